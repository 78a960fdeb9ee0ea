"""Pins for the multi-token (causal, several new tokens per sequence) oracle.

Pinned to an independent library routine (PyTorch's scaled_dot_product_attention
with an explicit mask, in float64), to the pinned decode oracle (one query token
is the decode step; the last query of a chunk sees the whole context), and to
causality (tokens after a query's position cannot change its output).  A wrong
diagonal offset, a transposed mask or a wrong head mapping fails one of them.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.multi_token import multi_token_attention


def _case(rng, L, Q, Hq=8, Hkv=2, D=16):
    q = rng.standard_normal((Q, Hq, D))
    k = rng.standard_normal((L, Hkv, D))
    v = rng.standard_normal((L, Hkv, D))
    return q, k, v


@pytest.mark.parametrize("L,Q", [(1, 1), (5, 5), (17, 4), (40, 16), (33, 1)])
def test_matches_library_sdpa_with_a_bottom_right_causal_mask(L, Q):
    rng = np.random.default_rng(L * 100 + Q)
    q, k, v = _case(rng, L, Q)
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    got = multi_token_attention([q], [k], [v], 0.3)[0]
    # query i may see key t iff t <= L - Q + i
    mask = torch.tensor([[t <= L - Q + i for t in range(L)] for i in range(Q)])
    qt = torch.from_numpy(q).permute(1, 0, 2)                      # [Hq, Q, D]
    kt = torch.from_numpy(np.repeat(k, G, axis=1)).permute(1, 0, 2)  # [Hq, L, D]
    vt = torch.from_numpy(np.repeat(v, G, axis=1)).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=0.3)
    assert np.allclose(got, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_one_query_is_the_decode_step():
    rng = np.random.default_rng(3)
    qs, ks, vs = zip(*[_case(rng, L, 1) for L in (1, 9, 70)])
    got = multi_token_attention(qs, ks, vs, 0.25)
    ref = oracle.decode_attention(np.stack([q[0] for q in qs]), ks, vs, 0.25)
    for s in range(3):
        assert np.allclose(got[s][0], ref[s], rtol=1e-12, atol=1e-13)


def test_last_query_sees_the_whole_context_and_earlier_ones_a_prefix():
    rng = np.random.default_rng(4)
    L, Q = 30, 6
    q, k, v = _case(rng, L, Q)
    got = multi_token_attention([q], [k], [v], 0.2)[0]
    for i in range(Q):
        p = L - Q + i
        ref = oracle.decode_attention(q[i][None], [k[:p + 1]], [v[:p + 1]], 0.2)[0]
        assert np.allclose(got[i], ref, rtol=1e-12, atol=1e-13)


def test_future_tokens_do_not_change_earlier_queries():
    rng = np.random.default_rng(5)
    L, Q = 25, 8
    q, k, v = _case(rng, L, Q)
    a = multi_token_attention([q], [k], [v], 0.5)[0]
    k2, v2 = k.copy(), v.copy()
    k2[L - 3:] += 7.0
    v2[L - 3:] -= 3.0
    b = multi_token_attention([q], [k2], [v2], 0.5)[0]
    # queries 0 .. Q-4 sit at positions <= L - 4: unchanged
    assert np.array_equal(a[:Q - 3], b[:Q - 3])
    assert not np.allclose(a[Q - 3:], b[Q - 3:])


def test_brute_force_tiny():
    q = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])   # Q 2, Hq 1, D 2
    k = np.array([[[1.0, 0.0]], [[0.0, 1.0]], [[1.0, 1.0]]])
    v = np.array([[[1.0, 2.0]], [[3.0, 4.0]], [[5.0, 6.0]]])
    got = multi_token_attention([q], [k], [v], 1.0)[0]
    # query 0 at position 1 sees tokens 0, 1: scores 1, 0
    w0 = np.exp([1.0, 0.0]); w0 /= w0.sum()
    # query 1 at position 2 sees tokens 0, 1, 2: scores 0, 1, 1
    w1 = np.exp([0.0, 1.0, 1.0]); w1 /= w1.sum()
    assert np.allclose(got[0, 0], w0 @ v[:2, 0])
    assert np.allclose(got[1, 0], w1 @ v[:, 0])


def test_more_queries_than_context_is_rejected():
    rng = np.random.default_rng(6)
    q, k, v = _case(rng, 3, 4)
    with pytest.raises(ValueError):
        multi_token_attention([q], [k], [v], 1.0)
