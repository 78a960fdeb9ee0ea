"""Multi-token paged attention (chunked prefill, verification of drafted tokens).

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``).

Source: "vLLM PagedAttention: Buoc dot pha ve thong luong suy luan LLM"
(vi.news.hada.io), the list of advanced features built on PagedAttention:
chunked prefill (a long prompt's prefill split into chunks) and speculative
decoding (tokens drafted by a smaller model, then checked).  Both attend
several new tokens of a sequence at once over its paged cache.  The page
gives no formula; the reading taken here is the plain causal one, the
aiwiki.vn page's statement of attention (a position attends to the positions
it may see) applied to every new token:

* sequence s has a context of L_s tokens in the cache, the last Q_s of which
  are this call's query tokens (their K/V already written);
* query i (0 <= i < Q_s) sits at position p = L_s - Q_s + i and attends to the
  tokens 0 .. p:
      out[i, h] = sum_{t <= p} softmax_t(scale * q[i, h] . K[t, g]) V[t, g],
  g = h // (Hq / Hkv).
Q_s = 1 is the decode step.
"""
from __future__ import annotations

import numpy as np


def multi_token_attention(q_seqs, k_seqs, v_seqs, scale):
    """fp64 causal attention of each sequence's last Q_s positions.

    q_seqs[s]: [Q_s, Hq, D]; k_seqs[s], v_seqs[s]: [L_s, Hkv, D] with
    Q_s <= L_s.  Returns a list of [Q_s, Hq, D] float64 arrays.
    """
    outs = []
    for q, k, v in zip(q_seqs, k_seqs, v_seqs):
        q = np.asarray(q, dtype=np.float64)
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        Q, Hq, D = q.shape
        L, Hkv = k.shape[0], k.shape[1]
        if Q > L:
            raise ValueError("a sequence cannot have more query tokens than context tokens")
        G = Hq // Hkv
        out = np.zeros((Q, Hq, D), dtype=np.float64)
        for i in range(Q):
            p = L - Q + i
            for h in range(Hq):
                g = h // G
                s = scale * (k[:p + 1, g, :] @ q[i, h, :])
                w = np.exp(s - s.max())
                out[i, h, :] = (w / w.sum()) @ v[:p + 1, g, :]
        outs.append(out)
    return outs
