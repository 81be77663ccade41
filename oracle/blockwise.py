"""The pages' tiled online-softmax forward, restated — used only to pin the oracle.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Sources:
  * FlashAttention paper summary (xyznot.com/vi/paper/2205.14135), "Theo dõi
    Softmax tăng dần" (incremental softmax statistics) and its four per-block
    steps: block scores, block max and exp-sum, merged statistics, rescaled
    output update.
  * The azimuth.plus FlashAttention explainer, "الخوارزمية خطوة بخطوة" (the
    step-by-step algorithm): outer loop over K/V blocks, inner loop over Q
    blocks, running (m, l) per row, division by l once at the end.

This module walks the blocks in that order and keeps the running row max m
and running exp-sum l.  It has no masks and no dropout: its only use is to
show that the direct definition in `attention.py` produces the same
statistics and output as the blockwise recurrence, for any block size.
"""

import numpy as np


def blockwise_forward(q, k, v, scale, block_r, block_c):
    """Tiled forward for one head; q, k, v: [N, d] fp64.

    Returns (O, m, l): the output normalised at the end, the running row max
    of the scaled scores and the running exp-sum relative to that max.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    N, d = q.shape
    acc = np.zeros((N, v.shape[1]))      # un-normalised output
    m = np.full(N, -np.inf)              # running row max
    l = np.zeros(N)                      # running exp-sum w.r.t. m
    for j0 in range(0, N, block_c):      # outer loop: K/V blocks
        kj = k[j0:j0 + block_c]
        vj = v[j0:j0 + block_c]
        for i0 in range(0, N, block_r):  # inner loop: Q blocks
            rs = slice(i0, i0 + block_r)
            s = scale * (q[rs] @ kj.T)
            m_blk = s.max(axis=1)                      # block row max
            p_blk = np.exp(s - m_blk[:, None])         # block probabilities
            l_blk = p_blk.sum(axis=1)                  # block exp-sum
            m_new = np.maximum(m[rs], m_blk)
            a_old = np.exp(m[rs] - m_new)              # rescale of old stats
            a_blk = np.exp(m_blk - m_new)              # rescale of block stats
            acc[rs] = a_old[:, None] * acc[rs] + a_blk[:, None] * (p_blk @ vj)
            l[rs] = a_old * l[rs] + a_blk * l_blk
            m[rs] = m_new
    return acc / l[:, None], m, l
