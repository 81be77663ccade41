"""Plain fp64 exact attention, forward and backward — the oracle.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  Only tests/, the package
smoke check and the bench's CPU-baseline leg may call this module.

What it computes, per (batch b, head h), on the exact fp64 upcast of the
inputs the GPU sees:

  1. S = c * Q K^T                         scaled scores ("3.3 Hiểu sâu cơ chế
                                            Self-Attention", §3.2–3.3, §4.1)
  2. S_ij = -inf where (i, j) is not allowed: causal (keep j <= i, the lower
     triangle with its diagonal, §10.2 of the same page), key padding
     (keep j < len_b, the masked_fill rule of §4.1), block mask (keep iff
     M[i // 128][j // 128] = 1, the block-sparse mask of the FlashAttention
     paper summary, "Block-Sparse FlashAttention" section).
  3. m = rowmax S; L = m + ln sum_j exp(S_ij - m)   (safe softmax, §7.2;
     L is the stored softmax statistic of the paper summary's
     "recomputation in the backward pass" idea, kept as one logsumexp)
  4. P = exp(S - L)                          (softmax, §3.4)
  5. P~ = P * Z / (1 - p')                   (dropout on the probabilities,
     fused between softmax and the second matmul per the kernel-fusion idea;
     Z is the Philox keep mask defined in `keep_mask`, p' = T / 2^16 its exact
     drop rate, see `dropout_threshold`)
  6. O = P~ V                                (§3.5)

A row with no allowed key has L = -inf, P = 0, O = 0 and contributes nothing
to any gradient.

Grouped-query attention ("3.3 Hiểu sâu cơ chế Self-Attention", §9.2 MQA and
§9.3 GQA): K and V may have H_kv heads, H_kv dividing H; the query heads are
split into H_kv groups of H / H_kv consecutive heads and every head of a group
reads the same key/value head, so query head h reads key/value head
h // (H / H_kv).  H_kv = H is ordinary multi-head attention and H_kv = 1 is
multi-query attention.  The gradient of a shared key/value head is the sum of
the per-head gradients over its group.

Backward (the chain rule applied to the definition above; the pages state only
that S and P are recomputed):

  dV = P~^T dO,  dP~ = dO V^T,  dP = dP~ * Z / (1 - p'),
  D = rowsum(dO * O)  (= rowsum(P * dP)),  dS = P * (dP - D),
  dQ = c * dS K,  dK = c * dS^T Q.

Evaluation order: query rows are processed in chunks so that no fp64 N x N
array is held; within a chunk every row's full score vector over the keys it
may attend is materialised.  Keys that no row of the chunk may attend are left
out of the chunk's products: their probability is exactly 0 by the definition.
"""

import math

import numpy as np

from .philox import philox4x32_10

BLOCK = 128          # block-mask granularity in rows and columns
_ROW_CHUNK = 256     # query rows per chunk


def dropout_threshold(p):
    """Integer drop threshold T = min(2^16 - 1, floor(p * 2^16)).

    p is taken at float32 precision (the width the C interface carries) and
    the product is formed in fp64, where it is exact.  An element is dropped
    iff its 16-bit uniform u satisfies u < T, so the drop probability is
    exactly T / 2^16 (within 2^-16 of p).
    """
    p32 = float(np.float32(p))
    if p32 <= 0.0:
        return 0
    return min(2 ** 16 - 1, int(math.floor(p32 * 2.0 ** 16)))


def keep_scale(p):
    """Scale of the kept probabilities: 1 / (1 - T / 2^16), the inverse keep rate."""
    T = dropout_threshold(p)
    return 2.0 ** 16 / (2.0 ** 16 - T) if T else 1.0


def keep_mask(rows, cols, bh, seed, offset, p):
    """Dropout keep mask Z[i, j] in {0, 1} for one (b, h).

    rows, cols: 1-D integer arrays of query/key indices; bh = b * H + h.
    Counter = (floor(j / 8), i, bh, offset), key = (low 32 bits of seed,
    high 32 bits of seed).  Of the four 32-bit Philox4x32-10 output words,
    word (j mod 8) div 2 holds keys j with j mod 2 = 0 in its low 16 bits and
    j mod 2 = 1 in its high 16 bits; that 16-bit value is the uniform u of
    element (i, j); keep iff u >= T (see dropout_threshold).
    """
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    T = dropout_threshold(p)
    if T == 0:
        return np.ones((rows.size, cols.size), dtype=bool)
    seed = int(seed)
    k0, k1 = seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF
    groups, inv = np.unique(cols // 8, return_inverse=True)
    words = philox4x32_10(groups[None, :], rows[:, None], bh, int(offset), k0, k1)
    stacked = np.stack(words, axis=-1)                 # [R, G, 4]
    w = stacked[:, inv, (cols % 8) // 2]               # [R, C]
    u16 = (w.astype(np.uint64) >> (16 * (cols % 2)).astype(np.uint64)) & np.uint64(0xFFFF)
    return u16 >= np.uint64(T)


def allowed_mask(rows, cols, causal=False, key_len=None, block_mask=None):
    """Boolean [len(rows), len(cols)]: True where key j may be attended by row i."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    a = np.ones((rows.size, cols.size), dtype=bool)
    if causal:
        a &= cols[None, :] <= rows[:, None]
    if key_len is not None:
        a &= (cols < int(key_len))[None, :]
    if block_mask is not None:
        bm = np.asarray(block_mask).astype(bool)
        a &= bm[np.ix_(rows // BLOCK, cols // BLOCK)]
    return a


class _Head:
    """One (b, h) problem in fp64, with its masking and dropout settings."""

    def __init__(self, q, k, v, scale, causal, key_len, block_mask,
                 dropout_p, seed, offset, bh):
        self.q = np.asarray(q, dtype=np.float64)
        self.k = np.asarray(k, dtype=np.float64)
        self.v = np.asarray(v, dtype=np.float64)
        self.N = self.q.shape[0]
        self.c = float(np.float32(scale))
        self.causal = bool(causal)
        self.key_len = None if key_len is None else int(key_len)
        self.block_mask = block_mask
        self.p = float(np.float32(dropout_p))
        self.seed, self.offset, self.bh = seed, offset, bh

    def chunk(self, rows):
        """Scores, softmax statistics and probabilities for a set of rows."""
        A = allowed_mask(rows, np.arange(self.N), self.causal, self.key_len,
                         self.block_mask)
        cols = np.nonzero(A.any(axis=0))[0]
        S = self.c * (self.q[rows] @ self.k[cols].T)
        S = np.where(A[:, cols], S, -np.inf)
        if cols.size:
            m = S.max(axis=1)
        else:
            m = np.full(len(rows), -np.inf)
        live = np.isfinite(m)
        L = np.full(len(rows), -np.inf)
        P = np.zeros_like(S)
        if live.any():
            Sl = S[live]
            ml = m[live]
            L[live] = ml + np.log(np.exp(Sl - ml[:, None]).sum(axis=1))
            P[live] = np.exp(Sl - L[live][:, None])
        if dropout_threshold(self.p) > 0:
            Z = keep_mask(rows, cols, self.bh, self.seed, self.offset, self.p)
            Zs = Z.astype(np.float64) * keep_scale(self.p)
        else:
            Zs = np.ones_like(P)
        return cols, P, Zs, L

    def forward(self, rows):
        cols, P, Zs, L = self.chunk(rows)
        O = (P * Zs) @ self.v[cols]
        return O, L

    def backward(self, rows, do_rows):
        """O, L, dQ for `rows`, and their contributions to dK, dV (full N)."""
        cols, P, Zs, L = self.chunk(rows)
        Pd = P * Zs
        O = Pd @ self.v[cols]
        D = (do_rows * O).sum(axis=1)
        dV = np.zeros_like(self.v)
        dK = np.zeros_like(self.k)
        dV[cols] = Pd.T @ do_rows
        dP = (do_rows @ self.v[cols].T) * Zs
        dS = P * (dP - D[:, None])
        dQ = self.c * (dS @ self.k[cols])
        dK[cols] = self.c * (dS.T @ self.q[rows])
        return O, L, dQ, dK, dV


def _chunks(rows, size=_ROW_CHUNK):
    rows = np.asarray(rows, dtype=np.int64)
    for s in range(0, rows.size, size):
        yield rows[s:s + size]


def _bm_for(block_mask, b, h):
    if block_mask is None:
        return None
    bm = np.asarray(block_mask)
    return bm if bm.ndim == 2 else bm[b, h]


def _group(q, k):
    """Query heads per key/value head (H / H_kv)."""
    H, H_kv = np.shape(q)[1], np.shape(k)[1]
    if H_kv < 1 or H % H_kv:
        raise ValueError(f"key/value heads ({H_kv}) must divide query heads ({H})")
    return H // H_kv


def _head(q, k, v, b, h, scale, causal, key_lens, block_mask, dropout_p,
          seed, offset):
    H = q.shape[1]
    hk = h // _group(q, k)
    kl = None if key_lens is None else int(np.asarray(key_lens)[b])
    return _Head(q[b, h], k[b, hk], v[b, hk], scale, causal, kl,
                 _bm_for(block_mask, b, h), dropout_p, seed, offset, b * H + h)


def forward_rows(q, k, v, b, h, rows, scale, causal=False, key_lens=None,
                 block_mask=None, dropout_p=0.0, seed=0, offset=0):
    """O[b, h, rows] and L[b, h, rows] for sampled rows of one head.

    q, k, v: arrays [B, H, N, d]; rows: 1-D indices.  Returns fp64 arrays.
    """
    hd = _head(q, k, v, b, h, scale, causal, key_lens, block_mask, dropout_p,
               seed, offset)
    outs = [hd.forward(r) for r in _chunks(rows)]
    O = np.concatenate([o for o, _ in outs]) if outs else np.zeros((0, hd.v.shape[1]))
    L = np.concatenate([l for _, l in outs]) if outs else np.zeros(0)
    return O, L


def backward_keys(q, k, v, do, b, hk, keys, scale, causal=False, key_lens=None,
                  block_mask=None, dropout_p=0.0, seed=0, offset=0):
    """dK[b, hk, keys] and dV[b, hk, keys] for sampled keys of key/value head hk.

    The query heads of hk's group all contribute.  Only query rows that may
    attend at least one of `keys` contribute, so only those rows are
    evaluated (each over its full score row).
    """
    g = _group(q, k)
    keys = np.asarray(keys, dtype=np.int64)
    dK = np.zeros(np.shape(k)[2:])
    dV = np.zeros(np.shape(v)[2:])
    for h in range(hk * g, (hk + 1) * g):
        hd = _head(q, k, v, b, h, scale, causal, key_lens, block_mask, dropout_p,
                   seed, offset)
        A = allowed_mask(np.arange(hd.N), keys, hd.causal, hd.key_len, hd.block_mask)
        rows = np.nonzero(A.any(axis=1))[0]
        dob = np.asarray(do[b, h], dtype=np.float64)
        for r in _chunks(rows):
            _, _, _, dk, dv = hd.backward(r, dob[r])
            dK += dk
            dV += dv
    return dK[keys], dV[keys]


def backward_rows(q, k, v, do, b, h, rows, scale, causal=False, key_lens=None,
                  block_mask=None, dropout_p=0.0, seed=0, offset=0):
    """dQ[b, h, rows] for sampled query rows of one head (each row in full)."""
    hd = _head(q, k, v, b, h, scale, causal, key_lens, block_mask, dropout_p,
               seed, offset)
    dob = np.asarray(do[b, h], dtype=np.float64)
    out = [hd.backward(r, dob[r])[2] for r in _chunks(rows)]
    return np.concatenate(out) if out else np.zeros((0, hd.q.shape[1]))


def attention_forward(q, k, v, scale, causal=False, key_lens=None,
                      block_mask=None, dropout_p=0.0, seed=0, offset=0):
    """Full forward.  q: [B, H, N, d]; k, v: [B, H_kv, N, d] with H_kv dividing H.
    Returns O [B,H,N,d], L [B,H,N] (fp64).

    block_mask: None, [nb, nb] shared by every (b, h), or [B, H, nb, nb].
    key_lens: None or [B] integers.
    """
    B, H, N, d = np.shape(q)
    O = np.zeros((B, H, N, d))
    L = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            hd = _head(q, k, v, b, h, scale, causal, key_lens, block_mask,
                       dropout_p, seed, offset)
            for r in _chunks(np.arange(N)):
                O[b, h, r], L[b, h, r] = hd.forward(r)
    return O, L


def attention_backward(q, k, v, do, scale, causal=False, key_lens=None,
                       block_mask=None, dropout_p=0.0, seed=0, offset=0):
    """Full forward + backward.  Returns (O, L, dQ, dK, dV) in fp64; dK and dV
    have the key/value heads of k and v."""
    B, H, N, d = np.shape(q)
    g = _group(q, k)
    O = np.zeros((B, H, N, d))
    L = np.zeros((B, H, N))
    dQ = np.zeros((B, H, N, d))
    dK = np.zeros(np.shape(k))
    dV = np.zeros(np.shape(v))
    for b in range(B):
        for h in range(H):
            hd = _head(q, k, v, b, h, scale, causal, key_lens, block_mask,
                       dropout_p, seed, offset)
            dob = np.asarray(do[b, h], dtype=np.float64)
            for r in _chunks(np.arange(N)):
                o, l, dq, dk, dv = hd.backward(r, dob[r])
                O[b, h, r], L[b, h, r], dQ[b, h, r] = o, l, dq
                dK[b, h // g] += dk
                dV[b, h // g] += dv
    return O, L, dQ, dK, dV


def decode_forward(q, k, v, scale, cache_lens, causal=True):
    """Attention of the newest query positions of each sequence against its
    key/value cache (the decode step of autoregressive generation).

    q: [B, H, N_q, d]; k, v: [B, H_kv, N_kv, d] (H_kv dividing H, grouped as
    above); cache_lens: [B] integers, 0 <= cache_lens[b] <= N_kv.  Query row t
    of batch b is the token at position cache_lens[b] - N_q + t, the last N_q
    positions of the cached sequence; it attends the cached keys
    j < cache_lens[b], and when `causal` only those with j <= its position
    (the causal mask of "3.3 Hiểu sâu cơ chế Self-Attention", §10.2, aligned
    to the end of the cache).  A row with no allowed key has O = 0 and
    L = -inf.  Returns O [B, H, N_q, d] and L [B, H, N_q] in fp64.
    """
    B, H, Nq, d = np.shape(q)
    g = _group(q, k)
    Nkv = np.shape(k)[2]
    lens = np.asarray(cache_lens, dtype=np.int64)
    c = float(np.float32(scale))
    O = np.zeros((B, H, Nq, d))
    L = np.full((B, H, Nq), -np.inf)
    cols = np.arange(Nkv)
    for b in range(B):
        n = int(lens[b])
        pos = n - Nq + np.arange(Nq)
        A = np.broadcast_to(cols[None, :] < n, (Nq, Nkv)).copy()
        if causal:
            A &= cols[None, :] <= pos[:, None]
        for h in range(H):
            qh = np.asarray(q[b, h], dtype=np.float64)
            kh = np.asarray(k[b, h // g], dtype=np.float64)
            vh = np.asarray(v[b, h // g], dtype=np.float64)
            S = np.where(A, c * (qh @ kh.T), -np.inf)
            live = A.any(axis=1)
            if not live.any():
                continue
            m = S[live].max(axis=1)
            Lr = m + np.log(np.exp(S[live] - m[:, None]).sum(axis=1))
            P = np.exp(S[live] - Lr[:, None])
            O[b, h, live] = P @ vh
            L[b, h, live] = Lr
    return O, L
