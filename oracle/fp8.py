"""FP8 (E4M3) attention forward — TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The FlashAttention explainer (azimuth.plus, the timeline entry
"FlashAttention-3") names FP8 arithmetic as the Hopper successor's next step
for throughput.  The pages fix nothing about the format, so this module takes
the plain reading: the inputs Q, K, V are stored as 8-bit E4M3 codes with one
fp32 de-scale factor per tensor, and the attention of the real values

    Q = q_descale * e4m3(Q8),  K = k_descale * e4m3(K8),  V = v_descale * e4m3(V8)

is the exact attention of attention.py (same masks, same O and L), evaluated
in fp64 on those values.

E4M3 is the format of the OCP "8-bit Floating Point Specification (OFP8)"
(revision 1.0, 2023): one sign bit, four exponent bits with bias 7, three
mantissa bits.  Exponent field 0 holds zero and the subnormals m/8 * 2^-6;
fields 1..15 hold (1 + m/8) * 2^(e - 7); the single NaN pattern per sign is
S.1111.111 and there are no infinities, so the largest finite value is
1.75 * 2^8 = 448.

The second half of the module gives the terms of the error bound a kernel
that rounds the probabilities to E4M3 before P V must meet (see
`rounding_terms`).
"""

import numpy as np

from .attention import allowed_mask, attention_forward, _group

E4M3_MAX = 448.0


def e4m3_value(codes):
    """fp64 values of E4M3 codes (uint8 array-like); NaN for S.1111.111."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 0xF) & (c & 0x7 == 0x7), np.nan, mag)
    return sign * mag


def dequantize(codes, descale):
    """Real values descale * e4m3(codes), fp64, same shape as `codes`."""
    return float(np.float32(descale)) * e4m3_value(codes)


def fp8_forward(q8, k8, v8, q_descale, k_descale, v_descale, scale, causal=False,
                key_lens=None, block_mask=None):
    """O [B,H,N,d] and L [B,H,N] (fp64) of the attention of the de-scaled E4M3
    inputs.  q8: uint8 codes [B,H,N,d]; k8, v8: [B,H_kv,N,d]."""
    q = dequantize(q8, q_descale)
    k = dequantize(k8, k_descale)
    v = dequantize(v8, v_descale)
    return attention_forward(q, k, v, scale, causal=causal, key_lens=key_lens,
                             block_mask=block_mask)


def rounding_terms_rows(q, k, v, b, h, rows, scale, causal=False, key_lens=None,
                        block_mask=None):
    """The terms of `rounding_terms` for the query rows `rows` of head (b, h)
    only: (A, T), each [len(rows), d].  q, k, v: real values, [B,H,N,d] and
    [B,H_kv,N,d]."""
    N, d = np.shape(q)[2], np.shape(q)[3]
    g = _group(q, k)
    c = float(np.float32(scale))
    rows = np.asarray(rows, dtype=np.int64)
    kl = None if key_lens is None else int(np.asarray(key_lens)[b])
    bm = None
    if block_mask is not None:
        bm = np.asarray(block_mask)
        bm = bm if bm.ndim == 2 else bm[b, h]
    allow = allowed_mask(rows, np.arange(N), causal, kl, bm)
    qh = np.asarray(q[b, h], dtype=np.float64)[rows]
    kh = np.asarray(k[b, h // g], dtype=np.float64)
    vh = np.abs(np.asarray(v[b, h // g], dtype=np.float64))
    A = np.zeros((rows.size, d))
    T = np.zeros((rows.size, d))
    live = allow.any(axis=1)
    if live.any():
        S = np.where(allow[live], c * (qh[live] @ kh.T), -np.inf)
        E = np.exp(S - S.max(axis=1, keepdims=True))
        l0 = E.sum(axis=1, keepdims=True)
        A[live] = (E / l0) @ vh
        T[live] = (allow[live].astype(np.float64) @ vh) / l0
    return A, T


def rounding_terms(q, k, v, scale, causal=False, key_lens=None, block_mask=None):
    """Per output element (b, h, i, c), the two sums the E4M3 rounding of the
    probabilities is bounded by.  q, k, v are real (de-scaled) values.

      A[b,h,i,c] = sum_j P_ij |V_jc|
      T[b,h,i,c] = (max_j P_ij) * sum_{j allowed} |V_jc|

    P is the softmax of the masked scaled scores (attention.py).  If a kernel
    forms unnormalised weights w_j = gamma * exp(S_ij - m_i) with gamma >= 1
    (m_i the row max; a lazily updated max gives gamma >= 1), rounds each to
    E4M3 (error at most 2^-4 w_j in the normal range, 2^-10 below 2^-6), and
    divides sum_j round(w_j) V_jc by the unrounded sum_j w_j, its error is at
    most 2^-4 A + 2^-10 T: max_j P_ij = exp(m_i - L_i) = 1 / sum_j exp(S_ij - m_i).
    Rows with no allowed key get 0.
    """
    B, H, N, d = np.shape(q)
    A = np.zeros((B, H, N, d))
    T = np.zeros((B, H, N, d))
    for b in range(B):
        for h in range(H):
            A[b, h], T[b, h] = rounding_terms_rows(q, k, v, b, h, np.arange(N), scale,
                                                   causal, key_lens, block_mask)
    return A, T
