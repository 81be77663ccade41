/*
 * exact_attention_12_gb300 — fused exact scaled dot-product attention for
 * NVIDIA GB300 (sm_103a).  C interface.
 *
 * The operation (FlashAttention: Fast and Memory-Efficient Exact Attention
 * with IO-Awareness, Dao et al. 2022, as summarised on the pages
 * "FlashAttention: Cơ chế Attention chính xác, nhanh và tối ưu bộ nhớ với
 * nhận thức IO" (xyznot.com, "Phương pháp"), "3.3 Hiểu sâu cơ chế
 * Self-Attention" (§3 Scaled Dot-Product Attention, §10 Causal Mask, §12
 * FlashAttention) and the azimuth.plus FlashAttention explainer
 * ("الخوارزمية خطوة بخطوة", the step-by-step algorithm)):
 *
 *   S = scale * Q K^T, with S_ij = -inf where key j is not allowed for query i
 *   L_i = logsumexp_j S_ij               (natural log, fp32)
 *   P = exp(S - L),  P~ = P * Z / (1 - p')  (Z: Philox dropout keep mask)
 *   O = P~ V
 *
 * Allowed(i, j) = (!causal || j <= i) && j < key_lens[b] &&
 *                 block_mask[i / 128][j / 128] != 0.
 * A row with no allowed key gets O_i = 0 and L_i = -inf.
 *
 * Backward (chain rule of the above; the pages state only that S and P are
 * recomputed from Q, K, V and the stored statistics):
 *   D = rowsum(dO * O),  dV = P~^T dO,  dP = (dO V^T) * Z / (1 - p'),
 *   dS = P * (dP - D),   dQ = scale * dS K,  dK = scale * dS^T Q.
 *
 * Dropout keep mask: Philox4x32-10 (Salmon et al., SC'11) at counter
 * (floor(j / 8), i, b * H + h, philox_offset) under key (low 32 bits of
 * philox_seed, high 32 bits) gives four 32-bit words; word (j mod 8) / 2
 * holds the 16-bit uniform u of element (b, h, i, j) in its low half when j
 * is even, its high half when j is odd.  The element is dropped iff u < T,
 * T = min(2^16 - 1, floor(dropout_p * 2^16)) computed in fp64 from the float
 * dropout_p: the drop rate is exactly p' = T / 2^16 (within 2^-16 of
 * dropout_p) and kept probabilities are scaled by 1 / (1 - p'), so P~ =
 * P * Z / (1 - p').  The backward call regenerates the same mask.
 *
 * Layout: Q, K, V, O, dO, dQ, dK, dV are logical [B, H, N, d] arrays with
 * unit stride along d and the element strides stride_b, stride_h, stride_n
 * (shared by all eight tensors).  lse is a contiguous fp32 [B, H, N].
 * Every device pointer must be 16-byte aligned; strides must be multiples
 * of 8 elements (bf16) or 4 elements (fp32).
 *
 * Ownership: the caller allocates and owns every buffer, including the
 * workspace `ws` (device memory, at least attn_workspace_size() bytes).  The
 * library allocates nothing and keeps no state between calls.  The first
 * 256 bytes of a workspace hold a device status word and the forward's work
 * counter, and must be zero before the workspace is first used; every
 * forward leaves the counter at zero when it completes, and attn_check()
 * reads and clears the status word.
 *
 * Streams: every call only enqueues work on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and returns.  Argument errors are detected on
 * the host before anything is enqueued.  Launch failures return
 * ATTN_ERR_CUDA.  A kernel that stops making progress gives up after a
 * bounded wait and records ATTN_ERR_TIMEOUT in the workspace status word,
 * which attn_check() returns.
 *
 * CUDA graphs: attn_fwd, attn_bwd and attn_decode neither synchronise nor
 * allocate, and every launch argument (tensor maps included) is passed by
 * value, so the calls can be captured into a CUDA graph and replayed.  Make
 * one uncaptured call of each kind first: it sets the kernels' attributes.
 * The forward and backward kernels are launched with programmatic stream
 * serialisation; each waits for the preceding work in the stream to complete
 * before it reads or writes global memory.
 *
 * Thread safety: calls on different workspaces may run concurrently; two
 * calls in flight on the same workspace race.
 */
#ifndef EXACT_ATTENTION_12_GB300_ATTN_H
#define EXACT_ATTENTION_12_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,   /* bad shape, stride, pointer, scale, p, ... */
  ATTN_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. fp32 bwd) */
  ATTN_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  ATTN_ERR_TIMEOUT = 4,       /* a kernel wait gave up (device status) */
  ATTN_ERR_WORKSPACE = 5      /* workspace missing, misaligned or too small */
} attn_status;

typedef enum { ATTN_BF16 = 0, ATTN_FP32 = 1, ATTN_FP8_E4M3 = 2 } attn_dtype;

typedef struct attn_params {
  int32_t B, H, N, d;        /* batch, heads, sequence length, head dim.
                                d in {64, 128}.  B, H or N = 0: no work. */
  int32_t dtype;             /* attn_dtype.  bf16: forward and backward;
                                fp32: forward only, on the tensor cores in
                                TF32 (the scores as three TF32 products of
                                the operands' high and low parts, P V as
                                one), fp32 o; fp8 (E4M3 q, k, v with the
                                de-scale factors below, bf16 o): forward
                                only, d = 128, no dropout. */
  float scale;               /* score scale, e.g. 1/sqrt(d); finite */
  int32_t causal;            /* nonzero: keep j <= i (top-left aligned) */
  float dropout_p;           /* drop probability in [0, 1); 0 = no dropout */
  uint64_t philox_seed;      /* Philox key */
  uint64_t philox_offset;    /* Philox counter word 3; must be < 2^32 */
  const int32_t* key_lens;   /* device [B]: keys j >= key_lens[b] masked;
                                NULL = all N keys valid.  Values are
                                clamped to [0, N]. */
  const uint8_t* block_mask; /* device uint8 [nb][nb], nb = ceil(N / 128),
                                row-major; nonzero = 128x128 block kept;
                                NULL = dense.  bf16 only. */
  int64_t block_mask_head_stride; /* bytes between the masks of consecutive
                                (b * H + h); 0 = one mask for all heads */
  int64_t stride_b, stride_h, stride_n; /* element strides of q, o, dout,
                                dq (and of k, v, dk, dv when the kv_stride
                                fields are 0) */
  /* Grouped-query attention ("3.3 Hiểu sâu cơ chế Self-Attention", §9.2
   * MQA and §9.3 GQA): the query heads are split into H_kv groups of H / H_kv
   * consecutive heads that share one key/value head, so query head h reads
   * key/value head h / (H / H_kv).  k, v, dk and dv are [B, H_kv, N, d]; dk
   * and dv of a shared head are the sums over its group.  H_kv = H (or 0) is
   * ordinary multi-head attention, H_kv = 1 multi-query attention. */
  int32_t H_kv;              /* key/value heads, dividing H; 0 = H */
  int32_t reserved;          /* must be 0 */
  int64_t kv_stride_b, kv_stride_h, kv_stride_n; /* element strides of k, v,
                                dk, dv; all three 0 = the strides above
                                (then H_kv must equal H) */
  /* FP8 inputs (dtype ATTN_FP8_E4M3).  The FlashAttention explainer
   * (azimuth.plus, timeline entry "FlashAttention-3") names FP8 as the
   * Hopper successor's step to higher throughput; the format is E4M3 of the
   * OCP 8-bit floating point specification (bias 7, largest value 448, no
   * infinities).  The attention is that of the real values
   *   Q = q_descale * q,  K = k_descale * k,  V = v_descale * v,
   * so the scores are scale * q_descale * k_descale * (q k^T).  The kernel
   * rounds the probabilities to E4M3 for the P V product (the row sums
   * that normalise O are taken before rounding), so O carries an error of
   * at most 2^-4 * sum_j P_ij |V_jc| + 2^-10 * max_j P_ij * sum_j |V_jc|
   * beyond the bf16 rounding of O; L is exact up to fp32 arithmetic.
   * o is bf16 [B, H, N, d] with the query strides.  Strides are in
   * elements and must be multiples of 16.  0 means 1 for each factor;
   * ignored for the other dtypes. */
  float q_descale, k_descale, v_descale;
  int32_t reserved2;         /* must be 0 */
} attn_params;

/* Bytes of device workspace a forward (for_backward = 0) or backward
 * (for_backward != 0) call needs.  Returns 0 if the parameters are invalid
 * (the call itself then reports why). */
size_t attn_workspace_size(const attn_params* p, int for_backward);

/* Forward: O [B,H,N,d] (same dtype as q; bf16 for fp8 inputs) and lse
 * [B,H,N] fp32.  For fp8 the workspace also holds a transposed copy of v
 * ([B, H_kv, d, N] padded to a multiple of 128 keys), written by the call;
 * for fp32 it holds the high and low TF32 parts of q and k and a transposed
 * copy of v, written by the call. */
attn_status attn_fwd(const attn_params* p, const void* q, const void* k,
                     const void* v, void* o, float* lse, void* ws,
                     size_t ws_bytes, void* stream);

/* Backward (bf16): needs o and lse from attn_fwd with the same parameters
 * (dropout seed and offset included).  Writes dq [B,H,N,d] and dk, dv
 * [B,H_kv,N,d] bf16. */
attn_status attn_bwd(const attn_params* p, const void* q, const void* k,
                     const void* v, const void* o, const float* lse,
                     const void* dout, void* dq, void* dk, void* dv, void* ws,
                     size_t ws_bytes, void* stream);

/* The three stages attn_bwd runs, callable one by one on the same workspace
 * (for callers that schedule or time them separately):
 *   attn_bwd_preprocess  D = rowsum(dO * O) and L * log2(e) into the
 *                        workspace (rows padded to a multiple of 128);
 *                        zeroes the workspace's fp32 dQ accumulator.
 *   attn_bwd_main        the fused recomputing backward: dK, dV written,
 *                        dQ accumulated into the workspace.  Reads what the
 *                        preprocess of the same call sequence wrote.
 *   attn_bwd_dq          dQ = scale * accumulator, converted to bf16.
 * Arguments mean the same as for attn_bwd; the workspace must be the same
 * and at least attn_workspace_size(p, 1) bytes. */
attn_status attn_bwd_preprocess(const attn_params* p, const void* o,
                                const float* lse, const void* dout, void* ws,
                                size_t ws_bytes, void* stream);
attn_status attn_bwd_main(const attn_params* p, const void* q, const void* k,
                          const void* v, const void* dout, void* dk, void* dv,
                          void* ws, size_t ws_bytes, void* stream);
attn_status attn_bwd_dq(const attn_params* p, void* dq, void* ws,
                        size_t ws_bytes, void* stream);

/* Backward without a caller workspace.  The pages have no counterpart: this
 * is an interface for callers that cannot allocate device memory (a plug-in
 * inside a host application that owns all device allocations, a runtime with
 * a fixed device-memory budget, a latency-critical loop where cudaMalloc
 * could synchronise the device).  Arguments and results are those of
 * attn_bwd; the scratch attn_bwd would take from `ws` comes from a 64 MiB
 * array built into the library, which every GPU that loads the library holds
 * until the process exits.
 *   - Problems needing more than 64 MiB of scratch (attn_workspace_size(p, 1))
 *     are rejected with ATTN_ERR_WORKSPACE before anything is enqueued.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and caches it; make that
 *     first call before any stream capture.
 *   - All calls share the one array and it keeps the previous call's
 *     contents: calls that overlap on the GPU (other streams, other host
 *     threads) race with each other.  The call clears the status words and
 *     rewrites everything else it reads.
 *   - A device-side time-out is recorded in the built-in array's status
 *     words: attn_check(NULL, stream) reports it (and clears it).  The next
 *     attn_bwd_noalloc call clears it too, so check before the next call. */
attn_status attn_bwd_noalloc(const attn_params* p, const void* q,
                             const void* k, const void* v, const void* o,
                             const float* lse, const void* dout, void* dq,
                             void* dk, void* dv, void* stream);

/* Decode step: the newest n_q query positions of each sequence against its
 * key/value cache.  The pages' pass is the training forward; this is the
 * same attention at generation time, where each new token attends the keys
 * cached so far (the KV cache of "3.3 Hiểu sâu cơ chế Self-Attention", §9).
 *   p->N          cache capacity: k and v are [B, H_kv, N, d] (key/value
 *                 strides and grouping as in attn_params)
 *   p->key_lens   required, device [B]: cached keys per sequence, clamped to
 *                 [0, N].  Query row t of sequence b is the token at position
 *                 key_lens[b] - n_q + t.
 *   p->causal     nonzero: query t attends keys j <= its position; otherwise
 *                 every cached key
 *   q, o          [B, H, n_q, d] with the query strides (stride_n steps over
 *                 the n_q rows); bf16
 *   lse           fp32 [B, H, n_q] (natural log; -inf for a row with no key)
 * 1 <= n_q and (H / H_kv) * n_q <= 64; dropout_p must be 0 and block_mask
 * NULL (ATTN_ERR_UNSUPPORTED otherwise).  The cache is split into chunks
 * processed in parallel and merged by the logsumexp rule; the workspace
 * (attn_decode_workspace_size bytes, the same 256-byte header rules as
 * above) holds the per-chunk partial results. */
size_t attn_decode_workspace_size(const attn_params* p, int32_t n_q);
attn_status attn_decode(const attn_params* p, int32_t n_q, const void* q, const void* k,
                        const void* v, void* o, float* lse, void* ws, size_t ws_bytes,
                        void* stream);

/* Diagnostic: runs the kernels' time-out path on purpose.  Enqueues one warp
 * that waits on a barrier nothing arrives at, giving up after `limit_ns`
 * (clamped to [1 ms, 2 s]); it records ATTN_ERR_TIMEOUT in the workspace's
 * status words exactly as a stalled attention kernel would, so a following
 * attn_check returns ATTN_ERR_TIMEOUT.  `ws` needs 256 bytes. */
attn_status attn_selftest_timeout(void* ws, uint64_t limit_ns, void* stream);

/* Test hook for the time-out path of the attention kernels themselves (the
 * pages have no counterpart: this checks this library's failure detection).
 * Arms a one-shot stall for the next launch of the named kernel made by a
 * call on the calling host thread:
 *   ATTN_STALL_FWD_SOFTMAX  the forward (attn_fwd, bf16 or fp8): in every CTA,
 *                           softmax warp 0 withholds its "P ready" arrive for
 *                           its first key tile;
 *   ATTN_STALL_BWD_COMPUTE  the backward main kernel (attn_bwd, attn_bwd_main,
 *                           attn_bwd_noalloc): in every CTA, compute warp 0
 *                           withholds its "P ready" arrive for its first
 *                           query tile.
 * The MMA warp's wait on that barrier then runs out; every wait of that launch
 * gives up after `limit_ns` (clamped to [1 ms, 2 s]).  The kernel drains its
 * copies and MMAs, frees its tensor memory and returns, and the status words
 * of the call's workspace hold ATTN_ERR_TIMEOUT and the wait site, which
 * attn_check reports.  That call's outputs are undefined; later calls are
 * unaffected.  Nothing faults, traps or hangs.  ATTN_STALL_NONE disarms;
 * other values give ATTN_ERR_INVALID_ARG. */
typedef enum {
  ATTN_STALL_NONE = 0,
  ATTN_STALL_FWD_SOFTMAX = 1,
  ATTN_STALL_BWD_COMPUTE = 2
} attn_stall;
attn_status attn_debug_stall(int32_t which, uint64_t limit_ns);

/* Synchronises `stream`, returns the workspace's device status (ATTN_OK or
 * ATTN_ERR_TIMEOUT) and clears it.  ws = NULL: the status of
 * attn_bwd_noalloc's built-in scratch on the current device. */
attn_status attn_check(void* ws, void* stream);

/* Static description of a status code. */
const char* attn_status_string(attn_status s);

/* Detail message of the last non-OK status returned on the calling thread. */
const char* attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTENTION_12_GB300_ATTN_H */
