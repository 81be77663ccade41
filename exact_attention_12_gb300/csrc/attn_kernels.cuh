// Kernel argument blocks and launcher declarations shared by the host API
// (attn_api.cu) and the kernel translation units.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <cuda_bf16.h>

#include <atomic>
#include <utility>

#include "philox.cuh"

namespace attn {

// Launch with programmatic stream serialisation: the kernel's CTAs may start
// while the previous kernel of the stream is still running (its prologue
// overlaps that kernel's tail, and the launch latency is hidden).  Every
// kernel launched this way calls grid_dep_wait() before touching global
// memory.  Captured into a CUDA graph the dependency becomes a programmatic
// edge.
template <typename... P, typename... A>
inline cudaError_t launch_pdl(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, A&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// One-time set-up of a kernel instance (its shared-memory limit, the
// register check) is per device: `done` remembers the devices it has run on
// (up to 64; beyond that it runs on every call).  Returns the current device
// in *dev and whether the set-up is still to do there; mark_done records it.
inline cudaError_t needs_setup(const std::atomic<uint64_t>& done, int* dev, bool* todo) {
  const cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (*dev >= 0 && *dev < 64) ? (uint64_t{1} << *dev) : 0;
  *todo = bit == 0 || (done.load(std::memory_order_acquire) & bit) == 0;
  return cudaSuccess;
}

inline void mark_done(std::atomic<uint64_t>& done, int dev) {
  if (dev >= 0 && dev < 64) done.fetch_or(uint64_t{1} << dev, std::memory_order_release);
}

constexpr int kTile = 128;            // query/key tile rows == block-mask granularity
constexpr float kRescaleTau = 8.0f;   // lazy-rescale threshold, log2 units

// Where a kernel gave up waiting (recorded next to the status code).
enum WaitSite : int {
  kSiteFwdQ = 1, kSiteFwdK, kSiteFwdV, kSiteFwdKvEmpty, kSiteFwdSFull, kSiteFwdSFree,
  kSiteFwdPFull, kSiteFwdPvDone, kSiteFwdUnit,
  kSiteBwdLoad = 20, kSiteBwdKV, kSiteBwdQ, kSiteBwdMma, kSiteBwdSoft, kSiteBwdDq,
  kSiteBwdEmpty, kSiteBwdFree, kSiteBwdSmem,
  kSiteDecode = 40,
  kSiteTf32Load = 50, kSiteTf32Mma, kSiteTf32Soft
};

// One-shot stalls armed by attn_debug_stall (a test of the kernels' own
// time-out path): the named role withholds one barrier arrive in its first
// tile, so the wait on that barrier runs out.
enum StallSite : int { kStallNone = 0, kStallFwdSoftmax = 1, kStallBwdCompute = 2 };

// Device status code for a kernel that found its shared memory misaligned
// and returned without doing anything (equals ATTN_ERR_CUDA in attn.h).
constexpr int kStatusSmemAlign = 3;

// Per-call mask/dropout settings common to every kernel.
struct MaskArgs {
  int B, H, N;
  int H_kv;                       // key/value heads (divides H)
  int kv_group;                   // H / H_kv: query head h reads key/value head h / kv_group
  int causal;
  const int32_t* key_lens;        // [B] or null
  // block mask, compacted: for mask m and tile t, cnt[m * nb + t] sorted
  // tile indices in idx[(m * nb + t) * nb + ...]; null when dense
  const int32_t* list_cnt;
  const uint16_t* list_idx;
  int nb;                         // ceil(N / 128)
  int mask_per_head;              // 0: one mask for all (b, h)
  // dense block mask (read by the fp32 kernel directly)
  const uint8_t* block_mask;
  int64_t block_mask_head_stride;
  // dropout
  uint32_t drop_threshold;        // 0 = no dropout
  float drop_scale;               // 1 / (1 - p)
  uint32_t seed_lo, seed_hi, offset;
  PhiloxRoundKeys rk;             // the ten round keys of (seed_lo, seed_hi)
  // CTAs are scheduled in groups of `head_group` consecutive (b, h) so that a
  // group's re-read operands stay in L2
  int head_group;
};

struct FwdArgs {
  MaskArgs m;
  int d;
  float scale;                    // c
  float scale_log2;               // c * log2(e) (FP8: times q_descale * k_descale)
  float o_scale;                  // factor on O: 1, or v_descale for FP8 inputs
  void* o;                        // [B,H,N,d]
  float* lse;                     // [B,H,N]
  int64_t stride_b, stride_h, stride_n;            // q, o
  int64_t kv_stride_b, kv_stride_h, kv_stride_n;   // k, v
  int* status;                    // workspace status words
  int* sched;                     // workspace scheduler words: next unit, CTAs finished
  uint64_t timeout_ns;
  // nonzero (with head_group = 1): number the units longest key range first,
  // the sequences in descending key length (ties by index), each head's
  // query-tile pairs together (key padding, not causal, B <= kLenOrderMaxB)
  int len_order;
  int stall;                      // kStallFwdSoftmax: softmax warp 0 withholds its first P-ready arrive
  // split pairs (too few query-tile pairs to fill the GPU): each pair's key
  // tiles are cut into `splits` pieces whose normalised O (fp32) and
  // logsumexp go to the workspace, then merged into o, lse; 1 = unsplit
  int splits;
  int part_rows;                  // rows per (b, h) in the partial arrays: pairs x 256
  float* part_o;                  // [splits][B*H][part_rows][d]
  float* part_l;                  // [splits][B*H][part_rows]
};

// Largest batch whose sequences the forward orders by key length (one warp
// ranks them at the start of the kernel, a lane per sequence).
constexpr int kLenOrderMaxB = 32;

struct BwdArgs {
  MaskArgs m;
  int d;
  float scale;
  float scale_log2;
  const float* lse;               // [B,H,N] from the forward (read by the preprocess)
  float* lse2;                    // workspace [B*H][npad]: -L * log2(e); -inf where the
                                  // row contributes nothing (padding rows, empty rows)
  float* dsum;                    // workspace [B*H][npad]: -rowsum(dO * O); 0 on padding
  int npad;                       // nb * 128
  float* dq_acc;                  // [B,H,N,d] fp32, zeroed by the preprocess
  void* dk;                       // [B,H_kv,N,d]
  void* dv;
  int64_t stride_b, stride_h, stride_n;            // q, o, dO, dQ
  int64_t kv_stride_b, kv_stride_h, kv_stride_n;   // k, v, dK, dV
  int* status;
  int* sched;                     // workspace scheduler words: next unit, CTAs finished
  uint64_t timeout_ns;
  int stall;                      // kStallBwdCompute: compute warp 0 withholds its first P-ready arrive
  // split key tiles (too few key tiles to fill the GPU): each key tile's
  // query tiles are cut into `splits` pieces whose dK, dV sums (fp32, dK
  // unscaled) go to the workspace, then added into dk, dv; 1 = unsplit
  int splits;
  int part_rows;                  // rows per (b, key/value head) in the partials: nb x 128
  float* part_dk;                 // [splits][B*H_kv][part_rows][d]
  float* part_dv;
};

// Decode step: query rows per CTA (the key/value group's heads x n_q) at most.
constexpr int kDecMaxRows = 64;
// Up to kDecMmaRows rows the warp-MMA kernel runs, on tiles of kDecMmaKeys
// keys (its k, v tensor maps have boxes of that many rows); above it the FMA
// kernel, on 64-key tiles.
constexpr int kDecMmaRows = 16;
constexpr int kDecMmaKeys = 32;

struct DecodeArgs {
  MaskArgs m;                     // N = cache capacity, key_lens = cache lengths
  int d;
  int n_q;                        // query rows per sequence (the newest positions)
  int rows;                       // kv_group * n_q: query rows of one CTA
  int chunk;                      // cache keys per split (multiple of 64)
  int splits;                     // ceil(N / chunk)
  float scale_log2;
  const __nv_bfloat16* q;         // [B, H, n_q, d] with the strides below
  int64_t stride_b, stride_h, stride_n;   // q and o
  float* part_o;                  // workspace [splits][B*H*n_q][d]
  float* part_l;                  // workspace [splits][B*H*n_q]
  int* status;
  uint64_t timeout_ns;
};

// Tensor maps: 4-D {d, N, H, B}, 64-element x 128-row boxes, 128-byte swizzle.
struct TensorMaps {
  CUtensorMap q, k, v, o, dout, dq_acc;
};

// Launchers (return the cudaGetLastError() of their launches).
cudaError_t launch_fwd_bf16(const TensorMaps& tm, const FwdArgs& a, cudaStream_t s);
// E4M3 forward (d = 128, no dropout); tm.v maps V^T [B, H_kv, d, N] with
// 128 x 128-byte boxes, written by launch_fp8_transpose_v.
cudaError_t launch_fwd_fp8(const TensorMaps& tm, const FwdArgs& a, cudaStream_t s);
cudaError_t launch_fp8_transpose_v(const uint8_t* v, int64_t sb, int64_t sh, int64_t sn, int B,
                                   int H_kv, int N, int d, int npad, uint8_t* vt, cudaStream_t s);
// fp32 inputs on the tensor cores (kind::tf32): the split kernel writes the
// TF32 hi and lo parts of q, k and the TF32 V^T into the workspace, the
// forward reads them through these maps (fp32, 32-column x 128-row boxes;
// V^T: 32-key x d-row boxes, 128-byte swizzle).
struct Tf32Maps {
  CUtensorMap qhi, qlo, khi, klo, vt;
};
struct Tf32Buffers {
  float *qhi, *qlo;               // [B*H][N][d]
  float *khi, *klo;               // [B*H_kv][N][d]
  float* vt;                      // [B*H_kv][d][npad]
  int npad;                       // keys per V^T row: N rounded up to 128
};
cudaError_t launch_tf32_split(const float* q, const float* k, const float* v, const FwdArgs& a,
                              const Tf32Buffers& buf, cudaStream_t s);
cudaError_t launch_fwd_tf32(const Tf32Maps& tm, const FwdArgs& a, cudaStream_t s);
cudaError_t launch_compact_mask(const uint8_t* mask, int64_t head_stride, int masks, int nb,
                                int by_column, int32_t* cnt, uint16_t* idx, cudaStream_t s);
cudaError_t launch_bwd_preprocess(const void* o, const void* dout, const BwdArgs& a,
                                  cudaStream_t s);
cudaError_t launch_bwd_bf16(const TensorMaps& tm, const BwdArgs& a, cudaStream_t s);
cudaError_t launch_dq_convert(void* dq, const BwdArgs& a, cudaStream_t s);
// k, v maps with boxes of kDecMmaKeys rows (rows <= kDecMmaRows) or 64 rows
cudaError_t launch_decode(const TensorMaps& tm, void* o, float* lse, const DecodeArgs& a,
                          cudaStream_t s);

// Records `msg` as the calling thread's last error (what attn_last_error()
// returns) and passes `status` through.
int record_error(int status, const char* msg);

// Device address of attn_bwd_noalloc's built-in scratch on the current
// device (looked up once per device); an attn_status.
int builtin_scratch(void** out);

}  // namespace attn
