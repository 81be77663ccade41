// Decode step: the newest n_q query positions of each sequence against its
// key/value cache, split over the cache and merged by the incremental-softmax
// rule.
//
// What it computes (the definition of "3.3 Hiểu sâu cơ chế Self-Attention",
// §3-§4, with the causal mask of §10.2 aligned to the end of the cache):
// query row t of sequence b sits at position len_b - n_q + t and attends the
// cached keys j < len_b (j <= its position when causal); O = softmax(c q K^T) V
// and L = logsumexp of the scaled scores.
//
// The step reads the whole cache once and does little arithmetic per byte
// (2 * rows multiply-adds per key element), so it is bound by HBM bandwidth,
// not by tensor throughput; what matters is issuing few instructions per
// byte.  To keep every SM streaming, each (b, key/value head) is split into
// chunks of the cache, one CTA each; a CTA stacks the query rows of the
// head's whole group (grouped heads share the cache, "3.3 ...", §9.3) so
// every key is read once.  Up to 16 rows use warp-level bf16 MMAs
// (decode_mma_kernel); more rows (up to 64) the FMA kernel decode_kernel.  Each
// CTA leaves a partial (O_s, L_s) normalised over its chunk; the merge kernel
// combines them with the statistics update of the FlashAttention paper
// summary ("Theo dõi Softmax tăng dần"): for a score row split into parts,
// m = max(m_1, m_2), l = e^(m_1 - m) l_1 + e^(m_2 - m) l_2, which in logsumexp
// form is L = log sum_s e^(L_s) and O = sum_s e^(L_s - L) O_s.
#include <cuda_bf16.h>

#include "attn_kernels.cuh"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr int kDecKeys = 64;      // keys per tile
constexpr int kDecStages = 2;     // K and V tiles in flight per CTA (three CTAs fit an SM)
constexpr int kDecThreads = 256;
constexpr float kLn2 = 0.693147180559945309f;

template <int D>
struct DecCfg {
  static constexpr int kBoxes = D / 64;                 // 64-column TMA boxes per tile
  static constexpr int kBoxBytes = kDecKeys * 128;      // 64 rows x 128 bytes
  static constexpr int kTileBytes = kDecKeys * D * 2;
  static constexpr int kRingBytes = 2 * kDecStages * kTileBytes;   // K and V
  // query rows (fp32) and scores/probabilities of one tile (fp32)
  static size_t smem(int rows) {
    return 1024 + kRingBytes + static_cast<size_t>(rows) * D * 4 +
           static_cast<size_t>(rows) * kDecKeys * 4;
  }
  // P V: thread t owns the column pair 2 (t % (D/2)) of rows t / (D/2) + kRowGroups i
  static constexpr int kRowGroups = kDecThreads / (D / 2);
};

// bf16 pair -> packed fp32 pair (exact: a bf16 is the top half of an fp32)
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t v) {
  return f2_pack(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

__device__ __forceinline__ uint64_t pack_u2(uint32_t lo, uint32_t hi) {
  return f2_pack(__uint_as_float(lo), __uint_as_float(hi));
}

struct DecodeShared {
  uint64_t kfull[kDecStages], vfull[kDecStages];
  float m[kDecMaxRows];         // running max of the scaled scores (log2 units)
  float l[kDecMaxRows];         // running sum of exponentials
  float alpha[kDecMaxRows];     // rescale of the accumulators for the current tile
  int abort_flag;
};

// More than 16 query rows per CTA (up to 64).  MAXR: a bound on the CTA's
// query rows (32 or 64), so that the accumulator loops cover only rows that
// can exist.
template <int D, int MAXR>
__global__ void __launch_bounds__(kDecThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                  const DecodeArgs a) {
  using C = DecCfg<D>;
  constexpr int kAcc = (MAXR + C::kRowGroups - 1) / C::kRowGroups;   // row pairs per thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + kDecStages * C::kTileBytes;
  float* sQ = reinterpret_cast<float*>(sV + kDecStages * C::kTileBytes);   // [rows][D]
  float* sP = sQ + a.rows * D;                                               // [rows][64]
  __shared__ DecodeShared sh;

  const int t = threadIdx.x;
  const MaskArgs& m = a.m;
  const int split = blockIdx.x;
  const int bhk = blockIdx.y;
  const int b = bhk / m.H_kv, hk = bhk - b * m.H_kv;
  const int R = a.rows;                       // kv_group * n_q query rows
  const int len = min(max(m.key_lens[b], 0), m.N);
  const int k_begin = split * a.chunk;
  const int k_end = min(len, k_begin + a.chunk);
  const int ntiles = k_end > k_begin ? (k_end - k_begin + kDecKeys - 1) / kDecKeys : 0;

  // thread 0: K or V of tile `tile` of this chunk into its stage.  K is
  // refilled as soon as the scores of the tile before have been formed, V once
  // its P V products are done, so each buffer is reloaded at the earliest.
  auto issue = [&](bool value, int tile) {
    const int s = tile % kDecStages;
    const int k0 = k_begin + tile * kDecKeys;
    uint64_t* bar = value ? &sh.vfull[s] : &sh.kfull[s];
    uint8_t* dst = (value ? sV : sK) + s * C::kTileBytes;
    mbar_arrive_expect_tx(bar, C::kTileBytes);
#pragma unroll
    for (int x = 0; x < C::kBoxes; ++x)
      tma_load_4d(dst + x * C::kBoxBytes, value ? &tv : &tk, bar, x * 64, k0, hk, b);
  };
  // the first copies go out before anything else, so their latency overlaps
  // the set-up below
  int k_issued = 0, v_issued = 0;   // tiles whose K / V copies thread 0 has issued
  if (t == 0) {
    sh.abort_flag = 0;
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(&sh.kfull[s], 1);
      mbar_init(&sh.vfull[s], 1);
    }
    fence_mbar_init();
    for (; k_issued < kDecStages && k_issued < ntiles; ++k_issued) {
      issue(false, k_issued);
      issue(true, k_issued);
    }
    v_issued = k_issued;
  }
  for (int r = t; r < R; r += kDecThreads) {
    sh.m[r] = -INFINITY;
    sh.l[r] = 0.f;
  }
  // the group's query rows r = local head * n_q + query index, fp32
  for (int e = t; e < R * D; e += kDecThreads) {
    const int r = e / D, c = e - r * D;
    const int h = hk * m.kv_group + r / a.n_q, qt = r % a.n_q;
    sQ[e] = __bfloat162float(a.q[b * a.stride_b + h * a.stride_h +
                                 static_cast<int64_t>(qt) * a.stride_n + c]);
  }
  __syncthreads();
  const WaitCtx wc{&sh.abort_flag, a.status, a.timeout_ns};

  // P V accumulators of the column pair (col, col + 1): the threads of a
  // column pair split the rows (rg, rg + kRowGroups, ...) and take every key.
  const int col = 2 * (t % (D / 2)), rg = t / (D / 2);
  uint64_t acc[kAcc];
#pragma unroll
  for (int i = 0; i < kAcc; ++i) acc[i] = f2_pack(0.f, 0.f);
  // byte offset of this thread's column pair in a swizzled tile row j, per j mod 8
  int voff[8];
#pragma unroll
  for (int jj = 0; jj < 8; ++jj)
    voff[jj] = (col >> 6) * C::kBoxBytes + ((((col & 63) >> 3) ^ jj) << 4) + (col & 7) * 2;
  const float c2 = a.scale_log2;
  bool ok = true;

  for (int tile = 0; tile < ntiles; ++tile) {
    const int s = tile % kDecStages;
    ok = __syncthreads_and(mbar_wait(&sh.kfull[s], (tile / kDecStages) & 1, wc, kSiteDecode));
    if (!ok) break;
    const uint8_t* tK = sK + s * C::kTileBytes;
    const uint8_t* tV = sV + s * C::kTileBytes;
    const int k0 = k_begin + tile * kDecKeys;
    // scores: lanes 2u, 2u + 1 of a row slot hold the two column halves of
    // keys u and u + 32 (packed fp32x2 products), summed with one shuffle;
    // a Q chunk loaded once serves both keys
    {
      const int u = t & (kDecKeys - 1), slot = t >> 6;
      const int ch = u & 1, jA = u >> 1, jB = jA + 32;
      const uint8_t* rowA = tK + jA * 128;
      const uint8_t* rowB = tK + jB * 128;
      const int xa = jA & 7, xb = jB & 7;
      for (int r = slot; r < R; r += kDecThreads / kDecKeys) {
        const float* qr = sQ + r * D;
        uint64_t a0 = f2_pack(0.f, 0.f), a1 = a0, b0 = a0, b1 = a0;
#pragma unroll
        for (int k8 = 0; k8 < D / 16; ++k8) {
          const int cc = ch * (D / 2) + k8 * 8;
          const int boff = (cc >> 6) * C::kBoxBytes;
          const int c8 = (cc & 63) >> 3;
          const uint4 ka = *reinterpret_cast<const uint4*>(rowA + boff + ((c8 ^ xa) << 4));
          const uint4 kb = *reinterpret_cast<const uint4*>(rowB + boff + ((c8 ^ xb) << 4));
          const uint4 qa = *reinterpret_cast<const uint4*>(qr + cc);
          const uint4 qb = *reinterpret_cast<const uint4*>(qr + cc + 4);
          const uint64_t q0 = pack_u2(qa.x, qa.y), q1 = pack_u2(qa.z, qa.w);
          const uint64_t q2 = pack_u2(qb.x, qb.y), q3 = pack_u2(qb.z, qb.w);
          a0 = f2_fma(bf16x2_to_f2(ka.x), q0, a0);
          a1 = f2_fma(bf16x2_to_f2(ka.y), q1, a1);
          a0 = f2_fma(bf16x2_to_f2(ka.z), q2, a0);
          a1 = f2_fma(bf16x2_to_f2(ka.w), q3, a1);
          b0 = f2_fma(bf16x2_to_f2(kb.x), q0, b0);
          b1 = f2_fma(bf16x2_to_f2(kb.y), q1, b1);
          b0 = f2_fma(bf16x2_to_f2(kb.z), q2, b0);
          b1 = f2_fma(bf16x2_to_f2(kb.w), q3, b1);
        }
        float x0, x1, x2, x3;
        f2_unpack(f2_add(a0, a1), x0, x1);
        f2_unpack(f2_add(b0, b1), x2, x3);
        float dA = x0 + x1, dB = x2 + x3;
        dA += __shfl_xor_sync(0xffffffffu, dA, 1);
        dB += __shfl_xor_sync(0xffffffffu, dB, 1);
        const int pos = len - a.n_q + r % a.n_q;   // this query row's position
        const int j = ch ? jB : jA;
        const int kj = k0 + j;
        const bool allowed = kj < k_end && (!m.causal || kj <= pos);
        sP[r * kDecKeys + j] = allowed ? (ch ? dB : dA) * c2 : -INFINITY;
      }
    }
    __syncthreads();   // the K stage is read: refill it
    if (t == 0 && k_issued < ntiles) issue(false, k_issued++);
    // online softmax per row, one warp per row
    {
      const int w = t >> 5, lane = t & 31;
      for (int r = w; r < R; r += kDecThreads / 32) {
        float* pr = sP + r * kDecKeys;
        const float s0 = pr[lane], s1 = pr[lane + 32];
        float mx = fmaxf(s0, s1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_old = sh.m[r];
        const float m_new = fmaxf(m_old, mx);
        // m_new = -inf only when the row has seen no allowed key yet
        const float base = m_new == -INFINITY ? 0.f : m_new;
        const float p0 = exp2f(s0 - base), p1 = exp2f(s1 - base);
        pr[lane] = p0;
        pr[lane + 32] = p1;
        float sum = p0 + p1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) {
          const float al = m_old == -INFINITY ? 0.f : exp2f(m_old - base);
          sh.alpha[r] = al;
          sh.l[r] = sh.l[r] * al + sum;
          sh.m[r] = m_new;
        }
      }
    }
    ok = __syncthreads_and(mbar_wait(&sh.vfull[s], (tile / kDecStages) & 1, wc, kSiteDecode));
    if (!ok) break;
    // O += P V: per key, one 32-bit load of the thread's two V columns and a
    // packed fma per row; the swizzled offsets of the 8 row phases are fixed
    // per thread
#pragma unroll
    for (int i = 0; i < kAcc; ++i) {
      const int r = rg + i * C::kRowGroups;
      if (r < R) {
        const float al = sh.alpha[r];
        acc[i] = f2_mul(acc[i], f2_pack(al, al));
      }
    }
#pragma unroll 2
    for (int j8 = 0; j8 < kDecKeys; j8 += 8) {
      uint64_t v2[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        v2[jj] = bf16x2_to_f2(*reinterpret_cast<const uint32_t*>(tV + (j8 + jj) * 128 + voff[jj]));
#pragma unroll
      for (int i = 0; i < kAcc; ++i) {
        const int r = rg + i * C::kRowGroups;
        if (r < R) {
          const float4 pa = *reinterpret_cast<const float4*>(sP + r * kDecKeys + j8);
          const float4 pb = *reinterpret_cast<const float4*>(sP + r * kDecKeys + j8 + 4);
          acc[i] = f2_fma(f2_pack(pa.x, pa.x), v2[0], acc[i]);
          acc[i] = f2_fma(f2_pack(pa.y, pa.y), v2[1], acc[i]);
          acc[i] = f2_fma(f2_pack(pa.z, pa.z), v2[2], acc[i]);
          acc[i] = f2_fma(f2_pack(pa.w, pa.w), v2[3], acc[i]);
          acc[i] = f2_fma(f2_pack(pb.x, pb.x), v2[4], acc[i]);
          acc[i] = f2_fma(f2_pack(pb.y, pb.y), v2[5], acc[i]);
          acc[i] = f2_fma(f2_pack(pb.z, pb.z), v2[6], acc[i]);
          acc[i] = f2_fma(f2_pack(pb.w, pb.w), v2[7], acc[i]);
        }
      }
    }
    __syncthreads();   // the stage and the scores are free
    if (t == 0 && v_issued < ntiles) issue(true, v_issued++);
  }

  if (!ok && t == 0) {   // let issued copies land before the ring is reused or the CTA exits
    for (int tile = max(0, k_issued - kDecStages); tile < k_issued; ++tile)
      mbar_wait_drain(&sh.kfull[tile % kDecStages], (tile / kDecStages) & 1, a.timeout_ns);
    for (int tile = max(0, v_issued - kDecStages); tile < v_issued; ++tile)
      mbar_wait_drain(&sh.vfull[tile % kDecStages], (tile / kDecStages) & 1, a.timeout_ns);
  }
  // partial O normalised over this chunk, and its logsumexp (natural log)
  const int64_t rows_total = static_cast<int64_t>(m.B) * m.H * a.n_q;
  auto write_row = [&](int r, int cc, float o0, float o1) {
    const int h = hk * m.kv_group + r / a.n_q, qt = r % a.n_q;
    const int64_t row = (static_cast<int64_t>(b) * m.H + h) * a.n_q + qt;
    const float l = ok ? sh.l[r] : 0.f;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    *reinterpret_cast<float2*>(&a.part_o[(split * rows_total + row) * D + cc]) =
        make_float2(o0 * inv, o1 * inv);
    if (cc == 0)
      a.part_l[split * rows_total + row] = l > 0.f ? (sh.m[r] + __log2f(l)) * kLn2 : -INFINITY;
  };
#pragma unroll
  for (int i = 0; i < kAcc; ++i) {
    const int r = rg + i * C::kRowGroups;
    if (r >= R) continue;
    float o0, o1;
    f2_unpack(acc[i], o0, o1);
    write_row(r, col, o0, o1);
  }
}

// ----------------------------------------------------------------------------
// Few query rows (the group's rows <= 16): warp-level tensor-core MMAs.
//
// The FMA kernel above spends about a dozen instructions per cached element,
// which leaves it far from the bandwidth bound.  Here the two contractions
// of a tile, S = Q K^T and O += P V, are 16 x 8 x 16 bf16 warp MMAs
// (mma.sync; the rows are padded to 16, the tensor work is irrelevant next
// to the bytes), so a 64-key tile of K and V (32 KB at d = 128) costs its
// warp about 300 instructions, where the FMA kernel issues some 6000 warp
// instructions for the same 32 KB.  Warp w takes the chunk's tiles w, w + kMmaWarps, ... and
// streams them itself: its lane 0 issues the TMA copies into the warp's own
// kStagesPerWarp stages and refills a stage as soon as the warp has read
// it, so no stage is shared between warps and every wait is on the warp's
// own previous copy.  Each warp keeps its own online-softmax state (max m,
// sum l, O in registers); the states are merged through shared memory at the
// end with the same rule as the split merge.
//
// Fragment layouts of mma.m16n8k16 (thread t = 4 g + q, g = t / 4, q = t % 4):
//   A (16 x 16): a0 = (row g, cols 2q, 2q+1), a1 = (row g+8, same),
//                a2 = (row g, cols 2q+8, 2q+9), a3 = (row g+8, same)
//   B (16 x 8):  b0 = (k 2q, 2q+1; n g), b1 = (k 2q+8, 2q+9; n g)
//   C (16 x 8):  c0, c1 = (row g, cols 2q, 2q+1), c2, c3 = (row g+8, same)
// ldmatrix delivers an 8 x 8 block as (row g, cols 2q, 2q+1) per thread,
// or transposed with .trans; the C fragment of the scores is the A fragment
// of P for the second product.

constexpr int kMmaWarps = 3;
constexpr int kMmaThreads = 32 * kMmaWarps;
constexpr int kMmaRows = kDecMmaRows;
constexpr int kMaxStagesPerWarp = 4;

// Tiles of kDecMmaKeys keys, two (d = 128) or four (d = 64) stages per warp:
// 96 KB of ring, two CTAs per SM, and each warp reads one tile while its
// next copy is in flight.
template <int D>
struct DecMmaCfg {
  static constexpr int kKeys = kDecMmaKeys;
  static constexpr int kBoxes = D / 64;
  static constexpr int kBoxBytes = kKeys * 128;           // kKeys rows x 128 bytes
  static constexpr int kTileBytes = kKeys * D * 2;
  static constexpr int kStagesPerWarp = D == 128 ? 2 : 4;
  static_assert(kStagesPerWarp <= kMaxStagesPerWarp, "barrier array");
  static constexpr int kStages = kMmaWarps * kStagesPerWarp;
  static constexpr int kRingBytes = 2 * kStages * kTileBytes;
  static constexpr int kSmem = 1024 + kRingBytes;
  static_assert(kMmaWarps * kMmaRows * D * 4 <= kRingBytes, "merge scratch fits the ring");
};

struct DecMmaShared {
  uint64_t full[kMaxStagesPerWarp * kMmaWarps];
  float m[kMmaWarps][kMmaRows], l[kMmaWarps][kMmaRows];
  int abort_flag;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// c += a b, 16 x 8 x 16, bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma_16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of the 16-byte chunk holding elements [col, col + 8) of row
// `key` in a 64-key tile stored as 64-column boxes with the 128-byte swizzle.
template <int D>
__device__ __forceinline__ uint32_t tile_off(int key, int col) {
  return static_cast<uint32_t>((col >> 6) * DecMmaCfg<D>::kBoxBytes + key * 128 +
                               ((((col & 63) >> 3) ^ (key & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kMmaThreads, 2)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                      const DecodeArgs a) {
  using C = DecMmaCfg<D>;
  constexpr int ST = C::kStages;
  constexpr int NT = D / 8;       // 8-column tiles of O
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ DecMmaShared sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const MaskArgs& m = a.m;
  const int split = blockIdx.x;
  const int bhk = blockIdx.y;
  const int b = bhk / m.H_kv, hk = bhk - b * m.H_kv;
  const int R = a.rows;
  const int len = min(max(m.key_lens[b], 0), m.N);
  const int k_begin = split * a.chunk;
  const int k_end = min(len, k_begin + a.chunk);
  constexpr int KT = C::kKeys;
  const int ntiles = k_end > k_begin ? (k_end - k_begin + KT - 1) / KT : 0;
  auto sK = [&](int s) { return smem + s * 2 * C::kTileBytes; };
  auto sV = [&](int s) { return smem + s * 2 * C::kTileBytes + C::kTileBytes; };

  if (threadIdx.x == 0) {
    sh.abort_flag = 0;
    for (int s = 0; s < ST; ++s) mbar_init(&sh.full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{&sh.abort_flag, a.status, a.timeout_ns};
  constexpr int SPW = C::kStagesPerWarp;
  // this warp's tiles: warp + kMmaWarps * u, u = 0, 1, ...; tile u sits in
  // stage warp * SPW + u % SPW
  const int my_tiles = ntiles > warp ? (ntiles - warp + kMmaWarps - 1) / kMmaWarps : 0;
  auto issue = [&](int u) {   // lane 0: K and V of the warp's tile u
    const int st = warp * SPW + u % SPW;
    const int k0 = k_begin + (warp + kMmaWarps * u) * KT;
    mbar_arrive_expect_tx(&sh.full[st], 2 * C::kTileBytes);
#pragma unroll
    for (int x = 0; x < C::kBoxes; ++x) {
      tma_load_4d(sK(st) + x * C::kBoxBytes, &tk, &sh.full[st], x * 64, k0, hk, b);
      tma_load_4d(sV(st) + x * C::kBoxBytes, &tv, &sh.full[st], x * 64, k0, hk, b);
    }
  };
  int issued = 0;
  if (lane == 0)
    for (; issued < SPW && issued < my_tiles; ++issued) issue(issued);

  // --------------------------------------------------------------- consumers
  const int g = lane >> 2, q = lane & 3;
  const int rows[2] = {g, g + 8};
  // Q fragments of rows g and g + 8 (zero past the group's rows)
  uint32_t qa[D / 16][4];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = rows[i];
    const __nv_bfloat16* qr = nullptr;
    if (r < R) {
      const int h = hk * m.kv_group + r / a.n_q, qt = r % a.n_q;
      qr = a.q + b * a.stride_b + h * a.stride_h + static_cast<int64_t>(qt) * a.stride_n;
    }
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][i] = qr ? *reinterpret_cast<const uint32_t*>(qr + kk * 16 + 2 * q) : 0u;
      qa[kk][i + 2] = qr ? *reinterpret_cast<const uint32_t*>(qr + kk * 16 + 8 + 2 * q) : 0u;
    }
  }
  int pos[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) pos[i] = len - a.n_q + rows[i] % a.n_q;
  const bool live[2] = {rows[0] < R, rows[1] < R};
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  const float c2 = a.scale_log2;
  // ldmatrix row address of this lane: block (lane / 8), row (lane % 8)
  const int lb = lane >> 3, lr = lane & 7;
  bool ok = true;

  for (int u = 0; u < my_tiles; ++u) {
    const int tile = warp + kMmaWarps * u;
    const int s = warp * SPW + u % SPW;
    if (!(ok = __all_sync(0xffffffffu, mbar_wait(&sh.full[s], (u / SPW) & 1, wc, kSiteDecode))))
      break;
    const uint32_t kb = smem_u32(sK(s)), vb = smem_u32(sV(s));
    const int k0 = k_begin + tile * KT;
    // S = Q K^T: KT/8 key blocks of 8; per 16 columns of d, one ldmatrix.x4
    // gives the B fragments of two key blocks
    float sc[KT / 8][4];
#pragma unroll
    for (int n = 0; n < KT / 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
      for (int n = 0; n < KT / 8; n += 2) {
        // blocks: (keys 8n, d 16kk), (8n, 16kk+8), (8n+8, 16kk), (8n+8, 16kk+8)
        const int key = 8 * n + 8 * (lb >> 1) + lr, col = 16 * kk + 8 * (lb & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + tile_off<D>(key, col), b0, b1, b2, b3);
        mma_16816(sc[n], qa[kk], b0, b1);
        mma_16816(sc[n + 1], qa[kk], b2, b3);
      }
    // mask, scale to log2 units, running max
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < KT / 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = e >> 1;
        const int kj = k0 + 8 * n + 2 * q + (e & 1);
        const bool allowed = live[i] && kj < k_end && (!m.causal || kj <= pos[i]);
        sc[n][e] = allowed ? sc[n][e] * c2 : -INFINITY;
        tmax[i] = fmaxf(tmax[i], sc[n][e]);
      }
    float alpha[2], base[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 1));
      tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 2));
      const float mn = fmaxf(mrow[i], tmax[i]);
      base[i] = mn == -INFINITY ? 0.f : mn;   // -inf: no allowed key seen yet
      alpha[i] = mrow[i] == -INFINITY ? 0.f : exp2f(mrow[i] - base[i]);
      mrow[i] = mn;
    }
    // P = 2^(S - m) as bf16 A fragments; row sums from the same fp32 values
    uint32_t pa[KT / 16][4];
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int n = 0; n < KT / 8; ++n) {
      const float p0 = exp2f(sc[n][0] - base[0]), p1 = exp2f(sc[n][1] - base[0]);
      const float p2 = exp2f(sc[n][2] - base[1]), p3 = exp2f(sc[n][3] - base[1]);
      psum[0] += p0 + p1;
      psum[1] += p2 + p3;
      // keys 16 kp .. 16 kp + 15: block 2 kp -> a0 / a1, block 2 kp + 1 -> a2 / a3
      pa[n >> 1][(n & 1) * 2] = pack_bf16x2(p0, p1);
      pa[n >> 1][(n & 1) * 2 + 1] = pack_bf16x2(p2, p3);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) lrow[i] = lrow[i] * alpha[i] + psum[i];
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][0] *= alpha[0];
        o[n][1] *= alpha[0];
        o[n][2] *= alpha[1];
        o[n][3] *= alpha[1];
      }
    }
    // O += P V: per 16 keys and 16 columns of d, one ldmatrix.x4.trans gives
    // the B fragments of two 8-column tiles
#pragma unroll
    for (int kp = 0; kp < KT / 16; ++kp)
#pragma unroll
      for (int n = 0; n < NT; n += 2) {
        // blocks: (keys 16kp, d 8n), (16kp+8, 8n), (16kp, 8n+8), (16kp+8, 8n+8)
        const int key = 16 * kp + 8 * (lb & 1) + lr, col = 8 * n + 8 * (lb >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + tile_off<D>(key, col), b0, b1, b2, b3);
        mma_16816(o[n], pa[kp], b0, b1);
        mma_16816(o[n + 1], pa[kp], b2, b3);
      }
    // the warp has read the stage: refill it with its tile u + SPW
    __syncwarp();
    if (lane == 0 && issued < my_tiles) {
      fence_proxy_async_smem();
      issue(issued++);
    }
  }
  if (lane == 0 && !ok)   // let issued copies land before the ring is reused or the CTA exits
    for (int u = max(0, issued - SPW); u < issued; ++u)   // each stage's last copy
      mbar_wait_drain(&sh.full[warp * SPW + u % SPW], (u / SPW) & 1, a.timeout_ns);

  // merge the four warps' states: m, l per row, then O through shared memory
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    lrow[i] += __shfl_xor_sync(0xffffffffu, lrow[i], 1);
    lrow[i] += __shfl_xor_sync(0xffffffffu, lrow[i], 2);
  }
  if (q == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      sh.m[warp][rows[i]] = mrow[i];
      sh.l[warp][rows[i]] = lrow[i];
    }
  }
  __syncthreads();   // every warp is done with the ring
  float scale[2], ltot[2], mtot[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) mx = fmaxf(mx, sh.m[w][rows[i]]);
    float lt = 0.f;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) {
      const float mw = sh.m[w][rows[i]];
      lt += mw == -INFINITY ? 0.f : sh.l[w][rows[i]] * exp2f(mw - mx);
    }
    mtot[i] = mx;
    ltot[i] = lt;
    // this warp's weight, with the final 1 / l folded in
    scale[i] = (mrow[i] == -INFINITY || !(lt > 0.f)) ? 0.f : exp2f(mrow[i] - mx) / lt;
  }
  float* red = reinterpret_cast<float*>(smem);   // [warp][16 rows][D]
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int col = 8 * n + 2 * q;
    *reinterpret_cast<float2*>(&red[(warp * kMmaRows + g) * D + col]) =
        make_float2(o[n][0] * scale[0], o[n][1] * scale[0]);
    *reinterpret_cast<float2*>(&red[(warp * kMmaRows + g + 8) * D + col]) =
        make_float2(o[n][2] * scale[1], o[n][3] * scale[1]);
  }
  __syncthreads();
  const int64_t rows_total = static_cast<int64_t>(m.B) * m.H * a.n_q;
  for (int e = threadIdx.x; e < R * (D / 2); e += 32 * kMmaWarps) {
    const int r = e / (D / 2), cc = 2 * (e - r * (D / 2));
    float o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) {
      const float2 v = *reinterpret_cast<const float2*>(&red[(w * kMmaRows + r) * D + cc]);
      o0 += v.x;
      o1 += v.y;
    }
    const int h = hk * m.kv_group + r / a.n_q, qt = r % a.n_q;
    const int64_t row = (static_cast<int64_t>(b) * m.H + h) * a.n_q + qt;
    *reinterpret_cast<float2*>(&a.part_o[(split * rows_total + row) * D + cc]) =
        ok ? make_float2(o0, o1) : make_float2(0.f, 0.f);
  }
  // logsumexp of the chunk (natural log): rows g, g + 8 by lanes with q == 0 of warp 0
  if (warp == 0 && q == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = rows[i];
      if (r >= R) continue;
      const int h = hk * m.kv_group + r / a.n_q, qt = r % a.n_q;
      const int64_t row = (static_cast<int64_t>(b) * m.H + h) * a.n_q + qt;
      a.part_l[split * rows_total + row] =
          (ok && ltot[i] > 0.f) ? (mtot[i] + __log2f(ltot[i])) * kLn2 : -INFINITY;
    }
  }
}

// Merge of the splits: L = log sum_s e^(L_s), O = sum_s e^(L_s - L) O_s.
// One CTA of D threads per query row.
template <int D>
__global__ void __launch_bounds__(128)
    decode_merge_kernel(__nv_bfloat16* o, float* lse, const DecodeArgs a) {
  const int64_t row = blockIdx.x;
  const int c = threadIdx.x;
  const MaskArgs& m = a.m;
  const int64_t rows_total = static_cast<int64_t>(m.B) * m.H * a.n_q;
  const int qt = static_cast<int>(row % a.n_q);
  const int64_t bh = row / a.n_q;
  const int b = static_cast<int>(bh / m.H), h = static_cast<int>(bh % m.H);
  float lmax = -INFINITY;
  for (int s = 0; s < a.splits; ++s) lmax = fmaxf(lmax, a.part_l[s * rows_total + row]);
  float L = -INFINITY, out = 0.f;
  if (lmax > -INFINITY) {
    float wsum = 0.f, acc = 0.f;
    for (int s = 0; s < a.splits; ++s) {
      const float ls = a.part_l[s * rows_total + row];
      const float w = ls == -INFINITY ? 0.f : __expf(ls - lmax);
      wsum += w;
      if (c < D) acc = fmaf(w, a.part_o[(s * rows_total + row) * D + c], acc);
    }
    L = lmax + __logf(wsum);
    out = acc / wsum;
  }
  if (c < D)
    o[b * a.stride_b + h * a.stride_h + static_cast<int64_t>(qt) * a.stride_n + c] =
        __float2bfloat16_rn(out);
  if (c == 0) lse[row] = L;
}

template <int D, int MAXR>
cudaError_t launch_rows(const TensorMaps& tm, const DecodeArgs& a, cudaStream_t s) {
  using C = DecCfg<D>;
  const size_t smem = C::smem(MAXR);
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, MAXR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(a.splits), static_cast<unsigned>(a.m.B * a.m.H_kv));
  decode_kernel<D, MAXR><<<grid, kDecThreads, smem, s>>>(tm.k, tm.v, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_mma(const TensorMaps& tm, const DecodeArgs& a, cudaStream_t s) {
  using C = DecMmaCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(a.splits), static_cast<unsigned>(a.m.B * a.m.H_kv));
  decode_mma_kernel<D><<<grid, kMmaThreads, C::kSmem, s>>>(tm.k, tm.v, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const TensorMaps& tm, void* o, float* lse, const DecodeArgs& a,
                     cudaStream_t s) {
  cudaError_t e;
  if (a.rows <= kMmaRows) e = launch_mma<D>(tm, a, s);
  else if (a.rows <= 32) e = launch_rows<D, 32>(tm, a, s);
  else e = launch_rows<D, kDecMaxRows>(tm, a, s);
  if (e != cudaSuccess) return e;
  const unsigned rows = static_cast<unsigned>(static_cast<int64_t>(a.m.B) * a.m.H * a.n_q);
  decode_merge_kernel<D><<<rows, 128, 0, s>>>(static_cast<__nv_bfloat16*>(o), lse, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const TensorMaps& tm, void* o, float* lse, const DecodeArgs& a,
                          cudaStream_t s) {
  return a.d == 64 ? launch_d<64>(tm, o, lse, a, s) : launch_d<128>(tm, o, lse, a, s);
}

}  // namespace attn
