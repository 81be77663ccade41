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
// not by the tensor cores: plain FMA arithmetic is enough.  To keep every SM
// streaming, each (b, key/value head) is split into chunks of the cache, one
// CTA each; a CTA stacks the query rows of the head's whole group (grouped
// heads share the cache, "3.3 ...", §9.3) so every key is read once.  Each
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

// MAXR: a bound on the CTA's query rows (4, 8, 16, 32 or 64), so that the
// accumulator loops cover only rows that can exist.
template <int D, int MAXR>
__global__ void __launch_bounds__(kDecThreads, MAXR <= 16 ? 3 : 2)
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

  // P V accumulators of the column pair (col, col + 1).  Few rows (<= 8):
  // the threads of a column pair split each tile's keys into kParts parts and
  // keep every row, so a V element loaded once serves all rows; the parts are
  // summed at the end.  Many rows: the threads split the rows (rg, rg +
  // kRowGroups, ...) and take every key.
  constexpr bool kKeySplit = MAXR <= 8;
  constexpr int kParts = kDecThreads / (D / 2);
  constexpr int kNAcc = kKeySplit ? MAXR : kAcc;
  const int col = 2 * (t % (D / 2)), rg = t / (D / 2);
  uint64_t acc[kNAcc];
#pragma unroll
  for (int i = 0; i < kNAcc; ++i) acc[i] = f2_pack(0.f, 0.f);
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
    if constexpr (kKeySplit) {
#pragma unroll
      for (int r = 0; r < MAXR; ++r)
        if (r < R) {
          const float al = sh.alpha[r];
          acc[r] = f2_mul(acc[r], f2_pack(al, al));
        }
      constexpr int kPer = kDecKeys / kParts;   // keys of this thread's part (8 or 16)
      const int j0 = rg * kPer;                  // rg is the key part here
#pragma unroll
      for (int j4 = 0; j4 < kPer; j4 += 4) {
        uint64_t v2[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = j0 + j4 + jj;
          v2[jj] = bf16x2_to_f2(*reinterpret_cast<const uint32_t*>(tV + j * 128 + voff[(j4 + jj) & 7]));
        }
#pragma unroll
        for (int r = 0; r < MAXR; ++r)
          if (r < R) {
            const float4 pv = *reinterpret_cast<const float4*>(sP + r * kDecKeys + j0 + j4);
            acc[r] = f2_fma(f2_pack(pv.x, pv.x), v2[0], acc[r]);
            acc[r] = f2_fma(f2_pack(pv.y, pv.y), v2[1], acc[r]);
            acc[r] = f2_fma(f2_pack(pv.z, pv.z), v2[2], acc[r]);
            acc[r] = f2_fma(f2_pack(pv.w, pv.w), v2[3], acc[r]);
          }
      }
    } else {
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
  if constexpr (kKeySplit) {
    // sum the key parts through shared memory (the K/V ring is free now)
    __syncthreads();
    float* red = reinterpret_cast<float*>(sK);   // [kParts][MAXR][D]
#pragma unroll
    for (int r = 0; r < MAXR; ++r)
      if (r < R) {
        float o0, o1;
        f2_unpack(acc[r], o0, o1);
        *reinterpret_cast<float2*>(&red[(rg * MAXR + r) * D + col]) = make_float2(o0, o1);
      }
    __syncthreads();
    for (int e = t; e < R * (D / 2); e += kDecThreads) {
      const int r = e / (D / 2), cc = 2 * (e - r * (D / 2));
      float o0 = 0.f, o1 = 0.f;
#pragma unroll
      for (int k = 0; k < kParts; ++k) {
        const float2 v = *reinterpret_cast<const float2*>(&red[(k * MAXR + r) * D + cc]);
        o0 += v.x;
        o1 += v.y;
      }
      write_row(r, cc, o0, o1);
    }
  } else {
#pragma unroll
    for (int i = 0; i < kAcc; ++i) {
      const int r = rg + i * C::kRowGroups;
      if (r >= R) continue;
      float o0, o1;
      f2_unpack(acc[i], o0, o1);
      write_row(r, col, o0, o1);
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
cudaError_t launch_d(const TensorMaps& tm, void* o, float* lse, const DecodeArgs& a,
                     cudaStream_t s) {
  cudaError_t e;
  if (a.rows <= 4) e = launch_rows<D, 4>(tm, a, s);
  else if (a.rows <= 8) e = launch_rows<D, 8>(tm, a, s);
  else if (a.rows <= 16) e = launch_rows<D, 16>(tm, a, s);
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
