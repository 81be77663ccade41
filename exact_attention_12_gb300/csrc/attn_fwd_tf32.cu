// Fused attention forward for fp32 inputs and outputs on the tensor cores:
// tcgen05.mma kind::tf32, fp32 accumulation in TMEM.
//
// Method: the tiled forward of FlashAttention (paper summary, "Theo dõi
// Softmax tăng dần" and its per-block steps; "3.3 Hiểu sâu cơ chế
// Self-Attention", §12.2 Tiling and §12.3 Online Softmax): a 128-row query
// tile streams the key/value tiles it may attend past it, keeping each row's
// running max m and exp-sum l on chip; only O and L = c*m + ln l are written.
//
// Precision.  TF32 keeps 10 of fp32's 23 mantissa bits (relative rounding
// 2^-11).  The scores, which L depends on directly, are formed in three TF32
// passes (the published "3xTF32" error compensation): with x_hi = tf32(x)
// and x_lo = tf32(x - x_hi),
//   Q K^T ~= Q_hi K_hi^T + Q_hi K_lo^T + Q_lo K_hi^T,
// which leaves out only Q_lo K_lo^T (~2^-22 relative) besides the fp32
// accumulation.  P V is one TF32 pass (P and V rounded to TF32), an error of
// about 2^-10 of sum_j P_ij |V_jc| in O.
//
// A split kernel first writes Q_hi, Q_lo, K_hi, K_lo (TF32-rounded fp32,
// [.., N, d] contiguous) and V^T (TF32, [.., d, keys padded to 128]) into the
// workspace, so every MMA operand is K-major and comes straight from TMA.
//
// CTA: one 128-row query tile of one (b, h); 256 threads.
//   warp 0     TMA producer: per key tile, d in chunks of 32 columns (one
//              128-byte swizzle box, 16 KB per 128 rows): the Q_hi, Q_lo,
//              K_hi, K_lo chunks through a two-stage ring; then V^T (four
//              boxes of 32 keys x d rows).
//   warp 1     TMEM owner; lane 0 issues the MMAs: per key tile three TF32
//              products per 8-column step of d into S, then, once the
//              softmax has written P over S, O += P V^T with P from TMEM.
//   warps 4-7  softmax: thread t owns row t (TMEM lane t).  Loads its S row,
//              masks it, updates m and l (rescaling O in TMEM when m grows),
//              forms P = 2^(c log2e (S - m)), applies the dropout keep mask
//              and writes P (TF32-rounded) over S.  Epilogue O / l, L.
//   warps 2-3  idle.
// Because every tcgen05.commit covers all earlier MMAs of the issuing thread,
// "S of key tile t + 1 is complete" implies "O += P V of tile t is
// complete": the softmax may then rescale O.
// TMEM columns: S (and P over it) [0, 128), O [128, 128 + d).
#include <climits>

#include "attn_kernels.cuh"
#include "philox.cuh"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr float kLn2 = 0.693147180559945309f;
constexpr int kChunkCols = 32;                 // fp32 columns per 128-byte box row
constexpr int kChunkBytes = kTile * 128;       // one box: 128 rows x 128 bytes
constexpr int kRing = 2;                       // chunk stages

template <int D>
struct Tf32Cfg {
  static constexpr int kChunks = D / kChunkCols;
  static constexpr int kStageBytes = 4 * kChunkBytes;      // Q_hi, Q_lo, K_hi, K_lo
  static constexpr int kVtBoxBytes = D * 128;              // 32 keys x d rows
  static constexpr int kVtBytes = 4 * kVtBoxBytes;         // 128 keys
  static constexpr int kSmem = 1024 + kRing * kStageBytes + kVtBytes;
  static constexpr int kThreads = 256;
  static constexpr uint32_t kSCol = 0, kOCol = 128;
};

struct Tf32Ctl {
  uint64_t full[kRing], empty[kRing];
  uint64_t vfull, vempty, sfull, pfull, done, final_bar;
  uint32_t tmem_base;
  int abort_flag;
};

// The key tiles query tile qt of head bh visits, in ascending order: those
// below the key limit (and, causal, at or below qt) that the block mask keeps.
struct Tf32Walk {
  const MaskArgs* m;
  int qt, bh, end;
  __device__ __forceinline__ int next(int j) const {   // first visited tile >= j, or end
    if (m->block_mask == nullptr) return j;
    const uint8_t* row = m->block_mask +
                         (m->mask_per_head ? static_cast<int64_t>(bh) * m->block_mask_head_stride
                                           : 0) +
                         static_cast<int64_t>(qt) * m->nb;
    while (j < end && row[j] == 0) ++j;
    return j;
  }
};

__device__ __forceinline__ Tf32Walk tf32_walk(const MaskArgs& m, int qt, int bh, int limit) {
  int end = (limit + kTile - 1) / kTile;
  if (m.causal) end = min(end, qt + 1);
  return Tf32Walk{&m, qt, bh, end};
}

template <int D, bool DROPOUT>
__global__ void __launch_bounds__(256, 1)
    fwd_tf32_kernel(const __grid_constant__ CUtensorMap tqh, const __grid_constant__ CUtensorMap tql,
                    const __grid_constant__ CUtensorMap tkh, const __grid_constant__ CUtensorMap tkl,
                    const __grid_constant__ CUtensorMap tvt, const FwdArgs a) {
  using C = Tf32Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sRing = smem;                               // kRing x (Q_hi, Q_lo, K_hi, K_lo chunk)
  uint8_t* sVt = smem + kRing * C::kStageBytes;        // V^T: 4 boxes of 32 keys x d rows
  __shared__ Tf32Ctl ctl;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const MaskArgs& m = a.m;
  const int qt = static_cast<int>(blockIdx.x);
  const int bh = static_cast<int>(blockIdx.y);
  const int b = bh / m.H, h = bh - b * m.H;
  const int hk = h / m.kv_group;
  const int limit = m.key_lens ? min(max(m.key_lens[b], 0), m.N) : m.N;
  const int q0 = qt * kTile;
  const Tf32Walk walk = tf32_walk(m, qt, bh, limit);

  if (threadIdx.x == 0) {
    ctl.abort_flag = 0;
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], 1);
    }
    mbar_init(&ctl.vfull, 1);
    mbar_init(&ctl.vempty, 1);
    mbar_init(&ctl.sfull, 1);
    mbar_init(&ctl.pfull, 4);
    mbar_init(&ctl.done, 1);
    mbar_init(&ctl.final_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl.tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const WaitCtx wc{&ctl.abort_flag, a.status, a.timeout_ns};

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int t = 0;    // chunks issued
      int nv = 0;   // V^T tiles issued
      bool ok = true;
      for (int j = walk.next(0); ok && j < walk.end; j = walk.next(j + 1)) {
        const int k0 = j * kTile;
        for (int c = 0; c < C::kChunks; ++c, ++t) {
          const int s = t % kRing;
          if (t >= kRing && !(ok = mbar_wait(&ctl.empty[s], ((t / kRing) - 1) & 1, wc, kSiteTf32Load)))
            break;
          uint8_t* st = sRing + s * C::kStageBytes;
          mbar_arrive_expect_tx(&ctl.full[s], C::kStageBytes);
          tma_load_4d(st, &tqh, &ctl.full[s], c * kChunkCols, q0, h, b);
          tma_load_4d(st + kChunkBytes, &tql, &ctl.full[s], c * kChunkCols, q0, h, b);
          tma_load_4d(st + 2 * kChunkBytes, &tkh, &ctl.full[s], c * kChunkCols, k0, hk, b);
          tma_load_4d(st + 3 * kChunkBytes, &tkl, &ctl.full[s], c * kChunkCols, k0, hk, b);
        }
        if (!ok) break;
        if (nv >= 1 && !(ok = mbar_wait(&ctl.vempty, (nv - 1) & 1, wc, kSiteTf32Load))) break;
        mbar_arrive_expect_tx(&ctl.vfull, C::kVtBytes);
#pragma unroll
        for (int x = 0; x < 4; ++x)
          tma_load_4d(sVt + x * C::kVtBoxBytes, &tvt, &ctl.vfull, k0 + x * kChunkCols, 0, hk, b);
        ++nv;
      }
      if (ctl.abort_flag) {   // let issued copies land before the CTA exits
        for (int tt = max(0, t - kRing); tt < t; ++tt)
          mbar_wait_drain(&ctl.full[tt % kRing], (tt / kRing) & 1, a.timeout_ns);
        if (nv >= 1) mbar_wait_drain(&ctl.vfull, (nv - 1) & 1, a.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_tf32(128, 128, false, false);
      constexpr uint32_t kIdO = idesc_tf32(128, D, false, false);
      int t = 0, nv = 0;
      bool ok = true;
      for (int j = walk.next(0); ok && j < walk.end; j = walk.next(j + 1), ++nv) {
        // S = Q_hi K_hi^T + Q_hi K_lo^T + Q_lo K_hi^T over d in chunks of 32
        for (int c = 0; c < C::kChunks && ok; ++c, ++t) {
          const int s = t % kRing;
          if (!(ok = mbar_wait(&ctl.full[s], (t / kRing) & 1, wc, kSiteTf32Mma))) break;
          tc_fence_after();
          const uint32_t base = smem_u32(sRing + s * C::kStageBytes);
          const uint64_t dqh = smem_desc(base, 16, 1024), dql = smem_desc(base + kChunkBytes, 16, 1024);
          const uint64_t dkh = smem_desc(base + 2 * kChunkBytes, 16, 1024);
          const uint64_t dkl = smem_desc(base + 3 * kChunkBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {   // 8 columns (32 bytes) per instruction
            const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
            mma_ss_tf32(tmem + C::kSCol, dqh + off, dkh + off, kIdS, (c > 0 || kk > 0) ? 1u : 0u);
            mma_ss_tf32(tmem + C::kSCol, dqh + off, dkl + off, kIdS, 1u);
            mma_ss_tf32(tmem + C::kSCol, dql + off, dkh + off, kIdS, 1u);
          }
          mma_commit(&ctl.empty[s]);
        }
        if (!ok) break;
        mma_commit(&ctl.sfull);
        // O (+)= P V once the softmax has written P over S
        if (!(ok = mbar_wait(&ctl.pfull, nv & 1, wc, kSiteTf32Mma) &&
                   mbar_wait(&ctl.vfull, nv & 1, wc, kSiteTf32Mma)))
          break;
        tc_fence_after();
        const uint64_t dv = smem_desc(smem_u32(sVt), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 8; ++kk) {   // 8 keys per instruction
          const uint64_t off =
              static_cast<uint64_t>(((kk >> 2) * C::kVtBoxBytes + (kk & 3) * 32) >> 4);
          mma_ts_tf32(tmem + C::kOCol, tmem + C::kSCol + kk * 8, dv + off, kIdO,
                      (nv > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&ctl.vempty);
      }
      if (ok && nv > 0) mma_commit(&ctl.done);
      mma_commit(&ctl.final_bar);   // every MMA done before TMEM is freed
      mbar_wait_drain(&ctl.final_bar, 0, a.timeout_ns);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------- softmax, epilogue
    const int row = (warp & 3) * 32 + lane;
    const int qi = q0 + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const float c2 = a.scale_log2;
    float m_run = -INFINITY;   // raw-score max the exponentials are taken against
    float l_sum = 0.f;
    int nv = 0;
    bool ok = true;
    for (int j = walk.next(0); j < walk.end; j = walk.next(j + 1), ++nv) {
      uint32_t keepw[4] = {~0u, ~0u, ~0u, ~0u};
      if constexpr (DROPOUT) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          keepw[q] = dropout_keep32(static_cast<uint32_t>(j * (kTile / 8) + 4 * q),
                                    static_cast<uint32_t>(qi), static_cast<uint32_t>(bh), m.offset,
                                    m.rk, m.drop_threshold);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl.sfull, nv & 1, wc, kSiteTf32Soft));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 128; c += 32) tmem_ld32(tl + C::kSCol + c, sr + c);
      tmem_wait_ld();
      const int kv0 = j * kTile;
      int lim = min(limit - kv0, kTile);
      if (m.causal) lim = min(lim, qi - kv0 + 1);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        if (c >= lim) sr[c] = __float_as_uint(-INFINITY);
        mx = fmaxf(mx, __uint_as_float(sr[c]));
      }
      // O and l hold sums against the old max: scale them by 2^(c2 (m_old -
      // m_new)) when the max grows.  The TMEM loads and stores are warp-wide
      // instructions, so the warp rescales together (alpha = 1 for rows whose
      // max did not grow).
      const bool grow = mx > m_run && m_run != -INFINITY;
      const float alpha = grow ? ex2_approx((m_run - mx) * c2) : 1.f;
      l_sum *= alpha;
      if (mx > m_run) m_run = mx;
      if (nv >= 1 && __any_sync(0xffffffffu, grow)) {
        // O holds the sum through the previous tile (complete: see above)
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tl + C::kOCol + c, o);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
          tmem_st32(tl + C::kOCol + c, o);
        }
      }
      const float mc = m_run == -INFINITY ? 0.f : m_run * c2;
#pragma unroll
      for (int c = 0; c < 128; c += 32) {
        uint32_t pk[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const float p = ex2_approx(fmaf(__uint_as_float(sr[c + u]), c2, -mc));
          l_sum += p;
          const bool keep = !DROPOUT || ((keepw[c / 32] >> u) & 1u);
          pk[u] = __float_as_uint(keep ? tf32_round(p) : 0.f);
        }
        tmem_st32(tl + C::kSCol + c, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.pfull);
    }
    if (ok && nv > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl.done, 0, wc, kSiteTf32Soft));
      if (ok) tc_fence_after();
    }
    if (ok) {   // (warp-uniform: the TMEM loads are warp-wide; rows past N only skip the stores)
      const bool live = l_sum > 0.f;
      const float inv = live ? m.drop_scale / l_sum : 0.f;
      float* orow = static_cast<float*>(a.o) + b * a.stride_b + h * a.stride_h +
                    static_cast<int64_t>(qi) * a.stride_n;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        if (nv > 0) {
          tmem_ld32(tl + C::kOCol + c, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = 0u;
        }
        if (qi < m.N) {
          float4* dst = reinterpret_cast<float4*>(orow + c);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            dst[u] = make_float4(__uint_as_float(o[4 * u]) * inv, __uint_as_float(o[4 * u + 1]) * inv,
                                 __uint_as_float(o[4 * u + 2]) * inv,
                                 __uint_as_float(o[4 * u + 3]) * inv);
        }
      }
      if (qi < m.N)
        a.lse[static_cast<int64_t>(bh) * m.N + qi] =
            live ? (m_run * c2 + __log2f(l_sum)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// Q, K -> TF32 hi and lo parts ([B*H][N][d] and [B*H_kv][N][d], contiguous);
// V -> V^T rounded to TF32 ([B*H_kv][d][npad], keys past N zero).
// blockIdx.y: 0 = Q, 1 = K, 2 = V.
__global__ void __launch_bounds__(256) tf32_split_kernel(const float* __restrict__ q,
                                                         const float* __restrict__ k,
                                                         const float* __restrict__ v,
                                                         const FwdArgs a, float* __restrict__ qhi,
                                                         float* __restrict__ qlo,
                                                         float* __restrict__ khi,
                                                         float* __restrict__ klo,
                                                         float* __restrict__ vt, int npad) {
  const MaskArgs& m = a.m;
  const int d = a.d;
  const int which = static_cast<int>(blockIdx.y);
  const int heads = which == 0 ? m.H : m.H_kv;
  const int64_t sb = which == 0 ? a.stride_b : a.kv_stride_b;
  const int64_t sh = which == 0 ? a.stride_h : a.kv_stride_h;
  const int64_t sn = which == 0 ? a.stride_n : a.kv_stride_n;
  const int64_t rows = static_cast<int64_t>(m.B) * heads * (which == 2 ? npad : m.N);
  const int64_t total = rows * d;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (which < 2) {   // e = ((bh * N) + n) * d + c
      const int c = static_cast<int>(e % d);
      const int64_t n = (e / d) % m.N;
      const int64_t bhx = e / (static_cast<int64_t>(d) * m.N);
      const int64_t bb = bhx / heads, hh = bhx % heads;
      const float x = (which == 0 ? q : k)[bb * sb + hh * sh + n * sn + c];
      const float hi = tf32_round(x);
      const float lo = tf32_round(x - hi);
      (which == 0 ? qhi : khi)[e] = hi;
      (which == 0 ? qlo : klo)[e] = lo;
    } else {           // e = ((bhk * d) + c) * npad + n
      const int64_t n = e % npad;
      const int c = static_cast<int>((e / npad) % d);
      const int64_t bhx = e / (static_cast<int64_t>(npad) * d);
      const int64_t bb = bhx / heads, hh = bhx % heads;
      vt[e] = n < m.N ? tf32_round(v[bb * sb + hh * sh + n * sn + c]) : 0.f;
    }
  }
}

template <int D, bool DROP>
cudaError_t launch_tf32(const Tf32Maps& tm, const FwdArgs& a, cudaStream_t s) {
  using C = Tf32Cfg<D>;
  static std::atomic<uint64_t> set_up{0};
  int dev = 0;
  bool todo = false;
  cudaError_t e = needs_setup(set_up, &dev, &todo);
  if (e != cudaSuccess) return e;
  if (todo) {
    e = cudaFuncSetAttribute(fwd_tf32_kernel<D, DROP>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    mark_done(set_up, dev);
  }
  const dim3 grid(static_cast<unsigned>(a.m.nb), static_cast<unsigned>(a.m.B * a.m.H));
  fwd_tf32_kernel<D, DROP><<<grid, C::kThreads, C::kSmem, s>>>(tm.qhi, tm.qlo, tm.khi, tm.klo,
                                                              tm.vt, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tf32_split(const float* q, const float* k, const float* v, const FwdArgs& a,
                              const Tf32Buffers& buf, cudaStream_t s) {
  const int64_t most = static_cast<int64_t>(a.m.B) * a.m.H * ((a.m.N + kTile - 1) / kTile * kTile) * a.d;
  int64_t blocks = (most + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  tf32_split_kernel<<<dim3(static_cast<unsigned>(blocks), 3), 256, 0, s>>>(
      q, k, v, a, buf.qhi, buf.qlo, buf.khi, buf.klo, buf.vt, buf.npad);
  return cudaGetLastError();
}

cudaError_t launch_fwd_tf32(const Tf32Maps& tm, const FwdArgs& a, cudaStream_t s) {
  const bool drop = a.m.drop_threshold != 0;
  if (a.d == 64) return drop ? launch_tf32<64, true>(tm, a, s) : launch_tf32<64, false>(tm, a, s);
  return drop ? launch_tf32<128, true>(tm, a, s) : launch_tf32<128, false>(tm, a, s);
}

}  // namespace attn
