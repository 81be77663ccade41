// Fused attention forward, bf16 in / bf16 out, tcgen05 tensor cores.
//
// Method: the tiled forward of FlashAttention (paper summary page, "Theo dõi
// Softmax tăng dần" and its four per-block steps; the "3.3 Self-Attention"
// page, §12.2 Tiling and §12.3 Online Softmax).  Each CTA owns one 128-row
// query tile Q_i of one (b, h) and streams the allowed 128-row key/value
// tiles K_j, V_j past it (query-outer order, §12.5 of the same page), keeping
// the running row max m and exp-sum l on chip; only O and the per-row
// logsumexp L = c*m + ln l are written.
//
// GB300 mapping (differs from the pages' A100 design: no B_r/B_c from the
// SRAM size; tiles are sized by TMEM and the 128-lane MMA):
//   warp 4      TMA producer: Q_i once, then K_j / V_j into a ring of
//               kStages shared-memory stages (128-byte swizzle).
//   warp 5      MMA issuer (one thread): S_j = Q_i K_j^T into one of two TMEM
//               S buffers, then O += P_j V_j with P_j read from TMEM.  S_{j+1}
//               is issued before O += P_j V_j so the tensor core works on the
//               next scores while the softmax warps handle the current ones.
//   warps 0-3   softmax: thread t owns row t (TMEM lane t).  Loads its S row,
//               applies the masks, updates m, rescales O in TMEM only when
//               the max grew by more than 2^8 (lazy rescale; the final O/l
//               is exact either way), computes P = 2^(S*c*log2e - m*c*log2e)
//               with ex2, applies the dropout keep mask, packs P to bf16 into
//               TMEM, and in the epilogue writes O / l and L.
// TMEM columns: S0 [0,128) S1 [128,256) P0 [256,320) P1 [320,384)
//               O [384, 384 + d).
#include <cuda_bf16.h>

#include "attn_kernels.cuh"
#include "philox.cuh"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr float kLn2 = 0.693147180559945309f;

template <int D>
struct FwdCfg {
  static constexpr int kBoxes = D / 64;               // 64-column TMA boxes per tile
  static constexpr int kBoxBytes = kTile * 128;       // 128 rows x 128 bytes
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static constexpr int kSmem = 1024 + kTileBytes * (1 + 2 * kStages);
  static constexpr uint32_t kSCol = 0, kPCol = 256, kOCol = 384;
  static constexpr int kThreads = 192;
};

template <int ST>
struct FwdCtl {
  uint64_t qfull;
  uint64_t kfull[ST], vfull[ST], kvempty[ST];
  uint64_t sfull[2], sfree[2], pfull[2], pvdone[2];
  uint64_t final_bar;
  uint32_t tmem_base;
  int abort_flag;
};

// The key tiles query tile `qt` of head `bh` visits, in ascending order.
struct TileList {
  const uint16_t* idx;   // compacted block-mask row, or null (dense)
  int n;
  __device__ __forceinline__ int operator[](int t) const { return idx ? int(idx[t]) : t; }
};

__device__ __forceinline__ int key_limit(const MaskArgs& m, int b) {
  int limit = m.N;
  if (m.key_lens != nullptr) limit = min(max(m.key_lens[b], 0), m.N);
  return limit;
}

__device__ __forceinline__ TileList fwd_tiles(const MaskArgs& m, int qt, int bh, int limit) {
  int cap = (limit + kTile - 1) / kTile;
  if (m.causal) cap = min(cap, qt + 1);
  TileList t{nullptr, cap};
  if (m.list_idx != nullptr) {
    const size_t row = static_cast<size_t>(m.mask_per_head ? bh : 0) * m.nb + qt;
    const uint16_t* p = m.list_idx + row * m.nb;
    int lo = 0, hi = m.list_cnt[row];
    while (lo < hi) {   // the list is sorted: the usable part is a prefix
      const int mid = (lo + hi) >> 1;
      if (int(p[mid]) < cap) lo = mid + 1; else hi = mid;
    }
    t.idx = p;
    t.n = lo;
  }
  return t;
}

template <int D, bool DROPOUT>
__global__ void __launch_bounds__(192, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const FwdArgs a) {
  using C = FwdCfg<D>;
  constexpr int ST = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + C::kTileBytes;
  uint8_t* sV = sK + ST * C::kTileBytes;
  __shared__ FwdCtl<ST> ctl;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const MaskArgs& m = a.m;
  const int BH = m.B * m.H;
  const int qt = m.nb - 1 - static_cast<int>(blockIdx.x / BH);   // heaviest tiles first
  const int bh = static_cast<int>(blockIdx.x % BH);
  const int b = bh / m.H, h = bh - b * m.H;
  const int q0 = qt * kTile;
  const int limit = key_limit(m, b);
  const TileList tiles = fwd_tiles(m, qt, bh, limit);
  const int n = tiles.n;

  if (threadIdx.x == 0) {
    ctl.abort_flag = 0;
    mbar_init(&ctl.qfull, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&ctl.kfull[s], 1);
      mbar_init(&ctl.vfull[s], 1);
      mbar_init(&ctl.kvempty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl.sfull[s], 1);
      mbar_init(&ctl.sfree[s], 4);
      mbar_init(&ctl.pfull[s], 4);
      mbar_init(&ctl.pvdone[s], 1);
    }
    mbar_init(&ctl.final_bar, 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&ctl.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const WaitCtx wc{&ctl.abort_flag, a.status, a.timeout_ns};

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_arrive_expect_tx(&ctl.qfull, C::kTileBytes);
#pragma unroll
      for (int x = 0; x < C::kBoxes; ++x)
        tma_load_4d(sQ + x * C::kBoxBytes, &tq, &ctl.qfull, x * 64, q0, h, b);
      int j = 0;
      for (; j < n; ++j) {
        const int s = j % ST;
        if (j >= ST && !mbar_wait(&ctl.kvempty[s], ((j / ST) - 1) & 1, wc, kSiteFwdKvEmpty)) break;
        const int kv0 = tiles[j] * kTile;
        uint8_t* dk = sK + s * C::kTileBytes;
        uint8_t* dv = sV + s * C::kTileBytes;
        mbar_arrive_expect_tx(&ctl.kfull[s], C::kTileBytes);
#pragma unroll
        for (int x = 0; x < C::kBoxes; ++x)
          tma_load_4d(dk + x * C::kBoxBytes, &tk, &ctl.kfull[s], x * 64, kv0, h, b);
        mbar_arrive_expect_tx(&ctl.vfull[s], C::kTileBytes);
#pragma unroll
        for (int x = 0; x < C::kBoxes; ++x)
          tma_load_4d(dv + x * C::kBoxBytes, &tv, &ctl.vfull[s], x * 64, kv0, h, b);
      }
      if (ctl.abort_flag) {   // let issued copies land before the CTA exits
        mbar_wait_drain(&ctl.qfull, 0, a.timeout_ns);
        for (int jj = max(0, j - ST); jj < j; ++jj) {
          mbar_wait_drain(&ctl.kfull[jj % ST], (jj / ST) & 1, a.timeout_ns);
          mbar_wait_drain(&ctl.vfull[jj % ST], (jj / ST) & 1, a.timeout_ns);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------- MMA issue
    if (lane == 0 && n > 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdO = idesc_bf16(128, D, false, true);
      const uint32_t q_base = smem_u32(sQ);
      bool ok = mbar_wait(&ctl.qfull, 0, wc, kSiteFwdQ);
      for (int j = 0; ok && j <= n; ++j) {
        if (j < n) {
          const int s = j % ST, bb = j & 1;
          ok = mbar_wait(&ctl.kfull[s], (j / ST) & 1, wc, kSiteFwdK);
          if (ok && j >= 2) ok = mbar_wait(&ctl.sfree[bb], ((j - 2) >> 1) & 1, wc, kSiteFwdSFree);
          if (!ok) break;
          tc_fence_after();
          const uint32_t k_base = smem_u32(sK + s * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kBoxBytes + (kk & 3) * 32;
            mma_ss(tmem + C::kSCol + bb * 128, smem_desc(q_base + off, 16, 1024),
                   smem_desc(k_base + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
          }
          mma_commit(&ctl.sfull[bb]);
        }
        if (j >= 1) {
          const int jj = j - 1, s = jj % ST, bb = jj & 1;
          ok = mbar_wait(&ctl.pfull[bb], (jj >> 1) & 1, wc, kSiteFwdPFull) &&
               mbar_wait(&ctl.vfull[s], (jj / ST) & 1, wc, kSiteFwdV);
          if (!ok) break;
          tc_fence_after();
          const uint32_t v_base = smem_u32(sV + s * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            mma_ts(tmem + C::kOCol, tmem + C::kPCol + bb * 64 + kk * 8,
                   smem_desc(v_base + kk * 2048, C::kBoxBytes, 1024), kIdO,
                   (jj > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&ctl.pvdone[bb]);
          mma_commit(&ctl.kvempty[s]);
        }
      }
      mma_commit(&ctl.final_bar);   // every MMA of this CTA done before TMEM is freed
      mbar_wait_drain(&ctl.final_bar, 0, a.timeout_ns);
    }
  } else {
    // ---------------------------------------------------- softmax, epilogue
    const int row = threadIdx.x;   // == TMEM lane == row within the tile
    const int qi = q0 + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float c2 = a.scale_log2;
    float m_used = -INFINITY;      // raw-score max the exponentials are taken against
    float l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int bb = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl.sfull[bb], (j >> 1) & 1, wc, kSiteFwdSFull));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tl + C::kSCol + bb * 128 + c * 32, sr + c * 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.sfree[bb]);

      const int kv0 = tiles[j] * kTile;
      const int col_lim = min(limit - kv0, kTile);
      const bool diag = m.causal && kv0 == q0;
      if (col_lim < kTile || diag) {
        const int lim = diag ? min(col_lim, row + 1) : col_lim;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= lim) sr[c] = __float_as_uint(-INFINITY);
      }
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; c += 4) {
        mx0 = fmaxf(mx0, __uint_as_float(sr[c]));
        mx1 = fmaxf(mx1, __uint_as_float(sr[c + 1]));
        mx2 = fmaxf(mx2, __uint_as_float(sr[c + 2]));
        mx3 = fmaxf(mx3, __uint_as_float(sr[c + 3]));
      }
      const float m_new = fmaxf(m_used, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)));
      const bool need =
          m_new > m_used && (m_used == -INFINITY || (m_new - m_used) * c2 > kRescaleTau);
      float alpha = 1.f;
      if (need) {
        alpha = ex2_approx((m_used - m_new) * c2);
        m_used = m_new;
        l_sum *= alpha;
      }
      if (j >= 1 && __any_sync(0xffffffffu, need)) {
        // O holds P_0 V_0 + ... + P_{j-1} V_{j-1} once that MMA is done
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl.pvdone[(j - 1) & 1], ((j - 1) >> 1) & 1, wc,
                                               kSiteFwdPvDone));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tl + C::kOCol + c, o);
          tmem_wait_ld();
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
          tmem_st32(tl + C::kOCol + c, o);
        }
      }
      if (j >= 2) {   // P buffer bb was last read by O += P_{j-2} V_{j-2}
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl.pvdone[bb], ((j - 2) >> 1) & 1, wc,
                                               kSiteFwdPvDone));
        if (!ok) break;
        tc_fence_after();
      }
      const float mc = (m_used == -INFINITY) ? 0.f : m_used * c2;
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int c = 0; c < 128; c += 32) {
        uint32_t keep = 0xffffffffu;
        if constexpr (DROPOUT) {
          keep = 0;
#pragma unroll
          for (int g = 0; g < 8; ++g)
            keep |= dropout_keep4(static_cast<uint32_t>((kv0 + c) / 4 + g), static_cast<uint32_t>(qi),
                                  static_cast<uint32_t>(bh), m.offset, m.seed_lo, m.seed_hi,
                                  m.drop_threshold)
                    << (4 * g);
        }
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          float p0 = ex2_approx(fmaf(__uint_as_float(sr[c + t]), c2, -mc));
          float p1 = ex2_approx(fmaf(__uint_as_float(sr[c + t + 1]), c2, -mc));
          ls0 += p0;
          ls1 += p1;
          if constexpr (DROPOUT) {
            p0 = ((keep >> t) & 1u) ? p0 : 0.f;
            p1 = ((keep >> (t + 1)) & 1u) ? p1 : 0.f;
          }
          pk[t / 2] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tl + C::kPCol + bb * 64 + c / 2, pk);
      }
      l_sum += ls0 + ls1;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.pfull[bb]);
    }

    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl.pvdone[(n - 1) & 1], ((n - 1) >> 1) & 1, wc,
                                             kSiteFwdPvDone));
      if (ok) tc_fence_after();
    }
    if (ok) {
      const bool live = l_sum > 0.f;
      const float inv = live ? m.drop_scale / l_sum : 0.f;
      const float L = live ? (m_used * c2 + __log2f(l_sum)) * kLn2 : -INFINITY;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.o) + b * a.stride_b + h * a.stride_h +
                            static_cast<int64_t>(qi) * a.stride_n;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        if (n > 0) {
          tmem_ld32(tl + C::kOCol + c, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2)
          pk[t / 2] = pack_bf16x2(__uint_as_float(o[t]) * inv, __uint_as_float(o[t + 1]) * inv);
        if (qi < m.N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
          for (int t = 0; t < 4; ++t)
            dst[t] = make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
        }
      }
      if (qi < m.N) a.lse[static_cast<int64_t>(bh) * m.N + qi] = L;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool DROP>
cudaError_t launch_one(const TensorMaps& tm, const FwdArgs& a, cudaStream_t s) {
  using C = FwdCfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(fwd_bf16_kernel<D, DROP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const unsigned grid = static_cast<unsigned>(a.m.nb) * a.m.B * a.m.H;
  fwd_bf16_kernel<D, DROP><<<grid, C::kThreads, C::kSmem, s>>>(tm.q, tm.k, tm.v, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const TensorMaps& tm, const FwdArgs& a, cudaStream_t s) {
  const bool drop = a.m.drop_threshold != 0;
  if (a.d == 64) return drop ? launch_one<64, true>(tm, a, s) : launch_one<64, false>(tm, a, s);
  return drop ? launch_one<128, true>(tm, a, s) : launch_one<128, false>(tm, a, s);
}

}  // namespace attn
