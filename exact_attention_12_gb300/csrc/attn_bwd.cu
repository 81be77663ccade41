// Fused attention backward, bf16, tcgen05 tensor cores.
//
// The pages state the idea (FlashAttention paper summary, "Tính toán lại
// trong lượt lan truyền ngược": store only O and the softmax statistics and
// recompute S and P block by block on chip in the backward pass); the
// gradients are the chain rule of the forward definition:
//   D = rowsum(dO * O), P = exp(S - L), dV = P~^T dO, dP = (dO V^T) * Z/(1-p),
//   dS = P * (dP - D), dQ = c dS K, dK = c dS^T Q.
//
// Kernels:
//   bwd_preprocess   D = rowsum(dO * O) per query row; zeroes the fp32 dQ
//                    accumulator.  Memory-bound.
//   bwd_kernel       one CTA per 128-row key/value tile K_j, V_j of one
//                    (b, key/value head); loops over the query heads that
//                    share it (one, or a group of H / H_kv) and for each over
//                    the query tiles Q_i that may attend it (all, the causal
//                    suffix i >= j, or the block mask's column list), so the
//                    group's dK, dV sum in TMEM.  Per query tile, five MMAs:
//                      S^T  = K_j Q_i^T      (TMEM)
//                      dP^T = V_j dO_i^T     (TMEM)
//                      dV  += P~^T dO_i      (A = P~^T in TMEM, bf16)
//                      dK  += dS^T Q_i       (A = dS^T in TMEM, bf16)
//                      dQ_i = dS K_j         (A = dS^T in shared memory, read
//                                             as an MN-major operand)
//                    dK and dV stay in TMEM for the whole loop; each dQ_i is
//                    staged through shared memory and added into the fp32
//                    accumulator with TMA bulk reduce-adds.  With fewer key
//                    tiles than SMs (few, long heads) a key tile's walk is
//                    cut into pieces, units of their own, each leaving fp32
//                    dK, dV partials (the kernel's SPLIT instances).
//   bwd_merge        the pieces' dK, dV added up -> bf16 (split key tiles only).
//   dq_convert       dQ = c * accumulator -> bf16.
//
// Warp roles of bwd_kernel (384 threads; registers re-split with setmaxnreg):
//   warps 0-7  compute: warp w owns key rows 32*(w%4) .. +31 (TMEM lanes) and
//              query columns 64*(w/4) .. +63 of the S^T / dP^T tiles.  The
//              backward needs no row reduction, so the 128 columns of a row
//              split freely between two warps.  Per query tile: P^T and the
//              dropout mask, P~^T into TMEM, dS^T into TMEM and shared
//              memory, and the drain of the previous dQ tile; epilogue
//              writes dK, dV.
//   warp 8     TMA producer (K_j, V_j once; Q_i, dO_i per query tile).
//   warp 9     MMA issuer, TMEM owner.  (warps 10-11 idle: they complete the
//              third warpgroup, whose registers go to the compute warps.)
// TMEM columns: S^T [0,128) -- P~^T (bf16 pairs) overwrites columns [0,32)
//   and [64,96), each half by the warps that read that half of S^T --,
//   dP^T [128,256) -- dS^T (bf16 pairs) overwrites [128,160) and [192,224)
//   the same way --, dV [256,256+d), dK [256+d,256+2d), dQ [384,448) for
//   d = 64 and over the dP^T columns for d = 128 (issued after dK, which
//   has read dS^T: the MMAs of one thread execute in order).
#include <cuda_bf16.h>

#include "attn_kernels.cuh"
#include "philox.cuh"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kComputeWarps = 8;

template <int D>
struct BwdCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kBoxBytes = kTile * 128;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kQStages = 2;                         // Q_i (+ its L, D) stages
  static constexpr int kDoStages = (D == 64) ? 2 : 1;        // dO_i stages
  static constexpr int kDsBytes = kTile * kTile * 2;          // dS^T tile, bf16
  static constexpr int kStageBytes = kComputeWarps * 4096;    // dQ staging, 4 KB per warp
  static constexpr int kLDBytes = 2 * kTile * 4;              // -L*log2e and -D of a query tile
  // every buffer is a multiple of 1024 bytes; the dynamic base must be
  // 1024-aligned (checked at run time), so no alignment slack is requested
  static constexpr int kSmem = 2 * kTileBytes + kQStages * kTileBytes + kDoStages * kTileBytes +
                               kDsBytes + kStageBytes;
  static constexpr uint32_t kSCol = 0, kDPCol = 128, kDVCol = 256, kDKCol = 256 + D;
  static constexpr uint32_t kDQCol = (D == 64) ? 384 : 128;
  static constexpr bool kDqAliasesDp = (D == 128);
  static constexpr int kHalf = D / 2;                         // dQ/dK/dV columns per warp
  // warpgroups 0, 1: compute; warpgroup 2: producer (warp 8), MMA issuer
  // (warp 9), two idle warps.  Registers are re-split after the start:
  // 256 * kRegsCompute + 128 * kRegsOther <= 384 * kRegsLaunch.
  static constexpr int kThreads = 384;
  static constexpr uint32_t kRegsLaunch = 168, kRegsCompute = 208, kRegsOther = 80;
};

// Barriers, TMEM address and the staged row statistics: the kernel's static
// shared memory, padded to 3 KB so that the dynamic buffers after it start on
// a 1024-byte boundary.
constexpr int kBwdUnitRing = 4;   // claimed units not yet handed to every role
constexpr int kBwdClaimAhead = 2;  // claim the next unit this many query tiles early

// A claimed unit (one key tile of one (b, key/value head), or one piece of
// its query tiles when key tiles are split) as the producer publishes it.
struct BwdUnit {
  int w;      // unit index; -1: no more units
  int kt, bhk, piece;
  int n;      // (query head, query tile) pairs it visits
};

struct __align__(1024) BwdCtl {
  float ld[2][2 * kTile];   // per Q stage: -L*log2e [0,128), -D [128,256)
  uint64_t kvfull, kvempty;
  uint64_t qfull[2], qempty[2], dofull[2], doempty[2];
  uint64_t sfull, dpfull, pfull, dsfull, dqfull, dqfree, done, dkvfree, claim;
  uint64_t unitfull[kBwdUnitRing], unitempty[kBwdUnitRing];
  uint64_t final_bar;
  BwdUnit unit[kBwdUnitRing];
  uint32_t tmem_base;
  int abort_flag;
  uint8_t pad[3072 - 2 * 2 * kTile * 4 - (23 + 2 * kBwdUnitRing) * 8 -
              kBwdUnitRing * sizeof(BwdUnit) - 8];
};
static_assert(sizeof(BwdCtl) == 3072, "static shared block must stay 3 KB");

struct QList {
  const uint16_t* idx;   // block-mask column list, or null (dense)
  int first, n;
  __device__ __forceinline__ int operator[](int t) const {
    return idx ? int(idx[first + t]) : first + t;
  }
};

// First position in the sorted list p[0, n) whose tile index is >= q.
__device__ __forceinline__ int lower_bound_q(const uint16_t* p, int n, int q) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (int(p[mid]) < q) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// The query tiles key tile kt of head bh is visited by, within piece `piece`
// of `splits`: the tiles [first, nb) (first = kt when causal) are cut into
// equal index ranges.
__device__ __forceinline__ QList bwd_tiles(const MaskArgs& m, int kt, int bh, int limit,
                                           int piece, int splits) {
  QList t{nullptr, 0, 0};
  if (kt * kTile >= limit) return t;   // every key of the tile is masked
  const int first = m.causal ? kt : 0;
  const int span = m.nb - first;
  const int qlo = first + piece * span / splits;
  const int qhi = first + (piece + 1) * span / splits;
  if (m.list_idx == nullptr) {
    t.first = qlo;
    t.n = qhi - qlo;
    return t;
  }
  const size_t col = static_cast<size_t>(m.mask_per_head ? bh : 0) * m.nb + kt;
  const uint16_t* p = m.list_idx + col * m.nb;
  const int cnt = m.list_cnt[col];
  t.idx = p;
  t.first = lower_bound_q(p, cnt, qlo);
  t.n = lower_bound_q(p, cnt, qhi) - t.first;
  return t;
}

__device__ __forceinline__ int key_limit(const MaskArgs& m, int b) {
  int limit = m.N;
  if (m.key_lens != nullptr) limit = min(max(m.key_lens[b], 0), m.N);
  return limit;
}

// The (query head, query tile) pairs a key tile of key/value head hk visits:
// the query heads h0 .. h0 + g - 1 of its group in order, each with its own
// query-tile list (the block mask may differ per head).
struct QHeadWalk {
  const MaskArgs* m;
  int kt, b, h0, g, limit, piece, splits;
  int qh = -1;
  QList list{nullptr, 0, 0};
  int i = 0;
  __device__ __forceinline__ bool next(int& h, int& qtile) {
    while (qh < 0 || i >= list.n) {
      if (++qh >= g) return false;
      list = bwd_tiles(*m, kt, b * m->H + h0 + qh, limit, piece, splits);
      i = 0;
    }
    h = h0 + qh;
    qtile = list[i++];
    return true;
  }
};

// 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled tile of 128-byte rows.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return r * 128 + ((c ^ (r & 7)) << 4);
}

// Drain this warp's share of a dQ tile: TMEM -> registers -> shared memory
// (32 rows x 32 fp32 boxes, 128-byte swizzle) -> TMA reduce-add into the
// accumulator.  Arrives on `dqfree` once the TMEM columns have been read.
// The reduce-adds run on while the warp goes on: the first box goes to the
// warp's slice of the dS^T buffer (free: dS^T of this tile is consumed) when
// there are two, the last to the warp's dedicated staging box; a box is only
// rewritten after its reduce has read it (cp.async.bulk.wait_group.read).
template <int D>
__device__ __forceinline__ void drain_dq(uint32_t tl_dq, uint8_t* stage, uint8_t* ds_slice,
                                         const CUtensorMap* tdq, uint64_t* dqfree, int q_row0,
                                         int col0, int h, int b, int lane) {
  constexpr int kChunks = (D / 2) / 32;
  uint32_t v[kChunks][32];
#pragma unroll
  for (int cc = 0; cc < kChunks; ++cc) tmem_ld32(tl_dq + cc * 32, v[cc]);
  tmem_wait_ld();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(dqfree);
#pragma unroll
  for (int cc = 0; cc < kChunks; ++cc) {
    const bool last = cc == kChunks - 1;
    uint8_t* box = last ? stage : ds_slice;
    // the staging box's previous reduce (one query tile ago) has read it;
    // for the dS^T slice nothing is pending
    if (last && lane == 0) {
      if (kChunks == 2)
        tma_store_wait_read_1();
      else
        tma_store_wait_read_all();
    }
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<uint4*>(box + swz(lane, c)) =
          make_uint4(v[cc][4 * c], v[cc][4 * c + 1], v[cc][4 * c + 2], v[cc][4 * c + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_reduce_add_4d(tdq, box, col0 + cc * 32, q_row0, h, b);
      tma_store_commit();
    }
  }
}

// Shared-memory descriptor of `base` + `off` bytes, from the descriptor of
// `base`: the offset goes into the 14-bit address field (addresses stay below
// 256 KB, so it cannot carry).  The MMA groups below build one descriptor
// per operand and step it this way, so the issuing thread issues instead of
// rebuilding descriptors.
__device__ __forceinline__ uint64_t desc_plus(uint64_t desc, uint32_t off) {
  return desc + static_cast<uint64_t>(off >> 4);
}

template <int D>
__device__ __forceinline__ void mma_kt_qt(uint32_t d_tmem, uint32_t a_base, uint32_t b_base) {
  // D[128 x 128] = A[128 x D] B[128 x D]^T, both K-major (K = D)
  constexpr uint32_t kId = idesc_bf16(128, 128, false, false);
  const uint64_t da = smem_desc(a_base, 16, 1024), db = smem_desc(b_base, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * BwdCfg<D>::kBoxBytes + (kk & 3) * 32;
    mma_ss(d_tmem, desc_plus(da, off), desc_plus(db, off), kId, kk > 0 ? 1u : 0u);
  }
}

// Unit w -> (key tile, b * H_kv + key/value head, piece): head groups of G
// consecutive (b, hk); within a group, key tiles in ascending order (heaviest
// first for causal), a key tile's K pieces together.
__device__ __forceinline__ void bwd_unit_of(const MaskArgs& m, int K, int w, int& kt, int& bhk,
                                            int& piece) {
  const int BHk = m.B * m.H_kv;
  const int G = m.head_group, per = G * m.nb * K, nfull = BHk / G;
  const int g = w < nfull * per ? w / per : nfull;
  const int gs = g < nfull ? G : BHk - nfull * G;
  const int rem = w - g * per;
  kt = rem / (gs * K);
  const int r2 = rem % (gs * K);
  bhk = g * G + r2 / K;
  piece = r2 % K;
}

// SPLIT: the key tiles are cut into pieces along their query tiles
// (a.splits > 1); the unsplit kernel is compiled without the pieces' code.
template <int D, bool DROPOUT, bool SPLIT>
__global__ void __launch_bounds__(384, 1)
    bwd_bf16_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const __grid_constant__ CUtensorMap tdq, const BwdArgs a) {
  using C = BwdCfg<D>;
  constexpr int QS = C::kQStages, DS = C::kDoStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ BwdCtl ctl;
  if ((smem_u32(smem_raw) & 1023u) != 0) {   // buffers need 1024-byte alignment
    grid_dep_wait();
    if (threadIdx.x == 0 && atomicCAS(a.status, 0, kStatusSmemAlign) == 0)
      atomicExch(a.status + 1, kSiteBwdSmem);
    return;
  }
  uint8_t* sK = smem_raw;
  uint8_t* sV = sK + C::kTileBytes;
  uint8_t* sQ = sV + C::kTileBytes;                 // QS tiles
  uint8_t* sdO = sQ + QS * C::kTileBytes;           // DS tiles
  uint8_t* sDS = sdO + DS * C::kTileBytes;          // dS^T [kv][q], two 64-column boxes
  uint8_t* sStage = sDS + C::kDsBytes;              // dQ staging, 4 KB per compute warp
  float* sLD = &ctl.ld[0][0];                       // QS x (-L2[128], -D[128])

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const MaskArgs& m = a.m;
  // persistent: CTA i starts with unit i (one key tile of one (b, key/value
  // head)); later units are claimed from the scheduler counter
  const int K = SPLIT ? a.splits : 1;   // pieces per key tile
  const int total = m.nb * m.B * m.H_kv * K;

  if (threadIdx.x == 0) {
    ctl.abort_flag = 0;
    mbar_init(&ctl.kvfull, 1);
    mbar_init(&ctl.kvempty, 1);
    mbar_init(&ctl.dkvfree, kComputeWarps);
    mbar_init(&ctl.claim, 1);
    for (int r = 0; r < kBwdUnitRing; ++r) {
      mbar_init(&ctl.unitfull[r], 1);
      mbar_init(&ctl.unitempty[r], 1 + kComputeWarps);   // the MMA thread, the compute warps
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl.qfull[s], 1);
      mbar_init(&ctl.qempty[s], 1);
      mbar_init(&ctl.dofull[s], 1);
      mbar_init(&ctl.doempty[s], 1);
    }
    mbar_init(&ctl.sfull, 1);
    mbar_init(&ctl.dpfull, 1);
    mbar_init(&ctl.pfull, kComputeWarps);
    mbar_init(&ctl.dsfull, kComputeWarps);
    mbar_init(&ctl.dqfull, 1);
    mbar_init(&ctl.dqfree, kComputeWarps);
    mbar_init(&ctl.done, 1);
    mbar_init(&ctl.final_bar, 1);
    fence_mbar_init();
  }
  if (warp == kComputeWarps + 1) {
    tmem_alloc(&ctl.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the set-up above touched no global memory: from here on the previous
  // kernel of the stream (the preprocess) must be complete
  grid_dep_wait();
  grid_dep_launch();
  const uint32_t tmem = ctl.tmem_base;
  const WaitCtx wc{&ctl.abort_flag, a.status, a.timeout_ns};
  const int wg = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 128, 0);

  if (wg == 2) {
    regs_decrease<C::kRegsOther>();
    if (warp == kComputeWarps) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&tdo);
        int iq = 0, id = 0;   // Q / dO tiles issued (all units)
        int kw = 0;           // units with work
        bool ok = true;
        for (int pub = 0;; ++pub) {
          // the current unit is close to its end: claim the next one
          if (kw >= 1 && !(ok = mbar_wait(&ctl.claim, (kw - 1) & 1, wc, kSiteBwdLoad))) break;
          const int w = pub == 0 ? static_cast<int>(blockIdx.x)
                                 : static_cast<int>(gridDim.x) + atomicAdd(a.sched, 1);
          BwdUnit u{-1, 0, 0, 0, 0};
          if (w < total) {
            u.w = w;
            bwd_unit_of(m, K, w, u.kt, u.bhk, u.piece);
            const int ub = u.bhk / m.H_kv, uhk = u.bhk - ub * m.H_kv;
            const int ulim = key_limit(m, ub);
            for (int qh = 0; qh < m.kv_group; ++qh)
              u.n += bwd_tiles(m, u.kt, ub * m.H + uhk * m.kv_group + qh, ulim, u.piece, K).n;
          }
          const int r = pub % kBwdUnitRing;
          if (pub >= kBwdUnitRing &&
              !(ok = mbar_wait(&ctl.unitempty[r], ((pub / kBwdUnitRing) - 1) & 1, wc,
                               kSiteBwdLoad)))
            break;
          ctl.unit[r] = u;
          mbar_arrive(&ctl.unitfull[r]);   // release: the consumers' wait acquires unit[r]
          if (u.w < 0) break;
          if (u.n == 0) continue;
          const int b = u.bhk / m.H_kv, hk = u.bhk - b * m.H_kv;
          const int k0 = u.kt * kTile;
          // K_j, V_j: the previous unit's MMAs are done with them
          if (kw >= 1 && !(ok = mbar_wait(&ctl.kvempty, (kw - 1) & 1, wc, kSiteBwdEmpty))) break;
          mbar_arrive_expect_tx(&ctl.kvfull, 2 * C::kTileBytes);
#pragma unroll
          for (int x = 0; x < C::kBoxes; ++x) {
            tma_load_4d(sK + x * C::kBoxBytes, &tk, &ctl.kvfull, x * 64, k0, hk, b);
            tma_load_4d(sV + x * C::kBoxBytes, &tv, &ctl.kvfull, x * 64, k0, hk, b);
          }
          ++kw;
          QHeadWalk walk{&m, u.kt, b, hk * m.kv_group, m.kv_group, key_limit(m, b), u.piece, K};
          int h, qtile;
          for (int i = 0; ok && walk.next(h, qtile); ++i) {
            const int q0 = qtile * kTile;
            const int bh = b * m.H + h;
            const int sq = iq % QS;
            if (iq >= QS &&
                !(ok = mbar_wait(&ctl.qempty[sq], ((iq / QS) - 1) & 1, wc, kSiteBwdEmpty)))
              break;
            mbar_arrive_expect_tx(&ctl.qfull[sq], C::kTileBytes + C::kLDBytes);
#pragma unroll
            for (int x = 0; x < C::kBoxes; ++x)
              tma_load_4d(sQ + sq * C::kTileBytes + x * C::kBoxBytes, &tq, &ctl.qfull[sq], x * 64,
                          q0, h, b);
            const int64_t row = static_cast<int64_t>(bh) * a.npad + q0;
            bulk_load(sLD + sq * 2 * kTile, a.lse2 + row, kTile * 4, &ctl.qfull[sq]);
            bulk_load(sLD + sq * 2 * kTile + kTile, a.dsum + row, kTile * 4, &ctl.qfull[sq]);
            ++iq;
            const int sd = id % DS;
            if (id >= DS &&
                !(ok = mbar_wait(&ctl.doempty[sd], ((id / DS) - 1) & 1, wc, kSiteBwdEmpty)))
              break;
            mbar_arrive_expect_tx(&ctl.dofull[sd], C::kTileBytes);
#pragma unroll
            for (int x = 0; x < C::kBoxes; ++x)
              tma_load_4d(sdO + sd * C::kTileBytes + x * C::kBoxBytes, &tdo, &ctl.dofull[sd],
                          x * 64, q0, h, b);
            ++id;
          }
          if (!ok) break;
        }
        // no further claims from this CTA; the last CTA to get here resets the
        // scheduler words for the next launch
        __threadfence();
        if (atomicAdd(a.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
          atomicExch(a.sched, 0);
          atomicExch(a.sched + 1, 0);
        }
        if (ctl.abort_flag) {   // let issued copies land before the CTA exits
          if (kw >= 1) mbar_wait_drain(&ctl.kvfull, (kw - 1) & 1, a.timeout_ns);
          for (int ii = max(0, iq - QS); ii < iq; ++ii)
            mbar_wait_drain(&ctl.qfull[ii % QS], (ii / QS) & 1, a.timeout_ns);
          for (int ii = max(0, id - DS); ii < id; ++ii)
            mbar_wait_drain(&ctl.dofull[ii % DS], (ii / DS) & 1, a.timeout_ns);
        }
      }
    } else if (warp == kComputeWarps + 1) {
      // ----------------------------------------------------------- MMA issue
      // Order: S^T_0, dP^T_0, then per query tile i:
      //   dV_i, S^T_{i+1}, dK_i, dQ_i, dP^T_{i+1}
      // so S^T_{i+1} runs while the compute warps form dS_i, and dK_i / dQ_i
      // run while they form P_{i+1}.
      if (lane == 0) {
        constexpr uint32_t kIdKN = idesc_bf16(128, D, false, true);   // K-major A, MN-major B
        constexpr uint32_t kIdNN = idesc_bf16(128, D, true, true);    // MN-major A and B
        const uint32_t k_base0 = smem_u32(sK), v_base0 = smem_u32(sV), ds_base0 = smem_u32(sDS);
        int it = 0;   // query tiles processed (all units): the phase of every per-tile barrier
        int kw = 0;   // units with work
        bool ok = true;
        for (int pub = 0; ok; ++pub) {
          const int r = pub % kBwdUnitRing;
          if (!(ok = mbar_wait(&ctl.unitfull[r], (pub / kBwdUnitRing) & 1, wc, kSiteBwdMma)))
            break;
          const BwdUnit u = ctl.unit[r];
          mbar_arrive(&ctl.unitempty[r]);
          if (u.w < 0) break;
          const int n = u.n;
          if (n == 0) continue;
          ok = mbar_wait(&ctl.kvfull, kw & 1, wc, kSiteBwdKV) &&
               mbar_wait(&ctl.qfull[it % QS], (it / QS) & 1, wc, kSiteBwdQ) &&
               mbar_wait(&ctl.dofull[it % DS], (it / DS) & 1, wc, kSiteBwdQ);
          // at d = 128 the dP^T columns hold the previous unit's last dQ until drained
          if (ok && C::kDqAliasesDp && it >= 1)
            ok = mbar_wait(&ctl.dqfree, (it - 1) & 1, wc, kSiteBwdMma);
          if (!ok) break;
          tc_fence_after();
          mma_kt_qt<D>(tmem + C::kSCol, opaque(k_base0),
                       smem_u32(sQ + (it % QS) * C::kTileBytes));   // S^T_0
          mma_commit(&ctl.sfull);
          mma_kt_qt<D>(tmem + C::kDPCol, opaque(v_base0),
                       smem_u32(sdO + (it % DS) * C::kTileBytes));  // dP^T_0
          mma_commit(&ctl.dpfull);
          // dK, dV of the previous unit have been read out by the epilogue
          if (kw >= 1) {
            if (!(ok = mbar_wait(&ctl.dkvfree, (kw - 1) & 1, wc, kSiteBwdMma))) break;
            tc_fence_after();
          }
          bool claimed = false;
          for (int i = 0; ok && i < n; ++i, ++it) {
            const uint32_t ph = it & 1;
            const uint32_t q_base = smem_u32(sQ + (it % QS) * C::kTileBytes);
            const uint32_t do_base = smem_u32(sdO + (it % DS) * C::kTileBytes);
            // the operand descriptors are rebuilt per tile from these (a few
            // integer ops per MMA group) rather than kept live across both
            // loops, where they do not fit this warp's registers
            const uint32_t k_base = opaque(k_base0);
            const uint32_t v_base = opaque(v_base0);
            const uint32_t ds_base = opaque(ds_base0);
            if (!claimed && n - i <= kBwdClaimAhead) {
              mbar_arrive(&ctl.claim);   // once per unit; at the latest in its last iteration
              claimed = true;
            }
            // dV += P~^T dO_i; P~^T pairs of query rows 0..63 sit in columns
            // [0,32), those of rows 64..127 in [64,96)
            if (!(ok = mbar_wait(&ctl.pfull, ph, wc, kSiteBwdMma))) break;
            tc_fence_after();
            {
              const uint64_t ddo = smem_desc(do_base, C::kBoxBytes, 1024);
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                mma_ts(tmem + C::kDVCol, tmem + C::kSCol + kk * 8 + (kk >= 4 ? 32 : 0),
                       desc_plus(ddo, kk * 2048), kIdKN, (i > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&ctl.doempty[it % DS]);
            // S^T_{i+1}: the S^T columns were read by the compute warps before
            // pfull and P~^T_i is consumed by dV_i, issued just before
            if (i + 1 < n) {
              if (!(ok = mbar_wait(&ctl.qfull[(it + 1) % QS], ((it + 1) / QS) & 1, wc, kSiteBwdQ)))
                break;
              tc_fence_after();
              mma_kt_qt<D>(tmem + C::kSCol, k_base,
                           smem_u32(sQ + ((it + 1) % QS) * C::kTileBytes));
              mma_commit(&ctl.sfull);
            }
            // dK += dS^T Q_i; dS^T pairs of query rows 0..63 sit in columns
            // [128,160), those of rows 64..127 in [192,224)
            if (!(ok = mbar_wait(&ctl.dsfull, ph, wc, kSiteBwdMma))) break;
            tc_fence_after();
            {
              const uint64_t dq = smem_desc(q_base, C::kBoxBytes, 1024);
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                mma_ts(tmem + C::kDKCol, tmem + C::kDPCol + kk * 8 + (kk >= 4 ? 32 : 0),
                       desc_plus(dq, kk * 2048), kIdKN, (i > 0 || kk > 0) ? 1u : 0u);
            }
            // dQ_i = dS K_j (its columns: drained copy of the previous dQ read out)
            if (!C::kDqAliasesDp && it >= 1) {
              if (!(ok = mbar_wait(&ctl.dqfree, (it - 1) & 1, wc, kSiteBwdMma))) break;
              tc_fence_after();
            }
            {
              const uint64_t dds = smem_desc(ds_base, C::kBoxBytes, 1024);
              const uint64_t dk = smem_desc(k_base, C::kBoxBytes, 1024);
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                mma_ss(tmem + C::kDQCol, desc_plus(dds, kk * 2048), desc_plus(dk, kk * 2048), kIdNN,
                       kk > 0 ? 1u : 0u);
            }
            mma_commit(&ctl.dqfull);
            mma_commit(&ctl.qempty[it % QS]);
            // dP^T_{i+1} (for d = 128 its columns hold dQ_i until drained)
            if (i + 1 < n) {
              if (C::kDqAliasesDp && !(ok = mbar_wait(&ctl.dqfree, it & 1, wc, kSiteBwdMma)))
                break;
              if (!(ok = mbar_wait(&ctl.dofull[(it + 1) % DS], ((it + 1) / DS) & 1, wc,
                                   kSiteBwdQ)))
                break;
              tc_fence_after();
              mma_kt_qt<D>(tmem + C::kDPCol, v_base,
                           smem_u32(sdO + ((it + 1) % DS) * C::kTileBytes));
              mma_commit(&ctl.dpfull);
            }
          }
          if (!ok) break;
          mma_commit(&ctl.kvempty);   // every MMA reading K_j, V_j of this unit is issued
          mma_commit(&ctl.done);      // ... and every one writing dK, dV
          ++kw;
        }
        mma_commit(&ctl.final_bar);
        mbar_wait_drain(&ctl.final_bar, 0, a.timeout_ns);
      }
    }
  } else {
    regs_increase<C::kRegsCompute>();
    // -------------------------------------------------------------- compute
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;     // key row within the tile == TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int qc0 = half * 64;             // this warp's first query column
    const float c2 = a.scale_log2;
    const float ds = m.drop_scale;
    // this warp's 4 KB of the dS^T buffer (its rows of box `half`) and its
    // dedicated dQ staging box
    uint8_t* region = sDS + half * C::kBoxBytes + quarter * 4096;
    uint8_t* stage = sStage + warp * 4096;
    bool ok = true;
    int it = 0;   // query tiles processed (all units): the phase of every per-tile barrier
    int kw = 0;   // units with work
    for (int pub = 0; ok; ++pub) {
    const int ur = pub % kBwdUnitRing;
    ok = __all_sync(0xffffffffu,
                    mbar_wait(&ctl.unitfull[ur], (pub / kBwdUnitRing) & 1, wc, kSiteBwdSoft));
    if (!ok) break;
    const BwdUnit u = ctl.unit[ur];
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl.unitempty[ur]);
    if (u.w < 0) break;
    const int n = u.n, kt = u.kt;
    const int b = u.bhk / m.H_kv, hk = u.bhk - b * m.H_kv;
    const int k0 = kt * kTile;
    const int limit = key_limit(m, b);
    const int kj = k0 + r;                 // global key index
    const bool key_ok = kj < limit;
    const bool tile_keys_ok = k0 + kTile <= limit;   // no key of the tile is masked
    QHeadWalk walk{&m, kt, b, hk * m.kv_group, m.kv_group, limit, u.piece, K};
    int h = 0, qtile = 0;
    int prev_h = 0, prev_q0 = 0;   // the pair whose dQ is drained next
    for (int i = 0; i < n && walk.next(h, qtile); ++i, ++it) {
      const uint32_t ph = it & 1;
      const int q0 = qtile * kTile;
      const int bh = b * m.H + h;
      // -L (log2 units) and -D of this warp's 64 query rows, staged by the producer
      const float* nLw = sLD + (it % QS) * 2 * kTile + qc0;
      const float* nDw = nLw + kTile;
      const bool diag = m.causal && qtile == kt;   // query q < key: masked
      const bool edge = diag || !tile_keys_ok;

      // this row's keep bits for the warp's 64 query columns, evaluated
      // before the scores are waited for, so they overlap the S^T MMA.
      // Element (query q, key kj): 16-bit half kj mod 2 of word (kj mod 8)/2
      // of the counter (kj/8, q, bh, offset).
      uint32_t keepbits[2] = {0xffffffffu, 0xffffffffu};
      if constexpr (DROPOUT) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
          keepbits[cc] = dropout_keep32_by_key(static_cast<uint32_t>(kj),
                                               static_cast<uint32_t>(q0 + qc0 + cc * 32),
                                               static_cast<uint32_t>(bh), m.offset, m.rk,
                                               m.drop_threshold, static_cast<uint32_t>(lane));
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl.sfull, ph, wc, kSiteBwdSoft));
      if (!ok) break;
      tc_fence_after();
      // P^T = 2^(S^T c log2e - L log2e), kept in fp32 for dS; P~^T into TMEM
      float p[64];
      {
        uint32_t srr[64];
        tmem_ld32(tl + C::kSCol + qc0, srr);
        tmem_ld32(tl + C::kSCol + qc0 + 32, srr + 32);
        tmem_wait_ld();
        const uint64_t c2x2 = f2_pack(c2, c2);
#pragma unroll
        for (int t = 0; t < 64; t += 4) {
          const float4 nl = *reinterpret_cast<const float4*>(nLw + t);
          float x0, x1, x2, x3;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(srr[t]), __uint_as_float(srr[t + 1])), c2x2,
                           f2_pack(nl.x, nl.y)), x0, x1);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(srr[t + 2]), __uint_as_float(srr[t + 3])), c2x2,
                           f2_pack(nl.z, nl.w)), x2, x3);
          p[t] = ex2_approx(x0);
          p[t + 1] = ex2_approx(x1);
          p[t + 2] = ex2_approx(x2);
          p[t + 3] = ex2_approx(x3);
        }
      }
      if (edge) {   // keys past the padding length; causal diagonal tile
#pragma unroll
        for (int t = 0; t < 64; ++t)
          if (!key_ok || (diag && qc0 + t < r)) p[t] = 0.f;
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const uint32_t keep = keepbits[cc];
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          float p0 = p[cc * 32 + t], p1 = p[cc * 32 + t + 1];
          if constexpr (DROPOUT) {
            p0 = ((keep >> t) & 1u) ? p0 * ds : 0.f;
            p1 = ((keep >> (t + 1)) & 1u) ? p1 * ds : 0.f;
          }
          pk[t / 2] = pack_bf16x2(p0, p1);
        }
        // pairs of query rows qc0+32cc .. +31 -> column 64*half + 16*cc (within
        // S^T's own half, already read by this warp)
        tmem_st16(tl + C::kSCol + half * 64 + cc * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      // (an armed test stall: warp 0 withholds its first arrive, so the MMA
      // warp's wait runs out and the CTA takes its time-out path)
      if (lane == 0 && !(a.stall == kStallBwdCompute && warp == 0 && it == 0))
        mbar_arrive(&ctl.pfull);

      if (i >= 1) {   // dQ of the previous query tile: its dS^T is consumed
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl.dqfull, (it - 1) & 1, wc, kSiteBwdDq));
        if (!ok) break;
        tc_fence_after();
        drain_dq<D>(tl + C::kDQCol + half * C::kHalf, stage, region, &tdq, &ctl.dqfree,
                    prev_q0 + quarter * 32, half * C::kHalf, prev_h, b, lane);
      }
      prev_h = h;
      prev_q0 = q0;

      // dS^T = P * (dP~ * Z/(1-p) - D)
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl.dpfull, ph, wc, kSiteBwdSoft));
      if (!ok) break;
      tc_fence_after();
      uint32_t drr[64];
      tmem_ld32(tl + C::kDPCol + qc0, drr);
      tmem_ld32(tl + C::kDPCol + qc0 + 32, drr + 32);
      tmem_wait_ld();
      if (C::kHalf > 32) {   // the dS^T slice held a dQ box: its reduce has read it
        if (lane == 0) tma_store_wait_read_1();
        __syncwarp();
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const uint32_t keep = keepbits[cc];
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 32; t += 4) {
          const int e = cc * 32 + t;
          const float4 nd = *reinterpret_cast<const float4*>(nDw + e);
          float d0 = __uint_as_float(drr[e]), d1 = __uint_as_float(drr[e + 1]);
          float d2 = __uint_as_float(drr[e + 2]), d3 = __uint_as_float(drr[e + 3]);
          if constexpr (DROPOUT) {
            d0 = ((keep >> t) & 1u) ? d0 * ds : 0.f;
            d1 = ((keep >> (t + 1)) & 1u) ? d1 * ds : 0.f;
            d2 = ((keep >> (t + 2)) & 1u) ? d2 * ds : 0.f;
            d3 = ((keep >> (t + 3)) & 1u) ? d3 * ds : 0.f;
          }
          float s0, s1, s2, s3;
          f2_unpack(f2_mul(f2_pack(p[e], p[e + 1]), f2_add(f2_pack(d0, d1), f2_pack(nd.x, nd.y))),
                    s0, s1);
          f2_unpack(f2_mul(f2_pack(p[e + 2], p[e + 3]),
                           f2_add(f2_pack(d2, d3), f2_pack(nd.z, nd.w))),
                    s2, s3);
          pk[t / 2] = pack_bf16x2(s0, s1);
          pk[t / 2 + 1] = pack_bf16x2(s2, s3);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4*>(region + swz(lane, cc * 4 + u)) =
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        // the dK MMA's A operand: over this warp's dP^T half, already read
        tmem_st16(tl + C::kDPCol + half * 64 + cc * 16, pk);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.dsfull);
    }
    if (!ok) break;
    if (n > 0) {   // dQ of the unit's last query tile
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl.dqfull, (it - 1) & 1, wc, kSiteBwdDq));
      if (ok) {
        tc_fence_after();
        drain_dq<D>(tl + C::kDQCol + half * C::kHalf, stage, region, &tdq, &ctl.dqfree,
                    prev_q0 + quarter * 32, half * C::kHalf, prev_h, b, lane);
      }
    }

    // epilogue: dV and c*dK, this warp's rows and half of the columns
    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl.done, kw & 1, wc, kSiteBwdSoft));
      if (ok) tc_fence_after();
    }
    if (ok && SPLIT) {
      // a piece of a split key tile: its dV and (unscaled) dK sums in fp32,
      // added up with the other pieces' afterwards
      const int64_t prow = (static_cast<int64_t>(u.piece) * m.B * m.H_kv + u.bhk) * a.part_rows + kj;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        float* dst = (which ? a.part_dk : a.part_dv) + prow * D + half * C::kHalf;
#pragma unroll
        for (int c = 0; c < C::kHalf; c += 32) {
          uint32_t o[32];
          if (n > 0) {
            tmem_ld32(tl + (which ? C::kDKCol : C::kDVCol) + half * C::kHalf + c, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = 0u;
          }
          if (kj < m.N) {
            float4* d4 = reinterpret_cast<float4*>(dst + c);
#pragma unroll
            for (int t = 0; t < 8; ++t)
              d4[t] = key_ok ? make_float4(__uint_as_float(o[4 * t]), __uint_as_float(o[4 * t + 1]),
                                           __uint_as_float(o[4 * t + 2]), __uint_as_float(o[4 * t + 3]))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
    } else if (ok) {
      const int64_t row_off = b * a.kv_stride_b + hk * a.kv_stride_h +
                              static_cast<int64_t>(kj) * a.kv_stride_n + half * C::kHalf;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(which ? a.dk : a.dv) + row_off;
        const float mul = which ? a.scale : 1.f;
#pragma unroll
        for (int c = 0; c < C::kHalf; c += 32) {
          uint32_t o[32];
          if (n > 0) {
            tmem_ld32(tl + (which ? C::kDKCol : C::kDVCol) + half * C::kHalf + c, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = 0u;
          }
          uint32_t pk[16];
#pragma unroll
          for (int t = 0; t < 32; t += 2)
            pk[t / 2] = pack_bf16x2(key_ok ? __uint_as_float(o[t]) * mul : 0.f,
                                    key_ok ? __uint_as_float(o[t + 1]) * mul : 0.f);
          if (kj < m.N) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
            for (int t = 0; t < 4; ++t)
              d4[t] = make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
          }
        }
      }
    }
    if (ok && n > 0) {   // dK, dV read out: the next unit's first dK, dV MMAs may overwrite them
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.dkvfree);
      ++kw;
    }
    }
    if (lane == 0) tma_store_wait_all();   // this warp's reduce-adds are complete
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kComputeWarps + 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Per query row of the padded [B*H][npad] layout (one row per group of d/8
// lanes): -D = -rowsum(dO * O) and -L * log2(e) (-inf for padding rows and
// rows with no allowed key, so they contribute nothing); and dQacc = 0.  The
// negated forms let the backward use one fused multiply-add per element.
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                                            const __nv_bfloat16* __restrict__ dout,
                                                            const BwdArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  constexpr int kLanes = D / 8;                 // lanes per row
  const int64_t rows = static_cast<int64_t>(a.m.B) * a.m.H * a.npad;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gtid / kLanes;
  const int part = static_cast<int>(gtid % kLanes);
  const int64_t n = row % a.npad;
  const int64_t bh = row / a.npad;
  const bool real = row < rows && n < a.m.N;
  float s = 0.f;
  if (real) {
    // zero this thread's 8 elements of the dQ accumulator ([B, H, N, d])
    float4* acc = reinterpret_cast<float4*>(a.dq_acc + (bh * a.m.N + n) * D + part * 8);
    acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t b = bh / a.m.H, h = bh % a.m.H;
    const int64_t off = b * a.stride_b + h * a.stride_h + n * a.stride_n + part * 8;
    const uint4 ov = *reinterpret_cast<const uint4*>(o + off);
    const uint4 gv = *reinterpret_cast<const uint4*>(dout + off);
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 x = __bfloat1622float2(o2[t]), y = __bfloat1622float2(g2[t]);
      s = fmaf(x.x, y.x, s);
      s = fmaf(x.y, y.y, s);
    }
  }
#pragma unroll
  for (int w = kLanes / 2; w > 0; w >>= 1) s += __shfl_xor_sync(0xffffffffu, s, w);
  if (row < rows && part == 0) {
    float nl2 = -INFINITY;
    if (real) {
      const float L = a.lse[bh * a.m.N + n];
      if (L != -INFINITY) nl2 = -L * kLog2e;
    }
    a.dsum[row] = -s;
    a.lse2[row] = nl2;
  }
}

template <int D>
__global__ void __launch_bounds__(256) dq_convert_kernel(__nv_bfloat16* __restrict__ dq,
                                                        const BwdArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t rows = static_cast<int64_t>(a.m.B) * a.m.H * a.m.N;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gtid / (D / 8);
  const int part = static_cast<int>(gtid % (D / 8));
  if (row >= rows) return;
  const int64_t n = row % a.m.N;
  const int64_t bh = row / a.m.N;
  const int64_t b = bh / a.m.H, h = bh % a.m.H;
  const float4* src = reinterpret_cast<const float4*>(a.dq_acc + row * D + part * 8);
  const float4 x = src[0], y = src[1];
  const float c = a.scale;
  uint4 out;
  out.x = pack_bf16x2(x.x * c, x.y * c);
  out.y = pack_bf16x2(x.z * c, x.w * c);
  out.z = pack_bf16x2(y.x * c, y.y * c);
  out.w = pack_bf16x2(y.z * c, y.w * c);
  *reinterpret_cast<uint4*>(dq + b * a.stride_b + h * a.stride_h + n * a.stride_n + part * 8) = out;
}

// dK, dV of split key tiles: the pieces' fp32 sums added up, dK scaled by c,
// converted to bf16.  One thread per eight columns of a key row.
template <int D>
__global__ void __launch_bounds__(256) bwd_merge_kernel(const BwdArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  constexpr int kLanes = D / 8;
  const MaskArgs& m = a.m;
  const int64_t rows = static_cast<int64_t>(m.B) * m.H_kv * m.N;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gtid / kLanes;
  if (row >= rows) return;
  const int part = static_cast<int>(gtid % kLanes);
  const int64_t n = row % m.N, bhk = row / m.N;
  const int64_t piece_stride = static_cast<int64_t>(m.B) * m.H_kv * a.part_rows * D;
  const int64_t off = (bhk * a.part_rows + n) * D + part * 8;
  float dk[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, dv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < a.splits; ++s) {
    const float4* pk = reinterpret_cast<const float4*>(a.part_dk + s * piece_stride + off);
    const float4* pv = reinterpret_cast<const float4*>(a.part_dv + s * piece_stride + off);
    const float4 k0 = pk[0], k1 = pk[1], v0 = pv[0], v1 = pv[1];
    dk[0] += k0.x; dk[1] += k0.y; dk[2] += k0.z; dk[3] += k0.w;
    dk[4] += k1.x; dk[5] += k1.y; dk[6] += k1.z; dk[7] += k1.w;
    dv[0] += v0.x; dv[1] += v0.y; dv[2] += v0.z; dv[3] += v0.w;
    dv[4] += v1.x; dv[5] += v1.y; dv[6] += v1.z; dv[7] += v1.w;
  }
  const int64_t b = bhk / m.H_kv, hk = bhk % m.H_kv;
  const int64_t dst = b * a.kv_stride_b + hk * a.kv_stride_h + n * a.kv_stride_n + part * 8;
  const float c = a.scale;
  uint4 ko, vo;
  ko.x = pack_bf16x2(dk[0] * c, dk[1] * c); ko.y = pack_bf16x2(dk[2] * c, dk[3] * c);
  ko.z = pack_bf16x2(dk[4] * c, dk[5] * c); ko.w = pack_bf16x2(dk[6] * c, dk[7] * c);
  vo.x = pack_bf16x2(dv[0], dv[1]); vo.y = pack_bf16x2(dv[2], dv[3]);
  vo.z = pack_bf16x2(dv[4], dv[5]); vo.w = pack_bf16x2(dv[6], dv[7]);
  *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dk) + dst) = ko;
  *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dv) + dst) = vo;
}

template <int D, bool DROP, bool SPLIT>
cudaError_t launch_main(const TensorMaps& tm, const BwdArgs& a, cudaStream_t s) {
  using C = BwdCfg<D>;
  static std::atomic<uint64_t> set_up{0};
  int dev = 0, sms = 0;
  bool todo = false;
  cudaError_t e = needs_setup(set_up, &dev, &todo);
  if (e != cudaSuccess) return e;
  if (todo) {
    e = cudaFuncSetAttribute(bwd_bf16_kernel<D, DROP, SPLIT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    // the register re-split inside the kernel assumes the launch allocation
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, bwd_bf16_kernel<D, DROP, SPLIT>)) != cudaSuccess) return e;
    if (static_cast<uint32_t>(fa.numRegs) < C::kRegsLaunch) return cudaErrorInvalidConfiguration;
    mark_done(set_up, dev);
  }
  // persistent: at most one CTA per SM, each claiming units (one key tile of
  // one (b, key/value head)) until none are left
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long units = static_cast<long long>(a.m.nb) * a.m.B * a.m.H_kv * a.splits;
  const unsigned grid = static_cast<unsigned>(units < sms ? units : sms);
  e = launch_pdl(bwd_bf16_kernel<D, DROP, SPLIT>, dim3(grid), dim3(C::kThreads), C::kSmem, s,
                 tm.q, tm.k, tm.v, tm.dout, tm.dq_acc, a);
  if (e != cudaSuccess || !SPLIT) return e;
  const int64_t threads = static_cast<int64_t>(a.m.B) * a.m.H_kv * a.m.N * (D / 8);
  return launch_pdl(bwd_merge_kernel<D>, dim3(static_cast<unsigned>((threads + 255) / 256)),
                    dim3(256), 0, s, a);
}

template <int D, bool DROP>
cudaError_t launch_main(const TensorMaps& tm, const BwdArgs& a, cudaStream_t s) {
  return a.splits > 1 ? launch_main<D, DROP, true>(tm, a, s) : launch_main<D, DROP, false>(tm, a, s);
}

unsigned blocks_for(int64_t threads) {
  const int64_t b = (threads + 255) / 256;
  return static_cast<unsigned>(b < 1 ? 1 : (b > 2147483647 ? 2147483647 : b));
}

}  // namespace

cudaError_t launch_bwd_preprocess(const void* o, const void* dout, const BwdArgs& a,
                                  cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(a.m.B) * a.m.H * a.npad;
  const unsigned grid = blocks_for(rows * (a.d / 8));
  const auto* o16 = static_cast<const __nv_bfloat16*>(o);
  const auto* g16 = static_cast<const __nv_bfloat16*>(dout);
  return a.d == 64 ? launch_pdl(bwd_preprocess_kernel<64>, dim3(grid), dim3(256), 0, s, o16, g16, a)
                   : launch_pdl(bwd_preprocess_kernel<128>, dim3(grid), dim3(256), 0, s, o16, g16,
                                a);
}

cudaError_t launch_bwd_bf16(const TensorMaps& tm, const BwdArgs& a, cudaStream_t s) {
  const bool drop = a.m.drop_threshold != 0;
  if (a.d == 64) return drop ? launch_main<64, true>(tm, a, s) : launch_main<64, false>(tm, a, s);
  return drop ? launch_main<128, true>(tm, a, s) : launch_main<128, false>(tm, a, s);
}

cudaError_t launch_dq_convert(void* dq, const BwdArgs& a, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(a.m.B) * a.m.H * a.m.N;
  const unsigned grid = blocks_for(rows * (a.d / 8));
  auto* dq16 = static_cast<__nv_bfloat16*>(dq);
  return a.d == 64 ? launch_pdl(dq_convert_kernel<64>, dim3(grid), dim3(256), 0, s, dq16, a)
                   : launch_pdl(dq_convert_kernel<128>, dim3(grid), dim3(256), 0, s, dq16, a);
}

}  // namespace attn
