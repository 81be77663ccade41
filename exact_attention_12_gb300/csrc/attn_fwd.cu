// Fused attention forward, bf16 in / bf16 out, tcgen05 tensor cores.
//
// Method: the tiled forward of FlashAttention (paper summary page, "Theo dõi
// Softmax tăng dần" and its four per-block steps; the "3.3 Self-Attention"
// page, §12.2 Tiling and §12.3 Online Softmax).  Query tiles of 128 rows
// stream the allowed 128-row key/value tiles past them (query-outer order,
// §12.5 of the same page), keeping the running row max m and exp-sum l on
// chip; only O and the per-row logsumexp L = c*m + ln l are written.
//
// GB300 mapping (the pages' A100 block sizes B_r/B_c from the SRAM size do
// not apply: tiles are sized by the 128-lane MMA and TMEM):
//   * One CTA owns a pair of query tiles A = 2u and B = 2u+1 of one (b, h)
//     and walks the union of their key-tile lists once; K_j / V_j are loaded
//     once for both tiles.  A key tile that only one of the two needs (the
//     causal diagonal, block-sparse lists) is skipped by the other.
//   * warp 8     TMA producer: Q_A, Q_B once, then K_j / V_j into a ring of
//                kStages shared-memory stages (128-byte swizzle).
//   * warp 9     MMA issuer (one thread) in the order
//                  ... O_A += P_A V_t, S_A = Q_A K_{t+1}^T, O_B += P_B V_t,
//                  S_B = Q_B K_{t+1}^T ...
//                so each tile's softmax runs while the tensor core works on
//                the other tile: the two tiles ping-pong.
//   * warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: thread t
//                owns row t of its tile (TMEM lane t).  It loads its whole
//                S row from TMEM into registers (four loads in flight), takes
//                the masked row max; if the max grew by more than 2^8 the
//                row's O is rescaled in TMEM (lazy rescale; the final O / l is
//                exact either way); then forms P = 2^(S c log2e - m c log2e)
//                (packed f32x2 FMA, ex2), applies the dropout keep mask and
//                writes P as bf16 over the first 64 columns of S, where
//                O += P V reads it.  With dropout the thread evaluates its
//                row's 128 keep bits (16 Philox calls) before it waits for
//                the tile's scores, so the random numbers overlap the score
//                MMA.
//   * warps 10-11 idle (they complete the third warpgroup, whose registers
//                go to the softmax warps).
//   * With few, long heads (fewer pairs than SMs) each pair's key tiles are
//     cut into pieces, units of their own; a piece leaves O normalised over
//     its keys (fp32) and its L in the workspace, and fwd_merge_kernel
//     combines the pieces.  That code is compiled only into the kernel's
//     SPLIT instances.
//   Because every tcgen05.commit covers all earlier MMAs of the issuing
//   thread, "S_X(t+1) is complete" already implies "O_X += P_X V_t is
//   complete": the softmax may then overwrite P_X and rescale O_X.
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256, 256+d),
//               O_B [256+d, 256+2d).
#include <climits>

#include <cuda_bf16.h>

#include "attn_kernels.cuh"
#include "philox.cuh"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr float kLn2 = 0.693147180559945309f;

template <int D, bool DROPOUT = false, bool FP8 = false>
struct FwdCfg {
  static constexpr int kElem = FP8 ? 1 : 2;           // bytes per operand element
  static constexpr int kBoxCols = 128 / kElem;        // elements per 128-byte box row
  static constexpr int kBoxes = D * kElem / 128;      // 128-byte-wide TMA boxes per tile
  static constexpr int kBoxBytes = kTile * 128;       // 128 rows x 128 bytes
  static constexpr int kTileBytes = kTile * D * kElem;
  static constexpr int kStages = (D == 64 || FP8) ? 4 : 2;
  static constexpr int kSmem = 1024 + kTileBytes * (2 + 2 * kStages);
  static constexpr uint32_t kSCol = 0, kOCol = 256;   // S_X at kSCol + 128X, O_X at kOCol + D*X
  // At d = 64 the bf16 P_X has columns of its own (kPCol + 64X), so the
  // scores of the next key tile can be computed while the softmax still
  // works on P; at d = 128 the TMEM is full and P_X overwrites S_X.
  static constexpr bool kSepP = (D == 64);
  static constexpr uint32_t kPCol = 384;
  // warpgroups 0, 1: softmax of tiles A, B (with dropout each thread also
  // evaluates its row's keep bits); warpgroup 2: producer (warp 8), MMA
  // issuer (warp 9), two idle warps.  Registers are re-split after the
  // start: kRegsSoftmax for the softmax warpgroups, kRegsOther for
  // warpgroup 2: 256 * 216 + 128 * 72 <= 384 * 168.
  static constexpr int kThreads = 384;
  static constexpr uint32_t kRegsLaunch = 168;
  static constexpr uint32_t kRegsSoftmax = 216;
  static constexpr uint32_t kRegsOther = 72;
  static_assert(256 * kRegsSoftmax + 128 * kRegsOther <= kThreads * kRegsLaunch,
                "register re-split exceeds the launch allocation");
};

// A claimed unit as the producer publishes it to the other roles.
struct UnitInfo {
  const uint16_t* idx[2];   // block-mask rows of query tiles A, B from their first
                            // visited entry (null: dense)
  int base[2];              // dense: first key tile A, B visit
  int n[2];                 // key tiles A and B visit
  int pair, bh, b, h, limit;
  int piece;                // key-range piece of a split pair (0 when unsplit)
  int w;                    // unit index; -1: no more units
};

// Units a CTA has claimed and not yet handed to every role.
constexpr int kUnitRing = 4;
constexpr int kClaimAhead = 2;

template <int ST>
struct FwdCtl {
  uint64_t qfull, qempty, claim;
  uint64_t kfull[ST], vfull[ST], kvempty[ST];
  uint64_t sfull[2], pfull[2], oempty[2];
  uint64_t sfree[2], pvdone[2];   // separate-P pipeline only
  uint64_t done, final_bar;
  uint64_t unitfull[kUnitRing], unitempty[kUnitRing];
  UnitInfo unit[kUnitRing];
  uint32_t tmem_base;
  int abort_flag;
  int16_t len_order[kLenOrderMaxB];   // sequences by descending key length (len_order mode)
};

// Named barrier between softmax warp 0 (ranks the sequences) and the
// producer warp (reads the ranking), in len_order mode.
constexpr int kBarLenOrder = 1;

// One unit of work: a pair of query tiles of one (b, h) and their key-tile
// lists, or, when the pairs are split along the keys (too few pairs to
// fill the GPU), one of `splits` pieces of a pair, each over a contiguous
// range of key-tile indices.  Units are numbered in head groups of G
// consecutive (b, h), within a group heaviest pair first, a pair's pieces
// together; CTAs take units round-robin.
struct FwdUnit {
  int pair, bh, b, h, limit, piece;
};


// CTA i starts with unit i; after that CTAs claim units dynamically from a
// global ticket counter (the scheduler word pair in the workspace header:
// [0] units claimed beyond the first gridDim.x, [1] CTAs finished).  The producer claims the next unit when the MMA warp signals
// that the current unit has at most kClaimAhead key tiles left to score (a
// global atomic takes microseconds, so the claim is made early enough to be
// answered before the current unit ends, and late enough that a CTA holds no
// more than one unit it has not started), and publishes it to the MMA and
// softmax warps through a ring of kUnitRing slots.  The last CTA to make its
// final claim resets both words to zero for the next launch.

// The key tiles query tile `qt` of head `bh` visits, in ascending order.
struct TileList {
  const uint16_t* idx;   // compacted block-mask row from the first visited entry, or null (dense)
  int base;              // dense: the first visited key tile
  int n;
  __device__ __forceinline__ int operator[](int t) const { return idx ? int(idx[t]) : base + t; }
};

__device__ __forceinline__ int key_limit(const MaskArgs& m, int b) {
  int limit = m.N;
  if (m.key_lens != nullptr) limit = min(max(m.key_lens[b], 0), m.N);
  return limit;
}

// First position in the sorted list p[0, n) whose tile index is >= j.
__device__ __forceinline__ int lower_bound_tile(const uint16_t* p, int n, int j) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (int(p[mid]) < j) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// The key tiles with index in [jlo, jhi) that query tile qt may attend.
__device__ __forceinline__ TileList fwd_tiles(const MaskArgs& m, int qt, int bh, int limit,
                                              int jlo, int jhi) {
  if (qt >= m.nb) return TileList{nullptr, 0, 0};   // past the last query tile
  int cap = (limit + kTile - 1) / kTile;
  if (m.causal) cap = min(cap, qt + 1);
  const int end = min(cap, jhi);
  if (m.list_idx == nullptr) return TileList{nullptr, jlo, max(0, end - jlo)};
  const size_t row = static_cast<size_t>(m.mask_per_head ? bh : 0) * m.nb + qt;
  const uint16_t* p = m.list_idx + row * m.nb;
  const int cnt = m.list_cnt[row];
  const int lo = lower_bound_tile(p, cnt, jlo);
  const int hi = lower_bound_tile(p, cnt, end);
  return TileList{p + lo, 0, max(0, hi - lo)};
}

// The key-tile range [jlo, jhi) of piece `piece` of `splits` of a query-tile
// pair: the pair's key tiles [0, J) cut into equal parts (J: the tiles below
// the key limit and, causal, at or below the pair's second tile).
__device__ __forceinline__ void piece_range(const MaskArgs& m, int pair, int limit, int piece,
                                            int splits, int& jlo, int& jhi) {
  int J = min((limit + kTile - 1) / kTile, m.nb);
  if (m.causal) J = min(J, 2 * pair + 2);
  jlo = piece * J / splits;
  jhi = (piece + 1) * J / splits;
}

// Walks the union of two sorted key-tile lists in ascending order.
struct PairWalk {
  TileList a, b;
  int ia = 0, ib = 0;
  __device__ __forceinline__ bool next(int& j, bool& na, bool& nb) {
    const int ja = ia < a.n ? a[ia] : INT_MAX;
    const int jb = ib < b.n ? b[ib] : INT_MAX;
    if (ja == INT_MAX && jb == INT_MAX) return false;
    j = min(ja, jb);
    na = ja == j;
    nb = jb == j;
    ia += na ? 1 : 0;
    ib += nb ? 1 : 0;
    return true;
  }
};

// S = Q K^T: both operands K-major; one instruction per 32 bytes of d
// (16 bf16 or 32 E4M3 elements).  The descriptors are built once per group
// and stepped by adding the (compile-time) offset to their address field:
// the issuing thread spends its time issuing, not rebuilding descriptors
// (shared-memory addresses stay below 256 KB, so the 14-bit field cannot
// carry into the next one).
template <int D, bool FP8>
__device__ __forceinline__ void mma_scores(uint32_t d_tmem, uint32_t q_base, uint32_t k_base) {
  constexpr int kSteps = D * FwdCfg<D, false, FP8>::kElem / 32;
  const uint64_t da0 = smem_desc(q_base, 16, 1024), db0 = smem_desc(k_base, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < kSteps; ++kk) {
    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * FwdCfg<D>::kBoxBytes + (kk & 3) * 32) >> 4);
    if constexpr (FP8)
      mma_ss_f8(d_tmem, da0 + off, db0 + off, idesc_e4m3(128, 128, false, false), kk > 0 ? 1u : 0u);
    else
      mma_ss(d_tmem, da0 + off, db0 + off, idesc_bf16(128, 128, false, false), kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V with P in TMEM.  bf16: V [keys, d] is the MN-major B operand,
// 16 keys per instruction.  E4M3: the B operand is the transposed tile V^T
// [d, keys] (K-major), 32 keys per instruction; P holds four keys per column.
template <int D, bool FP8>
__device__ __forceinline__ void mma_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_base,
                                       bool accumulate) {
  if constexpr (FP8) {
    constexpr uint32_t kId = idesc_e4m3(128, D, false, false);
    const uint64_t dv0 = smem_desc(v_base, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < kTile / 32; ++kk)
      mma_ts_f8(o_tmem, p_tmem + kk * 8, dv0 + static_cast<uint64_t>((kk * 32) >> 4), kId,
                (accumulate || kk > 0) ? 1u : 0u);
  } else {
    constexpr uint32_t kId = idesc_bf16(128, D, false, true);
    const uint64_t dv0 = smem_desc(v_base, FwdCfg<D>::kBoxBytes, 1024);
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk)
      mma_ts(o_tmem, p_tmem + kk * 8, dv0 + static_cast<uint64_t>((kk * 2048) >> 4), kId,
             (accumulate || kk > 0) ? 1u : 0u);
  }
}

// The forward of one CTA.  FP8: q, k are E4M3 [B,H,N,d] / [B,H_kv,N,d] maps
// with 128 x 128-byte boxes and tv maps the transposed V^T [B,H_kv,d,N].
// SPLIT: the pairs are cut into pieces along the keys (a.splits > 1); the
// unsplit kernel is compiled without the pieces' code.
template <int D, bool DROPOUT, bool FP8, bool SPLIT>
__device__ __forceinline__ void fwd_body(const CUtensorMap& tq, const CUtensorMap& tk,
                                         const CUtensorMap& tv, const FwdArgs& a) {
  using C = FwdCfg<D, DROPOUT, FP8>;
  constexpr int ST = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                          // Q_A, Q_B
  uint8_t* sK = smem + 2 * C::kTileBytes;
  uint8_t* sV = sK + ST * C::kTileBytes;
  __shared__ FwdCtl<ST> ctl;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const MaskArgs& m = a.m;
  const int BH = m.B * m.H;
  const int npairs = (m.nb + 1) / 2;
  const int K = SPLIT ? a.splits : 1;   // pieces per pair
  const int total = npairs * BH * K;
  auto unit_of = [&](int w) {
    const int G = m.head_group, per = G * npairs * K, nfull = BH / G;
    const int g = w < nfull * per ? w / per : nfull;
    const int gs = g < nfull ? G : BH - nfull * G;
    const int rem = w - g * per;
    FwdUnit u;
    u.pair = npairs - 1 - rem / (gs * K);
    const int r2 = rem % (gs * K);
    u.bh = g * G + r2 / K;
    u.piece = r2 % K;
    u.b = u.bh / m.H;
    u.h = u.bh - u.b * m.H;
    if (a.len_order) {   // (groups of one head) the sequences in their ranked order
      u.b = ctl.len_order[u.b];
      u.bh = u.b * m.H + u.h;
    }
    u.limit = key_limit(m, u.b);
    return u;
  };

  if (threadIdx.x == 0) {
    ctl.abort_flag = 0;
    mbar_init(&ctl.qfull, 1);
    mbar_init(&ctl.qempty, 1);
    mbar_init(&ctl.claim, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&ctl.kfull[s], 1);
      mbar_init(&ctl.vfull[s], 1);
      mbar_init(&ctl.kvempty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&ctl.sfull[x], 1);
      mbar_init(&ctl.pfull[x], 4);
      mbar_init(&ctl.oempty[x], 4);
      mbar_init(&ctl.sfree[x], 4);
      mbar_init(&ctl.pvdone[x], 1);
    }
    mbar_init(&ctl.done, 1);
    mbar_init(&ctl.final_bar, 1);
    for (int r = 0; r < kUnitRing; ++r) {
      mbar_init(&ctl.unitfull[r], 1);
      mbar_init(&ctl.unitempty[r], 9);   // the MMA thread and the eight softmax warps
    }
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&ctl.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the set-up above touched no global memory: from here on the previous
  // kernel of the stream must be complete
  grid_dep_wait();
  grid_dep_launch();
  const uint32_t tmem = ctl.tmem_base;
  const WaitCtx wc{&ctl.abort_flag, a.status, a.timeout_ns};
  const int wg = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 128, 0);

  if (wg == 2) {
    regs_decrease<C::kRegsOther>();
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (a.len_order) named_barrier_sync(kBarLenOrder, 64);   // warp 0 has ranked the sequences
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      int t = 0;      // key/value tiles loaded by this CTA (all units)
      int kw = 0;     // units with work
      bool ok = true;
      for (int pub = 0;; ++pub) {
        // the previous unit is close to its end: claim the next one
        if (kw >= 1 && !(ok = mbar_wait(&ctl.claim, (kw - 1) & 1, wc, kSiteFwdUnit))) break;
        // CTA i starts with unit i; later units come from the counter
        const int w = pub == 0 ? static_cast<int>(blockIdx.x)
                               : static_cast<int>(gridDim.x) + atomicAdd(a.sched, 1);
        UnitInfo ui{};
        ui.w = -1;
        if (w < total) {
          const FwdUnit u = unit_of(w);
          int jlo, jhi;
          piece_range(m, u.pair, u.limit, u.piece, K, jlo, jhi);
          const TileList la = fwd_tiles(m, 2 * u.pair, u.bh, u.limit, jlo, jhi);
          const TileList lb = fwd_tiles(m, 2 * u.pair + 1, u.bh, u.limit, jlo, jhi);
          ui = UnitInfo{{la.idx, lb.idx}, {la.base, lb.base}, {la.n, lb.n}, u.pair, u.bh,
                        u.b, u.h, u.limit, u.piece, w};
        }
        const int r = pub % kUnitRing;
        if (pub >= kUnitRing &&
            !(ok = mbar_wait(&ctl.unitempty[r], ((pub / kUnitRing) - 1) & 1, wc, kSiteFwdUnit)))
          break;
        ctl.unit[r] = ui;
        mbar_arrive(&ctl.unitfull[r]);   // release: the consumers' wait acquires unit[r]
        if (ui.w < 0) break;
        const FwdUnit u{ui.pair, ui.bh, ui.b, ui.h, ui.limit, ui.piece};
        const TileList listA{ui.idx[0], SPLIT ? ui.base[0] : 0, ui.n[0]},
            listB{ui.idx[1], SPLIT ? ui.base[1] : 0, ui.n[1]};
        if (listA.n == 0 && listB.n == 0) continue;
        // the previous unit's score MMAs are done with Q
        if (kw >= 1 && !(ok = mbar_wait(&ctl.qempty, (kw - 1) & 1, wc, kSiteFwdQ))) break;
        mbar_arrive_expect_tx(&ctl.qfull, 2 * C::kTileBytes);
#pragma unroll
        for (int x = 0; x < C::kBoxes; ++x) {
          tma_load_4d(sQ + x * C::kBoxBytes, &tq, &ctl.qfull, x * C::kBoxCols,
                      2 * u.pair * kTile, u.h, u.b);
          tma_load_4d(sQ + C::kTileBytes + x * C::kBoxBytes, &tq, &ctl.qfull, x * C::kBoxCols,
                      (2 * u.pair + 1) * kTile, u.h, u.b);
        }
        ++kw;
        const int hk = u.h / m.kv_group;   // the key/value head of query head h
        PairWalk walk{listA, listB};
        int j;
        bool na, nb;
        while (walk.next(j, na, nb)) {
          const int s = t % ST;
          if (t >= ST && !(ok = mbar_wait(&ctl.kvempty[s], ((t / ST) - 1) & 1, wc, kSiteFwdKvEmpty)))
            break;
          const int kv0 = j * kTile;
          uint8_t* dk = sK + s * C::kTileBytes;
          uint8_t* dv = sV + s * C::kTileBytes;
          mbar_arrive_expect_tx(&ctl.kfull[s], C::kTileBytes);
#pragma unroll
          for (int x = 0; x < C::kBoxes; ++x)
            tma_load_4d(dk + x * C::kBoxBytes, &tk, &ctl.kfull[s], x * C::kBoxCols, kv0, hk, u.b);
          mbar_arrive_expect_tx(&ctl.vfull[s], C::kTileBytes);
          if constexpr (FP8) {   // V^T: d rows of 128 keys
            tma_load_4d(dv, &tv, &ctl.vfull[s], kv0, 0, hk, u.b);
          } else {
#pragma unroll
            for (int x = 0; x < C::kBoxes; ++x)
              tma_load_4d(dv + x * C::kBoxBytes, &tv, &ctl.vfull[s], x * 64, kv0, hk, u.b);
          }
          ++t;
        }
      }
      // this CTA makes no further claims; the last CTA to get here resets the
      // scheduler words for the next launch (every other CTA's claims are
      // ordered before its count by the fence)
      __threadfence();
      if (atomicAdd(a.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
        atomicExch(a.sched, 0);
        atomicExch(a.sched + 1, 0);
      }
      if (ctl.abort_flag) {   // let issued copies land before the CTA exits
        if (kw >= 1) mbar_wait_drain(&ctl.qfull, (kw - 1) & 1, a.timeout_ns);
        for (int tt = max(0, t - ST); tt < t; ++tt) {
          mbar_wait_drain(&ctl.kfull[tt % ST], (tt / ST) & 1, a.timeout_ns);
          mbar_wait_drain(&ctl.vfull[tt % ST], (tt / ST) & 1, a.timeout_ns);
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t q_base0 = smem_u32(sQ);
      // the Q descriptors are rebuilt where they are used (a few integer ops
      // per MMA) instead of being kept live through the whole unit loop
      auto q_base = [&](int x) { return opaque(q_base0) + static_cast<uint32_t>(x) * C::kTileBytes; };
      uint32_t cnt[2] = {0, 0};   // P tiles consumed per query-tile slot (all units)
      uint32_t cs_issued[2] = {0, 0};   // S tiles issued per slot (separate-P pipeline)
      int t = 0;                  // key/value tiles consumed (all units)
      int kw = 0;                 // units with work
      bool ok = true;
      for (int pub = 0; ok; ++pub) {
        const int r = pub % kUnitRing;
        if (!(ok = mbar_wait(&ctl.unitfull[r], (pub / kUnitRing) & 1, wc, kSiteFwdUnit))) break;
        const UnitInfo ui = ctl.unit[r];
        mbar_arrive(&ctl.unitempty[r]);
        if (ui.w < 0) break;
        const TileList listA{ui.idx[0], SPLIT ? ui.base[0] : 0, ui.n[0]},
            listB{ui.idx[1], SPLIT ? ui.base[1] : 0, ui.n[1]};
        if (listA.n == 0 && listB.n == 0) continue;
        if (!(ok = mbar_wait(&ctl.qfull, kw & 1, wc, kSiteFwdQ))) break;
        PairWalk walk{listA, listB};
        int j;
        bool need[2], need_next[2];
        bool have = walk.next(j, need[0], need[1]);
        // scores of the first key tile
        if (!(ok = mbar_wait(&ctl.kfull[t % ST], (t / ST) & 1, wc, kSiteFwdK))) break;
        tc_fence_after();
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if (need[x]) {
            if constexpr (C::kSepP) {   // the softmax has read the previous S_X
              if (cs_issued[x] >= 1 &&
                  !(ok = mbar_wait(&ctl.sfree[x], (cs_issued[x] - 1) & 1, wc, kSiteFwdSFree)))
                break;
              tc_fence_after();
              ++cs_issued[x];
            }
            mma_scores<D, FP8>(tmem + C::kSCol + 128 * x, q_base(x), smem_u32(sK + (t % ST) * C::kTileBytes));
            mma_commit(&ctl.sfull[x]);
          }
        if (!ok) break;
        // O of both tiles was read by the previous unit's epilogues
        if (kw >= 1) {
          if (!(ok = mbar_wait(&ctl.oempty[0], (kw - 1) & 1, wc, kSiteFwdPvDone) &&
                     mbar_wait(&ctl.oempty[1], (kw - 1) & 1, wc, kSiteFwdPvDone)))
            break;
          tc_fence_after();
        }
        bool first[2] = {true, true};
        bool claimed = false;
        for (; ok && have; ++t) {
          const int s = t % ST;
          const int s1 = (t + 1) % ST;
          int jn;
          const bool have_next = walk.next(jn, need_next[0], need_next[1]);
          if (!have_next) mma_commit(&ctl.qempty);   // every score MMA of the unit is issued
          if (!claimed && walk.a.n - walk.ia <= kClaimAhead && walk.b.n - walk.ib <= kClaimAhead) {
            mbar_arrive(&ctl.claim);   // once per unit; at the latest in its last iteration
            claimed = true;
          }
          if constexpr (C::kSepP) {
            // S_X = Q_X K_{t+1}^T as soon as the softmax has read S_X(t) ...
            bool k_next_ready = false;
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              if (!(have_next && need_next[x])) continue;
              if (cs_issued[x] >= 1 &&
                  !(ok = mbar_wait(&ctl.sfree[x], (cs_issued[x] - 1) & 1, wc, kSiteFwdSFree)))
                break;
              if (!k_next_ready &&
                  !(ok = k_next_ready = mbar_wait(&ctl.kfull[s1], ((t + 1) / ST) & 1, wc, kSiteFwdK)))
                break;
              tc_fence_after();
              mma_scores<D, FP8>(tmem + C::kSCol + 128 * x, q_base(x), smem_u32(sK + s1 * C::kTileBytes));
              mma_commit(&ctl.sfull[x]);
              ++cs_issued[x];
            }
            if (!ok) break;
            // ... then O_X += P_X V_t once P_X(t) is written
            bool v_ready = false;
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              if (!need[x]) continue;
              ok = mbar_wait(&ctl.pfull[x], cnt[x] & 1, wc, kSiteFwdPFull);
              if (ok && !v_ready) ok = v_ready = mbar_wait(&ctl.vfull[s], (t / ST) & 1, wc, kSiteFwdV);
              if (!ok) break;
              tc_fence_after();
              mma_pv<D, FP8>(tmem + C::kOCol + D * x, tmem + C::kPCol + 64 * x,
                        smem_u32(sV + s * C::kTileBytes), !first[x]);
              mma_commit(&ctl.pvdone[x]);
              first[x] = false;
              ++cnt[x];
            }
            if (!ok) break;
            mma_commit(&ctl.kvempty[s]);   // K_t, V_t no longer needed
          } else {
            bool k_next_ready = false, v_ready = false;
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              if (need[x]) {   // O_X += P_X V_t
                ok = mbar_wait(&ctl.pfull[x], cnt[x] & 1, wc, kSiteFwdPFull);
                if (ok && !v_ready) ok = v_ready = mbar_wait(&ctl.vfull[s], (t / ST) & 1, wc, kSiteFwdV);
                if (!ok) break;
                tc_fence_after();
                mma_pv<D, FP8>(tmem + C::kOCol + D * x, tmem + C::kSCol + 128 * x,
                          smem_u32(sV + s * C::kTileBytes), !first[x]);
                first[x] = false;
                ++cnt[x];
              }
              if (x == 1) mma_commit(&ctl.kvempty[s]);   // K_t, V_t no longer needed
              if (have_next && need_next[x]) {   // S_X = Q_X K_{t+1}^T
                if (!k_next_ready) {
                  ok = k_next_ready = mbar_wait(&ctl.kfull[s1], ((t + 1) / ST) & 1, wc, kSiteFwdK);
                  if (!ok) break;
                  tc_fence_after();
                }
                mma_scores<D, FP8>(tmem + C::kSCol + 128 * x, q_base(x), smem_u32(sK + s1 * C::kTileBytes));
                mma_commit(&ctl.sfull[x]);
              }
            }
          }
          j = jn;
          need[0] = need_next[0];
          need[1] = need_next[1];
          have = have_next;
        }
        if (ok) mma_commit(&ctl.done);
        ++kw;
      }
      mma_commit(&ctl.final_bar);   // every MMA of this CTA done before TMEM is freed
      mbar_wait_drain(&ctl.final_bar, 0, a.timeout_ns);
    }
  }
  } else {
    regs_increase<C::kRegsSoftmax>();
    if (a.len_order && warp == 0) {
      // rank the sequences by descending key length (ties: lower index
      // first) for the producer's unit_of: lane l ranks sequence l
      const int lb = lane < m.B ? key_limit(m, lane) : -1;
      int rank = 0;
#pragma unroll
      for (int o = 0; o < 32; ++o) {
        const int lo = __shfl_sync(0xffffffffu, lb, o);
        rank += (lo > lb || (lo == lb && o < lane)) ? 1 : 0;
      }
      if (lane < m.B) ctl.len_order[rank] = static_cast<int16_t>(lane);
      named_barrier_arrive(kBarLenOrder, 64);
    }
    // ---------------------------------------------------- softmax, epilogue
    const int x = warp >> 2;                        // query tile: 0 = A, 1 = B
    const int row = (warp & 3) * 32 + lane;         // TMEM lane == row within the tile
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t sc = tl + C::kSCol + 128 * x;    // this tile's S (and P) columns
    const uint32_t oc = tl + C::kOCol + D * x;      // this tile's O columns
    const uint32_t pc = tl + C::kPCol + 64 * x;     // this tile's P columns (separate-P)
    const float c2 = a.scale_log2;
    uint32_t cs = 0;   // score tiles of this slot processed (all units)
    int kw = 0;        // units with work
    bool ok = true;
    for (int pub = 0; ok; ++pub) {
      const int r = pub % kUnitRing;
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&ctl.unitfull[r], (pub / kUnitRing) & 1, wc, kSiteFwdUnit));
      if (!ok) break;
      const UnitInfo ui = ctl.unit[r];
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.unitempty[r]);
      if (ui.w < 0) break;
      const TileList tiles{x ? ui.idx[1] : ui.idx[0], SPLIT ? (x ? ui.base[1] : ui.base[0]) : 0,
                           x ? ui.n[1] : ui.n[0]};
      const bool any = ui.n[0] > 0 || ui.n[1] > 0;
      const int bh = ui.bh, b = ui.b, h = ui.h, limit = ui.limit;
      const int q0 = (2 * ui.pair + x) * kTile;
      const int qi = q0 + row;
      const int n = tiles.n;
      float m_used = -INFINITY;      // raw-score max the exponentials are taken against
      float l_sum = 0.f;
      for (int jj = 0; jj < n; ++jj, ++cs) {
        // this row's 128 keep bits, evaluated while the tensor core forms the
        // scores (bit t of word q: key 32q + t of the tile is kept)
        uint32_t keepw[4] = {~0u, ~0u, ~0u, ~0u};
        if constexpr (DROPOUT) {
          const uint32_t j8 = static_cast<uint32_t>(tiles[jj] * (kTile / 8));
#pragma unroll
          for (int q = 0; q < 4; ++q)
            keepw[q] = dropout_keep32(j8 + 4 * q, static_cast<uint32_t>(qi),
                                      static_cast<uint32_t>(bh), m.offset, m.rk, m.drop_threshold);
        }
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl.sfull[x], cs & 1, wc, kSiteFwdSFull));
        if (!ok) break;
        tc_fence_after();
        const int kv0 = tiles[jj] * kTile;
        const int col_lim = min(limit - kv0, kTile);
        const bool diag = m.causal && kv0 == q0;
        // the whole S row: four loads in flight, one wait
        uint32_t sr[128];
  #pragma unroll
        for (int c = 0; c < 128; c += 32) tmem_ld32(sc + c, sr + c);
        tmem_wait_ld();
        if constexpr (C::kSepP) {   // S_X may be overwritten by the next key tile's scores
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.sfree[x]);
        }
        if (col_lim < kTile || diag) {
          const int lim = diag ? min(col_lim, row + 1) : col_lim;
  #pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim) sr[c] = __float_as_uint(-INFINITY);
        }
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
  #pragma unroll
        for (int c = 0; c < 128; c += 8) {
          mx0 = max3f(mx0, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
          mx1 = max3f(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
          mx2 = max3f(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
          mx3 = max3f(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
        }
        const float m_new = max3f(m_used, max3f(mx0, mx1, mx2), mx3);
        const bool need =
            m_new > m_used && (m_used == -INFINITY || (m_new - m_used) * c2 > kRescaleTau);
        float alpha = 1.f;
        if (need) {
          alpha = ex2_approx((m_used - m_new) * c2);
          m_used = m_new;
          l_sum *= alpha;
        }
        if constexpr (C::kSepP) {   // O_X += P_X V of the previous key tile is complete
          if (jj >= 1) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&ctl.pvdone[x], (cs - 1) & 1, wc, kSiteFwdPvDone));
            if (!ok) break;
            tc_fence_after();
          }
        }
        // P = 2^(S c2 - m c2) (masked entries are -inf: 2^-inf = 0), bf16 over
        // the first 64 columns of S (E4M3: the first 32)
        const float mc = (m_used == -INFINITY) ? 0.f : m_used * c2;
        const uint64_t c2x2 = f2_pack(c2, c2), nmc2 = f2_pack(-mc, -mc);
        uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
  #pragma unroll
        for (int c = 0; c < 128; c += 32) {
          const uint32_t keep = keepw[c / 32];
          uint32_t pk[16];
  #pragma unroll
          for (int t = 0; t < 32; t += 4) {
            float x0, x1, x2, x3;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c + t]), __uint_as_float(sr[c + t + 1])),
                             c2x2, nmc2), x0, x1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c + t + 2]), __uint_as_float(sr[c + t + 3])),
                             c2x2, nmc2), x2, x3);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            acc0 = f2_add(acc0, f2_pack(p0, p1));
            acc1 = f2_add(acc1, f2_pack(p2, p3));
            if constexpr (DROPOUT) {
              p0 = ((keep >> t) & 1u) ? p0 : 0.f;
              p1 = ((keep >> (t + 1)) & 1u) ? p1 : 0.f;
              p2 = ((keep >> (t + 2)) & 1u) ? p2 : 0.f;
              p3 = ((keep >> (t + 3)) & 1u) ? p3 : 0.f;
            }
            if constexpr (FP8) {
              pk[t / 4] = pack_e4m3x4(p0, p1, p2, p3);
            } else {
              pk[t / 2] = pack_bf16x2(p0, p1);
              pk[t / 2 + 1] = pack_bf16x2(p2, p3);
            }
          }
          if constexpr (FP8)
            tmem_st8(sc + c / 4, pk);
          else if constexpr (C::kSepP)
            tmem_st16(pc + c / 2, pk);
          else
            tmem_st16(sc + c / 2, pk);   // S columns [c/2, c/2+16) are already in registers
        }
        if (jj >= 1 && __any_sync(0xffffffffu, need)) {
          // O holds the sum through the previous key tile (complete: see
          // above).  Rescaled after P is formed, so that the O columns'
          // registers are not live together with the S row's.
  #pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_ld32(oc + c, o);
            tmem_wait_ld();
  #pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
            tmem_st32(oc + c, o);
          }
        }
        float ls0, ls1, ls2, ls3;
        f2_unpack(acc0, ls0, ls1);
        f2_unpack(acc1, ls2, ls3);
        ls0 += ls2;
        ls1 += ls3;
        l_sum += ls0 + ls1;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        // (an armed test stall: warp 0 withholds its first arrive, so the MMA
        // warp's wait runs out and the CTA takes its time-out path)
        if (lane == 0 && !(a.stall == kStallFwdSoftmax && warp == 0 && cs == 0))
          mbar_arrive(&ctl.pfull[x]);
      }
      if (!ok) break;
      if (any) {   // every warp takes every phase of `done`, so none falls two behind
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl.done, kw & 1, wc, kSiteFwdPvDone));
        if (!ok) break;
        tc_fence_after();
      }
      if (SPLIT && q0 < m.N) {
        // a piece of a split pair: O normalised over the piece's keys (fp32)
        // and its logsumexp, merged with the other pieces' afterwards
        const bool live = l_sum > 0.f;
        const float inv = live ? a.o_scale * (m.drop_scale / l_sum) : 0.f;
        const float L = live ? (m_used * c2 + __log2f(l_sum)) * kLn2 : -INFINITY;
        const int64_t prow = (static_cast<int64_t>(ui.piece) * BH + bh) * a.part_rows + qi;
        float* po = a.part_o + prow * D;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          if (n > 0) {
            tmem_ld32(oc + c, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = 0u;
          }
          if (qi < m.N) {
            float4* dst = reinterpret_cast<float4*>(po + c);
#pragma unroll
            for (int t = 0; t < 8; ++t)
              dst[t] = make_float4(__uint_as_float(o[4 * t]) * inv, __uint_as_float(o[4 * t + 1]) * inv,
                                   __uint_as_float(o[4 * t + 2]) * inv, __uint_as_float(o[4 * t + 3]) * inv);
          }
        }
        if (qi < m.N) a.part_l[prow] = L;
      } else if (q0 < m.N) {
        const bool live = l_sum > 0.f;
        const float inv = live ? a.o_scale * (m.drop_scale / l_sum) : 0.f;
        const float L = live ? (m_used * c2 + __log2f(l_sum)) * kLn2 : -INFINITY;
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.o) + b * a.stride_b + h * a.stride_h +
                              static_cast<int64_t>(qi) * a.stride_n;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          if (n > 0) {
            tmem_ld32(oc + c, o);
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
      if (any) {   // this tile's O has been read: the next unit may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.oempty[x]);
        ++kw;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool DROPOUT, bool SPLIT>
__global__ void __launch_bounds__(FwdCfg<D, DROPOUT>::kThreads, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const FwdArgs a) {
  fwd_body<D, DROPOUT, false, SPLIT>(tq, tk, tv, a);
}

template <int D, bool SPLIT>
__global__ void __launch_bounds__(FwdCfg<D, false, true>::kThreads, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tvt, const FwdArgs a) {
  fwd_body<D, false, true, SPLIT>(tq, tk, tvt, a);
}

template <int D, bool DROP, bool FP8, bool SPLIT>
cudaError_t launch_split(const TensorMaps& tm, const FwdArgs& a, cudaStream_t s) {
  using C = FwdCfg<D, DROP, FP8>;
  auto kernel = [] {
    if constexpr (FP8) return fwd_fp8_kernel<D, SPLIT>;
    else return fwd_bf16_kernel<D, DROP, SPLIT>;
  }();
  static std::atomic<uint64_t> set_up{0};
  int dev = 0, sms = 0;
  bool todo = false;
  cudaError_t e = needs_setup(set_up, &dev, &todo);
  if (e != cudaSuccess) return e;
  if (todo) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    // the register re-split inside the kernel assumes the launch allocation
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kernel)) != cudaSuccess) return e;
    if (static_cast<uint32_t>(fa.numRegs) < C::kRegsLaunch) return cudaErrorInvalidConfiguration;
    mark_done(set_up, dev);
  }
  // persistent: at most one CTA per SM, each walking its share of the units
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long units = static_cast<long long>((a.m.nb + 1) / 2) * a.m.B * a.m.H * a.splits;
  const unsigned grid = static_cast<unsigned>(units < sms ? units : sms);
  return launch_pdl(kernel, dim3(grid), dim3(C::kThreads), C::kSmem, s, tm.q, tm.k, tm.v, a);
}

template <int D, bool DROP, bool FP8>
cudaError_t launch_one(const TensorMaps& tm, const FwdArgs& a, cudaStream_t s) {
  return a.splits > 1 ? launch_split<D, DROP, FP8, true>(tm, a, s)
                      : launch_split<D, DROP, FP8, false>(tm, a, s);
}

// The pieces of split query-tile pairs merged by the incremental-softmax
// rule (the paper summary's running statistics, "Theo dõi Softmax tăng dần";
// the online-softmax update of the azimuth.plus explainer): with pieces s
// holding O_s normalised over their keys and L_s = logsumexp of their
// scores, L = log sum_s e^{L_s} and O = sum_s e^{L_s - L} O_s.  A piece with
// no allowed key has L_s = -inf and weight 0; a row with none at all gets
// O = 0, L = -inf.  One thread per eight columns of a row.
template <int D>
__global__ void __launch_bounds__(256) fwd_merge_kernel(const FwdArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  constexpr int kLanes = D / 8;
  const MaskArgs& m = a.m;
  const int64_t rows = static_cast<int64_t>(m.B) * m.H * m.N;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gtid / kLanes;
  if (row >= rows) return;
  const int part = static_cast<int>(gtid % kLanes);
  const int64_t n = row % m.N, bh = row / m.N;
  const int64_t piece_stride = static_cast<int64_t>(m.B) * m.H * a.part_rows;
  const int64_t prow = bh * a.part_rows + n;
  float lmax = -INFINITY;
  for (int s = 0; s < a.splits; ++s) lmax = fmaxf(lmax, a.part_l[s * piece_stride + prow]);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float L = -INFINITY;
  if (lmax > -INFINITY) {
    float wsum = 0.f;
    for (int s = 0; s < a.splits; ++s) {
      const float ls = a.part_l[s * piece_stride + prow];
      if (ls == -INFINITY) continue;
      const float w = __expf(ls - lmax);
      wsum += w;
      const float4* src = reinterpret_cast<const float4*>(a.part_o + (s * piece_stride + prow) * D + part * 8);
      const float4 x = src[0], y = src[1];
      acc[0] = fmaf(w, x.x, acc[0]); acc[1] = fmaf(w, x.y, acc[1]);
      acc[2] = fmaf(w, x.z, acc[2]); acc[3] = fmaf(w, x.w, acc[3]);
      acc[4] = fmaf(w, y.x, acc[4]); acc[5] = fmaf(w, y.y, acc[5]);
      acc[6] = fmaf(w, y.z, acc[6]); acc[7] = fmaf(w, y.w, acc[7]);
    }
    L = lmax + __logf(wsum);
    const float inv = 1.f / wsum;
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[t] *= inv;
  }
  const int64_t b = bh / m.H, h = bh % m.H;
  uint4 out;
  out.x = pack_bf16x2(acc[0], acc[1]);
  out.y = pack_bf16x2(acc[2], acc[3]);
  out.z = pack_bf16x2(acc[4], acc[5]);
  out.w = pack_bf16x2(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o) + b * a.stride_b + h * a.stride_h +
                            n * a.stride_n + part * 8) = out;
  if (part == 0) a.lse[row] = L;
}

template <int D>
cudaError_t launch_merge(const FwdArgs& a, cudaStream_t s) {
  const int64_t threads = static_cast<int64_t>(a.m.B) * a.m.H * a.m.N * (D / 8);
  const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
  return launch_pdl(fwd_merge_kernel<D>, dim3(grid), dim3(256), 0, s, a);
}

// V [B, H_kv, N, d] E4M3 -> V^T [B * H_kv][d][npad]: one CTA per 64 keys of
// one head; keys past N are written as zeros.
constexpr int kTrKeys = 64;

template <int D>
__global__ void __launch_bounds__(256) fp8_transpose_v_kernel(const uint8_t* __restrict__ v,
                                                              int64_t sb, int64_t sh, int64_t sn,
                                                              int H_kv, int N, int npad,
                                                              uint8_t* __restrict__ vt) {
  __shared__ uint8_t tile[kTrKeys][D + 16];
  const int bh = blockIdx.y, b = bh / H_kv, h = bh - b * H_kv;
  const int k0 = blockIdx.x * kTrKeys;
  const uint8_t* src = v + b * sb + h * sh;
  constexpr int kRowVecs = D / 16;   // 16-byte vectors per key row
  for (int i = threadIdx.x; i < kTrKeys * kRowVecs; i += blockDim.x) {
    const int r = i / kRowVecs, c = (i % kRowVecs) * 16;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (k0 + r < N) x = *reinterpret_cast<const uint4*>(src + static_cast<int64_t>(k0 + r) * sn + c);
    uint32_t* t = reinterpret_cast<uint32_t*>(&tile[r][c]);
    t[0] = x.x;
    t[1] = x.y;
    t[2] = x.z;
    t[3] = x.w;
  }
  __syncthreads();
  uint8_t* dst = vt + static_cast<int64_t>(bh) * D * npad;
  constexpr int kColVecs = kTrKeys / 16;   // 16-byte vectors per output row
  for (int i = threadIdx.x; i < D * kColVecs; i += blockDim.x) {
    const int c = i / kColVecs, r0 = (i % kColVecs) * 16;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      w[q] = static_cast<uint32_t>(tile[r0 + 4 * q][c]) |
             (static_cast<uint32_t>(tile[r0 + 4 * q + 1][c]) << 8) |
             (static_cast<uint32_t>(tile[r0 + 4 * q + 2][c]) << 16) |
             (static_cast<uint32_t>(tile[r0 + 4 * q + 3][c]) << 24);
    *reinterpret_cast<uint4*>(dst + static_cast<int64_t>(c) * npad + k0 + r0) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

cudaError_t launch_fwd_bf16(const TensorMaps& tm, const FwdArgs& a, cudaStream_t s) {
  const bool drop = a.m.drop_threshold != 0;
  cudaError_t e;
  if (a.d == 64)
    e = drop ? launch_one<64, true, false>(tm, a, s) : launch_one<64, false, false>(tm, a, s);
  else
    e = drop ? launch_one<128, true, false>(tm, a, s) : launch_one<128, false, false>(tm, a, s);
  if (e != cudaSuccess || a.splits <= 1) return e;
  return a.d == 64 ? launch_merge<64>(a, s) : launch_merge<128>(a, s);
}

cudaError_t launch_fp8_transpose_v(const uint8_t* v, int64_t sb, int64_t sh, int64_t sn, int B,
                                   int H_kv, int N, int d, int npad, uint8_t* vt, cudaStream_t s) {
  if (d != 128) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>((npad + kTrKeys - 1) / kTrKeys),
                  static_cast<unsigned>(B * H_kv));
  fp8_transpose_v_kernel<128><<<grid, 256, 0, s>>>(v, sb, sh, sn, H_kv, N, npad, vt);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const TensorMaps& tm, const FwdArgs& a, cudaStream_t s) {
  if (a.d != 128 || a.m.drop_threshold != 0) return cudaErrorInvalidValue;
  const cudaError_t e = launch_one<128, false, true>(tm, a, s);
  if (e != cudaSuccess || a.splits <= 1) return e;
  return launch_merge<128>(a, s);
}

}  // namespace attn
