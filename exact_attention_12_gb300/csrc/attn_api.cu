// Host side of the C interface declared in include/attn.h: argument
// validation, workspace layout, TMA tensor-map encoding and kernel launches.
// Nothing here allocates device memory.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "attn.h"
#include "attn_kernels.cuh"

namespace {

using attn::kTile;

thread_local std::string g_last_error;

// A test stall armed by attn_debug_stall for the next launch of the named
// kernel on this host thread, and the wait limit that launch gets.
thread_local int g_stall = attn::kStallNone;
thread_local uint64_t g_stall_limit_ns = 0;

// Takes the armed stall if it names `which`: sets the launch's stall and
// wait limit, and disarms it.
template <typename Args>
void take_stall(int which, Args* a) {
  if (g_stall == which && which != attn::kStallNone) {
    a->stall = which;
    a->timeout_ns = g_stall_limit_ns;
    g_stall = attn::kStallNone;
  }
}

attn_status fail(attn_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

attn_status cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr size_t kHeaderBytes = 256;   // status words [0, 8), scheduler words [128, 136)
constexpr size_t kSchedOffset = 128;
constexpr uint64_t kTimeoutNs = 2000000000ull;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t list_cnt = 0, list_idx = 0;   // compacted block mask (0 = none)
  size_t vt = 0;                       // FP8 forward: V^T [B * H_kv][d][nb * 128]
  size_t part_o = 0, part_l = 0;       // forward of split pairs: partial O, L
  int splits = 1;
  size_t qhi = 0, qlo = 0, khi = 0, klo = 0, vt32 = 0;   // fp32 forward: TF32 parts
  size_t lse2 = 0, dsum = 0, dq_acc = 0;   // backward only
  size_t part_dk = 0, part_dv = 0;         // backward of split key tiles: partial dK, dV
  int bwd_splits = 1;
  size_t total = 0;
};

int num_masks(const attn_params* p) {
  return p->block_mask_head_stride != 0 ? p->B * p->H : 1;
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    sms = 148;
  return sms;
}

// Key padding without the causal mask, up to kLenOrderMaxB sequences: the
// forward numbers its units longest sequence first (ranked in the kernel).
bool fwd_len_order(const attn_params* p) {
  return p->key_lens != nullptr && !p->causal && p->B <= attn::kLenOrderMaxB;
}

// Key tiles a piece of a split pair keeps at least.  A unit has fixed
// costs (claim, Q load, pipeline fill, epilogue) of a few key steps, and the
// pieces' partials must be merged afterwards, so short pieces lose more
// than the fuller GPU gains (measured: causal d = 128 with 16 heads at
// N = 1024, cut into pieces of 1-2 key tiles, took 41 us against 24 us
// unsplit).
constexpr long long kMinPieceTiles = 8;

// Pieces per query-tile pair in the forward.  With fewer pairs than SMs and
// long rows (few heads, long sequences) the pairs are cut along the keys
// into pieces merged afterwards: about two units per SM, each piece at least
// kMinPieceTiles key tiles of the longest pair, at most 16; otherwise 1.
// Rows under 32 key tiles are cut only when the pairs fill at most half of
// the SMs: with more, the pieces' fp32 partials and their merge cost more
// than the idle SMs (measured: 16 heads at N = 2048, 128 pairs, 39 us
// unsplit against 46 us in pieces of up to 8 key tiles).
int fwd_splits(const attn_params* p) {
  if (p->dtype == ATTN_FP32 || fwd_len_order(p)) return 1;
  const long long nb = (static_cast<long long>(p->N) + kTile - 1) / kTile;
  const long long units = (nb + 1) / 2 * p->B * p->H;
  const long long sms = sm_count();
  if (units <= 0 || units >= sms) return 1;
  if (nb < 32 && 2 * units > sms) return 1;
  long long k = (2 * sms + units - 1) / units;
  if (k > nb / kMinPieceTiles) k = nb / kMinPieceTiles;
  if (k > 16) k = 16;
  return k < 1 ? 1 : static_cast<int>(k);
}

// Pieces per key tile in the backward, by the same rule: with fewer key
// tiles (of all key/value heads) than SMs, each key tile's query tiles are
// cut into pieces of at least kMinPieceTiles (counted over the longest walk:
// nb query tiles of each of the H / H_kv query heads), about two units per
// SM, at most 16; otherwise 1.
int bwd_splits(const attn_params* p) {
  const long long nb = (static_cast<long long>(p->N) + kTile - 1) / kTile;
  const long long H_kv = p->H_kv == 0 ? p->H : p->H_kv;
  const long long units = nb * p->B * H_kv;
  const long long sms = sm_count();
  if (units <= 0 || units >= sms) return 1;
  const long long walk = nb * (H_kv > 0 ? p->H / H_kv : 1);
  long long k = (2 * sms + units - 1) / units;
  if (k > walk / kMinPieceTiles) k = walk / kMinPieceTiles;
  if (k > 16) k = 16;
  return k < 1 ? 1 : static_cast<int>(k);
}

WsLayout layout(const attn_params* p, bool bwd) {
  WsLayout L;
  size_t off = kHeaderBytes;
  const size_t nb = (static_cast<size_t>(p->N) + kTile - 1) / kTile;
  const size_t bhn = static_cast<size_t>(p->B) * p->H * p->N;
  if (p->block_mask != nullptr && p->dtype != ATTN_FP32) {
    const size_t masks = static_cast<size_t>(num_masks(p));
    L.list_cnt = off;
    off = round_up(off + masks * nb * sizeof(int32_t), 256);
    L.list_idx = off;
    off = round_up(off + masks * nb * nb * sizeof(uint16_t), 256);
  }
  if (p->dtype == ATTN_FP8_E4M3 && !bwd) {
    L.vt = off;
    const size_t H_kv = static_cast<size_t>(p->H_kv == 0 ? p->H : p->H_kv);
    off = round_up(off + static_cast<size_t>(p->B) * H_kv * p->d * nb * kTile, 256);
  }
  if (p->dtype == ATTN_FP32 && !bwd) {
    const size_t H_kv = static_cast<size_t>(p->H_kv == 0 ? p->H : p->H_kv);
    const size_t qn = static_cast<size_t>(p->B) * p->H * p->N * p->d * sizeof(float);
    const size_t kn = static_cast<size_t>(p->B) * H_kv * p->N * p->d * sizeof(float);
    L.qhi = off;
    off = round_up(off + qn, 256);
    L.qlo = off;
    off = round_up(off + qn, 256);
    L.khi = off;
    off = round_up(off + kn, 256);
    L.klo = off;
    off = round_up(off + kn, 256);
    L.vt32 = off;
    off = round_up(off + static_cast<size_t>(p->B) * H_kv * p->d * nb * kTile * sizeof(float), 256);
  }
  if (!bwd && (L.splits = fwd_splits(p)) > 1) {
    const size_t prows = static_cast<size_t>(L.splits) * p->B * p->H * ((nb + 1) / 2) * 2 * kTile;
    L.part_o = off;
    off = round_up(off + prows * p->d * sizeof(float), 256);
    L.part_l = off;
    off = round_up(off + prows * sizeof(float), 256);
  }
  if (bwd) {
    const size_t bhpad = static_cast<size_t>(p->B) * p->H * nb * kTile;
    L.lse2 = off;
    off = round_up(off + bhpad * sizeof(float), 256);
    L.dsum = off;
    off = round_up(off + bhpad * sizeof(float), 256);
    L.dq_acc = off;
    off = round_up(off + bhn * p->d * sizeof(float), 256);
    if ((L.bwd_splits = bwd_splits(p)) > 1) {
      const size_t prows =
          static_cast<size_t>(L.bwd_splits) * p->B * (p->H_kv == 0 ? p->H : p->H_kv) * nb * kTile;
      L.part_dk = off;
      off = round_up(off + prows * p->d * sizeof(float), 256);
      L.part_dv = off;
      off = round_up(off + prows * p->d * sizeof(float), 256);
    }
  }
  L.total = off;
  return L;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Key/value heads (H_kv = 0 means H) and the key/value strides (all zero
// means the query strides).
int kv_heads(const attn_params* p) { return p->H_kv == 0 ? p->H : p->H_kv; }

bool kv_strides_given(const attn_params* p) {
  return p->kv_stride_b != 0 || p->kv_stride_h != 0 || p->kv_stride_n != 0;
}

void kv_strides(const attn_params* p, int64_t* sb, int64_t* sh, int64_t* sn) {
  const bool own = kv_strides_given(p);
  *sb = own ? p->kv_stride_b : p->stride_b;
  *sh = own ? p->kv_stride_h : p->stride_h;
  *sn = own ? p->kv_stride_n : p->stride_n;
}

attn_status validate(const attn_params* p, bool bwd) {
  if (p == nullptr) return fail(ATTN_ERR_INVALID_ARG, "params is NULL");
  if (p->B < 0 || p->H < 0 || p->N < 0)
    return fail(ATTN_ERR_INVALID_ARG, "negative shape B=%d H=%d N=%d", p->B, p->H, p->N);
  if (p->reserved != 0) return fail(ATTN_ERR_INVALID_ARG, "reserved field must be 0");
  if (p->H_kv < 0 || (p->H > 0 && (kv_heads(p) < 1 || p->H % kv_heads(p) != 0)))
    return fail(ATTN_ERR_INVALID_ARG, "H_kv=%d must divide H=%d", p->H_kv, p->H);
  if (!kv_strides_given(p) && kv_heads(p) != p->H)
    return fail(ATTN_ERR_INVALID_ARG, "H_kv=%d != H=%d needs the key/value strides", p->H_kv,
                p->H);
  if (p->d != 64 && p->d != 128)
    return fail(ATTN_ERR_UNSUPPORTED, "head dim d=%d (supported: 64, 128)", p->d);
  if (p->dtype != ATTN_BF16 && p->dtype != ATTN_FP32 && p->dtype != ATTN_FP8_E4M3)
    return fail(ATTN_ERR_INVALID_ARG, "dtype %d", p->dtype);
  if (bwd && p->dtype != ATTN_BF16)
    return fail(ATTN_ERR_UNSUPPORTED, "backward is implemented for bf16 only");
  if (p->reserved2 != 0) return fail(ATTN_ERR_INVALID_ARG, "reserved2 field must be 0");
  if (p->dtype == ATTN_FP8_E4M3) {
    if (p->d != 128) return fail(ATTN_ERR_UNSUPPORTED, "fp8 forward needs d=128 (got %d)", p->d);
    if (p->dropout_p != 0.f) return fail(ATTN_ERR_UNSUPPORTED, "fp8 forward without dropout only");
    const float ds[3] = {p->q_descale, p->k_descale, p->v_descale};
    for (float x : ds)
      if (!std::isfinite(x) || x < 0.f)
        return fail(ATTN_ERR_INVALID_ARG, "fp8 de-scale factors must be finite and >= 0 (0 = 1)");
  }
  if (!std::isfinite(p->scale) || !(p->scale > 0.f))
    return fail(ATTN_ERR_INVALID_ARG, "scale must be positive and finite (got %g)", p->scale);
  if (!(p->dropout_p >= 0.f && p->dropout_p < 1.f))
    return fail(ATTN_ERR_INVALID_ARG, "dropout_p must be in [0, 1) (got %g)", p->dropout_p);
  if (p->philox_offset >= (1ull << 32))
    return fail(ATTN_ERR_INVALID_ARG, "philox_offset must be < 2^32");
  if (static_cast<int64_t>(p->N) > (int64_t{1} << 30))
    return fail(ATTN_ERR_UNSUPPORTED, "N=%d too large", p->N);
  if (p->block_mask != nullptr) {
    if (p->block_mask_head_stride < 0)
      return fail(ATTN_ERR_INVALID_ARG, "negative block_mask_head_stride");
    if ((p->N + kTile - 1) / kTile > 65535)
      return fail(ATTN_ERR_UNSUPPORTED, "block mask with more than 65535 blocks per side");
    if (num_masks(p) > 65535)
      return fail(ATTN_ERR_UNSUPPORTED, "more than 65535 per-head block masks");
  }
  // elements per 16 bytes (fp8: 16, which also aligns the bf16 output)
  const int64_t align = p->dtype == ATTN_BF16 ? 8 : (p->dtype == ATTN_FP32 ? 4 : 16);
  const int64_t st[3] = {p->stride_b, p->stride_h, p->stride_n};
  for (int i = 0; i < 3; ++i) {
    if (st[i] <= 0 || st[i] % align != 0)
      return fail(ATTN_ERR_INVALID_ARG,
                  "strides must be positive multiples of %lld elements (b=%lld h=%lld n=%lld)",
                  static_cast<long long>(align), static_cast<long long>(p->stride_b),
                  static_cast<long long>(p->stride_h), static_cast<long long>(p->stride_n));
  }
  if (p->stride_n < p->d) return fail(ATTN_ERR_INVALID_ARG, "stride_n < d");
  int64_t kst[3];
  kv_strides(p, &kst[0], &kst[1], &kst[2]);
  for (int i = 0; i < 3; ++i) {
    if (kst[i] <= 0 || kst[i] % align != 0)
      return fail(ATTN_ERR_INVALID_ARG,
                  "key/value strides must be positive multiples of %lld elements "
                  "(b=%lld h=%lld n=%lld)",
                  static_cast<long long>(align), static_cast<long long>(kst[0]),
                  static_cast<long long>(kst[1]), static_cast<long long>(kst[2]));
  }
  if (kst[2] < p->d) return fail(ATTN_ERR_INVALID_ARG, "kv_stride_n < d");
  return ATTN_OK;
}

attn_status check_ptrs(std::initializer_list<const void*> ptrs) {
  int i = 0;
  for (const void* ptr : ptrs) {
    if (ptr == nullptr) return fail(ATTN_ERR_INVALID_ARG, "tensor argument %d is NULL", i);
    if (!aligned16(ptr)) return fail(ATTN_ERR_INVALID_ARG, "tensor argument %d is not 16-byte aligned", i);
    ++i;
  }
  return ATTN_OK;
}

attn_status check_ws(const attn_params* p, bool bwd, const void* ws, size_t ws_bytes) {
  const size_t need = layout(p, bwd).total;
  if (ws == nullptr) return fail(ATTN_ERR_WORKSPACE, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(ATTN_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < need)
    return fail(ATTN_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, need);
  return ATTN_OK;
}

// ------------------------------------------------------------ tensor maps --

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// [B, H, N, d] tensor with element strides; boxes of `box_cols` x `box_rows`.
attn_status make_map(CUtensorMap* map, const void* ptr, CUtensorMapDataType dt, int elem_bytes,
                     int B, int H, int N, int d, int64_t sb, int64_t sh, int64_t sn, int box_cols,
                     int box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(sn * elem_bytes),
                                 static_cast<cuuint64_t>(sh * elem_bytes),
                                 static_cast<cuuint64_t>(sb * elem_bytes)};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = enc(map, dt, 4, const_cast<void*>(ptr), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return ATTN_OK;
}

attn_status make_bf16_map(CUtensorMap* map, const void* ptr, const attn_params* p) {
  return make_map(map, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->B, p->H, p->N, p->d,
                  p->stride_b, p->stride_h, p->stride_n, 64, kTile, CU_TENSOR_MAP_SWIZZLE_128B);
}

// k or v: [B, H_kv, N, d] with the key/value strides
attn_status make_kv_map(CUtensorMap* map, const void* ptr, const attn_params* p) {
  int64_t sb, sh, sn;
  kv_strides(p, &sb, &sh, &sn);
  return make_map(map, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->B, kv_heads(p), p->N, p->d,
                  sb, sh, sn, 64, kTile, CU_TENSOR_MAP_SWIZZLE_128B);
}

float descale_or_one(float x) { return x == 0.f ? 1.f : x; }

attn::MaskArgs mask_args(const attn_params* p, const WsLayout& L, char* ws, bool by_column) {
  attn::MaskArgs m{};
  m.B = p->B;
  m.H = p->H;
  m.N = p->N;
  m.H_kv = kv_heads(p);
  m.kv_group = m.H_kv > 0 ? p->H / m.H_kv : 1;
  m.causal = p->causal != 0;
  m.key_lens = p->key_lens;
  m.nb = (p->N + kTile - 1) / kTile;
  m.block_mask = p->block_mask;
  m.block_mask_head_stride = p->block_mask_head_stride;
  m.mask_per_head = p->block_mask_head_stride != 0;
  if (L.list_idx != 0) {
    m.list_cnt = reinterpret_cast<const int32_t*>(ws + L.list_cnt);
    m.list_idx = reinterpret_cast<const uint16_t*>(ws + L.list_idx);
  }
  (void)by_column;
  // 16-bit uniforms: drop iff u < T, T = min(2^16 - 1, floor(p * 2^16)); the
  // drop rate is exactly T / 2^16 and kept values are scaled by its inverse
  const double p32 = static_cast<double>(p->dropout_p);
  uint32_t T = 0;
  if (p32 > 0.0) {
    const double t = std::floor(p32 * 65536.0);
    T = t >= 65535.0 ? 65535u : static_cast<uint32_t>(t);
  }
  m.drop_threshold = T;
  m.drop_scale = T ? static_cast<float>(65536.0 / (65536.0 - T)) : 1.0f;
  m.seed_lo = static_cast<uint32_t>(p->philox_seed & 0xFFFFFFFFull);
  m.seed_hi = static_cast<uint32_t>(p->philox_seed >> 32);
  m.offset = static_cast<uint32_t>(p->philox_offset);
  m.rk = attn::philox_round_keys(m.seed_lo, m.seed_hi);
  return m;
}

bool empty_problem(const attn_params* p) { return p->B == 0 || p->H == 0 || p->N == 0; }

// Heads per scheduling group, out of `bh` (b, head) units: as many as keep
// `bytes_per_head` of re-read operands within a share of the 129 MB L2.
// Causal work is not grouped: its tiles differ in length, and a group's long
// tiles starting late would leave a tail; longest-first over all heads
// balances better.
int head_group(const attn_params* p, int bh, double bytes_per_head) {
  const double budget = 48.0 * 1024 * 1024;
  if (p->causal) return bh > 0 ? bh : 1;
  const int g = static_cast<int>(budget / (bytes_per_head > 1.0 ? bytes_per_head : 1.0));
  return g < 1 ? 1 : (g > bh ? bh : g);
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace

int attn::record_error(int status, const char* msg) {
  return static_cast<int>(fail(static_cast<attn_status>(status), "%s", msg));
}

extern "C" {

size_t attn_workspace_size(const attn_params* p, int for_backward) {
  if (validate(p, for_backward != 0) != ATTN_OK) return 0;
  return layout(p, for_backward != 0).total;
}

attn_status attn_fwd(const attn_params* p, const void* q, const void* k, const void* v, void* o,
                     float* lse, void* ws, size_t ws_bytes, void* stream) {
  attn_status st = validate(p, false);
  if (st != ATTN_OK) return st;
  if ((st = check_ws(p, false, ws, ws_bytes)) != ATTN_OK) return st;
  if (empty_problem(p)) return ATTN_OK;
  if ((st = check_ptrs({q, k, v, o, lse})) != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  const WsLayout L = layout(p, false);

  attn::FwdArgs a{};
  a.m = mask_args(p, L, w, false);
  a.m.head_group = head_group(p, p->B * p->H, 4.0 * p->N * p->d);   // K and V, bf16
  // key padding makes the units' costs differ by sequence: claim the
  // longest first so that the last claims are short
  a.len_order = fwd_len_order(p) ? 1 : 0;
  if (a.len_order) a.m.head_group = 1;   // each head's pairs together, heads in ranked order
  a.d = p->d;
  a.scale = p->scale;
  a.scale_log2 = p->scale * kLog2e;
  a.o_scale = 1.f;
  a.o = o;
  a.lse = lse;
  a.stride_b = p->stride_b;
  a.stride_h = p->stride_h;
  a.stride_n = p->stride_n;
  kv_strides(p, &a.kv_stride_b, &a.kv_stride_h, &a.kv_stride_n);
  a.status = reinterpret_cast<int*>(w);
  a.sched = reinterpret_cast<int*>(w + kSchedOffset);
  a.timeout_ns = kTimeoutNs;
  a.splits = L.splits;
  a.part_rows = (a.m.nb + 1) / 2 * 2 * kTile;
  if (L.splits > 1) {
    a.part_o = reinterpret_cast<float*>(w + L.part_o);
    a.part_l = reinterpret_cast<float*>(w + L.part_l);
  }

  cudaError_t e;
  if (p->dtype == ATTN_FP32) {
    // TF32 hi / lo parts of q, k and TF32 V^T into the workspace, then the
    // tensor-core forward on them
    const int H_kv = kv_heads(p);
    const int npad = a.m.nb * kTile;
    const int64_t d64 = p->d;
    attn::Tf32Buffers buf{reinterpret_cast<float*>(w + L.qhi), reinterpret_cast<float*>(w + L.qlo),
                          reinterpret_cast<float*>(w + L.khi), reinterpret_cast<float*>(w + L.klo),
                          reinterpret_cast<float*>(w + L.vt32), npad};
    attn::Tf32Maps tm{};
    const int64_t qsh = static_cast<int64_t>(p->N) * d64, ksh = qsh;
    if ((st = make_map(&tm.qhi, buf.qhi, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p->B, p->H, p->N,
                       p->d, p->H * qsh, qsh, d64, 32, kTile, CU_TENSOR_MAP_SWIZZLE_128B)) != ATTN_OK ||
        (st = make_map(&tm.qlo, buf.qlo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p->B, p->H, p->N,
                       p->d, p->H * qsh, qsh, d64, 32, kTile, CU_TENSOR_MAP_SWIZZLE_128B)) != ATTN_OK ||
        (st = make_map(&tm.khi, buf.khi, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p->B, H_kv, p->N,
                       p->d, H_kv * ksh, ksh, d64, 32, kTile, CU_TENSOR_MAP_SWIZZLE_128B)) != ATTN_OK ||
        (st = make_map(&tm.klo, buf.klo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p->B, H_kv, p->N,
                       p->d, H_kv * ksh, ksh, d64, 32, kTile, CU_TENSOR_MAP_SWIZZLE_128B)) != ATTN_OK)
      return st;
    // V^T [B, H_kv, d, N]: rows of npad keys, N of them valid (the rest read as 0)
    const int64_t dn = d64 * npad;
    if ((st = make_map(&tm.vt, buf.vt, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p->B, H_kv, p->d, p->N,
                       H_kv * dn, dn, npad, 32, p->d, CU_TENSOR_MAP_SWIZZLE_128B)) != ATTN_OK)
      return st;
    e = attn::launch_tf32_split(static_cast<const float*>(q), static_cast<const float*>(k),
                                static_cast<const float*>(v), a, buf, s);
    if (e != cudaSuccess) return cuda_fail(e, "fp32 split launch");
    e = attn::launch_fwd_tf32(tm, a, s);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "forward (fp32, tf32 tensor cores) launch");
  }
  attn::TensorMaps tm{};
  const bool fp8 = p->dtype == ATTN_FP8_E4M3;
  const int npad = a.m.nb * kTile;
  if (fp8) {
    // E4M3 q, k with 128 x 128-byte boxes; v goes through V^T in the workspace
    int64_t sb, sh, sn;
    kv_strides(p, &sb, &sh, &sn);
    const int H_kv = kv_heads(p);
    if ((st = make_map(&tm.q, q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p->B, p->H, p->N, p->d,
                       p->stride_b, p->stride_h, p->stride_n, kTile, kTile,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != ATTN_OK)
      return st;
    if ((st = make_map(&tm.k, k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p->B, H_kv, p->N, p->d, sb,
                       sh, sn, kTile, kTile, CU_TENSOR_MAP_SWIZZLE_128B)) != ATTN_OK)
      return st;
    // V^T [B, H_kv, d, N]: rows of npad keys, N of them valid (the rest read as 0)
    const int64_t dn = static_cast<int64_t>(p->d) * npad;
    if ((st = make_map(&tm.v, w + L.vt, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p->B, H_kv, p->d, p->N,
                       static_cast<int64_t>(H_kv) * dn, dn, npad, kTile, kTile,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != ATTN_OK)
      return st;
    const float qs = descale_or_one(p->q_descale), ks = descale_or_one(p->k_descale);
    a.scale = p->scale * qs * ks;
    a.scale_log2 = a.scale * kLog2e;
    a.o_scale = descale_or_one(p->v_descale);
    e = attn::launch_fp8_transpose_v(static_cast<const uint8_t*>(v), sb, sh, sn, p->B, H_kv, p->N,
                                     p->d, npad, reinterpret_cast<uint8_t*>(w + L.vt), s);
    if (e != cudaSuccess) return cuda_fail(e, "fp8 V transpose launch");
  } else {
    if ((st = make_bf16_map(&tm.q, q, p)) != ATTN_OK) return st;
    if ((st = make_kv_map(&tm.k, k, p)) != ATTN_OK) return st;
    if ((st = make_kv_map(&tm.v, v, p)) != ATTN_OK) return st;
  }
  if (p->block_mask != nullptr) {
    e = attn::launch_compact_mask(p->block_mask, p->block_mask_head_stride, num_masks(p), a.m.nb,
                                  0, reinterpret_cast<int32_t*>(w + L.list_cnt),
                                  reinterpret_cast<uint16_t*>(w + L.list_idx), s);
    if (e != cudaSuccess) return cuda_fail(e, "block-mask compaction launch");
  }
  take_stall(attn::kStallFwdSoftmax, &a);
  e = fp8 ? attn::launch_fwd_fp8(tm, a, s) : attn::launch_fwd_bf16(tm, a, s);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "forward launch");
}

}  // extern "C"

namespace {

// Validation and argument block shared by the backward entry points.
attn_status bwd_setup(const attn_params* p, void* ws, size_t ws_bytes, attn::BwdArgs* a,
                      WsLayout* L) {
  attn_status st = validate(p, true);
  if (st != ATTN_OK) return st;
  if ((st = check_ws(p, true, ws, ws_bytes)) != ATTN_OK) return st;
  char* w = static_cast<char*>(ws);
  *L = layout(p, true);
  *a = attn::BwdArgs{};
  a->m = mask_args(p, *L, w, true);
  // a key/value head's CTAs re-read the Q, dO (bf16) and dQ accumulator (fp32)
  // of its group's query heads
  a->m.head_group = head_group(p, p->B * kv_heads(p), 8.0 * a->m.kv_group * p->N * p->d);
  a->d = p->d;
  a->scale = p->scale;
  a->scale_log2 = p->scale * kLog2e;
  a->lse2 = reinterpret_cast<float*>(w + L->lse2);
  a->dsum = reinterpret_cast<float*>(w + L->dsum);
  a->npad = a->m.nb * kTile;
  a->dq_acc = reinterpret_cast<float*>(w + L->dq_acc);
  a->stride_b = p->stride_b;
  a->stride_h = p->stride_h;
  a->stride_n = p->stride_n;
  kv_strides(p, &a->kv_stride_b, &a->kv_stride_h, &a->kv_stride_n);
  a->status = reinterpret_cast<int*>(w);
  a->sched = reinterpret_cast<int*>(w + kSchedOffset);
  a->timeout_ns = kTimeoutNs;
  a->splits = L->bwd_splits;
  a->part_rows = a->npad;
  if (L->bwd_splits > 1) {
    a->part_dk = reinterpret_cast<float*>(w + L->part_dk);
    a->part_dv = reinterpret_cast<float*>(w + L->part_dv);
  }
  return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status attn_bwd_preprocess(const attn_params* p, const void* o, const float* lse,
                                const void* dout, void* ws, size_t ws_bytes, void* stream) {
  attn::BwdArgs a;
  WsLayout L;
  attn_status st = bwd_setup(p, ws, ws_bytes, &a, &L);
  if (st != ATTN_OK) return st;
  if (empty_problem(p)) return ATTN_OK;
  if ((st = check_ptrs({o, lse, dout})) != ATTN_OK) return st;
  a.lse = lse;
  const cudaError_t e = attn::launch_bwd_preprocess(o, dout, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "backward preprocess launch");
}

attn_status attn_bwd_main(const attn_params* p, const void* q, const void* k, const void* v,
                          const void* dout, void* dk, void* dv, void* ws, size_t ws_bytes,
                          void* stream) {
  attn::BwdArgs a;
  WsLayout L;
  attn_status st = bwd_setup(p, ws, ws_bytes, &a, &L);
  if (st != ATTN_OK) return st;
  if (empty_problem(p)) return ATTN_OK;
  if ((st = check_ptrs({q, k, v, dout, dk, dv})) != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  a.dk = dk;
  a.dv = dv;
  attn::TensorMaps tm{};
  if ((st = make_bf16_map(&tm.q, q, p)) != ATTN_OK) return st;
  if ((st = make_kv_map(&tm.k, k, p)) != ATTN_OK) return st;
  if ((st = make_kv_map(&tm.v, v, p)) != ATTN_OK) return st;
  if ((st = make_bf16_map(&tm.dout, dout, p)) != ATTN_OK) return st;
  // fp32 dQ accumulator: contiguous [B, H, N, d]; 32 x 32 boxes, 128-byte swizzle
  const int64_t d64 = p->d;
  if ((st = make_map(&tm.dq_acc, a.dq_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p->B, p->H, p->N,
                     p->d, static_cast<int64_t>(p->H) * p->N * d64,
                     static_cast<int64_t>(p->N) * d64, d64, 32, 32,
                     CU_TENSOR_MAP_SWIZZLE_128B)) != ATTN_OK)
    return st;
  cudaError_t e;
  if (p->block_mask != nullptr) {
    e = attn::launch_compact_mask(p->block_mask, p->block_mask_head_stride, num_masks(p), a.m.nb,
                                  1, reinterpret_cast<int32_t*>(w + L.list_cnt),
                                  reinterpret_cast<uint16_t*>(w + L.list_idx), s);
    if (e != cudaSuccess) return cuda_fail(e, "block-mask compaction launch");
  }
  take_stall(attn::kStallBwdCompute, &a);
  e = attn::launch_bwd_bf16(tm, a, s);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "backward launch");
}

attn_status attn_bwd_dq(const attn_params* p, void* dq, void* ws, size_t ws_bytes, void* stream) {
  attn::BwdArgs a;
  WsLayout L;
  attn_status st = bwd_setup(p, ws, ws_bytes, &a, &L);
  if (st != ATTN_OK) return st;
  if (empty_problem(p)) return ATTN_OK;
  if ((st = check_ptrs({dq})) != ATTN_OK) return st;
  const cudaError_t e = attn::launch_dq_convert(dq, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "dQ conversion launch");
}

attn_status attn_bwd(const attn_params* p, const void* q, const void* k, const void* v,
                     const void* o, const float* lse, const void* dout, void* dq, void* dk,
                     void* dv, void* ws, size_t ws_bytes, void* stream) {
  attn::BwdArgs a;
  WsLayout L;
  attn_status st = bwd_setup(p, ws, ws_bytes, &a, &L);
  if (st != ATTN_OK) return st;
  if (empty_problem(p)) return ATTN_OK;
  if ((st = check_ptrs({q, k, v, o, lse, dout, dq, dk, dv})) != ATTN_OK) return st;
  if ((st = attn_bwd_preprocess(p, o, lse, dout, ws, ws_bytes, stream)) != ATTN_OK) return st;
  if ((st = attn_bwd_main(p, q, k, v, dout, dk, dv, ws, ws_bytes, stream)) != ATTN_OK)
    return st;
  return attn_bwd_dq(p, dq, ws, ws_bytes, stream);
}

// ------------------------------------------------------------ decode step --

namespace {

// Cache keys per split, in multiples of the 64-key tile: enough splits that
// the grid covers every SM several times over (short CTAs balance the
// sequences' different lengths; much shorter ones spend their time in
// set-up).  The warp-MMA kernel (rows <= 16, two CTAs of four streaming
// warps per SM) takes chunks twice as long as the FMA kernel.
int decode_chunk(const attn_params* p, int rows) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 148;
  const int64_t heads = static_cast<int64_t>(p->B) * kv_heads(p);
  const int64_t want = (rows <= 16 ? 4LL : 8LL) * sms;
  int64_t per = heads > 0 ? (static_cast<int64_t>(p->N) * heads + want - 1) / want : p->N;
  per = (per + 63) / 64 * 64;
  if (per < 256) per = 256;
  return static_cast<int>(per);
}

attn_status validate_decode(const attn_params* p, int32_t n_q) {
  attn_status st = validate(p, false);
  if (st != ATTN_OK) return st;
  if (p->dtype != ATTN_BF16) return fail(ATTN_ERR_UNSUPPORTED, "decode is implemented for bf16");
  if (p->dropout_p != 0.f || p->block_mask != nullptr)
    return fail(ATTN_ERR_UNSUPPORTED, "decode takes no dropout and no block mask");
  if (p->key_lens == nullptr) return fail(ATTN_ERR_INVALID_ARG, "decode needs key_lens (cache lengths)");
  if (n_q < 1) return fail(ATTN_ERR_INVALID_ARG, "n_q=%d must be >= 1", n_q);
  if (p->H > 0 && static_cast<int64_t>(p->H / kv_heads(p)) * n_q > attn::kDecMaxRows)
    return fail(ATTN_ERR_UNSUPPORTED, "(H / H_kv) * n_q = %lld exceeds %d",
                static_cast<long long>(p->H / kv_heads(p)) * n_q, attn::kDecMaxRows);
  return ATTN_OK;
}

struct DecodeLayout {
  size_t part_o = 0, part_l = 0, total = 0;
  int chunk = 0, splits = 0;
};

DecodeLayout decode_layout(const attn_params* p, int32_t n_q) {
  DecodeLayout L;
  L.chunk = decode_chunk(p, p->H > 0 ? (p->H / kv_heads(p)) * n_q : 1);
  L.splits = p->N > 0 ? (p->N + L.chunk - 1) / L.chunk : 0;
  const size_t rows = static_cast<size_t>(p->B) * p->H * n_q;
  size_t off = kHeaderBytes;
  L.part_o = off;
  off = round_up(off + static_cast<size_t>(L.splits) * rows * p->d * 4, 256);
  L.part_l = off;
  off = round_up(off + static_cast<size_t>(L.splits) * rows * 4, 256);
  L.total = off;
  return L;
}

}  // namespace

size_t attn_decode_workspace_size(const attn_params* p, int32_t n_q) {
  if (validate_decode(p, n_q) != ATTN_OK) return 0;
  return decode_layout(p, n_q).total;
}

attn_status attn_decode(const attn_params* p, int32_t n_q, const void* q, const void* k,
                        const void* v, void* o, float* lse, void* ws, size_t ws_bytes,
                        void* stream) {
  attn_status st = validate_decode(p, n_q);
  if (st != ATTN_OK) return st;
  const DecodeLayout L = decode_layout(p, n_q);
  if (ws == nullptr) return fail(ATTN_ERR_WORKSPACE, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(ATTN_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < L.total)
    return fail(ATTN_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, L.total);
  if (empty_problem(p)) return ATTN_OK;
  if ((st = check_ptrs({q, k, v, o, lse})) != ATTN_OK) return st;
  char* w = static_cast<char*>(ws);
  attn::DecodeArgs a{};
  a.m = mask_args(p, WsLayout{}, w, false);
  a.d = p->d;
  a.n_q = n_q;
  a.rows = (p->H / kv_heads(p)) * n_q;
  a.chunk = L.chunk;
  a.splits = L.splits;
  a.scale_log2 = p->scale * kLog2e;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.stride_b = p->stride_b;
  a.stride_h = p->stride_h;
  a.stride_n = p->stride_n;
  a.part_o = reinterpret_cast<float*>(w + L.part_o);
  a.part_l = reinterpret_cast<float*>(w + L.part_l);
  a.status = reinterpret_cast<int*>(w);
  a.timeout_ns = kTimeoutNs;
  // k, v with boxes of the tile the chosen kernel streams
  attn::TensorMaps tm{};
  int64_t sb, sh, sn;
  kv_strides(p, &sb, &sh, &sn);
  const int box_rows = a.rows <= attn::kDecMmaRows ? attn::kDecMmaKeys : 64;
  if ((st = make_map(&tm.k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->B, kv_heads(p), p->N,
                     p->d, sb, sh, sn, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B)) != ATTN_OK)
    return st;
  if ((st = make_map(&tm.v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->B, kv_heads(p), p->N,
                     p->d, sb, sh, sn, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B)) != ATTN_OK)
    return st;
  const cudaError_t e = attn::launch_decode(tm, o, lse, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "decode launch");
}

attn_status attn_debug_stall(int32_t which, uint64_t limit_ns) {
  if (which != ATTN_STALL_NONE && which != ATTN_STALL_FWD_SOFTMAX &&
      which != ATTN_STALL_BWD_COMPUTE)
    return fail(ATTN_ERR_INVALID_ARG, "unknown stall %d", which);
  if (limit_ns < 1000000ull) limit_ns = 1000000ull;          // 1 ms
  if (limit_ns > kTimeoutNs) limit_ns = kTimeoutNs;          // 2 s
  g_stall = which;
  g_stall_limit_ns = limit_ns;
  return ATTN_OK;
}

attn_status attn_check(void* ws, void* stream) {
  if (ws == nullptr) {   // the built-in scratch of attn_bwd_noalloc on this device
    const attn_status st = static_cast<attn_status>(attn::builtin_scratch(&ws));
    if (st != ATTN_OK) return st;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int words[2] = {0, 0};
  if ((e = cudaMemcpy(words, ws, sizeof(words), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "status read");
  if (words[0] == 0) return ATTN_OK;
  if ((e = cudaMemset(ws, 0, sizeof(words))) != cudaSuccess) return cuda_fail(e, "status clear");
  return fail(static_cast<attn_status>(words[0]), "device status %d at wait site %d", words[0],
              words[1]);
}

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device wait timed out";
    case ATTN_ERR_WORKSPACE: return "bad workspace";
  }
  return "unknown status";
}

const char* attn_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
