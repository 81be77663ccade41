// Fused attention forward for fp32 inputs and outputs, computed in fp32 on
// the FMA pipes.
//
// Same method as the bf16 kernel (the FlashAttention tiled forward with the
// online-softmax statistics of the paper summary's "Theo dõi Softmax tăng
// dần" section), in its plainest form: each thread owns one query row, key
// and value tiles of 64 rows are staged in shared memory, and the row keeps
// its running max m, exp-sum l and un-normalised output in registers.  The
// fp32 path exists for fp32 callers and small problems; the tensor-core
// path is the bf16 one.
#include "attn_kernels.cuh"
#include "philox.cuh"

namespace attn {
namespace {

constexpr int kRows = 64;   // query rows per CTA (one per thread)
constexpr int kKeys = 64;   // keys per shared-memory tile
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
constexpr int fp32_smem_bytes() {
  return (kRows * (D + 1) + 2 * kKeys * D + kRows * (kKeys + 1)) * 4;
}

template <int D, bool DROPOUT>
__global__ void __launch_bounds__(kRows) fwd_fp32_kernel(const float* __restrict__ q,
                                                        const float* __restrict__ k,
                                                        const float* __restrict__ v,
                                                        const FwdArgs a) {
  extern __shared__ float sm[];
  float* sQ = sm;                        // [kRows][D + 1]
  float* sK = sQ + kRows * (D + 1);      // [kKeys][D]
  float* sV = sK + kKeys * D;            // [kKeys][D]
  float* sS = sV + kKeys * D;            // [kRows][kKeys + 1] scores of each row
  const MaskArgs& m = a.m;
  const int BH = m.B * m.H;
  const int nq = (m.N + kRows - 1) / kRows;
  const int qt = nq - 1 - static_cast<int>(blockIdx.x / BH);
  const int bh = static_cast<int>(blockIdx.x % BH);
  const int b = bh / m.H, h = bh - b * m.H;
  const int q0 = qt * kRows;
  const int t = threadIdx.x;
  const int qi = q0 + t;
  const int64_t head = b * a.stride_b + h * a.stride_h;
  // the key/value head of query head h
  const int64_t kv_head = b * a.kv_stride_b + (h / m.kv_group) * a.kv_stride_h;
  const float* qrow = sQ + t * (D + 1);
  float* srow = sS + t * (kKeys + 1);

  for (int e = t; e < kRows * D; e += kRows) {
    const int r = e / D, c = e - r * D;
    sQ[r * (D + 1) + c] = (q0 + r < m.N) ? q[head + static_cast<int64_t>(q0 + r) * a.stride_n + c] : 0.f;
  }
  int limit = m.N;
  if (m.key_lens != nullptr) limit = min(max(m.key_lens[b], 0), m.N);
  int kend = limit;
  if (m.causal) kend = min(kend, q0 + kRows);
  const uint8_t* bmask =
      m.block_mask ? m.block_mask + (m.block_mask_head_stride ? bh * m.block_mask_head_stride : 0)
                   : nullptr;

  float o[D];
#pragma unroll
  for (int c = 0; c < D; ++c) o[c] = 0.f;
  float mrow = -INFINITY, lrow = 0.f;

  for (int kv0 = 0; kv0 < kend; kv0 += kKeys) {
    if (bmask && !bmask[static_cast<int64_t>(q0 / kTile) * m.nb + kv0 / kTile]) continue;
    __syncthreads();
    for (int e = t; e < kKeys * D; e += kRows) {
      const int r = e / D, c = e - r * D;
      const bool in = kv0 + r < m.N;
      const int64_t g = kv_head + static_cast<int64_t>(kv0 + r) * a.kv_stride_n + c;
      sK[e] = in ? k[g] : 0.f;
      sV[e] = in ? v[g] : 0.f;
    }
    __syncthreads();
    float mt = -INFINITY;
    for (int j = 0; j < kKeys; ++j) {
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 16
      for (int c = 0; c < D; c += 2) {
        acc0 = fmaf(qrow[c], sK[j * D + c], acc0);
        acc1 = fmaf(qrow[c + 1], sK[j * D + c + 1], acc1);
      }
      const int kj = kv0 + j;
      const bool allowed = kj < limit && (!m.causal || kj <= qi);
      const float sj = allowed ? (acc0 + acc1) * a.scale : -INFINITY;
      srow[j] = sj;
      mt = fmaxf(mt, sj);
    }
    const float m_new = fmaxf(mrow, mt);
    if (m_new == -INFINITY) continue;          // nothing allowed in this tile for this row
    const float alpha = exp2f((mrow - m_new) * kLog2e);
    lrow *= alpha;
#pragma unroll
    for (int c = 0; c < D; ++c) o[c] *= alpha;
    mrow = m_new;
    uint32_t keep = 0xFFu;
    for (int j = 0; j < kKeys; ++j) {
      if constexpr (DROPOUT) {
        if ((j & 7) == 0)
          keep = dropout_keep8(static_cast<uint32_t>((kv0 + j) / 8), static_cast<uint32_t>(qi),
                               static_cast<uint32_t>(bh), m.offset, m.rk, m.drop_threshold);
      }
      const float p = exp2f((srow[j] - m_new) * kLog2e);
      lrow += p;
      const float pd = ((keep >> (j & 7)) & 1u) ? p : 0.f;
#pragma unroll
      for (int c = 0; c < D; ++c) o[c] = fmaf(pd, sV[j * D + c], o[c]);
    }
  }
  if (qi < m.N) {
    const bool live = lrow > 0.f;
    const float inv = live ? m.drop_scale / lrow : 0.f;
    float* orow = static_cast<float*>(a.o) + head + static_cast<int64_t>(qi) * a.stride_n;
#pragma unroll
    for (int c = 0; c < D; ++c) orow[c] = o[c] * inv;
    a.lse[static_cast<int64_t>(bh) * m.N + qi] = live ? mrow + logf(lrow) : -INFINITY;
  }
}

template <int D, bool DROP>
cudaError_t launch_one(const float* q, const float* k, const float* v, const FwdArgs& a,
                       cudaStream_t s) {
  constexpr int smem = fp32_smem_bytes<D>();
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(fwd_fp32_kernel<D, DROP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const unsigned grid = static_cast<unsigned>((a.m.N + kRows - 1) / kRows) * a.m.B * a.m.H;
  fwd_fp32_kernel<D, DROP><<<grid, kRows, smem, s>>>(q, k, v, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp32(const float* q, const float* k, const float* v, const FwdArgs& a,
                            cudaStream_t s) {
  const bool drop = a.m.drop_threshold != 0;
  if (a.d == 64) return drop ? launch_one<64, true>(q, k, v, a, s) : launch_one<64, false>(q, k, v, a, s);
  return drop ? launch_one<128, true>(q, k, v, a, s) : launch_one<128, false>(q, k, v, a, s);
}

}  // namespace attn
