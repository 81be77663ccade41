// Block-mask compaction for block-sparse attention.
//
// The block-sparse extension (FlashAttention paper summary, "Mở rộng:
// Block-Sparse FlashAttention"; azimuth.plus explainer, block-sparse
// section) restricts the computation to the nonzero blocks of a mask
// M in {0,1}^{N/128 x N/128} and skips zero blocks with no load, no compute
// and no write.  This kernel turns the dense uint8 mask into sorted lists:
// by row (the key tiles each query tile visits, forward) or by column (the
// query tiles each key tile visits, backward).  One warp per row/column; the
// ballot prefix keeps the indices in ascending order.
#include "attn_kernels.cuh"

namespace attn {
namespace {

__global__ void __launch_bounds__(32) compact_mask_kernel(const uint8_t* __restrict__ mask,
                                                          int64_t head_stride, int nb,
                                                          int by_column, int32_t* __restrict__ cnt,
                                                          uint16_t* __restrict__ idx) {
  const int t = blockIdx.x;      // row (or column) of the block mask
  const int mi = blockIdx.y;     // which mask (0 when shared by every head)
  const uint8_t* mk = mask + static_cast<int64_t>(mi) * head_stride;
  uint16_t* out = idx + (static_cast<size_t>(mi) * nb + t) * nb;
  const uint32_t lane = threadIdx.x;
  int total = 0;
  for (int base = 0; base < nb; base += 32) {
    const int u = base + static_cast<int>(lane);
    bool on = false;
    if (u < nb)
      on = (by_column ? mk[static_cast<size_t>(u) * nb + t] : mk[static_cast<size_t>(t) * nb + u]) != 0;
    const uint32_t bal = __ballot_sync(0xffffffffu, on);
    if (on) out[total + __popc(bal & ((1u << lane) - 1u))] = static_cast<uint16_t>(u);
    total += __popc(bal);
  }
  if (lane == 0) cnt[static_cast<size_t>(mi) * nb + t] = total;
}

}  // namespace

cudaError_t launch_compact_mask(const uint8_t* mask, int64_t head_stride, int masks, int nb,
                                int by_column, int32_t* cnt, uint16_t* idx, cudaStream_t s) {
  compact_mask_kernel<<<dim3(nb, masks), 32, 0, s>>>(mask, head_stride, nb, by_column, cnt, idx);
  return cudaGetLastError();
}

}  // namespace attn
