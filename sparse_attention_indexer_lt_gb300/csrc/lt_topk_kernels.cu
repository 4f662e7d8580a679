// lt_topk_kernels.cu -- the per-row top-k kernel.
#include "lt_kernels.cuh"
#include "lt_launch.h"

namespace lt {

// One CTA (or one cluster of CTAs) per row: select the top K = min(k, L)
// positions and write them ordered by (score desc, index asc).
__global__ void __launch_bounds__(kThreads, 2) topk_kernel(Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  Row R;
  setup_row<4>(R, p, smem);
  float4 va[kVecPerRound], vb[kVecPerRound];
  int na[Geo<4>::kSlots], nb[Geo<4>::kSlots];
  const uint32_t K = (uint32_t)(R.L < (int64_t)p.k ? R.L : (int64_t)p.k);
  bool intact;
  select_stage<4, false>(R, p, va, na, vb, nb, false, K, R.L, p.row_stride, KeepAll{}, &intact, true);
  write_ordered(R, p, K, (uint32_t)p.k, [&R](uint32_t idx) { return in_slice(R, idx); });
  finish_row(R);
}

const void* topk_kernel_ptr() { return reinterpret_cast<const void*>(&topk_kernel); }

}  // namespace lt
