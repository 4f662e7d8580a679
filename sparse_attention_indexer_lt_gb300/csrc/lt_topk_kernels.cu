// lt_topk_kernels.cu -- the per-row top-k kernel.
#include "lt_kernels.cuh"
#include "lt_launch.h"

namespace lt {

// One CTA (or one cluster of CTAs) per row: select the top K = min(k, L)
// positions and write them ordered by (score desc, index asc).
template <int T, int U>
__global__ void __launch_bounds__(T, (T <= 256 ? 3 : 1)) topk_kernel(Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  using G = Geo<T, U, 4>;
  Row R;
  stamp(p, kTrStart);
  setup_row<T, U, 4>(R, p, smem);
  float4 va[U], vb[U];
  int na[G::kSlots], nb[G::kSlots];
  const uint32_t K = (uint32_t)(R.L < (int64_t)p.k ? R.L : (int64_t)p.k);
  bool intact;
  uint64_t Tc;
  const bool exact = select_stage<T, U, 4, false>(R, p, va, na, vb, nb, false, K, R.L, p.row_stride,
                                                  KeepAll{}, true, &intact, &Tc, 0);
  output_positions<T>(R, p, exact, Tc, K, p.row_stride);
  wait_init(R);
}

const void* topk_kernel_ptr(int threads) {
  if (threads == 256) return reinterpret_cast<const void*>(&topk_kernel<256, 4>);
  if (threads == 512) return reinterpret_cast<const void*>(&topk_kernel<512, 8>);
  return nullptr;
}

}  // namespace lt
