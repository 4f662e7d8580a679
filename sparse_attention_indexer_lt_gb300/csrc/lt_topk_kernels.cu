// lt_topk_kernels.cu -- the per-row top-k kernel.
#include "lt_kernels.cuh"
#include "lt_launch.h"

namespace lt {

// One CTA (or one cluster of CTAs) per row: select the top K = min(k, L)
// positions and write them ordered by (score desc, index asc). kOne: every
// CTA's slice is a single register round (the planner guarantees it).
template <int T, int U, bool kOne>
__global__ void __launch_bounds__(T, (T <= 256 ? 3 : 1)) topk_kernel(Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  using G = Geo<T, U, 4>;
  Row R;
  stamp(p, kTrStart);
  grid_dependents_launch();
  setup_row<T, U, 4>(R, p, smem);
  float4 va[U];
  int na[G::kSlots];
  const uint32_t K = (uint32_t)(R.L < (int64_t)p.k ? R.L : (int64_t)p.k);
  uint64_t Tc;
  bool exact;
  if constexpr (kOne) {
    exact = select_one<T, U, 4>(R, p, va, na, K, &Tc);
  } else {
    float4 vb[U];
    int nb[G::kSlots];
    bool intact;
    exact = select_stage<T, U, 4, false>(R, p, va, na, vb, nb, false, K, R.L, p.row_stride, KeepAll{}, true,
                                         &intact, &Tc, 0);
  }
  output_positions<T>(R, p, exact, Tc, K, p.row_stride, true);
  wait_init(R);
}

const void* topk_kernel_ptr(int threads, bool one_round) {
  if (threads == 256)
    return one_round ? reinterpret_cast<const void*>(&topk_kernel<256, 4, true>)
                     : reinterpret_cast<const void*>(&topk_kernel<256, 4, false>);
  if (threads == 512)
    return one_round ? reinterpret_cast<const void*>(&topk_kernel<512, 8, true>)
                     : reinterpret_cast<const void*>(&topk_kernel<512, 8, false>);
  return nullptr;
}

// Positions one CTA covers in a single register round.
int64_t topk_round_positions(int threads) { return threads == 256 ? 256 * 4 * 4 : 512 * 8 * 4; }

}  // namespace lt
