// lt_topk_kernels.cu -- the per-row top-k kernel.
#include "lt_kernels.cuh"
#include "lt_launch.h"

namespace lt {

// One CTA (or one cluster of CTAs) per row: select the top K = min(k, L)
// positions and write them ordered by (score desc, index asc). kOne: every
// CTA's slice is a single register round (the planner guarantees it).
// S: the score type (float, or uint16_t holding bf16 bits). kHint: rows
// start from the output of an earlier row (batches of single-CTA rows).
template <int T, int U, bool kOne, class S, bool kHint = false>
__global__ void __launch_bounds__(T, (T <= 256 ? 3 : 1)) topk_kernel(Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  using G = Geo<T, U, 4>;
  RowT<S> R;
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
    // Batches of single-CTA rows (256 threads): start from the (k/2)-th and
    // k-th values of the row hint_rows earlier (two waves of CTAs, so almost
    // surely finished; see Hint). Another CTA may still be writing them: they
    // are a guess the filter checks; a miss takes the exact path. Whether a
    // row is hinted depends only on values every thread reads alike (the
    // row's length, the launch), so all warps take the same branch.
    if constexpr (kHint) {
      Hint hint = {};
      const bool hinted = p.out_val != nullptr && K == (uint32_t)p.k && p.k >= 2 && R.row >= p.hint_rows &&
                          R.L > (int64_t)(p.cap / 2);
      if (hinted) {
        const float* prev = p.out_val + (R.row - p.hint_rows) * (int64_t)p.k;
        hint.hi = ld_relaxed(prev + p.k / 2 - 1);
        hint.lo = ld_relaxed(prev + p.k - 1);
      }
      exact = select_stage<T, U, 4, false>(R, p, va, na, vb, nb, false, K, R.L, p.row_stride, KeepAll{}, true,
                                           &intact, &Tc, 0, hinted ? &hint : nullptr);
    } else {
      exact = select_stage<T, U, 4, false>(R, p, va, na, vb, nb, false, K, R.L, p.row_stride, KeepAll{}, true,
                                           &intact, &Tc, 0);
    }
  }
  output_positions<T>(R, p, exact, Tc, K, p.row_stride, true);
  wait_init(R);
}

template <class S>
const void* topk_ptr(int threads, bool one_round) {
  if (threads == 256)
    return one_round ? reinterpret_cast<const void*>(&topk_kernel<256, 4, true, S>)
                     : reinterpret_cast<const void*>(&topk_kernel<256, 4, false, S>);
  if (threads == 512)
    return one_round ? reinterpret_cast<const void*>(&topk_kernel<512, 8, true, S>)
                     : reinterpret_cast<const void*>(&topk_kernel<512, 8, false, S>);
  return nullptr;
}

const void* topk_kernel_ptr(int threads, bool one_round, bool bf16) {
  return bf16 ? topk_ptr<uint16_t>(threads, one_round) : topk_ptr<float>(threads, one_round);
}

const void* topk_hint_kernel_ptr(bool bf16) {
  return bf16 ? reinterpret_cast<const void*>(&topk_kernel<256, 4, false, uint16_t, true>)
              : reinterpret_cast<const void*>(&topk_kernel<256, 4, false, float, true>);
}

const void* blocked_kernel_ptr(int threads, int block, bool bf16) {
  if (threads == 256) return bf16 ? blocked_kernel_ptr_of<256, uint16_t>(block) : blocked_kernel_ptr_of<256, float>(block);
  if (threads == 512) return bf16 ? blocked_kernel_ptr_of<512, uint16_t>(block) : blocked_kernel_ptr_of<512, float>(block);
  return nullptr;
}

// Positions one CTA covers in a single register round.
int64_t topk_round_positions(int threads) { return threads == 256 ? 256 * 4 * 4 : 512 * 8 * 4; }

}  // namespace lt
