// lt_stream_kernels.cu -- the streamed, persistent top-k kernel.
#include "lt_launch.h"
#include "lt_stream.cuh"

namespace lt {

// A cluster of C CTAs (C = 1 without cluster launch) serves rows
// cluster_id, cluster_id + clusters, ...; every CTA of the cluster walks the
// same rows, each over its own slice.
template <int T, int UC, int UR, int kMinCtas>
__global__ void __launch_bounds__(T, kMinCtas) stream_kernel(Params p) {
  using SG = SGeo<T, UC>;
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t ns = (uint32_t)p.ring_stages;
  const StreamLayout sl = make_stream_layout(p.clustered != 0, (uint32_t)p.cap, (uint32_t)p.sel_cap, ns,
                                             (uint32_t)SG::kChunk * 4u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + sl.bars);
  float* ring = reinterpret_cast<float*>(smem + sl.ring);
  const uint32_t nclus = p.clustered ? cluster_size() : 1u;
  const uint32_t rank = p.clustered ? cluster_rank() : 0u;
  const int64_t first = (int64_t)(blockIdx.x / nclus);
  const int64_t step = (int64_t)(gridDim.x / nclus);

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < ns; ++i) mbar_init(&bars[i], 1);
    mbar_fence_init();
  }
  grid_dependents_launch();
  // the producer reads lengths and scores, which the previous kernel may write
  grid_dependency_wait();
  Prod& P = *reinterpret_cast<Prod*>(smem + sl.prod);  // thread 0 only
  if (threadIdx.x == 0) {
    P.scores = static_cast<const float*>(p.scores);
    P.lengths = p.lengths;
    P.row_stride = p.row_stride;
    P.rows = p.rows;
    P.step = step;
    P.bars = bars;
    P.ring = ring;
    P.ns = ns;
    P.rank = rank;
    P.nclus = nclus;
    P.seq = 0;
    P.released = 0;
    P.skip_last = p.stall_polls > 0;
    prod_row<T, UC>(P, first);
    produce<T, UC>(P, ns);
  }

  uint32_t g0 = 0;
  for (int64_t row = first; row < p.rows; row += step) {
    __syncthreads();  // the previous row is done with shared memory
    Row R;
    setup_row<T, UR, 4>(R, p, smem, row);
    // phase timestamps of one row per CTA: the third (steady state) when the
    // CTA has three rows, else its last
    const int64_t traced = first + 2 * step < p.rows ? first + 2 * step
                                                     : first + (p.rows - 1 - first) / step * step;
    if (row != traced) R.trace = nullptr;
    stamp(R, kTrStart);
    int64_t b, e, per;
    slice_of(p, row, rank, nclus, &b, &e, &per);
    const int rounds = chunk_rounds<T, UC>(e - b);
    const int rounds_max = chunk_rounds<T, UC>(per);
    bool late = false;
    stream_row<T, UC, UR>(R, p, bars, ring, ns, g0, rounds, rounds_max, P, late);
    if (__syncthreads_or(late ? 1 : 0)) bump(p, R, kCntTimeout);
    g0 += (uint32_t)rounds;
    wait_init(R);
  }
  // Every chunk issued was waited on. Stages whose wait gave up may still have
  // copies in flight: give them a bounded chance to land before the CTA exits.
  __syncthreads();
  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < ns && i < g0; ++i) {
      const uint32_t seq = g0 - 1u - i;
      (void)ring_wait(bars, ns, seq, p.stall_polls > 0 ? (uint32_t)p.stall_polls : kWaitPolls);
    }
  }
  __syncthreads();
}

const void* stream_kernel_ptr(int threads) {
  if (threads == 256) return reinterpret_cast<const void*>(&stream_kernel<256, 4, 4, 3>);
  if (threads == 512) return reinterpret_cast<const void*>(&stream_kernel<512, 2, 4, 2>);
  return nullptr;
}

}  // namespace lt
