// lt_blocked.cuh -- the two-level (candidate-restricted) top-k kernel.
#pragma once

#include "lt_kernels.cuh"

namespace lt {

// Stage A's kept blocks straight from the candidate segments, which the
// exchange replicated in every CTA of the cluster. 1024 linear buckets over
// the candidates' key range [lo, hi] locate the bucket b* holding the KA-th
// composite; one more pass keeps every item above b* and stages the items of
// b*, whose exact rank among themselves decides the rest. On the way each CTA
// marks its own kept blocks in a bitmap and counts the kept blocks of the
// lower-ranked slices (a block belongs to the slice holding its id: slices
// hold whole blocks), then writes its own kept ids in ascending order after
// them. Expects the bucket counts (R.hist) zeroed and a barrier passed since,
// and this CTA's slice to hold at most 32 * kBins blocks. Returns false, having
// written nothing, when b* holds more than kMaxBucket items.
template <int T, int W>
__device__ __forceinline__ bool kept_from_segments(RowCore& R, const Params& p, uint32_t KA, uint32_t lo,
                                                   uint32_t hi) {
  constexpr int NB = kOutBuckets;
  constexpr int BPT = NB / T;
  Misc* m = R.m;
  const uint32_t b0s = (uint32_t)(R.begin / W), b1s = (uint32_t)((R.end + W - 1) / W);
  const uint32_t words = (b1s - b0s + 31u) >> 5;
  uint32_t* bits = R.aux;
  for (uint32_t i = threadIdx.x; i < words; i += T) bits[i] = 0u;
  if (threadIdx.x == 0) {
    m->aux[2] = 0u;  // items staged from b*
    m->aux[6] = 0u;  // kept blocks of the lower-ranked slices
  }
  const float scale = (float)NB / ((float)(hi - lo) + 1.0f);
  auto bucket = [lo, scale](uint32_t key) -> uint32_t { return out_bucket(key, lo, scale); };
  for_each_cand<T>(R, [&](uint2 e) { atomicAdd(&R.hist[bucket(e.x)], 1u); });
  __syncthreads();
  uint32_t v[BPT];
#pragma unroll
  for (int j = 0; j < BPT; ++j) v[j] = R.hist[threadIdx.x * BPT + j];
  uint32_t tot = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) tot += v[j];
  uint32_t a = block_suffix_excl<T>(tot, m);
#pragma unroll
  for (int j = BPT - 1; j >= 0; --j) {
    if (a < KA && KA <= a + v[j]) {
      m->res_digit = threadIdx.x * BPT + j;
      m->res_above = a;
      m->res_cnt = v[j];
    }
    a += v[j];
  }
  __syncthreads();
  const uint32_t bstar = m->res_digit, above = m->res_above, cstar = m->res_cnt;
  if (cstar > (uint32_t)kMaxBucket) return false;
  uint32_t before = 0;
  auto keep = [&](uint32_t id) {
    if (id < b0s) ++before;
    else if (id < b1s) atomicOr(&bits[(id - b0s) >> 5], 1u << ((id - b0s) & 31u));
  };
  for_each_cand<T>(R, [&](uint2 e) {
    const uint32_t b = bucket(e.x);
    if (b > bstar) {
      keep(e.y);
    } else if (b == bstar) {
      const uint32_t pos = atomicAdd(&m->aux[2], 1u);
      if (pos < R.stage_cap) R.stage[pos] = composite(e.x, e.y);
    }
  });
  __syncthreads();
  const uint32_t need = KA - above;  // 1 <= need <= cstar
  for (uint32_t i = threadIdx.x; i < cstar; i += T) {
    const uint64_t c = R.stage[i];
    uint32_t r = 0;
    for (uint32_t j = 0; j < cstar; ++j) r += (R.stage[j] > c) ? 1u : 0u;
    if (r < need) keep(~(uint32_t)c);
  }
  before = __reduce_add_sync(kFull, before);
  if (lane_id() == 0 && before != 0u) atomicAdd(&m->aux[6], before);
  __syncthreads();
  int32_t* ob = p.out_blocks + R.row * (int64_t)p.k_blocks;
  const uint32_t wpt = (words + T - 1) / T;
  const uint32_t w0 = threadIdx.x * wpt;
  const uint32_t w1 = min(w0 + wpt, words);
  uint32_t cnt = 0;
  for (uint32_t w = w0; w < w1; ++w) cnt += (uint32_t)__popc(bits[w]);
  uint32_t out = m->aux[6] + block_prefix_excl<T>(cnt, m);
  for (uint32_t w = w0; w < w1; ++w)
    for (uint32_t x = bits[w]; x; x &= x - 1u) ob[out++] = (int32_t)(b0s + 32u * w + (uint32_t)(__ffs(x) - 1));
  if (R.rank == 0) {
    for (uint32_t j = KA + threadIdx.x; j < (uint32_t)p.k_blocks; j += T) ob[j] = -1;
  }
  return true;
}

// The roles other than stage A run out of line: a CTA runs its row's code
// once, fetching it as it goes, and with these bodies inlined ahead of stage
// A the side-by-side launch stalled longer on instruction fetch (cold
// launch 30.9 against 25.9 us; back to back 20.3 against 20.2 us, and 19.8
// with the general tail below out of line as well).
//
// The plain top-k of a row (group 1 of the side-by-side launch): items are
// single positions, so it runs on four-position slots (the top-k kernel's
// streaming filter: paired register rounds, compare masks without per-slot
// bookkeeping).
template <int T, int U, class S>
__device__ __noinline__ void blocked_plain_row(const Params p, unsigned char* smem, int64_t row) {
  RowT<S> R;
  float4 va[U], vb[U];
  setup_row<T, U, 4>(R, p, smem, row);
  int na4[U], nb4[U];
  const uint32_t K = (uint32_t)(R.L < (int64_t)p.k ? R.L : (int64_t)p.k);
  bool intact;
  uint64_t Tc;
  const bool exact = select_stage<T, U, 4, false>(R, p, va, na4, vb, nb4, false, K, R.L, p.row_stride, KeepAll{},
                                                  true, &intact, &Tc, kTrStageB);
  output_positions<T>(R, p, exact, Tc, K, p.row_stride, true);
  wait_init(R);
}

// Stage B over a given block list (role 3: the listed candidates of a later
// layer when the listed kernel does not apply).
template <int T, int U, int W, class S>
__device__ __noinline__ void blocked_listed_row(RowT<S> R, const Params p) {
  using G = Geo<T, U, W>;
  Misc* m = R.m;
  float4 va[U], vb[U];
  int na[G::kSlots], nb[G::kSlots];
  // a bitmap of this CTA's slice of blocks (slices hold whole blocks) in the
  // output's bucket-start area (unused until the ordered output); the
  // listed positions of the row are summed over the cluster
  const int64_t nblocks = (R.L + W - 1) / W;
  const int64_t b0 = R.begin / W, b1 = (R.end + W - 1) / W;
  const uint32_t words = (uint32_t)((b1 - b0 + 31) >> 5);  // <= kBins: checked by the host
  uint32_t* bits = R.aux;
  for (uint32_t i = threadIdx.x; i < words; i += T) bits[i] = 0u;
  __syncthreads();
  const int32_t* listed = p.cand_blocks + R.row * (int64_t)p.n_cand;
  for (int32_t j = (int32_t)threadIdx.x; j < p.n_cand; j += T) {
    const int64_t b = listed[j];
    if (b >= b0 && b < b1) atomicOr(&bits[(b - b0) >> 5], 1u << ((b - b0) & 31));
  }
  __syncthreads();
  uint32_t cnt = 0;
  for (uint32_t i = threadIdx.x; i < words; i += T) cnt += (uint32_t)__popc(bits[i]);
  const uint32_t nlisted = block_sum<T>(cnt, m);
  const int64_t lastb = nblocks - 1;  // may be partial: its positions past L do not count
  const bool last = lastb >= b0 && lastb < b1 && ((bits[(lastb - b0) >> 5] >> ((lastb - b0) & 31)) & 1u) != 0u;
  int64_t ncand = (int64_t)nlisted * W - (last ? nblocks * W - R.L : 0);
  if (R.nclus > 1) {
    // every CTA adds its count into every peer (zeroed before the start-up barrier)
    wait_init(R);
    if (threadIdx.x < R.nclus)
      dsmem_red_add(peer_addr(smem_addr(&m->aux[7]), threadIdx.x), (uint32_t)ncand);
    cluster_sync();
    ncand = (int64_t)m->aux[7];
  }
  const uint32_t K = (uint32_t)(ncand < (int64_t)p.k ? ncand : (int64_t)p.k);
  bool intact;
  uint64_t Tc;
  const bool exact = select_stage<T, U, W, false>(R, p, va, na, vb, nb, false, K, ncand, p.row_stride,
                                                  KeepListed<T, U, W>{bits, b0, words * 32u}, true, &intact,
                                                  &Tc, 0);
  output_positions<T>(R, p, exact, Tc, K, p.row_stride, true);
  wait_init(R);
}

// Kept blocks off the fast path (the exact stage A, a bucket past kMaxBucket
// items, or stage A and B in turn), then stage B when both stages run in
// turn. Out of line like the other rare paths; the two register rounds come
// along for a stage B that reuses them.
template <int T, int U, int W, class S>
__device__ __noinline__ void blocked_general_tail(RowT<S> R, const Params p, int role, uint64_t TA, uint32_t KA,
                                                  bool intact, RoundRegs<U, Geo<T, U, W>::kSlots> ra,
                                                  RoundRegs<U, Geo<T, U, W>::kSlots> rb) {
  Misc* m = R.m;
  float4 (&va)[U] = ra.v;
  float4 (&vb)[U] = rb.v;
  int (&na)[Geo<T, U, W>::kSlots] = ra.n;
  int (&nb)[Geo<T, U, W>::kSlots] = rb.n;
  // ---- kept block ids in ascending order: this CTA's own kept blocks,
  // sorted, placed after the kept blocks of the lower-ranked slices.
  const int64_t b0 = R.begin / W, b1 = (R.end + W - 1) / W;
  uint32_t before = 0, ncand_part = 0;
  for (uint32_t i = threadIdx.x; i < KA; i += T) {
    const uint32_t bid = ~(uint32_t)R.stage[i];
    before += ((int64_t)bid < b0) ? 1u : 0u;
    const int64_t lo = (int64_t)bid * W;
    const int64_t hi = lo + W < R.L ? lo + W : R.L;
    ncand_part += (uint32_t)(hi - lo);
  }
  const uint32_t n_before = block_sum<T>(before, m);
  const uint32_t ncand = block_sum<T>(ncand_part, m);
  if (p.out_blocks) {
    int32_t* ob = p.out_blocks + R.row * (int64_t)p.k_blocks;
    const int64_t nbo = b1 - b0;
    if (nbo <= 32 * (int64_t)kBins) {
      // a bitmap of this CTA's kept blocks, then an ascending prefix over its
      // words: each thread writes the ids of its own words in order
      uint32_t* bits = R.hist;
      const uint32_t words = (uint32_t)((nbo + 31) >> 5);
      for (uint32_t i = threadIdx.x; i < words; i += T) bits[i] = 0u;
      __syncthreads();
      for (uint32_t i = threadIdx.x; i < KA; i += T) {
        const uint32_t bid = ~(uint32_t)R.stage[i];
        if ((int64_t)bid >= b0 && (int64_t)bid < b1) {
          const uint32_t o = (uint32_t)((int64_t)bid - b0);
          atomicOr(&bits[o >> 5], 1u << (o & 31u));
        }
      }
      __syncthreads();
      const uint32_t wpt = (words + T - 1) / T;
      const uint32_t w0 = threadIdx.x * wpt;
      const uint32_t w1 = min(w0 + wpt, words);
      uint32_t cnt = 0;
      for (uint32_t w = w0; w < w1; ++w) cnt += (uint32_t)__popc(bits[w]);
      uint32_t out = n_before + block_prefix_excl<T>(cnt, m);
      for (uint32_t w = w0; w < w1; ++w)
        for (uint32_t x = bits[w]; x; x &= x - 1u)
          ob[out++] = (int32_t)(b0 + 32 * (int64_t)w + (__ffs(x) - 1));
      if (R.rank == 0) {
        for (uint32_t j = KA + threadIdx.x; j < (uint32_t)p.k_blocks; j += T) ob[j] = -1;
      }
    } else {
      uint32_t* ids = R.hist;  // own kept ids as ~id, so a descending sort is ascending
      if (threadIdx.x == 0) m->own_count = 0;
      __syncthreads();
      for (uint32_t base = 0; base < KA; base += T) {
        const uint32_t i = base + threadIdx.x;
        uint32_t bid = 0;
        bool mine = false;
        if (i < KA) {
          bid = ~(uint32_t)R.stage[i];
          mine = (int64_t)bid >= b0 && (int64_t)bid < b1;
        }
        const unsigned msk = __ballot_sync(kFull, mine);
        if (msk) {
          const uint32_t lane = lane_id();
          const int leader = __ffs(msk) - 1;
          uint32_t bb = 0;
          if ((int)lane == leader) bb = atomicAdd(&m->own_count, (uint32_t)__popc(msk));
          bb = __shfl_sync(kFull, bb, leader);
          const uint32_t pos = bb + (uint32_t)__popc(msk & ((1u << lane) - 1u));
          if (mine && pos < (uint32_t)kBins) ids[pos] = ~bid;
        }
      }
      __syncthreads();
      const uint32_t n_own = m->own_count < (uint32_t)kBins ? m->own_count : (uint32_t)kBins;
      uint32_t P = 2;
      while (P < n_own) P <<= 1;
      for (uint32_t i = n_own + threadIdx.x; i < P; i += T) ids[i] = 0u;
      __syncthreads();
      bitonic_sort_desc<T>(ids, P);
      for (uint32_t i = threadIdx.x; i < n_own; i += T) ob[n_before + i] = (int32_t)(~ids[i]);
      if (R.rank == 0) {
        for (uint32_t j = KA + threadIdx.x; j < (uint32_t)p.k_blocks; j += T) ob[j] = -1;
      }
    }
  }
  __syncthreads();
  if (role == 2) {
    stamp(R, kTrOutput);
    wait_init(R);
    return;
  }

  // ---- stage B: the top k among the positions of the kept blocks
  const uint32_t KB = ncand < (uint32_t)p.k ? ncand : (uint32_t)p.k;
  bool intact_b;
  uint64_t TcB;
  const bool exactB = select_stage<T, U, W, false>(R, p, va, na, vb, nb, intact, KB, (int64_t)ncand,
                                                   p.row_stride, KeepBlocks<T, U, W>{TA}, false,
                                                   &intact_b, &TcB, kTrStageB);
  output_positions<T>(R, p, exactB, TcB, KB, p.row_stride, true);
  wait_init(R);
}

// Stage A selects the top k_blocks blocks of W positions by block key (the
// key of the block's best score), ties by lowest block id; stage B selects the
// top k positions inside the kept blocks, ties by lowest position. The kept
// block ids are also written in ascending order.
//
// With k_blocks >= k the stages are independent: every block holding one of
// the row's plain top-k positions is kept (each block ranked above it has its
// own maximum, a distinct position ranked above that position, so fewer than
// k blocks rank above it), hence stage B returns exactly the plain top-k. The
// launch then holds two groups of clusters (split): group 1 (clusters
// [0, rows)) computes the plain top-k of its row, group 2 (clusters
// [rows, 2 rows), launched only when out_blocks is wanted) stage A alone. Both
// read the row once, side by side, instead of one stage after the other.
//
// Rounds are four float4 per thread (eight only for 32-position blocks): with
// eight, the 512-thread kernel (128 registers a thread) spilled, and the
// side-by-side 16-row launch took 22.8 us against 21.5 with four.
template <int T, int W, class S>
__global__ void __launch_bounds__(T, (T <= 256 ? 3 : 1)) blocked_kernel(Params p) {
  constexpr int U0 = 4;  // float4 per thread per round
  constexpr int U = (W / 4 > U0) ? W / 4 : U0;
  using G = Geo<T, U, W>;
  extern __shared__ __align__(128) unsigned char smem[];
  RowT<S> R;
  stamp(p, kTrStart);
  grid_dependents_launch();
  const int64_t cid = (int64_t)(blockIdx.x / (p.clustered ? cluster_size() : 1u));
  // 0: both stages in turn; 1 / 2: plain top-k / stage A side by side;
  // 3: stage B over a given block list
  const int role = p.external ? 3 : (p.split ? (cid < p.rows ? 1 : 2) : 0);
  float4 va[U], vb[U];
  if (role == 1) {
    blocked_plain_row<T, U, S>(p, smem, cid % p.rows);
    return;
  }
  setup_row<T, U, W>(R, p, smem, p.split ? cid % p.rows : cid);
  Misc* m = R.m;
  int na[G::kSlots], nb[G::kSlots];
  if (role == 3) {
    blocked_listed_row<T, U, W, S>(R, p);
    return;
  }
  const int64_t nblocks = (R.L + W - 1) / W;
  const uint32_t KA = (uint32_t)(nblocks < (int64_t)p.k_blocks ? nblocks : (int64_t)p.k_blocks);

  // ---- stage A: the top k_blocks blocks by (block key desc, block id asc)
  bool intact;
  uint64_t TcA;
  const bool exactA = select_stage<T, U, W, true>(R, p, va, na, vb, nb, false, KA, nblocks, nblocks,
                                                  KeepAll{}, true, &intact, &TcA, 0);
  uint64_t TA = 0;
  if (KA > 0) {
    if (role == 2 && !exactA && (R.end - R.begin + W - 1) / W <= 32 * (int64_t)kBins && p.out_blocks) {
      // stage-A-only clusters on the fast path: every CTA holds every segment
      uint32_t lo = 0xffffffffu, hi = 0u;
      for (uint32_t q = 0; q < m->nseg; ++q) {
        if (m->seg_cnt[q] == 0) continue;
        lo = min(lo, m->seg_min[q]);
        hi = max(hi, m->seg_max[q]);
      }
      if (kept_from_segments<T, W>(R, p, KA, lo, hi)) {
        __syncthreads();
        stamp(R, kTrOutput);
        wait_init(R);
        return;
      }
    }
    TA = exactA ? TcA : select_local<T>(R, KA, nblocks);
    compact_selected<T>(R, TA);  // stage[0, KA) = kept block composites
  }
  {
    RoundRegs<U, G::kSlots> ra, rb;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      ra.v[u] = va[u];
      rb.v[u] = vb[u];
    }
#pragma unroll
    for (int q = 0; q < G::kSlots; ++q) {
      ra.n[q] = na[q];
      rb.n[q] = nb[q];
    }
    blocked_general_tail<T, U, W, S>(R, p, role, TA, KA, intact, ra, rb);
  }
}

template <int T, class S>
const void* blocked_kernel_ptr_of(int block) {
  switch (block) {
    case 4: return reinterpret_cast<const void*>(&blocked_kernel<T, 4, S>);
    case 8: return reinterpret_cast<const void*>(&blocked_kernel<T, 8, S>);
    case 16: return reinterpret_cast<const void*>(&blocked_kernel<T, 16, S>);
    case 32: return reinterpret_cast<const void*>(&blocked_kernel<T, 32, S>);
    default: return nullptr;
  }
}

}  // namespace lt
