// lt_stream.cuh -- the streamed top-k kernel: rows move from HBM into shared
// memory through a ring of stages filled by asynchronous bulk copies, so the
// bytes in flight per SM no longer depend on registers, and a CTA's next row
// is already arriving while it selects and writes the current one.
//
// Geometry. A CTA's slice [begin, end) of a row is cut into tiles of
// kTilePos positions (one bulk copy each). A chunk is kSlots tiles; chunk c,
// slot s holds tile c + rounds * s, so chunk 0 is spread over the whole slice
// and is the sample of the threshold estimate (chunks 0 and 1 are the whole
// slice when it has at most two). Thread t owns float4 t + T * u (u < UC) of
// a chunk; consecutive threads read consecutive 16-byte words.
//
// Ring. Stage i (of ring_stages) holds one chunk and one mbarrier. Thread 0
// is the producer: it arms the stage's barrier with the chunk's byte count
// and issues the chunk's tile copies; the other threads wait on the barrier's
// phase parity. A stage is refilled -- with the rest of this row, then with
// the next row of this CTA -- after the block barrier that follows the
// chunk's filter. Chunks are numbered in the order the CTA consumes them over
// all of its rows: chunk g lives in stage g % ring_stages, phase parity
// (g / ring_stages) & 1.
//
// Selection is the same as in the register-resident kernel (sampled digit
// histogram, cluster merge, filter, candidate exchange, exact streaming radix
// select on a miss, bucket select-sort output), sharing its functions.
//
// Waits. Every mbarrier wait makes at most kWaitPolls try_wait calls, each
// suspending the thread for at most kSuspendNs (about 1.3 s in all). A wait
// that gives up marks the row in counters[kCntTimeout] (when counters are
// given); the CTA then keeps going, and before it exits it waits on each stage
// that may still have copies in flight, again a bounded number of times.

#pragma once

#include "lt_async.cuh"
#include "lt_kernels.cuh"

namespace lt {

constexpr int kTilePos = 1024;            // positions per bulk copy (4 KB)

template <int T, int UC>
struct SGeo {
  static constexpr int kChunk = T * UC * 4;  // positions per chunk
  static constexpr int kSlots = kChunk / kTilePos;
  static_assert(kChunk % kTilePos == 0 && kSlots >= 1, "a chunk holds whole tiles");
  static_assert(4 * UC <= 32, "the filter mask holds 32 positions");
};

struct StreamLayout {
  uint32_t prod, bars, ring, total;
};

constexpr uint32_t kProdBytes = 192;  // producer state (thread 0), see Prod

__host__ __device__ inline StreamLayout make_stream_layout(bool clustered, uint32_t cap, uint32_t sel_cap,
                                                           uint32_t stages, uint32_t chunk_bytes) {
  StreamLayout s;
  const Layout l = make_layout(clustered, cap, sel_cap, 0);
  s.prod = align_up_u32(l.total, 16);
  s.bars = align_up_u32(s.prod + kProdBytes, 8);
  s.ring = align_up_u32(s.bars + 8 * stages, 128);
  s.total = s.ring + stages * chunk_bytes;
  return s;
}

// ------------------------------------------------------------------ geometry

// The slice of `row` owned by cluster rank `rank` (same split as setup_row
// with W = 4).
__device__ __forceinline__ void slice_of(const Params& p, int64_t row, uint32_t rank, uint32_t nclus,
                                         int64_t* begin, int64_t* end, int64_t* per_out) {
  int64_t L = p.row_stride;
  if (p.lengths) {
    L = (int64_t)p.lengths[row];
    L = L < 0 ? 0 : (L > p.row_stride ? p.row_stride : L);
  }
  const int cl2 = 31 - __clz((int)nclus);
  int64_t per = (L + nclus - 1) >> cl2;
  per = (per + 3) & ~(int64_t)3;
  const int64_t b = (int64_t)rank * per;
  *begin = b < L ? b : L;
  *end = (*begin + per) < L ? (*begin + per) : L;
  if (per_out) *per_out = per;
}

template <int T, int UC>
__device__ __forceinline__ int chunk_rounds(int64_t len) {
  constexpr int64_t C = SGeo<T, UC>::kChunk;
  return (int)((len + C - 1) / C);
}

// Offset from the slice start of the first of the four scores in float4 f of
// chunk c (slices are shorter than 2^31 positions).
__device__ __forceinline__ uint32_t chunk_rel(int c, int rounds, uint32_t f) {
  constexpr uint32_t kF4 = kTilePos / 4;
  return (uint32_t)(c + rounds * (int)(f / kF4)) * kTilePos + 4u * (f % kF4);
}

// Whether every position of chunk c lies inside a slice of `len` positions.
template <int T, int UC>
__device__ __forceinline__ bool chunk_full(int c, int rounds, uint32_t len) {
  return (uint32_t)(c + rounds * (SGeo<T, UC>::kSlots - 1) + 1) * kTilePos <= len;
}

// Valid positions in chunk 0 of all slices of a row of L positions -- the
// sample, whose level-1 histogram holds exactly this many items -- from the
// slice geometry alone: slice r covers [r*per, min(L, (r+1)*per)), and its
// chunk 0 holds its tiles 0, rounds_r, 2*rounds_r, ... (rounds_r = that
// slice's chunk count), each clipped to the slice.
template <int T, int UC>
__device__ __forceinline__ uint32_t sample_size(int64_t L, uint32_t nclus) {
  constexpr int S = SGeo<T, UC>::kSlots;
  const int cl2 = 31 - __clz((int)nclus);
  int64_t per = (L + nclus - 1) >> cl2;
  per = (per + 3) & ~(int64_t)3;
  uint64_t n = 0;
  for (uint32_t r = 0; r < nclus; ++r) {
    const int64_t b = (int64_t)r * per < L ? (int64_t)r * per : L;
    const int64_t e = (b + per) < L ? (b + per) : L;
    const int64_t len = e - b;
    const int rounds = chunk_rounds<T, UC>(len);
    for (int s = 0; s < S; ++s) {
      const int64_t t0 = (int64_t)rounds * s * kTilePos;
      if (t0 < len) n += (uint64_t)(len - t0 < kTilePos ? len - t0 : kTilePos);
    }
  }
  return (uint32_t)n;
}

// ------------------------------------------------------------------ producer (thread 0)

struct Prod {
  // fixed for the launch
  const float* scores;
  const int32_t* lengths;
  int64_t row_stride, rows, step;
  uint64_t* bars;
  float* ring;
  uint32_t ns, rank, nclus;
  // the row being issued
  const float* rowp;
  int64_t row, begin, end4;
  int chunk, rounds;
  uint32_t seq;       // next chunk number to issue
  uint32_t released;  // chunks whose stage is free again
  bool skip_last;     // tests only: never issue this CTA's final chunk
};
static_assert(sizeof(Prod) <= kProdBytes, "producer state does not fit its shared-memory slot");

template <int T, int UC>
__device__ __forceinline__ void prod_row(Prod& P, int64_t row) {
  P.row = row;
  P.chunk = 0;
  P.rounds = 0;
  if (row >= P.rows) return;
  int64_t L = P.row_stride;
  if (P.lengths) {
    L = (int64_t)P.lengths[row];
    L = L < 0 ? 0 : (L > P.row_stride ? P.row_stride : L);
  }
  const int cl2 = 31 - __clz((int)P.nclus);
  int64_t per = (L + P.nclus - 1) >> cl2;
  per = (per + 3) & ~(int64_t)3;
  const int64_t b = (int64_t)P.rank * per;
  const int64_t bb = b < L ? b : L;
  const int64_t e = (bb + per) < L ? (bb + per) : L;
  P.rowp = P.scores + row * P.row_stride;
  P.begin = bb;
  // rows are 16-byte aligned and row_stride % 4 == 0, so reading up to the
  // next multiple of four positions stays inside the row
  P.end4 = (e + 3) & ~(int64_t)3;
  P.rounds = chunk_rounds<T, UC>(e - bb);
}

// Issue chunks while their stage is free (chunk numbers below `limit`).
template <int T, int UC>
__device__ __forceinline__ void produce(Prod& P, uint32_t limit) {
  using SG = SGeo<T, UC>;
  while (P.row < P.rows && (int32_t)(limit - P.seq) > 0) {
    if (P.chunk >= P.rounds) {
      prod_row<T, UC>(P, P.row + P.step);
      continue;
    }
    const uint32_t st = P.seq % P.ns;
    if (P.skip_last && P.chunk == P.rounds - 1 && P.row + P.step >= P.rows) {
      // tests only: the CTA's final chunk is never issued, so its stage's
      // barrier never completes and the consumers' bounded wait gives up;
      // no copy is in flight for it
      ++P.chunk;
      ++P.seq;
      continue;
    }
    float* dst = P.ring + (size_t)st * SG::kChunk;
    uint32_t n[SG::kSlots];
    uint32_t bytes = 0;
#pragma unroll
    for (int s = 0; s < SG::kSlots; ++s) {
      const int64_t pos = P.begin + (int64_t)(P.chunk + P.rounds * s) * kTilePos;
      n[s] = pos < P.end4 ? (uint32_t)(P.end4 - pos < kTilePos ? P.end4 - pos : kTilePos) : 0u;
      bytes += 4u * n[s];
    }
    mbar_arrive_tx(&P.bars[st], bytes);
#pragma unroll
    for (int s = 0; s < SG::kSlots; ++s) {
      const int64_t pos = P.begin + (int64_t)(P.chunk + P.rounds * s) * kTilePos;
      if (n[s] > 0) bulk_g2s(dst + s * kTilePos, P.rowp + pos, 4u * n[s], &P.bars[st]);
    }
    ++P.chunk;
    ++P.seq;
  }
}

// ------------------------------------------------------------------ consumers

// Sample histogram of one chunk (level 1: top 11 key bits; level 2: the next
// 11 bits of the keys whose top 11 bits equal d1).
template <int T, int UC, int kLevel>
__device__ __forceinline__ void hist_chunk(Row& R, const float* buf, int c, int rounds, uint32_t d1) {
  const float4* b4 = reinterpret_cast<const float4*>(buf);
  const uint32_t len = (uint32_t)(R.end - R.begin);
  const bool full = chunk_full<T, UC>(c, rounds, len);
#pragma unroll
  for (int u = 0; u < UC; ++u) {
    const uint32_t f = threadIdx.x + T * u;
    const uint32_t rel = chunk_rel(c, rounds, f);
    const int left = full ? 4 : (rel >= len ? 0 : (int)min(len - rel, 4u));
    if (left == 0) continue;
    const float4 q = b4[f];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (e < left) {
        const uint32_t kk = raw_key(__float_as_uint(lane4(q, e)));
        if (kLevel == 1) atomicAdd(&R.hist[kk >> 21], 1u);
        else if ((kk >> 21) == d1) atomicAdd(&R.hist[(kk >> 10) & (kBins - 1)], 1u);
      }
    }
  }
}

// Append every valid position of the chunk whose score passes (x >= g, or
// every valid position when `all`) to the list. The scores sit in shared
// memory, so each lane with candidates reserves its slots with one shared
// atomic and writes them itself (list order is irrelevant: the output ranks).
template <int T, int UC>
__device__ __forceinline__ void filter_chunk(Row& R, const float* buf, int c, int rounds, float g, bool all,
                                             uint32_t* counter, uint2* list, uint32_t cap) {
  const float4* b4 = reinterpret_cast<const float4*>(buf);
  const uint32_t len = (uint32_t)(R.end - R.begin);
  const bool full = chunk_full<T, UC>(c, rounds, len);
  uint32_t mask = 0;
#pragma unroll
  for (int u = 0; u < UC; ++u) {
    const uint32_t f = threadIdx.x + T * u;
    uint32_t b = 15u;
    if (!all) {
      // one compare per float4 on the common path: fmaxf ignores a NaN
      // operand and NaN never passes, so the max passes iff some lane does
      const float4 q = b4[f];
      b = 0u;
      if (fmaxf(fmaxf(q.x, q.y), fmaxf(q.z, q.w)) >= g)
        b = (q.x >= g ? 1u : 0u) | (q.y >= g ? 2u : 0u) | (q.z >= g ? 4u : 0u) | (q.w >= g ? 8u : 0u);
    }
    if (!full) {
      const uint32_t rel = chunk_rel(c, rounds, f);
      b &= rel >= len ? 0u : (len - rel >= 4u ? 15u : (1u << (len - rel)) - 1u);
    }
    mask |= b << (4 * u);
  }
  if (__ballot_sync(kFull, mask != 0) == 0) return;
  uint32_t kmn = 0xffffffffu, kmx = 0u;
  if (mask) {
    uint32_t slot = atomicAdd(counter, (uint32_t)__popc(mask));
    for (; mask; mask &= mask - 1u, ++slot) {
      const uint32_t bit = (uint32_t)(__ffs(mask) - 1);
      const uint32_t f = threadIdx.x + T * (bit >> 2), e = bit & 3u;
      const uint32_t kk = key_of(buf[4 * f + e]);
      kmn = min(kmn, kk);
      kmx = max(kmx, kk);
      if (slot < cap) list[slot] = make_uint2(kk, (uint32_t)(R.begin + (int64_t)(chunk_rel(c, rounds, f) + e)));
    }
  }
  kmn = __reduce_min_sync(kFull, kmn);
  kmx = __reduce_max_sync(kFull, kmx);
  if (lane_id() == 0) {
    atomicMin(&R.m->local_min, kmn);
    atomicMax(&R.m->local_max, kmx);
  }
}

// One row: estimate -> filter every chunk -> exchange -> (exact select) ->
// ordered output. g0 is the number of this row's chunk 0.
template <int T, int UC, int UR>
__device__ __forceinline__ void stream_row(Row& R, const Params& p, uint64_t* bars, float* ring, uint32_t ns,
                                           uint32_t g0, int rounds, int rounds_max, Prod& P, bool& late) {
  using SG = SGeo<T, UC>;
  Misc* m = R.m;
  const uint32_t K = (uint32_t)(R.L < (int64_t)p.k ? R.L : (int64_t)p.k);
  const uint32_t seg = 1u << R.seg_shift;
  uint2* list = R.cand + (R.rank << R.seg_shift);
  uint32_t* counter = &m->local_count;
  const uint32_t cap = (uint32_t)p.cap;
  const bool full = rounds_max <= 2;
  auto stage = [&](int c) -> float* { return ring + (size_t)((g0 + (uint32_t)c) % ns) * SG::kChunk; };
  const uint32_t polls = p.stall_polls > 0 ? (uint32_t)p.stall_polls : kWaitPolls;
  auto wait_chunk = [&](int c) {
    if (!ring_wait(bars, ns, g0 + (uint32_t)c, polls)) late = true;
  };
  // block barrier (every thread is done with the chunk's stage), then refill
  auto release_chunk = [&](int c) {
    __syncthreads();
    if (threadIdx.x == 0) {
      P.released = g0 + (uint32_t)c + 1u;
      produce<T, UC>(P, P.released + ns);
    }
  };

  bool exact = p.force_exact != 0;
  bool consumed = false;
  int stat = kCntFast;
  uint64_t Tc = 0;
  if (!exact && K > 0) {
    uint32_t t = 0;
    if (R.L > (int64_t)(cap / 2)) {
      const int nsr = full ? (rounds < 2 ? rounds : 2) : (rounds < 1 ? rounds : 1);
      for (int c = 0; c < nsr; ++c) wait_chunk(c);
      uint32_t r = 0, d1 = 0, above1 = 0;
#pragma unroll 1
      for (int level = 1; level <= 2; ++level) {
        zero_bins<T>(R.hist);
        for (int c = 0; c < nsr; ++c) {
          if (level == 1) hist_chunk<T, UC, 1>(R, stage(c), c, rounds, 0);
          else hist_chunk<T, UC, 2>(R, stage(c), c, rounds, d1);
        }
        if (level == 1) stamp(R, kTrHist);
        const uint32_t lo_rank = (level == 1 && full && R.nclus >= 8) ? (K < (uint32_t)R.L ? K : (uint32_t)R.L) : 0u;
        const uint32_t* bins = merge_hist<T>(R, level - 1, lo_rank);
        if (level == 1) stamp(R, kTrMerge);
        if (level == 1) {
          const uint32_t nsamp = full ? (uint32_t)R.L : sample_size<T, UC>(R.L, R.nclus);
          if (nsamp == 0) {
            release_merged<T>(R, 0);
            break;
          }
          r = sample_target(K, nsamp, R.L, full);
          find_digit<T>(bins, r, m);
          d1 = m->res_digit;
          above1 = m->res_above;
          const uint32_t cnt1 = m->res_cnt;
          release_merged<T>(R, 0);
          t = d1 << 21;
          const float predicted = full ? (float)(above1 + cnt1)
                                       : (float)(above1 + cnt1) * ((float)R.L / (float)nsamp);
          if (predicted <= kLevel2Frac * (float)cap) break;  // one 11-bit level is selective enough
        } else {
          find_digit<T>(bins, r - above1, m);
          t |= m->res_digit << 10;
          release_merged<T>(R, 1);
        }
      }
    }
    stamp(R, kTrEstimate);
    {
      // the output's bucket counts start from zero; the exchange's barrier
      // orders these stores before them
      uint4* z = reinterpret_cast<uint4*>(R.hist);
      for (int i = threadIdx.x; i < kOutBuckets / 4; i += T) z[i] = make_uint4(0, 0, 0, 0);
    }
    const bool all = (t == 0u);
    const float g = threshold_float(all ? 1u : t);
#pragma unroll 1
    for (int c = 0; c < rounds; ++c) {
      wait_chunk(c);
      filter_chunk<T, UC>(R, stage(c), c, rounds, g, all, counter, list, seg);
      release_chunk(c);
    }
    consumed = true;
    stamp(R, kTrFilter);
    exchange_segments<T>(R, false);
    stamp(R, kTrExchange);
    const uint32_t cs = lane_id() < R.nclus ? m->seg_cnt[lane_id()] : 0u;
    const uint32_t total = __reduce_add_sync(kFull, cs);
    const bool overflow = __any_sync(kFull, cs > seg);
    if (overflow || total < K) {
      exact = true;
      stat = overflow ? kCntOverflow : kCntShort;
    }
  }
  if (!consumed) {
    // keep the ring in step: this row's chunks were issued all the same
#pragma unroll 1
    for (int c = 0; c < rounds; ++c) {
      wait_chunk(c);
      release_chunk(c);
    }
  }
  if (exact && K > 0) {
    if (stat != kCntFast) bump(p, R, stat);
    wait_init(R);
    Tc = exact_select<T, UR, 4, false>(R, p, K, p.row_stride, KeepAll{});
    stamp(R, kTrExact);
    bump(p, R, kCntExact);
  } else {
    stamp(R, kTrExact);
    if (K > 0) bump(p, R, kCntFast);
  }
  output_positions<T>(R, p, exact, Tc, K, p.row_stride, false);
}

}  // namespace lt
