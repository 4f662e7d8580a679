// lt_kernels.cuh -- per-row selection machinery shared by the kernels.
//
// Data movement: a CTA's slice [begin, end) of the row is cut into tiles of
// T * W positions (one W-wide slot per thread per tile, W/4 float4 loads). A
// "round" is U float4 per thread. Round r, slot s covers tile r + rounds * s,
// so round 0 is spread over the whole slice and serves as a representative
// sample. Two register buffers hold the current and the next round; rounds
// stream through them. For the top-k kernel W = 4 (items are positions); for
// the two-level kernel W = block (stage A items are blocks, stage B items are
// the positions of the kept blocks).
//
// Code layout: a row's code runs once per CTA, so its latency includes
// fetching that code. Everything a normal row executes is inlined once; the
// paths only adversarial rows take (the streaming exact select, the
// radix-select + bitonic fallback of the output, the single-round path's
// second estimate level) are separate functions, and slices of one register
// round use select_one, which has no streaming code at all.

#pragma once

#include "lt_device.cuh"

namespace lt {

template <int T, int U, int W>
struct Geo {
  static constexpr int kVS = W / 4;        // float4 loads per slot
  static constexpr int kSlots = U / kVS;   // slots per round
  static constexpr int64_t kTile = (int64_t)T * W;
  static_assert(W % 4 == 0 && U % kVS == 0 && kSlots >= 1, "bad geometry");
};

// Per-row state of one CTA. RowCore holds everything but the score pointer;
// RowT<S> adds it for the score type S (float, or uint16_t holding bf16 bits).
struct RowCore {
  Misc* m;
  uint32_t* hist;
  uint32_t* aux;
  uint32_t* merged0;     // cluster merge targets (== hist with one CTA)
  uint32_t* merged1;
  uint2* cand;           // nclus segments of (1 << seg_shift) slots
  uint64_t* stage;
  float4* wst;           // this warp's staging area: [kStageF4][32] float4
  int64_t row;
  int64_t L;             // valid positions of the row
  int64_t begin, end;    // this CTA's slice of positions
  int64_t tbase;         // begin + threadIdx.x * W
  uint32_t rank, nclus;
  uint32_t stage_cap;
  uint32_t seg_shift;
  int rounds;            // rounds of this CTA's slice
  int rounds_max;        // cluster-wide maximum
  bool init_pending;     // the start-up cluster barrier has not been waited on
  int64_t* trace;        // phase timestamps of this row (nullable)
};

template <class S>
struct RowT : RowCore {
  const S* rowp;         // scores of this row
};
using Row = RowT<float>;

// Phase timestamp of this row (thread 0 of each CTA), when traced.
__device__ __forceinline__ void stamp(const RowCore& R, int slot) {
  if (R.trace != nullptr && threadIdx.x == 0) {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    R.trace[(int64_t)blockIdx.x * kTraceSlots + slot] = (int64_t)t;
  }
}

// Items of this CTA's own slice (ranks in the output are written by their owner).
struct OwnSlice {
  int64_t b, e;
  bool all;
  __device__ __forceinline__ bool operator()(uint32_t idx) const {
    return all || ((int64_t)idx >= b && (int64_t)idx < e);
  }
};
__device__ __forceinline__ OwnSlice own_slice(const RowCore& R) { return OwnSlice{R.begin, R.end, R.nclus == 1}; }

// Filler of positions past the slice end: a NaN (never passes x >= g) whose
// raw key is 0 (lands in the lowest histogram bin).
__device__ __forceinline__ float nan_f() { return __int_as_float((int)0xffffffffu); }

template <int T, int U, int W>
__device__ __forceinline__ int64_t slot_pos(const RowCore& R, int r, int s) {
  return R.tbase + (int64_t)(r + R.rounds * s) * Geo<T, U, W>::kTile;
}

// Scalar load of a ragged or unaligned group of four positions: [0, nv) are
// read, the rest are NaN (no threshold compare accepts NaN).
template <class S>
__device__ __forceinline__ float4 load4_scalar(const S* p, int nv) {
  float e[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) e[q] = (q < nv) ? load1(p + q) : nan_f();
  return make_float4(e[0], e[1], e[2], e[3]);
}

// Load round r; n[s] = valid positions of slot s (a prefix of the slot).
template <int T, int U, int W, class S>
__device__ __forceinline__ void load_round(const RowT<S>& R, bool vec, int r, float4 (&v)[U],
                                           int (&n)[Geo<T, U, W>::kSlots]) {
  using G = Geo<T, U, W>;
  // every slot full (the last one is the furthest): one straight run of loads
  if (vec && slot_pos<T, U, W>(R, r, G::kSlots - 1) + W <= R.end) {
    gather_round<U, G::kVS>(R.rowp + slot_pos<T, U, W>(R, r, 0), (int64_t)R.rounds * G::kTile, v);
#pragma unroll
    for (int s = 0; s < G::kSlots; ++s) n[s] = W;
    return;
  }
#pragma unroll
  for (int s = 0; s < G::kSlots; ++s) {
    const int64_t pos = slot_pos<T, U, W>(R, r, s);
    int64_t nv = R.end - pos;
    nv = nv < 0 ? 0 : (nv > W ? W : nv);
    n[s] = (int)nv;
    if (nv == W && vec) {
#pragma unroll
      for (int j = 0; j < G::kVS; ++j) v[s * G::kVS + j] = ldg4(R.rowp + pos + 4 * j);
    } else {
#pragma unroll
      for (int j = 0; j < G::kVS; ++j) {
        const int64_t left = nv - 4 * j;
        v[s * G::kVS + j] = load4_scalar(R.rowp + pos + 4 * j, left < 0 ? 0 : (left > 4 ? 4 : (int)left));
      }
    }
  }
}

// Bulk prefetch of this CTA's slice [begin, end) into L2, in 32 pieces (one
// per lane of the calling warp); pieces that do not start on a 16-byte
// boundary are skipped (a prefetch only changes timing).
template <class S>
__device__ __forceinline__ void prefetch_slice_l2(const RowT<S>& R) {
  const char* b = reinterpret_cast<const char*>(R.rowp + R.begin);
  const int64_t bytes = (R.end - R.begin) * (int64_t)sizeof(S);
  const int64_t piece = ((bytes + 31) / 32 + 15) & ~(int64_t)15;
  const int64_t off = (int64_t)lane_id() * piece;
  int64_t n = bytes - off;
  n = (n < piece ? n : piece) & ~(int64_t)15;
  if (n > 0 && (reinterpret_cast<uintptr_t>(b + off) & 15u) == 0)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(b + off), "r"((uint32_t)n) : "memory");
}

// Four-position slots (W = 4): round r lies wholly inside the slice.
template <int T, int U>
__device__ __forceinline__ bool round_whole(const RowCore& R, int r) {
  return (int64_t)(r + R.rounds * (U - 1) + 1) * Geo<T, U, 4>::kTile <= R.end - R.begin;
}

// Load round r of four-position slots: a whole round takes U vector loads
// from this thread's slot pointers, others go through load_round.
template <int T, int U, class S>
__device__ __forceinline__ void load_round4(const RowT<S>& R, bool vec, int r, float4 (&v)[U], int (&n)[U]) {
  using G = Geo<T, U, 4>;
  if (vec && round_whole<T, U>(R, r)) {
    gather_round<U, 1>(R.rowp + R.tbase + (int64_t)r * G::kTile, (int64_t)R.rounds * G::kTile, v);
#pragma unroll
    for (int s = 0; s < U; ++s) n[s] = 4;
  } else {
    load_round<T, U, 4>(R, vec, r, v, n);
  }
}

template <int S>
__device__ __forceinline__ void clear_round(int (&n)[S]) {
#pragma unroll
  for (int s = 0; s < S; ++s) n[s] = 0;
}

// Key of the block held in slot s (max of the keys of its valid positions).
template <int T, int U, int W>
__device__ __forceinline__ uint32_t slot_block_key(const float4 (&v)[U], int s, int nv) {
  // key_of is monotone on non-NaN scores and maps NaN lowest; fmaxf skips a
  // NaN operand, so the key of the float maximum is the maximum key (an
  // all-NaN block gives NaN, key 0). Positions past the slice end hold NaN.
  constexpr int VS = Geo<T, U, W>::kVS;
  (void)nv;
  float best = fmaxf(fmaxf(v[s * VS].x, v[s * VS].y), fmaxf(v[s * VS].z, v[s * VS].w));
#pragma unroll
  for (int j = 1; j < VS; ++j) {
    const float4 q = v[s * VS + j];
    best = fmaxf(best, fmaxf(fmaxf(q.x, q.y), fmaxf(q.z, q.w)));
  }
  return key_of(best);
}

struct KeepAll {
  static constexpr bool kAll = true;
  template <class V>
  __device__ __forceinline__ bool operator()(const RowCore&, int, const V&, int, int) const { return true; }
};

// Stage B of the two-level kernel: keep a slot (one block) when its block
// composite is >= the stage-A threshold composite Tc.
// Keep the positions of listed blocks: bits covers blocks [b0, b0 + nbits) of
// the row (this CTA's slice), bit i of bits[i >> 5] marking block b0 + i;
// blocks outside it are not listed.
template <int T, int U, int W>
struct KeepListed {
  static constexpr bool kAll = false;
  const uint32_t* bits;
  int64_t b0;
  uint32_t nbits;
  __device__ __forceinline__ bool operator()(const RowCore& R, int r, const float4 (&)[U], int s, int) const {
    const int64_t bid = slot_pos<T, U, W>(R, r, s) / W - b0;
    return bid >= 0 && bid < (int64_t)nbits && ((bits[bid >> 5] >> (bid & 31)) & 1u) != 0u;
  }
};

template <int T, int U, int W>
struct KeepBlocks {
  static constexpr bool kAll = false;
  uint64_t Tc;
  __device__ __forceinline__ bool operator()(const RowCore& R, int r, const float4 (&v)[U], int s, int nv) const {
    const uint32_t bid = (uint32_t)(slot_pos<T, U, W>(R, r, s) / W);
    return composite(slot_block_key<T, U, W>(v, s, nv), bid) >= Tc;
  }
};

// ------------------------------------------------------------------ setup

// row < 0: the row of this CTA's cluster (one row per cluster); otherwise the
// given row (persistent kernels).
template <int T, int U, int W, class S>
__device__ __forceinline__ void setup_row(RowT<S>& R, const Params& p, unsigned char* smem, int64_t row = -1) {
  using G = Geo<T, U, W>;
  R.nclus = p.clustered ? cluster_size() : 1u;
  R.rank = p.clustered ? cluster_rank() : 0u;
  R.row = row >= 0 ? row : (int64_t)(blockIdx.x / R.nclus);
  const Layout lay = make_layout(p.clustered != 0, (uint32_t)p.cap, (uint32_t)p.sel_cap, (uint32_t)p.wstage);
  R.m = reinterpret_cast<Misc*>(smem + lay.misc);
  R.hist = reinterpret_cast<uint32_t*>(smem + lay.hist);
  R.aux = reinterpret_cast<uint32_t*>(smem + lay.aux);
  R.merged0 = reinterpret_cast<uint32_t*>(smem + lay.merged0);
  R.merged1 = reinterpret_cast<uint32_t*>(smem + lay.merged1);
  R.cand = reinterpret_cast<uint2*>(smem + lay.cand);
  R.stage = reinterpret_cast<uint64_t*>(smem + lay.stage);
  static_assert(U <= kStageF4, "a lane stages at most kStageF4 float4");
  R.wst = reinterpret_cast<float4*>(smem + lay.wstage) + (threadIdx.x >> 5) * 32 * kStageF4;
  R.stage_cap = (uint32_t)p.sel_cap + kMaxBucket;
  R.trace = p.trace;
  R.seg_shift = (uint32_t)p.seg_shift;

  // shared-memory initialisation first: it overlaps the previous kernel of
  // the stream under programmatic dependent launch
  Misc* m = R.m;
  if (threadIdx.x == 0) {
    m->cand_count = 0;
    m->local_count = 0;
    m->local_min = 0xffffffffu;
    m->local_max = 0u;
    m->flags = 0;
    m->own_count = 0;
    m->aux[7] = 0;  // cluster-wide sums pushed by peers (listed positions)
    for (int i = 0; i < 2; ++i) {
      m->hint_min[i] = 0xffffffffu;
      m->hint_max[i] = 0u;
    }
  }
  if (p.clustered) {
    uint4* z0 = reinterpret_cast<uint4*>(R.merged0);
    uint4* z1 = reinterpret_cast<uint4*>(R.merged1);
    for (int i = threadIdx.x; i < kBins / 4; i += T) {
      z0[i] = make_uint4(0, 0, 0, 0);
      z1[i] = make_uint4(0, 0, 0, 0);
    }
  }
  // lengths, scores and the outputs may belong to the previous kernel
  grid_dependency_wait();

  int64_t L = p.row_stride;
  if (p.lengths) {
    L = (int64_t)p.lengths[R.row];
    L = L < 0 ? 0 : (L > p.row_stride ? p.row_stride : L);
  }
  R.L = L;
  R.rowp = static_cast<const S*>(p.scores) + R.row * p.row_stride;
  // the cluster size, T, W and the slots per round are powers of two
  const int cl2 = 31 - __clz((int)R.nclus);
  int64_t per = (L + R.nclus - 1) >> cl2;
  per = (per + W - 1) & ~(int64_t)(W - 1);
  const int64_t b = (int64_t)R.rank * per;
  R.begin = b < L ? b : L;
  R.end = (R.begin + per) < L ? (R.begin + per) : L;
  R.tbase = R.begin + (int64_t)threadIdx.x * W;
  constexpr int kTile2 = __builtin_ctz((unsigned)(T * W));
  constexpr int kSl2 = __builtin_ctz((unsigned)G::kSlots);
  const int64_t nt = (R.end - R.begin + G::kTile - 1) >> kTile2;
  R.rounds = (int)((nt + G::kSlots - 1) >> kSl2);
  const int64_t ntm = (per + G::kTile - 1) >> kTile2;
  R.rounds_max = (int)((ntm + G::kSlots - 1) >> kSl2);
  __syncthreads();
  R.init_pending = false;
  if (R.nclus > 1) {
    cluster_arrive();  // "my merged buffers and counters are zero"; waited on before the first push
    R.init_pending = true;
  }
}

__device__ __forceinline__ void wait_init(RowCore& R) {
  if (R.init_pending) {
    cluster_wait();
    R.init_pending = false;
  }
}

template <int T>
__device__ __forceinline__ void zero_bins(uint32_t* b) {
  uint4* p = reinterpret_cast<uint4*>(b);
  for (int i = threadIdx.x; i < kBins / 4; i += T) p[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
}

__device__ __forceinline__ void bump(const Params& p, const RowCore& R, int which) {
  if (p.counters && R.rank == 0 && threadIdx.x == 0) atomicAdd(&p.counters[which], 1);
}

__device__ __forceinline__ void dsmem_st_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}

// ------------------------------------------------------------------ candidates

// Visit every candidate: the array holds nseg segments of (1 << shift) slots,
// segment q holding seg_cnt[q] entries. Warps are spread over the segments
// (several warps per segment when there are fewer segments than warps).
template <int T, class F>
__device__ __forceinline__ void for_each_cand(const RowCore& R, F f) {
  constexpr uint32_t NW = T / 32;
  const Misc* m = R.m;
  const uint32_t nseg = m->nseg, shift = m->shift;
  const uint32_t seg = 1u << shift;
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  if (nseg >= NW) {
    for (uint32_t q = warp; q < nseg; q += NW) {
      const uint32_t n = min(m->seg_cnt[q], seg);
      const uint2* c = R.cand + (q << shift);
      for (uint32_t j = lane; j < n; j += 32) f(c[j]);
    }
  } else {
    // 2^lp warps per segment (nseg and NW are powers of two)
    const uint32_t lp = (uint32_t)(__clz(nseg) - __clz((int)NW));
    const uint32_t q = warp >> lp, sub = warp & ((1u << lp) - 1u);
    const uint32_t n = min(m->seg_cnt[q], seg);
    const uint2* c = R.cand + (q << shift);
    for (uint32_t j = sub * 32 + lane; j < n; j += 32u << lp) f(c[j]);
  }
}

__device__ __forceinline__ void reset_candidate_range(Misc* m) {
  m->kmin = 0xffffffffu;
  m->kmax = 0u;
  m->res_max = 0u;
  m->aux[1] = 0u;
}

// ------------------------------------------------------------------ cluster exchange

// Push the non-empty bins of the local histogram into merged buffer `buf` of
// every CTA of the cluster (this one included), then cluster-sync. With one
// CTA the local histogram is the merged one.
// With lo_rank > 0 only the bins at or above this CTA's own lo_rank-th key
// are pushed: the cluster-wide lo_rank-th key is at least that large, so every
// bin at or above its digit still arrives complete (used with a full sample).
template <int T>
__device__ __forceinline__ const uint32_t* merge_hist(RowCore& R, int buf, uint32_t lo_rank = 0) {
  __syncthreads();
  if (R.nclus == 1) return R.hist;
  uint32_t dlo = 0;
  if (lo_rank > 0) {
    if (threadIdx.x == 0) R.m->res_digit = 0;  // stays 0 when this CTA holds fewer than lo_rank keys
    find_digit<T>(R.hist, lo_rank, R.m);
    dlo = R.m->res_digit;
  }
  wait_init(R);
  uint32_t* dst = buf ? R.merged1 : R.merged0;
  const uint32_t base = smem_addr(dst);
  for (int b = threadIdx.x; b < kBins; b += T) {
    const uint32_t v = (uint32_t)b >= dlo ? R.hist[b] : 0u;
    if (v) {
      for (uint32_t q = 0; q < R.nclus; ++q) dsmem_red_add(peer_addr(base + 4u * b, q), v);
    }
  }
  cluster_sync();
  return dst;
}

// After the digit search on merged buffer `buf`: clear it for its next use.
// Peers only write it again after a later cluster barrier.
template <int T>
__device__ __forceinline__ void release_merged(RowCore& R, int buf) {
  if (R.nclus == 1) return;
  uint4* p = reinterpret_cast<uint4*>(buf ? R.merged1 : R.merged0);
  for (int i = threadIdx.x; i < kBins / 4; i += T) p[i] = make_uint4(0, 0, 0, 0);
}

// Fast-path exchange: this CTA's count and key range go to every peer, its
// segment to the same segment of every peer, or with `gather` to rank 0 only
// (which then orders and writes the whole row). One cluster barrier, no
// remote atomics.
template <int T>
__device__ __forceinline__ void exchange_segments(RowCore& R, bool gather) {
  Misc* m = R.m;
  __syncthreads();
  const uint32_t n = m->local_count;
  if (threadIdx.x == 0) {
    reset_candidate_range(m);
    m->nseg = R.nclus;
    m->shift = R.seg_shift;
  }
  const uint32_t kmn = m->local_min, kmx = m->local_max;
  if (R.nclus == 1) {
    if (threadIdx.x == 0) {
      m->seg_cnt[0] = n;
      m->seg_min[0] = kmn;
      m->seg_max[0] = kmx;
    }
    __syncthreads();
    return;
  }
  wait_init(R);
  const uint32_t seg = 1u << R.seg_shift;
  const uint32_t n_put = n < seg ? n : seg;
  const uint32_t off = R.rank << R.seg_shift;
  if (threadIdx.x < R.nclus) {
    dsmem_st_u32(peer_addr(smem_addr(&m->seg_cnt[R.rank]), threadIdx.x), n);
    dsmem_st_u32(peer_addr(smem_addr(&m->seg_min[R.rank]), threadIdx.x), kmn);
    dsmem_st_u32(peer_addr(smem_addr(&m->seg_max[R.rank]), threadIdx.x), kmx);
  }
  const uint2* mine = R.cand + off;
  const uint32_t src = smem_addr(R.cand) + 8u * off;
  if (gather) {
    if (R.rank != 0) {
      for (uint32_t i = threadIdx.x; i < n_put; i += T) dsmem_st_v2(peer_addr(src + 8u * i, 0), mine[i]);
    }
    cluster_sync();
    return;
  }
  // (peer, entry) pairs flattened over the threads; peers rank+1 .. rank+nclus-1.
  // x / n_put from a float estimate and one correction (x < 2^22 is exact
  // in a float and the estimate is off by at most one).
  const uint32_t pairs = n_put * (R.nclus - 1);
  const float inv = 1.0f / (float)(n_put > 0 ? n_put : 1u);
  for (uint32_t x = threadIdx.x; x < pairs; x += T) {
    uint32_t d = (uint32_t)((float)x * inv);
    int32_t i = (int32_t)x - (int32_t)(d * n_put);
    if (i < 0) {
      --d;
      i += (int32_t)n_put;
    } else if (i >= (int32_t)n_put) {
      ++d;
      i -= (int32_t)n_put;
    }
    const uint32_t q = (R.rank + 1 + d) & (R.nclus - 1);
    dsmem_st_v2(peer_addr(src + 8u * (uint32_t)i, q), mine[i]);
  }
  cluster_sync();
}

// ------------------------------------------------------------------ position items

// Sample histogram of one round. level 1: top 11 bits of the raw key;
// level 2: the next 11 bits of the items whose top 11 bits equal d1.
template <int T, int U, int W, int kLevel, class Keep>
__device__ __forceinline__ void hist_round(RowCore& R, int r, const float4 (&v)[U],
                                           const int (&n)[Geo<T, U, W>::kSlots], uint32_t d1, Keep keep) {
  using G = Geo<T, U, W>;
#pragma unroll
  for (int s = 0; s < G::kSlots; ++s) {
    const int ns = n[s];
    if (ns == 0 || !keep(R, r, v, s, ns)) continue;
#pragma unroll
    for (int j = 0; j < G::kVS; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (ns == W || 4 * j + e < ns) {
          const uint32_t kk = raw_key(__float_as_uint(lane4(v[s * G::kVS + j], e)));
          if (kLevel == 1) atomicAdd(&R.hist[kk >> 21], 1u);
          else if ((kk >> 21) == d1) atomicAdd(&R.hist[(kk >> 10) & (kBins - 1)], 1u);
        }
      }
  }
}

// Bit mask of this lane's passing positions in round r: bit 4*f + e is
// element e of float4 f (x >= g, or every valid position when `all`), for
// kept slots only.
template <int T, int U, int W, class Keep>
__device__ __forceinline__ uint32_t round_mask(const RowCore& R, int r, const float4 (&v)[U],
                                               const int (&n)[Geo<T, U, W>::kSlots], float g, bool all,
                                               Keep keep) {
  using G = Geo<T, U, W>;
  static_assert(4 * U <= 32, "mask holds 32 positions");
  uint32_t mask = 0;
#pragma unroll
  for (int s = 0; s < G::kSlots; ++s) {
    const int ns = n[s];
    uint32_t sm = 0;
    if (!all) {
      // positions past the slice end hold NaN, which fails x >= g
#pragma unroll
      for (int j = 0; j < G::kVS; ++j) {
        const float4 q = v[s * G::kVS + j];
        const uint32_t b = 4 * j;
        sm |= (q.x >= g ? 1u : 0u) << b;
        sm |= (q.y >= g ? 1u : 0u) << (b + 1);
        sm |= (q.z >= g ? 1u : 0u) << (b + 2);
        sm |= (q.w >= g ? 1u : 0u) << (b + 3);
      }
    } else {
      sm = ns >= 32 ? 0xffffffffu : ((1u << ns) - 1u);
    }
    if (sm != 0 && !keep(R, r, v, s, ns)) sm = 0;
    mask |= sm << (4 * G::kVS * s);
  }
  return mask;
}

// Append the positions of round r flagged in this lane's mask to the list.
// One shared atomic reserves the lane's slots; the lane stages its round in
// its own slots of the warp's staging area (read back by index, by this lane
// only) and walks its set bits, so the warp takes as many steps as its
// busiest lane holds candidates. Bit 4*f + e is element e of float4 f, i.e.
// slot f / kVS, float4 f % kVS. kmn/kmx collect the lane's key range.
template <int T, int U, int W>
__device__ __forceinline__ void extract_lane(const RowCore& R, int r, const float4 (&v)[U], uint32_t mask,
                                             uint32_t* counter, uint2* list, uint32_t cap, uint32_t& kmn,
                                             uint32_t& kmx) {
  using G = Geo<T, U, W>;
  if (mask == 0) return;
  uint32_t o = atomicAdd(counter, (uint32_t)__popc(mask));
  const uint32_t lane = lane_id();
#pragma unroll
  for (int f = 0; f < U; ++f) R.wst[f * 32 + lane] = v[f];
  const float* st = reinterpret_cast<const float*>(R.wst) + 4 * lane;
  // row-relative positions fit 32 bits (a row holds fewer than 2^31)
  const uint32_t p0 = (uint32_t)R.tbase + (uint32_t)r * (uint32_t)G::kTile;
  const uint32_t sstride = (uint32_t)R.rounds * (uint32_t)G::kTile;
  do {
    const uint32_t bit = (uint32_t)(__ffs(mask) - 1);
    mask &= mask - 1u;
    const uint32_t f = bit >> 2, e = bit & 3u;
    const uint32_t kk = key_of(st[128 * f + e]);
    kmn = min(kmn, kk);
    kmx = max(kmx, kk);
    if (o < cap) list[o] = make_uint2(kk, p0 + (f / G::kVS) * sstride + 4 * (f % G::kVS) + e);
    ++o;
  } while (mask);
}

// Fold the warp's key range into the CTA's (local_min / local_max).
__device__ __forceinline__ void flush_key_range(const RowCore& R, uint32_t kmn, uint32_t kmx) {
  kmn = __reduce_min_sync(kFull, kmn);
  kmx = __reduce_max_sync(kFull, kmx);
  if (lane_id() == 0 && kmn <= kmx) {
    atomicMin(&R.m->local_min, kmn);
    atomicMax(&R.m->local_max, kmx);
  }
}

// Append every kept position whose score passes the threshold (x >= g, or
// every valid position when `all`) to the list.
template <int T, int U, int W, class Keep>
__device__ __forceinline__ void filter_round(RowCore& R, int r, const float4 (&v)[U],
                                             const int (&n)[Geo<T, U, W>::kSlots], float g, bool all,
                                             uint32_t* counter, uint2* list, uint32_t cap, Keep keep) {
  uint32_t kmn = 0xffffffffu, kmx = 0u;
  extract_lane<T, U, W>(R, r, v, round_mask<T, U, W>(R, r, v, n, g, all, keep), counter, list, cap, kmn, kmx);
  flush_key_range(R, kmn, kmx);
}

// Per-lane walk over the staged float4s of one or two rounds (see
// filter_rounds_all): bit 4*F + e of mask is element e of staged float4 F,
// float4 F < U being slot F of round r (first position p0 of this lane) and
// F >= U slot F - U of round r + 1. kPos: every flagged score is > 0 (the
// threshold is positive), so its key is its bits with the sign bit set.
template <int T, int U, bool kPos>
__device__ __forceinline__ void walk_lane(const RowCore& R, uint32_t mask, uint32_t p0, uint32_t sstride,
                                          uint32_t* counter, uint2* list, uint32_t cap, uint32_t& kmn,
                                          uint32_t& kmx) {
  constexpr uint32_t kTile = (uint32_t)Geo<T, U, 4>::kTile;
  if (mask == 0) return;
  uint32_t o = atomicAdd(counter, (uint32_t)__popc(mask));
  const float* st = reinterpret_cast<const float*>(R.wst) + 4 * lane_id();
  do {
    const uint32_t bit = (uint32_t)(__ffs(mask) - 1);
    mask &= mask - 1u;
    const uint32_t F = bit >> 2, e = bit & 3u;
    const uint32_t u = __float_as_uint(st[128 * F + e]);
    const uint32_t kk = kPos ? (u | 0x80000000u) : key_of(u);
    kmn = min(kmn, kk);
    kmx = max(kmx, kk);
    const uint32_t pos = p0 + (F >= (uint32_t)U ? kTile : 0u) + (F & (uint32_t)(U - 1)) * sstride + e;
    if (o < cap) list[o] = make_uint2(kk, pos);
    ++o;
  } while (mask);
}

// The streaming filter of the plain top-k (every position kept, W = 4) over
// rounds 0 .. rounds-1, rounds 0 and 1 already in a and b. The two register
// buffers alternate (round r + 2 loads into the buffer round r just left), and
// a round lying wholly inside the slice loads and compares without any
// validity bookkeeping, from per-thread slot pointers. A round's flagged
// lanes stage it in shared memory before its buffer reloads, so the next
// loads leave before the candidates are written; with 16-position rounds
// (U = 4) both rounds of a pair share one walk over a 32-bit mask.
template <int T, int U, bool kPos, class S>
__device__ __forceinline__ void filter_rounds_all(RowT<S>& R, bool vec, float4 (&a)[U], int (&na)[U], float4 (&b)[U],
                                                  int (&nb)[U], float g, bool all, uint32_t* counter, uint2* list,
                                                  uint32_t cap) {
  using G = Geo<T, U, 4>;
  static_assert(G::kSlots == U, "one float4 per slot");
  constexpr bool kPair = 8 * U <= 32;
  const int rounds = R.rounds;
  const uint32_t lane = lane_id();
  auto load = [&](int r, float4 (&v)[U], int (&n)[U]) { load_round4<T, U>(R, vec, r, v, n); };
  // kPos (never "all"): positions past the slice end hold NaN, which fails
  // x >= g, so every round takes the plain compare mask
  auto mask_of = [&](int r, const float4 (&v)[U], const int (&n)[U]) -> uint32_t {
    if (kPos || (!all && round_whole<T, U>(R, r))) return ge_mask<U>(v, g);
    return round_mask<T, U, 4>(R, r, v, n, g, all, KeepAll{});
  };
  auto stage = [&](int F0, const float4 (&v)[U]) {
#pragma unroll
    for (int f = 0; f < U; ++f) R.wst[(F0 + f) * 32 + lane] = v[f];
  };
  const uint32_t q0 = (uint32_t)R.tbase, ss = (uint32_t)rounds * (uint32_t)G::kTile;
  uint32_t kmn = 0xffffffffu, kmx = 0u;
#pragma unroll 1
  for (int r = 0; r < rounds; r += 2) {
    const uint32_t ma = mask_of(r, a, na);
    if (ma) stage(0, a);
    if (r + 2 < rounds) load(r + 2, a, na);
    const uint32_t pr = q0 + (uint32_t)r * (uint32_t)G::kTile;
    if constexpr (kPair) {
      uint32_t mb = 0;
      if (r + 1 < rounds) {
        mb = mask_of(r + 1, b, nb);
        if (mb) stage(U, b);
        if (r + 3 < rounds) load(r + 3, b, nb);
      }
      walk_lane<T, U, kPos>(R, ma | (mb << (4 * U)), pr, ss, counter, list, cap, kmn, kmx);
    } else {
      walk_lane<T, U, kPos>(R, ma, pr, ss, counter, list, cap, kmn, kmx);
      if (r + 1 < rounds) {
        const uint32_t mb = mask_of(r + 1, b, nb);
        if (mb) stage(0, b);
        if (r + 3 < rounds) load(r + 3, b, nb);
        walk_lane<T, U, kPos>(R, mb, pr + (uint32_t)G::kTile, ss, counter, list, cap, kmn, kmx);
      }
    }
  }
  flush_key_range(R, kmn, kmx);
}

// ------------------------------------------------------------------ block items (stage A)

template <int T, int U, int W, int kLevel>
__device__ __forceinline__ void hist_round_blocks(RowCore& R, const float4 (&v)[U],
                                                  const int (&n)[Geo<T, U, W>::kSlots], uint32_t d1) {
#pragma unroll
  for (int s = 0; s < Geo<T, U, W>::kSlots; ++s) {
    if (n[s] == 0) continue;
    const uint32_t kk = slot_block_key<T, U, W>(v, s, n[s]);
    if (kLevel == 1) atomicAdd(&R.hist[kk >> 21], 1u);
    else if ((kk >> 21) == d1) atomicAdd(&R.hist[(kk >> 10) & (kBins - 1)], 1u);
  }
}

template <int T, int U, int W>
__device__ __forceinline__ void filter_round_blocks(RowCore& R, int r, const float4 (&v)[U],
                                                    const int (&n)[Geo<T, U, W>::kSlots], uint32_t t,
                                                    uint32_t* counter, uint2* list, uint32_t cap) {
  uint32_t kmn = 0xffffffffu, kmx = 0u;
#pragma unroll
  for (int s = 0; s < Geo<T, U, W>::kSlots; ++s) {
    const int ns = n[s];
    const uint32_t kk = ns > 0 ? slot_block_key<T, U, W>(v, s, ns) : 0u;
    const bool pe = ns > 0 && kk >= t;
    if (pe) {
      kmn = min(kmn, kk);
      kmx = max(kmx, kk);
    }
    const uint32_t bid = (uint32_t)(slot_pos<T, U, W>(R, r, s) / W);
    warp_append(pe, kk, bid, counter, list, cap);
  }
  kmn = __reduce_min_sync(kFull, kmn);
  kmx = __reduce_max_sync(kFull, kmx);
  if (lane_id() == 0 && kmn <= kmx) {
    atomicMin(&R.m->local_min, kmn);
    atomicMax(&R.m->local_max, kmx);
  }
}

// ------------------------------------------------------------------ local select (radix, fallback)

// Sample-rank target for the threshold estimate. With the whole slice sampled
// the target is exact; otherwise a margin keeps the k-th item above the
// estimated threshold with high probability (a miss only costs the exact path).
__device__ __forceinline__ uint32_t sample_target(uint32_t K, uint32_t ns, int64_t items, bool full) {
  if (full) return K;
  const float lam = (float)K * (float)ns / (float)items;
  const float r = ceilf(1.15f * lam + 3.5f * sqrtf(lam) + 2.0f);
  const uint32_t ri = (uint32_t)fminf(r, (float)ns);
  return ri < 1u ? 1u : ri;
}

template <int T>
__device__ __forceinline__ uint32_t bins_total(const uint32_t* bins, Misc* m) {
  constexpr int BPT = kBins / T;
  uint32_t v[BPT];
  load_bins<T>(bins, v);
  uint32_t s = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) s += v[j];
  return block_sum<T>(s, m);
}

// Exact MSD radix select over the valid candidates: the composite Tc with
// exactly K of them >= Tc. Requires 1 <= K <= number of valid candidates and
// all composites distinct.
template <int T>
__device__ __forceinline__ uint64_t select_local(RowCore& R, uint32_t K, int64_t idx_limit) {
  Misc* m = R.m;
  uint64_t tval = 0, tmask = 0;
  uint32_t need = K;
  for (int di = 0; di < 6; ++di) {
    const int s = digit_shift(di), w = digit_width(di);
    const uint64_t dmask = ((1ull << w) - 1ull) << s;
    if (di == 3 && idx_limit <= (int64_t(1) << 21)) {  // ~index bits 31..21 are all ones
      tval |= dmask;
      tmask |= dmask;
      continue;
    }
    zero_bins<T>(R.hist);
    for_each_cand<T>(R, [&](uint2 e) {
      const uint64_t c = composite(e.x, e.y);
      if ((c & tmask) == tval) atomicAdd(&R.hist[(uint32_t)(c >> s) & ((1u << w) - 1u)], 1u);
    });
    __syncthreads();
    find_digit<T>(R.hist, need, m);
    const uint32_t d = m->res_digit, above = m->res_above, cnt = m->res_cnt;
    need -= above;
    tval |= (uint64_t)d << s;
    tmask |= dmask;
    if (cnt == need) break;
  }
  __syncthreads();
  return tval;
}

// Compact every candidate with composite >= Tc into stage[] (as composites).
template <int T>
__device__ __forceinline__ uint32_t compact_selected(RowCore& R, uint64_t Tc) {
  Misc* m = R.m;
  if (threadIdx.x == 0) m->aux[0] = 0;
  __syncthreads();
  for_each_cand<T>(R, [&](uint2 e) {
    const uint64_t c = composite(e.x, e.y);
    if (c >= Tc) {
      const uint32_t pos = atomicAdd(&m->aux[0], 1u);
      if (pos < R.stage_cap) R.stage[pos] = c;
    }
  });
  __syncthreads();
  const uint32_t cnt = m->aux[0];
  __syncthreads();
  return cnt;
}

// ------------------------------------------------------------------ ordered output

template <class S>
__device__ __forceinline__ void write_slot(int32_t* oi, float* ov, uint32_t slot, uint64_t c, const S* rowp) {
  const uint32_t key = (uint32_t)(c >> 32), idx = ~(uint32_t)c;
  oi[slot] = (int32_t)idx;
  if (ov) ov[slot] = value_of(key, rowp, idx);
}

template <int T>
__device__ __forceinline__ void write_padding(const RowCore& R, int32_t* oi, float* ov, uint32_t K, uint32_t kout) {
  if (R.rank != 0) return;
  for (uint32_t j = K + threadIdx.x; j < kout; j += T) {
    oi[j] = -1;
    if (ov) ov[j] = -__int_as_float(0x7f800000);
  }
}

// Output fallback for candidate sets with heavily populated buckets: radix
// select of the K-th composite, compaction, then a bitonic sort (one CTA or
// large own slices) or a rank count per own item.
template <int T, class S>
__device__ __noinline__ void sorted_fallback(RowT<S> R, bool exact, uint64_t Tc, uint32_t K, uint32_t kout,
                                             int32_t* oi, float* ov, int64_t idx_limit, OwnSlice owner) {
  Misc* m = R.m;
  const uint64_t T64 = exact ? Tc : select_local<T>(R, K, idx_limit);
  compact_selected<T>(R, T64);
  const bool use_sort = (R.nclus == 1) || (K > 64u * R.nclus);
  if (use_sort) {
    uint32_t P = 2;
    while (P < K) P <<= 1;
    for (uint32_t i = K + threadIdx.x; i < P; i += T) R.stage[i] = 0ull;
    __syncthreads();
    bitonic_sort_desc<T>(R.stage, P);
    for (uint32_t j = R.rank + threadIdx.x * R.nclus; j < K; j += T * R.nclus) write_slot(oi, ov, j, R.stage[j], R.rowp);
  } else {
    uint32_t* own = R.aux;
    if (threadIdx.x == 0) m->own_count = 0;
    __syncthreads();
    for (uint32_t base = 0; base < K; base += T) {
      const uint32_t i = base + threadIdx.x;
      const bool mine = (i < K) && owner(~(uint32_t)R.stage[i]);
      const unsigned msk = __ballot_sync(kFull, mine);
      if (msk) {
        const uint32_t lane = lane_id();
        const int leader = __ffs(msk) - 1;
        uint32_t b = 0;
        if ((int)lane == leader) b = atomicAdd(&m->own_count, (uint32_t)__popc(msk));
        b = __shfl_sync(kFull, b, leader);
        const uint32_t pos = b + (uint32_t)__popc(msk & ((1u << lane) - 1u));
        if (mine && pos < (uint32_t)kBins) own[pos] = i;
      }
    }
    __syncthreads();
    const uint32_t n_own = m->own_count < (uint32_t)kBins ? m->own_count : (uint32_t)kBins;
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    for (uint32_t o = warp; o < n_own; o += T / 32) {
      const uint64_t c = R.stage[own[o]];
      uint32_t cnt = 0;
      for (uint32_t j = lane; j < K; j += 32) cnt += (R.stage[j] > c) ? 1u : 0u;
      cnt = __reduce_add_sync(kFull, cnt);
      if (lane == 0 && cnt < kout) write_slot(oi, ov, cnt, c, R.rowp);
    }
  }
  write_padding<T>(R, oi, ov, K, kout);
  __syncthreads();
}

// Select the top K of the valid candidates and write them in order (see step
// 4 at the top of lt_device.cuh). Returns false, having written nothing, when
// some bucket holds more than kMaxBucket candidates. With have_range the
// caller knows the candidates' key range [lo, hi] and count N and the
// histogram is already zero (the fast path clears it before the filter and
// the exchange's barrier follows); otherwise one pass finds them. Expects
// res_max reset.
template <int T, class S>
__device__ __forceinline__ bool bucket_select_sort(RowT<S>& R, uint32_t K, uint32_t kout, int32_t* oi, float* ov,
                                                   OwnSlice owner, bool have_range, uint32_t lo, uint32_t hi,
                                                   uint32_t N) {
  constexpr int NB = kOutBuckets;
  constexpr int BPT = NB / T;
  static_assert(NB % T == 0 && NB <= kBins, "bucket count");
  Misc* m = R.m;
  if (!have_range) {
    uint32_t l = 0xffffffffu, h = 0u, nloc = 0;
    for_each_cand<T>(R, [&](uint2 e) {
      l = min(l, e.x);
      h = max(h, e.x);
      ++nloc;
    });
    nloc = __reduce_add_sync(kFull, nloc);
    l = __reduce_min_sync(kFull, l);
    h = __reduce_max_sync(kFull, h);
    if (lane_id() == 0) {
      atomicMin(&m->kmin, l);
      atomicMax(&m->kmax, h);
      atomicAdd(&m->aux[1], nloc);
    }
    {
      uint4* z = reinterpret_cast<uint4*>(R.hist);
      for (int i = threadIdx.x; i < NB / 4; i += T) z[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    lo = m->kmin;
    hi = m->kmax;
    N = m->aux[1];
  }
  if (hi == lo && N > (uint32_t)kMaxBucket) return false;
  const float scale = (float)NB / ((float)(hi - lo) + 1.0f);
  auto bucket = [lo, scale](uint32_t key) -> uint32_t { return out_bucket(key, lo, scale); };
  for_each_cand<T>(R, [&](uint2 e) { atomicAdd(&R.hist[bucket(e.x)], 1u); });
  __syncthreads();
  // exclusive suffix starts -> aux; the bucket b* holding the K-th item; the
  // largest bucket
  uint32_t v[BPT];
#pragma unroll
  for (int j = 0; j < BPT; ++j) v[j] = R.hist[threadIdx.x * BPT + j];
  uint32_t tot = 0, mx = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    tot += v[j];
    mx = max(mx, v[j]);
  }
  uint32_t a = block_suffix_excl<T>(tot, m);
#pragma unroll
  for (int j = BPT - 1; j >= 0; --j) {
    R.aux[threadIdx.x * BPT + j] = a;
    if (a < K && K <= a + v[j]) {
      m->res_digit = threadIdx.x * BPT + j;
      m->res_above = a;
      m->res_cnt = v[j];
    }
    a += v[j];
  }
  mx = __reduce_max_sync(kFull, mx);
  if (lane_id() == 0) atomicMax(&m->res_max, mx);
  __syncthreads();
  if (m->res_max > (uint32_t)kMaxBucket) return false;
  const uint32_t bstar = m->res_digit, above = m->res_above, cstar = m->res_cnt;
  // scatter the items of buckets >= b* into stage, grouped by bucket
  for_each_cand<T>(R, [&](uint2 e) {
    const uint32_t b = bucket(e.x);
    if (b >= bstar) {
      const uint32_t pos = atomicAdd(&R.aux[b], 1u);
      if (pos < R.stage_cap) R.stage[pos] = composite(e.x, e.y);
    }
  });
  __syncthreads();
  const uint32_t M = above + cstar;
  for (uint32_t i = threadIdx.x; i < M; i += T) {
    const uint64_t c = R.stage[i];
    if (!owner(~(uint32_t)c)) continue;
    const uint32_t b = bucket((uint32_t)(c >> 32));
    const uint32_t e = R.aux[b], s0 = e - R.hist[b];
    uint32_t r = 0;
    for (uint32_t j = s0; j < e; ++j) r += (R.stage[j] > c) ? 1u : 0u;
    const uint32_t rank = s0 + r;
    if (rank < K) write_slot(oi, ov, rank, c, R.rowp);
  }
  write_padding<T>(R, oi, ov, K, kout);
  return true;
}

// ------------------------------------------------------------------ streaming exact select (rare)

// Streaming radix select over this stage's items: 11/11/10-bit digit passes
// over the composites (skipping the constant high bits of ~index), each pass
// re-reading the slice and merging histograms over DSMEM, then one capture
// pass of the K items >= the K-th composite into a flat candidate array.
// Returns that composite. Requires R.init_pending == false.
template <int T, int U, int W, bool kBlocks, class Keep, class S>
__device__ __noinline__ uint64_t exact_select(RowT<S> R, const Params p, uint32_t K, int64_t idx_limit, Keep keep) {
  using G = Geo<T, U, W>;
  Misc* m = R.m;
  const bool vec = p.vec_ok != 0;
  float4 va[U];
  int na[G::kSlots];
  __syncthreads();
  if (threadIdx.x == 0) {
    m->cand_count = 0;
    m->aux[0] = 0;
  }
  __syncthreads();
  uint64_t tval = 0, tmask = 0;
  uint32_t need = K;
  int buf = 0;
  for (int di = 0; di < 6; ++di) {
    const int sh = digit_shift(di), w = digit_width(di);
    const uint64_t dmask = ((1ull << w) - 1ull) << sh;
    const uint32_t wmask = (1u << w) - 1u;
    if (di == 3 && idx_limit <= (int64_t(1) << 21)) {
      tval |= dmask;
      tmask |= dmask;
      continue;
    }
    zero_bins<T>(R.hist);
    for (int r = 0; r < R.rounds; ++r) {
      load_round<T, U, W>(R, vec, r, va, na);
#pragma unroll
      for (int s = 0; s < G::kSlots; ++s) {
        if (na[s] == 0) continue;
        const int64_t pos = slot_pos<T, U, W>(R, r, s);
        if (kBlocks) {
          const uint64_t c = composite(slot_block_key<T, U, W>(va, s, na[s]), (uint32_t)(pos / W));
          if ((c & tmask) == tval) atomicAdd(&R.hist[(uint32_t)(c >> sh) & wmask], 1u);
        } else {
          if (!keep(R, r, va, s, na[s])) continue;
#pragma unroll
          for (int j = 0; j < G::kVS; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int o = 4 * j + e;
              if (o < na[s]) {
                const uint64_t c = composite(key_of(lane4(va[s * G::kVS + j], e)), (uint32_t)(pos + o));
                if ((c & tmask) == tval) atomicAdd(&R.hist[(uint32_t)(c >> sh) & wmask], 1u);
              }
            }
        }
      }
    }
    const uint32_t* bins = merge_hist<T>(R, buf);
    find_digit<T>(bins, need, m);
    const uint32_t d = m->res_digit, above = m->res_above, cnt = m->res_cnt;
    release_merged<T>(R, buf);
    buf ^= 1;
    need -= above;
    tval |= (uint64_t)d << sh;
    tmask |= dmask;
    if (cnt == need) break;
  }
  // capture the K items >= tval into stage[] (local), then into every CTA's
  // candidate array at offsets reserved with remote atomics
  uint2* lst = reinterpret_cast<uint2*>(R.stage);
  const uint32_t lcap = R.stage_cap;
  for (int r = 0; r < R.rounds; ++r) {
    load_round<T, U, W>(R, vec, r, va, na);
#pragma unroll
    for (int s = 0; s < G::kSlots; ++s) {
      const int64_t pos = slot_pos<T, U, W>(R, r, s);
      if (kBlocks) {
        const uint32_t kk = na[s] > 0 ? slot_block_key<T, U, W>(va, s, na[s]) : 0u;
        const uint32_t bid = (uint32_t)(pos / W);
        warp_append(na[s] > 0 && composite(kk, bid) >= tval, kk, bid, &m->aux[0], lst, lcap);
      } else {
        const bool kept = na[s] > 0 && keep(R, r, va, s, na[s]);
#pragma unroll
        for (int j = 0; j < G::kVS; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int o = 4 * j + e;
            const uint32_t kk = key_of(lane4(va[s * G::kVS + j], e));
            const bool pe = kept && o < na[s] && composite(kk, (uint32_t)(pos + o)) >= tval;
            warp_append(pe, kk, (uint32_t)(pos + o), &m->aux[0], lst, lcap);
          }
      }
    }
  }
  __syncthreads();
  const uint32_t n = m->aux[0] < lcap ? m->aux[0] : lcap;
  const uint32_t cap = (uint32_t)p.cap;
  if (R.nclus == 1) {
    for (uint32_t i = threadIdx.x; i < n; i += T) R.cand[i] = lst[i];
    if (threadIdx.x == 0) m->cand_count = n;
    __syncthreads();
  } else {
    if (threadIdx.x < R.nclus)
      m->peer_base[threadIdx.x] = dsmem_atom_add(peer_addr(smem_addr(&m->cand_count), threadIdx.x), n);
    __syncthreads();
    const uint32_t cand_base = smem_addr(R.cand);
    for (uint32_t q = 0; q < R.nclus; ++q) {
      const uint32_t pb = m->peer_base[q];
      const uint32_t dst = peer_addr(cand_base, q);
      for (uint32_t i = threadIdx.x; i < n; i += T)
        if (pb + i < cap) dsmem_st_v2(dst + 8u * (pb + i), lst[i]);
    }
    cluster_sync();
  }
  // flat layout: one segment holding the K captured items
  if (threadIdx.x == 0) {
    reset_candidate_range(m);
    m->nseg = 1;
    m->shift = 31 - __clz(cap);
    m->seg_cnt[0] = m->cand_count < cap ? m->cand_count : cap;
  }
  __syncthreads();
  return tval;
}

// Positions in round 0 of this CTA's slice, from the geometry: round 0 holds
// tiles 0, rounds, 2 rounds, ... (each clipped to the slice).
template <int T, int U, int W>
__device__ __forceinline__ uint32_t round0_size(const RowCore& R) {
  using G = Geo<T, U, W>;
  const int64_t len = R.end - R.begin;
  uint32_t n = 0;
#pragma unroll
  for (int s = 0; s < G::kSlots; ++s) {
    const int64_t t0 = (int64_t)R.rounds * s * G::kTile;
    if (t0 < len) n += (uint32_t)(len - t0 < G::kTile ? len - t0 : G::kTile);
  }
  return n;
}

// Threshold estimate of a single-CTA, 256-thread row from its spread round-0
// sample (not the whole slice) with two 8-bit digit levels of 256 bins, one
// bin per thread: the top 8 bits of the raw key, then the next 8 bits of the
// keys in the chosen bin. The threshold resolves 16 key bits -- 1/128 of an
// octave, each bf16 value its own bin -- with two one-bin-per-thread scans
// instead of 2048-bin ones. Returns the lower edge of the 16-bit bin holding
// the r-th largest sample key.
template <int T, int U, int W>
__device__ __forceinline__ uint32_t estimate_small(RowCore& R, const float4 (&v)[U],
                                                   const int (&n)[Geo<T, U, W>::kSlots], uint32_t K,
                                                   int64_t items) {
  using G = Geo<T, U, W>;
  static_assert(T == 256 && W == 4, "one 8-bit bin per thread, position items");
  Misc* m = R.m;
  uint32_t* h1 = R.hist;
  uint32_t* h2 = R.hist + 256;
  h1[threadIdx.x] = 0u;
  h2[threadIdx.x] = 0u;
  __syncthreads();
  // positions past the slice end hold NaN (raw key 0): counted in the lowest
  // bins, they can only lower the threshold
  (void)n;
#pragma unroll
  for (int s = 0; s < G::kSlots; ++s) {
#pragma unroll
    for (int e = 0; e < 4; ++e) atomicAdd(&h1[raw_key(__float_as_uint(lane4(v[s], e))) >> 24], 1u);
  }
  const uint32_t nsamp = round0_size<T, U, W>(R);
  const uint32_t r = sample_target(K, nsamp, items, false);
  __syncthreads();
  const uint32_t v1[1] = {h1[threadIdx.x]};
  find_rank<T, 1>(v1, r, m);
  const uint32_t d1 = m->res_digit, r2 = r - m->res_above;
#pragma unroll
  for (int s = 0; s < G::kSlots; ++s) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t kk = raw_key(__float_as_uint(lane4(v[s], e)));
      if ((kk >> 24) == d1) atomicAdd(&h2[(kk >> 16) & 255u], 1u);
    }
  }
  __syncthreads();
  const uint32_t v2[1] = {h2[threadIdx.x]};
  find_rank<T, 1>(v2, r2, m);
  return (d1 << 24) | (m->res_digit << 16);
}

// ------------------------------------------------------------------ one selection stage

// Estimate -> filter -> exchange over the items of this stage (positions, or
// blocks when kBlocks); on a miss, the streaming exact select. Returns true
// when the exact select ran (the candidate array then holds exactly the K
// selected items and *Tc is their threshold composite); false on the fast
// path (the candidates are every item >= a lower bound of the K-th item).
// cur/nxt hold rounds 0 and 1 on entry when `loaded`; *regs_intact tells
// whether they still do on return.
//
// hint (nullable): the (k/2)-th and k-th values an earlier row of the batch
// wrote to its output. Rows of one batch score the same context, so from
// lo = k-th and hi = (k/2)-th the filter can start at lo - 0.75 (hi - lo):
// about 1.4k to 1.5k of a similar row pass it (the scores thin out above the
// k-th), a margin of many times the row-to-row spread of the k-th value. The
// estimate is then skipped. Whether it fits is decided by the filter's own
// count check: fewer than K kept or more than the candidate area holds, and
// the row takes the exact path, as any miss does. With hi == lo (ties) the
// margin is a sixteenth of lo; values that give no usable threshold (NaN,
// infinities) keep every position, which the same check settles.
struct Hint {
  float hi, lo;  // the earlier row's (k/2)-th and k-th values
};

__device__ __forceinline__ uint32_t hint_threshold(const Hint& h) {
  // finite (NaN fails every compare); key 0 would mean "keep all"
  if (!(fabsf(h.lo) <= 3.4e38f)) return 0u;
  // with the (k/2)-th value tied to the k-th (scores with few distinct
  // values) the spread gives no margin: one sixteenth of the value instead
  const float t = (h.hi > h.lo && fabsf(h.hi) <= 3.4e38f) ? h.lo - 0.75f * (h.hi - h.lo)
                                                          : h.lo - 0.0625f * fabsf(h.lo);
  if (!(fabsf(t) <= 3.4e38f)) return 0u;
  return key_of(t);
}

template <int T, int U, int W, bool kBlocks, class Keep, class S>
__device__ __forceinline__ bool select_stage(RowT<S>& R, const Params& p, float4 (&cur)[U],
                                             int (&nc)[Geo<T, U, W>::kSlots], float4 (&nxt)[U],
                                             int (&nn)[Geo<T, U, W>::kSlots], bool loaded, uint32_t K,
                                             int64_t items, int64_t idx_limit, Keep keep, bool first,
                                             bool* regs_intact, uint64_t* Tc, int tr, Hint* hint = nullptr) {
  using G = Geo<T, U, W>;
  Misc* m = R.m;
  const bool vec = p.vec_ok != 0;
  if (!first) {
    // A later stage reuses the candidate array: clear the counts, and make
    // sure no peer pushes into it before this CTA has finished with it.
    __syncthreads();
    if (threadIdx.x == 0) {
      m->local_count = 0;
      m->local_min = 0xffffffffu;
      m->local_max = 0u;
      m->cand_count = 0;
    }
    __syncthreads();
    if (R.nclus > 1) {
      wait_init(R);
      cluster_sync();
    }
  }
  const uint32_t seg = 1u << R.seg_shift;
  uint2* list = R.cand + (R.rank << R.seg_shift);
  uint32_t* counter = &m->local_count;
  const uint32_t cap = (uint32_t)p.cap;
  const bool full = R.rounds_max <= 2;
  const bool resident = R.rounds <= 2;
  *regs_intact = resident;
  *Tc = 0;

  if constexpr (!kBlocks && W == 4) {
    if (!loaded) {
      if (R.rounds > 0) load_round4<T, U>(R, vec, 0, cur, nc);
      else clear_round(nc);
      if (R.rounds > 1) load_round4<T, U>(R, vec, 1, nxt, nn);
      else clear_round(nn);
      loaded = true;
      if constexpr (T == 256) {
        // Single-CTA rows of many rounds (the batched rows, three CTAs per
        // SM): the whole slice is asked into L2 at once, so the rounds the
        // registers load later come from L2 while HBM keeps streaming.
        if (R.rounds > 2 && threadIdx.x < 32 && p.host_scores == 0) prefetch_slice_l2(R);
      }
    }
  }
  if (!loaded) {
    // rounds 0 and 1 into cur and nxt (one load site: shift, then load);
    // with a single round, round 0 ends in cur and nxt is empty
    clear_round(nc);
    clear_round(nn);
#pragma unroll 1
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int u = 0; u < U; ++u) cur[u] = nxt[u];
#pragma unroll
      for (int s = 0; s < G::kSlots; ++s) nc[s] = nn[s];
      if (i < R.rounds) load_round<T, U, W>(R, vec, i, nxt, nn);
      else clear_round(nn);
    }
  }

  bool exact = p.force_exact != 0;
  int stat = kCntFast;
  if (!exact && K > 0) {
    // ---- threshold estimate from the digit histogram of the sample
    uint32_t t = 0;
    bool estimated = false;
    bool hinted = false;
    if constexpr (!kBlocks && W == 4 && Keep::kAll) {
      if (hint != nullptr && R.nclus == 1) {
        // from an earlier row's output, taken without a block barrier, so
        // the warps go on filtering at their own pace. Each warp takes its
        // lane 0's reading; that row's CTA may still have been writing it, so
        // the warps' readings are compared after the filter and any
        // difference counts as a miss. An unusable reading gives t = 0
        // (keep everything), which the count check also settles.
        Hint h;
        h.hi = __shfl_sync(kFull, hint->hi, 0);
        h.lo = __shfl_sync(kFull, hint->lo, 0);
        *hint = h;
        if (lane_id() == 0) {
          const uint32_t w[2] = {__float_as_uint(h.hi), __float_as_uint(h.lo)};
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            atomicMin(&m->hint_min[i], w[i]);
            atomicMax(&m->hint_max[i], w[i]);
          }
        }
        t = hint_threshold(h);
        hinted = true;
        estimated = true;
      }
    }
    if constexpr (!kBlocks && T == 256 && W == 4 && Keep::kAll) {
      if (!estimated && items > (int64_t)(cap / 2) && !full && R.nclus == 1) {
        t = estimate_small<T, U, W>(R, cur, nc, K, items);
        estimated = true;
      }
    }
    if (!estimated && items > (int64_t)(cap / 2)) {
      const int nsr = full ? (R.rounds < 2 ? R.rounds : 2) : (R.rounds < 1 ? R.rounds : 1);
      uint32_t r = 0, d1 = 0, above1 = 0;
#pragma unroll 1
      for (int level = 1; level <= 2; ++level) {
        zero_bins<T>(R.hist);
        if (level == 1) {
          if (kBlocks) {
            if (nsr > 0) hist_round_blocks<T, U, W, 1>(R, cur, nc, 0);
            if (nsr > 1) hist_round_blocks<T, U, W, 1>(R, nxt, nn, 0);
          } else {
            if (nsr > 0) hist_round<T, U, W, 1>(R, 0, cur, nc, 0, keep);
            if (nsr > 1) hist_round<T, U, W, 1>(R, 1, nxt, nn, 0, keep);
          }
          stamp(R, tr + kTrHist);
        } else {
          if (kBlocks) {
            if (nsr > 0) hist_round_blocks<T, U, W, 2>(R, cur, nc, d1);
            if (nsr > 1) hist_round_blocks<T, U, W, 2>(R, nxt, nn, d1);
          } else {
            if (nsr > 0) hist_round<T, U, W, 2>(R, 0, cur, nc, d1, keep);
            if (nsr > 1) hist_round<T, U, W, 2>(R, 1, nxt, nn, d1, keep);
          }
        }
        const uint32_t lo_rank = (level == 1 && full && R.nclus >= 8) ? (K < (uint32_t)items ? K : (uint32_t)items) : 0u;
        const uint32_t* bins = merge_hist<T>(R, level - 1, lo_rank);
        if (level == 1) stamp(R, tr + kTrMerge);
        if (level == 1) {
          const uint32_t ns = full ? (uint32_t)items : bins_total<T>(bins, m);
          if (ns == 0) {  // no sample: keep every item
            release_merged<T>(R, 0);
            break;
          }
          r = sample_target(K, ns, items, full);
          find_digit<T>(bins, r, m);
          d1 = m->res_digit;
          above1 = m->res_above;
          const uint32_t cnt1 = m->res_cnt;
          release_merged<T>(R, 0);
          t = d1 << 21;
          const float predicted = full ? (float)(above1 + cnt1)
                                       : (float)(above1 + cnt1) * ((float)items / (float)ns);
          if (predicted <= kLevel2Frac * (float)cap) break;  // one 11-bit level is selective enough
        } else {
          find_digit<T>(bins, r - above1, m);
          t |= m->res_digit << 10;
          release_merged<T>(R, 1);
        }
      }
    }
    stamp(R, tr + kTrEstimate);
    {
      // the output's bucket counts start from zero; the exchange's barrier
      // orders these stores before them
      uint4* z = reinterpret_cast<uint4*>(R.hist);
      for (int i = threadIdx.x; i < kOutBuckets / 4; i += T) z[i] = make_uint4(0, 0, 0, 0);
    }
    // ---- filter every round against the threshold
    const bool all = (t == 0u);
    const float g = threshold_float(all ? 1u : t);
    if (resident) {
      if (R.rounds > 0) {
        if (kBlocks) filter_round_blocks<T, U, W>(R, 0, cur, nc, t, counter, list, seg);
        else filter_round<T, U, W>(R, 0, cur, nc, g, all, counter, list, seg, keep);
      }
      if (R.rounds > 1) {
        if (kBlocks) filter_round_blocks<T, U, W>(R, 1, nxt, nn, t, counter, list, seg);
        else filter_round<T, U, W>(R, 1, nxt, nn, g, all, counter, list, seg, keep);
      }
    } else if constexpr (!kBlocks && W == 4 && Keep::kAll) {
      if (!all && g > 0.0f) filter_rounds_all<T, U, true>(R, vec, cur, nc, nxt, nn, g, all, counter, list, seg);
      else filter_rounds_all<T, U, false>(R, vec, cur, nc, nxt, nn, g, all, counter, list, seg);
    } else {
      // the two register buffers alternate: round r + 2 loads into the buffer
      // round r just left, so two rounds are in flight while one is filtered
#pragma unroll 1
      for (int r = 0; r < R.rounds; r += 2) {
        if (kBlocks) filter_round_blocks<T, U, W>(R, r, cur, nc, t, counter, list, seg);
        else filter_round<T, U, W>(R, r, cur, nc, g, all, counter, list, seg, keep);
        if (r + 2 < R.rounds) load_round<T, U, W>(R, vec, r + 2, cur, nc);
        else clear_round(nc);
        if (r + 1 < R.rounds) {
          if (kBlocks) filter_round_blocks<T, U, W>(R, r + 1, nxt, nn, t, counter, list, seg);
          else filter_round<T, U, W>(R, r + 1, nxt, nn, g, all, counter, list, seg, keep);
          if (r + 3 < R.rounds) load_round<T, U, W>(R, vec, r + 3, nxt, nn);
          else clear_round(nn);
        }
      }
    }
    stamp(R, tr + kTrFilter);
    exchange_segments<T>(R, !kBlocks);
    stamp(R, tr + kTrExchange);
    const uint32_t cq = lane_id() < R.nclus ? m->seg_cnt[lane_id()] : 0u;
    const uint32_t total = __reduce_add_sync(kFull, cq);
    const bool overflow = __any_sync(kFull, cq > seg);
    const bool split_hint = hinted && (m->hint_min[0] != m->hint_max[0] || m->hint_min[1] != m->hint_max[1]);
    if (overflow || total < K || split_hint) {
      if (hinted) bump(p, R, kCntHintMiss);  // the earlier row's threshold does not fit this one
      exact = true;
      stat = overflow ? kCntOverflow : kCntShort;
    } else if (hinted) {
      bump(p, R, kCntHintUsed);
    }
  }

  if (exact && K > 0) {
    if (stat != kCntFast) bump(p, R, stat);
    wait_init(R);
    *Tc = exact_select<T, U, W, kBlocks>(R, p, K, idx_limit, keep);
    *regs_intact = false;
    stamp(R, tr + kTrExact);
    bump(p, R, kCntExact);
    return true;
  }
  stamp(R, tr + kTrExact);
  if (K > 0) bump(p, R, kCntFast);
  return false;
}

// ------------------------------------------------------------------ single-round path

template <int U, int S>
struct RoundRegs {
  float4 v[U];
  int n[S];
};

// Second 11-bit level of the threshold for the single-round path: the next
// 11 key bits of the items in first-level bin d1, merged over the cluster; r2
// is the rank sought inside that bin. Rare (heavily populated first-level
// bins), so it lives out of line and the common path stays compact.
template <int T, int U, int W>
__device__ __noinline__ uint32_t refine_level2(RowCore R, RoundRegs<U, Geo<T, U, W>::kSlots> rr, uint32_t d1,
                                               uint32_t r2) {
  zero_bins<T>(R.hist);
  hist_round<T, U, W, 2>(R, 0, rr.v, rr.n, d1, KeepAll{});
  const uint32_t* bins = merge_hist<T>(R, 1);
  find_digit<T>(bins, r2, R.m);
  const uint32_t d2 = R.m->res_digit;
  release_merged<T>(R, 1);
  return (d1 << 21) | (d2 << 10);
}

// Single-round path: every CTA's slice is one register round, so the sample
// is the whole slice and its histogram is exact. The same steps as
// select_stage (first stage, every position kept) without the second
// register buffer, the streaming filter and the inline second estimate level:
// the code a row executes once per CTA is what its latency pays to fetch.
template <int T, int U, int W, class S>
__device__ __forceinline__ bool select_one(RowT<S>& R, const Params& p, float4 (&v)[U], int (&n)[Geo<T, U, W>::kSlots],
                                           uint32_t K, uint64_t* Tc) {
  using G = Geo<T, U, W>;
  Misc* m = R.m;
  const uint32_t seg = 1u << R.seg_shift;
  uint2* list = R.cand + (R.rank << R.seg_shift);
  const uint32_t cap = (uint32_t)p.cap;
  *Tc = 0;
  if (R.rounds > 0) load_round<T, U, W>(R, p.vec_ok != 0, 0, v, n);
  else clear_round(n);

  bool exact = p.force_exact != 0;
  int stat = kCntFast;
  if (!exact && K > 0) {
    uint32_t t = 0;
    if (R.L > (int64_t)(cap / 2)) {
      zero_bins<T>(R.hist);
      // every position of the round: the NaN fillers past the slice end have
      // raw key 0 and land in bin 0, below any threshold but t = 0 ("all")
#pragma unroll
      for (int u = 0; u < U; ++u) {
        atomicAdd(&R.hist[raw_key(__float_as_uint(v[u].x)) >> 21], 1u);
        atomicAdd(&R.hist[raw_key(__float_as_uint(v[u].y)) >> 21], 1u);
        atomicAdd(&R.hist[raw_key(__float_as_uint(v[u].z)) >> 21], 1u);
        atomicAdd(&R.hist[raw_key(__float_as_uint(v[u].w)) >> 21], 1u);
      }
      stamp(R, kTrHist);
      // K <= L: with large clusters each CTA pushes only the bins at or above
      // its own K-th digit (the cluster's K-th key is at least as large)
      const uint32_t* bins = merge_hist<T>(R, 0, R.nclus >= 8 ? K : 0u);
      stamp(R, kTrMerge);
      find_digit<T>(bins, K, m);
      const uint32_t d1 = m->res_digit, above1 = m->res_above, cnt1 = m->res_cnt;
      release_merged<T>(R, 0);
      t = d1 << 21;
      if ((float)(above1 + cnt1) > kLevel2Frac * (float)cap) {
        RoundRegs<U, G::kSlots> rr;
#pragma unroll
        for (int u = 0; u < U; ++u) rr.v[u] = v[u];
#pragma unroll
        for (int s = 0; s < G::kSlots; ++s) rr.n[s] = n[s];
        t = refine_level2<T, U, W>(R, rr, d1, K - above1);
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
    {
      // positions past the slice end hold NaN, which fails x >= g
      const uint32_t mask = all ? round_mask<T, U, W>(R, 0, v, n, 0.0f, true, KeepAll{})
                                : ge_mask<U>(v, threshold_float(t));
      uint32_t kmn = 0xffffffffu, kmx = 0u;
      extract_lane<T, U, W>(R, 0, v, mask, &m->local_count, list, seg, kmn, kmx);
      flush_key_range(R, kmn, kmx);
    }
    stamp(R, kTrFilter);
    exchange_segments<T>(R, true);
    stamp(R, kTrExchange);
    const uint32_t cq = lane_id() < R.nclus ? m->seg_cnt[lane_id()] : 0u;
    const uint32_t total = __reduce_add_sync(kFull, cq);
    const bool overflow = __any_sync(kFull, cq > seg);
    if (overflow || total < K) {
      exact = true;
      stat = overflow ? kCntOverflow : kCntShort;
    }
  }
  if (exact && K > 0) {
    if (stat != kCntFast) bump(p, R, stat);
    wait_init(R);
    *Tc = exact_select<T, U, W, false>(R, p, K, p.row_stride, KeepAll{});
    stamp(R, kTrExact);
    bump(p, R, kCntExact);
    return true;
  }
  stamp(R, kTrExact);
  if (K > 0) bump(p, R, kCntFast);
  return false;
}

// Select and write the top K positions of this row after select_stage.
// gather: the fast-path exchange gathered every candidate in rank 0, which
// writes the whole row alone; the other CTAs are done.
template <int T, class S>
__device__ __forceinline__ void output_positions(RowT<S>& R0, const Params& p, bool exact, uint64_t Tc, uint32_t K,
                                                 int64_t idx_limit, bool gather) {
  RowT<S> R = R0;
  if (gather && !exact && R.nclus > 1) {
    if (R.rank != 0) {
      stamp(R, kTrOutput);
      return;
    }
    R.nclus = 1;  // rank 0 owns every position
  }
  const uint32_t kout = (uint32_t)p.k;
  int32_t* oi = p.out_idx + R.row * (int64_t)kout;
  float* ov = p.out_val ? p.out_val + R.row * (int64_t)kout : nullptr;
  if (K == 0) {
    write_padding<T>(R, oi, ov, 0, kout);
  } else {
    const OwnSlice own = own_slice(R);
    // fast path: the filter recorded each segment's key range and count
    const Misc* m = R.m;
    uint32_t lo = 0xffffffffu, hi = 0u, n = 0;
    if (!exact) {
      // lane q reads segment q's count and key range
      const uint32_t q = lane_id();
      uint32_t c = 0, mn = 0xffffffffu, mx = 0u;
      if (q < m->nseg) {
        c = min(m->seg_cnt[q], 1u << m->shift);
        if (c) {
          mn = m->seg_min[q];
          mx = m->seg_max[q];
        }
      }
      n = __reduce_add_sync(kFull, c);
      lo = __reduce_min_sync(kFull, mn);
      hi = __reduce_max_sync(kFull, mx);
    }
    if (!bucket_select_sort<T>(R, K, kout, oi, ov, own, !exact, lo, hi, n))
      sorted_fallback<T>(R, exact, Tc, K, kout, oi, ov, idx_limit, own);
  }
  stamp(R, kTrOutput);
}

}  // namespace lt
