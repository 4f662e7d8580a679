// lt_kernels.cuh -- per-row selection machinery shared by the kernels.
//
// Data movement: a CTA's slice [begin, end) of the row is cut into tiles of
// T * W positions (one W-wide slot per thread per tile, W/4 float4 loads). A
// "round" is U float4 per thread. Round r, slot s covers tile r + rounds * s,
// so round 0 is spread over the whole slice and serves as a representative
// sample. Rounds 0 and 1 are loaded up front and kept in registers; later
// rounds stream through the same two register sets. For the top-k kernel
// W = 4 (items are positions); for the two-level kernel W = block (stage A
// items are blocks, stage B items are the positions of the kept blocks).

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

struct Row {
  Misc* m;
  uint32_t* hist;
  uint32_t* aux;
  uint32_t* merged0;     // cluster merge targets (== hist with one CTA)
  uint32_t* merged1;
  uint2* cand;
  uint2* local;
  uint64_t* stage;
  const float* rowp;
  int64_t row;
  int64_t L;             // valid positions of the row
  int64_t begin, end;    // this CTA's slice of positions
  int64_t tbase;         // begin + threadIdx.x * W
  uint32_t rank, nclus;
  uint32_t stage_cap;
  int rounds;            // rounds of this CTA's slice
  int rounds_max;        // cluster-wide maximum
  bool init_pending;     // the start-up cluster barrier has not been waited on
};

__device__ __forceinline__ float nan_f() { return __int_as_float(0x7fffffff); }

template <int T, int U, int W>
__device__ __forceinline__ int64_t slot_pos(const Row& R, int r, int s) {
  return R.tbase + (int64_t)(r + R.rounds * s) * Geo<T, U, W>::kTile;
}

// Load round r; n[s] = valid positions of slot s (a prefix of the slot).
// Invalid positions read as NaN, which no threshold compare accepts.
template <int T, int U, int W>
__device__ __forceinline__ void load_round(const Row& R, bool vec, int r, float4 (&v)[U],
                                           int (&n)[Geo<T, U, W>::kSlots]) {
  using G = Geo<T, U, W>;
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
        float e[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int o = 4 * j + q;
          e[q] = (o < nv) ? __ldg(R.rowp + pos + o) : nan_f();
        }
        v[s * G::kVS + j] = make_float4(e[0], e[1], e[2], e[3]);
      }
    }
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
  constexpr int VS = Geo<T, U, W>::kVS;
  uint32_t best = 0;
#pragma unroll
  for (int j = 0; j < VS; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t kk = key_of(lane4(v[s * VS + j], e));
      if (4 * j + e < nv && kk > best) best = kk;
    }
  return best;
}

struct KeepAll {
  template <class V>
  __device__ __forceinline__ bool operator()(const Row&, int, const V&, int, int) const { return true; }
};

// Stage B of the two-level kernel: keep a slot (one block) when its block
// composite is >= the stage-A threshold composite Tc.
template <int T, int U, int W>
struct KeepBlocks {
  uint64_t Tc;
  __device__ __forceinline__ bool operator()(const Row& R, int r, const float4 (&v)[U], int s, int nv) const {
    const uint32_t bid = (uint32_t)(slot_pos<T, U, W>(R, r, s) / W);
    return composite(slot_block_key<T, U, W>(v, s, nv), bid) >= Tc;
  }
};

// ------------------------------------------------------------------ setup

template <int T, int U, int W>
__device__ __forceinline__ void setup_row(Row& R, const Params& p, unsigned char* smem) {
  using G = Geo<T, U, W>;
  R.nclus = p.clustered ? cluster_size() : 1u;
  R.rank = p.clustered ? cluster_rank() : 0u;
  R.row = (int64_t)(blockIdx.x / R.nclus);
  const Layout lay = make_layout(p.clustered != 0, (uint32_t)p.cap, (uint32_t)p.sel_cap);
  R.m = reinterpret_cast<Misc*>(smem + lay.misc);
  R.hist = reinterpret_cast<uint32_t*>(smem + lay.hist);
  R.aux = reinterpret_cast<uint32_t*>(smem + lay.aux);
  R.merged0 = reinterpret_cast<uint32_t*>(smem + lay.merged0);
  R.merged1 = reinterpret_cast<uint32_t*>(smem + lay.merged1);
  R.cand = reinterpret_cast<uint2*>(smem + lay.cand);
  R.local = reinterpret_cast<uint2*>(smem + lay.local);
  R.stage = reinterpret_cast<uint64_t*>(smem + lay.stage);
  R.stage_cap = (uint32_t)p.sel_cap + kMaxBucket;
  int64_t L = p.row_stride;
  if (p.lengths) {
    L = (int64_t)p.lengths[R.row];
    L = L < 0 ? 0 : (L > p.row_stride ? p.row_stride : L);
  }
  R.L = L;
  R.rowp = p.scores + R.row * p.row_stride;
  int64_t per = (L + R.nclus - 1) / R.nclus;
  per = (per + W - 1) / W * W;
  const int64_t b = (int64_t)R.rank * per;
  R.begin = b < L ? b : L;
  R.end = (R.begin + per) < L ? (R.begin + per) : L;
  R.tbase = R.begin + (int64_t)threadIdx.x * W;
  const int64_t nt = (R.end - R.begin + G::kTile - 1) / G::kTile;
  R.rounds = (int)((nt + G::kSlots - 1) / G::kSlots);
  const int64_t ntm = (per + G::kTile - 1) / G::kTile;
  R.rounds_max = (int)((ntm + G::kSlots - 1) / G::kSlots);

  Misc* m = R.m;
  if (threadIdx.x == 0) {
    m->cand_count = 0;
    m->local_count = 0;
    m->flags = 0;
    m->own_count = 0;
  }
  if (p.clustered) {
    uint4* z0 = reinterpret_cast<uint4*>(R.merged0);
    uint4* z1 = reinterpret_cast<uint4*>(R.merged1);
    for (int i = threadIdx.x; i < kBins / 4; i += T) {
      z0[i] = make_uint4(0, 0, 0, 0);
      z1[i] = make_uint4(0, 0, 0, 0);
    }
  }
  __syncthreads();
  R.init_pending = false;
  if (R.nclus > 1) {
    cluster_arrive();  // "my merged buffers and counters are zero"; waited on before the first push
    R.init_pending = true;
  }
}

__device__ __forceinline__ void finish_row(Row& R) {
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

__device__ __forceinline__ void bump(const Params& p, const Row& R, int which) {
  if (p.counters && R.rank == 0 && threadIdx.x == 0) atomicAdd(&p.counters[which], 1);
}

// ------------------------------------------------------------------ cluster exchange

// Push the non-empty bins of the local histogram into merged buffer `buf` of every
// CTA of the cluster (this one included), then cluster-sync. With one CTA
// the local histogram is the merged one.
template <int T>
__device__ __forceinline__ const uint32_t* merge_hist(Row& R, int buf) {
  __syncthreads();
  if (R.nclus == 1) return R.hist;
  if (R.init_pending) { cluster_wait(); R.init_pending = false; }
  uint32_t* dst = buf ? R.merged1 : R.merged0;
  const uint32_t base = smem_addr(dst);
  for (int b = threadIdx.x; b < kBins; b += T) {
    const uint32_t v = R.hist[b];
    if (v) {
      for (uint32_t q = 0; q < R.nclus; ++q) dsmem_red_add(peer_addr(base + 4u * b, q), v);
    }
  }
  cluster_sync();
  return dst;
}

// After the digit search on merged buffer `buf`: clear it for its next use. Peers only
// write it again after a later cluster barrier.
template <int T>
__device__ __forceinline__ void release_merged(Row& R, int buf) {
  if (R.nclus == 1) return;
  uint4* p = reinterpret_cast<uint4*>(buf ? R.merged1 : R.merged0);
  for (int i = threadIdx.x; i < kBins / 4; i += T) p[i] = make_uint4(0, 0, 0, 0);
}

// Copy the local candidate list into cand[] of every CTA of the cluster, then
// cluster-sync. Afterwards cand[0, cand_count) holds the union (in an order
// that may differ between CTAs) unless an overflow flag is set.
template <int T>
__device__ __forceinline__ void exchange(Row& R, uint32_t cap) {
  __syncthreads();
  if (R.nclus == 1) return;  // single CTA: local == cand, already counted
  if (R.init_pending) { cluster_wait(); R.init_pending = false; }
  Misc* m = R.m;
  const uint32_t n = m->local_count;
  const uint32_t n_put = n < cap ? n : cap;
  if (threadIdx.x < R.nclus) {
    const uint32_t q = threadIdx.x;
    m->peer_base[q] = dsmem_atom_add(peer_addr(smem_addr(&m->cand_count), q), n);
    if (n > cap) dsmem_red_or(peer_addr(smem_addr(&m->flags), q), 1u);
  }
  __syncthreads();
  const uint32_t cand_base = smem_addr(R.cand);
  for (uint32_t q = 0; q < R.nclus; ++q) {
    const uint32_t pb = m->peer_base[q];
    const uint32_t dst = peer_addr(cand_base, q);
    for (uint32_t i = threadIdx.x; i < n_put; i += T) {
      if (pb + i < cap) dsmem_st_v2(dst + 8u * (pb + i), R.local[i]);
    }
  }
  cluster_sync();
}

__device__ __forceinline__ void reset_lists(Row& R) {
  __syncthreads();
  if (threadIdx.x == 0) {
    R.m->cand_count = 0;
    R.m->local_count = 0;
    R.m->flags = 0;
  }
  __syncthreads();
}

// ------------------------------------------------------------------ position items

template <int T, int U, int W, class Keep>
__device__ __forceinline__ void hist_round(Row& R, int r, const float4 (&v)[U],
                                           const int (&n)[Geo<T, U, W>::kSlots], int level,
                                           uint32_t d1, Keep keep) {
  using G = Geo<T, U, W>;
#pragma unroll
  for (int s = 0; s < G::kSlots; ++s) {
    if (n[s] == 0 || !keep(R, r, v, s, n[s])) continue;
#pragma unroll
    for (int j = 0; j < G::kVS; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (4 * j + e < n[s]) {
          const uint32_t kk = key_of(lane4(v[s * G::kVS + j], e));
          if (level == 1) atomicAdd(&R.hist[kk >> 21], 1u);
          else if ((kk >> 21) == d1) atomicAdd(&R.hist[(kk >> 10) & (kBins - 1)], 1u);
        }
      }
  }
}

// Append every kept position whose score passes the threshold (x >= g, or
// every position when `all`) to the list: a bit mask per thread, one warp
// scan and one shared atomic per warp, then each lane writes its own items.
template <int T, int U, int W, class Keep>
__device__ __forceinline__ void filter_round(Row& R, int r, const float4 (&v)[U],
                                             const int (&n)[Geo<T, U, W>::kSlots], float g, bool all,
                                             uint32_t* counter, uint2* list, uint32_t cap, Keep keep) {
  using G = Geo<T, U, W>;
  static_assert(4 * U <= 32, "mask holds 32 positions");
  uint32_t mask = 0;
#pragma unroll
  for (int s = 0; s < G::kSlots; ++s) {
    const bool kept = n[s] > 0 && keep(R, r, v, s, n[s]);
#pragma unroll
    for (int j = 0; j < G::kVS; ++j) {
      const float4 q = v[s * G::kVS + j];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool pe = kept && (4 * j + e < n[s]) && (all || lane4(q, e) >= g);
        mask |= pe ? (1u << (4 * (s * G::kVS + j) + e)) : 0u;
      }
    }
  }
  const uint32_t c = (uint32_t)__popc(mask);
  const uint32_t incl = warp_incl_scan(c);
  const uint32_t total = __shfl_sync(kFull, incl, 31);
  if (total == 0) return;
  uint32_t base = 0;
  if (lane_id() == 31) base = atomicAdd(counter, total);
  base = __shfl_sync(kFull, base, 31);
  uint32_t pos = base + incl - c;
#pragma unroll
  for (int f = 0; f < U; ++f) {
    uint32_t nib = (mask >> (4 * f)) & 15u;
    if (nib) {
      const int64_t p0 = slot_pos<T, U, W>(R, r, f / G::kVS) + 4 * (f % G::kVS);
      const float4 q = v[f];
      do {
        const int e = __ffs(nib) - 1;
        nib &= nib - 1;
        if (pos < cap) list[pos] = make_uint2(key_of(lane4(q, e)), (uint32_t)(p0 + e));
        ++pos;
      } while (nib);
    }
  }
}

// One pass of the streaming radix select: histogram digit (shift s, mask
// wmask) of every kept composite that matches the prefix (tval under tmask).
template <int T, int U, int W, class Keep>
__device__ __forceinline__ void exact_hist_round(Row& R, int r, const float4 (&v)[U],
                                                 const int (&n)[Geo<T, U, W>::kSlots], uint64_t tval,
                                                 uint64_t tmask, int s, uint32_t wmask, Keep keep) {
  using G = Geo<T, U, W>;
#pragma unroll
  for (int sl = 0; sl < G::kSlots; ++sl) {
    if (n[sl] == 0 || !keep(R, r, v, sl, n[sl])) continue;
    const int64_t pos = slot_pos<T, U, W>(R, r, sl);
#pragma unroll
    for (int j = 0; j < G::kVS; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int o = 4 * j + e;
        if (o < n[sl]) {
          const uint64_t c = composite(key_of(lane4(v[sl * G::kVS + j], e)), (uint32_t)(pos + o));
          if ((c & tmask) == tval) atomicAdd(&R.hist[(uint32_t)(c >> s) & wmask], 1u);
        }
      }
  }
}

template <int T, int U, int W, class Keep>
__device__ __forceinline__ void capture_round(Row& R, int r, const float4 (&v)[U],
                                              const int (&n)[Geo<T, U, W>::kSlots], uint64_t Tc,
                                              uint32_t* counter, uint2* list, uint32_t cap, Keep keep) {
  using G = Geo<T, U, W>;
#pragma unroll
  for (int sl = 0; sl < G::kSlots; ++sl) {
    const bool kept = n[sl] > 0 && keep(R, r, v, sl, n[sl]);
    const int64_t pos = slot_pos<T, U, W>(R, r, sl);
#pragma unroll
    for (int j = 0; j < G::kVS; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int o = 4 * j + e;
        const uint32_t kk = key_of(lane4(v[sl * G::kVS + j], e));
        const bool pe = kept && o < n[sl] && composite(kk, (uint32_t)(pos + o)) >= Tc;
        warp_append(pe, kk, (uint32_t)(pos + o), counter, list, cap);
      }
  }
}

// ------------------------------------------------------------------ block items (stage A)

template <int T, int U, int W>
__device__ __forceinline__ void hist_round_blocks(Row& R, const float4 (&v)[U],
                                                  const int (&n)[Geo<T, U, W>::kSlots], int level,
                                                  uint32_t d1) {
#pragma unroll
  for (int s = 0; s < Geo<T, U, W>::kSlots; ++s) {
    if (n[s] == 0) continue;
    const uint32_t kk = slot_block_key<T, U, W>(v, s, n[s]);
    if (level == 1) atomicAdd(&R.hist[kk >> 21], 1u);
    else if ((kk >> 21) == d1) atomicAdd(&R.hist[(kk >> 10) & (kBins - 1)], 1u);
  }
}

template <int T, int U, int W>
__device__ __forceinline__ void filter_round_blocks(Row& R, int r, const float4 (&v)[U],
                                                    const int (&n)[Geo<T, U, W>::kSlots], uint32_t t,
                                                    uint32_t* counter, uint2* list, uint32_t cap) {
#pragma unroll
  for (int s = 0; s < Geo<T, U, W>::kSlots; ++s) {
    const uint32_t kk = n[s] > 0 ? slot_block_key<T, U, W>(v, s, n[s]) : 0u;
    const bool pe = n[s] > 0 && kk >= t;
    const uint32_t bid = (uint32_t)(slot_pos<T, U, W>(R, r, s) / W);
    warp_append(pe, kk, bid, counter, list, cap);
  }
}

template <int T, int U, int W>
__device__ __forceinline__ void exact_hist_round_blocks(Row& R, int r, const float4 (&v)[U],
                                                        const int (&n)[Geo<T, U, W>::kSlots],
                                                        uint64_t tval, uint64_t tmask, int s,
                                                        uint32_t wmask) {
#pragma unroll
  for (int sl = 0; sl < Geo<T, U, W>::kSlots; ++sl) {
    if (n[sl] == 0) continue;
    const uint64_t c = composite(slot_block_key<T, U, W>(v, sl, n[sl]),
                                 (uint32_t)(slot_pos<T, U, W>(R, r, sl) / W));
    if ((c & tmask) == tval) atomicAdd(&R.hist[(uint32_t)(c >> s) & wmask], 1u);
  }
}

template <int T, int U, int W>
__device__ __forceinline__ void capture_round_blocks(Row& R, int r, const float4 (&v)[U],
                                                     const int (&n)[Geo<T, U, W>::kSlots], uint64_t Tc,
                                                     uint32_t* counter, uint2* list, uint32_t cap) {
#pragma unroll
  for (int sl = 0; sl < Geo<T, U, W>::kSlots; ++sl) {
    const uint32_t kk = n[sl] > 0 ? slot_block_key<T, U, W>(v, sl, n[sl]) : 0u;
    const uint32_t bid = (uint32_t)(slot_pos<T, U, W>(R, r, sl) / W);
    const bool pe = n[sl] > 0 && composite(kk, bid) >= Tc;
    warp_append(pe, kk, bid, counter, list, cap);
  }
}

// ------------------------------------------------------------------ local select / output

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

// Exact MSD radix select over cand[0, n): the composite Tc with exactly K
// entries >= Tc. Requires 1 <= K <= n and all composites distinct.
template <int T>
__device__ __forceinline__ uint64_t select_local(Row& R, uint32_t n, uint32_t K, int64_t idx_limit) {
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
    for (uint32_t i = threadIdx.x; i < n; i += T) {
      const uint2 e = R.cand[i];
      const uint64_t c = composite(e.x, e.y);
      if ((c & tmask) == tval) atomicAdd(&R.hist[(uint32_t)(c >> s) & ((1u << w) - 1u)], 1u);
    }
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

// Compact every cand entry with composite >= Tc into stage[] (as composites).
template <int T>
__device__ __forceinline__ uint32_t compact_selected(Row& R, uint32_t n, uint64_t Tc) {
  Misc* m = R.m;
  if (threadIdx.x == 0) m->aux[0] = 0;
  __syncthreads();
  for (uint32_t base = 0; base < n; base += T) {
    const uint32_t i = base + threadIdx.x;
    uint64_t c = 0;
    bool pr = false;
    if (i < n) {
      const uint2 e = R.cand[i];
      c = composite(e.x, e.y);
      pr = c >= Tc;
    }
    const unsigned msk = __ballot_sync(kFull, pr);
    if (msk) {
      const uint32_t lane = lane_id();
      const int leader = __ffs(msk) - 1;
      uint32_t b = 0;
      if ((int)lane == leader) b = atomicAdd(&m->aux[0], (uint32_t)__popc(msk));
      b = __shfl_sync(kFull, b, leader);
      const uint32_t pos = b + (uint32_t)__popc(msk & ((1u << lane) - 1u));
      if (pr && pos < R.stage_cap) R.stage[pos] = c;
    }
  }
  __syncthreads();
  const uint32_t cnt = m->aux[0];
  __syncthreads();
  return cnt;
}

__device__ __forceinline__ void write_slot(int32_t* oi, float* ov, uint32_t slot, uint64_t c, const float* rowp) {
  const uint32_t key = (uint32_t)(c >> 32), idx = ~(uint32_t)c;
  oi[slot] = (int32_t)idx;
  if (ov) ov[slot] = value_of(key, rowp, idx);
}

template <int T>
__device__ __forceinline__ void write_padding(const Row& R, int32_t* oi, float* ov, uint32_t K, uint32_t kout) {
  if (R.rank != 0) return;
  for (uint32_t j = K + threadIdx.x; j < kout; j += T) {
    oi[j] = -1;
    if (ov) ov[j] = -__int_as_float(0x7f800000);
  }
}

// Ordered output from stage[0, K) (any order): bitonic sort when one CTA owns
// the row or own slices are large, else each CTA ranks its own items by counting.
template <int T, class Owner>
__device__ __forceinline__ void write_sorted_fallback(Row& R, uint32_t K, uint32_t kout, int32_t* oi, float* ov,
                                                      Owner owner) {
  Misc* m = R.m;
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

// Select the top K of cand[0, N) and write them in order (see step 4 at the
// top of lt_device.cuh). Returns false, having written nothing, when a bucket
// at or above the k-th item's bucket holds more than kMaxBucket items.
template <int T, class Owner>
__device__ __forceinline__ bool bucket_select_sort(Row& R, uint32_t N, uint32_t K, uint32_t kout, int32_t* oi,
                                                   float* ov, Owner owner) {
  constexpr int BPT = kBins / T;
  Misc* m = R.m;
  uint32_t lo = 0xffffffffu, hi = 0u;
  for (uint32_t i = threadIdx.x; i < N; i += T) {
    const uint32_t kk = R.cand[i].x;
    lo = min(lo, kk);
    hi = max(hi, kk);
  }
  block_minmax<T>(lo, hi, m);
  if (hi == lo && N > (uint32_t)kMaxBucket) return false;
  const float scale = (float)kBins / ((float)(hi - lo) + 1.0f);
  auto bucket = [lo, scale](uint32_t key) -> uint32_t {
    const uint32_t b = (uint32_t)((float)(key - lo) * scale);
    return b > (uint32_t)(kBins - 1) ? (uint32_t)(kBins - 1) : b;
  };
  zero_bins<T>(R.hist);
  for (uint32_t i = threadIdx.x; i < N; i += T) atomicAdd(&R.hist[bucket(R.cand[i].x)], 1u);
  __syncthreads();
  // exclusive suffix starts -> aux; the bucket b* holding the K-th item
  uint32_t v[BPT];
  load_bins<T>(R.hist, v);
  uint32_t tot = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) tot += v[j];
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
  __syncthreads();
  const uint32_t bstar = m->res_digit, above = m->res_above, cstar = m->res_cnt;
  uint32_t mx = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j)
    if (threadIdx.x * BPT + j >= bstar) mx = max(mx, v[j]);
  uint32_t dummy = 0;
  block_minmax<T>(dummy, mx, m);
  if (mx > (uint32_t)kMaxBucket) return false;
  // scatter the items of buckets >= b* into stage, grouped by bucket
  for (uint32_t i = threadIdx.x; i < N; i += T) {
    const uint2 e = R.cand[i];
    const uint32_t b = bucket(e.x);
    if (b >= bstar) {
      const uint32_t pos = atomicAdd(&R.aux[b], 1u);
      if (pos < R.stage_cap) R.stage[pos] = composite(e.x, e.y);
    }
  }
  __syncthreads();
  const uint32_t M = above + cstar;
  for (uint32_t i = threadIdx.x; i < M; i += T) {
    const uint64_t c = R.stage[i];
    if (!owner(~(uint32_t)c)) continue;
    const uint32_t b = bucket((uint32_t)(c >> 32));
    const uint32_t e = R.aux[b], s = e - R.hist[b];
    uint32_t r = 0;
    for (uint32_t j = s; j < e; ++j) r += (R.stage[j] > c) ? 1u : 0u;
    const uint32_t rank = s + r;
    if (rank < K) write_slot(oi, ov, rank, c, R.rowp);
  }
  write_padding<T>(R, oi, ov, K, kout);
  __syncthreads();
  return true;
}

// ------------------------------------------------------------------ one selection stage

// Estimate -> filter -> exchange over the items of this stage (positions, or
// blocks when kBlocks). Returns true when the exact streaming select ran:
// then cand[0, K) holds exactly the selected items and *Tc their threshold
// composite. Returns false on the fast path: cand[0, cand_count) holds every
// item >= a lower bound of the K-th item, with K <= cand_count <= cap.
// va/vb hold rounds 0 and 1 on entry when `loaded`.
template <int T, int U, int W, bool kBlocks, class Keep>
__device__ __forceinline__ bool select_stage(Row& R, const Params& p, float4 (&va)[U],
                                             int (&na)[Geo<T, U, W>::kSlots], float4 (&vb)[U],
                                             int (&nb)[Geo<T, U, W>::kSlots], bool loaded, uint32_t K,
                                             int64_t items, int64_t idx_limit, Keep keep, bool first,
                                             bool* regs_intact, uint64_t* Tc, int tr) {
  Misc* m = R.m;
  const bool vec = p.vec_ok != 0;
  const uint32_t cap = (uint32_t)p.cap;
  if (!first) {
    // A later stage reuses the candidate lists: clear them, and make sure no
    // peer pushes into them before this CTA has finished with the last stage.
    reset_lists(R);
    if (R.nclus > 1) {
      if (R.init_pending) { cluster_wait(); R.init_pending = false; }
      cluster_sync();
    }
  }
  uint32_t* counter = (R.nclus > 1) ? &m->local_count : &m->cand_count;
  uint2* list = (R.nclus > 1) ? R.local : R.cand;
  const bool full = R.rounds_max <= 2;
  *regs_intact = R.rounds <= 2;
  *Tc = 0;

  if (!loaded) {
    if (R.rounds > 0) load_round<T, U, W>(R, vec, 0, va, na); else clear_round(na);
    if (R.rounds > 1) load_round<T, U, W>(R, vec, 1, vb, nb); else clear_round(nb);
  }

  bool exact = p.force_exact != 0;
  int stat = kCntFast;
  if (!exact && K > 0) {
    // ---- threshold estimate from the digit histogram of the sample
    uint32_t t = 0;
    if (items > (int64_t)(cap / 2)) {
      zero_bins<T>(R.hist);
      if (kBlocks) {
        hist_round_blocks<T, U, W>(R, va, na, 1, 0);
        if (full) hist_round_blocks<T, U, W>(R, vb, nb, 1, 0);
      } else {
        hist_round<T, U, W>(R, 0, va, na, 1, 0, keep);
        if (full) hist_round<T, U, W>(R, 1, vb, nb, 1, 0, keep);
      }
      stamp(p, tr + kTrHist);
      const uint32_t* bins = merge_hist<T>(R, 0);
      stamp(p, tr + kTrMerge);
      const uint32_t ns = full ? (uint32_t)items : bins_total<T>(bins, m);
      if (ns > 0) {
        const uint32_t r = sample_target(K, ns, items, full);
        find_digit<T>(bins, r, m);
        const uint32_t d1 = m->res_digit, above1 = m->res_above, cnt1 = m->res_cnt;
        release_merged<T>(R, 0);
        const float predicted = full ? (float)(above1 + cnt1)
                                     : (float)(above1 + cnt1) * ((float)items / (float)ns);
        t = d1 << 21;
        if (predicted > 0.5f * (float)cap) {
          zero_bins<T>(R.hist);
          if (kBlocks) {
            hist_round_blocks<T, U, W>(R, va, na, 2, d1);
            if (full) hist_round_blocks<T, U, W>(R, vb, nb, 2, d1);
          } else {
            hist_round<T, U, W>(R, 0, va, na, 2, d1, keep);
            if (full) hist_round<T, U, W>(R, 1, vb, nb, 2, d1, keep);
          }
          const uint32_t* bins2 = merge_hist<T>(R, 1);
          find_digit<T>(bins2, r - above1, m);
          const uint32_t d2 = m->res_digit;
          release_merged<T>(R, 1);
          t |= d2 << 10;
        }
      } else {
        release_merged<T>(R, 0);
      }
    }
    stamp(p, tr + kTrEstimate);
    // ---- filter every round against the threshold
    const bool all = (t == 0u);
    const float g = threshold_float(all ? 1u : t);
    for (int r = 0; r < R.rounds; r += 2) {
      if (kBlocks) filter_round_blocks<T, U, W>(R, r, va, na, t, counter, list, cap);
      else filter_round<T, U, W>(R, r, va, na, g, all, counter, list, cap, keep);
      if (r + 2 < R.rounds) load_round<T, U, W>(R, vec, r + 2, va, na);
      if (r + 1 < R.rounds) {
        if (kBlocks) filter_round_blocks<T, U, W>(R, r + 1, vb, nb, t, counter, list, cap);
        else filter_round<T, U, W>(R, r + 1, vb, nb, g, all, counter, list, cap, keep);
        if (r + 3 < R.rounds) load_round<T, U, W>(R, vec, r + 3, vb, nb);
      }
    }
    stamp(p, tr + kTrFilter);
    exchange<T>(R, cap);
    stamp(p, tr + kTrExchange);
    const uint32_t N = m->cand_count;
    const bool overflow = (m->flags & 1u) || N > cap;
    if (overflow || N < K) {
      exact = true;
      stat = overflow ? kCntOverflow : kCntShort;
      __syncthreads();
    }
  }

  if (exact && K > 0) {
    // ---- streaming radix select: every pass re-reads the slice
    if (stat != kCntFast) bump(p, R, stat);
    *regs_intact = false;
    reset_lists(R);
    uint64_t tval = 0, tmask = 0;
    uint32_t need = K;
    int buf = 0;
    for (int di = 0; di < 6; ++di) {
      const int s = digit_shift(di), w = digit_width(di);
      const uint64_t dmask = ((1ull << w) - 1ull) << s;
      if (di == 3 && idx_limit <= (int64_t(1) << 21)) {
        tval |= dmask;
        tmask |= dmask;
        continue;
      }
      zero_bins<T>(R.hist);
      for (int r = 0; r < R.rounds; ++r) {
        load_round<T, U, W>(R, vec, r, va, na);
        if (kBlocks) exact_hist_round_blocks<T, U, W>(R, r, va, na, tval, tmask, s, (1u << w) - 1u);
        else exact_hist_round<T, U, W>(R, r, va, na, tval, tmask, s, (1u << w) - 1u, keep);
      }
      const uint32_t* bins = merge_hist<T>(R, buf);
      find_digit<T>(bins, need, m);
      const uint32_t d = m->res_digit, above = m->res_above, cnt = m->res_cnt;
      release_merged<T>(R, buf);
      buf ^= 1;
      need -= above;
      tval |= (uint64_t)d << s;
      tmask |= dmask;
      if (cnt == need) break;
    }
    *Tc = tval;
    for (int r = 0; r < R.rounds; ++r) {
      load_round<T, U, W>(R, vec, r, va, na);
      if (kBlocks) capture_round_blocks<T, U, W>(R, r, va, na, tval, counter, list, cap);
      else capture_round<T, U, W>(R, r, va, na, tval, counter, list, cap, keep);
    }
    exchange<T>(R, cap);
    stamp(p, tr + kTrExact);
    bump(p, R, kCntExact);
    return true;
  }
  stamp(p, tr + kTrExact);
  if (K > 0) bump(p, R, kCntFast);
  return false;
}

// Select and write the top K positions of this row after select_stage.
template <int T, class Owner>
__device__ __forceinline__ void output_positions(Row& R, const Params& p, bool exact, uint64_t Tc, uint32_t K,
                                                 int64_t idx_limit, Owner owner) {
  const uint32_t kout = (uint32_t)p.k;
  int32_t* oi = p.out_idx + R.row * (int64_t)kout;
  float* ov = p.out_val ? p.out_val + R.row * (int64_t)kout : nullptr;
  if (K == 0) {
    write_padding<T>(R, oi, ov, 0, kout);
    return;
  }
  const uint32_t cap = (uint32_t)p.cap;
  const uint32_t N = exact ? K : (R.m->cand_count < cap ? R.m->cand_count : cap);
  if (!bucket_select_sort<T>(R, N, K, kout, oi, ov, owner)) {
    const uint64_t T64 = exact ? Tc : select_local<T>(R, N, K, idx_limit);
    compact_selected<T>(R, N, T64);
    write_sorted_fallback<T>(R, K, kout, oi, ov, owner);
  }
  stamp(p, kTrOutput);
}

__device__ __forceinline__ bool in_slice(const Row& R, uint32_t idx) {
  return (int64_t)idx >= R.begin && (int64_t)idx < R.end;
}

}  // namespace lt
