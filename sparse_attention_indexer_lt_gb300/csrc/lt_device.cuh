// lt_device.cuh -- device code of the GB300 (sm_103a) indexer top-k.
//
// One row of indexer scores is owned by one thread-block cluster of C CTAs
// (C = 1 when there are enough rows to fill the GPU). Each CTA streams its
// contiguous slice of the row with 128-bit loads and keeps the first two
// rounds of it in registers. The selection then runs in five steps:
//
//   1. key transform + digit histogram. Every score maps to an unsigned key
//      that orders like the score (larger key = larger score; -0 -> +0; NaN
//      -> 0, below -inf). Each CTA histograms the top 11 bits of the keys of
//      its sample in shared memory ("each CTA builds a local histogram",
//      AICon 2026 Shenzhen speaker page, outline section 3.2).
//   2. cluster merge. The non-empty bins are added into every CTA's merged
//      histogram with distributed-shared-memory reductions, so the reduce
//      travels over the SM-to-SM network, not HBM (same passage). A suffix
//      scan gives the digit of the k-th key; a second 11-bit level runs when
//      that bucket is still wide. The result is a key threshold t <= the k-th
//      key (exact when the sample is the whole slice).
//   3. filter + candidate exchange. Every key >= t is appended, with warp
//      ballots, to a per-CTA list; the lists are then pushed into every CTA of
//      the cluster, so each CTA holds the same candidate multiset.
//   4. exact select. A most-significant-digit radix select over the unique
//      64-bit composites (key << 32 | ~index) finds the k-th composite T.
//      Everything with composite > (key << 32 | ~0) is strictly above the
//      threshold key; among keys equal to the threshold the larger ~index,
//      i.e. the lower index, wins: the lowest-index tie fill falls out of the
//      low word of the composite.
//   5. ordered output. The k selected composites are ranked (bitonic sort in
//      one CTA, or each CTA counting the ranks of the items from its own
//      slice) and written as (index, score) pairs.
//
// When the sampled threshold keeps fewer than k candidates or more than the
// candidate capacity (adversarial orderings, massive ties), the row falls
// back to an exact streaming radix select: 11/11/10-bit passes over the keys
// (and index digits while ties remain), each pass re-reading the slice and
// merging histograms over DSMEM, then one capture pass. Both paths produce the
// same, unique answer.
//
// No kernel here waits on a flag: the only cross-CTA synchronisation is the
// hardware cluster barrier, which every thread of every CTA reaches the same
// number of times, and no CTA touches a peer's shared memory after the last
// barrier.

#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace lt {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;                    // 11-bit digits
constexpr int kBinsPerThread = kBins / kThreads;
constexpr int kVecPerRound = 8;                // float4 loads per thread per round
constexpr int kMaxCluster = 16;
constexpr unsigned kFull = 0xffffffffu;

enum Counter { kCntFast = 0, kCntExact = 1, kCntOverflow = 2, kCntShort = 3 };

struct Params {
  const float* scores;
  const int32_t* lengths;
  int64_t row_stride;
  int32_t* out_idx;
  float* out_val;
  int32_t* out_blocks;
  int32_t* counters;
  int32_t rows;
  int32_t k;
  int32_t k_blocks;
  int32_t cap;          // candidate capacity per CTA (entries)
  int32_t sel_cap;      // power of two >= max(k, k_blocks)
  int32_t force_exact;
  int32_t vec_ok;       // every row start is 16-byte aligned
  int32_t clustered;    // launched with cluster size > 1
};

// ------------------------------------------------------------------ smem layout

struct Misc {
  uint32_t cand_count;   // entries in cand[] (receives peers' reservations)
  uint32_t local_count;  // entries in local[]
  uint32_t flags;        // bit 0: some CTA's list overflowed
  uint32_t own_count;
  uint32_t res_digit, res_above, res_cnt, res_pad;
  uint32_t warp_tot[kWarps];
  uint32_t peer_base[kMaxCluster];
  uint32_t aux[8];
};

struct Layout {
  uint32_t misc, hist, merged0, merged1, cand, local, sel, total;
};

__host__ __device__ inline uint32_t align_up_u32(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline Layout make_layout(bool clustered, uint32_t cap, uint32_t sel_cap) {
  Layout l;
  uint32_t o = 0;
  l.misc = o;    o = align_up_u32(o + (uint32_t)sizeof(Misc), 16);
  l.hist = o;    o += kBins * 4;
  if (clustered) {
    l.merged0 = o; o += kBins * 4;
    l.merged1 = o; o += kBins * 4;
  } else {
    l.merged0 = l.merged1 = l.hist;
  }
  l.cand = o;    o += cap * 8;
  if (clustered) { l.local = o; o += cap * 8; } else { l.local = l.cand; }
  l.sel = o;     o += sel_cap * 8;
  l.total = align_up_u32(o, 128);
  return l;
}

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() { cluster_arrive(); cluster_wait(); }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void dsmem_red_add(uint32_t addr, uint32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.add.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void dsmem_red_or(uint32_t addr, uint32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.or.b32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t dsmem_atom_add(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.relaxed.cluster.shared::cluster.add.u32 %0, [%1], %2;"
               : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void dsmem_st_v2(uint32_t addr, uint2 v) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" :: "r"(addr), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ float4 ldg4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

// ------------------------------------------------------------------ keys

// Order-preserving float -> uint32: larger key <=> larger score; -0 and +0
// share a key; every NaN maps to 0, below key(-inf) = 0x007fffff.
__device__ __forceinline__ uint32_t key_of(uint32_t u) {
  u = (u == 0x80000000u) ? 0u : u;
  const uint32_t k = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
  return ((u & 0x7fffffffu) > 0x7f800000u) ? 0u : k;
}
__device__ __forceinline__ uint32_t key_of(float x) { return key_of(__float_as_uint(x)); }

__device__ __forceinline__ uint64_t composite(uint32_t key, uint32_t idx) {
  return ((uint64_t)key << 32) | (uint64_t)(~idx);
}

// For t >= 1 and any non-NaN x: key_of(x) >= t  <=>  x >= threshold_float(t).
// NaN never satisfies x >= g, matching key 0 < t.
__device__ __forceinline__ float threshold_float(uint32_t t) {
  if (t <= 0x007fffffu) return -__int_as_float(0x7f800000);  // -inf
  if (t >= 0x80000000u) {
    const uint32_t b = t & 0x7fffffffu;
    return b > 0x7f800000u ? __int_as_float(0x7fffffff) : __uint_as_float(b);
  }
  return __uint_as_float(~t);
}

// Score bits from a key. The key loses the sign of zero and the NaN payload,
// so those two cases re-read the score itself.
__device__ __forceinline__ float value_of(uint32_t key, const float* rowp, uint32_t idx) {
  if (key == 0u || key == 0x80000000u) return rowp[idx];
  const uint32_t b = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
  return __uint_as_float(b);
}

// ------------------------------------------------------------------ block-wide helpers

// Warp-aggregated append of (key, idx) into list[] via counter. All 32 lanes call.
__device__ __forceinline__ void warp_append(bool pred, uint32_t key, uint32_t idx, uint32_t* counter,
                                            uint2* list, uint32_t cap) {
  const unsigned m = __ballot_sync(kFull, pred);
  if (m == 0) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(m) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(counter, (uint32_t)__popc(m));
  base = __shfl_sync(kFull, base, leader);
  if (pred) {
    const uint32_t pos = base + (uint32_t)__popc(m & ((1u << lane) - 1u));
    if (pos < cap) list[pos] = make_uint2(key, idx);
  }
}

// Find digit d with suffix(d + 1) < r <= suffix(d), suffix(d) = sum of bins[b >= d].
// Requires 1 <= r <= sum(bins). Results land in m->res_*. Ends with __syncthreads.
__device__ __forceinline__ void find_digit(const uint32_t* bins, uint32_t r, Misc* m) {
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const uint4 a = reinterpret_cast<const uint4*>(bins)[2 * t];
  const uint4 b = reinterpret_cast<const uint4*>(bins)[2 * t + 1];
  const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t tot = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) tot += v[j];
  uint32_t incl = tot;  // sum over lanes >= lane within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_down_sync(kFull, incl, o);
    if (lane + o < 32) incl += n;
  }
  if (lane == 0) m->warp_tot[warp] = incl;
  __syncthreads();
  uint32_t after = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w)
    if (w > warp) after += m->warp_tot[w];
  uint32_t acc = after + (incl - tot);  // keys in bins owned by threads > t
  if (acc < r && r <= acc + tot) {
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      if (acc + v[j] >= r) {
        m->res_digit = (uint32_t)(t * 8 + j);
        m->res_above = acc;
        m->res_cnt = v[j];
        break;
      }
      acc += v[j];
    }
  }
  __syncthreads();
}

__device__ __forceinline__ uint32_t block_sum(uint32_t x, Misc* m) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  x = __reduce_add_sync(kFull, x);
  __syncthreads();
  if (lane == 0) m->warp_tot[warp] = x;
  __syncthreads();
  uint32_t s = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) s += m->warp_tot[w];
  __syncthreads();
  return s;
}

// Bitonic sort of s[0, n) descending; n a power of two >= 2. Ends with __syncthreads.
template <class T>
__device__ void bitonic_sort_desc(T* s, uint32_t n) {
  for (uint32_t size = 2; size <= n; size <<= 1) {
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (uint32_t i = threadIdx.x; i < (n >> 1); i += kThreads) {
        const uint32_t lo = 2 * i - (i & (stride - 1));
        const uint32_t hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const T x = s[lo], y = s[hi];
        if ((x < y) == desc) { s[lo] = y; s[hi] = x; }
      }
      __syncthreads();
    }
  }
}

// Digits of the 64-bit composite, most significant first: the key in
// 11/11/10 bits, then ~index in 11/11/10 bits.
__device__ __forceinline__ int digit_shift(int i) {
  return i == 0 ? 53 : i == 1 ? 42 : i == 2 ? 32 : i == 3 ? 21 : i == 4 ? 10 : 0;
}
__device__ __forceinline__ int digit_width(int i) { return (i == 2 || i == 5) ? 10 : 11; }

// ------------------------------------------------------------------ per-row context

struct Row {
  Misc* m;
  uint32_t* hist;
  uint32_t* merged[2];
  uint2* cand;
  uint2* local;
  unsigned char* sel;    // uint64_t[sel_cap] or uint32_t[2 * sel_cap]
  const float* rowp;
  int64_t row;
  int64_t L;             // valid positions of the row
  int64_t begin, end;    // this CTA's slice of positions
  int64_t chunk;
  uint32_t rank, nclus;
  int rounds;            // rounds of this CTA's slice
  int rounds_max;        // cluster-wide maximum
  bool init_pending;     // the start-up cluster barrier has not been waited on
  uint32_t sel_cap;      // entries of sel[]
};

// Push the non-empty bins of the local histogram into merged[buf] of every CTA
// of the cluster (including this one), then cluster-sync. With one CTA the
// local histogram is the merged one. Returns the merged bins.
__device__ __forceinline__ const uint32_t* merge_hist(Row& R, int buf) {
  __syncthreads();
  if (R.nclus == 1) return R.hist;
  if (R.init_pending) { cluster_wait(); R.init_pending = false; }
  const uint32_t base = smem_addr(R.merged[buf]);
  for (int b = threadIdx.x; b < kBins; b += kThreads) {
    const uint32_t v = R.hist[b];
    if (v) {
      for (uint32_t q = 0; q < R.nclus; ++q) dsmem_red_add(peer_addr(base + 4u * b, q), v);
    }
  }
  cluster_sync();
  return R.merged[buf];
}

// After the digit search on merged[buf]: clear it for its next use. Peers only
// write it again after a later cluster barrier.
__device__ __forceinline__ void release_merged(Row& R, int buf) {
  if (R.nclus == 1) return;
  uint4* p = reinterpret_cast<uint4*>(R.merged[buf]);
  for (int i = threadIdx.x; i < kBins / 4; i += kThreads) p[i] = make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ void zero_hist(Row& R) {
  uint4* p = reinterpret_cast<uint4*>(R.hist);
  for (int i = threadIdx.x; i < kBins / 4; i += kThreads) p[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
}

// Copy the local candidate list into cand[] of every CTA of the cluster, then
// cluster-sync. Afterwards cand[0, cand_count) holds the union (in an order
// that may differ between CTAs) unless an overflow flag is set.
__device__ inline void exchange(Row& R, uint32_t cap) {
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
    for (uint32_t i = threadIdx.x; i < n_put; i += kThreads) {
      if (pb + i < cap) dsmem_st_v2(dst + 8u * (pb + i), R.local[i]);
    }
  }
  cluster_sync();
}

// Exact radix select over cand[0, n): the composite T with exactly K entries
// >= T. Requires 1 <= K <= n and all composites distinct.
__device__ inline uint64_t select_local(Row& R, uint32_t n, uint32_t K, int64_t idx_limit) {
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
    zero_hist(R);
    for (uint32_t i = threadIdx.x; i < n; i += kThreads) {
      const uint2 e = R.cand[i];
      const uint64_t c = composite(e.x, e.y);
      if ((c & tmask) == tval) atomicAdd(&R.hist[(uint32_t)(c >> s) & ((1u << w) - 1u)], 1u);
    }
    __syncthreads();
    find_digit(R.hist, need, m);
    const uint32_t d = m->res_digit, above = m->res_above, cnt = m->res_cnt;
    need -= above;
    tval |= (uint64_t)d << s;
    tmask |= dmask;
    if (cnt == need) break;
  }
  __syncthreads();
  return tval;
}

// Compact every cand entry with composite >= T into sel (as composites).
__device__ inline uint32_t compact_selected(Row& R, uint32_t n, uint64_t T) {
  Misc* m = R.m;
  if (threadIdx.x == 0) m->aux[0] = 0;
  __syncthreads();
  uint64_t* sel = reinterpret_cast<uint64_t*>(R.sel);
  for (uint32_t base = 0; base < n; base += kThreads) {
    const uint32_t i = base + threadIdx.x;
    uint64_t c = 0;
    bool p = false;
    if (i < n) {
      const uint2 e = R.cand[i];
      c = composite(e.x, e.y);
      p = c >= T;
    }
    const unsigned msk = __ballot_sync(kFull, p);
    if (msk) {
      const int lane = threadIdx.x & 31, leader = __ffs(msk) - 1;
      uint32_t b = 0;
      if (lane == leader) b = atomicAdd(&m->aux[0], (uint32_t)__popc(msk));
      b = __shfl_sync(kFull, b, leader);
      const uint32_t pos = b + (uint32_t)__popc(msk & ((1u << lane) - 1u));
      if (p && pos < R.sel_cap) sel[pos] = c;
    }
  }
  __syncthreads();
  const uint32_t cnt = m->aux[0];
  __syncthreads();
  return cnt;
}

}  // namespace lt
