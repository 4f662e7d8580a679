// lt_device.cuh -- device primitives of the GB300 (sm_103a) indexer top-k.
//
// One row of indexer scores is owned by one thread-block cluster of C CTAs
// (C = 1 when the batch alone fills the GPU). Each CTA streams its contiguous
// slice of the row with 128-bit loads; the first rounds of the slice stay in
// registers. The selection runs in five steps:
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
//      that bucket is still wide. The result is a key threshold t no larger
//      than the k-th key (exact when the sample is the whole slice).
//   3. filter + candidate exchange. Every key >= t is appended to this CTA's
//      segment of its candidate array (one shared atomic per lane and round
//      that has candidates; the lane then walks its own flagged elements),
//      recording the segment's key range; each CTA then stores its count
//      and key range into every peer and its segment into the same segment
//      of rank 0 over DSMEM, so after one cluster barrier rank 0 holds every
//      candidate. (The two-level kernel's block stage stores segments into
//      every peer: each CTA then writes its own kept blocks.)
//   4. select + order. The candidates are spread over kOutBuckets buckets
//      that are linear in the key between the smallest and largest candidate
//      key; a suffix scan of the bucket counts finds the bucket of the k-th
//      item and the first output slot of every bucket above it; an item's
//      slot is its bucket's first slot plus the number of items of its bucket
//      with a larger composite (key << 32 | ~index). The composite is unique,
//      and among equal keys the larger ~index -- the lower index -- wins: the
//      lowest-index tie fill is the low word of the composite. When a bucket
//      holds more than kMaxBucket items (massive ties), an MSD radix select
//      over the composites and a bitonic sort take over.
//   5. rank 0 writes every slot. (After the exact path every CTA holds the
//      selected items and writes the slots of those from its own slice.)
//
// Every kernel is launched with programmatic dependent launch: it initialises
// shared memory while the previous kernel of its stream finishes, then waits
// for that grid (griddepcontrol.wait) before touching global memory.
//
// When the sampled threshold keeps fewer than k candidates or more than the
// candidate capacity (adversarial orderings, massive ties), the row falls
// back to an exact streaming radix select: 11/11/10-bit passes over the keys
// (and over index digits while ties remain), each pass re-reading the slice
// and merging histograms over DSMEM, then one capture pass. Both paths give
// the same, unique answer.
//
// No kernel here waits on a flag: the only cross-CTA synchronisation is the
// hardware cluster barrier, which every thread of every CTA reaches the same
// number of times (every branch that contains one depends only on values all
// CTAs of the cluster share), and no CTA touches a peer's shared memory after
// the last cluster barrier. The streamed kernel's mbarrier waits are bounded.

#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace lt {

constexpr int kBins = 2048;       // 11-bit digits / linear buckets
constexpr int kMaxCluster = 16;
// Positions a row's block list may cover on the listed kernel: one register
// round of a 512-thread CTA (512 threads x 8 float4).
constexpr int64_t kListedPositions = 512 * 8 * 4;
constexpr int kMaxWarps = 32;
constexpr int kMaxBucket = 256;   // largest bucket ranked by counting
constexpr int kOutBuckets = 1024; // linear key buckets of the ordered output
constexpr int kStageF4 = 8;        // float4 staging slots per lane (two 4-float4 rounds or one of 8)
constexpr unsigned kFull = 0xffffffffu;
// A second 11-bit level refines the sampled threshold only when the first
// predicts more candidates than this fraction of the candidate capacity.
constexpr float kLevel2Frac = 0.75f;

enum Counter {
  kCntFast = 0, kCntExact = 1, kCntOverflow = 2, kCntShort = 3, kCntTimeout = 4,
  kCntHintMiss = 5,  // rows whose threshold from an earlier row did not fit (then redone)
  kCntHintUsed = 6   // rows that finished from a threshold taken from an earlier row
};

// Phase timestamps (nanoseconds of the global timer) written by thread 0 of
// each CTA when a trace buffer is given: slot i of CTA b at trace[b * 16 + i].
constexpr int kTraceSlots = 16;
enum TracePoint {
  kTrStart = 0,     // kernel entry
  kTrHist = 1,      // sample histogram built (rounds 0/1 have arrived)
  kTrMerge = 2,     // first cluster merge done
  kTrEstimate = 3,  // threshold known
  kTrFilter = 4,    // every round filtered
  kTrExchange = 5,  // candidates replicated
  kTrExact = 6,     // streaming radix select done (equal to kTrExchange when not taken)
  kTrOutput = 7,    // outputs written
  kTrStageB = 8     // offset of the second stage of the two-level kernel
};

struct Params {
  const void* scores;   // float, or uint16_t bf16 bits (the kernel's score type)
  const int32_t* lengths;
  int64_t row_stride;
  int32_t* out_idx;
  float* out_val;
  int32_t* out_blocks;
  int32_t* counters;
  int64_t* trace;       // nullable: per-CTA phase timestamps (kTraceSlots per CTA)
  int32_t rows;
  int32_t k;
  int32_t k_blocks;
  int32_t cap;          // candidate slots: clusters * (1 << seg_shift)
  int32_t seg_shift;    // log2 of the candidate slots one CTA may fill
  int32_t sel_cap;      // power of two >= max(k, k_blocks)
  int32_t wstage;       // bytes of the candidate staging area (threads * 16 * kStageF4)
  int32_t force_exact;
  int32_t vec_ok;       // every row start is 16-byte aligned
  int32_t clustered;    // launched with cluster size > 1
  int32_t ring_stages;  // streamed kernel: shared-memory ring stages
  int32_t split;        // two-level kernel: stages run as independent cluster groups
  const int32_t* cand_blocks;  // listed-candidate call: n_cand block ids per row
  int32_t n_cand;
  int32_t external;     // two-level kernel: stage B over the listed blocks only
  int32_t hint_rows;    // > 0: row r starts from the output of row r - hint_rows (batches
                        // of single-CTA rows; see Hint in lt_kernels.cuh), else 0
  int32_t stall_polls;  // streamed kernel, tests only (0 normally): the final chunk of
                        // each CTA is never issued and every wait gives up after
                        // this many polls (see lt_test_inject)
  int32_t host_scores;  // the scores are host memory read over the host link (no L2 bulk prefetch)
};

// ------------------------------------------------------------------ smem layout

struct Misc {
  uint32_t cand_count;   // flat candidate count (streaming exact select)
  uint32_t local_count;  // candidates this CTA appended to its own segment
  uint32_t flags;
  uint32_t own_count;
  uint32_t res_digit, res_above, res_cnt, res_max;
  uint32_t kmin, kmax;   // candidate key range (bucket select)
  uint32_t nseg, shift;  // current candidate layout: nseg segments of 1 << shift slots
  uint32_t local_min, local_max;  // key range of this CTA's candidates (fast path)
  uint32_t seg_cnt[kMaxCluster];  // entries in each segment (may exceed the segment: overflow)
  uint32_t seg_min[kMaxCluster];  // key range of each segment's entries
  uint32_t seg_max[kMaxCluster];
  uint32_t peer_base[kMaxCluster];
  uint32_t warp_a[kMaxWarps];
  uint32_t warp_b[kMaxWarps];
  uint32_t aux[8];
  uint32_t hint_min[2], hint_max[2];  // bits of the warps' hint readings (hi, lo)
};

struct Layout {
  uint32_t misc, hist, aux, merged0, merged1, cand, stage, wstage, total;
};

// Output bucket of a candidate key: kOutBuckets buckets linear in the key
// from lo (every candidate's key is >= lo), clamped at the top. Monotone in
// the key, so a higher bucket never holds a smaller key.
__device__ __forceinline__ uint32_t out_bucket(uint32_t key, uint32_t lo, float scale) {
  const uint32_t b = (uint32_t)((float)(key - lo) * scale);
  return b > (uint32_t)(kOutBuckets - 1) ? (uint32_t)(kOutBuckets - 1) : b;
}

__host__ __device__ inline uint32_t align_up_u32(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// stage holds sel_cap + kMaxBucket composites (bucket scatter, fallback sort).
__host__ __device__ inline Layout make_layout(bool clustered, uint32_t cap, uint32_t sel_cap, uint32_t wstage) {
  Layout l;
  uint32_t o = 0;
  l.misc = o;    o = align_up_u32(o + (uint32_t)sizeof(Misc), 16);
  l.hist = o;    o += kBins * 4;
  l.aux = o;     o += kBins * 4;
  if (clustered) {
    l.merged0 = o; o += kBins * 4;
    l.merged1 = o; o += kBins * 4;
  } else {
    l.merged0 = l.merged1 = l.hist;
  }
  l.cand = o;    o += cap * 8;
  l.stage = o;   o += (sel_cap + kMaxBucket) * 8;
  o = align_up_u32(o, 16);
  l.wstage = o;  o += wstage;
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
__device__ __forceinline__ uint32_t dsmem_atom_add(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.relaxed.cluster.shared::cluster.add.u32 %0, [%1], %2;"
               : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void dsmem_st_v2(uint32_t addr, uint2 v) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" :: "r"(addr), "r"(v.x), "r"(v.y) : "memory");
}

// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization may start while the previous kernel of its stream still runs:
// everything before grid_dependency_wait() overlaps that kernel (so it must
// not touch global memory the previous kernel may write), and the wait returns
// once the previous grid has completed and its writes are visible. Without the
// launch attribute (or with no previous kernel) the wait returns at once.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel of the stream start launching (its CTAs still wait for
// this grid to complete before touching global memory).
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void stamp(const Params& p, int slot) {
  if (p.trace != nullptr && threadIdx.x == 0) {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    p.trace[(int64_t)blockIdx.x * kTraceSlots + slot] = (int64_t)t;
  }
}

// Scores are read as fp32 or as bf16. A bf16 value is the upper half of the
// fp32 with the same sign, exponent and leading seven mantissa bits, so
// widening it is exact: its 16 bits move to the top of a 32-bit word. Every
// later step (keys, compares, copied values) sees the widened fp32.
__device__ __forceinline__ float bf16_widen(uint32_t h) { return __uint_as_float(h << 16); }

__device__ __forceinline__ float load1(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load1(const uint16_t* p) { return bf16_widen(__ldg(p)); }

// Four consecutive scores; p 16-byte (fp32) or 8-byte (bf16) aligned.
// A load that may race with another CTA's store to the same word (the value
// is only used as a guess that is checked afterwards).
__device__ __forceinline__ float ld_relaxed(const float* p) {
  float v;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ float4 ldg4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}
// four bf16 scores as loaded (element 2i in the low half of word i), widened
__device__ __forceinline__ float4 widen4(uint2 q) {
  return make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xffff0000u),
                     __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xffff0000u));
}
__device__ __forceinline__ float4 ldg4(const uint16_t* p) {
  return widen4(__ldg(reinterpret_cast<const uint2*>(p)));
}

// A whole round of vector loads: slot s of this thread starts at
// p0 + s * sstride and holds VS consecutive float4. Every load is issued
// before any of its results is used; bf16 rows keep the raw 64-bit words
// until the last load has left and widen them afterwards (widening each word
// as it arrives would make the next load wait for it).
template <int U, int VS>
__device__ __forceinline__ void gather_round(const float* p0, int64_t sstride, float4 (&v)[U]) {
#pragma unroll
  for (int s = 0; s < U / VS; ++s)
#pragma unroll
    for (int j = 0; j < VS; ++j) v[s * VS + j] = ldg4(p0 + s * sstride + 4 * j);
}
template <int U, int VS>
__device__ __forceinline__ void gather_round(const uint16_t* p0, int64_t sstride, float4 (&v)[U]) {
  uint2 raw[U];
#pragma unroll
  for (int s = 0; s < U / VS; ++s)
#pragma unroll
    for (int j = 0; j < VS; ++j) raw[s * VS + j] = __ldg(reinterpret_cast<const uint2*>(p0 + s * sstride + 4 * j));
#pragma unroll
  for (int i = 0; i < U; ++i) v[i] = widen4(raw[i]);
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

// The same order map without the -0 and NaN fix-ups, for histogram digits
// only: -0 lands one 11-bit bin below +0 and a positive NaN in the top bins.
// Both can only lower the estimated threshold or push the row onto the exact
// path, never change a result.
__device__ __forceinline__ uint32_t raw_key(uint32_t u) {
  return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

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
template <class S>
__device__ __forceinline__ float value_of(uint32_t key, const S* rowp, uint32_t idx) {
  if (key == 0u || key == 0x80000000u) return load1(rowp + idx);
  const uint32_t b = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
  return __uint_as_float(b);
}

// All ones when x >= g (ordered: false for NaN), else zero.
__device__ __forceinline__ uint32_t ge_bits(float x, float g) {
  uint32_t r;
  asm("set.ge.u32.f32 %0, %1, %2;" : "=r"(r) : "f"(x), "f"(g));
  return r;
}

// (a & c) | (b & ~c): the bits of a where c is set, of b elsewhere.
__device__ __forceinline__ uint32_t bit_merge(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

__device__ __forceinline__ float lane4(const float4& q, int e) {
  return e == 0 ? q.x : e == 1 ? q.y : e == 2 ? q.z : q.w;
}

// Bit 4*f + e set when element e of v[f] >= g (NaN never passes): compare i
// gives all ones or zero, and bit i is taken from it while the bits below i
// are kept.
template <int U>
__device__ __forceinline__ uint32_t ge_mask(const float4 (&v)[U], float g) {
  static_assert(4 * U <= 32, "mask holds 32 positions");
  uint32_t m = ge_bits(v[0].x, g);
#pragma unroll
  for (int i = 1; i < 4 * U; ++i) m = bit_merge(m, ge_bits(lane4(v[i / 4], i % 4), g), (1u << i) - 1u);
  return 4 * U == 32 ? m : (m & ((1u << (4 * U)) - 1u));
}

// ------------------------------------------------------------------ warp / block helpers

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t x) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= (uint32_t)o) x += y;
  }
  return x;
}

// Warp-aggregated append of (key, idx) into list[] via counter. All 32 lanes call.
__device__ __forceinline__ void warp_append(bool pred, uint32_t key, uint32_t idx, uint32_t* counter,
                                            uint2* list, uint32_t cap) {
  const unsigned m = __ballot_sync(kFull, pred);
  if (m == 0) return;
  const uint32_t lane = lane_id();
  const int leader = __ffs(m) - 1;
  uint32_t base = 0;
  if ((int)lane == leader) base = atomicAdd(counter, (uint32_t)__popc(m));
  base = __shfl_sync(kFull, base, leader);
  if (pred) {
    const uint32_t pos = base + (uint32_t)__popc(m & ((1u << lane) - 1u));
    if (pos < cap) list[pos] = make_uint2(key, idx);
  }
}

// Block-wide sum: warp sums land in smem, warp 0 adds them, everyone reads
// the result. Ends with __syncthreads.
template <int T>
__device__ __forceinline__ uint32_t block_sum(uint32_t x, Misc* m) {
  constexpr int NW = T / 32;
  x = __reduce_add_sync(kFull, x);
  __syncthreads();
  if (lane_id() == 0) m->warp_a[threadIdx.x >> 5] = x;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t y = threadIdx.x < NW ? m->warp_a[threadIdx.x] : 0u;
    y = __reduce_add_sync(kFull, y);
    if (threadIdx.x == 0) m->warp_b[0] = y;
  }
  __syncthreads();
  return m->warp_b[0];
}

// Each thread owns BPT = kBins / T consecutive bins. Loads them into v[].
template <int T>
__device__ __forceinline__ void load_bins(const uint32_t* bins, uint32_t (&v)[kBins / T]) {
  constexpr int BPT = kBins / T;
  const uint32_t* p = bins + threadIdx.x * BPT;
  if constexpr (BPT % 4 == 0) {
#pragma unroll
    for (int j = 0; j < BPT; j += 4) {
      const uint4 q = *reinterpret_cast<const uint4*>(p + j);
      v[j] = q.x; v[j + 1] = q.y; v[j + 2] = q.z; v[j + 3] = q.w;
    }
  } else if constexpr (BPT == 2) {
    const uint2 q = *reinterpret_cast<const uint2*>(p);
    v[0] = q.x; v[1] = q.y;
  } else {
#pragma unroll
    for (int j = 0; j < BPT; ++j) v[j] = p[j];
  }
}

// Exclusive suffix sum over threads of per-thread totals (the keys in bins
// owned by threads with a larger index). One __syncthreads; each lane then
// reads one warp total and one warp reduction adds those after its warp.
// The caller must __syncthreads before warp_a is written again.
template <int T>
__device__ __forceinline__ uint32_t block_suffix_excl(uint32_t tot, Misc* m) {
  constexpr int NW = T / 32;
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  uint32_t incl = tot;  // sum over lanes >= lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_down_sync(kFull, incl, o);
    if (lane + o < 32) incl += n;
  }
  if (lane == 0) m->warp_a[warp] = incl;
  __syncthreads();
  const uint32_t after = __reduce_add_sync(kFull, (lane > warp && lane < (uint32_t)NW) ? m->warp_a[lane] : 0u);
  return after + (incl - tot);
}

// Exclusive prefix sum over threads of per-thread values (the sum over threads
// with a smaller index). One __syncthreads; the caller must __syncthreads
// before warp_a is written again.
template <int T>
__device__ __forceinline__ uint32_t block_prefix_excl(uint32_t x, Misc* m) {
  static_assert(T % 32 == 0 && T / 32 <= kMaxWarps, "whole warps");
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  const uint32_t incl = warp_incl_scan(x);
  if (lane == 31) m->warp_a[warp] = incl;
  __syncthreads();
  const uint32_t before = __reduce_add_sync(kFull, lane < warp ? m->warp_a[lane] : 0u);
  return before + incl - x;
}

// Thread t owns bins t*BPT .. t*BPT + BPT-1 with counts v[]. Finds the bin d
// with suffix(d + 1) < r <= suffix(d), suffix(d) = sum of bins >= d, for
// 1 <= r <= sum. Warp totals locate the warp holding it; only that warp
// scans its lanes. Results land in m->res_digit / res_above / res_cnt. Ends
// with __syncthreads; the caller must __syncthreads before warp_a is written
// again.
template <int T, int BPT>
__device__ __forceinline__ void find_rank(const uint32_t (&v)[BPT], uint32_t r, Misc* m) {
  constexpr int NW = T / 32;
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  uint32_t tot = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) tot += v[j];
  const uint32_t wsum = __reduce_add_sync(kFull, tot);
  if (lane == 0) m->warp_a[warp] = wsum;
  __syncthreads();
  const uint32_t after_w =
      __reduce_add_sync(kFull, (lane > warp && lane < (uint32_t)NW) ? m->warp_a[lane] : 0u);
  if (after_w < r && r <= after_w + wsum) {
    uint32_t incl = tot;  // sum over lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_down_sync(kFull, incl, o);
      if (lane + o < 32) incl += n;
    }
    uint32_t acc = after_w + incl - tot;
    if (acc < r && r <= acc + tot) {
#pragma unroll
      for (int j = BPT - 1; j >= 0; --j) {
        if (acc + v[j] >= r) {
          m->res_digit = (uint32_t)(threadIdx.x * BPT + j);
          m->res_above = acc;
          m->res_cnt = v[j];
          break;
        }
        acc += v[j];
      }
    }
  }
  __syncthreads();
}

// find_rank over the kBins bins of a histogram.
template <int T>
__device__ __forceinline__ void find_digit(const uint32_t* bins, uint32_t r, Misc* m) {
  uint32_t v[kBins / T];
  load_bins<T>(bins, v);
  find_rank<T, kBins / T>(v, r, m);
}

// Bitonic sort of s[0, n) descending; n a power of two >= 2. Ends with __syncthreads.
template <int T, class E>
__device__ __forceinline__ void bitonic_sort_desc(E* s, uint32_t n) {
  for (uint32_t size = 2; size <= n; size <<= 1) {
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (uint32_t i = threadIdx.x; i < (n >> 1); i += T) {
        const uint32_t lo = 2 * i - (i & (stride - 1));
        const uint32_t hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const E x = s[lo], y = s[hi];
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

}  // namespace lt
