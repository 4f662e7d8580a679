// lt_listed_kernels.cu -- top-k among the positions of a short block list,
// reading only those blocks.
#include "lt_kernels.cuh"
#include "lt_launch.h"

namespace lt {

// The U float4 at block bid[f] * W + off of a row, every one full and aligned.
template <int U>
__device__ __forceinline__ void gather_listed(const float* row, const uint32_t (&bid)[U], int W, int off,
                                              float4 (&v)[U]) {
#pragma unroll
  for (int f = 0; f < U; ++f) v[f] = ldg4(row + (int64_t)bid[f] * W + off);
}
template <int U>
__device__ __forceinline__ void gather_listed(const uint16_t* row, const uint32_t (&bid)[U], int W, int off,
                                              float4 (&v)[U]) {
  uint2 raw[U];
#pragma unroll
  for (int f = 0; f < U; ++f) raw[f] = __ldg(reinterpret_cast<const uint2*>(row + (int64_t)bid[f] * W + off));
#pragma unroll
  for (int f = 0; f < U; ++f) v[f] = widen4(raw[f]);
}

// The unique valid ids of the row's list (at most T * BPT entries: host) in
// ids[0, *n_u) -- in no particular order -- through an open-addressing hash
// set of 2 * T * BPT slots placed after them in the candidate area; *last:
// whether the row's last block is listed. For rows too long for a bitmap of
// their blocks. Probing is bounded: the set is never more than half full.
template <int T, int BPT>
__device__ __noinline__ void listed_ids_hashed(const Params p, const RowCore R, int64_t nblocks, uint32_t* ids,
                                               uint32_t* n_u, bool* last) {
  constexpr uint32_t kSlotsH = 2u * T * BPT;  // a power of two
  constexpr uint32_t kEmpty = 0xffffffffu;
  Misc* m = R.m;
  uint32_t* tab = ids + T * BPT;
  for (uint32_t i = threadIdx.x; i < kSlotsH; i += T) tab[i] = kEmpty;
  if (threadIdx.x == 0) m->aux[1] = 0u;  // the last block seen
  __syncthreads();
  const int32_t* listed = p.cand_blocks + R.row * (int64_t)p.n_cand;
  uint32_t mine[BPT];
  uint32_t cnt = 0;
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    const int32_t j = (int32_t)threadIdx.x + i * T;
    const int32_t b = j < p.n_cand ? __ldg(listed + j) : -1;
    mine[i] = kEmpty;
    if (b >= 0 && (int64_t)b < nblocks) {
      uint32_t h = ((uint32_t)b * 2654435761u) & (kSlotsH - 1u);
      for (uint32_t probe = 0; probe < kSlotsH; ++probe) {
        const uint32_t old = atomicCAS(&tab[h], kEmpty, (uint32_t)b);
        if (old == kEmpty) {  // first occurrence of b
          mine[i] = (uint32_t)b;
          ++cnt;
          if ((int64_t)b == nblocks - 1) m->aux[1] = 1u;
          break;
        }
        if (old == (uint32_t)b) break;  // a repeat
        h = (h + 1u) & (kSlotsH - 1u);
      }
    }
  }
  uint32_t o = block_prefix_excl<T>(cnt, m);
#pragma unroll
  for (int i = 0; i < BPT; ++i)
    if (mine[i] != kEmpty) ids[o++] = mine[i];
  if (threadIdx.x == T - 1) m->aux[0] = o;
  __syncthreads();
  *n_u = m->aux[0];
  *last = m->aux[1] != 0u;
  __syncthreads();
}

// The i-th of a thread's block ids (i < B).
template <int B>
__device__ __forceinline__ uint32_t pick_id(const uint32_t (&a)[B], uint32_t i) {
  uint32_t r = a[0];
#pragma unroll
  for (int j = 1; j < B; ++j) r = (i == (uint32_t)j) ? a[j] : r;
  return r;
}

// One CTA, or one cluster of C CTAs, per row. The row's listed blocks (ids
// outside the row ignored, repeats once) -- at most kListedPositions / W of
// them (host) -- form the ascending unique list, which every CTA of the row
// builds (ascending, from a bitmap of the row's blocks; rows too long for
// one build it unordered in a hash set and run on one CTA); CTA q gathers the
// q-th of C equal shares of it in one register
// round, so the row's scattered reads are spread over C SMs and only the
// listed blocks' scores are read. Then the single-round selection: exact
// 11-bit histogram of the keys of every gathered score (key_of: NaN lowest,
// like the fillers past the list), merged over the cluster, so the threshold
// -- the lower edge of the bin holding the K-th key -- keeps at least K;
// filter; rank 0 gathers the candidates and writes the ordered row. Each
// CTA's segment of the candidate area holds every position of its share, so
// no row can overflow it. Should a filter ever keep fewer than K, it is redone
// keeping every position.
template <int T, int W, class S>
__global__ void __launch_bounds__(T, 1) listed_kernel(Params p) {
  constexpr int U = 8;          // float4 per thread: the round
  constexpr int VS = W / 4;     // float4 per block
  constexpr int BPT = (int)(kListedPositions / W) / T;  // list entries per thread
  constexpr int NW = T / 32;
  using G = Geo<T, U, W>;
  static_assert(BPT >= 1 && BPT * T * W == (int)kListedPositions, "the list divides over the threads");
  (void)sizeof(G);
  extern __shared__ __align__(128) unsigned char smem[];
  RowT<S> R;
  stamp(p, kTrStart);
  grid_dependents_launch();
  setup_row<T, U, W>(R, p, smem);
  Misc* m = R.m;
  const int64_t nblocks = (R.L + W - 1) / W;
  const uint32_t words = (uint32_t)((nblocks + 31) >> 5);
  uint32_t* ids = reinterpret_cast<uint32_t*>(R.cand);
  uint32_t n_u;
  bool last;
  if (words > (uint32_t)kBins) {
    // rows of more than 32 * kBins blocks: the unique listed ids through a
    // hash set in the candidate area instead of a bitmap of the row
    listed_ids_hashed<T, BPT>(p, R, nblocks, ids, &n_u, &last);
  } else {
  // (1) bitmap of the listed blocks, then their ids ascending in the
  // candidate area (free until the filter)
  uint32_t* bits = R.aux;
  for (uint32_t i = threadIdx.x; i < words; i += T) bits[i] = 0u;
  __syncthreads();
  {
    // the list (at most T * BPT entries: host) read with all loads in flight
    const int32_t* listed = p.cand_blocks + R.row * (int64_t)p.n_cand;
    int32_t lb[BPT];
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      const int32_t j = (int32_t)threadIdx.x + i * T;
      lb[i] = j < p.n_cand ? __ldg(listed + j) : -1;
    }
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      const int32_t b = lb[i];
      if (b >= 0 && (int64_t)b < nblocks) atomicOr(&bits[b >> 5], 1u << (b & 31));
    }
  }
  __syncthreads();
  const uint32_t wpt = (words + T - 1) / T;
  const uint32_t w0 = threadIdx.x * wpt;
  const uint32_t w1 = min(w0 + wpt, words);
  uint32_t cnt = 0;
  for (uint32_t w = w0; w < w1; ++w) cnt += (uint32_t)__popc(bits[w]);
  uint32_t o = block_prefix_excl<T>(cnt, m);
  for (uint32_t w = w0; w < w1; ++w)
    for (uint32_t x = bits[w]; x; x &= x - 1u) ids[o++] = 32u * w + (uint32_t)(__ffs(x) - 1);
  if (threadIdx.x == T - 1) m->aux[0] = o;  // the number of unique listed blocks (<= T * BPT: host)
  const int64_t lastb = nblocks - 1;
  last = nblocks > 0 && ((bits[lastb >> 5] >> (lastb & 31)) & 1u) != 0u;
  __syncthreads();
  n_u = m->aux[0];
  }

  // (2) the gathered round over this CTA's share [s0, s1) of the list: its
  // float4 f of lane l of warp w is float4 l % VS of share block
  // f * NW * LPB + w * LPB + l / VS, so the lanes of one load share whole
  // blocks (each 32-byte sector of a block is requested once) and a small
  // share still spreads over every warp. Positions past the share or the row
  // hold NaN; nf[f] counts a float4's valid positions.
  constexpr int LPB = 32 / VS;  // blocks per warp load
  const uint32_t lane = lane_id();
  const uint32_t q = lane % VS;
  const uint32_t per = (n_u + R.nclus - 1) / R.nclus;
  const uint32_t s0 = min(R.rank * per, n_u), s1 = min(s0 + per, n_u);
  const uint32_t ubase = s0 + (threadIdx.x >> 5) * LPB + lane / VS;
  uint32_t bidf[U];
#pragma unroll
  for (int f = 0; f < U; ++f) {
    const uint32_t u = ubase + (uint32_t)f * (uint32_t)(NW * LPB);
    bidf[f] = u < s1 ? ids[u] : 0u;
  }
  __syncthreads();  // the id list is in registers: the candidate area is free
  float4 v[U];
  int nf[U];
  const bool vec = p.vec_ok != 0;
  bool whole = vec;
#pragma unroll
  for (int f = 0; f < U; ++f) {
    const int64_t p0 = (int64_t)bidf[f] * W + 4 * q;
    int64_t nv = ubase + (uint32_t)f * (uint32_t)(NW * LPB) < s1 ? R.L - p0 : 0;
    nv = nv < 0 ? 0 : (nv > 4 ? 4 : nv);
    nf[f] = (int)nv;
    whole = whole && nv == 4;
  }
  if (whole) {
    // every float4 full: all loads in flight before any is used
    gather_listed(R.rowp, bidf, W, 4 * q, v);
  } else {
#pragma unroll
    for (int f = 0; f < U; ++f) {
      const int64_t p0 = (int64_t)bidf[f] * W + 4 * q;
      if (vec && nf[f] == 4) v[f] = ldg4(R.rowp + p0);
      else v[f] = load4_scalar(R.rowp + p0, nf[f]);
    }
  }
  const int64_t ncand = (int64_t)n_u * W - (last ? nblocks * W - R.L : 0);
  const uint32_t K = (uint32_t)(ncand < (int64_t)p.k ? ncand : (int64_t)p.k);
  const uint32_t cap = (uint32_t)p.cap;
  const uint32_t seg = 1u << R.seg_shift;  // this CTA's segment: every position of its share fits
  if (R.nclus > 1 && K > 0 && ncand <= (int64_t)(cap / 2)) {
    // no histogram merge (whose barrier would do it) before the first push
    // into rank 0's candidate area, which held rank 0's id list until now
    wait_init(R);
    cluster_sync();
  }

  if (K > 0) {
    // (3) threshold from the exact histogram of the gathered keys (the NaN
    // fillers have key 0 and land in bin 0, below any threshold but t = 0,
    // "all")
    uint32_t t = 0;
    if (ncand > (int64_t)(cap / 2)) {
      zero_bins<T>(R.hist);
      // the gathered positions only (fillers past a small share would pile
      // up on bin 0)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (nf[u] > 0) atomicAdd(&R.hist[key_of(v[u].x) >> 21], 1u);
        if (nf[u] > 1) atomicAdd(&R.hist[key_of(v[u].y) >> 21], 1u);
        if (nf[u] > 2) atomicAdd(&R.hist[key_of(v[u].z) >> 21], 1u);
        if (nf[u] > 3) atomicAdd(&R.hist[key_of(v[u].w) >> 21], 1u);
      }
      stamp(R, kTrHist);
      // the cluster's histogram; a CTA holding K keys pushes only the bins at
      // or above its own K-th key's (the row's K-th key is no lower)
      const uint32_t* bins = merge_hist<T>(R, 0, R.nclus > 1 ? K : 0u);
      stamp(R, kTrMerge);
      find_digit<T>(bins, K, m);
      t = m->res_digit << 21;
      release_merged<T>(R, 0);
    }
    stamp(R, kTrEstimate);
    {
      // the output's bucket counts start from zero; the exchange's barrier
      // orders these stores before them
      uint4* z = reinterpret_cast<uint4*>(R.hist);
      for (int i = threadIdx.x; i < kOutBuckets / 4; i += T) z[i] = make_uint4(0, 0, 0, 0);
    }
    // (4) filter: every gathered position whose score passes (NaN fillers fail)
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      const bool all = pass == 1 || t == 0u;
      uint32_t mask = 0;
      if (all) {
#pragma unroll
        for (int f = 0; f < U; ++f) mask |= ((1u << nf[f]) - 1u) << (4 * f);
      } else {
        mask = ge_mask<U>(v, threshold_float(t));
      }
      uint32_t kmn = 0xffffffffu, kmx = 0u;
      if (mask) {
        uint2* list = R.cand + (R.rank << R.seg_shift);
        uint32_t oc = atomicAdd(&m->local_count, (uint32_t)__popc(mask));
#pragma unroll
        for (int f = 0; f < U; ++f) R.wst[f * 32 + lane] = v[f];
        const float* st = reinterpret_cast<const float*>(R.wst) + 4 * lane;
        do {
          const uint32_t bit = (uint32_t)(__ffs(mask) - 1);
          mask &= mask - 1u;
          const uint32_t F = bit >> 2, e = bit & 3u;
          const uint32_t kk = key_of(st[128 * F + e]);
          kmn = min(kmn, kk);
          kmx = max(kmx, kk);
          const uint32_t pos = pick_id<U>(bidf, F) * W + 4u * q + e;
          if (oc < seg) list[oc] = make_uint2(kk, pos);
          ++oc;
        } while (mask);
      }
      flush_key_range(R, kmn, kmx);
      stamp(R, kTrFilter);
      // one CTA: segment 0 is the whole list; a cluster gathers to rank 0
      exchange_segments<T>(R, R.nclus > 1);
      stamp(R, kTrExchange);
      const uint32_t cq = lane < R.nclus ? m->seg_cnt[lane] : 0u;
      if (__reduce_add_sync(kFull, cq) >= K) break;
      // fewer than K kept (the threshold above guarantees at least K): start
      // over keeping every position
      __syncthreads();
      if (threadIdx.x == 0) {
        m->local_count = 0;
        m->local_min = 0xffffffffu;
        m->local_max = 0u;
      }
      __syncthreads();
    }
    stamp(R, kTrExact);
    bump(p, R, kCntFast);
  }
  output_positions<T>(R, p, false, 0, K, p.row_stride, R.nclus > 1);
  wait_init(R);
}

template <int T, class S>
const void* listed_ptr(int block) {
  switch (block) {
    case 4: return reinterpret_cast<const void*>(&listed_kernel<T, 4, S>);
    case 8: return reinterpret_cast<const void*>(&listed_kernel<T, 8, S>);
    case 16: return reinterpret_cast<const void*>(&listed_kernel<T, 16, S>);
    case 32: return reinterpret_cast<const void*>(&listed_kernel<T, 32, S>);
    default: return nullptr;
  }
}

const void* listed_kernel_ptr(int threads, int block, bool bf16) {
  if (threads == 512) return bf16 ? listed_ptr<512, uint16_t>(block) : listed_ptr<512, float>(block);
  if (threads == 256) return bf16 ? listed_ptr<256, uint16_t>(block) : listed_ptr<256, float>(block);
  return nullptr;
}

// Listed blocks a row may have on the listed kernel.
int64_t listed_round_blocks(int block) { return kListedPositions / block; }

}  // namespace lt
