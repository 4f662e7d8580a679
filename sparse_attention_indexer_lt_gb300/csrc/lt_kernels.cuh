// lt_kernels.cuh -- the top-k and two-level top-k kernels (sm_103a).
//
// Data movement: a CTA's slice [begin, end) of the row is cut into tiles of
// kThreads * W positions (one W-wide slot per thread per tile, W/4 float4
// loads). A "round" is kSlots tiles, i.e. kVecPerRound float4 per thread.
// Round r, slot u covers tile r + rounds * u, so the first rounds are spread
// over the whole slice (a representative sample). Rounds 0 and 1 are loaded
// up front and stay in registers; later rounds stream through the same two
// register sets. For the top-k kernel W = 4 (items are positions); for the
// two-level kernel W = block (stage A items are blocks, stage B items are the
// positions of the kept blocks).

#pragma once

#include "lt_device.cuh"

namespace lt {

template <int W>
struct Geo {
  static constexpr int kVecPerSlot = W / 4;
  static constexpr int kSlots = kVecPerRound / kVecPerSlot;
  static constexpr int64_t kTile = (int64_t)kThreads * W;
};

__device__ __forceinline__ float nanf_bits() { return __int_as_float(0x7fffffff); }

__device__ __forceinline__ float lane4(const float4& q, int e) {
  return e == 0 ? q.x : e == 1 ? q.y : e == 2 ? q.z : q.w;
}

// Position of slot u of round r for this thread.
template <int W>
__device__ __forceinline__ int64_t slot_pos(const Row& R, int r, int u) {
  const int64_t tile = (int64_t)r + (int64_t)R.rounds * u;
  return R.begin + (tile * kThreads + threadIdx.x) * W;
}

// Load round r into v; n[u] = valid positions of slot u (a prefix of the slot).
// Invalid positions read as NaN so that no threshold compare accepts them.
template <int W>
__device__ __forceinline__ void load_round(const Row& R, const Params& p, int r, float4 (&v)[kVecPerRound],
                                           int (&n)[Geo<W>::kSlots]) {
  constexpr int VS = Geo<W>::kVecPerSlot;
  const int64_t ntiles = (R.end - R.begin + Geo<W>::kTile - 1) / Geo<W>::kTile;
#pragma unroll
  for (int u = 0; u < Geo<W>::kSlots; ++u) {
    const int64_t tile = (int64_t)r + (int64_t)R.rounds * u;
    const int64_t pos = R.begin + (tile * kThreads + threadIdx.x) * W;
    int64_t nv = (tile < ntiles && r < R.rounds) ? R.end - pos : 0;
    nv = nv < 0 ? 0 : (nv > W ? W : nv);
    n[u] = (int)nv;
    if (nv == W && p.vec_ok) {
#pragma unroll
      for (int j = 0; j < VS; ++j) v[u * VS + j] = ldg4(R.rowp + pos + 4 * j);
    } else {
#pragma unroll
      for (int j = 0; j < VS; ++j) {
        float e[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int o = 4 * j + q;
          e[q] = (o < nv) ? __ldg(R.rowp + pos + o) : nanf_bits();
        }
        v[u * VS + j] = make_float4(e[0], e[1], e[2], e[3]);
      }
    }
  }
}

template <int W>
__device__ __forceinline__ void clear_round(int (&n)[Geo<W>::kSlots]) {
#pragma unroll
  for (int u = 0; u < Geo<W>::kSlots; ++u) n[u] = 0;
}

// Key of the block held in slot u (max of the keys of its valid positions).
template <int W>
__device__ __forceinline__ uint32_t slot_block_key(const float4 (&v)[kVecPerRound], int u, int nv) {
  constexpr int VS = Geo<W>::kVecPerSlot;
  uint32_t best = 0;
#pragma unroll
  for (int j = 0; j < VS; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t kk = key_of(lane4(v[u * VS + j], e));
      if (4 * j + e < nv && kk > best) best = kk;
    }
  }
  return best;
}

// ------------------------------------------------------------------ common setup

template <int W>
__device__ __forceinline__ void setup_row(Row& R, const Params& p, unsigned char* smem) {
  R.nclus = p.clustered ? cluster_size() : 1u;
  R.rank = p.clustered ? cluster_rank() : 0u;
  R.row = (int64_t)(blockIdx.x / R.nclus);
  const Layout lay = make_layout(p.clustered != 0, (uint32_t)p.cap, (uint32_t)p.sel_cap);
  R.m = reinterpret_cast<Misc*>(smem + lay.misc);
  R.hist = reinterpret_cast<uint32_t*>(smem + lay.hist);
  R.merged[0] = reinterpret_cast<uint32_t*>(smem + lay.merged0);
  R.merged[1] = reinterpret_cast<uint32_t*>(smem + lay.merged1);
  R.cand = reinterpret_cast<uint2*>(smem + lay.cand);
  R.local = reinterpret_cast<uint2*>(smem + lay.local);
  R.sel = smem + lay.sel;
  R.sel_cap = (uint32_t)p.sel_cap;
  int64_t L = p.row_stride;
  if (p.lengths) {
    L = (int64_t)p.lengths[R.row];
    L = L < 0 ? 0 : (L > p.row_stride ? p.row_stride : L);
  }
  R.L = L;
  R.rowp = p.scores + R.row * p.row_stride;
  int64_t per = (L + R.nclus - 1) / R.nclus;
  per = (per + W - 1) / W * W;
  R.chunk = per;
  const int64_t b = (int64_t)R.rank * per;
  R.begin = b < L ? b : L;
  R.end = (R.begin + per) < L ? (R.begin + per) : L;
  const int64_t nt = (R.end - R.begin + Geo<W>::kTile - 1) / Geo<W>::kTile;
  R.rounds = (int)((nt + Geo<W>::kSlots - 1) / Geo<W>::kSlots);
  const int64_t ntm = (per + Geo<W>::kTile - 1) / Geo<W>::kTile;
  R.rounds_max = (int)((ntm + Geo<W>::kSlots - 1) / Geo<W>::kSlots);

  Misc* m = R.m;
  if (threadIdx.x == 0) {
    m->cand_count = 0;
    m->local_count = 0;
    m->flags = 0;
    m->own_count = 0;
  }
  if (p.clustered) {
    uint4* z0 = reinterpret_cast<uint4*>(R.merged[0]);
    uint4* z1 = reinterpret_cast<uint4*>(R.merged[1]);
    for (int i = threadIdx.x; i < kBins / 4; i += kThreads) {
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

__device__ __forceinline__ void reset_lists(Row& R) {
  __syncthreads();
  if (threadIdx.x == 0) {
    R.m->cand_count = 0;
    R.m->local_count = 0;
    R.m->flags = 0;
  }
  __syncthreads();
}

// Sample-rank target for the threshold estimate. With the whole slice sampled
// the target is exact; otherwise a margin keeps the k-th item above the
// estimated threshold with high probability (a miss only costs the exact path).
__device__ __forceinline__ uint32_t sample_target(uint32_t K, uint32_t ns, int64_t items, bool full) {
  if (full) return K;
  const float lam = (float)K * (float)ns / (float)items;
  float r = ceilf(1.15f * lam + 3.5f * sqrtf(lam) + 2.0f);
  uint32_t ri = (uint32_t)fminf(r, (float)ns);
  return ri < 1u ? 1u : ri;
}

__device__ __forceinline__ uint32_t bins_total(const uint32_t* bins, Misc* m) {
  const uint4 a = reinterpret_cast<const uint4*>(bins)[2 * threadIdx.x];
  const uint4 b = reinterpret_cast<const uint4*>(bins)[2 * threadIdx.x + 1];
  return block_sum(a.x + a.y + a.z + a.w + b.x + b.y + b.z + b.w, m);
}

__device__ __forceinline__ void bump(const Params& p, const Row& R, int which) {
  if (p.counters && R.rank == 0 && threadIdx.x == 0) atomicAdd(&p.counters[which], 1);
}

// ------------------------------------------------------------------ ordered output

// Write the K selected composites of sel[] (any order) to out_idx/out_val of
// this row in (score desc, index asc) order, padding slots [K, k).
// owner(idx) tells whether this CTA owns an item in the counting scheme.
template <class Owner>
__device__ void write_ordered(Row& R, const Params& p, uint32_t K, uint32_t kout, Owner owner) {
  Misc* m = R.m;
  uint64_t* sel = reinterpret_cast<uint64_t*>(R.sel);
  int32_t* oi = p.out_idx + R.row * (int64_t)kout;
  float* ov = p.out_val ? p.out_val + R.row * (int64_t)kout : nullptr;
  const bool use_sort = (R.nclus == 1) || (K > 64u * R.nclus);
  if (use_sort) {
    uint32_t P = 2;
    while (P < K) P <<= 1;
    for (uint32_t i = K + threadIdx.x; i < P; i += kThreads) sel[i] = 0ull;
    __syncthreads();
    bitonic_sort_desc(sel, P);
    for (uint32_t j = R.rank + threadIdx.x * R.nclus; j < kout; j += kThreads * R.nclus) {
      if (j < K) {
        const uint64_t c = sel[j];
        const uint32_t key = (uint32_t)(c >> 32), idx = ~(uint32_t)c;
        oi[j] = (int32_t)idx;
        if (ov) ov[j] = value_of(key, R.rowp, idx);
      } else {
        oi[j] = -1;
        if (ov) ov[j] = -__int_as_float(0x7f800000);
      }
    }
  } else {
    // each CTA ranks the selected items of its own slice by counting
    uint32_t* own = R.hist;  // free after the select
    if (threadIdx.x == 0) m->own_count = 0;
    __syncthreads();
    for (uint32_t base = 0; base < K; base += kThreads) {
      const uint32_t i = base + threadIdx.x;
      const bool mine = (i < K) && owner(~(uint32_t)sel[i]);
      const unsigned msk = __ballot_sync(kFull, mine);
      if (msk) {
        const int lane = threadIdx.x & 31, leader = __ffs(msk) - 1;
        uint32_t b = 0;
        if (lane == leader) b = atomicAdd(&m->own_count, (uint32_t)__popc(msk));
        b = __shfl_sync(kFull, b, leader);
        if (mine && b + __popc(msk & ((1u << lane) - 1u)) < (uint32_t)kBins)
          own[b + __popc(msk & ((1u << lane) - 1u))] = i;
      }
    }
    __syncthreads();
    const uint32_t n_own = m->own_count < (uint32_t)kBins ? m->own_count : (uint32_t)kBins;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (uint32_t o = warp; o < n_own; o += kWarps) {
      const uint64_t c = sel[own[o]];
      uint32_t cnt = 0;
      for (uint32_t j = lane; j < K; j += 32) cnt += (sel[j] > c) ? 1u : 0u;
      cnt = __reduce_add_sync(kFull, cnt);
      if (lane == 0 && cnt < kout) {
        const uint32_t key = (uint32_t)(c >> 32), idx = ~(uint32_t)c;
        oi[cnt] = (int32_t)idx;
        if (ov) ov[cnt] = value_of(key, R.rowp, idx);
      }
    }
    if (R.rank == 0) {
      for (uint32_t j = K + threadIdx.x; j < kout; j += kThreads) {
        oi[j] = -1;
        if (ov) ov[j] = -__int_as_float(0x7f800000);
      }
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------ position items (W = 4 per slot)

// Items of the top-k kernel and of stage B: positions. keep(u) masks whole
// slots (stage B keeps only positions of selected blocks).
struct KeepAll {
  __device__ __forceinline__ bool operator()(const Row&, int, const float4 (&)[kVecPerRound], int, int) const {
    return true;
  }
};

// Stage B of the two-level kernel: keep the slot (one block) when its block
// composite is >= the stage-A threshold composite T.
template <int W>
struct KeepBlocks {
  uint64_t T;
  __device__ __forceinline__ bool operator()(const Row& R, int r, const float4 (&v)[kVecPerRound], int u,
                                             int nv) const {
    return composite(slot_block_key<W>(v, u, nv), (uint32_t)(slot_pos<W>(R, r, u) / W)) >= T;
  }
};

template <int W, class Keep>
__device__ __forceinline__ void hist_level1(Row& R, int r, const float4 (&v)[kVecPerRound],
                                            const int (&n)[Geo<W>::kSlots], Keep keep) {
  constexpr int VS = Geo<W>::kVecPerSlot;
  if (r >= R.rounds) return;
#pragma unroll
  for (int u = 0; u < Geo<W>::kSlots; ++u) {
    if (n[u] == 0 || !keep(R, r, v, u, n[u])) continue;
#pragma unroll
    for (int j = 0; j < VS; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (4 * j + e < n[u]) atomicAdd(&R.hist[key_of(lane4(v[u * VS + j], e)) >> 21], 1u);
  }
}

template <int W, class Keep>
__device__ __forceinline__ void hist_level2(Row& R, int r, const float4 (&v)[kVecPerRound],
                                            const int (&n)[Geo<W>::kSlots], uint32_t d1, Keep keep) {
  constexpr int VS = Geo<W>::kVecPerSlot;
  if (r >= R.rounds) return;
#pragma unroll
  for (int u = 0; u < Geo<W>::kSlots; ++u) {
    if (n[u] == 0 || !keep(R, r, v, u, n[u])) continue;
#pragma unroll
    for (int j = 0; j < VS; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t kk = key_of(lane4(v[u * VS + j], e));
        if (4 * j + e < n[u] && (kk >> 21) == d1) atomicAdd(&R.hist[(kk >> 10) & (kBins - 1)], 1u);
      }
  }
}

// Append every kept position whose score passes the threshold (x >= g, or all
// positions when capture_all) to the list. Warp-uniform.
template <int W, class Keep>
__device__ __forceinline__ void filter_round(Row& R, int r, const float4 (&v)[kVecPerRound],
                                             const int (&n)[Geo<W>::kSlots], float g, bool capture_all,
                                             uint32_t* counter, uint2* list, uint32_t cap, Keep keep) {
  constexpr int VS = Geo<W>::kVecPerSlot;
#pragma unroll
  for (int u = 0; u < Geo<W>::kSlots; ++u) {
    const bool kept = n[u] > 0 && keep(R, r, v, u, n[u]);
    float mx = nanf_bits();
#pragma unroll
    for (int j = 0; j < VS; ++j) {
      const float4 q = v[u * VS + j];
      mx = fmaxf(mx, fmaxf(fmaxf(q.x, q.y), fmaxf(q.z, q.w)));
    }
    const bool any = kept && (capture_all || mx >= g);
    if (__any_sync(kFull, any)) {
      const int64_t pos = slot_pos<W>(R, r, u);
#pragma unroll
      for (int j = 0; j < VS; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int o = 4 * j + e;
          const float x = lane4(v[u * VS + j], e);
          const bool pe = kept && o < n[u] && (capture_all || x >= g);
          warp_append(pe, key_of(x), (uint32_t)(pos + o), counter, list, cap);
        }
    }
  }
}

// One pass of the streaming radix select over positions: histogram digit
// (shift s, width w) of every kept composite that matches the prefix.
template <int W, class Keep>
__device__ __forceinline__ void exact_hist_round(Row& R, int r, const float4 (&v)[kVecPerRound],
                                                 const int (&n)[Geo<W>::kSlots], uint64_t tval,
                                                 uint64_t tmask, int s, uint32_t wmask, Keep keep) {
  constexpr int VS = Geo<W>::kVecPerSlot;
#pragma unroll
  for (int u = 0; u < Geo<W>::kSlots; ++u) {
    if (n[u] == 0 || !keep(R, r, v, u, n[u])) continue;
    const int64_t pos = slot_pos<W>(R, r, u);
#pragma unroll
    for (int j = 0; j < VS; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int o = 4 * j + e;
        if (o < n[u]) {
          const uint64_t c = composite(key_of(lane4(v[u * VS + j], e)), (uint32_t)(pos + o));
          if ((c & tmask) == tval) atomicAdd(&R.hist[(uint32_t)(c >> s) & wmask], 1u);
        }
      }
  }
}

template <int W, class Keep>
__device__ __forceinline__ void capture_round(Row& R, int r, const float4 (&v)[kVecPerRound],
                                              const int (&n)[Geo<W>::kSlots], uint64_t T,
                                              uint32_t* counter, uint2* list, uint32_t cap, Keep keep) {
  constexpr int VS = Geo<W>::kVecPerSlot;
#pragma unroll
  for (int u = 0; u < Geo<W>::kSlots; ++u) {
    const bool kept = n[u] > 0 && keep(R, r, v, u, n[u]);
    const int64_t pos = slot_pos<W>(R, r, u);
#pragma unroll
    for (int j = 0; j < VS; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int o = 4 * j + e;
        const uint32_t kk = key_of(lane4(v[u * VS + j], e));
        const bool pe = kept && o < n[u] && composite(kk, (uint32_t)(pos + o)) >= T;
        warp_append(pe, kk, (uint32_t)(pos + o), counter, list, cap);
      }
  }
}

// ------------------------------------------------------------------ block items (stage A)

template <int W>
__device__ __forceinline__ void hist_level1_blocks(Row& R, int r, const float4 (&v)[kVecPerRound],
                                                   const int (&n)[Geo<W>::kSlots]) {
  if (r >= R.rounds) return;
#pragma unroll
  for (int u = 0; u < Geo<W>::kSlots; ++u)
    if (n[u] > 0) atomicAdd(&R.hist[slot_block_key<W>(v, u, n[u]) >> 21], 1u);
}

template <int W>
__device__ __forceinline__ void hist_level2_blocks(Row& R, int r, const float4 (&v)[kVecPerRound],
                                                   const int (&n)[Geo<W>::kSlots], uint32_t d1) {
  if (r >= R.rounds) return;
#pragma unroll
  for (int u = 0; u < Geo<W>::kSlots; ++u) {
    if (n[u] == 0) continue;
    const uint32_t kk = slot_block_key<W>(v, u, n[u]);
    if ((kk >> 21) == d1) atomicAdd(&R.hist[(kk >> 10) & (kBins - 1)], 1u);
  }
}

template <int W>
__device__ __forceinline__ void filter_round_blocks(Row& R, int r, const float4 (&v)[kVecPerRound],
                                                    const int (&n)[Geo<W>::kSlots], uint32_t t,
                                                    uint32_t* counter, uint2* list, uint32_t cap) {
#pragma unroll
  for (int u = 0; u < Geo<W>::kSlots; ++u) {
    const uint32_t kk = n[u] > 0 ? slot_block_key<W>(v, u, n[u]) : 0u;
    const bool pe = n[u] > 0 && kk >= t;
    const uint32_t bid = (uint32_t)(slot_pos<W>(R, r, u) / W);
    warp_append(pe, kk, bid, counter, list, cap);
  }
}

template <int W>
__device__ __forceinline__ void exact_hist_round_blocks(Row& R, int r, const float4 (&v)[kVecPerRound],
                                                        const int (&n)[Geo<W>::kSlots], uint64_t tval,
                                                        uint64_t tmask, int s, uint32_t wmask) {
#pragma unroll
  for (int u = 0; u < Geo<W>::kSlots; ++u) {
    if (n[u] == 0) continue;
    const uint64_t c = composite(slot_block_key<W>(v, u, n[u]), (uint32_t)(slot_pos<W>(R, r, u) / W));
    if ((c & tmask) == tval) atomicAdd(&R.hist[(uint32_t)(c >> s) & wmask], 1u);
  }
}

template <int W>
__device__ __forceinline__ void capture_round_blocks(Row& R, int r, const float4 (&v)[kVecPerRound],
                                                     const int (&n)[Geo<W>::kSlots], uint64_t T,
                                                     uint32_t* counter, uint2* list, uint32_t cap) {
#pragma unroll
  for (int u = 0; u < Geo<W>::kSlots; ++u) {
    const uint32_t kk = n[u] > 0 ? slot_block_key<W>(v, u, n[u]) : 0u;
    const uint32_t bid = (uint32_t)(slot_pos<W>(R, r, u) / W);
    const bool pe = n[u] > 0 && composite(kk, bid) >= T;
    warp_append(pe, kk, bid, counter, list, cap);
  }
}

// ------------------------------------------------------------------ one selection stage

// Items are either positions (kBlocks = false; keep masks whole slots) or
// blocks (kBlocks = true). Runs estimate -> filter -> exchange -> select (or
// the streaming exact select) and leaves the K selected composites in sel[].
// va/vb hold rounds 0 and 1 on entry when `loaded`; they may be overwritten.
// Returns the threshold composite T (valid when K > 0).
template <int W, bool kBlocks, class Keep>
__device__ uint64_t select_stage(Row& R, const Params& p, float4 (&va)[kVecPerRound],
                                 int (&na)[Geo<W>::kSlots], float4 (&vb)[kVecPerRound],
                                 int (&nb)[Geo<W>::kSlots], bool loaded, uint32_t K, int64_t items,
                                 int64_t idx_limit, Keep keep, bool* regs_intact, bool first) {
  Misc* m = R.m;
  if (!first) {
    // A later stage reuses the candidate lists: clear them, and make sure no
    // peer pushes into them before this CTA has finished with the last stage.
    reset_lists(R);
    if (R.nclus > 1) {
      if (R.init_pending) {
        cluster_wait();
        R.init_pending = false;
      }
      cluster_sync();
    }
  }
  const uint32_t cap = (uint32_t)p.cap;
  uint32_t* counter = (R.nclus > 1) ? &m->local_count : &m->cand_count;
  uint2* list = (R.nclus > 1) ? R.local : R.cand;
  const bool full = R.rounds_max <= 2;

  if (!loaded) {
    if (R.rounds > 0) load_round<W>(R, p, 0, va, na); else clear_round<W>(na);
    if (R.rounds > 1) load_round<W>(R, p, 1, vb, nb); else clear_round<W>(nb);
  }

  bool exact = p.force_exact != 0;
  int stat = kCntFast;
  *regs_intact = R.rounds <= 2;
  uint64_t T = 0;
  if (!exact && K > 0) {
    // ---- threshold estimate from the digit histogram of the sample
    uint32_t t = 0;
    if (items > (int64_t)(cap / 2)) {
      zero_hist(R);
      if (kBlocks) {
        hist_level1_blocks<W>(R, 0, va, na);
        hist_level1_blocks<W>(R, 1, vb, nb);
      } else {
        hist_level1<W>(R, 0, va, na, keep);
        hist_level1<W>(R, 1, vb, nb, keep);
      }
      const uint32_t* bins = merge_hist(R, 0);
      const uint32_t ns = full ? (uint32_t)items : bins_total(bins, m);
      if (ns > 0) {
        const uint32_t r = sample_target(K, ns, items, full);
        find_digit(bins, r, m);
        const uint32_t d1 = m->res_digit, above1 = m->res_above, cnt1 = m->res_cnt;
        release_merged(R, 0);
        const float predicted = full ? (float)(above1 + cnt1)
                                     : (float)(above1 + cnt1) * ((float)items / (float)ns);
        t = d1 << 21;
        if (predicted > 0.5f * (float)cap) {
          zero_hist(R);
          if (kBlocks) {
            hist_level2_blocks<W>(R, 0, va, na, d1);
            hist_level2_blocks<W>(R, 1, vb, nb, d1);
          } else {
            hist_level2<W>(R, 0, va, na, d1, keep);
            hist_level2<W>(R, 1, vb, nb, d1, keep);
          }
          const uint32_t* bins2 = merge_hist(R, 1);
          find_digit(bins2, r - above1, m);
          const uint32_t d2 = m->res_digit;
          release_merged(R, 1);
          t |= d2 << 10;
        }
      } else {
        release_merged(R, 0);
      }
    }
    // ---- filter every round against the threshold
    const bool all = (t == 0u);
    const float g = threshold_float(t == 0u ? 1u : t);
    for (int r = 0; r < R.rounds; r += 2) {
      if (kBlocks) filter_round_blocks<W>(R, r, va, na, t, counter, list, cap);
      else filter_round<W>(R, r, va, na, g, all, counter, list, cap, keep);
      if (r + 2 < R.rounds) load_round<W>(R, p, r + 2, va, na);
      if (r + 1 < R.rounds) {
        if (kBlocks) filter_round_blocks<W>(R, r + 1, vb, nb, t, counter, list, cap);
        else filter_round<W>(R, r + 1, vb, nb, g, all, counter, list, cap, keep);
        if (r + 3 < R.rounds) load_round<W>(R, p, r + 3, vb, nb);
      }
    }
    exchange(R, cap);
    const uint32_t N = m->cand_count;
    const bool overflow = (m->flags & 1u) || N > cap;
    if (overflow || N < K) {
      exact = true;
      stat = overflow ? kCntOverflow : kCntShort;
      __syncthreads();
    } else {
      T = select_local(R, N, K, idx_limit);
    }
  }

  if (exact && K > 0) {
    // ---- streaming radix select: every pass re-reads the slice
    if (stat != kCntFast) bump(p, R, stat);
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
      zero_hist(R);
      for (int r = 0; r < R.rounds; ++r) {
        load_round<W>(R, p, r, va, na);
        if (kBlocks) exact_hist_round_blocks<W>(R, r, va, na, tval, tmask, s, (1u << w) - 1u);
        else exact_hist_round<W>(R, r, va, na, tval, tmask, s, (1u << w) - 1u, keep);
      }
      const uint32_t* bins = merge_hist(R, buf);
      find_digit(bins, need, m);
      const uint32_t d = m->res_digit, above = m->res_above, cnt = m->res_cnt;
      release_merged(R, buf);
      buf ^= 1;
      need -= above;
      tval |= (uint64_t)d << s;
      tmask |= dmask;
      if (cnt == need) break;
    }
    T = tval;
    *regs_intact = false;
    for (int r = 0; r < R.rounds; ++r) {
      load_round<W>(R, p, r, va, na);
      if (kBlocks) capture_round_blocks<W>(R, r, va, na, T, counter, list, cap);
      else capture_round<W>(R, r, va, na, T, counter, list, cap, keep);
    }
    exchange(R, cap);
    bump(p, R, kCntExact);
  } else if (K > 0) {
    bump(p, R, kCntFast);
  }
  if (K > 0) {
    compact_selected(R, m->cand_count < cap ? m->cand_count : cap, T);
  }
  return T;
}

__device__ __forceinline__ bool in_slice(const Row& R, uint32_t idx) {
  return (int64_t)idx >= R.begin && (int64_t)idx < R.end;
}

}  // namespace lt
