// lt_compress.cu -- the fused KV compressor: each compressed entry is made
// from one read of its block's KV vectors and scores and one store.
//
// Unfused, the compressor is a chain of five passes over memory (read, add,
// softmax, dot, store: SGLang DeepSeek-V4 inference talk notes, section 3.1);
// here the add, the softmax over the block's tokens and the weighted sum run
// in registers between the read and the store (the fusion the AICon 2026
// Shenzhen speaker page calls FlashCompressor, outline section 3.1).
//
// Work split. A work item is one channel group (V consecutive channels) of
// one block (ratio consecutive tokens) of one row. A CTA is a TX x TY grid of
// threads: x runs over the channel groups of a block (consecutive threads read
// consecutive 16- or 8-byte words of a token's vector), y over blocks; CTAs
// walk the blocks grid-stride. A thread walks its block's tokens in chunks of
// U, with an online softmax: the chunk's scores are loaded together (2U loads
// in flight per thread), the running maximum is raised to the chunk's, the
// running sums are rescaled by exp(old max - new max) and the chunk's terms
// are added. The block's entry is the weighted sum over the sum of weights.
//
// No cross-CTA communication, no shared memory: the kernel is bound by HBM
// (kv and score read once, one entry written per block).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/lt_compress.h"
#include "lt_async.cuh"

namespace {

using lt::bulk_g2s;
using lt::kWaitPolls;
using lt::mbar_arrive_tx;
using lt::mbar_fence_init;
using lt::mbar_init;
using lt::ring_wait;

constexpr int kThreads = 256;
constexpr int kChunk = 4;  // tokens loaded together

struct CParams {
  const void* kv;
  const void* score;
  const float* bias;
  const int32_t* lengths;
  void* out;
  int64_t row_tokens;
  int64_t nblk;     // blocks per row: row_tokens / ratio
  int64_t blocks;   // rows * nblk
  int32_t dim;
  int32_t ratio;
  int32_t groups;   // channel groups per block: dim / V
};

struct DParams {
  const void* kv_new;
  const void* score_new;
  const float* bias;
  void* ring_kv;
  void* ring_score;
  const int32_t* pos;
  void* out;
  int32_t seqs, dim, ratio, groups;
};

// ---- V scores as floats (bf16 widens exactly: its bits are the top half of an fp32)

__device__ __forceinline__ float widen(uint32_t h) { return __uint_as_float(h << 16); }

template <int V>
__device__ __forceinline__ void load_v(const float* p, float (&x)[V]) {
  if constexpr (V == 4) {
    const float4 q = __ldg(reinterpret_cast<const float4*>(p));
    x[0] = q.x; x[1] = q.y; x[2] = q.z; x[3] = q.w;
  } else {
#pragma unroll
    for (int c = 0; c < V; ++c) x[c] = __ldg(p + c);
  }
}
template <int V>
__device__ __forceinline__ void load_v(const uint16_t* p, float (&x)[V]) {
  if constexpr (V == 4) {
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
    x[0] = widen(q.x & 0xffffu); x[1] = __uint_as_float(q.x & 0xffff0000u);
    x[2] = widen(q.y & 0xffffu); x[3] = __uint_as_float(q.y & 0xffff0000u);
  } else {
#pragma unroll
    for (int c = 0; c < V; ++c) x[c] = widen(__ldg(p + c));
  }
}
// plain (not read-only-path) loads for the ring buffers, which this kernel also writes
template <int V>
__device__ __forceinline__ void load_rw(const float* p, float (&x)[V]) {
#pragma unroll
  for (int c = 0; c < V; ++c) x[c] = p[c];
}
template <int V>
__device__ __forceinline__ void load_rw(const uint16_t* p, float (&x)[V]) {
#pragma unroll
  for (int c = 0; c < V; ++c) x[c] = widen(p[c]);
}

template <int V>
__device__ __forceinline__ void store_v(float* p, const float (&y)[V]) {
  if constexpr (V == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(y[0], y[1], y[2], y[3]);
  } else {
#pragma unroll
    for (int c = 0; c < V; ++c) p[c] = y[c];
  }
}
__device__ __forceinline__ uint32_t bf16_bits(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}
template <int V>
__device__ __forceinline__ void store_v(uint16_t* p, const float (&y)[V]) {
  if constexpr (V == 4) {
    *reinterpret_cast<uint2*>(p) = make_uint2(bf16_bits(y[0]) | (bf16_bits(y[1]) << 16),
                                              bf16_bits(y[2]) | (bf16_bits(y[3]) << 16));
  } else {
#pragma unroll
    for (int c = 0; c < V; ++c) p[c] = (uint16_t)bf16_bits(y[c]);
  }
}
// copy V raw elements (the new token into its ring slot)
template <class S, int V>
__device__ __forceinline__ void copy_v(S* dst, const S* src) {
#pragma unroll
  for (int c = 0; c < V; ++c) dst[c] = src[c];
}

// ---- the online softmax-weighted sum, in base 2
//
// exp(v) = 2^(v log2 e): the biased score is formed directly in base-2 units,
// l = score * log2(e) + bias * log2(e) (one fused multiply-add), and every
// weight is one hardware base-2 exponential (ex2.approx, relative error of a
// few ulps; results below 2^-126 flush to zero, a weight far below what can
// change the sum). The running maximum is kept in the same units.

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// the biased score of one channel in base-2 units
__device__ __forceinline__ float logit2(float z, float b) { return fmaf(z, kLog2e, b * kLog2e); }

template <int V>
struct Acc {
  float m[V], s[V], a[V];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int c = 0; c < V; ++c) {
      m[c] = -__int_as_float(0x7f800000);
      s[c] = 0.0f;
      a[c] = 0.0f;
    }
  }
  // add the n <= U tokens of a chunk: base-2 biased scores v, values x
  template <int U>
  __device__ __forceinline__ void add(const float (&v)[U][V], const float (&x)[U][V], int n) {
#pragma unroll
    for (int c = 0; c < V; ++c) {
      float cm = v[0][c];
#pragma unroll
      for (int u = 1; u < U; ++u)
        if (u < n) cm = fmaxf(cm, v[u][c]);
      const float mn = fmaxf(m[c], cm);
      const float r = ex2(m[c] - mn);  // 0 for the first chunk (m = -inf)
      float sc = s[c] * r, ac = a[c] * r;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (u < n) {
          const float e = ex2(v[u][c] - mn);
          sc += e;
          ac = fmaf(e, x[u][c], ac);
        }
      }
      m[c] = mn;
      s[c] = sc;
      a[c] = ac;
    }
  }
  __device__ __forceinline__ void result(float (&y)[V]) const {
#pragma unroll
    for (int c = 0; c < V; ++c) y[c] = a[c] / s[c];
  }
};

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- prefill: every complete block of every row

template <class S, int V>
__global__ void __launch_bounds__(kThreads) compress_kernel(CParams p) {
  grid_dependents_launch();
  grid_dependency_wait();  // kv, score and lengths may come from the previous kernel
  const S* kv = static_cast<const S*>(p.kv);
  const S* sc = static_cast<const S*>(p.score);
  S* out = static_cast<S*>(p.out);
  const int64_t step = (int64_t)gridDim.x * blockDim.y;
  int64_t b = (int64_t)blockIdx.x * blockDim.y + threadIdx.y;
  if (b >= p.blocks) return;
  // row and block of b, then advanced by `step` without dividing again
  int64_t r = b / p.nblk, g = b - r * p.nblk;
  int64_t lim = -1;  // complete blocks of row r (read lazily)
  int64_t lim_row = -1;
  for (; b < p.blocks; b += step) {
    if (r != lim_row) {
      int64_t L = p.row_tokens;
      if (p.lengths) {
        L = (int64_t)__ldg(p.lengths + r);
        L = L < 0 ? 0 : (L > p.row_tokens ? p.row_tokens : L);
      }
      lim = L / p.ratio;
      lim_row = r;
    }
    if (g < lim) {
      const int64_t t0 = r * p.row_tokens + g * p.ratio;
      for (int cg = threadIdx.x; cg < p.groups; cg += blockDim.x) {
        const int64_t c0 = (int64_t)cg * V;
        const S* xk = kv + t0 * p.dim + c0;
        const S* zk = sc + t0 * p.dim + c0;
        const float* bk = p.bias + c0;
        Acc<V> acc;
        acc.init();
        for (int j = 0; j < p.ratio; j += kChunk) {
          const int n = p.ratio - j < kChunk ? p.ratio - j : kChunk;
          float x[kChunk][V], v[kChunk][V];
#pragma unroll
          for (int u = 0; u < kChunk; ++u) {
            if (u < n) {
              const int64_t o = (int64_t)(j + u) * p.dim;
              float z[V], bb[V];
              load_v<V>(xk + o, x[u]);
              load_v<V>(zk + o, z);
              load_v<V>(bk + (int64_t)(j + u) * p.dim, bb);
#pragma unroll
              for (int c = 0; c < V; ++c) v[u][c] = logit2(z[c], bb[c]);  // add
            }
          }
          acc.add<kChunk>(v, x, n);  // softmax terms and weighted sum
        }
        float y[V];
        acc.result(y);
        store_v<V>(out + (r * p.nblk + g) * p.dim + c0, y);  // store
      }
    }
    g += step;
    if (g >= p.nblk) {
      const int64_t q = g / p.nblk;
      r += q;
      g -= q * p.nblk;
    }
  }
}

// ---- prefill through a ring of shared-memory stages (bulk copies)
//
// The register kernel above keeps only a few loads in flight per thread; on
// GB300 that leaves HBM idle. Here thread 0 of each (persistent) CTA copies
// whole token ranges of kv and score -- contiguous in memory -- into a ring of
// shared-memory stages with cp.async.bulk, each stage completing on its own
// mbarrier, so the bytes in flight no longer depend on registers. A unit of
// work is either several whole blocks (small ratios: a block fits a stage;
// the bias then lives in shared memory for the whole launch) or one block
// streamed over several stages (large ratios: each stage also carries the
// bias rows of its tokens, and the two threads of a channel group take
// alternate tokens and merge their partial sums with a shuffle at the end).
// Producer and consumers walk the same unit sequence (units of this CTA that
// hold at least one complete block), so no descriptors are exchanged. Waits
// are bounded (a copy that never lands leaves that unit's output undefined
// rather than hanging).

constexpr uint32_t kRingInSmall = 16384;  // kv bytes per stage when a block fits (score the same)
constexpr uint32_t kRingInLarge = 8192;   // kv bytes per stage of a streamed block (+ bias rows)
constexpr uint32_t kRingBudget = 112 * 1024;  // two CTAs per SM
constexpr int kRingMaxStages = 4;

struct RParams {
  const void* kv;
  const void* score;
  const float* bias;
  const int32_t* lengths;
  void* out;
  int64_t row_tokens;
  int64_t nblk;           // blocks per row
  int64_t units_per_row;
  int64_t units;          // rows * units_per_row
  int32_t dim, ratio, groups;
  int32_t st;             // tokens per full stage
  int32_t bpu;            // blocks per unit (streamed: blocks that stream side by side)
  int32_t subtiles;       // stages per unit
  int32_t tpg;            // streamed blocks: threads per channel group (power of two)
  int32_t stages;
  uint32_t in_bytes;      // kv bytes of a full stage
  uint32_t stage_bytes;   // kv + score (+ bias rows)
  uint32_t bias_off, ring_off;  // shared-memory offsets
};

// Unit u of the launch: row r, first block g0 and its complete blocks nb
// (0 when the unit lies past the row's last complete block).
__device__ __forceinline__ int unit_blocks(const RParams& p, int64_t u, int64_t* r, int64_t* g0) {
  *r = u / p.units_per_row;
  const int64_t ui = u - *r * p.units_per_row;
  int64_t L = p.row_tokens;
  if (p.lengths) {
    L = (int64_t)__ldg(p.lengths + *r);
    L = L < 0 ? 0 : (L > p.row_tokens ? p.row_tokens : L);
  }
  *g0 = ui * p.bpu;
  const int64_t n = L / p.ratio - *g0;
  return n <= 0 ? 0 : (n < p.bpu ? (int)n : p.bpu);
}

// The next unit at or after u (stepping by the grid) that has work.
__device__ __forceinline__ bool next_unit(const RParams& p, int64_t& u, int64_t* r, int64_t* g0, int* nb) {
  for (; u < p.units; u += gridDim.x) {
    *nb = unit_blocks(p, u, r, g0);
    if (*nb > 0) return true;
  }
  return false;
}

// Tokens of stage `sub` of a unit: first token (row-relative) and count.
__device__ __forceinline__ void stage_tokens(const RParams& p, int64_t g0, int nb, int sub, int64_t* t0, int* n) {
  if (p.subtiles == 1) {
    *t0 = g0 * p.ratio;
    *n = nb * p.ratio;
  } else {
    *t0 = g0 * p.ratio + (int64_t)sub * p.st;
    const int left = p.ratio - sub * p.st;
    *n = left < p.st ? left : p.st;
  }
}

template <int V>
__device__ __forceinline__ void lds_v(const float* p, float (&x)[V]) {
  const float4 q = *reinterpret_cast<const float4*>(p);
  x[0] = q.x; x[1] = q.y; x[2] = q.z; x[3] = q.w;
}
template <int V>
__device__ __forceinline__ void lds_v(const uint16_t* p, float (&x)[V]) {
  const uint2 q = *reinterpret_cast<const uint2*>(p);
  x[0] = widen(q.x & 0xffffu); x[1] = __uint_as_float(q.x & 0xffff0000u);
  x[2] = widen(q.y & 0xffffu); x[3] = __uint_as_float(q.y & 0xffff0000u);
}

// Whole blocks of one stage, any ratio: one item per (block, channel group).
// Offsets inside a stage fit 32 bits.
template <class S>
__device__ __forceinline__ void ring_blocks(const RParams& p, const S* xs, const S* zs, const float* bias_s, int nb,
                                            S* ob, int tid) {
  constexpr int V = 4;
  const int items = nb * p.groups;
  for (int it = tid; it < items; it += kThreads) {
    const int q = it / p.groups;
    const int cg = it - q * p.groups;
    const uint32_t o = (uint32_t)(q * p.ratio) * (uint32_t)p.dim + (uint32_t)cg * V;
    Acc<V> a;
    a.init();
    for (int j = 0; j < p.ratio; j += kChunk) {
      const int m = p.ratio - j < kChunk ? p.ratio - j : kChunk;
      float x[kChunk][V], v[kChunk][V];
#pragma unroll
      for (int u = 0; u < kChunk; ++u) {
        if (u < m) {
          float z[V], bb[V];
          const uint32_t tok = (uint32_t)(j + u) * (uint32_t)p.dim;
          lds_v<V>(xs + o + tok, x[u]);
          lds_v<V>(zs + o + tok, z);
          lds_v<V>(bias_s + tok + (uint32_t)cg * V, bb);
#pragma unroll
          for (int c = 0; c < V; ++c) v[u][c] = logit2(z[c], bb[c]);
        }
      }
      a.add<kChunk>(v, x, m);
    }
    float y[V];
    a.result(y);
    store_v<V>(ob + (uint32_t)q * (uint32_t)p.dim + (uint32_t)cg * V, y);
  }
}

// The same for a compile-time ratio R <= kChunk when the threads divide into
// whole channel-group columns: each thread keeps one channel group for the
// whole launch, with its R bias rows (already in base-2 units) in registers.
template <class S, int R>
__device__ __forceinline__ void ring_blocks_fixed(const S* xs, const S* zs, const float (&b2)[R > 0 ? R : 1][4],
                                                  int nb, int dim, int cg, int q0, int qs, S* ob) {
  constexpr int V = 4;
  static_assert(R >= 1 && R <= kChunk, "one chunk per block");
  for (int q = q0; q < nb; q += qs) {
    const uint32_t o = (uint32_t)(q * R) * (uint32_t)dim + (uint32_t)cg * V;
    float x[kChunk][V], v[kChunk][V];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      float z[V];
      lds_v<V>(xs + o + (uint32_t)u * (uint32_t)dim, x[u]);
      lds_v<V>(zs + o + (uint32_t)u * (uint32_t)dim, z);
#pragma unroll
      for (int c = 0; c < V; ++c) v[u][c] = fmaf(z[c], kLog2e, b2[u][c]);
    }
    Acc<V> a;
    a.init();
    a.add<kChunk>(v, x, R);
    float y[V];
    a.result(y);
    store_v<V>(ob + (uint32_t)q * (uint32_t)dim + (uint32_t)cg * V, y);
  }
}

// R: a compile-time ratio for the fixed-column path (blocks of R <= kChunk
// tokens, threads a multiple of the channel groups), else 0.
template <class S, int R>
__global__ void __launch_bounds__(kThreads, 2) compress_ring_kernel(RParams p) {
  constexpr int V = 4;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  float* bias_s = reinterpret_cast<float*>(smem + p.bias_off);
  unsigned char* ring = smem + p.ring_off;
  const int tid = threadIdx.x;
  const uint32_t ns = (uint32_t)p.stages;
  if (tid == 0) {
    for (uint32_t i = 0; i < ns; ++i) mbar_init(&bars[i], 1);
    mbar_fence_init();
  }
  grid_dependents_launch();
  grid_dependency_wait();  // inputs and lengths may come from the previous kernel
  if (p.subtiles == 1) {
    for (int i = tid; i < p.ratio * p.dim; i += kThreads) bias_s[i] = __ldg(p.bias + i);
  }
  __syncthreads();
  // fixed-column path: this thread's channel group, first block, block step
  // and bias rows (base-2 units)
  const int fixed_cg = R > 0 ? tid % p.groups : 0;
  const int fixed_q0 = R > 0 ? tid / p.groups : 0;
  const int fixed_qs = R > 0 ? kThreads / p.groups : 1;
  float bfix[R > 0 ? R : 1][4];
#pragma unroll
  for (int u = 0; u < (R > 0 ? R : 1); ++u)
#pragma unroll
    for (int c = 0; c < 4; ++c) bfix[u][c] = R > 0 ? bias_s[u * p.dim + fixed_cg * 4 + c] * kLog2e : 0.0f;

  const S* kv = static_cast<const S*>(p.kv);
  const S* sc = static_cast<const S*>(p.score);
  // ---- producer state (thread 0)
  int64_t pu = blockIdx.x, pr = 0, pg0 = 0;
  int pnb = 0, psub = 0;
  bool pvalid = false;
  uint32_t pseq = 0;
  auto produce = [&](uint32_t limit) {
    while (pvalid && (int32_t)(limit - pseq) > 0) {
      int64_t t0;
      int n;
      stage_tokens(p, pg0, pnb, psub, &t0, &n);
      unsigned char* dst = ring + (size_t)(pseq % ns) * p.stage_bytes;
      const uint32_t bytes = (uint32_t)n * (uint32_t)p.dim * (uint32_t)sizeof(S);
      uint64_t* bar = &bars[pseq % ns];
      if (R > 0 || p.subtiles == 1) {
        // whole blocks, contiguous: kv, then score (the fixed-column kernel
        // only ever sees these)
        mbar_arrive_tx(bar, 2u * bytes);
        const int64_t e0 = (pr * p.row_tokens + t0) * p.dim;
        bulk_g2s(dst, kv + e0, bytes, bar);
        bulk_g2s(dst + p.in_bytes, sc + e0, bytes, bar);
      } else {
        // the same tokens of each of the unit's pnb streamed blocks (kv of
        // block b at b * in_bytes, its score at (bpu + b) * in_bytes), then
        // those tokens' bias rows once for all of them
        const uint32_t bbytes = (uint32_t)n * (uint32_t)p.dim * 4u;
        mbar_arrive_tx(bar, 2u * bytes * (uint32_t)pnb + bbytes);
        for (int b = 0; b < pnb; ++b) {
          const int64_t e0 = (pr * p.row_tokens + t0 + (int64_t)b * p.ratio) * p.dim;
          bulk_g2s(dst + (uint32_t)b * p.in_bytes, kv + e0, bytes, bar);
          bulk_g2s(dst + (uint32_t)(p.bpu + b) * p.in_bytes, sc + e0, bytes, bar);
        }
        bulk_g2s(dst + 2u * (uint32_t)p.bpu * p.in_bytes, p.bias + (int64_t)psub * p.st * p.dim, bbytes, bar);
      }
      ++pseq;
      if (++psub == p.subtiles) {
        psub = 0;
        pu += gridDim.x;
        pvalid = next_unit(p, pu, &pr, &pg0, &pnb);
      }
    }
  };
  if (tid == 0) {
    pvalid = next_unit(p, pu, &pr, &pg0, &pnb);
    produce(ns);
  }

  // ---- consumers (every thread)
  S* out = static_cast<S*>(p.out);
  int64_t cu = blockIdx.x, cr = 0, cg0 = 0;
  int cnb = 0;
  bool cvalid = next_unit(p, cu, &cr, &cg0, &cnb);
  uint32_t seq = 0;
  bool late = false;
  // streamed blocks: this thread's block of the unit, channel group and token phase
  const int laneB = tid / (p.groups * p.tpg);
  const int jB = tid - laneB * (p.groups * p.tpg);
  const int cgB = jB / p.tpg, hB = jB - cgB * p.tpg;
  Acc<V> acc;
  while (cvalid) {
    for (int sub = 0; sub < p.subtiles; ++sub) {
      if (!ring_wait(bars, ns, seq, kWaitPolls)) late = true;
      const unsigned char* stg = ring + (size_t)(seq % ns) * p.stage_bytes;
      const S* xs = reinterpret_cast<const S*>(stg);
      const S* zs = reinterpret_cast<const S*>(stg + p.in_bytes);
      int64_t t0;
      int n;
      stage_tokens(p, cg0, cnb, sub, &t0, &n);
      if (R > 0 || p.subtiles == 1) {
        S* ob = out + (cr * p.nblk + cg0) * p.dim;
        if constexpr (R > 0) {
          ring_blocks_fixed<S, R>(xs, zs, bfix, cnb, p.dim, fixed_cg, fixed_q0, fixed_qs, ob);
        } else {
          ring_blocks<S>(p, xs, zs, bias_s, cnb, ob, tid);
        }
      } else {
        // a unit's blocks over several stages: this thread's block laneB,
        // tokens t with t mod tpg == hB
        if (sub == 0) acc.init();
        const float* bs = reinterpret_cast<const float*>(stg + 2u * (uint32_t)p.bpu * p.in_bytes);
        xs = reinterpret_cast<const S*>(stg + (uint32_t)laneB * p.in_bytes);
        zs = reinterpret_cast<const S*>(stg + (uint32_t)(p.bpu + laneB) * p.in_bytes);
        if (laneB < cnb && cgB < p.groups) {
          const int base = sub * p.st;
          int i = (hB - base) % p.tpg;
          if (i < 0) i += p.tpg;
          const uint32_t oc = (uint32_t)cgB * V;
          while (i < n) {
            float x[kChunk][V], v[kChunk][V];
            int m = 0;
#pragma unroll
            for (int u = 0; u < kChunk; ++u) {
              const int ii = i + u * p.tpg;
              if (ii < n) {
                float z[V], bb[V];
                const uint32_t ot = (uint32_t)ii * (uint32_t)p.dim + oc;
                lds_v<V>(xs + ot, x[u]);
                lds_v<V>(zs + ot, z);
                lds_v<V>(bs + ot, bb);
#pragma unroll
                for (int c = 0; c < V; ++c) v[u][c] = logit2(z[c], bb[c]);
                m = u + 1;
              }
            }
            acc.add<kChunk>(v, x, m);
            i += kChunk * p.tpg;
          }
        }
        if (sub == p.subtiles - 1) {
          // merge the tpg partial sums of each channel group (adjacent lanes)
          for (int off = 1; off < p.tpg; off <<= 1) {
#pragma unroll
            for (int c = 0; c < V; ++c) {
              const float m2 = __shfl_xor_sync(0xffffffffu, acc.m[c], off);
              const float s2 = __shfl_xor_sync(0xffffffffu, acc.s[c], off);
              const float a2 = __shfl_xor_sync(0xffffffffu, acc.a[c], off);
              const float mn = fmaxf(acc.m[c], m2);
              const float r1 = acc.m[c] == mn ? 1.0f : ex2(acc.m[c] - mn);
              const float r2 = m2 == mn ? 1.0f : ex2(m2 - mn);
              acc.s[c] = acc.s[c] * r1 + s2 * r2;
              acc.a[c] = acc.a[c] * r1 + a2 * r2;
              acc.m[c] = mn;
            }
          }
          if (laneB < cnb && cgB < p.groups && hB == 0) {
            float y[V];
            acc.result(y);
            store_v<V>(out + (cr * p.nblk + cg0 + laneB) * p.dim + (int64_t)cgB * V, y);
          }
        }
      }
      __syncthreads();  // every thread is done with this stage
      if (tid == 0) produce(seq + 1 + ns);
      ++seq;
    }
    cu += gridDim.x;
    cvalid = next_unit(p, cu, &cr, &cg0, &cnb);
  }
  // A wait that gave up may leave its copy in flight: give the last stages a
  // bounded chance to land before the CTA's shared memory goes away.
  if (__syncthreads_or(late ? 1 : 0) && tid == 0) {
    for (uint32_t i = 0; i < ns && i < seq; ++i) (void)ring_wait(bars, ns, seq - 1u - i, kWaitPolls);
  }
  __syncthreads();
}

// ---- decode: one new token per sequence, state in the two rings

template <class S, int V>
__global__ void __launch_bounds__(kThreads) compress_decode_kernel(DParams p) {
  grid_dependents_launch();
  grid_dependency_wait();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)p.seqs * p.groups) return;
  const int32_t s = (int32_t)(i / p.groups);
  const int32_t cg = (int32_t)(i - (int64_t)s * p.groups);
  const int32_t pos = __ldg(p.pos + s);
  if (pos < 0) return;
  const int32_t slot = pos % p.ratio;
  const int64_t c0 = (int64_t)cg * V;
  const S* xn = static_cast<const S*>(p.kv_new) + (int64_t)s * p.dim + c0;
  const S* zn = static_cast<const S*>(p.score_new) + (int64_t)s * p.dim + c0;
  S* rk = static_cast<S*>(p.ring_kv) + (int64_t)s * p.ratio * p.dim + c0;
  S* rs = static_cast<S*>(p.ring_score) + (int64_t)s * p.ratio * p.dim + c0;
  copy_v<S, V>(rk + (int64_t)slot * p.dim, xn);
  copy_v<S, V>(rs + (int64_t)slot * p.dim, zn);
  if (slot != p.ratio - 1) return;
  // the block is complete: the earlier slots come from the ring (written by
  // earlier steps), the new token from its input; chunked as in the prefill
  // kernel, so both give the same bits
  Acc<V> acc;
  acc.init();
  for (int j = 0; j < p.ratio; j += kChunk) {
    const int n = p.ratio - j < kChunk ? p.ratio - j : kChunk;
    float x[kChunk][V], v[kChunk][V];
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      if (u < n) {
        float z[V], bb[V];
        if (j + u == slot) {
          load_v<V>(xn, x[u]);
          load_v<V>(zn, z);
        } else {
          load_rw<V>(rk + (int64_t)(j + u) * p.dim, x[u]);
          load_rw<V>(rs + (int64_t)(j + u) * p.dim, z);
        }
        load_v<V>(p.bias + (int64_t)(j + u) * p.dim + c0, bb);
#pragma unroll
        for (int c = 0; c < V; ++c) v[u][c] = logit2(z[c], bb[c]);
      }
    }
    acc.add<kChunk>(v, x, n);
  }
  float y[V];
  acc.result(y);
  store_v<V>(static_cast<S*>(p.out) + (int64_t)s * p.dim + c0, y);
}

// ---- host side

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_ctas_per_sm[kMaxDevices][4];  // prefill kernels: resident CTAs per SM (0: not asked yet)
int g_sms[kMaxDevices];

int g_ring_smem_set[kMaxDevices][4];  // dynamic shared memory granted to the ring kernels
int g_ring_ctas[kMaxDevices][4];      // their resident CTAs per SM

template <class S, int V>
const void* prefill_ptr() { return reinterpret_cast<const void*>(&compress_kernel<S, V>); }

bool aligned_to(const void* p, unsigned a);

// Ring geometry for this launch; false when the layout does not allow bulk
// copies (then the register kernel runs).
bool ring_plan(const void* kv, const void* score, const float* bias, const void* out, int64_t row_tokens,
               int32_t dim, int32_t ratio, bool bf16, RParams* r, uint32_t* smem) {
  const uint32_t es = bf16 ? 2u : 4u;
  const uint64_t row_bytes = (uint64_t)dim * es;
  if (dim % 4 != 0 || row_bytes % 16 != 0) return false;
  if (!aligned_to(kv, 16) || !aligned_to(score, 16) || !aligned_to(bias, 16) || !aligned_to(out, bf16 ? 8 : 16))
    return false;
  const uint32_t groups = (uint32_t)dim / 4;
  uint32_t bias_bytes = 0;
  if ((uint64_t)ratio * row_bytes <= kRingInSmall) {
    r->bpu = (int32_t)(kRingInSmall / ((uint64_t)ratio * row_bytes));
    r->st = r->bpu * ratio;
    r->subtiles = 1;
    r->tpg = 1;
    r->in_bytes = (uint32_t)(r->st * row_bytes);
    r->stage_bytes = 2u * r->in_bytes;
    bias_bytes = (uint32_t)ratio * (uint32_t)dim * 4u;
  } else {
    if (groups > (uint32_t)kThreads || row_bytes > kRingInLarge) return false;
    r->st = (int32_t)(kRingInLarge / row_bytes);
    r->subtiles = (ratio + r->st - 1) / r->st;
    // two blocks stream side by side when both fit the threads (one thread
    // per channel group of each): a stage's bias rows then serve both;
    // otherwise one block, its channel groups split over tpg threads
    if (2u * groups <= (uint32_t)kThreads) {
      r->bpu = 2;
      r->tpg = 1;
    } else {
      r->bpu = 1;
      int tpg = 1;
      while (tpg * 2 <= 32 && (uint32_t)(tpg * 2) * groups <= (uint32_t)kThreads) tpg *= 2;
      r->tpg = tpg;
    }
    r->in_bytes = (uint32_t)(r->st * row_bytes);
    r->stage_bytes = 2u * (uint32_t)r->bpu * r->in_bytes + (uint32_t)r->st * (uint32_t)dim * 4u;
  }
  r->bias_off = 128;
  r->ring_off = (r->bias_off + bias_bytes + 127u) / 128u * 128u;
  if (r->ring_off + 2u * r->stage_bytes > kRingBudget) return false;
  r->stages = (int32_t)((kRingBudget - r->ring_off) / r->stage_bytes);
  if (r->stages > kRingMaxStages) r->stages = kRingMaxStages;
  *smem = r->ring_off + (uint32_t)r->stages * r->stage_bytes;
  r->groups = (int32_t)groups;
  r->dim = dim;
  r->ratio = ratio;
  r->row_tokens = row_tokens;
  r->nblk = row_tokens / ratio;
  r->units_per_row = (r->nblk + r->bpu - 1) / r->bpu;
  return true;
}

lt_status launch(const void* func, dim3 grid, dim3 block, void* args, void* stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  void* a[] = {args};
  return cudaLaunchKernelExC(&cfg, func, a) == cudaSuccess ? LT_OK : LT_ERR_CUDA;
}

bool aligned_to(const void* p, unsigned a) { return p == nullptr || reinterpret_cast<uintptr_t>(p) % a == 0; }

lt_status device_sms(int* dev, int* sms) {
  if (cudaGetDevice(dev) != cudaSuccess) return LT_ERR_CUDA;
  if (*dev < 0 || *dev >= kMaxDevices) return LT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sms[*dev] == 0 &&
      cudaDeviceGetAttribute(&g_sms[*dev], cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess)
    return LT_ERR_CUDA;
  *sms = g_sms[*dev];
  return LT_OK;
}

}  // namespace

extern "C" {

lt_status lt_compress(const void* kv, const void* score, const float* bias, const int32_t* lengths,
                      int32_t rows, int64_t row_tokens, int32_t dim, int32_t ratio, void* out,
                      int32_t dtype, void* stream) {
  if (rows < 0 || row_tokens < 1 || dim < 1 || ratio < 1) return LT_ERR_INVALID_ARG;
  if (dtype != LT_DTYPE_F32 && dtype != LT_DTYPE_BF16) return LT_ERR_INVALID_ARG;
  if (rows > 0 && (kv == nullptr || score == nullptr || bias == nullptr || out == nullptr))
    return LT_ERR_INVALID_ARG;
  if (ratio > LT_MAX_RATIO) return LT_ERR_UNSUPPORTED;
  const int64_t nblk = row_tokens / ratio;
  if (rows == 0 || nblk == 0) return LT_OK;
  const bool bf16 = dtype == LT_DTYPE_BF16;
  {
    // the ring kernel whenever the layout allows bulk copies
    RParams rp = {};
    uint32_t smem = 0;
    if (ring_plan(kv, score, bias, out, row_tokens, dim, ratio, bf16, &rp, &smem)) {
      rp.kv = kv;
      rp.score = score;
      rp.bias = bias;
      rp.lengths = lengths;
      rp.out = out;
      rp.units = (int64_t)rows * rp.units_per_row;
      // CSA's 4:1 blocks take the fixed-column variant
      const bool fixed = rp.subtiles == 1 && ratio == 4 && kThreads % rp.groups == 0;
      const void* func =
          bf16 ? (fixed ? reinterpret_cast<const void*>(&compress_ring_kernel<uint16_t, 4>)
                        : reinterpret_cast<const void*>(&compress_ring_kernel<uint16_t, 0>))
               : (fixed ? reinterpret_cast<const void*>(&compress_ring_kernel<float, 4>)
                        : reinterpret_cast<const void*>(&compress_ring_kernel<float, 0>));
      const int kslot = (bf16 ? 2 : 0) + (fixed ? 1 : 0);
      int dev = 0, sms = 0;
      lt_status st = device_sms(&dev, &sms);
      if (st != LT_OK) return st;
      int per_sm = 0;
      {
        std::lock_guard<std::mutex> lk(g_mu);
        const int k = kslot;
        if ((int)smem > g_ring_smem_set[dev][k]) {
          if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return LT_ERR_CUDA;
          g_ring_smem_set[dev][k] = (int)smem;
          g_ring_ctas[dev][k] = 0;
        }
        if (g_ring_ctas[dev][k] == 0 &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_ring_ctas[dev][k], func, kThreads, smem) != cudaSuccess)
          return LT_ERR_CUDA;
        per_sm = g_ring_ctas[dev][k];
      }
      if (per_sm < 1) return LT_ERR_UNSUPPORTED;
      int64_t ctas = (int64_t)sms * per_sm;
      if (ctas > rp.units) ctas = rp.units;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)ctas);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = static_cast<cudaStream_t>(stream);
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr.val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      void* a[] = {&rp};
      return cudaLaunchKernelExC(&cfg, func, a) == cudaSuccess ? LT_OK : LT_ERR_CUDA;
    }
  }
  const unsigned va = bf16 ? 8u : 16u;
  const bool vec = dim % 4 == 0 && aligned_to(kv, va) && aligned_to(score, va) && aligned_to(out, va) &&
                   aligned_to(bias, 16u);
  const int V = vec ? 4 : 1;
  const int kind = (bf16 ? 2 : 0) + (vec ? 1 : 0);
  const void* func = bf16 ? (vec ? prefill_ptr<uint16_t, 4>() : prefill_ptr<uint16_t, 1>())
                          : (vec ? prefill_ptr<float, 4>() : prefill_ptr<float, 1>());
  CParams p = {};
  p.kv = kv;
  p.score = score;
  p.bias = bias;
  p.lengths = lengths;
  p.out = out;
  p.row_tokens = row_tokens;
  p.nblk = nblk;
  p.blocks = (int64_t)rows * nblk;
  p.dim = dim;
  p.ratio = ratio;
  p.groups = dim / V;
  // threads: x over a block's channel groups, y over blocks
  const int tx = p.groups < kThreads ? p.groups : kThreads;
  const int ty = kThreads / tx;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LT_ERR_UNSUPPORTED;
  int per_sm = 0, sms = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    per_sm = g_ctas_per_sm[dev][kind];
    sms = g_sms[dev];
  }
  if (per_sm == 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return LT_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, func, kThreads, 0) != cudaSuccess || per_sm < 1)
      return LT_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    g_ctas_per_sm[dev][kind] = per_sm;
    g_sms[dev] = sms;
  }
  // persistent grid: every resident CTA slot once, fewer when there are fewer blocks
  int64_t ctas = (p.blocks + ty - 1) / ty;
  const int64_t full = (int64_t)sms * per_sm;
  if (ctas > full) ctas = full;
  return launch(func, dim3((unsigned)ctas), dim3((unsigned)tx, (unsigned)ty), &p, stream);
}

lt_status lt_compress_decode(const void* kv_new, const void* score_new, const float* bias,
                             void* ring_kv, void* ring_score, const int32_t* pos, int32_t seqs,
                             int32_t dim, int32_t ratio, void* out, int32_t dtype, void* stream) {
  if (seqs < 0 || dim < 1 || ratio < 1) return LT_ERR_INVALID_ARG;
  if (dtype != LT_DTYPE_F32 && dtype != LT_DTYPE_BF16) return LT_ERR_INVALID_ARG;
  if (seqs > 0 && (kv_new == nullptr || score_new == nullptr || bias == nullptr || ring_kv == nullptr ||
                   ring_score == nullptr || pos == nullptr || out == nullptr))
    return LT_ERR_INVALID_ARG;
  if (ratio > LT_MAX_RATIO) return LT_ERR_UNSUPPORTED;
  if (seqs == 0) return LT_OK;
  const bool bf16 = dtype == LT_DTYPE_BF16;
  const unsigned va = bf16 ? 8u : 16u;
  const bool vec = dim % 4 == 0 && aligned_to(kv_new, va) && aligned_to(score_new, va) && aligned_to(out, va) &&
                   aligned_to(bias, 16u);
  DParams p = {};
  p.kv_new = kv_new;
  p.score_new = score_new;
  p.bias = bias;
  p.ring_kv = ring_kv;
  p.ring_score = ring_score;
  p.pos = pos;
  p.out = out;
  p.seqs = seqs;
  p.dim = dim;
  p.ratio = ratio;
  p.groups = vec ? dim / 4 : dim;
  const void* func =
      bf16 ? (vec ? reinterpret_cast<const void*>(&compress_decode_kernel<uint16_t, 4>)
                  : reinterpret_cast<const void*>(&compress_decode_kernel<uint16_t, 1>))
           : (vec ? reinterpret_cast<const void*>(&compress_decode_kernel<float, 4>)
                  : reinterpret_cast<const void*>(&compress_decode_kernel<float, 1>));
  const int64_t items = (int64_t)seqs * p.groups;
  return launch(func, dim3((unsigned)((items + kThreads - 1) / kThreads)), dim3(kThreads), &p, stream);
}

}  // extern "C"
