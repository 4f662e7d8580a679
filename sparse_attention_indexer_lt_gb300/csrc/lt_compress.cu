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

namespace {

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

// ---- the online softmax-weighted sum

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
  // add the n <= U tokens of a chunk: biased scores v, values x
  template <int U>
  __device__ __forceinline__ void add(const float (&v)[U][V], const float (&x)[U][V], int n) {
#pragma unroll
    for (int c = 0; c < V; ++c) {
      float cm = v[0][c];
#pragma unroll
      for (int u = 1; u < U; ++u)
        if (u < n) cm = fmaxf(cm, v[u][c]);
      const float mn = fmaxf(m[c], cm);
      const float r = __expf(m[c] - mn);  // 0 for the first chunk (m = -inf)
      float sc = s[c] * r, ac = a[c] * r;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (u < n) {
          const float e = __expf(v[u][c] - mn);
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
              for (int c = 0; c < V; ++c) v[u][c] = z[c] + bb[c];  // add
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
        for (int c = 0; c < V; ++c) v[u][c] = z[c] + bb[c];
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

template <class S, int V>
const void* prefill_ptr() { return reinterpret_cast<const void*>(&compress_kernel<S, V>); }

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
