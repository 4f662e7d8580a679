// lt_api.cu -- the C ABI: argument checks, launch planning and launches.
//
// Planning. One cluster of C CTAs owns one row. Two CTA shapes exist:
//   narrow: 256 threads, several CTAs per SM -- used when the batch alone has
//           at least one row per SM (C = 1: no cluster traffic at all);
//   wide:   512 threads, one CTA per SM -- used for few rows. C doubles (up
//           to 16, the largest cluster a GPC can host) while the whole grid
//           still fits on the SMs and each CTA still gets at least one round
//           (16384 positions) of the row.
// A 16-CTA cluster is non-portable. The plan asks the occupancy calculator how
// many clusters of the chosen shape can be resident at once and halves C until
// all rows fit in one wave (a cluster must sit inside one GPC, so sixteen
// 8-CTA clusters of one-CTA-per-SM kernels may not all fit although 128 SMs
// would). When every CTA's slice is a single register round the top-k kernel
// is its compact single-round variant. The two-level call with k_blocks >= k
// plans twice the rows (its plain top-k and stage-A groups run side by side).
// The streamed kernel is used only when asked for (force_kernel).

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "../../include/lt_topk.h"
#include "lt_device.cuh"
#include "lt_launch.h"
#include "lt_stream.cuh"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kWideThreads = 512;
constexpr int kNarrowThreads = 256;
constexpr int64_t kWideRound = 512 * 8 * 4;  // positions per CTA per round (wide)
constexpr int kTypeSlots = 23;                // kernel variants per score type
constexpr int kSlots = 2 * kTypeSlots;        // fp32, then bf16
// the streamed kernel's launch bounds: CTAs per SM for 256 / 512 threads
constexpr int stream_ctas_per_sm(int threads) { return threads == 256 ? 3 : 2; }
constexpr int kStreamMaxStages = 8;

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int smem_optin = 0;
  int smem_per_sm = 0;
  int smem_reserved = 0;
};

std::mutex g_mu;
// test hooks (lt_test_inject): launches still to fail, polls of the next
// streamed launch's stalled wait
std::atomic<int32_t> g_fail_launches{0};
std::atomic<int32_t> g_stall_polls{0};

bool take_one(std::atomic<int32_t>& n) {
  int32_t v = n.load(std::memory_order_relaxed);
  while (v > 0 && !n.compare_exchange_weak(v, v - 1, std::memory_order_relaxed)) {
  }
  return v > 0;
}
DeviceInfo g_dev[kMaxDevices];
int g_smem_set[kMaxDevices][kSlots];  // largest dynamic smem already granted per kernel
bool g_nonportable_set[kMaxDevices][kSlots];

int block_index(int block) {
  switch (block) {
    case 4: return 0;
    case 8: return 1;
    case 16: return 2;
    case 32: return 3;
    default: return -1;
  }
}

// slots 14..17: the listed-candidate kernel, by block size (512 threads, one
// CTA per row); 18: the top-k whose rows start from an earlier row's output;
// 19..22: the listed-candidate kernel with 256 threads (a cluster per row);
// bf16 kernels follow the fp32 ones (kTypeSlots later)
int kernel_slot(bool blocked, int block, int threads, bool stream = false, bool one_round = false,
                bool bf16 = false) {
  const int wide = threads == kWideThreads ? 1 : 0;
  const int base = bf16 ? kTypeSlots : 0;
  if (stream) return 10 + wide;
  if (!blocked) return base + (one_round ? 12 : 0) + wide;
  const int b = block_index(block);
  return b < 0 ? -1 : base + 2 + 2 * b + wide;
}

uint32_t next_pow2(uint32_t x) {
  uint32_t p = 1;
  while (p < x) p <<= 1;
  return p;
}

struct Plan {
  int kernel = LT_KERNEL_RESIDENT;
  int cluster = 1;
  int threads = kNarrowThreads;
  int grid = 0;             // CTAs launched
  bool one_round = false;   // top-k: every slice fits one register round
  uint32_t stages = 0;      // streamed kernel: ring stages
  uint32_t cap = 0;        // candidate slots: cluster * (1 << seg_shift)
  uint32_t seg_shift = 0;  // log2 of the slots each CTA of the cluster may fill
  uint32_t wstage = 0;     // candidate staging bytes (threads * 16 * kStageF4)
  uint32_t sel_cap = 0;
  uint32_t smem = 0;
  int hint_rows = 0;       // > 0: rows start from the output of the row this many earlier
  const void* func = nullptr;
};

lt_status device_info(DeviceInfo** out, int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return LT_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return LT_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
      return LT_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
      return LT_ERR_CUDA;
    d.ready = true;
  }
  *out = &d;
  *dev_out = dev;
  return LT_OK;
}

// Grant the kernel the shared memory and cluster size it needs (once per device).
lt_status prepare_kernel(int dev, int slot, const void* func, uint32_t smem, int cluster) {
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)smem > g_smem_set[dev][slot]) {
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return LT_ERR_CUDA;
    g_smem_set[dev][slot] = (int)smem;
  }
  if (cluster > 8 && !g_nonportable_set[dev][slot]) {
    // refused on devices without 16-CTA clusters: the plan then shrinks, so
    // the error is cleared (only when no earlier error was pending)
    const bool clean = cudaPeekAtLastError() == cudaSuccess;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
      if (clean) (void)cudaGetLastError();
      return LT_ERR_UNSUPPORTED;
    }
    g_nonportable_set[dev][slot] = true;
  }
  return LT_OK;
}

// Clusters of this shape that can be resident at once (0 when none fits).
// Queried once per device, kernel, cluster size and shared-memory size.
struct ActiveEntry {
  uint32_t smem = 0;
  int n = -1;
};
ActiveEntry g_active[kMaxDevices][kSlots][5];

int active_clusters_query(const void* func, int cluster, int threads, uint32_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cluster);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = (unsigned)cluster;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  // a caller's pending error must survive: clear only an error this query set
  const bool clean = cudaPeekAtLastError() == cudaSuccess;
  if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess) {
    if (clean) (void)cudaGetLastError();
    return 0;
  }
  return n;
}

int active_clusters(int dev, int slot, const void* func, int cluster, int threads, uint32_t smem) {
  int lc = 0;
  while ((1 << lc) < cluster) ++lc;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const ActiveEntry& e = g_active[dev][slot][lc];
    if (e.n >= 0 && e.smem == smem) return e.n;
  }
  const int n = active_clusters_query(func, cluster, threads, smem);
  std::lock_guard<std::mutex> lk(g_mu);
  g_active[dev][slot][lc].smem = smem;
  g_active[dev][slot][lc].n = n;
  return n;
}

lt_status make_stream_plan(int32_t rows, int64_t row_stride, int32_t k, int32_t force_cluster,
                           int32_t force_threads, DeviceInfo* di, int dev, Plan* plan);

lt_status make_plan(int32_t rows, int64_t row_stride, int32_t k, bool blocked, int32_t block,
                    int32_t k_blocks, int32_t force_cluster, int32_t force_threads, int32_t force_kernel,
                    bool aligned, bool bf16, Plan* plan, int* dev_out) {
  DeviceInfo* di = nullptr;
  int dev = 0;
  lt_status st = device_info(&di, &dev);
  if (st != LT_OK) return st;
  // The streamed kernel (bulk copies need 16-byte aligned rows) runs only
  // when asked for: measured on GB300 it does not yet beat the register-
  // resident kernel on the batched shapes, whose loads are all in flight from
  // their first instruction and which keeps three CTAs per SM.
  bool stream = false;
  if (force_kernel == LT_KERNEL_STREAM) {
    if (blocked || !aligned || bf16) return LT_ERR_UNSUPPORTED;
    stream = true;
  }
  if (stream) {
    st = make_stream_plan(rows, row_stride, k, force_cluster, force_threads, di, dev, plan);
    if (st == LT_OK) *dev_out = dev;
    return st;
  }

  int threads = force_threads;
  if (threads == 0) threads = (int64_t)rows >= di->sms ? kNarrowThreads : kWideThreads;
  if (kernel_slot(blocked, block, threads, false, false, bf16) < 0) return LT_ERR_UNSUPPORTED;
  plan->threads = threads;
  // the top-k kernel has a variant for slices of one register round
  auto pick = [&](int c, int* slot) -> const void* {
    if (blocked) {
      *slot = kernel_slot(true, block, threads, false, false, bf16);
      return lt::blocked_kernel_ptr(threads, block, bf16);
    }
    int64_t per = (row_stride + c - 1) / c;
    per = (per + 3) & ~(int64_t)3;
    plan->one_round = per <= lt::topk_round_positions(threads);
    *slot = kernel_slot(false, 4, threads, false, plan->one_round, bf16);
    return lt::topk_kernel_ptr(threads, plan->one_round, bf16);
  };
  int slot = 0;
  plan->func = pick(1, &slot);
  // candidate staging: kStageF4 float4 per thread
  plan->wstage = (uint32_t)threads * 16u * (uint32_t)lt::kStageF4;
  if (!plan->func) return LT_ERR_UNSUPPORTED;

  // Candidate capacity: about 4k slots per row (the sampled threshold keeps
  // roughly k to 1.5k items), split into one segment per CTA of the cluster,
  // each segment at least 256 slots so uneven slices still fit. Plans of one
  // 512-thread CTA per SM have shared memory to spare and take at least 4096
  // slots: the second estimate level (a histogram pass, a merge and a search,
  // about 3 us on a 262144-position row) then only runs when the first level
  // predicts more than 3072 candidates, instead of 1536.
  const uint32_t kmax = (uint32_t)(blocked ? (k > k_blocks ? k : k_blocks) : k);
  uint32_t base_cap = next_pow2(4 * kmax);
  base_cap = base_cap < 2048u ? 2048u : (base_cap > 4096u ? 4096u : base_cap);
  if (threads == kWideThreads && !blocked && base_cap < 4096u) base_cap = 4096u;
  plan->sel_cap = next_pow2(kmax < 32u ? 32u : kmax);

  int c = 1;
  if (force_cluster > 0) {
    c = force_cluster;
  } else if (threads == kWideThreads) {
    while (c < 16 && (int64_t)rows * 2 * c <= di->sms && (int64_t)c * kWideRound < row_stride) c *= 2;
  }
  for (;;) {
    plan->func = pick(c, &slot);
    if (!plan->func) return LT_ERR_UNSUPPORTED;
    uint32_t seg = base_cap;
    if (c > 1) {
      seg = next_pow2((base_cap + (uint32_t)c - 1) / (uint32_t)c);
      if (seg < 256u) seg = 256u;
    }
    plan->cap = (uint32_t)c * seg;
    plan->seg_shift = 0;
    while ((1u << plan->seg_shift) < seg) ++plan->seg_shift;
    const uint32_t smem = lt::make_layout(c > 1, plan->cap, plan->sel_cap, plan->wstage).total;
    if ((int)smem > di->smem_optin) return LT_ERR_UNSUPPORTED;
    st = prepare_kernel(dev, slot, plan->func, smem, c);
    if (st != LT_OK && !(st == LT_ERR_UNSUPPORTED && force_cluster == 0 && c > 8)) return st;
    // automatic plans also want every row's cluster resident at once (one
    // wave): large clusters need that many SMs free inside one GPC
    const int need = force_cluster > 0 ? 1 : (rows < 1 ? 1 : rows);
    if (st == LT_OK && (c == 1 || active_clusters(dev, slot, plan->func, c, threads, smem) >= need)) {
      plan->cluster = c;
      plan->smem = smem;
      break;
    }
    if (force_cluster > 0 || c == 1) return LT_ERR_UNSUPPORTED;
    c /= 2;
  }
  if ((int64_t)rows * plan->cluster > 0x7fffffffLL) return LT_ERR_UNSUPPORTED;
  plan->grid = rows * plan->cluster;
  // Batches of single-CTA rows of several rounds: a row may start from the
  // output of the row two waves of CTAs earlier, which has almost surely
  // finished (the automatic plan only).
  if (!blocked && force_kernel == LT_KERNEL_AUTO && threads == kNarrowThreads && plan->cluster == 1 &&
      !plan->one_round) {
    const int two_waves = 2 * di->sms * lt::kNarrowCtasPerSm;
    if (rows > two_waves) {
      const void* f = lt::topk_hint_kernel_ptr(bf16);
      st = prepare_kernel(dev, (bf16 ? kTypeSlots : 0) + 18, f, plan->smem, 1);
      if (st != LT_OK) return st;
      plan->func = f;
      plan->hint_rows = two_waves;
    }
  }
  *dev_out = dev;
  return LT_OK;
}

// Streamed kernel: three (256 threads) or two (512) CTAs per SM, as many ring
// stages as fit in that share of an SM's shared memory, persistent CTAs (each
// walks rows grid-stride). C doubles while every row's cluster still fits on the SMs
// twice over and each CTA keeps at least two chunks of the row.
lt_status make_stream_plan(int32_t rows, int64_t row_stride, int32_t k, int32_t force_cluster,
                           int32_t force_threads, DeviceInfo* di, int dev, Plan* plan) {
  int threads = force_threads;
  if (threads == 0) threads = (int64_t)rows >= 2 * di->sms ? kNarrowThreads : kWideThreads;
  const int slot = kernel_slot(false, 4, threads, true);
  plan->kernel = LT_KERNEL_STREAM;
  plan->threads = threads;
  plan->func = lt::stream_kernel_ptr(threads);
  if (!plan->func) return LT_ERR_UNSUPPORTED;
  plan->wstage = 0;
  const uint32_t chunk_pos = threads == kNarrowThreads ? (uint32_t)lt::SGeo<256, 4>::kChunk
                                                       : (uint32_t)lt::SGeo<512, 2>::kChunk;
  const uint32_t kmax = (uint32_t)k;
  uint32_t base_cap = next_pow2(4 * kmax);
  base_cap = base_cap < 2048u ? 2048u : (base_cap > 4096u ? 4096u : base_cap);
  plan->sel_cap = next_pow2(kmax < 32u ? 32u : kmax);
  const int cps = stream_ctas_per_sm(threads);
  const int slots_total = di->sms * cps;
  int c = 1;
  if (force_cluster > 0) {
    c = force_cluster;
  } else {
    while (c < 16 && (int64_t)rows * 2 * c <= slots_total && (int64_t)c * 2 * chunk_pos < row_stride) c *= 2;
  }
  // shared memory per CTA: the SM's share when several CTAs per SM are
  // wanted; the whole opt-in amount when the grid is one CTA per SM anyway
  const bool sparse = (int64_t)rows * c <= di->sms;
  const uint32_t budget = sparse ? (uint32_t)di->smem_optin
                                 : (uint32_t)(di->smem_per_sm / cps - di->smem_reserved);
  for (;;) {
    uint32_t seg = base_cap;
    if (c > 1) {
      seg = next_pow2((base_cap + (uint32_t)c - 1) / (uint32_t)c);
      if (seg < 256u) seg = 256u;
    }
    plan->cap = (uint32_t)c * seg;
    plan->seg_shift = 0;
    while ((1u << plan->seg_shift) < seg) ++plan->seg_shift;
    uint32_t ns = kStreamMaxStages;
    while (ns > 2 && lt::make_stream_layout(c > 1, plan->cap, plan->sel_cap, ns, 4 * chunk_pos).total > budget) --ns;
    const uint32_t smem = lt::make_stream_layout(c > 1, plan->cap, plan->sel_cap, ns, 4 * chunk_pos).total;
    if ((int)smem > di->smem_optin) return LT_ERR_UNSUPPORTED;
    lt_status st = prepare_kernel(dev, slot, plan->func, smem, c);
    if (st != LT_OK && !(st == LT_ERR_UNSUPPORTED && force_cluster == 0 && c > 8)) return st;
    int resident = 0;
    if (st == LT_OK) {
      if (c == 1) {
        int per_sm = 0;
        const bool clean = cudaPeekAtLastError() == cudaSuccess;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, plan->func, threads, smem) != cudaSuccess) {
          if (clean) (void)cudaGetLastError();
          per_sm = 0;
        }
        resident = per_sm * di->sms;
      } else {
        resident = active_clusters(dev, slot, plan->func, c, threads, smem);
      }
    }
    const int need = force_cluster > 0 ? 1 : (c == 1 ? 1 : rows);
    if (resident >= need) {
      plan->cluster = c;
      plan->smem = smem;
      plan->stages = ns;
      const int64_t clusters = rows < resident ? rows : resident;
      plan->grid = (int)(clusters * c);
      return LT_OK;
    }
    if (force_cluster > 0 || c == 1) return LT_ERR_UNSUPPORTED;
    c /= 2;
  }
}

// The listed-candidate call's launch: the listed kernel (reads only the
// listed blocks) or role 3 of the two-level kernel (whole-row scan). Sets
// *listed accordingly.
lt_status make_candidates_plan(int32_t rows, int64_t row_stride, int32_t block, int32_t n_cand, int32_t k,
                               bool bf16, bool aligned, int32_t force_cluster, int32_t force_threads,
                               int32_t force_exact, Plan* plan, int* dev, bool* listed) {
  lt_status st = LT_OK;
  // A list of at most one register round of blocks goes to the listed
  // kernel, which reads only those blocks; longer lists, forced cluster
  // shapes and force_exact scan whole rows with the two-level kernel.
  bool gathered = force_exact == 0 && (force_cluster == 0 || force_cluster == 1) &&
                  (force_threads == 0 || force_threads == kWideThreads) &&
                  (int64_t)n_cand <= lt::listed_round_blocks(block);
  if (gathered) {
    DeviceInfo* di = nullptr;
    st = device_info(&di, dev);
    if (st != LT_OK) return st;
    // a row's scattered block reads spread over a cluster of up to 8 CTAs
    // (256 threads each) while the rows' clusters still fit the SMs once;
    // rows enough to fill the SMs take one 512-thread CTA each
    // (rows too long for a bitmap of their blocks build the id list in a
    // hash set, in an order the CTAs of a cluster would not agree on: one CTA)
    int c = 1;
    const bool bitmap = (row_stride + block - 1) / block <= (int64_t)32 * lt::kBins;
    if (force_cluster == 0 && force_threads == 0 && bitmap)
      while (c < 8 && (int64_t)rows * c * 2 <= di->sms) c *= 2;
    const uint32_t sel_cap = next_pow2(k < 32 ? 32u : (uint32_t)k);
    for (;; c /= 2) {
      const int threads = c > 1 ? kNarrowThreads : kWideThreads;
      plan->threads = threads;
      plan->cluster = c;
      plan->grid = rows * c;
      // every CTA's segment holds every position of its share of the list
      plan->cap = (uint32_t)lt::kListedPositions;
      plan->seg_shift = 0;
      while ((1u << plan->seg_shift) < plan->cap / (uint32_t)c) ++plan->seg_shift;
      plan->wstage = (uint32_t)threads * 16u * (uint32_t)lt::kStageF4;
      plan->sel_cap = sel_cap;
      plan->func = lt::listed_kernel_ptr(threads, block, bf16);
      plan->smem = lt::make_layout(c > 1, plan->cap, plan->sel_cap, plan->wstage).total;
      gathered = plan->func != nullptr && (int)plan->smem <= di->smem_optin;
      if (!gathered) {
        if (c == 1) break;
        gathered = true;  // try a smaller cluster
        continue;
      }
      const int slot = (bf16 ? kTypeSlots : 0) + (c > 1 ? 19 : 14) + block_index(block);
      st = prepare_kernel(*dev, slot, plan->func, plan->smem, c);
      if (st != LT_OK) return st;
      if (c == 1 || active_clusters(*dev, slot, plan->func, c, threads, plan->smem) >= rows) break;
    }
  }
  if (!gathered) {
    st = make_plan(rows, row_stride, k, true, block, 1, force_cluster, force_threads, LT_KERNEL_AUTO,
                   aligned, bf16, plan, dev);
    if (st != LT_OK) return st;
    // every CTA holds a bitmap of its slice's blocks in kBins words
    int64_t per = (row_stride + plan->cluster - 1) / plan->cluster;
    per = (per + block - 1) / block;
    if (per > (int64_t)32 * lt::kBins) return LT_ERR_UNSUPPORTED;
  }
  *listed = gathered;
  return LT_OK;
}

lt_status check_common(const void* scores, int32_t rows, int64_t row_stride, int32_t k,
                       const int32_t* out_idx, int32_t force_cluster, int32_t force_threads) {
  if (rows < 0 || row_stride < 1 || k < 1) return LT_ERR_INVALID_ARG;
  if (!(force_threads == 0 || force_threads == kNarrowThreads || force_threads == kWideThreads))
    return LT_ERR_INVALID_ARG;
  if (rows > 0 && (scores == nullptr || out_idx == nullptr)) return LT_ERR_INVALID_ARG;
  if (!(force_cluster == 0 || force_cluster == 1 || force_cluster == 2 || force_cluster == 4 ||
        force_cluster == 8 || force_cluster == 16))
    return LT_ERR_INVALID_ARG;
  if (k > LT_MAX_K || row_stride > LT_MAX_ROW_STRIDE) return LT_ERR_UNSUPPORTED;
  return LT_OK;
}

lt_status launch(const Plan& plan, const lt::Params& prm, void* stream) {
  if (take_one(g_fail_launches)) return LT_ERR_CUDA;  // injected by a test
  lt::Params p = prm;
  if (plan.kernel == LT_KERNEL_STREAM) p.stall_polls = g_stall_polls.exchange(0, std::memory_order_relaxed);
  p.cap = (int32_t)plan.cap;
  p.seg_shift = (int32_t)plan.seg_shift;
  p.wstage = (int32_t)plan.wstage;
  p.sel_cap = (int32_t)plan.sel_cap;
  p.clustered = plan.cluster > 1 ? 1 : 0;
  p.ring_stages = (int32_t)plan.stages;
  p.hint_rows = plan.hint_rows;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan.grid);
  cfg.blockDim = dim3((unsigned)plan.threads);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  // programmatic dependent launch: this kernel's shared-memory setup may
  // overlap the previous kernel of the stream; every kernel waits for that
  // kernel's completion before it touches global memory
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = (unsigned)plan.cluster;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = plan.cluster > 1 ? 2 : 1;
  void* args[] = {&p};
  return cudaLaunchKernelExC(&cfg, plan.func, args) == cudaSuccess ? LT_OK : LT_ERR_CUDA;
}

// Every row start allows the vector loads of four scores: 16 bytes of fp32,
// 8 bytes of bf16.
bool rows_aligned(const void* p, int64_t row_stride, bool bf16) {
  return (reinterpret_cast<uintptr_t>(p) % (bf16 ? 8u : 16u)) == 0 && (row_stride % 4) == 0;
}

// A data pointer may be device memory or page-locked host memory mapped into
// the device's address space (the kernels then reach it over the host link,
// which on a Grace host is NVLink-C2C). Replaces *ptr with the address the
// device uses; unregistered host memory is refused. nullptr stays nullptr.
template <class P>
lt_status resolve_ptr(P** ptr, bool* host) {
  *host = false;
  if (*ptr == nullptr) return LT_OK;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, static_cast<const void*>(*ptr)) != cudaSuccess) return LT_ERR_CUDA;
  if (a.type == cudaMemoryTypeHost) {
    if (a.devicePointer == nullptr) return LT_ERR_INVALID_ARG;
    *ptr = static_cast<P*>(a.devicePointer);
    *host = true;
  } else if (a.type == cudaMemoryTypeUnregistered) {
    return LT_ERR_INVALID_ARG;
  }
  return LT_OK;
}

// The scores, lengths, lists and outputs of a call (counters and trace stay
// device memory).
lt_status resolve_data(const void** scores, bool* host_scores, const int32_t** lengths,
                       const int32_t** cand_blocks, int32_t** out_idx, float** out_val, int32_t** out_blocks) {
  bool h = false;
  lt_status st = resolve_ptr(scores, host_scores);
  if (st == LT_OK) st = resolve_ptr(lengths, &h);
  if (st == LT_OK && cand_blocks != nullptr) st = resolve_ptr(cand_blocks, &h);
  if (st == LT_OK) st = resolve_ptr(out_idx, &h);
  if (st == LT_OK && out_val != nullptr) st = resolve_ptr(out_val, &h);
  if (st == LT_OK && out_blocks != nullptr) st = resolve_ptr(out_blocks, &h);
  return st;
}

lt_status check_dtype(int32_t dtype) {
  return (dtype == LT_DTYPE_F32 || dtype == LT_DTYPE_BF16) ? LT_OK : LT_ERR_INVALID_ARG;
}

}  // namespace

extern "C" {

lt_status lt_topk_ex(const void* scores, int32_t dtype, const int32_t* lengths, int32_t rows,
                     int64_t row_stride, int32_t k, int32_t* out_idx, float* out_val, int32_t force_cluster,
                     int32_t force_threads, int32_t force_exact, int32_t force_kernel, int32_t* counters,
                     int64_t* trace, void* stream) {
  lt_status st = check_common(scores, rows, row_stride, k, out_idx, force_cluster, force_threads);
  if (st != LT_OK) return st;
  if (check_dtype(dtype) != LT_OK) return LT_ERR_INVALID_ARG;
  if (force_kernel < LT_KERNEL_AUTO || force_kernel > LT_KERNEL_STREAM) return LT_ERR_INVALID_ARG;
  if (rows == 0) return LT_OK;
  bool host = false;
  st = resolve_data(&scores, &host, &lengths, nullptr, &out_idx, &out_val, nullptr);
  if (st != LT_OK) return st;
  if (host && force_kernel == LT_KERNEL_STREAM) return LT_ERR_UNSUPPORTED;  // bulk copies read device memory
  const bool bf16 = dtype == LT_DTYPE_BF16;
  const bool aligned = rows_aligned(scores, row_stride, bf16);
  Plan plan;
  int dev = 0;
  st = make_plan(rows, row_stride, k, false, 4, 1, force_cluster, force_threads, force_kernel, aligned, bf16,
                 &plan, &dev);
  if (st != LT_OK) return st;
  lt::Params p = {};
  p.host_scores = host ? 1 : 0;
  p.scores = scores;
  p.lengths = lengths;
  p.row_stride = row_stride;
  p.out_idx = out_idx;
  p.out_val = out_val;
  p.out_blocks = nullptr;
  p.counters = counters;
  p.trace = trace;
  p.rows = rows;
  p.k = k;
  p.k_blocks = 1;
  p.force_exact = force_exact ? 1 : 0;
  p.vec_ok = aligned ? 1 : 0;
  return launch(plan, p, stream);
}

lt_status lt_topk(const float* scores, const int32_t* lengths, int32_t rows, int64_t row_stride,
                  int32_t k, int32_t* out_idx, float* out_val, void* stream) {
  return lt_topk_ex(scores, LT_DTYPE_F32, lengths, rows, row_stride, k, out_idx, out_val, 0, 0, 0,
                    LT_KERNEL_AUTO, nullptr, nullptr, stream);
}

lt_status lt_topk_bf16(const uint16_t* scores, const int32_t* lengths, int32_t rows, int64_t row_stride,
                       int32_t k, int32_t* out_idx, float* out_val, void* stream) {
  return lt_topk_ex(scores, LT_DTYPE_BF16, lengths, rows, row_stride, k, out_idx, out_val, 0, 0, 0,
                    LT_KERNEL_AUTO, nullptr, nullptr, stream);
}

lt_status lt_topk_blocked_ex(const void* scores, int32_t dtype, const int32_t* lengths, int32_t rows,
                             int64_t row_stride, int32_t block, int32_t k_blocks, int32_t k,
                             int32_t* out_idx, float* out_val, int32_t* out_blocks,
                             int32_t force_cluster, int32_t force_threads, int32_t force_exact,
                             int32_t* counters, int64_t* trace, void* stream) {
  lt_status st = check_common(scores, rows, row_stride, k, out_idx, force_cluster, force_threads);
  if (st != LT_OK) return st;
  if (check_dtype(dtype) != LT_OK) return LT_ERR_INVALID_ARG;
  const bool bf16 = dtype == LT_DTYPE_BF16;
  if (block < 1 || k_blocks < 1) return LT_ERR_INVALID_ARG;
  if (k_blocks > LT_MAX_K || block_index(block) < 0) return LT_ERR_UNSUPPORTED;
  if (rows == 0) return LT_OK;
  bool host = false;
  st = resolve_data(&scores, &host, &lengths, nullptr, &out_idx, &out_val, &out_blocks);
  if (st != LT_OK) return st;
  const bool aligned = rows_aligned(scores, row_stride, bf16);
  // k_blocks >= k: stage B equals the plain top-k, so the stages run as two
  // independent groups of clusters (see lt_blocked.cuh); the stage-A group
  // exists only when the kept blocks are wanted.
  const bool split = k_blocks >= k;
  const int groups = (split && out_blocks != nullptr) ? 2 : 1;
  if ((int64_t)rows * groups > 0x7fffffffLL) return LT_ERR_UNSUPPORTED;
  Plan plan;
  int dev = 0;
  st = make_plan(rows * groups, row_stride, k, true, block, k_blocks, force_cluster, force_threads,
                 LT_KERNEL_AUTO, aligned, bf16, &plan, &dev);
  if (st != LT_OK) return st;
  lt::Params p = {};
  p.host_scores = host ? 1 : 0;
  p.split = split ? 1 : 0;
  p.scores = scores;
  p.lengths = lengths;
  p.row_stride = row_stride;
  p.out_idx = out_idx;
  p.out_val = out_val;
  p.out_blocks = out_blocks;
  p.counters = counters;
  p.trace = trace;
  p.rows = rows;
  p.k = k;
  p.k_blocks = k_blocks;
  p.force_exact = force_exact ? 1 : 0;
  p.vec_ok = aligned ? 1 : 0;
  return launch(plan, p, stream);
}

lt_status lt_topk_blocked(const float* scores, const int32_t* lengths, int32_t rows,
                          int64_t row_stride, int32_t block, int32_t k_blocks, int32_t k,
                          int32_t* out_idx, float* out_val, int32_t* out_blocks, void* stream) {
  return lt_topk_blocked_ex(scores, LT_DTYPE_F32, lengths, rows, row_stride, block, k_blocks, k, out_idx,
                            out_val, out_blocks, 0, 0, 0, nullptr, nullptr, stream);
}

lt_status lt_topk_blocked_bf16(const uint16_t* scores, const int32_t* lengths, int32_t rows,
                               int64_t row_stride, int32_t block, int32_t k_blocks, int32_t k,
                               int32_t* out_idx, float* out_val, int32_t* out_blocks, void* stream) {
  return lt_topk_blocked_ex(scores, LT_DTYPE_BF16, lengths, rows, row_stride, block, k_blocks, k, out_idx,
                            out_val, out_blocks, 0, 0, 0, nullptr, nullptr, stream);
}

lt_status lt_topk_candidates_ex(const void* scores, int32_t dtype, const int32_t* lengths, int32_t rows,
                                int64_t row_stride, int32_t block, const int32_t* cand_blocks,
                                int32_t n_cand, int32_t k, int32_t* out_idx, float* out_val,
                                int32_t force_cluster, int32_t force_threads, int32_t force_exact,
                                int32_t* counters, int64_t* trace, void* stream) {
  lt_status st = check_common(scores, rows, row_stride, k, out_idx, force_cluster, force_threads);
  if (st != LT_OK) return st;
  if (check_dtype(dtype) != LT_OK) return LT_ERR_INVALID_ARG;
  const bool bf16 = dtype == LT_DTYPE_BF16;
  if (block < 1 || n_cand < 0 || (n_cand > 0 && cand_blocks == nullptr && rows > 0))
    return LT_ERR_INVALID_ARG;
  if (block_index(block) < 0) return LT_ERR_UNSUPPORTED;
  if (rows == 0) return LT_OK;
  bool host = false;
  st = resolve_data(&scores, &host, &lengths, &cand_blocks, &out_idx, &out_val, nullptr);
  if (st != LT_OK) return st;
  const bool aligned = rows_aligned(scores, row_stride, bf16);
  Plan plan;
  int dev = 0;
  bool listed = false;
  st = make_candidates_plan(rows, row_stride, block, n_cand, k, bf16, aligned, force_cluster, force_threads,
                            force_exact, &plan, &dev, &listed);
  if (st != LT_OK) return st;
  lt::Params p = {};
  p.host_scores = host ? 1 : 0;
  p.external = 1;
  p.cand_blocks = cand_blocks;
  p.n_cand = n_cand;
  p.scores = scores;
  p.lengths = lengths;
  p.row_stride = row_stride;
  p.out_idx = out_idx;
  p.out_val = out_val;
  p.out_blocks = nullptr;
  p.counters = counters;
  p.trace = trace;
  p.rows = rows;
  p.k = k;
  p.k_blocks = 1;
  p.force_exact = force_exact ? 1 : 0;
  p.vec_ok = aligned ? 1 : 0;
  return launch(plan, p, stream);
}

lt_status lt_topk_candidates(const float* scores, const int32_t* lengths, int32_t rows,
                             int64_t row_stride, int32_t block, const int32_t* cand_blocks,
                             int32_t n_cand, int32_t k, int32_t* out_idx, float* out_val,
                             void* stream) {
  return lt_topk_candidates_ex(scores, LT_DTYPE_F32, lengths, rows, row_stride, block, cand_blocks, n_cand,
                               k, out_idx, out_val, 0, 0, 0, nullptr, nullptr, stream);
}

lt_status lt_topk_candidates_bf16(const uint16_t* scores, const int32_t* lengths, int32_t rows,
                                  int64_t row_stride, int32_t block, const int32_t* cand_blocks,
                                  int32_t n_cand, int32_t k, int32_t* out_idx, float* out_val,
                                  void* stream) {
  return lt_topk_candidates_ex(scores, LT_DTYPE_BF16, lengths, rows, row_stride, block, cand_blocks,
                               n_cand, k, out_idx, out_val, 0, 0, 0, nullptr, nullptr, stream);
}

lt_status lt_topk_plan(int32_t rows, int64_t row_stride, int32_t k, int32_t blocked, int32_t block,
                       int32_t k_blocks, int32_t force_cluster, int32_t force_threads, int32_t force_kernel,
                       int32_t aligned, lt_plan_info* info) {
  if (rows < 1 || row_stride < 1 || k < 1 || info == nullptr) return LT_ERR_INVALID_ARG;
  if (!(force_threads == 0 || force_threads == kNarrowThreads || force_threads == kWideThreads))
    return LT_ERR_INVALID_ARG;
  if (force_kernel < LT_KERNEL_AUTO || force_kernel > LT_KERNEL_STREAM) return LT_ERR_INVALID_ARG;
  if (blocked && block_index(block) < 0) return LT_ERR_UNSUPPORTED;
  if (k > LT_MAX_K || row_stride > LT_MAX_ROW_STRIDE) return LT_ERR_UNSUPPORTED;
  if (blocked && (k_blocks < 1 || k_blocks > LT_MAX_K)) return LT_ERR_INVALID_ARG;
  Plan plan;
  int dev = 0;
  // the two-level call with k_blocks >= k launches two groups of clusters
  // (plain top-k, stage A) when kept blocks are wanted, as assumed here
  const int groups = (blocked && k_blocks >= k) ? 2 : 1;
  if ((int64_t)rows * groups > 0x7fffffffLL) return LT_ERR_UNSUPPORTED;
  lt_status st = make_plan(rows * groups, row_stride, k, blocked != 0, blocked ? block : 4, blocked ? k_blocks : 1,
                           force_cluster, force_threads, force_kernel, aligned != 0 && row_stride % 4 == 0,
                           false, &plan, &dev);
  if (st != LT_OK) return st;
  info->kernel = plan.kernel;
  info->cluster_size = plan.cluster;
  info->threads_per_cta = plan.threads;
  info->smem_bytes = (int32_t)plan.smem;
  info->grid_ctas = plan.grid;
  info->ring_stages = (int32_t)plan.stages;
  info->one_round = plan.one_round ? 1 : 0;
  return LT_OK;
}

lt_status lt_topk_candidates_plan(int32_t rows, int64_t row_stride, int32_t block, int32_t n_cand, int32_t k,
                                  int32_t dtype, int32_t force_cluster, int32_t force_threads,
                                  int32_t force_exact, int32_t aligned, lt_plan_info* info) {
  if (rows < 1 || row_stride < 1 || k < 1 || n_cand < 0 || block < 1 || info == nullptr) return LT_ERR_INVALID_ARG;
  if (check_dtype(dtype) != LT_OK) return LT_ERR_INVALID_ARG;
  if (!(force_threads == 0 || force_threads == kNarrowThreads || force_threads == kWideThreads))
    return LT_ERR_INVALID_ARG;
  if (!(force_cluster == 0 || force_cluster == 1 || force_cluster == 2 || force_cluster == 4 ||
        force_cluster == 8 || force_cluster == 16))
    return LT_ERR_INVALID_ARG;
  if (block_index(block) < 0 || k > LT_MAX_K || row_stride > LT_MAX_ROW_STRIDE) return LT_ERR_UNSUPPORTED;
  Plan plan;
  int dev = 0;
  bool listed = false;
  const lt_status st = make_candidates_plan(rows, row_stride, block, n_cand, k, dtype == LT_DTYPE_BF16,
                                            aligned != 0 && row_stride % 4 == 0, force_cluster, force_threads,
                                            force_exact, &plan, &dev, &listed);
  if (st != LT_OK) return st;
  info->kernel = listed ? LT_KERNEL_LISTED : plan.kernel;
  info->cluster_size = plan.cluster;
  info->threads_per_cta = plan.threads;
  info->smem_bytes = (int32_t)plan.smem;
  info->grid_ctas = plan.grid;
  info->ring_stages = (int32_t)plan.stages;
  info->one_round = plan.one_round ? 1 : 0;
  return LT_OK;
}

const char* lt_status_string(lt_status status) {
  switch (status) {
    case LT_OK: return "ok";
    case LT_ERR_INVALID_ARG: return "invalid argument";
    case LT_ERR_UNSUPPORTED: return "unsupported by this build (size, block or cluster limit)";
    case LT_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

int32_t lt_version(void) { return 400; }

lt_status lt_test_inject(int32_t what, int32_t value) {
  if (value < 0) return LT_ERR_INVALID_ARG;
  switch (what) {
    case LT_TEST_FAIL_LAUNCHES: g_fail_launches.store(value, std::memory_order_relaxed); return LT_OK;
    case LT_TEST_STALL_STREAMED: g_stall_polls.store(value, std::memory_order_relaxed); return LT_OK;
    default: return LT_ERR_INVALID_ARG;
  }
}

}  // extern "C"
