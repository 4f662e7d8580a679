/*
 * lt_topk.h -- C ABI of the GB300 (sm_103a) indexer top-k library.
 *
 * The operation. Compressed sparse attention scores every compressed KV
 * position of a query row with an indexer and keeps only the k best positions
 * ("CSA: 4:1 compression + TopK selection", AICon 2026 Shenzhen speaker page,
 * abstract and outline section 1.1). At a million tokens that is a top-512 over
 * 262,144 positions, run in every layer; the pages name the kernel that does it
 * Lightning TopK: the row is split over the CTAs of one thread-block cluster,
 * each CTA builds a local histogram and the partial results are combined over
 * the SM-to-SM network instead of HBM (AICon page, outline section 3.2; SGLang
 * DeepSeek-V4 inference talk notes, section 3.2 "LightningTopK"). The two-level
 * variant restricts the top-512 to the positions of up to 2048 eight-position
 * candidate blocks chosen by block score (SGLang and Miles day-0 support for
 * DeepSeek-V4.1, Q&A on cross-layer sharing).
 *
 * The pages fix neither a tie rule nor an output order; this library fixes
 * both so that every row has exactly one correct answer:
 *   - positions are ranked by score descending, ties by index ascending;
 *   - -0.0 and +0.0 are equal; NaN ranks below -inf (NaNs tie, index decides);
 *   - the k outputs of a row are written in that rank order.
 *
 * Memory. Every pointer argument is DEVICE memory owned by the caller, with
 * one exception: scores, lengths, cand_blocks and the outputs may also be
 * page-locked host memory mapped into the device's address space
 * (cudaHostAlloc, or cudaHostRegister with mapping; mapped by default under
 * unified addressing), which the kernels then read or write over the host
 * link -- NVLink-C2C on a Grace host -- without staging copies (counters and
 * trace stay device memory). Other host memory returns LT_ERR_INVALID_ARG,
 * and the streamed kernel (LT_KERNEL_STREAM) returns LT_ERR_UNSUPPORTED for
 * host scores. The library allocates nothing, keeps no per-call state and
 * never synchronises the stream. Layouts are row-major:
 *   scores      float  [rows][row_stride]; row r is read on [0, L_r) only
 *               (the _bf16 calls: uint16_t bf16 bit patterns, same layout)
 *   lengths     int32  [rows] or NULL; L_r = clamp(lengths[r], 0, row_stride),
 *                      NULL means L_r = row_stride for every row
 *   out_idx     int32  [rows][k]; row-relative, 0-based positions
 *   out_val     float  [rows][k] or NULL; bit copies of scores[r][out_idx]
 *   out_blocks  int32  [rows][k_blocks] or NULL (two-level only)
 * A row with L_r < k fills slots [L_r, k) with index -1 and value -inf.
 * Rows whose start is 16-byte aligned (scores 16-byte aligned and row_stride a
 * multiple of 4) use 128-bit loads; bf16 rows need 8-byte aligned starts for
 * their 64-bit loads. Any other alignment takes scalar loads.
 *
 * bf16 scores. A low-precision indexer (the day-0 post on SGLang and Miles
 * for DeepSeek-V4.1 credits fused kernels and an FP4 indexer in its summary)
 * can hand its scores over in bf16, which halves the bytes this selection
 * reads. A bf16 score is ranked as the fp32 number it denotes
 * (its 16 bits as the upper half of an fp32, the rest zero: exact), under the
 * same rules; out_val receives that fp32 number.
 *
 * Errors. Argument errors return LT_ERR_INVALID_ARG or LT_ERR_UNSUPPORTED
 * synchronously and launch nothing. A failed launch returns LT_ERR_CUDA
 * (the CUDA error is left for cudaGetLastError). The kernels contain no
 * unbounded waits and no device-side traps.
 */
#ifndef LT_TOPK_H
#define LT_TOPK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum lt_status {
  LT_OK = 0,
  LT_ERR_INVALID_ARG = 1,  /* null pointer, k < 1, rows < 0, ... */
  LT_ERR_UNSUPPORTED = 2,  /* valid but outside this build's limits */
  LT_ERR_CUDA = 3          /* a CUDA runtime call failed */
} lt_status;

/* Score element types of the _ex calls. */
#define LT_DTYPE_F32 0
#define LT_DTYPE_BF16 1

/* Largest k and k_blocks accepted. */
#define LT_MAX_K 2048
/* Largest row_stride accepted (positions must fit a signed 32-bit index). */
#define LT_MAX_ROW_STRIDE 1073741824LL

/*
 * lt_topk -- per-row top-k of the indexer scores.
 *
 * For every row r in [0, rows): order the positions i in [0, L_r) by
 * (scores[r][i] descending, i ascending) and write the first min(k, L_r) to
 * out_idx[r][*] (and the copied scores to out_val[r][*]); pad the remaining
 * slots with (-1, -inf).
 *
 *   scores, lengths, rows, row_stride  as described above (rows >= 0,
 *                                      1 <= row_stride <= LT_MAX_ROW_STRIDE)
 *   k        1 <= k <= LT_MAX_K
 *   stream   a cudaStream_t (passed as void*); 0 is the legacy default stream
 *
 * rows == 0 returns LT_OK and launches nothing.
 */
lt_status lt_topk(const float* scores, const int32_t* lengths, int32_t rows, int64_t row_stride,
                  int32_t k, int32_t* out_idx, float* out_val, void* stream);

/* lt_topk over bf16 scores (uint16_t bit patterns); otherwise identical. */
lt_status lt_topk_bf16(const uint16_t* scores, const int32_t* lengths, int32_t rows, int64_t row_stride,
                       int32_t k, int32_t* out_idx, float* out_val, void* stream);

/*
 * lt_topk_blocked -- two-level, candidate-restricted top-k.
 *
 * Per row (L = L_r, nblocks = ceil(L / block)):
 *   stage A: block score of block j = max of scores[r][i] over its valid
 *            positions i in [j*block, min(L, (j+1)*block)); keep the first
 *            min(k_blocks, nblocks) blocks by (block score desc, block id asc);
 *   stage B: among the valid positions of the kept blocks, keep the first
 *            min(k, ncand) by (score desc, position asc).
 * out_idx / out_val are written as for lt_topk; out_blocks[r][*] (if not NULL)
 * receives the kept block ids in ascending order, padded with -1.
 *
 *   block     4, 8, 16 or 32 (the pages use 8)
 *   k_blocks  1 <= k_blocks <= LT_MAX_K
 *   k         1 <= k <= LT_MAX_K
 *
 * With k_blocks >= k every block holding one of the row's plain top-k
 * positions is kept, so stage B equals the plain top-k of the row; the
 * library then computes the two stages independently, side by side (same
 * results, bit for bit).
 */
lt_status lt_topk_blocked(const float* scores, const int32_t* lengths, int32_t rows,
                          int64_t row_stride, int32_t block, int32_t k_blocks, int32_t k,
                          int32_t* out_idx, float* out_val, int32_t* out_blocks, void* stream);

/* lt_topk_blocked over bf16 scores; otherwise identical. */
lt_status lt_topk_blocked_bf16(const uint16_t* scores, const int32_t* lengths, int32_t rows,
                               int64_t row_stride, int32_t block, int32_t k_blocks, int32_t k,
                               int32_t* out_idx, float* out_val, int32_t* out_blocks, void* stream);

/*
 * lt_topk_candidates -- top-k restricted to the positions of given blocks.
 *
 * The later layers' side of the cross-layer candidate sharing (SGLang and
 * Miles day-0 support for DeepSeek-V4.1, Q&A on cross-layer sharing): one
 * layer publishes its kept blocks (for example out_blocks of
 * lt_topk_blocked) and a later layer ranks its own scores only inside them.
 * Per row (L = L_r, nblocks = ceil(L / block)): the candidate positions are
 * the valid positions i < L of the listed blocks; keep the first
 * min(k, ncand) by (score desc, position asc), written as for lt_topk.
 *
 *   block        4, 8, 16 or 32
 *   cand_blocks  device int32[rows][n_cand], owned by the caller, read only:
 *                block ids in any order; ids outside [0, nblocks) are
 *                ignored (-1 pads a short list), a repeated id counts once
 *   n_cand       >= 0 (0: every row is all padding)
 *   k            1 <= k <= LT_MAX_K
 * Errors as for lt_topk; cand_blocks NULL with n_cand > 0 and rows > 0, a
 * negative n_cand or block < 1 return LT_ERR_INVALID_ARG.
 *
 * A list of at most 16384 / block entries per row (2048 blocks of 8) is
 * served by a kernel that reads only the listed blocks (any row length):
 * with few rows each row's unique blocks are shared out over a cluster of up
 * to 8 CTAs (rows of at most 65536 blocks), with enough rows to fill the SMs,
 * or a forced cluster of 1 or 512 threads, one CTA per row; longer lists,
 * and the _ex call with any other forced cluster or thread count or with
 * force_exact, scan whole rows, each
 * CTA of a row's cluster holding a bitmap of its own slice: those rows may
 * have at most 65536 blocks per CTA (for example 8,388,608 positions of
 * 8-blocks on 16 CTAs), else LT_ERR_UNSUPPORTED. Same results either way.
 */
lt_status lt_topk_candidates(const float* scores, const int32_t* lengths, int32_t rows,
                             int64_t row_stride, int32_t block, const int32_t* cand_blocks,
                             int32_t n_cand, int32_t k, int32_t* out_idx, float* out_val,
                             void* stream);

/* lt_topk_candidates over bf16 scores; otherwise identical. */
lt_status lt_topk_candidates_bf16(const uint16_t* scores, const int32_t* lengths, int32_t rows,
                                  int64_t row_stride, int32_t block, const int32_t* cand_blocks,
                                  int32_t n_cand, int32_t k, int32_t* out_idx, float* out_val,
                                  void* stream);

/* Kernels (force_kernel, lt_plan_info.kernel). */
#define LT_KERNEL_AUTO 0
/* Register-resident: each CTA holds its first rounds of the row in registers
 * and streams the rest with 128-bit loads; any alignment; one row per cluster. */
#define LT_KERNEL_RESIDENT 1
/* Streamed: 16-byte aligned rows move into a shared-memory ring by bulk
 * copies; persistent CTAs walk the rows and prefetch the next one. */
#define LT_KERNEL_STREAM 2
/* Listed: the listed-candidate kernel, which reads only the listed blocks
 * (reported by lt_topk_candidates_plan; not a force_kernel value). */
#define LT_KERNEL_LISTED 3

/*
 * Launch-plan control, for tests and measurement (not needed for normal use).
 *
 *   scores, dtype  the scores as for the plain calls; dtype LT_DTYPE_F32
 *                  (float) or LT_DTYPE_BF16 (uint16_t bf16 bits), anything
 *                  else returns LT_ERR_INVALID_ARG
 *   force_cluster  0 lets the planner choose; 1, 2, 4, 8 or 16 forces the
 *                  number of CTAs that share one row (16 needs a device that
 *                  can schedule a 16-CTA cluster, else LT_ERR_UNSUPPORTED)
 *   force_threads  0 lets the planner choose; 256 (several CTAs per SM, for
 *                  large batches) or 512 (one CTA per SM, for few rows)
 *   force_exact    nonzero skips the sampled-threshold fast path and runs the
 *                  streaming radix select on every row (same results)
 *   force_kernel   LT_KERNEL_AUTO lets the planner choose (register-resident;
 *                  in batches of more rows than one wave of single-CTA rows,
 *                  a row may start from the threshold implied by the output
 *                  of the row one wave earlier -- see below); forcing
 *                  LT_KERNEL_RESIDENT makes every row estimate its own;
 *                  LT_KERNEL_STREAM on unaligned or bf16 rows returns
 *                  LT_ERR_UNSUPPORTED
 *   counters       NULL, or device int32[LT_NUM_COUNTERS] that the kernel
 *                  increments atomically, once per row: [0] rows finished on
 *                  the fast path, [1] rows finished on the streaming radix
 *                  select, [2] rows whose candidate set overflowed, [3] rows
 *                  whose sampled threshold kept fewer than k candidates,
 *                  [4] rows of the streamed kernel during which a wait for a
 *                  bulk copy gave up after its poll limit (a hardware fault,
 *                  or lt_test_inject; that row's output is undefined),
 *                  [5] rows that started from an earlier row's threshold and
 *                  found it did not fit (they then count in [1] and [2] or
 *                  [3]), [6] rows that finished from such a threshold.
 *                  For the two-level call, each row counts once per stage
 *                  (with k_blocks >= k and out_blocks NULL, only stage B
 *                  runs: once); for the listed-candidate call, once (the
 *                  kernel that reads only the listed blocks always counts
 *                  [0]).
 *   trace          NULL, or device int64[grid CTAs * 16] receiving, from
 *                  thread 0 of each CTA, global-timer nanoseconds at phase
 *                  boundaries (entry, sample histogram, first cluster merge,
 *                  threshold, filter, candidate exchange, exact select,
 *                  output; the two-level kernel's second stage uses slots
 *                  9..14). CTA b of the grid is row b / cluster_size; a CTA
 *                  of the streamed kernel serves several rows and traces its
 *                  third (or, with fewer, its last). The entry timestamp is
 *                  written before the launch waits for the previous kernel
 *                  of the stream: give traced launches their own buffer or
 *                  synchronise between them.
 *
 * Thresholds from earlier rows. In a batch of single-CTA rows (256 threads,
 * several register rounds, more rows than two waves of resident CTAs) row r
 * reads the (k/2)-th and k-th values that row r - G wrote to out_val (G =
 * the CTAs of two waves; that row has almost surely finished) and, instead of
 * estimating, keeps the positions at or above k-th - 0.75 ((k/2)-th - k-th):
 * about 1.4k to 1.5k of a row like that one. The filter's count check accepts it
 * only if at least k and at most the candidate area pass; otherwise the row
 * takes the exact streaming select, as any miss does. Row r - G may still be being written (the
 * values are then stale, e.g. from a previous call into the same buffer):
 * a wrong guess costs time, never correctness. Needs out_val; results are
 * identical with or without it.
 *
 * Every launch uses programmatic dependent launch: a kernel may start while
 * the previous kernel of the stream finishes, and waits for it (device-side)
 * before it reads lengths or scores or writes outputs, counters or trace
 * slots other than the entry timestamp.
 */
#define LT_NUM_COUNTERS 7
lt_status lt_topk_ex(const void* scores, int32_t dtype, const int32_t* lengths, int32_t rows,
                     int64_t row_stride, int32_t k, int32_t* out_idx, float* out_val,
                     int32_t force_cluster, int32_t force_threads, int32_t force_exact,
                     int32_t force_kernel, int32_t* counters, int64_t* trace, void* stream);
lt_status lt_topk_blocked_ex(const void* scores, int32_t dtype, const int32_t* lengths, int32_t rows,
                             int64_t row_stride, int32_t block, int32_t k_blocks, int32_t k,
                             int32_t* out_idx, float* out_val, int32_t* out_blocks,
                             int32_t force_cluster, int32_t force_threads, int32_t force_exact,
                             int32_t* counters, int64_t* trace, void* stream);
lt_status lt_topk_candidates_ex(const void* scores, int32_t dtype, const int32_t* lengths, int32_t rows,
                                int64_t row_stride, int32_t block, const int32_t* cand_blocks,
                                int32_t n_cand, int32_t k, int32_t* out_idx, float* out_val,
                                int32_t force_cluster, int32_t force_threads, int32_t force_exact,
                                int32_t* counters, int64_t* trace, void* stream);

/*
 * lt_topk_plan -- the launch the planner would make, without launching.
 * blocked selects the two-level kernel (block and k_blocks are ignored
 * otherwise); aligned says whether the rows will be 16-byte aligned. Fills
 * *info (host memory, owned by the caller).
 */
typedef struct lt_plan_info {
  int32_t kernel;           /* LT_KERNEL_RESIDENT, LT_KERNEL_STREAM or LT_KERNEL_LISTED */
  int32_t cluster_size;     /* CTAs that share one row */
  int32_t threads_per_cta;
  int32_t smem_bytes;       /* dynamic shared memory per CTA */
  int32_t grid_ctas;        /* CTAs launched (streamed: persistent, rows grid-stride) */
  int32_t ring_stages;      /* streamed kernel: shared-memory ring stages, else 0 */
  int32_t one_round;        /* register-resident top-k: every CTA's slice is one
                               register round (the compact single-round variant) */
} lt_plan_info;
lt_status lt_topk_plan(int32_t rows, int64_t row_stride, int32_t k, int32_t blocked,
                       int32_t block, int32_t k_blocks, int32_t force_cluster,
                       int32_t force_threads, int32_t force_kernel, int32_t aligned,
                       lt_plan_info* info);
/* The launch lt_topk_candidates_ex would make for n_cand listed blocks per
 * row (dtype LT_DTYPE_F32 or LT_DTYPE_BF16): kernel LT_KERNEL_LISTED with its
 * cluster and grid, or the whole-row scan's plan (LT_KERNEL_RESIDENT). */
lt_status lt_topk_candidates_plan(int32_t rows, int64_t row_stride, int32_t block, int32_t n_cand,
                                  int32_t k, int32_t dtype, int32_t force_cluster,
                                  int32_t force_threads, int32_t force_exact, int32_t aligned,
                                  lt_plan_info* info);

/* Static description of a status code. */
const char* lt_status_string(lt_status status);

/* Library version, major*10000 + minor*100 + patch. */
int32_t lt_version(void);

/*
 * lt_test_inject -- failure injection for tests of the error paths (off unless
 * called; host-side state of the library, shared by all threads).
 *
 *   LT_TEST_FAIL_LAUNCHES   the next `value` launches return LT_ERR_CUDA
 *                           without launching anything and without setting a
 *                           CUDA error (0 cancels)
 *   LT_TEST_STALL_STREAMED  the next launch of the streamed kernel
 *                           (LT_KERNEL_STREAM) never issues the final bulk
 *                           copy of each CTA, and every one of its mbarrier
 *                           waits gives up after `value` polls (0 cancels):
 *                           the wait for that chunk runs out, counters[4]
 *                           records it, the kernel still finishes (no copy is
 *                           left in flight) and the affected rows' outputs are
 *                           undefined
 *
 * Returns LT_ERR_INVALID_ARG for an unknown `what` or a negative value.
 */
#define LT_TEST_FAIL_LAUNCHES 1
#define LT_TEST_STALL_STREAMED 2
lt_status lt_test_inject(int32_t what, int32_t value);

#ifdef __cplusplus
}
#endif

#endif /* LT_TOPK_H */
