// lt_launch.h -- internal: kernel entry points shared by the C-ABI translation unit.
#pragma once

namespace lt {
// threads is 256 (batched rows, several CTAs per SM) or 512 (few rows, one CTA per SM);
// one_round: the variant for slices of at most topk_round_positions(threads) positions.
const void* topk_kernel_ptr(int threads, bool one_round);
int64_t topk_round_positions(int threads);
// nullptr for an unsupported block size.
const void* blocked_kernel_ptr(int threads, int block);
const void* blocked_kernel_ptr_narrow(int block);
const void* blocked_kernel_ptr_wide(int block);
// the streamed top-k kernel: 256 threads (three CTAs per SM) or 512 (two)
const void* stream_kernel_ptr(int threads);
// listed-candidate kernel (512 threads, one CTA per row, only the listed
// blocks read): nullptr for an unsupported block size
const void* listed_kernel_ptr(int block);
int64_t listed_round_blocks(int block);
}  // namespace lt
