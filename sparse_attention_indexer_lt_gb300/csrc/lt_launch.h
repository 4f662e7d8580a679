// lt_launch.h -- internal: kernel entry points shared by the C-ABI translation unit.
// bf16: the kernel reading bf16 scores (uint16_t bits) instead of fp32.
#pragma once

#include <cstdint>

namespace lt {
// threads is 256 (batched rows, several CTAs per SM) or 512 (few rows, one CTA per SM);
// one_round: the variant for slices of at most topk_round_positions(threads) positions.
const void* topk_kernel_ptr(int threads, bool one_round, bool bf16);
int64_t topk_round_positions(int threads);
// the 256-thread multi-round top-k whose rows start from an earlier row's output
const void* topk_hint_kernel_ptr(bool bf16);
// resident CTAs per SM of the 256-thread kernels (their launch bounds)
constexpr int kNarrowCtasPerSm = 3;
// nullptr for an unsupported block size or thread count.
const void* blocked_kernel_ptr(int threads, int block, bool bf16);
// one instantiation per (threads, score type), each in its own translation unit
template <int T, class S>
const void* blocked_kernel_ptr_of(int block);
extern template const void* blocked_kernel_ptr_of<256, float>(int);
extern template const void* blocked_kernel_ptr_of<256, uint16_t>(int);
extern template const void* blocked_kernel_ptr_of<512, float>(int);
extern template const void* blocked_kernel_ptr_of<512, uint16_t>(int);
// the streamed top-k kernel (fp32 scores): 256 threads (three CTAs per SM) or 512 (two)
const void* stream_kernel_ptr(int threads);
// listed-candidate kernel (only the listed blocks read): 512 threads with one
// CTA per row, 256 threads with a cluster per row; nullptr for an unsupported
// block size or thread count
const void* listed_kernel_ptr(int threads, int block, bool bf16);
int64_t listed_round_blocks(int block);
}  // namespace lt
