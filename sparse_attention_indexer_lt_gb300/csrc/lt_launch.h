// lt_launch.h -- internal: kernel entry points shared by the C-ABI translation unit.
#pragma once

namespace lt {
// threads is 256 (batched rows, several CTAs per SM) or 512 (few rows, one CTA per SM).
const void* topk_kernel_ptr(int threads);
// nullptr for an unsupported block size.
const void* blocked_kernel_ptr(int threads, int block);
const void* blocked_kernel_ptr_narrow(int block);
const void* blocked_kernel_ptr_wide(int block);
// the streamed top-k kernel: 256 threads (three CTAs per SM) or 512 (two)
const void* stream_kernel_ptr(int threads);
}  // namespace lt
