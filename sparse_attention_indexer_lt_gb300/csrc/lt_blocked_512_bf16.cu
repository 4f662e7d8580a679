// lt_blocked_512_bf16.cu -- two-level kernels with 512 threads per CTA, bf16 scores
// (one translation unit per thread count and score type, so they compile in parallel).
#include "lt_blocked.cuh"
#include "lt_launch.h"

namespace lt {
template const void* blocked_kernel_ptr_of<512, uint16_t>(int);
}  // namespace lt
