// lt_blocked_256_f32.cu -- two-level kernels with 256 threads per CTA, fp32 scores
// (one translation unit per thread count and score type, so they compile in parallel).
#include "lt_blocked.cuh"
#include "lt_launch.h"

namespace lt {
template const void* blocked_kernel_ptr_of<256, float>(int);
}  // namespace lt
