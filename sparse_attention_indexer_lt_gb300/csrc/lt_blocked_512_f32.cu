// lt_blocked_512_f32.cu -- two-level kernels with 512 threads per CTA, fp32 scores
// (one translation unit per thread count and score type, so they compile in parallel).
#include "lt_blocked.cuh"
#include "lt_launch.h"

namespace lt {
template const void* blocked_kernel_ptr_of<512, float>(int);
}  // namespace lt
