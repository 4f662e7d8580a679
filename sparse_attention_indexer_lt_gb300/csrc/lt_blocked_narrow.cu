// lt_blocked_narrow.cu -- two-level kernels with 256 threads per CTA.
#include "lt_blocked.cuh"
#include "lt_launch.h"

namespace lt {
const void* blocked_kernel_ptr_narrow(int block) { return blocked_ptr<256>(block); }
}  // namespace lt
