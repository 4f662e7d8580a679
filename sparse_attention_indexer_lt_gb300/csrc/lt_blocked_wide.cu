// lt_blocked_wide.cu -- two-level kernels with 512 threads per CTA.
#include "lt_blocked.cuh"
#include "lt_launch.h"

namespace lt {
const void* blocked_kernel_ptr_wide(int block) { return blocked_ptr<512>(block); }
const void* blocked_kernel_ptr(int threads, int block) {
  if (threads == 256) return blocked_kernel_ptr_narrow(block);
  if (threads == 512) return blocked_kernel_ptr_wide(block);
  return nullptr;
}
}  // namespace lt
