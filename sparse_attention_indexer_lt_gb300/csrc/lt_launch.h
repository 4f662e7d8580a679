// lt_launch.h -- internal: kernel entry points shared by the C-ABI translation unit.
#pragma once

namespace lt {
struct Params;
const void* topk_kernel_ptr();
const void* blocked_kernel_ptr(int block);  // nullptr for an unsupported block size
}  // namespace lt
