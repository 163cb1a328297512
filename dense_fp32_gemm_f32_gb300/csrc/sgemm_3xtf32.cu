// The three-product TF32 tensor-core kernel (registry entry).
#include "kernels.h"
#include "sgemm_3xtf32.cuh"

namespace gb300 {

KernelEntry tf32x3_kernel() {
    return {reinterpret_cast<const void*>(&sgemm_3xtf32_kernel), kTcSmemBytes, kTcThreads};
}

}  // namespace gb300
