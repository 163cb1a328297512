// The direct-A three-product TF32 kernel (registry entry).
#include "kernels.h"
#include "sgemm_3xtf32_direct.cuh"

namespace gb300 {

KernelEntry tf32x3_direct_kernel() {
    return {reinterpret_cast<const void*>(&sgemm_3xtf32_direct_kernel), kTdSmemBytes, kTdThreads};
}

}  // namespace gb300
