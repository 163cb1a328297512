// The three-product TF32 tensor-core kernels (registry entries).
#include "kernels.h"
#include "sgemm_3xtf32.cuh"

namespace gb300 {

KernelEntry tf32x3_kernel() {
    return {reinterpret_cast<const void*>(&sgemm_3xtf32_kernel<128, 32>), TcShape<128, 32>::kSmemBytes, kTcThreads};
}

KernelEntry tf32x3_res_kernel() {
    return {reinterpret_cast<const void*>(&sgemm_3xtf32_kernel<128, 32, false, true>),
            TcShape<128, 32, false, true>::kSmemBytes, kTcThreads};
}

KernelEntry tf32x3_wide_kernel() {
    return {reinterpret_cast<const void*>(&sgemm_3xtf32_kernel<256, 16>), TcShape<256, 16>::kSmemBytes, kTcThreads};
}

KernelEntry tf32x3_wide_pb_kernel() {
    return {reinterpret_cast<const void*>(&sgemm_3xtf32_kernel<256, 16, true>), TcShape<256, 16, true>::kSmemBytes,
            kTcThreads};
}

}  // namespace gb300
