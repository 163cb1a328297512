// Instantiations of the FFMA kernel for the general entry: the scaled
// epilogue (C = alpha * A B + beta * C) in the variants its automatic plan
// picks (TMA producer with 2 stages, cp.async with 4; paired FMA; 128 x 128
// tiles), and the transposed-A kernels (TMA producer, 2 stages, paired FMA;
// plain and scaled).
#include "kernels.h"
#include "sgemm_ffma.cuh"

namespace gb300 {

KernelEntry ffma_kernel_scaled(int producer, int stages, int math) {
    if (math != kMathFfma2) return {nullptr, 0, 0};
    if (producer == kProducerTma && stages == 2)
        return {reinterpret_cast<const void*>(&sgemm_ffma_kernel<2, kProducerTma, kMathFfma2, kBN, true>),
                ffma_smem_bytes<2>(), ffma_threads<kProducerTma>()};
    if (producer == kProducerCpAsync && stages == 4)
        return {reinterpret_cast<const void*>(&sgemm_ffma_kernel<4, kProducerCpAsync, kMathFfma2, kBN, true>),
                ffma_smem_bytes<4>(), ffma_threads<kProducerCpAsync>()};
    return {nullptr, 0, 0};
}

KernelEntry ffma_kernel_amn(int stages, int math, bool scaled) {
    if (math != kMathFfma2 || stages != 2) return {nullptr, 0, 0};
    const void* fn = scaled
                         ? reinterpret_cast<const void*>(&sgemm_ffma_kernel<2, kProducerTma, kMathFfma2, kBN, true, true>)
                         : reinterpret_cast<const void*>(&sgemm_ffma_kernel<2, kProducerTma, kMathFfma2, kBN, false, true>);
    return {fn, ffma_smem_bytes<2>(), ffma_threads<kProducerTma>()};
}

}  // namespace gb300
