// Instantiations of the FFMA kernel on 128 x 256 tiles (8 x 16 accumulators
// per consumer thread), TMA producer warpgroup with the register split; A as
// stored, and (2 stages, paired FMA) A stored transposed.
#include "kernels.h"
#include "sgemm_ffma.cuh"

namespace gb300 {

template <int S, int MATH>
static KernelEntry entry() {
    return {reinterpret_cast<const void*>(&sgemm_ffma_kernel<S, kProducerTmaWg, MATH, kBNWide>),
            ffma_smem_bytes<S, kBNWide>(), ffma_threads<kProducerTmaWg>()};
}

KernelEntry ffma_kernel_tma_wide(int stages, int math) {
    if (math == kMathFfma) {
        switch (stages) {
            case 2: return entry<2, kMathFfma>();
            case 3: return entry<3, kMathFfma>();
            case 4: return entry<4, kMathFfma>();
        }
    } else if (math == kMathFfma2) {
        switch (stages) {
            case 2: return entry<2, kMathFfma2>();
            case 3: return entry<3, kMathFfma2>();
            case 4: return entry<4, kMathFfma2>();
        }
    }
    return {nullptr, 0, 0};
}

KernelEntry ffma_kernel_tma_wide_amn(int stages, int math) {
    if (math != kMathFfma2 || stages != 2) return {nullptr, 0, 0};
    return {reinterpret_cast<const void*>(&sgemm_ffma_kernel<2, kProducerTmaWg, kMathFfma2, kBNWide, false, true>),
            ffma_smem_bytes<2, kBNWide>(), ffma_threads<kProducerTmaWg>()};
}

}  // namespace gb300
