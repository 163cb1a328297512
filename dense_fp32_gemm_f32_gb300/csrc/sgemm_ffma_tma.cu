// Instantiations of the FFMA kernel with the tensor-map (TMA) producer.
#include "kernels.h"
#include "sgemm_ffma.cuh"

namespace gb300 {

template <int S, int MATH>
static KernelEntry entry() {
    return {reinterpret_cast<const void*>(&sgemm_ffma_kernel<S, kProducerTma, MATH>), ffma_smem_bytes<S>(),
            ffma_threads<kProducerTma>()};
}

KernelEntry ffma_kernel_tma(int stages, int math) {
    if (math == kMathFfma) {
        switch (stages) {
            case 1: return entry<1, kMathFfma>();
            case 2: return entry<2, kMathFfma>();
            case 3: return entry<3, kMathFfma>();
            case 4: return entry<4, kMathFfma>();
            case 5: return entry<5, kMathFfma>();
            case 6: return entry<6, kMathFfma>();
        }
    } else if (math == kMathFfma2) {
        switch (stages) {
            case 1: return entry<1, kMathFfma2>();
            case 2: return entry<2, kMathFfma2>();
            case 3: return entry<3, kMathFfma2>();
            case 4: return entry<4, kMathFfma2>();
            case 5: return entry<5, kMathFfma2>();
            case 6: return entry<6, kMathFfma2>();
        }
    }
    return {nullptr, 0, 0};
}

}  // namespace gb300
