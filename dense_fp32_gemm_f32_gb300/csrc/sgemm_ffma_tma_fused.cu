// Instantiations of the FFMA kernel with the fused producer: 4-warp CTAs on
// 128 x 64 tiles, two per SM, thread 0 issuing the TMA copies.
#include "kernels.h"
#include "sgemm_ffma.cuh"

namespace gb300 {

template <int S, int MATH>
static KernelEntry entry() {
    return {reinterpret_cast<const void*>(&sgemm_ffma_kernel<S, kProducerFused, MATH, kBNFused>),
            ffma_smem_bytes<S, kBNFused>(), ffma_threads<kProducerFused>()};
}

KernelEntry ffma_kernel_tma_fused(int stages, int math) {
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

}  // namespace gb300
