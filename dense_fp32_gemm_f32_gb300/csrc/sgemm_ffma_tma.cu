// Instantiations of the FFMA kernel with the tensor-map (TMA) producer:
// producer warp + 8 consumer warps (PRODUCER = kProducerTma), or, when this
// file is compiled with FFMA_TMA_WG defined, producer warpgroup with the
// register split (kProducerTmaWg).
#include "kernels.h"
#include "sgemm_ffma.cuh"

namespace gb300 {

#ifdef FFMA_TMA_WG
constexpr int kProd = kProducerTmaWg;
#define FFMA_TMA_REGISTRY ffma_kernel_tma_wg
#else
constexpr int kProd = kProducerTma;
#define FFMA_TMA_REGISTRY ffma_kernel_tma
#endif

template <int S, int MATH>
static KernelEntry entry() {
    return {reinterpret_cast<const void*>(&sgemm_ffma_kernel<S, kProd, MATH>), ffma_smem_bytes<S>(),
            ffma_threads<kProd>()};
}

KernelEntry FFMA_TMA_REGISTRY(int stages, int math) {
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
