// Instantiations of the FFMA kernel with A transposed in shared memory
// (kProducerTmaX: TMA producer warp + two transposing warps); 128 x 128 tiles.
#include "kernels.h"
#include "sgemm_ffma.cuh"

namespace gb300 {

template <int S, int MATH, bool SCALED, bool EDGE = false>
static KernelEntry entry() {
    return {reinterpret_cast<const void*>(
                &sgemm_ffma_kernel<S, kProducerTmaX, MATH, kBN, SCALED, false, false, kBK, false, EDGE>),
            ffma_smem_bytes<S, kBN, true, false, ffma_tma_store<S, kProducerTmaX, kBN, SCALED, false>(), kBK,
                            false, EDGE>(),
            ffma_threads<kProducerTmaX>(), ffma_tma_store<S, kProducerTmaX, kBN, SCALED, false>()};
}

KernelEntry ffma_kernel_tma_x(int stages, int math, bool scaled, bool edge) {
    if (scaled) return (stages == 2 && math == kMathFfma2 && !edge) ? entry<2, kMathFfma2, true>()
                                                                    : KernelEntry{nullptr, 0, 0};
    if (edge) {
        if (math != kMathFfma2) return {nullptr, 0, 0};
        switch (stages) {
            case 2: return entry<2, kMathFfma2, false, true>();
            case 3: return entry<3, kMathFfma2, false, true>();
            case 4: return entry<4, kMathFfma2, false, true>();
        }
        return {nullptr, 0, 0};
    }
    if (math == kMathFfma) {
        switch (stages) {
            case 2: return entry<2, kMathFfma, false>();
            case 3: return entry<3, kMathFfma, false>();
            case 4: return entry<4, kMathFfma, false>();
        }
    } else if (math == kMathFfma2) {
        switch (stages) {
            case 2: return entry<2, kMathFfma2, false>();
            case 3: return entry<3, kMathFfma2, false>();
            case 4: return entry<4, kMathFfma2, false>();
        }
    }
    return {nullptr, 0, 0};
}

}  // namespace gb300
