// Instantiations of the FFMA kernel with the cp.async producer (any alignment).
#include "kernels.h"
#include "sgemm_ffma.cuh"

namespace gb300 {

template <int S, int MATH>
static KernelEntry entry() {
    return {reinterpret_cast<const void*>(&sgemm_ffma_kernel<S, kProducerCpAsync, MATH>), ffma_smem_bytes<S>(),
            ffma_threads<kProducerCpAsync>()};
}

KernelEntry ffma_kernel_cpasync(int stages, int math) {
    if (math == kMathFfma) {
        switch (stages) {
            case 2: return entry<2, kMathFfma>();
            case 4: return entry<4, kMathFfma>();
        }
    } else if (math == kMathFfma2) {
        switch (stages) {
            case 2: return entry<2, kMathFfma2>();
            case 4: return entry<4, kMathFfma2>();
        }
    }
    return {nullptr, 0, 0};
}

}  // namespace gb300
