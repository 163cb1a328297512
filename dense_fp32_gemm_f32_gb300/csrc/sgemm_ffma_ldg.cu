// Instantiations of the FFMA kernel with loader warps (kProducerLdg: A and
// B of any alignment read from global memory by four producer warps); 128 x
// 128 tiles, paired FMA, plain epilogue; 2, 3 or 4 stages.
#include "kernels.h"
#include "sgemm_ffma.cuh"

namespace gb300 {

template <int S>
static KernelEntry entry() {
    constexpr bool kStg = ffma_tma_store<S, kProducerLdg, kBN, false, false>();
    return {reinterpret_cast<const void*>(&sgemm_ffma_kernel<S, kProducerLdg, kMathFfma2, kBN>),
            ffma_smem_bytes<S, kBN, false, false, kStg>(), ffma_threads<kProducerLdg>(), kStg};
}

KernelEntry ffma_kernel_ldg(int stages, int math) {
    if (math != kMathFfma2) return {nullptr, 0, 0};
    switch (stages) {
        case 2: return entry<2>();
        case 3: return entry<3>();
        case 4: return entry<4>();
    }
    return {nullptr, 0, 0};
}

}  // namespace gb300
