// Instantiations of the FFMA kernel with A transposed in shared memory
// (kProducerTmaX) on 16-deep K slices (sgemm_options.tile_k = 16); 128 x 128
// tiles, paired FMA, plain epilogue.
#include "kernels.h"
#include "sgemm_ffma.cuh"

namespace gb300 {

template <int S>
static KernelEntry entry() {
    constexpr bool kStg = ffma_tma_store<S, kProducerTmaX, kBN, false, false, kBK16>();
    return {reinterpret_cast<const void*>(
                &sgemm_ffma_kernel<S, kProducerTmaX, kMathFfma2, kBN, false, false, false, kBK16>),
            ffma_smem_bytes<S, kBN, true, false, kStg, kBK16>(), ffma_threads<kProducerTmaX>(), kStg};
}

KernelEntry ffma_kernel_tma_x16(int stages, int math) {
    if (math != kMathFfma2) return {nullptr, 0, 0};
    switch (stages) {
        case 2: return entry<2>();
        case 3: return entry<3>();
        case 4: return entry<4>();
        case 6: return entry<6>();
    }
    return {nullptr, 0, 0};
}

}  // namespace gb300
