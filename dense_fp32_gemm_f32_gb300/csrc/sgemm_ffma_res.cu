// Instantiations of the FFMA kernel on residue-class tensor maps (operands of
// any alignment read in place; res_maps.cuh): TMA producer warp, two
// A-transposing warps and one B-shifting warp; 128 x 128 tiles, paired FMA,
// plain epilogue.
#include "kernels.h"
#include "sgemm_ffma.cuh"

namespace gb300 {

template <int S>
static KernelEntry entry() {
    constexpr bool kStg = ffma_tma_store<S, kProducerTmaX, kBN, false, false, kBK, true>();
    return {reinterpret_cast<const void*>(
                &sgemm_ffma_kernel<S, kProducerTmaX, kMathFfma2, kBN, false, false, false, kBK, true>),
            ffma_smem_bytes<S, kBN, true, false, kStg, kBK, true>(), ffma_threads<kProducerTmaX, true>(), kStg};
}

KernelEntry ffma_kernel_res(int stages, int math) {
    if (math != kMathFfma2) return {nullptr, 0, 0};
    switch (stages) {
        case 2: return entry<2>();
        case 3: return entry<3>();
        case 4: return entry<4>();
    }
    return {nullptr, 0, 0};
}

}  // namespace gb300
