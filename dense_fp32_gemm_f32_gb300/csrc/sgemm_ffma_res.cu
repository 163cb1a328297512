// Instantiations of the FFMA kernel on residue-class tensor maps (operands of
// any alignment read in place; res_maps.cuh): TMA producer warp, two
// A-transposing warps and one B-shifting warp; 128 x 128 tiles, paired FMA;
// plain epilogue (2-4 stages) and the general entry's scaled one (2 stages).
#include "kernels.h"
#include "sgemm_ffma.cuh"

namespace gb300 {

template <int S, bool SCALED = false, bool EDGE = false>
static KernelEntry entry() {
    constexpr bool kStg = ffma_tma_store<S, kProducerTmaX, kBN, SCALED, false, kBK, true>();
    return {reinterpret_cast<const void*>(
                &sgemm_ffma_kernel<S, kProducerTmaX, kMathFfma2, kBN, SCALED, false, false, kBK, true, EDGE>),
            ffma_smem_bytes<S, kBN, true, false, kStg, kBK, true, EDGE>(), ffma_threads<kProducerTmaX, true>(), kStg};
}

KernelEntry ffma_kernel_res(int stages, int math, bool scaled, bool edge) {
    if (math != kMathFfma2) return {nullptr, 0, 0};
    if (scaled) return (stages == 2 && !edge) ? entry<2, true>() : KernelEntry{nullptr, 0, 0};
    switch (stages) {
        case 2: return edge ? entry<2, false, true>() : entry<2>();
        case 3: return edge ? entry<3, false, true>() : entry<3>();
        case 4: return edge ? entry<4, false, true>() : entry<4>();
    }
    return {nullptr, 0, 0};
}

}  // namespace gb300
