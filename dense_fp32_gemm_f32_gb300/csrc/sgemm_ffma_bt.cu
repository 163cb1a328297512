// Instantiations of the FFMA kernel for the general entry's op(B) = B^T read
// in place (B stored N x K): TMA producer warp + one B-transposing warp, with
// A either transposed in shared memory by two more warps (op(A) = A, stored
// M x K) or loaded as stored transposed (op(A) = A^T, stored K x M); 128 x 128
// tiles, 2 stages, paired FMA; plain and scaled epilogues.
#include "kernels.h"
#include "sgemm_ffma.cuh"

namespace gb300 {

template <int PROD, bool SCALED, bool AMN>
static KernelEntry entry() {
    constexpr bool kStg = ffma_tma_store<2, PROD, kBN, SCALED, true>();
    return {reinterpret_cast<const void*>(&sgemm_ffma_kernel<2, PROD, kMathFfma2, kBN, SCALED, AMN, true>),
            ffma_smem_bytes<2, kBN, PROD == kProducerTmaX, true, kStg>(), ffma_threads<PROD, true>(), kStg};
}

KernelEntry ffma_kernel_bnk(bool a_mn, bool scaled) {
    if (a_mn) return scaled ? entry<kProducerTma, true, true>() : entry<kProducerTma, false, true>();
    return scaled ? entry<kProducerTmaX, true, false>() : entry<kProducerTmaX, false, false>();
}

}  // namespace gb300
