// Instantiations of the FFMA kernel with the TMA producer in a warpgroup of
// its own and the setmaxnreg register split (kProducerTmaWg).
#define FFMA_TMA_WG 1
#include "sgemm_ffma_tma.cu"
