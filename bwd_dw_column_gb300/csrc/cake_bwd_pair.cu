// cake_bwd_pair.cu -- instantiates the deterministic pair's main kernel
// for every row layout and dw accumulation (see cake_bwd.cuh).
#include "cake_bwd.cuh"

namespace cake {

template cudaError_t launch_bwd_form<kFormPair>(const BwdParams &, int, int, int, int, size_t, cudaStream_t);
template cudaError_t occ_bwd_form<kFormPair>(int, int, int, int, size_t, int *);

} // namespace cake
