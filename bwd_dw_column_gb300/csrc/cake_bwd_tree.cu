// cake_bwd_tree.cu -- instantiates the single kernel with a two-level fixed-order reduce by the last CTAs
// for every row layout and dw accumulation (see cake_bwd.cuh).
#include "cake_bwd.cuh"

namespace cake {

template cudaError_t launch_bwd_form<kFormTree>(const BwdParams &, int, int, int, int, size_t, cudaStream_t);
template cudaError_t occ_bwd_form<kFormTree>(int, int, int, int, size_t, int *);

} // namespace cake
