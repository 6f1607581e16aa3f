// cake_bwd_grid.cu -- instantiates the cooperative single kernel with a grid barrier
// for every row layout and dw accumulation (see cake_bwd.cuh).
#include "cake_bwd.cuh"

namespace cake {

template cudaError_t launch_bwd_form<kFormGrid>(const BwdParams &, int, int, int, int, size_t, cudaStream_t);
template cudaError_t occ_bwd_form<kFormGrid>(int, int, int, int, size_t, int *);

} // namespace cake
