// cake_bwd_atomic.cu -- instantiates the single kernel with FP64 column atomics
// for every row layout and dw accumulation (see cake_bwd.cuh).
#include "cake_bwd.cuh"

namespace cake {

template cudaError_t launch_bwd_form<kFormAtomic>(const BwdParams &, int, int, int, int, size_t, cudaStream_t);
template cudaError_t occ_bwd_form<kFormAtomic>(int, int, int, int, size_t, int *);

} // namespace cake
