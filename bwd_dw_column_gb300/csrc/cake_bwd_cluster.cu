// cake_bwd_cluster.cu -- instantiates the cluster form (one cluster of CTAs
// reducing dw over distributed shared memory) for every row layout and dw
// accumulation (see cake_bwd.cuh).
#include "cake_bwd.cuh"

namespace cake {

template cudaError_t launch_bwd_form<kFormCluster>(const BwdParams &, int, int, int, int, size_t, cudaStream_t);
template cudaError_t occ_bwd_form<kFormCluster>(int, int, int, int, size_t, int *);

} // namespace cake
