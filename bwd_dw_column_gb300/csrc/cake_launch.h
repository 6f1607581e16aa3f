// cake_launch.h -- private interface between the C ABI (cake_api.cu) and the
// kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include "cake_params.h"

namespace cake {

// Raise a kernel's dynamic shared memory limit once per (device, kernel).
cudaError_t ensure_smem_attr(const void *kernel, size_t smem);

cudaError_t launch_fwd(const FwdParams &p, int vpt, int ctas, size_t smem, cudaStream_t stream);
// The backward row kernel: the pair's main kernel (single = 0) or the
// single kernel (single = 1).
cudaError_t launch_bwd_rows(const BwdParams &p, int vpt, int single, int dwm, int ctas, size_t smem,
                            cudaStream_t stream);
// The pair's fixed-order reduce of the CTA partials.
cudaError_t launch_dw_reduce(const ReduceParams &rp, cudaStream_t stream);

// Resident CTAs per SM the runtime reports for a row kernel and launch shape.
cudaError_t occupancy_fwd(int vpt, int lanes, int threads, size_t smem, int *n);
cudaError_t occupancy_bwd(int vpt, int w, int rpg, int lanes, int single, int dwm, int threads, size_t smem, int *n);

cudaError_t fwd_status(int *code, int clear);
cudaError_t bwd_status(int *code, int clear);

} // namespace cake
