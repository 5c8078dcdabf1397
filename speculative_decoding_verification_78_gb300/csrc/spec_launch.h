// spec_launch.h -- internal: per-translation-unit launchers of the verify kernel instances.
#pragma once

#include <cuda_runtime.h>

#include "spec_device.cuh"

namespace specv {

// Each launcher enqueues verify_kernel<E, MODE> (E chosen by dtype) and returns the launch
// status from cudaGetLastError.
cudaError_t launch_chain(int mode, int dtype, const Params &p, int grid, size_t smem,
                         cudaStream_t stream);
cudaError_t launch_tree(int dtype, const Params &p, int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_probs(int mode, int dtype, const Params &p, int grid, size_t smem,
                         cudaStream_t stream);

}  // namespace specv
