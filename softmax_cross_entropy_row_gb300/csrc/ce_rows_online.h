// Host-side interface of the loss-only warp-per-row kernel (ce_rows_online.cu).
// Internal to the library.
#pragma once

#include <cuda_runtime.h>

#include "ce_device.cuh"

namespace ce {

// One warp per row, rows of any length read once from global memory with a
// running max and a rescaled sum per lane: the loss alone (no gradient, no
// softmax output).  kOnlineWarps warps per CTA; `build` (0 .. kOnlineBuilds-1)
// selects the vectors per lane per step and the registers per thread.
constexpr int kOnlineWarps = 8;
constexpr int kOnlineBuilds = 5;
cudaError_t launch_rows_online(const ParamsEx &p, int dtype, int build, int ctas, cudaStream_t s);
cudaError_t rows_online_max_ctas_per_sm(int dtype, int build, int *ctas);

}  // namespace ce
