// Pass 2 of rumus 0.1.1's cross_entropy.wgsl as a launch of its own: the batch
// loss from row losses that earlier launches wrote (the host-buffer entry
// points compute a batch in chunks of rows, each chunk's kernel writing its
// rows' losses).  One CTA sums them in the fixed order every fused kernel's
// last CTA uses, so the loss has the same bits as a single fused launch.
#include "ce_launch.h"

namespace ce {
namespace {

__global__ void __launch_bounds__(kTailThreads) batch_loss_kernel(Params p) {
    __shared__ float2 scratch[kTailWarps];
    pdl_wait();  // the row losses of the launches before
    batch_tail(p, scratch);
}

}  // namespace

cudaError_t launch_batch_loss(const Params &p, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(kTailThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, batch_loss_kernel, p);
}

}  // namespace ce
