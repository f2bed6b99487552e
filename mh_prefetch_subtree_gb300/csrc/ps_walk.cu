// K3: the MH walk over each chain's prefetched subtree (PreSTO section 3.2
// step (3); Example 5; Algorithm 2, MHTransition), one warp per chain, four
// chains per CTA.  The walk of one chain is walk_chain() in ps_walk_chain.cuh,
// which the fused suffix-sum + walk kernel runs as well.
#include "ps_walk_chain.cuh"

namespace ps {
namespace {

constexpr int kWalkWarps = 4;

__global__ void __launch_bounds__(kWalkWarps * 32) walk_kernel(const WalkParams p) {
    __shared__ WalkSmem sm[kWalkWarps];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int c = blockIdx.x * kWalkWarps + warp;
    if (c >= p.n_chains) return;
    // Launched with programmatic dependent launch: wait for the previous
    // kernel in the stream before any load, since log A comes from it and the
    // caller may have written the tree or the uniforms with a kernel just
    // before this call.
    pdl_wait_prerequisites();
    walk_chain(p, c, sm[warp], lane);
}

}  // namespace

cudaError_t launch_walk(const WalkParams &p, cudaStream_t stream) {
    if (p.n_chains <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.n_chains + kWalkWarps - 1) / kWalkWarps));
    cfg.blockDim = dim3(kWalkWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, walk_kernel, p);
}

}  // namespace ps
