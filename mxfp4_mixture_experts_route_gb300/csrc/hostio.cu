// Host input staging for moe_forward_host: the step's x, in pinned host
// memory the GPU addresses over the CPU-GPU link, copied into the workspace
// by a kernel instead of a copy-engine transfer, so that the router (launched
// after it with programmatic dependent launch) starts and issues its weight
// loads while x crosses the link.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int STAGE_THREADS = 256;

// dst[i] = src[i] for i < n16 (16-byte chunks), one chunk a thread.  The
// loads go out at once, before the wait (the host buffer is an input of the
// call); the stores only after it: the previous call's kernels may still read
// the workspace's copy of x until then.
__global__ void __launch_bounds__(STAGE_THREADS) k_stage_in(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                            int n16) {
    pdl_trigger();
    const int i = blockIdx.x * STAGE_THREADS + threadIdx.x;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (i < n16) v = src[i];
    pdl_wait();
    if (i < n16) dst[i] = v;
}

}  // namespace

cudaError_t launch_stage_in(const void* src, void* dst, size_t bytes, cudaStream_t st) {
    const int n16 = (int)(bytes / 16);
    return launch_pdl(k_stage_in, dim3((n16 + STAGE_THREADS - 1) / STAGE_THREADS), dim3(STAGE_THREADS), 0, st,
                      reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), n16);
}

}  // namespace moe
