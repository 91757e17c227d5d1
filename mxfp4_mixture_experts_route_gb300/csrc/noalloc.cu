// moe_forward_noalloc: the whole block without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// block: a plugin or operator interface that hands over only input and output
// buffers, an application whose memory pool owns every byte of the GPU and
// forbids outside cudaMalloc calls, or a latency-critical serving loop where a
// cudaMalloc (which may synchronise the device) is not acceptable.  For them
// this entry point uses a fixed scratch area that lives in the library itself:
// a file-scope static device array, held by every GPU that loads it until the
// process exits.  The library's translation units are separate device
// modules, loaded lazily by default (CUDA_MODULE_LOADING=LAZY): the array is
// reserved when the first call on a device loads this file's module (the
// address lookup below).  A caller whose memory pool takes the whole GPU makes
// that first call, as a warm-up, before the pool claims its memory (and
// before any stream capture).  No call here allocates or frees memory itself.
#include "moe_internal.cuh"

#include <mutex>
#include <stdio.h>

namespace moe {

namespace {

// Size of the static scratch area.  A shape whose workspace (moe_workspace_bytes)
// is larger is rejected with MOE_ERR_WORKSPACE.
constexpr size_t kNoallocScratchBytes = size_t(32) << 20;   // 32 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};   // device address of the array, per device
std::mutex g_setup_mutex;

// The array's name is only a host-side stand-in in host code; its device
// address comes from cudaGetSymbolAddress, asked once per device with that
// device current.
int scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_NO_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            fprintf(stderr,
                    "libmoe: moe_forward_noalloc could not load its %zu-byte scratch array on device %d: %s%s\n",
                    kNoallocScratchBytes, dev, cudaGetErrorString(e),
                    e == cudaErrorMemoryAllocation ? " (make the first call before a memory pool takes the GPU)" : "");
            return MOE_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" int moe_forward_noalloc(const moe_shape* shape, const void* x, const void* w_gate,
                                   const float* bias, const float* logit_off, const uint8_t* w13,
                                   const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s,
                                   const float* norm_w, int32_t* ids, float* weights, float* out,
                                   int32_t* status, void* stream) {
    size_t need = 0;
    int rc = moe_workspace_bytes(shape, &need);
    if (rc) return rc;
    if (need > kNoallocScratchBytes) return MOE_ERR_WORKSPACE;
    // every argument check of moe_forward first: a rejected call touches
    // neither the device nor the array (which an earlier call may still use)
    rc = check_forward_args(shape, x, w_gate, bias, logit_off, w13, w13s, w2, w2s, norm_w, ids, weights, out);
    if (rc) return rc;
    void* ws = nullptr;
    rc = scratch_for_current_device(&ws);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    // the array keeps the previous call's contents: the status block (error
    // latch, per-call counters) and the sort counters must start at zero
    if (cudaMemsetAsync(ws, 0, WS_ZERO_PREFIX, st) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    rc = moe_forward(shape, x, w_gate, bias, logit_off, w13, w13s, w2, w2s, norm_w, ids, weights, out, ws,
                     kNoallocScratchBytes, stream);
    if (rc) return rc;
    if (status != nullptr &&
        cudaMemcpyAsync(status, ws, 2 * sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}
