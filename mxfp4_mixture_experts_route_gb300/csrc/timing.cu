// Diagnostic per-kernel timing (moe_timing_enable / moe_timing_collect): a
// fixed ring of CUDA event pairs recorded around the library's launches.
#include "moe_internal.cuh"

#include <vector>

namespace moe {

namespace {

struct Rec {
    int kernel;
    cudaEvent_t a, b;
};

std::vector<Rec> g_recs;   // event pairs, created by moe_timing_enable
int g_used = 0;            // pairs recorded since the last collect
int g_open = -1;           // pair started by timing_begin, not yet ended

const char* const kNames[K_NUM] = {"router_logits", "topk", "sort", "gather", "experts", "combine", "topk_sort_gather",
                                   "latent_down", "latent_mid", "latent_up"};

void free_all() {
    for (auto& r : g_recs) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    g_recs.clear();
    g_used = 0;
    g_open = -1;
}

}  // namespace

void timing_begin(int kernel_id, cudaStream_t st) {
    if (g_used >= (int)g_recs.size()) return;
    g_open = g_used++;
    g_recs[g_open].kernel = kernel_id;
    cudaEventRecord(g_recs[g_open].a, st);
}

void timing_end(cudaStream_t st) {
    if (g_open < 0) return;
    cudaEventRecord(g_recs[g_open].b, st);
    g_open = -1;
}

#ifdef MOE_TRACE
unsigned long long* g_kt_dev = nullptr;
#endif

}  // namespace moe

using namespace moe;

extern "C" {

int moe_timing_enable(int max_launches) {
    if (max_launches < 0) return MOE_ERR_INVALID_ARG;
    free_all();
    for (int i = 0; i < max_launches; ++i) {
        Rec r{-1, nullptr, nullptr};
        if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) {
            cudaGetLastError();
            free_all();
            return MOE_ERR_CUDA;
        }
        g_recs.push_back(r);
    }
    return MOE_OK;
}

int moe_timing_collect(int32_t* kernel_ids, float* ms, int cap, int* n) {
    if (!kernel_ids || !ms || !n || cap < 0) return MOE_ERR_INVALID_ARG;
    int m = 0;
    for (int i = 0; i < g_used && m < cap; ++i) {
        float t = 0.f;
        if (cudaEventSynchronize(g_recs[i].b) != cudaSuccess ||
            cudaEventElapsedTime(&t, g_recs[i].a, g_recs[i].b) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        kernel_ids[m] = g_recs[i].kernel;
        ms[m] = t;
        ++m;
    }
    *n = m;
    g_used = 0;
    g_open = -1;
    return MOE_OK;
}

const char* moe_kernel_name(int kernel_id) {
    return (kernel_id >= 0 && kernel_id < K_NUM) ? kNames[kernel_id] : nullptr;
}

}  // extern "C"

#ifdef MOE_TRACE
// Diagnostics export of the trace build: dst == NULL allocates the stamp table
// on first use and resets it (minima to all ones, maxima to zero); otherwise
// it synchronises the device and copies the table ([K_NUM][16] u64, see
// kt_mark) to the host buffer dst of `bytes` bytes.
extern "C" int moe_ktrace(unsigned long long* dst, size_t bytes) {
    const size_t n = (size_t)K_NUM * KT_SLOTS;
    if (g_kt_dev == nullptr && cudaMalloc(&g_kt_dev, n * sizeof(unsigned long long)) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    if (dst == nullptr) {
        unsigned long long init[K_NUM * KT_SLOTS];
        for (size_t i = 0; i < n; ++i) init[i] = (i % 2 == 0) ? ~0ull : 0ull;
        return cudaMemcpy(g_kt_dev, init, sizeof(init), cudaMemcpyHostToDevice) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    if (bytes > n * sizeof(unsigned long long)) bytes = n * sizeof(unsigned long long);
    return cudaMemcpy(dst, g_kt_dev, bytes, cudaMemcpyDeviceToHost) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
#endif
