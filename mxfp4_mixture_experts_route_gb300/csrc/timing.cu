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

const char* const kNames[K_NUM] = {"router_logits", "topk", "sort", "gather", "experts", "combine", "topk_sort",
                                   "latent_down", "latent_norm", "latent_up", "shared_gate_up", "shared_act",
                                   "shared_down"};

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
