// Per-pick post-expert norm and weighted combine.
//
// vllm.models.muse_spark.amd.mono.kernels.k3, stage E: "per-pick post-expert
// norm and weighted sum".  On one GPU with every expert resident there is no
// EP partial to reduce-scatter: the weighted sum over a token's k picks is the
// block's output, out[t] = sum_j w_j * [RMSNorm](y_{t,j}), summed in pick
// order j (ascending expert id for ids from moe_route).
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int CB_THREADS = 256;

// one CTA per token; y rows of the token's picks are read from the sorted
// per-pick buffer through pos[t*k + j]
__global__ void __launch_bounds__(CB_THREADS) k_combine(const float* __restrict__ y,
                                                        const int32_t* __restrict__ pos,
                                                        const float* __restrict__ w, const float* __restrict__ norm_w,
                                                        float eps, int k, int d, float* __restrict__ out) {
    const int t = blockIdx.x;
    __shared__ float coef[16];
    __shared__ int32_t prow[16];
    __shared__ float red[CB_THREADS / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int j = 0; j < k; ++j) {
        const int p = pos[(size_t)t * k + j];
        float c = (p >= 0) ? w[(size_t)t * k + j] : 0.f;
        if (norm_w != nullptr && p >= 0) {
            const float4* yr = reinterpret_cast<const float4*>(y + (size_t)p * d);
            float ss = 0.f;
            for (int i = tid; i < d / 4; i += CB_THREADS) {
                const float4 v = yr[i];
                ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
            }
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
            if (lane == 0) red[warp] = ss;
            __syncthreads();
            if (tid == 0) {
                float tot = 0.f;
                for (int i = 0; i < CB_THREADS / 32; ++i) tot += red[i];
                coef[j] = c * rsqrtf(tot / (float)d + eps);
            }
            __syncthreads();
        } else if (tid == 0) {
            coef[j] = c;
        }
        if (tid == 0) prow[j] = p;
    }
    __syncthreads();
    for (int i = tid; i < d / 4; i += CB_THREADS) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const int p = prow[j];
            if (p < 0) continue;
            const float4 v = reinterpret_cast<const float4*>(y + (size_t)p * d)[i];
            const float c = coef[j];
            acc.x = fmaf(c, v.x, acc.x);
            acc.y = fmaf(c, v.y, acc.y);
            acc.z = fmaf(c, v.z, acc.z);
            acc.w = fmaf(c, v.w, acc.w);
        }
        if (norm_w != nullptr) {
            const float4 nw = reinterpret_cast<const float4*>(norm_w)[i];
            acc.x *= nw.x;
            acc.y *= nw.y;
            acc.z *= nw.z;
            acc.w *= nw.w;
        }
        reinterpret_cast<float4*>(out + (size_t)t * d)[i] = acc;
    }
}

}  // namespace

cudaError_t launch_combine(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    timing_begin(K_COMBINE, st);
    k_combine<<<s.S, CB_THREADS, 0, st>>>(reinterpret_cast<const float*>(p.ws + L.y),
                                          reinterpret_cast<const int32_t*>(p.ws + L.pos), p.weights, p.norm_w,
                                          s.norm_eps, s.k, s.d, p.out);
    timing_end(st);
    return cudaGetLastError();
}

}  // namespace moe
