// Router logits (fp32) and sigmoid top-k.
//
// vllm.models.muse_spark.amd.mono.kernels.k3, stage A: "router logits (fp32)";
// stage route: every token's top-8; route_token: "sigmoid + ..." over a wave's
// tokens.  vllm.models.muse_spark.amd.mono.kernels.k5, HA: "router (fp32) ...
// top-8 (CTA t routes token t) ... top-k ids / weights".
// vllm.models.kimi_k3.amd.specialized_decode.mono.layer, k2_launch: w_gate and
// an fp32 bias.
//
// GB300 design: the pages split the router's K over 8-CTA groups of a rank and
// all-gather the partial logits; on one GPU the logits are one [S, d] x [d, E]
// product, split over CTAs by (8 experts) x (16 tokens) so every SM takes part,
// then one warp a token does the selection (the k3 "every CTA routes every
// token" redundancy is not needed: the ids are produced once).
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int RT_EXPERTS = 8;    // experts per CTA (one warp each)
constexpr int RT_TOKENS = 16;    // tokens per CTA

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// L[t, e] = sum_c x[t, c] * w_gate[e, c] in fp32 (+ logit_off[e]).
// grid (ceil(E/8), ceil(S/16)), 256 threads: warp w <-> expert 8*bx + w; each
// lane covers K-columns 8*lane + 256*i; partials are summed by a butterfly.
__global__ void __launch_bounds__(256) k_router_logits(const __nv_bfloat16* __restrict__ x,
                                                       const __nv_bfloat16* __restrict__ wg,
                                                       const float* __restrict__ off,
                                                       float* __restrict__ L, int S, int d, int E) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * RT_EXPERTS + warp;
    const int t0 = blockIdx.y * RT_TOKENS;
    if (e >= E) return;
    const int nt = min(RT_TOKENS, S - t0);
    float acc[RT_TOKENS];
#pragma unroll
    for (int j = 0; j < RT_TOKENS; ++j) acc[j] = 0.f;
    const uint4* wrow = reinterpret_cast<const uint4*>(wg + (size_t)e * d);
    const int nc = d >> 3;  // 16-byte chunks of a row
    for (int c = lane; c < nc; c += 32) {
        float wf[8];
        bf16x8_to_f32(__ldg(wrow + c), wf);
#pragma unroll
        for (int j = 0; j < RT_TOKENS; ++j) {
            if (j < nt) {
                float xf[8];
                bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + j) * d) + c), xf);
                float a = acc[j];
#pragma unroll
                for (int q = 0; q < 8; ++q) a = fmaf(xf[q], wf[q], a);
                acc[j] = a;
            }
        }
    }
    const float o = off ? off[e] : 0.f;
#pragma unroll
    for (int j = 0; j < RT_TOKENS; ++j) {
        float a = acc[j];
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) a += __shfl_xor_sync(0xffffffffu, a, m);
        if (lane == 0 && j < nt) L[(size_t)(t0 + j) * E + e] = a + o;
    }
}

// One warp per token: s = sigmoid(L), sel = s + bias, k rounds of a warp
// argmax (ties -> lower expert id), then the picks in ascending id with
// w_j = s_j / sum s.  Lane l holds experts l, l+32, ... (E <= 512).
__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ L, const float* __restrict__ bias,
                                              int S, int E, int k, int32_t* __restrict__ ids,
                                              float* __restrict__ wout) {
    const int lane = threadIdx.x & 31;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= S) return;
    constexpr int MAXE = 512 / 32;
    float s[MAXE], sel[MAXE];
#pragma unroll
    for (int i = 0; i < MAXE; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            const float z = L[(size_t)t * E + e];
            s[i] = 1.0f / (1.0f + expf(-z));
            const float v = s[i] + bias[e];
            sel[i] = (v == v) ? v : -INFINITY;
        } else {
            s[i] = 0.f;
            sel[i] = -INFINITY;
        }
    }
    int my_id = 0x7fffffff;   // lane j < k keeps pick j
    float my_s = 0.f;
    for (int r = 0; r < k; ++r) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < MAXE; ++i) {
            const int e = lane + 32 * i;
            if (e < E && (sel[i] > bv || (sel[i] == bv && e < bi))) { bv = sel[i]; bi = e; }
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, m);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, m);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        // the owner lane retires the winner and broadcasts its unbiased score
        const int owner = bi & 31, slot = bi >> 5;
        float sv = 0.f;
#pragma unroll
        for (int i = 0; i < MAXE; ++i)
            if (lane == owner && i == slot) { sv = s[i]; sel[i] = -INFINITY; }
        sv = __shfl_sync(0xffffffffu, sv, owner);
        if (lane == r) { my_id = bi; my_s = sv; }
    }
    // ascending id order: rank of my pick among the k picks
    float tot = 0.f;
    int rank = 0;
    for (int j = 0; j < k; ++j) {
        const int oid = __shfl_sync(0xffffffffu, my_id, j);
        tot += __shfl_sync(0xffffffffu, my_s, j);
        rank += (oid < my_id) ? 1 : 0;
    }
    if (lane < k) {
        ids[(size_t)t * k + rank] = my_id;
        wout[(size_t)t * k + rank] = my_s / tot;
    }
}

}  // namespace

cudaError_t launch_route(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    float* logits = reinterpret_cast<float*>(p.ws + L.logits);
    dim3 g1((s.E + RT_EXPERTS - 1) / RT_EXPERTS, (s.S + RT_TOKENS - 1) / RT_TOKENS);
    timing_begin(K_ROUTER, st);
    k_router_logits<<<g1, 256, 0, st>>>(p.x, p.w_gate, p.logit_off, logits, s.S, s.d, s.E);
    timing_end(st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int warps_per_block = 8;
    timing_begin(K_TOPK, st);
    k_topk<<<(s.S + warps_per_block - 1) / warps_per_block, 32 * warps_per_block, 0, st>>>(
        logits, p.bias, s.S, s.E, s.k, p.ids, p.weights);
    timing_end(st);
    return cudaGetLastError();
}

}  // namespace moe
