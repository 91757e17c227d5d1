// The elementwise steps of the latent-MoE layer around the routed block.
//
// vllm.models.kimi_k3.amd.specialized_decode.mono.layer, K2b's stage list:
// the latent parts project the layer input to the experts' latent width, the
// routed experts run there, "lnorm" normalises their combined output with
// ln_w and "up" projects it back; the shared expert's gate/up, its activation
// and its down projection run beside them.  The dense products are the
// tensor-core kernel of route_tc.cu; here are the two steps between them:
//   - the latent norm: zl = RMSNorm(yl) * ln_w, rounded to bf16 for the up
//     projection's bf16 operand;
//   - the shared expert's activation: hs = silu(g) * u, rounded to bf16 for
//     the shared down projection.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int LN_THREADS = 256;

// grid (S): zl[t, :] = bf16(yl[t, :] * rsqrt(mean(yl[t, :]^2) + eps) * ln_w).
// The sum of squares: each thread over columns tid, tid + 256, ..., then a
// fixed tree (warp shuffles, then the eight warp sums in order).
__global__ void __launch_bounds__(LN_THREADS) k_latent_norm(const float* yl, const float* __restrict__ ln_w,
                                                             float eps, int n, __nv_bfloat16* __restrict__ zl) {
    pdl_trigger();
    __shared__ float wsum[LN_THREADS / 32];
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    const float* row = yl + (size_t)t * n;
    float q = 0.f;
    for (int c = tid; c < n; c += LN_THREADS) {
        const float v = ld_dep(row + c);
        q = fmaf(v, v, q);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) q += __shfl_xor_sync(0xffffffffu, q, m);
    if (lane == 0) wsum[warp] = q;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < LN_THREADS / 32; ++w) tot += wsum[w];
    const float r = rsqrtf(tot / (float)n + eps);
    for (int c = tid; c < n; c += LN_THREADS)
        zl[(size_t)t * n + c] = __float2bfloat16_rn(ld_dep(row + c) * r * ln_w[c]);
}

// grid (S, ceil(SI / 256)): hs[t, i] = bf16(silu(g) * u), g = gu[t, i],
// u = gu[t, SI + i] (gate rows first, then up rows, as in w_sgu).
__global__ void __launch_bounds__(256) k_shared_act(const float* gu, int si, __nv_bfloat16* __restrict__ hs) {
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x, i = blockIdx.y * 256 + threadIdx.x;
    if (i >= si) return;
    const float g = ld_dep(gu + (size_t)t * 2 * si + i), u = ld_dep(gu + (size_t)t * 2 * si + si + i);
    hs[(size_t)t * si + i] = __float2bfloat16_rn(g / (1.0f + __expf(-g)) * u);
}

}  // namespace

cudaError_t launch_latent_norm(const float* yl, const float* ln_w, float eps, int S, int n, __nv_bfloat16* zl,
                               cudaStream_t st) {
    return launch_pdl(k_latent_norm, dim3(S), dim3(LN_THREADS), 0, st, yl, ln_w, eps, n, zl);
}

cudaError_t launch_shared_act(const float* gu, int S, int si, __nv_bfloat16* hs, cudaStream_t st) {
    return launch_pdl(k_shared_act, dim3(S, (si + 255) / 256), dim3(256), 0, st, gu, si, hs);
}

}  // namespace moe
