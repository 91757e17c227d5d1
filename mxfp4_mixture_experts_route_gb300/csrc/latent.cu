// The elementwise steps of the latent-MoE layer around the routed block, in
// one kernel.
//
// vllm.models.kimi_k3.amd.specialized_decode.mono.layer, K2b's stage list:
// the latent parts project the layer input to the experts' latent width, the
// routed experts run there, "lnorm" normalises their combined output with
// ln_w and "up" projects it back; the shared expert's gate/up, its activation
// and its down projection run beside them.  The dense products are the
// tensor-core kernel of route_tc.cu; here are the two steps between them
// (both read what the products before them wrote, both feed the products
// after them):
//   - the latent norm: zl = RMSNorm(yl) * ln_w, rounded to bf16 for the up
//     projection's bf16 operand;
//   - the shared expert's activation: hs = silu(g) * u, rounded to bf16 for
//     the shared down projection.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int MID_THREADS = 1024;
constexpr int MID_VEC = 4;   // float4 vectors a thread holds: rows of up to 16384 elements

// The steps between the dense products, one CTA a token t and step:
// blockIdx.y == 0, the latent norm: zl[t, :] = bf16(yl[t, :] * rsqrt(mean(
// yl[t, :]^2) + eps) * ln_w), the row held in registers (every load in flight
// at once), its sum of squares in a fixed order (each thread's vectors, warp
// shuffles, the warp sums in warp order); blockIdx.y == 1 (when si > 0), the
// shared expert's activation: hs[t, i] = bf16(silu(g) * u), g = gu[t, i],
// u = gu[t, si + i] (gate rows first, then up rows, as in w_sgu).
__global__ void __launch_bounds__(MID_THREADS) k_latent_mid(const float* yl, const float* __restrict__ ln_w, float eps,
                                                           int n, __nv_bfloat16* __restrict__ zl, const float* gu,
                                                           int si, __nv_bfloat16* __restrict__ hs) {
    KT_MARK(K_LATENT_MID, 0);
    pdl_trigger();
    __shared__ float wsum[MID_THREADS / 32];
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    KT_MARK(K_LATENT_MID, 1);
    if (blockIdx.y == 1) {
        const float* g = gu + (size_t)t * 2 * si;
        for (int i = tid; i < si; i += MID_THREADS) {
            const float gv = ld_dep(g + i), uv = ld_dep(g + si + i);
            hs[(size_t)t * si + i] = __float2bfloat16_rn(gv / (1.0f + __expf(-gv)) * uv);
        }
        return;
    }
    const float4* row = reinterpret_cast<const float4*>(yl + (size_t)t * n);
    const int nv = n / 4;
    float4 v[MID_VEC];
#pragma unroll
    for (int j = 0; j < MID_VEC; ++j) {
        const int c = tid + j * MID_THREADS;
        v[j] = c < nv ? ld_dep(row + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float q = 0.f;
#pragma unroll
    for (int j = 0; j < MID_VEC; ++j) {
        q = fmaf(v[j].x, v[j].x, q);
        q = fmaf(v[j].y, v[j].y, q);
        q = fmaf(v[j].z, v[j].z, q);
        q = fmaf(v[j].w, v[j].w, q);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) q += __shfl_xor_sync(0xffffffffu, q, m);
    if (lane == 0) wsum[warp] = q;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < MID_THREADS / 32; ++w) tot += wsum[w];
    const float r = rsqrtf(tot / (float)n + eps);
    const float4* lw = reinterpret_cast<const float4*>(ln_w);
#pragma unroll
    for (int j = 0; j < MID_VEC; ++j) {
        const int c = tid + j * MID_THREADS;
        if (c < nv) {
            const float4 w4 = lw[c];
            __nv_bfloat162 lo = __floats2bfloat162_rn(v[j].x * r * w4.x, v[j].y * r * w4.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(v[j].z * r * w4.z, v[j].w * r * w4.w);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(zl + (size_t)t * n + 4 * c) = pk;
        }
    }
    KT_MARK(K_LATENT_MID, 2);
}

}  // namespace

bool latent_mid_fits(int n) { return n % 4 == 0 && n <= 4 * MID_VEC * MID_THREADS; }

cudaError_t launch_latent_mid(const float* yl, const float* ln_w, float eps, int S, int n, __nv_bfloat16* zl,
                              const float* gu, int si, __nv_bfloat16* hs, cudaStream_t st) {
    KT_BIND();
    return launch_pdl(k_latent_mid, dim3(S, si > 0 ? 2 : 1), dim3(MID_THREADS), 0, st, yl, ln_w, eps, n, zl, gu, si,
                      hs);
}

}  // namespace moe
