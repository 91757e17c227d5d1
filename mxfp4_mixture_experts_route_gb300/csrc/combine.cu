// Per-pick post-expert norm and weighted combine.
//
// vllm.models.muse_spark.amd.mono.kernels.k3, stage E (a norm of each pick's
// expert output, then the weighted sum).  On one GPU with every expert resident there is no
// EP partial to reduce-scatter: the weighted sum over a token's k picks is the
// block's output, out[t] = sum_j w_j * [RMSNorm](y_{t,j}), summed in pick
// order j (ascending expert id for ids from moe_route).
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int CB_THREADS = 256;
constexpr int CB_COLS = 4 * CB_THREADS;   // columns of out per CTA
constexpr int CB_MAXK = 16;               // picks per token (k <= 16)

// grid (S, ceil(d / 1024)): CTA (t, c) writes out[t, 1024c .. 1024c+1023] =
// sum_j coef_j * y[pos(t, j), cols] (* norm_w[cols]), with coef_j = w_j, or
// for the post-expert norm w_j * rsqrt(mean(y_j^2) + eps).  y_j's sum of
// squares comes from the per-128-row-block sums the down GEMM's epilogue
// writes: warp w adds up the blocks of picks w and w + 8 (lanes over blocks,
// then a fixed shuffle tree), so the CTA never reads a whole y row twice.
// y rows are addressed through pos[t*k + j] (the sorted per-pick buffer).
// ids_out / w_out (host buffers of moe_forward_host, each or both null): the
// CTAs of column block 0 also copy the token's ids and routing weights there from
// the workspace, so that those writes over the CPU-GPU link go out with the
// block's last kernel instead of holding up the routing kernel's completion.
// At most 32 registers a thread (eight CTAs an SM's worth): a combine CTA
// starts beside an expert CTA (programmatic dependent launch) only if it fits
// in what that CTA leaves of each SM sub-partition's register file, 2048
// registers where four of the expert CTA's warps sit (4 x 32 x 112 of 16384),
// i.e. two warps of 32 registers a thread.
__global__ void __launch_bounds__(CB_THREADS, 8) k_combine(const float* y, const float* ssq, const int32_t* pos, const float* w,
                                                        const float* __restrict__ norm_w, float eps, int k, int d,
                                                        float* __restrict__ out, const int32_t* ids,
                                                        int32_t* __restrict__ ids_out, float* __restrict__ w_out) {
    KT_MARK(K_COMBINE, 0);
    pdl_trigger();
    pdl_wait();
    KT_MARK(K_COMBINE, 1);
    const int t = blockIdx.x;
    __shared__ float coef[CB_MAXK];
    __shared__ int32_t prow[CB_MAXK];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#pragma unroll
    for (int h = 0; h < CB_MAXK / 8; ++h) {
        const int j = warp + 8 * h;
        if (j < k) {
            const int p = ld_dep(pos + (size_t)t * k + j);
            float c = ld_dep(w + (size_t)t * k + j);
            if (blockIdx.y == 0 && lane == 0) {   // either may be null
                if (ids_out != nullptr) ids_out[(size_t)t * k + j] = ld_dep(ids + (size_t)t * k + j);
                if (w_out != nullptr) w_out[(size_t)t * k + j] = c;
            }
            if (norm_w != nullptr && p >= 0) {
                const int nb = d / 128;                // <= 128 row blocks
                float q = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int b = lane + 32 * i;
                    if (b < nb) q += ld_dep(ssq + (size_t)p * nb + b);
                }
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) q += __shfl_xor_sync(0xffffffffu, q, m);
                c *= rsqrtf(q / (float)d + eps);
            }
            if (lane == 0) {
                coef[j] = p >= 0 ? c : 0.f;
                prow[j] = p;
            }
        }
    }
    __syncthreads();
    const int col = blockIdx.y * CB_COLS + 4 * tid;
    if (col >= d) {
        KT_MARK(K_COMBINE, 2);
        return;
    }
    float4 v[CB_MAXK];
#pragma unroll
    for (int j = 0; j < CB_MAXK; ++j) {           // every pick's load in flight at once
        v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < k && prow[j] >= 0) v[j] = ld_dep(reinterpret_cast<const float4*>(y + (size_t)prow[j] * d + col));
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < CB_MAXK; ++j) {           // summed in pick order j
        if (j < k) {
            const float c = coef[j];
            acc.x = fmaf(c, v[j].x, acc.x);
            acc.y = fmaf(c, v[j].y, acc.y);
            acc.z = fmaf(c, v[j].z, acc.z);
            acc.w = fmaf(c, v[j].w, acc.w);
        }
    }
    if (norm_w != nullptr) {
        const float4 nw = *reinterpret_cast<const float4*>(norm_w + col);
        acc.x *= nw.x;
        acc.y *= nw.y;
        acc.z *= nw.z;
        acc.w *= nw.w;
    }
    *reinterpret_cast<float4*>(out + (size_t)t * d + col) = acc;
    KT_MARK(K_COMBINE, 2);
}

}  // namespace

// ids_out / w_out: see k_combine (both null: the plain combine)
cudaError_t launch_combine_host(const moe_shape& s, const WsLayout& L, const Ptrs& p, int32_t* ids_out, float* w_out,
                                cudaStream_t st) {
    KT_BIND();
    timing_begin(K_COMBINE, st);
    const dim3 grid(s.S, (s.d + CB_COLS - 1) / CB_COLS);
    const cudaError_t e =
        launch_pdl(k_combine, grid, dim3(CB_THREADS), 0, st, reinterpret_cast<const float*>(p.ws + L.y),
                   reinterpret_cast<const float*>(p.ws + L.ssq), reinterpret_cast<const int32_t*>(p.ws + L.pos),
                   (const float*)p.weights, p.norm_w, s.norm_eps, s.k, s.d, p.out, (const int32_t*)p.ids, ids_out,
                   w_out);
    timing_end(st);
    return e;
}

cudaError_t launch_combine(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    return launch_combine_host(s, L, p, nullptr, nullptr, st);
}

}  // namespace moe
