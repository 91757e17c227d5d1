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
// product, split over CTAs by 16 experts x K-ranges x 128 tokens so that about
// two CTAs per SM take part, with fp32 partials per K-range; one warp a token
// then sums the partials in a fixed order and does the selection (the k3
// "every CTA routes every token" redundancy is not needed: the ids are
// produced once).
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int RT_EXPERTS = 16;   // experts per CTA (two per warp)
constexpr int RT_TOKENS = 128;   // token rows per CTA (four per lane)
constexpr int RT_KC = 128;       // K elements staged per round
constexpr int RT_THREADS = 256;
constexpr int XS = RT_KC / 2 + 1;   // padded row stride of the staged tiles, in 32-bit words

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Partial router logits: Lp[ks][t][e] = sum over K-range ks of x[t, c] * w_gate[e, c]
// (fp32).  grid (E/16, KS, ceil(S/128)); the CTA stages 128-K slices of its 16
// weight rows and 128 token rows in shared memory (rows padded by one word so
// the 32 lanes, one token each, hit 32 banks) and accumulates over its K-range.
// Warp w owns experts 2w, 2w+1 of the block; lane l owns tokens l, l+32, l+64,
// l+96 of the tile.
__global__ void __launch_bounds__(RT_THREADS) k_router_partial(const __nv_bfloat16* __restrict__ x,
                                                               const __nv_bfloat16* __restrict__ wg,
                                                               float* __restrict__ Lp, int S, int d, int E,
                                                               int kslices) {
    __shared__ uint32_t ws_[RT_EXPERTS * XS];
    __shared__ uint32_t xs_[RT_TOKENS * XS];
    const int e0 = blockIdx.x * RT_EXPERTS, ks = blockIdx.y, t0 = blockIdx.z * RT_TOKENS;
    const int nk = d / 128;                                  // 128-K units of a row
    const int k_begin = (int)((long long)nk * ks / kslices) * 128;
    const int k_end = (int)((long long)nk * (ks + 1) / kslices) * 128;
    const int nt = min(RT_TOKENS, S - t0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float acc[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int kc = k_begin; kc < k_end; kc += RT_KC) {
        const int klen = min(RT_KC, k_end - kc);             // multiple of 128
        const int q16 = klen / 8;                            // 16-byte pieces of a row slice
        __syncthreads();
        for (int i = threadIdx.x; i < RT_EXPERTS * q16; i += RT_THREADS) {
            const int r = i / q16, c = i % q16;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (e0 + r < E) v = __ldg(reinterpret_cast<const uint4*>(wg + (size_t)(e0 + r) * d + kc) + c);
            uint32_t* dst = ws_ + r * XS + 4 * c;
            dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
        }
        for (int i = threadIdx.x; i < nt * q16; i += RT_THREADS) {
            const int r = i / q16, c = i % q16;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + r) * d + kc) + c);
            uint32_t* dst = xs_ + r * XS + 4 * c;
            dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
        }
        __syncthreads();
        const uint32_t* w0 = ws_ + (2 * warp) * XS;
        const uint32_t* w1 = w0 + XS;
        for (int kk = 0; kk < klen / 2; ++kk) {
            const uint32_t a0 = w0[kk], a1 = w1[kk];
            const float a0l = bf_lo(a0), a0h = bf_hi(a0), a1l = bf_lo(a1), a1h = bf_hi(a1);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = lane + 32 * j;
                if (t < nt) {
                    const uint32_t b = xs_[t * XS + kk];
                    const float bl = bf_lo(b), bh = bf_hi(b);
                    acc[0][j] = fmaf(bl, a0l, fmaf(bh, a0h, acc[0][j]));
                    acc[1][j] = fmaf(bl, a1l, fmaf(bh, a1h, acc[1][j]));
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int t = lane + 32 * j;
        if (t < nt) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int e = e0 + 2 * warp + i;
                if (e < E) Lp[((size_t)ks * S + t0 + t) * E + e] = acc[i][j];
            }
        }
    }
}

// One warp per token: L = sum of the K-range partials (fixed order) + offset;
// s = sigmoid(L), sel = s + bias, k rounds of a warp argmax (ties -> lower
// expert id), then the picks in ascending id with w_j = s_j / sum s.  Lane l
// holds experts l, l+32, ... (E <= 512).
__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ Lp, int kslices,
                                              const float* __restrict__ off, const float* __restrict__ bias,
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
            float z = 0.f;
            for (int ks = 0; ks < kslices; ++ks) z += Lp[((size_t)ks * S + t) * E + e];
            if (off) z += off[e];
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

int router_kslices(const moe_shape& s, int num_sms) {
    const int blocks = (s.E + RT_EXPERTS - 1) / RT_EXPERTS * ((s.S + RT_TOKENS - 1) / RT_TOKENS);
    int ks = (2 * num_sms + blocks - 1) / blocks;     // about two CTAs per SM
    const int nk = s.d / 128;
    if (ks > nk) ks = nk;
    if (ks < 1) ks = 1;
    return ks;
}

cudaError_t launch_route(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    float* Lp = reinterpret_cast<float*>(p.ws + L.logits);
    const int ks = L.router_kslices;
    dim3 g1((s.E + RT_EXPERTS - 1) / RT_EXPERTS, ks, (s.S + RT_TOKENS - 1) / RT_TOKENS);
    timing_begin(K_ROUTER, st);
    k_router_partial<<<g1, RT_THREADS, 0, st>>>(p.x, p.w_gate, Lp, s.S, s.d, s.E, ks);
    timing_end(st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int warps_per_block = 8;
    timing_begin(K_TOPK, st);
    k_topk<<<(s.S + warps_per_block - 1) / warps_per_block, 32 * warps_per_block, 0, st>>>(
        Lp, ks, p.logit_off, p.bias, s.S, s.E, s.k, p.ids, p.weights);
    timing_end(st);
    return cudaGetLastError();
}

}  // namespace moe
