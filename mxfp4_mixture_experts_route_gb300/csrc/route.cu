// Router logits (fp32) and sigmoid top-k.
//
// vllm.models.muse_spark.amd.mono.kernels.k3, stage A (the router's logits in
// fp32), stage route (every token's top 8) and route_token (a sigmoid score per
// expert, over a wave's tokens); vllm.models.muse_spark.amd.mono.kernels.k5,
// stage HA (fp32 router, top 8 with one CTA per token, ids and weights handed
// to the next stage); vllm.models.kimi_k3.amd.specialized_decode.mono.layer,
// k2_launch (the router weight w_gate and an fp32 bias).
//
// GB300 design: the pages split the router's K over 8-CTA groups of a rank and
// all-gather the partial logits; on one GPU the logits are one [S, d] x [d, E]
// product.  It is split over CTAs by 8 experts x 32 tokens, and when that
// leaves SMs idle, over K as well: the K-ranges of one output tile run as one
// thread-block cluster and are added up in the cluster's shared memory in a
// fixed order.  One warp a token then does the selection (k3 repeats the
// routing in every CTA; here the ids are produced once and read by the sort).
#include "moe_internal.cuh"
#include "topk.cuh"

#include <cooperative_groups.h>

namespace cg = cooperative_groups;

namespace moe {

namespace {

constexpr int RT_EXPERTS = 8;    // experts per CTA (one per warp)
constexpr int RT_TOKENS = 32;    // token rows per CTA
constexpr int RT_KC = 256;       // K elements per round: 8 per lane
constexpr int RT_THREADS = 32 * RT_EXPERTS;
constexpr int RT_MAX_CLUSTER = 8;   // portable cluster size

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Router logits L[t][e] = x[t] . w_gate[e] (+ offset[e]), fp32 accumulation.
// grid (E/8, KS, ceil(S/32)) in clusters of (1, KS, 1): the KS CTAs of a
// cluster split K.  Warp w owns expert 8*bx + w; in each 256-K round lane l
// holds that expert's elements 8l..8l+7 in registers and reads the same 16
// bytes of every staged token row from shared memory (one 128-bit load a
// token, no bank conflict); the lanes' sums are reduced across the warp once,
// after the CTA's whole K-range.  The cluster's first CTA then adds the KS
// partial tiles (distributed shared memory, K-range order) and writes L.
__global__ void __launch_bounds__(RT_THREADS) k_router(const __nv_bfloat16* __restrict__ x,
                                                       const __nv_bfloat16* __restrict__ wg,
                                                       const float* __restrict__ off, float* __restrict__ L,
                                                       int S, int d, int E, int kslices) {
    __shared__ uint4 xs_[2][RT_TOKENS * (RT_KC / 8)];
    __shared__ float part[RT_TOKENS * RT_EXPERTS];
    KT_MARK(K_ROUTER, 0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * RT_EXPERTS + warp, ks = blockIdx.y, t0 = blockIdx.z * RT_TOKENS;
    const int nk = d / 128;                                  // 128-K units of a row
    const int k_begin = (int)((long long)nk * ks / kslices) * 128;
    const int k_end = (int)((long long)nk * (ks + 1) / kslices) * 128;
    const int nt = min(RT_TOKENS, S - t0);
    float acc[RT_TOKENS];
#pragma unroll
    for (int t = 0; t < RT_TOKENS; ++t) acc[t] = 0.f;
    // one 256-K round: the lane's 8 weights against every staged token row
    auto fma_round = [&](const uint4 w, const uint4* xr, int q16) {
        if (lane < q16) {
            const float w0 = bf_lo(w.x), w1 = bf_hi(w.x), w2 = bf_lo(w.y), w3 = bf_hi(w.y);
            const float w4 = bf_lo(w.z), w5 = bf_hi(w.z), w6 = bf_lo(w.w), w7 = bf_hi(w.w);
#pragma unroll
            for (int t = 0; t < RT_TOKENS; ++t) {
                if (t < nt) {
                    const uint4 v = xr[t * (RT_KC / 8) + lane];
                    float a = acc[t];
                    a = fmaf(bf_lo(v.x), w0, a);
                    a = fmaf(bf_hi(v.x), w1, a);
                    a = fmaf(bf_lo(v.y), w2, a);
                    a = fmaf(bf_hi(v.y), w3, a);
                    a = fmaf(bf_lo(v.z), w4, a);
                    a = fmaf(bf_hi(v.z), w5, a);
                    a = fmaf(bf_lo(v.w), w6, a);
                    a = fmaf(bf_hi(v.w), w7, a);
                    acc[t] = a;
                }
            }
        }
    };
    auto stage = [&](uint4* xr, int kc, int q16) {
        for (int i = threadIdx.x; i < nt * q16; i += RT_THREADS) {
            const int r = i / q16, c = i % q16;
            xr[r * (RT_KC / 8) + c] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + r) * d + kc) + c);
        }
    };
    if (k_end - k_begin <= 2 * RT_KC) {
        // a K range of at most two rounds: both weight slices in flight before
        // the wait, both rounds of token rows staged at once (one round trip)
        uint4 w[2];
        int q16[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int kc = k_begin + r * RT_KC;
            q16[r] = kc < k_end ? min(RT_KC, k_end - kc) / 8 : 0;
            w[r] = make_uint4(0, 0, 0, 0);
            if (e < E && lane < q16[r]) w[r] = __ldg(reinterpret_cast<const uint4*>(wg + (size_t)e * d + kc) + lane);
        }
        pdl_wait();      // x may come from the stream's last kernel
        pdl_trigger();   // the call's first kernel: successors start once the call's inputs are final
        KT_MARK(K_ROUTER, 1);
#pragma unroll
        for (int r = 0; r < 2; ++r)
            if (q16[r] > 0) stage(xs_[r], k_begin + r * RT_KC, q16[r]);
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 2; ++r) fma_round(w[r], xs_[r], q16[r]);
    } else {
        for (int kc = k_begin; kc < k_end; kc += RT_KC) {
            const int klen = min(RT_KC, k_end - kc);             // 256 or 128
            const int q16 = klen / 8;                            // 16-byte pieces of a row slice
            uint4 w = make_uint4(0, 0, 0, 0);
            if (e < E && lane < q16) w = __ldg(reinterpret_cast<const uint4*>(wg + (size_t)e * d + kc) + lane);
            if (kc == k_begin) {
                pdl_wait();      // the first weight slice is in flight; x may come from the stream's last kernel
                pdl_trigger();   // the call's first kernel: successors start once the call's inputs are final
                KT_MARK(K_ROUTER, 1);
            }
            __syncthreads();
            stage(xs_[0], kc, q16);
            __syncthreads();
            fma_round(w, xs_[0], q16);
        }
    }
#pragma unroll
    for (int t = 0; t < RT_TOKENS; ++t) {
        float a = acc[t];
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) a += __shfl_xor_sync(0xffffffffu, a, m);
        if (lane == 0) part[t * RT_EXPERTS + warp] = a;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (ks == 0) {
        // thread i: token i / 8, expert i % 8 of the tile
        const int t = threadIdx.x / RT_EXPERTS, ee = threadIdx.x % RT_EXPERTS;
        const int eg = blockIdx.x * RT_EXPERTS + ee;
        float pz[RT_MAX_CLUSTER];
#pragma unroll
        for (int r = 0; r < RT_MAX_CLUSTER; ++r)   // the remote loads, all in flight together
            pz[r] = r < kslices ? cluster.map_shared_rank(part, r)[t * RT_EXPERTS + ee] : 0.f;
        float z = 0.f;
#pragma unroll
        for (int r = 0; r < RT_MAX_CLUSTER; ++r) z += pz[r];   // K-range order
        if (t < nt && eg < E) L[(size_t)(t0 + t) * E + eg] = off ? z + off[eg] : z;
    }
    cluster.sync();   // every CTA keeps its shared memory until the first has read it
    KT_MARK(K_ROUTER, 2);
}

// The same logits for a few tokens (S <= NTOK) and at most NR 256-K rounds per
// CTA: a lane issues every load of its weight slice (before the wait on the
// previous kernel) and of the token rows at once, straight from global memory
// (the rows are shared by all CTAs through L2), with no shared-memory staging.
template <int NTOK, int NR>
__global__ void __launch_bounds__(RT_THREADS) k_router_few(const __nv_bfloat16* __restrict__ x,
                                                           const __nv_bfloat16* __restrict__ wg,
                                                           const float* __restrict__ off, float* __restrict__ L,
                                                           int S, int d, int E, int kslices) {
    __shared__ float part[NTOK * RT_EXPERTS];
    KT_MARK(K_ROUTER, 0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * RT_EXPERTS + warp, ks = blockIdx.y;
    const int nk = d / 128;
    const int k_begin = (int)((long long)nk * ks / kslices) * 128;
    const int k_end = (int)((long long)nk * (ks + 1) / kslices) * 128;
    uint4 w[NR];
    int q16[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const int kc = k_begin + RT_KC * r;
        q16[r] = kc < k_end ? min(RT_KC, k_end - kc) / 8 : 0;
        w[r] = make_uint4(0, 0, 0, 0);
        if (e < E && lane < q16[r]) w[r] = __ldg(reinterpret_cast<const uint4*>(wg + (size_t)e * d + kc) + lane);
    }
    pdl_wait();      // x may come from the stream's previous kernel
    pdl_trigger();   // the call's first kernel: successors start once the call's inputs are final
    KT_MARK(K_ROUTER, 1);
    uint4 xv[NR][NTOK];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int t = 0; t < NTOK; ++t) {
            xv[r][t] = make_uint4(0, 0, 0, 0);
            if (t < S && lane < q16[r])
                xv[r][t] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * d + k_begin + RT_KC * r) + lane);
        }
    float acc[NTOK];
#pragma unroll
    for (int t = 0; t < NTOK; ++t) {
        float a = 0.f;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const uint4 v = xv[r][t], ww = w[r];
            a = fmaf(bf_lo(v.x), bf_lo(ww.x), a);
            a = fmaf(bf_hi(v.x), bf_hi(ww.x), a);
            a = fmaf(bf_lo(v.y), bf_lo(ww.y), a);
            a = fmaf(bf_hi(v.y), bf_hi(ww.y), a);
            a = fmaf(bf_lo(v.z), bf_lo(ww.z), a);
            a = fmaf(bf_hi(v.z), bf_hi(ww.z), a);
            a = fmaf(bf_lo(v.w), bf_lo(ww.w), a);
            a = fmaf(bf_hi(v.w), bf_hi(ww.w), a);
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) a += __shfl_xor_sync(0xffffffffu, a, m);
        acc[t] = a;
    }
    KT_MARK(K_ROUTER, 3);
    if (lane == 0) {
#pragma unroll
        for (int t = 0; t < NTOK; ++t) part[t * RT_EXPERTS + warp] = acc[t];
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    KT_MARK(K_ROUTER, 4);
    if (ks == 0 && threadIdx.x < NTOK * RT_EXPERTS) {
        const int t = threadIdx.x / RT_EXPERTS, ee = threadIdx.x % RT_EXPERTS;
        const int eg = blockIdx.x * RT_EXPERTS + ee;
        float pz[RT_MAX_CLUSTER];
#pragma unroll
        for (int r = 0; r < RT_MAX_CLUSTER; ++r)
            pz[r] = r < kslices ? cluster.map_shared_rank(part, r)[t * RT_EXPERTS + ee] : 0.f;
        float z = 0.f;
#pragma unroll
        for (int r = 0; r < RT_MAX_CLUSTER; ++r) z += pz[r];
        if (t < S && eg < E) L[(size_t)t * E + eg] = off ? z + off[eg] : z;
    }
    cluster.sync();
    KT_MARK(K_ROUTER, 2);
}

// One warp per token (see topk_select).
template <int MAXE>
__device__ __forceinline__ void topk_rows(const float* L, const float* __restrict__ bias, int S, int E, int k,
                                          int32_t* __restrict__ ids, float* __restrict__ wout, float* s_sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    float b[MAXE];
    load_bias(bias, E, lane, b);   // an input of the call: read before the wait
    pdl_wait();
    KT_MARK(K_TOPK, 1);
    if (t < S) {
        int id, rank;
        float w;
        float z[MAXE];
        topk_load(L + (size_t)t * E, E, lane, z);
        topk_select(z, b, E, k, lane, s_sh + warp * 32 * MAXE, id, w, rank);
        if (lane < k) {
            ids[(size_t)t * k + rank] = id;
            wout[(size_t)t * k + rank] = w;
        }
    }
}

constexpr int TOPK_WARPS = 8;
__global__ void __launch_bounds__(32 * TOPK_WARPS) k_topk(const float* L, const float* __restrict__ bias,
                                                          int S, int E, int k, int32_t* __restrict__ ids,
                                                          float* __restrict__ wout) {
    __shared__ float s_sh[TOPK_WARPS * 512];
    KT_MARK(K_TOPK, 0);
    pdl_trigger();
    if (E <= 256) topk_rows<256 / 32>(L, bias, S, E, k, ids, wout, s_sh);
    else topk_rows<512 / 32>(L, bias, S, E, k, ids, wout, s_sh);
    KT_MARK(K_TOPK, 2);
}

}  // namespace

int router_kslices(const moe_shape& s, int num_sms) {
    const int blocks = (s.E + RT_EXPERTS - 1) / RT_EXPERTS * ((s.S + RT_TOKENS - 1) / RT_TOKENS);
    int ks = (2 * num_sms + blocks - 1) / blocks;     // about two CTAs per SM
    const int nk = s.d / 128;
    if (ks > nk) ks = nk;
    if (ks > RT_MAX_CLUSTER) ks = RT_MAX_CLUSTER;
    if (ks < 1) ks = 1;
    return ks;
}

cudaError_t launch_router_logits(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    KT_BIND();
    if (router_tc_fits(s)) {
        timing_begin(K_ROUTER, st);
        const cudaError_t e = launch_router_tc(s, L, p, st);
        timing_end(st);
        return e;
    }
    float* logits = reinterpret_cast<float*>(p.ws + L.logits);
    const int ks = L.router_kslices;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((s.E + RT_EXPERTS - 1) / RT_EXPERTS, ks, (s.S + RT_TOKENS - 1) / RT_TOKENS);
    cfg.blockDim = dim3(RT_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = ks;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    // few tokens and at most two 256-K rounds per CTA: the variant without staging
    const int nk = s.d / 128;
    const bool few = s.S <= 8 && (nk + ks - 1) / ks <= 2 * (RT_KC / 128);
    if (few) cfg.gridDim = dim3((s.E + RT_EXPERTS - 1) / RT_EXPERTS, ks, 1);
    timing_begin(K_ROUTER, st);
    cudaError_t e = few ? cudaLaunchKernelEx(&cfg, k_router_few<8, 2>, p.x, p.w_gate, p.logit_off, logits, s.S, s.d,
                                             s.E, ks)
                        : cudaLaunchKernelEx(&cfg, k_router, p.x, p.w_gate, p.logit_off, logits, s.S, s.d, s.E, ks);
    timing_end(st);
    return e;
}

cudaError_t launch_topk(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    KT_BIND();
    timing_begin(K_TOPK, st);
    const cudaError_t e =
        launch_pdl(k_topk, dim3((s.S + TOPK_WARPS - 1) / TOPK_WARPS), dim3(32 * TOPK_WARPS), 0, st,
                   reinterpret_cast<const float*>(p.ws + L.logits), p.bias, s.S, s.E, s.k, p.ids, p.weights);
    timing_end(st);
    return e;
}

cudaError_t launch_route(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    cudaError_t e = launch_router_logits(s, L, p, st);
    if (e != cudaSuccess) return e;
    return launch_topk(s, L, p, st);
}

}  // namespace moe
