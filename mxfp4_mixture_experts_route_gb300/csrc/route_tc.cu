// Dense bf16 products on the tensor cores: the router's logits for batches of
// 9 to 32 and of 64 tokens and more, and the latent-MoE layer's dense projections (latent
// down and up, the shared expert), at any batch.
//
// vllm.models.muse_spark.amd.mono.kernels.k3, stage A (the router's logits in
// fp32); the pages split the router's K over 8-CTA groups.  At larger batches the
// logits are a dense [E, d] x [d, S] product, so here they are one: M = 128
// experts x N = 128 tokens per tile, tcgen05.mma kind::f16 (bf16 x bf16, fp32
// accumulate in TMEM; each product is exact in fp32), both operands by TMA in
// 128-byte swizzled 64-element slabs through a six-stage ring.  When there are
// fewer tiles than SMs, K is split over a thread-block cluster and the
// cluster's fp32 partial tiles are added in a fixed order through distributed
// shared memory.
//
// Warps: 0 TMA producer, 1 MMA issuer (and TMEM owner), 2-5 epilogue (TMEM ->
// shared-memory partial tile), then all warps take part in the cluster sum.
#include "moe_internal.cuh"
#include "tc_ptx.cuh"

#include <cooperative_groups.h>
#include <cudaTypedefs.h>
#include <climits>

namespace cg = cooperative_groups;

namespace moe {

namespace {

constexpr int RM = 128;                    // weight rows per tile (MMA M)
constexpr int RK = 64;                     // K elements per stage (one 128-byte slab)
constexpr int R_A = RM * RK * 2;           // 16 KB of weights a stage
constexpr int R_THREADS = 192;
constexpr int R_MAX_CLUSTER = 8;
constexpr uint64_t R_WAIT_NS = 2000000000ull;

// RN: token rows a tile (the MMA N): 128 for batches, 16 for a few tokens,
// where a 2 KB token slab a stage leaves room for twice the weight stages
// (the weight stream is the cost of a small-batch product).
template <int RN>
struct DCfg {
    static constexpr int R_B = RN * RK * 2;
    static constexpr int R_STAGE = R_A + R_B;
    static constexpr int RS_FIT = (232448 - 1024 - 256) / R_STAGE;
    static constexpr int RS = RS_FIT < 12 ? RS_FIT : 12;
    static constexpr int SMEM = 1024 + RS * R_STAGE + 256;
    static constexpr int TMEM_COLS = RN < 32 ? 32 : RN;
    static_assert(RS >= 4 && SMEM <= 232448, "stages");
    static_assert(RS * R_STAGE >= RM * RN * 4, "the partial tile reuses the stage ring");
};

// Up to three products of the same x in one launch, concatenated along N:
// part i (weights w, w2, w3) starts at tile tile0[i] (INT_MAX: absent) and
// writes its rows to out[i] (width[i] columns a token, mode[i]); or two
// products into one output concatenated along K: slabs from k_split on take
// x2 and w2 (INT_MAX: none).  The logit offset applies to part 0.
struct DenseParts {
    void* out[3];
    int tile0[3], width[3], mode[3];
    int k_split;
};

// out[t, n] = sum_k x[t, k] * w[n, k]: x [S, K] bf16, w [N, K] bf16, fp32
// accumulation in TMEM.  grid (N / 128, ceil(S / RN), kslices) in clusters of
// (1, 1, kslices) over K.  The weight slabs of the first stages are issued
// before the wait on the preceding kernel (the weights are inputs of the
// call); the token slabs after it.
template <int RN>
__global__ void __launch_bounds__(R_THREADS, 1)
    k_dense_tc(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
               const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_x2,
               const __grid_constant__ CUtensorMap tm_w3, const float* __restrict__ off, int S, int K, int kslices,
               int w_evict_first, StatusBlock* __restrict__ sb, int kt_id, const DenseParts parts) {
    using C = DCfg<RN>;
    constexpr int RS = C::RS, R_STAGE = C::R_STAGE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + RS * R_STAGE);
    uint64_t* empty = full + RS;
    uint64_t* done = empty + RS;
    uint32_t* holder = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(holder + 1);
    float* part = reinterpret_cast<float*>(sm);   // [RN][RM] partial products, after the MMAs

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    KT_MARK(kt_id, 0);
    const int e0 = blockIdx.x * RM, t0 = blockIdx.y * RN, ks = blockIdx.z;
    const int bx = (int)blockIdx.x;
    const int pidx = bx >= parts.tile0[2] ? 2 : bx >= parts.tile0[1] ? 1 : 0;   // the tile's product
    const int row0 = e0 - parts.tile0[pidx] * RM;                               // its first row in its weights
    // the weight map of slab k, and its slab within that map
    auto wmap = [&](int k) {
        return pidx == 2 ? &tm_w3 : (pidx == 1 || k >= parts.k_split) ? &tm_w2 : &tm_w;
    };
    auto wslab = [&](int k) { return k >= parts.k_split ? k - parts.k_split : k; };
    const int nk = K / RK;
    const int kb = (int)((long long)nk * ks / kslices), ke = (int)((long long)nk * (ks + 1) / kslices);
    if (threadIdx.x == 0) {
        for (int i = 0; i < RS; ++i) {
            ptx::mbar_init(&full[i], 1);
            ptx::mbar_init(&empty[i], 1);
        }
        ptx::mbar_init(done, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(holder, C::TMEM_COLS);
    const uint64_t pol_w = w_evict_first ? ptx::policy_evict_first() : ptx::policy_evict_last();
    const uint64_t pol_x = ptx::policy_evict_last();
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tm_w);
        ptx::prefetch_tensormap(&tm_x);
        if (pidx == 1 || parts.k_split != INT_MAX) ptx::prefetch_tensormap(&tm_w2);
        if (parts.k_split != INT_MAX) ptx::prefetch_tensormap(&tm_x2);
        if (pidx == 2) ptx::prefetch_tensormap(&tm_w3);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *holder;
    const int n_pre = ke - kb < RS ? ke - kb : RS;   // stages whose weights go out before the wait
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < n_pre; ++i) {
            ptx::mbar_arrive_expect_tx(&full[i], R_STAGE);
            ptx::tma_load_2d(sm + i * R_STAGE, wmap(kb + i), wslab(kb + i) * RK, row0, &full[i], pol_w);
        }
    }
    pdl_wait();      // x may come from the stream's previous kernel
    pdl_trigger();   // successors start once this kernel's inputs are final
    KT_MARK(kt_id, 1);

    auto fail = [&](int site) {
        latch_status(sb, MOE_ERR_TIMEOUT, 100 + site);
        *abort_flag = 1;
    };
    if (warp == 0) {
        if (lane == 0) {
            for (int k = kb, i = 0; k < ke; ++k, ++i) {
                const int s = i % RS;
                uint8_t* st = sm + s * R_STAGE;
                if (i >= n_pre) {
                    if (!ptx::mbar_wait(&empty[s], ((i / RS) & 1) ^ 1, abort_flag, R_WAIT_NS)) {
                        fail(1);
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&full[s], R_STAGE);
                    ptx::tma_load_2d(st, wmap(k), wslab(k) * RK, row0, &full[s], pol_w);
                }
                ptx::tma_load_2d(st + R_A, k >= parts.k_split ? &tm_x2 : &tm_x, wslab(k) * RK, t0, &full[s], pol_x);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(RM, RN);
            for (int k = kb, i = 0; k < ke; ++k, ++i) {
                const int s = i % RS;
                if (!ptx::mbar_wait(&full[s], (i / RS) & 1, abort_flag, R_WAIT_NS)) {
                    fail(2);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t a0 = ptx::smem_u32(sm + s * R_STAGE), b0 = a0 + R_A;
#pragma unroll
                for (int j = 0; j < RK / 16; ++j)
                    ptx::mma_bf16_ss(tmem, ptx::smem_desc_sw128(a0 + 32 * j), ptx::smem_desc_sw128(b0 + 32 * j), idesc,
                                     (i > 0 || j > 0) ? 1u : 0u);
                ptx::mma_commit(&empty[s]);
            }
            ptx::mma_commit(done);   // arrives once every MMA above has completed
        }
    } else {
        // epilogue: row m = 32 (warp mod 4) + lane of the tile, RN token columns
        const int q = warp & 3;
        const int m = 32 * q + lane;
        const bool got = ptx::mbar_wait_warp(done, 0, abort_flag, R_WAIT_NS);
        if (warp == 2) KT_MARK(kt_id, 4);
        if (!got && lane == 0) fail(3);
        if (got) {
            ptx::tc_fence_after();
            const uint32_t lane_base = (uint32_t)(32 * q) << 16;
#pragma unroll 1
            for (int c = 0; c < RN; c += 16) {
                uint32_t v[16];
                ptx::tmem_ld16(tmem + lane_base + c, v);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) part[(c + j) * RM + m] = __uint_as_float(v[j]);
            }
        }
    }
    ptx::tc_fence_before();
    // the cluster's partial tiles, added in K-range order; CTA r of the cluster
    // writes tokens [r RN / KS, (r + 1) RN / KS) of the tile
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    KT_MARK(kt_id, 5);
    if (!*abort_flag) {
        const int n0 = RN * ks / kslices, n1 = RN * (ks + 1) / kslices;
        for (int idx = threadIdx.x; idx < (n1 - n0) * RM; idx += R_THREADS) {
            const int n = n0 + idx / RM, mm = idx % RM;
            float pz[R_MAX_CLUSTER];
#pragma unroll
            for (int r = 0; r < R_MAX_CLUSTER; ++r)
                pz[r] = r < kslices ? cluster.map_shared_rank(part, r)[n * RM + mm] : 0.f;
            float z = 0.f;
#pragma unroll
            for (int r = 0; r < R_MAX_CLUSTER; ++r) z += pz[r];
            const int t = t0 + n, e = row0 + mm;
            const int width = parts.width[pidx], md = parts.mode[pidx];
            void* dst = parts.out[pidx];
            if (t < S && e < width) {
                const size_t o = (size_t)t * width + e;
                if (md == DENSE_BF16) {
                    reinterpret_cast<__nv_bfloat16*>(dst)[o] = __float2bfloat16_rn(z);
                } else if (md == DENSE_F32_ADD) {
                    float* of = reinterpret_cast<float*>(dst);
                    of[o] = ld_dep(of + o) + z;
                } else {
                    reinterpret_cast<float*>(dst)[o] = (off && pidx == 0) ? z + off[e] : z;
                }
            }
        }
    }
    cluster.sync();   // every CTA keeps its partial tile until the others have read it
    KT_MARK(kt_id, 2);
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, C::TMEM_COLS);
}

// One launch of k_dense_tc<RN>: x [S, K] times the parts' weights (N-
// concatenation: w[i] [N[i], K], N[i] = 0 for an absent part), or
// x . w^T + x2 . w2^T (K-concatenation: K2 > 0, w [N, K], w2 [N, K2],
// x2 [S, K2]).
struct DenseArgs {
    const void* x;
    const void* x2;
    const void* w[3];
    int S, K, K2;
    int N[3];
    const float* off;
    void* out[3];
    int mode[3];
};

template <int RN>
cudaError_t launch_dense_rn(const DenseArgs& d, bool w_once, StatusBlock* sb, cudaStream_t st, int kt_id) {
    using C = DCfg<RN>;
    KT_BIND();
    CUtensorMap tm[3], tm_x, tm_x2;
    const uint32_t w_b[2] = {RK, RM}, x_b[2] = {RK, RN};
    auto map2d = [&](CUtensorMap* m, const void* base, int cols, int rows, const uint32_t* box) {
        const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows}, str[1] = {(uint64_t)cols * 2};
        return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
    };
    if (!map2d(&tm[0], d.w[0], d.K, d.N[0], w_b) || !map2d(&tm_x, d.x, d.K, d.S, x_b)) return cudaErrorInvalidValue;
    tm[1] = tm[2] = tm[0];
    tm_x2 = tm_x;
    if (d.K2 > 0) {
        if (!map2d(&tm[1], d.w[1], d.K2, d.N[0], w_b) || !map2d(&tm_x2, d.x2, d.K2, d.S, x_b))
            return cudaErrorInvalidValue;
    } else {
        for (int i = 1; i < 3; ++i)
            if (d.N[i] > 0 && !map2d(&tm[i], d.w[i], d.K, d.N[i], w_b)) return cudaErrorInvalidValue;
    }
    DenseParts parts;
    int ntile = 0;
    for (int i = 0; i < 3; ++i) {
        const bool on = i == 0 || (d.K2 == 0 && d.N[i] > 0);
        parts.tile0[i] = on ? ntile : INT_MAX;
        parts.out[i] = d.out[i];
        parts.width[i] = d.N[i];
        parts.mode[i] = d.mode[i];
        if (on) ntile += d.N[i] / RM;
    }
    parts.k_split = d.K2 > 0 ? d.K / RK : INT_MAX;
    const int tiles = ntile * ((d.S + RN - 1) / RN);
    const int nk = (d.K + (d.K2 > 0 ? d.K2 : 0)) / RK;
    int ks = num_sms() / tiles;                 // at most one CTA per SM: a second wave would double the time
    if (ks > R_MAX_CLUSTER) ks = R_MAX_CLUSTER;
    if (ks > nk / 4) ks = nk / 4;               // at least four slabs per CTA
    if (ks < 1) ks = 1;
    cudaError_t e = cudaFuncSetAttribute(k_dense_tc<RN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ntile, (d.S + RN - 1) / RN, ks);
    cfg.blockDim = dim3(R_THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = ks;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k_dense_tc<RN>, tm[0], tm_x, tm[1], tm_x2, tm[2], d.off, d.S, nk * RK, ks,
                              w_once ? 1 : 0, sb, kt_id, parts);
}

cudaError_t launch_dense_args(const DenseArgs& d, StatusBlock* sb, cudaStream_t st, int kt_id) {
    // one token tile of 16 for up to 16 tokens (a weight-streaming product), else tiles of 128; the
    // weights are read once (evict first) unless several token tiles read them
    if (d.S <= 16) return launch_dense_rn<16>(d, true, sb, st, kt_id);
    return launch_dense_rn<128>(d, d.S <= 128, sb, st, kt_id);
}

}  // namespace

// Which batches the router runs on the tensor cores (E a multiple of 128):
// 9 to 32 tokens in 16-token tiles (S = 32: 10.7 us against 14.5 us for the
// CUDA-core router), 64 and more in 128-token tiles.  Up to 8 tokens the
// CUDA-core kernel without staging is faster (the step 53 us against 59 us);
// at 128 tokens 16-token tiles were slower than 128-token ones (20.8 against
// 16.7 us: eight token tiles each read all the weights).
bool router_tc_fits(const moe_shape& s) {
    return ((s.S >= 9 && s.S <= 32) || s.S >= 64) && s.E % RM == 0 && s.d % RK == 0;
}

bool dense_fits(int S, int K, int N) { return S >= 1 && N % RM == 0 && K % RK == 0 && K / RK >= 1; }

cudaError_t launch_dense(const void* x, const void* w, int S, int K, int N, const float* off, void* out, int mode,
                         StatusBlock* sb, cudaStream_t st, int kt_id) {
    const DenseArgs d{x, nullptr, {w, nullptr, nullptr}, S, K, 0, {N, 0, 0}, off, {out, nullptr, nullptr},
                      {mode, 0, 0}};
    return launch_dense_args(d, sb, st, kt_id);
}

cudaError_t launch_dense_ncat(const void* x, int S, int K, const DensePart* p, int n_parts, const float* off,
                              StatusBlock* sb, cudaStream_t st, int kt_id) {
    DenseArgs d{x, nullptr, {nullptr, nullptr, nullptr}, S, K, 0, {0, 0, 0}, off, {nullptr, nullptr, nullptr},
                {0, 0, 0}};
    for (int i = 0; i < n_parts && i < 3; ++i) {
        d.w[i] = p[i].w;
        d.N[i] = p[i].N;
        d.out[i] = p[i].out;
        d.mode[i] = p[i].mode;
    }
    return launch_dense_args(d, sb, st, kt_id);
}

cudaError_t launch_dense_kcat(const void* x, const void* w, int K, const void* x2, const void* w2, int K2, int S,
                              int N, void* out, int mode, StatusBlock* sb, cudaStream_t st, int kt_id) {
    const DenseArgs d{x, x2, {w, w2, nullptr}, S, K, K2, {N, 0, 0}, nullptr, {out, nullptr, nullptr}, {mode, 0, 0}};
    return launch_dense_args(d, sb, st, kt_id);
}

cudaError_t launch_router_tc(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    const DenseArgs d{p.x, nullptr, {p.w_gate, nullptr, nullptr}, s.S, s.d, 0, {s.E, 0, 0}, p.logit_off,
                      {p.ws + L.logits, nullptr, nullptr}, {DENSE_F32, 0, 0}};
    StatusBlock* sb = reinterpret_cast<StatusBlock*>(p.ws + L.status);
    // up to 32 tokens, tiles of 16: E/128 x S/16 tiles, K split over a
    // cluster, spread the weight rows over more CTAs than one 128-token tile
    if (s.S <= 32) return launch_dense_rn<16>(d, s.S <= 16, sb, st, K_ROUTER);
    return launch_dense_rn<128>(d, false, sb, st, K_ROUTER);
}

}  // namespace moe
