// Router logits on the tensor cores, for batches of 64 tokens and more.
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

namespace cg = cooperative_groups;

namespace moe {

namespace {

constexpr int RM = 128;                    // experts per tile (MMA M)
constexpr int RN = 128;                    // tokens per tile (MMA N)
constexpr int RK = 64;                     // K elements per stage (one 128-byte slab)
constexpr int RS = 6;                      // stages
constexpr int R_A = RM * RK * 2;           // 16 KB
constexpr int R_B = RN * RK * 2;           // 16 KB
constexpr int R_STAGE = R_A + R_B;
constexpr int R_THREADS = 192;
constexpr int R_MAX_CLUSTER = 8;
constexpr int R_SMEM = 1024 + RS * R_STAGE + 256;
constexpr uint64_t R_WAIT_NS = 2000000000ull;
static_assert(RS * R_STAGE >= RM * RN * 4, "the partial tile reuses the stage ring");

__global__ void __launch_bounds__(R_THREADS, 1)
    k_router_tc(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                const float* __restrict__ off, float* __restrict__ L, int S, int d, int E, int kslices,
                StatusBlock* __restrict__ sb) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + RS * R_STAGE);
    uint64_t* empty = full + RS;
    uint64_t* done = empty + RS;
    uint32_t* holder = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(holder + 1);
    float* part = reinterpret_cast<float*>(sm);   // [RN][RM] partial logits, after the MMAs

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e0 = blockIdx.x * RM, t0 = blockIdx.y * RN, ks = blockIdx.z;
    const int nk = d / RK;
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
    if (warp == 1) ptx::tmem_alloc(holder, RN);
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tm_w);
        ptx::prefetch_tensormap(&tm_x);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *holder;
    pdl_wait();      // x may come from the stream's previous kernel
    pdl_trigger();   // the call's first kernel: successors start once the call's inputs are final

    auto fail = [&](int site) {
        latch_status(sb, MOE_ERR_TIMEOUT, 100 + site);
        *abort_flag = 1;
    };
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = ptx::policy_evict_last();   // w_gate is read by every token tile
            for (int k = kb, i = 0; k < ke; ++k, ++i) {
                const int s = i % RS;
                if (i >= RS && !ptx::mbar_wait(&empty[s], ((i / RS) & 1) ^ 1, abort_flag, R_WAIT_NS)) {
                    fail(1);
                    break;
                }
                uint8_t* st = sm + s * R_STAGE;
                ptx::mbar_arrive_expect_tx(&full[s], R_STAGE);
                ptx::tma_load_2d(st, &tm_w, k * RK, e0, &full[s], pol);
                ptx::tma_load_2d(st + R_A, &tm_x, k * RK, t0, &full[s], pol);
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
        // epilogue: row m = 32 (warp mod 4) + lane of the tile, 128 token columns
        const int q = warp & 3;
        const int m = 32 * q + lane;
        const bool got = ptx::mbar_wait_warp(done, 0, abort_flag, R_WAIT_NS);
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
            const int t = t0 + n, e = e0 + mm;
            if (t < S && e < E) L[(size_t)t * E + e] = off ? z + off[e] : z;
        }
    }
    cluster.sync();   // every CTA keeps its partial tile until the others have read it
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, RN);
}

}  // namespace

bool router_tc_fits(const moe_shape& s) { return s.S >= 64 && s.E % RM == 0 && s.d % RK == 0; }

cudaError_t launch_router_tc(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    CUtensorMap tm_w, tm_x;
    const uint64_t d = s.d, E = s.E, S = s.S;
    const uint64_t w_d[2] = {d, E}, w_s[1] = {d * 2};
    const uint64_t x_d[2] = {d, S}, x_s[1] = {d * 2};
    const uint32_t w_b[2] = {RK, RM}, x_b[2] = {RK, RN};
    if (!make_map(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.w_gate, 2, w_d, w_s, w_b, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.x, 2, x_d, x_s, x_b, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int tiles = (s.E / RM) * ((s.S + RN - 1) / RN);
    const int nk = s.d / RK;
    int ks = (num_sms() + tiles - 1) / tiles;   // about one CTA per SM
    if (ks > R_MAX_CLUSTER) ks = R_MAX_CLUSTER;
    if (ks > nk / 4) ks = nk / 4;               // at least four slabs per CTA
    if (ks < 1) ks = 1;
    cudaError_t e = cudaFuncSetAttribute(k_router_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, R_SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(s.E / RM, (s.S + RN - 1) / RN, ks);
    cfg.blockDim = dim3(R_THREADS);
    cfg.dynamicSmemBytes = R_SMEM;
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
    return cudaLaunchKernelEx(&cfg, k_router_tc, tm_w, tm_x, p.logit_off, reinterpret_cast<float*>(p.ws + L.logits),
                              s.S, s.d, s.E, ks, reinterpret_cast<StatusBlock*>(p.ws + L.status));
}

}  // namespace moe
