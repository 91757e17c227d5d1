// Expert GEMMs on the CUDA cores (first, straightforward version).
//
// vllm.models.muse_spark.amd.mono.kernels.k3, stages C, D: "gate_up / down of
// the local experts: MXFP4 weights ..., decoded in registers".  Each thread
// owns one weight row (a gate row and its up row, or a down row), decodes 32
// e2m1 elements of one e8m0 block at a time and applies the block scale to the
// 32-element partial sums; the tile's picks (<= NT) are staged in shared
// memory as fp32.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int ROWS = 128;   // weight rows per CTA (one per thread)
constexpr int KC = 256;     // K elements staged per round

// e2m1 code -> value (OCP MX v1.0 FP4: sign, 2-bit exponent with bias 1,
// 1 mantissa bit; exponent 0 is the subnormal 0.5 * m)
__device__ __forceinline__ float e2m1_f32(uint32_t c) {
    const uint32_t ex = (c >> 1) & 3u, m = c & 1u;
    const float mag = ex == 0 ? 0.5f * (float)m : __int_as_float((126u + ex) << 23) * (1.0f + 0.5f * (float)m);
    return (c & 8u) ? -mag : mag;
}

// 2^(b - 127) for an e8m0 byte b in 0..128; a larger byte latches
// MOE_ERR_BAD_SCALE and reads as 0
__device__ __forceinline__ float e8m0_f32(uint32_t b, StatusBlock* sb) {
    if (b > 128u) {
        latch_status(sb, MOE_ERR_BAD_SCALE, (int)b);
        return 0.f;
    }
    return b ? __int_as_float(b << 23) : __int_as_float(0x00400000);
}

__device__ __forceinline__ void decode32(const uint4 q, float* v) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int n = 0; n < 8; ++n) v[8 * i + n] = e2m1_f32((w[i] >> (4 * n)) & 15u);
}

// stage rows p0 .. p0+n-1 (K slice kc .. kc+KC) of a bf16 [*, K] matrix into xs
__device__ __forceinline__ void stage(float (*xs)[KC], const __nv_bfloat16* __restrict__ a, int p0, int n,
                                      int K, int kc) {
    for (int idx = threadIdx.x; idx < NT * KC; idx += ROWS) {
        const int j = idx / KC, c = idx % KC;
        xs[j][c] = (j < n && kc + c < K) ? __bfloat162float(a[(size_t)(p0 + j) * K + kc + c]) : 0.f;
    }
}

// h[p, i] = silu(W1_e x_p)[i] * (W3_e x_p)[i] for the picks p of one tile.
// grid (max_tiles, I/ROWS)
__global__ void __launch_bounds__(ROWS) k_gateup_simt(const Tile* __restrict__ tiles,
                                                      const __nv_bfloat16* __restrict__ xg,
                                                      const uint8_t* __restrict__ w13,
                                                      const uint8_t* __restrict__ w13s, int d, int I,
                                                      __nv_bfloat16* __restrict__ h, StatusBlock* sb) {
    if ((int)blockIdx.x >= sb->n_tiles) return;
    const Tile tl = tiles[blockIdx.x];
    const int i = blockIdx.y * ROWS + threadIdx.x;
    __shared__ float xs[NT][KC];
    const size_t gr = (size_t)tl.e * 2 * I + i, ur = gr + I;
    const uint8_t* gq = w13 + gr * (d / 2);
    const uint8_t* uq = w13 + ur * (d / 2);
    const uint8_t* gs = w13s + gr * (d / 32);
    const uint8_t* us = w13s + ur * (d / 32);
    float ag[NT], au[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) ag[j] = au[j] = 0.f;
    for (int kc = 0; kc < d; kc += KC) {
        __syncthreads();
        stage(xs, xg, tl.p0, tl.n, d, kc);
        __syncthreads();
        const int nb = min(KC, d - kc) / 32;
        for (int b = 0; b < nb; ++b) {
            const int k0 = kc + 32 * b;
            float vg[32], vu[32];
            decode32(__ldg(reinterpret_cast<const uint4*>(gq + k0 / 2)), vg);
            decode32(__ldg(reinterpret_cast<const uint4*>(uq + k0 / 2)), vu);
            const float sg = e8m0_f32(gs[k0 / 32], sb), su = e8m0_f32(us[k0 / 32], sb);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if (j < tl.n) {
                    float dg = 0.f, du = 0.f;
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        dg = fmaf(vg[c], xs[j][32 * b + c], dg);
                        du = fmaf(vu[c], xs[j][32 * b + c], du);
                    }
                    ag[j] = fmaf(sg, dg, ag[j]);
                    au[j] = fmaf(su, du, au[j]);
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        if (j < tl.n) {
            const float g = ag[j];
            const float hv = g / (1.0f + expf(-g)) * au[j];
            h[(size_t)(tl.p0 + j) * I + i] = __float2bfloat16_rn(hv);
        }
    }
}

// y[p, m] = (W2_e h_p)[m] for the picks p of one tile.  grid (max_tiles, d/ROWS)
__global__ void __launch_bounds__(ROWS) k_down_simt(const Tile* __restrict__ tiles,
                                                    const __nv_bfloat16* __restrict__ h,
                                                    const uint8_t* __restrict__ w2, const uint8_t* __restrict__ w2s,
                                                    int d, int I, float* __restrict__ y, StatusBlock* sb) {
    if ((int)blockIdx.x >= sb->n_tiles) return;
    const Tile tl = tiles[blockIdx.x];
    const int m = blockIdx.y * ROWS + threadIdx.x;
    __shared__ float hs[NT][KC];
    const size_t r = (size_t)tl.e * d + m;
    const uint8_t* q = w2 + r * (I / 2);
    const uint8_t* sc = w2s + r * (I / 32);
    float acc[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j] = 0.f;
    for (int kc = 0; kc < I; kc += KC) {
        __syncthreads();
        stage(hs, h, tl.p0, tl.n, I, kc);
        __syncthreads();
        const int nb = min(KC, I - kc) / 32;
        for (int b = 0; b < nb; ++b) {
            const int k0 = kc + 32 * b;
            float v[32];
            decode32(__ldg(reinterpret_cast<const uint4*>(q + k0 / 2)), v);
            const float s = e8m0_f32(sc[k0 / 32], sb);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if (j < tl.n) {
                    float dv = 0.f;
#pragma unroll
                    for (int c = 0; c < 32; ++c) dv = fmaf(v[c], hs[j][32 * b + c], dv);
                    acc[j] = fmaf(s, dv, acc[j]);
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j)
        if (j < tl.n) y[(size_t)(tl.p0 + j) * d + m] = acc[j];
}

}  // namespace

cudaError_t launch_experts(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    StatusBlock* sb = reinterpret_cast<StatusBlock*>(p.ws + L.status);
    const Tile* tiles = reinterpret_cast<const Tile*>(p.ws + L.tiles);
    __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(p.ws + L.h);
    timing_begin(K_GATEUP, st);
    k_gateup_simt<<<dim3(L.max_tiles, s.I / ROWS), ROWS, 0, st>>>(
        tiles, reinterpret_cast<const __nv_bfloat16*>(p.ws + L.xg), p.w13, p.w13s, s.d, s.I, h, sb);
    timing_end(st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    timing_begin(K_DOWN, st);
    k_down_simt<<<dim3(L.max_tiles, s.d / ROWS), ROWS, 0, st>>>(tiles, h, p.w2, p.w2s, s.d, s.I,
                                                                reinterpret_cast<float*>(p.ws + L.y), sb);
    timing_end(st);
    return cudaGetLastError();
}

}  // namespace moe
