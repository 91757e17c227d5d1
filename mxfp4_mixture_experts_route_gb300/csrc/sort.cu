// Expert sort, work-tile schedule and token gather.
//
// vllm.models.muse_spark.amd.mono.kernels.k3, dn_loads: "Task (u, j)'s w2
// operands ... expert etab[u], u clamped below nv" -- the pages keep a table of
// the local experts that have picks and run tasks (expert, tile).  Here that
// table is built once per call: picks are counted per expert, sorted by
// (expert, token) with a stable counting sort, and cut into tiles of at most
// NT picks of one expert (k5 page: "Every row tile is 16 tokens").  Experts
// without picks get no tile, so no weight byte of an untouched expert is read.
#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int MAX_K = 16;

// One CTA of SORT_WARPS warps.  Warp w owns a range of 32-token groups and
// walks it with lane = token.
//   pass 1: validate ids, per-warp per-expert counts (smem)
//   pass 2: per-expert exclusive scan over warps, scan over experts -> offsets,
//           tile schedule, active list
//   pass 3: positions: offset[e] + base[w][e] + rank among earlier tokens of
//           the group that picked e (a 32-bit lane mask per expert)
// Output: counts[E], offsets[E+1], pos[t*k+j] (-1 for an invalid pick),
// src[p] = t*k+j, tiles[], active[], and n_picks / n_tiles / n_active.
// Global memory is only read for the ids (all of a token's ids in flight at
// once); everything the passes share stays in shared memory.
template <int SORT_WARPS>
__global__ void __launch_bounds__(SORT_WARPS * 32) k_sort(const int32_t* __restrict__ ids, int S, int E, int k,
                                                          int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ pos, int32_t* __restrict__ src,
                                                          Tile* __restrict__ tiles, int32_t* __restrict__ active,
                                                          uint32_t* __restrict__ tile_ready, int max_tiles,
                                                          StatusBlock* __restrict__ sb) {
    constexpr int SORT_THREADS = SORT_WARPS * 32;
    extern __shared__ int32_t smem[];
    int32_t* cnt = smem;                        // [SORT_WARPS][E]
    uint32_t* mask = reinterpret_cast<uint32_t*>(smem + SORT_WARPS * E);  // [SORT_WARPS][E]
    int32_t* etot = smem + 2 * SORT_WARPS * E;  // [E] totals, then exclusive offsets
    int32_t* etil = etot + E;                   // [E] tiles per expert, then tile offsets
    int32_t* eact = etil + E;                   // [E] active flag, then active slot
    int32_t* ecnt = eact + E;                   // [E] picks per expert
    __shared__ int32_t scan_tmp[32];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < 2 * SORT_WARPS * E; i += SORT_THREADS) smem[i] = 0;
    for (int i = tid; i < max_tiles; i += SORT_THREADS) tile_ready[i] = 0u;
    __syncthreads();

    const int groups = (S + 31) / 32;
    const int gpw = (groups + SORT_WARPS - 1) / SORT_WARPS;   // groups per warp
    const int g0 = warp * gpw, g1 = min(groups, g0 + gpw);

    // token t's k ids; bit j of the result is set when pick j is an id in
    // [0, E) that no earlier pick of the token repeats
    auto load_ids = [&](int t, int* my) -> uint32_t {
#pragma unroll
        for (int j = 0; j < MAX_K; ++j) my[j] = (j < k) ? __ldg(ids + (size_t)t * k + j) : -1;
        uint32_t valid = 0;
#pragma unroll
        for (int j = 0; j < MAX_K; ++j) {
            bool ok = j < k && my[j] >= 0 && my[j] < E;
#pragma unroll
            for (int q = 0; q < j; ++q) ok = ok && (my[q] != my[j]);
            valid |= ok ? 1u << j : 0u;
        }
        return valid;
    };

    // pass 1 ------------------------------------------------------------
    for (int g = g0; g < g1; ++g) {
        const int t = g * 32 + lane;
        if (t < S) {
            int my[MAX_K];
            const uint32_t valid = load_ids(t, my);
#pragma unroll
            for (int j = 0; j < MAX_K; ++j) {
                if (valid >> j & 1u) atomicAdd(&cnt[warp * E + my[j]], 1);
                else if (j < k) latch_status(sb, MOE_ERR_BAD_IDS, t * k + j);
            }
        }
    }
    __syncthreads();

    // pass 2 ------------------------------------------------------------
    for (int e = tid; e < E; e += SORT_THREADS) {
        int run = 0;
        for (int w = 0; w < SORT_WARPS; ++w) {
            const int c = cnt[w * E + e];
            cnt[w * E + e] = run;
            run += c;
        }
        etot[e] = run;
        ecnt[e] = run;
        etil[e] = (run + NT - 1) / NT;
        eact[e] = run > 0 ? 1 : 0;
    }
    __syncthreads();
    // three exclusive scans over E (E <= 512): each thread scans a run of
    // consecutive elements, then the runs' sums are scanned across the block
    auto block_scan = [&](int32_t* a, int32_t* total) {
        const int per = (E + SORT_THREADS - 1) / SORT_THREADS;
        const int b0 = tid * per, b1 = min(E, b0 + per);
        int v = 0;
        for (int i = b0; i < b1; ++i) v += a[i];
        int inc = v;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, inc, m);
            if (lane >= m) inc += o;
        }
        if (lane == 31) scan_tmp[warp] = inc;
        __syncthreads();
        if (warp == 0) {
            const int w = lane < SORT_WARPS ? scan_tmp[lane] : 0;
            int wi = w;
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, wi, m);
                if (lane >= m) wi += o;
            }
            if (lane < SORT_WARPS) scan_tmp[lane] = wi - w;   // exclusive prefix of the warp sums
            if (lane == 31) *total = wi;
        }
        __syncthreads();
        int run = scan_tmp[warp] + inc - v;
        for (int i = b0; i < b1; ++i) {
            const int x = a[i];
            a[i] = run;
            run += x;
        }
        __syncthreads();
    };
    __shared__ int32_t tot_picks, tot_tiles, tot_active;
    for (int e = tid; e < E; e += SORT_THREADS) counts[e] = ecnt[e];
    block_scan(etot, &tot_picks);
    block_scan(etil, &tot_tiles);
    block_scan(eact, &tot_active);
    for (int e = tid; e < E; e += SORT_THREADS) {
        const int n = ecnt[e];
        offsets[e] = etot[e];
        if (n > 0) active[eact[e]] = e;
        for (int i = 0, tb = etil[e]; i * NT < n; ++i) {
            Tile tl;
            tl.e = e;
            tl.p0 = etot[e] + i * NT;
            tl.n = min(NT, n - i * NT);
            tl.pad = 0;
            tiles[tb + i] = tl;
        }
    }
    if (tid == 0) {
        offsets[E] = tot_picks;
        sb->n_picks = tot_picks;
        sb->n_tiles = tot_tiles;
        sb->n_active = tot_active;
        sb->work_next = 0;
        sb->work_next2 = 0;
    }

    // pass 3 ------------------------------------------------------------
    const uint32_t lt = (1u << lane) - 1u;
    for (int g = g0; g < g1; ++g) {
        const int t = g * 32 + lane;
        int my[MAX_K];
        uint32_t valid = 0;
        if (t < S) {
            valid = load_ids(t, my);
#pragma unroll
            for (int j = 0; j < MAX_K; ++j) {
                if (valid >> j & 1u) atomicOr(&mask[warp * E + my[j]], 1u << lane);
                else if (j < k) pos[(size_t)t * k + j] = -1;
            }
        }
        __syncwarp();
        int rank0[MAX_K];
#pragma unroll
        for (int j = 0; j < MAX_K; ++j) {
            rank0[j] = -1;
            if (valid >> j & 1u) {
                const int e = my[j];
                const uint32_t m = mask[warp * E + e];
                const int r = __popc(m & lt);
                const int p = etot[e] + cnt[warp * E + e] + r;
                pos[(size_t)t * k + j] = p;
                src[p] = t * k + j;
                rank0[j] = (r == 0) ? __popc(m) : -1;
            }
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < MAX_K; ++j) {
            if (rank0[j] >= 0) {
                const int e = my[j];
                cnt[warp * E + e] += rank0[j];
                mask[warp * E + e] = 0u;
            }
        }
        __syncwarp();
    }
}

// Token rows of the expert GEMMs.  For every valid pick p < n_picks, token
// t = src[p] / k: rows 2p and 2p + 1 of xq hold hi = e4m3(x[t] / 2^s) and
// lo = e4m3(x[t] / 2^s - hi) for every 32-element block, and the scale table
// xs holds the block's e8m0 byte s + 127, chosen so that the block's largest
// magnitude divided by 2^s lies in [128, 256) (clamped to bytes 1..247).  For
// a bf16 x the two rows add up to x / 2^s exactly, but for elements more than
// 2^9 below the block maximum (there the error is below 2^-17 of it).  The
// unused bytes of the last stage's scale rows of xs and hs (K / 32 not a
// multiple of 8) are set to 127 (scale 1), as their codes are zero.
// grid (max_picks), 128 threads; a thread takes 8 elements, four threads a
// block.
__global__ void __launch_bounds__(128) k_quant_gather(const __nv_bfloat16* __restrict__ x,
                                                      const int32_t* __restrict__ src, int k, int d, int I, int P,
                                                      uint8_t* __restrict__ xq, uint8_t* __restrict__ xs,
                                                      uint8_t* __restrict__ hs,
                                                      const StatusBlock* __restrict__ sb) {
    const int p = blockIdx.x;
    const int sp = src[p];                 // read beside n_picks: src has max_picks entries
    if (p >= sb->n_picks) return;
    const int t = sp / k;
    const size_t rows = (size_t)P + NT;
    const uint4* in = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    uint8_t* hi_row = xq + (size_t)(2 * p) * d;
    uint8_t* lo_row = hi_row + d;
    for (int c0 = 0; c0 < d / 8; c0 += blockDim.x) {
        const int c = c0 + threadIdx.x;
        const bool act = c < d / 8;        // whole blocks of four threads (d / 8 is a multiple of 16)
        const uint4 v = act ? __ldg(in + c) : make_uint4(0, 0, 0, 0);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        float f[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[2 * j] = __uint_as_float(wv[j] << 16);
            f[2 * j + 1] = __uint_as_float(wv[j] & 0xFFFF0000u);
        }
        uint32_t amax = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = max(amax, __float_as_uint(fabsf(f[j])));
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        int e = (int)((amax >> 23) & 0xFFu) - 7;
        e = e < 1 ? 1 : (e > 247 ? 247 : e);
        const float mult = __uint_as_float((uint32_t)(254 - e) << 23);   // 2^-(e - 127)
        uint32_t hw[2] = {0, 0}, lw[2] = {0, 0};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a0 = f[2 * j] * mult, a1 = f[2 * j + 1] * mult;
            const uint32_t h2 = ptx::cvt_e4m3x2(a0, a1);
            float b0, b1;
            ptx::e4m3x2_to_f32(h2, b0, b1);
            const uint32_t l2 = ptx::cvt_e4m3x2(a0 - b0, a1 - b1);
            hw[j >> 1] |= h2 << (16 * (j & 1));
            lw[j >> 1] |= l2 << (16 * (j & 1));
        }
        if (act) {
            *reinterpret_cast<uint2*>(hi_row + 8 * c) = make_uint2(hw[0], hw[1]);
            *reinterpret_cast<uint2*>(lo_row + 8 * c) = make_uint2(lw[0], lw[1]);
            if ((c & 3) == 0) {
                const int blk = c >> 2;
                xs[((size_t)(blk >> 3) * rows + p) * TOKEN_SCALE_ROW + (blk & 7)] = (uint8_t)e;
            }
        }
    }
    if (threadIdx.x < 8) {
        const int j = threadIdx.x;
        const int nbx = d / 32, nbh = I / 32;
        if ((nbx & 7) && j >= (nbx & 7)) xs[((size_t)(nbx >> 3) * rows + p) * TOKEN_SCALE_ROW + j] = 127;
        if ((nbh & 7) && j >= (nbh & 7)) hs[((size_t)(nbh >> 3) * rows + p) * TOKEN_SCALE_ROW + j] = 127;
    }
}

}  // namespace

cudaError_t launch_sort_gather(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    char* ws = p.ws;
    StatusBlock* sb = reinterpret_cast<StatusBlock*>(ws + L.status);
    // small batches: 8 warps (the per-warp tables are then 8 x E); large: 32
    const bool big = (size_t)s.S * s.k > 2048;
    const int warps = big ? 32 : 8;
    const size_t smem = (size_t)(2 * warps * s.E + 4 * s.E) * sizeof(int32_t);
    auto kern = big ? k_sort<32> : k_sort<8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    timing_begin(K_SORT, st);
    kern<<<1, warps * 32, smem, st>>>(p.ids, s.S, s.E, s.k, reinterpret_cast<int32_t*>(ws + L.counts),
                                          reinterpret_cast<int32_t*>(ws + L.offsets),
                                          reinterpret_cast<int32_t*>(ws + L.pos),
                                          reinterpret_cast<int32_t*>(ws + L.src),
                                          reinterpret_cast<Tile*>(ws + L.tiles),
                                          reinterpret_cast<int32_t*>(ws + L.active),
                                          reinterpret_cast<uint32_t*>(ws + L.tile_ready), L.max_tiles, sb);
    timing_end(st);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    timing_begin(K_GATHER, st);
    k_quant_gather<<<L.max_picks, 128, 0, st>>>(p.x, reinterpret_cast<const int32_t*>(ws + L.src), s.k, s.d, s.I,
                                                L.max_picks, reinterpret_cast<uint8_t*>(ws + L.xq),
                                                reinterpret_cast<uint8_t*>(ws + L.xs),
                                                reinterpret_cast<uint8_t*>(ws + L.hs), sb);
    timing_end(st);
    return cudaGetLastError();
}

}  // namespace moe
