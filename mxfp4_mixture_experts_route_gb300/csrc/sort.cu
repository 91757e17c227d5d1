// Expert sort, work-tile schedule and token gather.
//
// vllm.models.muse_spark.amd.mono.kernels.k3, dn_loads: "Task (u, j)'s w2
// operands ... expert etab[u], u clamped below nv" -- the pages keep a table of
// the local experts that have picks and run tasks (expert, tile).  Here that
// table is built once per call: picks are counted per expert, placed in one
// segment per expert, and each segment is cut into tiles of at most nt picks
// (k5 page: "Every row tile is 16 tokens").  Experts without picks get no
// tile, so no weight byte of an untouched expert is read.
#include "moe_internal.cuh"
#include "tc_ptx.cuh"
#include "topk.cuh"
#include "quant.cuh"

#include <algorithm>

namespace moe {

namespace {

constexpr int SORT_THREADS = 1024;

struct SortOut {
    int32_t* counts;
    int32_t* offsets;
    int32_t* pos;
    int32_t* src;
    Tile* tiles;
    int32_t* active;
    uint32_t* tile_ready;
    int max_tiles;
    int nt;               // picks per tile
    StatusBlock* sb;
};

// shared-memory ints of sort_picks: per expert a count, a segment offset and a
// tile offset (E + 1 each)
__host__ __device__ constexpr int sort_smem_ints(int E) { return 3 * (E + 1); }

// Sort of the S * k picks by expert, one CTA of SORT_THREADS threads.
//   1. every pick p = t*k + j whose id e is in [0, E) and not repeated by an
//      earlier pick of token t takes a rank within expert e (a shared-memory
//      atomic); the others get pos[p] = -1 and latch MOE_ERR_BAD_IDS
//   2. one warp scans the counts over the experts: segment offsets, tile
//      offsets and active-expert slots
//   3. every thread places its picks (pos[p] = offset[e] + rank, src[pos] = p)
//      and writes tile entries (expert e, first pick, picks in the tile)
// The order of the picks inside a segment is the order the atomics came in:
// each pick is an independent column of the expert GEMMs, so the results do
// not depend on it.  ids may be in global or shared memory.
// Output: counts[E], offsets[E+1], pos[S*k], src[n_picks], tiles[n_tiles],
// active[n_active] and n_picks / n_tiles / n_active; tile_ready[] zeroed.
__device__ __forceinline__ void sort_picks(const int32_t* ids, int S, int E, int k, const SortOut& o,
                                           int32_t* smem) {
    int32_t* cnt = smem;               // [E + 1] counts
    int32_t* off = cnt + (E + 1);      // [E + 1] segment offsets
    int32_t* toff = off + (E + 1);     // [E + 1] tile offsets
    __shared__ int32_t tot_tiles;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = S * k;
    const int nt = o.nt;
    StatusBlock* sb = o.sb;

    for (int i = tid; i <= E; i += SORT_THREADS) cnt[i] = 0;
    for (int i = tid; i < o.max_tiles; i += SORT_THREADS) o.tile_ready[i] = 0u;
    __syncthreads();

    // 1 ----------------------------------------------------------------------
    // the lanes of a warp that hold the same expert share one atomic
    const uint32_t lower = (1u << lane) - 1u;
    for (int p0 = warp * 32; p0 < P; p0 += SORT_THREADS) {
        const int p = p0 + lane;
        int e = -1;
        bool ok = false;
        if (p < P) {
            const int t = p / k, j = p - t * k;
            e = ids[p];
            ok = e >= 0 && e < E;
            for (int q = 0; q < j && ok; ++q) ok = ids[(size_t)t * k + q] != e;
        }
        const uint32_t grp = __match_any_sync(0xffffffffu, ok ? e : -1 - lane);
        const int leader = __ffs(grp) - 1;
        int base = 0;
        if (ok && lane == leader) base = atomicAdd(&cnt[e], __popc(grp));
        base = __shfl_sync(0xffffffffu, base, leader);
        if (p < P) {
            if (ok) {
                o.pos[p] = base + __popc(grp & lower);   // rank within the expert, for now
            } else {
                o.pos[p] = -1;
                latch_status(sb, MOE_ERR_BAD_IDS, p);
            }
        }
    }
    __syncthreads();

    // 2 ----------------------------------------------------------------------
    if (warp == 0) {
        // lane l scans experts [l*per, (l+1)*per); three exclusive scans at once
        const int per = (E + 31) / 32;
        const int e0 = lane * per, e1 = min(E, e0 + per);
        int sp = 0, st = 0, sa = 0;
        for (int e = e0; e < e1; ++e) {
            const int n = cnt[e];
            sp += n;
            st += (n + nt - 1) / nt;
            sa += n > 0 ? 1 : 0;
        }
        int ip = sp, it = st, ia = sa;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, ip, m);
            const int b = __shfl_up_sync(0xffffffffu, it, m);
            const int c = __shfl_up_sync(0xffffffffu, ia, m);
            if (lane >= m) {
                ip += a;
                it += b;
                ia += c;
            }
        }
        int rp = ip - sp, rt = it - st, ra = ia - sa;   // exclusive prefixes of this lane's run
        for (int e = e0; e < e1; ++e) {
            const int n = cnt[e];
            off[e] = rp;
            toff[e] = rt;
            o.counts[e] = n;
            o.offsets[e] = rp;
            if (n > 0) o.active[ra++] = e;
            rp += n;
            rt += (n + nt - 1) / nt;
        }
        if (lane == 31) {
            off[E] = ip;
            toff[E] = it;
            tot_tiles = it;
            o.offsets[E] = ip;
            sb->n_picks = ip;
            sb->n_tiles = it;
            sb->n_active = ia;
            sb->work_next = 0;
            sb->work_next2 = 0;
        }
    }
    __syncthreads();

    // 3 ----------------------------------------------------------------------
    for (int p = warp * 32 + lane; p < P; p += SORT_THREADS) {
        const int r = o.pos[p];
        if (r >= 0) {
            const int q = off[ids[p]] + r;
            o.pos[p] = q;
            o.src[q] = p;
        }
    }
    const int n_tiles = tot_tiles;
    for (int ti = tid; ti < n_tiles; ti += SORT_THREADS) {
        // expert of tile ti: the last e with toff[e] <= ti (binary search)
        int lo = 0, hi = E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (toff[mid] <= ti) lo = mid;
            else hi = mid - 1;
        }
        const int i = ti - toff[lo];
        Tile tl;
        tl.e = lo;
        tl.p0 = off[lo] + i * nt;
        tl.n = min(nt, cnt[lo] - i * nt);
        tl.pad = 0;
        o.tiles[ti] = tl;
    }
}

__global__ void __launch_bounds__(SORT_THREADS) k_sort(const int32_t* __restrict__ ids, int S, int E, int k,
                                                       SortOut o) {
    extern __shared__ int32_t smem[];
    pdl_trigger();
    pdl_wait();
    sort_picks(ids, S, E, k, o, smem);
}

// moe_forward at small S: the sigmoid top-k of every token (one warp a token,
// see topk_token) and the sort of its picks in one CTA.  The ids go to the
// caller's buffer and, for the sort, to shared memory.
template <int MAXE>
__global__ void __launch_bounds__(SORT_THREADS) k_topk_sort(const float* __restrict__ L,
                                                            const float* __restrict__ bias, int S, int E, int k,
                                                            int32_t* __restrict__ ids,
                                                            float* __restrict__ weights, SortOut o) {
    extern __shared__ int32_t smem[];
    pdl_trigger();
    int32_t* sids = smem + sort_smem_ints(E);   // [S][k]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float b[MAXE];
    load_bias(bias, E, lane, b);   // an input of the call: read before the wait
    pdl_wait();
    for (int t = warp; t < S; t += SORT_THREADS / 32)
        topk_token(L + (size_t)t * E, b, E, k, lane, sids + (size_t)t * k, weights + (size_t)t * k);
    __syncthreads();
    for (int i = threadIdx.x; i < S * k; i += SORT_THREADS) ids[i] = sids[i];
    sort_picks(sids, S, E, k, o, smem);
}

// Token rows of the expert GEMMs (see quantize_pick).  grid (max_picks),
// blockDim = d / 8 rounded up to a warp (at most 1024), one pick a CTA.
__global__ void __launch_bounds__(1024) k_quant_gather(const __nv_bfloat16* __restrict__ x,
                                                      const int32_t* __restrict__ src, int k, int d, int I, int P,
                                                      uint8_t* __restrict__ xq, uint8_t* __restrict__ xs,
                                                      uint8_t* __restrict__ hs,
                                                      const StatusBlock* __restrict__ sb) {
    pdl_trigger();
    pdl_wait();
    const int p = blockIdx.x;
    const int sp = src[p];                 // read beside n_picks: src has max_picks entries
    if (p >= sb->n_picks) return;
    quantize_pick(x, sp / k, p, d, I, (size_t)P + NT_MAX, xq, xs, hs, threadIdx.x, blockDim.x);
}

}  // namespace

static SortOut sort_out(const WsLayout& L, char* ws) {
    SortOut o;
    o.counts = reinterpret_cast<int32_t*>(ws + L.counts);
    o.offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
    o.pos = reinterpret_cast<int32_t*>(ws + L.pos);
    o.src = reinterpret_cast<int32_t*>(ws + L.src);
    o.tiles = reinterpret_cast<Tile*>(ws + L.tiles);
    o.active = reinterpret_cast<int32_t*>(ws + L.active);
    o.tile_ready = reinterpret_cast<uint32_t*>(ws + L.tile_ready);
    o.max_tiles = L.max_tiles;
    o.nt = L.nt;
    o.sb = reinterpret_cast<StatusBlock*>(ws + L.status);
    return o;
}

static cudaError_t launch_gather(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    char* ws = p.ws;
    timing_begin(K_GATHER, st);
    const int threads = std::min(1024, (s.d / 8 + 31) / 32 * 32);
    const cudaError_t e = launch_pdl(k_quant_gather, dim3(L.max_picks), dim3(threads), 0, st, p.x,
                                     reinterpret_cast<const int32_t*>(ws + L.src), s.k, s.d, s.I, L.max_picks,
                                     reinterpret_cast<uint8_t*>(ws + L.xq), reinterpret_cast<uint8_t*>(ws + L.xs),
                                     reinterpret_cast<uint8_t*>(ws + L.hs),
                                     reinterpret_cast<const StatusBlock*>(ws + L.status));
    timing_end(st);
    return e;
}

cudaError_t launch_sort_gather(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    const size_t smem = (size_t)sort_smem_ints(s.E) * sizeof(int32_t);
    timing_begin(K_SORT, st);
    cudaError_t e = launch_pdl(k_sort, dim3(1), dim3(SORT_THREADS), smem, st, (const int32_t*)p.ids, s.S, s.E, s.k,
                               sort_out(L, p.ws));
    timing_end(st);
    if (e != cudaSuccess) return e;
    return launch_gather(s, L, p, st);
}

bool topk_sort_fits(const moe_shape& s) {
    // one token a warp (beyond that the top-k kernel spreads the tokens over
    // more SMs), and the ids of the call in shared memory
    return s.S <= SORT_THREADS / 32 && (size_t)s.S * s.k <= 8192;
}

cudaError_t launch_topk_sort_gather(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    const size_t smem = ((size_t)sort_smem_ints(s.E) + (size_t)s.S * s.k) * sizeof(int32_t);
    auto kern = s.E <= 256 ? k_topk_sort<256 / 32> : k_topk_sort<512 / 32>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    timing_begin(K_TOPK_SORT, st);
    e = launch_pdl(kern, dim3(1), dim3(SORT_THREADS), smem, st, reinterpret_cast<const float*>(p.ws + L.logits),
                   p.bias, s.S, s.E, s.k, p.ids, p.weights, sort_out(L, p.ws));
    timing_end(st);
    if (e != cudaSuccess) return e;
    return launch_gather(s, L, p, st);
}

}  // namespace moe
