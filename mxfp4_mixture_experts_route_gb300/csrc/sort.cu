// Expert sort, work-tile schedule and token gather.
//
// vllm.models.muse_spark.amd.mono.kernels.k3, dn_loads: a task (u, j) loads the
// down weights of the u-th entry of a table of the local experts that have
// picks, so the work runs as tasks (expert, tile).  Here that
// table is built once per call: picks are counted per expert, placed in one
// segment per expert, and each segment is cut into tiles of at most nt picks
// (the k5 page uses 16-token row tiles).  Experts without picks get no
// tile, so no weight byte of an untouched expert is read.
#include "moe_internal.cuh"
#include "tc_ptx.cuh"
#include "topk.cuh"
#include "quant.cuh"

#include <algorithm>

namespace moe {

namespace {

struct SortOut {
    int32_t* pos;
    Tile* tiles;
    uint32_t* tile_ready;
    int max_tiles;
    int nt;               // picks per tile
    StatusBlock* sb;
};

constexpr int GATHER_PASSES = 2;   // chunks of 8 elements a thread of k_gather_tok: d <= 16384
constexpr int SMALL_SORT_PICKS = 128;   // up to this many picks, moe_experts places them in k_route_gather

// moe_forward at small S: the top k of every token, the sort of all S * k
// picks and the gather in one kernel.  grid (S * k), one pick p = t * k + j a
// CTA, as the gather.  Every CTA selects every token's top k (a warp takes
// one or two tokens, topk_select) into shared memory, from the same logits
// with the same code, so all CTAs hold the same ids.  Each then places only
// its own pick, in the order of a stable sort by expert: with cnt[e] the picks of expert e,
// r_p = sum_{e < e_p} cnt[e] + #{q < p : e_q = e_p}; a tile opens where that
// index inside the segment is a multiple of nt, and tiles are numbered in
// position order: sum_{e < e_p} ceil(cnt[e] / nt) + index / nt.  It writes
// ids[p], weights[p], pos[p], that tile entry when its pick opens one, and
// token t's row (quantised before the wait) at r_p; CTA 0 writes the counts.
// The picks of a token are distinct valid experts.  With FROM_IDS the ids
// come from the top-k kernel (more tokens than each CTA should select again)
// or from moe_experts' caller (up to 128 picks): every CTA reads them, checks
// them (an id out of range or repeated by an earlier pick of its token is left
// out, latching MOE_ERR_BAD_IDS), and only places and gathers.  The rows are
// quantised before the wait when every kernel that could write them has
// completed before this one may start (after the router, which lets its
// successors start only past its own wait), after it otherwise
// (x_after_wait: rows an earlier kernel of the call wrote, or the first
// kernel of moe_experts, whose predecessor is the caller's).
constexpr int RG_THREADS = 512;        // at most; 16 warps: two tokens a warp at S = 32
constexpr int RG_PASSES = 4;           // chunks of 8 elements a thread, at most: d <= 16384
constexpr int RG_TOKENS_PER_WARP = 2;
constexpr size_t RG_ONE_PER_SM_SMEM = 117 * 1024;   // over half an SM's 228 KB
template <int MAXE, int PASSES, bool FROM_IDS>
__global__ void __launch_bounds__(RG_THREADS) k_route_gather(const float* L, const float* __restrict__ bias,
                                                            const __nv_bfloat16* __restrict__ x, int S, int E,
                                                            int k, int d, int I, int P_tab,
                                                            int32_t* __restrict__ ids, float* __restrict__ weights,
                                                            SortOut o, uint8_t* __restrict__ xq,
                                                            uint8_t* __restrict__ xs, uint8_t* __restrict__ hs,
                                                            int x_after_wait) {
    extern __shared__ int32_t smem[];
    KT_MARK(K_ROUTE_GATHER, 0);
    pdl_trigger();
    const int P = S * k, nt = o.nt;
    __shared__ int32_t r_sh;
    int32_t* key = smem;           // [P] expert of pick q = t * k + j (-1: not a valid pick)
    int32_t* cnt = key + P;        // [E] picks of expert e
    float* s_sh = reinterpret_cast<float*>(cnt + E);   // [min(S, warps)][32 * MAXE] (selecting)
    int32_t* raw = cnt + E;        // [P] the ids as given (FROM_IDS)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = (int)blockDim.x >> 5;
    const int p = blockIdx.x, t = p / k;
    const uint4* in = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    const int nc = d / 8;
    QuantChunk q[PASSES];
    if (!x_after_wait) {
#pragma unroll
        for (int i = 0; i < PASSES; ++i) {
            const int c = i * (int)blockDim.x + tid;
            if (i * (int)blockDim.x < nc) q[i] = quantize_chunk(in, c, c < nc);   // block-uniform condition
        }
    }
    float b[MAXE];
    if constexpr (!FROM_IDS) load_bias(bias, E, lane, b);
    for (int i = tid; i < E; i += blockDim.x) cnt[i] = 0;
    pdl_wait();
    KT_MARK(K_ROUTE_GATHER, 1);
    if (x_after_wait) {
#pragma unroll
        for (int i = 0; i < PASSES; ++i) {
            const int c = i * (int)blockDim.x + tid;
            if (i * (int)blockDim.x < nc) q[i] = quantize_chunk_dep(in, c, c < nc);
        }
    }
    if constexpr (FROM_IDS) {
        // ids from the top-k kernel or from the caller: a pick is valid when its
        // id is in [0, E) and not an id of an earlier pick of its token; the
        // others are left out (pos = -1) and latch MOE_ERR_BAD_IDS
        for (int i = tid; i < P; i += blockDim.x) raw[i] = ld_dep(ids + i);
        __syncthreads();
        for (int i = tid; i < P; i += blockDim.x) {
            const int t2 = i / k, j = i - t2 * k, e = raw[i];
            bool ok = e >= 0 && e < E;
            for (int q2 = 0; q2 < j && ok; ++q2) ok = raw[t2 * k + q2] != e;
            key[i] = ok ? e : -1;
            if (!ok && p == 0) latch_status(o.sb, MOE_ERR_BAD_IDS, i);
        }
    } else {
        // the warp's tokens warp and warp + nw: both rows of logits in flight first
        float z[RG_TOKENS_PER_WARP][MAXE];
#pragma unroll
        for (int u = 0; u < RG_TOKENS_PER_WARP; ++u)
            if (warp + u * nw < S) topk_load(L + (size_t)(warp + u * nw) * E, E, lane, z[u]);
#pragma unroll
        for (int u = 0; u < RG_TOKENS_PER_WARP; ++u) {
            const int tt = warp + u * nw;
            if (tt < S) {
                int id, rank;
                float w;
                topk_select(z[u], b, E, k, lane, s_sh + warp * 32 * MAXE, id, w, rank);
                if (lane < k) {
                    key[tt * k + rank] = id;
                    if (tt * k + rank == p) {
                        ids[p] = id;
                        weights[p] = w;
                    }
                }
            }
        }
    }
    __syncthreads();
    KT_MARK(K_ROUTE_GATHER, 3);
    for (int i = tid; i < P; i += blockDim.x)
        if (key[i] >= 0) atomicAdd(&cnt[key[i]], 1);
    __syncthreads();
    if (warp == 0) {
        const int ep = key[p];
        int off = 0, toff = 0, ntiles = 0, nvalid = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int n = e < E ? cnt[e] : 0;
            const int tn = (n + nt - 1) / nt;
            off += e < ep ? n : 0;
            toff += e < ep ? tn : 0;
            ntiles += tn;
            nvalid += n;
        }
        off = __reduce_add_sync(0xffffffffu, off);
        toff = __reduce_add_sync(0xffffffffu, toff);
        ntiles = __reduce_add_sync(0xffffffffu, ntiles);
        nvalid = __reduce_add_sync(0xffffffffu, nvalid);
        int idx = 0;   // picks of expert ep before p
        for (int q0 = 0; q0 < p; q0 += 32) {
            const int qq = q0 + lane;
            idx += __popc(__ballot_sync(0xffffffffu, qq < p && key[qq] == ep));
        }
        if (lane == 0) {
            const int r = ep >= 0 ? off + idx : -1;
            r_sh = r;
            o.pos[p] = r;
            if (ep >= 0 && idx % nt == 0) {
                Tile tl;
                tl.e = ep;
                tl.p0 = r;
                tl.n = min(nt, cnt[ep] - idx);
                tl.pad = 0;
                o.tiles[toff + idx / nt] = tl;
            }
            if (p == 0) {
                o.sb->n_picks = nvalid;
                o.sb->n_tiles = ntiles;
                o.sb->work_next = 0;
                o.sb->work_next2 = 0;
            }
        }
    }
    __syncthreads();
    KT_MARK(K_ROUTE_GATHER, 4);
    const int r = r_sh;
    for (int i = p + (int)gridDim.x * tid; i < o.max_tiles; i += (int)gridDim.x * (int)blockDim.x) o.tile_ready[i] = 0u;
    const size_t tab_rows = (size_t)P_tab + NT_MAX;
    if (r >= 0) {
#pragma unroll
        for (int i = 0; i < PASSES; ++i) {
            const int cc = i * (int)blockDim.x + tid;
            if (cc < nc) store_chunk(q[i], cc, r, d, tab_rows, xq, xs);
        }
        pad_scale_rows(r, d, I, tab_rows, xs, hs, tid);
    }
    KT_MARK(K_ROUTE_GATHER, 2);
}

// Whether pick j of token t (id e) is valid: e in [0, E) and not an id of the
// token's earlier picks, which are read all at once (k <= 16), not one
// round trip after another.
__device__ __forceinline__ bool pick_valid(const int32_t* ids, int t, int j, int k, int e, int E) {
    if (e < 0 || e >= E) return false;
    int prev[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) prev[q] = q < j ? ld_dep(ids + (size_t)t * k + q) : -1;
    bool ok = true;
#pragma unroll
    for (int q = 0; q < 16; ++q) ok = ok && prev[q] != e;
    return ok;
}

// Sort of more than 128 picks over many CTAs, for the gather below.
//   k_count: every pick p = t*k + j whose id e is in [0, E) and not repeated
//   by an earlier pick of token t counts itself into cnt[e] (warp-aggregated
//   global atomics; the others latch MOE_ERR_BAD_IDS); the last CTA to finish
//   (a counter in the status block) turns the counts into segment offsets
//   off[e] and tile offsets (one warp: two exclusive scans), writes every tile entry
//   (expert e, first position off[e] + i nt, min(nt, cnt[e] - i nt) picks),
//   the call's counts, clears cnt, the placement counters cnt2 and tile_ready
//   for the call, and resets its own counter.
//   k_gather_tok: one CTA a token: its row quantised once, then each valid
//   pick takes the position off[e] + atomicAdd(cnt2[e], 1) and gets a copy.
// The order of the picks inside a segment is the order the atomics came in:
// each pick is an independent column of the expert GEMMs, so the results do
// not depend on it; tiles and counts do not either.
constexpr int CNT_THREADS = 1024;
struct CountOut {
    int32_t* cnt;
    int32_t* off;
    int32_t* cnt2;
    SortOut o;
};

__global__ void __launch_bounds__(CNT_THREADS) k_count(const int32_t* ids, int S, int E, int k, CountOut c) {
    __shared__ int32_t s_cnt[SORT_CNT_MAX_E], s_off[SORT_CNT_MAX_E + 1], s_toff[SORT_CNT_MAX_E + 1];
    __shared__ int32_t last;
    KT_MARK(K_SORT, 0);
    pdl_wait();
    pdl_trigger();   // the call's first kernel for moe_experts: k_gather_tok reads x before its wait
    KT_MARK(K_SORT, 1);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = S * k, p = blockIdx.x * CNT_THREADS + tid;
    const SortOut& o = c.o;
    int e = -1;
    bool ok = false;
    if (p < P) {
        const int t = p / k, j = p - t * k;
        e = ld_dep(ids + p);
        ok = pick_valid(ids, t, j, k, e, E);
        if (!ok) latch_status(o.sb, MOE_ERR_BAD_IDS, p);
    }
    const uint32_t grp = __match_any_sync(0xffffffffu, ok ? e : -1 - lane);
    if (ok && lane == __ffs(grp) - 1) atomicAdd(&c.cnt[e], __popc(grp));
    __threadfence();
    __syncthreads();
    if (tid == 0) last = atomicAdd(&o.sb->count_done, 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    const int nt = o.nt;
    for (int i = tid; i < E; i += CNT_THREADS) {
        s_cnt[i] = ld_dep(c.cnt + i);
        c.cnt[i] = 0;    // clear for the next call
        c.cnt2[i] = 0;   // placement counters of this call
    }
    for (int i = tid; i < o.max_tiles; i += CNT_THREADS) o.tile_ready[i] = 0u;
    __syncthreads();
    if (warp == 0) {
        // lane l scans experts [l*per, (l+1)*per); two exclusive scans at once
        const int per = (E + 31) / 32;
        const int e0 = lane * per, e1 = min(E, e0 + per);
        int sp = 0, st = 0;
        for (int ee = e0; ee < e1; ++ee) {
            sp += s_cnt[ee];
            st += (s_cnt[ee] + nt - 1) / nt;
        }
        int ip = sp, it = st;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, ip, m);
            const int b = __shfl_up_sync(0xffffffffu, it, m);
            if (lane >= m) {
                ip += a;
                it += b;
            }
        }
        int rp = ip - sp, rt = it - st;
        for (int ee = e0; ee < e1; ++ee) {
            s_off[ee] = rp;
            s_toff[ee] = rt;
            rp += s_cnt[ee];
            rt += (s_cnt[ee] + nt - 1) / nt;
        }
        if (lane == 31) {
            o.sb->n_picks = ip;
            o.sb->n_tiles = it;
            o.sb->work_next = 0;
            o.sb->work_next2 = 0;
            o.sb->count_done = 0;
        }
    }
    __syncthreads();
    for (int ee = tid; ee < E; ee += CNT_THREADS) {
        c.off[ee] = s_off[ee];
        const int n = s_cnt[ee];
        for (int i = 0; i * nt < n; ++i) {
            Tile tl;
            tl.e = ee;
            tl.p0 = s_off[ee] + i * nt;
            tl.n = min(nt, n - i * nt);
            tl.pad = 0;
            o.tiles[s_toff[ee] + i] = tl;
        }
    }
    KT_MARK(K_SORT, 2);
}

// grid (S), a thread per GATHER_PASSES chunks of 8 elements of a row (see
// k_count).  The row's loads go out before the wait and are quantised only
// after the placement (the token's ids read once, each pick's position an
// L2 round trip), so that the two latencies overlap.
__global__ void __launch_bounds__(1024) k_gather_tok(const __nv_bfloat16* __restrict__ x, const int32_t* ids, int k,
                                                    int E, int d, int I, int P, CountOut c,
                                                    uint8_t* __restrict__ xq, uint8_t* __restrict__ xs,
                                                    uint8_t* __restrict__ hs) {
    __shared__ int32_t r_sh[16], id_sh[16];
    KT_MARK(K_GATHER, 0);
    pdl_trigger();
    const int t = blockIdx.x, tid = threadIdx.x;
    const uint4* in = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    const int nc = d / 8;
    uint4 raw[GATHER_PASSES];
#pragma unroll
    for (int i = 0; i < GATHER_PASSES; ++i) {
        const int cc = i * (int)blockDim.x + tid;
        raw[i] = cc < nc ? __ldg(in + cc) : make_uint4(0, 0, 0, 0);
    }
    pdl_wait();
    KT_MARK(K_GATHER, 1);
    if (tid < k) id_sh[tid] = ld_dep(ids + (size_t)t * k + tid);
    __syncthreads();
    if (tid < k) {
        // a pick is placed when its id is in [0, E) and not an id of an
        // earlier pick of the token (k_count latched the others)
        const int e = id_sh[tid];
        bool ok = e >= 0 && e < E;
        for (int q2 = 0; q2 < tid; ++q2) ok = ok && id_sh[q2] != e;
        const int r = ok ? ld_dep(c.off + e) + atomicAdd(&c.cnt2[e], 1) : -1;
        c.o.pos[(size_t)t * k + tid] = r;
        r_sh[tid] = r;
    }
    QuantChunk q[GATHER_PASSES];
#pragma unroll
    for (int i = 0; i < GATHER_PASSES; ++i) q[i] = quantize_vals(raw[i]);
    __syncthreads();
    const size_t tab_rows = (size_t)P + NT_MAX;
    for (int j = 0; j < k; ++j) {
        const int r = r_sh[j];
        if (r < 0) continue;
#pragma unroll
        for (int i = 0; i < GATHER_PASSES; ++i) {
            const int cc = i * (int)blockDim.x + tid;
            if (cc < nc) store_chunk(q[i], cc, r, d, tab_rows, xq, xs);
        }
        pad_scale_rows(r, d, I, tab_rows, xs, hs, tid);
    }
    KT_MARK(K_GATHER, 2);
}

}  // namespace

static SortOut sort_out(const WsLayout& L, char* ws) {
    SortOut o;
    o.pos = reinterpret_cast<int32_t*>(ws + L.pos);
    o.tiles = reinterpret_cast<Tile*>(ws + L.tiles);
    o.tile_ready = reinterpret_cast<uint32_t*>(ws + L.tile_ready);
    o.max_tiles = L.max_tiles;
    o.nt = L.nt;
    o.sb = reinterpret_cast<StatusBlock*>(ws + L.status);
    return o;
}

static CountOut count_out(const WsLayout& L, char* ws) {
    CountOut c;
    int32_t* base = reinterpret_cast<int32_t*>(ws + L.sortcnt);
    c.cnt = base;
    c.off = base + SORT_CNT_MAX_E;
    c.cnt2 = base + 2 * SORT_CNT_MAX_E;
    c.o = sort_out(L, ws);
    return c;
}


// The fused top-k + sort + gather selects again in every CTA; above this
// many picks (as many CTAs) the top-k kernel selects once and the fused
// kernel only sorts and gathers.
constexpr int RG_MAX_SELECT_PICKS = 128;

bool topk_sort_fits(const moe_shape& s) {
    // a CTA's threads hold the row's chunks (RG_PASSES a thread), its warps
    // one or two tokens each
    return s.S <= RG_TOKENS_PER_WARP * (RG_THREADS / 32) && s.S * s.k <= 1024 &&
           s.d / 8 <= RG_PASSES * RG_THREADS;
}

bool route_gather_selects(const moe_shape& s) { return topk_sort_fits(s) && s.S * s.k <= RG_MAX_SELECT_PICKS; }

// a thread per chunk of 8 elements of a row, and a warp for every two tokens
// (at least), within RG_THREADS
static int route_gather_threads(const moe_shape& s) {
    const int rows = (s.d / 8 + 31) / 32 * 32;
    const int tok = 32 * ((s.S + RG_TOKENS_PER_WARP - 1) / RG_TOKENS_PER_WARP);
    return std::min(RG_THREADS, std::max(rows, tok));
}

template <int MAXE, bool FROM_IDS>
static cudaError_t launch_rg(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st, bool x_after_wait) {
    const int threads = route_gather_threads(s);
    const int P = s.S * s.k;
    size_t smem = (size_t)(P + s.E) * sizeof(int32_t) +
                  (FROM_IDS ? (size_t)P * sizeof(int32_t)
                            : (size_t)std::min(s.S, threads / 32) * 32 * MAXE * sizeof(float));
    // one CTA an SM when the picks fit one wave: two CTAs on an SM finished
    // their selection up to 1.3 us apart, and the slowest CTA decides when the
    // expert kernel's wait returns (S = 8: the step 52.3 against 53.0 us).  The
    // shared memory asked for is what makes a second CTA not fit.
    if (P <= num_sms() && smem < RG_ONE_PER_SM_SMEM) smem = RG_ONE_PER_SM_SMEM;
    const int passes = (s.d / 8 + threads - 1) / threads;   // 1, 2 or 4 (d <= 16384)
    auto kern = passes == 1 ? k_route_gather<MAXE, 1, FROM_IDS>
                            : passes == 2 ? k_route_gather<MAXE, 2, FROM_IDS> : k_route_gather<MAXE, 4, FROM_IDS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    char* ws = p.ws;
    timing_begin(FROM_IDS ? K_GATHER : K_ROUTE_GATHER, st);
    e = launch_pdl(kern, dim3(P), dim3(threads), smem, st, reinterpret_cast<const float*>(ws + L.logits), p.bias,
                   p.x, s.S, s.E, s.k, s.d, s.I, L.max_picks, p.ids, p.weights, sort_out(L, ws),
                   reinterpret_cast<uint8_t*>(ws + L.xq), reinterpret_cast<uint8_t*>(ws + L.xs),
                   reinterpret_cast<uint8_t*>(ws + L.hs), x_after_wait ? 1 : 0);
    timing_end(st);
    return e;
}

cudaError_t launch_topk_sort_gather(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st,
                                    bool x_after_wait) {
    KT_BIND();
    if (!route_gather_selects(s)) {
        cudaError_t e = launch_topk(s, L, p, st);
        if (e != cudaSuccess) return e;
        return launch_rg<8, true>(s, L, p, st, x_after_wait);
    }
    return s.E <= 256 ? launch_rg<8, false>(s, L, p, st, x_after_wait) : launch_rg<16, false>(s, L, p, st, x_after_wait);
}

cudaError_t launch_sort_gather(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st,
                               bool x_after_wait) {
    KT_BIND();
    const int P = s.S * s.k;
    if (P > SMALL_SORT_PICKS) {
        // k_gather_tok reads the rows before its wait even when an earlier
        // kernel of the call wrote them: k_count lets it start only past its
        // own wait, when every kernel before k_count has completed
        const CountOut c = count_out(L, p.ws);
        timing_begin(K_SORT, st);
        cudaError_t e = launch_pdl(k_count, dim3((P + CNT_THREADS - 1) / CNT_THREADS), dim3(CNT_THREADS), 0, st,
                                   (const int32_t*)p.ids, s.S, s.E, s.k, c);
        timing_end(st);
        if (e != cudaSuccess) return e;
        // GATHER_PASSES chunks a thread: several tokens' CTAs an SM
        const int threads = std::min(1024, ((s.d / 8 + GATHER_PASSES - 1) / GATHER_PASSES + 31) / 32 * 32);
        timing_begin(K_GATHER, st);
        e = launch_pdl(k_gather_tok, dim3(s.S), dim3(threads), 0, st, p.x, (const int32_t*)p.ids, s.k, s.E, s.d, s.I,
                       L.max_picks, c, reinterpret_cast<uint8_t*>(p.ws + L.xq), reinterpret_cast<uint8_t*>(p.ws + L.xs),
                       reinterpret_cast<uint8_t*>(p.ws + L.hs));
        timing_end(st);
        return e;
    }
    // up to 128 picks: the fused kernel reads the ids, checks them, places
    // every pick and gathers its row in one launch (after its wait when an
    // earlier kernel of the call wrote the rows: the top-k kernel before it
    // lets it start before that kernel's own wait)
    return launch_rg<8, true>(s, L, p, st, x_after_wait);
}

}  // namespace moe
