// MXFP4 expert GEMMs on the 5th-generation tensor cores: one persistent kernel
// runs every gate_up unit and then every down unit of the call.
//
// vllm.models.muse_spark.amd.mono.kernels.k3, stages C, D: "gate_up / down of
// the local experts: MXFP4 weights ..., decoded in registers, bf16 MFMA";
// fp4_mma: "Chunk c (256 K) of a 16-row MXFP4 group: 8 MFMA steps"; mx_chunk:
// rows x K chunk of an MXFP4 weight and its e8m0 scales; task_ring: compute
// the current task with the next tasks' loads in flight.
// vllm.models.kimi_k3.amd.specialized_decode.mono.layer: the static weights
// stream while earlier stages settle, weights issued before the first wait.
//
// GB300 design (one CTA per SM, 14 warps):
//   warp 0      producer: TMA of the weight tile (128 rows x 128 K of packed
//               e2m1, 8 KB) and of the token tile (N picks x 128 K bf16) into a
//               ring of NS shared-memory stages; the 128 x 4 e8m0 bytes of the
//               stage by cp.async, completing on the same mbarrier.
//   warp 1      MMA issuer (one thread): tcgen05.mma kind::f16, M = 128, N =
//               picks, K = 16, A = decoded weights in TMEM, B = token tile in
//               shared memory (128-byte swizzle), fp32 accumulators in TMEM.
//   warps 6-13  decoders (two groups of four, alternate stages): each thread
//               owns one weight row, reads its 64 bytes (128 e2m1) from shared
//               memory, turns them into bf16 with the block scale applied and
//               stores them into a TMEM A stage (tcgen05.st).
//   warps 2-5   epilogue: accumulators -> h = silu(g) * u (bf16) for gate_up,
//               y (fp32) for down.
// Work units, in a static round-robin over the CTAs: gate_up units first
// (64 gate rows stacked on the matching 64 up rows = one M = 128 operand), then
// down units (128 rows of w2).  A down unit needs the h rows of its tile: its
// producer issues the weight loads first and waits (bounded) on the tile's
// counter, which every finished gate_up unit of the tile increments.
//
// Decode: an e2m1 code (s, e1, e0, m) is placed in a bf16 as sign bit 15 and
// bits 8..6 = (e1, e0, m): that bf16 equals the e2m1 value times 2^-126
// (exact, subnormal for e = 0), so one bf16x2 multiply by 2^(b - 1) applies
// the e8m0 scale 2^(b - 127) exactly for b in 0..128.  Two codes 16 bits apart
// in a 32-bit word share one integer multiply (x 0x1040 or x 0x104) and one
// mask.  The K order inside every group of 8 elements is therefore
// (0, 4, 1, 5, 2, 6, 3, 7); the gathered tokens and h are stored in the same
// order, so the MMA sums matching pairs.
#include "moe_internal.cuh"
#include "tc_ptx.cuh"

#include <cudaTypedefs.h>

namespace moe {

namespace {

constexpr int KC = 128;                      // K elements per stage
constexpr int AROWS = 128;                   // MMA M
constexpr int A_BYTES = AROWS * KC / 2;      // packed e2m1 per stage
constexpr int SC_BYTES = AROWS * 4;          // e8m0 bytes per stage
constexpr int NS = 12;                       // shared-memory stages
constexpr int NA = 4;                        // TMEM A stages
constexpr int A_COLS = KC / 2;               // TMEM columns of one A stage
constexpr int A_COL0 = 256;                  // first A-stage column
constexpr int TMEM_COLS = 512;
constexpr int NUM_WARPS = 14;
constexpr int NUM_THREADS = 32 * NUM_WARPS;
constexpr int EPI_WARP0 = 2, DEC_WARP0 = 6;
constexpr uint64_t WAIT_NS = 2000000000ull;  // bounded waits: 2 s

template <int N>
struct Cfg {
    static constexpr int B_BOX = N * 128;                      // N rows x 64 bf16
    static constexpr int B_BYTES = 2 * B_BOX;                  // KC = 128 bf16 per row
    static constexpr int STAGE = ((A_BYTES + B_BYTES + SC_BYTES) + 1023) / 1024 * 1024;
    static constexpr int XCH_STRIDE = N + 1;
    static constexpr int SMEM = 1024 /*align slack*/ + NS * STAGE + 64 * XCH_STRIDE * 4 + 1024 /*barriers*/;
    static_assert(N % 16 == 0 && N >= 16 && N <= 128, "MMA N");
    static_assert(2 * N <= A_COL0, "accumulators below the A stages");
};

struct Args {
    const Tile* tiles;
    StatusBlock* sb;
    const uint8_t* w13s;
    const uint8_t* w2s;
    __nv_bfloat16* h;
    float* y;
    uint32_t* tile_ready;
    int d, I;
};

struct Unit {
    int down;        // 0: gate_up, 1: down
    int tile, mb;    // tile index and row block
    int e, p0, n;
    int chunks;
};

__device__ __forceinline__ Unit get_unit(int u, int U1, const Args& a) {
    Unit U;
    const int mb1 = a.I / 64, mb2 = a.d / AROWS;
    if (u < U1) {
        U.down = 0;
        U.tile = u / mb1;
        U.mb = u % mb1;
        U.chunks = a.d / KC;
    } else {
        const int v = u - U1;
        U.down = 1;
        U.tile = v / mb2;
        U.mb = v % mb2;
        U.chunks = a.I / KC;
    }
    const Tile t = a.tiles[U.tile];
    U.e = t.e;
    U.p0 = t.p0;
    U.n = t.n;
    return U;
}

// global row (in the [E * rows, K/2] view) of weight row r (0..127) of unit U
__device__ __forceinline__ int weight_row(const Unit& U, int r, const Args& a) {
    if (!U.down) {
        const int base = U.e * 2 * a.I + U.mb * 64;
        return r < 64 ? base + r : base + a.I + (r - 64);
    }
    return U.e * a.d + U.mb * AROWS + r;
}

// e2m1 x 32 (16 bytes) + e8m0 byte -> 16 bf16x2 words in MMA K order
__device__ __forceinline__ void decode_block(const uint4 q, uint32_t sbyte, uint32_t* out, StatusBlock* sb) {
    uint32_t mult;
    if (sbyte <= 128u) {
        mult = (sbyte + 126u) << 7;          // bf16 bits of 2^(b - 1)
    } else {
        latch_status(sb, MOE_ERR_BAD_SCALE, (int)sbyte);
        mult = 0u;
    }
    mult |= mult << 16;
    const __nv_bfloat162 m2 = *reinterpret_cast<const __nv_bfloat162*>(&mult);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t x = w[i], x8 = x >> 8;
        uint32_t o[4];
        o[0] = ((x & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;    // codes 0 and 4 of the word
        o[1] = ((x & 0x00F000F0u) * 0x104u) & 0x81C081C0u;     // codes 1 and 5
        o[2] = ((x8 & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;   // codes 2 and 6
        o[3] = ((x8 & 0x00F000F0u) * 0x104u) & 0x81C081C0u;   // codes 3 and 7
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&o[j]);
            v = __hmul2(v, m2);
            out[4 * i + j] = *reinterpret_cast<const uint32_t*>(&v);
        }
    }
}

// position of K-element i in the MMA order of its group of 8
__device__ __forceinline__ int kperm(int i) {
    const int e = i & 7;
    return (i & ~7) | (e < 4 ? 2 * e : 2 * (e - 4) + 1);
}

template <int N>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_experts_tc(const __grid_constant__ CUtensorMap tm_w13, const __grid_constant__ CUtensorMap tm_w2,
                 const __grid_constant__ CUtensorMap tm_xg, const __grid_constant__ CUtensorMap tm_h,
                 const Args a) {
    using C = Cfg<N>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    float* xch = reinterpret_cast<float*>(smem + NS * C::STAGE);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NS * C::STAGE + 64 * C::XCH_STRIDE * 4);
    uint64_t* full = bars;                  // [NS]
    uint64_t* empty = full + NS;            // [NS]
    uint64_t* a_full = empty + NS;          // [NA]
    uint64_t* a_empty = a_full + NA;        // [NA]
    uint64_t* acc_full = a_empty + NA;      // [2]
    uint64_t* acc_empty = acc_full + 2;     // [2]
    uint64_t* fin = acc_empty + 2;          // [1]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(fin + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* epi_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    StatusBlock* sb = a.sb;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            ptx::mbar_init(&full[i], 1 + 32);   // producer expect_tx + 32 cp.async arrivals
            ptx::mbar_init(&empty[i], 4 + 1);   // 4 decoder warps + MMA commit
        }
        for (int i = 0; i < NA; ++i) {
            ptx::mbar_init(&a_full[i], 4);
            ptx::mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&acc_full[i], 1);
            ptx::mbar_init(&acc_empty[i], 4);
        }
        ptx::mbar_init(fin, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(tmem_holder, TMEM_COLS);
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tm_w13);
        ptx::prefetch_tensormap(&tm_w2);
        ptx::prefetch_tensormap(&tm_xg);
        ptx::prefetch_tensormap(&tm_h);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    const int n_tiles = sb->n_tiles;
    const int U1 = n_tiles * (a.I / 64);
    const int total = U1 + n_tiles * (a.d / AROWS);
    const int mb1 = a.I / 64;

    auto fail = [&](int site) {
        latch_status(sb, MOE_ERR_TIMEOUT, site);
        *abort_flag = 1;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const uint64_t pol_w = ptx::policy_evict_first();
        const uint64_t pol_x = ptx::policy_evict_last();
        int seq = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
            const Unit U = get_unit(u, U1, a);
            const CUtensorMap* tmB = U.down ? &tm_h : &tm_xg;
            bool b_ok = !U.down;
            int pend = seq;   // first stage sequence number whose B is not issued yet
            for (int c = 0; c < U.chunks; ++c, ++seq) {
                const int s = seq % NS;
                if (!ptx::mbar_wait_warp(&empty[s], ((seq / NS) & 1) ^ 1, abort_flag, WAIT_NS)) {
                    if (lane == 0) fail(1);
                    ok = false;
                    break;
                }
                uint8_t* st = stages + s * C::STAGE;
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(&full[s], A_BYTES + C::B_BYTES);
                    if (!U.down) {
                        const int r0 = U.e * 2 * a.I + U.mb * 64;
                        ptx::tma_load_2d(st, &tm_w13, c * (KC / 2), r0, &full[s], pol_w);
                        ptx::tma_load_2d(st + A_BYTES / 2, &tm_w13, c * (KC / 2), r0 + a.I, &full[s], pol_w);
                    } else {
                        ptx::tma_load_2d(st, &tm_w2, c * (KC / 2), U.e * a.d + U.mb * AROWS, &full[s], pol_w);
                    }
                }
                // e8m0 bytes of this stage: rows lane, lane+32, lane+64, lane+96
                {
                    const uint8_t* sbase = U.down ? a.w2s : a.w13s;
                    const int kb = U.down ? a.I / 32 : a.d / 32;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int r = lane + 32 * j;
                        ptx::cp_async_4(st + A_BYTES + C::B_BYTES + 4 * r,
                                        sbase + (size_t)weight_row(U, r, a) * kb + 4 * c);
                    }
                    ptx::cp_async_mbar_arrive_noinc(&full[s]);
                }
                if (!b_ok) {
                    // a down unit: its h rows must be complete; check without
                    // blocking while weight stages are still being issued
                    uint32_t ready = 0;
                    if (lane == 0) ready = ptx::ld_acquire_gpu(&a.tile_ready[U.tile]) >= (uint32_t)mb1;
                    ready = __shfl_sync(0xffffffffu, ready, 0);
                    if (!ready && (c == U.chunks - 1 || seq - pend + 1 >= NS / 2)) {
                        // every stage we may fill without it is filled: wait
                        if (lane == 0) {
                            const uint64_t t0 = ptx::globaltimer();
                            uint32_t it = 0;
                            while (ptx::ld_acquire_gpu(&a.tile_ready[U.tile]) < (uint32_t)mb1) {
                                __nanosleep(64);
                                if ((++it & 63u) == 0u && (*abort_flag || ptx::globaltimer() - t0 > WAIT_NS)) {
                                    fail(2);
                                    break;
                                }
                            }
                            ready = *abort_flag ? 0u : 1u;
                        }
                        ready = __shfl_sync(0xffffffffu, ready, 0);
                        if (!ready) {
                            ok = false;
                            ++seq;
                            break;
                        }
                    }
                    if (ready) {
                        b_ok = true;
                        if (lane == 0) {
                            ptx::fence_proxy_async_global();
                            for (int q = pend; q < seq; ++q) {   // earlier stages of this unit
                                const int cc = c - (seq - q);
                                uint8_t* sq = stages + (q % NS) * C::STAGE + A_BYTES;
                                ptx::tma_load_2d(sq, tmB, cc * KC, U.p0, &full[q % NS], pol_x);
                                ptx::tma_load_2d(sq + C::B_BOX, tmB, cc * KC + 64, U.p0, &full[q % NS], pol_x);
                            }
                        }
                    }
                }
                if (b_ok) {
                    if (lane == 0) {
                        ptx::tma_load_2d(st + A_BYTES, tmB, c * KC, U.p0, &full[s], pol_x);
                        ptx::tma_load_2d(st + A_BYTES + C::B_BOX, tmB, c * KC + 64, U.p0, &full[s], pol_x);
                    }
                    pend = seq + 1;
                }
                __syncwarp();
            }
        }
        ptx::cp_async_wait_all();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(AROWS, N);
            int seq = 0, uc = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x, ++uc) {
                const Unit U = get_unit(u, U1, a);
                const int ab = uc & 1;
                if (!ptx::mbar_wait(&acc_empty[ab], ((uc >> 1) & 1) ^ 1, abort_flag, WAIT_NS)) {
                    fail(3);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + ab * N;
                for (int c = 0; c < U.chunks; ++c, ++seq) {
                    const int s = seq % NS, as = seq % NA;
                    if (!ptx::mbar_wait(&full[s], (seq / NS) & 1, abort_flag, WAIT_NS) ||
                        !ptx::mbar_wait(&a_full[as], (seq / NA) & 1, abort_flag, WAIT_NS)) {
                        fail(4);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t b0 = ptx::smem_u32(stages + s * C::STAGE + A_BYTES);
                    const uint32_t a0 = tmem + A_COL0 + as * A_COLS;
#pragma unroll
                    for (int kk = 0; kk < KC / 16; ++kk) {
                        const uint64_t bd = ptx::smem_desc_sw128(b0 + (kk >> 2) * C::B_BOX + (kk & 3) * 32);
                        ptx::mma_bf16_ts(d_tmem, a0 + kk * 8, bd, idesc, (c | kk) != 0);
                    }
                    ptx::mma_commit(&a_empty[as]);
                    ptx::mma_commit(&empty[s]);
                }
                if (!ok) break;
                ptx::mma_commit(&acc_full[ab]);
            }
            // every MMA issued above has completed before TMEM is released
            ptx::mma_commit(fin);
            ptx::mbar_wait(fin, 0, abort_flag, WAIT_NS);
        }
        __syncwarp();
    } else if (warp >= DEC_WARP0) {
        // ------------------------------------------------------------ decoders
        const int dw = warp - DEC_WARP0;
        const int g = dw >> 2;            // stage parity handled by this group
        const int qd = warp & 3;          // TMEM lane quarter of this warp
        const int r = 32 * qd + lane;     // weight row of this thread
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        int seq = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
            const Unit U = get_unit(u, U1, a);
            for (int c = 0; c < U.chunks; ++c, ++seq) {
                if ((seq & 1) != g) continue;
                const int s = seq % NS, as = seq % NA;
                if (!ptx::mbar_wait_warp(&full[s], (seq / NS) & 1, abort_flag, WAIT_NS)) {
                    if (lane == 0) fail(5);
                    ok = false;
                    break;
                }
                const uint8_t* st = stages + s * C::STAGE;
                uint4 q[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    q[j] = *reinterpret_cast<const uint4*>(st + r * 64 + ((j ^ ((r >> 1) & 3)) << 4));
                const uint32_t sc = *reinterpret_cast<const uint32_t*>(st + A_BYTES + C::B_BYTES + 4 * r);
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&empty[s]);
                if (!ptx::mbar_wait_warp(&a_empty[as], ((seq / NA) & 1) ^ 1, abort_flag, WAIT_NS)) {
                    if (lane == 0) fail(6);
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t ta = tmem + lane_base + A_COL0 + as * A_COLS;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t v[16];
                    decode_block(q[j], (sc >> (8 * j)) & 0xFFu, v, sb);
                    ptx::tmem_st16(ta + 16 * j, v);
                }
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&a_full[as]);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int qd = warp & 3;
        const int r = 32 * qd + lane;
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        int uc = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x, ++uc) {
            const Unit U = get_unit(u, U1, a);
            const int ab = uc & 1;
            // the four epilogue warps take one decision before their named
            // barriers: carry on, or leave together
            if (!ptx::mbar_wait_warp(&acc_full[ab], (uc >> 1) & 1, abort_flag, WAIT_NS) && lane == 0) fail(7);
            ptx::named_bar_sync(1, 128);
            if (threadIdx.x == EPI_WARP0 * 32) *epi_flag = *abort_flag;
            ptx::named_bar_sync(1, 128);
            if (*epi_flag) break;
            ptx::tc_fence_after();
            uint32_t v[N];
#pragma unroll
            for (int j = 0; j < N / 16; ++j) ptx::tmem_ld16(tmem + lane_base + ab * N + 16 * j, v + 16 * j);
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&acc_empty[ab]);
            if (!U.down) {
                // lanes 0..63: gate of rows mb*64 + r; lanes 64..127: up of the same rows
                if (r >= 64) {
#pragma unroll
                    for (int n = 0; n < N; ++n) xch[(r - 64) * C::XCH_STRIDE + n] = __uint_as_float(v[n]);
                }
                ptx::named_bar_sync(1, 128);
                if (r < 64) {
                    const int i = U.mb * 64 + r;
                    const int col = kperm(i);
#pragma unroll
                    for (int n = 0; n < N; ++n) {
                        if (n < U.n) {
                            const float gv = __uint_as_float(v[n]);
                            const float uv = xch[r * C::XCH_STRIDE + n];
                            const float hv = gv / (1.0f + __expf(-gv)) * uv;
                            a.h[(size_t)(U.p0 + n) * a.I + col] = __float2bfloat16_rn(hv);
                        }
                    }
                    ptx::fence_proxy_async_global();
                }
                ptx::named_bar_sync(1, 128);
                if (warp == EPI_WARP0 && lane == 0) {
                    __threadfence();
                    ptx::red_release_gpu_add(&a.tile_ready[U.tile], 1u);
                }
            } else {
                const int m = U.mb * AROWS + r;
#pragma unroll
                for (int n = 0; n < N; ++n)
                    if (n < U.n) a.y[(size_t)(U.p0 + n) * a.d + m] = __uint_as_float(v[n]);
            }
        }
    }

    __syncthreads();
    if (*abort_flag) {
        // let copies still in flight into this CTA's shared memory land
        const uint64_t t0 = ptx::globaltimer();
        while (ptx::globaltimer() - t0 < 200000ull) {
        }
    }
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------------------
// host side: tensor maps and launch
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
    static int n[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!n[dev]) cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
    return n[dev];
}

template <int N>
cudaError_t launch_tc(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    using C = Cfg<N>;
    CUtensorMap tm_w13, tm_w2, tm_xg, tm_h;
    const uint64_t P = (uint64_t)L.max_picks;
    if (!make_map_2d(&tm_w13, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.w13, s.d / 2, (uint64_t)s.E * 2 * s.I, s.d / 2,
                     KC / 2, 64, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map_2d(&tm_w2, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.w2, s.I / 2, (uint64_t)s.E * s.d, s.I / 2, KC / 2,
                     AROWS, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map_2d(&tm_xg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.ws + L.xg, s.d, P, (uint64_t)s.d * 2, 64, N,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&tm_h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.ws + L.h, s.I, P, (uint64_t)s.I * 2, 64, N,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_experts_tc<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    Args a;
    a.tiles = reinterpret_cast<const Tile*>(p.ws + L.tiles);
    a.sb = reinterpret_cast<StatusBlock*>(p.ws + L.status);
    a.w13s = p.w13s;
    a.w2s = p.w2s;
    a.h = reinterpret_cast<__nv_bfloat16*>(p.ws + L.h);
    a.y = reinterpret_cast<float*>(p.ws + L.y);
    a.tile_ready = reinterpret_cast<uint32_t*>(p.ws + L.tile_ready);
    a.d = s.d;
    a.I = s.I;
    k_experts_tc<N><<<num_sms(), NUM_THREADS, C::SMEM, st>>>(tm_w13, tm_w2, tm_xg, tm_h, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_experts(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    timing_begin(K_EXPERTS, st);
    cudaError_t e = launch_tc<NT>(s, L, p, st);
    timing_end(st);
    return e;
}

}  // namespace moe
