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
// GB300 design (one persistent CTA per SM, 24 warps):
//   warp 0      weight producer: per 256-K stage of a unit, the weight tile
//               (128 rows x 256 K of packed e2m1, 16 KB; gate and up rows in
//               one 4-D box) and its e8m0 bytes into a ring of weight stages,
//               and an L2 prefetch of the weight tile PF stages ahead.  Under
//               full load the HBM latency is several microseconds, more than
//               the shared memory can cover at the bandwidth wanted; the L2
//               prefetch keeps the rest of the bytes in flight.
//   warp 7      token producer: the token tile (N picks x 256 K bf16, one 3-D
//               box of four 128-byte-swizzled slabs) into a ring of its own;
//               for a down unit it first waits (bounded) for the tile's h.
//   warps 1-2   MMA issuers (lane 0 of each): tcgen05.mma kind::f16, M = 128,
//               N = picks, K = 16, A = decoded weights in TMEM, B = token tile
//               in shared memory.  Issuer m takes the 128-K sub-chunks q = m
//               mod 2 of every unit into an fp32 accumulator of its own (double
//               buffered); the epilogue sums the two.  One thread issues one
//               MMA every ~50 cycles and each wait on an mbarrier drains its
//               MMAs, so at N = 16 one issuer caps the tensor rate below what
//               the weight stream needs; two issuers overlap.  Each TMEM A stage
//               belongs to one issuer (stage q mod NA has the parity of q), so
//               all uses of a stage complete in that issuer's order and no
//               waiter is ever two phases ahead of an mbarrier.
//   warps 8-23  decoders (groups of four warps; group g takes the 128-K
//               sub-chunks g, g+G, ...): each thread owns one weight row, reads
//               its 64 bytes (128 e2m1) and scale byte from shared memory
//               (releasing the weight stage at once), turns them into bf16 with
//               the block scale applied and stores them into a TMEM A stage.
//   warps 3-6   epilogue: accumulators -> h = silu(g) * u (bf16) for gate_up,
//               y (fp32) for down.
// Work units, in a static round-robin over the CTAs: gate_up units first
// (64 gate rows stacked on the matching 64 up rows = one M = 128 operand), then
// down units (128 rows of w2).  A down unit needs the h rows of its tile: the
// counter of the tile, which every finished gate_up unit of it increments.
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

constexpr int KC = 128;                      // K elements of one decode sub-chunk (one TMEM A stage)
constexpr int KS = 256;                      // K elements of one shared-memory stage (two sub-chunks)
constexpr int AROWS = 128;                   // MMA M
constexpr int A_SUB = AROWS * KC / 2;        // packed e2m1 of one sub-chunk: 8 KB
constexpr int A_BYTES = 2 * A_SUB;           // of one stage: 16 KB
#ifndef MOE_TC_TOKEN_STAGES
#define MOE_TC_TOKEN_STAGES 4
#endif
#ifndef MOE_TC_DEC_GROUPS
#define MOE_TC_DEC_GROUPS 4
#endif
#ifndef MOE_TC_PREFETCH
#define MOE_TC_PREFETCH 16
#endif
constexpr int NSB = MOE_TC_TOKEN_STAGES;       // token-tile stages
constexpr int DEC_GROUPS = MOE_TC_DEC_GROUPS;  // decoder groups of 4 warps
constexpr int PF = MOE_TC_PREFETCH;            // L2 prefetch distance in weight stages
constexpr int A_COLS = KC / 2;               // TMEM columns of one A stage
constexpr int TMEM_COLS = 512;
constexpr int NMMA = 2;                      // MMA-issuing warps (one thread each)
constexpr int MMA_WARP0 = 1, EPI_WARP0 = 3, TOK_WARP = 7, DEC_WARP0 = 8;
static_assert(MOE_TC_DEC_GROUPS % NMMA == 0, "decoder group g feeds issuer g mod NMMA");
constexpr int NUM_WARPS = DEC_WARP0 + 4 * DEC_GROUPS;
constexpr int NUM_THREADS = 32 * NUM_WARPS;
constexpr int UR = 32;                       // unit ring entries
constexpr uint64_t WAIT_NS = 2000000000ull;  // bounded waits: 2 s

// STMA: the e8m0 bytes come by TMA, 16 bytes (512 K) of each row per stage,
// when the scale rows are 16-byte aligned (K % 512 == 0); otherwise by 4-byte
// cp.async, 8 bytes (256 K) of each row per stage.
template <int N, bool STMA>
struct Cfg {
    static constexpr int B_BOX = N * 128;                      // N rows x 64 bf16 (one slab)
    static constexpr int B_BYTES = 4 * B_BOX;                  // token tile of a stage (256 K)
    static constexpr int SC_ROW = STMA ? 16 : 8;               // e8m0 bytes of a row in a stage
    static constexpr int SC_BYTES = AROWS * SC_ROW;
    static constexpr int SC_OFF = A_BYTES;                     // within a weight stage
    static constexpr int A_STAGE = ((A_BYTES + SC_BYTES) + 1023) / 1024 * 1024;
    static constexpr int B_STAGE = (B_BYTES + 1023) / 1024 * 1024;
    static constexpr int XCH_STRIDE = N + 1;
    static constexpr int XCH_BYTES = 64 * XCH_STRIDE * 4;
    static constexpr int RING_BYTES = UR * 32;
    static constexpr int MISC = 1024 /*align slack*/ + XCH_BYTES + RING_BYTES + 1024 /*barriers*/;
    // weight stages: an even count, so that each stage's two sub-chunks always
    // go to the same two decoder groups (no group is ever two phases ahead)
    static constexpr int NSA = (232448 - MISC - NSB * B_STAGE) / A_STAGE / 2 * 2;
    static constexpr int SMEM = MISC + NSB * B_STAGE + NSA * A_STAGE;
    // TMEM: 2 buffers x NMMA fp32 accumulators of N columns, then as many A
    // stages as fit
    static constexpr int A_COL0 = (2 * NMMA * N + 63) / 64 * 64;
    static constexpr int NA = (TMEM_COLS - A_COL0) / A_COLS / NMMA * NMMA;   // a multiple of NMMA
    static_assert(N % 16 == 0 && N >= 16 && N <= 64, "MMA N");
    static_assert(NA >= 2 * NMMA && NA % NMMA == 0, "TMEM A stages: two or more per issuer");
    static_assert(NSA >= 4 && (2 * NSA) % DEC_GROUPS == 0, "weight stages");
    static_assert(SMEM <= 232448, "shared memory per CTA");
};

struct Args {
    const Tile* tiles;
    StatusBlock* sb;
    const uint8_t* w13s;
    const uint8_t* w2s;
    __nv_bfloat16* h;
    float* y;
    float* ssq;      // per-pick sums of y^2 by 128-row block, or null
    uint32_t* tile_ready;
    int d, I;
};

struct Unit {
    int down;        // 0: gate_up, 1: down
    int tile, mb;    // tile index and row block
    int e, p0, n;
    int stages;      // shared-memory stages (256 K each) of the unit
    int pad;
};

// unit u of the call (u < U1: gate_up units, tile-major; then down units)
__device__ __forceinline__ void unit_coords(int u, int U1, const Args& a, int& down, int& tile, int& mb) {
    const int mb1 = a.I / 64, mb2 = a.d / AROWS;
    if (u < U1) {
        down = 0;
        tile = u / mb1;
        mb = u % mb1;
    } else {
        const int v = u - U1;
        down = 1;
        tile = v / mb2;
        mb = v % mb2;
    }
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

template <int N, bool STMA>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_experts_tc(const __grid_constant__ CUtensorMap tm_w13, const __grid_constant__ CUtensorMap tm_w2,
                 const __grid_constant__ CUtensorMap tm_xg, const __grid_constant__ CUtensorMap tm_h,
                 const __grid_constant__ CUtensorMap tm_w13s, const __grid_constant__ CUtensorMap tm_w2s,
                 const Args a) {
    using C = Cfg<N, STMA>;
    constexpr int NSA = C::NSA, NA = C::NA, A_COL0 = C::A_COL0;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* wst = smem;                                  // weight stages [NSA][A_STAGE]
    uint8_t* tst = smem + NSA * C::A_STAGE;               // token stages [NSB][B_STAGE]
    float* xch = reinterpret_cast<float*>(tst + NSB * C::B_STAGE);
    Unit* uring = reinterpret_cast<Unit*>(reinterpret_cast<uint8_t*>(xch) + C::XCH_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(uring) + C::RING_BYTES);
    uint64_t* full_a = bars;                // [NSA]
    uint64_t* empty_a = full_a + NSA;       // [NSA]
    uint64_t* full_b = empty_a + NSA;       // [NSB]
    uint64_t* empty_b = full_b + NSB;       // [NSB]
    uint64_t* a_full = empty_b + NSB;       // [NA]
    uint64_t* a_empty = a_full + NA;        // [NA]
    uint64_t* acc_full = a_empty + NA;      // [2]
    uint64_t* acc_empty = acc_full + 2;     // [2]
    uint64_t* u_full = acc_empty + 2;       // [UR]
    uint64_t* u_empty = u_full + UR;        // [UR]
    uint64_t* fin = u_empty + UR;           // [NMMA]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(fin + NMMA);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* epi_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    StatusBlock* sb = a.sb;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSA; ++i) {
            ptx::mbar_init(&full_a[i], STMA ? 1 : 1 + 32);   // expect_tx (+ 32 cp.async arrivals)
            ptx::mbar_init(&empty_a[i], 2 * 4);             // the 4 decoder warps of each sub-chunk
        }
        for (int i = 0; i < NSB; ++i) {
            ptx::mbar_init(&full_b[i], 1);
            ptx::mbar_init(&empty_b[i], 2);                 // MMA commits of the stage's two sub-chunks
        }
        for (int i = 0; i < NA; ++i) {
            ptx::mbar_init(&a_full[i], 4);
            ptx::mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&acc_full[i], NMMA);
            ptx::mbar_init(&acc_empty[i], 4);
        }
        for (int i = 0; i < UR; ++i) {
            ptx::mbar_init(&u_full[i], 1);
            ptx::mbar_init(&u_empty[i], NMMA + 1 + 4 * DEC_GROUPS + 4);   // MMA, token producer, decoders, epilogue
        }
        for (int i = 0; i < NMMA; ++i) ptx::mbar_init(&fin[i], 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == MMA_WARP0) ptx::tmem_alloc(tmem_holder, TMEM_COLS);
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tm_w13);
        ptx::prefetch_tensormap(&tm_w2);
        if (STMA) {
            ptx::prefetch_tensormap(&tm_w13s);
            ptx::prefetch_tensormap(&tm_w2s);
        }
    }
    if (warp == TOK_WARP && lane == 0) {
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
    const int my_units = total > (int)blockIdx.x ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int mb1 = a.I / 64;

    auto fail = [&](int site) {
        latch_status(sb, MOE_ERR_TIMEOUT, site);
        *abort_flag = 1;
    };
    // consumers: unit i of this CTA from the ring (warp-uniform; false = give up)
    auto take_unit = [&](int i, Unit& U) -> bool {
        if (!ptx::mbar_wait_warp(&u_full[i % UR], (i / UR) & 1, abort_flag, WAIT_NS)) return false;
        U = uring[i % UR];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&u_empty[i % UR]);
        return true;
    };
    // unit i of this CTA without its tile entry (e, p0, n)
    auto unit_shape = [&](int i, Unit& U) {
        unit_coords(blockIdx.x + i * gridDim.x, U1, a, U.down, U.tile, U.mb);
        U.stages = ((U.down ? a.I : a.d) + KS - 1) / KS;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ weight producer
        const uint64_t pol_w = ptx::policy_evict_first();
        // L2 prefetch cursor: unit pi, stage pc, PF stages ahead of the loads
        int pi = 0, pc = 0;
        Unit PU;
        Tile pnext = {0, 0, 0, 0};
        if (my_units > 0) {
            unit_shape(0, PU);
            PU.e = a.tiles[PU.tile].e;
            if (my_units > 1) {
                Unit t;
                unit_shape(1, t);
                pnext = a.tiles[t.tile];
            }
        }
        auto prefetch_one = [&]() {
            if (pi >= my_units) return;
            if (lane == 0) {
                if (!PU.down) {
                    const int r0 = PU.mb * 64;
                    ptx::tma_prefetch_4d(&tm_w13, 0, r0, 2 * PU.e, 2 * pc);
                    if (STMA && !(pc & 1)) ptx::tma_prefetch_3d(&tm_w13s, (pc >> 1) * 16, r0, 2 * PU.e);
                } else {
                    const int r0 = PU.e * a.d + PU.mb * AROWS;
                    ptx::tma_prefetch_3d(&tm_w2, 0, r0, 2 * pc);
                    if (STMA && !(pc & 1)) ptx::tma_prefetch_2d(&tm_w2s, (pc >> 1) * 16, r0);
                }
            }
            if (++pc == PU.stages) {
                pc = 0;
                if (++pi < my_units) {
                    unit_shape(pi, PU);
                    PU.e = pnext.e;
                    if (pi + 1 < my_units) {
                        Unit t;
                        unit_shape(pi + 1, t);
                        pnext = a.tiles[t.tile];
                    }
                }
            }
        };
        for (int j = 0; j < PF; ++j) prefetch_one();

        int ts = 0;   // stage sequence number
        bool ok = true;
        Tile tnext = {0, 0, 0, 0};
        if (my_units > 0) {
            Unit t;
            unit_shape(0, t);
            tnext = a.tiles[t.tile];
        }
        for (int i = 0; i < my_units && ok; ++i) {
            Unit U;
            unit_shape(i, U);
            U.e = tnext.e;
            U.p0 = tnext.p0;
            U.n = tnext.n;
            U.pad = 0;
            if (i + 1 < my_units) {   // the next unit's tile entry, in flight while this one is issued
                Unit t;
                unit_shape(i + 1, t);
                tnext = a.tiles[t.tile];
            }
            if (!ptx::mbar_wait_warp(&u_empty[i % UR], ((i / UR) & 1) ^ 1, abort_flag, WAIT_NS)) {
                if (lane == 0) fail(8);
                break;
            }
            if (lane == 0) {
                uring[i % UR] = U;
                ptx::mbar_arrive(&u_full[i % UR]);
            }
            const int K = U.down ? a.I : a.d;
            const int r0 = U.down ? U.e * a.d + U.mb * AROWS : U.mb * 64;
            for (int c = 0; c < U.stages; ++c, ++ts) {
                const int s = ts % NSA;
                if (!ptx::mbar_wait_warp(&empty_a[s], ((ts / NSA) & 1) ^ 1, abort_flag, WAIT_NS)) {
                    if (lane == 0) fail(1);
                    ok = false;
                    break;
                }
                uint8_t* st = wst + s * C::A_STAGE;
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(&full_a[s], A_BYTES + (STMA ? C::SC_BYTES : 0));
                    if (!U.down) {
                        // gate rows mb*64.. and up rows I + mb*64.. of expert e, 2 slabs of 128 K
                        ptx::tma_load_4d(st, &tm_w13, 0, r0, 2 * U.e, 2 * c, &full_a[s], pol_w);
                        if (STMA) ptx::tma_load_3d(st + C::SC_OFF, &tm_w13s, (c >> 1) * 16, r0, 2 * U.e, &full_a[s], pol_w);
                    } else {
                        ptx::tma_load_3d(st, &tm_w2, 0, r0, 2 * c, &full_a[s], pol_w);
                        if (STMA) ptx::tma_load_2d(st + C::SC_OFF, &tm_w2s, (c >> 1) * 16, r0, &full_a[s], pol_w);
                    }
                }
                if (!STMA) {
                    // e8m0 bytes of this stage: rows lane, lane+32, lane+64, lane+96, 4 bytes a
                    // sub-chunk; a sub-chunk past K (odd K/128) reads the row's first bytes
                    // (its weights are zero-filled, so they are multiplied by zero)
                    const uint8_t* sbase = U.down ? a.w2s : a.w13s;
                    const int kb = K / 32;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int r = lane + 32 * j;
                        const uint8_t* row = sbase + (size_t)weight_row(U, r, a) * kb;
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int sub = 2 * c + hh;
                            ptx::cp_async_4(st + C::SC_OFF + 8 * r + 4 * hh, row + (sub * 4 < kb ? sub * 4 : 0));
                        }
                    }
                    ptx::cp_async_mbar_arrive_noinc(&full_a[s]);
                }
                prefetch_one();
                __syncwarp();
            }
        }
        ptx::cp_async_wait_all();
    } else if (warp == TOK_WARP) {
        // ------------------------------------------------------------ token producer
        const uint64_t pol_x = ptx::policy_evict_last();
        int ts = 0;
        bool ok = true;
        for (int i = 0; i < my_units && ok; ++i) {
            Unit U;
            if (!take_unit(i, U)) {
                if (lane == 0) fail(12);
                break;
            }
            const CUtensorMap* tmB = U.down ? &tm_h : &tm_xg;
            if (U.down) {
                // the tile's h rows: complete once all its gate_up units are done
                uint32_t ready = 0;
                if (lane == 0) {
                    const uint64_t t0 = ptx::globaltimer();
                    uint32_t it = 0;
                    ready = 1;
                    while (ptx::ld_acquire_gpu(&a.tile_ready[U.tile]) < (uint32_t)mb1) {
                        __nanosleep(32);
                        if ((++it & 63u) == 0u && (*abort_flag || ptx::globaltimer() - t0 > WAIT_NS)) {
                            fail(2);
                            ready = 0;
                            break;
                        }
                    }
                    if (ready) ptx::fence_proxy_async_global();
                }
                if (!__shfl_sync(0xffffffffu, ready, 0)) break;
            }
            for (int c = 0; c < U.stages; ++c, ++ts) {
                const int s = ts % NSB;
                if (!ptx::mbar_wait_warp(&empty_b[s], ((ts / NSB) & 1) ^ 1, abort_flag, WAIT_NS)) {
                    if (lane == 0) fail(13);
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(&full_b[s], C::B_BYTES);
                    ptx::tma_load_3d(tst + s * C::B_STAGE, tmB, 0, U.p0, 4 * c, &full_b[s], pol_x);
                }
                __syncwarp();
            }
        }
    } else if (warp >= MMA_WARP0 && warp < MMA_WARP0 + NMMA) {
        // ------------------------------------------------------------ MMA issuers
        constexpr uint32_t idesc = ptx::idesc_bf16_f32(AROWS, N);
        const int m = warp - MMA_WARP0;   // this issuer takes sub-chunks q = m mod NMMA (every unit
                                          // has an even number of sub-chunks, so it gets at least one)
        int q = 0;                        // sub-chunk sequence number
        for (int i = 0; i < my_units; ++i) {
            Unit U;
            if (!take_unit(i, U)) {
                if (lane == 0) fail(9);
                break;
            }
            bool ok = true;
            if (lane == 0) {
                const int ab = i & 1;
                const uint32_t d_tmem = tmem + (ab * NMMA + m) * N;
                bool first = true;
                for (int cc = 0; cc < 2 * U.stages && ok; ++cc, ++q) {
                    if (q % NMMA != m) continue;
                    if (first && !ptx::mbar_wait(&acc_empty[ab], ((i >> 1) & 1) ^ 1, abort_flag, WAIT_NS)) {
                        fail(3);
                        ok = false;
                        break;
                    }
                    const int ts = q >> 1, sbi = ts % NSB, as = q % NA, hh = q & 1;
                    if (!ptx::mbar_wait(&full_b[sbi], (ts / NSB) & 1, abort_flag, WAIT_NS) ||
                        !ptx::mbar_wait(&a_full[as], (q / NA) & 1, abort_flag, WAIT_NS)) {
                        fail(4);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t b0 = ptx::smem_u32(tst + sbi * C::B_STAGE + 2 * hh * C::B_BOX);
                    const uint32_t a0 = tmem + A_COL0 + as * A_COLS;
#pragma unroll
                    for (int kk = 0; kk < KC / 16; ++kk) {
                        const uint64_t bd = ptx::smem_desc_sw128(b0 + (kk >> 2) * C::B_BOX + (kk & 3) * 32);
                        ptx::mma_bf16_ts(d_tmem, a0 + kk * 8, bd, idesc, (!first || kk) ? 1u : 0u);
                    }
                    first = false;
                    ptx::mma_commit(&a_empty[as]);
                    ptx::mma_commit(&empty_b[sbi]);
                }
                if (ok) ptx::mma_commit(&acc_full[ab]);
            }
            q = __shfl_sync(0xffffffffu, q, 0);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
        }
        if (lane == 0) {
            // every MMA issued above has completed before TMEM is released
            ptx::mma_commit(&fin[m]);
            ptx::mbar_wait(&fin[m], 0, abort_flag, WAIT_NS);
        }
        __syncwarp();
    } else if (warp >= DEC_WARP0) {
        // ------------------------------------------------------------ decoders
        const int dw = warp - DEC_WARP0;
        const int g = dw >> 2;            // this group takes sub-chunks g mod DEC_GROUPS
        const int qd = warp & 3;          // TMEM lane quarter of this warp
        const int r = 32 * qd + lane;     // weight row of this thread
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        int q = 0;
        bool ok = true;
        for (int i = 0; i < my_units && ok; ++i) {
            Unit U;
            if (!take_unit(i, U)) {
                if (lane == 0) fail(10);
                break;
            }
            for (int cc = 0; cc < 2 * U.stages; ++cc, ++q) {
                if (q % DEC_GROUPS != g) continue;
                const int ts = q >> 1, s = ts % NSA, as = q % NA, hh = q & 1;
                if (!ptx::mbar_wait_warp(&full_a[s], (ts / NSA) & 1, abort_flag, WAIT_NS)) {
                    if (lane == 0) fail(5);
                    ok = false;
                    break;
                }
                const uint8_t* st = wst + s * C::A_STAGE;
                const uint8_t* arow = st + hh * A_SUB + r * 64;
                uint4 w4[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    w4[j] = *reinterpret_cast<const uint4*>(arow + ((j ^ ((r >> 1) & 3)) << 4));
                const uint32_t sc = *reinterpret_cast<const uint32_t*>(
                    st + C::SC_OFF + C::SC_ROW * r + (STMA ? 4 * (cc & 3) : 4 * hh));
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&empty_a[s]);
                if (!ptx::mbar_wait_warp(&a_empty[as], ((q / NA) & 1) ^ 1, abort_flag, WAIT_NS)) {
                    if (lane == 0) fail(6);
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t ta = tmem + lane_base + A_COL0 + as * A_COLS;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t v[16];
                    decode_block(w4[j], (sc >> (8 * j)) & 0xFFu, v, sb);
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
        for (int i = 0; i < my_units; ++i) {
            const int ab = i & 1;
            // the four epilogue warps take one decision before their named
            // barriers: carry on, or leave together
            Unit U;
            if (!take_unit(i, U) && lane == 0) fail(11);
            if (!*abort_flag && !ptx::mbar_wait_warp(&acc_full[ab], (i >> 1) & 1, abort_flag, WAIT_NS) &&
                lane == 0)
                fail(7);
            ptx::named_bar_sync(1, 128);
            if (threadIdx.x == EPI_WARP0 * 32) *epi_flag = *abort_flag;
            ptx::named_bar_sync(1, 128);
            if (*epi_flag) break;
            ptx::tc_fence_after();
            // sum the issuers' accumulators (each issuer had sub-chunks of the unit)
            float v[N];
#pragma unroll
            for (int n = 0; n < N; ++n) v[n] = 0.f;
#pragma unroll
            for (int mm = 0; mm < NMMA; ++mm) {
                uint32_t t[N];
#pragma unroll
                for (int j = 0; j < N / 16; ++j)
                    ptx::tmem_ld16(tmem + lane_base + (ab * NMMA + mm) * N + 16 * j, t + 16 * j);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int n = 0; n < N; ++n) v[n] += __uint_as_float(t[n]);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&acc_empty[ab]);
            if (!U.down) {
                // lanes 0..63: gate of rows mb*64 + r; lanes 64..127: up of the same rows
                if (r >= 64) {
#pragma unroll
                    for (int n = 0; n < N; ++n) xch[(r - 64) * C::XCH_STRIDE + n] = v[n];
                }
                ptx::named_bar_sync(1, 128);
                if (r < 64) {
                    const int ii = U.mb * 64 + r;
                    const int col = kperm(ii);
#pragma unroll
                    for (int n = 0; n < N; ++n) {
                        if (n < U.n) {
                            const float gv = v[n];
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
                    if (n < U.n) a.y[(size_t)(U.p0 + n) * a.d + m] = v[n];
                if (a.ssq != nullptr) {
                    // sum of y^2 over the unit's 128 rows for every pick: a
                    // reduce-scatter across the warp (lane l ends with picks
                    // [idx, idx + c)), then the four warps' sums in warp order
                    float q[N];
#pragma unroll
                    for (int n = 0; n < N; ++n) q[n] = v[n] * v[n];
                    int idx = 0;
#pragma unroll
                    for (int step = 0; step < 5; ++step) {
                        const int o = 16 >> step;
                        const int c = N >> step;        // values a lane holds before this step
                        const bool hi = (lane & o) != 0;
                        if (c > 1) {
#pragma unroll
                            for (int j = 0; j < c / 2; ++j) {
                                const float send = hi ? q[j] : q[j + c / 2];
                                const float keep = hi ? q[j + c / 2] : q[j];
                                q[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                            }
                            idx += hi ? c / 2 : 0;
                        } else {
                            q[0] += __shfl_xor_sync(0xffffffffu, q[0], o);
                        }
                    }
                    constexpr int C_END = N >= 32 ? N / 32 : 1;   // values a lane holds at the end
                    constexpr int SHARE = 32 * C_END / N;          // lanes holding the same values
                    float* part = xch;                             // [4][N]
                    if (lane % SHARE == 0) {
#pragma unroll
                        for (int j = 0; j < C_END; ++j) part[qd * N + idx + j] = q[j];
                    }
                    ptx::named_bar_sync(1, 128);
                    if (r < U.n)
                        a.ssq[(size_t)(U.p0 + r) * (a.d / AROWS) + U.mb] =
                            ((part[r] + part[N + r]) + part[2 * N + r]) + part[3 * N + r];
                }
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
    if (warp == MMA_WARP0) ptx::tmem_dealloc(tmem, TMEM_COLS);
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

// rank-r tiled map: dims[0] innermost; strides[i] = byte stride of dims[i+1]
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) gs[i] = strides[i];
    }
    return fn(m, dt, rank, const_cast<void*>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
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

template <int N, bool STMA>
cudaError_t launch_tc(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    using C = Cfg<N, STMA>;
    CUtensorMap tm_w13, tm_w2, tm_xg, tm_h, tm_w13s, tm_w2s;
    const uint64_t P = (uint64_t)L.max_picks, E = s.E, d = s.d, I = s.I;
    const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8, BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // w13 [E][2][I][d/2] as {64 bytes, I rows, 2E halves, d/128 slabs}
    const uint64_t w13_d[4] = {64, I, 2 * E, d / 128}, w13_s[3] = {d / 2, I * d / 2, 64};
    const uint32_t w13_b[4] = {64, 64, 2, 2};
    // w2 [E d][I/2] as {64 bytes, E d rows, I/128 slabs}
    const uint64_t w2_d[3] = {64, E * d, I / 128}, w2_s[2] = {I / 2, 64};
    const uint32_t w2_b[3] = {64, AROWS, 2};
    // xg [P][d] / h [P][I] bf16 as {64 elements, P rows, K/64 slabs}
    const uint64_t xg_d[3] = {64, P, d / 64}, xg_s[2] = {d * 2, 128};
    const uint64_t h_d[3] = {64, P, I / 64}, h_s[2] = {I * 2, 128};
    const uint32_t tok_b[3] = {64, (uint32_t)N, 4};
    if (!make_map(&tm_w13, U8, p.w13, 4, w13_d, w13_s, w13_b, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&tm_w2, U8, p.w2, 3, w2_d, w2_s, w2_b, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&tm_xg, BF, p.ws + L.xg, 3, xg_d, xg_s, tok_b, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tm_h, BF, p.ws + L.h, 3, h_d, h_s, tok_b, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (STMA) {
        // w13s [E][2][I][d/32] as {d/32 bytes, I rows, 2E halves}; w2s [E d][I/32]
        const uint64_t a_d[3] = {d / 32, I, 2 * E}, a_s[2] = {d / 32, I * d / 32};
        const uint32_t a_b[3] = {16, 64, 2};
        const uint64_t b_d[2] = {I / 32, E * d}, b_s[1] = {I / 32};
        const uint32_t b_b[2] = {16, AROWS};
        if (!make_map(&tm_w13s, U8, p.w13s, 3, a_d, a_s, a_b, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_map(&tm_w2s, U8, p.w2s, 2, b_d, b_s, b_b, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        tm_w13s = tm_w13;   // unused
        tm_w2s = tm_w2;
    }
    cudaError_t e = cudaFuncSetAttribute(k_experts_tc<N, STMA>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    Args a;
    a.tiles = reinterpret_cast<const Tile*>(p.ws + L.tiles);
    a.sb = reinterpret_cast<StatusBlock*>(p.ws + L.status);
    a.w13s = p.w13s;
    a.w2s = p.w2s;
    a.h = reinterpret_cast<__nv_bfloat16*>(p.ws + L.h);
    a.y = reinterpret_cast<float*>(p.ws + L.y);
    a.ssq = p.norm_w != nullptr ? reinterpret_cast<float*>(p.ws + L.ssq) : nullptr;
    a.tile_ready = reinterpret_cast<uint32_t*>(p.ws + L.tile_ready);
    a.d = s.d;
    a.I = s.I;
    k_experts_tc<N, STMA><<<num_sms(), NUM_THREADS, C::SMEM, st>>>(tm_w13, tm_w2, tm_xg, tm_h, tm_w13s, tm_w2s, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_experts(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    timing_begin(K_EXPERTS, st);
    const bool stma = (s.d % 512 == 0) && (s.I % 512 == 0);
    cudaError_t e = stma ? launch_tc<NT, true>(s, L, p, st) : launch_tc<NT, false>(s, L, p, st);
    timing_end(st);
    return e;
}

}  // namespace moe
