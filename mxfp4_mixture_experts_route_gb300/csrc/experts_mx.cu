// MXFP4 expert GEMMs on the 5th-generation tensor cores with hardware block
// scaling: one persistent kernel runs every gate_up unit and then every down
// unit of the call.
//
// vllm.models.muse_spark.amd.mono.kernels.k3, stages C and D (the local
// experts' gate_up and down projections on MXFP4 weights): the weights stay in their MX form,
// e2m1 codes with one e8m0 scale per 32 elements of a row; fp4_mma: a 256-K
// chunk of a row group per step; task_ring: compute the current task with the
// next tasks' loads in flight.  vllm.models.kimi_k3.amd.specialized_decode.
// mono.layer: the static weights stream while earlier stages settle, weights
// issued before the first wait.
//
// GB300 design.  The pages decode the e2m1 codes to 16-bit values in
// registers for a bf16 MMA.  On sm_103a the tensor core takes e2m1 operands
// and e8m0 block scales itself (tcgen05.mma kind::mxf8f6f4 block_scale), and
// the TMA unpacks packed 4-bit codes into the tensor core's operand layout on
// the way to shared memory, so no thread touches a weight byte.  The other
// operand must then be an 8-bit float: each bf16 token row x (and each fp32 h
// row) is written as two e4m3 rows, hi = e4m3(x / 2^s) and lo = e4m3(x / 2^s
// - hi), with 2^s an e8m0 scale per 32 elements chosen so that the block's
// largest magnitude lands in [128, 256).  hi carries the leading 4 significant
// bits and lo the next 4, so hi + lo is x / 2^s exactly for a bf16 x (to
// within 2^-17 of the block maximum for elements more than 2^9 below it).
// The MMA's N = 2 nt columns are the hi and lo rows of an nt-pick tile (nt =
// 8, 16, 32 or 64, by the picks an expert gets on average); the epilogue adds
// each pick's two columns.
//
// One persistent CTA per SM, 13 warps:
//   warp 0      weight producer: per 256-K stage of a unit, the weight tile
//               (128 rows x 256 K e2m1 = 16 KB of HBM, 32 KB in shared memory
//               in the tensor core's 4-bit layout, which the tensor map writes;
//               gate and up rows in one 4-D box) and its e8m0 bytes into a ring
//               of weight stages.
//   warp 7      token producer: the token tile (2 nt e4m3 rows x 256 K, one
//               3-D box of two 128-byte-swizzled slabs) and the tile's nt rows
//               of block scales (one bulk copy) into a ring of its own; for a
//               down unit it first waits (bounded) for the tile's h.
//   warps 8-11  scale movers: copy the stage's weight and token block scales
//               from shared memory into TMEM, in the layout the MMA reads.
//   warp 12     unit scheduler: claims units and reads their tile entries
//               (global-memory round trips) at most LOOKAHEAD units ahead of the
//               weight producer, and publishes them in the CTA's unit ring.
//   warps 1-2   MMA issuers (lane 0 of each): M = 128 weight rows, N = 2 nt,
//               K = 32; issuer m takes the stages of parity m of every unit
//               into an fp32 accumulator of its own (buffered by unit).  One
//               thread needs several hundred cycles per stage for its waits,
//               MMAs and commits, more than a stage lasts at full HBM
//               bandwidth; two issuers on alternate stages keep up (64-pick
//               tiles, whose stages last longer, have one).
//   warps 3-6   epilogue: the issuers' accumulators and each pick's hi and lo
//               column added; h = silu(g) * u split into e4m3 hi/lo rows with a
//               block scale per 32 rows for gate_up; y (fp32) and per-128-row
//               sums of squares for down.
// Work units: CTA b starts with unit b and claims the next ones from a
// device-wide counter (reset by the sort kernel), so that a CTA that finishes
// early takes more.  Gate_up units
// first (64 gate rows stacked on the matching 64 up rows = one M = 128
// operand), then down units (128 rows of w2).  A down unit needs the h rows of
// its tile: the counter of the tile, which every finished gate_up unit of it
// increments.  Every gate_up unit is claimed before any down unit and a
// gate_up unit waits on nothing, so each of these waits ends.
#include "moe_internal.cuh"
#include "tc_ptx.cuh"

#include <cudaTypedefs.h>

namespace moe {

namespace {

constexpr int KS = 256;                      // K elements of one stage
constexpr int AROWS = 128;                   // MMA M
constexpr int A_SLAB = AROWS * 128;          // one 128-K slab of the weight tile in shared memory (unpacked)
constexpr int A_SMEM = 2 * A_SLAB;           // 32 KB
constexpr int A_TX = AROWS * KS / 2;         // packed bytes of a weight tile: the TMA transaction count
#ifndef MOE_MX_TOKEN_STAGES
#define MOE_MX_TOKEN_STAGES 4
#endif
#ifndef MOE_MX_WIDE_TOKEN_STAGES
#define MOE_MX_WIDE_TOKEN_STAGES 3
#endif
#ifndef MOE_MX_DOWN_BLOCKS
#define MOE_MX_DOWN_BLOCKS 2
#endif

constexpr int NSB_DEF = MOE_MX_TOKEN_STAGES; // token-tile stages (MOE_MX_WIDE_TOKEN_STAGES for 64-pick tiles)
constexpr int TMEM_COLS = 512;
constexpr int NMMA_MAX = 2;                  // MMA-issuing warps (one thread each; one for 64-pick tiles)
// One stage's scale slot in TMEM, 64 columns: the weight scales of K steps
// 0-3 at +0 and of K steps 4-7 at +16 (row m of the tile in lane m, column
// + m / 32), the token scales at +32 and +48 (column n in lane n mod 32 of
// every lane quarter, column + n / 32).  Every scale address the MMA gets is a
// multiple of 16 columns.
constexpr int SF_SLOT = 64;
constexpr int SF_A1 = 16, SF_B0 = 32, SF_B1 = 48;
constexpr int MMA_WARP0 = 1, EPI_WARP0 = 3, TOK_WARP = 7, SF_WARP0 = 8, SCHED_WARP = 12;
constexpr int NUM_WARPS = 13;
constexpr int LOOKAHEAD = 1;                 // units the scheduler publishes ahead of the weight producer
constexpr int NUM_THREADS = 32 * NUM_WARPS;
constexpr int UR = 32;                       // unit ring entries
// Diagnostics build (-DMOE_TRACE): %globaltimer stamps per CTA, read back
// with moe_trace_copy: [cta][TR_KINDS][TR_CAP] u64, kinds below (index = the
// CTA's stage or unit sequence number; slot 0 of TR_MISC = kernel start, 1 =
// after the wait on the preceding kernel, 2 = end).
#ifdef MOE_TRACE
constexpr int TR_CAP = 1024, TR_KINDS = 8, TR_MAX_CTAS = 160;
enum { TR_UNIT = 0, TR_ISSUE = 1, TR_LANDED = 2, TR_MMA = 3, TR_MISC = 4, TR_UDESC = 5, TR_ACCE = 6, TR_EPI = 7 };
__device__ uint64_t g_trace[TR_MAX_CTAS][TR_KINDS][TR_CAP];
#define MOE_TR(kind, idx)                                                                    \
    do {                                                                                     \
        if (blockIdx.x < TR_MAX_CTAS && (idx) < TR_CAP) g_trace[blockIdx.x][kind][idx] = ptx::globaltimer(); \
    } while (0)
#else
#define MOE_TR(kind, idx) \
    do {                  \
    } while (0)
#endif

#ifndef MOE_WAIT_TEST
constexpr uint64_t WAIT_NS = 2000000000ull;  // bounded waits: 2 s
constexpr uint64_t WAIT_NS_H = WAIT_NS;      // the token producer's wait for a tile's h rows
#else
// test-only build: waits give up after 1 ms, and one down unit can be made to
// wait for a readiness count that is never reached; that wait gives up first
// (the waits behind it, on the unit's MMAs, would run out 1 ms after they began)
constexpr uint64_t WAIT_NS = 1000000ull;
constexpr uint64_t WAIT_NS_H = WAIT_NS / 4;
int g_unreachable_wait = 0;
#endif

struct Unit {
    int down;        // 0: gate_up, 1: down, -1: no more units
    int tile, mb;    // tile index; row block (gate_up) or group of RD row blocks (down)
    int e, p0, n;
    int stages;      // 256-K stages of the unit
    int nblk;        // down: 128-row blocks of the unit (<= RD)
    int h_ready;     // down: the scheduler saw the tile's h rows complete
};

// STMA: the e8m0 bytes of the weights come by TMA, 16 bytes (512 K) of each
// row per stage, when the scale rows are 16-byte aligned (K % 512 == 0);
// otherwise by 4-byte cp.async, 8 bytes (256 K) of each row per stage.
// NTT: picks per tile (8 or 16); the MMA N is 2 NTT.
template <bool STMA, int NTT>
struct Cfg {
    static constexpr int NB = 2 * NTT;                         // MMA N: a hi and a lo row per pick
    static constexpr int NMMA = NTT >= 64 ? 1 : NMMA_MAX;      // issuers (TMEM: one N = 128 accumulator each)
    static constexpr int NSB = NTT >= 64 ? MOE_MX_WIDE_TOKEN_STAGES : NSB_DEF;   // token stages (32 KB at 64 picks)
    static constexpr int EC = NTT < 16 ? NTT : 16;             // picks per epilogue chunk
    static constexpr int B_SLAB = NB * 128;                    // one 128-K slab of the token tile
    static constexpr int B_SMEM = 2 * B_SLAB;                  // a token stage (4 or 8 KB)
    static constexpr int BS_BYTES = NTT * TOKEN_SCALE_ROW;     // the tile's token scale rows
    // 128-row blocks of w2 in one down unit: a down unit is short (I / 256
    // stages a block), and every unit costs a claim, a tile-entry read and a
    // readiness check of its h rows; several blocks of one tile can share
    // them where the accumulators fit in TMEM beside the scale slots
    static constexpr int RD = NTT == 8 ? MOE_MX_DOWN_BLOCKS : 1;
    // fp32 accumulators: ACCB buffers (by unit) of RD x NMMA accumulators of
    // NB columns: block b of the unit, issuer slot j (the issuers take
    // alternate stages of a block); 4 buffers when they fit beside six scale
    // slots, so that short units do not wait for the epilogue to drain the
    // buffer of two units back
    static constexpr int ACC_UNIT = RD * NMMA;
    static constexpr int BW = ACC_UNIT * NB;
    static constexpr int ACCB = (NTT == 8 && RD == 1) ? 4 : 2;
    static constexpr int BSG = (NB + 31) / 32;                 // TMEM columns of one group of token scales
    static_assert(NTT <= NT_MAX, "token tables are padded by NT_MAX rows");
    static constexpr int SF_COL0 = ACCB * BW;                  // TMEM columns of the scale slots

    static constexpr int SC_ROW = STMA ? 16 : 8;               // e8m0 bytes of a row in a stage
    static constexpr int SC_BYTES = AROWS * SC_ROW;
    static constexpr int SC_OFF = A_SMEM;                      // within a weight stage
    static constexpr int A_STAGE = (A_SMEM + SC_BYTES + 1023) / 1024 * 1024;
    static constexpr int B_STAGE = B_SMEM;                     // the token scale rows sit apart
    static constexpr int XCH_STRIDE = EC + 1;
    static constexpr int XCH_BYTES = 64 * XCH_STRIDE * 4;
    static constexpr int RING_BYTES = (UR * (int)sizeof(Unit) + 15) / 16 * 16;
    static constexpr int TSC_BYTES = NSB * BS_BYTES;
    static constexpr int MISC = 1024 /*align slack*/ + XCH_BYTES + RING_BYTES + TSC_BYTES + 1024 /*barriers*/;
    static constexpr int NSA_FIT = (232448 - MISC - NSB * B_STAGE) / A_STAGE;
    static constexpr int NSA_TMEM = (TMEM_COLS - SF_COL0) / SF_SLOT;
    static constexpr int NSA = NSA_FIT < NSA_TMEM ? NSA_FIT : NSA_TMEM;
    static constexpr int SMEM = MISC + NSB * B_STAGE + NSA * A_STAGE;
    static_assert(NSA >= 3, "weight stages");
    static_assert(SMEM <= 232448, "shared memory per CTA");
    static_assert(SF_COL0 + NSA * SF_SLOT <= TMEM_COLS, "TMEM columns");
};

struct Args {
    const Tile* tiles;
    StatusBlock* sb;
    const uint8_t* w13s;
    const uint8_t* w2s;
    uint8_t* hq;          // [2P][I] e4m3: row 2p = hi, row 2p + 1 = lo of pick p's h
    uint8_t* hs;          // [ceil(I/256)][P + NT_MAX][16] e8m0 block scales of h
    float* y;
    float* ssq;           // per-pick sums of y^2 by 128-row block, or null
    uint32_t* tile_ready;
    const uint8_t* xs;    // [ceil(d/256)][P + NT_MAX][16] e8m0 block scales of the gathered tokens
    int d, I, P;
    int max_tiles;
#ifdef MOE_WAIT_TEST
    int unreachable;      // the first down unit of tile 0 waits for one gate_up unit too many
#endif
};

// A tile entry of the sort's table (an earlier kernel's output: read through L2)
__device__ __forceinline__ Tile load_tile(const Tile* p) {
    const int4 v = ld_dep(reinterpret_cast<const int4*>(p));
    Tile t;
    t.e = v.x;
    t.p0 = v.y;
    t.n = v.z;
    t.pad = v.w;
    return t;
}


// unit u of the call (u < U1: gate_up units, tile-major; then down units, g2
// groups of rd row blocks a tile)
__device__ __forceinline__ void unit_coords(int u, int U1, int g2, const Args& a, int& down, int& tile, int& mb) {
    const int mb1 = a.I / 64;
    if (u < U1) {
        down = 0;
        tile = u / mb1;
        mb = u % mb1;
    } else {
        const int v = u - U1;
        down = 1;
        tile = v / g2;
        mb = v % g2;
    }
}

// Walks the stages of a unit in order: stage c is 256-K stage kc of the
// unit's 128-row block blk (down units: kst stages a block; gate_up units:
// one block, kc = c).  Incremental, so that the per-stage loops of the
// pipeline's roles carry no division.
struct StageWalk {
    int blk = 0, kc = 0, kst;
    __device__ __forceinline__ explicit StageWalk(const Unit& U, int kst_down) : kst(U.down ? kst_down : 1 << 30) {}
    __device__ __forceinline__ void next() {
        if (++kc == kst) {
            kc = 0;
            ++blk;
        }
    }
};

// global row (in the [E * rows, K/2] view) of weight row r (0..127) of block
// blk of unit U (rd row blocks a down unit)
__device__ __forceinline__ int weight_row(const Unit& U, int blk, int r, int rd, const Args& a) {
    if (!U.down) {
        const int base = U.e * 2 * a.I + U.mb * 64;
        return r < 64 ? base + r : base + a.I + (r - 64);
    }
    return U.e * a.d + (U.mb * rd + blk) * AROWS + r;
}

// The CTA's first unit, unit blockIdx.x, when it is a gate_up unit (there
// are n_tiles * I / 64 of them): the two producers compute it themselves
// from the tile table, so that their first copies wait for no ring round
// trip.  The scheduler publishes the same unit (from the same entries) first.
__device__ __forceinline__ bool first_gate_up_unit(const Args& a, Unit& U) {
    const int mb1 = a.I / 64, u = (int)blockIdx.x;
    const int n_tiles = ld_dep(&a.sb->n_tiles);
    const Tile tl = load_tile(a.tiles + min(u / mb1, a.max_tiles - 1));
    if (u >= n_tiles * mb1) return false;
    U.down = 0;
    U.tile = u / mb1;
    U.mb = u % mb1;
    U.e = tl.e;
    U.p0 = tl.p0;
    U.n = tl.n;
    U.nblk = 0;
    U.stages = (a.d + KS - 1) / KS;
    U.h_ready = 0;
    return true;
}

template <bool STMA, int NTT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_experts_mx(const __grid_constant__ CUtensorMap tm_w13, const __grid_constant__ CUtensorMap tm_w2,
                 const __grid_constant__ CUtensorMap tm_xq, const __grid_constant__ CUtensorMap tm_hq,
                 const __grid_constant__ CUtensorMap tm_w13s, const __grid_constant__ CUtensorMap tm_w2s,
                 const Args a) {
    using C = Cfg<STMA, NTT>;
    constexpr int NSA = C::NSA, NB = C::NB, B_SLAB = C::B_SLAB, B_SMEM = C::B_SMEM, BS_BYTES = C::BS_BYTES;
    constexpr int SF_COL0 = C::SF_COL0, ACCB = C::ACCB, NSB = C::NSB, NMMA = C::NMMA, EC = C::EC;
    constexpr int RD = C::RD, BW = C::BW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* wst = smem;                                  // weight stages [NSA][A_STAGE]
    uint8_t* tst = smem + NSA * C::A_STAGE;               // token stages [NSB][B_STAGE]
    float* xch = reinterpret_cast<float*>(tst + NSB * C::B_STAGE);
    uint8_t* tsc = reinterpret_cast<uint8_t*>(xch) + C::XCH_BYTES;   // token scale rows [NSB][BS_BYTES]
    Unit* uring = reinterpret_cast<Unit*>(tsc + C::TSC_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(uring) + C::RING_BYTES);
    uint64_t* full_a = bars;                // [NSA] weight tile + its scales landed
    uint64_t* empty_a = full_a + NSA;       // [NSA] both issuers done with the weight stage
    uint64_t* full_b = empty_a + NSA;       // [NSB] token tile + its scales landed
    uint64_t* empty_b = full_b + NSB;       // [NSB] both issuers done with the token stage
    // [NMMA_MAX][NSA] the stage's scales are in TMEM: one barrier per issuer
    // and slot, arrived on for the stages that issuer owns, so that each issuer
    // waits on the phases of its own barriers strictly in order (an issuer
    // skips the other's stages; a shared barrier could be a full phase ahead
    // of it, which a parity wait cannot tell from the phase it wants)
    uint64_t* sf_full = empty_b + NSB;
    uint64_t* acc_full = sf_full + NMMA_MAX * NSA;   // [ACCB]
    uint64_t* acc_empty = acc_full + ACCB;  // [ACCB]
    uint64_t* u_full = acc_empty + ACCB;    // [UR]
    uint64_t* u_empty = u_full + UR;        // [UR]
    uint64_t* fin = u_empty + UR;           // [NMMA_MAX]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(fin + NMMA_MAX);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* taken = abort_flag + 1;   // units the weight producer has taken
    volatile int* epi_flag = abort_flag + 2;   // [2] the epilogue's leave decision, by unit parity

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    StatusBlock* sb = a.sb;
    if (threadIdx.x == 0) MOE_TR(TR_MISC, 0);
    KT_MARK(K_EXPERTS, 0);
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSA; ++i) {
            ptx::mbar_init(&full_a[i], STMA ? 1 : 1 + 32);   // expect_tx (+ 32 cp.async arrivals)
            ptx::mbar_init(&empty_a[i], 1);                 // the stage's issuer
            for (int m = 0; m < NMMA_MAX; ++m) ptx::mbar_init(&sf_full[m * NSA + i], 4);   // the four scale movers
        }
        for (int i = 0; i < NSB; ++i) {
            ptx::mbar_init(&full_b[i], 1);
            ptx::mbar_init(&empty_b[i], 1);
        }
        for (int i = 0; i < ACCB; ++i) {
            ptx::mbar_init(&acc_full[i], NMMA);
            ptx::mbar_init(&acc_empty[i], 4);
        }
        for (int i = 0; i < UR; ++i) {
            ptx::mbar_init(&u_full[i], 1);
            ptx::mbar_init(&u_empty[i], NMMA + 1 + 4 + 4 + 1);   // MMA, token, scale movers, epilogue, weights
        }
        for (int i = 0; i < NMMA; ++i) ptx::mbar_init(&fin[i], 1);
        *abort_flag = 0;
        *taken = 0;
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
        ptx::prefetch_tensormap(&tm_xq);
        ptx::prefetch_tensormap(&tm_hq);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // the set-up above needs nothing from the preceding kernels; everything
    // below reads their results
    pdl_wait();
    if (threadIdx.x == 0) MOE_TR(TR_MISC, 1);
    KT_MARK(K_EXPERTS, 1);

    const int mb1 = a.I / 64;
    const int kst_down = (a.I + KS - 1) / KS;             // 256-K stages of one down row block
    const int mb2 = a.d / AROWS;                          // 128-row blocks of w2 per expert
    const int g2 = (mb2 + RD - 1) / RD;                   // down units per tile
    // a down unit's h rows are complete when all mb1 gate_up units of its
    // tile have counted themselves in tile_ready
    auto h_target = [&](const Unit& U) -> uint32_t {
#ifndef MOE_WAIT_TEST
        return (uint32_t)mb1;
#else
        return (uint32_t)mb1 + (a.unreachable && U.tile == 0 && U.mb == 0 ? 1u : 0u);
#endif
    };
    auto ld_acquire_h = [&](const Unit& U) -> uint32_t { return ptx::ld_acquire_gpu(&a.tile_ready[U.tile]); };

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

    if (warp == 0) {
        // ------------------------------------------------------------ weight producer
        const uint64_t pol_w = ptx::policy_evict_first();
        int ts = 0;   // stage sequence number
        bool ok = true;
        if (lane == 0) MOE_TR(TR_MISC, 7);
        // lane 0: the weight tile (and its e8m0 bytes, STMA) of stage c of
        // unit U into ring slot s
        auto issue = [&](const Unit& U, const StageWalk& sa, int s) {
            uint8_t* st = wst + s * C::A_STAGE;
            const int r0 = U.down ? U.e * a.d + (U.mb * RD + sa.blk) * AROWS : U.mb * 64;
            ptx::mbar_arrive_expect_tx(&full_a[s], A_TX + (STMA ? C::SC_BYTES : 0));
            if (!U.down) {
                // gate rows mb*64.. and up rows I + mb*64.. of expert e, 2 slabs of 128 K
                ptx::tma_load_4d(st, &tm_w13, 0, r0, 2 * U.e, 2 * sa.kc, &full_a[s], pol_w);
                if (STMA) ptx::tma_load_3d(st + C::SC_OFF, &tm_w13s, (sa.kc >> 1) * 16, r0, 2 * U.e, &full_a[s], pol_w);
            } else {
                ptx::tma_load_3d(st, &tm_w2, 0, r0, 2 * sa.kc, &full_a[s], pol_w);
                if (STMA) ptx::tma_load_2d(st + C::SC_OFF, &tm_w2s, (sa.kc >> 1) * 16, r0, &full_a[s], pol_w);
            }
        };
        // the first unit's first stages, before it comes through the ring (the
        // ring of weight stages is empty: no slot to wait for)
        int pre = 0;
        if (STMA) {
            Unit U0;
            if (lane == 0 && first_gate_up_unit(a, U0)) {
                pre = min(NSA, U0.stages);
                StageWalk sa(U0, kst_down);
                for (int c = 0; c < pre; ++c, sa.next()) {
                    MOE_TR(TR_ISSUE, c);
                    issue(U0, sa, c);
                }
            }
            pre = __shfl_sync(0xffffffffu, pre, 0);
        }
        for (int i = 0; ok; ++i) {
            Unit U;
            if (!take_unit(i, U)) {
                if (lane == 0) fail(14);
                break;
            }
            if (lane == 0 && i == 0) MOE_TR(TR_MISC, 5);
            if (lane == 0) *taken = i + 1;
            if (lane == 0) MOE_TR(TR_UNIT, i);
#ifdef MOE_TRACE
            if (lane == 0 && blockIdx.x < TR_MAX_CTAS && i < TR_CAP)
                g_trace[blockIdx.x][TR_UDESC][i] = 1ull << 63 | (uint64_t)(U.down + 1) << 48 |
                                                   (uint64_t)U.tile << 24 | (uint64_t)U.mb << 8 | (uint64_t)U.stages;
#endif
            if (U.down < 0) break;
            const int K = U.down ? a.I : a.d;
            StageWalk sa(U, kst_down);
            for (int c = 0; c < U.stages; ++c, ++ts, sa.next()) {
                if (i == 0 && c < pre) continue;   // issued above
                const int s = ts % NSA;
                if (!ptx::mbar_wait_warp(&empty_a[s], ((ts / NSA) & 1) ^ 1, abort_flag, WAIT_NS)) {
                    if (lane == 0) fail(1);
                    ok = false;
                    break;
                }
                uint8_t* st = wst + s * C::A_STAGE;
                if (lane == 0) {
                    MOE_TR(TR_ISSUE, ts);
                    issue(U, sa, s);
                }
                if (!STMA) {
                    // e8m0 bytes of this stage: rows lane, lane+32, lane+64, lane+96, 4 bytes a
                    // 128-K half; a half past K (odd K/128) reads the row's first bytes (its
                    // codes are zero-filled, so they are multiplied by zero)
                    const uint8_t* sbase = U.down ? a.w2s : a.w13s;
                    const int kb = K / 32;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int r = lane + 32 * j;
                        const uint8_t* row = sbase + (size_t)weight_row(U, sa.blk, r, RD, a) * kb;
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int sub = 2 * sa.kc + hh;
                            ptx::cp_async_4(st + C::SC_OFF + 8 * r + 4 * hh, row + (sub * 4 < kb ? sub * 4 : 0));
                        }
                    }
                    ptx::cp_async_mbar_arrive_noinc(&full_a[s]);
                }
                __syncwarp();
            }
        }
        ptx::cp_async_wait_all();
    } else if (warp == SCHED_WARP) {
        // ------------------------------------------------------------ unit scheduler
        // CTA b's first unit is unit b; the later ones are claimed from the
        // counter (offset by the grid size).  The tile count, the first unit's
        // tile entry (read as if it were a gate_up unit, the usual case, and
        // read again below if not) and the second claim are all in flight at
        // once.
        const int n_tiles = ld_dep(&sb->n_tiles);
        const Tile tile0 = load_tile(a.tiles + min((int)blockIdx.x / mb1, a.max_tiles - 1));
        int claim1 = 0;
        if (lane == 0) claim1 = atomicAdd(&sb->work_next, 1);   // raw counter value
        const int U1 = n_tiles * mb1;
        const int total = U1 + n_tiles * g2;
        auto tile_of = [&](int u) { return u < U1 ? u / mb1 : (u - U1) / g2; };
        // Ring entry i is published once the weight producer has taken entry
        // i - 1, and only then is entry i + 1 claimed (its claim, then its tile
        // entry: a round trip of about two unit-stages, hidden behind the
        // stages of entry i - 1 and i still to issue).  So a CTA holds at most
        // two units beyond the one it streams when the counter runs out, and
        // the CTAs end within about a unit of one another.  Entry 1's claim
        // was issued at the start (a claim is kept as the raw counter value
        // until it is used: arithmetic on it would wait for the atomic).
        int u = (int)blockIdx.x;
        Tile tl = tile0;
        if (lane == 0) MOE_TR(TR_MISC, 3);
        if (u >= U1 && u < total) tl = load_tile(a.tiles + tile_of(u));
        for (int i = 0;; ++i) {
            Unit U;
            if (u < total) {
                unit_coords(u, U1, g2, a, U.down, U.tile, U.mb);
                U.e = tl.e;
                U.p0 = tl.p0;
                U.n = tl.n;
                U.nblk = U.down ? min(RD, mb2 - U.mb * RD) : 0;
                U.stages = U.down ? U.nblk * kst_down : (a.d + KS - 1) / KS;
                // a down unit's h rows, read now (a unit before the token
                // producer needs them): when complete, it skips its own wait
                U.h_ready = U.down ? (int)(ld_acquire_h(U) >= h_target(U)) : 0;
            } else {
                U.down = -1;
                U.tile = U.mb = U.e = U.p0 = U.n = U.stages = U.nblk = U.h_ready = 0;
            }
            bool go = true;
            if (lane == 0 && i >= LOOKAHEAD) {
                const uint64_t t0 = ptx::globaltimer();
                uint32_t it = 0;
                while (*taken < i - LOOKAHEAD + 1) {
                    __nanosleep(32);
                    if ((++it & 63u) == 0u && (*abort_flag || ptx::globaltimer() - t0 > WAIT_NS)) {
                        fail(15);
                        go = false;
                        break;
                    }
                }
            }
            if (!__shfl_sync(0xffffffffu, go ? 1 : 0, 0)) break;
            if (!ptx::mbar_wait_warp(&u_empty[i % UR], ((i / UR) & 1) ^ 1, abort_flag, WAIT_NS)) {
                if (lane == 0) fail(8);
                break;
            }
            if (lane == 0) {
                uring[i % UR] = U;
                ptx::mbar_arrive(&u_full[i % UR]);
                if (i == 0) MOE_TR(TR_MISC, 4);
            }
            if (U.down < 0) break;
            int claim = claim1;
            if (i > 0 && lane == 0) claim = atomicAdd(&sb->work_next, 1);
            u = (int)gridDim.x + __shfl_sync(0xffffffffu, claim, 0);
            if (u < total) tl = load_tile(a.tiles + tile_of(u));
            else u = total;
        }
    } else if (warp == TOK_WARP) {
        // ------------------------------------------------------------ token producer
        const uint64_t pol_x = ptx::policy_evict_last();
        const size_t tab_rows = (size_t)a.P + NT_MAX;
        int ts = 0;
        bool ok = true;
        // lane 0: token stage kc of unit U (x rows, or h rows for a down unit)
        // and its block scales into ring slot s
        auto issue = [&](const Unit& U, int kc, int s) {
            uint8_t* st = tst + s * C::B_STAGE;
            const CUtensorMap* tmB = U.down ? &tm_hq : &tm_xq;
            const uint8_t* tab = U.down ? a.hs : a.xs;
            ptx::mbar_arrive_expect_tx(&full_b[s], B_SMEM + BS_BYTES);
            ptx::tma_load_3d(st, tmB, 0, 2 * U.p0, 2 * kc, &full_b[s], pol_x);
            ptx::bulk_load(tsc + s * BS_BYTES, tab + ((size_t)kc * tab_rows + U.p0) * TOKEN_SCALE_ROW, BS_BYTES,
                           &full_b[s], pol_x);
        };
        // the first unit's first stages, before it comes through the ring
        int pre = 0;
        {
            Unit U0;
            if (lane == 0 && first_gate_up_unit(a, U0)) {
                pre = min(NSB, U0.stages);
                for (int c = 0; c < pre; ++c) issue(U0, c, c);   // gate_up: stage c reads K chunk c
            }
            pre = __shfl_sync(0xffffffffu, pre, 0);
        }
        for (int i = 0; ok; ++i) {
            Unit U;
            if (!take_unit(i, U)) {
                if (lane == 0) fail(12);
                break;
            }
            if (U.down < 0) break;
            if (U.down) {
                // the tile's h rows: complete once all its gate_up units are
                // done (seen by the scheduler already, or waited for here);
                // the scheduler's acquire orders them before its ring entry,
                // which this warp's wait on the entry orders before its copies
                uint32_t ready = 0;
                if (lane == 0) {
                    const uint64_t t0 = ptx::globaltimer();
                    uint32_t it = 0;
                    ready = 1;
                    const uint32_t target = h_target(U);
                    while (!U.h_ready && ptx::ld_acquire_gpu(&a.tile_ready[U.tile]) < target) {
                        __nanosleep(32);
                        if ((++it & 63u) == 0u && (*abort_flag || ptx::globaltimer() - t0 > WAIT_NS_H)) {
                            fail(2);
                            ready = 0;
                            break;
                        }
                    }
                    if (ready) ptx::fence_proxy_async_global();
                }
                if (!__shfl_sync(0xffffffffu, ready, 0)) break;
            }
            StageWalk sw(U, kst_down);
            for (int c = 0; c < U.stages; ++c, ++ts, sw.next()) {
                if (i == 0 && c < pre) continue;   // issued above
                const int s = ts % NSB;
                if (!ptx::mbar_wait_warp(&empty_b[s], ((ts / NSB) & 1) ^ 1, abort_flag, WAIT_NS)) {
                    if (lane == 0) fail(13);
                    ok = false;
                    break;
                }
                // a down unit's blocks read the same h rows: stage kc of h
                if (lane == 0) issue(U, sw.kc, s);
                __syncwarp();
            }
        }
    } else if (warp >= SF_WARP0 && warp < SF_WARP0 + 4) {
        // ------------------------------------------------------------ scale movers
        const int q = warp - SF_WARP0;    // TMEM lane quarter of this warp
        const int r = 32 * q + lane;      // weight row of this thread
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        int ts = 0;
        bool ok = true;
        for (int i = 0; ok; ++i) {
            Unit U;
            if (!take_unit(i, U)) {
                if (lane == 0) fail(10);
                break;
            }
            if (U.down < 0) break;
            StageWalk sa(U, kst_down);
            for (int c = 0; c < U.stages; ++c, ++ts, sa.next()) {
                const int s = ts % NSA, sbi = ts % NSB;
                if (!ptx::mbar_wait_warp(&full_a[s], (ts / NSA) & 1, abort_flag, WAIT_NS) ||
                    !ptx::mbar_wait_warp(&full_b[sbi], (ts / NSB) & 1, abort_flag, WAIT_NS)) {
                    if (lane == 0) fail(5);
                    ok = false;
                    break;
                }
                if (q == 0 && lane == 0) MOE_TR(TR_LANDED, ts);
                const uint8_t* st = wst + s * C::A_STAGE;
                const int kc = sa.kc;
                const int owner = c % NMMA;   // the stage's MMA issuer
                const uint2 wa = *reinterpret_cast<const uint2*>(st + C::SC_OFF + C::SC_ROW * r + (STMA ? 8 * (kc & 1) : 0));
                // token column n = 32 g + lane (g < BSG): pick n / 2 (its hi and lo
                // row); columns past the tile's 2 NTT are never read
                uint32_t bx[C::BSG], by[C::BSG];
#pragma unroll
                for (int g = 0; g < C::BSG; ++g) {
                    const uint2 wb = *reinterpret_cast<const uint2*>(
                        tsc + sbi * BS_BYTES + TOKEN_SCALE_ROW * ((16 * g + (lane >> 1)) & (NTT - 1)));
                    bx[g] = wb.x;
                    by[g] = wb.y;
                }
                // 0xFF is NaN in e8m0
                const uint32_t nan_a = __vcmpeq4(wa.x, 0xFFFFFFFFu) | __vcmpeq4(wa.y, 0xFFFFFFFFu);
                if (nan_a) latch_status(sb, MOE_ERR_BAD_SCALE, 255);
                const uint32_t col = SF_COL0 + s * SF_SLOT;
                // row r = 32q + lane is read at column col + q (K steps 0-3) and
                // col + SF_A1 + q (K steps 4-7); the warp writes its word into all
                // four columns of a group (aligned stores): the other lane quarters'
                // columns of these lanes are never read
                ptx::tmem_st4_rep(tmem + lane_base + col, wa.x);
                ptx::tmem_st4_rep(tmem + lane_base + col + SF_A1, wa.y);
                // token column n: lane n mod 32 of every lane quarter, column + n / 32
                if constexpr (C::BSG == 1) {
                    ptx::tmem_st4_rep(tmem + lane_base + col + SF_B0, bx[0]);
                    ptx::tmem_st4_rep(tmem + lane_base + col + SF_B1, by[0]);
                } else if constexpr (C::BSG == 2) {
                    ptx::tmem_st2(tmem + lane_base + col + SF_B0, bx[0], bx[1]);
                    ptx::tmem_st2(tmem + lane_base + col + SF_B1, by[0], by[1]);
                } else {
                    static_assert(C::BSG == 4, "token scale groups of one, two or four columns");
                    ptx::tmem_st4(tmem + lane_base + col + SF_B0, bx[0], bx[1], bx[2], bx[3]);
                    ptx::tmem_st4(tmem + lane_base + col + SF_B1, by[0], by[1], by[2], by[3]);
                }
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sf_full[owner * NSA + s]);
            }
        }
    } else if (warp >= MMA_WARP0 && warp < MMA_WARP0 + NMMA) {
        // ------------------------------------------------------------ MMA issuers
        // Issuer m takes the stages c of every unit with c mod NMMA == m (all
        // eight K steps of each), so two issue loops overlap on different
        // stages.  It waits only on sf_full: the scale movers arrive there
        // after they have waited on the stage's weight and token barriers, so
        // both TMA copies are complete and visible once sf_full completes.
        const int m = warp - MMA_WARP0;
        int ts = 0;
        uint32_t sf_par = 0;   // bit s: parity of the next phase of this issuer's sf_full[s]
        for (int i = 0;; ++i) {
            Unit U;
            if (!take_unit(i, U)) {
                if (lane == 0) fail(9);
                break;
            }
            if (U.down < 0) break;
            bool ok = true;
            if (lane == 0) {
                const int ab = i % ACCB;
                // every issuer waits for the accumulator buffer of every unit
                // (drained by the epilogue ACCB units back), also when it has no
                // stage in it, so that it never waits two phases ahead
                if (!ptx::mbar_wait(&acc_empty[ab], ((i / ACCB) & 1) ^ 1, abort_flag, WAIT_NS)) {
                    fail(3);
                    ok = false;
                }
                if (m == 0) MOE_TR(TR_ACCE, i);
                StageWalk sa(U, kst_down);
                for (int c = 0; ok && c < U.stages; ++c, ++ts, sa.next()) {
                    // issuer m takes the stages c = m (mod NMMA) of the unit; stage
                    // kc of row block b goes to accumulator slot kc mod NMMA of the
                    // block (every stage of a slot has the same issuer)
                    if (c % NMMA != m) continue;
                    const uint32_t d_tmem = tmem + ab * BW + (sa.blk * NMMA + sa.kc % NMMA) * NB;
                    const bool acc = sa.kc >= NMMA;
                    const int s = ts % NSA, sbi = ts % NSB;
                    if (!ptx::mbar_wait(&sf_full[m * NSA + s], (sf_par >> s) & 1u, abort_flag, WAIT_NS)) {
                        fail(4);
                        ok = false;
                        break;
                    }
                    sf_par ^= 1u << s;
                    MOE_TR(TR_MMA, ts);
                    ptx::tc_fence_after();
                    const uint32_t a0 = ptx::smem_u32(wst + s * C::A_STAGE);
                    const uint32_t b0 = ptx::smem_u32(tst + sbi * C::B_STAGE);
                    const uint32_t col = SF_COL0 + s * SF_SLOT;
#pragma unroll
                    for (int kk = 0; kk < KS / 32; ++kk) {
                        const int h = kk >> 2, j = kk & 3;   // 128-K slab, K step within it
                        ptx::mma_mx_ss(d_tmem, ptx::smem_desc_sw128(a0 + h * A_SLAB + 32 * j),
                                       ptx::smem_desc_sw128(b0 + h * B_SLAB + 32 * j),
                                       ptx::idesc_mx_e2m1_e4m3(AROWS, NB, j, j), (acc || kk > 0) ? 1u : 0u,
                                       tmem + col + SF_A1 * h, tmem + col + SF_B0 + (SF_B1 - SF_B0) * h);
                    }
                    ptx::mma_commit(&empty_a[s]);
                    ptx::mma_commit(&empty_b[sbi]);
                }
                // an issuer without a stage in this unit (one-stage units) commits
                // nothing of its own; the epilogue reads only the issuers that had one
                if (ok) ptx::mma_commit(&acc_full[ab]);
            }
            ts = __shfl_sync(0xffffffffu, ts, 0);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
        }
        if (lane == 0) {
            // every MMA issued above has completed before TMEM is released
            ptx::mma_commit(&fin[m]);
            ptx::mbar_wait(&fin[m], 0, abort_flag, WAIT_NS);
        }
        __syncwarp();
    } else if (warp >= MMA_WARP0 && warp < MMA_WARP0 + NMMA_MAX) {
        // an issuer warp with nothing to do: the widest tiles have a single issuer
    } else {
        // ------------------------------------------------------------ epilogue
        const int qd = warp & 3;
        const int r = 32 * qd + lane;
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        const size_t tab_rows = (size_t)a.P + NT_MAX;
        for (int i = 0;; ++i) {
            const int ab = i % ACCB;
            // the four epilogue warps take one decision before their named
            // barriers: carry on, or leave together (they all read the same
            // ring entry, so they all see the end of the units together)
            Unit U;
            const bool got = take_unit(i, U);
            if (!got && lane == 0) fail(11);
            const bool end = got && U.down < 0;
            if (!end && !*abort_flag && !ptx::mbar_wait_warp(&acc_full[ab], (i / ACCB) & 1, abort_flag, WAIT_NS) &&
                lane == 0)
                fail(7);
            // one barrier a unit: the decision flags alternate, so that a flag
            // is written again only after every warp has passed the next barrier
            if (threadIdx.x == EPI_WARP0 * 32) epi_flag[i & 1] = *abort_flag;
            ptx::named_bar_sync(1, 128);
            if (epi_flag[i & 1] || end) break;
            if (threadIdx.x == EPI_WARP0 * 32) MOE_TR(TR_EPI, i);
            ptx::tc_fence_after();
            // accumulators of a row block: one per issuer slot that had a stage
            // in the block, added
            const int kst_blk = U.down ? kst_down : U.stages;
            const int nacc = kst_blk < NMMA ? kst_blk : NMMA;
            // the tile's picks in chunks of EC: v[n] = the block's accumulators,
            // hi + lo column of pick ch + n (8-pick chunks: every TMEM load in
            // flight before one wait; wider chunks one accumulator at a time,
            // within the registers a thread has)
            auto read_chunk = [&](uint32_t acc_col, int ch, float (&v)[EC]) {
                constexpr int NL = EC <= 8 ? NMMA : 1;   // accumulators loaded before a wait
#pragma unroll
                for (int n = 0; n < EC; ++n) v[n] = 0.f;
#pragma unroll
                for (int m0 = 0; m0 < NMMA; m0 += NL) {
                    if (m0 >= nacc) break;
                    uint32_t t[NL][2 * EC];
#pragma unroll
                    for (int mm = 0; mm < NL; ++mm) {
                        if (m0 + mm < nacc) {
#pragma unroll
                            for (int j = 0; j < 2 * EC / 16; ++j)
                                ptx::tmem_ld16(tmem + lane_base + acc_col + (m0 + mm) * NB + 2 * ch + 16 * j,
                                               t[mm] + 16 * j);
                        }
                    }
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int mm = 0; mm < NL; ++mm) {
                        if (m0 + mm < nacc) {
#pragma unroll
                            for (int n = 0; n < EC; ++n)
                                v[n] += __uint_as_float(t[mm][2 * n]) + __uint_as_float(t[mm][2 * n + 1]);
                        }
                    }
                }
            };
            auto release_acc = [&]() {   // the unit's accumulators are read out
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&acc_empty[ab]);
            };
            if (!U.down) {
                const int ii = U.mb * 64 + r;        // h row of lanes 0..63
                const int blk = ii / 32;             // its 32-row block of h
#pragma unroll 1
                for (int ch = 0; ch < NTT; ch += EC) {
                    float v[EC];
                    read_chunk(ab * BW, ch, v);
                    if (ch + EC >= NTT) release_acc();
                    // lanes 0..63: gate of rows mb*64 + r; lanes 64..127: up of the same rows
                    if (r >= 64) {
#pragma unroll
                        for (int n = 0; n < EC; ++n) xch[(r - 64) * C::XCH_STRIDE + n] = v[n];
                    }
                    ptx::named_bar_sync(1, 128);
                    if (r < 64) {
                        // warp qd (0 or 1) holds the 32 rows of h block mb*2 + qd
                        float h[EC];
#pragma unroll
                        for (int n = 0; n < EC; ++n) {
                            const float gv = v[n];
                            const float uv = xch[r * C::XCH_STRIDE + n];
                            h[n] = ch + n < U.n ? gv / (1.0f + __expf(-gv)) * uv : 0.f;
                        }
#pragma unroll
                        for (int n = 0; n < EC; n += 2) {
                            uint32_t byte2[2];
                            float hs2[2];
#pragma unroll
                            for (int z = 0; z < 2; ++z) {
                                const uint32_t amax = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h[n + z])));
                                int e = (int)((amax >> 23) & 0xFFu) - 7;
                                e = e < 1 ? 1 : (e > 247 ? 247 : e);
                                byte2[z] = (uint32_t)e;
                                hs2[z] = h[n + z] * __uint_as_float((uint32_t)(254 - e) << 23);   // h / 2^(e - 127)
                            }
                            const uint32_t hi2 = ptx::cvt_e4m3x2(hs2[0], hs2[1]);
                            float f0, f1;
                            ptx::e4m3x2_to_f32(hi2, f0, f1);
                            const uint32_t lo2 = ptx::cvt_e4m3x2(hs2[0] - f0, hs2[1] - f1);
#pragma unroll
                            for (int z = 0; z < 2; ++z) {
                                if (ch + n + z < U.n) {
                                    const size_t p = (size_t)(U.p0 + ch + n + z);
                                    a.hq[(2 * p) * a.I + ii] = (uint8_t)(hi2 >> (8 * z));
                                    a.hq[(2 * p + 1) * a.I + ii] = (uint8_t)(lo2 >> (8 * z));
                                    if (lane == 0)
                                        a.hs[((size_t)(blk >> 3) * tab_rows + p) * TOKEN_SCALE_ROW + (blk & 7)] =
                                            (uint8_t)byte2[z];
                                }
                            }
                        }
                    }
                    ptx::named_bar_sync(1, 128);   // xch is written again by the next chunk
                }
            } else {
#pragma unroll 1
                for (int b = 0; b < U.nblk; ++b) {
                    const int yrow = (U.mb * RD + b) * AROWS + r;   // row of y
#pragma unroll 1
                    for (int ch = 0; ch < NTT; ch += EC) {
                        float v[EC];
                        read_chunk(ab * BW + b * NMMA * NB, ch, v);
                        if (b + 1 == U.nblk && ch + EC >= NTT) release_acc();
#pragma unroll
                        for (int n = 0; n < EC; ++n)
                            if (ch + n < U.n) a.y[(size_t)(U.p0 + ch + n) * a.d + yrow] = v[n];
                        if (a.ssq != nullptr) {
                            // sum of y^2 over the block's 128 rows for every pick of the
                            // chunk: a reduce-scatter across the warp (lane l ends with
                            // pick idx), then (below) the four warps' sums in warp order
                            float q[EC];
#pragma unroll
                            for (int n = 0; n < EC; ++n) q[n] = v[n] * v[n];
                            int idx = 0;
#pragma unroll
                            for (int step = 0; step < 5; ++step) {
                                const int o = 16 >> step;
                                const int c = EC >> step;       // values a lane holds before this step
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
                            // every pick's sum now sits on 32 / EC lanes
                            float* part = xch;                             // [4][NTT]
                            if ((lane & (32 / EC - 1)) == 0) part[qd * NTT + ch + idx] = q[0];
                        }
                    }
                    if (a.ssq != nullptr) {
                        const float* part = xch;
                        ptx::named_bar_sync(1, 128);
                        for (int pr = r; pr < U.n; pr += 128)
                            a.ssq[(size_t)(U.p0 + pr) * mb2 + (U.mb * RD + b)] =
                                ((part[pr] + part[NTT + pr]) + part[2 * NTT + pr]) + part[3 * NTT + pr];
                        ptx::named_bar_sync(1, 128);   // part is written again by the next block or unit
                    }
                }
            }
            if (!U.down) {
                // the writers' h rows, generic stores, are read by other CTAs'
                // TMA copies: each writer fences its stores against the async
                // proxy, the barrier orders them before the release (a release
                // is cumulative over what its thread has synchronised with)
                if (r < 64) ptx::fence_proxy_async_global();
                ptx::named_bar_sync(1, 128);
                if (warp == EPI_WARP0 && lane == 0) ptx::red_release_gpu_add(&a.tile_ready[U.tile], 1u);
            }
        }
    }

    __syncthreads();
    if (threadIdx.x == 0) MOE_TR(TR_MISC, 2);
    KT_MARK(K_EXPERTS, 2);
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
template <bool STMA, int NTT>
cudaError_t launch_mx(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    using C = Cfg<STMA, NTT>;
    CUtensorMap tm_w13, tm_w2, tm_xq, tm_hq, tm_w13s, tm_w2s;
    const uint64_t P = (uint64_t)L.max_picks, E = s.E, d = s.d, I = s.I;
    const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8, U4 = CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B;
    // w13 [E][2][I][d/2] as 4-bit codes {128 codes, I rows, 2E halves, d/128 slabs}
    const uint64_t w13_d[4] = {128, I, 2 * E, d / 128}, w13_s[3] = {d / 2, I * d / 2, 64};
    const uint32_t w13_b[4] = {128, 64, 2, 2};
    // w2 [E][d][I/2] as {128 codes, E d rows, I/128 slabs}
    const uint64_t w2_d[3] = {128, E * d, I / 128}, w2_s[2] = {I / 2, 64};
    const uint32_t w2_b[3] = {128, AROWS, 2};
    // xq [2P][d] / hq [2P][I] e4m3 as {128 bytes, 2P rows, K/128 slabs}
    const uint64_t xq_d[3] = {128, 2 * P, d / 128}, xq_s[2] = {d, 128};
    const uint64_t hq_d[3] = {128, 2 * P, I / 128}, hq_s[2] = {I, 128};
    const uint32_t tok_b[3] = {128, (uint32_t)C::NB, 2};
    if (!make_map(&tm_w13, U4, p.w13, 4, w13_d, w13_s, w13_b, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tm_w2, U4, p.w2, 3, w2_d, w2_s, w2_b, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tm_xq, U8, p.ws + L.xq, 3, xq_d, xq_s, tok_b, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tm_hq, U8, p.ws + L.hq, 3, hq_d, hq_s, tok_b, CU_TENSOR_MAP_SWIZZLE_128B))
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
    cudaError_t e = cudaFuncSetAttribute(k_experts_mx<STMA, NTT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    Args a;
    a.tiles = reinterpret_cast<const Tile*>(p.ws + L.tiles);
    a.sb = reinterpret_cast<StatusBlock*>(p.ws + L.status);
    a.w13s = p.w13s;
    a.w2s = p.w2s;
    a.hq = reinterpret_cast<uint8_t*>(p.ws + L.hq);
    a.hs = reinterpret_cast<uint8_t*>(p.ws + L.hs);
    a.y = reinterpret_cast<float*>(p.ws + L.y);
    a.ssq = p.norm_w != nullptr ? reinterpret_cast<float*>(p.ws + L.ssq) : nullptr;
    a.tile_ready = reinterpret_cast<uint32_t*>(p.ws + L.tile_ready);
    a.xs = reinterpret_cast<const uint8_t*>(p.ws + L.xs);
    a.d = s.d;
    a.I = s.I;
    a.P = L.max_picks;
    a.max_tiles = L.max_tiles;
#ifdef MOE_WAIT_TEST
    a.unreachable = g_unreachable_wait;
#endif
    return launch_pdl(k_experts_mx<STMA, NTT>, dim3(num_sms()), dim3(NUM_THREADS), C::SMEM, st, tm_w13, tm_w2, tm_xq, tm_hq,
                      tm_w13s, tm_w2s, a);
}

}  // namespace

// Tensor-map and device helpers shared with the router's tensor-core kernel.
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

cudaError_t launch_experts(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    KT_BIND();
    timing_begin(K_EXPERTS, st);
    const bool stma = (s.d % 512 == 0) && (s.I % 512 == 0);
    cudaError_t e;
    if (L.nt == 8)
        e = stma ? launch_mx<true, 8>(s, L, p, st) : launch_mx<false, 8>(s, L, p, st);
    else if (L.nt == 16)
        e = stma ? launch_mx<true, 16>(s, L, p, st) : launch_mx<false, 16>(s, L, p, st);
    else if (L.nt == 32)
        e = stma ? launch_mx<true, 32>(s, L, p, st) : launch_mx<false, 32>(s, L, p, st);
    else
        e = stma ? launch_mx<true, 64>(s, L, p, st) : launch_mx<false, 64>(s, L, p, st);
    timing_end(st);
    return e;
}

}  // namespace moe

#ifdef MOE_TRACE
// Diagnostics export of the trace build: copies the stamp table to `dst`
// (host memory, `bytes` <= its size), after synchronising the device.
// dst == NULL clears the table instead.
extern "C" int moe_trace_copy(void* dst, size_t bytes) {
    if (bytes > sizeof(moe::g_trace)) bytes = sizeof(moe::g_trace);
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    if (dst == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, moe::g_trace) != cudaSuccess) return MOE_ERR_CUDA;
        return cudaMemset(p, 0, sizeof(moe::g_trace)) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    return cudaMemcpyFromSymbol(dst, moe::g_trace, bytes) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
#endif

#ifdef MOE_WAIT_TEST
// Test-only export of the wait-test build: on != 0 makes the next launches'
// first down unit of tile 0 wait for a count no kernel reaches, so its bounded
// wait runs out (MOE_ERR_TIMEOUT, detail 2) and the kernel takes its abort path.
extern "C" int moe_test_unreachable_wait(int on) {
    moe::g_unreachable_wait = on != 0;
    return 0;
}
#endif
