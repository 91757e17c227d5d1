// Internal declarations shared by the translation units of libmoe.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

#include <utility>

namespace moe {

// ---------------------------------------------------------------------------
// device status block (first 256 bytes of the workspace)
// ---------------------------------------------------------------------------
struct StatusBlock {
    int32_t status;     // first latched MOE_ERR_* (0 = none)
    int32_t detail;     // code-specific detail of that error
    int32_t n_picks;    // valid picks of the current call (written by the sort)
    int32_t n_tiles;    // gate_up work tiles of the current call
    int32_t work_next;  // persistent-kernel work counters (reset each call)
    int32_t work_next2;
    int32_t count_done; // CTAs of the counting kernel done (its last CTA resets it)
    int32_t pad[57];
};
static_assert(sizeof(StatusBlock) == 256, "status block is 256 bytes");

// Token-tile width of the expert GEMMs: one tile holds up to nt picks of one
// expert (an MMA N of 2 nt: hi and lo row per pick), nt = 16 (the pages'
// 16-row tiles, k5 page), 8 when the call's experts get few picks each, 32 or
// 64 when they get many.
constexpr int NT_MAX = 64;
int tile_picks(const moe_shape& s);

// Block scales of the gathered tokens and of h (e8m0, one per 32 elements):
// a table [ceil(K/256) stages][P + NT picks][TOKEN_SCALE_ROW bytes], bytes
// 0..7 of a row holding the stage's eight scales (16-byte rows, so that the
// rows of a tile are one aligned bulk copy; NT_MAX rows of padding so that
// the last tile's copy stays inside the table).
constexpr int TOKEN_SCALE_ROW = 16;

// The sort counters of the picks above 128 (right after the status block):
// cnt [E] picks per expert, off [E] segment offsets, cnt2 [E] picks placed
// per expert; E <= 512.  Zero before a call (moe_workspace_init, and every
// call leaves them so), with the status block the workspace's zeroed prefix.
constexpr int SORT_CNT_MAX_E = 512;
constexpr size_t SORT_CNT_BYTES = 3 * SORT_CNT_MAX_E * sizeof(int32_t);
constexpr size_t WS_ZERO_PREFIX = sizeof(StatusBlock) + SORT_CNT_BYTES;

// One work tile: expert e, first sorted pick p0, n picks (n <= nt).
struct Tile {
    int32_t e, p0, n, pad;
};

// Byte offsets of the workspace regions (all 256-byte aligned).
struct WsLayout {
    size_t status, sortcnt, logits, pos, tiles, tile_ready, xq, xs, hq, hs, y, ssq;
    size_t xin, hio_ids, hio_w, hio_out;  // moe_forward_host staging
    size_t total;
    int max_tiles;
    int nt;               // picks per tile (8 or 16)
    int max_picks;
    int router_kslices;   // K-ranges of the router (CTAs of one cluster)
};

WsLayout ws_layout(const moe_shape& s);

// moe_forward's host-side checks except the workspace's (moe_abi.cu)
int check_forward_args(const moe_shape* s, const void* x, const void* w_gate, const float* bias,
                       const float* logit_off, const uint8_t* w13, const uint8_t* w13s, const uint8_t* w2,
                       const uint8_t* w2s, const float* norm_w, const int32_t* ids, const float* w,
                       const float* out);

// Host helpers of the tensor-core kernels (experts_mx.cu): a rank-r tiled
// tensor map (dims[0] innermost; strides[i] = byte stride of dims[i+1]) and
// the device's SM count.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw);
int num_sms();
int router_kslices(const moe_shape& s, int num_sms);

__device__ __forceinline__ void latch_status(StatusBlock* sb, int code, int detail) {
    if (atomicCAS(&sb->status, 0, code) == 0) sb->detail = detail;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  The block's kernels are launched so that the
// next one may start while its predecessor is still running: a kernel allows
// its successor to launch (pdl_trigger), does the work that needs no
// predecessor's data, and calls pdl_wait, which returns when the predecessor
// grid has completed and its writes are visible, before it reads or writes
// anything the stream's earlier kernels of the call touch.  The first kernel
// of a call triggers only after its own wait has returned, i.e. once the
// stream's work before the call (which wrote x) has completed; every later
// kernel triggers at its start.  So before its wait a kernel may read the
// call's inputs (weights, bias, x), which none of the block's kernels writes.
// Without the launch attribute pdl_wait returns at once.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Loads of what an earlier kernel of the call wrote go through L2 (ld.global.cg):
// that kernel may still have been running when this one started, so the data
// is not read-only for this kernel's lifetime, which the non-coherent path
// (__ldg, or a const __restrict__ pointer the compiler may read that way)
// requires; a stale line there was seen to survive the wait.
template <typename T>
__device__ __forceinline__ T ld_dep(const T* p) { return __ldcg(p); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// per-kernel timing hooks (moe_timing_*): no-ops unless enabled
// ---------------------------------------------------------------------------
enum KernelId {
    K_ROUTER = 0, K_TOPK, K_SORT, K_GATHER, K_EXPERTS, K_COMBINE, K_ROUTE_GATHER,
    K_LATENT_DOWN, K_LATENT_MID, K_LATENT_UP, K_NUM
};
void timing_begin(int kernel_id, cudaStream_t st);
void timing_end(cudaStream_t st);

// Diagnostics build (-DMOE_TRACE): every CTA of the library's kernels stamps
// %globaltimer at its start (point 0), after its wait on the preceding kernel
// (1), at its end (2) and at kernel-specific points 3..7 into a table
// [K_NUM][8 points][min, max] (moe_ktrace).  The table lives in device memory the trace
// build allocates (timing.cu); each translation unit binds its own copy of the
// pointer before its first launch.
#ifdef MOE_TRACE
constexpr int KT_SLOTS = 16;
extern unsigned long long* g_kt_dev;
static __constant__ unsigned long long* g_ktp;
static bool g_kt_bound = false;
static inline void kt_bind() {
    if (!g_kt_bound && g_kt_dev != nullptr) {
        cudaMemcpyToSymbol(g_ktp, &g_kt_dev, sizeof(g_kt_dev));
        g_kt_bound = true;
    }
}
// what: 0 start, 1 after the wait, 2 end, 3..7 inner points (thread 0 of the CTA)
__device__ __forceinline__ void kt_mark(int kid, int what) {
    if (threadIdx.x != 0 || threadIdx.y != 0 || g_ktp == nullptr) return;
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    atomicMin(g_ktp + kid * KT_SLOTS + 2 * what, t);
    atomicMax(g_ktp + kid * KT_SLOTS + 2 * what + 1, t);
}
#define KT_BIND() kt_bind()
#define KT_MARK(kid, what) kt_mark(kid, what)
#else
#define KT_BIND() \
    do {          \
    } while (0)
#define KT_MARK(kid, what) \
    do {                   \
    } while (0)
#endif

// ---------------------------------------------------------------------------
// launchers (one per kernel); all return cudaGetLastError() of the launch
// ---------------------------------------------------------------------------
struct Ptrs {
    const __nv_bfloat16* x;
    const __nv_bfloat16* w_gate;
    const float* bias;
    const float* logit_off;
    const uint8_t* w13;
    const uint8_t* w13s;
    const uint8_t* w2;
    const uint8_t* w2s;
    const float* norm_w;
    int32_t* ids;
    float* weights;
    float* out;
    char* ws;
};

cudaError_t launch_router_logits(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st);
// the router's tensor-core kernel (9 <= S <= 32 or S >= 64, E a multiple of 128)
bool router_tc_fits(const moe_shape& s);
cudaError_t launch_router_tc(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st);
// dense bf16 product out[S, N] = x[S, K] . w[N, K]^T on the tensor cores
// (route_tc.cu): N % 128 == 0, K % 64 == 0; out fp32 (store, or add to what
// the stream's earlier kernels wrote) or bf16
enum DenseOut { DENSE_F32 = 0, DENSE_F32_ADD = 1, DENSE_BF16 = 2 };
bool dense_fits(int S, int K, int N);
// (kt_id: the KernelId its diagnostics stamps go under)
cudaError_t launch_dense(const void* x, const void* w, int S, int K, int N, const float* off, void* out, int mode,
                         StatusBlock* sb, cudaStream_t st, int kt_id);
// up to three products of the same x in one launch: part i = x . w^T into
// out (N cols a token, mode), the logit offset added to part 0's; or
// x . w^T + x2 . w2^T (K and K2 long rows) into one out
struct DensePart {
    const void* w;
    int N;
    void* out;
    int mode;
};
cudaError_t launch_dense_ncat(const void* x, int S, int K, const DensePart* p, int n_parts, const float* off,
                              StatusBlock* sb, cudaStream_t st, int kt_id);
cudaError_t launch_dense_kcat(const void* x, const void* w, int K, const void* x2, const void* w2, int K2, int S,
                              int N, void* out, int mode, StatusBlock* sb, cudaStream_t st, int kt_id);
cudaError_t launch_topk(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st);
cudaError_t launch_route(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st);
// moe_forward at small S: top-k, sort and gather in one kernel (needs the
// logits); above 128 picks the top-k kernel first, then sort and gather
bool topk_sort_fits(const moe_shape& s);
// ... and the fused kernel selects the top k itself (no top-k kernel before it)
bool route_gather_selects(const moe_shape& s);
// (x_after_wait: the rows to gather were written by an earlier kernel of the
// call, not an input of it)
cudaError_t launch_topk_sort_gather(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st,
                                    bool x_after_wait = false);
// the ids given (moe_experts, or the top-k kernel's); x_after_wait as above
cudaError_t launch_sort_gather(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st,
                               bool x_after_wait = false);
cudaError_t launch_experts(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st);
cudaError_t launch_combine(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st);
// the latent-MoE layer's elementwise steps (latent.cu)
// zl = bf16(RMSNorm(yl) ln_w) and, when si > 0, hs = bf16(silu(g) u) of the
// shared expert's gate/up rows gu, in one launch (n <= 16384, n % 4 == 0)
bool latent_mid_fits(int n);
cudaError_t launch_latent_mid(const float* yl, const float* ln_w, float eps, int S, int n, __nv_bfloat16* zl,
                              const float* gu, int si, __nv_bfloat16* hs, cudaStream_t st);

}  // namespace moe
