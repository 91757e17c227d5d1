/*
 * moe.h -- C ABI of libmoe: the routed MXFP4 mixture-of-experts block of a
 * speculative-decode verify step, on one GB300 GPU (sm_103a), all experts
 * resident, no collectives.
 *
 * The block (pages cited by their vLLM module names):
 *   vllm.models.muse_spark.amd.mono.kernels.k3, stage list:
 *     A      the router's logits, in fp32
 *     route  the top 8 of every token (each CTA repeats the same routing);
 *            route_token starts from a sigmoid score (its summary is cut off)
 *     C, D   the local experts' gate_up and down projections, MXFP4 weights
 *     E      a norm of each pick's expert output, then the weighted sum
 *   vllm.models.muse_spark.amd.mono.kernels.k5, stage HA: fp32 router, top 8,
 *     ids and weights handed to the expert stage
 *   vllm.models.kimi_k3.amd.specialized_decode.mono.layer, k2_launch: the MoE
 *     arguments w_gate, bias, w13, w13s, w2, w2s and the output out [S, 7168].
 *
 * What is computed, for token t (0 <= t < S):
 *   L[t,e]   = sum_c x[t,c] * w_gate[e,c]  (fp32)  [+ logit_off[e]]
 *   s[t,e]   = sigmoid(L[t,e]);  sel = s + bias[e]
 *   picks    = the k experts with the largest sel (ties -> lower id),
 *              reported in ascending expert id; weight w_j = s_j / sum_j s_j
 *   g, u     = W1_e x_t, W3_e x_t   (W1 = rows 0..I-1 of w13, W3 = rows I..2I-1)
 *   h        = silu(g) * u;   y = W2_e h
 *   [post]   y <- y * rsqrt(mean(y^2) + norm_eps) * norm_w      (MOE_POST_NORM)
 *   out[t]   = sum_j w_j * y_j                                      (fp32)
 *
 * MXFP4 encoding (OCP Microscaling v1.0): an e2m1 element is a 4-bit code
 * (sign, 2 exponent bits with bias 1, 1 mantissa bit); an e8m0 scale byte b
 * means 2^(b-127) and covers 32 consecutive K-elements of one row.  Packed
 * rows are row-major with K contiguous: byte j holds element 2j in its low
 * nibble and element 2j+1 in its high nibble.  Scale bytes 0..254 (block
 * scales 2^-127 .. 2^127) are supported; the byte 255, NaN in the MX format,
 * latches MOE_ERR_BAD_SCALE on the device (the affected outputs are NaN).
 *
 * Precision: the expert GEMMs run on the tensor core's block-scaled e2m1 x
 * e4m3 path with fp32 accumulation.  The weights enter exactly; each bf16
 * token row enters as two e4m3 rows (leading and trailing 4 significant
 * bits) under a power-of-two scale per 32 elements, which is exact up to
 * 2^-17 of the block's largest magnitude; h = silu(g) * u enters the same
 * way from fp32 (about 9 significant bits, like a bf16 rounding).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers (cudaMalloc'd or equivalent),
 *     16-byte aligned (the packed weights w13 and w2: 32-byte aligned),
 *     owned by the caller, and must stay valid until the
 *     work queued on `stream` has finished.  Nothing is allocated, freed or
 *     cached by the library on these paths; it keeps no state between calls
 *     except per-device kernel attributes.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls only enqueue work; they do not synchronise, except
 *     moe_device_status.  The library's kernels are launched with
 *     programmatic dependent launch: later kernels of a call read its inputs
 *     (weights, bias, x) before waiting on their predecessors, which is safe
 *     because the call's first kernel lets them start only once the stream's
 *     earlier work has completed.  A caller kernel launched the same way that
 *     writes an input must therefore not signal launch completion before the
 *     input is written.
 *   - `ws` is a device workspace of at least moe_workspace_bytes() bytes,
 *     256-byte aligned, prepared once with moe_workspace_init.  Its first
 *     bytes hold the device status word; calls that share one workspace must
 *     be ordered on one stream.
 *   - Return value: MOE_OK or a negative MOE_ERR_* code.  Host-side checks
 *     (arguments, shape, alignment, workspace size) run before anything is
 *     enqueued and enqueue nothing when they fail.  Errors found on the
 *     device (bad ids, bad scale bytes, a bounded wait that ran out) are
 *     latched in the workspace status word and reported by
 *     moe_device_status.  The library never aborts, traps or asserts.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1

/* status codes */
#define MOE_OK                     0
#define MOE_ERR_INVALID_ARG       -1  /* NULL pointer, negative size, bad flags */
#define MOE_ERR_UNSUPPORTED_SHAPE -2  /* shape outside the supported set (below) */
#define MOE_ERR_ALIGNMENT         -3  /* a pointer is not 16-byte (w13, w2: 32; ws: 256) aligned */
#define MOE_ERR_WORKSPACE         -4  /* ws_bytes < moe_workspace_bytes() */
#define MOE_ERR_CUDA              -5  /* a CUDA runtime call or launch failed */
#define MOE_ERR_TIMEOUT           -6  /* device: a bounded wait ran out */
#define MOE_ERR_BAD_IDS           -7  /* device: an expert id outside [0, E) */
#define MOE_ERR_BAD_SCALE         -8  /* device: an e8m0 scale byte of 255 (NaN) */
#define MOE_ERR_NO_DEVICE         -9  /* current device is not sm_103 (GB300) */

/* moe_shape.flags */
#define MOE_POST_NORM    1u  /* per-pick RMSNorm of y before the weighted sum */
#define MOE_LOGIT_OFFSET 2u  /* add logit_off[e] to the router logits */

/*
 * Problem shape.  Supported: S >= 1, S * k <= 1<<20; d % 128 == 0 and
 * 128 <= d <= 16384; I % 128 == 0 and 128 <= I <= 8192; 1 <= k <= 16;
 * k <= E <= 512; norm_eps >= 0 (used with MOE_POST_NORM only).
 */
typedef struct moe_shape {
    int32_t S;        /* token rows */
    int32_t d;        /* hidden size (K of gate_up, N-rows of down) */
    int32_t E;        /* experts */
    int32_t k;        /* picks per token */
    int32_t I;        /* expert intermediate size */
    uint32_t flags;   /* MOE_POST_NORM | MOE_LOGIT_OFFSET */
    float norm_eps;   /* RMSNorm epsilon */
} moe_shape;

/* ABI version of the loaded library (MOE_ABI_VERSION). */
int moe_abi_version(void);

/* Static English text for a status code; never NULL. */
const char* moe_strerror(int code);

/*
 * Workspace size for `shape` in *bytes.  Returns MOE_OK, MOE_ERR_INVALID_ARG
 * or MOE_ERR_UNSUPPORTED_SHAPE.  Pure host function.
 */
int moe_workspace_bytes(const moe_shape* shape, size_t* bytes);

/*
 * Clears the workspace's status block and its per-expert sort counters (the
 * first 6400 bytes, or ws_bytes if fewer; enqueued on `stream`).  Call once
 * after allocating a workspace, before its first use; the library's kernels
 * leave the counters cleared after every call that completes.
 */
int moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/*
 * Router + sigmoid top-k (k3 stages A and route; k5 HA).
 *   x         [S, d]  bf16, row-major
 *   w_gate    [E, d]  bf16, row-major (the router weight)
 *   bias      [E]     fp32, selection bias (affects the choice, not w_j)
 *   logit_off [E]     fp32, added to the logits when MOE_LOGIT_OFFSET is
 *                     set, else ignored (may be NULL)
 *   ids       [S, k]  int32 out: picks in ascending expert id
 *   weights   [S, k]  fp32 out: renormalised sigmoid of the picks, aligned
 *                     with ids
 */
int moe_route(const moe_shape* shape, const void* x, const void* w_gate,
              const float* bias, const float* logit_off,
              int32_t* ids, float* weights,
              void* ws, size_t ws_bytes, void* stream);

/*
 * Experts + combine (k3 stages C, D, E; k2_launch w13/w13s/w2/w2s/out).
 *   x         [S, d]        bf16
 *   ids       [S, k]        int32, expert of each pick, distinct within a
 *                           token, any order (an id outside [0, E), or one
 *                           repeated within its token, latches
 *                           MOE_ERR_BAD_IDS and that pick contributes
 *                           nothing)
 *   weights   [S, k]        fp32, aligned with ids
 *   w13       [E, 2I, d/2]  packed e2m1; rows 0..I-1 gate, I..2I-1 up
 *   w13s      [E, 2I, d/32] e8m0
 *   w2        [E, d, I/2]   packed e2m1
 *   w2s       [E, d, I/32]  e8m0
 *   norm_w    [d]           fp32 post-expert norm weight (MOE_POST_NORM),
 *                           else ignored (may be NULL)
 *   out       [S, d]        fp32, overwritten
 */
int moe_experts(const moe_shape* shape, const void* x,
                const int32_t* ids, const float* weights,
                const uint8_t* w13, const uint8_t* w13s,
                const uint8_t* w2, const uint8_t* w2s,
                const float* norm_w, float* out,
                void* ws, size_t ws_bytes, void* stream);

/*
 * The whole block: moe_route then moe_experts on one stream, with the same
 * arguments as those two (ids and weights are written, then consumed).
 */
int moe_forward(const moe_shape* shape, const void* x, const void* w_gate,
                const float* bias, const float* logit_off,
                const uint8_t* w13, const uint8_t* w13s,
                const uint8_t* w2, const uint8_t* w2s,
                const float* norm_w,
                int32_t* ids, float* weights, float* out,
                void* ws, size_t ws_bytes, void* stream);

/*
 * moe_forward with the step's input and outputs in HOST memory: x_host [S, d]
 * bf16 in, ids_host [S, k], weights_host [S, k], out_host [S, d] out, all
 * enqueued on `stream`.  An output in a small pinned buffer the GPU can
 * address (cudaHostAlloc'd or cudaHostRegister'ed memory; on GB300 over the
 * coherent CPU-GPU link), 16-byte aligned, is written in place by the kernels:
 * ids and weights when S <= 32 and S * k <= 128, out when S * d * 4 <= 256 KiB.
 * x is copied into the workspace, from a pinned buffer up to 1 MiB by a kernel
 * (which lets the router start meanwhile), else with one cudaMemcpyAsync; every
 * other host buffer (pageable, unaligned or larger) is staged through the
 * workspace with one cudaMemcpyAsync.  The weights (w_gate,
 * bias, logit_off, w13, w13s, w2, w2s, norm_w) stay device pointers.  The host
 * buffers must not be touched until the stream has been synchronised.
 * ids_host / weights_host may be NULL (then only out is returned).
 */
int moe_forward_host(const moe_shape* shape, const void* x_host, const void* w_gate,
                     const float* bias, const float* logit_off,
                     const uint8_t* w13, const uint8_t* w13s,
                     const uint8_t* w2, const uint8_t* w2s,
                     const float* norm_w,
                     int32_t* ids_host, float* weights_host, float* out_host,
                     void* ws, size_t ws_bytes, void* stream);

/*
 * moe_forward without a workspace argument, for callers that cannot allocate
 * device memory where they run the block (an operator or plugin interface
 * that passes only inputs and outputs, an application whose memory pool owns
 * the whole GPU, a serving loop that must not call cudaMalloc).  The pages have
 * no counterpart: their launchers always receive a scratch buffer.
 *
 * Scratch comes from a 32 MiB static device array inside the library, which
 * every GPU that uses this entry point holds until the process exits.  The
 * library's device modules load lazily (CUDA's default), so the 32 MiB are
 * reserved by the first call on a device, which loads the array's module and
 * looks up its device address once (cudaGetSymbolAddress, with that device
 * current).  Make that first call as a warm-up: before a memory pool claims
 * the whole GPU (else it fails with MOE_ERR_CUDA, reported on stderr) and
 * before any stream capture.  No call allocates or frees memory itself.
 * Shapes whose moe_workspace_bytes() exceeds 32 MiB are rejected with
 * MOE_ERR_WORKSPACE (S * k <= 256 at d = 4096, I = 1024, E = 256 fits), and
 * every argument check of moe_forward runs, with the same codes, before the
 * array is touched: a rejected call enqueues nothing.
 *
 * Every call on a device shares the one array, which keeps the previous
 * call's contents; each call clears its status block first.  Calls that
 * overlap on the GPU (other streams, other host threads) race on the array:
 * order them on one stream.  Arguments are those of moe_forward minus the
 * workspace; `status` (device int32[2], may be NULL) receives this call's
 * device status and detail (see moe_device_status) when the call's work is
 * done.
 */
int moe_forward_noalloc(const moe_shape* shape, const void* x, const void* w_gate,
                        const float* bias, const float* logit_off,
                        const uint8_t* w13, const uint8_t* w13s,
                        const uint8_t* w2, const uint8_t* w2s,
                        const float* norm_w,
                        int32_t* ids, float* weights, float* out,
                        int32_t* status, void* stream);

/*
 * The latent-MoE layer around the routed block, with a shared expert
 * (vllm.models.kimi_k3.amd.specialized_decode.mono.layer: K2b's stage list --
 * router parts and latent parts, route, the shared gate/up and its
 * activation, ug and down of the routed experts, the shared down, lnorm, up --
 * and k2_launch's arguments w_gate, bias, w_ld, w_sgu, w_sd, w13, w13s, w2,
 * w2s, ln_w, w_up, out [S, 7168]).  For token t:
 *   picks, w_j = the sigmoid top-k of x[t] (as moe_route, over H)
 *   xl        = x[t] . w_ld^T                   latent input, [LAT] (bf16)
 *   yl        = sum_j w_j * expert_j(xl)        the routed block at d = LAT
 *   zl        = yl * rsqrt(mean(yl^2) + norm_eps) * ln_w             (bf16)
 *   out[t]    = zl . w_up^T  +  (silu(g) * u) . w_sd^T,
 *               g, u = x[t] . w_sgu[0:SI]^T, x[t] . w_sgu[SI:2SI]^T  (fp32)
 * The pages give the stages and the argument names, not the formulas or the
 * formats: the dense weights carry no scale tensors and are bf16 here; the
 * latent norm is an RMSNorm with weight ln_w; the shared expert is a SwiGLU
 * expert on the layer input, its output added to the up projection's.  The
 * intermediate activations xl, zl and silu(g) * u are rounded to bf16, the
 * operand type of the dense products (bf16 x bf16 on the tensor cores, fp32
 * accumulation); every sum is fp32.
 *
 * Shape: H and LAT multiples of 128 (LAT <= 16384, H <= 16384), SI a
 * multiple of 128 or 0 (no shared expert), E, k, I as in moe_shape, S * k
 * <= 1<<20; flags may hold MOE_LOGIT_OFFSET only.
 */
typedef struct moe_latent_shape {
    int32_t S;        /* token rows */
    int32_t H;        /* hidden size of the layer input and output */
    int32_t LAT;      /* latent width: the routed experts' d */
    int32_t E;        /* routed experts */
    int32_t k;        /* picks per token */
    int32_t I;        /* routed expert intermediate size */
    int32_t SI;       /* shared expert intermediate size (0: none) */
    uint32_t flags;   /* MOE_LOGIT_OFFSET */
    float norm_eps;   /* latent RMSNorm epsilon */
} moe_latent_shape;

/* Workspace size of moe_latent_forward in *bytes (pure host function). */
int moe_latent_workspace_bytes(const moe_latent_shape* shape, size_t* bytes);

/*
 * The latent-MoE layer, all device pointers (16-byte aligned; w13, w2:
 * 32-byte aligned), enqueued on `stream`:
 *   x      [S, H] bf16           w_gate [E, H] bf16     bias [E] fp32
 *   logit_off [E] fp32 (MOE_LOGIT_OFFSET) or NULL
 *   w_ld   [LAT, H] bf16         latent down projection
 *   w13 [E, 2I, LAT/2], w13s [E, 2I, LAT/32], w2 [E, LAT, I/2], w2s
 *   [E, LAT, I/32]               the routed experts (MXFP4, as moe_experts)
 *   ln_w   [LAT] fp32            latent norm weight
 *   w_up   [H, LAT] bf16         up projection
 *   w_sgu  [2 SI, H] bf16        shared gate (rows 0..SI-1) and up rows
 *   w_sd   [H, SI] bf16          shared down (both NULL when SI == 0)
 *   ids, weights [S, k] out      the routing, as moe_route
 *   out    [S, H] fp32 out       overwritten
 * ws: at least moe_latent_workspace_bytes(), 256-byte aligned, prepared with
 * moe_workspace_init.  Errors as for moe_forward.
 */
int moe_latent_forward(const moe_latent_shape* shape, const void* x, const void* w_gate,
                       const float* bias, const float* logit_off, const void* w_ld,
                       const uint8_t* w13, const uint8_t* w13s,
                       const uint8_t* w2, const uint8_t* w2s,
                       const float* ln_w, const void* w_up,
                       const void* w_sgu, const void* w_sd,
                       int32_t* ids, float* weights, float* out,
                       void* ws, size_t ws_bytes, void* stream);

/*
 * Synchronises `stream`, returns the status latched in the workspace by the
 * device since the last call (MOE_OK, MOE_ERR_BAD_IDS, MOE_ERR_BAD_SCALE or
 * MOE_ERR_TIMEOUT; MOE_ERR_CUDA if the synchronisation itself failed) and
 * clears it.  *detail (may be NULL) receives a code-specific value: the first
 * offending flat pick index, the first bad scale byte's value, or the site of
 * the wait that ran out.
 */
int moe_device_status(void* ws, int32_t* detail, void* stream);

/*
 * Workspace regions (diagnostics, pure host function): byte offset and size
 * of one region of the workspace of `shape`, for reading intermediate results
 * back after a call (tests and profiling).  Returns MOE_OK, or
 * MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED_SHAPE.  P = S * k picks; a pick's
 * sorted position r groups the picks by ascending expert id (k3 page,
 * dn_loads: tasks over a table of the experts that have picks).
 *   MOE_WS_STATUS  int32 [64]: status, detail, valid picks, work tiles, ...
 *   MOE_WS_POS     int32 [P]: sorted position r of pick t*k + j (-1: invalid)
 *   MOE_WS_TILES   int32 [max tiles][4]: expert, first position, picks, 0;
 *                  the first "work tiles" entries are this call's tiles
 *   MOE_WS_XQ      uint8 [2P][d]: e4m3 rows 2r (hi) and 2r + 1 (lo) of the
 *                  token of the pick at position r
 *   MOE_WS_XS      uint8 [ceil(d/256)][P + 64][16]: e8m0 scale of 32-element
 *                  block b of position r at [b / 8][r][b % 8]
 *   MOE_WS_HQ, MOE_WS_HS  the same for h = silu(g) * u (K = I)
 *   MOE_WS_Y       fp32 [P][d]: expert output of the pick at position r
 *   MOE_WS_LOGITS  fp32 [S][E]: the router's logits (moe_route, moe_forward)
 */
#define MOE_WS_STATUS 0
#define MOE_WS_POS    1
#define MOE_WS_TILES  2
#define MOE_WS_XQ     3
#define MOE_WS_XS     4
#define MOE_WS_HQ     5
#define MOE_WS_HS     6
#define MOE_WS_Y      7
#define MOE_WS_LOGITS 8
int moe_workspace_region(const moe_shape* shape, int region, size_t* offset, size_t* bytes);

/*
 * Per-kernel timing (diagnostics, host side).  After moe_timing_enable(n) with
 * n > 0, the next n kernels the library launches are each bracketed by a pair
 * of CUDA events recorded on their launch stream; n = 0 turns this off and
 * frees the events.  moe_timing_collect waits for the recorded events and
 * writes up to `cap` (kernel id, milliseconds) pairs in launch order, the
 * count to *n, and starts a new recording of the same size.  Kernel ids name
 * the launched kernels (moe_kernel_name; NULL past the last id).  Not
 * thread-safe; event records add a few microseconds of host time per launch.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG or MOE_ERR_CUDA.
 */
int moe_timing_enable(int max_launches);
int moe_timing_collect(int32_t* kernel_ids, float* ms, int cap, int* n);
const char* moe_kernel_name(int kernel_id);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
