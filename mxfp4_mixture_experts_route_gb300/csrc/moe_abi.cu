// The C ABI of libmoe: argument checks, workspace layout and the launch order
// of the block (router -> top-k -> expert sort/gather -> gate_up -> down ->
// combine) on the caller's stream.  Declarations and contracts: include/moe.h.
#include "moe_internal.cuh"

#include <stdio.h>

namespace moe {

// x from pinned host memory into the workspace by a kernel (hostio.cu):
// bytes a multiple of 16, both addresses 16-byte aligned
cudaError_t launch_stage_in(const void* src, void* dst, size_t bytes, cudaStream_t st);
// the combine that also copies ids and weights to host buffers (combine.cu)
cudaError_t launch_combine_host(const moe_shape& s, const WsLayout& L, const Ptrs& p, int32_t* ids_out, float* w_out,
                                cudaStream_t st);

static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Picks per expert tile: 8 while the average expert gets at most 2 picks (the
// tile then carries little padding, and the expert kernel's smaller token
// stages leave room for one more weight stage); 32 once it gets 32 or more
// (fewer, wider MMAs per weight byte where the expert GEMMs turn compute
// bound); else 16 (with more picks per expert a second tile, which reads the
// expert's weights again, gets likely).
int tile_picks(const moe_shape& s) {
    const int64_t picks = (int64_t)s.S * s.k;
    if (picks <= 2 * (int64_t)s.E) return 8;
    if (picks >= 64 * (int64_t)s.E) return 64;
    return picks >= 32 * (int64_t)s.E ? 32 : 16;
}

WsLayout ws_layout(const moe_shape& s) {
    WsLayout L{};
    const size_t P = (size_t)s.S * s.k;                  // picks
    L.max_picks = (int)P;
    L.nt = tile_picks(s);
    const size_t nt = (size_t)L.nt;
    // sum_e ceil(n_e / nt) <= P / nt + (experts with a pick) <= ceil(P / nt) + min(E, P)
    L.max_tiles = (int)((P + nt - 1) / nt + (P < (size_t)s.E ? P : (size_t)s.E));
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align256(o + bytes); return at; };
    L.status = take(sizeof(StatusBlock));
    L.sortcnt = take(SORT_CNT_BYTES);   // right after the status block: the zeroed prefix
    // router K-split (its cluster size): chosen for 152 SMs (GB300); another
    // SM count only changes how the work is split
    L.router_kslices = router_kslices(s, 152);
    L.logits = take((size_t)s.S * s.E * 4);
    L.pos = take(P * 4);
    L.tiles = take((size_t)L.max_tiles * sizeof(Tile));
    L.tile_ready = take((size_t)L.max_tiles * 4);
    // e4m3 hi / lo rows of the gathered tokens and of h, and their block scales
    const size_t rows = P + NT_MAX;
    L.xq = take(2 * P * s.d);
    L.xs = take((size_t)((s.d + 255) / 256) * rows * TOKEN_SCALE_ROW);
    L.hq = take(2 * P * s.I);
    L.hs = take((size_t)((s.I + 255) / 256) * rows * TOKEN_SCALE_ROW);
    L.y = take(P * s.d * 4);
    L.ssq = take(P * (s.d / 128) * 4);                   // per-pick sums of y^2 by 128-row block
    L.xin = take((size_t)s.S * s.d * 2);                 // host-I/O staging
    L.hio_ids = take(P * 4);
    L.hio_w = take(P * 4);
    L.hio_out = take((size_t)s.S * s.d * 4);
    L.total = o;
    return L;
}

static int check_shape(const moe_shape* s) {
    if (!s) return MOE_ERR_INVALID_ARG;
    if (s->flags & ~(MOE_POST_NORM | MOE_LOGIT_OFFSET)) return MOE_ERR_INVALID_ARG;
    if (s->S < 1 || s->d < 1 || s->E < 1 || s->k < 1 || s->I < 1) return MOE_ERR_INVALID_ARG;
    if (!(s->norm_eps >= 0.0f)) return MOE_ERR_INVALID_ARG;
    if (s->d % 128 || s->d > 16384) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (s->I % 128 || s->I > 8192) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (s->k > 16 || s->k > s->E || s->E > 512) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((int64_t)s->S * s->k > (1 << 20)) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

static bool a16(const void* p) { return ((uintptr_t)p & 15) == 0; }
static bool a32(const void* p) { return ((uintptr_t)p & 31) == 0; }   // the 4-bit tensor maps' base rule

static int check_ws(const moe_shape* s, void* ws, size_t ws_bytes) {
    if (!ws) return MOE_ERR_INVALID_ARG;
    if ((uintptr_t)ws & 255) return MOE_ERR_ALIGNMENT;
    if (ws_bytes < ws_layout(*s).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

static int check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return MOE_ERR_NO_DEVICE; }
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_NO_DEVICE;
    }
    return (major == 10 && minor == 3) ? MOE_OK : MOE_ERR_NO_DEVICE;
}

static int cuda_rc(cudaError_t e) {
    if (e == cudaSuccess) return MOE_OK;
    fprintf(stderr, "libmoe: CUDA error %d (%s)\n", (int)e, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
}

static int check_route_args(const moe_shape* s, const void* x, const void* w_gate, const float* bias,
                            const float* logit_off, const int32_t* ids, const float* w) {
    if (!x || !w_gate || !bias || !ids || !w) return MOE_ERR_INVALID_ARG;
    if ((s->flags & MOE_LOGIT_OFFSET) && !logit_off) return MOE_ERR_INVALID_ARG;
    if (!a16(x) || !a16(w_gate) || !a16(bias) || !a16(ids) || !a16(w)) return MOE_ERR_ALIGNMENT;
    if ((s->flags & MOE_LOGIT_OFFSET) && !a16(logit_off)) return MOE_ERR_ALIGNMENT;
    return MOE_OK;
}

static int check_expert_args(const moe_shape* s, const void* x, const int32_t* ids, const float* w,
                             const uint8_t* w13, const uint8_t* w13s, const uint8_t* w2,
                             const uint8_t* w2s, const float* norm_w, const float* out) {
    if (!x || !ids || !w || !w13 || !w13s || !w2 || !w2s || !out) return MOE_ERR_INVALID_ARG;
    if ((s->flags & MOE_POST_NORM) && !norm_w) return MOE_ERR_INVALID_ARG;
    if (!a16(x) || !a16(ids) || !a16(w) || !a32(w13) || !a16(w13s) || !a32(w2) || !a16(w2s) || !a16(out))
        return MOE_ERR_ALIGNMENT;
    if ((s->flags & MOE_POST_NORM) && !a16(norm_w)) return MOE_ERR_ALIGNMENT;
    return MOE_OK;
}

static int run_route(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st) {
    return cuda_rc(launch_route(s, L, p, st));
}

// first: the sort + gather is the call's first kernel (moe_experts), so it
// reads x only after its wait, whatever the caller's previous kernel does;
// after the top-k kernel (moe_forward) x is final before it may start
static int run_experts(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st, bool first) {
    int rc = cuda_rc(launch_sort_gather(s, L, p, st, first));
    if (rc) return rc;
    rc = cuda_rc(launch_experts(s, L, p, st));
    if (rc) return rc;
    return cuda_rc(launch_combine(s, L, p, st));
}

// Every host-side check of moe_forward (shape, pointers, alignment, device),
// without the workspace: moe_forward_noalloc runs them before it touches its
// scratch array, so a rejected call enqueues nothing.
int check_forward_args(const moe_shape* s, const void* x, const void* w_gate, const float* bias,
                       const float* logit_off, const uint8_t* w13, const uint8_t* w13s, const uint8_t* w2,
                       const uint8_t* w2s, const float* norm_w, const int32_t* ids, const float* w,
                       const float* out) {
    int rc = check_shape(s);
    if (!rc) rc = check_route_args(s, x, w_gate, bias, logit_off, ids, w);
    if (!rc) rc = check_expert_args(s, x, ids, w, w13, w13s, w2, w2s, norm_w, out);
    if (!rc) rc = check_device();
    return rc;
}

// The whole block.  At small S the top-k, the sort and the gather share one
// kernel (two launches and two kernel boundaries fewer).
// ids_out / w_out (moe_forward_host at small S, or null): host buffers the
// combine copies the ids and weights to.
static int run_forward(const moe_shape& s, const WsLayout& L, const Ptrs& p, cudaStream_t st,
                       int32_t* ids_out = nullptr, float* w_out = nullptr) {
    if (!topk_sort_fits(s)) {
        const int rc = run_route(s, L, p, st);
        return rc ? rc : run_experts(s, L, p, st, false);
    }
    int rc = cuda_rc(launch_router_logits(s, L, p, st));
    if (!rc) rc = cuda_rc(launch_topk_sort_gather(s, L, p, st));
    if (!rc) rc = cuda_rc(launch_experts(s, L, p, st));
    if (!rc) rc = cuda_rc(launch_combine_host(s, L, p, ids_out, w_out, st));
    return rc;
}

// moe_forward; ids_out / w_out (host buffers, or null): the combine also
// copies the ids and weights there (moe_forward_host at small S)
static int forward_impl(const moe_shape* shape, const void* x, const void* w_gate, const float* bias,
                        const float* logit_off, const uint8_t* w13, const uint8_t* w13s, const uint8_t* w2,
                        const uint8_t* w2s, const float* norm_w, int32_t* ids, float* weights, float* out,
                        void* ws, size_t ws_bytes, void* stream, int32_t* ids_out, float* w_out) {
    int rc = check_shape(shape);
    if (!rc) rc = check_route_args(shape, x, w_gate, bias, logit_off, ids, weights);
    if (!rc) rc = check_expert_args(shape, x, ids, weights, w13, w13s, w2, w2s, norm_w, out);
    if (!rc) rc = check_ws(shape, ws, ws_bytes);
    if (!rc) rc = check_device();
    if (rc) return rc;
    WsLayout L = ws_layout(*shape);
    Ptrs p{};
    p.x = (const __nv_bfloat16*)x;
    p.w_gate = (const __nv_bfloat16*)w_gate;
    p.bias = bias;
    p.logit_off = (shape->flags & MOE_LOGIT_OFFSET) ? logit_off : nullptr;
    p.w13 = w13; p.w13s = w13s; p.w2 = w2; p.w2s = w2s;
    p.norm_w = (shape->flags & MOE_POST_NORM) ? norm_w : nullptr;
    p.ids = ids;
    p.weights = weights;
    p.out = out;
    p.ws = (char*)ws;
    return run_forward(*shape, L, p, (cudaStream_t)stream, ids_out, w_out);
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_strerror(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MOE_ERR_ALIGNMENT: return "misaligned pointer";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "device wait timed out";
        case MOE_ERR_BAD_IDS: return "expert id out of range or repeated within a token";
        case MOE_ERR_BAD_SCALE: return "e8m0 scale byte 255 (NaN)";
        case MOE_ERR_NO_DEVICE: return "no sm_103 device";
        default: return "unknown status";
    }
}

int moe_workspace_bytes(const moe_shape* shape, size_t* bytes) {
    int rc = check_shape(shape);
    if (rc) return rc;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = ws_layout(*shape).total;
    return MOE_OK;
}

int moe_workspace_region(const moe_shape* shape, int region, size_t* offset, size_t* bytes) {
    int rc = check_shape(shape);
    if (rc) return rc;
    if (!offset || !bytes) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*shape);
    const size_t P = (size_t)shape->S * shape->k, rows = P + NT_MAX;
    switch (region) {
        case MOE_WS_STATUS: *offset = L.status; *bytes = sizeof(StatusBlock); break;
        case MOE_WS_POS: *offset = L.pos; *bytes = P * 4; break;
        case MOE_WS_TILES: *offset = L.tiles; *bytes = (size_t)L.max_tiles * sizeof(Tile); break;
        case MOE_WS_XQ: *offset = L.xq; *bytes = 2 * P * shape->d; break;
        case MOE_WS_XS: *offset = L.xs; *bytes = (size_t)((shape->d + 255) / 256) * rows * TOKEN_SCALE_ROW; break;
        case MOE_WS_HQ: *offset = L.hq; *bytes = 2 * P * shape->I; break;
        case MOE_WS_HS: *offset = L.hs; *bytes = (size_t)((shape->I + 255) / 256) * rows * TOKEN_SCALE_ROW; break;
        case MOE_WS_Y: *offset = L.y; *bytes = P * shape->d * 4; break;
        case MOE_WS_LOGITS: *offset = L.logits; *bytes = (size_t)shape->S * shape->E * 4; break;
        default: return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

int moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (!ws) return MOE_ERR_INVALID_ARG;
    if ((uintptr_t)ws & 255) return MOE_ERR_ALIGNMENT;
    if (ws_bytes < sizeof(StatusBlock)) return MOE_ERR_WORKSPACE;
    int rc = check_device();
    if (rc) return rc;
    const size_t n = ws_bytes < WS_ZERO_PREFIX ? ws_bytes : WS_ZERO_PREFIX;
    return cuda_rc(cudaMemsetAsync(ws, 0, n, (cudaStream_t)stream));
}

int moe_route(const moe_shape* shape, const void* x, const void* w_gate, const float* bias,
              const float* logit_off, int32_t* ids, float* weights, void* ws, size_t ws_bytes,
              void* stream) {
    int rc = check_shape(shape);
    if (!rc) rc = check_route_args(shape, x, w_gate, bias, logit_off, ids, weights);
    if (!rc) rc = check_ws(shape, ws, ws_bytes);
    if (!rc) rc = check_device();
    if (rc) return rc;
    WsLayout L = ws_layout(*shape);
    Ptrs p{};
    p.x = (const __nv_bfloat16*)x;
    p.w_gate = (const __nv_bfloat16*)w_gate;
    p.bias = bias;
    p.logit_off = (shape->flags & MOE_LOGIT_OFFSET) ? logit_off : nullptr;
    p.ids = ids;
    p.weights = weights;
    p.ws = (char*)ws;
    return run_route(*shape, L, p, (cudaStream_t)stream);
}

int moe_experts(const moe_shape* shape, const void* x, const int32_t* ids, const float* weights,
                const uint8_t* w13, const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s,
                const float* norm_w, float* out, void* ws, size_t ws_bytes, void* stream) {
    int rc = check_shape(shape);
    if (!rc) rc = check_expert_args(shape, x, ids, weights, w13, w13s, w2, w2s, norm_w, out);
    if (!rc) rc = check_ws(shape, ws, ws_bytes);
    if (!rc) rc = check_device();
    if (rc) return rc;
    WsLayout L = ws_layout(*shape);
    Ptrs p{};
    p.x = (const __nv_bfloat16*)x;
    p.ids = const_cast<int32_t*>(ids);
    p.weights = const_cast<float*>(weights);
    p.w13 = w13; p.w13s = w13s; p.w2 = w2; p.w2s = w2s;
    p.norm_w = (shape->flags & MOE_POST_NORM) ? norm_w : nullptr;
    p.out = out;
    p.ws = (char*)ws;
    return run_experts(*shape, L, p, (cudaStream_t)stream, true);
}

int moe_forward(const moe_shape* shape, const void* x, const void* w_gate, const float* bias,
                const float* logit_off, const uint8_t* w13, const uint8_t* w13s, const uint8_t* w2,
                const uint8_t* w2s, const float* norm_w, int32_t* ids, float* weights, float* out,
                void* ws, size_t ws_bytes, void* stream) {
    return forward_impl(shape, x, w_gate, bias, logit_off, w13, w13s, w2, w2s, norm_w, ids, weights, out, ws, ws_bytes,
                        stream, nullptr, nullptr);
}

}  // extern "C"

namespace {
// The latent layer's workspace: the block's workspace for the larger of its
// two shapes (the router over H, the experts over LAT; the two calls run one
// after the other on the stream, so they share it), then the layer's own
// activations.
struct LatentLayout {
    moe_shape sr, sx;      // routing over H; experts over LAT
    WsLayout Lr, Lx;
    size_t xl, yl, zl, gu, hs, total;
};

int latent_layout(const moe_latent_shape* ls, LatentLayout& o) {
    if (!ls) return MOE_ERR_INVALID_ARG;
    if (ls->flags & ~MOE_LOGIT_OFFSET) return MOE_ERR_INVALID_ARG;
    if (ls->SI < 0 || ls->H < 1 || ls->LAT < 1) return MOE_ERR_INVALID_ARG;
    if (ls->SI % 128 || ls->SI > 16384) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!latent_mid_fits(ls->LAT)) return MOE_ERR_UNSUPPORTED_SHAPE;
    o.sr = moe_shape{ls->S, ls->H, ls->E, ls->k, ls->I, ls->flags, ls->norm_eps};
    o.sx = moe_shape{ls->S, ls->LAT, ls->E, ls->k, ls->I, 0u, ls->norm_eps};
    int rc = check_shape(&o.sr);
    if (!rc) rc = check_shape(&o.sx);
    if (rc) return rc;
    o.Lr = ws_layout(o.sr);
    o.Lx = ws_layout(o.sx);
    size_t at = align256(o.Lr.total > o.Lx.total ? o.Lr.total : o.Lx.total);
    auto take = [&](size_t bytes) { size_t r = at; at = align256(at + bytes); return r; };
    const size_t S = (size_t)ls->S;
    o.xl = take(S * ls->LAT * 2);
    o.yl = take(S * ls->LAT * 4);
    o.zl = take(S * ls->LAT * 2);
    o.gu = take(S * 2 * (size_t)ls->SI * 4);
    o.hs = take(S * (size_t)ls->SI * 2);
    o.total = at;
    return MOE_OK;
}

// The device address of a 16-byte aligned pinned host buffer the GPU reads and
// writes in place (cudaHostAlloc'd or registered memory under unified
// addressing; on GB300 over the coherent CPU-GPU link), else nullptr: pageable
// or unaligned memory is staged.
void* device_view(const void* host) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, host) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return nullptr;
    return ((uintptr_t)at.devicePointer & 15) == 0 ? at.devicePointer : nullptr;
}
}  // namespace

extern "C" {

int moe_forward_host(const moe_shape* shape, const void* x_host, const void* w_gate, const float* bias,
                     const float* logit_off, const uint8_t* w13, const uint8_t* w13s, const uint8_t* w2,
                     const uint8_t* w2s, const float* norm_w, int32_t* ids_host, float* weights_host,
                     float* out_host, void* ws, size_t ws_bytes, void* stream) {
    int rc = check_shape(shape);
    if (rc) return rc;
    if (!x_host || !out_host) return MOE_ERR_INVALID_ARG;
    if (!w_gate || !bias || !w13 || !w13s || !w2 || !w2s) return MOE_ERR_INVALID_ARG;
    if ((shape->flags & MOE_LOGIT_OFFSET) && !logit_off) return MOE_ERR_INVALID_ARG;
    if ((shape->flags & MOE_POST_NORM) && !norm_w) return MOE_ERR_INVALID_ARG;
    if (!a16(w_gate) || !a16(bias) || !a32(w13) || !a16(w13s) || !a32(w2) || !a16(w2s))
        return MOE_ERR_ALIGNMENT;
    rc = check_ws(shape, ws, ws_bytes);
    if (!rc) rc = check_device();
    if (rc) return rc;
    // A small pinned host buffer for an output is written over the link by a
    // kernel (measured faster than a copy afterwards at S = 8: 7 to 8 us a step
    // for each of out and ids + weights): out up to 256 KB by the combine, and
    // ids and weights, when the fused top-k + sort + gather produces them,
    // copied from the workspace by the combine too (so that those writes do
    // not hold up the routing kernel's completion).  x, which the router and
    // the gather both read, and every other buffer go through the workspace's
    // host-I/O staging regions (xin, hio_ids, hio_w, hio_out).
    WsLayout L = ws_layout(*shape);
    cudaStream_t st = (cudaStream_t)stream;
    char* w = (char*)ws;
    const size_t P = (size_t)shape->S * shape->k;
    const bool small_out = (size_t)shape->S * shape->d * 4 <= (256u << 10);
    // ids and weights go to the workspace; the combine copies them to pinned
    // host buffers at small S, a copy afterwards does otherwise
    int32_t* ids_view = ids_host && route_gather_selects(*shape) ? (int32_t*)device_view(ids_host) : nullptr;
    float* wts_view = weights_host && route_gather_selects(*shape) ? (float*)device_view(weights_host) : nullptr;
    float* out_dev = small_out ? (float*)device_view(out_host) : nullptr;
    const bool ids_staged = !ids_view, wts_staged = !wts_view, out_staged = !out_dev;
    int32_t* ids_dev = (int32_t*)(w + L.hio_ids);
    float* wts_dev = (float*)(w + L.hio_w);
    if (!out_dev) out_dev = (float*)(w + L.hio_out);
    // x by a kernel from a pinned buffer up to 1 MB (the router starts while
    // it runs), by the copy engine otherwise
    void* x_dev = w + L.xin;
    const size_t x_bytes = (size_t)shape->S * shape->d * 2;
    const void* x_view = x_bytes <= (1u << 20) ? device_view(x_host) : nullptr;
    rc = cuda_rc(x_view ? launch_stage_in(x_view, x_dev, x_bytes, st)
                        : cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, st));
    if (rc) return rc;
    rc = forward_impl(shape, x_dev, w_gate, bias, logit_off, w13, w13s, w2, w2s, norm_w, ids_dev, wts_dev, out_dev,
                      ws, ws_bytes, stream, ids_view, wts_view);
    if (rc) return rc;
    if (out_staged)
        rc = cuda_rc(cudaMemcpyAsync(out_host, out_dev, (size_t)shape->S * shape->d * 4, cudaMemcpyDeviceToHost, st));
    if (!rc && ids_host && ids_staged)
        rc = cuda_rc(cudaMemcpyAsync(ids_host, ids_dev, P * 4, cudaMemcpyDeviceToHost, st));
    if (!rc && weights_host && wts_staged)
        rc = cuda_rc(cudaMemcpyAsync(weights_host, wts_dev, P * 4, cudaMemcpyDeviceToHost, st));
    return rc;
}

int moe_latent_workspace_bytes(const moe_latent_shape* shape, size_t* bytes) {
    LatentLayout LL;
    const int rc = latent_layout(shape, LL);
    if (rc) return rc;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = LL.total;
    return MOE_OK;
}

int moe_latent_forward(const moe_latent_shape* shape, const void* x, const void* w_gate, const float* bias,
                       const float* logit_off, const void* w_ld, const uint8_t* w13, const uint8_t* w13s,
                       const uint8_t* w2, const uint8_t* w2s, const float* ln_w, const void* w_up, const void* w_sgu,
                       const void* w_sd, int32_t* ids, float* weights, float* out, void* ws, size_t ws_bytes,
                       void* stream) {
    LatentLayout LL;
    int rc = latent_layout(shape, LL);
    if (rc) return rc;
    const moe_latent_shape& ls = *shape;
    const bool shared = ls.SI > 0;
    if (!x || !w_gate || !bias || !w_ld || !w13 || !w13s || !w2 || !w2s || !ln_w || !w_up || !ids || !weights || !out)
        return MOE_ERR_INVALID_ARG;
    if ((ls.flags & MOE_LOGIT_OFFSET) && !logit_off) return MOE_ERR_INVALID_ARG;
    if (shared && (!w_sgu || !w_sd)) return MOE_ERR_INVALID_ARG;
    if (!a16(x) || !a16(w_gate) || !a16(bias) || !a16(w_ld) || !a32(w13) || !a16(w13s) || !a32(w2) || !a16(w2s) ||
        !a16(ln_w) || !a16(w_up) || !a16(ids) || !a16(weights) || !a16(out))
        return MOE_ERR_ALIGNMENT;
    if ((ls.flags & MOE_LOGIT_OFFSET) && !a16(logit_off)) return MOE_ERR_ALIGNMENT;
    if (shared && (!a16(w_sgu) || !a16(w_sd))) return MOE_ERR_ALIGNMENT;
    if (!ws) return MOE_ERR_INVALID_ARG;
    if ((uintptr_t)ws & 255) return MOE_ERR_ALIGNMENT;
    if (ws_bytes < LL.total) return MOE_ERR_WORKSPACE;
    rc = check_device();
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    char* w = (char*)ws;
    StatusBlock* sb = reinterpret_cast<StatusBlock*>(w + LL.Lr.status);
    const int S = ls.S;
    // k2 page, K2b's stages, in six launches at small S:
    //   1. the router's logits L = x . w_gate^T (+ offset), latent down
    //      xl = bf16(x . w_ld^T) and the shared expert's gate/up gu = x . w_sgu^T,
    //      one launch (products of the same x over H, the weights one after
    //      the other along N; the router in its own kernel before it when E is
    //      not a multiple of 128)
    //   2. top-k, sort and gather of xl (the block's workspace over LAT shares
    //      the router's status, logits, pos and tile regions)
    //   3-4. the expert GEMMs and the combine: yl
    //   5. zl = bf16(RMSNorm(yl) ln_w) and hs = bf16(silu(g) u)
    //   6. out = zl . w_up^T + hs . w_sd^T, one launch (the two products
    //      concatenated along K)
    Ptrs pr{};
    pr.x = (const __nv_bfloat16*)x;
    pr.w_gate = (const __nv_bfloat16*)w_gate;
    pr.bias = bias;
    pr.logit_off = (ls.flags & MOE_LOGIT_OFFSET) ? logit_off : nullptr;
    pr.ids = ids;
    pr.weights = weights;
    pr.ws = w;
    // the router's logits join the latent-down launch as its first part when
    // its experts fill whole 128-row tiles; otherwise the router's own kernel
    const bool router_part = ls.E % 128 == 0;
    if (!router_part) rc = cuda_rc(launch_router_logits(LL.sr, LL.Lr, pr, st));
    if (!rc) {
        DensePart parts[3];
        int np = 0;
        if (router_part) parts[np++] = DensePart{w_gate, ls.E, w + LL.Lr.logits, DENSE_F32};
        parts[np++] = DensePart{w_ld, ls.LAT, w + LL.xl, DENSE_BF16};
        if (shared) parts[np++] = DensePart{w_sgu, 2 * ls.SI, w + LL.gu, DENSE_F32};
        timing_begin(K_LATENT_DOWN, st);
        rc = cuda_rc(launch_dense_ncat(x, S, ls.H, parts, np, router_part ? pr.logit_off : nullptr, sb, st,
                                       K_LATENT_DOWN));
        timing_end(st);
    }
    Ptrs px{};
    px.x = (const __nv_bfloat16*)(w + LL.xl);
    px.bias = bias;
    px.ids = ids;
    px.weights = weights;
    px.w13 = w13; px.w13s = w13s; px.w2 = w2; px.w2s = w2s;
    px.norm_w = nullptr;
    px.out = (float*)(w + LL.yl);
    px.ws = w;
    if (!rc) {
        if (topk_sort_fits(LL.sx)) {
            rc = cuda_rc(launch_topk_sort_gather(LL.sx, LL.Lx, px, st, true));
        } else {
            rc = cuda_rc(launch_topk(LL.sx, LL.Lx, px, st));
            if (!rc) rc = cuda_rc(launch_sort_gather(LL.sx, LL.Lx, px, st, true));
        }
    }
    if (!rc) rc = cuda_rc(launch_experts(LL.sx, LL.Lx, px, st));
    if (!rc) rc = cuda_rc(launch_combine(LL.sx, LL.Lx, px, st));
    if (!rc) {
        timing_begin(K_LATENT_MID, st);
        rc = cuda_rc(launch_latent_mid((const float*)(w + LL.yl), ln_w, ls.norm_eps, S, ls.LAT,
                                       (__nv_bfloat16*)(w + LL.zl), (const float*)(w + LL.gu), ls.SI,
                                       (__nv_bfloat16*)(w + LL.hs), st));
        timing_end(st);
    }
    if (!rc) {
        timing_begin(K_LATENT_UP, st);
        rc = shared ? cuda_rc(launch_dense_kcat(w + LL.zl, w_up, ls.LAT, w + LL.hs, w_sd, ls.SI, S, ls.H, out,
                                                DENSE_F32, sb, st, K_LATENT_UP))
                    : cuda_rc(launch_dense(w + LL.zl, w_up, S, ls.LAT, ls.H, nullptr, out, DENSE_F32, sb, st,
                                           K_LATENT_UP));
        timing_end(st);
    }
    return rc;
}

int moe_device_status(void* ws, int32_t* detail, void* stream) {
    if (!ws) return MOE_ERR_INVALID_ARG;
    if ((uintptr_t)ws & 255) return MOE_ERR_ALIGNMENT;
    cudaStream_t st = (cudaStream_t)stream;
    StatusBlock hb{};
    if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_rc(cudaGetLastError());
    if (cudaMemcpy(&hb, ws, 2 * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return cuda_rc(cudaGetLastError());
    if (hb.status != 0) {
        int32_t zero[2] = {0, 0};
        if (cudaMemcpy(ws, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return cuda_rc(cudaGetLastError());
    }
    if (detail) *detail = hb.detail;
    return hb.status;
}

}  // extern "C"
