"""GPU path vs the CPU oracle, through the C ABI (needs a GB300).

Bars: routing ids bit-exact; routing weights checked through the router's
fp32 logits (within the error of an fp32 sum in any order of the oracle's
exact logits, and the weights within 2e-6 of those logits renormalised:
check_routing_weights); outputs max|out - ref| / max|ref| <= 1e-2 (the expert
GEMMs take x exactly, as two e4m3 halves under a block scale, and h to about
9 significant bits; the oracle keeps fp64 throughout).
"""
import numpy as np
import pytest

import moe_inputs as mi
import mxfp4_mixture_experts_route_gb300 as moe
import oracle as O
from libmoe_util import check_routing_weights, device_block, ensure_built, gpu_forward, shape_of
from oracle.gap_tables import enforce_gap

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _check(inp, ids, w, out, L, rows=None):
    rows = np.arange(inp.cfg.S) if rows is None else np.asarray(rows)
    rids, rw, rout, _ = O.moe_forward(inp, rows)
    assert np.array_equal(ids[rows], rids), "routing ids differ"
    check_routing_weights(L, inp.x, inp.w_gate, inp.logit_off, ids, w, rows)
    err = O.parity_error(out[rows], rout)
    assert err <= OUT_TOL, f"out parity {err:.3e}"
    return err


def _gap_inputs(cfg, seed):
    return mi.make_inputs(cfg, seed, attempts=enforce_gap(cfg, seed), use_stored_attempts=False)


@pytest.mark.parametrize("ci", [0, 1, 2])
def test_configs_full(ci):
    inp = mi.make_inputs(mi.CONFIGS[ci])
    ids, w, out, L = gpu_forward(inp)
    _check(inp, ids, w, out, L)


def _tile_picks(cfg):
    """Picks per tile, as the library chooses it from the average picks per
    expert (8 up to 2, 16 below 32, 32 below 64, else 64)."""
    P = cfg.S * cfg.k
    if P <= 2 * cfg.E:
        return 8
    if P >= 64 * cfg.E:
        return 64
    return 32 if P >= 32 * cfg.E else 16


def _sort_state(blk, ids):
    """The GPU's expert sort of the last call, read back from the workspace, and
    checked for what is unique about it: every expert's picks fill one segment
    of positions (experts in ascending order), cut into tiles of nt picks (the
    last one partial).  The order of picks inside a segment is not unique.
    Returns (slot [S, k], tile [S, k], tiles [n_tiles, 4], nt)."""
    import torch
    s = blk.shape
    S, k, E = s.S, s.k, s.E
    st = moe.read_region(s, blk.ws, moe.MOE_WS_STATUS, torch.int32).numpy()
    pos = moe.read_region(s, blk.ws, moe.MOE_WS_POS, torch.int32).numpy()
    n_tiles = int(st[3])
    tiles = moe.read_region(s, blk.ws, moe.MOE_WS_TILES, torch.int32).numpy().reshape(-1, 4)[:n_tiles]
    nt = _tile_picks(mi.MoEConfig("x", S=S, d=s.d, E=E, k=k, I=s.I))
    assert int(st[2]) == S * k
    cnt = np.bincount(ids.ravel(), minlength=E)
    seg = np.concatenate([[0], np.cumsum(cnt)])
    flat_ids = ids.ravel()
    # positions: a permutation of 0..P-1 with expert e's picks in its segment
    assert np.array_equal(np.sort(pos), np.arange(S * k))
    assert np.all(pos >= seg[flat_ids]) and np.all(pos < seg[flat_ids + 1])
    # tiles: expert e's segment in order, nt picks each but the last
    want = [(e, seg[e] + i, min(nt, cnt[e] - i)) for e in range(E) for i in range(0, cnt[e], nt)]
    got = sorted((int(t[0]), int(t[1]), int(t[2])) for t in tiles)
    assert got == sorted(want)
    pos2tile = np.empty(S * k, np.int64)
    for ti, (e, p0, n, _) in enumerate(tiles):
        pos2tile[p0:p0 + n] = ti
    tile = pos2tile[pos]
    slot = pos - tiles[tile, 1]
    return slot.reshape(S, k), tile.reshape(S, k), tiles, nt


def _cover_rows(ids, slot, tile, targets_of, min_rows, seed=0):
    """Token rows whose picks cover every target (greedy: most new targets
    first, then fewest experts the oracle has not dequantised yet), topped up
    to min_rows with rows that add as few experts as possible."""
    S = ids.shape[0]
    rng = np.random.default_rng(seed)
    cov = [set(targets_of(t)) for t in range(S)]
    need = set().union(*cov)
    chosen, experts = [], set()
    while need:
        best = max(range(S), key=lambda t: (len(cov[t] & need), -len(set(ids[t]) - experts)))
        assert cov[best] & need
        chosen.append(best)
        need -= cov[best]
        experts |= set(ids[best])
    rest = [t for t in rng.permutation(S) if t not in chosen]
    rest.sort(key=lambda t: len(set(ids[t]) - experts))
    for t in rest:
        if len(chosen) >= min_rows:
            break
        chosen.append(int(t))
        experts |= set(ids[t])
    return sorted(chosen)


def _full_size_parity(ci, min_rows, hot_targets):
    cfg = mi.CONFIGS[ci]
    inp = mi.make_inputs(cfg)
    blk = device_block(inp)
    ids_t, w_t, out_t = blk.forward()
    moe.check_device_status(blk.ws, "forward")
    ids, w, out = ids_t.cpu().numpy(), w_t.cpu().numpy(), out_t.cpu().numpy().astype(np.float64)
    import torch
    Lg = moe.read_region(blk.shape, blk.ws, moe.MOE_WS_LOGITS, torch.float32).numpy().reshape(cfg.S, cfg.E)
    # every token's routing: ids exactly, weights through the logits
    L = O.router_logits(inp.x, inp.w_gate, inp.logit_off)
    rids, rw = O.route(L, inp.bias, cfg.k)
    assert np.array_equal(ids, rids)
    check_routing_weights(Lg, inp.x, inp.w_gate, inp.logit_off, ids, w)
    slot, tile, tiles, nt = _sort_state(blk, ids)
    extra = hot_targets(ids, tiles, nt)

    def targets_of(t):
        tg = {("slot", int(s)) for s in slot[t]}
        tg |= {("tile", int(ti)) for ti in tile[t] if ("tile", int(ti)) in extra}
        tg |= {("chunk", int(ti), int(s) // 16) for ti, s in zip(tile[t], slot[t])
               if ("chunk", int(ti), int(s) // 16) in extra}
        return tg

    rows = _cover_rows(ids, slot, tile, targets_of, min_rows)
    covered = set().union(*(targets_of(t) for t in rows))
    assert {("slot", s) for s in range(nt)} <= covered and extra <= covered
    assert len(rows) >= min_rows
    _check(inp, ids, w, out, Lg, rows=rows)
    return rows, nt


def test_config3_full_size_tiles():
    """S = 128 (16-pick tiles, per-pick norm): the checked rows cover every
    tile slot and every tile of each expert that got more than one."""
    def multi_tile(ids, tiles, nt):
        per_e = {}
        for ti, t in enumerate(tiles):
            per_e.setdefault(int(t[0]), []).append(ti)
        return {("tile", ti) for tis in per_e.values() if len(tis) > 1 for ti in tis}

    rows, nt = _full_size_parity(3, 32, multi_tile)
    assert nt == 16


def test_config4_full_size_tiles():
    """S = 4096 (64-pick tiles, Zipf-skewed experts): the checked rows cover
    every tile slot (so every 16-pick epilogue chunk), the last tile of the
    hottest expert (partial unless its picks are a multiple of 64) and every
    chunk of one of its middle tiles."""
    def hottest(ids, tiles, nt):
        cnt = np.bincount(ids.ravel())
        e = int(np.argmax(cnt))
        tis = sorted((int(t[1]), ti) for ti, t in enumerate(tiles) if int(t[0]) == e)
        assert len(tis) >= 3, "the hottest expert has a middle tile"
        mid = tis[len(tis) // 2][1]
        # and the last tile of every expert that got more than one
        per_e = {}
        for ti, t in enumerate(tiles):
            per_e.setdefault(int(t[0]), []).append((int(t[1]), ti))
        multi = {("tile", max(v)[1]) for v in per_e.values() if len(v) > 1}
        return {("tile", tis[-1][1])} | {("chunk", mid, c) for c in range(nt // 16)} | multi

    rows, nt = _full_size_parity(4, 64, hottest)
    assert nt == 64


SMALL = [
    mi.MoEConfig("s1", S=1, d=128, E=8, k=1, I=128),
    mi.MoEConfig("s3", S=3, d=384, E=16, k=2, I=256),
    mi.MoEConfig("s17", S=17, d=256, E=40, k=8, I=128, post_norm=True),
    mi.MoEConfig("s33", S=33, d=512, E=12, k=3, I=384, zipf=1.1),
    mi.MoEConfig("kE", S=5, d=128, E=4, k=4, I=128),
    mi.MoEConfig("s70", S=70, d=256, E=8, k=2, I=256),      # > NT picks per expert
    mi.MoEConfig("s160", S=160, d=256, E=8, k=2, I=128),    # 32-pick tiles (40 picks per expert)
    mi.MoEConfig("maxEk", S=4, d=256, E=512, k=16, I=128),  # E and k at their maxima
    mi.MoEConfig("maxd", S=2, d=16384, E=8, k=2, I=128),    # d at its maximum (two gather passes)
    mi.MoEConfig("maxI", S=2, d=256, E=4, k=1, I=8192),     # I at its maximum
    # E a multiple of 128 above 8 tokens: the router on the tensor cores, in
    # 16-token tiles up to 32 tokens (one ragged tile; two, the last ragged),
    # in one ragged 128-token tile at 100
    mi.MoEConfig("tc9", S=9, d=384, E=128, k=4, I=128),
    mi.MoEConfig("tc30", S=30, d=256, E=256, k=8, I=128, zipf=1.1),
    mi.MoEConfig("tc100", S=100, d=512, E=256, k=8, I=128, zipf=1.1),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[c.name for c in SMALL])
def test_small_shapes(cfg):
    inp = _gap_inputs(cfg, 1)
    ids, w, out, L = gpu_forward(inp)
    _check(inp, ids, w, out, L)


def test_route_then_experts_separately():
    import torch
    inp = mi.make_inputs(mi.CONFIGS[0])
    blk = device_block(inp)
    s = blk.shape
    moe.route(s, blk.x, blk.w_gate, blk.bias, blk.logit_off, blk.ids, blk.weights, blk.ws)
    # experts on the oracle's ids / weights (reversed pick order: any order is allowed)
    L = O.router_logits(inp.x, inp.w_gate)
    rids, rw = O.route(L, inp.bias, inp.cfg.k)
    ids_t = torch.as_tensor(rids[:, ::-1].copy()).cuda()
    w_t = torch.as_tensor(rw[:, ::-1].astype(np.float32).copy()).cuda()
    moe.experts(s, blk.x, ids_t, w_t, blk.w13, blk.w13s, blk.w2, blk.w2s, blk.norm_w, blk.out, blk.ws)
    moe.check_device_status(blk.ws)
    assert np.array_equal(blk.ids.cpu().numpy(), rids)
    _, _, rout, _ = O.moe_forward(inp)
    assert O.parity_error(blk.out.cpu().numpy(), rout) <= OUT_TOL


def test_one_expert_takes_every_token():
    cfg = mi.MoEConfig("hot", S=40, d=256, E=8, k=2, I=128)
    inp = mi.make_inputs(cfg, 2, use_stored_attempts=False)
    inp.bias = np.zeros(cfg.E, np.float32)
    inp.bias[3] = 5.0           # expert 3 wins every token; 40 picks > NT
    inp.bias[6] = 4.0
    ids, w, out, L = gpu_forward(inp)
    assert np.all(ids == np.array([3, 6]))
    _check(inp, ids, w, out, L)


@pytest.mark.parametrize("S", [8, 24, 40], ids=["fused_select", "topk_then_fused_sort", "topk_kernel"])
def test_exact_ties_go_to_the_lower_id(S):
    """Zero router weights: every logit is 0 and every score 0.5, so the
    selection scores are the bias, drawn from three values: whole groups of
    experts tie exactly, and the k picks must be the experts of the largest
    bias values, lower ids first (the pages' order on equal scores: the
    lower expert index)."""
    cfg = mi.MoEConfig("ties", S=S, d=256, E=64, k=8, I=128)
    inp = mi.make_inputs(cfg, 3, use_stored_attempts=False)
    inp.w_gate = np.zeros_like(inp.w_gate)
    rng = np.random.default_rng(5)
    inp.bias = rng.choice(np.array([0.0, 0.25, 0.5], np.float32), size=cfg.E).astype(np.float32)
    ids, w, out, L = gpu_forward(inp)
    want = sorted(sorted(range(cfg.E), key=lambda e: (-float(inp.bias[e]), e))[:cfg.k])
    assert np.array_equal(ids, np.tile(np.array(want, np.int32), (S, 1)))
    assert np.allclose(w, 1.0 / cfg.k, rtol=1e-6, atol=0)
    _check(inp, ids, w, out, L)


def test_bad_ids_latch_status():
    import torch
    inp = mi.make_inputs(mi.CONFIGS[0])
    blk = device_block(inp)
    s = blk.shape
    ids = torch.tensor([[0, 1]] * 8, dtype=torch.int32).cuda()
    ids[2, 1] = 9          # out of range
    ids[5, 1] = 0          # repeated within token 5
    w = torch.full((8, 2), 0.5, dtype=torch.float32).cuda()
    moe.experts(s, blk.x, ids, w, blk.w13, blk.w13s, blk.w2, blk.w2s, None, blk.out, blk.ws)
    rc, det = moe.device_status(blk.ws)
    assert rc == moe.MOE_ERR_BAD_IDS and det in (2 * 2 + 1, 5 * 2 + 1)
    out = blk.out.cpu().numpy()
    assert np.all(np.isfinite(out))
    # the valid picks still contribute: token 2 = 0.5 * expert 0 only
    xf = O.bf16_to_f64(inp.x)
    y0 = O.expert_ffn(xf[2:3], inp.w13[0], inp.w13s[0], inp.w2[0], inp.w2s[0])[0]
    assert O.parity_error(out[2], 0.5 * y0) <= OUT_TOL
    assert moe.device_status(blk.ws)[0] == moe.MOE_OK      # cleared


def test_bad_ids_latch_status_many_picks():
    """More than 128 picks (the multi-CTA count and the per-token gather):
    an out-of-range id and a repeated one latch MOE_ERR_BAD_IDS, are left out
    of the sums, and every valid pick still contributes."""
    import torch
    cfg = mi.MoEConfig("bad_many", S=40, d=256, E=8, k=4, I=128)
    inp = mi.make_inputs(cfg, 4, use_stored_attempts=False)
    blk = device_block(inp)
    s = blk.shape
    rng = np.random.default_rng(11)
    ids_np = np.stack([np.sort(rng.choice(cfg.E, cfg.k, replace=False)) for _ in range(cfg.S)]).astype(np.int32)
    w_np = np.full((cfg.S, cfg.k), 0.25, np.float32)
    ids_np[7, 2] = 8                      # out of range
    ids_np[30, 3] = ids_np[30, 0]         # repeated within token 30
    moe.experts(s, blk.x, torch.as_tensor(ids_np).cuda(), torch.as_tensor(w_np).cuda(), blk.w13, blk.w13s, blk.w2,
                blk.w2s, None, blk.out, blk.ws)
    rc, det = moe.device_status(blk.ws)
    assert rc == moe.MOE_ERR_BAD_IDS and det in (7 * 4 + 2, 30 * 4 + 3)
    out = blk.out.cpu().numpy()
    xf = O.bf16_to_f64(inp.x)
    for t in (7, 30, 0):
        valid = [j for j in range(cfg.k) if 0 <= ids_np[t, j] < cfg.E and ids_np[t, j] not in ids_np[t, :j]]
        ref = sum(0.25 * O.expert_ffn(xf[t:t + 1], inp.w13[e], inp.w13s[e], inp.w2[e], inp.w2s[e])[0]
                  for e in ids_np[t, valid])
        assert O.parity_error(out[t], ref) <= OUT_TOL
    assert moe.device_status(blk.ws)[0] == moe.MOE_OK      # cleared
    # the counters are left clear: a valid call on the same workspace matches the oracle
    good = np.stack([np.sort(rng.choice(cfg.E, cfg.k, replace=False)) for _ in range(cfg.S)]).astype(np.int32)
    moe.experts(s, blk.x, torch.as_tensor(good).cuda(), torch.as_tensor(w_np).cuda(), blk.w13, blk.w13s, blk.w2,
                blk.w2s, None, blk.out, blk.ws)
    moe.check_device_status(blk.ws, "second call")
    out = blk.out.cpu().numpy()
    for t in (0, 7, 39):
        ref = sum(0.25 * O.expert_ffn(xf[t:t + 1], inp.w13[e], inp.w13s[e], inp.w2[e], inp.w2s[e])[0]
                  for e in good[t])
        assert O.parity_error(out[t], ref) <= OUT_TOL


def test_bad_scale_latches_status():
    # e8m0 255 is NaN (OCP MX v1.0); it is reported, not silently used
    inp = mi.make_inputs(mi.CONFIGS[0])
    inp.w2s = inp.w2s.copy()
    inp.w2s[:, 7, 1] = 255
    blk = device_block(inp)
    blk.forward()
    rc, det = moe.device_status(blk.ws)
    assert rc == moe.MOE_ERR_BAD_SCALE and det == 255


@pytest.mark.parametrize("shift13,shift2", [(24, -24), (-20, 20), (40, -40)])
def test_scale_range(shift13, shift2):
    # every e8m0 byte 0..254 is a valid scale: gate_up scales moved up (down)
    # by 2^shift13 and the down scales back, so h spans a very different range
    # from y (kept well inside fp32: h grows as 2^(2 shift13)); the routing is
    # unchanged
    inp = mi.make_inputs(mi.CONFIGS[0])
    inp.w13s = np.clip(inp.w13s.astype(np.int64) + shift13, 0, 254).astype(np.uint8)
    inp.w2s = np.clip(inp.w2s.astype(np.int64) + shift2, 0, 254).astype(np.uint8)
    ids, w, out, L = gpu_forward(inp)
    _check(inp, ids, w, out, L)


@pytest.mark.parametrize("ci,pinned", [(1, True), (1, False), (2, True), (3, True)])
def test_forward_host_matches_forward(ci, pinned):
    """Host buffers: a small pinned x is copied in by the staging kernel (S = 8
    and 32), small pinned outputs are written over the link by the combine
    (out, ids and weights at S = 8), the others go through the workspace and a
    copy (pageable ones, S = 128's x); either way the bytes equal moe_forward's."""
    import torch
    inp = mi.make_inputs(mi.CONFIGS[ci])
    blk = device_block(inp)
    ids, w, out = [t.cpu().numpy() for t in blk.forward()]
    s = blk.shape

    def host(t):
        return t.pin_memory() if pinned else t

    xh = host(torch.as_tensor(inp.x).view(torch.bfloat16).clone())
    oh = host(torch.empty((s.S, s.d), dtype=torch.float32))
    ih = host(torch.empty((s.S, s.k), dtype=torch.int32))
    wh = host(torch.empty((s.S, s.k), dtype=torch.float32))
    moe.forward_host(s, xh, blk.w_gate, blk.bias, blk.logit_off, blk.w13, blk.w13s, blk.w2, blk.w2s,
                     blk.norm_w, ih, wh, oh, blk.ws)
    torch.cuda.current_stream().synchronize()
    moe.check_device_status(blk.ws)
    assert np.array_equal(ih.numpy(), ids) and np.array_equal(wh.numpy(), w)
    assert np.array_equal(oh.numpy(), out)


@pytest.mark.parametrize("want", ["ids", "weights", "neither"])
def test_forward_host_one_routing_output(want):
    """ids_host and weights_host may each be NULL: the other (pinned, written
    by the combine at S = 8) and out still come back."""
    import torch
    inp = mi.make_inputs(mi.CONFIGS[1])
    blk = device_block(inp)
    ids, w, out = [t.cpu().numpy() for t in blk.forward()]
    s = blk.shape
    xh = torch.as_tensor(inp.x).view(torch.bfloat16).clone().pin_memory()
    oh = torch.empty((s.S, s.d), dtype=torch.float32).pin_memory()
    ih = torch.full((s.S, s.k), -7, dtype=torch.int32).pin_memory() if want == "ids" else None
    wh = torch.full((s.S, s.k), -7.0, dtype=torch.float32).pin_memory() if want == "weights" else None
    moe.forward_host(s, xh, blk.w_gate, blk.bias, blk.logit_off, blk.w13, blk.w13s, blk.w2, blk.w2s,
                     blk.norm_w, ih, wh, oh, blk.ws)
    torch.cuda.current_stream().synchronize()
    moe.check_device_status(blk.ws)
    assert np.array_equal(oh.numpy(), out)
    if ih is not None:
        assert np.array_equal(ih.numpy(), ids)
    if wh is not None:
        assert np.array_equal(wh.numpy(), w)


@pytest.mark.parametrize("ci", [2, 3])
def test_repeat_calls_are_deterministic(ci):
    """Synchronised calls with other work on the stream in between (a write
    larger than L2) give identical bytes: every kernel reads its predecessors'
    outputs coherently, whatever the caches hold from the previous call."""
    import torch
    inp = mi.make_inputs(mi.CONFIGS[ci])
    blk = device_block(inp)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ref = None
    for _ in range(6):
        flush.zero_()
        got = [t.cpu().numpy().copy() for t in blk.forward()]
        moe.check_device_status(blk.ws, "repeat")
        if ref is None:
            ref = got
        for u, v in zip(got, ref):
            assert np.array_equal(u, v)


@pytest.mark.parametrize("ci", [0, 1, 2, 3])
def test_back_to_back_calls_with_different_routing(ci):
    """Calls enqueued one after another on one stream, with nothing between
    them, overlap on the device (each kernel may start before its predecessor
    ends, and the expert kernel before the token gather ends).  Four inputs with
    different routing, each called many times in turn into fresh outputs, must
    give exactly what each gives alone."""
    import torch
    inp = mi.make_inputs(mi.CONFIGS[ci])
    blk = device_block(inp)
    s = blk.shape
    xs = [blk.x, blk.x.roll(1, 0).contiguous(), blk.x.flip(1).contiguous(), (-blk.x).contiguous()]

    def outs():
        return (torch.empty((s.S, s.k), dtype=torch.int32, device="cuda"),
                torch.empty((s.S, s.k), dtype=torch.float32, device="cuda"),
                torch.empty((s.S, s.d), dtype=torch.float32, device="cuda"))

    def call(x, o):
        moe.forward(s, x, blk.w_gate, blk.bias, blk.logit_off, blk.w13, blk.w13s, blk.w2, blk.w2s,
                    blk.norm_w, *o, blk.ws)

    refs = []
    for x in xs:
        o = outs()
        call(x, o)
        torch.cuda.synchronize()
        moe.check_device_status(blk.ws, "alone")
        refs.append(o)
    rounds = 12 if ci < 3 else 4
    got = []
    for _ in range(rounds):
        for v, x in enumerate(xs):
            o = outs()
            call(x, o)
            got.append((v, o))
    torch.cuda.synchronize()
    moe.check_device_status(blk.ws, "back to back")
    for v, o in got:
        for a, b in zip(o, refs[v]):
            assert torch.equal(a, b), f"input {v} differs when enqueued back to back"
