"""GPU parity: every step of the hot path and the whole layer against the CPU
oracle, through the C ABI, on seeded inputs of the workloads' shapes.

Sizes: the small R1- and BF16-shaped layers run in full against the oracle
(several tiles in every dimension, ragged tails); the full-size R1 layers
(128, 1024 and 4096 tokens) are checked bit for bit on routing and dispatch
for every token and on the layer output for a seeded sample of tokens, in
the same launch configuration the benchmark times.  Tolerances are stated
in tests/_gpu_common.py.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_07_gb300 as moe
import synth
from oracle import layer as olayer
from oracle import permute as opermute
from oracle import quant as oquant
from oracle import routing as orouting

from _gpu_common import (BF16_TOL, FP8_TOL, W_RTOL, Workload, build_library, check_close,
                         fp8_codes_equal, oracle_layer, rms, to_np)

pytestmark = pytest.mark.gpu

SMALL = ["tiny_bf16", "v2lite_bf16", "r1_mini", "r1_mini_zipf", "r1_mini_i512", "bf16_mini"]
FULL = ["r1_decode_t128", "r1_zipf_t1024", "r1_prefill_t4096"]
# tokens of the full-size layers whose output is compared with the oracle: all
# 128 of the decode batch (every active expert's FFN output enters some
# token), 64 seeded tokens of the wider batches
SAMPLE = {"r1_decode_t128": 128, "r1_zipf_t1024": 64, "r1_prefill_t4096": 64}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    return build_library()


_cache = {}


def workload(name, seed=0, perm=None, T=None):
    key = (name, seed, perm, T)
    if key not in _cache:
        if any(k[0] in FULL for k in _cache) and name in FULL:
            for k in [k for k in _cache if k[0] in FULL]:
                del _cache[k]          # one full-size layer resident at a time
            torch.cuda.empty_cache()
        shape = synth.CONFIGS[name]
        if T is not None:
            shape = shape.with_tokens(T)
        _cache[key] = Workload(shape, seed=seed, perm=perm)
    return _cache[key]


def run_route(wl, T=None):
    s = wl.shape
    T = s.tokens if T is None else T
    dev = wl.dev
    logits = torch.full((T, s.num_experts), float("nan"), device="cuda")
    ids = torch.full((T, s.top_k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, s.top_k), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    l2p = None if wl.log2phys is None else torch.as_tensor(wl.log2phys, device="cuda")
    moe.route(moe.make_config(s), T, dev["x"], dev["wg"], dev["e_bias"], dev["logit_offset"],
              l2p, logits, ids, w, st)
    torch.cuda.synchronize()
    return to_np(logits), to_np(ids), to_np(w), int(st.item())


# ------------------------------------------------------------------ routing
@pytest.mark.parametrize("name", SMALL + FULL)
def test_route_bit_exact(lib, name):
    wl = workload(name)
    logits, ids, w, st = run_route(wl)
    n = wl.np
    ref_l = orouting.gate_logits(n["x_bits"], n["wg_bits"], n["logit_offset"])
    assert np.array_equal(logits.view(np.uint32), ref_l.view(np.uint32)), "logits differ"
    phys, ref_w, _ = orouting.route(ref_l, wl.shape, n["e_bias"], n["log2phys"])
    assert np.array_equal(ids, phys)
    np.testing.assert_allclose(w, ref_w, rtol=W_RTOL, atol=0)
    assert st == 0


@pytest.mark.parametrize("T", [1, 2, 5, 33])
def test_route_small_batches(lib, T):
    wl = workload("r1_mini", seed=3, T=T)
    logits, ids, w, st = run_route(wl)
    n = wl.np
    ref_l = orouting.gate_logits(n["x_bits"], n["wg_bits"], n["logit_offset"])
    phys, ref_w, _ = orouting.route(ref_l, wl.shape, n["e_bias"], None)
    assert np.array_equal(ids, phys) and st == 0
    np.testing.assert_allclose(w, ref_w, rtol=W_RTOL, atol=0)


def test_route_with_random_permutation(lib):
    wl = workload("r1_mini", seed=5, perm="random")
    _, ids, w, _ = run_route(wl)
    n = wl.np
    ref_l = orouting.gate_logits(n["x_bits"], n["wg_bits"], n["logit_offset"])
    phys, ref_w, logical = orouting.route(ref_l, wl.shape, n["e_bias"], n["log2phys"])
    assert np.array_equal(ids, phys) and np.array_equal(ids, wl.log2phys[logical])


def test_sigmoid_score_equals_fp64_bit_for_bit(lib):
    """The selection kernel's sigmoid score (double-float fp32 arithmetic,
    with the fp64 expression wherever that cannot decide the rounding) is
    the fp64 sigmoid rounded to fp32 on every input: 8M normal logits at four
    spreads, a dense sweep of [-90, 90] (it crosses many rounding midpoints)
    and the edges of the fast range.  The oracle's numpy evaluation agrees as
    well."""
    g = torch.Generator(device="cuda").manual_seed(5)
    parts = [torch.randn(2_000_000, device="cuda", generator=g) * sd for sd in (0.5, 2.0, 8.0, 30.0)]
    parts.append(torch.linspace(-90.0, 90.0, 1_000_001, device="cuda"))
    parts.append(torch.tensor([0.0, -0.0, 1e-30, -1e-30, 1e-7, -1e-7, 80.0, -80.0, 80.00001,
                               -80.00001, 87.3, -87.3, 88.8, -88.8, 100.0, -100.0, 1e4, -1e4,
                               float("inf"), float("-inf")], device="cuda"))
    lg = torch.cat(parts).contiguous()
    n = lg.numel()
    fast, ref = torch.empty_like(lg), torch.empty_like(lg)
    fb = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = moe.lib().moe_selftest_sigmoid(lg.data_ptr(), n, fast.data_ptr(), ref.data_ptr(),
                                        fb.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert torch.equal(fast.view(torch.int32), ref.view(torch.int32))
    # inputs beyond |l| = 80 always take the fp64 expression; the others rarely
    out_of_range = int((~(lg.abs() <= 80.0)).sum().item())
    assert int(fb.item()) - out_of_range < (n - out_of_range) // 1000
    with np.errstate(over="ignore"):   # exp(1e4) is inf, as it should be
        want = orouting.sigmoid_scores(lg.cpu().numpy())
    assert np.array_equal(to_np(fast).view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("name", ["r1_mini", "bf16_mini", "tiny_bf16"])
def test_route_ties_go_to_the_lower_index(lib, name):
    """Every odd expert's gate row (and bias) copies the even expert below it,
    so scores tie in pairs: the selection, group scores and slot order must
    break every tie toward the lower index, as the oracle does."""
    shape = synth.CONFIGS[name]
    wl = Workload(shape, seed=7)
    for key in ("wg", "e_bias", "logit_offset"):
        if wl.dev.get(key) is not None:
            t = wl.dev[key].clone()
            t[1::2] = t[0::2]
            wl.dev[key] = t
    wl._np = None
    logits, ids, w, st = run_route(wl)
    assert st == 0
    assert np.array_equal(logits[:, 1::2], logits[:, 0::2])   # the ties are real
    n = wl.np
    ref_l = orouting.gate_logits(n["x_bits"], n["wg_bits"], n["logit_offset"])
    phys, ref_w, _ = orouting.route(ref_l, shape, n["e_bias"], n.get("log2phys"))
    assert np.array_equal(ids, phys)
    np.testing.assert_allclose(w, ref_w, rtol=W_RTOL)


# ------------------------------------------------------------ quantisation
def _quant_x(cfg, x, T, H):
    q = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    s = torch.empty((T, H // 128), dtype=torch.float32, device="cuda")
    moe.act_requant(cfg, moe.ACT_IDENTITY, T, x, q, s)
    torch.cuda.synchronize()
    return to_np(q), to_np(s)


@pytest.mark.parametrize("name", ["r1_mini", "r1_decode_t128"])
def test_quant_x_bit_exact(lib, name):
    wl = workload(name)
    s = wl.shape
    q, sc = _quant_x(moe.make_config(s), wl.dev["x"], s.tokens, s.hidden)
    rq, rs = oquant.quant_groups_fp8(oquant.bf16_from_bits(wl.np["x_bits"]))
    assert fp8_codes_equal(q, rq) and np.array_equal(sc, rs)


@pytest.mark.parametrize("name,T", [("r1_mini", None), ("r1_decode_t128", None),
                                    ("r1_prefill_t4096", None), ("r1_mini", 1)])
def test_route_quantize_equals_route_then_quantize(lib, name, T):
    """Routing with the x quantisation in the selection kernel (the layer's own
    launch sequence) gives the bits of moe_route followed by moe_act_requant."""
    wl = workload(name, T=T)
    s = wl.shape
    T = s.tokens
    cfg = moe.make_config(s)
    dev = wl.dev
    l2p = None if wl.log2phys is None else torch.as_tensor(wl.log2phys, device="cuda")
    outs = []
    for fused in (False, True):
        logits = torch.full((T, s.num_experts), float("nan"), device="cuda")
        ids = torch.full((T, s.top_k), -7, dtype=torch.int32, device="cuda")
        w = torch.full((T, s.top_k), float("nan"), device="cuda")
        xq = torch.full((T, s.hidden), 0x55, dtype=torch.uint8, device="cuda")
        xs = torch.full((T, s.hidden // 128), -1.0, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            moe.route_quantize(cfg, T, dev["x"], dev["wg"], dev["e_bias"], dev["logit_offset"],
                               l2p, logits, ids, w, xq, xs, st)
        else:
            moe.route(cfg, T, dev["x"], dev["wg"], dev["e_bias"], dev["logit_offset"], l2p,
                      logits, ids, w, st)
            moe.act_requant(cfg, moe.ACT_IDENTITY, T, dev["x"], xq, xs)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        outs.append((logits, ids, w, xq, xs))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_quant_x_ties_zeros_and_extremes(lib):
    s = synth.CONFIGS["r1_mini"]
    H = s.hidden
    x = torch.randn(6, H, device="cuda").to(torch.bfloat16)
    x[0] = 0                                       # all-zero row: scale 1, codes 0
    x[1, :128] = 0.53125                           # midpoints of the e4m3 grid ...
    x[1, 1::2] = -3.125
    x[1, 0] = 448.0                                # ... with scale exactly 1
    x[2] *= 1e-30                                  # tiny magnitudes
    x[3] *= 1e30                                   # huge magnitudes
    x[4, 128:256] = 0
    q, sc = _quant_x(moe.make_config(s), x, 6, H)
    bits = x.view(torch.int16).cpu().numpy().view(np.uint16)
    rq, rs = oquant.quant_groups_fp8(oquant.bf16_from_bits(bits))
    assert fp8_codes_equal(q, rq) and np.array_equal(sc, rs)
    assert sc[1, 0] == 1.0 and sc[0].tolist() == [1.0] * (H // 128)


@pytest.mark.parametrize("fp8", [True, False])
def test_silu_mul_requant(lib, fp8):
    s = synth.CONFIGS["r1_mini" if fp8 else "bf16_mini"]
    cfg = moe.make_config(s)
    rows, I = 37, s.inter
    gen = torch.Generator(device="cuda").manual_seed(11)
    g = (torch.randn(rows, 2 * I, device="cuda", generator=gen) * 3).contiguous()
    g[5] = 0                                        # a zero row
    rows_dev = torch.tensor([30], dtype=torch.int32, device="cuda")
    if fp8:
        out = torch.full((rows, I), 0x55, dtype=torch.uint8, device="cuda")
        sc = torch.full((rows, I // 128), -1.0, device="cuda")
    else:
        out = torch.zeros((rows, I), dtype=torch.bfloat16, device="cuda")
        sc = None
    moe.act_requant(cfg, moe.ACT_SILU_MUL, rows, g, out, sc, rows_dev=rows_dev)
    torch.cuda.synchronize()
    h = olayer.silu_mul(to_np(g)[:30])
    if fp8:
        rq, rs = oquant.quant_groups_fp8(h.astype(np.float32))
        q = to_np(out)
        gs = to_np(sc)
        np.testing.assert_allclose(gs[:30], rs, rtol=1e-6, atol=0)
        deq = oquant.dequant_groups_fp8(q[:30], gs[:30])
        ref = oquant.dequant_groups_fp8(rq, rs)
        qn = np.where(q[:30] == 0x80, 0, q[:30])
        rn = np.where(rq == 0x80, 0, rq)
        diff = qn != rn
        # a code may differ only where fp32 silu rounding straddles a midpoint:
        # by one e4m3 step, rarely
        assert diff.mean() < 1e-3
        step = np.maximum(np.abs(ref) * 2.0 ** -3, np.repeat(rs, 128, axis=1) * 2.0 ** -9)
        assert np.all(np.abs(deq - ref)[diff] <= step[diff] * 1.0001)
        assert np.all(q[30:] == 0x55) and np.all(gs[30:] == -1.0)
    else:
        hb = to_np(out.float())
        ref = oquant.bf16_round(h)
        # fp32 silu on the device against fp64 here: a value may round to the
        # neighbouring bf16 (one unit in the last place), rarely
        a = np.abs(ref)
        _, ex = np.frexp(np.where(a > 0, a, 1.0))
        ulp = np.where(a > 0, np.ldexp(1.0, ex.astype(np.int64) - 1 - 7), 0.0)
        diff = hb[:30] != ref
        assert diff.mean() < 1e-3
        assert np.all(np.abs(hb[:30] - ref)[diff] <= ulp[diff])
        assert np.all(hb[30:] == 0)


# ------------------------------------------------------------------ permute
def run_permute(cfg, s, ids_t, x_rows, x_scales):
    T, k, E, S, H = ids_t.shape[0], s.top_k, s.num_experts, s.num_shared, s.hidden
    rows = T * (k + S)
    fp8 = s.dtype == "fp8"
    off = torch.full((E + S + 1,), -5, dtype=torch.int32, device="cuda")
    src = torch.full((rows,), -5, dtype=torch.int32, device="cuda")
    ros = torch.full((T, k), -5, dtype=torch.int32, device="cuda")
    xp = torch.zeros((rows, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device="cuda")
    xps = torch.zeros((rows, H // 128), device="cuda") if fp8 else None
    nws = moe.permute_workspace_size(cfg, T)
    ws = torch.empty(max(nws, 1), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.permute(cfg, T, ids_t, x_rows, x_scales, off, src, ros, xp, xps, ws, nws, st)
    torch.cuda.synchronize()
    return dict(off=to_np(off), src=to_np(src), ros=to_np(ros), xp=xp, xps=xps,
                status=int(st.item()))


@pytest.mark.parametrize("name", ["r1_mini", "bf16_mini", "v2lite_bf16", "r1_decode_t128",
                                  "r1_zipf_t1024", "r1_prefill_t4096"])
def test_permute_bit_exact(lib, name):
    wl = workload(name)
    s = wl.shape
    cfg = moe.make_config(s)
    _, ids, _, _ = run_route(wl)
    ids_t = torch.as_tensor(ids, device="cuda")
    if s.dtype == "fp8":
        xq = torch.empty((s.tokens, s.hidden), dtype=torch.uint8, device="cuda")
        xs = torch.empty((s.tokens, s.hidden // 128), device="cuda")
        moe.act_requant(cfg, moe.ACT_IDENTITY, s.tokens, wl.dev["x"], xq, xs)
        rows_src, rows_sc = xq, xs
    else:
        rows_src, rows_sc = wl.dev["x"], None
    r = run_permute(cfg, s, ids_t, rows_src, rows_sc)
    off, src, ros = opermute.permute(ids, s.num_experts, s.num_shared)
    assert np.array_equal(r["off"], off)
    assert np.array_equal(r["src"], src)
    assert np.array_equal(r["ros"], ros)
    tok = opermute.token_of_slot(src, s.tokens, s.top_k)
    assert torch.equal(r["xp"], rows_src[torch.as_tensor(tok, device="cuda")])
    if rows_sc is not None:
        assert torch.equal(r["xps"], rows_sc[torch.as_tensor(tok, device="cuda")])
    assert r["status"] == 0


def test_permute_edge_cases(lib):
    s = synth.CONFIGS["bf16_mini"]
    cfg = moe.make_config(s)
    T, k, E = 40, s.top_k, s.num_experts
    x = torch.randn(T, s.hidden, device="cuda").to(torch.bfloat16)
    # every token to the same experts (others empty); then invalid ids
    ids = np.tile(np.array([3, 0, 6], np.int32), (T, 1))
    r = run_permute(cfg, s, torch.as_tensor(ids, device="cuda"), x, None)
    off, src, ros = opermute.permute(ids, E, s.num_shared)
    assert np.array_equal(r["off"], off) and np.array_equal(r["ros"], ros)
    assert np.array_equal(r["src"], src) and r["status"] == 0
    bad = ids.copy()
    bad[7, 1] = -1
    bad[9, 2] = E
    r = run_permute(cfg, s, torch.as_tensor(bad, device="cuda"), x, None)
    assert r["status"] & moe.DEV_BAD_EXPERT_ID
    assert r["ros"][7, 1] == -1 and r["ros"][9, 2] == -1
    valid = np.ones_like(bad, bool)
    valid[7, 1] = valid[9, 2] = False
    counts = np.bincount(bad[valid], minlength=E)
    assert np.array_equal(np.diff(r["off"])[:E], counts)


# ------------------------------------------------------------- grouped GEMM
GEMM_ROWS = [0, 1, 15, 16, 17, 0, 63, 64, 65, 129, 3]


@pytest.mark.parametrize("fp8,N,K,out_bf16", [(True, 256, 384, False), (True, 384, 1024, True),
                                              (False, 256, 320, False), (False, 128, 512, True)])
def test_grouped_gemm(lib, fp8, N, K, out_bf16):
    s = synth.CONFIGS["r1_mini" if fp8 else "bf16_mini"]
    cfg = moe.make_config(s)
    counts = np.array(GEMM_ROWS)
    G = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(off[-1]) + 5                      # 5 trailing rows outside every group
    g = torch.Generator(device="cuda").manual_seed(7)
    a32 = torch.randn(rows, K, device="cuda", generator=g)
    w32 = torch.randn(G, N, K, device="cuda", generator=g) * 0.05
    if fp8:
        a = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
        asc = torch.empty((rows, K // 128), device="cuda")
        cfg_q = moe.make_config(synth.MoEShape("q", rows, K, 128, 1, 0, 1, dtype="fp8"))
        moe.act_requant(cfg_q, moe.ACT_IDENTITY, rows, a32.to(torch.bfloat16), a, asc)
        w, wsc = synth.block_quantize_e4m3(w32)
    else:
        a, asc = a32.to(torch.bfloat16), None
        w, wsc = w32.to(torch.bfloat16), None
    c = torch.full((rows, N), float("nan"), device="cuda",
                   dtype=torch.bfloat16 if out_bf16 else torch.float32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.grouped_gemm(cfg, G, N, K, rows, a, asc, torch.as_tensor(off, device="cuda"), w, wsc, c,
                     moe.OUT_BF16 if out_bf16 else moe.OUT_F32, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    if fp8:
        ref = olayer.grouped_gemm(s, off, to_np(a), to_np(w), to_np(asc), to_np(wsc))
    else:
        ref = olayer.grouped_gemm(s, off, to_np(a.view(torch.int16)).view(np.uint16),
                                  to_np(w.view(torch.int16)).view(np.uint16))
    got = to_np(c.float())
    inside = off[-1]
    check_close(got[:inside], ref[:inside], 1e-3 if not out_bf16 else 1e-4, bf16_out=out_bf16)
    assert np.all(np.isnan(got[inside:]))


WIDE_ROWS = [0, 1, 127, 128, 129, 0, 255, 64, 300, 17]


@pytest.mark.parametrize("N,K,counts", [(384, 1024, WIDE_ROWS), (512, 1024, WIDE_ROWS),
                                         (7168, 2048, [150, 130, 120, 0, 140, 600, 7])])
def test_grouped_gemm_tile_variants_agree(lib, N, K, counts):
    """The kernels chosen by rows per group promote per K block in the same
    order: the same bits, within the oracle's tolerance.  Empty groups
    appended to the same problem move it between them: 32-row activation
    tiles for few rows per group; for 16 or more, 128 token rows against 256
    output columns when N is a multiple of 256 (512, and the R1 down
    projection's 7168 with ragged 128-row token tiles), else 64-row tiles."""
    s = synth.CONFIGS["r1_mini"]
    cfg = moe.make_config(s)
    counts = np.array(counts)
    rows = int(counts.sum())
    g = torch.Generator(device="cuda").manual_seed(11)
    a32 = torch.randn(rows, K, device="cuda", generator=g)
    a = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
    asc = torch.empty((rows, K // 128), device="cuda")
    cfg_q = moe.make_config(synth.MoEShape("q", rows, K, 128, 1, 0, 1, dtype="fp8"))
    moe.act_requant(cfg_q, moe.ACT_IDENTITY, rows, a32.to(torch.bfloat16), a, asc)
    w, wsc = synth.block_quantize_e4m3(
        torch.randn(len(counts), N, K, device="cuda", generator=g) * 0.05)
    outs = []
    for extra in (0, 40, 70):   # WIDE_ROWS: 102, 20 and 13 rows per group
        G = len(counts) + extra
        off = np.concatenate([[0], np.cumsum(np.concatenate([counts, np.zeros(extra, int)]))])
        wpad = torch.cat([w, torch.zeros((extra, N, K), dtype=w.dtype, device="cuda")])
        spad = torch.cat([wsc, torch.ones((extra,) + tuple(wsc.shape[1:]), device="cuda")])
        c = torch.full((rows, N), float("nan"), device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        moe.grouped_gemm(cfg, G, N, K, rows, a, asc,
                         torch.as_tensor(off.astype(np.int32), device="cuda"), wpad, spad, c,
                         moe.OUT_F32, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        outs.append(c)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ref = olayer.grouped_gemm(s, off, to_np(a), to_np(w), to_np(asc), to_np(wsc))
    check_close(to_np(outs[0]), ref, 1e-3)


def test_grouped_gemm_rejects_inconsistent_offsets(lib):
    s = synth.CONFIGS["r1_mini"]
    cfg = moe.make_config(s)
    K, N, rows = 128, 128, 32
    a = torch.zeros((rows, K), dtype=torch.uint8, device="cuda")
    asc = torch.ones((rows, 1), device="cuda")
    w = torch.zeros((2, N, K), dtype=torch.uint8, device="cuda")
    wsc = torch.ones((2, 1, 1), device="cuda")
    c = torch.full((rows, N), 3.0, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    off = torch.tensor([0, 20, 10], dtype=torch.int32, device="cuda")   # decreasing
    moe.grouped_gemm(cfg, 2, N, K, rows, a, asc, off, w, wsc, c, moe.OUT_F32, st)
    torch.cuda.synchronize()
    assert int(st.item()) & moe.DEV_BAD_OFFSETS
    assert torch.all(c == 3.0)                  # nothing was written


def test_swiglu_wide_rejects_inconsistent_offsets(lib):
    """The token-rows-on-M SwiGLU kernel (16+ rows per group) flags offsets that
    run backwards or past the rows, and writes nothing."""
    s = synth.CONFIGS["r1_mini"]
    cfg = moe.make_config(s)
    K, inter, rows = 128, 128, 64
    a = torch.zeros((rows, K), dtype=torch.uint8, device="cuda")
    asc = torch.ones((rows, 1), device="cuda")
    w = torch.zeros((2, 2 * inter, K), dtype=torch.uint8, device="cuda")
    wsc = torch.ones((2, 2, 1), device="cuda")
    for bad in ([0, 40, 20], [0, 30, 70]):      # decreasing; past the rows
        h = torch.full((rows, inter), 7, dtype=torch.uint8, device="cuda")
        hs = torch.full((rows, 1), 3.0, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        off = torch.tensor(bad, dtype=torch.int32, device="cuda")
        moe.grouped_gemm_swiglu(cfg, 2, inter, K, rows, a, asc, off, w, wsc, h, hs, st)
        torch.cuda.synchronize()
        assert int(st.item()) & moe.DEV_BAD_OFFSETS
        assert torch.all(h == 7) and torch.all(hs == 3.0)


# ------------------------------------------------------------------ combine
@pytest.mark.parametrize("out_bf16", [False, True])
def test_combine(lib, out_bf16):
    s = synth.CONFIGS["v2lite_bf16"]
    cfg = moe.make_config(s)
    T, k, E, S, H = 50, s.top_k, s.num_experts, s.num_shared, s.hidden
    rng = np.random.default_rng(3)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    off, src, ros = opermute.permute(ids, E, S)
    rows = int(off[-1])
    y = torch.randn(rows, H, device="cuda")
    w = torch.rand(T, k, device="cuda")
    out = torch.empty((T, H), device="cuda", dtype=torch.bfloat16 if out_bf16 else torch.float32)
    moe.combine(cfg, T, y, torch.as_tensor(ros, device="cuda"), w,
                torch.as_tensor(off, device="cuda"), out, moe.OUT_BF16 if out_bf16 else moe.OUT_F32)
    torch.cuda.synchronize()
    ref = olayer.combine(to_np(y.float()), ros, to_np(w), off, E, S)
    check_close(to_np(out.float()), ref, 1e-5, bf16_out=out_bf16)


# ------------------------------------------------------------- whole layer
def run_layer(wl, T=None, out_bf16=False, layer=None):
    s = wl.shape
    T = s.tokens if T is None else T
    layer = layer or wl.layer()
    out = torch.full((max(T, 1), s.hidden), float("nan"), device="cuda",
                     dtype=torch.bfloat16 if out_bf16 else torch.float32)
    layer.forward(wl.dev["x"][:T] if T else wl.dev["x"][:1], out,
                  moe.OUT_BF16 if out_bf16 else moe.OUT_F32, T=T)
    torch.cuda.synchronize()
    return layer, out


def _check_layer_routing(layer, s, ref):
    T, k, E, S = s.tokens, s.top_k, s.num_experts, s.num_shared
    ids = to_np(layer.view("topk_ids", torch.int32, (T, k)))
    off = to_np(layer.view("expert_offsets", torch.int32, (E + S + 1,)))
    assert np.array_equal(ids, ref["topk_ids"])
    assert np.array_equal(off, ref["expert_offsets"])


@pytest.mark.parametrize("name", SMALL)
def test_layer_parity_small(lib, name):
    wl = workload(name)
    s = wl.shape
    layer, out = run_layer(wl)
    ref = oracle_layer(wl)
    _check_layer_routing(layer, s, ref)
    tol = FP8_TOL if s.dtype == "fp8" else BF16_TOL
    rel = check_close(to_np(out), ref["out"], tol)
    assert layer.status() == 0
    print(f"{name}: max|gpu-oracle|/rms = {rel:.2e}")


@pytest.mark.parametrize("name", FULL)
def test_layer_parity_full_size(lib, name):
    wl = workload(name)
    s = wl.shape
    layer, out = run_layer(wl)
    rng = np.random.default_rng(1234)
    tokens = np.sort(rng.choice(s.tokens, SAMPLE[name], replace=False))
    ref = oracle_layer(wl, tokens=tokens)
    _check_layer_routing(layer, s, ref)
    rel = check_close(to_np(out)[tokens], ref["out"], FP8_TOL)
    assert layer.status() == 0
    print(f"{name}: max|gpu-oracle|/rms over {len(tokens)} tokens = {rel:.2e}")
    if s.balanced_perm:
        # the report (section "Load balancing across GPUs") brings the sets
        # within 5% of each other with the balanced grouping
        assert wl.imbalance <= wl.naive_imbalance
        assert wl.imbalance <= 1.05
        print(f"{name}: set imbalance balanced {wl.imbalance:.4f}, contiguous {wl.naive_imbalance:.4f}")


def test_layer_bf16_output_and_partial_batch(lib):
    wl = workload("r1_mini")
    s = wl.shape
    layer = wl.layer()
    _, out = run_layer(wl, out_bf16=True, layer=layer)
    ref = oracle_layer(wl)
    check_close(to_np(out.float()), ref["out"], FP8_TOL, bf16_out=True)
    # T below max_tokens reuses the same workspace
    T = 20
    _, out2 = run_layer(wl, T=T, layer=layer)
    ref20 = olayer.layer_forward(s.with_tokens(T), {**wl.np, "x_bits": wl.np["x_bits"][:T]})
    check_close(to_np(out2)[:T], ref20["out"], FP8_TOL)


def test_layer_single_token_and_empty(lib):
    wl = workload("r1_mini", seed=2, T=1)
    _, out = run_layer(wl)
    check_close(to_np(out), oracle_layer(wl)["out"], FP8_TOL)
    layer = wl.layer()
    out = torch.full((1, wl.shape.hidden), 5.0, device="cuda")
    layer.forward(wl.dev["x"], out, T=0)
    torch.cuda.synchronize()
    assert torch.all(out == 5.0) and layer.status() == 0


def test_layer_all_tokens_on_few_experts(lib):
    # a large bias on experts 0..7 sends every token to them (several N tiles
    # per expert, a ragged last tile); the other experts receive no rows
    shape = synth.CONFIGS["r1_mini"].with_tokens(130)
    wl = Workload(shape, seed=4)
    wl.dev["e_bias"] = wl.dev["e_bias"].clone()
    wl.dev["e_bias"][:8] += 10.0
    wl._np = None
    layer, out = run_layer(wl)
    ref = oracle_layer(wl)
    assert set(np.unique(ref["topk_ids"]).tolist()) == set(range(8))
    _check_layer_routing(layer, shape, ref)
    check_close(to_np(out), ref["out"], FP8_TOL)


@pytest.mark.parametrize("name,T", [("r1_mini", None), ("r1_mini_i512", None),
                                    ("r1_mini", 130)])   # 130 tokens: the wide-batch path
def test_layer_deterministic_and_graph_capturable(lib, name, T):
    wl = workload(name, T=T)
    layer, out1 = run_layer(wl)
    _, out2 = run_layer(wl, layer=layer)
    assert torch.equal(out1, out2)
    out3 = torch.zeros_like(out1)
    x = wl.dev["x"]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(x, out3)                  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    out3.zero_()
    with torch.cuda.graph(graph):
        layer.forward(x, out3)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out1, out3)


@pytest.mark.parametrize("name,T", [("r1_mini_i512", None),   # FP8 one-kernel FFN
                                     ("bf16_mini", None),      # BF16 one-kernel FFN
                                     ("r1_mini", 96)])         # 26 rows per group: GEMM path
def test_layer_back_to_back_calls_bit_identical(lib, name, T):
    """Layer calls queued with no host synchronisation between them overlap
    through programmatic dependent launch and reuse one workspace; every call
    must give the same bits (no race in the persistent kernels' barriers,
    completion counters or workspace reuse)."""
    wl = workload(name, T=T)
    s = wl.shape
    layer = wl.layer()
    outs = [torch.full((s.tokens, s.hidden), float("nan"), device="cuda") for _ in range(12)]
    for o in outs:
        layer.forward(wl.dev["x"], o)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert not torch.isnan(outs[0]).any()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_stream_read_utility(lib):
    """The read-stream utility bench.py uses for the read-only HBM rate: a
    1 GiB pass ends with a clear status at a plausible rate (1 to 10 TB/s)."""
    nbytes = 1 << 30
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.stream_read(buf, nbytes, st)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    moe.stream_read(buf, nbytes, st)
    b.record()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    gbs = nbytes / (a.elapsed_time(b) * 1e-3) / 1e9
    assert 1000 < gbs < 10000, gbs


def test_bounded_wait_reports_timeout_and_context_survives(lib):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = moe.lib().moe_selftest_bounded_wait(st.data_ptr(), 2_000_000, res.data_ptr(),
                                             torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(res.item()) == 3 and int(st.item()) & moe.DEV_TIMEOUT
    # the context is still usable
    wl = workload("bf16_mini")
    _, out = run_layer(wl)
    check_close(to_np(out), oracle_layer(wl)["out"], BF16_TOL)


@pytest.mark.parametrize("fp8,inter,K,counts", [
    (True, 384, 1024, GEMM_ROWS), (True, 2048, 7168, [3, 0, 17, 40, 128, 1]),
    (True, 384, 1024, [127, 128, 129, 0, 255, 256, 300, 1, 520, 33]),
    (True, 2048, 7168, [150, 130, 120, 0, 140, 600, 7]),
    (True, 384, 1024, [0, 1, 15, 16, 17, 3, 9, 2, 0, 5, 31]),
    (True, 2048, 7168, [2, 0, 9, 1, 14, 3]),
    (False, 384, 512, GEMM_ROWS)])
def test_swiglu_epilogue_equals_gemm_then_silu_requant(lib, fp8, inter, K, counts):
    """The fused gate/up + SwiGLU kernels give the bits of the two-kernel path,
    for groups averaging 16 rows or more (the first four cases: the
    token-rows-on-M kernel, with ragged 128-row token tiles, empty groups and
    a group of 600 rows; the plain GEMM takes 64-row tiles there) and fewer
    (the next two: 32-row activation tiles)."""
    s = synth.CONFIGS["r1_mini" if fp8 else "bf16_mini"]
    cfg = moe.make_config(s)
    counts = np.array(counts)
    G = len(counts)
    off_np = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(off_np[-1])
    off = torch.as_tensor(off_np, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(9)
    a32 = torch.randn(rows, K, device="cuda", generator=g)
    w32 = torch.randn(G, 2 * inter, K, device="cuda", generator=g) * 0.05
    if fp8:
        a = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
        asc = torch.empty((rows, K // 128), device="cuda")
        cfg_q = moe.make_config(synth.MoEShape("q", rows, K, 128, 1, 0, 1, dtype="fp8"))
        moe.act_requant(cfg_q, moe.ACT_IDENTITY, rows, a32.to(torch.bfloat16), a, asc)
        w, wsc = synth.block_quantize_e4m3(w32)
        h_ref = torch.empty((rows, inter), dtype=torch.uint8, device="cuda")
        hs_ref = torch.empty((rows, inter // 128), device="cuda")
        h = torch.full_like(h_ref, 0x55)
        hs = torch.full_like(hs_ref, -1.0)
    else:
        a, asc = a32.to(torch.bfloat16), None
        w, wsc = w32.to(torch.bfloat16), None
        h_ref = torch.empty((rows, inter), dtype=torch.bfloat16, device="cuda")
        h = torch.zeros_like(h_ref)
        hs_ref = hs = None
    cfg_i = moe.make_config(dataclasses_replace(s, inter=inter, hidden=K))
    gu = torch.empty((rows, 2 * inter), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.grouped_gemm(cfg, G, 2 * inter, K, rows, a, asc, off, w, wsc, gu, moe.OUT_F32, st)
    moe.act_requant(cfg_i, moe.ACT_SILU_MUL, rows, gu, h_ref, hs_ref)
    moe.grouped_gemm_swiglu(cfg, G, inter, K, rows, a, asc, off, w, wsc, h, hs, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(h, h_ref)
    if fp8:
        assert torch.equal(hs, hs_ref)


def dataclasses_replace(shape, **kw):
    import dataclasses
    return dataclasses.replace(shape, **kw)


@pytest.mark.parametrize("name,T,window", [("r1_mini", 130, (0, moe.ALL_ROWS)),
                                           ("r1_mini", 130, (33, moe.ALL_ROWS)),
                                           ("r1_mini_zipf", None, (0, moe.ALL_ROWS)),
                                           ("r1_mini", 1, (0, moe.ALL_ROWS)),
                                           ("r1_prefill_t4096", None, (33, moe.ALL_ROWS))])
def test_swiglu_gather_equals_swiglu_on_dispatched_rows(lib, name, T, window):
    """The gate/up GEMM that gathers its rows from the token rows of x (TMA
    gather4) gives the bits of moe_grouped_gemm_swiglu on the rows the
    dispatch copies; the dispatch's copy window leaves the other groups' rows
    uncopied and its tables unchanged."""
    wl = workload(name, T=T)
    s = wl.shape
    T = s.tokens
    cfg = moe.make_config(s)
    G, H, I = s.groups, s.hidden, s.inter
    rows = T * (s.top_k + s.num_shared)
    layer = wl.layer()
    out = torch.empty((T, H), device="cuda")
    layer.forward(wl.dev["x"], out)   # routing, x quantisation and dispatch
    torch.cuda.synchronize()
    L, base = layer.layout, layer.ws.data_ptr()
    xq, xs = base + L.xq, base + L.xs
    ids = layer.view("topk_ids", torch.int32, (T, s.top_k))
    off_full = layer.view("expert_offsets", torch.int32, (G + 1,)).clone()
    src_full = layer.view("src_of_row", torch.int32, (rows,)).clone()
    # the dispatch again, copying every row, and with the layer's copy window
    perm = {}
    for cap in (moe.ALL_ROWS, 32):
        r = dict(off=torch.full((G + 1,), -5, dtype=torch.int32, device="cuda"),
                 src=torch.full((rows,), -5, dtype=torch.int32, device="cuda"),
                 ros=torch.full((T, s.top_k), -5, dtype=torch.int32, device="cuda"),
                 xp=torch.full((rows, H), 0x55, dtype=torch.uint8, device="cuda"),
                 xps=torch.full((rows, H // 128), -1.0, device="cuda"))
        nws = moe.permute_workspace_size(cfg, T)
        ws = torch.empty(max(nws, 1), dtype=torch.uint8, device="cuda")
        moe.permute(cfg, T, ids, xq, xs, r["off"], r["src"], r["ros"], r["xp"], r["xps"], ws, nws,
                    copy_max_group_rows=cap)
        perm[cap] = r
    torch.cuda.synchronize()
    a, b = perm[moe.ALL_ROWS], perm[32]
    for key in ("off", "src", "ros"):
        assert torch.equal(a[key], b[key])
    assert torch.equal(a["off"], off_full) and torch.equal(a["src"], src_full)
    offs = to_np(a["off"])
    counts = np.diff(offs)
    small = np.zeros(rows, bool)
    for g in np.nonzero(counts <= 32)[0]:
        small[offs[g]:offs[g + 1]] = True
    small_t = torch.as_tensor(small, device="cuda")
    assert torch.equal(b["xp"][small_t], a["xp"][small_t])
    assert torch.all(b["xp"][~small_t] == 0x55) and torch.all(b["xps"][~small_t] == -1.0)
    # gate/up + SwiGLU on the copied rows against the gathered ones
    w = layer._keep
    outs = []
    for gather in (False, True):
        h = torch.full((rows, I), 0x55, dtype=torch.uint8, device="cuda")
        hs = torch.full((rows, I // 128), -1.0, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        if gather:
            moe.grouped_gemm_swiglu_gather(cfg, G, I, H, rows, xq, xs, T, a["src"], a["off"],
                                           w["w13"], w["w13_s"], h, hs, st,
                                           w_layout=layer.expert_layout,
                                           min_group_rows=window[0], max_group_rows=window[1])
        else:
            moe.grouped_gemm_swiglu(cfg, G, I, H, rows, a["xp"], a["xps"], a["off"], w["w13"],
                                    w["w13_s"], h, hs, st, w_layout=layer.expert_layout,
                                    min_group_rows=window[0], max_group_rows=window[1])
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        outs.append((h, hs))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    if window[0] > 0:   # the window's groups only
        inside = torch.as_tensor(np.repeat(counts >= window[0], counts), device="cuda")
        assert torch.all(outs[1][0][~inside] == 0x55)


@pytest.mark.parametrize("name,T", [("r1_mini_zipf", None), ("r1_mini", 130), ("bf16_mini", None)])
def test_group_row_windows_partition_the_groups(lib, name, T):
    """The group row windows of the expert entry points: the one-kernel FFN on
    the groups of at most X rows, then the gate/up and down GEMMs on the
    others, give the bits of the FFN over every group; a windowed call leaves
    the other groups' rows as they were.  (130 tokens of r1_mini: the GEMMs
    take their token-rows-on-M kernels; the others their 32/64-row tiles.)"""
    wl = workload(name, T=T)
    layer = wl.layer()
    s = wl.shape
    out = torch.empty((s.tokens, s.hidden), device="cuda")
    layer.forward(wl.dev["x"], out)   # routing and dispatch into the workspace
    cfg, w, wlay = layer.cfg, layer._keep, layer.expert_layout
    G, H, I = s.groups, s.hidden, s.inter
    rows = s.tokens * (s.top_k + s.num_shared)
    L, base = layer.layout, layer.ws.data_ptr()
    fp8 = s.dtype == "fp8"
    xp, xps, off = base + L.xp, (base + L.xp_scales) if fp8 else None, base + L.expert_offsets
    # the dispatch again with every row copied (wide layer calls copy only the
    # groups the FFN reads and let the gate/up GEMM gather the others)
    nws = moe.permute_workspace_size(cfg, s.tokens)
    moe.permute(cfg, s.tokens, base + L.topk_ids, (base + L.xq) if fp8 else wl.dev["x"],
                (base + L.xs) if fp8 else None, off, base + L.src_of_row, base + L.row_of_slot,
                xp, xps, base + L.perm_scratch, nws)
    torch.cuda.synchronize()
    offs = to_np(layer.view("expert_offsets", torch.int32, (G + 1,)))
    counts = np.diff(offs)
    X = int(np.median(counts[counts > 0]))
    assert (counts > X).any() and ((counts > 0) & (counts <= X)).any()
    nb = moe.expert_ffn_sched_bytes(G, rows)
    small = np.zeros(rows, bool)
    for g in np.nonzero(counts <= X)[0]:
        small[offs[g]:offs[g + 1]] = True
    small_t = torch.as_tensor(small, device="cuda")

    def run_ffn(**kw):
        h = torch.zeros((rows, I), dtype=torch.uint8 if fp8 else torch.bfloat16, device="cuda")
        hs = torch.zeros((rows, I // 128), device="cuda") if fp8 else None
        y = torch.full((rows, H), float("nan"), device="cuda")
        sched = torch.zeros(nb // 4 + 1, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        moe.expert_ffn(cfg, G, rows, xp, xps, off, w["w13"], w.get("w13_s"), w["w2"],
                       w.get("w2_s"), h, hs, y, sched, nb, st, w_layout=wlay, **kw)
        return h, hs, y, st

    _, _, y_all, st0 = run_ffn()
    h, hs, y, st = run_ffn(max_group_rows=X)
    torch.cuda.synchronize()
    assert torch.isnan(y[~small_t]).all() and torch.equal(y[small_t], y_all[small_t])
    moe.grouped_gemm_swiglu(cfg, G, I, H, rows, xp, xps, off, w["w13"], w.get("w13_s"), h, hs, st,
                            w_layout=wlay, min_group_rows=X + 1)
    moe.grouped_gemm(cfg, G, H, I, rows, h, hs, off, w["w2"], w.get("w2_s"), y, moe.OUT_F32, st,
                     w_layout=wlay, min_group_rows=X + 1)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st0.item()) == 0
    assert torch.equal(y, y_all)


@pytest.mark.parametrize("name,T", [("r1_mini_i512", None), ("bf16_mini", None),
                                    ("r1_mini", None), ("r1_mini", 130)])
def test_bench_steps_equal_the_layer_call(lib, name, T):
    """bench.py times the layer as C-ABI steps; they compute the layer call's bits
    (130 tokens of r1_mini average 35 rows per group: the wide-batch path, the
    one-kernel FFN on the groups of at most 32 rows and the GEMMs on the rest)."""
    import bench
    wl = workload(name, T=T)
    layer = wl.layer()
    s = wl.shape
    ref = torch.full((s.tokens, s.hidden), float("nan"), device="cuda")
    layer.forward(wl.dev["x"], ref)
    out = torch.full_like(ref, float("nan"))
    stepper = bench.Stepper(layer, wl.dev["x"], out)
    assert stepper.wide == (T is not None)
    stepper.step(record="all")
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(out, ref)
    assert set(stepper.kernel_ms()) == set(stepper.NAMES)
