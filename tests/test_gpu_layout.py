"""Expert weights packed into 128 x 128-byte tiles (MOE_LAYOUT_TILES).

The packing is a pure permutation of bytes (checked against a torch view),
and every kernel that reads expert weights gives the same bits from the
packed copy as from the row-major one.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import moe_expert_layer_07_gb300 as moe
import synth

from _gpu_common import build_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    return build_library()


def _cfg(dtype, H=1024, I=512):
    return moe.make_config(synth.MoEShape("lay", 1, H, I, 32, 1, 8, num_groups=8, topk_groups=4,
                                          group_topn=2, scoring="sigmoid", dtype=dtype))


def _tiles_reference(w, fp8):
    """Tiles of 128 rows x 128 bytes, tile-major, and within a tile the
    16-byte chunk c of row r at chunk position c ^ (r mod 8)."""
    G, N, K = w.shape
    kt = 128 if fp8 else 64
    t = w.view(G, N // 128, 128, K // kt, kt).permute(0, 1, 3, 2, 4).contiguous()
    t = t.view(G, N // 128, K // kt, 128, 8, kt // 8)          # [..., row, chunk, element]
    r = torch.arange(128, device=w.device)[:, None]
    c = torch.arange(8, device=w.device)[None, :]
    t = t[:, :, :, r, c ^ (r % 8), :]                          # position c holds chunk c ^ (r mod 8)
    return t.contiguous().view(G, N, K)


@pytest.mark.parametrize("fp8,G,N,K", [(True, 3, 256, 384), (True, 1, 128, 128),
                                       (False, 2, 384, 320), (False, 5, 128, 64)])
def test_pack_is_the_tile_permutation(lib, fp8, G, N, K):
    g = torch.Generator(device="cuda").manual_seed(1)
    if fp8:
        w = torch.randint(0, 256, (G, N, K), dtype=torch.uint8, device="cuda", generator=g)
    else:
        w = torch.randn(G, N, K, device="cuda", generator=g).to(torch.bfloat16)
    packed = moe.pack_expert_weights(_cfg("fp8" if fp8 else "bf16"), w)
    torch.cuda.synchronize()
    ref = _tiles_reference(w, fp8)
    assert torch.equal(packed.view(torch.uint8) if fp8 else packed.view(torch.int16),
                       ref.view(torch.uint8) if fp8 else ref.view(torch.int16))


def _quantised_problem(H, N, counts, seed):
    counts = np.asarray(counts)
    off = torch.as_tensor(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32), device="cuda")
    rows = int(counts.sum())
    g = torch.Generator(device="cuda").manual_seed(seed)
    a32 = torch.randn(rows, H, device="cuda", generator=g)
    a = torch.empty((rows, H), dtype=torch.uint8, device="cuda")
    asc = torch.empty((rows, H // 128), device="cuda")
    moe.act_requant(moe.make_config(synth.MoEShape("q", rows, H, 128, 1, 0, 1, dtype="fp8")),
                    moe.ACT_IDENTITY, rows, a32.to(torch.bfloat16), a, asc)
    w, ws = synth.block_quantize_e4m3(
        torch.randn(len(counts), N, H, device="cuda", generator=g) * 0.05)
    return off, rows, a, asc, w, ws


@pytest.mark.parametrize("counts", [[3, 0, 17, 40, 128, 1], [0, 300, 129, 64, 2]])
def test_fp8_gemms_same_bits_from_tiles(lib, counts):
    H, I = 1024, 512
    cfg = _cfg("fp8", H, I)
    G = len(counts)
    off, rows, a, asc, w13, w13s = _quantised_problem(H, 2 * I, counts, 5)
    t13 = moe.pack_expert_weights(cfg, w13)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for w, lay in ((w13, moe.LAYOUT_ROWS), (t13, moe.LAYOUT_TILES)):
        c = torch.full((rows, 2 * I), float("nan"), device="cuda")
        moe.grouped_gemm(cfg, G, 2 * I, H, rows, a, asc, off, w, w13s, c, moe.OUT_F32, st,
                         w_layout=lay)
        h = torch.zeros((rows, I), dtype=torch.uint8, device="cuda")
        hs = torch.zeros((rows, I // 128), device="cuda")
        moe.grouped_gemm_swiglu(cfg, G, I, H, rows, a, asc, off, w, w13s, h, hs, st, w_layout=lay)
        outs.append((c, h, hs))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for x, y in zip(outs[0], outs[1]):
        assert torch.equal(x, y)


def test_expert_ffn_same_bits_from_tiles(lib):
    H, I = 1024, 512
    cfg = _cfg("fp8", H, I)
    counts = [3, 0, 17, 40, 128, 1]
    G = len(counts)
    off, rows, a, asc, w13, w13s = _quantised_problem(H, 2 * I, counts, 6)
    w2, w2s = synth.block_quantize_e4m3(
        torch.randn(G, H, I, device="cuda", generator=torch.Generator(device="cuda").manual_seed(8))
        * 0.05)
    t13, t2 = moe.pack_expert_weights(cfg, w13), moe.pack_expert_weights(cfg, w2)
    nbytes = moe.expert_ffn_sched_bytes(G, rows)
    sched = torch.zeros(nbytes // 4, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ys = []
    for (x13, x2, lay) in ((w13, w2, moe.LAYOUT_ROWS), (t13, t2, moe.LAYOUT_TILES)):
        h = torch.zeros((rows, I), dtype=torch.uint8, device="cuda")
        hs = torch.zeros((rows, I // 128), device="cuda")
        y = torch.full((rows, H), float("nan"), device="cuda")
        moe.expert_ffn(cfg, G, rows, a, asc, off, x13, w13s, x2, w2s, h, hs, y, sched, nbytes, st,
                       w_layout=lay)
        ys.append(y)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(ys[0], ys[1])


def test_bf16_gemm_same_bits_from_tiles(lib):
    H, N = 512, 384
    cfg = _cfg("bf16", H, 384)
    counts = [5, 0, 70, 33]
    G = len(counts)
    off = torch.as_tensor(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32), device="cuda")
    rows = int(sum(counts))
    g = torch.Generator(device="cuda").manual_seed(9)
    a = torch.randn(rows, H, device="cuda", generator=g).to(torch.bfloat16)
    w = (torch.randn(G, N, H, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    t = moe.pack_expert_weights(cfg, w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cs = []
    for ww, lay in ((w, moe.LAYOUT_ROWS), (t, moe.LAYOUT_TILES)):
        c = torch.full((rows, N), float("nan"), device="cuda")
        moe.grouped_gemm(cfg, G, N, H, rows, a, None, off, ww, None, c, moe.OUT_F32, st,
                         w_layout=lay)
        cs.append(c)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and torch.equal(cs[0], cs[1])


@pytest.mark.parametrize("name", ["r1_mini_i512", "bf16_mini", "r1_mini"])
def test_layer_same_bits_packed_or_not(lib, name):
    shape = synth.CONFIGS[name]
    inp = synth.make_inputs(shape, seed=0, device="cuda")
    outs = []
    for pack in (False, True):
        layer = moe.MoELayer(shape, inp, pack_weights=pack)
        assert layer.expert_layout == (moe.LAYOUT_TILES if pack else moe.LAYOUT_ROWS)
        out = torch.full((shape.tokens, shape.hidden), float("nan"), device="cuda")
        layer.forward(inp["x"], out)
        torch.cuda.synchronize()
        assert layer.status() == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
