"""Pins of the oracle's expert FFN, grouped GEMM, combine and whole layer.

The one-expert layer is a dense SwiGLU FFN, recomputed here with torch's own
fp64 matmul, silu and casts; the permuted layer equals the unpermuted one
bit for bit; linearity and the shared-expert-only case are closed forms.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import layer, permute, quant


def _cfg(**kw):
    base = dict(name="t", tokens=13, hidden=256, inter=128, num_experts=1, num_shared=0,
                top_k=1, scoring="softmax", norm_topk=True)
    base.update(kw)
    return synth.MoEShape(**base)


def _torch_dense_ffn(x_bf16, w13, w2, fp8, w13_s=None, w2_s=None):
    """Dense SwiGLU with the layer's quantisation points, in torch fp64."""
    I = w2.shape[1]
    if fp8:
        def deq(q, s, n, k):
            v = q.view(torch.float8_e4m3fn).to(torch.float64)
            return v * s.to(torch.float64).repeat_interleave(128, 0).repeat_interleave(128, 1)[:n, :k]
        x32 = x_bf16.to(torch.float32)
        T, H = x32.shape
        g = x32.view(T, H // 128, 128)
        sx = g.abs().amax(dim=2) / 448.0
        xq = (g / sx[..., None]).to(torch.float8_e4m3fn).to(torch.float64)
        xd = (xq * sx[..., None].to(torch.float64)).view(T, H)
        W13 = deq(w13, w13_s, 2 * I, H)
        W2 = deq(w2, w2_s, H, I)
        gu = xd @ W13.T
        h = (torch.nn.functional.silu(gu[:, :I]) * gu[:, I:]).to(torch.float32)
        hg = h.view(T, I // 128, 128)
        sh = hg.abs().amax(dim=2) / 448.0
        hq = (hg / sh[..., None]).to(torch.float8_e4m3fn).to(torch.float64)
        hd = (hq * sh[..., None].to(torch.float64)).view(T, I)
        y = hd @ W2.T
    else:
        xd = x_bf16.to(torch.float64)
        gu = xd @ w13.to(torch.float64).T
        h = (torch.nn.functional.silu(gu[:, :I]) * gu[:, I:]).to(torch.bfloat16).to(torch.float64)
        y = h @ w2.to(torch.float64).T
    return y.numpy()


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_one_expert_layer_is_dense_ffn(oracle_lib, dtype):
    cfg = _cfg(dtype=dtype)
    inp = synth.make_inputs(cfg, seed=3)
    res = layer.layer_forward(cfg, synth.to_numpy(inp))
    assert np.all(res["topk_ids"] == 0) and np.all(res["topk_w"] == 1.0)
    ref = _torch_dense_ffn(inp["x"], inp["w13"][0], inp["w2"][0], dtype == "fp8",
                           inp["w13_s"][0] if dtype == "fp8" else None,
                           inp["w2_s"][0] if dtype == "fp8" else None)
    # what is left is fp64 summation order (and, in principle, a rounding
    # decision of h flipped by it)
    err = np.abs(res["out"] - ref)
    rms = np.sqrt(np.mean(ref ** 2))
    assert err.max() <= 1e-9 * rms


@pytest.mark.parametrize("name", ["r1_mini", "bf16_mini"])
def test_permuted_layer_equals_unpermuted(oracle_lib, name):
    cfg = synth.CONFIGS[name].with_tokens(9)
    inp = synth.make_inputs(cfg, seed=1)
    base = layer.layer_forward(cfg, synth.to_numpy(inp))
    rng = np.random.default_rng(0)
    phys2log = rng.permutation(cfg.num_experts)
    log2phys = np.argsort(phys2log).astype(np.int32)
    moved = synth.relayout_experts(inp, cfg, phys2log)
    perm = layer.layer_forward(cfg, synth.to_numpy(moved, log2phys))
    assert np.array_equal(perm["topk_ids"], log2phys[base["topk_ids"]])
    assert np.array_equal(perm["topk_w"], base["topk_w"])
    assert np.array_equal(perm["out"], base["out"])


def test_shared_experts_only_and_linearity(oracle_lib):
    cfg = synth.CONFIGS["bf16_mini"].with_tokens(6)
    inp = synth.make_inputs(cfg, seed=2)
    E = cfg.num_experts
    zeroed = dict(inp)
    zeroed["w2"] = inp["w2"].clone()
    zeroed["w2"][:E] = 0
    res = layer.layer_forward(cfg, synth.to_numpy(zeroed))
    shared = sum(_torch_dense_ffn(inp["x"], inp["w13"][E + s], inp["w2"][E + s], False)
                 for s in range(cfg.num_shared))
    rms = np.sqrt(np.mean(shared ** 2))
    assert np.abs(res["out"] - shared).max() <= 1e-2 * rms
    # doubling every W2 doubles each expert output exactly
    doubled = dict(inp)
    doubled["w2"] = inp["w2"] * 2
    a = layer.layer_forward(cfg, synth.to_numpy(inp))["out"]
    b = layer.layer_forward(cfg, synth.to_numpy(doubled))["out"]
    assert np.array_equal(b, 2 * a)


def test_layer_output_on_token_subset_matches_full(oracle_lib):
    cfg = synth.CONFIGS["r1_mini"]
    inp = synth.to_numpy(synth.make_inputs(cfg, seed=4))
    full = layer.layer_forward(cfg, inp)
    sub = layer.layer_forward(cfg, inp, tokens=[0, 17, 36])
    assert np.allclose(sub["out"], full["out"][[0, 17, 36]], rtol=0, atol=1e-12)


def test_grouped_gemm_against_torch(oracle_lib):
    rng = np.random.default_rng(5)
    cfg = _cfg(dtype="fp8")
    G, N, K = 3, 256, 384
    offsets = np.array([0, 5, 5, 12], np.int32)
    a = rng.standard_normal((14, K)).astype(np.float32)
    aq, asc = quant.quant_groups_fp8(a)
    w = torch.from_numpy(rng.standard_normal((G, N, K)).astype(np.float32) * 0.02)
    wq, ws = synth.block_quantize_e4m3(w)
    c = layer.grouped_gemm(cfg, offsets, aq, wq.numpy(), asc, ws.numpy())
    ad = quant.dequant_groups_fp8(aq, asc)
    for g in range(G):
        wd = wq[g].view(torch.float8_e4m3fn).to(torch.float64) * \
            ws[g].to(torch.float64).repeat_interleave(128, 0).repeat_interleave(128, 1)
        r0, r1 = offsets[g], offsets[g + 1]
        ref = torch.from_numpy(ad[r0:r1]) @ wd.T
        assert np.allclose(c[r0:r1], ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.all(c[12:] == 0)


def test_combine_closed_form():
    T, k, E, S, H = 4, 3, 5, 2, 16
    rng = np.random.default_rng(6)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    off, src, ros = permute.permute(ids, E, S)
    rows = off[-1]
    # row r holds the constant (r + 1): combine is then a weighted row-index sum
    y = np.repeat((np.arange(rows) + 1.0)[:, None], H, axis=1)
    w = rng.random((T, k)).astype(np.float32)
    out = layer.combine(y, ros, w, off, E, S)
    for t in range(T):
        want = sum(off[E + s] + t + 1.0 for s in range(S)) + \
            sum(float(w[t, j]) * (ros[t, j] + 1.0) for j in range(k))
        assert np.allclose(out[t], want, rtol=1e-15)
