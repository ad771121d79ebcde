"""The one-kernel expert FFN (gate/up + SwiGLU + FP8 requant + down) on the GPU.

It must give the bits of the two-kernel path (SwiGLU GEMM, then the down
GEMM), whose parity with the oracle the layer tests establish; the layer
tests on r1_mini_i512 and the full-size R1 decode layer run it against the
oracle directly.
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


def _cfg(H, I):
    return moe.make_config(synth.MoEShape("ffn", 1, H, I, 32, 1, 8, num_groups=8,
                                          topk_groups=4, group_topn=2, scoring="sigmoid",
                                          dtype="fp8"))


def _problem(H, I, counts, seed):
    counts = np.asarray(counts)
    G = len(counts)
    off_np = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(off_np[-1])
    g = torch.Generator(device="cuda").manual_seed(seed)
    a32 = torch.randn(max(rows, 1), H, device="cuda", generator=g)
    a = torch.empty((max(rows, 1), H), dtype=torch.uint8, device="cuda")
    asc = torch.empty((max(rows, 1), H // 128), device="cuda")
    cfg_q = moe.make_config(synth.MoEShape("q", max(rows, 1), H, 128, 1, 0, 1, dtype="fp8"))
    moe.act_requant(cfg_q, moe.ACT_IDENTITY, max(rows, 1), a32.to(torch.bfloat16), a, asc)
    w13, w13s = synth.block_quantize_e4m3(
        torch.randn(G, 2 * I, H, device="cuda", generator=g) * 0.05)
    w2, w2s = synth.block_quantize_e4m3(torch.randn(G, H, I, device="cuda", generator=g) * 0.05)
    off = torch.as_tensor(off_np, device="cuda")
    return G, rows, a, asc, off, w13, w13s, w2, w2s


def _two_kernels(cfg, G, rows, H, I, a, asc, off, w13, w13s, w2, w2s):
    h = torch.empty((rows, I), dtype=torch.uint8, device="cuda")
    hs = torch.empty((rows, I // 128), device="cuda")
    y = torch.empty((rows, H), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.grouped_gemm_swiglu(cfg, G, I, H, rows, a, asc, off, w13, w13s, h, hs, st)
    moe.grouped_gemm(cfg, G, H, I, rows, h, hs, off, w2, w2s, y, moe.OUT_F32, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return h, hs, y


def _fused(cfg, G, rows, H, I, a, asc, off, w13, w13s, w2, w2s, sched=None):
    h = torch.full((rows, I), 0x55, dtype=torch.uint8, device="cuda")
    hs = torch.full((rows, I // 128), -1.0, device="cuda")
    y = torch.full((rows, H), float("nan"), device="cuda")
    nbytes = moe.expert_ffn_sched_bytes(G, rows)
    if sched is None:
        sched = torch.full((nbytes // 4,), 12345, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.expert_ffn(cfg, G, rows, a, asc, off, w13, w13s, w2, w2s, h, hs, y, sched, nbytes, st)
    torch.cuda.synchronize()
    return h, hs, y, int(st.item()), sched


CASES = [
    # hidden, inter, rows per group: empty groups, groups spanning several
    # 32-row activation tiles, ragged tails
    (1024, 512, [3, 0, 17, 40, 128, 1]),
    (384, 256, [5]),                                   # one group, one down step
    (7168, 2048, [3, 0, 17, 40, 128, 1]),             # R1 sizes
    (2048, 768, [0, 0, 33, 0, 64, 0, 1, 31, 32]),     # exact tile edges
    (1024, 384, [3, 0, 17, 40, 128, 1]),              # 3 K blocks of W2: a 1-block last stage
]


@pytest.mark.parametrize("H,I,counts", CASES)
def test_expert_ffn_equals_two_kernel_path(lib, H, I, counts):
    cfg = _cfg(H, I)
    p = _problem(H, I, counts, seed=3)
    G, rows = p[0], p[1]
    h_ref, hs_ref, y_ref = _two_kernels(cfg, G, rows, H, I, *p[2:])
    h, hs, y, st, sched = _fused(cfg, G, rows, H, I, *p[2:])
    assert st == 0
    assert torch.equal(h, h_ref)
    assert torch.equal(hs, hs_ref)
    assert torch.equal(y, y_ref)
    # every gate/up tile of every activation tile reported completion once
    nt = int(sum((c + 31) // 32 for c in counts))
    done = sched[1:1 + nt].cpu().numpy()
    assert np.all(done == I // 128)
    units = (I // 128 + H // 128) * nt
    assert int(sched[0].item()) >= units   # claims past the end stop each CTA


def test_expert_ffn_decode_many_groups_repeatable(lib):
    """257 groups of decode-sized rows (as the 128-token R1 layer): the same
    bits twice over, whichever CTA claims which unit."""
    H, I = 1024, 512
    rng = np.random.default_rng(5)
    counts = np.bincount(rng.integers(0, 256, size=128 * 8), minlength=256).tolist() + [128]
    cfg = _cfg(H, I)
    p = _problem(H, I, counts, seed=4)
    G, rows = p[0], p[1]
    h_ref, hs_ref, y_ref = _two_kernels(cfg, G, rows, H, I, *p[2:])
    for _ in range(2):
        h, hs, y, st, _ = _fused(cfg, G, rows, H, I, *p[2:])
        assert st == 0
        assert torch.equal(h, h_ref) and torch.equal(hs, hs_ref) and torch.equal(y, y_ref)


def test_expert_ffn_no_rows_and_bad_offsets(lib):
    H, I = 1024, 512
    cfg = _cfg(H, I)
    G, rows, a, asc, off, w13, w13s, w2, w2s = _problem(H, I, [0, 0, 0], seed=1)
    assert rows == 0
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # rows = 0: nothing to do, nothing launched (no output buffers needed)
    moe.expert_ffn(cfg, G, 0, a, asc, off, w13, w13s, w2, w2s, None, None, None, None, 0, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # offsets that leave [0, rows]: reported, nothing written, no hang
    p = _problem(H, I, [4, 4], seed=2)
    G, rows = p[0], p[1]
    bad = torch.as_tensor(np.array([0, 6, 4], np.int32), device="cuda")
    args = list(p[2:])
    args[2] = bad
    h, hs, y, stv, _ = _fused(cfg, G, rows, H, I, *args)
    assert stv & moe.DEV_BAD_OFFSETS
    assert bool(torch.isnan(y).all())


def test_flag_wait_gives_up_and_context_survives(lib):
    """A down unit whose h rows nobody writes: the bounded wait expires, the
    device status says so, and the next launches run normally."""
    n = moe.lib().moe_selftest_ffn_flag_timeout_scratch_bytes()
    scratch = torch.empty(n, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = moe.lib().moe_selftest_ffn_flag_timeout(scratch.data_ptr(), n, st.data_ptr(),
                                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(st.item()) & moe.DEV_TIMEOUT
    H, I, counts = 1024, 512, [3, 0, 17, 40, 128, 1]
    cfg = _cfg(H, I)
    p = _problem(H, I, counts, seed=3)
    G, rows = p[0], p[1]
    h_ref, hs_ref, y_ref = _two_kernels(cfg, G, rows, H, I, *p[2:])
    h, hs, y, stv, _ = _fused(cfg, G, rows, H, I, *p[2:])
    assert stv == 0 and torch.equal(y, y_ref) and torch.equal(h, h_ref)


def _bf16_problem(H, I, counts, seed):
    counts = np.asarray(counts)
    G = len(counts)
    off = torch.as_tensor(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32), device="cuda")
    rows = int(counts.sum())
    g = torch.Generator(device="cuda").manual_seed(seed)
    a = torch.randn(rows, H, device="cuda", generator=g).to(torch.bfloat16)
    w13 = (torch.randn(G, 2 * I, H, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    w2 = (torch.randn(G, H, I, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    return G, rows, a, off, w13, w2


@pytest.mark.parametrize("H,I,counts", [(1024, 512, [3, 0, 17, 40, 128, 1]),
                                        (2048, 1408, [24, 0, 256, 5, 33]),   # V2-Lite sizes
                                        (512, 384, [7])])
def test_expert_ffn_bf16_equals_two_kernel_path(lib, H, I, counts):
    """Both BF16 configurations of the kernel: the first and last cases have
    few enough gate/up units for one CTA per SM with the five-stage ring,
    the V2-Lite-sized one takes two CTAs per SM with two stages."""
    cfg = moe.make_config(synth.MoEShape("ffn16", 1, H, I, 32, 1, 8, scoring="softmax",
                                         dtype="bf16"))
    G, rows, a, off, w13, w2 = _bf16_problem(H, I, counts, 12)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    h_ref = torch.empty((rows, I), dtype=torch.bfloat16, device="cuda")
    y_ref = torch.empty((rows, H), device="cuda")
    moe.grouped_gemm_swiglu(cfg, G, I, H, rows, a, None, off, w13, None, h_ref, None, st)
    moe.grouped_gemm(cfg, G, H, I, rows, h_ref, None, off, w2, None, y_ref, moe.OUT_F32, st)
    h = torch.zeros_like(h_ref)
    y = torch.full_like(y_ref, float("nan"))
    nbytes = moe.expert_ffn_sched_bytes(G, rows)
    sched = torch.full((nbytes // 4,), 77, dtype=torch.int32, device="cuda")
    moe.expert_ffn(cfg, G, rows, a, None, off, w13, None, w2, None, h, None, y, sched, nbytes, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(h.view(torch.int16), h_ref.view(torch.int16))
    assert torch.equal(y, y_ref)
