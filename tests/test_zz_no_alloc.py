"""moe_permute_static_scratch: the dispatch permutation for callers that cannot
allocate device memory (a plugin whose host framework owns every device
allocation, a runtime held to a fixed memory budget).  It must give the same
rows, tables and offsets as moe_permute with a caller workspace, call after
call, although every call reuses the one static scratch array.

Collected last on purpose (file name), so that a run stopping at its first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_expert_layer_07_gb300 as moe
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from moe_expert_layer_07_gb300 import _build
    _build.build()
    return moe.lib()


def _outputs(shape, T):
    k, E, S, H = shape.top_k, shape.num_experts, shape.num_shared, shape.hidden
    rows = T * (k + S)
    return dict(off=torch.full((E + S + 1,), -5, dtype=torch.int32, device="cuda"),
                src=torch.full((rows,), -5, dtype=torch.int32, device="cuda"),
                ros=torch.full((T, k), -5, dtype=torch.int32, device="cuda"),
                xp=torch.zeros((rows, H), dtype=torch.uint8, device="cuda"),
                xps=torch.zeros((rows, H // 128), device="cuda"),
                st=torch.zeros(1, dtype=torch.int32, device="cuda"))


# up to 1024 routed slots the dispatch counts and scans in one CTA; above it
# (129 and 1024 tokens at the R1 shape, and 21824, where the per-chunk counts,
# chunk bases and per-slot ranks fill the 1 MiB array exactly) it takes the
# multi-chunk kernels, whose scratch all lives in the static array
@pytest.mark.parametrize("name,T", [("r1_mini", 37), ("r1_decode_t128", 128),
                                    ("r1_decode_t128", 129), ("r1_decode_t128", 1024),
                                    ("r1_decode_t128", 21824)])
def test_static_scratch_permute_matches_workspace_permute(lib, name, T):
    shape = synth.CONFIGS[name]
    cfg = moe.make_config(shape, max_tokens=T)
    k, E, H = shape.top_k, shape.num_experts, shape.hidden
    if T > 1024:
        assert moe.permute_workspace_size(cfg, T) > moe.permute_workspace_size(cfg, 128)
    if T == 21824:
        assert moe.permute_workspace_size(cfg, T) == lib.moe_permute_static_scratch_capacity()
    for call in range(2):   # two calls in a row: the second reuses the scratch
        g = torch.Generator(device="cuda").manual_seed(100 + call)
        # k distinct experts per token, skewed towards low ids on the second call
        scores = torch.rand(T, E, device="cuda", generator=g)
        if call == 1:
            scores[:, : E // 8] += 0.5
        ids = scores.topk(k, dim=1).indices.to(torch.int32).contiguous()
        x = torch.randint(0, 255, (T, H), dtype=torch.uint8, device="cuda", generator=g)
        xs = torch.rand(T, H // 128, device="cuda", generator=g)

        ref = _outputs(shape, T)
        nws = moe.permute_workspace_size(cfg, T)
        ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
        moe.permute(cfg, T, ids, x, xs, ref["off"], ref["src"], ref["ros"], ref["xp"],
                    ref["xps"], ws, nws, ref["st"])

        got = _outputs(shape, T)
        moe.permute_static_scratch(cfg, T, ids, x, xs, got["off"], got["src"], got["ros"],
                                   got["xp"], got["xps"], got["st"])
        torch.cuda.synchronize()
        for key in ("off", "src", "ros", "xp", "xps", "st"):
            assert torch.equal(got[key], ref[key]), f"call {call}: {key} differs"
        assert int(got["st"].item()) == 0


def test_static_scratch_rejects_sizes_beyond_capacity(lib):
    shape = synth.CONFIGS["r1_decode_t128"]
    cap = lib.moe_permute_static_scratch_capacity()
    T = 21825   # one token beyond the capacity at the R1 shape
    cfg = moe.make_config(shape, max_tokens=T)
    assert moe.permute_workspace_size(cfg, T) > cap
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: rejected before any launch
    rc = lib.moe_permute_static_scratch(ctypes.byref(cfg), T, fake, fake, fake, fake, fake,
                                        fake, fake, fake, None, None)
    assert rc == -2   # MOE_ERR_UNSUPPORTED_SHAPE
    assert moe.permute_workspace_size(moe.make_config(shape, max_tokens=21824), 21824) <= cap
