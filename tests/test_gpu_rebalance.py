"""Continuous load balancing on the GPU: on-device row counting against the
oracle's histogram, the block re-layout against a direct gather, and a
re-balance that moves experts without changing the layer's output."""
import numpy as np
import pytest
import torch

import moe_expert_layer_07_gb300 as moe
import synth
from oracle import routing as orouting

from _gpu_common import build_library, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    return build_library()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _oracle_phys_ids(shape, inp, x, log2phys=None):
    off = None if inp["logit_offset"] is None else inp["logit_offset"].cpu().numpy()
    bias = None if inp["e_bias"] is None else inp["e_bias"].cpu().numpy()
    l = orouting.gate_logits(_bits(x), _bits(inp["wg"]), off)
    phys, _, logical = orouting.route(l, shape, bias, log2phys)
    return phys, logical


def test_count_rows_accumulates_the_histogram(lib):
    shape = synth.CONFIGS["r1_mini_zipf"]
    inp = synth.make_inputs(shape, seed=1, device="cuda")
    layer = moe.MoELayer(shape, inp)
    reb = moe.ExpertRebalancer(layer, shape.num_sets)
    want = np.zeros(shape.num_experts, np.int64)
    out = torch.empty((shape.tokens, shape.hidden), device="cuda")
    for b in range(3):
        x = synth.make_inputs(shape, seed=10 + b, device="cuda")["x"]
        layer.forward(x, out)
        reb.observe()
        phys, _ = _oracle_phys_ids(shape, inp, x)
        want += np.bincount(phys.reshape(-1), minlength=shape.num_experts)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(reb.counts), want)
    assert np.array_equal(reb.logical_counts(), want)     # identity permutation so far


def test_relayout_is_a_block_gather(lib):
    g = torch.Generator(device="cuda").manual_seed(5)
    G, block = 9, 4096 + 48
    src = torch.randint(0, 256, (G, block), dtype=torch.uint8, device="cuda", generator=g)
    slot = torch.randperm(G, device="cuda", generator=g).to(torch.int32)
    dst = torch.zeros_like(src)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.relayout_experts(src, dst, slot, G, block, st)
    torch.cuda.synchronize()
    assert torch.equal(dst, src[slot.long()]) and int(st.item()) == 0
    bad = slot.clone()
    bad[3] = G
    dst2 = torch.zeros_like(src)
    moe.relayout_experts(src, dst2, bad, G, block, st)
    torch.cuda.synchronize()
    assert int(st.item()) & moe.DEV_BAD_EXPERT_ID
    assert torch.all(dst2[3] == 0)
    assert torch.equal(dst2[[0, 1, 2, 4]], src[bad[[0, 1, 2, 4]].long()])


@pytest.mark.parametrize("name", ["r1_mini_zipf", "r1_zipf_t1024"])
def test_rebalance_moves_experts_without_changing_the_output(lib, name):
    shape = synth.CONFIGS[name]
    inp = synth.make_inputs(shape, seed=0, device="cuda")
    layer = moe.MoELayer(shape, inp)
    reb = moe.ExpertRebalancer(layer, shape.num_sets)
    x = inp["x"]
    out_a = torch.empty((shape.tokens, shape.hidden), device="cuda")
    layer.forward(x, out_a)
    reb.observe()
    before, after = reb.rebalance()
    assert after <= before
    out_b = torch.empty_like(out_a)
    layer.forward(x, out_b)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(out_a, out_b)
    ids = to_np(layer.view("topk_ids", torch.int32, (shape.tokens, shape.top_k)))
    _, logical = _oracle_phys_ids(shape, inp, x)
    assert np.array_equal(ids, reb.log2phys[logical])
    assert np.array_equal(np.sort(reb.log2phys), np.arange(shape.num_experts))
    assert int(reb.counts.sum().item()) == 0          # the window restarts
    print(f"{name}: set imbalance {before:.4f} -> {after:.4f}")


def test_coactivation_counts_equal_the_oracle(lib):
    from oracle import affinity as oaff
    shape = synth.CONFIGS["r1_mini_zipf"]
    inp = synth.make_inputs(shape, seed=2, device="cuda")
    rng = np.random.default_rng(4)
    p2l = rng.permutation(shape.num_experts)
    l2p = np.argsort(p2l).astype(np.int32)
    moved = synth.relayout_experts(inp, shape, p2l)
    layer = moe.MoELayer(shape, moved, log2phys=l2p)
    reb = moe.ExpertRebalancer(layer, shape.num_sets, affinity_slack=0.05)
    out = torch.empty((shape.tokens, shape.hidden), device="cuda")
    want = np.zeros((shape.num_experts, shape.num_experts), np.int64)
    for b in range(2):
        x = synth.make_inputs(shape, seed=20 + b, device="cuda")["x"]
        layer.forward(x, out)
        reb.observe()
        _, logical = _oracle_phys_ids(shape, inp, x)
        want += oaff.coactivation_n(logical, shape.num_experts)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(reb.coact), want)
    before, after = reb.rebalance()
    out_b = torch.empty_like(out)
    layer.forward(x, out_b)
    torch.cuda.synchronize()
    assert torch.equal(out, out_b) and layer.status() == 0
    assert 0.0 <= reb.last_intra_fraction <= 1.0
