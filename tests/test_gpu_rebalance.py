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


def test_periodic_rebalance_retightens_a_drifting_stream(lib):
    """A stream whose expert popularity drifts (a new seeded Zipf order every
    three batches): the every-3-batches policy re-balances at the end of each
    phase.  Each re-balance brings the phase's counts from their imbalance
    under the old permutation down to the balanced partition's, and the layer
    gives the same bits for the same batch before and after each move."""
    shape = synth.CONFIGS["r1_mini_zipf"]
    inp = synth.make_inputs(shape, seed=0, device="cuda")
    layer = moe.MoELayer(shape, inp)
    reb = moe.ExpertRebalancer(layer, shape.num_sets, every=3)
    offset = layer._keep["logit_offset"]          # the prior the layer routes with
    T, H = shape.tokens, shape.hidden
    out = torch.empty((T, H), device="cuda")
    g = torch.Generator(device="cuda").manual_seed(77)
    befores, afters = [], []
    for phase in range(3):
        offset.copy_(synth.zipf_logit_offset(shape, 100 + phase, "cuda"))
        for b in range(3):
            x = torch.randn((T, H), device="cuda", generator=g).to(torch.bfloat16)
            layer.forward(x, out)
            counted = reb.logical_counts() + np.bincount(
                _oracle_phys_ids(shape, {**inp, "logit_offset": offset}, x)[1].reshape(-1),
                minlength=shape.num_experts)
            prev_l2p = reb.log2phys.copy()
            res = reb.step()
            assert (res is not None) == (b == 2)
        before, after = res
        # the policy's figures are those of the phase's counts
        assert before == pytest.approx(moe.set_imbalance(counted, prev_l2p, shape.num_sets))
        assert after == pytest.approx(moe.set_imbalance(counted, reb.log2phys, shape.num_sets))
        _, _, best = moe.balance_permutation(counted, shape.num_sets)
        assert after == pytest.approx(best) and after <= before
        ref = out.clone()
        layer.forward(x, out)                       # the same batch after the move
        torch.cuda.synchronize()
        assert torch.equal(out, ref) and layer.status() == 0
        befores.append(before)
        afters.append(after)
    assert [h[0] for h in reb.history] == [3, 3, 3]
    # after the first phase the stream drifts: the old placement no longer fits
    assert all(b > a for b, a in zip(befores[1:], afters[1:]))
    print(f"set imbalance per phase, before -> after: "
          f"{[(round(b, 3), round(a, 3)) for b, a in zip(befores, afters)]}")
