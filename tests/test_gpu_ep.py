"""The expert-parallel step with the CUDA kernels: P ranks of the product's
ep_forward/GpuRank (their own routed experts, the shared experts, the
global gate) run as host threads of one process on one GPU.  Their
exchanges are host-side copies between launches, after each rank's stream
has drained, so no kernel ever waits on another rank's kernel.

Every rank's output must equal the single-GPU layer (moe_layer_forward) on
the same tokens bit for bit: a row's FFN result does not depend on which
rows share its tile, whether the rank's expert groups take the one-kernel
FFN (few rows per group) or the wide GEMMs (37 tokens against 200 below),
and in a BF16 layer with two shared experts.
"""
import threading

import numpy as np
import pytest
import torch

import moe_expert_layer_07_gb300 as moe
import synth
from moe_expert_layer_07_gb300.ep import EPPlan, Exchange, GpuRank, ep_forward, split_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from moe_expert_layer_07_gb300 import _build
    _build.build()
    return moe.lib()


class _Loopback:
    """The collectives of P in-process ranks: each rank posts its buffer, all
    meet at a barrier, each copies what it is owed, and all meet again."""

    def __init__(self, world):
        self.world = world
        self.bar = threading.Barrier(world, timeout=300)
        self.slots = [None] * world

    def rank(self, r):
        return _RankView(self, r)


class _RankView(Exchange):
    def __init__(self, lb, r):
        self.lb, self.r = lb, r

    def counts(self, send):
        lb, r = self.lb, self.r
        lb.slots[r] = np.asarray(send)
        lb.bar.wait()
        recv = np.stack([lb.slots[s][r] for s in range(lb.world)])
        lb.bar.wait()
        return recv

    def rows(self, out, inp, out_splits, in_splits):
        lb, r = self.lb, self.r
        torch.cuda.current_stream().synchronize()   # the rows to send are complete
        lb.slots[r] = (inp, list(in_splits))
        lb.bar.wait()
        o = 0
        for s in range(lb.world):
            src, sp = lb.slots[s]
            start, n = sum(sp[:r]), sp[r]
            assert n == out_splits[s]
            if n:
                out[o:o + n].copy_(src[start:start + n])
            o += n
        torch.cuda.current_stream().synchronize()   # copied before the sender moves on
        lb.bar.wait()


def _balanced(shape, inp):
    layer = moe.MoELayer(shape, inp)
    reb = moe.ExpertRebalancer(layer, 1)
    out = torch.empty((shape.tokens, shape.hidden), device="cuda")
    layer.forward(inp["x"], out)
    reb.observe()
    counts = reb.logical_counts()
    return counts


@pytest.mark.parametrize("name,T,world", [("r1_mini", 37, 2), ("r1_mini", 37, 4),
                                          ("r1_mini", 200, 2), ("bf16_mini", 29, 2)])
def test_expert_parallel_ranks_equal_the_single_gpu_layer(lib, name, T, world):
    shape = synth.CONFIGS[name].with_tokens(T)
    inp = synth.make_inputs(shape, seed=5, device="cuda")
    # one balanced expert set per rank, weights re-laid in that order
    l2p, p2l, _ = moe.balance_permutation(_balanced(shape, inp), world)
    inp = synth.relayout_experts(inp, shape, p2l)
    ref_layer = moe.MoELayer(shape, inp, log2phys=l2p)
    rng = np.random.default_rng(T + world)
    cuts = np.sort(rng.choice(np.arange(1, T), world - 1, replace=False))
    edges = np.concatenate([[0], cuts, [T]])
    ranges = list(zip(edges[:-1].tolist(), edges[1:].tolist()))
    x = inp["x"]
    lb = _Loopback(world)
    outs, recs, errs = [None] * world, [None] * world, []

    def worker(r):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                plan = EPPlan(shape.num_experts, world, r)
                ops = GpuRank(shape, split_weights(inp, plan, shape.num_shared), plan,
                              log2phys=l2p)
                a, b = ranges[r]
                out = torch.full((b - a, shape.hidden), float("nan"), device="cuda")
                recs[r] = ep_forward(ops, plan, lb.rank(r), x[a:b].contiguous(), out)
                stream.synchronize()
                assert int(ops.status.item()) == 0
                outs[r] = out
        except BaseException as e:   # noqa: BLE001 -- reported below
            errs.append(e)
            lb.bar.abort()

    threads = [threading.Thread(target=worker, args=(r,)) for r in range(world)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=600)
    assert not errs, errs
    for r, (a, b) in enumerate(ranges):
        ref = torch.full((b - a, shape.hidden), float("nan"), device="cuda")
        ref_layer.forward(x[a:b].contiguous(), ref, T=b - a)
        torch.cuda.synchronize()
        assert torch.equal(outs[r], ref), f"rank {r} differs from the layer"
        for s in range(world):
            assert np.array_equal(recs[r]["recv_counts"][s], recs[s]["send_counts"][r])
    assert ref_layer.status() == 0


def _nccl_rank(port, results):
    import os
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        import moe_expert_layer_07_gb300 as moe
        import synth
        from moe_expert_layer_07_gb300 import _build
        from moe_expert_layer_07_gb300.ep import DistExchange, EPPlan, GpuRank, ep_forward, split_weights
        _build.build()
        shape = synth.CONFIGS["r1_mini"]
        inp = synth.make_inputs(shape, seed=6, device="cuda")
        plan = EPPlan(shape.num_experts, 1, 0)
        ops = GpuRank(shape, split_weights(inp, plan, shape.num_shared), plan)
        out = torch.full((shape.tokens, shape.hidden), float("nan"), device="cuda")
        rec = ep_forward(ops, plan, DistExchange(device="cuda"), inp["x"], out)
        ref = torch.full_like(out, float("nan"))
        moe.MoELayer(shape, inp).forward(inp["x"], ref)
        torch.cuda.synchronize()
        results["equal"] = bool(torch.equal(out, ref))
        results["rows"] = (rec["rows_sent"], rec["rows_received"])
        results["status"] = int(ops.status.item())
    finally:
        dist.destroy_process_group()


def test_dist_exchange_over_nccl_single_rank(lib):
    """ep_forward over a real NCCL process group (one rank, one GPU: each
    all-to-all is a copy to itself) gives the single-GPU layer's bits; the
    calls are those a multi-GPU run makes."""
    import os
    import torch.multiprocessing as mp
    port = 29700 + os.getpid() % 1000
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        p = ctx.Process(target=_nccl_rank, args=(port, results))
        p.start()
        p.join(timeout=600)
        assert p.exitcode == 0
        res = dict(results)
    assert res["equal"] and res["status"] == 0
    s = synth.CONFIGS["r1_mini"]
    assert res["rows"] == (s.tokens * s.top_k, s.tokens * s.top_k)
