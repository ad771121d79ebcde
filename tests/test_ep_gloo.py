"""Expert parallelism across ranks on the CPU: two (and four) gloo ranks run the
product's expert-parallel step (moe_expert_layer_07_gb300.ep.ep_forward: plan,
count and row all-to-alls, regrouping, inverse all-to-all, combine) with the
oracle standing in for each rank's kernels (tests/_ep_oracle_rank.py).

Checked against the oracle's single-process layer:
  * every rank's routing ids and expert offsets, bit for bit;
  * the send / receive tables agree across ranks (what d receives from s is
    what s sent to d);
  * every received row -- codes and scales, in arrival order (source-major,
    then expert, then the source's slot order) -- is the row the oracle's
    dispatch of the source's tokens holds for that expert;
  * each rank's output against the oracle layer on its tokens (the FP8
    tolerance; with the oracle as the local computation it agrees to
    rounding of the fp64 sums).
The balanced permutation gives each rank one set (Moreh report, section
"Load balancing across GPUs"); empty expert sets and a rank with one token
are covered.
"""
import os
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

from moe_expert_layer_07_gb300.ep import EPPlan  # noqa: E402

FP8_TOL = 2e-2


def _inputs(name, world):
    import synth
    import moe_expert_layer_07_gb300 as moe
    from oracle import routing as orouting
    shape = synth.CONFIGS[name]
    inp = synth.make_inputs(shape, seed=3, device="cpu")
    npin0 = synth.to_numpy(inp)
    logits = orouting.gate_logits(npin0["x_bits"], npin0["wg_bits"], npin0.get("logit_offset"))
    _, _, logical = orouting.route(logits, shape, npin0.get("e_bias"))
    counts = np.bincount(logical.reshape(-1), minlength=shape.num_experts)
    l2p, p2l, _ = moe.balance_permutation(counts, world)   # host call: one set per rank
    inp = synth.relayout_experts(inp, shape, p2l)
    return shape, synth.to_numpy(inp, l2p)


def _rank_main(rank, world, port, name, ranges, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from _ep_oracle_rank import OracleRank
    from moe_expert_layer_07_gb300.ep import DistExchange, ep_forward
    shape, npin = _inputs(name, world)
    plan = EPPlan(shape.num_experts, world, rank)
    ops = OracleRank(shape, npin, plan)
    a, b = ranges[rank]
    x = np.ascontiguousarray(npin["x_bits"][a:b])
    out = torch.zeros((b - a, shape.hidden), dtype=torch.float64)
    rec = ep_forward(ops, plan, DistExchange(device="cpu"), x, out)
    st = ops.dispatch(x)   # the rank's own routing tables, for the checks
    results[rank] = dict(out=out.numpy(), send=rec["send_counts"], recv=rec["recv_counts"],
                         ids=st.tensors["ids"], offsets=st.offsets,
                         received=ops.received)
    dist.barrier()
    dist.destroy_process_group()


def _run(name, world, ranges):
    port = 29600 + (os.getpid() + 37 * world) % 1000
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, name, ranges, results))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=600)
            assert p.exitcode == 0
        return dict(results)


@pytest.mark.parametrize("name,world,ranges", [
    ("r1_mini", 2, [(0, 20), (20, 37)]),
    ("r1_mini", 4, [(0, 1), (1, 12), (12, 30), (30, 37)]),
    ("bf16_mini", 2, [(0, 11), (11, 29)])])        # BF16, two shared experts, top-3
def test_expert_parallel_step_matches_the_oracle(oracle_lib, name, world, ranges):
    from oracle import layer as olayer
    from oracle import permute as opermute
    res = _run(name, world, ranges)
    shape, npin = _inputs(name, world)
    full = olayer.layer_forward(shape, npin)      # routing of every token, all outputs
    E, k, S = shape.num_experts, shape.top_k, shape.num_shared
    plan0 = EPPlan(E, world, 0)
    m = plan0.m
    for r in range(world):
        a, b = ranges[r]
        got = res[r]
        # routing and dispatch tables of the rank's tokens, bit for bit
        assert np.array_equal(got["ids"], full["topk_ids"][a:b])
        off, _, _ = opermute.permute(full["topk_ids"][a:b], E, S)
        assert np.array_equal(got["offsets"], off)
        assert np.array_equal(got["send"], np.diff(off[:E + 1]).reshape(world, m))
        for s in range(world):   # what r received from s is what s sent to r
            assert np.array_equal(got["recv"][s], res[s]["send"][r])
        # every received row, in arrival order
        exp_codes, exp_scales, exp_ids = [], [], []
        for s in range(world):
            sa, sb = ranges[s]
            ids_s = full["topk_ids"][sa:sb]
            for j in range(m):
                e = r * m + j
                tt, _ = np.nonzero(ids_s == e)          # slot order: t, then j
                if shape.dtype == "fp8":
                    exp_codes.append(full["xq"][sa + tt])
                    exp_scales.append(full["xs"][sa + tt])
                else:
                    exp_codes.append(npin["x_bits"][sa + tt])
                exp_ids.append(np.full(len(tt), j, np.int32))
        rec = got["received"]
        assert np.array_equal(rec["local_ids"], np.concatenate(exp_ids))
        assert np.array_equal(rec["xp"], np.concatenate(exp_codes))
        if shape.dtype == "fp8":
            assert np.array_equal(rec["xps"], np.concatenate(exp_scales))
        # the rank's output against the oracle layer on its tokens
        ref = full["out"][a:b]
        err = np.abs(got["out"] - ref).max()
        rms = np.sqrt(np.mean(full["out"] ** 2))
        assert err <= (FP8_TOL if shape.dtype == "fp8" else 5e-3) * rms
        assert err <= 1e-9 * rms    # same computation, different summation of rows
    # the balanced permutation spreads the routed rows evenly over the ranks
    loads = [int(res[r]["recv"].sum()) for r in range(world)]
    assert sum(loads) == (ranges[-1][1]) * k


def test_plan_tables():
    p = EPPlan(8, 4, 2)
    assert list(p.local_experts) == [4, 5]
    off = np.array([0, 1, 1, 4, 6, 6, 9, 9, 12, 20])   # 8 routed experts + 1 shared
    send = p.send_counts(off)
    assert send.tolist() == [[1, 0], [3, 2], [0, 3], [0, 3]]
    assert p.splits(send) == [1, 5, 3, 3]
    recv = np.array([[2, 0], [0, 1], [1, 1], [0, 0]])
    assert p.recv_local_ids(recv).tolist() == [0, 0, 1, 0, 1]
    assert p.recv_local_ids(np.zeros((4, 2), np.int64)).size == 0
    with pytest.raises(ValueError):
        EPPlan(10, 4, 0)
    with pytest.raises(ValueError):
        EPPlan(8, 4, 4)
    with pytest.raises(ValueError):
        p.recv_local_ids(np.array([[1, -1], [0, 0], [0, 0], [0, 0]]))
