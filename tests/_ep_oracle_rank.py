"""A CPU rank for the expert-parallel step, for tests only: each local step of
moe_expert_layer_07_gb300.ep.GpuRank computed by the oracle instead of the
CUDA kernels, with host tensors for the gloo collectives.  The step's
orchestration (plan, exchanges, reassembly) is the product's ep_forward."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from moe_expert_layer_07_gb300.ep import EPPlan, StepState
from oracle import layer as olayer
from oracle import permute as opermute
from oracle import quant as oquant
from oracle import routing as orouting


class OracleRank:
    def __init__(self, shape, npin: dict, plan: EPPlan):
        """npin: the full layer's numpy inputs (synth.to_numpy): weights in
        physical order, shared experts last, and log2phys."""
        self.shape, self.np, self.plan = shape, npin, plan
        self.received = None

    def dispatch(self, x_bits: np.ndarray) -> StepState:
        s, n = self.shape, self.np
        T, E, k, S = x_bits.shape[0], s.num_experts, s.top_k, s.num_shared
        logits = orouting.gate_logits(x_bits, n["wg_bits"], n.get("logit_offset"))
        phys, w, _ = orouting.route(logits, s, n.get("e_bias"), n.get("log2phys"))
        off, src, ros = opermute.permute(phys, E, S)
        tok = opermute.token_of_slot(src, T, k)
        if self.fp8:
            xq, xs = oquant.quant_groups_fp8(oquant.bf16_from_bits(x_bits))
            rows = dict(xp=torch.from_numpy(np.ascontiguousarray(xq[tok])),
                        xps=torch.from_numpy(np.ascontiguousarray(xs[tok])))
        else:   # bf16 rows travel as their bytes
            xq, xs = np.ascontiguousarray(x_bits, np.uint16), None
            rows = dict(xp=torch.from_numpy(np.ascontiguousarray(xq[tok]).view(np.uint8)))
        d = dict(ids=phys, w=w, ros=ros, src=src, xq=xq, xs=xs,
                 y=torch.zeros((len(src), s.hidden), dtype=torch.float64), **rows)
        return StepState(T=T, offsets=off, tensors=d)

    @property
    def fp8(self):
        return self.shape.dtype == "fp8"

    def new_rows(self, nrows):
        H = self.shape.hidden
        if not self.fp8:
            return {"xp": torch.empty((nrows, 2 * H), dtype=torch.uint8)}
        return {"xp": torch.empty((nrows, H), dtype=torch.uint8),
                "xps": torch.empty((nrows, H // 128), dtype=torch.float32)}

    def sent_rows(self, st, name, R):
        return st.tensors[name][:R]

    def returned_rows(self, st, R):
        return st.tensors["y"][:R]

    def local_experts(self, plan, local_ids, bufs):
        xp = bufs["xp"].numpy()
        if not self.fp8:
            xp = np.ascontiguousarray(xp).view(np.uint16)
        xps = bufs["xps"].numpy() if self.fp8 else None
        self.received = {"local_ids": local_ids.copy(), "xp": xp.copy(),
                         "xps": None if xps is None else xps.copy()}
        n, H = len(local_ids), self.shape.hidden
        y = np.zeros((n, H), dtype=np.float64)
        for j in np.unique(local_ids):
            rows = np.nonzero(local_ids == j)[0]
            e = plan.rank * plan.m + int(j)                   # physical expert
            y[rows] = self._ffn(e, xp[rows], None if xps is None else xps[rows])
        return torch.from_numpy(y)

    def finish(self, st, out):
        s, d = self.shape, st.tensors
        T, E, S = st.T, s.num_experts, s.num_shared
        y = d["y"].numpy()
        for sh in range(S):
            r0 = int(st.offsets[E + sh])
            y[r0:r0 + T] = self._ffn(E + sh, d["xq"], d["xs"])
        out[:] = torch.from_numpy(olayer.combine(y, d["ros"], d["w"], st.offsets, E, S))
        return out

    def _ffn(self, e, xq, xs):
        n = self.np
        if not self.fp8:
            return olayer.expert_ffn(self.shape, xq, n["w13"][e], n["w2"][e])
        return olayer.expert_ffn(self.shape, xq, n["w13"][e], n["w2"][e], n["w13_s"][e],
                                 n["w2_s"][e], xs)


def token_split(T: int, world: int, seed: int = 0):
    """Uneven contiguous token ranges, one per rank (at least one token each)."""
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, T), world - 1, replace=False))
    edges = np.concatenate([[0], cuts, [T]])
    return [(int(a), int(b)) for a, b in zip(edges[:-1], edges[1:])]


def shape_with_tokens(shape, T):
    return dataclasses.replace(shape, tokens=T)
