"""Expert parallelism: the layer's routed experts split over P ranks, tokens
carried to their experts' ranks by an all-to-all dispatch and the expert
outputs brought back by an all-to-all combine.

Report "21K output tokens/s DeepSeek inference on MI300X with Expert
Parallelism": section "Parallelisation" runs the routed experts expert-
parallel (EP8: 32 of the 256 experts on each GPU) and the rest of the layer
data-parallel, each GPU on its own tokens, with the shared expert on every
GPU; section "Load balancing across GPUs" gives every GPU one set of a
balanced expert permutation (the sets hold equal activation totals within a
few percent); section "Compute-communication overlap" moves the tokens with
an all-to-all dispatch and the results with an all-to-all combine.

One step on rank r of P (m = E / P routed experts per rank; physical experts
[d m, (d + 1) m) live on rank d):
  1. route, quantise and dispatch the rank's own tokens exactly as the
     single-GPU layer does.  The dispatched rows are ordered by physical
     expert, so the rows bound for rank d are one contiguous slice,
     [offsets[d m], offsets[(d + 1) m]);
  2. exchange the rows per (destination rank, expert) -- a P x m table --
     then the rows themselves (FP8 codes and their scales, or bf16): one
     all-to-all, rows arriving source-major, expert-minor;
  3. group the received rows by local expert (the dispatch kernel with one
     choice per row), run the local experts' FFN, and put the outputs back
     in arrival order (the combine kernel with one choice of weight 1, which
     is exact);
  4. return the outputs with the inverse all-to-all, into the rows they left;
  5. run the shared experts on the rank's own rows and combine.
A row's FFN output does not depend on which other rows share its tile, so
each rank's output equals the single-GPU layer's on its tokens, bit for bit.

The split sizes of the all-to-alls come from the expert counts, which this
path reads to the host (steps 1 and 2), so unlike moe_layer_forward it
synchronises the host once per exchange and is not graph-capturable.

This module is orchestration: plan arithmetic on the host, collectives, and
calls into the C ABI (GpuRank).  The exchange is any object with the two
methods of Exchange; DistExchange runs it over torch.distributed (NCCL for
device tensors, gloo for host tensors).
"""
from __future__ import annotations

import dataclasses

import numpy as np


class EPPlan:
    """Host arithmetic of one step on one rank: which experts are local, the
    send table from the rank's expert offsets and the local expert of every
    received row."""

    def __init__(self, num_experts: int, world: int, rank: int):
        if world <= 0 or num_experts % world:
            raise ValueError(f"{num_experts} experts do not split over {world} ranks")
        if not 0 <= rank < world:
            raise ValueError(f"rank {rank} outside 0..{world - 1}")
        self.E, self.P, self.rank = num_experts, world, rank
        self.m = num_experts // world

    @property
    def local_experts(self) -> range:
        """Physical ids of this rank's routed experts."""
        return range(self.rank * self.m, (self.rank + 1) * self.m)

    def send_counts(self, offsets) -> np.ndarray:
        """Rows per (destination rank, its expert), int64 [P, m], from this
        rank's expert offsets (routed experts first)."""
        off = np.asarray(offsets, dtype=np.int64)
        return np.diff(off[:self.E + 1]).reshape(self.P, self.m)

    @staticmethod
    def splits(counts) -> list[int]:
        """Rows per peer rank of a P x m table."""
        return [int(v) for v in np.asarray(counts, dtype=np.int64).sum(axis=1)]

    def recv_local_ids(self, recv_counts) -> np.ndarray:
        """Local expert (0..m-1) of every received row, in arrival order
        (source-major, expert-minor), int32."""
        c = np.asarray(recv_counts, dtype=np.int64)
        if c.shape != (self.P, self.m) or (c < 0).any():
            raise ValueError("received counts must be a non-negative P x m table")
        return np.tile(np.arange(self.m, dtype=np.int32), self.P).repeat(c.reshape(-1))


class Exchange:
    """What a step needs from the collectives (one call per rank)."""

    def counts(self, send: np.ndarray) -> np.ndarray:
        """All-to-all of a P x m int64 table: row s of the result is what rank
        s sent to this rank."""
        raise NotImplementedError

    def rows(self, out, inp, out_splits, in_splits):
        """All-to-all of row blocks: inp's rows [sum(in_splits[:d]), +in_splits[d])
        go to rank d; out's rows [sum(out_splits[:s]), +out_splits[s]) come from rank s."""
        raise NotImplementedError


class DistExchange(Exchange):
    """Exchange over torch.distributed (the default group unless given)."""

    def __init__(self, group=None, device=None):
        self.group, self.device = group, device

    def counts(self, send):
        import torch
        import torch.distributed as dist
        t = torch.as_tensor(np.ascontiguousarray(send, dtype=np.int64), device=self.device)
        out = torch.empty_like(t)
        dist.all_to_all_single(out, t, group=self.group)
        return out.cpu().numpy()

    def rows(self, out, inp, out_splits, in_splits):
        import torch.distributed as dist
        dist.all_to_all_single(out, inp, output_split_sizes=list(out_splits),
                               input_split_sizes=list(in_splits), group=self.group)


@dataclasses.dataclass
class StepState:
    """One rank's intermediates of a step, on its device (host: offsets)."""
    T: int
    offsets: np.ndarray        # int32 [E + S + 1], host copy
    tensors: dict              # the rank's own device buffers


def ep_forward(rank_ops, plan: EPPlan, exchange: Exchange, x, out):
    """One expert-parallel step of the layer on this rank's tokens x [T, H]
    into out [T, H] (fp32).  rank_ops supplies the local computation (GpuRank
    on a GPU); exchange the collectives.  Returns the step's host-side record
    (send and receive tables)."""
    st = rank_ops.dispatch(x)                         # 1. route, quantise, dispatch
    send = plan.send_counts(st.offsets)
    recv = exchange.counts(send)                      # 2. counts, then rows
    s_split, r_split = plan.splits(send), plan.splits(recv)
    R = int(st.offsets[plan.E])
    n_recv = int(sum(r_split))
    recv_bufs = rank_ops.new_rows(n_recv)
    for name, buf in recv_bufs.items():
        exchange.rows(buf, rank_ops.sent_rows(st, name, R), r_split, s_split)
    y_recv = rank_ops.local_experts(plan, plan.recv_local_ids(recv), recv_bufs)   # 3.
    exchange.rows(rank_ops.returned_rows(st, R), y_recv, s_split, r_split)        # 4.
    rank_ops.finish(st, out)                          # 5. shared experts + combine
    return {"send_counts": send, "recv_counts": recv, "rows_sent": R, "rows_received": n_recv}


class GpuRank:
    """The local computation of one rank through the C ABI: routing over all
    E experts (gate, bias and permutation are global), this rank's m routed
    experts and the shared experts.

    weights: dict of device tensors as for MoELayer, with w13/w2 (+ scales)
    holding only the rank's m routed experts (physical ids [r m, (r + 1) m),
    in order) followed by the shared experts; log2phys (global) optional.
    """

    def __init__(self, shape, weights: dict, plan: EPPlan, log2phys=None, pack_weights=True,
                 stream=None):
        import torch
        from . import (LAYOUT_ROWS, LAYOUT_TILES, make_config, pack_expert_weights)
        self.shape, self.plan, self.stream = shape, plan, stream
        self.fp8 = shape.dtype == "fp8"
        self.cfg = make_config(shape)
        m, S = plan.m, shape.num_shared
        w = dict(weights)
        if w["w13"].shape[0] != m + S:
            raise ValueError(f"expected {m} local + {S} shared experts, got {w['w13'].shape[0]}")
        # the local experts' config: m groups, one choice per received row
        self.cfg_local = make_config(dataclasses.replace(
            shape, num_experts=m, num_shared=0, top_k=1, num_groups=1, topk_groups=1,
            group_topn=1, scoring="softmax"))
        if pack_weights and w.get("expert_layout", LAYOUT_ROWS) == LAYOUT_ROWS:
            w["w13"] = pack_expert_weights(self.cfg_local, w["w13"], stream=stream)
            w["w2"] = pack_expert_weights(self.cfg_local, w["w2"], stream=stream)
            w["expert_layout"] = LAYOUT_TILES
        self.layout = w.get("expert_layout", LAYOUT_ROWS)
        self.w = w
        self.l2p = None if log2phys is None else torch.as_tensor(
            np.asarray(log2phys, np.int32), device=w["w13"].device)
        self.device = w["w13"].device

    # -- helpers
    def _empty(self, shape, dtype):
        import torch
        return torch.empty(shape, dtype=dtype, device=self.device)

    def _code_dtype(self):
        import torch
        return torch.uint8 if self.fp8 else torch.bfloat16

    def _ffn(self, cfg, groups, rows, xp, xps, offsets, w13, w13s, w2, w2s, y):
        """The FFN of `groups` expert groups on dispatched rows (h scratch here)."""
        import torch
        from . import expert_ffn_sched_bytes, experts_forward
        s = self.shape
        h = self._empty((max(rows, 1), s.inter), self._code_dtype())
        hs = self._empty((max(rows, 1), s.inter // 128), torch.float32) if self.fp8 else None
        nb = expert_ffn_sched_bytes(groups, rows)
        sched = self._empty((max(nb, 4) // 4,), torch.int32)
        experts_forward(cfg, groups, rows, xp, xps, offsets, w13, w13s, w2, w2s, h, hs, y,
                        sched, nb, self.status, stream=self.stream, w_layout=self.layout)

    # -- the step
    def dispatch(self, x) -> StepState:
        import torch
        from . import ACT_IDENTITY, act_requant, permute, permute_workspace_size, route
        s, cfg = self.shape, self.cfg
        T, H, E, k, S = x.shape[0], s.hidden, s.num_experts, s.top_k, s.num_shared
        rows = T * (k + S)
        d = {}
        self.status = self._empty((1,), torch.int32)
        self.status.zero_()
        d["logits"] = self._empty((max(T, 1), E), torch.float32)
        d["ids"] = self._empty((max(T, 1), k), torch.int32)
        d["w"] = self._empty((max(T, 1), k), torch.float32)
        d["offsets"] = self._empty((E + S + 1,), torch.int32)
        d["src"] = self._empty((max(rows, 1),), torch.int32)
        d["ros"] = self._empty((max(T, 1), k), torch.int32)
        d["xp"] = self._empty((max(rows, 1), H), self._code_dtype())
        d["xps"] = self._empty((max(rows, 1), H // 128), torch.float32) if self.fp8 else None
        d["y"] = self._empty((max(rows, 1), H), torch.float32)
        route(cfg, T, x, self.w["wg"], self.w.get("e_bias"), self.w.get("logit_offset"), self.l2p,
              d["logits"], d["ids"], d["w"], self.status, stream=self.stream)
        src_rows, src_sc = x, None
        if self.fp8:
            d["xq"] = self._empty((max(T, 1), H), torch.uint8)
            d["xs"] = self._empty((max(T, 1), H // 128), torch.float32)
            act_requant(cfg, ACT_IDENTITY, T, x, d["xq"], d["xs"], stream=self.stream)
            src_rows, src_sc = d["xq"], d["xs"]
        nws = permute_workspace_size(cfg, T)
        ws = self._empty((max(nws, 1),), torch.uint8)
        permute(cfg, T, d["ids"], src_rows, src_sc, d["offsets"], d["src"], d["ros"], d["xp"],
                d["xps"], ws, nws, self.status, stream=self.stream)
        off = d["offsets"].cpu().numpy() if self.stream is None else _to_host(d["offsets"],
                                                                               self.stream)
        return StepState(T=T, offsets=off, tensors=d)

    def new_rows(self, n):
        """Receive buffers for n rows of the dispatch all-to-all."""
        import torch
        H = self.shape.hidden
        bufs = {"xp": self._empty((n, H), self._code_dtype())}
        if self.fp8:
            bufs["xps"] = self._empty((n, H // 128), torch.float32)
        return bufs

    def sent_rows(self, st: StepState, name: str, R: int):
        return st.tensors[name][:R]

    def returned_rows(self, st: StepState, R: int):
        return st.tensors["y"][:R]

    def local_experts(self, plan: EPPlan, local_ids: np.ndarray, bufs: dict):
        """Outputs of this rank's experts for the received rows, in arrival order."""
        import torch
        from . import OUT_F32, combine, permute, permute_workspace_size
        n, H, m = len(local_ids), self.shape.hidden, plan.m
        y_recv = self._empty((n, H), torch.float32)
        if n == 0:
            return y_recv
        cl = self.cfg_local
        ids = torch.as_tensor(local_ids.reshape(n, 1), device=self.device)
        off = self._empty((m + 1,), torch.int32)
        src = self._empty((n,), torch.int32)
        ros = self._empty((n, 1), torch.int32)
        xg = self._empty((n, H), self._code_dtype())
        xgs = self._empty((n, H // 128), torch.float32) if self.fp8 else None
        nws = permute_workspace_size(cl, n)
        ws = self._empty((max(nws, 1),), torch.uint8)
        permute(cl, n, ids, bufs["xp"], bufs.get("xps"), off, src, ros, xg, xgs, ws, nws,
                self.status, stream=self.stream)
        yg = self._empty((n, H), torch.float32)
        w = self.w
        self._ffn(cl, m, n, xg, xgs, off, w["w13"], w.get("w13_s"), w["w2"], w.get("w2_s"), yg)
        ones = torch.ones((n, 1), dtype=torch.float32, device=self.device)
        combine(cl, n, yg, ros, ones, off, y_recv, OUT_F32, stream=self.stream)
        return y_recv

    def finish(self, st: StepState, out):
        """The shared experts on this rank's rows, then the combine into out."""
        from . import OUT_F32, combine
        s, d, m = self.shape, st.tensors, self.plan.m
        T, E, S = st.T, s.num_experts, s.num_shared
        if T == 0:
            return out
        rows = T * (s.top_k + S)
        if S:
            w = self.w
            # groups E .. E + S - 1 of the rank's offsets; shared weights follow
            # the m local experts in the rank's weight tensors
            def shared(key):
                t = w.get(key)
                return None if t is None else t[m:]
            self._ffn(self.cfg, S, rows, d["xp"], d["xps"], d["offsets"][E:], shared("w13"),
                      shared("w13_s"), shared("w2"), shared("w2_s"), d["y"])
        combine(self.cfg, T, d["y"], d["ros"], d["w"], d["offsets"], out, OUT_F32,
                stream=self.stream)
        return out


def _to_host(t, stream):
    import torch
    with torch.cuda.stream(stream):
        h = t.to("cpu", non_blocking=False)
    return h.numpy()


def split_weights(weights: dict, plan: EPPlan, num_shared: int) -> dict:
    """A rank's share of full-layer weights (physical order, shared last):
    its m routed experts, then the shared experts; gate, bias and offsets as
    they are."""
    import torch
    E = plan.E
    lo, hi = plan.rank * plan.m, (plan.rank + 1) * plan.m
    out = dict(weights)
    for key in ("w13", "w13_s", "w2", "w2_s"):
        t = weights.get(key)
        if t is not None:
            out[key] = torch.cat([t[lo:hi], t[E:E + num_shared]]).contiguous()
    return out
