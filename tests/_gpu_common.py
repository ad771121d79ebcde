"""Helpers shared by the GPU parity tests: workloads on the device, their
oracle view, and the tolerances the tests apply.

Tolerances
  * routing ids, expert offsets, permutation tables, x quantisation codes:
    bit-exact (both sides take the decision in the same fp32 arithmetic);
  * routing weights: relative 1e-6 (fp32 on the device, fp64 rounded once in
    the oracle: a few fp32 roundings apart, < 4e-7);
  * layer outputs: max |gpu - oracle| <= 2e-2 * rms(oracle) for FP8 layers
    and <= 5e-3 * rms(oracle) for BF16 layers (fp32 output); with a bf16
    output half a bf16 unit of the value is added to the bound;
  * fp32 grouped-GEMM output: max error <= 1e-3 * rms (fp32 accumulation of
    at most 7168 exact products against fp64: about sqrt(K) * 2^-24
    relative, far inside the bound).
"""
from __future__ import annotations

import numpy as np
import torch

import moe_expert_layer_07_gb300 as moe
import synth
from oracle import balance as obal
from oracle import layer as olayer
from oracle import routing as orouting

FP8_TOL = 2e-2
BF16_TOL = 5e-3
W_RTOL = 1e-6


def build_library():
    from moe_expert_layer_07_gb300 import _build
    _build.build()
    return moe.lib()


class Workload:
    """Device tensors of one seeded workload plus its oracle (numpy) view."""

    def __init__(self, shape: synth.MoEShape, seed: int = 0, perm: str | None = None):
        self.shape = shape
        inp = synth.make_inputs(shape, seed=seed, device="cuda")
        self.log2phys = None
        if perm == "random":
            rng = np.random.default_rng(seed + 99)
            p2l = rng.permutation(shape.num_experts)
            self.log2phys = np.argsort(p2l).astype(np.int32)
        elif perm == "balanced" or (perm is None and shape.balanced_perm):
            # counts from routing the same batch without a permutation
            logical = self.oracle_logical_ids(inp)
            counts = np.bincount(logical.reshape(-1), minlength=shape.num_experts)
            l2p, p2l, self.imbalance = moe.balance_permutation(counts, shape.num_sets)
            self.naive_imbalance = obal.imbalance(obal.contiguous_loads(counts, shape.num_sets))
            self.counts = counts
            self.log2phys = l2p
        if self.log2phys is not None:
            inp = synth.relayout_experts(inp, shape, np.argsort(self.log2phys))
        self.dev = inp
        self._np = None

    def oracle_logical_ids(self, inp):
        def bits(t):
            return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        off = None if inp["logit_offset"] is None else inp["logit_offset"].cpu().numpy()
        bias = None if inp["e_bias"] is None else inp["e_bias"].cpu().numpy()
        l = orouting.gate_logits(bits(inp["x"]), bits(inp["wg"]), off)
        _, _, logical = orouting.route(l, self.shape, bias)
        return logical

    @property
    def np(self):
        if self._np is None:
            self._np = synth.to_numpy(self.dev, self.log2phys)
        return self._np

    def layer(self, max_tokens=None):
        w = dict(self.dev)
        return moe.MoELayer(self.shape, w, max_tokens=max_tokens, log2phys=self.log2phys)


def rms(a):
    return float(np.sqrt(np.mean(np.asarray(a, np.float64) ** 2)))


def check_close(gpu, ref, tol, bf16_out=False):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    r = rms(ref)
    bound = tol * r
    if bf16_out:   # plus half a bf16 unit in the last place of the value
        a = np.abs(ref)
        _, ex = np.frexp(np.where(a > 0, a, 1.0))
        bound = bound + np.where(a > 0, np.ldexp(1.0, ex.astype(np.int64) - 1 - 8), 0.0)
    err = np.abs(gpu - ref)
    worst = float((err / np.maximum(bound, 1e-300)).max()) if err.size else 0.0
    assert np.all(err <= bound), f"max err {err.max():.3e} vs rms {r:.3e} (ratio {worst:.3f})"
    return float(err.max()) / r if r > 0 else 0.0


def fp8_codes_equal(a, b):
    """e4m3 codes compared as values: +0 and -0 (0x00, 0x80) are the same zero."""
    a = np.where(np.asarray(a) == 0x80, 0, np.asarray(a))
    b = np.where(np.asarray(b) == 0x80, 0, np.asarray(b))
    return np.array_equal(a, b)


def oracle_layer(wl: Workload, tokens=None):
    return olayer.layer_forward(wl.shape, wl.np, tokens=tokens)


def to_np(t):
    return t.detach().cpu().numpy()
