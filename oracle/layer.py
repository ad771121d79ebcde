"""The MoE FFN layer and its steps, by definition, on the CPU.

Test infrastructure only (see oracle/__init__.py).

Sources.  Moreh report "21K output tokens/s DeepSeek inference on MI300X
with Expert Parallelism": section "Overview" (experts are small FFNs, a
light gate picks a few per token), section "Parallelisation" (an always-on
shared expert besides the routed ones) and section "Library optimisation"
(horizontal fusion of the shared expert's GEMMs).  SGLang/H20 article,
sections "MoE" (prefill: block-scale handling, down-projection input) and
"SwapAB GEMM" (grouped GEMMs over variable per-expert row counts).

Readings taken where the pages say nothing:
  * an expert is a SwiGLU MLP: y = W2 (silu(W_gate x) * (W_up x)), with
    silu(z) = z / (1 + e^-z); W13 = [W_gate; W_up] is [2I, H], W2 is [H, I];
  * the layer output is out[t] = sum_s y_s(t) + sum_j w[t,j] * y_(e_j)(t),
    shared experts with weight 1 and no routed_scaling;
  * a model with n shared experts of width I has n shared groups;
  * quantisation points are part of the layer: in the FP8 layer x is
    quantised per token and 128-column group, h likewise (from its fp32
    value, the precision the decision is taken in); in the BF16 layer h is
    rounded to bf16 (the tensor-core operand format);
  * an expert output y is not rounded: on one GPU it never crosses a link
    (the all-to-all combine of the report's section "Compute-communication
    overlap" is where a narrower wire format would apply), so it is summed
    into the output at full precision;
  * everything else is exact: products and sums here are fp64.
"""
from __future__ import annotations

import numpy as np

from . import _clib
from .permute import permute
from .quant import (bf16_from_bits, bf16_round, dequant_groups_fp8,
                    quant_groups_fp8)
from .routing import gate_logits, route


def matmul_fp8(a64: np.ndarray, q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """a [n, K] fp64 times dequantised (q * block scale) [N, K] transposed."""
    a = np.ascontiguousarray(a64, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.float32)
    n, K = a.shape
    N = q.shape[0]
    assert q.shape == (N, K) and s.shape == (N // 128, K // 128)
    out = np.empty((n, N), dtype=np.float64)
    if n:
        _clib.lib().oracle_matmul_fp8(n, N, K, _clib.ptr(a), _clib.ptr(q),
                                      _clib.ptr(s), _clib.ptr(out))
    return out


def matmul_bf16(a64: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """a [n, K] fp64 times bf16 w [N, K] transposed, in fp64."""
    a = np.ascontiguousarray(a64, dtype=np.float64)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    n, K = a.shape
    N = w.shape[0]
    assert w.shape == (N, K)
    out = np.empty((n, N), dtype=np.float64)
    if n:
        _clib.lib().oracle_matmul_bf16(n, N, K, _clib.ptr(a), _clib.ptr(w),
                                       _clib.ptr(out))
    return out


def silu(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def silu_mul(g: np.ndarray) -> np.ndarray:
    """h = silu(gate) * up for rows [gate (I cols) | up (I cols)], fp64."""
    g = np.asarray(g, dtype=np.float64)
    I = g.shape[1] // 2
    return silu(g[:, :I]) * g[:, I:]


def expert_ffn(cfg, x_rows, w13, w2, w13_s=None, w2_s=None, x_scales=None):
    """One expert's SwiGLU MLP on n rows; returns fp64 [n, H].

    FP8 layer: x_rows are e4m3 codes [n, H] with x_scales [n, H/128], the
    weights e4m3 codes with 128x128 block scales.  BF16 layer: x_rows and
    weights are bf16 bit patterns.
    """
    if cfg.dtype == "fp8":
        a = dequant_groups_fp8(x_rows, x_scales)
        g = matmul_fp8(a, w13, w13_s)
        h = silu_mul(g).astype(np.float32)
        hq, hs = quant_groups_fp8(h)
        y = matmul_fp8(dequant_groups_fp8(hq, hs), w2, w2_s)
    else:
        a = bf16_from_bits(x_rows).astype(np.float64)
        g = matmul_bf16(a, w13)
        h = bf16_round(silu_mul(g))
        y = matmul_bf16(h, _bits(w2))
    return y


def _bits(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def grouped_gemm(cfg, offsets, a_rows, w, a_scales=None, w_scales=None):
    """C[r] = A[r] W[g]^T for the rows r of each group g, fp64 [rows, N].

    Rows outside [offsets[0], offsets[G]) are left at zero.
    """
    off = np.asarray(offsets, dtype=np.int64)
    G = len(off) - 1
    N = w.shape[1]
    out = np.zeros((a_rows.shape[0], N), dtype=np.float64)
    for g in range(G):
        r0, r1 = off[g], off[g + 1]
        if r1 <= r0:
            continue
        if cfg.dtype == "fp8":
            a = dequant_groups_fp8(a_rows[r0:r1], a_scales[r0:r1])
            out[r0:r1] = matmul_fp8(a, w[g], w_scales[g])
        else:
            a = bf16_from_bits(a_rows[r0:r1]).astype(np.float64)
            out[r0:r1] = matmul_bf16(a, _bits(w[g]))
    return out


def combine(y_rows, row_of_slot, topk_w, offsets, num_experts, num_shared):
    """out[t] = sum_s Y[shared row of t] + sum_j w[t,j] Y[row_of_slot[t,j]]."""
    y = np.asarray(y_rows, dtype=np.float64)
    ros = np.asarray(row_of_slot, dtype=np.int64)
    w = np.asarray(topk_w, dtype=np.float32).astype(np.float64)
    off = np.asarray(offsets, dtype=np.int64)
    T, k = ros.shape
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    for s in range(num_shared):
        out += y[off[num_experts + s] + np.arange(T)]
    for j in range(k):
        out += w[:, j:j + 1] * y[ros[:, j]]
    return out


def layer_forward(cfg, inp: dict, tokens=None) -> dict:
    """The whole layer.  `inp` holds numpy arrays:
        x_bits [T, H] uint16 (bf16), wg_bits [E, H] uint16 (bf16, logical
        expert order), e_bias [E] fp32 or None, logit_offset [E] fp32 or
        None, log2phys [E] int32 or None, w13 [G, 2I, H] and w2 [G, H, I]
        (uint8 e4m3 codes or uint16 bf16 bits, physical order, shared
        experts last), w13_s [G, 2I/128, H/128] and w2_s [G, H/128, I/128]
        fp32 (FP8 layer).
    Routing runs for every token; the expert FFNs and the output run for
    `tokens` (default: all), a list of token indices.
    """
    x = inp["x_bits"]
    T, H = x.shape
    E, k, S = cfg.num_experts, cfg.top_k, cfg.num_shared
    logits = gate_logits(x, inp["wg_bits"], inp.get("logit_offset"))
    phys, weights, logical = route(logits, cfg, inp.get("e_bias"), inp.get("log2phys"))
    offsets, src_of_row, row_of_slot = permute(phys, E, S)
    if tokens is None:
        tokens = np.arange(T)
    tokens = np.asarray(tokens, dtype=np.int64)

    if cfg.dtype == "fp8":
        xq, xs = quant_groups_fp8(bf16_from_bits(x))
    else:
        xq, xs = x, None

    n = len(tokens)
    y_routed = np.zeros((n, k, H), dtype=np.float64)
    y_shared = np.zeros((n, S, H), dtype=np.float64)
    w13, w2 = inp["w13"], inp["w2"]
    w13_s, w2_s = inp.get("w13_s"), inp.get("w2_s")

    def run(e, rows):
        return expert_ffn(cfg, xq[rows], w13[e], w2[e],
                          None if w13_s is None else w13_s[e],
                          None if w2_s is None else w2_s[e],
                          None if xs is None else xs[rows])

    sub = phys[tokens]                                  # [n, k]
    for e in np.unique(sub):
        ii, jj = np.nonzero(sub == e)
        y_routed[ii, jj] = run(int(e), tokens[ii])
    for s in range(S):
        y_shared[:, s] = run(E + s, tokens)

    w = weights[tokens].astype(np.float64)
    out = y_shared.sum(axis=1) + (w[:, :, None] * y_routed).sum(axis=1)
    return dict(logits=logits, topk_ids=phys, topk_w=weights, logical_ids=logical,
                expert_offsets=offsets, src_of_row=src_of_row,
                row_of_slot=row_of_slot, tokens=tokens, out=out,
                xq=xq if cfg.dtype == "fp8" else None, xs=xs)
