"""Gating and top-k expert selection, by definition, one token at a time.

Test infrastructure only (see oracle/__init__.py).

Sources.  Moreh report "21K output tokens/s DeepSeek inference on MI300X with
Expert Parallelism": section "Overview" (a light gating network picks a small
subset of experts for each token), section "Parallelisation" (DeepSeek-R1:
256 experts, 8 active per token, plus an always-on shared expert) and
section "Load balancing across GPUs" (after the experts are permuted, the
gate must emit routing results in the new expert order).

The pages print no gating formula.  Readings (each the plainest one that
the R1- and V2-Lite-shaped workloads support):
  * softmax scoring: p = softmax(l) over all experts in fp64; experts are
    chosen by l; weight = p of the chosen expert, divided by the sum over
    the chosen ones when renormalised, times routed_scaling; rounded to fp32.
  * sigmoid scoring: s = fp32(1 / (1 + exp(-l))) computed in fp64;
    selection score s' = s + bias (fp32 add); weight = s / sum(s of chosen)
    times routed_scaling (bias excluded from the weight).
  * group-limited routing: experts form num_groups contiguous groups; a
    group's score is the fp32 sum, best first, of its top group_topn
    selection scores; the topk_groups best groups are kept and top_k
    experts are chosen among them.
  * ties: the lower expert index (or group index) wins.
  * slot order j: descending selection score, then ascending expert index.
  * routing is defined on logical expert ids; a permutation table log2phys
    only renames the chosen ids (phys = log2phys[logical]).
"""
from __future__ import annotations

import numpy as np

from . import _clib


def gate_logits(x_bits: np.ndarray, wg_bits: np.ndarray,
                offset: np.ndarray | None = None) -> np.ndarray:
    """fp32 gate logits [T, E] from bf16 bit patterns x [T, H], Wg [E, H].

    The summation order is fixed (see oracle_gate_logits in moe_oracle.c);
    the optional per-expert offset is added afterwards in fp32.
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w = np.ascontiguousarray(wg_bits, dtype=np.uint16)
    T, H = x.shape
    E, H2 = w.shape
    assert H == H2
    off = None if offset is None else np.ascontiguousarray(offset, dtype=np.float32)
    out = np.empty((T, E), dtype=np.float32)
    _clib.lib().oracle_gate_logits(T, E, H, _clib.ptr(x), _clib.ptr(w),
                                   _clib.ptr(off), _clib.ptr(out))
    return out


def _beats(va, ia, vb, ib) -> bool:
    """Total order of candidates: higher score first, then lower index."""
    return va > vb or (va == vb and ia < ib)


def _top_n(scores, candidates, n):
    """The n best of `candidates` (indices into scores), best first."""
    chosen = []
    pool = list(candidates)
    for _ in range(n):
        best = None
        for c in pool:
            if best is None or _beats(scores[c], c, scores[best], best):
                best = c
        chosen.append(best)
        pool.remove(best)
    return chosen


def sigmoid_scores(logits_row: np.ndarray) -> np.ndarray:
    """fp32 sigmoid of fp32 logits, evaluated in fp64 and rounded once."""
    l64 = np.asarray(logits_row, dtype=np.float32).astype(np.float64)
    return (1.0 / (1.0 + np.exp(-l64))).astype(np.float32)


def select_token(logits_row: np.ndarray, cfg, bias: np.ndarray | None):
    """Route one token.  Returns (logical ids [k], fp32 weights [k])."""
    E = cfg.num_experts
    l = np.asarray(logits_row, dtype=np.float32)
    if cfg.scoring == "sigmoid":
        s = sigmoid_scores(l)
        sel = s if bias is None else (s + np.asarray(bias, np.float32)).astype(np.float32)
    elif cfg.scoring == "softmax":
        if bias is not None:
            raise ValueError("softmax scoring takes no selection bias")
        s = None
        sel = l
    else:
        raise ValueError(cfg.scoring)

    if cfg.num_groups > 1:
        gs = E // cfg.num_groups
        gscore = []
        for g in range(cfg.num_groups):
            members = range(g * gs, (g + 1) * gs)
            best = _top_n(sel, members, cfg.group_topn)
            acc = np.float32(sel[best[0]])
            for b in best[1:]:
                acc = np.float32(acc + sel[b])
            gscore.append(acc)
        groups = _top_n(gscore, range(cfg.num_groups), cfg.topk_groups)
        allowed = [e for g in sorted(groups) for e in range(g * gs, (g + 1) * gs)]
    else:
        allowed = range(E)

    ids = _top_n(sel, allowed, cfg.top_k)

    if cfg.scoring == "sigmoid":
        chosen = s[ids].astype(np.float64)
        w = chosen / chosen.sum() if cfg.norm_topk else chosen
    else:
        l64 = l.astype(np.float64)
        p = np.exp(l64 - l64.max())
        p = p / p.sum()
        chosen = p[ids]
        w = chosen / chosen.sum() if cfg.norm_topk else chosen
    w = (w * cfg.routed_scaling).astype(np.float32)
    return np.asarray(ids, dtype=np.int32), w


def route(logits: np.ndarray, cfg, bias: np.ndarray | None = None,
          log2phys: np.ndarray | None = None):
    """Route every token of a batch.

    Returns (phys ids int32 [T, k], weights fp32 [T, k], logical ids [T, k]).
    """
    T = logits.shape[0]
    k = cfg.top_k
    logical = np.empty((T, k), dtype=np.int32)
    weights = np.empty((T, k), dtype=np.float32)
    for t in range(T):
        logical[t], weights[t] = select_token(logits[t], cfg, bias)
    if log2phys is None:
        phys = logical.copy()
    else:
        phys = np.asarray(log2phys, dtype=np.int32)[logical]
    return phys, weights, logical
