"""Pins of the oracle's gate logits and expert selection (CPU only).

Logits: exact integer dot products, the fp64 dot within the fp32 error bound,
one-hot inputs.  Selection: brute force over every group subset and every
k-subset of experts on tiny inputs with many ties; the routing weights'
closed forms; library sigmoid/softmax as checks.
"""
import dataclasses
import itertools

import numpy as np
import pytest
import scipy.special

from oracle import quant, routing


@dataclasses.dataclass
class Cfg:
    num_experts: int
    top_k: int
    num_groups: int = 1
    topk_groups: int = 1
    group_topn: int = 1
    scoring: str = "sigmoid"
    norm_topk: bool = True
    routed_scaling: float = 1.0


def _bits(v):
    return quant.bf16_bits(np.asarray(v, np.float32))


def test_logits_exact_on_integer_inputs(oracle_lib):
    rng = np.random.default_rng(0)
    T, E, H = 5, 7, 1024
    x = rng.integers(-8, 9, size=(T, H)).astype(np.float32)
    w = rng.integers(-8, 9, size=(E, H)).astype(np.float32)
    # every partial sum is an integer below 2^24, so any order is exact
    l = routing.gate_logits(_bits(x), _bits(w))
    assert np.array_equal(l.astype(np.float64), x.astype(np.float64) @ w.T.astype(np.float64))
    off = rng.integers(-3, 4, size=E).astype(np.float32)
    l2 = routing.gate_logits(_bits(x), _bits(w), off)
    assert np.array_equal(l2, l + off)


def test_logits_one_hot_and_ragged_hidden(oracle_lib):
    rng = np.random.default_rng(1)
    E, H = 9, 7168 + 8          # H not a multiple of 256: a short last slice
    w = quant.bf16_round(rng.standard_normal((E, H)) * 0.02).astype(np.float32)
    for h in (0, 7, 8, 255, 256, 4097, H - 1):
        x = np.zeros((1, H), np.float32)
        x[0, h] = 1.0
        l = routing.gate_logits(_bits(x), _bits(w))
        assert np.array_equal(l[0], w[:, h])


def test_logits_summation_order_by_absorption(oracle_lib):
    """The fixed summation order, pinned by fp32 absorption (2^24 + 1 rounds to
    2^24): each case's value is worked out by hand for the order the routing
    reading fixes -- hidden index h in lane slice (h/8) mod 32, each slice
    summed in increasing h, the 32 slices meeting in an xor butterfly
    (16, 8, 4, 2, 1) -- and differs under the plausible alternatives."""
    H, big = 1024, 2.0 ** 24

    def logit(products):
        x = np.zeros((1, H), np.float32)
        w = np.zeros((1, H), np.float32)
        for h, p in products.items():
            x[0, h], w[0, h] = 1.0, p        # bf16-exact values
        return float(routing.gate_logits(_bits(x), _bits(w))[0, 0])

    # three slices (lanes 0, 1, 2): the butterfly adds lane 2 to lane 0 (2^24 - 2^24)
    # before lane 1 joins: 1; summed in increasing h it would be (2^24 + 1) - 2^24 = 0
    assert logit({0: big, 8: 1.0, 16: -big}) == 1.0
    # one slice, increasing h: 2^24 absorbs each 1; in decreasing h, 1 + 1 + 2^24
    assert logit({0: big, 1: 1.0, 2: 1.0}) == big
    assert logit({2: big, 1: 1.0, 0: 1.0}) == big + 2.0
    # slices of 8 consecutive elements: h = 0, 1 share lane 0 (the 1 is absorbed)
    # and h = 32 is lane 4: 0; with h mod 32 lanes, h = 0 and 32 would cancel in
    # lane 0 and the 1 would survive in lane 1
    assert logit({0: big, 1: 1.0, 32: -big}) == 0.0
    # h = 256 returns to lane 0 after h = 0..255: (2^24 + 1) absorbed, then -2^24
    assert logit({0: big, 256: 1.0, 512: -big}) == 0.0


def test_logits_within_fp32_bound_of_fp64_dot(oracle_lib):
    rng = np.random.default_rng(2)
    T, E, H = 6, 16, 7168
    x = quant.bf16_round(rng.standard_normal((T, H))).astype(np.float32)
    w = quant.bf16_round(rng.standard_normal((E, H)) * 0.02).astype(np.float32)
    l = routing.gate_logits(_bits(x), _bits(w)).astype(np.float64)
    exact = x.astype(np.float64) @ w.T.astype(np.float64)
    # 224 sequential adds per slice + 5 butterfly levels: gamma_n with n = 229
    bound = 229 * 2.0 ** -24 * (np.abs(x).astype(np.float64) @ np.abs(w).T.astype(np.float64))
    assert np.all(np.abs(l - exact) <= bound)
    assert not np.array_equal(l, exact.astype(np.float32))   # rounding is visible


def _brute_groups(sel, cfg):
    """Groups chosen by exhaustive search: the best-scoring subset in the
    (score desc, index asc) order, i.e. each kept group beats each dropped one."""
    gs = cfg.num_experts // cfg.num_groups
    gscore = []
    for g in range(cfg.num_groups):
        vals = sorted(((sel[e], -e) for e in range(g * gs, (g + 1) * gs)), reverse=True)
        acc = np.float32(vals[0][0])
        for v, _ in vals[1:cfg.group_topn]:
            acc = np.float32(acc + v)
        gscore.append(acc)
    good = []
    for sub in itertools.combinations(range(cfg.num_groups), cfg.topk_groups):
        rest = [g for g in range(cfg.num_groups) if g not in sub]
        if all(gscore[a] > gscore[b] or (gscore[a] == gscore[b] and a < b)
               for a in sub for b in rest):
            good.append(set(sub))
    assert len(good) == 1
    return good[0]


def _brute_topk(sel, allowed, k):
    good = []
    for sub in itertools.combinations(allowed, k):
        rest = [e for e in allowed if e not in sub]
        if all(sel[a] > sel[b] or (sel[a] == sel[b] and a < b) for a in sub for b in rest):
            good.append(set(sub))
    assert len(good) == 1
    return good[0]


@pytest.mark.parametrize("E,G,TG,N,k", [(16, 4, 2, 2, 4), (12, 3, 2, 2, 3), (16, 8, 3, 2, 5),
                                         (8, 1, 1, 1, 3), (16, 4, 1, 3, 2)])
def test_selection_matches_brute_force_with_ties(E, G, TG, N, k):
    rng = np.random.default_rng(E * 100 + k)
    cfg = Cfg(num_experts=E, top_k=k, num_groups=G, topk_groups=TG, group_topn=N,
              routed_scaling=2.5)
    for trial in range(60):
        # logits and biases on a coarse grid so that ties are common
        l = (rng.integers(-3, 4, size=E) * 0.5).astype(np.float32)
        bias = (rng.integers(-2, 3, size=E) * 0.125).astype(np.float32) if trial % 2 else None
        ids, w = routing.select_token(l, cfg, bias)
        s = routing.sigmoid_scores(l)
        sel = s if bias is None else (s + bias).astype(np.float32)
        if G > 1:
            groups = _brute_groups(sel, cfg)
            gs = E // G
            allowed = [e for e in range(E) if e // gs in groups]
        else:
            allowed = list(range(E))
        assert set(ids.tolist()) == _brute_topk(sel, allowed, k)
        # slot order: descending score, ties by ascending index
        keys = [(-sel[e], e) for e in ids]
        assert keys == sorted(keys)
        # weights: un-biased sigmoid, normalised, times routed_scaling
        assert abs(float(w.astype(np.float64).sum()) - 2.5) < 2.5 * 4e-7
        ref = s[ids].astype(np.float64) / s[ids].astype(np.float64).sum() * 2.5
        assert np.allclose(w, ref, rtol=1e-7, atol=0)


def test_softmax_weights_against_scipy():
    rng = np.random.default_rng(7)
    for norm in (True, False):
        cfg = Cfg(num_experts=64, top_k=6, scoring="softmax", norm_topk=norm, routed_scaling=1.0)
        for _ in range(20):
            l = (rng.standard_normal(64) * 0.3).astype(np.float32)
            ids, w = routing.select_token(l, cfg, None)
            p = scipy.special.softmax(l.astype(np.float64))
            assert set(ids.tolist()) == set(np.argsort(-l, kind="stable")[:6].tolist())
            ref = p[ids] / p[ids].sum() if norm else p[ids]
            assert np.allclose(w, ref, rtol=1e-7, atol=0)
            if norm:
                assert abs(float(w.astype(np.float64).sum()) - 1.0) < 4e-7


def test_sigmoid_scores_against_scipy_expit():
    rng = np.random.default_rng(8)
    l = (rng.standard_normal(100000) * 4).astype(np.float32)
    ours = routing.sigmoid_scores(l)
    ref = scipy.special.expit(l.astype(np.float64)).astype(np.float32)
    assert np.array_equal(ours, ref)


def test_route_applies_permutation_to_ids_only(oracle_lib):
    rng = np.random.default_rng(9)
    cfg = Cfg(num_experts=32, top_k=8, num_groups=8, topk_groups=4, group_topn=2,
              routed_scaling=2.5)
    logits = (rng.standard_normal((11, 32))).astype(np.float32)
    bias = (rng.standard_normal(32) * 0.01).astype(np.float32)
    perm = rng.permutation(32).astype(np.int32)
    p0, w0, l0 = routing.route(logits, cfg, bias)
    p1, w1, l1 = routing.route(logits, cfg, bias, perm)
    assert np.array_equal(l0, l1) and np.array_equal(w0, w1)
    assert np.array_equal(p1, perm[l0]) and np.array_equal(p0, l0)
