"""The C-ABI library on the host (no GPU needed): it loads, exports every
function include/moe_gb300.h declares, rejects bad arguments before any
launch, and its host-only balanced permutation matches the oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

import moe_expert_layer_07_gb300 as moe
import synth
from oracle import balance

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def L():
    from moe_expert_layer_07_gb300 import _build
    _build.build()
    return moe.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    return sorted({n for n in names if n.startswith(("moe_", "expert_")) and n != "moe_config"})


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(L, n), f"{n} declared in the header but not exported"


def test_error_detail_is_a_thread_local_text(L):
    """moe_last_error_detail names the CUDA call behind a MOE_ERR_CUDA; a thread
    that has seen none reads an empty text (argument errors do not set it)."""
    import threading
    cfg = moe.make_config(synth.CONFIGS["r1_mini"])
    seen = []

    def fresh_thread():
        assert L.moe_route(ctypes.byref(cfg), 4, None, None, None, None, None, None, None, None,
                           None, None) == -1
        seen.append(moe.last_error_detail())

    t = threading.Thread(target=fresh_thread)
    t.start()
    t.join()
    assert seen == [""]


def test_status_strings(L):
    assert moe.status_string(0) == "ok"
    for code in (-1, -2, -3, -4, -5, -6):
        assert moe.status_string(code) not in ("ok", "unknown status")
    assert moe.status_string(-99) == "unknown status"


def test_workspace_size_r1_decode(L):
    shape = synth.CONFIGS["r1_decode_t128"]
    cfg = moe.make_config(shape)
    n = moe.workspace_size(cfg)
    lay = moe.workspace_layout(cfg)
    assert lay.total == n and lay.status == 0
    rows = 128 * 9
    # the largest buffers: fp32 y [rows, 7168], fp8 xp [rows, 7168], fp8 h [rows, 2048]
    floor = rows * 7168 * 4 + rows * 7168 + rows * 2048
    assert floor < n < floor * 1.2
    offs = [lay.status, lay.logits, lay.topk_ids, lay.topk_w, lay.xq, lay.xs, lay.expert_offsets,
            lay.src_of_row, lay.row_of_slot, lay.perm_scratch, lay.xp, lay.xp_scales, lay.gate_up,
            lay.h, lay.h_scales, lay.y]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    # the one-kernel FFN's scheduler counters follow the status word, so one
    # memset clears both
    assert lay.ffn_sched == 256
    assert lay.logits - lay.ffn_sched >= moe.expert_ffn_sched_bytes(257, rows)


def test_layer_kernel_counts(L):
    # route (2, the FP8 quantisation of x inside) + permute (2 for at most 1024
    # routed slots, else 3) + experts' FFN + combine
    r1 = moe.make_config(synth.CONFIGS["r1_decode_t128"])
    assert moe.layer_kernel_count(r1, 128) == 6        # one-kernel FFN, 1024 slots
    assert moe.layer_kernel_count(r1, 129) == 7        # 1032 slots: count and scan apart
    assert moe.layer_kernel_count(r1, 4096) == 9       # wide: FFN (small groups), 2 GEMMs
    mini = moe.make_config(synth.CONFIGS["r1_mini"])   # inter 384: odd K blocks of W2
    assert moe.layer_kernel_count(mini, 37) == 6
    b16 = moe.make_config(synth.CONFIGS["bf16_mini"])   # BF16: one-kernel FFN
    assert moe.layer_kernel_count(b16, 29) == 6
    assert moe.layer_kernel_count(r1, 0) == 0


def test_bad_arguments_are_rejected_before_launch(L):
    shape = synth.CONFIGS["r1_mini"]
    cfg = moe.make_config(shape)
    P = ctypes.c_void_p
    fake = P(0x1000)   # never dereferenced: every call below fails validation first
    # null pointers
    assert L.moe_route(ctypes.byref(cfg), 4, None, fake, None, None, None, fake, fake, fake,
                       None, None) == -1
    # misaligned activation pointer
    assert L.moe_route(ctypes.byref(cfg), 4, P(0x1001), fake, None, None, None, fake, fake, fake,
                       None, None) == -1
    # shapes the kernels do not handle
    bad = moe.make_config(shape)
    bad.hidden = 1000
    assert L.moe_route(ctypes.byref(bad), 4, fake, fake, None, None, None, fake, fake, fake,
                       None, None) == -2
    ALL = moe.ALL_ROWS
    assert L.moe_grouped_gemm(ctypes.byref(cfg), 3, 200, 128, 10, fake, fake, fake, fake, fake,
                              0, fake, 0, 0, ALL, None, None) == -2
    assert L.moe_grouped_gemm(ctypes.byref(cfg), 2000, 128, 128, 10, fake, fake, fake, fake,
                              fake, 0, fake, 0, 0, ALL, None, None) == -2
    # unknown weight layout
    assert L.moe_grouped_gemm(ctypes.byref(cfg), 3, 256, 128, 10, fake, fake, fake, fake, fake,
                              7, fake, 0, 0, ALL, None, None) == -1
    assert L.moe_grouped_gemm_swiglu(ctypes.byref(cfg), 3, 256, 128, 10, fake, fake, fake, fake,
                                     fake, 2, fake, fake, 0, ALL, None, None) == -1
    # a group row window that starts below zero
    assert L.moe_grouped_gemm(ctypes.byref(cfg), 3, 256, 128, 10, fake, fake, fake, fake, fake,
                              0, fake, 0, -1, ALL, None, None) == -1
    assert L.moe_grouped_gemm_swiglu(ctypes.byref(cfg), 3, 256, 128, 10, fake, fake, fake, fake,
                                     fake, 0, fake, fake, -1, ALL, None, None) == -1
    # packing: shapes and overlap
    assert L.moe_pack_expert_weights(ctypes.byref(cfg), 2, 200, 128, fake, P(0x100000),
                                     None) == -2
    assert L.moe_pack_expert_weights(ctypes.byref(cfg), 2, 256, 128, fake, P(0x1000 + 4096),
                                     None) == -1
    assert L.moe_pack_expert_weights(ctypes.byref(cfg), 2, 256, 128, P(0x1008), P(0x100000),
                                     None) == -1
    # workspace too small
    need = moe.permute_workspace_size(cfg, 37)
    assert L.moe_permute(ctypes.byref(cfg), 37, fake, fake, fake, fake, fake, fake, fake, fake,
                         fake, need - 1, ALL, None, None) == -3
    assert L.moe_permute(ctypes.byref(cfg), 37, fake, fake, fake, fake, fake, fake, fake, fake,
                         fake, need, -1, None, None) == -1   # a negative copy window
    # the gathering gate/up GEMM: FP8 only, token rows needed, known layouts
    gg = lambda c, T, rows, layout=0, lo=0, xr=fake: L.moe_grouped_gemm_swiglu_gather(
        ctypes.byref(c), 3, 256, 1024, rows, xr, fake, T, fake, fake, fake, fake, layout, fake,
        fake, lo, ALL, None, None)
    b16c = moe.make_config(synth.CONFIGS["bf16_mini"])
    assert gg(b16c, 4, 10) == -1          # BF16 layer
    assert gg(cfg, 4, 10, layout=3) == -1
    assert gg(cfg, 4, 10, lo=-1) == -1
    assert gg(cfg, 0, 10) == -1           # rows to fill, no token rows
    assert gg(cfg, 4, 10, xr=None) == -1
    assert gg(cfg, 4, 10, xr=P(0x1004)) == -1   # unaligned token rows
    assert gg(cfg, 4, 0) == 0             # nothing to do
    # identity quantisation (alone or with routing) needs an FP8 layer; unknown enums
    b16 = moe.make_config(synth.CONFIGS["bf16_mini"])
    assert L.moe_route_quantize(ctypes.byref(b16), 4, fake, fake, None, None, None, fake, fake,
                                fake, fake, fake, None, None) == -1
    assert L.moe_route_quantize(ctypes.byref(cfg), 4, fake, fake, None, None, None, fake, fake,
                                fake, None, fake, None, None) == -1
    assert L.moe_route_quantize(ctypes.byref(cfg), 0, None, None, None, None, None, None, None,
                                None, None, None, None, None) == 0
    assert L.moe_act_requant(ctypes.byref(b16), moe.ACT_IDENTITY, 4, None, fake, fake, fake,
                             None) == -1
    assert L.moe_act_requant(ctypes.byref(cfg), 7, 4, None, fake, fake, fake, None) == -1
    # softmax takes no selection bias
    assert L.moe_route(ctypes.byref(b16), 4, fake, fake, fake, None, None, fake, fake, fake,
                       None, None) == -1
    # group-limited routing that cannot supply k candidates
    g = moe.make_config(shape)
    g.topk_groups = 1
    g.top_k = 8   # 1 group of 4 experts
    assert L.moe_route(ctypes.byref(g), 4, fake, fake, None, None, None, fake, fake, fake,
                       None, None) == -1
    # T beyond max_tokens
    w = moe.Weights(w_gate=0x1000, w13=0x1000, w2=0x1000, w13_scales=0x1000, w2_scales=0x1000)
    bad_layout = moe.Weights(w_gate=0x1000, w13=0x1000, w2=0x1000, w13_scales=0x1000,
                             w2_scales=0x1000, expert_layout=3)
    assert L.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(bad_layout), 4, fake, fake, 0,
                               fake, 1 << 40, None) == -1
    assert L.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(w), 38, fake, fake, 0, fake,
                               1 << 40, None) == -1
    assert L.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(w), 4, fake, fake, 0, fake,
                               16, None) == -3
    # the one-kernel expert FFN: enough scratch, known layouts
    r1 = moe.make_config(synth.CONFIGS["r1_decode_t128"])
    ffn = lambda c, groups, rows, nbytes, layout=0, lo=0: L.moe_expert_ffn(
        ctypes.byref(c), groups, rows, fake, fake, fake, fake, fake, fake, fake, layout, fake,
        fake, fake, fake, nbytes, lo, moe.ALL_ROWS, None, None)
    need = moe.expert_ffn_sched_bytes(257, 1152)
    assert need == 4 * (1 + 257 + 36)
    assert ffn(r1, 257, 1152, need - 4) == -3
    assert ffn(r1, 0, 10, need) == -1
    assert ffn(r1, 2000, 10, 1 << 20) == -2
    assert ffn(r1, 257, 1152, need, layout=5) == -1
    assert ffn(r1, 257, 1152, need, lo=-3) == -1
    assert L.moe_expert_ffn(ctypes.byref(r1), 257, 1152, P(0x1001), fake, fake, fake, fake, fake,
                            fake, 0, fake, fake, fake, fake, need, 0, moe.ALL_ROWS, None,
                            None) == -1
    assert L.moe_expert_ffn(ctypes.byref(r1), 257, 0, None, None, None, None, None, None, None,
                            0, None, None, None, None, 0, 0, moe.ALL_ROWS, None, None) == 0
    # the experts' FFN with the layer's choice of kernels: the same checks
    fwd = lambda c, groups, rows, nbytes, layout=0: L.moe_experts_forward(
        ctypes.byref(c), groups, rows, fake, fake, fake, fake, fake, fake, fake, layout, fake,
        fake, fake, fake, nbytes, None, None)
    assert fwd(r1, 257, 1152, need - 4) == -3
    assert fwd(r1, 0, 10, need) == -1
    assert fwd(r1, 2000, 10, 1 << 20) == -2
    assert fwd(r1, 257, 1152, need, layout=5) == -1
    assert L.moe_experts_forward(ctypes.byref(r1), 257, 1152, fake, None, fake, fake, fake, fake,
                                 fake, 0, fake, fake, fake, fake, need, None, None) == -1
    assert L.moe_experts_forward(ctypes.byref(r1), 257, 0, None, None, None, None, None, None,
                                 None, 0, None, None, None, None, 0, None, None) == 0
    # the read-stream utility: aligned, whole granules
    g = L.moe_stream_read_granule()
    assert g == 65536
    assert L.moe_stream_read(None, g, None, None) == -1
    assert L.moe_stream_read(P(0x1008), g, None, None) == -1
    assert L.moe_stream_read(fake, g + 16, None, None) == -1
    assert L.moe_stream_read(fake, 0, None, None) == 0
    # the FFN flag self-test needs its scratch
    n = L.moe_selftest_ffn_flag_timeout_scratch_bytes()
    assert 0 < n < (1 << 20)
    assert L.moe_selftest_ffn_flag_timeout(fake, n - 1, fake, None) == -1
    assert L.moe_selftest_ffn_flag_timeout(None, n, fake, None) == -1
    assert L.moe_selftest_ffn_flag_timeout(fake, n, None, None) == -1
    # zero tokens enqueue nothing and succeed
    assert L.moe_route(ctypes.byref(cfg), 0, None, None, None, None, None, None, None, None,
                       None, None) == 0
    assert L.moe_combine(ctypes.byref(cfg), 0, None, None, None, None, None, 0, None) == 0


@pytest.mark.parametrize("E,S", [(4, 2), (6, 3), (8, 2), (8, 4), (12, 3), (12, 4), (12, 6)])
def test_balance_is_optimal_on_tiny_counts(L, E, S):
    rng = np.random.default_rng(E * 7 + S)
    for trial in range(4):
        counts = rng.integers(0, 100, size=E)
        if trial == 0:
            counts = np.sort(counts)[::-1].copy()
        l2p, p2l, mom = moe.balance_permutation(counts, S)
        assert sorted(l2p.tolist()) == list(range(E))
        assert np.array_equal(p2l[l2p], np.arange(E))
        loads = balance.set_loads(counts, l2p, S)
        assert loads.max() == balance.optimum_max_load(counts.tolist(), S)
        assert abs(mom - balance.imbalance(loads)) < 1e-12
        m = E // S
        for s in range(S):   # logical ids ascend inside a set
            members = p2l[s * m:(s + 1) * m]
            assert list(members) == sorted(members)


@pytest.mark.parametrize("skew", [0.5, 1.0, 1.2])
def test_balance_on_skewed_large_counts_reaches_lower_bound(L, skew):
    rng = np.random.default_rng(11)
    counts = (1e4 / np.arange(1, 257) ** skew).astype(np.int64)[rng.permutation(256)]
    l2p, p2l, mom = moe.balance_permutation(counts, 8)
    loads = balance.set_loads(counts, l2p, 8)
    # no partition beats the mean, nor the heaviest expert with the 31 lightest others
    srt = np.sort(counts)
    lower = max(int(np.ceil(counts.sum() / 8)), int(counts.max() + srt[:31].sum()))
    assert lower <= loads.max() <= 1.01 * lower
    assert mom <= balance.imbalance(balance.contiguous_loads(counts, 8))


def test_balance_rejects_bad_arguments(L):
    c = np.ones(10, np.int64)
    out = np.empty(10, np.int32)
    assert L.expert_balance_permutation(c.ctypes.data, 10, 3, out.ctypes.data, out.ctypes.data,
                                        None) == -1
    c[2] = -1
    assert L.expert_balance_permutation(c.ctypes.data, 10, 5, out.ctypes.data, out.ctypes.data,
                                        None) == -1


def test_set_imbalance_of_a_given_permutation(L):
    """The library's set-imbalance figure against the oracle's definition, for
    the identity, random and balanced permutations; bad tables are rejected."""
    rng = np.random.default_rng(5)
    for E, S in ((8, 2), (32, 4), (256, 8)):
        counts = rng.integers(0, 1000, size=E)
        for l2p in (None, rng.permutation(E).astype(np.int32),
                    moe.balance_permutation(counts, S)[0]):
            ref_perm = np.arange(E) if l2p is None else l2p
            ref = balance.imbalance(balance.set_loads(counts, ref_perm, S))
            assert abs(moe.set_imbalance(counts, l2p, S) - ref) < 1e-12
    assert moe.set_imbalance(np.zeros(8, np.int64), None, 2) == 1.0
    c = np.ones(8, np.int64)
    bad = np.arange(8, dtype=np.int32)
    bad[3] = 2                                    # repeated id
    v = ctypes.c_double()
    assert L.expert_set_imbalance(c.ctypes.data, bad.ctypes.data, 8, 2, ctypes.byref(v)) == -1
    bad[3] = 8                                    # out of range
    assert L.expert_set_imbalance(c.ctypes.data, bad.ctypes.data, 8, 2, ctypes.byref(v)) == -1
    assert L.expert_set_imbalance(c.ctypes.data, None, 8, 3, ctypes.byref(v)) == -1


def test_source_slots_apply_a_new_permutation():
    rng = np.random.default_rng(21)
    E, G = 32, 34
    for _ in range(5):
        old_p2l = rng.permutation(E)
        old_l2p = np.argsort(old_p2l)
        new_p2l = rng.permutation(E)
        src = moe.source_slots(old_l2p, new_p2l, E, G)
        blocks_old = np.concatenate([old_p2l, np.arange(E, G)])   # logical id held per slot
        assert np.array_equal(blocks_old[src], np.concatenate([new_p2l, np.arange(E, G)]))


from oracle import affinity as oaff   # noqa: E402


@pytest.mark.parametrize("E,S", [(6, 2), (8, 2), (8, 4), (12, 3), (12, 4)])
def test_affinity_placement_is_optimal_on_tiny_inputs(L, E, S):
    rng = np.random.default_rng(E * 13 + S)
    for _ in range(3):
        counts = rng.integers(1, 40, size=E)
        A = np.triu(rng.integers(0, 12, size=(E, E)), 1)
        A = A + A.T
        l2p, p2l, mom, intra = moe.affinity_permutation(counts, A, S, 0.05)
        assert sorted(l2p.tolist()) == list(range(E)) and np.array_equal(p2l[l2p], np.arange(E))
        sets = oaff.set_of_logical(l2p, E, S)
        bound = oaff.load_bound(counts, S, balance.optimum_max_load(counts.tolist(), S), 0.05)
        assert balance.set_loads(counts, l2p, S).max() <= bound
        assert oaff.intra_affinity(A, sets) == oaff.optimum_affinity(counts, A, S, bound)
        assert abs(intra - oaff.intra_affinity(A, sets) / oaff.total_affinity(A)) < 1e-12


def test_affinity_placement_recovers_co_selected_clusters(L):
    rng = np.random.default_rng(3)
    E, S, k, T = 64, 8, 4, 4000
    hidden = rng.permutation(E).reshape(S, E // S)      # 8 clusters under a random numbering
    ids = []
    for t in range(T):
        c = hidden[rng.integers(S)]
        pick = list(rng.choice(c, k - 1, replace=False)) + [int(rng.integers(E))]
        while len(set(pick)) < k:
            pick[-1] = int(rng.integers(E))
        ids.append(pick)
    ids = np.array(ids)
    counts = np.bincount(ids.reshape(-1), minlength=E)
    A = oaff.coactivation_n(ids, E)
    l2p_b, _, mom_b = moe.balance_permutation(counts, S)
    l2p_a, _, mom_a, intra = moe.affinity_permutation(counts, A, S, 0.05)
    sets_contig = np.arange(E) // (E // S)
    m_contig = oaff.mean_sets_per_token(ids, sets_contig)
    m_bal = oaff.mean_sets_per_token(ids, oaff.set_of_logical(l2p_b, E, S))
    m_aff = oaff.mean_sets_per_token(ids, oaff.set_of_logical(l2p_a, E, S))
    planted = np.zeros(E, np.int64)
    for s in range(S):
        planted[hidden[s]] = s
    m_planted = oaff.mean_sets_per_token(ids, planted)
    # within 15% of the planted clustering, far below the load-only layouts
    assert m_aff <= 1.15 * m_planted and m_aff < 0.7 * min(m_contig, m_bal)
    assert intra >= 0.85 * oaff.intra_affinity(A, planted) / oaff.total_affinity(A)
    assert mom_a <= max(mom_b, 1.05) + 1e-12
    assert oaff.intra_affinity(A, oaff.set_of_logical(l2p_a, E, S)) >= \
        oaff.intra_affinity(A, oaff.set_of_logical(l2p_b, E, S))


def test_affinity_placement_rejects_bad_matrices(L):
    c = np.ones(8, np.int64)
    A = np.zeros((8, 8), np.int64)
    A[0, 1] = 3                                          # not symmetric
    out = np.empty(8, np.int32)
    assert L.expert_affinity_permutation(c.ctypes.data, A.ctypes.data, 8, 2, ctypes.c_double(0.05),
                                         out.ctypes.data, out.ctypes.data, None, None) == -1
