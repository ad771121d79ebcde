"""The benchmark's byte accounting on the CPU: the per-expert figure of the R1
layer, the method's bytes against this path's own (which add fp32
intermediates), and the share of weights at decode."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_r1_expert_bytes():
    # gate/up [4096, 7168] and down [7168, 2048] e4m3 codes plus one fp32 scale
    # per 128 x 128 block: 44,040,192 code bytes and 10,752 scale bytes
    w13, w2 = bench.expert_weight_bytes(synth.CONFIGS["r1_decode_t128"])
    assert (w13, w2) == (29_360_128 + 7_168, 14_680_064 + 3_584)
    assert w13 + w2 == 44_040_192 + 10_752


def _offsets(shape, active):
    rows = shape.tokens * (shape.top_k + shape.num_shared)
    counts = np.zeros(shape.groups, dtype=np.int64)
    counts[:active] = rows // active
    counts[0] += rows - counts.sum()
    return np.concatenate([[0], np.cumsum(counts)])


def test_method_bytes_below_path_bytes_and_weights_dominate_decode():
    for name in ("r1_decode_t128", "r1_zipf_t1024", "r1_prefill_t4096", "v2lite_bf16",
                 "tiny_bf16"):
        s = synth.CONFIGS[name]
        per, active, _ = bench.path_bytes(s, _offsets(s, s.groups))
        m = bench.method_bytes(s, active)
        assert 0 < m <= sum(per.values())
    s = synth.CONFIGS["r1_decode_t128"]
    w13, w2 = bench.expert_weight_bytes(s)
    m = bench.method_bytes(s, 250)
    assert 250 * (w13 + w2) < m < 1.01 * 250 * (w13 + w2) + 2 * s.num_experts * s.hidden


def test_wide_path_intermediates_not_counted():
    # at 4096 tokens the path's fp32 Y (written and read) is its own choice:
    # the method counts Y as bf16, so the path moves at least 4 bytes more per
    # element of Y; the wide path keeps no fp32 gate/up rows (its gate/up
    # GEMM writes FP8 h directly)
    s = synth.CONFIGS["r1_prefill_t4096"]
    per, active, _ = bench.path_bytes(s, _offsets(s, s.groups))
    rows = s.tokens * (s.top_k + s.num_shared)
    y_extra = 4 * rows * s.hidden
    gate_up_rows = 2 * rows * 2 * s.inter * 4
    diff = sum(per.values()) - bench.method_bytes(s, active)
    assert y_extra < diff < y_extra + gate_up_rows / 2
    assert "silu_mul" not in per and "gemm_gate_up_swiglu" in per


def test_weights_that_fit_in_l2_are_rotated():
    """Layers whose expert weights fit in L2 are timed over enough copies that
    two uses of one copy are at least 2.5 L2 capacities apart; the R1 and
    V2-Lite layers (far beyond L2) use one copy and say so in their config."""
    for name in ("r1_decode_t128", "r1_zipf_t1024", "r1_prefill_t4096", "v2lite_bf16"):
        s = synth.CONFIGS[name]
        assert bench.l2_rotation(s) == 1
        assert bench.l2_note(s).startswith("inputs larger than L2 (expert weights streamed")
    s = synth.CONFIGS["tiny_bf16"]
    r = bench.l2_rotation(s)
    w13, w2 = bench.expert_weight_bytes(s)
    per_layer = s.groups * (w13 + w2)
    assert per_layer < bench.L2_BYTES                    # 53.5 MB: the case this is for
    assert (r - 1) * per_layer >= 2.5 * bench.L2_BYTES   # others' weights in between
    assert (r - 2) * per_layer < 2.5 * bench.L2_BYTES    # and no more copies than that
    assert f"{r} copies" in bench.l2_note(s)
