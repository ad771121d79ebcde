"""moe_expert_layer_07_gb300: the DeepSeek-style MoE decode layer on one GB300.

A thin ctypes binding of the C-ABI library libmoe_gb300.so (declared in
include/moe_gb300.h).  The functions here only marshal arguments: every step
of the layer runs in the library's CUDA kernels.  PyTorch supplies device
memory and streams.  If the library has not been built, importing the
compute entry points raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB as LIB_PATH

__all__ = ["Config", "Weights", "WsLayout", "lib", "make_config", "route", "route_quantize",
           "act_requant",
           "permute", "permute_workspace_size", "permute_static_scratch", "grouped_gemm", "combine", "layer_forward",
           "workspace_size", "workspace_layout", "get_device_status", "status_string",
           "last_error_detail", "stream_read", "stream_read_granule",
           "balance_permutation", "set_imbalance", "rebalance_due", "layer_kernel_count", "MoELayer", "MoEError",
           "count_expert_rows", "relayout_experts", "source_slots", "ExpertRebalancer",
           "count_coactivation", "affinity_permutation", "grouped_gemm_swiglu",
           "expert_ffn", "experts_forward", "expert_ffn_sched_bytes", "pack_expert_weights", "LAYOUT_ROWS",
           "LAYOUT_TILES",
           "SOFTMAX", "SIGMOID", "BF16", "FP8", "OUT_F32", "OUT_BF16", "ACT_IDENTITY",
           "ACT_SILU_MUL"]

SOFTMAX, SIGMOID = 0, 1
BF16, FP8 = 0, 1
OUT_F32, OUT_BF16 = 0, 1
ACT_IDENTITY, ACT_SILU_MUL = 0, 1
DEV_BAD_EXPERT_ID, DEV_BAD_OFFSETS, DEV_TIMEOUT = 1, 2, 4
LAYOUT_ROWS, LAYOUT_TILES = 0, 1


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = f"{where}: {status_string(code)} ({code})"
        if code == -4:   # MOE_ERR_CUDA: add what the library saw fail
            msg += f" [{last_error_detail()}]"
        super().__init__(msg)
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("hidden", "inter", "num_experts", "num_shared", "top_k", "num_groups",
                 "topk_groups", "group_topn", "scoring", "norm_topk", "dtype", "max_tokens")] + \
               [("routed_scaling", ctypes.c_float)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_gate", "e_bias", "logit_offset", "log2phys", "w13", "w13_scales", "w2",
                 "w2_scales")] + [("expert_layout", ctypes.c_int32)]


class WsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("status", "logits", "topk_ids", "topk_w", "xq", "xs", "expert_offsets",
                 "src_of_row", "row_of_slot", "perm_scratch", "xp", "xp_scales", "gate_up",
                 "h", "h_scales", "y", "ffn_sched", "total")]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int32
_CP = ctypes.POINTER(Config)

_SIGS = {
    "moe_route": [_CP, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_act_requant": [_CP, _I, _I, _P, _P, _P, _P, _P],
    "moe_route_quantize": [_CP, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_permute_workspace_size": [_CP, _I, ctypes.POINTER(ctypes.c_size_t)],
    "moe_permute": [_CP, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _I, _P, _P],
    "moe_grouped_gemm_swiglu_gather": [_CP, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P, _I, _P,
                                       _P, _I, _I, _P, _P],
    "moe_grouped_gemm": [_CP, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _P, _P],
    "moe_combine": [_CP, _I, _P, _P, _P, _P, _P, _I, _P],
    "moe_workspace_size": [_CP, ctypes.POINTER(ctypes.c_size_t)],
    "moe_layer_forward": [_CP, ctypes.POINTER(Weights), _I, _P, _P, _I, _P, ctypes.c_size_t, _P],
    "moe_workspace_layout": [_CP, ctypes.POINTER(WsLayout)],
    "moe_get_device_status": [_P, ctypes.POINTER(ctypes.c_int32)],
    "moe_layer_kernel_count": [_CP, _I],
    "expert_balance_permutation": [_P, _I, _I, _P, _P, ctypes.POINTER(ctypes.c_double)],
    "expert_set_imbalance": [_P, _P, _I, _I, ctypes.POINTER(ctypes.c_double)],
    "moe_selftest_bounded_wait": [_P, ctypes.c_int64, _P, _P],
    "moe_permute_static_scratch": [_CP, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_count_expert_rows": [_CP, _P, _P, _P],
    "moe_grouped_gemm_swiglu": [_CP, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _P,
                                _P],
    "moe_pack_expert_weights": [_CP, _I, _I, _I, _P, _P, _P],
    "moe_count_coactivation": [_CP, _I, _P, _P, _P, _P],
    "expert_affinity_permutation": [_P, _P, _I, _I, ctypes.c_double, _P, _P,
                                    ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)],
    "moe_relayout_experts": [_P, _P, _P, _I, ctypes.c_int64, _P, _P],
    "moe_selftest_ffn_flag_timeout": [_P, ctypes.c_size_t, _P, _P],
    "moe_selftest_sigmoid": [_P, _I, _P, _P, _P, _P],
    "moe_expert_ffn": [_CP, _I, _I, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P,
                       ctypes.c_size_t, _I, _I, _P, _P],
    "moe_experts_forward": [_CP, _I, _I, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P,
                            ctypes.c_size_t, _P, _P],
    "moe_stream_read": [_P, ctypes.c_size_t, _P, _P],
}


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                              "(there is no non-CUDA fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.moe_permute_static_scratch_capacity.argtypes = []
        L.moe_permute_static_scratch_capacity.restype = ctypes.c_size_t
        L.moe_stream_read_granule.argtypes = []
        L.moe_stream_read_granule.restype = ctypes.c_size_t
        L.moe_expert_ffn_sched_bytes.argtypes = [_I, _I]
        L.moe_expert_ffn_sched_bytes.restype = ctypes.c_size_t
        L.moe_selftest_ffn_flag_timeout_scratch_bytes.argtypes = []
        L.moe_selftest_ffn_flag_timeout_scratch_bytes.restype = ctypes.c_size_t
        L.moe_status_string.argtypes = [ctypes.c_int32]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_last_error_detail.argtypes = []
        L.moe_last_error_detail.restype = ctypes.c_char_p
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def last_error_detail() -> str:
    """What the last MOE_ERR_CUDA on this thread failed at."""
    return lib().moe_last_error_detail().decode()


def _check(rc: int, where: str):
    if rc != 0:
        raise MoEError(rc, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


_RAW_STREAM = []


def _current_stream_handle():
    """torch's current CUDA stream as a cudaStream_t value.  The raw-handle
    query costs about 0.3 us against 3 us for torch.cuda.current_stream()
    (which builds a Stream object); the latter stays as the fallback."""
    import torch
    if not _RAW_STREAM:
        _RAW_STREAM.append(getattr(torch._C, "_cuda_getCurrentRawStream", None))
    raw = _RAW_STREAM[0]
    if raw is not None:
        return raw(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _stream(stream):
    if stream is None:
        return _current_stream_handle()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_config(shape, max_tokens: int | None = None) -> Config:
    """Config from any object with the layer's fields (e.g. synth.MoEShape)."""
    return Config(hidden=shape.hidden, inter=shape.inter, num_experts=shape.num_experts,
                  num_shared=shape.num_shared, top_k=shape.top_k, num_groups=shape.num_groups,
                  topk_groups=shape.topk_groups, group_topn=shape.group_topn,
                  scoring=SIGMOID if shape.scoring == "sigmoid" else SOFTMAX,
                  norm_topk=int(bool(shape.norm_topk)),
                  dtype=FP8 if shape.dtype == "fp8" else BF16,
                  max_tokens=shape.tokens if max_tokens is None else max_tokens,
                  routed_scaling=float(shape.routed_scaling))


def route(cfg: Config, T, x, w_gate, e_bias, logit_offset, log2phys, logits, topk_ids, topk_w,
          status=None, stream=None):
    _check(lib().moe_route(ctypes.byref(cfg), T, _ptr(x), _ptr(w_gate), _ptr(e_bias),
                           _ptr(logit_offset), _ptr(log2phys), _ptr(logits), _ptr(topk_ids),
                           _ptr(topk_w), _ptr(status), _stream(stream)), "moe_route")


def route_quantize(cfg: Config, T, x, w_gate, e_bias, logit_offset, log2phys, logits, topk_ids,
                   topk_w, xq, xs, status=None, stream=None):
    """moe_route and the FP8 quantisation of x in the selection kernel (FP8 layers)."""
    _check(lib().moe_route_quantize(ctypes.byref(cfg), T, _ptr(x), _ptr(w_gate), _ptr(e_bias),
                                    _ptr(logit_offset), _ptr(log2phys), _ptr(logits),
                                    _ptr(topk_ids), _ptr(topk_w), _ptr(xq), _ptr(xs),
                                    _ptr(status), _stream(stream)), "moe_route_quantize")


def act_requant(cfg: Config, mode, rows, inp, out, out_scales=None, rows_dev=None, stream=None):
    _check(lib().moe_act_requant(ctypes.byref(cfg), mode, rows, _ptr(rows_dev), _ptr(inp),
                                 _ptr(out), _ptr(out_scales), _stream(stream)), "moe_act_requant")


def permute_workspace_size(cfg: Config, T: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_permute_workspace_size(ctypes.byref(cfg), T, ctypes.byref(n)),
           "moe_permute_workspace_size")
    return n.value


def permute(cfg: Config, T, topk_ids, x_rows, x_scales, expert_offsets, src_of_row,
            row_of_slot, xp, xp_scales, ws, ws_bytes, status=None, stream=None,
            copy_max_group_rows=0x7FFFFFFF):
    _check(lib().moe_permute(ctypes.byref(cfg), T, _ptr(topk_ids), _ptr(x_rows), _ptr(x_scales),
                             _ptr(expert_offsets), _ptr(src_of_row), _ptr(row_of_slot),
                             _ptr(xp), _ptr(xp_scales), _ptr(ws), ws_bytes, copy_max_group_rows,
                             _ptr(status), _stream(stream)), "moe_permute")


def permute_static_scratch(cfg: Config, T, topk_ids, x_rows, x_scales, expert_offsets,
                           src_of_row, row_of_slot, xp, xp_scales, status=None, stream=None):
    """moe_permute with its scratch in the library's static device array, for
    callers that cannot allocate device memory (limits: include/moe_gb300.h)."""
    _check(lib().moe_permute_static_scratch(ctypes.byref(cfg), T, _ptr(topk_ids), _ptr(x_rows),
                                            _ptr(x_scales), _ptr(expert_offsets),
                                            _ptr(src_of_row), _ptr(row_of_slot), _ptr(xp),
                                            _ptr(xp_scales), _ptr(status), _stream(stream)),
           "moe_permute_static_scratch")


# group row window [min_group_rows, max_group_rows] of the expert entry points: all groups
ALL_ROWS = 0x7FFFFFFF


def grouped_gemm(cfg: Config, groups, n_out, k_dim, rows, a, a_scales, expert_offsets, w,
                 w_scales, c, c_dtype, status=None, stream=None, w_layout=None,
                 min_group_rows=0, max_group_rows=ALL_ROWS):
    _check(lib().moe_grouped_gemm(ctypes.byref(cfg), groups, n_out, k_dim, rows, _ptr(a),
                                  _ptr(a_scales), _ptr(expert_offsets), _ptr(w), _ptr(w_scales),
                                  LAYOUT_ROWS if w_layout is None else w_layout, _ptr(c),
                                  c_dtype, min_group_rows, max_group_rows, _ptr(status),
                                  _stream(stream)),
           "moe_grouped_gemm")


def grouped_gemm_swiglu(cfg: Config, groups, inter, k_dim, rows, a, a_scales, expert_offsets,
                        w13, w13_scales, h, h_scales, status=None, stream=None, w_layout=None,
                        min_group_rows=0, max_group_rows=ALL_ROWS):
    _check(lib().moe_grouped_gemm_swiglu(ctypes.byref(cfg), groups, inter, k_dim, rows, _ptr(a),
                                         _ptr(a_scales), _ptr(expert_offsets), _ptr(w13),
                                         _ptr(w13_scales),
                                         LAYOUT_ROWS if w_layout is None else w_layout, _ptr(h),
                                         _ptr(h_scales), min_group_rows, max_group_rows,
                                         _ptr(status), _stream(stream)),
           "moe_grouped_gemm_swiglu")


def grouped_gemm_swiglu_gather(cfg: Config, groups, inter, k_dim, rows, x_rows, x_scales, T,
                               src_of_row, expert_offsets, w13, w13_scales, h, h_scales,
                               status=None, stream=None, w_layout=None, min_group_rows=0,
                               max_group_rows=ALL_ROWS):
    """The gate/up GEMM with SwiGLU on rows gathered from the token rows of x (FP8)."""
    _check(lib().moe_grouped_gemm_swiglu_gather(
        ctypes.byref(cfg), groups, inter, k_dim, rows, _ptr(x_rows), _ptr(x_scales), T,
        _ptr(src_of_row), _ptr(expert_offsets), _ptr(w13), _ptr(w13_scales),
        LAYOUT_ROWS if w_layout is None else w_layout, _ptr(h), _ptr(h_scales), min_group_rows,
        max_group_rows, _ptr(status), _stream(stream)), "moe_grouped_gemm_swiglu_gather")


def pack_expert_weights(cfg: Config, w, out=None, stream=None):
    """W [groups, N, K] row-major -> the same tensor shape in MOE_LAYOUT_TILES
    (a new tensor unless `out` is given)."""
    import torch
    out = torch.empty_like(w) if out is None else out
    G, N, K = w.shape
    _check(lib().moe_pack_expert_weights(ctypes.byref(cfg), G, N, K, _ptr(w), _ptr(out),
                                         _stream(stream)), "moe_pack_expert_weights")
    return out


def expert_ffn_sched_bytes(groups, rows) -> int:
    """Bytes of the scheduler scratch moe_expert_ffn needs."""
    return int(lib().moe_expert_ffn_sched_bytes(groups, rows))


def expert_ffn(cfg: Config, groups, rows, a, a_scales, expert_offsets, w13, w13_scales, w2,
               w2_scales, h, h_scales, y, sched, sched_bytes, status=None, stream=None,
               w_layout=None, min_group_rows=0, max_group_rows=ALL_ROWS):
    """Both expert GEMMs with SwiGLU between them, one persistent kernel (FP8 or BF16)."""
    _check(lib().moe_expert_ffn(ctypes.byref(cfg), groups, rows, _ptr(a), _ptr(a_scales),
                                _ptr(expert_offsets), _ptr(w13), _ptr(w13_scales), _ptr(w2),
                                _ptr(w2_scales), LAYOUT_ROWS if w_layout is None else w_layout,
                                _ptr(h), _ptr(h_scales), _ptr(y), _ptr(sched), sched_bytes,
                                min_group_rows, max_group_rows, _ptr(status), _stream(stream)),
           "moe_expert_ffn")


def experts_forward(cfg: Config, groups, rows, a, a_scales, expert_offsets, w13, w13_scales, w2,
                    w2_scales, h, h_scales, y, sched, sched_bytes, status=None, stream=None,
                    w_layout=None):
    """The experts' FFN with the kernels the layer would pick for this batch."""
    _check(lib().moe_experts_forward(ctypes.byref(cfg), groups, rows, _ptr(a), _ptr(a_scales),
                                     _ptr(expert_offsets), _ptr(w13), _ptr(w13_scales), _ptr(w2),
                                     _ptr(w2_scales), LAYOUT_ROWS if w_layout is None else w_layout,
                                     _ptr(h), _ptr(h_scales), _ptr(y), _ptr(sched), sched_bytes,
                                     _ptr(status), _stream(stream)), "moe_experts_forward")


def combine(cfg: Config, T, y, row_of_slot, topk_w, expert_offsets, out, out_dtype, stream=None):
    _check(lib().moe_combine(ctypes.byref(cfg), T, _ptr(y), _ptr(row_of_slot), _ptr(topk_w),
                             _ptr(expert_offsets), _ptr(out), out_dtype, _stream(stream)),
           "moe_combine")


def count_expert_rows(cfg: Config, expert_offsets, counts, stream=None):
    """counts[p] += rows of routed expert p (physical) in the batch behind expert_offsets."""
    _check(lib().moe_count_expert_rows(ctypes.byref(cfg), _ptr(expert_offsets), _ptr(counts),
                                       _stream(stream)), "moe_count_expert_rows")


def count_coactivation(cfg: Config, T, topk_ids, phys2log, coact, stream=None):
    """coact[a, b] += tokens selecting both logical experts a and b (device int64 [E, E])."""
    _check(lib().moe_count_coactivation(ctypes.byref(cfg), T, _ptr(topk_ids), _ptr(phys2log),
                                        _ptr(coact), _stream(stream)), "moe_count_coactivation")


def affinity_permutation(counts, coact, num_sets: int, load_slack: float = 0.05):
    """Host call: (log2phys, phys2log, max_over_mean, intra_fraction)."""
    import numpy as np
    c = np.ascontiguousarray(counts, dtype=np.int64)
    A = np.ascontiguousarray(coact, dtype=np.int64)
    E = len(c)
    l2p = np.empty(E, dtype=np.int32)
    p2l = np.empty(E, dtype=np.int32)
    mom, intra = ctypes.c_double(), ctypes.c_double()
    _check(lib().expert_affinity_permutation(c.ctypes.data, A.ctypes.data, E, num_sets,
                                             float(load_slack), l2p.ctypes.data, p2l.ctypes.data,
                                             ctypes.byref(mom), ctypes.byref(intra)),
           "expert_affinity_permutation")
    return l2p, p2l, mom.value, intra.value


def relayout_experts(src, dst, src_slot, groups, block_bytes, status=None, stream=None):
    """dst block p = src block src_slot[p] (device tensors/pointers)."""
    _check(lib().moe_relayout_experts(_ptr(src), _ptr(dst), _ptr(src_slot), groups, block_bytes,
                                      _ptr(status), _stream(stream)), "moe_relayout_experts")


def source_slots(old_log2phys, new_phys2log, num_experts: int, groups: int):
    """Re-layout table: new physical slot p takes the block now at
    old_log2phys[new_phys2log[p]]; shared experts (p >= num_experts) stay."""
    import numpy as np
    old = np.asarray(old_log2phys, dtype=np.int64)
    new = np.asarray(new_phys2log, dtype=np.int64)
    return np.concatenate([old[new], np.arange(num_experts, groups)]).astype(np.int32)


def stream_read(src, nbytes: int, status=None, stream=None):
    """Reads nbytes of device memory at src through shared memory (a timing utility)."""
    _check(lib().moe_stream_read(_ptr(src), nbytes, _ptr(status), _stream(stream)),
           "moe_stream_read")


def stream_read_granule() -> int:
    return int(lib().moe_stream_read_granule())


def workspace_size(cfg: Config) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def workspace_layout(cfg: Config) -> WsLayout:
    L = WsLayout()
    _check(lib().moe_workspace_layout(ctypes.byref(cfg), ctypes.byref(L)), "moe_workspace_layout")
    return L


def layer_kernel_count(cfg: Config, T: int) -> int:
    return int(lib().moe_layer_kernel_count(ctypes.byref(cfg), T))


def layer_forward(cfg: Config, weights: Weights, T, x, out, out_dtype, ws, ws_bytes, stream=None):
    _check(lib().moe_layer_forward(ctypes.byref(cfg), ctypes.byref(weights), T, _ptr(x), _ptr(out),
                                   out_dtype, _ptr(ws), ws_bytes, _stream(stream)),
           "moe_layer_forward")


def get_device_status(ws) -> int:
    v = ctypes.c_int32()
    lib().moe_get_device_status(_ptr(ws), ctypes.byref(v))
    return v.value


def balance_permutation(counts, num_sets: int):
    """Host call: (log2phys, phys2log, max_over_mean) from per-expert counts."""
    import numpy as np
    c = np.ascontiguousarray(counts, dtype=np.int64)
    E = len(c)
    l2p = np.empty(E, dtype=np.int32)
    p2l = np.empty(E, dtype=np.int32)
    mom = ctypes.c_double()
    _check(lib().expert_balance_permutation(c.ctypes.data, E, num_sets, l2p.ctypes.data,
                                            p2l.ctypes.data, ctypes.byref(mom)),
           "expert_balance_permutation")
    return l2p, p2l, mom.value


def set_imbalance(counts, log2phys, num_sets: int) -> float:
    """Host call: largest set load / mean set load of a permutation."""
    import numpy as np
    c = np.ascontiguousarray(counts, dtype=np.int64)
    l2p = None if log2phys is None else np.ascontiguousarray(log2phys, dtype=np.int32)
    v = ctypes.c_double()
    _check(lib().expert_set_imbalance(c.ctypes.data, None if l2p is None else l2p.ctypes.data,
                                      len(c), num_sets, ctypes.byref(v)), "expert_set_imbalance")
    return v.value


def rebalance_due(batches: int, every, max_imbalance, check_every: int, imbalance) -> bool:
    """The periodic re-balancing policy: due after `every` counted batches, or,
    with max_imbalance set, when imbalance() (called only on every
    check_every-th batch) exceeds it."""
    if every is not None and batches >= every:
        return True
    if max_imbalance is not None and batches % check_every == 0:
        return imbalance() > max_imbalance
    return False


class MoELayer:
    """One MoE layer: device weights, a workspace and the forward call.

    weights: dict of device tensors with keys wg, e_bias, logit_offset, w13,
    w13_s, w2, w2_s (expert weights in physical order, shared experts last)
    and optionally log2phys (int32) and expert_layout (LAYOUT_*, default
    row-major).  With pack_weights (the default) row-major expert weights are
    packed once into 128 x 128-byte tiles (MOE_LAYOUT_TILES), which the
    tensor-core kernels stream faster; the caller's tensors are not changed.
    """

    def __init__(self, shape, weights: dict, max_tokens: int | None = None, log2phys=None,
                 pack_weights: bool = True):
        import torch
        self.cfg = make_config(shape, max_tokens)
        self.shape = shape
        weights = dict(weights)
        if pack_weights and weights.get("expert_layout", LAYOUT_ROWS) == LAYOUT_ROWS:
            weights["w13"] = pack_expert_weights(self.cfg, weights["w13"])
            weights["w2"] = pack_expert_weights(self.cfg, weights["w2"])
            weights["expert_layout"] = LAYOUT_TILES
        self.set_weights(weights, log2phys)
        self.ws_bytes = workspace_size(self.cfg)
        self.layout = workspace_layout(self.cfg)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=weights["w13"].device)

    def set_weights(self, weights: dict, log2phys=None):
        """Point the layer at (new) device weights; keeps references alive."""
        import torch
        keep = dict(weights)
        if log2phys is not None:
            keep["log2phys"] = torch.as_tensor(log2phys, dtype=torch.int32,
                                               device=weights["w13"].device)
        else:
            keep.pop("log2phys", None)
        self._keep = keep
        keep.setdefault("expert_layout", LAYOUT_ROWS)
        self.expert_layout = keep["expert_layout"]
        self.weights = Weights(w_gate=_ptr(keep["wg"]), e_bias=_ptr(keep.get("e_bias")),
                               logit_offset=_ptr(keep.get("logit_offset")),
                               log2phys=_ptr(keep.get("log2phys")), w13=_ptr(keep["w13"]),
                               w13_scales=_ptr(keep.get("w13_s")), w2=_ptr(keep["w2"]),
                               w2_scales=_ptr(keep.get("w2_s")),
                               expert_layout=self.expert_layout)

    def forward(self, x, out, out_dtype=OUT_F32, T=None, stream=None):
        """x bf16 [T, H] and out [T, H] (fp32 or bf16) device tensors."""
        T = x.shape[0] if T is None else T
        layer_forward(self.cfg, self.weights, T, x, out, out_dtype, self.ws, self.ws_bytes, stream)
        return out

    def forward_host(self, x_host, out_host, x_dev, out_dev, out_dtype=OUT_F32, stream=None):
        """End to end from pinned host memory: copy x in, run, copy out back."""
        x_dev.copy_(x_host, non_blocking=True)
        self.forward(x_dev, out_dev, out_dtype, stream=stream)
        out_host.copy_(out_dev, non_blocking=True)
        return out_host

    def view(self, name, dtype, shape):
        """A tensor view of one intermediate inside the workspace."""
        import math
        import torch
        off = getattr(self.layout, name)
        n = math.prod(shape)
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype).view(*shape)

    def status(self) -> int:
        return get_device_status(self.ws)


class ExpertRebalancer:
    """Continuous load balancing of one MoELayer: counts each batch's rows per
    expert on the device, and -- on request (rebalance) or by the periodic
    policy of step() -- derives a new balanced permutation from the counts
    and re-lays the expert weights into it on a side stream (report "21K
    output tokens/s DeepSeek inference on MI300X with Expert Parallelism",
    section "Load balancing across GPUs": activation frequencies are
    re-measured at regular intervals and the permutation renewed).

    The layer's output does not change when its experts move: routing is
    defined on logical ids and each expert's rows are computed the same way
    wherever its weights sit.
    """

    _BLOCKS = ("w13", "w13_s", "w2", "w2_s")

    def __init__(self, layer: MoELayer, num_sets: int, affinity_slack: float | None = None,
                 every: int | None = None, max_imbalance: float | None = None,
                 check_every: int = 1):
        """affinity_slack: None for plain balancing; a value (e.g. 0.05) to
        also track co-activation and place co-selected experts together with
        set totals allowed up to (1 + slack) x the mean.

        The periodic policy of step() (the report's re-measurement "at
        regular intervals"): every -- re-balance after this many counted
        batches; max_imbalance -- re-balance as soon as the counts since the
        last re-balance put the busiest set above this multiple of the mean
        under the current permutation, looked at every check_every batches
        (the look reads the counts to the host)."""
        import numpy as np
        import torch
        if every is not None and every < 1:
            raise ValueError("every must be at least 1")
        if max_imbalance is not None and max_imbalance < 1.0:
            raise ValueError("max_imbalance is a max / mean ratio, at least 1")
        if check_every < 1:
            raise ValueError("check_every must be at least 1")
        self.layer = layer
        self.num_sets = num_sets
        self.affinity_slack = affinity_slack
        self.every, self.max_imbalance, self.check_every = every, max_imbalance, check_every
        self.batches = 0          # batches counted since the last re-balance
        self.history = []         # (batches counted, imbalance before, after) per re-balance
        s = layer.shape
        dev = layer._keep["w13"].device
        self.counts = torch.zeros(s.num_experts, dtype=torch.int64, device=dev)
        self.coact = (torch.zeros((s.num_experts, s.num_experts), dtype=torch.int64, device=dev)
                      if affinity_slack is not None else None)
        l2p = layer._keep.get("log2phys")
        self.log2phys = (np.arange(s.num_experts, dtype=np.int32) if l2p is None
                         else l2p.cpu().numpy().astype(np.int32))
        self._p2l = torch.as_tensor(np.argsort(self.log2phys).astype(np.int32), device=dev)
        self.side = torch.cuda.Stream(device=dev)
        self.last_intra_fraction = None

    def observe(self, T=None, stream=None):
        """Add the last forward's rows per expert (and co-activation), enqueued."""
        lay = self.layer
        count_expert_rows(lay.cfg, lay.ws.data_ptr() + lay.layout.expert_offsets, self.counts,
                          stream)
        if self.coact is not None:
            count_coactivation(lay.cfg, lay.shape.tokens if T is None else T,
                               lay.ws.data_ptr() + lay.layout.topk_ids, self._p2l, self.coact,
                               stream)

    def logical_counts(self):
        """Rows per logical expert since the last re-balance (synchronous read)."""
        return self.counts.cpu().numpy()[self.log2phys]

    def current_imbalance(self) -> float:
        """Busiest set / mean set of the counts since the last re-balance under
        the current permutation (synchronous read)."""
        return set_imbalance(self.logical_counts(), self.log2phys, self.num_sets)

    def step(self, T=None, stream=None):
        """Counts the batch the layer just ran and applies the periodic policy
        given at construction.  Returns (imbalance before, after) when it
        re-balanced, else None."""
        self.observe(T, stream)
        self.batches += 1
        if not rebalance_due(self.batches, self.every, self.max_imbalance, self.check_every,
                             self.current_imbalance):
            return None
        n = self.batches
        before, after = self.rebalance()
        self.history.append((n, before, after))
        return before, after

    def rebalance(self, counts=None):
        """New permutation from the counts; weights re-laid on a side stream,
        then the layer switches to them (the current stream waits for the copy).
        Returns (set imbalance before, after)."""
        import numpy as np
        import torch
        lay, s = self.layer, self.layer.shape
        c = self.logical_counts() if counts is None else np.asarray(counts, np.int64)
        before = set_imbalance(c, self.log2phys, self.num_sets)
        if self.coact is not None:
            new_l2p, new_p2l, after, self.last_intra_fraction = affinity_permutation(
                c, self.coact.cpu().numpy(), self.num_sets, self.affinity_slack)
        else:
            new_l2p, new_p2l, after = balance_permutation(c, self.num_sets)
        src = torch.as_tensor(source_slots(self.log2phys, new_p2l, s.num_experts, s.groups),
                              device=self.counts.device)
        cur = torch.cuda.current_stream(self.counts.device)
        self.side.wait_stream(cur)
        new_w = dict(lay._keep)
        self._events = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        self.relayout_bytes = 0
        with torch.cuda.stream(self.side):
            self._events[0].record(self.side)
            for key in self._BLOCKS:
                t = lay._keep.get(key)
                if t is None:
                    continue
                out = torch.empty_like(t)
                relayout_experts(t, out, src, s.groups, t[0].numel() * t.element_size(),
                                 stream=self.side)
                new_w[key] = out
                self.relayout_bytes += 2 * t.numel() * t.element_size()
            self._events[1].record(self.side)
            self.counts.zero_()
            if self.coact is not None:
                self.coact.zero_()
        cur.wait_stream(self.side)
        self.batches = 0
        for key in self._BLOCKS:   # old buffers stay valid until the copy is done
            if lay._keep.get(key) is not None:
                lay._keep[key].record_stream(self.side)
        new_w.pop("log2phys", None)
        lay.set_weights(new_w, new_l2p)
        self.log2phys = new_l2p.astype(np.int32)
        self._p2l = torch.as_tensor(new_p2l.astype(np.int32), device=self.counts.device)
        return before, float(after)

    def last_relayout_ms(self):
        """Device time of the last re-layout (waits for it)."""
        self._events[1].synchronize()
        return self._events[0].elapsed_time(self._events[1])
