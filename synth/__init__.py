"""Seeded synthetic workloads of the MoE decode layer.

This module only draws inputs: shapes, random numbers and the storage
formats the layer consumes.  It computes no step of the layer; the CUDA
path and the CPU oracle both take its tensors as given.

Workload shapes (the pages' model is DeepSeek-R1; Moreh report "21K output
tokens/s DeepSeek inference on MI300X with Expert Parallelism", section
"Parallelisation": 256 routed experts, 8 active per token, one shared
expert):

  tiny_bf16        64 tokens, hidden 1024, 16 experts, top-4 softmax
                   (renormalised), 1 shared expert, intermediate 512, BF16
  v2lite_bf16      256 tokens, hidden 2048, 64 experts, top-6 softmax (not
                   renormalised), 2 shared experts, intermediate 1408, BF16
  r1_decode_t128   128 tokens, hidden 7168, 256 experts + 1 shared,
                   intermediate 2048, FP8 e4m3 weights with 128x128 fp32
                   block scales, sigmoid + bias N(0, 0.01), 8 groups, top-4
                   groups by top-2 sum, top-8, normalised x 2.5
  r1_zipf_t1024    the same layer at 1024 tokens with Zipf(1.0)-skewed
                   expert popularity and a balanced expert permutation
  r1_prefill_t4096 the same layer at 4096 tokens, uniform routing

Values: x ~ N(0, 1) as bf16; gate ~ N(0, 0.02) as bf16; expert weights ~
N(0, 0.02) (BF16 layers: rounded to bf16; FP8 layers: block-quantised with
torch's own float8_e4m3fn cast, scale = block amax / 448).  Each tensor has
its own generator seeded with seed * 16 + tensor id.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class MoEShape:
    name: str
    tokens: int
    hidden: int
    inter: int
    num_experts: int
    num_shared: int
    top_k: int
    num_groups: int = 1
    topk_groups: int = 1
    group_topn: int = 1
    scoring: str = "softmax"       # "softmax" | "sigmoid"
    norm_topk: bool = True
    routed_scaling: float = 1.0
    dtype: str = "bf16"            # "bf16" | "fp8"
    bias_std: float | None = None  # per-expert selection bias (sigmoid)
    zipf_s: float | None = None    # logit offset -s*ln(rank) over a seeded order
    balanced_perm: bool = False    # route through a balanced expert permutation
    num_sets: int = 8              # sets of the balanced permutation

    @property
    def groups(self) -> int:
        return self.num_experts + self.num_shared

    def with_tokens(self, T: int) -> "MoEShape":
        return dataclasses.replace(self, tokens=T)


_R1 = dict(hidden=7168, inter=2048, num_experts=256, num_shared=1, top_k=8,
           num_groups=8, topk_groups=4, group_topn=2, scoring="sigmoid",
           norm_topk=True, routed_scaling=2.5, dtype="fp8", bias_std=0.01)

CONFIGS = {
    "tiny_bf16": MoEShape("tiny_bf16", tokens=64, hidden=1024, inter=512,
                          num_experts=16, num_shared=1, top_k=4,
                          scoring="softmax", norm_topk=True),
    "v2lite_bf16": MoEShape("v2lite_bf16", tokens=256, hidden=2048, inter=1408,
                            num_experts=64, num_shared=2, top_k=6,
                            scoring="softmax", norm_topk=False),
    "r1_decode_t128": MoEShape("r1_decode_t128", tokens=128, **_R1),
    "r1_zipf_t1024": MoEShape("r1_zipf_t1024", tokens=1024, zipf_s=1.0,
                              balanced_perm=True, **_R1),
    "r1_prefill_t4096": MoEShape("r1_prefill_t4096", tokens=4096, **_R1),
    # four times the prefill-sized batch: about 576 rows per routed expert,
    # the regime where the layer's FLOPs start to weigh against its bytes
    "r1_prefill_t16384": MoEShape("r1_prefill_t16384", tokens=16384, **_R1),
    # R1-shaped layers small enough for the oracle in seconds: several tiles
    # in every dimension and ragged tails (37 tokens, 3 k-blocks in the
    # down projection).
    "r1_mini": MoEShape("r1_mini", tokens=37, hidden=1024, inter=384,
                        num_experts=32, num_shared=1, top_k=8, num_groups=8,
                        topk_groups=4, group_topn=2, scoring="sigmoid",
                        norm_topk=True, routed_scaling=2.5, dtype="fp8",
                        bias_std=0.01),
    "r1_mini_zipf": MoEShape("r1_mini_zipf", tokens=53, hidden=1024, inter=384,
                             num_experts=32, num_shared=1, top_k=8, num_groups=8,
                             topk_groups=4, group_topn=2, scoring="sigmoid",
                             norm_topk=True, routed_scaling=2.5, dtype="fp8",
                             bias_std=0.01, zipf_s=1.0, balanced_perm=True,
                             num_sets=4),
    # as r1_mini with a 512-wide intermediate (the size the one-kernel expert
    # FFN takes) and Zipf-skewed routing, so hot experts span several 32-row
    # activation tiles
    "r1_mini_i512": MoEShape("r1_mini_i512", tokens=53, hidden=1024, inter=512,
                             num_experts=32, num_shared=1, top_k=8, num_groups=8,
                             topk_groups=4, group_topn=2, scoring="sigmoid",
                             norm_topk=True, routed_scaling=2.5, dtype="fp8",
                             bias_std=0.01, zipf_s=1.0),
    "bf16_mini": MoEShape("bf16_mini", tokens=29, hidden=512, inter=384,
                          num_experts=8, num_shared=2, top_k=3,
                          scoring="softmax", norm_topk=True),
    # R1 hidden/intermediate sizes with 32 experts: a few GB on the device,
    # the cases kernel profiles are captured on (16 tokens: decode-sized
    # groups of a few rows, as in the 128-token, 256-expert layer).
    "r1_e32_t16": MoEShape("r1_e32_t16", tokens=16, hidden=7168, inter=2048,
                           num_experts=32, num_shared=1, top_k=8, num_groups=8,
                           topk_groups=4, group_topn=2, scoring="sigmoid",
                           norm_topk=True, routed_scaling=2.5, dtype="fp8",
                           bias_std=0.01),
    # about 128 rows per routed expert, as in the 4096-token, 256-expert layer
    "r1_e32_t512": MoEShape("r1_e32_t512", tokens=512, hidden=7168, inter=2048,
                            num_experts=32, num_shared=1, top_k=8, num_groups=8,
                            topk_groups=4, group_topn=2, scoring="sigmoid",
                            norm_topk=True, routed_scaling=2.5, dtype="fp8",
                            bias_std=0.01),
    "r1_e32_t128": MoEShape("r1_e32_t128", tokens=128, hidden=7168, inter=2048,
                            num_experts=32, num_shared=1, top_k=8, num_groups=8,
                            topk_groups=4, group_topn=2, scoring="sigmoid",
                            norm_topk=True, routed_scaling=2.5, dtype="fp8",
                            bias_std=0.01),
}

# tensor ids for per-tensor seeds
_TID = dict(x=0, wg=1, bias=2, w13=3, w2=4, zipf=5)


def _gen(seed: int, tid: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 16 + _TID[tid])
    return g


def _normal(shape, std, gen, device, dtype=torch.float32):
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=gen)
    return t.to(dtype)


def block_quantize_e4m3(w: torch.Tensor):
    """[..., N, K] fp32 -> (e4m3 codes as uint8, fp32 scales [..., N/128, K/128]).

    Storage-format preparation of synthetic weights: scale = amax/448 per
    128x128 block, codes from torch's float8_e4m3fn cast.
    """
    *lead, N, K = w.shape
    b = w.reshape(*lead, N // 128, 128, K // 128, 128)
    amax = b.abs().amax(dim=(-3, -1))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (b / scale[..., :, None, :, None]).clamp(-448.0, 448.0)
    q = q.to(torch.float8_e4m3fn).reshape(*lead, N, K).view(torch.uint8)
    return q, scale.to(torch.float32).contiguous()


def zipf_logit_offset(cfg: MoEShape, seed: int, device) -> torch.Tensor:
    """-s * ln(rank_e) with rank_e = order_e + 1 for a seeded permutation."""
    g = _gen(seed, "zipf", "cpu")
    order = torch.randperm(cfg.num_experts, generator=g)
    rank = order.to(torch.float64) + 1.0
    return (-cfg.zipf_s * torch.log(rank)).to(torch.float32).to(device)


def make_inputs(cfg: MoEShape, seed: int = 0, device="cpu") -> dict:
    """All tensors of one workload, on `device`, in the layer's formats.

    Keys: x [T,H] bf16; wg [E,H] bf16 (logical order); e_bias [E] fp32 or
    None; logit_offset [E] fp32 or None; w13 [G,2I,H], w2 [G,H,I] (bf16, or
    uint8 e4m3 codes); w13_s [G,2I/128,H/128], w2_s [G,H/128,I/128] fp32
    (FP8 only).  Expert weights are in logical order, shared experts last.
    """
    T, H, I, E, G = cfg.tokens, cfg.hidden, cfg.inter, cfg.num_experts, cfg.groups
    out = {}
    out["x"] = _normal((T, H), 1.0, _gen(seed, "x", device), device, torch.bfloat16)
    out["wg"] = _normal((E, H), 0.02, _gen(seed, "wg", device), device, torch.bfloat16)
    out["e_bias"] = (_normal((E,), cfg.bias_std, _gen(seed, "bias", device), device)
                     if cfg.bias_std else None)
    out["logit_offset"] = zipf_logit_offset(cfg, seed, device) if cfg.zipf_s else None
    g13, g2 = _gen(seed, "w13", device), _gen(seed, "w2", device)
    if cfg.dtype == "bf16":
        out["w13"] = _normal((G, 2 * I, H), 0.02, g13, device, torch.bfloat16)
        out["w2"] = _normal((G, H, I), 0.02, g2, device, torch.bfloat16)
        out["w13_s"] = out["w2_s"] = None
    else:
        w13 = torch.empty((G, 2 * I, H), dtype=torch.uint8, device=device)
        w2 = torch.empty((G, H, I), dtype=torch.uint8, device=device)
        s13 = torch.empty((G, 2 * I // 128, H // 128), dtype=torch.float32, device=device)
        s2 = torch.empty((G, H // 128, I // 128), dtype=torch.float32, device=device)
        for e in range(G):   # one expert at a time bounds the fp32 staging
            w13[e], s13[e] = block_quantize_e4m3(_normal((2 * I, H), 0.02, g13, device))
            w2[e], s2[e] = block_quantize_e4m3(_normal((H, I), 0.02, g2, device))
        out.update(w13=w13, w2=w2, w13_s=s13, w2_s=s2)
    return out


def relayout_experts(inputs: dict, cfg: MoEShape, phys2log) -> dict:
    """Expert weights in physical order: slot p holds logical expert phys2log[p].

    Shared experts stay last.  Gate rows, bias and offsets stay logical.
    """
    idx = torch.as_tensor(list(phys2log) + list(range(cfg.num_experts, cfg.groups)),
                          dtype=torch.long, device=inputs["w13"].device)
    out = dict(inputs)
    for key in ("w13", "w2", "w13_s", "w2_s"):
        if inputs.get(key) is not None:
            out[key] = inputs[key].index_select(0, idx)
    return out


def to_numpy(inputs: dict, log2phys=None) -> dict:
    """The oracle's view: bf16 as uint16 bit patterns, e4m3 as uint8 codes."""
    def bits(t):
        return t.contiguous().view(torch.int16).cpu().numpy().view("uint16")

    out = dict(x_bits=bits(inputs["x"]), wg_bits=bits(inputs["wg"]))
    for key in ("e_bias", "logit_offset", "w13_s", "w2_s"):
        v = inputs.get(key)
        out[key] = None if v is None else v.contiguous().cpu().numpy()
    for key in ("w13", "w2"):
        v = inputs[key]
        out[key] = bits(v) if v.dtype == torch.bfloat16 else v.contiguous().cpu().numpy()
    out["log2phys"] = None if log2phys is None else \
        torch.as_tensor(log2phys).to(torch.int32).cpu().numpy()
    return out


def weight_bytes_per_expert(cfg: MoEShape) -> int:
    H, I = cfg.hidden, cfg.inter
    if cfg.dtype == "fp8":
        return 3 * H * I + 4 * (2 * I // 128) * (H // 128) + 4 * (H // 128) * (I // 128)
    return 2 * 3 * H * I


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = ["MoEShape", "CONFIGS", "make_inputs", "relayout_experts", "to_numpy",
           "block_quantize_e4m3", "zipf_logit_offset", "weight_bytes_per_expert",
           "ceil_div", "math"]
