"""Pins of the oracle's number formats (CPU only).

e4m3 and bf16 rounding are checked against torch's own casts (a library used
as a check), and the per-128 group quantiser against closed-form bounds.
"""
import numpy as np
import pytest
import torch

from oracle import quant


def _torch_e4m3_codes(v32):
    return torch.from_numpy(np.asarray(v32, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = quant.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_torch_on_every_bf16_value_in_range():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) <= 464.0)]
    assert np.array_equal(quant.e4m3_encode(v), _torch_e4m3_codes(v))


def test_e4m3_encode_ties_and_random_fp32():
    finite = quant.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = ((finite[:-1] + finite[1:]) / 2).astype(np.float32)   # exact midpoints
    rng = np.random.default_rng(1)
    rnd = (rng.standard_normal(200000) * rng.choice([1e-3, 0.1, 1, 30, 200], 200000)).astype(np.float32)
    for v in (mids, -mids, rnd[np.abs(rnd) <= 464]):
        assert np.array_equal(quant.e4m3_encode(v), _torch_e4m3_codes(v))
    # ties go to the even code
    ties = quant.e4m3_encode(mids)
    assert np.all(ties % 2 == 0)


def test_e4m3_saturates():
    v = np.array([448.0, 449.0, 470.0, 1e6, -470.0, -1e30], dtype=np.float32)
    assert list(quant.e4m3_encode(v)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_e4m3_round_trip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = quant.e4m3_decode(codes).astype(np.float32)
    back = quant.e4m3_encode(vals)
    assert np.array_equal(quant.e4m3_decode(back), quant.e4m3_decode(codes))


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(300000) * rng.choice([1e-30, 1e-3, 1, 1e3, 1e30], 300000)).astype(np.float32)
    # exact ties: bf16 value + half a quantum
    base = torch.from_numpy(v[:1000]).to(torch.bfloat16).to(torch.float32).numpy()
    ties = (base.view(np.uint32) | np.uint32(0x8000)).view(np.float32)
    for x in (v, ties):
        ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
        assert np.array_equal(quant.bf16_round(x), ref)


def test_bf16_bits_round_trip():
    rng = np.random.default_rng(3)
    v = torch.from_numpy(rng.standard_normal(1000).astype(np.float32)).to(torch.bfloat16)
    bits = v.view(torch.int16).numpy().view(np.uint16)
    f = quant.bf16_from_bits(bits)
    assert np.array_equal(f, v.to(torch.float32).numpy())
    assert np.array_equal(quant.bf16_bits(f), bits)


@pytest.mark.parametrize("scale", [1e-4, 1.0, 50.0])
def test_group_quant_bounds(scale):
    rng = np.random.default_rng(4)
    v = (rng.standard_normal((7, 512)) * scale).astype(np.float32)
    v[3, 128:256] = 0.0                          # an all-zero group
    codes, s = quant.quant_groups_fp8(v)
    assert codes.shape == v.shape and s.shape == (7, 4) and s.dtype == np.float32
    assert s[3, 1] == 1.0 and np.all(codes[3, 128:256] == 0)
    g = v.reshape(7, 4, 128)
    amax = np.abs(g).max(axis=2)
    nz = amax > 0
    # scale = amax / 448 exactly as an fp32 division
    assert np.array_equal(s[nz], (amax / np.float32(448.0))[nz])
    # the largest element of each group lands on +-448
    c = codes.reshape(7, 4, 128)
    arg = np.abs(g).argmax(axis=2)
    top = np.take_along_axis(c, arg[..., None], axis=2)[..., 0]
    assert np.all(np.isin(top[nz], [0x7E, 0xFE]))
    # dequantised error: half an e4m3 quantum (3 mantissa bits, subnormal quantum 2^-9)
    deq = quant.dequant_groups_fp8(codes, s)
    err = np.abs(deq - v.astype(np.float64))
    bound = np.maximum(np.abs(v) * 2.0 ** -4, np.repeat(s, 128, axis=1) * 2.0 ** -10)
    assert np.all(err <= bound * (1 + 1e-6))


def test_group_quant_is_torch_cast_of_fp32_quotient():
    rng = np.random.default_rng(5)
    v = rng.standard_normal((5, 256)).astype(np.float32)
    codes, s = quant.quant_groups_fp8(v)
    t = torch.from_numpy(v).view(5, 2, 128)
    amax = t.abs().amax(dim=2)
    ts = amax / 448.0
    q = (t / ts[..., None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(5, 256).numpy()
    assert np.array_equal(s, ts.numpy())
    assert np.array_equal(codes, q)
