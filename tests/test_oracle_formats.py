"""Pins of the oracle's number formats (bf16, OCP E4M3) and of its per-128-column
FP8 cast, against library converters, closed forms and hand-worked values.

The e4m3 encoder is checked against torch's float8_e4m3fn conversion (round to
nearest even; torch turns magnitudes past 464 into NaN, where the satfinite
rule of the cast saturates to 448), the bf16 encoder against torch's bfloat16
conversion (round to nearest even).
"""
import numpy as np
import pytest
import torch


def _torch_e4m3(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_e4m3_decode_table_matches_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_to_f32(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ours[~nan], ref[~nan])
    # anchors from the format definition
    assert ours[0x7E] == 448.0 and ours[0xFE] == -448.0
    assert ours[0x38] == 1.0
    assert ours[0x08] == 2.0 ** -6 and ours[0x01] == 2.0 ** -9 and ours[0x07] == 7 * 2.0 ** -9


def test_e4m3_roundtrip_every_finite_code(orc):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    back = orc.f32_to_e4m3(orc.e4m3_to_f32(codes))
    assert np.array_equal(back, codes)


def test_e4m3_encoder_matches_torch_on_sweep(orc):
    # strided sweep over every binary32 magnitude up to 464, both signs
    lim = np.float32(464.0).view(np.uint32)
    bits = np.arange(0, int(lim) + 1, 997, dtype=np.uint32)
    x = bits.view(np.float32)
    x = np.concatenate([x, -x])
    assert np.array_equal(orc.f32_to_e4m3(x), _torch_e4m3(x))


def test_e4m3_encoder_ties_and_neighbours(orc):
    finite = np.array(sorted({float(v) for v in orc.e4m3_to_f32(np.arange(0, 0x7F, dtype=np.uint8))}))
    mids = (finite[:-1] + finite[1:]) / 2  # exact in binary32
    mids = mids.astype(np.float32)
    around = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
                             finite.astype(np.float32)])
    x = np.concatenate([around, -around])
    assert np.array_equal(orc.f32_to_e4m3(x), _torch_e4m3(x))
    # ties go to the even code: 17 lies between 16 (0x58) and 18 (0x59)
    assert orc.f32_to_e4m3(np.array([17.0, 19.0], np.float32)).tolist() == [0x58, 0x5A]


def test_e4m3_saturates_past_largest_finite(orc):
    x = np.array([448.0, 464.0, 464.0001, 480.0, 1e4, 3.0e38, np.inf], np.float32)
    assert orc.f32_to_e4m3(x).tolist() == [0x7E] * 7
    assert orc.f32_to_e4m3(-x).tolist() == [0xFE] * 7
    # torch agrees wherever it does not produce NaN
    t = _torch_e4m3(x[:2])
    assert t.tolist() == [0x7E, 0x7E]


def test_e4m3_encoder_monotone_over_all_positive_floats(orc):
    # every positive finite binary32 in chunks: codes never decrease
    prev = 0
    step = 1 << 26
    top = int(np.float32(np.inf).view(np.uint32))
    for first in range(0, top, step):
        n = min(step, top - first)
        c = orc.e4m3_of_bits(first, n)
        assert c[0] >= prev
        assert np.all(np.diff(c.astype(np.int16)) >= 0)
        prev = int(c[-1])
    assert prev == 0x7E


def test_bf16_encoder_matches_torch_on_sweep(orc):
    bits = np.arange(0, 1 << 32, 4099, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    assert np.array_equal(orc.f32_to_bf16(x), _torch_bf16(x))
    # ties to even around 1.0
    t = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -20], np.float32)
    assert orc.f32_to_bf16(t).tolist() == [0x3F80, 0x3F82, 0x3F81]


def _bf16_bits(v):
    return _torch_bf16(np.asarray(v, np.float32))


def test_fp8_cast_hand_worked_group(orc):
    # amax = 2 -> inv = 448/2 = 224 exactly; sf = 2/448 rounded to binary32
    g = np.zeros(128, np.float32)
    g[:4] = [1.0, -2.0, 0.5, 0.0]
    q, sf = orc.cast_row_fp8(_bf16_bits(g))
    assert sf[0] == np.float32(2.0) / np.float32(448.0)
    # 1*224 = 224 = 1.75*2^7 -> 0x76; -2*224 = -448 -> 0xFE; 0.5*224 = 112 -> 0x6E
    assert q[:4].tolist() == [0x76, 0xFE, 0x6E, 0x00]
    assert np.all(q[4:] == 0)


def test_fp8_cast_all_zero_group(orc):
    q, sf = orc.cast_row_fp8(np.zeros(256, np.uint16))
    assert np.all(q == 0)
    assert np.all(sf == np.float32(1e-4) / np.float32(448.0))


def test_fp8_cast_properties_random(orc):
    rng = np.random.default_rng(1)
    H = 1024
    for trial in range(40):
        scale = 10.0 ** rng.uniform(-6, 4)
        x = (rng.standard_normal(H) * scale).astype(np.float32)
        if trial % 5 == 0:
            x[rng.integers(0, H, 50)] = 0.0
        xb = _bf16_bits(x)
        xf = orc.bf16_to_f32(xb)
        q, sf = orc.cast_row_fp8(xb)
        deq = orc.e4m3_to_f32(q).astype(np.float64) * np.repeat(sf.astype(np.float64), 128)
        # e4m3 keeps 3 mantissa bits: rounding error <= 2^-4 relative (normal range)
        # or 2^-10 in scaled units (subnormals); sf*inv is 1 within a few ulp.
        bound = (2.0 ** -4 + 1e-6) * np.abs(xf) + 2.0 ** -10 * np.repeat(sf, 128) * 1.0001
        assert np.all(np.abs(deq - xf) <= bound)
        amax = np.abs(xf).reshape(-1, 128).max(1)
        for gi in range(H // 128):
            grp = xf[gi * 128:(gi + 1) * 128]
            if amax[gi] >= 1e-4:
                # the largest element lands on +-448
                j = int(np.argmax(np.abs(grp)))
                assert q[gi * 128 + j] in (0x7E, 0xFE)
                assert sf[gi] == np.float32(amax[gi]) / np.float32(448.0)
            else:
                assert sf[gi] == np.float32(1e-4) / np.float32(448.0)


def test_fp8_cast_power_of_two_scaling_invariance(orc):
    rng = np.random.default_rng(2)
    x = rng.standard_normal(512).astype(np.float32)
    q0, sf0 = orc.cast_row_fp8(_bf16_bits(x))
    for p in (-6, -1, 3, 9):
        q, sf = orc.cast_row_fp8(_bf16_bits(x * np.float32(2.0 ** p)))
        assert np.array_equal(q, q0)
        assert np.array_equal(sf, sf0 * np.float32(2.0 ** p))


# ---- packed power-of-two scales (reading of num_sf_packs) -------------------

def test_packed_cast_hand_worked_group(orc):
    g = np.zeros(512, np.float32)
    g[:4] = [1.0, -2.0, 0.5, 0.0]
    q, words = orc.cast_row_fp8_ue8m0(_bf16_bits(g))
    # group 0: amax 2 -> 2/448 lies in (2^-8, 2^-7] -> e = -7, byte 120 = 0x78;
    # q = x * 2^7: 128 -> 0x70, -256 -> 0xF8, 64 -> 0x68.
    # groups 1..3 are zero: amax clamps to 1e-4, 1e-4/448 in (2^-23, 2^-22] -> 0x69
    assert q[:4].tolist() == [0x70, 0xF8, 0x68, 0x00]
    assert words.tolist() == [0x69696978]


def test_packed_cast_properties(orc):
    rng = np.random.default_rng(5)
    H = 1152  # 9 groups: the third word holds one group and three zero bytes
    for trial in range(30):
        x = (rng.standard_normal(H) * 10.0 ** rng.uniform(-5, 5)).astype(np.float32)
        xb = _bf16_bits(x)
        xf = orc.bf16_to_f32(xb).astype(np.float64)
        q, words = orc.cast_row_fp8_ue8m0(xb)
        assert words.size == 3
        b = words.view(np.uint8)  # little-endian: group g is byte g
        assert not b[9:].any()
        e = b[:9].astype(np.int64) - 127
        amax = np.maximum(np.abs(xf).reshape(9, 128).max(1), np.float64(np.float32(1e-4)))
        # the smallest power of two at or above amax / 448
        assert np.all(amax <= 448.0 * 2.0 ** e) and np.all(amax > 448.0 * 2.0 ** (e - 1))
        deq = orc.e4m3_to_f32(q).astype(np.float64).reshape(9, 128) * (2.0 ** e)[:, None]
        err = np.abs(deq - xf.reshape(9, 128))
        assert np.all(err <= 2.0 ** -4 * np.abs(xf.reshape(9, 128)) + 2.0 ** -10 * (2.0 ** e)[:, None])
        assert np.all((q & 0x7F) <= 0x7E)


def test_packed_cast_equals_fp32_cast_when_the_scale_is_a_power_of_two(orc):
    # amax = 448 * 2^-3 = 56: the fp32 scale amax/448 is exactly 2^-3 = the packed one
    rng = np.random.default_rng(9)
    x = np.clip(rng.standard_normal(256).astype(np.float32) * 10, -55, 55)
    x[7], x[200] = 56.0, -56.0
    xb = _bf16_bits(x)
    q1, sf = orc.cast_row_fp8(xb)
    q2, words = orc.cast_row_fp8_ue8m0(xb)
    assert np.all(sf == np.float32(0.125)) and words.view(np.uint8)[:2].tolist() == [124, 124]
    assert np.array_equal(q1, q2)
