"""Pins of the oracle's 8-bit KV format (FP8 E4M3 codes with one fp32 scale per row).

The format's facts come from the OCP 8-bit floating-point definition (1 sign, 4 exponent
bits with bias 7, 3 mantissa bits, no infinities, NaN only at S.1111.111, largest finite
magnitude 448). The encoder is also compared with torch's float8_e4m3fn conversion, a
library routine, on values inside the finite range.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from split_kv_decode_distattention_gb300 import workloads as W

FINITE = [c for c in range(256) if c not in (0x7F, 0xFF)]


def test_named_codes_have_their_values(orc):
    assert orc.e4m3_value(0x00) == 0.0
    assert math.copysign(1.0, orc.e4m3_value(0x80)) == -1.0  # -0
    assert orc.e4m3_value(0x38) == 1.0
    assert orc.e4m3_value(0x40) == 2.0
    assert orc.e4m3_value(0xB8) == -1.0
    assert orc.e4m3_value(0x7E) == 448.0  # largest finite
    assert orc.e4m3_value(0x08) == 2.0 ** -6  # smallest normal
    assert orc.e4m3_value(0x01) == 2.0 ** -9  # smallest subnormal
    assert math.isnan(orc.e4m3_value(0x7F)) and math.isnan(orc.e4m3_value(0xFF))


def test_positive_codes_are_strictly_increasing(orc):
    vals = [orc.e4m3_value(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(vals, vals[1:]))
    assert len(set(orc.e4m3_value(c) for c in FINITE)) == 253  # +0 and -0 compare equal


def test_values_match_torch_float8_e4m3fn(orc):
    codes = torch.tensor(FINITE, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.e4m3_value(c) for c in FINITE])
    np.testing.assert_array_equal(got, ref)


def test_encoder_round_trips_every_finite_code(orc):
    for c in FINITE:
        assert orc.e4m3_code(orc.e4m3_value(c)) == c


def test_encoder_matches_torch_on_a_dense_sweep(orc):
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-448, 448, 4000),
                        rng.normal(0, 1, 4000) * 2.0 ** rng.integers(-12, 8, 4000)])
    x = x.astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_code(float(v)) for v in x], np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_encoder_ties_to_even_and_saturates(orc):
    pos = sorted((orc.e4m3_value(c), c) for c in range(0x7F))
    for (a, ca), (b, cb) in zip(pos, pos[1:]):
        mid = (a + b) / 2
        if np.float32(mid) != mid:
            continue  # the midpoint is not an fp32 value
        even = ca if ca % 2 == 0 else cb
        assert orc.e4m3_code(mid) == even, (a, b)
    assert orc.e4m3_code(1000.0) == 0x7E and orc.e4m3_code(-1000.0) == 0xFE
    assert orc.e4m3_code(450.0) == 0x7E  # between 448 and the unrepresentable 480
    assert orc.e4m3_code(2.0 ** -11) == 0x00  # below half the smallest subnormal
    assert orc.e4m3_code(-(2.0 ** -11)) == 0x80


def test_quantized_row_uses_the_full_range_and_bounds_the_error(orc):
    rng = np.random.default_rng(4)
    for trial in range(40):
        x = torch.from_numpy(rng.normal(0, 1 + trial, 128).astype(np.float32)).to(torch.bfloat16)
        codes, scale = orc.quantize_rows_fp8(x)
        xf = x.to(torch.float64).numpy()
        j = int(np.argmax(np.abs(xf)))
        assert orc.e4m3_value(codes[j]) == math.copysign(448.0, xf[j])
        assert scale == np.float32(np.float32(np.abs(xf).max()) / np.float32(448.0))
        deq = orc.dequantize_rows_fp8(codes, scale)
        # 3 mantissa bits: relative error <= 2^-4 for normals, 2^-10 * scale absolute below
        bound = np.maximum(np.abs(xf) * 2.0 ** -4, 2.0 ** -10 * float(scale))
        assert np.all(np.abs(deq - xf) <= bound * (1 + 1e-12))


def test_zero_row_has_zero_scale_and_codes(orc):
    codes, scale = orc.quantize_rows_fp8(np.zeros(64, np.uint16))
    assert scale == 0.0 and not codes.any()
    assert not orc.dequantize_rows_fp8(codes, scale).any()


def test_fp8_pool_write_matches_row_quantization_and_bf16_layout(orc):
    case = W.Case("fp8w", B=1, Hq=4, Hkv=2, d=64, P=16, lens=[0], seed=5, shuffle=False)
    T = 40
    K, V = case.kv(0, 0, T, "cpu")
    num_pages = 4
    kp = np.zeros((num_pages, 2, 16, 64), np.uint8)
    vp = np.zeros_like(kp)
    ks = np.zeros((num_pages, 2, 16), np.float32)
    vs = np.zeros_like(ks)
    bt = np.array([2, 0, 3, -1], np.int32)
    assert orc.kv_write_fp8(kp, vp, ks, vs, 16, bt, num_pages, K, V, 0) == 0
    kc, kscale = orc.quantize_rows_fp8(K)
    vc, vscale = orc.quantize_rows_fp8(V)
    for t in range(T):
        page, slot = bt[t // 16], t % 16
        for h in range(2):
            np.testing.assert_array_equal(kp[page, h, slot], kc[t, h])
            np.testing.assert_array_equal(vp[page, h, slot], vc[t, h])
            assert ks[page, h, slot] == kscale[t, h] and vs[page, h, slot] == vscale[t, h]
    # the unmapped fourth page is skipped, and nothing else is written
    assert orc.kv_write_fp8(kp, vp, ks, vs, 16, bt, num_pages, K[:1], V[:1], 48) == 1


def test_f64_attention_equals_bf16_attention_on_bf16_values(orc):
    rng = np.random.default_rng(6)
    K = torch.from_numpy(rng.normal(size=(300, 64)).astype(np.float32)).to(torch.bfloat16)
    V = torch.from_numpy(rng.normal(size=(300, 64)).astype(np.float32)).to(torch.bfloat16)
    q = torch.from_numpy(rng.normal(size=64).astype(np.float32)).to(torch.bfloat16)
    rows = np.arange(5, 280, 3)
    out, m, e = orc.attention(q, K, V, 0.125, rows=rows)
    out2, m2, e2 = orc.attention_f64(q, K.double().numpy(), V.double().numpy(), 0.125, rows=rows)
    np.testing.assert_array_equal(out, out2)
    assert m == m2 and e == e2
    mj, ej, MA = orc.partial(q, K, V, 0.125, rows=rows)
    mj2, ej2, MA2 = orc.partial_f64(q, K.double().numpy(), V.double().numpy(), 0.125, rows=rows)
    np.testing.assert_array_equal(MA, MA2)
    assert mj == mj2 and ej == ej2
