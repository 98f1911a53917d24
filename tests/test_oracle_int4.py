"""Pins of the oracle's 4-bit KV format (reading R12 of the oracle).

A row of d bf16 values keeps one fp32 scale, max|x| / 7, and d symmetric integer codes
x / scale rounded to the nearest integer (ties to even) in [-7, 7]; byte i holds code + 8 of
channel 2i in its low nibble and of channel 2i + 1 in its high nibble. The expected codes
below are worked out by hand from that definition; the rest are properties every row must
have (range, the largest element at +-7, the rounding error bound, sign symmetry).
"""
import numpy as np
import torch

from split_kv_decode_distattention_gb300 import workloads as W


def _bf16(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)


def test_golden_row(orc):
    # max |x| = 3.5, scale = 0.5; x / scale = 3.5, -7, 1, 0, 6.5, -0.5, 2, -2
    # -> codes 4 (tie to even), -7, 1, 0, 6 (tie to even), 0 (tie to even), 2, -2
    x = _bf16([1.75, -3.5, 0.5, 0.0, 3.25, -0.25, 1.0, -1.0])
    packed, scale = orc.quantize_rows_int4(x)
    assert scale == 0.5
    # nibbles 12, 1 | 9, 8 | 14, 8 | 10, 6
    np.testing.assert_array_equal(packed, np.array([0x1C, 0x89, 0x8E, 0x6A], np.uint8))
    np.testing.assert_array_equal(orc.int4_codes(packed), [4, -7, 1, 0, 6, 0, 2, -2])
    np.testing.assert_array_equal(orc.dequantize_rows_int4(packed, scale),
                                  [2.0, -3.5, 0.5, 0.0, 3.0, 0.0, 1.0, -1.0])


def test_ties_go_to_the_even_code(orc):
    # max 7 gives scale 1: x / scale is x itself
    x = _bf16([7.0, 0.5, 1.5, 2.5, -2.5, -1.5, 3.5, -4.5])
    packed, scale = orc.quantize_rows_int4(x)
    assert scale == 1.0
    np.testing.assert_array_equal(orc.int4_codes(packed), [7, 0, 2, 2, -2, -2, 4, -4])


def test_rows_use_the_full_range_and_bound_the_error(orc):
    rng = np.random.default_rng(12)
    for trial in range(40):
        x = _bf16(rng.normal(0, 1 + trial, 128))
        packed, scale = orc.quantize_rows_int4(x)
        xf = x.to(torch.float64).numpy()
        codes = orc.int4_codes(packed)
        nib = np.stack([packed & 15, packed >> 4], axis=-1).reshape(-1)
        assert nib.min() >= 1 and nib.max() <= 15  # codes never reach -8
        assert scale == np.float32(np.float32(np.abs(xf).max()) / np.float32(7.0))
        j = int(np.argmax(np.abs(xf)))
        assert codes[j] == (7 if xf[j] > 0 else -7)
        deq = orc.dequantize_rows_int4(packed, scale)
        # half a step, plus the fp32 rounding of x / scale (|x / scale| <= 7)
        assert np.all(np.abs(deq - xf) <= float(scale) * (0.5 + 7 * 2.0 ** -23))


def test_negated_row_negates_the_codes(orc):
    rng = np.random.default_rng(13)
    x = _bf16(rng.normal(0, 2, 64))
    p1, s1 = orc.quantize_rows_int4(x)
    p2, s2 = orc.quantize_rows_int4(-x)
    assert s1 == s2
    np.testing.assert_array_equal(orc.int4_codes(p2), -orc.int4_codes(p1).astype(np.int16))


def test_zero_row_has_zero_scale_and_zero_codes(orc):
    packed, scale = orc.quantize_rows_int4(np.zeros(64, np.uint16))
    assert scale == 0.0
    assert (packed == 0x88).all()
    assert not orc.dequantize_rows_int4(packed, scale).any()


def test_int4_pool_write_matches_row_quantization_and_layout(orc):
    case = W.Case("int4w", B=1, Hq=4, Hkv=2, d=64, P=16, lens=[0], seed=7, shuffle=False)
    T = 40
    K, V = case.kv(0, 0, T, "cpu")
    num_pages = 4
    kp = np.zeros((num_pages, 2, 16, 32), np.uint8)
    vp = np.zeros_like(kp)
    ks = np.zeros((num_pages, 2, 16), np.float32)
    vs = np.zeros_like(ks)
    bt = np.array([2, 0, 3, -1], np.int32)
    assert orc.kv_write_int4(kp, vp, ks, vs, 16, bt, num_pages, K, V, 0) == 0
    kc, kscale = orc.quantize_rows_int4(K)
    vc, vscale = orc.quantize_rows_int4(V)
    for t in range(T):
        page, slot = bt[t // 16], t % 16
        for h in range(2):
            np.testing.assert_array_equal(kp[page, h, slot], kc[t, h])
            np.testing.assert_array_equal(vp[page, h, slot], vc[t, h])
            assert ks[page, h, slot] == kscale[t, h] and vs[page, h, slot] == vscale[t, h]
    # the unmapped fourth page is skipped, and nothing else is written
    assert orc.kv_write_int4(kp, vp, ks, vs, 16, bt, num_pages, K[:1], V[:1], 48) == 1
