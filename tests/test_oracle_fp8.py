"""Pins of the FP8 (E4M3) cache oracle: code values fixed by the format's
definition, a round trip of every finite code, agreement with PyTorch's
float8_e4m3fn cast where both define the result, ties to even, saturation,
planted mistakes, and exactness when the cached values are representable."""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as ofp8


def test_code_values_follow_the_bit_fields():
    # (code, value): zero, the smallest and largest subnormal, the smallest
    # normal, one, the largest finite value, negative zero and -448
    cases = [(0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
             (0x38, 1.0), (0x3C, 1.5), (0x40, 2.0), (0x7E, 448.0), (0x80, -0.0), (0xFE, -448.0),
             (0xB8, -1.0)]
    for code, want in cases:
        got = float(oracle.e4m3_value(np.uint8(code)))
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got)
    assert np.isnan(oracle.e4m3_value(np.uint8(0x7F)))
    assert np.isnan(oracle.e4m3_value(np.uint8(0xFF)))
    assert oracle.E4M3_MAX == float(oracle.e4m3_value(np.uint8(0x7E)))


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_value(codes).astype(np.float32)
    back = oracle.e4m3_encode(vals)
    assert np.array_equal(back, codes)


def test_encode_matches_torch_below_the_saturation_point():
    # a dense sweep including every midpoint between neighbouring codes (the
    # ties) and values just off them; torch maps |y| >= 464 to NaN, the reading
    # here saturates, so the comparison stops below 464
    pos = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2
    rng = np.random.default_rng(0)
    y = np.concatenate([pos, mids, np.nextafter(mids, 0), np.nextafter(mids, 1000),
                        rng.uniform(-460, 460, 4000), rng.normal(0, 0.01, 2000)])
    y = np.concatenate([y, -y]).astype(np.float32)
    y = y[np.abs(y) < 464]
    ours = oracle.e4m3_encode(y)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_ties_go_to_the_even_mantissa():
    cases = [(1.0 + 1 / 16, 0x38),      # between 1.0 (m=0) and 1.125 (m=1): m=0
             (1.0 + 3 / 16, 0x3A),      # between 1.125 (m=1) and 1.25 (m=2): m=2
             (2.0 ** -10, 0x00),        # between 0 and the smallest subnormal: 0
             (3 * 2.0 ** -10, 0x02),    # between 2^-9 (m=1) and 2^-8 (m=2): m=2
             (-(1.0 + 1 / 16), 0xB8)]
    for y, want in cases:
        assert int(oracle.e4m3_encode(np.float32(y))) == want, y


def test_saturation_and_nan():
    y = np.array([448.0, 460.0, 464.0, 500.0, 1e10, -1e10, np.inf, -np.inf], dtype=np.float32)
    assert oracle.e4m3_encode(y).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE]
    assert int(oracle.e4m3_encode(np.float32(np.nan))) & 0x7F == 0x7F


def test_quantize_rows_divides_by_the_heads_scale_in_float32():
    x = torch.tensor([[[3.0, -6.0], [1.0, 0.5]]], dtype=torch.bfloat16)  # [1, Hkv=2, d=2]
    scale = np.array([2.0, 0.25], dtype=np.float32)
    got = oracle.quantize_rows(x.float().numpy(), scale)
    want = oracle.e4m3_encode(np.array([[[1.5, -3.0], [4.0, 2.0]]], dtype=np.float32))
    assert np.array_equal(got, want)
    # an inexact quotient is rounded to float32 first, as the library does
    y = np.float32(1.0) / np.float32(3.0)
    assert int(oracle.quantize_rows(np.ones((1, 1, 1), np.float32), [3.0])[0, 0, 0]) == \
        int(oracle.e4m3_encode(y))


def test_fp8_cache_is_exact_for_representable_values():
    """With values that E4M3 holds exactly (times a power-of-two scale),
    quantise + dequantise is the identity, so the FP8 decode equals the
    bf16-cache decode of the same values."""
    rng = np.random.default_rng(1)
    lengths = [5, 37, 16]
    hkv, d, hq = 2, 8, 4
    nb = sum((n + 15) // 16 for n in lengths) + 1
    codes_k = rng.integers(0, 0x7F, size=(nb, 16, hkv, d)).astype(np.uint8)
    codes_k |= (rng.integers(0, 2, size=codes_k.shape) * 0x80).astype(np.uint8)
    codes_v = rng.integers(0, 0x7E, size=(nb, 16, hkv, d)).astype(np.uint8)
    k_scale = np.array([0.5, 2.0], np.float32)
    v_scale = np.array([0.125, 1.0], np.float32)
    table, nxt = [], 0
    perm = rng.permutation(nb)
    for n in lengths:
        m = (n + 15) // 16
        table.append([int(x) for x in perm[nxt:nxt + m]] + [-1] * (3 - m))
        nxt += m
    q = rng.normal(size=(3, hq, d)) * 0.05
    o8, l8 = oracle.decode_paged_fp8(q, codes_k, codes_v, k_scale, v_scale, table, lengths,
                                     block_size=16)
    kd = oracle.e4m3_value(codes_k) * k_scale.reshape(-1, 1)
    vd = oracle.e4m3_value(codes_v) * v_scale.reshape(-1, 1)
    o, l = oracle.decode_paged(q, kd, vd, table, lengths, block_size=16)
    assert np.abs(o8 - o).max() == 0 and np.abs(l8 - l).max() == 0
    # and quantising those exact values gives the codes back (scale divides exactly)
    assert np.array_equal(oracle.quantize_rows(kd.astype(np.float32), k_scale), codes_k)


def test_append_paged_fp8_writes_quantised_rows_only_at_their_slots():
    before, new = [3, 16], [2, 1]
    hkv, d = 2, 4
    nb = 4
    table = [[2, -1], [0, 3]]
    rng = np.random.default_rng(2)
    kc = rng.integers(0, 256, size=(nb, 16, hkv, d)).astype(np.uint8)
    vc = rng.integers(0, 256, size=(nb, 16, hkv, d)).astype(np.uint8)
    kn = rng.normal(size=(3, hkv, d)).astype(np.float32)
    vn = rng.normal(size=(3, hkv, d)).astype(np.float32)
    ks, vs = np.array([0.5, 0.25], np.float32), np.array([1.0, 2.0], np.float32)
    k2, v2 = oracle.append_paged_fp8(kc, vc, kn, vn, ks, vs, table, before, [0, 2, 3], 16)
    changed = np.argwhere((k2 != kc).any(axis=(2, 3)))
    assert set(map(tuple, changed.tolist())) <= {(2, 3), (2, 4), (3, 0)}
    assert np.array_equal(k2[2, 3], oracle.quantize_rows(kn[0:1], ks)[0])
    assert np.array_equal(v2[3, 0], oracle.quantize_rows(vn[2:3], vs)[0])


def test_fp8_halves_the_page_kv_bytes():
    # "Генерация и KV-кэш", section "Сколько весит KV-кэш": 1 byte per number in
    # FP8 against 2 in BF16; Llama 3 8B keeps 128 KiB per token in BF16
    bf16 = oracle.kv_cache_bytes(32, 8, 1, 128, 2)
    assert bf16 == 128 * 1024
    assert oracle.kv_cache_bytes(32, 8, 1, 128, 1) == bf16 // 2


@pytest.mark.parametrize("mistake", ["truncate", "bias8", "nan_overflow"])
def test_planted_fp8_mistakes_are_caught(mistake, monkeypatch):
    """Each plausible codec bug fails at least one of the pins above."""
    good_encode = ofp8.e4m3_encode
    if mistake == "truncate":
        def bad(y):
            y = np.asarray(y, dtype=np.float32).astype(np.float64)
            out = good_encode(y)
            # round toward zero instead of to nearest
            vals = ofp8.e4m3_value(out)
            over = np.abs(vals) > np.abs(y)
            out = out.astype(np.int64)
            out[over] -= 1
            return out.astype(np.uint8)
        monkeypatch.setattr(ofp8, "e4m3_encode", bad)
        monkeypatch.setattr(oracle, "e4m3_encode", bad)
        with pytest.raises(AssertionError):
            test_ties_go_to_the_even_mantissa()
    elif mistake == "bias8":
        vals = ofp8._VALUES.copy()
        bad_vals = np.where(np.isnan(vals), vals, vals / 2)
        monkeypatch.setattr(ofp8, "_VALUES", bad_vals)
        with pytest.raises(AssertionError):
            test_code_values_follow_the_bit_fields()
    else:
        def bad(y):
            out = good_encode(y)
            big = np.abs(np.asarray(y, dtype=np.float32)) >= 464
            out = np.where(big, np.uint8(0x7F), out).astype(np.uint8)
            return out
        monkeypatch.setattr(oracle, "e4m3_encode", bad)
        with pytest.raises(AssertionError):
            test_saturation_and_nan()
