"""Pins of the compact 656-byte latent row (oracle/compact_row.py), and the
plausible mistakes they catch.

The row is a reading of the "ESS: Latent-Cache Offload" page: 512 e4m3
latent values in four tiles with power-of-two scales, four float32 scales
and the 64 bf16 RoPE values.  The pins: the page's byte split, the e4m3
definition (every byte's value, rounding to nearest with ties to the even
code, saturation), exact round trips of values already on the scaled grid,
the scale rule and the rounding error bound, decoded values exact in bf16,
the batched decoder against the per-row one, and the layout of the bytes.
"""
import inspect
import os
import sys

import numpy as np
import pytest

from oracle import compact_row as X
from host_latent_cache_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ess_entry_split.txt")


def _golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line:
                out[line[0]] = float(line[1])
    return out


def _bits(x):
    return W.float_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_row_size_matches_the_pages_split():
    g = _golden()
    assert X.ROW_BYTES == 512 + 16 + 128 == g["transfer_bytes"]
    indexer = 128 + 4                                   # e4m3 key and its float32 scale
    total = X.ROW_BYTES + indexer
    assert round(100 * indexer / total, 1) == g["indexer_share_pct"]
    assert round(100 * X.ROW_BYTES / total, 1) == g["latent_share_pct"]


def test_e4m3_values_from_the_definition():
    # the largest finite value, the smallest normal and subnormal, one, NaN
    assert X.e4m3_value(0x7E) == 448.0
    assert X.e4m3_value(0x08) == 2.0 ** -6
    assert X.e4m3_value(0x01) == 2.0 ** -9
    assert X.e4m3_value(0x38) == 1.0
    assert X.e4m3_value(0xB8) == -1.0
    assert np.isnan(X.e4m3_value(0x7F)) and np.isnan(X.e4m3_value(0xFF))
    vals = [X.e4m3_value(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(vals, vals[1:]))   # codes are ordered by value


def test_e4m3_rounding_ties_to_even_and_saturates():
    assert X.e4m3_encode(1.0625) == 0x38                # between 1 (even) and 1.125
    assert X.e4m3_encode(1.1875) == 0x3A                # between 1.125 and 1.25 (even)
    assert X.e4m3_encode(1.07) == 0x39
    assert X.e4m3_encode(-1.0625) == 0xB8
    assert X.e4m3_encode(500.0) == 0x7E and X.e4m3_encode(-1e9) == 0xFE
    assert X.e4m3_encode(2.0 ** -11) == 0x00            # below half the smallest subnormal
    assert X.e4m3_encode(-(2.0 ** -11)) == 0x80         # the sign of zero is kept
    assert X.e4m3_encode(3 * 2.0 ** -10) == 0x02        # 1.5 subnormal steps: even code 2


def test_values_on_the_scaled_grid_round_trip_exactly():
    # tile j holds e4m3 values times 2^(j-2), with 448 * 2^(j-2) present, so
    # its scale is exactly 2^(j-2) and every value survives
    rng = np.random.default_rng(3)
    levels = np.array([X.e4m3_value(c) for c in range(0x7F)])
    lat = []
    for j in range(4):
        v = rng.choice(levels, 128) * rng.choice([-1.0, 1.0], 128)
        v[5] = 448.0
        lat.append(v * 2.0 ** (j - 2))
    row = np.concatenate(lat + [rng.standard_normal(64)]).astype(np.float32)
    bits = _bits(row)
    assert np.array_equal(W.bf16_bits_to_float(bits)[:512], row[:512])   # exact in bf16 too
    enc = X.encode_row(bits)
    assert enc[512:528].view("<f4").tolist() == [0.25, 0.5, 1.0, 2.0]
    dec = X.decode_row(enc)
    assert np.array_equal(dec[:512], row[:512].astype(np.float64))


def test_rounding_error_bound_and_layout():
    rng = np.random.default_rng(4)
    for _ in range(20):
        x = (rng.standard_normal(576) * 0.5).astype(np.float32)
        x[:128] *= 30.0                                 # tiles of different ranges
        bits = _bits(x)
        xv = W.bf16_bits_to_float(bits).astype(np.float64)
        enc = X.encode_row(bits)
        assert enc.shape == (656,) and enc.dtype == np.uint8
        dec = X.decode_row(enc)
        scales = enc[512:528].view("<f4").astype(np.float64)
        for j in range(4):
            t = slice(128 * j, 128 * (j + 1))
            amax = np.max(np.abs(xv[t]))
            # the smallest power of two at or above amax / 448 (float32)
            m, e = np.frexp(scales[j])
            assert m == 0.5
            q = np.float32(np.float32(amax) / np.float32(448.0))
            assert scales[j] >= q and scales[j] / 2 < q
            assert 224.0 < amax / scales[j] <= 448.0
            err = np.abs(dec[t] - xv[t])
            # half a step: 2^-4 of the value in the normal range, 2^-10 of the
            # scale in the subnormal range (plus the float32 division's rounding)
            bound = np.maximum(np.abs(xv[t]) * 2.0 ** -4, scales[j] * 2.0 ** -10) * (1 + 2.0 ** -20)
            assert np.all(err <= bound)
        assert np.array_equal(enc[528:].view("<u2"), bits[512:])          # RoPE untouched
        assert np.array_equal(dec[512:], xv[512:])


def test_decoded_values_are_exact_in_bf16():
    # the point of power-of-two scales: a GPU widens rows to bf16 exactly
    rng = np.random.default_rng(5)
    for _ in range(10):
        x = (rng.standard_normal(576) * rng.choice([0.01, 0.5, 40.0])).astype(np.float32)
        dec = X.decode_row(X.encode_row(_bits(x)))
        f32 = dec.astype(np.float32)
        assert np.array_equal(f32.astype(np.float64), dec)
        assert np.array_equal(W.bf16_bits_to_float(_bits(f32)), f32)


def test_decode_rows_equals_decode_row():
    rng = np.random.default_rng(6)
    rows = rng.integers(0, 256, size=(7, 656), dtype=np.uint8)
    rows[:, :512] &= 0xFE                               # no NaN codes (0x7F / 0xFF)
    rows[:, 512:528] = np.repeat(np.array([[2.0 ** -8, 0.5, 1.0, 2.0 ** 3]], "<f4").view(np.uint8),
                                 7, axis=0)
    rope = _bits(rng.standard_normal((7, 64)).astype(np.float32))
    rows[:, 528:] = rope.astype("<u2").view(np.uint8).reshape(7, 128)
    got = X.decode_rows(rows)
    for i in range(7):
        assert np.array_equal(got[i], X.decode_row(rows[i]))


def test_zero_tile_has_unit_scale():
    x = np.zeros(576, np.float32)
    x[200] = 14.0                                       # scale 14/448 = 2^-5, exact
    enc = X.encode_row(_bits(x))
    assert enc[512:528].view("<f4").tolist()[0] == 1.0
    assert np.all(enc[:128] == 0)
    assert np.array_equal(X.decode_row(enc)[:512], x[:512].astype(np.float64))


# ------------------------------------------------------------------ mutants

ORIG_ENCODE = X.e4m3_encode
ORIG_ROW = X.encode_row


def _encode_truncates(v):
    sign = 0x80 if (v < 0 or (v == 0 and np.signbit(v))) else 0
    a = min(abs(float(v)), 448.0)
    i = int(np.searchsorted(X._POS_VALUES, a, side="right")) - 1
    return sign | int(X._POS_CODES[i])


def _encode_ties_away(v):
    sign = 0x80 if (v < 0 or (v == 0 and np.signbit(v))) else 0
    a = min(abs(float(v)), 448.0)
    i = int(np.argmin(np.abs(X._POS_VALUES - a) - 1e-12 * X._POS_VALUES))
    return sign | int(X._POS_CODES[i])


def _row_one_scale(bits):
    out = ORIG_ROW(bits)
    x = W.bf16_bits_to_float(np.asarray(bits, np.uint16))[:512]
    amax = np.float32(np.max(np.abs(x)))
    s = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
    out[:512] = [ORIG_ENCODE(float(v)) for v in (x / s).astype(np.float32)]
    out[512:528] = np.full(4, s, "<f4").view(np.uint8)
    return out


def _row_wrong_max(bits):
    x = W.bf16_bits_to_float(np.asarray(bits, np.uint16))
    out = ORIG_ROW(bits)
    for j in range(4):
        t = x[128 * j:128 * (j + 1)]
        amax = np.float32(np.max(np.abs(t)))
        s = np.float32(amax / np.float32(240.0)) if amax > 0 else np.float32(1.0)
        out[128 * j:128 * (j + 1)] = [ORIG_ENCODE(float(v)) for v in (t / s).astype(np.float32)]
        out[512 + 4 * j:516 + 4 * j] = np.array([s], "<f4").view(np.uint8)
    return out


def _row_scale_not_a_power_of_two(bits):
    x = W.bf16_bits_to_float(np.asarray(bits, np.uint16))
    out = ORIG_ROW(bits)
    for j in range(4):
        t = x[128 * j:128 * (j + 1)]
        amax = np.float32(np.max(np.abs(t)))
        s = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
        out[128 * j:128 * (j + 1)] = [ORIG_ENCODE(float(v)) for v in (t / s).astype(np.float32)]
        out[512 + 4 * j:516 + 4 * j] = np.array([s], "<f4").view(np.uint8)
    return out


def _row_rope_quantized(bits):
    out = ORIG_ROW(bits)
    out[528:] = 0
    return out


MUTANTS = [("e4m3_encode", _encode_truncates), ("e4m3_encode", _encode_ties_away),
           ("encode_row", _row_one_scale), ("encode_row", _row_wrong_max),
           ("encode_row", _row_rope_quantized), ("encode_row", _row_scale_not_a_power_of_two)]
PINS = [f for name, f in sorted(vars(sys.modules[__name__]).items())
        if name.startswith("test_") and inspect.isfunction(f) and name != "test_pins_catch_mutant"]


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=[m.__name__ for _, m in MUTANTS])
def test_pins_catch_mutant(monkeypatch, name, mutant):
    monkeypatch.setattr(X, name, mutant)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (Exception, pytest.fail.Exception) as e:   # an assertion or a pytest.raises miss
            failed.append(f"{pin.__name__}: {type(e).__name__}")
            break
    assert failed, f"no pin notices {mutant.__name__}"
