"""Pins for the oracle's NF4 codec (CPU only).

The codec follows the frozen-base precision of the method: 4-bit
NormalFloat codes with one fp32 absmax per 64 consecutive weights of a row
(Poros docs, "Limitations" page, "What 0.00e+00 means": NF4 is the only
bitwise precision; research page "Poros": the block-streamed NF4 loader
quantises each tensor).  Each test checks the oracle against something other
than the oracle itself: the published table, the quantile construction that
defines NF4, brute-force nearest-level search, exact round trips, and bounds.
"""
import os

import numpy as np
import pytest

from weight_streaming_nf4_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden", "nf4_levels.txt")


def _golden_levels():
    vals = [float(l) for l in open(GOLD) if l.strip() and not l.startswith("#")]
    return np.array(vals, dtype=np.float32)


def test_levels_match_printed_table(orc):
    lv = orc.nf4_levels()
    assert lv.dtype == np.float32 and lv.shape == (16,)
    assert np.array_equal(lv, _golden_levels())
    assert np.all(np.diff(lv) > 0)


def test_levels_match_normalfloat_construction(orc):
    """NF4 = normalised quantiles of N(0,1): 8 positive levels from 9 equally
    spaced probabilities in [0.5, 1-d], 7 negative from 8, plus an exact zero,
    with d = (1/32 + 1/30)/2, scaled so the largest level is 1 (QLoRA,
    section 3).  The printed 4-decimal table must round from it."""
    scipy_stats = pytest.importorskip("scipy.stats")
    top = 1.0 - 0.5 * (1.0 / 32.0 + 1.0 / 30.0)
    pos = scipy_stats.norm.ppf(np.linspace(top, 0.5, 9)[:-1])
    neg = -scipy_stats.norm.ppf(np.linspace(top, 0.5, 8)[:-1])
    v = np.sort(np.concatenate([pos, [0.0], neg]))
    v = v / v.max()
    lv = orc.nf4_levels().astype(np.float64)
    # printed to 4 decimals; 1e-5 slack for the construction's own float error
    assert np.max(np.abs(lv - v)) <= 0.5e-4 + 1e-5


def _unpack(codes):
    hi = codes >> 4
    lo = codes & 15
    return np.stack([hi, lo], axis=-1).reshape(codes.shape[0], -1)


def test_roundtrip_of_levels_times_scale(orc):
    """A block whose entries are bf16(c_i * a) (with +-a present) quantises to
    code i exactly, with absmax = bf16(a)."""
    lv = orc.nf4_levels().astype(np.float64)
    rng = np.random.default_rng(1)
    for a in [1.0, 0.5, 0.037, 3.75e-3, 17.0]:
        idx = rng.integers(0, 16, size=(8, 64))
        idx[:, 0] = 15
        w = synth.to_bf16_bits(lv[idx] * a)
        codes, absmax = orc.quantize_nf4(w)
        assert np.array_equal(_unpack(codes), idx)
        assert np.all(absmax == synth.bf16_bits_to_f32(synth.to_bf16_bits(np.array([a])))[0])


def test_absmax_is_block_max_and_extremes_map_to_end_codes(orc):
    W = synth.normal_bf16(0, "nf4.inv", (24, 256), 0.02)
    codes, absmax = orc.quantize_nf4(W)
    wf = synth.bf16_bits_to_f32(W).reshape(24, 4, 64)
    want = np.abs(wf).max(axis=2).T  # [K/64, N]
    assert np.array_equal(absmax, want.astype(np.float32))
    c = _unpack(codes).reshape(24, 4, 64)
    for n in range(24):
        for kb in range(4):
            i = np.argmax(np.abs(wf[n, kb]))
            assert c[n, kb, i] == (15 if wf[n, kb, i] > 0 else 0)


def test_codes_are_nearest_level_bruteforce(orc):
    W = synth.normal_bf16(0, "nf4.near", (64, 512), 0.02)
    codes, absmax = orc.quantize_nf4(W)
    c = _unpack(codes)
    wf = synth.bf16_bits_to_f32(W)
    amax = np.repeat(absmax.T, 64, axis=1)  # [N, K]
    v = (wf / amax).astype(np.float32).astype(np.float64)   # IEEE fp32 division
    lv = orc.nf4_levels().astype(np.float64)
    dist = np.abs(v[..., None] - lv[None, None, :])
    best = dist.min(axis=-1)
    got = dist[np.arange(64)[:, None], np.arange(512)[None, :], c]
    # nearest up to the fp32 rounding of the midpoints
    assert np.all(got <= best + 1e-7)
    # ties (to 1e-7) are rare; away from them the code is the unique argmin
    assert np.mean(c == dist.argmin(axis=-1)) > 0.9999


def test_codes_monotone_within_block(orc):
    W = synth.normal_bf16(0, "nf4.mono", (16, 128), 0.02)
    codes, _ = orc.quantize_nf4(W)
    c = _unpack(codes).reshape(16, 2, 64)
    wf = synth.bf16_bits_to_f32(W).reshape(16, 2, 64)
    for n in range(16):
        for kb in range(2):
            o = np.argsort(wf[n, kb], kind="stable")
            assert np.all(np.diff(c[n, kb][o].astype(int)) >= 0)


def test_zero_block_and_nibble_order(orc):
    W = np.zeros((2, 128), np.uint16)
    W[1, 64] = synth.to_bf16_bits(np.array([-0.5]))[0]   # k=64: level 0
    W[1, 65] = synth.to_bf16_bits(np.array([0.3]))[0]    # k=65: v ~ 0.6016 -> 0.5626 (13)
    codes, absmax = orc.quantize_nf4(W)
    assert np.all(codes[0] == 0x77) and np.all(absmax[:, 0] == 0)
    assert codes[1, 32] == (0 << 4) | 13
    assert absmax[1, 1] == 0.5 and absmax[0, 1] == 0.0
    Wq = orc.dequant_nf4(codes, absmax)
    assert np.all(Wq[0] == 0)


def test_dequant_is_single_rounding_of_fp32_product(orc):
    rng = np.random.default_rng(3)
    N, K = 32, 256
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    absmax = np.abs(rng.normal(0, 0.05, size=(K // 64, N))).astype(np.float32)
    Wq = orc.dequant_nf4(codes, absmax)
    c = _unpack(codes)
    lv = orc.nf4_levels()
    prod = lv[c] * np.repeat(absmax.T, 64, axis=1)   # numpy fp32 multiply
    assert np.array_equal(Wq, synth.to_bf16_bits(prod))
    # end codes reproduce +-bf16(absmax), code 7 is an exact zero
    a = np.repeat(absmax.T, 64, axis=1)
    sel15 = c == 15
    assert np.array_equal(synth.bf16_bits_to_f32(Wq)[sel15],
                          synth.bf16_bits_to_f32(synth.to_bf16_bits(a[sel15])))
    assert np.all(Wq[c == 7] == 0)


def test_quantisation_error_bound(orc):
    W = synth.normal_bf16(0, "nf4.err", (32, 512), 0.02)
    codes, absmax = orc.quantize_nf4(W)
    Wq = orc.dequant_nf4(codes, absmax)
    lv = orc.nf4_levels().astype(np.float64)
    gap = np.max(np.diff(lv))
    a = np.repeat(absmax.T, 64, axis=1).astype(np.float64)
    err = np.abs(synth.bf16_bits_to_f32(W).astype(np.float64)
                 - synth.bf16_bits_to_f32(Wq).astype(np.float64))
    assert np.all(err <= a * (gap / 2 + 2.0 ** -8) + 1e-12)
