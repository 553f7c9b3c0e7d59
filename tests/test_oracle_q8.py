"""Pins of the oracle's int8 key quantiser and its logit error bound.

RetrievalAttention review, Appendix C "CPU memory minimization" (8-bit
scalar quantisation of keys, scheme unspecified) and the future-work item
"Scalar quantization of KV vectors with accuracy-preservation guarantees"
(per-channel symmetric is one of the schemes it names; the concern is that
quantised keys shift the nearest-neighbour ranking, which the exact
rescoring of the quantised scan's shortlist removes).

Checked against closed forms (an exact grid of multiples of the scale, ties
to even, an all-zero channel, saturation of an appended value), the
invariants of the definition (codes in [1, 255], the channel maximum maps
to +-127, fitted errors at most half a step) and the bound's tightness on a
constructed row where every channel's error has the sign of q_j.
"""
import numpy as np

import oracle as orc
from test_oracle import exact_bf16, f32_to_bf16_bits, widen

rng = np.random.default_rng(4242)
D = 128


def test_exact_grid_has_zero_error():
    # maxabs = 127/16 -> s = 1/16 exactly; every k = m/16 is a code m exactly
    m = rng.integers(-127, 128, size=(64, D))
    m[0, :] = 127  # the channel maximum
    k = f32_to_bf16_bits((m / 16.0).astype(np.float32))
    assert np.array_equal(widen(k), m / 16.0)
    s, codes, err = orc.q8_fit(k)
    assert np.all(s == np.float32(1.0 / 16.0))
    assert np.array_equal(codes.astype(np.int64) - 128, m)
    assert np.all(err == 0.0)


def test_ties_go_to_even():
    # channel 0: maxabs 127 -> s = 1; 2.5 -> 2, 3.5 -> 4, -2.5 -> -2, -3.5 -> -4
    vals = [127.0, 2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 1.5]
    k = np.zeros((len(vals), D), np.uint16)
    for i, v in enumerate(vals):
        k[i, 0] = exact_bf16(v)
    s, codes, err = orc.q8_fit(k)
    assert s[0] == np.float32(1.0)
    got = codes[:, 0].astype(np.int64) - 128
    assert got.tolist() == [127, 2, 4, -2, -4, 0, 0, 2]
    assert err[0] == 0.5


def test_zero_channel():
    k = f32_to_bf16_bits(rng.standard_normal((32, D)).astype(np.float32))
    k[:, 7] = 0
    s, codes, err = orc.q8_fit(k)
    assert s[7] == 0.0 and err[7] == 0.0
    assert np.all(codes[:, 7] == 128)
    # an appended nonzero value on a zero-scale channel keeps code 0 and
    # its whole magnitude is the error
    extra = np.zeros((1, D), np.uint16)
    extra[0, 7] = exact_bf16(-3.0)
    c2, e2 = orc.q8_append(extra, s, err)
    assert c2[0, 7] == 128 and e2[7] == 3.0


def test_fit_invariants_random():
    x = 0.7 + rng.standard_normal((500, D)) * (0.5 + 1.5 * rng.random(D))
    k = f32_to_bf16_bits(x.astype(np.float32))
    kd = widen(k)
    s, codes, err = orc.q8_fit(k)
    maxabs = np.abs(kd).max(axis=0)
    # s is the binary32 quotient maxabs / 127 (the decision's precision)
    assert np.array_equal(s, (maxabs.astype(np.float32) / np.float32(127.0)).astype(np.float32))
    assert codes.min() >= 1 and codes.max() <= 255
    c = codes.astype(np.int64) - 128
    arg = np.abs(kd).argmax(axis=0)
    assert np.all(np.abs(c[arg, np.arange(D)]) == 127)
    assert np.all(np.sign(c[arg, np.arange(D)]) == np.sign(kd[arg, np.arange(D)]))
    # fitted rows: at most half a step, up to the binary32 rounding of k/s
    # (|k/s| <= 127, so that quotient is off by at most 127 * 2^-24 steps: a
    # value just below a half-way point can round onto it and go to even)
    sd = s.astype(np.float64)
    resid = np.abs(kd - sd * c)
    assert np.all(resid <= sd * (0.5 + 2.0 ** -16))
    assert np.array_equal(err, resid.max(axis=0))
    # the code is the nearest multiple, up to the same rounding
    for dc in (-1, 1):
        alt = np.clip(c + dc, -127, 127)
        assert np.all(np.abs(kd - sd * alt) >= resid - sd * 2.0 ** -16)


def test_append_saturates_and_updates_error():
    k = f32_to_bf16_bits(rng.standard_normal((100, D)).astype(np.float32))
    s, codes, err = orc.q8_fit(k)
    kd = widen(k)
    maxabs = np.abs(kd).max(axis=0)
    big = f32_to_bf16_bits((np.where(np.arange(D) % 2 == 0, 3.0, -3.0) * maxabs)
                           .astype(np.float32)[None, :])
    c2, e2 = orc.q8_append(big, s, err)
    c = c2[0].astype(np.int64) - 128
    assert np.all(c[0::2] == 127) and np.all(c[1::2] == -127)
    bd = widen(big)[0]
    expect = np.abs(bd) - 127.0 * s.astype(np.float64)
    assert np.allclose(e2, np.maximum(err, expect), rtol=0, atol=0)
    # the input error array is left alone; a second append of nothing keeps it
    c3, e3 = orc.q8_append(np.zeros((0, D), np.uint16), s, e2)
    assert c3.shape == (0, D) and np.array_equal(e3, e2)


def test_bound_holds_on_every_row():
    x = 0.3 + rng.standard_normal((800, D)) * (0.5 + 1.5 * rng.random(D))
    k = f32_to_bf16_bits(x.astype(np.float32))
    s, codes, err = orc.q8_fit(k)
    kd = widen(k)
    deq = s.astype(np.float64) * (codes.astype(np.int64) - 128)
    scale = 1.0 / np.sqrt(D)
    for _ in range(5):
        q = f32_to_bf16_bits(rng.standard_normal(D).astype(np.float32) * 2)
        qd = widen(q)
        z = scale * (kd @ qd)
        zh = scale * (deq @ qd)
        eps = orc.q8_bound(q, scale, err)
        assert np.all(np.abs(z - zh) <= eps * (1 + 1e-12))
        # and it is not vacuous: within a factor of the channels' worst case
        assert eps <= scale * np.abs(qd) @ (s.astype(np.float64) * 0.5) * (1 + 1e-9)


def test_bound_is_attained():
    # row 0 fixes the scales (maxabs 127/16 -> s = 1/16), row 1 sits a
    # quarter step off the grid on every channel, alternating sides; a query
    # with q_j of the error's sign makes the logit error equal the bound
    sgn = np.where(np.arange(D) % 3 == 0, -1.0, 1.0)
    row0 = np.full(D, 127.0 / 16.0)
    base = rng.integers(-31, 32, size=D) / 16.0  # (4m +- 1)/64: exact in bf16
    row1 = base + sgn * (1.0 / 64.0)
    k = f32_to_bf16_bits(np.stack([row0, row1]).astype(np.float32))
    assert np.array_equal(widen(k)[1], row1)
    s, codes, err = orc.q8_fit(k)
    assert np.all(err == 1.0 / 64.0)
    mag = 1.0 + rng.integers(0, 4, size=D)  # small integers: every sum is exact
    q = f32_to_bf16_bits((sgn * mag).astype(np.float32))
    scale = 0.125
    eps = orc.q8_bound(q, scale, err)
    assert eps == scale * np.sum(mag) / 64.0
    kd = widen(k)
    deq = 1.0 / 16.0 * (codes.astype(np.int64) - 128)
    gap = scale * (kd[1] @ widen(q)) - scale * (deq[1] @ widen(q))
    assert gap == eps
