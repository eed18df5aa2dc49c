"""The quantisers' shortcut, checked in plain fp32 on the CPU (no kernel): the
code round_half_even(fl(v / scale)) is computed as rint(fl(v * fl(1/scale)))
whenever that product lies farther than 2^-14 from every half-integer, and by
the IEEE division otherwise.  Wherever the shortcut is taken it must give the
division's integer; the test draws scales and values over the whole range the
quantiser sees (|v| <= 127.5 * scale), plus values placed next to ties."""
import numpy as np

MARGIN = np.float32(0.5) - np.float32(2.0 ** -14)


def _check(v, scale):
    v = v.astype(np.float32)
    scale = scale.astype(np.float32)
    r = (np.float32(1.0) / scale).astype(np.float32)            # RN(1/scale)
    p = (v * r).astype(np.float32)                               # RN(v * r)
    k = np.rint(p)
    fast = np.abs((p - k).astype(np.float32)) <= MARGIN
    exact = np.rint((v / scale).astype(np.float32))              # round half even of RN(v/scale)
    bad = fast & (k != exact)
    assert not bad.any(), (v[bad][:5], scale[bad][:5])
    return fast.mean()


def test_shortcut_matches_division_on_random_rows():
    rng = np.random.default_rng(0)
    n = 2_000_000
    scale = np.exp2(rng.uniform(-60, 60, n)).astype(np.float32)
    v = (rng.uniform(-127.5, 127.5, n) * scale).astype(np.float32)
    frac_fast = _check(v, scale)
    assert frac_fast > 0.999                                     # the division is rare


def test_shortcut_matches_division_next_to_ties():
    rng = np.random.default_rng(1)
    n = 1_000_000
    scale = np.exp2(rng.uniform(-30, 30, n)).astype(np.float32)
    half = rng.integers(-127, 127, n) + 0.5                     # half-integers in range
    # values whose quotient lies within a few ulp of a tie, on both sides
    q = (half * (1.0 + rng.integers(-8, 9, n) * 2.0 ** -23)).astype(np.float32)
    v = (q.astype(np.float64) * scale.astype(np.float64)).astype(np.float32)
    frac_fast = _check(v, scale)
    assert frac_fast < 0.5                                       # these mostly take the division


def test_row_maximum_codes_to_127():
    """scale = fl(amax / 127): the element equal to amax codes to exactly 127
    through either path."""
    rng = np.random.default_rng(2)
    amax = np.exp2(rng.uniform(-60, 60, 500_000)).astype(np.float32)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    r = (np.float32(1.0) / scale).astype(np.float32)
    p = (amax * r).astype(np.float32)
    assert np.all(np.rint((amax / scale).astype(np.float32)) == 127)
    assert np.all(np.abs(p - 127.0) < 2.0 ** -14)


def _static_code(v, scale):
    """The Smooth-Static shortcut: p = fl(v * fl(1/scale)); |p| >= 128 saturates;
    otherwise rint(p) clamped, unless p is within 2^-14 of a half-integer, where
    the IEEE division decides.  Returns (code, took_division)."""
    r = (np.float32(1.0) / scale).astype(np.float32)
    p = (v * r).astype(np.float32)
    sat = np.abs(p) >= np.float32(128.0)
    k = np.rint(p)
    fast = ~sat & (np.abs((p - k).astype(np.float32)) <= MARGIN)
    div = np.rint((v / scale).astype(np.float32))
    code = np.where(sat, np.copysign(np.float32(127.0), p),
                    np.clip(np.where(fast, k, div), -127, 127)).astype(np.float32)
    return code, ~sat & ~fast


def test_static_shortcut_matches_saturating_division():
    """Values far beyond the calibrated range included: the shortcut's code
    equals clamp(round_half_even(fl(v / scale)), -127, 127) everywhere."""
    rng = np.random.default_rng(3)
    n = 2_000_000
    scale = np.exp2(rng.uniform(-50, 50, n)).astype(np.float32)
    mag = np.exp2(rng.uniform(-10, 20, n)) * rng.choice([-1.0, 1.0], n)   # |v/scale| up to 2^20
    v = (mag * scale.astype(np.float64)).astype(np.float32)
    # and values next to the saturation boundary 127.5 and to ties inside it
    m = 200_000
    edge = (np.float32(127.5) * (1.0 + rng.integers(-6, 7, m) * 2.0 ** -23)).astype(np.float32)
    v[:m] = (edge.astype(np.float64) * scale[:m].astype(np.float64)
             * rng.choice([-1.0, 1.0], m)).astype(np.float32)
    finite = np.isfinite(v) & (v != 0)
    v, scale = v[finite], scale[finite]
    code, _ = _static_code(v, scale)
    ref = np.clip(np.rint((v / scale).astype(np.float32)), -127, 127)
    bad = code != ref
    assert not bad.any(), (v[bad][:5], scale[bad][:5])
