"""Host check of the argument behind the nucleus kernel's bf16 prefilter.

Pass C of nucleus_row_kernel scans a row for the tokens of one bin, whose
logits lie in a range [zl, zh] of bf16 values. For bf16 rows a 16-byte
vector passes the prefilter when, for one of its elements v, the sign bit
of q = (v - c)^2 - rr is set. There d = v - c is rounded to bf16 and
q = d d - rr is rounded once (a packed bf16 FMA). c, rb and rr come from
zl and zh as the kernel's NearBf16 takes them:
  c  = bf16_rn(f32(0.5 zl + 0.5 zh))
  rb = bf16_ru(max(f32_ru(zh - c), f32_ru(c - zl)))
  rr = max(bf16_ru(f32_ru(f32_ru(rb rb) (1 + 2^-7))), 2^-100)
The exact test that follows keeps only the tokens in [zl, zh], so the
prefilter may pass more tokens but must never drop one. Here the roundings
are emulated in float64, and every bf16 value v in [zl, zh] is checked to
give d^2 < rr (so q < 0), over many ranges. Among them are one-value ranges,
ranges across zero, negative ranges and wide ones. Values far outside the
range must fail, so the filter is not vacuous.

Results on the GPU are covered by the top-p parity tests, and the outputs
do not depend on the prefilter (it only decides which vectors get the exact
test)."""
import numpy as np


def _round_bits(x, bits, up):
    """x (float64, finite, normal or zero) rounded to `bits` significant bits:
    to nearest even, or up (toward +inf) when `up`."""
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    s = m * 2.0 ** bits
    s = np.ceil(s) if up else np.rint(s)
    return np.ldexp(s, e - bits)


def _bf16_rn(x):
    return _round_bits(x, 8, False)


def _bf16_ru(x):
    return _round_bits(x, 8, True)


def _f32_ru(x):
    return _round_bits(x, 24, True)


def _all_finite_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):   # the NaN patterns, dropped below
        v = (bits << 16).view(np.float32).astype(np.float64)
    v = v[np.isfinite(v)]
    return np.unique(v)  # sorted; -0 and +0 merge


ALL = _all_finite_bf16()


def _near_params(zl, zh):
    mid = np.float32(0.5) * np.float32(zl) + np.float32(0.5) * np.float32(zh)
    c = float(_bf16_rn(float(mid)))
    rb = float(_bf16_ru(max(float(_f32_ru(zh - c)), float(_f32_ru(c - zl)))))
    rr = float(_f32_ru(float(_f32_ru(rb * rb)) * (1.0 + 2.0 ** -7)))
    rr = max(float(_bf16_ru(rr)), 2.0 ** -100)
    return c, rb, rr


def _passes(v, c, rr):
    d = _bf16_rn(v - c)
    return d * d < rr


def _ranges(seed=7, n=3000):
    rng = np.random.default_rng(seed)
    finite = ALL[np.abs(ALL) <= 300.0]
    out = []
    for _ in range(n):
        i = int(rng.integers(0, finite.size))
        width = int(rng.choice([0, 1, 2, 3, 7, 15, 31, 63, 127, 255, 256, 511, 2000]))
        j = min(i + width, finite.size - 1)
        out.append((float(finite[i]), float(finite[j])))
    # ranges around zero, tiny magnitudes and single values at the extremes
    z0 = int(np.searchsorted(finite, 0.0))
    for w in (1, 5, 40, 300, 3000):
        out.append((float(finite[max(z0 - w, 0)]), float(finite[min(z0 + w, finite.size - 1)])))
    out += [(float(finite[0]), float(finite[0])), (float(finite[-1]), float(finite[-1])),
            (-1.0, -1.0), (0.0, 0.0), (2.0 ** -90, 2.0 ** -90)]
    return out


def test_every_value_in_the_range_passes():
    bad = []
    for zl, zh in _ranges():
        c, rb, rr = _near_params(zl, zh)
        v = ALL[(ALL >= zl) & (ALL <= zh)]
        assert v.size >= 1
        ok = _passes(v, c, rr)
        if not ok.all():
            bad.append((zl, zh, float(v[~ok][0])))
    assert not bad, f"values in range rejected: {bad[:5]}"


def test_values_far_outside_fail():
    """Not vacuous: a value more than twice the half-width rb from the centre
    (or, for rb = 0, more than 2^-49 from it) never passes."""
    for zl, zh in _ranges(seed=11, n=500):
        c, rb, rr = _near_params(zl, zh)
        far = ALL[np.abs(ALL - c) > 2.0 * rb + 2.0 ** -49]
        if far.size:
            assert not _passes(far, c, rr).any(), (zl, zh)


def test_emulated_roundings():
    # to nearest even at 8 bits, and upward
    assert _bf16_rn(1.0 + 2.0 ** -8) == 1.0          # a tie goes to even
    assert _bf16_rn(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert _bf16_ru(1.0 + 2.0 ** -20) == 1.0 + 2.0 ** -7
    assert _f32_ru(1.0 + 2.0 ** -40) == 1.0 + 2.0 ** -23
    # every bf16 value is a fixed point of both roundings
    v = ALL[np.abs(ALL) < 1e30]
    assert np.array_equal(_bf16_rn(v), v) and np.array_equal(_bf16_ru(v), v)
