"""The fp32 block-sparse tensor-core path forms every product from fp16 (hi, lo) splits of
power-of-two scaled operands. These CPU checks restate that number format (the shift rule,
the split, the three-term product) in numpy and bound its error, independently of the GPU
and of the oracle."""
import numpy as np


def scale_shift(m):
    """Shift s that brings a largest magnitude m into [2^14, 2^15), at most 120."""
    e = int((np.float32(m).view(np.uint32) >> 23) & 0xFF)
    return min(141 - e, 120)


def split(x):
    """fp16 hi = fp16(x), lo = fp16(x - hi) of an fp32 array already scaled."""
    x = np.asarray(x, dtype=np.float32)
    hi = x.astype(np.float16)
    lo = (x - hi.astype(np.float32)).astype(np.float16)
    return hi, lo


def three_term_dot(q, K):
    """<q, k_j> for every row of K from the scaled splits: hi.hi + hi.lo + lo.hi summed in
    fp64 (the tensor core sums exact fp16 products in fp32; fp64 isolates the split error),
    scaled back by the exact powers of two."""
    sq = scale_shift(np.abs(q).max())
    sk = scale_shift(np.abs(K).max())
    qh, ql = split(q * np.float32(2.0 ** sq))
    kh, kl = split(K * np.float32(2.0 ** sk))
    f = lambda a, b: b.astype(np.float64) @ a.astype(np.float64)
    return (f(qh, kh) + f(qh, kl) + f(ql, kh)) * 2.0 ** -(sq + sk)


def test_shift_puts_the_largest_magnitude_in_range():
    rng = np.random.default_rng(0)
    for e in range(-100, 101, 7):
        m = np.float32(rng.uniform(1.0, 2.0) * 2.0 ** e)
        s = scale_shift(m)
        scaled = float(m) * 2.0 ** s
        assert 2.0 ** 14 <= scaled < 2.0 ** 15, (e, s)
        assert np.float16(np.float32(scaled)) < np.inf
    # zero and the smallest magnitudes: the shift is clamped, 2^s stays a finite float
    assert scale_shift(0.0) == 120 and np.isfinite(np.float32(2.0 ** 120))
    assert scale_shift(np.float32(2.0 ** -120)) == 120
    # the largest finite float still gives a representable 2^-s
    assert np.isfinite(np.float32(2.0 ** -scale_shift(np.float32(3.0e38))))


def test_split_keeps_22_bits_over_the_scaled_range():
    # magnitudes from 2^-2 (lo still a normal fp16 number) up to the 2^15 ceiling
    rng = np.random.default_rng(1)
    sign = np.where(rng.random(200000) < 0.5, -1.0, 1.0)
    x = (sign * 2.0 ** rng.uniform(-2, 15, 200000)).astype(np.float32)
    hi, lo = split(x)
    rel = np.abs(hi.astype(np.float64) + lo.astype(np.float64) - x.astype(np.float64))
    rel /= np.abs(x.astype(np.float64))
    assert rel.max() <= 2.0 ** -21


def test_three_term_product_is_fp32_accurate_at_any_magnitude():
    rng = np.random.default_rng(2)
    for eq, ek in ((0, 0), (40, -40), (-50, 45), (90, -100), (-110, 20)):
        q = (rng.standard_normal(128) * 2.0 ** eq).astype(np.float32)
        K = (rng.standard_normal((64, 128)) * 2.0 ** ek).astype(np.float32)
        K[::7] *= np.float32(2.0 ** -6)   # rows of smaller magnitude inside the block
        got = three_term_dot(q, K)
        ref = K.astype(np.float64) @ q.astype(np.float64)
        scale = np.linalg.norm(q.astype(np.float64)) * np.linalg.norm(K.astype(np.float64), axis=1)
        assert (np.abs(got - ref) / scale).max() <= 2.0 ** -20, (eq, ek)


def test_weight_split_with_the_2_to_14_factor():
    # P' = 2^14 P for P in [0, 1]: hi + lo within 2^-21 of P' for every weight whose lo
    # part is a normal fp16 number (P' >= 2^-2), and within 2^-24 absolutely below that
    # (2^-38 of the largest weight)
    rng = np.random.default_rng(3)
    p = np.concatenate([rng.uniform(0, 1, 100000), 2.0 ** -rng.uniform(0, 40, 100000), [0.0, 1.0]])
    pp = (p * 2.0 ** 14).astype(np.float32)
    hi, lo = split(pp)
    err = np.abs(hi.astype(np.float64) + lo.astype(np.float64) - pp.astype(np.float64))
    big = pp >= 2.0 ** -2
    assert (err[big] / pp[big]).max() <= 2.0 ** -21
    assert err[~big].max() <= 2.0 ** -24
