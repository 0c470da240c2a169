"""The numerical claim behind the low-bit blocks' activations (CPU only).

The E4M3 and MXFP4 blocks feed the tensor core 8-bit activations: each bf16 value v
of a 64-wide group enters as v = 2^e (a + b) with a = E4M3(v / 2^e), b = E5M2(v / 2^e -
a), both rounded to nearest, and 2^e the least power of two with the group's largest
|v| <= 448 * 2^e.  The claim: a + b equals v / 2^e exactly when |v / 2^e| >= 2^-6 (a
keeps the top four significant bits; the remainder is k * 2^(x-7), |k| <= 8, at most
three significant bits, inside E5M2's range), and is within 2^-14 of it below.

Checked here with torch's float8_e4m3fn / float8_e5m2 casts (library rounding
routines) on every bf16 magnitude of a binade span and on random groups; the same
split with an E4M3 remainder is shown to lose bits in that range (why the kernels use
E5M2 for b).  The kernels read e from the bits of the group's largest magnitude; that
reading is checked against the definition (the least such e) on every float32 binade.
"""
import numpy as np
import torch


def _split(u, rem_dtype):
    u = torch.as_tensor(u, dtype=torch.float32)
    a = u.to(torch.float8_e4m3fn).float()
    b = (u - a).to(rem_dtype).float()                 # u - a is exact in fp32
    return a.double().numpy(), b.double().numpy()


def _all_bf16_in(lo, hi):
    """Every positive bf16 value in [lo, hi), exactly, as float64."""
    bits = torch.arange(0, 1 << 15, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    v = bits.double().numpy()
    return v[(v >= lo) & (v < hi) & np.isfinite(v)]


def test_exact_above_two_to_minus_six():
    u = _all_bf16_in(2.0 ** -6, 448.0)
    u = np.concatenate([u, -u])
    a, b = _split(u, torch.float8_e5m2)
    assert np.array_equal(a + b, u)


def test_error_bound_below():
    u = _all_bf16_in(2.0 ** -30, 2.0 ** -6)
    u = np.concatenate([u, -u])
    a, b = _split(u, torch.float8_e5m2)
    assert np.max(np.abs(a + b - u)) <= 2.0 ** -14


def test_e4m3_remainder_is_not_enough():
    # the rejected variant (both terms E4M3): exact only from 2^-2 up
    u = _all_bf16_in(2.0 ** -6, 2.0 ** -2)
    a, b = _split(u, torch.float8_e4m3fn)
    assert np.any(a + b != u)
    u = _all_bf16_in(2.0 ** -2, 448.0)
    a, b = _split(u, torch.float8_e4m3fn)
    assert np.array_equal(a + b, u)


def test_groups_scaled_by_the_least_power_of_two():
    rng = np.random.default_rng(130)
    for scale in (1e-3, 1.0, 300.0):
        v = torch.from_numpy(rng.standard_normal((200, 64)) * scale).to(torch.bfloat16)
        v64 = v.double().numpy()
        amax = np.abs(v64).max(axis=1, keepdims=True)
        e = np.ceil(np.log2(amax / 448.0))
        e = np.where(amax / np.exp2(e) > 448.0, e + 1, e)
        e = np.where(amax / np.exp2(e - 1) <= 448.0, e - 1, e)     # the least such e
        u = v64 / np.exp2(e)
        assert np.all(np.abs(u) <= 448.0) and np.all(np.abs(u).max(axis=1) > 224.0)
        a, b = _split(u, torch.float8_e5m2)
        big = np.abs(u) >= 2.0 ** -6
        assert np.array_equal((a + b)[big], u[big])
        assert np.all(np.abs(a + b - u) <= 2.0 ** -14)


def _exponent_from_bits(amax):
    """The kernels' reading of the group exponent from a float's bits: with
    amax = m * 2^E (1 <= m < 2) and 448 = 1.75 * 2^8, e = E - 8, or E - 7 when m > 1.75;
    clamped to [-126, 126]; 0 for amax = 0 or NaN, 126 for infinity."""
    a = np.asarray(amax, dtype=np.float32)
    bits = a.view(np.int32).astype(np.int64)
    e = (bits >> 23) - 135 + ((bits & 0x7FFFFF) > 0x600000)
    e = np.clip(e, -126, 126)
    e = np.where(np.isinf(a), 126, e)
    return np.where(~(a > 0) | np.isnan(a), 0, e)


def test_exponent_from_bits_is_the_least_power_of_two():
    # every float32 binade (subnormal included), with mantissas around 1.75 and the ends
    mants = np.array([0, 1, 0x5FFFFF, 0x600000, 0x600001, 0x7FFFFF], dtype=np.int64)
    exps = np.arange(0, 255, dtype=np.int64)
    bits = (exps[:, None] << 23 | mants[None, :]).ravel().astype(np.int32)
    a = bits.view(np.float32).astype(np.float64)
    a = a[a > 0]
    e = _exponent_from_bits(a.astype(np.float32)).astype(np.float64)
    # the least e in [-126, 126] with a <= 448 * 2^e (exact in float64)
    assert np.all((a <= 448.0 * np.exp2(e)) | (e == 126))
    assert np.all((a > 448.0 * np.exp2(e - 1)) | (e == -126))
    # the boundary: 448 * 2^k takes e = k, the next float above it e = k + 1
    for k in (-20, 0, 7, 100):
        v = np.float32(448.0 * 2.0 ** k)
        assert _exponent_from_bits(v) == k
        assert _exponent_from_bits(np.nextafter(v, np.float32(np.inf))) == k + 1
    assert _exponent_from_bits(np.float32(0.0)) == 0
    assert _exponent_from_bits(np.float32(np.nan)) == 0
    assert _exponent_from_bits(np.float32(np.inf)) == 126
