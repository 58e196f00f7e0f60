"""Pins for the oracle's compression arithmetic and attention (no GPU).

What each test ties the oracle to:
  quantizer      exhaustive search over every code with exact rationals;
                 torch's E4M3 cast for the metadata; the textbook error bound
  LS coefficient brute-force grid search and golden-section search
  rotation       orthogonality / norm preservation of the seeded R
  residual       zero-residual special case reached exactly; the
                 reconstruction error equals the residual quantization error
                 (R orthogonal), which a wrong sign, a dropped c or R used
                 in place of R^T all break
  attention      one key, identical keys, scipy's softmax
"""
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

import synth
from oracle import formats as F
from oracle import method as M


def _e4m3_torch(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def _nearest_e4m3_exact(t: Fraction) -> float:
    """Nearest finite E4M3 value to an exact rational (ties to the even code), saturating."""
    codes = np.arange(0x7F, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mag = abs(t)
    if mag >= 448:
        return float(np.copysign(448.0, float(t)))
    dist = [abs(Fraction(float(v)) - mag) for v in vals]
    best = min(dist)
    ks = [k for k in range(len(vals)) if dist[k] == best]
    k = ks[0] if len(ks) == 1 else [k for k in ks if k % 2 == 0][0]
    return float(np.copysign(vals[k], float(t))) if t != 0 else 0.0


@pytest.mark.parametrize("bits", [4, 2])
def test_quantizer_codes_are_exact_nearest_grid_points(bits):
    """Exhaustive: the metadata is the exact nearest E4M3 value of min and of
    range / (2^bits - 1); every code is the nearest grid point o + k s among
    all 2^bits codes (exact rationals), ties to the even code."""
    rng = np.random.default_rng(10 + bits)
    g = 8
    qmax = (1 << bits) - 1
    for trial in range(150):
        v = rng.standard_normal((4, g)).astype(np.float32).astype(np.float64)
        if trial % 5 == 0:   # put some values on a coarse grid
            v[1] = np.round(v[1] * 4) / 4
        # a group whose scale and offset are E4M3-exact and whose inner values sit
        # exactly halfway between grid points: the code must be the even neighbour
        s_t = [0.25, 0.125, 0.5, 0.0625][trial % 4]
        o_t = [0.0, -1.0, 0.5, -2.0][(trial // 4) % 4]
        k_t = rng.integers(0, qmax, size=g - 2)
        v[2] = np.concatenate([[o_t, o_t + qmax * s_t], o_t + (k_t + 0.5) * s_t])
        codes, s_b, o_b = M.quantize(v, bits, g)
        s = F.e4m3_decode(s_b)[:, 0]
        o = F.e4m3_decode(o_b)[:, 0]
        for row in range(v.shape[0]):
            lo, hi = Fraction(v[row].min()), Fraction(v[row].max())
            assert s[row] == _nearest_e4m3_exact((hi - lo) / qmax)
            assert o[row] == _nearest_e4m3_exact(lo)
            if s[row] == 0:
                assert np.all(codes[row] == 0)
                continue
            fo, fs = Fraction(o[row]), Fraction(s[row])
            for i in range(g):
                fv = Fraction(v[row, i])
                dist = [abs(fv - (fo + k * fs)) for k in range(qmax + 1)]
                best = min(dist)
                ks = [k for k in range(qmax + 1) if dist[k] == best]
                want = ks[0] if len(ks) == 1 else [k for k in ks if k % 2 == 0][0]
                assert codes[row, i] == want, (v[row, i], o[row], s[row], codes[row, i], want)


def test_quantizer_constant_group():
    v = np.full((3, 32), 0.7109375)           # a BF16 value, not an E4M3 value
    codes, s_b, o_b = M.quantize(v, 4, 32)
    assert np.all(codes == 0)
    assert np.all(F.e4m3_decode(s_b) == 0.0)
    xhat = M.dequantize(codes, s_b, o_b, 32)
    assert np.all(xhat == F.e4m3_round(0.7109375))


def test_quantizer_error_bound():
    """|v - v_hat| <= s/2 for every element inside the grid's span; elements
    past the span (offset/scale rounding) are clamped to the end codes."""
    rng = np.random.default_rng(11)
    for bits in (4, 2):
        v = (rng.standard_normal((2000, 32)) * rng.uniform(0.01, 20, (2000, 1))).astype(np.float32).astype(np.float64)
        codes, s_b, o_b = M.quantize(v, bits, 32)
        xhat = M.dequantize(codes, s_b, o_b, 32)
        s = F.e4m3_decode(s_b)[:, :, None].repeat(32, 2).reshape(v.shape)
        o = F.e4m3_decode(o_b)[:, :, None].repeat(32, 2).reshape(v.shape)
        qmax = (1 << bits) - 1
        inside = (v >= o) & (v <= o + qmax * s)
        assert np.all(np.abs(v - xhat)[inside] <= s[inside] / 2)
        assert np.all(codes[(v < o)] == 0)
        assert np.all(codes[(v > o + qmax * s)] == qmax)


def test_ls_coefficient_minimises_squared_error():
    rng = np.random.default_rng(12)
    for _ in range(50):
        y = rng.standard_normal(128)
        x = 0.8 * y + 0.3 * rng.standard_normal(128)
        c = float(M.ls_coefficient(x, y))
        f = lambda cc: float(np.sum((x - cc * y) ** 2))
        grid = np.linspace(c - 1, c + 1, 10001)
        errs = np.array([f(cc) for cc in grid])
        assert errs.min() >= f(c) - 1e-9
        assert abs(grid[errs.argmin()] - c) <= 2e-4
        # golden-section search on [-3, 3] lands on c
        a, b = -3.0, 3.0
        gr = (np.sqrt(5) - 1) / 2
        for _ in range(200):
            c1, c2 = b - gr * (b - a), a + gr * (b - a)
            if f(c1) < f(c2):
                b = c2
            else:
                a = c1
        assert abs((a + b) / 2 - c) < 1e-7
    assert float(M.ls_coefficient(np.ones(8), np.zeros(8))) == 0.0


def test_rotation_is_orthogonal():
    for d in (96, 128):
        R = synth.rotation(d, seed=0)
        assert np.abs(R.T @ R - np.eye(d)).max() < 1e-13
        assert np.all(np.diag(np.linalg.qr(np.random.default_rng(np.random.PCG64(0)).standard_normal((d, d)))[1]) != 0)
        u = np.random.default_rng(5).standard_normal((10, d))
        assert np.allclose(np.linalg.norm(u @ R.T, axis=1), np.linalg.norm(u, axis=1), rtol=1e-13)
        q = np.random.default_rng(6).standard_normal(d)
        # query-side rotation identity: (R q) . (R u) == q . u
        assert np.allclose((R @ q) @ (u @ R.T).T, q @ u.T, rtol=1e-12, atol=1e-12)


def _grid_anchor(rng, d=128, g=32):
    """An anchor already on the INT4 grid with E4M3-exact scale and offset per group,
    every group spanning its full 0..15 range."""
    ng = d // g
    s = np.array([0.25, 0.125, 0.5, 0.0625])[:ng]
    o = np.array([-2.0, -1.0, -4.0, -0.5])[:ng]
    codes = rng.integers(0, 16, size=(ng, g))
    codes[:, 0], codes[:, 1] = 0, 15
    return (s[:, None] * codes + o[:, None]).reshape(d), codes.reshape(d)


def test_zero_residual_is_reached_exactly():
    """x_l = 0.75 * anchor with the anchor on its INT4 grid: c = 0.75 exactly (BF16-exact),
    the residual is 0, its codes and scale are 0, and the loop is rebuilt exactly."""
    rng = np.random.default_rng(13)
    a, a_codes = _grid_anchor(rng)
    R = synth.rotation(128)
    x = np.stack([0.75 * a, 0.75 * a, 0.75 * a, a])
    comp = M.compress_group(x, R, 32)
    assert np.array_equal(comp["anchor"][0], a_codes)
    for j in range(3):
        r_codes, r_s, r_o, c_bits = comp["res"][j]
        assert float(F.bf16_decode(c_bits)) == 0.75
        assert np.all(comp["u"][j] == 0.0)
        assert np.all(r_codes == 0) and np.all(F.e4m3_decode(r_s) == 0) and np.all(F.e4m3_decode(r_o) == 0)
        assert np.array_equal(comp["recon"][j], x[j])


@pytest.mark.parametrize("chained", [False, True])
def test_reconstruction_error_is_the_residual_quantization_error(chained):
    """With R orthogonal, x_l - x_hat_l = R^T (u - r_hat): its norm equals the
    residual's quantization error, which is at most s/2 per element."""
    w = synth.WORKLOADS["toy"]
    _, kv = synth.looped_kv(0, w, batch=1, ntok=64)
    R = synth.rotation(128)
    comp = M.compress_group(kv, R, 32, chained=chained, precision="f64")
    for j in range(3):
        r_codes, r_s, r_o, _ = comp["res"][j]
        r_hat = M.dequantize(r_codes, r_s, r_o, 32)
        err_u = np.linalg.norm(comp["u"][j] - r_hat, axis=-1)
        err_x = np.linalg.norm(kv[j] - comp["recon"][j], axis=-1)
        assert np.allclose(err_x, err_u, rtol=1e-10, atol=1e-12)
        s = F.e4m3_decode(r_s)
        assert np.all(np.abs(comp["u"][j] - r_hat).reshape(r_codes.shape[:-1] + (4, 32)).max(-1) <= s / 2 + 1e-12)
        # the ablation's direction (ai4snews summary, Figure 1 ladder): coding the
        # rotated residual beats coding the loop directly at the same 2 bits
        rel = np.linalg.norm(kv[j] - comp["recon"][j]) / np.linalg.norm(kv[j])
        direct = M.dequantize(*M.quantize(kv[j], 2, 32), 32)
        rel_direct = np.linalg.norm(kv[j] - direct) / np.linalg.norm(kv[j])
        assert rel < 0.5 * rel_direct


def test_norm_ratio_coefficient():
    """Norm ratio ||x|| / ||y||: exact for x = lambda * y (lambda a power of two),
    equal to a separately computed norm quotient, 0 for a zero reference."""
    rng = np.random.default_rng(5)
    y = rng.standard_normal((3, 128)).astype(np.float32).astype(np.float64)
    for lam in (0.5, -2.0, 4.0):      # powers of two scale every rounded sum exactly
        c = M.norm_ratio_coefficient(lam * y, y)
        assert np.all(c == abs(lam))
    for lam in (0.75, -1.5, 3.0):
        c = M.norm_ratio_coefficient(lam * y, y)
        assert np.allclose(c, abs(lam), rtol=1e-15, atol=0)
    x = rng.standard_normal((3, 128))
    c = M.norm_ratio_coefficient(x, y)
    want = np.linalg.norm(x, axis=-1) / np.linalg.norm(y, axis=-1)
    assert np.allclose(c, want, rtol=1e-14, atol=0)
    assert float(M.norm_ratio_coefficient(np.ones(8), np.zeros(8))) == 0.0
    assert float(M.norm_ratio_coefficient(np.zeros(8), np.ones(8))) == 0.0


@pytest.mark.parametrize("chained", [False, True])
def test_compress_group_stores_the_norm_ratio(chained):
    """In norm-ratio mode the stored BF16 coefficient of every loop is the norm ratio
    of that loop against its reference (the dequantized anchor, or the rebuilt
    next loop when chained), and never negative."""
    _, kv = synth.looped_kv(8, synth.WORKLOADS["toy"], batch=1, ntok=5)
    R = synth.rotation(128).astype(np.float32).astype(np.float64)
    x = kv[:, 0]                                      # K: [P, 1, H, n, d]
    comp = M.compress_group(x, R, 32, chained=chained, scaling="norm")
    P = x.shape[0]
    for j in range(P - 1):
        ref = comp["recon"][j + 1] if chained else comp["recon"][P - 1]
        c_bits = comp["res"][j][3]
        if not chained:   # the encoder's reference is exactly the decoder's anchor
            assert np.array_equal(c_bits, F.bf16_encode(M.norm_ratio_coefficient(x[j], ref)))
        assert np.all(F.bf16_decode(c_bits) >= 0)


def test_residual_uses_bf16_coefficient_and_dequantized_anchor():
    w = synth.WORKLOADS["toy"]
    _, kv = synth.looped_kv(1, w, batch=1, ntok=8)
    R = synth.rotation(128)
    comp = M.compress_group(kv, R, 32, precision="f64")
    a_hat = M.dequantize(*comp["anchor"], 32)
    for j in range(3):
        c = M.ls_coefficient(kv[j], a_hat)
        c_bits = comp["res"][j][3]
        assert np.array_equal(c_bits, F.bf16_encode(c))
        cb = F.bf16_decode(c_bits)[..., None]
        assert np.allclose(comp["u"][j], (kv[j] - cb * a_hat) @ R.T, rtol=0, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(14)
    q = rng.standard_normal(64)
    v = rng.standard_normal((1, 64))
    k = rng.standard_normal((1, 64))
    assert np.array_equal(M.attention(q, k, v, 0.125), v[0])
    K = np.repeat(k, 7, axis=0)
    V = rng.standard_normal((7, 64))
    assert np.allclose(M.attention(q, K, V, 0.125), V.mean(0), rtol=1e-14, atol=1e-14)
    K = rng.standard_normal((300, 64)) * 3
    V = rng.standard_normal((300, 64))
    ref = scipy.special.softmax(0.125 * K @ q) @ V
    assert np.allclose(M.attention(q, K, V, 0.125), ref, rtol=1e-12, atol=1e-13)
    # log-sum-exp form
    s = 0.125 * K @ q
    lse = scipy.special.logsumexp(s)
    assert np.allclose(M.attention(q, K, V, 0.125), np.exp(s - lse) @ V, rtol=1e-12, atol=1e-13)


def test_fma_f32_is_one_rounding_of_the_exact_value():
    """Against exact rationals (Fraction) and a binary32 round-to-nearest-even
    written from the format (24-bit significand)."""
    from fractions import Fraction

    def rne32(fr):
        if fr == 0:
            return 0.0
        sgn, fr = (-1 if fr < 0 else 1), abs(fr)
        e = fr.numerator.bit_length() - fr.denominator.bit_length()
        while Fraction(2) ** e > fr:
            e -= 1
        while Fraction(2) ** (e + 1) <= fr:
            e += 1
        q = Fraction(2) ** (e - 23)
        k = fr / q
        fl = k.numerator // k.denominator
        rem = k - fl
        if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
            fl += 1
        return sgn * float(fl * q)

    # one rounding, not two: the exact a*b is halfway between two binary32 values
    # and c is far below float64's precision there, so rounding a*b + c to float64
    # first would land on the tie and send it to the even neighbour; the single
    # rounding goes the way c points.  Both directions (even neighbour below, above).
    tiny = float.fromhex("0x1p-80")
    for a, b, c in [(1 + 2.0 ** -12, 1 + 2.0 ** -12, tiny), (1 + 2.0 ** -12, 1 + 3 * 2.0 ** -12, -tiny),
                    (-(1 + 2.0 ** -12), 1 + 2.0 ** -12, -tiny)]:
        a32, b32, c32 = np.float32(a), np.float32(b), np.float32(c)
        assert float(a32) == a and float(b32) == b and float(c32) == c
        want = rne32(Fraction(a) * Fraction(b) + Fraction(c))
        assert float(F.fma_f32(a32, b32, c32)) == want
        assert want != float(np.float32(np.float64(a) * np.float64(b) + np.float64(c)))   # the trap is real

    rng = np.random.default_rng(21)
    for i in range(6000):
        a, b, c = rng.standard_normal(3).astype(np.float32)
        if i % 3 == 0:
            c = np.float32(-(np.float64(a) * np.float64(b)))     # near-total cancellation
        if i % 7 == 0:
            c = np.float32(c * 1e-8)
        want = rne32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))
        assert float(F.fma_f32(a, b, c)) == want


def test_f32_rotation_special_cases_and_error_bound():
    rng = np.random.default_rng(22)
    e = rng.standard_normal((50, 128)).astype(np.float32)
    # identity and signed permutation: exact
    assert np.array_equal(M.rotate_f32(np.eye(128, dtype=np.float32), e), e)
    perm = rng.permutation(128)
    Pm = np.zeros((128, 128), np.float32)
    Pm[np.arange(128), perm] = rng.choice([-1.0, 1.0], 128).astype(np.float32)
    assert np.array_equal(M.rotate_f32(Pm, e), e @ Pm.T)
    assert np.array_equal(M.rotate_back_f32(Pm, e), e @ Pm)
    # general R: within the textbook bound of a binary32 recursive sum, d * 2^-24 * sum|R_ik e_k|
    R = synth.rotation(128).astype(np.float32)
    u32 = M.rotate_f32(R, e).astype(np.float64)
    u64 = e.astype(np.float64) @ R.astype(np.float64).T
    bound = 128 * 2.0 ** -24 * (np.abs(e.astype(np.float64)) @ np.abs(R.astype(np.float64)).T)
    assert np.all(np.abs(u32 - u64) <= bound)
    assert np.abs(u32 - u64).max() > 0      # it is a genuinely different rounding


@pytest.mark.parametrize("chained", [False, True])
def test_f32_and_f64_readings_agree_up_to_rounding(chained):
    """The binary32 reading of the residual changes codes only where the float64
    reading sits on a rounding boundary."""
    w = synth.WORKLOADS["toy"]
    _, kv = synth.looped_kv(3, w, batch=1, ntok=64)
    R = synth.rotation(128).astype(np.float32).astype(np.float64)
    c32 = M.compress_group(kv, R, 32, chained=chained, precision="f32")
    c64 = M.compress_group(kv, R, 32, chained=chained, precision="f64")
    assert np.array_equal(c32["anchor"][0], c64["anchor"][0])
    for j in range(3):
        assert np.allclose(c32["u"][j], c64["u"][j], rtol=0, atol=1e-4)
        diff = (c32["res"][j][0] != c64["res"][j][0]).mean()
        assert diff < 1e-3


# ---- Walsh-Hadamard rotation ----

def _popcount_hadamard(d):
    """H_d by its entry formula (-1)^popcount(i & k), independent of the recursion
    and of the butterflies."""
    i = np.arange(d)
    bits = np.bitwise_and(i[:, None], i[None, :])
    pc = np.zeros_like(bits)
    for b in range(int(np.log2(d))):
        pc += (bits >> b) & 1
    return np.where(pc % 2 == 0, 1.0, -1.0)


@pytest.mark.parametrize("d", [2, 8, 128])
def test_fwht_is_the_sylvester_matrix_exactly(d):
    """On small integers every butterfly sum is exact in binary32, so the fast
    transform must equal H_d e exactly; a wrong pairing, sign or stage order fails."""
    rng = np.random.default_rng(d)
    e = rng.integers(-50, 50, size=(6, d)).astype(np.float64)
    H = _popcount_hadamard(d)
    assert np.array_equal(M.fwht_f32(e).astype(np.float64), e @ H.T)
    assert np.array_equal(M.hadamard_matrix(d) * np.sqrt(d), H)
    assert np.array_equal(H @ H.T, d * np.eye(d))


def test_hadamard_rotation_close_to_the_dense_product():
    """Random data: the binary32 transform is within a few roundings of the float64
    product, keeps norms (orthogonal), and is its own inverse (symmetric R)."""
    rng = np.random.default_rng(11)
    e = rng.standard_normal((50, 128))
    R = M.hadamard_matrix(128)
    u32 = M.hadamard_f32(e).astype(np.float64)
    u64 = e @ R.T
    assert np.abs(u32 - u64).max() <= 1e-5 * np.abs(e).max()
    assert np.allclose(np.linalg.norm(u32, axis=-1), np.linalg.norm(e, axis=-1), rtol=1e-6)
    back = M.hadamard_f32(u32).astype(np.float64)
    assert np.abs(back - e).max() <= 1e-5 * np.abs(e).max()
    assert np.float32(1.0 / np.sqrt(128)) == np.float32(float.fromhex("0x1.6a09e6p-4"))


@pytest.mark.parametrize("chained", [False, True])
def test_compress_group_with_hadamard_rotation(chained):
    """The binary32 fast-transform path and the float64 dense reading of the same
    R give the same codes except at rounding boundaries; the reconstruction
    error of a loop equals its residual's quantization error (R orthogonal,
    R^T used to rebuild)."""
    w = synth.Workload("t", 1, 4, 1, 2, 128, 32, 2, 64, synth.OURO_ALPHAS, True)
    _, kv = synth.looped_kv(3, w, batch=2, ntok=40)
    R = M.hadamard_matrix(128)
    c32 = M.compress_group(kv, R, 32, chained=chained, rotation="hadamard")
    c64 = M.compress_group(kv, R, 32, chained=chained, precision="f64", rotation="hadamard")
    same = np.mean([np.mean(c32["res"][j][0] == c64["res"][j][0]) for j in range(3)])
    assert same > 0.99
    for j in range(3):
        if chained:
            continue   # the reference itself carries the later loops' errors
        # x_j = cb a_hat + R^T u, so ||recon_j - x_j|| = ||r_hat - u|| for an orthogonal R
        r_hat = M.dequantize(*c64["res"][j][:3], 32)
        lhs = np.linalg.norm(c64["recon"][j] - kv[j], axis=-1)
        rhs = np.linalg.norm(r_hat - c64["u"][j], axis=-1)
        assert np.allclose(lhs, rhs, rtol=1e-9, atol=1e-12)
