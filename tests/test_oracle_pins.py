"""Pins for the fp64 CPU oracle: each check ties an oracle function to
something other than itself -- the pages' printed values, a library routine
(scipy's Sylvester Hadamard matrix, numpy's IEEE float16 conversion, scipy
quadrature), exact rational arithmetic, brute force over every candidate
code, closed forms and invariants.  A dropped term, a wrong sign, a swapped
index or an off-by-one in a rounding rule fails at least one of them."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.integrate
import scipy.linalg
import scipy.stats

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# storage formats
# --------------------------------------------------------------------------

def _all_bf16_values():
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        f = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    return bits.astype(np.uint16), f


def test_bf16_decode_and_roundtrip_exhaustive():
    bits, vals = _all_bf16_values()
    for b, v in zip(bits[::97], vals[::97]):
        got = O.bf16_to_f64(int(b))
        if math.isnan(v):
            assert math.isnan(got)
            continue
        assert got == v
        if math.isfinite(v):
            assert O.f64_to_bf16(v) == int(b)


def _nearest_bf16_bruteforce(x, table, table_bits):
    """Nearest finite bf16 by exhaustive search, ties to the even pattern."""
    i = np.searchsorted(table, x)
    cands = [j for j in (i - 1, i) if 0 <= j < len(table)]
    best = min(cands, key=lambda j: (abs(Fraction(table[j]) - Fraction(x)), int(table_bits[j]) & 1))
    return int(table_bits[best])


def test_bf16_rounding_against_bruteforce():
    bits, vals = _all_bf16_values()
    pos = np.isfinite(vals) & (vals >= 0) & ~((bits == 0x8000))
    pb, pv = bits[pos], vals[pos]
    order = np.argsort(pv, kind="stable")
    pb, pv = pb[order], pv[order]
    rng = np.random.default_rng(1)
    xs = list(np.exp(rng.uniform(np.log(1e-40), np.log(3e38), 3000)))
    # exact midpoints between neighbours (ties) and points just beside them
    for j in rng.integers(0, len(pv) - 1, 400):
        mid = (pv[j] + pv[j + 1]) / 2.0     # exact in fp64 (bf16 has 8 bits)
        xs += [mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf)]
    for x in xs:
        want = _nearest_bf16_bruteforce(float(x), pv, pb)
        assert O.f64_to_bf16(float(x)) == want, x
        assert O.f64_to_bf16(-float(x)) == want | 0x8000, x
    # overflow: halfway between the largest finite and 2^128 ties to even (inf)
    big = (2 - 2 ** -7) * 2.0 ** 127
    assert O.f64_to_bf16(big) == 0x7F7F
    assert O.f64_to_bf16(big + 2.0 ** 119) == 0x7F80
    assert O.f64_to_bf16(np.nextafter(big + 2.0 ** 119, 0)) == 0x7F7F


def test_f16_against_numpy_ieee_half():
    rng = np.random.default_rng(2)
    xs = np.concatenate([
        rng.normal(size=2000) * 100,
        np.exp(rng.uniform(np.log(1e-9), np.log(7e4), 4000)) * rng.choice([-1, 1], 4000),
        np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float64)[::13],
        [65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14, 0.0, -0.0],
    ])
    xs = xs[np.isfinite(xs)]
    with np.errstate(over="ignore"):
        want = xs.astype(np.float16).view(np.uint16)
    got = np.array([O.f64_to_f16(float(x)) for x in xs], np.uint16)
    np.testing.assert_array_equal(got, want)
    hb = np.arange(0, 65536, 7, dtype=np.uint16)
    ref = hb.view(np.float16).astype(np.float64)
    for b, r in zip(hb, ref):
        g = O.f16_to_f64(int(b))
        assert (math.isnan(g) and math.isnan(r)) or g == r


# --------------------------------------------------------------------------
# Walsh-Hadamard rotation ("PolyKV" 2.B.2 rotation)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("d", [1, 2, 4, 8, 16, 32, 64, 128])
def test_fwht_is_sylvester_hadamard(d):
    rng = np.random.default_rng(d)
    x = rng.normal(size=d)
    Hm = scipy.linalg.hadamard(d).astype(np.float64)
    np.testing.assert_allclose(O.fwht(x), Hm @ x, rtol=0, atol=1e-12 * d)


@pytest.mark.parametrize("d", [64, 128])
def test_fwht_orthogonality_involution_parseval(d):
    cols = np.stack([O.fwht(e) for e in np.eye(d)], axis=1)
    np.testing.assert_array_equal(cols @ cols.T, d * np.eye(d))
    np.testing.assert_array_equal(cols[:, 0], np.ones(d))          # H e0 = 1
    rng = np.random.default_rng(7)
    x = rng.standard_t(5, size=d)
    y = O.fwht(x) / math.sqrt(d)
    assert abs(np.dot(y, y) - np.dot(x, x)) < 1e-12 * np.dot(x, x)
    np.testing.assert_allclose(O.fwht(y) / math.sqrt(d), x, atol=1e-12)


# --------------------------------------------------------------------------
# Lloyd-Max codebook ("PolyKV" 2.B.2 quantization)
# --------------------------------------------------------------------------

def test_lloyd_iteration_reproduces_published_codebook():
    g = golden("lloyd_max_gauss8.json")
    c, mse, it = O.lloyd_max_gauss(8)
    assert it < 100000
    pos = np.array(g["positive_centroids"])
    np.testing.assert_allclose(c[4:], pos, atol=g["printed_precision"])
    np.testing.assert_allclose(c[:4], -pos[::-1], atol=g["printed_precision"])
    assert abs(mse - g["mse"]) < g["mse_printed_precision"]
    # the codebook the codec uses is the published one; thresholds are midpoints
    np.testing.assert_array_equal(O.centroids()[4:], pos)
    np.testing.assert_allclose(O.thresholds()[4:], g["positive_thresholds_midpoints"], atol=1e-15)
    np.testing.assert_allclose(O.thresholds()[:3], -np.array(g["positive_thresholds_midpoints"])[::-1], atol=1e-15)
    assert O.thresholds()[3] == 0.0


def test_lloyd_fixed_point_by_quadrature():
    """Each centroid is the conditional mean of its cell (numerical integral)."""
    c, _, _ = O.lloyd_max_gauss(8)
    edges = [-np.inf] + list((c[:-1] + c[1:]) / 2) + [np.inf]
    for i in range(8):
        a, b = edges[i], edges[i + 1]
        num = scipy.integrate.quad(lambda x: x * scipy.stats.norm.pdf(x), a, b)[0]
        den = scipy.integrate.quad(scipy.stats.norm.pdf, a, b)[0]
        assert abs(num / den - c[i]) < 1e-9
    mse = sum(scipy.integrate.quad(lambda x, ci=c[i]: (x - ci) ** 2 * scipy.stats.norm.pdf(x),
                                   edges[i], edges[i + 1])[0] for i in range(8))
    assert abs(mse - O.lloyd_max_gauss(8)[1]) < 1e-9


def test_v_code_is_nearest_centroid():
    c = O.centroids()
    rng = np.random.default_rng(3)
    t = O.thresholds()
    # a value on a (fp64) threshold goes to the upper cell
    for j, tj in enumerate(t):
        assert O.v_code(float(tj)) == j + 1
        assert O.v_code(float(np.nextafter(tj, -np.inf))) == j
    us = list(rng.normal(size=5000) * 1.5) + [-0.0, 0.0, 5.0, -5.0]
    us += [tj + e for tj in t for e in (1e-9, -1e-9)]
    for u in us:
        dist = [abs(Fraction(float(u)) - Fraction(float(ci))) for ci in c]
        m = min(dist)
        want = max(j for j in range(8) if dist[j] == m)      # a tie goes to the upper cell
        assert O.v_code(float(u)) == want, u


# --------------------------------------------------------------------------
# keys: per-tensor symmetric int8 ("PolyKV" 2.B.1)
# --------------------------------------------------------------------------

def _fp32_nearest(fr):
    """Correctly rounded fp32 of a positive Fraction, by bracketing."""
    f = np.float32(float(fr))
    cands = [np.nextafter(f, np.float32(0)), f, np.nextafter(f, np.float32(np.inf))]
    return min(cands, key=lambda c: (abs(Fraction(float(c)) - fr), int(np.float32(c).view(np.uint32)) & 1))


def _bf16(a):
    return np.asarray(a, np.float32).view(np.uint32).__rshift__(16).astype(np.uint16)


def test_k_scale_is_correctly_rounded_quotient():
    rng = np.random.default_rng(4)
    _, vals = _all_bf16_values()
    ms = vals[np.isfinite(vals) & (vals > 0)]
    for m in list(rng.choice(ms, 800)) + [1.0, 127.0, 254.0, float(ms.min()), float(ms.max())]:
        want = _fp32_nearest(Fraction(float(m)) / 127)
        assert O.k_scale(float(m)) == want, m
    assert O.k_scale(0.0) == 0.0


def test_k_codes_bruteforce_exact():
    rng = np.random.default_rng(5)
    for trial in range(30):
        x = rng.normal(size=64) * (10.0 ** rng.uniform(-3, 3))
        x[rng.integers(0, 64)] *= 20
        kb = _bf16(x)
        m, bad = O.k_absmax(kb)
        assert not bad
        kv = np.array([O.bf16_to_f64(int(b)) for b in kb])
        assert m == np.max(np.abs(kv))
        s = O.k_scale(m)
        S = Fraction(float(s))
        for b, k in zip(kb, kv):
            K = Fraction(float(k))
            best = min(range(-127, 128), key=lambda q: (abs(K - q * S), q & 1))
            q = O.k_code(int(b), s)
            assert q == best
            assert abs(K - q * S) <= S / 2
        # the absmax element maps to +-127
        j = int(np.argmax(np.abs(kv)))
        assert abs(O.k_code(int(kb[j]), s)) == 127


def test_k_codes_ties_go_to_even():
    s = np.float32(1.0)
    for k, want in [(0.5, 0), (1.5, 2), (2.5, 2), (-0.5, 0), (-1.5, -2), (-2.5, -2), (126.5, 126)]:
        assert O.k_code(int(_bf16(k)), s) == want


def test_k_on_grid_and_zero_tensor():
    ints = np.arange(-127, 128, dtype=np.float64)
    kb = _bf16(ints)
    m, _ = O.k_absmax(kb)
    s = O.k_scale(m)
    assert m == 127.0 and s == 1.0
    assert [O.k_code(int(b), s) for b in kb] == list(range(-127, 128))
    assert [O.k_decode(q, s) for q in range(-127, 128)] == list(kb)
    z = np.zeros(16, np.uint16)
    m, _ = O.k_absmax(z)
    assert m == 0.0 and O.k_scale(m) == 0.0 and O.k_code(0, np.float32(0)) == 0
    assert O.k_decode(0, np.float32(0)) == 0


def test_k_nonfinite_flag():
    kb = _bf16(np.array([1.0, np.inf, -2.0]))
    m, bad = O.k_absmax(kb)
    assert bad and m == 2.0
    kb = np.array([0x7FC0, 0x3F80], np.uint16)
    assert O.k_absmax(kb)[1]


# --------------------------------------------------------------------------
# values: FWHT + sigma + Lloyd-Max codes + 3-bit pack ("PolyKV" 2.B.2)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("d", [64, 128])
def test_v_encode_against_library_rotation(d):
    rng = np.random.default_rng(d + 1)
    Hm = scipy.linalg.hadamard(d).astype(np.float64)
    c = O.centroids()
    t = O.thresholds()
    for _ in range(40):
        v = rng.standard_t(5, size=d) * 0.5
        vb = _bf16(v)
        vv = vb.astype(np.uint32).__lshift__(16).astype(np.uint32).view(np.float32).astype(np.float64)
        codes, sh, u, flags = O.v_encode_vec(vb)
        assert flags == 0
        nrm = np.linalg.norm(vv)
        u_ref = (Hm @ vv) / nrm
        np.testing.assert_allclose(u, u_ref, atol=1e-12)
        # sigma = ||v|| / sqrt(d), stored as IEEE half
        assert sh == int(np.float16(nrm / math.sqrt(d)).view(np.uint16))
        far = np.min(np.abs(u_ref[:, None] - t[None, :]), axis=1) > 1e-9
        want = np.argmin(np.abs(u_ref[:, None] - c[None, :]), axis=1)
        np.testing.assert_array_equal(codes[far], want[far])


@pytest.mark.parametrize("d", [64, 128])
def test_v_one_hot_and_hadamard_row_closed_forms(d):
    # v = a e_0: y = a (1,...,1), u_i = sign(a) -> cell of 1.0 is [0.50055, 1.05): code 5 (2 if a<0)
    for a, code in [(3.0, 5), (-0.75, 2)]:
        v = np.zeros(d)
        v[0] = a
        codes, sh, u, _ = O.v_encode_vec(_bf16(v))
        assert set(codes) == {code}
        assert sh == int(np.float16(abs(a) / math.sqrt(d)).view(np.uint16))
    # v = row j of H (entries +-1): y = d e_j, ||v|| = sqrt(d), u_j = sqrt(d) > 1.748
    j = 5
    v = scipy.linalg.hadamard(d)[j].astype(np.float64)
    codes, sh, u, _ = O.v_encode_vec(_bf16(v))
    assert codes[j] == 7 and np.all(np.delete(codes, j) == 4)
    assert sh == int(np.float16(1.0).view(np.uint16))
    # zero vector: every code is the cell just above 0, sigma 0
    codes, sh, u, flags = O.v_encode_vec(np.zeros(d, np.uint16))
    assert np.all(codes == 4) and sh == 0 and flags == 0
    # negative zeros behave like zeros
    codes, sh, u, flags = O.v_encode_vec(np.full(d, 0x8000, np.uint16))
    assert np.all(codes == 4) and sh == 0


def test_v_flags():
    """Non-finite input is NONFINITE only; a finite vector whose sigma exceeds
    the fp16 range is RANGE only."""
    d = 64
    for bad in (np.inf, -np.inf, np.nan):
        v = np.zeros(d)
        v[3] = bad
        assert O.v_encode_vec(_bf16(v))[3] == O.FLAG_NONFINITE
    v = np.full(d, 70000.0)          # sigma = 70000 > fp16 max
    assert O.v_encode_vec(_bf16(v))[3] == O.FLAG_RANGE
    v = np.full(d, 65000.0)          # sigma = 65000 fits
    assert O.v_encode_vec(_bf16(v))[3] == 0


def test_group_flags():
    x = np.linspace(-1, 1, 32)
    x[4] = np.nan
    assert O.group_quant(x, 4)[4] == O.FLAG_NONFINITE
    x[4] = np.inf
    assert O.group_quant(x, 4)[4] == O.FLAG_NONFINITE
    x = np.linspace(-70000.0, 0.0, 32)      # zero point below -65504
    assert O.group_quant(x, 4)[4] == O.FLAG_RANGE


def test_pack3_layout():
    d = 64
    assert list(O.pack3(np.full(d, 7, np.uint8))) == [0xFF] * (3 * d // 8)
    c = np.zeros(d, np.uint8)
    c[1] = 1                                   # code 1 at bits 3..5
    c[8] = 4                                   # second group, code 4 at bits 0..2 -> 0x04
    c[15] = 7                                  # second group, bits 21..23 -> byte 2 = 0xE0
    p = O.pack3(c)
    assert list(p[:6]) == [0x08, 0x00, 0x00, 0x04, 0x00, 0xE0]
    rng = np.random.default_rng(0)
    for d in (64, 128):
        c = rng.integers(0, 8, d).astype(np.uint8)
        np.testing.assert_array_equal(O.unpack3(O.pack3(c), d), c)


@pytest.mark.parametrize("d", [64, 128])
def test_v_decode_closed_form(d):
    # all codes 4: c_hat = 0.2451 * ones, H c_hat = 0.2451 d e_0,
    # x_hat = sigma_h * 0.2451 * d / sqrt(d) at index 0, zero elsewhere
    sig = int(np.float16(1.5).view(np.uint16))
    out = O.v_decode_vec(np.full(d, 4, np.uint8), sig)
    want0 = 1.5 * 0.2451 * math.sqrt(d)
    assert out[0] == int(_bf16(np.float32(want0))) or abs(O.bf16_to_f64(int(out[0])) - want0) <= 2 ** -8 * want0
    assert np.all(out[1:] == 0)
    # decode is linear in the centroids: against the library matrix product
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 8, d).astype(np.uint8)
    ref = 1.5 * (scipy.linalg.hadamard(d) @ O.centroids()[codes]) / math.sqrt(d)
    got = np.array([O.bf16_to_f64(int(b)) for b in O.v_decode_vec(codes, sig)])
    np.testing.assert_allclose(got, ref, rtol=2 ** -8, atol=1e-6)


def test_v_centroid_inputs_roundtrip():
    """Vectors whose normalised rotated coordinates sit on centroids far from
    the cell edges decode and re-encode to the same codes."""
    rng = np.random.default_rng(11)
    for d in (64, 128):
        for _ in range(10):
            codes = rng.choice(np.array([1, 2, 5, 6], np.uint8), d)
            x = O.v_decode_vec(codes, int(np.float16(0.7).view(np.uint16)))
            codes2, _, _, _ = O.v_encode_vec(x)
            np.testing.assert_array_equal(codes2, codes)


def test_v_relative_mse_matches_lloyd_max():
    """Gaussian vectors: after rotation and normalisation the coordinates are
    ~N(0,1), so the relative MSE is the Lloyd-Max MSE 0.03455 (within 10%)."""
    rng = np.random.default_rng(12)
    d = 128
    num = den = 0.0
    for _ in range(8000):                      # 1.02e6 coordinates
        vb = _bf16(rng.normal(size=d))
        v = vb.astype(np.uint32).__lshift__(16).astype(np.uint32).view(np.float32).astype(np.float64)
        codes, sh, _, _ = O.v_encode_vec(vb)
        # compare in the rotated, normalised domain the quantizer works in
        nrm = np.linalg.norm(v)
        u = O.fwht(v) / nrm
        num += np.sum((u - O.centroids()[codes]) ** 2)
        den += d
    assert abs(num / den - 0.03455) < 0.1 * 0.03455


# --------------------------------------------------------------------------
# pool image and ratios ("PolyKV" 2.A, compression-ratio equation, 4)
# --------------------------------------------------------------------------

def test_ratio_closed_forms():
    g = golden("polykv_ratio.json")
    ratio = g["bits_fp"] / ((g["bits_k"] + g["bits_v"]) / 2)
    assert round(ratio, g["ratio_printed_decimals"]) == g["ratio_printed"]
    red = 1 - 1 / (g["agents"] * ratio)
    assert round(100 * red, g["reduction_printed_decimals"]) == g["reduction_printed_percent"]
    # achieved ratio of the pool payload per (token, head): K d bytes, V 3d/8 + fp16 sigma
    for d, want in [(128, 2.8764), (64, 2.8444)]:
        raw = 2 * d * 2
        comp = d + 3 * d // 8 + 2
        assert abs(raw / comp - want) < 1e-4
        L, H, T = 4, 8, 1024
        geo = O.pool_geometry(L, H, d, T)
        payload = geo["layer_stride"] * L
        assert abs(raw * H * T * L / payload - raw / comp) < 1e-3


def test_pool_geometry_closed_form():
    L, H, d, T = 3, 5, 64, 37
    g = O.pool_geometry(L, H, d, T)
    al = lambda x: (x + 255) // 256 * 256
    nv = H * T
    assert g["off_scales"] == 256
    assert g["off_layers"] == al(256 + 4 * L)
    assert g["sec_v"] == al(nv * d)
    assert g["sec_sigma"] == al(g["sec_v"] + nv * 3 * d // 8)
    assert g["layer_stride"] == al(g["sec_sigma"] + 2 * nv)
    assert g["total"] == g["off_layers"] + L * g["layer_stride"] == O.pool_bytes(L, H, d, T)


def _tiny_kv(L, H, T, d, seed):
    rng = np.random.default_rng(seed)
    ks, vs = [], []
    for _ in range(L):
        k = rng.normal(size=(H, T, d))
        for h in range(H):
            k[h, :, rng.choice(d, 4, replace=False)] *= 20
        ks.append(_bf16(k))
        vs.append(_bf16(rng.standard_t(5, size=(H, T, d)) * 0.5))
    return ks, vs


def _f(bits):
    return np.asarray(bits, np.uint16).astype(np.uint32).__lshift__(16).astype(np.uint32).view(np.float32).astype(np.float64)


def test_pool_encode_decode_consistent_with_pieces():
    L, H, T, d = 2, 3, 11, 64
    ks, vs = _tiny_kv(L, H, T, d, 13)
    pool, flags, u = O.pool_encode(ks, vs, want_u=True)
    assert flags == 0
    g = O.pool_geometry(L, H, d, T)
    hdr = pool[:32].view(np.uint32)
    assert hdr[0] == 0x4C50564B and hdr[1] == 1 and list(hdr[2:6]) == [L, H, d, T]
    for l in range(L):
        m, _ = O.k_absmax(ks[l])
        s = O.k_scale(m)
        assert pool[g["off_scales"] + 4 * l: g["off_scales"] + 4 * l + 4].view(np.float32)[0] == s
        base = g["off_layers"] + l * g["layer_stride"]
        kc = pool[base: base + H * T * d].view(np.int8)
        np.testing.assert_array_equal(kc, [O.k_code(int(b), s) for b in ks[l].ravel()])
        for n in (0, 7, H * T - 1):
            codes, sh, _, _ = O.v_encode_vec(vs[l].reshape(-1, d)[n])
            vc = pool[base + g["sec_v"] + n * 3 * d // 8: base + g["sec_v"] + (n + 1) * 3 * d // 8]
            np.testing.assert_array_equal(O.unpack3(vc, d), codes)
            assert pool[base + g["sec_sigma"] + 2 * n: base + g["sec_sigma"] + 2 * n + 2].view(np.uint16)[0] == sh
    # fan-out decode: every agent gets identical layers; values within the codec's error
    k_out, v_out = O.pool_decode_into(pool, 0, L, 3)
    for a in range(3):
        for l in range(L):
            np.testing.assert_array_equal(k_out[a][l], k_out[0][l])
            np.testing.assert_array_equal(v_out[a][l], v_out[0][l])
    for l in range(L):
        s = float(O.k_scale(O.k_absmax(ks[l])[0]))
        err = np.abs(_f(k_out[0][l]) - _f(ks[l]))
        assert np.all(err <= s / 2 + 2 ** -8 * np.abs(_f(ks[l])) + 1e-30)
        rel = np.sum((_f(v_out[0][l]) - _f(vs[l])) ** 2) / np.sum(_f(vs[l]) ** 2)
        assert rel < 0.06


def test_pool_decode_layer_range():
    L, H, T, d = 3, 2, 5, 128
    ks, vs = _tiny_kv(L, H, T, d, 14)
    pool, _, _ = O.pool_encode(ks, vs)
    k_all, v_all = O.pool_decode_into(pool, 0, L, 1)
    k_mid, v_mid = O.pool_decode_into(pool, 1, 2, 2)
    assert k_mid[0][0] is None and k_mid[1][2] is None
    np.testing.assert_array_equal(k_mid[1][1], k_all[0][1])
    np.testing.assert_array_equal(v_mid[0][1], v_all[0][1])


# --------------------------------------------------------------------------
# CacheCard ("QKVShare" Methodology 1-3)
# --------------------------------------------------------------------------

def test_card_record_bytes_golden():
    g = golden("cachecard_record_bytes.json")
    for b, want in g["record_bytes"].items():
        assert O.card_record_bytes(int(b), g["n_kv_heads"], g["head_dim"]) == want


def test_card_bytes_is_sum_of_records():
    rng = np.random.default_rng(15)
    L, H, d, T = 3, 1, 64, 29
    bits = rng.choice(np.array([2, 4, 8, 16], np.uint8), T)
    g = O.card_geometry(L, H, d, T, bits)
    rec = sum(O.card_record_bytes(int(b), H, d) for b in bits)
    assert g["layer_stride"] == (rec + 255) // 256 * 256
    assert g["off_offsets"] % 16 == 0 and g["off_offsets"] >= 128 + T
    assert g["off_layers"] % 256 == 0 and g["off_layers"] >= g["off_offsets"] + 4 * T
    assert g["total"] == O.card_bytes(L, H, d, T, bits) == g["off_layers"] + L * g["layer_stride"]
    # H=1, d=64, b=2: 2*(16 + 2*4) = 48, already a multiple of 16; b=4: 2*(32+8) = 80
    assert O.card_record_bytes(2, 1, 64) == 48 and O.card_record_bytes(4, 1, 64) == 80
    # odd sizes are padded to 16 bytes: H=3, d=64, b=2: 2*(48+24) = 144; b=8: 2*(192+24) = 432
    assert O.card_record_bytes(8, 3, 64) == 432
    bad = bits.copy()
    bad[3] = 3
    assert O.card_bytes(L, H, d, T, bad) == 0


@pytest.mark.parametrize("b", [2, 4, 8])
def test_group_quant_bruteforce(b):
    rng = np.random.default_rng(b)
    qmax = 2 ** b - 1
    for _ in range(60):
        x = _f(_bf16(rng.normal(size=32) * 10.0 ** rng.uniform(-2, 2) + rng.normal() * 3))
        q, sb, zb, r, flags = O.group_quant(x, b)
        assert flags == 0
        assert sb == int(np.float16((x.max() - x.min()) / qmax).view(np.uint16))
        assert zb == int(np.float16(x.min()).view(np.uint16))
        S, Z = Fraction(O.f16_to_f64(sb)), Fraction(O.f16_to_f64(zb))
        for xi, qi in zip(x, q):
            X = Fraction(float(xi))
            best = min(range(qmax + 1), key=lambda c: (abs(X - (c * S + Z)), c & 1))
            assert qi == best


def test_group_quant_on_grid_and_degenerate():
    for b in (2, 4, 8):
        qmax = 2 ** b - 1
        rng = np.random.default_rng(b + 100)
        q0 = rng.integers(0, qmax + 1, 32)
        q0[0], q0[1] = 0, qmax
        x = q0.astype(np.float64) * 0.5 - 3.0        # s = 0.5, z = -3 exactly in fp16
        q, sb, zb, r, _ = O.group_quant(x, b)
        np.testing.assert_array_equal(q, q0)
        assert O.f16_to_f64(sb) == 0.5 and O.f16_to_f64(zb) == -3.0
    q, sb, zb, r, _ = O.group_quant(np.full(32, 2.5), 4)     # constant group: s = 0
    assert sb == 0 and np.all(q == 0) and O.f16_to_f64(zb) == 2.5


def test_card_pack_unpack_roundtrip():
    L, H, T, d = 2, 3, 9, 64
    ks, vs = _tiny_kv(L, H, T, d, 16)
    bits = np.array([2, 4, 8, 16, 16, 8, 4, 2, 4], np.uint8)
    card, flags, r = O.card_pack(ks, vs, bits, model_id=0x1234567890ABCDEF, pos_offset=-77, want_r=True)
    assert flags == 0
    hdr = card[:128]
    assert hdr[:4].view(np.uint32)[0] == 0x4343564B
    assert list(hdr[8:32].view(np.int32)) == [T, L, H, d, 32, 1]
    assert hdr[32:40].view(np.uint64)[0] == 0x1234567890ABCDEF
    assert hdr[40:48].view(np.int64)[0] == -77
    g = O.card_geometry(L, H, d, T, bits)
    np.testing.assert_array_equal(card[g["off_bits"]: g["off_bits"] + T], bits)
    offs = card[g["off_offsets"]: g["off_offsets"] + 4 * T].view(np.uint32)
    sizes = [O.card_record_bytes(int(b), H, d) for b in bits]
    np.testing.assert_array_equal(offs, np.concatenate([[0], np.cumsum(sizes)[:-1]]))
    k2, v2 = O.card_unpack(card)
    for l in range(L):
        for t in range(T):
            for src, out in ((ks[l], k2[l]), (vs[l], v2[l])):
                if bits[t] == 16:
                    np.testing.assert_array_equal(out[:, t], src[:, t])
                    continue
                x = _f(src[:, t]).reshape(H, d // 32, 32)
                xh = _f(out[:, t]).reshape(H, d // 32, 32)
                step = (x.max(-1, keepdims=True) - x.min(-1, keepdims=True)) / (2 ** int(bits[t]) - 1)
                assert np.all(np.abs(xh - x) <= 0.5 * step * (1 + 2 ** -9) + 2 ** -8 * np.abs(x) + 2 ** -9 * np.abs(x.min(-1, keepdims=True)) + 1e-6)


def test_card_invalid_bits():
    ks, vs = _tiny_kv(1, 1, 3, 64, 17)
    _, flags, _ = O.card_pack(ks, vs, np.array([2, 5, 4], np.uint8))
    assert flags == O.FLAG_BITS


# --------------------------------------------------------------------------
# attention over the pool (next row: fused attention on the quantized cache)
# --------------------------------------------------------------------------

def _decoded_fp64(pool, L, H, d, T, layer):
    """Exact dequantized K and V of one layer, from the oracle's pieces."""
    g = O.pool_geometry(L, H, d, T)
    base = g["off_layers"] + layer * g["layer_stride"]
    s = float(pool[g["off_scales"] + 4 * layer: g["off_scales"] + 4 * layer + 4].view(np.float32)[0])
    kc = pool[base: base + H * T * d].view(np.int8).astype(np.float64).reshape(H, T, d) * s
    vp = pool[base + g["sec_v"]: base + g["sec_v"] + H * T * 3 * d // 8].reshape(H * T, 3 * d // 8)
    sig = pool[base + g["sec_sigma"]: base + g["sec_sigma"] + 2 * H * T].view(np.uint16)
    Hm = scipy.linalg.hadamard(d).astype(np.float64)
    c = O.centroids()
    v = np.zeros((H * T, d))
    for n in range(H * T):
        codes = O.unpack3(vp[n], d)
        v[n] = O.f16_to_f64(int(sig[n])) * (Hm @ c[codes]) / math.sqrt(d)
    return kc, v.reshape(H, T, d)


def test_pool_attend_against_library_softmax():
    """Against numpy matmuls and scipy's softmax / logsumexp over the exactly
    dequantized caches, with GQA (4 query heads per KV head) and 3 agents."""
    import scipy.special
    L, H, T, d = 2, 2, 37, 64
    ks, vs = _tiny_kv(L, H, T, d, 21)
    pool, _, _ = O.pool_encode(ks, vs)
    rng = np.random.default_rng(22)
    na, nq = 3, 8
    q = _bf16(rng.normal(size=(na, nq, d)))
    qf = _f(q)
    for layer in range(L):
        out, lse = O.pool_attend(pool, layer, q, 0.125)
        kf, vf = _decoded_fp64(pool, L, H, d, T, layer)
        for a in range(na):
            for j in range(nq):
                h = j // (nq // H)
                sc = 0.125 * (kf[h] @ qf[a, j])
                np.testing.assert_allclose(out[a, j], scipy.special.softmax(sc) @ vf[h], rtol=1e-10, atol=1e-12)
                assert abs(lse[a, j] - scipy.special.logsumexp(sc)) < 1e-10


def test_pool_attend_closed_forms():
    L, H, T, d = 1, 1, 16, 128
    ks, vs = _tiny_kv(L, H, T, d, 23)
    pool, _, _ = O.pool_encode(ks, vs)
    kf, vf = _decoded_fp64(pool, L, H, d, T, 0)
    # q = 0: uniform weights -> the mean of the values, lse = log T
    out, lse = O.pool_attend(pool, 0, np.zeros((1, 1, d), np.uint16), 1.0)
    np.testing.assert_allclose(out[0, 0], vf[0].mean(0), rtol=1e-12, atol=1e-14)
    assert abs(lse[0, 0] - math.log(T)) < 1e-12
    # a large scale makes the softmax one-hot on the top-scoring token
    q = _bf16(kf[0, 5][None, None, :] / np.abs(kf[0, 5]).max())
    sc = kf[0] @ _f(q)[0, 0]
    top = np.sort(sc)
    scale = 60.0 / (top[-1] - top[-2])          # the runner-up weighs < e^-60
    out, lse = O.pool_attend(pool, 0, q, scale)
    np.testing.assert_allclose(out[0, 0], vf[0, int(np.argmax(sc))], rtol=1e-9, atol=1e-12)
    assert abs(lse[0, 0] - scale * top[-1]) < 1e-9 * scale * abs(top[-1])


# --------------------------------------------------------------------------
# card unpack re-aligned to other positions (next row: rotary realignment)
# --------------------------------------------------------------------------

def _rope_complex(x, pos, w):
    """Rotary embedding written as complex multiplication, independently of
    the oracle's real 2x2 form: pair (i, i + d/2) is z = x_i + 1j x_{i+d/2},
    turned by exp(1j * pos * w_i).  x [..., T, d], pos [T] (int), w [d/2]."""
    half = x.shape[-1] // 2
    z = x[..., :half] + 1j * x[..., half:]
    ang = np.multiply.outer(np.asarray(pos, np.float64), np.asarray(w, np.float64))
    z = z * np.exp(1j * ang)
    return np.concatenate([z.real, z.imag], axis=-1)


def _bf16_rne(x):
    import torch
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _llama_inv_freq(d, base=500000.0):
    return (1.0 / base ** (np.arange(0, d, 2, dtype=np.float64) / d)).astype(np.float32)


def _pair_norm(x):
    half = x.shape[-1] // 2
    n = np.sqrt(x[..., :half] ** 2 + x[..., half:] ** 2)
    return np.concatenate([n, n], axis=-1)


def test_card_unpack_at_zero_shift_is_plain_unpack():
    L, H, T, d = 2, 3, 9, 128
    ks, vs = _tiny_kv(L, H, T, d, 21)
    bits = np.array([2, 4, 8, 16, 16, 8, 4, 2, 4], np.uint8)
    card, flags, _ = O.card_pack(ks, vs, bits, pos_offset=300)
    assert flags == 0
    k0, v0 = O.card_unpack(card)
    k1, v1 = O.card_unpack_at(card, 300, _llama_inv_freq(d))
    for l in range(L):
        np.testing.assert_array_equal(k1[l], k0[l])
        np.testing.assert_array_equal(v1[l], v0[l])


@pytest.mark.parametrize("d,p_src,p_dst,w", [
    (64, -77, 1000, "llama"), (128, 5000, 12, "llama"), (128, 0, 30000, "unit"), (64, 7, 8, "ramp")])
def test_card_unpack_at_matches_complex_rotation(d, p_src, p_dst, w):
    """Keys embedded at p_src + t, carried verbatim (16-bit tokens), come out
    as the keys embedded at p_dst + t; values are untouched."""
    L, H, T = 2, 3, 7
    rng = np.random.default_rng(d + p_dst)
    freq = {"llama": _llama_inv_freq(d), "unit": np.ones(d // 2, np.float32),
            "ramp": np.linspace(0.01, 3.0, d // 2).astype(np.float32)}[w]
    k0 = [rng.normal(size=(H, T, d)) * 2.0 for _ in range(L)]
    ks = [_bf16_rne(_rope_complex(k, p_src + np.arange(T), freq)) for k in k0]
    vs = [_bf16_rne(rng.normal(size=(H, T, d))) for _ in range(L)]
    card, flags, _ = O.card_pack(ks, vs, np.full(T, 16, np.uint8), pos_offset=p_src)
    assert flags == 0
    ko, vo = O.card_unpack_at(card, p_dst, freq)
    for l in range(L):
        want = _rope_complex(k0[l], p_dst + np.arange(T), freq)
        assert np.all(np.abs(_f(ko[l]) - want) <= 2.0 ** -7 * _pair_norm(want) + 1e-12)
        np.testing.assert_array_equal(vo[l], vs[l])


@pytest.mark.parametrize("d", [64, 128])
def test_card_unpack_at_quarter_and_half_turns(d):
    """w_i = pi/2 per position: a shift of 1 maps (a, b) to (-b, a), a shift
    of 2 negates every key and a shift of -1 maps (a, b) to (b, -a)."""
    L, H, T = 1, 2, 5
    rng = np.random.default_rng(3)
    ks = [_bf16_rne(rng.normal(size=(H, T, d)) + np.sign(rng.normal(size=(H, T, d))))]
    vs = [_bf16_rne(rng.normal(size=(H, T, d)))]
    card, _, _ = O.card_pack(ks, vs, np.full(T, 16, np.uint8), pos_offset=10)
    x = _f(ks[0])
    half = d // 2
    freq = np.full(half, np.pi / 2, np.float32)
    k1, _ = O.card_unpack_at(card, 11, freq)
    np.testing.assert_array_equal(_f(k1[0]), np.concatenate([-x[..., half:], x[..., :half]], -1))
    k2, _ = O.card_unpack_at(card, 12, freq)
    np.testing.assert_array_equal(_f(k2[0]), -x)
    k3, _ = O.card_unpack_at(card, 9, freq)
    np.testing.assert_array_equal(_f(k3[0]), np.concatenate([x[..., half:], -x[..., :half]], -1))


def test_card_unpack_at_quantized_tokens_and_round_trip():
    """Quantized tokens: the re-aligned key is the turned dequantized key (to
    the bf16 rounding of the plain unpack); re-packing the result at the new
    offset and re-aligning back restores the plain unpack."""
    L, H, T, d = 2, 2, 8, 128
    ks, vs = _tiny_kv(L, H, T, d, 22)
    bits = np.array([2, 4, 8, 16, 2, 4, 8, 16], np.uint8)
    freq = _llama_inv_freq(d, base=10000.0)
    card, _, _ = O.card_pack(ks, vs, bits, pos_offset=-1234)
    k0, v0 = O.card_unpack(card)
    k1, v1 = O.card_unpack_at(card, 4321, freq)
    for l in range(L):
        want = _rope_complex(_f(k0[l]), 5555 + np.zeros(T), freq)
        assert np.all(np.abs(_f(k1[l]) - want) <= 2.0 ** -7 * _pair_norm(want) + 1e-12)
        np.testing.assert_array_equal(v1[l], v0[l])
    card2, _, _ = O.card_pack(k1, v1, np.full(T, 16, np.uint8), pos_offset=4321)
    k2, _ = O.card_unpack_at(card2, -1234, freq)
    for l in range(L):
        ref = _f(k0[l])
        assert np.all(np.abs(_f(k2[l]) - ref) <= 2.0 ** -7 * _pair_norm(ref) + 1e-12)


# --------------------------------------------------------------------------
# q8_0 key blocks (next row: block-wise int8 keys with fp16 scales)
# --------------------------------------------------------------------------

def _fp16_nearest(fr):
    """Correctly rounded fp16 of a non-negative Fraction (ties to even), by
    bracketing with numpy's fp16 neighbours."""
    f = np.float16(float(fr))
    cands = [np.nextafter(f, np.float16(0)), f, np.nextafter(f, np.float16(np.inf))]
    cands = [c for c in cands if np.isfinite(c)]
    return min(cands, key=lambda c: (abs(Fraction(float(c)) - fr), int(np.float16(c).view(np.uint16)) & 1))


def _q8_block(x):
    kb = _bf16(x)
    sb, bad, rng = O.k_block_scale(kb)
    return kb, sb, bad, rng


def test_k_block_scale_is_correctly_rounded_fp16():
    rng = np.random.default_rng(31)
    mags = [1.0, 127.0, 3.5, 127 * 2.0 ** -25, 127 * 2.0 ** -14, 127 * 2.0 ** -24 * 3, 5.0e4, 8.0e6, 1e-7]
    mags += list(10.0 ** rng.uniform(-7, 6.5, 300))
    for m in mags:
        x = rng.normal(size=32) * 0.3 * m
        x[rng.integers(0, 32)] = m * (1 if rng.random() < 0.5 else -1)
        kb, sb, bad, rng_flag = _q8_block(x)
        mm = max(abs(O.bf16_to_f64(int(b))) for b in kb)
        want = _fp16_nearest(Fraction(mm) / 127)
        s = np.float16(O.f16_to_f64(sb))
        if np.isinf(np.float16(float(Fraction(mm) / 127))) or float(Fraction(mm) / 127) >= 65520:
            assert rng_flag and (sb & 0x7C00) == 0x7C00
            continue
        assert not bad and not rng_flag
        assert s == want, (m, s, want)


def test_k_block_codes_bruteforce_exact():
    rng = np.random.default_rng(32)
    for trial in range(40):
        x = rng.normal(size=32) * (10.0 ** rng.uniform(-6, 3))
        x[rng.integers(0, 32)] *= 20
        kb, sb, _, _ = _q8_block(x)
        S = Fraction(O.f16_to_f64(sb))
        assert S > 0
        clamped = 0
        for b in kb:
            K = Fraction(O.bf16_to_f64(int(b)))
            best = min(range(-127, 128), key=lambda q: (abs(K - q * S), q & 1))
            q = O.k_block_code(int(b), sb)
            assert q == best
            if abs(K - q * S) > S / 2:
                clamped += 1
                assert abs(q) == 127
            assert O.k_block_decode(q, sb) == int(_bf16_rne(float(q * S)))
        if O.f16_to_f64(sb) >= 2.0 ** -14:  # normal scale: nothing clamps, the absmax maps to +-127
            assert clamped == 0
            j = int(np.argmax(np.abs(_f(kb))))
            assert abs(O.k_block_code(int(kb[j]), sb)) == 127


def test_k_block_on_grid_zero_and_flags():
    for e in (-10, -3, 0, 5):
        qs = np.arange(-127, 128, 8)[:32].astype(np.float64)
        qs[0] = -127
        x = qs * 2.0 ** e
        kb, sb, bad, rng_flag = _q8_block(x)
        assert O.f16_to_f64(sb) == 2.0 ** e and not bad and not rng_flag
        assert [O.k_block_code(int(b), sb) for b in kb] == [int(q) for q in qs]
        assert [O.k_block_decode(int(q), sb) for q in qs] == list(kb)
    kb, sb, bad, rng_flag = _q8_block(np.zeros(32))
    assert sb == 0 and O.k_block_code(int(kb[0]), sb) == 0 and O.k_block_decode(0, sb) == 0
    kb, sb, bad, rng_flag = _q8_block(np.full(32, 127 * 2.0 ** -26))  # below half the least scale
    assert sb == 0 and all(O.k_block_code(int(b), sb) == 0 for b in kb)
    x = np.ones(32)
    x[3] = np.nan
    assert _q8_block(x)[2]
    x = np.ones(32)
    x[5] = 1.0e7  # 1e7 / 127 overflows fp16
    kb, sb, bad, rng_flag = _q8_block(x)
    assert rng_flag and not bad


def test_pool_q8_layout_and_consistency():
    L, H, T, d = 2, 3, 11, 64
    ks, vs = _tiny_kv(L, H, T, d, 33)
    p0, f0, _ = O.pool_encode(ks, vs)
    p1, f1, _ = O.pool_encode(ks, vs, k_mode=1)
    assert f0 == 0 and f1 == 0
    g = O.pool_geometry(L, H, d, T)
    off_ks, total = O.pool_geometry_q8(L, H, d, T)
    nb = H * T * d // 32
    assert off_ks == g["total"] and total == g["total"] + ((L * nb * 2 + 255) // 256) * 256 == p1.size
    hdr = p1[:80]
    assert hdr[28:32].view(np.uint32)[0] == 1 and p0[28:32].view(np.uint32)[0] == 0
    assert hdr[72:80].view(np.uint64)[0] == total
    assert not p1[g["off_scales"]: g["off_scales"] + 4 * L].any()       # no per-tensor scales
    for l in range(L):
        base = g["off_layers"] + l * g["layer_stride"]
        # values and sigma do not depend on the key format
        np.testing.assert_array_equal(p1[base + g["sec_v"]: base + g["layer_stride"]],
                                      p0[base + g["sec_v"]: base + g["layer_stride"]])
        kc = p1[base: base + H * T * d].view(np.int8)
        sc = p1[off_ks + l * nb * 2: off_ks + (l + 1) * nb * 2].view(np.uint16)
        kflat = ks[l].reshape(-1)
        for b in range(nb):
            sb, _, _ = O.k_block_scale(kflat[32 * b: 32 * b + 32])
            assert sc[b] == sb
            assert [O.k_block_code(int(x), sb) for x in kflat[32 * b: 32 * b + 32]] == list(kc[32 * b: 32 * b + 32])
    kd, vd = O.pool_decode_into(p1, 0, L, 1)
    k0, v0 = O.pool_decode_into(p0, 0, L, 1)
    for l in range(L):
        base = g["off_layers"] + l * g["layer_stride"]
        kc = p1[base: base + H * T * d].view(np.int8)
        sc = p1[off_ks + l * nb * 2: off_ks + (l + 1) * nb * 2].view(np.uint16)
        want = [O.k_block_decode(int(kc[i]), int(sc[i // 32])) for i in range(H * T * d)]
        np.testing.assert_array_equal(kd[0][l].reshape(-1), np.array(want, np.uint16))
        np.testing.assert_array_equal(vd[0][l], v0[0][l])


def test_q8_blocks_beat_one_scale_on_outlier_channels():
    """Keys with a few 20x channels per head (the synthetic recipe): per-block
    scales confine the outliers' range to their own blocks, so the mean
    reconstruction error is several times below the per-tensor scale's."""
    L, H, T, d = 1, 2, 64, 128
    ks, vs = _tiny_kv(L, H, T, d, 34)
    x = _f(ks[0])
    errs = []
    for mode in (0, 1):
        p, _, _ = O.pool_encode(ks, vs, k_mode=mode)
        kd, _ = O.pool_decode_into(p, 0, 1, 1)
        errs.append(np.mean(np.abs(_f(kd[0][0]) - x)))
    assert errs[1] < errs[0] / 3, errs


def test_pool_attend_q8_against_library_softmax():
    import scipy.special
    L, H, T, d = 1, 2, 45, 128
    ks, vs = _tiny_kv(L, H, T, d, 35)
    pool, _, _ = O.pool_encode(ks, vs, k_mode=1)
    g = O.pool_geometry(L, H, d, T)
    off_ks, _ = O.pool_geometry_q8(L, H, d, T)
    kc = pool[g["off_layers"]: g["off_layers"] + H * T * d].view(np.int8).astype(np.float64)
    sc = np.array([O.f16_to_f64(int(s)) for s in pool[off_ks: off_ks + H * T * d // 32 * 2].view(np.uint16)])
    kf = (kc.reshape(-1, 32) * sc[:, None]).reshape(H, T, d)
    _, vf = _decoded_fp64(pool, L, H, d, T, 0)
    rng = np.random.default_rng(36)
    q = _bf16(rng.normal(size=(2, 4, d)))
    out, lse = O.pool_attend(pool, 0, q, 0.1)
    for a in range(2):
        for j in range(4):
            h = j // 2
            s = 0.1 * (kf[h] @ _f(q)[a, j])
            np.testing.assert_allclose(out[a, j], scipy.special.softmax(s) @ vf[h], rtol=1e-10, atol=1e-12)
            assert abs(lse[a, j] - scipy.special.logsumexp(s)) < 1e-10


# --------------------------------------------------------------------------
# attention with a shared low-rank value cache (next row: Flash-LoRA reorder)
# --------------------------------------------------------------------------

def _lora_inputs(T, d, H, na, rank, seed):
    rng = np.random.default_rng(seed)
    vlr = _bf16(rng.normal(size=(T, rank)))
    b = _bf16(rng.normal(size=(na, rank, H * d)) * 0.05)
    return vlr, b


def test_pool_attend_lora_zero_b_is_plain_attention():
    L, H, T, d = 1, 2, 37, 64
    ks, vs = _tiny_kv(L, H, T, d, 41)
    pool, _, _ = O.pool_encode(ks, vs)
    q = _bf16(np.random.default_rng(42).normal(size=(3, 8, d)))
    vlr, _ = _lora_inputs(T, d, H, 3, 16, 43)
    out0, lse0 = O.pool_attend(pool, 0, q, 0.125)
    out1, lse1 = O.pool_attend_lora(pool, 0, q, 0.125, vlr, np.zeros((3, 16, H * d), np.uint16))
    np.testing.assert_array_equal(out1, out0)
    np.testing.assert_array_equal(lse1, lse0)


@pytest.mark.parametrize("k_mode", [0, 1])
def test_pool_attend_lora_against_reordered_library_form(k_mode):
    """The oracle forms every agent's values first; numpy's softmax with the
    reordered product P V_base + (P V_lr) B_a must agree."""
    import scipy.special
    L, H, T, d, na, nq, rank = 1, 2, 45, 128, 3, 8, 32
    ks, vs = _tiny_kv(L, H, T, d, 44)
    pool, _, _ = O.pool_encode(ks, vs, k_mode=k_mode)
    vlr, b = _lora_inputs(T, d, H, na, rank, 45)
    q = _bf16(np.random.default_rng(46).normal(size=(na, nq, d)))
    out, lse = O.pool_attend_lora(pool, 0, q, 0.09, vlr, b)
    kf, _ = _decoded_fp64(pool, L, H, d, T, 0) if k_mode == 0 else (None, None)
    if k_mode == 1:
        g = O.pool_geometry(L, H, d, T)
        off_ks, _ = O.pool_geometry_q8(L, H, d, T)
        kc = pool[g["off_layers"]: g["off_layers"] + H * T * d].view(np.int8).astype(np.float64)
        sc = np.array([O.f16_to_f64(int(s)) for s in pool[off_ks: off_ks + H * T * d // 32 * 2].view(np.uint16)])
        kf = (kc.reshape(-1, 32) * sc[:, None]).reshape(H, T, d)
    _, vf = _decoded_fp64(pool, L, H, d, T, 0)
    vl, bf = _f(vlr), _f(b)
    for a in range(na):
        for j in range(nq):
            h = j // (nq // H)
            p = scipy.special.softmax(0.09 * (kf[h] @ _f(q)[a, j]))
            want = p @ vf[h] + (p @ vl) @ bf[a][:, h * d:(h + 1) * d]
            np.testing.assert_allclose(out[a, j], want, rtol=1e-10, atol=1e-12)
            assert abs(lse[a, j] - scipy.special.logsumexp(0.09 * (kf[h] @ _f(q)[a, j]))) < 1e-10


def test_pool_attend_lora_one_hot_low_rank_cache():
    """Every token's low-rank activation is e_k: the attention-weighted sum is
    e_k whatever the weights, so the output shifts by row k of the agent's
    up-projection, restricted to the query's KV head."""
    L, H, T, d, na, nq, rank = 1, 4, 21, 64, 2, 8, 16
    ks, vs = _tiny_kv(L, H, T, d, 47)
    pool, _, _ = O.pool_encode(ks, vs)
    _, b = _lora_inputs(T, d, H, na, rank, 48)
    q = _bf16(np.random.default_rng(49).normal(size=(na, nq, d)))
    out0, _ = O.pool_attend(pool, 0, q, 0.2)
    for k in (0, 5, rank - 1):
        vlr = np.zeros((T, rank), np.uint16)
        vlr[:, k] = _bf16(1.0)
        out, _ = O.pool_attend_lora(pool, 0, q, 0.2, vlr, b)
        for a in range(na):
            for j in range(nq):
                h = j // (nq // H)
                np.testing.assert_allclose(out[a, j] - out0[a, j], _f(b)[a, k, h * d:(h + 1) * d], atol=1e-12)
