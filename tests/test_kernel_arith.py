"""Arithmetic shortcuts the CUDA kernels take, checked on the CPU against the
oracle over every input they can see (no GPU needed).

q8_0 key blocks ("PolyKV" section 2, the q8_0 key format): the encoder forms
the fp16 block scale as fp16(fl32(max|k|) * fl32(1/127)) instead of an IEEE
division.  Over all 32,640 finite bf16 maxima that must give the oracle's
scale, the fp16 nearest to the real max|k|/127, including the fp16 subnormal
range and the overflow to Inf (reported as a range error).

Values ("PolyKV" section 2.B.2): the encoder's tensor-core rotation (its lane,
fragment and staging layout, restated here) computes the oracle's transform;
its codes, taken from the sign bits of y^2 - t_k^2 S / d and two products in
fp32 and packed by funnel shifts, equal the oracle's wherever the oracle's u
is not within 1e-4 of a threshold.
"""
import numpy as np

import oracle as O


def _kernel_block_scale(m_bits):
    m = (np.asarray(m_bits, dtype=np.uint32) << 16).view(np.float32)
    with np.errstate(over="ignore"):
        return (m * (np.float32(1.0) / np.float32(127.0))).astype(np.float16).view(np.uint16)


def test_q8_block_scale_product_matches_oracle_for_every_bf16_maximum():
    m_bits = np.arange(0, 0x7F80, dtype=np.uint32)
    got = _kernel_block_scale(m_bits)
    block = np.zeros(32, dtype=np.uint16)
    for i, b in enumerate(m_bits):
        block[5] = b
        block[17] = b | 0x8000  # a negative key of the same magnitude
        sb, bad, rng = O.k_block_scale(block)
        assert not bad
        assert int(got[i]) == sb, (hex(int(b)), hex(int(got[i])), hex(sb))
        assert rng == ((sb & 0x7C00) == 0x7C00)


def test_q8_block_scale_plain_division_would_differ_in_fp32():
    # The fp32 product and fp32 quotient differ for some maxima; only the
    # fp16 results agree, so the identity above is not a tautology.
    m = (np.arange(0x0080, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    q = m / np.float32(127.0)
    r = m * (np.float32(1.0) / np.float32(127.0))
    assert np.count_nonzero(q != r) > 0


# --- values: the encoder's tensor-core rotation and compare-free codes ------
#
# The value encoder (csrc/kvpool_encode.cu) takes the Walsh-Hadamard rotation
# ("PolyKV" section 2.B.2) as H_16 on four index bits through mma.m16n8k16 and
# register butterflies on the rest, with a lane / register layout chosen so
# that 16-byte input chunks are A fragments as they stand.  The functions
# below restate that layout (the PTX fragment layouts of m16n8k16: A row
# groupID + 8 * (i >> 1 & 1), column 2 * tig + (i & 1) + 8 * (i >> 2); B row
# 2 * tig + (i & 1) + 8 * (i >> 1), column groupID; C row groupID + 8 * (i >> 1),
# column 2 * tig + (i & 1)) and check that it computes the oracle's transform.

def _h16_entry(k, n):
    return -1.0 if bin(k & n).count("1") & 1 else 1.0


def _swizzled_slot(d, v, c):
    if d == 128:
        return v * 16 + (c ^ (((c >> 3) & 1) << 1) ^ (v & 1))
    return v * 8 + (c ^ (v & 1))


def _encoder_rotation(V, d):
    """The kernel's rotation of one warp step (8 vectors at d = 128, 16 at
    d = 64), fragment by fragment, in exact arithmetic."""
    cpv = d // 8
    smem = {}
    for j in range(4):                      # the coalesced cp.async fill
        for lane in range(32):
            C = 32 * j + lane
            v, c = C // cpv, C % cpv
            smem[_swizzled_slot(d, v, c)] = V[v, 8 * c:8 * c + 8]
    out = np.zeros_like(V)
    A = [np.zeros((16, 16)) for _ in range(4)]
    for lane in range(32):                  # A fragments: the chunk as it stands
        g, q = lane >> 2, lane & 3
        for m in range(4):
            vec, c = (g, 4 * q + m) if d == 128 else (8 * (m >> 1) + g, 2 * q + (m & 1))
            w = smem[_swizzled_slot(d, vec, c)]
            regs = [w[0:2], w[2:4], w[4:6], w[6:8]]   # registers x, y, z, w
            for i in range(8):
                A[m][g + 8 * ((i >> 1) & 1), 2 * q + (i & 1) + 8 * (i >> 2)] = regs[i >> 1][i & 1]
    B = np.zeros((16, 16))
    for lane in range(32):                  # B fragments as h16_fragments builds them
        g, q = lane >> 2, lane & 3
        for nt in range(2):
            for i in range(4):
                k = 2 * q + (i & 1) + 8 * (i >> 1)
                B[k, 8 * nt + g] = _h16_entry(k, 8 * nt + g)
    for lane in range(32):
        g, q = lane >> 2, lane & 3
        y = np.zeros((4, 2, 2, 2))          # y[m][nt][h] = (c_2h, c_2h+1)
        for m in range(4):
            Cm = A[m] @ B
            for nt in range(2):
                for i in range(4):
                    y[m, nt, i >> 1, i & 1] = Cm[g + 8 * (i >> 1), 8 * nt + 2 * q + (i & 1)]
        for m in range(4):                  # butterflies: h, then bit 0 of m, then bit 1 (d = 128)
            for nt in range(2):
                a_, b_ = y[m, nt, 0].copy(), y[m, nt, 1].copy()
                y[m, nt, 0], y[m, nt, 1] = a_ + b_, a_ - b_
        pairs = [(0, 1), (2, 3)] + ([(0, 2), (1, 3)] if d == 128 else [])
        for m0, m1 in pairs:
            for nt in range(2):
                for h in range(2):
                    a_, b_ = y[m0, nt, h].copy(), y[m1, nt, h].copy()
                    y[m0, nt, h], y[m1, nt, h] = a_ + b_, a_ - b_
        for m in range(4):
            for nt in range(2):
                for h in range(2):
                    for e in range(2):
                        t = m if d == 128 else m & 1
                        vec = g if d == 128 else 8 * (m >> 1) + g
                        out[vec, (d // 4) * q + 8 * t + 4 * nt + 2 * h + e] = y[m, nt, h, e]
    return out


def test_value_rotation_fragment_layout_is_the_oracle_transform():
    rng = np.random.default_rng(11)
    for d in (128, 64):
        V = rng.standard_normal((1024 // d, d))
        got = _encoder_rotation(V, d)
        for v in range(V.shape[0]):
            assert np.allclose(got[v], O.fwht(V[v]), rtol=0, atol=1e-9)


def test_value_staging_swizzle_is_conflict_free():
    for d in (128, 64):
        cpv = d // 8
        seen = set()
        for j in range(4):
            slots = []
            for lane in range(32):
                C = 32 * j + lane
                slots.append(_swizzled_slot(d, C // cpv, C % cpv))
            seen.update(slots)
            for qw in range(4):   # a quarter-warp's 8 16-byte accesses hit 8 bank groups
                assert len({slots[8 * qw + k] % 8 for k in range(8)}) == 8
        assert seen == set(range(128))
        for m in range(4):
            slots = []
            for lane in range(32):
                g, q = lane >> 2, lane & 3
                vec, c = (g, 4 * q + m) if d == 128 else (8 * (m >> 1) + g, 2 * q + (m & 1))
                slots.append(_swizzled_slot(d, vec, c))
            for qw in range(4):
                assert len({slots[8 * qw + k] % 8 for k in range(8)}) == 8


def _fma32(a, b, c):
    """fp32 fma: the exact a * b + c rounded once (exact in fp64 for these
    operands: a product of two fp32 values has at most 48 significant bits)."""
    return np.float32(np.float64(a) * np.float64(b) + np.float64(c))


def _encoder_codes(y32, S):
    """The kernel's codes from the fp32 rotated vector y32 and S = sum y^2:
    sign bits of d_k = y^2 - (t_k^2 / d) S, of P = d_2 y and of Q = d_1 ^ d_3 ^ P,
    inverted, as code bits 0-2 (bit 2 from y, bit 1 from P, bit 0 from Q)."""
    d = y32.size
    t = O.thresholds()[4:]                 # t_1 < t_2 < t_3
    tsq = [np.float32(np.float64(np.float32(x)) ** 2) for x in t]
    nt = [np.float32(-(np.float32(S) * np.float32(tq / np.float32(d)))) for tq in tsq]
    codes = np.zeros(d, np.uint8)
    sign = lambda x: int(np.float32(x).view(np.uint32) >> 31)
    for i, yy in enumerate(y32):
        dk = [_fma32(yy, yy, n) for n in nt]
        P = np.float32(np.float64(dk[1]) * np.float64(yy))
        s, p, q = sign(yy), sign(P), sign(dk[0]) ^ sign(dk[2]) ^ sign(P)
        codes[i] = ((1 - s) << 2) | ((1 - p) << 1) | (1 - q)
    return codes


def _funnel_pack(codes):
    """Codes appended bit by bit (bit 31 of the source shifted in below the
    word's bits), highest coordinate first, into 32-bit words; the kernel
    stores the words' bytes in order."""
    n = codes.size
    words = [0] * ((3 * n + 31) // 32)
    for j in range(n - 1, -1, -1):
        for b in (2, 1, 0):
            p = 3 * j + b
            words[p >> 5] = ((words[p >> 5] << 1) | ((int(codes[j]) >> b) & 1)) & 0xFFFFFFFF
    return np.array(words, np.uint32).view(np.uint8)[: 3 * n // 8]


def test_value_codes_from_signs_match_the_oracle():
    rng = np.random.default_rng(5)
    for d in (128, 64):
        for trial in range(60):
            x = rng.standard_normal(d) * rng.choice([1e-3, 1.0, 30.0])
            if trial % 7 == 0:
                x = np.round(x * 2) / 2          # coarse values: many exact ties
            v_bits = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)  # any bf16 will do
            codes, _, u, flags = O.v_encode_vec(v_bits)
            assert flags == 0
            v = (v_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            y32 = O.fwht(v).astype(np.float32)
            S = np.float32(np.sum(y32.astype(np.float64) ** 2))
            got = _encoder_codes(y32, S)
            t = O.thresholds()
            near = np.min(np.abs(u[:, None] - t[None, :]), axis=1) < 1e-4
            assert np.array_equal(got[~near], codes[~near]), (d, trial)
            # the packing of the kernel's codes is the pool's 3-bit layout
            assert np.array_equal(_funnel_pack(got), O.pack3(got))


def test_value_codes_zero_vector_is_all_fours():
    """A zero vector: y = +0, S = 0, and the kernel uses thresholds of -FLT_MAX
    (finite, so that P = d2 * y is -0 and not inf * 0)."""
    d = 128
    y32 = np.zeros(d, np.float32)
    t = O.thresholds()[4:]
    codes = np.zeros(d, np.uint8)
    sign = lambda x: int(np.float32(x).view(np.uint32) >> 31)
    fmax = np.finfo(np.float32).max
    for i, yy in enumerate(y32):
        dk = [_fma32(yy, yy, -fmax) for _ in t]
        P = np.float32(np.float64(dk[1]) * np.float64(yy))
        s, p, q = sign(yy), sign(P), sign(dk[0]) ^ sign(dk[2]) ^ sign(P)
        codes[i] = ((1 - s) << 2) | ((1 - p) << 1) | (1 - q)
    assert np.all(codes == 4)
    assert np.all(O.v_encode_vec(np.zeros(d, np.uint16))[0] == 4)
