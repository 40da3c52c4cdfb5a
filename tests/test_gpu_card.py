"""GPU parity of the CacheCard path ("QKVShare" Methodology 1-3) against the
fp64 oracle: offsets and header, per-token {2,4,8,16}-bit group
quantization with fp16 scale / zero point, and unpack to bf16
past_key_values, through the C ABI.  Criteria: tests/kvhelp.py."""
import numpy as np
import pytest
import torch

import agent_shared_compressed_gb300 as kv
from agent_shared_compressed_gb300 import build as kvbuild
from agent_shared_compressed_gb300 import synth
import oracle as O
from kvhelp import CARD_BAND, Guarded, assert_bf16_close, bf16_dev_layers, card_tokens, split_record

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    kvbuild.build()
    kv.load()


def inputs(L, H, T, d, seed):
    ks, vs = synth.kv_layers(L, H, T, d, seed=seed, device="cpu")
    bits = synth.card_bits(T, seed=seed).numpy()
    return [synth.bits16(k) for k in ks], [synth.bits16(v) for v in vs], bits


def gpu_pack(kd, vd, bits, shape, model_id=0, pos=0, nbytes=None):
    n = kv.cachecard_bytes(shape, bits) if nbytes is None else nbytes
    card = Guarded(n, fill=0x5A)
    bits_dev = torch.from_numpy(np.ascontiguousarray(bits, np.uint8)).cuda()
    st = torch.cuda.current_stream()
    rc = kv.cachecard_pack(shape, model_id, pos, bits_dev, kd, vd, card.t, card.nbytes, st)
    assert rc == kv.KVP_OK, kv.kvp_strerror(rc)
    status = kv.cachecard_status(card.t, st)
    assert card.canary_ok()
    return card, status


def gpu_unpack(card, L, H, T, d):
    hdr = kv.CardHeader()
    assert kv.cachecard_read_header(card.t, hdr) == kv.KVP_OK
    ko = [Guarded(H * T * d * 2, fill=0xFF) for _ in range(L)]
    vo = [Guarded(H * T * d * 2, fill=0xFF) for _ in range(L)]
    assert kv.cachecard_unpack(card.t, hdr, [g.t for g in ko], [g.t for g in vo]) == kv.KVP_OK
    torch.cuda.synchronize()
    assert all(g.canary_ok() for g in ko + vo)
    return hdr, [synth.bits16(g.bf16((H, T, d))) for g in ko], [synth.bits16(g.bf16((H, T, d))) for g in vo]


def assert_card_parity(gimg, oimg, r, L, H, d, T, bits):
    geo = O.card_geometry(L, H, d, T, bits)
    np.testing.assert_array_equal(gimg[: geo["off_layers"]], oimg[: geo["off_layers"]])  # header, bits, offsets
    G = card_tokens(gimg, geo, L, H, d, T, bits)
    R = card_tokens(oimg, geo, L, H, d, T, bits)
    n_band = 0
    for b, (idx, grec) in G.items():
        orec = R[b][1]
        if b == 16:
            np.testing.assert_array_equal(grec, orec)
            continue
        gc, gp = split_record(grec, b, H, d)
        oc, op = split_record(orec, b, H, d)
        np.testing.assert_array_equal(gp, op, err_msg="fp16 scale/zero, b=%d" % b)
        rr = r[:, idx].reshape(L, idx.size, 2, H * d)
        band = np.abs(rr - np.floor(rr) - 0.5) < CARD_BAND
        bad = (gc != oc) & ~band
        assert not bad.any(), "b=%d: %d codes differ outside the band" % (b, bad.sum())
        n_band += int(((gc != oc) & band).sum())
    # layer tails after the last record: zero
    used = int(gimg[geo["off_offsets"] + 4 * (T - 1): geo["off_offsets"] + 4 * T].view(np.uint32)[0]) + \
        O.card_record_bytes(int(bits[-1]), H, d)
    for l in range(L):
        base = geo["off_layers"] + l * geo["layer_stride"]
        assert not gimg[base + used: base + geo["layer_stride"]].any()
    return n_band


@pytest.mark.parametrize("shape", [(3, 5, 64, 37), (2, 8, 128, 64), (1, 1, 64, 1), (2, 3, 128, 50),
                                   (1, 8, 128, 1500), (2, 32, 64, 129), (1, 32, 128, 33)])
def test_card_pack_unpack_match_oracle(shape):
    L, H, d, T = shape
    ks, vs, bits = inputs(L, H, T, d, seed=T + L)
    if T >= 4:
        bits[:4] = [2, 4, 8, 16]                      # every bitwidth present
    kd, vd = bf16_dev_layers(ks), bf16_dev_layers(vs)
    card, status = gpu_pack(kd, vd, bits, shape, model_id=0xFEEDFACE12345678, pos=-4096)
    assert status == kv.KVP_OK
    oimg, flags, r = O.card_pack(ks, vs, bits, model_id=0xFEEDFACE12345678, pos_offset=-4096, want_r=True)
    assert flags == 0
    gimg = card.host()
    assert gimg.size == oimg.size
    assert_card_parity(gimg, oimg, r, L, H, d, T, bits)
    hdr, ku, vu = gpu_unpack(card, L, H, T, d)
    assert (hdr.seq_len, hdr.n_layers, hdr.n_kv_heads, hdr.head_dim) == (T, L, H, d)
    assert hdr.model_id == 0xFEEDFACE12345678 and hdr.pos_offset == -4096 and hdr.error == 0
    ok_, ov = O.card_unpack(gimg)                      # oracle decodes the GPU's own card
    for l in range(L):
        assert_bf16_close(ku[l], ok_[l], "K layer %d" % l)
        assert_bf16_close(vu[l], ov[l], "V layer %d" % l)
        full = bits == 16                                # 16-bit tokens: verbatim
        np.testing.assert_array_equal(ku[l][:, full], ks[l][:, full])
        np.testing.assert_array_equal(vu[l][:, full], vs[l][:, full])


@pytest.mark.parametrize("shape", [(2, 8, 128, 64), (2, 3, 64, 37)])
def test_card_pack_from_16_byte_aligned_layers(shape):
    """Layers with only the 16-byte alignment the ABI asks for (not 32-byte)
    pack to a card byte-identical to the one packed from 512-byte aligned
    copies, and it matches the oracle's."""
    L, H, d, T = shape
    ks, vs, bits = inputs(L, H, T, d, seed=T + 7)
    kd, vd = bf16_dev_layers(ks), bf16_dev_layers(vs)

    def shifted(t):
        buf = torch.empty(t.numel() + 8, dtype=torch.bfloat16, device="cuda")
        view = buf[8:8 + t.numel()]                      # 16 bytes past a 512-byte aligned start
        view.copy_(t.reshape(-1))
        assert view.data_ptr() % 32 == 16
        return view

    card_a, st_a = gpu_pack(kd, vd, bits, shape)
    card_u, st_u = gpu_pack([shifted(k) for k in kd], [shifted(v) for v in vd], bits, shape)
    assert st_a == kv.KVP_OK and st_u == kv.KVP_OK
    np.testing.assert_array_equal(card_u.host(), card_a.host())
    oimg, flags, r = O.card_pack(ks, vs, bits, want_r=True)
    assert flags == 0
    assert_card_parity(card_u.host(), oimg, r, L, H, d, T, bits)


def test_card_on_grid_values_roundtrip_exactly():
    """Groups whose values sit on their own quantization grid (s, z exact in
    fp16, every value z + q*s exact in bf16) come back bit-exact."""
    L, H, d, T = 1, 2, 64, 12
    rng = np.random.default_rng(4)
    bits = np.array([2, 4, 8, 2, 4, 8, 2, 4, 8, 16, 4, 8], np.uint8)
    ks, vs = [], []
    for _ in range(2):
        x = np.zeros((H, T, d))
        for t in range(T):
            b = int(bits[t]) if bits[t] < 16 else 8
            qm = 2 ** b - 1
            for h in range(H):
                for g in range(d // 32):
                    q = rng.integers(0, qm + 1, 32)
                    q[0], q[1] = 0, qm
                    x[h, t, 32 * g: 32 * g + 32] = -2.0 + 0.5 * q     # s = 0.5, z = -2
        (ks if not ks else vs).append((np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16))
    card, status = gpu_pack(bf16_dev_layers(ks), bf16_dev_layers(vs), bits, (L, H, d, T))
    assert status == kv.KVP_OK
    _, ku, vu = gpu_unpack(card, L, H, T, d)
    np.testing.assert_array_equal(ku[0], ks[0])
    np.testing.assert_array_equal(vu[0], vs[0])


def test_card_invalid_bits_and_small_buffer():
    L, H, d, T = 2, 2, 64, 10
    ks, vs, bits = inputs(L, H, T, d, seed=2)
    kd, vd = bf16_dev_layers(ks), bf16_dev_layers(vs)
    bad = bits.copy()
    bad[5] = 3
    good_bytes = kv.cachecard_bytes((L, H, d, T), bits)
    card, status = gpu_pack(kd, vd, bad, (L, H, d, T), nbytes=good_bytes)
    assert status == kv.KVP_ERR_BITS
    hdr = kv.CardHeader()
    assert kv.cachecard_read_header(card.t, hdr) == kv.KVP_OK
    assert kv.cachecard_unpack(card.t, hdr, [0x10000] * L, [0x10000] * L) == kv.KVP_ERR_HEADER
    # records untouched (the fill pattern survives past the offsets table)
    geo = O.card_geometry(L, H, d, T, bits)
    assert np.all(card.host()[geo["off_layers"]:] == 0x5A)
    small = kv.cachecard_bytes((L, H, d, T), bits) - 256
    card2, status2 = gpu_pack(kd, vd, bits, (L, H, d, T), nbytes=small)
    assert status2 == kv.KVP_ERR_SIZE
    assert np.all(card2.host()[geo["off_layers"]:] == 0x5A)


@pytest.mark.parametrize("shape", [(2, 8, 128, 20), (1, 32, 128, 9)])
def test_card_unpack_rejects_corrupt_records(shape):
    """A card corrupted after packing: one token's record offset moved off its
    16-byte boundary, another's bitwidth byte set to 3.  Both records are
    rejected before anything is read from them (the staged kernel, first
    shape, and the direct one, second); cachecard_status reports
    KVP_ERR_HEADER, and every other token unpacks as from the intact card."""
    L, H, d, T = shape
    ks, vs, bits = inputs(L, H, T, d, seed=T + 3)
    kd, vd = bf16_dev_layers(ks), bf16_dev_layers(vs)
    card, status = gpu_pack(kd, vd, bits, shape)
    assert status == kv.KVP_OK
    hdr0, k0, v0 = gpu_unpack(card, L, H, T, d)
    img = card.host().copy()
    offs = img[hdr0.off_offsets:hdr0.off_offsets + 4 * T].view(np.uint32)
    offs[3] += 8                                        # misaligned, still inside the layer
    img[hdr0.off_bits + 6] = 3                          # not a bitwidth
    bad = Guarded(img.size)
    bad.t[: img.size].copy_(torch.from_numpy(img))
    hdr = kv.CardHeader()
    assert kv.cachecard_read_header(bad.t, hdr) == kv.KVP_OK
    ko = [Guarded(H * T * d * 2, fill=0xFF) for _ in range(L)]
    vo = [Guarded(H * T * d * 2, fill=0xFF) for _ in range(L)]
    assert kv.cachecard_unpack(bad.t, hdr, [g.t for g in ko], [g.t for g in vo]) == kv.KVP_OK
    torch.cuda.synchronize()
    assert kv.cachecard_status(bad.t) == kv.KVP_ERR_HEADER
    assert all(g.canary_ok() for g in ko + vo)
    keep = np.ones(T, bool)
    keep[[3, 6]] = False
    for l in range(L):
        ku, vu = synth.bits16(ko[l].bf16((H, T, d))), synth.bits16(vo[l].bf16((H, T, d)))
        np.testing.assert_array_equal(ku[:, keep], k0[l][:, keep])
        np.testing.assert_array_equal(vu[:, keep], v0[l][:, keep])
        assert np.all(ku[:, ~keep] == 0xFFFF) and np.all(vu[:, ~keep] == 0xFFFF)   # left unwritten


def test_card_nonfinite_and_range_flags():
    L, H, d, T = 1, 1, 64, 4
    ks, vs, _ = inputs(L, H, T, d, seed=3)
    bits = np.array([2, 4, 8, 16], np.uint8)
    k = ks[0].copy()
    k[0, 1, 5] = 0x7FC0                                       # NaN in a 4-bit token
    card, status = gpu_pack(bf16_dev_layers([k]), bf16_dev_layers(vs), bits, (L, H, d, T))
    assert status == kv.KVP_ERR_NONFINITE
    v = vs[0].copy()
    v[0, 2, :32] = (np.full(32, 1e5, np.float32).view(np.uint32) >> 16).astype(np.uint16)   # z > fp16 max
    card, status = gpu_pack(bf16_dev_layers(ks), bf16_dev_layers([v]), bits, (L, H, d, T))
    assert status == kv.KVP_ERR_RANGE
    _, f, _ = O.card_pack(ks, [v], bits)
    assert f == O.FLAG_RANGE


def test_card_full_size():
    """The Llama-3.1-8B-shaped CacheCard at 8192 tokens with i.i.d. bitwidths,
    packed and unpacked in the benchmark's launch configuration; packed
    records compared with the oracle on sampled tokens, the unpacked cache
    compared in full with the oracle's unpack of the same card."""
    w = synth.WORKLOADS["llama31-8b-cachecard-8k"]
    L, H, d, T = w["L"], w["H"], w["d"], w["T"]
    shape = (L, H, d, T)
    ks_t, vs_t = synth.kv_layers(L, H, T, d, seed=0, device="cuda")
    bits = synth.card_bits(T, seed=0).numpy()
    card, status = gpu_pack(ks_t, vs_t, bits, shape, model_id=42, pos=0)
    assert status == kv.KVP_OK
    gimg = card.host()
    geo = O.card_geometry(L, H, d, T, bits)
    assert gimg.size == geo["total"]
    offs = gimg[geo["off_offsets"]: geo["off_offsets"] + 4 * T].view(np.uint32)
    sizes = np.array([O.card_record_bytes(int(b), H, d) for b in bits])
    np.testing.assert_array_equal(offs, np.concatenate([[0], np.cumsum(sizes)[:-1]]))
    rng = np.random.default_rng(0)
    for l in rng.choice(L, 4, replace=False):
        kb, vb = synth.bits16(ks_t[l]), synth.bits16(vs_t[l])
        for t in rng.choice(T, 60, replace=False):
            b = int(bits[t])
            rec = gimg[geo["off_layers"] + l * geo["layer_stride"] + int(offs[t]):][: O.card_record_bytes(b, H, d)]
            if b == 16:
                np.testing.assert_array_equal(rec[: H * d * 2].view(np.uint16).reshape(H, d), kb[:, t])
                continue
            codes, par = split_record(rec[None], b, H, d)
            for kvi, src in enumerate((kb, vb)):
                for h in range(H):
                    for gi in range(d // 32):
                        x = ((src[h, t, 32 * gi: 32 * gi + 32].astype(np.uint32) << 16).view(np.float32)).astype(np.float64)
                        q, sb, zb, r, _ = O.group_quant(x, b)
                        p = int(par[0, kvi, h * (d // 32) + gi])
                        assert (p & 0xFFFF, p >> 16) == (sb, zb)
                        got = codes[0, kvi, h * d + 32 * gi: h * d + 32 * gi + 32]
                        band = np.abs(r - np.floor(r) - 0.5) < CARD_BAND
                        assert np.all((got == q) | band)
    _, ku, vu = gpu_unpack(card, L, H, T, d)
    ok_, ov = O.card_unpack(gimg)
    for l in range(L):
        assert_bf16_close(ku[l], ok_[l], "K layer %d" % l)
        assert_bf16_close(vu[l], ov[l], "V layer %d" % l)


def test_card_group_scales_across_fp16_range():
    """Groups whose scale (max - min) / (2^b - 1) falls in fp16's subnormal
    range, at zero (constant groups), in the normal range and near its top, and
    zero points up to 3e4, on every bitwidth: the exactly rounded fp16 scale
    and zero point, the codes (outside the half-integer band) and the unpacked
    values match the oracle."""
    L, H, d, T = 1, 2, 64, 16
    rng = np.random.default_rng(8)
    spans = [0.0, 1e-8, 2e-7, 3e-6, 4e-5, 1e-3, 0.5, 20.0, 900.0, 3e4]
    bases = [0.0, -1e-6, 5e-5, 1.0, -30.0, 3e4]
    x = np.zeros((2, H, T, d), np.float64)
    for part in range(2):
        for h in range(H):
            for t in range(T):
                for gi in range(d // 32):
                    span = spans[(t + 3 * gi + part + h) % len(spans)]
                    base = bases[(2 * t + gi + h) % len(bases)]
                    x[part, h, t, 32 * gi: 32 * gi + 32] = base + span * rng.uniform(0, 1, 32)
    bits16 = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)   # bf16 by truncation
    ks, vs = [bits16[0]], [bits16[1]]
    bits = np.array([[2, 4, 8, 16][t % 4] for t in range(T)], np.uint8)
    card, status = gpu_pack(bf16_dev_layers(ks), bf16_dev_layers(vs), bits, (L, H, d, T))
    assert status == kv.KVP_OK
    oimg, flags, r = O.card_pack(ks, vs, bits, want_r=True)
    assert flags == 0
    gimg = card.host()
    assert_card_parity(gimg, oimg, r, L, H, d, T, bits)
    _, gk, gv = gpu_unpack(card, L, H, T, d)
    ok_, ov = O.card_unpack(gimg)
    assert_bf16_close(gk[0], ok_[0], "K")
    assert_bf16_close(gv[0], ov[0], "V")
