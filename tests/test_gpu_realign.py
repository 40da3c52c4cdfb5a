"""GPU parity of cachecard_unpack_at -- CacheCard unpack with every key moved
from the card's position offset to another (rotary realignment: "KVCMAS",
How it is used; the offset travels in the card, "QKVShare" Methodology 2) --
against the fp64 oracle's realigned unpack of the same card image.

Criteria: keys within one bf16 ulp of the oracle plus 2^-20 of their rotary
pair's norm (the kernel dequantizes and turns in fp32, a few fp32 ulps before
its one rounding to bf16); values bit-identical to cachecard_unpack's; a zero
shift reproduces cachecard_unpack bit for bit."""
import numpy as np
import pytest
import torch

import agent_shared_compressed_gb300 as kv
from agent_shared_compressed_gb300 import build as kvbuild
from agent_shared_compressed_gb300 import synth
import oracle as O
from kvhelp import Guarded, assert_bf16_close, bf16_dev_layers, f32_of_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    kvbuild.build()
    kv.load()


def inv_freq(d, kind):
    if kind == "llama3":  # Llama-3 rotary base
        return (1.0 / 500000.0 ** (np.arange(0, d, 2, dtype=np.float64) / d)).astype(np.float32)
    if kind == "unit":    # one radian per position on every pair: the largest angles
        return np.ones(d // 2, np.float32)
    return np.linspace(0.001, 2.5, d // 2).astype(np.float32)


def pack(kd, vd, bits, shape, pos):
    n = kv.cachecard_bytes(shape, bits)
    card = Guarded(n, fill=0x5A)
    bits_dev = torch.from_numpy(np.ascontiguousarray(bits, np.uint8)).cuda()
    rc = kv.cachecard_pack(shape, 7, pos, bits_dev, kd, vd, card.t, card.nbytes, torch.cuda.current_stream())
    assert rc == kv.KVP_OK and kv.cachecard_status(card.t) == kv.KVP_OK
    return card


def unpack(card, L, H, T, d, pos_dst=None, w=None):
    hdr = kv.CardHeader()
    assert kv.cachecard_read_header(card.t, hdr) == kv.KVP_OK
    ko = [Guarded(H * T * d * 2, fill=0xFF) for _ in range(L)]
    vo = [Guarded(H * T * d * 2, fill=0xFF) for _ in range(L)]
    if pos_dst is None:
        rc = kv.cachecard_unpack(card.t, hdr, [g.t for g in ko], [g.t for g in vo])
    else:
        rc = kv.cachecard_unpack_at(card.t, hdr, pos_dst, w, [g.t for g in ko], [g.t for g in vo])
    assert rc == kv.KVP_OK, kv.kvp_strerror(rc)
    torch.cuda.synchronize()
    assert all(g.canary_ok() for g in ko + vo)
    assert kv.cachecard_status(card.t) == kv.KVP_OK
    return [synth.bits16(g.bf16((H, T, d))) for g in ko], [synth.bits16(g.bf16((H, T, d))) for g in vo]


def assert_keys_close(gpu_bits, ora_bits, what):
    a, b = f32_of_bf16(gpu_bits).astype(np.float64), f32_of_bf16(ora_bits).astype(np.float64)
    half = b.shape[-1] // 2
    pn = np.sqrt(b[..., :half] ** 2 + b[..., half:] ** 2)
    pn = np.concatenate([pn, pn], -1)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(b), 2.0 ** -126))) - 7)
    bad = np.abs(a - b) > ulp + 2.0 ** -20 * pn
    assert not bad.any(), "%s: %d keys off (worst %r vs %r)" % (what, bad.sum(), a[bad][:3], b[bad][:3])
    return float(np.mean(gpu_bits == ora_bits))


CASES = [  # (L, H, d, T, pos_src, pos_dst, frequencies)
    (2, 3, 64, 37, -4096, 123457, "llama3"),
    (1, 8, 128, 300, 0, 4096, "llama3"),
    (3, 2, 128, 9, 5000, 12, "unit"),
    (2, 4, 64, 65, 17, -40000, "ramp"),
    (1, 16, 128, 40, 3, 700, "llama3"),  # staged in more than 48 KB of shared memory per block
    (1, 32, 128, 20, 9, 2000, "ramp"),   # records too large to stage: the direct kernel
]


@pytest.mark.parametrize("case", CASES)
def test_unpack_at_matches_oracle(case):
    L, H, d, T, p0, p1, kind = case
    shape = (L, H, d, T)
    ks, vs = synth.kv_layers(L, H, T, d, seed=T, device="cpu")
    ks, vs = [synth.bits16(k) for k in ks], [synth.bits16(v) for v in vs]
    bits = synth.card_bits(T, seed=T).numpy()
    bits[:4] = [2, 4, 8, 16]
    card = pack(bf16_dev_layers(ks), bf16_dev_layers(vs), bits, shape, p0)
    w = inv_freq(d, kind)
    ku, vu = unpack(card, L, H, T, d, p1, w)
    kp, vp = unpack(card, L, H, T, d)
    ok_, _ = O.card_unpack_at(card.host(), p1, w)
    for l in range(L):
        same = assert_keys_close(ku[l], ok_[l], "K layer %d" % l)
        assert same > 0.9, same
        np.testing.assert_array_equal(vu[l], vp[l])


def test_unpack_at_zero_shift_is_unpack():
    L, H, d, T = 2, 8, 128, 100
    ks, vs = synth.kv_layers(L, H, T, d, seed=5, device="cuda")
    bits = synth.card_bits(T, seed=5).numpy()
    card = pack(ks, vs, bits, (L, H, d, T), 777)
    ku, vu = unpack(card, L, H, T, d, 777, inv_freq(d, "unit"))
    kp, vp = unpack(card, L, H, T, d)
    for l in range(L):
        np.testing.assert_array_equal(ku[l], kp[l])
        np.testing.assert_array_equal(vu[l], vp[l])


def test_unpack_at_full_size():
    """The Llama-3.1-8B-shaped card at 8192 tokens, re-aligned by 4096
    positions in the benchmark's launch configuration, compared in full with
    the oracle's realigned unpack of the same card."""
    w = synth.WORKLOADS["llama31-8b-cachecard-8k"]
    L, H, d, T = w["L"], w["H"], w["d"], w["T"]
    ks_t, vs_t = synth.kv_layers(L, H, T, d, seed=0, device="cuda")
    bits = synth.card_bits(T, seed=0).numpy()
    card = pack(ks_t, vs_t, bits, (L, H, d, T), 0)
    fr = inv_freq(d, "llama3")
    ku, vu = unpack(card, L, H, T, d, 4096, fr)
    ok_, _ = O.card_unpack_at(card.host(), 4096, fr)
    for l in range(L):
        assert_keys_close(ku[l], ok_[l], "K layer %d" % l)
    # values: the plain unpack's (itself checked against the oracle elsewhere)
    _, vp = unpack(card, L, H, T, d)
    for l in range(L):
        np.testing.assert_array_equal(vu[l], vp[l])


@pytest.mark.parametrize("realign", [False, True])
def test_unpack_wait_timeout_is_reported(realign):
    """The staged unpack's bounded wait for a record's bulk copies, made to run
    out on every warp's first record, is reported by cachecard_status as
    KVP_ERR_TIMEOUT with the context still usable; the hook applies to one
    call only, and the next unpack of a fresh card is whole and correct."""
    L, H, d, T = 2, 8, 128, 300
    ks, vs = synth.kv_layers(L, H, T, d, seed=11, device="cuda")
    bits = synth.card_bits(T, seed=11).numpy()
    w = inv_freq(d, "llama3")
    card = pack(ks, vs, bits, (L, H, d, T), 0)
    hdr = kv.CardHeader()
    assert kv.cachecard_read_header(card.t, hdr) == kv.KVP_OK
    ko = [torch.empty(H * T * d, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    vo = [torch.empty(H * T * d, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    assert kv.kvp_test_limit_next_unpack(0) == kv.KVP_OK
    if realign:
        rc = kv.cachecard_unpack_at(card.t, hdr, 4096, w, ko, vo)
    else:
        rc = kv.cachecard_unpack(card.t, hdr, ko, vo)
    assert rc == kv.KVP_OK
    torch.cuda.synchronize()
    assert kv.cachecard_status(card.t) == kv.KVP_ERR_TIMEOUT
    card2 = pack(ks, vs, bits, (L, H, d, T), 0)          # the first card keeps its error word
    ku, vu = unpack(card2, L, H, T, d, 4096 if realign else None, w if realign else None)
    if realign:
        ok_, _ = O.card_unpack_at(card2.host(), 4096, w)
        for l in range(L):
            assert_keys_close(ku[l], ok_[l], "K layer %d" % l)
    kp, vp = unpack(card2, L, H, T, d)
    for l in range(L):
        np.testing.assert_array_equal(vu[l], vp[l])
        if not realign:
            np.testing.assert_array_equal(ku[l], kp[l])


@pytest.mark.parametrize("shape,fill", [((1, 8, 128, 1), 16), ((1, 8, 128, 1), 2), ((2, 8, 128, 5), 16),
                                        ((2, 8, 128, 5), 2), ((1, 4, 64, 3), 8), ((3, 2, 128, 2), 4)])
def test_staged_unpack_edge_cases(shape, fill):
    """The staged unpack (every shape here stages) at its edges: a single
    token, fewer tokens than a block has warps, and every record at the
    largest (16-bit) or smallest (2-bit) size; plain and realigning unpack
    against the oracle, values of the two bit-identical."""
    L, H, d, T = shape
    ks, vs = synth.kv_layers(L, H, T, d, seed=T + fill, device="cpu")
    ks, vs = [synth.bits16(k) for k in ks], [synth.bits16(v) for v in vs]
    bits = np.full(T, fill, np.uint8)
    card = pack(bf16_dev_layers(ks), bf16_dev_layers(vs), bits, shape, 11)
    kp, vp = unpack(card, L, H, T, d)
    ok_, ov = O.card_unpack(card.host())
    for l in range(L):
        assert_bf16_close(kp[l], ok_[l], "K layer %d" % l)
        assert_bf16_close(vp[l], ov[l], "V layer %d" % l)
        if fill == 16:
            np.testing.assert_array_equal(kp[l], ks[l])
            np.testing.assert_array_equal(vp[l], vs[l])
    w = inv_freq(d, "llama3")
    ku, vu = unpack(card, L, H, T, d, 11 + 3000, w)
    oka, _ = O.card_unpack_at(card.host(), 11 + 3000, w)
    for l in range(L):
        assert_keys_close(ku[l], oka[l], "K layer %d" % l)
        np.testing.assert_array_equal(vu[l], vp[l])
