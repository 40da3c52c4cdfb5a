"""GPU parity of the q8_0 key format (KVP_K_Q8_0; "PolyKV" 2.B.1 labels its
int8 key step "q8_0": 32 keys along d share an fp16 scale) against the fp64
oracle, through the C ABI: the whole pool image from kvpool_encode_ex (header
with the format word, int8 codes, block scales, and the value sections that
do not depend on the key format), fan-out decode and pool attention over a
q8_0 pool.  Key codes and block scales are compared bit for bit: the
kernel's rounding decisions are exact.  Other criteria: tests/kvhelp.py and
tests/test_gpu_attend.py."""
import math

import numpy as np
import pytest
import torch

import agent_shared_compressed_gb300 as kv
from agent_shared_compressed_gb300 import build as kvbuild
from agent_shared_compressed_gb300 import synth
import oracle as O
from kvhelp import (Guarded, assert_bf16_close, assert_pool_parity, bf16_dev_layers, f32_of_bf16,
                    guarded_caches, pool_sections, unpack3_np)
from test_gpu_attend import _attend, _check

pytestmark = pytest.mark.gpu
Q8 = kv.KVP_K_Q8_0


@pytest.fixture(scope="module", autouse=True)
def built():
    kvbuild.build()
    kv.load()


def encode_q8(kd, vd, shape):
    pool = Guarded(kv.kvpool_pool_bytes_ex(shape, Q8), fill=0x5A)
    ws = Guarded(kv.kvpool_workspace_bytes(shape), fill=0x77)
    st = torch.cuda.current_stream()
    rc = kv.kvpool_encode_ex(shape, Q8, kd, vd, pool.t, pool.nbytes, ws.t, ws.nbytes, st)
    assert rc == kv.KVP_OK, kv.kvp_strerror(rc)
    status = kv.kvpool_status(pool.t, st)
    assert pool.canary_ok() and ws.canary_ok()
    return pool, status


def kscales(img, L, H, d, T):
    off, total = O.pool_geometry_q8(L, H, d, T)
    nb = H * T * d // 32
    return img[off: off + L * nb * 2].view(np.uint16).reshape(L, H, T, d // 32), img[off + L * nb * 2: total]


def assert_q8_pool(gimg, oimg, u, L, H, d, T):
    assert gimg.size == oimg.size == kv.kvpool_pool_bytes_ex((L, H, d, T), Q8)
    assert_pool_parity(gimg, oimg, u, L, H, d, T)   # header (format word 1), codes, values, gaps
    sg, tail = kscales(gimg, L, H, d, T)
    so, _ = kscales(oimg, L, H, d, T)
    np.testing.assert_array_equal(sg, so)
    assert not tail.any()


SMALL = [(1, 8, 128, 512), (2, 32, 64, 1851), (3, 5, 64, 37), (2, 3, 128, 7), (1, 1, 64, 1), (4, 2, 128, 129)]


@pytest.mark.parametrize("shape", SMALL)
def test_encode_q8_matches_oracle(shape):
    L, H, d, T = shape
    ks, vs = synth.kv_layers(L, H, T, d, seed=L * 100 + T, device="cpu")
    ks, vs = [synth.bits16(k) for k in ks], [synth.bits16(v) for v in vs]
    pool, status = encode_q8(bf16_dev_layers(ks), bf16_dev_layers(vs), shape)
    assert status == kv.KVP_OK
    ora, flags, u = O.pool_encode(ks, vs, want_u=True, k_mode=1)
    assert flags == 0
    assert_q8_pool(pool.host(), ora, u, L, H, d, T)


def test_encode_q8_edge_blocks():
    """Zero blocks, blocks whose scale is an fp16 subnormal (codes clamp) or
    rounds to zero, on-grid blocks and large blocks, bit for bit; then a
    non-finite key and a scale beyond fp16 reported by kvpool_status."""
    L, H, d, T = 1, 2, 128, 6
    rng = np.random.default_rng(8)
    x = rng.normal(size=(H, T, d))
    x[0, 0, :32] = 0.0
    x[0, 1, 32:64] = rng.normal(size=32) * 1e-6          # scale below 2^-14: subnormal
    x[0, 2, 64:96] = rng.normal(size=32) * 127 * 2.0 ** -22
    x[0, 3, 96:] = np.full(32, 127 * 2.0 ** -26)          # scale rounds to zero
    x[1, 0, :32] = np.arange(-127, 128, 8)[:32] * 2.0 ** -3
    x[1, 1] = rng.normal(size=d) * 3000.0
    x[1, 5, 5] *= 1.0e3
    ks = [synth.bits16(torch.from_numpy(x).to(torch.bfloat16))]
    vs = [synth.bits16(torch.from_numpy(rng.normal(size=(H, T, d))).to(torch.bfloat16))]
    pool, status = encode_q8(bf16_dev_layers(ks), bf16_dev_layers(vs), (L, H, d, T))
    assert status == kv.KVP_OK
    ora, flags, u = O.pool_encode(ks, vs, want_u=True, k_mode=1)
    assert flags == 0
    assert_q8_pool(pool.host(), ora, u, L, H, d, T)
    for value, want in ((float("nan"), kv.KVP_ERR_NONFINITE), (1.0e7, kv.KVP_ERR_RANGE)):
        y = x.copy()
        y[1, 3, 40] = value
        kb = [synth.bits16(torch.from_numpy(y).to(torch.bfloat16))]
        _, st = encode_q8(bf16_dev_layers(kb), bf16_dev_layers(vs), (L, H, d, T))
        assert st == want, kv.kvp_strerror(st)


@pytest.mark.parametrize("shape,n", [((1, 8, 128, 512), 2), ((2, 32, 64, 1851), 3), ((3, 5, 64, 37), 1)])
def test_decode_q8_matches_oracle(shape, n):
    L, H, d, T = shape
    ks_t, vs_t = synth.kv_layers(L, H, T, d, seed=3 + T, device="cuda")
    pool, status = encode_q8(ks_t, vs_t, shape)
    assert status == kv.KVP_OK
    img = pool.host()
    ck = guarded_caches(L, H, T, d, n)
    cv = guarded_caches(L, H, T, d, n)
    rc = kv.kvpool_decode_into(pool.t, shape, 0, L, n, [c.t for a in ck for c in a], [c.t for a in cv for c in a])
    assert rc == kv.KVP_OK
    torch.cuda.synchronize()
    assert kv.kvpool_status(pool.t) == kv.KVP_OK
    ok_, ov = O.pool_decode_into(img, 0, L, 1)
    sc, _ = kscales(img, L, H, d, T)
    for l in range(L):
        k0, v0 = synth.bits16(ck[0][l].bf16((H, T, d))), synth.bits16(cv[0][l].bf16((H, T, d)))
        np.testing.assert_array_equal(k0, ok_[0][l])   # q * s_b, one rounding: bit-exact
        assert_bf16_close(v0, ov[0][l], "V layer %d" % l)
        for a in range(1, n):
            assert torch.equal(ck[a][l].t, ck[0][l].t) and torch.equal(cv[a][l].t, cv[0][l].t)
        s_b = np.repeat(np.array([O.f16_to_f64(int(b)) for b in sc[l].ravel()]).reshape(H, T, d // 32), 32, -1)
        x = f32_of_bf16(synth.bits16(ks_t[l]))
        err = np.abs(f32_of_bf16(k0) - x)
        assert np.all(err <= s_b / 2 + 2.0 ** -8 * np.abs(x) + 1e-30)


ATT_CASES = [(2, 2, 64, 37, 3, 8), (1, 8, 128, 512, 15, 32), (1, 4, 128, 1000, 4, 32), (2, 4, 128, 129, 20, 16)]


@pytest.mark.parametrize("case", ATT_CASES)
def test_attend_q8_matches_oracle(case):
    L, H, d, T, na, nq = case
    shape = (L, H, d, T)
    ks_t, vs_t = synth.kv_layers(L, H, T, d, seed=T + na, device="cuda")
    pool, status = encode_q8(ks_t, vs_t, shape)
    assert status == kv.KVP_OK
    img = pool.host()
    g = torch.Generator(device="cpu").manual_seed(9)
    q = torch.randn(na, nq, d, generator=g).to(torch.bfloat16)
    for layer in {0, L - 1}:
        out, lse = _attend(pool.t, shape, layer, q.cuda(), 1.0 / math.sqrt(d))
        _check(img, shape, layer, synth.bits16(q), 1.0 / math.sqrt(d), out, lse)


def test_q8_full_size_sampled():
    """The 4K-token, 15-agent Llama-3-8B workload encoded with q8_0 keys in
    one launch: sampled layers compared with the oracle's encode of those
    layers, a decode of two agents compared with the oracle's decode of the
    same image, and attention over the last layer."""
    w = synth.WORKLOADS["llama3-8b-4k-15agents"]
    L, H, d, T, N = w["L"], w["H"], w["d"], w["T"], w["N"]
    shape = (L, H, d, T)
    ks_t, vs_t = synth.kv_layers(L, H, T, d, seed=0, device="cuda")
    pool, status = encode_q8(ks_t, vs_t, shape)
    assert status == kv.KVP_OK
    img = pool.host()
    sec = pool_sections(img, L, H, d, T)
    sc, tail = kscales(img, L, H, d, T)
    assert not tail.any() and not sec["scales"].any()
    rng = np.random.default_rng(2)
    for l in rng.choice(L, 3, replace=False):
        kb, vb = synth.bits16(ks_t[l]), synth.bits16(vs_t[l])
        ora, flags, u = O.pool_encode([kb], [vb], want_u=True, k_mode=1)
        assert flags == 0
        so = pool_sections(ora, 1, H, d, T)
        np.testing.assert_array_equal(sec["k"][l], so["k"][0])
        np.testing.assert_array_equal(sc[l], kscales(ora, 1, H, d, T)[0][0])
        cg, co = unpack3_np(sec["vpacked"][l], d), unpack3_np(so["vpacked"][0], d)
        band = np.zeros(cg.shape, bool)
        for t in O.thresholds():
            band |= np.abs(u[0].reshape(H * T, d) - t) < 1e-4
        assert not ((cg != co) & ~band).any()
        assert np.abs(sec["sigma"][l].astype(np.int32) - so["sigma"][0].astype(np.int32)).max() <= 1
    lb, le = L - 2, L
    ck = [[torch.empty((H, T, d), dtype=torch.bfloat16, device="cuda") for _ in range(L)] for _ in range(2)]
    cv = [[torch.empty((H, T, d), dtype=torch.bfloat16, device="cuda") for _ in range(L)] for _ in range(2)]
    rc = kv.kvpool_decode_into(pool.t, shape, lb, le, 2, [c for a in ck for c in a], [c for a in cv for c in a])
    assert rc == kv.KVP_OK
    torch.cuda.synchronize()
    ok_, ov = O.pool_decode_into(img, lb, le, 1)
    for l in range(lb, le):
        np.testing.assert_array_equal(synth.bits16(ck[1][l]), ok_[0][l])
        assert_bf16_close(synth.bits16(cv[1][l]), ov[0][l], "V layer %d" % l)
    g = torch.Generator(device="cpu").manual_seed(11)
    q = torch.randn(N, 32, d, generator=g).to(torch.bfloat16)
    out, lse = _attend(pool.t, shape, L - 1, q.cuda(), 1.0 / math.sqrt(d))
    _check(img, shape, L - 1, synth.bits16(q), 1.0 / math.sqrt(d), out, lse)
