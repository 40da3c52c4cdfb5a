"""GPU parity of the SharedKVPool path ("PolyKV" 2.A, 2.B) against the fp64
oracle: encode (K absmax / scale / int8 codes, V FWHT / sigma / 3-bit codes /
packing, header and layout) and fan-out decode into N agent caches, through
the C ABI, on seeded synthetic caches.  Criteria: tests/kvhelp.py."""
import numpy as np
import pytest
import torch

import agent_shared_compressed_gb300 as kv
from agent_shared_compressed_gb300 import build as kvbuild
from agent_shared_compressed_gb300 import synth
import oracle as O
from kvhelp import (Guarded, assert_bf16_close, assert_pool_parity, bf16_dev_layers, f32_of_bf16,
                    guarded_caches, pool_sections, unpack3_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    kvbuild.build()
    kv.load()


def cpu_inputs(L, H, T, d, seed):
    ks, vs = synth.kv_layers(L, H, T, d, seed=seed, device="cpu")
    return [synth.bits16(k) for k in ks], [synth.bits16(v) for v in vs]


def gpu_encode(ks_np, vs_np, shape, stream=None):
    kd, vd = bf16_dev_layers(ks_np), bf16_dev_layers(vs_np)
    pool = Guarded(kv.kvpool_pool_bytes(shape), fill=0x5A)
    ws = Guarded(kv.kvpool_workspace_bytes(shape), fill=0x77)
    st = stream or torch.cuda.current_stream()
    rc = kv.kvpool_encode(shape, kd, vd, pool.t, pool.nbytes, ws.t, ws.nbytes, st)
    assert rc == kv.KVP_OK, kv.kvp_strerror(rc)
    status = kv.kvpool_status(pool.t, st)
    assert pool.canary_ok() and ws.canary_ok()
    return pool, status, (kd, vd)


def gpu_decode(pool, shape, lb, le, n):
    L, H, d, T = shape
    ck = guarded_caches(L, H, T, d, n)
    cv = guarded_caches(L, H, T, d, n)
    kd = [ck[a][l].t if lb <= l < le else None for a in range(n) for l in range(L)]
    vd = [cv[a][l].t if lb <= l < le else None for a in range(n) for l in range(L)]
    rc = kv.kvpool_decode_into(pool.t, shape, lb, le, n, kd, vd, torch.cuda.current_stream())
    assert rc == kv.KVP_OK, kv.kvp_strerror(rc)
    torch.cuda.synchronize()
    for a in range(n):
        for l in range(L):
            assert ck[a][l].canary_ok() and cv[a][l].canary_ok()
            if not (lb <= l < le):                      # untouched outside the range
                assert bool((ck[a][l].t == 0xFF).all()) and bool((cv[a][l].t == 0xFF).all())
    return ck, cv


SMALL = [  # (L, H, d, T): several tiles and ragged tails, both head_dims
    (1, 8, 128, 512),       # one Llama-3-8B layer, 512 tokens
    (2, 32, 64, 1851),      # two SmolLM2-1.7B layers at 1851 tokens (odd T)
    (3, 5, 64, 37),
    (2, 3, 128, 7),
    (1, 1, 64, 1),
    (1, 1, 128, 1),
    (4, 2, 128, 129),
    (2, 1, 64, 15),         # fewer vectors than one warp step (16 at d=64)
]


@pytest.mark.parametrize("shape", SMALL)
def test_encode_matches_oracle(shape):
    L, H, d, T = shape
    ks, vs = cpu_inputs(L, H, T, d, seed=L * 1000 + T)
    pool, status, _ = gpu_encode(ks, vs, shape)
    assert status == kv.KVP_OK
    ora, flags, u = O.pool_encode(ks, vs, want_u=True)
    assert flags == 0
    assert_pool_parity(pool.host(), ora, u, L, H, d, T)


@pytest.mark.parametrize("shape,n", [((1, 8, 128, 512), 1), ((2, 32, 64, 1851), 3), ((3, 5, 64, 37), 4),
                                     ((2, 3, 128, 7), 2), ((1, 1, 64, 1), 5)])
def test_decode_fanout_matches_oracle(shape, n):
    L, H, d, T = shape
    ks, vs = cpu_inputs(L, H, T, d, seed=7 + T)
    pool, _, _ = gpu_encode(ks, vs, shape)
    img = pool.host()
    ck, cv = gpu_decode(pool, shape, 0, L, n)
    ok_, ov = O.pool_decode_into(img, 0, L, 1)       # the oracle decodes the GPU's own codes
    for l in range(L):
        k0, v0 = synth.bits16(ck[0][l].bf16((H, T, d))), synth.bits16(cv[0][l].bf16((H, T, d)))
        assert_bf16_close(k0, ok_[0][l], "K layer %d" % l)
        assert_bf16_close(v0, ov[0][l], "V layer %d" % l)
        for a in range(1, n):                          # every agent gets the same bytes
            assert torch.equal(ck[a][l].t, ck[0][l].t) and torch.equal(cv[a][l].t, cv[0][l].t)
        # reconstruction error of K is bounded by half a quantization step (plus bf16 rounding)
        s = float(pool_sections(img, L, H, d, T)["scales"][l])
        err = np.abs(f32_of_bf16(k0) - f32_of_bf16(ks[l]))
        assert np.all(err <= s / 2 + 2.0 ** -8 * np.abs(f32_of_bf16(ks[l])) + 1e-30)


def test_decode_layer_ranges_and_agent_split():
    shape = (5, 4, 128, 33)
    L, H, d, T = shape
    ks, vs = cpu_inputs(L, H, T, d, seed=3)
    pool, _, _ = gpu_encode(ks, vs, shape)
    ck_all, cv_all = gpu_decode(pool, shape, 0, L, 1)
    for lb, le, n in [(2, 3, 3), (1, 4, 2), (4, 5, 1)]:
        ck, cv = gpu_decode(pool, shape, lb, le, n)
        for a in range(n):
            for l in range(lb, le):
                assert torch.equal(ck[a][l].t, ck_all[0][l].t) and torch.equal(cv[a][l].t, cv_all[0][l].t)


def test_decode_many_destinations_split_into_launches():
    # 300 agents x 4 layers = 1200 destinations > 1024 per launch
    shape = (4, 1, 64, 16)
    L, H, d, T = shape
    ks, vs = cpu_inputs(L, H, T, d, seed=5)
    pool, _, _ = gpu_encode(ks, vs, shape)
    n = 300
    ck = [[torch.full((H, T, d), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(L)] for _ in range(n)]
    cv = [[torch.full((H, T, d), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(L)] for _ in range(n)]
    rc = kv.kvpool_decode_into(pool.t, shape, 0, L, n, [c for a in ck for c in a], [c for a in cv for c in a])
    assert rc == kv.KVP_OK
    ref_k, ref_v = gpu_decode(pool, shape, 0, L, 1)
    for a in range(n):
        for l in range(L):
            assert torch.equal(ck[a][l].view(torch.uint8).flatten(), ref_k[0][l].t)
            assert torch.equal(cv[a][l].view(torch.uint8).flatten(), ref_v[0][l].t)


def test_decode_rejects_mismatched_shape():
    shape = (2, 2, 64, 8)
    ks, vs = cpu_inputs(2, 2, 8, 64, seed=9)
    pool, status, _ = gpu_encode(ks, vs, shape)
    assert status == kv.KVP_OK
    other = (2, 2, 64, 9)                                  # same layout class, wrong T
    big = Guarded(kv.kvpool_pool_bytes(other))
    big.t[: pool.nbytes].copy_(pool.t)
    ck = guarded_caches(2, 2, 9, 64, 1)
    cv = guarded_caches(2, 2, 9, 64, 1)
    rc = kv.kvpool_decode_into(big.t, other, 0, 2, 1, [c.t for c in ck[0]], [c.t for c in cv[0]])
    assert rc == kv.KVP_OK
    assert kv.kvpool_status(big.t) == kv.KVP_ERR_HEADER
    for c in ck[0] + cv[0]:
        assert bool((c.t == 0xFF).all())                    # nothing written
    junk = Guarded(4096, fill=0)
    assert kv.kvpool_status(junk.t) == kv.KVP_ERR_HEADER


def test_encode_is_deterministic_and_overwrites_everything():
    shape = (2, 3, 64, 21)
    ks, vs = cpu_inputs(2, 3, 21, 64, seed=11)
    p1, _, _ = gpu_encode(ks, vs, shape)
    kd, vd = bf16_dev_layers(ks), bf16_dev_layers(vs)
    p2 = Guarded(p1.nbytes, fill=0xC3)
    ws = Guarded(kv.kvpool_workspace_bytes(shape), fill=0x00)
    assert kv.kvpool_encode(shape, kd, vd, p2.t, p2.nbytes, ws.t, ws.nbytes) == kv.KVP_OK
    torch.cuda.synchronize()
    assert torch.equal(p1.t, p2.t)


# --- degenerate inputs ------------------------------------------------------

def _bits(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("d", [128, 64])
def test_degenerate_layers_match_oracle(d):
    """Zero tensors (s = 0, codes 0 / 4, sigma 0), a tiny-magnitude layer (key
    scale below 2^-100, value norms below 2^-50), exact ties in k/s (s = 1,
    half-integer keys), one-hot and constant value vectors; both head_dims
    (at 64 each lane of the value encoder holds two vectors)."""
    L, H, T = 4, 2, 24
    rng = np.random.default_rng(0)
    ks, vs = [], []
    ks.append(np.zeros((H, T, d), np.uint16)); vs.append(np.zeros((H, T, d), np.uint16))
    ks.append(_bits(rng.normal(size=(H, T, d)) * 1e-34)); vs.append(_bits(rng.normal(size=(H, T, d)) * 1e-20))
    k = np.round(rng.uniform(-127, 127, size=(H, T, d)) * 2) / 2          # half-integers, |k| <= 127
    k[0, 0, 0] = 127.0
    ks.append(_bits(k))
    v = np.zeros((H, T, d))
    v[:, np.arange(T), np.arange(T) % d] = rng.choice([-3.0, 2.0], T)      # one-hot vectors
    v[1, 5:10, :] = 0.75                                                    # constant vectors
    vs.append(_bits(v))
    ks.append(_bits(rng.normal(size=(H, T, d)))); vs.append(_bits(rng.standard_t(5, size=(H, T, d))))
    ks, vs = ks[:L], vs[:L]
    shape = (L, H, d, T)
    pool, status, _ = gpu_encode(ks, vs, shape)
    assert status == kv.KVP_OK
    ora, flags, u = O.pool_encode(ks, vs, want_u=True)
    assert flags == 0
    assert_pool_parity(pool.host(), ora, u, L, H, d, T)
    sec = pool_sections(pool.host(), L, H, d, T)
    assert sec["scales"][0] == 0 and not sec["k"][0].any()
    assert np.all(unpack3_np(sec["vpacked"][0], d) == 4) and not sec["sigma"][0].any()
    assert sec["scales"][1] < 2.0 ** -100 and sec["scales"][2] == 1.0
    ck, cv = gpu_decode(pool, shape, 0, L, 2)
    ok_, ov = O.pool_decode_into(pool.host(), 0, L, 1)
    for l in range(L):
        assert_bf16_close(synth.bits16(ck[1][l].bf16((H, T, d))), ok_[0][l], "K layer %d" % l)
        assert_bf16_close(synth.bits16(cv[1][l].bf16((H, T, d))), ov[0][l], "V layer %d" % l)
    assert not ck[0][0].t.any() and not cv[0][0].t.any()


@pytest.mark.parametrize("d", [128, 64])
def test_mixed_magnitude_vectors_in_one_warp_step(d):
    """Zero, tiny (norm below 2^-50), ordinary and large value vectors next to
    one another, so one warp step of the value encoder holds all of them:
    the zero vectors code as 4, the tiny ones are rescaled, the others not."""
    L, H, T = 1, 2, 40
    rng = np.random.default_rng(3)
    scale = np.array([0.0, 1e-20, 1.0, 1e3, 1e-30, 7.0, 0.0, 1e-3])[np.arange(T) % 8]
    v = rng.normal(size=(H, T, d)) * scale[None, :, None]
    ks = [_bits(rng.normal(size=(H, T, d)))]
    vs = [_bits(v)]
    shape = (L, H, d, T)
    pool, status, _ = gpu_encode(ks, vs, shape)
    assert status == kv.KVP_OK
    ora, flags, u = O.pool_encode(ks, vs, want_u=True)
    assert flags == 0
    assert_pool_parity(pool.host(), ora, u, L, H, d, T)
    sec = pool_sections(pool.host(), L, H, d, T)
    codes = unpack3_np(sec["vpacked"][0], d).reshape(H, T, d)
    assert np.all(codes[:, scale == 0.0, :] == 4)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("where,value,code", [("k", np.nan, kv.KVP_ERR_NONFINITE), ("k", np.inf, kv.KVP_ERR_NONFINITE),
                                              ("v", np.nan, kv.KVP_ERR_NONFINITE), ("v", -np.inf, kv.KVP_ERR_NONFINITE),
                                              ("v", 1e6, kv.KVP_ERR_RANGE)])
def test_device_detected_errors(where, value, code, d):
    L, H, T = 2, 2, 16
    ks, vs = cpu_inputs(L, H, T, d, seed=1)
    arr = (ks if where == "k" else vs)[1].copy()
    if value == 1e6:
        arr[1, 3, :] = _bits(np.full(d, value))
    else:
        arr[1, 3, 7] = _bits(np.array([value]))[0]
    (ks if where == "k" else vs)[1] = arr
    _, status, _ = gpu_encode(ks, vs, (L, H, d, T))
    assert status == code
    _, flags, _ = O.pool_encode(ks, vs)
    assert flags == {kv.KVP_ERR_NONFINITE: O.FLAG_NONFINITE, kv.KVP_ERR_RANGE: O.FLAG_RANGE}[code]


@pytest.mark.parametrize("d", [64, 128])
def test_sigma_near_the_fp16_limit(d):
    """A constant value vector has sigma = |x|: 59,904 is an fp16 value just
    below the largest (no error, sigma stored exactly); 70,144 is above it (a
    range error).  Both sides agree with the oracle."""
    L, H, T = 1, 2, 16
    for x, code in ((6.0e4, kv.KVP_OK), (7.0e4, kv.KVP_ERR_RANGE)):
        ks, vs = cpu_inputs(L, H, T, d, seed=2)
        arr = vs[0].copy()
        arr[1, 5, :] = _bits(np.full(d, x))
        vs[0] = arr
        pool, status, _ = gpu_encode(ks, vs, (L, H, d, T))
        assert status == code
        ora, flags, _ = O.pool_encode(ks, vs)
        assert flags == (0 if code == kv.KVP_OK else O.FLAG_RANGE)
        if code == kv.KVP_OK:
            xv = float((np.uint32(_bits(np.array([x]))[0]) << np.uint32(16)).view(np.float32))
            sec = pool_sections(pool.host(), L, H, d, T)
            assert int(sec["sigma"][0][1, 5]) == O.f64_to_f16(xv)


# --- full-size workloads, sampled -------------------------------------------

@pytest.mark.parametrize("name", ["llama3-8b-4k-15agents", "llama3-8b-32k-4agents", "smollm2-1.7b-1851"])
def test_full_size_sampled(name):
    """The benchmark's workloads at full size, in the launch configuration the
    benchmark times (all layers in one encode, all layers x all agents in one
    decode); outputs compared with the oracle on sampled vectors / elements,
    agent copies compared in full."""
    w = synth.WORKLOADS[name]
    L, H, d, T, N = w["L"], w["H"], w["d"], w["T"], w["N"]
    shape = (L, H, d, T)
    ks_t, vs_t = synth.kv_layers(L, H, T, d, seed=0, device="cuda")
    pool = Guarded(kv.kvpool_pool_bytes(shape))
    ws = Guarded(kv.kvpool_workspace_bytes(shape))
    st = torch.cuda.current_stream()
    assert kv.kvpool_encode(shape, ks_t, vs_t, pool.t, pool.nbytes, ws.t, ws.nbytes, st) == kv.KVP_OK
    assert kv.kvpool_status(pool.t, st) == kv.KVP_OK
    assert pool.canary_ok()
    ck = [[torch.empty((H, T, d), dtype=torch.bfloat16, device="cuda") for _ in range(L)] for _ in range(N)]
    cv = [[torch.empty((H, T, d), dtype=torch.bfloat16, device="cuda") for _ in range(L)] for _ in range(N)]
    assert kv.kvpool_decode_into(pool.t, shape, 0, L, N, [c for a in ck for c in a], [c for a in cv for c in a],
                                 st) == kv.KVP_OK
    torch.cuda.synchronize()
    img = pool.host()
    sec = pool_sections(img, L, H, d, T)
    rng = np.random.default_rng(1)
    for l in rng.choice(L, min(L, 6), replace=False):
        kb = synth.bits16(ks_t[l])
        m, bad = O.k_absmax(kb)
        assert not bad
        s = O.k_scale(m)
        assert sec["scales"][l] == s
        flat = kb.ravel()
        idx = rng.choice(flat.size, 20000, replace=False)
        want = np.array([O.k_code(int(flat[i]), s) for i in idx])
        np.testing.assert_array_equal(sec["k"][l].ravel()[idx], want)
        vb = synth.bits16(vs_t[l]).reshape(H * T, d)
        codes_g = unpack3_np(sec["vpacked"][l], d)
        sig_g = sec["sigma"][l].ravel()
        kout = synth.bits16(ck[N - 1][l]).reshape(H * T, d)
        vout = synth.bits16(cv[N - 1][l]).reshape(H * T, d)
        for n in rng.choice(H * T, 300, replace=False):
            codes, sh, u, fl = O.v_encode_vec(vb[n])
            band = np.zeros(d, bool)
            for t in O.thresholds():
                band |= np.abs(u - t) < 1e-4
            assert np.all((codes_g[n] == codes) | band)
            assert abs(int(sig_g[n]) - int(sh)) <= 1
            assert_bf16_close(vout[n], O.v_decode_vec(codes_g[n], int(sig_g[n])), "V decode")
            kd_ = np.array([O.k_decode(int(q), s) for q in sec["k"][l].reshape(H * T, d)[n]], np.uint16)
            assert_bf16_close(kout[n], kd_, "K decode")
    for a in range(N - 1):
        for l in range(L):
            assert torch.equal(ck[a][l], ck[N - 1][l]) and torch.equal(cv[a][l], cv[N - 1][l])


def test_encode_wait_timeout_is_reported_and_context_survives():
    """The key-quantize work waits (bounded) for its layer's scale, released by
    another block.  With that release withheld for one layer, the wait runs out
    after a short limit, kvpool_status reports KVP_ERR_TIMEOUT, and the next
    encode on the same context is correct."""
    shape = (3, 4, 128, 64)
    L, H, d, T = shape
    ks, vs = cpu_inputs(L, H, T, d, seed=31)
    assert kv.kvp_test_fail_next_encode(1, 20000) == kv.KVP_OK   # ~2-3 ms per waiting slice
    pool, status, _ = gpu_encode(ks, vs, shape)
    assert status == kv.KVP_ERR_TIMEOUT
    pool2, status2, _ = gpu_encode(ks, vs, shape)                 # the hook applies to one call only
    assert status2 == kv.KVP_OK
    ora, flags, u = O.pool_encode(ks, vs, want_u=True)
    assert_pool_parity(pool2.host(), ora, u, L, H, d, T)
