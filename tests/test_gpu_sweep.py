"""A seeded sweep over random cache shapes: on each, every entry point of the
path runs once on the same synthetic cache and is compared with the fp64
oracle under the criteria of tests/kvhelp.py:
  * pool encode (per-tensor and q8_0 keys): the whole image;
  * fan-out decode into N agents: agent 0 within the bf16 bound of the
    oracle's decode of the GPU's own pool, every agent identical;
  * CacheCard pack: the whole image; unpack: within the bf16 bound of the
    oracle's unpack of the GPU's own card;
  * attention over the pool's last layer: out within 1e-3 of the largest
    |value|, lse within 1e-4 (1 + |lse|).
Shapes: L in 1..3, H in {1, 2, 3, 4, 8}, d in {64, 128}, T in 1..700,
N in 1..5 agents, 1, 2 or 4 query heads per KV head."""
import math

import numpy as np
import pytest
import torch

import agent_shared_compressed_gb300 as kv
from agent_shared_compressed_gb300 import build as kvbuild
from agent_shared_compressed_gb300 import synth
import oracle as O
from kvhelp import Guarded, assert_bf16_close, assert_pool_parity, bf16_dev_layers, guarded_caches
from test_gpu_card import assert_card_parity, gpu_pack, gpu_unpack
from test_gpu_q8 import assert_q8_pool, encode_q8

pytestmark = pytest.mark.gpu


def _shapes(n, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        L = int(rng.integers(1, 4))
        H = int(rng.choice([1, 2, 3, 4, 8]))
        d = int(rng.choice([64, 128]))
        T = int(rng.integers(1, 701))
        N = int(rng.integers(1, 6))
        G = int(rng.choice([1, 2, 4]))
        out.append((L, H, d, T, N, G))
    return out


SHAPES = _shapes(8)


@pytest.fixture(scope="module", autouse=True)
def built():
    kvbuild.build()
    kv.load()


@pytest.mark.parametrize("case", SHAPES, ids=["L%dH%dd%dT%dN%dG%d" % c for c in SHAPES])
def test_sweep_every_entry_point(case):
    L, H, d, T, N, G = case
    shape = (L, H, d, T)
    seed = (L * 131 + H * 17 + d + T * 7 + N) % 100003
    ks_t, vs_t = synth.kv_layers(L, H, T, d, seed=seed, device="cpu")
    ks, vs = [synth.bits16(k) for k in ks_t], [synth.bits16(v) for v in vs_t]
    kd, vd = bf16_dev_layers(ks), bf16_dev_layers(vs)
    st = torch.cuda.current_stream()

    # pool encode, per-tensor keys
    pool = Guarded(kv.kvpool_pool_bytes(shape), fill=0x5A)
    ws = Guarded(kv.kvpool_workspace_bytes(shape), fill=0x77)
    assert kv.kvpool_encode(shape, kd, vd, pool.t, pool.nbytes, ws.t, ws.nbytes, st) == kv.KVP_OK
    assert kv.kvpool_status(pool.t, st) == kv.KVP_OK
    assert pool.canary_ok() and ws.canary_ok()
    img = pool.host()
    ora, flags, u = O.pool_encode(ks, vs, want_u=True)
    assert flags == 0
    assert_pool_parity(img, ora, u, L, H, d, T)

    # fan-out decode into N agents
    ck, cv = guarded_caches(L, H, T, d, N), guarded_caches(L, H, T, d, N)
    rc = kv.kvpool_decode_into(pool.t, shape, 0, L, N, [c.t for a in ck for c in a], [c.t for a in cv for c in a], st)
    assert rc == kv.KVP_OK
    torch.cuda.synchronize()
    ok_, ov = O.pool_decode_into(img, 0, L, 1)
    for l in range(L):
        assert_bf16_close(synth.bits16(ck[0][l].bf16((H, T, d))), ok_[0][l], "K layer %d" % l)
        assert_bf16_close(synth.bits16(cv[0][l].bf16((H, T, d))), ov[0][l], "V layer %d" % l)
        for a in range(1, N):
            assert torch.equal(ck[a][l].t, ck[0][l].t) and torch.equal(cv[a][l].t, cv[0][l].t)
    assert all(c.canary_ok() for a in ck + cv for c in a)

    # pool encode, q8_0 keys
    pool8, status8 = encode_q8(kd, vd, shape)
    assert status8 == kv.KVP_OK
    ora8, flags8, u8 = O.pool_encode(ks, vs, want_u=True, k_mode=1)
    assert flags8 == 0
    assert_q8_pool(pool8.host(), ora8, u8, L, H, d, T)

    # CacheCard pack and unpack
    bits = synth.card_bits(T, seed=seed).numpy()
    card, cstatus = gpu_pack(kd, vd, bits, shape, model_id=seed, pos=T)
    assert cstatus == kv.KVP_OK
    cimg = card.host()
    ocard, cflags, r = O.card_pack(ks, vs, bits, model_id=seed, pos_offset=T, want_r=True)
    assert cflags == 0
    assert_card_parity(cimg, ocard, r, L, H, d, T, bits)
    _, uk, uv = gpu_unpack(card, L, H, T, d)
    rk, rv = O.card_unpack(cimg)
    for l in range(L):
        assert_bf16_close(uk[l], rk[l], "card K layer %d" % l)
        assert_bf16_close(uv[l], rv[l], "card V layer %d" % l)

    # attention over the last layer
    nq = H * G
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn(N, nq, d, generator=g).to(torch.bfloat16)
    out = torch.empty(N, nq, d, dtype=torch.float32, device="cuda")
    lse = torch.empty(N, nq, dtype=torch.float32, device="cuda")
    wsb = kv.kvpool_attend_workspace_bytes(shape, N, nq)
    wsa = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(d)
    assert kv.kvpool_attend(pool.t, shape, L - 1, N, nq, q.cuda(), scale, out, lse, wsa, wsb, st) == kv.KVP_OK
    assert kv.kvpool_status(pool.t, st) == kv.KVP_OK
    ref, ref_lse = O.pool_attend(img, L - 1, synth.bits16(q), scale)
    vmax = np.abs(((ov[0][L - 1].astype(np.uint32) << 16).view(np.float32))).reshape(H, -1).max(1)
    o = out.cpu().numpy()
    for j in range(nq):
        assert np.abs(o[:, j] - ref[:, j]).max() <= 1e-3 * vmax[j // G] + 1e-6, "attention head %d" % j
    assert np.all(np.abs(lse.cpu().numpy() - ref_lse) <= 1e-4 * (1 + np.abs(ref_lse)))
