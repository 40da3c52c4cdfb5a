"""GPU parity of kvpool_attend -- attention of N agents' queries over one pool
layer straight from the compressed bytes (next row: QKVShare's deferred fused
attention over the quantized cache) -- against the fp64 oracle's attention
over the same pool image (exact dequantization).

Criteria: out within 1e-3 of the largest |value| of the KV head's tokens
(probabilities times sigma enter the value product as fp16, relative 2^-11;
centroids as fp16, relative 2.5e-4 at most); lse within 1e-4 (1 + |lse|)."""
import math

import numpy as np
import pytest
import torch

import agent_shared_compressed_gb300 as kv
from agent_shared_compressed_gb300 import build as kvbuild
from agent_shared_compressed_gb300 import synth
import oracle as O
from kvhelp import Guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    kvbuild.build()
    kv.load()


def _pool(ks_t, vs_t, shape):
    pool = torch.empty(kv.kvpool_pool_bytes(shape), dtype=torch.uint8, device="cuda")
    ws = torch.empty(kv.kvpool_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    assert kv.kvpool_encode(shape, ks_t, vs_t, pool, pool.numel(), ws, ws.numel()) == kv.KVP_OK
    assert kv.kvpool_status(pool) == kv.KVP_OK
    return pool


def _attend(pool, shape, layer, q_t, scale):
    na, nq, d = q_t.shape
    out = Guarded(na * nq * d * 4)
    lse = Guarded(na * nq * 4)
    wsb = kv.kvpool_attend_workspace_bytes(shape, na, nq)
    ws = Guarded(wsb, fill=0x7F)
    rc = kv.kvpool_attend(pool, shape, layer, na, nq, q_t, scale, out.t, lse.t, ws.t, wsb)
    assert rc == kv.KVP_OK, kv.kvp_strerror(rc)
    torch.cuda.synchronize()
    assert out.canary_ok() and lse.canary_ok() and ws.canary_ok()
    return (out.t.view(torch.float32).view(na, nq, d).cpu().numpy(),
            lse.t.view(torch.float32).view(na, nq).cpu().numpy())


def _check(pool_img, shape, layer, q_bits, scale, out, lse):
    L, H, d, T = shape
    ref, ref_lse = O.pool_attend(pool_img, layer, q_bits, scale)
    # per KV head: the largest |value| of its tokens bounds any output
    _, vref = O.pool_decode_into(pool_img, layer, layer + 1, 1)
    vmax = np.abs((vref[0][layer].astype(np.uint32) << 16).view(np.float32)).reshape(H, -1).max(1)
    na, nq, _ = q_bits.shape
    G = nq // H
    worst = 0.0
    for j in range(nq):
        tol = 1e-3 * vmax[j // G] + 1e-6
        err = np.abs(out[:, j] - ref[:, j]).max()
        assert err <= tol, "head %d: max error %g > %g" % (j, err, tol)
        worst = max(worst, err / tol)
    print("attend %s layer %d: worst out error / tolerance %.3f" % (tuple(shape), layer, worst))
    assert np.all(np.abs(lse - ref_lse) <= 1e-4 * (1 + np.abs(ref_lse)))


CASES = [  # (L, H, d, T, n_agents, n_q_heads)
    (2, 2, 64, 37, 3, 8),        # GQA 4, T < 64, ragged
    (1, 8, 128, 512, 15, 32),    # one Llama-3-8B layer, 15 agents x 32 query heads (60 rows per KV head)
    (2, 4, 128, 129, 20, 16),    # 80 rows per KV head: two query tiles; T = 2*64 + 1
    (1, 32, 64, 300, 3, 32),     # SmolLM2-like: no grouping (1 query head per KV head)
    (1, 1, 128, 1, 1, 1),        # one token
    (1, 2, 128, 4096, 2, 8),     # many sub-chunks per split
    (1, 4, 128, 1000, 4, 32),    # 32 rows per KV head: two 16-row tiles, four token slices
]


@pytest.mark.parametrize("case", CASES)
def test_attend_matches_oracle(case):
    L, H, d, T, na, nq = case
    shape = (L, H, d, T)
    ks_t, vs_t = synth.kv_layers(L, H, T, d, seed=T + na, device="cuda")
    pool = _pool(ks_t, vs_t, shape)
    img = pool.cpu().numpy()
    g = torch.Generator(device="cpu").manual_seed(7)
    q = torch.randn(na, nq, d, generator=g).to(torch.bfloat16)
    qb = synth.bits16(q)
    for layer in {0, L - 1}:
        out, lse = _attend(pool, shape, layer, q.cuda(), 1.0 / math.sqrt(d))
        _check(img, shape, layer, qb, 1.0 / math.sqrt(d), out, lse)


def test_attend_peaked_and_flat_softmax():
    """A large scale (nearly one-hot weights) and a zero query (uniform
    weights: the mean value, lse = log T)."""
    shape = (1, 2, 128, 200)
    L, H, d, T = shape
    ks_t, vs_t = synth.kv_layers(L, H, T, d, seed=5, device="cuda")
    pool = _pool(ks_t, vs_t, shape)
    img = pool.cpu().numpy()
    q = torch.zeros(2, 4, d, dtype=torch.bfloat16)
    q[1] = torch.randn(4, d)
    qb = synth.bits16(q)
    out, lse = _attend(pool, shape, 0, q.cuda(), 1.0)
    _check(img, shape, 0, qb, 1.0, out, lse)
    assert np.allclose(lse[0], math.log(T), atol=1e-5)
    out, lse = _attend(pool, shape, 0, q.cuda(), 8.0)
    _check(img, shape, 0, qb, 8.0, out, lse)


def test_attend_argument_errors():
    shape = (2, 4, 128, 64)
    ok = 0x10000
    wsb = kv.kvpool_attend_workspace_bytes(shape, 2, 8)
    assert kv.kvpool_attend_workspace_bytes(shape, 2, 6) == 0            # 6 query heads over 4 KV heads
    assert kv.kvpool_attend(ok, shape, 2, 2, 8, ok, 1.0, ok, ok, ok, wsb) == kv.KVP_ERR_ARG   # layer
    assert kv.kvpool_attend(ok, shape, 0, 2, 6, ok, 1.0, ok, ok, ok, wsb) == kv.KVP_ERR_ARG   # heads
    assert kv.kvpool_attend(ok, shape, 0, 2, 8, ok + 8, 1.0, ok, ok, ok, wsb) == kv.KVP_ERR_ALIGN
    assert kv.kvpool_attend(ok, shape, 0, 2, 8, ok, 1.0, ok, ok, ok, wsb - 1) == kv.KVP_ERR_SIZE


@pytest.mark.parametrize("name,n_q", [("llama3-8b-4k-15agents", 32), ("llama3-8b-32k-4agents", 32)])
def test_attend_full_size_layers(name, n_q):
    """The 4K/15-agent and 32K/4-agent pools (Llama-3-8B: 32 query heads over
    8 KV heads), first and last layer, against the oracle."""
    w = synth.WORKLOADS[name]
    L, H, d, T, N = w["L"], w["H"], w["d"], w["T"], w["N"]
    shape = (L, H, d, T)
    ks_t, vs_t = synth.kv_layers(L, H, T, d, seed=0, device="cuda")
    pool = _pool(ks_t, vs_t, shape)
    img = pool.cpu().numpy()
    g = torch.Generator(device="cpu").manual_seed(11)
    q = torch.randn(N, n_q, d, generator=g).to(torch.bfloat16)
    qb = synth.bits16(q)
    for layer in (0, L - 1):
        out, lse = _attend(pool, shape, layer, q.cuda(), 1.0 / math.sqrt(d))
        _check(img, shape, layer, qb, 1.0 / math.sqrt(d), out, lse)


def test_attend_wait_timeout_is_reported_and_context_survives():
    """The split kernel waits (bounded) for each sub-chunk's bulk copies.  With
    the next call limited to zero polls every block gives up on its first
    sub-chunk: it lets the copies it issued land, records the timeout in the
    pool's error word (kvpool_status: KVP_ERR_TIMEOUT) and returns.  The
    context stays usable and the next call, on a fresh pool, is correct.
    Four sub-chunks per block here, so each block drains a full ring."""
    shape = (1, 8, 128, 8192)
    L, H, d, T = shape
    ks_t, vs_t = synth.kv_layers(L, H, T, d, seed=41, device="cuda")
    pool = _pool(ks_t, vs_t, shape)
    g = torch.Generator(device="cpu").manual_seed(3)
    q = torch.randn(2, 32, d, generator=g).to(torch.bfloat16)
    na, nq = q.shape[0], q.shape[1]
    out = torch.empty(na, nq, d, dtype=torch.float32, device="cuda")
    lse = torch.empty(na, nq, dtype=torch.float32, device="cuda")
    wsb = kv.kvpool_attend_workspace_bytes(shape, na, nq)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    assert kv.kvp_test_limit_next_attend(0) == kv.KVP_OK
    assert kv.kvpool_attend(pool, shape, 0, na, nq, q.cuda(), 0.1, out, lse, ws, wsb) == kv.KVP_OK
    assert kv.kvpool_status(pool) == kv.KVP_ERR_TIMEOUT
    torch.cuda.synchronize()
    pool2 = _pool(ks_t, vs_t, shape)                   # the hook applies to one call only
    res, res_lse = _attend(pool2, shape, 0, q.cuda(), 0.1)
    assert kv.kvpool_status(pool2) == kv.KVP_OK
    _check(pool2.cpu().numpy(), shape, 0, synth.bits16(q), 0.1, res, res_lse)


def test_attend_calls_chained_without_synchronization():
    """Attention calls back to back on one stream, with no host
    synchronization in between: every layer of a pool, then the pool
    re-encoded from other caches in place and attended again.  The split
    kernel may be placed while the previous call's combine still runs (a
    programmatic dependent launch), so each call must still see the
    queries, the pool and the previous kernels' writes in stream order."""
    shape = (3, 8, 128, 700)
    L, H, d, T = shape
    ks_a, vs_a = synth.kv_layers(L, H, T, d, seed=51, device="cuda")
    ks_b, vs_b = synth.kv_layers(L, H, T, d, seed=52, device="cuda")
    pool = torch.empty(kv.kvpool_pool_bytes(shape), dtype=torch.uint8, device="cuda")
    pws = torch.empty(kv.kvpool_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cpu").manual_seed(9)
    q = torch.randn(3, 32, d, generator=g).to(torch.bfloat16)
    qd = q.cuda()
    na, nq = q.shape[0], q.shape[1]
    wsb = kv.kvpool_attend_workspace_bytes(shape, na, nq)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    outs, lses = [], []

    def attend_all():
        for layer in range(L):
            o = torch.empty(na, nq, d, dtype=torch.float32, device="cuda")
            s = torch.empty(na, nq, dtype=torch.float32, device="cuda")
            assert kv.kvpool_attend(pool, shape, layer, na, nq, qd, 0.09, o, s, ws, wsb) == kv.KVP_OK
            outs.append(o)
            lses.append(s)

    assert kv.kvpool_encode(shape, ks_a, vs_a, pool, pool.numel(), pws, pws.numel()) == kv.KVP_OK
    attend_all()
    img_a = pool.clone()
    assert kv.kvpool_encode(shape, ks_b, vs_b, pool, pool.numel(), pws, pws.numel()) == kv.KVP_OK
    attend_all()
    torch.cuda.synchronize()
    assert kv.kvpool_status(pool) == kv.KVP_OK
    qb = synth.bits16(q)
    for i, img in enumerate([img_a.cpu().numpy(), pool.cpu().numpy()]):
        for layer in range(L):
            k = i * L + layer
            _check(img, shape, layer, qb, 0.09, outs[k].cpu().numpy(), lses[k].cpu().numpy())
