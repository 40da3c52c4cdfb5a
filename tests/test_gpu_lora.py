"""GPU parity of kvpool_attend_lora -- pool attention for agents that differ by
a LoRA adapter on the value projection, with one shared low-rank cache
("LRAgent", BaseLRShared and Flash-LoRA-Attention: P V_base + (P V_lr) B) --
against the fp64 oracle, which forms every agent's values first and attends
over them.

Criteria: out within 1e-3 of the largest |value| any agent sees (base value
plus adapter term), lse within 1e-4 (1 + |lse|); a zero up-projection gives
kvpool_attend's output."""
import math

import numpy as np
import pytest
import torch

import agent_shared_compressed_gb300 as kv
from agent_shared_compressed_gb300 import build as kvbuild
from agent_shared_compressed_gb300 import synth
import oracle as O
from kvhelp import Guarded, f32_of_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    kvbuild.build()
    kv.load()


def make_pool(shape, seed, k_mode=0):
    L, H, d, T = shape
    ks_t, vs_t = synth.kv_layers(L, H, T, d, seed=seed, device="cuda")
    pool = torch.empty(kv.kvpool_pool_bytes_ex(shape, k_mode), dtype=torch.uint8, device="cuda")
    ws = torch.empty(kv.kvpool_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    assert kv.kvpool_encode_ex(shape, k_mode, ks_t, vs_t, pool, pool.numel(), ws, ws.numel()) == kv.KVP_OK
    assert kv.kvpool_status(pool) == kv.KVP_OK
    return pool


def attend_lora(pool, shape, layer, q, scale, rank, vlr, b):
    na, nq, d = q.shape
    out = Guarded(na * nq * d * 4)
    lse = Guarded(na * nq * 4)
    wsb = kv.kvpool_attend_lora_workspace_bytes(shape, na, nq, rank)
    ws = Guarded(wsb, fill=0x7F)
    rc = kv.kvpool_attend_lora(pool, shape, layer, na, nq, q, scale, rank, vlr, b, out.t, lse.t, ws.t, wsb)
    assert rc == kv.KVP_OK, kv.kvp_strerror(rc)
    torch.cuda.synchronize()
    assert out.canary_ok() and lse.canary_ok() and ws.canary_ok()
    assert kv.kvpool_status(pool) == kv.KVP_OK
    return (out.t.view(torch.float32).view(na, nq, d).cpu().numpy(),
            lse.t.view(torch.float32).view(na, nq).cpu().numpy())


def check(img, shape, layer, q, scale, vlr, b, out, lse):
    L, H, d, T = shape
    qb, vb, bb = synth.bits16(q), synth.bits16(vlr), synth.bits16(b)
    ref, ref_lse = O.pool_attend_lora(img, layer, qb, scale, vb, bb)
    _, vref = O.pool_decode_into(img, layer, layer + 1, 1)
    vbase = np.abs(f32_of_bf16(vref[0][layer])).max()
    adapter = np.abs(f32_of_bf16(vb).astype(np.float64) @ f32_of_bf16(bb).astype(np.float64)).max()
    tol = 1e-3 * (vbase + adapter) + 1e-6
    err = np.abs(out - ref).max()
    assert err <= tol, "max error %g > %g" % (err, tol)
    assert np.all(np.abs(lse - ref_lse) <= 1e-4 * (1 + np.abs(ref_lse)))
    print("lora attend %s: worst error / tolerance %.3f" % (tuple(shape), err / tol))


CASES = [  # (L, H, d, T, n_agents, n_q_heads, rank, key format)
    (2, 2, 64, 37, 3, 8, 16, 0),
    (1, 8, 128, 512, 15, 32, 32, 0),
    (1, 4, 128, 1000, 4, 32, 16, 0),
    (2, 4, 128, 129, 20, 16, 32, 0),
    (1, 8, 128, 300, 6, 32, 32, 1),
    (1, 32, 64, 300, 3, 32, 32, 0),
]


@pytest.mark.parametrize("case", CASES)
def test_attend_lora_matches_oracle(case):
    L, H, d, T, na, nq, rank, km = case
    shape = (L, H, d, T)
    pool = make_pool(shape, T + rank, km)
    img = pool.cpu().numpy()
    vlr, b = synth.lora_inputs(T, H, d, na, rank, seed=T, device="cuda")
    g = torch.Generator(device="cpu").manual_seed(3)
    q = torch.randn(na, nq, d, generator=g).to(torch.bfloat16).cuda()
    for layer in {0, L - 1}:
        out, lse = attend_lora(pool, shape, layer, q, 1.0 / math.sqrt(d), rank, vlr, b)
        check(img, shape, layer, q, 1.0 / math.sqrt(d), vlr, b, out, lse)


def test_attend_lora_zero_up_projection_is_plain_attention():
    shape = (1, 8, 128, 700)
    L, H, d, T = shape
    pool = make_pool(shape, 5)
    vlr, _ = synth.lora_inputs(T, H, d, 5, 32, seed=1, device="cuda")
    b = torch.zeros(5, 32, H * d, dtype=torch.bfloat16, device="cuda")
    q = torch.randn(5, 32, d, device="cuda").to(torch.bfloat16)
    out, lse = attend_lora(pool, shape, 0, q, 0.1, 32, vlr, b)
    wsb = kv.kvpool_attend_workspace_bytes(shape, 5, 32)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    o2 = torch.empty(5, 32, d, device="cuda")
    l2 = torch.empty(5, 32, device="cuda")
    assert kv.kvpool_attend(pool, shape, 0, 5, 32, q, 0.1, o2, l2, ws, wsb) == kv.KVP_OK
    torch.cuda.synchronize()
    np.testing.assert_allclose(out, o2.cpu().numpy(), rtol=0, atol=1e-6)
    np.testing.assert_allclose(lse, l2.cpu().numpy(), rtol=0, atol=1e-6)


def test_attend_lora_argument_errors():
    shape = (2, 4, 128, 64)
    ok = 0x10000
    wsb = kv.kvpool_attend_lora_workspace_bytes(shape, 2, 8, 16)
    assert wsb > kv.kvpool_attend_workspace_bytes(shape, 2, 8)
    assert kv.kvpool_attend_lora_workspace_bytes(shape, 2, 8, 8) == 0
    args = (ok, shape, 0, 2, 8, ok, 1.0)
    assert kv.kvpool_attend_lora(*args, 8, ok, ok, ok, ok, ok, wsb) == kv.KVP_ERR_ARG      # rank
    assert kv.kvpool_attend_lora(*args, 16, None, ok, ok, ok, ok, wsb) == kv.KVP_ERR_ARG   # no low-rank cache
    assert kv.kvpool_attend_lora(*args, 16, ok, None, ok, ok, ok, wsb) == kv.KVP_ERR_ARG   # no up-projection
    assert kv.kvpool_attend_lora(*args, 16, ok + 8, ok, ok, ok, ok, wsb) == kv.KVP_ERR_ALIGN
    assert kv.kvpool_attend_lora(*args, 16, ok, ok, ok, ok, ok, wsb - 1) == kv.KVP_ERR_SIZE


def test_attend_lora_full_size_layer():
    """The 4K-token, 15-agent Llama-3-8B pool at rank 32, last layer."""
    w = synth.WORKLOADS["llama3-8b-4k-15agents"]
    L, H, d, T, N = w["L"], w["H"], w["d"], w["T"], w["N"]
    shape = (L, H, d, T)
    pool = make_pool(shape, 0)
    img = pool.cpu().numpy()
    vlr, b = synth.lora_inputs(T, H, d, N, 32, seed=2, device="cuda")
    q = torch.randn(N, 32, d, generator=torch.Generator(device="cpu").manual_seed(4)).to(torch.bfloat16).cuda()
    out, lse = attend_lora(pool, shape, L - 1, q, 1.0 / math.sqrt(d), 32, vlr, b)
    check(img, shape, L - 1, q, 1.0 / math.sqrt(d), vlr, b, out, lse)
