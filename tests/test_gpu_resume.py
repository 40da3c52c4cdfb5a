"""Checkpoint / resume of the two shareable artefacts.  A SharedKVPool
("PolyKV" 2.A) and a CacheCard ("QKVShare" Methodology 2) are self-describing
byte images (header plus offsets, no pointers), so saving one is a copy: the
pool and the card go device -> host -> file -> host -> device, into buffers at
other addresses, and decode, attention and unpack from the restored copies
give exactly the bytes they give from the originals.  Also: calls on several
streams at once give the bytes of a sequential run."""
import numpy as np
import pytest
import torch

import agent_shared_compressed_gb300 as kv
from agent_shared_compressed_gb300 import build as kvbuild
from agent_shared_compressed_gb300 import synth
from kvhelp import Guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    kvbuild.build()
    kv.load()


def _restore(img, tmp_path, name, pad):
    """img (numpy bytes) through a file into a device buffer `pad` bytes into a
    larger allocation (another address, still 256-byte aligned)."""
    f = tmp_path / name
    img.tofile(f)
    back = np.fromfile(f, dtype=np.uint8)
    assert np.array_equal(back, img)
    big = torch.empty(pad + back.size, dtype=torch.uint8, device="cuda")
    dev = big[pad:]
    dev.copy_(torch.from_numpy(back))
    assert dev.data_ptr() % 256 == 0
    return dev


def _decode(pool, shape, n):
    L, H, d, T = shape
    ck = [[torch.empty(H * T * d * 2, dtype=torch.uint8, device="cuda") for _ in range(L)] for _ in range(n)]
    cv = [[torch.empty(H * T * d * 2, dtype=torch.uint8, device="cuda") for _ in range(L)] for _ in range(n)]
    rc = kv.kvpool_decode_into(pool, shape, 0, L, n, [c for a in ck for c in a], [c for a in cv for c in a])
    assert rc == kv.KVP_OK
    torch.cuda.synchronize()
    return torch.stack([torch.stack(a) for a in ck]), torch.stack([torch.stack(a) for a in cv])


def _attend(pool, shape, q, layer):
    L, H, d, T = shape
    na, nq = q.shape[0], q.shape[1]
    out = torch.empty(na, nq, d, dtype=torch.float32, device="cuda")
    lse = torch.empty(na, nq, dtype=torch.float32, device="cuda")
    wsb = kv.kvpool_attend_workspace_bytes(shape, na, nq)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    assert kv.kvpool_attend(pool, shape, layer, na, nq, q, 0.125, out, lse, ws, wsb) == kv.KVP_OK
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("k_mode", [kv.KVP_K_PER_TENSOR, kv.KVP_K_Q8_0])
def test_pool_and_card_survive_a_file_round_trip(tmp_path, k_mode):
    shape = (3, 4, 128, 300)
    L, H, d, T = shape
    ks_t, vs_t = synth.kv_layers(L, H, T, d, seed=77, device="cuda")
    pool = torch.empty(kv.kvpool_pool_bytes_ex(shape, k_mode), dtype=torch.uint8, device="cuda")
    ws = torch.empty(kv.kvpool_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    assert kv.kvpool_encode_ex(shape, k_mode, ks_t, vs_t, pool, pool.numel(), ws, ws.numel()) == kv.KVP_OK
    assert kv.kvpool_status(pool) == kv.KVP_OK
    bits = synth.card_bits(T, seed=77).numpy()
    card = Guarded(kv.cachecard_bytes(shape, bits))
    bits_dev = torch.from_numpy(bits).cuda()
    assert kv.cachecard_pack(shape, 5, 1234, bits_dev, ks_t, vs_t, card.t, card.nbytes) == kv.KVP_OK
    assert kv.cachecard_status(card.t) == kv.KVP_OK

    pool2 = _restore(pool.cpu().numpy(), tmp_path, "pool.bin", 768)
    card2 = _restore(card.host(), tmp_path, "card.bin", 1280)
    assert kv.kvpool_status(pool2) == kv.KVP_OK and kv.cachecard_status(card2) == kv.KVP_OK

    k1, v1 = _decode(pool, shape, 2)
    k2, v2 = _decode(pool2, shape, 2)
    assert torch.equal(k1, k2) and torch.equal(v1, v2)

    q = torch.randn(2, 8, d, generator=torch.Generator(device="cpu").manual_seed(3)).to(torch.bfloat16).cuda()
    o1, l1 = _attend(pool, shape, q, L - 1)
    o2, l2 = _attend(pool2, shape, q, L - 1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)

    outs = []
    for c in (card.t, card2):
        hdr = kv.CardHeader()
        assert kv.cachecard_read_header(c, hdr) == kv.KVP_OK
        assert hdr.model_id == 5 and hdr.pos_offset == 1234 and hdr.seq_len == T
        uk = [torch.empty(H, T, d, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
        uv = [torch.empty(H, T, d, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
        assert kv.cachecard_unpack(c, hdr, uk, uv) == kv.KVP_OK
        torch.cuda.synchronize()
        outs.append((torch.stack(uk), torch.stack(uv)))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_concurrent_streams_match_sequential_results():
    """Decode (into two agents), attention and a CacheCard pack of the same
    source, issued on three streams with no ordering between them, give the
    bytes a sequential run gives: the calls share no hidden state (the pool
    is only read; each call has its own outputs and workspace)."""
    shape = (2, 4, 128, 700)
    L, H, d, T = shape
    ks_t, vs_t = synth.kv_layers(L, H, T, d, seed=91, device="cuda")
    pool = torch.empty(kv.kvpool_pool_bytes(shape), dtype=torch.uint8, device="cuda")
    ws = torch.empty(kv.kvpool_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    assert kv.kvpool_encode(shape, ks_t, vs_t, pool, pool.numel(), ws, ws.numel()) == kv.KVP_OK
    bits = synth.card_bits(T, seed=91).numpy()
    bits_dev = torch.from_numpy(bits).cuda()
    q = torch.randn(3, 16, d, generator=torch.Generator(device="cpu").manual_seed(9)).to(torch.bfloat16).cuda()
    torch.cuda.synchronize()

    def run(streams):
        ck = [torch.empty(H * T * d * 2, dtype=torch.uint8, device="cuda") for _ in range(2 * L)]
        cv = [torch.empty(H * T * d * 2, dtype=torch.uint8, device="cuda") for _ in range(2 * L)]
        out = torch.empty(3, 16, d, dtype=torch.float32, device="cuda")
        lse = torch.empty(3, 16, dtype=torch.float32, device="cuda")
        wsb = kv.kvpool_attend_workspace_bytes(shape, 3, 16)
        wsa = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        card = torch.empty(kv.cachecard_bytes(shape, bits), dtype=torch.uint8, device="cuda")
        s1, s2, s3 = streams
        assert kv.kvpool_decode_into(pool, shape, 0, L, 2, ck, cv, s1) == kv.KVP_OK
        assert kv.kvpool_attend(pool, shape, L - 1, 3, 16, q, 0.1, out, lse, wsa, wsb, s2) == kv.KVP_OK
        assert kv.cachecard_pack(shape, 1, 0, bits_dev, ks_t, vs_t, card, card.numel(), s3) == kv.KVP_OK
        torch.cuda.synchronize()
        return torch.cat(ck + cv), out, lse, card

    cur = torch.cuda.current_stream()
    seq = run((cur, cur, cur))
    side = [torch.cuda.Stream() for _ in range(3)]
    for s in side:
        s.wait_stream(cur)
    par = run(side)
    for a, b in zip(seq, par):
        assert torch.equal(a, b)
    assert kv.kvpool_status(pool) == kv.KVP_OK
