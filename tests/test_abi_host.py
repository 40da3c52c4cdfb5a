"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every function include/kvpool.h declares; host-computed sizes agree
with the oracle's byte formats; every error the host can detect is returned
before any work is enqueued (each call below fails validation, so nothing
reaches the device even on a GPU machine)."""
import ctypes as C

import numpy as np
import pytest

import agent_shared_compressed_gb300 as kv
from agent_shared_compressed_gb300 import build as kvbuild
import oracle as O


@pytest.fixture(scope="module", autouse=True)
def built():
    kvbuild.build()
    kv.load()


def test_exports_every_declared_function():
    names = kv.declared_functions()
    assert set(names) >= {"kvpool_pool_bytes", "kvpool_workspace_bytes", "kvpool_encode", "kvpool_decode_into",
                          "kvpool_status", "cachecard_bytes", "cachecard_pack", "cachecard_read_header",
                          "cachecard_unpack", "cachecard_unpack_at", "cachecard_status", "kvp_strerror",
                          "kvp_launch_count"}
    lib = C.CDLL(kv.binding.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


SHAPES = [(1, 8, 128, 512), (24, 32, 64, 1851), (32, 8, 128, 4096), (32, 8, 128, 32768),
          (3, 5, 64, 37), (1, 1, 64, 1), (2, 3, 128, 7), (512, 1, 64, 3)]


@pytest.mark.parametrize("shape", SHAPES)
def test_pool_bytes_match_oracle_format(shape):
    L, H, d, T = shape
    assert kv.kvpool_pool_bytes((L, H, d, T)) == O.pool_bytes(L, H, d, T)
    assert kv.kvpool_pool_bytes_ex((L, H, d, T), kv.KVP_K_PER_TENSOR) == O.pool_bytes(L, H, d, T)
    assert kv.kvpool_pool_bytes_ex((L, H, d, T), kv.KVP_K_Q8_0) == O.pool_bytes_mode(L, H, d, T, 1)
    assert kv.kvpool_pool_bytes_ex((L, H, d, T), 2) == 0
    assert kv.kvpool_workspace_bytes((L, H, d, T)) > 0


def test_pool_bytes_of_the_named_configurations():
    # per layer: K H*T*d + V H*T*3d/8 + sigma 2*H*T, each section 256-aligned
    assert kv.kvpool_pool_bytes((1, 8, 128, 512)) == 512 + 729088
    assert kv.kvpool_pool_bytes((32, 8, 128, 4096)) - 512 == 186646528
    # payload bytes independent of agents; achieved ratio 2.8764 at d=128
    assert abs(2 * 32 * 8 * 4096 * 128 * 2 / (kv.kvpool_pool_bytes((32, 8, 128, 4096)) - 512) - 2.8764) < 1e-4


@pytest.mark.parametrize("shape", [(3, 5, 64, 37), (32, 8, 128, 8192), (2, 1, 64, 1), (4, 3, 128, 100)])
def test_card_bytes_match_oracle_format(shape):
    L, H, d, T = shape
    rng = np.random.default_rng(T)
    bits = rng.choice(np.array([2, 4, 8, 16], np.uint8), T, p=[0.25, 0.4, 0.25, 0.1])
    assert kv.cachecard_bytes((L, H, d, T), bits) == O.card_bytes(L, H, d, T, bits)
    bad = bits.copy()
    bad[-1] = 6
    assert kv.cachecard_bytes((L, H, d, T), bad) == 0


@pytest.mark.parametrize("shape,code", [((0, 8, 128, 16), kv.KVP_ERR_ARG), ((1, 0, 128, 16), kv.KVP_ERR_ARG),
                                        ((1, 8, 96, 16), kv.KVP_ERR_UNSUPPORTED_D),
                                        ((1, 8, 128, 0), kv.KVP_ERR_ARG), ((513, 8, 128, 16), kv.KVP_ERR_SIZE)])
def test_invalid_shapes(shape, code):
    assert kv.kvpool_pool_bytes(shape) == 0
    assert kv.kvpool_workspace_bytes(shape) == 0
    assert kv.kvpool_encode(shape, [0x1000], [0x1000], 0x1000, 1 << 30, 0x1000, 1 << 20) == code
    assert kv.kvpool_decode_into(0x1000, shape, 0, 1, 1, [0x1000], [0x1000]) == code
    assert kv.cachecard_pack(shape, 0, 0, 0x1000, [0x1000], [0x1000], 0x1000, 1 << 30) == code


def test_encode_argument_errors():
    s = (2, 8, 128, 64)
    pb, wb = kv.kvpool_pool_bytes(s), kv.kvpool_workspace_bytes(s)
    ok = 0x10000
    assert kv.kvpool_encode(s, [ok, None], [ok, ok], ok, pb, ok, wb) == kv.KVP_ERR_ARG
    assert kv.kvpool_encode(s, [ok, ok], [ok, ok], None, pb, ok, wb) == kv.KVP_ERR_ARG
    assert kv.kvpool_encode(s, [ok, ok + 8], [ok, ok], ok, pb, ok, wb) == kv.KVP_ERR_ALIGN
    assert kv.kvpool_encode(s, [ok, ok], [ok, ok], ok + 16, pb, ok, wb) == kv.KVP_ERR_ALIGN
    assert kv.kvpool_encode(s, [ok, ok], [ok, ok], ok, pb - 1, ok, wb) == kv.KVP_ERR_SIZE
    assert kv.kvpool_encode(s, [ok, ok], [ok, ok], ok, pb, ok, wb - 1) == kv.KVP_ERR_SIZE


def test_decode_argument_errors():
    s = (3, 8, 128, 64)
    ok = 0x10000
    dst = [ok] * 6
    assert kv.kvpool_decode_into(ok, s, 0, 4, 2, dst, dst) == kv.KVP_ERR_ARG      # layer range
    assert kv.kvpool_decode_into(ok, s, 2, 2, 2, dst, dst) == kv.KVP_ERR_ARG      # empty range
    assert kv.kvpool_decode_into(ok, s, 0, 3, 0, dst, dst) == kv.KVP_ERR_ARG      # no agents
    assert kv.kvpool_decode_into(ok + 128, s, 0, 3, 2, dst, dst) == kv.KVP_ERR_ALIGN
    bad = list(dst)
    bad[4] = ok + 2                                                               # agent 1, layer 1
    assert kv.kvpool_decode_into(ok, s, 0, 3, 2, bad, dst) == kv.KVP_ERR_ALIGN
    bad[4] = None
    assert kv.kvpool_decode_into(ok, s, 0, 3, 2, dst, bad) == kv.KVP_ERR_ARG
    # layers outside the range are not read: a NULL there is fine up to validation
    # (range [1,2) with an unaligned pool still fails on the pool, before launch)
    assert kv.kvpool_decode_into(ok + 64, s, 1, 2, 2, [None, ok, None] * 2, [None, ok, None] * 2) == kv.KVP_ERR_ALIGN


def test_encode_ex_argument_errors():
    """Host-side checks of the key-format encode, all before any launch."""
    s = (2, 4, 128, 64)
    ok = 0x10000
    pb, wb = kv.kvpool_pool_bytes_ex(s, kv.KVP_K_Q8_0), kv.kvpool_workspace_bytes(s)
    assert pb > kv.kvpool_pool_bytes(s)
    assert kv.kvpool_encode_ex(s, 7, [ok] * 2, [ok] * 2, ok, pb, ok, wb) == kv.KVP_ERR_ARG
    assert kv.kvpool_encode_ex(s, -1, [ok] * 2, [ok] * 2, ok, pb, ok, wb) == kv.KVP_ERR_ARG
    # a per-tensor-sized buffer is too small for q8_0 keys
    assert kv.kvpool_encode_ex(s, kv.KVP_K_Q8_0, [ok] * 2, [ok] * 2, ok, kv.kvpool_pool_bytes(s), ok,
                               wb) == kv.KVP_ERR_SIZE
    assert kv.kvpool_encode_ex(s, kv.KVP_K_Q8_0, [ok] * 2, [ok] * 2, ok + 16, pb, ok, wb) == kv.KVP_ERR_ALIGN
    assert kv.kvpool_encode_ex(s, kv.KVP_K_Q8_0, [ok, None], [ok] * 2, ok, pb, ok, wb) == kv.KVP_ERR_ARG


def test_card_argument_errors():
    s = (2, 8, 128, 64)
    ok = 0x10000
    assert kv.cachecard_pack(s, 1, 2, None, [ok, ok], [ok, ok], ok, 1 << 24) == kv.KVP_ERR_ARG
    assert kv.cachecard_pack(s, 1, 2, ok, [ok, ok], [ok, ok], ok + 16, 1 << 24) == kv.KVP_ERR_ALIGN
    assert kv.cachecard_pack(s, 1, 2, ok, [ok, ok], [ok, ok], ok, 128) == kv.KVP_ERR_SIZE
    h = kv.CardHeader()
    h.magic = 0x12345678
    assert kv.cachecard_unpack(ok, h, [ok, ok], [ok, ok]) == kv.KVP_ERR_HEADER
    assert kv.cachecard_unpack(None, h, [ok], [ok]) == kv.KVP_ERR_ARG
    assert kv.kvpool_status(None) == kv.KVP_ERR_ARG
    assert kv.cachecard_status(None) == kv.KVP_ERR_ARG


def _consistent_header(L, H, d, T, bits):
    g = O.card_geometry(L, H, d, T, bits)
    h = kv.CardHeader()
    h.magic, h.version, h.seq_len, h.n_layers, h.n_kv_heads, h.head_dim = 0x4343564B, 1, T, L, H, d
    h.group_size, h.dtype, h.pos_offset = 32, 1, -5
    h.off_bits, h.off_offsets, h.off_layers = g["off_bits"], g["off_offsets"], g["off_layers"]
    h.layer_stride = g["layer_stride"]
    h.total_bytes = g["off_layers"] + L * g["layer_stride"]
    return h


def test_card_unpack_at_argument_errors():
    """Host-side checks of the re-aligning unpack, all before any launch."""
    L, H, d, T = 2, 8, 128, 64
    ok = 0x10000
    h = _consistent_header(L, H, d, T, np.full(T, 4, np.uint8))
    w = [1.0] * (d // 2)
    assert kv.cachecard_unpack_at(ok, h, 0, None, [ok] * L, [ok] * L) == kv.KVP_ERR_ARG
    assert kv.cachecard_unpack_at(ok, h, 0, w[:-1] + [float("nan")], [ok] * L, [ok] * L) == kv.KVP_ERR_ARG
    assert kv.cachecard_unpack_at(ok, h, 0, w[:-1] + [float("inf")], [ok] * L, [ok] * L) == kv.KVP_ERR_ARG
    assert kv.cachecard_unpack_at(ok, h, 2 ** 63 - 1, w, [ok] * L, [ok] * L) == kv.KVP_ERR_ARG  # shift overflows
    assert kv.cachecard_unpack_at(ok + 16, h, 0, w, [ok] * L, [ok] * L) == kv.KVP_ERR_ALIGN
    assert kv.cachecard_unpack_at(ok, h, 0, w, [ok + 2] * L, [ok] * L) == kv.KVP_ERR_ALIGN
    h.magic = 1
    assert kv.cachecard_unpack_at(ok, h, 0, w, [ok] * L, [ok] * L) == kv.KVP_ERR_HEADER


def test_strerror_and_counter():
    for code in range(-9, 1):
        assert kv.kvp_strerror(code) and kv.kvp_strerror(code) != "unknown status"
    assert kv.kvp_strerror(-100) == "unknown status"
    assert kv.kvp_launch_count() >= 0


def _attend_ws(H, d, T, na, nq, rank=0):
    """The attention workspace the split plan implies: the splits of each KV
    head (64-token sub-chunks) are as many as keep the grid of H x splits
    blocks within one wave of resident blocks, which a host without a GPU
    takes as 304 (two per SM on the GB300's 152 SMs); one partial row of
    d + rank floats and one (max, sum) pair per query row (padded to 64) per
    split."""
    nsub = (T + 63) // 64
    want = max(1, min(304 // H, nsub))
    per = (nsub + want - 1) // want
    nsplit = (nsub + per - 1) // per
    qhp = (na * (nq // H) + 63) // 64 * 64
    rows = H * nsplit * qhp
    a256 = lambda x: (x + 255) // 256 * 256
    return a256(a256(rows * (d + rank) * 4) + rows * 8), H * nsplit


@pytest.mark.parametrize("H,d,T,na,nq", [(8, 128, 4096, 15, 32), (8, 128, 32768, 4, 32), (32, 64, 1851, 3, 32),
                                          (1, 128, 1, 1, 1), (4, 128, 1000, 4, 32), (2, 64, 37, 3, 8)])
def test_attention_plan_stays_within_one_wave(H, d, T, na, nq):
    shape = (1, H, d, T)
    ws, blocks = _attend_ws(H, d, T, na, nq)
    assert blocks <= 304
    assert kv.kvpool_attend_workspace_bytes(shape, na, nq) == ws
    for rank in (16, 32):
        assert kv.kvpool_attend_lora_workspace_bytes(shape, na, nq, rank) == _attend_ws(H, d, T, na, nq, rank)[0]


def test_bandwidth_probe_argument_errors():
    ok = 0x10000
    assert kv.kvp_bandwidth_probe(7, ok, ok, 4096) == kv.KVP_ERR_ARG          # unknown mode
    assert kv.kvp_bandwidth_probe(kv.KVP_PROBE_STORE, None, None, 4096) == kv.KVP_ERR_ARG
    assert kv.kvp_bandwidth_probe(kv.KVP_PROBE_STORE, ok, None, 0) == kv.KVP_ERR_ARG
    assert kv.kvp_bandwidth_probe(kv.KVP_PROBE_STORE, ok + 16, None, 4096) == kv.KVP_ERR_ALIGN
    assert kv.kvp_bandwidth_probe(kv.KVP_PROBE_STORE, ok, None, 4100) == kv.KVP_ERR_SIZE
    assert kv.kvp_bandwidth_probe(kv.KVP_PROBE_BULK_STORE, ok, None, 4096 + 16) == kv.KVP_ERR_SIZE
    assert kv.kvp_bandwidth_probe(kv.KVP_PROBE_COPY, ok, None, 4096) == kv.KVP_ERR_ARG
    assert kv.kvp_bandwidth_probe(kv.KVP_PROBE_COPY, ok, ok + 16, 4096) == kv.KVP_ERR_ALIGN
    assert kv.kvp_bandwidth_probe(kv.KVP_PROBE_COPY, ok, ok, 4100) == kv.KVP_ERR_SIZE
