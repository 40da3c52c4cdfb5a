"""fp64 CPU oracle for the shared multi-agent KV codec -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it: the C source ``kv_oracle.c`` restates the method from
the pages ("PolyKV: A Shared Asymmetrically-Compressed KV Cache Pool for
Multi-Agent LLM Inference", 2.A and 2.B; "QKVShare: Quantized KV-Cache Handoff
for Multi-Agent On-Device LLMs", Methodology 1-3) in plain double precision.

This module is argument marshalling only: numpy arrays in, numpy arrays out.
bf16 and fp16 tensors travel as their raw ``uint16`` bit patterns.

Every oracle function is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_pins.py``; none is marked "parity unpinned".
"""
import ctypes as C
import numpy as np

from . import build as _build

_lib = None

FLAG_NONFINITE = 1
FLAG_RANGE = 2
FLAG_BITS = 4

_u16p = C.POINTER(C.c_uint16)
_u8p = C.POINTER(C.c_uint8)
_dp = C.POINTER(C.c_double)
_u64p = C.POINTER(C.c_uint64)


def lib():
    """Load (building first if needed) the oracle shared object.  The
    KV_ORACLE_LIB environment variable points at another build of the same
    source (used by the mutation test to load deliberately broken copies)."""
    global _lib
    if _lib is not None:
        return _lib
    import os
    path = os.environ.get("KV_ORACLE_LIB") or _build.build()
    L = C.CDLL(path)
    sig = {
        "orc_set_threads": (None, [C.c_int]),
        "orc_get_threads": (C.c_int, []),
        "orc_bf16_to_f64": (C.c_double, [C.c_uint16]),
        "orc_f64_to_bf16": (C.c_uint16, [C.c_double]),
        "orc_f16_to_f64": (C.c_double, [C.c_uint16]),
        "orc_f64_to_f16": (C.c_uint16, [C.c_double]),
        "orc_fwht": (None, [_dp, C.c_int]),
        "orc_lloyd_max_gauss": (C.c_int, [C.c_int, C.c_int, C.c_double, _dp, _dp]),
        "orc_centroids": (None, [_dp]),
        "orc_thresholds": (None, [_dp]),
        "orc_v_code": (C.c_int, [C.c_double]),
        "orc_k_absmax": (C.c_double, [_u16p, C.c_size_t, C.POINTER(C.c_int)]),
        "orc_k_scale": (C.c_float, [C.c_double]),
        "orc_k_code": (C.c_int, [C.c_uint16, C.c_float]),
        "orc_k_decode": (C.c_uint16, [C.c_int, C.c_float]),
        "orc_k_block_scale": (C.c_uint16, [_u16p, C.POINTER(C.c_int), C.POINTER(C.c_int)]),
        "orc_k_block_code": (C.c_int, [C.c_uint16, C.c_uint16]),
        "orc_k_block_decode": (C.c_uint16, [C.c_int, C.c_uint16]),
        "orc_v_encode_vec": (C.c_uint32, [_u16p, C.c_int, _u8p, _u16p, _dp]),
        "orc_pack3": (None, [_u8p, C.c_int, _u8p]),
        "orc_unpack3": (None, [_u8p, C.c_int, _u8p]),
        "orc_v_decode_vec": (None, [_u8p, C.c_uint16, C.c_int, _u16p]),
        "orc_pool_bytes": (C.c_size_t, [C.c_int] * 4),
        "orc_pool_geometry": (None, [C.c_int] * 4 + [_u64p]),
        "orc_pool_encode": (C.c_uint32, [C.c_int] * 4 + [C.POINTER(_u16p), C.POINTER(_u16p), _u8p, _dp]),
        "orc_pool_encode_mode": (C.c_uint32, [C.c_int] * 5 + [C.POINTER(_u16p), C.POINTER(_u16p), _u8p, _dp]),
        "orc_pool_bytes_mode": (C.c_size_t, [C.c_int] * 5),
        "orc_pool_geometry_q8": (None, [C.c_int] * 4 + [_u64p]),
        "orc_pool_decode_into": (C.c_int, [_u8p, C.c_int, C.c_int, C.c_int, C.POINTER(_u16p), C.POINTER(_u16p)]),
        "orc_card_record_bytes": (C.c_uint64, [C.c_int, C.c_int, C.c_int]),
        "orc_card_bytes": (C.c_size_t, [C.c_int] * 4 + [_u8p]),
        "orc_card_geometry": (None, [C.c_int] * 4 + [_u8p, _u64p]),
        "orc_group_quant": (C.c_uint32, [_dp, C.c_int, _u8p, _u16p, _u16p, _dp]),
        "orc_card_pack": (C.c_uint32, [C.c_int] * 4 + [C.c_uint64, C.c_int64, _u8p,
                                                      C.POINTER(_u16p), C.POINTER(_u16p), _u8p, _dp]),
        "orc_card_unpack": (C.c_int, [_u8p, C.POINTER(_u16p), C.POINTER(_u16p)]),
        "orc_pool_attend_lora": (C.c_int, [_u8p, C.c_int, C.c_int, C.c_int, _u16p, C.c_double, C.c_int, _u16p, _u16p,
                                          _dp, _dp]),
        "orc_card_unpack_at": (C.c_int, [_u8p, C.c_int64, C.POINTER(C.c_float), C.POINTER(_u16p),
                                         C.POINTER(_u16p)]),
        "orc_pool_attend": (C.c_int, [_u8p, C.c_int, C.c_int, C.c_int, _u16p, C.c_double, _dp, _dp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _p(a, t):
    return a.ctypes.data_as(t)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def set_threads(n):
    lib().orc_set_threads(int(n))


def get_threads():
    return int(lib().orc_get_threads())


# --- scalar formats ---------------------------------------------------------

def bf16_to_f64(bits):
    return lib().orc_bf16_to_f64(int(bits))


def f64_to_bf16(x):
    return int(lib().orc_f64_to_bf16(float(x)))


def f16_to_f64(bits):
    return lib().orc_f16_to_f64(int(bits))


def f64_to_f16(x):
    return int(lib().orc_f64_to_f16(float(x)))


# --- building blocks --------------------------------------------------------

def fwht(x):
    """Unnormalised Sylvester-order Walsh-Hadamard transform of a 1-D array."""
    y = _c(x, np.float64).copy()
    lib().orc_fwht(_p(y, _dp), int(y.size))
    return y


def lloyd_max_gauss(levels=8, max_iter=100000, tol=1e-14):
    c = np.zeros(levels, np.float64)
    mse = C.c_double()
    it = lib().orc_lloyd_max_gauss(levels, max_iter, tol, _p(c, _dp), C.byref(mse))
    return c, mse.value, it


def centroids():
    c = np.zeros(8, np.float64)
    lib().orc_centroids(_p(c, _dp))
    return c


def thresholds():
    t = np.zeros(7, np.float64)
    lib().orc_thresholds(_p(t, _dp))
    return t


def v_code(u):
    return int(lib().orc_v_code(float(u)))


def k_absmax(k_bits):
    k = _c(k_bits, np.uint16).ravel()
    bad = C.c_int(0)
    m = lib().orc_k_absmax(_p(k, _u16p), k.size, C.byref(bad))
    return m, bool(bad.value)


def k_scale(m):
    return np.float32(lib().orc_k_scale(float(m)))


def k_code(k_bits, s):
    return int(lib().orc_k_code(int(k_bits), float(s)))


def k_decode(q, s):
    return int(lib().orc_k_decode(int(q), float(s)))


def k_block_scale(k32_bits):
    """q8_0 block: (fp16 scale bits, nonfinite, range) of 32 bf16 keys."""
    k = _c(k32_bits, np.uint16)
    assert k.size == 32
    bad, rng = C.c_int(0), C.c_int(0)
    sb = lib().orc_k_block_scale(_p(k, _u16p), C.byref(bad), C.byref(rng))
    return int(sb), bool(bad.value), bool(rng.value)


def k_block_code(k_bits, s_bits):
    return int(lib().orc_k_block_code(int(k_bits), int(s_bits)))


def k_block_decode(q, s_bits):
    return int(lib().orc_k_block_decode(int(q), int(s_bits)))


def v_encode_vec(v_bits):
    v = _c(v_bits, np.uint16).ravel()
    d = v.size
    codes = np.zeros(d, np.uint8)
    sh = np.zeros(1, np.uint16)
    u = np.zeros(d, np.float64)
    flags = lib().orc_v_encode_vec(_p(v, _u16p), d, _p(codes, _u8p), _p(sh, _u16p), _p(u, _dp))
    return codes, int(sh[0]), u, int(flags)


def pack3(codes):
    c = _c(codes, np.uint8).ravel()
    out = np.zeros(c.size * 3 // 8, np.uint8)
    lib().orc_pack3(_p(c, _u8p), c.size, _p(out, _u8p))
    return out


def unpack3(packed, d):
    p = _c(packed, np.uint8).ravel()
    out = np.zeros(d, np.uint8)
    lib().orc_unpack3(_p(p, _u8p), d, _p(out, _u8p))
    return out


def v_decode_vec(codes, sigma_bits):
    c = _c(codes, np.uint8).ravel()
    out = np.zeros(c.size, np.uint16)
    lib().orc_v_decode_vec(_p(c, _u8p), int(sigma_bits), c.size, _p(out, _u16p))
    return out


# --- SharedKVPool -----------------------------------------------------------

def pool_bytes(L, H, d, T):
    return int(lib().orc_pool_bytes(L, H, d, T))


def pool_geometry(L, H, d, T):
    g = np.zeros(6, np.uint64)
    lib().orc_pool_geometry(L, H, d, T, _p(g, _u64p))
    keys = ("off_scales", "off_layers", "layer_stride", "sec_v", "sec_sigma", "total")
    return {k: int(v) for k, v in zip(keys, g)}


def _ptr_table(arrays, t):
    arr = (t * len(arrays))()
    for i, a in enumerate(arrays):
        arr[i] = _p(a, t)
    return arr


def pool_encode(k_layers, v_layers, want_u=False, k_mode=0):
    """k_layers/v_layers: lists of uint16 arrays shaped [H, T, d] (bf16 bits).
    k_mode: 0 one key scale per layer tensor, 1 q8_0 key blocks.

    Returns (pool image uint8, error flags, u or None) where u is the fp64
    rotated coordinate behind every V code, shaped [L, H, T, d]."""
    k_layers = [_c(k, np.uint16) for k in k_layers]
    v_layers = [_c(v, np.uint16) for v in v_layers]
    L = len(k_layers)
    H, T, d = k_layers[0].shape
    pool = np.zeros(pool_bytes_mode(L, H, d, T, k_mode), np.uint8)
    u = np.zeros((L, H, T, d), np.float64) if want_u else None
    if k_mode == 0:
        flags = lib().orc_pool_encode(L, H, d, T, _ptr_table(k_layers, _u16p), _ptr_table(v_layers, _u16p),
                                      _p(pool, _u8p), _p(u, _dp) if want_u else None)
    else:
        flags = lib().orc_pool_encode_mode(L, H, d, T, k_mode, _ptr_table(k_layers, _u16p),
                                           _ptr_table(v_layers, _u16p), _p(pool, _u8p),
                                           _p(u, _dp) if want_u else None)
    return pool, int(flags), u


def pool_bytes_mode(L, H, d, T, k_mode):
    return int(lib().orc_pool_bytes_mode(L, H, d, T, int(k_mode)))


def pool_geometry_q8(L, H, d, T):
    """(off_kscales, total bytes) of a q8_0-key pool."""
    g = np.zeros(2, np.uint64)
    lib().orc_pool_geometry_q8(L, H, d, T, _p(g, _u64p))
    return int(g[0]), int(g[1])


def pool_decode_into(pool, layer_begin, layer_end, n_agents):
    """Decode layers [layer_begin, layer_end) into n_agents caches.

    Returns (k, v): lists over agents of lists over all L layers; layers
    outside the range are None."""
    pool = _c(pool, np.uint8)
    hdr = pool[:32].view(np.int32)
    L, H, d, T = int(hdr[2]), int(hdr[3]), int(hdr[4]), int(hdr[5])
    k = [[None] * L for _ in range(n_agents)]
    v = [[None] * L for _ in range(n_agents)]
    kt = (_u16p * (n_agents * L))()
    vt = (_u16p * (n_agents * L))()
    for a in range(n_agents):
        for l in range(layer_begin, layer_end):
            k[a][l] = np.zeros((H, T, d), np.uint16)
            v[a][l] = np.zeros((H, T, d), np.uint16)
            kt[a * L + l] = _p(k[a][l], _u16p)
            vt[a * L + l] = _p(v[a][l], _u16p)
    rc = lib().orc_pool_decode_into(_p(pool, _u8p), layer_begin, layer_end, n_agents, kt, vt)
    if rc != 0:
        raise ValueError("oracle: not a version-1 pool")
    return k, v


# --- CacheCard --------------------------------------------------------------

def card_record_bytes(b, H, d):
    return int(lib().orc_card_record_bytes(b, H, d))


def card_bytes(L, H, d, T, bits):
    b = _c(bits, np.uint8)
    return int(lib().orc_card_bytes(L, H, d, T, _p(b, _u8p)))


def card_geometry(L, H, d, T, bits):
    b = _c(bits, np.uint8)
    g = np.zeros(5, np.uint64)
    lib().orc_card_geometry(L, H, d, T, _p(b, _u8p), _p(g, _u64p))
    keys = ("off_bits", "off_offsets", "off_layers", "layer_stride", "total")
    return {k: int(v) for k, v in zip(keys, g)}


def group_quant(x, b):
    x = _c(x, np.float64)
    assert x.size == 32
    q = np.zeros(32, np.uint8)
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    r = np.zeros(32, np.float64)
    flags = lib().orc_group_quant(_p(x, _dp), int(b), _p(q, _u8p), _p(s, _u16p), _p(z, _u16p), _p(r, _dp))
    return q, int(s[0]), int(z[0]), r, int(flags)


def card_pack(k_layers, v_layers, bits, model_id=0, pos_offset=0, want_r=False):
    """Returns (card image uint8, error flags, r or None); r = (x - z_h)/s_h
    for every element, shaped [L, T, 2, H, d]."""
    k_layers = [_c(k, np.uint16) for k in k_layers]
    v_layers = [_c(v, np.uint16) for v in v_layers]
    bits = _c(bits, np.uint8)
    L = len(k_layers)
    H, T, d = k_layers[0].shape
    n = card_bytes(L, H, d, T, bits)
    card = np.zeros(max(n, 128), np.uint8)
    r = np.zeros((L, T, 2, H, d), np.float64) if want_r else None
    flags = lib().orc_card_pack(L, H, d, T, C.c_uint64(model_id), C.c_int64(pos_offset), _p(bits, _u8p),
                                _ptr_table(k_layers, _u16p), _ptr_table(v_layers, _u16p),
                                _p(card, _u8p), _p(r, _dp) if want_r else None)
    return card, int(flags), r


def card_unpack(card):
    card = _c(card, np.uint8)
    hdr = card[:32].view(np.int32)
    T, L, H, d = int(hdr[2]), int(hdr[3]), int(hdr[4]), int(hdr[5])
    k = [np.zeros((H, T, d), np.uint16) for _ in range(L)]
    v = [np.zeros((H, T, d), np.uint16) for _ in range(L)]
    rc = lib().orc_card_unpack(_p(card, _u8p), _ptr_table(k, _u16p), _ptr_table(v, _u16p))
    if rc != 0:
        raise ValueError("oracle: not a version-1 card")
    return k, v


def card_unpack_at(card, pos_dst, inv_freq):
    """Unpack with K re-aligned from the card's position offset to pos_dst
    (rotary pairs (i, i + d/2), frequencies inv_freq[d/2] in radians per
    position)."""
    card = _c(card, np.uint8)
    hdr = card[:32].view(np.int32)
    T, L, H, d = int(hdr[2]), int(hdr[3]), int(hdr[4]), int(hdr[5])
    w = _c(inv_freq, np.float32)
    assert w.size == d // 2
    k = [np.zeros((H, T, d), np.uint16) for _ in range(L)]
    v = [np.zeros((H, T, d), np.uint16) for _ in range(L)]
    rc = lib().orc_card_unpack_at(_p(card, _u8p), C.c_int64(pos_dst), _p(w, C.POINTER(C.c_float)),
                                  _ptr_table(k, _u16p), _ptr_table(v, _u16p))
    if rc != 0:
        raise ValueError("oracle: not a version-1 card")
    return k, v


# --- attention over the pool -------------------------------------------------

def pool_attend(pool, layer, q_bits, scale):
    """q_bits: uint16 [n_agents, n_q_heads, d] (bf16).  Returns (out fp64
    [n_agents, n_q_heads, d], lse fp64 [n_agents, n_q_heads])."""
    pool = _c(pool, np.uint8)
    q = _c(q_bits, np.uint16)
    na, nq, d = q.shape
    out = np.zeros((na, nq, d), np.float64)
    lse = np.zeros((na, nq), np.float64)
    rc = lib().orc_pool_attend(_p(pool, _u8p), int(layer), na, nq, _p(q, _u16p), float(scale),
                               _p(out, _dp), _p(lse, _dp))
    if rc != 0:
        raise ValueError("oracle: bad pool header, layer or head count")
    return out, lse


def pool_attend_lora(pool, layer, q_bits, scale, vlr_bits, lora_b_bits):
    """Attention of agents' queries over one pool layer with each agent's
    values v_base + vlr @ B_a.  q_bits: bf16 [n_agents][n_q_heads][d];
    vlr_bits: bf16 [T][rank]; lora_b_bits: bf16 [n_agents][rank][H*d].
    Returns (out [n_agents][n_q_heads][d] fp64, lse [n_agents][n_q_heads])."""
    pool = _c(pool, np.uint8)
    q = _c(q_bits, np.uint16)
    vlr = _c(vlr_bits, np.uint16)
    b = _c(lora_b_bits, np.uint16)
    na, nq, d = q.shape
    rank = vlr.shape[1]
    assert b.shape[0] == na and b.shape[1] == rank
    out = np.zeros((na, nq, d), np.float64)
    lse = np.zeros((na, nq), np.float64)
    rc = lib().orc_pool_attend_lora(_p(pool, _u8p), int(layer), na, nq, _p(q, _u16p), float(scale), int(rank),
                                    _p(vlr, _u16p), _p(b, _u16p), _p(out, _dp), _p(lse, _dp))
    if rc != 0:
        raise ValueError("oracle: bad pool header or head count")
    return out, lse
