"""ctypes binding of include/kvpool.h -- argument marshalling only.

Every function has the C name and returns the C status (0 = KVP_OK,
negative = KVP_ERR_*); all computation happens in the CUDA library.
Arguments that the C API takes as device pointers accept a torch tensor
(its data_ptr()), a plain int address or None (NULL).  Per-layer pointer
lists accept Python sequences of the same.  `stream` accepts a
torch.cuda.Stream, a raw cudaStream_t int, or None (legacy default stream).

The library is loaded from this package's directory (built in-tree by
agent_shared_compressed_gb300.build); if it is missing, load() raises -- there
is no fallback.
"""
import ctypes as C
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvcodec.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "kvpool.h")

KVP_OK = 0
KVP_ERR_ARG = -1
KVP_ERR_UNSUPPORTED_D = -2
KVP_ERR_ALIGN = -3
KVP_ERR_SIZE = -4
KVP_ERR_CUDA = -5
KVP_ERR_NONFINITE = -6
KVP_ERR_RANGE = -7
KVP_ERR_BITS = -8
KVP_ERR_HEADER = -9
KVP_ERR_TIMEOUT = -10
KVP_MAX_LAYERS = 512
KVP_K_PER_TENSOR = 0
KVP_K_Q8_0 = 1
KVP_NOALLOC_SCRATCH_BYTES = 262144
KVP_PROBE_STORE = 0
KVP_PROBE_BULK_STORE = 1
KVP_PROBE_COPY = 2


class Shape(C.Structure):
    """kvp_shape: n_layers tensors of [n_kv_heads][n_tokens][head_dim]."""
    _fields_ = [("n_layers", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("n_tokens", C.c_int32)]

    def __repr__(self):
        return "Shape(L=%d, H=%d, d=%d, T=%d)" % (self.n_layers, self.n_kv_heads, self.head_dim, self.n_tokens)


class CardHeader(C.Structure):
    """kvp_card_header: the first 128 bytes of a CacheCard."""
    _fields_ = [("magic", C.c_uint32), ("version", C.c_uint32), ("seq_len", C.c_int32),
                ("n_layers", C.c_int32), ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("group_size", C.c_int32), ("dtype", C.c_int32), ("model_id", C.c_uint64),
                ("pos_offset", C.c_int64), ("off_bits", C.c_uint64), ("off_offsets", C.c_uint64),
                ("off_layers", C.c_uint64), ("layer_stride", C.c_uint64), ("total_bytes", C.c_uint64),
                ("error", C.c_uint32), ("reserved", C.c_uint32 * 9)]


assert C.sizeof(CardHeader) == 128

_vp = C.c_void_p
_SIGS = {
    "kvpool_pool_bytes": (C.c_size_t, [C.POINTER(Shape)]),
    "kvpool_workspace_bytes": (C.c_size_t, [C.POINTER(Shape)]),
    "kvpool_encode": (C.c_int, [C.POINTER(Shape), C.POINTER(_vp), C.POINTER(_vp), _vp, C.c_size_t,
                                _vp, C.c_size_t, _vp]),
    "kvpool_pool_bytes_ex": (C.c_size_t, [C.POINTER(Shape), C.c_int]),
    "kvpool_encode_ex": (C.c_int, [C.POINTER(Shape), C.c_int, C.POINTER(_vp), C.POINTER(_vp), _vp, C.c_size_t,
                                   _vp, C.c_size_t, _vp]),
    "kvpool_decode_into": (C.c_int, [_vp, C.POINTER(Shape), C.c_int, C.c_int, C.c_int,
                                     C.POINTER(_vp), C.POINTER(_vp), _vp]),
    "kvpool_status": (C.c_int, [_vp, _vp]),
    "kvpool_attend_workspace_bytes": (C.c_size_t, [C.POINTER(Shape), C.c_int, C.c_int]),
    "kvpool_attend": (C.c_int, [_vp, C.POINTER(Shape), C.c_int, C.c_int, C.c_int, _vp, C.c_float, _vp, _vp, _vp,
                                C.c_size_t, _vp]),
    "kvpool_attend_lora_workspace_bytes": (C.c_size_t, [C.POINTER(Shape), C.c_int, C.c_int, C.c_int]),
    "kvpool_attend_lora": (C.c_int, [_vp, C.POINTER(Shape), C.c_int, C.c_int, C.c_int, _vp, C.c_float, C.c_int, _vp,
                                     _vp, _vp, _vp, _vp, C.c_size_t, _vp]),
    "kvpool_encode_noalloc": (C.c_int, [C.POINTER(Shape), C.POINTER(_vp), C.POINTER(_vp), _vp, C.c_size_t, _vp]),
    "cachecard_bytes": (C.c_size_t, [C.POINTER(Shape), C.POINTER(C.c_uint8)]),
    "cachecard_pack": (C.c_int, [C.POINTER(Shape), C.c_uint64, C.c_int64, _vp, C.POINTER(_vp),
                                 C.POINTER(_vp), _vp, C.c_size_t, _vp]),
    "cachecard_read_header": (C.c_int, [_vp, C.POINTER(CardHeader), _vp]),
    "cachecard_unpack": (C.c_int, [_vp, C.POINTER(CardHeader), C.POINTER(_vp), C.POINTER(_vp), _vp]),
    "cachecard_unpack_at": (C.c_int, [_vp, C.POINTER(CardHeader), C.c_int64, C.POINTER(C.c_float), C.POINTER(_vp),
                                      C.POINTER(_vp), _vp]),
    "cachecard_status": (C.c_int, [_vp, _vp]),
    "kvp_strerror": (C.c_char_p, [C.c_int]),
    "kvp_launch_count": (C.c_uint64, []),
    "kvp_bandwidth_probe": (C.c_int, [C.c_int, _vp, _vp, C.c_size_t, _vp]),
    "kvp_test_fail_next_encode": (C.c_int, [C.c_int, C.c_uint32]),
    "kvp_test_limit_next_attend": (C.c_int, [C.c_uint32]),
    "kvp_test_limit_next_unpack": (C.c_int, [C.c_uint32]),
}

_lib = None


def load(path=None):
    """Load the CUDA codec library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError("CUDA codec library not built: %s (run agent_shared_compressed_gb300.build.build())" % p)
    lib = C.CDLL(p)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = lib
    return lib


def declared_functions(header=HEADER):
    """Names of the functions include/kvpool.h declares."""
    src = open(header).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\([^;{]*\)\s*;", src)))


# --- marshalling helpers ---------------------------------------------------

def _addr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError("expected a tensor, an int address or None, got %r" % type(x))


def _ptrs(seq):
    seq = list(seq)
    arr = (_vp * max(1, len(seq)))()
    for i, x in enumerate(seq):
        arr[i] = _addr(x)
    return arr


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _shape(s):
    if isinstance(s, Shape):
        return s
    L, H, d, T = s
    return Shape(L, H, d, T)


# --- C API -----------------------------------------------------------------

def kvpool_pool_bytes(shape):
    return int(load().kvpool_pool_bytes(C.byref(_shape(shape))))


def kvpool_workspace_bytes(shape):
    return int(load().kvpool_workspace_bytes(C.byref(_shape(shape))))


def kvpool_encode(shape, k_layers, v_layers, pool, pool_bytes, ws, ws_bytes, stream=None):
    return load().kvpool_encode(C.byref(_shape(shape)), _ptrs(k_layers), _ptrs(v_layers), _addr(pool),
                                int(pool_bytes), _addr(ws), int(ws_bytes), _stream(stream))


def kvpool_pool_bytes_ex(shape, k_mode):
    return int(load().kvpool_pool_bytes_ex(C.byref(_shape(shape)), int(k_mode)))


def kvpool_encode_ex(shape, k_mode, k_layers, v_layers, pool, pool_bytes, ws, ws_bytes, stream=None):
    """k_mode: KVP_K_PER_TENSOR or KVP_K_Q8_0."""
    return load().kvpool_encode_ex(C.byref(_shape(shape)), int(k_mode), _ptrs(k_layers), _ptrs(v_layers),
                                   _addr(pool), int(pool_bytes), _addr(ws), int(ws_bytes), _stream(stream))


def kvpool_encode_noalloc(shape, k_layers, v_layers, pool, pool_bytes, stream=None):
    """kvpool_encode with the library's own scratch array as workspace (for
    callers that cannot allocate device memory)."""
    return load().kvpool_encode_noalloc(C.byref(_shape(shape)), _ptrs(k_layers), _ptrs(v_layers), _addr(pool),
                                        int(pool_bytes), _stream(stream))


def kvpool_decode_into(pool, shape, layer_begin, layer_end, n_agents, k_dst, v_dst, stream=None):
    """k_dst/v_dst: n_agents * n_layers pointers, agent-major (a*L + l)."""
    return load().kvpool_decode_into(_addr(pool), C.byref(_shape(shape)), int(layer_begin), int(layer_end),
                                     int(n_agents), _ptrs(k_dst), _ptrs(v_dst), _stream(stream))


def kvpool_attend_workspace_bytes(shape, n_agents, n_q_heads):
    return int(load().kvpool_attend_workspace_bytes(C.byref(_shape(shape)), int(n_agents), int(n_q_heads)))


def kvpool_attend(pool, shape, layer, n_agents, n_q_heads, q, scale, out, lse, ws, ws_bytes, stream=None):
    return load().kvpool_attend(_addr(pool), C.byref(_shape(shape)), int(layer), int(n_agents), int(n_q_heads),
                                _addr(q), C.c_float(scale), _addr(out), _addr(lse), _addr(ws), int(ws_bytes),
                                _stream(stream))


def kvpool_attend_lora_workspace_bytes(shape, n_agents, n_q_heads, rank):
    return int(load().kvpool_attend_lora_workspace_bytes(C.byref(_shape(shape)), int(n_agents), int(n_q_heads),
                                                         int(rank)))


def kvpool_attend_lora(pool, shape, layer, n_agents, n_q_heads, q, scale, rank, v_lr, lora_b, out, lse, ws,
                       ws_bytes, stream=None):
    return load().kvpool_attend_lora(_addr(pool), C.byref(_shape(shape)), int(layer), int(n_agents),
                                     int(n_q_heads), _addr(q), C.c_float(scale), int(rank), _addr(v_lr),
                                     _addr(lora_b), _addr(out), _addr(lse), _addr(ws), int(ws_bytes),
                                     _stream(stream))


def kvpool_status(pool, stream=None):
    return load().kvpool_status(_addr(pool), _stream(stream))


def cachecard_bytes(shape, bits_host):
    b = bytes(bytearray(int(x) for x in bits_host))
    arr = (C.c_uint8 * max(1, len(b))).from_buffer_copy(b if b else b"\0")
    return int(load().cachecard_bytes(C.byref(_shape(shape)), arr))


def cachecard_pack(shape, model_id, pos_offset, bits_dev, k_layers, v_layers, card, card_bytes, stream=None):
    return load().cachecard_pack(C.byref(_shape(shape)), C.c_uint64(model_id), C.c_int64(pos_offset),
                                 _addr(bits_dev), _ptrs(k_layers), _ptrs(v_layers), _addr(card),
                                 int(card_bytes), _stream(stream))


def cachecard_read_header(card, out, stream=None):
    """Fills `out` (a CardHeader); returns the status."""
    return load().cachecard_read_header(_addr(card), C.byref(out), _stream(stream))


def cachecard_unpack(card, hdr, k_dst, v_dst, stream=None):
    return load().cachecard_unpack(_addr(card), C.byref(hdr), _ptrs(k_dst), _ptrs(v_dst), _stream(stream))


def cachecard_unpack_at(card, hdr, pos_dst, inv_freq, k_dst, v_dst, stream=None):
    """inv_freq: head_dim/2 host floats (any sequence; None passes NULL)."""
    if inv_freq is None:
        w = None
    else:
        vals = [float(x) for x in inv_freq]
        w = (C.c_float * max(1, len(vals)))(*vals)
    return load().cachecard_unpack_at(_addr(card), C.byref(hdr), C.c_int64(int(pos_dst)), w, _ptrs(k_dst),
                                      _ptrs(v_dst), _stream(stream))


def cachecard_status(card, stream=None):
    return load().cachecard_status(_addr(card), _stream(stream))


def kvp_strerror(status):
    return load().kvp_strerror(int(status)).decode()


def kvp_launch_count():
    return int(load().kvp_launch_count())


def kvp_bandwidth_probe(mode, dst, src, nbytes, stream=None):
    return load().kvp_bandwidth_probe(int(mode), _addr(dst), _addr(src), int(nbytes), _stream(stream))


def kvp_test_fail_next_encode(layer, spin_iters):
    return load().kvp_test_fail_next_encode(int(layer), int(spin_iters))


def kvp_test_limit_next_attend(polls):
    return load().kvp_test_limit_next_attend(int(polls))


def kvp_test_limit_next_unpack(polls):
    return load().kvp_test_limit_next_unpack(int(polls))


class KVPError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__("%s%s (%d)" % (what + ": " if what else "", kvp_strerror(status), status))


def check(status, what=""):
    """Raise KVPError for a non-zero status."""
    if status != KVP_OK:
        raise KVPError(status, what)
    return status
