"""Helpers for the GPU parity tests: canary-guarded device buffers, readers
of the pool / card byte images, and the parity criteria.

Parity criteria (GPU vs the fp64 oracle on the same inputs):
  * integer / byte outputs (K codes, layouts, headers, CacheCard codes and
    fp16 scale/zero points, copied 16-bit tokens): bit-exact, except
  * V codes where the oracle's rotated coordinate u lies within 1e-4 of a
    decision threshold, and CacheCard codes where the oracle's (x - z)/s lies
    within 1e-4 of a half-integer (the GPU decides these in fp32);
  * sigma (fp16): within 1 ulp;
  * decoded bf16: |gpu - oracle| <= 2^-7 |oracle| + 1e-3, decoding the GPU's
    own codes with both decoders so decode parity does not depend on encode
    parity.
"""
import numpy as np
import torch

import agent_shared_compressed_gb300 as kv
from agent_shared_compressed_gb300 import synth
import oracle as O

CANARY = 0xA5
CANARY_BYTES = 4096
V_BAND = 1e-4
CARD_BAND = 1e-4


def f32_of_bf16(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class Guarded:
    """A device byte buffer followed by a 4 KiB canary."""

    def __init__(self, nbytes, fill=None, device="cuda"):
        self.nbytes = int(nbytes)
        self.buf = torch.empty(self.nbytes + CANARY_BYTES, dtype=torch.uint8, device=device)
        if fill is not None:
            self.buf[: self.nbytes].fill_(fill)
        self.buf[self.nbytes:].fill_(CANARY)
        self.t = self.buf[: self.nbytes]

    def ptr(self):
        return self.t.data_ptr()

    def canary_ok(self):
        return bool((self.buf[self.nbytes:] == CANARY).all().item())

    def bf16(self, shape):
        return self.t.view(torch.bfloat16).view(*shape)

    def host(self):
        return self.t.cpu().numpy()


def bf16_dev_layers(np_layers):
    return [synth.from_bits16(a, "cuda") for a in np_layers]


def guarded_caches(L, H, T, d, n):
    """n * L guarded bf16 [H, T, d] caches (agent-major), pre-filled with NaN bits."""
    return [[Guarded(H * T * d * 2, fill=0xFF) for _ in range(L)] for _ in range(n)]


# --- pool image readers -----------------------------------------------------

def pool_sections(img, L, H, d, T):
    g = O.pool_geometry(L, H, d, T)
    nv = H * T
    out = {"geo": g, "scales": img[g["off_scales"]: g["off_scales"] + 4 * L].view(np.float32).copy()}
    ks, vs, ss = [], [], []
    for l in range(L):
        b = g["off_layers"] + l * g["layer_stride"]
        ks.append(img[b: b + nv * d].view(np.int8).reshape(H, T, d))
        vs.append(img[b + g["sec_v"]: b + g["sec_v"] + nv * 3 * d // 8].reshape(nv, 3 * d // 8))
        ss.append(img[b + g["sec_sigma"]: b + g["sec_sigma"] + 2 * nv].view(np.uint16).reshape(H, T))
    out["k"], out["vpacked"], out["sigma"] = ks, vs, ss
    return out


def unpack3_np(packed, d):
    p = packed.reshape(packed.shape[0], d // 8, 3).astype(np.uint32)
    w = p[..., 0] | (p[..., 1] << 8) | (p[..., 2] << 16)
    e = np.arange(8, dtype=np.uint32)
    return ((w[..., None] >> (3 * e)) & 7).reshape(packed.shape[0], d).astype(np.uint8)


def v_band_mask(u):
    """True where a V code may legitimately differ (u within 1e-4 of a threshold)."""
    t = O.thresholds()
    m = np.zeros(u.shape, bool)
    for tj in t:
        m |= np.abs(u - tj) < V_BAND
    return m


def assert_pool_parity(gpu_img, ora_img, u, L, H, d, T):
    g = O.pool_geometry(L, H, d, T)
    # header and the gap after the scales: bit-exact
    np.testing.assert_array_equal(gpu_img[:256], ora_img[:256])
    np.testing.assert_array_equal(gpu_img[g["off_scales"] + 4 * L: g["off_layers"]],
                                  ora_img[g["off_scales"] + 4 * L: g["off_layers"]])
    G, R = pool_sections(gpu_img, L, H, d, T), pool_sections(ora_img, L, H, d, T)
    np.testing.assert_array_equal(G["scales"].view(np.uint32), R["scales"].view(np.uint32))
    n_band = 0
    for l in range(L):
        np.testing.assert_array_equal(G["k"][l], R["k"][l], err_msg="K codes, layer %d" % l)
        cg, cr = unpack3_np(G["vpacked"][l], d), unpack3_np(R["vpacked"][l], d)
        band = v_band_mask(u[l].reshape(H * T, d))
        diff = (cg != cr) & ~band
        assert not diff.any(), "V codes differ outside the 1e-4 band at layer %d: %d" % (l, diff.sum())
        n_band += int(((cg != cr) & band).sum())
        ds = np.abs(G["sigma"][l].astype(np.int32) - R["sigma"][l].astype(np.int32))
        assert ds.max() <= 1, "sigma differs by more than 1 fp16 ulp at layer %d" % l
        # alignment gaps inside the layer: zero on both
        b = g["off_layers"] + l * g["layer_stride"]
        for lo, hi in ((H * T * d, g["sec_v"]), (g["sec_v"] + H * T * 3 * d // 8, g["sec_sigma"]),
                       (g["sec_sigma"] + 2 * H * T, g["layer_stride"])):
            assert not gpu_img[b + lo: b + hi].any()
    return n_band


def assert_bf16_close(gpu_bits, ora_bits, what=""):
    a, b = f32_of_bf16(gpu_bits), f32_of_bf16(ora_bits)
    tol = 2.0 ** -7 * np.abs(b) + 1e-3
    bad = ~(np.abs(a - b) <= tol)
    assert not bad.any(), "%s: %d values outside 2^-7|x|+1e-3 (worst %r vs %r)" % (
        what, bad.sum(), a[bad][:3], b[bad][:3])


# --- card image readers -----------------------------------------------------

def card_tokens(img, hdr_geo, L, H, d, T, bits):
    """Per bitwidth b: (token indices, records [L, n_b, rec_bytes]) gathered
    from a card image."""
    offs = img[hdr_geo["off_offsets"]: hdr_geo["off_offsets"] + 4 * T].view(np.uint32).astype(np.int64)
    out = {}
    for b in (2, 4, 8, 16):
        idx = np.nonzero(bits == b)[0]
        if idx.size == 0:
            continue
        rb = O.card_record_bytes(b, H, d)
        base = hdr_geo["off_layers"] + np.arange(L)[:, None] * hdr_geo["layer_stride"] + offs[idx][None, :]
        recs = img[base[..., None] + np.arange(rb)[None, None, :]]
        out[b] = (idx, recs)
    return out


def unpack_group_codes(codes_bytes, b, n_coords):
    """codes_bytes [..., n_coords*b/8] -> codes [..., n_coords] (LE bit strings)."""
    bitsarr = np.unpackbits(codes_bytes, axis=-1, bitorder="little")
    bitsarr = bitsarr.reshape(*codes_bytes.shape[:-1], n_coords, b)
    w = (1 << np.arange(b)).astype(np.uint32)
    return (bitsarr.astype(np.uint32) * w).sum(-1)


def split_record(recs, b, H, d):
    """recs [..., rec_bytes] -> (codes [..., 2, H*d], params [..., 2, H*d/32] u32) for b < 16."""
    cb = H * d * b // 8
    npar = H * (d // 32)
    codes = np.stack([unpack_group_codes(recs[..., kv * cb:(kv + 1) * cb], b, H * d) for kv in (0, 1)], -2)
    par = recs[..., 2 * cb: 2 * cb + 2 * npar * 4].copy().view(np.uint32).reshape(*recs.shape[:-1], 2, npar)
    return codes, par
