// kvpool_encode.cu -- SharedKVPool encoder ("PolyKV" 2.B asymmetric
// compression): int8 keys with one symmetric scale per layer tensor; values
// rotated by a Walsh-Hadamard transform, normalised by sigma = ||v||/sqrt(d)
// (fp16), quantized to the 8-level Lloyd-Max codebook and packed 8 codes to 3
// bytes.
//
// One persistent kernel, encode_pool, works through an ordered queue of
// items.  For every layer l (queue order in item_of):
//   1. P key slices "absmax": max|k| over 128 KB of K_l, folded into the
//      layer's maximum with atomicMax.  The block that finishes the layer's
//      last slice computes the scale s = m/127, writes it to the pool and the
//      key quantizer's parameters to the workspace, and releases ready[l].
//   2. the layer's value batches (4 warp steps of 1024 value coordinates per
//      warp, each step copied into shared memory with cp.async while the
//      previous one is encoded; the rotation runs on the tensor cores),
//      interleaved with P key slices "quantize": each waits (bounded) for
//      ready[l], then writes the int8 codes = the integer nearest to the
//      exact k/s.  The key slice is re-read soon after its first read, from
//      L2 (first read marked evict-last, second evict-first).
// Items are taken in queue order by running blocks, so every item a wait
// depends on was taken earlier by a block that does not wait: no deadlock,
// whatever the number of resident blocks.  The last block to finish writes
// the pool header with the OR of every error bit.  The workspace's control
// block is zeroed on the stream before the kernel.
#include <cfloat>

#include "kvp_vec.cuh"

namespace kvp {

constexpr int ENC_THREADS = 256;
constexpr int ENC_WARPS = ENC_THREADS / 32;
constexpr uint64_t SLICE_CHUNKS = 8192;      // 16-byte chunks (128 KB of keys) per slice, at most
constexpr float RNE_MAGIC = 12582912.0f;     // 1.5 * 2^23
constexpr uint32_t SPIN_LIMIT = 1u << 24;    // ~1.7 s of 100 ns sleeps
constexpr int VSTEPS = 4;                    // value warp steps per warp per item

enum : int { ITEM_ABSMAX = 0, ITEM_KEYS = 1, ITEM_VALUES = 2 };

// Start of the workspace; zeroed before every encode.
struct EncodeCtl {
    uint32_t next_item;                    // work queue head
    uint32_t flags;                        // OR of every block's error bits
    uint32_t blocks_done;                  // last-block ticket
    uint32_t pad;
    uint32_t slices_done[KVP_MAX_LAYERS];  // absmax slices finished, per layer
    uint32_t ready[KVP_MAX_LAYERS];        // 1 once the layer's key parameters are written
    uint32_t kmax[KVP_MAX_LAYERS];         // max of the layer's sign-cleared bf16 key patterns
};

struct EncodeArgs {
    const uint4 *k[KVP_MAX_LAYERS];
    const uint4 *v[KVP_MAX_LAYERS];
    uint8_t *pool;
    EncodeCtl *ctl;
    float4 *kparams;     // [L]: s_eff, 1/s_eff, prescale1, prescale2
    PoolGeom geo;
    uint64_t chunks;            // 16-byte chunks per layer of K (H*T*d/8)
    uint64_t chunks_per_slice;  // per absmax / quantize slice
    uint64_t nvec;              // vectors per layer (H*T)
    uint64_t steps_per_layer;   // value warp steps per layer
    uint32_t vitems;            // value batches per layer
    uint32_t vhead;             // value batches of a layer queued before its first quantize slice
    uint32_t lag;               // layer l's value/quantize items follow layer l+lag's absmax items
    uint32_t seg0, seg1;        // queue positions where the middle / last stretch of rounds begin
    uint32_t total_items;
    uint32_t spin_limit;
    int L, H, T, d, P;
    int fail_layer;             // failure-path testing: this layer's flag is never released
    uint32_t kmode;             // KVP_K_PER_TENSOR or KVP_K_Q8_0
};

struct WsLayout {
    uint64_t ctl, kparams, total;
};

static inline int slices_per_layer(uint64_t chunks) {
    const uint64_t p = (chunks + SLICE_CHUNKS - 1) / SLICE_CHUNKS;
    return int(p < 1 ? 1 : p);
}

static inline WsLayout ws_layout(int L) {
    WsLayout w;
    w.ctl = 0;
    w.kparams = align256(sizeof(EncodeCtl));
    w.total = align16(w.kparams + 16ull * uint64_t(L));
    return w;
}

// Item t of the queue.  The queue is a sequence of rounds r = 0 .. L+lag-1;
// round r holds layer r's P absmax slices (if r < L), then the mixed items of
// layer r - lag (if that layer exists): its value batches with its P quantize
// slices spread evenly among them after a head of vhead value batches.  The
// lag (0-2 layers, chosen so that the keys of the layers in between still fit
// in L2) and the head put enough items between a layer's absmax slices and
// its quantize slices that the latter rarely wait.
__device__ __forceinline__ void mixed_item(const EncodeArgs &a, uint32_t o, int &kind, uint32_t &id) {
    if (o < a.vhead) {
        kind = ITEM_VALUES;
        id = o;
        return;
    }
    const uint64_t k = o - a.vhead;
    const uint64_t n = uint64_t(a.P) + a.vitems - a.vhead;
    const uint64_t qb = (k * uint64_t(a.P)) / n, qa = ((k + 1) * uint64_t(a.P)) / n;
    if (qa > qb) {
        kind = ITEM_KEYS;
        id = uint32_t(qb);
    } else {
        kind = ITEM_VALUES;
        id = uint32_t(a.vhead + k - qb);
    }
}

__device__ __forceinline__ void item_of(const EncodeArgs &a, uint32_t t, int &kind, int &layer, uint32_t &id) {
    const uint32_t P = uint32_t(a.P), M = P + a.vitems;
    if (t < a.seg0) {  // rounds 0 .. lag-1: absmax only
        layer = int(t / P);
        kind = ITEM_ABSMAX;
        id = t % P;
        return;
    }
    if (t < a.seg1) {  // rounds lag .. L-1: absmax of layer r, mixed of layer r - lag
        const uint32_t u = t - a.seg0;
        const uint32_t r = a.lag + u / (P + M), o = u % (P + M);
        if (o < P) {
            layer = int(r);
            kind = ITEM_ABSMAX;
            id = o;
        } else {
            layer = int(r - a.lag);
            mixed_item(a, o - P, kind, id);
        }
        return;
    }
    const uint32_t u = t - a.seg1;  // rounds L .. L+lag-1: mixed only
    layer = int(uint32_t(a.L) - a.lag + u / M);
    mixed_item(a, u % M, kind, id);
}

// ---------------------------------------------------------------------------
// Keys, pass 1: max|k| of one slice, folded into the layer's maximum, on the
// bf16 bit patterns with the sign cleared (for finite values their order is
// the order of the magnitudes; Inf/NaN patterns sort above every finite one,
// so they flag themselves).
// ---------------------------------------------------------------------------
__device__ void absmax_slice(const EncodeArgs &a, int l, uint32_t p, uint64_t pol, uint32_t *red) {
    const uint64_t c0 = uint64_t(p) * a.chunks_per_slice;
    const uint64_t c1 = min(c0 + a.chunks_per_slice, a.chunks);
    const uint4 *src = a.k[l];
    // per-halfword unsigned max of the bf16 patterns with the sign cleared
    // (Inf / NaN patterns sort above every finite value)
    uint32_t m2 = 0;
    uint64_t c = c0 + threadIdx.x;
    for (; c + 7 * ENC_THREADS < c1; c += 8 * ENC_THREADS) {
        uint4 w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) w[u] = ld_v4_policy(src + c + u * ENC_THREADS, pol);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            m2 = __vmaxu2(m2, __vmaxu2(w[u].x & 0x7FFF7FFFu, w[u].y & 0x7FFF7FFFu));
            m2 = __vmaxu2(m2, __vmaxu2(w[u].z & 0x7FFF7FFFu, w[u].w & 0x7FFF7FFFu));
        }
    }
    for (; c < c1; c += ENC_THREADS) {
        const uint4 w = ld_v4_policy(src + c, pol);
        m2 = __vmaxu2(m2, __vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu));
        m2 = __vmaxu2(m2, __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu));
    }
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t r = red[0];
#pragma unroll
        for (int i = 1; i < ENC_WARPS; ++i) r = max(r, red[i]);
        atomicMax(&a.ctl->kmax[l], r);
    }
    __syncthreads();
}

// Layer l's absmax slices are all done: its scale, quantizer parameters and
// alignment gaps; then release ready[l].  Whole block.
// Zero a layer's alignment gaps so the pool image is deterministic (block-wide).
__device__ void zero_layer_gaps(const EncodeArgs &a, int l) {
    uint8_t *lay = a.pool + a.geo.off_layers + uint64_t(l) * a.geo.layer_stride;
    const uint64_t gaps[3][2] = {{a.nvec * uint64_t(a.d), a.geo.sec_v},
                                 {a.geo.sec_v + a.nvec * uint64_t(3 * a.d / 8), a.geo.sec_sigma},
                                 {a.geo.sec_sigma + 2 * a.nvec, a.geo.layer_stride}};
    for (int gi = 0; gi < 3; ++gi)
        for (uint64_t i = gaps[gi][0] + threadIdx.x; i < gaps[gi][1]; i += ENC_THREADS) lay[i] = 0;
}

__device__ void finalize_layer(const EncodeArgs &a, int l) {
    if (threadIdx.x == 0) {
        __threadfence();  // the other blocks' maxima (folded in before their counter increments)
        const uint32_t r = *reinterpret_cast<volatile uint32_t *>(&a.ctl->kmax[l]);
        const bool finite = r < 0x7F80u;
        if (!finite) atomicOr(&a.ctl->flags, FLAG_NONFINITE);
        const float mk = __uint_as_float(r << 16);  // max|k|, exact
        // s = m/127, IEEE division: the correctly rounded fp32 quotient.
        const float s = finite ? mk / 127.0f : 0.0f;
        float4 kp = make_float4(0.f, 0.f, 1.f, 1.f);
        if (s > 0.0f) {
            if (s >= 0x1p-100f) {
                kp = make_float4(s, 1.0f / s, 1.0f, 1.0f);
            } else {
                // Tiny scale: quantize k*2^p against s*2^p with s*2^p in [1,2)
                // (both scalings exact), so 1/s cannot overflow and the exact
                // tie test cannot underflow.
                int e;
                frexpf(s, &e);
                const int p = 1 - e;
                const int p1 = p > 120 ? 120 : p;
                const float f1 = ldexpf(1.0f, p1), f2 = ldexpf(1.0f, p - p1);
                const float se = (s * f1) * f2;
                kp = make_float4(se, 1.0f / se, f1, f2);
            }
        }
        a.kparams[l] = kp;
        reinterpret_cast<float *>(a.pool + a.geo.off_scales)[l] = s;
    }
    zero_layer_gaps(a, l);
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (l != a.fail_layer) st_release_u32(&a.ctl->ready[l], 1u);
    }
}

// ---------------------------------------------------------------------------
// Keys, pass 2: int8 codes ("PolyKV" 2.B.1).  q = the integer nearest to the
// real k/s, ties to even.  Fast path: t = fma(k, 1/s, 1.5*2^23) rounds k/s'
// (k/s within 1.6e-5) to an integer held in t's low mantissa bits, whose low
// byte is the two's-complement code.  Only when that estimate is within 1e-4
// of a half-integer is the decision taken exactly: the sign of
// k - (q0 +- 1/2) s is exact under one fma rounding.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int k_code_exact_int(float k, float s, float q0) {
    const float hi = fmaf(-(q0 + 0.5f), s, k);
    const float lo = fmaf(-(q0 - 0.5f), s, k);
    int q = int(q0);
    if (hi > 0.0f)
        q += 1;
    else if (hi == 0.0f)
        q += (q & 1);
    else if (lo < 0.0f)
        q -= 1;
    else if (lo == 0.0f)
        q -= (q & 1);
    return q;
}

__device__ __forceinline__ uint32_t k_code_exact(float k, float s, float q0) {
    return uint32_t(k_code_exact_int(k, s, q0)) & 0xFFu;
}

template <bool PRESCALE>
__device__ __forceinline__ uint2 k_quant8(uint4 w, float4 kp) {
    // pairs of keys (low and high bf16 half of each word), on f32x2 lanes
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    float2 k[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) k[i] = make_float2(bf16_lo(ws[i]), bf16_hi(ws[i]));
    if (PRESCALE) {
#pragma unroll
        for (int i = 0; i < 4; ++i) k[i] = __fmul2_rn(__fmul2_rn(k[i], make_float2(kp.z, kp.z)), make_float2(kp.w, kp.w));
    }
    const float2 r = make_float2(kp.y, kp.y), mg = make_float2(RNE_MAGIC, RNE_MAGIC);
    float2 tf[4];
    bool near = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        tf[i] = __ffma2_rn(k[i], r, mg);
        const float2 nq0 = __ffma2_rn(tf[i], make_float2(-1.0f, -1.0f), mg);  // -q0, exact
        const float2 e = __ffma2_rn(k[i], r, nq0);
        near |= fabsf(e.x) > 0.4999f;
        near |= fabsf(e.y) > 0.4999f;
    }
    uint32_t t[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        t[2 * i] = __float_as_uint(tf[i].x);
        t[2 * i + 1] = __float_as_uint(tf[i].y);
    }
    if (near) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            t[2 * i] = k_code_exact(k[i].x, kp.x, tf[i].x - RNE_MAGIC);
            t[2 * i + 1] = k_code_exact(k[i].y, kp.x, tf[i].y - RNE_MAGIC);
        }
    }
    uint2 r8;
    r8.x = __byte_perm(__byte_perm(t[0], t[1], 0x0040), __byte_perm(t[2], t[3], 0x0040), 0x5410);
    r8.y = __byte_perm(__byte_perm(t[4], t[5], 0x0040), __byte_perm(t[6], t[7], 0x0040), 0x5410);
    return r8;
}

__device__ void quant_slice(const EncodeArgs &a, int l, uint32_t p, uint64_t pol) {
    // written by another block in this kernel: plain (coherent) loads
    const volatile float *kpv = reinterpret_cast<const volatile float *>(a.kparams + l);
    const float4 kp = make_float4(kpv[0], kpv[1], kpv[2], kpv[3]);
    const bool pre = kp.z != 1.0f || kp.w != 1.0f;
    const uint64_t c0 = uint64_t(p) * a.chunks_per_slice;
    const uint64_t c1 = min(c0 + a.chunks_per_slice, a.chunks);
    const uint4 *src = a.k[l];
    uint2 *dst = reinterpret_cast<uint2 *>(a.pool + a.geo.off_layers + uint64_t(l) * a.geo.layer_stride);
    uint64_t c = c0 + threadIdx.x;
    for (; c + 7 * ENC_THREADS < c1; c += 8 * ENC_THREADS) {
        uint4 w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) w[u] = ld_v4_policy(src + c + u * ENC_THREADS, pol);
        if (pre) {
#pragma unroll
            for (int u = 0; u < 8; ++u) __stcs(dst + c + u * ENC_THREADS, k_quant8<true>(w[u], kp));
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) __stcs(dst + c + u * ENC_THREADS, k_quant8<false>(w[u], kp));
        }
    }
    for (; c < c1; c += ENC_THREADS) {
        const uint4 w0 = ld_v4_policy(src + c, pol);
        __stcs(dst + c, pre ? k_quant8<true>(w0, kp) : k_quant8<false>(w0, kp));
    }
}

// ---------------------------------------------------------------------------
// Values ("PolyKV" 2.B.2): one warp step encodes 1024 coordinates, the 8
// vectors of d = 128 or 16 of d = 64 that follow one another in the layer.
//
// Rotation.  The Sylvester-order Walsh-Hadamard matrix is the Kronecker
// product of H_2 over the bits of the coordinate index, so any 4 of the
// index bits can be transformed at once by H_16 and the others separately.
// Four bits go through the tensor cores: mma.m16n8k16 with the vector's bf16
// elements as A and H_16 (entries +-1, exact in bf16) as B, so every product
// is exact and the sums are fp32.  The other 3 bits (d = 128) or 2 bits
// (d = 64) are butterflies on fp32 pairs in registers.
//
// The MMA's k and n index bits (k0, k1, k2, k3) stand for the coordinate
// bits (i0, i5, i6, i2) at d = 128 and (i0, i4, i5, i2) at d = 64: the same
// relabelling on both sides, so B is H_16 in natural order.  An A row is a
// (vector, i1, i3 [, i4]) combination, rows g and g + 8 differing in i1.
// Then each 16-byte chunk of the input is one A fragment as it stands
// (registers x, y, z, w), and lane (g, q) = (lane / 4, lane % 4) ends up
// with the consecutive rotated coordinates [q d/4, (q+1) d/4) of vector g
// (and of vector 8 + g at d = 64): the C element c_{2h+e} of M-tile m,
// N-tile nt is local coordinate 8t + 4nt + 2h + e, t = m (d = 128) or m % 2
// (d = 64).
//
// Codes.  u = y / ||v|| (y = H_d v, unnormalised) falls in cell
// cnt ^ (y >= 0 ? 4 : 3) with cnt = #{k : |y| >= t_k ||v||}.  With
// S = ||y||^2 = d ||v||^2 (Parseval), |y| >= t_k ||v|| exactly when
// y^2 - (t_k^2 / d) S >= 0, and one fma gives that difference with an exact
// sign.  Let n_k be the sign bits of the three differences and s the sign
// of y.  The cells are nested (n1 >= n2 >= n3), so
//     code bit 2 = ~s,  bit 1 = ~(n2 ^ s),  bit 0 = ~(n1 ^ n2 ^ n3 ^ s):
// the sign bits of y, of P = d2 * y (a product's sign is the xor of its
// factors' signs) and of Q = d1 ^ d3 ^ P, inverted.  Each bit is funnel-
// shifted into the little-endian code words, highest coordinate first.
// ---------------------------------------------------------------------------

// Slow path for the rare vector whose S is not finite: Inf/NaN in the input
// (NONFINITE) or finite values too large for sigma (RANGE).
__device__ uint32_t classify_nonfinite(const uint4 *vec, int nchunks) {
    for (int c = 0; c < nchunks; ++c) {
        const uint4 w = vec[c];
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        for (int i = 0; i < 4; ++i)
            if ((ws[i] & 0x7F80u) == 0x7F80u || (ws[i] & 0x7F800000u) == 0x7F800000u) return FLAG_NONFINITE;
    }
    return FLAG_RANGE;
}

// Staging layout.  Chunk c of vector v of a warp step sits at slot
// v * d/8 + (c ^ ((c >> 3 & 1) << 1) ^ (v & 1)) (d = 128) or
// v * d/8 + (c ^ (v & 1)) (d = 64) of the warp's 2 KB buffer.  The XOR
// swizzle makes both the coalesced fill and the fragment reads
// conflict-free: the 8 lanes of a quarter-warp always reach 8 different
// 16-byte bank groups.  The fill copies chunk 32j + lane (j = 0..3) of the
// step, which lands at slot 32j + v_fill_slot(lane).
template <int D>
__device__ __forceinline__ int v_fill_slot(int lane) {
    if (D == 128) {
        const int c = lane & 15, v = lane >> 4;
        return 16 * v + (c ^ (((c >> 3) & 1) << 1) ^ v);
    }
    const int c = lane & 7, v = lane >> 3;
    return 8 * v + (c ^ (v & 1));
}

// Issue the cp.async copies of one warp step's 2 KB of value data (chunks
// [128 step, 128 step + 128) of the layer's values, which hold nvec vectors)
// into the staging buffer.  Chunks past the layer's end get zeros.  Always
// commits one group.
template <int D>
__device__ __forceinline__ void v_prefetch(const uint4 *vlayer, uint32_t nvec, uint32_t step, uint4 *buf,
                                           int fill_slot, uint64_t pol) {
    constexpr uint32_t VPW = 1024 / D;
    const int lane = threadIdx.x & 31;
    const uint32_t n0 = step * VPW;
    const uint32_t left = n0 < nvec ? min(nvec - n0, VPW) * (D / 8) : 0u;
    const uint4 *src = vlayer + uint64_t(step) * 128u + lane;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const bool valid = uint32_t(32 * j + lane) < left;
        cp_async16(buf + 32 * j + fill_slot, valid ? src + 32 * j : vlayer, valid ? 16u : 0u, pol);
    }
    cp_async_commit();
}

// The B fragments of H_16 for N-tiles 0 and 1: lane (g, q) holds the entries
// (k, n) = (2q + {0, 1}, 8nt + g) and (2q + 8 + {0, 1}, 8nt + g), +-1 in bf16
// with the lower k in the low half.
__device__ __forceinline__ void h16_fragments(uint32_t (&hb)[2][2]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int k = 2 * q + 8 * r, n = 8 * nt + g;
            const uint32_t lo = (__popc(k & n) & 1) ? 0xBF80u : 0x3F80u;
            const uint32_t hi = (__popc((k + 1) & n) & 1) ? 0xBF80u : 0x3F80u;
            hb[nt][r] = lo | (hi << 16);
        }
}

__device__ __forceinline__ void mma_h16(float2 &lo, float2 &hi, uint4 w, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(lo.x), "=f"(lo.y), "=f"(hi.x), "=f"(hi.y)
        : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ void bfly2(float2 &a, float2 &b) {
    const float2 s = f2add(a, b);
    b = f2sub(a, b);
    a = s;
}

// Appends bit 31 of src below the bits already in word.
__device__ __forceinline__ void put_bit(uint32_t &word, float src) {
    word = __funnelshift_l(__float_as_uint(src), word, 1);
}
__device__ __forceinline__ void put_bit(uint32_t &word, uint32_t src) { word = __funnelshift_l(src, word, 1); }

// Codes of one lane's coordinates of one vector: pairs y[p] hold local
// coordinates (2p, 2p + 1); nt_k = -(t_k^2 / d) S.  W gets the 3 NP * 2 bits,
// code of local coordinate j at bits 3j .. 3j + 2 (inverted afterwards).
template <int NP>
__device__ __forceinline__ void v_codes(const float2 (&y)[NP], float nt1, float nt2, float nt3,
                                        uint32_t (&W)[(6 * NP + 31) / 32]) {
    const float2 n1 = make_float2(nt1, nt1), n2 = make_float2(nt2, nt2), n3 = make_float2(nt3, nt3);
#pragma unroll
    for (int p = NP - 1; p >= 0; --p) {
        const float2 yy = y[p];
        const float2 d1 = __ffma2_rn(yy, yy, n1), d2 = __ffma2_rn(yy, yy, n2), d3 = __ffma2_rn(yy, yy, n3);
        const float2 P = __fmul2_rn(d2, yy);
        const uint32_t qx = __float_as_uint(d1.x) ^ __float_as_uint(d3.x) ^ __float_as_uint(P.x);
        const uint32_t qy = __float_as_uint(d1.y) ^ __float_as_uint(d3.y) ^ __float_as_uint(P.y);
        const int j1 = 2 * p + 1, j0 = 2 * p;
        put_bit(W[(3 * j1 + 2) >> 5], yy.y);
        put_bit(W[(3 * j1 + 1) >> 5], P.y);
        put_bit(W[(3 * j1) >> 5], qy);
        put_bit(W[(3 * j0 + 2) >> 5], yy.x);
        put_bit(W[(3 * j0 + 1) >> 5], P.x);
        put_bit(W[(3 * j0) >> 5], qx);
    }
}

// t_k^2 for the Lloyd-Max decision thresholds t_k (kvp_vec.cuh).
constexpr float TSQ1 = float(double(THR1) * double(THR1));
constexpr float TSQ2 = float(double(THR2) * double(THR2));
constexpr float TSQ3 = float(double(THR3) * double(THR3));

// Square root for sigma: the approximate instruction is within 2^-22 of the
// real root, well inside the fp16 rounding that follows.
__device__ __forceinline__ float sqrt_approx(float x) {
    float r;
    asm("sqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// One warp step: vectors [step * VPW, step * VPW + VPW) of a layer of nvec
// vectors whose values start at vlayer, whose packed codes go to vsec and
// whose sigmas go to ssec.
template <int D>
__device__ uint32_t v_encode_step(const uint4 *vlayer, uint8_t *vsec, uint16_t *ssec, uint32_t nvec, uint32_t step,
                                  const uint4 *buf, const uint32_t (&hb)[2][2]) {
    constexpr int VPW = 1024 / D;           // vectors per warp step
    constexpr int NV = D == 128 ? 1 : 2;    // vectors per lane
    constexpr int NP = D / 8;               // coordinate pairs per lane and vector
    constexpr int CPV = D / 8;              // 16-byte chunks per vector
    constexpr int CB = 3 * D / 8;           // code bytes per vector
    constexpr float INV_D = 1.0f / float(D);
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const uint32_t n0 = step * VPW;

    // y[m][nt][h] = (c_{2h}, c_{2h+1}) of M-tile m, N-tile nt.  M-tile m
    // reads chunk 4q + m of vector g (d = 128) or chunk 2q + m % 2 of vector
    // 8 (m / 2) + g (d = 64); the staging layout puts it at rd + off(m).
    const uint4 *rd = buf + (D == 128 ? 16 * g + 4 * q : 8 * g + 2 * q);
    const int X = D == 128 ? 2 * (q >> 1) + (g & 1) : (g & 1);
    float2 y[4][2][2];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint4 w = rd[D == 128 ? (m ^ X) : 64 * (m >> 1) + ((m & 1) ^ X)];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) mma_h16(y[m][nt][0], y[m][nt][1], w, hb[nt][0], hb[nt][1]);
    }
    // the register-held index bits: i1 (h), i3 (bit 0 of m) and, at d = 128, i4 (bit 1 of m)
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) bfly2(y[m][nt][0], y[m][nt][1]);
#pragma unroll
    for (int m = 0; m < 4; m += 2)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) bfly2(y[m][nt][h], y[m + 1][nt][h]);
    if (D == 128) {
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h) bfly2(y[m][nt][h], y[m + 2][nt][h]);
    }

    // the lane's pairs per vector, in local-coordinate order: pair p = 4t + 2nt + h
    float2 yp[NV][NP];
#pragma unroll
    for (int vi = 0; vi < NV; ++vi)
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            const int t = p >> 2, nt = (p >> 1) & 1, h = p & 1;
            yp[vi][p] = y[D == 128 ? t : 2 * vi + t][nt][h];
        }

    float S[NV];
#pragma unroll
    for (int vi = 0; vi < NV; ++vi) {
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int p = 0; p < NP; ++p) acc = __ffma2_rn(yp[vi][p], yp[vi][p], acc);
        S[vi] = acc.x + acc.y;
        S[vi] += __shfl_xor_sync(0xffffffffu, S[vi], 1);
        S[vi] += __shfl_xor_sync(0xffffffffu, S[vi], 2);
    }
    bool tiny[NV];
    bool any_tiny = false;
#pragma unroll
    for (int vi = 0; vi < NV; ++vi) {
        tiny[vi] = S[vi] < 0x1p-100f;
        any_tiny |= tiny[vi];
    }
    // S below 2^-100 loses precision to underflow in the squares: rescale the
    // rotated vector by 2^60 (exact) and take S again (codes are scale-free;
    // sigma is below 2^-56, an fp16 zero).  A zero vector gets +0 everywhere
    // and thresholds above every square: every code 4.
    if (__any_sync(0xffffffffu, any_tiny)) {
#pragma unroll
        for (int vi = 0; vi < NV; ++vi) {
            const float f = tiny[vi] ? 0x1p60f : 1.0f;
            float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                yp[vi][p] = __fmul2_rn(yp[vi][p], make_float2(f, f));
                acc = __ffma2_rn(yp[vi][p], yp[vi][p], acc);
            }
            float s2 = acc.x + acc.y;
            s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
            s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
            if (tiny[vi]) {
                S[vi] = s2;
                if (s2 == 0.0f) {
#pragma unroll
                    for (int p = 0; p < NP; ++p) yp[vi][p] = make_float2(0.0f, 0.0f);
                }
            }
        }
    }

    // sigma; the rare non-finite or out-of-range vector is classified off the
    // common path (RANGE: finite input whose sigma exceeds fp16; non-finite
    // input is NONFINITE only)
    uint32_t flags = 0;
    uint32_t n[NV];
    bool valid[NV];
    uint16_t sig[NV];
    bool bad = false;
#pragma unroll
    for (int vi = 0; vi < NV; ++vi) {
        n[vi] = n0 + uint32_t(D == 128 ? g : 8 * vi + g);
        valid[vi] = n[vi] < nvec;
        sig[vi] = tiny[vi] ? 0 : __half_as_ushort(__float2half_rn(sqrt_approx(S[vi]) * INV_D));
        bad |= valid[vi] && (!(S[vi] <= 3.0e38f) || (sig[vi] & 0x7C00u) == 0x7C00u);
    }
    if (__any_sync(0xffffffffu, bad)) {
#pragma unroll
        for (int vi = 0; vi < NV; ++vi) {
            if (valid[vi] && !(S[vi] <= 3.0e38f))
                flags |= classify_nonfinite(vlayer + uint64_t(n[vi]) * CPV, CPV);
            else if (valid[vi] && (sig[vi] & 0x7C00u) == 0x7C00u)
                flags |= FLAG_RANGE;
        }
    }
#pragma unroll
    for (int vi = 0; vi < NV; ++vi) {
        const float s = S[vi];
        // a zero vector (y = +0): thresholds below every square, but finite,
        // so that P = d2 * y is -0 and not inf * 0
        const float nt1 = s == 0.0f ? -FLT_MAX : -(s * (TSQ1 * INV_D));
        const float nt2 = s == 0.0f ? -FLT_MAX : -(s * (TSQ2 * INV_D));
        const float nt3 = s == 0.0f ? -FLT_MAX : -(s * (TSQ3 * INV_D));
        uint32_t W[(6 * NP + 31) / 32];
#pragma unroll
        for (int i = 0; i < (6 * NP + 31) / 32; ++i) W[i] = 0;
        v_codes<NP>(yp[vi], nt1, nt2, nt3, W);
        uint8_t *dst = vsec + uint64_t(n[vi]) * CB + uint32_t(q) * (CB / 4);
        if (valid[vi]) {
            if (D == 128) {
#pragma unroll
                for (int i = 0; i < 3; ++i) __stcs(reinterpret_cast<unsigned int *>(dst) + i, ~W[i]);
            } else {
                unsigned short *d16 = reinterpret_cast<unsigned short *>(dst);
                __stcs(d16 + 0, (unsigned short)(~W[0]));
                __stcs(d16 + 1, (unsigned short)(~W[0] >> 16));
                __stcs(d16 + 2, (unsigned short)(~W[1]));
            }
        }
        if (valid[vi] && q == 0) __stcs(reinterpret_cast<unsigned short *>(ssec) + n[vi], (unsigned short)sig[vi]);
    }
    return flags;
}

// The pool header, written by the last block (all error bits are in).
__device__ void write_header(const EncodeArgs &a) {
    __threadfence();
    for (uint64_t i = 80 + threadIdx.x; i < POOL_HEADER_BYTES; i += ENC_THREADS) a.pool[i] = 0;
    for (uint64_t i = a.geo.off_scales + 4ull * a.L + threadIdx.x; i < a.geo.off_layers; i += ENC_THREADS)
        a.pool[i] = 0;
    if (threadIdx.x == 0) {
        uint32_t *h = reinterpret_cast<uint32_t *>(a.pool);
        h[0] = POOL_MAGIC;
        h[1] = POOL_VERSION;
        h[2] = uint32_t(a.L);
        h[3] = uint32_t(a.H);
        h[4] = uint32_t(a.d);
        h[5] = uint32_t(a.T);
        h[POOL_ERR_WORD] = *reinterpret_cast<volatile uint32_t *>(&a.ctl->flags);
        h[POOL_KMODE_WORD] = a.kmode;
        uint64_t *h64 = reinterpret_cast<uint64_t *>(a.pool);
        h64[4] = a.geo.off_scales;
        h64[5] = a.geo.off_layers;
        h64[6] = a.geo.layer_stride;
        h64[7] = a.geo.sec_v;
        h64[8] = a.geo.sec_sigma;
        h64[9] = a.kmode == KVP_K_Q8_0 ? a.geo.total_q8 : a.geo.total;
    }
}

template <int D>
__global__ void __launch_bounds__(ENC_THREADS, 3) encode_pool(const __grid_constant__ EncodeArgs a) {
    __shared__ __align__(16) uint4 vbuf[ENC_WARPS][2][128];  // per warp: two steps of value data
    __shared__ uint32_t red[ENC_WARPS];
    __shared__ uint4 s_item[2];  // (queue index, kind, layer, id), decoded once by thread 0
    __shared__ uint32_t s_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t keep = l2_evict_last_policy(), drop = l2_evict_first_policy();
    uint32_t hb[2][2];
    h16_fragments(hb);
    const int fill_slot = v_fill_slot<D>(lane);
    uint32_t flags = 0;
    // The next queue index is fetched while the current item runs (thread 0
    // holds it in a register) and decoded by thread 0 alone; the broadcast
    // slot alternates between two entries so one barrier per item suffices.
    uint32_t next = 0;
    if (threadIdx.x == 0) next = atomicAdd(&a.ctl->next_item, 1u);
    for (uint32_t k = 0;; ++k) {
        if (threadIdx.x == 0) {
            int kd = 0, ly = 0;
            uint32_t ix = 0;
            if (next < a.total_items) item_of(a, next, kd, ly, ix);
            s_item[k & 1u] = make_uint4(next, uint32_t(kd), uint32_t(ly), ix);
        }
        __syncthreads();
        const uint4 it = s_item[k & 1u];
        if (it.x >= a.total_items) break;
        if (threadIdx.x == 0) next = atomicAdd(&a.ctl->next_item, 1u);
        const int kind = int(it.y), layer = int(it.z);
        const uint32_t id = it.w;
        if (kind == ITEM_ABSMAX) {
            absmax_slice(a, layer, id, keep, red);
            if (threadIdx.x == 0) {
                __threadfence();  // this slice's partial before the count
                s_flag = atomicAdd(&a.ctl->slices_done[layer], 1u) == uint32_t(a.P) - 1u;
            }
            __syncthreads();
            if (s_flag) finalize_layer(a, layer);
        } else if (kind == ITEM_KEYS) {
            if (threadIdx.x == 0) {
                // bounded wait for the layer's scale (released by another block)
                uint32_t ok = 1, i = 0;
                while (ld_acquire_u32(&a.ctl->ready[layer]) == 0u) {
                    if (++i >= a.spin_limit) {
                        ok = 0;
                        break;
                    }
                    __nanosleep(100);
                }
                __threadfence();
                s_flag = ok;
            }
            __syncthreads();
            if (s_flag)
                quant_slice(a, layer, id, drop);
            else if (threadIdx.x == 0)
                flags |= FLAG_TIMEOUT;
        } else {
            // the warp's VSTEPS steps, each prefetched while the previous one is encoded
            const uint32_t step0 = id * uint32_t(VSTEPS * ENC_WARPS) + uint32_t(warp);
            const uint32_t nvec = uint32_t(a.nvec), nsteps = uint32_t(a.steps_per_layer);
            const uint4 *vlayer = a.v[layer];
            uint8_t *lay = a.pool + a.geo.off_layers + uint64_t(layer) * a.geo.layer_stride;
            uint8_t *vsec = lay + a.geo.sec_v;
            uint16_t *ssec = reinterpret_cast<uint16_t *>(lay + a.geo.sec_sigma);
            v_prefetch<D>(vlayer, nvec, step0, vbuf[warp][0], fill_slot, drop);
#pragma unroll 1
            for (int vs = 0; vs < VSTEPS; ++vs) {
                const uint32_t step = step0 + uint32_t(vs * ENC_WARPS);
                if (vs + 1 < VSTEPS)
                    v_prefetch<D>(vlayer, nvec, step + ENC_WARPS, vbuf[warp][(vs + 1) & 1], fill_slot, drop);
                else
                    cp_async_commit();  // keep one group per iteration
                cp_async_wait<1>();     // this lane's copies of this step have landed
                __syncwarp();           // ... and every other lane's
                if (step < nsteps)  // warp-uniform
                    flags |= v_encode_step<D>(vlayer, vsec, ssec, nvec, step, vbuf[warp][vs & 1], hb);
                __syncwarp();           // the buffer is read before it is refilled
            }
            cp_async_wait<0>();
        }
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (lane == 0 && flags) atomicOr(&a.ctl->flags, flags);
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_flag = atomicAdd(&a.ctl->blocks_done, 1u) == gridDim.x - 1u;
    }
    __syncthreads();
    if (s_flag) write_header(a);
}

// ---------------------------------------------------------------------------
// q8_0 keys (KVP_K_Q8_0): every 32 consecutive keys of a vector share an fp16
// scale s_b = fp16(max|k| / 127); codes as above against s_b, clamped to
// [-127, 127].  No layer-wide maximum, so one sweep encodes keys and values
// on the block-level queue: per layer, key slices (4 lanes per 32-key block:
// two shuffles give the block's maximum) spread among the value batches, and
// nothing waits.  The fp16 scale is fp16(max|k| * fl(1/127)): that
// fp32 product is within 2^-23 relative of the real quotient max|k|/127,
// which never lies closer than 2^-20 relative to an fp16 midpoint (a bf16
// over 127 is at least that far from any 12-bit fraction), so the fp16
// rounding is the correct one.
// ---------------------------------------------------------------------------
constexpr float Q8_INV127 = 1.0f / 127.0f;

// Fast path as k_quant8: the code is the low byte of fma(k, r, 1.5*2^23),
// with r an approximate 1/s (relative error below 2^-21, so k*r is within
// 4e-5 of k/s for |k/s| <= 127.1).  The chunk is redone exactly when an
// estimate is within 1e-4 of a half-integer or not finite, and when s is an
// fp16 subnormal (then |k/s| may exceed 127.5 and the code is clamped);
// non-finite keys code as 0.
__device__ __forceinline__ uint2 k_quant8_block(uint4 w, float s, float rcp, bool subnormal_scale) {
    const float k[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                        bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
    uint32_t t[8];
    bool slow = subnormal_scale;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float tf = fmaf(k[i], rcp, RNE_MAGIC);
        const float e = fmaf(k[i], rcp, -(tf - RNE_MAGIC));
        slow |= !(fabsf(e) <= 0.4999f);
        t[i] = __float_as_uint(tf);
    }
    if (slow) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int q = k_code_exact_int(k[i], s, __uint_as_float(t[i]) - RNE_MAGIC);
            q = max(-127, min(127, q));
            if (!(fabsf(k[i]) <= 3.0e38f)) q = 0;  // Inf / NaN: code 0 (reported)
            t[i] = uint32_t(q) & 0xFFu;
        }
    }
    uint2 r;
    r.x = __byte_perm(__byte_perm(t[0], t[1], 0x0040), __byte_perm(t[2], t[3], 0x0040), 0x5410);
    r.y = __byte_perm(__byte_perm(t[4], t[5], 0x0040), __byte_perm(t[6], t[7], 0x0040), 0x5410);
    return r;
}

// One 16-byte key chunk c of layer l (w: its 8 keys; valid: c < chunks),
// with the warp's lanes 4k .. 4k+3 holding the 4 chunks of one 32-key block
// (every lane of the warp takes part: the block maximum is two shuffles).
__device__ __forceinline__ uint32_t q8_chunk(const EncodeArgs &a, uint2 *dst, uint16_t *ksc, uint64_t c, uint4 w,
                                             bool valid) {
    const int lane = threadIdx.x & 31;
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    // block maximum: per-halfword max of the sign-cleared patterns; Inf /
    // NaN patterns sort above every finite one, so a block holding one is
    // redone with those halves masked out (its maximum over finite keys)
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) m2 = __vmaxu2(m2, ws[i] & 0x7FFF7FFFu);
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
    const bool bad = m >= 0x7F80u;
    if (__any_sync(0xffffffffu, bad)) {
        uint32_t f2 = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t ab = ws[i] & 0x7FFF7FFFu;
            f2 = __vmaxu2(f2, ab & ~__vcmpgeu2(ab, 0x7F807F80u));  // 0xFFFF in each Inf / NaN half
        }
        uint32_t f = max(f2 & 0xFFFFu, f2 >> 16);
        f = max(f, __shfl_xor_sync(0xffffffffu, f, 1));
        f = max(f, __shfl_xor_sync(0xffffffffu, f, 2));
        if (bad) m = f;
    }
    // fp16(max|k| * fl(1/127)): for every finite bf16 maximum this is the
    // fp16 nearest to the real max|k|/127 (checked over all of them)
    const __half sh = __float2half_rn(__fmul_rn(__uint_as_float(m << 16), Q8_INV127));
    const uint16_t sb = __half_as_ushort(sh);
    const float s = __half2float(sh);
    uint32_t flags = 0;
    if (valid) {
        if (bad)
            flags |= FLAG_NONFINITE;
        else if ((sb & 0x7C00u) == 0x7C00u)
            flags |= FLAG_RANGE;
        const uint2 codes =
            (s > 0.0f && s <= 65504.0f) ? k_quant8_block(w, s, __fdividef(1.0f, s), s < 0x1p-14f) : make_uint2(0, 0);
        __stcs(dst + c, codes);
        if ((lane & 3) == 0) __stcs(reinterpret_cast<unsigned short *>(ksc) + (c >> 2), (unsigned short)sb);
    }
    return flags;
}

// One key slice of layer l on the block-level queue: chunks
// [p * chunks_per_slice, ...) (slice bounds are multiples of 4 chunks, so
// lanes 4k .. 4k+3 hold one 32-key block), 4 chunks per thread in flight.
__device__ uint32_t q8_slice(const EncodeArgs &a, int l, uint32_t p, uint64_t pol) {
    const uint64_t c0 = uint64_t(p) * a.chunks_per_slice;
    const uint64_t c1 = min(c0 + a.chunks_per_slice, a.chunks);
    const uint4 *src = a.k[l];
    uint2 *dst = reinterpret_cast<uint2 *>(a.pool + a.geo.off_layers + uint64_t(l) * a.geo.layer_stride);
    uint16_t *ksc = reinterpret_cast<uint16_t *>(a.pool + a.geo.off_kscales) + uint64_t(l) * (a.chunks / 4);
    uint32_t flags = 0;
    for (uint64_t cb = c0; cb < c1; cb += 4 * ENC_THREADS) {  // the same trip count in every thread
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint64_t c = cb + threadIdx.x + uint64_t(u) * ENC_THREADS;
            w[u] = c < c1 ? ld_v4_policy(src + c, pol) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint64_t c = cb + threadIdx.x + uint64_t(u) * ENC_THREADS;
            flags |= q8_chunk(a, dst, ksc, c, w[u], c < c1);
        }
    }
    return flags;
}

// The q8_0 encoder on the block-level queue: per layer, its P key slices
// spread evenly among its value batches (there is no layer-wide maximum, so
// nothing waits); item t belongs to layer t / (P + vitems).
template <int D>
__global__ void __launch_bounds__(ENC_THREADS, 3) encode_pool_q8q(const __grid_constant__ EncodeArgs a) {
    __shared__ __align__(16) uint4 vbuf[ENC_WARPS][2][128];  // per warp: two steps of value data
    __shared__ uint4 s_item[2];  // (queue index, kind, layer, id), decoded once by thread 0
    __shared__ uint32_t s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t drop = l2_evict_first_policy();
    uint32_t hb[2][2];
    h16_fragments(hb);
    const int fill_slot = v_fill_slot<D>(lane);
    const uint32_t M = uint32_t(a.P) + a.vitems;
    uint32_t flags = 0;
    uint32_t next = 0;
    if (threadIdx.x == 0) next = atomicAdd(&a.ctl->next_item, 1u);
    for (uint32_t k = 0;; ++k) {
        if (threadIdx.x == 0) {
            int kd = 0;
            uint32_t ix = 0;
            if (next < a.total_items) mixed_item(a, next % M, kd, ix);
            s_item[k & 1u] = make_uint4(next, uint32_t(kd), next / M, ix);
        }
        __syncthreads();
        const uint4 it = s_item[k & 1u];
        if (it.x >= a.total_items) break;
        if (threadIdx.x == 0) next = atomicAdd(&a.ctl->next_item, 1u);
        const int kind = int(it.y), layer = int(it.z);
        const uint32_t id = it.w;
        if (kind == ITEM_KEYS) {
            flags |= q8_slice(a, layer, id, drop);
        } else {
            // the warp's VSTEPS steps, each prefetched while the previous one is encoded
            const uint32_t step0 = id * uint32_t(VSTEPS * ENC_WARPS) + uint32_t(warp);
            const uint32_t nvec = uint32_t(a.nvec), nsteps = uint32_t(a.steps_per_layer);
            const uint4 *vlayer = a.v[layer];
            uint8_t *lay = a.pool + a.geo.off_layers + uint64_t(layer) * a.geo.layer_stride;
            uint8_t *vsec = lay + a.geo.sec_v;
            uint16_t *ssec = reinterpret_cast<uint16_t *>(lay + a.geo.sec_sigma);
            v_prefetch<D>(vlayer, nvec, step0, vbuf[warp][0], fill_slot, drop);
#pragma unroll 1
            for (int vs = 0; vs < VSTEPS; ++vs) {
                const uint32_t step = step0 + uint32_t(vs * ENC_WARPS);
                if (vs + 1 < VSTEPS)
                    v_prefetch<D>(vlayer, nvec, step + ENC_WARPS, vbuf[warp][(vs + 1) & 1], fill_slot, drop);
                else
                    cp_async_commit();  // keep one group per iteration
                cp_async_wait<1>();     // this lane's copies of this step have landed
                __syncwarp();           // ... and every other lane's
                if (step < nsteps)  // warp-uniform
                    flags |= v_encode_step<D>(vlayer, vsec, ssec, nvec, step, vbuf[warp][vs & 1], hb);
                __syncwarp();           // the buffer is read before it is refilled
            }
            cp_async_wait<0>();
        }
    }
    // deterministic image: layer gaps, the unused per-tensor scales, the
    // tail of the block-scale region
    for (int l = blockIdx.x; l < a.L; l += gridDim.x) zero_layer_gaps(a, l);
    if (blockIdx.x == gridDim.x - 1) {
        for (uint64_t i = threadIdx.x; i < 4ull * uint64_t(a.L); i += ENC_THREADS) a.pool[a.geo.off_scales + i] = 0;
        for (uint64_t i = a.geo.off_kscales + 2ull * uint64_t(a.L) * (a.chunks / 4) + threadIdx.x;
             i < a.geo.total_q8; i += ENC_THREADS)
            a.pool[i] = 0;
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (lane == 0 && flags) atomicOr(&a.ctl->flags, flags);
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(&a.ctl->blocks_done, 1u) == gridDim.x - 1u;
    }
    __syncthreads();
    if (s_last) write_header(a);
}

template <int D>
static int encode_occupancy() {
    static int occ = 0;
    if (occ == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, encode_pool<D>, ENC_THREADS, 0) != cudaSuccess ||
            occ < 1)
            occ = 1;
    }
    return occ;
}

// Failure-path testing (kvp_test_fail_next_encode): consumed by the next
// encode on the calling thread.
static thread_local int t_fail_layer = -1;
static thread_local uint32_t t_fail_spin = SPIN_LIMIT;

}  // namespace kvp

using namespace kvp;

extern "C" int kvp_test_fail_next_encode(int layer, uint32_t spin_iters) {
    t_fail_layer = layer < 0 ? -1 : layer;
    t_fail_spin = layer < 0 ? SPIN_LIMIT : (spin_iters > 0 ? spin_iters : 1u);
    return KVP_OK;
}

extern "C" size_t kvpool_workspace_bytes(const kvp_shape *s) {
    if (shape_ok(s) != KVP_OK) return 0;
    return size_t(ws_layout(s->n_layers).total);
}

extern "C" size_t kvpool_pool_bytes_ex(const kvp_shape *s, int k_mode) {
    if (shape_ok(s) != KVP_OK || (k_mode != KVP_K_PER_TENSOR && k_mode != KVP_K_Q8_0)) return 0;
    const PoolGeom g = pool_geom(s->n_layers, s->n_kv_heads, s->head_dim, s->n_tokens);
    return size_t(k_mode == KVP_K_Q8_0 ? g.total_q8 : g.total);
}

template <int D>
static int encode_q8_occupancy() {
    static int occ = 0;
    if (occ == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, encode_pool_q8q<D>, ENC_THREADS, 0) != cudaSuccess ||
            occ < 1)
            occ = 1;
    }
    return occ;
}

extern "C" int kvpool_encode(const kvp_shape *s, const void *const *k_layers, const void *const *v_layers,
                             void *pool, size_t pool_bytes, void *ws, size_t ws_bytes, void *stream) {
    return kvpool_encode_ex(s, KVP_K_PER_TENSOR, k_layers, v_layers, pool, pool_bytes, ws, ws_bytes, stream);
}

extern "C" int kvpool_encode_ex(const kvp_shape *s, int k_mode, const void *const *k_layers,
                                const void *const *v_layers, void *pool, size_t pool_bytes, void *ws,
                                size_t ws_bytes, void *stream) {
    int rc = shape_ok(s);
    if (rc != KVP_OK) return rc;
    if (k_mode != KVP_K_PER_TENSOR && k_mode != KVP_K_Q8_0) return KVP_ERR_ARG;
    if (!k_layers || !v_layers || !pool || !ws) return KVP_ERR_ARG;
    const int L = s->n_layers;
    for (int l = 0; l < L; ++l) {
        if (!k_layers[l] || !v_layers[l]) return KVP_ERR_ARG;
        if (!aligned(k_layers[l], 16) || !aligned(v_layers[l], 16)) return KVP_ERR_ALIGN;
    }
    if (!aligned(pool, 256) || !aligned(ws, 16)) return KVP_ERR_ALIGN;
    const PoolGeom geo = pool_geom(L, s->n_kv_heads, s->head_dim, s->n_tokens);
    if (pool_bytes < (k_mode == KVP_K_Q8_0 ? geo.total_q8 : geo.total)) return KVP_ERR_SIZE;
    const uint64_t chunks = uint64_t(s->n_kv_heads) * uint64_t(s->n_tokens) * uint64_t(s->head_dim) / 8;
    const WsLayout wl = ws_layout(L);
    if (ws_bytes < wl.total) return KVP_ERR_SIZE;

    EncodeArgs a;
    for (int l = 0; l < L; ++l) {
        a.k[l] = static_cast<const uint4 *>(k_layers[l]);
        a.v[l] = static_cast<const uint4 *>(v_layers[l]);
    }
    for (int l = L; l < KVP_MAX_LAYERS; ++l) a.k[l] = a.v[l] = nullptr;
    a.pool = static_cast<uint8_t *>(pool);
    uint8_t *w = static_cast<uint8_t *>(ws);
    a.ctl = reinterpret_cast<EncodeCtl *>(w + wl.ctl);
    a.kparams = reinterpret_cast<float4 *>(w + wl.kparams);
    a.geo = geo;
    a.chunks = chunks;
    a.L = L;
    a.H = s->n_kv_heads;
    a.T = s->n_tokens;
    a.d = s->head_dim;
    a.kmode = uint32_t(k_mode);
    a.P = slices_per_layer(chunks);
    a.chunks_per_slice = (chunks + a.P - 1) / a.P;
    a.nvec = uint64_t(a.H) * uint64_t(a.T);
    const int vpw = a.d == 128 ? 8 : 16;
    a.steps_per_layer = (a.nvec + vpw - 1) / vpw;
    const uint64_t vitems = (a.steps_per_layer + ENC_WARPS * VSTEPS - 1) / (ENC_WARPS * VSTEPS);
    const uint64_t ipl = 2ull * uint64_t(a.P) + vitems;
    if (ipl * uint64_t(L) >= (1ull << 32)) return KVP_ERR_SIZE;
    a.vitems = uint32_t(vitems);
    a.total_items = uint32_t(ipl * uint64_t(L));
    const uint64_t resident =
        uint64_t(sm_count()) * uint64_t(a.d == 128 ? encode_occupancy<128>() : encode_occupancy<64>());
    const unsigned grid = unsigned(resident < a.total_items ? resident : a.total_items);
    // Between a layer's last absmax slice and its first quantize slice the
    // queue holds about two grids' worth of items, so the absmax slices are
    // done by then: `lag` whole rounds (as many as needed, while the keys of
    // lag+1 layers fit in 48 MB of L2), then a head of value batches for the
    // rest.
    const uint64_t kbytes = chunks * 16u;
    const uint64_t want = 2ull * grid;
    const uint64_t lag_l2 = kbytes >= (48ull << 20) ? 0 : (48ull << 20) / kbytes - 1;
    uint64_t lag = (want + ipl - 1) / ipl;
    if (lag > lag_l2) lag = lag_l2;
    if (lag > uint64_t(L)) lag = uint64_t(L);
    a.lag = uint32_t(lag);
    const uint64_t covered = lag * ipl;
    const uint64_t head = covered >= want ? 0 : want - covered;
    a.vhead = uint32_t(head < vitems ? head : vitems);
    a.seg0 = lag * uint32_t(a.P);
    a.seg1 = a.seg0 + (uint32_t(L) - lag) * uint32_t(ipl);
    a.fail_layer = t_fail_layer;
    a.spin_limit = t_fail_spin;
    t_fail_layer = -1;
    t_fail_spin = SPIN_LIMIT;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(a.ctl, 0, sizeof(EncodeCtl), st) != cudaSuccess) return KVP_ERR_CUDA;
    if (k_mode == KVP_K_Q8_0) {
        // the block-level queue without absmax items: per layer, key slices (a
        // multiple of 4 chunks each: whole 32-key blocks) spread among the
        // value batches; nothing waits
        a.chunks_per_slice = (a.chunks_per_slice + 3) & ~uint64_t(3);
        a.P = int((chunks + a.chunks_per_slice - 1) / a.chunks_per_slice);
        a.vhead = 0;
        const uint64_t items = (uint64_t(a.P) + vitems) * uint64_t(L);
        if (items >= (1ull << 32)) return KVP_ERR_SIZE;
        a.total_items = uint32_t(items);
        const uint64_t res_q8 =
            uint64_t(sm_count()) * uint64_t(a.d == 128 ? encode_q8_occupancy<128>() : encode_q8_occupancy<64>());
        const unsigned g8 = unsigned(items < res_q8 ? items : res_q8);
        if (a.d == 128)
            encode_pool_q8q<128><<<g8, ENC_THREADS, 0, st>>>(a);
        else
            encode_pool_q8q<64><<<g8, ENC_THREADS, 0, st>>>(a);
    } else if (a.d == 128) {
        encode_pool<128><<<grid, ENC_THREADS, 0, st>>>(a);
    } else {
        encode_pool<64><<<grid, ENC_THREADS, 0, st>>>(a);
    }
    count_launch(1);
    return launch_status();
}
