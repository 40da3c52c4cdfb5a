// kvpool_encode.cu -- SharedKVPool encoder ("PolyKV" 2.B asymmetric
// compression): int8 keys with one symmetric scale per layer tensor; values
// rotated by a Walsh-Hadamard transform, normalised by sigma = ||v||/sqrt(d)
// (fp16), quantized to the 8-level Lloyd-Max codebook and packed 8 codes to 3
// bytes.
//
// Three launches on the caller's stream:
//   1. encode_phase1: a persistent grid of G blocks works through L*P key
//      slices (max|k| of one slice of one layer -> a partial) interleaved
//      with the value batches (every value vector of every layer: it does not
//      depend on the key scale), recording error bits in one slot per block.
//   2. encode_finalize: one block per layer folds its P partials into the
//      layer's maximum, writes the fp32 scale s = m/127 into the pool and the
//      key-quantizer parameters into the workspace; block 0 writes the pool
//      header (with the OR of every error bit) and zeroes alignment gaps.
//   3. encode_keys: int8 codes = the integer nearest to the exact k/s.
// No block waits on another; the workspace needs no initialisation.
#include "kvp_vec.cuh"

namespace kvp {

constexpr int ENC_THREADS = 256;
constexpr int ENC_WARPS = ENC_THREADS / 32;
constexpr uint64_t ABSMAX_MIN_CHUNKS = 2048;  // 16-byte chunks per absmax block, at least
constexpr int ABSMAX_MAX_BLOCKS = 256;        // per layer
constexpr int VFLAG_SLOTS = 1024;             // value-encode blocks, at most
constexpr float RNE_MAGIC = 12582912.0f;      // 1.5 * 2^23

struct EncodeArgs {
    const uint4 *k[KVP_MAX_LAYERS];
    const uint4 *v[KVP_MAX_LAYERS];
    uint8_t *pool;
    uint32_t *partials;  // [L][P]
    uint32_t *vflags;    // [G]
    float4 *kparams;     // [L]: s_eff, 1/s_eff, prescale1, prescale2
    PoolGeom geo;
    uint64_t chunks;           // 16-byte chunks per layer of K (H*T*d/8)
    uint64_t chunks_per_block; // per absmax block
    int L, H, T, d, P, G;
};

// Workspace: partials, value flags, key parameters (each 16-byte aligned).
struct WsLayout {
    uint64_t partials, vflags, kparams, total;
};

static inline int absmax_blocks(uint64_t chunks) {
    uint64_t p = (chunks + ABSMAX_MIN_CHUNKS - 1) / ABSMAX_MIN_CHUNKS;
    if (p < 1) p = 1;
    if (p > ABSMAX_MAX_BLOCKS) p = ABSMAX_MAX_BLOCKS;
    return int(p);
}

static inline WsLayout ws_layout(int L, uint64_t chunks) {
    WsLayout w;
    const int P = absmax_blocks(chunks);
    w.partials = 0;
    w.vflags = align16(4ull * uint64_t(L) * uint64_t(P));
    w.kparams = align16(w.vflags + 4ull * VFLAG_SLOTS);
    w.total = align16(w.kparams + 16ull * uint64_t(L));
    return w;
}

// ---------------------------------------------------------------------------
// Phase 1a: partial max|k| of one slice of one layer, on the bf16 bit
// patterns with the sign cleared (for finite values the order of the
// patterns is the order of the magnitudes; Inf/NaN patterns sort above
// every finite one, so they flag themselves).
// ---------------------------------------------------------------------------
__device__ void absmax_slice(const EncodeArgs &a, int bid) {
    const int l = bid / a.P, p = bid % a.P;
    const uint64_t c0 = uint64_t(p) * a.chunks_per_block;
    const uint64_t c1 = min(c0 + a.chunks_per_block, a.chunks);
    const uint4 *src = a.k[l];
    uint32_t mlo = 0, mhi = 0;
    uint64_t c = c0 + threadIdx.x;
    for (; c + 3 * ENC_THREADS < c1; c += 4 * ENC_THREADS) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) w[u] = ld_stream_v4(src + c + u * ENC_THREADS);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            mlo = max(mlo, max(max(w[u].x & 0x7FFFu, w[u].y & 0x7FFFu), max(w[u].z & 0x7FFFu, w[u].w & 0x7FFFu)));
            mhi = max(mhi, max(max(w[u].x & 0x7FFF0000u, w[u].y & 0x7FFF0000u),
                               max(w[u].z & 0x7FFF0000u, w[u].w & 0x7FFF0000u)));
        }
    }
    for (; c < c1; c += ENC_THREADS) {
        const uint4 w = ld_stream_v4(src + c);
        mlo = max(mlo, max(max(w.x & 0x7FFFu, w.y & 0x7FFFu), max(w.z & 0x7FFFu, w.w & 0x7FFFu)));
        mhi = max(mhi, max(max(w.x & 0x7FFF0000u, w.y & 0x7FFF0000u), max(w.z & 0x7FFF0000u, w.w & 0x7FFF0000u)));
    }
    uint32_t m = max(mlo, mhi >> 16);
    m = __reduce_max_sync(0xffffffffu, m);
    __shared__ uint32_t red[ENC_WARPS];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t r = red[0];
#pragma unroll
        for (int i = 1; i < ENC_WARPS; ++i) r = max(r, red[i]);
        a.partials[bid] = r;
    }
    __syncthreads();  // red[] is reused by the block's next slice
}

// ---------------------------------------------------------------------------
// Phase 1b: value vectors ("PolyKV" 2.B.2).  One warp handles VPW vectors per
// step; see kvp_vec.cuh for the lane mapping.
// ---------------------------------------------------------------------------

// Slow path for the rare vector whose squared norm is not finite: Inf/NaN in
// the input (NONFINITE) or finite values too large for sigma (RANGE).
__device__ uint32_t classify_nonfinite(const uint4 *vec, int nchunks) {
    for (int c = 0; c < nchunks; ++c) {
        const uint4 w = vec[c];
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        for (int i = 0; i < 4; ++i)
            if ((ws[i] & 0x7F80u) == 0x7F80u || (ws[i] & 0x7F800000u) == 0x7F800000u) return FLAG_NONFINITE;
    }
    return FLAG_RANGE;
}

// One warp step: VPW consecutive vectors of one layer (see kvp_vec.cuh for
// the lane mapping).  Returns error bits.
template <int D>
__device__ uint32_t v_encode_step(const EncodeArgs &a, uint64_t step, uint64_t steps_per_layer, uint8_t *stage) {
    constexpr int LPV = D / 32;      // lanes per vector
    constexpr int VPW = 32 / LPV;    // vectors per warp step
    constexpr int CPV = D / 8;       // 16-byte chunks per vector
    constexpr int CB = 3 * D / 8;    // code bytes per vector
    static_assert(VPW * CB == 384, "a warp step stages 384 code bytes");
    const int lane = threadIdx.x & 31;
    const int g = lane / LPV, l = lane % LPV;
    const uint64_t nvec = uint64_t(a.H) * uint64_t(a.T);
    const float inv_d = 1.0f / float(D);
    uint32_t flags = 0;

    const int layer = int(step / steps_per_layer);
    const uint64_t n0 = (step % steps_per_layer) * VPW;
    const uint64_t n = n0 + g;
    const bool valid = n < nvec;
    const uint4 *vec = a.v[layer] + n * CPV;

    // x[j][p] = (v_a + v_b, v_a - v_b) for the coordinate pair (a, b) = (2p, 2p+1)
    // of chunk j: the first butterfly stage is applied while unpacking.
    uint4 w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = valid ? ld_stream_v4(vec + j * LPV + l) : make_uint4(0, 0, 0, 0);
    float2 x[4][4];
    float2 n2v = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t ws[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float2 v = make_float2(bf16_lo(ws[p]), bf16_hi(ws[p]));
            n2v = __ffma2_rn(v, v, n2v);
            x[j][p] = make_float2(v.x + v.y, v.x - v.y);
        }
    }
    float n2 = n2v.x + n2v.y;
#pragma unroll
    for (int m = 1; m < LPV; m <<= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, m);

    fwht_pairs<LPV>(x, lane);

    // Thresholds t_k * ||v|| in the unnormalised rotated domain.
    float nrm = sqrtf(n2);
    uint16_t sig_bits = __half_as_ushort(__float2half_rn(sqrtf(n2 * inv_d)));
    // A norm below 2^-50 loses precision to underflow in n2: rescale the
    // rotated vector by 2^60 (exact) and take the norm from it through
    // Parseval (||y||^2 = d ||v||^2).  sigma is below 2^-53: fp16 zero.
    const bool tiny = n2 < 0x1p-100f;
    if (__any_sync(0xffffffffu, tiny)) {
        float s2 = 0.0f;
        const float2 sc = make_float2(0x1p60f, 0x1p60f);
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float2 ys = __fmul2_rn(x[j][p], sc);
                if (tiny) x[j][p] = ys;
                s2 = fmaf(ys.x, ys.x, fmaf(ys.y, ys.y, s2));
            }
#pragma unroll
        for (int m = 1; m < LPV; m <<= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, m);
        if (tiny) {
            nrm = sqrtf(s2 * inv_d);
            sig_bits = 0;
        }
    }
    // RANGE: finite input whose sigma exceeds fp16; non-finite input is
    // NONFINITE only.
    if (valid && !(n2 <= 3.0e38f))
        flags |= classify_nonfinite(vec, CPV);
    else if (valid && (sig_bits & 0x7C00u) == 0x7C00u)
        flags |= FLAG_RANGE;

    float T1 = THR1 * nrm, T2 = THR2 * nrm, T3 = THR3 * nrm;
    if (nrm == 0.0f) T1 = T2 = T3 = __int_as_float(0x7F800000);  // zero vector: all codes 4

    uint8_t *st = stage + g * CB;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t cw = 0;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            cw |= v_code(x[j][p].x, T1, T2, T3) << (6 * p);
            cw |= v_code(x[j][p].y, T1, T2, T3) << (6 * p + 3);
        }
        const int c = j * LPV + l;
        st[3 * c + 0] = uint8_t(cw);
        st[3 * c + 1] = uint8_t(cw >> 8);
        st[3 * c + 2] = uint8_t(cw >> 16);
    }
    __syncwarp();

    uint8_t *lay = a.pool + a.geo.off_layers + uint64_t(layer) * a.geo.layer_stride;
    const uint64_t nv_here = min(uint64_t(VPW), nvec - n0);
    const uint32_t bytes = uint32_t(nv_here) * CB;
    uint8_t *vdst = lay + a.geo.sec_v + n0 * CB;
    const uint32_t off = uint32_t(lane) * 16u;
    if (off + 16u <= bytes) {
        *reinterpret_cast<uint4 *>(vdst + off) = *reinterpret_cast<const uint4 *>(stage + off);
    } else if (off < bytes) {  // bytes is a multiple of 8
        *reinterpret_cast<uint2 *>(vdst + off) = *reinterpret_cast<const uint2 *>(stage + off);
    }
    if (valid && l == 0) reinterpret_cast<uint16_t *>(lay + a.geo.sec_sigma)[n] = sig_bits;
    __syncwarp();
    return flags;
}

// Phase 1 work items: L*P key-absmax slices and ceil(value steps / 8)
// value batches (8 warp steps, one per warp), interleaved so that both kinds
// run on every SM at once (key reads overlap the value transform's ALU work).
struct Phase1Items {
    uint64_t na, nv, total;
    __device__ __forceinline__ void at(uint64_t t, bool &is_abs, uint64_t &id) const {
        const uint64_t both = 2 * min(na, nv);
        if (t < both) {
            is_abs = (t & 1u) == 0;
            id = t >> 1;
        } else {
            is_abs = na > nv;
            id = t - both + min(na, nv);
        }
    }
};

template <int D>
__global__ void __launch_bounds__(ENC_THREADS, 3) encode_phase1(const __grid_constant__ EncodeArgs a) {
    constexpr int VPW = 32 / (D / 32);
    __shared__ __align__(16) uint8_t stage[ENC_WARPS][384];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t nvec = uint64_t(a.H) * uint64_t(a.T);
    const uint64_t steps_per_layer = (nvec + VPW - 1) / VPW;
    const uint64_t vsteps = steps_per_layer * uint64_t(a.L);
    Phase1Items items;
    items.na = uint64_t(a.L) * uint64_t(a.P);
    items.nv = (vsteps + ENC_WARPS - 1) / ENC_WARPS;
    items.total = items.na + items.nv;
    uint32_t flags = 0;
    for (uint64_t t = blockIdx.x; t < items.total; t += gridDim.x) {
        bool is_abs;
        uint64_t id;
        items.at(t, is_abs, id);
        if (is_abs) {
            absmax_slice(a, int(id));
        } else {
            const uint64_t step = id * ENC_WARPS + warp;
            if (step < vsteps) flags |= v_encode_step<D>(a, step, steps_per_layer, stage[warp]);
        }
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    __shared__ uint32_t fl[ENC_WARPS];
    if (lane == 0) fl[warp] = flags;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t f = 0;
#pragma unroll
        for (int i = 0; i < ENC_WARPS; ++i) f |= fl[i];
        a.vflags[blockIdx.x] = f;
    }
}

// ---------------------------------------------------------------------------
// Phase 2: per-layer scale and key-quantizer parameters; the pool header.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(ENC_THREADS) encode_finalize(const __grid_constant__ EncodeArgs a) {
    const int l = blockIdx.x;
    __shared__ uint32_t red[ENC_WARPS];
    uint32_t m = 0;
    for (int i = threadIdx.x; i < a.P; i += ENC_THREADS) m = max(m, a.partials[l * a.P + i]);
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t r = red[0];
        for (int i = 1; i < ENC_WARPS; ++i) r = max(r, red[i]);
        const bool finite = r < 0x7F80u;
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
                // tie test below cannot underflow.
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
    // Zero this layer's alignment gaps so the pool image is deterministic.
    {
        uint8_t *lay = a.pool + a.geo.off_layers + uint64_t(l) * a.geo.layer_stride;
        const uint64_t nv = uint64_t(a.H) * uint64_t(a.T);
        const uint64_t gaps[3][2] = {{nv * uint64_t(a.d), a.geo.sec_v},
                                     {a.geo.sec_v + nv * uint64_t(3 * a.d / 8), a.geo.sec_sigma},
                                     {a.geo.sec_sigma + 2 * nv, a.geo.layer_stride}};
        for (int gi = 0; gi < 3; ++gi)
            for (uint64_t i = gaps[gi][0] + threadIdx.x; i < gaps[gi][1]; i += ENC_THREADS) lay[i] = 0;
    }
    if (l == 0) {
        // Error bits: every value-encode slot and every key partial.
        uint32_t f = 0;
        for (int i = threadIdx.x; i < a.G; i += ENC_THREADS) f |= a.vflags[i];
        for (int i = threadIdx.x; i < a.L * a.P; i += ENC_THREADS)
            if (a.partials[i] >= 0x7F80u) f |= FLAG_NONFINITE;
        f = __reduce_or_sync(0xffffffffu, f);
        __syncthreads();
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = f;
        __syncthreads();
        uint32_t *h = reinterpret_cast<uint32_t *>(a.pool);
        // bytes 80..(off_layers): header tail and the gap after the scales
        for (uint64_t i = 80 + threadIdx.x; i < POOL_HEADER_BYTES; i += ENC_THREADS) a.pool[i] = 0;
        for (uint64_t i = a.geo.off_scales + 4ull * a.L + threadIdx.x; i < a.geo.off_layers; i += ENC_THREADS)
            a.pool[i] = 0;
        if (threadIdx.x == 0) {
            uint32_t ff = 0;
            for (int i = 0; i < ENC_WARPS; ++i) ff |= red[i];
            h[0] = POOL_MAGIC;
            h[1] = POOL_VERSION;
            h[2] = uint32_t(a.L);
            h[3] = uint32_t(a.H);
            h[4] = uint32_t(a.d);
            h[5] = uint32_t(a.T);
            h[POOL_ERR_WORD] = ff;
            h[7] = 0;
            uint64_t *h64 = reinterpret_cast<uint64_t *>(a.pool);
            h64[4] = a.geo.off_scales;
            h64[5] = a.geo.off_layers;
            h64[6] = a.geo.layer_stride;
            h64[7] = a.geo.sec_v;
            h64[8] = a.geo.sec_sigma;
            h64[9] = a.geo.total;
        }
    }
}

// ---------------------------------------------------------------------------
// Phase 3: int8 key codes ("PolyKV" 2.B.1).  q = the integer nearest to the
// real k/s, ties to even.  Fast path: t = fma(k, 1/s, 1.5*2^23) rounds k/s'
// (k/s within 1.6e-5) to an integer held in t's low mantissa bits, whose low
// byte is the two's-complement code.  Only when that estimate is within 1e-4
// of a half-integer is the decision taken exactly: the sign of
// k - (q0 +- 1/2) s is exact under one fma rounding.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t k_code_exact(float k, float s, float q0) {
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
    return uint32_t(q) & 0xFFu;
}

template <bool PRESCALE>
__device__ __forceinline__ uint2 k_quant8(uint4 w, float4 kp) {
    float k[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                  bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
    if (PRESCALE) {
#pragma unroll
        for (int i = 0; i < 8; ++i) k[i] = (k[i] * kp.z) * kp.w;
    }
    uint32_t t[8];
    bool near = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float tf = fmaf(k[i], kp.y, RNE_MAGIC);
        const float q0 = tf - RNE_MAGIC;
        const float e = fmaf(k[i], kp.y, -q0);
        near |= fabsf(e) > 0.4999f;
        t[i] = __float_as_uint(tf);
    }
    if (near) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float q0 = __uint_as_float(t[i]) - RNE_MAGIC;
            t[i] = k_code_exact(k[i], kp.x, q0);
        }
    }
    uint2 r;
    r.x = __byte_perm(__byte_perm(t[0], t[1], 0x0040), __byte_perm(t[2], t[3], 0x0040), 0x5410);
    r.y = __byte_perm(__byte_perm(t[4], t[5], 0x0040), __byte_perm(t[6], t[7], 0x0040), 0x5410);
    return r;
}

__global__ void __launch_bounds__(ENC_THREADS) encode_keys(const __grid_constant__ EncodeArgs a, int blocks_per_layer) {
    const int l = blockIdx.x / blocks_per_layer, b = blockIdx.x % blocks_per_layer;
    const float4 kp = a.kparams[l];
    const uint4 *src = a.k[l];
    uint2 *dst = reinterpret_cast<uint2 *>(a.pool + a.geo.off_layers + uint64_t(l) * a.geo.layer_stride);
    const uint64_t stride = uint64_t(blocks_per_layer) * ENC_THREADS;
    const bool pre = kp.z != 1.0f || kp.w != 1.0f;
    uint64_t c = uint64_t(b) * ENC_THREADS + threadIdx.x;
    for (; c + stride < a.chunks; c += 2 * stride) {
        const uint4 w0 = ld_stream_v4(src + c), w1 = ld_stream_v4(src + c + stride);
        if (pre) {
            dst[c] = k_quant8<true>(w0, kp);
            dst[c + stride] = k_quant8<true>(w1, kp);
        } else {
            dst[c] = k_quant8<false>(w0, kp);
            dst[c + stride] = k_quant8<false>(w1, kp);
        }
    }
    for (; c < a.chunks; c += stride) {
        const uint4 w0 = ld_stream_v4(src + c);
        dst[c] = pre ? k_quant8<true>(w0, kp) : k_quant8<false>(w0, kp);
    }
}

template <int D>
static int phase1_occupancy() {
    static int occ = 0;
    if (occ == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, encode_phase1<D>, ENC_THREADS, 0) != cudaSuccess ||
            occ < 1)
            occ = 1;
    }
    return occ;
}

}  // namespace kvp

using namespace kvp;

extern "C" size_t kvpool_workspace_bytes(const kvp_shape *s) {
    if (shape_ok(s) != KVP_OK) return 0;
    const uint64_t chunks = uint64_t(s->n_kv_heads) * uint64_t(s->n_tokens) * uint64_t(s->head_dim) / 8;
    return size_t(ws_layout(s->n_layers, chunks).total);
}

extern "C" int kvpool_encode(const kvp_shape *s, const void *const *k_layers, const void *const *v_layers,
                             void *pool, size_t pool_bytes, void *ws, size_t ws_bytes, void *stream) {
    int rc = shape_ok(s);
    if (rc != KVP_OK) return rc;
    if (!k_layers || !v_layers || !pool || !ws) return KVP_ERR_ARG;
    const int L = s->n_layers;
    for (int l = 0; l < L; ++l) {
        if (!k_layers[l] || !v_layers[l]) return KVP_ERR_ARG;
        if (!aligned(k_layers[l], 16) || !aligned(v_layers[l], 16)) return KVP_ERR_ALIGN;
    }
    if (!aligned(pool, 256) || !aligned(ws, 16)) return KVP_ERR_ALIGN;
    const PoolGeom geo = pool_geom(L, s->n_kv_heads, s->head_dim, s->n_tokens);
    if (pool_bytes < geo.total) return KVP_ERR_SIZE;
    const uint64_t chunks = uint64_t(s->n_kv_heads) * uint64_t(s->n_tokens) * uint64_t(s->head_dim) / 8;
    const WsLayout wl = ws_layout(L, chunks);
    if (ws_bytes < wl.total) return KVP_ERR_SIZE;

    EncodeArgs a;
    for (int l = 0; l < L; ++l) {
        a.k[l] = static_cast<const uint4 *>(k_layers[l]);
        a.v[l] = static_cast<const uint4 *>(v_layers[l]);
    }
    for (int l = L; l < KVP_MAX_LAYERS; ++l) a.k[l] = a.v[l] = nullptr;
    a.pool = static_cast<uint8_t *>(pool);
    uint8_t *w = static_cast<uint8_t *>(ws);
    a.partials = reinterpret_cast<uint32_t *>(w + wl.partials);
    a.vflags = reinterpret_cast<uint32_t *>(w + wl.vflags);
    a.kparams = reinterpret_cast<float4 *>(w + wl.kparams);
    a.geo = geo;
    a.chunks = chunks;
    a.L = L;
    a.H = s->n_kv_heads;
    a.T = s->n_tokens;
    a.d = s->head_dim;
    a.P = absmax_blocks(chunks);
    a.chunks_per_block = (chunks + a.P - 1) / a.P;
    const int sms = sm_count();
    const uint64_t nvec = uint64_t(a.H) * uint64_t(a.T);
    const uint64_t vsteps = (nvec + (a.d == 128 ? 8 : 16) - 1) / (a.d == 128 ? 8 : 16) * uint64_t(L);
    // persistent phase-1 grid: one block per resident slot, one flag slot per block
    const uint64_t items = uint64_t(a.L) * uint64_t(a.P) + (vsteps + ENC_WARPS - 1) / ENC_WARPS;
    const uint64_t gmax = uint64_t(sms) * uint64_t(a.d == 128 ? phase1_occupancy<128>() : phase1_occupancy<64>());
    uint64_t g = items < gmax ? items : gmax;
    if (g > VFLAG_SLOTS) g = VFLAG_SLOTS;
    a.G = int(g < 1 ? 1 : g);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (a.d == 128)
        encode_phase1<128><<<unsigned(a.G), ENC_THREADS, 0, st>>>(a);
    else
        encode_phase1<64><<<unsigned(a.G), ENC_THREADS, 0, st>>>(a);
    encode_finalize<<<L, ENC_THREADS, 0, st>>>(a);
    uint64_t bpl = (chunks + 2ull * ENC_THREADS * 4 - 1) / (2ull * ENC_THREADS * 4);
    const uint64_t bmax = (uint64_t(sms) * 8 + L - 1) / L;
    if (bpl > bmax) bpl = bmax;
    if (bpl < 1) bpl = 1;
    encode_keys<<<unsigned(uint64_t(L) * bpl), ENC_THREADS, 0, st>>>(a, int(bpl));
    count_launch(3);
    return launch_status();
}
