// cachecard.cu -- QKVShare CacheCard ("QKVShare: Quantized KV-Cache Handoff
// for Multi-Agent On-Device LLMs", Methodology 1-3): per-token bitwidth from
// {2,4,8,16}; asymmetric min/max quantization in groups of 32 coordinates
// with fp16 scale and zero point; the receiver rebuilds bf16 past_key_values.
//
// cachecard_pack: card_scan (one block: bitwidths -> record offsets, header)
// then card_pack (one warp per (layer, token, K|V) record half).
// cachecard_unpack: the inverse, one warp per record half: card_unpack_staged
// (the next record brought into shared memory by bulk copies while the
// current one is unpacked) where its buffers fit, else card_unpack.
// cachecard_unpack_at: the same with the keys turned to new positions.
#include <cmath>

#include "kvp_async.cuh"
#include "kvp_internal.cuh"

namespace kvp {

constexpr int CARD_THREADS = 256;
constexpr int CARD_WARPS = CARD_THREADS / 32;
constexpr int SCAN_THREADS = 1024;
constexpr float RNE_MAGIC_C = 12582912.0f;  // 1.5 * 2^23

struct CardArgs {
    const uint4 *src[2][KVP_MAX_LAYERS];  // pack: K, V inputs.  unpack: unused
    uint4 *dst[2][KVP_MAX_LAYERS];        // unpack: K, V outputs
    uint8_t *card;
    const uint8_t *bits_dev;
    uint64_t card_bytes;
    uint64_t model_id;
    int64_t pos_offset;
    uint64_t off_offsets, off_layers, layer_stride;
    int L, H, T, d;
    uint32_t it_dt, it_dl;  // staged unpack: (token, layer) step of a warp's tasks
    uint32_t wait_polls;    // staged unpack: polls of a buffer's copies before giving up
    int64_t shift;      // unpack_at: target offset - card offset
    float2 rot[64];     // unpack_at: (cos, sin) of shift * w_i for the d/2 rotary frequencies w_i
};

// ---------------------------------------------------------------------------
// Offsets and header ("QKVShare" Methodology 2: bitwidths + metadata).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(SCAN_THREADS) card_scan(const __grid_constant__ CardArgs a) {
    __shared__ unsigned long long wsum[SCAN_THREADS / 32];
    __shared__ uint32_t wbad[SCAN_THREADS / 32];
    const int T = a.T;
    const int per = (T + SCAN_THREADS - 1) / SCAN_THREADS;
    const int t0 = min(T, int(threadIdx.x) * per), t1 = min(T, t0 + per);
    unsigned long long sum = 0;
    uint32_t bad = 0;
    for (int t = t0; t < t1; ++t) {
        const int b = a.bits_dev[t];
        if (valid_bits(b)) sum += card_record_bytes(b, a.H, a.d);
        else bad = 1;
    }
    // block-wide exclusive scan of the per-thread sums
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 31) wsum[warp] = incl;
    if (lane == 0) wbad[warp] = bad;
    __syncthreads();
    unsigned long long wpre = 0, total = 0;
    uint32_t anybad = 0;
    for (int w = 0; w < SCAN_THREADS / 32; ++w) {
        if (w < warp) wpre += wsum[w];
        total += wsum[w];
        anybad |= wbad[w];
    }
    unsigned long long run = wpre + incl - sum;
    uint8_t *bits = a.card + CARD_HEADER_BYTES;
    uint32_t *offs = reinterpret_cast<uint32_t *>(a.card + a.off_offsets);
    for (int t = t0; t < t1; ++t) {
        const int b = a.bits_dev[t];
        bits[t] = uint8_t(b);
        offs[t] = uint32_t(run);
        if (valid_bits(b)) run += card_record_bytes(b, a.H, a.d);
    }
    // zero the gaps after bits[] and after off[]
    for (uint64_t i = CARD_HEADER_BYTES + uint64_t(T) + threadIdx.x; i < a.off_offsets; i += SCAN_THREADS) a.card[i] = 0;
    for (uint64_t i = a.off_offsets + 4ull * uint64_t(T) + threadIdx.x; i < a.off_layers; i += SCAN_THREADS)
        a.card[i] = 0;
    if (threadIdx.x == 0) {
        const uint64_t stride = align256(total);
        const uint64_t bytes = a.off_layers + uint64_t(a.L) * stride;
        uint32_t err = 0;
        if (anybad) err |= FLAG_BITS;
        if (total >= (1ull << 32) || bytes > a.card_bytes) err |= FLAG_SIZE;
        kvp_card_header h;
        h.magic = CARD_MAGIC;
        h.version = CARD_VERSION;
        h.seq_len = T;
        h.n_layers = a.L;
        h.n_kv_heads = a.H;
        h.head_dim = a.d;
        h.group_size = CARD_GROUP;
        h.dtype = 1;
        h.model_id = a.model_id;
        h.pos_offset = a.pos_offset;
        h.off_bits = CARD_HEADER_BYTES;
        h.off_offsets = a.off_offsets;
        h.off_layers = a.off_layers;
        h.layer_stride = stride;
        h.total_bytes = bytes;
        h.error = err;
        for (int i = 0; i < 9; ++i) h.reserved[i] = 0;
        *reinterpret_cast<kvp_card_header *>(a.card) = h;
    }
}

// ---------------------------------------------------------------------------
// fp16 group scale, correctly rounded: s_h = RNE_fp16((mx - mn) / qmax).
// mx - mn is carried exactly as hi + lo (two-sum); the fp16 estimate from
// fp32 arithmetic is then checked against its two neighbouring fp16
// midpoints m, where the sign of (hi + lo) - m*qmax is exact (m*qmax has at
// most 20 significant bits; hi - m*qmax is exact when the two are within a
// factor 2, and dominates lo otherwise).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int cmp_mid(float hi, float lo, float m, float qmax) {
    const float r = fmaf(-m, qmax, hi) + lo;
    return r > 0.0f ? 1 : (r < 0.0f ? -1 : 0);
}

// fp32 value of the midpoint between normal fp16 h and the next fp16 value
// (65520 above 65504): h's bits widened to fp32 with the rounding bit set.
__device__ __forceinline__ float f16_mid_above(uint32_t h) {
    return __uint_as_float(((h << 13) | 0x1000u) + 0x38000000u);
}

__device__ uint16_t group_scale_f16(float mx, float mn, float qmax, float rcp_qmax) {
    const float hi = mx - mn;
    const float bb = hi - mx;
    const float lo = (mx - (hi - bb)) + (-mn - bb);
    // estimate within one fp16 step of the answer; the checks below make it exact
    uint32_t h = __half_as_ushort(__float2half_rn(hi * rcp_qmax));
    if (h >= 0x0401u && h <= 0x7BFFu) {  // h and h - 1 normal: midpoints by bit arithmetic
        // at most one of the two moves applies (the midpoints are ordered)
        const float ru = fmaf(-f16_mid_above(h), qmax, hi) + lo;
        const float rl = fmaf(-f16_mid_above(h - 1), qmax, hi) + lo;
        const bool odd = (h & 1u) != 0;
        const uint32_t up = (ru > 0.0f || (ru == 0.0f && odd)) ? 1u : 0u;
        const uint32_t dn = (rl < 0.0f || (rl == 0.0f && odd)) ? 1u : 0u;
        return uint16_t(h + up - dn);
    }
    if (h == 0x7C00u) return cmp_mid(hi, lo, 65520.0f, qmax) < 0 ? uint16_t(0x7BFFu) : uint16_t(h);
    const float vh = __half2float(__ushort_as_half(uint16_t(h)));
    const float vn = h == 0x7BFFu ? 65536.0f : __half2float(__ushort_as_half(uint16_t(h + 1)));
    int c = cmp_mid(hi, lo, 0.5f * (vh + vn), qmax);
    if (c > 0 || (c == 0 && (h & 1u))) return uint16_t(h + 1);
    if (h == 0) return uint16_t(h);
    const float vp = __half2float(__ushort_as_half(uint16_t(h - 1)));
    c = cmp_mid(hi, lo, 0.5f * (vp + vh), qmax);
    if (c < 0 || (c == 0 && (h & 1u))) return uint16_t(h - 1);
    return uint16_t(h);
}

// ---------------------------------------------------------------------------
// Pack: one warp per (layer, token, K|V) task; one thread per group of 32
// coordinates (a task with more than 32 groups takes several rounds).  A
// thread loads its group's 64 contiguous bytes (L1-cached, so the warp's
// 2 KB are fetched once), reduces min / max, takes the exactly rounded fp16
// scale, quantizes and packs its 32 codes (4b bytes) and stores them with the
// group's (s_h, z_h); a 16-bit token's group is copied as it is.  The warp's
// rounds form one sequence, software-pipelined: the next round's group is
// loaded before the current one is quantized, so a warp keeps two rounds'
// loads in flight.  Codes are formed and packed eight at a time, which keeps
// the live registers to the two groups and the packed output.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bytes4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
    return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

// A pack task's coordinates: layer l, token t, kv (0 keys, 1 values).  A
// warp's tasks advance by a fixed stride, so the coordinates are stepped
// rather than divided out of the task index.
struct PackPos {
    uint32_t t;
    int l, kv;
};

template <bool FULL>
__device__ __forceinline__ void pack_load(const CardArgs &a, const PackPos &pos, int gi, int ngroups, int cpr,
                                          int gshift, uint32_t T, uint4 (&w)[4]) {
    if (FULL || gi < ngroups) {
        const int h = gi >> gshift, gg = gi & ((1 << gshift) - 1);
        const uint32_t row = uint32_t(h) * T + pos.t;  // H T < 2^31
        const uint4 *p = a.src[pos.kv][pos.l] + uint64_t(row) * uint32_t(cpr) + gg * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q) w[q] = __ldg(p + q);
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) w[q] = make_uint4(0, 0, 0, 0);
    }
}

// The group's 32 codes from its 16 words of bf16 pairs: the low mantissa
// bits of (x - z_h) * r + 1.5*2^23, clamped to [0, qmax] only when the
// group's extremes leave the code range (CLAMP), packed b bits each.
template <bool CLAMP>
__device__ __forceinline__ void pack_codes(const uint32_t (&ws)[16], int b, float2 negz, float2 inv2, float lo_c,
                                           float hi_c, uint32_t (&out)[8]) {
    const float2 mg = make_float2(RNE_MAGIC_C, RNE_MAGIC_C);
#pragma unroll
    for (int e = 0; e < 4; ++e) {  // 8 values (4 words) at a time
        uint32_t q[8];  // the code in the low bits, higher bits not cleared
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t wv = ws[4 * e + i];
            float2 tf = __ffma2_rn(__fadd2_rn(make_float2(bf16_lo(wv), bf16_hi(wv)), negz), inv2, mg);
            if (CLAMP) {
                tf.x = fminf(fmaxf(tf.x, lo_c), hi_c);
                tf.y = fminf(fmaxf(tf.y, lo_c), hi_c);
            }
            q[2 * i] = __float_as_uint(tf.x);
            q[2 * i + 1] = __float_as_uint(tf.y);
        }
        if (b == 8) {
            out[2 * e] = pack_bytes4(q[0], q[1], q[2], q[3]);
            out[2 * e + 1] = pack_bytes4(q[4], q[5], q[6], q[7]);
        } else if (b == 4) {
            uint32_t by[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) by[i] = (q[2 * i] & 0xFu) | ((q[2 * i + 1] & 0xFu) << 4);
            out[e] = pack_bytes4(by[0], by[1], by[2], by[3]);
        } else {
            const uint32_t b0 = (q[0] & 3u) | ((q[1] & 3u) << 2) | ((q[2] & 3u) << 4) | ((q[3] & 3u) << 6);
            const uint32_t b1 = (q[4] & 3u) | ((q[5] & 3u) << 2) | ((q[6] & 3u) << 4) | ((q[7] & 3u) << 6);
            if (e & 1)
                out[e >> 1] |= (b0 << 16) | (b1 << 24);
            else
                out[e >> 1] = b0 | (b1 << 8);
        }
    }
}

// The codes and group parameters of one group (one lane) of a b-bit pack
// round, B < 16: min / max, the fp16 scale and zero point, the codes.  B is a
// template argument so that each bitwidth's code path is straight-line (with
// a run-time b the 4K-token step's pack took 0.149 against 0.135 ms).
template <int B, bool FULL>
__device__ __forceinline__ void pack_group(const CardArgs &a, uint8_t *rec, const uint4 (&w)[4], int gi, int ngroups,
                                           int kv, uint32_t hd, int lane, int round, int rounds, uint32_t &flags) {
    const uint32_t code_bytes = hd * uint32_t(B) / 8u;
    if (FULL || gi < ngroups) {
        const float qmax = float((1 << B) - 1);
        const uint32_t ws[16] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w,
                                 w[2].x, w[2].y, w[2].z, w[2].w, w[3].x, w[3].y, w[3].z, w[3].w};
        // min / max on the packed bf16 pairs (exact).  The maximum
        // propagates NaN, so a group holding Inf or NaN has a non-finite
        // min or max.
        __nv_bfloat162 mnp = *reinterpret_cast<const __nv_bfloat162 *>(&ws[0]), mxp = mnp;
#pragma unroll
        for (int i = 1; i < 16; ++i) {
            const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162 *>(&ws[i]);
            mnp = __hmin2(mnp, pr);
            mxp = __hmax2_nan(mxp, pr);
        }
        const float mn = fminf(__low2float(mnp), __high2float(mnp));
        const float mx0 = __low2float(mxp), mx1 = __high2float(mxp);
        const float mx = fmaxf(mx0, mx1);
        const bool nf = !(fabsf(mn) <= 3.0e38f) || !(fabsf(mx0) <= 3.0e38f) || !(fabsf(mx1) <= 3.0e38f);
        const uint32_t sb = group_scale_f16(mx, mn, qmax, 1.0f / qmax);
        const uint32_t zb = __half_as_ushort(__float2half_rn(mn));
        if (nf)
            flags |= FLAG_NONFINITE;
        else if (((sb & 0x7C00u) == 0x7C00u) || ((zb & 0x7C00u) == 0x7C00u))
            flags |= FLAG_RANGE;
        const float sf = __half2float(__ushort_as_half(uint16_t(sb)));
        const float zf = __half2float(__ushort_as_half(uint16_t(zb)));
        const float inv = (sf > 0.0f && sf <= 65504.0f) ? __fdividef(1.0f, sf) : 0.0f;
        // code = clamp(round((x - z_h) / s_h), 0, 2^b - 1): the low mantissa
        // bits of (x - z_h) * r + 1.5*2^23, r the fast reciprocal of s_h
        // (within 2 ulp): for codes up to 255 the estimate is within 8e-5
        // of the exact quotient, so it rounds the same way unless that
        // quotient lies within 8e-5 of a half-integer.  The map is
        // monotone, so the clamp is needed only if the group's extremes
        // fall outside the code range.
        const float lo_c = RNE_MAGIC_C, hi_c = RNE_MAGIC_C + qmax;
        const float tmn = fmaf(mn - zf, inv, RNE_MAGIC_C), tmx = fmaf(mx - zf, inv, RNE_MAGIC_C);
        const bool clamp = !(tmn >= lo_c && tmx <= hi_c);
        const float2 negz = make_float2(-zf, -zf), inv2 = make_float2(inv, inv);
        uint32_t out[8];  // packed codes: 4b bytes
        if (clamp)
            pack_codes<true>(ws, B, negz, inv2, lo_c, hi_c, out);
        else
            pack_codes<false>(ws, B, negz, inv2, lo_c, hi_c, out);
        uint8_t *codes = rec + (kv ? code_bytes : 0u);
        if (B == 8) {
            uint4 *o = reinterpret_cast<uint4 *>(codes) + 2 * gi;
            o[0] = make_uint4(out[0], out[1], out[2], out[3]);
            o[1] = make_uint4(out[4], out[5], out[6], out[7]);
        } else if (B == 4) {
            reinterpret_cast<uint4 *>(codes)[gi] = make_uint4(out[0], out[1], out[2], out[3]);
        } else {
            reinterpret_cast<uint2 *>(codes)[gi] = make_uint2(out[0], out[1]);
        }
        uint32_t *par = reinterpret_cast<uint32_t *>(rec + 2u * code_bytes + (kv ? hd / 8u : 0u));
        par[gi] = sb | (zb << 16);
    }
    // zero the record's padding (sizes are multiples of 8, records of 16)
    if (kv == 1 && lane == 0 && round == rounds - 1) {
        const uint64_t used = 2ull * code_bytes + hd / 4u;
        const uint64_t padded = card_record_bytes(B, a.H, a.d);
        if (padded > used) *reinterpret_cast<uint2 *>(rec + used) = make_uint2(0, 0);
    }
}

// FULL: every round holds 32 groups (H d / 32 is a multiple of 32), so no
// lane is idle and the per-lane group checks drop out.
template <bool FULL>
__global__ void __launch_bounds__(CARD_THREADS, 4) card_pack(const __grid_constant__ CardArgs a) {
    const kvp_card_header *hdr = reinterpret_cast<const kvp_card_header *>(a.card);
    if (hdr->error & (FLAG_BITS | FLAG_SIZE)) return;
    const uint64_t stride = hdr->layer_stride;  // depends on the device-resident bitwidths
    const int lane = threadIdx.x & 31;
    const int cpr = a.d / 8;                     // 16-byte chunks per head row (8 or 16)
    const int gshift = a.d == 128 ? 2 : 1;       // log2(groups per head row)
    const int ngroups = a.H * (a.d / 32);
    const int rounds = (ngroups + 31) >> 5;
    const uint32_t T = uint32_t(a.T);
    const uint32_t tasks = uint32_t(a.L) * T * 2u;  // fits: checked on the host
    const uint8_t *bits = a.card + CARD_HEADER_BYTES;
    const uint32_t *offs = reinterpret_cast<const uint32_t *>(a.card + a.off_offsets);
    const uint32_t tstep = gridDim.x * CARD_WARPS;
    uint32_t flags = 0;

    uint32_t task = blockIdx.x * CARD_WARPS + (threadIdx.x >> 5);
    // task = 2 (l T + t) + kv; the stride (a multiple of 2 CARD_WARPS) keeps kv
    // and moves (l, t) by dl layers and dt tokens, with a carry
    const uint32_t dlt = tstep >> 1, dt = dlt % T;
    const int dl = int(dlt / T);
    PackPos pos;
    pos.kv = int(task & 1u);
    pos.t = (task >> 1) % T;
    pos.l = int((task >> 1) / T);
    int round = 0;
    uint4 w[4];
    int b = 0;         // the task's bitwidth and record offset, loaded with its first round
    uint32_t off = 0;
    if (task < tasks) {
        pack_load<FULL>(a, pos, lane, ngroups, cpr, gshift, T, w);
        b = bits[pos.t];
        off = offs[pos.t];
    }
    while (task < tasks) {
        // the next round of this warp's sequence, loaded now (with the next
        // task's bitwidth and offset, so that no header load is waited for)
        uint32_t ntask = task;
        PackPos npos = pos;
        int nround = round + 1;
        int nb = b;
        uint32_t noff = off;
        if (nround == rounds) {
            nround = 0;
            ntask += tstep;
            npos.t += dt;
            npos.l += dl;
            if (npos.t >= T) {
                npos.t -= T;
                npos.l += 1;
            }
        }
        uint4 wn[4];
        if (ntask < tasks) {
            pack_load<FULL>(a, npos, nround * 32 + lane, ngroups, cpr, gshift, T, wn);
            if (nround == 0) {
                nb = bits[npos.t];
                noff = offs[npos.t];
            }
        }

        const int gi = round * 32 + lane;
        const int kv = pos.kv;
        const int l = pos.l;
        uint8_t *rec = a.card + a.off_layers + uint64_t(uint32_t(l)) * stride + off;
        const uint32_t hd = uint32_t(a.H) * uint32_t(a.d);  // H d < 2^31
        if (b == 16) {
            if (FULL || gi < ngroups) {
                uint4 *out = reinterpret_cast<uint4 *>(rec + (kv ? 2u * hd : 0u)) + 4 * gi;
#pragma unroll
                for (int q = 0; q < 4; ++q) out[q] = w[q];
            }
        } else if (b == 2) {
            pack_group<2, FULL>(a, rec, w, gi, ngroups, kv, hd, lane, round, rounds, flags);
        } else if (b == 4) {
            pack_group<4, FULL>(a, rec, w, gi, ngroups, kv, hd, lane, round, rounds, flags);
        } else {  // 8: card_scan has flagged any other bitwidth, and this kernel then returns at once
            pack_group<8, FULL>(a, rec, w, gi, ngroups, kv, hd, lane, round, rounds, flags);
        }
        task = ntask;
        pos = npos;
        round = nround;
        b = nb;
        off = noff;
#pragma unroll
        for (int q = 0; q < 4; ++q) w[q] = wn[q];
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (lane == 0 && flags) atomicOr(const_cast<uint32_t *>(&hdr->error), flags);
}

// Zero each layer's tail after its last record (layer_stride is 256-aligned),
// one block per layer, so the card image is fully determined.
__global__ void card_zero_tails(const __grid_constant__ CardArgs a) {
    const kvp_card_header *hdr = reinterpret_cast<const kvp_card_header *>(a.card);
    if (hdr->error & (FLAG_BITS | FLAG_SIZE)) return;
    const uint64_t stride = hdr->layer_stride;
    const uint8_t *bits = a.card + CARD_HEADER_BYTES;
    const uint32_t *offs = reinterpret_cast<const uint32_t *>(a.card + a.off_offsets);
    const uint64_t used = uint64_t(offs[a.T - 1]) + card_record_bytes(bits[a.T - 1], a.H, a.d);
    for (uint64_t i = used + threadIdx.x; i < stride; i += blockDim.x)
        a.card[a.off_layers + uint64_t(blockIdx.x) * stride + i] = 0;
}

// ---------------------------------------------------------------------------
// Unpack ("QKVShare" Methodology 3): x = bf16(q * s_h + z_h); 16-bit tokens
// verbatim.
// ---------------------------------------------------------------------------

// The 8 values of one chunk (8 consecutive dims) of a b-bit group record:
// codes cw (2, 4 or 8 bits each, low bits first), group parameters pw
// (fp16 scale | fp16 zero point << 16).
__device__ __forceinline__ void card_chunk_values(int b, uint2 cw, uint32_t pw, float (&y)[8]) {
    uint32_t q[8];  // the fp32 bit patterns of 2^23 + code
    if (b == 2) {
#pragma unroll
        for (int e = 0; e < 8; ++e) q[e] = ((cw.x >> (2 * e)) & 3u) | 0x4B000000u;
    } else if (b == 4) {
#pragma unroll
        for (int e = 0; e < 8; ++e) q[e] = ((cw.x >> (4 * e)) & 15u) | 0x4B000000u;
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            q[e] = __byte_perm(cw.x, 0x4B000000u, 0x7650u | e);
            q[4 + e] = __byte_perm(cw.y, 0x4B000000u, 0x7650u | e);
        }
    }
    const float sf = __half2float(__ushort_as_half(uint16_t(pw & 0xFFFFu)));
    const float zf = __half2float(__ushort_as_half(uint16_t(pw >> 16)));
    // (2^23 + code) - 2^23 (exact), then code * s + z rounded once: two lanes at a time
    const float2 off = make_float2(-8388608.0f, -8388608.0f), s2 = make_float2(sf, sf), z2 = make_float2(zf, zf);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const float2 c = __fadd2_rn(make_float2(__uint_as_float(q[e]), __uint_as_float(q[e + 1])), off);
        const float2 v = __ffma2_rn(c, s2, z2);
        y[e] = v.x;
        y[e + 1] = v.y;
    }
}

// Codes of chunk c of a b-bit record part.
__device__ __forceinline__ uint2 card_chunk_codes(int b, const uint8_t *codes, int c) {
    if (b == 2) return make_uint2(reinterpret_cast<const uint16_t *>(codes)[c], 0u);
    if (b == 4) return make_uint2(reinterpret_cast<const uint32_t *>(codes)[c], 0u);
    return reinterpret_cast<const uint2 *>(codes)[c];
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&y)[8]) {
    return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                      pack_bf16x2(y[6], y[7]));
}

// One (layer, token, K|V) task of a plain unpack, by one warp: lanes over
// the H * d/8 chunks of the token.  B: the token's bitwidth, a template
// argument so that each bitwidth's code path is straight-line (a run-time b
// inside the chunk loop costs the 4K-token step's unpack 3 %).
template <int B>
__device__ __forceinline__ void unpack_task_b(const CardArgs &a, const uint8_t *rec, uint4 *dst, int kv, uint32_t t,
                                              int lane) {
    const int cpr = a.d / 8;
    const int cshift = a.d == 128 ? 4 : 3;
    const int nchunks = a.H * cpr;
    const uint32_t T = uint32_t(a.T);
    const uint32_t hd = uint32_t(a.H) * uint32_t(a.d);
    if (B == 16) {
        const uint4 *in = reinterpret_cast<const uint4 *>(rec + (kv ? 2u * hd : 0u));
        for (int c = lane; c < nchunks; c += 32) {
            const int h = c >> cshift, ch = c & (cpr - 1);
            st_stream_v4(dst + (uint64_t(h) * T + t) * cpr + ch, ld_stream_v4(in + c));
        }
        return;
    }
    const uint32_t code_bytes = hd * uint32_t(B) / 8u;
    const uint8_t *codes = rec + (kv ? code_bytes : 0u);
    const uint32_t *par = reinterpret_cast<const uint32_t *>(rec + 2u * code_bytes + (kv ? hd / 8u : 0u));
    for (int c0 = 0; c0 < nchunks; c0 += 4 * 32) {
        // up to 4 chunks' codes and group parameters per lane in flight
        uint2 cw[4];
        uint32_t pw[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int c = c0 + it * 32 + lane;
            cw[it] = make_uint2(0, 0);
            pw[it] = 0;
            if (c < nchunks) {
                cw[it] = card_chunk_codes(B, codes, c);
                pw[it] = par[c >> 2];
            }
        }
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int c = c0 + it * 32 + lane;
            if (c >= nchunks) break;
            float y[8];
            card_chunk_values(B, cw[it], pw[it], y);
            const int h = c >> cshift, ch = c & (cpr - 1);
            st_stream_v4(dst + (uint64_t(h) * T + t) * cpr + ch, pack_bf16x8(y));
        }
    }
}

// b: a checked bitwidth (2, 4, 8 or 16).
__device__ __forceinline__ void unpack_task_plain(const CardArgs &a, const uint8_t *rec, uint4 *dst, int b, int kv,
                                                  uint32_t t, int lane) {
    switch (b) {
    case 2: unpack_task_b<2>(a, rec, dst, kv, t, lane); break;
    case 4: unpack_task_b<4>(a, rec, dst, kv, t, lane); break;
    case 8: unpack_task_b<8>(a, rec, dst, kv, t, lane); break;
    default: unpack_task_b<16>(a, rec, dst, kv, t, lane); break;
    }
}

// The record of (layer l, token t), or null (and the card's error flag set)
// when its bitwidth or offset does not fit the card's own layer stride.
__device__ __forceinline__ const uint8_t *unpack_record(const CardArgs &a, int l, uint32_t t, int &b, int lane) {
    const uint8_t *bits = a.card + CARD_HEADER_BYTES;
    const uint32_t *offs = reinterpret_cast<const uint32_t *>(a.card + a.off_offsets);
    b = bits[t];
    if (!valid_bits(b) || (offs[t] & 15u) != 0 || uint64_t(offs[t]) + card_record_bytes(b, a.H, a.d) > a.layer_stride) {
        if (lane == 0) atomicOr(&reinterpret_cast<kvp_card_header *>(a.card)->error, FLAG_HEADER);
        return nullptr;
    }
    return a.card + a.off_layers + uint64_t(l) * a.layer_stride + offs[t];
}

// 48 registers, 5 blocks/SM (at 52 the allocator drops to 4 and the 8K-token
// card unpack takes 0.266 against 0.244 ms)
__global__ void __launch_bounds__(CARD_THREADS, 5) card_unpack(const __grid_constant__ CardArgs a) {
    const int lane = threadIdx.x & 31;
    const uint32_t T = uint32_t(a.T);
    const uint32_t tasks = uint32_t(a.L) * T * 2u;  // fits: checked on the host
    for (uint32_t task = blockIdx.x * CARD_WARPS + (threadIdx.x >> 5); task < tasks;
         task += gridDim.x * CARD_WARPS) {
        const int kv = int(task & 1u);
        const uint32_t lt = task >> 1;
        const uint32_t t = lt % T;
        const int l = int(lt / T);
        int b;
        const uint8_t *rec = unpack_record(a, l, t, b, lane);
        if (rec) unpack_task_plain(a, rec, a.dst[kv][l], b, kv, t, lane);
    }
}

// ---------------------------------------------------------------------------
// Unpack with the keys moved to other positions: rotary position embedding
// turns dims (i, i + d/2) through p * w_i at position p, and turns compose,
// so keys embedded at (card offset + t) become the keys at (pos_dst + t) by a
// turn through shift * w_i, shift = pos_dst - card offset ("KVCMAS", How it
// is used: the source cache's key positions are re-aligned to the target's;
// "QKVShare", Methodology 2: the card carries the position offset).  The
// angle is formed and its sine / cosine taken in fp64 on the host, once per
// call, and rounded to fp32; each key is dequantized and turned in fp32, two
// coordinates per packed f32x2 instruction, and rounded to bf16 once.  Values
// are unpacked as by card_unpack.
// ---------------------------------------------------------------------------
// The keys of one token, turned: lanes over the H d/16 pairs of chunks
// (c, c + d/16) of a head row, which hold the coordinates (i, i + d/2) that
// one rotary frequency couples; two pairs (four chunks) per lane in flight.
// B: the token's bitwidth, a template argument so that each bitwidth's
// code path is straight-line.  rc, rs: (cos, sin) of the lane's 8
// frequencies, two per packed register.
template <int B>
__device__ __forceinline__ void rope_keys(const CardArgs &a, const uint8_t *rec, uint4 *dst, uint32_t t, int lane,
                                          const float2 (&rc)[4], const float2 (&rs)[4]) {
    constexpr int b = B;
    const int cpr = a.d / 8, half = cpr / 2;  // chunks per row, per half row
    const int hshift = a.d == 128 ? 3 : 2;     // log2(half)
    const int npairs = a.H * half;
    const int chl = lane & (half - 1);  // the lane's chunk within the half row, the same for every pair
    const uint32_t T = uint32_t(a.T);
    const uint64_t code_bytes = uint64_t(a.H) * a.d * b / 8;
    const uint32_t *par = reinterpret_cast<const uint32_t *>(rec + 2 * code_bytes);
    for (int p0 = 0; p0 < npairs; p0 += 2 * 32) {
        uint4 ra[2], rb[2];
        uint32_t pa[2], pb[2];
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int p = p0 + it * 32 + lane;
            ra[it] = rb[it] = make_uint4(0, 0, 0, 0);
            pa[it] = pb[it] = 0;
            if (p < npairs) {
                const int ca = (p >> hshift) * cpr + (p & (half - 1)), cb = ca + half;
                if (b == 16) {  // resolved at compile time
                    ra[it] = ld_stream_v4(reinterpret_cast<const uint4 *>(rec) + ca);
                    rb[it] = ld_stream_v4(reinterpret_cast<const uint4 *>(rec) + cb);
                } else {
                    const uint2 x = card_chunk_codes(b, rec, ca), y = card_chunk_codes(b, rec, cb);
                    ra[it] = make_uint4(x.x, x.y, 0, 0);
                    rb[it] = make_uint4(y.x, y.y, 0, 0);
                    pa[it] = par[ca >> 2];
                    pb[it] = par[cb >> 2];
                }
            }
        }
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int p = p0 + it * 32 + lane;
            if (p >= npairs) break;
            const int h = p >> hshift;
            const int ca = h * cpr + chl, cb = ca + half;
            float ya[8], yb[8];
            if (b == 16) {
                const uint32_t wa[4] = {ra[it].x, ra[it].y, ra[it].z, ra[it].w};
                const uint32_t wb[4] = {rb[it].x, rb[it].y, rb[it].z, rb[it].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    ya[2 * e] = bf16_lo(wa[e]);
                    ya[2 * e + 1] = bf16_hi(wa[e]);
                    yb[2 * e] = bf16_lo(wb[e]);
                    yb[2 * e + 1] = bf16_hi(wb[e]);
                }
            } else {
                card_chunk_values(b, make_uint2(ra[it].x, ra[it].y), pa[it], ya);
                card_chunk_values(b, make_uint2(rb[it].x, rb[it].y), pb[it], yb);
            }
            // oa = ya cos - yb sin, ob = ya sin + yb cos: one product rounded, then one fma
            float oa[8], ob[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 xa = make_float2(ya[2 * e], ya[2 * e + 1]), xb = make_float2(yb[2 * e], yb[2 * e + 1]);
                const float2 ta = __fmul2_rn(xb, rs[e]), tb = __fmul2_rn(xb, rc[e]);
                const float2 u = __ffma2_rn(xa, rc[e], make_float2(-ta.x, -ta.y));
                const float2 w = __ffma2_rn(xa, rs[e], tb);
                oa[2 * e] = u.x, oa[2 * e + 1] = u.y;
                ob[2 * e] = w.x, ob[2 * e + 1] = w.y;
            }
            st_stream_v4(dst + (uint64_t(h) * T + t) * cpr + (ca - h * cpr), pack_bf16x8(oa));
            st_stream_v4(dst + (uint64_t(h) * T + t) * cpr + (cb - h * cpr), pack_bf16x8(ob));
        }
    }
}

__global__ void __launch_bounds__(CARD_THREADS, 4) card_unpack_rope(const __grid_constant__ CardArgs a) {
    const int lane = threadIdx.x & 31;
    // a lane's chunk within the half row is the same for every pair it takes
    const int chl = lane & (a.d / 16 - 1);
    float2 rc[4], rs[4];  // (cos, sin) of the lane's 8 frequencies, two per packed register
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 r0 = a.rot[chl * 8 + 2 * e], r1 = a.rot[chl * 8 + 2 * e + 1];
        rc[e] = make_float2(r0.x, r1.x);
        rs[e] = make_float2(r0.y, r1.y);
    }
    const uint32_t T = uint32_t(a.T);
    const uint32_t tasks = uint32_t(a.L) * T * 2u;
    // The grid's warp count is even, so task = 2 (l T + t) + kv would give each
    // warp one half (keys or values) for good, and the warps with the heavier
    // key turns would run on alone at the end.  The half is flipped on each of
    // the warp's turns instead: warps 2j and 2j + 1 still take complementary
    // halves of the same token, so every (token, half) is taken once.
    int flip = 0;
    for (uint32_t task = blockIdx.x * CARD_WARPS + (threadIdx.x >> 5); task < tasks;
         task += gridDim.x * CARD_WARPS, flip ^= 1) {
        const int kv = int(task & 1u) ^ flip;
        const uint32_t lt = task >> 1;
        const uint32_t t = lt % T;
        const int l = int(lt / T);
        int b;
        const uint8_t *rec = unpack_record(a, l, t, b, lane);
        if (!rec) continue;
        uint4 *dst = a.dst[kv][l];
        if (kv == 1) {
            unpack_task_plain(a, rec, dst, b, kv, t, lane);
            continue;
        }
        switch (b) {  // unpack_record has checked b
        case 2: rope_keys<2>(a, rec, dst, t, lane, rc, rs); break;
        case 4: rope_keys<4>(a, rec, dst, t, lane, rc, rs); break;
        case 8: rope_keys<8>(a, rec, dst, t, lane, rc, rs); break;
        default: rope_keys<16>(a, rec, dst, t, lane, rc, rs); break;
        }
    }
}

// ---------------------------------------------------------------------------
// Staged unpack.  Each warp has two shared-memory buffers, each with its
// mbarrier.  While it dequantizes task k from one buffer, the half-record
// (codes and group parameters, or the bf16 half of a 16-bit token) of task
// k + 1 lands in the other by bulk copies that its lane 0 issued, and the
// bitwidth and offset of task k + 2 are loaded: a task's record reads are in
// flight through the previous task's arithmetic and stores, with no
// registers held for them.  A warp's tasks advance by a fixed (token, layer)
// step, and the halves are taken as in card_unpack (ROPE = false) and
// card_unpack_rope (ROPE = true).  Used where two buffers of 2 H d bytes per
// warp fit 96 KB per block and every part of a record starts on a 16-byte
// boundary (d = 128, or H even).
// ---------------------------------------------------------------------------
constexpr uint32_t CARD_WAIT_LIMIT = 1u << 22;  // polls, about half a second

// A task's position, bitwidth and record offset; ok: its record may be read.
struct StagedTask {
    uint32_t t, l, off;
    int b;
    bool ok;
};

__device__ __forceinline__ void staged_load_hdr(const CardArgs &a, StagedTask &x) {
    x.b = 0;
    x.off = 0;
    x.ok = false;
    if (x.l < uint32_t(a.L)) {
        x.b = (a.card + CARD_HEADER_BYTES)[x.t];
        x.off = reinterpret_cast<const uint32_t *>(a.card + a.off_offsets)[x.t];
    }
}

__device__ __forceinline__ void staged_check(const CardArgs &a, StagedTask &x) {
    x.ok = x.l < uint32_t(a.L) && valid_bits(x.b) && (x.off & 15u) == 0 &&
           uint64_t(x.off) + card_record_bytes(x.b, a.H, a.d) <= a.layer_stride;
}

__device__ __forceinline__ StagedTask staged_next(const CardArgs &a, const StagedTask &x) {
    StagedTask n;
    n.t = x.t + a.it_dt;
    n.l = x.l + a.it_dl;
    if (n.t >= uint32_t(a.T)) {
        n.t -= uint32_t(a.T);
        n.l += 1;
    }
    staged_load_hdr(a, n);
    return n;
}

// Lane 0: the bulk copies of half kv of task x's record into `stage`
// (codes, then group parameters), completing on `bar`.
__device__ __forceinline__ void staged_issue(const CardArgs &a, const StagedTask &x, int kv, uint32_t stage,
                                             uint32_t bar, uint64_t pol) {
    const uint8_t *rec = a.card + a.off_layers + uint64_t(x.l) * a.layer_stride + x.off;
    const uint32_t hd = uint32_t(a.H) * uint32_t(a.d);
    fence_proxy_async();  // the warp's reads of this buffer (last task) come first
    if (x.b == 16) {
        mbar_expect_tx(bar, 2u * hd);
        bulk_g2s(stage, rec + (kv ? 2u * hd : 0u), 2u * hd, bar, pol);
    } else {
        const uint32_t cb = hd * uint32_t(x.b) / 8u, pb = hd / 8u;
        mbar_expect_tx(bar, cb + pb);
        bulk_g2s(stage, rec + (kv ? cb : 0u), cb, bar, pol);
        bulk_g2s(stage + cb, rec + 2u * cb + (kv ? pb : 0u), pb, bar, pol);
    }
}

// One plain half-task from its staged half-record.
template <int B>
__device__ __forceinline__ void unpack_staged_b(const CardArgs &a, const uint8_t *stage, uint4 *dst, uint32_t t,
                                                int lane) {
    const int cpr = a.d / 8;
    const int cshift = a.d == 128 ? 4 : 3;
    const int nchunks = a.H * cpr;
    const uint32_t T = uint32_t(a.T);
    const uint32_t code_bytes = uint32_t(a.H) * uint32_t(a.d) * uint32_t(B) / 8u;
    for (int c0 = 0; c0 < nchunks; c0 += 4 * 32) {
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int c = c0 + it * 32 + lane;
            if (c >= nchunks) break;
            const int h = c >> cshift, ch = c & (cpr - 1);
            uint4 v;
            if (B == 16) {
                v = reinterpret_cast<const uint4 *>(stage)[c];
            } else {
                float y[8];
                card_chunk_values(B, card_chunk_codes(B, stage, c),
                                  reinterpret_cast<const uint32_t *>(stage + code_bytes)[c >> 2], y);
                v = pack_bf16x8(y);
            }
            st_stream_v4(dst + (uint64_t(h) * T + t) * cpr + ch, v);
        }
    }
}

// The keys of one token, turned, from the staged half-record (pairs of chunks
// as in rope_keys).
template <int B>
__device__ __forceinline__ void rope_staged_b(const CardArgs &a, const uint8_t *stage, uint4 *dst, uint32_t t,
                                              int lane, const float2 (&rc)[4], const float2 (&rs)[4]) {
    const int cpr = a.d / 8, half = cpr / 2;
    const int hshift = a.d == 128 ? 3 : 2;
    const int npairs = a.H * half;
    const int chl = lane & (half - 1);
    const uint32_t T = uint32_t(a.T);
    const uint32_t code_bytes = uint32_t(a.H) * uint32_t(a.d) * uint32_t(B) / 8u;
    const uint32_t *par = reinterpret_cast<const uint32_t *>(stage + code_bytes);
    for (int p0 = 0; p0 < npairs; p0 += 2 * 32) {
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int p = p0 + it * 32 + lane;
        if (p >= npairs) break;
        const int h = p >> hshift;
        const int ca = h * cpr + chl, cb = ca + half;
        float ya[8], yb[8];
        if (B == 16) {
            const uint4 ra = reinterpret_cast<const uint4 *>(stage)[ca], rb = reinterpret_cast<const uint4 *>(stage)[cb];
            const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                ya[2 * e] = bf16_lo(wa[e]);
                ya[2 * e + 1] = bf16_hi(wa[e]);
                yb[2 * e] = bf16_lo(wb[e]);
                yb[2 * e + 1] = bf16_hi(wb[e]);
            }
        } else {
            card_chunk_values(B, card_chunk_codes(B, stage, ca), par[ca >> 2], ya);
            card_chunk_values(B, card_chunk_codes(B, stage, cb), par[cb >> 2], yb);
        }
        // oa = ya cos - yb sin, ob = ya sin + yb cos: one product rounded, then one fma
        float oa[8], ob[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 xa = make_float2(ya[2 * e], ya[2 * e + 1]), xb = make_float2(yb[2 * e], yb[2 * e + 1]);
            const float2 ta = __fmul2_rn(xb, rs[e]), tb = __fmul2_rn(xb, rc[e]);
            const float2 u = __ffma2_rn(xa, rc[e], make_float2(-ta.x, -ta.y));
            const float2 w = __ffma2_rn(xa, rs[e], tb);
            oa[2 * e] = u.x, oa[2 * e + 1] = u.y;
            ob[2 * e] = w.x, ob[2 * e + 1] = w.y;
        }
        uint4 *row = dst + (uint64_t(h) * T + t) * cpr;
        st_stream_v4(row + chl, pack_bf16x8(oa));
        st_stream_v4(row + chl + half, pack_bf16x8(ob));
      }
    }
}

template <bool ROPE>
__global__ void __launch_bounds__(CARD_THREADS, ROPE ? 4 : 5) card_unpack_staged(const __grid_constant__ CardArgs a,
                                                                        uint32_t stage_bytes) {
    extern __shared__ uint4 s_stage[];  // [warp][2] mbarriers (128 bytes), then [warp][2] buffers
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *base = reinterpret_cast<uint8_t *>(s_stage);
    const uint32_t bar0 = smem_addr(base) + 16u * uint32_t(warp);
    uint8_t *stages = base + 16u * CARD_WARPS + uint32_t(warp) * 2u * stage_bytes;
    const uint32_t st0 = smem_addr(stages);
    if (lane == 0) {
        mbar_init1(bar0);
        mbar_init1(bar0 + 8);
        mbar_init_fence();
    }
    __syncwarp();
    float2 rc[4], rs[4];  // ROPE: (cos, sin) of the lane's 8 frequencies, two per packed register
    if (ROPE) {
        const int chl = lane & (a.d / 16 - 1);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 r0 = a.rot[chl * 8 + 2 * e], r1 = a.rot[chl * 8 + 2 * e + 1];
            rc[e] = make_float2(r0.x, r1.x);
            rs[e] = make_float2(r0.y, r1.y);
        }
    }
    const uint64_t pol = l2_evict_first_policy();  // the card is read once
    const uint32_t w = blockIdx.x * CARD_WARPS + uint32_t(warp);
    const int kv0 = int(w & 1u);
    StagedTask c;  // task k
    c.t = (w >> 1) % uint32_t(a.T);
    c.l = (w >> 1) / uint32_t(a.T);
    staged_load_hdr(a, c);
    staged_check(a, c);
    if (lane == 0 && c.ok) staged_issue(a, c, kv0, st0, bar0, pol);
    StagedTask n = staged_next(a, c);  // task k + 1
    uint32_t phase = 0;                // bit s: parity of buffer s's next phase
    for (uint32_t k = 0; c.l < uint32_t(a.L); ++k) {
        const uint32_t s = k & 1u;
        const int kv = kv0 ^ (ROPE ? int(s) : 0);
        staged_check(a, n);
        if (lane == 0 && n.ok) staged_issue(a, n, kv ^ (ROPE ? 1 : 0), st0 + (s ^ 1u) * stage_bytes, bar0 + 8u * (s ^ 1u), pol);
        const StagedTask nn = staged_next(a, n);  // task k + 2: its header lands during this task
        if (c.ok) {
            const bool ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8u * s, (phase >> s) & 1u, a.wait_polls));
            if (!ok) {
                // give up: record it, let the copies in flight (this buffer's
                // and the other's) land, with the normal limit, and leave
                if (lane == 0) atomicOr(&reinterpret_cast<kvp_card_header *>(a.card)->error, FLAG_TIMEOUT);
                mbar_wait(bar0 + 8u * s, (phase >> s) & 1u, CARD_WAIT_LIMIT);
                if (n.ok) mbar_wait(bar0 + 8u * (s ^ 1u), (phase >> (s ^ 1u)) & 1u, CARD_WAIT_LIMIT);
                return;
            }
            phase ^= 1u << s;
            const uint8_t *stage = stages + s * stage_bytes;
            uint4 *dst = a.dst[kv][c.l];
            if (ROPE && kv == 0) {
                switch (c.b) {
                case 2: rope_staged_b<2>(a, stage, dst, c.t, lane, rc, rs); break;
                case 4: rope_staged_b<4>(a, stage, dst, c.t, lane, rc, rs); break;
                case 8: rope_staged_b<8>(a, stage, dst, c.t, lane, rc, rs); break;
                default: rope_staged_b<16>(a, stage, dst, c.t, lane, rc, rs); break;
                }
            } else {
                switch (c.b) {
                case 2: unpack_staged_b<2>(a, stage, dst, c.t, lane); break;
                case 4: unpack_staged_b<4>(a, stage, dst, c.t, lane); break;
                case 8: unpack_staged_b<8>(a, stage, dst, c.t, lane); break;
                default: unpack_staged_b<16>(a, stage, dst, c.t, lane); break;
                }
            }
        } else if (lane == 0) {
            atomicOr(&reinterpret_cast<kvp_card_header *>(a.card)->error, FLAG_HEADER);
        }
        __syncwarp();  // every lane is done with this buffer before it is refilled
        c = n;
        n = nn;
    }
}

// Dynamic shared memory above the default 48 KB is opted into once per device
// and kernel, for the largest size asked so far.
template <bool ROPE>
static bool unpack_smem_ready(size_t smem) {
    if (smem <= 48u * 1024u) return true;
    static size_t done[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return false;
    }
    if (done[dev] >= smem) return true;
    if (cudaFuncSetAttribute(card_unpack_staged<ROPE>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
        cudaSuccess) {
        (void)cudaGetLastError();  // leave no sticky error for the next call to report
        return false;
    }
    done[dev] = smem;
    return true;
}

// The (token, layer) step of a warp's staged-unpack tasks for a grid of
// `grid` blocks: half the grid's warp count, in tokens.
static void set_unpack_steps(CardArgs &a, int grid) {
    const uint32_t dlt = uint32_t(grid) * uint32_t(CARD_WARPS / 2);
    a.it_dt = dlt % uint32_t(a.T);
    a.it_dl = dlt / uint32_t(a.T);
}

// Bytes of one staging buffer (the largest half-record, 2 H d bytes) when the
// staged unpack applies to the shape, else 0: the block's buffers fit 96 KB
// (above 48 KB by opt-in; SmolLM2-1.7B's H d = 2048 takes 64 KB and unpacks
// in 0.080 against 0.085 ms direct).
static uint32_t unpack_stage_bytes(const CardArgs &a) {
    const uint64_t hd = uint64_t(a.H) * uint64_t(a.d);
    if (a.d != 128 && (a.H & 1)) return 0;  // V group parameters would start 8 bytes off a 16-byte boundary
    if (16u * CARD_WARPS + uint64_t(CARD_WARPS) * 2u * 2u * hd > 96u * 1024u) return 0;
    return uint32_t(2u * hd);
}

template <typename K>
static int card_grid(K kernel, uint64_t tasks, int waves, size_t smem = 0) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, CARD_THREADS, smem) != cudaSuccess || occ < 1)
        occ = 1;
    const uint64_t want = (tasks + CARD_WARPS - 1) / CARD_WARPS;
    const uint64_t cap = uint64_t(sm_count()) * uint64_t(occ) * uint64_t(waves);
    return int(want < cap ? (want < 1 ? 1 : want) : cap);
}

}  // namespace kvp

using namespace kvp;

extern "C" int cachecard_pack(const kvp_shape *s, uint64_t model_id, int64_t pos_offset, const uint8_t *bits_dev,
                              const void *const *k_layers, const void *const *v_layers, void *card, size_t card_bytes,
                              void *stream) {
    int rc = shape_ok(s);
    if (rc != KVP_OK) return rc;
    if (!bits_dev || !k_layers || !v_layers || !card) return KVP_ERR_ARG;
    const int L = s->n_layers;
    for (int l = 0; l < L; ++l) {
        if (!k_layers[l] || !v_layers[l]) return KVP_ERR_ARG;
        if (!aligned(k_layers[l], 16) || !aligned(v_layers[l], 16)) return KVP_ERR_ALIGN;
    }
    if (!aligned(card, 256)) return KVP_ERR_ALIGN;
    // the header, bits and offsets must fit whatever the bitwidths are
    if (card_bytes < card_off_layers(s->n_tokens)) return KVP_ERR_SIZE;
    // record offsets are 32-bit: the largest possible layer must fit
    if (uint64_t(s->n_tokens) * card_record_bytes(16, s->n_kv_heads, s->head_dim) >= (1ull << 32)) return KVP_ERR_SIZE;
    // (layer, token, K|V) tasks are counted in 32 bits
    if (uint64_t(s->n_layers) * uint64_t(s->n_tokens) * 2ull >= (1ull << 32)) return KVP_ERR_SIZE;

    CardArgs a;
    for (int l = 0; l < L; ++l) {
        a.src[0][l] = static_cast<const uint4 *>(k_layers[l]);
        a.src[1][l] = static_cast<const uint4 *>(v_layers[l]);
    }
    a.card = static_cast<uint8_t *>(card);
    a.bits_dev = bits_dev;
    a.card_bytes = card_bytes;
    a.model_id = model_id;
    a.pos_offset = pos_offset;
    a.L = L;
    a.H = s->n_kv_heads;
    a.T = s->n_tokens;
    a.d = s->head_dim;
    a.off_offsets = card_off_offsets(a.T);
    a.off_layers = card_off_layers(a.T);
    a.layer_stride = 0;  // depends on device-resident bits: kernels read it from the header
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    card_scan<<<1, SCAN_THREADS, 0, st>>>(a);
    const uint64_t tasks = uint64_t(L) * uint64_t(a.T) * 2u;
    // 64 registers (4 blocks/SM) and two resident grids' worth of blocks: more
    // loads in flight for this latency-bound kernel (measured 0.185 -> 0.176 ms
    // on the 4K-token Llama-3-8B step; 5 blocks/SM is slower)
    if ((s->n_kv_heads * (s->head_dim / 32)) % 32 == 0)
        card_pack<true><<<card_grid(card_pack<true>, tasks, 2), CARD_THREADS, 0, st>>>(a);
    else
        card_pack<false><<<card_grid(card_pack<false>, tasks, 2), CARD_THREADS, 0, st>>>(a);
    card_zero_tails<<<L, CARD_THREADS, 0, st>>>(a);
    count_launch(3);
    return launch_status();
}

// Failure-path testing (kvp_test_limit_next_unpack): consumed by the next
// unpack call on the calling thread.
static thread_local uint32_t t_unpack_polls = CARD_WAIT_LIMIT;

// Host checks and launch arguments shared by both unpack entry points.
static int unpack_setup(const void *card, const kvp_card_header *hdr, void *const *k_dst, void *const *v_dst,
                        CardArgs &a) {
    if (!card || !hdr || !k_dst || !v_dst) return KVP_ERR_ARG;
    if (hdr->magic != CARD_MAGIC || hdr->version != CARD_VERSION || hdr->group_size != CARD_GROUP || hdr->dtype != 1)
        return KVP_ERR_HEADER;
    kvp_shape s = {hdr->n_layers, hdr->n_kv_heads, hdr->head_dim, hdr->seq_len};
    int rc = shape_ok(&s);
    if (rc != KVP_OK) return rc == KVP_ERR_ARG ? KVP_ERR_HEADER : rc;
    if (hdr->error & (FLAG_BITS | FLAG_SIZE)) return KVP_ERR_HEADER;
    if (hdr->off_offsets != card_off_offsets(s.n_tokens) || hdr->off_layers != card_off_layers(s.n_tokens) ||
        hdr->off_bits != CARD_HEADER_BYTES || (hdr->layer_stride & 255u) != 0 ||
        hdr->total_bytes != hdr->off_layers + uint64_t(s.n_layers) * hdr->layer_stride)
        return KVP_ERR_HEADER;
    if (!aligned(card, 256)) return KVP_ERR_ALIGN;
    if (uint64_t(s.n_layers) * uint64_t(s.n_tokens) * 2ull >= (1ull << 32)) return KVP_ERR_SIZE;
    const int L = s.n_layers;
    for (int l = 0; l < L; ++l) {
        if (!k_dst[l] || !v_dst[l]) return KVP_ERR_ARG;
        if (!aligned(k_dst[l], 16) || !aligned(v_dst[l], 16)) return KVP_ERR_ALIGN;
        a.dst[0][l] = static_cast<uint4 *>(k_dst[l]);
        a.dst[1][l] = static_cast<uint4 *>(v_dst[l]);
    }
    a.card = static_cast<uint8_t *>(const_cast<void *>(card));
    a.bits_dev = nullptr;
    a.card_bytes = hdr->total_bytes;
    a.model_id = hdr->model_id;
    a.pos_offset = hdr->pos_offset;
    a.off_offsets = hdr->off_offsets;
    a.off_layers = hdr->off_layers;
    a.layer_stride = hdr->layer_stride;
    a.L = L;
    a.H = s.n_kv_heads;
    a.T = s.n_tokens;
    a.d = s.head_dim;
    a.shift = 0;
    a.wait_polls = t_unpack_polls;
    t_unpack_polls = CARD_WAIT_LIMIT;
    return KVP_OK;
}

extern "C" int cachecard_unpack(const void *card, const kvp_card_header *hdr, void *const *k_dst, void *const *v_dst,
                                void *stream) {
    CardArgs a;
    const int rc = unpack_setup(card, hdr, k_dst, v_dst, a);
    if (rc != KVP_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint64_t tasks = uint64_t(a.L) * uint64_t(a.T) * 2u;
    // store-heavy: several resident grids' worth of blocks spread the
    // concurrent stores (as in the pool decoder)
    const uint32_t sb = unpack_stage_bytes(a);
    if (sb) {
        const size_t smem = 16u * CARD_WARPS + size_t(CARD_WARPS) * 2u * sb;
        // eight resident grids' worth of blocks: 4K-token step unpack 0.117 ms
        // against 0.121 (three) and 0.119 (six); 8K-token card 0.231 against 0.242
        if (!unpack_smem_ready<false>(smem)) return KVP_ERR_CUDA;
        const int grid = card_grid(card_unpack_staged<false>, tasks, 8, smem);
        set_unpack_steps(a, grid);
        card_unpack_staged<false><<<grid, CARD_THREADS, smem, st>>>(a, sb);
    } else {
        card_unpack<<<card_grid(card_unpack, tasks, 3), CARD_THREADS, 0, st>>>(a);
    }
    count_launch(1);
    return launch_status();
}

extern "C" int cachecard_unpack_at(const void *card, const kvp_card_header *hdr, int64_t pos_dst,
                                   const float *inv_freq, void *const *k_dst, void *const *v_dst, void *stream) {
    if (!inv_freq) return KVP_ERR_ARG;
    CardArgs a;
    const int rc = unpack_setup(card, hdr, k_dst, v_dst, a);
    if (rc != KVP_OK) return rc;
    if (__builtin_sub_overflow(pos_dst, hdr->pos_offset, &a.shift)) return KVP_ERR_ARG;
    for (int i = 0; i < a.d / 2; ++i) {
        if (!std::isfinite(inv_freq[i])) return KVP_ERR_ARG;
        const double ang = double(a.shift) * double(inv_freq[i]);
        a.rot[i] = make_float2(float(std::cos(ang)), float(std::sin(ang)));
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint64_t tasks = uint64_t(a.L) * uint64_t(a.T) * 2u;
    const uint32_t sb = unpack_stage_bytes(a);
    if (sb) {
        const size_t smem = 16u * CARD_WARPS + size_t(CARD_WARPS) * 2u * sb;
        // four resident grids' worth of blocks (8K-token card: 0.250 ms; one, two,
        // three, six, eight and twelve: 0.267, 0.257, 0.251, 0.251, 0.253, 0.258)
        if (!unpack_smem_ready<true>(smem)) return KVP_ERR_CUDA;
        const int grid = card_grid(card_unpack_staged<true>, tasks, 4, smem);
        set_unpack_steps(a, grid);
        card_unpack_staged<true><<<grid, CARD_THREADS, smem, st>>>(a, sb);
    } else {
        card_unpack_rope<<<card_grid(card_unpack_rope, tasks, 3), CARD_THREADS, 0, st>>>(a);
    }
    count_launch(1);
    return launch_status();
}

extern "C" int kvp_test_limit_next_unpack(uint32_t polls) {
    t_unpack_polls = polls;
    return KVP_OK;
}
