// kvpool_attend.cu -- attention of N agents' queries over one layer of a
// SharedKVPool without materialising any cache: the fused attention over the
// quantized cache that "QKVShare: Quantized KV-Cache Handoff for Multi-Agent
// On-Device LLMs" defers (Significance), applied to "PolyKV" 2.A's shared
// pool: one read of the compressed layer serves every agent.
//
// For agent a, query head j (GQA: KV head h = j / (n_q_heads / H)):
//   s_t = scale * s_l * (q . kq_t)          kq_t: the int8 key codes
//   out = sum_t p_t v_t,  p = softmax(s),   lse = log sum_t exp(s_t)
//   v_t = sigma_t * (H_d c_t) / sqrt(d)  =>  out = H_d (sum_t p_t sigma_t c_t) / sqrt(d)
// so values are accumulated in the rotated domain and transformed once per
// query at the end.
//
// attend_split: one block per (KV head, token split); the split's 64-token
// sub-chunks are staged in shared memory (keys as exact bf16 integers,
// centroids as fp16 hi + lo parts, transposed), and two warp-level tensor-core
// products run per sub-chunk: S = Q K^T (bf16 in, fp32 accumulate: exact
// products) and A += P' C (P' = p * sigma in fp16; C = C_hi + C_lo), with an
// online softmax across sub-chunks.  attend_combine merges the splits
// (log-sum-exp), applies the inverse transform and writes out / lse.
#include "kvp_vec.cuh"

namespace kvp {

constexpr int ATT_THREADS = 256;
constexpr int ATT_TC = 64;  // tokens per sub-chunk
constexpr int ATT_MT = 64;  // query rows per tile
constexpr int ATT_TARGET_BLOCKS = 304;

struct AttendArgs {
    const uint8_t *pool;
    const uint16_t *q;  // bf16 [NA][NQ][d]
    float *out;         // [NA][NQ][d]
    float *lse;         // [NA][NQ]
    float *part;        // [H][nsplit][QHP][d] rotated-domain partial sums
    float2 *stats;      // [H][nsplit][QHP]: (running max, running sum)
    PoolGeom geo;
    float scale;
    int L, H, T, layer, NA, NQ, G, QH, QHP, nsub, per_split, nsplit;
};

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int D>
struct AttendSmem {
    static constexpr int KW = D / 2 + 4;       // 32-bit words per Q / K row (padded: conflict-free fragments)
    static constexpr int CW = ATT_TC / 2 + 4;  // words per P / C row
    static constexpr size_t words = size_t(ATT_MT) * KW + size_t(ATT_TC) * KW + size_t(ATT_MT) * CW +
                                    2 * size_t(D) * CW + ATT_TC + 4 * ATT_MT + 2 * ATT_MT;
    static constexpr size_t bytes = words * 4 + 16 * 4;  // + the centroid table
};

template <int D>
__global__ void __launch_bounds__(ATT_THREADS, 2) attend_split(const __grid_constant__ AttendArgs a) {
    using SM = AttendSmem<D>;
    constexpr int KW = SM::KW, CW = SM::CW;
    constexpr int NT_S = 32 / 8;         // S: a warp covers 32 tokens (4 n8 tiles)
    constexpr int NT_V = D / 2 / 8;      // PV: a warp covers D/2 dims
    extern __shared__ __align__(16) uint32_t smem[];
    uint32_t *Qs = smem;                  // [ATT_MT][KW]  bf16 pairs
    uint32_t *Kb = Qs + ATT_MT * KW;      // [ATT_TC][KW]  bf16 pairs
    uint32_t *Ps = Kb + ATT_TC * KW;      // [ATT_MT][CW]  fp16 pairs
    uint32_t *Ch = Ps + ATT_MT * CW;      // [D][CW]       fp16 pairs, token-contiguous
    uint32_t *Cl = Ch + D * CW;           // [D][CW]
    float *sig = reinterpret_cast<float *>(Cl + D * CW);  // [ATT_TC]
    float *rmax = sig + ATT_TC;           // [2][ATT_MT] per-half row maxima
    float *rsum = rmax + 2 * ATT_MT;      // [2][ATT_MT] per-half row sums
    float *row_m = rsum + 2 * ATT_MT;     // [ATT_MT] running max
    float *row_l = row_m + ATT_MT;        // [ATT_MT] running sum
    __half2 *ctab = reinterpret_cast<__half2 *>(row_l + ATT_MT);  // [8] (hi, lo) per code

    const int h = blockIdx.x, split = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int mi = warp & 3, nh = warp >> 2;  // m16 tile; half (tokens for S, dims for PV)
    const int r0 = mi * 16;
    const uint8_t *lay = a.pool + a.geo.off_layers + uint64_t(a.layer) * a.geo.layer_stride;
    const float qk = a.scale * reinterpret_cast<const float *>(a.pool + a.geo.off_scales)[a.layer];
    const uint64_t vbase = uint64_t(h) * uint64_t(a.T);  // first vector of this KV head
    const int sub0 = split * a.per_split, sub1 = min(a.nsub, sub0 + a.per_split);

    if (tid < 8) {  // centroids as fp16 hi + lo parts: c = hi + lo to ~2^-22 relative
        const float c = centroid_e4(uint32_t(tid)) * 1e-4f;
        const __half hi = __float2half_rn(c);
        ctab[tid] = __halves2half2(hi, __float2half_rn(c - __half2float(hi)));
    }

    for (int m0 = 0; m0 < a.QH; m0 += ATT_MT) {
        __syncthreads();
        // query rows m0..m0+63 of this KV head: agent r / G, head h*G + r % G
        for (int e = tid; e < ATT_MT * (D / 8); e += ATT_THREADS) {
            const int r = e / (D / 8), c8 = e % (D / 8);
            uint4 v = make_uint4(0, 0, 0, 0);
            if (m0 + r < a.QH) {
                const int ag = (m0 + r) / a.G, j = h * a.G + (m0 + r) % a.G;
                v = *reinterpret_cast<const uint4 *>(a.q + (uint64_t(ag) * a.NQ + j) * D + c8 * 8);
            }
            *reinterpret_cast<uint4 *>(Qs + r * KW + c8 * 4) = v;
        }
        if (tid < ATT_MT) {
            row_m[tid] = -INFINITY;
            row_l[tid] = 0.0f;
        }
        float acc[NT_V][4];
#pragma unroll
        for (int nt = 0; nt < NT_V; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;

        for (int sub = sub0; sub < sub1; ++sub) {
            const int t0 = sub * ATT_TC;
            __syncthreads();  // (1) the previous sub-chunk's tiles and statistics are settled
            {   // keys: int8 codes -> exact bf16 (|q| <= 127: at most 7 significant bits)
                const int t = tid >> 2, part = tid & 3;  // 64 tokens x 4 quarters of d
                constexpr int DQ = D / 4;                // codes per quarter (32 or 16)
                uint32_t wds[DQ / 4];
                if (t0 + t < a.T) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(lay + (vbase + t0 + t) * D + part * DQ);
#pragma unroll
                    for (int u = 0; u < DQ / 16; ++u) {
                        const uint4 w = ld_stream_v4(src + u);
                        wds[4 * u] = w.x;
                        wds[4 * u + 1] = w.y;
                        wds[4 * u + 2] = w.z;
                        wds[4 * u + 3] = w.w;
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < DQ / 4; ++u) wds[u] = 0u;  // codes 0 (scores are masked anyway)
                }
                uint32_t *row = Kb + t * KW + part * (DQ / 2);
#pragma unroll
                for (int u = 0; u < DQ / 4; ++u) {
                    const uint32_t x = wds[u] ^ 0x80808080u;
                    float f[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        f[i] = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7650u | i)) - 8388736.0f;
                    row[2 * u] = __byte_perm(__float_as_uint(f[0]), __float_as_uint(f[1]), 0x7632u);
                    row[2 * u + 1] = __byte_perm(__float_as_uint(f[2]), __float_as_uint(f[3]), 0x7632u);
                }
            }
            // values: 3-bit codes -> centroid hi / lo, transposed [dim][token]; each
            // work item is 32 codes (12 bytes) of one token
            for (int e = tid; e < ATT_TC * (D / 32); e += ATT_THREADS) {
                const int t = e & (ATT_TC - 1), ig = e / ATT_TC;
                const bool ok = t0 + t < a.T;
                uint32_t w[4];
#pragma unroll
                for (int u = 0; u < 3; ++u)
                    w[u] = ok ? ld_stream_u32(lay + a.geo.sec_v + (vbase + t0 + t) * (3 * D / 8) + ig * 12 + 4 * u)
                              : 0u;
                w[3] = 0u;
                __half *chh = reinterpret_cast<__half *>(Ch), *cll = reinterpret_cast<__half *>(Cl);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int bit = 3 * c, wi = bit >> 5, sh = bit & 31;
                    uint32_t code = w[wi] >> sh;
                    if (sh > 29) code |= w[wi + 1] << (32 - sh);
                    const __half2 cv = ctab[code & 7u];
                    const int dim = ig * 32 + c;
                    chh[dim * (2 * CW) + t] = ok ? __low2half(cv) : __float2half_rn(0.0f);
                    cll[dim * (2 * CW) + t] = ok ? __high2half(cv) : __float2half_rn(0.0f);
                }
            }
            if (tid < ATT_TC)
                sig[tid] = (t0 + tid < a.T) ? __half2float(__ushort_as_half(reinterpret_cast<const uint16_t *>(
                                                  lay + a.geo.sec_sigma)[vbase + t0 + tid]))
                                            : 0.0f;
            __syncthreads();  // (2) tiles staged

            // S = Q K^T: rows r0.., tokens nh*32..
            float s[NT_S][4];
#pragma unroll
            for (int nt = 0; nt < NT_S; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.0f;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const int kw = ks * 8;
                const uint32_t a0 = Qs[(r0 + g) * KW + kw + tig], a1 = Qs[(r0 + g + 8) * KW + kw + tig];
                const uint32_t a2 = Qs[(r0 + g) * KW + kw + tig + 4], a3 = Qs[(r0 + g + 8) * KW + kw + tig + 4];
#pragma unroll
                for (int nt = 0; nt < NT_S; ++nt) {
                    const int n0 = nh * 32 + nt * 8;
                    mma_bf16(s[nt], a0, a1, a2, a3, Kb[(n0 + g) * KW + kw + tig], Kb[(n0 + g) * KW + kw + tig + 4]);
                }
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < NT_S; ++nt) {
                const int tk = t0 + nh * 32 + nt * 8 + 2 * tig;
                s[nt][0] = tk < a.T ? s[nt][0] * qk : -INFINITY;
                s[nt][1] = tk + 1 < a.T ? s[nt][1] * qk : -INFINITY;
                s[nt][2] = tk < a.T ? s[nt][2] * qk : -INFINITY;
                s[nt][3] = tk + 1 < a.T ? s[nt][3] * qk : -INFINITY;
                mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
                mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
            }
#pragma unroll
            for (int m = 1; m < 4; m <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, m));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, m));
            }
            if (tig == 0) {
                rmax[nh * ATT_MT + r0 + g] = mx0;
                rmax[nh * ATT_MT + r0 + g + 8] = mx1;
            }
            __syncthreads();  // (3) both halves' maxima in

            // new running max of the warp's two rows (every sub-chunk has a valid token)
            const float om0 = row_m[r0 + g], om1 = row_m[r0 + g + 8];
            const float nm0 = fmaxf(om0, fmaxf(rmax[r0 + g], rmax[ATT_MT + r0 + g]));
            const float nm1 = fmaxf(om1, fmaxf(rmax[r0 + g + 8], rmax[ATT_MT + r0 + g + 8]));
            float sm0 = 0.0f, sm1 = 0.0f;
#pragma unroll
            for (int nt = 0; nt < NT_S; ++nt) {
                const int tl = nh * 32 + nt * 8 + 2 * tig;
                const float p0 = __expf(s[nt][0] - nm0), p1 = __expf(s[nt][1] - nm0);
                const float p2 = __expf(s[nt][2] - nm1), p3 = __expf(s[nt][3] - nm1);
                sm0 += p0 + p1;
                sm1 += p2 + p3;
                const __half2 u = __floats2half2_rn(p0 * sig[tl], p1 * sig[tl + 1]);
                const __half2 v = __floats2half2_rn(p2 * sig[tl], p3 * sig[tl + 1]);
                Ps[(r0 + g) * CW + tl / 2] = *reinterpret_cast<const uint32_t *>(&u);
                Ps[(r0 + g + 8) * CW + tl / 2] = *reinterpret_cast<const uint32_t *>(&v);
            }
#pragma unroll
            for (int m = 1; m < 4; m <<= 1) {
                sm0 += __shfl_xor_sync(0xffffffffu, sm0, m);
                sm1 += __shfl_xor_sync(0xffffffffu, sm1, m);
            }
            if (tig == 0) {
                rsum[nh * ATT_MT + r0 + g] = sm0;
                rsum[nh * ATT_MT + r0 + g + 8] = sm1;
            }
            __syncthreads();  // (4) P' and the partial sums in

            // rescale to the new max, then A += P' (C_hi + C_lo): rows r0.., dims nh*D/2..
            const float al0 = __expf(om0 - nm0), al1 = __expf(om1 - nm1);  // 0 on the first sub-chunk
#pragma unroll
            for (int nt = 0; nt < NT_V; ++nt) {
                acc[nt][0] *= al0;
                acc[nt][1] *= al0;
                acc[nt][2] *= al1;
                acc[nt][3] *= al1;
            }
#pragma unroll
            for (int ks = 0; ks < ATT_TC / 16; ++ks) {
                const int kw = ks * 8;
                const uint32_t a0 = Ps[(r0 + g) * CW + kw + tig], a1 = Ps[(r0 + g + 8) * CW + kw + tig];
                const uint32_t a2 = Ps[(r0 + g) * CW + kw + tig + 4], a3 = Ps[(r0 + g + 8) * CW + kw + tig + 4];
#pragma unroll
                for (int nt = 0; nt < NT_V; ++nt) {
                    const int n0 = nh * (D / 2) + nt * 8;
                    mma_f16(acc[nt], a0, a1, a2, a3, Ch[(n0 + g) * CW + kw + tig], Ch[(n0 + g) * CW + kw + tig + 4]);
                    mma_f16(acc[nt], a0, a1, a2, a3, Cl[(n0 + g) * CW + kw + tig], Cl[(n0 + g) * CW + kw + tig + 4]);
                }
            }
            __syncthreads();  // (5) every warp has read the old statistics and P'
            if (tid < ATT_MT) {
                const float om = row_m[tid];
                const float nm = fmaxf(om, fmaxf(rmax[tid], rmax[ATT_MT + tid]));
                row_l[tid] = row_l[tid] * __expf(om - nm) + rsum[tid] + rsum[ATT_MT + tid];
                row_m[tid] = nm;
            }
        }
        __syncthreads();
        // this split's partial sums and statistics for the tile's real rows
        const uint64_t pbase = (uint64_t(h) * a.nsplit + split) * uint64_t(a.QHP);
#pragma unroll
        for (int nt = 0; nt < NT_V; ++nt) {
            const int dim = nh * (D / 2) + nt * 8 + 2 * tig;
            const int ra = m0 + r0 + g, rb = ra + 8;
            if (ra < a.QH)
                *reinterpret_cast<float2 *>(a.part + (pbase + ra) * D + dim) = make_float2(acc[nt][0], acc[nt][1]);
            if (rb < a.QH)
                *reinterpret_cast<float2 *>(a.part + (pbase + rb) * D + dim) = make_float2(acc[nt][2], acc[nt][3]);
        }
        if (tid < ATT_MT && m0 + tid < a.QH) a.stats[pbase + m0 + tid] = make_float2(row_m[tid], row_l[tid]);
    }
}

// One warp per (agent, query head): merge the splits, inverse transform.
template <int D>
__global__ void __launch_bounds__(256) attend_combine(const __grid_constant__ AttendArgs a) {
    constexpr int PL = D / 32;  // dims per lane, indices lane*PL + e
    const int wq = int((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
    if (wq >= a.NA * a.NQ) return;
    const int ag = wq / a.NQ, j = wq % a.NQ;
    const int h = j / a.G, r = ag * a.G + j % a.G;
    float m = -INFINITY, l = 0.0f, acc[PL];
#pragma unroll
    for (int e = 0; e < PL; ++e) acc[e] = 0.0f;
    for (int sp = 0; sp < a.nsplit; ++sp) {
        const uint64_t row = (uint64_t(h) * a.nsplit + sp) * uint64_t(a.QHP) + r;
        const float2 st = a.stats[row];
        const float nm = fmaxf(m, st.x);
        const float a1 = __expf(m - nm), a2 = __expf(st.x - nm);
        l = l * a1 + st.y * a2;
        const float *pp = a.part + row * D + lane * PL;
#pragma unroll
        for (int e = 0; e < PL; ++e) acc[e] = acc[e] * a1 + pp[e] * a2;
        m = nm;
    }
    // unnormalised Walsh-Hadamard transform over d: register bits, then lane bits
#pragma unroll
    for (int hb = 1; hb < PL; hb <<= 1)
#pragma unroll
        for (int e = 0; e < PL; ++e)
            if ((e & hb) == 0) {
                const float p = acc[e], q = acc[e + hb];
                acc[e] = p + q;
                acc[e + hb] = p - q;
            }
#pragma unroll
    for (int mb = 1; mb < 32; mb <<= 1) {
        const float sg = (lane & mb) ? -1.0f : 1.0f;
#pragma unroll
        for (int e = 0; e < PL; ++e) acc[e] = fmaf(sg, acc[e], __shfl_xor_sync(0xffffffffu, acc[e], mb));
    }
    const float f = (D == 128 ? 0.08838834764831845f : 0.125f) / l;  // 1/sqrt(d) / l
    float *o = a.out + (uint64_t(ag) * a.NQ + j) * D + lane * PL;
#pragma unroll
    for (int e = 0; e < PL; ++e) o[e] = acc[e] * f;
    if (lane == 0) a.lse[uint64_t(ag) * a.NQ + j] = m + __logf(l);
}

// The split kernel's dynamic shared memory exceeds the default 48 KB: raise
// the limit once per device (the first call on a device does it).
template <int D>
static bool attend_smem_ready() {
    static bool done[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (!done[dev]) {
        if (cudaFuncSetAttribute(attend_split<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(AttendSmem<D>::bytes)) != cudaSuccess)
            return false;
        done[dev] = true;
    }
    return true;
}

struct AttendPlan {
    int G, QH, QHP, nsub, per_split, nsplit;
    uint64_t part_off, stats_off, total;
};

static inline AttendPlan attend_plan(const kvp_shape *s, int na, int nq) {
    AttendPlan p;
    p.G = nq / s->n_kv_heads;
    p.QH = na * p.G;
    p.QHP = (p.QH + ATT_MT - 1) / ATT_MT * ATT_MT;
    p.nsub = (s->n_tokens + ATT_TC - 1) / ATT_TC;
    int want = (ATT_TARGET_BLOCKS + s->n_kv_heads - 1) / s->n_kv_heads;
    if (want < 1) want = 1;
    if (want > p.nsub) want = p.nsub;
    p.per_split = (p.nsub + want - 1) / want;
    p.nsplit = (p.nsub + p.per_split - 1) / p.per_split;
    const uint64_t rows = uint64_t(s->n_kv_heads) * uint64_t(p.nsplit) * uint64_t(p.QHP);
    p.part_off = 0;
    p.stats_off = align256(rows * uint64_t(s->head_dim) * 4u);
    p.total = align256(p.stats_off + rows * 8u);
    return p;
}

}  // namespace kvp

using namespace kvp;

extern "C" size_t kvpool_attend_workspace_bytes(const kvp_shape *s, int n_agents, int n_q_heads) {
    if (shape_ok(s) != KVP_OK || n_agents < 1 || n_q_heads < 1 || n_q_heads % s->n_kv_heads != 0) return 0;
    return size_t(attend_plan(s, n_agents, n_q_heads).total);
}

extern "C" int kvpool_attend(const void *pool, const kvp_shape *s, int layer, int n_agents, int n_q_heads,
                             const void *q, float scale, float *out, float *lse, void *ws, size_t ws_bytes,
                             void *stream) {
    int rc = shape_ok(s);
    if (rc != KVP_OK) return rc;
    if (!pool || !q || !out || !lse || !ws) return KVP_ERR_ARG;
    if (layer < 0 || layer >= s->n_layers || n_agents < 1 || n_q_heads < 1 || n_q_heads % s->n_kv_heads != 0)
        return KVP_ERR_ARG;
    if (uint64_t(n_agents) * uint64_t(n_q_heads) >= (1ull << 24)) return KVP_ERR_SIZE;
    if (!aligned(pool, 256) || !aligned(q, 16) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(ws, 16))
        return KVP_ERR_ALIGN;
    const AttendPlan p = attend_plan(s, n_agents, n_q_heads);
    if (ws_bytes < p.total) return KVP_ERR_SIZE;
    AttendArgs a;
    a.pool = static_cast<const uint8_t *>(pool);
    a.q = static_cast<const uint16_t *>(q);
    a.out = out;
    a.lse = lse;
    a.part = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + p.part_off);
    a.stats = reinterpret_cast<float2 *>(static_cast<uint8_t *>(ws) + p.stats_off);
    a.geo = pool_geom(s->n_layers, s->n_kv_heads, s->head_dim, s->n_tokens);
    a.scale = scale;
    a.L = s->n_layers;
    a.H = s->n_kv_heads;
    a.T = s->n_tokens;
    a.layer = layer;
    a.NA = n_agents;
    a.NQ = n_q_heads;
    a.G = p.G;
    a.QH = p.QH;
    a.QHP = p.QHP;
    a.nsub = p.nsub;
    a.per_split = p.per_split;
    a.nsplit = p.nsplit;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const dim3 grid(unsigned(a.H), unsigned(a.nsplit));
    const unsigned cgrid = unsigned((uint64_t(n_agents) * n_q_heads * 32 + 255) / 256);
    if (s->head_dim == 128) {
        if (!attend_smem_ready<128>()) return KVP_ERR_CUDA;
        attend_split<128><<<grid, ATT_THREADS, AttendSmem<128>::bytes, st>>>(a);
        attend_combine<128><<<cgrid, 256, 0, st>>>(a);
    } else {
        if (!attend_smem_ready<64>()) return KVP_ERR_CUDA;
        attend_split<64><<<grid, ATT_THREADS, AttendSmem<64>::bytes, st>>>(a);
        attend_combine<64><<<cgrid, 256, 0, st>>>(a);
    }
    count_launch(2);
    return launch_status();
}
