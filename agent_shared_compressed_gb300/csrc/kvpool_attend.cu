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
// attend_split: one block per (KV head, token split).  The split's 64-token
// sub-chunks arrive as raw pool bytes in a shared-memory ring that bulk
// copies (the TMA engine) keep up to four sub-chunks ahead; the current one
// is staged from there into tiles (keys as exact bf16 integers, centroids as
// fp16, both [token][dim]) and multiplied.  Warp
// (mi, th) owns query rows mi*16.. and a token slice th of every sub-chunk; it
// runs its own online softmax over that slice with warp-level tensor-core
// products: S = Q K^T (bf16 in, fp32 accumulate: exact products) and
// A += P' C (P' = p * sigma, fp16, kept in registers as the next product's
// A operand).  The warps' states are merged in shared memory at the end.
// attend_combine merges the splits (log-sum-exp), applies the inverse
// transform and writes out / lse.  Exponentials are base 2 throughout.
#include "kvp_async.cuh"
#include "kvp_vec.cuh"

namespace kvp {

constexpr int ATT_THREADS = 256;
constexpr int ATT_WARPS = ATT_THREADS / 32;
constexpr int ATT_TC = 64;  // tokens per sub-chunk
constexpr int ATT_MT = 64;  // query rows per tile (the Q buffer)

struct AttendArgs {
    const uint8_t *pool;
    const uint16_t *q;  // bf16 [NA][NQ][d]
    float *out;         // [NA][NQ][d]
    float *lse;         // [NA][NQ]
    float *part;        // [H][nsplit][QHP][d + R] rotated-domain partial sums (+ P V_lr columns)
    float2 *stats;      // [H][nsplit][QHP]: (running max, running sum), base 2
    PoolGeom geo;
    float scale;
    int L, H, T, layer, NA, NQ, G, QH, QHP, nsub, per_split, nsplit;
    const uint16_t *vlr;     // LoRA attention: bf16 [T][R] shared low-rank value cache
    const uint16_t *lora_b;  // LoRA attention: bf16 [NA][R][H*d] per-agent up-projections
    uint32_t wait_polls;     // polls of a sub-chunk's barrier before giving up
};

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Four 8x8 b16 tiles from shared memory; lane l supplies the row address of
// tile l/8, row l%8.  .trans delivers each tile transposed.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Waits on the bulk-copy ring give up after ATT_WAIT_LIMIT polls (about half
// a second) and report KVP_ERR_TIMEOUT.
constexpr uint32_t ATT_WAIT_LIMIT = 1u << 22;

// Shared memory of the split kernel (bytes).  A ring of NST raw sub-chunks
// (the pool's bytes as they are, filled by bulk copies), then the staged
// tiles of the current sub-chunk: Q, K as exact bf16 integers, values as fp16
// centroids (rows of RW words: 16-byte multiples, conflict-free ldmatrix),
// sigma, the centroid pair table, q8_0 block scales and the low-rank tile.
// After the loop the warps' states are merged from offset BAR_BYTES on.
// PIPE (passes of at most 32 query rows, no low-rank tile): two sets of
// staged tiles, so that a sub-chunk is staged while the one before it is
// multiplied; the ring is two slots deep and the Q tile 32 rows.
template <int D, int R = 0, bool PIPE = false>
struct AttendSmem {
    static constexpr int NST = PIPE ? 2 : (R > 0 ? 3 : 4);  // ring depth
    static constexpr int QROWS = PIPE ? 32 : ATT_MT;        // rows of the Q tile
    static constexpr int RW = D / 2 + 4;       // 32-bit words per Q / K / C row
    static constexpr int LW = R / 2 + 4;       // words per low-rank row (LoRA attention)
    static constexpr int MS = D + R + 8;       // floats per row of a warp's merge slot (conflict-free float2 stores)
    // one raw slot; the V, sigma and block-scale windows start at the 16-byte
    // boundary below their first byte, hence 16 bytes of slack each
    static constexpr uint32_t RAW_K = 0;                                   // [64][D] int8 codes
    static constexpr uint32_t RAW_V = RAW_K + ATT_TC * D;                  // [64][3D/8] code bytes
    static constexpr uint32_t RAW_SG = RAW_V + ATT_TC * 3 * D / 8 + 16;    // [64] fp16 sigma
    static constexpr uint32_t RAW_KS = RAW_SG + ATT_TC * 2 + 16;           // [64][D/32] fp16 block scales
    static constexpr uint32_t RAW_LR = RAW_KS + ATT_TC * (D / 32) * 2 + 16;  // [64][R] bf16 low-rank values
    static constexpr uint32_t SLOT = RAW_LR + ATT_TC * R * 2;
    static constexpr uint32_t BAR_BYTES = 64;
    static constexpr uint32_t OFF_RING = BAR_BYTES;
    static constexpr uint32_t OFF_Q = OFF_RING + NST * SLOT;
    static constexpr uint32_t OFF_K = OFF_Q + QROWS * RW * 4;
    static constexpr uint32_t OFF_C = OFF_K + ATT_TC * RW * 4;
    static constexpr uint32_t OFF_SIG = OFF_C + ATT_TC * RW * 4;
    static constexpr uint32_t OFF_LUT = OFF_SIG + ATT_TC * 4;
    static constexpr uint32_t OFF_KSB = OFF_LUT + 64 * 4;
    static constexpr uint32_t OFF_LS = OFF_KSB + ATT_TC * (D / 32) * 4;
    static constexpr uint32_t END0 = OFF_LS + (R > 0 ? ATT_TC * LW * 4 : 0);
    // PIPE: the second set of staged tiles (the pair table is shared)
    static constexpr uint32_t OFF_K1 = END0;
    static constexpr uint32_t OFF_C1 = OFF_K1 + ATT_TC * RW * 4;
    static constexpr uint32_t OFF_SIG1 = OFF_C1 + ATT_TC * RW * 4;
    static constexpr uint32_t OFF_KSB1 = OFF_SIG1 + ATT_TC * 4;
    static constexpr uint32_t OFF_LS1 = OFF_KSB1 + ATT_TC * (D / 32) * 4;
    static constexpr uint32_t STAGE_END = PIPE ? OFF_LS1 + (R > 0 ? ATT_TC * LW * 4 : 0) : END0;
    static constexpr uint32_t MERGE_END = BAR_BYTES + ATT_WARPS * (16 * MS + 32) * 4;
    static constexpr size_t bytes = STAGE_END > MERGE_END ? STAGE_END : MERGE_END;
    static_assert(SLOT % 16 == 0 && RAW_V % 16 == 0 && RAW_SG % 16 == 0 && RAW_KS % 16 == 0 && RAW_LR % 16 == 0,
                  "bulk-copy destinations are 16-byte aligned");
    static_assert(NST * 8 <= BAR_BYTES, "one mbarrier per slot");
    static_assert(END0 % 16 == 0 && OFF_C1 % 16 == 0, "staged tiles are 16-byte aligned");
};

// The split kernel's shared memory: pipelined for passes of at most 32 query
// rows (TPW = 16) without a low-rank tile.
template <int D, int TPW, int R>
using SplitSmem = AttendSmem<D, R, TPW == 16 && R == 0>;

// Thread 0: the bulk copies of sub-chunk tokens t0 .. t0 + nt - 1 of KV head
// (vbase / T) into one raw slot, completing on its barrier.  Every source is
// a 16-byte aligned run inside its section (sections are 256-byte aligned):
// keys exactly; value codes, sigma and block scales as the 16-byte aligned
// window around their bytes.
template <int D, bool Q8, int R>
__device__ __forceinline__ void issue_chunk(uint8_t *raw, uint32_t bar, const uint8_t *lay, const PoolGeom &geo,
                                            uint64_t vbase, int t0, int T, const uint16_t *kscales,
                                            const uint16_t *vlr) {
    using SM = AttendSmem<D, R>;
    const uint32_t nt = uint32_t(min(ATT_TC, T - t0));
    const uint64_t n0 = vbase + uint64_t(t0);
    const uint8_t *ksrc = lay + n0 * D;
    const uintptr_t v = reinterpret_cast<uintptr_t>(lay + geo.sec_v + n0 * (3 * D / 8));
    const uintptr_t sg = reinterpret_cast<uintptr_t>(lay + geo.sec_sigma + n0 * 2);
    const uint32_t kb = nt * D;
    const uint32_t vb = uint32_t(align16(v + nt * (3 * D / 8)) - (v & ~uintptr_t(15)));
    const uint32_t sb = uint32_t(align16(sg + nt * 2) - (sg & ~uintptr_t(15)));
    uint32_t qb = 0, lb = 0;
    uintptr_t qs = 0;
    if constexpr (Q8) {
        qs = reinterpret_cast<uintptr_t>(kscales + n0 * (D / 32));
        qb = uint32_t(align16(qs + nt * (D / 32) * 2) - (qs & ~uintptr_t(15)));
    }
    if constexpr (R > 0) lb = nt * R * 2;
    mbar_expect_tx(bar, kb + vb + sb + qb + lb);
    bulk_g2s(smem_addr(raw + SM::RAW_K), ksrc, kb, bar);
    bulk_g2s(smem_addr(raw + SM::RAW_V), reinterpret_cast<const void *>(v & ~uintptr_t(15)), vb, bar);
    bulk_g2s(smem_addr(raw + SM::RAW_SG), reinterpret_cast<const void *>(sg & ~uintptr_t(15)), sb, bar);
    if constexpr (Q8)
        bulk_g2s(smem_addr(raw + SM::RAW_KS), reinterpret_cast<const void *>(qs & ~uintptr_t(15)), qb, bar);
    if constexpr (R > 0) bulk_g2s(smem_addr(raw + SM::RAW_LR), vlr + uint64_t(t0) * R, lb, bar);
}

// Raw slot -> staged tiles (whole block): keys int8 -> exact bf16 (|q| <= 127
// has at most 7 significant bits); value codes -> fp16 centroids, two dims
// per word via the pair table.  Tokens at or past T stage as zeros.  Thread
// mapping: the eight lanes of a quarter-warp take eight consecutive tokens;
// for keys each lane starts at a different 16-byte chunk of its token, so
// the raw reads and the tile stores of a quarter-warp both fall on eight
// distinct bank groups (d = 128).  voff / soff / qoff: where the value,
// sigma and block-scale bytes start within their 16-byte aligned windows.
template <int D, bool Q8, int R>
__device__ __forceinline__ void stage_raw(const uint8_t *raw, int t0, int T, int tid, uint32_t voff, uint32_t soff,
                                          uint32_t qoff, uint32_t *Kb, uint32_t *Cs, float *sig, const uint32_t *lut,
                                          float *ksb, uint32_t *Ls) {
    using SM = AttendSmem<D, R>;
    constexpr int RW = SM::RW, VPT = D / 32, CPT = D / 16;
    const int q = tid >> 3, l8 = tid & 7;
    {
        const int tl = l8 + 8 * (q >> 2);
        const bool real = t0 + tl < T;
        uint32_t *row = Kb + tl * RW;
#pragma unroll
        for (int u = 0; u < D / 64; ++u) {
            const int c = ((q & 3) * (D / 64) + u + l8) % CPT;  // 16-byte chunk of the token
            const uint4 w = real ? *reinterpret_cast<const uint4 *>(raw + SM::RAW_K + tl * D + c * 16)
                                 : make_uint4(0, 0, 0, 0);
            const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
            uint32_t o[8];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const uint32_t x = w4[b] ^ 0x80808080u;  // byte i: q + 128
                // 2^23 + q + 128 as fp32, minus 2^23 + 128 (exact), two at a time
                const float2 off = make_float2(-8388736.0f, -8388736.0f);
                const float2 f01 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7650u)),
                                                          __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7651u))), off);
                const float2 f23 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7652u)),
                                                          __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7653u))), off);
                o[2 * b] = __byte_perm(__float_as_uint(f01.x), __float_as_uint(f01.y), 0x7632u);
                o[2 * b + 1] = __byte_perm(__float_as_uint(f23.x), __float_as_uint(f23.y), 0x7632u);
            }
            *reinterpret_cast<uint4 *>(row + 8 * c) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4 *>(row + 8 * c + 4) = make_uint4(o[4], o[5], o[6], o[7]);
        }
    }
    if (q < 8 * VPT) {
        const int tl = l8 + 8 * (q / VPT);
        uint32_t *row = Cs + tl * RW + (q % VPT) * 16;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (t0 + tl < T) {
            const uint32_t *src =
                reinterpret_cast<const uint32_t *>(raw + SM::RAW_V + voff + tl * (3 * D / 8) + (q % VPT) * 12);
            w[0] = src[0];
            w[1] = src[1];
            w[2] = src[2];
        }
        uint32_t o[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {  // codes 2k, 2k+1: bits 6k .. 6k+5
            const int bit = 6 * k, wi = bit >> 5, sh = bit & 31;
            o[k] = lut[__funnelshift_r(w[wi], w[wi + 1], sh) & 63u];
        }
#pragma unroll
        for (int k = 0; k < 16; k += 4) *reinterpret_cast<uint4 *>(row + k) = make_uint4(o[k], o[k + 1], o[k + 2], o[k + 3]);
    }
    if (tid < ATT_TC)
        sig[tid] = t0 + tid < T ? __half2float(*reinterpret_cast<const __half *>(raw + SM::RAW_SG + soff + 2 * tid))
                                : 0.0f;
    if constexpr (Q8)
        if (tid < ATT_TC * (D / 32))
            ksb[tid] = t0 + tid / (D / 32) < T
                           ? __half2float(*reinterpret_cast<const __half *>(raw + SM::RAW_KS + qoff + 2 * tid))
                           : 0.0f;
    if constexpr (R > 0)
        if (tid < ATT_TC * (R / 8)) {  // bf16 -> fp16, exact within fp16's normal range
            uint32_t o[4] = {0u, 0u, 0u, 0u};
            if (t0 + tid / (R / 8) < T) {
                const uint4 x = *reinterpret_cast<const uint4 *>(raw + SM::RAW_LR + 16 * tid);
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) o[i] = pack_half2(bf16_lo(w[i]), bf16_hi(w[i]));
            }
            *reinterpret_cast<uint4 *>(Ls + (tid / (R / 8)) * SM::LW + (tid % (R / 8)) * 4) =
                make_uint4(o[0], o[1], o[2], o[3]);
        }
}

// TPW: tokens of a sub-chunk per warp (32: four 16-row tiles per pass; 16:
// two 16-row tiles per pass, for blocks with at most 32 query rows).
template <int D, int TPW, bool Q8, int R>
__device__ __forceinline__ void attend_passes(const AttendArgs &a, uint32_t *smem, const uint16_t *kscales) {
    using SM = SplitSmem<D, TPW, R>;
    constexpr bool PIPE = TPW == 16 && R == 0;  // sub-chunk i + 1 staged while sub-chunk i is multiplied
    constexpr int RW = SM::RW, MSW = SM::MS;
    constexpr int MS = TPW / 8;       // 16-row tiles per pass
    constexpr int RP = 16 * MS;       // query rows per pass
    constexpr int NS = TPW / 8;       // S n-tiles per warp
    constexpr int NV = D / 8;         // PV n-tiles per warp (all dims)
    constexpr int NL = R / 8;         // P V_lr n-tiles per warp (LoRA attention)
    constexpr int LW = SM::LW;
    constexpr int PW = D + R;         // floats per partial row
    constexpr int NST = SM::NST;
    static_assert(RP <= SM::QROWS, "the Q tile holds a pass's rows");
    uint8_t *sm8 = reinterpret_cast<uint8_t *>(smem);
    const uint32_t bar0 = smem_addr(sm8);                                   // [NST] mbarriers, 8 bytes each
    uint8_t *ring = sm8 + SM::OFF_RING;                                    // [NST] raw sub-chunks
    uint32_t *Qs = reinterpret_cast<uint32_t *>(sm8 + SM::OFF_Q);          // [ATT_MT][RW] bf16 pairs
    uint32_t *Kt = reinterpret_cast<uint32_t *>(sm8 + SM::OFF_K);          // [ATT_TC][RW] bf16 pairs
    uint32_t *Ct = reinterpret_cast<uint32_t *>(sm8 + SM::OFF_C);          // [ATT_TC][RW] fp16 pairs
    float *st = reinterpret_cast<float *>(sm8 + SM::OFF_SIG);              // [ATT_TC] sigma
    uint32_t *lut = reinterpret_cast<uint32_t *>(sm8 + SM::OFF_LUT);       // [64] (c[lo], c[hi]) fp16 pairs
    float *kst = reinterpret_cast<float *>(sm8 + SM::OFF_KSB);             // [ATT_TC][D/32] q8_0 key block scales
    uint32_t *Lt = reinterpret_cast<uint32_t *>(sm8 + SM::OFF_LS);         // [ATT_TC][LW] low-rank fp16 pairs
    // PIPE: the second tile set (never touched otherwise)
    uint32_t *Kt1 = reinterpret_cast<uint32_t *>(sm8 + SM::OFF_K1);
    uint32_t *Ct1 = reinterpret_cast<uint32_t *>(sm8 + SM::OFF_C1);
    float *st1 = reinterpret_cast<float *>(sm8 + SM::OFF_SIG1);
    float *kst1 = reinterpret_cast<float *>(sm8 + SM::OFF_KSB1);
    uint32_t *Lt1 = reinterpret_cast<uint32_t *>(sm8 + SM::OFF_LS1);
    float *mrg = reinterpret_cast<float *>(sm8 + SM::BAR_BYTES);  // after the loop: [warps][16][MSW] acc, [warps][32] m, l

    const int h = blockIdx.x, split = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int mi = warp % MS, th = warp / MS;
    const uint8_t *lay = a.pool + a.geo.off_layers + uint64_t(a.layer) * a.geo.layer_stride;
    // base-2 score scale; q8_0 block scales enter the scores themselves
    const float qk2 = a.scale * 1.4426950408889634f *
                      (Q8 ? 1.0f : reinterpret_cast<const float *>(a.pool + a.geo.off_scales)[a.layer]);
    const uint64_t vbase = uint64_t(h) * uint64_t(a.T);
    const int sub0 = split * a.per_split, sub1 = min(a.nsub, sub0 + a.per_split);
    const int nsubs = sub1 - sub0;
    if (tid == 0) {
        for (int sl = 0; sl < NST; ++sl) mbar_init1(bar0 + 8 * sl);
        mbar_init_fence();
    }
    uint32_t phases = 0;  // bit sl: parity of slot sl's next completion (the same in every thread)

    for (int m0 = 0; m0 < a.QH; m0 += RP) {
        __syncthreads();  // the barriers are set up; the previous pass's merge slots are read
        if (tid == 0) {   // the ring's first sub-chunks are requested before the query tile
            fence_proxy_async();
            for (int sl = 0; sl < NST && sl < nsubs; ++sl)
                issue_chunk<D, Q8, R>(ring + sl * SM::SLOT, bar0 + 8 * sl, lay, a.geo, vbase, (sub0 + sl) * ATT_TC,
                                      a.T, kscales, a.vlr);
        }
        if (tid < 64) {
            const float c0 = centroid_e4(uint32_t(tid & 7)) * 1e-4f, c1 = centroid_e4(uint32_t(tid >> 3)) * 1e-4f;
            lut[tid] = pack_half2(c0, c1);
        }
        // the kernel before this one (see attend_split) has completed and its
        // writes are visible past this point; the queries are read, and the
        // workspace written, only after it
        asm volatile("griddepcontrol.wait;" ::: "memory");
        {   // the query tile: every load of a thread issued before its stores
            constexpr int QPT = (RP * (D / 8) + ATT_THREADS - 1) / ATT_THREADS;
            uint4 v[QPT];
#pragma unroll
            for (int u = 0; u < QPT; ++u) {
                const int e = tid + u * ATT_THREADS, r = e / (D / 8), c8 = e % (D / 8);
                v[u] = make_uint4(0, 0, 0, 0);
                if (e < RP * (D / 8) && m0 + r < a.QH) {
                    const int ag = (m0 + r) / a.G, j = h * a.G + (m0 + r) % a.G;
                    v[u] = *reinterpret_cast<const uint4 *>(a.q + (uint64_t(ag) * a.NQ + j) * D + c8 * 8);
                }
            }
#pragma unroll
            for (int u = 0; u < QPT; ++u) {
                const int e = tid + u * ATT_THREADS, r = e / (D / 8), c8 = e % (D / 8);
                if (e < RP * (D / 8)) *reinterpret_cast<uint4 *>(Qs + r * RW + c8 * 4) = v[u];
            }
        }
        const bool active = m0 + mi * 16 < a.QH;  // warp-uniform: this tile has real rows
        float acc[NV][4];
#pragma unroll
        for (int nt = 0; nt < NV; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
        float mx[2] = {-INFINITY, -INFINITY}, ls[2] = {0.0f, 0.0f};
        float lracc[NL > 0 ? NL : 1][4];  // P V_lr (LoRA attention)
#pragma unroll
        for (int nt = 0; nt < (NL > 0 ? NL : 1); ++nt) lracc[nt][0] = lracc[nt][1] = lracc[nt][2] = lracc[nt][3] = 0.0f;

        __syncthreads();  // the pair table and the query tile are in
        int failed_at = -1;
        // sub-chunk j (raw slot j % NST) staged into tile set `set`
        auto stage_sub = [&](int j, int set) {
            const int t0 = (sub0 + j) * ATT_TC;
            const uint64_t n0 = vbase + uint64_t(t0);
            const uint32_t voff = uint32_t(reinterpret_cast<uintptr_t>(lay + a.geo.sec_v + n0 * (3 * D / 8)) & 15u);
            const uint32_t soff = uint32_t(reinterpret_cast<uintptr_t>(lay + a.geo.sec_sigma + n0 * 2) & 15u);
            const uint32_t qoff = Q8 ? uint32_t(reinterpret_cast<uintptr_t>(kscales + n0 * (D / 32)) & 15u) : 0u;
            stage_raw<D, Q8, R>(ring + (j % NST) * SM::SLOT, t0, a.T, tid, voff, soff, qoff, set ? Kt1 : Kt,
                                set ? Ct1 : Ct, set ? st1 : st, lut, set ? kst1 : kst, set ? Lt1 : Lt);
        };
        // thread 0: sub-chunk j's slot refilled with the sub-chunk NST ahead
        auto refill = [&](int j) {
            if (tid == 0 && j + NST < nsubs) {
                const int sl = j % NST;
                fence_proxy_async();
                issue_chunk<D, Q8, R>(ring + sl * SM::SLOT, bar0 + 8 * sl, lay, a.geo, vbase,
                                      (sub0 + j + NST) * ATT_TC, a.T, kscales, a.vlr);
            }
        };
        if constexpr (PIPE) {
            if (nsubs > 0) {  // sub-chunk 0 into the first tile set
                const bool ok = mbar_wait(bar0, phases & 1u, a.wait_polls);
                phases ^= 1u;
                stage_sub(0, 0);
                if (__syncthreads_or(!ok))
                    failed_at = 0;
                else
                    refill(0);
            }
        }
        for (int i = 0; i < nsubs && failed_at < 0; ++i) {
            const int sub = sub0 + i;
            int cur = 0;           // the tile set sub-chunk i is in
            bool ok_next = true;   // PIPE: sub-chunk i + 1's copies landed in time
            if constexpr (PIPE) {
                cur = i & 1;
                if (i + 1 < nsubs) {  // the next sub-chunk into the other tile set
                    const int sl = (i + 1) % NST;
                    ok_next = mbar_wait(bar0 + 8 * sl, (phases >> sl) & 1u, a.wait_polls);
                    phases ^= 1u << sl;
                    stage_sub(i + 1, cur ^ 1);
                }
            } else {
                const int sl = i % NST;
                if (i > 0) __syncthreads();  // every warp is done with the staged tiles
                const bool ok = mbar_wait(bar0 + 8 * sl, (phases >> sl) & 1u, a.wait_polls);
                phases ^= 1u << sl;
                stage_sub(i, 0);
                if (__syncthreads_or(!ok)) {  // the tiles are staged and the slot is free, unless a wait ran out
                    failed_at = i;
                    break;
                }
                refill(i);
            }
            const uint32_t *Kc = cur ? Kt1 : Kt, *Cc = cur ? Ct1 : Ct, *Lc = cur ? Lt1 : Lt;
            const float *sc = cur ? st1 : st, *kc = cur ? kst1 : kst;
            if (active) {

                // S = Q K^T for rows mi*16.., tokens th*TPW..
                float s[NS][4];
    #pragma unroll
                for (int nt = 0; nt < NS; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.0f;
                if constexpr (!Q8) {
    #pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        uint32_t qa[4];
                        ldsm_x4(qa, Qs + (mi * 16 + (lane & 15)) * RW + ks * 8 + (lane >> 4) * 4);
    #pragma unroll
                        for (int np = 0; np < NS; np += 2) {
                            uint32_t kb[4];
                            const int tok = th * TPW + np * 8 + (lane & 7) + ((lane >> 4) << 3);
                            ldsm_x4(kb, Kc + tok * RW + ks * 8 + ((lane >> 3) & 1) * 4);
                            mma_bf16(s[np], qa, kb[0], kb[1]);
                            mma_bf16(s[np + 1], qa, kb[2], kb[3]);
                        }
                    }
                } else {
                    // q8_0: each 32-key block's exact partial products, one n-tile
                    // at a time, added in scaled by that token's block scale
    #pragma unroll
                    for (int nt = 0; nt < NS; ++nt) {
                        const int tok = th * TPW + nt * 8 + (lane & 7);
                        const int tl = th * TPW + nt * 8 + 2 * tig;
    #pragma unroll 1
                        for (int blk = 0; blk < D / 32; ++blk) {
                            float t1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                            uint32_t kb[4];  // k-steps 2 blk and 2 blk + 1 of this n-tile
                            ldsm_x4(kb, Kc + tok * RW + blk * 16 + (lane >> 3) * 4);
    #pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                uint32_t qa[4];
                                ldsm_x4(qa, Qs + (mi * 16 + (lane & 15)) * RW + (2 * blk + kk) * 8 + (lane >> 4) * 4);
                                mma_bf16(t1, qa, kb[2 * kk], kb[2 * kk + 1]);
                            }
                            const float c0 = kc[tl * (D / 32) + blk], c1 = kc[(tl + 1) * (D / 32) + blk];
                            s[nt][0] = fmaf(t1[0], c0, s[nt][0]);
                            s[nt][1] = fmaf(t1[1], c1, s[nt][1]);
                            s[nt][2] = fmaf(t1[2], c0, s[nt][2]);
                            s[nt][3] = fmaf(t1[3], c1, s[nt][3]);
                        }
                    }
                }
                // online softmax over this warp's slice (rows g and g+8 of the tile)
                const int tbase = sub * ATT_TC + th * TPW;
                float cm[2] = {-INFINITY, -INFINITY};
                if (tbase + TPW <= a.T) {  // warp-uniform: every token of the slice is real
    #pragma unroll
                    for (int nt = 0; nt < NS; ++nt) {
                        const float2 lo = __fmul2_rn(make_float2(s[nt][0], s[nt][1]), make_float2(qk2, qk2));
                        const float2 hi = __fmul2_rn(make_float2(s[nt][2], s[nt][3]), make_float2(qk2, qk2));
                        s[nt][0] = lo.x, s[nt][1] = lo.y, s[nt][2] = hi.x, s[nt][3] = hi.y;
                        cm[0] = fmaxf(cm[0], fmaxf(s[nt][0], s[nt][1]));
                        cm[1] = fmaxf(cm[1], fmaxf(s[nt][2], s[nt][3]));
                    }
                } else {
    #pragma unroll
                    for (int nt = 0; nt < NS; ++nt) {
                        const int tk = tbase + nt * 8 + 2 * tig;
                        s[nt][0] = tk < a.T ? s[nt][0] * qk2 : -INFINITY;
                        s[nt][1] = tk + 1 < a.T ? s[nt][1] * qk2 : -INFINITY;
                        s[nt][2] = tk < a.T ? s[nt][2] * qk2 : -INFINITY;
                        s[nt][3] = tk + 1 < a.T ? s[nt][3] * qk2 : -INFINITY;
                        cm[0] = fmaxf(cm[0], fmaxf(s[nt][0], s[nt][1]));
                        cm[1] = fmaxf(cm[1], fmaxf(s[nt][2], s[nt][3]));
                    }
                }
                float ref[2], al[2];
    #pragma unroll
                for (int i = 0; i < 2; ++i) {
                    cm[i] = fmaxf(cm[i], __shfl_xor_sync(0xffffffffu, cm[i], 1));
                    cm[i] = fmaxf(cm[i], __shfl_xor_sync(0xffffffffu, cm[i], 2));
                    const float nm = fmaxf(mx[i], cm[i]);
                    ref[i] = nm == -INFINITY ? 0.0f : nm;  // a slice with no token yet: p = 0, nothing to rescale
                    al[i] = exp2f(mx[i] - ref[i]);
                    mx[i] = nm;
                    ls[i] *= al[i];
                }
                {
                    const float2 a0 = make_float2(al[0], al[0]), a1 = make_float2(al[1], al[1]);
    #pragma unroll
                    for (int nt = 0; nt < NV; ++nt) {
                        const float2 lo = __fmul2_rn(make_float2(acc[nt][0], acc[nt][1]), a0);
                        const float2 hi = __fmul2_rn(make_float2(acc[nt][2], acc[nt][3]), a1);
                        acc[nt][0] = lo.x, acc[nt][1] = lo.y, acc[nt][2] = hi.x, acc[nt][3] = hi.y;
                    }
                }
                if constexpr (R > 0) {
    #pragma unroll
                    for (int nt = 0; nt < NL; ++nt) {
                        lracc[nt][0] *= al[0];
                        lracc[nt][1] *= al[0];
                        lracc[nt][2] *= al[1];
                        lracc[nt][3] *= al[1];
                    }
                }
                // P' = p * sigma as fp16 A fragments: the S accumulator of n-tiles
                // 2kk, 2kk+1 is the A operand of k-step kk
    #pragma unroll
                for (int kk = 0; kk < NS / 2; ++kk) {
                    uint32_t pa[4], pl[4];  // p * sigma for the pool's values; p for the low-rank cache
    #pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int nt = 2 * kk + hf;
                        const int tl = th * TPW + nt * 8 + 2 * tig;
                        const float s0 = sc[tl], s1 = sc[tl + 1];
                        const float p0 = exp2f(s[nt][0] - ref[0]), p1 = exp2f(s[nt][1] - ref[0]);
                        const float p2 = exp2f(s[nt][2] - ref[1]), p3 = exp2f(s[nt][3] - ref[1]);
                        ls[0] += p0 + p1;
                        ls[1] += p2 + p3;
                        pa[2 * hf] = pack_half2(p0 * s0, p1 * s1);
                        pa[2 * hf + 1] = pack_half2(p2 * s0, p3 * s1);
                        if constexpr (R > 0) {
                            pl[2 * hf] = pack_half2(p0, p1);
                            pl[2 * hf + 1] = pack_half2(p2, p3);
                        }
                    }
                    // A += P' C over tokens th*TPW + kk*16 .. +15, every dim
    #pragma unroll
                    for (int np = 0; np < NV; np += 2) {
                        uint32_t cb[4];
                        const int tok = th * TPW + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                        ldsm_x4_t(cb, Cc + tok * RW + np * 4 + (lane >> 4) * 4);
                        mma_f16(acc[np], pa, cb[0], cb[1]);
                        mma_f16(acc[np + 1], pa, cb[2], cb[3]);
                    }
                    if constexpr (R > 0) {
                        // Flash-LoRA reorder: P V_lr over the same tokens, r columns
    #pragma unroll
                        for (int np = 0; np < NL; np += 2) {
                            uint32_t lb[4];
                            const int tok = th * TPW + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                            ldsm_x4_t(lb, Lc + tok * LW + np * 4 + (lane >> 4) * 4);
                            mma_f16(lracc[np], pl, lb[0], lb[1]);
                            mma_f16(lracc[np + 1], pl, lb[2], lb[3]);
                        }
                    }
                }
            }
            if constexpr (PIPE) {
                // the next tile set is staged and this one is free, unless a wait ran out
                if (__syncthreads_or(!ok_next)) {
                    failed_at = i + 1;
                    break;
                }
                refill(i + 1);
            }
        }
        if (failed_at >= 0) {
            // a bulk copy did not complete in time: report it, let the copies
            // still outstanding (sub-chunks failed_at .. failed_at + NST - 1)
            // land (bounded), and give up on this block
            if (tid == 0) {
                atomicOr(const_cast<uint32_t *>(reinterpret_cast<const uint32_t *>(a.pool)) + POOL_ERR_WORD,
                         FLAG_TIMEOUT);
                for (int k = failed_at; k < nsubs && k < failed_at + NST; ++k) {
                    const int sl = k % NST;
                    mbar_wait(bar0 + 8 * sl, ((phases >> sl) & 1u) ^ (k == failed_at ? 1u : 0u), ATT_WAIT_LIMIT);
                }
            }
            return;
        }
        // the combine kernel (launched as this kernel's programmatic
        // dependent) may be placed once every block is this far; it waits for
        // this grid's completion before it reads
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        // merge the token slices of each row tile
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            ls[i] += __shfl_xor_sync(0xffffffffu, ls[i], 1);
            ls[i] += __shfl_xor_sync(0xffffffffu, ls[i], 2);
        }
        __syncthreads();  // every warp is done with the staged tiles
        {
            float *slot = mrg + warp * (16 * MSW);
#pragma unroll
            for (int nt = 0; nt < NV; ++nt) {
                *reinterpret_cast<float2 *>(slot + g * MSW + nt * 8 + 2 * tig) = make_float2(acc[nt][0], acc[nt][1]);
                *reinterpret_cast<float2 *>(slot + (g + 8) * MSW + nt * 8 + 2 * tig) =
                    make_float2(acc[nt][2], acc[nt][3]);
            }
            if constexpr (R > 0) {
#pragma unroll
                for (int nt = 0; nt < NL; ++nt) {
                    *reinterpret_cast<float2 *>(slot + g * MSW + D + nt * 8 + 2 * tig) =
                        make_float2(lracc[nt][0], lracc[nt][1]);
                    *reinterpret_cast<float2 *>(slot + (g + 8) * MSW + D + nt * 8 + 2 * tig) =
                        make_float2(lracc[nt][2], lracc[nt][3]);
                }
            }
            float *ms = mrg + ATT_WARPS * 16 * MSW + warp * 32;
            if (tig == 0) {
                ms[g] = mx[0];
                ms[g + 8] = mx[1];
                ms[16 + g] = ls[0];
                ms[16 + g + 8] = ls[1];
            }
        }
        __syncthreads();
        const uint64_t pbase = (uint64_t(h) * a.nsplit + split) * uint64_t(a.QHP);
        for (int e = tid; e < RP * (PW / 4); e += ATT_THREADS) {
            const int r = e / (PW / 4), c4 = e % (PW / 4);
            if (m0 + r >= a.QH) continue;
            const int ti = r >> 4, rr = r & 15;
            const float *ms = mrg + ATT_WARPS * 16 * MSW;
            float M = -INFINITY;
#pragma unroll
            for (int w = ti; w < ATT_WARPS; w += MS) M = fmaxf(M, ms[w * 32 + rr]);
            float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            float l = 0.0f;
#pragma unroll
            for (int w = ti; w < ATT_WARPS; w += MS) {
                const float f = exp2f(ms[w * 32 + rr] - M);  // 0 for a slice that saw no token
                const float4 x = *reinterpret_cast<const float4 *>(mrg + w * (16 * MSW) + rr * MSW + c4 * 4);
                o.x = fmaf(f, x.x, o.x);
                o.y = fmaf(f, x.y, o.y);
                o.z = fmaf(f, x.z, o.z);
                o.w = fmaf(f, x.w, o.w);
                l = fmaf(f, ms[w * 32 + 16 + rr], l);
            }
            *reinterpret_cast<float4 *>(a.part + (pbase + m0 + r) * PW + c4 * 4) = o;
            if (c4 == 0) a.stats[pbase + m0 + r] = make_float2(M, l);
        }
    }
}

template <int D, int TPW, int R>
__global__ void __launch_bounds__(ATT_THREADS, 2) attend_split(const __grid_constant__ AttendArgs a) {
    extern __shared__ __align__(16) uint32_t smem[];
    // Launched as a programmatic dependent of whatever precedes it on the
    // stream, and waits for it (griddepcontrol.wait) before it reads the
    // queries or writes its workspace.  The pool (and a LoRA cache) is read
    // before that wait: the only kernel that lets this grid start early is the
    // combine of a previous attention call, which writes neither, and any
    // other kernel before it (an encode, a caller's kernel) has completed
    // before this grid starts.
    const uint32_t *hdr = reinterpret_cast<const uint32_t *>(a.pool);
    const uint32_t kmode = hdr[POOL_KMODE_WORD];
    if (hdr[0] != POOL_MAGIC || hdr[1] != POOL_VERSION || hdr[2] != uint32_t(a.L) || hdr[3] != uint32_t(a.H) ||
        hdr[4] != uint32_t(D) || hdr[5] != uint32_t(a.T) || (kmode != KVP_K_PER_TENSOR && kmode != KVP_K_Q8_0)) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && hdr[0] == POOL_MAGIC)
            atomicOr(const_cast<uint32_t *>(hdr) + POOL_ERR_WORD, FLAG_HEADER);
        return;
    }
    if (kmode == KVP_K_Q8_0)
        attend_passes<D, TPW, true, R>(
            a, smem,
            reinterpret_cast<const uint16_t *>(a.pool + a.geo.off_kscales) + uint64_t(a.layer) * a.H * a.T * (D / 32));
    else
        attend_passes<D, TPW, false, R>(a, smem, nullptr);
}

// One 128-thread block per (agent, query head): merge the splits, inverse
// transform.  Warp w merges splits w, w+4, ... online, with the statistics
// and partial rows of up to eight splits in flight at once; the four warps'
// states are then merged in shared memory and warp 0 applies the transform.
// LoRA attention (R > 0): lane k < R also merges column k of P V_lr, and the
// agent's up-projection is applied once, after the transform:
// out += (P V_lr / l) B_a[:, h*d .. h*d + d).
constexpr int CMB_THREADS = 128;
constexpr int CMB_WARPS = CMB_THREADS / 32;

template <int D, int R>
__global__ void __launch_bounds__(CMB_THREADS) attend_combine(const __grid_constant__ AttendArgs a) {
    constexpr int PL = D / 32;  // dims per lane, indices lane*PL + e
    constexpr int UN = 8;       // splits in flight per warp
    constexpr int PW = D + R;   // floats per partial row
    __shared__ float wacc[CMB_WARPS][D + (R > 0 ? 32 : 0)];
    __shared__ float wml[CMB_WARPS][2];
    __shared__ __align__(16) uint16_t sb[R > 0 ? R : 1][R > 0 ? D : 8];  // LoRA: B_a's rows, this head's columns
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ag = blockIdx.x / a.NQ, j = blockIdx.x % a.NQ;
    const int h = j / a.G, r = ag * a.G + j % a.G;
    // a following split kernel (the next layer's attention) may be placed
    // now: it waits for this grid's completion before it reads anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if constexpr (R > 0) {
        // the agent's up-projection is an input, not a result of the split
        // kernel (which runs after every earlier kernel of the stream is
        // done), so it is requested before the wait, by asynchronous copies
        // that stay in flight beside the partial-row loads below
        const uint16_t *bh = a.lora_b + uint64_t(ag) * R * uint64_t(a.H) * D + uint64_t(h) * D;
        const uint64_t keep = l2_evict_last_policy();  // read by the agent's other query heads too
        for (int i = threadIdx.x; i < R * (D / 8); i += CMB_THREADS) {
            const int k = i / (D / 8), c = i % (D / 8);
            cp_async16(&sb[k][c * 8], bh + uint64_t(k) * a.H * D + c * 8, 16, keep);
        }
        cp_async_commit();
    }
    // launched as a programmatic dependent of the split kernel: its partial
    // rows and statistics are complete and visible after this wait
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint64_t row0 = uint64_t(h) * a.nsplit * uint64_t(a.QHP) + r;  // split sp: row0 + sp * QHP
    float m = -INFINITY, l = 0.0f, acc[PL], lrv = 0.0f;
#pragma unroll
    for (int e = 0; e < PL; ++e) acc[e] = 0.0f;
    for (int sp0 = warp; sp0 < a.nsplit; sp0 += CMB_WARPS * UN) {
        float2 st[UN];
        float v[UN][PL], vl[UN];
#pragma unroll
        for (int u = 0; u < UN; ++u) {
            const int sp = sp0 + u * CMB_WARPS;
            st[u] = make_float2(-INFINITY, 0.0f);
            vl[u] = 0.0f;
#pragma unroll
            for (int e = 0; e < PL; ++e) v[u][e] = 0.0f;
            if (sp < a.nsplit) {
                const uint64_t row = row0 + uint64_t(sp) * a.QHP;
                st[u] = a.stats[row];
                const float *pp = a.part + row * PW + lane * PL;
                if constexpr (R > 0)
                    if (lane < R) vl[u] = a.part[row * PW + D + lane];
                if constexpr (PL == 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(pp);
                    v[u][0] = x.x, v[u][1] = x.y, v[u][2] = x.z, v[u][3] = x.w;
                } else {
                    const float2 x = *reinterpret_cast<const float2 *>(pp);
                    v[u][0] = x.x, v[u][1] = x.y;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < UN; ++u) {
            if (st[u].x == -INFINITY) continue;  // past the last split
            const float nm = fmaxf(m, st[u].x);
            const float f0 = exp2f(m - nm), f1 = exp2f(st[u].x - nm);
            l = l * f0 + st[u].y * f1;
#pragma unroll
            for (int e = 0; e < PL; ++e) acc[e] = acc[e] * f0 + v[u][e] * f1;
            if constexpr (R > 0) lrv = lrv * f0 + vl[u] * f1;
            m = nm;
        }
    }
#pragma unroll
    for (int e = 0; e < PL; ++e) wacc[warp][lane * PL + e] = acc[e];
    if constexpr (R > 0) {
        wacc[warp][D + lane] = lrv;
        cp_async_wait<0>();  // this thread's share of B_a is in (the barrier below publishes it)
    }
    if (lane == 0) {
        wml[warp][0] = m;
        wml[warp][1] = l;
    }
    __syncthreads();
    if (warp != 0) return;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < CMB_WARPS; ++w) M = fmaxf(M, wml[w][0]);
    l = 0.0f;
    lrv = 0.0f;
#pragma unroll
    for (int e = 0; e < PL; ++e) acc[e] = 0.0f;
#pragma unroll
    for (int w = 0; w < CMB_WARPS; ++w) {
        const float f = wml[w][0] == -INFINITY ? 0.0f : exp2f(wml[w][0] - M);  // a warp with no split
        l = fmaf(f, wml[w][1], l);
#pragma unroll
        for (int e = 0; e < PL; ++e) acc[e] = fmaf(f, wacc[w][lane * PL + e], acc[e]);
        if constexpr (R > 0) lrv = fmaf(f, wacc[w][D + lane], lrv);
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
    for (int e = 0; e < PL; ++e) acc[e] *= f;
    if constexpr (R > 0) {
        // (P V_lr / l) B_a, restricted to this KV head's d columns
        const float il = 1.0f / l;
#pragma unroll 4
        for (int k = 0; k < R; ++k) {
            const float c = __shfl_sync(0xffffffffu, lrv, k) * il;
            const uint16_t *bk = &sb[k][lane * PL];
            if constexpr (PL == 4) {
                const uint2 w = *reinterpret_cast<const uint2 *>(bk);
                acc[0] = fmaf(c, bf16_lo(w.x), acc[0]);
                acc[1] = fmaf(c, bf16_hi(w.x), acc[1]);
                acc[2] = fmaf(c, bf16_lo(w.y), acc[2]);
                acc[3] = fmaf(c, bf16_hi(w.y), acc[3]);
            } else {
                const uint32_t w = *reinterpret_cast<const uint32_t *>(bk);
                acc[0] = fmaf(c, bf16_lo(w), acc[0]);
                acc[1] = fmaf(c, bf16_hi(w), acc[1]);
            }
        }
    }
#pragma unroll
    for (int e = 0; e < PL; ++e) o[e] = acc[e];
    if (lane == 0) a.lse[uint64_t(ag) * a.NQ + j] = (M + __log2f(l)) * 0.6931471805599453f;
}

// The split kernel's dynamic shared memory exceeds the default 48 KB: raise
// the limit once per device (the first call on a device does it).
template <int D, int TPW, int R>
static bool attend_smem_ready() {
    static bool done[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (!done[dev]) {
        // two blocks per SM need the largest shared-memory carveout; without
        // the preference the driver may configure the SM for one block
        if (cudaFuncSetAttribute(attend_split<D, TPW, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(SplitSmem<D, TPW, R>::bytes)) != cudaSuccess ||
            cudaFuncSetAttribute(attend_split<D, TPW, R>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 int(cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
            return false;
        done[dev] = true;
    }
    return true;
}

template <int D, int TPW, int R>
static int attend_launch(const AttendArgs &a, dim3 grid, unsigned cgrid, cudaStream_t st) {
    if (!attend_smem_ready<D, TPW, R>()) return KVP_ERR_CUDA;
    // programmatic dependent launch on both kernels: the split's blocks may be
    // placed while the kernel before it (a previous layer's combine) finishes,
    // and wait (griddepcontrol.wait) for it before reading
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t scfg = {};
    scfg.gridDim = grid;
    scfg.blockDim = dim3(ATT_THREADS);
    scfg.dynamicSmemBytes = SplitSmem<D, TPW, R>::bytes;
    scfg.stream = st;
    scfg.attrs = attr;
    scfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&scfg, attend_split<D, TPW, R>, a) != cudaSuccess) return KVP_ERR_CUDA;
    // programmatic dependent launch: the combine's blocks are placed while the
    // split runs and wait (griddepcontrol.wait) for its results
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cgrid);
    cfg.blockDim = dim3(CMB_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, attend_combine<D, R>, a) != cudaSuccess) return KVP_ERR_CUDA;
    return KVP_OK;
}

// head_dim, token-slice width (at most 32 query rows per KV head: 16) and rank
template <int R>
static int attend_dispatch(const AttendArgs &a, int d, bool narrow, dim3 grid, unsigned cgrid, cudaStream_t st) {
    if (d == 128)
        return narrow ? attend_launch<128, 16, R>(a, grid, cgrid, st) : attend_launch<128, 32, R>(a, grid, cgrid, st);
    return narrow ? attend_launch<64, 16, R>(a, grid, cgrid, st) : attend_launch<64, 32, R>(a, grid, cgrid, st);
}

// Blocks of the split kernel resident at once: SMs times blocks per SM (two:
// about 100 KB of shared memory and 128 registers per thread each).  The
// plan keeps the grid within that one wave.  Without a device (a size query
// on a host without a GPU) it is made for the GB300's 152 SMs.
static int attend_target_blocks() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        (void)cudaGetLastError();
        return 2 * 152;
    }
    static int cached[64] = {0};
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int occ = 0;
    if (!attend_smem_ready<128, 32, 0>() ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, attend_split<128, 32, 0>, ATT_THREADS,
                                                      SplitSmem<128, 32, 0>::bytes) != cudaSuccess ||
        occ < 1) {
        (void)cudaGetLastError();
        occ = 1;
    }
    const int n = sms * occ;
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
}

struct AttendPlan {
    int G, QH, QHP, nsub, per_split, nsplit;
    uint64_t part_off, stats_off, total;
};

static inline AttendPlan attend_plan(const kvp_shape *s, int na, int nq, int rank = 0) {
    AttendPlan p;
    p.G = nq / s->n_kv_heads;
    p.QH = na * p.G;
    p.QHP = (p.QH + ATT_MT - 1) / ATT_MT * ATT_MT;
    p.nsub = (s->n_tokens + ATT_TC - 1) / ATT_TC;
    int want = attend_target_blocks() / s->n_kv_heads;  // splits per KV head: the grid stays within one wave
    if (want < 1) want = 1;
    if (want > p.nsub) want = p.nsub;
    p.per_split = (p.nsub + want - 1) / want;
    p.nsplit = (p.nsub + p.per_split - 1) / p.per_split;
    const uint64_t rows = uint64_t(s->n_kv_heads) * uint64_t(p.nsplit) * uint64_t(p.QHP);
    p.part_off = 0;
    p.stats_off = align256(rows * uint64_t(s->head_dim + rank) * 4u);
    p.total = align256(p.stats_off + rows * 8u);
    return p;
}

// Failure-path testing (kvp_test_limit_next_attend): consumed by the next
// attention call on the calling thread.
static thread_local uint32_t t_att_polls = ATT_WAIT_LIMIT;

// Checks, arguments and launches shared by plain (rank 0) and LoRA attention.
static int attend_common(const void *pool, const kvp_shape *s, int layer, int n_agents, int n_q_heads,
                         const void *q, float scale, int rank, const void *v_lr, const void *lora_b, float *out,
                         float *lse, void *ws, size_t ws_bytes, void *stream) {
    int rc = shape_ok(s);
    if (rc != KVP_OK) return rc;
    if (!pool || !q || !out || !lse || !ws) return KVP_ERR_ARG;
    if (layer < 0 || layer >= s->n_layers || n_agents < 1 || n_q_heads < 1 || n_q_heads % s->n_kv_heads != 0)
        return KVP_ERR_ARG;
    if (rank != 0 && (!v_lr || !lora_b)) return KVP_ERR_ARG;
    if (uint64_t(n_agents) * uint64_t(n_q_heads) >= (1ull << 24)) return KVP_ERR_SIZE;
    if (!aligned(pool, 256) || !aligned(q, 16) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(ws, 16))
        return KVP_ERR_ALIGN;
    if (rank != 0 && (!aligned(v_lr, 16) || !aligned(lora_b, 16))) return KVP_ERR_ALIGN;
    const AttendPlan p = attend_plan(s, n_agents, n_q_heads, rank);
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
    a.vlr = static_cast<const uint16_t *>(v_lr);
    a.lora_b = static_cast<const uint16_t *>(lora_b);
    a.wait_polls = t_att_polls;
    t_att_polls = ATT_WAIT_LIMIT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const dim3 grid(unsigned(a.H), unsigned(a.nsplit));
    const unsigned cgrid = unsigned(n_agents) * unsigned(n_q_heads);  // one block per query
    const bool narrow = p.QH <= 32;
    if (rank == 0)
        rc = attend_dispatch<0>(a, s->head_dim, narrow, grid, cgrid, st);
    else if (rank == 16)
        rc = attend_dispatch<16>(a, s->head_dim, narrow, grid, cgrid, st);
    else
        rc = attend_dispatch<32>(a, s->head_dim, narrow, grid, cgrid, st);
    if (rc != KVP_OK) return rc;
    count_launch(2);
    return launch_status();
}

static inline bool rank_ok(int rank) { return rank == 16 || rank == 32; }


}  // namespace kvp

using namespace kvp;

extern "C" int kvp_test_limit_next_attend(uint32_t polls) {
    t_att_polls = polls;
    return KVP_OK;
}

extern "C" size_t kvpool_attend_workspace_bytes(const kvp_shape *s, int n_agents, int n_q_heads) {
    if (shape_ok(s) != KVP_OK || n_agents < 1 || n_q_heads < 1 || n_q_heads % s->n_kv_heads != 0) return 0;
    return size_t(attend_plan(s, n_agents, n_q_heads).total);
}

extern "C" int kvpool_attend(const void *pool, const kvp_shape *s, int layer, int n_agents, int n_q_heads,
                             const void *q, float scale, float *out, float *lse, void *ws, size_t ws_bytes,
                             void *stream) {
    return attend_common(pool, s, layer, n_agents, n_q_heads, q, scale, 0, nullptr, nullptr, out, lse, ws, ws_bytes,
                         stream);
}

extern "C" size_t kvpool_attend_lora_workspace_bytes(const kvp_shape *s, int n_agents, int n_q_heads, int rank) {
    if (shape_ok(s) != KVP_OK || n_agents < 1 || n_q_heads < 1 || n_q_heads % s->n_kv_heads != 0 || !rank_ok(rank))
        return 0;
    return size_t(attend_plan(s, n_agents, n_q_heads, rank).total);
}

extern "C" int kvpool_attend_lora(const void *pool, const kvp_shape *s, int layer, int n_agents, int n_q_heads,
                                  const void *q, float scale, int rank, const void *v_lr, const void *lora_b,
                                  float *out, float *lse, void *ws, size_t ws_bytes, void *stream) {
    if (!rank_ok(rank)) return KVP_ERR_ARG;
    return attend_common(pool, s, layer, n_agents, n_q_heads, q, scale, rank, v_lr, lora_b, out, lse, ws, ws_bytes,
                         stream);
}
