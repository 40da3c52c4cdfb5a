// kvpool_decode.cu -- fan-out decode of a SharedKVPool ("PolyKV" 2.A: each
// PooledAgent receives the decompressed KV layer by layer in its own cache;
// 2.B.2 dequantization: centroid lookup, inverse Walsh-Hadamard transform,
// rescale).  The pool is read once per launch; every decoded tile is stored
// to all agents' caches by bulk copies from shared memory, so HBM traffic is
// the pool plus N x the bf16 cache -- the write side is the roofline.
#include "kvp_vec.cuh"

namespace kvp {

constexpr int DEC_THREADS = 256;
constexpr int DEC_WARPS = DEC_THREADS / 32;
constexpr int DEC_MAX_PTRS = 1024;  // (agent, layer) destinations per launch
// Fan-out by bulk copies: each warp decodes a unit into shared memory once and
// its lanes hand the agents' copies to the bulk-copy (TMA) engine, so the
// stores take no issue slots or registers of the SM.  Used from this many
// agents per launch; fewer are written with direct stores.
constexpr int DEC_BULK_MIN_AGENTS = 2;

// Asynchronous bulk copy shared -> global (16-byte aligned addresses, size a
// multiple of 16), tracked per thread in bulk async-groups.
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(gdst), "r"(static_cast<uint32_t>(__cvta_generic_to_shared(ssrc))), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every committed group of this thread has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every committed group of this thread is complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// generic-proxy shared-memory writes become visible to the bulk-copy engine
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

struct DecodeArgs {
    uint4 *kd[DEC_MAX_PTRS];  // index a * nl + r: agent a, layer lb + r
    uint4 *vd[DEC_MAX_PTRS];
    const uint8_t *pool;
    PoolGeom geo;
    int L, H, T, d;
    int lb, nl, na;
};

// 8 int8 key codes -> 8 bf16 values q*s.  A code byte c is turned into the
// float 2^23 + (c + 128) by byte permutation (exact), then offset (exact) and
// scaled, two lanes of f32x2 at a time.
__device__ __forceinline__ uint4 k_decode8(uint2 raw, float s) {
    const uint32_t a0 = raw.x ^ 0x80808080u, a1 = raw.y ^ 0x80808080u;
    const float2 off = make_float2(8388736.0f, 8388736.0f), ss = make_float2(s, s);
    float2 f[4];
    f[0] = make_float2(__uint_as_float(__byte_perm(a0, 0x4B000000u, 0x7650u)),
                       __uint_as_float(__byte_perm(a0, 0x4B000000u, 0x7651u)));
    f[1] = make_float2(__uint_as_float(__byte_perm(a0, 0x4B000000u, 0x7652u)),
                       __uint_as_float(__byte_perm(a0, 0x4B000000u, 0x7653u)));
    f[2] = make_float2(__uint_as_float(__byte_perm(a1, 0x4B000000u, 0x7650u)),
                       __uint_as_float(__byte_perm(a1, 0x4B000000u, 0x7651u)));
    f[3] = make_float2(__uint_as_float(__byte_perm(a1, 0x4B000000u, 0x7652u)),
                       __uint_as_float(__byte_perm(a1, 0x4B000000u, 0x7653u)));
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = __fmul2_rn(f2sub(f[i], off), ss);
    return make_uint4(pack_bf16x2(f[0].x, f[0].y), pack_bf16x2(f[1].x, f[1].y), pack_bf16x2(f[2].x, f[2].y),
                      pack_bf16x2(f[3].x, f[3].y));
}

// One warp step ("unit"): VPW consecutive vectors of one layer.  The pool
// bytes of the unit are loaded up front (keys 4 x 8 B per lane, value codes
// 16 B on 24 lanes, sigma 2 B).  Value codes are staged in shared memory and
// each pair of codes (a, b) is looked up in a 64-entry table of
// (c_a + c_b, c_a - c_b), which is also the transform's first butterfly
// stage.  The decoded keys and values (2 KB each: VPW contiguous vectors)
// are written to the warp's staging area, and lane a hands agent a's two
// copies to the bulk-copy engine.
// The grid-stride walk over units; Q8: keys carry q8_0 block scales.
template <int D, bool Q8, bool BULK>
__device__ __forceinline__ void decode_units(const DecodeArgs &a, uint8_t (*stage)[384 + 16], const float2 *pair_lut,
                                             uint4 *ostage) {
    constexpr int LPV = D / 32;
    constexpr int VPW = 32 / LPV;
    constexpr int CPV = D / 8;
    constexpr int CB = 3 * D / 8;
    constexpr int KCH = VPW * D / 8 / 32;  // 8-byte key chunks per lane per step (4)
    // 1 / (sqrt(d) * 10^4): the orthonormal 1/sqrt(d) and the codebook's 10^4.
    constexpr float KS = D == 128 ? 8.838834764831845e-6f : 1.25e-5f;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane / LPV, l = lane % LPV;
    const uint64_t nvec = uint64_t(a.H) * uint64_t(a.T);
    const uint64_t upl = (nvec + VPW - 1) / VPW;
    const uint64_t total = upl * uint64_t(a.nl);
    const float *scales = reinterpret_cast<const float *>(a.pool + a.geo.off_scales);
    const uint16_t *kscales = reinterpret_cast<const uint16_t *>(a.pool + a.geo.off_kscales);
    uint4 *osk = ostage + warp * (2 * VPW * CPV);  // this warp's decoded unit: keys, then values
    uint4 *osv = osk + VPW * CPV;

    for (uint64_t u = uint64_t(blockIdx.x) * DEC_WARPS + warp; u < total; u += uint64_t(gridDim.x) * DEC_WARPS) {
        const int r = int(u / upl);
        const int layer = a.lb + r;
        const uint64_t n0 = (u % upl) * VPW;
        const uint32_t cnt = uint32_t(min(uint64_t(VPW), nvec - n0));
        const uint8_t *lay = a.pool + a.geo.off_layers + uint64_t(layer) * a.geo.layer_stride;

        // --- all loads of the unit first
        const uint2 *kc = reinterpret_cast<const uint2 *>(lay) + n0 * (D / 8);
        const uint32_t kvalid = cnt * (D / 8);
        uint2 kraw[KCH];
#pragma unroll
        for (int it = 0; it < KCH; ++it) {
            const uint32_t k = uint32_t(it) * 32u + uint32_t(lane);
            kraw[it] = k < kvalid ? ld_stream_v2(kc + k) : make_uint2(0x80808080u, 0x80808080u);
        }
        const uint32_t bytes = cnt * CB;
        const uint32_t off = uint32_t(lane) * 16u;
        const uint8_t *vsrc = lay + a.geo.sec_v + n0 * CB;
        uint4 vraw = make_uint4(0, 0, 0, 0);
        if (off + 16u <= bytes) {
            vraw = ld_stream_v4(vsrc + off);
        } else if (off < bytes) {
            const uint2 h = ld_stream_v2(vsrc + off);
            vraw.x = h.x;
            vraw.y = h.y;
        }
        const uint64_t n = n0 + g;
        const bool valid = n < nvec;
        const uint16_t sh = valid ? reinterpret_cast<const uint16_t *>(lay + a.geo.sec_sigma)[n] : uint16_t(0);
        if constexpr (BULK) {
            // the previous unit's copies have read this warp's staging area
            bulk_wait_read_all();
            __syncwarp();
        }
        float ks[KCH];  // each 8-key chunk's scale: the layer's, or its q8_0 block's
        if constexpr (Q8) {
            // chunk k of the unit holds keys 8k .. 8k+7 from vector n0: block (n0 * D + 8k) / 32
            const uint16_t *bs = kscales + (uint64_t(layer) * nvec + n0) * (D / 32);
#pragma unroll
            for (int it = 0; it < KCH; ++it) {
                const uint32_t k = uint32_t(it) * 32u + uint32_t(lane);
                ks[it] = k < kvalid ? __half2float(__ushort_as_half(bs[k >> 2])) : 0.0f;
            }
        } else {
            const float s = scales[layer];
#pragma unroll
            for (int it = 0; it < KCH; ++it) ks[it] = s;
        }

        // --- keys: decode, fan out
        {
            uint4 kout[KCH];
#pragma unroll
            for (int it = 0; it < KCH; ++it) kout[it] = k_decode8(kraw[it], ks[it]);
            if constexpr (BULK) {
#pragma unroll
                for (int it = 0; it < KCH; ++it) {
                    const uint32_t k = uint32_t(it) * 32u + uint32_t(lane);
                    if (k < kvalid) osk[k] = kout[it];
                }
            } else {
                for (int ag = 0; ag < a.na; ++ag) {
                    uint4 *kd = a.kd[ag * a.nl + r] + n0 * (D / 8);
#pragma unroll
                    for (int it = 0; it < KCH; ++it) {
                        const uint32_t k = uint32_t(it) * 32u + uint32_t(lane);
                        if (k < kvalid) st_stream_v4(kd + k, kout[it]);
                    }
                }
            }
        }

        // --- values: stage codes, look up pairs, transform, rescale, fan out
        if (off < 384u) *reinterpret_cast<uint4 *>(stage[warp] + off) = vraw;
        __syncwarp();
        float2 x[4][4];
        const uint32_t *st32 = reinterpret_cast<const uint32_t *>(stage[warp]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t o = uint32_t(g * CB + 3 * (j * LPV + l));
            const uint32_t w = __funnelshift_r(st32[o >> 2], st32[(o >> 2) + 1], (o & 3u) * 8u);
#pragma unroll
            for (int p = 0; p < 4; ++p) x[j][p] = pair_lut[(w >> (6 * p)) & 63u];
        }
        __syncwarp();
        fwht_pairs<LPV>(x, lane);
        const float f = __half2float(__ushort_as_half(sh)) * KS;
        const float2 ff = make_float2(f, f);
        uint4 vout[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 y0 = __fmul2_rn(x[j][0], ff), y1 = __fmul2_rn(x[j][1], ff);
            const float2 y2 = __fmul2_rn(x[j][2], ff), y3 = __fmul2_rn(x[j][3], ff);
            vout[j] = make_uint4(pack_bf16x2(y0.x, y0.y), pack_bf16x2(y1.x, y1.y), pack_bf16x2(y2.x, y2.y),
                                 pack_bf16x2(y3.x, y3.y));
        }
        if constexpr (BULK) {
            if (valid) {
#pragma unroll
                for (int j = 0; j < 4; ++j) osv[g * CPV + j * LPV + l] = vout[j];
            }
            fence_proxy_async_smem();
            __syncwarp();
            // lane a sends the unit (cnt contiguous vectors of keys and of values) to agent a
            const uint32_t nbytes = cnt * uint32_t(D) * 2u;
            for (int ag = lane; ag < a.na; ag += 32) {
                bulk_store(a.kd[ag * a.nl + r] + n0 * (D / 8), osk, nbytes);
                bulk_store(a.vd[ag * a.nl + r] + n0 * CPV, osv, nbytes);
            }
            if (lane < a.na) bulk_commit();
        } else if (valid) {
            for (int ag = 0; ag < a.na; ++ag) {
                uint4 *vd = a.vd[ag * a.nl + r] + n * CPV;
#pragma unroll
                for (int j = 0; j < 4; ++j) st_stream_v4(vd + j * LPV + l, vout[j]);
            }
        }
    }
    if constexpr (BULK) bulk_wait_all();
}

// BULK: fan-out by bulk copies (several agents); otherwise direct streaming
// stores from registers (one agent: the copies would be too few to pay).
template <int D, bool BULK>
__global__ void __launch_bounds__(DEC_THREADS, 4) decode_fanout(const __grid_constant__ DecodeArgs a) {
    __shared__ __align__(16) uint8_t stage[DEC_WARPS][384 + 16];
    __shared__ float2 pair_lut[64];
    // per warp: one decoded unit (keys, then values) for the bulk copies
    __shared__ __align__(128) uint4 ostage[BULK ? DEC_WARPS * 2 * (32 / (D / 32)) * (D / 8) : 1];

    if (threadIdx.x < 64) {
        const float ca = centroid_e4(threadIdx.x & 7u), cb = centroid_e4(threadIdx.x >> 3);
        pair_lut[threadIdx.x] = make_float2(ca + cb, ca - cb);  // exact: integers < 2^16
    }
    __syncthreads();

    const uint32_t *hdr = reinterpret_cast<const uint32_t *>(a.pool);
    if (hdr[0] != POOL_MAGIC || hdr[1] != POOL_VERSION) return;
    const uint32_t kmode = hdr[POOL_KMODE_WORD];
    if (hdr[2] != uint32_t(a.L) || hdr[3] != uint32_t(a.H) || hdr[4] != uint32_t(a.d) || hdr[5] != uint32_t(a.T) ||
        (kmode != KVP_K_PER_TENSOR && kmode != KVP_K_Q8_0)) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            atomicOr(const_cast<uint32_t *>(hdr) + POOL_ERR_WORD, FLAG_HEADER);
        return;
    }
    if (kmode == KVP_K_Q8_0)
        decode_units<D, true, BULK>(a, stage, pair_lut, ostage);
    else
        decode_units<D, false, BULK>(a, stage, pair_lut, ostage);
}


template <int D, bool BULK>
static int decode_grid(uint64_t total_units) {
    const uint64_t want = (total_units + DEC_WARPS - 1) / DEC_WARPS;
    if (BULK) {
        // One unit per warp: every warp decodes one tile, hands its copies to
        // the bulk-copy engine and retires, so as many units as the SMs can
        // hold are being written at any time (measured on the 4K/15-agent
        // pool: 1.242 ms with three resident grids' worth of blocks, 1.183 ms
        // with one unit per warp; 2.88 -> 2.69 ms on the 32K/4-agent pool).
        return int(want < 1 ? 1 : (want < 0x7FFFFFFFull ? want : 0x7FFFFFFFull));
    }
    static int occ[2] = {0, 0};
    int &o = occ[D == 128 ? 1 : 0];
    if (o == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, decode_fanout<D, false>, DEC_THREADS, 0) != cudaSuccess ||
            o < 1)
            o = 1;
    }
    // Direct stores: three resident grids' worth of blocks, each block's
    // grid-stride walk spreading the concurrent stores over more of the
    // destination (measured 7-9 % faster than a single resident grid).
    const uint64_t cap = uint64_t(sm_count()) * uint64_t(o) * 3u;
    return int(want < cap ? (want < 1 ? 1 : want) : cap);
}

}  // namespace kvp

using namespace kvp;

extern "C" int kvpool_decode_into(const void *pool, const kvp_shape *s, int lb, int le, int na,
                                  void *const *k_dst, void *const *v_dst, void *stream) {
    int rc = shape_ok(s);
    if (rc != KVP_OK) return rc;
    if (!pool || !k_dst || !v_dst) return KVP_ERR_ARG;
    const int L = s->n_layers;
    if (lb < 0 || le > L || lb >= le || na < 1) return KVP_ERR_ARG;
    if (!aligned(pool, 256)) return KVP_ERR_ALIGN;
    for (int ag = 0; ag < na; ++ag)
        for (int l = lb; l < le; ++l) {
            const void *kp = k_dst[size_t(ag) * L + l], *vp = v_dst[size_t(ag) * L + l];
            if (!kp || !vp) return KVP_ERR_ARG;
            if (!aligned(kp, 16) || !aligned(vp, 16)) return KVP_ERR_ALIGN;
        }

    DecodeArgs a;
    a.pool = static_cast<const uint8_t *>(pool);
    a.geo = pool_geom(L, s->n_kv_heads, s->head_dim, s->n_tokens);
    a.L = L;
    a.H = s->n_kv_heads;
    a.T = s->n_tokens;
    a.d = s->head_dim;
    const uint64_t nvec = uint64_t(a.H) * uint64_t(a.T);
    const int vpw = a.d == 128 ? 8 : 16;
    const uint64_t upl = (nvec + vpw - 1) / vpw;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // Split (agent, layer) destinations into launches of at most
    // DEC_MAX_PTRS pointers each (one launch for every shape in practice).
    const int ac = na < DEC_MAX_PTRS ? na : DEC_MAX_PTRS;
    const int lc_max = DEC_MAX_PTRS / ac;
    int launches = 0;
    for (int a0 = 0; a0 < na; a0 += ac) {
        const int nag = (na - a0) < ac ? (na - a0) : ac;
        for (int l0 = lb; l0 < le; l0 += lc_max) {
            const int nl = (le - l0) < lc_max ? (le - l0) : lc_max;
            a.lb = l0;
            a.nl = nl;
            a.na = nag;
            for (int ag = 0; ag < nag; ++ag)
                for (int r = 0; r < nl; ++r) {
                    a.kd[ag * nl + r] = static_cast<uint4 *>(k_dst[size_t(a0 + ag) * L + l0 + r]);
                    a.vd[ag * nl + r] = static_cast<uint4 *>(v_dst[size_t(a0 + ag) * L + l0 + r]);
                }
            const uint64_t units = upl * uint64_t(nl);
            // bulk copies pay from DEC_BULK_MIN_AGENTS destinations per unit up
            if (nag >= DEC_BULK_MIN_AGENTS) {
                if (a.d == 128)
                    decode_fanout<128, true><<<decode_grid<128, true>(units), DEC_THREADS, 0, st>>>(a);
                else
                    decode_fanout<64, true><<<decode_grid<64, true>(units), DEC_THREADS, 0, st>>>(a);
            } else if (a.d == 128) {
                decode_fanout<128, false><<<decode_grid<128, false>(units), DEC_THREADS, 0, st>>>(a);
            } else {
                decode_fanout<64, false><<<decode_grid<64, false>(units), DEC_THREADS, 0, st>>>(a);
            }
            ++launches;
        }
    }
    count_launch(launches);
    return launch_status();
}
