// kvp_internal.cuh -- definitions shared by the library's translation units:
// byte-format geometry of the SharedKVPool and the CacheCard, error bits,
// bf16 helpers and streaming memory access.  Device code targets sm_103a.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kvpool.h"

namespace kvp {

// ---------------------------------------------------------------------------
// Error bits kept in the pool / card header (device-written).
// ---------------------------------------------------------------------------
constexpr uint32_t FLAG_NONFINITE = 1u;  // an input element was Inf or NaN
constexpr uint32_t FLAG_RANGE = 2u;      // a scale / zero point overflowed fp16
constexpr uint32_t FLAG_BITS = 4u;       // a CacheCard bitwidth not in {2,4,8,16}
constexpr uint32_t FLAG_SIZE = 8u;       // card buffer smaller than the bits need
constexpr uint32_t FLAG_HEADER = 16u;    // decode asked for a shape the pool lacks
constexpr uint32_t FLAG_TIMEOUT = 32u;   // a bounded wait on another block ran out

// ---------------------------------------------------------------------------
// SharedKVPool geometry ("PolyKV" 2.A: one object, size independent of the
// number of agents).  Header fields (little-endian, byte offsets):
//   0 magic "KVPL"  4 version  8 L  12 H  16 d  20 T  24 error  28 reserved
//   32 off_scales  40 off_layers  48 layer_stride  56 sec_v  64 sec_sigma
//   72 total_bytes; zero to 256.
// ---------------------------------------------------------------------------
constexpr uint32_t POOL_MAGIC = 0x4C50564Bu;
constexpr uint32_t POOL_VERSION = 1u;
constexpr uint64_t POOL_HEADER_BYTES = 256;
constexpr int POOL_ERR_WORD = 6;  // u32 index of the error word
constexpr int POOL_KMODE_WORD = 7;  // u32 index of the key format word (KVP_K_PER_TENSOR / KVP_K_Q8_0)

__host__ __device__ inline uint64_t align256(uint64_t x) { return (x + 255u) & ~uint64_t(255); }
__host__ __device__ inline uint64_t align16(uint64_t x) { return (x + 15u) & ~uint64_t(15); }

struct PoolGeom {
    uint64_t off_scales, off_layers, layer_stride, sec_v, sec_sigma, total;
    uint64_t off_kscales, total_q8;  // q8_0 keys: fp16 block scales [L][H][T][d/32] after the last layer
};

__host__ __device__ inline PoolGeom pool_geom(int L, int H, int d, int T) {
    PoolGeom g;
    const uint64_t nv = uint64_t(H) * uint64_t(T);
    g.off_scales = POOL_HEADER_BYTES;
    g.off_layers = align256(POOL_HEADER_BYTES + 4ull * uint64_t(L));
    g.sec_v = align256(nv * uint64_t(d));
    g.sec_sigma = align256(g.sec_v + nv * uint64_t(3 * d / 8));
    g.layer_stride = align256(g.sec_sigma + 2ull * nv);
    g.total = g.off_layers + uint64_t(L) * g.layer_stride;
    g.off_kscales = g.total;
    g.total_q8 = g.off_kscales + align256(uint64_t(L) * nv * uint64_t(d / 32) * 2ull);
    return g;
}

// ---------------------------------------------------------------------------
// CacheCard geometry ("QKVShare" Methodology 2).  The header is
// kvp_card_header (128 bytes); bits[T] at 128; off[T] 16-byte aligned after
// it; layers 256-byte aligned after that.
// ---------------------------------------------------------------------------
constexpr uint32_t CARD_MAGIC = 0x4343564Bu;
constexpr uint32_t CARD_VERSION = 1u;
constexpr uint64_t CARD_HEADER_BYTES = 128;
constexpr int CARD_GROUP = 32;

__host__ __device__ inline uint64_t card_record_bytes(int b, int H, int d) {
    uint64_t r;
    if (b == 16)
        r = 4ull * uint64_t(H) * uint64_t(d);
    else
        r = 2ull * (uint64_t(H) * uint64_t(d) * uint64_t(b) / 8ull + uint64_t(H) * uint64_t(d / CARD_GROUP) * 4ull);
    return align16(r);
}

__host__ __device__ inline bool valid_bits(int b) { return b == 2 || b == 4 || b == 8 || b == 16; }

__host__ __device__ inline uint64_t card_off_offsets(int T) { return align16(CARD_HEADER_BYTES + uint64_t(T)); }
__host__ __device__ inline uint64_t card_off_layers(int T) { return align256(card_off_offsets(T) + 4ull * uint64_t(T)); }

// ---------------------------------------------------------------------------
// Host-side helpers (kvp_host.cu).
// ---------------------------------------------------------------------------
int shape_ok(const kvp_shape *s);            // KVP_OK or an error code
int sm_count();                              // SMs of the current device (cached)
void count_launch(int n = 1);                // adds to kvp_launch_count()
int launch_status();                         // KVP_OK or KVP_ERR_CUDA after launches
inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// ---------------------------------------------------------------------------
// Device helpers.
// ---------------------------------------------------------------------------

// 16-byte load of data read exactly once: bypass L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ld_stream_v2(const void *p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void *p) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

// L2 eviction-priority policies for loads: keep (evict_last) data that is read
// again soon, drop (evict_first) data read for the last time.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ld_v4_policy(const void *p, uint64_t pol) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p), "l"(pol));
    return r;
}

// Asynchronous 16-byte global -> shared copies (completion tracked per thread
// with commit / wait groups).  src_bytes = 0 fills the 16 bytes with zeros
// and reads nothing.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, uint32_t src_bytes, uint64_t pol) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;"
                 ::"r"(s), "l"(gmem), "r"(src_bytes), "l"(pol) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Acquire / release on a 32-bit flag in global memory (GPU scope).
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 16-byte store of write-once output (evict-first in L2).
__device__ __forceinline__ void st_stream_v4(void *p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// The two bf16 halves of a 32-bit word as fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values rounded to nearest-even bf16, packed (a in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

}  // namespace kvp
