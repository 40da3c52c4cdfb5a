// kvp_probe.cu -- HBM bandwidth ceilings measured by the library's own
// kernels, so a benchmark can report the codec's kernels against the ceiling
// of the access pattern they use (the pages have no counterpart: this is
// measurement support only).
//
//  KVP_PROBE_STORE       16-byte streaming stores (st.global.cs.v4) over a
//                        grid-stride walk with one resident grid: the store
//                        pattern of the one-agent decode and the card unpack.
//  KVP_PROBE_BULK_STORE  4 KB shared -> global bulk copies, one per warp, one
//                        unit per warp: the fan-out decode's store pattern.
//  KVP_PROBE_COPY        16-byte loads and stores (read + write), a plain
//                        device copy.
#include "kvp_internal.cuh"

namespace kvp {

constexpr int PROBE_THREADS = 256;
constexpr int PROBE_WARPS = PROBE_THREADS / 32;
constexpr uint32_t PROBE_TILE = 4096;  // bytes per bulk copy

__global__ void __launch_bounds__(PROBE_THREADS) probe_store(uint4 *dst, uint64_t n16) {
    const uint4 v = make_uint4(threadIdx.x, blockIdx.x, 0x5A5A5A5Au, 0xA5A5A5A5u);
    const uint64_t stride = uint64_t(gridDim.x) * PROBE_THREADS;
    uint64_t i = uint64_t(blockIdx.x) * PROBE_THREADS + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        st_stream_v4(dst + i, v);
        st_stream_v4(dst + i + stride, v);
        st_stream_v4(dst + i + 2 * stride, v);
        st_stream_v4(dst + i + 3 * stride, v);
    }
    for (; i < n16; i += stride) st_stream_v4(dst + i, v);
}

__global__ void __launch_bounds__(PROBE_THREADS) probe_copy(uint4 *dst, const uint4 *src, uint64_t n16) {
    const uint64_t stride = uint64_t(gridDim.x) * PROBE_THREADS;
    uint64_t i = uint64_t(blockIdx.x) * PROBE_THREADS + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = ld_stream_v4(src + i), b = ld_stream_v4(src + i + stride);
        const uint4 c = ld_stream_v4(src + i + 2 * stride), d = ld_stream_v4(src + i + 3 * stride);
        st_stream_v4(dst + i, a);
        st_stream_v4(dst + i + stride, b);
        st_stream_v4(dst + i + 2 * stride, c);
        st_stream_v4(dst + i + 3 * stride, d);
    }
    for (; i < n16; i += stride) st_stream_v4(dst + i, ld_stream_v4(src + i));
}

// Each warp fills its 4 KB tile in shared memory and hands one bulk copy of
// it to the copy engine (lane 0), then waits for the copy before retiring.
__global__ void __launch_bounds__(PROBE_THREADS) probe_bulk_store(uint8_t *dst, uint64_t tiles) {
    __shared__ __align__(128) uint4 tile[PROBE_WARPS][PROBE_TILE / 16];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t t = uint64_t(blockIdx.x) * PROBE_WARPS + warp;
    if (t >= tiles) return;
    for (int i = lane; i < int(PROBE_TILE / 16); i += 32) tile[warp][i] = make_uint4(i, warp, blockIdx.x, 0x5A5A5A5Au);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                     :: "l"(dst + t * PROBE_TILE),
                        "r"(static_cast<uint32_t>(__cvta_generic_to_shared(&tile[warp][0]))), "r"(PROBE_TILE)
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
}

}  // namespace kvp

using namespace kvp;

extern "C" int kvp_bandwidth_probe(int mode, void *dst, const void *src, size_t bytes, void *stream) {
    if (!dst || bytes == 0) return KVP_ERR_ARG;
    if (!aligned(dst, 256)) return KVP_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    static int occ_store = 0, occ_copy = 0;
    switch (mode) {
        case KVP_PROBE_STORE: {
            if (bytes % 16) return KVP_ERR_SIZE;
            if (occ_store == 0 &&
                (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_store, probe_store, PROBE_THREADS, 0) !=
                     cudaSuccess || occ_store < 1))
                occ_store = 1;
            probe_store<<<sm_count() * occ_store, PROBE_THREADS, 0, st>>>(static_cast<uint4 *>(dst), bytes / 16);
            break;
        }
        case KVP_PROBE_COPY: {
            if (!src) return KVP_ERR_ARG;
            if (!aligned(src, 256)) return KVP_ERR_ALIGN;
            if (bytes % 16) return KVP_ERR_SIZE;
            if (occ_copy == 0 &&
                (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_copy, probe_copy, PROBE_THREADS, 0) !=
                     cudaSuccess || occ_copy < 1))
                occ_copy = 1;
            probe_copy<<<sm_count() * occ_copy, PROBE_THREADS, 0, st>>>(static_cast<uint4 *>(dst),
                                                                     static_cast<const uint4 *>(src), bytes / 16);
            break;
        }
        case KVP_PROBE_BULK_STORE: {
            if (bytes % PROBE_TILE) return KVP_ERR_SIZE;
            const uint64_t tiles = bytes / PROBE_TILE;
            const uint64_t blocks = (tiles + PROBE_WARPS - 1) / PROBE_WARPS;
            if (blocks > 0x7FFFFFFFull) return KVP_ERR_SIZE;
            probe_bulk_store<<<unsigned(blocks), PROBE_THREADS, 0, st>>>(static_cast<uint8_t *>(dst), tiles);
            break;
        }
        default:
            return KVP_ERR_ARG;
    }
    count_launch(1);
    return launch_status();
}
