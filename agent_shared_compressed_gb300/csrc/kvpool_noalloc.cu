// kvpool_noalloc.cu -- kvpool_encode for callers that cannot allocate device
// memory.
//
// kvpool_encode takes a caller-provided workspace for its per-block partial
// maxima, value-block error flags and per-layer key parameters.  Some callers
// have no way to provide one: a plug-in loaded into another program's process
// that must not allocate behind its host's memory manager (for instance a
// server whose caching allocator already holds the GPU memory), or a caller on
// a latency-critical path where a cudaMalloc may synchronise the device.  For
// them, kvpool_encode_noalloc runs the same encoder with the workspace taken
// from a fixed array in the library's own device memory.
//
// The array is a file-scope __device__ variable of KVP_NOALLOC_SCRATCH_BYTES:
// every GPU on which the library is loaded holds it until the process exits.
// Host code cannot use the array's name as a device address, so the first
// call on each device looks the address up with cudaGetSymbolAddress (with
// that device current) and caches it.
#include "kvp_internal.cuh"

namespace kvp {

static __device__ __align__(256) uint8_t g_encode_scratch[KVP_NOALLOC_SCRATCH_BYTES];

constexpr int NOALLOC_MAX_DEVICES = 64;
static void *g_scratch_addr[NOALLOC_MAX_DEVICES] = {nullptr};

// Device address of the scratch array on the current device (nullptr on
// failure).  Done once per device.
static void *scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NOALLOC_MAX_DEVICES) return nullptr;
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_encode_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace kvp

using namespace kvp;

extern "C" int kvpool_encode_noalloc(const kvp_shape *s, const void *const *k_layers, const void *const *v_layers,
                                     void *pool, size_t pool_bytes, void *stream) {
    const size_t need = kvpool_workspace_bytes(s);
    if (need == 0) {
        const int rc = shape_ok(s);
        return rc != KVP_OK ? rc : KVP_ERR_ARG;
    }
    if (need > size_t(KVP_NOALLOC_SCRATCH_BYTES)) return KVP_ERR_SIZE;
    void *ws = scratch_address();
    if (ws == nullptr) return KVP_ERR_CUDA;
    return kvpool_encode(s, k_layers, v_layers, pool, pool_bytes, ws, size_t(KVP_NOALLOC_SCRATCH_BYTES), stream);
}
