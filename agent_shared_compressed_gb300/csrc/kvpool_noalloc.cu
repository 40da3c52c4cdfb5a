// kvpool_noalloc.cu -- kvpool_encode for callers that cannot allocate device
// memory.
//
// kvpool_encode takes a caller-provided workspace for its work-queue control
// block and per-layer key parameters.  Some callers
// have no way to provide one: a plug-in loaded into another program's process
// that must not allocate behind its host's memory manager (for instance a
// server whose caching allocator already holds the GPU memory), or a caller on
// a latency-critical path where a cudaMalloc may synchronise the device.  For
// them, kvpool_encode_noalloc runs the same encoder with the workspace taken
// from a fixed array in the library's own device memory.
//
// The array is a file-scope __device__ variable of KVP_NOALLOC_SCRATCH_BYTES:
// every GPU on which the library is loaded holds it until the process exits.
// Host code cannot use the array's name as a device address, so the address
// is looked up with cudaGetSymbolAddress, with the device current.  The
// lookup is cached per CUDA context, keyed by the driver's context id, which
// is never reused within a process: after cudaDeviceReset (or any teardown
// and re-creation of the primary context) the next call sees a new id and
// looks the address up again instead of handing the encoder a stale one.
#include <cuda.h>

#include <mutex>

#include "kvp_internal.cuh"

namespace kvp {

static __device__ __align__(256) uint8_t g_encode_scratch[KVP_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*ctx_get_current_fn)(CUcontext *);
typedef CUresult (*ctx_get_id_fn)(CUcontext, unsigned long long *);

constexpr int NOALLOC_CACHE = 16;
struct ScratchEntry {
    unsigned long long ctx_id;
    void *addr;
};
static std::mutex g_scratch_mu;
static ScratchEntry g_scratch_cache[NOALLOC_CACHE];
static int g_scratch_used = 0, g_scratch_next = 0;

// Id of the CUDA context current on this thread.  False if none is current
// yet (the runtime binds the device's primary context on its first call on a
// thread) or the driver cannot say.
static bool current_context_id(unsigned long long *id) {
    static ctx_get_current_fn get_current = nullptr;
    static ctx_get_id_fn get_id = nullptr;
    static bool resolved = false;
    if (!resolved) {  // called under g_scratch_mu
        cudaDriverEntryPointQueryResult q1, q2;
        void *f1 = nullptr, *f2 = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
            return false;
        get_current = reinterpret_cast<ctx_get_current_fn>(f1);
        get_id = reinterpret_cast<ctx_get_id_fn>(f2);
        resolved = true;
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current context (nullptr on
// failure).  Looked up once per context; a context the driver cannot name is
// looked up on every call.
static void *scratch_address() {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    unsigned long long id = 0;
    bool have_id = current_context_id(&id);
    if (have_id)
        for (int i = 0; i < g_scratch_used; i++)
            if (g_scratch_cache[i].ctx_id == id) return g_scratch_cache[i].addr;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_encode_scratch) != cudaSuccess || p == nullptr) return nullptr;
    if (!have_id) have_id = current_context_id(&id);  // the lookup has bound the primary context
    if (have_id) {
        const int slot = g_scratch_used < NOALLOC_CACHE ? g_scratch_used++ : (g_scratch_next++ % NOALLOC_CACHE);
        g_scratch_cache[slot] = ScratchEntry{id, p};
    }
    return p;
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
    if (ws == nullptr) {
        (void)cudaGetLastError();  // leave no sticky error for the next, unrelated call to report
        return KVP_ERR_CUDA;
    }
    return kvpool_encode(s, k_layers, v_layers, pool, pool_bytes, ws, size_t(KVP_NOALLOC_SCRATCH_BYTES), stream);
}
