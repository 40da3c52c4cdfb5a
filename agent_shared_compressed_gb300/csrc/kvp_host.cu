// kvp_host.cu -- host-side parts of the C ABI that launch no kernel: sizes,
// status read-back, error text, launch accounting.
#include <atomic>

#include "kvp_internal.cuh"

namespace kvp {

static std::atomic<uint64_t> g_launches{0};

void count_launch(int n) { g_launches.fetch_add(uint64_t(n), std::memory_order_relaxed); }

int launch_status() { return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA; }

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
}

int shape_ok(const kvp_shape *s) {
    if (!s) return KVP_ERR_ARG;
    if (s->n_layers <= 0 || s->n_kv_heads <= 0 || s->n_tokens <= 0) return KVP_ERR_ARG;
    if (s->n_layers > KVP_MAX_LAYERS) return KVP_ERR_SIZE;
    if (s->head_dim != 64 && s->head_dim != 128) return KVP_ERR_UNSUPPORTED_D;
    // vectors per layer and elements per layer must fit the kernels' indexing
    const uint64_t nv = uint64_t(s->n_kv_heads) * uint64_t(s->n_tokens);
    if (nv >= (1ull << 31)) return KVP_ERR_SIZE;
    return KVP_OK;
}

}  // namespace kvp

using namespace kvp;

extern "C" {

size_t kvpool_pool_bytes(const kvp_shape *s) {
    if (shape_ok(s) != KVP_OK) return 0;
    return size_t(pool_geom(s->n_layers, s->n_kv_heads, s->head_dim, s->n_tokens).total);
}

const char *kvp_strerror(int st) {
    switch (st) {
        case KVP_OK: return "ok";
        case KVP_ERR_ARG: return "invalid argument (null pointer, count or range)";
        case KVP_ERR_UNSUPPORTED_D: return "unsupported head_dim (64 or 128)";
        case KVP_ERR_ALIGN: return "pointer not aligned as required";
        case KVP_ERR_SIZE: return "buffer too small or shape too large";
        case KVP_ERR_CUDA: return "CUDA call or kernel launch failed";
        case KVP_ERR_NONFINITE: return "input holds Inf or NaN";
        case KVP_ERR_RANGE: return "a scale or zero point overflowed fp16";
        case KVP_ERR_BITS: return "CacheCard bitwidth not in {2,4,8,16}";
        case KVP_ERR_HEADER: return "not a pool / card, or its shape does not match";
        case KVP_ERR_TIMEOUT: return "a bounded device-side wait ran out";
        default: return "unknown status";
    }
}

uint64_t kvp_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

static int flags_to_status(uint32_t f) {
    if (f & FLAG_HEADER) return KVP_ERR_HEADER;
    if (f & FLAG_TIMEOUT) return KVP_ERR_TIMEOUT;
    if (f & FLAG_BITS) return KVP_ERR_BITS;
    if (f & FLAG_SIZE) return KVP_ERR_SIZE;
    if (f & FLAG_NONFINITE) return KVP_ERR_NONFINITE;
    if (f & FLAG_RANGE) return KVP_ERR_RANGE;
    return KVP_OK;
}

int kvpool_status(const void *pool, void *stream) {
    if (!pool) return KVP_ERR_ARG;
    uint32_t h[8];
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(h, pool, sizeof h, cudaMemcpyDeviceToHost, st) != cudaSuccess) return KVP_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KVP_ERR_CUDA;
    if (h[0] != POOL_MAGIC || h[1] != POOL_VERSION) return KVP_ERR_HEADER;
    return flags_to_status(h[POOL_ERR_WORD]);
}

int cachecard_read_header(const void *card, kvp_card_header *out, void *stream) {
    if (!card || !out) return KVP_ERR_ARG;
    static_assert(sizeof(kvp_card_header) == 128, "CacheCard header is 128 bytes");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(out, card, sizeof *out, cudaMemcpyDeviceToHost, st) != cudaSuccess) return KVP_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KVP_ERR_CUDA;
    if (out->magic != CARD_MAGIC || out->version != CARD_VERSION) return KVP_ERR_HEADER;
    return KVP_OK;
}

int cachecard_status(const void *card, void *stream) {
    kvp_card_header h;
    int rc = cachecard_read_header(card, &h, stream);
    if (rc != KVP_OK) return rc;
    return flags_to_status(h.error);
}

size_t cachecard_bytes(const kvp_shape *s, const uint8_t *bits) {
    if (shape_ok(s) != KVP_OK || !bits) return 0;
    uint64_t sum = 0;
    for (int t = 0; t < s->n_tokens; t++) {
        if (!valid_bits(bits[t])) return 0;
        sum += card_record_bytes(bits[t], s->n_kv_heads, s->head_dim);
    }
    if (sum >= (1ull << 32)) return 0;  // record offsets are 32-bit
    return size_t(card_off_layers(s->n_tokens) + uint64_t(s->n_layers) * align256(sum));
}

}  // extern "C"
