/*
 * kvpool.h -- C ABI of the GB300 (sm_103a) KV-cache codec for multi-agent
 * KV sharing.
 *
 * Two containers, both position-independent byte blobs in device memory:
 *
 *  SharedKVPool -- "PolyKV: A Shared Asymmetrically-Compressed KV Cache Pool
 *    for Multi-Agent LLM Inference", 2.A (write once, read many; one object
 *    whose size does not depend on the number of agents) and 2.B (keys int8
 *    with one symmetric scale per layer tensor; values rotated by a fast
 *    Walsh-Hadamard transform, normalised, mapped to the 8-level Lloyd-Max
 *    codebook for N(0,1) and packed at 3 bits).
 *
 *  CacheCard -- "QKVShare: Quantized KV-Cache Handoff for Multi-Agent
 *    On-Device LLMs", Methodology 1-3 (per-token bitwidth from {2,4,8,16},
 *    quantized KV groups plus metadata seq_len / model_id / position offset;
 *    the receiver rebuilds 16-bit past_key_values from it).
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - KV tensors are bf16, one tensor per layer, layout [H][T][d] contiguous
 *    (the Hugging Face past_key_values layout at batch 1).  head_dim d must
 *    be 64 or 128.
 *  - Arrays of per-layer tensor pointers (k_layers, k_dst, ...) are HOST
 *    arrays of DEVICE pointers; the library reads them during the call only
 *    (they are copied into the kernel launch), so the caller may reuse them
 *    as soon as the call returns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every compute call only enqueues work on that stream and
 *    returns; it never allocates, frees or synchronises device memory.  The
 *    only synchronising calls are kvpool_status, cachecard_status and
 *    cachecard_read_header, which say so.
 *  - The caller owns every buffer.  Device pointers to KV tensors must be
 *    16-byte aligned; pool and card buffers 256-byte aligned; workspaces
 *    16-byte aligned.
 *  - Errors: 0 is success, negative values are KVP_ERR_*.  Everything the
 *    host can check (null pointers, shapes, alignment, buffer sizes) is
 *    checked before any work is enqueued, and nothing is enqueued on error.
 *    Conditions only the device can see (non-finite input, a value whose
 *    fp16 scale overflows, an invalid bitwidth in device memory) are
 *    recorded in an error word inside the pool / card header and returned
 *    by the *_status calls.  No kernel traps or asserts.  Two kinds of
 *    device-side wait exist, both bounded: the pool encoder's key-quantize
 *    work waits for its layer's scale, released by another block of the same
 *    kernel; pool attention and CacheCard unpack wait on mbarriers for their
 *    own bulk copies into shared memory.  A wait that runs out is recorded in
 *    the pool's or the card's error word and reported as KVP_ERR_TIMEOUT by
 *    kvpool_status / cachecard_status; the CUDA context stays usable.
 */
#ifndef KVPOOL_H
#define KVPOOL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define KVP_OK 0
#define KVP_ERR_ARG (-1)            /* null pointer, bad count or range      */
#define KVP_ERR_UNSUPPORTED_D (-2)  /* head_dim other than 64 or 128         */
#define KVP_ERR_ALIGN (-3)          /* pointer not aligned as required       */
#define KVP_ERR_SIZE (-4)           /* buffer too small / shape too large    */
#define KVP_ERR_CUDA (-5)           /* a CUDA call or kernel launch failed   */
#define KVP_ERR_NONFINITE (-6)      /* input held Inf or NaN                 */
#define KVP_ERR_RANGE (-7)          /* a scale or zero point overflowed fp16 */
#define KVP_ERR_BITS (-8)           /* CacheCard bitwidth not in {2,4,8,16}  */
#define KVP_ERR_HEADER (-9)         /* not a pool / card, or shape mismatch  */
#define KVP_ERR_TIMEOUT (-10)       /* a bounded device-side wait ran out    */

/* Largest layer count one call accepts. */
#define KVP_MAX_LAYERS 512

/* Key formats of a pool (the pool header records which one it holds). */
#define KVP_K_PER_TENSOR 0  /* one fp32 scale per layer's key tensor ("PolyKV" 2.B.1 text) */
#define KVP_K_Q8_0 1        /* q8_0 blocks: 32 keys along d share an fp16 scale (the label
                               "q8_0" that "PolyKV" 2.B.1 gives the same step)            */

/* Shape of one KV cache: n_layers tensors of [n_kv_heads][n_tokens][head_dim]. */
typedef struct kvp_shape {
    int32_t n_layers;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t n_tokens;
} kvp_shape;

/* CacheCard header, byte-for-byte the first 128 bytes of a card. */
typedef struct kvp_card_header {
    uint32_t magic;         /* 0x4343564B, bytes "KVCC"                        */
    uint32_t version;       /* 1                                              */
    int32_t seq_len;        /* T                                              */
    int32_t n_layers;       /* L                                              */
    int32_t n_kv_heads;     /* H                                              */
    int32_t head_dim;       /* d                                              */
    int32_t group_size;     /* 32                                             */
    int32_t dtype;          /* 1 = bf16                                       */
    uint64_t model_id;      /* opaque id of the model that produced the cache */
    int64_t pos_offset;     /* position of token 0 in the sender's sequence   */
    uint64_t off_bits;      /* byte offset of uint8 bits[T]                    */
    uint64_t off_offsets;   /* byte offset of uint32 off[T] (record offsets)   */
    uint64_t off_layers;    /* byte offset of layer 0's records                */
    uint64_t layer_stride;  /* bytes per layer                                 */
    uint64_t total_bytes;   /* bytes of the whole card                         */
    uint32_t error;         /* device-detected error bits                      */
    uint32_t reserved[9];
} kvp_card_header;

/* ---------------------------------------------------------------------- */
/* SharedKVPool                                                            */
/* ---------------------------------------------------------------------- */

/* Exact byte size of the pool for this shape, or 0 for an invalid shape.
 * Independent of how many agents will read it ("PolyKV" 2.A).
 * Pool layout (every section 256-byte aligned): 256-byte header (magic
 * "KVPL", version 1, L, H, d, T, error word, section offsets), fp32 K scale
 * per layer, then per layer: int8 K codes [H][T][d], 3-bit V codes
 * [H][T][3d/8] (8 codes c_0..c_7 = the 24-bit little-endian word
 * sum c_j << 3j), fp16 sigma [H][T]. */
size_t kvpool_pool_bytes(const kvp_shape *shape);

/* Bytes of device workspace kvpool_encode needs for this shape (0 for an
 * invalid shape).  The workspace holds the encoder's work-queue control
 * block (queue head, per-layer key maxima and ready flags) and per-layer
 * quantization parameters; its contents need no initialisation and are
 * dead after the encode's kernels finish. */
size_t kvpool_workspace_bytes(const kvp_shape *shape);

/* Encode a whole KV cache into a pool ("PolyKV" 2.B).
 *  k_layers, v_layers: host arrays of n_layers device pointers, each a bf16
 *    [H][T][d] tensor (16-byte aligned).
 *  Keys: per layer, s = max|k| / 127 rounded once to fp32; code = the
 *    integer nearest to the exact k/s (ties to even), in [-127,127]; s = 0
 *    gives all-zero codes.
 *  Values: per (token, head) vector v, y = H_d v (Sylvester-order
 *    Walsh-Hadamard), sigma = ||v||/sqrt(d) stored as fp16, u = y/||v||, and
 *    code = number of Lloyd-Max thresholds (midpoints of
 *    +-0.2451/0.7560/1.3440/2.1520) not above u; a zero vector codes as 4.
 *  pool: pool_bytes >= kvpool_pool_bytes(shape), 256-byte aligned; fully
 *    overwritten.  ws: ws_bytes >= kvpool_workspace_bytes(shape).
 * Non-finite input or a sigma above the fp16 range is reported by
 * kvpool_status (the affected codes are then unspecified). */
int kvpool_encode(const kvp_shape *shape, const void *const *k_layers,
                  const void *const *v_layers, void *pool, size_t pool_bytes,
                  void *ws, size_t ws_bytes, void *stream);

/* Pool bytes for key format k_mode (KVP_K_PER_TENSOR: as kvpool_pool_bytes;
 * KVP_K_Q8_0: that plus the block scales, 2 * n_layers * H * T * d/32 bytes
 * rounded up to 256).  0 for an invalid shape or format. */
size_t kvpool_pool_bytes_ex(const kvp_shape *shape, int k_mode);

/* kvpool_encode with the key format chosen by k_mode.  KVP_K_PER_TENSOR is
 * kvpool_encode.  KVP_K_Q8_0 ("PolyKV" 2.B.1 labels the key step "q8_0"):
 * every 32 consecutive keys of a vector share the scale
 * s_b = fp16(max|k| / 127) (round to nearest even); code = the integer
 * nearest to the exact k / s_b (ties to even) clamped to [-127, 127] (the
 * clamp only acts when s_b is an fp16 subnormal); s_b = 0 gives codes 0.  No
 * layer-wide maximum is needed, so keys and values are encoded in one pass.
 * Values as kvpool_encode.  pool_bytes >= kvpool_pool_bytes_ex(shape,
 * k_mode); ws as kvpool_encode.  A block whose scale overflows fp16 is
 * reported as KVP_ERR_RANGE by kvpool_status, non-finite keys as
 * KVP_ERR_NONFINITE (they code as 0).  Returns KVP_ERR_ARG for an unknown
 * k_mode. */
int kvpool_encode_ex(const kvp_shape *shape, int k_mode, const void *const *k_layers,
                     const void *const *v_layers, void *pool, size_t pool_bytes,
                     void *ws, size_t ws_bytes, void *stream);

/* Fan-out decode ("PolyKV" 2.A PooledAgent, 2.B.2 dequantization): read
 * layers [layer_begin, layer_end) of the pool once and write the decoded
 * bf16 K and V into each of n_agents caches.
 *  K: bf16(q * s_l), or bf16(q * s_b) with the key's block scale in a
 *    q8_0 pool (the format is read from the pool header on the device).
 *    V: bf16(sigma_h * (H_d c) / sqrt(d)) with c the centroids of the codes
 *    (the orthonormal transform is its own inverse).
 *  shape must equal the shape the pool was encoded with.
 *  k_dst, v_dst: host arrays of n_agents * n_layers device pointers,
 *    agent-major (entry a * n_layers + l is agent a's layer l, a bf16
 *    [H][T][d] tensor, 16-byte aligned).  Only entries of layers in the
 *    range are read; the others may be NULL.
 * The pool is only read, so decodes of one pool may run concurrently on
 * several streams.  A pool whose header does not match `shape` is left
 * undecoded and kvpool_status reports KVP_ERR_HEADER. */
int kvpool_decode_into(const void *pool, const kvp_shape *shape, int layer_begin,
                       int layer_end, int n_agents, void *const *k_dst,
                       void *const *v_dst, void *stream);

/* Synchronises `stream`, then returns KVP_OK or the first device-detected
 * error recorded in the pool's header (KVP_ERR_HEADER if `pool` does not
 * hold a version-1 pool). */
int kvpool_status(const void *pool, void *stream);

/* Size of the library's own device scratch array used by
 * kvpool_encode_noalloc (256 KiB on every GPU that loads the library, held
 * until the process exits). */
#define KVP_NOALLOC_SCRATCH_BYTES 262144

/* kvpool_encode without a caller workspace.  This entry point has no
 * counterpart in the papers; it exists for callers that cannot allocate
 * device memory -- e.g. a plug-in inside another program's process that must
 * not allocate behind its host's memory manager, or a latency-critical caller
 * for which a cudaMalloc could synchronise the device.  It allocates nothing
 * (no cudaMalloc, cudaFree or allocating library call): the workspace is a
 * fixed array of KVP_NOALLOC_SCRATCH_BYTES in the library's device memory.
 *  Arguments and results are those of kvpool_encode minus ws / ws_bytes.
 *  The encoder's workspace is a control block of about 6 KB plus 16 bytes
 *    per layer, so every shape kvpool_encode accepts fits in the array.  A
 *    shape it refuses is refused here with the same code, before anything
 *    is enqueued.
 *  The first call in each CUDA context looks up the array's device address
 *    (with that context current) and caches it under the driver's context
 *    id; make that first call before any stream capture.  A context created
 *    later (after cudaDeviceReset, say) gets a fresh lookup on its first
 *    call, so the library may outlive a context.
 *  Every call on a device shares the one array.  The encoder overwrites
 *    everything it reads from it, so nothing needs clearing between calls,
 *    but calls that overlap on the GPU (other streams, no ordering between
 *    them) race on the array: order them on one stream or with events. */
int kvpool_encode_noalloc(const kvp_shape *shape, const void *const *k_layers,
                          const void *const *v_layers, void *pool, size_t pool_bytes,
                          void *stream);

/* ---------------------------------------------------------------------- */
/* Attention over the pool                                                 */
/* ---------------------------------------------------------------------- */

/* Bytes of device workspace kvpool_attend needs (0 for an invalid shape or
 * head count).  Holds per-split partial results; no initialisation. */
size_t kvpool_attend_workspace_bytes(const kvp_shape *shape, int n_agents, int n_q_heads);

/* One decode step of attention of n_agents agents' queries over layer
 * `layer` of the pool, computed from the compressed bytes without writing any
 * bf16 cache: the fused attention over the quantized cache that "QKVShare"
 * (Significance) leaves as future work, on "PolyKV" 2.A's shared pool.
 *  q: device bf16 [n_agents][n_q_heads][head_dim], 16-byte aligned; query head
 *    j reads KV head j / (n_q_heads / n_kv_heads) (n_q_heads a multiple of
 *    n_kv_heads: grouped-query attention).
 *  For each (agent, head): s_t = scale * (q . k_t) over the T pooled tokens
 *    with k_t = code_t * s_layer (q8_0 pools: code * s_b per 32-key block;
 *    the format is read from the pool header); out = sum_t softmax(s)_t v_t with v_t the
 *    decoded value (sigma_t * H_d c_t / sqrt(d), accumulated in the rotated
 *    domain and transformed once); lse = log sum_t exp(s_t) (natural log), so a
 *    caller can merge with attention over its own further tokens.
 *  out: device fp32 [n_agents][n_q_heads][head_dim] (16-byte aligned); lse:
 *    device fp32 [n_agents][n_q_heads].  ws: kvpool_attend_workspace_bytes.
 *  Precision: scores are exact products accumulated in fp32 (q8_0: exact
 *  per-block partial sums, each scaled by its block scale in fp32);
 *  probabilities times sigma enter the value product as fp16, centroids as
 *  fp16.  A pool whose header does not match `shape` is not read and
 *  kvpool_status reports KVP_ERR_HEADER.  The kernel streams the pool's bytes
 *  into shared memory with bulk copies and waits on them for at most about
 *  half a second; should a wait run out, out / lse are unspecified and
 *  kvpool_status reports KVP_ERR_TIMEOUT.  Errors are recorded in the pool's
 *  error word (the only bytes of the pool a call may write). */
int kvpool_attend(const void *pool, const kvp_shape *shape, int layer, int n_agents, int n_q_heads,
                  const void *q, float scale, float *out, float *lse, void *ws, size_t ws_bytes,
                  void *stream);

/* Bytes of device workspace kvpool_attend_lora needs (0 for an invalid shape,
 * head count or rank). */
size_t kvpool_attend_lora_workspace_bytes(const kvp_shape *shape, int n_agents, int n_q_heads, int rank);

/* Pool attention for agents that differ by a LoRA adapter on the value
 * projection, with one shared low-rank cache ("LRAgent": BaseLRShared shares
 * the base cache and the low-rank cache X A between agents, each agent keeping
 * its own up-projection B; Flash-LoRA-Attention computes
 * P (V_base + V_lr B) as P V_base + (P V_lr) B, so the up-projection is
 * applied once per query instead of expanding the cache).  Agent a's value of
 * token t at KV head h is
 *   v = (the pool's decoded value) + sum_k v_lr[t][k] * lora_b[a][k][h*d + i];
 * otherwise as kvpool_attend (same out, lse, GQA map and key formats).
 *  rank: 16 or 32 (KVP_ERR_ARG otherwise).
 *  v_lr: device bf16 [n_tokens][rank], the layer's shared low-rank cache
 *    (16-byte aligned).  It enters the product as fp16: exact for values in
 *    fp16's normal range, |x| in [2^-14, 65504].
 *  lora_b: device bf16 [n_agents][rank][n_kv_heads * head_dim], each agent's
 *    up-projection with rank-major rows (the transpose of a PyTorch LoRA
 *    B weight), 16-byte aligned.
 *  ws: kvpool_attend_lora_workspace_bytes. */
int kvpool_attend_lora(const void *pool, const kvp_shape *shape, int layer, int n_agents, int n_q_heads,
                       const void *q, float scale, int rank, const void *v_lr, const void *lora_b, float *out,
                       float *lse, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* CacheCard                                                               */
/* ---------------------------------------------------------------------- */

/* Exact byte size of a card for these per-token bitwidths (host array of
 * n_tokens values), or 0 if the shape or any bitwidth is invalid.
 * Card layout: 128-byte header (kvp_card_header), uint8 bits[T], uint32
 * off[T] (16-byte aligned; exclusive prefix sum of record sizes), then
 * n_layers layers of layer_stride bytes (256-byte aligned).  A token's
 * record in one layer, b in {2,4,8}: K codes [H][d] then V codes [H][d] at b
 * bits (each group of 32 coordinates a little-endian bit string, code j at
 * bits j*b..j*b+b-1), then K (fp16 scale, fp16 zero) [H][d/32], then V
 * (scale, zero) [H][d/32]; b = 16: K then V verbatim.  Records are padded to
 * 16 bytes. */
size_t cachecard_bytes(const kvp_shape *shape, const uint8_t *bits_host);

/* Pack a CacheCard ("QKVShare" Methodology 1-2).
 *  bits_dev: device array of n_tokens bitwidths in {2,4,8,16}.
 *  For b < 16, per group of 32 coordinates of one (layer, token, K|V, head):
 *    s_h = fp16((max-min)/(2^b-1)), z_h = fp16(min), code =
 *    clamp(nearest integer to (x - z_h)/s_h, 0, 2^b-1) (0 when s_h = 0).
 *    b = 16 copies the bf16 values.
 *  card: card_bytes bytes, 256-byte aligned; must hold cachecard_bytes()
 *    for these bits, otherwise nothing but the header is written and
 *    cachecard_status reports KVP_ERR_SIZE (KVP_ERR_BITS for an invalid
 *    bitwidth). */
int cachecard_pack(const kvp_shape *shape, uint64_t model_id, int64_t pos_offset,
                   const uint8_t *bits_dev, const void *const *k_layers,
                   const void *const *v_layers, void *card, size_t card_bytes,
                   void *stream);

/* Copy the card's 128-byte header to *out (synchronises `stream`).  Returns
 * KVP_ERR_HEADER if the magic or version is wrong. */
int cachecard_read_header(const void *card, kvp_card_header *out, void *stream);

/* Receiver injection ("QKVShare" Methodology 3): rebuild every layer's bf16
 * K and V ([H][T][d]) from the card: x = bf16(q * s_h + z_h), 16-bit tokens
 * verbatim.  hdr is the header read by cachecard_read_header.  k_dst, v_dst:
 * host arrays of n_layers device pointers (16-byte aligned).  The header's
 * fields are checked on the host (KVP_ERR_HEADER); a token whose bitwidth is
 * invalid or whose record offset is not 16-byte aligned or does not fit the
 * layer stride is left unwritten, and cachecard_status then reports
 * KVP_ERR_HEADER.  Where the shape allows it (see kvp_test_limit_next_unpack)
 * records are staged through shared memory by bulk copies. */
int cachecard_unpack(const void *card, const kvp_card_header *hdr,
                     void *const *k_dst, void *const *v_dst, void *stream);

/* Receiver injection at other positions: as cachecard_unpack, but every key
 * is moved from its position in the sender's sequence (hdr->pos_offset + t)
 * to pos_dst + t.  The card's metadata carries the position offset
 * ("QKVShare" Methodology 2), and a reused segment's key positions are
 * re-aligned to the target agent's ("KVCMAS", How it is used).  Under rotary
 * position embedding -- dims i and i + d/2 turned through p * w_i at
 * position p, the Hugging Face Llama pairing -- that is one further turn of
 * every pair through (pos_dst - hdr->pos_offset) * w_i.
 *   inv_freq: HOST array of head_dim/2 fp32 frequencies w_i (radians per
 *     position; the model's rotary inverse frequencies, any scaling already
 *     applied).  Copied into the launch, so it may be freed on return.
 *   The angle is formed and its sine and cosine taken in fp64; each key is
 *   dequantized and turned in fp32 and rounded to bf16 once.  Values are
 *   unpacked exactly as by cachecard_unpack.  pos_dst == hdr->pos_offset
 *   gives cachecard_unpack's output bit for bit.
 * Returns KVP_ERR_ARG for a null inv_freq, a non-finite frequency or a shift
 * that overflows int64; otherwise as cachecard_unpack. */
int cachecard_unpack_at(const void *card, const kvp_card_header *hdr, int64_t pos_dst,
                        const float *inv_freq, void *const *k_dst, void *const *v_dst,
                        void *stream);

/* Synchronises `stream`, then returns KVP_OK or the first device-detected
 * error recorded in the card's header. */
int cachecard_status(const void *card, void *stream);

/* ---------------------------------------------------------------------- */
/* Diagnostics                                                             */
/* ---------------------------------------------------------------------- */

/* Static, human-readable text for a status code. */
const char *kvp_strerror(int status);

/* Number of kernels this library has launched in this process. */
uint64_t kvp_launch_count(void);

/* Bandwidth probes (the papers have no counterpart: measurement support).
 * They give the HBM ceiling of the access pattern each codec kernel uses, so
 * a benchmark can report a kernel against its own pattern's ceiling.
 *  KVP_PROBE_STORE: write `bytes` to dst with 16-byte streaming stores, one
 *    resident grid walking the buffer (the one-agent decode's and the card
 *    unpack's store pattern).  bytes a multiple of 16.
 *  KVP_PROBE_BULK_STORE: write `bytes` to dst as 4 KB bulk copies from
 *    shared memory, one per warp (the fan-out decode's store pattern).
 *    bytes a multiple of 4096.
 *  KVP_PROBE_COPY: copy `bytes` from src to dst with 16-byte loads and
 *    stores (read + write).  bytes a multiple of 16; src 256-byte aligned.
 * dst: device buffer of at least `bytes`, 256-byte aligned; its contents are
 * overwritten with an arbitrary pattern.  Enqueues one kernel on `stream`.
 * Returns KVP_ERR_ARG (unknown mode, null pointer, zero bytes),
 * KVP_ERR_ALIGN or KVP_ERR_SIZE before launching anything. */
#define KVP_PROBE_STORE 0
#define KVP_PROBE_BULK_STORE 1
#define KVP_PROBE_COPY 2
int kvp_bandwidth_probe(int mode, void *dst, const void *src, size_t bytes, void *stream);

/* Failure-path testing.  The pool encoder's key-quantization work waits, with
 * an iteration limit, for a per-layer "scale ready" flag set by other blocks
 * of the same kernel; a wait that runs out is reported by kvpool_status as
 * KVP_ERR_TIMEOUT and leaves the CUDA context usable.  Calling this with
 * layer >= 0 makes the NEXT kvpool_encode on this thread leave that layer's
 * flag unset and wait at most spin_iters iterations (about 100 ns each), so
 * a test can exercise that path; layer < 0 restores normal operation.
 * Returns KVP_OK. */
int kvp_test_fail_next_encode(int layer, uint32_t spin_iters);

/* Failure-path testing of pool attention.  Its split kernel waits, with a
 * bounded number of polls, for the bulk copies of each sub-chunk; a wait that
 * runs out is reported by kvpool_status as KVP_ERR_TIMEOUT (the block first
 * lets its copies in flight land, with the normal limit) and leaves the CUDA
 * context usable.  Makes the NEXT kvpool_attend / kvpool_attend_lora on this
 * thread poll each sub-chunk's copies at most `polls` times (0: not at all, so
 * every block gives up on its first sub-chunk).  Returns KVP_OK. */
int kvp_test_limit_next_attend(uint32_t polls);

/* Failure-path testing of CacheCard unpack.  Where the shape lets it stage
 * records in shared memory (d = 128 or an even n_kv_heads, and 32 n_kv_heads
 * head_dim bytes of buffers per block within 96 KB), unpack waits, with a
 * bounded number of polls, for the bulk copies of each record; a wait that
 * runs out is reported by cachecard_status as KVP_ERR_TIMEOUT (the warp
 * first lets its copies in flight land, with the normal limit, and leaves
 * that layer's outputs incomplete) and leaves the CUDA context usable.
 * Makes the NEXT cachecard_unpack / cachecard_unpack_at on this thread poll
 * each record's copies at most `polls` times (0: not at all, so every warp
 * gives up on its first record); other shapes ignore it.  Returns KVP_OK. */
int kvp_test_limit_next_unpack(uint32_t polls);

#ifdef __cplusplus
}
#endif

#endif /* KVPOOL_H */
