/*
 * kvarn.h -- C ABI of the KVarN KV-cache hot path on GB300 (sm_103a).
 *
 * The method (sources are web write-ups of KVarN; titles as published):
 *  - "KVarN: 2-Bit KV-Cache That Beats FP16 Throughput, and Where the Catch
 *    Lives", section "What KVarN does differently": each KV tile is rotated
 *    by a Hadamard transform along the channel dimension, then its variance
 *    is equalised by a Sinkhorn-like alternation of column and row
 *    standard-deviation normalisation in log space.
 *  - "Huawei's KVarN puts KV-cache quantization inside vLLM's backend",
 *    section "What KVarN changes in vLLM's serving path": preset
 *    kvarn_k4v2_g128 stores 4-bit keys and 2-bit values per 128-token tile
 *    (one paged block) with dual FP8 scales and FP16 zero-points; section
 *    "The four-stage pipeline": rotation, variance normalisation, asymmetric
 *    round-to-nearest, and dequantisation at read time inside attention;
 *    FAQ "Is the tile size configurable": the tile is fixed at 128 tokens.
 *
 * Conventions for every entry point:
 *  - All pointers documented "device" are CUDA device pointers the caller
 *    owns and keeps alive until the stream work completes.  The library
 *    allocates nothing.  Its only process-wide state is the fixed scratch
 *    array of kvarn_decode_attention_noalloc and host-side caches filled on
 *    first use and never changed afterwards: the array's device address per
 *    device, the driver's tensor-map encoder entry point, and per kernel a
 *    mark of the devices on which its shared-memory limit is already set.
 *    They are safe to fill from several host threads at once.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL is the legacy default stream).  Device pointers must be 16-byte
 *    aligned; the library checks this on the host.
 *  - Host-side validation fails synchronously with KVARN_ERR_INVALID (bad
 *    argument) or KVARN_ERR_UNSUPPORTED (a configuration the library does not
 *    implement) and launches nothing.  A failed launch returns
 *    KVARN_ERR_CUDA.
 *  - Faults found on the device (a block id outside [0, num_blocks), a
 *    token index or length out of range) store the first error code into
 *    *dev_err (a device int32 the caller zeroes) and the affected unit skips
 *    its work.  Kernels never trap and never wait without a bound; a bounded
 *    wait that expires reports KVARN_DEV_ERR_TIMEOUT.  No C++ exception
 *    crosses this interface.
 *
 * Packed format (one record per tile x KV head, 16-byte aligned):
 *   K record 8704 B: g[128] FP8 E4M3 per-channel scale | a[128] FP8 E4M3
 *     per-token step | b[128] FP16 (little-endian) per-token zero-point |
 *     codes[128 tokens][64 B], byte i of token t = code[t][2i] |
 *     code[t][2i+1] << 4.
 *   V record 4608 B: same 512-byte header | codes[128 channels][32 B]:
 *     channel c holds 8 little-endian 32-bit words; word w carries tokens
 *     16w .. 16w+15, token 16w+u at bit u (u even) or bit 15+u (u odd),
 *     i.e. even tokens in the low half-word and odd tokens in the high
 *     half-word, 2 bits each.
 *   K2 record 4608 B (k_bits = 2): same 512-byte header | codes[128 tokens]
 *     [32 B], byte i of token t = sum over k < 4 of code[t][4i+k] << 2k.
 *   V4 record 8704 B (v_bits = 4): same 512-byte header | codes[128
 *     channels][64 B]: channel c holds 16 little-endian 32-bit words; word w
 *     carries tokens 8w .. 8w+7, token 8w+u at bit 2u (u even) or 14+2u (u
 *     odd), 4 bits each.
 *   Block b of the pool = for each KV head h: [K record | V record], i.e.
 *     num_kv_heads * R bytes with R = 13312 (K4/V2), 9216 (K2/V2) or 17408
 *     (K4/V4); head h of block b starts at b * kvarn_block_bytes() + h * R.
 *   Dequantised value (rotated domain): R[t][c] = g[c] * (a[t]*code + b[t]);
 *   the cache value is R H with H the 128-point Sylvester Hadamard matrix
 *   divided by sqrt(128).  4.25 bits/element for K, 2.25 for V (and for
 *   2-bit K).
 *
 * Presets: k_bits = 4, v_bits = 2 is kvarn_k4v2_g128, the one the pages
 * ship.  k_bits = 2, v_bits = 2 (2-bit keys) and k_bits = 4, v_bits = 4
 * (4-bit values, levels 0..15) follow the same kvarn_k<bits>v<bits>_g<tile>
 * naming ("Huawei's KVarN puts KV-cache quantization inside vLLM's
 * backend", section "What KVarN changes in vLLM's serving path"); the pages
 * name no other preset, so their records are the shipped ones with the code
 * field narrowed or widened.  Other combinations return
 * KVARN_ERR_UNSUPPORTED.
 */
#ifndef KVARN_H
#define KVARN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvarn_status {
  KVARN_OK = 0,
  KVARN_ERR_INVALID = 1,     /* bad pointer, size, alignment or stride */
  KVARN_ERR_UNSUPPORTED = 2, /* valid request outside what the library implements */
  KVARN_ERR_CUDA = 3         /* a kernel launch or CUDA runtime call failed */
} kvarn_status;

typedef enum kvarn_dtype {
  KVARN_DTYPE_F16 = 0,
  KVARN_DTYPE_BF16 = 1
} kvarn_dtype;

/* Codes stored into *dev_err by a kernel (first error wins). */
#define KVARN_DEV_ERR_BLOCK_RANGE 1 /* a block id outside [0, num_blocks) */
#define KVARN_DEV_ERR_TOKEN_RANGE 2 /* a token index, position or length out of range */
#define KVARN_DEV_ERR_TIMEOUT 3     /* a bounded wait on an async copy expired */
#define KVARN_DEV_ERR_BOUNDS 4      /* checked (debug) build only: an access outside its buffer was skipped */

typedef struct kvarn_config {
  int32_t head_dim;       /* channels per head; must be 128 */
  int32_t tile_tokens;    /* tokens per tile = paged block size; must be 128 */
  int32_t num_kv_heads;   /* KV heads of the layer, >= 1 */
  int32_t num_q_heads;    /* query heads; a multiple of num_kv_heads with group size <= 8 */
  int32_t num_blocks;     /* blocks in the packed block pool (device bounds check); with 0 blocks
                             the pool pointer may be NULL */
  int32_t k_bits;         /* key code width; 4 or 2 */
  int32_t v_bits;         /* value code width; 2, or 4 with k_bits = 4 */
  int32_t sinkhorn_iters; /* normalisation iterations, 0..64 (the preset uses 8) */
  int32_t dtype;          /* kvarn_dtype of K/V/query inputs and of the open-tile buffer */
} kvarn_config;

/* Bytes of one block of the packed pool: num_kv_heads * (K record + V
 * record): 13312 (K4/V2), 9216 (K2/V2) or 17408 (K4/V4).  0 if cfg is
 * invalid. */
size_t kvarn_block_bytes(const kvarn_config* cfg);

/* Bytes of the open-tile (tail) buffer for `batch` sequences:
 * batch * num_kv_heads * 2 * 128 * 128 * 2.  Layout [seq][kv_head][K=0,V=1]
 * [token slot 0..127][channel], 16-bit elements of cfg->dtype; token p of a
 * sequence lives in slot p % 128 until its tile closes.  0 if invalid. */
size_t kvarn_tail_bytes(const kvarn_config* cfg, int32_t batch);

/*
 * Quantise whole 128-token tiles into the packed pool (write path: rotation,
 * Sinkhorn-like normalisation, FP8/FP16 scales, asymmetric round-to-nearest,
 * bit packing -- the first three stages of "The four-stage pipeline").
 *
 *  k, v              device, 16-bit (cfg->dtype).  Element (token r, head h,
 *                    channel c) at k[r * token_stride_elems + h * 128 + c];
 *                    e.g. a [seq][token][head][128] array flattened over
 *                    (seq, token).  token_stride_elems: multiple of 8,
 *                    >= num_kv_heads * 128.
 *  n_tokens          number of token rows addressable from k and v (bound for
 *                    the device check).
 *  tile_first_token  device int64[n_tiles]: first token row of tile i.
 *  tile_dst_block    device int32[n_tiles]: destination block of tile i; all
 *                    num_kv_heads heads of the tile go into that block.
 *  block_pool        device, num_blocks * kvarn_block_bytes() bytes.
 *  dev_err           device int32 (see above); tiles whose first token or
 *                    block is out of range are skipped.
 * n_tiles == 0 is a no-op.  Records of different tiles must not alias.
 */
kvarn_status kvarn_quantize_tiles(const kvarn_config* cfg, const void* k, const void* v,
                                  int64_t token_stride_elems, int64_t n_tokens,
                                  const int64_t* tile_first_token, const int32_t* tile_dst_block,
                                  int32_t n_tiles, void* block_pool, int32_t* dev_err, void* stream);

/*
 * Append one token per sequence to the open tile; when a tile fills (its
 * 128th token arrives) quantise it into block_table[s][pos/128] (the write
 * path "happens every decode step", "The four-stage pipeline").  The open
 * tile stays raw 16-bit until it fills.
 *
 *  k_new, v_new  device, 16-bit [batch][num_kv_heads][128].
 *  pos           device int32[batch]: position of the new token in its
 *                sequence (0-based); must be >= 0 and pos/128 < max_blocks.
 *  block_table   device int32[batch][max_blocks]: physical block of each
 *                128-token tile of each sequence.
 *  tail_pool     device, kvarn_tail_bytes(cfg, batch) bytes (layout above).
 *  block_pool    device packed pool.
 * Out-of-range positions or blocks set *dev_err and skip that sequence.
 * KVARN_ERR_INVALID if batch * num_kv_heads * 2 exceeds 2^31 - 1.
 */
kvarn_status kvarn_append_tokens(const kvarn_config* cfg, const void* k_new, const void* v_new,
                                 const int32_t* pos, const int32_t* block_table, int32_t max_blocks,
                                 int32_t batch, void* tail_pool, void* block_pool, int32_t* dev_err,
                                 void* stream);

/* Workspace bytes kvarn_decode_attention needs for this batch and table
 * width (split-K partial results).  0 if invalid. */
size_t kvarn_decode_workspace_bytes(const kvarn_config* cfg, int32_t batch, int32_t max_blocks);

/*
 * Decode attention over the packed paged cache plus the raw open tile
 * ("Dequantization at read time", "The four-stage pipeline"): for each
 * sequence s and query head j (KV head j / (num_q_heads/num_kv_heads)),
 *   out[s][j] = softmax(scale * q K^T) V
 * over the seq_lens[s] tokens of s: tiles 0 .. seq_lens[s]/128 - 1 packed in
 * block_table[s][.], then seq_lens[s] % 128 raw tokens in the open tile.
 * Scales and the key rotation are folded into the query, the per-channel
 * value scales into the accumulator, and one inverse rotation is applied to
 * the output.
 *
 *  q           device, 16-bit (cfg->dtype) [batch][num_q_heads][128].
 *  block_table device int32[batch][max_blocks], max_blocks >= 1 (a batch
 *              without a closed tile still passes one column).
 *  seq_lens    device int32[batch]; 0 gives a zero output row; must satisfy
 *              seq_lens[s] <= 128 * max_blocks.
 *  out         device float32 [batch][num_q_heads][128].
 *  workspace   device, >= kvarn_decode_workspace_bytes(cfg, batch, max_blocks).
 */
kvarn_status kvarn_decode_attention(const kvarn_config* cfg, const void* q, const int32_t* block_table,
                                    int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                                    const void* block_pool, const void* tail_pool, float softmax_scale,
                                    float* out, void* workspace, size_t workspace_bytes,
                                    int32_t* dev_err, void* stream);

/* Workspace bytes kvarn_multiquery_attention needs for this batch, table
 * width and query count (split-K partial rows).  0 if invalid. */
size_t kvarn_multiquery_workspace_bytes(const kvarn_config* cfg, int32_t batch, int32_t max_blocks,
                                        int32_t n_queries);

/*
 * Causal attention of several new query tokens per sequence over the packed
 * paged cache plus the raw open tile: the read side of the pages' pipeline
 * ("Huawei's KVarN puts KV-cache quantization inside vLLM's backend",
 * section "The four-stage pipeline": dequantisation at read time inside
 * attention) for a chunk of prefill or a speculative step that verifies
 * several draft tokens.  The caller has already appended the n_queries new
 * tokens (kvarn_append_tokens, kvarn_quantize_tiles), so sequence s holds
 * seq_lens[s] tokens laid out as for kvarn_decode_attention.  Query i of
 * sequence s sits at position seq_lens[s] - n_queries + i and attends to the
 * tokens at positions 0 .. seq_lens[s] - n_queries + i:
 *   out[s][i][j] = softmax(scale * q[s][i][j] K[0..pos]^T) V[0..pos].
 *
 *  q           device, 16-bit (cfg->dtype) [batch][n_queries][num_q_heads][128].
 *  n_queries   1 .. 4096.
 *  seq_lens    device int32[batch]; each must satisfy n_queries <= seq_lens[s]
 *              <= 128 * max_blocks, else KVARN_DEV_ERR_TOKEN_RANGE is stored
 *              and the rows of s are zero.
 *  out         device float32 [batch][n_queries][num_q_heads][128].
 *  workspace   device, >= kvarn_multiquery_workspace_bytes(cfg, batch,
 *              max_blocks, n_queries).
 * Other arguments as kvarn_decode_attention.  The query rows of a KV head
 * (n_queries x group size) run in blocks of 128 on the tensor cores.
 */
kvarn_status kvarn_multiquery_attention(const kvarn_config* cfg, const void* q, int32_t n_queries,
                                        const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                                        int32_t batch, const void* block_pool, const void* tail_pool,
                                        float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                                        int32_t* dev_err, void* stream);

/* Size of the fixed device scratch used by kvarn_decode_attention_noalloc. */
#define KVARN_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * kvarn_decode_attention without a workspace argument, for callers that
 * cannot allocate device memory: for example an inference engine whose
 * memory manager has already reserved the free device memory for its paged
 * cache and forbids ad-hoc allocations, or a latency-critical decode loop in
 * which cudaMalloc/cudaFree would synchronise the device.  The pages describe
 * nothing like it; it is this library's own addition.
 *
 * Arguments, layouts and results are those of kvarn_decode_attention (the
 * caller still passes every input and the output).  The split-K partials go
 * to a fixed device array of KVARN_NOALLOC_SCRATCH_BYTES (16 MiB) that the
 * library defines at file scope; every GPU that loads the library holds it
 * until the process exits.  Nothing is allocated: no cudaMalloc, no cudaFree.
 *  - A request that needs more scratch than that (batch * num_kv_heads *
 *    (ceil(max_blocks / 16) + 1) * group * 528 bytes) returns
 *    KVARN_ERR_UNSUPPORTED and launches nothing; use kvarn_decode_attention.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls share the one array and it keeps the last call's contents;
 *    every partial a call reads was written earlier in that same call, so no
 *    clearing is needed.  Calls that overlap on the GPU (two streams, two
 *    host threads) race on the array and must be serialised by the caller.
 */
kvarn_status kvarn_decode_attention_noalloc(const kvarn_config* cfg, const void* q, const int32_t* block_table,
                                            int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                                            const void* block_pool, const void* tail_pool, float softmax_scale,
                                            float* out, int32_t* dev_err, void* stream);

/*
 * Dequantise packed blocks back to the unrotated domain (tests and tools).
 *  blocks  device int32[n]: block ids.
 *  out     device float32 [n][2 (K,V)][num_kv_heads][128 tokens][128].
 */
kvarn_status kvarn_dequantize(const kvarn_config* cfg, const void* block_pool, const int32_t* blocks,
                              int32_t n, float* out, int32_t* dev_err, void* stream);

/* Scratch bytes kvarn_token_errors needs: one record per (tile, head). */
size_t kvarn_token_errors_scratch_bytes(const kvarn_config* cfg, int32_t n_tiles, int32_t is_v);

/*
 * Per-token reconstruction errors (an analysis tool, not part of serving):
 * quantise each (tile, KV head) of x as the K (is_v = 0) or V (is_v = 1)
 * record of cfg's preset, dequantise it and compare with the input.  The
 * pages single out the per-token error distribution ("Huawei's KVarN puts
 * KV-cache quantization inside vLLM's backend", section "Why KV-cache
 * quantization degrades under autoregressive decoding": the largest 5% of
 * per-token errors cause most of the loss); rotate = 0 skips the Hadamard
 * rotation and sinkhorn_iters = 0 the variance normalisation, so the same
 * call measures each stage's effect.
 *  x, token_stride_elems, n_tokens, tile_first_token, n_tiles: as
 *              kvarn_quantize_tiles (one input tensor).
 *  scratch     device, >= kvarn_token_errors_scratch_bytes(cfg, n_tiles, is_v).
 *  out         device float32 [n_tiles][num_kv_heads][128 tokens][2]:
 *              (sum_c (xhat - x)^2, sum_c x^2) per token.
 * A tile whose first token is out of range stores KVARN_DEV_ERR_TOKEN_RANGE
 * and leaves its rows unwritten.
 */
kvarn_status kvarn_token_errors(const kvarn_config* cfg, const void* x, int64_t token_stride_elems, int64_t n_tokens,
                                const int64_t* tile_first_token, int32_t n_tiles, int32_t is_v, int32_t rotate,
                                int32_t sinkhorn_iters, void* scratch, size_t scratch_bytes, float* out,
                                int32_t* dev_err, void* stream);

/* Bytes of one block of the 16-bit comparison pool: num_kv_heads * 2 * 128 *
 * 128 * 2, layout [kv_head][K=0,V=1][token][channel]. */
size_t kvarn_fp16_block_bytes(const kvarn_config* cfg);

/*
 * Comparison point: the same decode attention over an unquantised 16-bit
 * paged cache (cfg->dtype elements, pool of num_blocks blocks laid out as in
 * kvarn_fp16_block_bytes).  seq_lens[s] tokens of sequence s live in
 * block_table[s][0 .. ceil(seq_lens[s]/128) - 1]; slots past the length in
 * the last block are ignored.  Arguments otherwise as kvarn_decode_attention.
 */
kvarn_status kvarn_fp16_decode_attention(const kvarn_config* cfg, const void* q,
                                         const int32_t* block_table, int32_t max_blocks,
                                         const int32_t* seq_lens, int32_t batch, const void* fp16_pool,
                                         float softmax_scale, float* out, void* workspace,
                                         size_t workspace_bytes, int32_t* dev_err, void* stream);

/*
 * Error-path test of kvarn_decode_attention (not for serving): the same call
 * with the copy of the first key record of one unit (sequence 0, KV head 0,
 * its first split-K chunk, first warp) left out and every wait on a record
 * copy limited to wait_polls polls of its mbarrier.  Nothing is in flight
 * for the left-out record, so its wait expires: the kernel stores
 * KVARN_DEV_ERR_TIMEOUT into *dev_err, waits (bounded) for the unit's copies
 * that did start, skips the rest of that warp's tiles and returns; the call
 * completes and the device stays usable.  The outputs of sequence 0 are
 * unspecified; the other sequences are decoded normally.  wait_polls >= 1
 * (KVARN_ERR_INVALID otherwise); other arguments as kvarn_decode_attention.
 * This is the timeout path every bounded wait of the library takes ("Kernels
 * never trap and never wait without a bound" above); the pages describe
 * nothing like it.
 */
kvarn_status kvarn_test_decode_wait_expiry(const kvarn_config* cfg, const void* q, const int32_t* block_table,
                                           int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                                           const void* block_pool, const void* tail_pool, float softmax_scale,
                                           float* out, void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                           int32_t wait_polls, void* stream);

/* Static description of a status code. */
const char* kvarn_status_string(kvarn_status s);

#ifdef __cplusplus
}
#endif

#endif /* KVARN_H */
