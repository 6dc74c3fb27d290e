// kvarn_abi.cu -- the extern "C" entry points declared in include/kvarn.h:
// host-side validation, launch configuration and status codes.  No
// allocation, no global state, no exceptions across the boundary.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/kvarn.h"

#include "params.h"

namespace kvarn {
constexpr int kChunkTiles = 16;  // packed tiles per split-K CTA of an ordinary call (sizes the workspace)
constexpr int kSmallChunkTiles = 8;  // of a small call: two tiles per warp of its 4-warp CTAs
// A call whose table spans fewer (sequence, KV head, tile) units than this
// is small: 16-tile chunks would give it under three waves of two 8-warp
// CTAs per SM on 152 SMs (3 x 304 x 16), so it takes 8-tile chunks, twice
// the CTAs.  The rule depends only on the call's shape, so the workspace
// size does too.
constexpr long long kSmallCallUnits = 3LL * 304 * 16;

static bool small_call(int batch, int num_kv_heads, int max_blocks) {
  return (long long)batch * num_kv_heads * max_blocks < kSmallCallUnits;
}

// Fewest packed tiles per split-K CTA a call of this shape may use.
static int min_chunk_tiles(int batch, int num_kv_heads, int max_blocks) {
  return small_call(batch, num_kv_heads, max_blocks) ? kSmallChunkTiles : kChunkTiles;
}

// Packed tiles per split-K CTA for one call: 8 for a small call; else the
// longest of 64 and 32 (longer CTAs amortise the per-CTA query set-up and
// merge) that still gives at least three waves of CTAs at two per SM, else 16.
// The K4/V4 preset, whose CTAs have 4 warps, stops at 32 (8 tiles a warp).
static int choose_chunk_tiles(const kvarn_config* cfg, int batch, int num_kv_heads, int max_blocks) {
  if (small_call(batch, num_kv_heads, max_blocks)) return kSmallChunkTiles;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return kChunkTiles;
  const long long units = (long long)batch * num_kv_heads;
  for (int chunk : {64, 32})
    if ((chunk == 32 || cfg->v_bits != 4) && units * ((max_blocks + chunk - 1) / chunk) >= 6LL * sms) return chunk;
  return kChunkTiles;
}
constexpr int kF16ChunkTiles = 16;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by every entry point.
static kvarn_status check_config(const kvarn_config* c) {
  if (!c) return KVARN_ERR_INVALID;
  if (c->num_kv_heads < 1 || c->num_q_heads < 1 || c->num_blocks < 0 || c->sinkhorn_iters < 0 ||
      c->sinkhorn_iters > 64 || c->head_dim < 1 || c->tile_tokens < 1)
    return KVARN_ERR_INVALID;
  if (c->num_q_heads % c->num_kv_heads) return KVARN_ERR_INVALID;
  if (c->dtype != KVARN_DTYPE_F16 && c->dtype != KVARN_DTYPE_BF16) return KVARN_ERR_INVALID;
  // presets: kvarn_k4v2 (4-bit keys, 2-bit values), K2/V2 and K4/V4
  const bool preset = (c->k_bits == 4 && c->v_bits == 2) || (c->k_bits == 2 && c->v_bits == 2) ||
                      (c->k_bits == 4 && c->v_bits == 4);
  if (c->head_dim != 128 || c->tile_tokens != 128 || !preset) return KVARN_ERR_UNSUPPORTED;
  if (c->num_q_heads / c->num_kv_heads > 8) return KVARN_ERR_UNSUPPORTED;
  return KVARN_OK;
}

static kvarn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVARN_OK : KVARN_ERR_CUDA; }
}  // namespace kvarn

using namespace kvarn;

extern "C" {

size_t kvarn_block_bytes(const kvarn_config* cfg) {
  if (check_config(cfg) != KVARN_OK) return 0;
  return static_cast<size_t>(cfg->num_kv_heads) * head_rec(cfg->k_bits, cfg->v_bits);
}

size_t kvarn_tail_bytes(const kvarn_config* cfg, int32_t batch) {
  if (check_config(cfg) != KVARN_OK || batch < 0) return 0;
  return static_cast<size_t>(batch) * cfg->num_kv_heads * 2 * 128 * 128 * 2;
}

size_t kvarn_fp16_block_bytes(const kvarn_config* cfg) {
  if (check_config(cfg) != KVARN_OK) return 0;
  return static_cast<size_t>(cfg->num_kv_heads) * 2 * 128 * 128 * 2;
}

size_t kvarn_decode_workspace_bytes(const kvarn_config* cfg, int32_t batch, int32_t max_blocks) {
  if (check_config(cfg) != KVARN_OK || batch < 0 || max_blocks < 1) return 0;
  const int G = cfg->num_q_heads / cfg->num_kv_heads;
  const size_t a = decode_ws_bytes(batch, cfg->num_kv_heads, G, max_blocks,
                                   min_chunk_tiles(batch, cfg->num_kv_heads, max_blocks));
  const size_t b = decode_ws_bytes(batch, cfg->num_kv_heads, G, max_blocks, kF16ChunkTiles);
  return a > b ? a : b;
}

kvarn_status kvarn_quantize_tiles(const kvarn_config* cfg, const void* k, const void* v, int64_t token_stride_elems,
                                  int64_t n_tokens, const int64_t* tile_first_token, const int32_t* tile_dst_block,
                                  int32_t n_tiles, void* block_pool, int32_t* dev_err, void* stream) {
  kvarn_status st = check_config(cfg);
  if (st != KVARN_OK) return st;
  if (n_tiles < 0 || n_tokens < 0) return KVARN_ERR_INVALID;
  if (n_tiles == 0) return KVARN_OK;
  if (!k || !v || !tile_first_token || !tile_dst_block || (!block_pool && cfg->num_blocks > 0)) return KVARN_ERR_INVALID;
  if (!aligned16(k) || !aligned16(v) || !aligned16(block_pool)) return KVARN_ERR_INVALID;
  if (token_stride_elems % 8 || token_stride_elems < static_cast<int64_t>(cfg->num_kv_heads) * 128)
    return KVARN_ERR_INVALID;
  if (static_cast<int64_t>(n_tiles) * cfg->num_kv_heads * 2 > 0x7fffffffLL) return KVARN_ERR_INVALID;
  QuantizeParams p{k, v, token_stride_elems, n_tokens, tile_first_token, tile_dst_block,
                   static_cast<unsigned char*>(block_pool), static_cast<int64_t>(kvarn_block_bytes(cfg)),
                   cfg->num_kv_heads, cfg->num_blocks, cfg->sinkhorn_iters, cfg->k_bits, cfg->v_bits, dev_err};
  return cuda_status(launch_quantize(p, cfg->dtype, n_tiles, static_cast<cudaStream_t>(stream)));
}

size_t kvarn_token_errors_scratch_bytes(const kvarn_config* cfg, int32_t n_tiles, int32_t is_v) {
  if (check_config(cfg) != KVARN_OK || n_tiles < 0) return 0;
  return static_cast<size_t>(n_tiles) * cfg->num_kv_heads *
         static_cast<size_t>(is_v ? rec_bytes(cfg->v_bits) : rec_bytes(cfg->k_bits));
}

kvarn_status kvarn_token_errors(const kvarn_config* cfg, const void* x, int64_t token_stride_elems, int64_t n_tokens,
                                const int64_t* tile_first_token, int32_t n_tiles, int32_t is_v, int32_t rotate,
                                int32_t sinkhorn_iters, void* scratch, size_t scratch_bytes, float* out,
                                int32_t* dev_err, void* stream) {
  kvarn_status st = check_config(cfg);
  if (st != KVARN_OK) return st;
  if (n_tiles < 0 || n_tokens < 0 || (is_v != 0 && is_v != 1) || (rotate != 0 && rotate != 1) ||
      sinkhorn_iters < 0 || sinkhorn_iters > 64)
    return KVARN_ERR_INVALID;
  if (n_tiles == 0) return KVARN_OK;
  if (!x || !tile_first_token || !scratch || !out) return KVARN_ERR_INVALID;
  if (!aligned16(x) || !aligned16(scratch) || !aligned16(out)) return KVARN_ERR_INVALID;
  if (token_stride_elems % 8 || token_stride_elems < static_cast<int64_t>(cfg->num_kv_heads) * 128)
    return KVARN_ERR_INVALID;
  if (static_cast<int64_t>(n_tiles) * cfg->num_kv_heads > 0x7fffffffLL) return KVARN_ERR_INVALID;
  if (scratch_bytes < kvarn_token_errors_scratch_bytes(cfg, n_tiles, is_v)) return KVARN_ERR_INVALID;
  ErrParams p{x, token_stride_elems, n_tokens, tile_first_token, static_cast<unsigned char*>(scratch), out,
              cfg->num_kv_heads, sinkhorn_iters, cfg->k_bits, cfg->v_bits, is_v, rotate, dev_err};
  return cuda_status(launch_token_errors(p, cfg->dtype, n_tiles, static_cast<cudaStream_t>(stream)));
}

kvarn_status kvarn_append_tokens(const kvarn_config* cfg, const void* k_new, const void* v_new, const int32_t* pos,
                                 const int32_t* block_table, int32_t max_blocks, int32_t batch, void* tail_pool,
                                 void* block_pool, int32_t* dev_err, void* stream) {
  kvarn_status st = check_config(cfg);
  if (st != KVARN_OK) return st;
  if (batch < 0 || max_blocks < 1) return KVARN_ERR_INVALID;
  if (batch == 0) return KVARN_OK;
  if (static_cast<int64_t>(batch) * cfg->num_kv_heads * 2 > 0x7fffffffLL) return KVARN_ERR_INVALID;
  if (!k_new || !v_new || !pos || !block_table || !tail_pool || (!block_pool && cfg->num_blocks > 0)) return KVARN_ERR_INVALID;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(tail_pool) || !aligned16(block_pool))
    return KVARN_ERR_INVALID;
  AppendParams p{k_new, v_new, pos, block_table, max_blocks, cfg->num_kv_heads, cfg->num_blocks, cfg->sinkhorn_iters,
                 tail_pool, static_cast<unsigned char*>(block_pool), static_cast<int64_t>(kvarn_block_bytes(cfg)),
                 cfg->k_bits, cfg->v_bits, dev_err};
  return cuda_status(launch_append(p, cfg->dtype, batch, static_cast<cudaStream_t>(stream)));
}

static kvarn_status check_decode(const kvarn_config* cfg, const void* q, const int32_t* block_table,
                                 int32_t max_blocks, const int32_t* seq_lens, int32_t batch, const void* pool,
                                 float* out, void* workspace, size_t workspace_bytes) {
  kvarn_status st = check_config(cfg);
  if (st != KVARN_OK) return st;
  if (batch < 0 || max_blocks < 1 || batch > 65535) return KVARN_ERR_INVALID;
  if (batch == 0) return KVARN_OK;
  if (!q || !block_table || !seq_lens || (!pool && cfg->num_blocks > 0) || !out || !workspace) return KVARN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(pool) || !aligned16(out) || !aligned16(workspace)) return KVARN_ERR_INVALID;
  if (workspace_bytes < kvarn_decode_workspace_bytes(cfg, batch, max_blocks)) return KVARN_ERR_INVALID;
  return KVARN_OK;
}

static kvarn_status decode_call(const kvarn_config* cfg, const void* q, const int32_t* block_table,
                                int32_t max_blocks, const int32_t* seq_lens, int32_t batch, const void* block_pool,
                                const void* tail_pool, float softmax_scale, float* out, void* workspace,
                                size_t workspace_bytes, int32_t* dev_err, void* stream, int32_t wait_polls,
                                int32_t skip_first_copy) {
  kvarn_status st = check_decode(cfg, q, block_table, max_blocks, seq_lens, batch, block_pool, out, workspace,
                                 workspace_bytes);
  if (st != KVARN_OK || batch == 0) return st;
  if (!tail_pool || !aligned16(tail_pool)) return KVARN_ERR_INVALID;
  const int chunk = choose_chunk_tiles(cfg, batch, cfg->num_kv_heads, max_blocks);
  const int n_chunks = (max_blocks + chunk - 1) / chunk;
  DecodeParams p{q, block_table, seq_lens, static_cast<const unsigned char*>(block_pool), tail_pool,
                 static_cast<float*>(workspace), dev_err, static_cast<int64_t>(kvarn_block_bytes(cfg)), softmax_scale,
                 max_blocks, cfg->num_kv_heads, cfg->num_q_heads, cfg->num_q_heads / cfg->num_kv_heads,
                 cfg->num_blocks, chunk, n_chunks, cfg->k_bits, cfg->v_bits, wait_polls, skip_first_copy,
                 static_cast<int64_t>(workspace_bytes)};
  return cuda_status(launch_decode(p, cfg->dtype, batch, out, static_cast<cudaStream_t>(stream)));
}

kvarn_status kvarn_decode_attention(const kvarn_config* cfg, const void* q, const int32_t* block_table,
                                    int32_t max_blocks, const int32_t* seq_lens, int32_t batch, const void* block_pool,
                                    const void* tail_pool, float softmax_scale, float* out, void* workspace,
                                    size_t workspace_bytes, int32_t* dev_err, void* stream) {
  return decode_call(cfg, q, block_table, max_blocks, seq_lens, batch, block_pool, tail_pool, softmax_scale, out,
                     workspace, workspace_bytes, dev_err, stream, 0, 0);
}

kvarn_status kvarn_test_decode_wait_expiry(const kvarn_config* cfg, const void* q, const int32_t* block_table,
                                           int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                                           const void* block_pool, const void* tail_pool, float softmax_scale,
                                           float* out, void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                           int32_t wait_polls, void* stream) {
  if (wait_polls < 1) return KVARN_ERR_INVALID;
  return decode_call(cfg, q, block_table, max_blocks, seq_lens, batch, block_pool, tail_pool, softmax_scale, out,
                     workspace, workspace_bytes, dev_err, stream, wait_polls, 1);
}

// Packed tiles per split-K CTA of the multi-query kernel (one CTA per SM):
// 32 while that leaves at least three waves, else 16 (sizes the workspace).
static int choose_mq_chunk(int units, int max_blocks) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return kChunkTiles;
  const long long ctas = (long long)units * ((max_blocks + 31) / 32);
  return ctas >= 3LL * sms ? 32 : kChunkTiles;
}

static int mq_rowblocks(const kvarn_config* cfg, int n_queries) {
  const int G = cfg->num_q_heads / cfg->num_kv_heads;
  return (n_queries * G + 127) / 128;
}

size_t kvarn_multiquery_workspace_bytes(const kvarn_config* cfg, int32_t batch, int32_t max_blocks,
                                        int32_t n_queries) {
  if (check_config(cfg) != KVARN_OK || batch < 0 || max_blocks < 1 || n_queries < 1 || n_queries > 4096) return 0;
  return multiquery_ws_bytes(batch, cfg->num_kv_heads, mq_rowblocks(cfg, n_queries), max_blocks, kChunkTiles);
}

kvarn_status kvarn_multiquery_attention(const kvarn_config* cfg, const void* q, int32_t n_queries,
                                        const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                                        int32_t batch, const void* block_pool, const void* tail_pool,
                                        float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                                        int32_t* dev_err, void* stream) {
  kvarn_status st = check_config(cfg);
  if (st != KVARN_OK) return st;
  if (batch < 0 || max_blocks < 1 || batch > 65535 || n_queries < 1 || n_queries > 4096) return KVARN_ERR_INVALID;
  if (batch == 0) return KVARN_OK;
  if (!q || !block_table || !seq_lens || (!block_pool && cfg->num_blocks > 0) || !tail_pool || !out || !workspace)
    return KVARN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(block_pool) || !aligned16(tail_pool) || !aligned16(out) || !aligned16(workspace))
    return KVARN_ERR_INVALID;
  if (workspace_bytes < kvarn_multiquery_workspace_bytes(cfg, batch, max_blocks, n_queries)) return KVARN_ERR_INVALID;
  const int n_rb = mq_rowblocks(cfg, n_queries);
  if ((long long)cfg->num_kv_heads * n_rb > 65535) return KVARN_ERR_UNSUPPORTED;
  const int chunk = choose_mq_chunk(batch * cfg->num_kv_heads * n_rb, max_blocks);
  const int n_chunks = (max_blocks + chunk - 1) / chunk;
  MQParams p{q, block_table, seq_lens, static_cast<const unsigned char*>(block_pool), tail_pool,
             static_cast<float*>(workspace), dev_err, static_cast<int64_t>(kvarn_block_bytes(cfg)), softmax_scale,
             max_blocks, cfg->num_kv_heads, cfg->num_q_heads, cfg->num_q_heads / cfg->num_kv_heads, cfg->num_blocks,
             n_queries, n_rb, chunk, n_chunks, cfg->k_bits, cfg->v_bits, static_cast<int64_t>(workspace_bytes)};
  return cuda_status(launch_multiquery(p, cfg->dtype, batch, out, static_cast<cudaStream_t>(stream)));
}

kvarn_status kvarn_decode_attention_noalloc(const kvarn_config* cfg, const void* q, const int32_t* block_table,
                                            int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                                            const void* block_pool, const void* tail_pool, float softmax_scale,
                                            float* out, int32_t* dev_err, void* stream) {
  kvarn_status st = check_config(cfg);
  if (st != KVARN_OK) return st;
  if (batch < 0 || max_blocks < 1 || batch > 65535) return KVARN_ERR_INVALID;
  if (batch == 0) return KVARN_OK;
  if (!q || !block_table || !seq_lens || (!block_pool && cfg->num_blocks > 0) || !tail_pool || !out) return KVARN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(block_pool) || !aligned16(tail_pool) || !aligned16(out)) return KVARN_ERR_INVALID;
  const int G = cfg->num_q_heads / cfg->num_kv_heads;
  if (decode_ws_bytes(batch, cfg->num_kv_heads, G, max_blocks, kChunkTiles) > KVARN_NOALLOC_SCRATCH_BYTES)
    return KVARN_ERR_UNSUPPORTED;  // larger than the fixed scratch: use kvarn_decode_attention
  int chunk = choose_chunk_tiles(cfg, batch, cfg->num_kv_heads, max_blocks);
  if (decode_ws_bytes(batch, cfg->num_kv_heads, G, max_blocks, chunk) > KVARN_NOALLOC_SCRATCH_BYTES)
    chunk = kChunkTiles;  // a small call's finer split does not fit: the ordinary split does
  const int n_chunks = (max_blocks + chunk - 1) / chunk;
  DecodeParams p{q, block_table, seq_lens, static_cast<const unsigned char*>(block_pool), tail_pool, nullptr, dev_err,
                 static_cast<int64_t>(kvarn_block_bytes(cfg)), softmax_scale, max_blocks, cfg->num_kv_heads,
                 cfg->num_q_heads, G, cfg->num_blocks, chunk, n_chunks, cfg->k_bits, cfg->v_bits};
  return cuda_status(launch_decode_noalloc(p, cfg->dtype, batch, out, static_cast<cudaStream_t>(stream)));
}

kvarn_status kvarn_fp16_decode_attention(const kvarn_config* cfg, const void* q, const int32_t* block_table,
                                         int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                                         const void* fp16_pool, float softmax_scale, float* out, void* workspace,
                                         size_t workspace_bytes, int32_t* dev_err, void* stream) {
  kvarn_status st = check_decode(cfg, q, block_table, max_blocks, seq_lens, batch, fp16_pool, out, workspace,
                                 workspace_bytes);
  if (st != KVARN_OK || batch == 0) return st;
  if (cfg->num_blocks < 1) return KVARN_ERR_INVALID;
  const int n_chunks = (max_blocks + kF16ChunkTiles - 1) / kF16ChunkTiles;
  DecodeParams p{q, block_table, seq_lens, nullptr, nullptr, static_cast<float*>(workspace), dev_err, 0,
                 softmax_scale, max_blocks, cfg->num_kv_heads, cfg->num_q_heads,
                 cfg->num_q_heads / cfg->num_kv_heads, cfg->num_blocks, kF16ChunkTiles, n_chunks, 16, 16, 0, 0,
                 static_cast<int64_t>(workspace_bytes)};
  cudaError_t e = launch_decode_f16(p, fp16_pool, cfg->dtype, batch, out, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidValue) return KVARN_ERR_INVALID;
  if (e == cudaErrorNotSupported) return KVARN_ERR_UNSUPPORTED;
  return cuda_status(e);
}

kvarn_status kvarn_dequantize(const kvarn_config* cfg, const void* block_pool, const int32_t* blocks, int32_t n,
                              float* out, int32_t* dev_err, void* stream) {
  kvarn_status st = check_config(cfg);
  if (st != KVARN_OK) return st;
  if (n < 0) return KVARN_ERR_INVALID;
  if (n == 0) return KVARN_OK;
  if ((!block_pool && cfg->num_blocks > 0) || !blocks || !out || !aligned16(block_pool) || !aligned16(out))
    return KVARN_ERR_INVALID;
  if (cfg->num_kv_heads > 65535) return KVARN_ERR_INVALID;
  return cuda_status(launch_dequantize(static_cast<const unsigned char*>(block_pool),
                                       static_cast<int64_t>(kvarn_block_bytes(cfg)), blocks, n, cfg->num_blocks,
                                       cfg->num_kv_heads, cfg->k_bits, cfg->v_bits, out, dev_err,
                                       static_cast<cudaStream_t>(stream)));
}

const char* kvarn_status_string(kvarn_status s) {
  switch (s) {
    case KVARN_OK: return "ok";
    case KVARN_ERR_INVALID: return "invalid argument";
    case KVARN_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVARN_ERR_CUDA: return "CUDA launch or runtime error";
  }
  return "unknown status";
}

}  // extern "C"
