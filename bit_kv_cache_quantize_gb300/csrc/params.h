// params.h -- launch parameter blocks and launcher declarations shared by
// the C-ABI layer (kvarn_abi.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace kvarn {
// Bytes of one (tile, head) record of one role: a 512-byte header (per-channel
// and per-token FP8 scales, per-token FP16 zero-points) + 128 x 128 codes of
// `bits` bits; a head holds its key record then its value record.
__host__ __device__ constexpr int rec_bytes(int bits) { return 512 + 128 * 128 * bits / 8; }
__host__ __device__ constexpr int head_rec(int k_bits, int v_bits) { return rec_bytes(k_bits) + rec_bytes(v_bits); }

struct QuantizeParams {
  const void* k;
  const void* v;
  int64_t token_stride;
  int64_t n_tokens;
  const int64_t* tile_first_token;
  const int32_t* tile_dst_block;
  unsigned char* pool;
  int64_t block_bytes;
  int32_t num_kv_heads;
  int32_t num_blocks;
  int32_t iters;
  int32_t k_bits;  // key code width: 4 or 2
  int32_t v_bits;  // value code width: 2 or 4
  int32_t* err;
};
struct AppendParams {
  const void* k_new;
  const void* v_new;
  const int32_t* pos;
  const int32_t* block_table;
  int32_t max_blocks;
  int32_t num_kv_heads;
  int32_t num_blocks;
  int32_t iters;
  void* tail;
  unsigned char* pool;
  int64_t block_bytes;
  int32_t k_bits;
  int32_t v_bits;
  int32_t* err;
  int32_t batch;  // sequences (set by the launcher)
};
struct DecodeParams {
  const void* q;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const unsigned char* pool;
  const void* tail;
  float* ws;
  int32_t* err;
  int64_t block_bytes;
  float scale;
  int32_t max_blocks;
  int32_t num_kv_heads;
  int32_t num_q_heads;
  int32_t G;
  int32_t num_blocks;
  int32_t chunk_tiles;
  int32_t n_chunks;
  int32_t k_bits;
  int32_t v_bits;
  // Error-path test only (both 0 in every normal call): the bounded-wait
  // limit in polls (0 = the default) and a flag that leaves out the first
  // key-record copy of warp 0 of the unit (chunk 0, KV head 0, sequence 0),
  // so that its wait expires with nothing in flight.
  int32_t wait_polls;
  int32_t skip_first_copy;
  int64_t ws_bytes;  // bytes of ws (the bounds checks of the checked build)
};
// Multi-query causal attention: n_queries query tokens per sequence at the
// last n_queries positions, grouped with their GQA heads into row blocks of
// 128 (query, head-in-group) rows per KV head.
struct MQParams {
  const void* q;  // [batch][n_queries][num_q_heads][128]
  const int32_t* block_table;
  const int32_t* seq_lens;
  const unsigned char* pool;
  const void* tail;
  float* ws;
  int32_t* err;
  int64_t block_bytes;
  float scale;
  int32_t max_blocks;
  int32_t num_kv_heads;
  int32_t num_q_heads;
  int32_t G;
  int32_t num_blocks;
  int32_t n_queries;
  int32_t n_rowblocks;
  int32_t chunk_tiles;
  int32_t n_chunks;
  int32_t k_bits;
  int32_t v_bits;
  int64_t ws_bytes;  // bytes of ws (the bounds checks of the checked build)
};

// Per-token reconstruction errors of quantised tiles (the error study):
// quantise (rotation and normalisation optional), dequantise, compare.
struct ErrParams {
  const void* x;
  int64_t token_stride;
  int64_t n_tokens;
  const int64_t* tile_first_token;
  unsigned char* scratch;  // one record per (tile, head)
  float* out;              // [n_tiles][num_kv_heads][128] x (err2, norm2)
  int32_t num_kv_heads;
  int32_t iters;
  int32_t k_bits;
  int32_t v_bits;
  int32_t is_v;
  int32_t rotate;
  int32_t* err;
};
cudaError_t launch_token_errors(const ErrParams& p, int dtype, int n_tiles, cudaStream_t s);

cudaError_t launch_quantize(const QuantizeParams& p, int dtype, int n_tiles, cudaStream_t s);
cudaError_t launch_append(const AppendParams& p, int dtype, int batch, cudaStream_t s);
cudaError_t launch_dequantize(const unsigned char* pool, int64_t block_bytes, const int32_t* blocks, int n,
                              int num_blocks, int num_kv_heads, int k_bits, int v_bits, float* out, int32_t* err,
                              cudaStream_t s);
cudaError_t launch_decode(const DecodeParams& p, int dtype, int batch, float* out, cudaStream_t s);
cudaError_t launch_decode_noalloc(DecodeParams p, int dtype, int batch, float* out, cudaStream_t s);
cudaError_t launch_decode_f16(const DecodeParams& p, const void* pool16, int dtype, int batch, float* out,
                              cudaStream_t s);
cudaError_t launch_multiquery(const MQParams& p, int dtype, int batch, float* out, cudaStream_t s);
size_t multiquery_ws_bytes(int batch, int num_kv_heads, int n_rowblocks, int max_blocks, int chunk_tiles);
size_t decode_ws_bytes(int batch, int num_kv_heads, int G, int max_blocks, int chunk_tiles);

}  // namespace kvarn
