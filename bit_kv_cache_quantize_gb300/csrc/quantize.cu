// quantize.cu -- write path of the KVarN cache: one CTA quantises one
// 128-token x 128-channel tile of one KV head into a packed record.
//
// Steps (page "KVarN: 2-Bit KV-Cache That Beats FP16 Throughput, and Where
// the Catch Lives", section "What KVarN does differently"; page "Huawei's
// KVarN puts KV-cache quantization inside vLLM's backend", sections "What
// KVarN changes in vLLM's serving path" and "The four-stage pipeline"):
//   1. Hadamard rotation along channels, R = X H: a 128x128x128 product on
//      the tensor cores (A = the 16-bit tile, exact; B = the +-1 Sylvester
//      signs generated in registers; fp32 accumulate), scaled by 1/sqrt(128).
//   2. Sinkhorn-like normalisation in log space: N iterations of a column
//      step (log std over tokens of every channel) then a row step (log std
//      over channels of every token).  Column steps read a channel-major
//      register copy of R, row steps a token-major copy, so both reductions
//      finish inside a quad of lanes.  Each std is a shifted one-pass sum
//      (shift = the first element), exact for a constant row or column.
//   3. Column factors centred (geometric mean 1) -> FP8 E4M3 scale g.
//   4. Per token: Y = R / g, FP16 zero-point b = round-down(min Y), FP8 step
//      a = round-up((max Y - b) / L).
//   5. Codes rne((Y - b) * (1/a)), clamped to [0, L]; packed and stored with
//      16-byte stores.
#include "common.cuh"
#include "params.h"

namespace kvarn {

// Shared memory of one quantiser CTA (dynamic, ~78 KB).
struct QSmem {
  alignas(128) unsigned char big[65536];   // X staging (128 x 272 B), then R fp32 (swizzled)
  alignas(16) unsigned char rec[512 + 128 * 68];  // header | codes (K rows padded to 68 B)
  float alpha[4 * 36];                     // row factors exp(-u), padded per 32 tokens
  float beta[128];                         // column factors exp(-v)
  float inv_g[128];
  float inv_a[128];
  float bval[128];
  float red[8];
};

constexpr int X_ROW = 272;                 // staging row stride: 256 B + 16 B pad

__device__ __forceinline__ int alpha_idx(int t) { return (t >> 5) * 36 + (t & 31); }

// Byte offset of the float2 holding R[t][2*c2 .. 2*c2+1] (XOR swizzle keeps
// both the token-major writes and the channel-major reads conflict-free).
__device__ __forceinline__ int r_off(int t, int c2) {
  return t * 512 + ((c2 ^ (((t ^ (t >> 5)) & 3) << 2)) << 3);
}

// New log factor from shifted sums over n = 128 values: s1 = sum(w - K),
// s2 = sum((w - K)^2).  Keeps `old` when the std is at most 1e-6 of the rms
// (constant or all-zero row/column).
__device__ __forceinline__ float log_std_or_keep(float s1, float s2, float K, float old) {
  const float inv_n = 1.0f / 128.0f;
  float md = s1 * inv_n;
  float var = fmaxf(s2 * inv_n - md * md, 0.0f);
  float mw = K + md;
  float ms = var + mw * mw;
  return (var > 1e-12f * ms) ? logf(sqrtf(var)) : old;
}

// Quantise one tile.  src: token rows of 128 16-bit channels, consecutive
// rows row_stride elements apart (16-byte aligned).  dst: the record in the
// pool.  All 256 threads of the CTA must call this.
template <typename E, bool IS_V>
__device__ void quantize_tile_cta(const E* __restrict__ src, int64_t row_stride, unsigned char* __restrict__ dst,
                                  int iters, QSmem& sm) {
  constexpr int L = IS_V ? 3 : 15;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, j = lane & 3;  // copy 1: token g (+8) of the warp's 16, channel pair j of each 8
  const int p = g, q = j;                 // copy 2: channel pair p of the warp's 16, tokens 32q..32q+31

  // ---- 1. stage X (16-bit) into shared memory
  for (int i = tid; i < T * 16; i += 256) {
    int row = i >> 4, ch16 = i & 15;
    cp_async16(sm.big + row * X_ROW + ch16 * 16, src + row * row_stride + ch16 * 8);
  }
  for (int i = tid; i < T; i += 256) sm.alpha[alpha_idx(i)] = 1.0f;
  cp_async_wait_all();
  __syncthreads();

  uint32_t afr[8][4];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    ldmatrix_x4(afr[ks], sm.big + (16 * warp + (lane & 15)) * X_ROW + (16 * ks + (lane >> 4) * 8) * 2);
  __syncthreads();  // the staging area is reused for R below

  // ---- 2. R = X H on the tensor cores; H[k][n] = (-1)^popcount(k & n)
  // For k = 16ks + kk, n = 8nb + g:  popcount(k & n) = popcount(kk & g)
  // + (kk >> 3) * (nb & 1) + popcount(ks & (nb >> 1)), so every B fragment is
  // +-F with F the lane's base sign pair.
  const uint32_t one = Bits16<E>::one;
  const uint32_t F = ((__popc((2 * j) & g) & 1) ? (one | 0x8000u) : one) |
                     (((__popc((2 * j + 1) & g) & 1) ? (one | 0x8000u) : one) << 16);
  const uint32_t NF = F ^ 0x80008000u;
  float r1[16][4];  // copy 1: R[16w+g][8nb+2j+{0,1}] and R[16w+g+8][...]
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int P = __builtin_popcount(ks & (nb >> 1)) & 1;
      const uint32_t b0 = P ? NF : F;
      const uint32_t b1 = (P ^ (nb & 1)) ? NF : F;
      mma16816<E>(c, afr[ks], b0, b1);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) r1[nb][e] = c[e] * INV_SQRT_D;
  }

  // ---- transpose through shared memory into copy 2 (channel-major)
  const int t0 = 16 * warp + g, t1 = t0 + 8;
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) {
    *reinterpret_cast<float2*>(sm.big + r_off(t0, 4 * nb + j)) = make_float2(r1[nb][0], r1[nb][1]);
    *reinterpret_cast<float2*>(sm.big + r_off(t1, 4 * nb + j)) = make_float2(r1[nb][2], r1[nb][3]);
  }
  __syncthreads();
  const int c0 = 16 * warp + 2 * p;  // copy-2 channels c0, c0 + 1
  float2 r2[32];                     // R[32q + i][c0 .. c0+1]
#pragma unroll
  for (int i = 0; i < 32; ++i) r2[i] = *reinterpret_cast<const float2*>(sm.big + r_off(32 * q + i, 8 * warp + p));

  // ---- 3. Sinkhorn-like iterations
  float v0 = 0.f, v1 = 0.f;  // log column factors of c0, c0+1 (replicated over q)
  float u0 = 0.f, u1 = 0.f;  // log row factors of t0, t1 (replicated over j)
  for (int it = 0; it < iters; ++it) {
    // column step on copy 2: std over tokens of w = alpha_t * R[t][c], as
    // shifted sums of d = alpha_t * R - K (K = token 0's value), two channels
    // per packed f32x2 op
    {
      const float* al = sm.alpha + q * 36;
      const float2 w0 = make_float2(al[0] * r2[0].x, al[0] * r2[0].y);
      const float Ka = __shfl_sync(0xffffffffu, w0.x, lane & ~3);
      const float Kb = __shfl_sync(0xffffffffu, w0.y, lane & ~3);
      const float2 nK = make_float2(-Ka, -Kb);
      float2 s1e = make_float2(0.f, 0.f), s2e = s1e, s1o = s1e, s2o = s1e;
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 de = ffma2(make_float2(al[i], al[i]), r2[i], nK);
        const float2 dd = ffma2(make_float2(al[i + 1], al[i + 1]), r2[i + 1], nK);
        s1e = fadd2(s1e, de); s2e = ffma2(de, de, s2e);
        s1o = fadd2(s1o, dd); s2o = ffma2(dd, dd, s2o);
      }
      s1e = fadd2(s1e, s1o); s2e = fadd2(s2e, s2o);
      const float s1a = quad_sum(s1e.x), s2a = quad_sum(s2e.x), s1b = quad_sum(s1e.y), s2b = quad_sum(s2e.y);
      v0 = log_std_or_keep(s1a, s2a, Ka, v0);
      v1 = log_std_or_keep(s1b, s2b, Kb, v1);
      if (q == 0) { sm.beta[c0] = expf(-v0); sm.beta[c0 + 1] = expf(-v1); }
    }
    __syncthreads();
    // row step on copy 1: std over channels of w = beta_c * R[t][c]; packed
    // over the channel pair, the two lanes of a pair accumulate separately
    {
      const float2 be0 = *reinterpret_cast<const float2*>(sm.beta + 2 * j);
      const float Ka = __shfl_sync(0xffffffffu, be0.x * r1[0][0], lane & ~3);  // channel 0 of token t0
      const float Kb = __shfl_sync(0xffffffffu, be0.x * r1[0][2], lane & ~3);  // channel 0 of token t1
      const float2 nKa = make_float2(-Ka, -Ka), nKb = make_float2(-Kb, -Kb);
      float2 s1a = make_float2(0.f, 0.f), s2a = s1a, s1b = s1a, s2b = s1a;
#pragma unroll
      for (int nb = 0; nb < 16; ++nb) {
        const float2 be = *reinterpret_cast<const float2*>(sm.beta + 8 * nb + 2 * j);
        const float2 da = ffma2(be, make_float2(r1[nb][0], r1[nb][1]), nKa);
        const float2 db = ffma2(be, make_float2(r1[nb][2], r1[nb][3]), nKb);
        s1a = fadd2(s1a, da); s2a = ffma2(da, da, s2a);
        s1b = fadd2(s1b, db); s2b = ffma2(db, db, s2b);
      }
      const float S1a = quad_sum(s1a.x + s1a.y), S2a = quad_sum(s2a.x + s2a.y);
      const float S1b = quad_sum(s1b.x + s1b.y), S2b = quad_sum(s2b.x + s2b.y);
      u0 = log_std_or_keep(S1a, S2a, Ka, u0);
      u1 = log_std_or_keep(S1b, S2b, Kb, u1);
      if (j == 0) { sm.alpha[alpha_idx(t0)] = expf(-u0); sm.alpha[alpha_idx(t1)] = expf(-u1); }
    }
    __syncthreads();
  }

  // ---- 4. gauge and per-channel FP8 scales
  {
    float s = (q == 0) ? (v0 + v1) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) sm.red[warp] = s;
  }
  __syncthreads();
  {
    float mean = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) mean += sm.red[w];
    mean *= (1.0f / 128.0f);
    if (q == 0) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = e ? v1 : v0;
        uint8_t gc = float_to_e4m3_rn(expf(v - mean));
        if (gc == 0) gc = 0x01;
        sm.rec[c0 + e] = gc;
        sm.inv_g[c0 + e] = __frcp_rn(e4m3_to_float(gc));
      }
    }
  }
  __syncthreads();

  // ---- 5. per-token zero-point and step (copy 1)
  float ig[16][2];
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) {
    const float2 v = *reinterpret_cast<const float2*>(sm.inv_g + 8 * nb + 2 * j);
    ig[nb][0] = v.x; ig[nb][1] = v.y;
  }
  float ba, bb, ia, ib;  // zero-point and 1/step of t0, t1
  {
    float mn0 = INFINITY, mx0 = -INFINITY, mn1 = INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 16; ++nb) {
      const float y0 = __fmul_rn(r1[nb][0], ig[nb][0]), y1 = __fmul_rn(r1[nb][1], ig[nb][1]);
      const float y2 = __fmul_rn(r1[nb][2], ig[nb][0]), y3 = __fmul_rn(r1[nb][3], ig[nb][1]);
      mn0 = fminf(mn0, fminf(y0, y1)); mx0 = fmaxf(mx0, fmaxf(y0, y1));
      mn1 = fminf(mn1, fminf(y2, y3)); mx1 = fmaxf(mx1, fmaxf(y2, y3));
    }
    mn0 = quad_min(mn0); mx0 = quad_max(mx0); mn1 = quad_min(mn1); mx1 = quad_max(mx1);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float mn = e ? mn1 : mn0, mx = e ? mx1 : mx0;
      __half bh = (mn <= -65504.f) ? __float2half_rn(-65504.f) : __float2half_rd(mn);
      const float bv = __half2float(bh);
      const float step = __fdiv_ru(__fsub_ru(mx, bv), (float)L);
      uint8_t ac = float_to_e4m3_ru(step);
      if (ac == 0) ac = 0x01;
      const float inv_a = __frcp_rn(e4m3_to_float(ac));
      if (e) { bb = bv; ib = inv_a; } else { ba = bv; ia = inv_a; }
      if (j == 0) {
        const int t = e ? t1 : t0;
        sm.rec[128 + t] = ac;
        *reinterpret_cast<__half*>(sm.rec + 256 + 2 * t) = bh;
        sm.inv_a[t] = inv_a;
        sm.bval[t] = bv;
      }
    }
  }

  // ---- 6. codes and packing
  if constexpr (!IS_V) {
    // token-major nibbles: byte 4nb+j of token t holds channels 8nb+2j, +1
#pragma unroll
    for (int nb = 0; nb < 16; ++nb) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float bv = e ? bb : ba, inv_a = e ? ib : ia;
        int k0 = __float2int_rn(__fmul_rn(__fsub_rn(__fmul_rn(r1[nb][2 * e], ig[nb][0]), bv), inv_a));
        int k1 = __float2int_rn(__fmul_rn(__fsub_rn(__fmul_rn(r1[nb][2 * e + 1], ig[nb][1]), bv), inv_a));
        k0 = min(max(k0, 0), L);
        k1 = min(max(k1, 0), L);
        const int t = e ? t1 : t0;
        sm.rec[512 + t * 68 + 4 * nb + j] = static_cast<unsigned char>(k0 | (k1 << 4));
      }
    }
    __syncthreads();
    // header (32 x 16 B) then 128 rows x 4 x 16 B of codes
    for (int i = tid; i < 32 + T * 4; i += 256) {
      uint4 v;
      if (i < 32) {
        v = *reinterpret_cast<const uint4*>(sm.rec + 16 * i);
      } else {
        const int k = i - 32, t = k >> 2, part = k & 3;
        const uint32_t* s = reinterpret_cast<const uint32_t*>(sm.rec + 512 + t * 68 + 16 * part);
        v = make_uint4(s[0], s[1], s[2], s[3]);
      }
      *reinterpret_cast<uint4*>(dst + 16 * i) = v;
    }
  } else {
    __syncthreads();  // inv_a / bval of every token are needed by copy 2
    const float ga = sm.inv_g[c0], gb = sm.inv_g[c0 + 1];
    uint64_t pa = 0, pb = 0;  // channel-major 2-bit codes of tokens 32q .. 32q+31
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int t = 32 * q + i;
      const float bv = sm.bval[t], inv_a = sm.inv_a[t];
      int ka = __float2int_rn(__fmul_rn(__fsub_rn(__fmul_rn(r2[i].x, ga), bv), inv_a));
      int kb = __float2int_rn(__fmul_rn(__fsub_rn(__fmul_rn(r2[i].y, gb), bv), inv_a));
      ka = min(max(ka, 0), L);
      kb = min(max(kb, 0), L);
      pa |= static_cast<uint64_t>(ka) << (2 * i);
      pb |= static_cast<uint64_t>(kb) << (2 * i);
    }
    *reinterpret_cast<uint64_t*>(sm.rec + 512 + c0 * 32 + 8 * q) = pa;
    *reinterpret_cast<uint64_t*>(sm.rec + 512 + (c0 + 1) * 32 + 8 * q) = pb;
    __syncthreads();
    for (int i = tid; i < V_REC / 16; i += 256)
      *reinterpret_cast<uint4*>(dst + 16 * i) = *reinterpret_cast<const uint4*>(sm.rec + 16 * i);
  }
}

// ------------------------------------------------------------------ kernels

// One CTA per (tile, head, K|V): blockIdx.x = (tile * H + head) * 2 + kv.
template <typename E>
__global__ void __launch_bounds__(256, 1) quantize_tiles_kernel(QuantizeParams prm) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  QSmem& sm = *reinterpret_cast<QSmem*>(smem_raw);
  const int job = blockIdx.x;
  const int kv = job & 1;
  const int h = (job >> 1) % prm.num_kv_heads;
  const int tile = (job >> 1) / prm.num_kv_heads;
  const int64_t first = prm.tile_first_token[tile];
  const int32_t blk = prm.tile_dst_block[tile];
  if (first < 0 || first + T > prm.n_tokens) {
    if (threadIdx.x == 0) set_error(prm.err, KVARN_DEV_ERR_TOKEN_RANGE);
    return;
  }
  if (blk < 0 || blk >= prm.num_blocks) {
    if (threadIdx.x == 0) set_error(prm.err, KVARN_DEV_ERR_BLOCK_RANGE);
    return;
  }
  const E* src = static_cast<const E*>(kv ? prm.v : prm.k) + first * prm.token_stride + h * D;
  unsigned char* dst = prm.pool + blk * prm.block_bytes + h * HEAD_REC + kv * K_REC;
  if (kv) quantize_tile_cta<E, true>(src, prm.token_stride, dst, prm.iters, sm);
  else quantize_tile_cta<E, false>(src, prm.token_stride, dst, prm.iters, sm);
}


// One CTA per (sequence, head, K|V): copy the new token into the open tile;
// the CTA whose token fills the tile quantises it into the sequence's block.
template <typename E>
__global__ void __launch_bounds__(256, 1) append_tokens_kernel(AppendParams prm) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  QSmem& sm = *reinterpret_cast<QSmem*>(smem_raw);
  const int b = blockIdx.x, h = blockIdx.y, kv = blockIdx.z;
  const int pos = prm.pos[b];
  if (pos < 0 || pos / T >= prm.max_blocks) {
    if (threadIdx.x == 0 && h == 0 && kv == 0) set_error(prm.err, KVARN_DEV_ERR_TOKEN_RANGE);
    return;
  }
  E* tile = static_cast<E*>(prm.tail) + ((static_cast<int64_t>(b) * prm.num_kv_heads + h) * 2 + kv) * (T * D);
  const int slot = pos & (T - 1);
  if (threadIdx.x < 16) {
    const E* src = static_cast<const E*>(kv ? prm.v_new : prm.k_new) + (static_cast<int64_t>(b) * prm.num_kv_heads + h) * D;
    reinterpret_cast<uint4*>(tile + slot * D)[threadIdx.x] = reinterpret_cast<const uint4*>(src)[threadIdx.x];
  }
  if (slot != T - 1) return;
  const int32_t blk = prm.block_table[static_cast<int64_t>(b) * prm.max_blocks + pos / T];
  if (blk < 0 || blk >= prm.num_blocks) {
    if (threadIdx.x == 0) set_error(prm.err, KVARN_DEV_ERR_BLOCK_RANGE);
    return;
  }
  __threadfence();
  __syncthreads();
  unsigned char* dst = prm.pool + blk * prm.block_bytes + h * HEAD_REC + kv * K_REC;
  if (kv) quantize_tile_cta<E, true>(tile, D, dst, prm.iters, sm);
  else quantize_tile_cta<E, false>(tile, D, dst, prm.iters, sm);
}

// Dequantise (tests): one CTA of 128 threads per (block, head, K|V); thread
// t rebuilds token t: R[t][c] = g[c] (a[t] code + b[t]), then X = R H by an
// in-register fast Walsh-Hadamard transform.
__global__ void __launch_bounds__(128) dequantize_kernel(const unsigned char* __restrict__ pool, int64_t block_bytes,
                                                         const int32_t* __restrict__ blocks, int32_t num_blocks,
                                                         int32_t num_kv_heads, float* __restrict__ out, int32_t* err) {
  __shared__ __align__(16) unsigned char rec[K_REC];
  const int n = blockIdx.x, h = blockIdx.y, kv = blockIdx.z, t = threadIdx.x;
  const int32_t blk = blocks[n];
  if (blk < 0 || blk >= num_blocks) {
    if (t == 0) set_error(err, KVARN_DEV_ERR_BLOCK_RANGE);
    return;
  }
  const unsigned char* src = pool + blk * block_bytes + h * HEAD_REC + kv * K_REC;
  const int bytes = kv ? V_REC : K_REC;
  for (int i = t; i < bytes / 16; i += 128)
    reinterpret_cast<uint4*>(rec)[i] = reinterpret_cast<const uint4*>(src)[i];
  __syncthreads();
  const float a = e4m3_to_float(rec[128 + t]);
  const float b = __half2float(*reinterpret_cast<const __half*>(rec + 256 + 2 * t));
  float x[D];
#pragma unroll
  for (int c = 0; c < D; ++c) {
    int code = kv ? (rec[512 + c * 32 + (t >> 2)] >> (2 * (t & 3))) & 3
                  : (rec[512 + t * 64 + (c >> 1)] >> (4 * (c & 1))) & 15;
    x[c] = e4m3_to_float(rec[c]) * fmaf(a, static_cast<float>(code), b);
  }
#pragma unroll
  for (int hh = 1; hh < D; hh <<= 1)
#pragma unroll
    for (int i = 0; i < D; ++i)
      if ((i & hh) == 0) {
        const float u = x[i], w = x[i + hh];
        x[i] = u + w;
        x[i + hh] = u - w;
      }
  float* o = out + (((static_cast<int64_t>(n) * 2 + kv) * num_kv_heads + h) * T + t) * D;
#pragma unroll
  for (int c = 0; c < D; c += 4)
    *reinterpret_cast<float4*>(o + c) =
        make_float4(x[c] * INV_SQRT_D, x[c + 1] * INV_SQRT_D, x[c + 2] * INV_SQRT_D, x[c + 3] * INV_SQRT_D);
}

// ------------------------------------------------------------------ launchers
size_t quantize_smem_bytes() { return sizeof(QSmem); }

template <typename E>
static cudaError_t launch_quantize_t(const QuantizeParams& p, int n_tiles, cudaStream_t s) {
  const size_t smem = sizeof(QSmem);
  cudaError_t e = cudaFuncSetAttribute(quantize_tiles_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t jobs = static_cast<int64_t>(n_tiles) * p.num_kv_heads * 2;
  quantize_tiles_kernel<E><<<static_cast<unsigned>(jobs), 256, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const QuantizeParams& p, int dtype, int n_tiles, cudaStream_t s) {
  return dtype == KVARN_DTYPE_BF16 ? launch_quantize_t<__nv_bfloat16>(p, n_tiles, s)
                                   : launch_quantize_t<__half>(p, n_tiles, s);
}

template <typename E>
static cudaError_t launch_append_t(const AppendParams& p, int batch, cudaStream_t s) {
  const size_t smem = sizeof(QSmem);
  cudaError_t e = cudaFuncSetAttribute(append_tokens_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  append_tokens_kernel<E><<<dim3(batch, p.num_kv_heads, 2), 256, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendParams& p, int dtype, int batch, cudaStream_t s) {
  return dtype == KVARN_DTYPE_BF16 ? launch_append_t<__nv_bfloat16>(p, batch, s) : launch_append_t<__half>(p, batch, s);
}

cudaError_t launch_dequantize(const unsigned char* pool, int64_t block_bytes, const int32_t* blocks, int n,
                              int num_blocks, int num_kv_heads, float* out, int32_t* err, cudaStream_t s) {
  dequantize_kernel<<<dim3(n, num_kv_heads, 2), 128, 0, s>>>(pool, block_bytes, blocks, num_blocks, num_kv_heads, out, err);
  return cudaGetLastError();
}

}  // namespace kvarn
