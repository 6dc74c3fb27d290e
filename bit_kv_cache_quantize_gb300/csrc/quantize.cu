// quantize.cu -- write path of the KVarN cache: one CTA quantises one
// 128-token x 128-channel tile of one KV head into a packed record.
//
// Steps (page "KVarN: 2-Bit KV-Cache That Beats FP16 Throughput, and Where
// the Catch Lives", section "What KVarN does differently"; page "Huawei's
// KVarN puts KV-cache quantization inside vLLM's backend", sections "What
// KVarN changes in vLLM's serving path" and "The four-stage pipeline"):
//   1. Hadamard rotation along channels, R = X H with the Sylvester H =
//      H8 (x) H16: a block-diagonal product with H16 on the tensor cores
//      (A = the 16-bit tile, exact; B = the +-1 signs generated in
//      registers; fp32 accumulate), then an 8-point Walsh-Hadamard transform
//      across the 16-channel groups in registers; scaled by 1/sqrt(128).
//   2. Sinkhorn-like normalisation in log space: N iterations of a column
//      step (log std over tokens of every channel) then a row step (log std
//      over channels of every token).  Each thread holds an 8-token x
//      8-channel block of R; the column step reduces across the lane pair
//      and the 8 warps through shared memory, the row step across the 16
//      lanes of a half-warp.  Each std is a shifted one-pass sum (shift = the
//      first element), exact for a constant row or column.
//   3. Column factors centred (geometric mean 1) -> FP8 E4M3 scale g.
//   4. Per token: Y = R / g, FP16 zero-point b = round-down(min Y), FP8 step
//      a = round-up((max Y - b) / L).
//   5. Codes rne((Y - b) * (1/a)), clamped to [0, L]; packed and stored with
//      16-byte stores.
#include <algorithm>

#include "common.cuh"
#include "params.h"

namespace kvarn {

// Shared memory of one quantiser CTA (~66 KB).  One area is reused: first
// the 16-bit tile (128 x 272 B), then per-warp transposition slabs (8 x 8 KB),
// then the packed record, the column partial sums and per-token scale pairs.
struct QSmem {
  alignas(128) unsigned char xs[65536];
  float beta[D + 12];                       // column factors exp(-v) of the last column step (beta_slot)
  float inv_g[D];
  float g[D];                               // the channel scales themselves (unrotated path)
  float vred[8];
};
constexpr int X_ROW = 272;                 // staging row stride: 256 B + 16 B pad
constexpr int OFF_PART = 9216;             // float2 [8 warps][PART_STRIDE]: column (mean, M2) over 16 tokens
// channel c of a warp's partials at c + c / 16: the lanes of a half-warp
// write channels 8 apart, which the skew spreads over all 16 bank pairs
// (without it they share 2), and the merge's 32 consecutive channels still
// take each bank pair twice, the minimum for 256 bytes
constexpr int PART_STRIDE = 136;
__host__ __device__ constexpr int part_slot(int c) { return c + (c >> 4); }
// channel c of the column factors at c + 4 (c / 32): each lane reads 8
// channels as two float4, 8 channels apart from the next lane's; shifting
// each 32-channel block by 4 more words spreads a half-warp over 8 bank
// quads instead of 4
__host__ __device__ constexpr int beta_slot(int c) { return c + 4 * (c >> 5); }
constexpr int OFF_TOK = 17408;             // float2 [128]: (zero-point, 1/step) per token
constexpr int OFF_ROW = 18432;             // per half-warp row-step slot: 8 x 36 partials, 8 shifts, 8 factors
constexpr int ROW_SLOT = 304;              // floats per slot
// Value codes staged for the record: channel c, word w at word
// ((c & 7) * 16 + (c >> 3)) * stride + w, stride 9 (2-bit, 8 words per
// channel) or 17 (4-bit, 16 words), so that the lanes of a warp, which hold
// channels 8 apart, store into different banks (the record's own 32- or
// 64-byte channel rows would put 16 lanes on one bank).
constexpr int OFF_STG = 40960;
__host__ __device__ constexpr int stg_stride(int kind_words) { return kind_words + 1; }
__device__ __forceinline__ int stg_index(int c, int w, int stride) { return ((c & 7) * 16 + (c >> 3)) * stride + w; }
static_assert(OFF_ROW + 16 * ROW_SLOT * 4 <= OFF_STG && T * 272 <= 65536, "staging reuse overflows");
static_assert(beta_slot(D - 1) < D + 12, "column factors overflow");
static_assert(OFF_PART + 8 * PART_STRIDE * 8 <= OFF_ROW && part_slot(D - 1) < PART_STRIDE,
              "column partials overflow (they may overlap the per-token values, which step 5 writes later)");
static_assert(OFF_STG + 4 * (127 * 17 + 16) <= 65536, "value staging overflows");

// New log factor ln(std) from a population variance and mean over 128
// values; keeps `old` when the std is at most 1e-6 of the rms (a constant or
// all-zero row/column).
__device__ __forceinline__ float log_std_or_keep(float var, float mean, float old) {
  var = fmaxf(var, 0.0f);
  return (var > 1e-12f * (var + mean * mean)) ? 0.5f * __logf(var) : old;
}

// Sum of 16 values (8 tokens x 2 quantities, index 2i + m) across the 16 lanes
// of a half-warp: recursive halving over lane bits 3, 2, 1, then a butterfly
// over bit 0.  Lane ends with the two totals of token ti = (lane & 15) >> 1.
// Selects keep every register index static.
template <typename Op>
__device__ __forceinline__ void halve16(float (&t)[8][2], int lane, Op op, float& r0, float& r1) {
  const bool b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
  float a[4][2];
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const float keep = b3 ? t[q + 4][m] : t[q][m];
      const float send = b3 ? t[q][m] : t[q + 4][m];
      a[q][m] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
  float c[2][2];
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const float keep = b2 ? a[q + 2][m] : a[q][m];
      const float send = b2 ? a[q][m] : a[q + 2][m];
      c[q][m] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
  float d[2];
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const float keep = b1 ? c[1][m] : c[0][m];
    const float send = b1 ? c[0][m] : c[1][m];
    d[m] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  }
  r0 = op(d[0], __shfl_xor_sync(0xffffffffu, d[0], 1));
  r1 = op(d[1], __shfl_xor_sync(0xffffffffu, d[1], 1));
}

// The 8 per-token values v[0..7] (identical in every lane of the half-warp)
// reduced the same way: value of token ti.
__device__ __forceinline__ float pick8(const float (&v)[8], int lane) {
  const int ti = (lane & 15) >> 1;
  float r = v[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) r = (ti == i) ? v[i] : r;
  return r;
}

// Record kinds written by the quantiser.
constexpr int KIND_K4 = 0;  // 4-bit keys, token-major nibbles (kvarn_k4v2 preset)
constexpr int KIND_V2 = 1;  // 2-bit values, channel-major even/odd token half-words
constexpr int KIND_K2 = 2;  // 2-bit keys, token-major, four codes per byte (K2/V2 preset)
constexpr int KIND_V4 = 3;  // 4-bit values, channel-major even/odd token half-words (K4/V4 preset)
__host__ __device__ constexpr int kind_levels(int kind) { return (kind == KIND_K4 || kind == KIND_V4) ? 15 : 3; }
__host__ __device__ constexpr int kind_rec_bytes(int kind) {
  return (kind == KIND_K4 || kind == KIND_V4) ? K_REC : V_REC;
}

struct AddOp { __device__ float operator()(float a, float b) const { return a + b; } };
struct MinOp { __device__ float operator()(float a, float b) const { return fminf(a, b); } };
struct MaxOp { __device__ float operator()(float a, float b) const { return fmaxf(a, b); } };

// Step 6 for this thread's 8 tokens x 8 channels: code = rne((Y - b) * (1/a))
// (two fp32 roundings, as written), clamped below at 0 when CLAMP; adding
// 1.5 * 2^23 leaves the rounded integer in the low mantissa bits.  With
// EXACT (the unrotated path, whose Y are exact quotients of the 16-bit
// inputs, so that (Y - b) / a often is exactly k + 1/2) the quotient is the
// correctly rounded IEEE division instead, and an exact tie goes to the
// even level as the definition says; tokv then holds a, not 1/a.  K4: byte
// pair p of token t = code[2p] | code[2p+1] << 4.  K2: byte i of token t =
// sum_k code[4i+k] << 2k.  V2: token 16w + u of a channel at bit u (u even)
// or 15 + u (u odd) of the channel's word w; tokens tok0 .. tok0+7
// (u = 8h + i) fill byte h (even i, at bit i) and byte 2 + h (odd i, at bit i - 1).
template <int KIND, bool CLAMP, bool EXACT = false>
__device__ __forceinline__ void encode_pack(const float2 (&r)[8][4], const float2* tokv, unsigned char* rec,
                                            int tok0, int cb) {
  constexpr int L = kind_levels(KIND);
  constexpr float RNE_MAGIC = 12582912.0f;
  const float2 MAG2 = make_float2(RNE_MAGIC, RNE_MAGIC);
  auto code2 = [&](float2 y, float2 nb, float2 ia) {
    float2 q2;
    if constexpr (EXACT) {
      const float2 d = fadd2(y, nb);
      q2 = make_float2(__fdiv_rn(d.x, ia.x), __fdiv_rn(d.y, ia.y));
    } else {
      q2 = fmul2(fadd2(y, nb), ia);
    }
    // a min between the product and the rounding add keeps the two from being
    // fused into one FMA (which would round once instead of twice); without
    // saturation it only ever trims L (1 + 2^-23) to L
    if constexpr (CLAMP) q2.x = fmaxf(q2.x, 0.f), q2.y = fmaxf(q2.y, 0.f);
    q2.x = fminf(q2.x, (float)L);
    q2.y = fminf(q2.y, (float)L);
    return fadd2(q2, MAG2);
  };
  if constexpr (KIND == KIND_K2) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 ta = tokv[tok0 + i];
      const float2 nb = make_float2(-ta.x, -ta.x), ia = make_float2(ta.y, ta.y);
      uint32_t bits16 = 0;  // channels 8cb .. 8cb+7 of token tok0 + i, channel 8cb + k at bits 2k
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const float2 q2 = code2(r[i][pp], nb, ia);
        bits16 |= ((__float_as_uint(q2.x) & 3u) << (4 * pp)) | ((__float_as_uint(q2.y) & 3u) << (4 * pp + 2));
      }
      *reinterpret_cast<uint16_t*>(rec + 512 + (tok0 + i) * 32 + 2 * cb) = (uint16_t)bits16;
    }
  } else if constexpr (KIND == KIND_K4) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 ta = tokv[tok0 + i];
      const float2 nb = make_float2(-ta.x, -ta.x), ia = make_float2(ta.y, ta.y);
      uint32_t u[4];
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const float2 q2 = code2(r[i][pp], nb, ia);
        // low byte = code_x + 16 code_y (both codes in [0, 15], the bits above them zero)
        u[pp] = (__float_as_uint(q2.y) << 4) + (__float_as_uint(q2.x) & 0xFu);
      }
      const uint32_t word = __byte_perm(__byte_perm(u[0], u[1], 0x0040), __byte_perm(u[2], u[3], 0x0040), 0x5410);
      *reinterpret_cast<uint32_t*>(rec + 512 + (tok0 + i) * 64 + 4 * cb) = word;
    }
  } else if constexpr (KIND == KIND_V4) {
    // the thread's 8 tokens are one 32-bit word per channel: token tok0 + u at
    // bit 2u (u even) or 14 + 2u (u odd); staged, see OFF_STG
    uint32_t word[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) word[k] = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 ta = tokv[tok0 + i];
      const float2 nb = make_float2(-ta.x, -ta.x), ia = make_float2(ta.y, ta.y);
      const int sh = (i & 1) ? 14 + 2 * i : 2 * i;
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const float2 q2 = code2(r[i][pp], nb, ia);
        word[2 * pp] |= (__float_as_uint(q2.x) & 15u) << sh;
        word[2 * pp + 1] |= (__float_as_uint(q2.y) & 15u) << sh;
      }
    }
    uint32_t* stg = reinterpret_cast<uint32_t*>(rec + OFF_STG);
#pragma unroll
    for (int k = 0; k < 8; ++k) stg[stg_index(8 * cb + k, tok0 >> 3, stg_stride(16))] = word[k];
  } else {
    uint32_t half[8];  // channel 8cb + k: even-token byte in bits 0-7, odd-token byte in bits 16-23
#pragma unroll
    for (int k = 0; k < 8; ++k) half[k] = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 ta = tokv[tok0 + i];
      const float2 nb = make_float2(-ta.x, -ta.x), ia = make_float2(ta.y, ta.y);
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const float2 q2 = code2(r[i][pp], nb, ia);
        const int sh = (i & 1) ? 15 + i : i;
        half[2 * pp] |= (__float_as_uint(q2.x) & 3u) << sh;
        half[2 * pp + 1] |= (__float_as_uint(q2.y) & 3u) << sh;
      }
    }
    // word (tok0 >> 4) of channel 8cb + k: bytes 0 / 2 from the half-warp with
    // the first 8 tokens (even / odd), bytes 1 / 3 from the one with the next
    // 8; the lane pair (cb, cb + 16) swaps its halves, and each lane stages
    // four of the eight words (see OFF_STG)
    const int hb = (tok0 >> 3) & 1;
    uint32_t* stg = reinterpret_cast<uint32_t*>(rec + OFF_STG);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t other = __shfl_xor_sync(0xffffffffu, half[k], 16);
      const uint32_t w = hb ? __byte_perm(other, half[k], 0x6240) : __byte_perm(half[k], other, 0x6240);
      if ((k >> 2) == hb) stg[stg_index(8 * cb + k, tok0 >> 4, stg_stride(8))] = w;
    }
  }
}

// Quantise one tile.  src: token rows of 128 16-bit channels, consecutive
// rows row_stride elements apart (16-byte aligned).  dst: the record in the
// pool.  All 256 threads of the CTA must call this.  After the rotation every
// thread holds one 8-token x 8-channel block of R: tokens 16w + 8(l >> 4) +
// 0..7, channels 8(l & 15) + 0..7 (warp w, lane l).
template <typename E, int KIND, bool ROT = true>
__device__ void quantize_tile_cta(const E* __restrict__ src, int64_t row_stride, unsigned char* __restrict__ dst,
                                  int iters, QSmem& sm) {
  constexpr int L = kind_levels(KIND);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, j = lane & 3;          // MMA fragment coordinates
  const int tbl = lane >> 4, cb = lane & 15;       // 8x8 block coordinates
  const int tok0 = 16 * warp + 8 * tbl;            // first token of this thread's block

  // ---- 1. stage X (16-bit) into shared memory
  for (int i = tid; i < T * 16; i += 256) {
    const int row = i >> 4, ch16 = i & 15;
    cp_async16(sm.xs + row * X_ROW + ch16 * 16, src + row * row_stride + ch16 * 8);
  }
  cp_async_wait_all();
  __syncthreads();
  float2 r[8][4];  // r[i][p] = R[tok0 + i][8cb + 2p .. 2p+1]
  if constexpr (!ROT) {  // the no-rotation ablation: R = X
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(sm.xs + (tok0 + i) * X_ROW + (8 * cb + 2 * pp) * 2);
        r[i][pp] = make_float2(bits2f<E>((uint16_t)(w & 0xFFFFu)), bits2f<E>((uint16_t)(w >> 16)));
      }
  } else {
  uint32_t afr[8][4];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    ldmatrix_x4(afr[ks], sm.xs + (16 * warp + (lane & 15)) * X_ROW + (16 * ks + (lane >> 4) * 8) * 2);
  __syncthreads();  // the staging area is reused below

  // ---- 2. R = X H; H[k][n] = (-1)^popcount(k & n) (Sylvester order)
  // With k = 16a' + b', n = 16a + b the sign splits, popcount(k & n) =
  // popcount(a' & a) + popcount(b' & b): H = H8 (x) H16.  So first
  // Y = X (I8 (x) H16) on the tensor cores, one MMA per 8-column block nb
  // (its 16-channel group a = nb >> 1 is k-block a), then R = Y (H8 (x) I16),
  // an 8-point Walsh-Hadamard transform across the groups that each lane does
  // in registers (it holds column 8nb + 2j (+1) of every block).  For
  // kk = k - 16a, n = 8nb + g: the H16 sign is popcount(kk & g) +
  // (kk >> 3)(nb & 1), so every B fragment is +-F, F the lane's base sign pair.
  {
    const uint32_t one = Bits16<E>::one;
    const uint32_t F = ((__popc((2 * j) & g) & 1) ? (one | 0x8000u) : one) |
                       (((__popc((2 * j + 1) & g) & 1) ? (one | 0x8000u) : one) << 16);
    const uint32_t NF = F ^ 0x80008000u;
    float acc[16][4];
#pragma unroll
    for (int nb = 0; nb < 16; ++nb) {
      acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
      mma16816<E>(acc[nb], afr[nb >> 1], F, (nb & 1) ? NF : F);
    }
#pragma unroll
    for (int st = 1; st < 8; st <<= 1)    // butterflies over the group index a, block nb = 2a + h
#pragma unroll
      for (int a = 0; a < 8; ++a)
        if (!(a & st))
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float u = acc[2 * a + h][e], v = acc[2 * (a ^ st) + h][e];
              acc[2 * a + h][e] = u + v;
              acc[2 * (a ^ st) + h][e] = u - v;
            }
    // transpose the warp's 16 x 128 slab into 8x8 blocks through 8 KB of
    // shared memory.  Column c of row r sits at c ^ 8 (r & 3) ^ 4 ((c >> 5) & 1):
    // both sides then take the minimum number of wavefronts (the readers'
    // 16 float4 of one row are 32 bytes apart, which without the second term
    // shares 4 bank quads among 16 lanes)
    float* slab = reinterpret_cast<float*>(sm.xs) + warp * 2048;
#pragma unroll
    for (int nb = 0; nb < 16; ++nb) {
      const int col = (8 * nb + 2 * j) ^ (8 * (g & 3)) ^ (4 * ((nb >> 2) & 1));
      *reinterpret_cast<float2*>(slab + g * 128 + col) = make_float2(acc[nb][0] * INV_SQRT_D, acc[nb][1] * INV_SQRT_D);
      *reinterpret_cast<float2*>(slab + (g + 8) * 128 + col) =
          make_float2(acc[nb][2] * INV_SQRT_D, acc[nb][3] * INV_SQRT_D);
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float4 v = *reinterpret_cast<const float4*>(slab + (8 * tbl + i) * 128 +
                                                          ((8 * cb + 4 * hh) ^ (8 * (i & 3)) ^ (4 * ((cb >> 2) & 1))));
        r[i][2 * hh] = make_float2(v.x, v.y);
        r[i][2 * hh + 1] = make_float2(v.z, v.w);
      }
  }
  }
  float2* part = reinterpret_cast<float2*>(sm.xs + OFF_PART);
  float2* tokv = reinterpret_cast<float2*>(sm.xs + OFF_TOK);
  __syncthreads();  // slabs done: the staging area now holds partials and the record

  // ---- 3. Sinkhorn-like iterations
  // column step: per thread, shifted sums over its 8 tokens of w = alpha_t
  // R[t][c] with shift = w at its first token (exact zero for a constant
  // column), turned into (mean, M2) and merged across threads pairwise
  // (M2 = M2a + M2b + d^2 na nb / (na + nb), d = difference of the means);
  // row step: shifted sums over channels of w = beta_c R[t][c], shift = the
  // row's channel-0 value, the same in every lane of the half-warp.
  float al[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) al[i] = 1.f;
  float v_c = 0.f;   // log factor of channel tid (tid < 128)
  float u_t = 0.f;   // log factor of token tok0 + ((lane & 15) >> 1)
  for (int it = 0; it < iters; ++it) {
    {
      const float2 a0 = make_float2(al[0], al[0]);
      float2 nK[4], s1[4], s2[4];
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const float2 K = fmul2(a0, r[0][pp]);
        nK[pp] = make_float2(-K.x, -K.y);
        s1[pp] = s2[pp] = make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 a2 = make_float2(al[i], al[i]);
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const float2 d = ffma2(a2, r[i][pp], nK[pp]);
          s1[pp] = fadd2(s1[pp], d);
          s2[pp] = ffma2(d, d, s2[pp]);
        }
      }
      float2 mean[4], M2[4];   // over this thread's 8 tokens
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        mean[pp] = ffma2(s1[pp], make_float2(0.125f, 0.125f), make_float2(-nK[pp].x, -nK[pp].y));
        M2[pp] = ffma2(fmul2(s1[pp], make_float2(-0.125f, -0.125f)), s1[pp], s2[pp]);
      }
      // lane pair (tbl 0, tbl 1) shares channels: tbl 0 keeps pairs 0-1, tbl 1 keeps 2-3
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float2 km = tbl ? mean[q + 2] : mean[q], kM = tbl ? M2[q + 2] : M2[q];
        const float2 om = tbl ? mean[q] : mean[q + 2], oM = tbl ? M2[q] : M2[q + 2];
        const float2 pm = make_float2(__shfl_xor_sync(0xffffffffu, om.x, 16), __shfl_xor_sync(0xffffffffu, om.y, 16));
        const float2 pM = make_float2(__shfl_xor_sync(0xffffffffu, oM.x, 16), __shfl_xor_sync(0xffffffffu, oM.y, 16));
        const float2 dl = make_float2(km.x - pm.x, km.y - pm.y);
        const float2 m16 = fmul2(fadd2(km, pm), make_float2(0.5f, 0.5f));
        const float2 M16 = ffma2(fmul2(dl, make_float2(4.f, 4.f)), dl, fadd2(kM, pM));
        const int c = 8 * cb + 4 * tbl + 2 * q;
        part[warp * PART_STRIDE + part_slot(c)] = make_float2(m16.x, M16.x);
        part[warp * PART_STRIDE + part_slot(c + 1)] = make_float2(m16.y, M16.y);
      }
    }
    __syncthreads();
    if (tid < D) {
      float mw[8], msum = 0.f, M2 = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float2 v = part[w * PART_STRIDE + part_slot(tid)];
        mw[w] = v.x; msum += v.x; M2 += v.y;
      }
      const float mean = msum * 0.125f;
#pragma unroll
      for (int w = 0; w < 8; ++w) M2 = fmaf(16.f * (mw[w] - mean), mw[w] - mean, M2);
      v_c = log_std_or_keep(M2 * (1.0f / 128.0f), mean, v_c);
      sm.beta[beta_slot(tid)] = __expf(-v_c);
    }
    __syncthreads();
    // row step: the half-warp holding tokens tok0 .. tok0+7 reduces through
    // its own shared-memory slot: row shifts, 16 partial pairs per lane, then
    // each token's owner lanes (cb = 2i, 2i+1) sum the 16 partials of token i
    {
      float* rs = reinterpret_cast<float*>(sm.xs + OFF_ROW) + (2 * warp + tbl) * ROW_SLOT;
      const float4 b0 = *reinterpret_cast<const float4*>(sm.beta + beta_slot(8 * cb));
      const float4 b1 = *reinterpret_cast<const float4*>(sm.beta + beta_slot(8 * cb) + 4);
      const float2 bp[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                            make_float2(b1.z, b1.w)};
      if (cb == 0) {  // channel 0 of each token: the shift of its row
        *reinterpret_cast<float4*>(rs + 288) =
            make_float4(bp[0].x * r[0][0].x, bp[0].x * r[1][0].x, bp[0].x * r[2][0].x, bp[0].x * r[3][0].x);
        *reinterpret_cast<float4*>(rs + 292) =
            make_float4(bp[0].x * r[4][0].x, bp[0].x * r[5][0].x, bp[0].x * r[6][0].x, bp[0].x * r[7][0].x);
      }
      __syncwarp();
      float Kt[8];
      {
        const float4 k0 = *reinterpret_cast<const float4*>(rs + 288), k1 = *reinterpret_cast<const float4*>(rs + 292);
        Kt[0] = k0.x; Kt[1] = k0.y; Kt[2] = k0.z; Kt[3] = k0.w; Kt[4] = k1.x; Kt[5] = k1.y; Kt[6] = k1.z; Kt[7] = k1.w;
      }
      float t2[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 nK = make_float2(-Kt[i], -Kt[i]);
        float2 s1 = make_float2(0.f, 0.f), s2 = s1;
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const float2 d = ffma2(bp[pp], r[i][pp], nK);
          s1 = fadd2(s1, d);
          s2 = ffma2(d, d, s2);
        }
        t2[2 * i] = s1.x + s1.y;
        t2[2 * i + 1] = s2.x + s2.y;
      }
      // partial pairs: slot layout [token i (stride 36)][lane cb] float2: the owner's 16 reads are
      // contiguous and the 8 owners hit different banks
#pragma unroll
      for (int i = 0; i < 8; ++i) *reinterpret_cast<float2*>(rs + 36 * i + 2 * cb) = make_float2(t2[2 * i], t2[2 * i + 1]);
      __syncwarp();
      const int ti = cb >> 1;
      float2 S = make_float2(0.f, 0.f);
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const float4 v = *reinterpret_cast<const float4*>(rs + 36 * ti + 4 * q4);
        S = fadd2(S, make_float2(v.x + v.z, v.y + v.w));
      }
      const float md = S.x * (1.0f / 128.0f);
      u_t = log_std_or_keep(S.y * (1.0f / 128.0f) - md * md, rs[288 + ti] + md, u_t);
      __syncwarp();
      if ((cb & 1) == 0) rs[296 + ti] = __expf(-u_t);
      __syncwarp();
      const float4 a0 = *reinterpret_cast<const float4*>(rs + 296), a1 = *reinterpret_cast<const float4*>(rs + 300);
      al[0] = a0.x; al[1] = a0.y; al[2] = a0.z; al[3] = a0.w; al[4] = a1.x; al[5] = a1.y; al[6] = a1.z; al[7] = a1.w;
      __syncwarp();
    }
  }

  // ---- 4. gauge and per-channel FP8 scales
  unsigned char* rec = sm.xs;
  {
    float s = (tid < D) ? v_c : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) sm.vred[warp] = s;
  }
  __syncthreads();
  if (tid < D) {
    float mean = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) mean += sm.vred[w];
    mean *= (1.0f / 128.0f);
    uint8_t gc = float_to_e4m3_rn(expf(v_c - mean));
    if (gc == 0) gc = 0x01;
    rec[tid] = gc;
    sm.inv_g[tid] = __frcp_rn(e4m3_to_float(gc));
    sm.g[tid] = e4m3_to_float(gc);
  }
  __syncthreads();

  // ---- 5. per-token zero-point and step
  bool sat;
  float2 ig[4];
  {
    const float4 g0 = *reinterpret_cast<const float4*>(sm.inv_g + 8 * cb);
    const float4 g1 = *reinterpret_cast<const float4*>(sm.inv_g + 8 * cb + 4);
    ig[0] = make_float2(g0.x, g0.y); ig[1] = make_float2(g0.z, g0.w);
    ig[2] = make_float2(g1.x, g1.y); ig[3] = make_float2(g1.z, g1.w);
  }
  if constexpr (ROT) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) r[i][pp] = fmul2(r[i][pp], ig[pp]);   // r now holds Y = R / g
  } else {  // unrotated: Y = X / g correctly rounded (exact whenever the quotient is an fp32 number)
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int pp = 0; pp < 4; ++pp)
        r[i][pp] = make_float2(__fdiv_rn(r[i][pp].x, sm.g[8 * cb + 2 * pp]), __fdiv_rn(r[i][pp].y, sm.g[8 * cb + 2 * pp + 1]));
  }
  {
    float mm[8][2];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float a = fminf(r[i][0].x, r[i][0].y), bmax = fmaxf(r[i][0].x, r[i][0].y);
#pragma unroll
      for (int pp = 1; pp < 4; ++pp) {
        a = fminf(a, fminf(r[i][pp].x, r[i][pp].y));
        bmax = fmaxf(bmax, fmaxf(r[i][pp].x, r[i][pp].y));
      }
      mm[i][0] = -a;     // max of -Y = -(min of Y): one max-reduction for both
      mm[i][1] = bmax;
    }
    float nymin, ymax;
    halve16(mm, lane, MaxOp(), nymin, ymax);
    const float ymin = -nymin;
    const __half bh = (ymin <= -65504.f) ? __float2half_rn(-65504.f) : __float2half_rd(ymin);
    const float bv = __half2float(bh);
    const float step = __fdiv_ru(__fsub_ru(ymax, bv), (float)L);
    uint8_t ac = float_to_e4m3_ru(step);
    if (ac == 0) ac = 0x01;
    const float inv_a = __frcp_rn(e4m3_to_float(ac));
    // without saturation b <= min Y and a >= (max Y - b) / L, so every
    // (Y - b) * (1/a) lies in [0, L (1 + 2^-23)]: no clamp at 0 needed
    sat = !(ymin > -65504.f) || !(step <= 448.f);
    if ((lane & 1) == 0) {
      const int tk = tok0 + ((lane & 15) >> 1);
      rec[128 + tk] = ac;
      *reinterpret_cast<__half*>(rec + 256 + 2 * tk) = bh;
      tokv[tk] = make_float2(bv, ROT ? inv_a : e4m3_to_float(ac));
    }
  }
  const bool clamp_codes = __syncthreads_or(sat);

  // ---- 6. codes and packing: code = rne((Y - b) * (1/a)), clamped to [0, L]
  // only in a tile where some token saturated its zero-point or step
  if (clamp_codes) encode_pack<KIND, true, !ROT>(r, tokv, rec, tok0, cb);
  else encode_pack<KIND, false, !ROT>(r, tokv, rec, tok0, cb);
  __syncthreads();
  const int bytes = kind_rec_bytes(KIND);
  if constexpr (KIND == KIND_V2 || KIND == KIND_V4) {  // header from the record, codes from the staging
    constexpr int WPC = KIND == KIND_V2 ? 8 : 16;      // code words per channel
    const uint32_t* stg = reinterpret_cast<const uint32_t*>(rec + OFF_STG);
    for (int i = tid; i < bytes / 16; i += 256) {
      uint4 v;
      if (i < 32) {
        v = *reinterpret_cast<const uint4*>(rec + 16 * i);
      } else {
        const int q = 4 * (i - 32), c = q / WPC, w = q % WPC;
        const uint32_t* src = stg + stg_index(c, w, stg_stride(WPC));
        v = make_uint4(src[0], src[1], src[2], src[3]);
      }
      *reinterpret_cast<uint4*>(dst + 16 * i) = v;
    }
  } else {
    for (int i = tid; i < bytes / 16; i += 256)
      *reinterpret_cast<uint4*>(dst + 16 * i) = *reinterpret_cast<const uint4*>(rec + 16 * i);
  }
}

// ------------------------------------------------------------------ kernels

// One CTA per (tile, head, K|V): blockIdx.x = (tile * H + head) * 2 + kv.
template <typename E>
__global__ void __launch_bounds__(256, 2) quantize_tiles_kernel(QuantizeParams prm) {
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
  unsigned char* dst =
      prm.pool + blk * prm.block_bytes + h * head_rec(prm.k_bits, prm.v_bits) + kv * rec_bytes(prm.k_bits);
  if (!kcheck(dst, rec_bytes(kv ? prm.v_bits : prm.k_bits), prm.pool, (size_t)prm.num_blocks * prm.block_bytes,
              prm.err) ||
      !kcheck(src, ((T - 1) * prm.token_stride + D) * sizeof(E), kv ? prm.v : prm.k,
              (size_t)prm.n_tokens * prm.token_stride * sizeof(E), prm.err))
    return;
  if (kv && prm.v_bits == 4) quantize_tile_cta<E, KIND_V4>(src, prm.token_stride, dst, prm.iters, sm);
  else if (kv) quantize_tile_cta<E, KIND_V2>(src, prm.token_stride, dst, prm.iters, sm);
  else if (prm.k_bits == 4) quantize_tile_cta<E, KIND_K4>(src, prm.token_stride, dst, prm.iters, sm);
  else quantize_tile_cta<E, KIND_K2>(src, prm.token_stride, dst, prm.iters, sm);
}


// Append one token per (sequence, head, K|V) unit to its open tile; a token
// that fills the tile has the whole CTA quantise it into the sequence's block.
// The grid is at most two CTAs per SM: most units only copy 256 bytes, and a
// grid of one 66 KB CTA per unit would take batch x heads x 2 / (2 x SMs)
// waves to do it.
template <typename E>
__global__ void __launch_bounds__(256, 2) append_tokens_kernel(AppendParams prm) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  QSmem& sm = *reinterpret_cast<QSmem*>(smem_raw);
  __shared__ int32_t close_blk[16];  // per unit of the current pass: block its tile closes into, or -1
  const int64_t units = static_cast<int64_t>(prm.batch) * prm.num_kv_heads * 2;
  const size_t tail_bytes = (size_t)units * T * D * sizeof(E);
  const int grp = threadIdx.x >> 4, gl = threadIdx.x & 15;
  // This CTA owns units blockIdx.x + k * gridDim.x (unit = (sequence, head,
  // K|V)), sixteen per pass.
  for (int64_t r0 = blockIdx.x; r0 < units; r0 += 16LL * gridDim.x) {
    // 1. sixteen threads per unit copy its token into the open tile and note
    //    whether the token closes the tile
    const int64_t u = r0 + static_cast<int64_t>(grp) * gridDim.x;
    int32_t cb = -1;
    if (u < units) {
      const int kv = static_cast<int>(u & 1);
      const int h = static_cast<int>((u >> 1) % prm.num_kv_heads), b = static_cast<int>((u >> 1) / prm.num_kv_heads);
      const int pos = prm.pos[b];
      if (pos < 0 || pos / T >= prm.max_blocks) {
        if (gl == 0 && h == 0 && kv == 0) set_error(prm.err, KVARN_DEV_ERR_TOKEN_RANGE);
      } else {
        E* tile = static_cast<E*>(prm.tail) + u * (T * D);
        const int slot = pos & (T - 1);
        if (kcheck(tile, T * D * sizeof(E), prm.tail, tail_bytes, prm.err)) {
          const E* src = static_cast<const E*>(kv ? prm.v_new : prm.k_new) + (u >> 1) * D;
          reinterpret_cast<uint4*>(tile + slot * D)[gl] = reinterpret_cast<const uint4*>(src)[gl];
          if (slot == T - 1) {
            const int32_t blk = prm.block_table[static_cast<int64_t>(b) * prm.max_blocks + pos / T];
            if (blk >= 0 && blk < prm.num_blocks) {
              cb = blk;
              __threadfence();  // the token reaches L2 before the CTA's cp.async reads the tile
            } else if (gl == 0) {
              set_error(prm.err, KVARN_DEV_ERR_BLOCK_RANGE);
            }
          }
        }
      }
    }
    if (gl == 0) close_blk[grp] = cb;
    __syncthreads();
    // 2. the whole CTA quantises the closed tiles one after another
    for (int j = 0; j < 16; ++j) {
      const int32_t blk = close_blk[j];
      if (blk < 0) continue;
      const int64_t uj = r0 + static_cast<int64_t>(j) * gridDim.x;
      const int kv = static_cast<int>(uj & 1), h = static_cast<int>((uj >> 1) % prm.num_kv_heads);
      const E* tile = static_cast<const E*>(prm.tail) + uj * (T * D);
      unsigned char* dst =
          prm.pool + blk * prm.block_bytes + h * head_rec(prm.k_bits, prm.v_bits) + kv * rec_bytes(prm.k_bits);
      if (!kcheck(dst, rec_bytes(kv ? prm.v_bits : prm.k_bits), prm.pool, (size_t)prm.num_blocks * prm.block_bytes,
                  prm.err))
        continue;
      if (kv && prm.v_bits == 4) quantize_tile_cta<E, KIND_V4>(tile, D, dst, prm.iters, sm);
      else if (kv) quantize_tile_cta<E, KIND_V2>(tile, D, dst, prm.iters, sm);
      else if (prm.k_bits == 4) quantize_tile_cta<E, KIND_K4>(tile, D, dst, prm.iters, sm);
      else quantize_tile_cta<E, KIND_K2>(tile, D, dst, prm.iters, sm);
      __syncthreads();  // the next tile reuses the shared memory
    }
    __syncthreads();  // close_blk is rewritten by the next pass
  }
}

// Dequantise (tests): one CTA of 128 threads per (block, head, K|V); thread
// t rebuilds token t: R[t][c] = g[c] (a[t] code + b[t]), then X = R H by an
// in-register fast Walsh-Hadamard transform.
__global__ void __launch_bounds__(128) dequantize_kernel(const unsigned char* __restrict__ pool, int64_t block_bytes,
                                                         const int32_t* __restrict__ blocks, int32_t num_blocks,
                                                         int32_t num_kv_heads, int32_t k_bits, int32_t v_bits,
                                                         float* __restrict__ out,
                                                         int32_t* err) {
  __shared__ __align__(16) unsigned char rec[K_REC];
  const int n = blockIdx.x, h = blockIdx.y, kv = blockIdx.z, t = threadIdx.x;
  const int32_t blk = blocks[n];
  if (blk < 0 || blk >= num_blocks) {
    if (t == 0) set_error(err, KVARN_DEV_ERR_BLOCK_RANGE);
    return;
  }
  const unsigned char* src = pool + blk * block_bytes + h * head_rec(k_bits, v_bits) + kv * rec_bytes(k_bits);
  const int bytes = kv ? rec_bytes(v_bits) : rec_bytes(k_bits);
  float* const o0 = out + ((static_cast<int64_t>(n) * 2 + kv) * num_kv_heads + h) * T * D;  // this CTA's rows
  if (!kcheck(src, bytes, pool, (size_t)num_blocks * block_bytes, err) ||
      !kcheck(o0, T * D * sizeof(float), out, (size_t)gridDim.x * 2 * num_kv_heads * T * D * sizeof(float), err))
    return;
  float* o = o0 + t * D;
  for (int i = t; i < bytes / 16; i += 128)
    reinterpret_cast<uint4*>(rec)[i] = reinterpret_cast<const uint4*>(src)[i];
  __syncthreads();
  const float a = e4m3_to_float(rec[128 + t]);
  const float b = __half2float(*reinterpret_cast<const __half*>(rec + 256 + 2 * t));
  float x[D];
#pragma unroll
  for (int c = 0; c < D; ++c) {
    const int vb = (t & 1) ? 15 + (t & 15) : (t & 15);          // bit of token t in its 2-bit V word
    const int vb4 = (t & 1) ? 14 + 2 * (t & 7) : 2 * (t & 7);  // bit of token t in its 4-bit V word
    int code = kv ? (v_bits == 4 ? (rec[512 + c * 64 + 4 * (t >> 3) + (vb4 >> 3)] >> (vb4 & 7)) & 15
                                 : (rec[512 + c * 32 + 4 * (t >> 4) + (vb >> 3)] >> (vb & 7)) & 3)
               : k_bits == 4 ? (rec[512 + t * 64 + (c >> 1)] >> (4 * (c & 1))) & 15
                             : (rec[512 + t * 32 + (c >> 2)] >> (2 * (c & 3))) & 3;
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
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = smem_attr_once(attr_done, (const void*)quantize_tiles_kernel<E>, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t jobs = static_cast<int64_t>(n_tiles) * p.num_kv_heads * 2;
  quantize_tiles_kernel<E><<<static_cast<unsigned>(jobs), 256, smem, s>>>(p);
  return cudaGetLastError();
}

// ---- per-token errors: quantise a tile into a scratch record, dequantise it
// and compare with the input.  One CTA (256 threads) per (tile, head); in the
// comparison thread 2t + hf takes channels 64 hf .. 64 hf + 63 of token t.
template <typename E, int KIND, bool ROT>
__global__ void __launch_bounds__(256, 2) token_errors_kernel(ErrParams prm) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  QSmem& sm = *reinterpret_cast<QSmem*>(smem_raw);
  const int job = blockIdx.x, h = job % prm.num_kv_heads, tile = job / prm.num_kv_heads;
  const int64_t first = prm.tile_first_token[tile];
  if (first < 0 || first + T > prm.n_tokens) {
    if (threadIdx.x == 0) set_error(prm.err, KVARN_DEV_ERR_TOKEN_RANGE);
    return;
  }
  const E* src = static_cast<const E*>(prm.x) + first * prm.token_stride + h * D;
  unsigned char* rec = prm.scratch + (int64_t)job * kind_rec_bytes(KIND);
  if (!kcheck(rec, kind_rec_bytes(KIND), prm.scratch, (size_t)gridDim.x * kind_rec_bytes(KIND), prm.err) ||
      !kcheck(prm.out + (int64_t)job * T * 2, T * 2 * sizeof(float), prm.out, (size_t)gridDim.x * T * 2 * sizeof(float),
              prm.err) ||
      !kcheck(src, ((T - 1) * prm.token_stride + D) * sizeof(E), prm.x,
              (size_t)prm.n_tokens * prm.token_stride * sizeof(E), prm.err))
    return;
  quantize_tile_cta<E, KIND, ROT>(src, prm.token_stride, rec, prm.iters, sm);
  __syncthreads();  // the record is in global memory, written by this CTA
  const int t = threadIdx.x >> 1, hf = threadIdx.x & 1;
  const float a = e4m3_to_float(rec[128 + t]);
  const float b = __half2float(*reinterpret_cast<const __half*>(rec + 256 + 2 * t));
  float x[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const int c = 64 * hf + i;
    int code;
    if constexpr (KIND == KIND_V2) {
      const int vb = (t & 1) ? 15 + (t & 15) : (t & 15);  // bit of token t in its channel word
      code = (rec[512 + c * 32 + 4 * (t >> 4) + (vb >> 3)] >> (vb & 7)) & 3;
    } else if constexpr (KIND == KIND_V4) {
      const int vb = (t & 1) ? 14 + 2 * (t & 7) : 2 * (t & 7);
      code = (rec[512 + c * 64 + 4 * (t >> 3) + (vb >> 3)] >> (vb & 7)) & 15;
    } else if constexpr (KIND == KIND_K4) {
      code = (rec[512 + t * 64 + (c >> 1)] >> (4 * (c & 1))) & 15;
    } else {
      code = (rec[512 + t * 32 + (c >> 2)] >> (2 * (c & 3))) & 3;
    }
    x[i] = e4m3_to_float(rec[c]) * fmaf(a, static_cast<float>(code), b);
  }
  if constexpr (ROT) {  // x = R H / sqrt(128): 64-point butterflies here, the last stage across the lane pair
#pragma unroll
    for (int m = 1; m < 64; m <<= 1)
#pragma unroll
      for (int i = 0; i < 64; ++i)
        if (!(i & m)) {
          const float u = x[i], w = x[i + m];
          x[i] = u + w;
          x[i + m] = u - w;
        }
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, x[i], 1);
      x[i] = (hf ? (o - x[i]) : (x[i] + o)) * INV_SQRT_D;
    }
  }
  float e2 = 0.f, n2 = 0.f;
  const E* row = src + (int64_t)t * prm.token_stride + 64 * hf;
#pragma unroll
  for (int i = 0; i < 64; i += 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float x0 = bits2f<E>((uint16_t)(w[k] & 0xFFFFu)), x1 = bits2f<E>((uint16_t)(w[k] >> 16));
      const float d0 = x[i + 2 * k] - x0, d1 = x[i + 2 * k + 1] - x1;
      e2 = fmaf(d0, d0, fmaf(d1, d1, e2));
      n2 = fmaf(x0, x0, fmaf(x1, x1, n2));
    }
  }
  e2 += __shfl_xor_sync(0xffffffffu, e2, 1);
  n2 += __shfl_xor_sync(0xffffffffu, n2, 1);
  if (hf == 0) *reinterpret_cast<float2*>(prm.out + ((int64_t)job * T + t) * 2) = make_float2(e2, n2);
}

template <typename E, int KIND>
static cudaError_t launch_errors_k(const ErrParams& p, int n_tiles, cudaStream_t s) {
  const size_t smem = sizeof(QSmem);
  const dim3 grid(n_tiles * p.num_kv_heads);
  if (p.rotate) {
    static std::atomic<uint64_t> attr_done{0};
    cudaError_t e = smem_attr_once(attr_done, (const void*)token_errors_kernel<E, KIND, true>, (int)smem);
    if (e != cudaSuccess) return e;
    token_errors_kernel<E, KIND, true><<<grid, 256, smem, s>>>(p);
  } else {
    static std::atomic<uint64_t> attr_done{0};
    cudaError_t e = smem_attr_once(attr_done, (const void*)token_errors_kernel<E, KIND, false>, (int)smem);
    if (e != cudaSuccess) return e;
    token_errors_kernel<E, KIND, false><<<grid, 256, smem, s>>>(p);
  }
  return cudaGetLastError();
}

template <typename E>
static cudaError_t launch_errors_t(const ErrParams& p, int n_tiles, cudaStream_t s) {
  if (p.is_v) return p.v_bits == 4 ? launch_errors_k<E, KIND_V4>(p, n_tiles, s) : launch_errors_k<E, KIND_V2>(p, n_tiles, s);
  return p.k_bits == 2 ? launch_errors_k<E, KIND_K2>(p, n_tiles, s) : launch_errors_k<E, KIND_K4>(p, n_tiles, s);
}

cudaError_t launch_token_errors(const ErrParams& p, int dtype, int n_tiles, cudaStream_t s) {
  return dtype == KVARN_DTYPE_BF16 ? launch_errors_t<__nv_bfloat16>(p, n_tiles, s) : launch_errors_t<__half>(p, n_tiles, s);
}

cudaError_t launch_quantize(const QuantizeParams& p, int dtype, int n_tiles, cudaStream_t s) {
  return dtype == KVARN_DTYPE_BF16 ? launch_quantize_t<__nv_bfloat16>(p, n_tiles, s)
                                   : launch_quantize_t<__half>(p, n_tiles, s);
}

template <typename E>
static cudaError_t launch_append_t(const AppendParams& p, int batch, cudaStream_t s) {
  const size_t smem = sizeof(QSmem);
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = smem_attr_once(attr_done, (const void*)append_tokens_kernel<E>, (int)smem);
  if (e != cudaSuccess) return e;
  // at most two CTAs per SM (the 66 KB of shared memory a closing tile needs)
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  AppendParams q = p;
  q.batch = batch;
  const long long units = (long long)batch * p.num_kv_heads * 2;
  int grid = (int)std::min<long long>(units, 2LL * std::max(sms, 1));
  if (grid > 1 && grid % 2 == 0) --grid;  // odd: each CTA's units alternate K and V tiles
  append_tokens_kernel<E><<<grid, 256, smem, s>>>(q);
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendParams& p, int dtype, int batch, cudaStream_t s) {
  return dtype == KVARN_DTYPE_BF16 ? launch_append_t<__nv_bfloat16>(p, batch, s) : launch_append_t<__half>(p, batch, s);
}

cudaError_t launch_dequantize(const unsigned char* pool, int64_t block_bytes, const int32_t* blocks, int n,
                              int num_blocks, int num_kv_heads, int k_bits, int v_bits, float* out, int32_t* err,
                              cudaStream_t s) {
  dequantize_kernel<<<dim3(n, num_kv_heads, 2), 128, 0, s>>>(pool, block_bytes, blocks, num_blocks, num_kv_heads,
                                                              k_bits, v_bits, out, err);
  return cudaGetLastError();
}

}  // namespace kvarn
