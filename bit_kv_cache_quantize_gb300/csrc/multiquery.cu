// multiquery.cu -- causal multi-query attention over the packed paged cache.
//
// Several new query tokens per sequence (a chunk of prefill, or the draft
// tokens a speculative step verifies) attend to the cache the way one decode
// query does: the closed tiles are read as packed records and dequantised
// inside the attention loop, the open tile is read raw ("Huawei's KVarN puts
// KV-cache quantization inside vLLM's backend", section "The four-stage
// pipeline": dequantisation at read time inside attention).  Query i of a
// sequence of length L sits at position L - n_queries + i and sees the
// tokens at positions <= its own.
//
// With the GQA group folded in, one KV head carries n_queries * G query rows;
// 128 of them form a row block, which makes both contractions full
// 128-row tensor-core tiles.  Per packed tile (128 tokens, one KV head):
//
//   QK (tcgen05, fp16, M = 128 rows, N = 144, K = 128 channels):
//     A = Q' (rotated, scaled query rows; fp16 hi and lo halves, two passes),
//     B = K~ with K~[t][c] = gK_c code_tc / 64 (exact in fp16) for the 128
//     tokens and K~[128][c] = gK_c / 64, so that
//       score_t = (64 / qs) (aK_t D[t] + bK_t D[128]).
//   softmax (two threads per row, one per 64-token half, scores from tensor
//     memory; the halves exchange their maxima through shared memory):
//     running reference m per row, moved only when a tile maximum exceeds it
//     by more than 8 (log2 units), which rescales the accumulator.
//   PV (tcgen05, bf16, M = 128 rows, N = 128 channels, K = 144):
//     A = P~ with P~[t] = p_t aV_t (bf16 hi and lo, two passes) and
//     P~[128], P~[129] = hi and lo of beta = sum_t p_t bV_t; B = V~ with
//     V~[c][t] = gV_c codeV_tc and V~[c][128] = V~[c][129] = gV_c (exact in
//     bf16), so the accumulator collects sum_t p_t gV_c (aV_t code + bV_t).
//
// Warp roles per CTA (13 warps, one CTA per SM): warps 0-7 run the softmax
// (warp w: rows 32 (w & 3) .. + 31, token half w >> 2), warps 8-11 unpack
// records into the K~ / V~ operands (their first thread refills a record
// stage once all of them are done with it), one thread of warp 12 issues
// the first bulk copies and the MMAs.  Operands that a later tile reuses are
// double-buffered (K~, scores, scales) or guarded by the previous PV (V~).
#include <type_traits>

#include "common.cuh"
#include "tcgen05.cuh"

namespace kvarn {
namespace {

constexpr float MQ_LOG2E = 1.4426950408889634f;
constexpr uint32_t MAGIC_F16 = 0x64006400u;  // 1024.0 in both fp16 halves
constexpr uint32_t MAGIC_BF16 = 0x43004300u; // 128.0 in both bf16 halves
constexpr int MQ_ROWS = 128;
constexpr int MQ_THREADS = 416;  // warps 0-7 softmax (two per row quarter), 8-11 unpack, 12 issue
constexpr int MQ_PART = D + 4;  // floats per split-K partial row: m, l, 2 pad, acc[128]
constexpr int MQ_PACC = 4;
constexpr int KT_ROWS = 144;                 // 128 tokens, the g row, 15 zero rows
constexpr int KT_BYTES = KT_ROWS * D * 2;    // K~, fp16, K-major core matrices
constexpr int VT_K = 144;                    // 128 tokens, beta hi / lo, 14 zero columns
constexpr int VT_BYTES = D * VT_K * 2;       // V~, bf16, K-major core matrices
constexpr int QA_BYTES = MQ_ROWS * D * 2;
constexpr int REC_STAGES = 3;
// tensor-memory columns: accumulator O, then two score buffers S (144 each).
// The softmax overwrites a tile's scores in place, first with the scaled
// scores, then with the P~ operand: for tokens 16 j .. 16 j + 15 the bf16 hi
// parts go to columns 16 j .. 16 j + 7 and the lo parts to 16 j + 8 .. 16 j + 15
// (exactly the columns those tokens' scores occupied); columns 128..135 take
// the beta entries (k 128..143).
constexpr uint32_t TM_O = 0, TM_S = 128, TM_SSTRIDE = 144, TM_COLS = 512;
constexpr uint32_t TM_QA = 416;  // Q' hi (the A operand of the first QK pass), 64 columns
constexpr uint32_t IDESC_QK = umma_idesc(128, KT_ROWS, 0);
constexpr uint32_t IDESC_PV = umma_idesc(128, D, 1);
constexpr float MQ_TAU = 8.f;  // log2 headroom before the row reference moves

struct MQSmem {
  alignas(128) unsigned char qa_lo[QA_BYTES];  // Q' lo (the hi half lives in tensor memory)
  alignas(128) unsigned char kt[2][KT_BYTES];
  alignas(128) unsigned char vt[VT_BYTES];
  alignas(128) unsigned char rec[REC_STAGES][HEAD_REC_MAX];  // K record | V record (either widths)
  alignas(16) float ka[2][T], kb[2][T];  // aK, bK per token (per K~ stage)
  alignas(16) float va[2][T], vb[2][T];  // aV, bV per token
  alignas(16) float xmax[2][2][MQ_ROWS];  // tile maximum of each row half (exchanged between halves)
  alignas(16) float xl[2][MQ_ROWS];       // row sums of the two halves at the end
  float qsi[MQ_ROWS];                     // 1 / qs of each row
  uint64_t rec_full[REC_STAGES], rec_empty[REC_STAGES], kt_full[2], qk_done[2], p_full[2], xbar[2];
  uint64_t s_full[2], vt_full, pv_done, fin, lbar;
  uint32_t tmem;
  uint32_t vmask;  // bit k: block id of tile k of this chunk is in range
};
struct MQTailSmem {
  float k[T][D];
  float v[T][D];
};
static_assert(sizeof(MQTailSmem) <= sizeof(MQSmem), "tail buffers fit the packed layout");

template <typename E>
__device__ __forceinline__ float tof(E x) {
  if constexpr (std::is_same<E, __half>::value) return __half2float(x);
  else return __bfloat162float(x);
}
// Two 16-bit values of E (low half first) -> exact floats.
template <typename E>
__device__ __forceinline__ float2 pair_to_float2(uint32_t u) {
  if constexpr (std::is_same<E, __half>::value) return __half22float2(*reinterpret_cast<__half2*>(&u));
  else return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t x) { return *reinterpret_cast<__half2*>(&x); }
__device__ __forceinline__ uint32_t b2u(__nv_bfloat162 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __nv_bfloat162 u2b(uint32_t x) { return *reinterpret_cast<__nv_bfloat162*>(&x); }

// Byte offset of element (row r, k) of a K-major operand made of 8-row x
// 16-byte core matrices, `kb` core matrices per row group along K.
__host__ __device__ constexpr int cm_off(int r, int k, int kb) {
  return ((r >> 3) * kb + (k >> 3)) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

// Channel held by contraction slot k of the QK operands.  A key word of
// 4-bit codes yields channel pairs (c, c + 4) per masked field, a word of
// 2-bit codes pairs (c, c + 8), and a pair fills two adjacent slots.
template <int KBITS>
__host__ __device__ constexpr int perm_k(int k) {
  if constexpr (KBITS == 4) {
    const int j = k & 7;
    return (k & ~7) + (j >> 1) + 4 * (j & 1);
  } else {
    const int j = k & 15;
    return (k & ~15) + (j >> 1) + 8 * (j & 1);
  }
}

// (x & mask) | magic as one three-input logic op, then y * m + a (one
// rounding; exact whenever the result is representable).
__device__ __forceinline__ uint32_t lop_magic(uint32_t x, uint32_t mask, uint32_t magic) {
  uint32_t y;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(y) : "r"(x), "r"(mask), "r"(magic));
  return y;
}
__device__ __forceinline__ uint32_t fma_h(uint32_t y, __half2 m, __half2 a) { return h2u(__hfma2(u2h(y), m, a)); }
__device__ __forceinline__ uint32_t fma_b(uint32_t y, __nv_bfloat162 m, __nv_bfloat162 a) {
  return b2u(__hfma2(u2b(y), m, a));
}

__device__ __forceinline__ float* mq_part(const MQParams& p, int b, int h, int rb, int chunk, int r) {
  return p.ws + (((((int64_t)b * p.num_kv_heads + h) * p.n_rowblocks + rb) * (p.n_chunks + 1) + chunk) * MQ_ROWS + r) *
                    MQ_PART;
}

// Rows of row block rb, the last position any of them sees, and the number
// of closed tiles the block reads.
__device__ __forceinline__ void mq_block_extent(const MQParams& p, int rb, int len, int& rows, int& n_need) {
  rows = min(MQ_ROWS, p.n_queries * p.G - rb * MQ_ROWS);
  const int pos_hi = len - p.n_queries + (rb * MQ_ROWS + rows - 1) / p.G;
  n_need = min(len / T, pos_hi / T + 1);
}

// Warp-uniform bounded wait: every lane waits, all report failure together.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, int32_t* err) {
  const bool ok = mbar_wait_parked(bar, parity, err);
  return __all_sync(0xffffffffu, ok);
}

// ---- producers: K~ rows of 8 tokens x 16 channels per thread
// Thread pth takes channels 16 cg .. 16 cg + 15 of tokens 8 (tq + 2 i) + tl,
// i = 0..7, so the 8 lanes of a store phase write 8 rows of one core matrix.
__device__ __forceinline__ int k_token(int pth, int i) { return 8 * ((pth >> 6) + 2 * i) + (pth & 7); }

template <int KBITS>
__device__ __forceinline__ void unpack_k(const unsigned char* kr, unsigned char* kt, int pth) {
  const int cg = (pth >> 3) & 7;
  const uint4 g16 = *reinterpret_cast<const uint4*>(kr + 16 * cg);
  const uint32_t gw[4] = {g16.x, g16.y, g16.z, g16.w};
  auto gval = [&](int c) { return e4m3_to_float((uint8_t)(gw[c >> 2] >> (8 * (c & 3)))); };
  if constexpr (KBITS == 4) {
    // word w (channels 8w' .. 8w'+7 of this group) -> pairs (0,4),(1,5) at bits 0 / 4, (2,6),(3,7) after >> 8
    __half2 mul[2][4], add[2][4];
#pragma unroll
    for (int w = 0; w < 2; ++w)
#pragma unroll
      for (int f = 0; f < 4; ++f) {
        const int c0 = 8 * w + f, c1 = c0 + 4;
        const float sh = (f & 1) ? 1.f / 1024.f : 1.f / 64.f;   // field at bit 4 (f odd) or bit 0
        const float ad = (f & 1) ? -1.f : -16.f;
        mul[w][f] = __floats2half2_rn(gval(c0) * sh, gval(c1) * sh);
        add[w][f] = __floats2half2_rn(gval(c0) * ad, gval(c1) * ad);
      }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = k_token(pth, i);
      const uint2 cw = *reinterpret_cast<const uint2*>(kr + 512 + 64 * t + 8 * cg);
      const uint32_t wv[2] = {cw.x, cw.y};
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const uint32_t x = wv[w], x8 = x >> 8;
        uint4 o;
        o.x = fma_h(lop_magic(x, 0x000F000Fu, MAGIC_F16), mul[w][0], add[w][0]);
        o.y = fma_h(lop_magic(x, 0x00F000F0u, MAGIC_F16), mul[w][1], add[w][1]);
        o.z = fma_h(lop_magic(x8, 0x000F000Fu, MAGIC_F16), mul[w][2], add[w][2]);
        o.w = fma_h(lop_magic(x8, 0x00F000F0u, MAGIC_F16), mul[w][3], add[w][3]);
        *reinterpret_cast<uint4*>(kt + cm_off(t, 16 * cg + 8 * w, 16)) = o;
      }
    }
  } else {
    // one word per token: channel pairs (j, j+8) at crumb j (j < 4) or, after >> 8, crumb j - 4
    __half2 mul[8], add[8];
#pragma unroll
    for (int f = 0; f < 8; ++f) {
      const int c0 = f, c1 = f + 8;
      const int pos = 2 * (f & 3);  // bit position of the field
      const float sh = 1.f / (64.f * (float)(1 << pos)), ad = -16.f / (float)(1 << pos);
      mul[f] = __floats2half2_rn(gval(c0) * sh, gval(c1) * sh);
      add[f] = __floats2half2_rn(gval(c0) * ad, gval(c1) * ad);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = k_token(pth, i);
      const uint32_t x = *reinterpret_cast<const uint32_t*>(kr + 512 + 32 * t + 4 * cg), x8 = x >> 8;
      uint32_t o[8];
#pragma unroll
      for (int f = 0; f < 8; ++f)
        o[f] = fma_h(lop_magic(f < 4 ? x : x8, 0x00030003u << (2 * (f & 3)), MAGIC_F16), mul[f], add[f]);
      *reinterpret_cast<uint4*>(kt + cm_off(t, 16 * cg, 16)) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(kt + cm_off(t, 16 * cg + 8, 16)) = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
}

// ---- producers: zero operands for a tile whose block id is out of range
// (its record buffer holds no data; the rows mask every token of it)
__device__ __forceinline__ void zero_k(unsigned char* kt, int pth) {
  const int cg = (pth >> 3) & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    *reinterpret_cast<uint4*>(kt + cm_off(k_token(pth, i), 16 * cg, 16)) = make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(kt + cm_off(k_token(pth, i), 16 * cg + 8, 16)) = make_uint4(0u, 0u, 0u, 0u);
  }
}
__device__ __forceinline__ void zero_v(unsigned char* vt, int c) {
#pragma unroll
  for (int k8 = 0; k8 < 17; ++k8) *reinterpret_cast<uint4*>(vt + cm_off(c, 8 * k8, VT_K / 8)) = make_uint4(0u, 0u, 0u, 0u);
}

// ---- producers: V~ row of channel c (128 tokens) plus its gV entries
template <int VBITS>
__device__ __forceinline__ void unpack_v(const unsigned char* vr, unsigned char* vt, int c) {
  if constexpr (VBITS == 4) {
    // 16 words of 8 tokens; token pair (2s, 2s + 1) of word w at bits 4s, 16 + 4s:
    // shifted to bits 0 and 16, each field reads 128 + code in bf16
    const float gv = e4m3_to_float(vr[c]);
    const __nv_bfloat162 m0 = __float2bfloat162_rn(gv), a0 = __float2bfloat162_rn(-128.f * gv);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 c4 = *reinterpret_cast<const uint4*>(vr + 512 + 64 * c + 16 * q);
      const uint32_t wv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t x = wv[e];
        uint32_t o[4];
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2) o[s2] = fma_b(lop_magic(x >> (4 * s2), 0x000F000Fu, MAGIC_BF16), m0, a0);
        *reinterpret_cast<uint4*>(vt + cm_off(c, 8 * (4 * q + e), VT_K / 8)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    const uint32_t g2 = b2u(m0);  // k 128..131: beta hi, lo of the two row halves
    *reinterpret_cast<uint4*>(vt + cm_off(c, 128, VT_K / 8)) = make_uint4(g2, g2, 0u, 0u);
    return;
  }
  // a field at bit q reads 128 + 2^q code: times gV / 2^q, minus 128 gV / 2^q
  const float gv = e4m3_to_float(vr[c]);
  const __nv_bfloat162 m0 = __float2bfloat162_rn(gv), m2 = __float2bfloat162_rn(gv * 0.25f),
                       m4 = __float2bfloat162_rn(gv * 0.0625f);
  const __nv_bfloat162 a0 = __float2bfloat162_rn(-128.f * gv), a2 = __float2bfloat162_rn(-32.f * gv),
                       a4 = __float2bfloat162_rn(-8.f * gv);
  const uint4 c0 = *reinterpret_cast<const uint4*>(vr + 512 + 32 * c);
  const uint4 c1 = *reinterpret_cast<const uint4*>(vr + 512 + 32 * c + 16);
  const uint32_t wv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    // tokens 16w + (2s, 2s+1) sit at bits 2s of the low / high half-word
    const uint32_t x = wv[w], y = x >> 6, z = x >> 12;
    uint32_t o[8];
    o[0] = fma_b(lop_magic(x, 0x00030003u, MAGIC_BF16), m0, a0);
    o[1] = fma_b(lop_magic(x, 0x000C000Cu, MAGIC_BF16), m2, a2);
    o[2] = fma_b(lop_magic(x, 0x00300030u, MAGIC_BF16), m4, a4);
    o[3] = fma_b(lop_magic(y, 0x00030003u, MAGIC_BF16), m0, a0);
    o[4] = fma_b(lop_magic(y, 0x000C000Cu, MAGIC_BF16), m2, a2);
    o[5] = fma_b(lop_magic(y, 0x00300030u, MAGIC_BF16), m4, a4);
    o[6] = fma_b(lop_magic(z, 0x00030003u, MAGIC_BF16), m0, a0);
    o[7] = fma_b(lop_magic(z, 0x000C000Cu, MAGIC_BF16), m2, a2);
    *reinterpret_cast<uint4*>(vt + cm_off(c, 16 * w, VT_K / 8)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(vt + cm_off(c, 16 * w + 8, VT_K / 8)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
  const uint32_t g2 = b2u(m0);  // k 128..131: beta hi, lo of the two row halves
  *reinterpret_cast<uint4*>(vt + cm_off(c, 128, VT_K / 8)) = make_uint4(g2, g2, 0u, 0u);
}

// Raw open tile: rows of this row block against its len % 128 tokens, fp32
// on the CUDA cores; two threads per row (64 channels each).
template <typename E>
__device__ void mq_tail(const MQParams& p, int b, int h, int rb, int len, unsigned char* smem) {
  const int n = len % T;
  if (n == 0) return;
  MQTailSmem& sm = *reinterpret_cast<MQTailSmem*>(smem);
  const int tid = threadIdx.x;
  const E* kt = static_cast<const E*>(p.tail) + (((int64_t)b * p.num_kv_heads + h) * 2 + 0) * (T * D);
  const E* vt = kt + T * D;
  for (int i = tid; i < n * D; i += blockDim.x) {
    sm.k[i / D][i % D] = tof(kt[i]);
    sm.v[i / D][i % D] = tof(vt[i]);
  }
  __syncthreads();
  if (tid >= 2 * MQ_ROWS) return;
  const int r = tid >> 1, half = tid & 1;
  int rows, n_need;
  mq_block_extent(p, rb, len, rows, n_need);
  const int R = rb * MQ_ROWS + r;
  const bool rv = r < rows;
  const int qi = rv ? R / p.G : 0, gq = rv ? R % p.G : 0;
  const int pos = rv ? len - p.n_queries + qi : -1;
  const int t0 = len - n;  // position of slot 0
  const int nv = min(n, pos - t0 + 1);  // tail tokens this row sees (may be <= 0)
  // the query half row stays in its 16-bit pairs (exact); scale after the dot product
  uint32_t q2[32];
  float acc[64];
  {
    const uint4* qr = reinterpret_cast<const uint4*>(
        static_cast<const E*>(p.q) +
        (((int64_t)b * p.n_queries + qi) * p.num_q_heads + (int64_t)h * p.G + gq) * D + 64 * half);
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      const uint4 v = rv ? qr[c8] : make_uint4(0u, 0u, 0u, 0u);
      q2[4 * c8] = v.x; q2[4 * c8 + 1] = v.y; q2[4 * c8 + 2] = v.z; q2[4 * c8 + 3] = v.w;
    }
#pragma unroll
    for (int c = 0; c < 64; ++c) acc[c] = 0.f;
  }
  const float fscale = p.scale * MQ_LOG2E;
  float m = -INFINITY, l = 0.f;
  for (int tb = 0; tb < n; tb += 8) {
    float s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = min(tb + i, T - 1);
      float a = 0.f;
      const float4* kk = reinterpret_cast<const float4*>(&sm.k[t][64 * half]);
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 kv = kk[c4];
        const float2 q01 = pair_to_float2<E>(q2[2 * c4]), q23 = pair_to_float2<E>(q2[2 * c4 + 1]);
        a = fmaf(q01.x, kv.x, a);
        a = fmaf(q01.y, kv.y, a);
        a = fmaf(q23.x, kv.z, a);
        a = fmaf(q23.y, kv.w, a);
      }
      a += __shfl_xor_sync(0xffffffffu, a, 1);
      s[i] = (tb + i < nv) ? a * fscale : -INFINITY;
    }
    float bm = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) bm = fmaxf(bm, s[i]);
    if (bm == -INFINITY) continue;
    if (bm > m) {
      const float corr = (m == -INFINITY) ? 0.f : exp2f(m - bm);
      l *= corr;
#pragma unroll
      for (int c = 0; c < 64; ++c) acc[c] *= corr;
      m = bm;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float pr = exp2f(s[i] - m);
      l += pr;
      if (pr != 0.f) {
        const float4* vv = reinterpret_cast<const float4*>(&sm.v[min(tb + i, T - 1)][64 * half]);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 v4 = vv[c4];
          acc[4 * c4] = fmaf(pr, v4.x, acc[4 * c4]);
          acc[4 * c4 + 1] = fmaf(pr, v4.y, acc[4 * c4 + 1]);
          acc[4 * c4 + 2] = fmaf(pr, v4.z, acc[4 * c4 + 2]);
          acc[4 * c4 + 3] = fmaf(pr, v4.w, acc[4 * c4 + 3]);
        }
      }
    }
  }
  if (!rv) return;
  float* o = mq_part(p, b, h, rb, p.n_chunks, r);
  if (!kcheck(o, MQ_PART * sizeof(float), p.ws, (size_t)p.ws_bytes, p.err)) return;
  if (half == 0) { o[0] = m; o[1] = l; }
#pragma unroll
  for (int c4 = 0; c4 < 16; ++c4)
    *reinterpret_cast<float4*>(o + MQ_PACC + 64 * half + 4 * c4) =
        make_float4(acc[4 * c4], acc[4 * c4 + 1], acc[4 * c4 + 2], acc[4 * c4 + 3]);
}

// grid (n_chunks + 1, num_kv_heads * n_rowblocks, batch) x 416 threads;
// chunk n_chunks handles the raw open tile.
template <typename E, int KBITS, int VBITS>
__global__ void __launch_bounds__(MQ_THREADS, 1) mq_kernel(MQParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  allow_dependents();  // the combine may be scheduled once every CTA has started
  const int chunk = blockIdx.x, h = blockIdx.y / p.n_rowblocks, rb = blockIdx.y % p.n_rowblocks, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int len = p.seq_lens[b];
  if (len < p.n_queries || len > T * p.max_blocks) {
    if (tid == 0 && chunk == 0 && blockIdx.y == 0) set_error(p.err, KVARN_DEV_ERR_TOKEN_RANGE);
    return;
  }
  const uint32_t sbase = smem_u32(smem_raw);
  unsigned char* base = smem_raw + (((sbase + 127u) & ~127u) - sbase);
  if (chunk == p.n_chunks) {
    mq_tail<E>(p, b, h, rb, len, base);
    return;
  }
  int rows, n_need;
  mq_block_extent(p, rb, len, rows, n_need);
  const int first = chunk * p.chunk_tiles;
  const int n_tiles = min(p.chunk_tiles, n_need - first);
  if (n_tiles <= 0) return;
  constexpr int KREC = rec_bytes(KBITS), VREC = rec_bytes(VBITS);
  MQSmem& sm = *reinterpret_cast<MQSmem*>(base);
  const int32_t* tab = p.block_table + (int64_t)b * p.max_blocks + first;

  if (warp == 12) tmem_alloc(&sm.tmem, TM_COLS);
  if (tid == 0) {
    for (int s = 0; s < REC_STAGES; ++s) {
      mbar_init(&sm.rec_full[s], 1);
      mbar_init(&sm.rec_empty[s], 128);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.kt_full[s], 128);
      mbar_init(&sm.qk_done[s], 1);
      mbar_init(&sm.p_full[s], 256);
      mbar_init(&sm.xbar[s], 256);
    }
    mbar_init(&sm.s_full[0], 1);
    mbar_init(&sm.s_full[1], 1);
    mbar_init(&sm.vt_full, 128);
    mbar_init(&sm.pv_done, 1);
    mbar_init(&sm.fin, 1);
    mbar_init(&sm.lbar, 256);
    fence_mbar_init();
    uint32_t vm = 0;
    for (int k = 0; k < n_tiles; ++k) vm |= (tab[k] >= 0 && tab[k] < p.num_blocks) ? (1u << k) : 0u;
    sm.vmask = vm;
  }

  // ---- prologue: query operand (warps 0-3, a thread per row), constant
  // operand regions (producers)
  const int q4 = warp & 3, half = (warp >> 2) & 1;  // softmax warps: row quarter, token half
  const int r = 32 * q4 + lane;
  const int R = rb * MQ_ROWS + r;
  const bool rv = warp < 8 && r < rows;
  const int qi = rv ? R / p.G : 0;
  if (warp < 8) {
    // warp w rotates rows 16 w .. 16 w + 15, 4 channels per lane: x = q H
    // (4-point butterflies in registers, then across lanes), 8 rows at a
    // time staged in shared memory (the second K~ buffer, free until the
    // main loop), then written as fp16 hi / lo core-matrix rows so that the
    // 8 lanes of a store phase write 8 different rows
    float* stage = reinterpret_cast<float*>(sm.kt[1]) + warp * (8 * 132);  // 8 rows of 132 floats per warp
    for (int rg = 0; rg < 2; ++rg) {
      for (int rr = 0; rr < 8; ++rr) {
        const int row = 16 * warp + 8 * rg + rr, Rr = rb * MQ_ROWS + row;
        const bool ok = row < rows;
        const int qr_i = ok ? Rr / p.G : 0, qr_g = ok ? Rr % p.G : 0;
        const E* qr = static_cast<const E*>(p.q) +
                      (((int64_t)b * p.n_queries + qr_i) * p.num_q_heads + (int64_t)h * p.G + qr_g) * D + 4 * lane;
        float x[4];
        {
          const uint2 v = ok ? *reinterpret_cast<const uint2*>(qr) : make_uint2(0u, 0u);
          const E* e = reinterpret_cast<const E*>(&v);
#pragma unroll
          for (int i = 0; i < 4; ++i) x[i] = tof(e[i]);
        }
        float u = x[0], v = x[1];
        x[0] = u + v; x[1] = u - v;
        u = x[2]; v = x[3];
        x[2] = u + v; x[3] = u - v;
        u = x[0]; v = x[2];
        x[0] = u + v; x[2] = u - v;
        u = x[1]; v = x[3];
        x[1] = u + v; x[3] = u - v;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
          const bool upper = (lane & m) != 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, x[i], m);
            x[i] = upper ? (o - x[i]) : (x[i] + o);
          }
        }
        const float f = p.scale * MQ_LOG2E * INV_SQRT_D;
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          x[i] *= f;
          amax = fmaxf(amax, fabsf(x[i]));
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
        int ex = 0;
        if (amax > 0.f) frexpf(amax, &ex);
        const float qs = ldexpf(1.f, 7 - ex);  // max |Q'| in [64, 128)
        if (lane == 0) sm.qsi[row] = ldexpf(1.f, ex - 7);
        *reinterpret_cast<float4*>(stage + rr * 132 + 4 * lane) = make_float4(x[0] * qs, x[1] * qs, x[2] * qs, x[3] * qs);
      }
      __syncwarp();
      // lane: row rr = lane & 7, core-matrix columns g = (lane >> 3) + 4 j
      const int rr = lane & 7, row = 16 * warp + 8 * rg + rr;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int g = (lane >> 3) + 4 * j;
        // slot pairs (2i, 2i + 1) hold channels (ca + i, cb + i): K4 (8g, 8g + 4), K2 (16 (g/2) + 4 (g&1), + 8)
        const int ca = (KBITS == 4) ? 8 * g : 16 * (g >> 1) + 4 * (g & 1), cb = ca + ((KBITS == 4) ? 4 : 8);
        const float4 va = *reinterpret_cast<const float4*>(stage + rr * 132 + ca);
        const float4 vb = *reinterpret_cast<const float4*>(stage + rr * 132 + cb);
        const float av[4] = {va.x, va.y, va.z, va.w}, bv[4] = {vb.x, vb.y, vb.z, vb.w};
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half2 hi = __floats2half2_rn(av[i], bv[i]);
          const float2 hf = __half22float2(hi);
          hw[i] = h2u(hi);
          lw[i] = h2u(__floats2half2_rn(av[i] - hf.x, bv[i] - hf.y));
        }
        // hi: staged in the V~ buffer (free until the main loop), lo: the shared-memory operand
        *reinterpret_cast<uint4*>(sm.vt + cm_off(row, 8 * g, 16)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(sm.qa_lo + cm_off(row, 8 * g, 16)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      __syncwarp();
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  const uint32_t vmask = sm.vmask;
  if (warp < 4) {  // Q' hi of row r -> tensor-memory lane r, columns TM_QA .. +63 (the A operand layout)
    const uint32_t lb = tmem + ((uint32_t)(warp * 32) << 16) + TM_QA;
    const int row = tid;
#pragma unroll
    for (int c = 0; c < 64; c += 16) {
      uint32_t w16[16];
#pragma unroll
      for (int g2 = 0; g2 < 4; ++g2) {
        const uint4 v4 = *reinterpret_cast<const uint4*>(sm.vt + cm_off(row, 2 * c + 8 * g2, 16));
        w16[4 * g2] = v4.x; w16[4 * g2 + 1] = v4.y; w16[4 * g2 + 2] = v4.z; w16[4 * g2 + 3] = v4.w;
      }
      tmem_st16(lb + c, w16);
    }
    tmem_wait_st();
  } else if (warp >= 8 && warp < 12) {
    const int pth = tid - 256;
    for (int i = pth; i < 2 * 15 * 16; i += 128) {  // K~ rows 129..143 of both stages
      const int s = i / (15 * 16), rr = 129 + (i / 16) % 15, kg = i % 16;
      *reinterpret_cast<uint4*>(sm.kt[s] + cm_off(rr, 8 * kg, 16)) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // one bulk copy of the K and V records of tile k into its stage (one thread)
  auto issue_rec = [&](int k) {
    const int s = k % REC_STAGES;
    const unsigned char* src = p.pool + tab[k] * p.block_bytes + (int64_t)h * (KREC + VREC);
    if (((vmask >> k) & 1u) && kcheck(src, KREC + VREC, p.pool, (size_t)p.num_blocks * p.block_bytes, p.err)) {
      mbar_expect_tx(&sm.rec_full[s], KREC + VREC);
      bulk_g2s(sm.rec[s], src, KREC + VREC, &sm.rec_full[s]);
    } else {
      set_error(p.err, KVARN_DEV_ERR_BLOCK_RANGE);
      mbar_arrive(&sm.rec_full[s]);
    }
  };
  if (warp == 12) {
    // ------------------------------------------------------------ MMA issue (one thread)
    if (lane == 0) {
      const uint64_t qa_lo = umma_desc(smem_u32(sm.qa_lo), 128, 2048);
      auto issue_qk = [&](int k) {  // S[k & 1] = Q' K~^T over the hi then the lo query halves
        const uint32_t kb = smem_u32(sm.kt[k & 1]), d = tmem + TM_S + TM_SSTRIDE * (k & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(d, tmem + TM_QA + 8 * kk, umma_desc(kb + 256 * kk, 128, 2048), IDESC_QK, kk > 0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(d, qa_lo + (uint64_t)(16 * kk), umma_desc(kb + 256 * kk, 128, 2048), IDESC_QK, 1);
        umma_commit(&sm.qk_done[k & 1]);
        umma_commit(&sm.s_full[k & 1]);
      };
      auto issue_pv = [&](int k) {  // D_O += P~ V~^T over the hi (with beta) then the lo halves
        const uint32_t vb = smem_u32(sm.vt), pa = tmem + TM_S + TM_SSTRIDE * (k & 1);
#pragma unroll
        for (int kk = 0; kk < 9; ++kk)  // hi parts of tokens 16 kk .. 16 kk + 15, then the beta block
          umma_ts(tmem + TM_O, pa + 16 * kk, umma_desc(vb + 256 * kk, 128, VT_K * 16), IDESC_PV,
                  (k > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // lo parts
          umma_ts(tmem + TM_O, pa + 16 * kk + 8, umma_desc(vb + 256 * kk, 128, VT_K * 16), IDESC_PV, 1);
        umma_commit(&sm.pv_done);
      };
      bool ok = true;
      for (int k = 0; k < min(n_tiles, REC_STAGES); ++k) issue_rec(k);
      for (int k = 0; ok && k < min(n_tiles, 2); ++k) {  // both score buffers start free
        ok = mbar_wait_parked(&sm.kt_full[k], 0, p.err);
        if (!ok) break;
        tc_fence_after();
        issue_qk(k);
      }
      for (int k = 0; ok && k < n_tiles; ++k) {
        ok = mbar_wait_parked(&sm.p_full[k & 1], (k >> 1) & 1, p.err) && mbar_wait_parked(&sm.vt_full, k & 1, p.err);
        if (!ok) break;
        tc_fence_after();
        issue_pv(k);
        if (k + 2 < n_tiles) {  // buffer k & 1 is free once PV(k) has read its P~
          ok = mbar_wait_parked(&sm.kt_full[k & 1], ((k + 2) >> 1) & 1, p.err) &&
               mbar_wait_parked(&sm.pv_done, k & 1, p.err);
          if (!ok) break;
          tc_fence_after();
          issue_qk(k + 2);
        }
      }
      // every MMA this thread issued has finished before the memory is released
      umma_commit(&sm.fin);
      mbar_wait_parked(&sm.fin, 0, p.err);
    }
    __syncwarp();
  } else if (warp >= 8) {
    // ------------------------------------------------------------ producers
    const int pth = tid - 256;
    // V~ columns 136..143 stay zero (the buffer held the query staging until the last barrier)
    *reinterpret_cast<uint4*>(sm.vt + cm_off(pth, 136, VT_K / 8)) = make_uint4(0u, 0u, 0u, 0u);
    bool ok = true;
    for (int k = -1; k < n_tiles; ++k) {
      const int j = k + 1;  // K~ of the next tile first, then V~ of this one
      if (j < n_tiles) {
        const int s = j % REC_STAGES;
        ok = wait_all(&sm.rec_full[s], (j / REC_STAGES) & 1, p.err);
        if (ok && j >= 2)
          ok = wait_all(&sm.qk_done[j & 1], ((j - 2) >> 1) & 1, p.err) &&
               wait_all(&sm.p_full[j & 1], ((j - 2) >> 1) & 1, p.err);
        if (!ok) break;
        const unsigned char* kr = sm.rec[s];
        const unsigned char* vr = kr + KREC;
        if ((vmask >> j) & 1u) {
          sm.ka[j & 1][pth] = e4m3_to_float(kr[128 + pth]);
          sm.kb[j & 1][pth] = __half2float(*reinterpret_cast<const __half*>(kr + 256 + 2 * pth));
          sm.va[j & 1][pth] = e4m3_to_float(vr[128 + pth]);
          sm.vb[j & 1][pth] = __half2float(*reinterpret_cast<const __half*>(vr + 256 + 2 * pth));
          unpack_k<KBITS>(kr, sm.kt[j & 1], pth);
          if (pth < 16) {  // the g row: K~[128][k] = gK of the slot's channel / 64
            uint32_t o[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
              o[jj] = h2u(__floats2half2_rn(e4m3_to_float(kr[perm_k<KBITS>(8 * pth + 2 * jj)]) * (1.f / 64.f),
                                            e4m3_to_float(kr[perm_k<KBITS>(8 * pth + 2 * jj + 1)]) * (1.f / 64.f)));
            *reinterpret_cast<uint4*>(sm.kt[j & 1] + cm_off(128, 8 * pth, 16)) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        } else {
          sm.ka[j & 1][pth] = sm.kb[j & 1][pth] = sm.va[j & 1][pth] = sm.vb[j & 1][pth] = 0.f;
          zero_k(sm.kt[j & 1], pth);
          if (pth < 16)
            *reinterpret_cast<uint4*>(sm.kt[j & 1] + cm_off(128, 8 * pth, 16)) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async();
        mbar_arrive(&sm.kt_full[j & 1]);
      }
      if (k >= 0) {
        if (k >= 1) ok = wait_all(&sm.pv_done, (k - 1) & 1, p.err);
        if (!ok) break;
        if ((vmask >> k) & 1u) unpack_v<VBITS>(sm.rec[k % REC_STAGES] + KREC, sm.vt, pth);
        else zero_v(sm.vt, pth);
        fence_proxy_async();
        mbar_arrive(&sm.vt_full);
        mbar_arrive(&sm.rec_empty[k % REC_STAGES]);
        if (pth == 0 && k + REC_STAGES < n_tiles) {  // every producer is done with this stage: refill it
          if (mbar_wait_parked(&sm.rec_empty[k % REC_STAGES], (k / REC_STAGES) & 1, p.err)) issue_rec(k + REC_STAGES);
        }
      }
    }
    // copies still in flight (an early exit) land before the CTA ends
    if (!ok && pth == 0) {
      for (int k = 0; k < n_tiles; ++k) mbar_wait_parked(&sm.rec_full[k % REC_STAGES], (k / REC_STAGES) & 1, p.err);
    }
  } else {
    // ------------------------------------------------------------ softmax: row r, tokens 64 half .. +63
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    const int pos = rv ? len - p.n_queries + qi : -1;
    const float cr = 64.f * sm.qsi[r];  // score (log2) = cr (aK D_t + bK D_128)
    const float2 cr2 = make_float2(cr, cr);
    float m_ref = -INFINITY, l_sum = 0.f;
    bool dead = false;
    for (int k = 0; k < n_tiles; ++k) {
      const int s = k & 1;
      const uint32_t sb = lane_base + TM_S + TM_SSTRIDE * s;  // this tile's score / P~ buffer
      if (!wait_all(&sm.s_full[s], (k >> 1) & 1, p.err)) { dead = true; break; }
      tc_fence_after();
      // pass 1: scores s = aK D_t + bK D_128 (units of 1 / cr) of this half's 64
      // tokens, written back in place, and their maximum; masked tokens -> -inf
      float d128;
      {
        uint32_t d1;
        tmem_ld1(sb + 128, d1);
        tmem_wait_ld();
        d128 = __uint_as_float(d1);
      }
      // the scales of this tile (written with its K~; that phase is complete)
      if (!wait_all(&sm.kt_full[s], (k >> 1) & 1, p.err)) { dead = true; break; }
      const int t0 = (first + k) * T + 64 * half;
      const int nvis = ((vmask >> k) & 1u) ? min(64, pos - t0 + 1) : 0;  // tokens of this half the row sees
      const float2 d2 = make_float2(d128, d128);
      float tmax = -INFINITY;
      // the causal mask, in a second copy of the loop that only a tile with
      // hidden tokens takes (padded rows are never written, so they may skip it)
      auto pass1 = [&](auto mask_c) {
        constexpr bool MASK = decltype(mask_c)::value;
#pragma unroll 1
        for (int c = 0; c < 64; c += 16) {
          uint32_t d[16];
          tmem_ld16(sb + 64 * half + c, d);
          const float4* ka4 = reinterpret_cast<const float4*>(sm.ka[s] + 64 * half + c);
          const float4* kb4 = reinterpret_cast<const float4*>(sm.kb[s] + 64 * half + c);
          float4 a4[4], b4[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) { a4[j] = ka4[j]; b4[j] = kb4[j]; }
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float2 s01 = ffma2(make_float2(a4[j].x, a4[j].y),
                               make_float2(__uint_as_float(d[4 * j]), __uint_as_float(d[4 * j + 1])),
                               fmul2(make_float2(b4[j].x, b4[j].y), d2));
            float2 s23 = ffma2(make_float2(a4[j].z, a4[j].w),
                               make_float2(__uint_as_float(d[4 * j + 2]), __uint_as_float(d[4 * j + 3])),
                               fmul2(make_float2(b4[j].z, b4[j].w), d2));
            const int t = c + 4 * j;
            if (MASK && nvis < 64) {
              if (t >= nvis) s01.x = -INFINITY;
              if (t + 1 >= nvis) s01.y = -INFINITY;
              if (t + 2 >= nvis) s23.x = -INFINITY;
              if (t + 3 >= nvis) s23.y = -INFINITY;
            }
            tmax = fmaxf(tmax, fmaxf(fmaxf(s01.x, s01.y), fmaxf(s23.x, s23.y)));
            d[4 * j] = __float_as_uint(s01.x); d[4 * j + 1] = __float_as_uint(s01.y);
            d[4 * j + 2] = __float_as_uint(s23.x); d[4 * j + 3] = __float_as_uint(s23.y);
          }
          tmem_st16(sb + 64 * half + c, d);
        }
      };
      if (__all_sync(0xffffffffu, !rv || nvis >= 64)) pass1(std::false_type{});
      else pass1(std::true_type{});
      tmem_wait_st();
      tc_fence_before();  // both halves read D_128 before either writes beta (ordered by xbar)
      // the row maximum: exchange with the other half through shared memory
      sm.xmax[k & 1][half][r] = tmax;
      mbar_arrive(&sm.xbar[k & 1]);
      if (!wait_all(&sm.xbar[k & 1], (k >> 1) & 1, p.err)) { dead = true; break; }
      tc_fence_after();
      tmax = fmaxf(tmax, sm.xmax[k & 1][half ^ 1][r]) * cr;
      float corr = 1.f;
      bool resc = false;
      if (tmax > m_ref + MQ_TAU) {
        if (m_ref != -INFINITY) {
          corr = ex2_ftz(m_ref - tmax);
          resc = true;
        }
        m_ref = tmax;
        l_sum *= corr;
      }
      const bool live = m_ref != -INFINITY;
      if (__any_sync(0xffffffffu, resc)) {  // rescale the accumulator once the previous PV is done
        if (k > 0 && !wait_all(&sm.pv_done, (k - 1) & 1, p.err)) { dead = true; break; }
        tc_fence_after();
        uint32_t d[16];
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
          tmem_ld16(lane_base + TM_O + 64 * half + c, d);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) d[i] = __float_as_uint(__uint_as_float(d[i]) * corr);
          tmem_st16(lane_base + TM_O + 64 * half + c, d);
        }
      }
      // pass 2: P~ = p aV (bf16 hi, lo) over the scores of each 16-token group,
      // l += sum p, beta += sum p bV
      const float2 nm2 = make_float2(-m_ref, -m_ref);
      float2 lt = make_float2(0.f, 0.f), bt = make_float2(0.f, 0.f);
      // a row that has seen no token yet (reference still -inf) gets p = 0, in
      // a second copy of the loop that only such tiles take
      auto pass2 = [&](auto zero_c) {
        constexpr bool ZERO = decltype(zero_c)::value;
#pragma unroll 1
        for (int c = 0; c < 64; c += 16) {
          uint32_t d[16];
          tmem_ld16(sb + 64 * half + c, d);
          const float4* va4 = reinterpret_cast<const float4*>(sm.va[s] + 64 * half + c);
          const float4* vb4 = reinterpret_cast<const float4*>(sm.vb[s] + 64 * half + c);
          float4 a4[4], b4[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) { a4[j] = va4[j]; b4[j] = vb4[j]; }
          tmem_wait_ld();
          uint32_t pw[16];  // hi words 0..7, lo words 8..15
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 e01 = ffma2(cr2, make_float2(__uint_as_float(d[4 * j]), __uint_as_float(d[4 * j + 1])), nm2);
            const float2 e23 = ffma2(cr2, make_float2(__uint_as_float(d[4 * j + 2]), __uint_as_float(d[4 * j + 3])), nm2);
            float2 p01 = make_float2(ex2_ftz(e01.x), ex2_ftz(e01.y)), p23 = make_float2(ex2_ftz(e23.x), ex2_ftz(e23.y));
            if (ZERO && !live) p01 = p23 = make_float2(0.f, 0.f);
            lt = fadd2(lt, fadd2(p01, p23));
            bt = ffma2(p01, make_float2(b4[j].x, b4[j].y), ffma2(p23, make_float2(b4[j].z, b4[j].w), bt));
            const float2 x01 = fmul2(p01, make_float2(a4[j].x, a4[j].y)), x23 = fmul2(p23, make_float2(a4[j].z, a4[j].w));
            const __nv_bfloat162 h01 = __floats2bfloat162_rn(x01.x, x01.y), h23 = __floats2bfloat162_rn(x23.x, x23.y);
            const float2 r01 = ffma2(__bfloat1622float2(h01), make_float2(-1.f, -1.f), x01);  // x - hi, exact product
            const float2 r23 = ffma2(__bfloat1622float2(h23), make_float2(-1.f, -1.f), x23);
            pw[2 * j] = b2u(h01);
            pw[2 * j + 1] = b2u(h23);
            pw[8 + 2 * j] = b2u(__floats2bfloat162_rn(r01.x, r01.y));
            pw[8 + 2 * j + 1] = b2u(__floats2bfloat162_rn(r23.x, r23.y));
          }
          tmem_st16(sb + 64 * half + c, pw);
        }
      };
      if (__all_sync(0xffffffffu, !rv || live)) pass2(std::false_type{});
      else pass2(std::true_type{});
      l_sum += lt.x + lt.y;
      {
        const float beta = bt.x + bt.y;
        const __nv_bfloat16 bh = __float2bfloat16_rn(beta);
        const __nv_bfloat16 bl = __float2bfloat16_rn(beta - __bfloat162float(bh));
        tmem_st1(sb + 128 + half, (uint32_t)__bfloat16_as_ushort(bh) | ((uint32_t)__bfloat16_as_ushort(bl) << 16));
        if (half) {  // k 132..143 of the beta block are zero
          tmem_st2(sb + 130, 0u, 0u);
          tmem_st4(sb + 132, 0u, 0u, 0u, 0u);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&sm.p_full[s]);
    }
    // ---- this CTA's partial of each row: half h writes channels 64 h .. 64 h + 63
    bool ok = !dead && wait_all(&sm.pv_done, (n_tiles - 1) & 1, p.err);
    sm.xl[half][r] = l_sum;
    mbar_arrive(&sm.lbar);
    ok = wait_all(&sm.lbar, 0, p.err) && ok;
    tc_fence_after();
    float* o = mq_part(p, b, h, rb, chunk, rv ? r : 0);
    const bool wv = rv && kcheck(o, MQ_PART * sizeof(float), p.ws, (size_t)p.ws_bytes, p.err);
    if (wv && half == 0) {
      o[0] = ok ? m_ref : -INFINITY;
      o[1] = ok ? l_sum + sm.xl[1][r] : 0.f;
    }
#pragma unroll
    for (int c = 0; c < 64; c += 16) {
      uint32_t d[16];
      tmem_ld16(lane_base + TM_O + 64 * half + c, d);
      tmem_wait_ld();
      if (wv) {
        float* oa = o + MQ_PACC + 64 * half + c;
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          *reinterpret_cast<float4*>(oa + i) = ok ? make_float4(__uint_as_float(d[i]), __uint_as_float(d[i + 1]),
                                                                __uint_as_float(d[i + 2]), __uint_as_float(d[i + 3]))
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 12) tmem_dealloc(tmem, TM_COLS);
}

// One warp per output row (sequence, query, query head): merge the split-K
// partials, rotate the packed part back, add the raw part, normalise.
__global__ void __launch_bounds__(128) mq_combine_kernel(MQParams p, int batch, float* __restrict__ out) {
  wait_prerequisite();  // the split-K kernel's partial rows
  const int wid = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int per_seq = p.n_queries * p.num_q_heads;
  if (wid >= batch * per_seq) return;
  const int b = wid / per_seq, qi = (wid % per_seq) / p.num_q_heads, hq = wid % p.num_q_heads;
  const int h = hq / p.G, gq = hq % p.G;
  const int R = qi * p.G + gq, rb = R / MQ_ROWS, r = R % MQ_ROWS;
  const int len = p.seq_lens[b];
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* plo = mq_part(p, b, h, rb, 0, r);
  const size_t pspan = (size_t)(mq_part(p, b, h, rb, p.n_chunks, r) + MQ_PART - plo) * sizeof(float);
  if (len >= p.n_queries && len <= T * p.max_blocks && kcheck(plo, pspan, p.ws, (size_t)p.ws_bytes, p.err)) {
    int rows, n_need;
    mq_block_extent(p, rb, len, rows, n_need);
    const int n_c = (n_need + p.chunk_tiles - 1) / p.chunk_tiles;
    const bool has_tail = (len % T) != 0;
    float M = -INFINITY;
    for (int i = 0; i < n_c; ++i) M = fmaxf(M, mq_part(p, b, h, rb, i, r)[0]);
    if (has_tail) M = fmaxf(M, mq_part(p, b, h, rb, p.n_chunks, r)[0]);
    float Lsum = 0.f;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (M != -INFINITY) {
      for (int i = 0; i < n_c; ++i) {
        const float* pp = mq_part(p, b, h, rb, i, r);
        const float f = (pp[0] == -INFINITY) ? 0.f : exp2f(pp[0] - M);
        Lsum += f * pp[1];
        const float4 a = *reinterpret_cast<const float4*>(pp + MQ_PACC + 4 * lane);
        x[0] += f * a.x; x[1] += f * a.y; x[2] += f * a.z; x[3] += f * a.w;
      }
    }
    // x = x H / sqrt(128) over the 128 channels held 4 per lane
    float u = x[0], v = x[1];
    x[0] = u + v; x[1] = u - v;
    u = x[2]; v = x[3];
    x[2] = u + v; x[3] = u - v;
    u = x[0]; v = x[2];
    x[0] = u + v; x[2] = u - v;
    u = x[1]; v = x[3];
    x[1] = u + v; x[3] = u - v;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float other = __shfl_xor_sync(0xffffffffu, x[e], m);
        x[e] = upper ? (other - x[e]) : (x[e] + other);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] *= INV_SQRT_D;
    if (has_tail && M != -INFINITY) {
      const float* pp = mq_part(p, b, h, rb, p.n_chunks, r);
      const float f = (pp[0] == -INFINITY) ? 0.f : exp2f(pp[0] - M);
      Lsum += f * pp[1];
      const float4 a = *reinterpret_cast<const float4*>(pp + MQ_PACC + 4 * lane);
      x[0] += f * a.x; x[1] += f * a.y; x[2] += f * a.z; x[3] += f * a.w;
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    o = make_float4(x[0] * inv, x[1] * inv, x[2] * inv, x[3] * inv);
  }
  float* dst = out + (((int64_t)b * p.n_queries + qi) * p.num_q_heads + hq) * D + 4 * lane;
  if (kcheck(dst, sizeof(float4), out, (size_t)batch * p.n_queries * p.num_q_heads * D * sizeof(float), p.err))
    *reinterpret_cast<float4*>(dst) = o;
}

template <typename E, int KBITS, int VBITS>
cudaError_t launch_mq_t(const MQParams& p, int batch, float* out, cudaStream_t s) {
  const size_t smem = sizeof(MQSmem) + 128;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = smem_attr_once(attr_done, (const void*)mq_kernel<E, KBITS, VBITS>, (int)smem);
  if (e != cudaSuccess) return e;
  mq_kernel<E, KBITS, VBITS><<<dim3(p.n_chunks + 1, p.num_kv_heads * p.n_rowblocks, batch), MQ_THREADS, smem, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int warps = batch * p.n_queries * p.num_q_heads;
  return launch_after(mq_combine_kernel, dim3((warps + 3) / 4), dim3(128), s, p, batch, out);
}

}  // namespace

cudaError_t launch_multiquery(const MQParams& p, int dtype, int batch, float* out, cudaStream_t s) {
  if (p.k_bits == 2)
    return dtype == KVARN_DTYPE_BF16 ? launch_mq_t<__nv_bfloat16, 2, 2>(p, batch, out, s)
                                     : launch_mq_t<__half, 2, 2>(p, batch, out, s);
  if (p.v_bits == 4)
    return dtype == KVARN_DTYPE_BF16 ? launch_mq_t<__nv_bfloat16, 4, 4>(p, batch, out, s)
                                     : launch_mq_t<__half, 4, 4>(p, batch, out, s);
  return dtype == KVARN_DTYPE_BF16 ? launch_mq_t<__nv_bfloat16, 4, 2>(p, batch, out, s)
                                   : launch_mq_t<__half, 4, 2>(p, batch, out, s);
}

size_t multiquery_ws_bytes(int batch, int num_kv_heads, int n_rowblocks, int max_blocks, int chunk_tiles) {
  const size_t n_chunks = (size_t)(max_blocks + chunk_tiles - 1) / chunk_tiles;
  return (size_t)batch * num_kv_heads * n_rowblocks * (n_chunks + 1) * MQ_ROWS * MQ_PART * sizeof(float);
}

}  // namespace kvarn
