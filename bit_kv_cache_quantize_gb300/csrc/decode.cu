// decode.cu -- read path of the KVarN cache: split-K paged decode attention
// over packed 4-bit K / 2-bit V tiles plus the raw open tile, the split-K
// combine (with the single inverse rotation), and a 16-bit paged decode
// kernel on the same shapes as a comparison point.
//
// Scales are applied at read time (page "Huawei's KVarN puts KV-cache
// quantization inside vLLM's backend", section "The four-stage pipeline",
// fourth stage).  With R[t][c] = g[c] (a[t] code + b[t]) and K = R H:
//   score_t = scale <q, k_t> = a_t <qg, code_t> + b_t S,  qg = (q H scale) * gK,
//                                                       S = sum_c qg[c]
//   sum_t p_t v_t = (gV * (sum_t p_t a_t code_t + sum_t p_t b_t)) H
// so the key rotation and per-channel key scales fold into the query once
// per tile, the per-token scale/zero into the scores, the per-channel value
// scales into the accumulator, and one inverse rotation (in the combine)
// finishes the output.
//
// The two contractions per tile (QK: 128 tokens x 128 channels x G queries,
// PV: 128 channels x 128 tokens x G queries) run as warp MMAs m16n8k16 with
// the codes unpacked in registers straight into the fragments: rows 0-7 of
// the A operand are the fp16 high parts of the G <= 8 queries (or
// probabilities), rows 8-15 their fp16 low parts, so each product is exact
// to ~2^-22 while the 4-/2-bit codes are exact small integers.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "params.h"

namespace kvarn {

constexpr float LOG2E = 1.4426950408889634f;
constexpr uint32_t MAGIC = 0x64006400u;  // 1024.0 in both fp16 halves
constexpr int kMaxDevices = 64;
constexpr int PART = D + 4;  // floats per split-K partial: m, l, 2 pad, acc[128] (16-byte aligned)
constexpr int PACC = 4;      // offset of acc[] in a partial


__device__ __forceinline__ float* part_ptr(const DecodeParams& p, int b, int h, int chunk, int g) {
  return p.ws + ((((int64_t)b * p.num_kv_heads + h) * (p.n_chunks + 1) + chunk) * p.G + g) * PART;
}


__device__ __forceinline__ __half2 u2h2(uint32_t x) { return *reinterpret_cast<__half2*>(&x); }
__device__ __forceinline__ uint32_t h22u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Two fp16 codes (1024 + c) in a half2 -> exact (c0, c1).
__device__ __forceinline__ uint32_t unbias(uint32_t x) {
  __half2 h = *reinterpret_cast<__half2*>(&x);
  h = __hsub2(h, __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
  return *reinterpret_cast<uint32_t*>(&h);
}


template <typename E>
__device__ __forceinline__ float to_f(E x) {
  if constexpr (std::is_same_v<E, __half>) return __half2float(x);
  else return __bfloat162float(x);
}

constexpr int PV_ILP = 4;  // independent MMA chains interleaved in PV

// Shared memory of one packed-decode CTA: per warp one K-record buffer and
// one V-record buffer -- the next tile's K record streams in while this
// tile's V record is in use and vice versa -- the query operand fragments,
// and the cross-warp merge area (aliases the K buffers at the end).
// Warps per CTA (NW): 8, two CTAs per SM at 128 registers; or 4, two CTAs
// per SM at the registers such CTAs may have (no spills).  The K4/V4 preset,
// whose 17 KB records leave room for fewer buffers, always takes 4 (measured
// 10 % faster on the 16K decode than one 8-warp CTA per SM); the others take
// 4 for small calls (8-tile chunks, 7 % faster on the Qwen3-4B layer) and 8
// otherwise.
template <int KBITS, int VBITS, int NW>
struct DecSmem {
  alignas(128) unsigned char krec[NW][rec_bytes(KBITS)];
  alignas(128) unsigned char vrec[NW][rec_bytes(VBITS)];
  alignas(16) uint4 qf[8][32];  // [kb][lane]: fp16 query pairs in A-fragment order: hi, lo of the first
                                // channel pair, hi, lo of the second, each over its field multiplier
  alignas(16) float qr[8][D];   // rotated, scaled queries (set-up only)
  float qsi[8];                 // per query: inverse of its power-of-two operand scale
  uint64_t kbar[NW];
  uint64_t vbar[NW];
};
template <int NW>
struct DecMerge {
  float m[NW][8];
  float l[NW][8];
  float acc[NW][8][D];
};
static_assert(sizeof(DecMerge<8>) <= sizeof(DecSmem<2, 2, 8>::krec), "merge area must fit");
static_assert(sizeof(DecMerge<4>) <= sizeof(DecSmem<2, 2, 4>::krec), "merge area must fit");
static_assert(K_REC % 128 == 0 && K2_REC % 128 == 0 && V_REC % 128 == 0 && V4_REC % 128 == 0,
              "record buffers stay 128-byte aligned");

// Key layouts.  KBITS = 4: token rows of 64 B, byte i = channels 2i, 2i+1 (nibbles).
// KBITS = 2: token rows of 32 B, byte i = channels 4i .. 4i+3 (crumbs at bits 2k).
// A QK k-block kb takes, from the lane's 32 channels 32j .. 32j+31, two channel
// pairs (one per B register) whose codes sit at the same bits of the two
// half-words of one 32-bit code word; their entries of the query operand are
// divided by the power of two the field position multiplies the code by.
template <int KBITS>
struct KeyLayout;
template <>
struct KeyLayout<4> {
  // channels (c0, c0+4) at x1 and (c0+1, c0+5) at x16, c0 = 8 (kb >> 1) + 2 (kb & 1)
  __device__ static int ch_a(int kb) { return 8 * (kb >> 1) + 2 * (kb & 1); }
  __device__ static int ch_b(int kb) { return ch_a(kb) + 1; }
  static constexpr int PAIR = 4;                        // distance between the two channels of a pair
  __device__ static float scale_a(int) { return 1.f; }
  __device__ static float scale_b(int) { return 1.f / 16.f; }
  __device__ static int gword_lo(int kb) { return 2 * (kb >> 1); }  // g bytes: word of ch_a, word of ch_a + PAIR
  __device__ static int gword_hi(int kb) { return 2 * (kb >> 1) + 1; }
};
template <>
struct KeyLayout<2> {
  // word w = kb >> 2 holds channels 16w .. 16w+15 (low half 0-7, high half 8-15);
  // (kb >> 1) & 1 selects the word shifted by 8; fields at crumbs s0 = 2 (kb & 1), s0 + 1
  __device__ static int ch_a(int kb) { return 16 * (kb >> 2) + 4 * ((kb >> 1) & 1) + 2 * (kb & 1); }
  __device__ static int ch_b(int kb) { return ch_a(kb) + 1; }
  static constexpr int PAIR = 8;
  __device__ static float scale_a(int kb) { return (kb & 1) ? 1.f / 16.f : 1.f; }
  __device__ static float scale_b(int kb) { return (kb & 1) ? 1.f / 64.f : 1.f / 4.f; }
  __device__ static int gword_lo(int kb) { return 4 * (kb >> 2) + ((kb >> 1) & 1); }
  __device__ static int gword_hi(int kb) { return gword_lo(kb) + 2; }
};

template <typename E>
__device__ void tail_chunk(const DecodeParams& p, int b, int h, int len, unsigned char* smem);

// Unpacking codes to exact fp16 operands.  A code field ORed into the
// mantissa of 1024.0 (0x6400) and 1024 subtracted gives the code exactly.
// A field at mantissa bits 4s .. 4s+3 (nibble) or 2s .. 2s+1 (crumb) comes
// out multiplied by 16^s or 4^s; the matching entries of the other operand
// carry the inverse power of two, which is exact.
// (x & mask) | MAGIC as one explicit three-input logic op (the C expression
// compiles to two), then the exact fp16 subtraction of 1024.
__device__ __forceinline__ uint32_t field(uint32_t x, uint32_t mask) {
  uint32_t y;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(y) : "r"(x), "r"(mask), "r"(MAGIC));
  return unbias(y);
}

// Two E4M3 bytes (low byte first) -> fp16 pair, exact.
__device__ __forceinline__ __half2 e4m3x2_to_half2(uint32_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
  return __half2(h);
}

// grid (n_chunks + 1, H_kv, B) x 32 NW threads; chunk n_chunks handles the
// raw open tile.  Warp w of a chunk takes its tiles first + w, first + w + NW, ....
//
// Per tile and warp, with lane = 4 g + j:
//   QK (m16n8k16, M = 8 queries hi | lo, N = 8 tokens, K = 16 channels):
//     A = qg = q * gK as an exact fp16 high part plus low part, formed per
//     tile from the fp16 query pairs with HMUL2/HFMA2; B = 4-bit codes of
//     token 32 (g >> 1) + 2 nb + (g & 1), channels 32 j .. 32 j + 31 in the
//     order (c0, c0+4 | c0+1, c0+5), c0 = 32 j + 8 (kb >> 1) + 2 (kb & 1).
//     Lane (g, j) receives the scores of query g for tokens 32 j + 2 nb, +1.
//   S = sum_c qg_c from eight more MMAs against constant B = 1 | 16.
//   PV: A = p aV 64 / 4^(nb & 3) (hi | lo) of the same tokens, which k-block
//     kb = nb >> 1 takes as k = 2j, 2j+1 (nb even) and 2j+8, 2j+9 (nb odd);
//     B = 2-bit codes of channel 8 nbp + g, whose 32-bit words keep even
//     tokens in the low half and odd tokens in the high half, so each B
//     register is one masked field of one word.
// Two CTAs per SM: 8 warps at 128 registers a thread, or 4 warps at the
// registers two 4-warp CTAs may have (no spills).
template <typename E, int KBITS, int VBITS, int NW>
__global__ void __launch_bounds__(32 * NW, 2) decode_packed_kernel(DecodeParams p) {
  using KL = KeyLayout<KBITS>;
  constexpr int KREC = rec_bytes(KBITS), KROW = D * KBITS / 8;  // KROW: code bytes per token
  constexpr int VREC = rec_bytes(VBITS);
  static_assert(KROW == 16 * KBITS, "token row");
  extern __shared__ __align__(128) unsigned char smem_raw[];
  allow_dependents();  // the combine may be scheduled once every CTA has started
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, j = lane & 3;
  const int len = p.seq_lens[b];
  if (len < 0 || len > T * p.max_blocks) {
    if (tid == 0 && chunk == 0 && h == 0) set_error(p.err, KVARN_DEV_ERR_TOKEN_RANGE);
    return;
  }
  if (chunk == p.n_chunks) {
    tail_chunk<E>(p, b, h, len, smem_raw);
    return;
  }
  const int n_closed = len / T;
  const int first = chunk * p.chunk_tiles;
  const int n_tiles = min(p.chunk_tiles, n_closed - first);
  if (n_tiles <= 0) return;
  const uint32_t sbase = smem_u32(smem_raw);
  DecSmem<KBITS, VBITS, NW>& sm =
      *reinterpret_cast<DecSmem<KBITS, VBITS, NW>*>(smem_raw + (((sbase + 127u) & ~127u) - sbase));
  const int G = p.G;
  const int32_t* tab = p.block_table + (int64_t)b * p.max_blocks;
  const int my_n = (n_tiles > warp) ? (n_tiles - warp + NW - 1) / NW : 0;
  const int polls = p.wait_polls > 0 ? p.wait_polls : kWaitPolls;

  // start this warp's first tile before anything else
  if (lane == 0) {
    mbar_init(&sm.kbar[warp], 1);
    mbar_init(&sm.vbar[warp], 1);
    fence_mbar_init();
  }
  __syncwarp();
  auto issue = [&](int k, bool is_v) {  // lane 0: copy the K or V record of this warp's k-th tile
    if (p.skip_first_copy && k == 0 && !is_v && warp == 0 && chunk == 0 && h == 0 && b == 0)
      return;  // error-path test: this copy never starts, so its wait must expire
    const int32_t blk = tab[first + warp + k * NW];
    uint64_t* bar = is_v ? &sm.vbar[warp] : &sm.kbar[warp];
    const unsigned char* src = p.pool + blk * p.block_bytes + (int64_t)h * head_rec(KBITS, VBITS) + (is_v ? KREC : 0);
    const uint32_t bytes = is_v ? VREC : KREC;
    if (blk >= 0 && blk < p.num_blocks && kcheck(src, bytes, p.pool, (size_t)p.num_blocks * p.block_bytes, p.err)) {
      mbar_expect_tx(bar, bytes);
      bulk_g2s_stream(is_v ? sm.vrec[warp] : sm.krec[warp], src, bytes, bar);
    } else {
      set_error(p.err, KVARN_DEV_ERR_BLOCK_RANGE);
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
    }
  };
  if (lane == 0 && my_n > 0) { issue(0, false); issue(0, true); }

  // rotated, scaled queries: warp w rotates queries w, w + NW, ... (rows past
  // G stay zero) with a 128-point butterfly over 4 channels per lane;
  // qr = qs * scale * log2(e) * (q H), qs a power of two putting max |qr| in
  // [64, 128), so |qr gK| <= 128 * 448 stays inside fp16
#pragma unroll
  for (int it = 0; it < 8 / NW; ++it) {
    const int qq = warp + NW * it;
    const E* qb = static_cast<const E*>(p.q) + ((int64_t)b * p.num_q_heads + (int64_t)h * G) * D;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (qq < G) {
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = to_f(qb[qq * D + 4 * lane + e]);
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
      for (int e = 0; e < 4; ++e) {
        const float o = __shfl_xor_sync(0xffffffffu, x[e], m);
        x[e] = upper ? (o - x[e]) : (x[e] + o);
      }
    }
    const float f = p.scale * LOG2E * INV_SQRT_D;
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[e] *= f;
      amax = fmaxf(amax, fabsf(x[e]));
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    int ex = 0;
    if (amax > 0.f) frexpf(amax, &ex);
    const float qs = ldexpf(1.f, 7 - ex);
    *reinterpret_cast<float4*>(&sm.qr[qq][4 * lane]) = make_float4(x[0] * qs, x[1] * qs, x[2] * qs, x[3] * qs);
    if (lane == 0) sm.qsi[qq] = ldexpf(1.f, ex - 7);
  }
  __syncthreads();
#pragma unroll
  for (int it = 0; it < 8 / NW; ++it) {  // thread (kb, lane) forms the fp16 high/low query pairs of its A-fragment slot
    const int kb = warp + NW * it;
    const int ca = 32 * j + KL::ch_a(kb), cb = 32 * j + KL::ch_b(kb);
    const float* q = sm.qr[g];
    const float sa = KL::scale_a(kb), sb = KL::scale_b(kb);
    const float v0 = q[ca] * sa, v1 = q[ca + KL::PAIR] * sa, v2 = q[cb] * sb, v3 = q[cb + KL::PAIR] * sb;
    const __half2 h01 = __floats2half2_rn(v0, v1), h23 = __floats2half2_rn(v2, v3);
    const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
    const __half2 l01 = __floats2half2_rn(v0 - f01.x, v1 - f01.y), l23 = __floats2half2_rn(v2 - f23.x, v3 - f23.y);
    sm.qf[kb][lane] = make_uint4(h22u(h01), h22u(l01), h22u(h23), h22u(l23));
  }
  __syncthreads();

  const float qsi = sm.qsi[g];
  float m_run = -INFINITY, l_run = 0.f;
  float2 acc[16];  // query g, channels 8 nbp + 2j, +1
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) acc[nb] = make_float2(0.f, 0.f);

  for (int k = 0; k < my_n; ++k) {
    const int32_t blk = tab[first + warp + k * NW];
    const bool valid = blk >= 0 && blk < p.num_blocks;
    const unsigned char* kr = sm.krec[warp];
    const unsigned char* vr = sm.vrec[warp];
    // a wait that gives up ends this warp's loop (after waiting, bounded, for
    // the V copy it still has in flight); the error word is already set
    if (__any_sync(0xffffffffu, !mbar_wait_bounded(&sm.kbar[warp], k & 1, p.err, polls))) {
      mbar_wait_bounded(&sm.vbar[warp], k & 1, p.err);
      break;
    }

    float2 sc[16];  // scores x qs of query g, tokens 32j + 2nb, +1
    float tmax = -INFINITY;
    if (valid) {
      // ---- A operand: qg = q gK, high part RN(q_hi gK), low part q_lo gK + (q_hi gK - high)
      uint32_t afr[8][4];
      {
        const uint4 gA = *reinterpret_cast<const uint4*>(kr + 32 * j);
        const uint4 gB = *reinterpret_cast<const uint4*>(kr + 32 * j + 16);
        const uint32_t gw[8] = {gA.x, gA.y, gA.z, gA.w, gB.x, gB.y, gB.z, gB.w};  // channels 32j + 4i .. +3
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          const uint32_t lo = gw[KL::gword_lo(kb)], hi = gw[KL::gword_hi(kb)];
          const uint32_t pr = __byte_perm(lo, hi, (kb & 1) ? 0x7362 : 0x5140);
          const __half2 g01 = e4m3x2_to_half2(pr), g23 = e4m3x2_to_half2(pr >> 16);
          const uint4 qv = sm.qf[kb][lane];
          const __half2 h01 = __hmul2_rn(u2h2(qv.x), g01);
          const __half2 l01 = __hfma2(u2h2(qv.y), g01, __hfma2(u2h2(qv.x), g01, __hneg2(h01)));
          const __half2 h23 = __hmul2_rn(u2h2(qv.z), g23);
          const __half2 l23 = __hfma2(u2h2(qv.w), g23, __hfma2(u2h2(qv.z), g23, __hneg2(h23)));
          afr[kb][0] = h22u(h01); afr[kb][1] = h22u(l01);
          afr[kb][2] = h22u(h23); afr[kb][3] = h22u(l23);
        }
      }
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {  // B = the field multipliers (1 | 16 for 4-bit keys; 1 | 4, 16 | 64 for 2-bit)
        const uint32_t b0 = (KBITS == 4 || !(kb & 1)) ? 0x3C003C00u : 0x4C004C00u;
        const uint32_t b1 = KBITS == 4 ? 0x4C004C00u : ((kb & 1) ? 0x54005400u : 0x44004400u);
        mma_f16(sacc, afr[kb], b0, b1);
      }
      const float S = sacc[0] + sacc[2];
      const float2 S2 = make_float2(S, S);

      // ---- QK: scores x qs = aK <qg, code> + bK S
      const unsigned char* kc = kr + 512 + (32 * (g >> 1) + (g & 1)) * KROW + (KROW / 4) * j;
      const unsigned char* ka = kr + 128 + 32 * j;
      const unsigned char* kz = kr + 256 + 64 * j;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint2 a8 = *reinterpret_cast<const uint2*>(ka + 8 * q4);
        const uint4 b8 = *reinterpret_cast<const uint4*>(kz + 16 * q4);
        const uint32_t bw[4] = {b8.x, b8.y, b8.z, b8.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int nb = 4 * q4 + i;
          float c[4] = {0.f, 0.f, 0.f, 0.f};
          if constexpr (KBITS == 4) {
            const uint4 v4 = *reinterpret_cast<const uint4*>(kc + nb * 2 * KROW);
            const uint32_t kw[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) {
              const uint32_t x = (kb & 1) ? (kw[kb >> 1] >> 8) : kw[kb >> 1];
              mma_f16(c, afr[kb], field(x, 0x000F000Fu), field(x, 0x00F000F0u));
            }
          } else {
            const uint2 v2 = *reinterpret_cast<const uint2*>(kc + nb * 2 * KROW);
            const uint32_t kw[2] = {v2.x, v2.y};
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) {
              const uint32_t x = ((kb >> 1) & 1) ? (kw[kb >> 2] >> 8) : kw[kb >> 2];
              const uint32_t m0 = 0x00030003u << (4 * (kb & 1));
              mma_f16(c, afr[kb], field(x, m0), field(x, m0 << 2));
            }
          }
          const float2 a2 = __half22float2(e4m3x2_to_half2(((i & 2) ? a8.y : a8.x) >> (16 * (i & 1))));
          const float2 b2 = __half22float2(u2h2(bw[i]));
          const float2 s2 = ffma2(a2, fadd2(make_float2(c[0], c[1]), make_float2(c[2], c[3])), fmul2(b2, S2));
          sc[nb] = s2;
          tmax = fmaxf(tmax, fmaxf(s2.x, s2.y));
        }
      }
    }
    __syncwarp();
    if (lane == 0 && k + 1 < my_n) {  // this K buffer is free: fetch the next tile's K
      fence_proxy_async();
      issue(k + 1, false);
    }
    if (__any_sync(0xffffffffu, !mbar_wait_bounded(&sm.vbar[warp], k & 1, p.err, polls))) {
      if (k + 1 < my_n) mbar_wait_bounded(&sm.kbar[warp], (k + 1) & 1, p.err);
      break;
    }
    if (valid) {
      // ---- online softmax (log2 domain)
      tmax = quad_max(tmax);
      const float m_new = fmaxf(m_run, tmax * qsi);
      const float corr = ex2_ftz(m_run - m_new);
      const float nm = -m_new;
      const float2 nm2 = make_float2(nm, nm), qsi2 = make_float2(qsi, qsi);
      m_run = m_new;
      // ---- P = p aV 64 / 4^(nb & 3), hi rows 0-7 / lo rows 8-15
      uint32_t pfr[8][4];
      float2 psum = make_float2(0.f, 0.f), pb = psum;
      const unsigned char* va = vr + 128 + 32 * j;
      const unsigned char* vz = vr + 256 + 64 * j;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint2 a8 = *reinterpret_cast<const uint2*>(va + 8 * q4);
        const uint4 b8 = *reinterpret_cast<const uint4*>(vz + 16 * q4);
        const uint32_t bw[4] = {b8.x, b8.y, b8.z, b8.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int nb = 4 * q4 + i;
          const float2 ea = ffma2(sc[nb], qsi2, nm2);  // per element the same fused multiply-add as fmaf
          const float2 pr = make_float2(ex2_ftz(ea.x), ex2_ftz(ea.y));
          psum = fadd2(psum, pr);
          pb = ffma2(pr, __half22float2(u2h2(bw[i])), pb);
          // undo the field multiplier of the V operand: 4^(nb & 3) for 2-bit fields, 16^(nb & 1) for 4-bit
          const __half2 f2 = __float2half2_rn(VBITS == 2 ? 64.f / (float)(1 << (2 * (nb & 3)))
                                                         : 16.f / (float)(1 << (4 * (nb & 1))));
          const __half2 av = __hmul2(e4m3x2_to_half2(((i & 2) ? a8.y : a8.x) >> (16 * (i & 1))), f2);  // exact
          const float2 pa = fmul2(pr, __half22float2(av));
          const __half2 hi = __float22half2_rn(pa);
          const float2 lo = ffma2(__half22float2(hi), make_float2(-1.f, -1.f), pa);  // pa - hi, exact product
          pfr[nb >> 1][(nb & 1) ? 2 : 0] = h22u(hi);
          pfr[nb >> 1][(nb & 1) ? 3 : 1] = h22u(__float22half2_rn(lo));
        }
      }
      l_run = l_run * corr + quad_sum(psum.x + psum.y);
      const float pbs = quad_sum(pb.x + pb.y);
      const float2 corr2 = make_float2(corr, corr), pbs2 = make_float2(pbs, pbs);
      constexpr float PSC = VBITS == 2 ? 1.f / 64.f : 1.f / 16.f;  // the constant factor of P'
      const float2 inv64 = make_float2(PSC, PSC);
      if constexpr (VBITS == 4) {
      // ---- PV: B = 4-bit codes of channel 8 nbp + g, tokens 32j .. 32j+31 (words 4j .. 4j+3)
      const unsigned char* vc = vr + 512 + g * 64 + 16 * j;
#pragma unroll
      for (int n4 = 0; n4 < 16; n4 += PV_ILP) {
        uint4 vw[PV_ILP];
#pragma unroll
        for (int i = 0; i < PV_ILP; ++i) vw[i] = *reinterpret_cast<const uint4*>(vc + (n4 + i) * 512);
        float c[PV_ILP][4];
#pragma unroll
        for (int i = 0; i < PV_ILP; ++i) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          // tokens 32j + 4kb + {0,1} | {2,3}: nibbles at bits 0 | 4 of word kb >> 1, shifted by 8 when kb & 1
#pragma unroll
          for (int i = 0; i < PV_ILP; ++i) {
            const uint32_t w = (kb >> 1) == 0 ? vw[i].x : (kb >> 1) == 1 ? vw[i].y : (kb >> 1) == 2 ? vw[i].z : vw[i].w;
            const uint32_t x = (kb & 1) ? (w >> 8) : w;
            mma_f16(c[i], pfr[kb], field(x, 0x000F000Fu), field(x, 0x00F000F0u));
          }
        }
#pragma unroll
        for (int i = 0; i < PV_ILP; ++i) {
          const int nbp = n4 + i;
          const float2 gv = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(vr + 8 * nbp + 2 * j));
          const float2 o = ffma2(fadd2(make_float2(c[i][0], c[i][1]), make_float2(c[i][2], c[i][3])), inv64, pbs2);
          acc[nbp] = ffma2(acc[nbp], corr2, fmul2(gv, o));
        }
      }
      } else {
      // ---- PV: B = 2-bit codes of channel 8 nbp + g, tokens 32j .. 32j+31
      const unsigned char* vc = vr + 512 + g * 32 + 8 * j;
#pragma unroll
      for (int n4 = 0; n4 < 16; n4 += PV_ILP) {
        uint2 vw[PV_ILP];
#pragma unroll
        for (int i = 0; i < PV_ILP; ++i) vw[i] = *reinterpret_cast<const uint2*>(vc + (n4 + i) * 256);
        float c[PV_ILP][4];
#pragma unroll
        for (int i = 0; i < PV_ILP; ++i) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          // tokens 32j + 4kb + {0,1} | {2,3}: fields at bits 4 (kb & 1) | +2 of word kb >> 2, shifted by 8 when kb & 2
          const uint32_t m0 = 0x00030003u << (4 * (kb & 1));
#pragma unroll
          for (int i = 0; i < PV_ILP; ++i) {
            const uint32_t w = (kb & 4) ? vw[i].y : vw[i].x;
            const uint32_t x = (kb & 2) ? (w >> 8) : w;
            mma_f16(c[i], pfr[kb], field(x, m0), field(x, m0 << 2));
          }
        }
#pragma unroll
        for (int i = 0; i < PV_ILP; ++i) {
          const int nbp = n4 + i;
          const float2 gv = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(vr + 8 * nbp + 2 * j));
          const float2 o = ffma2(fadd2(make_float2(c[i][0], c[i][1]), make_float2(c[i][2], c[i][3])), inv64, pbs2);
          acc[nbp] = ffma2(acc[nbp], corr2, fmul2(gv, o));
        }
      }
      }
    }
    __syncwarp();
    if (lane == 0 && k + 1 < my_n) {  // this V buffer is free: fetch the next tile's V
      fence_proxy_async();
      issue(k + 1, true);
    }
  }

  // ---- merge the warps and write this CTA's partial
  __syncthreads();
  DecMerge<NW>& mg = *reinterpret_cast<DecMerge<NW>*>(sm.krec);
  if (j == 0) { mg.m[warp][g] = m_run; mg.l[warp][g] = l_run; }
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) *reinterpret_cast<float2*>(&mg.acc[warp][g][8 * nb + 2 * j]) = acc[nb];
  __syncthreads();
  for (int i = tid; i < G * D; i += 32 * NW) {
    const int gg = i / D, c = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mg.m[w][gg]);
    float Lsum = 0.f, A = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = exp2f(mg.m[w][gg] - M);
        Lsum += f * mg.l[w][gg];
        A += f * mg.acc[w][gg][c];
      }
    }
    float* o = part_ptr(p, b, h, chunk, gg);
    if (!kcheck(o, PART * sizeof(float), p.ws, (size_t)p.ws_bytes, p.err)) continue;
    if (c == 0) { o[0] = M; o[1] = Lsum; }
    o[PACC + c] = A;
  }
}

// Raw open tile of (b, h): len % 128 tokens in 16-bit, unrotated query.
template <typename E>
__device__ void tail_chunk(const DecodeParams& p, int b, int h, int len, unsigned char* smem) {
  const int n = len % T;
  if (n == 0) return;
  const int tid = threadIdx.x, G = p.G;
  float* qs = reinterpret_cast<float*>(smem);  // [8][128]
  float* pr = qs + 8 * D;                      // [8][128] scores, then probabilities
  float* ml = pr + 8 * T;                      // [8][2]
  const E* qb = static_cast<const E*>(p.q) + ((int64_t)b * p.num_q_heads + (int64_t)h * G) * D;
  const float f = p.scale * LOG2E;
  for (int i = tid; i < G * D; i += blockDim.x) qs[i] = to_f(qb[i]) * f;
  __syncthreads();
  const E* kt = static_cast<const E*>(p.tail) + (((int64_t)b * p.num_kv_heads + h) * 2 + 0) * (T * D);
  const E* vt = kt + T * D;
  if (!kcheck(kt, 2 * T * D * sizeof(E), p.tail, (size_t)gridDim.z * p.num_kv_heads * 2 * T * D * sizeof(E), p.err))
    return;
  if (tid < n) {
    float s[8];
#pragma unroll
    for (int gg = 0; gg < 8; ++gg) s[gg] = 0.f;
    for (int c = 0; c < D; ++c) {
      const float kv = to_f(kt[tid * D + c]);
#pragma unroll
      for (int gg = 0; gg < 8; ++gg)
        if (gg < G) s[gg] = fmaf(qs[gg * D + c], kv, s[gg]);
    }
    for (int gg = 0; gg < G; ++gg) pr[gg * T + tid] = s[gg];
  }
  __syncthreads();
  if (tid < G) {
    float m = -INFINITY, l = 0.f;
    for (int t = 0; t < n; ++t) m = fmaxf(m, pr[tid * T + t]);
    for (int t = 0; t < n; ++t) {
      const float e = exp2f(pr[tid * T + t] - m);
      pr[tid * T + t] = e;
      l += e;
    }
    ml[2 * tid] = m;
    ml[2 * tid + 1] = l;
  }
  __syncthreads();
  if (tid >= D) return;
  float a[8];
#pragma unroll
  for (int gg = 0; gg < 8; ++gg) a[gg] = 0.f;
  for (int t = 0; t < n; ++t) {
    const float v = to_f(vt[t * D + tid]);
#pragma unroll
    for (int gg = 0; gg < 8; ++gg)
      if (gg < G) a[gg] = fmaf(pr[gg * T + t], v, a[gg]);
  }
  for (int gg = 0; gg < G; ++gg) {
    float* out = part_ptr(p, b, h, p.n_chunks, gg);
    if (!kcheck(out, PART * sizeof(float), p.ws, (size_t)p.ws_bytes, p.err)) continue;
    if (tid == 0) { out[0] = ml[2 * gg]; out[1] = ml[2 * gg + 1]; }
    out[PACC + tid] = a[gg];
  }
}

// One warp per (sequence, query head): merge the split-K partials, apply
// the inverse rotation to the packed-tile part, add the raw part, normalise.
__global__ void __launch_bounds__(128) combine_kernel(DecodeParams p, int rotate, int batch, float* __restrict__ out) {
  wait_prerequisite();  // the split-K kernel's partials
  const int wid = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (wid >= batch * p.num_q_heads) return;
  const int b = wid / p.num_q_heads, hq = wid % p.num_q_heads;
  const int h = hq / p.G, g = hq % p.G;
  const int len = p.seq_lens[b];
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* plo = part_ptr(p, b, h, 0, g);
  const size_t pspan = (size_t)(part_ptr(p, b, h, p.n_chunks, g) + PART - plo) * sizeof(float);
  if (len > 0 && len <= T * p.max_blocks && kcheck(plo, pspan, p.ws, (size_t)p.ws_bytes, p.err)) {
    const int n_tc = rotate ? ((len / T) + p.chunk_tiles - 1) / p.chunk_tiles
                            : (((len + T - 1) / T) + p.chunk_tiles - 1) / p.chunk_tiles;
    const bool has_tail = rotate && (len % T) != 0;
    float M = -INFINITY;
    for (int i = 0; i < n_tc; ++i) M = fmaxf(M, part_ptr(p, b, h, i, g)[0]);
    if (has_tail) M = fmaxf(M, part_ptr(p, b, h, p.n_chunks, g)[0]);
    float Lsum = 0.f;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < n_tc; ++i) {
      const float* pp = part_ptr(p, b, h, i, g);
      const float f = (pp[0] == -INFINITY) ? 0.f : exp2f(pp[0] - M);
      Lsum += f * pp[1];
      const float4 a = *reinterpret_cast<const float4*>(pp + PACC + 4 * lane);
      x[0] += f * a.x; x[1] += f * a.y; x[2] += f * a.z; x[3] += f * a.w;
    }
    if (rotate) {  // x = x H over the 128 channels held 4 per lane
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
    }
    if (has_tail) {
      const float* pp = part_ptr(p, b, h, p.n_chunks, g);
      const float f = exp2f(pp[0] - M);
      Lsum += f * pp[1];
      const float4 a = *reinterpret_cast<const float4*>(pp + PACC + 4 * lane);
      x[0] += f * a.x; x[1] += f * a.y; x[2] += f * a.z; x[3] += f * a.w;
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    o = make_float4(x[0] * inv, x[1] * inv, x[2] * inv, x[3] * inv);
  }
  float* dst = out + ((int64_t)b * p.num_q_heads + hq) * D + 4 * lane;
  if (kcheck(dst, sizeof(float4), out, (size_t)batch * p.num_q_heads * D * sizeof(float), p.err))
    *reinterpret_cast<float4*>(dst) = o;
}

// ------------------------------------------------------------------ 16-bit comparison kernel
// Pool block = [kv_head][K,V][128 tokens][128 channels] 16-bit.  Each tile is
// loaded by TMA as four 64-channel x 128-token boxes with the 128-byte
// swizzle; 8 warps each take 16 tokens of every tile.
constexpr int F16_WARPS = 8;
constexpr int F16_STAGES = 3;
constexpr int F16_TILE = 2 * T * D * 2;  // K + V, 64 KB
struct F16Smem {
  alignas(1024) unsigned char stage[F16_STAGES][F16_TILE];
  uint64_t bar[F16_STAGES];
};
struct F16Merge {
  float m[F16_WARPS][8];
  float l[F16_WARPS][8];
  float acc[F16_WARPS][8][D];
};
static_assert(sizeof(F16Merge) <= sizeof(F16Smem::stage), "merge area must fit the stages");

// Byte offset of 16-byte chunk `ch` (0..15) of row r in a swizzled K or V
// matrix made of two 64-channel boxes of 128 rows x 128 B.
__device__ __forceinline__ int f16_off(int r, int ch) {
  return (ch >> 3) * (T * 128) + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
}

template <typename E>
__global__ void __launch_bounds__(256, 1) decode_f16_kernel(const __grid_constant__ CUtensorMap tmap, DecodeParams p) {
  extern __shared__ __align__(1024) unsigned char smem_f16[];
  allow_dependents();
  // the 128-byte TMA swizzle needs 1024-byte aligned boxes: align explicitly
  const uint32_t base = smem_u32(smem_f16);
  F16Smem& sm = *reinterpret_cast<F16Smem*>(smem_f16 + (((base + 1023u) & ~1023u) - base));
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, j = lane & 3;
  const int len = p.seq_lens[b];
  if (len < 0 || len > T * p.max_blocks) {
    if (tid == 0 && chunk == 0 && h == 0) set_error(p.err, KVARN_DEV_ERR_TOKEN_RANGE);
    return;
  }
  const int n_all = (len + T - 1) / T;
  const int first = chunk * p.chunk_tiles;
  const int n_tiles = min(p.chunk_tiles, n_all - first);
  if (n_tiles <= 0) return;
  const int G = p.G;
  const int32_t* tab = p.block_table + (int64_t)b * p.max_blocks;

  if (tid == 0) {
    for (int s = 0; s < F16_STAGES; ++s) mbar_init(&sm.bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int k) {  // thread 0
    const int s = k % F16_STAGES;
    const int32_t blk = tab[first + k];
    if (blk >= 0 && blk < p.num_blocks) {
      mbar_expect_tx(&sm.bar[s], F16_TILE);
      const int row0 = ((blk * p.num_kv_heads + h) * 2) * T;
#pragma unroll
      for (int part = 0; part < 4; ++part) {  // K lo, K hi, V lo, V hi
        const int x = (part & 1) * 64, y = row0 + (part >> 1) * T;
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
                smem_u32(sm.stage[s] + part * (T * 128))),
            "l"(&tmap), "r"(x), "r"(y), "r"(smem_u32(&sm.bar[s]))
            : "memory");
      }
    } else {
      set_error(p.err, KVARN_DEV_ERR_BLOCK_RANGE);
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&sm.bar[s])) : "memory");
    }
  };
  if (tid == 0)
    for (int k = 0; k < min(n_tiles, F16_STAGES); ++k) issue(k);

  // query fragments: rows 0-7 = queries (exact 16-bit), rows 8-15 zero
  uint32_t qa[8][2];
  {
    const E* qb = static_cast<const E*>(p.q) + ((int64_t)b * p.num_q_heads + (int64_t)h * G) * D;
#pragma unroll
    for (int kb = 0; kb < 8; ++kb)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int c = 16 * kb + 2 * j + 8 * hh;
        qa[kb][hh] = (g < G) ? *reinterpret_cast<const uint32_t*>(qb + g * D + c) : 0u;
      }
  }
  const float sl2 = p.scale * LOG2E;
  float m_run = -INFINITY, l_run = 0.f;
  float acc[16][4];
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;

  for (int k = 0; k < n_tiles; ++k) {
    const int s = k % F16_STAGES;
    const int32_t blk = tab[first + k];
    // a wait that gives up (error word set) ends the loop for the whole CTA
    if (__syncthreads_or(!mbar_wait_bounded(&sm.bar[s], (k / F16_STAGES) & 1, p.err))) break;
    const bool ok = true;
    const int valid = min(T, len - (first + k) * T);
    if (ok && blk >= 0 && blk < p.num_blocks && 16 * warp < valid) {
      const unsigned char* kt = sm.stage[s];
      const unsigned char* vt = kt + 2 * T * 128;
      // QK for tokens 16w .. 16w+15 (two n-blocks)
      float sc[2][4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {  // channel chunks 4kp .. 4kp+3 (k-blocks 2kp, 2kp+1)
          uint32_t r[4];
          const int row = 16 * warp + 8 * nb + (lane & 7);
          ldmatrix_x4(r, kt + f16_off(row, 4 * kp + (lane >> 3)));
          const uint32_t a0[4] = {qa[2 * kp][0], 0u, qa[2 * kp][1], 0u};
          const uint32_t a1[4] = {qa[2 * kp + 1][0], 0u, qa[2 * kp + 1][1], 0u};
          mma16816<E>(c, a0, r[0], r[1]);
          mma16816<E>(c, a1, r[2], r[3]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = 16 * warp + 8 * nb + 2 * j + (e & 1);
          sc[nb][e] = (tok < valid) ? c[e] * sl2 : -INFINITY;
        }
      }
      float tmax = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
      const float m_new = fmaxf(m_run, tmax);
      const float corr = exp2f(m_run - m_new);
      m_run = m_new;
      uint16_t ph[2][2], pl[2][2];
      float psum = 0.f;
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float pr = exp2f(sc[nb][e] - m_new);
          psum += pr;
          split_hl<E>(pr, ph[nb][e], pl[nb][e]);
        }
      psum = quad_sum(psum);
      l_run = l_run * corr + psum;
      const uint32_t pa[4] = {pack2(ph[0][0], ph[0][1]), pack2(pl[0][0], pl[0][1]), pack2(ph[1][0], ph[1][1]),
                              pack2(pl[1][0], pl[1][1])};
      // PV: tokens 16w .. 16w+15 (one k-block) x 128 channels
#pragma unroll
      for (int np = 0; np < 8; ++np) {  // channel n-blocks 2np, 2np+1
        uint32_t r[4];
        const int row = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1);
        ldmatrix_x4_trans(r, vt + f16_off(row, 2 * np + (lane >> 4)));
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816<E>(c0, pa, r[0], r[1]);
        mma16816<E>(c1, pa, r[2], r[3]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[2 * np][e] = fmaf(acc[2 * np][e], corr, c0[e]);
          acc[2 * np + 1][e] = fmaf(acc[2 * np + 1][e], corr, c1[e]);
        }
      }
    }
    __syncthreads();
    if (tid == 0 && k + F16_STAGES < n_tiles) {
      fence_proxy_async();
      issue(k + F16_STAGES);
    }
  }

  F16Merge& mg = *reinterpret_cast<F16Merge*>(sm.stage);
  if (j == 0) { mg.m[warp][g] = m_run; mg.l[warp][g] = l_run; }
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) {
    mg.acc[warp][g][8 * nb + 2 * j] = acc[nb][0] + acc[nb][2];
    mg.acc[warp][g][8 * nb + 2 * j + 1] = acc[nb][1] + acc[nb][3];
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += 256) {
    const int gg = i / D, c = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < F16_WARPS; ++w) M = fmaxf(M, mg.m[w][gg]);
    float Lsum = 0.f, A = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < F16_WARPS; ++w) {
        const float f = exp2f(mg.m[w][gg] - M);
        Lsum += f * mg.l[w][gg];
        A += f * mg.acc[w][gg][c];
      }
    }
    float* o = part_ptr(p, b, h, chunk, gg);
    if (!kcheck(o, PART * sizeof(float), p.ws, (size_t)p.ws_bytes, p.err)) continue;
    if (c == 0) { o[0] = M; o[1] = Lsum; }
    o[PACC + c] = A;
  }
}

// ------------------------------------------------------------------ launchers
size_t decode_ws_bytes(int batch, int num_kv_heads, int G, int max_blocks, int chunk_tiles) {
  const int n_chunks = (max_blocks + chunk_tiles - 1) / chunk_tiles;
  return (size_t)batch * num_kv_heads * (n_chunks + 1) * G * PART * sizeof(float);
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode();

template <typename E, int KBITS, int VBITS, int NW>
static cudaError_t launch_decode_t(DecodeParams p, int batch, float* out, cudaStream_t s) {
  const size_t smem = sizeof(DecSmem<KBITS, VBITS, NW>) + 128;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = smem_attr_once(attr_done, (const void*)decode_packed_kernel<E, KBITS, VBITS, NW>, (int)smem);
  if (e != cudaSuccess) return e;
  decode_packed_kernel<E, KBITS, VBITS, NW><<<dim3(p.n_chunks + 1, p.num_kv_heads, batch), 32 * NW, smem, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int warps = batch * p.num_q_heads;
  return launch_after(combine_kernel, dim3((warps + 3) / 4), dim3(128), s, p, 1, batch, out);
}

template <typename E, int KBITS, int VBITS>
static cudaError_t launch_decode_w(const DecodeParams& p, int batch, float* out, cudaStream_t s) {
  if constexpr (KBITS == 4 && VBITS == 4) {
    return launch_decode_t<E, KBITS, VBITS, 4>(p, batch, out, s);
  } else {  // a small call's 8-tile chunks take the 4-warp CTAs too
    return p.chunk_tiles <= 8 ? launch_decode_t<E, KBITS, VBITS, 4>(p, batch, out, s)
                              : launch_decode_t<E, KBITS, VBITS, 8>(p, batch, out, s);
  }
}

cudaError_t launch_decode(const DecodeParams& p, int dtype, int batch, float* out, cudaStream_t s) {
  const bool bf = dtype == KVARN_DTYPE_BF16;
  if (p.v_bits == 4)  // the K4/V4 preset
    return bf ? launch_decode_w<__nv_bfloat16, 4, 4>(p, batch, out, s) : launch_decode_w<__half, 4, 4>(p, batch, out, s);
  if (p.k_bits == 2)
    return bf ? launch_decode_w<__nv_bfloat16, 2, 2>(p, batch, out, s) : launch_decode_w<__half, 2, 2>(p, batch, out, s);
  return bf ? launch_decode_w<__nv_bfloat16, 4, 2>(p, batch, out, s) : launch_decode_w<__half, 4, 2>(p, batch, out, s);
}

// ---- fixed-scratch variant of the packed decode (no allocation anywhere)
//
// The split-K partials normally live in a caller-provided workspace.  Some
// callers cannot hand one over: an inference engine whose memory manager has
// already claimed the free device memory for its paged cache and forbids
// ad-hoc allocations, or a latency-critical decode loop where cudaMalloc /
// cudaFree would synchronise the device.  For them the partials go into this
// file-scope device array instead.  Every device that loads the library holds
// it until the process exits.  In host code `g_decode_scratch` only names a
// host-side stand-in, so its device address is looked up per device.
static __device__ __align__(256) unsigned char g_decode_scratch[KVARN_NOALLOC_SCRATCH_BYTES];

// Device address of g_decode_scratch on the current device, looked up once
// per device (on the first call that runs with that device current).
static cudaError_t scratch_address(float** out) {
  static std::atomic<void*> addr[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = addr[dev].load(std::memory_order_acquire);
  if (!p) {
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    addr[dev].store(p, std::memory_order_release);
  }
  *out = static_cast<float*>(p);
  return cudaSuccess;
}

cudaError_t launch_decode_noalloc(DecodeParams p, int dtype, int batch, float* out, cudaStream_t s) {
  float* ws = nullptr;
  cudaError_t e = scratch_address(&ws);
  if (e != cudaSuccess) return e;
  p.ws = ws;
  p.ws_bytes = KVARN_NOALLOC_SCRATCH_BYTES;
  return launch_decode(p, dtype, batch, out, s);
}

// The driver's tensor-map encoder, looked up once (a function-local static
// with an initialiser is initialised exactly once, even under concurrent
// first calls).
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    return nullptr;
  }();
  return fn;
}

template <typename E>
static cudaError_t launch_f16_t(DecodeParams p, const void* pool16, int batch, float* out, cudaStream_t s) {
  auto encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)p.num_blocks * p.num_kv_heads * 2 * T};
  const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)T};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(&tmap, std::is_same_v<E, __half> ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      2, const_cast<void*>(pool16), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const size_t smem = sizeof(F16Smem) + 1024;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = smem_attr_once(attr_done, (const void*)decode_f16_kernel<E>, (int)smem);
  if (e != cudaSuccess) return e;
  decode_f16_kernel<E><<<dim3(p.n_chunks, p.num_kv_heads, batch), 256, smem, s>>>(tmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int warps = batch * p.num_q_heads;
  return launch_after(combine_kernel, dim3((warps + 3) / 4), dim3(128), s, p, 0, batch, out);
}

cudaError_t launch_decode_f16(const DecodeParams& p, const void* pool16, int dtype, int batch, float* out,
                              cudaStream_t s) {
  return dtype == KVARN_DTYPE_BF16 ? launch_f16_t<__nv_bfloat16>(p, pool16, batch, out, s)
                                   : launch_f16_t<__half>(p, pool16, batch, out, s);
}

}  // namespace kvarn
