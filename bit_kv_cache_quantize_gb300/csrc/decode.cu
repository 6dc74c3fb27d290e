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
__device__ __forceinline__ uint32_t nib2(uint32_t w, int s) { return unbias(((w >> (4 * s)) & 0x000F000Fu) | 0x64006400u); }
__device__ __forceinline__ uint32_t crumb2(uint32_t w, int s) { return unbias(((w >> (2 * s)) & 0x00030003u) | 0x64006400u); }


template <typename E>
__device__ __forceinline__ float to_f(E x) {
  if constexpr (std::is_same_v<E, __half>) return __half2float(x);
  else return __bfloat162float(x);
}

// Shared memory of one packed-decode CTA: per warp one K-record buffer and
// one V-record buffer -- the next tile's K record streams in while this
// tile's V record is in use and vice versa -- the rotated queries, and the
// cross-warp merge area (aliases the record buffers at the end).
constexpr int DEC_WARPS = 8;
#ifndef KVARN_QK_ILP
#define KVARN_QK_ILP 1
#endif
#ifndef KVARN_PV_ILP
#define KVARN_PV_ILP 4
#endif
constexpr int QK_ILP = KVARN_QK_ILP;  // independent MMA chains interleaved in QK
constexpr int PV_ILP = KVARN_PV_ILP;  // and in PV
constexpr int QR_STRIDE = D + 4;  // padded query rows: lanes g, g+1 hit different banks
// The K codes (128 tokens x 64 B) arrive by a 2-D TMA load of 64 rows of
// 128 B (two tokens per row) with the 128-byte swizzle: 16-byte chunk c of
// row r lands at chunk c ^ (r & 7).  Tokens t and t + 8, which lanes g and
// g + 1 read together, then sit in different banks.
struct DecSmem {
  alignas(1024) unsigned char kcodes[DEC_WARPS][T * D / 2];
  alignas(128) unsigned char khdr[DEC_WARPS][512];
  alignas(128) unsigned char vbuf[DEC_WARPS][V_REC];
  alignas(16) float qr[8][QR_STRIDE];
  uint64_t kbar[DEC_WARPS];
  uint64_t vbar[DEC_WARPS];
};
struct DecMerge {
  float m[DEC_WARPS][8];
  float l[DEC_WARPS][8];
  float acc[DEC_WARPS][8][D];
};
static_assert(sizeof(DecMerge) <= sizeof(DecSmem::kcodes), "merge area must fit");

// Byte offset, inside a warp's swizzled K-code buffer, of the 16 bytes of
// token t's codes for channels 32j .. 32j+31.
__device__ __forceinline__ int kcode_off(int t, int j) {
  const int row = t >> 1, chunk = ((t & 1) << 2) | j;
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

template <typename E>
__device__ void tail_chunk(const DecodeParams& p, int b, int h, int len, unsigned char* smem);

// Unpacking codes to exact fp16 operands.  A code field ORed into the
// mantissa of 1024.0 (0x6400) and 1024 subtracted gives the code exactly.
// Fields at mantissa bits 0-3 / 4-7 of each 16-bit half are taken without a
// shift; a field at bit offset 4 (nibble) or 2k (crumb) comes out multiplied
// by 16 or 4^k, and the matching entries of the other operand are divided by
// the same power of two, which is exact.
__device__ __forceinline__ uint32_t field(uint32_t x, uint32_t mask) { return unbias((x & mask) | MAGIC); }

// grid (n_chunks + 1, H_kv, B) x 256 threads; chunk n_chunks handles the
// raw open tile.  Warp w of a chunk takes its tiles first + w, first + w + 8.
template <typename E>
__global__ void __launch_bounds__(256, 2) decode_packed_kernel(const __grid_constant__ CUtensorMap kmap, DecodeParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
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
  DecSmem& sm = *reinterpret_cast<DecSmem*>(smem_raw + (((sbase + 1023u) & ~1023u) - sbase));
  const int G = p.G;
  const int32_t* tab = p.block_table + (int64_t)b * p.max_blocks;
  const int my_n = (n_tiles > warp) ? (n_tiles - warp + DEC_WARPS - 1) / DEC_WARPS : 0;

  // start this warp's first tile before anything else
  if (lane == 0) {
    mbar_init(&sm.kbar[warp], 1);
    mbar_init(&sm.vbar[warp], 1);
    fence_mbar_init();
  }
  __syncwarp();
  auto issue = [&](int k, bool is_v) {  // lane 0: copy the K or V record of this warp's k-th tile
    const int32_t blk = tab[first + warp + k * DEC_WARPS];
    uint64_t* bar = is_v ? &sm.vbar[warp] : &sm.kbar[warp];
    if (blk >= 0 && blk < p.num_blocks) {
      const int64_t rec = blk * p.block_bytes + (int64_t)h * HEAD_REC;
      if (is_v) {
        mbar_expect_tx(bar, V_REC);
        bulk_g2s(sm.vbuf[warp], p.pool + rec + K_REC, V_REC, bar);
      } else {
        mbar_expect_tx(bar, K_REC);
        bulk_g2s(sm.khdr[warp], p.pool + rec, 512, bar);
        tma_load_2d(sm.kcodes[warp], &kmap, 0, (int)((rec + 512) >> 7), bar);
      }
    } else {
      set_error(p.err, KVARN_DEV_ERR_BLOCK_RANGE);
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
    }
  };
  if (lane == 0 && my_n > 0) { issue(0, false); issue(0, true); }

  // rotated, scaled queries: warp w < G rotates query w with a 128-point
  // butterfly over 4 channels per lane; qr = scale * log2(e) * (q H)
  {
    const E* qb = static_cast<const E*>(p.q) + ((int64_t)b * p.num_q_heads + (int64_t)h * G) * D;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (warp < G) {
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = to_f(qb[warp * D + 4 * lane + e]);
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
    *reinterpret_cast<float4*>(&sm.qr[warp][4 * lane]) = make_float4(x[0] * f, x[1] * f, x[2] * f, x[3] * f);
  }
  __syncthreads();

  float m_run = -INFINITY, l_run = 0.f;
  float acc[16][2];
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) acc[nb][0] = acc[nb][1] = 0.f;

  for (int k = 0; k < my_n; ++k) {
    const int32_t blk = tab[first + warp + k * DEC_WARPS];
    const bool valid = blk >= 0 && blk < p.num_blocks;
    const unsigned char* krec = sm.khdr[warp];
    const unsigned char* kcodes = sm.kcodes[warp];
    const unsigned char* vrec = sm.vbuf[warp];
    // a wait that gives up ends this warp's loop (after waiting, bounded, for
    // the V copy it still has in flight); the error word is already set
    if (__any_sync(0xffffffffu, !mbar_wait_bounded(&sm.kbar[warp], k & 1, p.err))) {
      mbar_wait_bounded(&sm.vbar[warp], k & 1, p.err);
      break;
    }
    const bool kok = valid;

    // ---- query fold: qg = q' * gK over channels 32j..32j+31, scaled so max |qg| is in [512, 1024)
    uint32_t afr[8][4];
    float S = 0.f, qs_inv = 1.f;
    float sc[16][2];
    float tmax = -INFINITY;
    if (kok) {
      float qg[32];
      const uint4 g0 = *reinterpret_cast<const uint4*>(krec + 32 * j);
      const uint4 g1 = *reinterpret_cast<const uint4*>(krec + 32 * j + 16);
      const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      const float* q = &sm.qr[g][32 * j];
      float amax = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float4 qv = *reinterpret_cast<const float4*>(q + 4 * w);
        const float2 lo = e4m3x2_to_float2((uint16_t)(gw[w] & 0xFFFF));
        const float2 hi = e4m3x2_to_float2((uint16_t)(gw[w] >> 16));
        qg[4 * w] = qv.x * lo.x; qg[4 * w + 1] = qv.y * lo.y;
        qg[4 * w + 2] = qv.z * hi.x; qg[4 * w + 3] = qv.w * hi.y;
#pragma unroll
        for (int e = 0; e < 4; ++e) { S += qg[4 * w + e]; amax = fmaxf(amax, fabsf(qg[4 * w + e])); }
      }
      S = quad_sum(S);
      amax = quad_max(amax);
      int ex = 0;
      if (amax > 0.f) frexpf(amax, &ex);
      const float qs = ldexpf(1.f, 10 - ex), qs16 = ldexpf(1.f, 6 - ex);
      qs_inv = ldexpf(1.f, ex - 10);
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        const int c0 = 8 * (kb >> 1) + 2 * (kb & 1);  // b0: channels c0, c0+4 (x1); b1: c0+1, c0+5 (x16)
        uint16_t h00, l00, h01, l01, h10, l10, h11, l11;
        split_hl<__half>(qg[c0] * qs, h00, l00);
        split_hl<__half>(qg[c0 + 4] * qs, h01, l01);
        split_hl<__half>(qg[c0 + 1] * qs16, h10, l10);
        split_hl<__half>(qg[c0 + 5] * qs16, h11, l11);
        afr[kb][0] = pack2(h00, h01);
        afr[kb][1] = pack2(l00, l01);
        afr[kb][2] = pack2(h10, h11);
        afr[kb][3] = pack2(l10, l11);
      }

      // ---- QK: n-block nb holds tokens off(nb), off(nb) + 8 of this lane's 32
      // (off = nb for nb < 8, nb + 8 otherwise); B rows = K codes of token
      // 32 (g >> 1) + off(nb) + 8 (g & 1), channels 32j .. 32j+31
      const __half* bz = reinterpret_cast<const __half*>(krec + 256) + 32 * j;
      const unsigned char* az = krec + 128 + 32 * j;
#pragma unroll
      for (int n4 = 0; n4 < 16; n4 += QK_ILP) {
        uint32_t kw[QK_ILP][4];
#pragma unroll
        for (int i = 0; i < QK_ILP; ++i) {
          const int nb = n4 + i;
          const int off = nb < 8 ? nb : nb + 8;
          const uint4 v4 = *reinterpret_cast<const uint4*>(kcodes + kcode_off(32 * (g >> 1) + off + 8 * (g & 1), j));
          kw[i][0] = v4.x; kw[i][1] = v4.y; kw[i][2] = v4.z; kw[i][3] = v4.w;
        }
        float c[QK_ILP][4];
#pragma unroll
        for (int i = 0; i < QK_ILP; ++i) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
#pragma unroll
          for (int i = 0; i < QK_ILP; ++i) {
            const uint32_t x = (kb & 1) ? (kw[i][kb >> 1] >> 8) : kw[i][kb >> 1];
            mma_f16(c[i], afr[kb], field(x, 0x000F000Fu), field(x, 0x00F000F0u));
          }
        }
#pragma unroll
        for (int i = 0; i < QK_ILP; ++i) {
          const int nb = n4 + i;
          const int off = nb < 8 ? nb : nb + 8;
          const float2 dot = fmul2(fadd2(make_float2(c[i][0], c[i][1]), make_float2(c[i][2], c[i][3])),
                                   make_float2(qs_inv, qs_inv));
          const float2 a = make_float2(e4m3_to_float(az[off]), e4m3_to_float(az[off + 8]));
          const float2 bb = make_float2(__half2float(bz[off]), __half2float(bz[off + 8]));
          const float2 s2 = ffma2(a, dot, fmul2(bb, make_float2(S, S)));
          sc[nb][0] = s2.x; sc[nb][1] = s2.y;
          tmax = fmaxf(tmax, fmaxf(s2.x, s2.y));
        }
      }
    }
    __syncwarp();
    if (lane == 0 && k + 1 < my_n) {  // this K buffer is free: fetch the next tile's K
      fence_proxy_async();
      issue(k + 1, false);
    }
    if (__any_sync(0xffffffffu, !mbar_wait_bounded(&sm.vbar[warp], k & 1, p.err))) {
      if (k + 1 < my_n) mbar_wait_bounded(&sm.kbar[warp], (k + 1) & 1, p.err);
      break;
    }
    const bool vok = kok;
    if (vok) {
      // ---- online softmax (log2 domain)
      tmax = quad_max(tmax);
      const float m_new = fmaxf(m_run, tmax);
      const float corr = exp2f(m_run - m_new);
      m_run = m_new;
      // ---- P = p * aV * 64 / slot scale, hi rows 0-7 / lo rows 8-15
      uint32_t pfr[8][4];
      float2 psum = make_float2(0.f, 0.f), pb = psum;
      const __half* bz = reinterpret_cast<const __half*>(vrec + 256) + 32 * j;
      const unsigned char* az = vrec + 128 + 32 * j;
#pragma unroll
      for (int nb = 0; nb < 16; ++nb) {
        const int off = nb < 8 ? nb : nb + 8;
        const float2 pr = make_float2(exp2f(sc[nb][0] - m_new), exp2f(sc[nb][1] - m_new));
        psum = fadd2(psum, pr);
        pb = ffma2(pr, make_float2(__half2float(bz[off]), __half2float(bz[off + 8])), pb);
        const float f = 64.f / (float)(1 << (2 * (nb & 3)));  // undo the slot scale of this pair
        const float2 pa = fmul2(pr, make_float2(e4m3_to_float(az[off]) * f, e4m3_to_float(az[off + 8]) * f));
        const __half2 hi = __floats2half2_rn(pa.x, pa.y);
        const float2 hf = __half22float2(hi);
        const __half2 lo = __floats2half2_rn(pa.x - hf.x, pa.y - hf.y);
        const uint32_t hb = *reinterpret_cast<const uint32_t*>(&hi), lb = *reinterpret_cast<const uint32_t*>(&lo);
        pfr[nb >> 1][(nb & 1) ? 2 : 0] = hb;
        pfr[nb >> 1][(nb & 1) ? 3 : 1] = lb;
      }
      const float ps = quad_sum(psum.x + psum.y);
      const float pbs = quad_sum(pb.x + pb.y);
      l_run = l_run * corr + ps;
      // ---- PV: B = 2-bit V codes of channel 8nb + g, tokens 32j .. 32j+31
#pragma unroll
      for (int n4 = 0; n4 < 16; n4 += PV_ILP) {
        uint32_t vw[PV_ILP][2];
#pragma unroll
        for (int i = 0; i < PV_ILP; ++i) {
          const uint2 v2 = *reinterpret_cast<const uint2*>(vrec + 512 + (8 * (n4 + i) + g) * 32 + 8 * j);
          vw[i][0] = v2.x; vw[i][1] = v2.y;
        }
        float c[PV_ILP][4];
#pragma unroll
        for (int i = 0; i < PV_ILP; ++i) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          // pairs 2kb, 2kb+1 = crumb fields s, s+1 (s = 2kb & 7) of word kb >> 2
          const int sh = (2 * kb) & 7;
#pragma unroll
          for (int i = 0; i < PV_ILP; ++i) {
            const uint32_t x = (sh & 4) ? (vw[i][kb >> 2] >> 8) : vw[i][kb >> 2];
            const uint32_t m0 = 0x00030003u << (2 * (sh & 3));
            mma_f16(c[i], pfr[kb], field(x, m0), field(x, m0 << 2));
          }
        }
#pragma unroll
        for (int i = 0; i < PV_ILP; ++i) {
          const int nb = n4 + i;
          const float2 gv = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(vrec + 8 * nb + 2 * j));
          const float o0 = fmaf(c[i][0] + c[i][2], 1.f / 64.f, pbs);
          const float o1 = fmaf(c[i][1] + c[i][3], 1.f / 64.f, pbs);
          acc[nb][0] = fmaf(acc[nb][0], corr, gv.x * o0);
          acc[nb][1] = fmaf(acc[nb][1], corr, gv.y * o1);
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
  DecMerge& mg = *reinterpret_cast<DecMerge*>(sm.kcodes);
  if (j == 0) { mg.m[warp][g] = m_run; mg.l[warp][g] = l_run; }
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) {
    mg.acc[warp][g][8 * nb + 2 * j] = acc[nb][0];
    mg.acc[warp][g][8 * nb + 2 * j + 1] = acc[nb][1];
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += 256) {
    const int gg = i / D, c = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) M = fmaxf(M, mg.m[w][gg]);
    float Lsum = 0.f, A = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < DEC_WARPS; ++w) {
        const float f = exp2f(mg.m[w][gg] - M);
        Lsum += f * mg.l[w][gg];
        A += f * mg.acc[w][gg][c];
      }
    }
    float* o = part_ptr(p, b, h, chunk, gg);
    if (c == 0) { o[0] = M; o[1] = Lsum; }
    o[PACC + c] = A;
  }
}

// ------------------------------------------------------------------ tcgen05 decode
// One CTA of 128 threads per (sequence, KV head, chunk of tiles).  Per tile:
//   QK: thread t unpacks token t's 4-bit K codes (scaled by its step a_t,
//       exactly, in the same fp16 FMA that removes the 1024 bias) into tensor
//       memory lane t; the MMA  D1[t][n] = sum_c A_K[t][c] B_q[c][n]  with
//       B_q = qg hi | lo (n = 0..7 | 8..15) from shared memory gives a_t <qg, code_t>.
//       A second MMA against an all-ones A gives S = sum_c qg_c for every row.
//   PV: thread c unpacks channel c's 2-bit V codes into lane c; the MMA
//       D2[c][n] = sum_t A_V[c][t] B_P[t][n]  with B_P = p_t aV_t (hi | lo) gives
//       the packed part of the output; an all-ones MMA over B_Pb = p_t bV_t
//       gives sum_t p_t bV_t.
// The only CTA-wide reduction per tile is the running maximum of the scores.
constexpr int TCW = 4;                    // warps per CTA
constexpr uint32_t TC_COLS = 128;         // tensor-memory columns per CTA
constexpr uint32_t TC_A = 0;              // A operand: 64 columns = 128 fp16
constexpr uint32_t TC_D1 = 64, TC_DS = 80, TC_D2 = 96, TC_DPB = 112;
constexpr uint32_t TC_IDESC = umma_idesc_f16(128, 16, 1);

struct TcSmem {
  alignas(128) unsigned char rec[2][HEAD_REC];  // two stages of one (tile, head) K+V record pair
  alignas(128) unsigned char bq[4096];          // B: qg hi|lo, MN-major, K = 128 channels (permuted), N = 16
  alignas(128) unsigned char bp[4096];          // B: p aV 64 / 4^(t & 3) hi|lo, K = 128 tokens (permuted)
  alignas(128) unsigned char bpb[4096];         // B: p bV hi|lo, K = 128 tokens
  alignas(128) unsigned char ones[128];         // one 8 x 8 core matrix of fp16 1.0
  alignas(16) float qr[8][D];                   // rotated, scaled queries
  alignas(16) float red[TCW][8];
  uint64_t rbar[2];
  uint64_t mbar;
  uint32_t tmem;
};

// Byte offset of element (n, k) in an MN-major B operand (K x 16, no
// swizzle): 8 x 8 core matrices, K-groups 256 B apart, N-groups 128 B apart.
__device__ __forceinline__ int bmn_off(int k) { return (k >> 3) * 256 + (k & 7) * 16; }

template <typename E>
__device__ void tail_chunk(const DecodeParams& p, int b, int h, int len, unsigned char* smem);

template <typename E>
__global__ void __launch_bounds__(TCW * 32) decode_tc_kernel(DecodeParams p) {
  extern __shared__ __align__(128) unsigned char smem_tc[];
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int len = p.seq_lens[b];
  if (len < 0 || len > T * p.max_blocks) {
    if (tid == 0 && chunk == 0 && h == 0) set_error(p.err, KVARN_DEV_ERR_TOKEN_RANGE);
    return;
  }
  if (chunk == p.n_chunks) {
    tail_chunk<E>(p, b, h, len, smem_tc);
    return;
  }
  const int first = chunk * p.chunk_tiles;
  const int n_tiles = min(p.chunk_tiles, len / T - first);
  if (n_tiles <= 0) return;
  TcSmem& sm = *reinterpret_cast<TcSmem*>(smem_tc);
  const int G = p.G;
  const int32_t* tab = p.block_table + (int64_t)b * p.max_blocks;

  if (warp == 0) tmem_alloc(&sm.tmem, TC_COLS);
  if (tid == 0) {
    mbar_init(&sm.rbar[0], 1);
    mbar_init(&sm.rbar[1], 1);
    mbar_init(&sm.mbar, 1);
    fence_mbar_init();
  }
  if (tid < 64) reinterpret_cast<uint32_t*>(sm.ones)[tid & 31] = 0x3C003C00u;
  auto issue = [&](int k) {  // thread 0: copy tile k's K+V record pair
    const int s = k & 1;
    const int32_t blk = tab[first + k];
    if (blk >= 0 && blk < p.num_blocks) {
      mbar_expect_tx(&sm.rbar[s], HEAD_REC);
      bulk_g2s(sm.rec[s], p.pool + blk * p.block_bytes + (int64_t)h * HEAD_REC, HEAD_REC, &sm.rbar[s]);
    } else {
      set_error(p.err, KVARN_DEV_ERR_BLOCK_RANGE);
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&sm.rbar[s])) : "memory");
    }
  };
  __syncthreads();
  if (tid == 0) {
    issue(0);
    if (n_tiles > 1) issue(1);
  }

  // rotated queries: warp w rotates queries w and w + 4 (128-point butterfly,
  // 4 channels per lane); then one power-of-two scale for the CTA puts
  // max |q'| in [0.5, 1) so the fp16 hi/lo parts of q' g stay normal
  {
    const E* qb = static_cast<const E*>(p.q) + ((int64_t)b * p.num_q_heads + (int64_t)h * G) * D;
    float amax = 0.f;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int qq = warp + 4 * r;
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
#pragma unroll
      for (int e = 0; e < 4; ++e) { x[e] *= f; amax = fmaxf(amax, fabsf(x[e])); }
      *reinterpret_cast<float4*>(&sm.qr[qq][4 * lane]) = make_float4(x[0], x[1], x[2], x[3]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) sm.red[warp][0] = amax;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);  // this thread's lane
  float qscale, qscale_inv;
  {
    float amax = fmaxf(fmaxf(sm.red[0][0], sm.red[1][0]), fmaxf(sm.red[2][0], sm.red[3][0]));
    int ex = 0;
    if (amax > 0.f) frexpf(amax, &ex);
    qscale = ldexpf(1.f, -ex);
    qscale_inv = ldexpf(1.f, ex);
  }
  // this thread's channel c = tid: its queries (scaled) and its place in B_q
  float qc[8];
#pragma unroll
  for (int qq = 0; qq < 8; ++qq) qc[qq] = sm.qr[qq][tid] * qscale;
  const int c = tid, t = tid;
  const int kq = 8 * (c >> 3) + 2 * (c & 3) + ((c & 7) >> 2);   // K slot of channel c
  const int kp = 16 * (t >> 4) + 2 * (t & 7) + ((t >> 3) & 1);  // K slot of token t
  const float pscale = 64.f / (float)(1 << (2 * (t & 3)));       // undo the 4^k field scale of token t
  const uint64_t ones_desc = umma_desc(smem_u32(sm.ones), 0, 0);
  const uint32_t bq_s = smem_u32(sm.bq), bp_s = smem_u32(sm.bp), bpb_s = smem_u32(sm.bpb);

  float m_run[8], l_run[8], acc[8];
#pragma unroll
  for (int qq = 0; qq < 8; ++qq) { m_run[qq] = -INFINITY; l_run[qq] = 0.f; acc[qq] = 0.f; }
  uint32_t mphase = 0;
  bool dead = false;

  for (int k = 0; k < n_tiles && !dead; ++k) {
    const int s = k & 1;
    const int32_t blk = tab[first + k];
    const bool valid = blk >= 0 && blk < p.num_blocks;
    if (__syncthreads_or(!mbar_wait_bounded(&sm.rbar[s], (k >> 1) & 1, p.err))) { dead = true; break; }
    const unsigned char* krec = sm.rec[s];
    const unsigned char* vrec = krec + K_REC;

    // ---- QK operands: B_q (thread c) and A_K = a_t * codes of token t
    {
      const float g = e4m3_to_float(krec[c]);
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int qq = 0; qq < 8; qq += 2) {
        uint16_t h0, l0, h1, l1;
        split_hl<__half>(qc[qq] * g, h0, l0);
        split_hl<__half>(qc[qq + 1] * g, h1, l1);
        hw[qq >> 1] = pack2(h0, h1);
        lw[qq >> 1] = pack2(l0, l1);
      }
      *reinterpret_cast<uint4*>(sm.bq + bmn_off(kq)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(sm.bq + bmn_off(kq) + 128) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
    {
      const float a = e4m3_to_float(krec[128 + t]);
      const __half2 A1 = __float2half2_rn(a), A16 = __float2half2_rn(a * 0.0625f);
      const __half2 N1 = __float2half2_rn(-1024.f * a), N16 = __float2half2_rn(-64.f * a);
      uint32_t f[64];
      const unsigned char* row = krec + 512 + t * 64;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint4 v4 = *reinterpret_cast<const uint4*>(row + 16 * q4);
        const uint32_t wv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int w = 4 * q4 + e;
          const uint32_t x = wv[e], x8 = x >> 8;
          __half2 y0 = __hfma2(u2h2((x & 0x000F000Fu) | MAGIC), A1, N1);
          __half2 y1 = __hfma2(u2h2((x & 0x00F000F0u) | MAGIC), A16, N16);
          __half2 y2 = __hfma2(u2h2((x8 & 0x000F000Fu) | MAGIC), A1, N1);
          __half2 y3 = __hfma2(u2h2((x8 & 0x00F000F0u) | MAGIC), A16, N16);
          f[4 * w] = h22u(y0); f[4 * w + 1] = h22u(y1); f[4 * w + 2] = h22u(y2); f[4 * w + 3] = h22u(y3);
        }
      }
      tmem_st64(lane_base + TC_A, f);
    }
    tmem_wait_st();
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t bd = umma_desc(bq_s + 512 * kk, 256, 128);
        umma_ts(tmem + TC_D1, tmem + TC_A + 8 * kk, bd, TC_IDESC, kk);
        umma_ss(tmem + TC_DS, ones_desc, bd, TC_IDESC, kk);
      }
      umma_commit(&sm.mbar);
    }
    // ---- meanwhile: V codes of channel c (fields scaled by 4^(s & 3))
    uint32_t fv[64];
    {
      const unsigned char* row = vrec + 512 + c * 32;
      const __half2 M = u2h2(MAGIC);
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {
        const uint4 v4 = *reinterpret_cast<const uint4*>(row + 16 * q2);
        const uint32_t wv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int ww = 4 * q2 + e;
          const uint32_t x = wv[e], x8 = x >> 8;
#pragma unroll
          for (int sh = 0; sh < 4; ++sh) {
            const uint32_t m = 0x00030003u << (2 * sh);
            fv[8 * ww + sh] = h22u(__hsub2(u2h2((x & m) | MAGIC), M));
            fv[8 * ww + 4 + sh] = h22u(__hsub2(u2h2((x8 & m) | MAGIC), M));
          }
        }
      }
    }
    const float bK = __half2float(*reinterpret_cast<const __half*>(krec + 256 + 2 * t));
    const float aV = e4m3_to_float(vrec[128 + t]);
    const float bV = __half2float(*reinterpret_cast<const __half*>(vrec + 256 + 2 * t));
    const float gV = e4m3_to_float(vrec[c]);
    if (__syncthreads_or(!mbar_wait_bounded(&sm.mbar, mphase, p.err))) { dead = true; break; }
    mphase ^= 1;
    tc_fence_after();
    // ---- scores of token t
    float sc[8];
    {
      float d1[16], ds[16];
      tmem_ld16(lane_base + TC_D1, d1);
      tmem_ld16(lane_base + TC_DS, ds);
      tmem_wait_ld();
#pragma unroll
      for (int qq = 0; qq < 8; ++qq) sc[qq] = qscale_inv * fmaf(bK, ds[qq] + ds[8 + qq], d1[qq] + d1[8 + qq]);
    }
    tmem_st64(lane_base + TC_A, fv);  // QK is done with the A columns
    // ---- tile maximum of each query: reduce-scatter in the warp, then across warps
    {
      const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
      float r4[4], r2[2], r1;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float keep = b4 ? sc[i + 4] : sc[i], send = b4 ? sc[i] : sc[i + 4];
        r4[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 16));
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float keep = b3 ? r4[i + 2] : r4[i], send = b3 ? r4[i] : r4[i + 2];
        r2[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 8));
      }
      {
        const float keep = b2 ? r2[1] : r2[0], send = b2 ? r2[0] : r2[1];
        r1 = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 4));
      }
      r1 = fmaxf(r1, __shfl_xor_sync(0xffffffffu, r1, 2));
      r1 = fmaxf(r1, __shfl_xor_sync(0xffffffffu, r1, 1));
      if ((lane & 3) == 0) sm.red[warp][(b4 ? 4 : 0) + (b3 ? 2 : 0) + (b2 ? 1 : 0)] = r1;
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    float corr[8];
    {
      const float4 r00 = *reinterpret_cast<const float4*>(&sm.red[0][0]), r01 = *reinterpret_cast<const float4*>(&sm.red[0][4]);
      const float4 r10 = *reinterpret_cast<const float4*>(&sm.red[1][0]), r11 = *reinterpret_cast<const float4*>(&sm.red[1][4]);
      const float4 r20 = *reinterpret_cast<const float4*>(&sm.red[2][0]), r21 = *reinterpret_cast<const float4*>(&sm.red[2][4]);
      const float4 r30 = *reinterpret_cast<const float4*>(&sm.red[3][0]), r31 = *reinterpret_cast<const float4*>(&sm.red[3][4]);
      const float tm[8] = {fmaxf(fmaxf(r00.x, r10.x), fmaxf(r20.x, r30.x)), fmaxf(fmaxf(r00.y, r10.y), fmaxf(r20.y, r30.y)),
                           fmaxf(fmaxf(r00.z, r10.z), fmaxf(r20.z, r30.z)), fmaxf(fmaxf(r00.w, r10.w), fmaxf(r20.w, r30.w)),
                           fmaxf(fmaxf(r01.x, r11.x), fmaxf(r21.x, r31.x)), fmaxf(fmaxf(r01.y, r11.y), fmaxf(r21.y, r31.y)),
                           fmaxf(fmaxf(r01.z, r11.z), fmaxf(r21.z, r31.z)), fmaxf(fmaxf(r01.w, r11.w), fmaxf(r21.w, r31.w))};
      uint32_t pw[4], plw[4], bw[4], blw[4];
#pragma unroll
      for (int qq = 0; qq < 8; ++qq) {
        const float mn = valid ? fmaxf(m_run[qq], tm[qq]) : m_run[qq];
        corr[qq] = (m_run[qq] == -INFINITY) ? 0.f : exp2f(m_run[qq] - mn);
        m_run[qq] = mn;
        const float pr = valid ? exp2f(sc[qq] - mn) : 0.f;
        l_run[qq] = fmaf(l_run[qq], corr[qq], pr);
        uint16_t ph, pl, bh, bl;
        split_hl<__half>(pr * aV * pscale, ph, pl);
        split_hl<__half>(pr * bV, bh, bl);
        if (qq & 1) {
          pw[qq >> 1] |= (uint32_t)ph << 16; plw[qq >> 1] |= (uint32_t)pl << 16;
          bw[qq >> 1] |= (uint32_t)bh << 16; blw[qq >> 1] |= (uint32_t)bl << 16;
        } else {
          pw[qq >> 1] = ph; plw[qq >> 1] = pl; bw[qq >> 1] = bh; blw[qq >> 1] = bl;
        }
      }
      *reinterpret_cast<uint4*>(sm.bp + bmn_off(kp)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      *reinterpret_cast<uint4*>(sm.bp + bmn_off(kp) + 128) = make_uint4(plw[0], plw[1], plw[2], plw[3]);
      *reinterpret_cast<uint4*>(sm.bpb + bmn_off(t)) = make_uint4(bw[0], bw[1], bw[2], bw[3]);
      *reinterpret_cast<uint4*>(sm.bpb + bmn_off(t) + 128) = make_uint4(blw[0], blw[1], blw[2], blw[3]);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        umma_ts(tmem + TC_D2, tmem + TC_A + 8 * kk, umma_desc(bp_s + 512 * kk, 256, 128), TC_IDESC, kk);
        umma_ss(tmem + TC_DPB, ones_desc, umma_desc(bpb_s + 512 * kk, 256, 128), TC_IDESC, kk);
      }
      umma_commit(&sm.mbar);
      if (k + 2 < n_tiles) {  // every thread is done reading this stage
        fence_proxy_async();
        issue(k + 2);
      }
    }
    if (__syncthreads_or(!mbar_wait_bounded(&sm.mbar, mphase, p.err))) { dead = true; break; }
    mphase ^= 1;
    tc_fence_after();
    {
      float d2[16], dpb[16];
      tmem_ld16(lane_base + TC_D2, d2);
      tmem_ld16(lane_base + TC_DPB, dpb);
      tmem_wait_ld();
#pragma unroll
      for (int qq = 0; qq < 8; ++qq)
        acc[qq] = fmaf(acc[qq], corr[qq], valid ? gV * fmaf(d2[qq] + d2[8 + qq], 1.f / 64.f, dpb[qq] + dpb[8 + qq]) : 0.f);
    }
    tc_fence_before();
  }

  // ---- partial of this CTA: m (uniform), l = sum over threads, acc per channel
#pragma unroll
  for (int qq = 0; qq < 8; ++qq) {
    float v = l_run[qq];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    l_run[qq] = v;
  }
  __syncthreads();
  if (lane == 0) {
#pragma unroll
    for (int qq = 0; qq < 8; ++qq) sm.red[warp][qq] = l_run[qq];
  }
  __syncthreads();
  for (int qq = 0; qq < G; ++qq) {
    float* o = part_ptr(p, b, h, chunk, qq);
    if (tid == 0) {
      o[0] = dead ? -INFINITY : m_run[qq];
      o[1] = dead ? 0.f : sm.red[0][qq] + sm.red[1][qq] + sm.red[2][qq] + sm.red[3][qq];
    }
    o[PACC + c] = dead ? 0.f : acc[qq];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, TC_COLS);
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
    if (tid == 0) { out[0] = ml[2 * gg]; out[1] = ml[2 * gg + 1]; }
    out[PACC + tid] = a[gg];
  }
}

// One warp per (sequence, query head): merge the split-K partials, apply
// the inverse rotation to the packed-tile part, add the raw part, normalise.
__global__ void __launch_bounds__(128) combine_kernel(DecodeParams p, int rotate, int batch, float* __restrict__ out) {
  const int wid = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (wid >= batch * p.num_q_heads) return;
  const int b = wid / p.num_q_heads, hq = wid % p.num_q_heads;
  const int h = hq / p.G, g = hq % p.G;
  const int len = p.seq_lens[b];
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  if (len > 0 && len <= T * p.max_blocks) {
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
  *reinterpret_cast<float4*>(out + ((int64_t)b * p.num_q_heads + hq) * D + 4 * lane) = o;
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

// 2-D view of the packed pool as rows of 128 bytes, read in boxes of 64 rows
// (one tile's K codes) with the 128-byte swizzle.
static cudaError_t pool_tensor_map(const DecodeParams& p, CUtensorMap* m) {
  auto encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {128, (cuuint64_t)p.num_blocks * (cuuint64_t)p.block_bytes / 128};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, 64};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<unsigned char*>(p.pool), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <typename E>
static cudaError_t launch_decode_t(DecodeParams p, int batch, float* out, cudaStream_t s) {
  CUtensorMap kmap;
  cudaError_t e = pool_tensor_map(p, &kmap);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(DecSmem) + 1024;
  e = cudaFuncSetAttribute(decode_packed_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  decode_packed_kernel<E><<<dim3(p.n_chunks + 1, p.num_kv_heads, batch), 256, smem, s>>>(kmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int warps = batch * p.num_q_heads;
  combine_kernel<<<(warps + 3) / 4, 128, 0, s>>>(p, 1, batch, out);
  return cudaGetLastError();
}

template <typename E>
static cudaError_t launch_decode_tc_t(DecodeParams p, int batch, float* out, cudaStream_t s) {
  const size_t smem = sizeof(TcSmem);
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<E><<<dim3(p.n_chunks + 1, p.num_kv_heads, batch), TCW * 32, smem, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int warps = batch * p.num_q_heads;
  combine_kernel<<<(warps + 3) / 4, 128, 0, s>>>(p, 1, batch, out);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, int dtype, int batch, float* out, cudaStream_t s) {
#ifdef KVARN_DECODE_TC
  return dtype == KVARN_DTYPE_BF16 ? launch_decode_tc_t<__nv_bfloat16>(p, batch, out, s)
                                   : launch_decode_tc_t<__half>(p, batch, out, s);
#else
  return dtype == KVARN_DTYPE_BF16 ? launch_decode_t<__nv_bfloat16>(p, batch, out, s)
                                   : launch_decode_t<__half>(p, batch, out, s);
#endif
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
  return launch_decode(p, dtype, batch, out, s);
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
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
  cudaError_t e = cudaFuncSetAttribute(decode_f16_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  decode_f16_kernel<E><<<dim3(p.n_chunks, p.num_kv_heads, batch), 256, smem, s>>>(tmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int warps = batch * p.num_q_heads;
  combine_kernel<<<(warps + 3) / 4, 128, 0, s>>>(p, 0, batch, out);
  return cudaGetLastError();
}

cudaError_t launch_decode_f16(const DecodeParams& p, const void* pool16, int dtype, int batch, float* out,
                              cudaStream_t s) {
  return dtype == KVARN_DTYPE_BF16 ? launch_f16_t<__nv_bfloat16>(p, pool16, batch, out, s)
                                   : launch_f16_t<__half>(p, pool16, batch, out, s);
}

}  // namespace kvarn
