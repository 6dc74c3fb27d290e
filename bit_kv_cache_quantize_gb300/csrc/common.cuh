// common.cuh -- device helpers shared by the KVarN kernels (sm_103a).
//
// Inline-PTX wrappers for the warp-level tensor-core MMA (m16n8k16, fp32
// accumulate), ldmatrix, 16-byte cp.async, 1-D bulk copies completed on an
// mbarrier, and the FP8 E4M3 / FP16 conversions the packed format needs.
#pragma once

#include "params.h"
#include <atomic>
#include <cstdint>
#include <type_traits>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "../../include/kvarn.h"

namespace kvarn {

constexpr int D = 128;               // channels per token (head_dim)
constexpr int T = 128;               // tokens per tile (one paged block)
constexpr int K_REC = rec_bytes(4);  // 4-bit keys (kvarn_k4v2 preset): 8704 B
constexpr int K2_REC = rec_bytes(2); // 2-bit keys (K2/V2 preset): 4608 B
constexpr int V_REC = rec_bytes(2);  // 2-bit values: 4608 B
constexpr int V4_REC = rec_bytes(4); // 4-bit values (K4/V4 preset): 8704 B
constexpr int HEAD_REC_MAX = K_REC + V4_REC;  // largest (tile, head) pair of records
constexpr float INV_SQRT_D = 0.08838834764831845f;  // 1/sqrt(128)

// First error wins; the failing unit skips its work.  Never traps, never waits.
__device__ __forceinline__ void set_error(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

// Programmatic dependent launch.  A split-K combine is launched with
// launch_after() so that the GPU may schedule it while the kernel ahead of it
// in the stream is still running, once every CTA of that kernel has called
// allow_dependents(); its threads then block in wait_prerequisite() until the
// kernel ahead has completed and its memory is visible.  For a kernel
// launched the ordinary way wait_prerequisite() returns at once.
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void wait_prerequisite() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

template <typename... Params, typename... Args>
static cudaError_t launch_after(void (*kernel)(Params...), dim3 grid, dim3 block, cudaStream_t s, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Bounds check of the checked (debug) build, compiled with KVARN_CHECK: an
// access of n bytes at p must lie inside [base, base + bytes); otherwise the
// first error is recorded as KVARN_DEV_ERR_BOUNDS and the caller skips the
// access.  In the normal build it is the constant true and compiles away.
__device__ __forceinline__ bool kcheck(const void* p, size_t n, const void* base, size_t bytes, int32_t* err) {
#ifdef KVARN_CHECK
  const char* a = static_cast<const char*>(p);
  const char* lo = static_cast<const char*>(base);
  if (a >= lo && n <= bytes && static_cast<size_t>(a - lo) <= bytes - n) return true;
  set_error(err, KVARN_DEV_ERR_BOUNDS);
  return false;
#else
  (void)p; (void)n; (void)base; (void)bytes; (void)err;
  return true;
#endif
}

// ------------------------------------------------------------------ MMA
// Bits of +1.0 in the 16-bit element type E.
template <typename E> struct Bits16;
template <> struct Bits16<__half> { static constexpr uint32_t one = 0x3C00u; };
template <> struct Bits16<__nv_bfloat16> { static constexpr uint32_t one = 0x3F80u; };

__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <typename E>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (std::is_same_v<E, __half>) mma_f16(c, a, b0, b1);
  else mma_bf16(c, a, b0, b1);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// ------------------------------------------------------------------ copies
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::);
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes));
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem, const void* gmem, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(smem)),
      "l"(gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// The same copy for data read once (the decode's record stream): the L2
// lines it brings in are the first evicted, which keeps the split-K
// partials and the other small buffers of the step resident.
__device__ __forceinline__ void bulk_g2s_stream(void* smem, const void* gmem, uint32_t bytes, uint64_t* bar) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(
          smem_u32(smem)),
      "l"(gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// 2-D tiled TMA load global -> shared (box and swizzle from the tensor map),
// completion counted on an mbarrier.  x * element size must be a multiple of
// 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* smem, const void* tmap, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          smem_u32(smem)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: false (and the error word set) if the phase has not
// completed after `polls` polls (each poll may itself wait a short,
// hardware-defined time).
constexpr int kWaitPolls = 1 << 22;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int32_t* err,
                                                  int polls = kWaitPolls) {
  for (int i = 0; i < polls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  set_error(err, KVARN_DEV_ERR_TIMEOUT);
  return false;
}

// Bounded wait in which the hardware may park the thread until the phase
// completes (try_wait with a suspend-time hint of 0.2 ms) instead of
// re-polling; false (and the error word set) after about 2 s.
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool mbar_wait_parked(uint64_t* bar, uint32_t parity, int32_t* err) {
  const uint64_t t0 = global_ns();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(200000u)
        : "memory");
    if (ok) return true;
    if (global_ns() - t0 > 2000000000ull) break;
  }
  set_error(err, KVARN_DEV_ERR_TIMEOUT);
  return false;
}

// 2^x, flushing results below the normal range to zero (PTX ex2.approx.ftz).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ formats
__device__ __forceinline__ float e4m3_to_float(uint8_t b) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
  return __half2float(__half(h));
}

// Two E4M3 bytes (low byte first) -> two floats.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  return __half22float2(__half2(h));
}

// Round to nearest even, saturating to +-448.
__device__ __forceinline__ uint8_t float_to_e4m3_rn(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

// Smallest E4M3 value >= x for x >= 0, saturating at 448 (code 0x7E).
__device__ __forceinline__ uint8_t float_to_e4m3_ru(float x) {
  if (!(x > 0.f)) return 0;
  if (x >= 448.f) return 0x7E;
  uint8_t c = float_to_e4m3_rn(x);
  if (e4m3_to_float(c) < x) ++c;  // the next code is the next value up
  return c;
}

// Packed two-lane fp32 arithmetic (one instruction for two IEEE operations,
// each rounded to nearest even exactly as the scalar forms).
__device__ __forceinline__ unsigned long long f2_bits(float2 a) { return *reinterpret_cast<unsigned long long*>(&a); }
__device__ __forceinline__ float2 bits_f2(unsigned long long b) { return *reinterpret_cast<float2*>(&b); }
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
  return bits_f2(d);
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}

// Reductions over the 4 lanes of a quad (lanes 4k .. 4k+3).
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}
__device__ __forceinline__ float quad_min(float x) {
  x = fminf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fminf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}
__device__ __forceinline__ float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}

// fp32 -> 16-bit bits of E, round to nearest even.
template <typename E>
__device__ __forceinline__ uint16_t f2bits(float x) {
  if constexpr (std::is_same_v<E, __half>) return __half_as_ushort(__float2half_rn(x));
  else return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
template <typename E>
__device__ __forceinline__ float bits2f(uint16_t b) {
  if constexpr (std::is_same_v<E, __half>) return __half2float(__ushort_as_half(b));
  else return __bfloat162float(__ushort_as_bfloat16(b));
}
// x -> (hi, lo) in E with hi + lo = x to within E's precision squared.
template <typename E>
__device__ __forceinline__ void split_hl(float x, uint16_t& hi, uint16_t& lo) {
  hi = f2bits<E>(x);
  lo = f2bits<E>(x - bits2f<E>(hi));
}
__device__ __forceinline__ uint32_t pack2(uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); }

// ------------------------------------------------------------------ host
// Raises the dynamic shared memory limit of one kernel to `bytes`, once per
// device: `done` (one static per kernel instance at the call site) keeps a
// bit per device whose attribute is already set, so the decode-step path
// makes no attribute call after the first launch.
inline cudaError_t smem_attr_once(std::atomic<uint64_t>& done, const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

}  // namespace kvarn
