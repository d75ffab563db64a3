// Device helpers shared by the hot-path kernels: bf16 widening, segmented
// warp reductions, mbarrier + bulk-copy staging with bounded waits, the
// sticky error word, the per-sequence arrival counter, and the e4m3 / e2m1
// conversions of the read copy.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace rs {

__device__ __forceinline__ float bf(uint16_t v) { return __uint_as_float(static_cast<uint32_t>(v) << 16); }

// 8 bf16 packed in a uint4 -> 8 floats
__device__ __forceinline__ void bf8(const uint4 raw, float out[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[2 * i] = __uint_as_float(w[i] << 16);
    out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// 4 bf16 packed in a uint2 -> float4
__device__ __forceinline__ float4 bf4(const uint2 raw) {
  return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                     __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
}

// Sum over aligned groups of SEG lanes (SEG a power of two <= 32); every lane
// of the group receives the total.
template <int SEG>
__device__ __forceinline__ float seg_sum(float v) {
#pragma unroll
  for (int o = SEG / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int SEG>
__device__ __forceinline__ float seg_max(float v) {
#pragma unroll
  for (int o = SEG / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Inclusive suffix sum over lanes 0..last of one value per lane (lanes past
// `last` contribute nothing).
__device__ __forceinline__ float suffix_sum(float v, int lane, int last) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float w = __shfl_down_sync(0xffffffffu, v, o);
    if (lane + o <= last) v += w;
  }
  return v;
}

__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
  return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, a.x * b.x)));
}

__device__ __forceinline__ float4 axpy4(float a, const float4 x, float4 y) {
  y.x = fmaf(a, x.x, y.x);
  y.y = fmaf(a, x.y, y.y);
  y.z = fmaf(a, x.z, y.z);
  y.w = fmaf(a, x.w, y.w);
  return y;
}

// y += a * x with packed two-lane FP32 FMAs (fma.rn.f32x2: two IEEE fmaf)
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float4 axpy4x2(float a, const float4 x, const float4 y) {
  const float2 lo = fma2(make_float2(a, a), make_float2(x.x, x.y), make_float2(y.x, y.y));
  const float2 hi = fma2(make_float2(a, a), make_float2(x.z, x.w), make_float2(y.z, y.w));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// Unit range of this CTA in a persistent launch: blockIdx.x, or the debug
// permutation (c * mult + 7) mod grid when mult > 0 (mult coprime with the grid).
__device__ __forceinline__ int cta_index(int mult) {
  if (mult <= 0) return static_cast<int>(blockIdx.x);
  return static_cast<int>((static_cast<long long>(blockIdx.x) * mult + 7) % gridDim.x);
}

// a . b with two packed FMAs (pairs (x, y) and (z, w)) and one add
__device__ __forceinline__ float dot4p(const float4 a, const float4 b) {
  float2 t = fma2(make_float2(a.x, a.y), make_float2(b.x, b.y), make_float2(0.f, 0.f));
  t = fma2(make_float2(a.z, a.w), make_float2(b.z, b.w), t);
  return t.x + t.y;
}

__device__ __forceinline__ float4 scale4(float a, const float4 x) {
  return make_float4(a * x.x, a * x.y, a * x.z, a * x.w);
}

// Draft sigma lies on the path from the committed records to draft tau (tau
// itself included) in the ancestor mask of a verify (bit 4 tau + sigma).
__device__ __forceinline__ bool on_tree_path(uint32_t anc, int tau, int sigma) {
  return sigma >= 0 && sigma < 4 && tau >= 0 && tau < 4 && ((anc >> (4 * tau + sigma)) & 1u) != 0;
}

// ---- error word and cursor bookkeeping -------------------------------------

__device__ __forceinline__ void report_error(int* err, int code, int seq) {
  if (atomicCAS(err, 0, code) == 0) atomicExch(err + 1, seq);
}

// Thread 0 of a CTA, after all of the CTA's global writes: counts this CTA in
// and returns true for the last of the `nctas` CTAs of sequence b, after
// resetting the counter for the next launch.
__device__ __forceinline__ bool arrive_last(int* arrive, int b, int nctas) {
  __threadfence();
  const int prev = atomicAdd(arrive + b, 1);
  if (prev == nctas - 1) {
    atomicExch(arrive + b, 0);
    return true;
  }
  return false;
}

// ---- barriers among the kThreads computing threads (named barrier 1) ---------
// Kernels with a producer warp keep it out of these.

__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

// Barrier that also returns whether `v` held in every computing thread.
__device__ __forceinline__ bool compute_sync_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kThreads)
      : "memory");
  return r != 0;
}

// ---- mbarrier + bulk copy (cp.async.bulk, the untiled TMA path) -------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Global -> shared bulk copy; dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of the barrier, giving up after about `limit_ns`
// (and at most 2^22 polls).  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = 1000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < (1u << 22); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0 && global_ns() - t0 > limit_ns) break;
  }
  return mbar_try_wait(bar, parity);
}

// ---- e4m3 / e2m1 conversions (hardware cvt: round to nearest even, satfinite)

// (lo, hi) -> two e4m3 codes, lo in bits 0..7
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
  const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
  return __half22float2(hv);
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  return e4m3x2_to_f32x2(static_cast<uint16_t>(code & 0xFFu)).x;
}

// four floats -> four e2m1 codes packed in 16 bits (element i in nibble i)
__device__ __forceinline__ uint32_t f32x4_to_e2m1x4(float a0, float a1, float a2, float a3) {
  uint16_t r;
  asm("{\n\t.reg .b8 q0, q1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "mov.b16 %0, {q0, q1};\n\t}"
      : "=h"(r)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  return r;
}

// two packed e2m1 codes (one byte, element 0 in the low nibble) -> two floats
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t byte) {
  uint32_t h2;
  const uint16_t in16 = static_cast<uint16_t>(byte & 0xFFu);
  asm("{\n\t.reg .b8 q, qz;\n\t"
      "mov.b16 {q, qz}, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, q;\n\t}"
      : "=r"(h2)
      : "h"(in16));
  const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
  return __half22float2(hv);
}

// eight packed e2m1 codes (one word, element 0 in the low nibble) -> eight floats
__device__ __forceinline__ void e2m1x8_to_f32x2(uint32_t word, float2 out[4]) {
  uint32_t h[4];
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "mov.b32 {q0, q1, q2, q3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, q0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, q1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, q2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, q3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(word));
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
}

// the correctly rounded reciprocal of 448 (the FP8 e4m3 maximum), for div_by: an
// FP8 row scale amax / 448 is correctly rounded for every amax above 2^-117
constexpr float kInv448 = 1.0f / 448.0f;

// x / d rounded to nearest for many x over one divisor d, given r = the
// correctly rounded reciprocal of d (__frcp_rn): q = x r is within one ulp of
// x / d, and one fused correction q + (x - q d) r rounds it correctly
// (Markstein's theorem on FMA-based division), away from overflow and
// underflow -- which the read-copy quotients stay clear of wherever a code's
// rounding depends on them (|x / d| <= 448 and codes below 2^-10 are 0).
__device__ __forceinline__ float div_by(float x, float d, float r) {
  const float q = __fmul_rn(x, r);
  return __fmaf_rn(__fmaf_rn(-q, d, x), r, q);
}

// Sum each of v[0..7] over the eight lanes that share lane >> 3 (transpose-reduce:
// 7 shuffles).  Lane L returns the total of v[L & 7] over its eight lanes.
__device__ __forceinline__ float reduce8_lanes3(const float v[8], int lane) {
  const bool b2 = (lane & 4) != 0, b1 = (lane & 2) != 0, b0 = (lane & 1) != 0;
  float w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b2 ? v[i] : v[i + 4];
    const float keep = b2 ? v[i + 4] : v[i];
    w[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  float x[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b1 ? w[i] : w[i + 2];
    const float keep = b1 ? w[i + 2] : w[i];
    x[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  return (b0 ? x[1] : x[0]) + __shfl_xor_sync(0xffffffffu, b0 ? x[0] : x[1], 1);
}

// Maximum of each of v[0..7] over the 32 lanes of the warp (transpose-reduce: 9
// shuffles).  Lane L returns the maximum of v[(L >> 2) & 7].
__device__ __forceinline__ float reduce8_max(const float v[8], int lane) {
  const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
  float w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b4 ? v[i] : v[i + 4];
    const float keep = b4 ? v[i + 4] : v[i];
    w[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
  float x[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b3 ? w[i] : w[i + 2];
    const float keep = b3 ? w[i + 2] : w[i];
    x[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
  float z = fmaxf(b2 ? x[1] : x[0], __shfl_xor_sync(0xffffffffu, b2 ? x[0] : x[1], 4));
  z = fmaxf(z, __shfl_xor_sync(0xffffffffu, z, 2));
  z = fmaxf(z, __shfl_xor_sync(0xffffffffu, z, 1));
  return z;
}

// Sum each of v[0..7] over the 32 lanes of the warp (transpose-reduce: 9
// shuffles).  Lane L returns the total of v[(L >> 2) & 7].
__device__ __forceinline__ float reduce8(const float v[8], int lane) {
  const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
  float w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b4 ? v[i] : v[i + 4];
    const float keep = b4 ? v[i + 4] : v[i];
    w[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
  float x[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b3 ? w[i] : w[i + 2];
    const float keep = b3 ? w[i + 2] : w[i];
    x[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  float z = (b2 ? x[1] : x[0]) + __shfl_xor_sync(0xffffffffu, b2 ? x[0] : x[1], 4);
  z += __shfl_xor_sync(0xffffffffu, z, 2);
  z += __shfl_xor_sync(0xffffffffu, z, 1);
  return z;
}

}  // namespace rs
