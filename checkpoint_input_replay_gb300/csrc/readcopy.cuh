// Low-precision read copy of one state matrix, written from the folded FP32
// matrix held in shared memory.  The copy serves only the checkpoint read of
// later non-flush steps; the FP32 checkpoint stays the recurrence's state
// ("ReplaySSM caches SSM inputs instead of state" (richland.au), "What
// shipped", the paragraph on quantization).
//
// FP8 per-row:  scale = amax(row) / 448, code = e4m3(x / scale).
// NVFP4:        s = amax(matrix) / (448 * 6); per 16-element block along N a
//               block scale e4m3(amax_blk / (6 s)); code = e2m1(x / (bs * s)),
//               element 2i in the low nibble of byte i.
// Scales and scaled values are float32 with IEEE round-to-nearest division
// (__fdiv_rn), element codes from the hardware cvt (round to nearest even,
// saturating); a zero divisor gives zero codes.
#pragma once

#include "common.cuh"

namespace rs {

// sT: folded matrix [P][N] f32 in shared memory; sred: kThreads/32 floats.
// Called by the kThreads computing threads (threads 0..kThreads-1) of the CTA.
template <int N, int READ>
__device__ __forceinline__ void write_read_copy(const LayerDev& d, int bh, const float* sT, float* sred) {
  constexpr int SEG = N / 4;
  const int P = d.P;
  const int t = threadIdx.x;
  const int c4 = t % SEG;
  const int nf4 = P * N / 4;
  const float4* sT4 = reinterpret_cast<const float4*>(sT);
  if (READ == READ_FP8) {
    uint32_t* codes = reinterpret_cast<uint32_t*>(d.rc_codes + static_cast<size_t>(bh) * P * N);
    float* rowscale = d.rc_rowscale + static_cast<size_t>(bh) * P;
    for (int f = t; f < nf4; f += kThreads) {
      const float4 v = sT4[f];
      float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
      m = seg_max<SEG>(m);
      const float scale = __fdiv_rn(m, 448.0f);
      uint32_t packed = 0;
      if (scale != 0.0f) {
        const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(v.x, scale), __fdiv_rn(v.y, scale));
        const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(v.z, scale), __fdiv_rn(v.w, scale));
        packed = lo | (hi << 16);
      }
      codes[f] = packed;
      if (c4 == 0) rowscale[f / SEG] = scale;
    }
  } else if (READ == READ_NVFP4) {
    // matrix amax
    float m = 0.0f;
    for (int f = t; f < nf4; f += kThreads) {
      const float4 v = sT4[f];
      m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    m = seg_max<32>(m);
    if ((t & 31) == 0) sred[t >> 5] = m;
    compute_sync();
    float amax = 0.0f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) amax = fmaxf(amax, sred[w]);
    const float s = __fdiv_rn(amax, 2688.0f);  // 448 * 6
    const float six_s = __fmul_rn(6.0f, s);
    uint16_t* codes = reinterpret_cast<uint16_t*>(d.rc_codes + static_cast<size_t>(bh) * P * (N / 2));
    uint8_t* blk = d.rc_blkscale + static_cast<size_t>(bh) * P * (N / 16);
    for (int f = t; f < nf4; f += kThreads) {
      const float4 v = sT4[f];
      float mb = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
      mb = seg_max<4>(mb);  // 4 lanes = one 16-element block
      uint32_t bcode = 0;
      if (six_s != 0.0f) bcode = f32x2_to_e4m3x2(__fdiv_rn(mb, six_s), 0.0f) & 0xFFu;
      const float dd = __fmul_rn(e4m3_to_f32(bcode), s);
      uint32_t q = 0;
      if (dd != 0.0f)
        q = f32x4_to_e2m1x4(__fdiv_rn(v.x, dd), __fdiv_rn(v.y, dd), __fdiv_rn(v.z, dd), __fdiv_rn(v.w, dd));
      codes[f] = static_cast<uint16_t>(q);
      if ((c4 & 3) == 0) blk[f / 4] = static_cast<uint8_t>(bcode);
    }
    if (t == 0) d.rc_matscale[bh] = s;
  }
}

}  // namespace rs
