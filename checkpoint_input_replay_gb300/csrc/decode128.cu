// Standard decode step for d_state = 128 (every configuration the workloads
// measure): the output-only non-flush body and the flush body, per sequence,
// in one persistent launch.  Same arithmetic as decode.cu (the unrolled
// checkpoint-plus-buffer form of "ReplaySSM caches SSM inputs instead of
// state" (richland.au), "What shipped"); this file differs in how the work is
// fed and split:
//
//  * a work unit is one (sequence, head) state matrix [P][128]; CTA c owns a
//    contiguous range of units, so it meets each group (and sequence) once;
//  * a producer warp stages each unit with two bulk copies (cp.async.bulk):
//    the state matrix (or its read copy) and the buffered records of that
//    head.  Everything the heads of a group share or that is small -- the
//    group's keys and query, the current tokens of all its heads, the ring's
//    per-head decay rows, the current per-head scalars, the read-copy scales --
//    is staged once per group into one of two group buffers;
//  * a prologue warp turns each unit into scalars (key dot products once per
//    group, the decay suffix scan, per-record coefficients) and signals
//    `ready`;
//  * eight computing warps each own rows w, w+8, .. of every unit: lane = 4
//    columns, 4 lanes per row split the buffered records, an 8-row
//    transpose-reduce forms the row sums.  A flush unit folds in registers
//    (register-held coefficients, shuffles, packed fma.rn.f32x2) and stores the
//    checkpoint once.  No barrier spans the warps, except an NVFP4 flush unit,
//    whose matrix amax is exchanged through a bounded mbarrier.
#include "common.cuh"

namespace rs {
namespace {

constexpr int N = 128;               // d_state of this kernel
constexpr int SEG = N / 4;           // lanes per state row (one float4 each)
constexpr int kMaxSeq128 = 64;       // sequences one CTA may cover
constexpr int kThreads128 = kThreads + 64;  // 8 computing warps, prologue warp, producer warp

__host__ __device__ __forceinline__ int al16(int x) { return (x + 15) & ~15; }
__host__ __device__ __forceinline__ int al128(int x) { return (x + 127) & ~127; }

// Shared-memory layout (bytes): [stages][2 group buffers][persistent].
struct Lay128 {
  // stage
  int st_tile, st_rec, st_scal, st_size;
  // group buffer
  int gb_key, gb_q, gb_cur, gb_la, gb_dt, gb_s1, gb_s2, gb_rs, gb_ms, gb_size;
  // persistent
  int pe_A, pe_bars, pe_seq, pe_misc, pe_size;
};

__host__ __device__ __forceinline__ Lay128 lay128(int kind, int read, int P, int C, int Cp, int H, int hpg) {
  Lay128 l;
  int o = 0;
  l.st_tile = o;  o += P * N * 4;
  l.st_rec = o;   o += kind == 0 ? al16(C * P * 2) : C * P * 4;
  l.st_scal = o;  o += al16((3 * C + 2 * P + 8) * 4);
  l.st_size = al128(o);
  o = 0;
  const int span = al16(hpg * 4) + 16;
  l.gb_key = o;   o += C * N * 2;
  l.gb_q = o;     o += N * 2;
  l.gb_cur = o;   o += al16(hpg * P * 2);
  l.gb_la = o;    o += hpg * Cp * 4;
  l.gb_dt = o;    o += kind == 0 ? hpg * Cp * 2 : 0;
  l.gb_s1 = o;    o += span;
  l.gb_s2 = o;    o += kind == 0 ? 0 : span;
  l.gb_rs = o;    o += read == READ_FP8 ? hpg * P * 4 : (read == READ_NVFP4 ? hpg * P * (N / 16) : 0);
  l.gb_ms = o;    o += read == READ_NVFP4 ? span : 0;
  l.gb_size = al128(o);
  o = 0;
  l.pe_A = o;     o += al16(H * 4);
  l.pe_bars = o;  o += 4 * 8 * 8;       // full, empty, ready, amax x 8 stages
  l.pe_seq = o;   o += 3 * kMaxSeq128 * 4;
  l.pe_misc = o;  o += 16;
  l.pe_size = al128(o);
  return l;
}

__device__ __forceinline__ int ring_slot(int head, int j, int C) {
  int s = head + j;
  return s >= C ? s - C : s;
}

struct Unit {
  int u, b, h, g, hh, k, head, n;
  bool ok, flush, first;
};

template <int KIND, int READ>
__global__ void __launch_bounds__(kThreads128, 1) decode128_kernel(const LayerDev d, const TokenIn in,
                                                                   float* __restrict__ y, const int units_per_cta,
                                                                   const int stages) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int P = d.P, H = d.H, G = d.G, C = d.C, L = d.L, Cp = d.Cp;
  const int hpg = H / G;
  const int tile = P * N;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const Lay128 LY = lay128(KIND, READ, P, C, Cp, H, hpg);
  unsigned char* gbase = smem + static_cast<size_t>(LY.st_size) * stages;
  unsigned char* pbase = gbase + 2 * LY.gb_size;
  const float* sA = reinterpret_cast<const float*>(pbase + LY.pe_A);
  uint64_t* full = reinterpret_cast<uint64_t*>(pbase + LY.pe_bars);
  uint64_t* empty = full + 8;
  uint64_t* ready = full + 16;
  uint64_t* amaxbar = full + 24;
  int* sseq = reinterpret_cast<int*>(pbase + LY.pe_seq);
  volatile int* smisc = reinterpret_cast<volatile int*>(pbase + LY.pe_misc);  // abort, issued, producer done

  const int total_units = d.B * H;
  const int u0 = blockIdx.x * units_per_cta;
  const int u1 = min(u0 + units_per_cta, total_units);
  if (u0 >= u1) return;
  const int nunits = u1 - u0;
  const int b0 = u0 / H, b1 = (u1 - 1) / H;
  const int nseq = b1 - b0 + 1;

  // --- cursors of the covered sequences; arrival; new cursors by the last arriver ---
  if (t < nseq) {
    const int b = b0 + t;
    const int head = d.cursor[4 * b], cnt = d.cursor[4 * b + 1];
    const bool ok = static_cast<unsigned>(head) < static_cast<unsigned>(C) &&
                    static_cast<unsigned>(cnt) < static_cast<unsigned>(L);
    sseq[3 * t] = head;
    sseq[3 * t + 1] = cnt;
    sseq[3 * t + 2] = ok ? 1 : 0;
    const int lo = max(u0, b * H), hi = min(u1, (b + 1) * H);
    __threadfence();
    const int prev = atomicAdd(d.arrive + b, hi - lo);
    if (prev + (hi - lo) == H) {  // every CTA of this sequence has read its cursor
      atomicExch(d.arrive + b, 0);
      if (!ok) {
        report_error(d.err, DEVERR_CURSOR, b);
      } else if (cnt + 1 == L) {
        d.cursor[4 * b] = ring_slot(head, cnt + 1, C);
        d.cursor[4 * b + 1] = 0;
        d.cursor[4 * b + 2] = 1;
      } else {
        d.cursor[4 * b + 1] = cnt + 1;
        d.cursor[4 * b + 2] = 0;
      }
    }
  }
  if (t == kThreads) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kThreads / 32);
      mbar_init(ready + s, 1);
      mbar_init(amaxbar + s, kThreads / 32);
    }
    smisc[0] = 0;
    smisc[1] = 0;
    smisc[2] = 0;
  }
  __syncthreads();

  auto unit_of = [&](int i) {
    Unit v;
    v.u = u0 + i;
    v.b = v.u / H;
    v.h = v.u - v.b * H;
    v.g = v.h / hpg;
    v.hh = v.h - v.g * hpg;
    v.k = v.b - b0;
    v.ok = sseq[3 * v.k + 2] != 0;
    v.head = v.ok ? sseq[3 * v.k] : 0;  // a rejected cursor stages nothing from the ring
    const int cnt = sseq[3 * v.k + 1];
    v.n = v.ok ? cnt : 0;
    v.flush = v.ok && (cnt + 1 == L);
    v.first = (i == 0) || (v.hh == 0);
    return v;
  };
  // first element of the 16-byte block holding element e, for 2-byte / 4-byte arrays
  auto blk2 = [](size_t e) { return e & ~static_cast<size_t>(7); };
  auto blk4 = [](size_t e) { return e & ~static_cast<size_t>(3); };

  // =============================== producer warp ===============================
  if (warp == kThreads / 32 + 1) {
    if (lane != 0) return;
    int gi = -1;
    for (int i = 0; i < nunits; ++i) {
      const int s = i % stages;
      if (i >= stages && !mbar_wait_bounded(empty + s, static_cast<uint32_t>(((i / stages) - 1) & 1))) break;
      if (smisc[0]) break;
      const Unit v = unit_of(i);
      if (v.first) ++gi;
      unsigned char* st = smem + static_cast<size_t>(LY.st_size) * s;
      unsigned char* gb = gbase + static_cast<size_t>(LY.gb_size) * (gi & 1);
      uint64_t* bar = full + s;
      const size_t u = static_cast<size_t>(v.u);
      const int n = v.n;
      const int seg1 = min(n, C - v.head), seg2 = n - seg1;
      const int esz = KIND == 0 ? 2 : 4;
      const uint32_t tb = (READ == READ_NONE || v.flush) ? tile * 4 : (READ == READ_FP8 ? tile : tile / 2);
      uint32_t bytes = tb + static_cast<uint32_t>(n) * P * esz;
      // group data (first unit of a group in this CTA)
      const size_t ug = static_cast<size_t>(v.b) * H + static_cast<size_t>(v.g) * hpg;  // first unit of the group
      const size_t bg = static_cast<size_t>(v.b) * G + v.g;
      const uint32_t s1b = KIND == 0 ? static_cast<uint32_t>((blk2(ug + hpg + 7) - blk2(ug)) * 2)
                                     : static_cast<uint32_t>((blk4(ug + hpg + 3) - blk4(ug)) * 4);
      const uint32_t s4b = static_cast<uint32_t>((blk4(ug + hpg + 3) - blk4(ug)) * 4);
      if (v.first) {
        bytes += static_cast<uint32_t>(n + 1) * N * 2 + N * 2 + hpg * P * 2 + hpg * Cp * 4 + s1b;
        if (KIND == 0) bytes += hpg * Cp * 2;
        else bytes += s4b;
        if (READ == READ_FP8) bytes += hpg * P * 4;
        if (READ == READ_NVFP4) bytes += hpg * P * (N / 16) + s4b;
      }
      if (KIND == 0 && i == 0) bytes += al16(H * 4);  // A (Mamba-2 only)
      mbar_expect_tx(bar, bytes);
      // the unit: state matrix (or read copy) and this head's buffered records
      if (READ == READ_NONE || v.flush) bulk_g2s(st + LY.st_tile, d.ckpt + u * tile, tb, bar);
      else bulk_g2s(st + LY.st_tile, d.rc_codes + u * tb, tb, bar);
      const unsigned char* rsrc = KIND == 0 ? reinterpret_cast<const unsigned char*>(d.r_x)
                                            : reinterpret_cast<const unsigned char*>(d.r_u);
      const size_t rrow = static_cast<size_t>(P) * esz;
      if (seg1) bulk_g2s(st + LY.st_rec, rsrc + (u * C + v.head) * rrow, seg1 * rrow, bar);
      if (seg2) bulk_g2s(st + LY.st_rec + seg1 * rrow, rsrc + u * C * rrow, seg2 * rrow, bar);
      // the group: keys and query, current tokens, decay rows, scalars, scales
      if (v.first) {
        const uint16_t* rk = (KIND == 0 ? d.r_B : d.r_k) + bg * C * N;
        if (seg1) bulk_g2s(gb + LY.gb_key, rk + static_cast<size_t>(v.head) * N, seg1 * N * 2, bar);
        if (seg2) bulk_g2s(gb + LY.gb_key + seg1 * N * 2, rk, seg2 * N * 2, bar);
        bulk_g2s(gb + LY.gb_key + n * N * 2, (KIND == 0 ? in.Bm : in.k) + bg * N, N * 2, bar);
        bulk_g2s(gb + LY.gb_q, (KIND == 0 ? in.Cm : in.q) + bg * N, N * 2, bar);
        bulk_g2s(gb + LY.gb_cur, (KIND == 0 ? in.x : in.v) + ug * P, hpg * P * 2, bar);
        if (KIND == 0) {
          bulk_g2s(gb + LY.gb_la, d.r_la + ug * Cp, hpg * Cp * 4, bar);
          bulk_g2s(gb + LY.gb_dt, d.r_dt + ug * Cp, hpg * Cp * 2, bar);
          bulk_g2s(gb + LY.gb_s1, in.dt + blk2(ug), s1b, bar);
        } else {
          bulk_g2s(gb + LY.gb_la, d.r_g + ug * Cp, hpg * Cp * 4, bar);
          bulk_g2s(gb + LY.gb_s1, in.g + blk4(ug), s1b, bar);
          bulk_g2s(gb + LY.gb_s2, in.beta + blk4(ug), s4b, bar);
        }
        if (READ == READ_FP8) bulk_g2s(gb + LY.gb_rs, d.rc_rowscale + ug * P, hpg * P * 4, bar);
        if (READ == READ_NVFP4) {
          bulk_g2s(gb + LY.gb_rs, d.rc_blkscale + ug * (P * (N / 16)), hpg * P * (N / 16), bar);
          bulk_g2s(gb + LY.gb_ms, d.rc_matscale + blk4(ug), s4b, bar);
        }
      }
      if (KIND == 0 && i == 0) bulk_g2s(pbase + LY.pe_A, in.A, al16(H * 4), bar);
      smisc[1] = i + 1;
    }
    smisc[2] = 1;
    return;
  }

  const int RW = P / 8;  // rows per computing warp
  const int kq = (lane >> 2) & 7, jl = lane & 3;

  // =============================== prologue warp ===============================
  if (warp == kThreads / 32) {
    float dq = 0.f, dk = 0.f;  // lane j: k_j . q, k_j . k_cur of the current group
    int gi = -1, consumed = 0;
    for (int i = 0; i < nunits; ++i) {
      if (smisc[0]) break;
      const int s = i % stages;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(full + s, static_cast<uint32_t>((i / stages) & 1)))) {
        if (lane == 0) {
          report_error(d.err, DEVERR_TIMEOUT, (u0 + i) / H);
          smisc[0] = 1;
        }
        break;
      }
      consumed = i + 1;
      const Unit v = unit_of(i);
      if (v.first) ++gi;
      unsigned char* st = smem + static_cast<size_t>(LY.st_size) * s;
      const unsigned char* gb = gbase + static_cast<size_t>(LY.gb_size) * (gi & 1);
      float* sc = reinterpret_cast<float*>(st + LY.st_scal);
      if (v.ok) {
        const int n = v.n;
        const int slot_lane = lane < n ? ring_slot(v.head, lane, C) : 0;
        const float* la_row = reinterpret_cast<const float*>(gb + LY.gb_la) + v.hh * Cp;
        const size_t ug = static_cast<size_t>(v.b) * H + static_cast<size_t>(v.g) * hpg;
        if (v.first) {
          const uint16_t* kb = reinterpret_cast<const uint16_t*>(gb + LY.gb_key);
          const float4 q4 = bf4(reinterpret_cast<const uint2*>(gb + LY.gb_q)[lane]);
          const float4 kc4 = bf4(reinterpret_cast<const uint2*>(kb + n * N)[lane]);
          for (int j0 = 0; j0 <= n; j0 += 8) {
            float pq[8], pk[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int j = j0 + k;
              const float4 kj = j <= n ? bf4(reinterpret_cast<const uint2*>(kb + j * N)[lane])
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
              pq[k] = dot4(kj, q4);
              pk[k] = KIND == 1 ? dot4(kj, kc4) : 0.f;
            }
            const float tq = __shfl_sync(0xffffffffu, reduce8(pq, lane), 4 * (lane & 7));
            if ((lane >> 3) == (j0 >> 3)) dq = tq;
            if (KIND == 1) {
              const float tk = __shfl_sync(0xffffffffu, reduce8(pk, lane), 4 * (lane & 7));
              if ((lane >> 3) == (j0 >> 3)) dk = tk;
            }
          }
        }
        if (KIND == 0) {
          const uint16_t* dt_row = reinterpret_cast<const uint16_t*>(gb + LY.gb_dt) + v.hh * Cp;
          const uint16_t* s1 = reinterpret_cast<const uint16_t*>(gb + LY.gb_s1);
          const float dt_cur = bf(s1[(ug & 7) + v.hh]);
          const float la_cur = dt_cur * sA[v.h];
          // records 0..n (current at n): w_j = exp(sum_{i=j+1..n} la_i), gamma = exp(sum_{i<=n} la_i)
          const float sv = suffix_sum(lane < n ? la_row[slot_lane] : (lane == n ? la_cur : 0.f), lane, n);
          const float excl = __shfl_down_sync(0xffffffffu, sv, 1);
          const float Wl = lane <= n ? expf(lane < n ? excl : 0.f) : 0.f;
          const float dtl = lane < n ? bf(dt_row[slot_lane]) : (lane == n ? dt_cur : 0.f);
          if (lane <= n) {
            sc[lane] = Wl * dtl * dq;     // output coefficient on x_j[r]
            sc[2 * C + lane] = Wl * dtl;  // fold coefficient on x_j[r]
          }
          if (lane == 0) {
            sc[3 * C + 2 * P] = expf(sv);
            sc[3 * C + 2 * P + 4] = la_cur;
          }
        } else {
          const float* s1 = reinterpret_cast<const float*>(gb + LY.gb_s1);
          const float* s2 = reinterpret_cast<const float*>(gb + LY.gb_s2);
          // buffered records 0..n-1: w_j = exp(sum_{i=j+1..n-1} g_i), gamma = exp(sum_{i<n} g_i)
          const float sv = suffix_sum(lane < n ? la_row[slot_lane] : 0.f, lane, n - 1);
          const float excl = __shfl_down_sync(0xffffffffu, sv, 1);
          const float Wl = lane < n ? expf(lane + 1 < n ? excl : 0.f) : 0.f;
          const float g_cur = s1[(ug & 3) + v.hh];
          const float a = expf(g_cur);
          if (lane < n) {
            sc[lane] = Wl * dk;         // coefficient of u_j[r] in S k
            sc[C + lane] = Wl * dq;     // coefficient of u_j[r] in S q
            sc[2 * C + lane] = a * Wl;  // fold coefficient of u_j[r]
          }
          const float kq_dot = __shfl_sync(0xffffffffu, dq, n);
          if (lane == 0) {
            sc[3 * C + 2 * P] = n > 0 ? expf(sv) : 1.f;
            sc[3 * C + 2 * P + 1] = a;
            sc[3 * C + 2 * P + 2] = s2[(ug & 3) + v.hh];
            sc[3 * C + 2 * P + 3] = kq_dot;
            sc[3 * C + 2 * P + 4] = g_cur;
          }
        }
      }
      if (lane == 0) reinterpret_cast<int*>(sc)[3 * C + 2 * P + 6] = 0;  // NVFP4 matrix amax slot
      __syncwarp();
      if (lane == 0) mbar_arrive(ready + s);
    }
    // after an abort: let the copies already issued land before the CTA exits
    if (smisc[0] && lane == 0) {
      const uint64_t t0 = global_ns();
      while (!smisc[2] && global_ns() - t0 < 2000000000ull) {
      }
      const int issued = smisc[1];
      for (int j = consumed; j < issued; ++j)
        mbar_wait_bounded(full + (j % stages), static_cast<uint32_t>((j / stages) & 1));
    }
    return;
  }

  // =============================== computing warps ===============================
  uint32_t amax_phase = 0;
  int gi = -1;
  for (int i = 0; i < nunits; ++i) {
    if (smisc[0]) break;
    const int s = i % stages;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(ready + s, static_cast<uint32_t>((i / stages) & 1)))) {
      if (lane == 0) {
        report_error(d.err, DEVERR_TIMEOUT, (u0 + i) / H);
        smisc[0] = 1;
      }
      break;
    }
    const Unit v = unit_of(i);
    if (v.first) ++gi;
    unsigned char* st = smem + static_cast<size_t>(LY.st_size) * s;
    const unsigned char* gb = gbase + static_cast<size_t>(LY.gb_size) * (gi & 1);
    const float* sc = reinterpret_cast<const float*>(st + LY.st_scal);
    if (v.ok) {
      const size_t u = static_cast<size_t>(v.u);
      const int n = v.n;
      const int slot = ring_slot(v.head, n, C);
      const size_t ug = static_cast<size_t>(v.b) * H + static_cast<size_t>(v.g) * hpg;
      const uint16_t* kb = reinterpret_cast<const uint16_t*>(gb + LY.gb_key);
      const uint16_t* cur = reinterpret_cast<const uint16_t*>(gb + LY.gb_cur) + v.hh * P;  // x or v of this head
      float* yrow = y + u * P;
      float4* sT4 = reinterpret_cast<float4*>(st + LY.st_tile);
      float4* gS4 = reinterpret_cast<float4*>(d.ckpt + u * tile);
      const float4 q4 = bf4(reinterpret_cast<const uint2*>(gb + LY.gb_q)[lane]);
      const float4 kc4 = bf4(reinterpret_cast<const uint2*>(kb + n * N)[lane]);
      const float gamma = sc[3 * C + 2 * P];
      if (KIND == 0) {
        const uint16_t* xb = reinterpret_cast<const uint16_t*>(st + LY.st_rec);
        for (int r0 = 0; r0 < RW; r0 += 8) {
          const int Rq = warp + 8 * (r0 + kq);
          const bool vq = r0 + kq < RW;
          // buffered term of row slot kq: lanes 4kq..4kq+3 split the records 0..n
          float ry = 0.f;
          for (int j0 = 0; j0 <= n; j0 += 4) {
            const int j = j0 + jl;
            if (j <= n && vq) ry = fmaf(sc[j], bf(j < n ? xb[j * P + Rq] : cur[Rq]), ry);
          }
          ry += __shfl_xor_sync(0xffffffffu, ry, 1);
          ry += __shfl_xor_sync(0xffffffffu, ry, 2);
          float4 s4[8];
          float part[8];
          float row_scale = 1.f;
          if (READ != READ_NONE && !v.flush) {
            // non-flush: the checkpoint term from the low-precision copy
            const unsigned char* cb = st + LY.st_tile;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int R = warp + 8 * (r0 + k);
              float pv = 0.f;
              if (r0 + k < RW) {
                if (READ == READ_FP8) {
                  const uint32_t w = reinterpret_cast<const uint32_t*>(cb + R * N)[lane];
                  const float2 lo = e4m3x2_to_f32x2(static_cast<uint16_t>(w & 0xFFFFu));
                  const float2 hi = e4m3x2_to_f32x2(static_cast<uint16_t>(w >> 16));
                  pv = dot4(make_float4(lo.x, lo.y, hi.x, hi.y), q4);
                } else {
                  const uint32_t w = reinterpret_cast<const uint16_t*>(cb + R * (N / 2))[lane];
                  const float2 lo = e2m1x2_to_f32x2(w & 0xFFu);
                  const float2 hi = e2m1x2_to_f32x2(w >> 8);
                  const float bs =
                      e4m3_to_f32(gb[LY.gb_rs + (v.hh * P + R) * (N / 16) + (lane >> 2)]);
                  pv = bs * dot4(make_float4(lo.x, lo.y, hi.x, hi.y), q4);
                }
              }
              part[k] = pv;
            }
            if (vq) {
              if (READ == READ_FP8)
                row_scale = reinterpret_cast<const float*>(gb + LY.gb_rs)[v.hh * P + Rq];
              else
                row_scale = reinterpret_cast<const float*>(gb + LY.gb_ms)[(ug & 3) + v.hh];
            }
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              s4[k] = r0 + k < RW ? sT4[(warp + 8 * (r0 + k)) * SEG + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
              part[k] = dot4(s4[k], q4);
            }
          }
          const float tot = reduce8(part, lane);
          if (jl == 0 && vq) {
            yrow[Rq] = fmaf(gamma * row_scale, tot, ry);
            if (!v.flush) d.r_x[(u * C + slot) * P + Rq] = cur[Rq];
          }
          if (v.flush) {
            // lane (kq, jl) holds m_j[Rq] = w_j dt_j x_j[Rq] for records j = 4 jc + jl
            float mreg[kMaxRec / 4];
#pragma unroll
            for (int jc = 0; jc < kMaxRec / 4; ++jc) {
              const int j = 4 * jc + jl;
              mreg[jc] = (j <= n && vq) ? sc[2 * C + j] * bf(j < n ? xb[j * P + Rq] : cur[Rq]) : 0.f;
            }
            float4 acc[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = scale4(gamma, s4[k]);
#pragma unroll
            for (int jc = 0; jc < kMaxRec / 4; ++jc) {
              if (4 * jc > n) break;
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const int j = 4 * jc + jj;
                if (j > n) break;
                const float4 k4 = bf4(reinterpret_cast<const uint2*>(kb + j * N)[lane]);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                  acc[k] = axpy4x2(__shfl_sync(0xffffffffu, mreg[jc], 4 * k + jj), k4, acc[k]);
              }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (r0 + k < RW) {
                __stcs(gS4 + (warp + 8 * (r0 + k)) * SEG + lane, acc[k]);
                if (READ != READ_NONE) sT4[(warp + 8 * (r0 + k)) * SEG + lane] = acc[k];
              }
            }
          }
        }
        if (READ != READ_NONE && v.flush) {
          // refresh the read copy of this warp's rows from the folded rows in shared memory
          if (READ == READ_FP8) {
            uint32_t* codes = reinterpret_cast<uint32_t*>(d.rc_codes + u * tile);
            for (int m = 0; m < RW; ++m) {
              const int R = warp + 8 * m;
              const float4 v4 = sT4[R * SEG + lane];
              float mx = fmaxf(fmaxf(fabsf(v4.x), fabsf(v4.y)), fmaxf(fabsf(v4.z), fabsf(v4.w)));
              mx = seg_max<32>(mx);
              const float scale = __fdiv_rn(mx, 448.0f);
              uint32_t packed = 0;
              if (scale != 0.0f) {
                const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(v4.x, scale), __fdiv_rn(v4.y, scale));
                const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(v4.z, scale), __fdiv_rn(v4.w, scale));
                packed = lo | (hi << 16);
              }
              codes[R * SEG + lane] = packed;
              if (lane == 0) d.rc_rowscale[u * P + R] = scale;
            }
          } else {
            float mloc = 0.f;
            for (int m = 0; m < RW; ++m) {
              const float4 v4 = sT4[(warp + 8 * m) * SEG + lane];
              mloc = fmaxf(mloc, fmaxf(fmaxf(fabsf(v4.x), fabsf(v4.y)), fmaxf(fabsf(v4.z), fabsf(v4.w))));
            }
            mloc = seg_max<32>(mloc);
            int* slot_amax = reinterpret_cast<int*>(st + LY.st_scal) + 3 * C + 2 * P + 6;
            if (lane == 0) atomicMax(slot_amax, __float_as_int(mloc));  // non-negative floats order as ints
            __syncwarp();
            if (lane == 0) mbar_arrive(amaxbar + s);
            const bool got =
                __all_sync(0xffffffffu, mbar_wait_bounded(amaxbar + s, (amax_phase >> s) & 1u));
            amax_phase ^= 1u << s;
            if (!got) {
              if (lane == 0) {
                report_error(d.err, DEVERR_TIMEOUT, v.b);
                smisc[0] = 1;
              }
            } else {
              const float amax = __int_as_float(*reinterpret_cast<volatile int*>(slot_amax));
              const float smat = __fdiv_rn(amax, 2688.0f);  // 448 * 6
              const float six_s = __fmul_rn(6.0f, smat);
              uint16_t* codes = reinterpret_cast<uint16_t*>(d.rc_codes + u * (tile / 2));
              uint8_t* blk = d.rc_blkscale + u * (tile / 16);
              for (int m = 0; m < RW; ++m) {
                const int R = warp + 8 * m;
                const float4 v4 = sT4[R * SEG + lane];
                float mb = fmaxf(fmaxf(fabsf(v4.x), fabsf(v4.y)), fmaxf(fabsf(v4.z), fabsf(v4.w)));
                mb = seg_max<4>(mb);  // 4 lanes = one 16-element block
                uint32_t bcode = 0;
                if (six_s != 0.0f) bcode = f32x2_to_e4m3x2(__fdiv_rn(mb, six_s), 0.0f) & 0xFFu;
                const float dd = __fmul_rn(e4m3_to_f32(bcode), smat);
                uint32_t q = 0;
                if (dd != 0.0f)
                  q = f32x4_to_e2m1x4(__fdiv_rn(v4.x, dd), __fdiv_rn(v4.y, dd), __fdiv_rn(v4.z, dd),
                                      __fdiv_rn(v4.w, dd));
                codes[R * SEG + lane] = static_cast<uint16_t>(q);
                if ((lane & 3) == 0) blk[R * (N / 16) + (lane >> 2)] = static_cast<uint8_t>(bcode);
              }
              if (warp == 0 && lane == 0) d.rc_matscale[u] = smat;
            }
          }
        }
        if (!v.flush && warp == 0) {
          if (lane == 0) {
            const uint16_t* s1 = reinterpret_cast<const uint16_t*>(gb + LY.gb_s1);
            d.r_dt[u * Cp + slot] = s1[(ug & 7) + v.hh];
            d.r_la[u * Cp + slot] = sc[3 * C + 2 * P + 4];
          }
          if (v.hh == 0) {
            const size_t bg = static_cast<size_t>(v.b) * G + v.g;
            reinterpret_cast<uint2*>(d.r_B + (bg * C + slot) * N)[lane] =
                reinterpret_cast<const uint2*>(kb + n * N)[lane];
          }
        }
      } else {
        const float* ub = reinterpret_cast<const float*>(st + LY.st_rec);
        const float a = sc[3 * C + 2 * P + 1], beta = sc[3 * C + 2 * P + 2];
        const float kq_dot = sc[3 * C + 2 * P + 3];
        float* urow = d.r_u + (u * C + slot) * P;
        for (int r0 = 0; r0 < RW; r0 += 8) {
          const int Rq = warp + 8 * (r0 + kq);
          const bool vq = r0 + kq < RW;
          float rk = 0.f, rq = 0.f;
          for (int j0 = 0; j0 < n; j0 += 4) {
            const int j = j0 + jl;
            if (j < n && vq) {
              const float uj = ub[j * P + Rq];
              rk = fmaf(sc[j], uj, rk);
              rq = fmaf(sc[C + j], uj, rq);
            }
          }
          rk += __shfl_xor_sync(0xffffffffu, rk, 1);
          rk += __shfl_xor_sync(0xffffffffu, rk, 2);
          rq += __shfl_xor_sync(0xffffffffu, rq, 1);
          rq += __shfl_xor_sync(0xffffffffu, rq, 2);
          float4 s4[8];
          float pk[8], pq[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            s4[k] = r0 + k < RW ? sT4[(warp + 8 * (r0 + k)) * SEG + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
            pk[k] = dot4(s4[k], kc4);
            pq[k] = dot4(s4[k], q4);
          }
          const float tk = reduce8(pk, lane);
          const float tq = reduce8(pq, lane);
          float uu = 0.f;
          if (vq) {
            const float Sk = fmaf(gamma, tk, rk);
            const float Sq = fmaf(gamma, tq, rq);
            uu = beta * (bf(cur[Rq]) - a * Sk);
            if (jl == 0) {
              yrow[Rq] = fmaf(a, Sq, uu * kq_dot);
              if (!v.flush) urow[Rq] = uu;
            }
          }
          if (v.flush) {
            // lane (kq, jl) holds m_j[Rq] = a w_j u_j[Rq] for records j = 4 jc + jl
            float mreg[kMaxRec / 4];
#pragma unroll
            for (int jc = 0; jc < kMaxRec / 4; ++jc) {
              const int j = 4 * jc + jl;
              mreg[jc] = (j < n && vq) ? sc[2 * C + j] * ub[j * P + Rq] : 0.f;
            }
            float4 acc[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              acc[k] = axpy4(__shfl_sync(0xffffffffu, uu, 4 * k), kc4, scale4(a * gamma, s4[k]));
#pragma unroll
            for (int jc = 0; jc < kMaxRec / 4; ++jc) {
              if (4 * jc >= n) break;
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const int j = 4 * jc + jj;
                if (j >= n) break;
                const float4 k4 = bf4(reinterpret_cast<const uint2*>(kb + j * N)[lane]);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                  acc[k] = axpy4x2(__shfl_sync(0xffffffffu, mreg[jc], 4 * k + jj), k4, acc[k]);
              }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k)
              if (r0 + k < RW) __stcs(gS4 + (warp + 8 * (r0 + k)) * SEG + lane, acc[k]);
          }
        }
        if (!v.flush && warp == 0) {
          if (lane == 0) d.r_g[u * Cp + slot] = sc[3 * C + 2 * P + 4];
          if (v.hh == 0) {
            const size_t bg = static_cast<size_t>(v.b) * G + v.g;
            reinterpret_cast<uint2*>(d.r_k + (bg * C + slot) * N)[lane] =
                reinterpret_cast<const uint2*>(kb + n * N)[lane];
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + s);
  }
}

template <int KIND, int READ>
cudaError_t launch128(const LayerDev& d, const TokenIn& in, float* y, cudaStream_t s) {
  const int hpg = d.H / d.G;
  const Lay128 LY = lay128(KIND, READ, d.P, d.C, d.Cp, d.H, hpg);
  const long budget = 227L * 1024 - 2L * LY.gb_size - LY.pe_size;
  long stages = budget / LY.st_size;
  if (stages > 8) stages = 8;
  // a group buffer is rewritten two groups later: every unit of that earlier
  // group must have left the pipeline, which holds when stages <= hpg + 1
  if (stages > hpg + 1) stages = hpg + 1;
  if (stages < 1) return cudaErrorInvalidConfiguration;
  const size_t smem = static_cast<size_t>(LY.st_size) * stages + 2u * LY.gb_size + LY.pe_size;
  const int total = d.B * d.H;
  int grid = d.num_sms > 0 ? d.num_sms : 1;
  if (grid > total) grid = total;
  int per = (total + grid - 1) / grid;
  while (per / d.H + 2 > kMaxSeq128) {
    grid *= 2;
    per = (total + grid - 1) / grid;
  }
  grid = (total + per - 1) / per;
  auto kernel = decode128_kernel<KIND, READ>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads128, smem, s>>>(d, in, y, per, static_cast<int>(stages));
  return cudaGetLastError();
}

}  // namespace

size_t decode128_smem_bytes(const LayerDev& d) {
  const Lay128 LY = lay128(d.kind, d.read_mode, d.P, d.C, d.Cp, d.H, d.H / d.G);
  return static_cast<size_t>(LY.st_size) + 2u * LY.gb_size + LY.pe_size;
}

cudaError_t launch_decode128(const LayerDev& d, const TokenIn& in, float* y, cudaStream_t s) {
  if (d.N != N) return cudaErrorInvalidValue;
  if (d.kind == 0) {
    if (d.read_mode == READ_FP8) return launch128<0, READ_FP8>(d, in, y, s);
    if (d.read_mode == READ_NVFP4) return launch128<0, READ_NVFP4>(d, in, y, s);
    return launch128<0, READ_NONE>(d, in, y, s);
  }
  return launch128<1, READ_NONE>(d, in, y, s);
}

}  // namespace rs
