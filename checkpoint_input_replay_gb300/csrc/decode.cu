// Standard decode step: the output-only non-flush body and the flush body,
// selected per sequence from its device-resident cursor inside one launch.
//
// Unrolled form ("ReplaySSM caches SSM inputs instead of state" (richland.au),
// "What shipped", the paragraph on unrolling the recurrence): with records
// j = 0..n-1 buffered since the checkpoint and the current token as record n,
//   S_n = gamma S_ckpt + sum_{j<=n} w_j v_j k_j^T,
//   w_j = prod_{i=j+1..n} a_i,  gamma = prod_{i=0..n} a_i,
// so the Mamba-2 output is
//   y = gamma (S_ckpt q) + sum_{j<=n} w_j (k_j . q) v_j
// and S_ckpt is only read.  Gated DeltaNet buffers (g, u, k) records with
// u = b (v - a S_{t-1} k), which gives S_t = a S_{t-1} + u k^T the same form;
// its step needs S_{t-1} k and S_{t-1} q from one pass over S_ckpt.
//
// Kernel structure (one persistent CTA per SM):
//  * a work unit is one (sequence, head) state matrix [P][N]; CTA c owns a
//    contiguous range of units, so it meets each group (and sequence) once;
//  * at start the CTA reads the cursors of the sequences it covers and counts
//    itself in on their arrival counters; the last CTA of a sequence to arrive
//    (every reader has then read the old cursor) writes the new cursor;
//  * thread 0 keeps `stages` units of input in flight with bulk copies
//    (cp.async.bulk, the untiled TMA path) into a shared-memory ring: the state
//    matrix (or its low-precision read copy), exactly the buffered records, the
//    current token, and the group's keys when the group changes;
//  * all warps compute unit i from shared memory while units i+1.. load: the
//    per-group key dot products once per group, the decay weights with a warp
//    scan, the buffered term per row, then one pass over the matrix;
//  * a dedicated producer warp issues the copies; the eight computing warps
//    release a stage through an mbarrier when they are done with it;
//  * for d_state = 128 a unit is computed warp-locally: warp w owns rows
//    w, w+8, ..; lanes split the buffered records four per row and the row
//    sums use a transpose-reduce over 8 rows (9 shuffles);
//  * a flush unit folds the records in registers and writes the checkpoint
//    back once; a non-flush unit stores no state.
#include "common.cuh"
#include "readcopy.cuh"

namespace rs {
namespace {

constexpr int kMaxSeq = 64;  // sequences one CTA may cover

__host__ __device__ __forceinline__ int a16(int x) { return (x + 15) & ~15; }
__host__ __device__ __forceinline__ int a128(int x) { return (x + 127) & ~127; }

// Byte offsets inside one pipeline stage.
struct Stage {
  int tile;   // f32 [P][N] state matrix, or the read copy (codes, then scales)
  int rec;    // Mamba-2: x bf16 [C][P] records 0..n (n = current); GDN: u f32 [C][P] records 0..n-1
  int key;    // bf16 [C][N] keys of records 0..n (current at n), only for the first unit of a group
  int q;      // bf16 [N], with the keys
  int v;      // GDN: current v bf16 [P]
  int la;     // f32 [Cp] log decays in slot order
  int dt;     // Mamba-2: dt bf16 [Cp] in slot order
  int chunk;  // three 16-byte chunks: Mamba-2 dt_cur, A, matrix scale; GDN g_cur, beta, -
  int scal;   // f32 [3C + 2P + 8]: per-record coefficients, per-row buffered terms, scalars
  int size;
};

__host__ __device__ __forceinline__ Stage stage_layout(int kind, int P, int N, int C, int Cp) {
  Stage s;
  int o = 0;
  s.tile = o;
  o += P * N * 4;
  s.rec = o;
  o += kind == 0 ? a16(C * P * 2) : C * P * 4;
  s.key = o;
  o += C * N * 2;
  s.q = o;
  o += N * 2;
  s.v = o;
  o += kind == 0 ? 0 : a16(P * 2);
  s.la = o;
  o += Cp * 4;
  s.dt = o;
  o += kind == 0 ? a16(Cp * 2) : 0;
  s.chunk = o;
  o += 48;
  s.scal = o;
  o += (3 * C + 2 * P + 8) * 4;
  s.size = a128(o);
  return s;
}

// Persistent (non-stage) shared memory, in floats, after the stages.
struct Persist {
  int q, keys, dots, dots2, W, row, row2, coef, red, misc, bars, seq, size_floats;
};

__host__ __device__ __forceinline__ Persist persist_layout(int P, int N, int C) {
  Persist p;
  int o = 0;
  p.q = o;      o += N;          // group query f32
  p.keys = o;   o += C * N;      // group keys f32 [C][N] (records 0..n)
  p.dots = o;   o += C;          // k_j . q   (GDN: with k_cur . q at n)
  p.dots2 = o;  o += C;          // GDN: k_j . k_cur
  p.W = o;      o += C + 4;      // decay weights; gamma, dt_cur | a, log a_cur | beta
  p.row = o;    o += P;          // buffered term per row (GDN: for S k)
  p.row2 = o;   o += P;          // GDN: buffered term for S q
  p.coef = o;   o += C * P;      // flush coefficients [C][P]
  p.red = o;    o += kThreads / 32;
  p.misc = o;   o += 4;
  p.bars = (o + 3) & ~3;         // 16-byte aligned: 8 full, empty, ready, amax mbarriers (u64)
  o = p.bars + 2 * 32;
  p.seq = o;    o += 3 * kMaxSeq;  // cached cursors: head, count, ok
  p.size_floats = o;
  return p;
}

__device__ __forceinline__ int ring_slot(int head, int j, int C) {
  int s = head + j;
  return s >= C ? s - C : s;
}

// bulk copy of `bytes` (a multiple of 16, possibly 0)
__device__ __forceinline__ void copy_in(unsigned char* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  if (bytes) bulk_g2s(dst, src, bytes, bar);
}

struct UnitInfo {
  int u, b, h, g, k;  // unit, sequence, head, group, cached-sequence index
  int head, n;        // cursor head and buffered records
  bool ok, flush, first_of_group;
};

// Non-flush output rows from the FP8 per-row read copy staged in shared memory:
// codes [P][N] then row scales f32 [P].  Loops run whole warps so the
// segmented shuffles always see all 32 lanes.
template <int N>
__device__ __forceinline__ void rc_rows_fp8(const unsigned char* sC, const float* sRS, const float* sq, int P,
                                            float gamma, const float* sry, float* yrow) {
  constexpr int E = 16;
  constexpr int TPR = N / E;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int c = t % TPR;
  float qv[E];
#pragma unroll
  for (int i = 0; i < E; ++i) qv[i] = sq[c * E + i];
  const int total = P * TPR;
  for (int f0 = warp * 32; f0 < total; f0 += kThreads) {
    const int f = f0 + lane;
    float acc = 0.f;
    if (f < total) {
      const uint4 raw = reinterpret_cast<const uint4*>(sC)[f];
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 lo = e4m3x2_to_f32x2(static_cast<uint16_t>(w[k] & 0xFFFFu));
        const float2 hi = e4m3x2_to_f32x2(static_cast<uint16_t>(w[k] >> 16));
        acc = fmaf(lo.x, qv[4 * k], acc);
        acc = fmaf(lo.y, qv[4 * k + 1], acc);
        acc = fmaf(hi.x, qv[4 * k + 2], acc);
        acc = fmaf(hi.y, qv[4 * k + 3], acc);
      }
    }
    acc = seg_sum<TPR>(acc);
    if (f < total && c == 0) {
      const int r = f / TPR;
      yrow[r] = fmaf(gamma * sRS[r], acc, sry[r]);
    }
  }
}

// Non-flush output rows from the NVFP4 read copy staged in shared memory:
// codes [P][N/2] (element 2i in the low nibble) then block scales [P][N/16].
template <int N>
__device__ __forceinline__ void rc_rows_nvfp4(const unsigned char* sC, const unsigned char* sBS, float smat,
                                              const float* sq, int P, float gamma, const float* sry, float* yrow) {
  constexpr int E = N >= 32 ? 32 : 16;
  constexpr int TPR = N / E;
  constexpr int WORDS = E / 8;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int c = t % TPR;
  float qv[E];
#pragma unroll
  for (int i = 0; i < E; ++i) qv[i] = sq[c * E + i];
  const int total = P * TPR;
  for (int f0 = warp * 32; f0 < total; f0 += kThreads) {
    const int f = f0 + lane;
    float acc = 0.f;
    if (f < total) {
      const int r = f / TPR;
      uint32_t w[4];
      if (WORDS == 4) {
        const uint4 raw = reinterpret_cast<const uint4*>(sC)[f];
        w[0] = raw.x; w[1] = raw.y; w[2] = raw.z; w[3] = raw.w;
      } else {
        const uint2 raw = reinterpret_cast<const uint2*>(sC)[f];
        w[0] = raw.x; w[1] = raw.y; w[2] = 0; w[3] = 0;
      }
#pragma unroll
      for (int blk = 0; blk < E / 16; ++blk) {
        float part = 0.f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t word = w[2 * blk + k];
#pragma unroll
          for (int by = 0; by < 4; ++by) {
            const float2 v = e2m1x2_to_f32x2((word >> (8 * by)) & 0xFFu);
            const int e = blk * 16 + k * 8 + by * 2;
            part = fmaf(v.x, qv[e], part);
            part = fmaf(v.y, qv[e + 1], part);
          }
        }
        const float bs = e4m3_to_f32(sBS[r * (N / 16) + c * (E / 16) + blk]);
        acc = fmaf(bs, part, acc);
      }
    }
    acc = seg_sum<TPR>(acc);
    if (f < total && c == 0) {
      const int r = f / TPR;
      yrow[r] = fmaf(gamma * smat, acc, sry[r]);
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel (KIND 0: Mamba-2, 1: Gated DeltaNet)
// ---------------------------------------------------------------------------
// 8 computing warps + 1 producer warp, + 1 prologue warp on the warp-local path
template <int N, int READ>
constexpr int decode_threads() {
  return kThreads + (N == 128 ? 64 : 32);
}

template <int KIND, int N, int READ>
__global__ void __launch_bounds__(decode_threads<N, READ>(), 1) decode_kernel(const LayerDev d, const TokenIn in,
                                                                   float* __restrict__ y, const int units_per_cta,
                                                                   const int stages) {
  constexpr int SEG = N / 4;  // lanes per state row, one float4 each
  // d_state 128: every warp computes its rows of a unit on its own
  constexpr bool kWarpLocal = (N == 128);
  extern __shared__ __align__(1024) unsigned char smem[];

  const int P = d.P, H = d.H, G = d.G, C = d.C, L = d.L, Cp = d.Cp;
  const int hpg = H / G;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int tile = P * N;
  const Stage SL = stage_layout(KIND, P, N, C, Cp);
  const Persist PL = persist_layout(P, N, C);
  float* pf = reinterpret_cast<float*>(smem + static_cast<size_t>(SL.size) * stages);
  float* sq = pf + PL.q;
  float* sK = pf + PL.keys;
  float* sdot = pf + PL.dots;
  float* sdot2 = pf + PL.dots2;
  float* sW = pf + PL.W;
  float* srow = pf + PL.row;
  float* srow2 = pf + PL.row2;
  float* scoef = pf + PL.coef;
  float* sred = pf + PL.red;
  volatile int* smisc = reinterpret_cast<volatile int*>(pf + PL.misc);  // abort, issued, producer done
  uint64_t* full = reinterpret_cast<uint64_t*>(pf + PL.bars);
  uint64_t* empty = full + 8;
  uint64_t* ready = full + 16;
  uint64_t* amaxbar = full + 24;  // NVFP4 flush units: the eight computing warps exchange the matrix amax
  int* sseq = reinterpret_cast<int*>(pf + PL.seq);

  const int total_units = d.B * H;
  const int u0 = blockIdx.x * units_per_cta;
  const int u1 = min(u0 + units_per_cta, total_units);
  if (u0 >= u1) return;
  const int nunits = u1 - u0;
  const int b0 = u0 / H, b1 = (u1 - 1) / H;  // sequences covered
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
      mbar_init(empty + s, kWarpLocal ? kThreads / 32 : 1);
      mbar_init(ready + s, 1);
      mbar_init(amaxbar + s, kThreads / 32);
    }
    smisc[0] = 0;  // abort
    smisc[1] = 0;  // units issued
    smisc[2] = 0;  // producer finished
  }
  __syncthreads();

  auto unit_info = [&](int i) {
    UnitInfo ui;
    ui.u = u0 + i;
    ui.b = ui.u / H;
    ui.h = ui.u - ui.b * H;
    ui.g = ui.h / hpg;
    ui.k = ui.b - b0;
    ui.head = sseq[3 * ui.k];
    const int cnt = sseq[3 * ui.k + 1];
    ui.ok = sseq[3 * ui.k + 2] != 0;
    ui.n = ui.ok ? cnt : 0;
    ui.flush = ui.ok && (cnt + 1 == L);
    ui.first_of_group = (i == 0) || (ui.h % hpg == 0);
    return ui;
  };

  // =========================== producer warp ===============================
  if (warp == kThreads / 32 + (kWarpLocal ? 1 : 0)) {
    if (lane != 0) return;
    for (int i = 0; i < nunits; ++i) {
      const int s = i % stages;
      if (i >= stages && !mbar_wait_bounded(empty + s, static_cast<uint32_t>(((i / stages) - 1) & 1))) break;
      if (smisc[0]) break;
      const UnitInfo ui = unit_info(i);
      unsigned char* st = smem + static_cast<size_t>(SL.size) * s;
      uint64_t* bar = full + s;
      const size_t u = static_cast<size_t>(ui.u);
      const size_t bg = static_cast<size_t>(ui.b) * G + ui.g;
      const int n = ui.n;
      const int seg1 = min(n, C - ui.head), seg2 = n - seg1;
      const int resz = KIND == 0 ? 2 : 4;  // record element size
      uint32_t tb0 = 0, tb1 = 0;
      if (READ == READ_NONE || ui.flush) {
        tb0 = tile * 4;
      } else if (READ == READ_FP8) {
        tb0 = tile;
        tb1 = P * 4;
      } else {
        tb0 = tile / 2;
        tb1 = tile / 16;
      }
      uint32_t bytes = tb0 + tb1;
      bytes += static_cast<uint32_t>(n) * P * resz;                        // buffered records
      bytes += KIND == 0 ? P * 2 : a16(P * 2);                              // current x / v
      // all buffered keys for the first unit of a group (dot products) and for a
      // fold; the current key and q for every unit on the warp-local path
      const bool all_keys = ui.first_of_group || (kWarpLocal && ui.flush);
      const bool cur_key = kWarpLocal || all_keys;
      if (all_keys) bytes += static_cast<uint32_t>(n) * N * 2;
      if (cur_key) bytes += 2 * N * 2;
      bytes += Cp * 4 + (KIND == 0 ? a16(Cp * 2) : 0) + 48;               // log decays, dt, chunks
      mbar_expect_tx(bar, bytes);
      if (READ == READ_NONE || ui.flush) {
        copy_in(st + SL.tile, d.ckpt + u * tile, tb0, bar);
      } else if (READ == READ_FP8) {
        copy_in(st + SL.tile, d.rc_codes + u * tile, tb0, bar);
        copy_in(st + SL.tile + tile, d.rc_rowscale + u * P, tb1, bar);
      } else {
        copy_in(st + SL.tile, d.rc_codes + u * (tile / 2), tb0, bar);
        copy_in(st + SL.tile + tile / 2, d.rc_blkscale + u * (tile / 16), tb1, bar);
      }
      if (KIND == 0) {
        const uint16_t* rx = d.r_x + u * C * P;
        copy_in(st + SL.rec, rx + static_cast<size_t>(ui.head) * P, seg1 * P * 2, bar);
        copy_in(st + SL.rec + seg1 * P * 2, rx, seg2 * P * 2, bar);
        copy_in(st + SL.rec + n * P * 2, in.x + u * P, P * 2, bar);
      } else {
        const float* ru = d.r_u + u * C * P;
        copy_in(st + SL.rec, ru + static_cast<size_t>(ui.head) * P, seg1 * P * 4, bar);
        copy_in(st + SL.rec + seg1 * P * 4, ru, seg2 * P * 4, bar);
        copy_in(st + SL.v, in.v + u * P, a16(P * 2), bar);
      }
      if (all_keys) {
        const uint16_t* rk = (KIND == 0 ? d.r_B : d.r_k) + bg * C * N;
        copy_in(st + SL.key, rk + static_cast<size_t>(ui.head) * N, seg1 * N * 2, bar);
        copy_in(st + SL.key + seg1 * N * 2, rk, seg2 * N * 2, bar);
      }
      if (cur_key) {
        copy_in(st + SL.key + n * N * 2, (KIND == 0 ? in.Bm : in.k) + bg * N, N * 2, bar);
        copy_in(st + SL.q, (KIND == 0 ? in.Cm : in.q) + bg * N, N * 2, bar);
      }
      if (KIND == 0) {
        copy_in(st + SL.la, d.r_la + u * Cp, Cp * 4, bar);
        copy_in(st + SL.dt, d.r_dt + u * Cp, a16(Cp * 2), bar);
        copy_in(st + SL.chunk, in.dt + (u & ~static_cast<size_t>(7)), 16, bar);
        copy_in(st + SL.chunk + 16, in.A + (ui.h & ~3), 16, bar);
        if (READ == READ_NVFP4)
          copy_in(st + SL.chunk + 32, d.rc_matscale + (u & ~static_cast<size_t>(3)), 16, bar);
        else
          copy_in(st + SL.chunk + 32, in.A + (ui.h & ~3), 16, bar);
      } else {
        copy_in(st + SL.la, d.r_g + u * Cp, Cp * 4, bar);
        copy_in(st + SL.chunk, in.g + (u & ~static_cast<size_t>(3)), 16, bar);
        copy_in(st + SL.chunk + 16, in.beta + (u & ~static_cast<size_t>(3)), 16, bar);
        copy_in(st + SL.chunk + 32, in.g + (u & ~static_cast<size_t>(3)), 16, bar);
      }
      smisc[1] = i + 1;
    }
    smisc[2] = 1;
    return;
  }

  // =========================== computing warps ==============================
  if constexpr (kWarpLocal) {
    const int RW = P / 8;  // rows per computing warp
    const int kq = (lane >> 2) & 7, jl = lane & 3;
    // ===================== prologue warp =====================
    // Runs ahead of the computing warps: per unit it turns the staged records
    // into scalars -- key dot products (once per group, kept in registers),
    // decay weights, per-record coefficients and the buffered term of every
    // row -- writes them into the stage and signals `ready`.
    if (warp == kThreads / 32) {
      float dq = 0.f, dk = 0.f;  // lane j: k_j . q, k_j . k_cur of the current group
      int consumed = 0;
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
        const UnitInfo ui = unit_info(i);
        unsigned char* st = smem + static_cast<size_t>(SL.size) * s;
        float* sc = reinterpret_cast<float*>(st + SL.scal);
        if (ui.ok) {
          const size_t u = static_cast<size_t>(ui.u);
          const int n = ui.n;
          const int slot_lane = lane < n ? ring_slot(ui.head, lane, C) : 0;
          const float* la_slot = reinterpret_cast<const float*>(st + SL.la);
          const float* chunk = reinterpret_cast<const float*>(st + SL.chunk);
          if (ui.first_of_group) {
            const uint16_t* kb = reinterpret_cast<const uint16_t*>(st + SL.key);
            const float4 q4 = bf4(reinterpret_cast<const uint2*>(st + SL.q)[lane]);
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
            const uint16_t* dtr = reinterpret_cast<const uint16_t*>(st + SL.dt);
            const uint16_t* dtc = reinterpret_cast<const uint16_t*>(st + SL.chunk);
            const float dt_cur = bf(dtc[u & 7]);
            const float la_cur = dt_cur * chunk[4 + (ui.h & 3)];
            // records 0..n (current at n): w_j = exp(sum_{i=j+1..n} la_i), gamma = exp(sum_{i<=n} la_i)
            const float v = suffix_sum(lane < n ? la_slot[slot_lane] : (lane == n ? la_cur : 0.f), lane, n);
            const float excl = __shfl_down_sync(0xffffffffu, v, 1);
            const float Wl = lane <= n ? expf(lane < n ? excl : 0.f) : 0.f;
            const float dtl = lane < n ? bf(dtr[slot_lane]) : (lane == n ? dt_cur : 0.f);
            if (lane <= n) {
              sc[lane] = Wl * dtl * dq;     // output coefficient on x_j[r]
              sc[2 * C + lane] = Wl * dtl;  // fold coefficient on x_j[r]
            }
            if (lane == 0) {
              sc[3 * C + 2 * P] = expf(v);
              sc[3 * C + 2 * P + 4] = la_cur;
            }
          } else {
            // buffered records 0..n-1: w_j = exp(sum_{i=j+1..n-1} g_i), gamma = exp(sum_{i<n} g_i)
            const float v = suffix_sum(lane < n ? la_slot[slot_lane] : 0.f, lane, n - 1);
            const float excl = __shfl_down_sync(0xffffffffu, v, 1);
            const float Wl = lane < n ? expf(lane + 1 < n ? excl : 0.f) : 0.f;
            const float a = expf(chunk[u & 3]);
            if (lane < n) {
              sc[lane] = Wl * dk;          // coefficient of u_j[r] in S k
              sc[C + lane] = Wl * dq;      // coefficient of u_j[r] in S q
              sc[2 * C + lane] = a * Wl;   // fold coefficient of u_j[r]
            }
            const float kq_dot = __shfl_sync(0xffffffffu, dq, n);
            if (lane == 0) {
              sc[3 * C + 2 * P] = n > 0 ? expf(v) : 1.f;
              sc[3 * C + 2 * P + 1] = a;
              sc[3 * C + 2 * P + 2] = chunk[4 + (u & 3)];
              sc[3 * C + 2 * P + 3] = kq_dot;
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
    // ===================== computing warps =====================
    // warp w owns rows w, w+8, ..; lane = column chunk; no barrier across warps
    // (an NVFP4 flush unit exchanges its matrix amax through a bounded mbarrier)
    uint32_t amax_phase = 0;
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
      const UnitInfo ui = unit_info(i);
      unsigned char* st = smem + static_cast<size_t>(SL.size) * s;
      const float* sc = reinterpret_cast<const float*>(st + SL.scal);
      if (ui.ok) {
        const size_t u = static_cast<size_t>(ui.u);
        const int n = ui.n;
        const int slot = ring_slot(ui.head, n, C);
        const uint16_t* kb = reinterpret_cast<const uint16_t*>(st + SL.key);
        float* yrow = y + u * P;
        float4* sT4 = reinterpret_cast<float4*>(st + SL.tile);
        float4* gS4 = reinterpret_cast<float4*>(d.ckpt + u * tile);
        const float4 q4 = bf4(reinterpret_cast<const uint2*>(st + SL.q)[lane]);
        const float4 kc4 = bf4(reinterpret_cast<const uint2*>(kb + n * N)[lane]);
        const float gamma = sc[3 * C + 2 * P];
        if (KIND == 0) {
          const uint16_t* xb = reinterpret_cast<const uint16_t*>(st + SL.rec);
          for (int r0 = 0; r0 < RW; r0 += 8) {
            const int Rq = warp + 8 * (r0 + kq);
            const bool vq = r0 + kq < RW;
            // buffered term of row slot kq: lanes 4kq..4kq+3 split the records
            float ry = 0.f;
            for (int j0 = 0; j0 <= n; j0 += 4) {
              const int j = j0 + jl;
              if (j <= n && vq) ry = fmaf(sc[j], bf(xb[j * P + Rq]), ry);
            }
            ry += __shfl_xor_sync(0xffffffffu, ry, 1);
            ry += __shfl_xor_sync(0xffffffffu, ry, 2);
            float4 s4[8];
            float part[8];
            float row_scale = 1.f;  // read-copy scale of row slot kq
            if (READ != READ_NONE && !ui.flush) {
              // non-flush: the checkpoint term from the low-precision copy
              const unsigned char* cb = st + SL.tile;
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
                    const float bs = e4m3_to_f32(cb[P * (N / 2) + R * (N / 16) + (lane >> 2)]);
                    pv = bs * dot4(make_float4(lo.x, lo.y, hi.x, hi.y), q4);
                  }
                }
                part[k] = pv;
              }
              if (vq) {
                if (READ == READ_FP8)
                  row_scale = reinterpret_cast<const float*>(cb + P * N)[Rq];
                else
                  row_scale = reinterpret_cast<const float*>(st + SL.chunk)[8 + (u & 3)];
              }
            } else {
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                s4[k] = r0 + k < RW ? sT4[(warp + 8 * (r0 + k)) * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
                part[k] = dot4(s4[k], q4);
              }
            }
            const float tot = reduce8(part, lane);
            if (jl == 0 && vq) {
              yrow[Rq] = fmaf(gamma * row_scale, tot, ry);
              if (!ui.flush) d.r_x[(u * C + slot) * P + Rq] = xb[n * P + Rq];
            }
            if (ui.flush) {
              // lane (kq, jl) holds m_j[Rq] = w_j dt_j x_j[Rq] for records j = 4 jc + jl
              float mreg[kMaxRec / 4];
#pragma unroll
              for (int jc = 0; jc < kMaxRec / 4; ++jc) {
                const int j = 4 * jc + jl;
                mreg[jc] = (j <= n && vq) ? sc[2 * C + j] * bf(xb[j * P + Rq]) : 0.f;
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
                  __stcs(gS4 + (warp + 8 * (r0 + k)) * 32 + lane, acc[k]);
                  if (READ != READ_NONE) sT4[(warp + 8 * (r0 + k)) * 32 + lane] = acc[k];
                }
              }
            }
          }
          if (READ != READ_NONE && ui.flush) {
            // refresh the read copy of this warp's rows from the folded rows in shared memory
            if (READ == READ_FP8) {
              uint32_t* codes = reinterpret_cast<uint32_t*>(d.rc_codes + u * tile);
              for (int m = 0; m < RW; ++m) {
                const int R = warp + 8 * m;
                const float4 v4 = sT4[R * 32 + lane];
                float mx = fmaxf(fmaxf(fabsf(v4.x), fabsf(v4.y)), fmaxf(fabsf(v4.z), fabsf(v4.w)));
                mx = seg_max<32>(mx);
                const float scale = __fdiv_rn(mx, 448.0f);
                uint32_t packed = 0;
                if (scale != 0.0f) {
                  const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(v4.x, scale), __fdiv_rn(v4.y, scale));
                  const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(v4.z, scale), __fdiv_rn(v4.w, scale));
                  packed = lo | (hi << 16);
                }
                codes[R * 32 + lane] = packed;
                if (lane == 0) d.rc_rowscale[u * P + R] = scale;
              }
            } else {
              float mloc = 0.f;
              for (int m = 0; m < RW; ++m) {
                const float4 v4 = sT4[(warp + 8 * m) * 32 + lane];
                mloc = fmaxf(mloc, fmaxf(fmaxf(fabsf(v4.x), fabsf(v4.y)), fmaxf(fabsf(v4.z), fabsf(v4.w))));
              }
              mloc = seg_max<32>(mloc);
              volatile int* slot_amax = reinterpret_cast<volatile int*>(
                  reinterpret_cast<int*>(st + SL.scal) + 3 * C + 2 * P + 6);
              if (lane == 0) {
                atomicMax(const_cast<int*>(slot_amax), __float_as_int(mloc));  // non-negative floats order as ints
                __threadfence_block();
              }
              __syncwarp();
              if (lane == 0) mbar_arrive(amaxbar + s);
              const bool got = __all_sync(0xffffffffu,
                                          mbar_wait_bounded(amaxbar + s, (amax_phase >> s) & 1u));
              amax_phase ^= 1u << s;
              if (!got) {
                if (lane == 0) {
                  report_error(d.err, DEVERR_TIMEOUT, ui.b);
                  smisc[0] = 1;
                }
              } else {
                const float amax = __int_as_float(*slot_amax);
                const float smat = __fdiv_rn(amax, 2688.0f);  // 448 * 6
                const float six_s = __fmul_rn(6.0f, smat);
                uint16_t* codes = reinterpret_cast<uint16_t*>(d.rc_codes + u * (tile / 2));
                uint8_t* blk = d.rc_blkscale + u * (tile / 16);
                for (int m = 0; m < RW; ++m) {
                  const int R = warp + 8 * m;
                  const float4 v4 = sT4[R * 32 + lane];
                  float mb = fmaxf(fmaxf(fabsf(v4.x), fabsf(v4.y)), fmaxf(fabsf(v4.z), fabsf(v4.w)));
                  mb = seg_max<4>(mb);  // 4 lanes = one 16-element block
                  uint32_t bcode = 0;
                  if (six_s != 0.0f) bcode = f32x2_to_e4m3x2(__fdiv_rn(mb, six_s), 0.0f) & 0xFFu;
                  const float dd = __fmul_rn(e4m3_to_f32(bcode), smat);
                  uint32_t q = 0;
                  if (dd != 0.0f)
                    q = f32x4_to_e2m1x4(__fdiv_rn(v4.x, dd), __fdiv_rn(v4.y, dd), __fdiv_rn(v4.z, dd),
                                        __fdiv_rn(v4.w, dd));
                  codes[R * 32 + lane] = static_cast<uint16_t>(q);
                  if ((lane & 3) == 0) blk[R * (N / 16) + (lane >> 2)] = static_cast<uint8_t>(bcode);
                }
                if (warp == 0 && lane == 0) d.rc_matscale[u] = smat;
              }
            }
          }
          if (!ui.flush && warp == 0) {
            if (lane == 0) {
              const uint16_t* dtc = reinterpret_cast<const uint16_t*>(st + SL.chunk);
              d.r_dt[u * Cp + slot] = dtc[u & 7];
              d.r_la[u * Cp + slot] = sc[3 * C + 2 * P + 4];
            }
            if (ui.h % hpg == 0) {
              const size_t bg = static_cast<size_t>(ui.b) * G + ui.g;
              reinterpret_cast<uint2*>(d.r_B + (bg * C + slot) * N)[lane] =
                  reinterpret_cast<const uint2*>(kb + n * N)[lane];
            }
          }
        } else {
          const float* ub = reinterpret_cast<const float*>(st + SL.rec);
          const uint16_t* vb = reinterpret_cast<const uint16_t*>(st + SL.v);
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
              s4[k] = r0 + k < RW ? sT4[(warp + 8 * (r0 + k)) * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
              pk[k] = dot4(s4[k], kc4);
              pq[k] = dot4(s4[k], q4);
            }
            const float tk = reduce8(pk, lane);
            const float tq = reduce8(pq, lane);
            float uu = 0.f;
            if (vq) {
              const float Sk = fmaf(gamma, tk, rk);
              const float Sq = fmaf(gamma, tq, rq);
              uu = beta * (bf(vb[Rq]) - a * Sk);
              if (jl == 0) {
                yrow[Rq] = fmaf(a, Sq, uu * kq_dot);
                if (!ui.flush) urow[Rq] = uu;
              }
            }
            if (ui.flush) {
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
                if (r0 + k < RW) __stcs(gS4 + (warp + 8 * (r0 + k)) * 32 + lane, acc[k]);
            }
          }
          if (!ui.flush && warp == 0) {
            const float* chunk = reinterpret_cast<const float*>(st + SL.chunk);
            if (lane == 0) d.r_g[u * Cp + slot] = chunk[u & 3];
            if (ui.h % hpg == 0) {
              const size_t bg = static_cast<size_t>(ui.b) * G + ui.g;
              reinterpret_cast<uint2*>(d.r_k + (bg * C + slot) * N)[lane] =
                  reinterpret_cast<const uint2*>(kb + n * N)[lane];
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
    }
    return;
  }

  const int c4 = t % SEG;
  int consumed = 0;
  for (int i = 0; i < nunits; ++i) {
    const UnitInfo ui = unit_info(i);
    const int s = i % stages;
    unsigned char* st = smem + static_cast<size_t>(SL.size) * s;
    const uint32_t parity = static_cast<uint32_t>((i / stages) & 1);
    const bool arrived = compute_sync_and(mbar_wait_bounded(full + s, parity));
    if (!arrived) {
      if (t == 0) {
        report_error(d.err, DEVERR_TIMEOUT, ui.b);
        smisc[0] = 1;
      }
      break;
    }
    consumed = i + 1;
    const size_t u = static_cast<size_t>(ui.u);
    const int n = ui.n;
    const int slot = ring_slot(ui.head, n, C);
    const int slot_lane = lane < n ? ring_slot(ui.head, lane, C) : 0;
    const float* la_slot = reinterpret_cast<const float*>(st + SL.la);
    const float* chunk = reinterpret_cast<const float*>(st + SL.chunk);
    float* yrow = y + u * P;
    float4* sT4 = reinterpret_cast<float4*>(st + SL.tile);
    float4* gS4 = reinterpret_cast<float4*>(d.ckpt + u * tile);
    const int nf4 = tile / 4;

    // ---- per group: keys, query and their dot products (once per group) ----
    if (ui.first_of_group) {
      const uint16_t* kb = reinterpret_cast<const uint16_t*>(st + SL.key);
      const uint16_t* qb = reinterpret_cast<const uint16_t*>(st + SL.q);
      for (int e = t; e < (n + 1) * N; e += kThreads) sK[e] = bf(kb[e]);
      for (int e = t; e < N; e += kThreads) sq[e] = bf(qb[e]);
      compute_sync();
      for (int j = warp; j <= n; j += kThreads / 32) {  // one warp per record
        float aq = 0.f, ak = 0.f;
        for (int e = lane; e < N; e += 32) {
          const float kv = sK[j * N + e];
          aq = fmaf(kv, sq[e], aq);
          if (KIND == 1) ak = fmaf(kv, sK[n * N + e], ak);
        }
        aq = seg_sum<32>(aq);
        if (KIND == 1) ak = seg_sum<32>(ak);
        if (lane == 0) {
          sdot[j] = aq;
          if (KIND == 1) sdot2[j] = ak;
        }
      }
      compute_sync();
    }

    const bool fast = (N == 128) && (READ == READ_NONE || ui.flush);
    if (fast && ui.ok) {
      // ======== warp-local unit: warp w owns rows w, w+8, ...; lane = column chunk ========
      const int RW = P / 8;  // rows per warp
      if (KIND == 0) {
        const uint16_t* xb = reinterpret_cast<const uint16_t*>(st + SL.rec);
        const uint16_t* dtr = reinterpret_cast<const uint16_t*>(st + SL.dt);
        const uint16_t* dtc = reinterpret_cast<const uint16_t*>(st + SL.chunk);
        const float dt_cur = bf(dtc[u & 7]);
        const float la_cur = dt_cur * chunk[4 + (ui.h & 3)];
        // records 0..n (current at n): w_j = exp(sum_{i=j+1..n} la_i), gamma = exp(sum_{i<=n} la_i)
        const float v = suffix_sum(lane < n ? la_slot[slot_lane] : (lane == n ? la_cur : 0.f), lane, n);
        const float excl = __shfl_down_sync(0xffffffffu, v, 1);
        const float Wl = lane <= n ? expf(lane < n ? excl : 0.f) : 0.f;
        const float gamma = expf(__shfl_sync(0xffffffffu, v, 0));
        const float dtl = lane < n ? bf(dtr[slot_lane]) : (lane == n ? dt_cur : 0.f);
        const float cy = lane <= n ? Wl * dtl * sdot[lane] : 0.f;  // output coefficient on x_j[r]
        const float cf = Wl * dtl;                                 // fold coefficient on x_j[r]
        const float4 q4 = reinterpret_cast<const float4*>(sq)[lane];
        const int kq = (lane >> 2) & 7, jl = lane & 3;
        for (int r0 = 0; r0 < RW; r0 += 8) {
          // buffered term of row slot kq: lanes 4kq..4kq+3 split the records
          const int Rq = warp + 8 * (r0 + kq);
          const bool vq = r0 + kq < RW;
          float ry = 0.f;
          for (int j0 = 0; j0 <= n; j0 += 4) {
            const int j = j0 + jl;
            const float c = __shfl_sync(0xffffffffu, cy, j & 31);
            if (j <= n && vq) ry = fmaf(c, bf(xb[j * P + Rq]), ry);
          }
          ry += __shfl_xor_sync(0xffffffffu, ry, 1);
          ry += __shfl_xor_sync(0xffffffffu, ry, 2);
          float4 s4[8];
          float part[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const bool vk = r0 + k < RW;
            s4[k] = vk ? sT4[(warp + 8 * (r0 + k)) * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
            part[k] = dot4(s4[k], q4);
          }
          const float tot = reduce8(part, lane);
          if (jl == 0 && vq) yrow[Rq] = fmaf(gamma, tot, ry);
          if (ui.flush) {
            float4 acc[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = scale4(gamma, s4[k]);
            for (int j = 0; j <= n; ++j) {
              const float4 k4 = reinterpret_cast<const float4*>(sK + j * N)[lane];
              const float c = __shfl_sync(0xffffffffu, cf, j);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const int R = warp + 8 * (r0 + k);
                if (r0 + k < RW) acc[k] = axpy4(c * bf(xb[j * P + R]), k4, acc[k]);
              }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (r0 + k < RW) {
                const int f = (warp + 8 * (r0 + k)) * 32 + lane;
                __stcs(gS4 + f, acc[k]);
                if (READ != READ_NONE) sT4[f] = acc[k];
              }
            }
          }
        }
      } else {
        const float* ub = reinterpret_cast<const float*>(st + SL.rec);
        const uint16_t* vb = reinterpret_cast<const uint16_t*>(st + SL.v);
        // buffered records 0..n-1: w_j = exp(sum_{i=j+1..n-1} g_i), gamma = exp(sum_{i<n} g_i)
        const float v = suffix_sum(lane < n ? la_slot[slot_lane] : 0.f, lane, n - 1);
        const float excl = __shfl_down_sync(0xffffffffu, v, 1);
        const float Wl = lane < n ? expf(lane + 1 < n ? excl : 0.f) : 0.f;
        const float gamma = n > 0 ? expf(__shfl_sync(0xffffffffu, v, 0)) : 1.f;
        const float a = expf(chunk[u & 3]);
        const float beta = chunk[4 + (u & 3)];
        const float kq_dot = sdot[n];
        const float ck = lane < n ? Wl * sdot2[lane] : 0.f;   // coefficient of u_j[r] in S k
        const float cq = lane < n ? Wl * sdot[lane] : 0.f;    // coefficient of u_j[r] in S q
        const float cf = a * Wl;                              // fold coefficient of u_j[r]
        const float4 q4 = reinterpret_cast<const float4*>(sq)[lane];
        const float4 k4c = reinterpret_cast<const float4*>(sK + n * N)[lane];
        float* urow = d.r_u + (u * C + slot) * P;
        const int kq = (lane >> 2) & 7, jl = lane & 3;
        for (int r0 = 0; r0 < RW; r0 += 8) {
          const int Rq = warp + 8 * (r0 + kq);
          const bool vq = r0 + kq < RW;
          float rk = 0.f, rq = 0.f;
          for (int j0 = 0; j0 < n; j0 += 4) {
            const int j = j0 + jl;
            const float c1 = __shfl_sync(0xffffffffu, ck, j & 31);
            const float c2 = __shfl_sync(0xffffffffu, cq, j & 31);
            if (j < n && vq) {
              const float uj = ub[j * P + Rq];
              rk = fmaf(c1, uj, rk);
              rq = fmaf(c2, uj, rq);
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
            const bool vk = r0 + k < RW;
            s4[k] = vk ? sT4[(warp + 8 * (r0 + k)) * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
            pk[k] = dot4(s4[k], k4c);
            pq[k] = dot4(s4[k], q4);
          }
          const float Sk = fmaf(gamma, reduce8(pk, lane), rk);
          const float Sq = fmaf(gamma, reduce8(pq, lane), rq);
          const float uu = vq ? beta * (bf(vb[Rq]) - a * Sk) : 0.f;
          if (jl == 0 && vq) {
            yrow[Rq] = fmaf(a, Sq, uu * kq_dot);
            if (!ui.flush) urow[Rq] = uu;
          }
          if (ui.flush) {
            float4 acc[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              acc[k] = axpy4(__shfl_sync(0xffffffffu, uu, 4 * k), k4c, scale4(a * gamma, s4[k]));
            for (int j = 0; j < n; ++j) {
              const float4 k4 = reinterpret_cast<const float4*>(sK + j * N)[lane];
              const float c = __shfl_sync(0xffffffffu, cf, j);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const int R = warp + 8 * (r0 + k);
                if (r0 + k < RW) acc[k] = axpy4(c * ub[j * P + R], k4, acc[k]);
              }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (r0 + k < RW) __stcs(gS4 + (warp + 8 * (r0 + k)) * 32 + lane, acc[k]);
            }
          }
        }
      }
    } else if (ui.ok) {
      // ======== shared-memory path (d_state < 128, or a read-copy non-flush unit) ========
      if (warp == 0) {
        if (KIND == 0) {
          const uint16_t* dtc = reinterpret_cast<const uint16_t*>(st + SL.chunk);
          const float dt_cur = bf(dtc[u & 7]);
          const float la_cur = dt_cur * chunk[4 + (ui.h & 3)];
          const float v = suffix_sum(lane < n ? la_slot[slot_lane] : (lane == n ? la_cur : 0.f), lane, n);
          const float excl = __shfl_down_sync(0xffffffffu, v, 1);
          if (lane <= n) sW[lane] = expf(lane < n ? excl : 0.f);
          if (lane == 0) {
            sW[C] = expf(v);
            sW[C + 1] = dt_cur;
            sW[C + 2] = la_cur;
          }
        } else {
          const float v = suffix_sum(lane < n ? la_slot[slot_lane] : 0.f, lane, n - 1);
          const float excl = __shfl_down_sync(0xffffffffu, v, 1);
          if (lane < n) sW[lane] = expf(lane + 1 < n ? excl : 0.f);
          if (lane == 0) {
            sW[C] = n > 0 ? expf(v) : 1.f;
            sW[C + 1] = expf(chunk[u & 3]);
            sW[C + 2] = chunk[4 + (u & 3)];
          }
        }
      }
      compute_sync();
      if (KIND == 0) {
        const uint16_t* xb = reinterpret_cast<const uint16_t*>(st + SL.rec);
        const uint16_t* dtr = reinterpret_cast<const uint16_t*>(st + SL.dt);
        const float dt_cur = sW[C + 1];
        for (int r = t; r < P; r += kThreads) {
          float acc = 0.f;
          for (int j = 0; j <= n; ++j) {
            const float dtj = j < n ? bf(dtr[ring_slot(ui.head, j, C)]) : dt_cur;
            const float v = dtj * bf(xb[j * P + r]);
            acc = fmaf(sW[j] * sdot[j], v, acc);
            if (ui.flush) scoef[j * P + r] = sW[j] * v;
          }
          srow[r] = acc;
        }
      } else {
        const float* ub = reinterpret_cast<const float*>(st + SL.rec);
        const float a = sW[C + 1];
        for (int r = t; r < P; r += kThreads) {
          float ak = 0.f, aq = 0.f;
          for (int j = 0; j < n; ++j) {
            const float wu = sW[j] * ub[j * P + r];
            ak = fmaf(wu, sdot2[j], ak);
            aq = fmaf(wu, sdot[j], aq);
            if (ui.flush) scoef[j * P + r] = a * wu;
          }
          srow[r] = ak;
          srow2[r] = aq;
        }
      }
      compute_sync();
      const float gamma = sW[C];
      if (KIND == 0) {
        const float4 q4 = reinterpret_cast<const float4*>(sq)[c4];
        if (!ui.flush && READ == READ_FP8) {
          const unsigned char* sC = st + SL.tile;
          rc_rows_fp8<N>(sC, reinterpret_cast<const float*>(sC + tile), sq, P, gamma, srow, yrow);
        } else if (!ui.flush && READ == READ_NVFP4) {
          const unsigned char* sC = st + SL.tile;
          rc_rows_nvfp4<N>(sC, sC + tile / 2, chunk[8 + (u & 3)], sq, P, gamma, srow, yrow);
        } else if (!ui.flush) {
          for (int f = t; f < nf4; f += kThreads) {
            const float part = seg_sum<SEG>(dot4(sT4[f], q4));
            if (c4 == 0) yrow[f / SEG] = fmaf(gamma, part, srow[f / SEG]);
          }
        } else {
          for (int f = t; f < nf4; f += kThreads) {
            const float4 s4 = sT4[f];
            const int r = f / SEG;
            const float part = seg_sum<SEG>(dot4(s4, q4));
            if (c4 == 0) yrow[r] = fmaf(gamma, part, srow[r]);
            float4 acc = scale4(gamma, s4);
            for (int j = 0; j <= n; ++j)
              acc = axpy4(scoef[j * P + r], reinterpret_cast<const float4*>(sK + j * N)[c4], acc);
            __stcs(gS4 + f, acc);
            sT4[f] = acc;
          }
        }
      } else {
        const float4 q4 = reinterpret_cast<const float4*>(sq)[c4];
        const float4 k4 = reinterpret_cast<const float4*>(sK + n * N)[c4];
        const float a = sW[C + 1], beta = sW[C + 2], kq = sdot[n];
        const uint16_t* vb = reinterpret_cast<const uint16_t*>(st + SL.v);
        float* urow = d.r_u + (u * C + slot) * P;
        for (int f = t; f < nf4; f += kThreads) {
          const float4 s4 = sT4[f];
          const int r = f / SEG;
          const float pk = seg_sum<SEG>(dot4(s4, k4));
          const float pq = seg_sum<SEG>(dot4(s4, q4));
          const float Sk = fmaf(gamma, pk, srow[r]);
          const float Sq = fmaf(gamma, pq, srow2[r]);
          const float uu = beta * (bf(vb[r]) - a * Sk);
          if (c4 == 0) {
            yrow[r] = fmaf(a, Sq, uu * kq);
            if (!ui.flush) urow[r] = uu;
          }
          if (ui.flush) {
            float4 acc = axpy4(uu, k4, scale4(a * gamma, s4));
            for (int j = 0; j < n; ++j)
              acc = axpy4(scoef[j * P + r], reinterpret_cast<const float4*>(sK + j * N)[c4], acc);
            __stcs(gS4 + f, acc);
          }
        }
      }
    }

    // ---- flush: refresh the read copy from the folded matrix in shared memory ----
    if (READ != READ_NONE && ui.ok && ui.flush) {
      compute_sync();
      write_read_copy<N, READ>(d, static_cast<int>(u), reinterpret_cast<const float*>(st + SL.tile), sred);
    }

    // ---- append this token's record (non-flush units) ----
    if (ui.ok && !ui.flush) {
      if (KIND == 0) {
        const uint16_t* xb = reinterpret_cast<const uint16_t*>(st + SL.rec);
        for (int r = t; r < P; r += kThreads) d.r_x[(u * C + slot) * P + r] = xb[n * P + r];
        if (t == 0) {
          const uint16_t* dtc = reinterpret_cast<const uint16_t*>(st + SL.chunk);
          d.r_dt[u * Cp + slot] = dtc[u & 7];
          d.r_la[u * Cp + slot] = bf(dtc[u & 7]) * chunk[4 + (ui.h & 3)];
        }
      } else {
        if (t == 0) d.r_g[u * Cp + slot] = chunk[u & 3];
      }
      if (ui.h % hpg == 0) {
        const uint16_t* kb = reinterpret_cast<const uint16_t*>(st + SL.key);
        const size_t bg = static_cast<size_t>(ui.b) * G + ui.g;
        uint16_t* rk = (KIND == 0 ? d.r_B : d.r_k) + (bg * C + slot) * N;
        for (int e = t; e < N; e += kThreads) rk[e] = kb[n * N + e];
      }
    }

    compute_sync();  // every computing thread is done with stage s
    if (t == 0) mbar_arrive(empty + s);
  }
  // after an abort: let the copies already issued land before the CTA exits
  if (smisc[0] && t == 0) {
    const uint64_t t0 = global_ns();
    while (smisc[1] < min(consumed + stages, nunits) && global_ns() - t0 < 1000000000ull) {
    }
    const int issued = smisc[1];
    for (int j = consumed; j < issued; ++j)
      mbar_wait_bounded(full + (j % stages), static_cast<uint32_t>((j / stages) & 1));
  }
}

int stages_for(const LayerDev& d) {
  const Stage SL = stage_layout(d.kind, d.P, d.N, d.C, d.Cp);
  const Persist PL = persist_layout(d.P, d.N, d.C);
  const long budget = 227L * 1024 - static_cast<long>(PL.size_floats) * 4;
  long s = budget / SL.size;
  if (s > 8) s = 8;
  return static_cast<int>(s);
}

template <int KIND, int N, int READ>
cudaError_t launch_one(const LayerDev& d, const TokenIn& in, float* y, cudaStream_t s) {
  const int stages = stages_for(d);
  if (stages < 1) return cudaErrorInvalidConfiguration;
  const Stage SL = stage_layout(d.kind, d.P, d.N, d.C, d.Cp);
  const Persist PL = persist_layout(d.P, d.N, d.C);
  const size_t smem = static_cast<size_t>(SL.size) * stages + static_cast<size_t>(PL.size_floats) * 4;
  const int total = d.B * d.H;
  int grid = d.num_sms > 0 ? d.num_sms : 1;
  if (grid > total) grid = total;
  int per = (total + grid - 1) / grid;
  while (per / d.H + 2 > kMaxSeq) {  // bound the sequences one CTA covers
    grid *= 2;
    per = (total + grid - 1) / grid;
  }
  grid = (total + per - 1) / per;
  auto kernel = decode_kernel<KIND, N, READ>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, decode_threads<N, READ>(), smem, s>>>(d, in, y, per, stages);
  return cudaGetLastError();
}

template <int KIND, int N>
cudaError_t launch_kn(const LayerDev& d, const TokenIn& in, float* y, cudaStream_t s) {
  if (KIND == 0 && d.read_mode == READ_FP8) return launch_one<KIND, N, READ_FP8>(d, in, y, s);
  if (KIND == 0 && d.read_mode == READ_NVFP4) return launch_one<KIND, N, READ_NVFP4>(d, in, y, s);
  return launch_one<KIND, N, READ_NONE>(d, in, y, s);
}

}  // namespace

size_t decode_smem_bytes(const LayerDev& d) {
  const Stage SL = stage_layout(d.kind, d.P, d.N, d.C, d.Cp);
  const Persist PL = persist_layout(d.P, d.N, d.C);
  return static_cast<size_t>(SL.size) + static_cast<size_t>(PL.size_floats) * 4;
}

cudaError_t launch_decode(const LayerDev& d, const TokenIn& in, float* y, cudaStream_t s) {
  if (d.kind == RS_KDA) return launch_kda_decode(d, in, y, s);
  // d_state 128, d_head 64 or 128: the grouped kernel (decode128.cu)
  if (decode128_supports(d)) return launch_decode128(d, in, y, s);
  if (d.kind == 0) {
    switch (d.N) {
      case 16: return launch_kn<0, 16>(d, in, y, s);
      case 32: return launch_kn<0, 32>(d, in, y, s);
      case 64: return launch_kn<0, 64>(d, in, y, s);
      case 128: return launch_kn<0, 128>(d, in, y, s);
    }
  } else {
    switch (d.N) {
      case 16: return launch_kn<1, 16>(d, in, y, s);
      case 32: return launch_kn<1, 32>(d, in, y, s);
      case 64: return launch_kn<1, 64>(d, in, y, s);
      case 128: return launch_kn<1, 128>(d, in, y, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace rs
