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
//  * a flush unit folds the records into the matrix in shared memory and a bulk
//    store writes the checkpoint back once; a non-flush unit stores no state.
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
  p.bars = (o + 3) & ~3;         // 16-byte aligned, up to 8 mbarriers (u64)
  o = p.bars + 2 * 8;
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

__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

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
template <int KIND, int N, int READ>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const LayerDev d, const TokenIn in,
                                                             float* __restrict__ y, const int units_per_cta,
                                                             const int stages) {
  constexpr int SEG = N / 4;  // lanes per state row, one float4 each
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
  uint64_t* bars = reinterpret_cast<uint64_t*>(pf + PL.bars);
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
  if (t == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(bars + s, 1);
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

  // --- producer: stage the inputs of unit i (thread 0 only) ---
  auto issue = [&](int i) {
    const UnitInfo ui = unit_info(i);
    unsigned char* st = smem + static_cast<size_t>(SL.size) * (i % stages);
    uint64_t* bar = bars + (i % stages);
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
    if (ui.first_of_group) bytes += static_cast<uint32_t>(n + 1) * N * 2 + N * 2;  // keys + q
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
    if (ui.first_of_group) {
      const uint16_t* rk = (KIND == 0 ? d.r_B : d.r_k) + bg * C * N;
      copy_in(st + SL.key, rk + static_cast<size_t>(ui.head) * N, seg1 * N * 2, bar);
      copy_in(st + SL.key + seg1 * N * 2, rk, seg2 * N * 2, bar);
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
  };

  if (t == 0) {
    for (int i = 0; i < min(stages, nunits); ++i) issue(i);
  }

  const int c4 = t % SEG;
  for (int i = 0; i < nunits; ++i) {
    const UnitInfo ui = unit_info(i);
    unsigned char* st = smem + static_cast<size_t>(SL.size) * (i % stages);
    const uint32_t parity = static_cast<uint32_t>((i / stages) & 1);
    const bool arrived = __syncthreads_and(mbar_wait_bounded(bars + (i % stages), parity) ? 1 : 0) != 0;
    if (!arrived) {
      if (t == 0) {
        report_error(d.err, DEVERR_TIMEOUT, ui.b);
        // wait (bounded) for every copy already issued, then stop
        for (int j = i; j < min(i + stages, nunits); ++j)
          mbar_wait_bounded(bars + (j % stages), static_cast<uint32_t>((j / stages) & 1));
      }
      __syncthreads();
      break;
    }
    const size_t u = static_cast<size_t>(ui.u);
    const int n = ui.n;
    const int slot = ring_slot(ui.head, n, C);
    const int slot_lane = lane < n ? ring_slot(ui.head, lane, C) : 0;

    // ---- per group: keys, query and their dot products (once per group) ----
    if (ui.first_of_group) {
      const uint16_t* kb = reinterpret_cast<const uint16_t*>(st + SL.key);
      const uint16_t* qb = reinterpret_cast<const uint16_t*>(st + SL.q);
      for (int e = t; e < (n + 1) * N; e += kThreads) sK[e] = bf(kb[e]);
      for (int e = t; e < N; e += kThreads) sq[e] = bf(qb[e]);
      __syncthreads();
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
    }

    // ---- decay weights (warp 0): suffix sums of log decays ----
    const float* la_slot = reinterpret_cast<const float*>(st + SL.la);
    const float* chunk = reinterpret_cast<const float*>(st + SL.chunk);
    if (warp == 0) {
      if (KIND == 0) {
        // records 0..n (current at n): w_j = exp(sum_{i=j+1..n} la_i), gamma = exp(sum_{i<=n} la_i)
        const uint16_t* dtc = reinterpret_cast<const uint16_t*>(st + SL.chunk);
        const float dt_cur = bf(dtc[u & 7]);
        const float la_cur = dt_cur * chunk[4 + (ui.h & 3)];
        float v = lane < n ? la_slot[slot_lane] : (lane == n ? la_cur : 0.f);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float w = __shfl_down_sync(0xffffffffu, v, o);
          if (lane + o <= n) v += w;
        }
        const float excl = __shfl_down_sync(0xffffffffu, v, 1);
        if (lane <= n) sW[lane] = expf(lane < n ? excl : 0.f);
        if (lane == 0) {
          sW[C] = expf(v);
          sW[C + 1] = dt_cur;
          sW[C + 2] = la_cur;
        }
      } else {
        // buffered records 0..n-1: w_j = exp(sum_{i=j+1..n-1} g_i), gamma = exp(sum_{i<n} g_i)
        float v = lane < n ? la_slot[slot_lane] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float w = __shfl_down_sync(0xffffffffu, v, o);
          if (lane + o < n) v += w;
        }
        const float excl = __shfl_down_sync(0xffffffffu, v, 1);
        if (lane < n) sW[lane] = expf(lane + 1 < n ? excl : 0.f);
        if (lane == 0) {
          sW[C] = n > 0 ? expf(v) : 1.f;
          sW[C + 1] = expf(chunk[u & 3]);
          sW[C + 2] = chunk[4 + (u & 3)];
        }
      }
    }
    __syncthreads();

    // ---- per-row buffered terms; fold coefficients on flush units ----
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
    __syncthreads();

    // ---- one pass over the state matrix ----
    float* yrow = y + u * P;
    float4* sT4 = reinterpret_cast<float4*>(st + SL.tile);
    const int nf4 = tile / 4;
    const float gamma = sW[C];
    if (ui.ok) {
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
            sT4[f] = acc;
          }
        }
      }
    }

    // ---- flush: write the folded matrix back once (bulk store), refresh the read copy ----
    if (ui.ok && ui.flush) {
      fence_proxy_async();
      __syncthreads();
      if (t == 0) bulk_s2g(d.ckpt + u * tile, st + SL.tile, static_cast<uint32_t>(tile) * 4u);
      if (READ != READ_NONE)
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
          d.r_la[u * Cp + slot] = sW[C + 2];
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

    __syncthreads();  // stage i % stages is free
    if (t == 0 && i + stages < nunits) {
      if (ui.ok && ui.flush) bulk_wait_read_all();  // the bulk store has read the stage
      issue(i + stages);
    }
  }
  if (t == 0) bulk_wait_all();
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
  kernel<<<grid, kThreads, smem, s>>>(d, in, y, per, stages);
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
