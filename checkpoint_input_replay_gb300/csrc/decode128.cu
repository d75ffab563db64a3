// Standard decode step for d_state = 128 and d_head 64 or 128 (the layer
// shapes the workloads use): the output-only non-flush body and the flush
// body, per sequence, in one persistent launch.  Same arithmetic as decode.cu
// (the unrolled checkpoint-plus-buffer form of "ReplaySSM caches SSM inputs
// instead of state" (richland.au), "What shipped"); this file differs in how
// the work is fed and split, so that the computing warps do little besides the
// pass over the state matrix:
//
//  * a work unit is one (sequence, head) state matrix [P][128] -- a Gated
//    DeltaNet head of d_head 128 is two units of 64 rows; on a layer with a
//    low-precision read copy, the non-flush units hold four heads of a group,
//    whose codes fit where one FP32 matrix goes -- and CTA c owns a contiguous
//    range of units, so it meets each group (and sequence) once;
//  * a producer warp stages each unit with bulk copies (cp.async.bulk): the
//    state matrix (or its read copy) and the buffered records of that head.
//    What the heads of a group share, or what is small -- the group's keys and
//    query, the current tokens of all its heads, the ring's per-head decay rows,
//    the current per-head scalars, the read-copy scales -- is staged once per
//    group, one group ahead, into one of three group buffers;
//  * two builder warps, one group ahead of the computing warps: the query (and
//    current key) in FP32, the group's key dot products (eight keys per
//    transpose-reduce; on Gated DeltaNet layers, whose groups hold two heads,
//    one builder takes the k_j . q and the other the k_j . k_cur), the per-head
//    coefficient tables (one decay suffix scan per head; on Mamba-2 layers two
//    heads at once in 16-lane halves when the records fit, on Gated DeltaNet
//    layers one head per builder), and the ring appends of the group's current
//    tokens;
//  * a prologue warp publishes per unit a 16-byte descriptor and signals
//    `ready` (at a group's first unit, once its tables are in place);
//  * the eight computing warps form one or two teams that take units in turn;
//    a team's warps own rows w, w+T, .. of each of its units: lane = 4
//    columns, 4 lanes per row split the buffered records, an 8-row
//    transpose-reduce forms the row sums.  A flush unit folds in registers:
//    each warp writes the fold coefficients of its 8 rows into a small table
//    in shared memory, reads them back four records at a time by broadcast,
//    and accumulates with packed fma.rn.f32x2; it stores the checkpoint once.
//    No barrier spans the warps, except an NVFP4 flush unit, whose matrix
//    amax is exchanged through a bounded mbarrier.
#include "common.cuh"

namespace rs {
namespace {

constexpr int N = 128;               // d_state of this kernel
constexpr int SEG = N / 4;           // lanes per state row (one float4 each)
constexpr int kMaxSeq128 = 64;       // sequences one CTA may cover
// the weighted work split (batches up to kBalanceMaxB sequences): relative cost of
// a unit that folds this step and of one that does not (measured: flush step
// ~2.2x a non-flush step at the workload shapes)
constexpr int kBalanceMaxB = 4096;
constexpr int kWPlain = 4, kWFlush = 9;
constexpr int kThreads128 = kThreads + 128;  // 8 computing warps, prologue, producer, 2 builders
constexpr int kPrologueWarp = kThreads / 32;
constexpr int kProducerWarp = kThreads / 32 + 1;
constexpr int kBuilderWarp = kThreads / 32 + 2;  // first builder warp
constexpr int kGroupBufs = 3;                    // group buffers (staged one group ahead)
// row stride (floats) of a warp's fold-coefficient table: kMaxRec padded so the
// 32 lanes' stores (8 rows x 4 records) fall in 32 different banks
constexpr int kMtabRow = kMaxRec + 4;
// rows of a warp's fold-coefficient table: 16 where a flush unit folds both of a
// warp's 8-row blocks in one pass (Mamba-2, d_head 64, FP32 reads), else 8
__host__ __device__ __forceinline__ constexpr int mtab_rows(int kind, int read, int P) {
  return (kind == 0 && read == 0 && P == 64) ? 16 : 8;
}

__host__ __device__ __forceinline__ int al16(int x) { return (x + 15) & ~15; }
__host__ __device__ __forceinline__ int al128(int x) { return (x + 127) & ~127; }
// floats per head in a coefficient table: 3 rows of C record coefficients, 8 scalars
__host__ __device__ __forceinline__ int coef_stride(int C) { return (3 * C + 8 + 3) & ~3; }

// per-head scalars after the 3C record coefficients
enum : int { CO_GAMMA = 0, CO_A = 1, CO_BETA = 2, CO_KQ = 3, CO_MATSCALE = 4 };

// Shared-memory layout (bytes): [stages][3 group buffers][persistent].
struct Lay128 {
  int st_tile, st_rec, st_meta, st_size, rec_stride, urow;
  int gb_key, gb_q, gb_cur, gb_la, gb_dt, gb_s1, gb_s2, gb_rs, gb_ms, gb_qf, gb_kf, gb_coef, gb_size;
  int pe_A, pe_bars, pe_seq, pe_misc, pe_cnt, pe_mtab, pe_dq, pe_size;
};

// Barriers of the two builder warps (named barrier 3, 64 threads); the _and form
// returns whether `v` held in both.
__device__ __forceinline__ void builder_pair_sync() { asm volatile("bar.sync 3, 64;" ::: "memory"); }
__device__ __forceinline__ bool builder_pair_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 3, 64, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

// heads in a non-flush unit of a read-copy layer: 4 heads' codes fit where one
// FP32 matrix goes, and the unit's fixed costs are shared by 4 heads
__host__ __device__ __forceinline__ int read_heads(int read) { return read == READ_NONE ? 1 : 4; }

// units per head: a Gated DeltaNet head of d_head 128 is two units of 64 rows,
// so that a stage holds 32 KB of state and five stages fit
__host__ __device__ __forceinline__ int splits(int kind, int P) { return (kind == 1 && P == 128) ? 2 : 1; }


__host__ __device__ __forceinline__ Lay128 lay128(int kind, int read, int P, int C, int Cp, int H, int hpg) {
  Lay128 l;
  int o = 0;
  const int rpu = P / splits(kind, P);  // state rows per unit
  l.st_tile = o;  o += rpu * N * 4;
  // a read-copy unit's heads' record blocks sit 16 bytes off the 128-byte bank period
  l.rec_stride = al16(C * P * 2) + (read == READ_NONE ? 0 : 16);
  // Gated DeltaNet records are staged whole (all P rows of u_j, both units of a
  // head), by at most two copies per unit
  l.urow = P;
  l.st_rec = o;   o += kind == 0 ? read_heads(read) * l.rec_stride : C * l.urow * 4;
  l.st_meta = o;  o += 32;              // int4 descriptor, NVFP4 amax word
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
  l.gb_qf = o;    o += N * 4;
  l.gb_kf = o;    o += kind == 0 ? 0 : N * 4;
  l.gb_coef = o;  o += hpg * coef_stride(C) * 4;
  l.gb_size = al128(o);
  o = 0;
  l.pe_A = o;     o += al16(H * 4);
  l.pe_bars = o;  o += 48 * 8;  // full, empty, ready x 8 stages; amax x 2 teams x 8 stages; group full, tables x 3
  l.pe_seq = o;   o += 3 * kMaxSeq128 * 4;
  l.pe_misc = o;  o += 16;
  l.pe_cnt = o;   o += 16;  // computing warps that have finished this CTA's units
  l.pe_mtab = o;  o += (kThreads / 32) * mtab_rows(kind, read, P) * kMtabRow * 4;  // per computing warp: fold coefficients [rows][records]
  l.pe_dq = o;    o += 2 * 2 * kMaxRec * 4;                 // key dots: per builder (Mamba-2) or per group parity (GDN)
  l.pe_size = al128(o);
  return l;
}

// the weighted work split needs the batch's per-sequence weights in shared memory
// (in the computing warps' fold tables, before they are used), and its weight sums
// (units x kWFlush at most) in 32 bits
__host__ __device__ __forceinline__ bool balanced(const Lay128& l, int B, int upseq) {
  return B <= kBalanceMaxB && ((B + 3) & ~3) * 4 + B * 8 + 8 <= l.pe_dq - l.pe_mtab &&
         static_cast<long long>(B) * upseq * kWFlush < (1LL << 30);
}

__device__ __forceinline__ int ring_slot(int head, int j, int C) {
  int s = head + j;
  return s >= C ? s - C : s;
}

// One warp: count this CTA in on the launch-wide counter (arrive[0]); the last CTA
// advances every sequence's cursor and returns the counter to zero.
__device__ __forceinline__ void finish_launch(const LayerDev& d, int lane, int C, int L) {
  int last = 0;
  if (lane == 0) {
    __threadfence();
    last = atomicAdd(d.arrive, 1) == static_cast<int>(gridDim.x) - 1;
  }
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  // eight cursors a lane per round: all loads of a round before its stores
  for (int b0r = 0; b0r < d.B; b0r += 8 * 32) {
    int4 cur[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int b = b0r + 32 * k + lane;
      cur[k] = b < d.B ? reinterpret_cast<const int4*>(d.cursor)[b] : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int b = b0r + 32 * k + lane;
      if (b >= d.B) continue;
      const int head = cur[k].x, cnt = cur[k].y;
      if (static_cast<unsigned>(head) >= static_cast<unsigned>(C) || static_cast<unsigned>(cnt) >= static_cast<unsigned>(L)) {
        report_error(d.err, DEVERR_CURSOR, b);
      } else if (cnt + 1 == L) {
        reinterpret_cast<int4*>(d.cursor)[b] = make_int4(ring_slot(head, cnt + 1, C), 0, 1, cur[k].w);
      } else {
        reinterpret_cast<int4*>(d.cursor)[b] = make_int4(head, cnt + 1, 0, cur[k].w);
      }
    }
  }
  if (lane == 0) atomicExch(d.arrive, 0);
}


// Position of a unit: its index ui, sequence b, head (u = b H + h), group g,
// head-in-group hh and part sp of a split head; advanced one unit at a time so
// that no role divides per unit.
struct Walk {
  int ui, u, b, h, g, hh, sp;
  __device__ __forceinline__ void start(int u0, int H, int hpg, int spl) {
    ui = u0;
    b = u0 / (H * spl);
    const int r = u0 - b * H * spl;
    h = r / spl;
    sp = r - h * spl;
    u = b * H + h;
    g = h / hpg;
    hh = h - g * hpg;
  }
  // advance one unit: the next part of a split head, or `step` heads (1, or HR
  // for a non-flush read-copy unit; HR divides heads-per-group and H)
  __device__ __forceinline__ void next(int H, int hpg, int step, int spl) {
    if (spl > 1) {
      ++ui;
      if (++sp < spl) return;
      sp = 0;
      step = 1;
    } else {
      ui += step;
    }
    u += step;
    h += step;
    hh += step;
    if (hh == hpg) {
      hh = 0;
      ++g;
    }
    if (h == H) {
      h = 0;
      g = 0;
      ++b;
    }
  }
};

// Position of a group: sequence b, group g, and its first head-in-group hh0, part
// sp0 and unit index ui0 in this CTA (a CTA's first group may start mid-group).
struct GWalk {
  int b, g, hh0, sp0, ui0;
  __device__ __forceinline__ void start(int u0, int H, int hpg, int spl) {
    b = u0 / (H * spl);
    const int r = u0 - b * H * spl;
    const int h = r / spl;
    sp0 = r - h * spl;
    g = h / hpg;
    hh0 = h - g * hpg;
    ui0 = u0;
  }
  __device__ __forceinline__ void next(int H, int G, int hpg, int spl) {
    if (++g == G) {
      g = 0;
      ++b;
    }
    hh0 = 0;
    sp0 = 0;
    ui0 = (b * H + g * hpg) * spl;
  }
  // one past the last head-in-group of this group that has a unit in [ui0, u1)
  __device__ __forceinline__ int hh_end(int u1, int hpg, int spl) const {
    return min(hpg, hh0 + (u1 - ui0 + sp0 + spl - 1) / spl);
  }
};

// TEAMS: the eight computing warps form TEAMS teams of 8 / TEAMS warps; team t
// takes units t, t + TEAMS, ..., so that TEAMS units are computed at once
template <int KIND, int READ, int P, int TEAMS>
__global__ void __launch_bounds__(kThreads128, 1) decode128_kernel(const LayerDev d, const TokenIn in,
                                                                   float* __restrict__ y, const int units_per_cta,
                                                                   const int stages) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int SPL = (KIND == 1 && P == 128) ? 2 : 1;  // units per head
  constexpr int RPU = P / SPL;                          // state rows per unit
  static_assert(TEAMS == 1 || TEAMS == 2 || TEAMS == 4, "teams: a power of two dividing the 8 computing warps");
  constexpr int TW = 8 / TEAMS;                         // warps of a team
  constexpr int RW = RPU / TW;                          // rows per computing warp and unit
  constexpr int NB = 2;                                  // builder warps
  constexpr int tile = P * N;                           // floats of one head's state
  constexpr int HR = READ == READ_NONE ? 1 : 4;         // heads of a non-flush read-copy unit
  const int H = d.H, G = d.G, C = d.C, L = d.L, Cp = d.Cp;
  const int hpg = H / G;
  const int CS = coef_stride(C);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const Lay128 LY = lay128(KIND, READ, P, C, Cp, H, hpg);
  unsigned char* gbase = smem + static_cast<size_t>(LY.st_size) * stages;
  unsigned char* pbase = gbase + kGroupBufs * LY.gb_size;
  const float* sA = reinterpret_cast<const float*>(pbase + LY.pe_A);
  uint64_t* full = reinterpret_cast<uint64_t*>(pbase + LY.pe_bars);
  uint64_t* empty = full + 8;
  uint64_t* ready = full + 16;
  uint64_t* amaxbar = full + 24;  // [team][stage]: NVFP4 matrix amax of a flushed unit
  uint64_t* gfull = full + 40;    // [group buffer]: the group's copies have landed
  uint64_t* tready = full + 43;   // [group buffer]: the group's tables are in place
  int* sseq = reinterpret_cast<int*>(pbase + LY.pe_seq);
  // abort, unit copies issued, producer done, group copies issued
  volatile int* smisc = reinterpret_cast<volatile int*>(pbase + LY.pe_misc);
  // this warp's fold-coefficient table (computing warps)
  constexpr int MR = mtab_rows(KIND, READ, P);
  float* mt = reinterpret_cast<float*>(pbase + LY.pe_mtab) + (warp < kThreads / 32 ? warp : 0) * MR * kMtabRow;

  const int upseq = H * SPL;  // units of a sequence
  const int total_units = d.B * upseq;
  const int cta = cta_index(d.cta_mult);
  int u0, u1;
  const bool bal = balanced(LY, d.B, upseq) && !d.uniform_split;
  // scratch before the computing warps' fold tables are used: per-sequence weights,
  // the batch's cursors (head, count) and the two range bounds
  int* wts = reinterpret_cast<int*>(pbase + LY.pe_mtab);
  int2* snap = reinterpret_cast<int2*>(wts + ((d.B + 3) & ~3));
  int* sbound = reinterpret_cast<int*>(snap + d.B);
  if (bal) {
    // Work split by weight: a unit of a sequence that folds this step costs about
    // kWFlush / kWPlain times a non-flush unit, so in a batch whose sequences are
    // at different window positions the CTAs take equal shares of the weighted
    // total rather than of the units.  Every CTA computes every boundary from the
    // same cursors: no CTA changes a cursor before all have read them (below).
    for (int b = t; b < d.B; b += kThreads128) {
      const int2 hc = reinterpret_cast<const int2*>(d.cursor)[2 * b];
      const int head = hc.x, cnt = hc.y;
      const bool fl = static_cast<unsigned>(head) < static_cast<unsigned>(C) &&
                      static_cast<unsigned>(cnt) < static_cast<unsigned>(L) && cnt + 1 == L;
      wts[b] = fl ? kWFlush : kWPlain;
      snap[b] = make_int2(head, cnt);
    }
    __syncthreads();
    if (warp == 0) {
      // 32-bit sums (the launcher keeps total_units * kWFlush below 2^31) and
      // constant divisors: this scan delays every CTA's first copy
      const int per_l = (d.B + 31) / 32;
      const int lo = min(lane * per_l, d.B), hi = min(lo + per_l, d.B);
      int sw = 0;
      for (int b = lo; b < hi; ++b) sw += wts[b];
      int incl = sw;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int W = __shfl_sync(0xffffffffu, incl, 31) * upseq;
      const int cum0 = (incl - sw) * upseq;  // weight before this lane's first sequence
      const int share = (W + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        // units whose weight interval starts before T = (cta + e) ceil(W / grid): with
        // equal weights these are the even split's boundaries
        const int T = min(W, (cta + e) * share);
        int cum = cum0;
        int cntu = 0;
        for (int b = lo; b < hi; ++b) {
          const int w = wts[b];
          if (T > cum) {
            const int x = T - cum;
            cntu += min(upseq, w == kWPlain ? (x + kWPlain - 1) / kWPlain : (x + kWFlush - 1) / kWFlush);
          }
          cum += w * upseq;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cntu += __shfl_xor_sync(0xffffffffu, cntu, o);
        // a non-flush read-copy unit spans HR heads; the last CTA ends the batch
        if (lane == 0) sbound[e] = (e == 1 && cta + 1 == static_cast<int>(gridDim.x)) ? total_units : cntu - cntu % HR;
      }
    }
    __syncthreads();
    u0 = sbound[0];
    u1 = sbound[1];
  } else {
    u0 = cta * units_per_cta;
    u1 = min(u0 + units_per_cta, total_units);
  }
  const int b0 = u0 / upseq, b1 = u1 > u0 ? (u1 - 1) / upseq : b0;
  const int nseq = u1 > u0 ? b1 - b0 + 1 : 0;

  // --- cursors of the covered sequences ---
  if (t < nseq) {
    const int b = b0 + t;
    const int2 hc = bal ? snap[b] : make_int2(d.cursor[4 * b], d.cursor[4 * b + 1]);
    const int head = hc.x, cnt = hc.y;
    const bool ok = static_cast<unsigned>(head) < static_cast<unsigned>(C) &&
                    static_cast<unsigned>(cnt) < static_cast<unsigned>(L);
    sseq[3 * t] = ok ? head : 0;  // a rejected cursor stages nothing from the ring
    sseq[3 * t + 1] = ok ? cnt : 0;
    sseq[3 * t + 2] = ok ? 1 : 0;
  }
  if (t == kThreads) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, TW);
      mbar_init(ready + s, 1);
      for (int k = 0; k < TEAMS; ++k) mbar_init(amaxbar + 8 * k + s, TW);
    }
    for (int k = 0; k < kGroupBufs; ++k) {
      mbar_init(gfull + k, 1);
      mbar_init(tready + k, NB);
    }
    smisc[0] = 0;
    smisc[1] = 0;
    smisc[2] = 0;
    smisc[3] = 0;
    *reinterpret_cast<int*>(pbase + LY.pe_cnt) = 0;
  }
  __syncthreads();
  // An empty CTA counts itself in at once (the others when their units are done, at the end)
  if (u0 >= u1) {
    if (warp == 0) finish_launch(d, lane, C, L);
    return;
  }

  // heads in the unit that starts at sequence b: HR unless b flushes this step
  auto step_of = [&](int b) {
    const int k = b - b0;
    return (HR > 1 && !(sseq[3 * k + 2] != 0 && sseq[3 * k + 1] + 1 == L)) ? HR : 1;
  };
  // first element of the 16-byte block holding element e, for 2-byte / 4-byte arrays
  auto blk2 = [](size_t e) { return e & ~static_cast<size_t>(7); };
  auto blk4 = [](size_t e) { return e & ~static_cast<size_t>(3); };

  // =============================== producer warp ===============================
  if (warp == kProducerWarp) {
    if (lane != 0) return;
    // the copies of group gw (its buffer x, barrier gfull[x]): keys and query,
    // current tokens, decay rows, scalars, scales (and A with the first group)
    auto stage_group = [&](const GWalk& gw, int x, bool with_A) {
      const int k = gw.b - b0;
      const int head = sseq[3 * k], n = sseq[3 * k + 1];
      const int seg1 = min(n, C - head), seg2 = n - seg1;
      const size_t ug = static_cast<size_t>(gw.b) * H + static_cast<size_t>(gw.g) * hpg;  // first head
      const size_t bg = static_cast<size_t>(gw.b) * G + gw.g;
      const uint32_t s1b = KIND == 0 ? static_cast<uint32_t>((blk2(ug + hpg + 7) - blk2(ug)) * 2)
                                     : static_cast<uint32_t>((blk4(ug + hpg + 3) - blk4(ug)) * 4);
      const uint32_t s4b = static_cast<uint32_t>((blk4(ug + hpg + 3) - blk4(ug)) * 4);
      uint32_t bytes = static_cast<uint32_t>(n + 1) * N * 2 + N * 2 + hpg * P * 2 + hpg * Cp * 4 + s1b;
      if (KIND == 0) bytes += hpg * Cp * 2;
      else bytes += s4b;
      if (READ == READ_FP8) bytes += hpg * P * 4;
      if (READ == READ_NVFP4) bytes += hpg * P * (N / 16) + s4b;
      if (with_A) bytes += al16(H * 4);
      unsigned char* gb = gbase + static_cast<size_t>(LY.gb_size) * x;
      uint64_t* bar = gfull + x;
      mbar_expect_tx(bar, bytes);
      const uint16_t* rk = (KIND == 0 ? d.r_B : d.r_k) + bg * C * N;
      if (seg1) bulk_g2s(gb + LY.gb_key, rk + static_cast<size_t>(head) * N, seg1 * N * 2, bar);
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
      if (with_A) bulk_g2s(pbase + LY.pe_A, in.A, al16(H * 4), bar);
    };
    Walk w;
    w.start(u0, H, hpg, SPL);
    GWalk gn;  // the next group to stage
    gn.start(u0, H, hpg, SPL);
    int gi = -1, staged = 0;
    int si = 0;        // stage of unit i
    uint32_t ph = 0;   // parity of the stage's uses before unit i
    for (int i = 0; w.ui < u1; ++i, w.next(H, hpg, step_of(w.b), SPL)) {
      const int s = si;
      const uint32_t par = ph ^ 1u;  // release of the stage's previous unit
      if (++si == stages) {
        si = 0;
        ph ^= 1u;
      }
      if (i >= stages && !mbar_try_wait(empty + s, par)) {
        if (smisc[0] || !mbar_wait_bounded(empty + s, par)) break;
      }
      const bool first = i == 0 || (w.hh == 0 && w.sp == 0);
      if (first) ++gi;
      // group buffers: the CTA's first group with its first unit, then group gi + 1
      // at the first unit of group gi (its buffer's earlier group, gi - 2, has left
      // the pipeline: stages <= units per group + 1)
      if (i == 0) {
        stage_group(gn, 0, KIND == 0);
        gn.next(H, G, hpg, SPL);
        smisc[3] = staged = 1;
      }
      const int k = w.b - b0;
      const int head = sseq[3 * k], n = sseq[3 * k + 1];
      const bool flush = sseq[3 * k + 2] != 0 && n + 1 == L;
      unsigned char* st = smem + static_cast<size_t>(LY.st_size) * s;
      uint64_t* bar = full + s;
      const size_t u = static_cast<size_t>(w.u);
      const int seg1 = min(n, C - head), seg2 = n - seg1;
      constexpr int esz = KIND == 0 ? 2 : 4;
      const int nh = step_of(w.b);  // heads in this unit
      const uint32_t tb = (READ == READ_NONE || flush) ? RPU * N * 4 : (READ == READ_FP8 ? tile : tile / 2);
      mbar_expect_tx(bar, nh * (tb + static_cast<uint32_t>(n) * (KIND == 0 ? RPU : P) * esz));
      // the unit: state matrix (or read copy) and this head's buffered records
      if (READ == READ_NONE || flush) bulk_g2s(st + LY.st_tile, d.ckpt + u * tile + w.sp * RPU * N, tb, bar);
      else bulk_g2s(st + LY.st_tile, d.rc_codes + u * tb, nh * tb, bar);  // nh consecutive heads
      const unsigned char* rsrc = KIND == 0 ? reinterpret_cast<const unsigned char*>(d.r_x)
                                            : reinterpret_cast<const unsigned char*>(d.r_u);
      constexpr size_t rrow = static_cast<size_t>(P) * esz;
      if (KIND == 0) {
        for (int hu = 0; hu < nh; ++hu) {
          unsigned char* rdst = st + LY.st_rec + static_cast<size_t>(hu) * LY.rec_stride;
          const size_t uh = u + hu;
          if (seg1) bulk_g2s(rdst, rsrc + (uh * C + head) * rrow, seg1 * rrow, bar);
          if (seg2) bulk_g2s(rdst + seg1 * rrow, rsrc + uh * C * rrow, seg2 * rrow, bar);
        }
      } else {
        // the head's buffered records, whole (the ring's slots are contiguous up to the wrap)
        if (seg1) bulk_g2s(st + LY.st_rec, rsrc + (u * C + head) * rrow, seg1 * rrow, bar);
        if (seg2) bulk_g2s(st + LY.st_rec + seg1 * rrow, rsrc + u * C * rrow, seg2 * rrow, bar);
      }
      smisc[1] = i + 1;
      if (first && gn.ui0 < u1) {
        stage_group(gn, (gi + 1) % kGroupBufs, false);
        gn.next(H, G, hpg, SPL);
        smisc[3] = ++staged;
      }
    }
    smisc[2] = 1;
    return;
  }

  // =============================== builder warps ===============================
  if (warp >= kBuilderWarp) {
    const int bi = warp - kBuilderWarp;
    if (bi >= NB) return;
    float* pdq = reinterpret_cast<float*>(pbase + LY.pe_dq) + bi * 2 * kMaxRec;  // k_j . q (Mamba-2)
    GWalk gw;
    gw.start(u0, H, hpg, SPL);
    int built = 0;
    for (int gi = 0; gw.ui0 < u1; ++gi, gw.next(H, G, hpg, SPL)) {
      const int x = gi % kGroupBufs;
      if (KIND == 1) {
        // the two builders split each group's work and meet at a barrier, so they
        // decide together whether to go on
        const bool go = !smisc[0] && mbar_wait_bounded(gfull + x, static_cast<uint32_t>((gi / kGroupBufs) & 1));
        if (!builder_pair_and(go)) {
          if (lane == 0 && !smisc[0]) {
            report_error(d.err, DEVERR_TIMEOUT, gw.b);
            smisc[0] = 1;
          }
          break;
        }
      } else {
        if (smisc[0]) break;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(gfull + x, static_cast<uint32_t>((gi / kGroupBufs) & 1)))) {
          if (lane == 0) {
            report_error(d.err, DEVERR_TIMEOUT, gw.b);
            smisc[0] = 1;
          }
          break;
        }
      }
      built = gi + 1;
      const int k = gw.b - b0;
      const int head = sseq[3 * k], n = sseq[3 * k + 1];
      const bool ok = sseq[3 * k + 2] != 0;
      const bool flush = ok && n + 1 == L;
      const int slot = ring_slot(head, n, C);
      unsigned char* gb = gbase + static_cast<size_t>(LY.gb_size) * x;
      const size_t ug = static_cast<size_t>(gw.b) * H + static_cast<size_t>(gw.g) * hpg;  // first head of the group
      const int hh_hi = gw.hh_end(u1, hpg, SPL);
      const uint16_t* kb = reinterpret_cast<const uint16_t*>(gb + LY.gb_key);
      if (ok) {
        // the query (and current key) in FP32
        const float4 q4 = bf4(reinterpret_cast<const uint2*>(gb + LY.gb_q)[lane]);
        const float4 kc4 = bf4(reinterpret_cast<const uint2*>(kb + n * N)[lane]);
        if (bi == 0) {
          reinterpret_cast<float4*>(gb + LY.gb_qf)[lane] = q4;
          if (KIND == 1) reinterpret_cast<float4*>(gb + LY.gb_kf)[lane] = kc4;
        }
        // key dot products of records 0..n, eight keys per transpose-reduce (Gated
        // DeltaNet: builder 0 the k_j . q, builder 1 the k_j . k_cur, into tables of
        // the group's parity that both read)
        float* gdq = reinterpret_cast<float*>(pbase + LY.pe_dq) + (gi & 1) * 2 * kMaxRec;
        float* gdk = gdq + kMaxRec;
        const float4 o4 = (KIND == 1 && bi == 1) ? kc4 : q4;
        for (int jb = 0; jb <= n; jb += 8) {
          float pq[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 kj = jb + e <= n ? bf4(reinterpret_cast<const uint2*>(kb + (jb + e) * N)[lane])
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
            pq[e] = dot4(kj, o4);
          }
          const float tq = reduce8(pq, lane);
          const int j = jb + (lane >> 2);
          if ((lane & 3) == 0 && j <= n) {
            if (KIND == 0) pdq[j] = tq;
            else (bi == 0 ? gdq : gdk)[j] = tq;
          }
        }
        if (KIND == 1) builder_pair_sync();
        else __syncwarp();
        // coefficient tables: two heads at once in the 16-lane halves when records
        // 0..n fit in 16 lanes; passes shared out over the builders
        // (Gated DeltaNet: one head per builder and pass)
        const int sw = (KIND == 0 && n < 16) ? 16 : 32;
        const int jl = lane & (sw - 1);
        const float dq = jl <= n ? (KIND == 0 ? pdq : gdq)[jl] : 0.f;
        const float dk = (KIND == 1 && jl <= n) ? gdk[jl] : 0.f;
        const int slot_j = jl < n ? ring_slot(head, jl, C) : 0;
        for (int e0 = gw.hh0 + bi * (32 / sw); e0 < hh_hi; e0 += NB * (32 / sw)) {
          const int e = e0 + lane / sw;
          const bool act = e < hh_hi;
          const float* la_row = reinterpret_cast<const float*>(gb + LY.gb_la) + e * Cp;
          float* co = reinterpret_cast<float*>(gb + LY.gb_coef) + e * CS;
          if (KIND == 0) {
            // records 0..n (current at n): w_j = exp(sum_{i=j+1..n} la_i), gamma = exp(sum_{i<=n} la_i)
            float dt_cur = 0.f, la_cur = 0.f;
            if (act) {
              dt_cur = bf(reinterpret_cast<const uint16_t*>(gb + LY.gb_s1)[(ug & 7) + e]);
              la_cur = dt_cur * sA[gw.g * hpg + e];
            }
            float v = act ? (jl < n ? la_row[slot_j] : (jl == n ? la_cur : 0.f)) : 0.f;
            for (int o = 1; o < sw; o <<= 1) {  // suffix sums within the segment
              const float wv = __shfl_down_sync(0xffffffffu, v, o);
              if (jl + o <= n) v += wv;
            }
            const float excl = __shfl_down_sync(0xffffffffu, v, 1);
            if (act) {
              const float Wl = jl <= n ? expf(jl < n ? excl : 0.f) : 0.f;
              const uint16_t* dt_row = reinterpret_cast<const uint16_t*>(gb + LY.gb_dt) + e * Cp;
              const float dtl = jl < n ? bf(dt_row[slot_j]) : (jl == n ? dt_cur : 0.f);
              if (jl <= n) {
                co[jl] = Wl * dtl * dq;     // output coefficient on x_j[r]
                co[2 * C + jl] = Wl * dtl;  // fold coefficient on x_j[r]
              }
              if (jl == 0) {
                co[3 * C + CO_GAMMA] = expf(v);
                if (READ == READ_NVFP4)
                  co[3 * C + CO_MATSCALE] = reinterpret_cast<const float*>(gb + LY.gb_ms)[(ug & 3) + e];
              }
            }
          } else {
            // buffered records 0..n-1: w_j = exp(sum_{i=j+1..n-1} g_i), gamma = exp(sum_{i<n} g_i)
            float v = act && jl < n ? la_row[slot_j] : 0.f;
            for (int o = 1; o < sw; o <<= 1) {  // suffix sums within the segment
              const float wv = __shfl_down_sync(0xffffffffu, v, o);
              if (jl + o <= n - 1) v += wv;
            }
            const float excl = __shfl_down_sync(0xffffffffu, v, 1);
            const float kq_dot = __shfl_sync(0xffffffffu, dq, (lane & ~(sw - 1)) + n);  // k_cur . q
            if (act) {
              const float Wl = jl < n ? expf(jl + 1 < n ? excl : 0.f) : 0.f;
              const float a = expf(reinterpret_cast<const float*>(gb + LY.gb_s1)[(ug & 3) + e]);
              if (jl < n) {
                co[jl] = Wl * dk;         // coefficient of u_j[r] in S k
                co[C + jl] = Wl * dq;     // coefficient of u_j[r] in S q
                co[2 * C + jl] = a * Wl;  // fold coefficient of u_j[r]
              }
              if (jl == 0) {
                co[3 * C + CO_GAMMA] = n > 0 ? expf(v) : 1.f;
                co[3 * C + CO_A] = a;
                co[3 * C + CO_BETA] = reinterpret_cast<const float*>(gb + LY.gb_s2)[(ug & 3) + e];
                co[3 * C + CO_KQ] = kq_dot;
              }
            }
          }
        }
        if (!flush) {
          // ring appends: the current tokens of the group's heads in this CTA (a head
          // whose first part another CTA holds is appended by that CTA), and the group's
          // key row from the CTA that holds the group's first head
          for (int e = gw.hh0 + (gw.sp0 > 0 ? 1 : 0) + bi; e < hh_hi; e += NB) {
            const size_t ue = ug + e;
            if (KIND == 0) {
              const uint16_t* xc = reinterpret_cast<const uint16_t*>(gb + LY.gb_cur) + e * P;
              uint16_t* dst = d.r_x + (ue * C + slot) * P;
              if (P == 64)
                reinterpret_cast<uint32_t*>(dst)[lane] = reinterpret_cast<const uint32_t*>(xc)[lane];
              else
                reinterpret_cast<uint2*>(dst)[lane] = reinterpret_cast<const uint2*>(xc)[lane];
              if (lane == 0) {
                const uint16_t dt_bits = reinterpret_cast<const uint16_t*>(gb + LY.gb_s1)[(ug & 7) + e];
                d.r_dt[ue * Cp + slot] = dt_bits;
                d.r_la[ue * Cp + slot] = bf(dt_bits) * sA[gw.g * hpg + e];
              }
            } else if (lane == 0) {
              d.r_g[ue * Cp + slot] = reinterpret_cast<const float*>(gb + LY.gb_s1)[(ug & 3) + e];
            }
          }
          if (bi == 0 && gw.hh0 == 0 && gw.sp0 == 0) {
            const size_t bg = static_cast<size_t>(gw.b) * G + gw.g;
            reinterpret_cast<uint2*>((KIND == 0 ? d.r_B : d.r_k) + (bg * C + slot) * N)[lane] =
                reinterpret_cast<const uint2*>(kb + n * N)[lane];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(tready + x);
    }
    // after an abort: let the group copies already issued land before the CTA exits
    if (smisc[0] && bi == 0 && lane == 0) {
      const uint64_t t0 = global_ns();
      while (!smisc[2] && global_ns() - t0 < 2000000000ull) {
      }
      const int issued = smisc[3];
      for (int j = built; j < issued; ++j)
        mbar_wait_bounded(gfull + (j % kGroupBufs), static_cast<uint32_t>((j / kGroupBufs) & 1));
    }
    return;
  }

  const int kq = (lane >> 2) & 7, jl = lane & 3;

  // =============================== prologue warp ===============================
  if (warp == kPrologueWarp) {
    Walk w;
    w.start(u0, H, hpg, SPL);
    int gi = -1, gx = 0, consumed = 0;
    int si = 0;
    uint32_t ph = 0;
    for (int i = 0; w.ui < u1; ++i, w.next(H, hpg, step_of(w.b), SPL)) {
      const int s = si;
      const uint32_t par = ph;
      if (++si == stages) {
        si = 0;
        ph ^= 1u;
      }
      if (!__all_sync(0xffffffffu, mbar_try_wait(full + s, par))) {
        if (smisc[0]) break;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(full + s, par))) {
          if (lane == 0) {
            report_error(d.err, DEVERR_TIMEOUT, w.b);
            smisc[0] = 1;
          }
          break;
        }
      }
      consumed = i + 1;
      const bool first = i == 0 || (w.hh == 0 && w.sp == 0);
      if (first) {
        ++gi;
        gx = gi % kGroupBufs;
        // the group's tables are in place
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(tready + gx, static_cast<uint32_t>((gi / kGroupBufs) & 1)))) {
          if (lane == 0) {
            report_error(d.err, DEVERR_TIMEOUT, w.b);
            smisc[0] = 1;
          }
          break;
        }
      }
      if (lane == 0) {
        const int k = w.b - b0;
        const int head = sseq[3 * k], n = sseq[3 * k + 1];
        const bool ok = sseq[3 * k + 2] != 0;
        const bool flush = ok && n + 1 == L;
        unsigned char* st = smem + static_cast<size_t>(LY.st_size) * s;
        *reinterpret_cast<int4*>(st + LY.st_meta) =
            make_int4(w.u, n | (flush ? 0x100 : 0) | (ok ? 0x200 : 0) | (first ? 0x400 : 0),
                      ring_slot(head, n, C), w.hh | (gx << 16) | (w.sp << 24));
        reinterpret_cast<int*>(st + LY.st_meta)[4] = 0;  // NVFP4 matrix amax
        mbar_arrive(ready + s);
      }
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
  const int team = warp / TW, tw = warp - team * TW;  // team, warp in the team
  uint32_t amax_phase = 0;
  Walk wc;
  wc.start(u0, H, hpg, SPL);
  int si = 0;
  uint32_t ph = 0;
  for (int i = 0; wc.ui < u1; ++i, wc.next(H, hpg, step_of(wc.b), SPL)) {
    const int s = si;
    const uint32_t par = ph;
    if (++si == stages) {
      si = 0;
      ph ^= 1u;
    }
    if (TEAMS > 1 && (i & (TEAMS - 1)) != team) continue;
    // the abort flag is read only when the unit is not ready at the first poll
    if (!__all_sync(0xffffffffu, mbar_try_wait(ready + s, par))) {
      if (smisc[0]) break;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(ready + s, par))) {
        if (lane == 0) {
          report_error(d.err, DEVERR_TIMEOUT, wc.b);
          smisc[0] = 1;
        }
        break;
      }
    }
    unsigned char* st = smem + static_cast<size_t>(LY.st_size) * s;
    const int4 meta = *reinterpret_cast<const int4*>(st + LY.st_meta);
    const int nh_unit = (READ != READ_NONE && !(meta.y & 0x100)) ? HR : 1;  // heads of this unit
    if constexpr (KIND == 0 && READ != READ_NONE) if (nh_unit == HR && (meta.y & 0x200)) {
      // Non-flush unit of a read-copy layer: HR heads of one group; warp tw takes
      // rows RW tw .. RW tw + RW - 1 of each.  Codes: in pass f, lane 8 rq + cb
      // decodes channels 16 cb .. 16 cb + 15 of row RW tw + 4 f + rq (one 16- or
      // 8-byte shared load, one NVFP4 block scale), and the eight lanes of a row
      // add their block dot products by a transpose-reduce that leaves each
      // (head, row) total in one lane.  That lane also sums the row's buffered
      // records (lanes of a warp read 16 distinct banks: the heads' record
      // blocks are 16 bytes off the 128-byte period) and writes y.
      static_assert(HR == 4 && RW % 4 == 0 && (RW / 4 * HR) % 8 == 0, "read-copy unit shape");
      constexpr int NPASS = RW / 4;
      constexpr int NV = NPASS * HR;  // block dot products per lane, reduced 8 at a time
      const int n = meta.y & 0xFF;
      const int hh0 = meta.w & 0xFFFF;
      const size_t uh0 = static_cast<size_t>(meta.x);
      const unsigned char* gb = gbase + static_cast<size_t>(LY.gb_size) * ((meta.w >> 16) & 3);
      const float* cob = reinterpret_cast<const float*>(gb + LY.gb_coef);
      const uint16_t* curb = reinterpret_cast<const uint16_t*>(gb + LY.gb_cur);
      constexpr int TBH = READ == READ_FP8 ? tile : tile / 2;  // code bytes per head
      const int rq = lane >> 3, cbk = lane & 7;
      float2 qv[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 q4 = reinterpret_cast<const float4*>(gb + LY.gb_qf)[4 * cbk + i];
        qv[2 * i] = make_float2(q4.x, q4.y);
        qv[2 * i + 1] = make_float2(q4.z, q4.w);
      }
      float v[NV];
#pragma unroll
      for (int f = 0; f < NPASS; ++f) {
        const int R = RW * tw + 4 * f + rq;
#pragma unroll
        for (int hu = 0; hu < HR; ++hu) {
          const unsigned char* cbp = st + LY.st_tile + hu * TBH;
          float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
          if (READ == READ_FP8) {
            const uint4 wv = *reinterpret_cast<const uint4*>(cbp + R * N + 16 * cbk);
            const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              a0 = fma2(e4m3x2_to_f32x2(static_cast<uint16_t>(wd[i] & 0xFFFFu)), qv[2 * i], a0);
              a1 = fma2(e4m3x2_to_f32x2(static_cast<uint16_t>(wd[i] >> 16)), qv[2 * i + 1], a1);
            }
            v[f * HR + hu] = (a0.x + a0.y) + (a1.x + a1.y);
          } else {
            const uint2 wv = *reinterpret_cast<const uint2*>(cbp + R * (N / 2) + 8 * cbk);
            const uint32_t wd[2] = {wv.x, wv.y};
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              float2 c[4];
              e2m1x8_to_f32x2(wd[i], c);
              a0 = fma2(c[0], qv[4 * i], a0);
              a1 = fma2(c[1], qv[4 * i + 1], a1);
              a0 = fma2(c[2], qv[4 * i + 2], a0);
              a1 = fma2(c[3], qv[4 * i + 3], a1);
            }
            const float bs = e4m3_to_f32(gb[LY.gb_rs + ((hh0 + hu) * P + R) * (N / 16) + cbk]);
            v[f * HR + hu] = bs * ((a0.x + a0.y) + (a1.x + a1.y));
          }
        }
      }
#pragma unroll
      for (int g = 0; g < NV / 8; ++g) {
        // this lane's total: value 8 g + cb, i.e. head cb mod 4, pass 2 g + cb / 4
        const float tot = reduce8_lanes3(v + 8 * g, lane);
        const int hu = cbk & 3;
        const int R = RW * tw + 4 * (2 * g + (cbk >> 2)) + rq;
        const float* co = cob + (hh0 + hu) * CS;
        const uint16_t* xr = reinterpret_cast<const uint16_t*>(st + LY.st_rec + hu * LY.rec_stride) + R;
        float r0 = co[n] * bf(curb[(hh0 + hu) * P + R]), r1 = 0.f;
        int j = 0;
        for (; j + 1 < n; j += 2) {
          r0 = fmaf(co[j], bf(xr[j * P]), r0);
          r1 = fmaf(co[j + 1], bf(xr[(j + 1) * P]), r1);
        }
        if (j < n) r0 = fmaf(co[j], bf(xr[j * P]), r0);
        const float gsc = co[3 * C + CO_GAMMA] * (READ == READ_FP8
                                                      ? reinterpret_cast<const float*>(gb + LY.gb_rs)[(hh0 + hu) * P + R]
                                                      : co[3 * C + CO_MATSCALE]);
        y[(uh0 + hu) * P + R] = fmaf(gsc, tot, r0 + r1);
      }
    }
    for (int hu = 0; hu < 1 && nh_unit == 1 && (meta.y & 0x200); ++hu) {
      const size_t u = static_cast<size_t>(meta.x) + hu;
      const int n = meta.y & 0xFF;
      const bool flush = (meta.y & 0x100) != 0;
      const int slot = meta.z;
      const int hh = (meta.w & 0xFFFF) + hu;
      const int sp = meta.w >> 24;  // part of a split head: rows sp RPU .. sp RPU + RPU - 1
      const unsigned char* gb = gbase + static_cast<size_t>(LY.gb_size) * ((meta.w >> 16) & 3);
      const float* co = reinterpret_cast<const float*>(gb + LY.gb_coef) + hh * CS;
      const uint16_t* kb = reinterpret_cast<const uint16_t*>(gb + LY.gb_key);
      const uint16_t* cur = reinterpret_cast<const uint16_t*>(gb + LY.gb_cur) + hh * P + sp * RPU;  // x or v
      float* yrow = y + u * P + sp * RPU;
      float4* sT4 = reinterpret_cast<float4*>(st + LY.st_tile);
      float4* gS4 = reinterpret_cast<float4*>(d.ckpt + u * tile + sp * RPU * N);
      const float4 q4 = reinterpret_cast<const float4*>(gb + LY.gb_qf)[lane];
      const float gamma = co[3 * C + CO_GAMMA];
      if (KIND == 0) {
        const uint16_t* xb = reinterpret_cast<const uint16_t*>(st + LY.st_rec + static_cast<size_t>(hu) * LY.rec_stride);
        if (MR == 16 && RW == 16 && flush) {
          // flush unit, both of this warp's 8-row blocks in one pass over the records:
          // the keys are loaded once for the two, and the two blocks' accumulations
          // interleave (table rows 8 bk + kq hold block bk's fold coefficients)
          float4 acc[2][8];
#pragma unroll
          for (int bk = 0; bk < 2; ++bk) {
            const int Rq = tw + TW * (8 * bk + kq);
            float ry = jl == 0 ? co[n] * bf(cur[Rq]) : 0.f;
            for (int j = jl; j < n; j += 4) ry = fmaf(co[j], bf(xb[j * P + Rq]), ry);
            ry += __shfl_xor_sync(0xffffffffu, ry, 1);
            ry += __shfl_xor_sync(0xffffffffu, ry, 2);
            float part[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float4 s4 = sT4[(tw + TW * (8 * bk + e)) * SEG + lane];
              part[e] = dot4(s4, q4);
              acc[bk][e] = scale4(gamma, s4);
            }
            const float tot = reduce8(part, lane);
            if (jl == 0) yrow[Rq] = fmaf(gamma, tot, ry);
            for (int jc = 0; 4 * jc <= n; ++jc) {
              const int j = 4 * jc + jl;
              mt[(8 * bk + kq) * kMtabRow + j] = j <= n ? co[2 * C + j] * bf(j < n ? xb[j * P + Rq] : cur[Rq]) : 0.f;
            }
          }
          __syncwarp();
          for (int jq = 0; 4 * jq <= n; ++jq) {
            float4 k4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              k4[i] = 4 * jq + i <= n ? bf4(reinterpret_cast<const uint2*>(kb + (4 * jq + i) * N)[lane])
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float4 m4 = *reinterpret_cast<const float4*>(mt + e * kMtabRow + 4 * jq);
              float4& a = acc[e >> 3][e & 7];
              a = axpy4x2(m4.x, k4[0], a);
              a = axpy4x2(m4.y, k4[1], a);
              a = axpy4x2(m4.z, k4[2], a);
              a = axpy4x2(m4.w, k4[3], a);
            }
          }
          __syncwarp();
#pragma unroll
          for (int e = 0; e < 16; ++e) __stcs(gS4 + (tw + TW * e) * SEG + lane, acc[e >> 3][e & 7]);
        }
#pragma unroll
        for (int r0 = 0; r0 < RW && !(MR == 16 && RW == 16 && flush); r0 += 8) {
          const int Rq = tw + TW * (r0 + kq);
          // buffered term of row Rq: lanes 4kq..4kq+3 split the records 0..n-1, lane jl = 0 adds record n
          float ry = jl == 0 ? co[n] * bf(cur[Rq]) : 0.f;
          for (int j = jl; j < n; j += 4) ry = fmaf(co[j], bf(xb[j * P + Rq]), ry);
          ry += __shfl_xor_sync(0xffffffffu, ry, 1);
          ry += __shfl_xor_sync(0xffffffffu, ry, 2);
          float4 s4[8];
          float part[8];
          float row_scale = 1.f;
          if (READ != READ_NONE && !flush) {
            // non-flush: the checkpoint term from the low-precision copy of head hu of the unit
            const unsigned char* cb = st + LY.st_tile + hu * (READ == READ_FP8 ? tile : tile / 2);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int R = tw + TW * (r0 + e);
              if (READ == READ_FP8) {
                const uint32_t wd = reinterpret_cast<const uint32_t*>(cb + R * N)[lane];
                const float2 lo = e4m3x2_to_f32x2(static_cast<uint16_t>(wd & 0xFFFFu));
                const float2 hi = e4m3x2_to_f32x2(static_cast<uint16_t>(wd >> 16));
                part[e] = dot4p(make_float4(lo.x, lo.y, hi.x, hi.y), q4);
              } else {
                const uint32_t wd = reinterpret_cast<const uint16_t*>(cb + R * (N / 2))[lane];
                const float2 lo = e2m1x2_to_f32x2(wd & 0xFFu);
                const float2 hi = e2m1x2_to_f32x2(wd >> 8);
                const float bs = e4m3_to_f32(gb[LY.gb_rs + (hh * P + R) * (N / 16) + (lane >> 2)]);
                part[e] = bs * dot4p(make_float4(lo.x, lo.y, hi.x, hi.y), q4);
              }
            }
            row_scale = READ == READ_FP8 ? reinterpret_cast<const float*>(gb + LY.gb_rs)[hh * P + Rq]
                                         : co[3 * C + CO_MATSCALE];
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              s4[e] = sT4[(tw + TW * (r0 + e)) * SEG + lane];
              part[e] = dot4(s4[e], q4);
            }
          }
          const float tot = reduce8(part, lane);
          if (jl == 0) yrow[Rq] = fmaf(gamma * row_scale, tot, ry);
          if (flush) {
            // m_j[row] = w_j dt_j x_j[row] for records j = 0..n (current at n) into this warp's
            // table (lane (kq, jl) writes records jl, jl + 4, .. of row slot kq; zero past n to
            // the end of the last quad), then four records per broadcast read
            for (int jc = 0; 4 * jc <= n; ++jc) {
              const int j = 4 * jc + jl;
              mt[kq * kMtabRow + j] = j <= n ? co[2 * C + j] * bf(j < n ? xb[j * P + Rq] : cur[Rq]) : 0.f;
            }
            __syncwarp();
            float4 acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = scale4(gamma, s4[e]);
            for (int jq = 0; 4 * jq <= n; ++jq) {
              float4 k4[4];
#pragma unroll
              for (int i = 0; i < 4; ++i)
                k4[i] = 4 * jq + i <= n ? bf4(reinterpret_cast<const uint2*>(kb + (4 * jq + i) * N)[lane])
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float4 m4 = *reinterpret_cast<const float4*>(mt + e * kMtabRow + 4 * jq);
                acc[e] = axpy4x2(m4.x, k4[0], acc[e]);
                acc[e] = axpy4x2(m4.y, k4[1], acc[e]);
                acc[e] = axpy4x2(m4.z, k4[2], acc[e]);
                acc[e] = axpy4x2(m4.w, k4[3], acc[e]);
              }
            }
            __syncwarp();
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              __stcs(gS4 + (tw + TW * (r0 + e)) * SEG + lane, acc[e]);
              if (READ == READ_NVFP4 && RW != 8) sT4[(tw + TW * (r0 + e)) * SEG + lane] = acc[e];
            }
            if (READ == READ_NVFP4 && RW == 8) {
              // NVFP4 with the warp's rows all in registers: the head's amax over the team
              // (its matrix scale), then these rows' codes straight from the registers
              float mloc = 0.f;
#pragma unroll
              for (int e = 0; e < 8; ++e)
                mloc = fmaxf(mloc, fmaxf(fmaxf(fabsf(acc[e].x), fabsf(acc[e].y)), fmaxf(fabsf(acc[e].z), fabsf(acc[e].w))));
              mloc = seg_max<32>(mloc);
              int* slot_amax = reinterpret_cast<int*>(st + LY.st_meta) + 4;
              if (lane == 0) atomicMax(slot_amax, __float_as_int(mloc));  // non-negative floats order as ints
              __syncwarp();
              if (lane == 0) mbar_arrive(amaxbar + 8 * team + s);
              const bool got =
                  __all_sync(0xffffffffu, mbar_wait_bounded(amaxbar + 8 * team + s, (amax_phase >> s) & 1u));
              amax_phase ^= 1u << s;
              if (!got) {
                if (lane == 0) {
                  report_error(d.err, DEVERR_TIMEOUT, static_cast<int>(u / H));
                  smisc[0] = 1;
                }
              } else {
                const float amax = __int_as_float(*reinterpret_cast<volatile int*>(slot_amax));
                const float smat = __fdiv_rn(amax, 2688.0f);  // 448 * 6
                const float six_s = __fmul_rn(6.0f, smat);
                const float r6 = six_s != 0.0f ? __frcp_rn(six_s) : 0.0f;
                uint16_t* codes = reinterpret_cast<uint16_t*>(d.rc_codes + u * (tile / 2));
                uint8_t* blk = d.rc_blkscale + u * (tile / 16);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const int R = tw + TW * (r0 + e);
                  const float4 v4 = acc[e];
                  float mb = fmaxf(fmaxf(fabsf(v4.x), fabsf(v4.y)), fmaxf(fabsf(v4.z), fabsf(v4.w)));
                  mb = seg_max<4>(mb);  // 4 lanes = one 16-element block
                  uint32_t bcode = 0;
                  if (six_s != 0.0f) bcode = f32x2_to_e4m3x2(div_by(mb, six_s, r6), 0.0f) & 0xFFu;
                  const float dd = __fmul_rn(e4m3_to_f32(bcode), smat);
                  uint32_t qv = 0;
                  if (dd != 0.0f) {
                    const float rd = __frcp_rn(dd);
                    qv = f32x4_to_e2m1x4(div_by(v4.x, dd, rd), div_by(v4.y, dd, rd), div_by(v4.z, dd, rd),
                                         div_by(v4.w, dd, rd));
                  }
                  codes[R * SEG + lane] = static_cast<uint16_t>(qv);
                  if ((lane & 3) == 0) blk[R * (N / 16) + (lane >> 2)] = static_cast<uint8_t>(bcode);
                }
                if (tw == 0 && lane == 0) d.rc_matscale[u] = smat;
              }
            }
            if (READ == READ_FP8) {
              // refresh the FP8 copy of these eight rows from the folded rows in registers:
              // the rows' amax by one transpose-reduce, then per row scale = amax / 448 and
              // code = e4m3(x / scale), both divisions correctly rounded
              float am[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                am[e] = fmaxf(fmaxf(fabsf(acc[e].x), fabsf(acc[e].y)), fmaxf(fabsf(acc[e].z), fabsf(acc[e].w)));
              const float amx = reduce8_max(am, lane);  // row (lane >> 2) & 7
              uint32_t* codes = reinterpret_cast<uint32_t*>(d.rc_codes + u * tile);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int R = tw + TW * (r0 + e);
                const float mx = __shfl_sync(0xffffffffu, amx, 4 * e);
                const float scale = div_by(mx, 448.0f, kInv448);
                uint32_t packed = 0;
                if (scale != 0.0f) {
                  const float rs = __frcp_rn(scale);
                  const uint32_t lo = f32x2_to_e4m3x2(div_by(acc[e].x, scale, rs), div_by(acc[e].y, scale, rs));
                  const uint32_t hi = f32x2_to_e4m3x2(div_by(acc[e].z, scale, rs), div_by(acc[e].w, scale, rs));
                  packed = lo | (hi << 16);
                }
                codes[R * SEG + lane] = packed;
                if (lane == 0) d.rc_rowscale[u * P + R] = scale;
              }
            }
          }
        }
        if (READ == READ_NVFP4 && RW != 8 && flush) {
          // refresh the NVFP4 copy of this warp's rows from the folded rows in shared memory
          // (the matrix scale needs the amax of the whole head first)
          {
            float mloc = 0.f;
#pragma unroll
            for (int m = 0; m < RW; ++m) {
              const float4 v4 = sT4[(tw + TW * m) * SEG + lane];
              mloc = fmaxf(mloc, fmaxf(fmaxf(fabsf(v4.x), fabsf(v4.y)), fmaxf(fabsf(v4.z), fabsf(v4.w))));
            }
            mloc = seg_max<32>(mloc);
            int* slot_amax = reinterpret_cast<int*>(st + LY.st_meta) + 4;
            if (lane == 0) atomicMax(slot_amax, __float_as_int(mloc));  // non-negative floats order as ints
            __syncwarp();
            if (lane == 0) mbar_arrive(amaxbar + 8 * team + s);
            const bool got =
                __all_sync(0xffffffffu, mbar_wait_bounded(amaxbar + 8 * team + s, (amax_phase >> s) & 1u));
            amax_phase ^= 1u << s;
            if (!got) {
              if (lane == 0) {
                report_error(d.err, DEVERR_TIMEOUT, static_cast<int>(u / H));
                smisc[0] = 1;
              }
            } else {
              const float amax = __int_as_float(*reinterpret_cast<volatile int*>(slot_amax));
              const float smat = __fdiv_rn(amax, 2688.0f);  // 448 * 6
              const float six_s = __fmul_rn(6.0f, smat);
              const float r6 = six_s != 0.0f ? __frcp_rn(six_s) : 0.0f;
              uint16_t* codes = reinterpret_cast<uint16_t*>(d.rc_codes + u * (tile / 2));
              uint8_t* blk = d.rc_blkscale + u * (tile / 16);
#pragma unroll
              for (int m = 0; m < RW; ++m) {
                const int R = tw + TW * m;
                const float4 v4 = sT4[R * SEG + lane];
                float mb = fmaxf(fmaxf(fabsf(v4.x), fabsf(v4.y)), fmaxf(fabsf(v4.z), fabsf(v4.w)));
                mb = seg_max<4>(mb);  // 4 lanes = one 16-element block
                uint32_t bcode = 0;
                if (six_s != 0.0f) bcode = f32x2_to_e4m3x2(div_by(mb, six_s, r6), 0.0f) & 0xFFu;
                const float dd = __fmul_rn(e4m3_to_f32(bcode), smat);
                uint32_t qv = 0;
                if (dd != 0.0f) {
                  const float rd = __frcp_rn(dd);
                  qv = f32x4_to_e2m1x4(div_by(v4.x, dd, rd), div_by(v4.y, dd, rd), div_by(v4.z, dd, rd),
                                       div_by(v4.w, dd, rd));
                }
                codes[R * SEG + lane] = static_cast<uint16_t>(qv);
                if ((lane & 3) == 0) blk[R * (N / 16) + (lane >> 2)] = static_cast<uint8_t>(bcode);
              }
              if (tw == 0 && lane == 0) d.rc_matscale[u] = smat;
            }
          }
        }
      } else {
        const float* ub = reinterpret_cast<const float*>(st + LY.st_rec) + sp * RPU;  // this unit's rows
        const float4 kc4 = reinterpret_cast<const float4*>(gb + LY.gb_kf)[lane];
        const float a = co[3 * C + CO_A], beta = co[3 * C + CO_BETA];
        const float kq_dot = co[3 * C + CO_KQ];
        float* urow = d.r_u + (u * C + slot) * P + sp * RPU;
        if (!flush) {
          // Lane 8 rq + cb takes the 16 channels 4 (8 i + cb) .. + 3 (i < 4: the eight
          // lanes of a row read 128 contiguous bytes a load) of the warp's rows
          // RW tw + 4 f + rq, pass f; its 2 NPASS partial dot products (S k, S q per
          // pass) are summed over the row's eight lanes by transpose-reduces, which
          // leave S k and S q of one row in the lane pair (cb = 2 f', 2 f' + 1); that
          // pair splits the row's records by parity and writes u and o.
          constexpr int NPASS = RW / 4;
          static_assert(KIND != 1 || NPASS % 4 == 0, "rows per warp: a multiple of 16");
          const int rq = lane >> 3, cbk = lane & 7;
          float2 kv[8], qv[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 k4 = reinterpret_cast<const float4*>(gb + LY.gb_kf)[8 * i + cbk];
            const float4 qq = reinterpret_cast<const float4*>(gb + LY.gb_qf)[8 * i + cbk];
            kv[2 * i] = make_float2(k4.x, k4.y);
            kv[2 * i + 1] = make_float2(k4.z, k4.w);
            qv[2 * i] = make_float2(qq.x, qq.y);
            qv[2 * i + 1] = make_float2(qq.z, qq.w);
          }
#pragma unroll
          for (int g4 = 0; g4 < NPASS / 4; ++g4) {
            float v[8];
#pragma unroll
            for (int f4 = 0; f4 < 4; ++f4) {
              const int R = RW * tw + 4 * (4 * g4 + f4) + rq;
              float2 ak0 = make_float2(0.f, 0.f), ak1 = ak0, aq0 = ak0, aq1 = ak0;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 s4 = sT4[R * SEG + 8 * i + cbk];
                const float2 lo = make_float2(s4.x, s4.y), hi = make_float2(s4.z, s4.w);
                ak0 = fma2(lo, kv[2 * i], ak0);
                ak1 = fma2(hi, kv[2 * i + 1], ak1);
                aq0 = fma2(lo, qv[2 * i], aq0);
                aq1 = fma2(hi, qv[2 * i + 1], aq1);
              }
              v[2 * f4] = (ak0.x + ak0.y) + (ak1.x + ak1.y);
              v[2 * f4 + 1] = (aq0.x + aq0.y) + (aq1.x + aq1.y);
            }
            // this lane: value cb = dot (cb & 1) of pass 4 g4 + cb / 2
            const float tot = reduce8_lanes3(v, lane);
            const float oth = __shfl_xor_sync(0xffffffffu, tot, 1);
            const float tk = (cbk & 1) ? oth : tot, tq = (cbk & 1) ? tot : oth;
            const int R = RW * tw + 4 * (4 * g4 + (cbk >> 1)) + rq;
            float r1 = 0.f, r2 = 0.f;
            for (int j = cbk & 1; j < n; j += 2) {
              const float uj = ub[j * LY.urow + R];
              r1 = fmaf(co[j], uj, r1);
              r2 = fmaf(co[C + j], uj, r2);
            }
            r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
            r2 += __shfl_xor_sync(0xffffffffu, r2, 1);
            const float uu = beta * (bf(cur[R]) - a * fmaf(gamma, tk, r1));
            if ((cbk & 1) == 0) {
              yrow[R] = fmaf(a, fmaf(gamma, tq, r2), uu * kq_dot);
              urow[R] = uu;
            }
          }
        }
#pragma unroll
        for (int r0 = 0; r0 < RW && flush; r0 += 8) {
          const int Rq = tw + TW * (r0 + kq);
          float rk = 0.f, rq = 0.f;
          for (int j = jl; j < n; j += 4) {
            const float uj = ub[j * LY.urow + Rq];
            rk = fmaf(co[j], uj, rk);
            rq = fmaf(co[C + j], uj, rq);
          }
          rk += __shfl_xor_sync(0xffffffffu, rk, 1);
          rk += __shfl_xor_sync(0xffffffffu, rk, 2);
          rq += __shfl_xor_sync(0xffffffffu, rq, 1);
          rq += __shfl_xor_sync(0xffffffffu, rq, 2);
          float4 s4[8];
          float pk[8], pq[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            s4[e] = sT4[(tw + TW * (r0 + e)) * SEG + lane];
            pk[e] = dot4p(s4[e], kc4);
            pq[e] = dot4p(s4[e], q4);
          }
          const float tk = reduce8(pk, lane);
          const float tq = reduce8(pq, lane);
          const float Sk = fmaf(gamma, tk, rk);
          const float Sq = fmaf(gamma, tq, rq);
          const float uu = beta * (bf(cur[Rq]) - a * Sk);
          if (jl == 0) {
            yrow[Rq] = fmaf(a, Sq, uu * kq_dot);
            if (!flush) urow[Rq] = uu;
          }
          if (flush) {
            // m_j[row] = a w_j u_j[row] for records j < n into this warp's table (zero past n to
            // the end of the last quad), then four records per broadcast read
            for (int jc = 0; 4 * jc < n; ++jc) {
              const int j = 4 * jc + jl;
              mt[kq * kMtabRow + j] = j < n ? co[2 * C + j] * ub[j * LY.urow + Rq] : 0.f;
            }
            __syncwarp();
            float4 acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              acc[e] = axpy4(__shfl_sync(0xffffffffu, uu, 4 * e), kc4, scale4(a * gamma, s4[e]));
            for (int jq = 0; 4 * jq < n; ++jq) {
              float4 k4[4];
#pragma unroll
              for (int i = 0; i < 4; ++i)
                k4[i] = 4 * jq + i < n ? bf4(reinterpret_cast<const uint2*>(kb + (4 * jq + i) * N)[lane])
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float4 m4 = *reinterpret_cast<const float4*>(mt + e * kMtabRow + 4 * jq);
                acc[e] = axpy4x2(m4.x, k4[0], acc[e]);
                acc[e] = axpy4x2(m4.y, k4[1], acc[e]);
                acc[e] = axpy4x2(m4.z, k4[2], acc[e]);
                acc[e] = axpy4x2(m4.w, k4[3], acc[e]);
              }
            }
            __syncwarp();
#pragma unroll
            for (int e = 0; e < 8; ++e) __stcs(gS4 + (tw + TW * (r0 + e)) * SEG + lane, acc[e]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + s);
  }
  // This CTA's units are done (or it aborted): the last of its computing warps counts
  // the CTA in; the launch's last CTA writes every new cursor.  Every CTA read all the
  // cursors it needed before its first unit, so none can see a cursor of this step
  // already advanced.
  int done = 0;
  if (lane == 0) done = atomicAdd(reinterpret_cast<int*>(pbase + LY.pe_cnt), 1);
  if (__shfl_sync(0xffffffffu, done, 0) == kThreads / 32 - 1) finish_launch(d, lane, C, L);
}

template <int KIND, int READ, int P, int TEAMS>
cudaError_t launch128(const LayerDev& d, const TokenIn& in, float* y, cudaStream_t s) {
  const int hpg = d.H / d.G;
  const Lay128 LY = lay128(KIND, READ, P, d.C, d.Cp, d.H, hpg);
  const long budget = 227L * 1024 - static_cast<long>(kGroupBufs) * LY.gb_size - LY.pe_size;
  long stages = budget / LY.st_size;
  if (stages > 8) stages = 8;
  // a group buffer is restaged for the group three later, at the first unit of
  // the group two later: every unit of the buffer's earlier group must have left
  // the pipeline, which holds when stages <= (units per group) + 1; a non-flush
  // read-copy unit holds read_heads(READ) heads
  constexpr int SPL = (KIND == 1 && P == 128) ? 2 : 1;
  const int upg = hpg * SPL / read_heads(READ);
  if (stages > upg + 1) stages = upg + 1;
  if (stages < 1) return cudaErrorInvalidConfiguration;
  const size_t smem = static_cast<size_t>(LY.st_size) * stages + static_cast<size_t>(kGroupBufs) * LY.gb_size + LY.pe_size;
  // each CTA takes a contiguous range of heads, a multiple of read_heads(READ)
  const int hr = read_heads(READ);
  const int total = d.B * d.H * SPL;
  int grid = d.num_sms > 0 ? d.num_sms : 1;
  if (grid > total / hr) grid = total / hr;
  int per = ((total + grid - 1) / grid + hr - 1) / hr * hr;
  // a weighted share may stretch to kWFlush / kWPlain times the even share
  auto span_seqs = [&](int p) {
    return (balanced(LY, d.B, d.H * SPL) ? p * kWFlush / kWPlain : p) / (d.H * SPL) + 2;
  };
  while (span_seqs(per) > kMaxSeq128) {
    grid *= 2;
    per = ((total + grid - 1) / grid + hr - 1) / hr * hr;
  }
  grid = (total + per - 1) / per;
  auto kernel = decode128_kernel<KIND, READ, P, TEAMS>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  LayerDev dd = d;
  dd.cta_mult = coprime_mult(d.cta_mult, grid);
  kernel<<<grid, kThreads128, smem, s>>>(dd, in, y, per, static_cast<int>(stages));
  return cudaGetLastError();
}

// two computing teams where a unit is one FP32 matrix; one team on a read-copy
// layer, whose non-flush units already interleave four heads' chains
template <int P>
cudaError_t launch128_p(const LayerDev& d, const TokenIn& in, float* y, cudaStream_t s) {
  if (d.kind == 0) {
    if (d.read_mode == READ_FP8) return launch128<0, READ_FP8, P, 1>(d, in, y, s);
    if (d.read_mode == READ_NVFP4) return launch128<0, READ_NVFP4, P, 1>(d, in, y, s);
    return launch128<0, READ_NONE, P, 2>(d, in, y, s);
  }
  return launch128<1, READ_NONE, P, 2>(d, in, y, s);
}

}  // namespace

bool decode128_supports(const LayerDev& d) {
  if (d.N != N || (d.P != 64 && d.P != 128)) return false;
  // a read-copy layer's non-flush units span read_heads heads of one group
  if (d.H % read_heads(d.read_mode) != 0 || (d.H / d.G) % read_heads(d.read_mode) != 0) return false;
  const Lay128 LY = lay128(d.kind, d.read_mode, d.P, d.C, d.Cp, d.H, d.H / d.G);
  return static_cast<long>(LY.st_size) + static_cast<long>(kGroupBufs) * LY.gb_size + LY.pe_size <= 227L * 1024;
}

cudaError_t launch_decode128(const LayerDev& d, const TokenIn& in, float* y, cudaStream_t s) {
  if (!decode128_supports(d)) return cudaErrorInvalidValue;
  return d.P == 64 ? launch128_p<64>(d, in, y, s) : launch128_p<128>(d, in, y, s);
}

}  // namespace rs
