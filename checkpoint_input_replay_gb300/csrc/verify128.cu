// Speculative verification of T <= 4 draft tokens for d_state = 128 and
// d_head 64 or 128 (the layer shapes the workloads use), chunkwise form
//   O = S_ckpt Q D + V (W ⊙ (K^T Q))
// ("ReplaySSM caches SSM inputs instead of state" (richland.au), "What
// shipped", the paragraph on the second benefit), with the Gated DeltaNet
// drafts obtained by forward substitution of the unit lower-triangular T x T
// system (same arithmetic and notation as verify.cu, which serves the other
// shapes).  Two launches:
//
// 1. verify_prep_kernel, one CTA per (sequence, group): K^T Q (and K^T K_draft)
//    once for the group, then per head the decay weights W, D (and for Gated
//    DeltaNet the T x T system) folded into a coefficient table in scratch
//    memory, and the drafts' keys and per-head scalars into the ring.  This is
//    the latency-bound scalar part; thousands of independent groups hide its
//    latency.
//
// 2. verify128_kernel, the pass over the state.  A work unit is 128
//    consecutive state rows of one group: two heads of d_head 64, or one head
//    of d_head 128, so one tcgen05 MMA with M = 128 covers it.  The dense part
//    S_ckpt [128][128] x [K_draft | Q] [128][16] runs on the tensor cores in
//    kind::f16 with bf16 operands and FP32 accumulation in tensor memory.  The
//    FP32 state is split exactly into three bf16 parts, hi = bf16(S),
//    mid = bf16(S - hi), lo = bf16(S - hi - mid) (each difference is exact,
//    and 24 significand bits fit in three round-to-nearest pieces of 8), and
//    the three parts accumulate into one result: 24 MMAs of K = 16 per unit,
//    where the earlier kind::tf32 form (raw state + lo = S - trunc(S), K = 8)
//    took 32.  The A operands are read from tensor memory (an MMA with A in
//    shared memory costs about 1.7x one with A in tensor memory at these
//    shapes): the split warps write each 32-column block of the state rows,
//    as hi | mid | lo, into a ring of tensor-memory chunks that the MMA thread
//    consumes block by block.  The drafts' queries and keys are bf16 already.
//    Roles (15 warps, one persistent CTA per SM):
//     * producer (1 thread): per unit, the state tile by four 2D TMA loads
//       into one of two tile stages, and the unit's committed records and
//       coefficient tables by bulk copies into one of up to three record
//       stages; once per group, the draft keys, queries and values into one
//       of two group buffers;
//     * prologue warp: once per group, the MMA B operand; per unit a
//       descriptor;
//     * eight split warps (two per tensor-memory lane quarter, one for the
//       even and one for the odd 32-column blocks): per block, the three bf16
//       parts of the rows into a tensor-memory chunk (row r to lane r); the
//       shared-memory tile is released once it has been read;
//     * MMA thread: per chunk, two MMAs on each of the three parts, into one
//       of two accumulators;
//     * four epilogue warps: accumulator rows back from tensor memory, the
//       buffered-record terms, the triangular solve (Gated DeltaNet), outputs
//       and the drafts' x (Mamba-2) or u (Gated DeltaNet) records.
//    Every wait is bounded; on a timeout the CTA records an error and drains
//    its copies and MMAs before it frees tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tcgen05.cuh"

namespace rs {
namespace {

constexpr int N = 128;            // d_state
constexpr int kT = 4;             // drafts per verify, at most
constexpr int kNmma = 16;         // MMA N: T draft keys (GDN) and T draft queries, zero-padded
constexpr int kRows = 128;        // state rows per unit = MMA M
constexpr int kMaxSeqV = 64;      // sequences one CTA may cover
constexpr int kNT = 2;            // tile stages
constexpr int kMaxNR = 3;         // record stages, at most
constexpr uint32_t kTileBytes = kRows * N * 4;
constexpr int kSplitWarps = 8;  // two per tensor-memory lane quarter: one for the even, one for the odd blocks
constexpr int kWarpEpi = 8;      // epilogue warps 8..11
constexpr int kWarpPro = 12, kWarpProd = 13, kWarpMma = 14;
constexpr int kThreadsV = 15 * 32;
constexpr int kPrepThreads = 128;
// tensor memory: a ring of six A-operand chunks, each the 32 K-columns of one
// 128-byte block of the state rows as three bf16 parts [hi | mid | lo], 16
// columns each (two bf16 a column), then two accumulators
constexpr int kSlots = 6;
constexpr uint32_t kSlotCols = 64;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = kSlots * kSlotCols;

__host__ __device__ __forceinline__ int al16(int x) { return (x + 15) & ~15; }
__host__ __device__ __forceinline__ int al128(int x) { return (x + 127) & ~127; }

// floats per head in a coefficient table (a multiple of 4)
//   Mamba-2: C1[C][4] (output coefficient of x_j for draft position tau), D[4]
//   GDN:     C1[C][4] (coefficient of u_j in S k_tau), C2[C][4] (in S q_tau),
//            then G2[4] G1[4] a[4] beta[4] M[4][4] Qd[4][4]
__host__ __device__ __forceinline__ int head_stride(int kind, int C) { return kind == 0 ? 4 * C + 4 : 8 * C + 48; }

__device__ __forceinline__ int ring_slot(int head, int j, int C) {
  int s = head + j;
  return s >= C ? s - C : s;
}

// ============================================================================
// prep kernel
// ============================================================================
// One CTA of four warps per (sequence, group).  Its work is a short chain of
// dependent global loads, so every load is issued up front: the cursor, then
// the keys and queries together with the per-head ring scalars (up to four
// heads per warp per batch, held in registers) before any arithmetic.
constexpr int kPrepWarps = kPrepThreads / 32;
constexpr int kHB = 4;  // heads per warp per batch
constexpr int kKeyRow = N / 4 + 8;  // uint2 per padded key row (320 bytes)

// CTAs per SM the registers must allow: Mamba-2 (many heads per group, a long
// per-head phase) gains from ten; GDN (two heads per group) from fewer spills at eight
template <int KIND>
__global__ void __launch_bounds__(kPrepThreads, KIND == 0 ? 10 : 8)
    verify_prep_kernel(const LayerDev d, const TokenIn in, const int T) {
  const int H = d.H, G = d.G, C = d.C, L = d.L, Cp = d.Cp;
  const int hpg = H / G, HS = head_stride(KIND, C);
  const int bg = blockIdx.x, b = bg / G, g = bg - b * G;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  // the main kernel may be scheduled as SMs free up: it waits for this grid only
  // before it reads the coefficient tables (programmatic dependent launch)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int kNCol = KIND == 0 ? kT : 2 * kT;
  // keys of records 0..n+T-1 (committed, then drafts) as bf16, each row padded to
  // 320 bytes so that the four rows a warp reads at once fill both bank halves
  __shared__ __align__(16) uint2 skey[kMaxRec][kKeyRow];
  // dot-product columns in FP32: the draft queries in 0..3, the drafts' keys
  // (GDN) in 4..7, zero for tau >= T
  __shared__ __align__(16) float scol[kNCol][N];
  __shared__ float sdq[kMaxRec][kT];      // k_j . q_tau
  __shared__ float sdk[kMaxRec][kT];      // k_j . k_{n+tau} (GDN)

  const int head = d.cursor[4 * b], cnt = d.cursor[4 * b + 1];
  const bool ok = static_cast<unsigned>(head) < static_cast<unsigned>(C) &&
                  static_cast<unsigned>(cnt) < static_cast<unsigned>(L) && cnt + T <= C;
  if (!ok) {
    if (g == 0 && t == 0) report_error(d.err, DEVERR_CURSOR, b);
    return;
  }
  if (g == 0 && t == 0) d.cursor[4 * b + 2] = 0;  // verify folds nothing
  const int n = cnt, nr = n + T;
  const int slot_lane = lane < n ? ring_slot(head, lane, C) : 0;
  const int sigma = lane - n;  // draft index of record `lane`
  const bool is_draft = sigma >= 0 && sigma < T;

  // per-head scalars of record `lane`: log decay, and dt (Mamba-2) or beta (GDN)
  float pl[kHB], px[kHB];
  auto load_heads = [&](int batch) {
#pragma unroll
    for (int hb = 0; hb < kHB; ++hb) {
      const int e = batch * (kHB * kPrepWarps) + hb * kPrepWarps + warp;
      pl[hb] = 0.f;
      px[hb] = 0.f;
      if (e < hpg) {
        const int h = g * hpg + e;
        const size_t bh = static_cast<size_t>(b) * H + h;
        const size_t idx_d = is_draft ? (static_cast<size_t>(b) * T + sigma) * H + h : 0;
        if (KIND == 0) {
          if (lane < n) {
            pl[hb] = d.r_la[bh * Cp + slot_lane];
            px[hb] = bf(d.r_dt[bh * Cp + slot_lane]);
          } else if (is_draft) {
            const float dt = bf(in.dt[idx_d]);
            pl[hb] = dt * in.A[h];
            px[hb] = dt;
          }
        } else {
          if (lane < n) {
            pl[hb] = d.r_g[bh * Cp + slot_lane];
          } else if (is_draft) {
            pl[hb] = in.g[idx_d];
            px[hb] = in.beta[idx_d];
          }
        }
      }
    }
  };

  uint16_t* rk = (KIND == 0 ? d.r_B : d.r_k) + static_cast<size_t>(bg) * C * N;
  const uint16_t* kin = KIND == 0 ? in.Bm : in.k;
  const uint16_t* qin = KIND == 0 ? in.Cm : in.q;
  // 16-byte pieces: 16 per 128-channel bf16 row
  for (int e = t; e < nr * 16; e += kPrepThreads) {
    const int j = e >> 4, c = e & 15;
    const uint16_t* src = j < n ? rk + static_cast<size_t>(ring_slot(head, j, C)) * N
                                : kin + ((static_cast<size_t>(b) * T + (j - n)) * G + g) * N;
    const uint4 raw = reinterpret_cast<const uint4*>(src)[c];
    reinterpret_cast<uint4*>(&skey[j][0])[c] = raw;
    if constexpr (KIND == 1) {
      if (j >= n) {
        float4* dst = reinterpret_cast<float4*>(&scol[kT + j - n][8 * c]);
        dst[0] = bf4(make_uint2(raw.x, raw.y));
        dst[1] = bf4(make_uint2(raw.z, raw.w));
      }
    }
  }
  for (int e = t; e < kT * 16; e += kPrepThreads) {
    const int tau = e >> 4, c = e & 15;
    float4* dst = reinterpret_cast<float4*>(&scol[tau][8 * c]);
    if (tau < T) {
      const uint4 raw = reinterpret_cast<const uint4*>(qin + ((static_cast<size_t>(b) * T + tau) * G + g) * N)[c];
      dst[0] = bf4(make_uint2(raw.x, raw.y));
      dst[1] = bf4(make_uint2(raw.z, raw.w));
    } else {
      dst[0] = dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if constexpr (KIND == 1) {
        float4* dk4 = reinterpret_cast<float4*>(&scol[kT + tau][8 * c]);
        dk4[0] = dk4[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  load_heads(0);
  __syncthreads();
  // the drafts' keys into the ring, after the committed records
  for (int e = t; e < T * 16; e += kPrepThreads) {
    const int tau = e >> 4, c = e & 15;
    reinterpret_cast<uint4*>(rk + static_cast<size_t>(ring_slot(head, n + tau, C)) * N)[c] =
        reinterpret_cast<const uint4*>(&skey[n + tau][0])[c];
  }
  // key dot products.  A pass of one warp covers 4 * RPL records: lane 8 rq + cb
  // holds channels 4 (8 i + cb) .. + 3 (i < 4) of record jb + 4 r + rq (r < RPL)
  // and forms its partial dots with every column; the transpose-reduce over the
  // eight lanes of rq leaves value cb = r * kNCol + col in lane cb.
  {
    constexpr int RPL = 8 / kNCol;
    const int rq = lane >> 3, cb = lane & 7;
    const int npass = (nr + 4 * RPL - 1) / (4 * RPL);
    for (int p = warp; p < npass; p += kPrepWarps) {
      const int jb = p * 4 * RPL;
      int jr[RPL];
#pragma unroll
      for (int r = 0; r < RPL; ++r) jr[r] = min(jb + 4 * r + rq, nr - 1);
      float2 acc[RPL][kNCol];
#pragma unroll
      for (int r = 0; r < RPL; ++r)
#pragma unroll
        for (int col = 0; col < kNCol; ++col) acc[r][col] = make_float2(0.f, 0.f);
      // one 16-byte chunk of channels at a time (unrolled, the loop's column loads are
      // all hoisted and the registers spill)
#pragma unroll 1
      for (int i = 0; i < 4; ++i) {
        float4 kr[RPL];
#pragma unroll
        for (int r = 0; r < RPL; ++r) kr[r] = bf4(skey[jr[r]][8 * i + cb]);
#pragma unroll
        for (int col = 0; col < kNCol; ++col) {
          const float4 o = reinterpret_cast<const float4*>(scol[col])[8 * i + cb];
#pragma unroll
          for (int r = 0; r < RPL; ++r) {
            acc[r][col] = fma2(make_float2(kr[r].x, kr[r].y), make_float2(o.x, o.y), acc[r][col]);
            acc[r][col] = fma2(make_float2(kr[r].z, kr[r].w), make_float2(o.z, o.w), acc[r][col]);
          }
        }
      }
      float part[8];
#pragma unroll
      for (int r = 0; r < RPL; ++r)
#pragma unroll
        for (int col = 0; col < kNCol; ++col) part[r * kNCol + col] = acc[r][col].x + acc[r][col].y;
      const float tot = reduce8_lanes3(part, lane);
      const int j = jb + 4 * (cb / kNCol) + rq, col = cb % kNCol;
      if (j < nr) {
        if (col < kT) {
          if (col < T) sdq[j][col] = tot;
        } else if (col - kT < T) {
          sdk[j][col - kT] = tot;
        }
      }
    }
  }
  __syncthreads();
  float dq[kT], dk[kT];
#pragma unroll
  for (int tau = 0; tau < kT; ++tau) {
    dq[tau] = (lane < nr && tau < T) ? sdq[lane][tau] : 0.f;
    dk[tau] = (KIND == 1 && lane < nr && tau < T) ? sdk[lane][tau] : 0.f;
  }
  // per head: decay weights and the coefficient table (all draft positions in one
  // warp), the drafts' appends
  const int nbatch = (hpg + kHB * kPrepWarps - 1) / (kHB * kPrepWarps);
  for (int batch = 0; batch < nbatch; ++batch) {
    if (batch > 0) load_heads(batch);
#pragma unroll
    for (int hb = 0; hb < kHB; ++hb) {
      const int e = batch * (kHB * kPrepWarps) + hb * kPrepWarps + warp;
      if (e >= hpg) continue;
      const int h = g * hpg + e;
      const size_t bh = static_cast<size_t>(b) * H + h;
      float* co = d.vtab + bh * HS;
      const float lj = pl[hb];
      // log-decay sums along draft tau's path, built from terms of one sign so that
      // nothing cancels: the committed records by one suffix scan
      // (sc_j = sum_{i=j..n-1} l_i), the drafts by direct sums of at most four terms
      float sc = lane < n ? lj : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float w = __shfl_down_sync(0xffffffffu, sc, o);
        if (lane + o < 32) sc += w;
      }
      const float tot_c = __shfl_sync(0xffffffffu, sc, 0);          // every committed record
      const float sc_next = __shfl_down_sync(0xffffffffu, sc, 1);
      const float sc_after = lane < n ? sc_next : 0.f;  // records j+1..n-1
      float ld[kT];  // the drafts' log decays
#pragma unroll
      for (int s = 0; s < kT; ++s) ld[s] = __shfl_sync(0xffffffffu, lj, min(n + s, 31));
      // for draft tau: ex_q = sum over the path records after `lane` up to tau, ex_k
      // the same before tau, and a_q, a_k the path drafts' totals
      auto path_sums = [&](int tau, float& ex_q, float& ex_k, float& a_q, float& a_k) {
        float dq_ = 0.f, dk_ = 0.f, aq = 0.f, ak = 0.f;
#pragma unroll
        for (int s = 0; s < kT; ++s) {
          if (s < T && on_tree_path(d.tree_anc, tau, s)) {
            aq += ld[s];
            if (s != tau) ak += ld[s];
            if (s > sigma) {
              dq_ += ld[s];
              if (s != tau) dk_ += ld[s];
            }
          }
        }
        ex_q = sc_after + dq_;
        ex_k = sc_after + dk_;
        a_q = aq;
        a_k = ak;
      };
      if (KIND == 0) {
        const float dtj = px[hb];
        float c1[kT], Dv[kT];
#pragma unroll
        for (int tau = 0; tau < kT; ++tau) {
          // w_j = prod_{i=j+1..m} a_i, D = prod_{i<=m} a_i over draft tau's path
          const int m = n + tau;
          float ex, ex_k, aq, ak;  // ex_k and ak serve the GDN table only
          path_sums(tau, ex, ex_k, aq, ak);
          const bool onp = lane < n || on_tree_path(d.tree_anc, tau, sigma);  // record on draft tau's path
          const float W = onp ? __expf(lane < m ? ex : 0.f) : 0.f;
          c1[tau] = tau < T ? W * dq[tau] * dtj : 0.f;
          Dv[tau] = tau < T ? __expf(tot_c + aq) : 0.f;
        }
        if (lane < nr) reinterpret_cast<float4*>(co)[lane] = make_float4(c1[0], c1[1], c1[2], c1[3]);
        if (lane == 0) reinterpret_cast<float4*>(co)[C] = make_float4(Dv[0], Dv[1], Dv[2], Dv[3]);
        // the drafts into the ring: dt and log decay (the x rows are appended by
        // the main kernel, which stages them anyway)
        if (is_draft) {
          d.r_dt[bh * Cp + ring_slot(head, lane, C)] = static_cast<uint16_t>(__float_as_uint(dtj) >> 16);
          d.r_la[bh * Cp + ring_slot(head, lane, C)] = lj;
        }
      } else {
        const float g_d = is_draft ? lj : 0.f;
        const float beta_d = px[hb];
        float c1[kT], c2[kT], G1[kT], G2[kT], a_t[kT], b_t[kT], Mv[kT], Qv[kT];
#pragma unroll
        for (int tau = 0; tau < kT; ++tau) {
          const int m = n + tau;  // draft tau is record m
          float exq, exk, aq, ak;
          path_sums(tau, exq, exk, aq, ak);
          const float gm = __shfl_sync(0xffffffffu, g_d, min(m, 31));
          const float bm = __shfl_sync(0xffffffffu, beta_d, min(m, 31));
          // over draft tau's path: tW_j = prod_{i=j+1..m} a_i (j <= m),
          // tWk_j = prod_{i=j+1..m-1} a_i (j < m)
          const float tW = lane <= m ? __expf(lane < m ? exq : 0.f) : 0.f;
          const float tWk = lane < m ? __expf(lane + 1 < m ? exk : 0.f) : 0.f;
          const bool live = tau < T;
          G2[tau] = live ? __expf(tot_c + aq) : 0.f;
          G1[tau] = live ? (m > 0 ? __expf(tot_c + ak) : 1.f) : 0.f;
          a_t[tau] = live ? __expf(gm) : 0.f;
          b_t[tau] = live ? bm : 0.f;
          c1[tau] = (live && lane < n) ? tWk * dk[tau] : 0.f;  // coefficient of u_j[r] in S k_tau
          c2[tau] = (live && lane < n) ? tW * dq[tau] : 0.f;   // coefficient of u_j[r] in S q_tau
          // lane n + s: M[tau][s] (s < tau), Qd[tau][s] (s <= tau)
          const bool anc = is_draft && on_tree_path(d.tree_anc, tau, sigma);
          Mv[tau] = (live && anc && sigma != tau) ? b_t[tau] * a_t[tau] * tWk * dk[tau] : 0.f;
          Qv[tau] = (live && anc) ? tW * dq[tau] : 0.f;
        }
        if (lane < n) {
          reinterpret_cast<float4*>(co)[lane] = make_float4(c1[0], c1[1], c1[2], c1[3]);
          reinterpret_cast<float4*>(co)[C + lane] = make_float4(c2[0], c2[1], c2[2], c2[3]);
        }
        float* sc = co + 8 * C;
        if (lane == 0) {
          reinterpret_cast<float4*>(sc)[0] = make_float4(G2[0], G2[1], G2[2], G2[3]);
          reinterpret_cast<float4*>(sc)[1] = make_float4(G1[0], G1[1], G1[2], G1[3]);
          reinterpret_cast<float4*>(sc)[2] = make_float4(a_t[0], a_t[1], a_t[2], a_t[3]);
          reinterpret_cast<float4*>(sc)[3] = make_float4(b_t[0], b_t[1], b_t[2], b_t[3]);
        }
        if (is_draft) {
#pragma unroll
          for (int tau = 0; tau < kT; ++tau) {
            sc[16 + tau * 4 + sigma] = Mv[tau];
            sc[32 + tau * 4 + sigma] = Qv[tau];
          }
          d.r_g[bh * Cp + ring_slot(head, lane, C)] = g_d;
        }
      }
    }
  }
}

// ============================================================================
// main kernel
// ============================================================================
struct VL {
  int tile, rec, rec_size, rec_tab, rec_meta;
  int gb, gb_size;
  int g_key, g_q, g_B, g_dx;
  int bars, seq, misc;
  int total;
};

__host__ __device__ __forceinline__ VL vlayout(int kind, int C, int hpg, int P, int NR) {
  const int HPU = kRows / P;
  VL l;
  int o = 0;
  l.tile = o;     o += kNT * static_cast<int>(kTileBytes);
  l.rec = o;
  l.rec_tab = kind == 0 ? 256 * C : 512 * C;                 // records of the unit's 128 rows
  l.rec_meta = l.rec_tab + HPU * head_stride(kind, C) * 4;   // coefficient tables of its heads
  l.rec_size = al128(l.rec_meta + 32);                       // 32 bytes of descriptor
  o += NR * l.rec_size;
  int g = 0;
  l.g_B = g;      g += kNmma * N * 2;
  l.g_key = g;    g += kT * N * 2;  // draft keys
  l.g_q = g;      g += kT * N * 2;  // draft queries
  l.g_dx = g;     g += al16(kT * hpg * P * 2);
  l.gb_size = al128(g);
  l.gb = o;       o += 2 * l.gb_size;
  l.bars = o;     o += 32 * 8;
  l.seq = o;      o += 3 * kMaxSeqV * 4;
  l.misc = o;     o += 16;
  l.total = al128(o) + 1024;  // + slack to align the base to 1024 bytes
  return l;
}

// Barrier among the four epilogue warps (named barrier 2, 128 threads) that
// also returns whether `v` held in all of them.
__device__ __forceinline__ bool epi_sync_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

// Unit position (sequence, first head, group, head-in-group of the first head),
// advanced one unit at a time.
struct VWalk {
  int b, h0, g, hh0;
  __device__ __forceinline__ void start(int u0, int UPH, int HPU, int hpg) {
    b = u0 / UPH;
    h0 = (u0 - b * UPH) * HPU;
    g = h0 / hpg;
    hh0 = h0 - g * hpg;
  }
  __device__ __forceinline__ void next(int H, int HPU, int hpg) {
    h0 += HPU;
    hh0 += HPU;
    if (hh0 == hpg) {
      hh0 = 0;
      ++g;
    }
    if (h0 == H) {
      h0 = 0;
      g = 0;
      hh0 = 0;
      ++b;
    }
  }
};

template <int KIND, int P>
__global__ void __launch_bounds__(kThreadsV, 1)
    verify128_kernel(const __grid_constant__ CUtensorMap tmap, const LayerDev d, const TokenIn in, const int T,
                     float* __restrict__ y, const int units_per_cta, const int NR) {
  constexpr int HPU = kRows / P;  // heads per unit
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int H = d.H, G = d.G, C = d.C, L = d.L;
  const int hpg = H / G;
  const int UPH = H / HPU;
  const int HS = head_stride(KIND, C);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const VL LY = vlayout(KIND, C, hpg, P, NR);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY.bars);
  uint64_t* tile_full = bars;        // [2]
  uint64_t* tile_empty = bars + 2;   // [2]
  uint64_t* acc_full = bars + 4;     // [2]
  uint64_t* acc_empty = bars + 6;    // [2]
  uint64_t* drain = bars + 8;        // [1]
  uint64_t* chunk_full = bars + 10;  // [6]
  uint64_t* chunk_free = bars + 16;  // [6]
  uint64_t* rec_full = bars + 22;    // [NR]
  uint64_t* rec_empty = bars + 25;   // [NR]
  uint64_t* ready = bars + 28;       // [NR]
  int* sseq = reinterpret_cast<int*>(smem + LY.seq);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + LY.misc);
  volatile int* smisc = reinterpret_cast<volatile int*>(smem + LY.misc + 4);  // abort, tiles issued, records issued

  const int total_units = d.B * UPH;
  const int u0 = blockIdx.x * units_per_cta;
  const int u1 = min(u0 + units_per_cta, total_units);
  if (u0 >= u1) return;
  const int nunits = u1 - u0;
  const int b0 = u0 / UPH, b1 = (u1 - 1) / UPH;
  const int nseq = b1 - b0 + 1;

  if (t < nseq) {
    const int b = b0 + t;
    const int head = d.cursor[4 * b], cnt = d.cursor[4 * b + 1];
    const bool ok = static_cast<unsigned>(head) < static_cast<unsigned>(C) &&
                    static_cast<unsigned>(cnt) < static_cast<unsigned>(L) && cnt + T <= C;
    sseq[3 * t] = ok ? head : 0;
    sseq[3 * t + 1] = ok ? cnt : 0;
    sseq[3 * t + 2] = ok ? 1 : 0;
  }
  if (t == 0) {
    for (int s = 0; s < kNT; ++s) {
      mbar_init(tile_full + s, 1);
      mbar_init(tile_empty + s, kSplitWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(acc_full + s, 1);
      mbar_init(acc_empty + s, 4);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(chunk_full + s, 4);
      mbar_init(chunk_free + s, 1);
    }
    mbar_init(drain, 1);
    for (int s = 0; s < NR; ++s) {
      mbar_init(rec_full + s, 1);
      mbar_init(rec_empty + s, 4);
      mbar_init(ready + s, 1);
    }
    smisc[0] = 0;
    smisc[1] = 0;
    smisc[2] = 0;
  }
  if (warp == 0) tmem_alloc(tslot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  auto abort_with = [&](int b) {
    report_error(d.err, DEVERR_TIMEOUT, b);
    smisc[0] = 1;
  };
  auto tile_at = [&](int ts) { return smem + LY.tile + ts * kTileBytes; };
  auto rec_at = [&](int rs) { return smem + LY.rec + rs * LY.rec_size; };
  auto gb_at = [&](int gs) { return smem + LY.gb + gs * LY.gb_size; };

  if (warp == kWarpProd) {
    // ================================ producer ================================
    if (lane == 0) {
      VWalk w;
      w.start(u0, UPH, HPU, hpg);
      int gi = -1;
      for (int i = 0; i < nunits; ++i, w.next(H, HPU, hpg)) {
        const bool first = i == 0 || w.hh0 == 0;
        if (first) ++gi;
        const int ts = i % kNT, rs = i % NR;
        if (i >= kNT && !mbar_wait_bounded(tile_empty + ts, static_cast<uint32_t>(((i / kNT) - 1) & 1))) {
          abort_with(w.b);
          break;
        }
        if (smisc[0]) break;
        mbar_expect_tx(tile_full + ts, kTileBytes);
        const int row0 = (w.b * H + w.h0) * P;
        for (int kb = 0; kb < 4; ++kb)
          tma_load_2d(tile_at(ts) + kb * (kTileBytes / 4), &tmap, kb * 32, row0, tile_full + ts);
        smisc[1] = i + 1;
        if (i >= NR && !mbar_wait_bounded(rec_empty + rs, static_cast<uint32_t>(((i / NR) - 1) & 1))) {
          abort_with(w.b);
          break;
        }
        if (smisc[0]) break;
        const int k = w.b - b0;
        const int head = sseq[3 * k], n = sseq[3 * k + 1];
        const int seg1 = min(n, C - head), seg2 = n - seg1;
        unsigned char* rec = rec_at(rs);
        unsigned char* gb = gb_at(gi & 1);
        uint64_t* bar = rec_full + rs;
        const size_t bh0 = static_cast<size_t>(w.b) * H + w.h0;
        constexpr int esz = KIND == 0 ? 2 : 4;
        uint32_t bytes = static_cast<uint32_t>(HPU * n * P * esz + HPU * HS * 4);
        if (first) bytes += static_cast<uint32_t>(2 * T * N * 2 + T * hpg * P * 2);
        mbar_expect_tx(bar, bytes);
        // committed records of the unit's rows, the coefficient tables of its heads
        for (int hu = 0; hu < HPU; ++hu) {
          const size_t base = (bh0 + hu) * C;
          unsigned char* dst = rec + static_cast<size_t>(hu) * C * P * esz;
          const unsigned char* src = KIND == 0 ? reinterpret_cast<const unsigned char*>(d.r_x)
                                               : reinterpret_cast<const unsigned char*>(d.r_u);
          if (seg1) bulk_g2s(dst, src + (base + head) * P * esz, seg1 * P * esz, bar);
          if (seg2) bulk_g2s(dst + static_cast<size_t>(seg1) * P * esz, src + base * P * esz, seg2 * P * esz, bar);
        }
        // the tables come from the prep kernel, which may still be running
        if (i == 0) {
          asm volatile("griddepcontrol.wait;" ::: "memory");
          asm volatile("fence.proxy.async.global;" ::: "memory");  // then read by the bulk copies
        }
        bulk_g2s(rec + LY.rec_tab, d.vtab + bh0 * HS, HPU * HS * 4, bar);
        if (first) {
          for (int tau = 0; tau < T; ++tau) {
            const size_t bt = static_cast<size_t>(w.b) * T + tau;
            const size_t kq = (bt * G + w.g) * N;
            bulk_g2s(gb + LY.g_key + tau * N * 2, (KIND == 0 ? in.Bm : in.k) + kq, N * 2, bar);
            bulk_g2s(gb + LY.g_q + tau * N * 2, (KIND == 0 ? in.Cm : in.q) + kq, N * 2, bar);
            const size_t i0 = bt * H + static_cast<size_t>(w.g) * hpg;
            bulk_g2s(gb + LY.g_dx + tau * hpg * P * 2, (KIND == 0 ? in.x : in.v) + i0 * P, hpg * P * 2, bar);
          }
        }
        smisc[2] = i + 1;
      }
      // after an abort: the copies already issued land before the CTA frees its memory
      if (smisc[0]) {
        const int nt = smisc[1], nr = smisc[2];
        for (int j = max(0, nt - kNT); j < nt; ++j)
          mbar_wait_bounded(tile_full + j % kNT, static_cast<uint32_t>((j / kNT) & 1));
        for (int j = max(0, nr - NR); j < nr; ++j)
          mbar_wait_bounded(rec_full + j % NR, static_cast<uint32_t>((j / NR) & 1));
      }
    }
  } else if (warp == kWarpPro) {
    // ================================ prologue ================================
    VWalk w;
    w.start(u0, UPH, HPU, hpg);
    int gi = -1;
    for (int i = 0; i < nunits; ++i, w.next(H, HPU, hpg)) {
      if (smisc[0]) break;
      const int rs = i % NR;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(rec_full + rs, static_cast<uint32_t>((i / NR) & 1)))) {
        if (lane == 0) abort_with(w.b);
        break;
      }
      const bool first = i == 0 || w.hh0 == 0;
      if (first) ++gi;
      const int k = w.b - b0;
      const int head = sseq[3 * k], n = sseq[3 * k + 1];
      const bool ok = sseq[3 * k + 2] != 0;
      unsigned char* gb = gb_at(gi & 1);
      if (first && ok) {
        // the MMA B operand in bf16, canonical K-major: rows = [K_draft | Q] (GDN) or [Q]
        // (Mamba-2), zero-padded to kNmma rows; one 16-byte core-matrix row per store
        const uint16_t* kb = reinterpret_cast<const uint16_t*>(gb + LY.g_key);
        const uint16_t* qb = reinterpret_cast<const uint16_t*>(gb + LY.g_q);
        uint16_t* Bs = reinterpret_cast<uint16_t*>(gb + LY.g_B);
        for (int it = 0; it < kNmma * N / 8 / 32; ++it) {
          const int rho = 2 * it + (lane >> 4);  // B row
          const int c = lane & 15;               // 8-element block along K
          const uint16_t* src = nullptr;
          if (KIND == 0) {
            if (rho < T) src = qb + rho * N;
          } else {
            if (rho < T) src = kb + rho * N;
            else if (rho < 2 * T) src = qb + (rho - T) * N;
          }
          const uint4 v = src ? reinterpret_cast<const uint4*>(src)[c] : make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(Bs + canon_offset16(rho, 8 * c, N)) = v;
        }
      }
      if (lane == 0) {
        int* meta = reinterpret_cast<int*>(rec_at(rs) + LY.rec_meta);
        *reinterpret_cast<int4*>(meta) = make_int4(w.b, w.h0, n | (ok ? 0x100 : 0), w.hh0 | ((gi & 1) << 16));
        meta[4] = head;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // B operand -> tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(ready + rs);
    }
  } else if (warp == kWarpMma) {
    // ================================ MMA thread ================================
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kRows, kNmma);
      int issued = 0;
      for (int i = 0; i < nunits; ++i) {
        if (smisc[0]) break;
        const int rs = i % NR, ab = i & 1;
        bool okw = mbar_wait_bounded(ready + rs, static_cast<uint32_t>((i / NR) & 1));
        if (i >= 2) okw = okw && mbar_wait_bounded(acc_empty + ab, static_cast<uint32_t>(((i / 2) - 1) & 1));
        if (!okw) {
          abort_with((u0 + i) / UPH);
          break;
        }
        const int4 meta = *reinterpret_cast<const int4*>(rec_at(rs) + LY.rec_meta);
        const uint32_t bsm = smem_u32(gb_at(meta.w >> 16) + LY.g_B);
        const uint32_t dacc = tmem + kAccCol + ab * 32;
        bool okc = true;
        for (int kb = 0; kb < 4; ++kb) {
          const int q = 4 * i + kb, slot = q % kSlots;
          if (!mbar_wait_bounded(chunk_full + slot, static_cast<uint32_t>((q / kSlots) & 1))) {
            okc = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = tmem + slot * kSlotCols;
          // the three bf16 parts (hi, mid, lo) of the chunk's 32 K-columns, K = 16 per MMA
          for (int part = 0; part < 3; ++part)
            for (int kk = 0; kk < 2; ++kk)
              mma_bf16_ta(dacc, a0 + part * 16 + kk * 8, umma_desc(bsm + (2 * kb + kk) * 256, 128, (N / 8) * 128),
                          idesc, kb > 0 || part > 0 || kk > 0);
          mma_commit(chunk_free + slot);
          issued = i + 1;
        }
        if (!okc) {
          abort_with((u0 + i) / UPH);
          break;
        }
        mma_commit(acc_full + ab);
      }
      // every MMA issued has completed before tensor memory is freed
      mma_commit(drain);
      if (issued > 0 || smisc[0]) mbar_wait_bounded(drain, 0);
    }
  } else if (warp < kSplitWarps) {
    // ================================ split warps ================================
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;
    for (int i = 0; i < nunits; ++i) {
      if (smisc[0]) break;
      const int ts = i % kNT;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(tile_full + ts, static_cast<uint32_t>((i / kNT) & 1)))) {
        if (lane == 0) abort_with((u0 + i) / UPH);
        break;
      }
      const unsigned char* tl = tile_at(ts) + r * 128;
      bool okc = true;
#pragma unroll 1
      for (int kb = half; kb < 4; kb += 2) {
        const int q = 4 * i + kb, slot = q % kSlots;
        if (q >= kSlots &&
            !__all_sync(0xffffffffu, mbar_wait_bounded(chunk_free + slot, static_cast<uint32_t>(((q / kSlots) - 1) & 1)))) {
          okc = false;
          break;
        }
        // exact split x = hi + mid + lo into three bf16 (24 significand bits in three
        // round-to-nearest pieces of 8; both differences are exact), two K-columns a word
        uint32_t hm[32], lo[16];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const float4 x = *reinterpret_cast<const float4*>(tl + kb * (kTileBytes / 4) + ((cc ^ (r & 7)) << 4));
          const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const float a = xs[e], b = xs[e + 1];
            const uint32_t h = pack_bf16x2(a, b);
            const float ra = a - __uint_as_float(h << 16), rb = b - __uint_as_float(h & 0xFFFF0000u);
            const uint32_t m = pack_bf16x2(ra, rb);
            const float sa = ra - __uint_as_float(m << 16), sb = rb - __uint_as_float(m & 0xFFFF0000u);
            hm[2 * cc + e / 2] = h;
            hm[16 + 2 * cc + e / 2] = m;
            lo[2 * cc + e / 2] = pack_bf16x2(sa, sb);
          }
        }
        const uint32_t ta = tmem + slot * kSlotCols + (static_cast<uint32_t>(quarter * 32) << 16);
        tmem_st32(ta, hm);
        tmem_st16(ta + 32, lo);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(chunk_full + slot);
      }
      if (!okc) {
        if (lane == 0) abort_with((u0 + i) / UPH);
        break;
      }
      // the tile has been read: the producer may refill the stage
      if (lane == 0) mbar_arrive(tile_empty + ts);
    }
  } else {
    // ================================ epilogue warps ================================
    // The four warps decide together (named barrier 2) whether to go on, so
    // that none of them is left waiting at the barrier.
    const int ew = warp - kWarpEpi;  // also the tensor-memory lane quarter
    const int r = ew * 32 + lane;
    const int hu = r / P, p = r - hu * P;
    for (int i = 0; i < nunits; ++i) {
      const int rs = i % NR, ab = i & 1;
      bool got = mbar_wait_bounded(ready + rs, static_cast<uint32_t>((i / NR) & 1));
      got = got && mbar_wait_bounded(acc_full + ab, static_cast<uint32_t>((i / 2) & 1));
      if (!epi_sync_and(got)) {
        if (ew == 0 && lane == 0) abort_with((u0 + i) / UPH);
        break;
      }
      tc_fence_after();
      float acc[8];
      tmem_ld8(tmem + kAccCol + ab * 32 + (static_cast<uint32_t>(ew * 32) << 16), acc);
      const unsigned char* rec = rec_at(rs);
      const int* meta = reinterpret_cast<const int*>(rec + LY.rec_meta);
      const int b = meta[0], h0 = meta[1], n = meta[2] & 0xFF;
      const bool ok = (meta[2] & 0x100) != 0;
      const int hh = (meta[3] & 0xFFFF) + hu;
      const int head = meta[4];
      const unsigned char* gb = gb_at(meta[3] >> 16);
      const float* co = reinterpret_cast<const float*>(rec + LY.rec_tab) + hu * HS;
      const float4* co4 = reinterpret_cast<const float4*>(co);
      const int h = h0 + hu;
      if (ok) {
        if (KIND == 0) {
          const uint16_t* xr = reinterpret_cast<const uint16_t*>(rec) + hu * C * P + p;
          const uint16_t* xd = reinterpret_cast<const uint16_t*>(gb + LY.g_dx) + hh * P + p;
          float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 4
          for (int j = 0; j < n; ++j) {
            const float4 c = co4[j];
            const float xv = bf(xr[j * P]);
            a0 = fmaf(c.x, xv, a0);
            a1 = fmaf(c.y, xv, a1);
            a2 = fmaf(c.z, xv, a2);
            a3 = fmaf(c.w, xv, a3);
          }
          uint16_t* xring = d.r_x + (static_cast<size_t>(b) * H + h) * C * P + p;
          for (int s = 0; s < T; ++s) {
            const float4 c = co4[n + s];
            const uint16_t xbits = xd[s * hpg * P];
            xring[static_cast<size_t>(ring_slot(head, n + s, C)) * P] = xbits;  // the draft into the ring
            const float xv = bf(xbits);
            a0 = fmaf(c.x, xv, a0);
            a1 = fmaf(c.y, xv, a1);
            a2 = fmaf(c.z, xv, a2);
            a3 = fmaf(c.w, xv, a3);
          }
          const float4 Dv = co4[C];
          const float av[kT] = {a0, a1, a2, a3};
          const float dv[kT] = {Dv.x, Dv.y, Dv.z, Dv.w};
#pragma unroll
          for (int tau = 0; tau < kT; ++tau)
            if (tau < T) y[((static_cast<size_t>(b) * T + tau) * H + h) * P + p] = fmaf(dv[tau], acc[tau], av[tau]);
        } else {
          const float* ur = reinterpret_cast<const float*>(rec) + hu * C * P + p;
          float rk[kT] = {0.f, 0.f, 0.f, 0.f}, rq[kT] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
          for (int j = 0; j < n; ++j) {
            const float4 c1 = co4[j], c2 = co4[C + j];
            const float uj = ur[j * P];
            rk[0] = fmaf(c1.x, uj, rk[0]);
            rk[1] = fmaf(c1.y, uj, rk[1]);
            rk[2] = fmaf(c1.z, uj, rk[2]);
            rk[3] = fmaf(c1.w, uj, rk[3]);
            rq[0] = fmaf(c2.x, uj, rq[0]);
            rq[1] = fmaf(c2.y, uj, rq[1]);
            rq[2] = fmaf(c2.z, uj, rq[2]);
            rq[3] = fmaf(c2.w, uj, rq[3]);
          }
          const float* sc = co + 8 * C;
          const uint16_t* vd = reinterpret_cast<const uint16_t*>(gb + LY.g_dx) + hh * P + p;
          const size_t bh = static_cast<size_t>(b) * H + h;
          float uu[kT];
#pragma unroll
          for (int tau = 0; tau < kT; ++tau) {
            uu[tau] = 0.f;
            if (tau < T) {
              const float Sk = fmaf(sc[4 + tau], acc[tau], rk[tau]);  // G1 * (S_ckpt k) + buffered
              float rhs = sc[12 + tau] * (bf(vd[tau * hpg * P]) - sc[8 + tau] * Sk);
#pragma unroll
              for (int s = 0; s < kT; ++s)
                if (s < tau) rhs = fmaf(-sc[16 + tau * 4 + s], uu[s], rhs);
              uu[tau] = rhs;
            }
          }
#pragma unroll
          for (int tau = 0; tau < kT; ++tau) {
            if (tau < T) {
              float o = fmaf(sc[tau], acc[T + tau], rq[tau]);  // G2 * (S_ckpt q) + buffered
#pragma unroll
              for (int s = 0; s < kT; ++s)
                if (s <= tau) o = fmaf(sc[32 + tau * 4 + s], uu[s], o);
              y[((static_cast<size_t>(b) * T + tau) * H + h) * P + p] = o;
              d.r_u[(bh * C + ring_slot(head, n + tau, C)) * P + p] = uu[tau];
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(acc_empty + ab);
        mbar_arrive(rec_empty + rs);
      }
    }
  }

  // ---- teardown: all copies and MMAs have completed; free tensor memory ----
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int KIND, int P>
cudaError_t launch_v128(const LayerDev& d, const CUtensorMap& tmap, const TokenIn& in, int T, float* y,
                        cudaStream_t s) {
  constexpr int HPU = kRows / P;
  const int hpg = d.H / d.G;
  const int U = hpg / HPU;  // units per group
  const int NR = U + 1 < kMaxNR ? U + 1 : kMaxNR;
  const VL LY = vlayout(KIND, d.C, hpg, P, NR);
  if (LY.total > 227 * 1024) return cudaErrorInvalidConfiguration;
  verify_prep_kernel<KIND><<<d.B * d.G, kPrepThreads, 0, s>>>(d, in, T);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int UPH = d.H / HPU;
  const int total = d.B * UPH;
  int grid = d.num_sms > 0 ? d.num_sms : 1;
  if (grid > total) grid = total;
  int per = (total + grid - 1) / grid;
  while (per / UPH + 2 > kMaxSeqV) {
    grid *= 2;
    per = (total + grid - 1) / grid;
  }
  grid = (total + per - 1) / per;
  auto kernel = verify128_kernel<KIND, P>;
  e = set_smem_limit(reinterpret_cast<const void*>(kernel), LY.total);
  if (e != cudaSuccess) return e;
  // launched as a programmatic dependent of the prep kernel: its setup and first
  // tile loads overlap the prep kernel's last wave (see griddepcontrol.wait)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreadsV);
  cfg.dynamicSmemBytes = LY.total;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, tmap, d, in, T, y, per, NR);
}

}  // namespace

int verify_table_stride(int kind, int C) { return head_stride(kind, C); }

bool verify128_supports(const LayerDev& d) {
  if (d.N != N || (d.P != 64 && d.P != 128) || d.T_max > kT || d.C > kMaxRec || !d.vtab) return false;
  const int HPU = kRows / d.P, hpg = d.H / d.G;
  if (hpg % HPU != 0) return false;
  const int U = hpg / HPU;
  const int NR = U + 1 < kMaxNR ? U + 1 : kMaxNR;
  return vlayout(d.kind, d.C, hpg, d.P, NR).total <= 227 * 1024;
}

cudaError_t make_ckpt_tmap(const LayerDev& d, CUtensorMap* out) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult qr;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr);
    if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  // the checkpoint as a 2D tensor [B*H*P rows][d_state] of FP32; box 32 x 128, 128-byte swizzle
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(d.B) * d.H * d.P};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 4};
  const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(kRows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, d.ckpt, dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_verify128(const LayerDev& d, const CUtensorMap& tmap, const TokenIn& in, int T, float* y,
                             cudaStream_t s) {
  if (!verify128_supports(d) || T < 1 || T > kT) return cudaErrorInvalidValue;
  if (d.kind == 0)
    return d.P == 64 ? launch_v128<0, 64>(d, tmap, in, T, y, s) : launch_v128<0, 128>(d, tmap, in, T, y, s);
  return d.P == 64 ? launch_v128<1, 64>(d, tmap, in, T, y, s) : launch_v128<1, 128>(d, tmap, in, T, y, s);
}

}  // namespace rs
