// Speculative verification of T <= 4 draft tokens for d_state = 128 and
// d_head 64 or 128 (the layer shapes the workloads use), chunkwise form
//   O = S_ckpt Q D + V (W ⊙ (K^T Q))
// ("ReplaySSM caches SSM inputs instead of state" (richland.au), "What
// shipped", the paragraph on the second benefit), with the Gated DeltaNet
// drafts obtained by forward substitution of the unit lower-triangular T x T
// system (same arithmetic and notation as verify.cu, which serves the other
// shapes).
//
// A work unit is 128 consecutive state rows of one group: two heads of d_head
// 64, or one head of d_head 128, so one tcgen05 MMA with M = 128 covers it.
// The dense part S_ckpt [128][128] x [K_draft | Q] [128][16] runs on the
// tensor cores in kind::tf32 with FP32 accumulation in tensor memory.  The FP32
// state is split exactly: kind::tf32 reads an FP32 operand with its low 13
// mantissa bits ignored, so the first pass takes the raw state as loaded by
// TMA (128-byte swizzle, the layout the MMA reads directly), and the second
// pass takes lo = S - trunc(S), computed in registers and stored to tensor
// memory, as its A operand.  The drafts' queries and keys are bf16, which TF32
// holds exactly.
//
// Roles (11 warps, one persistent CTA per SM):
//  * producer (1 thread): per unit, the state tile by four 2D TMA loads into
//    one of two tile stages, and the unit's committed records by bulk copies
//    into one of up to three record stages; once per group, the group's keys,
//    draft queries, draft values, per-head scalars and ring decay rows into
//    one of two group buffers;
//  * prologue warp: once per group, the MMA B operand and the drafts' ring
//    appends; per unit a descriptor;
//  * four split warps: lo = S - trunc(S), row r to tensor-memory lane r;
//  * MMA thread: the two passes into one of two accumulators;
//  * four epilogue warps: once per group the key dot products K^T Q (and
//    K^T K_draft); per unit the decay weights and coefficient tables of its
//    heads (one suffix scan per head and draft position, spread over the
//    warps), then the accumulator rows back from
//    tensor memory, the buffered-record terms, the triangular solve (Gated
//    DeltaNet), outputs and the drafts' u records.
// Every wait is bounded; on a timeout the CTA records an error and drains its
// copies and MMAs before it frees tensor memory and exits.
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
constexpr int kWarpPro = 8, kWarpProd = 9, kWarpMma = 10;
constexpr int kThreadsV = 11 * 32;
// tensor memory: two lo operands (128 columns each), then two accumulators
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kLoCol = 0, kAccCol = 256;

__host__ __device__ __forceinline__ int al16(int x) { return (x + 15) & ~15; }
__host__ __device__ __forceinline__ int al128(int x) { return (x + 127) & ~127; }

// floats per head in a coefficient table
//   Mamba-2: C1[C][4], then D[4]
//   GDN:     C1[C][4], C2[C][4], then G2[4] G1[4] a[4] beta[4] M[4][4] Qd[4][4]
__host__ __device__ __forceinline__ int head_stride(int kind, int C) { return kind == 0 ? 4 * C + 4 : 8 * C + 48; }

struct VL {
  int tile, rec, rec_size, rec_meta;
  int gb, gb_size;
  int g_key, g_q, g_B, g_dx, g_s1, g_s2, g_la, g_dt, g_dq, g_dk, g_coef;
  int span;  // bytes of one per-draft scalar span
  int bars, seq, A, misc;
  int total;
};

__host__ __device__ __forceinline__ VL vlayout(int kind, int C, int Cp, int H, int hpg, int P, int NR) {
  VL l;
  int o = 0;
  l.tile = o;     o += kNT * static_cast<int>(kTileBytes);
  l.rec = o;
  l.rec_meta = kind == 0 ? 256 * C : 512 * C;  // records of the unit's 128 rows, then 32 bytes of descriptor
  l.rec_size = al128(l.rec_meta + 32);
  o += NR * l.rec_size;
  l.span = al16(hpg * 4) + 16;
  int g = 0;
  l.g_B = g;      g += kNmma * N * 4;
  l.g_key = g;    g += C * N * 2;
  l.g_q = g;      g += kT * N * 2;
  l.g_dx = g;     g += al16(kT * hpg * P * 2);
  l.g_s1 = g;     g += kT * l.span;
  l.g_s2 = g;     g += kind == 0 ? 0 : kT * l.span;
  l.g_la = g;     g += hpg * Cp * 4;
  l.g_dt = g;     g += kind == 0 ? al16(hpg * Cp * 2) : 0;
  l.g_dq = g;     g += C * 16;
  l.g_dk = g;     g += kind == 0 ? 0 : C * 16;
  l.g_coef = g;   g += hpg * head_stride(kind, C) * 4;
  l.gb_size = al128(g);
  l.gb = o;       o += 2 * l.gb_size;
  l.bars = o;     o += 32 * 8;
  l.seq = o;      o += 3 * kMaxSeqV * 4;
  l.A = o;        o += al16(H * 4);
  l.misc = o;     o += 16;
  l.total = al128(o) + 1024;  // + slack to align the base to 1024 bytes
  return l;
}

// Barrier among the four epilogue warps (named barrier 2, 128 threads); the
// _and form also returns whether `v` held in all of them.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
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

__device__ __forceinline__ int ring_slot(int head, int j, int C) {
  int s = head + j;
  return s >= C ? s - C : s;
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
  const int H = d.H, G = d.G, C = d.C, L = d.L, Cp = d.Cp;
  const int hpg = H / G;
  const int UPH = H / HPU;
  const int HS = head_stride(KIND, C);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const VL LY = vlayout(KIND, C, Cp, H, hpg, P, NR);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY.bars);
  uint64_t* tile_full = bars;        // [2]
  uint64_t* tile_empty = bars + 2;   // [2]
  uint64_t* lo_ready = bars + 4;     // [2]
  uint64_t* lo_free = bars + 6;      // [2]
  uint64_t* acc_full = bars + 8;     // [2]
  uint64_t* acc_empty = bars + 10;   // [2]
  uint64_t* drain = bars + 12;       // [1]
  uint64_t* rec_full = bars + 16;    // [NR]
  uint64_t* rec_empty = bars + 20;   // [NR]
  uint64_t* ready = bars + 24;       // [NR]
  int* sseq = reinterpret_cast<int*>(smem + LY.seq);
  const float* sA = reinterpret_cast<const float*>(smem + LY.A);
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
      mbar_init(tile_empty + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(lo_ready + s, 4);
      mbar_init(lo_free + s, 1);
      mbar_init(acc_full + s, 1);
      mbar_init(acc_empty + s, 4);
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
  // first element of the 16-byte block holding element e, for 2-byte / 4-byte arrays
  auto blk2 = [](size_t e) { return e & ~static_cast<size_t>(7); };
  auto blk4 = [](size_t e) { return e & ~static_cast<size_t>(3); };

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
        for (int kb = 0; kb < 4; ++kb) tma_load_2d(tile_at(ts) + kb * (kTileBytes / 4), &tmap, kb * 32, row0, tile_full + ts);
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
        const size_t ug = static_cast<size_t>(w.b) * H + static_cast<size_t>(w.g) * hpg;  // first head of the group
        const size_t bg = static_cast<size_t>(w.b) * G + w.g;
        constexpr int esz = KIND == 0 ? 2 : 4;
        uint32_t bytes = static_cast<uint32_t>(HPU * n * P * esz);
        if (first) {
          bytes += static_cast<uint32_t>((n + T) * N * 2 + T * N * 2 + T * hpg * P * 2 + hpg * Cp * 4);
          for (int tau = 0; tau < T; ++tau) {
            const size_t i0 = (static_cast<size_t>(w.b) * T + tau) * H + static_cast<size_t>(w.g) * hpg;
            if (KIND == 0) {
              bytes += static_cast<uint32_t>((blk2(i0 + hpg + 7) - blk2(i0)) * 2);
            } else {
              bytes += 2u * static_cast<uint32_t>((blk4(i0 + hpg + 3) - blk4(i0)) * 4);
            }
          }
          if (KIND == 0) bytes += static_cast<uint32_t>(hpg * Cp * 2);
        }
        if (KIND == 0 && i == 0) bytes += al16(H * 4);
        mbar_expect_tx(bar, bytes);
        // committed records of the unit's rows
        for (int hu = 0; hu < HPU; ++hu) {
          const size_t base = (bh0 + hu) * C;
          unsigned char* dst = rec + static_cast<size_t>(hu) * C * P * esz;
          const unsigned char* src = KIND == 0 ? reinterpret_cast<const unsigned char*>(d.r_x)
                                               : reinterpret_cast<const unsigned char*>(d.r_u);
          if (seg1) bulk_g2s(dst, src + (base + head) * P * esz, seg1 * P * esz, bar);
          if (seg2) bulk_g2s(dst + static_cast<size_t>(seg1) * P * esz, src + base * P * esz, seg2 * P * esz, bar);
        }
        if (first) {
          const uint16_t* rk = (KIND == 0 ? d.r_B : d.r_k) + bg * C * N;
          if (seg1) bulk_g2s(gb + LY.g_key, rk + static_cast<size_t>(head) * N, seg1 * N * 2, bar);
          if (seg2) bulk_g2s(gb + LY.g_key + seg1 * N * 2, rk, seg2 * N * 2, bar);
          for (int tau = 0; tau < T; ++tau) {
            const size_t bt = static_cast<size_t>(w.b) * T + tau;
            const size_t kq = (bt * G + w.g) * N;
            bulk_g2s(gb + LY.g_key + (n + tau) * N * 2, (KIND == 0 ? in.Bm : in.k) + kq, N * 2, bar);
            bulk_g2s(gb + LY.g_q + tau * N * 2, (KIND == 0 ? in.Cm : in.q) + kq, N * 2, bar);
            const size_t i0 = bt * H + static_cast<size_t>(w.g) * hpg;
            bulk_g2s(gb + LY.g_dx + tau * hpg * P * 2, (KIND == 0 ? in.x : in.v) + i0 * P, hpg * P * 2, bar);
            if (KIND == 0) {
              bulk_g2s(gb + LY.g_s1 + tau * LY.span, in.dt + blk2(i0),
                       static_cast<uint32_t>((blk2(i0 + hpg + 7) - blk2(i0)) * 2), bar);
            } else {
              const uint32_t sb = static_cast<uint32_t>((blk4(i0 + hpg + 3) - blk4(i0)) * 4);
              bulk_g2s(gb + LY.g_s1 + tau * LY.span, in.g + blk4(i0), sb, bar);
              bulk_g2s(gb + LY.g_s2 + tau * LY.span, in.beta + blk4(i0), sb, bar);
            }
          }
          if (KIND == 0) {
            bulk_g2s(gb + LY.g_la, d.r_la + ug * Cp, hpg * Cp * 4, bar);
            bulk_g2s(gb + LY.g_dt, d.r_dt + ug * Cp, hpg * Cp * 2, bar);
          } else {
            bulk_g2s(gb + LY.g_la, d.r_g + ug * Cp, hpg * Cp * 4, bar);
          }
        }
        if (KIND == 0 && i == 0) bulk_g2s(smem + LY.A, in.A, al16(H * 4), bar);
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
        const uint16_t* kb = reinterpret_cast<const uint16_t*>(gb + LY.g_key);
        const uint16_t* qb = reinterpret_cast<const uint16_t*>(gb + LY.g_q);
        // ---- the MMA B operand, canonical K-major: rows = [K_draft | Q] (GDN) or [Q] (Mamba-2) ----
        float* Bs = reinterpret_cast<float*>(gb + LY.g_B);
        for (int it = 0; it < kNmma * N / 4 / 32; ++it) {
          const int rho = (it >> 3) * 8 + (lane & 7);
          const int c = (it & 7) * 4 + (lane >> 3);
          const uint16_t* src = nullptr;
          if (KIND == 0) {
            if (rho < T) src = qb + rho * N;
          } else {
            if (rho < T) src = kb + (n + rho) * N;
            else if (rho < 2 * T) src = qb + (rho - T) * N;
          }
          const float4 v = src ? bf4(reinterpret_cast<const uint2*>(src)[c]) : make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(Bs + canon_offset(rho, 4 * c, N)) = v;
        }
        // ---- the drafts into the ring after the committed records ----
        const int sigma = lane - n;  // draft index of record `lane`
        const bool is_draft = sigma >= 0 && sigma < T;
        const size_t i0s = is_draft ? (static_cast<size_t>(w.b) * T + sigma) * H + static_cast<size_t>(w.g) * hpg : 0;
        const int hh_hi = min(hpg, w.hh0 + (nunits - i) * HPU);  // heads of this group in this CTA
        for (int e = w.hh0; e < hh_hi; ++e) {
          const int h = w.g * hpg + e;
          const size_t bhe = static_cast<size_t>(w.b) * H + h;
          if (KIND == 0) {
            for (int tau = 0; tau < T; ++tau) {
              const uint16_t* xs = reinterpret_cast<const uint16_t*>(gb + LY.g_dx) + (tau * hpg + e) * P;
              uint16_t* xd = d.r_x + (bhe * C + ring_slot(head, n + tau, C)) * P;
              if (P == 64)
                reinterpret_cast<uint32_t*>(xd)[lane] = reinterpret_cast<const uint32_t*>(xs)[lane];
              else
                reinterpret_cast<uint2*>(xd)[lane] = reinterpret_cast<const uint2*>(xs)[lane];
            }
            if (is_draft) {
              const uint16_t dt_bits = reinterpret_cast<const uint16_t*>(gb + LY.g_s1 + sigma * LY.span)[(i0s & 7) + e];
              const int sl = ring_slot(head, lane, C);
              d.r_dt[bhe * Cp + sl] = dt_bits;
              d.r_la[bhe * Cp + sl] = bf(dt_bits) * sA[h];
            }
          } else if (is_draft) {
            d.r_g[bhe * Cp + ring_slot(head, lane, C)] =
                reinterpret_cast<const float*>(gb + LY.g_s1 + sigma * LY.span)[(i0s & 3) + e];
          }
        }
        if (w.hh0 == 0) {
          // the drafts' key rows: appended by the CTA that holds the group's first head
          const size_t bg = static_cast<size_t>(w.b) * G + w.g;
          uint16_t* rk = KIND == 0 ? d.r_B : d.r_k;
          for (int tau = 0; tau < T; ++tau)
            reinterpret_cast<uint2*>(rk + (bg * C + ring_slot(head, n + tau, C)) * N)[lane] =
                reinterpret_cast<const uint2*>(kb + (n + tau) * N)[lane];
        }
      }
      if (lane == 0) {
        if (w.h0 == 0) {
          if (ok) d.cursor[4 * w.b + 2] = 0;  // verify folds nothing
          else report_error(d.err, DEVERR_CURSOR, w.b);
        }
        int* meta = reinterpret_cast<int*>(rec_at(rs) + LY.rec_meta);
        *reinterpret_cast<int4*>(meta) =
            make_int4(w.b, w.h0, n | (ok ? 0x100 : 0) | (first ? 0x200 : 0), w.hh0 | ((gi & 1) << 16));
        meta[4] = head;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // B operand -> tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(ready + rs);
    }
  } else if (warp == kWarpMma) {
    // ================================ MMA thread ================================
    if (lane == 0) {
      const uint32_t idesc = idesc_tf32(kRows, kNmma);
      int issued = 0;
      for (int i = 0; i < nunits; ++i) {
        if (smisc[0]) break;
        const int ts = i % kNT, rs = i % NR, ab = i & 1, lb = i & 1;
        bool okw = mbar_wait_bounded(tile_full + ts, static_cast<uint32_t>((i / kNT) & 1));
        okw = okw && mbar_wait_bounded(ready + rs, static_cast<uint32_t>((i / NR) & 1));
        if (i >= 2) okw = okw && mbar_wait_bounded(acc_empty + ab, static_cast<uint32_t>(((i / 2) - 1) & 1));
        if (!okw) {
          abort_with((u0 + i) / UPH);
          break;
        }
        const int4 meta = *reinterpret_cast<const int4*>(rec_at(rs) + LY.rec_meta);
        const uint32_t bsm = smem_u32(gb_at(meta.w >> 16) + LY.g_B);
        const uint32_t asm_ = smem_u32(tile_at(ts));
        const uint32_t dacc = tmem + kAccCol + ab * 32;
        tc_fence_after();
        for (int ks = 0; ks < N / 8; ++ks)
          mma_tf32(dacc, umma_desc_sw128(asm_ + (ks >> 2) * (kTileBytes / 4) + (ks & 3) * 32, 1024),
                   umma_desc(bsm + ks * 256, 128, (N / 4) * 128), idesc, ks > 0);
        issued = i + 1;
        if (!mbar_wait_bounded(lo_ready + lb, static_cast<uint32_t>((i / 2) & 1))) {
          abort_with((u0 + i) / UPH);
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < N / 8; ++ks)
          mma_tf32_ta(dacc, tmem + kLoCol + lb * 128 + ks * 8, umma_desc(bsm + ks * 256, 128, (N / 4) * 128), idesc,
                      true);
        mma_commit(acc_full + ab);
        mma_commit(tile_empty + ts);
        mma_commit(lo_free + lb);
      }
      // every MMA issued has completed before tensor memory is freed
      mma_commit(drain);
      if (issued > 0 || smisc[0]) mbar_wait_bounded(drain, 0);
    }
  } else if (warp < 4) {
    // ================================ split warps ================================
    const int r = warp * 32 + lane;
    for (int i = 0; i < nunits; ++i) {
      if (smisc[0]) break;
      const int ts = i % kNT, lb = i & 1;
      bool okw = mbar_wait_bounded(tile_full + ts, static_cast<uint32_t>((i / kNT) & 1));
      if (i >= 2) okw = okw && mbar_wait_bounded(lo_free + lb, static_cast<uint32_t>(((i / 2) - 1) & 1));
      if (!__all_sync(0xffffffffu, okw)) {
        if (lane == 0) abort_with((u0 + i) / UPH);
        break;
      }
      const unsigned char* tl = tile_at(ts) + r * 128;
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) {
        uint32_t v[32];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const float4 x = *reinterpret_cast<const float4*>(tl + kb * (kTileBytes / 4) + ((cc ^ (r & 7)) << 4));
          v[4 * cc + 0] = __float_as_uint(x.x - __uint_as_float(__float_as_uint(x.x) & 0xFFFFE000u));
          v[4 * cc + 1] = __float_as_uint(x.y - __uint_as_float(__float_as_uint(x.y) & 0xFFFFE000u));
          v[4 * cc + 2] = __float_as_uint(x.z - __uint_as_float(__float_as_uint(x.z) & 0xFFFFE000u));
          v[4 * cc + 3] = __float_as_uint(x.w - __uint_as_float(__float_as_uint(x.w) & 0xFFFFE000u));
        }
        tmem_st32(tmem + kLoCol + lb * 128 + (static_cast<uint32_t>(warp * 32) << 16) + kb * 32, v);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(lo_ready + lb);
    }
  } else {
    // ================================ epilogue warps ================================
    // The four warps decide together (named barrier 2) whether to go on, so
    // that none of them is left waiting at the barrier.
    const int ew = warp - 4;  // also the tensor-memory lane quarter
    const int r = ew * 32 + lane;
    const int hu = r / P, p = r - hu * P;
    for (int i = 0; i < nunits; ++i) {
      const int rs = i % NR, ab = i & 1;
      const bool got = mbar_wait_bounded(ready + rs, static_cast<uint32_t>((i / NR) & 1));
      if (!epi_sync_and(got)) {
        if (ew == 0 && lane == 0) abort_with((u0 + i) / UPH);
        break;
      }
      const unsigned char* rec = rec_at(rs);
      const int* meta = reinterpret_cast<const int*>(rec + LY.rec_meta);
      const int b = meta[0], h0 = meta[1], n = meta[2] & 0xFF;
      const bool ok = (meta[2] & 0x100) != 0, first = (meta[2] & 0x200) != 0;
      const int hh0 = meta[3] & 0xFFFF;
      const int head = meta[4];
      unsigned char* gb = gb_at(meta[3] >> 16);
      const int nr = n + T;
      float* dqt = reinterpret_cast<float*>(gb + LY.g_dq);  // [C][4]: k_j . q_tau
      float* dkt = reinterpret_cast<float*>(gb + LY.g_dk);  // [C][4]: k_j . k_{n+tau} (GDN)
      const uint16_t* kb = reinterpret_cast<const uint16_t*>(gb + LY.g_key);
      if (ok && first) {
        // key dot products of the group, shared by its heads; item = (8 records, one column)
        const uint16_t* qb = reinterpret_cast<const uint16_t*>(gb + LY.g_q);
        const int ncol = KIND == 0 ? T : 2 * T;
        const int nblk = (nr + 7) >> 3;
        for (int it = ew; it < nblk * ncol; it += 4) {
          const int jb = it / ncol, c = it - jb * ncol;
          const uint16_t* other = c < T ? qb + c * N : kb + (n + c - T) * N;
          const float4 o4 = bf4(reinterpret_cast<const uint2*>(other)[lane]);
          float part[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = 8 * jb + e;
            part[e] = j < nr ? dot4(bf4(reinterpret_cast<const uint2*>(kb + j * N)[lane]), o4) : 0.f;
          }
          const float tot = reduce8(part, lane);
          const int j = 8 * jb + (lane >> 2);
          if ((lane & 3) == 0 && j < nr) {
            if (c < T) dqt[j * 4 + c] = tot;
            else dkt[j * 4 + c - T] = tot;
          }
        }
      }
      epi_sync();
      if (ok) {
        // decay weights and coefficient tables, one (head, draft position) item per warp
        // at a time; each item is a suffix scan over the records 0..n+tau (FP32, as in
        // the decode kernels), lane j holding record j
        const int slot_lane = lane < n ? ring_slot(head, lane, C) : 0;
        const int sigma = lane - n;
        const bool is_draft = sigma >= 0 && sigma < T;
        for (int it = ew; it < HPU * T; it += 4) {
          const int hu_t = it / T, tau = it - hu_t * T;
          const int hh = hh0 + hu_t, h = h0 + hu_t;
          float* co = reinterpret_cast<float*>(gb + LY.g_coef) + hh * HS;
          const float* la_row = reinterpret_cast<const float*>(gb + LY.g_la) + hh * Cp;
          const size_t i0s = is_draft ? (static_cast<size_t>(b) * T + sigma) * H + static_cast<size_t>(h - hh) : 0;
          const int m = n + tau;  // draft tau is record m
          const float dqj = lane < nr ? dqt[lane * 4 + tau] : 0.f;
          if (KIND == 0) {
            const uint16_t dt_bits =
                is_draft ? reinterpret_cast<const uint16_t*>(gb + LY.g_s1 + sigma * LY.span)[(i0s & 7) + hh] : 0;
            const uint16_t* dtr = reinterpret_cast<const uint16_t*>(gb + LY.g_dt) + hh * Cp;
            const float lj = lane < n ? la_row[slot_lane] : (is_draft ? bf(dt_bits) * sA[h] : 0.f);
            const float dtj = lane < n ? bf(dtr[slot_lane]) : (is_draft ? bf(dt_bits) : 0.f);
            // w_j = prod_{i=j+1..m} a_i, D = prod_{i<=m} a_i
            const float v = suffix_sum(lane <= m ? lj : 0.f, lane, m);
            const float ex = __shfl_down_sync(0xffffffffu, v, 1);
            const float W = lane <= m ? expf(lane < m ? ex : 0.f) : 0.f;
            if (lane < nr) co[lane * 4 + tau] = W * dqj * dtj;
            if (lane == 0) co[4 * C + tau] = expf(v);
          } else {
            float g_d = 0.f, beta_d = 0.f;
            if (is_draft) {
              g_d = reinterpret_cast<const float*>(gb + LY.g_s1 + sigma * LY.span)[(i0s & 3) + hh];
              beta_d = reinterpret_cast<const float*>(gb + LY.g_s2 + sigma * LY.span)[(i0s & 3) + hh];
            }
            const float lj = lane < n ? la_row[slot_lane] : g_d;
            const float dkj = lane < nr ? dkt[lane * 4 + tau] : 0.f;
            // tW_j = prod_{i=j+1..m} a_i (j <= m), tWk_j = prod_{i=j+1..m-1} a_i (j < m)
            const float vq = suffix_sum(lane <= m ? lj : 0.f, lane, m);
            const float exq = __shfl_down_sync(0xffffffffu, vq, 1);
            const float tW = lane <= m ? expf(lane < m ? exq : 0.f) : 0.f;
            const float vk = suffix_sum(lane < m ? lj : 0.f, lane, m - 1);
            const float exk = __shfl_down_sync(0xffffffffu, vk, 1);
            const float tWk = lane < m ? expf(lane + 1 < m ? exk : 0.f) : 0.f;
            const float a_t = expf(__shfl_sync(0xffffffffu, g_d, m));
            const float b_t = __shfl_sync(0xffffffffu, beta_d, m);
            if (lane < n) {
              co[lane * 4 + tau] = tWk * dkj;        // coefficient of u_j[r] in S k_tau
              co[(C + lane) * 4 + tau] = tW * dqj;   // coefficient of u_j[r] in S q_tau
            }
            float* sc = co + 8 * C;
            if (lane == 0) {
              sc[tau] = expf(vq);                   // G2
              sc[4 + tau] = m > 0 ? expf(vk) : 1.f;  // G1
              sc[8 + tau] = a_t;
              sc[12 + tau] = b_t;
            }
            if (is_draft) {  // lane n + s: M[tau][s] (s < tau), Qd[tau][s] (s <= tau)
              sc[16 + tau * 4 + sigma] = sigma < tau ? b_t * a_t * tWk * dkj : 0.f;
              sc[32 + tau * 4 + sigma] = sigma <= tau ? tW * dqj : 0.f;
            }
            if (lane >= T && lane < kT) {  // unused draft slots of the T x T tables
              sc[16 + tau * 4 + lane] = 0.f;
              sc[32 + tau * 4 + lane] = 0.f;
            }
          }
        }
      }
      // the tables are complete; the accumulator of this unit is needed next
      const bool acc_ok = mbar_wait_bounded(acc_full + ab, static_cast<uint32_t>((i / 2) & 1));
      if (!epi_sync_and(acc_ok)) {
        if (ew == 0 && lane == 0) abort_with(b);
        break;
      }
      tc_fence_after();
      float acc[8];
      tmem_ld8(tmem + kAccCol + ab * 32 + (static_cast<uint32_t>(ew * 32) << 16), acc);
      const int hh = hh0 + hu;
      const float* co = reinterpret_cast<const float*>(gb + LY.g_coef) + hh * HS;
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
          for (int s = 0; s < T; ++s) {
            const float4 c = co4[n + s];
            const float xv = bf(xd[s * hpg * P]);
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
  const VL LY = vlayout(KIND, d.C, d.Cp, d.H, hpg, P, NR);
  if (LY.total > 227 * 1024) return cudaErrorInvalidConfiguration;
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
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kernel), LY.total);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreadsV, LY.total, s>>>(tmap, d, in, T, y, per, NR);
  return cudaGetLastError();
}

}  // namespace

bool verify128_supports(const LayerDev& d) {
  if (d.N != N || (d.P != 64 && d.P != 128) || d.T_max > kT || d.C > kMaxRec) return false;
  const int HPU = kRows / d.P, hpg = d.H / d.G;
  if (hpg % HPU != 0) return false;
  const int U = hpg / HPU;
  const int NR = U + 1 < kMaxNR ? U + 1 : kMaxNR;
  return vlayout(d.kind, d.C, d.Cp, d.H, hpg, d.P, NR).total <= 227 * 1024;
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
  if (d.kind == 0) return d.P == 64 ? launch_v128<0, 64>(d, tmap, in, T, y, s) : launch_v128<0, 128>(d, tmap, in, T, y, s);
  return d.P == 64 ? launch_v128<1, 64>(d, tmap, in, T, y, s) : launch_v128<1, 128>(d, tmap, in, T, y, s);
}

}  // namespace rs
