// Speculative verification of T draft tokens per sequence, chunkwise form.
//
// With n committed records j = 0..n-1 buffered since the checkpoint and the
// T drafts appended as records n..n+T-1, the output of draft position tau is
//   O = S_ckpt Q D + V (W ⊙ (K^T Q))
// Q = [q_0..q_{T-1}], D = diag(prod_{i<=n+tau} a_i), K and V the keys and
// value vectors of the n+T records, W[j][tau] = prod_{i=j+1..n+tau} a_i for
// j <= n+tau and 0 above ("ReplaySSM caches SSM inputs instead of state"
// (richland.au), "What shipped", the paragraph on the second, subtler
// benefit).  K^T Q is formed once per group for the group's keys and draft
// queries.  For Gated DeltaNet the draft deltas u_tau solve the unit
// lower-triangular T x T system
//   u_tau + sum_{s<tau} M[tau][s] u_s = R_tau,
//   R_tau     = b_tau (v_tau - a_tau (S_{n+tau} k_tau over the committed records)),
//   M[tau][s] = b_tau a_tau prod_{n+s<i<n+tau} a_i (k_{n+s} . k_tau),
// by forward substitution per state row; V then holds the committed u_j and
// the draft u_tau.
//
// The dense part S_ckpt [rows][d_state] x [Q | K_draft] [d_state][<=16] runs on
// the tensor cores: tcgen05 kind::tf32 with the FP32 state split into a
// TF32-exact high part and the remainder (two MMA passes; the draft queries
// and keys are bf16, which TF32 holds exactly), FP32 accumulation in tensor
// memory.  M = 128 rows per MMA; a work unit is a 64-row chunk of one head's
// state and the other 64 rows of the MMA are ignored.
//
// Structure: persistent CTAs over (sequence, head, row chunk) units, one
// producer warp staging each unit with bulk copies (state rows, buffered
// records, drafts, the group's keys and queries when the group changes), eight
// computing warps that split the state into the canonical MMA layout, issue
// the MMAs, form decays and per-row buffered terms while the tensor cores
// run, then read the accumulator back and finish each row.  The drafts are
// appended to the ring after the committed records; the cursor does not move.
#include "common.cuh"
#include "readcopy.cuh"
#include "tcgen05.cuh"

namespace rs {
namespace {

constexpr int kTMax = 4;        // drafts per verify
constexpr int kNmma = 16;       // MMA N (columns: T queries, or T keys + T queries)
constexpr int kRowChunk = 64;   // state rows per work unit
constexpr int kMaxSeqV = 64;    // sequences one CTA may cover
constexpr int kVerifyThreads = kThreads + 32;

__host__ __device__ __forceinline__ int a16v(int x) { return (x + 15) & ~15; }
__host__ __device__ __forceinline__ int a128v(int x) { return (x + 127) & ~127; }

__device__ __forceinline__ int ring_slot(int head, int j, int C) {
  int s = head + j;
  return s >= C ? s - C : s;
}

struct VStage {
  int tile;   // f32 [RC][N] state rows
  int rec;    // Mamba-2: x bf16 [C][RC] (committed, then drafts); GDN: u f32 [C][RC] committed
  int vd;     // GDN: draft v bf16 [T][RC]
  int key;    // bf16 [C][N]: committed keys then draft keys (first unit of a group)
  int qry;    // bf16 [T][N] draft queries (first unit of a group)
  int la;     // f32 [Cp] log decays, slot order
  int dt;     // Mamba-2: dt bf16 [Cp], slot order
  int chunk;  // 16-byte chunks: Mamba-2 dt_tau (T), A; GDN g_tau (T), beta_tau (T)
  int size;
};

__host__ __device__ __forceinline__ VStage vstage_layout(int kind, int RC, int N, int C, int Cp) {
  VStage s;
  int o = 0;
  s.tile = o;  o += RC * N * 4;
  s.rec = o;   o += kind == 0 ? a16v(C * RC * 2) : C * RC * 4;
  s.vd = o;    o += kind == 0 ? 0 : kTMax * RC * 2;
  s.key = o;   o += C * N * 2;
  s.qry = o;   o += kTMax * N * 2;
  s.la = o;    o += Cp * 4;
  s.dt = o;    o += kind == 0 ? a16v(Cp * 2) : 0;
  s.chunk = o; o += (2 * kTMax + 1) * 16;
  s.size = a128v(o);
  return s;
}

// Shared memory outside the stages, bytes.  The operand buffers come first:
// MMA rows beyond the chunk read the memory that follows them.
struct VPersist {
  int ahi, alo, b, tab, bars, seq, slot, size;
};

__host__ __device__ __forceinline__ VPersist vpersist_layout(int RC, int N, int C) {
  VPersist p;
  int o = 0;
  p.ahi = o;  o += RC * N * 4;
  p.alo = o;  o += RC * N * 4;
  p.b = o;    o += kNmma * N * 4;
  p.tab = o;  o += (8 * C * kTMax + 4 * kTMax * kRowChunk + 8 * kTMax + 2 * kTMax * kTMax + 16) * 4;
  p.bars = a16v(o);  o = p.bars + 8 * 17;  // 8 full, 8 empty, 1 mma
  p.seq = o;  o += 3 * kMaxSeqV * 4;
  p.slot = o; o += 16;
  p.size = a128v(o);
  return p;
}

template <int KIND, int N>
__global__ void __launch_bounds__(kVerifyThreads, 1) verify_kernel(const LayerDev d, const TokenIn in, const int T,
                                                                   float* __restrict__ y, const int units_per_cta,
                                                                   const int stages) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int P = d.P, H = d.H, G = d.G, C = d.C, L = d.L, Cp = d.Cp;
  const int hpg = H / G;
  const int RC = P < kRowChunk ? P : kRowChunk;
  const int NCH = P / RC;  // row chunks per head
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const VPersist PL = vpersist_layout(RC, N, C);
  const VStage SL = vstage_layout(KIND, RC, N, C, Cp);
  float* sAhi = reinterpret_cast<float*>(smem + PL.ahi);
  float* sAlo = reinterpret_cast<float*>(smem + PL.alo);
  float* sB = reinterpret_cast<float*>(smem + PL.b);
  float* tab = reinterpret_cast<float*>(smem + PL.tab);
  // tables (floats)
  float* tD = tab;                        // [C][4]  k_j . q_tau            (GDN: k_j . q_tau)
  float* tDk = tD + C * kTMax;            // [C][4]  GDN k_j . k_tau
  float* tW = tDk + C * kTMax;            // [C][4]  prod_{i=j+1..n+tau} a_i
  float* tWk = tW + C * kTMax;            // [C][4]  GDN prod_{i=j+1..n+tau-1} a_i
  float* tC1 = tWk + C * kTMax;           // [C][4]  per-record coefficient (output / S k)
  float* tC2 = tC1 + C * kTMax;           // [C][4]  GDN per-record coefficient of S q
  float* tR1 = tab + 8 * C * kTMax;       // [4][RC] per-row buffered term (Mamba-2 y / GDN S k)
  float* tR2 = tR1 + kTMax * kRowChunk;   // [4][RC] GDN buffered term of S q
  float* tS = tR1 + 4 * kTMax * kRowChunk;  // [8][4] per-draft scalars: D|G2, G1, a, beta, ...
  float* tM = tS + 8 * kTMax;             // [4][4] GDN solve coefficients
  float* tQd = tM + kTMax * kTMax;        // [4][4] GDN draft-draft output coefficients
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + PL.bars);
  uint64_t* empty = full + 8;
  uint64_t* mma_bar = full + 16;
  int* sseq = reinterpret_cast<int*>(smem + PL.seq);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + PL.slot);
  volatile int* smisc = reinterpret_cast<volatile int*>(smem + PL.slot + 4);  // abort, issued, done
  unsigned char* stage0 = smem + PL.size;

  const int total_units = d.B * H * NCH;
  const int u0 = blockIdx.x * units_per_cta;
  const int u1 = min(u0 + units_per_cta, total_units);
  if (u0 >= u1) return;
  const int nunits = u1 - u0;
  const int b0 = u0 / (H * NCH), b1 = (u1 - 1) / (H * NCH);
  const int nseq = b1 - b0 + 1;

  if (t < nseq) {
    const int b = b0 + t;
    const int head = d.cursor[4 * b], cnt = d.cursor[4 * b + 1];
    const bool ok = static_cast<unsigned>(head) < static_cast<unsigned>(C) &&
                    static_cast<unsigned>(cnt) < static_cast<unsigned>(L) && cnt + T <= C;
    sseq[3 * t] = head;
    sseq[3 * t + 1] = cnt;
    sseq[3 * t + 2] = ok ? 1 : 0;
  }
  if (t == kThreads) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    mbar_init(mma_bar, 1);
    smisc[0] = 0;
    smisc[1] = 0;
    smisc[2] = 0;
  }
  if (warp == 0) tmem_alloc(tslot, 32);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  struct VUnit {
    int u, b, h, g, rc, head, n;
    size_t bh;
    bool ok, first_of_group;
  };
  auto unit_of = [&](int i) {
    VUnit v;
    v.u = u0 + i;
    v.rc = v.u % NCH;
    const int bhh = v.u / NCH;
    v.b = bhh / H;
    v.h = bhh - v.b * H;
    v.g = v.h / hpg;
    v.bh = static_cast<size_t>(bhh);
    const int k = v.b - b0;
    v.head = sseq[3 * k];
    v.ok = sseq[3 * k + 2] != 0;
    v.n = v.ok ? sseq[3 * k + 1] : 0;
    v.first_of_group = (i == 0) || (v.h % hpg == 0 && v.rc == 0);
    return v;
  };

  // ============================ producer warp ==============================
  if (warp == kThreads / 32) {
    if (lane != 0) return;
    for (int i = 0; i < nunits; ++i) {
      const int s = i % stages;
      if (i >= stages && !mbar_wait_bounded(empty + s, static_cast<uint32_t>(((i / stages) - 1) & 1))) break;
      if (smisc[0]) break;
      const VUnit v = unit_of(i);
      unsigned char* st = stage0 + static_cast<size_t>(SL.size) * s;
      uint64_t* bar = full + s;
      const int n = v.n;
      const size_t bg = static_cast<size_t>(v.b) * G + v.g;
      const int esz = KIND == 0 ? 2 : 4;
      uint32_t bytes = RC * N * 4 + static_cast<uint32_t>(n) * RC * esz + Cp * 4 + (KIND == 0 ? a16v(Cp * 2) : 0);
      bytes += KIND == 0 ? static_cast<uint32_t>(T) * RC * 2 : static_cast<uint32_t>(T) * RC * 2;
      bytes += KIND == 0 ? (T + 1) * 16 : 2 * T * 16;
      if (v.first_of_group) bytes += static_cast<uint32_t>(n + T) * N * 2 + static_cast<uint32_t>(T) * N * 2;
      mbar_expect_tx(bar, bytes);
      // state rows of this chunk
      bulk_g2s(st + SL.tile, d.ckpt + (v.bh * P + static_cast<size_t>(v.rc) * RC) * N, RC * N * 4, bar);
      // committed records (rows of this chunk): one or two contiguous runs of
      // slots when the chunk is the whole head row, else one copy per record
      if (RC == P) {
        const int seg1 = min(n, C - v.head), seg2 = n - seg1;
        const size_t base = v.bh * C * P;
        if (KIND == 0) {
          if (seg1) bulk_g2s(st + SL.rec, d.r_x + base + static_cast<size_t>(v.head) * P, seg1 * P * 2, bar);
          if (seg2) bulk_g2s(st + SL.rec + seg1 * P * 2, d.r_x + base, seg2 * P * 2, bar);
        } else {
          if (seg1) bulk_g2s(st + SL.rec, d.r_u + base + static_cast<size_t>(v.head) * P, seg1 * P * 4, bar);
          if (seg2) bulk_g2s(st + SL.rec + seg1 * P * 4, d.r_u + base, seg2 * P * 4, bar);
        }
      } else {
        for (int j = 0; j < n; ++j) {
          const size_t row = (v.bh * C + ring_slot(v.head, j, C)) * P + static_cast<size_t>(v.rc) * RC;
          if (KIND == 0)
            bulk_g2s(st + SL.rec + j * RC * 2, d.r_x + row, RC * 2, bar);
          else
            bulk_g2s(st + SL.rec + j * RC * 4, d.r_u + row, RC * 4, bar);
        }
      }
      // draft values, per-head scalars
      for (int tau = 0; tau < T; ++tau) {
        const size_t bt = static_cast<size_t>(v.b) * T + tau;
        const size_t src = (bt * H + v.h) * P + static_cast<size_t>(v.rc) * RC;
        if (KIND == 0) {
          bulk_g2s(st + SL.rec + (n + tau) * RC * 2, in.x + src, RC * 2, bar);
          bulk_g2s(st + SL.chunk + tau * 16, in.dt + ((bt * H + v.h) & ~static_cast<size_t>(7)), 16, bar);
        } else {
          bulk_g2s(st + SL.vd + tau * RC * 2, in.v + src, RC * 2, bar);
          bulk_g2s(st + SL.chunk + tau * 16, in.g + ((bt * H + v.h) & ~static_cast<size_t>(3)), 16, bar);
          bulk_g2s(st + SL.chunk + (kTMax + tau) * 16, in.beta + ((bt * H + v.h) & ~static_cast<size_t>(3)), 16,
                   bar);
        }
      }
      if (KIND == 0) {
        bulk_g2s(st + SL.chunk + 2 * kTMax * 16, in.A + (v.h & ~3), 16, bar);
        bulk_g2s(st + SL.la, d.r_la + v.bh * Cp, Cp * 4, bar);
        bulk_g2s(st + SL.dt, d.r_dt + v.bh * Cp, a16v(Cp * 2), bar);
      } else {
        bulk_g2s(st + SL.la, d.r_g + v.bh * Cp, Cp * 4, bar);
      }
      if (v.first_of_group) {
        const uint16_t* rk = (KIND == 0 ? d.r_B : d.r_k) + bg * C * N;
        const int seg1 = min(n, C - v.head), seg2 = n - seg1;
        if (seg1) bulk_g2s(st + SL.key, rk + static_cast<size_t>(v.head) * N, seg1 * N * 2, bar);
        if (seg2) bulk_g2s(st + SL.key + seg1 * N * 2, rk, seg2 * N * 2, bar);
        for (int tau = 0; tau < T; ++tau) {
          const size_t src = ((static_cast<size_t>(v.b) * T + tau) * G + v.g) * N;
          bulk_g2s(st + SL.key + (n + tau) * N * 2, (KIND == 0 ? in.Bm : in.k) + src, N * 2, bar);
          bulk_g2s(st + SL.qry + tau * N * 2, (KIND == 0 ? in.Cm : in.q) + src, N * 2, bar);
        }
      }
      smisc[1] = i + 1;
    }
    smisc[2] = 1;
    return;
  }

  // ============================ computing warps ============================
  const uint32_t idesc = idesc_tf32(128, kNmma);
  const uint32_t sbo = static_cast<uint32_t>(N / 4) * 128u;
  int consumed = 0;
  bool mma_pending = false;
  for (int i = 0; i < nunits; ++i) {
    const int s = i % stages;
    if (!compute_sync_and(mbar_wait_bounded(full + s, static_cast<uint32_t>((i / stages) & 1)))) {
      if (t == 0) {
        report_error(d.err, DEVERR_TIMEOUT, (u0 + i) / (H * NCH));
        smisc[0] = 1;
      }
      break;
    }
    consumed = i + 1;
    const VUnit v = unit_of(i);
    const unsigned char* st = stage0 + static_cast<size_t>(SL.size) * s;
    const int n = v.n, nr = n + T;

    // ---- per group: the MMA B operand and the key dot products ----
    if (v.first_of_group) {
      const uint16_t* kb = reinterpret_cast<const uint16_t*>(st + SL.key);
      const uint16_t* qb = reinterpret_cast<const uint16_t*>(st + SL.qry);
      const int ncols = KIND == 0 ? T : 2 * T;
      for (int e = t; e < kNmma * N; e += kThreads) {
        const int row = e / N, k = e - row * N;
        float val = 0.f;
        if (row < ncols) {
          if (KIND == 0) val = bf(qb[row * N + k]);
          else val = row < T ? bf(kb[(n + row) * N + k]) : bf(qb[(row - T) * N + k]);
        }
        sB[canon_offset(row, k, N)] = val;
      }
      // K^T Q (and GDN K^T K_draft): one warp per record
      for (int j = warp; j < nr; j += kThreads / 32) {
        float aq[kTMax], ak[kTMax];
#pragma unroll
        for (int tau = 0; tau < kTMax; ++tau) aq[tau] = ak[tau] = 0.f;
        for (int e = lane; e < N; e += 32) {
          const float kv = bf(kb[j * N + e]);
#pragma unroll
          for (int tau = 0; tau < kTMax; ++tau) {
            if (tau < T) {
              aq[tau] = fmaf(kv, bf(qb[tau * N + e]), aq[tau]);
              if (KIND == 1) ak[tau] = fmaf(kv, bf(kb[(n + tau) * N + e]), ak[tau]);
            }
          }
        }
#pragma unroll
        for (int tau = 0; tau < kTMax; ++tau) {
          if (tau < T) {
            aq[tau] = seg_sum<32>(aq[tau]);
            if (KIND == 1) ak[tau] = seg_sum<32>(ak[tau]);
            if (lane == 0) {
              tD[j * kTMax + tau] = aq[tau];
              if (KIND == 1) tDk[j * kTMax + tau] = ak[tau];
            }
          }
        }
      }
    }

    // ---- split the state rows into the canonical TF32 operand (hi + lo) ----
    {
      const float4* src = reinterpret_cast<const float4*>(st + SL.tile);
      const int total4 = RC * N / 4;
      for (int e = t; e < total4; e += kThreads) {
        int r, c;
        if (N >= 32) {  // diagonal order: conflict-free row-major reads and core-matrix writes
          constexpr int CB = N >= 32 ? N / 32 : 1;  // 8-chunk column blocks per row
          const int blk = e >> 6, w = e & 63, q = w & 7, dd = w >> 3;
          const int rb = blk / CB, cb = blk - rb * CB;
          r = 8 * rb + q;
          c = 8 * cb + ((q + dd) & 7);
        } else {
          r = e / (N / 4);
          c = e - r * (N / 4);
        }
        const float4 val = src[r * (N / 4) + c];
        float4 hi, lo;
        hi.x = __uint_as_float(__float_as_uint(val.x) & 0xFFFFE000u);
        hi.y = __uint_as_float(__float_as_uint(val.y) & 0xFFFFE000u);
        hi.z = __uint_as_float(__float_as_uint(val.z) & 0xFFFFE000u);
        hi.w = __uint_as_float(__float_as_uint(val.w) & 0xFFFFE000u);
        lo = make_float4(val.x - hi.x, val.y - hi.y, val.z - hi.z, val.w - hi.w);
        const int off = canon_offset(r, 4 * c, N);
        *reinterpret_cast<float4*>(sAhi + off) = hi;
        *reinterpret_cast<float4*>(sAlo + off) = lo;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    compute_sync();

    // ---- tensor cores: S_chunk x [Q | K_draft], two passes (hi, lo) ----
    if (t == 0) {
      tc_fence_after();
      const uint32_t ah = smem_u32(sAhi), al = smem_u32(sAlo), bb = smem_u32(sB);
      bool acc = false;
      for (int pass = 0; pass < 2; ++pass) {
        const uint32_t a = pass == 0 ? ah : al;
        for (int k = 0; k < N / 8; ++k) {
          mma_tf32(tmem, umma_desc(a + k * 256, 128, sbo), umma_desc(bb + k * 256, 128, sbo), idesc, acc);
          acc = true;
        }
      }
      mma_commit(mma_bar);
    }
    mma_pending = true;

    // ---- decay weights per draft position (warp tau), while the MMAs run ----
    const float* la_slot = reinterpret_cast<const float*>(st + SL.la);
    const float* chunk = reinterpret_cast<const float*>(st + SL.chunk);
    if (warp < T) {
      const int tau = warp, last = n + tau;  // records 0..n+tau
      const size_t idx = (static_cast<size_t>(v.b) * T + tau) * H + v.h;
      float la_d;  // log decay of draft record n + tau', read by lane n + tau'
      const int dl = lane - n;
      if (KIND == 0) {
        const uint16_t* dtc = reinterpret_cast<const uint16_t*>(st + SL.chunk);
        const float A = chunk[2 * kTMax * 4 + (v.h & 3)];
        const size_t idx_l = (static_cast<size_t>(v.b) * T + (dl >= 0 && dl < T ? dl : 0)) * H + v.h;
        la_d = bf(dtc[(dl >= 0 && dl < T ? dl : 0) * 8 + (idx_l & 7)]) * A;
      } else {
        const size_t idx_l = (static_cast<size_t>(v.b) * T + (dl >= 0 && dl < T ? dl : 0)) * H + v.h;
        la_d = chunk[(dl >= 0 && dl < T ? dl : 0) * 4 + (idx_l & 3)];
      }
      // records on draft tau's path: the committed ones, then tau's ancestors and tau
      const bool onp = lane < n || on_tree_path(d.tree_anc, tau, dl);
      const float lj = lane < n ? la_slot[lane < n ? ring_slot(v.head, lane, C) : 0] : (onp ? la_d : 0.f);
      const float vq = suffix_sum(lj, lane, last);
      const float exq = __shfl_down_sync(0xffffffffu, vq, 1);
      if (lane <= last) tW[lane * kTMax + tau] = expf(lane < last ? exq : 0.f);
      if (lane == 0) tS[tau] = expf(vq);  // D (Mamba-2) / G2 (GDN)
      if (KIND == 1) {
        const float vk = suffix_sum((onp && dl != tau) ? lj : 0.f, lane, last - 1);
        const float exk = __shfl_down_sync(0xffffffffu, vk, 1);
        if (lane < last) tWk[lane * kTMax + tau] = expf(lane + 1 < last ? exk : 0.f);
        if (lane == 0) {
          tS[kTMax + tau] = last > 0 ? expf(vk) : 1.f;                    // G1
          tS[2 * kTMax + tau] = expf(chunk[tau * 4 + (idx & 3)]);         // a_tau
          tS[3 * kTMax + tau] = chunk[(kTMax + tau) * 4 + (idx & 3)];     // beta_tau
        }
      }
    }
    compute_sync();
    // per-record coefficients
    for (int e = t; e < nr * kTMax; e += kThreads) {
      const int j = e / kTMax, tau = e - j * kTMax;
      if (tau >= T) continue;
      if (KIND == 0) {
        float dtj;
        if (j < n) {
          dtj = bf(reinterpret_cast<const uint16_t*>(st + SL.dt)[ring_slot(v.head, j, C)]);
        } else {
          const size_t idx = (static_cast<size_t>(v.b) * T + (j - n)) * H + v.h;
          dtj = bf(reinterpret_cast<const uint16_t*>(st + SL.chunk)[(j - n) * 8 + (idx & 7)]);
        }
        tC1[e] = (j < n || on_tree_path(d.tree_anc, tau, j - n)) ? tW[e] * tD[e] * dtj : 0.f;
      } else if (j < n) {
        tC1[e] = tWk[e] * tDk[e];  // coefficient of u_j[r] in S k_tau
        tC2[e] = tW[e] * tD[e];    // coefficient of u_j[r] in S q_tau
      }
    }
    if (KIND == 1 && t < kTMax * kTMax) {
      const int tau = t / kTMax, sg = t - tau * kTMax;
      const int j = n + sg;
      tM[t] = (tau < T && sg != tau && on_tree_path(d.tree_anc, tau, sg)) ? tS[3 * kTMax + tau] * tS[2 * kTMax + tau] * tWk[j * kTMax + tau] *
                                          tDk[j * kTMax + tau]
                                    : 0.f;
      tQd[t] = (tau < T && on_tree_path(d.tree_anc, tau, sg)) ? tW[j * kTMax + tau] * tD[j * kTMax + tau] : 0.f;
    }
    compute_sync();
    // per-row buffered terms
    for (int e = t; e < T * RC; e += kThreads) {
      const int tau = e / RC, r = e - tau * RC;
      float a1 = 0.f, a2 = 0.f;
      if (KIND == 0) {
        const uint16_t* xb = reinterpret_cast<const uint16_t*>(st + SL.rec);
        for (int j = 0; j <= n + tau; ++j) a1 = fmaf(tC1[j * kTMax + tau], bf(xb[j * RC + r]), a1);
      } else {
        const float* ub = reinterpret_cast<const float*>(st + SL.rec);
        for (int j = 0; j < n; ++j) {
          const float uj = ub[j * RC + r];
          a1 = fmaf(tC1[j * kTMax + tau], uj, a1);
          a2 = fmaf(tC2[j * kTMax + tau], uj, a2);
        }
      }
      tR1[tau * kRowChunk + r] = a1;
      tR2[tau * kRowChunk + r] = a2;
    }

    // ---- accumulator back, finish each row ----
    const bool mma_ok = compute_sync_and(mbar_wait_bounded(mma_bar, static_cast<uint32_t>(i & 1)));
    mma_pending = false;
    if (!mma_ok) {
      if (t == 0) {
        report_error(d.err, DEVERR_TIMEOUT, v.b);
        smisc[0] = 1;
      }
      mbar_wait_bounded(mma_bar, static_cast<uint32_t>(i & 1));
      break;
    }
    tc_fence_after();
    if (warp * 32 < RC) {
      float acc[16];
      tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16), acc);
      const int r = warp * 32 + lane;
      if (r < RC && v.ok) {
        const int prow = v.rc * RC + r;
        if (KIND == 0) {
          for (int tau = 0; tau < T; ++tau)
            y[((static_cast<size_t>(v.b) * T + tau) * H + v.h) * P + prow] =
                fmaf(tS[tau], acc[tau], tR1[tau * kRowChunk + r]);
        } else {
          const uint16_t* vdb = reinterpret_cast<const uint16_t*>(st + SL.vd);
          float uu[kTMax];
#pragma unroll
          for (int tau = 0; tau < kTMax; ++tau) {
            if (tau < T) {
              const float Sk = fmaf(tS[kTMax + tau], acc[tau], tR1[tau * kRowChunk + r]);
              float rhs = tS[3 * kTMax + tau] * (bf(vdb[tau * RC + r]) - tS[2 * kTMax + tau] * Sk);
#pragma unroll
              for (int sg = 0; sg < kTMax; ++sg)
                if (sg < tau) rhs = fmaf(-tM[tau * kTMax + sg], uu[sg], rhs);
              uu[tau] = rhs;
            }
          }
#pragma unroll
          for (int tau = 0; tau < kTMax; ++tau) {
            if (tau < T) {
              float o = fmaf(tS[tau], acc[T + tau], tR2[tau * kRowChunk + r]);
#pragma unroll
              for (int sg = 0; sg < kTMax; ++sg)
                if (sg <= tau) o = fmaf(tQd[tau * kTMax + sg], uu[sg], o);
              y[((static_cast<size_t>(v.b) * T + tau) * H + v.h) * P + prow] = o;
              d.r_u[(v.bh * C + ring_slot(v.head, n + tau, C)) * P + prow] = uu[tau];
            }
          }
        }
      }
    }
    tc_fence_before();

    // ---- append the drafts after the committed records ----
    if (v.ok) {
      if (KIND == 0) {
        const uint16_t* xb = reinterpret_cast<const uint16_t*>(st + SL.rec);
        for (int e = t; e < T * RC; e += kThreads) {
          const int tau = e / RC, r = e - tau * RC;
          d.r_x[(v.bh * C + ring_slot(v.head, n + tau, C)) * P + v.rc * RC + r] = xb[(n + tau) * RC + r];
        }
      }
      if (v.rc == 0 && t < T) {
        const int tau = t;
        const size_t idx = (static_cast<size_t>(v.b) * T + tau) * H + v.h;
        const int sl = ring_slot(v.head, n + tau, C);
        if (KIND == 0) {
          const uint16_t dtb = reinterpret_cast<const uint16_t*>(st + SL.chunk)[tau * 8 + (idx & 7)];
          d.r_dt[v.bh * Cp + sl] = dtb;
          d.r_la[v.bh * Cp + sl] = bf(dtb) * chunk[2 * kTMax * 4 + (v.h & 3)];
        } else {
          d.r_g[v.bh * Cp + sl] = chunk[tau * 4 + (idx & 3)];
        }
      }
      if (v.h % hpg == 0 && v.rc == 0) {
        const uint16_t* kb = reinterpret_cast<const uint16_t*>(st + SL.key);
        const size_t bg = static_cast<size_t>(v.b) * G + v.g;
        uint16_t* rk = KIND == 0 ? d.r_B : d.r_k;
        for (int e = t; e < T * N; e += kThreads) {
          const int tau = e / N, k = e - tau * N;
          rk[(bg * C + ring_slot(v.head, n + tau, C)) * N + k] = kb[(n + tau) * N + k];
        }
      }
      if (v.h == 0 && v.rc == 0 && t == 0) d.cursor[4 * v.b + 2] = 0;  // verify folds nothing
    } else if (v.h == 0 && v.rc == 0 && t == 0) {
      report_error(d.err, DEVERR_CURSOR, v.b);
    }
    compute_sync();
    if (t == 0) mbar_arrive(empty + s);
  }
  // ---- teardown: no tensor-core work or copy may be in flight when the CTA exits ----
  if (smisc[0]) {
    if (t == 0) {
      if (mma_pending) mbar_wait_bounded(mma_bar, static_cast<uint32_t>((consumed - 1) & 1));
      const uint64_t t0 = global_ns();
      while (!smisc[2] && global_ns() - t0 < 2000000000ull) {
      }
      const int issued = smisc[1];
      for (int j = consumed; j < issued; ++j)
        mbar_wait_bounded(full + (j % stages), static_cast<uint32_t>((j / stages) & 1));
    }
  }
  compute_sync();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
}

template <int KIND, int N>
cudaError_t launch_kn(const LayerDev& d, const TokenIn& in, int T, float* y, cudaStream_t s) {
  const int RC = d.P < kRowChunk ? d.P : kRowChunk;
  const VPersist PL = vpersist_layout(RC, d.N, d.C);
  const VStage SL = vstage_layout(d.kind, RC, d.N, d.C, d.Cp);
  long budget = 227L * 1024 - PL.size;
  int stages = static_cast<int>(budget / SL.size);
  if (stages > 4) stages = 4;
  if (stages < 1) return cudaErrorInvalidConfiguration;
  size_t smem = static_cast<size_t>(PL.size) + static_cast<size_t>(SL.size) * stages;
  // MMA rows past the chunk read the 128-row span after each operand buffer
  const size_t need = static_cast<size_t>(PL.alo) + 128u * static_cast<size_t>(d.N) * 4u;
  if (smem < need) smem = need;
  if (smem > 227u * 1024u) return cudaErrorInvalidConfiguration;
  const int total = d.B * d.H * (d.P / RC);
  int grid = d.num_sms > 0 ? d.num_sms : 1;
  if (grid > total) grid = total;
  int per = (total + grid - 1) / grid;
  while (per / (d.H * (d.P / RC)) + 2 > kMaxSeqV) {
    grid *= 2;
    per = (total + grid - 1) / grid;
  }
  grid = (total + per - 1) / per;
  auto kernel = verify_kernel<KIND, N>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kVerifyThreads, smem, s>>>(d, in, T, y, per, stages);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify(const LayerDev& d, const TokenIn& in, int T, float* y, cudaStream_t s) {
  if (T < 1 || T > kTMax) return cudaErrorInvalidValue;
  if (d.kind == 0) {
    switch (d.N) {
      case 16: return launch_kn<0, 16>(d, in, T, y, s);
      case 32: return launch_kn<0, 32>(d, in, T, y, s);
      case 64: return launch_kn<0, 64>(d, in, T, y, s);
      case 128: return launch_kn<0, 128>(d, in, T, y, s);
    }
  } else {
    switch (d.N) {
      case 16: return launch_kn<1, 16>(d, in, T, y, s);
      case 32: return launch_kn<1, 32>(d, in, T, y, s);
      case 64: return launch_kn<1, 64>(d, in, T, y, s);
      case 128: return launch_kn<1, 128>(d, in, T, y, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace rs
