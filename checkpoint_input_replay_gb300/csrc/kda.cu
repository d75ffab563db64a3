// Decode step and fold for the delta rule with a per-key-channel gate (the gate
// form of Kimi Delta Attention), to which the checkpoint-plus-buffer method
// generalises ("ReplaySSM caches SSM inputs instead of state" (richland.au),
// "Why it matters"):
//   S_t = S_{t-1} Diag(a_t) (I - b_t k_t k_t^T) + b_t v_t k_t^T,  o_t = S_t q_t,
// with a_t = exp(g_t) a vector over the key channels.  Written as
//   S_t = S_{t-1} Diag(a_t) + u_t k_t^T,  u_t = b_t (v_t - S_{t-1} (a_t * k_t)),
// the state n records after the checkpoint unrolls to
//   S_n = S_ckpt Diag(G_n) + sum_j u_j (k_j * W_j(n))^T,
// G_n the channel-wise product of all n decays and W_j(n) that of the decays
// after record j.  A record is (g_j over the key channels, u_j, k_j).  Unlike
// the scalar gate, the decayed keys k_j * W_j differ per value head, so the
// record dot products are formed per head, not per key group.
//
// One CTA of 256 threads per (sequence, head, block of up to 64 rows).  The
// block's checkpoint rows (contiguous) are requested first, by one bulk copy
// into shared memory, so that they are in flight while the CTA stages the
// buffered records (log decays, keys, its rows' deltas), forms the decayed keys
// by a channel-wise suffix scan and the record dot products; then it finishes
// its rows:
//   S k' = S_ckpt (G' * k) + sum_j u_j (k_j * W'_j . k),   S q' likewise,
// with G', W' including this token's decay; u = b (v - S k'), o = S q' + u (k . q).
// A non-flush step appends (g, u, k) to the ring and stores no state; the flush
// step (the L-th record) writes S_ckpt Diag(G') + sum_j u_j (k_j * W'_j)^T + u k^T
// once.  The fold without a token (rs_flush) writes S_ckpt Diag(G_n) +
// sum_j u_j (k_j * W_j(n))^T.  The last CTA of a sequence to read its cursor
// advances it.
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace rs {
namespace {

constexpr int kKdaThreads = 256;
constexpr int kWarps = kKdaThreads / 32;
constexpr int kPass = 8;  // row passes per warp: one 16-byte load each in flight per thread

__device__ __forceinline__ int kslot(int head, int j, int C) {
  const int s = head + j;
  return s >= C ? s - C : s;
}

// rows of one CTA: every warp takes kPass passes of 32 / (N/4) rows
__host__ __device__ __forceinline__ int kda_rows(int N, int P) {
  const int rows = kWarps * kPass * (32 / (N / 4));
  return P < rows ? P : rows;
}

struct KdaSmem {
  int tile, bar, kt, u, kb, k, q, G, gq, gk, ck, cq, misc, size;  // float offsets
  int ustride;                                                     // floats per row of the deltas
};

__host__ __device__ __forceinline__ KdaSmem kda_smem(int R, int N, int C) {
  KdaSmem m;
  int o = 0;
  m.ustride = C | 1;        // odd: the lanes of a row read consecutive records without bank conflicts
  m.tile = o; o += R * N;   // the CTA's checkpoint rows, by one bulk copy
  m.bar = o;  o += 4;       // its mbarrier
  m.kt = o;   o += C * N;   // decayed keys k_j * W'_j [records][N] (the log decays first, in place)
  m.u = o;    o += (R * m.ustride + 3) & ~3;  // this CTA's rows' deltas [rows][records]
  m.kb = o;   o += C * N / 2;  // the records' keys, bf16 [records][N]
  m.k = o;    o += N;       // this token's key
  m.q = o;    o += N;       // this token's query
  m.G = o;    o += N;       // G' (fold: G_n), the checkpoint's channel decay
  m.gk = o;   o += N;       // G' * k
  m.gq = o;   o += N;       // G' * q
  m.ck = o;   o += C;       // (k_j * W'_j) . k
  m.cq = o;   o += C;       // (k_j * W'_j) . q
  m.misc = o; o += 4;       // k . q
  m.size = o;
  return m;
}

// FOLD = false: one decode token per sequence; true: fold the buffered records
// of the masked sequences (no token).
template <int N, bool FOLD>
__global__ void __launch_bounds__(kKdaThreads, 4) kda_kernel(const LayerDev d, const TokenIn in,
                                                              float* __restrict__ y,
                                                              const uint8_t* __restrict__ mask) {
  constexpr int SEG = N / 4, RPP = 32 / SEG, ROWS = kPass * RPP;
  extern __shared__ __align__(16) float sm[];
  const int P = d.P, H = d.H, G = d.G, C = d.C, L = d.L;
  const int R = kda_rows(N, P), parts = (P + R - 1) / R;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int c = lane % SEG, rsub = lane / SEG;
  const int blk = blockIdx.x;
  const int u = blk / parts, part = blk - u * parts;
  const int b = u / H, h = u - b * H;
  const int g = h / (H / G);
  const int r0 = part * R;  // first row of this CTA
  const size_t bh = static_cast<size_t>(u), bg = static_cast<size_t>(b) * G + g;
  const KdaSmem M = kda_smem(R, N, C);
  float* skt = sm + M.kt;
  float* su = sm + M.u;
  uint16_t* skb = reinterpret_cast<uint16_t*>(sm + M.kb);
  float* sk = sm + M.k;
  float* sq = sm + M.q;
  float* sG = sm + M.G;
  float* sgk = sm + M.gk;
  float* sgq = sm + M.gq;
  float* sck = sm + M.ck;
  float* scq = sm + M.cq;
  float* smisc = sm + M.misc;

  // The CTA's checkpoint rows (contiguous) by one bulk copy into shared memory, in
  // flight during the staging below; this thread's rows' values v.
  float4* S4 = reinterpret_cast<float4*>(d.ckpt + bh * static_cast<size_t>(P) * N);
  const int nrows = min(R, P - r0);
  uint64_t* tbar = reinterpret_cast<uint64_t*>(sm + M.bar);
  if (t == 0) {
    mbar_init(tbar, 1);
    mbar_expect_tx(tbar, static_cast<uint32_t>(nrows * N * 4));
    bulk_g2s(sm + M.tile, d.ckpt + (bh * P + r0) * static_cast<size_t>(N), static_cast<uint32_t>(nrows * N * 4), tbar);
  }
  __syncthreads();  // the barrier's initialisation before anyone waits on it
  const int wrow = r0 + warp * ROWS + rsub;  // row of pass 0 (pass k adds k RPP)
  float vr[kPass];
#pragma unroll
  for (int k = 0; k < kPass; ++k) {
    const int row = wrow + k * RPP;
    vr[k] = (!FOLD && row < r0 + nrows) ? bf(in.v[bh * P + row]) : 0.f;
  }

  // this token's key, query and channel decay (thread t < N holds channel t), beta
  const float gch = (!FOLD && t < N) ? in.g[bh * N + t] : 0.f;
  const uint16_t kbits = (!FOLD && t < N) ? in.k[bg * N + t] : 0, qbits = (!FOLD && t < N) ? in.q[bg * N + t] : 0;
  const float beta = FOLD ? 0.f : in.beta[bh];

  const int head = d.cursor[4 * b], cnt = d.cursor[4 * b + 1];
  const bool ok = static_cast<unsigned>(head) < static_cast<unsigned>(C) &&
                  static_cast<unsigned>(cnt) < static_cast<unsigned>(L);
  const bool work = ok && (!FOLD || mask == nullptr || mask[b] != 0);
  const int n = work ? cnt : 0;                  // buffered records
  const bool flush = work && (FOLD || cnt + 1 == L);
  // The last CTA of the sequence to have read its cursor advances it (no CTA reads
  // another sequence's cursor); thread 0's atomic overlaps the staging below.
  if (t == 0 && arrive_last(d.arrive, b, H * parts)) {
    if (!ok) {
      report_error(d.err, DEVERR_CURSOR, b);
    } else if (flush) {
      d.cursor[4 * b] = kslot(head, FOLD ? cnt : cnt + 1, C);
      d.cursor[4 * b + 1] = 0;
      d.cursor[4 * b + 2] = 1;
    } else if (FOLD) {
      d.cursor[4 * b + 2] = 0;
    } else {
      d.cursor[4 * b + 1] = cnt + 1;
      d.cursor[4 * b + 2] = 0;
    }
  }

  if (work) {
    // stage: the records' log decays (into skt, turned into decayed keys below) and
    // keys, this CTA's rows' deltas, this token's key and query
    const float* rg = d.r_g + bh * C * N;
    const uint16_t* rk = d.r_k + bg * C * N;
    const float* ru = d.r_u + bh * C * P;
    for (int e = t; e < n * N; e += kKdaThreads) {
      const int j = e / N, ch = e - j * N;
      const size_t src = static_cast<size_t>(kslot(head, j, C)) * N + ch;
      skt[e] = rg[src];
      skb[e] = rk[src];
    }
    for (int e = t; e < n * R; e += kKdaThreads) {
      const int j = e / R, r = e - j * R;
      su[r * M.ustride + j] = r0 + r < P ? ru[static_cast<size_t>(kslot(head, j, C)) * P + r0 + r] : 0.f;
    }
    if (!FOLD && t < N) {
      sk[t] = bf(kbits);
      sq[t] = bf(qbits);
    }
    __syncthreads();
    // channel-wise suffix scan: W'_j = exp(sum of the log decays after record j,
    // this token's included), decayed key k_j * W'_j; G' = exp(all of them)
    for (int ch = t; ch < N; ch += kKdaThreads) {
      float acc = gch;  // this token's log decay (0 for a fold)
      for (int j = n - 1; j >= 0; --j) {
        const float gj = skt[j * N + ch];
        skt[j * N + ch] = bf(skb[j * N + ch]) * expf(acc);
        acc += gj;
      }
      const float Gp = expf(acc);
      sG[ch] = Gp;
      if (!FOLD) {
        sgk[ch] = Gp * sk[ch];
        sgq[ch] = Gp * sq[ch];
      }
    }
    __syncthreads();
    if (!FOLD) {
      // record dots (k_j * W'_j) . k and . q, and k . q: one warp per item
      for (int it = warp; it < 2 * n + 1; it += kWarps) {
        const float* a = it < 2 * n ? skt + (it >> 1) * N : sk;
        const float* bvec = (it < 2 * n && (it & 1) == 0) ? sk : sq;
        float sacc = 0.f;
        for (int ch = lane; ch < N; ch += 32) sacc = fmaf(a[ch], bvec[ch], sacc);
        sacc = seg_sum<32>(sacc);
        if (lane == 0) {
          if (it == 2 * n) smisc[0] = sacc;
          else if ((it & 1) == 0) sck[it >> 1] = sacc;
          else scq[it >> 1] = sacc;
        }
      }
      __syncthreads();
    }

    // the rows have landed (bounded wait; on a timeout the CTA reports it, waits once
    // more for its copy and skips the sequence)
    if (!__syncthreads_and(mbar_wait_bounded(tbar, 0))) {
      if (t == 0) report_error(d.err, DEVERR_TIMEOUT, b);
      mbar_wait_bounded(tbar, 0);
      return;
    }
    float4 s[kPass];
#pragma unroll
    for (int k = 0; k < kPass; ++k) {
      const int row = wrow + k * RPP;
      s[k] = row < r0 + nrows ? reinterpret_cast<const float4*>(sm + M.tile)[(row - r0) * SEG + c]
                              : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float4 G4 = reinterpret_cast<const float4*>(sG)[c];
    const float4 gk4 = FOLD ? make_float4(0.f, 0.f, 0.f, 0.f) : reinterpret_cast<const float4*>(sgk)[c];
    const float4 gq4 = FOLD ? make_float4(0.f, 0.f, 0.f, 0.f) : reinterpret_cast<const float4*>(sgq)[c];
    const float4 k4 = FOLD ? make_float4(0.f, 0.f, 0.f, 0.f) : reinterpret_cast<const float4*>(sk)[c];
    const float kq = FOLD ? 0.f : smisc[0];
    const int slot = kslot(head, n, C);
    float ud[kPass];
    if (!FOLD) {
      // checkpoint terms (row totals over the row's lanes) and buffered-record terms
      // (the row's lanes split the records)
      float tk[kPass], tq[kPass];
#pragma unroll
      for (int k = 0; k < kPass; ++k) {
        const int row = wrow + k * RPP;
        float pk = dot4(s[k], gk4), pq = dot4(s[k], gq4);
        if (row < r0 + R && row < P) {
          const float* urow = su + (row - r0) * M.ustride;
          for (int j = c; j < n; j += SEG) {
            const float uj = urow[j];
            pk = fmaf(uj, sck[j], pk);
            pq = fmaf(uj, scq[j], pq);
          }
        }
        tk[k] = seg_sum<SEG>(pk);
        tq[k] = seg_sum<SEG>(pq);
      }
#pragma unroll
      for (int k = 0; k < kPass; ++k) {
        const int row = wrow + k * RPP;
        ud[k] = 0.f;
        if (row < r0 + R && row < P) {
          ud[k] = beta * (vr[k] - tk[k]);  // u = b (v - S k')
          if (c == 0) {
            y[bh * P + row] = fmaf(ud[k], kq, tq[k]);  // o = S q' + u (k . q)
            if (!flush) d.r_u[(bh * C + slot) * P + row] = ud[k];
          }
        }
      }
    }
    if (flush) {
      // S_new = S_ckpt Diag(G') + sum_j u_j (k_j * W'_j)^T (+ u k^T for a token)
#pragma unroll
      for (int k = 0; k < kPass; ++k) {
        const int row = wrow + k * RPP;
        if (row >= r0 + R || row >= P) continue;
        const float* urow = su + (row - r0) * M.ustride;
        float4 acc = make_float4(s[k].x * G4.x, s[k].y * G4.y, s[k].z * G4.z, s[k].w * G4.w);
        for (int j = 0; j < n; ++j) acc = axpy4(urow[j], reinterpret_cast<const float4*>(skt + j * N)[c], acc);
        if (!FOLD) acc = axpy4(ud[k], k4, acc);
        __stcs(S4 + static_cast<size_t>(row) * SEG + c, acc);
      }
    }
    // a non-flush step appends this token's record: g over the key channels and u
    // (above) per head, k once per key group (by the CTAs of the group's first head)
    if (!FOLD && !flush && part == 0 && t < N) {
      d.r_g[(bh * C + slot) * N + t] = gch;
      if (h % (H / G) == 0) d.r_k[(bg * C + slot) * N + t] = kbits;
    }
  } else {
    // nothing to do for this sequence: the rows' copy must still land before the
    // CTA's shared memory is released
    mbar_wait_bounded(tbar, 0);
  }
}

// ---- persistent decode step for d_state 128 ---------------------------------
//
// The same arithmetic as kda_kernel, organised like the other d_state-128 decode
// kernels: a CTA (two per SM) takes a contiguous range of units (sequence, head,
// block of 64 rows) and a producer warp stages the next unit by bulk copies into
// the other of two shared-memory stages while the eight computing warps work on
// the current one.  The first unit of a head stages the buffered records (log
// decays and keys over the key channels, the deltas of its rows) and this
// token's log decay, key, query and values, and builds the head's tables: the
// channel-wise suffix scan (the eight warps, two halves of the records) gives the
// decayed keys k_j W'_j and G', then the record dot products (a warp per item).
// The head's next units, when this CTA takes them right after, reuse those
// tables and stage only their checkpoint rows, their rows of the deltas and
// values.  Then eight rows a warp:
// the two checkpoint dot products (a transpose-reduce over the row's lanes), the
// records' terms (four lanes a row split the records), u, o and, on a flush
// step, the folded rows.  The CTAs read their sequences' cursors once, at the
// start; the last CTA of a sequence to count its units in advances the cursor.

constexpr int kPN = 128;                 // d_state
constexpr int kPR = 64;                  // state rows per unit
constexpr int kPThreads = kThreads + 32;  // eight computing warps and the producer warp
constexpr int kPMaxSeq = 64;             // sequences one CTA may cover
constexpr int kUStride = kPR + 8;        // floats per record row of the staged deltas (bank skew)

struct KdaPStage {  // byte offsets within one stage
  int tile, g, kb, u, tg, tk, tq, tv, size;
};

__host__ __device__ __forceinline__ KdaPStage kdap_stage(int C) {
  KdaPStage m;
  int o = 0;
  m.tile = o; o += kPR * kPN * 4;       // the unit's checkpoint rows
  m.g = o;    o += C * kPN * 4;         // records' log decays [j][N] (first unit of a head)
  m.kb = o;   o += C * kPN * 2;         // records' keys, bf16 [j][N] (first unit of a head)
  m.u = o;    o += C * kUStride * 4;    // records' deltas of the unit's rows [j][kUStride]
  m.tg = o;   o += kPN * 4;             // this token's log decay over the channels
  m.tk = o;   o += kPN * 2;             // this token's key, bf16
  m.tq = o;   o += kPN * 2;             // this token's query, bf16
  m.tv = o;   o += kPR * 2;             // this token's values of the unit's rows, bf16
  m.size = (o + 127) & ~127;
  return m;
}

struct KdaPTab {  // byte offsets of the head's tables (one set per CTA)
  int kt, vec, dots, ktok, size;
};

__host__ __device__ __forceinline__ KdaPTab kdap_tab(int C) {
  KdaPTab m;
  int o = 0;
  m.kt = o;   o += C * kPN * 4;         // decayed keys k_j W'_j [j][N]
  m.vec = o;  o += 3 * kPN * 4;         // G', G' k, G' q
  m.dots = o; o += (2 * C + 4) * 4;     // (k_j W'_j) . k and . q interleaved, then k . q
  m.ktok = o; o += kPN * 2;             // this token's key, bf16 (for the fold)
  m.size = (o + 127) & ~127;
  return m;
}

__host__ __device__ __forceinline__ int kdap_pers_bytes() { return 32 + 16 * kPMaxSeq + 16; }

__global__ void __launch_bounds__(kPThreads, 2) kdap_kernel(const LayerDev d, const TokenIn in,
                                                            float* __restrict__ y, const int per) {
  extern __shared__ __align__(128) unsigned char psm[];
  const int H = d.H, G = d.G, C = d.C, L = d.L, P = d.P;
  const int parts = P / kPR, ups = H * parts;  // units of a sequence
  const int total = d.B * ups;
  const int u0 = static_cast<int>(blockIdx.x) * per, u1 = min(u0 + per, total);
  if (u0 >= u1) return;
  const KdaPStage M = kdap_stage(C);
  const KdaPTab TB = kdap_tab(C);
  unsigned char* tab = psm + 2 * M.size;
  unsigned char* pers = tab + TB.size;
  uint64_t* full = reinterpret_cast<uint64_t*>(pers);  // [2] stage landed
  uint64_t* empty = full + 2;                          // [2] stage released by the eight computing warps
  int4* scur = reinterpret_cast<int4*>(pers + 32);     // per covered sequence: head, count, flags (1 ok, 2 flush)
  volatile int* sabort = reinterpret_cast<volatile int*>(pers + 32 + 16 * kPMaxSeq);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int b0 = u0 / ups, nseq = (u1 - 1) / ups - b0 + 1;
  if (t < nseq) {
    const int b = b0 + t;
    const int4 cv = reinterpret_cast<const int4*>(d.cursor)[b];
    const bool ok = static_cast<unsigned>(cv.x) < static_cast<unsigned>(C) &&
                    static_cast<unsigned>(cv.y) < static_cast<unsigned>(L);
    const bool fl = ok && cv.y + 1 == L;
    scur[t] = make_int4(ok ? cv.x : 0, ok ? cv.y : 0, (ok ? 1 : 0) | (fl ? 2 : 0), 0);
    // count this CTA's units of the sequence in (after its cursor has been read);
    // the last CTA of the sequence advances the cursor
    const int cnt = min(u1, (b + 1) * ups) - max(u0, b * ups);
    const int prev = atomicAdd(d.arrive + b, cnt);
    if (prev + cnt == ups) {
      atomicExch(d.arrive + b, 0);
      if (!ok) report_error(d.err, DEVERR_CURSOR, b);
      else if (fl) reinterpret_cast<int4*>(d.cursor)[b] = make_int4(kslot(cv.x, cv.y + 1, C), 0, 1, cv.w);
      else reinterpret_cast<int4*>(d.cursor)[b] = make_int4(cv.x, cv.y + 1, 0, cv.w);
    }
  }
  if (t == kThreads) {
    mbar_init(full, 1);
    mbar_init(full + 1, 1);
    mbar_init(empty, kThreads / 32);
    mbar_init(empty + 1, kThreads / 32);
    *sabort = 0;
  }
  __syncthreads();

  if (warp == kThreads / 32) {
    // ================================ producer ================================
    if (lane == 0) {
      int k = 0;           // units staged
      long long prev = -1;  // (b H + h) parts + part of the last staged unit
      for (int uu = u0; uu < u1; ++uu) {
        const int b = uu / ups, rem = uu - b * ups, h = rem / parts, part = rem - h * parts;
        const int4 cs = scur[b - b0];
        if (!(cs.z & 1)) continue;
        const long long key = static_cast<long long>(uu);
        const bool reuse = part > 0 && prev == key - 1;  // the head's tables are in place
        prev = key;
        const int s = k & 1;
        if (k >= 2 && !mbar_wait_bounded(empty + s, static_cast<uint32_t>(((k >> 1) - 1) & 1))) {
          report_error(d.err, DEVERR_TIMEOUT, b);
          *sabort = 1;
          break;
        }
        if (*sabort) break;
        unsigned char* st = psm + static_cast<size_t>(s) * M.size;
        const int head = cs.x, n = cs.y;
        const size_t bh = static_cast<size_t>(b) * H + h, bg = static_cast<size_t>(b) * G + h / (H / G);
        const int r0 = part * kPR;
        uint64_t* bar = full + s;
        mbar_expect_tx(bar, static_cast<uint32_t>(kPR * kPN * 4 + n * kPR * 4 + kPR * 2 +
                                                  (reuse ? 0 : n * kPN * 6 + kPN * 8)));
        bulk_g2s(st + M.tile, d.ckpt + (bh * P + r0) * kPN, kPR * kPN * 4, bar);
        for (int j = 0; j < n; ++j)
          bulk_g2s(st + M.u + j * kUStride * 4, d.r_u + (bh * C + kslot(head, j, C)) * P + r0, kPR * 4, bar);
        bulk_g2s(st + M.tv, in.v + bh * P + r0, kPR * 2, bar);
        if (!reuse) {
          const int seg1 = min(n, C - head), seg2 = n - seg1;
          if (seg1) {
            bulk_g2s(st + M.g, d.r_g + (bh * C + head) * kPN, seg1 * kPN * 4, bar);
            bulk_g2s(st + M.kb, d.r_k + (bg * C + head) * kPN, seg1 * kPN * 2, bar);
          }
          if (seg2) {
            bulk_g2s(st + M.g + seg1 * kPN * 4, d.r_g + bh * C * kPN, seg2 * kPN * 4, bar);
            bulk_g2s(st + M.kb + seg1 * kPN * 2, d.r_k + bg * C * kPN, seg2 * kPN * 2, bar);
          }
          bulk_g2s(st + M.tg, in.g + bh * kPN, kPN * 4, bar);
          bulk_g2s(st + M.tk, in.k + bg * kPN, kPN * 2, bar);
          bulk_g2s(st + M.tq, in.q + bg * kPN, kPN * 2, bar);
        }
        ++k;
      }
      // the copies in flight land before the CTA's shared memory is released
      for (int j = max(0, k - 2); j < k; ++j) mbar_wait_bounded(full + (j & 1), static_cast<uint32_t>((j >> 1) & 1));
    }
    return;
  }

  // ============================== computing warps ==============================
  const int rq = (lane >> 2) & 7, jl = lane & 3;  // row of the warp's eight, record lane
  float* kt = reinterpret_cast<float*>(tab + TB.kt);
  float* vec = reinterpret_cast<float*>(tab + TB.vec);
  float* dots = reinterpret_cast<float*>(tab + TB.dots);
  uint16_t* ktok = reinterpret_cast<uint16_t*>(tab + TB.ktok);
  int k = 0;
  long long prev = -1;
  for (int uu = u0; uu < u1; ++uu) {
    const int b = uu / ups, rem = uu - b * ups, h = rem / parts, part = rem - h * parts;
    const int4 cs = scur[b - b0];
    if (!(cs.z & 1)) continue;
    const bool reuse = part > 0 && prev == static_cast<long long>(uu) - 1;
    prev = uu;
    const int s = k & 1;
    const uint32_t par = static_cast<uint32_t>((k >> 1) & 1);
    ++k;
    const size_t bh = static_cast<size_t>(b) * H + h, bg = static_cast<size_t>(b) * G + h / (H / G);
    const int r0 = part * kPR;
    const int head = cs.x, n = cs.y;
    const bool flush = (cs.z & 2) != 0;
    const float beta = in.beta[bh];  // in flight during the scan
    // (also the barrier that keeps the head's tables until every warp is past the
    // previous unit)
    if (!compute_sync_and(mbar_wait_bounded(full + s, par))) {
      if (t == 0) {
        report_error(d.err, DEVERR_TIMEOUT, b);
        *sabort = 1;
      }
      break;
    }
    unsigned char* st = psm + static_cast<size_t>(s) * M.size;
    const float* su = reinterpret_cast<const float*>(st + M.u);
    const uint16_t* tv = reinterpret_cast<const uint16_t*>(st + M.tv);
    if (!reuse) {
      const float* rg = reinterpret_cast<const float*>(st + M.g);
      const uint16_t* kb = reinterpret_cast<const uint16_t*>(st + M.kb);
      const float* tg = reinterpret_cast<const float*>(st + M.tg);
      const uint16_t* tk = reinterpret_cast<const uint16_t*>(st + M.tk);
      const uint16_t* tq = reinterpret_cast<const uint16_t*>(st + M.tq);
      // channel-wise suffix scan: W'_j = exp(sum of the log decays after record j, this
      // token's included), decayed key k_j W'_j; G' = exp(all).  (The fast exponential:
      // its relative error, a few 1e-7 at these arguments, is far below the FP32
      // path's tolerance.)
      // All eight warps: threads 128-255 take records m..n-1 (m = n / 2), threads 0-127
      // records 0..m-1 after adding up the later records' log decays themselves.
      {
        const int ch = t & (kPN - 1), m = n >> 1;
        const bool late = t >= kPN;
        float acc = tg[ch];
        if (!late)
          for (int j = n - 1; j >= m; --j) acc += rg[j * kPN + ch];
        for (int j = late ? n - 1 : m - 1; j >= (late ? m : 0); --j) {
          kt[j * kPN + ch] = bf(kb[j * kPN + ch]) * __expf(acc);
          acc += rg[j * kPN + ch];
        }
        if (!late) {
          const float Gp = __expf(acc);
          vec[ch] = Gp;
          vec[kPN + ch] = Gp * bf(tk[ch]);
          vec[2 * kPN + ch] = Gp * bf(tq[ch]);
          ktok[ch] = tk[ch];
        }
      }
      compute_sync();
      // record dots (k_j W'_j) . k and . q (items 2 j and 2 j + 1), and k . q (item 2 n)
      for (int it = warp; it < 2 * n + 1; it += kThreads / 32) {
        const float4 a4 = it < 2 * n ? reinterpret_cast<const float4*>(kt + (it >> 1) * kPN)[lane]
                                     : bf4(reinterpret_cast<const uint2*>(tk)[lane]);
        const float4 b4 = bf4(reinterpret_cast<const uint2*>((it < 2 * n && (it & 1) == 0) ? tk : tq)[lane]);
        const float v = seg_sum<32>(dot4(a4, b4));
        if (lane == 0) dots[it] = v;
      }
      compute_sync();
    }
    // the warp's eight rows: checkpoint dot products, records' terms, u and o
    const int lr = 8 * warp + rq;  // this lane's row (of the unit) after the reductions
    const float4* tile4 = reinterpret_cast<const float4*>(st + M.tile);
    const float4 gk4 = reinterpret_cast<const float4*>(vec + kPN)[lane];
    const float4 gq4 = reinterpret_cast<const float4*>(vec + 2 * kPN)[lane];
    float4 srow[8];
    float pk[8], pq[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      srow[e] = tile4[(8 * warp + e) * (kPN / 4) + lane];
      pk[e] = dot4p(srow[e], gk4);
      pq[e] = dot4p(srow[e], gq4);
    }
    const float sk = reduce8(pk, lane), sq = reduce8(pq, lane);
    float rk = 0.f, rqv = 0.f;
    for (int j = jl; j < n; j += 4) {
      const float uj = su[j * kUStride + lr];
      rk = fmaf(uj, dots[2 * j], rk);
      rqv = fmaf(uj, dots[2 * j + 1], rqv);
    }
    rk += __shfl_xor_sync(0xffffffffu, rk, 1);
    rk += __shfl_xor_sync(0xffffffffu, rk, 2);
    rqv += __shfl_xor_sync(0xffffffffu, rqv, 1);
    rqv += __shfl_xor_sync(0xffffffffu, rqv, 2);
    const float kq = dots[2 * n];
    const float ut = beta * (bf(tv[lr]) - (sk + rk));  // u = b (v - S k')
    if (jl == 0) {
      y[bh * P + r0 + lr] = fmaf(ut, kq, sq + rqv);  // o = S q' + u (k . q)
      if (!flush) d.r_u[(bh * C + kslot(head, n, C)) * P + r0 + lr] = ut;
    }
    if (flush) {
      // S_new = S_ckpt Diag(G') + sum_j u_j (k_j W'_j)^T + u k^T, stored once
      const float4 G4 = reinterpret_cast<const float4*>(vec)[lane];
      const float4 k4 = bf4(reinterpret_cast<const uint2*>(ktok)[lane]);
      float4 acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        acc[e] = make_float4(srow[e].x * G4.x, srow[e].y * G4.y, srow[e].z * G4.z, srow[e].w * G4.w);
      for (int j = 0; j < n; ++j) {
        const float4 kt4 = reinterpret_cast<const float4*>(kt + j * kPN)[lane];
        const float4* uj4 = reinterpret_cast<const float4*>(su + j * kUStride + 8 * warp);
        const float4 ua = uj4[0], ub = uj4[1];
        const float ue[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = axpy4x2(ue[e], kt4, acc[e]);
      }
      float4* gS4 = reinterpret_cast<float4*>(d.ckpt + (bh * P + r0 + 8 * warp) * kPN);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float ue = __shfl_sync(0xffffffffu, ut, 4 * e);
        __stcs(gS4 + e * (kPN / 4) + lane, axpy4(ue, k4, acc[e]));
      }
    } else if (part == 0 && t < kPN) {
      // this token's record: g over the key channels per head, k once per key group
      // (the first unit of a head stages this token's inputs)
      const int slot = kslot(head, n, C);
      d.r_g[(bh * C + slot) * kPN + t] = reinterpret_cast<const float*>(st + M.tg)[t];
      if (h % (H / G) == 0) d.r_k[(bg * C + slot) * kPN + t] = ktok[t];
    }
    // the warp is done with the stage
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + s);
  }
}

template <int N, bool FOLD>
cudaError_t launch_kda_n(const LayerDev& d, const TokenIn& in, float* y, const uint8_t* mask, cudaStream_t s) {
  const int R = kda_rows(N, d.P);
  const int parts = (d.P + R - 1) / R;
  const size_t smem = static_cast<size_t>(kda_smem(R, N, d.C).size) * 4;
  auto kernel = kda_kernel<N, FOLD>;
  const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  kernel<<<d.B * d.H * parts, kKdaThreads, smem, s>>>(d, in, y, mask);
  return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// the persistent decode: d_state 128, whole 64-row units, every staged source
// 16-byte aligned, two stages in shared memory
size_t kdap_smem(const LayerDev& d) {
  return 2 * static_cast<size_t>(kdap_stage(d.C).size) + kdap_tab(d.C).size + kdap_pers_bytes();
}

bool kdap_supports(const LayerDev& d, const TokenIn& in) {
  return d.N == kPN && d.P % kPR == 0 && d.H % d.G == 0 && kdap_smem(d) <= 227u * 1024u && aligned16(d.ckpt) &&
         aligned16(d.r_g) && aligned16(d.r_k) && aligned16(d.r_u) && aligned16(in.g) && aligned16(in.k) &&
         aligned16(in.q) && aligned16(in.v);
}

cudaError_t launch_kdap(const LayerDev& d, const TokenIn& in, float* y, cudaStream_t s) {
  const size_t smem = kdap_smem(d);
  const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kdap_kernel), smem);
  if (e != cudaSuccess) return e;
  const int ups = d.H * (d.P / kPR);
  const int total = d.B * ups;
  const int per_sm = smem + 1024 <= 114u * 1024u ? 2 : 1;
  int grid = (d.num_sms > 0 ? d.num_sms : 1) * per_sm;
  if (grid > total) grid = total;
  int per = (total + grid - 1) / grid;
  while (per / ups + 2 > kPMaxSeq) {  // sequences a CTA covers
    grid *= 2;
    per = (total + grid - 1) / grid;
  }
  grid = (total + per - 1) / per;
  kdap_kernel<<<grid, kPThreads, smem, s>>>(d, in, y, per);
  return cudaGetLastError();
}

template <bool FOLD>
cudaError_t launch_kda_any(const LayerDev& d, const TokenIn& in, float* y, const uint8_t* mask, cudaStream_t s) {
  switch (d.N) {
    case 16: return launch_kda_n<16, FOLD>(d, in, y, mask, s);
    case 32: return launch_kda_n<32, FOLD>(d, in, y, mask, s);
    case 64: return launch_kda_n<64, FOLD>(d, in, y, mask, s);
    case 128: return launch_kda_n<128, FOLD>(d, in, y, mask, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_kda_decode(const LayerDev& d, const TokenIn& in, float* y, cudaStream_t s) {
  if (kdap_supports(d, in)) return launch_kdap(d, in, y, s);
  return launch_kda_any<false>(d, in, y, nullptr, s);
}

cudaError_t launch_kda_fold(const LayerDev& d, const uint8_t* mask, cudaStream_t s) {
  return launch_kda_any<true>(d, TokenIn{}, nullptr, mask, s);
}

}  // namespace rs
