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
  return launch_kda_any<false>(d, in, y, nullptr, s);
}

cudaError_t launch_kda_fold(const LayerDev& d, const uint8_t* mask, cudaStream_t s) {
  return launch_kda_any<true>(d, TokenIn{}, nullptr, mask, s);
}

}  // namespace rs
