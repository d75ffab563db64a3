// Speculative verification of T draft tokens per sequence, chunkwise form.
//
// With n committed records j = 0..n-1 buffered since the checkpoint and the
// T drafts appended as records n..n+T-1, the output of draft position tau is
// never formed through a state:
//   O = S_ckpt Q D + V (W ⊙ (K^T Q))
// Q = [q_0..q_{T-1}], D = diag(prod_{i<=n+tau} a_i), K and V the keys and
// value vectors of the n+T records, W[j][tau] = prod_{i=j+1..n+tau} a_i for
// j <= n+tau and 0 above ("ReplaySSM caches SSM inputs instead of state"
// (richland.au), "What shipped", the paragraph on the second, subtler
// benefit).  K^T Q is formed once per CTA for the group's keys and queries.
// For Gated DeltaNet the draft deltas u_tau are unknown until S_{n+tau} k_tau
// is known; they solve the unit lower-triangular T x T system
//   u_tau + sum_{s<tau} M[tau][s] u_s = R_tau,
//   R_tau   = b_tau (v_tau - a_tau (S_{n+tau} k_tau restricted to committed records)),
//   M[tau][s] = b_tau a_tau prod_{n+s<i<n+tau} a_i (k_{n+s} . k_tau),
// solved per state row by forward substitution, after which V above holds
// the committed u_j followed by the draft u_tau.
//
// The drafts are appended to the ring after the committed records; the
// cursor does not move (commit advances it).
#include "common.cuh"

namespace rs {
namespace {

constexpr int kTMax = 4;   // drafts per verify handled by one instantiation

__device__ __forceinline__ int ring_slot(int head, int j, int C) {
  int s = head + j;
  return s >= C ? s - C : s;
}

template <int N>
__device__ __forceinline__ void dots_rows(float* dst, int stride, const float* sK, const float* vec, int count) {
  // dst[j * stride] = sK[j] . vec, one warp per record
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int j = warp; j < count; j += kThreads / 32) {
    float acc = 0.f;
    for (int e = lane; e < N; e += 32) acc = fmaf(sK[j * N + e], vec[e], acc);
    acc = seg_sum<32>(acc);
    if (lane == 0) dst[j * stride] = acc;
  }
}

// ---------------------------------------------------------------------------
template <int N>
__global__ void __launch_bounds__(kThreads) m2_verify_kernel(const LayerDev d, const TokenIn in, const int T,
                                                             float* __restrict__ y) {
  constexpr int SEG = N / 4;
  extern __shared__ __align__(128) unsigned char smem[];
  const int P = d.P, H = d.H, G = d.G, C = d.C, L = d.L;
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh - b * H;
  const int hpg = H / G, g = h / hpg;
  const int t = threadIdx.x;
  const int tile = P * N;

  float* sS = reinterpret_cast<float*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sS + tile);
  float* sQ = reinterpret_cast<float*>(bar + 2);  // [kTMax][N]
  float* sK = sQ + kTMax * N;                     // [C][N]
  float* sX = sK + C * N;                         // [C][P]
  float* sD = sX + C * P;                         // [C][kTMax]  k_j . q_tau
  float* sW = sD + C * kTMax;                     // [C][kTMax]  decay weights
  float* sla = sW + C * kTMax;                    // [C]
  float* sdt = sla + C;                           // [C]
  float* sry = sdt + C;                           // [kTMax][P]
  float* scS = sry + kTMax * P;                   // [kTMax]

  float* gS = d.ckpt + static_cast<size_t>(bh) * tile;
  if (t == 0) {
    mbar_init(bar, 1);
    mbar_expect_tx(bar, static_cast<uint32_t>(tile) * 4u);
    bulk_g2s(sS, gS, static_cast<uint32_t>(tile) * 4u, bar);
  }

  const int head = d.cursor[4 * b], cnt = d.cursor[4 * b + 1];
  const bool ok = static_cast<unsigned>(head) < static_cast<unsigned>(C) &&
                  static_cast<unsigned>(cnt) < static_cast<unsigned>(L) && cnt + T <= C;
  const int n = ok ? cnt : 0;
  const int nr = n + T;
  const size_t bg = static_cast<size_t>(b) * G + g;

  // queries and keys of the drafts; keys, log decays, dt and x of all records
  for (int i = t; i < T * N; i += kThreads) {
    const int tau = i / N, e = i - tau * N;
    const size_t src = ((static_cast<size_t>(b) * T + tau) * G + g) * N + e;
    sQ[i] = bf(in.Cm[src]);
    sK[(n + tau) * N + e] = bf(in.Bm[src]);
  }
  for (int i = t; i < n * N; i += kThreads) {
    const int j = i / N, e = i - j * N;
    sK[i] = bf(d.r_B[(bg * C + ring_slot(head, j, C)) * N + e]);
  }
  if (t < nr) {
    if (t < n) {
      const size_t s = static_cast<size_t>(bh) * d.Cp + ring_slot(head, t, C);
      sla[t] = d.r_la[s];
      sdt[t] = bf(d.r_dt[s]);
    } else {
      const float dtc = bf(in.dt[(static_cast<size_t>(b) * T + (t - n)) * H + h]);
      sdt[t] = dtc;
      sla[t] = dtc * in.A[h];
    }
  }
  for (int i = t; i < nr * P; i += kThreads) {
    const int j = i / P, r = i - j * P;
    const uint16_t xv = j < n ? d.r_x[(static_cast<size_t>(bh) * C + ring_slot(head, j, C)) * P + r]
                              : in.x[((static_cast<size_t>(b) * T + (j - n)) * H + h) * P + r];
    sX[i] = bf(xv);
  }
  __syncthreads();

  // K^T Q for all records and draft queries
  for (int tau = 0; tau < T; ++tau) dots_rows<N>(sD + tau, kTMax, sK, sQ + tau * N, nr);
  // decay weights: W[j][tau] = prod_{i=j+1..n+tau} a_i, D[tau] = prod_{i<=n+tau} a_i
  if (t < T) {
    const int tau = t;
    float e = 0.f;
    for (int j = nr - 1; j > n + tau; --j) sW[j * kTMax + tau] = 0.f;
    for (int j = n + tau; j >= 0; --j) {
      sW[j * kTMax + tau] = expf(e);
      e += sla[j];
    }
    scS[tau] = expf(e);
  }
  __syncthreads();
  for (int i = t; i < T * P; i += kThreads) {
    const int tau = i / P, r = i - tau * P;
    float acc = 0.f;
    for (int j = 0; j <= n + tau; ++j)
      acc = fmaf(sW[j * kTMax + tau] * sD[j * kTMax + tau], sdt[j] * sX[j * P + r], acc);
    sry[i] = acc;
  }

  const bool tile_ok = __syncthreads_and(mbar_wait_bounded(bar, 0) ? 1 : 0) != 0;
  if (!tile_ok) {
    if (t == 0) report_error(d.err, DEVERR_TIMEOUT, b);
    mbar_wait_bounded(bar, 0);
  }
  if (!ok) {
    if (t == 0) report_error(d.err, DEVERR_CURSOR, b);
    return;
  }
  if (!tile_ok) return;
  if (h == 0 && t == 0) d.cursor[4 * b + 2] = 0;  // verify folds nothing

  // O[tau][r] = D[tau] (S_ckpt q_tau)[r] + sum_j W[j][tau] (k_j . q_tau) v_j[r]
  const int c4 = t % SEG;
  float4 q4[kTMax];
#pragma unroll
  for (int tau = 0; tau < kTMax; ++tau)
    q4[tau] = tau < T ? reinterpret_cast<const float4*>(sQ + tau * N)[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* sS4 = reinterpret_cast<const float4*>(sS);
  const int nf4 = tile / 4;
  for (int f = t; f < nf4; f += kThreads) {
    const float4 s4 = sS4[f];
    const int r = f / SEG;
#pragma unroll
    for (int tau = 0; tau < kTMax; ++tau) {
      if (tau < T) {
        const float part = seg_sum<SEG>(dot4(s4, q4[tau]));
        if (c4 == 0)
          y[((static_cast<size_t>(b) * T + tau) * H + h) * P + r] = fmaf(scS[tau], part, sry[tau * P + r]);
      }
    }
  }
  // append the drafts after the committed records
  for (int i = t; i < T * P; i += kThreads) {
    const int tau = i / P, r = i - tau * P;
    d.r_x[(static_cast<size_t>(bh) * C + ring_slot(head, n + tau, C)) * P + r] =
        in.x[((static_cast<size_t>(b) * T + tau) * H + h) * P + r];
  }
  if (t < T) {
    const size_t s = static_cast<size_t>(bh) * d.Cp + ring_slot(head, n + t, C);
    d.r_dt[s] = in.dt[(static_cast<size_t>(b) * T + t) * H + h];
    d.r_la[s] = sla[n + t];
  }
  if (h % hpg == 0) {
    for (int i = t; i < T * N; i += kThreads) {
      const int tau = i / N, e = i - tau * N;
      d.r_B[(bg * C + ring_slot(head, n + tau, C)) * N + e] =
          in.Bm[((static_cast<size_t>(b) * T + tau) * G + g) * N + e];
    }
  }
}

// ---------------------------------------------------------------------------
template <int N>
__global__ void __launch_bounds__(kThreads) gdn_verify_kernel(const LayerDev d, const TokenIn in, const int T,
                                                              float* __restrict__ o) {
  constexpr int SEG = N / 4;
  extern __shared__ __align__(128) unsigned char smem[];
  const int P = d.P, H = d.H, G = d.G, C = d.C, L = d.L;
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh - b * H;
  const int hpg = H / G, g = h / hpg;
  const int t = threadIdx.x;
  const int tile = P * N;

  float* sS = reinterpret_cast<float*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sS + tile);
  float* sQ = reinterpret_cast<float*>(bar + 2);  // [kTMax][N] draft queries
  float* sK = sQ + kTMax * N;                     // [C][N] keys: committed, then drafts
  float* sU = sK + C * N;                         // [C][P] committed u_j
  float* sDk = sU + C * P;                        // [C][kTMax] k_j . k_tau
  float* sDq = sDk + C * kTMax;                   // [C][kTMax] k_j . q_tau
  float* sWk = sDq + C * kTMax;                   // [C][kTMax] prod_{i=j+1..n+tau-1} a_i
  float* sWq = sWk + C * kTMax;                   // [C][kTMax] prod_{i=j+1..n+tau} a_i
  float* sla = sWq + C * kTMax;                   // [C]
  float* srk = sla + C;                           // [kTMax][P]
  float* srq = srk + kTMax * P;                   // [kTMax][P]
  float* sv = srq + kTMax * P;                    // [kTMax][P] draft v
  float* sM = sv + kTMax * P;                     // [kTMax][kTMax] solve coefficients
  float* sg1 = sM + kTMax * kTMax;                // [kTMax] prod_{i<n+tau} a_i
  float* sg2 = sg1 + kTMax;                       // [kTMax] prod_{i<=n+tau} a_i
  float* sab = sg2 + kTMax;                       // [2][kTMax] a_tau, beta_tau

  float* gS = d.ckpt + static_cast<size_t>(bh) * tile;
  if (t == 0) {
    mbar_init(bar, 1);
    mbar_expect_tx(bar, static_cast<uint32_t>(tile) * 4u);
    bulk_g2s(sS, gS, static_cast<uint32_t>(tile) * 4u, bar);
  }

  const int head = d.cursor[4 * b], cnt = d.cursor[4 * b + 1];
  const bool ok = static_cast<unsigned>(head) < static_cast<unsigned>(C) &&
                  static_cast<unsigned>(cnt) < static_cast<unsigned>(L) && cnt + T <= C;
  const int n = ok ? cnt : 0;
  const int nr = n + T;
  const size_t bg = static_cast<size_t>(b) * G + g;

  for (int i = t; i < T * N; i += kThreads) {
    const int tau = i / N, e = i - tau * N;
    const size_t src = ((static_cast<size_t>(b) * T + tau) * G + g) * N + e;
    sQ[i] = bf(in.q[src]);
    sK[(n + tau) * N + e] = bf(in.k[src]);
  }
  for (int i = t; i < n * N; i += kThreads) {
    const int j = i / N, e = i - j * N;
    sK[i] = bf(d.r_k[(bg * C + ring_slot(head, j, C)) * N + e]);
  }
  for (int i = t; i < n * P; i += kThreads) {
    const int j = i / P, r = i - j * P;
    sU[i] = d.r_u[(static_cast<size_t>(bh) * C + ring_slot(head, j, C)) * P + r];
  }
  for (int i = t; i < T * P; i += kThreads) {
    const int tau = i / P, r = i - tau * P;
    sv[i] = bf(in.v[((static_cast<size_t>(b) * T + tau) * H + h) * P + r]);
  }
  if (t < nr) {
    if (t < n) {
      sla[t] = d.r_g[static_cast<size_t>(bh) * d.Cp + ring_slot(head, t, C)];
    } else {
      const size_t s = (static_cast<size_t>(b) * T + (t - n)) * H + h;
      sla[t] = in.g[s];
      sab[t - n] = expf(in.g[s]);
      sab[kTMax + t - n] = in.beta[s];
    }
  }
  __syncthreads();

  for (int tau = 0; tau < T; ++tau) {
    dots_rows<N>(sDk + tau, kTMax, sK, sK + (n + tau) * N, nr);
    dots_rows<N>(sDq + tau, kTMax, sK, sQ + tau * N, nr);
  }
  if (t < T) {
    const int tau = t;
    // sWq[j][tau] = prod_{i=j+1..n+tau} a_i ; sWk[j][tau] = prod_{i=j+1..n+tau-1} a_i
    float e = 0.f;
    for (int j = n + tau; j >= 0; --j) {
      sWq[j * kTMax + tau] = expf(e);
      e += sla[j];
    }
    sg2[tau] = expf(e);
    e = 0.f;
    for (int j = n + tau - 1; j >= 0; --j) {
      sWk[j * kTMax + tau] = expf(e);
      e += sla[j];
    }
    sg1[tau] = expf(e);
  }
  __syncthreads();
  if (t < T * kTMax) {
    const int tau = t / kTMax, s = t - tau * kTMax;
    sM[t] = (s < tau) ? sab[kTMax + tau] * sab[tau] * sWk[(n + s) * kTMax + tau] * sDk[(n + s) * kTMax + tau]
                      : 0.f;
  }
  for (int i = t; i < T * P; i += kThreads) {
    const int tau = i / P, r = i - tau * P;
    float ak = 0.f, aq = 0.f;
    for (int j = 0; j < n; ++j) {
      const float u = sU[j * P + r];
      ak = fmaf(sWk[j * kTMax + tau] * sDk[j * kTMax + tau], u, ak);
      aq = fmaf(sWq[j * kTMax + tau] * sDq[j * kTMax + tau], u, aq);
    }
    srk[i] = ak;
    srq[i] = aq;
  }

  const bool tile_ok = __syncthreads_and(mbar_wait_bounded(bar, 0) ? 1 : 0) != 0;
  if (!tile_ok) {
    if (t == 0) report_error(d.err, DEVERR_TIMEOUT, b);
    mbar_wait_bounded(bar, 0);
  }
  if (!ok) {
    if (t == 0) report_error(d.err, DEVERR_CURSOR, b);
    return;
  }
  if (!tile_ok) return;
  if (h == 0 && t == 0) d.cursor[4 * b + 2] = 0;  // verify folds nothing

  const int c4 = t % SEG;
  float4 k4[kTMax], q4[kTMax];
#pragma unroll
  for (int tau = 0; tau < kTMax; ++tau) {
    k4[tau] = tau < T ? reinterpret_cast<const float4*>(sK + (n + tau) * N)[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
    q4[tau] = tau < T ? reinterpret_cast<const float4*>(sQ + tau * N)[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float4* sS4 = reinterpret_cast<const float4*>(sS);
  const int nf4 = tile / 4;
  for (int f = t; f < nf4; f += kThreads) {
    const float4 s4 = sS4[f];
    const int r = f / SEG;
    float pk[kTMax], pq[kTMax];
#pragma unroll
    for (int tau = 0; tau < kTMax; ++tau) {
      pk[tau] = 0.f;
      pq[tau] = 0.f;
      if (tau < T) {
        pk[tau] = seg_sum<SEG>(dot4(s4, k4[tau]));
        pq[tau] = seg_sum<SEG>(dot4(s4, q4[tau]));
      }
    }
    if (c4 == 0) {
      float u[kTMax];
#pragma unroll
      for (int tau = 0; tau < kTMax; ++tau) {
        if (tau < T) {
          const float Sk = fmaf(sg1[tau], pk[tau], srk[tau * P + r]);
          float rhs = sab[kTMax + tau] * (sv[tau * P + r] - sab[tau] * Sk);
#pragma unroll
          for (int s = 0; s < kTMax; ++s)
            if (s < tau) rhs = fmaf(-sM[tau * kTMax + s], u[s], rhs);
          u[tau] = rhs;
        }
      }
#pragma unroll
      for (int tau = 0; tau < kTMax; ++tau) {
        if (tau < T) {
          float acc = fmaf(sg2[tau], pq[tau], srq[tau * P + r]);
#pragma unroll
          for (int s = 0; s < kTMax; ++s)
            if (s <= tau) acc = fmaf(sWq[(n + s) * kTMax + tau] * sDq[(n + s) * kTMax + tau], u[s], acc);
          o[((static_cast<size_t>(b) * T + tau) * H + h) * P + r] = acc;
          d.r_u[(static_cast<size_t>(bh) * C + ring_slot(head, n + tau, C)) * P + r] = u[tau];
        }
      }
    }
  }
  if (t < T) {
    d.r_g[static_cast<size_t>(bh) * d.Cp + ring_slot(head, n + t, C)] = sla[n + t];
  }
  if (h % hpg == 0) {
    for (int i = t; i < T * N; i += kThreads) {
      const int tau = i / N, e = i - tau * N;
      d.r_k[(bg * C + ring_slot(head, n + tau, C)) * N + e] =
          in.k[((static_cast<size_t>(b) * T + tau) * G + g) * N + e];
    }
  }
}

size_t verify_smem_bytes(const LayerDev& d) {
  const size_t tile = static_cast<size_t>(d.P) * d.N * 4;
  const size_t C = d.C, P = d.P, N = d.N, TM = kTMax;
  size_t floats;
  if (d.kind == 0)
    floats = TM * N + C * N + C * P + 2 * C * TM + 2 * C + TM * P + TM;
  else
    floats = TM * N + C * N + C * P + 4 * C * TM + C + 3 * TM * P + TM * TM + 4 * TM;
  return tile + 16 + floats * 4;
}

template <typename K>
cudaError_t run(K kernel, const LayerDev& d, const TokenIn& in, int T, float* y, size_t smem, cudaStream_t s) {
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  kernel<<<d.B * d.H, kThreads, smem, s>>>(d, in, T, y);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify(const LayerDev& d, const TokenIn& in, int T, float* y, cudaStream_t s) {
  if (T < 1 || T > kTMax) return cudaErrorInvalidValue;
  const size_t smem = verify_smem_bytes(d);
  if (d.kind == 0) {
    switch (d.N) {
      case 16: return run(m2_verify_kernel<16>, d, in, T, y, smem, s);
      case 32: return run(m2_verify_kernel<32>, d, in, T, y, smem, s);
      case 64: return run(m2_verify_kernel<64>, d, in, T, y, smem, s);
      case 128: return run(m2_verify_kernel<128>, d, in, T, y, smem, s);
    }
  } else {
    switch (d.N) {
      case 16: return run(gdn_verify_kernel<16>, d, in, T, y, smem, s);
      case 32: return run(gdn_verify_kernel<32>, d, in, T, y, smem, s);
      case 64: return run(gdn_verify_kernel<64>, d, in, T, y, smem, s);
      case 128: return run(gdn_verify_kernel<128>, d, in, T, y, smem, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace rs
