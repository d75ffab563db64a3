// Standard decode step: the output-only non-flush body and the flush body,
// selected per sequence from its device-resident cursor inside one launch.
//
// One CTA serves one (sequence, head) state matrix S_ckpt [P][N].  Thread 0
// starts a bulk copy (cp.async.bulk, the untiled TMA path) of the whole
// matrix into shared memory before anything else; while it is in flight the
// CTA gathers the token's inputs and the buffered records, forms the per-group
// key dot products and the decay weights, and only then waits for the tile.
// The matrix is read from HBM exactly once.  A non-flush CTA writes only the
// output row and the appended record; a flush CTA also writes the folded
// checkpoint once.  The last CTA of a sequence to finish advances its cursor.
//
// Unrolled form ("ReplaySSM caches SSM inputs instead of state" (richland.au),
// "What shipped", the paragraph on unrolling the recurrence): with records
// j = 0..n-1 buffered since the checkpoint and the current token as record n,
//   S_n = gamma S_ckpt + sum_{j<=n} w_j v_j k_j^T,
//   w_j = prod_{i=j+1..n} a_i,  gamma = prod_{i=0..n} a_i,
// so the Mamba-2 output is
//   y = gamma (S_ckpt q) + sum_{j<=n} w_j (k_j . q) v_j,
// with the key dot products k_j . q shared by the heads of a group.  Gated
// DeltaNet buffers (g, u, k) records with u = b (v - a S_{t-1} k), which makes
// its state S_t = a S_{t-1} + u k^T of the same form; its step needs S_{t-1} k
// and S_{t-1} q from the same pass over S_ckpt.
#include "common.cuh"

namespace rs {
namespace {

__device__ __forceinline__ int ring_slot(int head, int j, int C) {
  int s = head + j;
  return s >= C ? s - C : s;
}

// Records per 16-byte-chunk pass when TPR threads share one key row.
template <int N>
struct KeyLoad {
  static constexpr int TPR = N / 8;
  static constexpr int RPP = kThreads / TPR;
  static constexpr int NPASS = (kMaxRec + RPP - 1) / RPP;
};

// Load bf16 key rows of records 0..n-1 from the ring (slot order from head)
// into sK[j][N] as f32.
template <int N>
__device__ __forceinline__ void load_ring_keys(float* sK, const uint16_t* ring_keys_bg, int head, int n,
                                               int C) {
  using KL = KeyLoad<N>;
  const int t = threadIdx.x;
#pragma unroll
  for (int pass = 0; pass < KL::NPASS; ++pass) {
    const int j = pass * KL::RPP + t / KL::TPR;
    const int e0 = (t % KL::TPR) * 8;
    if (j < n) {
      const uint4 raw =
          *reinterpret_cast<const uint4*>(ring_keys_bg + static_cast<size_t>(ring_slot(head, j, C)) * N + e0);
      float v[8];
      bf8(raw, v);
      float4* dst = reinterpret_cast<float4*>(sK + j * N + e0);
      dst[0] = make_float4(v[0], v[1], v[2], v[3]);
      dst[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

// dst[j] = sK[j] . vec for j = 0..count-1 (TPR threads per record).
template <int N>
__device__ __forceinline__ void key_dots(float* dst, const float* sK, const float* vec, int count) {
  using KL = KeyLoad<N>;
  const int t = threadIdx.x;
#pragma unroll
  for (int pass = 0; pass < KL::NPASS; ++pass) {
    const int j = pass * KL::RPP + t / KL::TPR;
    const int e0 = (t % KL::TPR) * 8;
    float acc = 0.f;
    if (j < count) {
      const float4* kk = reinterpret_cast<const float4*>(sK + j * N + e0);
      const float4* vv = reinterpret_cast<const float4*>(vec + e0);
      acc = dot4(kk[0], vv[0]) + dot4(kk[1], vv[1]);
    }
    acc = seg_sum<KL::TPR>(acc);
    if (j < count && (t % KL::TPR) == 0) dst[j] = acc;
  }
}

__device__ __forceinline__ void start_tile_copy(float* sS, const float* gS, uint32_t bytes, uint64_t* bar) {
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_expect_tx(bar, bytes);
    bulk_g2s(sS, gS, bytes, bar);
  }
}

// All threads: wait for the staged tile.  CTA-uniform result; on timeout the
// error word is set and the copy is waited for once more before returning.
__device__ __forceinline__ bool finish_tile_copy(uint64_t* bar, int* err, int seq) {
  const bool ok = __syncthreads_and(mbar_wait_bounded(bar, 0) ? 1 : 0) != 0;
  if (!ok) {
    if (threadIdx.x == 0) report_error(err, DEVERR_TIMEOUT, seq);
    mbar_wait_bounded(bar, 0);
  }
  return ok;
}

// ---------------------------------------------------------------------------
// Mamba-2
// ---------------------------------------------------------------------------
template <int N>
__global__ void __launch_bounds__(kThreads) m2_decode_kernel(const LayerDev d, const TokenIn in,
                                                             float* __restrict__ y) {
  constexpr int SEG = N / 4;  // lanes per state row, one float4 each
  extern __shared__ __align__(128) unsigned char smem[];

  const int P = d.P, H = d.H, G = d.G, C = d.C, L = d.L;
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh - b * H;
  const int hpg = H / G, g = h / hpg;
  const int t = threadIdx.x;
  const int tile = P * N;
  const size_t bg = static_cast<size_t>(b) * G + g;

  float* sS = reinterpret_cast<float*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sS + tile);
  float* sq = reinterpret_cast<float*>(bar + 2);  // [N]   q = C of the group
  float* sK = sq + N;                             // [C][N] keys of records 0..n
  float* sX = sK + C * N;                         // [C][P] x_j, then fold coefficients
  float* sdot = sX + C * P;                       // [C]   k_j . q
  float* sW = sdot + C;                           // [C]   w_j
  float* sla = sW + C;                            // [C]   log a_j
  float* sdt = sla + C;                           // [C]   dt_j
  float* sry = sdt + C;                           // [P]   sum_j w_j (k_j . q) v_j
  float* sc = sry + P;                            // [1]   gamma

  float* gS = d.ckpt + static_cast<size_t>(bh) * tile;
  start_tile_copy(sS, gS, static_cast<uint32_t>(tile) * 4u, bar);

  // --- cursor and gathers (overlap the tile copy) ---
  const int head = d.cursor[4 * b], cnt = d.cursor[4 * b + 1];
  const bool ok = static_cast<unsigned>(head) < static_cast<unsigned>(C) &&
                  static_cast<unsigned>(cnt) < static_cast<unsigned>(L);
  const int n = ok ? cnt : 0;
  const bool flush = ok && (cnt + 1 == L);

  for (int i = t; i < N; i += kThreads) {
    sq[i] = bf(in.Cm[bg * N + i]);
    sK[n * N + i] = bf(in.Bm[bg * N + i]);
  }
  load_ring_keys<N>(sK, d.r_B + bg * C * N, head, n, C);
  if (t < n) {
    const size_t s = static_cast<size_t>(bh) * C + ring_slot(head, t, C);
    sla[t] = d.r_la[s];
    sdt[t] = bf(d.r_dt[s]);
  } else if (t == n) {
    const float dtc = bf(in.dt[bh]);
    sdt[n] = dtc;
    sla[n] = dtc * in.A[h];
  }
  for (int i = t; i < (n + 1) * P; i += kThreads) {
    const int j = i / P, r = i - j * P;
    const uint16_t xv = j < n ? d.r_x[(static_cast<size_t>(bh) * C + ring_slot(head, j, C)) * P + r]
                              : in.x[static_cast<size_t>(bh) * P + r];
    sX[i] = bf(xv);
  }
  __syncthreads();

  // --- k_j . q for j = 0..n, decay weights ---
  key_dots<N>(sdot, sK, sq, n + 1);
  if (t == 0) {
    float e = 0.f;
    for (int j = n; j >= 0; --j) {
      sW[j] = expf(e);
      e += sla[j];
    }
    sc[0] = expf(e);
  }
  __syncthreads();

  // --- per-row buffered term; fold coefficients w_j v_j[r] on flush steps ---
  for (int r = t; r < P; r += kThreads) {
    float acc = 0.f;
    for (int j = 0; j <= n; ++j) {
      const float v = sdt[j] * sX[j * P + r];
      acc = fmaf(sW[j] * sdot[j], v, acc);
      if (flush) sX[j * P + r] = sW[j] * v;
    }
    sry[r] = acc;
  }

  const bool tile_ok = finish_tile_copy(bar, d.err, b);  // includes __syncthreads
  const bool work = ok && tile_ok;

  if (work) {
    const float gamma = sc[0];
    const int c4 = t % SEG;
    const float4 q4 = reinterpret_cast<const float4*>(sq)[c4];
    const float4* sS4 = reinterpret_cast<const float4*>(sS);
    float* yrow = y + static_cast<size_t>(bh) * P;
    const int nf4 = tile / 4;
    if (!flush) {
      for (int f = t; f < nf4; f += kThreads) {
        const float part = seg_sum<SEG>(dot4(sS4[f], q4));
        if (c4 == 0) yrow[f / SEG] = fmaf(gamma, part, sry[f / SEG]);
      }
    } else {
      float4* gS4 = reinterpret_cast<float4*>(gS);
      for (int f0 = 0; f0 < nf4; f0 += 8 * kThreads) {
        float4 acc[8];
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) {
          const int f = f0 + ii * kThreads + t;
          if (f < nf4) {
            const float4 s4 = sS4[f];
            const float part = seg_sum<SEG>(dot4(s4, q4));
            if (c4 == 0) yrow[f / SEG] = fmaf(gamma, part, sry[f / SEG]);
            acc[ii] = scale4(gamma, s4);
          }
        }
        for (int j0 = 0; j0 <= n; j0 += 8) {
          float4 kk[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            kk[jj] = (j0 + jj <= n) ? reinterpret_cast<const float4*>(sK + (j0 + jj) * N)[c4]
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int ii = 0; ii < 8; ++ii) {
            const int f = f0 + ii * kThreads + t;
            if (f < nf4) {
              const int r = f / SEG;
#pragma unroll
              for (int jj = 0; jj < 8; ++jj)
                if (j0 + jj <= n) acc[ii] = axpy4(sX[(j0 + jj) * P + r], kk[jj], acc[ii]);
            }
          }
        }
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) {
          const int f = f0 + ii * kThreads + t;
          if (f < nf4) __stcs(gS4 + f, acc[ii]);
        }
      }
    }
    // append this token's record (non-flush steps; a flush empties the ring)
    if (!flush) {
      const int slot = ring_slot(head, n, C);
      for (int r = t; r < P; r += kThreads)
        d.r_x[(static_cast<size_t>(bh) * C + slot) * P + r] = in.x[static_cast<size_t>(bh) * P + r];
      if (t == 0) {
        d.r_dt[static_cast<size_t>(bh) * C + slot] = in.dt[bh];
        d.r_la[static_cast<size_t>(bh) * C + slot] = sla[n];
      }
      if (h % hpg == 0)
        for (int i = t; i < N; i += kThreads) d.r_B[(bg * C + slot) * N + i] = in.Bm[bg * N + i];
    }
  }

  __syncthreads();
  if (t == 0 && arrive_last(d.arrive, b, H)) {
    if (!ok) {
      report_error(d.err, DEVERR_CURSOR, b);
    } else if (flush) {
      d.cursor[4 * b] = ring_slot(head, n + 1, C);
      d.cursor[4 * b + 1] = 0;
      d.cursor[4 * b + 2] = 1;
    } else {
      d.cursor[4 * b + 1] = n + 1;
      d.cursor[4 * b + 2] = 0;
    }
  }
}

// ---------------------------------------------------------------------------
// Gated DeltaNet
// ---------------------------------------------------------------------------
template <int N>
__global__ void __launch_bounds__(kThreads) gdn_decode_kernel(const LayerDev d, const TokenIn in,
                                                              float* __restrict__ o) {
  constexpr int SEG = N / 4;
  extern __shared__ __align__(128) unsigned char smem[];

  const int P = d.P, H = d.H, G = d.G, C = d.C, L = d.L;
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh - b * H;
  const int hpg = H / G, g = h / hpg;  // g: key head
  const int t = threadIdx.x;
  const int tile = P * N;
  const size_t bg = static_cast<size_t>(b) * G + g;

  float* sS = reinterpret_cast<float*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sS + tile);
  float* sq = reinterpret_cast<float*>(bar + 2);  // [N]
  float* sK = sq + N;                             // [C][N] keys of records 0..n (n: current)
  float* sU = sK + C * N;                         // [C][P] u_j, then fold coefficients
  float* sv = sU + C * P;                         // [P]   current v
  float* sdk = sv + P;                            // [C]   k_j . k
  float* sdq = sdk + C;                           // [C]   k_j . q  (sdq[n] = k . q)
  float* sW = sdq + C;                            // [C]
  float* sla = sW + C;                            // [C]
  float* srk = sla + C;                           // [P]
  float* srq = srk + P;                           // [P]
  float* sc = srq + P;                            // [4]: gamma, a, beta

  float* gS = d.ckpt + static_cast<size_t>(bh) * tile;
  start_tile_copy(sS, gS, static_cast<uint32_t>(tile) * 4u, bar);

  const int head = d.cursor[4 * b], cnt = d.cursor[4 * b + 1];
  const bool ok = static_cast<unsigned>(head) < static_cast<unsigned>(C) &&
                  static_cast<unsigned>(cnt) < static_cast<unsigned>(L);
  const int n = ok ? cnt : 0;
  const bool flush = ok && (cnt + 1 == L);

  for (int i = t; i < N; i += kThreads) {
    sq[i] = bf(in.q[bg * N + i]);
    sK[n * N + i] = bf(in.k[bg * N + i]);
  }
  for (int r = t; r < P; r += kThreads) sv[r] = bf(in.v[static_cast<size_t>(bh) * P + r]);
  load_ring_keys<N>(sK, d.r_k + bg * C * N, head, n, C);
  if (t < n) sla[t] = d.r_g[static_cast<size_t>(bh) * C + ring_slot(head, t, C)];
  for (int i = t; i < n * P; i += kThreads) {
    const int j = i / P, r = i - j * P;
    sU[i] = d.r_u[(static_cast<size_t>(bh) * C + ring_slot(head, j, C)) * P + r];
  }
  __syncthreads();

  key_dots<N>(sdk, sK, sK + n * N, n);
  key_dots<N>(sdq, sK, sq, n + 1);
  if (t == 0) {
    float e = 0.f;
    for (int j = n - 1; j >= 0; --j) {
      sW[j] = expf(e);
      e += sla[j];
    }
    sc[0] = expf(e);
    sc[1] = expf(in.g[bh]);
    sc[2] = in.beta[bh];
  }
  __syncthreads();

  const float a = sc[1];
  for (int r = t; r < P; r += kThreads) {
    float ak = 0.f, aq = 0.f;
    for (int j = 0; j < n; ++j) {
      const float wu = sW[j] * sU[j * P + r];
      ak = fmaf(wu, sdk[j], ak);
      aq = fmaf(wu, sdq[j], aq);
      if (flush) sU[j * P + r] = a * wu;
    }
    srk[r] = ak;
    srq[r] = aq;
  }

  const bool tile_ok = finish_tile_copy(bar, d.err, b);
  const bool work = ok && tile_ok;
  const int slot = ring_slot(head, n, C);

  if (work) {
    const float gamma = sc[0], beta = sc[2], kq = sdq[n];
    const int c4 = t % SEG;
    const float4 q4 = reinterpret_cast<const float4*>(sq)[c4];
    const float4 k4 = reinterpret_cast<const float4*>(sK + n * N)[c4];
    const float4* sS4 = reinterpret_cast<const float4*>(sS);
    float* orow = o + static_cast<size_t>(bh) * P;
    float* urow = d.r_u + (static_cast<size_t>(bh) * C + slot) * P;
    const int nf4 = tile / 4;
    if (!flush) {
      for (int f = t; f < nf4; f += kThreads) {
        const float4 s4 = sS4[f];
        const float pk = seg_sum<SEG>(dot4(s4, k4));
        const float pq = seg_sum<SEG>(dot4(s4, q4));
        if (c4 == 0) {
          const int r = f / SEG;
          const float Sk = fmaf(gamma, pk, srk[r]);
          const float Sq = fmaf(gamma, pq, srq[r]);
          const float u = beta * (sv[r] - a * Sk);
          orow[r] = fmaf(a, Sq, u * kq);
          urow[r] = u;
        }
      }
    } else {
      const float ag = a * gamma;
      float4* gS4 = reinterpret_cast<float4*>(gS);
      for (int f0 = 0; f0 < nf4; f0 += 8 * kThreads) {
        float4 acc[8];
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) {
          const int f = f0 + ii * kThreads + t;
          if (f < nf4) {
            const float4 s4 = sS4[f];
            const float pk = seg_sum<SEG>(dot4(s4, k4));
            const float pq = seg_sum<SEG>(dot4(s4, q4));
            const int r = f / SEG;
            const float Sk = fmaf(gamma, pk, srk[r]);
            const float Sq = fmaf(gamma, pq, srq[r]);
            const float u = beta * (sv[r] - a * Sk);
            if (c4 == 0) orow[r] = fmaf(a, Sq, u * kq);
            acc[ii] = axpy4(u, k4, scale4(ag, s4));
          }
        }
        for (int j0 = 0; j0 < n; j0 += 8) {
          float4 kk[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            kk[jj] = (j0 + jj < n) ? reinterpret_cast<const float4*>(sK + (j0 + jj) * N)[c4]
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int ii = 0; ii < 8; ++ii) {
            const int f = f0 + ii * kThreads + t;
            if (f < nf4) {
              const int r = f / SEG;
#pragma unroll
              for (int jj = 0; jj < 8; ++jj)
                if (j0 + jj < n) acc[ii] = axpy4(sU[(j0 + jj) * P + r], kk[jj], acc[ii]);
            }
          }
        }
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) {
          const int f = f0 + ii * kThreads + t;
          if (f < nf4) __stcs(gS4 + f, acc[ii]);
        }
      }
    }
    if (!flush) {
      if (t == 0) d.r_g[static_cast<size_t>(bh) * C + slot] = in.g[bh];
      if (h % hpg == 0)
        for (int i = t; i < N; i += kThreads) d.r_k[(bg * C + slot) * N + i] = in.k[bg * N + i];
    }
  }

  __syncthreads();
  if (t == 0 && arrive_last(d.arrive, b, H)) {
    if (!ok) {
      report_error(d.err, DEVERR_CURSOR, b);
    } else if (flush) {
      d.cursor[4 * b] = ring_slot(head, n + 1, C);
      d.cursor[4 * b + 1] = 0;
      d.cursor[4 * b + 2] = 1;
    } else {
      d.cursor[4 * b + 1] = n + 1;
      d.cursor[4 * b + 2] = 0;
    }
  }
}

template <typename K>
cudaError_t launch_with_smem(K kernel, const LayerDev& d, const TokenIn& in, float* y, size_t smem,
                             cudaStream_t s) {
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  kernel<<<d.B * d.H, kThreads, smem, s>>>(d, in, y);
  return cudaGetLastError();
}

}  // namespace

size_t decode_smem_bytes(const LayerDev& d) {
  const size_t tile = static_cast<size_t>(d.P) * d.N * 4;
  size_t floats;
  if (d.kind == 0)
    floats = d.N + static_cast<size_t>(d.C) * d.N + static_cast<size_t>(d.C) * d.P + 4 * d.C + d.P + 4;
  else
    floats = d.N + static_cast<size_t>(d.C) * d.N + static_cast<size_t>(d.C) * d.P + d.P + 4 * d.C + 2 * d.P + 4;
  return tile + 16 + floats * 4;
}

cudaError_t launch_decode(const LayerDev& d, const TokenIn& in, float* y, cudaStream_t s) {
  const size_t smem = decode_smem_bytes(d);
  if (d.kind == 0) {
    switch (d.N) {
      case 16: return launch_with_smem(m2_decode_kernel<16>, d, in, y, smem, s);
      case 32: return launch_with_smem(m2_decode_kernel<32>, d, in, y, smem, s);
      case 64: return launch_with_smem(m2_decode_kernel<64>, d, in, y, smem, s);
      case 128: return launch_with_smem(m2_decode_kernel<128>, d, in, y, smem, s);
    }
  } else {
    switch (d.N) {
      case 16: return launch_with_smem(gdn_decode_kernel<16>, d, in, y, smem, s);
      case 32: return launch_with_smem(gdn_decode_kernel<32>, d, in, y, smem, s);
      case 64: return launch_with_smem(gdn_decode_kernel<64>, d, in, y, smem, s);
      case 128: return launch_with_smem(gdn_decode_kernel<128>, d, in, y, smem, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace rs
