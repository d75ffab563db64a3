// Commit (pointer advance) and explicit flush: fold buffered records into the
// checkpoint where the cursor says so, and advance the cursor.
//
// Commit: count += accepted[b]; a sequence whose count reaches L is folded
// over all its records in this launch and its cursor moves past them.
// Rejected drafts stay in their slots and are overwritten later ("ReplaySSM
// caches SSM inputs instead of state" (richland.au), "What shipped": the
// accepted prefix is committed by advancing a pointer; records past the
// pointer are ignored and overwritten).  Flush: fold whatever is buffered for
// the masked sequences.
//
// The fold of n records j = 0..n-1 is
//   S_new = gamma S_ckpt + sum_j w_j d_j k_j^T,  w_j = prod_{i>j} a_i,  gamma = prod_i a_i
// with d_j = dt_j x_j (Mamba-2) or the buffered delta u_j (Gated DeltaNet):
// one read and one write of the state matrix.
#include "common.cuh"
#include "readcopy.cuh"

namespace rs {
namespace {

__device__ __forceinline__ int ring_slot(int head, int j, int C) {
  int s = head + j;
  return s >= C ? s - C : s;
}

template <int KIND, int N, int READ>
__global__ void __launch_bounds__(kThreads) fold_kernel(const LayerDev d, const int mode,
                                                        const int* __restrict__ accepted,
                                                        const uint8_t* __restrict__ mask, const int T_pending) {
  constexpr int SEG = N / 4;
  extern __shared__ __align__(128) unsigned char smem[];

  const int P = d.P, H = d.H, G = d.G, C = d.C, L = d.L;
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh - b * H;
  const int g = h / (H / G);
  const int t = threadIdx.x;
  const int tile = P * N;
  const size_t bg = static_cast<size_t>(b) * G + g;

  float* sS = reinterpret_cast<float*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sS + tile);
  float* sK = reinterpret_cast<float*>(bar + 2);  // [C][N]
  float* sV = sK + C * N;                         // [C][P] d_j[r], then w_j d_j[r]
  float* sla = sV + C * P;                        // [C]
  float* sW = sla + C;                            // [C]
  float* sdt = sW + C;                            // [C]
  float* sc = sdt + C;                            // [1]
  float* sred = sc + 4;                           // [kThreads / 32] read-copy reduction

  const int head = d.cursor[4 * b], cnt = d.cursor[4 * b + 1];
  bool ok = static_cast<unsigned>(head) < static_cast<unsigned>(C) &&
            static_cast<unsigned>(cnt) < static_cast<unsigned>(L);
  int nacc = 0;
  bool acc_ok = true;
  if (mode == FOLD_COMMIT) {
    nacc = accepted[b];
    acc_ok = nacc >= 0 && nacc <= T_pending;
    ok = ok && cnt + T_pending <= C;
  }
  const int n_new = cnt + nacc;
  const bool fold = ok && acc_ok && (mode == FOLD_FLUSH ? (mask == nullptr || mask[b] != 0) : n_new >= L);
  const int n = fold ? n_new : 0;
  const bool need_tile = fold && (n > 0 || READ != READ_NONE);

  float* gS = d.ckpt + static_cast<size_t>(bh) * tile;
  if (need_tile && t == 0) {
    mbar_init(bar, 1);
    mbar_expect_tx(bar, static_cast<uint32_t>(tile) * 4u);
    bulk_g2s(sS, gS, static_cast<uint32_t>(tile) * 4u, bar);
  }

  if (n > 0) {
    const uint16_t* rk = (KIND == 0 ? d.r_B : d.r_k) + bg * C * N;
    for (int i = t; i < n * N; i += kThreads) {
      const int j = i / N, e = i - j * N;
      sK[i] = bf(rk[static_cast<size_t>(ring_slot(head, j, C)) * N + e]);
    }
    if (t < n) {
      const size_t s = static_cast<size_t>(bh) * d.Cp + ring_slot(head, t, C);
      if (KIND == 0) {
        sla[t] = d.r_la[s];
        sdt[t] = bf(d.r_dt[s]);
      } else {
        sla[t] = d.r_g[s];
      }
    }
    for (int i = t; i < n * P; i += kThreads) {
      const int j = i / P, r = i - j * P;
      const size_t s = (static_cast<size_t>(bh) * C + ring_slot(head, j, C)) * P + r;
      sV[i] = KIND == 0 ? bf(d.r_x[s]) : d.r_u[s];
    }
  }
  __syncthreads();
  if (t == 0) {
    float e = 0.f;
    for (int j = n - 1; j >= 0; --j) {
      sW[j] = expf(e);
      e += sla[j];
    }
    sc[0] = expf(e);
  }
  __syncthreads();
  for (int i = t; i < n * P; i += kThreads) {
    const int j = i / P;
    sV[i] = KIND == 0 ? sW[j] * (sdt[j] * sV[i]) : sW[j] * sV[i];
  }

  bool tile_ok = true;
  if (need_tile) {
    const bool arrived = __syncthreads_and(mbar_wait_bounded(bar, 0) ? 1 : 0) != 0;
    if (!arrived) {
      if (t == 0) report_error(d.err, DEVERR_TIMEOUT, b);
      mbar_wait_bounded(bar, 0);
      tile_ok = false;
    }
  } else {
    __syncthreads();
  }

  if (need_tile && tile_ok) {
    const float gamma = sc[0];
    const int c4 = t % SEG;
    const float4* sS4 = reinterpret_cast<const float4*>(sS);
    float4* gS4 = reinterpret_cast<float4*>(gS);
    float4* sOut4 = reinterpret_cast<float4*>(sS);  // folded tile, in place (read copy source)
    const int nf4 = tile / 4;
    for (int f0 = 0; f0 < nf4; f0 += 8 * kThreads) {
      float4 acc[8];
#pragma unroll
      for (int ii = 0; ii < 8; ++ii) {
        const int f = f0 + ii * kThreads + t;
        if (f < nf4) acc[ii] = n > 0 ? scale4(gamma, sS4[f]) : sS4[f];
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
              if (j0 + jj < n) acc[ii] = axpy4(sV[(j0 + jj) * P + r], kk[jj], acc[ii]);
          }
        }
      }
#pragma unroll
      for (int ii = 0; ii < 8; ++ii) {
        const int f = f0 + ii * kThreads + t;
        if (f < nf4) {
          if (n > 0) __stcs(gS4 + f, acc[ii]);
          if (READ != READ_NONE) sOut4[f] = acc[ii];
        }
      }
    }
    if (READ != READ_NONE) {
      __syncthreads();
      write_read_copy<N, READ>(d, bh, sS, sred);
    }
  }

  __syncthreads();
  if (t == 0 && arrive_last(d.arrive, b, H)) {
    if (!ok) {
      report_error(d.err, DEVERR_CURSOR, b);
    } else if (!acc_ok) {
      report_error(d.err, DEVERR_ACCEPTED, b);
    } else if (fold) {
      d.cursor[4 * b] = ring_slot(head, n, C);
      d.cursor[4 * b + 1] = 0;
      d.cursor[4 * b + 2] = 1;
    } else {
      d.cursor[4 * b + 1] = n_new;
      d.cursor[4 * b + 2] = 0;
    }
  }
}

template <int KIND, int N>
cudaError_t launch_n(const LayerDev& d, int mode, const int* accepted, const uint8_t* mask, int T_pending,
                     size_t smem, cudaStream_t s) {
  auto run = [&](auto kernel) -> cudaError_t {
    cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kernel), smem);
    if (e != cudaSuccess) return e;
    kernel<<<d.B * d.H, kThreads, smem, s>>>(d, mode, accepted, mask, T_pending);
    return cudaGetLastError();
  };
  if (KIND == 0 && d.read_mode == READ_FP8) return run(fold_kernel<KIND, N, READ_FP8>);
  if (KIND == 0 && d.read_mode == READ_NVFP4) return run(fold_kernel<KIND, N, READ_NVFP4>);
  return run(fold_kernel<KIND, N, READ_NONE>);
}

}  // namespace

cudaError_t launch_fold(const LayerDev& d, int mode, const int* accepted, const uint8_t* mask, int T_pending,
                        cudaStream_t s) {
  if (d.kind == RS_KDA) return mode == FOLD_FLUSH ? launch_kda_fold(d, mask, s) : cudaErrorInvalidValue;
  // d_state 128, d_head 64 or 128: the persistent kernel that skips non-folding sequences (fold128.cu)
  if (fold128_supports(d)) return launch_fold128(d, mode, accepted, mask, T_pending, s);
  const size_t smem = static_cast<size_t>(d.P) * d.N * 4 + 16 +
                      (static_cast<size_t>(d.C) * d.N + static_cast<size_t>(d.C) * d.P + 3 * d.C + 4 +
                       kThreads / 32) * 4;
  if (d.kind == 0) {
    switch (d.N) {
      case 16: return launch_n<0, 16>(d, mode, accepted, mask, T_pending, smem, s);
      case 32: return launch_n<0, 32>(d, mode, accepted, mask, T_pending, smem, s);
      case 64: return launch_n<0, 64>(d, mode, accepted, mask, T_pending, smem, s);
      case 128: return launch_n<0, 128>(d, mode, accepted, mask, T_pending, smem, s);
    }
  } else {
    switch (d.N) {
      case 16: return launch_n<1, 16>(d, mode, accepted, mask, T_pending, smem, s);
      case 32: return launch_n<1, 32>(d, mode, accepted, mask, T_pending, smem, s);
      case 64: return launch_n<1, 64>(d, mode, accepted, mask, T_pending, smem, s);
      case 128: return launch_n<1, 128>(d, mode, accepted, mask, T_pending, smem, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace rs
