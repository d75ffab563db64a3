// The conventional SSM decode path on the same GPU, for comparison with the
// checkpoint-plus-ring path: a read-modify-write decode step that reads the
// whole recurrent state, applies the rank-1 update and writes the state back
// on every token, and a speculative path that keeps a state snapshot after
// every draft token (one state read and T snapshot writes per verify) and
// rolls back by selecting a snapshot ("ReplaySSM caches SSM inputs instead of
// state" (richland.au), "What shipped": the paragraph on why the conventional
// kernel is bandwidth-bound -- it loads the full state, applies a rank-1
// update and stores it back every token -- and the paragraph on the snapshot
// stored after every draft token; ai-jitan-hub.com, "何がどれだけ速くなったのか",
// items 1 and 2).
//
// Both are plain streaming kernels: one CTA of 256 threads per (sequence,
// head) state matrix, a lane holds four consecutive columns of a row, every
// thread keeps eight rows' 16-byte loads in flight, the row dot products are
// warp reductions, and the state never leaves registers between its load and
// its store(s).  Loads and stores are streaming (evict-first): each state
// byte is touched once per launch.
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace rs {
namespace {

constexpr int kConvThreads = 256;
constexpr int kPasses = 8;  // row passes per warp batch = 16-byte loads a thread keeps in flight

// Per-lane totals of the row each lane works on, for each of the 8 passes
// (a row spans N/4 lanes; N = 128: one row per pass, totals by transpose-reduce).
template <int N>
__device__ __forceinline__ void row_totals(const float part[kPasses], int lane, float tot[kPasses]) {
  if constexpr (N == 128) {
    const float z = reduce8(part, lane);  // lane 4k holds the total of pass k
#pragma unroll
    for (int k = 0; k < kPasses; ++k) tot[k] = __shfl_sync(0xffffffffu, z, 4 * k);
  } else {
#pragma unroll
    for (int k = 0; k < kPasses; ++k) tot[k] = seg_sum<N / 4>(part[k]);
  }
}

struct ConvShape {
  int B, H, G, P;
};

// One conventional decode token for every (sequence, head): S <- update(S), y = S q.
//   Mamba-2: S_t = a S_{t-1} + v k^T, a = exp(dt A_h), v = dt x, k = B, q = C
//   GDN:     S_t = a S_{t-1} + u k^T, u = b (v - a S_{t-1} k), a = exp(g)
//            (= a S_{t-1} (I - b k k^T) + b v k^T), o = S_t q = a S_{t-1} q + u (k . q)
template <int KIND, int N>
__global__ void __launch_bounds__(kConvThreads) conv_decode_kernel(const ConvShape sh, float* __restrict__ state,
                                                                    const TokenIn in, float* __restrict__ y) {
  constexpr int SEG = N / 4, RPP = 32 / SEG, ROWS = kPasses * RPP;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = lane % SEG, rsub = lane / SEG;
  const size_t u = blockIdx.x;
  const int b = static_cast<int>(u / sh.H), h = static_cast<int>(u % sh.H);
  const int g = h / (sh.H / sh.G);
  const size_t bg = static_cast<size_t>(b) * sh.G + g;
  const int P = sh.P;
  float4* S4 = reinterpret_cast<float4*>(state + u * static_cast<size_t>(P) * N);
  float a, scal;  // Mamba-2: a, dt; GDN: a, beta
  float4 k4, q4;
  if (KIND == 0) {
    const float dt = bf(in.dt[u]);
    a = expf(dt * in.A[h]);
    scal = dt;
    k4 = bf4(reinterpret_cast<const uint2*>(in.Bm + bg * N)[c]);
    q4 = bf4(reinterpret_cast<const uint2*>(in.Cm + bg * N)[c]);
  } else {
    a = expf(in.g[u]);
    scal = in.beta[u];
    k4 = bf4(reinterpret_cast<const uint2*>(in.k + bg * N)[c]);
    q4 = bf4(reinterpret_cast<const uint2*>(in.q + bg * N)[c]);
  }
  const float kq = KIND == 1 ? seg_sum<SEG>(dot4(k4, q4)) : 0.f;
  for (int base = warp * ROWS; base < P; base += (kConvThreads / 32) * ROWS) {
    float4 s[kPasses];
    float xr[kPasses];
#pragma unroll
    for (int k = 0; k < kPasses; ++k) {
      const int row = base + k * RPP + rsub;
      const bool valid = row < P;
      s[k] = valid ? __ldcs(S4 + static_cast<size_t>(row) * SEG + c) : make_float4(0.f, 0.f, 0.f, 0.f);
      xr[k] = valid ? bf(KIND == 0 ? in.x[u * P + row] : in.v[u * P + row]) : 0.f;
    }
    if (KIND == 0) {
      float part[kPasses], tot[kPasses];
#pragma unroll
      for (int k = 0; k < kPasses; ++k) {
        s[k] = axpy4(scal * xr[k], k4, scale4(a, s[k]));  // a S + (dt x) k^T
        part[k] = dot4(s[k], q4);
      }
      row_totals<N>(part, lane, tot);
#pragma unroll
      for (int k = 0; k < kPasses; ++k) {
        const int row = base + k * RPP + rsub;
        if (row < P) {
          __stcs(S4 + static_cast<size_t>(row) * SEG + c, s[k]);
          if (c == 0) y[u * P + row] = tot[k];
        }
      }
    } else {
      float pk[kPasses], pq[kPasses], Sk[kPasses], Sq[kPasses];
#pragma unroll
      for (int k = 0; k < kPasses; ++k) {
        pk[k] = dot4(s[k], k4);
        pq[k] = dot4(s[k], q4);
      }
      row_totals<N>(pk, lane, Sk);
      row_totals<N>(pq, lane, Sq);
#pragma unroll
      for (int k = 0; k < kPasses; ++k) {
        const int row = base + k * RPP + rsub;
        const float ud = scal * (xr[k] - a * Sk[k]);  // u = b (v - a S k)
        if (row < P) {
          __stcs(S4 + static_cast<size_t>(row) * SEG + c, axpy4(ud, k4, scale4(a, s[k])));
          if (c == 0) y[u * P + row] = fmaf(a, Sq[k], ud * kq);
        }
      }
    }
  }
}

// Snapshot-per-draft speculative verify: per (sequence, head), read the current
// state (slot cur of the sequence's T_max + 1 slots) once, run the T drafts
// token by token in registers, write the state after draft tau to slot
// (cur + 1 + tau) mod (T_max + 1) and emit every draft's output.
template <int KIND, int N>
__global__ void __launch_bounds__(kConvThreads) snapshot_verify_kernel(const ConvShape sh, const int n_slots,
                                                                        float* __restrict__ pool,
                                                                        const int* __restrict__ slots, int* err,
                                                                        const TokenIn in, const int T,
                                                                        float* __restrict__ y) {
  constexpr int SEG = N / 4, RPP = 32 / SEG, ROWS = kPasses * RPP;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = lane % SEG, rsub = lane / SEG;
  const int H = sh.H, G = sh.G, P = sh.P;
  const int b = static_cast<int>(blockIdx.x / H), h = static_cast<int>(blockIdx.x % H);
  const int g = h / (H / G);
  const size_t tile = static_cast<size_t>(P) * N;
  const int cur = slots[b];
  if (cur < 0 || cur >= n_slots) {
    if (threadIdx.x == 0 && h == 0) report_error(err, DEVERR_CURSOR, b);
    return;
  }
  auto slot_ptr = [&](int s) {
    return reinterpret_cast<float4*>(pool + ((static_cast<size_t>(b) * n_slots + s) * H + h) * tile);
  };
  const float4* src = slot_ptr(cur);
  for (int base = warp * ROWS; base < P; base += (kConvThreads / 32) * ROWS) {
    float4 s[kPasses];
#pragma unroll
    for (int k = 0; k < kPasses; ++k) {
      const int row = base + k * RPP + rsub;
      s[k] = row < P ? __ldcs(src + static_cast<size_t>(row) * SEG + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int tau = 0; tau < T; ++tau) {
      const size_t bt = static_cast<size_t>(b) * T + tau;
      const size_t ut = bt * H + h;     // per-head input index of draft tau
      const size_t gt = bt * G + g;     // per-group input index
      float a, scal;
      float4 k4, q4;
      if (KIND == 0) {
        const float dt = bf(in.dt[ut]);
        a = expf(dt * in.A[h]);
        scal = dt;
        k4 = bf4(reinterpret_cast<const uint2*>(in.Bm + gt * N)[c]);
        q4 = bf4(reinterpret_cast<const uint2*>(in.Cm + gt * N)[c]);
      } else {
        a = expf(in.g[ut]);
        scal = in.beta[ut];
        k4 = bf4(reinterpret_cast<const uint2*>(in.k + gt * N)[c]);
        q4 = bf4(reinterpret_cast<const uint2*>(in.q + gt * N)[c]);
      }
      float xr[kPasses];
#pragma unroll
      for (int k = 0; k < kPasses; ++k) {
        const int row = base + k * RPP + rsub;
        xr[k] = row < P ? bf(KIND == 0 ? in.x[ut * P + row] : in.v[ut * P + row]) : 0.f;
      }
      float tot[kPasses];
      if (KIND == 0) {
        float part[kPasses];
#pragma unroll
        for (int k = 0; k < kPasses; ++k) {
          s[k] = axpy4(scal * xr[k], k4, scale4(a, s[k]));
          part[k] = dot4(s[k], q4);
        }
        row_totals<N>(part, lane, tot);
      } else {
        const float kq = seg_sum<SEG>(dot4(k4, q4));
        float pk[kPasses], pq[kPasses], Sk[kPasses], Sq[kPasses];
#pragma unroll
        for (int k = 0; k < kPasses; ++k) {
          pk[k] = dot4(s[k], k4);
          pq[k] = dot4(s[k], q4);
        }
        row_totals<N>(pk, lane, Sk);
        row_totals<N>(pq, lane, Sq);
#pragma unroll
        for (int k = 0; k < kPasses; ++k) {
          const float ud = scal * (xr[k] - a * Sk[k]);
          s[k] = axpy4(ud, k4, scale4(a, s[k]));
          tot[k] = fmaf(a, Sq[k], ud * kq);
        }
      }
      float4* dst = slot_ptr((cur + 1 + tau) % n_slots);
#pragma unroll
      for (int k = 0; k < kPasses; ++k) {
        const int row = base + k * RPP + rsub;
        if (row < P) {
          __stcs(dst + static_cast<size_t>(row) * SEG + c, s[k]);
          if (c == 0) y[ut * P + row] = tot[k];
        }
      }
    }
  }
}

// Rollback by snapshot select: the state after the accepted prefix is the
// snapshot of draft n - 1 (n = 0: the state before the drafts).
__global__ void snapshot_commit_kernel(int B, int n_slots, int T, int* __restrict__ slots,
                                       const int* __restrict__ accepted, int* err) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int n = accepted[b], cur = slots[b];
  if (n < 0 || n > T) {
    report_error(err, DEVERR_ACCEPTED, b);
    return;
  }
  if (cur < 0 || cur >= n_slots) {
    report_error(err, DEVERR_CURSOR, b);
    return;
  }
  slots[b] = (cur + n) % n_slots;
}

template <int KIND>
cudaError_t launch_conv_k(const ConvShape& sh, int N, float* state, const TokenIn& in, float* y, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>(sh.B) * sh.H;
  switch (N) {
    case 16: conv_decode_kernel<KIND, 16><<<grid, kConvThreads, 0, s>>>(sh, state, in, y); break;
    case 32: conv_decode_kernel<KIND, 32><<<grid, kConvThreads, 0, s>>>(sh, state, in, y); break;
    case 64: conv_decode_kernel<KIND, 64><<<grid, kConvThreads, 0, s>>>(sh, state, in, y); break;
    default: conv_decode_kernel<KIND, 128><<<grid, kConvThreads, 0, s>>>(sh, state, in, y); break;
  }
  return cudaGetLastError();
}

template <int KIND>
cudaError_t launch_snap_k(const ConvShape& sh, int N, int n_slots, float* pool, const int* slots, int* err,
                          const TokenIn& in, int T, float* y, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>(sh.B) * sh.H;
  switch (N) {
    case 16: snapshot_verify_kernel<KIND, 16><<<grid, kConvThreads, 0, s>>>(sh, n_slots, pool, slots, err, in, T, y); break;
    case 32: snapshot_verify_kernel<KIND, 32><<<grid, kConvThreads, 0, s>>>(sh, n_slots, pool, slots, err, in, T, y); break;
    case 64: snapshot_verify_kernel<KIND, 64><<<grid, kConvThreads, 0, s>>>(sh, n_slots, pool, slots, err, in, T, y); break;
    default: snapshot_verify_kernel<KIND, 128><<<grid, kConvThreads, 0, s>>>(sh, n_slots, pool, slots, err, in, T, y); break;
  }
  return cudaGetLastError();
}

bool pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The shapes the conventional kernels serve (no ring, no read copy).
rs_status validate_conv(const rs_config* c, bool snapshot) {
  if (!c) return RS_ERR_NULL;
  if (c->kind != RS_MAMBA2 && c->kind != RS_GDN) return RS_ERR_RANGE;
  if (c->read_mode != RS_READ_NONE) return RS_ERR_UNSUPPORTED;
  if (c->batch < 1 || c->n_heads < 1 || c->n_groups < 1 || c->n_heads % c->n_groups != 0) return RS_ERR_SHAPE;
  if (static_cast<long long>(c->batch) * c->n_heads > (1LL << 31) - 1) return RS_ERR_SHAPE;
  if (!pow2_in(c->d_state, 16, 128) || !pow2_in(c->d_head, 16, 128)) return RS_ERR_UNSUPPORTED;
  if (snapshot && (c->max_draft < 1 || c->max_draft > 4)) return RS_ERR_RANGE;
  return RS_OK;
}

ConvShape shape_of(const rs_config* c) { return ConvShape{c->batch, c->n_heads, c->n_groups, c->d_head}; }

}  // namespace
}  // namespace rs

extern "C" {

rs_status rs_conventional_decode_step(const rs_config* cfg, float* state, const rs_inputs* in, float* y,
                                      rs_stream stream) {
  rs_status st = rs::validate_conv(cfg, false);
  if (st != RS_OK) return st;
  if (!state || !y) return RS_ERR_NULL;
  if (!rs::al16(state) || !rs::al16(y)) return RS_ERR_ALIGN;
  rs::TokenIn tok{};
  st = rs::bind_inputs(cfg->kind, in, &tok);
  if (st != RS_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const rs::ConvShape sh = rs::shape_of(cfg);
  const cudaError_t e = cfg->kind == RS_MAMBA2 ? rs::launch_conv_k<0>(sh, cfg->d_state, state, tok, y, s)
                                               : rs::launch_conv_k<1>(sh, cfg->d_state, state, tok, y, s);
  return e == cudaSuccess ? RS_OK : RS_ERR_CUDA;
}

rs_status rs_snapshot_query_sizes(const rs_config* cfg, size_t bytes[2]) {
  if (!bytes) return RS_ERR_NULL;
  const rs_status st = rs::validate_conv(cfg, true);
  if (st != RS_OK) return st;
  const size_t n_slots = static_cast<size_t>(cfg->max_draft) + 1;
  bytes[0] = static_cast<size_t>(cfg->batch) * n_slots * cfg->n_heads * cfg->d_head * cfg->d_state * 4;
  bytes[1] = static_cast<size_t>(cfg->batch) * 4 + 16;
  return RS_OK;
}

rs_status rs_snapshot_verify(const rs_config* cfg, float* pool, const int32_t* slots, int32_t T,
                             const rs_inputs* drafts, float* y, rs_stream stream) {
  rs_status st = rs::validate_conv(cfg, true);
  if (st != RS_OK) return st;
  if (!pool || !slots || !y) return RS_ERR_NULL;
  if (T < 1 || T > cfg->max_draft) return RS_ERR_RANGE;
  if (!rs::al16(pool) || !rs::al16(slots) || !rs::al16(y)) return RS_ERR_ALIGN;
  rs::TokenIn tok{};
  st = rs::bind_inputs(cfg->kind, drafts, &tok);
  if (st != RS_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const rs::ConvShape sh = rs::shape_of(cfg);
  int* err = const_cast<int*>(slots) + cfg->batch;
  const int n_slots = cfg->max_draft + 1;
  const cudaError_t e =
      cfg->kind == RS_MAMBA2 ? rs::launch_snap_k<0>(sh, cfg->d_state, n_slots, pool, slots, err, tok, T, y, s)
                             : rs::launch_snap_k<1>(sh, cfg->d_state, n_slots, pool, slots, err, tok, T, y, s);
  return e == cudaSuccess ? RS_OK : RS_ERR_CUDA;
}

rs_status rs_snapshot_commit(const rs_config* cfg, int32_t* slots, const int32_t* accepted, int32_t T,
                             rs_stream stream) {
  const rs_status st = rs::validate_conv(cfg, true);
  if (st != RS_OK) return st;
  if (!slots || !accepted) return RS_ERR_NULL;
  if (T < 1 || T > cfg->max_draft) return RS_ERR_RANGE;
  if (!rs::al16(slots) || !rs::al16(accepted)) return RS_ERR_ALIGN;
  const int threads = 256, blocks = (cfg->batch + threads - 1) / threads;
  rs::snapshot_commit_kernel<<<blocks, threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      cfg->batch, cfg->max_draft + 1, T, slots, accepted, slots + cfg->batch);
  return cudaGetLastError() == cudaSuccess ? RS_OK : RS_ERR_CUDA;
}

}  // extern "C"
