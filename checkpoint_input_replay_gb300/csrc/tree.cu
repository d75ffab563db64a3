// Tree-shaped speculative decoding: the records of an accepted path are moved
// next to the committed ones before the pointer advance.
//
// With drafts arranged as a tree (draft tau continues draft parent[tau]; -1 is
// the last committed record), the verify writes draft tau's record to slot
// head + count + tau like a chain, so the accepted path's records need not be
// contiguous in the buffer ("ReplaySSM：ハイブリッドモデルの高速デコーディングを
// 実現する状態ストレージ再考" (ai.warp-studio.com), "推測デコーディングにおける
// 革新と実装詳細", the sentence on tree-based speculative decoding).  The
// commit takes the accepted path as an index list: this kernel copies record
// path[i] to slot head + count + i (in place: every source is read before any
// destination is written), and hands the path length to the regular commit
// launch, which advances the pointer and folds when the buffer is full.  The
// records of a path depend only on the committed records and on the path's own
// earlier drafts, so the moved records (the Gated DeltaNet deltas included)
// are exactly the ones a chain of those drafts would have written.
#include "common.cuh"
#include "internal.h"

namespace rs {
namespace {

constexpr int kCompactThreads = 256;
constexpr int kMaxT = 4;

__device__ __forceinline__ int slot_of(int head, int j, int C) {
  const int s = head + j;
  return s >= C ? s - C : s;
}

// Copy element e of record path[i] to record i, for i < len, over `count`
// elements of one ring section; base(slot) gives the element's address.
template <typename TV, typename F>
__device__ __forceinline__ void move_section(int count, int len, const int* sp, int head, int n, int C, F base) {
  for (int e = threadIdx.x; e < count; e += kCompactThreads) {
    TV v[kMaxT];
#pragma unroll
    for (int i = 0; i < kMaxT; ++i)
      if (i < len) v[i] = *base(slot_of(head, n + sp[i], C), e);
#pragma unroll
    for (int i = 0; i < kMaxT; ++i)
      if (i < len && sp[i] != i) *base(slot_of(head, n + i, C), e) = v[i];
  }
}

__global__ void __launch_bounds__(kCompactThreads) tree_compact_kernel(const LayerDev d, const int* path_len,
                                                                       const int* path, const int stride,
                                                                       const int T, const uint32_t parents,
                                                                       int* accepted_out) {
  __shared__ int sp[kMaxT];
  __shared__ int smove;
  const int b = blockIdx.x;
  const int C = d.C, H = d.H, G = d.G, P = d.P, N = d.N, Cp = d.Cp;
  const int head = d.cursor[4 * b], n = d.cursor[4 * b + 1];
  if (threadIdx.x == 0) {
    const int len = path_len[b];
    bool ok = len >= 0 && len <= T && static_cast<unsigned>(head) < static_cast<unsigned>(C) && n >= 0 &&
              n + T <= C;
    int prev = -1;
    bool move = false;
    for (int i = 0; i < kMaxT; ++i) {
      if (!ok || i >= len) break;
      const int node = path[static_cast<size_t>(b) * stride + i];
      // a root-to-draft path: each node's parent is the previous node (the first's is -1)
      ok = node >= 0 && node < T && static_cast<int>((parents >> (8 * node)) & 0xFFu) - 1 == prev;
      prev = node;
      sp[i] = node;
      move = move || node != i;
    }
    accepted_out[b] = ok ? len : -1;
    smove = (ok && move) ? len : 0;
  }
  __syncthreads();
  const int len = smove;
  if (len == 0) return;
  const size_t bH = static_cast<size_t>(b) * H, bG = static_cast<size_t>(b) * G;
  // rows of a slot move 16 bytes at a time (P and N are multiples of 8, the ring's
  // sections 16-byte aligned)
  if (d.kind == RS_MAMBA2) {
    // x [B][H][C][P], dt and log a [B][H][Cp] per head, B [B][G][C][N] per group
    const int xv = P / 8, bv = N / 8;  // uint4 per row
    move_section<uint4>(H * xv, len, sp, head, n, C, [&](int slot, int e) {
      const int h = e / xv, c = e - h * xv;
      return reinterpret_cast<uint4*>(d.r_x + ((bH + h) * C + slot) * P) + c;
    });
    move_section<uint16_t>(H, len, sp, head, n, C, [&](int slot, int h) { return d.r_dt + (bH + h) * Cp + slot; });
    move_section<float>(H, len, sp, head, n, C, [&](int slot, int h) { return d.r_la + (bH + h) * Cp + slot; });
    move_section<uint4>(G * bv, len, sp, head, n, C, [&](int slot, int e) {
      const int g = e / bv, c = e - g * bv;
      return reinterpret_cast<uint4*>(d.r_B + ((bG + g) * C + slot) * N) + c;
    });
  } else {
    // u [B][H][C][P], g [B][H][Cp] per head, k [B][G][C][N] per group
    const int uv = P / 4, kv = N / 8;
    move_section<uint4>(H * uv, len, sp, head, n, C, [&](int slot, int e) {
      const int h = e / uv, c = e - h * uv;
      return reinterpret_cast<uint4*>(d.r_u + ((bH + h) * C + slot) * P) + c;
    });
    move_section<float>(H, len, sp, head, n, C, [&](int slot, int h) { return d.r_g + (bH + h) * Cp + slot; });
    move_section<uint4>(G * kv, len, sp, head, n, C, [&](int slot, int e) {
      const int g = e / kv, c = e - g * kv;
      return reinterpret_cast<uint4*>(d.r_k + ((bG + g) * C + slot) * N) + c;
    });
  }
}

}  // namespace

cudaError_t launch_tree_compact(const LayerDev& d, const int* path_len, const int* path, int path_stride,
                                int T_pending, uint32_t parents, int* accepted_out, cudaStream_t s) {
  if (T_pending < 1 || T_pending > kMaxT) return cudaErrorInvalidValue;
  tree_compact_kernel<<<d.B, kCompactThreads, 0, s>>>(d, path_len, path, path_stride, T_pending, parents,
                                                      accepted_out);
  return cudaGetLastError();
}

}  // namespace rs
