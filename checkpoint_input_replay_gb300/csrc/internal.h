// Host/device shared descriptors of one cache, passed by value to every kernel.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <cuda.h>

#include "replayssm.h"

namespace rs {

constexpr int kThreads = 256;          // threads per CTA of every hot-path kernel
constexpr int kMaxRec = 32;            // L + T_max limit (records per sequence)
constexpr int kMaxTileBytes = 65536;   // P * N * 4 limit (one head's state, staged in smem)

enum DevErr : int { DEVERR_NONE = 0, DEVERR_ACCEPTED = 1, DEVERR_CURSOR = 2, DEVERR_TIMEOUT = 3 };
enum ReadMode : int { READ_NONE = 0, READ_FP8 = 1, READ_NVFP4 = 2 };
enum FoldMode : int { FOLD_COMMIT = 0, FOLD_FLUSH = 1 };

struct LayerDev {
  int kind, B, H, G, P, N, L, C, T_max, read_mode;
  int Cp;                      // ring row stride of the per-head scalars: C rounded up to 8
  int num_sms;                 // SMs of the device (persistent grid size)
  // debug (ordering check): a persistent launch's CTA c takes unit range
  // (c * cta_mult + 7) mod grid instead of c; 0 = off.  Launchers make it coprime
  // with the grid, so the map is a permutation.
  int cta_mult;
  // debug (comparison): the d_state-128 decode splits its units evenly instead of
  // by weight; 0 = off
  int uniform_split;
  float* ckpt;                 // [B][H][P][N]
  // Mamba-2 ring
  uint16_t* r_x;               // bf16 [B][H][C][P]
  uint16_t* r_dt;              // bf16 [B][H][Cp]
  float* r_la;                 // f32  [B][H][Cp]  log decay dt*A
  uint16_t* r_B;               // bf16 [B][G][C][N]
  // GDN ring (and the per-channel-gate layer's: g f32 [B][H][C][N] there)
  float* r_u;                  // f32  [B][H][C][P] delta u
  float* r_g;                  // f32  [B][H][Cp]   log decay g
  uint16_t* r_k;               // bf16 [B][G][C][N]
  // cursor and bookkeeping
  int* cursor;                 // [B][4] head, count, last_flush, 0
  int* err;                    // [4] code, sequence
  int* arrive;                 // [B]
  // read copy
  uint8_t* rc_codes;           // FP8: [B][H][P][N]; NVFP4: [B][H][P][N/2]
  float* rc_rowscale;          // FP8: [B][H][P]
  uint8_t* rc_blkscale;        // NVFP4: [B][H][P][N/16]
  float* rc_matscale;          // NVFP4: [B][H]
  // verify coefficient tables (scratch): f32 [B][H][verify_table_stride]
  float* vtab;
  // verify: the drafts' tree as an ancestor mask, bit 4 tau + sigma set when draft
  // sigma lies on the path from the committed records to draft tau (sigma = tau
  // included); chain-shaped drafts have every bit with sigma <= tau.  Set per call.
  uint32_t tree_anc;
};

struct TokenIn {
  const uint16_t *x, *dt, *Bm, *Cm;   // Mamba-2
  const float* A;
  const uint16_t *q, *k, *v;          // GDN
  const float *g, *beta;
};

// Launchers (one per kernel family); each returns the launch status.
cudaError_t launch_decode(const LayerDev& d, const TokenIn& in, float* y, cudaStream_t s);
cudaError_t launch_verify(const LayerDev& d, const TokenIn& in, int T, float* y, cudaStream_t s);
cudaError_t launch_fold(const LayerDev& d, int mode, const int* accepted, const uint8_t* mask,
                        int T_pending, cudaStream_t s);

// Host helpers of api.cu shared with other entry points.
rs_status bind_layer(const rs_config* cfg, const rs_buffers* bufs, bool needs_scratch, LayerDev* out);
rs_status bind_inputs(int kind, const rs_inputs* in, TokenIn* out);

// Raise a kernel's dynamic shared-memory limit (once per kernel and size).
cudaError_t set_smem_limit(const void* func, size_t bytes);

// Dynamic shared memory the decode kernel needs for this layer.
size_t decode_smem_bytes(const LayerDev& d);
// grouped decode kernel for d_state 128, d_head 64 or 128, when one stage and
// both group buffers fit in shared memory
bool decode128_supports(const LayerDev& d);
cudaError_t launch_decode128(const LayerDev& d, const TokenIn& in, float* y, cudaStream_t s);

// verify kernel on tcgen05 for d_state 128, d_head 64 or 128 (verify128.cu); it
// reads the checkpoint through a TMA tensor map made once per cache
bool verify128_supports(const LayerDev& d);
// commit / flush for d_state 128, d_head 64 or 128 (fold128.cu)
bool fold128_supports(const LayerDev& d);
cudaError_t launch_fold128(const LayerDev& d, int mode, const int* accepted, const uint8_t* mask, int T_pending,
                           cudaStream_t s);
int verify_table_stride(int kind, int C);
cudaError_t make_ckpt_tmap(const LayerDev& d, CUtensorMap* out);
cudaError_t launch_verify128(const LayerDev& d, const CUtensorMap& tmap, const TokenIn& in, int T, float* y,
                             cudaStream_t s);

// Per-channel-gate layers (kind 2): decode step and fold (kda.cu).
cudaError_t launch_kda_decode(const LayerDev& d, const TokenIn& in, float* y, cudaStream_t s);
cudaError_t launch_kda_fold(const LayerDev& d, const uint8_t* mask, cudaStream_t s);

// Tree speculative commit: move the records of each sequence's accepted path
// (drafts path[b][0..len) of the pending verify, whose parents are packed one
// byte each, parent + 1, in `parents`) to the slots right after the committed
// records, and write the accepted count the commit launch then applies (the
// path length, or -1 for a path that is not one, which that launch reports).
cudaError_t launch_tree_compact(const LayerDev& d, const int* path_len, const int* path, int path_stride,
                                int T_pending, uint32_t parents, int* accepted_out, cudaStream_t s);

// smallest m' >= m coprime with g (a CTA permutation multiplier); 0 stays 0
inline int coprime_mult(int m, int g) {
  if (m <= 0) return 0;
  auto gcd = [](int a, int b) {
    while (b) {
      const int t = a % b;
      a = b;
      b = t;
    }
    return a;
  };
  while (gcd(m, g) != 1) ++m;
  return m;
}

}  // namespace rs
