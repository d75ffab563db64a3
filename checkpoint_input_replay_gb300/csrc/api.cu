// Host side of the C ABI declared in include/replayssm.h: argument
// validation, the buffer layout, call-order rules and kernel launches.
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <new>

#include "internal.h"
#include "replayssm.h"

struct rs_cache {
  CUtensorMap ckpt_map;  // the checkpoint as a TMA tensor (when the tcgen05 verify kernel serves the shape)
  rs_config cfg;
  rs::LayerDev dev;
  int pending;    // drafts appended by the last rs_verify and not yet committed
  uint32_t pending_parents;  // their tree: parent + 1 of draft tau in byte tau
  bool pending_chain;        // the pending drafts form a chain (a prefix commit applies)
  bool map_ok;
};

namespace {

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool is_pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Layout {
  size_t ckpt, ring, cursor, read_copy, scratch;
  size_t s1;  // scratch: offset of the verify coefficient tables (0 when there are none)
  // ring section offsets (bytes)
  size_t r0, r1, r2, r3;
  // read-copy section offsets
  size_t c0, c1, c2;
};

size_t decode_smem(const rs_config& c) {
  rs::LayerDev d{};
  d.kind = c.kind;
  d.P = c.d_head;
  d.N = c.d_state;
  d.C = c.ring_len + c.max_draft;
  return rs::decode_smem_bytes(d);
}

rs_status validate(const rs_config* c) {
  if (!c) return RS_ERR_NULL;
  if (c->kind != RS_MAMBA2 && c->kind != RS_GDN && c->kind != RS_KDA) return RS_ERR_RANGE;
  if (c->read_mode < RS_READ_NONE || c->read_mode > RS_READ_NVFP4) return RS_ERR_RANGE;
  if (c->batch < 1 || c->n_heads < 1 || c->n_groups < 1 || c->d_head < 1 || c->d_state < 1 ||
      c->ring_len < 1 || c->max_draft < 0)
    return RS_ERR_SHAPE;
  if (c->n_heads % c->n_groups != 0) return RS_ERR_SHAPE;
  if (static_cast<long long>(c->batch) * c->n_heads > (1LL << 31) - 1) return RS_ERR_SHAPE;
  if (!is_pow2_in(c->d_state, 16, 128) || !is_pow2_in(c->d_head, 16, 128)) return RS_ERR_UNSUPPORTED;
  if (static_cast<long long>(c->d_head) * c->d_state * 4 > rs::kMaxTileBytes) return RS_ERR_UNSUPPORTED;
  if (c->ring_len + c->max_draft > rs::kMaxRec || c->max_draft > 4) return RS_ERR_UNSUPPORTED;
  if (c->read_mode != RS_READ_NONE && c->kind != RS_MAMBA2) return RS_ERR_UNSUPPORTED;
  // the per-channel-gate layer is decoded and flushed; no speculative path
  if (c->kind == RS_KDA && c->max_draft != 0) return RS_ERR_UNSUPPORTED;
  if (decode_smem(*c) > 227 * 1024) return RS_ERR_UNSUPPORTED;
  return RS_OK;
}

Layout layout_of(const rs_config& c) {
  Layout L{};
  const size_t B = c.batch, H = c.n_heads, G = c.n_groups, P = c.d_head, N = c.d_state;
  const size_t C = static_cast<size_t>(c.ring_len) + c.max_draft;
  const size_t Cp = (C + 7) & ~static_cast<size_t>(7);
  L.ckpt = B * H * P * N * 4;
  if (c.kind == RS_MAMBA2) {
    L.r0 = 0;                                   // x  bf16 [B][H][C][P]
    L.r1 = L.r0 + align256(B * H * C * P * 2);  // dt bf16 [B][H][Cp]
    L.r2 = L.r1 + align256(B * H * Cp * 2);     // la f32  [B][H][Cp]
    L.r3 = L.r2 + align256(B * H * Cp * 4);     // B  bf16 [B][G][C][N]
    L.ring = L.r3 + align256(B * G * C * N * 2);
  } else if (c.kind == RS_GDN) {
    L.r0 = 0;                                   // u f32  [B][H][C][P]
    L.r1 = L.r0 + align256(B * H * C * P * 4);  // g f32  [B][H][Cp]
    L.r2 = L.r1 + align256(B * H * Cp * 4);     // k bf16 [B][G][C][N]
    L.r3 = L.r2;
    L.ring = L.r2 + align256(B * G * C * N * 2);
  } else {
    L.r0 = 0;                                   // u f32  [B][H][C][P]
    L.r1 = L.r0 + align256(B * H * C * P * 4);  // g f32  [B][H][C][N] (a log decay per key channel)
    L.r2 = L.r1 + align256(B * H * C * N * 4);  // k bf16 [B][G][C][N]
    L.r3 = L.r2;
    L.ring = L.r2 + align256(B * G * C * N * 2);
  }
  L.cursor = B * 16 + 16;
  if (c.read_mode == RS_READ_FP8_ROW) {
    L.c0 = 0;
    L.c1 = align256(B * H * P * N);             // row scales f32 [B][H][P]
    L.read_copy = L.c1 + align256(B * H * P * 4);
  } else if (c.read_mode == RS_READ_NVFP4) {
    L.c0 = 0;
    L.c1 = align256(B * H * P * N / 2);         // block scales u8 [B][H][P][N/16]
    L.c2 = L.c1 + align256(B * H * P * (N / 16));  // matrix scales f32 [B][H]
    L.read_copy = L.c2 + align256(B * H * 4);
  }
  L.scratch = B * 4;
  if (c.max_draft > 0) {
    // per-head coefficient tables of the tensor-core verify kernel
    L.s1 = align256(B * 4);
    L.scratch = L.s1 + B * H * static_cast<size_t>(rs::verify_table_stride(c.kind, static_cast<int>(C))) * 4;
  }
  return L;
}

rs_status from_cuda(cudaError_t e) { return e == cudaSuccess ? RS_OK : RS_ERR_CUDA; }

rs_status check_inputs(const rs_cache* h, const rs_inputs* in) {
  if (!in) return RS_ERR_NULL;
  const void* p[5];
  if (h->cfg.kind == RS_MAMBA2) {
    p[0] = in->x; p[1] = in->dt; p[2] = in->A; p[3] = in->Bm; p[4] = in->Cm;
  } else {
    p[0] = in->q; p[1] = in->k; p[2] = in->v; p[3] = in->g; p[4] = in->beta;
  }
  for (const void* q : p)
    if (!q) return RS_ERR_NULL;
  for (const void* q : p)
    if (!aligned16(q)) return RS_ERR_ALIGN;
  return RS_OK;
}

rs::TokenIn token_in(const rs_inputs* in) {
  rs::TokenIn t{};
  t.x = static_cast<const uint16_t*>(in->x);
  t.dt = static_cast<const uint16_t*>(in->dt);
  t.A = in->A;
  t.Bm = static_cast<const uint16_t*>(in->Bm);
  t.Cm = static_cast<const uint16_t*>(in->Cm);
  t.q = static_cast<const uint16_t*>(in->q);
  t.k = static_cast<const uint16_t*>(in->k);
  t.v = static_cast<const uint16_t*>(in->v);
  t.g = in->g;
  t.beta = in->beta;
  return t;
}

}  // namespace

namespace rs {

cudaError_t set_smem_limit(const void* func, size_t bytes) {
  // cudaFuncSetAttribute once per kernel and size: launches stay a plain <<<>>>.
  static std::mutex mu;
  static const void* keys[256];
  static size_t sizes[256];
  static int used = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (keys[i] == func && sizes[i] >= bytes) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  for (int i = 0; i < used; ++i)
    if (keys[i] == func) {
      sizes[i] = bytes;
      return cudaSuccess;
    }
  if (used < 256) {
    keys[used] = func;
    sizes[used] = bytes;
    ++used;
  }
  return cudaSuccess;
}

// Layer descriptor for caller buffers, validated like rs_create_cache but
// without a handle and without touching device memory.  The arrival counters
// are left unset when needs_scratch is false (the caller supplies them).
rs_status bind_layer(const rs_config* cfg, const rs_buffers* bufs, bool needs_scratch, LayerDev* out) {
  if (!cfg || !bufs || !out) return RS_ERR_NULL;
  const rs_status st = validate(cfg);
  if (st != RS_OK) return st;
  if (!bufs->ckpt || !bufs->ring || !bufs->cursor || (needs_scratch && !bufs->scratch)) return RS_ERR_NULL;
  if (cfg->read_mode != RS_READ_NONE && !bufs->read_copy) return RS_ERR_NULL;
  if (!aligned16(bufs->ckpt) || !aligned16(bufs->ring) || !aligned16(bufs->cursor) ||
      (needs_scratch && !aligned16(bufs->scratch)) || (bufs->read_copy && !aligned16(bufs->read_copy)))
    return RS_ERR_ALIGN;
  const Layout L = layout_of(*cfg);
  LayerDev d{};
  d.kind = cfg->kind;
  d.B = cfg->batch;
  d.H = cfg->n_heads;
  d.G = cfg->n_groups;
  d.P = cfg->d_head;
  d.N = cfg->d_state;
  d.L = cfg->ring_len;
  d.T_max = cfg->max_draft;
  d.C = cfg->ring_len + cfg->max_draft;
  d.Cp = (d.C + 7) & ~7;
  d.read_mode = cfg->read_mode;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return RS_ERR_CUDA;
  d.num_sms = sms;
  d.ckpt = static_cast<float*>(bufs->ckpt);
  char* ring = static_cast<char*>(bufs->ring);
  if (cfg->kind == RS_MAMBA2) {
    d.r_x = reinterpret_cast<uint16_t*>(ring + L.r0);
    d.r_dt = reinterpret_cast<uint16_t*>(ring + L.r1);
    d.r_la = reinterpret_cast<float*>(ring + L.r2);
    d.r_B = reinterpret_cast<uint16_t*>(ring + L.r3);
  } else {
    d.r_u = reinterpret_cast<float*>(ring + L.r0);
    d.r_g = reinterpret_cast<float*>(ring + L.r1);
    d.r_k = reinterpret_cast<uint16_t*>(ring + L.r2);
  }
  d.cursor = static_cast<int*>(bufs->cursor);
  d.err = d.cursor + 4 * d.B;
  d.arrive = needs_scratch ? static_cast<int*>(bufs->scratch) : nullptr;
  if (cfg->read_mode != RS_READ_NONE) {
    char* rc = static_cast<char*>(bufs->read_copy);
    d.rc_codes = reinterpret_cast<uint8_t*>(rc + L.c0);
    if (cfg->read_mode == RS_READ_FP8_ROW) {
      d.rc_rowscale = reinterpret_cast<float*>(rc + L.c1);
    } else {
      d.rc_blkscale = reinterpret_cast<uint8_t*>(rc + L.c1);
      d.rc_matscale = reinterpret_cast<float*>(rc + L.c2);
    }
  }
  *out = d;
  return RS_OK;
}

// Token inputs of one call, checked for the layer kind (NULL / alignment).
rs_status bind_inputs(int kind, const rs_inputs* in, TokenIn* out) {
  if (!in || !out) return RS_ERR_NULL;
  const void* p[5];
  if (kind == RS_MAMBA2) {
    p[0] = in->x; p[1] = in->dt; p[2] = in->A; p[3] = in->Bm; p[4] = in->Cm;
  } else {
    p[0] = in->q; p[1] = in->k; p[2] = in->v; p[3] = in->g; p[4] = in->beta;
  }
  for (const void* q : p)
    if (!q) return RS_ERR_NULL;
  for (const void* q : p)
    if (!aligned16(q)) return RS_ERR_ALIGN;
  *out = token_in(in);
  return RS_OK;
}

}  // namespace rs

extern "C" {

rs_status rs_query_sizes(const rs_config* cfg, size_t bytes[5]) {
  if (!cfg || !bytes) return RS_ERR_NULL;
  const rs_status st = validate(cfg);
  if (st != RS_OK) return st;
  const Layout L = layout_of(*cfg);
  bytes[0] = L.ckpt;
  bytes[1] = L.ring;
  bytes[2] = L.cursor;
  bytes[3] = L.read_copy;
  bytes[4] = L.scratch;
  return RS_OK;
}

rs_status rs_create_cache(const rs_config* cfg, const rs_buffers* bufs, rs_cache** out) {
  if (!cfg || !bufs || !out) return RS_ERR_NULL;
  const rs_status st = validate(cfg);
  if (st != RS_OK) return st;
  if (!bufs->ckpt || !bufs->ring || !bufs->cursor || !bufs->scratch) return RS_ERR_NULL;
  if (cfg->read_mode != RS_READ_NONE && !bufs->read_copy) return RS_ERR_NULL;
  if (!aligned16(bufs->ckpt) || !aligned16(bufs->ring) || !aligned16(bufs->cursor) ||
      !aligned16(bufs->scratch) || (bufs->read_copy && !aligned16(bufs->read_copy)))
    return RS_ERR_ALIGN;

  const Layout L = layout_of(*cfg);
  rs::LayerDev d{};
  d.kind = cfg->kind;
  d.B = cfg->batch;
  d.H = cfg->n_heads;
  d.G = cfg->n_groups;
  d.P = cfg->d_head;
  d.N = cfg->d_state;
  d.L = cfg->ring_len;
  d.T_max = cfg->max_draft;
  d.C = cfg->ring_len + cfg->max_draft;
  d.Cp = (d.C + 7) & ~7;
  d.read_mode = cfg->read_mode;
  {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return RS_ERR_CUDA;
    d.num_sms = sms;
  }
  // debug: RS_DEBUG_CTA_PERMUTE=<m> (m >= 2) permutes which CTA of the persistent
  // decode and commit launches takes which unit range, to check that no result
  // depends on the order in which CTAs run or arrive
  if (const char* e = getenv("RS_DEBUG_CTA_PERMUTE")) d.cta_mult = atoi(e) >= 2 ? atoi(e) : 0;
  // debug: RS_DEBUG_UNIFORM_SPLIT=1 makes the d_state-128 decode split its units evenly
  // rather than by weight (to measure what the weighted split buys)
  if (const char* e = getenv("RS_DEBUG_UNIFORM_SPLIT")) d.uniform_split = atoi(e) != 0;
  d.ckpt = static_cast<float*>(bufs->ckpt);
  char* ring = static_cast<char*>(bufs->ring);
  if (cfg->kind == RS_MAMBA2) {
    d.r_x = reinterpret_cast<uint16_t*>(ring + L.r0);
    d.r_dt = reinterpret_cast<uint16_t*>(ring + L.r1);
    d.r_la = reinterpret_cast<float*>(ring + L.r2);
    d.r_B = reinterpret_cast<uint16_t*>(ring + L.r3);
  } else {
    d.r_u = reinterpret_cast<float*>(ring + L.r0);
    d.r_g = reinterpret_cast<float*>(ring + L.r1);
    d.r_k = reinterpret_cast<uint16_t*>(ring + L.r2);
  }
  d.cursor = static_cast<int*>(bufs->cursor);
  d.err = d.cursor + 4 * d.B;
  d.arrive = static_cast<int*>(bufs->scratch);
  d.vtab = L.s1 ? reinterpret_cast<float*>(static_cast<char*>(bufs->scratch) + L.s1) : nullptr;
  if (cfg->read_mode != RS_READ_NONE) {
    char* rc = static_cast<char*>(bufs->read_copy);
    d.rc_codes = reinterpret_cast<uint8_t*>(rc + L.c0);
    if (cfg->read_mode == RS_READ_FP8_ROW) {
      d.rc_rowscale = reinterpret_cast<float*>(rc + L.c1);
    } else {
      d.rc_blkscale = reinterpret_cast<uint8_t*>(rc + L.c1);
      d.rc_matscale = reinterpret_cast<float*>(rc + L.c2);
    }
  }

  cudaError_t e = cudaMemset(bufs->cursor, 0, L.cursor);
  if (e == cudaSuccess) e = cudaMemset(bufs->scratch, 0, L.scratch);
  if (e == cudaSuccess) e = cudaStreamSynchronize(0);
  if (e != cudaSuccess) return RS_ERR_CUDA;

  rs_cache* h = new (std::nothrow) rs_cache;
  if (!h) return RS_ERR_CUDA;
  h->cfg = *cfg;
  h->dev = d;
  h->pending = 0;
  h->pending_parents = 0;
  h->pending_chain = true;
  h->map_ok = rs::verify128_supports(d) && rs::make_ckpt_tmap(d, &h->ckpt_map) == cudaSuccess;
  *out = h;
  return RS_OK;
}

void rs_destroy_cache(rs_cache* cache) { delete cache; }

rs_status rs_decode_step(rs_cache* h, const rs_inputs* in, float* y, rs_stream stream) {
  if (!h || !y) return RS_ERR_NULL;
  const rs_status st = check_inputs(h, in);
  if (st != RS_OK) return st;
  if (!aligned16(y)) return RS_ERR_ALIGN;
  if (h->pending) return RS_ERR_STATE;
  return from_cuda(rs::launch_decode(h->dev, token_in(in), y, reinterpret_cast<cudaStream_t>(stream)));
}

// ---- host-buffer decode steps ----------------------------------------------

struct rs_pipe {
  rs_cache* cache;
  cudaStream_t h2d, d2h;                              // input copies, output copies
  cudaEvent_t in_ready[2], step_done[2], y_out[2];  // per slot
  unsigned char* dev_in[2];                          // one step's inputs, five 256-byte-aligned sections
  float* dev_y[2];
  size_t off[5], bytes[5], in_bytes, y_bytes;
  int64_t steps;
};

namespace {

// the five input arrays of one decode step, in rs_inputs order for the kind
void pipe_sections(const rs_config& c, size_t bytes[5]) {
  const size_t B = c.batch, H = c.n_heads, G = c.n_groups, P = c.d_head, N = c.d_state;
  if (c.kind == RS_MAMBA2) {
    bytes[0] = B * H * P * 2;  // x
    bytes[1] = B * H * 2;      // dt
    bytes[2] = H * 4;          // A
    bytes[3] = B * G * N * 2;  // Bm
    bytes[4] = B * G * N * 2;  // Cm
  } else {
    bytes[0] = B * G * N * 2;  // q
    bytes[1] = B * G * N * 2;  // k
    bytes[2] = B * H * P * 2;  // v
    bytes[3] = c.kind == RS_KDA ? B * H * N * 4 : B * H * 4;  // g (per key channel for KDA)
    bytes[4] = B * H * 4;      // beta
  }
}

const void* pipe_src(const rs_config& c, const rs_inputs* in, int i) {
  if (c.kind == RS_MAMBA2) {
    const void* p[5] = {in->x, in->dt, in->A, in->Bm, in->Cm};
    return p[i];
  }
  const void* p[5] = {in->q, in->k, in->v, in->g, in->beta};
  return p[i];
}

void pipe_free(rs_pipe* p) {
  for (int k = 0; k < 2; ++k) {
    if (p->in_ready[k]) cudaEventDestroy(p->in_ready[k]);
    if (p->step_done[k]) cudaEventDestroy(p->step_done[k]);
    if (p->y_out[k]) cudaEventDestroy(p->y_out[k]);
    if (p->dev_in[k]) cudaFree(p->dev_in[k]);
    if (p->dev_y[k]) cudaFree(p->dev_y[k]);
  }
  if (p->h2d) cudaStreamDestroy(p->h2d);
  if (p->d2h) cudaStreamDestroy(p->d2h);
  delete p;
}

}  // namespace

rs_status rs_pipe_create(rs_cache* cache, rs_pipe** out) {
  if (!cache || !out) return RS_ERR_NULL;
  *out = nullptr;
  rs_pipe* p = new (std::nothrow) rs_pipe{};
  if (!p) return RS_ERR_CUDA;
  p->cache = cache;
  pipe_sections(cache->cfg, p->bytes);
  size_t o = 0;
  for (int i = 0; i < 5; ++i) {
    p->off[i] = o;
    o = align256(o + p->bytes[i]);
  }
  p->in_bytes = o;
  p->y_bytes = static_cast<size_t>(cache->cfg.batch) * cache->cfg.n_heads * cache->cfg.d_head * 4;
  bool ok = cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking) == cudaSuccess;
  for (int k = 0; k < 2 && ok; ++k) {
    ok = cudaEventCreateWithFlags(&p->in_ready[k], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->step_done[k], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->y_out[k], cudaEventDisableTiming) == cudaSuccess &&
         cudaMalloc(reinterpret_cast<void**>(&p->dev_in[k]), p->in_bytes) == cudaSuccess &&
         cudaMalloc(reinterpret_cast<void**>(&p->dev_y[k]), p->y_bytes) == cudaSuccess;
  }
  if (!ok) {
    pipe_free(p);
    return RS_ERR_CUDA;
  }
  *out = p;
  return RS_OK;
}

rs_status rs_pipe_decode_step(rs_pipe* p, const rs_inputs* host_in, float* host_y, rs_stream stream) {
  if (!p || !host_in || !host_y) return RS_ERR_NULL;
  const rs_config& c = p->cache->cfg;
  for (int i = 0; i < 5; ++i)
    if (!pipe_src(c, host_in, i)) return RS_ERR_NULL;
  if (p->cache->pending) return RS_ERR_STATE;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int k = static_cast<int>(p->steps & 1);
  cudaError_t e = cudaSuccess;
  // inputs: into slot k once the kernel of two steps ago has read it
  if (p->steps >= 2) e = cudaStreamWaitEvent(p->h2d, p->step_done[k], 0);
  for (int i = 0; i < 5 && e == cudaSuccess; ++i)
    e = cudaMemcpyAsync(p->dev_in[k] + p->off[i], pipe_src(c, host_in, i), p->bytes[i], cudaMemcpyHostToDevice,
                        p->h2d);
  if (e == cudaSuccess) e = cudaEventRecord(p->in_ready[k], p->h2d);
  // the step on the caller's stream, once its inputs are in and y's slot has been read back
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, p->in_ready[k], 0);
  if (e == cudaSuccess && p->steps >= 2) e = cudaStreamWaitEvent(s, p->y_out[k], 0);
  if (e != cudaSuccess) return RS_ERR_CUDA;
  rs_inputs din{};
  const void* dp[5];
  for (int i = 0; i < 5; ++i) dp[i] = p->dev_in[k] + p->off[i];
  if (c.kind == RS_MAMBA2) {
    din.x = dp[0]; din.dt = dp[1]; din.A = static_cast<const float*>(dp[2]); din.Bm = dp[3]; din.Cm = dp[4];
  } else {
    din.q = dp[0]; din.k = dp[1]; din.v = dp[2]; din.g = static_cast<const float*>(dp[3]);
    din.beta = static_cast<const float*>(dp[4]);
  }
  const rs_status st = rs_decode_step(p->cache, &din, p->dev_y[k], stream);
  if (st != RS_OK) return st;
  // y back to the host on the output stream
  e = cudaEventRecord(p->step_done[k], s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p->d2h, p->step_done[k], 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(host_y, p->dev_y[k], p->y_bytes, cudaMemcpyDeviceToHost, p->d2h);
  if (e == cudaSuccess) e = cudaEventRecord(p->y_out[k], p->d2h);
  if (e != cudaSuccess) return RS_ERR_CUDA;
  ++p->steps;
  return RS_OK;
}

rs_status rs_pipe_sync(rs_pipe* p, rs_stream stream) {
  if (!p) return RS_ERR_NULL;
  if (p->steps == 0) return RS_OK;
  return from_cuda(cudaStreamWaitEvent(reinterpret_cast<cudaStream_t>(stream), p->y_out[(p->steps - 1) & 1], 0));
}

void rs_pipe_destroy(rs_pipe* p) {
  if (!p) return;
  cudaStreamSynchronize(p->h2d);
  cudaStreamSynchronize(p->d2h);
  pipe_free(p);
}

namespace {

// Ancestor mask and packed parents of a draft tree (parents[tau] in -1..tau-1);
// false for an invalid tree.
bool tree_of(int T, const int32_t* parents, uint32_t* anc, uint32_t* packed, bool* chain) {
  *anc = 0;
  *packed = 0;
  *chain = true;
  for (int tau = 0; tau < T; ++tau) {
    const int p = parents[tau];
    if (p < -1 || p >= tau) return false;
    *chain = *chain && p == tau - 1;
    *packed |= static_cast<uint32_t>(p + 1) << (8 * tau);
    uint32_t row = 1u << tau;  // tau itself
    if (p >= 0) row |= (*anc >> (4 * p)) & 0xFu;
    *anc |= row << (4 * tau);
  }
  return true;
}

rs_status verify_with_tree(rs_cache* h, int32_t T, const int32_t* parents, const rs_inputs* in, float* y,
                           rs_stream stream) {
  if (!h || !y) return RS_ERR_NULL;
  if (T < 1 || T > h->cfg.max_draft) return RS_ERR_RANGE;
  uint32_t anc = 0, packed = 0;
  bool chain = true;
  if (!tree_of(T, parents, &anc, &packed, &chain)) return RS_ERR_RANGE;
  const rs_status st = check_inputs(h, in);
  if (st != RS_OK) return st;
  if (!aligned16(y)) return RS_ERR_ALIGN;
  if (h->pending) return RS_ERR_STATE;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rs::LayerDev d = h->dev;
  d.tree_anc = anc;
  const cudaError_t e = h->map_ok ? rs::launch_verify128(d, h->ckpt_map, token_in(in), T, y, s)
                                  : rs::launch_verify(d, token_in(in), T, y, s);
  if (e != cudaSuccess) return RS_ERR_CUDA;
  h->pending = T;
  h->pending_parents = packed;
  h->pending_chain = chain;
  return RS_OK;
}

}  // namespace

rs_status rs_verify(rs_cache* h, int32_t T, const rs_inputs* in, float* y, rs_stream stream) {
  const int32_t chain[4] = {-1, 0, 1, 2};
  return verify_with_tree(h, T, chain, in, y, stream);
}

rs_status rs_verify_tree(rs_cache* h, int32_t T, const int32_t* parents, const rs_inputs* in, float* y,
                         rs_stream stream) {
  if (!parents) return RS_ERR_NULL;
  return verify_with_tree(h, T, parents, in, y, stream);
}

rs_status rs_commit_path(rs_cache* h, const int32_t* path_len, const int32_t* path, rs_stream stream) {
  if (!h || !path_len || !path) return RS_ERR_NULL;
  if (!aligned16(path_len) || !aligned16(path)) return RS_ERR_ALIGN;
  if (!h->pending) return RS_ERR_STATE;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the accepted counts the commit launch applies live in the verify-table scratch,
  // which only rs_verify uses
  int* acc = reinterpret_cast<int*>(h->dev.vtab);
  cudaError_t e = rs::launch_tree_compact(h->dev, path_len, path, h->cfg.max_draft, h->pending,
                                          h->pending_parents, acc, s);
  if (e == cudaSuccess) e = rs::launch_fold(h->dev, rs::FOLD_COMMIT, acc, nullptr, h->pending, s);
  if (e != cudaSuccess) return RS_ERR_CUDA;
  h->pending = 0;
  return RS_OK;
}

rs_status rs_commit(rs_cache* h, const int32_t* accepted, rs_stream stream) {
  if (!h || !accepted) return RS_ERR_NULL;
  if (!aligned16(accepted)) return RS_ERR_ALIGN;
  if (!h->pending || !h->pending_chain) return RS_ERR_STATE;
  const cudaError_t e = rs::launch_fold(h->dev, rs::FOLD_COMMIT, accepted, nullptr, h->pending,
                                        reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return RS_ERR_CUDA;
  h->pending = 0;
  return RS_OK;
}

rs_status rs_flush(rs_cache* h, const uint8_t* seq_mask, rs_stream stream) {
  if (!h) return RS_ERR_NULL;
  if (seq_mask && !aligned16(seq_mask)) return RS_ERR_ALIGN;
  if (h->pending) return RS_ERR_STATE;
  return from_cuda(rs::launch_fold(h->dev, rs::FOLD_FLUSH, nullptr, seq_mask, 0,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

rs_status rs_get_device_error(rs_cache* h, rs_stream stream, int32_t* code) {
  if (!h || !code) return RS_ERR_NULL;
  int32_t word[2] = {0, 0};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(word, h->dev.err, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return RS_ERR_CUDA;
  *code = word[0];
  return word[0] == 0 ? RS_OK : RS_ERR_DEVICE;
}

const char* rs_status_string(rs_status s) {
  switch (s) {
    case RS_OK: return "ok";
    case RS_ERR_NULL: return "a required pointer is NULL";
    case RS_ERR_SHAPE: return "config dimensions inconsistent or out of range";
    case RS_ERR_ALIGN: return "a device pointer is not 16-byte aligned";
    case RS_ERR_RANGE: return "a scalar argument is out of range";
    case RS_ERR_STATE: return "call order violated (verify must be followed by one commit)";
    case RS_ERR_UNSUPPORTED: return "configuration outside the built kernels";
    case RS_ERR_CUDA: return "a CUDA runtime call failed";
    case RS_ERR_DEVICE: return "the device error word is set";
  }
  return "unknown status";
}

}  // extern "C"
