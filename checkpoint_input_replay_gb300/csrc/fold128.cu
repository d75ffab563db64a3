// Commit (pointer advance) and explicit flush for d_state = 128 and d_head 64
// or 128: the sequences whose window is complete (commit) or that the caller
// selects (flush) fold their buffered records into the checkpoint,
//   S_new = gamma S_ckpt + sum_{j<n} w_j d_j k_j^T,
//   w_j = prod_{i=j+1..n-1} a_i,  gamma = prod_{i<n} a_i,
// d_j = dt_j x_j (Mamba-2) or the buffered delta u_j (Gated DeltaNet), and
// every cursor moves ("ReplaySSM caches SSM inputs instead of state"
// (richland.au), "What shipped": the accepted prefix is committed by
// advancing a pointer; records past it are ignored and overwritten).  Same
// arithmetic as fold.cu, which serves the other shapes.
//
// Structure as in decode128.cu: one persistent CTA per SM.  Only the
// (sequence, head) units of folding sequences are work: every CTA scans all
// cursors, numbers the folding sequences in order and takes an equal
// contiguous share of their units, so a commit in which few sequences fold
// costs little more than their state traffic and no CTA carries more than its
// share.  The last CTA to finish the scan writes every cursor.  The producer
// warp stages each folding unit (the state matrix and its records) with bulk
// copies and, once per group, the group's keys and ring decay rows; the
// prologue warp computes, once per group, each head's fold weights from one
// suffix scan; eight computing warps fold in registers (fold coefficients from
// a per-warp shared-memory table, four records per broadcast read, packed
// fma.rn.f32x2), store the checkpoint once and refresh the low-precision read
// copy where there is one.
#include "common.cuh"

namespace rs {
namespace {

constexpr int N = 128;
constexpr int SEG = N / 4;
constexpr int kMaxSeqF = 64;
constexpr int kThreadsF = kThreads + 64;  // 8 computing warps, prologue warp, producer warp
constexpr int kPrologueWarp = kThreads / 32;
constexpr int kProducerWarp = kThreads / 32 + 1;
// row stride (floats) of a warp's fold-coefficient table: kMaxRec padded so the
// 32 lanes' stores (8 rows x 4 records) fall in 32 different banks
constexpr int kMtabRow = kMaxRec + 4;

__host__ __device__ __forceinline__ int al16(int x) { return (x + 15) & ~15; }
__host__ __device__ __forceinline__ int al128(int x) { return (x + 127) & ~127; }
// floats per head in a fold table: w_j d-scale for the C records, then gamma
__host__ __device__ __forceinline__ int fold_stride(int C) { return (C + 4 + 3) & ~3; }

struct LayF {
  int st_tile, st_rec, st_meta, st_size;
  int gb_key, gb_la, gb_dt, gb_coef, gb_size;
  int pe_bars, pe_seq, pe_misc, pe_cnt, pe_mtab, pe_size;
};

__host__ __device__ __forceinline__ LayF layf(int kind, int P, int C, int Cp, int hpg) {
  LayF l;
  int o = 0;
  l.st_tile = o;  o += P * N * 4;
  l.st_rec = o;   o += kind == 0 ? al16(C * P * 2) : C * P * 4;
  l.st_meta = o;  o += 32;  // int4 descriptor, NVFP4 amax word
  l.st_size = al128(o);
  o = 0;
  l.gb_key = o;   o += C * N * 2;
  l.gb_la = o;    o += hpg * Cp * 4;
  l.gb_dt = o;    o += kind == 0 ? al16(hpg * Cp * 2) : 0;
  l.gb_coef = o;  o += hpg * fold_stride(C) * 4;
  l.gb_size = al128(o);
  o = 0;
  l.pe_bars = o;  o += 4 * 8 * 8;  // full, empty, ready, amax x 8 stages
  l.pe_seq = o;   o += 3 * kMaxSeqF * 4;
  l.pe_misc = o;  o += 16;
  l.pe_cnt = o;   o += al16((kThreadsF / 32 + 1) * 4);  // per-warp counts of the sequence scan, last-CTA flag
  l.pe_mtab = o;  o += (kThreads / 32) * 8 * kMtabRow * 4;  // per computing warp: fold coefficients [8 rows][records]
  l.pe_size = al128(o);
  return l;
}

__device__ __forceinline__ int ring_slot(int head, int j, int C) {
  int s = head + j;
  return s >= C ? s - C : s;
}

// Position of a staged unit: the CTA's sequence slot k (its sequence is
// sseq[3k]), head h, group g, head-in-group hh; advanced one unit at a time.
struct FWalk {
  int k, h, g, hh;
  __device__ __forceinline__ void start(int u0, int H, int hpg) {
    k = 0;
    h = u0 - (u0 / H) * H;
    g = h / hpg;
    hh = h - g * hpg;
  }
  __device__ __forceinline__ void next(int H, int hpg) {
    ++h;
    if (++hh == hpg) {
      hh = 0;
      ++g;
    }
    if (h == H) {
      h = 0;
      g = 0;
      ++k;
    }
  }
};

template <int KIND, int READ, int P>
__global__ void __launch_bounds__(kThreadsF, 1)
    fold128_kernel(const LayerDev d, const int mode, const int* __restrict__ accepted,
                   const uint8_t* __restrict__ mask, const int T_pending, const int stages) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int RW = P / 8;
  constexpr int tile = P * N;
  const int H = d.H, G = d.G, C = d.C, L = d.L, Cp = d.Cp;
  const int hpg = H / G;
  const int FS = fold_stride(C);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const LayF LY = layf(KIND, P, C, Cp, hpg);
  unsigned char* gbase = smem + static_cast<size_t>(LY.st_size) * stages;
  unsigned char* pbase = gbase + 2 * LY.gb_size;
  uint64_t* full = reinterpret_cast<uint64_t*>(pbase + LY.pe_bars);
  uint64_t* empty = full + 8;
  uint64_t* ready = full + 16;
  uint64_t* amaxbar = full + 24;
  int* sseq = reinterpret_cast<int*>(pbase + LY.pe_seq);
  volatile int* smisc = reinterpret_cast<volatile int*>(pbase + LY.pe_misc);  // abort, issued, producer done
  // this warp's fold-coefficient table (computing warps)
  float* mt = reinterpret_cast<float*>(pbase + LY.pe_mtab) + (warp < kThreads / 32 ? warp : 0) * 8 * kMtabRow;

  // --- the folding sequences, numbered in order (every CTA computes the same list) ---
  int* s_cnt = reinterpret_cast<int*>(pbase + LY.pe_cnt);
  int& s_last = s_cnt[kThreadsF / 32];
  auto decide = [&](int b, int* head, int* n_new, int* flags) {
    const int hd = d.cursor[4 * b], cnt = d.cursor[4 * b + 1];
    bool ok = static_cast<unsigned>(hd) < static_cast<unsigned>(C) &&
              static_cast<unsigned>(cnt) < static_cast<unsigned>(L);
    int nacc = 0;
    bool acc_ok = true;
    if (mode == FOLD_COMMIT) {
      nacc = accepted[b];
      acc_ok = nacc >= 0 && nacc <= T_pending;
      ok = ok && cnt + T_pending <= C;
    }
    const bool fold = ok && acc_ok && (mode == FOLD_FLUSH ? (mask == nullptr || mask[b] != 0) : cnt + nacc >= L);
    *head = hd;
    *n_new = cnt + nacc;
    // bit 0: a unit is staged (records to fold, or a read copy to refresh); bit 1: folds;
    // bit 2: cursor invalid; bit 3: accepted count invalid
    *flags = ((fold && (cnt + nacc > 0 || READ != READ_NONE)) ? 1 : 0) | (fold ? 2 : 0) | (ok ? 0 : 4) |
             (acc_ok ? 0 : 8);
  };
  // pass 1: how many sequences are staged
  int mine = 0;
  for (int b = t; b < d.B; b += kThreadsF) {
    int hd, nn, fl;
    decide(b, &hd, &nn, &fl);
    mine += fl & 1;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) s_cnt[warp] = mine;
  __syncthreads();
  int K = 0;
  for (int w = 0; w < kThreadsF / 32; ++w) K += s_cnt[w];
  const int total_units = K * H;
  const int per = (total_units + gridDim.x - 1) / gridDim.x;
  const int u0 = min(cta_index(d.cta_mult) * per, total_units);
  const int u1 = min(u0 + per, total_units);
  const int nunits = u1 - u0;
  const int k0 = u0 / H;  // first staged sequence of this CTA (in the numbering)
  const int nseq = nunits > 0 ? (u1 - 1) / H - k0 + 1 : 0;
  // pass 2: the staged sequences numbered k0 .. k0 + nseq - 1, by a running prefix count
  int base = 0;
  for (int b0c = 0; b0c < d.B; b0c += kThreadsF) {
    const int b = b0c + t;
    int hd = 0, nn = 0, fl = 0;
    if (b < d.B) decide(b, &hd, &nn, &fl);
    const int f = fl & 1;
    const unsigned bal = __ballot_sync(0xffffffffu, f);
    const int pre_w = __popc(bal & ((1u << lane) - 1u));
    __syncthreads();
    if (lane == 0) s_cnt[warp] = __popc(bal);
    __syncthreads();
    int pre = base + pre_w;
    for (int w = 0; w < warp; ++w) pre += s_cnt[w];
    if (f && pre >= k0 && pre < k0 + nseq) {
      const int k = pre - k0;
      sseq[3 * k] = b;
      sseq[3 * k + 1] = hd;
      sseq[3 * k + 2] = (fl & 2) ? nn : 0;
    }
    for (int w = 0; w < kThreadsF / 32; ++w) base += s_cnt[w];
  }
  // every cursor has been read by this CTA: count it in; the last CTA writes the cursors
  __syncthreads();
  if (t == 0) {
    __threadfence();
    s_last = atomicAdd(d.arrive, 1) == static_cast<int>(gridDim.x) - 1;
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    for (int b = t; b < d.B; b += kThreadsF) {
      int hd, nn, fl;
      decide(b, &hd, &nn, &fl);
      if (fl & 4) {
        report_error(d.err, DEVERR_CURSOR, b);
      } else if (fl & 8) {
        report_error(d.err, DEVERR_ACCEPTED, b);
      } else if (fl & 2) {
        d.cursor[4 * b] = ring_slot(hd, nn, C);
        d.cursor[4 * b + 1] = 0;
        d.cursor[4 * b + 2] = 1;
      } else {
        d.cursor[4 * b + 1] = nn;
        d.cursor[4 * b + 2] = 0;
      }
    }
    if (t == 0) atomicExch(d.arrive, 0);
  }
  if (nunits <= 0) return;

  if (t == kThreads) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kThreads / 32);
      mbar_init(ready + s, 1);
      mbar_init(amaxbar + s, kThreads / 32);
    }
    smisc[0] = 0;
    smisc[1] = 0;
    smisc[2] = 0;
  }
  __syncthreads();

  // =============================== producer warp ===============================
  if (warp == kProducerWarp) {
    if (lane != 0) return;
    FWalk w;
    w.start(u0, H, hpg);
    int k = 0, gi = -1;  // active units issued, group ordinal
    for (int i = 0; i < nunits; ++i, w.next(H, hpg)) {
      const bool first = k == 0 || w.hh == 0;
      if (first) ++gi;
      const int s = k % stages;
      if (k >= stages && !mbar_wait_bounded(empty + s, static_cast<uint32_t>(((k / stages) - 1) & 1))) break;
      if (smisc[0]) break;
      const int b = sseq[3 * w.k], head = sseq[3 * w.k + 1], n = sseq[3 * w.k + 2];
      unsigned char* st = smem + static_cast<size_t>(LY.st_size) * s;
      unsigned char* gb = gbase + static_cast<size_t>(LY.gb_size) * (gi & 1);
      uint64_t* bar = full + s;
      const size_t u = static_cast<size_t>(b) * H + w.h;
      const int seg1 = min(n, C - head), seg2 = n - seg1;
      constexpr int esz = KIND == 0 ? 2 : 4;
      const size_t ug = static_cast<size_t>(b) * H + static_cast<size_t>(w.g) * hpg;
      const size_t bg = static_cast<size_t>(b) * G + w.g;
      uint32_t bytes = tile * 4 + static_cast<uint32_t>(n) * P * esz;
      if (first) {
        bytes += static_cast<uint32_t>(n) * N * 2 + hpg * Cp * 4;
        if (KIND == 0) bytes += hpg * Cp * 2;
      }
      mbar_expect_tx(bar, bytes);
      bulk_g2s(st + LY.st_tile, d.ckpt + u * tile, tile * 4, bar);
      const unsigned char* rsrc = KIND == 0 ? reinterpret_cast<const unsigned char*>(d.r_x)
                                            : reinterpret_cast<const unsigned char*>(d.r_u);
      constexpr size_t rrow = static_cast<size_t>(P) * esz;
      if (seg1) bulk_g2s(st + LY.st_rec, rsrc + (u * C + head) * rrow, seg1 * rrow, bar);
      if (seg2) bulk_g2s(st + LY.st_rec + seg1 * rrow, rsrc + u * C * rrow, seg2 * rrow, bar);
      if (first) {
        const uint16_t* rk = (KIND == 0 ? d.r_B : d.r_k) + bg * C * N;
        if (seg1) bulk_g2s(gb + LY.gb_key, rk + static_cast<size_t>(head) * N, seg1 * N * 2, bar);
        if (seg2) bulk_g2s(gb + LY.gb_key + seg1 * N * 2, rk, seg2 * N * 2, bar);
        bulk_g2s(gb + LY.gb_la, (KIND == 0 ? d.r_la : d.r_g) + ug * Cp, hpg * Cp * 4, bar);
        if (KIND == 0) bulk_g2s(gb + LY.gb_dt, d.r_dt + ug * Cp, hpg * Cp * 2, bar);
      }
      ++k;
      smisc[1] = k;
    }
    smisc[2] = 1;
    return;
  }

  const int kq = (lane >> 2) & 7, jl = lane & 3;

  // =============================== prologue warp ===============================
  if (warp == kPrologueWarp) {
    FWalk w;
    w.start(u0, H, hpg);
    int k = 0, gi = -1, consumed = 0;
    for (int i = 0; i < nunits; ++i, w.next(H, hpg)) {
      if (smisc[0]) break;
      const int s = k % stages;
      const int b = sseq[3 * w.k], head = sseq[3 * w.k + 1], n = sseq[3 * w.k + 2];
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(full + s, static_cast<uint32_t>((k / stages) & 1)))) {
        if (lane == 0) {
          report_error(d.err, DEVERR_TIMEOUT, b);
          smisc[0] = 1;
        }
        break;
      }
      consumed = k + 1;
      const bool first = k == 0 || w.hh == 0;
      if (first) ++gi;
      unsigned char* gb = gbase + static_cast<size_t>(LY.gb_size) * (gi & 1);
      if (first) {
        // fold weights of the heads of this group in this CTA: one suffix scan per head
        const int slot_lane = lane < n ? ring_slot(head, lane, C) : 0;
        int hh_hi = hpg;  // heads of this group in this CTA
        {
          const int left = nunits - i;
          if (w.hh + left < hh_hi) hh_hi = w.hh + left;
        }
        for (int e = w.hh; e < hh_hi; ++e) {
          float* co = reinterpret_cast<float*>(gb + LY.gb_coef) + e * FS;
          const float* la_row = reinterpret_cast<const float*>(gb + LY.gb_la) + e * Cp;
          // w_j = exp(sum_{i=j+1..n-1} la_i), gamma = exp(sum_{i<n} la_i)
          const float sv = suffix_sum(lane < n ? la_row[slot_lane] : 0.f, lane, n - 1);
          const float excl = __shfl_down_sync(0xffffffffu, sv, 1);
          const float Wl = lane < n ? expf(lane + 1 < n ? excl : 0.f) : 0.f;
          float scale = 1.f;
          if (KIND == 0) scale = lane < n ? bf(reinterpret_cast<const uint16_t*>(gb + LY.gb_dt)[e * Cp + slot_lane]) : 0.f;
          if (lane < n) co[lane] = Wl * scale;  // fold coefficient of the record's x (dt w_j) or u (w_j)
          if (lane == 0) co[C] = n > 0 ? expf(sv) : 1.f;
        }
      }
      if (lane == 0) {
        unsigned char* st = smem + static_cast<size_t>(LY.st_size) * s;
        *reinterpret_cast<int4*>(st + LY.st_meta) = make_int4(b * H + w.h, n, w.hh, gi & 1);
        reinterpret_cast<int*>(st + LY.st_meta)[4] = 0;  // NVFP4 matrix amax
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(ready + s);
      ++k;
    }
    // after an abort: let the copies already issued land before the CTA exits
    if (smisc[0] && lane == 0) {
      const uint64_t t0 = global_ns();
      while (!smisc[2] && global_ns() - t0 < 2000000000ull) {
      }
      const int issued = smisc[1];
      for (int j = consumed; j < issued; ++j)
        mbar_wait_bounded(full + (j % stages), static_cast<uint32_t>((j / stages) & 1));
    }
    return;
  }

  // =============================== computing warps ===============================
  uint32_t amax_phase = 0;
  int k = 0;
  for (int i = 0; i < nunits; ++i) {
    if (smisc[0]) break;
    const int s = k % stages;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(ready + s, static_cast<uint32_t>((k / stages) & 1)))) {
      if (lane == 0) {
        report_error(d.err, DEVERR_TIMEOUT, sseq[0]);
        smisc[0] = 1;
      }
      break;
    }
    ++k;
    unsigned char* st = smem + static_cast<size_t>(LY.st_size) * s;
    const int4 meta = *reinterpret_cast<const int4*>(st + LY.st_meta);
    const size_t u = static_cast<size_t>(meta.x);
    const int n = meta.y, hh = meta.z;
    const unsigned char* gb = gbase + static_cast<size_t>(LY.gb_size) * meta.w;
    const float* co = reinterpret_cast<const float*>(gb + LY.gb_coef) + hh * FS;
    const uint16_t* kb = reinterpret_cast<const uint16_t*>(gb + LY.gb_key);
    float4* sT4 = reinterpret_cast<float4*>(st + LY.st_tile);
    float4* gS4 = reinterpret_cast<float4*>(d.ckpt + u * tile);
    const float gamma = co[C];
    if (n > 0) {
#pragma unroll
      for (int r0 = 0; r0 < RW; r0 += 8) {
        const int Rq = warp + 8 * (r0 + kq);
        // m_j[row] = coefficient * record j (j < n) into this warp's table, lane (kq, jl)
        // writing records jl, jl + 4, .. of row slot kq (zero past n to the end of the
        // last quad); then four records per broadcast read
        for (int jc = 0; 4 * jc < n; ++jc) {
          const int j = 4 * jc + jl;
          float rv = 0.f;
          if (j < n) {
            if (KIND == 0) rv = bf(reinterpret_cast<const uint16_t*>(st + LY.st_rec)[j * P + Rq]);
            else rv = reinterpret_cast<const float*>(st + LY.st_rec)[j * P + Rq];
          }
          mt[kq * kMtabRow + j] = j < n ? co[j] * rv : 0.f;
        }
        __syncwarp();
        float4 acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = scale4(gamma, sT4[(warp + 8 * (r0 + e)) * SEG + lane]);
        for (int jq = 0; 4 * jq < n; ++jq) {
          float4 k4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            k4[i] = 4 * jq + i < n ? bf4(reinterpret_cast<const uint2*>(kb + (4 * jq + i) * N)[lane])
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 m4 = *reinterpret_cast<const float4*>(mt + e * kMtabRow + 4 * jq);
            acc[e] = axpy4x2(m4.x, k4[0], acc[e]);
            acc[e] = axpy4x2(m4.y, k4[1], acc[e]);
            acc[e] = axpy4x2(m4.z, k4[2], acc[e]);
            acc[e] = axpy4x2(m4.w, k4[3], acc[e]);
          }
        }
        __syncwarp();
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          __stcs(gS4 + (warp + 8 * (r0 + e)) * SEG + lane, acc[e]);
          if (READ != READ_NONE) sT4[(warp + 8 * (r0 + e)) * SEG + lane] = acc[e];
        }
      }
    }
    if (READ == READ_FP8) {
      // refresh the read copy of this warp's rows from the folded rows in shared memory
      uint32_t* codes = reinterpret_cast<uint32_t*>(d.rc_codes + u * tile);
#pragma unroll
      for (int m = 0; m < RW; ++m) {
        const int R = warp + 8 * m;
        const float4 v4 = sT4[R * SEG + lane];
        float mx = fmaxf(fmaxf(fabsf(v4.x), fabsf(v4.y)), fmaxf(fabsf(v4.z), fabsf(v4.w)));
        mx = seg_max<32>(mx);
        const float scale = div_by(mx, 448.0f, kInv448);
        uint32_t packed = 0;
        if (scale != 0.0f) {
          const float rs = __frcp_rn(scale);
          const uint32_t lo = f32x2_to_e4m3x2(div_by(v4.x, scale, rs), div_by(v4.y, scale, rs));
          const uint32_t hi = f32x2_to_e4m3x2(div_by(v4.z, scale, rs), div_by(v4.w, scale, rs));
          packed = lo | (hi << 16);
        }
        codes[R * SEG + lane] = packed;
        if (lane == 0) d.rc_rowscale[u * P + R] = scale;
      }
    } else if (READ == READ_NVFP4) {
      float mloc = 0.f;
#pragma unroll
      for (int m = 0; m < RW; ++m) {
        const float4 v4 = sT4[(warp + 8 * m) * SEG + lane];
        mloc = fmaxf(mloc, fmaxf(fmaxf(fabsf(v4.x), fabsf(v4.y)), fmaxf(fabsf(v4.z), fabsf(v4.w))));
      }
      mloc = seg_max<32>(mloc);
      int* slot_amax = reinterpret_cast<int*>(st + LY.st_meta) + 4;
      if (lane == 0) atomicMax(slot_amax, __float_as_int(mloc));  // non-negative floats order as ints
      __syncwarp();
      if (lane == 0) mbar_arrive(amaxbar + s);
      const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(amaxbar + s, (amax_phase >> s) & 1u));
      amax_phase ^= 1u << s;
      if (!got) {
        if (lane == 0) {
          report_error(d.err, DEVERR_TIMEOUT, static_cast<int>(u / H));
          smisc[0] = 1;
        }
      } else {
        const float amax = __int_as_float(*reinterpret_cast<volatile int*>(slot_amax));
        const float smat = __fdiv_rn(amax, 2688.0f);  // 448 * 6
        const float six_s = __fmul_rn(6.0f, smat);
        const float r6 = six_s != 0.0f ? __frcp_rn(six_s) : 0.0f;
        uint16_t* codes = reinterpret_cast<uint16_t*>(d.rc_codes + u * (tile / 2));
        uint8_t* blk = d.rc_blkscale + u * (tile / 16);
#pragma unroll
        for (int m = 0; m < RW; ++m) {
          const int R = warp + 8 * m;
          const float4 v4 = sT4[R * SEG + lane];
          float mb = fmaxf(fmaxf(fabsf(v4.x), fabsf(v4.y)), fmaxf(fabsf(v4.z), fabsf(v4.w)));
          mb = seg_max<4>(mb);  // 4 lanes = one 16-element block
          uint32_t bcode = 0;
          if (six_s != 0.0f) bcode = f32x2_to_e4m3x2(div_by(mb, six_s, r6), 0.0f) & 0xFFu;
          const float dd = __fmul_rn(e4m3_to_f32(bcode), smat);
          uint32_t qv = 0;
          if (dd != 0.0f) {
            const float rd = __frcp_rn(dd);
            qv = f32x4_to_e2m1x4(div_by(v4.x, dd, rd), div_by(v4.y, dd, rd), div_by(v4.z, dd, rd), div_by(v4.w, dd, rd));
          }
          codes[R * SEG + lane] = static_cast<uint16_t>(qv);
          if ((lane & 3) == 0) blk[R * (N / 16) + (lane >> 2)] = static_cast<uint8_t>(bcode);
        }
        if (warp == 0 && lane == 0) d.rc_matscale[u] = smat;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + s);
  }
}

template <int KIND, int READ, int P>
cudaError_t launch_f128(const LayerDev& d, int mode, const int* accepted, const uint8_t* mask, int T_pending,
                        cudaStream_t s) {
  const int hpg = d.H / d.G;
  const LayF LY = layf(KIND, P, d.C, d.Cp, hpg);
  const long budget = 227L * 1024 - 2L * LY.gb_size - LY.pe_size;
  long stages = budget / LY.st_size;
  if (stages > 8) stages = 8;
  // a group buffer is rewritten two groups later: every unit of that earlier
  // group must have left the pipeline, which holds when stages <= hpg + 1
  if (stages > hpg + 1) stages = hpg + 1;
  if (stages < 1) return cudaErrorInvalidConfiguration;
  const size_t smem = static_cast<size_t>(LY.st_size) * stages + 2u * LY.gb_size + LY.pe_size;
  // the share of each CTA is computed on the device from the number of folding
  // sequences; enough CTAs that a share spans at most kMaxSeqF - 2 sequences
  int grid = d.num_sms > 0 ? d.num_sms : 1;
  while ((d.B + grid - 1) / grid + 2 > kMaxSeqF) grid *= 2;
  auto kernel = fold128_kernel<KIND, READ, P>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  LayerDev dd = d;
  dd.cta_mult = coprime_mult(d.cta_mult, grid);
  kernel<<<grid, kThreadsF, smem, s>>>(dd, mode, accepted, mask, T_pending, static_cast<int>(stages));
  return cudaGetLastError();
}

template <int P>
cudaError_t launch_f128_p(const LayerDev& d, int mode, const int* accepted, const uint8_t* mask, int T_pending,
                          cudaStream_t s) {
  if (d.kind == 0) {
    if (d.read_mode == READ_FP8) return launch_f128<0, READ_FP8, P>(d, mode, accepted, mask, T_pending, s);
    if (d.read_mode == READ_NVFP4) return launch_f128<0, READ_NVFP4, P>(d, mode, accepted, mask, T_pending, s);
    return launch_f128<0, READ_NONE, P>(d, mode, accepted, mask, T_pending, s);
  }
  return launch_f128<1, READ_NONE, P>(d, mode, accepted, mask, T_pending, s);
}

}  // namespace

bool fold128_supports(const LayerDev& d) {
  if (d.N != N || (d.P != 64 && d.P != 128) || d.C > kMaxRec) return false;
  const LayF LY = layf(d.kind, d.P, d.C, d.Cp, d.H / d.G);
  return static_cast<long>(LY.st_size) + 2L * LY.gb_size + LY.pe_size <= 227L * 1024;
}

cudaError_t launch_fold128(const LayerDev& d, int mode, const int* accepted, const uint8_t* mask, int T_pending,
                           cudaStream_t s) {
  if (!fold128_supports(d)) return cudaErrorInvalidValue;
  return d.P == 64 ? launch_f128_p<64>(d, mode, accepted, mask, T_pending, s)
                   : launch_f128_p<128>(d, mode, accepted, mask, T_pending, s);
}

}  // namespace rs
