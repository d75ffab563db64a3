/*
 * replayssm.h -- C ABI of the ReplaySSM decode hot path for one SSM layer on
 * one GPU (sm_103a).
 *
 * The conventional SSM decoder reads the recurrent state, applies a rank-1
 * update and writes the state back for every token.  ReplaySSM keeps instead a
 * high-precision checkpoint plus a ring buffer of the last L input records;
 * non-flush steps compute the output from checkpoint + buffer without storing
 * any state, and the state is written once per window when the buffer fills
 * ("ReplaySSM caches SSM inputs instead of state, cutting hybrid-model decode
 * traffic in half" (richland.au), section "What shipped"; "NVIDIAとプリンストン
 * 大Dao AI Lab、ハイブリッドモデルの推論を速める「ReplaySSM」を公開"
 * (ai-jitan-hub.com), section "ReplaySSMは何をする手法か").
 *
 * Two recurrences, per head:
 *   Mamba-2:         S_t = a_t S_{t-1} + v_t k_t^T,                     y_t = S_t q_t
 *                    a_t = exp(dt_t A_h), v_t = dt_t x_t, k_t = B_t, q_t = C_t
 *   Gated DeltaNet:  S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T, o_t = S_t q_t
 *                    a_t = exp(g_t), b_t = beta_t
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every function returns rs_status.  Nothing throws across the ABI.
 *   Argument errors are detected on the host before any launch; the cache is
 *   then left unchanged.
 * - Device memory is owned by the caller (rs_query_sizes gives the sizes);
 *   the library owns only the opaque host handle rs_cache.
 * - All device pointers must be 16-byte aligned.  Device pointers may be any
 *   memory the GPU can load from with the same address (cudaMalloc, managed).
 * - Calls are asynchronous and stream-ordered on the caller's stream.  Calls
 *   on one cache must not overlap in time (use one stream, or order them).
 * - bf16 = IEEE bfloat16 bit patterns (uint16); f32 = float.
 * - Environment (debug only): RS_DEBUG_CTA_PERMUTE=<m>, m >= 2, read by
 *   rs_create_cache and by every rs_decode_step_noalloc call, permutes which
 *   CTA of the persistent decode and commit launches takes which range of
 *   work (an ordering check); results do not change.  RS_DEBUG_UNIFORM_SPLIT=1,
 *   read by rs_create_cache, makes the d_state-128 decode launch split its work
 *   evenly over its CTAs instead of by weight (a flush unit counts more), to
 *   measure what the weighted split buys in batches at mixed window positions;
 *   results do not change.  Unset in normal use.
 * - Kernels never trap.  A problem found on the device (corrupt cursor,
 *   accepted count out of range, a staged copy that did not arrive in time)
 *   sets a sticky device error word and leaves that sequence untouched;
 *   read it with rs_get_device_error.
 *
 * Notation: B batch, H heads (Mamba-2 nheads | GDN value heads), G groups
 * (Mamba-2 ngroups | GDN key heads), P = d_head (Mamba-2 headdim | GDN d_v),
 * N = d_state (Mamba-2 dstate | GDN d_k), L ring_len, T_max max_draft,
 * C = L + T_max ring capacity, Cp = C rounded up to a multiple of 8.
 * Head h uses group h / (H / G).
 */
#ifndef REPLAYSSM_H
#define REPLAYSSM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *rs_stream;

typedef enum {
  RS_OK = 0,
  RS_ERR_NULL = 1,        /* a required pointer is NULL                         */
  RS_ERR_SHAPE = 2,       /* config dimensions inconsistent or out of range     */
  RS_ERR_ALIGN = 3,       /* a device pointer is not 16-byte aligned            */
  RS_ERR_RANGE = 4,       /* a scalar argument (T, kind, mode) out of range     */
  RS_ERR_STATE = 5,       /* call order violated (see rs_verify / rs_commit)    */
  RS_ERR_UNSUPPORTED = 6, /* valid but not built (see rs_query_sizes)           */
  RS_ERR_CUDA = 7,        /* a CUDA runtime call failed                         */
  RS_ERR_DEVICE = 8       /* the device error word is set                       */
} rs_status;

/* RS_KDA: the Gated DeltaNet rule with a per-key-channel gate (the gate form of
 * Kimi Delta Attention), S_t = S_{t-1} Diag(a_t) (I - b_t k_t k_t^T) + b_t v_t k_t^T,
 * a_t = exp(g_t) over the d_state key channels, o_t = S_t q_t -- a recurrence the
 * method generalises to ("ReplaySSM caches SSM inputs..." (richland.au), "Why it
 * matters").  Decode and flush only (max_draft must be 0). */
typedef enum { RS_MAMBA2 = 0, RS_GDN = 1, RS_KDA = 2 } rs_kind;

/* Low-precision read copy of the checkpoint, used only for the checkpoint
 * read of non-flush decode steps and never fed back into the recurrence
 * ("ReplaySSM caches SSM inputs..." (richland.au), "What shipped", the
 * paragraph on quantization; ai-jitan-hub.com, "何がどれだけ速くなったのか",
 * item 3).  Mamba-2 only. */
typedef enum { RS_READ_NONE = 0, RS_READ_FP8_ROW = 1, RS_READ_NVFP4 = 2 } rs_read_mode;

/* Device error codes (the sticky word read by rs_get_device_error). */
enum {
  RS_DEVERR_NONE = 0,
  RS_DEVERR_ACCEPTED = 1, /* rs_commit: accepted[b] < 0 or > drafts pending   */
  RS_DEVERR_CURSOR = 2,   /* a cursor (head, count) outside its valid range   */
  RS_DEVERR_TIMEOUT = 3   /* a staged tile copy did not complete in time      */
};

typedef struct {
  int32_t kind;      /* rs_kind                                            */
  int32_t batch;     /* B >= 1                                             */
  int32_t n_heads;   /* H, a multiple of n_groups                          */
  int32_t n_groups;  /* G >= 1                                             */
  int32_t d_head;    /* P in {16, 32, 64, 128}                             */
  int32_t d_state;   /* N in {16, 32, 64, 128}; P * N * 4 <= 65536         */
  int32_t ring_len;  /* L >= 1                                             */
  int32_t max_draft; /* T_max >= 0 (0: standard decode only), L+T_max<=32  */
  int32_t read_mode; /* rs_read_mode (Mamba-2 only)                      */
} rs_config;

/*
 * Caller-owned device buffers (sizes from rs_query_sizes, in this order).
 *
 * ckpt       f32 [B][H][P][N], N contiguous: the FP32 checkpoint S_ckpt.  The
 *            caller writes the initial state here before the first call.
 * ring       the input-record ring, C slots per sequence; record j since the
 *            last flush lives in slot (head + j) mod C.  Sections, each
 *            starting on a 256-byte boundary:
 *              Mamba-2: x bf16 [B][H][C][P] | dt bf16 [B][H][Cp] |
 *                       log a = dt*A f32 [B][H][Cp] | B bf16 [B][G][C][N]
 *              GDN:     u f32 [B][H][C][P] (delta u = b (v - a S_{t-1} k)) |
 *                       g f32 [B][H][Cp] | k bf16 [B][G][C][N]
 *              KDA:     u f32 [B][H][C][P] (u = b (v - S_{t-1} (a * k))) |
 *                       g f32 [B][H][C][N] | k bf16 [B][G][C][N]
 * cursor     int32 [B][4] = {head, count, last_flush, 0} followed by the
 *            device error word int32 [4] = {code, sequence, 0, 0}.
 *            last_flush is 1 if the last call folded that sequence.
 * read_copy  NULL when read_mode == RS_READ_NONE, else (256-byte sections)
 *              FP8_ROW: e4m3 codes u8 [B][H][P][N] | row scale f32 [B][H][P]
 *              NVFP4:   e2m1 codes u8 [B][H][P][N/2] (element 2i in the low
 *                       nibble) | e4m3 block scales u8 [B][H][P][N/16] |
 *                       matrix scale f32 [B][H]
 * scratch    int32 [B] per-sequence arrival counters (the last CTA of a
 *            sequence to finish a launch advances its cursor).  Zeroed by
 *            rs_create_cache; every launch leaves it zero again.  When
 *            max_draft > 0 a second section follows on a 256-byte boundary:
 *            f32 [B][H][S] per-head coefficient tables that rs_verify writes
 *            and reads within one call (decay weights times key dot products
 *            of the chunkwise form), S = 4C + 4 for Mamba-2 and 8C + 48 for
 *            Gated DeltaNet.
 */
typedef struct {
  void *ckpt, *ring, *cursor, *read_copy, *scratch;
} rs_buffers;

/*
 * Per-call token inputs (device pointers).  Decode: one token per sequence,
 * lead dims [B].  Verify: T draft tokens per sequence, lead dims [B][T].
 *   Mamba-2: x bf16 [..][H][P], dt bf16 [..][H] (already softplus-ed),
 *            A f32 [H], Bm bf16 [..][G][N], Cm bf16 [..][G][N]
 *   GDN:     q bf16 [..][G][N], k bf16 [..][G][N], v bf16 [..][H][P],
 *            g f32 [..][H] (log decay), beta f32 [..][H]
 *   KDA:     as GDN, with g f32 [..][H][N] (log decay per key channel)
 * Pointers of the other kind are ignored and may be NULL.  The decode kernel
 * stages the per-head scalars (dt, A, g, beta) in 16-byte blocks, so each of
 * those arrays must stay readable up to the next 16-byte boundary after its
 * last element (every cudaMalloc or PyTorch allocation is).
 */
typedef struct {
  const void *x, *dt;
  const float *A;
  const void *Bm, *Cm;
  const void *q, *k, *v;
  const float *g, *beta;
} rs_inputs;

typedef struct rs_cache rs_cache;

/* Byte sizes of ckpt, ring, cursor, read_copy, scratch for this config: the
 * high-precision checkpoint plus the per-layer ring of the last L input
 * records that the method keeps instead of a per-token state ("ReplaySSM
 * caches SSM inputs..." (richland.au), "What shipped", the paragraph on
 * unrolling the recurrence: a checkpoint and a 16-record buffer per layer;
 * ai-jitan-hub.com, "ReplaySSMは何をする手法か", first bullet), with room for
 * T_max draft records after the committed ones ("What shipped", the paragraph
 * on speculative decoding: drafts are appended to the input buffer).
 * Pure host call.  RS_ERR_SHAPE / RS_ERR_RANGE for invalid configs,
 * RS_ERR_UNSUPPORTED for valid configs outside the built kernels. */
rs_status rs_query_sizes(const rs_config *cfg, size_t bytes[5]);

/* Bind a config to caller-owned buffers and zero the cursor, the error word
 * and the arrival counters (synchronously, on the legacy default stream):
 * an empty ring whose pointer starts at slot 0 ("ReplaySSM caches SSM
 * inputs..." (richland.au), "What shipped": the buffer holds the inputs since
 * the checkpoint and is addressed through a pointer, like a KV cache).
 * The checkpoint is not touched.  With a read copy, call rs_flush once after
 * the initial checkpoint is written so that the copy is quantised from it. */
rs_status rs_create_cache(const rs_config *cfg, const rs_buffers *bufs, rs_cache **out);

/* Free the handle (never the caller's buffers).  NULL is a no-op. */
void rs_destroy_cache(rs_cache *cache);

/* Standard decode step: one token per sequence, y f32 [B][H][P].
 * Per sequence with count = c records buffered: if c + 1 < L the step is a
 * non-flush step -- it reads the checkpoint (or its read copy) once, computes
 * y_t = S_t q_t from checkpoint + buffer + this token, appends this token's
 * record to slot (head + c) mod C, stores no state and sets count = c + 1.
 * If c + 1 == L it is a flush step: it folds the L records (this token's
 * included) into the checkpoint, writes it once (and refreshes the read
 * copy), sets head = (head + L) mod C, count = 0, last_flush = 1
 * ("ReplaySSM caches SSM inputs..." (richland.au), "What shipped", the
 * paragraph on unrolling the recurrence).
 * RS_ERR_STATE if drafts are pending (rs_verify without rs_commit). */
rs_status rs_decode_step(rs_cache *cache, const rs_inputs *in, float *y, rs_stream stream);

/* Speculative verification of T drafts per sequence (1 <= T <= max_draft):
 * appends the T draft records after the committed ones (GDN: the draft deltas
 * come from a unit-triangular T x T solve) and writes the outputs of all T
 * draft positions, y f32 [B][T][H][P], in the chunkwise form
 * O = S_ckpt Q D + V (W ⊙ (K^T Q)) with D the cumulative decay of each draft
 * position and W the causally masked decay matrix; K^T Q is formed once per
 * group.  The cursor does not move ("ReplaySSM caches SSM inputs..."
 * (richland.au), "What shipped", the paragraphs on speculative decoding).
 * Exactly one rs_commit (or rs_commit_path) must follow before the next
 * decode, verify or flush (RS_ERR_STATE otherwise). */
rs_status rs_verify(rs_cache *cache, int32_t T, const rs_inputs *in, float *y, rs_stream stream);

/* Commit accepted[b] (device int32 [B], 0 <= accepted[b] <= T of the pending
 * verify) drafts of each sequence by advancing its cursor: count += accepted.
 * Rejected draft slots are left to be overwritten.  A sequence whose count
 * reaches L or more is folded in the same launch (all its records), written
 * once, and its cursor moves to head += count, count = 0.  An out-of-range
 * accepted[b] sets RS_DEVERR_ACCEPTED and leaves that sequence unchanged.
 * The accepted prefix is committed by moving the ring pointer, with no state
 * snapshot; records past it are ignored and later overwritten ("ReplaySSM
 * caches SSM inputs..." (richland.au), "What shipped", the paragraph on the
 * second benefit for speculative decoding; ai.warp-studio.com,
 * "推測デコーディングにおける革新と実装詳細").
 * RS_ERR_STATE if no verify is pending, or if the pending drafts are a tree
 * that is not a chain (use rs_commit_path). */
rs_status rs_commit(rs_cache *cache, const int32_t *accepted, rs_stream stream);

/* Tree-shaped speculative verification: as rs_verify, but draft tau continues
 * draft parents[tau] (host int32 [T], parents[tau] in -1..tau-1, -1 = the last
 * committed record; one tree for the whole batch).  Each draft's output is the
 * recurrence along its own path from the committed state: in the chunkwise
 * form, W and the Gated DeltaNet T x T system keep only the records on that
 * path.  Draft tau's record goes to slot head + count + tau as for a chain, so
 * an accepted path need not be contiguous in the buffer ("ReplaySSM：ハイブリッド
 * モデルの高速デコーディングを実現する状態ストレージ再考" (ai.warp-studio.com),
 * "推測デコーディングにおける革新と実装詳細", the sentence on tree-based
 * speculative decoding).  parents = {-1, 0, 1, ..} is rs_verify.
 * RS_ERR_RANGE for an invalid tree; then exactly one rs_commit_path (or, for a
 * chain, rs_commit) must follow. */
rs_status rs_verify_tree(rs_cache *cache, int32_t T, const int32_t *parents, const rs_inputs *in, float *y,
                         rs_stream stream);

/* Commit by index list: per sequence b, path_len[b] (device int32 [B]) drafts
 * path[b][0..path_len[b]) (device int32 [B][T_max]) of the pending verify, a
 * path from the root (path[b][0]'s parent is -1, each next draft's parent the
 * previous one).  Their records are moved to the slots right after the
 * committed records, in path order, then the pointer advances by path_len[b]
 * and the sequence folds if its count reaches L, as in rs_commit.  A list that
 * is not such a path sets RS_DEVERR_ACCEPTED and leaves that sequence
 * unchanged.  Uses the verify-table section of the scratch buffer.
 * RS_ERR_STATE if no verify is pending. */
rs_status rs_commit_path(rs_cache *cache, const int32_t *path_len, const int32_t *path, rs_stream stream);

/* Fold all buffered records of the sequences with seq_mask[b] != 0 (device
 * u8 [B]; NULL = all sequences) into the checkpoint and refresh their read
 * copy; count = 0, last_flush = 1 for them, last_flush = 0 for the others.
 * Use after writing an initial checkpoint (read-copy quantisation), to export
 * the state (after rs_flush the checkpoint is the full state), or at the end
 * of a sequence.  This is the flush of the method -- fold the buffered
 * records into the checkpoint, write it to HBM once, clear the buffer
 * ("ReplaySSM caches SSM inputs..." (richland.au), "What shipped", the
 * paragraph on unrolling the recurrence; ai-jitan-hub.com,
 * "ReplaySSMは何をする手法か", third bullet) -- on demand rather than on fill.
 * RS_ERR_STATE if drafts are pending. */
rs_status rs_flush(rs_cache *cache, const uint8_t *seq_mask, rs_stream stream);

/* Synchronise the stream and read the device error word (RS_DEVERR_*) into
 * *code.  Returns RS_ERR_DEVICE if it is set, RS_OK otherwise.  The word is
 * sticky; a cache with a device error should be re-created. */
rs_status rs_get_device_error(rs_cache *cache, rs_stream stream, int32_t *code);

/* Standard decode step, as rs_decode_step, for callers that cannot allocate
 * device memory -- for example code running inside a server or plugin whose
 * device memory is owned and pre-allocated by someone else.  It takes the
 * config and the caller's buffers directly (no rs_cache handle; bufs->scratch
 * is ignored and may be NULL) and keeps the per-sequence arrival counters in
 * a fixed array of this library (64 KiB on every GPU that loads the library,
 * held until the process exits).  It calls no cudaMalloc, no cudaFree and no
 * allocating library routine.  The paper has no counterpart of this call.
 *   - batch must be <= 16384, else RS_ERR_UNSUPPORTED.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is kept per device and context: after a cudaDeviceReset
 *     (or any other replacement of the device's context) the next call looks
 *     it up again, so make that call, too, before any stream capture.
 *   - Every call clears the counters it uses on `stream`, then launches.  All
 *     calls on a device share the array: calls that overlap on the GPU (other
 *     streams, other caches, other threads) race and must be ordered by the
 *     caller.
 *   - No drafts may be pending on these buffers (rs_verify without rs_commit);
 *     without a handle this call cannot check that. */
rs_status rs_decode_step_noalloc(const rs_config *cfg, const rs_buffers *bufs, const rs_inputs *in, float *y,
                                 rs_stream stream);

/*
 * Host-buffer decode steps.  A pipe serves one cache; it owns two device
 * copies of one step's inputs and of y (allocated by rs_pipe_create, freed
 * by rs_pipe_destroy -- the one exception to caller-owned device memory) and
 * two non-blocking streams for the copies.  rs_pipe_decode_step copies the
 * step's inputs from host memory (rs_inputs with host pointers, layouts as
 * for rs_decode_step; pinned memory for overlap) into one slot, runs
 * rs_decode_step on `stream`, and copies y f32 [B][H][P] back to host_y.
 * Slots alternate, so step t's input copy overlaps step t-1's kernel and step
 * t's y copy overlaps step t+1's kernel; events order every reuse of a slot.
 * The paper has no counterpart of this call.
 *   - Host inputs must stay unchanged, and host_y must not be read, until the
 *     caller has called rs_pipe_sync(pipe, s) and synchronised s.
 *   - Same errors as rs_decode_step (RS_ERR_NULL for a missing host array);
 *     RS_ERR_CUDA for a failed copy or event call.
 *   - Calls on one pipe must come from one host thread in order.
 *   - The pipe keeps a pointer to its cache: destroy the pipe before the cache.
 */
typedef struct rs_pipe rs_pipe;
rs_status rs_pipe_create(rs_cache *cache, rs_pipe **out);
rs_status rs_pipe_decode_step(rs_pipe *pipe, const rs_inputs *host_in, float *host_y, rs_stream stream);
/* Make `stream` wait for every copy the pipe has issued (then synchronise it). */
rs_status rs_pipe_sync(rs_pipe *pipe, rs_stream stream);
/* Waits for the pipe's copies, then frees its device memory, streams and events. */
void rs_pipe_destroy(rs_pipe *pipe);

/*
 * The conventional path, on the same GPU, for comparison: the decoders the
 * method replaces.  Stateless calls (no rs_cache; the caller owns the state);
 * cfg->ring_len is ignored, read_mode must be RS_READ_NONE.
 *
 * rs_conventional_decode_step: one token per sequence, the plain per-token
 * recurrence -- read the whole state, apply the rank-1 update, write the state
 * back, y_t = S_t q_t ("ReplaySSM caches SSM inputs..." (richland.au), "What
 * shipped", the paragraph on why the conventional decode kernel is
 * bandwidth-bound; ai-jitan-hub.com, "何がどれだけ速くなったのか", item 1).
 *   state  f32 [B][H][P][N], updated in place;  y  f32 [B][H][P];
 *   in     as for rs_decode_step.
 * One read and one write of the state per token (2 |S| bytes).
 */
rs_status rs_conventional_decode_step(const rs_config *cfg, float *state, const rs_inputs *in, float *y,
                                      rs_stream stream);

/*
 * Snapshot-per-draft speculative decoding: the state of every sequence lives
 * in one of T_max + 1 slots; rs_snapshot_verify reads the current slot once,
 * runs the T drafts token by token and writes the state after each draft to
 * its own slot (one read and T writes of the state), and rs_snapshot_commit
 * rolls back by selecting the slot of the accepted prefix ("ReplaySSM caches
 * SSM inputs..." (richland.au), "What shipped", the paragraph on the snapshot
 * stored after every draft token; ai-jitan-hub.com, "何がどれだけ速くなったのか",
 * item 2).  cfg->max_draft = T_max in 1..4.
 *   pool   f32 [B][T_max+1][H][P][N]: slot s of sequence b at index (b, s).
 *   slots  int32 [B] (the current slot of each sequence, 0 initially: zero the
 *          array and write the initial state into slot 0), followed by a
 *          device error word int32 [4] = {code, sequence, 0, 0}.
 * rs_snapshot_query_sizes gives bytes[0] = pool, bytes[1] = slots + error word.
 * rs_snapshot_verify: drafts as for rs_verify ([B][T] lead dims), y f32
 * [B][T][H][P]; the state after draft tau goes to slot (cur + 1 + tau) mod
 * (T_max + 1); a slot index out of range sets RS_DEVERR_CURSOR and skips the
 * sequence.  rs_snapshot_commit: accepted int32 [B] in 0..T (the T of the
 * verify it follows) sets cur = (cur + accepted) mod (T_max + 1); out of range
 * sets RS_DEVERR_ACCEPTED and leaves the sequence unchanged.  Read the error
 * word with a device-to-host copy after synchronising.
 */
rs_status rs_snapshot_query_sizes(const rs_config *cfg, size_t bytes[2]);
rs_status rs_snapshot_verify(const rs_config *cfg, float *pool, const int32_t *slots, int32_t T,
                             const rs_inputs *drafts, float *y, rs_stream stream);
rs_status rs_snapshot_commit(const rs_config *cfg, int32_t *slots, const int32_t *accepted, int32_t T,
                             rs_stream stream);

/* Self-test of the bounded wait every kernel uses on its mbarriers: one GPU
 * thread waits on an mbarrier that nothing completes, giving up after
 * limit_us microseconds (1..1000000), with the same primitive and the same
 * give-up rule (time limit or 2^22 polls) as the hot-path kernels.  Writes the
 * outcome to *code_out: RS_DEVERR_TIMEOUT when the wait gave up (the expected
 * result), RS_DEVERR_NONE if the barrier was somehow seen complete.  No GPU
 * fault is involved and the context stays usable.  Synchronises `stream`.
 * RS_ERR_NULL / RS_ERR_RANGE for bad arguments, RS_ERR_CUDA on a CUDA error. */
rs_status rs_selftest_wait_timeout(int32_t limit_us, int32_t *code_out, rs_stream stream);

/* Static description of a status code. */
const char *rs_status_string(rs_status status);

#ifdef __cplusplus
}
#endif

#endif /* REPLAYSSM_H */
