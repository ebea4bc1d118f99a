/*
 * replayssm.h -- C ABI of the ReplaySSM decode library for one Mamba-2 layer (sm_103a).
 *
 * Source of the method: the NVIDIA Developer blog post "ReplaySSM: Rethinking State
 * Storage for Faster Hybrid-Model Decoding". Each call below names the section of that
 * page that defines the operation. The page's displayed formulas were lost; the
 * operation is stated here in full.
 *
 * Model (per sequence b and head h; head h reads group g = h / (H/G)):
 *     a_t = exp(dt_t * A_h)
 *     h_t = a_t * h_{t-1} + dt_t * x_t B_t^T          (P x N state)
 *     y_t = h_t C_t + D_h * x_t
 * ("Why SSM layers can become a decoding bottleneck".) ReplaySSM keeps h as an FP32
 * checkpoint h0 plus a ring of the input records (x_s, B_s, dt_s) appended since the
 * checkpoint ("How ReplaySSM represents the state"). With the n records numbered
 * s = 1..k (k = n + 1 including the current token):
 *     y_k = Gamma_k (h0 C_k) + sum_s gamma(k,s) dt_s (B_s . C_k) x_s + D x_k
 *     gamma(k,s) = exp(A sum_{r=s+1..k} dt_r),  Gamma_k = exp(A sum_{r=1..k} dt_r)
 *
 * Conventions for every call:
 *  - Ownership: all device memory (workspace, inputs, outputs, A, D) belongs to the
 *    caller and is passed as plain device pointers. The library owns only the small
 *    host handle returned by replay_alloc. It allocates no device memory.
 *  - Streams: `stream` is a cudaStream_t (NULL = the legacy default stream). Every
 *    device call is asynchronous on that stream and launches on no other stream. The calls
 *    on one store must run in the order they are made: issue them on one stream, or order
 *    the streams with events. Two consecutive replay_step calls on one stream may overlap on
 *    the GPU (a store with a read copy starts a step's first kernel while the previous
 *    step's last one finishes; the results are those of running them one after the other).
 *  - Return codes: REPLAY_OK, or a negative REPLAY_E* code for errors found on the host
 *    (nothing is launched then). Errors found on the device never trap: they set bits of
 *    the store's status word (REPLAY_DEV_*), read with replay_status.
 *  - Layouts: dense, row-major, last index fastest:
 *      x [batch][H][P], B and C [batch][G][N], dt [batch][H], y [batch][H][P]  (one token)
 *      x [batch][T][H][P], B and C [batch][T][G][N], dt [batch][T][H],
 *      y [batch][T][H][P]                                                     (T drafts)
 *      A, D [H] FP32 on the device; states [batch][H][P][N] FP32.
 *    x, B, C and dt are FP32 or bf16 (replay_config.in_dtype); y is always FP32.
 *    x, B, C and state buffers must be 16-byte aligned (REPLAY_EBADARG otherwise).
 *  - Limits: batch <= 65535 (REPLAY_ECAPACITY otherwise).
 *  - Supported shapes: headdim P = 64 and dstate N in {64, 128, 256}; H a multiple of G;
 *    ring capacity (see replay_layout) at most 64 records.
 */
#ifndef REPLAYSSM_H
#define REPLAYSSM_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 3: the workspace holds two step plans and at least two coefficient blocks (replay_layout
 * sizes changed); status bit REPLAY_DEV_COPY_TIMEOUT.
 * 4: replay_config.checkpoint_format (an FP16 checkpoint with stochastic rounding beside a
 * separate read copy). */
#define REPLAY_ABI_VERSION 4

/* element types of x, B, C, dt and of the ring records */
#define REPLAY_F32 0
#define REPLAY_BF16 1

/* low-precision read copy of the checkpoint */
#define REPLAY_RC_NONE 0
#define REPLAY_RC_BF16 1     /* bf16, round to nearest even */
#define REPLAY_RC_FP8E4M3 2  /* OCP E4M3, RNE, saturating; FP32 scale absmax/448 per (b, h) */
#define REPLAY_RC_FP16 3     /* IEEE binary16. As a separate copy: round to nearest even. As the
                              * shared checkpoint (shared_checkpoint = 1): stochastic rounding,
                              * saturating at +-65504 -- the FP16 recurrence checkpoint with
                              * stochastic rounding named in the post's section "State
                              * quantization". The draw for element e (row-major in P x N) of
                              * slab s = b*H + h, written by the sequence's flush number `epoch`
                              * (meta.w), is number d = (epoch*batch*H + s)*P*N + e: the 16-bit
                              * chunk d mod 4 (most significant first) of output d / 4 of the
                              * splitmix64 generator seeded 0x2545F4914F6CDD1D; u = chunk / 2^16,
                              * and the value rounds away from zero iff u is below its distance
                              * from the lower neighbour over the neighbours' spacing.
                              * dstate 64 and 128 only. */
#define REPLAY_RC_NVFP4 4    /* NVFP4: E2M1 codes, one E4M3 scale per 16 consecutive elements of
                              * a row, one FP32 scale per (b, h) slab: s_g = absmax / 2688 (1 if
                              * the slab is zero); s_b = e4m3(block_absmax / (6 s_g)); e = s_b s_g;
                              * q = e2m1(h / e) (RNE, saturating at 6; 0 where e = 0), each step
                              * one FP32 operation. The post's sections "Benefit 3" and "State
                              * quantization" read this format. dstate 128 only. Code layout of
                              * a row (64 bytes): quarter u (0..3) of block b (columns 16b+4u ..
                              * 16b+4u+3) is the 2-byte unit at byte 16u + 2b; the unit's byte 0
                              * holds columns 16b+4u (slot A) and 16b+4u+2 (slot B), byte 1
                              * columns 16b+4u+1 (A) and 16b+4u+3 (B); slot A keeps the code's
                              * sign in bit 7 and magnitude in bits 3..1, slot B the sign in bit
                              * 0 and magnitude in bits 6..4 (E2M1 code = sign * 8 + magnitude).
                              * Block scales are [P][N/16] row-major. */

/* format of the recurrence checkpoint (replay_config.checkpoint_format) */
#define REPLAY_CKPT_F32 0     /* FP32 */
#define REPLAY_CKPT_F16_SR 1  /* IEEE binary16 written by stochastic rounding (the draws and the
                               * rounding of REPLAY_RC_FP16 as a shared checkpoint, numbered by
                               * the same epoch), with a separate read copy cast independently
                               * from the same FP32 values: the FP16 recurrence with NVFP4 (or
                               * bf16, E4M3) reads of the post's sections "Benefit 3" and "State
                               * quantization". Needs read_copy BF16, FP8E4M3 or NVFP4,
                               * shared_checkpoint 0, dstate <= 128. */

/* host return codes */
#define REPLAY_OK 0
#define REPLAY_EBADARG (-1)      /* null pointer, bad count, store/shape mismatch */
#define REPLAY_EUNSUPPORTED (-2) /* shape or dtype this build has no kernel for */
#define REPLAY_ECAPACITY (-3)    /* ring capacity or draft count beyond the configured maximum */
#define REPLAY_ECUDA (-4)        /* a CUDA call or launch failed */

/* device status bits (sticky until cleared by replay_status or replay_reset) */
#define REPLAY_DEV_BAD_META 1    /* a sequence's ring metadata was out of range: its y is NaN */
#define REPLAY_DEV_BAD_ACCEPT 2  /* commit with accept < 0 or > drafts pending: not applied */
#define REPLAY_DEV_COPY_TIMEOUT 4 /* a step CTA's bulk copy of its checkpoint slab did not land
                                     within its wait limit (1 s): that slab's y is NaN and its
                                     ring and checkpoint are left as they were */

typedef struct replay_config {
  int batch;        /* sequences */
  int nheads;       /* H */
  int headdim;      /* P */
  int dstate;       /* N */
  int ngroups;      /* G: B and C are shared by the H/G heads of a group */
  int window_L;     /* records folded per flush (the window) */
  int max_draft_T;  /* largest T passed to replay_verify; 0 = no speculative verify */
  int in_dtype;     /* REPLAY_F32 or REPLAY_BF16 */
  int read_copy;    /* REPLAY_RC_* */
  int shared_checkpoint; /* 0: FP32 checkpoint + derived read copy ("Benefit 3", separate
                          * precisions). 1: the low-precision copy IS the checkpoint: flushes
                          * start from it and write only it, no FP32 checkpoint is kept (the
                          * "shared" low-precision checkpoint the pages compare against: rounded
                          * once per window, and fed back). Needs read_copy != REPLAY_RC_NONE. */
  int checkpoint_format; /* REPLAY_CKPT_F32 (0) or REPLAY_CKPT_F16_SR: the recurrence checkpoint
                          * h0 is kept in FP16, rounded stochastically at every write; flushes
                          * start from it, and non-flush steps and verify read the read copy. */
} replay_config;

/* Byte offsets of the regions inside the caller's workspace (each 256-byte aligned).
 *   h0     FP32 checkpoint            [batch][H][P][N]      (FP16 with REPLAY_CKPT_F16_SR)
 *   rc     read copy (bf16/E4M3/FP16) [batch][H][P][N]      (0 bytes without a copy)
 *          NVFP4 codes                [batch][H][P][N/2] bytes (row layout: REPLAY_RC_NVFP4)
 *   scale  FP32 slab scale            [batch][H]            (E4M3 and NVFP4 only)
 *   bscale NVFP4 E4M3 block scales    [batch][H][P][N/16]   (NVFP4 only)
 *   xbuf   ring of x records          [batch][H][cap][P]    (in_dtype)
 *   bbuf   ring of B records          [batch][G][cap][N]    (in_dtype)
 *   dtbuf  ring of dt records         [batch][H][cap]       (in_dtype)
 *   meta   per sequence int32 x4      {start, n, pending, epoch}: records live in ring slots
 *          (start + s) mod cap, s < n; `pending` drafts sit beyond them after a verify;
 *          `epoch` numbers the sequence's next checkpoint write (the load/reset write is
 *          number 0, so it is 1 after a load and grows by one at each flush)
 *   arrive per sequence int32 counter (internal; zero between calls)
 *   status int32 device status word (REPLAY_DEV_* bits)
 *   plan   2 x per sequence int32 x4  (internal, per step: the pointer the step runs on;
 *          consecutive steps alternate between the two)
 *   coef   FP32 [batch][H][max(T+1,2)][cap+1] (internal, per call: record weights and
 *          decays; T = max_draft_T; a step uses one of the region's first two blocks of
 *          batch x H x (cap+1) values, alternating, a verify the region as [batch][H][T+1][cap+1])
 * cap = window_L when max_draft_T == 0, else window_L + 2*max_draft_T - 1: the most
 * records a sequence can hold (window_L - 1 + T committed before a verify folds them)
 * plus T drafts written beyond them while those are being folded. */
typedef struct replay_layout {
  size_t h0, rc, scale, bscale, xbuf, bbuf, dtbuf, meta, arrive, status, plan, coef;
  size_t total;  /* workspace bytes */
  int cap;       /* ring capacity in records */
} replay_layout;

typedef struct replay_store replay_store; /* opaque host handle */

/* Validate a config and compute its workspace layout. No CUDA call. */
int replay_layout_of(const replay_config* cfg, replay_layout* out);

/* Workspace bytes the caller must allocate for cfg. No CUDA call. */
int replay_store_bytes(const replay_config* cfg, size_t* bytes);

/* Bind a store to a caller-owned device workspace of at least replay_store_bytes bytes
 * (256-byte aligned) and to the per-head A (< 0) and D vectors, which must stay valid
 * while the store is used. Launches a reset on `stream`: h0 = 0 and every ring empty.
 * The handle is freed with replay_free. */
int replay_alloc(const replay_config* cfg, void* workspace, size_t workspace_bytes,
                 const float* A, const float* D, void* stream, replay_store** out);

/* Free the host handle. The workspace stays the caller's. */
int replay_free(replay_store* st);

/* Reset sequences: h0 = 0, ring emptied, pending drafts dropped. seq_mask is a device
 * int32 [batch] (nonzero = reset) or NULL for all sequences; with NULL the status word is
 * cleared as well. */
int replay_reset(replay_store* st, const int* seq_mask, void* stream);

/* Import a state for every sequence: h0 = h (FP32 [batch][H][P][N], device), rings
 * emptied, and the read copy recast from h. Used to resume, or to hand over a state
 * computed elsewhere (e.g. by prefill). */
int replay_load_state(replay_store* st, const float* h, void* stream);

/* Write the current state of every sequence -- h0 with the committed records folded in
 * (the unrolled window of "How ReplaySSM represents the state") -- to h_out (FP32
 * [batch][H][P][N], device). The store is not modified. */
int replay_export_state(replay_store* st, float* h_out, void* stream);

/* One decode token for every sequence ("How ReplaySSM represents the state";
 * "Benefit 1: Reduce state memory traffic"). With k = n + 1:
 *  - k < window_L (non-flush step): y from checkpoint + records + the current inputs;
 *    the record (x, B, dt) is appended to the ring; no state is written.
 *  - k >= window_L (flush step): the k records (this token's included) are folded into
 *    h0, which is written once (and cast into the read copy, if any); y is read from the
 *    new FP32 checkpoint; the ring is emptied.
 * Non-flush steps read the read copy when one is configured; flushes always start from
 * the FP32 checkpoint ("Benefit 3"). Drafts pending from a verify are dropped. A sequence
 * with out-of-range ring metadata gets NaN outputs and REPLAY_DEV_BAD_META; a CTA whose bulk
 * copy of its state does not land within 1 s gives its slabs NaN outputs, leaves their state
 * unchanged and sets REPLAY_DEV_COPY_TIMEOUT (read with replay_status). */
int replay_step(replay_store* st, const void* x, const void* B, const void* C,
                const void* dt, float* y, void* stream);

/* Speculative verify of T drafts (1 <= T <= max_draft_T) for every sequence ("Benefit 2:
 * Simplify rollback and speed up verification"). If the sequence holds n >= window_L
 * committed records they are folded into h0 first (a flush of committed records only).
 * Then y[b][j] (j = 0..T-1) is the output the model would give after decoding drafts
 * 0..j in order, computed from checkpoint + committed records + drafts without forming a
 * state. The drafts' records are written to the ring beyond the committed ones; the
 * commit pointer does not move until replay_commit. */
int replay_verify(replay_store* st, int T, const void* x, const void* B, const void* C,
                  const void* dt, float* y, void* stream);

/* Commit the first accept[b] drafts of the last verify of each sequence (device int32
 * [batch], 0 <= accept[b] <= T): the ring pointer advances over them; the other drafts are
 * left beyond the pointer, ignored, and overwritten by the next append ("Benefit 2").
 * Nothing is restored. An out-of-range accept sets REPLAY_DEV_BAD_ACCEPT and commits
 * nothing for that sequence. */
int replay_commit(replay_store* st, const int* accept, void* stream);

/* Fold every sequence's committed records into h0 now (n > 0), writing h0 (and the read
 * copy) once and emptying the ring; pending drafts are dropped. */
int replay_flush(replay_store* st, void* stream);

/* Copy the device status word to *status_out (host), synchronising `stream`; clear it
 * afterwards if `clear` is nonzero. */
int replay_status(replay_store* st, int* status_out, int clear, void* stream);

/* replay_step for callers that must not allocate device memory. The paper has no
 * counterpart: this is a deployment aid of this library.
 * Who needs it: callers that cannot call cudaMalloc (or anything that allocates) when they
 * decode -- an engine plugin handed only its input, output and state buffers, a process
 * whose device memory is pre-claimed by another framework's pool, code running while a
 * stream is captured. replay_step's scratch memory -- the per-sequence arrival counters, the
 * step's plan and the per-head record coefficients, all only alive during one step -- is kept
 * by this call in a fixed array inside the library (the store's arrive, plan and coef regions
 * are not touched); otherwise it is replay_step: same arguments, kernels, results, errors.
 * Limits and rules:
 *  - batch <= REPLAY_STATIC_MAX_BATCH and batch * nheads * (cap + 1) <= REPLAY_STATIC_MAX_COEFS
 *    (cap: replay_layout), else REPLAY_ECAPACITY and nothing is launched. The array
 *    (16 KiB of counters, 64 KiB of plans, 4 MiB of coefficients) exists on every GPU that
 *    loads the library, until the process exits.
 *  - The first call on a device looks up the array's device address (once per device, with
 *    that device current); make that first call before any stream capture. The address is
 *    kept for the life of the process: after cudaDeviceReset (or any teardown of the device's
 *    primary context) this call must not be used again in that process.
 *  - Each call zeroes the counters it uses (an asynchronous memset on `stream`, no
 *    allocation) before its launch. All calls share the one array, so calls on the same
 *    device that can overlap on the GPU (different streams, no ordering between them) race
 *    and give wrong results: order them, or use replay_step. */
#define REPLAY_STATIC_MAX_BATCH 4096
#define REPLAY_STATIC_MAX_COEFS 1048576
int replay_step_static_scratch(replay_store* st, const void* x, const void* B, const void* C,
                               const void* dt, float* y, void* stream);

/* ---------------------------------------------------------------------------------
 * Conventional baselines ("Why SSM layers can become a decoding bottleneck"; "Rollback
 * for speculative decoding"). They use the config's shape fields and in_dtype only.
 * --------------------------------------------------------------------------------- */

/* Load-update-store decode step: state <- a * state + dt x B^T, y = state C + D x, state
 * stored back. state is [batch][H][P][N], FP32 (state_dtype REPLAY_F32) or bf16
 * (REPLAY_BF16: FP32 arithmetic, stored with round-to-nearest-even). */
int conv_step(const replay_config* cfg, void* state, int state_dtype, const float* A,
              const float* D, const void* x, const void* B, const void* C, const void* dt,
              float* y, void* stream);

/* Snapshot-per-draft verify: one read of snapshot slot cur[b], T updates, snapshot j
 * (after draft j) written to slot (cur[b] + 1 + j) mod (T + 1), outputs y[b][j].
 * snaps is FP32 [batch][T+1][H][P][N]; cur is device int32 [batch]. */
int conv_verify_snapshot(const replay_config* cfg, int T, float* snaps, const int* cur,
                         const float* A, const float* D, const void* x, const void* B,
                         const void* C, const void* dt, float* y, void* stream);

/* Pick the snapshot of the accepted prefix: cur[b] <- (cur[b] + accept[b]) mod (T + 1).
 * An accept outside 0..T leaves cur[b] and sets bit REPLAY_DEV_BAD_ACCEPT of *status
 * (device int32, may be NULL). */
int conv_commit(int batch, int T, int* cur, const int* accept, int* status, void* stream);

/* Text for a return code; library version. */
const char* replay_strerror(int code);
int replay_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* REPLAYSSM_H */
