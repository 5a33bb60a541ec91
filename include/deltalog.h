/*
 * deltalog.h — C ABI of libdeltalog: deferred materialisation of the recurrent
 * state in linear-attention decoding (DeltaLog), for Gated DeltaNet (GDN),
 * Kimi Delta Attention (KDA) and RWKV6, on one GB300 GPU (sm_103a).
 *
 * What it computes.  Each slot (a request or a branch) and head holds a
 * recurrent state S in R^{d_v x d_k}, stored value-major: S[v][i], row = value
 * index, contiguous along d_k.  One decode token updates it and reads it out:
 *
 *   GDN    u_t = beta_t (v_t - alpha_t S_{t-1} k_t)        alpha_t = exp(g_t), one per head
 *          S_t = alpha_t S_{t-1} + u_t k_t^T,   o_t = scale * S_t q_t
 *   KDA    S_t = S_{t-1} Diag(alpha_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *          (alpha_t = exp(g_t) one per key channel),       o_t = scale * S_t q_t
 *   RWKV6  S_t = S_{t-1} Diag(w_t) + v_t k_t^T              w_t = exp(g_t) per key channel
 *          o_t = scale * (S_{t-1} r_t + (sum_i r_i bonus_i k_i) v_t)
 *
 * (The RWKV6 rule is the key-major rule Z_t = Diag(w_t) Z_{t-1} + k_t v_t^T,
 * o_t = r_t^T (Z_{t-1} + Diag(bonus) k_t v_t^T) with S = Z^T.)  The operator
 * traits follow the DeltaLog page ("DeltaLog: Deferred Materialization of
 * Recurrent States for Linear Attention Decoding"), section "Kernel
 * implementation": GDN has a head-scalar decay and the delta-rule correction,
 * KDA a per-key decay and the delta rule, RWKV6 a per-key decay and raw-value
 * updates.
 *
 * How.  Section "Methodology — Base + Log" of the same page: the state is a
 * dense base S̄ (history up to the last merge) plus a bounded log of compressed
 * update factors with cumulative log-decay metadata.  For M-1 tokens a step
 * reads S̄ but does not rewrite it; it appends its factors (value side u_t,
 * or v_t for RWKV6; key side k_t; log-decay Λ_t) to the log.  Every M-th token
 * of a slot is a merge step: the same kernel also writes base + replayed log
 * back into S̄ and clears the log.  M = 1 is eager decoding.  The results are
 * those of the eager rules above, up to floating-point rounding order.
 * Section "Kernel implementation — Staged execution": per step a ReplayPrep
 * kernel computes the per slot-head coefficients once, and a value-tiled
 * AppendDecode kernel streams S̄ in value-row tiles, each with its shard of
 * the value-side log.
 *
 * Forking.  The Flide page ("같은 맥락에서 여러 판단을 빠르게 처리하는 Flide",
 * section "Research method step by step", second step) runs a shared context
 * once, saves the final recurrent state, and starts every question branch from
 * its own request's saved state by indexing it.  dl_fork does this: a branch
 * points at the source's dense base (no copy) and gets a copy of its log; the
 * branch writes a private base at its first merge.  A slot whose base is
 * indexed by another slot is frozen until every such branch has merged.
 *
 * Conventions for every call below.
 *   - Slot ids (int32) are HOST arrays; each call validates them on the host
 *     before anything is enqueued: every id in [0, num_slots), no id twice in
 *     one call.  An invalid argument returns DL_EINVAL and changes nothing;
 *     a frozen slot returns DL_EBUSY and changes nothing.
 *   - Every tensor pointer is a DEVICE pointer on the context's device,
 *     16-byte aligned, C-contiguous, owned by the caller, and must stay valid
 *     until the work enqueued on the context's stream has run.  Rows of
 *     per-token tensors follow the order of the slot list.
 *   - Work is enqueued asynchronously on the context's CUDA stream; calls that
 *     return host data (dl_get_meta, dl_get_timing, dl_sync) synchronise it.
 *   - bf16 tensors are raw IEEE bfloat16 (uint16 storage).
 *   - Errors: a CUDA error returns DL_ECUDA; a device-side error (a kernel
 *     gave up a bounded wait) is recorded in a device status word and returned
 *     as DL_EDEVICE by the next synchronising call.  Both are sticky for the
 *     context.  dl_last_error() gives a one-line description.  No exception
 *     crosses this interface.
 *   - A context is not thread-safe; use one per host thread.
 */
#ifndef DELTALOG_H
#define DELTALOG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DL_ABI_VERSION 2

typedef enum dl_status {
    DL_OK = 0,
    DL_EINVAL = 1,       /* bad argument (range, duplicate, shape, alignment, NULL) */
    DL_ENOMEM = 2,       /* device or host allocation failed                        */
    DL_ECUDA = 3,        /* a CUDA runtime call failed                              */
    DL_EBUSY = 4,        /* slot frozen: its base is indexed by a forked branch     */
    DL_EDEVICE = 5,      /* a kernel reported an error through the status word      */
    DL_EUNSUPPORTED = 6  /* configuration this library has no kernel for            */
} dl_status;

typedef enum dl_op { DL_GDN = 0, DL_KDA = 1, DL_RWKV6 = 2 } dl_op;

typedef struct dl_config {
    int32_t op;              /* dl_op                                                   */
    int32_t num_slots;       /* state slots (requests + branches), >= 1                 */
    int32_t num_heads;       /* H, >= 1                                                 */
    int32_t d_k;             /* key dimension: 64 or 128                                */
    int32_t d_v;             /* value dimension: equal to d_k in this library           */
    int32_t merge_interval;  /* M in [1, 32]; 1 = eager (every step merges)             */
    int32_t out_bf16;        /* 1: o is bf16; 0: o is fp32                              */
    float scale;             /* output scale (1.0 for the decode workloads)             */
    int32_t staging;         /* DL_STAGE_FUSED (0, default) or DL_STAGE_KERNELS (1)     */
} dl_config;

/* How a dl_step runs the two stages of the DeltaLog page's "Kernel
 * implementation" section.  FUSED: one kernel; a warp of each AppendDecode CTA
 * is the ReplayPrep stage and computes each slot-head's coefficients from the
 * unit's inputs in shared memory.  KERNELS: a ReplayPrep kernel writes the
 * coefficient blocks to HBM scratch, then AppendDecode (launched as its
 * programmatic dependent) reads them.  Both compute the same values. */
#define DL_STAGE_FUSED 0
#define DL_STAGE_KERNELS 1

/* ------------------------------------------------------------------------ */
/* Host bookkeeping (no GPU needed).  This is the slot table every context   */
/* keeps: per slot the log length n (0 <= n < M), the slot whose dense base  */
/* it reads (base_of), and how many other slots index its base (refs).       */
/* The rules are those stated for dl_step / dl_fork / dl_set_state /          */
/* dl_merge below; the table is exposed so that callers (and tests) can plan */
/* and check them without a device.                                           */
/* ------------------------------------------------------------------------ */
typedef struct dl_table dl_table;

/* Create a table of num_slots slots, all with n = 0 and base_of[s] = s. */
dl_status dl_table_create(int32_t num_slots, int32_t merge_interval, dl_table **out);
void dl_table_destroy(dl_table *t);
/* Advance the listed slots by one token.  If plan != NULL it receives, per
 * slot in argument order, 4 int32: slot, base read this step, n before the
 * step, 1 if this step is the slot's merge step.  A merge step resets n to 0
 * and makes the slot own its base (base_of[s] = s). */
dl_status dl_table_step(dl_table *t, const int32_t *slots, int32_t n, int32_t *plan);
/* Validate an eager step: each slot must own its base and have n == 0. */
dl_status dl_table_step_eager(dl_table *t, const int32_t *slots, int32_t n);
/* Fork: each dst releases whatever base it indexed, then indexes src's base and
 * takes src's log length.  dst must not contain src nor a frozen slot. */
dl_status dl_table_fork(dl_table *t, int32_t src, const int32_t *dsts, int32_t n);
/* Re-seed or merge: each slot releases its base reference, owns its base, n = 0. */
dl_status dl_table_reset(dl_table *t, const int32_t *slots, int32_t n);
/* Validate a slot list (range, duplicates). */
dl_status dl_table_check(const dl_table *t, const int32_t *slots, int32_t n);
/* Copy out the table; any pointer may be NULL.  Arrays have num_slots entries. */
dl_status dl_table_get(const dl_table *t, int32_t *n_log, int32_t *base_of, int32_t *refs);

/* ------------------------------------------------------------------------ */
/* Device context                                                            */
/* ------------------------------------------------------------------------ */
typedef struct dl_ctx dl_ctx;

/* The base + log representation of the DeltaLog page, "Methodology — Base +
 * Log".  Allocate, on the current CUDA device, the dense bases S̄ [num_slots, H, d_v,
 * d_k] fp32 (zeroed), the bounded log (value side [num_slots, H, M-1, d_v]
 * fp32, or bf16 for RWKV6; keys [num_slots, H, M-1, d_k] bf16; cumulative
 * log-decay [num_slots, H, M-1] or [num_slots, H, M-1, d_k] fp32), the slot
 * table on host and device, and per-step scratch.  stream is a cudaStream_t
 * (NULL = legacy default stream).  On failure *out is NULL. */
dl_status dl_create(const dl_config *cfg, void *stream, dl_ctx **out);
/* Synchronise the stream, free everything.  NULL is accepted. */
dl_status dl_destroy(dl_ctx *ctx);
/* Use another stream for subsequent calls (the caller orders the two). */
dl_status dl_set_stream(dl_ctx *ctx, void *stream);

/* Load initial states: S [n, H, d_v, d_k] fp32 device -> S̄ of the listed slots;
 * their logs are emptied (n = 0) and they own their bases again. */
dl_status dl_set_state(dl_ctx *ctx, const int32_t *slots, int32_t n, const float *S);

/* RWKV6 only: the per-head bonus, [H, d_k] fp32 device (copied). */
dl_status dl_set_bonus(dl_ctx *ctx, const float *bonus);

/* Flide-style fork of src into each dst (see above): no dense state is copied;
 * only src's log rows (n_src entries) are copied into each dst's log. */
dl_status dl_fork(dl_ctx *ctx, int32_t src, const int32_t *dsts, int32_t n);

/* One decode token for each listed slot: the step of the DeltaLog page,
 * "Methodology — Base + Log", run as in "Kernel implementation" (n slots, row
 * i of every tensor is slot slots[i]):
 *   q (r for RWKV6), k   [n, H, d_k] bf16
 *   v                    [n, H, d_v] bf16
 *   g                    [n, H] fp32 (GDN) or [n, H, d_k] fp32 (KDA, RWKV6): log-decay
 *   beta                 [n, H] fp32 (GDN, KDA); ignored for RWKV6 (may be NULL)
 *   o                    [n, H, d_v] bf16 or fp32 (dl_config.out_bf16), written
 * Runs the ReplayPrep and AppendDecode stages (dl_config.staging; the merge is
 * fused for the slots whose log is full).  With M = 1 every step is the eager
 * update; when every listed slot reads its own base it runs as the EagerStep
 * kernel (as dl_step_eager), else through the merge path.  A frozen slot in the
 * list returns DL_EBUSY. */
dl_status dl_step(dl_ctx *ctx, const int32_t *slots, int32_t n,
                  const void *q, const void *k, const void *v,
                  const float *g, const float *beta, void *o);

/* The dl_step operation with every tensor in HOST memory (pinned memory
 * gives full copy speed): same arguments and results as dl_step.  The call copies the inputs to
 * device staging buffers owned by the context, runs dl_step, copies o back
 * and synchronises the stream before returning. */
dl_status dl_step_host(dl_ctx *ctx, const int32_t *slots, int32_t n,
                       const void *q, const void *k, const void *v,
                       const float *g, const float *beta, void *o);

/* T dl_step operations (DeltaLog page, "Methodology — Base + Log") for the
 * same n slots from HOST buffers: q, k [T, n, H, d_k]
 * bf16, v [T, n, H, d_v] bf16, g [T, n, H] or [T, n, H, d_k] fp32, beta
 * [T, n, H] fp32 (NULL for RWKV6), o [T, n, H, d_v] (written); token t is
 * slice t of each.  Equivalent to T calls of dl_step_host, but the copies
 * overlap the computation: tokens travel in groups (one copy per tensor; small
 * tensors are grouped until a copy reaches 2 MiB, up to 8 tokens and 64 MiB of
 * staging a group), and while a group's tokens run on the
 * context's stream an upload stream copies the next groups' inputs into the
 * next of four device staging sets (a set is reused once its group's outputs
 * are back) and a download stream copies earlier groups' outputs back.  When
 * every listed slot owns its base with an empty log and T is a multiple of M
 * (M >= 2), each group is a whole decode window of M tokens, run as a window
 * graph (dl_window_create) captured on its staging set: the same kernels and
 * results, one graph launch per M tokens.  These windows are captured at the
 * first such call for a slot list and kept until a call with another list
 * (their staging takes at most 2 GiB; larger batches use the per-token path).
 * The staging sets, windows and streams are owned by the context and made on
 * first use.  Host memory must be pinned for the copies to run
 * asynchronously.  Returns once every output is in host memory; on an error
 * (for example DL_EBUSY for a frozen slot at the first token) the tokens
 * before it have been decoded and copied back. */
dl_status dl_decode_host(dl_ctx *ctx, const int32_t *slots, int32_t n, int32_t T,
                         const void *q, const void *k, const void *v,
                         const float *g, const float *beta, void *o);

/* The eager dense step, one kernel that reads and rewrites the whole state of
 * every listed slot-head (the "state-update tax" of the DeltaLog page, section
 * "Problem").  Same arguments as dl_step; each slot must own its base and
 * have an empty log (true for every slot of an M = 1 context), else DL_EINVAL. */
dl_status dl_step_eager(dl_ctx *ctx, const int32_t *slots, int32_t n,
                        const void *q, const void *k, const void *v,
                        const float *g, const float *beta, void *o);

/* The merge of the DeltaLog page, "Methodology — Base + Log", forced now:
 * S̄[s] <- base + replayed log, log emptied, slot owns its base.  Frozen slots
 * return DL_EBUSY. */
dl_status dl_merge(dl_ctx *ctx, const int32_t *slots, int32_t n);

/* Materialise the logical state of each listed slot (base + replayed log,
 * DeltaLog page, "Methodology — Base + Log") into S_out [n, H, d_v, d_k] fp32
 * device.  Does not change the context. */
dl_status dl_read_state(dl_ctx *ctx, const int32_t *slots, int32_t n, float *S_out);

/* Synchronise and copy the device slot table: n_log and base_of are host
 * arrays of num_slots int32 (either may be NULL).  Returns DL_EDEVICE if the
 * device table disagrees with the host table. */
dl_status dl_get_meta(dl_ctx *ctx, int32_t *n_log, int32_t *base_of);

/* Chunked prefill: feed T context tokens to each listed slot in one call and
 * leave the state after the last token in the slot's dense base (log empty).
 * Flide page, "Research method step by step", second step: the shared
 * context is processed once and its final state saved before branches fork.
 * Inputs are token-major: q (r for RWKV6), k [T, n, H, d_k] bf16, v
 * [T, n, H, d_v] bf16, g [T, n, H] (GDN) or [T, n, H, d_k] (KDA, RWKV6) fp32,
 * beta [T, n, H] fp32 (NULL for RWKV6, which needs dl_set_bonus first);
 * o [T, n, H, d_v] receives every token's output, or is NULL.  q, k, v (and g
 * for KDA, RWKV6) must be 16-byte aligned, the other tensors aligned to their
 * element size (else DL_EINVAL).  Every slot must own its base and have an
 * empty log (else DL_EINVAL).  Tokens are
 * processed C = 32 at a time: one pass over the state per chunk computes all
 * chunk outputs (base + log algebra with the chunk as the log, forward
 * substitution for the delta-rule factors), and the state is rewritten once
 * per chunk. */
dl_status dl_prefill(dl_ctx *ctx, const int32_t *slots, int32_t n, int32_t T,
                     const void *q, const void *k, const void *v,
                     const float *g, const float *beta, void *o);

/* Prefix checkpoints (Flide page, "Research method step by step", fourth step:
 * a growing agent trace resumes from a checkpoint saved at a matching prefix).
 * A checkpoint is the exact DeltaLog representation of a slot: the dense base
 * it reads (fp32 [H, d_v, d_k]), its log rows (value side, keys, log-decays)
 * and its log length, so that a restored slot continues bit for bit as the
 * saved one would have.  dl_checkpoint_bytes gives the size of one slot's
 * checkpoint; buffers are device memory owned by the caller, 16-byte aligned,
 * slot i at offset i * dl_checkpoint_bytes. */
int64_t dl_checkpoint_bytes(const dl_ctx *ctx);
dl_status dl_checkpoint_save(dl_ctx *ctx, const int32_t *slots, int32_t n, void *buf);
/* Restore: each listed slot becomes the saved state (it owns a private copy of
 * the saved base).  Frozen slots return DL_EBUSY.  Synchronises the stream
 * (the saved log lengths are read back to update the host table). */
dl_status dl_checkpoint_load(dl_ctx *ctx, const int32_t *slots, int32_t n, const void *buf);

/* CUDA-graph decode loop (Flide page, third step: prepared CUDA graphs cut the
 * per-step launch cost).  A window is one merge interval — M decode tokens —
 * of a fixed batch, captured once into a CUDA graph and replayed.  Every
 * listed slot must own its base and have an empty log when the window is
 * created and whenever it is launched; the window's last token is the merge,
 * so windows can be launched back to back.  q, k are [M, n, H, d_k] bf16, v
 * [M, n, H, d_v] bf16, g [M, n, H] or [M, n, H, d_k] fp32, beta [M, n, H] fp32
 * (NULL for RWKV6), o [M, n, H, d_v]: token j of a launch reads slice j of each
 * input and writes slice j of o; the graph keeps these device pointers, and the
 * caller refills the buffers between launches (in stream order).  The inputs
 * must not overlap o: a step may read its inputs while the step before it is
 * still writing its outputs.  n <= 1024.
 * dl_window_launch validates the slots, enqueues the graph on the context's
 * stream and advances the slot table by M tokens. */
typedef struct dl_window dl_window;
dl_status dl_window_create(dl_ctx *ctx, const int32_t *slots, int32_t n,
                           const void *q, const void *k, const void *v,
                           const float *g, const float *beta, void *o, dl_window **out);
dl_status dl_window_launch(dl_window *w);
dl_status dl_window_destroy(dl_window *w);

/* Ragged decode window (the same Flide step, for batches whose active set
 * changes from token to token, e.g. branches of different lengths).  Captured
 * once for up to n_max rows per token; the M per-token slot lists and counts
 * live in device memory and are refreshed from host memory by the graph's
 * first node at every launch, so one graph serves any active sets.  Token j
 * reads rows 0 .. counts[j]-1 of slice j of q, k [M, n_max, H, d_k] bf16,
 * v [M, n_max, H, d_v] bf16, g [M, n_max, H] or [M, n_max, H, d_k] fp32, beta
 * [M, n_max, H] fp32 (NULL for RWKV6) and writes the same rows of o
 * [M, n_max, H, d_v]; rows at or past counts[j] are neither read nor written
 * (a token may have no rows at all).  Unlike the fixed window, slots may have
 * any log length and may index a fork source's base.
 * dl_window_launch_ragged takes the slot ids as a host array [M][n_max] (row
 * i of token j at j*n_max + i) and the counts [M].  It validates every token
 * first (ids in range, no duplicates within a token, no fork source that
 * branches still index: DL_EINVAL / DL_EBUSY, and then nothing is launched),
 * plans the M tokens on the host slot table, and enqueues the graph on the
 * context's stream.  A launch waits for the previous launch of the same
 * window to finish before it rewrites the host plan.  n_max <= min(1024,
 * num_slots). */
dl_status dl_window_create_ragged(dl_ctx *ctx, int32_t n_max,
                                  const void *q, const void *k, const void *v,
                                  const float *g, const float *beta, void *o, dl_window **out);
dl_status dl_window_launch_ragged(dl_window *w, const int32_t *slots, const int32_t *counts);

/* ------------------------------------------------------------------------ */
/* A decode step that allocates no device memory.                            */
/* The paper has no counterpart: this entry point exists for callers that    */
/* cannot let a library call cudaMalloc while they run — engines that reserve */
/* almost all device memory for their own pools at start-up, code whose       */
/* device buffers must all come from the caller's own allocator, and loops    */
/* that cannot afford the device synchronisation an allocation can cause.    */
/* The caller owns every buffer (layouts as in dl_create); the coefficient    */
/* scratch of the step lives in a static device array of the library.        */
/* ------------------------------------------------------------------------ */
#define DL_NOALLOC_SCRATCH_FLOATS (4 * 1024 * 1024)   /* 16 MiB of fp32 scratch */

typedef struct dl_state_view {
    float *Sbar;         /* [num_slots, H, d_v, d_k] fp32 dense bases                     */
    void *alog;          /* [num_slots, H, max(M-1,1), d_v] fp32 (bf16 for RWKV6), value log */
    uint16_t *klog;      /* [num_slots, H, max(M-1,1), d_k] bf16 key log                    */
    float *Llog;         /* [num_slots, H, max(M-1,1)] (GDN) or [..., d_k] fp32 log-decays  */
    int32_t *n_log;      /* [num_slots] device slot table: log lengths (written)            */
    int32_t *base_of;    /* [num_slots] device slot table: base indices (written)           */
    const float *bonus;  /* [H, d_k] fp32 (RWKV6), else NULL                                */
} dl_state_view;

/* One token for n slots on caller-owned state, without allocating.  `plan` is
 * the host array that dl_table_step returns for this step ([n][4]: slot, base
 * read, log length before the step, merge flag); the caller keeps a dl_table
 * (host memory) for its slots.  Tensors and stream are as in dl_step.  The
 * step's coefficient scratch must fit DL_NOALLOC_SCRATCH_FLOATS (n * H * CB
 * floats; CB grows with M and, for KDA/RWKV6, with M * d_k); larger steps are
 * refused with DL_EINVAL — split them over several calls.  The scratch is one
 * array shared by every call and keeps the last call's contents: within a
 * call every coefficient used is written first, but calls that overlap on
 * the GPU race, so order them on one stream.  The first call on a device does
 * a one-time set-up with that device current (it looks up the device
 * addresses of the scratch and the status word, and sets kernel shared-memory
 * limits); make it before any stream capture.  If errbuf != NULL it receives a one-line reason
 * for a non-DL_OK status (at most errlen bytes, NUL-terminated).  The step
 * always runs as two kernels (the scratch holds the coefficient blocks that
 * pass between them); cfg->staging is not used.
 * Checked on the host before anything is enqueued (DL_EINVAL, nothing runs):
 * the plan's ids and log lengths are in range and its merge flags agree with
 * them, no slot appears twice, and no row reads the base of a slot that
 * merges in the same call (dl_table_step never plans that: a fork source is
 * frozen); q, k, v (and g for KDA / RWKV6), Sbar, alog, klog, the per-key
 * Llog and bonus are 16-byte aligned, the other pointers aligned to their
 * element size.
 * Device-side errors (a bounded wait in a kernel gave up) are recorded in one
 * static status word per device, which starts at zero and keeps the first
 * code until dl_noalloc_sync reads it. */
dl_status dl_step_noalloc(const dl_config *cfg, const dl_state_view *st,
                          const int32_t *plan, int32_t n,
                          const void *q, const void *k, const void *v,
                          const float *g, const float *beta, void *o,
                          void *stream, char *errbuf, int32_t errlen);

/* Companion of dl_step_noalloc (no paper counterpart either; allocates
 * nothing): synchronise `stream`, then read the current device's static status
 * word.  DL_OK if no dl_step_noalloc call since the last dl_noalloc_sync
 * reported a device-side error.  Otherwise DL_EDEVICE, *device_code (if not
 * NULL) receives the code, errbuf a one-line reason, and the word is cleared:
 * the outputs and state written by the calls since the last dl_noalloc_sync
 * must not be trusted.  A CUDA error returns DL_ECUDA. */
dl_status dl_noalloc_sync(void *stream, int32_t *device_code, char *errbuf, int32_t errlen);

/* Synchronise the stream and report any CUDA or device-side error. */
dl_status dl_sync(dl_ctx *ctx);

/* Kernel timing: when enabled, every launch is bracketed by CUDA events on the
 * context's stream (this disables launch overlap between ReplayPrep and
 * AppendDecode).  dl_get_timing synchronises and returns, per kernel kind
 * (0 ReplayPrep, 1 AppendDecode, 2 EagerStep, 3 Merge/ReadState), the summed
 * milliseconds and the number of launches since timing was enabled. */
dl_status dl_set_timing(dl_ctx *ctx, int32_t enable);
dl_status dl_get_timing(dl_ctx *ctx, double *ms, int64_t *launches);

/* One-line text for the last error of ctx (never NULL). */
const char *dl_last_error(const dl_ctx *ctx);
const char *dl_status_str(dl_status s);
int32_t dl_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DELTALOG_H */
