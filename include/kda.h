/*
 * kda.h -- C ABI of the KDA (Kimi Delta Attention) gated delta-rule serving
 * path on one NVIDIA GB300 (sm_103a).
 *
 * The rule, per head, with S a K x V FP32 state:
 *   S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *   o_t = scale * S_t^T q_t
 * with q, k optionally L2-normalised (x / sqrt(sum x^2 + 1e-6)), beta
 * optionally sigmoid(raw beta), and g either given (a log-decay) or the
 * bounded gate g = lower_bound * sigmoid(exp(A_log[h]) * (a + dt_bias[h,:])).
 *
 * The three serving phases and their contracts come from the pages:
 *   prefill  -- chunk_kda in "PR #35197 report: fix(kernel) Fix Helion
 *               small-token prefill bug" (key source snippet of
 *               kda_prefill.py; implementation steps 1-2),
 *   decode   -- validate_packed_decode_inputs in the same report (snippet of
 *               kda_decode.py; implementation step 3),
 *   verify   -- "[KDA] Support Helion MTP verification and harden prefill,
 *               decode" (sglang PR #42857), Modifications: chain/tree
 *               verification with per-candidate state snapshots; its review
 *               thread: commit a partially accepted prefix, then replay.
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller.  The
 *     library allocates nothing, never synchronises and never reads device
 *     memory from the host, so each call can be captured in a CUDA graph and
 *     replayed with new device-resident indices.
 *   - 16-bit token tensors (q, k, v, g, beta, mixed_qkv, a, b, o) are passed
 *     as raw bit patterns (kda_bf16): BF16, or FP16 when kda_dims.dtype is
 *     KDA_DTYPE_F16.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *   - Host-checkable errors return a status and launch nothing.  Buffer
 *     sizes are implied by the sizes passed (B, T, num_seqs, total_tokens,
 *     gb_rows, pool_slots) and cannot be checked through bare pointers: a
 *     buffer shorter than its documented shape is a caller error.  (The
 *     Python binding checks tensor shapes before it calls.)
 *   - Device-resident index errors (a state slot outside [-1, pool_slots), a
 *     tree parent outside [-1, i), a malformed cu_seqlens, an accepted index
 *     >= T) set bits in *err_flag when err_flag is non-NULL and the affected
 *     unit (sequence or request) is skipped; kernels never trap.  The caller
 *     zeroes *err_flag.
 *   - A state slot of -1 marks a padding sequence/request: it is skipped,
 *     its output rows are written as zero and its pool slot is not touched.
 *   - Slots within one call must be distinct (a caller error otherwise).
 *   - This build supports K == V == 128 and HV a multiple of H (grouped
 *     value heads; the pages' packed-decode validator takes HV from the
 *     state shape and the q/k widths from H); other shapes return
 *     KDA_ERR_UNSUPPORTED (non-power-of-two K or V are always rejected, as
 *     the packed-decode validator does).
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kda_bf16; /* raw 16-bit element bits: BF16, or FP16 per kda_dims.dtype */

typedef enum {
  KDA_OK = 0,
  KDA_ERR_NULL_ARG = 1,    /* a required pointer is NULL (e.g. no pool or no indices) */
  KDA_ERR_SHAPE = 2,       /* inconsistent sizes (e.g. gate/beta rows < tokens) */
  KDA_ERR_UNSUPPORTED = 3, /* a shape or option this build does not implement */
  KDA_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required */
  KDA_ERR_CUDA = 5,        /* a CUDA launch failed; see cudaGetLastError */
  KDA_ERR_ALIGNMENT = 6    /* a pointer or stride is not 16-byte aligned */
} kda_status;

/* device-side error bits written to *err_flag */
#define KDA_DEVERR_SLOT 1     /* state slot outside [-1, pool_slots) */
#define KDA_DEVERR_PARENT 2   /* tree parent outside [-1, i) */
#define KDA_DEVERR_SEQLENS 4  /* cu_seqlens not 0 .. total_tokens, non-decreasing */
#define KDA_DEVERR_ACCEPTED 8 /* accepted index >= T */
#define KDA_DEVERR_TIMEOUT 16 /* a kernel's bounded wait on its own copies or
                                 tensor-core work ran out; its unit was not
                                 written back */
#define KDA_DEVERR_INTERMEDIATE 32 /* the chunk-start state buffer holds fewer
                                      records than the call's sequences have
                                      chunks; the states past its end were not
                                      written */

/* element type of the token tensors (q, k, v, g, beta, mixed_qkv, a, b) and
 * of the output o: the "two precisions" of the pages' prefill sweep
 * ("PR #35197 report: fix(kernel) Fix Helion small-token prefill bug",
 * implementation step 4).  States, snapshots, rings and the gate parameters
 * are FP32 either way. */
#define KDA_DTYPE_BF16 0
#define KDA_DTYPE_F16 1

typedef struct {
  int H;  /* q/k heads */
  int HV; /* value heads, a multiple of H: value head h reads q/k head
             h / (HV / H) (grouped value heads); everything else is per
             value head */
  int K;  /* key head dim (128) */
  int V;  /* value head dim (128) */
  int dtype; /* KDA_DTYPE_BF16 (0, so a zeroed struct means BF16) or KDA_DTYPE_F16 */
} kda_dims;

typedef struct {
  const float *A_log;   /* device [HV] FP32, or NULL: g is already a log-decay */
  const float *dt_bias; /* device [HV*K] FP32, or NULL (zero bias) */
  float lower_bound;    /* bound of the gate (e.g. -5); NaN = none.  Required
                           when A_log is given: the unbounded gate formula is
                           not supported (KDA_ERR_UNSUPPORTED). */
  int beta_is_raw;      /* 1: beta <- sigmoid(beta) */
  int use_qk_l2norm;    /* 1: q, k <- x / sqrt(sum x^2 + 1e-6) */
  float scale;          /* output scale, usually K^-0.5 */
} kda_gate;

/* Human-readable name of a status. */
const char *kda_status_string(kda_status s);

/* Bytes of device workspace kda_prefill needs for this call shape (an upper
 * bound over every cu_seqlens with this many sequences and tokens):
 *   align256(4 * num_seqs + 4) + (total_tokens / 64 + num_seqs) * HV * 180352
 *     + num_seqs * HV * 65536
 * (per-sequence flags and a counter, one record per (chunk, head), one
 * staged start state per (sequence, head)).  total_tokens above INT32_MAX (cu_seqlens are int32)
 * gives SIZE_MAX. */
size_t kda_prefill_workspace_size(kda_dims dims, int num_seqs, int64_t total_tokens);

/*
 * Chunked varlen prefill from an indexed initial-state pool (chunk_kda).
 *   q, k          [total_tokens, H, K]    BF16
 *   v             [total_tokens, HV, V]   BF16
 *   g             [gb_rows, HV, K] BF16: gate input a (A_log given) or log-decay.
 *                 The chunk form needs per-token log-decays in [-5.5, 0].  A
 *                 bounded gate with lower_bound < -5.5 (the pages' gate uses
 *                 -5) runs every sequence token by token instead (one
 *                 recurrent step per token, like decode; same outputs, far
 *                 slower for long sequences).  Given log-decays (A_log NULL)
 *                 are checked on the device: a sequence with any value
 *                 outside [-5.5, 0] (or NaN) is left out of the chunk form
 *                 and computed token by token after it.  Decode and verify
 *                 take any log-decay.
 *   beta          [gb_rows, HV]    BF16: raw beta (beta_is_raw) or beta
 *   gb_rows       >= total_tokens (else KDA_ERR_SHAPE).  Rows past
 *                 total_tokens are CUDA-graph bucket padding and never read.
 *   state_pool    [pool_slots, HV, V, K] FP32, updated in place: sequence n
 *                 starts from slot state_idx[n] and its final state is
 *                 written back there.  NULL pool or indices: KDA_ERR_NULL_ARG.
 *   state_idx     [num_seqs] int32 (device)
 *   cu_seqlens    [num_seqs+1] int32 (device) or NULL for the fixed layout
 *                 (num_seqs equal lengths, total_tokens % num_seqs == 0).
 *                 A sequence of length 0 leaves its state unchanged.
 *   o             [total_tokens, HV, V] BF16 (round to nearest even)
 *   intermediate  NULL, or [sum_n ceil(T_n/64), HV, V, K] FP32: the state at
 *                 the start of every 64-token chunk of every sequence,
 *                 sequence-major.  The records of a padding sequence (slot
 *                 -1) are not written.
 *   intermediate_chunks
 *                 the number of [HV, V, K] records `intermediate` holds
 *                 (ignored when it is NULL).  The chunk count depends on
 *                 cu_seqlens, which only the device reads: records past this
 *                 capacity are not written and KDA_DEVERR_INTERMEDIATE is set.
 *   workspace     >= kda_prefill_workspace_size(...) bytes, 256-byte aligned.
 * T = 1 takes the same kernels as any other length.  The first call on each
 * device sets the kernels' shared-memory limits (cudaFuncSetAttribute); make
 * it before capturing calls into a CUDA graph.
 *
 * Schedule: everything runs on `stream`: the per-sequence decay check (given
 * log-decays only), the chunk transform, then the state pass.  When
 * 8 * HV * num_seqs does not exceed the SM count, each (sequence, head)
 * chain of chunks runs as two CTAs per value slice; the second starts behind
 * a chunk whose chain product is certainly left out (its map is zero, or too
 * small for the bounded state to matter), which it finds within 32 chunks
 * or else starts from the sequence's first chunk.  Results are bit for bit
 * those of a single CTA per slice.  With more (sequence, head, slice) chains
 * than SMs, the pass runs one CTA per SM, each claiming the next chain from
 * a counter in the workspace whenever it is free; there the chains run in
 * two parts too when the sequences average 1024 tokens or more.  The
 * pass is a programmatic dependent launch of the transform: its CTAs may
 * start on SMs the transform has left and wait for the transform before
 * reading its records.  The transform reads the token rows by TMA, through
 * tensor maps encoded on the host for each call.
 */
kda_status kda_prefill(kda_dims dims, kda_gate gate, const kda_bf16 *q, const kda_bf16 *k,
                       const kda_bf16 *v, const kda_bf16 *g, const kda_bf16 *beta,
                       int64_t gb_rows, float *state_pool, int pool_slots,
                       const int32_t *state_idx, const int32_t *cu_seqlens, int num_seqs,
                       int64_t total_tokens, kda_bf16 *o, float *intermediate,
                       int64_t intermediate_chunks, void *workspace, size_t workspace_bytes,
                       int32_t *err_flag, void *stream);

/*
 * Packed single-token decode (one token per request), state updated in place.
 *   mixed_qkv     [B, row_stride] BF16, each row [q (H*K) | k (H*K) | v (HV*V)];
 *                 row_stride >= 2*H*K + HV*V and a multiple of 8 elements.
 *   a             [B, HV*K] BF16 gate input (or log-decay when A_log is NULL)
 *   b             [B, HV]   BF16 raw beta (or beta)
 *   state_pool    [pool_slots, HV, V, K] FP32, slot state_idx[r] read and
 *                 written in place.
 *   o             [B, HV, V] BF16
 */
kda_status kda_decode_packed(kda_dims dims, kda_gate gate, const kda_bf16 *mixed_qkv,
                             int64_t row_stride, const kda_bf16 *a, const kda_bf16 *b, int B,
                             float *state_pool, int pool_slots, const int32_t *state_idx,
                             kda_bf16 *o, int32_t *err_flag, void *stream);

/*
 * Speculative chain verify: T draft tokens per request, request-major rows
 * (row r*T + i is draft token i of request r) in mixed_qkv, a and b, laid out
 * as for decode.  The pool is READ ONLY.
 *   o             [B, T, HV, V] BF16
 *   snapshots     [B, T, HV, V, K] FP32: snapshots[r][i] is the state after
 *                 draft token i (the per-candidate state snapshot).
 */
kda_status kda_verify_chain(kda_dims dims, kda_gate gate, const kda_bf16 *mixed_qkv,
                            int64_t row_stride, const kda_bf16 *a, const kda_bf16 *b, int B,
                            int T, const float *state_pool, int pool_slots,
                            const int32_t *state_idx, kda_bf16 *o, float *snapshots,
                            int32_t *err_flag, void *stream);

/*
 * Speculative tree verify: as kda_verify_chain, but node i of request r
 * continues from node parent_idx[r*T+i] (parent < i; -1 = the pool state).
 *   parent_idx    [B, T] int32 (device)
 */
kda_status kda_verify_tree(kda_dims dims, kda_gate gate, const kda_bf16 *mixed_qkv,
                           int64_t row_stride, const kda_bf16 *a, const kda_bf16 *b, int B,
                           int T, const int32_t *parent_idx, const float *state_pool,
                           int pool_slots, const int32_t *state_idx, kda_bf16 *o,
                           float *snapshots, int32_t *err_flag, void *stream);

/*
 * Commit of the accepted draft prefix: for each request r with
 * accepted[r] >= 0, state_pool[state_idx[r]] <- snapshots[r][accepted[r]]
 * (a bit-exact copy).  accepted[r] = -1 keeps the pool state.
 *   snapshots     [B, T, HV, V, K] FP32 as written by verify
 *   accepted      [B] int32 (device)
 */
kda_status kda_commit(kda_dims dims, const float *snapshots, int B, int T,
                      const int32_t *accepted, float *state_pool, int pool_slots,
                      const int32_t *state_idx, int32_t *err_flag, void *stream);

/*
 * kda_prefill without a caller-provided workspace.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory: a host whose whole device memory already belongs
 * to its own pools, code issuing the call while a CUDA graph is being
 * captured (cudaMalloc is not allowed there), or a plugin that only receives
 * tensors through this ABI and has no allocator.  It allocates nothing
 * (no cudaMalloc, no cudaFree, no allocating library call).
 *
 * Its scratch is a file-scope static device array of
 * KDA_PREFILL_STATIC_SCRATCH_BYTES that every GPU loading the library keeps
 * until the process exits.  Calls whose workspace need
 * (kda_prefill_workspace_size) exceeds it return KDA_ERR_WORKSPACE and
 * launch nothing.  The rule is
 *   align256(4 * num_seqs + 4) + (total_tokens / 64 + num_seqs) * HV * 180352
 *       + num_seqs * HV * 65536 <= KDA_PREFILL_STATIC_SCRATCH_BYTES,
 * so one sequence at 16 heads takes at most 2943 tokens (46 records per
 * head); the 1 x 4096 shape at 16 heads needs 65 and is refused.
 *
 * The first call on each device looks up the array's device address with
 * that device current; make that first call before any stream capture.
 * All calls in the process share the one array (per device): calls whose
 * work overlaps on the GPU race on it, so serialise them (one stream, or
 * events).  The per-sequence flags at the start of the scratch are cleared
 * by each call that uses them, and every other scratch byte a call reads it
 * has written itself, so nothing is left to clear between calls.  Arguments
 * and results are exactly those of kda_prefill.
 */
#define KDA_PREFILL_STATIC_SCRATCH_BYTES ((size_t)128 << 20)
kda_status kda_prefill_noalloc(kda_dims dims, kda_gate gate, const kda_bf16 *q,
                               const kda_bf16 *k, const kda_bf16 *v, const kda_bf16 *g,
                               const kda_bf16 *beta, int64_t gb_rows, float *state_pool,
                               int pool_slots, const int32_t *state_idx,
                               const int32_t *cu_seqlens, int num_seqs, int64_t total_tokens,
                               kda_bf16 *o, float *intermediate, int64_t intermediate_chunks,
                               int32_t *err_flag, void *stream);

/*
 * ReplaySSM verify ("[KDA] Default GLM-5-Next spec verify to the CuTe DSL KDA
 * kernel #42905", Results: the "ReplaySSM rings" columns beside the
 * "intermediate-state snapshots" ones; left out of scope in "[KDA] Support
 * Helion MTP verification and harden prefill, decode", Motivation): chain
 * verify that keeps no per-token state snapshots.  Outputs o
 * are those of kda_verify_chain, bit for bit; instead of snapshots, each draft
 * token's folded inputs (k-hat, exp(g), v, beta) are recorded in `ring`, and
 * kda_commit_replay replays the accepted prefix onto the pool.  The state is
 * read once and nothing state-sized is written, so the call moves about
 * 1/7 of the bytes of the snapshot verify at T = 6.
 *   ring          device, kda_replay_ring_bytes(dims, B, T) bytes, 16-byte
 *                 aligned; layout [B, T, HV, 388] FP32 (k-hat [128], exp(g)
 *                 [128], v [128], beta, 3 unused), owned by the caller and
 *                 read by the next kda_commit_replay.
 * Other arguments and errors as kda_verify_chain.  The pool is not written.
 */
size_t kda_replay_ring_bytes(kda_dims dims, int B, int T);
kda_status kda_verify_chain_replay(kda_dims dims, kda_gate gate, const kda_bf16 *mixed_qkv,
                                   int64_t row_stride, const kda_bf16 *a, const kda_bf16 *b,
                                   int B, int T, const float *state_pool, int pool_slots,
                                   const int32_t *state_idx, kda_bf16 *o, float *ring,
                                   int32_t *err_flag, void *stream);

/*
 * Commit for ReplaySSM verify: for each request r with accepted[r] >= 0, the
 * pool state is advanced through draft tokens 0..accepted[r] from `ring`,
 * with the verify's own arithmetic, so the new pool state equals, bit for
 * bit, the snapshot kda_verify_chain would have written after that token.
 * accepted[r] = -1 keeps the pool state; accepted[r] >= T sets
 * KDA_DEVERR_ACCEPTED and skips the request; slot -1 is skipped.
 *   ring          as written by kda_verify_chain_replay with the same B, T
 *   accepted      [B] int32 (device)
 */
kda_status kda_commit_replay(kda_dims dims, const float *ring, int B, int T,
                             const int32_t *accepted, float *state_pool, int pool_slots,
                             const int32_t *state_idx, int32_t *err_flag, void *stream);

/*
 * Profiling aid (not part of the pages' contract): per-kernel timing of every
 * entry point.  After kda_set_stage_events(ev) with three cudaEvent_t
 * handles passed as void*, each later call records ev[0] on its stream before
 * its first kernel and ev[2] after its last; kda_prefill records ev[1]
 * between its chunk-transform and state-pass kernels, the single-kernel entry
 * points record ev[1] together with ev[2].  Under stream capture they become
 * external event nodes, so every replay of the graph records them.  A NULL
 * entry is not recorded; a NULL array clears the setting, which is
 * process-wide and not meant for concurrent callers.
 */
void kda_set_stage_events(void *const *events);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
