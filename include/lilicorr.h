/*
 * lilicorr.h -- C ABI of the GB300 (sm_103a) LiLiCorr draft-time rerank path.
 *
 * The path (LiLiCorr: Lightweight Likelihood Correlation of Parallel Drafts for
 * Speculative Decoding, Sec. 3.2, Sec. 3.5 and App. A):
 *   a1  per drafted slot, one read of the vocabulary logits gives the full-vocabulary
 *       log-partition and the top-K candidates            (App. A "Serving"; serving PR
 *       "[Spec] Add LiLiCorr ...", section "Why the custom kernels")
 *   a2  each candidate becomes a node: embedding + drafter hidden + confidence MLP over
 *       five scalars + slot and rank tables                (Sec. 3.2; App. A "Architecture")
 *   a3  a two-layer bidirectional transformer over the (B-1) x K lattice (App. A)
 *   a4  target fusion, out/in/anchor heads, unit norm, matching scores
 *       phi(s,k,k') = sigma * cos(o_{s,k}, i_{s+1,k'})     (Sec. 3.2, Eq. 1)
 *   a5  greedy commit c_s = argmax_k phi(s-1, c_{s-1}, k)  (Sec. 3.5, Eq. 8)
 *
 * Conventions for every entry point:
 *   - Device pointers are caller-owned CUDA device memory, contiguous, row-major.
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy default stream.
 *     Device entry points only enqueue work on `stream`: they never allocate and never
 *     synchronise, so a call can be captured in a CUDA graph.
 *   - All arguments are checked on the host before any launch; a violation returns an
 *     error status and launches nothing.  A failed launch returns LILICORR_ERR_CUDA
 *     (lilicorr_last_error() has the CUDA message).  No device-side trap is used.
 *   - Logits are finite or -inf (no NaN, no +inf); each row holds a finite value.
 *   - Index arguments use 0-based slots for arrays; drafted slot s (1..B-1) is stored
 *     at index s-1 of [.., B-1, ..] arrays.
 */
#ifndef LILICORR_H_
#define LILICORR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LILICORR_OK = 0,
  LILICORR_ERR_INVALID_ARG = 1,     /* a size, pointer or alignment is out of contract   */
  LILICORR_ERR_UNSUPPORTED = 2,     /* legal but not built (e.g. K > 32, f32 weights)     */
  LILICORR_ERR_WEIGHTS_MISSING = 3, /* a required head tensor is absent                   */
  LILICORR_ERR_WEIGHTS_SURPLUS = 4, /* an unknown head tensor was given                   */
  LILICORR_ERR_WEIGHTS_SHAPE = 5,   /* a head tensor's shape or dtype disagrees with dims */
  LILICORR_ERR_CUDA = 6,            /* a CUDA call failed                                 */
  LILICORR_ERR_WORKSPACE = 7,       /* workspace missing, too small or misaligned         */
  LILICORR_ERR_DEVICE = 8           /* a kernel reported a device-side error (timeout)    */
} lilicorr_status;

typedef enum { LILICORR_F32 = 0, LILICORR_BF16 = 1 } lilicorr_dtype;

/* Head geometry (LiLiCorr App. A, Table 4).  Constraints checked at weight creation:
 * hidden % 64 == 0; heads divides hidden with hidden/heads in {32, 64, 128};
 * ffn % 64 == 0; d_e % 32 == 0 and d_e <= 256; 2 <= B_max <= 64; 1 <= K_max <= 32;
 * V >= 1.  sigma is the cosine scale (8.0 in Table 4), rms_eps the RMSNorm epsilon. */
typedef struct {
  int32_t layers, hidden, heads, ffn, d_e, B_max, K_max;
  int64_t V;
  float sigma;
  float rms_eps;
} lilicorr_dims;

/* One named head tensor in host memory.  Weights are bf16 bit patterns (dtype must be
 * LILICORR_BF16), row-major, with exactly these shapes (H hidden, F ffn, E d_e):
 *   embed [V,H]  slot_table [B_max-1,H]  rank_table [K_max,H]
 *   conf.w1 [H,5] conf.b1 [H] conf.w2 [H,H] conf.b2 [H]
 *   layers.{l}.norm1 [H] .in_proj_w [3H,H] .in_proj_b [3H] .out_proj_w [H,H]
 *     .out_proj_b [H] .dist_bias [heads,2*B_max-3] .same_bias [heads] .norm2 [H]
 *     .ffn.w1 [F,H] .ffn.b1 [F] .ffn.w2 [H,F] .ffn.b2 [H]
 *   fuse.w [H,3H] fuse.b [H]  head_out.w [E,H] head_out.b [E]
 *   head_in.w [E,H] head_in.b [E]  head_anchor.w [E,H] head_anchor.b [E]
 * The in_proj layout is nn.MultiheadAttention's packed [q; k; v] (serving PR, design
 * note 3).  The host data is copied; the caller may free it after the call returns. */
typedef struct {
  const char* name;
  const void* host_data;
  lilicorr_dtype dtype;
  int32_t ndim;
  int64_t shape[4];
} lilicorr_tensor;

typedef struct lilicorr_weights lilicorr_weights; /* opaque, library-owned device arena */

/* Validate the tensor set against dims and copy it into a device arena on `device`.
 * Missing names -> WEIGHTS_MISSING, unknown names -> WEIGHTS_SURPLUS (both directions
 * are refused, as the serving PR's loader does, design note 4), wrong shape or dtype ->
 * WEIGHTS_SHAPE.  Synchronous; allocates device memory (the only call that does). */
lilicorr_status lilicorr_weights_create(const lilicorr_dims* dims,
                                        const lilicorr_tensor* tensors, int32_t n,
                                        int device, lilicorr_weights** out);
void lilicorr_weights_destroy(lilicorr_weights* w);
/* Copy of the dims the weights were created with. */
lilicorr_status lilicorr_weights_dims(const lilicorr_weights* w, lilicorr_dims* out);

/* Bytes of device workspace lilicorr_rerank needs for this call shape (0 on bad args). */
size_t lilicorr_workspace_bytes(const lilicorr_weights* w, int64_t batch, int32_t B,
                                int32_t K);

/* Optional extra outputs of lilicorr_rerank (any member may be NULL; the struct
 * pointer itself may be NULL).  S = (B-1)*K lattice nodes per block, slot-major. */
typedef struct {
  int32_t* choice;      /* [batch,B-1]      committed candidate index per slot          */
  int32_t* cand_id;     /* [batch,B-1,K]    top-K token ids, (logit desc, id asc)        */
  float* cand_logit;    /* [batch,B-1,K]    their logits, exactly widened to f32         */
  float* lse;           /* [batch,B-1]      natural-log full-vocabulary log-partition    */
  float* pair_scores;   /* [batch,B-1,K,K]  [p,k,k'] = phi(p,k,k'); pair 0 row>0 = -inf */
  float* nodes;         /* [batch,S,H]      node vectors (encoder input)                 */
  float* hidden;        /* [batch,S,H]      encoder output                               */
  float* out_vec;       /* [batch,S,d_e]    unit out vectors                             */
  float* in_vec;        /* [batch,S,d_e]    unit in vectors                              */
  float* anchor_vec;    /* [batch,d_e]      unit anchor out vector o_0                   */
} lilicorr_taps;

/* The whole rerank on `stream`.
 *   logits       [batch,B,V] of ldtype (F32 or BF16); row 0 of each block (the anchor
 *                position) is not read.  Rows need only element alignment.
 *   B            2 <= B <= dims.B_max;  V == dims.V;  1 <= K <= min(dims.K_max, V)
 *   slot_hidden  nullable [batch,B,H] bf16: drafter hidden per slot (row 0 unused)
 *   target_state nullable [batch,H] bf16: projected target state t
 *                (both 16-byte aligned, else LILICORR_ERR_INVALID_ARG)
 *   anchor_ids   nullable [batch] int32: written to tokens[:,0] (else -1)
 *   tokens       [batch,B] int32 out;  path_score [batch,B-1] f32 out:
 *                path_score[b,s-1] = phi(s-1, c_{s-1}, c_s)
 *   workspace    device memory of >= lilicorr_workspace_bytes(...) bytes, 256-B aligned;
 *                its contents need no initialisation and are clobbered.
 * Concurrent calls must not share a workspace. */
lilicorr_status lilicorr_rerank(const lilicorr_weights* w, const void* logits,
                                lilicorr_dtype ldtype, int64_t batch, int32_t B, int64_t V,
                                int32_t K, const void* slot_hidden, const void* target_state,
                                const int32_t* anchor_ids, int32_t* tokens, float* path_score,
                                const lilicorr_taps* taps, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Host-memory form of lilicorr_rerank: logits, slot_hidden, target_state and anchor_ids
 * are host pointers (pinned memory makes the copies asynchronous), tokens and
 * path_score are host outputs.  The inputs are copied to device staging inside
 * `workspace` (size from lilicorr_workspace_bytes_host); the logits travel in up to 8
 * chunks of blocks on an internal copy stream, rows 1..B-1 only (row 0 is never read),
 * and each chunk is reranked on `stream` as soon as it has landed, so compute hides
 * under the copy.  The outputs are copied back and the call returns after synchronising
 * `stream`.  Results are identical to lilicorr_rerank on the whole batch. */
size_t lilicorr_workspace_bytes_host(const lilicorr_weights* w, int64_t batch, int32_t B,
                                     int32_t K, lilicorr_dtype ldtype);
lilicorr_status lilicorr_rerank_host(const lilicorr_weights* w, const void* logits_host,
                                     lilicorr_dtype ldtype, int64_t batch, int32_t B,
                                     int64_t V, int32_t K, const void* slot_hidden_host,
                                     const void* target_state_host,
                                     const int32_t* anchor_ids_host, int32_t* tokens_host,
                                     float* path_score_host, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* Step a1 alone (serving PR, "Why the custom kernels": exact per-row top-k plus the
 * full-vocabulary log-partition from one pass over the logits).  For every block b and
 * drafted slot s = 1..B-1 it reads row logits[b,s,:] once and writes
 *   cand_id[b,s-1,:K] int32, cand_logit[b,s-1,:K] f32 (logit desc, token id asc) and
 *   lse[b,s-1] = log sum_v exp(logits[b,s,v]) (f32, natural log).
 * 1 <= K <= min(32, V); one row is under 2 GiB.  Workspace: lilicorr_topk_lse_workspace_bytes
 * (may be 0). */
size_t lilicorr_topk_lse_workspace_bytes(int64_t batch, int32_t B, int64_t V, int32_t K,
                                         lilicorr_dtype ldtype);
lilicorr_status lilicorr_topk_lse(const void* logits, lilicorr_dtype ldtype, int64_t batch,
                                  int32_t B, int64_t V, int32_t K, int32_t* cand_id,
                                  float* cand_logit, float* lse, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* lilicorr_topk_lse without a workspace (the paper has no counterpart: this is a
 * convenience of this library).  Some callers cannot allocate device memory when they
 * run the logit pass: a serving loop whose memory is all handed to its own pool and that
 * forbids further cudaMalloc, code running while a CUDA graph is being captured (where
 * allocation is not allowed), or a plain C host that has no device allocator at all.
 * This form computes exactly what lilicorr_topk_lse computes, but keeps the split-row
 * scratch in a 4 MiB array compiled into the library (every GPU that loads the library
 * holds it until the process exits); it allocates nothing and frees nothing.
 *   - A shape that needs more scratch than 4 MiB returns LILICORR_ERR_WORKSPACE with a
 *     message in lilicorr_last_error(); use lilicorr_topk_lse for it.
 *   - The first call on each device looks up the scratch's device address (the library
 *     caches it per device); make that first call before any stream capture.  A
 *     cudaDeviceReset (or any re-creation of the device's primary context) invalidates
 *     the cached address and the library's per-device kernel settings: reload the library
 *     after one.
 *   - All calls share the one scratch array, which keeps the previous call's contents
 *     (the parts that must start at zero are cleared by every call).  Calls whose work
 *     overlaps on the GPU (different streams, or host threads without ordering) race on
 *     it: serialise them. */
lilicorr_status lilicorr_topk_lse_noalloc(const void* logits, lilicorr_dtype ldtype,
                                          int64_t batch, int32_t B, int64_t V, int32_t K,
                                          int32_t* cand_id, float* cand_logit, float* lse,
                                          void* stream);

/* Vocabulary-sharded form of step a1 (serving PR, "Why the custom kernels" and its
 * tensor-parallel notes: with the LM head sharded over the vocabulary, each rank reduces
 * its slice to a per-row top-K and a partial log-partition, one packed all-gather moves
 * K*(4+4) + 8 bytes per row, and a merge finishes the row).  On one GPU the ranks are
 * emulated by slices of one logits tensor.
 *   lilicorr_topk_lse_shard_record_bytes(K): bytes of one row record,
 *     {f32 m2, f32 s, f32 v[K], int32 id[K]} = K*8 + 8 (m2 = max * log2(e) of the
 *     slice, s = sum 2^(x*log2(e) - m2); v / id the slice's top-K by (value desc, id asc),
 *     ids global; a slice with fewer than K values pads with (-inf, INT32_MAX)).
 *   lilicorr_topk_lse_shard: logits points at element [0,0,0] of this shard's slice;
 *     rows are row_stride >= V_shard elements apart (V_total for a slice of a whole
 *     tensor); candidate ids are id_offset + column.  Writes records[batch*(B-1)] for the
 *     drafted rows 1..B-1 (row 0 is not read).  Workspace as lilicorr_topk_lse at V_shard.
 *   lilicorr_topk_lse_merge: records [n_shards][rows] -> cand_id, cand_logit [rows,K] and
 *     lse [rows] exactly as lilicorr_topk_lse on the unsharded rows (ids and logits
 *     identical; lse to f32 rounding).
 * Errors: LILICORR_ERR_INVALID_ARG for null pointers, sizes out of range (1 <= K <= 32,
 * id_offset + V_shard < 2^31 - 1), misaligned logits or records; LILICORR_ERR_WORKSPACE;
 * LILICORR_ERR_CUDA. */
size_t lilicorr_topk_lse_shard_record_bytes(int32_t K);
lilicorr_status lilicorr_topk_lse_shard(const void* logits, lilicorr_dtype ldtype,
                                        int64_t batch, int32_t B, int64_t V_shard,
                                        int64_t row_stride, int64_t id_offset, int32_t K,
                                        void* records, void* workspace, size_t workspace_bytes,
                                        void* stream);
lilicorr_status lilicorr_topk_lse_merge(const void* records, int32_t n_shards, int64_t rows,
                                        int32_t K, int32_t* cand_id, float* cand_logit,
                                        float* lse, void* stream);

/* The drafter's vocabulary projection fused with step a1 (the serving write-up's list of
 * follow-ons: the LM-head projection, 0.49 ms of a block in LiLiCorr Table 3, feeds the
 * top-K / log-partition pass directly, so the [rows, V] logits never reach HBM):
 *   logit[r,v] = sum_d hidden[r,d] * w_lm[v,d]     (bf16 operands, f32 accumulation)
 *   cand_id / cand_logit [rows,K] = the K largest logits of row r by (value desc, id asc),
 *   lse [rows] = log sum_v exp(logit[r,v]).
 * hidden [rows, D] and w_lm [V, D] are bf16, row-major, 16-byte aligned; D % 64 == 0;
 * 1 <= K <= min(32, V); V < 2^31 - 256.  The logits are f32 sums of exact bf16 products
 * in the tensor cores' order, so two logits closer than their rounding may swap places
 * against an exact reference.  Workspace: lilicorr_lm_head_workspace_bytes (0 for
 * unsupported sizes), 256-byte aligned; it holds one vocabulary-shard record per row and
 * vocabulary range, merged as lilicorr_topk_lse_merge does.
 * Errors: LILICORR_ERR_INVALID_ARG (null pointers, sizes, alignment),
 * LILICORR_ERR_WORKSPACE, LILICORR_ERR_CUDA. */
size_t lilicorr_lm_head_workspace_bytes(int64_t rows, int64_t V, int32_t D, int32_t K);
lilicorr_status lilicorr_lm_head_topk_lse(const void* hidden, const void* w_lm, int64_t rows,
                                          int64_t V, int32_t D, int32_t K, int32_t* cand_id,
                                          float* cand_logit, float* lse, void* workspace,
                                          size_t workspace_bytes, void* stream);

/* Step a5 alone (LiLiCorr Sec. 3.5, Eq. 8) on given scores pair_scores [batch,B-1,K,K]
 * (layout as in lilicorr_taps).  c_1 = argmax_k pair_scores[b,0,0,k]; c_s = argmax_k
 * pair_scores[b,s-1,c_{s-1},k]; ties go to the lowest k (serving PR: the Triton
 * argmax breaks ties toward the lower index).  cand_id [batch,B-1,K] maps choices to
 * tokens.  Outputs: tokens [batch,B] (tokens[:,0] = anchor_ids or -1), choice
 * [batch,B-1] (nullable), path_score [batch,B-1] (nullable).  1 <= K <= 32,
 * 2 <= B <= 64. */
lilicorr_status lilicorr_greedy_walk(const float* pair_scores, const int32_t* cand_id,
                                     const int32_t* anchor_ids, int64_t batch, int32_t B,
                                     int32_t K, int32_t* tokens, int32_t* choice,
                                     float* path_score, void* stream);

/* Exact best path on given scores (LiLiCorr App. E, Eq. 12; the follow-on the serving
 * write-up ranks first): the path c maximising g(c) = sum_s pair_scores[b,s-1,c_{s-1},c_s]
 * (c_0 = 0, so pair 0 uses its row 0), by max-plus dynamic programming with traceback.
 * Path sums are formed in double from the f32 scores; ties go to the lowest k, for every
 * back pointer and for the final candidate.  Same layouts as lilicorr_greedy_walk;
 * total [batch] (nullable, f64) receives g of the chosen path.  1 <= K <= 32,
 * 2 <= B <= 64.  Errors: LILICORR_ERR_INVALID_ARG for null required pointers or sizes
 * out of range, LILICORR_ERR_CUDA for a failed launch. */
lilicorr_status lilicorr_viterbi(const float* pair_scores, const int32_t* cand_id,
                                 const int32_t* anchor_ids, int64_t batch, int32_t B,
                                 int32_t K, int32_t* tokens, int32_t* choice,
                                 float* path_score, double* total, void* stream);

/* Sampled commit on given scores (serving PR, "Sampling the committed path"; LiLiCorr
 * Sec. 3.3, Eq. 2): slot s draws c_s from softmax_k(pair_scores[b,s-1,c_{s-1},k] / T_b)
 * given the previous draw (c_0 = 0), and publishes the distribution it drew from so a
 * verifier can accept by rejection sampling.
 *   temperature [batch] f32, nullable (null: every row greedy).  Rows with T_b <= 0 take
 *               the greedy argmax (f32, lowest k on ties), bit-identical to
 *               lilicorr_greedy_walk, with a one-hot proposal.
 *   uniforms    [batch,B-1] f32 in [0,1), the caller's random numbers (one per slot,
 *               e.g. from its own Philox stream); required when temperature is given.
 *               The draw is by inverse CDF: weights exp((z - max z)/T) and their running
 *               sums in double, in k order; c_s = the first k whose running sum exceeds
 *               u * (total).
 *   proposal    [batch,B-1,K] f32, nullable: the drawn-from distribution per slot.
 * Other layouts as lilicorr_greedy_walk.  1 <= K <= 32.  Errors: LILICORR_ERR_INVALID_ARG
 * for null required pointers, temperature without uniforms or sizes out of range;
 * LILICORR_ERR_CUDA for a failed launch. */
lilicorr_status lilicorr_sample_walk(const float* pair_scores, const int32_t* cand_id,
                                     const int32_t* anchor_ids, const float* temperature,
                                     const float* uniforms, int64_t batch, int32_t B,
                                     int32_t K, int32_t* tokens, int32_t* choice,
                                     float* path_score, float* proposal, void* stream);

/* Human-readable name of a status; never NULL. */
const char* lilicorr_status_string(lilicorr_status s);
/* Message of the most recent CUDA failure in this thread ("" if none). */
const char* lilicorr_last_error(void);
/* Kernels this library has launched since load (all threads). */
uint64_t lilicorr_launch_count(void);
/* Read and clear the device-side error words of the current device (synchronises the
 * device): 0 = no error; otherwise one bit per wait site that gave up (bits 0-7 the logit
 * pass, bits 8-15 the tensor-core GEMM, bits 16-23 the tensor-core attention). */
lilicorr_status lilicorr_device_error(uint32_t* code);
/* Self-check of the device-side timeouts (a diagnostic of this library; the pages have no
 * counterpart).  Runs the logit pass on one row of V bf16 logits (device memory, 16-byte
 * aligned, 1 <= V <= 16384 so that the row is a single stage) with that stage's bulk copy
 * announced to its barrier but never issued.  The consumer warps' bounded wait gives up
 * after limit_cycles SM cycles (1000 <= limit_cycles <= 1e8), then the producer's final
 * wait for its copies does too; each records its site bit (bit 0: stage wait, bit 1:
 * drain) in the device error word and the kernel returns without writing cand_id [1],
 * cand_logit [1] or lse [1] (device memory, still required).  Nothing faults, traps or
 * hangs: the context stays usable.  Read the bits with lilicorr_device_error.
 * Errors: LILICORR_ERR_INVALID_ARG for null pointers or sizes out of range,
 * LILICORR_ERR_CUDA for a failed launch. */
lilicorr_status lilicorr_diag_wait_timeout(const void* logits, int64_t V, uint32_t limit_cycles,
                                           int32_t* cand_id, float* cand_logit, float* lse,
                                           void* stream);

/* Per-kernel timing.  When enabled, lilicorr_rerank records a CUDA event on its stream
 * after each of its launches.  lilicorr_stage_times() synchronises on the recorded
 * events and, for every timing slot i < n (names: lilicorr_stage_name(i)), writes the
 * elapsed milliseconds summed over all calls since the last read into ms[i] and the
 * number of launches into launches[i] (either array may be NULL); *calls gets the
 * number of calls.  It returns the number of slots and resets the accumulators. */
void lilicorr_stage_timing(int enable);
int32_t lilicorr_stage_times(double* ms, int64_t* launches, int32_t n, int64_t* calls);
const char* lilicorr_stage_name(int32_t i);

#ifdef __cplusplus
}
#endif

#endif /* LILICORR_H_ */
