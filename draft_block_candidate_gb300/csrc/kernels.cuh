// Host-side launchers of the rerank kernels (one declaration shared by all units).
#pragma once

#include <utility>

#include "common.cuh"

namespace lilicorr {

// a1 logit pass (logit_pass.cu)
size_t k1_workspace_bytes(int64_t batch, int B, int64_t V, int esize);
// The logit pass splits rows into segments only in calls of fewer than this many rows.
constexpr int K1_SPLIT_BELOW_ROWS = 90;
cudaError_t k1_launch(const void* logits, int esize, int64_t batch, int B, int64_t V, int K,
                      int32_t* cand_id, float* cand_logit, float* lse, void* ws,
                      cudaStream_t stream, int64_t row_stride = 0, int id_offset = 0,
                      void* records = nullptr, long long wait_limit = WAIT_LIMIT_CYCLES,
                      bool withhold_first = false);
size_t k1_shard_record_bytes(int K);
cudaError_t k1_merge_launch(const void* records, int n, int64_t rows, int K, int32_t* cand_id,
                            float* cand_logit, float* lse, cudaStream_t stream);
cudaError_t k1_read_device_error(uint32_t* code);

// message returned by lilicorr_last_error() for this thread (lilicorr_api.cu)
void set_last_error(const char* msg);

// Per-device host state (lilicorr_api.cu), safe to call from several host threads:
// the SM count of the current device (148 when no device can be queried), and the
// dynamic shared-memory limit of a kernel raised to at least `bytes` on the current
// device (cudaFuncSetAttribute once per kernel, size and device).
int device_sm_count();
cudaError_t allow_dynamic_smem(const void* kernel, int bytes);

// a4 scores + a5 walk (walk.cu)
cudaError_t launch_pair_scores(const float* heads, const float* anchor_raw, int64_t anchor_stride,
                               int64_t batch, int B, int K, int E, float sigma, float* scores,
                               float* out_tap, float* in_tap, float* anchor_tap,
                               cudaStream_t stream);
cudaError_t launch_viterbi(const float* scores, const int32_t* cand_id,
                           const int32_t* anchor_ids, int64_t batch, int B, int K,
                           int32_t* tokens, int32_t* choice, float* path, double* total,
                           cudaStream_t stream);
cudaError_t launch_sample_walk(const float* scores, const int32_t* cand_id,
                               const int32_t* anchor_ids, const float* temperature,
                               const float* uniforms, int64_t batch, int B, int K,
                               int32_t* tokens, int32_t* choice, float* path, float* proposal,
                               cudaStream_t stream);
cudaError_t launch_greedy_walk(const float* scores, const int32_t* cand_id,
                               const int32_t* anchor_ids, int64_t batch, int B, int K,
                               int32_t* tokens, int32_t* choice, float* path,
                               cudaStream_t stream);

// a2/a3/a4 contractions (encoder.cu)
enum Epi : int { EPI_F32 = 0, EPI_RESID = 1, EPI_SPLIT = 2, EPI_SPLIT_SILU = 3, EPI_NODE = 4 };

struct GemmArgs {
  const __nv_bfloat16* A;  // [M, Ka] (Ka = Kw, or 2*Kw for a split operand [A_hi | A_lo])
  const __nv_bfloat16* W;  // [N, Kw]
  int64_t M;
  int N, Kw, Ka;
  const float* bias;       // [N], or one row per bias_group rows when bias_group > 0
  int64_t bias_group;      // rows sharing one bias row (0: one bias for all rows)
  int64_t bias_stride;     // elements between grouped bias rows (0: N)
  float* out;              // EPI_F32 / EPI_RESID / EPI_NODE: [M, N] f32
  __nv_bfloat16* out_split;  // EPI_SPLIT*: [M, 2N]
  // EPI_NODE extras: X = acc + bias + E[cand] + slot_table[s-1] + rank_table[k] + hidden
  const __nv_bfloat16* embed;       // [V, N]
  const int32_t* cand_id;           // [M]
  const float* slot_table;          // [B_max-1, N]
  const float* rank_table;          // [K_max, N]
  const __nv_bfloat16* slot_hidden; // [batch, B, N] or null
  int K, B;
  int64_t vocab;                    // rows of embed (gather index is clamped to it)
  float* nodes_tap;                 // [M, N] or null
  // A operand made in the kernel instead of read (A is then unused), split bf16 hi / lo
  // written straight into the shared-memory stages:
  //   ASRC_FUSION: A = [h, h * t] with h = a_x [M, Kw/2] f32 and t = a_t [M / a_group,
  //                Kw/2] bf16 (null: zero), the column blocks of h and h * t interleaved
  //   ASRC_CONF:   A = SiLU(a_w1 f + a_b1) [M, Kw], f the five confidence features of row
  //                m from a_cl [M] (candidate logits), a_lse [M / K] and its rank m % K
  int asrc;
  const float* a_x;
  const __nv_bfloat16* a_t;
  int64_t a_group;
  const float *a_cl, *a_lse, *a_w1, *a_b1;
  // The last tail_tiles output tiles run as tail_split column pieces each (128 x 256 /
  // tail_split), so that the last round of the persistent grid keeps more SMs busy; every
  // piece owns its outputs (no reduction).  Set by launch_gemm.
  int tail_tiles, tail_split;
};
enum ASrc : int { ASRC_TMA = 0, ASRC_FUSION = 1, ASRC_CONF = 2 };

// tcgen05 tensor-core GEMM (gemm_tc.cu)
cudaError_t launch_gemm(int epi, const GemmArgs& g, cudaStream_t stream);
// LM-head projection fused with the top-K / log-sum-exp pass (gemm_tc.cu)
bool lm_head_supported(int64_t rows, int64_t V, int D, int K);
size_t lm_head_records_bytes(int64_t rows, int64_t V, int K);
cudaError_t launch_lm_head_topk(const __nv_bfloat16* hidden, const __nv_bfloat16* w_lm,
                                int64_t rows, int64_t V, int D, int K, void* records,
                                int32_t* cand_id, float* cand_logit, float* lse,
                                cudaStream_t stream);
cudaError_t tc_read_device_error(uint32_t* code);
// confidence layer as its own pass, hidden width 256 only (encoder.cu)
cudaError_t launch_conf_hidden(const float* cand_logit, const float* lse, int64_t M, int K, int H,
                               const float* w1, const float* b1, __nv_bfloat16* U,
                               cudaStream_t stream);
cudaError_t launch_rmsnorm_split(const float* X, const float* gain, int64_t M, int H, float eps,
                                 __nv_bfloat16* out, cudaStream_t stream);
cudaError_t launch_attention(const __nv_bfloat16* qkv, int64_t batch, int S, int K, int H,
                             int heads, int B_max, const float* dist_bias,
                             const float* same_bias, __nv_bfloat16* out, cudaStream_t stream);
// tcgen05 attention for head dim 64, up to 256 tokens and a per-query-slot bias table
// that fits beside its operand tiles (S / K <= 25 query slots) (attn_tc.cu)
bool attention_tc_supported(int S, int K, int H, int heads, int B_max);
cudaError_t launch_attention_tc(const __nv_bfloat16* qkv, int64_t batch, int S, int K, int H,
                                int heads, int B_max, const float* dist_bias,
                                const float* same_bias, __nv_bfloat16* out, cudaStream_t stream);
// tcgen05 attention for head dim 64 and 257..512 tokens, keys in chunks of 128 with an
// online softmax (attn_tc.cu)
bool attention_tc_long_supported(int S, int K, int H, int heads, int B_max);
cudaError_t launch_attention_tc_long(const __nv_bfloat16* qkv, int64_t batch, int S, int K,
                                     int H, int heads, int B_max, const float* dist_bias,
                                     const float* same_bias, __nv_bfloat16* out,
                                     cudaStream_t stream);
cudaError_t at_read_device_error(uint32_t* code);
cudaError_t launch_rows_bias(const float* bias, int64_t rows, int N, float* out,
                             cudaStream_t stream);

// Programmatic dependent launch of the path's kernels (lilicorr_api.cu): while a
// PdlScope with `on` is alive in this host thread, launch_k lets each launch begin before
// the previous kernel on the stream has finished; the kernels order their memory
// accesses after it with pdl_wait.  Off by default (the standalone entry points).
bool pdl_enabled();
struct PdlScope {
  bool prev;
  explicit PdlScope(bool on);
  ~PdlScope();
  void set(bool on);
};
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
}  // namespace lilicorr
