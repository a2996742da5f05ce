// Steps a4 (normalise + matching scores) and a5 (greedy commit).
//
// Matching score (LiLiCorr: Lightweight Likelihood Correlation of Parallel Drafts for
// Speculative Decoding, Sec. 3.2, Eq. 1): phi(s,k,k') = sigma * cos(o_{s,k}, i_{s+1,k'})
// for s = 0..B-2, with one anchor out vector o_0 (K_0 = 1).  Sec. 3.5: the (B-2)K^2 + K
// terms are one small product per adjacent slot pair, batched over the block.
// Greedy commit (Sec. 3.5, Eq. 8): c_s = argmax_k phi(s-1, c_{s-1}, k), ties to the
// lowest k (serving PR "[Spec] Add LiLiCorr", "Why the custom kernels": the argmax
// breaks ties toward the lower index).
#include <float.h>
#include <limits.h>

#include "kernels.cuh"

namespace lilicorr {

// One CTA per (block b, pair p).  heads [batch*S, 2E] holds the raw out | in head
// outputs.  The p == 0 CTA of a block also evaluates the anchor head on the block's
// target state (anchor_raw = Wa t + ba, f32 accumulation of exact bf16 products).
// Vectors are normalised here (nrm(v) = v / max(||v||, 1e-12)) and dotted in f32.
__global__ void __launch_bounds__(256) pair_scores_kernel(
    const float* __restrict__ heads, const __nv_bfloat16* __restrict__ target,
    const __nv_bfloat16* __restrict__ Wa, const float* __restrict__ ba, int B, int K, int E, int H,
    float sigma, float* __restrict__ scores, float* __restrict__ out_tap,
    float* __restrict__ in_tap, float* __restrict__ anchor_tap) {
  extern __shared__ __align__(16) float ps_smem[];
  const int E1 = E + 4;  // row pitch: 16-byte rows, rows of a warp on distinct banks
  float* so = ps_smem;            // [K][E1] out vectors of slot p (or o_0 in row 0)
  float* si = ps_smem + K * E1;   // [K][E1] in vectors of slot p+1
  const int p = blockIdx.x, b = blockIdx.y;
  const int S = (B - 1) * K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int64_t blk_row0 = int64_t(b) * S;

  if (p == 0) {
    // raw anchor head output for this block, into row 0 of so
    const __nv_bfloat16* t = target ? target + int64_t(b) * H : nullptr;
    for (int e = warp; e < E; e += nw) {
      float acc = 0.f;
      if (t)
        for (int h = lane * 8; h < H; h += 256) {
          const uint4 wa = __ldg(reinterpret_cast<const uint4*>(Wa + int64_t(e) * H + h));
          const uint4 tv = __ldg(reinterpret_cast<const uint4*>(t + h));
          const uint32_t aw[4] = {wa.x, wa.y, wa.z, wa.w}, tw[4] = {tv.x, tv.y, tv.z, tv.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc = fmaf(__uint_as_float(aw[j] << 16), __uint_as_float(tw[j] << 16), acc);
            acc = fmaf(__uint_as_float(aw[j] & 0xffff0000u), __uint_as_float(tw[j] & 0xffff0000u),
                       acc);
          }
        }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(FULL_MASK, acc, o);
      if (lane == 0) so[e] = acc + ba[e];
    }
    __syncthreads();
  }

  // rows to normalise: out rows of slot p (p >= 1) or the anchor (p == 0); in rows of
  // slot p+1; the p == 0 CTA also normalises slot B-1's out rows for the tap.
  const int n_out = (p == 0) ? 1 : K;
  for (int r = warp; r < n_out + K; r += nw) {
    const float* src;
    float* dst;
    float* tap = nullptr;
    if (r < n_out) {
      if (p == 0) {
        src = so;  // normalised in place
        tap = anchor_tap ? anchor_tap + int64_t(b) * E : nullptr;
      } else {
        const int64_t row = blk_row0 + int64_t(p - 1) * K + r;
        src = heads + row * (2 * E);
        tap = out_tap ? out_tap + row * E : nullptr;
      }
      dst = so + r * E1;
    } else {
      const int k = r - n_out;
      const int64_t row = blk_row0 + int64_t(p) * K + k;
      src = heads + row * (2 * E) + E;
      tap = in_tap ? in_tap + row * E : nullptr;
      dst = si + k * E1;
    }
    float ss = 0.f;
    for (int e = lane; e < E; e += 32) {
      const float v = src[e];
      ss = fmaf(v, v, ss);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(FULL_MASK, ss, o);
    const float inv = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
    for (int e = lane; e < E; e += 32) {
      const float v = src[e] * inv;
      dst[e] = v;
      if (tap) tap[e] = v;
    }
  }
  if (p == 0 && out_tap) {
    for (int k = warp; k < K; k += nw) {
      const int64_t row = blk_row0 + int64_t(B - 2) * K + k;
      const float* src = heads + row * (2 * E);
      float ss = 0.f;
      for (int e = lane; e < E; e += 32) ss = fmaf(src[e], src[e], ss);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(FULL_MASK, ss, o);
      const float inv = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
      for (int e = lane; e < E; e += 32) out_tap[row * E + e] = src[e] * inv;
    }
  }
  __syncthreads();

  float* dst = scores + (int64_t(b) * (B - 1) + p) * K * K;
  for (int t = tid; t < K * K; t += blockDim.x) {
    const int k = t / K, kk = t % K;
    float v;
    if (p == 0 && k > 0) {
      v = -INFINITY;
    } else {
      const float* a = so + k * E1;
      const float* c = si + kk * E1;
      float acc = 0.f;
      for (int e = 0; e < E; e += 4) {  // E % 4 == 0
        const float4 a4 = *reinterpret_cast<const float4*>(a + e);
        const float4 c4 = *reinterpret_cast<const float4*>(c + e);
        acc = fmaf(a4.x, c4.x, acc);
        acc = fmaf(a4.y, c4.y, acc);
        acc = fmaf(a4.z, c4.z, acc);
        acc = fmaf(a4.w, c4.w, acc);
      }
      v = sigma * acc;
    }
    dst[t] = v;
  }
}

// One warp per block: the block's (B-1) K x K scores are staged in shared memory with
// independent coalesced loads, then the B-1 dependent argmaxes over K <= 32 candidates
// run from there.
__global__ void __launch_bounds__(32) greedy_walk_kernel(
    const float* __restrict__ scores, const int32_t* __restrict__ cand_id,
    const int32_t* __restrict__ anchor_ids, int64_t batch, int B, int K,
    int32_t* __restrict__ tokens, int32_t* __restrict__ choice, float* __restrict__ path,
    bool staged) {
  extern __shared__ __align__(16) float gw_smem[];
  const int lane = threadIdx.x & 31;
  const int64_t b = blockIdx.x;
  if (b >= batch) return;
  const int n = (B - 1) * K * K;
  const float* src = scores + b * n;
  if (staged) {
    // independent 16-byte loads, eight in flight per lane (n = (B-1) K^2 is a multiple of
    // 4 when K is even; an odd K takes the scalar loop)
    if ((K & 1) == 0) {
      const float4* s4 = reinterpret_cast<const float4*>(src);
      float4* d4 = reinterpret_cast<float4*>(gw_smem);
      const int n4 = n >> 2;
      for (int i0 = 0; i0 < n4; i0 += 256) {
        float4 t[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = i0 + j * 32 + lane;
          t[j] = i < n4 ? __ldg(s4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = i0 + j * 32 + lane;
          if (i < n4) d4[i] = t[j];
        }
      }
    } else {
      for (int i = lane; i < n; i += 32) gw_smem[i] = __ldg(src + i);
    }
    __syncwarp();
  }
  const float* sc = staged ? gw_smem : src;
  if (lane == 0) tokens[b * B] = anchor_ids ? anchor_ids[b] : -1;
  int prev = 0;
  for (int p = 0; p < B - 1; ++p) {
    const int64_t pr = b * (B - 1) + p;
    const float* row = sc + (p * K + prev) * K;
    float v = lane < K ? row[lane] : -INFINITY;
    int idx = lane < K ? lane : INT_MAX;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float ov = __shfl_xor_sync(FULL_MASK, v, o);
      const int oi = __shfl_xor_sync(FULL_MASK, idx, o);
      if (ov > v || (ov == v && oi < idx)) {
        v = ov;
        idx = oi;
      }
    }
    if (lane == 0) {
      if (choice) choice[pr] = idx;
      if (path) path[pr] = v;
      tokens[b * B + p + 1] = __ldg(cand_id + pr * K + idx);
    }
    prev = idx;
  }
}

// Exact best path (LiLiCorr App. E, Eq. 12): maximise g(c) = sum_s phi(s-1, c_{s-1}, c_s)
// by max-plus dynamic programming over the same scores, one warp per block, lane k' =
// candidate k' of the current slot.  Path sums are accumulated in double from the f32
// scores (each step is one addition per (k, k'), so the sums are those of the plain
// definition); ties go to the lowest k, both for the back pointers and for the final
// candidate.  Back pointers live in shared memory; lane 0 traces the path back.
__global__ void __launch_bounds__(32) viterbi_kernel(
    const float* __restrict__ scores, const int32_t* __restrict__ cand_id,
    const int32_t* __restrict__ anchor_ids, int64_t batch, int B, int K,
    int32_t* __restrict__ tokens, int32_t* __restrict__ choice, float* __restrict__ path,
    double* __restrict__ total, bool staged) {
  extern __shared__ __align__(16) float vt_smem[];
  const int lane = threadIdx.x & 31;
  const int64_t b = blockIdx.x;
  if (b >= batch) return;
  const int Bm1 = B - 1, KK = K * K;
  const int n = Bm1 * KK;
  const float* src = scores + b * n;
  if (staged)
    for (int i = lane; i < n; i += 32) vt_smem[i] = __ldg(src + i);
  uint8_t* back = reinterpret_cast<uint8_t*>(vt_smem + (staged ? n : 0));  // [B-1][K]
  int* chosen = reinterpret_cast<int*>(back + ((Bm1 * K + 15) & ~15));     // [B-1]
  __syncwarp();
  const float* sc = staged ? vt_smem : src;
  double best = lane < K ? double(sc[lane]) : -INFINITY;  // pair 0 uses row 0 only
  for (int s = 1; s < Bm1; ++s) {
    const float* zs = sc + s * KK;
    double nb = -INFINITY;
    int arg = 0;
    for (int k = 0; k < K; ++k) {
      const double bk = __shfl_sync(FULL_MASK, best, k);
      if (lane < K) {
        const double c = bk + double(zs[k * K + lane]);
        if (c > nb) {
          nb = c;
          arg = k;
        }
      }
    }
    if (lane < K) back[s * K + lane] = static_cast<uint8_t>(arg);
    best = lane < K ? nb : -INFINITY;
  }
  // final candidate: the best total, lowest k on ties
  double v = best;
  int idx = lane < K ? lane : INT_MAX;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const double ov = __shfl_xor_sync(FULL_MASK, v, o);
    const int oi = __shfl_xor_sync(FULL_MASK, idx, o);
    if (ov > v || (ov == v && oi < idx)) {
      v = ov;
      idx = oi;
    }
  }
  __syncwarp();
  if (lane == 0) {
    int c = idx;
    chosen[Bm1 - 1] = c;
    for (int s = Bm1 - 1; s >= 1; --s) {
      c = back[s * K + c];
      chosen[s - 1] = c;
    }
    if (total) total[b] = v;
    tokens[b * B] = anchor_ids ? anchor_ids[b] : -1;
  }
  __syncwarp();
  for (int s = lane; s < Bm1; s += 32) {
    const int c = chosen[s];
    const int prev = s == 0 ? 0 : chosen[s - 1];
    const int64_t pr = b * Bm1 + s;
    if (choice) choice[pr] = c;
    if (path) path[pr] = sc[s * KK + prev * K + c];
    tokens[b * B + s + 1] = __ldg(cand_id + pr * K + c);
  }
}

// Sampled commit (serving PR, "Sampling the committed path"; LiLiCorr Eq. 2): each
// slot draws c_s from softmax_k(z_s[k] / T_b) given the previous draw, by inverse CDF
// with the caller's uniform u[b, s]: w_k = exp((z_k - max z) / T) in double, W = their
// sum in k order, c_s = the first k whose running sum exceeds u * W (the last k with
// w > 0 if rounding leaves none).  Rows with T_b <= 0 (or no temperature array) take the
// same f32 argmax, lowest k on ties, as the greedy walk and publish a one-hot proposal.
// One warp per block; lane k holds candidate k; lane 0 forms the running sums in order.
__global__ void __launch_bounds__(32) sample_walk_kernel(
    const float* __restrict__ scores, const int32_t* __restrict__ cand_id,
    const int32_t* __restrict__ anchor_ids, const float* __restrict__ temperature,
    const float* __restrict__ uniforms, int64_t batch, int B, int K,
    int32_t* __restrict__ tokens, int32_t* __restrict__ choice, float* __restrict__ path,
    float* __restrict__ proposal) {
  __shared__ double s_w[32];
  const int lane = threadIdx.x & 31;
  const int64_t b = blockIdx.x;
  if (b >= batch) return;
  const int Bm1 = B - 1;
  const float T = temperature ? temperature[b] : 0.f;
  const float* src = scores + b * int64_t(Bm1) * K * K;
  if (lane == 0) tokens[b * B] = anchor_ids ? anchor_ids[b] : -1;
  int prev = 0;
  for (int s = 0; s < Bm1; ++s) {
    const int64_t pr = b * Bm1 + s;
    const float z = lane < K ? __ldg(src + (int64_t(s) * K + prev) * K + lane) : -INFINITY;
    // f32 argmax, lowest k on ties (the greedy decision)
    float v = z;
    int idx = lane < K ? lane : INT_MAX;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float ov = __shfl_xor_sync(FULL_MASK, v, o);
      const int oi = __shfl_xor_sync(FULL_MASK, idx, o);
      if (ov > v || (ov == v && oi < idx)) {
        v = ov;
        idx = oi;
      }
    }
    int c = idx;
    float q = lane == idx ? 1.f : 0.f;
    if (T > 0.f && v != -INFINITY) {
      const double w = lane < K ? exp((double(z) - double(v)) / double(T)) : 0.0;
      s_w[lane] = w;
      __syncwarp();
      int pick = 0;
      double W = 0.0;
      if (lane == 0) {
        for (int k = 0; k < K; ++k) W += s_w[k];
        const double thr = double(uniforms[pr]) * W;
        double cum = 0.0;
        int last = 0;
        pick = -1;
        for (int k = 0; k < K; ++k) {
          cum += s_w[k];
          if (s_w[k] > 0.0) last = k;
          if (pick < 0 && cum > thr) pick = k;
        }
        if (pick < 0) pick = last;
      }
      c = __shfl_sync(FULL_MASK, pick, 0);
      W = __shfl_sync(FULL_MASK, W, 0);
      q = static_cast<float>(w / W);
      __syncwarp();
    }
    if (proposal && lane < K) proposal[pr * K + lane] = q;
    if (lane == 0) {
      if (choice) choice[pr] = c;
      if (path) path[pr] = __ldg(src + (int64_t(s) * K + prev) * K + c);
      tokens[b * B + s + 1] = __ldg(cand_id + pr * K + c);
    }
    prev = c;
  }
}

cudaError_t launch_pair_scores(const float* heads, const __nv_bfloat16* target,
                               const __nv_bfloat16* Wa, const float* ba, int64_t batch, int B,
                               int K, int E, int H, float sigma, float* scores, float* out_tap,
                               float* in_tap, float* anchor_tap, cudaStream_t stream) {
  if (H % 8 || (reinterpret_cast<uintptr_t>(Wa) % 16) || (reinterpret_cast<uintptr_t>(target) % 16))
    return cudaErrorInvalidValue;
  if (E % 4) return cudaErrorInvalidValue;
  const size_t smem = size_t(2) * K * (E + 4) * sizeof(float);
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(pair_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         2 * 32 * 260 * 4);
    attr = true;
  }
  const dim3 grid(B - 1, static_cast<unsigned>(batch));
  pair_scores_kernel<<<grid, 256, smem, stream>>>(heads, target, Wa, ba, B, K, E, H, sigma, scores,
                                                  out_tap, in_tap, anchor_tap);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_greedy_walk(const float* scores, const int32_t* cand_id,
                               const int32_t* anchor_ids, int64_t batch, int B, int K,
                               int32_t* tokens, int32_t* choice, float* path,
                               cudaStream_t stream) {
  constexpr size_t kMaxStage = 96 * 1024;
  const size_t need = size_t(B - 1) * K * K * sizeof(float);
  const bool staged = need <= kMaxStage;  // otherwise the walk reads the scores in place
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(greedy_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(kMaxStage));
    attr = true;
  }
  greedy_walk_kernel<<<static_cast<unsigned>(batch), 32, staged ? need : 0, stream>>>(
      scores, cand_id, anchor_ids, batch, B, K, tokens, choice, path, staged);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_viterbi(const float* scores, const int32_t* cand_id,
                           const int32_t* anchor_ids, int64_t batch, int B, int K,
                           int32_t* tokens, int32_t* choice, float* path, double* total,
                           cudaStream_t stream) {
  constexpr size_t kMaxStage = 96 * 1024;
  const size_t need = size_t(B - 1) * K * K * sizeof(float);
  const bool staged = need <= kMaxStage;  // otherwise the scores are read in place
  const size_t aux = ((size_t(B - 1) * K + 15) & ~size_t(15)) + size_t(B - 1) * sizeof(int);
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(viterbi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(kMaxStage + 4096));
    attr = true;
  }
  viterbi_kernel<<<static_cast<unsigned>(batch), 32, (staged ? need : 0) + aux, stream>>>(
      scores, cand_id, anchor_ids, batch, B, K, tokens, choice, path, total, staged);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_sample_walk(const float* scores, const int32_t* cand_id,
                               const int32_t* anchor_ids, const float* temperature,
                               const float* uniforms, int64_t batch, int B, int K,
                               int32_t* tokens, int32_t* choice, float* path, float* proposal,
                               cudaStream_t stream) {
  sample_walk_kernel<<<static_cast<unsigned>(batch), 32, 0, stream>>>(
      scores, cand_id, anchor_ids, temperature, uniforms, batch, B, K, tokens, choice, path,
      proposal);
  note_launch();
  return cudaGetLastError();
}

}  // namespace lilicorr
