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

// One warp per (block b, pair p); a CTA holds up to four pairs of one block.  heads
// [batch*S, 2E] holds the raw out | in head outputs; anchor_raw (row stride anchor_stride)
// the block's raw anchor head output Wa t + ba.  The warp copies the raw out rows of slot
// p (the anchor for p == 0) and the in rows of slot p+1 to shared memory with 16-byte
// asynchronous copies, takes every row's inverse norm 1 / max(||v||, 1e-12) there, and
// forms phi = sigma * (o . i) * inv(o) * inv(i), the cosine of the normalised vectors up
// to f32 rounding.  The dot products run on the tensor cores (warp-level TF32 MMA with
// split operands, f32-level accuracy), reading each shared operand once.
constexpr int PS_MAX_WARPS = 4;

__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// x = hi + lo with hi, lo TF32 values (round to nearest, ties away from zero).
__device__ __forceinline__ void tf32_split(float x, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
  const float r = x - __uint_as_float(hi);
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(r));
}

// d += a . b for one m16n8k8 TF32 tile (f32 accumulate).
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__host__ __device__ inline size_t ps_warp_floats(int K, int E) {
  const int K16 = (K + 15) & ~15;
  return size_t(2) * K16 * (E + 4) + 2 * K16;
}

__global__ void __launch_bounds__(32 * PS_MAX_WARPS, 3) pair_scores_kernel(
    const float* __restrict__ heads, const float* __restrict__ anchor_raw, int64_t anchor_stride,
    int B, int K, int E, float sigma, float* __restrict__ scores, float* __restrict__ out_tap,
    float* __restrict__ in_tap, float* __restrict__ anchor_tap) {
  extern __shared__ __align__(16) float ps_smem[];
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int p = blockIdx.x * (blockDim.x >> 5) + warp;
  const int b = blockIdx.y;
  if (p >= B - 1) return;  // warp-uniform; no CTA-wide barrier follows
  const int E1 = E + 4;  // row pitch: 16-byte rows on shifted banks
  const int K16 = (K + 15) & ~15;
  float* so = ps_smem + size_t(warp) * ps_warp_floats(K, E);  // [K16][E1] out rows / anchor
  float* si = so + K16 * E1;                                   // [K16][E1] in rows of slot p+1
  float* inv = si + K16 * E1;                                  // [2*K16] inverse norms
  const int S = (B - 1) * K;
  const int64_t blk_row0 = int64_t(b) * S;
  const int E4 = E >> 2;  // float4 columns (E % 4 == 0)
  const int n_out = (p == 0) ? 1 : K;

  // rows 0..K16-1: out rows, K16..2*K16-1: in rows; rows past K (and past the anchor) zero
  for (int r = 0; r < 2 * K16; ++r) {
    const bool is_in = r >= K16;
    const int k = is_in ? r - K16 : r;
    float* dst = (is_in ? si : so) + k * E1;
    const float* src = nullptr;
    if (is_in) {
      if (k < K) src = heads + (blk_row0 + int64_t(p) * K + k) * (2 * E) + E;
    } else if (k < n_out) {
      src = p == 0 ? anchor_raw + int64_t(b) * anchor_stride
                   : heads + (blk_row0 + int64_t(p - 1) * K + k) * (2 * E);
    }
    for (int c = lane; c < E4; c += 32) {
      if (src)
        cp_async16(dst + 4 * c, src + 4 * c);
      else
        reinterpret_cast<float4*>(dst)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  cp_async_wait_all();
  __syncwarp();

  // inverse norms: lane per row
  for (int r = lane; r < 2 * K16; r += 32) {
    const float* v = r >= K16 ? si + (r - K16) * E1 : so + r * E1;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;  // independent chains
#pragma unroll 8
    for (int c = 0; c < E4; ++c) {
      const float4 x = reinterpret_cast<const float4*>(v)[c];
      s0 = fmaf(x.x, x.x, s0);
      s1 = fmaf(x.y, x.y, s1);
      s2 = fmaf(x.z, x.z, s2);
      s3 = fmaf(x.w, x.w, s3);
    }
    inv[r] = 1.0f / fmaxf(sqrtf((s0 + s1) + (s2 + s3)), 1e-12f);
  }
  __syncwarp();

  // taps of the normalised vectors (checking only)
  if (out_tap || in_tap || anchor_tap) {
    for (int r = 0; r < n_out + K; ++r) {
      const bool is_in = r >= n_out;
      const int k = is_in ? r - n_out : r;
      float* tap;
      if (is_in)
        tap = in_tap ? in_tap + (blk_row0 + int64_t(p) * K + k) * E : nullptr;
      else if (p == 0)
        tap = anchor_tap ? anchor_tap + int64_t(b) * E : nullptr;
      else
        tap = out_tap ? out_tap + (blk_row0 + int64_t(p - 1) * K + k) * E : nullptr;
      if (!tap) continue;
      const float* v = (is_in ? si : so) + k * E1;
      const float sc = inv[is_in ? K16 + k : k];
      for (int e = lane; e < E; e += 32) tap[e] = v[e] * sc;
    }
    if (p == 0 && out_tap) {  // slot B-1's out rows are used by no pair
      for (int k = 0; k < K; ++k) {
        const int64_t row = blk_row0 + int64_t(B - 2) * K + k;
        const float* src = heads + row * (2 * E);
        float ss = 0.f;
        for (int e = lane; e < E; e += 32) ss = fmaf(src[e], src[e], ss);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(FULL_MASK, ss, o);
        const float sc = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
        for (int e = lane; e < E; e += 32) out_tap[row * E + e] = src[e] * sc;
      }
    }
  }

  // K x K dot products on the tensor cores, 16 x 16 tiles: mma.sync m16n8k8 in TF32 with
  // each operand split hi + lo (hi = tf32(x), lo = tf32(x - hi)) and the three products
  // hi.hi + hi.lo + lo.hi accumulated in f32 (about 21 significant bits per product, the
  // dropped lo.lo term below 2^-22 relative).  Fragments: g = lane / 4 picks the row
  // (A) or column (B), t = lane % 4 the K index.
  float* dst_scores = scores + (int64_t(b) * (B - 1) + p) * K * K;
  const int g = lane >> 2, t = lane & 3;
  for (int t0 = 0; t0 < K; t0 += 16) {
    for (int u0 = 0; u0 < K; u0 += 16) {
      const float* A0 = so + (t0 + g) * E1;
      const float* A1 = so + (t0 + g + 8) * E1;
      const float* B0 = si + (u0 + g) * E1;
      const float* B1 = si + (u0 + 8 + g) * E1;
      float acc[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;
#pragma unroll 4
      for (int e = t; e < E; e += 8) {
        uint32_t ah[4], al[4], bh[2][2], bl[2][2];
        tf32_split(A0[e], ah[0], al[0]);
        tf32_split(A1[e], ah[1], al[1]);
        tf32_split(A0[e + 4], ah[2], al[2]);
        tf32_split(A1[e + 4], ah[3], al[3]);
        tf32_split(B0[e], bh[0][0], bl[0][0]);
        tf32_split(B0[e + 4], bh[0][1], bl[0][1]);
        tf32_split(B1[e], bh[1][0], bl[1][0]);
        tf32_split(B1[e + 4], bh[1][1], bl[1][1]);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          mma_tf32(acc[j], al, bh[j]);
          mma_tf32(acc[j], ah, bl[j]);
          mma_tf32(acc[j], ah, bh[j]);
        }
      }
      // acc[j] = C[g][2t], C[g][2t+1], C[g+8][2t], C[g+8][2t+1] of column block j
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int k = t0 + g + (i >= 2 ? 8 : 0), kk = u0 + 8 * j + 2 * t + (i & 1);
          if (k < K && kk < K)
            dst_scores[k * K + kk] =
                (p == 0 && k > 0) ? -INFINITY : sigma * acc[j][i] * inv[k] * inv[K16 + kk];
        }
    }
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
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t b = blockIdx.x;
  if (b >= batch) return;
  const int n = (B - 1) * K * K;
  const float* src = scores + b * n;
  if (staged) {
    // every 16-byte copy of the block's scores in flight at once (n = (B-1) K^2 is a
    // multiple of 4 when K is even; an odd K or an unaligned array takes the scalar loop)
    if ((K & 1) == 0 && (reinterpret_cast<uintptr_t>(scores) & 15) == 0) {
      for (int i = lane; i < (n >> 2); i += 32) cp_async16(gw_smem + 4 * i, src + 4 * i);
      cp_async_wait_all();
    } else {
      for (int i = lane; i < n; i += 32) gw_smem[i] = __ldg(src + i);
    }
    __syncwarp();
  }
  const float* sc = staged ? gw_smem : src;
  if (lane == 0) tokens[b * B] = anchor_ids ? anchor_ids[b] : -1;
  // The walk keeps step p's choice and value in lane p % 32 (two rounds for B - 1 > 32);
  // the outputs and the token lookups happen after the walk, in parallel, so no step
  // waits for a global load.
  int prev = 0;
  int c_lo = 0, c_hi = 0;
  float v_lo = 0.f, v_hi = 0.f;
  for (int p = 0; p < B - 1; ++p) {
    const float* row = sc + (p * K + prev) * K;
    // argmax as one warp max over ordered keys (-0.0 folded into +0.0 so that equal
    // values tie), then the lowest lane holding it
    const int key = lane < K ? float_key(row[lane] + 0.0f) : INT_MIN;
    const int kmax = __reduce_max_sync(FULL_MASK, key);
    const int idx = __ffs(__ballot_sync(FULL_MASK, key == kmax)) - 1;
    if (lane == (p & 31)) {
      if (p < 32) {
        c_lo = idx;
        v_lo = key_float(kmax);
      } else {
        c_hi = idx;
        v_hi = key_float(kmax);
      }
    }
    prev = idx;
  }
  for (int p = lane; p < B - 1; p += 32) {
    const int c = p < 32 ? c_lo : c_hi;
    const float v = p < 32 ? v_lo : v_hi;
    const int64_t pr = b * (B - 1) + p;
    if (choice) choice[pr] = c;
    if (path) path[pr] = v;
    tokens[b * B + p + 1] = __ldg(cand_id + pr * K + c);
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

cudaError_t launch_pair_scores(const float* heads, const float* anchor_raw, int64_t anchor_stride,
                               int64_t batch, int B, int K, int E, float sigma, float* scores,
                               float* out_tap, float* in_tap, float* anchor_tap,
                               cudaStream_t stream) {
  if (E % 4 || E > 256 || K < 1 || K > 32 || B < 2 || anchor_stride % 4 ||
      (reinterpret_cast<uintptr_t>(heads) % 16) || (reinterpret_cast<uintptr_t>(anchor_raw) % 16))
    return cudaErrorInvalidValue;
  const size_t per_warp = ps_warp_floats(K, E) * sizeof(float);
  int pw = PS_MAX_WARPS;
  while (pw > 1 && pw * per_warp > size_t(200) * 1024) --pw;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(pair_scores_kernel),
                                     static_cast<int>(pw * per_warp));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((B - 1 + pw - 1) / pw), static_cast<unsigned>(batch));
  e = launch_k(pair_scores_kernel, grid, dim3(32 * pw), pw * per_warp, stream, heads, anchor_raw,
               anchor_stride, B, K, E, sigma, scores, out_tap, in_tap, anchor_tap);
  if (e != cudaSuccess) return e;
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
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(greedy_walk_kernel),
                                     static_cast<int>(kMaxStage));
  if (e != cudaSuccess) return e;
  e = launch_k(greedy_walk_kernel, dim3(static_cast<unsigned>(batch)), dim3(32), staged ? need : 0,
               stream, scores, cand_id, anchor_ids, batch, B, K, tokens, choice, path, staged);
  if (e != cudaSuccess) return e;
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
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(viterbi_kernel),
                                     static_cast<int>(kMaxStage + 4096));
  if (e != cudaSuccess) return e;
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
