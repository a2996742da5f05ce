// Step a1: fused full-vocabulary log-partition + exact top-K, one read per logit row.
//
// What it computes (LiLiCorr: Lightweight Likelihood Correlation of Parallel Drafts for
// Speculative Decoding, Sec. 3.2 "retains the drafter's top-K candidate tokens" and
// App. A "log-probability ... under the full vocabulary"; serving PR "[Spec] Add
// LiLiCorr", section "Why the custom kernels": exact top-k plus the log-partition from a
// single pass over [n, V]):
//   for each block b and drafted slot s = 1..B-1 (row 0, the anchor, is never read)
//     lse[b,s-1]        = log sum_v exp(l[b,s,v])
//     cand_*[b,s-1,0:K] = the K largest logits ordered by (value desc, token id asc)
//
// GB300 design.  The pass is HBM-bound (one streaming read of batch*(B-1)*V elements), so
// each CTA streams a contiguous segment of one row through shared memory with 1-D bulk
// copies (cp.async.bulk, 16 KB stages, 3 in flight, 3 CTAs per SM) and every thread
// consumes 16-byte chunks:
//   * online log-sum-exp in base 2: per chunk one max, one FFMA + ex2 per element;
//   * top-K: warp 0 keeps the running top-32 (value, id) pairs sorted across its lanes.
//     Every thread compares its elements with the running K-th entry (floored in the
//     first stage by the K-th largest per-thread maximum, a valid lower bound), so after
//     warm-up almost every element costs one compare; the rare survivors go to a shared
//     buffer that warp 0 folds in 32 at a time (warp bitonic sort + bitonic merge)
//     during the next stage.
// Rows are split into P segments when there are too few rows to fill 152 SMs; the last
// CTA of a row (atomic counter, no waiting) merges the P partial results.
#include <float.h>
#include <limits.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <mutex>

#include "kernels.cuh"

namespace lilicorr {

static __device__ uint32_t g_err_k1;

constexpr int K1_THREADS = 512;
constexpr int K1_WARPS = K1_THREADS / 32;
constexpr int K1_STAGE_BYTES = 16384;
constexpr int K1_NSTAGES = 4;
constexpr int K1_CPT = K1_STAGE_BYTES / 16 / K1_THREADS;  // 16-byte chunks per thread per stage
constexpr int KQ = 32;                                      // queue slots per warp
constexpr float LOG2E = 1.4426950408889634f;
constexpr float M2_INIT = -1e30f;                           // "no element yet", finite

struct K1Partial {
  float m2, s;
  float v[KQ];
  int id[KQ];
};

struct K1Params {
  const char* logits;
  int64_t batch;
  int B;
  int64_t V;
  int K;
  int P;
  int64_t seg_bytes;
  int32_t* cand_id;
  float* cand_logit;
  float* lse;
  K1Partial* partials;
  unsigned* counters;
};

__device__ __forceinline__ int64_t i64min(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (va, ia) ranks before (vb, ib): larger value, then smaller id.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

struct WarpQueue {
  float qv;   // this lane's entry (lane = position in the sorted queue)
  int qid;
  float tv;   // the K-th entry, warp-uniform
  int tid;

  __device__ void init() {
    qv = -INFINITY;
    qid = INT_MAX;
    tv = -INFINITY;
    tid = INT_MAX;
  }
};

// Merge sorted list (bv, bi) (one entry per lane, descending) into (v, id): afterwards
// (v, id) holds the best 32 of the union, sorted.
__device__ __forceinline__ void bitonic_merge(float& v, int& id, float bv, int bi, int lane) {
  const float rv = __shfl_sync(FULL_MASK, bv, 31 - lane);
  const int ri = __shfl_sync(FULL_MASK, bi, 31 - lane);
  if (better(rv, ri, v, id)) {
    v = rv;
    id = ri;
  }
#pragma unroll
  for (int st = 16; st >= 1; st >>= 1) {
    const float ov = __shfl_xor_sync(FULL_MASK, v, st);
    const int oi = __shfl_xor_sync(FULL_MASK, id, st);
    const bool ob = better(ov, oi, v, id);
    const bool lower = (lane & st) == 0;
    if (lower ? ob : !ob) {
      v = ov;
      id = oi;
    }
  }
}

__device__ __forceinline__ void lse_merge(float& m2, float& s, float om2, float os) {
  const float M = fmaxf(m2, om2);
  s = s * ex2(m2 - M) + os * ex2(om2 - M);
  m2 = M;
}

template <typename T>
__device__ __forceinline__ float load_elem(const char* p);
template <>
__device__ __forceinline__ float load_elem<float>(const char* p) {
  return __ldg(reinterpret_cast<const float*>(p));
}
template <>
__device__ __forceinline__ float load_elem<__nv_bfloat16>(const char* p) {
  return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16*>(p)));
}

// Descending bitonic sort of one value per lane across the warp.
__device__ __forceinline__ float warp_sort_desc(float v, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(FULL_MASK, v, j);
      const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
      v = keep_max ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return v;
}

constexpr int K1_CAP = 256;  // candidate buffer entries per CTA and stage parity

// The running K-th entry (value, id) shared as one 64-bit word, so a reader never sees
// the value of one update with the id of another.
__device__ __forceinline__ unsigned long long pack_tau(float v, int id) {
  return (static_cast<unsigned long long>(__float_as_uint(v)) << 32) | static_cast<uint32_t>(id);
}
__device__ __forceinline__ void unpack_tau(unsigned long long w, float& v, int& id) {
  v = __uint_as_float(static_cast<uint32_t>(w >> 32));
  id = static_cast<int>(static_cast<uint32_t>(w));
}

// Sort one (value, id) pair per lane across the warp into (value desc, id asc) order
// (bitonic network, 15 compare-exchange steps).
__device__ __forceinline__ void warp_sort_pairs(float& v, int& id, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float ov = __shfl_xor_sync(FULL_MASK, v, j);
      const int oi = __shfl_xor_sync(FULL_MASK, id, j);
      const bool ob = better(ov, oi, v, id);
      const bool keep_better = ((lane & j) == 0) == ((lane & k) == 0);
      if (keep_better ? ob : !ob) {
        v = ov;
        id = oi;
      }
    }
  }
}

// Warp-uniform: fold one candidate per lane (sentinel -inf / INT_MAX for none) into the
// sorted 32-entry queue q, 32 candidates at a time: sort them, bitonic-merge, keep the
// best 32.  Skipped when no lane beats the queue's K-th entry.
__device__ __forceinline__ void queue_absorb(WarpQueue& q, float v, int id, int lane, int K) {
  if (!__any_sync(FULL_MASK, better(v, id, q.tv, q.tid))) return;
  warp_sort_pairs(v, id, lane);
  bitonic_merge(q.qv, q.qid, v, id, lane);
  q.tv = __shfl_sync(FULL_MASK, q.qv, K - 1);
  q.tid = __shfl_sync(FULL_MASK, q.qid, K - 1);
}

// Warp-uniform: fold the buffered candidates into the running queue, publish its K-th
// entry, empty the buffer.
__device__ __forceinline__ void merge_buffer(WarpQueue& run, const float* bv, const int* bi,
                                             int* cnt_p, volatile unsigned long long* tau,
                                             int lane, int K) {
  const int cnt = min(*cnt_p, K1_CAP);
  for (int c0 = 0; c0 < cnt; c0 += 32) {
    float v = -INFINITY;
    int vi = INT_MAX;
    if (c0 + lane < cnt) {
      v = bv[c0 + lane];
      vi = bi[c0 + lane];
    }
    queue_absorb(run, v, vi, lane, K);
  }
  __syncwarp();
  if (lane == 0) {
    *tau = pack_tau(run.tv, run.tid);
    *cnt_p = 0;
  }
}

// Unpack one 16-byte chunk (8 bf16 or 4 f32) into floats.
template <int NV>
__device__ __forceinline__ void unpack16(const uint4 w, float (&x)[NV]) {
  if constexpr (NV == 8) {
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __uint_as_float(ww[k] << 16);
      x[2 * k + 1] = __uint_as_float(ww[k] & 0xffff0000u);
    }
  } else {
    x[0] = __uint_as_float(w.x);
    x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z);
    x[3] = __uint_as_float(w.w);
  }
}

// Append this chunk's elements that can still enter the top-K to the stage buffer.
template <int NV>
__device__ __forceinline__ void append_chunk(const float (&x)[NV], int id0, float thr, float tv,
                                             int ti, float* bv, int* bi, int* cnt) {
#pragma unroll
  for (int j = 0; j < NV; ++j)
    if (x[j] >= thr && better(x[j], id0 + j, tv, ti)) {
      const int idx = atomicAdd(cnt, 1);
      if (idx < K1_CAP) {
        bv[idx] = x[j];
        bi[idx] = id0 + j;
      }
    }
}

template <typename T>
__global__ void __launch_bounds__(K1_THREADS, 3) logit_pass_kernel(const K1Params p) {
  constexpr int ES = sizeof(T);
  constexpr int NV = 16 / ES;
  extern __shared__ __align__(128) uint8_t k1_dyn_smem[];
  uint8_t(*stage)[K1_STAGE_BYTES] = reinterpret_cast<uint8_t(*)[K1_STAGE_BYTES]>(k1_dyn_smem);
  __shared__ __align__(8) uint64_t full_bar[K1_NSTAGES];
  __shared__ float sq_v[K1_WARPS][KQ];
  __shared__ int sq_i[K1_WARPS][KQ];
  __shared__ float s_buf_v[2][K1_CAP];
  __shared__ int s_buf_i[2][K1_CAP];
  __shared__ float s_m2[K1_WARPS], s_s[K1_WARPS];
  __shared__ float s_L0;
  __shared__ int s_abort;
  __shared__ int s_cnt[2];
  __shared__ volatile unsigned long long s_tau;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.K;
  const int64_t u = blockIdx.x;
  const int64_t r = u / p.P;
  const int seg = static_cast<int>(u % p.P);
  const int64_t b = r / (p.B - 1);
  const int64_t s_slot = r % (p.B - 1) + 1;

  // Row geometry in bytes relative to p.logits; body = 16-byte aligned part.
  const int64_t row_start = (b * p.B + s_slot) * p.V * ES;
  const int64_t row_end = row_start + p.V * ES;
  const uintptr_t base = reinterpret_cast<uintptr_t>(p.logits);
  int64_t body_start = static_cast<int64_t>(((base + row_start + 15) & ~uintptr_t(15)) - base);
  int64_t body_end = static_cast<int64_t>(((base + row_end) & ~uintptr_t(15)) - base);
  if (body_start >= body_end) body_start = body_end = row_end;
  const int64_t seg_lo = i64min(body_end, body_start + seg * p.seg_bytes);
  const int64_t seg_hi = i64min(body_end, seg_lo + p.seg_bytes);
  const int nstages = static_cast<int>((seg_hi - seg_lo + K1_STAGE_BYTES - 1) / K1_STAGE_BYTES);
  const int seg_bytes = static_cast<int>(seg_hi - seg_lo);
  const int seg_elem0 = static_cast<int>((seg_lo - row_start) / ES);  // id of first body elem

  if (tid == 0) {
    for (int i = 0; i < K1_NSTAGES; ++i) mbar_init(&full_bar[i], 1);
    fence_mbar_init();
    s_cnt[0] = s_cnt[1] = 0;
    s_abort = 0;
    s_tau = pack_tau(-INFINITY, INT_MAX);
  }
  __syncthreads();

  if (tid == 0)
    for (int st = 0; st < min(K1_NSTAGES - 1, nstages); ++st) {
      const int off = st * K1_STAGE_BYTES;
      const uint32_t bytes = static_cast<uint32_t>(min(K1_STAGE_BYTES, seg_bytes - off));
      mbar_arrive_expect_tx(&full_bar[st], bytes);
      bulk_g2s(stage[st], p.logits + seg_lo + off, bytes, &full_bar[st]);
    }

  float m2 = M2_INIT, ssum = 0.f;
  // Warp 0 owns the running top-32 of everything consumed so far (one entry per lane,
  // sorted); the other warps see its K-th entry through s_tau.
  WarpQueue run;
  run.init();

  // Unaligned head (segment 0) and tail (last segment) elements: plain loads by warp 0,
  // one element per lane, straight into the running queue.
  if (warp == 0) {
    const int64_t row_elem0 = row_start / ES;
    for (int part = 0; part < 2; ++part) {
      int64_t first = 0;
      int cnt = 0;
      if (part == 0 && seg == 0) {
        first = row_start;
        cnt = static_cast<int>((body_start - row_start) / ES);
      } else if (part == 1 && seg == p.P - 1 && body_end < row_end) {
        first = body_end;
        cnt = static_cast<int>((row_end - body_end) / ES);
      }
      if (cnt == 0) continue;  // warp-uniform
      const bool has = lane < cnt;
      const float xv = has ? load_elem<T>(p.logits + first + int64_t(lane) * ES) : -INFINITY;
      if (has) {
        const float c2 = xv * LOG2E;
        if (c2 > m2) {
          ssum *= ex2(m2 - c2);
          m2 = c2;
        }
        ssum += ex2(fmaf(xv, LOG2E, -m2));
      }
      queue_absorb(run, xv, has ? static_cast<int>(first / ES - row_elem0) + lane : INT_MAX, lane,
                   K);
    }
    if (lane == 0) s_tau = pack_tau(run.tv, run.tid);
  }

  float L0 = -INFINITY;  // lower bound of the segment's K-th largest value (from stage 0)
  bool ok = true;
  for (int st = 0; st < nstages; ++st) {
    const int slot = st % K1_NSTAGES;
    if (tid == 0 && st + K1_NSTAGES - 1 < nstages) {
      const int nx = st + K1_NSTAGES - 1, ns = nx % K1_NSTAGES;
      const int off = nx * K1_STAGE_BYTES;
      const uint32_t bytes = static_cast<uint32_t>(min(K1_STAGE_BYTES, seg_bytes - off));
      mbar_arrive_expect_tx(&full_bar[ns], bytes);
      bulk_g2s(stage[ns], p.logits + seg_lo + off, bytes, &full_bar[ns]);
    }
    if (!mbar_wait_bounded(&full_bar[slot], (st / K1_NSTAGES) & 1, &g_err_k1, ERR_K1_FULL_WAIT))
      s_abort = 1;
    const int soff = st * K1_STAGE_BYTES;
    const int nbytes = min(K1_STAGE_BYTES, seg_bytes - soff);
    const uint8_t* sbuf = stage[slot];
    const int bsel = st & 1;
    float* bv = s_buf_v[bsel];
    int* bi = s_buf_i[bsel];
    // the running K-th entry; warp 0 may raise it concurrently, either value is valid
    // (stage 0 re-reads it below, after barriers that order warp 0's head/tail update)
    float tv;
    int ti;
    unpack_tau(s_tau, tv, ti);
    const float thr = fmaxf(tv, L0);

    // ---- one 16-byte chunk at a time: log-sum-exp, then the (rare) candidate check
    float tmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < K1_CPT; ++i) {
      const int c = tid + i * K1_THREADS;
      if (c * 16 < nbytes) {
        float x[NV];
        unpack16<NV>(*reinterpret_cast<const uint4*>(sbuf + c * 16), x);
        float cm = x[0];
#pragma unroll
        for (int j = 1; j < NV; ++j) cm = fmaxf(cm, x[j]);
        const float cm2 = cm * LOG2E;
        if (cm2 > m2) {
          ssum *= ex2(m2 - cm2);
          m2 = cm2;
        }
#pragma unroll
        for (int j = 0; j < NV; ++j) ssum += ex2(fmaf(x[j], LOG2E, -m2));
        tmax = fmaxf(tmax, cm);
        if (st > 0 && cm >= thr)
          append_chunk<NV>(x, seg_elem0 + (soff + c * 16) / ES, thr, tv, ti, bv, bi, &s_cnt[bsel]);
      }
    }

    // ---- stage 0: floor L0 = the K-th largest per-thread maximum (K distinct threads
    // hold an element at least that large), then this stage's candidates.
    if (st == 0) {
      sq_v[warp][lane] = warp_sort_desc(tmax, lane);
      __syncthreads();
      for (int half = K1_WARPS / 2; half >= 1; half >>= 1) {
        if (warp < half) {
          float a = sq_v[warp][lane];
          int ai = 0;
          bitonic_merge(a, ai, sq_v[warp + half][lane], 0, lane);
          __syncwarp();
          sq_v[warp][lane] = a;
        }
        __syncthreads();
      }
      if (tid == 0) s_L0 = sq_v[0][K - 1];
      __syncthreads();
      L0 = s_L0;
      unpack_tau(s_tau, tv, ti);
      const float thr0 = fmaxf(tv, L0);
      if (tmax >= thr0) {
#pragma unroll
        for (int i = 0; i < K1_CPT; ++i) {
          const int c = tid + i * K1_THREADS;
          if (c * 16 < nbytes) {
            float x[NV];
            unpack16<NV>(*reinterpret_cast<const uint4*>(sbuf + c * 16), x);
            append_chunk<NV>(x, seg_elem0 + (soff + c * 16) / ES, thr0, tv, ti, bv, bi,
                             &s_cnt[bsel]);
          }
        }
      }
    }

    // ---- warp 0 folds the previous stage's buffer into the running queue while the
    // other warps go on (a stale threshold is still a valid lower bound)
    if (warp == 0 && st > 0)
      merge_buffer(run, s_buf_v[bsel ^ 1], s_buf_i[bsel ^ 1], &s_cnt[bsel ^ 1], &s_tau, lane, K);
    __syncthreads();
    if (s_cnt[bsel] > K1_CAP) {
      // Too many ties for the buffer: exact per-warp queues over this stage's elements,
      // re-read from shared memory (the slot is not refilled before the next iteration),
      // merged into the running queue; the buffer is dropped.
      WarpQueue q;
      q.init();
#pragma unroll
      for (int i = 0; i < K1_CPT; ++i) {
        const int c = tid + i * K1_THREADS;
        const bool has = c * 16 < nbytes;
        float x[NV];
        if (has) unpack16<NV>(*reinterpret_cast<const uint4*>(sbuf + c * 16), x);
        const int id0 = seg_elem0 + (soff + c * 16) / ES;
#pragma unroll
        for (int j = 0; j < NV; ++j)
          queue_absorb(q, has ? x[j] : -INFINITY, has ? id0 + j : INT_MAX, lane, K);
      }
      sq_v[warp][lane] = q.qv;
      sq_i[warp][lane] = q.qid;
      __syncthreads();
      for (int half = K1_WARPS / 2; half >= 1; half >>= 1) {
        if (warp < half) {
          float a = sq_v[warp][lane];
          int ai = sq_i[warp][lane];
          bitonic_merge(a, ai, sq_v[warp + half][lane], sq_i[warp + half][lane], lane);
          __syncwarp();
          sq_v[warp][lane] = a;
          sq_i[warp][lane] = ai;
        }
        __syncthreads();
      }
      if (warp == 0) {
        bitonic_merge(run.qv, run.qid, sq_v[0][lane], sq_i[0][lane], lane);
        run.tv = __shfl_sync(FULL_MASK, run.qv, K - 1);
        run.tid = __shfl_sync(FULL_MASK, run.qid, K - 1);
        if (lane == 0) {
          s_tau = pack_tau(run.tv, run.tid);
          s_cnt[bsel] = 0;
        }
      }
      __syncthreads();
    }
    if (s_abort) {
      ok = false;
      break;
    }
  }
  if (ok && warp == 0 && nstages > 0)
    merge_buffer(run, s_buf_v[(nstages - 1) & 1], s_buf_i[(nstages - 1) & 1],
                 &s_cnt[(nstages - 1) & 1], &s_tau, lane, K);
  if (!ok) {
    // Give copies still in flight a bounded chance to land before the CTA exits.
    if (tid == 0)
      for (int st = 0; st < nstages; ++st)
        if (!mbar_try_wait(&full_bar[st % K1_NSTAGES], (st / K1_NSTAGES) & 1))
          mbar_wait_bounded(&full_bar[st % K1_NSTAGES], (st / K1_NSTAGES) & 1, &g_err_k1,
                            ERR_K1_DRAIN);
    return;
  }

  // ---- CTA log-sum-exp reduction; the running queue is the CTA's top-K
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float om = __shfl_xor_sync(FULL_MASK, m2, o);
    const float os = __shfl_xor_sync(FULL_MASK, ssum, o);
    lse_merge(m2, ssum, om, os);
  }
  if (lane == 0) {
    s_m2[warp] = m2;
    s_s[warp] = ssum;
  }
  __syncthreads();
  if (warp != 0) return;

  float v = run.qv;
  int id = run.qid;
  float M = lane < K1_WARPS ? s_m2[lane] : M2_INIT;
  float S = lane < K1_WARPS ? s_s[lane] : 0.f;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float om = __shfl_xor_sync(FULL_MASK, M, o);
    const float os = __shfl_xor_sync(FULL_MASK, S, o);
    lse_merge(M, S, om, os);
  }

  if (p.P > 1) {
    K1Partial* part = p.partials + u;
    part->v[lane] = v;
    part->id[lane] = id;
    if (lane == 0) {
      part->m2 = M;
      part->s = S;
    }
    __threadfence();
    __syncwarp();
    unsigned prev = 0;
    if (lane == 0) prev = atomicAdd(&p.counters[r], 1u);
    prev = __shfl_sync(FULL_MASK, prev, 0);
    if (prev != static_cast<unsigned>(p.P - 1)) return;
    __threadfence();
    const K1Partial* parts = p.partials + r * p.P;
    v = __ldcg(&parts[0].v[lane]);
    id = __ldcg(&parts[0].id[lane]);
    M = __ldcg(&parts[0].m2);
    S = __ldcg(&parts[0].s);
    for (int k = 1; k < p.P; ++k) {
      bitonic_merge(v, id, __ldcg(&parts[k].v[lane]), __ldcg(&parts[k].id[lane]), lane);
      lse_merge(M, S, __ldcg(&parts[k].m2), __ldcg(&parts[k].s));
    }
    if (lane == 0) p.counters[r] = 0u;
  }

  if (lane < K) {
    p.cand_id[r * K + lane] = id;
    p.cand_logit[r * K + lane] = v;
  }
  if (lane == 0) {
    const double l2 = static_cast<double>(M) + log2(static_cast<double>(S));
    p.lse[r] = static_cast<float>(l2 / static_cast<double>(LOG2E));
  }
}

// ------------------------------------------------------------------------------ host

struct K1Plan {
  int P;
  int64_t seg_bytes;
  size_t ws_bytes;
};

static int g_num_sms = 0;

static int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 148;
  }
  return g_num_sms;
}

K1Plan k1_plan(int64_t batch, int B, int64_t V, int esize) {
  K1Plan pl{1, 0, 0};
  const int64_t rows = batch * (B - 1);
  const int64_t row_bytes = V * esize;
  const int64_t stages = (row_bytes + K1_STAGE_BYTES - 1) / K1_STAGE_BYTES;
  const int64_t conc = int64_t(num_sms()) * 2;  // resident CTAs
  // Smallest P (1..64, at least one stage per segment) whose work fills whole waves
  // of resident CTAs to within 5%; otherwise the best-filled P.
  int bestP = 1;
  double best_eff = -1.0;
  const int64_t pmax = std::max<int64_t>(1, std::min<int64_t>(64, stages));
  for (int P = 1; P <= pmax; ++P) {
    const double waves = double(rows * P) / double(conc);
    const double eff = waves / std::ceil(waves);
    if (eff >= 0.95) {
      bestP = P;
      break;
    }
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      bestP = P;
    }
  }
  pl.P = bestP;
  const int64_t seg = (row_bytes + pl.P - 1) / pl.P;
  pl.seg_bytes = std::max<int64_t>(16, (seg + 15) / 16 * 16);
  if (pl.P > 1)
    pl.ws_bytes = size_t(rows * pl.P) * sizeof(K1Partial) + size_t(rows) * sizeof(unsigned) + 256;
  return pl;
}

size_t k1_workspace_bytes(int64_t batch, int B, int64_t V, int esize) {
  return k1_plan(batch, B, V, esize).ws_bytes;
}

cudaError_t k1_launch(const void* logits, int esize, int64_t batch, int B, int64_t V, int K,
                      int32_t* cand_id, float* cand_logit, float* lse, void* ws,
                      cudaStream_t stream) {
  const K1Plan pl = k1_plan(batch, B, V, esize);
  K1Params prm;
  prm.logits = static_cast<const char*>(logits);
  prm.batch = batch;
  prm.B = B;
  prm.V = V;
  prm.K = K;
  prm.P = pl.P;
  prm.seg_bytes = pl.seg_bytes;
  prm.cand_id = cand_id;
  prm.cand_logit = cand_logit;
  prm.lse = lse;
  prm.partials = nullptr;
  prm.counters = nullptr;
  const int64_t rows = batch * (B - 1);
  if (pl.P > 1) {
    prm.partials = static_cast<K1Partial*>(ws);
    prm.counters = reinterpret_cast<unsigned*>(static_cast<char*>(ws) +
                                               size_t(rows * pl.P) * sizeof(K1Partial));
    cudaError_t e = cudaMemsetAsync(prm.counters, 0, size_t(rows) * sizeof(unsigned), stream);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(static_cast<unsigned>(rows * pl.P));
  constexpr int dyn = K1_NSTAGES * K1_STAGE_BYTES;
  static bool attr_done = false;
  if (!attr_done) {
    cudaFuncSetAttribute(logit_pass_kernel<__nv_bfloat16>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
    cudaFuncSetAttribute(logit_pass_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         dyn);
    attr_done = true;
  }
  if (esize == 2)
    logit_pass_kernel<__nv_bfloat16><<<grid, K1_THREADS, dyn, stream>>>(prm);
  else
    logit_pass_kernel<float><<<grid, K1_THREADS, dyn, stream>>>(prm);
  note_launch();
  return cudaGetLastError();
}

cudaError_t k1_read_device_error(uint32_t* code) {
  uint32_t v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_err_k1, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_err_k1, &zero, sizeof(zero));
  *code |= v;
  return e;
}

// ------------------------------------------------------------------ allocation-free form
// Scratch for lilicorr_topk_lse_noalloc: the split-row partial results and their
// arrival counters, compiled into the library so that a caller needs no workspace.
// Every device that loads the library holds these bytes until the process exits.
constexpr size_t K1_STATIC_SCRATCH_BYTES = size_t(4) << 20;
static __device__ __align__(256) uint8_t g_k1_static_scratch[K1_STATIC_SCRATCH_BYTES];

static std::mutex g_static_scratch_mu;
static void* g_static_scratch_dev[128] = {};  // device address of the array, per device

// Device address of the static scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once per device
// (with that device current) and cached.
static cudaError_t k1_static_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_static_scratch_mu);
  if (!g_static_scratch_dev[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_k1_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_scratch_dev[dev] = p;
  }
  *ptr = g_static_scratch_dev[dev];
  return cudaSuccess;
}

}  // namespace lilicorr

extern "C" lilicorr_status lilicorr_topk_lse_noalloc(const void* logits, lilicorr_dtype ldtype,
                                                     int64_t batch, int32_t B, int64_t V,
                                                     int32_t K, int32_t* cand_id,
                                                     float* cand_logit, float* lse,
                                                     void* stream) {
  using namespace lilicorr;
  if (!logits || !cand_id || !cand_logit || !lse) return LILICORR_ERR_INVALID_ARG;
  if (batch < 1 || B < 2 || V < 1 || V > (int64_t(1) << 31) - 2 || K < 1 || K > 32 || K > V)
    return LILICORR_ERR_INVALID_ARG;
  if (ldtype != LILICORR_F32 && ldtype != LILICORR_BF16) return LILICORR_ERR_INVALID_ARG;
  const int es = ldtype == LILICORR_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(logits) % es) return LILICORR_ERR_INVALID_ARG;
  if (V * es > (int64_t(1) << 31) - 64) return LILICORR_ERR_INVALID_ARG;
  const size_t need = k1_workspace_bytes(batch, B, V, es);
  if (need > K1_STATIC_SCRATCH_BYTES) {
    char msg[160];
    snprintf(msg, sizeof(msg),
             "lilicorr_topk_lse_noalloc: this shape needs %zu bytes of scratch; the static "
             "scratch holds %zu (use lilicorr_topk_lse with a workspace)",
             need, K1_STATIC_SCRATCH_BYTES);
    set_last_error(msg);
    return LILICORR_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  cudaError_t e = k1_static_scratch(&scratch);
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return LILICORR_ERR_CUDA;
  }
  // k1_launch zeroes the arrival counters inside the scratch before the kernel runs.
  e = k1_launch(logits, es, batch, B, V, K, cand_id, cand_logit, lse, scratch,
                static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return LILICORR_ERR_CUDA;
  }
  return LILICORR_OK;
}
