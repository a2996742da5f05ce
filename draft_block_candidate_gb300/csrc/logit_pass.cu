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
// copies (cp.async.bulk, 32 KB stages, 3 in flight, 2 CTAs per SM).  A producer warp
// refills a ring slot as soon as the 16 consumer warps have each released it (an
// mbarrier per slot; no CTA-wide barrier while streaming).  Every consumer thread copies
// its four 16-byte chunks of a stage into registers, takes their maxima and releases the
// slot at once; the rest of the stage's work runs from registers:
//   * online log-sum-exp in base 2: the running maximum is raised once per stage, then
//     packed f32x2 FFMA / FADD around one ex2 per element (two partial sums per thread);
//   * top-K: each consumer warp keeps its own running top-32 (value, id) pairs, sorted
//     across its lanes.  After a stage one vote compares every thread's stage maximum
//     with the warp's threshold, the better of its own K-th entry and a CTA-wide floor.
//     Only on a hit are the hit chunks unpacked and their elements at or above the
//     threshold appended to the warp's buffer, which is folded in 32 at a time (warp
//     bitonic sort + bitonic merge).
//   * the CTA floor is the K-th largest of 32 thread-group running maxima (of 64 above
//     K = 16; K distinct elements are at least that large).  After stage 0 the consumer
//     warps meet once so that the first floor covers the whole stage; afterwards the
//     producer warp raises it after every refill, and every fold raises it to the warp's
//     own K-th entry.
// At the end every warp offers its K-th entry to the floor; only queue and buffer entries
// at or above the final floor are gathered into one list, placed by rank (or folded by
// one warp when long).
// Rows are split into P segments only when fewer than about 90 rows are given (a single
// request); the last CTA of a row (atomic counter, no waiting) merges the P partials.
#include <float.h>
#include <limits.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <mutex>

#include "kernels.cuh"

namespace lilicorr {

static __device__ uint32_t g_err_k1;

constexpr int K1_CWARPS = 16;                      // consumer warps
constexpr int K1_CTHREADS = 32 * K1_CWARPS;
constexpr int K1_THREADS = K1_CTHREADS + 32;       // + one producer warp
#ifndef K1_MIN_BLOCKS
#define K1_MIN_BLOCKS 2
#endif
#ifndef K1_STAGE_KB
#define K1_STAGE_KB 32
#endif
#ifndef K1_POLL_NS
#define K1_POLL_NS 64
#endif
constexpr int K1_STAGE_BYTES = K1_STAGE_KB * 1024;
#ifndef K1_NST
#define K1_NST 3
#endif
constexpr int K1_NSTAGES = K1_NST;
constexpr int K1_CPT = K1_STAGE_BYTES / 16 / K1_CTHREADS;  // 16-byte chunks per consumer per stage
constexpr int KQ = 32;                                      // queue slots per warp
constexpr float LOG2E = 1.4426950408889634f;
constexpr float M2_INIT = -1e30f;                           // "no element yet", finite

// Natural-log lse of a base-2 pair (M, S), sum = S 2^M: (M + log2 S) / LOG2E, in float
// with one rounding's worth of care.  S = f 2^e with f in [0.5, 1), so log2 S = e + log2 f
// (the float log2 f within one ulp of a value below 1 in magnitude).  M + e is formed
// exactly as a head s and tail t (two-sum), the tail takes log2 f, and the pair is scaled
// by the reciprocal of the same float LOG2E that scaled the logits, held as a head and
// tail float: the head product exactly by an FMA, the rest added before the one final
// rounding.  Rounding-named intrinsics keep the compiler from contracting the steps.
__device__ __forceinline__ float lse_of(float M, float S) {
  constexpr double INV_L = 1.0 / static_cast<double>(LOG2E);
  constexpr float IH = static_cast<float>(INV_L);
  constexpr float IL = static_cast<float>(INV_L - static_cast<double>(IH));
  int e;
  const float f = frexpf(S, &e);
  const float E = static_cast<float>(e);
  const float s = __fadd_rn(M, E);
  const float bb = __fsub_rn(s, M);
  const float t = __fadd_rn(__fsub_rn(M, __fsub_rn(s, bb)), __fsub_rn(E, bb));
  const float lo = __fadd_rn(t, log2f(f));
  const float ph = __fmul_rn(s, IH);
  const float pe = __fmaf_rn(s, IH, -ph);
  return __fadd_rn(ph, __fadd_rn(pe, __fmaf_rn(s, IL, __fmul_rn(lo, IH))));
}

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
  int64_t row_stride;  // elements between consecutive rows (V for a whole-vocabulary pass)
  int id_offset;       // added to every candidate id (a vocabulary shard's first id)
  char* records;       // vocabulary-shard mode: packed per-row records instead of outputs
  long long wait_limit;  // SM cycles after which a wait gives up (WAIT_LIMIT_CYCLES)
  int withhold_first;    // self-check only: stage 0's copy is announced but never issued
  int64_t prefetch_ahead;  // > 0: at its last refill a CTA prefetches into L2 the first
                           // stage of unit blockIdx + prefetch_ahead (co-resident CTAs)
};

// Packed per-row record of a vocabulary shard: {m2, s, v[K], id[K]}, K * 8 + 8 bytes.
// m2 = max * log2(e) of the shard's logits, s = sum 2^(x log2(e) - m2); v / id its top-K
// (value desc, global id asc).
__host__ __device__ constexpr size_t k1_record_bytes(int K) { return 8 + size_t(K) * 8; }

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
// sorted 32-entry queue q: sort the 32 candidates, bitonic-merge, keep the best 32.
// Skipped when no lane beats the queue's K-th entry.
__device__ __forceinline__ void queue_absorb(WarpQueue& q, float v, int id, int lane, int K) {
  if (!__any_sync(FULL_MASK, better(v, id, q.tv, q.tid))) return;
  warp_sort_pairs(v, id, lane);
  bitonic_merge(q.qv, q.qid, v, id, lane);
  q.tv = __shfl_sync(FULL_MASK, q.qv, K - 1);
  q.tid = __shfl_sync(FULL_MASK, q.qid, K - 1);
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

// Element j of a 16-byte chunk (8 bf16 or 4 f32).
template <int NV>
__device__ __forceinline__ float elem_of(const uint4 w, int j) {
  const int k = NV == 8 ? j >> 1 : j;
  const uint32_t wd = k == 0 ? w.x : k == 1 ? w.y : k == 2 ? w.z : w.w;
  if constexpr (NV == 8) return __uint_as_float((j & 1) ? (wd & 0xffff0000u) : (wd << 16));
  else return __uint_as_float(wd);
}

constexpr int K1_WCAP = 64;    // per-warp candidate buffer entries
// Thread groups whose running maxima give the CTA floor: 32 (16 threads each) up to
// K = 16; 64 (8 threads each) above, where the K-th largest of 32 would be loose.
template <bool WIDE>
__host__ __device__ constexpr int k1_groups() { return WIDE ? 64 : 32; }
constexpr int K1_WIDE_ABOVE_K = 16;
// Final candidate list: at most every queue entry (17 warps) and every buffer entry.
constexpr int K1_UCAP = (K1_CWARPS + 1) * KQ + K1_CWARPS * K1_WCAP;
static_assert(K1_UCAP * 8 <= K1_STAGE_BYTES, "final candidate list must fit in one ring slot");
static_assert(K1_WCAP >= KQ, "a warp buffer holds the sorted result at the end");

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Maximum of one 16-byte chunk (8 bf16 compared as packed pairs, or 4 f32).
template <typename T>
__device__ __forceinline__ float chunk_max(const uint4 w);
template <>
__device__ __forceinline__ float chunk_max<__nv_bfloat16>(const uint4 w) {
  const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&w.x),
                                   *reinterpret_cast<const __nv_bfloat162*>(&w.y));
  const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&w.z),
                                   *reinterpret_cast<const __nv_bfloat162*>(&w.w));
  const __nv_bfloat162 c = __hmax2(a, b);
  return fmaxf(__low2float(c), __high2float(c));
}
template <>
__device__ __forceinline__ float chunk_max<float>(const uint4 w) {
  return fmaxf(max3f(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z)),
               __uint_as_float(w.w));
}

// Consumer-side log-sum-exp of one stage held in registers (chunk words w, validity bits,
// the thread's maximum smax over its chunks).  The running maximum m2 is raised once per stage; when it rises it
// is offered to the thread group's maximum in shared memory.  The sum is kept as two
// partial sums (even / odd elements) updated with packed f32x2 arithmetic.
template <int NV>
__device__ __forceinline__ void lse_stage(const uint4 (&w)[K1_CPT], unsigned valid, float smax,
                                          float& m2, float2& s2, int* gmax) {
  const float sm2 = smax * LOG2E;
  if (sm2 > m2) {
    const float sc = ex2(m2 - sm2);
    s2 = __fmul2_rn(s2, make_float2(sc, sc));
    m2 = sm2;
    atomicMax(gmax, float_key(smax));
  }
  const float2 l2 = make_float2(LOG2E, LOG2E);
  const float2 nm = make_float2(-m2, -m2);
#pragma unroll
  for (int i = 0; i < K1_CPT; ++i) {
    if ((valid >> i) & 1u) {
      float x[NV];
      unpack16<NV>(w[i], x);
#pragma unroll
      for (int j = 0; j < NV; j += 2) {
        const float2 y = __ffma2_rn(make_float2(x[j], x[j + 1]), l2, nm);
        s2 = __fadd2_rn(s2, make_float2(ex2(y.x), ex2(y.y)));
      }
    }
  }
}

// The 16-byte aligned byte range [lo, hi) of p.logits that unit u (row u / P, segment
// u % P) streams.
__device__ __forceinline__ void k1_unit_range(const K1Params& p, int64_t u, int es, int64_t& lo,
                                              int64_t& hi) {
  const int64_t r = u / p.P;
  const int64_t seg = u % p.P;
  const int64_t row_start = ((r / (p.B - 1)) * p.B + r % (p.B - 1) + 1) * p.row_stride * es;
  const int64_t row_end = row_start + p.V * es;
  const uintptr_t base = reinterpret_cast<uintptr_t>(p.logits);
  int64_t bs = static_cast<int64_t>(((base + row_start + 15) & ~uintptr_t(15)) - base);
  int64_t be = static_cast<int64_t>(((base + row_end) & ~uintptr_t(15)) - base);
  if (bs >= be) bs = be = row_end;
  lo = i64min(be, bs + seg * p.seg_bytes);
  hi = i64min(be, lo + p.seg_bytes);
}

__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Warp-uniform: the K-th largest of the group maxima.  Each group's maximum is an element
// of a distinct set of threads, so K elements of the segment are at least this large: a
// valid inclusive floor for the K-th largest value.  32 groups: one per lane, one sort.
// 64 groups: lane l holds groups l and l + 32; the first half sorted descending and the
// second ascending give, lane by lane, the larger of the two as a bitonic sequence of the
// 32 largest, which one merge sorts.
template <bool WIDE>
__device__ __forceinline__ float group_floor(const int* gmax, int lane, int K) {
  float g = key_float(*reinterpret_cast<const volatile int*>(&gmax[lane]));
  if constexpr (!WIDE) {
    if (K == 1) {
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) g = fmaxf(g, __shfl_xor_sync(FULL_MASK, g, o));
      return g;
    }
    return __shfl_sync(FULL_MASK, warp_sort_desc(g, lane), K - 1);
  } else {
    const float h = key_float(*reinterpret_cast<const volatile int*>(&gmax[lane + 32]));
    g = warp_sort_desc(g, lane);
    float c = fmaxf(g, __shfl_sync(FULL_MASK, warp_sort_desc(h, lane), 31 - lane));
#pragma unroll
    for (int j = 16; j >= 1; j >>= 1) {
      const float o = __shfl_xor_sync(FULL_MASK, c, j);
      c = (lane & j) == 0 ? fmaxf(c, o) : fminf(c, o);
    }
    return __shfl_sync(FULL_MASK, c, K - 1);
  }
}

template <typename T, bool WIDE>
__global__ void __launch_bounds__(K1_THREADS, K1_MIN_BLOCKS) logit_pass_kernel(const K1Params p) {
  constexpr int ES = sizeof(T);
  constexpr int NV = 16 / ES;
  constexpr int K1_GROUPS = k1_groups<WIDE>();
  extern __shared__ __align__(128) uint8_t k1_dyn_smem[];
  uint8_t(*stage)[K1_STAGE_BYTES] = reinterpret_cast<uint8_t(*)[K1_STAGE_BYTES]>(k1_dyn_smem);
  __shared__ __align__(8) uint64_t full_bar[K1_NSTAGES], empty_bar[K1_NSTAGES];
  __shared__ float s_bv[K1_CWARPS][K1_WCAP];  // per-warp candidate buffers
  __shared__ int s_bi[K1_CWARPS][K1_WCAP];
  __shared__ int s_ucnt;                       // entries of the final candidate list
  __shared__ int s_wcnt[K1_CWARPS];
  __shared__ int s_gmax[K1_GROUPS];  // float_key of each thread group's running maximum
  __shared__ int s_floor;            // float_key of the CTA floor (atomic max)
  __shared__ float s_m2[K1_CWARPS + 1], s_s[K1_CWARPS + 1];
  __shared__ int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.K;
  const int64_t u = blockIdx.x;
  const int64_t r = u / p.P;
  const int seg = static_cast<int>(u % p.P);
  const int64_t b = r / (p.B - 1);
  const int64_t s_slot = r % (p.B - 1) + 1;

  // Row geometry in bytes relative to p.logits; body = 16-byte aligned part.
  const int64_t row_start = (b * p.B + s_slot) * p.row_stride * ES;
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
    for (int i = 0; i < K1_NSTAGES; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], K1_CWARPS);
    }
    fence_mbar_init();
    s_abort = 0;
    s_ucnt = 0;
    s_floor = float_key(-INFINITY);
  }
  if (tid < K1_GROUPS) s_gmax[tid] = float_key(-INFINITY);
  if (tid < K1_CWARPS) s_wcnt[tid] = 0;
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  float m2 = M2_INIT, ssum = 0.f;
  WarpQueue q;  // this warp's running top-32 (one entry per lane, sorted)
  q.init();
  int issued = 0;  // copies issued (producer warp, lane 0)

  if (warp == K1_CWARPS) {
    // ================= producer warp =================
    auto issue = [&](int st) {
      const int off = st * K1_STAGE_BYTES;
      const int sl = st % K1_NSTAGES;
      const uint32_t bytes = static_cast<uint32_t>(min(K1_STAGE_BYTES, seg_bytes - off));
      mbar_arrive_expect_tx(&full_bar[sl], bytes);
      if (!(p.withhold_first && st == 0))
        bulk_g2s(stage[sl], p.logits + seg_lo + off, bytes, &full_bar[sl]);
      issued = st + 1;
    };
    if (lane == 0)
      for (int st = 0; st < min(K1_NSTAGES, nstages); ++st) issue(st);
    // Unaligned head (segment 0) and tail (last segment): one element per lane.
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
      if (has) lse_merge(m2, ssum, xv * LOG2E, 1.0f);
      queue_absorb(q, xv, has ? static_cast<int>(first / ES - row_elem0) + lane : INT_MAX, lane,
                   K);
    }
    // Refill each slot as soon as every consumer warp has released it (the wait only
    // polls, so a released slot is refilled at once); after each refill the CTA floor is
    // raised to the K-th largest of the group maxima.
    for (int st = K1_NSTAGES; st < nstages; ++st) {
      const int sl = st % K1_NSTAGES;
      const uint32_t par = ((st / K1_NSTAGES) - 1) & 1;
      const long long t0 = clock64();
      int ready = 0;
      for (;;) {
        if (lane == 0) {
          if (mbar_test_wait(&empty_bar[sl], par)) {
            ready = 1;
          } else if (s_abort) {
            ready = 2;
          } else if (clock64() - t0 > p.wait_limit) {
            atomicOr(&g_err_k1, ERR_K1_EMPTY_WAIT);
            s_abort = 1;
            ready = 2;
          }
        }
        ready = __shfl_sync(FULL_MASK, ready, 0);
        if (ready != 0) break;
        __nanosleep(K1_POLL_NS);
      }
      if (ready == 2) break;
      if (lane == 0) {
        issue(st);
        // the first stage of the unit a CTA will likely start on this slot when this one
        // ends, into L2 (a hint: its first copy then waits on L2, not on DRAM)
        if (st == nstages - 1 && p.prefetch_ahead > 0 && u + p.prefetch_ahead < gridDim.x) {
          int64_t lo, hi;
          k1_unit_range(p, u + p.prefetch_ahead, ES, lo, hi);
          if (hi > lo) prefetch_l2(p.logits + lo, static_cast<uint32_t>(i64min(K1_STAGE_BYTES, hi - lo)));
        }
      }
      {
        const float f = group_floor<WIDE>(s_gmax, lane, K);
        if (lane == 0) atomicMax(&s_floor, float_key(f));
      }
    }
  } else {
    // ================= consumer warps =================
    float* bv = s_bv[warp];
    int* bi = s_bi[warp];
    int* gmax = &s_gmax[tid / (K1_CTHREADS / K1_GROUPS)];
    int* wcnt = &s_wcnt[warp];
    int wprev = 0;  // *wcnt as this warp last left it (only this warp appends)
    float2 s2 = make_float2(0.f, 0.f);  // partial sums of this thread's exponentials

    // Candidates of stage st (chunk maxima cmx, validity bits vmask, chunk words from
    // chunk_at(i)): compare with the threshold tv, the better of the warp's K-th entry and
    // the CTA floor fl; append the elements of hit chunks at or above tv to the warp
    // buffer (a superset of those that beat the threshold in (value, id) order: the
    // queue's folds order ties by id); fold the buffer into the queue 32 entries at a time.
    auto check_stage = [&](int st, const float (&cmx)[K1_CPT], unsigned vmask, float smax,
                           float fl, auto&& chunk_at) {
      const int soff = st * K1_STAGE_BYTES;
      const float tv = fmaxf(q.tv, fl);
      if (!__any_sync(FULL_MASK, smax >= tv)) return;
      const int prev = wprev;
#pragma unroll
      for (int i = 0; i < K1_CPT; ++i) {
        if (((vmask >> i) & 1u) && cmx[i] >= tv) {
          const int c = tid + i * K1_CTHREADS;
          float x[NV];
          unpack16<NV>(chunk_at(i), x);
          const int id0 = seg_elem0 + (soff + c * 16) / ES;
#pragma unroll
          for (int j = 0; j < NV; ++j)
            if (x[j] >= tv) {
              const int idx = atomicAdd(wcnt, 1);
              if (idx < K1_WCAP) {
                bv[idx] = x[j];
                bi[idx] = id0 + j;
              }
            }
        }
      }
      __syncwarp();
      int cnt = *reinterpret_cast<volatile int*>(wcnt);
      if (cnt < 32) {
        wprev = cnt;
        return;
      }
      if (cnt > K1_WCAP) {
        // Too many ties for the buffer: fold the earlier stages' entries, then this
        // stage's chunks element by element; the buffer is dropped.
        const bool has = lane < prev;
        queue_absorb(q, has ? bv[lane] : -INFINITY, has ? bi[lane] : INT_MAX, lane, K);
        // (a rolled loop: one copy of the fold keeps the kernel's code small)
#pragma unroll 1
        for (int e = 0; e < K1_CPT * NV; ++e) {
          const int i = e / NV;
          uint4 cw = chunk_at(0);
#pragma unroll
          for (int k = 1; k < K1_CPT; ++k)
            if (i == k) cw = chunk_at(k);
          const bool hv = (vmask >> i) & 1u;
          const int id = seg_elem0 + (soff + (tid + i * K1_CTHREADS) * 16) / ES + e % NV;
          queue_absorb(q, hv ? elem_of<NV>(cw, e % NV) : -INFINITY, hv ? id : INT_MAX, lane, K);
        }
        cnt = 0;
      } else {
        while (cnt >= 32) {
          const float v = bv[lane];
          const int id = bi[lane];
          const bool more = lane + 32 < cnt;
          const float v2 = more ? bv[lane + 32] : 0.f;
          const int i2 = more ? bi[lane + 32] : 0;
          __syncwarp();
          if (more) {
            bv[lane] = v2;
            bi[lane] = i2;
          }
          cnt -= 32;
          queue_absorb(q, v, id, lane, K);
          __syncwarp();
        }
      }
      __syncwarp();
      wprev = cnt;
      if (lane == 0) {
        *wcnt = cnt;
        if (q.tv != -INFINITY) atomicMax(&s_floor, float_key(q.tv));
      }
    };

    for (int st = 0; st < nstages; ++st) {
      const int sl = st % K1_NSTAGES;
      if (!mbar_wait_bounded(&full_bar[sl], (st / K1_NSTAGES) & 1, &g_err_k1, ERR_K1_FULL_WAIT,
                             p.wait_limit))
        s_abort = 1;
      if (st > 0 && s_abort) break;  // stage 0 first meets the other consumer warps
      const int nbytes = min(K1_STAGE_BYTES, seg_bytes - st * K1_STAGE_BYTES);
      const uint8_t* sbuf = stage[sl];
      // This thread's chunks of the stage into registers, and their maxima.
      uint4 w[K1_CPT];
      float cm[K1_CPT];
      unsigned valid = 0;  // bit i: this thread has chunk i of the stage
#pragma unroll
      for (int i = 0; i < K1_CPT; ++i) {
        const int c = tid + i * K1_CTHREADS;
        w[i] = make_uint4(0u, 0u, 0u, 0u);
        if (c * 16 < nbytes) {
          valid |= 1u << i;
          w[i] = *reinterpret_cast<const uint4*>(sbuf + c * 16);
        }
      }
#pragma unroll
      for (int i = 0; i < K1_CPT; ++i) cm[i] = ((valid >> i) & 1u) ? chunk_max<T>(w[i]) : -INFINITY;
      // The stage is in registers: release the slot to the producer at once.
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[sl]);

      float smax = cm[0];  // this thread's maximum of the stage
#pragma unroll
      for (int i = 1; i < K1_CPT; ++i) smax = fmaxf(smax, cm[i]);
      float fl;
      if (st == 0) {
        // First CTA floor: every thread offers its stage-0 maximum to its group, the
        // consumer warps meet, and each takes the K-th largest of the group maxima.
        if (smax != -INFINITY) atomicMax(gmax, float_key(smax));
        named_bar_sync(1, K1_CTHREADS);
        if (s_abort) break;
        fl = group_floor<WIDE>(s_gmax, lane, K);
        if (warp == 0 && lane == 0) atomicMax(&s_floor, float_key(fl));
        lse_stage<NV>(w, valid, smax, m2, s2, gmax);
      } else {
        lse_stage<NV>(w, valid, smax, m2, s2, gmax);
        fl = key_float(*reinterpret_cast<volatile int*>(&s_floor));
      }
      check_stage(st, cm, valid, smax, fl, [&](int i) { return w[i]; });
    }
    ssum = s2.x + s2.y;
  }

  // ---- CTA reduction.  Log-sum-exp: within each warp, then across the warps.  Top-K:
  // every warp offers its K-th queue entry to the CTA floor; then only queue and buffer
  // entries at or above that final floor can be among the segment's K best, and they are
  // gathered into one list (in ring slot 0, free once every stage is consumed) that
  // warp 0 folds.
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float om = __shfl_xor_sync(FULL_MASK, m2, o);
    const float os = __shfl_xor_sync(FULL_MASK, ssum, o);
    lse_merge(m2, ssum, om, os);
  }
  if (lane == 0) {
    s_m2[warp] = m2;
    s_s[warp] = ssum;
    if (q.tv != -INFINITY) atomicMax(&s_floor, float_key(q.tv));
  }
  __syncthreads();
  if (s_abort) {
    // let every copy still in flight land before the CTA exits
    if (warp == K1_CWARPS && lane == 0)
      for (int st = max(0, issued - K1_NSTAGES); st < issued; ++st)
        mbar_wait_bounded(&full_bar[st % K1_NSTAGES], (st / K1_NSTAGES) & 1, &g_err_k1,
                          ERR_K1_DRAIN, p.wait_limit);
    return;
  }
  float* uv = reinterpret_cast<float*>(stage[0]);
  int* ui = reinterpret_cast<int*>(stage[0] + K1_UCAP * sizeof(float));
  {
    const float F = key_float(s_floor);
    if (q.qid != INT_MAX && q.qv >= F) {
      const int k = atomicAdd(&s_ucnt, 1);
      uv[k] = q.qv;
      ui[k] = q.qid;
    }
    if (warp < K1_CWARPS) {
      const int cnt = min(s_wcnt[warp], K1_WCAP);
      for (int j = lane; j < cnt; j += 32) {
        const float bvj = s_bv[warp][j];
        if (bvj >= F) {
          const int k = atomicAdd(&s_ucnt, 1);
          uv[k] = bvj;
          ui[k] = s_bi[warp][j];
        }
      }
    }
  }
  __syncthreads();
  if (warp != 0) return;

  const int nu = s_ucnt;
  float v = -INFINITY;
  int id = INT_MAX;
  if (nu <= 64) {
    // The list's entries are distinct (value, id) pairs, so under (value desc, id asc)
    // each has its own rank, the number of entries better than it: each lane ranks its
    // one or two entries and places those ranked below KQ in warp 0's buffer (no longer
    // read), which then holds the sorted result.
    float* rv = s_bv[0];
    int* ri = s_bi[0];
    const bool h0 = lane < nu, h1 = lane + 32 < nu;
    const float c0 = h0 ? uv[lane] : 0.f, c1 = h1 ? uv[lane + 32] : 0.f;
    const int i0 = h0 ? ui[lane] : 0, i1 = h1 ? ui[lane + 32] : 0;
    int r0 = 0, r1 = 0;
#pragma unroll 4
    for (int j = 0; j < nu; ++j) {
      const float vj = uv[j];
      const int ij = ui[j];
      r0 += better(vj, ij, c0, i0) ? 1 : 0;
      r1 += better(vj, ij, c1, i1) ? 1 : 0;
    }
    rv[lane] = -INFINITY;
    ri[lane] = INT_MAX;
    __syncwarp();
    if (h0 && r0 < KQ) {
      rv[r0] = c0;
      ri[r0] = i0;
    }
    if (h1 && r1 < KQ) {
      rv[r1] = c1;
      ri[r1] = i1;
    }
    __syncwarp();
    v = rv[lane];
    id = ri[lane];
  } else {
    WarpQueue fq;
    fq.init();
    for (int b0 = 0; b0 < nu; b0 += 32) {
      const bool has = b0 + lane < nu;
      queue_absorb(fq, has ? uv[b0 + lane] : -INFINITY, has ? ui[b0 + lane] : INT_MAX, lane, K);
    }
    v = fq.qv;
    id = fq.qid;
  }
  float M = lane <= K1_CWARPS ? s_m2[lane] : M2_INIT;
  float S = lane <= K1_CWARPS ? s_s[lane] : 0.f;
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

  if (p.records) {
    char* rec = p.records + r * k1_record_bytes(K);
    if (lane == 0) {
      reinterpret_cast<float*>(rec)[0] = M;
      reinterpret_cast<float*>(rec)[1] = S;
    }
    if (lane < K) {
      reinterpret_cast<float*>(rec + 8)[lane] = v;
      reinterpret_cast<int32_t*>(rec + 8 + 4 * K)[lane] = id == INT_MAX ? INT_MAX : id + p.id_offset;
    }
    return;
  }
  if (lane < K) {
    p.cand_id[r * K + lane] = id + p.id_offset;
    p.cand_logit[r * K + lane] = v;
  }
  if (lane == 0) p.lse[r] = lse_of(M, S);
}

// Merge of n vocabulary-shard records per row (one warp per row): the shards' sorted
// top-K lists by bitonic merge under the same (value desc, id asc) order, and their
// (m2, s) pairs by the online log-sum-exp rule.  Shards hold disjoint ids, so the result
// is the top-K of the whole row.
__global__ void __launch_bounds__(128) k1_merge_kernel(const char* __restrict__ records,
                                                       int n, int64_t rows, int K,
                                                       int32_t* __restrict__ cand_id,
                                                       float* __restrict__ cand_logit,
                                                       float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int64_t r = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const size_t rb = k1_record_bytes(K);
  float v = -INFINITY, M = M2_INIT, S = 0.f;
  int id = INT_MAX;
  for (int j = 0; j < n; ++j) {
    const char* rec = records + (int64_t(j) * rows + r) * rb;
    const float bv = lane < K ? __ldg(reinterpret_cast<const float*>(rec + 8) + lane) : -INFINITY;
    const int bi = lane < K ? __ldg(reinterpret_cast<const int32_t*>(rec + 8 + 4 * K) + lane) : INT_MAX;
    bitonic_merge(v, id, bv, bi, lane);
    lse_merge(M, S, __ldg(reinterpret_cast<const float*>(rec)), __ldg(reinterpret_cast<const float*>(rec) + 1));
  }
  if (lane < K) {
    cand_id[r * K + lane] = id;
    cand_logit[r * K + lane] = v;
  }
  if (lane == 0) lse[r] = lse_of(M, S);
}

// ------------------------------------------------------------------------------ host

struct K1Plan {
  int P;
  int64_t seg_bytes;
  size_t ws_bytes;
};

K1Plan k1_plan(int64_t batch, int B, int64_t V, int esize) {
  K1Plan pl{1, 0, 0};
  const int64_t rows = batch * (B - 1);
  const int64_t row_bytes = V * esize;
  const int64_t stages = (row_bytes + K1_STAGE_BYTES - 1) / K1_STAGE_BYTES;
  // A row is split into P segments only when there are too few rows to keep about 90
  // CTAs streaming.  Measured on GB300 at V = 151,936 bf16 (P = 1 vs the best split):
  // 15 rows 18.7 vs 15.7 us (P = 6); 60 rows 17.4 us, unsplit best; from 240 rows on,
  // every split is slower than one CTA per row (960 rows: 74 us unsplit, 104 us at P = 2,
  // 145 us at P = 4), because a CTA's start, first-stage latency and final gather cost
  // about as much as streaming a third of a row.
  const int64_t want = rows >= K1_SPLIT_BELOW_ROWS ? 1 : K1_SPLIT_BELOW_ROWS / rows;
  pl.P = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({want, 64, stages})));
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
                      cudaStream_t stream, int64_t row_stride, int id_offset, void* records,
                      long long wait_limit, bool withhold_first) {
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
  prm.row_stride = row_stride > 0 ? row_stride : V;
  prm.id_offset = id_offset;
  prm.records = static_cast<char*>(records);
  prm.wait_limit = wait_limit;
  prm.withhold_first = withhold_first ? 1 : 0;
  {
    const int64_t resident = int64_t(K1_MIN_BLOCKS) * device_sm_count();
    prm.prefetch_ahead = batch * (B - 1) * pl.P > resident ? resident : 0;
  }
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
  const bool wide = K > K1_WIDE_ABOVE_K;
  void (*kern)(const K1Params) =
      esize == 2 ? (wide ? logit_pass_kernel<__nv_bfloat16, true> : logit_pass_kernel<__nv_bfloat16, false>)
                 : (wide ? logit_pass_kernel<float, true> : logit_pass_kernel<float, false>);
  {
    cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), dyn);
    if (e != cudaSuccess) return e;
  }
  const cudaError_t e = launch_k(kern, grid, dim3(K1_THREADS), dyn, stream, prm);
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaGetLastError();
}

size_t k1_shard_record_bytes(int K) { return k1_record_bytes(K); }

cudaError_t k1_merge_launch(const void* records, int n, int64_t rows, int K, int32_t* cand_id,
                            float* cand_logit, float* lse, cudaStream_t stream) {
  const int wpb = 4;
  k1_merge_kernel<<<static_cast<unsigned>((rows + wpb - 1) / wpb), 32 * wpb, 0, stream>>>(
      static_cast<const char*>(records), n, rows, K, cand_id, cand_logit, lse);
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

// Self-check of the bounded waits: one row that fits one stage, its only copy announced
// to the stage's barrier but never issued.  The consumer warps' wait and the producer's
// final drain both give up after `limit_cycles`, set their site bits and return; no
// output is written.  Nothing else is in flight, so the kernel ends cleanly.
extern "C" lilicorr_status lilicorr_diag_wait_timeout(const void* logits, int64_t V,
                                                      uint32_t limit_cycles, int32_t* cand_id,
                                                      float* cand_logit, float* lse,
                                                      void* stream) {
  using namespace lilicorr;
  if (!logits || !cand_id || !cand_logit || !lse) return LILICORR_ERR_INVALID_ARG;
  if (V < 1 || V * 2 > K1_STAGE_BYTES || reinterpret_cast<uintptr_t>(logits) % 16)
    return LILICORR_ERR_INVALID_ARG;
  if (limit_cycles < 1000u || limit_cycles > 100000000u) return LILICORR_ERR_INVALID_ARG;
  const cudaError_t e = k1_launch(logits, 2, 1, 2, V, 1, cand_id, cand_logit, lse, nullptr,
                                  static_cast<cudaStream_t>(stream), 0, 0, nullptr,
                                  static_cast<long long>(limit_cycles), true);
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return LILICORR_ERR_CUDA;
  }
  return LILICORR_OK;
}
