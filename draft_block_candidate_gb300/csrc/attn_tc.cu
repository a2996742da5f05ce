// Lattice self-attention of step a3 on the 5th-generation tensor cores (head dim 64,
// up to 256 lattice tokens per block).
//
// Per head: softmax_j(q_i . k_j / sqrt(dh) + dist[slot_j - slot_i + B_max - 2]
//                     + [slot_i == slot_j] * same) v_j          (LiLiCorr App. A)
// over all tokens of the block (bidirectional, no mask).
//
// Persistent: one CTA per SM walks the (128-query tile, block, head) items, head-major (a
// CTA keeps one head's bias table for several items; the two query tiles of a (block,
// head) run on neighbouring CTAs at the same time, so its K / V tiles are read from DRAM
// once), 18 warps:
//   warp 0     TMA: Q (128 x 64), K and V (256 x 64), each as bf16 hi and lo, 128-byte
//              swizzle; the next item's Q and K load as soon as this item's S is formed,
//              each key half of its V as soon as this item's product over that half is
//              done; owns the TMEM allocation (S / P: 256 columns, O': 2 x 128 columns)
//   warp 1     MMA, per item: S0 / S1 = Q K^T over key halves 0-127 / 128-255 (three
//              split products), then both P V halves, then the next item's S0 and S1
//              O' = Ph [Vh | Vl] + Pl [Vh | Vl] (N 128: the hi and lo tiles of V are the two
//              64-column atoms of one MN-major operand) with P read from TMEM;
//              O = O'[:, 0:64] + O'[:, 64:128]
//   warps 2-17 four warps per query-row quarter, each taking a quarter of the keys:
//              pass 1 scales, adds the slot bias (a per-query-slot row of the head's
//              bias table, -inf beyond the block; one 16-byte load per four keys) and
//              takes the row max (the four parts combined through shared memory); pass 2
//              recomputes the biased logit, forms p = 2^(x - max) and its sum and writes
//              p as packed bf16 hi / lo over the logits it came from; the epilogue
//              divides this warp's 16 columns of O by the sum, splits them into a
//              swizzled shared-memory tile, and one thread per quarter stores the
//              quarter's 32 rows with a bulk tensor store (rows past the block clipped).
// Every mbarrier wait is bounded; on a timeout the CTA records it and still frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.cuh"

namespace lilicorr {

static __device__ uint32_t g_err_at;

constexpr int AT_DH = 64, AT_QT = 128, AT_KMAX = 256, AT_SOFT_WARPS = 16;
constexpr int AT_NSPLIT = AT_SOFT_WARPS / 4;      // softmax warps per 32-row quarter
constexpr int AT_OW = AT_DH / AT_NSPLIT;          // output columns per softmax warp
constexpr int AT_THREADS = 32 * (2 + AT_SOFT_WARPS);
constexpr int AT_TILE = 128 * 64 * 2;  // one [128 x 64] bf16 swizzled tile
constexpr int AT_SMEM = 12 * AT_TILE + 1024;  // + the bias table, sized per launch
constexpr int AT_SMEM_MAX = 227 * 1024 - 8 * 1024;  // dynamic share (static use < 8 KB)
constexpr int AT_BSTRIDE = AT_KMAX + 4;        // floats per bias-table row (bank offset)
constexpr uint32_t AT_TMEM_COLS = 512, AT_O_COL = 256, AT_O_W = 128;
constexpr float AT_LOG2E = 1.4426950408889634f;

enum AtErr : uint32_t {
  ERR_AT_QK = 1u << 0,
  ERR_AT_S = 1u << 1,
  ERR_AT_V = 1u << 2,
  ERR_AT_P = 1u << 3,
  ERR_AT_O = 1u << 4,
  ERR_AT_QKFREE = 1u << 5,
  ERR_AT_VFREE = 1u << 6,
  ERR_AT_OFREE = 1u << 7
};

__device__ __forceinline__ void at_tma(void* dst, const CUtensorMap* tm, int c0, int c1,
                                       uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void at_tma3(void* dst, const CUtensorMap* tm, int c0, int c1, int c2,
                                        uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void at_store4(const CUtensorMap* tm, const void* src, int c0, int c1,
                                          int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(tm)),
      "r"(smem_addr(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void at_store(const CUtensorMap* tm, const void* src, int c0, int c1,
                                         int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(tm)),
      "r"(smem_addr(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void at_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void at_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 128-byte-swizzle descriptor (K-major tiles of 64-element rows, or MN-major tiles whose
// rows are the K index); 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t at_desc(const void* p) {
  const uint64_t a = smem_addr(p);
  return ((a >> 4) & 0x3FFFull) | (1ull << 16) | ((1024ull >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}
// The same for an MN-major operand two atoms wide along N: [V hi | V lo], the lo tile
// 2 * AT_TILE bytes after the hi tile (leading-dimension byte offset).
__device__ __forceinline__ uint64_t at_desc_vhl(const void* p) {
  return at_desc(p) & ~(0x3FFFull << 16) | (uint64_t((2 * AT_TILE) >> 4) << 16);
}
__device__ __forceinline__ void at_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// A operand from TMEM (packed bf16 pairs, one row per lane), B from shared memory.
__device__ __forceinline__ void at_mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void at_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void at_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void at_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void at_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
__device__ __forceinline__ float at_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// idesc kind::f16, f32 D, bf16 A/B; b_mn selects an MN-major B operand.
__host__ __device__ constexpr uint32_t at_idesc(int M, int N, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn ? (1u << 16) : 0u) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// The four softmax warps of one 32-row quarter (named barriers 2-5).
__device__ __forceinline__ void quarter_sync(int q) {
  asm volatile("bar.sync %0, 128;" ::"r"(2 + q) : "memory");
}
__device__ __forceinline__ void at_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}
__device__ __forceinline__ void at_st16f(uint32_t taddr, const float (&v)[16]) {
  uint32_t u[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(v[i]);
  at_st16(taddr, u);
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// (query tile, block, head) of a CTA's items, head-major, advanced by the grid stride
// with carries instead of 64-bit divisions per item.
struct ItemPos {
  int qt, blk, h, dqt, dblk, dh, QT, batch;
  __device__ ItemPos(int64_t t, int64_t G, int QT_, int64_t batch_)
      : QT(QT_), batch(static_cast<int>(batch_)) {
    qt = static_cast<int>(t % QT);
    blk = static_cast<int>((t / QT) % batch_);
    h = static_cast<int>(t / (QT * batch_));
    dqt = static_cast<int>(G % QT);
    dblk = static_cast<int>((G / QT) % batch_);
    dh = static_cast<int>(G / (QT * batch_));
  }
  __device__ void next() {
    qt += dqt;
    int c = 0;
    if (qt >= QT) { qt -= QT; c = 1; }
    blk += dblk + c;
    c = 0;
    if (blk >= batch) { blk -= batch; c = 1; }
    h += dh + c;
  }
};

__device__ __forceinline__ void soft_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * AT_SOFT_WARPS) : "memory");
}

__global__ void __launch_bounds__(AT_THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ CUtensorMap tmo,
                   int S, int Kc, int H, int B_max, int heads, int64_t batch,
                   const float* __restrict__ dist_bias, const float* __restrict__ same_bias,
                   int dh) {
  extern __shared__ uint8_t at_smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(at_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQh = sm;                 // Q hi / lo: 1 tile each
  uint8_t* sQl = sm + AT_TILE;
  uint8_t* sKh = sm + 2 * AT_TILE;   // K hi / lo: 2 tiles each (256 keys)
  uint8_t* sKl = sm + 4 * AT_TILE;
  uint8_t* sVh = sm + 6 * AT_TILE;   // V hi / lo: 2 tiles each
  uint8_t* sVl = sm + 8 * AT_TILE;
  uint8_t* sOh = sm + 10 * AT_TILE;  // output hi / lo tiles [128 rows][64] (128-byte swizzle)
  uint8_t* sOl = sm + 11 * AT_TILE;
  // [query slot][key]: (dist + same-slot bias) * log2(e) of the current head, -inf for
  // keys beyond the block
  float* s_btab = reinterpret_cast<float*>(sm + 12 * AT_TILE);
  __shared__ __align__(8) uint64_t bar_qk, bar_qkfree, bar_v[2], bar_vfree[2], bar_s0, bar_s1,
      bar_p0, bar_p1, bar_pv0, bar_o, bar_ofree[2];
  __shared__ uint32_t s_tmem;
  __shared__ float s_pmax[2][AT_NSPLIT][128], s_psum[AT_NSPLIT][128];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int QT = (S + AT_QT - 1) / AT_QT;
  const int64_t nitems = batch * heads * QT;
  const int nd = 2 * B_max - 3;

  if (tid == 0) {
    mbar_init(&bar_qk, 1);
    mbar_init(&bar_qkfree, 1);
    mbar_init(&bar_v[0], 1);
    mbar_init(&bar_v[1], 1);
    mbar_init(&bar_vfree[0], 1);
    mbar_init(&bar_vfree[1], 1);
    mbar_init(&bar_s0, 1);
    mbar_init(&bar_s1, 1);
    mbar_init(&bar_p0, 32 * AT_SOFT_WARPS);
    mbar_init(&bar_p1, 32 * AT_SOFT_WARPS);
    mbar_init(&bar_pv0, 1);
    mbar_init(&bar_o, 1);
    mbar_init(&bar_ofree[0], 32 * AT_SOFT_WARPS);
    mbar_init(&bar_ofree[1], 32 * AT_SOFT_WARPS);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&s_tmem)),
                 "r"(AT_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  at_fence_before();
  __syncthreads();
  at_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_wait();
  pdl_trigger();
  // S / P of key half 0 in columns 0-127, of half 1 in 128-255; O' of even / odd items in
  // 256-319 / 320-383
  const uint32_t tS = tmem, tO0 = tmem + AT_O_COL;
  // this CTA's items: a contiguous range (query tile fastest), so that the query tiles of a
  // (block, head) follow each other and the later ones reuse the K / V tiles already in
  // shared memory (only Q is loaded), and the head (with its bias table) rarely changes
  const int64_t per = (nitems + gridDim.x - 1) / gridDim.x;
  const int64_t first = int64_t(blockIdx.x) * per;
  const int my_items = first < nitems ? static_cast<int>(min(per, nitems - first)) : 0;

  if (warp == 0 && lane == 0) {
    // ---- producer
    ItemPos it(first, 1, QT, batch);
    int pblk = -1, ph = -1;  // (block, head) whose K / V tiles are in shared memory
    for (int i = 0; i < my_items; ++i, it.next()) {
      const int qt = it.qt, h = it.h;
      const int tok0 = it.blk * S;
      const int cq = h * dh, ck = H + h * dh, cv = 2 * H + h * dh, lo = 3 * H;
      // a [128 x 64] tile at column col: plain 2-D box, or for head dim 32 the 3-D view
      // whose 64-wide box over 32-wide heads has its upper half zero-filled
      auto ld = [&](void* dst, int col, int row, uint64_t* bar) {
        if (dh == AT_DH)
          at_tma(dst, &tm, col, row, bar);
        else
          at_tma3(dst, &tm, 0, col >> 5, row, bar);
      };
      const bool same_kv = it.blk == pblk && h == ph;
      pblk = it.blk;
      ph = h;
      if (i > 0 && !mbar_wait_bounded(&bar_qkfree, (i - 1) & 1, &g_err_at, ERR_AT_QKFREE)) break;
      mbar_arrive_expect_tx(&bar_qk, (same_kv ? 2 : 6) * AT_TILE);
      ld(sQh, cq, tok0 + qt * AT_QT, &bar_qk);
      ld(sQl, lo + cq, tok0 + qt * AT_QT, &bar_qk);
      if (!same_kv) {
        ld(sKh, ck, tok0, &bar_qk);
        ld(sKh + AT_TILE, ck, tok0 + 128, &bar_qk);
        ld(sKl, lo + ck, tok0, &bar_qk);
        ld(sKl + AT_TILE, lo + ck, tok0 + 128, &bar_qk);
      }
      // V by key halves: half 0 is free once the previous item's first product is done
      bool vok = true;
      for (int vh = 0; vh < 2 && vok; ++vh) {
        if (i > 0 && !mbar_wait_bounded(&bar_vfree[vh], (i - 1) & 1, &g_err_at, ERR_AT_VFREE)) {
          vok = false;
          break;
        }
        if (same_kv) {
          mbar_arrive(&bar_v[vh]);  // the tiles in place serve this item too
        } else {
          mbar_arrive_expect_tx(&bar_v[vh], 2 * AT_TILE);
          ld(sVh + vh * AT_TILE, cv, tok0 + 128 * vh, &bar_v[vh]);
          ld(sVl + vh * AT_TILE, lo + cv, tok0 + 128 * vh, &bar_v[vh]);
        }
      }
      if (!vok) break;
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer.  Per item i: S0 = Q K[0:128]^T, S1 = Q K[128:256]^T (three-term
    // products, N 128), PV0 into O[i&1] once P0 is ready, PV1 once P1 is ready, then the
    // next item's S0 (over P0, once PV0 has completed) and S1 (once PV1 has), which run
    // while the softmax warps finish this item's epilogue.
    constexpr uint32_t id_s = at_idesc(128, 128, false);
    constexpr uint32_t id_o = at_idesc(128, 128, true);
    auto qk_half = [&](int half) {
      const uint32_t d = tS + uint32_t(128 * half);
      uint8_t* kh = sKh + half * AT_TILE;
      uint8_t* kl = sKl + half * AT_TILE;
#pragma unroll
      for (int ks = 0; ks < AT_DH / 16; ++ks) {
        at_mma(d, at_desc(sQh + ks * 32), at_desc(kh + ks * 32), id_s, ks > 0);
        at_mma(d, at_desc(sQh + ks * 32), at_desc(kl + ks * 32), id_s, 1);
        at_mma(d, at_desc(sQl + ks * 32), at_desc(kh + ks * 32), id_s, 1);
      }
    };
    auto pv_half = [&](int half, uint32_t tO) {
      // P for keys 32c..32c+31 sits in TMEM columns 32c (hi, 16 packed columns) and
      // 32c + 16 (lo); a 16-key step j uses 8 of them
#pragma unroll 4
      for (int jj = 0; jj < 8; ++jj) {
        const int j = 8 * half + jj;
        const uint32_t pc = uint32_t(32 * (j >> 1) + 8 * (j & 1));
        const uint64_t vhl = at_desc_vhl(sVh + 16 * j * 128);
        at_mma_ts(tO, tS + pc, vhl, id_o, (half > 0 || jj > 0));
        at_mma_ts(tO, tS + pc + 16, vhl, id_o, 1);
      }
    };
    bool ok = my_items > 0 && mbar_wait_bounded(&bar_qk, 0, &g_err_at, ERR_AT_QK);
    if (ok) {
      at_fence_after();
      qk_half(0);
      at_commit(&bar_s0);
      qk_half(1);
      at_commit(&bar_s1);
      at_commit(&bar_qkfree);
    }
    for (int i = 0; i < my_items && ok; ++i) {
      const bool more = i + 1 < my_items;
      const uint32_t tO = tO0 + AT_O_W * uint32_t(i & 1);
      ok = mbar_wait_bounded(&bar_p0, i & 1, &g_err_at, ERR_AT_P) &&
           mbar_wait_bounded(&bar_v[0], i & 1, &g_err_at, ERR_AT_V) &&
           (i < 2 || mbar_wait_bounded(&bar_ofree[i & 1], ((i >> 1) - 1) & 1, &g_err_at,
                                       ERR_AT_OFREE));
      if (!ok) break;
      at_fence_after();
      pv_half(0, tO);
      at_commit(&bar_pv0);
      at_commit(&bar_vfree[0]);
      ok = mbar_wait_bounded(&bar_p1, i & 1, &g_err_at, ERR_AT_P) &&
           mbar_wait_bounded(&bar_v[1], i & 1, &g_err_at, ERR_AT_V);
      if (!ok) break;
      at_fence_after();
      pv_half(1, tO);
      at_commit(&bar_o);
      at_commit(&bar_vfree[1]);
      if (more) {
        // S0 of the next item overwrites P0: after PV0 has completed
        ok = mbar_wait_bounded(&bar_pv0, i & 1, &g_err_at, ERR_AT_O) &&
             mbar_wait_bounded(&bar_qk, (i + 1) & 1, &g_err_at, ERR_AT_QK);
        if (!ok) break;
        at_fence_after();
        qk_half(0);
        at_commit(&bar_s0);
        ok = mbar_wait_bounded(&bar_o, i & 1, &g_err_at, ERR_AT_O);
        if (!ok) break;
        at_fence_after();
        qk_half(1);
        at_commit(&bar_s1);
        at_commit(&bar_qkfree);
      }
    }
  } else if (warp >= 2) {
    // ---- softmax and epilogue
    const int qq = warp & 3, hf = (warp - 2) >> 2;
    const int r = 32 * qq + lane;  // TMEM lane = query row of the tile
    const uint32_t lane_off = uint32_t(32 * qq) << 16;
    const int nq = S / Kc;         // query slots
    const float C = (dh == AT_DH ? 0.125f : 0.17677669529663687f) * AT_LOG2E;  // 1/sqrt(dh), log2 units
    constexpr float RESCALE_AT = 16.f;      // log2 headroom before half 1 re-bases
    int i = 0;
    int cur_h = -1;
    const int bj = (tid - 64) & (AT_KMAX - 1);  // this thread's key in the bias-table fill
    const int bks = bj / Kc;
    // Epilogue of item pi: O / l for this warp's 16 of the 64 output columns, split,
    // staged, stored by one thread per quarter.
    int p_qt = 0, p_h = 0, p_blk = 0;
    float p_inv = 0.f;
    bool p_ok = false;
    auto epilogue = [&](int pi) {
      const uint32_t tOp = tO0 + AT_O_W * uint32_t(pi & 1);
      const bool ok2 = mbar_wait_bounded(&bar_o, pi & 1, &g_err_at, ERR_AT_O) && p_ok;
      at_fence_after();
      float v[AT_OW], vl[AT_OW];
      at_ld16(tOp + lane_off + AT_OW * hf, v);
      at_ld16(tOp + lane_off + 64 + AT_OW * hf, vl);
      at_fence_before();
      mbar_arrive(&bar_ofree[pi & 1]);
      uint32_t hi[AT_OW / 2], lo[AT_OW / 2];
#pragma unroll
      for (int e = 0; e < AT_OW; e += 2)
        split2_bf16((v[e] + vl[e]) * p_inv, (v[e + 1] + vl[e + 1]) * p_inv, hi[e / 2], lo[e / 2]);
      // this warp's 16 columns = 16-byte chunks 2hf, 2hf + 1 of the row's 128 bytes, at
      // chunk ^ (row & 7) under the 128-byte swizzle
#pragma unroll
      for (int u = 0; u < AT_OW / 8; ++u) {
        const int off = r * 128 + 16 * ((AT_OW / 8 * hf + u) ^ (r & 7));
        *reinterpret_cast<uint4*>(sOh + off) =
            make_uint4(hi[4 * u], hi[4 * u + 1], hi[4 * u + 2], hi[4 * u + 3]);
        *reinterpret_cast<uint4*>(sOl + off) =
            make_uint4(lo[4 * u], lo[4 * u + 1], lo[4 * u + 2], lo[4 * u + 3]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      quarter_sync(qq);
      if (hf == 0 && lane == 0 && ok2 && p_qt * AT_QT + 32 * qq < S) {
        if (dh == AT_DH) {
          at_store(&tmo, sOh + 32 * qq * 128, p_h * AT_DH, p_qt * AT_QT + 32 * qq, p_blk);
          at_store(&tmo, sOl + 32 * qq * 128, H + p_h * AT_DH, p_qt * AT_QT + 32 * qq, p_blk);
        } else {
          // 4-D view over 32-wide heads: the box's upper 32 columns (zeros) are clipped
          at_store4(&tmo, sOh + 32 * qq * 128, 0, p_h, p_qt * AT_QT + 32 * qq, p_blk);
          at_store4(&tmo, sOl + 32 * qq * 128, 0, heads + p_h, p_qt * AT_QT + 32 * qq, p_blk);
        }
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    };
    ItemPos it(first, 1, QT, batch);
    for (; i < my_items; ++i, it.next()) {
      const int qt = it.qt, h = it.h, blk = it.blk;
      const int q = qt * AT_QT + r;
      const uint32_t tO = tO0 + AT_O_W * uint32_t(i & 1);
      if (h != cur_h) {  // bias table of this head (all softmax warps take the same items)
        soft_sync();
        // thread: key bj, query slots of its parity; distance entries from L1
        const float* drow = dist_bias + h * nd;
        const float same = same_bias[h];
        for (int qs = (tid - 64) / AT_KMAX; qs < nq; qs += 32 * AT_SOFT_WARPS / AT_KMAX) {
          const int k = bks - qs + B_max - 2;
          s_btab[qs * AT_BSTRIDE + bj] =
              bj < S ? (__ldg(drow + k) + (k == B_max - 2 ? same : 0.f)) * AT_LOG2E : -INFINITY;
        }
        soft_sync();
        cur_h = h;
      }
      const float* brow = s_btab + (min(q, S - 1) / Kc) * AT_BSTRIDE;
      bool ok = true;
      float m0 = 0.f, l0 = 0.f, l1 = 0.f;
      for (int half = 0; half < 2; ++half) {
        ok = mbar_wait_bounded(half ? &bar_s1 : &bar_s0, i & 1, &g_err_at, ERR_AT_S) && ok;
        at_fence_after();
        const int jb = 128 * half + 32 * hf;  // this warp's 32 keys of the half
        float v[32];
        at_ld32(tS + lane_off + jb, v);
        // x = v / 8 * log2(e) + bias (log2 units), two at a time; kept for pass 2
        float mx = -INFINITY;
        const float2 c2 = make_float2(C, C);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 b4 = *reinterpret_cast<const float4*>(brow + jb + 4 * u);
          const float2 xa = __ffma2_rn(make_float2(v[4 * u], v[4 * u + 1]), c2, make_float2(b4.x, b4.y));
          const float2 xb = __ffma2_rn(make_float2(v[4 * u + 2], v[4 * u + 3]), c2, make_float2(b4.z, b4.w));
          v[4 * u] = xa.x;
          v[4 * u + 1] = xa.y;
          v[4 * u + 2] = xb.x;
          v[4 * u + 3] = xb.y;
          mx = fmaxf(mx, fmaxf(fmaxf(xa.x, xa.y), fmaxf(xb.x, xb.y)));
        }
        s_pmax[half][hf][r] = mx;
        quarter_sync(qq);
        float mh = s_pmax[half][0][r];
#pragma unroll
        for (int k = 1; k < AT_NSPLIT; ++k) mh = fmaxf(mh, s_pmax[half][k][r]);
        float mref = mh;
        if (half == 0) {
          m0 = mh;
        } else {
          // Rows whose half 1 holds a much larger logit re-base on it: O[i] holds half 0's
          // products (wait for them), scaled down with l0; other rows keep half 0's base
          // (terms up to 2^RESCALE_AT).  The TMEM access is warp-wide.
          const bool rebase = mh > m0 + RESCALE_AT;
          if (!rebase) mref = m0;
          if (__any_sync(FULL_MASK, rebase)) {
            const float sc = rebase ? at_ex2(m0 - mh) : 1.f;
            l0 *= sc;
            mbar_wait_bounded(&bar_pv0, i & 1, &g_err_at, ERR_AT_O);
            at_fence_after();
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              float o[AT_OW];
              at_ld16(tO + lane_off + 64 * part + AT_OW * hf, o);
#pragma unroll
              for (int e = 0; e < AT_OW; ++e) o[e] *= sc;
              at_st16f(tO + lane_off + 64 * part + AT_OW * hf, o);
            }
          }
        }
        float2 l2 = make_float2(0.f, 0.f);
        uint32_t ph[16], pl[16];
        const float2 nm = make_float2(-mref, -mref);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float2 y = __fadd2_rn(make_float2(v[2 * u], v[2 * u + 1]), nm);
          const float p0 = at_ex2(y.x), p1 = at_ex2(y.y);
          l2 = __fadd2_rn(l2, make_float2(p0, p1));
          split2_bf16(p0, p1, ph[u], pl[u]);
        }
        const float l = l2.x + l2.y;
        at_st16(tS + lane_off + jb, ph);
        at_st16(tS + lane_off + jb + 16, pl);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        if (half == 0) l0 = l; else l1 = l;
        at_fence_before();
        mbar_arrive(half ? &bar_p1 : &bar_p0);
      }
      s_psum[hf][r] = l0 + l1;
      // the quarter's previous output store has finished reading its staging rows
      if (hf == 0 && lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      quarter_sync(qq);
      float lsum = 0.f;
#pragma unroll
      for (int k = 0; k < AT_NSPLIT; ++k) lsum += s_psum[k][r];
      p_inv = 1.0f / lsum;
      p_qt = qt;
      p_h = h;
      p_blk = blk;
      p_ok = ok;
      epilogue(i);
    }
  }
  if (warp >= 2 && ((warp - 2) >> 2) == 0 && lane == 0)
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  at_fence_before();
  __syncthreads();
  if (warp == 0) {
    at_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(AT_TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ long lattices
//
// Lattices of 257..512 tokens (the wide candidate pool: 15 slots x 32 candidates = 480
// tokens).  The keys no longer fit the shared memory at once, so each (128-query tile,
// block, head) item walks its keys in chunks of 128 with an online softmax:
//   warp 0     TMA: the item's Q (hi, lo) and per chunk K (hi, lo) into a two-stage ring;
//              warp 18 the V chunks (hi, lo) into their own; warp 0 owns the TMEM
//              allocation (S / P: three 128-column buffers,
//              O': one 128-column buffer, which the epilogue empties before the next item's
//              first product)
//   warp 1     MMA: S(g+1) = Q K(g+1)^T (three split products) while the softmax warps
//              work on chunk g, then O' += P(g) [V hi | V lo] (two products, N 128, P read
//              from TMEM); S into a buffer waits until the product that read its previous
//              P (three chunks back) has completed
//   warps 2-17 per chunk: scale, add the slot bias, row maximum (four warps per query-row
//              quarter, combined through shared memory), running maximum m: the first
//              chunk sets it; a later chunk whose maximum exceeds m by more than 2^16
//              re-bases the row (O' and the partial sums scaled down once the previous
//              product has landed), otherwise its terms stay relative to m; p = 2^(x - m)
//              written over S as packed bf16 hi / lo.  After the last chunk O / l is
//              split into hi / lo and stored straight from registers (rows past the
//              block skipped).
// The bias table holds one row per query slot over all keys (-inf past the block).
// Every wait is bounded and the first timeout makes every later wait of the CTA give up
// at once, so that all warps still reach their named barriers and the final teardown.
constexpr int AL_KC = 128;                     // keys per chunk
constexpr int AL_SBUF = 3;                     // S / P buffers in TMEM (+ one O' buffer)
constexpr int AL_VWARP = 2 + AT_SOFT_WARPS;    // the V producer, after the softmax warps
constexpr int AL_THREADS = AT_THREADS + 32;
constexpr int AL_KMAX = 512;
constexpr int AL_BSTRIDE = AL_KMAX + 4;        // floats per bias-table row (bank offset)
constexpr int AL_SMEM = 11 * AT_TILE + 1024;   // Q, K ring, V ring, output staging + bias table

__device__ __forceinline__ bool al_wait(uint64_t* bar, uint32_t parity, uint32_t site,
                                        volatile int* fail) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63) == 0 && (*fail || clock64() - t0 > WAIT_LIMIT_CYCLES)) {
      atomicOr(&g_err_at, site);
      *fail = 1;
      return false;
    }
  }
}

// MN-major [V hi | V lo] operand whose lo tile sits `lo_off` bytes after the hi tile.
__device__ __forceinline__ uint64_t al_desc_v(const void* p, uint32_t lo_off) {
  return (at_desc(p) & ~(0x3FFFull << 16)) | (uint64_t(lo_off >> 4) << 16);
}

__global__ void __launch_bounds__(AL_THREADS, 1)
    attn_tc_long_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ CUtensorMap tmo,
                        int S, int Kc, int H, int B_max, int heads, int64_t batch,
                        const float* __restrict__ dist_bias, const float* __restrict__ same_bias) {
  extern __shared__ uint8_t al_smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(al_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQh = sm;                // Q hi / lo
  uint8_t* sQl = sm + AT_TILE;
  uint8_t* sK = sm + 2 * AT_TILE;   // stage s: K hi at sK + 2 s AT_TILE, K lo one tile later
  uint8_t* sV = sm + 6 * AT_TILE;   // stage s: V hi at sV + 2 s AT_TILE, V lo one tile later
  uint8_t* sO = sm + 10 * AT_TILE;  // output staging [128 rows][64] (hi, then lo)
  // [query slot][key]: (dist + same-slot bias) * log2(e) of the current head, -inf for
  // keys beyond the block
  float* s_btab = reinterpret_cast<float*>(sm + 11 * AT_TILE);
  __shared__ __align__(8) uint64_t bar_q, bar_qfree, bar_k[2], bar_kfree[2], bar_v[2],
      bar_vfree[2], bar_s[AL_SBUF], bar_p[AL_SBUF], bar_pv[AL_SBUF], bar_o, bar_ofree;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_fail;
  __shared__ float s_pmax[2][AT_NSPLIT][128], s_psum[AT_NSPLIT][128];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int QT = (S + AT_QT - 1) / AT_QT;
  const int NC = (S + AL_KC - 1) / AL_KC;
  const int64_t nitems = batch * heads * QT;
  const int nd = 2 * B_max - 3;

  if (tid == 0) {
    mbar_init(&bar_q, 1);
    mbar_init(&bar_qfree, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_k[b], 1);
      mbar_init(&bar_kfree[b], 1);
      mbar_init(&bar_v[b], 1);
      mbar_init(&bar_vfree[b], 1);
    }
    for (int b = 0; b < AL_SBUF; ++b) {
      mbar_init(&bar_s[b], 1);
      mbar_init(&bar_p[b], 32 * AT_SOFT_WARPS);
      mbar_init(&bar_pv[b], 1);
    }
    mbar_init(&bar_o, 1);
    mbar_init(&bar_ofree, 32 * AT_SOFT_WARPS);
    s_fail = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&s_tmem)),
                 "r"(AT_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  at_fence_before();
  __syncthreads();
  at_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_wait();
  pdl_trigger();
  // S / P of chunk g in columns 128 (g % 3) .. +127; O' in columns 384..511
  const uint32_t tS = tmem, tO = tmem + AL_SBUF * AL_KC;
  // this CTA's items: a contiguous range, so that the four query tiles of a (block, head)
  // run back to back (their K / V chunks come from L2) and the head, with its bias table,
  // changes at most once or twice per CTA
  const int64_t per = (nitems + gridDim.x - 1) / gridDim.x;
  const int64_t first = int64_t(blockIdx.x) * per;
  const int my_items = first < nitems ? static_cast<int>(min(per, nitems - first)) : 0;
  const int total = my_items * NC;

  if ((warp == 0 || warp == AL_VWARP) && lane == 0) {
    // ---- producers: warp 0 loads Q and the K chunks, the last warp the V chunks, so
    // that a K load never waits behind a V slot (freed only by a later product)
    const bool kside = warp == 0;
    int g = 0;
    bool ok = true;
    ItemPos it(first, 1, QT, batch);
    for (int i = 0; i < my_items && ok; ++i, it.next()) {
      const int tok0 = it.blk * S;
      const int cq = it.h * AT_DH, ck = H + it.h * AT_DH, cv = 2 * H + it.h * AT_DH, lo = 3 * H;
      if (kside) {
        if (i > 0 && !al_wait(&bar_qfree, (i - 1) & 1, ERR_AT_QKFREE, &s_fail)) break;
        mbar_arrive_expect_tx(&bar_q, 2 * AT_TILE);
        at_tma(sQh, &tm, cq, tok0 + it.qt * AT_QT, &bar_q);
        at_tma(sQl, &tm, lo + cq, tok0 + it.qt * AT_QT, &bar_q);
      }
      for (int c = 0; c < NC; ++c, ++g) {
        const int st = g & 1, use = g >> 1;
        const int row = tok0 + c * AL_KC;
        uint64_t* freed = kside ? &bar_kfree[st] : &bar_vfree[st];
        if (use > 0 &&
            !al_wait(freed, (use - 1) & 1, kside ? ERR_AT_QKFREE : ERR_AT_VFREE, &s_fail)) {
          ok = false;
          break;
        }
        uint64_t* full = kside ? &bar_k[st] : &bar_v[st];
        uint8_t* dst = (kside ? sK : sV) + 2 * st * AT_TILE;
        const int col = kside ? ck : cv;
        mbar_arrive_expect_tx(full, 2 * AT_TILE);
        at_tma(dst, &tm, col, row, full);
        at_tma(dst + AT_TILE, &tm, lo + col, row, full);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: S(0); then per chunk g: S(g + 1), O' += P(g) V(g)
    constexpr uint32_t id_s = at_idesc(128, 128, false);
    constexpr uint32_t id_o = at_idesc(128, 128, true);
    auto qk = [&](int b, int st) {  // S into buffer b from K stage st
      const uint32_t d = tS + uint32_t(128 * b);
      const uint8_t* kh = sK + 2 * st * AT_TILE;
      const uint8_t* kl = kh + AT_TILE;
#pragma unroll
      for (int ks = 0; ks < AT_DH / 16; ++ks) {
        at_mma(d, at_desc(sQh + ks * 32), at_desc(kh + ks * 32), id_s, ks > 0);
        at_mma(d, at_desc(sQh + ks * 32), at_desc(kl + ks * 32), id_s, 1);
        at_mma(d, at_desc(sQl + ks * 32), at_desc(kh + ks * 32), id_s, 1);
      }
    };
    auto pv = [&](int b, int st, bool first) {
      // P for keys 32c..32c+31 of the chunk: TMEM columns 32c (hi, 16 packed columns) and
      // 32c + 16 (lo); a 16-key step j uses 8 of them
      const uint8_t* vh = sV + 2 * st * AT_TILE;
#pragma unroll 4
      for (int j = 0; j < AL_KC / 16; ++j) {
        const uint32_t pc = uint32_t(128 * b + 32 * (j >> 1) + 8 * (j & 1));
        const uint64_t vhl = al_desc_v(vh + 16 * j * 128, AT_TILE);
        at_mma_ts(tO, tS + pc, vhl, id_o, !(first && j == 0));
        at_mma_ts(tO, tS + pc + 16, vhl, id_o, 1);
      }
    };
    bool ok = total > 0 && al_wait(&bar_q, 0, ERR_AT_QK, &s_fail) &&
              al_wait(&bar_k[0], 0, ERR_AT_QK, &s_fail);
    if (ok) {
      at_fence_after();
      qk(0, 0);
      at_commit(&bar_s[0]);
      at_commit(&bar_kfree[0]);
    }
    int i = 0, c = 0;  // item and chunk of g
    int b = 0, u = 0;  // S / P buffer of g and its use count (g = 3 u + b)
    for (int g = 0; g < total && ok; ++g) {
      const int g1 = g + 1;
      const int b1 = b + 1 == AL_SBUF ? 0 : b + 1, u1 = b1 == 0 ? u + 1 : u;
      if (g1 < total) {
        // S(g + 1) into the buffer that PV(g - 2) read last: once that product is done
        const int c1 = c + 1 == NC ? 0 : c + 1;
        const int i1 = c1 == 0 ? i + 1 : i;
        ok = (c1 != 0 || al_wait(&bar_q, i1 & 1, ERR_AT_QK, &s_fail)) &&
             al_wait(&bar_k[g1 & 1], (g1 >> 1) & 1, ERR_AT_QK, &s_fail) &&
             (u1 == 0 || al_wait(&bar_pv[b1], (u1 - 1) & 1, ERR_AT_O, &s_fail));
        if (!ok) break;
        at_fence_after();
        qk(b1, g1 & 1);
        at_commit(&bar_s[b1]);
        at_commit(&bar_kfree[g1 & 1]);
        if (c1 == NC - 1) at_commit(&bar_qfree);
      }
      // O' of item i starts once the epilogue has read item i - 1's
      ok = al_wait(&bar_p[b], u & 1, ERR_AT_P, &s_fail) &&
           al_wait(&bar_v[g & 1], (g >> 1) & 1, ERR_AT_V, &s_fail) &&
           (c != 0 || i < 1 || al_wait(&bar_ofree, (i - 1) & 1, ERR_AT_OFREE, &s_fail));
      if (!ok) break;
      at_fence_after();
      pv(b, g & 1, c == 0);
      at_commit(&bar_pv[b]);
      at_commit(&bar_vfree[g & 1]);
      if (c == NC - 1) at_commit(&bar_o);
      if (++c == NC) {
        c = 0;
        ++i;
      }
      b = b1;
      u = u1;
    }
  } else if (warp >= 2 && warp < 2 + AT_SOFT_WARPS) {
    // ---- softmax and epilogue
    const int qq = warp & 3, hf = (warp - 2) >> 2;
    const int r = 32 * qq + lane;  // TMEM lane = query row of the tile
    const uint32_t lane_off = uint32_t(32 * qq) << 16;
    const int nq = S / Kc;         // query slots
    const int nk = NC * AL_KC;     // keys covered by the chunks
    constexpr float C = 0.125f * AT_LOG2E;  // 1 / sqrt(64), in log2 units
    constexpr float RESCALE_AT = 16.f;      // log2 headroom before a chunk re-bases a row
    const int jb = 32 * hf;                 // this warp's 32 keys of every chunk
    int cur_h = -1;
    int g = 0, sb = 0, su = 0;  // chunk, its S / P buffer and the buffer's use count
    int psb = 0, psu = 0;       // the same of chunk g - 1
    ItemPos it(first, 1, QT, batch);
    for (int i = 0; i < my_items; ++i, it.next()) {
      const int qt = it.qt, h = it.h, blk = it.blk;
      const int q = qt * AT_QT + r;
      if (h != cur_h) {  // bias table of this head (all softmax warps take the same items)
        soft_sync();
        // a thread per key column (no division per entry), all query slots down it
        const float* drow = dist_bias + h * nd;
        const float same = same_bias[h];
        for (int key = tid - 64; key < nk; key += 32 * AT_SOFT_WARPS) {
          const int ks = key / Kc;
          for (int qs = 0; qs < nq; ++qs) {
            const int k = ks - qs + B_max - 2;
            s_btab[qs * AL_BSTRIDE + key] =
                key < S ? (__ldg(drow + k) + (k == B_max - 2 ? same : 0.f)) * AT_LOG2E
                        : -INFINITY;
          }
        }
        soft_sync();
        cur_h = h;
      }
      const float* brow = s_btab + (min(q, S - 1) / Kc) * AL_BSTRIDE;
      bool ok = true;
      float m = -INFINITY, l = 0.f;
      for (int c = 0; c < NC; ++c, ++g) {
        ok = al_wait(&bar_s[sb], su & 1, ERR_AT_S, &s_fail) && ok;
        at_fence_after();
        float v[32];
        at_ld32(tS + lane_off + uint32_t(128 * sb + jb), v);
        // x = v / 8 * log2(e) + bias (log2 units), two at a time
        const float* bk = brow + c * AL_KC + jb;
        float mx = -INFINITY;
        const float2 c2 = make_float2(C, C);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 b4 = *reinterpret_cast<const float4*>(bk + 4 * u);
          const float2 xa = __ffma2_rn(make_float2(v[4 * u], v[4 * u + 1]), c2, make_float2(b4.x, b4.y));
          const float2 xb = __ffma2_rn(make_float2(v[4 * u + 2], v[4 * u + 3]), c2, make_float2(b4.z, b4.w));
          v[4 * u] = xa.x;
          v[4 * u + 1] = xa.y;
          v[4 * u + 2] = xb.x;
          v[4 * u + 3] = xb.y;
          mx = fmaxf(mx, fmaxf(fmaxf(xa.x, xa.y), fmaxf(xb.x, xb.y)));
        }
        s_pmax[c & 1][hf][r] = mx;
        quarter_sync(qq);
        float mh = s_pmax[c & 1][0][r];
#pragma unroll
        for (int k = 1; k < AT_NSPLIT; ++k) mh = fmaxf(mh, s_pmax[c & 1][k][r]);
        if (c == 0) {
          m = mh;
        } else {
          // a row whose new chunk holds a much larger logit re-bases on it: O' holds the
          // earlier chunks' products (wait for the last of them) and is scaled down with
          // the partial sum; other rows keep their base (terms up to 2^RESCALE_AT).  The
          // TMEM access is warp-wide.
          const bool rebase = mh > m + RESCALE_AT;
          if (__any_sync(FULL_MASK, rebase)) {
            const float sc = rebase ? at_ex2(m - mh) : 1.f;
            l *= sc;
            ok = al_wait(&bar_pv[psb], psu & 1, ERR_AT_O, &s_fail) && ok;
            at_fence_after();
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              float o[AT_OW];
              at_ld16(tO + lane_off + 64 * part + AT_OW * hf, o);
#pragma unroll
              for (int e = 0; e < AT_OW; ++e) o[e] *= sc;
              at_st16f(tO + lane_off + 64 * part + AT_OW * hf, o);
            }
          }
          if (rebase) m = mh;
        }
        // p = 2^(x - m) as packed bf16 hi / lo over the logits, 16 keys at a time (hi
        // words of keys 2u, 2u + 1 at column jb + u, lo words 16 columns further)
        float2 l2 = make_float2(0.f, 0.f);
        const float2 nm = make_float2(-m, -m);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t ph[8], pl[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int e = 16 * h2 + 2 * u;
            const float2 y = __fadd2_rn(make_float2(v[e], v[e + 1]), nm);
            const float p0 = at_ex2(y.x), p1 = at_ex2(y.y);
            l2 = __fadd2_rn(l2, make_float2(p0, p1));
            split2_bf16(p0, p1, ph[u], pl[u]);
          }
          at_st8(tS + lane_off + uint32_t(128 * sb + jb + 8 * h2), ph);
          at_st8(tS + lane_off + uint32_t(128 * sb + jb + 16 + 8 * h2), pl);
        }
        l += l2.x + l2.y;
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        at_fence_before();
        mbar_arrive(&bar_p[sb]);
        psb = sb;
        psu = su;
        if (++sb == AL_SBUF) {
          sb = 0;
          ++su;
        }
      }
      s_psum[hf][r] = l;
      // the quarter's previous output store has finished reading its staging rows
      if (hf == 0 && lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      quarter_sync(qq);
      float lsum = 0.f;
#pragma unroll
      for (int k = 0; k < AT_NSPLIT; ++k) lsum += s_psum[k][r];
      const float inv = 1.0f / lsum;
      // epilogue: O / l for this warp's 16 of the 64 output columns, split, stored from
      // registers (hi at column h * 64, lo at H + h * 64 of the [tokens, 2H] output)
      ok = al_wait(&bar_o, i & 1, ERR_AT_O, &s_fail) && ok;
      at_fence_after();
      float v[AT_OW], vl[AT_OW];
      at_ld16(tO + lane_off + AT_OW * hf, v);
      at_ld16(tO + lane_off + 64 + AT_OW * hf, vl);
      at_fence_before();
      mbar_arrive(&bar_ofree);
      uint32_t hi[AT_OW / 2], lo[AT_OW / 2];
#pragma unroll
      for (int e = 0; e < AT_OW; e += 2)
        split2_bf16((v[e] + vl[e]) * inv, (v[e + 1] + vl[e + 1]) * inv, hi[e / 2], lo[e / 2]);
      // stored through the staging tile by bulk tensor stores of the quarter's 32 rows
      // (rows past the block are clipped): first the hi words, then, once that store has
      // read the staging, the lo words.  This warp's 16 columns = 16-byte chunks 2 hf,
      // 2 hf + 1 of the row's 128 bytes, at chunk ^ (row & 7) under the 128-byte swizzle.
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t* wv = half ? lo : hi;
#pragma unroll
        for (int u = 0; u < AT_OW / 8; ++u) {
          const int off = r * 128 + 16 * ((AT_OW / 8 * hf + u) ^ (r & 7));
          *reinterpret_cast<uint4*>(sO + off) =
              make_uint4(wv[4 * u], wv[4 * u + 1], wv[4 * u + 2], wv[4 * u + 3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        quarter_sync(qq);
        if (hf == 0 && lane == 0) {
          if (ok && qt * AT_QT + 32 * qq < S) {
            at_store(&tmo, sO + 32 * qq * 128, (half ? H : 0) + h * AT_DH, qt * AT_QT + 32 * qq,
                     blk);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
          if (!half) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        }
        if (!half) quarter_sync(qq);
      }
    }
  }
  if (warp >= 2 && warp < 2 + AT_SOFT_WARPS && ((warp - 2) >> 2) == 0 && lane == 0)
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  at_fence_before();
  __syncthreads();
  if (warp == 0) {
    at_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(AT_TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host

static PFN_cuTensorMapEncodeTiled_v12000 at_encode_fn() {
  // looked up once per process (a thread-safe static initialisation)
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

static int at_smem_bytes(int S, int K) { return AT_SMEM + (S / K) * AT_BSTRIDE * 4; }

// Head dim 64, or 32 through zero-filled 64-wide tiles (the products then run at the
// head-dim-64 cost; the workloads' head-dim-32 lattice is the 12-token tiny one).
bool attention_tc_supported(int S, int K, int H, int heads, int B_max) {
  const int dh = heads > 0 ? H / heads : 0;
  return (dh == AT_DH || dh == 32) && dh * heads == H && S >= 1 && S <= AT_KMAX && K >= 1 &&
         H % 64 == 0 && B_max <= 64 && at_smem_bytes(S, K) <= AT_SMEM_MAX;
}

cudaError_t launch_attention_tc(const __nv_bfloat16* qkv, int64_t batch, int S, int K, int H,
                                int heads, int B_max, const float* dist_bias,
                                const float* same_bias, __nv_bfloat16* out,
                                cudaStream_t stream) {
  auto fn = at_encode_fn();
  if (!fn || !attention_tc_supported(S, K, H, heads, B_max)) return cudaErrorInvalidValue;
  const int64_t M = batch * S;
  const int dh = H / heads;
  CUtensorMap tm, tmo;
  if (dh == AT_DH) {
    const cuuint64_t dims[2] = {cuuint64_t(6 * H), cuuint64_t(M)};
    const cuuint64_t strides[1] = {cuuint64_t(6 * H) * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t estr[2] = {1, 1};
    if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(qkv), dims,
           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    // output [batch][S][2H] (hi | lo): 3-D so that a store box never runs into the next block
    const cuuint64_t odims[3] = {cuuint64_t(2 * H), cuuint64_t(S), cuuint64_t(batch)};
    const cuuint64_t ostrides[2] = {cuuint64_t(2 * H) * 2, cuuint64_t(S) * 2 * H * 2};
    const cuuint32_t obox[3] = {64, 32, 1};
    const cuuint32_t oestr[3] = {1, 1, 1};
    if (fn(&tmo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, odims, ostrides, obox, oestr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  } else {
    // head dim 32: qkv as [M][6H / 32][32], read in [128][1][64] boxes (the 32 columns
    // past each head's end zero-filled), and the output as [batch][S][2H / 32][32],
    // written in [1][32][1][64] boxes (the zero half clipped)
    const cuuint64_t dims[3] = {32, cuuint64_t(6 * H / 32), cuuint64_t(M)};
    const cuuint64_t strides[2] = {64, cuuint64_t(6 * H) * 2};
    const cuuint32_t box[3] = {64, 1, 128};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(qkv), dims,
           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    const cuuint64_t odims[4] = {32, cuuint64_t(2 * H / 32), cuuint64_t(S), cuuint64_t(batch)};
    const cuuint64_t ostrides[3] = {64, cuuint64_t(2 * H) * 2, cuuint64_t(S) * 2 * H * 2};
    const cuuint32_t obox[4] = {64, 1, 32, 1};
    const cuuint32_t oestr[4] = {1, 1, 1, 1};
    if (fn(&tmo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, out, odims, ostrides, obox, oestr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int smem = at_smem_bytes(S, K);
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(attn_tc_kernel), smem);
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count();
  const int64_t nitems = batch * heads * ((S + AT_QT - 1) / AT_QT);
  // contiguous item ranges of ceil(nitems / SMs): as many CTAs as that takes, none empty
  const int64_t per = (nitems + sms - 1) / sms;
  const dim3 grid(static_cast<unsigned>((nitems + per - 1) / per));
  e = launch_k(attn_tc_kernel, grid, dim3(AT_THREADS), smem, stream, tm, tmo, S, K, H, B_max,
               heads, batch, dist_bias, same_bias, dh);
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaGetLastError();
}

static int al_smem_bytes(int S, int K) { return AL_SMEM + (S / K) * AL_BSTRIDE * 4; }

bool attention_tc_long_supported(int S, int K, int H, int heads, int B_max) {
  return H / heads == AT_DH && S > AT_KMAX && S <= AL_KMAX && K >= 1 && H % 64 == 0 &&
         B_max <= 64 && al_smem_bytes(S, K) <= AT_SMEM_MAX;
}

cudaError_t launch_attention_tc_long(const __nv_bfloat16* qkv, int64_t batch, int S, int K,
                                     int H, int heads, int B_max, const float* dist_bias,
                                     const float* same_bias, __nv_bfloat16* out,
                                     cudaStream_t stream) {
  auto fn = at_encode_fn();
  if (!fn || !attention_tc_long_supported(S, K, H, heads, B_max) ||
      reinterpret_cast<uintptr_t>(out) % 16)
    return cudaErrorInvalidValue;
  const int64_t M = batch * S;
  CUtensorMap tm;
  const cuuint64_t dims[2] = {cuuint64_t(6 * H), cuuint64_t(M)};
  const cuuint64_t strides[1] = {cuuint64_t(6 * H) * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(qkv), dims, strides,
         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // output [batch][S][2H] (hi | lo): 3-D so that a store box never runs into the next block
  CUtensorMap tmo;
  const cuuint64_t odims[3] = {cuuint64_t(2 * H), cuuint64_t(S), cuuint64_t(batch)};
  const cuuint64_t ostrides[2] = {cuuint64_t(2 * H) * 2, cuuint64_t(S) * 2 * H * 2};
  const cuuint32_t obox[3] = {64, 32, 1};
  const cuuint32_t oestr[3] = {1, 1, 1};
  if (fn(&tmo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, odims, ostrides, obox, oestr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int smem = al_smem_bytes(S, K);
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(attn_tc_long_kernel), smem);
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count();
  const int64_t nitems = batch * heads * ((S + AT_QT - 1) / AT_QT);
  const dim3 grid(static_cast<unsigned>(nitems < sms ? nitems : sms));
  e = launch_k(attn_tc_long_kernel, grid, dim3(AL_THREADS), smem, stream, tm, tmo, S, K, H, B_max,
               heads, batch, dist_bias, same_bias);
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaGetLastError();
}

cudaError_t at_read_device_error(uint32_t* code) {
  uint32_t v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_err_at, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_err_at, &zero, sizeof(zero));
  *code |= v << 16;
  return e;
}

}  // namespace lilicorr
