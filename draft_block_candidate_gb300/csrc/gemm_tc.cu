// Dense contractions of steps a2-a4 on the 5th-generation tensor cores.
//
//   C[M, N] = A[M, Ka] . W[N, Kw]^T (+ fused epilogue),   Ka = Kw or 2 Kw
//
// A is an activation stored [A_hi | A_lo] (two bf16 halves whose sum carries ~16
// significant bits) when Ka = 2 Kw; W is an exact bf16 weight whose column index wraps
// (k mod Kw), so one accumulation gives A_hi W^T + A_lo W^T.
//
// Persistent: one CTA per SM walks the 128 x 256 output tiles (n fastest, so the CTAs
// working at the same time share A tiles through L2; 256 columns per tile halve the
// A re-reads of 128-wide tiles, which left these small-K contractions short of L2
// bandwidth).  10 warps:
//   warp 0      TMA producer (2-D tiled loads, 128-byte swizzle, 3-stage mbarrier ring
//               that runs on across tiles) and TMEM owner (2 x 256 f32 columns)
//   warp 1      MMA issuer: one elected thread issues tcgen05.mma (kind::f16, bf16 in,
//               f32 accumulate in TMEM, M 128 x N 256), 4 per 64-wide K block, and
//               tcgen05.commit
//   warps 2-9   epilogue: two warps per 32-lane TMEM quarter (= 32 output rows), each
//               taking half of the columns; tcgen05.ld, then the fused bias / SiLU /
//               hi-lo split in registers, 32 x 32 chunks staged through swizzled shared
//               memory and written by bulk tensor stores (the residual add is a bulk
//               tensor reduce-add into the f32 stream); the node epilogue's gathers and
//               sums store directly
// The accumulator is double-buffered: the epilogue of tile i overlaps the MMAs of tile
// i + 1.  Every mbarrier wait is bounded; a timeout sets a bit in this unit's error word
// and the CTA still frees its TMEM before exiting.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <float.h>
#include <limits.h>

#include <algorithm>

#include "kernels.cuh"

namespace lilicorr {

static __device__ uint32_t g_err_tc;

constexpr int TC_BM = 128, TC_BN = 256, TC_BK = 64;
constexpr int TC_EPI_WARPS = 8, TC_THREADS = 32 * (2 + TC_EPI_WARPS);
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;
constexpr int TC_B_BYTES = TC_BN * TC_BK * 2;
constexpr int TC_STG_BYTES = 4096;  // one 32 x 32 output chunk (f32, or bf16 hi + lo)
// Shared memory of a configuration: operand ring of ST stages + NB epilogue staging
// buffers per warp.  A stage holds one 64-wide K block of A and of W, or, for a split
// operand (pair), the A_hi and A_lo blocks that share one W block.  Configurations in
// use: 4 plain stages or 3 paired stages with 1 staging buffer per epilogue warp, 2 paired
// stages with 2 (node sum) or with 16 epilogue warps (short-K SiLU).
__host__ __device__ constexpr int tc_smem(int st, int nb, bool pair, int ew = TC_EPI_WARPS) {
  return st * ((pair ? 2 : 1) * TC_A_BYTES + TC_B_BYTES) + ew * nb * TC_STG_BYTES + 1024;
}
constexpr uint32_t TC_TMEM_COLS = 2 * TC_BN;  // two accumulator buffers

enum TcErr : uint32_t {
  ERR_TC_EMPTY = 1u << 0,
  ERR_TC_FULL = 1u << 1,
  ERR_TC_ACCUM = 1u << 2,
  ERR_TC_ACC_EMPTY = 1u << 3
};

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
      : "memory");
}

// Bulk tensor store / reduce-add of a shared-memory box to global memory.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, const void* src, int c0,
                                             int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(smem_addr(src)), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* tm, const void* src, int c0,
                                                  int c1) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(tm)),
      "r"(smem_addr(src)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most one committed bulk group still reads shared memory.
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand tile written by TMA with the 128-byte
// swizzle (rows of 64 bf16 = 128 bytes, 8-row / 1024-byte swizzle atoms).
//   bits  0-13 start address >> 4     bits 16-29 leading byte offset >> 4 (unused: 1)
//   bits 32-45 stride byte offset >> 4 (1024 B between 8-row groups)
//   bits 46-47 version (1)            bits 61-63 layout (2 = 128-byte swizzle)
__device__ __forceinline__ uint64_t sw128_desc(const void* smem_tile) {
  const uint64_t addr = smem_addr(smem_tile);
  return ((addr >> 4) & 0x3FFFull) | (1ull << 16) | ((1024ull >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}

// Instruction descriptor, kind::f16: f32 accumulator, bf16 A and B, both K-major.
//   bits 4-5 D format (1 = f32)  bits 7-9 A format (1 = bf16)  bits 10-12 B format (1 = bf16)
//   bit 15/16 A/B major (0 = K)  bits 17-22 N >> 3             bits 24-28 M >> 4
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// 32 consecutive f32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
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

// ------------------------------------------------------------------ epilogue

// Node epilogue terms of row m, columns n..n+31: v (the accumulator) += bias + E[cand]
// + slot_table[s-1] + rank_table[k] (+ drafter hidden); the optional tap is written here,
// X by the staged f32 store.
// Node sum of step a2 for one row: the row's gather sources, found once per tile.
struct NodeRow {
  const __nv_bfloat16* e;  // E[cand] row
  const __nv_bfloat16* h;  // drafter hidden row of the slot, or null
  const float* st;         // slot-table row
  const float* rk;         // rank-table row
};
__device__ __forceinline__ NodeRow tc_node_row(const GemmArgs& g, int64_t m) {
  const int S = (g.B - 1) * g.K;
  const int64_t b = m / S;
  const int t = static_cast<int>(m - b * S);
  const int slot = t / g.K + 1, k = t - (slot - 1) * g.K;
  int64_t id = g.cand_id[m];
  id = id < 0 ? 0 : (id >= g.vocab ? g.vocab - 1 : id);
  NodeRow r;
  r.e = g.embed + id * g.N;
  r.h = g.slot_hidden ? g.slot_hidden + (b * g.B + slot) * g.N : nullptr;
  r.st = g.slot_table + int64_t(slot - 1) * g.N;
  r.rk = g.rank_table + int64_t(k) * g.N;
  return r;
}
// The row's bf16 gathers of columns n..n+31 (issued before the accumulator is read).
__device__ __forceinline__ void tc_node_gather(const NodeRow& r, int n, uint4 (&ge)[4],
                                               uint4 (&gh)[4]) {
  const uint4* e4 = reinterpret_cast<const uint4*>(r.e + n);
#pragma unroll
  for (int j = 0; j < 4; ++j) ge[j] = __ldg(e4 + j);
  if (r.h) {
    const uint4* h4 = reinterpret_cast<const uint4*>(r.h + n);
#pragma unroll
    for (int j = 0; j < 4; ++j) gh[j] = __ldg(h4 + j);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) gh[j] = make_uint4(0u, 0u, 0u, 0u);
  }
}
__device__ __forceinline__ void tc_add_bf16x8(float* v, const uint4& e) {
  const uint32_t ew[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    v[2 * q] += __uint_as_float(ew[q] << 16);
    v[2 * q + 1] += __uint_as_float(ew[q] & 0xffff0000u);
  }
}
// v[0..31] = accumulator columns n..n+31 of row m: + bias + E[cand] + slot + rank +
// drafter hidden, in that order.
__device__ __forceinline__ void tc_node_terms(const GemmArgs& g, const NodeRow& r, int64_t m,
                                              int n, float (&v)[32], const uint4 (&ge)[4],
                                              const uint4 (&gh)[4]) {
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    const float4 b4 = __ldg(reinterpret_cast<const float4*>(g.bias + n + j));
    v[j] += b4.x;
    v[j + 1] += b4.y;
    v[j + 2] += b4.z;
    v[j + 3] += b4.w;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) tc_add_bf16x8(v + 8 * j, ge[j]);
  const float4* st4 = reinterpret_cast<const float4*>(r.st + n);
  const float4* rk4 = reinterpret_cast<const float4*>(r.rk + n);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 a = __ldg(st4 + j), c = __ldg(rk4 + j);
    v[4 * j] += a.x + c.x;
    v[4 * j + 1] += a.y + c.y;
    v[4 * j + 2] += a.z + c.z;
    v[4 * j + 3] += a.w + c.w;
  }
  if (r.h) {
#pragma unroll
    for (int j = 0; j < 4; ++j) tc_add_bf16x8(v + 8 * j, gh[j]);
  }
  // X itself leaves through the staged f32 store; only the optional tap is written here
  if (g.nodes_tap) {
    float4* tp = reinterpret_cast<float4*>(g.nodes_tap + m * g.N + n);
#pragma unroll
    for (int j = 0; j < 8; ++j) tp[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  }
}

// The bias of this lane's row, columns n..n+31 (one bias for all rows, or the row's block
// row when bias_group > 0; rows past M reuse the last one): loaded before the accumulator
// and the staging buffer are waited for, so its latency overlaps those waits.
__device__ __forceinline__ void tc_bias_fetch(const GemmArgs& g, int64_t row0, int lane, int n,
                                              float4 (&bq)[8]) {
  const float* bias = g.bias + n;
  if (g.bias_group > 0)
    bias += (std::min<int64_t>(row0 + lane, g.M - 1) / g.bias_group) *
            (g.bias_stride > 0 ? g.bias_stride : int64_t(g.N));
#pragma unroll
  for (int j = 0; j < 8; ++j) bq[j] = __ldg(reinterpret_cast<const float4*>(bias) + j);
}

// Staged form of the bias / SiLU / split / residual epilogues: v[0..31] = accumulator
// columns n..n+31 of this lane's row (bq its bias, or null); the warp's 32 x 32 chunk goes
// to shared memory in the layout of the output tensor map's swizzle (16-byte unit u of row
// r at u ^ f(r)), then one lane stores it (or adds it into the residual) with bulk tensor
// copies.
template <int EPI>
__device__ __forceinline__ void tc_epilogue_staged(const GemmArgs& g, const CUtensorMap* tmC,
                                                   uint8_t* stg, int lane, int64_t row0, int n,
                                                   float (&v)[32], const float4* bq) {
  if (bq) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[4 * j] += bq[j].x;
      v[4 * j + 1] += bq[j].y;
      v[4 * j + 2] += bq[j].z;
      v[4 * j + 3] += bq[j].w;
    }
  }
  if constexpr (EPI == EPI_SPLIT || EPI == EPI_SPLIT_SILU) {
    uint32_t hi[16], lo[16];
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      float a = v[j], b = v[j + 1];
      if constexpr (EPI == EPI_SPLIT_SILU) {
        a = silu(a);
        b = silu(b);
      }
      split2_bf16(a, b, hi[j / 2], lo[j / 2]);
    }
    // 64-byte rows, 64-byte swizzle: unit u of row r lands at u ^ ((r >> 1) & 3)
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int off = lane * 64 + ((u ^ sw) << 4);
      *reinterpret_cast<uint4*>(stg + off) = make_uint4(hi[4 * u], hi[4 * u + 1], hi[4 * u + 2], hi[4 * u + 3]);
      *reinterpret_cast<uint4*>(stg + 2048 + off) =
          make_uint4(lo[4 * u], lo[4 * u + 1], lo[4 * u + 2], lo[4 * u + 3]);
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tmC, stg, n, static_cast<int>(row0));
      tma_store_2d(tmC, stg + 2048, g.N + n, static_cast<int>(row0));
      bulk_commit();
    }
  } else {
    // 128-byte rows, 128-byte swizzle: unit u of row r lands at u ^ (r & 7)
    const int sw = lane & 7;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      *reinterpret_cast<float4*>(stg + lane * 128 + ((u ^ sw) << 4)) =
          make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      if constexpr (EPI == EPI_RESID)
        tma_reduce_add_2d(tmC, stg, n, static_cast<int>(row0));
      else
        tma_store_2d(tmC, stg, n, static_cast<int>(row0));
      bulk_commit();
    }
  }
}

// ------------------------------------------------------------------ work items
//
// Item i of a launch: tile t, columns [c0, c0 + bn) of it.  The first ntiles - tail_tiles
// items are whole tiles; the rest are the last tail_tiles tiles cut into tail_split column
// pieces, so that the last round of the persistent grid is spread over more SMs.
struct TcItem {
  int t, c0, bn;
};
__device__ __forceinline__ int tc_items(const GemmArgs& g, int ntiles) {
  return g.tail_split > 1 ? ntiles + g.tail_tiles * (g.tail_split - 1) : ntiles;
}
__device__ __forceinline__ TcItem tc_item(const GemmArgs& g, int ntiles, int i) {
  const int nfull = g.tail_split > 1 ? ntiles - g.tail_tiles : ntiles;
  if (i < nfull) return {i, 0, TC_BN};
  const int j = i - nfull, bn = TC_BN / g.tail_split;
  return {nfull + j / g.tail_split, (j % g.tail_split) * bn, bn};
}

// ------------------------------------------------------------------ A made in the kernel
//
// Two contractions read an A operand that is cheap to form from data already on hand, so
// forming it beside the MMAs saves its round trip through HBM (and the launch that wrote
// it).  TC_A_WARPS warps (256 threads) fill the A_hi / A_lo halves of each ring stage in
// the 128-byte-swizzled K-major layout the TMA would have written (16-byte unit u of
// row r at r * 128 + ((u ^ (r & 7)) << 4)), each thread one unit of rows r, r + 32,
// r + 64, r + 96; every thread arrives on the stage's full barrier after a proxy fence,
// and waits for the stage's empty barrier before rewriting it.  Rows past M are zero.
constexpr int TC_A_WARPS = 8;

__device__ __forceinline__ void a_store_unit(uint8_t* ahi, uint8_t* alo, int r, int unit,
                                             const float (&v)[8]) {
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) split2_bf16(v[2 * j], v[2 * j + 1], hi[j], lo[j]);
  const int off = r * 128 + ((unit ^ (r & 7)) << 4);
  *reinterpret_cast<uint4*>(ahi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  *reinterpret_cast<uint4*>(alo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

template <int ASRC, int STAGES>
__device__ __forceinline__ void a_producer(const GemmArgs& g, uint8_t* sA, int AST,
                                           uint64_t* full_bar, uint64_t* empty_bar, int KB,
                                           int NT, int ntiles, int unit, int rsub,
                                           const float* wt) {
  int it = 0;
  const int nitems = tc_items(g, ntiles);
  for (int w = blockIdx.x; w < nitems; w += gridDim.x) {
    const int t = tc_item(g, ntiles, w).t;  // the operand rows depend only on the tile
    const int64_t m0 = int64_t(t / NT) * TC_BM;
    if constexpr (ASRC == ASRC_FUSION) {
      // [h, h * t]: ring step kb = 2 cb + part holds column block cb of h (part 0) or of
      // h * t (part 1), so a block of X is loaded once for both; the loads are issued
      // before the wait for the stage, so their latency overlaps it
      const int H = g.Kw / 2;
      const float* xr[4];
      const __nv_bfloat16* tr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + rsub + 32 * i;
        const bool live = m < g.M;
        xr[i] = live ? g.a_x + m * H + unit * 8 : nullptr;
        tr[i] = live && g.a_t ? g.a_t + (m / g.a_group) * H + unit * 8 : nullptr;
      }
      float x[4][8];
      uint4 tw[4];
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int cb = kb >> 1, part = kb & 1;
        const int s = it % STAGES, use = it / STAGES;
        if (part == 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (xr[i]) {
              a = __ldg(reinterpret_cast<const float4*>(xr[i] + cb * TC_BK));
              b = __ldg(reinterpret_cast<const float4*>(xr[i] + cb * TC_BK + 4));
            }
            x[i][0] = a.x; x[i][1] = a.y; x[i][2] = a.z; x[i][3] = a.w;
            x[i][4] = b.x; x[i][5] = b.y; x[i][6] = b.z; x[i][7] = b.w;
            tw[i] = tr[i] ? __ldg(reinterpret_cast<const uint4*>(tr[i] + cb * TC_BK))
                          : make_uint4(0u, 0u, 0u, 0u);
          }
        }
        if (use > 0 &&
            !mbar_wait_bounded(&empty_bar[s], (use - 1) & 1, &g_err_tc, ERR_TC_EMPTY))
          return;
        uint8_t* ahi = sA + s * AST;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float v[8];
          if (part == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = x[i][j];
          } else {
            const uint32_t ww[4] = {tw[i].x, tw[i].y, tw[i].z, tw[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              v[2 * j] = x[i][2 * j] * __uint_as_float(ww[j] << 16);
              v[2 * j + 1] = x[i][2 * j + 1] * __uint_as_float(ww[j] & 0xffff0000u);
            }
          }
          a_store_unit(ahi, ahi + TC_A_BYTES, rsub + 32 * i, unit, v);
        }
        fence_async_smem();
        mbar_arrive(&full_bar[s]);
      }
    } else {
      // U = SiLU(W1 f + b1): the five features of each of this thread's rows once per tile
      // (log-prob, prob, gap to the slot's top candidate, normalised rank, top indicator),
      // then per ring step the 8 hidden units of this thread's unit
      float f[4][5];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + rsub + 32 * i;
#pragma unroll
        for (int c = 0; c < 5; ++c) f[i][c] = 0.f;
        if (m < g.M) {
          const int64_t j = m / g.K;
          const int k = static_cast<int>(m - j * g.K);
          const float l2 = __ldg(g.a_lse + j);
          const float lp = __ldg(g.a_cl + m) - l2;
          f[i][0] = lp;
          f[i][1] = expf(lp);
          f[i][2] = lp - (__ldg(g.a_cl + j * g.K) - l2);
          f[i][3] = g.K > 1 ? float(k) / float(g.K - 1) : 0.f;
          f[i][4] = k == 0 ? 1.f : 0.f;
        }
      }
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % STAGES, use = it / STAGES;
        // this unit's 8 hidden units: 48 consecutive floats of the weight table
        float w[48];
        const float4* w4 = reinterpret_cast<const float4*>(wt + (kb * TC_BK + unit * 8) * 6);
#pragma unroll
        for (int c = 0; c < 12; ++c) {
          const float4 q = w4[c];
          w[4 * c] = q.x;
          w[4 * c + 1] = q.y;
          w[4 * c + 2] = q.z;
          w[4 * c + 3] = q.w;
        }
        if (use > 0 &&
            !mbar_wait_bounded(&empty_bar[s], (use - 1) & 1, &g_err_tc, ERR_TC_EMPTY))
          return;
        uint8_t* ahi = sA + s * AST;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float v[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float acc = w[6 * q + 5];
#pragma unroll
            for (int c = 0; c < 5; ++c) acc = fmaf(w[6 * q + c], f[i][c], acc);
            v[q] = silu(acc);
          }
          a_store_unit(ahi, ahi + TC_A_BYTES, rsub + 32 * i, unit, v);
        }
        fence_async_smem();
        mbar_arrive(&full_bar[s]);
      }
    }
  }
}

// ------------------------------------------------------------------ kernel

// EW epilogue warps: 8 (two per TMEM quarter, each half the columns) or 16 (four per
// quarter, each a quarter of the columns: more warps to hide the epilogue's latencies).
// ASRC != ASRC_TMA: the A operand is made by TC_A_WARPS more warps (a_producer_stage)
// straight into the stages' A halves; the TMA warp then loads only W.
template <int EPI, int TC_STAGES, int TC_STG_BUFS, bool PAIR, int EW = TC_EPI_WARPS,
          int ASRC = ASRC_TMA>
__global__ void __launch_bounds__(32 * (2 + EW + (ASRC != ASRC_TMA ? TC_A_WARPS : 0)), 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmBp,
                   const GemmArgs g) {
  static_assert(ASRC == ASRC_TMA || PAIR, "a made A operand is always split");
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int AST = PAIR ? 2 * TC_A_BYTES : TC_A_BYTES;  // A bytes of a stage
  uint8_t* sA = smem;                                       // stage s at sA + s * AST
  uint8_t* sB = smem + TC_STAGES * AST;
  uint8_t* sStage = sB + TC_STAGES * TC_B_BYTES;  // epilogue staging
  __shared__ __align__(8) uint64_t full_bar[TC_STAGES], empty_bar[TC_STAGES];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2];
  __shared__ uint32_t s_tmem;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // ring steps per tile: 64-wide K blocks of A, or of W when A_hi / A_lo share a stage
  const int KB = (PAIR ? g.Kw : g.Ka) / TC_BK;
  const int NT = (g.N + TC_BN - 1) / TC_BN;
  const int MT = static_cast<int>((g.M + TC_BM - 1) / TC_BM);
  const int ntiles = NT * MT;

  if (tid == 0) {
    for (int s = 0; s < TC_STAGES; ++s) {
      // the TMA warp's expect-tx arrival, plus one arrival per A-producer thread
      mbar_init(&full_bar[s], 1 + (ASRC != ASRC_TMA ? 32 * TC_A_WARPS : 0));
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], EW);
    }
    fence_mbar_init();
  }
  if constexpr (ASRC == ASRC_CONF) {
    // the confidence layer's weights [Kw][5] and biases [Kw], as 6 floats per hidden unit
    float* wt = reinterpret_cast<float*>(sStage + EW * TC_STG_BUFS * TC_STG_BYTES);
    for (int i = tid; i < g.Kw * 6; i += blockDim.x) {
      const int h = i / 6, c = i - 6 * h;
      wt[i] = c < 5 ? g.a_w1[h * 5 + c] : g.a_b1[h];
    }
  }
  if (warp == 0) tmem_alloc(&s_tmem, TC_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_wait();
  pdl_trigger();

  if (warp == 0 && lane == 0) {
    // ---- producer: the smem ring runs on across this CTA's tiles
    int it = 0;
    bool ok = true;
    const int nitems = tc_items(g, ntiles);
    for (int w = blockIdx.x; w < nitems && ok; w += gridDim.x) {
      const TcItem item = tc_item(g, ntiles, w);
      const int t = item.t;
      // W rows of the tile, or of the piece (tmBp: boxes of the piece's width)
      const int m0 = (t / NT) * TC_BM, n0 = (t % NT) * TC_BN + item.c0;
      const CUtensorMap* wmap = item.bn == TC_BN ? &tmB : &tmBp;
      const uint32_t wbytes = uint32_t(item.bn) * TC_BK * 2;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % TC_STAGES, use = it / TC_STAGES;
        if (use > 0 && !mbar_wait_bounded(&empty_bar[s], (use - 1) & 1, &g_err_tc, ERR_TC_EMPTY)) {
          ok = false;
          break;
        }
        if constexpr (ASRC != ASRC_TMA) {
          // W block of ring step kb: for the fusion input the steps alternate between the
          // h and the h * t halves of one 64-column block
          const int wk = ASRC == ASRC_FUSION ? (kb & 1) * (g.Kw / 2) + (kb >> 1) * TC_BK : kb * TC_BK;
          mbar_arrive_expect_tx(&full_bar[s], wbytes);
          tma_load_2d(sB + s * TC_B_BYTES, wmap, wk, n0, &full_bar[s]);
          continue;
        }
        mbar_arrive_expect_tx(&full_bar[s], AST + wbytes);
        if constexpr (PAIR) {
          tma_load_2d(sA + s * AST, &tmA, kb * TC_BK, m0, &full_bar[s]);
          tma_load_2d(sA + s * AST + TC_A_BYTES, &tmA, g.Kw + kb * TC_BK, m0, &full_bar[s]);
          tma_load_2d(sB + s * TC_B_BYTES, wmap, kb * TC_BK, n0, &full_bar[s]);
        } else {
          tma_load_2d(sA + s * AST, &tmA, kb * TC_BK, m0, &full_bar[s]);
          tma_load_2d(sB + s * TC_B_BYTES, wmap, (kb * TC_BK) % g.Kw, n0, &full_bar[s]);
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    int it = 0, i = 0;
    bool ok = true;
    const int nitems = tc_items(g, ntiles);
    for (int w = blockIdx.x; w < nitems && ok; w += gridDim.x, ++i) {
      const uint32_t idesc = idesc_bf16(TC_BM, tc_item(g, ntiles, w).bn);
      const int buf = i & 1;
      const uint32_t acc = tmem + uint32_t(buf * TC_BN);
      if (i >= 2 && !mbar_wait_bounded(&acc_empty[buf], ((i >> 1) - 1) & 1, &g_err_tc,
                                        ERR_TC_ACC_EMPTY)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % TC_STAGES, use = it / TC_STAGES;
        if (!mbar_wait_bounded(&full_bar[s], use & 1, &g_err_tc, ERR_TC_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < TC_BK / 16; ++kk)
          umma_bf16(acc, sw128_desc(sA + s * AST + kk * 32),
                    sw128_desc(sB + s * TC_B_BYTES + kk * 32), idesc, (kb | kk) != 0);
        if constexpr (PAIR) {  // A_lo against the same W block
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk)
            umma_bf16(acc, sw128_desc(sA + s * AST + TC_A_BYTES + kk * 32),
                      sw128_desc(sB + s * TC_B_BYTES + kk * 32), idesc, 1u);
        }
        umma_commit(&empty_bar[s]);
      }
      umma_commit(&acc_full[buf]);
    }
  } else if (warp >= 2 && warp < 2 + EW) {
    // ---- epilogue: quarter q = warp % 4 owns TMEM lanes 32q..32q+31 (output rows);
    // the two warps of a quarter split the tile's columns in halves
    constexpr int CPP = (TC_BN / 32) / (EW / 4);  // 32-column chunks per epilogue warp
    const int q = warp & 3, half = (warp - 2) >> 2;  // half: this warp's column part
    uint8_t* stg = sStage + (warp - 2) * TC_STG_BUFS * TC_STG_BYTES;
    int sb = 0;  // staging buffer of the next chunk
    int i = 0;
    const int nitems = tc_items(g, ntiles);
    for (int w = blockIdx.x; w < nitems; w += gridDim.x, ++i) {
      const TcItem item = tc_item(g, ntiles, w);
      const int t = item.t;
      const int buf = i & 1;
      const int64_t m0 = int64_t(t / NT) * TC_BM;
      const int n0 = (t % NT) * TC_BN + item.c0;  // the accumulator's column 0
      const int64_t m = m0 + 32 * q + lane;
      // node sum: the row's gather sources before the accumulator is waited for
      NodeRow nr{};
      const bool mrow = m < g.M;
      if constexpr (EPI == EPI_NODE) {
        if (mrow) nr = tc_node_row(g, m);
      }
      if (!mbar_wait_bounded(&acc_full[buf], (i >> 1) & 1, &g_err_tc, ERR_TC_ACCUM)) break;
      tc_fence_after();
#pragma unroll 1
      for (int cc = half * CPP; cc < (half + 1) * CPP; ++cc) {
        if (cc * 32 >= item.bn) break;  // a piece: only its own columns
        float v[32];
        const int n = n0 + cc * 32;
        if constexpr (EPI == EPI_NODE) {
          // DRAM gathers first, then the accumulator, the sums and the staged f32 store
          uint4 ge[4], gh[4];
          const bool live = mrow && n < g.N;
          if (live) tc_node_gather(nr, n, ge, gh);
          tmem_ld32(tmem + (uint32_t(32 * q) << 16) + uint32_t(buf * TC_BN + cc * 32), v);
          if (live) tc_node_terms(g, nr, m, n, v, ge, gh);
          if (n < g.N) {
            if (lane == 0) {
              if constexpr (TC_STG_BUFS == 2)
                bulk_wait_read1();
              else
                bulk_wait_read0();
            }
            __syncwarp();
            tc_epilogue_staged<EPI_F32>(g, &tmC, stg + sb * TC_STG_BYTES, lane, m0 + 32 * q,
                                        n, v, nullptr);
            sb = (sb + 1) % TC_STG_BUFS;
          }
        } else if (n < g.N) {
          // the bias is loaded ahead of the waits where registers allow (8 epilogue warps,
          // no producer warps: 112+ registers a thread)
          constexpr bool EARLY = EW == 8 && ASRC == ASRC_TMA;
          float4 bq[8];
          if constexpr (EARLY) tc_bias_fetch(g, m0 + 32 * q, lane, n, bq);
          tmem_ld32(tmem + (uint32_t(32 * q) << 16) + uint32_t(buf * TC_BN + cc * 32), v);
          // the buffer's previous bulk copy must have finished reading it
          if (lane == 0) {
            if constexpr (TC_STG_BUFS == 2)
              bulk_wait_read1();
            else
              bulk_wait_read0();
          }
          __syncwarp();
          if constexpr (!EARLY) tc_bias_fetch(g, m0 + 32 * q, lane, n, bq);
          tc_epilogue_staged<EPI>(g, &tmC, stg + sb * TC_STG_BYTES, lane, m0 + 32 * q, n, v, bq);
          sb = (sb + 1) % TC_STG_BUFS;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  } else if (ASRC != ASRC_TMA && warp >= 2 + EW) {
    // ---- A producers: each thread makes the same 16-byte unit of 4 rows of every stage
    const int at = tid - 32 * (2 + EW);
    const int unit = at & 7, rsub = at >> 3;  // rows rsub + 32 i
    a_producer<ASRC, TC_STAGES>(g, sA, AST, full_bar, empty_bar, KB, NT, ntiles, unit, rsub,
                     reinterpret_cast<const float*>(sStage + EW * TC_STG_BUFS * TC_STG_BYTES));
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TC_TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// Row-major bf16 matrix [rows, cols] read in boxes of box_rows x 64 columns.
static bool make_tmap(CUtensorMap* tm, const void* ptr, uint64_t rows, uint64_t cols,
                      uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {TC_BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output matrix [rows, cols] (bf16 or f32) written in 32 x 32 boxes whose 64- or
// 128-byte rows use the matching swizzle.
static bool make_tmap_out(CUtensorMap* tm, void* ptr, uint64_t rows, uint64_t cols, bool f32) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t es = f32 ? 4 : 2;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * es};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr,
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool gemm_tc_supported(const GemmArgs& g) {
  return g.Kw % TC_BK == 0 && g.Ka % TC_BK == 0 && (g.Ka == g.Kw || g.Ka == 2 * g.Kw) &&
         g.N % 32 == 0 && g.M > 0 &&
         (reinterpret_cast<uintptr_t>(g.A) % 16) == 0 && (reinterpret_cast<uintptr_t>(g.W) % 16) == 0;
}

// The tail plan of a launch over ntiles tiles on `sms` SMs: the tiles of the last,
// part-filled round of the persistent grid (all of them when there are fewer tiles than
// SMs) run as 2, 4 or 8 column pieces, as many as keep the pieces within one round.
// Returns the number of work items (the grid is min(items, sms)).
static int64_t tc_tail_plan(GemmArgs& g, int64_t ntiles, int sms) {
  g.tail_tiles = 0;
  g.tail_split = 1;
  const int64_t r = ntiles % sms;
  if (r == 0) return ntiles;
  int sp = 1;
  while (sp < 8 && r * sp * 2 <= sms) sp *= 2;
  if (sp == 1) return ntiles;
  g.tail_tiles = static_cast<int>(r);
  g.tail_split = sp;
  return ntiles + r * (sp - 1);
}

cudaError_t launch_gemm(int epi, const GemmArgs& g_in, cudaStream_t stream) {
  GemmArgs g = g_in;
  CUtensorMap ta, tb, tc;
  if (g.asrc != ASRC_TMA) {
    // A made in the kernel: the fusion input under the SiLU-split epilogue, or the
    // confidence layer under the node epilogue; both split (Ka = 2 Kw)
    const bool fusion = g.asrc == ASRC_FUSION && epi == EPI_SPLIT_SILU && g.a_x &&
                        g.a_group > 0 && g.Kw % (2 * TC_BK) == 0 &&
                        reinterpret_cast<uintptr_t>(g.a_x) % 16 == 0 &&
                        reinterpret_cast<uintptr_t>(g.a_t) % 16 == 0;
    const bool conf = g.asrc == ASRC_CONF && epi == EPI_NODE && g.a_cl && g.a_lse && g.a_w1 &&
                      g.a_b1 && g.K >= 1;
    if (!(fusion || conf) || g.Ka != 2 * g.Kw || g.Kw % TC_BK || g.N % 32 || g.M <= 0 ||
        reinterpret_cast<uintptr_t>(g.W) % 16)
      return cudaErrorInvalidValue;
    // (the A tensor map is not read; it is encoded over W only to fill the argument)
    if (!make_tmap(&ta, g.W, uint64_t(g.N), uint64_t(g.Kw), TC_BM) ||
        !make_tmap(&tb, g.W, uint64_t(g.N), uint64_t(g.Kw), TC_BN))
      return cudaErrorInvalidValue;
    if (fusion) {
      if (!g.out_split || reinterpret_cast<uintptr_t>(g.out_split) % 16 ||
          !make_tmap_out(&tc, g.out_split, uint64_t(g.M), uint64_t(2 * g.N), false))
        return cudaErrorInvalidValue;
    } else if (!g.out || reinterpret_cast<uintptr_t>(g.out) % 16 ||
               !make_tmap_out(&tc, g.out, uint64_t(g.M), uint64_t(g.N), true)) {
      return cudaErrorInvalidValue;
    }
    const int sms = device_sm_count();
    const int64_t ntiles = int64_t((g.N + TC_BN - 1) / TC_BN) * ((g.M + TC_BM - 1) / TC_BM);
    const int64_t nitems = tc_tail_plan(g, ntiles, sms);
    const dim3 grid(static_cast<unsigned>(nitems < sms ? nitems : sms));
    CUtensorMap tbp = tb;  // W in boxes of a tail piece's width
    if (g.tail_split > 1 &&
        !make_tmap(&tbp, g.W, uint64_t(g.N), uint64_t(g.Kw), uint32_t(TC_BN / g.tail_split)))
      return cudaErrorInvalidValue;
    constexpr int threads = 32 * (2 + TC_EPI_WARPS + TC_A_WARPS);
    cudaError_t e;
    if (fusion) {
      constexpr int sm = tc_smem(3, 1, true);
      auto k = gemm_tc_kernel<EPI_SPLIT_SILU, 3, 1, true, TC_EPI_WARPS, ASRC_FUSION>;
      e = allow_dynamic_smem(reinterpret_cast<const void*>(k), sm);
      if (e == cudaSuccess) e = launch_k(k, grid, dim3(threads), sm, stream, ta, tb, tc, tbp, g);
    } else {
      const int sm = tc_smem(2, 2, true) + g.Kw * 6 * 4;  // + the layer's weight table
      if (sm > 227 * 1024) return cudaErrorInvalidValue;
      auto k = gemm_tc_kernel<EPI_NODE, 2, 2, true, TC_EPI_WARPS, ASRC_CONF>;
      e = allow_dynamic_smem(reinterpret_cast<const void*>(k), sm);
      if (e == cudaSuccess) e = launch_k(k, grid, dim3(threads), sm, stream, ta, tb, tc, tbp, g);
    }
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
  }
  if (!gemm_tc_supported(g)) return cudaErrorInvalidValue;
  if (!make_tmap(&ta, g.A, uint64_t(g.M), uint64_t(g.Ka), TC_BM) ||
      !make_tmap(&tb, g.W, uint64_t(g.N), uint64_t(g.Kw), TC_BN))
    return cudaErrorInvalidValue;
  if (epi == EPI_SPLIT || epi == EPI_SPLIT_SILU) {
    if (!g.out_split || reinterpret_cast<uintptr_t>(g.out_split) % 16 ||
        !make_tmap_out(&tc, g.out_split, uint64_t(g.M), uint64_t(2 * g.N), false))
      return cudaErrorInvalidValue;
  } else {
    if (!g.out || reinterpret_cast<uintptr_t>(g.out) % 16 ||
        !make_tmap_out(&tc, g.out, uint64_t(g.M), uint64_t(g.N), true))
      return cudaErrorInvalidValue;
  }
  // A split operand (Ka = 2 Kw) runs paired stages: A_hi and A_lo share one W block.
  // Measured per epilogue at the high-concurrency sizes: the node sum (embedding-row
  // gathers) runs faster with 2 paired stages in flight than with 3 (less operand traffic
  // competing with its gathers), with two staging buffers per epilogue warp; the others
  // with 3 stages.
  const bool pair = g.Ka == 2 * g.Kw;
  // The SiLU epilogue of short K (FFN1) is the longest epilogue per MMA: it runs 16
  // epilogue warps (2 paired stages leave room for their staging buffers).
  const bool wide = epi == EPI_SPLIT_SILU && g.Ka <= 512;
  const bool two = epi == EPI_NODE;
  constexpr int sp = tc_smem(3, 1, true), sp2 = tc_smem(2, 2, true), sn = tc_smem(4, 1, false);
  constexpr int sw = tc_smem(2, 1, true, 16);
  const int sms = device_sm_count();
  const int64_t ntiles = int64_t((g.N + TC_BN - 1) / TC_BN) * ((g.M + TC_BM - 1) / TC_BM);
  const int64_t nitems = tc_tail_plan(g, ntiles, sms);
  const dim3 grid(static_cast<unsigned>(nitems < sms ? nitems : sms));
  CUtensorMap tbp = tb;  // W in boxes of a tail piece's width
  if (g.tail_split > 1 &&
      !make_tmap(&tbp, g.W, uint64_t(g.N), uint64_t(g.Kw), uint32_t(TC_BN / g.tail_split)))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaSuccess;
  // the chosen instance's shared-memory limit (once per device), then its launch
#define LC_TC_RUN(E, KERNEL, THREADS, SMEM)                                                  \
  {                                                                                          \
    e = allow_dynamic_smem(reinterpret_cast<const void*>(KERNEL), SMEM);                     \
    if (e == cudaSuccess) e = launch_k(KERNEL, grid, dim3(THREADS), SMEM, stream, ta, tb, tc, tbp, g); \
  }
#define LC_TC_LAUNCH(E)                                                                      \
  if (pair && wide)                                                                          \
    LC_TC_RUN(E, (gemm_tc_kernel<E, 2, 1, true, 16>), 32 * 18, sw)                           \
  else if (pair && two)                                                                      \
    LC_TC_RUN(E, (gemm_tc_kernel<E, 2, 2, true>), TC_THREADS, sp2)                           \
  else if (pair)                                                                             \
    LC_TC_RUN(E, (gemm_tc_kernel<E, 3, 1, true>), TC_THREADS, sp)                            \
  else                                                                                       \
    LC_TC_RUN(E, (gemm_tc_kernel<E, 4, 1, false>), TC_THREADS, sn)
  switch (epi) {
    case EPI_F32: LC_TC_LAUNCH(EPI_F32) break;
    case EPI_RESID: LC_TC_LAUNCH(EPI_RESID) break;
    case EPI_SPLIT: LC_TC_LAUNCH(EPI_SPLIT) break;
    case EPI_SPLIT_SILU: LC_TC_LAUNCH(EPI_SPLIT_SILU) break;
    default: LC_TC_LAUNCH(EPI_NODE) break;
  }
#undef LC_TC_RUN
#undef LC_TC_LAUNCH
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------------------ LM head + top-K / LSE
//
// The drafter's vocabulary projection fused with step a1 (the follow-on the serving
// write-up lists after the rerank: the projection's logits go straight into the top-K /
// log-partition pass instead of a round trip through HBM):
//   logit[r, v] = hidden[r, :] . W[v, :]   (bf16 operands, f32 accumulation)
// and for every row its K best (value desc, id asc) and the online log-sum-exp.  A CTA
// owns one 128-row tile and one contiguous range of 256-column vocabulary tiles; the MMA
// side is the plain (non-split) form of the kernel above, and the epilogue warps keep,
// per (row, column half), a running base-2 log-sum-exp and a sorted top-K in registers.
// At the end the two halves of a row are merged and one record per (row, range) is
// written in the vocabulary-shard record format, which the shard merge reduces to the
// outputs.
constexpr float LM_LOG2E = 1.4426950408889634f;
constexpr float LM_M2_INIT = -1e30f;

struct LmArgs {
  int64_t rows, V;
  int D, K;
  int nr;   // vocabulary ranges per row tile
  int tpr;  // 256-column tiles per range
  char* records;  // [nr][rows] records of 8 + 8 K bytes
};

__device__ __forceinline__ bool lm_better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

template <int KM>
__global__ void __launch_bounds__(TC_THREADS, 1)
    lm_head_topk_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const LmArgs a) {
  constexpr int ST = 4;
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + ST * TC_A_BYTES;
  __shared__ __align__(8) uint64_t full_bar[ST], empty_bar[ST];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2];
  __shared__ uint32_t s_tmem;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int KB = a.D / TC_BK;
  const int NT = static_cast<int>((a.V + TC_BN - 1) / TC_BN);
  const int mt = blockIdx.x / a.nr, rg = blockIdx.x % a.nr;
  const int nt0 = rg * a.tpr, nt1 = min(NT, nt0 + a.tpr);
  const int64_t m0 = int64_t(mt) * TC_BM;

  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], TC_EPI_WARPS);
    }
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&s_tmem, TC_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0 && lane == 0) {
    // ---- producer: hidden rows of the tile and the vocabulary rows of each N tile
    int it = 0;
    bool ok = true;
    for (int nt = nt0; nt < nt1 && ok; ++nt) {
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % ST, use = it / ST;
        if (use > 0 && !mbar_wait_bounded(&empty_bar[s], (use - 1) & 1, &g_err_tc, ERR_TC_EMPTY)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full_bar[s], TC_A_BYTES + TC_B_BYTES);
        tma_load_2d(sA + s * TC_A_BYTES, &tmA, kb * TC_BK, static_cast<int>(m0), &full_bar[s]);
        tma_load_2d(sB + s * TC_B_BYTES, &tmB, kb * TC_BK, nt * TC_BN, &full_bar[s]);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    constexpr uint32_t idesc = idesc_bf16(TC_BM, TC_BN);
    int it = 0, i = 0;
    bool ok = true;
    for (int nt = nt0; nt < nt1 && ok; ++nt, ++i) {
      const int buf = i & 1;
      const uint32_t acc = tmem + uint32_t(buf * TC_BN);
      if (i >= 2 && !mbar_wait_bounded(&acc_empty[buf], ((i >> 1) - 1) & 1, &g_err_tc,
                                        ERR_TC_ACC_EMPTY)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % ST, use = it / ST;
        if (!mbar_wait_bounded(&full_bar[s], use & 1, &g_err_tc, ERR_TC_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < TC_BK / 16; ++kk)
          umma_bf16(acc, sw128_desc(sA + s * TC_A_BYTES + kk * 32),
                    sw128_desc(sB + s * TC_B_BYTES + kk * 32), idesc, (kb | kk) != 0);
        umma_commit(&empty_bar[s]);
      }
      umma_commit(&acc_full[buf]);
    }
  } else if (warp >= 2) {
    // ---- epilogue: quarter q = TMEM lanes 32q.. (rows), half = the tile's column half
    const int q = warp & 3, half = (warp - 2) >> 2;
    const int K = a.K;
    float m2 = LM_M2_INIT, ssum = 0.f;
    float tv[KM];
    int ti[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      tv[j] = -INFINITY;
      ti[j] = INT_MAX;
    }
    float kth = -INFINITY;  // tv[K - 1]
    bool done = false;
    int i = 0;
    for (int nt = nt0; nt < nt1; ++nt, ++i) {
      const int buf = i & 1;
      if (!mbar_wait_bounded(&acc_full[buf], (i >> 1) & 1, &g_err_tc, ERR_TC_ACCUM)) {
        done = true;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int cc = half * (TC_BN / 64); cc < (half + 1) * (TC_BN / 64); ++cc) {
        float v[32];
        tmem_ld32(tmem + (uint32_t(32 * q) << 16) + uint32_t(buf * TC_BN + cc * 32), v);
        const int64_t n = int64_t(nt) * TC_BN + cc * 32;
        const int64_t left = a.V - n;
        const int nvalid = left < 32 ? static_cast<int>(left) : 32;
        // online log-sum-exp over the chunk's valid columns
        float cmax = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nvalid) cmax = fmaxf(cmax, v[j]);
        const float c2 = cmax * LM_LOG2E;
        if (c2 > m2) {
          ssum *= exp2f(m2 - c2);
          m2 = c2;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nvalid) ssum += exp2f(fmaf(v[j], LM_LOG2E, -m2));
        // top-K: ids only grow along this thread's columns, so a value equal to the K-th
        // cannot enter; insertion keeps tv sorted (value desc, id asc)
        if (cmax > kth) {
#pragma unroll 1
          for (int j = 0; j < nvalid; ++j) {
            float x = v[0];
#pragma unroll
            for (int u = 1; u < 32; ++u)
              if (j == u) x = v[u];
            if (!(x > kth)) continue;
            const int id = static_cast<int>(n) + j;
            bool placed = false;
#pragma unroll
            for (int u = KM - 1; u >= 0; --u) {
              if (u >= K || placed) continue;
              if (u > 0 && lm_better(x, id, tv[u - 1], ti[u - 1])) {
                tv[u] = tv[u - 1];
                ti[u] = ti[u - 1];
              } else {
                tv[u] = x;
                ti[u] = id;
                placed = true;
              }
            }
#pragma unroll
            for (int u = 0; u < KM; ++u)
              if (u == K - 1) kth = tv[u];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
    // ---- merge the two column halves of each row through shared memory (the operand
    // ring is idle once the last accumulator has been read), then write the record
    tc_fence_before();
    asm volatile("bar.sync %0, 256;" ::"r"(1) : "memory");  // every epilogue warp is done
    float* scr = reinterpret_cast<float*>(sA);  // [128 rows][2 halves][2 + 2 KM]
    constexpr int RS = 2 + 2 * KM;
    const int r = 32 * q + lane;
    float* mine = scr + (r * 2 + half) * RS;
    mine[0] = m2;
    mine[1] = ssum;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      mine[2 + j] = tv[j];
      reinterpret_cast<int*>(mine)[2 + KM + j] = ti[j];
    }
    asm volatile("bar.sync %0, 256;" ::"r"(1) : "memory");
    const int64_t row = m0 + r;
    if (half == 0 && row < a.rows && !done) {
      const float* p0 = scr + (r * 2) * RS;
      const float* p1 = p0 + RS;
      float M = fmaxf(p0[0], p1[0]);
      const float S = p0[1] * exp2f(p0[0] - M) + p1[1] * exp2f(p1[0] - M);
      char* rec = a.records + (int64_t(rg) * a.rows + row) * (8 + 8 * int64_t(K));
      reinterpret_cast<float*>(rec)[0] = M;
      reinterpret_cast<float*>(rec)[1] = S;
      float* rv = reinterpret_cast<float*>(rec + 8);
      int* ri = reinterpret_cast<int*>(rec + 8 + 4 * K);
      const int* i0 = reinterpret_cast<const int*>(p0) + 2 + KM;
      const int* i1 = reinterpret_cast<const int*>(p1) + 2 + KM;
      int x = 0, y = 0;
      for (int o = 0; o < K; ++o) {
        const bool take0 = y >= K || (x < K && lm_better(p0[2 + x], i0[x], p1[2 + y], i1[y]));
        if (take0) {
          rv[o] = p0[2 + x];
          ri[o] = i0[x];
          ++x;
        } else {
          rv[o] = p1[2 + y];
          ri[o] = i1[y];
          ++y;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TC_TMEM_COLS);
  }
}

bool lm_head_supported(int64_t rows, int64_t V, int D, int K) {
  return rows >= 1 && V >= 1 && V < (int64_t(1) << 31) - 256 && D >= TC_BK && D % TC_BK == 0 &&
         K >= 1 && K <= 32 && K <= V;
}

static void lm_head_plan(int64_t rows, int64_t V, int* nr, int* tpr) {
  const int sms = device_sm_count();
  const int64_t MT = (rows + TC_BM - 1) / TC_BM, NT = (V + TC_BN - 1) / TC_BN;
  int64_t want = std::max<int64_t>(1, (sms + MT / 2) / MT);  // ranges so that MT x nr ~ SMs
  want = std::min<int64_t>(want, NT);
  *tpr = static_cast<int>((NT + want - 1) / want);
  *nr = static_cast<int>((NT + *tpr - 1) / *tpr);
}

size_t lm_head_records_bytes(int64_t rows, int64_t V, int K) {
  int nr = 1, tpr = 1;
  lm_head_plan(rows, V, &nr, &tpr);
  return size_t(nr) * size_t(rows) * (8 + 8 * size_t(K));
}

cudaError_t launch_lm_head_topk(const __nv_bfloat16* hidden, const __nv_bfloat16* w_lm,
                                int64_t rows, int64_t V, int D, int K, void* records,
                                int32_t* cand_id, float* cand_logit, float* lse,
                                cudaStream_t stream) {
  if (!lm_head_supported(rows, V, D, K) || reinterpret_cast<uintptr_t>(hidden) % 16 ||
      reinterpret_cast<uintptr_t>(w_lm) % 16 || reinterpret_cast<uintptr_t>(records) % 4)
    return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, hidden, uint64_t(rows), uint64_t(D), TC_BM) ||
      !make_tmap(&tb, w_lm, uint64_t(V), uint64_t(D), TC_BN))
    return cudaErrorInvalidValue;
  LmArgs la{};
  la.rows = rows;
  la.V = V;
  la.D = D;
  la.K = K;
  la.records = static_cast<char*>(records);
  lm_head_plan(rows, V, &la.nr, &la.tpr);
  const int64_t MT = (rows + TC_BM - 1) / TC_BM;
  const dim3 grid(static_cast<unsigned>(MT * la.nr));
  constexpr int sm = 4 * (TC_A_BYTES + TC_B_BYTES) + 1024;
  {
    cudaError_t e = allow_dynamic_smem(
        K <= 8    ? reinterpret_cast<const void*>(lm_head_topk_kernel<8>)
        : K <= 16 ? reinterpret_cast<const void*>(lm_head_topk_kernel<16>)
                  : reinterpret_cast<const void*>(lm_head_topk_kernel<32>),
        sm);
    if (e != cudaSuccess) return e;
  }
  if (K <= 8)
    lm_head_topk_kernel<8><<<grid, TC_THREADS, sm, stream>>>(ta, tb, la);
  else if (K <= 16)
    lm_head_topk_kernel<16><<<grid, TC_THREADS, sm, stream>>>(ta, tb, la);
  else
    lm_head_topk_kernel<32><<<grid, TC_THREADS, sm, stream>>>(ta, tb, la);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return k1_merge_launch(records, la.nr, rows, K, cand_id, cand_logit, lse, stream);
}

cudaError_t tc_read_device_error(uint32_t* code) {
  uint32_t v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_err_tc, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_err_tc, &zero, sizeof(zero));
  *code |= v << 8;
  return e;
}

}  // namespace lilicorr
