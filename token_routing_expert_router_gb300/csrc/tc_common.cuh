// Blackwell (sm_100 family, here sm_103a) primitives in inline PTX: mbarriers, TMA tensor
// loads, tcgen05 MMA / TMEM allocation / TMEM loads, and the shared-memory and instruction
// descriptors of tcgen05.mma. Each wrapper is one PTX instruction (or a short fixed
// sequence) as documented in the PTX ISA for tcgen05 and cp.async.bulk.tensor.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "moe_internal.cuh"

namespace moe {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- cluster (CTA pair)
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared::cluster address of the variable at shared::cta address `saddr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Every thread of both CTAs of the cluster (release/acquire: earlier memory operations,
// including mbarrier inits and remote arrives, are visible after it).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}


// Relaxed arrivals, for an epilogue handing a TMEM accumulator back to the MMA issuer. What
// must precede the arrival is the completion of the warp's tcgen05.ld reads of that buffer,
// and tcgen05.wait::ld has already blocked until they completed; the default release
// semantics would also hold the arrival until every global store the warp has issued is
// visible at the barrier's scope, which stalls the epilogue for nothing.
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// 16-byte copy from global to shared memory on the load/store pipe (completion tracked by
// commit/wait groups); the data is then made visible to the async proxy (the tensor core)
// with fence_proxy_async_smem before the stage's barrier arrival.
__device__ __forceinline__ void cp_async16(uint32_t dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `bar` with parity `parity`. Gives up when another role
// has aborted (*abort set) or after timeout_ns, in which case it records MOE_ERR_TIMEOUT,
// sets *abort so the other roles of the block stop too, and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t timeout_ns, DeviceStatus* st) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      *abort = 1;
      set_status(st, MOE_ERR_TIMEOUT, (int32_t)blockIdx.x);
      return false;
    }
  }
  return true;
}

// Bounded wait that ignores the abort flag: used when a block winds down, so that no TMA
// write or MMA completion is still in flight when it exits.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                                DeviceStatus* st) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) {
      set_status(st, MOE_ERR_TIMEOUT, (int32_t)blockIdx.x);
      return false;
    }
  }
  return true;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled load of the box at (x = inner coordinate, y = outer coordinate) into `dst`,
// completing `bytes` of transaction count on `bar`. x * element size is a multiple of 16.
__device__ __forceinline__ void tma_load_2d(const CUtensorMap* m, void* dst, uint64_t* bar, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_addr(bar)), "r"(x), "r"(y)
      : "memory");
}

// Pair form: the destination is this CTA's shared memory, the mbarrier (a shared::cluster
// address) may be in either CTA of the pair; used to complete the leader's barrier.
__device__ __forceinline__ void tma_load_2d_pair(const CUtensorMap* m, void* dst, uint32_t bar_cluster, int32_t x,
                                                 int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

// Row gather: four rows y0..y3 of a tensor whose map has a one-row box, columns [x, x + box
// width), written as four consecutive 128-byte rows at `dst` (the map's swizzle applies).
__device__ __forceinline__ void tma_gather4(const CUtensorMap* m, void* dst, uint64_t* bar, int32_t x, int32_t y0,
                                            int32_t y1, int32_t y2, int32_t y3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_addr(bar)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3)
      : "memory");
}

// Pair form of the row gather (the mbarrier may be in the other CTA of the pair).
__device__ __forceinline__ void tma_gather4_pair(const CUtensorMap* m, void* dst, uint32_t bar_cluster, int32_t x,
                                                 int32_t y0, int32_t y1, int32_t y2, int32_t y3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
// TMEM allocation by one warp of the CTA (CG = 1) or by one warp of each CTA of the pair
// (CG = 2); the address lands in shared memory.
template <int CG>
__device__ __forceinline__ void tmem_alloc_cg(uint32_t* dst_smem, uint32_t ncols) {
  if constexpr (CG == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc_cg(uint32_t taddr, uint32_t ncols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Pair MMA, issued by one thread of the leader CTA: A rows and B rows are split between the
// two CTAs' shared memory (same offsets), D rows between their TMEM (kind::f16, bf16).
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrival on the barrier at this shared::cta offset in every CTA of `mask` once all prior
// pair MMAs of this thread have completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "h"(mask)
               : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one elected thread; kind::f16 (bf16 inputs, fp32 acc).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same with kind::f8f6f4 (here e4m3 x e4m3, fp32 accumulate).
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier gets one arrival when every tcgen05 operation this thread issued before
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane (taddr.lane + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// (a0, a1) += (x0, x1) * f as one packed two-lane fp32 FMA (fma.rn.f32x2): each lane is
// rounded on its own, so the result is bit-identical to two fmaf calls at half the issue cost.
__device__ __forceinline__ void fma2(float& a0, float& a1, float x0, float x1, float f) {
  asm("{\n\t.reg .b64 a, x, s;\n\t"
      "mov.b64 a, {%0, %1};\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 s, {%4, %4};\n\t"
      "fma.rn.f32x2 a, x, s, a;\n\t"
      "mov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(x0), "f"(x1), "f"(f));
}

// A warp's 32 rows x 64 bytes, staged in shared memory so that the global stores are
// coalesced: each thread puts its own row's four 16-byte pieces in (stage_piece), then
// each store instruction of flush_rows_64B writes 8 rows x 64 contiguous bytes. Piece c of
// row r sits at r * 64 + 16 * (c ^ ((r >> 1) & 3)), which keeps both the row-wise writes
// and the column-wise reads free of bank conflicts. Row r goes to base + r * stride; rows
// r >= live (past the end of an expert's segment) are skipped.
__device__ __forceinline__ void stage_piece(uint8_t* stage, int lane, int c, uint4 v) {
  *reinterpret_cast<uint4*>(stage + lane * 64 + 16 * (c ^ ((lane >> 1) & 3))) = v;
}

__device__ __forceinline__ void flush_rows_64B(uint8_t* stage, int lane, uint8_t* base, int64_t stride, int live) {
  __syncwarp();
  const int c = lane & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int row = 8 * j + (lane >> 2);
    const uint4 v = *reinterpret_cast<const uint4*>(stage + row * 64 + 16 * (c ^ ((row >> 1) & 3)));
    if (row < live) *reinterpret_cast<uint4*>(base + row * stride + 16 * c) = v;
  }
  __syncwarp();
}

// Shared-memory matrix descriptor of tcgen05.mma for a K-major operand stored as rows of
// 128 bytes with the 128-byte swizzle (the layout a TMA load with SWIZZLE_128B writes):
// start address >> 4 (bits 0-13), leading byte offset 16 B (bits 16-29, unused for this
// layout), stride byte offset 1024 B between 8-row groups (bits 32-45), descriptor
// version 1 (bits 46-47), base offset 0, swizzle mode 2 = 128B (bits 61-63).
__device__ __forceinline__ uint64_t desc_k_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor: dense, D fp32 (bits 4-5 = 1), A/B type (bits 7-9, 10-12), both
// K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
// kind::f16: type 1 = bf16. kind::f8f6f4: type 0 = e4m3.
__host__ __device__ constexpr uint32_t idesc_make(uint32_t ab_type, int M, int N) {
  return (1u << 4) | (ab_type << 7) | (ab_type << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------- ragged tile schedule
// The grouped GEMMs' tiles over ragged groups: groups [0, G) are the routed experts (rows
// offsets[g + 1] - offsets[g], read on the device) and, when ngroups = G + 1, group G holds
// t_extra rows (the shared expert, or a single problem). One warp builds, 32 groups per
// step, seg_rows[g] and the exclusive prefix mt_prefix[0..ngroups] of the groups' m tiles
// ceil(rows / tm).
__device__ __forceinline__ void build_tile_prefix(const int32_t* offsets, int G, int ngroups, int t_extra, int tm,
                                                  int lane, int32_t* seg_rows, int32_t* mt_prefix) {
  int carry = 0;
  for (int g0 = 0; g0 < ngroups; g0 += 32) {
    const int g = g0 + lane;
    int rows = 0;
    if (g < G) rows = offsets[g + 1] - offsets[g];
    else if (g < ngroups) rows = t_extra;
    const int mt = (rows + tm - 1) / tm;
    int inc = mt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += o;
    }
    if (g < ngroups) {
      seg_rows[g] = rows;
      mt_prefix[g] = carry + inc - mt;
    }
    carry += __shfl_sync(0xffffffffu, inc, 31);
  }
  if (lane == 0) mt_prefix[ngroups] = carry;
}

struct TileCoord {
  int g, mb, nb, rows;  // group, m tile, n tile; rows: valid rows of the tile (<= tm)
};

// Tile index -> coordinates. Tiles run group-major, then n tile, then m tile, so the m
// tiles of one (group, n tile) run side by side and share the weight tile through L2; empty
// groups own no tiles.
__device__ __forceinline__ TileCoord decode_tile(int tile, const int32_t* mt_prefix, int ngroups, int n_tiles,
                                                 const int32_t* seg_rows, int tm) {
  int lo = 0, hi = ngroups - 1;  // largest g with n_tiles * mt_prefix[g] <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (n_tiles * mt_prefix[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  TileCoord c;
  c.g = lo;
  const int mt = mt_prefix[lo + 1] - mt_prefix[lo];
  const int local = tile - n_tiles * mt_prefix[lo];
  c.nb = local / mt;
  c.mb = local - c.nb * mt;
  c.rows = min(tm, seg_rows[lo] - c.mb * tm);
  return c;
}

}  // namespace tc
}  // namespace moe
