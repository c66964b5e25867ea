// Blackwell tensor-core (tcgen05 / TMEM) and TMA tensor-copy helpers for libdspark.
#pragma once

#include <cuda.h>  // CUtensorMap (types only; the encoder is fetched at run time)

#include "common.cuh"

namespace dspark {

// ---- host: 2-D tensor map for a row-major [rows, cols] 16-bit matrix ---------------
// Box = box_cols x box_rows elements, 128-byte swizzle (box_cols * 2 must be 128).
// Out-of-bounds elements of a box read as zero.
dspark_status make_tmap_2d(CUtensorMap *map, const void *base, bool bf16, uint64_t rows, uint64_t cols,
                           uint32_t box_rows, uint32_t box_cols);

// 3-D view of a row-major [rows, cols] 8-bit matrix (cols a multiple of 128) as
// [cols / 128][rows][128]: one box = box_katoms consecutive 128-byte column atoms of box_rows
// rows, stored atom after atom, each atom with the 128-byte swizzle (within each 1024-byte group
// of 8 rows, 16-byte chunk c of row r is stored at chunk c ^ (r & 7)).  One copy then reads
// box_katoms * 128 contiguous bytes of each row.  Out-of-bounds rows read as zero.
dspark_status make_tmap_kblocks_u8(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                                  uint32_t box_katoms);

// 3-D view of a row-major [rows, cols] 16-bit matrix (cols a multiple of 64) as
// [cols / 64][rows][64]: one box = box_kblocks consecutive 64-column blocks of box_rows rows,
// stored block after block, each in the 128-byte-swizzled layout of make_tmap_2d.
dspark_status make_tmap_kblocks(CUtensorMap *map, const void *base, bool bf16, uint64_t rows, uint64_t cols,
                                uint32_t box_rows, uint32_t box_kblocks);

// 3-D view of a row-major fp32 array [planes, rows, cols] (cols a multiple of 4, base 16-byte
// aligned): one box = box_cols consecutive columns of one row in each of box_planes planes,
// stored plane after plane without swizzle.  Out-of-range elements read as zero.
dspark_status make_tmap_rows_f32(CUtensorMap *map, const float *base, uint64_t planes, uint64_t rows, uint64_t cols,
                                 uint32_t box_planes, uint32_t box_cols);

// ---- device ----------------------------------------------------------------------
// Make this thread's generic-proxy shared-memory writes visible to the async proxy
// (tensor-core operand reads, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst_smem, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                            uint64_t l2_policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(l2_policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst_smem, const CUtensorMap *map, int x, int y, int z, uint64_t *bar,
                                            uint64_t l2_policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(l2_policy)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, both K-major; accumulate when acc != 0.
__device__ __forceinline__ void tc_mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// As tc_mma_f16 with the A operand read from tensor memory (128 lanes = rows, two 16-bit
// elements per 32-bit column along K) instead of shared memory.
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                              uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// Arrive (once) on `bar` when every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread t gets lane (taddr.lane + t).
__device__ __forceinline__ void tmem_ld_16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 8 consecutive 32-bit columns, waited for.
__device__ __forceinline__ void tmem_ld_8(uint32_t taddr, uint32_t (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// As tmem_ld_16 without the wait: several loads may be in flight; tmem_wait_ld() waits for all.
__device__ __forceinline__ void tmem_ld_16_async(uint32_t taddr, uint32_t *v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns from registers: thread t writes lane (taddr.lane + t).
// Completion is awaited with tmem_wait_st().
__device__ __forceinline__ void tmem_st_32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand in the 128-byte-swizzled layout a TMA
// tensor copy with CU_TENSOR_MAP_SWIZZLE_128B writes (rows of 128 B, 8-row atoms of
// 1024 B).  `addr` must lie in a 1024-byte-aligned tile; advancing along K inside the
// 128-byte row is done by adding the byte offset to `addr`.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);          // start address
    d |= static_cast<uint64_t>(1u) << 16;                         // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;                 // stride byte offset: 8-row atom
    d |= static_cast<uint64_t>(1u) << 46;                         // descriptor version
    d |= static_cast<uint64_t>(2u) << 61;                         // 128-byte swizzle
    return d;
}

// Instruction descriptor for kind::f16 with fp32 accumulation, K-major A and B.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int M, int N) {
    return (1u << 4)                                        // D = f32
           | ((bf16 ? 1u : 0u) << 7)                        // A type
           | ((bf16 ? 1u : 0u) << 10)                       // B type
           | (static_cast<uint32_t>(N >> 3) << 17)          // N
           | (static_cast<uint32_t>(M >> 4) << 24);         // M
}

}  // namespace dspark
