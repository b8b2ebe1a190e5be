// smx_tc.cuh -- fifth-generation tensor cores (tcgen05): tensor memory, shared-memory matrix
// descriptors and the bf16 MMA the attention uses.
//
// Operand tiles are bf16 [rows][128] in shared memory, K-major with the 128-byte swizzle: two
// K blocks of 64 elements, each rows x 128 B, in 8-row atoms of 1024 B; the 16-byte chunk c of
// row r sits at chunk c ^ (r % 8). One MMA step (K = 16, 32 bytes of every row) starts 32 * (k % 4)
// bytes into K block k / 4. The accumulator D (fp32, 128 rows x N columns) lives in tensor memory:
// row i in lane i, column j in column j of the allocation.
#pragma once

#include <stdint.h>

#include "smx_device.cuh"

namespace smx {

// Byte offset of element (r, k) of a bf16 [rows][128] tile in the layout above.
__host__ __device__ __forceinline__ uint32_t sw128_off(int r, int k, int rows) {
    const int kb = k >> 6, kk = k & 63;
    return (uint32_t)(kb * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + ((((kk >> 3) ^ (r & 7)) & 7) << 4) + (kk & 7) * 2);
}

// Byte offset of the 16-byte chunk holding elements 8c .. 8c + 7 of row r.
__host__ __device__ __forceinline__ uint32_t sw128_chunk(int r, int c, int rows) {
    return (uint32_t)((c >> 3) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);   // start address
    d |= (uint64_t)1 << 16;                     // leading byte offset (unused when swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset between 8-row atoms
    d |= (uint64_t)1 << 46;                     // descriptor version
    d |= (uint64_t)2 << 61;                     // 128-byte swizzle
    return d;
}

// Instruction descriptor: dense kind::f16, bf16 A and B (both K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Allocate ncols (a power of two >= 32) tensor-memory columns; one whole warp calls it and the
// base address lands in *slot (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Free the columns (one whole warp; no MMA or load may still be using them).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[128 x N] (+)= A[128 x 128] . B[N x 128]^T over the 8 K steps of the tiles at a_s, b_s (one
// thread), then arrive on bar when the MMAs are done.
__device__ __forceinline__ void tc_mma_tile(uint32_t d_tmem, uint32_t a_s, uint32_t b_s, int a_rows, int b_rows,
                                            uint32_t idesc, bool accumulate, uint64_t* bar) {
    // bar == nullptr: no commit (a later tc_mma_tile's commit covers these MMAs too)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint64_t ad = sw128_desc(a_s + (k >> 2) * a_rows * 128 + (k & 3) * 32);
        const uint64_t bd = sw128_desc(b_s + (k >> 2) * b_rows * 128 + (k & 3) * 32);
        const uint32_t acc = (accumulate || k > 0) ? 1u : 0u;
        asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
                     " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem), "l"(ad), "l"(bd),
                     "r"(idesc), "r"(acc)
                     : "memory");
    }
    if (bar != nullptr)
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                     : "memory");
}

// Arrive on bar once every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's lane (the warp's 32 lanes) from taddr.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive fp32 columns of this thread's lane from taddr (waits for the load).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Store 16 fp32 columns of this thread's lane at taddr (waits for the store).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 64 consecutive fp32 columns of this thread's lane from taddr (one load; waits for it).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
        " tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Store 64 fp32 columns of this thread's lane at taddr (waits for the store).
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const float (&v)[64]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n"
        " tcgen05.wait::st.sync.aligned;"
        ::"r"(taddr),
          "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
          "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
          "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
          "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
          "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
          "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
          "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
          "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31])),
          "r"(__float_as_uint(v[32])), "r"(__float_as_uint(v[33])), "r"(__float_as_uint(v[34])), "r"(__float_as_uint(v[35])),
          "r"(__float_as_uint(v[36])), "r"(__float_as_uint(v[37])), "r"(__float_as_uint(v[38])), "r"(__float_as_uint(v[39])),
          "r"(__float_as_uint(v[40])), "r"(__float_as_uint(v[41])), "r"(__float_as_uint(v[42])), "r"(__float_as_uint(v[43])),
          "r"(__float_as_uint(v[44])), "r"(__float_as_uint(v[45])), "r"(__float_as_uint(v[46])), "r"(__float_as_uint(v[47])),
          "r"(__float_as_uint(v[48])), "r"(__float_as_uint(v[49])), "r"(__float_as_uint(v[50])), "r"(__float_as_uint(v[51])),
          "r"(__float_as_uint(v[52])), "r"(__float_as_uint(v[53])), "r"(__float_as_uint(v[54])), "r"(__float_as_uint(v[55])),
          "r"(__float_as_uint(v[56])), "r"(__float_as_uint(v[57])), "r"(__float_as_uint(v[58])), "r"(__float_as_uint(v[59])),
          "r"(__float_as_uint(v[60])), "r"(__float_as_uint(v[61])), "r"(__float_as_uint(v[62])), "r"(__float_as_uint(v[63]))
        : "memory");
}

// Four 32-bit words into columns taddr .. taddr + 3 of this thread's lane (waits for the store).
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};\n"
        " tcgen05.wait::st.sync.aligned;" ::"r"(taddr), "r"(a), "r"(b), "r"(c), "r"(d)
        : "memory");
}

// ---- block-scaled fp4 x e4m3 and MN-major operands --------------------------------------------
// kind::mxf8f6f4 reads an fp4 operand as 16-element chunks of 8 nibble bytes followed by 8
// bytes of padding, so a K-major [rows][128] fp4 tile has the byte layout of an 8-bit [rows][128]
// tile (128-byte rows, swizzled as above) and one MMA (K = 32) covers 32 bytes of every row.
// Scale factors (E8M0, one per 32 elements) sit in tensor memory: A row i's in lane i, B row n's
// in lane n % 32 of column n / 32 of the scale block, in every 32-lane quadrant (a D row reads
// the copy in its own quadrant); byte j of each 32-bit cell is the scale the MMA with scale id j
// uses.

// Instruction descriptor: kind::mxf8f6f4 with E8M0 scales, A e4m3 and B e2m1 (both K-major),
// fp32 D, M x N, scale byte `sf` of both operands' cells.
__host__ __device__ constexpr uint32_t idesc_mx_e4m3_e2m1(int M, int N, int sf) {
    return ((uint32_t)sf << 4) | (0u << 7) | (5u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(M >> 4) << 24) | ((uint32_t)sf << 29);
}

// D[128 x 128] = sum over the four 32-element groups g of (A_g 2^sfa_g) (B_g 2^sfb_g)^T: A the
// e4m3 tile at a_s, B the fp4 tile at b_s (both [128][128 elements], 128-byte rows), scale blocks
// at tensor-memory columns sfa, sfb. One thread; no commit.
__device__ __forceinline__ void tc_mma_mx_tile(uint32_t d_tmem, uint32_t a_s, uint32_t b_s, uint32_t sfa, uint32_t sfb) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint64_t ad = sw128_desc(a_s + 32 * g);
        const uint64_t bd = sw128_desc(b_s + 32 * g);
        const uint32_t idesc = idesc_mx_e4m3_e2m1(128, 128, g);
        asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %6, 0;\n"
                     " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}"
                     ::"r"(d_tmem), "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"((uint32_t)(g > 0))
                     : "memory");
    }
}

// Shared-memory matrix descriptor of an MN-major bf16 operand of 128 elements per K row: rows of
// 64 elements (128 bytes, swizzled as above) in 8-row atoms 1024 B apart, the two 64-element
// halves 16384 B apart. Element (k, n) sits where element (k, n) of a K-major [128][128] tile
// would (sw128_off(k, n, 128)).
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);   // start address
    d |= (uint64_t)(16384 >> 4) << 16;          // leading byte offset: between the 64-element halves
    d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset: between 8-row K atoms
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// D[128 x N] (+)= A[128 x 128] . B[128 x N]: A K-major, its two 64-element K blocks at a_lo and
// a_hi (each [128 rows][64], 8-row atoms 1024 B apart), B MN-major [k][n] at b_s (sw128_desc_mn;
// each 16-row K step is two atoms, 2048 B). N a multiple of 16, at most 192. One thread; no commit.
__device__ __forceinline__ void tc_mma_tile_bmn(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_s, int N,
                                                bool accumulate) {
    const uint32_t idesc = idesc_bf16(128, N) | (1u << 16);   // B MN-major
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint64_t ad = sw128_desc((k < 4 ? a_lo : a_hi) + (k & 3) * 32);
        const uint64_t bd = sw128_desc_mn(b_s + 2048 * k);
        const uint32_t acc = (accumulate || k > 0) ? 1u : 0u;
        asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
                     " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem), "l"(ad), "l"(bd),
                     "r"(idesc), "r"(acc)
                     : "memory");
    }
}

// One fp32 column of this thread's lane (waits for the load).
__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
    uint32_t r;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n tcgen05.wait::ld.sync.aligned;" : "=r"(r) : "r"(taddr)
                 : "memory");
    return __uint_as_float(r);
}

// Store one fp32 column of this thread's lane (waits for the store).
__device__ __forceinline__ void tmem_st1(uint32_t taddr, float v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};\n tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
                 "r"(__float_as_uint(v))
                 : "memory");
}

}  // namespace smx
