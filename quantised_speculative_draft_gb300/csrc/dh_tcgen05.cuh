// dh_tcgen05.cuh -- inline-PTX wrappers for the 5th-generation tensor-core instructions
// (tcgen05.*) used by the coarse-pass kernels, sm_103a only.
#pragma once

#include "dh_common.cuh"

namespace dh {

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// The same two instructions issued by one elected lane of a warp that runs the loop around them
// together: the operands are warp-uniform, so the loop's arithmetic stays on the uniform
// datapath and the instruction stream per MMA is short.
__device__ __forceinline__ void mma_ts_f8_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p, e;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "elect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void mma_commit_elect(uint64_t *bar)
{
    asm volatile("{\n\t.reg .pred e;\n\t"
                 "elect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_st_x64(uint32_t taddr, const uint32_t (&r)[64])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {"
                 "%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
                 "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, "
                 "%33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, "
                 "%49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};" ::
                     "r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                 "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
                 "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
                 "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
                 "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]),
                 "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]),
                 "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]),
                 "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]),
                 "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]),
                 "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]),
                 "r"(r[62]), "r"(r[63])
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {"
                 "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// One 16-column chunk of each of T terms (term t at columns taddr + t * stride ..), read with T
// tcgen05.ld and one wait in a single asm block, returned as packed pairs: u[t][i] holds
// columns 2i, 2i + 1 of term t, ready as FFMA2 operands.
__device__ __forceinline__ float2 pair_f2(uint64_t u)
{
    return make_float2(__uint_as_float(static_cast<uint32_t>(u)),
                       __uint_as_float(static_cast<uint32_t>(u >> 32)));
}

__device__ __forceinline__ void tmem_ld_terms2(uint32_t taddr, uint32_t stride, uint64_t (&u)[2][8])
{
    asm volatile("{\n\t.reg .b32 a<16>, b<16>;\n\t"
                 "tcgen05.ld.sync.aligned.32x32b.x16.b32 {a0, a1, a2, a3, a4, a5, a6, a7, a8, a9, a10, a11, a12, a13, a14, a15}, [%16];\n\t"
                 "tcgen05.ld.sync.aligned.32x32b.x16.b32 {b0, b1, b2, b3, b4, b5, b6, b7, b8, b9, b10, b11, b12, b13, b14, b15}, [%17];\n\t"
                 "tcgen05.wait::ld.sync.aligned;\n\t"
                 "mov.b64 %0, {a0, a1};\n\t"
                 "mov.b64 %1, {a2, a3};\n\t"
                 "mov.b64 %2, {a4, a5};\n\t"
                 "mov.b64 %3, {a6, a7};\n\t"
                 "mov.b64 %4, {a8, a9};\n\t"
                 "mov.b64 %5, {a10, a11};\n\t"
                 "mov.b64 %6, {a12, a13};\n\t"
                 "mov.b64 %7, {a14, a15};\n\t"
                 "mov.b64 %8, {b0, b1};\n\t"
                 "mov.b64 %9, {b2, b3};\n\t"
                 "mov.b64 %10, {b4, b5};\n\t"
                 "mov.b64 %11, {b6, b7};\n\t"
                 "mov.b64 %12, {b8, b9};\n\t"
                 "mov.b64 %13, {b10, b11};\n\t"
                 "mov.b64 %14, {b12, b13};\n\t"
                 "mov.b64 %15, {b14, b15};\n\t"
                 "}"
                 : "=l"(u[0][0]), "=l"(u[0][1]), "=l"(u[0][2]), "=l"(u[0][3]), "=l"(u[0][4]),
                   "=l"(u[0][5]), "=l"(u[0][6]), "=l"(u[0][7]), "=l"(u[1][0]), "=l"(u[1][1]),
                   "=l"(u[1][2]), "=l"(u[1][3]), "=l"(u[1][4]), "=l"(u[1][5]), "=l"(u[1][6]),
                   "=l"(u[1][7])
                 : "r"(taddr), "r"(taddr + stride)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_terms3(uint32_t taddr, uint32_t stride, uint64_t (&u)[3][8])
{
    asm volatile("{\n\t.reg .b32 a<16>, b<16>, c<16>;\n\t"
                 "tcgen05.ld.sync.aligned.32x32b.x16.b32 {a0, a1, a2, a3, a4, a5, a6, a7, a8, a9, a10, a11, a12, a13, a14, a15}, [%24];\n\t"
                 "tcgen05.ld.sync.aligned.32x32b.x16.b32 {b0, b1, b2, b3, b4, b5, b6, b7, b8, b9, b10, b11, b12, b13, b14, b15}, [%25];\n\t"
                 "tcgen05.ld.sync.aligned.32x32b.x16.b32 {c0, c1, c2, c3, c4, c5, c6, c7, c8, c9, c10, c11, c12, c13, c14, c15}, [%26];\n\t"
                 "tcgen05.wait::ld.sync.aligned;\n\t"
                 "mov.b64 %0, {a0, a1};\n\t"
                 "mov.b64 %1, {a2, a3};\n\t"
                 "mov.b64 %2, {a4, a5};\n\t"
                 "mov.b64 %3, {a6, a7};\n\t"
                 "mov.b64 %4, {a8, a9};\n\t"
                 "mov.b64 %5, {a10, a11};\n\t"
                 "mov.b64 %6, {a12, a13};\n\t"
                 "mov.b64 %7, {a14, a15};\n\t"
                 "mov.b64 %8, {b0, b1};\n\t"
                 "mov.b64 %9, {b2, b3};\n\t"
                 "mov.b64 %10, {b4, b5};\n\t"
                 "mov.b64 %11, {b6, b7};\n\t"
                 "mov.b64 %12, {b8, b9};\n\t"
                 "mov.b64 %13, {b10, b11};\n\t"
                 "mov.b64 %14, {b12, b13};\n\t"
                 "mov.b64 %15, {b14, b15};\n\t"
                 "mov.b64 %16, {c0, c1};\n\t"
                 "mov.b64 %17, {c2, c3};\n\t"
                 "mov.b64 %18, {c4, c5};\n\t"
                 "mov.b64 %19, {c6, c7};\n\t"
                 "mov.b64 %20, {c8, c9};\n\t"
                 "mov.b64 %21, {c10, c11};\n\t"
                 "mov.b64 %22, {c12, c13};\n\t"
                 "mov.b64 %23, {c14, c15};\n\t"
                 "}"
                 : "=l"(u[0][0]), "=l"(u[0][1]), "=l"(u[0][2]), "=l"(u[0][3]), "=l"(u[0][4]),
                   "=l"(u[0][5]), "=l"(u[0][6]), "=l"(u[0][7]), "=l"(u[1][0]), "=l"(u[1][1]),
                   "=l"(u[1][2]), "=l"(u[1][3]), "=l"(u[1][4]), "=l"(u[1][5]), "=l"(u[1][6]),
                   "=l"(u[1][7]), "=l"(u[2][0]), "=l"(u[2][1]), "=l"(u[2][2]), "=l"(u[2][3]),
                   "=l"(u[2][4]), "=l"(u[2][5]), "=l"(u[2][6]), "=l"(u[2][7])
                 : "r"(taddr), "r"(taddr + stride), "r"(taddr + 2 * stride)
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Bounded wait taken by every lane of a warp; the warp agrees on the outcome so that the
// .sync.aligned tcgen05 instructions after it are never reached by part of a warp.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int *flag)
{
    // the common case, a phase that has already completed: one probe and one vote
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "vote.sync.all.pred p, p, 0xffffffff;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    if (done) return true;
    const bool ok = mbar_wait_bounded(bar, parity, flag);
    return __all_sync(0xffffffffu, ok);
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 B
// apart (SBO), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (1ull << 16) | (64ull << 32) |
           (1ull << 46) | (2ull << 61);
}


// D[tmem] (+)= A[tmem] * B[smem], kind::f8f6f4 (8-bit A and B, K = 32 per instruction)
__device__ __forceinline__ void mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {"
                 "%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
                 "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::
                     "r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                 "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
                 "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
                 "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
                 "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}

} // namespace dh
