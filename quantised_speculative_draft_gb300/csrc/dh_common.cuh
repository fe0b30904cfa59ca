// dh_common.cuh -- device helpers shared by the draft-head kernels (sm_103a only).
//
// Inline-PTX wrappers for mbarriers, TMA (cp.async.bulk[.tensor]), warp-level mma.sync and
// the bit-pattern dequant of the 2-bit planes, plus the launch-geometry constants.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dh_internal.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "this library is written for sm_103a only"
#endif

namespace dh {

// A bounded device-side wait gives up after this long and flags DH_ERR_DEVICE_TIMEOUT.
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

// ----------------------------------------------------------------------------------------
// small utilities
// ----------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b)
{
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// OCP e4m3 (the float8_e4m3fn format) byte -> fp32, exact.  Sign, 4 exponent bits (bias 7),
// 3 mantissa bits; exponent field 0 is subnormal, m * 2^-9.  A normal value's fp32 bits are
// its exponent and mantissa fields moved up by 20 bits with the bias raised from 7 to 127.
// The NaN codes (0x7F, 0xFF) decode as +-480: callers hold finite weights only.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b)
{
    const uint32_t mag = b & 0x7Fu;
    const float v = mag >= 8u ? __uint_as_float((mag << 20) + (120u << 23))
                              : static_cast<float>(mag) * 0.001953125f; // 2^-9
    return (b & 0x80u) ? -v : v;
}

// Order-preserving map of an fp32 value onto uint32 (larger value -> larger key).
__device__ __forceinline__ uint32_t f32_order_key(float v)
{
    uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float f32_from_order_key(uint32_t k)
{
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

// ----------------------------------------------------------------------------------------
// mbarrier (shared::cta) with bounded waits
// ----------------------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream serialization may
// start while its predecessor in the stream still runs; pdl_wait() blocks until that predecessor
// has completed and its memory is visible, pdl_trigger() lets this kernel's own dependents start.
// Both are no-ops for a kernel launched the ordinary way.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One bounded-latency probe of the phase: try_wait may park the thread for a short,
// system-chosen time while the phase is incomplete (no explicit suspend-time hint: a long hint
// delayed wake-ups on the handoffs of the pipelined kernels).
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and sets *flag) if
// it has not completed within kWaitTimeoutNs of the global timer or kWaitTimeoutCycles of
// the SM clock (two independent clocks, so the bound holds even if one of them stalls); the
// caller must then stop its work.
constexpr long long kWaitTimeoutCycles = 5000000000ll;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, int *flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    // the clocks are read only every 16 suspended polls: a wait that completes soon costs no
    // timer reads
    unsigned long long t0 = 0;
    long long c0 = 0;
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15u) == 0) {
            if (i == 16) {
                t0 = globaltimer_ns();
                c0 = clock64();
            } else if (globaltimer_ns() - t0 > kWaitTimeoutNs || clock64() - c0 > kWaitTimeoutCycles) {
                break;
            }
        }
    }
    atomicExch(flag, 1);
    return false;
}

// ----------------------------------------------------------------------------------------
// TMA
// ----------------------------------------------------------------------------------------

__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(void *smem_dst, const CUtensorMap *map, int x,
                                                 int y, uint64_t *bar, uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)),
                 "l"(policy)
                 : "memory");
}

// Plain (untiled) bulk copy global -> shared: both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1], %2, [%3];" ::"r"(smem_u32(smem_dst)),
                 "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ----------------------------------------------------------------------------------------
// Bit-pattern dequant (radiance_drafthead.py, docstring bullet "Bit-pattern dequant,
// hoisted"): the 2-bit code v in bits 5-6 of a bf16 with sign 0 and exponent 127 reads as
// 1 + v/4.  Working on a 32-bit word of four packed bytes, one shift and one and-or turn
// bytes (0, 2) -- or bytes (1, 3) -- of plane P into a bf16x2 pair.
// ----------------------------------------------------------------------------------------

template <int P>
__device__ __forceinline__ uint32_t deq_pair_even(uint32_t w) // bytes 0 and 2
{
    const uint32_t t = (P < 3) ? (w << (5 - 2 * P)) : (w >> 1);
    return (t & 0x00600060u) | 0x3F803F80u;
}

template <int P>
__device__ __forceinline__ uint32_t deq_pair_odd(uint32_t w) // bytes 1 and 3
{
    return ((w >> (3 + 2 * P)) & 0x00600060u) | 0x3F803F80u;
}

// ----------------------------------------------------------------------------------------
// warp-level tensor-core MMA: D[16x8] += A[16x16] * B[16x8], bf16 in, fp32 accumulate
// ----------------------------------------------------------------------------------------

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (value, index) ordering used by every selection: larger value first, equal values ->
// lower index first.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib)
{
    return va > vb || (va == vb && ia < ib);
}

} // namespace dh
