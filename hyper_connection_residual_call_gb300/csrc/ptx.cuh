// ptx.cuh -- inline-PTX helpers for sm_103a used by the hyper-connection
// kernels: mbarriers, bulk (TMA) copies, programmatic dependent launch,
// cluster barriers and distributed shared memory.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tshc {

// Device-side status values (mirrors TS_OK / TS_ERR_TIMEOUT of ts_hc.h).
constexpr unsigned kStatusTimeout = 5u;
// Upper bound on any in-kernel wait for an asynchronous copy (nanoseconds).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t arrivals)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(arrivals)
                 : "memory");
}

// Makes the initialised barrier visible to the async (TMA) proxy and the cluster.
__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// One arrival on the barrier (release at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for phase `parity` of the barrier, giving up after kWaitLimitNs.
// Returns false on timeout (the caller records it and carries on).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (global_timer_ns() - t0 > kWaitLimitNs)
            return false;
    }
}

// ---- bulk copies (TMA, non-tensor) -----------------------------------------

// Global -> this CTA's shared memory; completion counted on `bar` in bytes.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Asks L2 to fetch [src, src + bytes) from HBM; nothing is waited for or
// counted. src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Asks L2 to fetch this CTA's share of [base, base + bytes) (the grid's CTAs in
// order, pieces of at most 16 KB), issued by `lanes` threads, this one being
// `lane` of them. base 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_share_l2(const void *base, size_t bytes, int lane, int lanes)
{
    constexpr size_t kPiece = 16384;
    const size_t nb = (size_t)gridDim.x * gridDim.y, b = (size_t)blockIdx.y * gridDim.x + blockIdx.x;
    const size_t share = ((bytes + nb - 1) / nb + 15) & ~size_t(15);
    const size_t lo = min(bytes, b * share), hi = min(bytes, lo + share);
    for (size_t off = lo + (size_t)lane * kPiece; off < hi; off += (size_t)lanes * kPiece)
        bulk_prefetch_l2(static_cast<const unsigned char *>(base) + off, (uint32_t)min(kPiece, hi - off));
}

// ---- programmatic dependent launch -----------------------------------------

// Lets the next kernel in the stream start launching (its blocks then wait in
// pdl_wait() for this grid to complete). No-op without the launch attribute.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Blocks until the previous kernel in the stream has completed and its memory
// is visible. No-op when the kernel was not launched as a dependent.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---- clusters / distributed shared memory ----------------------------------

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Full cluster barrier with release/acquire ordering of shared memory. Called
// by every thread; the warp is reconverged first because the barrier is
// .aligned.
__device__ __forceinline__ void cluster_sync()
{
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void *local, uint32_t rank)
{
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_addr(local)), "r"(rank));
    return out;
}

__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// ---- number formats ----------------------------------------------------------

// The two bf16 values packed in a 32-bit word (element 0 in the low half).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// INT4 code word (element 2i in the low nibble of byte i) split by nibble:
// byte i of the low word holds element 2i, byte i of the high word 2i + 1.
__device__ __forceinline__ uint32_t int4_lo_nibbles(uint32_t codes) { return codes & 0x0F0F0F0Fu; }
__device__ __forceinline__ uint32_t int4_hi_nibbles(uint32_t codes) { return (codes >> 4) & 0x0F0F0F0Fu; }

// Byte i of a nibble word placed in the mantissa of 2^23 (one byte permute):
// the bits of the float 2^23 + q, exact for q < 2^23.
__device__ __forceinline__ uint32_t nibble_2p23_bits(uint32_t nibbles, int i)
{
    return __byte_perm(nibbles, 0x4B000000u, 0x7440u | (uint32_t)i);
}

// ---- packed fp32x2 arithmetic (two IEEE fp32 operations in one instruction) ----

__device__ __forceinline__ uint64_t f32x2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f32x2_unpack(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// d = a * b + c, lane-wise, round to nearest.
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// d = a + b, lane-wise, round to nearest.
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Elements 2i and 2i + 1 of an INT4 code word, given by its two nibble words,
// as an exact fp32 pair without an int-to-float conversion: (2^23 + q) - 2^23.
__device__ __forceinline__ uint64_t int4_pair_f32x2(uint32_t lo_nibbles, uint32_t hi_nibbles, int i)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(nibble_2p23_bits(lo_nibbles, i)), "r"(nibble_2p23_bits(hi_nibbles, i)));
    return fadd2(r, 0xCB000000CB000000ull);  // + (-2^23, -2^23)
}

}  // namespace tshc
