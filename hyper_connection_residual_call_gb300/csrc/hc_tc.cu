// hc_tc.cu -- the batched (M >= 2 tokens) hyper-connection call on the
// 5th-generation tensor cores: tcgen05.mma with TMEM accumulators, operands
// staged by tensor-map TMA in the 128-byte swizzled layout.
//
// At M tokens the projections are dense contractions (families/qwen4/hc.rs
// runs them as GEMVs per token; real_forward.rs batches such GEMVs into M-row
// GEMMs inside a prefill micro-batch). Four kernels, PDL-chained:
//
//  hc_tc_prep_kernel   per (token, stream): the fused inject-add (written back
//                      to the residual), inv_rms, and normed = raw * g * inv_rms
//                      stored as bf16 hi + lo (normed = hi + lo to ~16
//                      significant bits), so that the GEMMs keep fp32-level
//                      accuracy with bf16 operands.
//  hc_tc_down_kernel   D[128 rows][N tokens] = W[rows][K chunk] * normed^T, one
//                      MMA of N = 2 * tokens per K step over the stacked hi and
//                      lo tiles (their column halves added in the epilogue);
//                      CTA (chunk, row tile, token tile) writes its fp32
//                      partial tile to part[chunk][token][row].
//  hc_tc_reduce_kernel z = sum over chunks (fixed order); act = silu(z / C)
//                      (fp32, and bf16 hi + lo for the up GEMM), gates =
//                      2 sigmoid(z / C).
//  hc_tc_up_kernel     D[C*HBt rows][N] = Wu[rows {c*H + h}][L] * (act_hi + act_lo)^T,
//                      one stacked MMA per K step as in the down kernel,
//                      epilogue: w = sigmoid(D),
//                      mixed[h] = mean_c w * normed, with the normed tile
//                      (hi + lo) staged by TMA. act keeps ~16 significant bits
//                      so that w meets the fp32 bar where the sigmoid leaves
//                      its linear region (a bf16 act moves a small w by up to
//                      2^-9 of the up pre-activation, far past 1e-3 of w).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <set>
#include <utility>

#include "hc_tc.h"
#include "ptx.cuh"
#include "umma.cuh"

namespace tshc {

namespace {

constexpr int kThreads = 512;  // down kernel: 16 warps
constexpr int kUpThreads = 512;  // up kernel: 16 warps (the epilogue and the INT4 producers are latency-bound)
constexpr int kTileRows = 128; // UMMA M
constexpr int kKBlock = 64;    // bf16 elements per 128-byte swizzled row
constexpr int kProducers = kThreads - 64;  // down kernel: warps 2-15 dequantise INT4 weight tiles
constexpr int kUpProducers = kUpThreads - 64;  // up kernel: warps 2-15

// Sigmoid from the fast exponential and division intrinsics (relative error
// ~1e-6, far inside the 1e-3 bar), for the per-element epilogues.
__device__ __forceinline__ float sigm_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

__device__ __forceinline__ void record_timeout(unsigned *status)
{
    if (status)
        atomicExch(status, kStatusTimeout);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&b);
}

__host__ __device__ constexpr uint32_t tmem_cols(int n)
{
    return n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : 256u;
}

struct TcSmem {
    uint32_t stage_bytes, a_bytes, b_bytes;
    uint32_t ring, extra, bars, total;
};

// Dequantises 8 INT4-affine codes (element e in nibble e of `codes`) with one
// scale and bias (fp16 bits) and splits them into bf16 hi and lo parts:
// w = q * s + b in fp32, hi = bf16(w), lo = bf16(w - hi).
__device__ __forceinline__ void int4x8_hilo(uint32_t codes, uint16_t sb, uint16_t bb, uint4 &hi, uint4 &lo)
{
    const float sc = __half2float(__ushort_as_half(sb)), bi = __half2float(__ushort_as_half(bb));
    const uint64_t sc2 = f32x2(sc, sc), bi2 = f32x2(bi, bi);
    const uint32_t nlo = int4_lo_nibbles(codes), nhi = int4_hi_nibbles(codes);
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        // Elements 2e and 2e+1, exact, then w = q * s + b for both in one packed FMA.
        float wa, wb;
        f32x2_unpack(ffma2(int4_pair_f32x2(nlo, nhi, e), sc2, bi2), wa, wb);
        const uint32_t hh = pack_bf16x2(wa, wb);
        h[e] = hh;
        l[e] = pack_bf16x2(wa - bf16_lo(hh), wb - bf16_hi(hh));
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}


// ---------------------------------------------------------------- prep

constexpr int kPrepThreads = 512;
constexpr int kPrepVec = 4;  // 8-element vectors per thread: H <= 8 * kPrepThreads * kPrepVec = 16384

__device__ __forceinline__ float warp_sum_f(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Grid (M, C): CTA (m, c) owns stream c of token m, one 8-element vector per
// thread and round.
__global__ void __launch_bounds__(kPrepThreads) hc_tc_prep_kernel(const TcPrepParams p)
{
    __shared__ float red_s[kPrepThreads / 32];
    const int m = blockIdx.x, c = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int nv = p.H / 8;
    const size_t base = (size_t)m * p.W + (size_t)c * p.H;                        // [M][W] outputs
    const size_t rbase = (size_t)m * p.raw_mstride + (size_t)c * p.raw_cstride;  // the residual's view
    const bool fused = p.inj_out != nullptr;
    const bool write_back = p.raw_out != nullptr;
    pdl_launch_dependents();
    uint4 gq[kPrepVec];  // g is a weight: read before the dependency wait
#pragma unroll
    for (int k = 0; k < kPrepVec; ++k) {
        const int v = tid + k * blockDim.x;
        gq[k] = v < nv ? reinterpret_cast<const uint4 *>(p.g + (size_t)c * p.H)[v] : make_uint4(0, 0, 0, 0);
    }
    pdl_wait();  // the residual, the sublayer output and the previous gates come from earlier kernels

    // Every load first (the residual is written back below).
    uint4 rv[kPrepVec], ov[kPrepVec];
#pragma unroll
    for (int k = 0; k < kPrepVec; ++k) {
        const int v = tid + k * blockDim.x;
        rv[k] = v < nv ? reinterpret_cast<const uint4 *>(p.raw + rbase)[v] : make_uint4(0, 0, 0, 0);
        ov[k] = (fused && v < nv) ? reinterpret_cast<const uint4 *>(p.inj_out + (size_t)m * p.H)[v]
                                  : make_uint4(0, 0, 0, 0);
    }
    const float gate = fused ? p.inj_gate[(size_t)m * p.inj_stride + c] : 0.f;
    float q = 0.f;
#pragma unroll
    for (int k = 0; k < kPrepVec; ++k) {
        const int v = tid + k * blockDim.x;
        if (v >= nv)
            continue;
        uint32_t w[4] = {rv[k].x, rv[k].y, rv[k].z, rv[k].w};
        if (fused) {  // raw + out * gate, rounded as the inject-add kernel rounds
            const uint32_t o[4] = {ov[k].x, ov[k].y, ov[k].z, ov[k].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                w[e] = pack_bf16x2(fmaf(bf16_lo(o[e]), gate, bf16_lo(w[e])), fmaf(bf16_hi(o[e]), gate, bf16_hi(w[e])));
            rv[k] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (write_back)
            reinterpret_cast<uint4 *>(p.raw_out + base)[v] = rv[k];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = bf16_lo(w[e]), b = bf16_hi(w[e]);
            q = fmaf(a, a, q);
            q = fmaf(b, b, q);
        }
    }
    // The stream's sum of squares: warps, then the warp totals in warp order.
    q = warp_sum_f(q);
    if (lane == 0)
        red_s[warp] = q;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < nwarps; ++w)
        t += red_s[w];
    const float inv = rsqrtf(fmaf(t, p.inv_H, p.eps));
    if (tid == 0)
        p.inv_rms[(size_t)m * p.C + c] = inv;
#pragma unroll
    for (int k = 0; k < kPrepVec; ++k) {
        const int v = tid + k * blockDim.x;
        if (v >= nv)
            continue;
        const uint32_t w[4] = {rv[k].x, rv[k].y, rv[k].z, rv[k].w};
        const uint32_t gw[4] = {gq[k].x, gq[k].y, gq[k].z, gq[k].w};
        uint32_t h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float xa = bf16_lo(w[e]) * bf16_lo(gw[e]) * inv, xb = bf16_hi(w[e]) * bf16_hi(gw[e]) * inv;
            const uint32_t hh = pack_bf16x2(xa, xb);
            h[e] = hh;
            l[e] = pack_bf16x2(xa - bf16_lo(hh), xb - bf16_hi(hh));
        }
        reinterpret_cast<uint4 *>(p.x_hi + base)[v] = make_uint4(h[0], h[1], h[2], h[3]);
        reinterpret_cast<uint4 *>(p.x_lo + base)[v] = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

// ---------------------------------------------------------------- down

// Shared memory of the down kernel: a ring of stages [A_hi | A_lo (INT4
// weights only) | B_hi | B_lo], then the barriers.
__host__ __device__ inline TcSmem down_tc_layout(int NT, int ns, int wt)
{
    TcSmem s;
    s.a_bytes = kTileRows * 128;
    s.b_bytes = NT * 128;
    s.stage_bytes = s.a_bytes * (1 + wt) + 2 * s.b_bytes;
    s.ring = 0;
    s.extra = s.ring + ns * s.stage_bytes;
    s.bars = s.extra;
    s.total = s.bars + 8 * (3 * ns + 1) + 16;
    return s;
}

// Grid (nchunk, row tiles, token tiles). Warp 0 lane 0 streams the weight
// tiles (before the dependency wait) and the normed hi/lo tiles by TMA; with
// INT4 weights, warps 2-15 dequantise the weight tiles instead. Warp 1 lane 0
// issues the MMAs. All eight warps then move the fp32 tile from TMEM to
// part[chunk][row][token].
template <int WT>
__global__ void __launch_bounds__(kThreads, 1)
hc_tc_down_kernel(const TcDownParams p, const __grid_constant__ CUtensorMap map_d,
                  const __grid_constant__ CUtensorMap map_i, const __grid_constant__ CUtensorMap map_xhi,
                  const __grid_constant__ CUtensorMap map_xlo)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int NT = p.NT, NS = p.n_stages;
    const TcSmem lay = down_tc_layout(NT, NS, WT);
    const uint32_t b_off = lay.a_bytes * (1 + WT);  // B_hi within a stage
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bars);  // TMA bytes of a stage
    uint64_t *fullp = full + NS;                                      // INT4: producers' A tiles written
    uint64_t *empty = fullp + NS;
    uint64_t *done = empty + NS;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kc = blockIdx.x, rt = blockIdx.y, tile = blockIdx.z;
    const int r0 = rt * kTileRows;
    const int KBT = p.W / kKBlock, kb0 = kc * p.KBc;
    const int KB = min(p.KBc, KBT - kb0);
    const uint32_t ncols = tmem_cols(2 * NT);  // columns [0, NT): W * B_hi, [NT, 2 NT): W * B_lo

    // Boxes of 32 rows making up this row tile: from W_down, from
    // block_inject_weight (rows beyond its C are zero-filled), or skipped.
    int nbox = 0;
    for (int b = 0; b < 4; ++b) {
        const int gr = r0 + 32 * b;
        if (gr + 32 <= p.L || (gr == p.L && p.has_inject)) ++nbox;
    }

    pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&fullp[s], kProducers / 32);  // one arrival per producer warp
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        mbar_fence_init();
    }
    if (warp == 0) {
        __syncwarp();
        tmem_alloc(tslot, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool timed_out = false;

    if (warp == 0 && lane == 0) {
        const uint32_t a_tx = WT == 0 ? (uint32_t)nbox * 32 * 128 : 0u;
        const uint32_t b_tx = 2u * NT * 128;
        auto load_a = [&](int kb, int s) {
            uint8_t *a = smem + lay.ring + s * lay.stage_bytes;
            const int col = (kb0 + kb) * kKBlock;
            for (int b = 0; b < 4; ++b) {
                const int gr = r0 + 32 * b;
                if (gr + 32 <= p.L)
                    tma_load_2d(a + b * 32 * 128, &map_d, col, gr, &full[s]);
                else if (gr == p.L && p.has_inject)
                    tma_load_2d(a + b * 32 * 128, &map_i, col, 0, &full[s]);
            }
        };
        auto load_b = [&](int kb, int s) {
            uint8_t *bh = smem + lay.ring + s * lay.stage_bytes + b_off;
            const int col = (kb0 + kb) * kKBlock;
            tma_load_2d(bh, &map_xhi, col, tile * NT, &full[s]);
            tma_load_2d(bh + lay.b_bytes, &map_xlo, col, tile * NT, &full[s]);
        };
        if (WT == 0) {
            tma_prefetch_map(&map_d);
            if (p.has_inject) tma_prefetch_map(&map_i);
        }
        // The stages before the ring wraps: weights first (independent of the
        // previous kernels), then the activations once they exist.
        const int npre = KB < NS ? KB : NS;
        for (int kb = 0; kb < npre; ++kb) {
            mbar_arrive_expect_tx(&full[kb], a_tx + b_tx);
            if (WT == 0)
                load_a(kb, kb);
        }
        pdl_wait();  // normed comes from the prep kernel
        for (int kb = 0; kb < npre; ++kb)
            load_b(kb, kb);
        for (int kb = npre; kb < KB; ++kb) {
            const int s = kb % NS, u = kb / NS;
            if (!mbar_wait_bounded(&empty[s], (u - 1) & 1)) timed_out = true;
            mbar_arrive_expect_tx(&full[s], a_tx + b_tx);
            if (WT == 0)
                load_a(kb, s);
            load_b(kb, s);
        }
    } else if (WT == 1 && warp >= 2) {
        // INT4 weights: warps 2-15 dequantise the A tiles (weights only, so no
        // dependency wait). Thread t handles the 16-byte chunks t + kProducers j
        // of the 128 x 64 tile: row / 8, chunk t % 8 (8 codes, one scale and bias).
        const int t = tid - 64;
        const int ck = t & 7;
        constexpr int kItems = (kTileRows * 8 + kProducers - 1) / kProducers;
        const uint8_t *wq[kItems];
        const uint16_t *wsc[kItems];
        const uint16_t *wbi[kItems];
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            const int rr = (t + kProducers * j) >> 3, gr = r0 + rr;
            // Fields picked by value: taking a parameter's address would move
            // the parameters to local memory.
            const bool isd = gr < p.L, isi = !isd && p.has_inject && gr < p.L + p.C;
            const int row = isd ? gr : gr - p.L;
            const size_t srow = (size_t)row * (p.W >> p.dw.gshift);  // inject has down's group
            wq[j] = ((isd || isi) && rr < kTileRows)
                        ? static_cast<const uint8_t *>(isd ? p.dw.data : p.iw.data) + (size_t)row * (p.W / 2)
                        : nullptr;
            wsc[j] = wq[j] ? (isd ? p.dw.scales : p.iw.scales) + srow : nullptr;
            wbi[j] = wq[j] ? (isd ? p.dw.biases : p.iw.biases) + srow : nullptr;
        }
        uint32_t qn[kItems];
        uint16_t sn[kItems], bn[kItems];
        auto fetch = [&](int kb) {
            const int col = (kb0 + kb) * kKBlock + 8 * ck;
#pragma unroll
            for (int j = 0; j < kItems; ++j) {
                qn[j] = wq[j] ? *reinterpret_cast<const uint32_t *>(wq[j] + col / 2) : 0u;
                sn[j] = wq[j] ? wsc[j][col >> p.dw.gshift] : (uint16_t)0;
                bn[j] = wq[j] ? wbi[j][col >> p.dw.gshift] : (uint16_t)0;
            }
        };
        fetch(0);
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % NS, u = kb / NS;
            uint32_t qc[kItems];
            uint16_t sc[kItems], bc[kItems];
#pragma unroll
            for (int j = 0; j < kItems; ++j) {
                qc[j] = qn[j];
                sc[j] = sn[j];
                bc[j] = bn[j];
            }
            if (kb + 1 < KB)
                fetch(kb + 1);
            if (u > 0 && !mbar_wait_bounded(&empty[s], (u - 1) & 1)) timed_out = true;
            uint8_t *ahi = smem + lay.ring + s * lay.stage_bytes;
            uint8_t *alo = ahi + lay.a_bytes;
#pragma unroll
            for (int j = 0; j < kItems; ++j) {
                const int rr = (t + kProducers * j) >> 3;
                if (rr >= kTileRows)
                    continue;
                uint4 hi = make_uint4(0, 0, 0, 0), lo = make_uint4(0, 0, 0, 0);
                if (wq[j])
                    int4x8_hilo(qc[j], sc[j], bc[j], hi, lo);
                *reinterpret_cast<uint4 *>(ahi + sw128_offset(rr, 8 * ck)) = hi;
                *reinterpret_cast<uint4 *>(alo + sw128_offset(rr, 8 * ck)) = lo;
            }
            // Each thread's tile writes become visible to the tensor cores; the
            // warp then arrives once.
            fence_async_shared();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&fullp[s]);
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer. B_lo follows B_hi in the stage, a whole number of 8-row
        // swizzle atoms later, so [B_hi; B_lo] is one K-major operand of 2 NT rows:
        // one MMA of N = 2 NT per K step instead of one per part (an MMA
        // instruction costs about the same from N = 16 to N = 128).
        const uint32_t idesc2 = umma_idesc_bf16(kTileRows, 2 * NT);
        const uint32_t idesc1 = umma_idesc_bf16(kTileRows, NT);
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % NS, u = kb / NS;
            if (!mbar_wait_bounded(&full[s], u & 1)) timed_out = true;
            if (WT == 1 && !mbar_wait_bounded(&fullp[s], u & 1)) timed_out = true;
            tc_fence_after();
            const uint32_t a = smem_addr(smem + lay.ring + s * lay.stage_bytes);
            const uint32_t al = a + lay.a_bytes;  // A_lo (INT4 weights)
            const uint32_t bh = a + b_off;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                umma_bf16(tmem, umma_desc_sw128(a + 32 * k), umma_desc_sw128(bh + 32 * k), idesc2, (kb | k) != 0);
                if (WT == 1)  // the weight's lo part against the activation's hi part (columns [0, NT))
                    umma_bf16(tmem, umma_desc_sw128(al + 32 * k), umma_desc_sw128(bh + 32 * k), idesc1, 1);
            }
            umma_commit(&empty[s]);
        }
        umma_commit(done);
    }

    // Epilogue on all 16 warps: warp w reads TMEM lanes 32*(w%4).. (the tile's
    // rows) for the 16-column chunks 16*(w/4) + 64k, the hi and the lo parts --
    // all of them before the one wait -- adds the two, and stores them to
    // part[chunk][token][row]: the 32 lanes of a store write 32 consecutive rows
    // of one token (coalesced). The barrier reconverges the single-thread roles.
    __syncthreads();
    if (!mbar_wait_bounded(done, 0)) timed_out = true;
    __syncwarp();  // the TMEM loads below are .aligned
    tc_fence_after();
    {
        constexpr int kParts = kThreads / 128;      // warps sharing a TMEM lane quadrant
        constexpr int kChunks = 128 / (16 * kParts);  // NT <= 128: chunks per warp
        const int quad = warp & 3, part = warp >> 2;
        const int gr = r0 + quad * 32 + lane;
        const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16);
        uint32_t v[kChunks][16], w[kChunks][16];
#pragma unroll
        for (int k = 0; k < kChunks; ++k)
            if (16 * part + 16 * kParts * k < NT) {  // warp-uniform
                tmem_ld16_async(tbase + 16 * part + 16 * kParts * k, v[k]);
                tmem_ld16_async(tbase + NT + 16 * part + 16 * kParts * k, w[k]);
            }
#pragma unroll
        for (int k = 0; k < kChunks; ++k) {
            tmem_wait_ld(v[k]);
            tmem_wait_ld(w[k]);
        }
        if (gr < p.R) {
            float *dst = p.part + ((size_t)kc * p.Mp + (size_t)tile * NT) * p.R + gr;
#pragma unroll
            for (int k = 0; k < kChunks; ++k) {
                const int c0 = 16 * part + 16 * kParts * k;
                if (c0 < NT) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        dst[(size_t)(c0 + j) * p.R] = __uint_as_float(v[k][j]) + __uint_as_float(w[k][j]);
                }
            }
        }
    }
    if (timed_out) record_timeout(p.status);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        tmem_dealloc(tmem, ncols);
}

// ---------------------------------------------------------------- reduce

// One thread per (token, row): element i = m * R + r of every chunk's partial
// tile, so the loads of a warp are contiguous; the chunks are summed in order,
// every load of a thread in flight at once. The host sizes the grid to about
// one CTA per SM (and reserves shared memory to keep it so), on the SMs that
// the up kernel's CTAs leave free when those all fit beside it: the up CTAs
// then start, set up and stream their weights while this kernel runs. Before
// the dependency wait each CTA asks L2 for its share of the up kernel's
// weights. It triggers the up kernel only after that wait, so that the up
// kernel may read the prep kernel's normed tiles before its own.
constexpr int kReduceBatch = 40;

// A load through L2 that the compiler keeps in program order with the other
// loads of a batch (volatile), so that the batch is in flight at once.
__device__ __forceinline__ float ld_cg_f32(const float *ptr)
{
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
    return v;
}

__global__ void __launch_bounds__(1024) hc_tc_reduce_kernel(const TcReduceParams p)
{
    if (threadIdx.x < 32) {
        constexpr size_t kPiece = 16384;
        const size_t nb = gridDim.x, b = blockIdx.x;
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const size_t total = p.l2_next_bytes[i];
            const size_t share = ((total + nb - 1) / nb + 15) & ~size_t(15);
            const size_t lo = min(total, b * share), hi = min(total, lo + share);
            for (size_t off = lo + (size_t)threadIdx.x * kPiece; off < hi; off += 32 * kPiece)
                bulk_prefetch_l2(static_cast<const unsigned char *>(p.l2_next[i]) + off,
                                 (uint32_t)min(kPiece, hi - off));
        }
    }
    pdl_wait();
    pdl_launch_dependents();  // after the wait: the up kernel may read what came before this kernel
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long)p.M * p.R)
        return;
    const float *src = p.part + i;
    const size_t cstride = (size_t)p.Mp * p.R;
    float z = 0.f;
    for (int kc = 0; kc < p.nchunk; kc += kReduceBatch) {
        float v[kReduceBatch];
        if (kc + kReduceBatch <= p.nchunk) {  // a whole batch: every load issued before the first add
#pragma unroll
            for (int j = 0; j < kReduceBatch; ++j)
                v[j] = ld_cg_f32(src + (size_t)(kc + j) * cstride);
        } else {
#pragma unroll
            for (int j = 0; j < kReduceBatch; ++j)
                v[j] = kc + j < p.nchunk ? ld_cg_f32(src + (size_t)(kc + j) * cstride) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < kReduceBatch; ++j)
            z += v[j];
    }
    const int m = (int)(i / p.R), r = (int)(i % p.R);
    const float zc = z * p.inv_C;
    if (r < p.L) {
        const float a = zc * sigm_fast(zc);
        const __nv_bfloat16 ah = __float2bfloat16_rn(a);
        p.act[(size_t)m * p.L + r] = a;
        p.act_hi[(size_t)m * p.L + r] = __bfloat16_as_ushort(ah);
        p.act_lo[(size_t)m * p.L + r] = __bfloat16_as_ushort(__float2bfloat16_rn(a - __bfloat162float(ah)));
    } else {
        p.gate[(size_t)m * p.gate_stride + (r - p.L)] = 2.0f * sigm_fast(zc);
    }
}

// ---------------------------------------------------------------- up

// Up kernel shared memory: a ring of stages [A_hi | A_lo (INT4 weights only) |
// B_hi | B_lo (act)], then the normed hi and lo tiles [C][NT][HBt] bf16, then
// the barriers.
__host__ __device__ inline uint32_t up_tc_tile_bytes(int NT, int C, int HBt)
{
    return ((C * NT * HBt * 2 + 1023) / 1024) * 1024;
}

__host__ __device__ inline TcSmem up_tc_layout(int NT, int ns, int C, int HBt, int wt)
{
    TcSmem s;
    s.a_bytes = kTileRows * 128;
    s.b_bytes = NT * 128;
    s.stage_bytes = s.a_bytes * (1 + wt) + 2 * s.b_bytes;
    s.ring = 0;
    s.extra = s.ring + ns * s.stage_bytes;
    s.bars = s.extra + 2 * up_tc_tile_bytes(NT, C, HBt);
    s.total = s.bars + 8 * (3 * ns + 2) + 16;
    return s;
}

template <int WT>
__global__ void __launch_bounds__(kUpThreads, 1)
hc_tc_up_kernel(const TcUpParams p, const __grid_constant__ CUtensorMap map_u,
                const __grid_constant__ CUtensorMap map_act, const __grid_constant__ CUtensorMap map_alo,
                const __grid_constant__ CUtensorMap map_nhi, const __grid_constant__ CUtensorMap map_nlo)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int NT = p.NT, NS = p.n_stages, C = p.C, HBt = p.HBt;
    const TcSmem lay = up_tc_layout(NT, NS, C, HBt, WT);
    const uint32_t b_off = lay.a_bytes * (1 + WT);  // B_hi (act), then B_lo, within a stage
    const uint16_t *nhi_s = reinterpret_cast<const uint16_t *>(smem + lay.extra);  // [C][NT][HBt]
    const uint16_t *nlo_s = nhi_s + up_tc_tile_bytes(NT, C, HBt) / 2;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bars);
    uint64_t *empty = full + NS;
    uint64_t *fullp = empty + NS;  // INT4: the producers' A tiles of a stage are written
    uint64_t *done = fullp + NS;
    uint64_t *nbar = done + 1;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(nbar + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h0 = blockIdx.x * HBt;
    const int tile = blockIdx.y;
    const int KB = p.L / kKBlock;
    const uint32_t ncols = tmem_cols(2 * NT);  // columns [0, NT): Wu * act_hi, [NT, 2 NT): Wu * act_lo

    pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&fullp[s], kUpProducers / 32);  // one arrival per producer warp
        }
        mbar_init(done, 1);
        mbar_init(nbar, 1);
        mbar_fence_init();
    }
    if (warp == 0) {
        __syncwarp();
        tmem_alloc(tslot, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool timed_out = false;

    if (warp == 0 && lane == 0) {
        // Weights first (bf16: TMA; independent of the previous kernels) ...
        const int npre = WT == 0 ? (KB < NS ? KB : NS) : 0;
        if (WT == 0)
            tma_prefetch_map(&map_u);
        for (int kb = 0; kb < npre; ++kb) {
            uint8_t *a = smem + lay.ring + kb * lay.stage_bytes;
            mbar_arrive_expect_tx(&full[kb], C * HBt * 128 + 2 * NT * 128);
            for (int cc = 0; cc < C; ++cc)
                tma_load_2d(a + cc * HBt * 128, &map_u, kb * kKBlock, cc * p.H + h0, &full[kb]);
        }
        // The normed tiles come from the prep kernel, two kernels back: the reduce
        // kernel triggers only after its own wait, so they are complete here.
        mbar_arrive_expect_tx(nbar, 2 * C * NT * HBt * 2);
        for (int cc = 0; cc < C; ++cc) {
            tma_load_2d(const_cast<uint16_t *>(nhi_s) + cc * NT * HBt, &map_nhi, cc * p.H + h0, tile * NT, nbar);
            tma_load_2d(const_cast<uint16_t *>(nlo_s) + cc * NT * HBt, &map_nlo, cc * p.H + h0, tile * NT, nbar);
        }
        pdl_wait();  // ... then the activations
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % NS, u = kb / NS;
            uint8_t *a = smem + lay.ring + s * lay.stage_bytes;
            if (WT == 0 && kb >= npre) {
                if (!mbar_wait_bounded(&empty[s], (u - 1) & 1)) timed_out = true;
                mbar_arrive_expect_tx(&full[s], C * HBt * 128 + 2 * NT * 128);
                for (int cc = 0; cc < C; ++cc)
                    tma_load_2d(a + cc * HBt * 128, &map_u, kb * kKBlock, cc * p.H + h0, &full[s]);
            } else if (WT == 1) {
                if (u > 0 && !mbar_wait_bounded(&empty[s], (u - 1) & 1)) timed_out = true;
                mbar_arrive_expect_tx(&full[s], 2 * NT * 128);
            }
            tma_load_2d(a + b_off, &map_act, kb * kKBlock, tile * NT, &full[s]);
            tma_load_2d(a + b_off + lay.b_bytes, &map_alo, kb * kKBlock, tile * NT, &full[s]);
        }
    } else if (WT == 1 && warp >= 2) {
        // INT4 weights: warps 2-15 dequantise the A tiles (rows (stream, h) of
        // this CTA, 64 columns per stage) to bf16 hi + lo. Thread t handles the
        // 16-byte chunks t + kUpProducers j: row / 8, chunk t % 8. Weights only:
        // no dependency wait.
        const int t = tid - 64;
        const int ck = t & 7;
        constexpr int kItems = (kTileRows * 8 + kUpProducers - 1) / kUpProducers;
        const uint8_t *wq[kItems];
        const uint16_t *wsc[kItems];
        const uint16_t *wbi[kItems];
        const int ngr = p.L >> p.uw.gshift;
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            const int rr = (t + kUpProducers * j) >> 3;
            const int cc = rr / HBt, hl = rr % HBt;
            const bool ok = rr < kTileRows && cc < C && h0 + hl < p.H;
            const size_t row = (size_t)cc * p.H + h0 + hl;
            wq[j] = ok ? static_cast<const uint8_t *>(p.uw.data) + row * (p.L / 2) : nullptr;
            wsc[j] = ok ? p.uw.scales + row * ngr : nullptr;
            wbi[j] = ok ? p.uw.biases + row * ngr : nullptr;
        }
        // The next K block's codes, scales and biases are loaded while the
        // current one is converted.
        uint32_t qn[kItems];
        uint16_t sn[kItems], bn[kItems];
        auto fetch = [&](int kb) {
            const int col = kb * kKBlock + 8 * ck;
#pragma unroll
            for (int j = 0; j < kItems; ++j) {
                qn[j] = wq[j] ? *reinterpret_cast<const uint32_t *>(wq[j] + col / 2) : 0u;
                sn[j] = wq[j] ? wsc[j][col >> p.uw.gshift] : (uint16_t)0;
                bn[j] = wq[j] ? wbi[j][col >> p.uw.gshift] : (uint16_t)0;
            }
        };
        fetch(0);
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % NS, u = kb / NS;
            uint32_t q[kItems];
            uint16_t sc[kItems], bi[kItems];
#pragma unroll
            for (int j = 0; j < kItems; ++j) {
                q[j] = qn[j];
                sc[j] = sn[j];
                bi[j] = bn[j];
            }
            if (kb + 1 < KB)
                fetch(kb + 1);
            if (u > 0 && !mbar_wait_bounded(&empty[s], (u - 1) & 1)) timed_out = true;
            uint8_t *ahi = smem + lay.ring + s * lay.stage_bytes;
            uint8_t *alo = ahi + lay.a_bytes;
#pragma unroll
            for (int j = 0; j < kItems; ++j) {
                const int rr = (t + kUpProducers * j) >> 3;
                if (rr >= kTileRows)
                    continue;
                uint4 hi = make_uint4(0, 0, 0, 0), lo = make_uint4(0, 0, 0, 0);
                if (wq[j])
                    int4x8_hilo(q[j], sc[j], bi[j], hi, lo);
                *reinterpret_cast<uint4 *>(ahi + sw128_offset(rr, 8 * ck)) = hi;
                *reinterpret_cast<uint4 *>(alo + sw128_offset(rr, 8 * ck)) = lo;
            }
            // Each thread's tile writes become visible to the tensor cores; the
            // warp then arrives once.
            fence_async_shared();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&fullp[s]);
        }
    }

    if (warp == 1 && lane == 0) {
        // One MMA of N = 2 NT per K step over [act_hi; act_lo] (act_lo follows
        // act_hi in the stage, a whole number of swizzle atoms later).
        const uint32_t idesc2 = umma_idesc_bf16(kTileRows, 2 * NT);
        const uint32_t idesc1 = umma_idesc_bf16(kTileRows, NT);
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % NS, u = kb / NS;
            if (!mbar_wait_bounded(&full[s], u & 1)) timed_out = true;
            if (WT == 1 && !mbar_wait_bounded(&fullp[s], u & 1)) timed_out = true;
            tc_fence_after();
            const uint32_t a = smem_addr(smem + lay.ring + s * lay.stage_bytes);
            const uint32_t al = a + lay.a_bytes;  // A_lo (INT4 weights)
            const uint32_t b = a + b_off;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                umma_bf16(tmem, umma_desc_sw128(a + 32 * k), umma_desc_sw128(b + 32 * k), idesc2, (kb | k) != 0);
                if (WT == 1)  // the weight's lo part against act's hi part (columns [0, NT))
                    umma_bf16(tmem, umma_desc_sw128(al + 32 * k), umma_desc_sw128(b + 32 * k), idesc1, 1);
            }
            umma_commit(&empty[s]);
        }
        umma_commit(done);
    }
    __syncthreads();  // reconverges the single-thread roles

    // Epilogue on all 16 warps: warp w reads TMEM lanes 32*(w%4).. (rows = (stream,
    // h) pairs) for the 16-column chunks 16*(w/4) + 64k.
    float *mix_s = reinterpret_cast<float *>(smem + lay.ring);  // [C][NT][HBt], over the ring
    {
        if (!mbar_wait_bounded(done, 0)) timed_out = true;
        if (!mbar_wait_bounded(nbar, 0)) timed_out = true;
        __syncwarp();  // the TMEM loads below are .aligned
        tc_fence_after();
        const int quad = warp & 3, part = warp >> 2;
        constexpr int kStride = 16 * (kUpThreads / 128);  // columns between a warp's chunks
        const int row = quad * 32 + lane;
        const int cc = row / HBt, hl = row % HBt;
        const bool live = cc < C && h0 + hl < p.H;
        // The warp's 16-column chunks: chunk k+1 is loaded from TMEM while chunk
        // k is processed (two register buffers). A chunk's shared-memory loads
        // are all issued before its stores.
        auto process = [&](int c0, const uint32_t (&vr)[16]) {
            if (!live)
                return;
            float x[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int o = (cc * NT + c0 + j) * HBt + hl;
                x[j] = __bfloat162float(__ushort_as_bfloat16(nhi_s[o])) + __bfloat162float(__ushort_as_bfloat16(nlo_s[o]));
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float w = sigm_fast(__uint_as_float(vr[j]));
                mix_s[(cc * NT + c0 + j) * HBt + hl] = w * x[j];
                const int m = tile * NT + c0 + j;
                if (p.w_out && m < p.M)  // debug output of w (uniform branch)
                    p.w_out[(size_t)m * p.W + (size_t)cc * p.H + h0 + hl] = w;
            }
        };
        const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16);
        // NT <= 128 = 2 kStride: at most two chunks per warp; the hi and lo
        // columns of both are loaded before the one wait, then added.
        static_assert(2 * kStride >= 128, "two chunks per warp cover NT");
        uint32_t va[16], vb[16], wa[16], wb[16];
        const int c0 = 16 * part;
        if (c0 < NT) {  // warp-uniform
            tmem_ld16_async(tbase + c0, va);
            tmem_ld16_async(tbase + NT + c0, wa);
        }
        if (c0 + kStride < NT) {
            tmem_ld16_async(tbase + c0 + kStride, vb);
            tmem_ld16_async(tbase + NT + c0 + kStride, wb);
        }
        tmem_wait_ld(va);
        tmem_wait_ld(wa);
        tmem_wait_ld(vb);
        tmem_wait_ld(wb);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            va[j] = __float_as_uint(__uint_as_float(va[j]) + __uint_as_float(wa[j]));
            vb[j] = __float_as_uint(__uint_as_float(vb[j]) + __uint_as_float(wb[j]));
        }
        if (c0 < NT)
            process(c0, va);
        if (c0 + kStride < NT)
            process(c0 + kStride, vb);
    }
    tc_fence_before();
    __syncthreads();
    // Mean over the streams, 8 consecutive h of one token per item (stream order).
    for (int i = tid; i < NT * (HBt / 8); i += kUpThreads) {
        const int n = i / (HBt / 8), hv = (i % (HBt / 8)) * 8;
        const int m = tile * NT + n, h = h0 + hv;
        if (m < p.M && h + 8 <= p.H) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int cc = 0; cc < C; ++cc) {
                const float4 a = *reinterpret_cast<const float4 *>(mix_s + (cc * NT + n) * HBt + hv);
                const float4 b = *reinterpret_cast<const float4 *>(mix_s + (cc * NT + n) * HBt + hv + 4);
                acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
                acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
            }
            *reinterpret_cast<uint4 *>(p.mixed + (size_t)m * p.H + h) =
                make_uint4(pack_bf16x2(acc[0] * p.inv_C, acc[1] * p.inv_C), pack_bf16x2(acc[2] * p.inv_C, acc[3] * p.inv_C),
                           pack_bf16x2(acc[4] * p.inv_C, acc[5] * p.inv_C), pack_bf16x2(acc[6] * p.inv_C, acc[7] * p.inv_C));
        }
    }
    if (timed_out) record_timeout(p.status);
    __syncwarp();
    tc_fence_after();
    if (warp == 0)
        tmem_dealloc(tmem, ncols);
}

// ---------------------------------------------------------------- lm_head

// logits[m][v] = sum_h W[v][h] * mixed[m][h] for up to 16 tokens (families/qwen4/
// mod.rs, decoder pseudocode, exit lines: lm_head on the mixer's output, no
// softcap, no further norm). A plain bf16 GEMM: both operands are exact in bf16,
// so one MMA per K step, fp32 accumulation in TMEM. Persistent grid: CTA b takes
// the 128-row vocabulary tiles b, b + grid, ... (the tiles of w, then those of
// the optional second weight w2 against the same tokens). The tiles stream
// through one ring of stages of four K blocks: one 3-D TMA box of the weights
// (128 rows x 4 K blocks, so that each row yields 512 contiguous bytes per
// request instead of 128; it lands as four ordinary 128-row K-block tiles) and
// four 16-row token boxes (absent tokens and the ragged ends zero-filled by
// TMA). The first stages' weights are requested before the dependency wait.
// A tile's K range is accumulated in segments of at most kLmSegStages stages (64
// MMAs), alternating between two TMEM accumulators of 16 columns; the epilogue
// adds a tile's segments in fp32, in order, while the next segment accumulates. Roles: warp 0 lane 0 TMA, warp 1 lane 0 MMA, warps 2-5 the epilogue
// (TMEM lane quadrant warp % 4: 32 vocabulary rows, 16 tokens), whose stores
// of one token are 32 consecutive logits.
constexpr int kLmTcThreads = 192;
constexpr int kLmTcNT = kLmHeadMaxTokens;  // one 16-token tile, MMA N = 16
constexpr int kLmTcStages = 3;
// Stages one TMEM accumulation takes at most (64 MMAs): longer sums in one
// accumulator drift past the fp32 bar at H = 16384 (1024 MMAs).
constexpr int kLmSegStages = 4;
constexpr int kLmKbs = 4;                        // K blocks per stage (one 3-D weight box)
constexpr uint32_t kLmTcA = kLmKbs * kTileRows * 128;  // weight box: KBS K-block tiles of 128 rows x 128 bytes
constexpr uint32_t kLmTcB = kLmKbs * kLmTcNT * 128;    // token boxes: KBS x 16 rows x 128 bytes
constexpr uint32_t kLmTcStage = kLmTcA + kLmTcB;
constexpr uint32_t kLmTcBars = kLmTcStages * kLmTcStage;
constexpr size_t kLmTcSmem = kLmTcBars + 8 * (2 * kLmTcStages + 4) + 16 + 1024;

__global__ void __launch_bounds__(kLmTcThreads, 1)
hc_lm_head_tc_kernel(const LmHeadParams p, const __grid_constant__ CUtensorMap map_w,
                     const __grid_constant__ CUtensorMap map_w2, const __grid_constant__ CUtensorMap map_x)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kLmTcBars);
    uint64_t *empty = full + kLmTcStages;
    uint64_t *tfull = empty + kLmTcStages;  // [2] an accumulator's tile is complete
    uint64_t *tempty = tfull + 2;           // [2] the epilogue has read it
    uint32_t *tslot = reinterpret_cast<uint32_t *>(tempty + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nt1 = (p.V + kTileRows - 1) / kTileRows;  // tiles of w; those of w2 follow
    const int ntiles = nt1 + (p.V2 + kTileRows - 1) / kTileRows;
    const int KB = (p.H + kKBlock * kLmKbs - 1) / (kKBlock * kLmKbs);  // stages per tile
    const int my_tiles = (int)blockIdx.x < ntiles ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int nsteps = my_tiles * KB;

    pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < kLmTcStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);  // one arrival per epilogue warp
        }
        mbar_fence_init();
    }
    if (warp == 0) {
        __syncwarp();
        tmem_alloc(tslot, 2 * kLmTcNT);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool timed_out = false;

    if (warp == 0 && lane == 0) {
        // Step g: K block g % KB of the CTA's tile g / KB, in ring stage g % stages.
        auto load_w = [&](int g) {
            const int t = (int)blockIdx.x + (g / KB) * (int)gridDim.x;
            const bool first = t < nt1;
            tma_load_3d(smem + (g % kLmTcStages) * kLmTcStage, first ? &map_w : &map_w2, 0,
                        (first ? t : t - nt1) * kTileRows, (g % KB) * kLmKbs, &full[g % kLmTcStages]);
        };
        auto load_x = [&](int g) {
            for (int q = 0; q < kLmKbs; ++q)
                tma_load_2d(smem + (g % kLmTcStages) * kLmTcStage + kLmTcA + q * kLmTcNT * 128, &map_x,
                            ((g % KB) * kLmKbs + q) * kKBlock, 0, &full[g % kLmTcStages]);
        };
        tma_prefetch_map(&map_w);
        const int npre = nsteps < kLmTcStages ? nsteps : kLmTcStages;
        for (int g = 0; g < npre; ++g) {  // weights: independent of the kernels before
            mbar_arrive_expect_tx(&full[g], kLmTcStage);
            load_w(g);
        }
        pdl_wait();  // the tokens come from the kernel before
        for (int g = 0; g < npre; ++g)
            load_x(g);
        for (int g = npre; g < nsteps; ++g) {
            const int s = g % kLmTcStages, u = g / kLmTcStages;
            if (!mbar_wait_bounded(&empty[s], (u - 1) & 1)) timed_out = true;
            mbar_arrive_expect_tx(&full[s], kLmTcStage);
            load_w(g);
            load_x(g);
        }
    } else if (warp == 1 && lane == 0) {
        // A tile's K range in segments of at most kLmSegStages stages, each accumulated
        // in one of the two TMEM accumulators (alternating per segment) and added up
        // by the epilogue in fp32, in order.
        const uint32_t idesc = umma_idesc_bf16(kTileRows, kLmTcNT);
        int g = 0, acc = 0;  // acc: segments issued so far; accumulator acc & 1
        for (int j = 0; j < my_tiles; ++j) {
            for (int k0 = 0; k0 < KB; k0 += kLmSegStages, ++acc) {
                const int b = acc & 1;
                // The accumulator's previous segment (acc - 2) must have been read out.
                if (acc >= 2 && !mbar_wait_bounded(&tempty[b], ((acc >> 1) - 1) & 1)) timed_out = true;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * kLmTcNT);
                const int k1 = min(KB, k0 + kLmSegStages);
                for (int kb = k0; kb < k1; ++kb, ++g) {
                    const int s = g % kLmTcStages, u = g / kLmTcStages;
                    if (!mbar_wait_bounded(&full[s], u & 1)) timed_out = true;
                    tc_fence_after();
                    const uint32_t a0 = smem_addr(smem + s * kLmTcStage), x0 = a0 + kLmTcA;
#pragma unroll
                    for (int q = 0; q < kLmKbs; ++q) {
                        const uint32_t a = a0 + q * kTileRows * 128, x = x0 + q * kLmTcNT * 128;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            umma_bf16(d, umma_desc_sw128(a + 32 * k), umma_desc_sw128(x + 32 * k), idesc,
                                      (kb != k0 || q != 0 || k != 0) ? 1u : 0u);
                    }
                    umma_commit(&empty[s]);
                }
                umma_commit(&tfull[b]);
            }
        }
    } else if (warp >= 2) {
        const int quad = warp & 3;
        int acc = 0;
        for (int j = 0; j < my_tiles; ++j) {
            float sum[kLmTcNT];
            for (int k0 = 0; k0 < KB; k0 += kLmSegStages, ++acc) {
                const int b = acc & 1;
                if (!mbar_wait_bounded(&tfull[b], (acc >> 1) & 1)) timed_out = true;
                __syncwarp();  // the TMEM load below is .aligned
                tc_fence_after();
                uint32_t v[16];
                tmem_ld16_async(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(b * kLmTcNT), v);
                tmem_wait_ld(v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&tempty[b]);
#pragma unroll
                for (int m = 0; m < kLmTcNT; ++m)
                    sum[m] = k0 == 0 ? __uint_as_float(v[m]) : sum[m] + __uint_as_float(v[m]);
            }
            const int t = (int)blockIdx.x + j * (int)gridDim.x;
            const bool first = t < nt1;
            const int row = (first ? t : t - nt1) * kTileRows + quad * 32 + lane;
            float *out = first ? p.logits : p.logits2;
            const long stride = first ? p.logits_stride : p.logits2_stride;
            if (row < (first ? p.V : p.V2)) {
#pragma unroll
                for (int m = 0; m < kLmTcNT; ++m)
                    if (m < p.M)
                        out[(size_t)m * stride + row] = sum[m];
            }
        }
    }
    if (timed_out) record_timeout(p.status);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        tmem_dealloc(tmem, 2 * kLmTcNT);
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// A 2-D bf16 tensor map: `rows` x `cols` (row-major), box box_cols x box_rows.
bool make_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_cols,
              uint32_t box_rows, bool swizzle)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 3-D view of a bf16 [rows][cols] matrix for K-block boxes: dims (64 elements,
// rows, cols / 64), so that a box (64, box_rows, kbs) lands as kbs consecutive
// K-block tiles of box_rows x 128 bytes (128-byte swizzle).
bool make_map_kblocks(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                      uint32_t kbs)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[3] = {64, rows, (cols + 63) / 64};
    const cuuint64_t strides[2] = {cols * 2, 128};
    const cuuint32_t box[3] = {64, box_rows, kbs};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_tc(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                      int cluster_x, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int n = 0;
    if (cluster_x > 0) {
        attrs[n].id = cudaLaunchAttributeClusterDimension;
        attrs[n].val.clusterDim.x = cluster_x;
        attrs[n].val.clusterDim.y = 1;
        attrs[n].val.clusterDim.z = 1;
        ++n;
    }
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    cfg.attrs = attrs;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Once per kernel and device: the dynamic shared-memory limit (when
// `dynamic` is set) and the largest carveout.
template <typename K>
cudaError_t allow_smem_tc(K kernel, bool dynamic = true)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    static std::mutex mu;
    static std::set<std::pair<const void *, int>> done;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(reinterpret_cast<const void *>(kernel), dev);
    if (done.count(key))
        return cudaSuccess;
    e = dynamic ? cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmemLimit)
                : cudaSuccess;
    if (e == cudaSuccess)  // same carveout as every other kernel of the library (co-residency)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        done.insert(key);
    return e;
}

}  // namespace

size_t tc_down_smem(int NT, int ns, int wt) { return down_tc_layout(NT, ns, wt).total + 1024; }

bool lm_head_shape_ok(int M, int H, int V) { return M >= 1 && M <= kLmTcNT && H >= 64 && H % 64 == 0 && V >= 1; }

cudaError_t launch_lm_head(const LmHeadParams &p, const LaunchCfg &cfg, cudaStream_t stream)
{
    CUtensorMap map_w, map_w2, map_x;
    if (!lm_head_shape_ok(p.M, p.H, p.V) || p.V2 < 0 ||
        !make_map_kblocks(&map_w, p.w, (uint64_t)p.V, (uint64_t)p.H, kTileRows, kLmKbs) ||
        !make_map_kblocks(&map_w2, p.V2 > 0 ? p.w2 : p.w, (uint64_t)(p.V2 > 0 ? p.V2 : p.V), (uint64_t)p.H,
                          kTileRows, kLmKbs) ||
        !make_map(&map_x, p.mixed, (uint64_t)p.M, (uint64_t)p.H, kKBlock, kLmTcNT, true))
        return cudaErrorInvalidValue;
    const cudaError_t e = allow_smem_tc(hc_lm_head_tc_kernel);
    if (e != cudaSuccess)
        return e;
    const int ntiles = (p.V + kTileRows - 1) / kTileRows + (p.V2 + kTileRows - 1) / kTileRows;
    return launch_tc(hc_lm_head_tc_kernel, dim3((unsigned)std::min(ntiles, cfg.sm_count)), dim3(kLmTcThreads),
                     kLmTcSmem, stream, 0, p, map_w, map_w2, map_x);
}
size_t tc_up_smem(int NT, int ns, int C, int HBt, int wt) { return up_tc_layout(NT, ns, C, HBt, wt).total + 1024; }

cudaError_t launch_tc_call(const TcCall &t, cudaStream_t stream)
{
    CUtensorMap map_d, map_i, map_u, map_xhi, map_xlo, map_act, map_alo, map_nhi, map_nlo;
    const TcPrepParams &pp = t.prep;
    const TcDownParams &d = t.down;
    const TcUpParams &u = t.up;
    // INT4 weights are dequantised by producer warps; their (unused) weight
    // maps are encoded over the normed buffer, a valid bf16 tensor.
    const bool qd = d.wt == 1, qu = u.wt == 1;
    const int M = pp.M, W = pp.W;
    if (!make_map(&map_d, qd ? pp.x_hi : t.wd, qd ? M : d.L, W, kKBlock, 32, true) ||
        !make_map(&map_i, qd ? pp.x_hi : d.has_inject ? t.wi : t.wd, qd ? M : d.has_inject ? d.C : d.L, W, kKBlock,
                  32, true) ||
        !make_map(&map_u, qu ? pp.x_hi : t.wu, qu ? M : W, qu ? W : u.L, kKBlock, u.HBt, true) ||
        !make_map(&map_xhi, pp.x_hi, M, W, kKBlock, d.NT, true) ||
        !make_map(&map_xlo, pp.x_lo, M, W, kKBlock, d.NT, true) ||
        !make_map(&map_act, t.red.act_hi, M, u.L, kKBlock, u.NT, true) ||
        !make_map(&map_alo, t.red.act_lo, M, u.L, kKBlock, u.NT, true) ||
        !make_map(&map_nhi, pp.x_hi, M, W, u.HBt, u.NT, false) ||
        !make_map(&map_nlo, pp.x_lo, M, W, u.HBt, u.NT, false))
        return cudaErrorInvalidValue;

    auto kd = qd ? hc_tc_down_kernel<1> : hc_tc_down_kernel<0>;
    auto ku = qu ? hc_tc_up_kernel<1> : hc_tc_up_kernel<0>;
    cudaError_t e;
    if ((e = allow_smem_tc(kd)) != cudaSuccess) return e;
    if ((e = allow_smem_tc(ku)) != cudaSuccess) return e;
    if ((e = allow_smem_tc(hc_tc_reduce_kernel)) != cudaSuccess) return e;
    if ((e = allow_smem_tc(hc_tc_prep_kernel, false)) != cudaSuccess) return e;
    // Up to kPrepVec vectors per thread, so that the M * C CTAs fit the GPU at once.
    const int prep_threads = std::min(kPrepThreads, ((pp.H / 8 + kPrepVec - 1) / kPrepVec + 31) / 32 * 32);
    e = launch_tc(hc_tc_prep_kernel, dim3(M, pp.C), dim3(prep_threads), 0, stream, 0, pp);
    if (e != cudaSuccess)
        return e;
    const int ntiles = (M + d.NT - 1) / d.NT;
    e = launch_tc(kd, dim3(d.nchunk, (d.R + kTileRows - 1) / kTileRows, ntiles), dim3(kThreads),
                  tc_down_smem(d.NT, d.n_stages, d.wt), stream, 0, d, map_d, map_i, map_xhi, map_xlo);
    if (e != cudaSuccess)
        return e;
    // About one output per thread on one CTA per SM (more CTAs only past 1024 threads each),
    // on the SMs the up kernel's CTAs leave free when they all fit beside it.
    const long nred = (long)t.red.M * t.red.R;
    const int up_ctas = (int)(((u.H + u.HBt - 1) / u.HBt) * ntiles);
    const int red_ctas = up_ctas <= kTcChunkCtas - 32 ? kTcChunkCtas - up_ctas : kTcChunkCtas;
    const long per = (nred + red_ctas - 1) / red_ctas;
    const int rthreads = (int)std::min<long>(1024, (per + 31) / 32 * 32);
    e = launch_tc(hc_tc_reduce_kernel, dim3((unsigned)((nred + rthreads - 1) / rthreads)), dim3(rthreads),
                  kTcReduceSmemReserve, stream, 0, t.red);
    if (e != cudaSuccess)
        return e;
    return launch_tc(ku, dim3((u.H + u.HBt - 1) / u.HBt, ntiles), dim3(kUpThreads),
                     tc_up_smem(u.NT, u.n_stages, u.C, u.HBt, u.wt), stream, 0, u, map_u, map_act, map_alo, map_nhi,
                     map_nlo);
}

}  // namespace tshc
