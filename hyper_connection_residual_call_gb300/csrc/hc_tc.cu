// hc_tc.cu -- the batched (M >= 16 tokens) hyper-connection call on the
// 5th-generation tensor cores: tcgen05.mma with TMEM accumulators, weights
// streamed by tensor-map TMA in the 128-byte swizzled layout.
//
// At M tokens the projections are dense contractions (families/qwen4/hc.rs
// runs them as GEMVs per token; real_forward.rs batches such GEMVs into M-row
// GEMMs inside a prefill micro-batch). Three kernels, PDL-chained:
//
//  hc_tc_down_kernel   D[128 rows][N tokens] = W[rows][chunk] * X[chunk][tokens]
//                      with X = raw * g built by producer warps as bf16 hi + lo
//                      (x = hi + lo to ~16 significant bits; two MMAs per
//                      K step), so the down projection keeps fp32-level
//                      accuracy. A cluster of CS CTAs covers one stream; the
//                      partial tiles meet in distributed shared memory and the
//                      cluster writes the stream's partial z and the stream's
//                      per-token sum of squares.
//  hc_tc_reduce_kernel z = sum_c inv_rms[c] * part[c]; act = silu(z / C) (fp32 and
//                      bf16 hi/lo for the up GEMM), gates = 2 sigmoid(z / C).
//  hc_tc_up_kernel     D[C*HBt rows][N] = Wu[rows {c*H + h}][L] * act^T (hi + lo),
//                      epilogue: w = sigmoid(D), mixed[h] = mean_c w * raw *
//                      inv_rms * g, with the raw tile staged by TMA.
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

constexpr int kThreads = 256;  // 8 warps
constexpr int kTileRows = 128; // UMMA M
constexpr int kKBlock = 64;    // bf16 elements per 128-byte swizzled row
constexpr int kProducers = 192; // warps 2-7 build the down kernel's activation tiles

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Sigmoid from the fast exponential and division intrinsics (relative error
// ~1e-6, far inside the 1e-3 bar), for the per-element epilogues.
__device__ __forceinline__ float sigm_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

__device__ __forceinline__ float4 dsmem_ld_f32x4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
    return v;
}

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

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

__host__ __device__ constexpr uint32_t tmem_cols(int n)
{
    return n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : 256u;
}

struct TcSmem {
    uint32_t stage_bytes, a_bytes, b_bytes;
    uint32_t ring, extra, bars, total;
};

// Down kernel shared memory: ring of stages [A 16 KB | B_hi | B_lo], then the
// per-token sums of squares, then this CTA's chunk of g (bf16, at most
// kMaxChunk elements), then barriers.
constexpr int kMaxChunk = 2048;
// A stage is [A_hi | A_lo (INT4 weights only) | B_hi | B_lo].
__host__ __device__ inline TcSmem down_tc_layout(int NT, int ns, int wt)
{
    TcSmem s;
    s.a_bytes = kTileRows * 128;
    s.b_bytes = NT * 128;
    s.stage_bytes = s.a_bytes * (1 + wt) + 2 * s.b_bytes;
    s.ring = 0;
    s.extra = s.ring + ns * s.stage_bytes;          // ssq_s: NT floats, then g_s
    s.bars = s.extra + ((NT * 4 + 127) / 128) * 128 + kMaxChunk * 2;
    s.total = s.bars + 8 * (3 * ns + 2) + 16;
    return s;
}

// Dequantises 8 INT4-affine codes (element e in nibble e of `codes`) with one
// scale and bias (fp16 bits) and splits them into bf16 hi and lo parts:
// w = q * s + b in fp32, hi = bf16(w), lo = bf16(w - hi).
__device__ __forceinline__ void int4x8_hilo(uint32_t codes, uint16_t sb, uint16_t bb, uint4 &hi, uint4 &lo)
{
    const float sc = __half2float(__ushort_as_half(sb)), bi = __half2float(__ushort_as_half(bb));
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float wa = fmaf((float)((codes >> (8 * e)) & 0xFu), sc, bi);
        const float wb = fmaf((float)((codes >> (8 * e + 4)) & 0xFu), sc, bi);
        const uint32_t hh = pack_bf16x2(wa, wb);
        h[e] = hh;
        l[e] = pack_bf16x2(wa - bf16_lo(hh), wb - bf16_hi(hh));
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Up kernel: ring, then raw tile [C][NT][HBt] bf16, inv_rms tile [NT][C], and
// for a fused inject-add the sublayer-output tile [NT][HBt] bf16 and the
// previous gates [NT][C].
__host__ __device__ inline uint32_t up_tc_raw_bytes(int NT, int C, int HBt)
{
    return ((C * NT * HBt * 2 + 1023) / 1024) * 1024;
}
__host__ __device__ inline uint32_t up_tc_small_bytes(int NT, int C) { return ((NT * C * 4 + 127) / 128) * 128; }
__host__ __device__ inline uint32_t up_tc_out_bytes(int NT, int HBt) { return ((NT * HBt * 2 + 127) / 128) * 128; }

__host__ __device__ inline TcSmem up_tc_layout(int NT, int ns, int C, int HBt, int wt)
{
    TcSmem s;
    s.a_bytes = kTileRows * 128;
    s.b_bytes = NT * 128;
    s.stage_bytes = s.a_bytes * (1 + wt) + 2 * s.b_bytes;
    s.ring = 0;
    s.extra = s.ring + ns * s.stage_bytes;
    s.bars = s.extra + up_tc_raw_bytes(NT, C, HBt) + 2 * up_tc_small_bytes(NT, C) + up_tc_out_bytes(NT, HBt);
    s.total = s.bars + 8 * (4 * ns + 2) + 16;
    return s;
}

// ---------------------------------------------------------------- down

template <int WT>
__global__ void __launch_bounds__(kThreads, 1)
hc_tc_down_kernel(const TcDownParams p, const __grid_constant__ CUtensorMap map_d,
                  const __grid_constant__ CUtensorMap map_i)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int NT = p.NT, NS = p.n_stages;
    const TcSmem lay = down_tc_layout(NT, NS, WT);
    const uint32_t b_off = lay.a_bytes * (1 + WT);  // B_hi within a stage
    float *ssq_s = reinterpret_cast<float *>(smem + lay.extra);
    uint16_t *g_s = reinterpret_cast<uint16_t *>(smem + lay.extra + ((NT * 4 + 127) / 128) * 128);
    uint64_t *full_a = reinterpret_cast<uint64_t *>(smem + lay.bars);
    uint64_t *full_b = full_a + NS;
    uint64_t *empty = full_b + NS;
    uint64_t *done = empty + NS;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = blockIdx.x;                 // chunk within the stream == cluster rank
    const int c = blockIdx.y / p.RT;          // stream
    const int rt = blockIdx.y % p.RT;         // row tile
    const int tile = blockIdx.z;              // token tile
    const int r0 = rt * kTileRows;
    const int k0 = c * p.H + q * p.chunk;
    const int KB = p.chunk / kKBlock;
    const uint32_t ncols = tmem_cols(NT);

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
            mbar_init(&full_a[s], 1);
            mbar_init(&full_b[s], kProducers);
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
    // g is a weight: this CTA's chunk goes to shared memory before the wait
    // (read by the producers after this barrier; the TMA producer below runs
    // ahead without any further block barrier).
    for (int i = tid; i < p.chunk / 8; i += kThreads)
        reinterpret_cast<uint4 *>(g_s)[i] = reinterpret_cast<const uint4 *>(p.g + k0)[i];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool timed_out = false;

    if (WT == 0 && warp == 0 && lane == 0) {
        // TMA producer of the weight tiles (independent of the previous kernel).
        tma_prefetch_map(&map_d);
        if (p.has_inject) tma_prefetch_map(&map_i);
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % NS, u = kb / NS;
            if (u > 0 && !mbar_wait_bounded(&empty[s], (u - 1) & 1)) timed_out = true;
            uint8_t *a = smem + lay.ring + s * lay.stage_bytes;
            mbar_arrive_expect_tx(&full_a[s], nbox * 32 * 128);
            for (int b = 0; b < 4; ++b) {
                const int gr = r0 + 32 * b;
                if (gr + 32 <= p.L)
                    tma_load_2d(a + b * 32 * 128, &map_d, k0 + kb * kKBlock, gr, &full_a[s]);
                else if (gr == p.L && p.has_inject)
                    tma_load_2d(a + b * 32 * 128, &map_i, k0 + kb * kKBlock, 0, &full_a[s]);
            }
        }
    }
    if (warp < 2)
        pdl_wait();  // raw is produced by the previous kernel in the stream

    if (warp >= 2) {
        // Activation producers (warps 2-7): per K block, X = raw * g as bf16
        // hi + lo in the swizzled K-major layout. Thread t handles the 16-byte
        // chunks i = t + kProducers j of the NT x 64 block: token i / 8, chunk
        // i % 8, so eight consecutive lanes read one token's 128 contiguous
        // bytes (coalesced), and accumulate that token's sum of squares.
        const int t = tid - 64;
        const int ck = t & 7;                  // 16-byte chunk within the 64-element K block
        constexpr int kItems = (kTileRows * 8 + kProducers - 1) / kProducers;
        float ssq[kItems], inj_g[kItems];
        const uint4 *rrow[kItems];
        const uint4 *orow[kItems];
        bool live[kItems];
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            const int n = (t + kProducers * j) >> 3;   // token of chunk t + kProducers j
            const int m = tile * NT + n;
            live[j] = n < NT && m < p.M;
            ssq[j] = 0.f;
            rrow[j] = reinterpret_cast<const uint4 *>(p.raw + (size_t)(live[j] ? m : 0) * p.W + k0) + ck;
            orow[j] = p.inj_out ? reinterpret_cast<const uint4 *>(p.inj_out + (size_t)(live[j] ? m : 0) * p.H
                                                                  + q * p.chunk) + ck
                                : nullptr;
        }
        // INT4 weights: item j is also row (t + kProducers j) / 8 of the A tile,
        // chunk ck: 8 codes (4 bytes) and the group's scale and bias.
        const uint8_t *wq[kItems];
        const uint16_t *wsc[kItems];
        const uint16_t *wbi[kItems];
        if constexpr (WT == 1) {
#pragma unroll
            for (int j = 0; j < kItems; ++j) {
                const int rr = (t + kProducers * j) >> 3, gr = r0 + rr;
                const WeightView *v = gr < p.L ? &p.dw : (p.has_inject && gr < p.L + p.C) ? &p.iw : nullptr;
                const int row = gr < p.L ? gr : gr - p.L;
                wq[j] = (v && rr < kTileRows) ? static_cast<const uint8_t *>(v->data) + ((size_t)row * p.W + k0) / 2 : nullptr;
                wsc[j] = wq[j] ? v->scales + (size_t)row * (p.W / v->group) : nullptr;
                wbi[j] = wq[j] ? v->biases + (size_t)row * (p.W / v->group) : nullptr;
            }
        }
        // The next K block's chunks are loaded while the current one is converted.
        uint4 rnext[kItems], onext[kItems];
        uint32_t qnext[kItems];
        uint16_t snext[kItems], bnext[kItems];
        auto fetch_w = [&](int kb) {
            if constexpr (WT == 1) {
                const int col = kb * kKBlock + 8 * ck;  // within the chunk
#pragma unroll
                for (int j = 0; j < kItems; ++j) {
                    qnext[j] = wq[j] ? *reinterpret_cast<const uint32_t *>(wq[j] + col / 2) : 0u;
                    snext[j] = wq[j] ? wsc[j][(k0 + col) / p.dw.group] : (uint16_t)0;
                    bnext[j] = wq[j] ? wbi[j][(k0 + col) / p.dw.group] : (uint16_t)0;
                }
            }
        };
        auto fetch = [&](int kb) {
#pragma unroll
            for (int j = 0; j < kItems; ++j) {
                rnext[j] = live[j] ? rrow[j][kb * (kKBlock / 8)] : make_uint4(0, 0, 0, 0);
                onext[j] = (live[j] && p.inj_out) ? orow[j][kb * (kKBlock / 8)] : make_uint4(0, 0, 0, 0);
            }
            fetch_w(kb);
        };
        fetch_w(0);  // weights do not depend on the previous kernel
        pdl_wait();  // raw is produced by the previous kernel in the stream
        fetch(0);
        // The previous gates come from the previous call's reduce kernel, which
        // can still be running when this kernel starts: read only after the wait.
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            const int m = tile * NT + ((t + kProducers * j) >> 3);
            inj_g[j] = (live[j] && p.inj_out) ? p.inj_gate[(size_t)m * p.inj_stride + c] : 0.f;
        }
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % NS, u = kb / NS;
            uint4 rcur[kItems], ocur[kItems];
            uint32_t qcur[kItems];
            uint16_t scur[kItems], bcur[kItems];
#pragma unroll
            for (int j = 0; j < kItems; ++j) {
                rcur[j] = rnext[j];
                ocur[j] = onext[j];
                qcur[j] = qnext[j];
                scur[j] = snext[j];
                bcur[j] = bnext[j];
            }
            if (kb + 1 < KB)
                fetch(kb + 1);
            if (u > 0 && !mbar_wait_bounded(&empty[s], (u - 1) & 1)) timed_out = true;
            uint8_t *ahi = smem + lay.ring + s * lay.stage_bytes;
            uint8_t *bhi = ahi + b_off;
            uint8_t *blo = bhi + lay.b_bytes;
            if constexpr (WT == 1) {
                uint8_t *alo = ahi + lay.a_bytes;
#pragma unroll
                for (int j = 0; j < kItems; ++j) {
                    const int rr = (t + kProducers * j) >> 3;
                    if (rr >= kTileRows)
                        continue;
                    uint4 hi = make_uint4(0, 0, 0, 0), lo = make_uint4(0, 0, 0, 0);
                    if (wq[j])
                        int4x8_hilo(qcur[j], scur[j], bcur[j], hi, lo);
                    *reinterpret_cast<uint4 *>(ahi + sw128_offset(rr, 8 * ck)) = hi;
                    *reinterpret_cast<uint4 *>(alo + sw128_offset(rr, 8 * ck)) = lo;
                }
            }
            const uint4 gv = reinterpret_cast<const uint4 *>(g_s + kb * kKBlock)[ck];
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int j = 0; j < kItems; ++j) {
                const int n = (t + kProducers * j) >> 3;
                if (n >= NT)
                    continue;
                uint4 hi = make_uint4(0, 0, 0, 0), lo = make_uint4(0, 0, 0, 0);
                if (live[j]) {
                    const uint32_t rw[4] = {rcur[j].x, rcur[j].y, rcur[j].z, rcur[j].w};
                    const uint32_t ow[4] = {ocur[j].x, ocur[j].y, ocur[j].z, ocur[j].w};
                    uint32_t h[4], l[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        // Packed conversions: one bf16x2 rounding per pair.
                        float r_a = bf16_lo(rw[e]), r_b = bf16_hi(rw[e]);
                        if (p.inj_out) {  // fused inject-add, rounded as the inject-add kernel rounds
                            const uint32_t rr = pack_bf16x2(fmaf(bf16_lo(ow[e]), inj_g[j], r_a),
                                                            fmaf(bf16_hi(ow[e]), inj_g[j], r_b));
                            r_a = bf16_lo(rr);
                            r_b = bf16_hi(rr);
                        }
                        ssq[j] = fmaf(r_a, r_a, ssq[j]);
                        ssq[j] = fmaf(r_b, r_b, ssq[j]);
                        const float x_a = r_a * bf16_lo(gw[e]), x_b = r_b * bf16_hi(gw[e]);
                        const uint32_t hh = pack_bf16x2(x_a, x_b);
                        h[e] = hh;
                        l[e] = pack_bf16x2(x_a - bf16_lo(hh), x_b - bf16_hi(hh));
                    }
                    hi = make_uint4(h[0], h[1], h[2], h[3]);
                    lo = make_uint4(l[0], l[1], l[2], l[3]);
                }
                *reinterpret_cast<uint4 *>(bhi + sw128_offset(n, 8 * ck)) = hi;
                *reinterpret_cast<uint4 *>(blo + sw128_offset(n, 8 * ck)) = lo;
            }
            fence_async_shared();
            mbar_arrive(&full_b[s]);
        }
        // A token's sum of squares: its 8 lanes (one octet of the warp), fixed order.
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            float v = ssq[j];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            const int n = (t + kProducers * j) >> 3;
            if (ck == 0 && n < NT)
                ssq_s[n] = v;
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer.
        const uint32_t idesc = umma_idesc_bf16(kTileRows, NT);
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % NS, u = kb / NS;
            if (WT == 0 && !mbar_wait_bounded(&full_a[s], u & 1)) timed_out = true;
            if (!mbar_wait_bounded(&full_b[s], u & 1)) timed_out = true;
            tc_fence_after();
            const uint32_t a = smem_addr(smem + lay.ring + s * lay.stage_bytes);
            const uint32_t al = a + lay.a_bytes;  // A_lo (INT4 weights)
            const uint32_t bh = a + b_off, bl = bh + lay.b_bytes;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                umma_bf16(tmem, umma_desc_sw128(a + 32 * k), umma_desc_sw128(bh + 32 * k), idesc, (kb | k) != 0);
                umma_bf16(tmem, umma_desc_sw128(a + 32 * k), umma_desc_sw128(bl + 32 * k), idesc, 1);
                if (WT == 1)  // the weight's lo part against the activation's hi part
                    umma_bf16(tmem, umma_desc_sw128(al + 32 * k), umma_desc_sw128(bh + 32 * k), idesc, 1);
            }
            umma_commit(&empty[s]);
        }
        umma_commit(done);
    }

    // Epilogue: the 128 x NT fp32 partial tile, TMEM -> shared (over the ring).
    // The barrier also reconverges the warps whose lane 0 had a producer role.
    __syncthreads();
    float *ptile = reinterpret_cast<float *>(smem + lay.ring);
    const int pstride = NT + 4;
    if (warp < 4) {
        if (!mbar_wait_bounded(done, 0)) timed_out = true;
        __syncwarp();  // the TMEM loads below are .aligned
        tc_fence_after();
        const int row = warp * 32 + lane;
        for (int c0 = 0; c0 < NT; c0 += 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4 *>(ptile + row * pstride + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
    }
    if (timed_out) record_timeout(p.status);
    tc_fence_before();
    cluster_sync();  // every CTA of the stream has its partial tile and sums of squares in shared memory

    // Rank q sums rows [q*RS, (q+1)*RS) over the cluster, in rank order, four
    // tokens at a time; the remote loads of a group are all issued before any
    // is used, so their latencies overlap.
    const int RS = kTileRows / p.CS;
    const int NT4 = NT / 4;  // NT is a multiple of 16
    for (int i = tid; i < RS * NT4; i += kThreads) {
        const int r = q * RS + i / NT4, n = (i % NT4) * 4;
        const int gr = r0 + r;
        float4 v[8];
#pragma unroll
        for (int pr = 0; pr < 8; ++pr)
            v[pr] = pr < p.CS ? dsmem_ld_f32x4(dsmem_addr(ptile + r * pstride + n, pr)) : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 z = v[0];
#pragma unroll
        for (int pr = 1; pr < 8; ++pr) {
            if (pr < p.CS) {
                z.x += v[pr].x; z.y += v[pr].y; z.z += v[pr].z; z.w += v[pr].w;
            }
        }
        if (gr < p.R) {
            const float zz[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = tile * NT + n + e;
                if (m < p.M)
                    p.part[((size_t)c * p.R + gr) * p.M + m] = zz[e];
            }
        }
    }
    if (q == 0 && rt == 0) {
        for (int n = tid; n < NT; n += kThreads) {
            const int m = tile * NT + n;
            float s = 0.f;
            for (int pr = 0; pr < p.CS; ++pr)
                s += dsmem_ld_f32(dsmem_addr(ssq_s + n, pr));
            if (m < p.M)
                p.ssq[(size_t)c * p.M + m] = s;
        }
    }
    cluster_sync();  // peers have finished reading this CTA's shared memory
    tc_fence_after();
    if (warp == 0)
        tmem_dealloc(tmem, ncols);
}

// ---------------------------------------------------------------- reduce

// Grid (ceil(M / 32), ceil(R / 32)); 1024 threads, one element each. The
// partials are read along tokens and act is written along rows, through a
// shared-memory transpose, so both sides are coalesced.
__global__ void __launch_bounds__(1024) hc_tc_reduce_kernel(const TcReduceParams p)
{
    __shared__ float zt[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int m0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    pdl_launch_dependents();
    pdl_wait();
    {
        // z of row r0 + ty, token m0 + tx: every load first, then the sum in stream order.
        const int m = m0 + tx, r = r0 + ty;
        const bool ok = m < p.M && r < p.R;
        float sq[8], pt[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            sq[c] = (c < p.C && ok) ? p.ssq[(size_t)c * p.M + m] : 0.f;
            pt[c] = (c < p.C && ok) ? p.part[((size_t)c * p.R + r) * p.M + m] : 0.f;
        }
        float z = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            if (c < p.C && ok) {
                const float inv = 1.0f / sqrtf(sq[c] / (float)p.H + p.eps);
                z = fmaf(inv, pt[c], z);
                if (r == 0)
                    p.inv_rms[(size_t)m * p.C + c] = inv;
            }
        }
        zt[ty][tx] = z;
    }
    __syncthreads();
    // Row r0 + tx of token m0 + ty.
    const int r = r0 + tx, mm = m0 + ty;
    if (r >= p.R || mm >= p.M)
        return;
    const float zc = zt[tx][ty] * p.inv_C;
    if (r < p.L) {
        const float a = zc * sigm_fast(zc);
        const float hi = bf16_round(a);
        p.act[(size_t)mm * p.L + r] = a;
        p.act_hi[(size_t)mm * p.L + r] = __bfloat16_as_ushort(__float2bfloat16_rn(a));
        p.act_lo[(size_t)mm * p.L + r] = __bfloat16_as_ushort(__float2bfloat16_rn(a - hi));
    } else {
        p.gate[(size_t)mm * p.gate_stride + (r - p.L)] = 2.0f * sigm_fast(zc);
    }
}

// ---------------------------------------------------------------- up

template <int WT>
__global__ void __launch_bounds__(kThreads, 1)
hc_tc_up_kernel(const TcUpParams p, const __grid_constant__ CUtensorMap map_u,
                const __grid_constant__ CUtensorMap map_ahi, const __grid_constant__ CUtensorMap map_alo,
                const __grid_constant__ CUtensorMap map_raw)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int NT = p.NT, NS = p.n_stages, C = p.C, HBt = p.HBt;
    const TcSmem lay = up_tc_layout(NT, NS, C, HBt, WT);
    const uint32_t b_off = lay.a_bytes * (1 + WT);  // B_hi within a stage
    uint16_t *raw_s = reinterpret_cast<uint16_t *>(smem + lay.extra);  // [C][NT][HBt]
    float *inv_s = reinterpret_cast<float *>(smem + lay.extra + up_tc_raw_bytes(NT, C, HBt));  // [NT][C]
    float *pgate_s = inv_s + up_tc_small_bytes(NT, C) / 4;                                       // [NT][C]
    uint16_t *out_s = reinterpret_cast<uint16_t *>(pgate_s + up_tc_small_bytes(NT, C) / 4);     // [NT][HBt]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bars);
    uint64_t *empty = full + NS;
    uint64_t *fullp = empty + NS;  // INT4: the producers' A tiles of a stage are written
    uint64_t *done = fullp + NS;
    uint64_t *raw_bar = done + 1;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(raw_bar + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h0 = blockIdx.x * HBt;
    const int tile = blockIdx.y;
    const int KB = p.L / kKBlock;
    const uint32_t ncols = tmem_cols(NT);

    pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&fullp[s], kProducers);
        }
        mbar_init(done, 1);
        mbar_init(raw_bar, 1);
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
        pdl_wait();  // ... then the activations and the residual tile
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
            tma_load_2d(a + b_off, &map_ahi, kb * kKBlock, tile * NT, &full[s]);
            tma_load_2d(a + b_off + lay.b_bytes, &map_alo, kb * kKBlock, tile * NT, &full[s]);
        }
        mbar_arrive_expect_tx(raw_bar, C * NT * HBt * 2);
        for (int cc = 0; cc < C; ++cc)
            tma_load_2d(raw_s + cc * NT * HBt, &map_raw, cc * p.H + h0, tile * NT, raw_bar);
    } else if (WT == 1 && warp >= 2) {
        // INT4 weights: warps 2-7 dequantise the A tiles (rows (stream, h) of
        // this CTA, 64 columns per stage) to bf16 hi + lo. Thread t handles the
        // 16-byte chunks t + kProducers j: row / 8, chunk t % 8. The stages
        // before the ring wraps are written before the dependency wait.
        const int t = tid - 64;
        const int ck = t & 7;
        constexpr int kItems = (kTileRows * 8 + kProducers - 1) / kProducers;
        const uint8_t *wq[kItems];
        const uint16_t *wsc[kItems];
        const uint16_t *wbi[kItems];
        const int ngr = p.L / p.uw.group;
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            const int rr = (t + kProducers * j) >> 3;
            const int cc = rr / HBt, hl = rr % HBt;
            const bool ok = rr < kTileRows && cc < C && h0 + hl < p.H;
            const size_t row = (size_t)cc * p.H + h0 + hl;
            wq[j] = ok ? static_cast<const uint8_t *>(p.uw.data) + row * (p.L / 2) : nullptr;
            wsc[j] = ok ? p.uw.scales + row * ngr : nullptr;
            wbi[j] = ok ? p.uw.biases + row * ngr : nullptr;
        }
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % NS, u = kb / NS;
            if (kb == NS)
                pdl_wait();
            const int col = kb * kKBlock + 8 * ck;
            uint32_t q[kItems];
            uint16_t sc[kItems], bi[kItems];
#pragma unroll
            for (int j = 0; j < kItems; ++j) {
                q[j] = wq[j] ? *reinterpret_cast<const uint32_t *>(wq[j] + col / 2) : 0u;
                sc[j] = wq[j] ? wsc[j][col / p.uw.group] : (uint16_t)0;
                bi[j] = wq[j] ? wbi[j][col / p.uw.group] : (uint16_t)0;
            }
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
                    int4x8_hilo(q[j], sc[j], bi[j], hi, lo);
                *reinterpret_cast<uint4 *>(ahi + sw128_offset(rr, 8 * ck)) = hi;
                *reinterpret_cast<uint4 *>(alo + sw128_offset(rr, 8 * ck)) = lo;
            }
            fence_async_shared();
            mbar_arrive(&fullp[s]);
        }
        if (KB <= NS)
            pdl_wait();
    } else {
        pdl_wait();
    }

    if (warp == 1 && lane == 0) {
        const uint32_t idesc = umma_idesc_bf16(kTileRows, NT);
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % NS, u = kb / NS;
            if (!mbar_wait_bounded(&full[s], u & 1)) timed_out = true;
            if (WT == 1 && !mbar_wait_bounded(&fullp[s], u & 1)) timed_out = true;
            tc_fence_after();
            const uint32_t a = smem_addr(smem + lay.ring + s * lay.stage_bytes);
            const uint32_t al = a + lay.a_bytes;  // A_lo (INT4 weights)
            const uint32_t bh = a + b_off, bl = bh + lay.b_bytes;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                umma_bf16(tmem, umma_desc_sw128(a + 32 * k), umma_desc_sw128(bh + 32 * k), idesc, (kb | k) != 0);
                umma_bf16(tmem, umma_desc_sw128(a + 32 * k), umma_desc_sw128(bl + 32 * k), idesc, 1);
                if (WT == 1)  // the weight's lo part against the activation's hi part
                    umma_bf16(tmem, umma_desc_sw128(al + 32 * k), umma_desc_sw128(bh + 32 * k), idesc, 1);
            }
            umma_commit(&empty[s]);
        }
        umma_commit(done);
    }
    if (warp >= 4) {
        // While the MMAs run: inv_rms and, for a fused inject-add, the previous
        // gates and the sublayer-output tile of this CTA's h-block.
        // Every load of a thread is issued before any is stored (one round trip).
        constexpr int kPer = 16;  // NT * C <= 128 * 8 and NT * HBt / 8 <= 128 * 16
        float iv[kPer], gv2[kPer];
        uint4 ov[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int i = tid - 128 + 128 * j;
            const int n = i / C, cc = i % C, m = tile * NT + n;
            const bool ok = i < NT * C && m < p.M;
            iv[j] = ok ? p.inv_rms[(size_t)m * C + cc] : 0.f;
            gv2[j] = (ok && p.raw_out) ? p.inj_gate[(size_t)m * p.inj_stride + cc] : 0.f;
            const int v = i, nv = v / (HBt / 8), hv = (v % (HBt / 8)) * 8, mv = tile * NT + nv;
            const bool okv = p.raw_out && v < NT * HBt / 8 && mv < p.M && h0 + hv + 8 <= p.H;
            ov[j] = okv ? *reinterpret_cast<const uint4 *>(p.inj_out + (size_t)mv * p.H + h0 + hv)
                        : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int i = tid - 128 + 128 * j;
            if (i < NT * C) {
                inv_s[i] = iv[j];
                pgate_s[i] = gv2[j];
            }
            if (i < NT * HBt / 8)
                reinterpret_cast<uint4 *>(out_s)[i] = ov[j];
        }
    }
    __syncthreads();

    // Epilogue on all 8 warps: warp w reads TMEM lanes 32*(w%4).. (rows = (stream,
    // h) pairs) for the 16-column chunks of parity w/4.
    float *mix_s = reinterpret_cast<float *>(smem + lay.ring);  // [C][NT][HBt], over the ring
    {
        if (!mbar_wait_bounded(done, 0)) timed_out = true;
        if (!mbar_wait_bounded(raw_bar, 0)) timed_out = true;
        __syncwarp();  // the TMEM loads below are .aligned
        tc_fence_after();
        const int quad = warp & 3, half = warp >> 2;
        const int row = quad * 32 + lane;
        const int cc = row / HBt, hl = row % HBt;
        const bool live = cc < C && h0 + hl < p.H;
        const float gv = live ? __bfloat162float(__ushort_as_bfloat16(p.g[cc * p.H + h0 + hl])) : 0.f;
        // The warp's 16-column chunks c0 = 16*half + 32k: chunk k+1 is loaded from
        // TMEM while chunk k is processed (two register buffers; the loop body
        // stays small, which keeps the epilogue's code in the instruction cache).
        // Every shared-memory load of a chunk is issued before its first store:
        // the compiler cannot tell the global residual from the shared tiles,
        // so a load placed after a store would wait for it.
        const bool fused = p.raw_out != nullptr;
        uint16_t *rout = fused ? p.raw_out + (size_t)cc * p.H + h0 + hl : nullptr;
        auto process = [&](int c0, const uint32_t (&vr)[16]) {
            if (!live)
                return;
            float rv[16], sc[16], ov[16], pg[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int n = c0 + j;
                rv[j] = __bfloat162float(__ushort_as_bfloat16(raw_s[(cc * NT + n) * HBt + hl]));
                sc[j] = inv_s[n * C + cc] * gv;
                if (fused) {
                    ov[j] = __bfloat162float(__ushort_as_bfloat16(out_s[n * HBt + hl]));
                    pg[j] = pgate_s[n * C + cc];
                }
            }
            if (fused) {  // the inject-add: this thread owns residual elements (m, cc, h)
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    rv[j] = bf16_round(fmaf(ov[j], pg[j], rv[j]));
                    const int m = tile * NT + c0 + j;
                    if (m < p.M)
                        rout[(size_t)m * p.W] = __bfloat16_as_ushort(__float2bfloat16_rn(rv[j]));
                }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j)
                mix_s[(cc * NT + c0 + j) * HBt + hl] = sigm_fast(__uint_as_float(vr[j])) * (rv[j] * sc[j]);
        };
        const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16);
        uint32_t va[16], vb[16];
        int c0 = 16 * half;
        if (c0 < NT)  // warp-uniform
            tmem_ld16_async(tbase + c0, va);
        tmem_wait_ld(va);
#pragma unroll 1
        for (; c0 < NT; c0 += 64) {
            if (c0 + 32 < NT)
                tmem_ld16_async(tbase + c0 + 32, vb);
            process(c0, va);
            tmem_wait_ld(vb);
            if (c0 + 32 >= NT)
                break;
            if (c0 + 64 < NT)
                tmem_ld16_async(tbase + c0 + 64, va);
            process(c0 + 32, vb);
            tmem_wait_ld(va);
        }
    }
    tc_fence_before();
    __syncthreads();
    // Mean over the streams, 8 consecutive h of one token per item (stream order).
    for (int i = tid; i < NT * (HBt / 8); i += kThreads) {
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
size_t tc_up_smem(int NT, int ns, int C, int HBt, int wt) { return up_tc_layout(NT, ns, C, HBt, wt).total + 1024; }

cudaError_t launch_tc_call(const TcCall &t, cudaStream_t stream)
{
    CUtensorMap map_d, map_i, map_u, map_ahi, map_alo, map_raw;
    const TcDownParams &d = t.down;
    const TcUpParams &u = t.up;
    // INT4 weights are dequantised by producer warps; their (unused) weight
    // maps are encoded over the residual, a valid bf16 tensor.
    const bool q = d.wt == 1;
    if (!make_map(&map_d, q ? d.raw : t.wd, q ? d.M : d.L, d.W, kKBlock, 32, true) ||
        !make_map(&map_i, q ? d.raw : d.has_inject ? t.wi : t.wd, q ? d.M : d.has_inject ? d.C : d.L, d.W, kKBlock,
                  32, true) ||
        !make_map(&map_u, q ? u.raw : t.wu, q ? u.M : u.W, q ? u.W : u.L, kKBlock, u.HBt, true) ||
        !make_map(&map_ahi, t.red.act_hi, u.M, u.L, kKBlock, u.NT, true) ||
        !make_map(&map_alo, t.red.act_lo, u.M, u.L, kKBlock, u.NT, true) ||
        !make_map(&map_raw, u.raw, u.M, u.W, u.HBt, u.NT, false))
        return cudaErrorInvalidValue;

    auto kd = q ? hc_tc_down_kernel<1> : hc_tc_down_kernel<0>;
    auto ku = u.wt == 1 ? hc_tc_up_kernel<1> : hc_tc_up_kernel<0>;
    cudaError_t e;
    if ((e = allow_smem_tc(kd)) != cudaSuccess) return e;
    if ((e = allow_smem_tc(ku)) != cudaSuccess) return e;
    if ((e = allow_smem_tc(hc_tc_reduce_kernel, false)) != cudaSuccess) return e;
    const int ntiles = (d.M + d.NT - 1) / d.NT;
    e = launch_tc(kd, dim3(d.CS, d.C * d.RT, ntiles), dim3(kThreads),
                  tc_down_smem(d.NT, d.n_stages, d.wt), stream, d.CS, d, map_d, map_i);
    if (e != cudaSuccess)
        return e;
    e = launch_tc(hc_tc_reduce_kernel, dim3((t.red.M + 31) / 32, (t.red.R + 31) / 32), dim3(1024), 0, stream, 0,
                  t.red);
    if (e != cudaSuccess)
        return e;
    return launch_tc(ku, dim3((u.H + u.HBt - 1) / u.HBt, ntiles), dim3(kThreads),
                     tc_up_smem(u.NT, u.n_stages, u.C, u.HBt, u.wt), stream, 0, u, map_u, map_ahi, map_alo, map_raw);
}

}  // namespace tshc
