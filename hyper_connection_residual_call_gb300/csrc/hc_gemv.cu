// hc_gemv.cu -- CUDA-core kernels of the hyper-connection call for small
// token counts (weight-streaming GEMVs, HBM bound), the final mixer and the
// inject-add.
//
// The call (families/qwen4/mod.rs, "## Hyper-connections"; families/qwen4/
// hc.rs, encode_hyper_connection) runs as two kernels chained with
// programmatic dependent launch:
//
//  hc_down_kernel  grouped RMSNorm folded into a split-K down GEMV (plus the C
//                  block_inject_weight rows). A cluster of S CTAs shares a
//                  block of output rows; CTA s streams the weight columns of
//                  its chunk [s*KC, (s+1)*KC) into shared memory with bulk
//                  copies issued before it waits on the previous kernel, then
//                  forms x = raw * g for its chunk together with the chunk's
//                  sum of squares. Partial dots and sums of squares meet in
//                  distributed shared memory; rank q of the cluster finishes
//                  rows q, q+S, ... as z = sum_s inv_rms[stream(s)] * P_s, and
//                  writes silu(z / C) (down rows) or 2 sigmoid(z / C) (gate
//                  rows). The normalised vector never goes to HBM.
//  hc_up_kernel    CTA b streams up rows {c*H + h : h in its h-block} for all
//                  C streams into shared memory before waiting, then forms
//                  w = sigmoid(up . act) and the mean mix
//                  mixed[h] = (1/C) sum_c w[c*H+h] * raw[c*H+h] * inv_rms[c] * g[c*H+h].
//
// Reductions run in a fixed order: results are bit-identical run to run.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>
#include <set>
#include <utility>

#include "hc_kernels.h"
#include "ptx.cuh"

namespace tshc {

namespace {

constexpr int kMaxCluster = 8;  // CTAs per split-K cluster (portable maximum)

// Elements per 16-byte vector of weight storage: 8 bf16 or 32 INT4 codes.
template <int WT> struct Vec;
template <> struct Vec<0> { static constexpr int kElems = 8; };
template <> struct Vec<1> { static constexpr int kElems = 32; };

__host__ __device__ constexpr int round_up(int x, int m) { return (x + m - 1) / m * m; }
__host__ __device__ constexpr size_t round_up_sz(size_t x, size_t m) { return (x + m - 1) / m * m; }

// Activations x_s are stored permuted so that lane l of a warp reading "its"
// weight vector v = l + 32 i finds the matching activations as consecutive
// float4s across lanes (no shared-memory bank conflicts). Element j of the
// chunk, in vector v = j / VW at offset e = j % VW, sits at:
template <int VW>
__device__ __forceinline__ int xpos(int j)
{
    const int v = j / VW, e = j % VW;
    return (v >> 5) * (32 * VW) + (e >> 2) * 128 + (v & 31) * 4 + (e & 3);
}

struct DownSmem {
    size_t bar, w, sb, x, part, ssq, invr, red, total;
};

__host__ __device__ inline DownSmem down_layout(const DownParams &p, int mt)
{
    const int VW = p.down.type == 0 ? 8 : 32;
    const int kcp = round_up(p.KC, 32 * VW);
    const size_t seg = p.down.type == 0 ? (size_t)p.KC * 2 : (size_t)p.KC / 2;
    const int ng = p.down.type == 0 ? 0 : p.KC >> p.down.gshift;
    DownSmem s;
    s.bar = 0;
    s.w = 128;
    s.sb = round_up_sz(s.w + seg * p.rows_per_block, 128);
    s.x = round_up_sz(s.sb + sizeof(float) * 2 * (size_t)ng * p.rows_per_block, 128);
    s.part = round_up_sz(s.x + sizeof(float) * (size_t)mt * kcp, 128);
    s.ssq = round_up_sz(s.part + sizeof(float) * (size_t)mt * p.rows_per_block, 16);
    s.invr = round_up_sz(s.ssq + sizeof(float) * mt, 16);
    s.red = round_up_sz(s.invr + sizeof(float) * (size_t)mt * p.C, 16);
    s.total = round_up_sz(s.red + sizeof(float) * 32 * mt, 128);
    return s;
}

struct UpSmem {
    size_t bar, w, sb, act, wv, rv, gv, inv, total;
};

// Up kernel shared memory: weight rows, INT4 scales/biases, act tile, sigmoid
// outputs, and the mix operands staged right after the dependency wait:
// residual values rv [mt][C][HB], norm scale gv [C][HB], inv_rms [mt][C].
__host__ __device__ inline UpSmem up_layout(const UpParams &p, int mt)
{
    const size_t row = p.up.type == 0 ? (size_t)p.L * 2 : (size_t)p.L / 2;
    const int ng = p.up.type == 0 ? 0 : p.L >> p.up.gshift;
    UpSmem s;
    s.bar = 0;
    s.w = 128;
    s.sb = round_up_sz(s.w + row * p.C * p.HB, 128);
    s.act = round_up_sz(s.sb + sizeof(float) * 2 * (size_t)ng * p.C * p.HB, 128);
    s.wv = round_up_sz(s.act + sizeof(float) * (size_t)mt * p.L, 128);
    s.rv = round_up_sz(s.wv + sizeof(float) * (size_t)mt * p.C * p.HB, 128);
    s.gv = round_up_sz(s.rv + sizeof(float) * (size_t)mt * p.C * p.HB, 128);
    s.inv = round_up_sz(s.gv + sizeof(float) * (size_t)p.C * p.HB, 128);
    s.total = round_up_sz(s.inv + sizeof(float) * (size_t)mt * p.C, 128);
    return s;
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
// Shorter-latency sigmoid for the one-token kernels' dependency chain: the
// fast exponential and division intrinsics (relative error ~1e-6, far
// inside the 1e-3 bar on fp32 intermediates).
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

__device__ __forceinline__ void unpack_bf16x8(const uint4 &v, float (&f)[8])
{
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// rf[e] <- bf16(out[e] * gate + rf[e]): the inject-add of the previous
// sublayer, rounded exactly as the stand-alone inject-add kernel rounds it.
__device__ __forceinline__ void inject_bf16x8(float (&rf)[8], const uint16_t *out, float gate)
{
    float of[8];
    unpack_bf16x8(*reinterpret_cast<const uint4 *>(out), of);
#pragma unroll
    for (int e = 0; e < 8; ++e)
        rf[e] = __bfloat162float(__float2bfloat16_rn(fmaf(of[e], gate, rf[e])));
}

__device__ __forceinline__ float half_bits_to_float(uint16_t b)
{
    return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// A bf16 pair (element 2i in the low half of the word) as an fp32 pair.
__device__ __forceinline__ uint64_t bf16x2_as_f32x2(uint32_t w)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(w << 16), "r"(w & 0xffff0000u));
    return r;
}

// Sum of the two lanes: low + high.
__device__ __forceinline__ float f32x2_sum(uint64_t v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo + hi;
}

__device__ __forceinline__ void record_timeout(unsigned *status)
{
    if (status)
        atomicExch(status, kStatusTimeout);
}

// Dot of one weight row segment with MT activation rows, partial per lane.
// bf16: lane handles vectors v = lane + 32 i of 8 elements.
template <int MT>
__device__ __forceinline__ void row_dot_bf16(const uint4 *wrow, int nvec, const float *x, int xstride,
                                             int lane, float (&acc)[MT])
{
    // Two accumulation chains per token (even / odd elements) halve the
    // dependent-FMA depth; they are added once at the end.
    float a0[MT], a1[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) { a0[t] = 0.f; a1[t] = 0.f; }
#pragma unroll 2
    for (int v = lane; v < nvec; v += 32) {
        float wf[8];
        unpack_bf16x8(wrow[v], wf);
        const int p0 = xpos<8>(v * 8);
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            const float4 xa = *reinterpret_cast<const float4 *>(x + t * xstride + p0);
            const float4 xb = *reinterpret_cast<const float4 *>(x + t * xstride + p0 + 128);
            a0[t] = fmaf(wf[0], xa.x, a0[t]); a1[t] = fmaf(wf[1], xa.y, a1[t]);
            a0[t] = fmaf(wf[2], xa.z, a0[t]); a1[t] = fmaf(wf[3], xa.w, a1[t]);
            a0[t] = fmaf(wf[4], xb.x, a0[t]); a1[t] = fmaf(wf[5], xb.y, a1[t]);
            a0[t] = fmaf(wf[6], xb.z, a0[t]); a1[t] = fmaf(wf[7], xb.w, a1[t]);
        }
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t] += a0[t] + a1[t];
}

// INT4-affine: lane handles vectors of 32 codes (one group-aligned run of 32
// inputs, so one scale and bias).
template <int MT>
__device__ __forceinline__ void row_dot_int4(const uint4 *wrow, int nvec, const float *sb, int gshift,
                                             const float *x, int xstride, int lane, float (&acc)[MT])
{
    float a0[MT], a1[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) { a0[t] = 0.f; a1[t] = 0.f; }
    for (int v = lane; v < nvec; v += 32) {
        const uint4 q = wrow[v];
        const int gi = (v * 32) >> gshift;
        const float sc = sb[2 * gi], bi = sb[2 * gi + 1];
        const uint32_t words[4] = {q.x, q.y, q.z, q.w};
        const int base = (v >> 5) * 1024 + (v & 31) * 4;
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
            float wf[8];
#pragma unroll
            for (int n = 0; n < 8; ++n)
                wf[n] = fmaf((float)((words[wd] >> (4 * n)) & 0xFu), sc, bi);
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                // elements e = 8*wd .. 8*wd+7 sit in float4 groups e/4 = 2*wd, 2*wd+1
                const float4 xa = *reinterpret_cast<const float4 *>(x + t * xstride + base + (2 * wd) * 128);
                const float4 xb = *reinterpret_cast<const float4 *>(x + t * xstride + base + (2 * wd + 1) * 128);
                a0[t] = fmaf(wf[0], xa.x, a0[t]); a1[t] = fmaf(wf[1], xa.y, a1[t]);
                a0[t] = fmaf(wf[2], xa.z, a0[t]); a1[t] = fmaf(wf[3], xa.w, a1[t]);
                a0[t] = fmaf(wf[4], xb.x, a0[t]); a1[t] = fmaf(wf[5], xb.y, a1[t]);
                a0[t] = fmaf(wf[6], xb.z, a0[t]); a1[t] = fmaf(wf[7], xb.w, a1[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t] += a0[t] + a1[t];
}

template <int WT, int MT>
__global__ void __launch_bounds__(512) hc_down_kernel(const DownParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int VW = Vec<WT>::kElems;
    const DownSmem lay = down_layout(p, MT);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + lay.bar);
    unsigned char *w_s = smem + lay.w;
    float *sb_s = reinterpret_cast<float *>(smem + lay.sb);
    float *x_s = reinterpret_cast<float *>(smem + lay.x);
    float *part_s = reinterpret_cast<float *>(smem + lay.part);
    float *ssq_s = reinterpret_cast<float *>(smem + lay.ssq);
    float *invr_s = reinterpret_cast<float *>(smem + lay.invr);
    float *red_s = reinterpret_cast<float *>(smem + lay.red);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int s = blockIdx.x;  // chunk index == rank in the cluster (gridDim.x == cluster size)
    const int RPB = p.rows_per_block;
    const int r0 = blockIdx.y * RPB;
    const int nrows = min(RPB, p.R - r0);
    const int KC = p.KC, k0 = s * KC;
    const int kcp = round_up(KC, 32 * VW);
    const int nvec = KC / VW;
    const size_t seg = WT == 0 ? (size_t)KC * 2 : (size_t)KC / 2;

    pdl_launch_dependents();

    // Weights do not depend on the previous kernel: start streaming them now.
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(bar, (uint32_t)(seg * nrows));
        for (int r = 0; r < nrows; ++r) {
            const int gr = r0 + r;
            const WeightView &wv = gr < p.L ? p.down : p.inject;
            const int row = gr < p.L ? gr : gr - p.L;
            const unsigned char *src = static_cast<const unsigned char *>(wv.data)
                + (WT == 0 ? ((size_t)row * p.W + k0) * 2 : ((size_t)row * p.W + k0) / 2);
            bulk_copy_g2s(w_s + r * seg, src, (uint32_t)seg, bar);
        }
    }
    if constexpr (WT == 1) {
        const int ng = KC >> p.down.gshift;
        for (int i = tid; i < nrows * ng; i += blockDim.x) {
            const int r = i / ng, gi = i % ng;
            const int gr = r0 + r;
            const WeightView &wv = gr < p.L ? p.down : p.inject;
            const int row = gr < p.L ? gr : gr - p.L;
            const size_t off = (size_t)row * (p.W >> wv.gshift) + (k0 >> wv.gshift) + gi;
            sb_s[2 * i] = half_bits_to_float(wv.scales[off]);
            sb_s[2 * i + 1] = half_bits_to_float(wv.biases[off]);
        }
    }

    // The residual is written by the previous kernel in the stream.
    pdl_wait();

    bool have_weights = false, timed_out = false;
    for (int t0 = 0; t0 < p.M; t0 += MT) {
        const int mt = min(MT, p.M - t0);

        // x = raw * g over this chunk, and the chunk's sum of squares.
        float ssq[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) ssq[t] = 0.f;
        for (int v = tid; v < KC / 8; v += blockDim.x) {
            float gf[8];
            unpack_bf16x8(*reinterpret_cast<const uint4 *>(p.g + k0 + v * 8), gf);
            const int p0 = xpos<VW>(v * 8), p1 = xpos<VW>(v * 8 + 4);
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                float rf[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (t < mt) {
                    unpack_bf16x8(*reinterpret_cast<const uint4 *>(p.raw + (size_t)(t0 + t) * p.raw_mstride +
                                                                    (size_t)(k0 / p.H) * p.raw_cstride + k0 % p.H +
                                                                    v * 8), rf);
                    if (p.inj_out)
                        inject_bf16x8(rf, p.inj_out + (size_t)(t0 + t) * p.H + k0 % p.H + v * 8,
                                      p.inj_gate[(size_t)(t0 + t) * p.inj_stride + k0 / p.H]);
                }
                float q = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) q = fmaf(rf[e], rf[e], q);
                ssq[t] += q;
                *reinterpret_cast<float4 *>(x_s + t * kcp + p0) =
                    make_float4(rf[0] * gf[0], rf[1] * gf[1], rf[2] * gf[2], rf[3] * gf[3]);
                *reinterpret_cast<float4 *>(x_s + t * kcp + p1) =
                    make_float4(rf[4] * gf[4], rf[5] * gf[5], rf[6] * gf[6], rf[7] * gf[7]);
            }
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            const float v = warp_sum(ssq[t]);
            if (lane == 0) red_s[warp * MT + t] = v;
        }
        __syncthreads();
        if (tid < MT) {
            float v = 0.f;
            for (int w = 0; w < nwarps; ++w) v += red_s[w * MT + tid];
            ssq_s[tid] = v;
        }
        if (!have_weights) {
            timed_out = !mbar_wait_bounded(bar, 0);
            if (timed_out)
                record_timeout(p.status);
            have_weights = true;
        }

        // Partial dots of this CTA's rows over its chunk.
        for (int r = warp; r < nrows; r += nwarps) {
            float acc[MT];
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[t] = 0.f;
            const uint4 *wrow = reinterpret_cast<const uint4 *>(w_s + r * seg);
            if constexpr (WT == 0)
                row_dot_bf16<MT>(wrow, nvec, x_s, kcp, lane, acc);
            else
                row_dot_int4<MT>(wrow, nvec, sb_s + 2 * r * (KC >> p.down.gshift), p.down.gshift, x_s, kcp,
                                 lane, acc);
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const float v = warp_sum(acc[t]);
                if (lane == 0) part_s[t * RPB + r] = v;
            }
        }

        cluster_sync();  // every rank's partials and sums of squares are complete

        // Remote (DSMEM) loads are all issued before any is used, so their
        // latencies overlap; the sums then run in rank order.
        if (tid < mt) {
            float ssr[kMaxCluster];
#pragma unroll
            for (int q = 0; q < kMaxCluster; ++q)
                ssr[q] = q < p.S ? dsmem_ld_f32(dsmem_addr(ssq_s + tid, q)) : 0.f;
            for (int c = 0; c < p.C; ++c) {
                float ss = 0.f;
#pragma unroll
                for (int q = 0; q < kMaxCluster; ++q)
                    if (q / p.sps == c && q < p.S) ss += ssr[q];
                invr_s[tid * p.C + c] = 1.0f / sqrtf(ss / (float)p.H + p.eps);
            }
        }
        __syncthreads();
        if (blockIdx.y == 0 && s == 0) {
            for (int i = tid; i < mt * p.C; i += blockDim.x)
                p.inv_rms[(size_t)t0 * p.C + i] = invr_s[i];
        }

        // Rank s finishes rows s, s+S, ... of the block.
        const int my_rows = s < nrows ? (nrows - s + p.S - 1) / p.S : 0;
        for (int i = tid; i < my_rows * mt; i += blockDim.x) {
            const int r = s + p.S * (i / mt), t = i % mt;
            float pv[kMaxCluster];
#pragma unroll
            for (int q = 0; q < kMaxCluster; ++q)
                pv[q] = q < p.S ? dsmem_ld_f32(dsmem_addr(part_s + t * RPB + r, q)) : 0.f;
            float z = 0.f;
#pragma unroll
            for (int q = 0; q < kMaxCluster; ++q)
                if (q < p.S) z = fmaf(invr_s[t * p.C + q / p.sps], pv[q], z);
            const int gr = r0 + r;
            const int m = t0 + t;
            const float zc = z * p.inv_C;
            if (gr < p.L)
                p.act[(size_t)m * p.L + gr] = zc * sigmoidf_(zc);
            else
                p.gate[(size_t)m * p.gate_stride + (gr - p.L)] = 2.0f * sigmoidf_(zc);
        }

        cluster_sync();  // peers have read this CTA's partials before they are overwritten
    }
    if (timed_out)  // do not leave with a copy into this CTA's shared memory in flight
        mbar_wait_bounded(bar, 0);
}

template <int WT, int MT>
__global__ void __launch_bounds__(768, 1) hc_up_kernel(const UpParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const UpSmem lay = up_layout(p, MT);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + lay.bar);
    unsigned char *w_s = smem + lay.w;
    float *sb_s = reinterpret_cast<float *>(smem + lay.sb);
    float *act_s = reinterpret_cast<float *>(smem + lay.act);
    float *wv_s = reinterpret_cast<float *>(smem + lay.wv);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int HB = p.HB, h0 = blockIdx.x * HB;
    const int hb = min(HB, p.H - h0);
    const int L = p.L;
    const size_t row_bytes = WT == 0 ? (size_t)L * 2 : (size_t)L / 2;
    const int ng = WT == 0 ? 0 : L >> p.up.gshift;

    pdl_launch_dependents();

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(bar, (uint32_t)(row_bytes * hb * p.C));
        for (int c = 0; c < p.C; ++c)
            bulk_copy_g2s(w_s + (size_t)c * HB * row_bytes,
                          static_cast<const unsigned char *>(p.up.data) + ((size_t)c * p.H + h0) * row_bytes,
                          (uint32_t)(row_bytes * hb), bar);
    }
    if constexpr (WT == 1) {
        for (int i = tid; i < p.C * hb * ng; i += blockDim.x) {
            const int c = i / (hb * ng), rem = i % (hb * ng), hl = rem / ng, gi = rem % ng;
            const size_t off = ((size_t)c * p.H + h0 + hl) * ng + gi;
            const int srow = c * HB + hl;
            sb_s[2 * (srow * ng + gi)] = half_bits_to_float(p.up.scales[off]);
            sb_s[2 * (srow * ng + gi) + 1] = half_bits_to_float(p.up.biases[off]);
        }
    }

    const int team = lane >> 3, tl = lane & 7;  // 8 lanes per up row
    bool have_weights = false, timed_out = false;
    float *rv_s = reinterpret_cast<float *>(smem + lay.rv);
    float *gv_s = reinterpret_cast<float *>(smem + lay.gv);
    float *inv_s = reinterpret_cast<float *>(smem + lay.inv);
    // g is a weight: staged before the dependency wait.
    for (int i = tid; i < p.C * HB; i += blockDim.x) {
        const int c = i / HB, hl = i % HB;
        gv_s[i] = hl < hb ? __bfloat162float(__ushort_as_bfloat16(p.g[c * p.H + h0 + hl])) : 0.f;
    }

    // act and inv_rms come from the down kernel; raw from the kernel before it.
    pdl_wait();

    for (int t0 = 0; t0 < p.M; t0 += MT) {
        const int mt = min(MT, p.M - t0);
        // Everything the tile needs is loaded in one round: act, inv_rms and
        // the residual of this CTA's h-block (with a fused inject-add applied
        // and written back here -- this CTA owns these elements).
        for (int i = tid; i < MT * L; i += blockDim.x) {
            const int t = i / L, k = i % L;
            act_s[i] = t < mt ? p.act[(size_t)(t0 + t) * L + k] : 0.f;
        }
        for (int i = tid; i < MT * p.C; i += blockDim.x)
            inv_s[i] = i / p.C < mt ? p.inv_rms[(size_t)t0 * p.C + i] : 0.f;
        for (int i = tid; i < MT * p.C * HB; i += blockDim.x) {
            const int t = i / (p.C * HB), c = (i / HB) % p.C, hl = i % HB;
            float rv = 0.f;
            if (t < mt && hl < hb) {
                const size_t m = (size_t)(t0 + t);
                const int h = h0 + hl, j = c * p.H + h;
                rv = __bfloat162float(__ushort_as_bfloat16(p.raw[m * p.raw_mstride + (size_t)c * p.raw_cstride + h]));
                if (p.inj_out) {
                    const float ov = __bfloat162float(__ushort_as_bfloat16(p.inj_out[m * p.H + h]));
                    rv = __bfloat162float(__float2bfloat16_rn(fmaf(ov, p.inj_gate[m * p.inj_stride + c], rv)));
                }
                if (p.raw_out)
                    p.raw_out[m * p.W + j] = __bfloat16_as_ushort(__float2bfloat16_rn(rv));
            }
            rv_s[i] = rv;
        }
        __syncthreads();
        if (!have_weights) {
            timed_out = !mbar_wait_bounded(bar, 0);
            if (timed_out)
                record_timeout(p.status);
            have_weights = true;
        }

        // The loop bound is uniform across the warp (every lane reaches the
        // full-warp shuffles below); teams past the last row compute nothing.
        for (int base = warp * 4; base < p.C * hb; base += nwarps * 4) {
            const int rr = base + team;
            const bool row_ok = rr < p.C * hb;
            const int c = row_ok ? rr / hb : 0, hl = row_ok ? rr % hb : 0;
            const int srow = c * HB + hl;
            const uint4 *wrow = reinterpret_cast<const uint4 *>(w_s + srow * row_bytes);
            float acc[MT];
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[t] = 0.f;
            if (!row_ok) {
                // no row for this team
            } else if constexpr (WT == 0) {
                float a1[MT];  // second chain (odd elements), added at the end
#pragma unroll
                for (int t = 0; t < MT; ++t) a1[t] = 0.f;
#pragma unroll 2
                for (int v = tl; v < L / 8; v += 8) {
                    float wf[8];
                    unpack_bf16x8(wrow[v], wf);
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const float4 xa = *reinterpret_cast<const float4 *>(act_s + t * L + v * 8);
                        const float4 xb = *reinterpret_cast<const float4 *>(act_s + t * L + v * 8 + 4);
                        acc[t] = fmaf(wf[0], xa.x, acc[t]); a1[t] = fmaf(wf[1], xa.y, a1[t]);
                        acc[t] = fmaf(wf[2], xa.z, acc[t]); a1[t] = fmaf(wf[3], xa.w, a1[t]);
                        acc[t] = fmaf(wf[4], xb.x, acc[t]); a1[t] = fmaf(wf[5], xb.y, a1[t]);
                        acc[t] = fmaf(wf[6], xb.z, acc[t]); a1[t] = fmaf(wf[7], xb.w, a1[t]);
                    }
                }
#pragma unroll
                for (int t = 0; t < MT; ++t) acc[t] += a1[t];
            } else {
                // Lane tl of the team owns the 4-byte words (8 codes) w = tl + 8 i
                // of the row: the team reads 32 contiguous bytes of codes and act
                // rows 32 bytes apart per lane (no 128-byte-stride bank conflicts).
                const float *sb = sb_s + 2 * srow * ng;
                const uint32_t *wrow32 = reinterpret_cast<const uint32_t *>(wrow);
                for (int w = tl; w < L / 8; w += 8) {
                    const uint32_t codes = wrow32[w];
                    const int gi = (w * 8) >> p.up.gshift;
                    const float sc = sb[2 * gi], bi = sb[2 * gi + 1];
                    float wf[8];
#pragma unroll
                    for (int n = 0; n < 8; ++n)
                        wf[n] = fmaf((float)((codes >> (4 * n)) & 0xFu), sc, bi);
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const float *xr = act_s + t * L + w * 8;
                        const float4 xa = *reinterpret_cast<const float4 *>(xr);
                        const float4 xb = *reinterpret_cast<const float4 *>(xr + 4);
                        float a = acc[t];
                        a = fmaf(wf[0], xa.x, a); a = fmaf(wf[1], xa.y, a);
                        a = fmaf(wf[2], xa.z, a); a = fmaf(wf[3], xa.w, a);
                        a = fmaf(wf[4], xb.x, a); a = fmaf(wf[5], xb.y, a);
                        a = fmaf(wf[6], xb.z, a); a = fmaf(wf[7], xb.w, a);
                        acc[t] = a;
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                float v = acc[t];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                if (tl == 0 && row_ok) {
                    const float w = sigmoidf_(v);
                    wv_s[(t * p.C + c) * HB + hl] = w;
                    if (p.w_out && t < mt)  // debug output of w
                        p.w_out[(size_t)(t0 + t) * p.W + (size_t)c * p.H + h0 + hl] = w;
                }
            }
        }
        __syncthreads();

        for (int i = tid; i < mt * hb; i += blockDim.x) {
            const int t = i / hb, hl = i % hb;
            const int h = h0 + hl;
            const size_t m = (size_t)(t0 + t);
            float acc = 0.f;
            for (int c = 0; c < p.C; ++c) {
                const float nv = rv_s[(t * p.C + c) * HB + hl] * inv_s[t * p.C + c] * gv_s[c * HB + hl];
                acc = fmaf(wv_s[(t * p.C + c) * HB + hl], nv, acc);
            }
            p.mixed[m * p.H + h] = __bfloat16_as_ushort(__float2bfloat16_rn(acc * p.inv_C));
        }
        __syncthreads();
    }
    if (timed_out)  // do not leave with a copy into this CTA's shared memory in flight
        mbar_wait_bounded(bar, 0);
}

// ---- one token (M == 1): two kernels, no cluster, no cross-CTA wait ---------
//
// hc_down1_kernel  Grid (S, row blocks): CTA (s, rb) owns rows [rb*RPB, ...)
//                  over input chunk s (which lies inside stream s / sps).
//                  Before the dependency wait, warp 0 streams the block's
//                  weight row segments and the chunk of g into shared memory
//                  (one bulk copy per lane). Thread v of a group owns the
//                  chunk's inputs [8v, 8v + 8): after the wait it reads them
//                  once (applying a fused inject-add), keeps x = raw * g in
//                  registers and forms their dot with each of its group's rows
//                  (the block's rows are split evenly over G groups of
//                  threads). Partial sums leave the warp by a transposed
//                  butterfly and meet across warps in shared memory; the
//                  block writes part1[s][r] and (row block 0) the chunk's sum
//                  of squares ssq1[s].
// hc_up1_kernel    Every CTA forms inv_rms, z = sum_s inv_rms[stream(s)] * P_s
//                  and silu(z / C) for all rows from the partials in a fixed
//                  order (CTA 0 also writes act, inv_rms and the gates out).
//                  Warp w owns h = h0 + w and dots act with the C up rows
//                  {c*H + h}. bf16: lane l owns the act pairs l + 32i of every
//                  row. INT4: lane l owns the 8-input code words l + 32i of
//                  every row, or, with C = 4 compiled in, the words l/4 + 8i
//                  of row l & 3. Lane 4c then holds row c (after the transposed
//                  butterfly, or one shuffle), applies the sigmoid and its term
//                  of the mean mix, and lane 0 writes mixed[h]. With a fused
//                  inject-add, lane 4c also writes the updated residual
//                  element back.

// Sums v[0..7] over the 32 lanes of a warp. On return lane l holds the total
// of v[(l >> 2) & 7]. Every lane must take part; the order is fixed.
__device__ __forceinline__ float warp_transpose_sum8(float (&v)[8], int lane)
{
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // v[i] -> value 4*b4 + i
        const float send = b4 ? v[i] : v[i + 4];
        const float keep = b4 ? v[i + 4] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {  // v[i] -> value 4*b4 + 2*b3 + i
        const float send = b3 ? v[i] : v[i + 2];
        const float keep = b3 ? v[i + 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const float send = b2 ? v[0] : v[1];
    const float keep = b2 ? v[1] : v[0];
    float r = keep + __shfl_xor_sync(0xffffffffu, send, 4);  // value 4*b4 + 2*b3 + b2
    r += __shfl_xor_sync(0xffffffffu, r, 2);
    r += __shfl_xor_sync(0xffffffffu, r, 1);
    return r;
}

constexpr int kRowsPerGroup = 8;  // rows one thread of hc_down1_kernel dots

struct Down1Smem {
    size_t bar, w, g, red, total;
};

__host__ __device__ inline Down1Smem down1_layout(const DownParams &p)
{
    const size_t seg = p.down.type == 0 ? (size_t)p.KC * 2 : (size_t)p.KC / 2;
    Down1Smem s;
    s.bar = 0;
    s.w = 128;
    s.g = round_up_sz(s.w + seg * p.rows_per_block, 128);
    s.red = round_up_sz(s.g + (size_t)p.KC * 2, 128);
    s.total = round_up_sz(s.red + sizeof(float) * 32 * (kRowsPerGroup + 1), 128);
    return s;
}

// Threads of one group of hc_down1_kernel: one per 8 inputs of the chunk.
__host__ __device__ inline int down1_group_threads(const DownParams &p) { return round_up(p.KC / 8, 32); }
// Groups (the block's rows split evenly, at most kRowsPerGroup each).
__host__ __device__ inline int down1_groups(const DownParams &p)
{
    return (p.rows_per_block + kRowsPerGroup - 1) / kRowsPerGroup;
}

template <int WT>
__global__ void __launch_bounds__(1024, 1) hc_down1_kernel(const DownParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const Down1Smem lay = down1_layout(p);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + lay.bar);
    const unsigned char *w_s = smem + lay.w;
    const uint16_t *g_s = reinterpret_cast<const uint16_t *>(smem + lay.g);
    float *red_s = reinterpret_cast<float *>(smem + lay.red);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = blockIdx.x;
    const int r0 = blockIdx.y * p.rows_per_block;
    const int nrows = min(p.rows_per_block, p.R - r0);
    const int KC = p.KC, k0 = s * KC, nv = KC / 8;
    const size_t seg = WT == 0 ? (size_t)KC * 2 : (size_t)KC / 2;
    const int tpg = down1_group_threads(p), wpg = tpg / 32;
    const int ngroups = blockDim.x / tpg;
    const int rpg = (nrows + ngroups - 1) / ngroups;  // rows per group (<= kRowsPerGroup)
    const int grp = tid / tpg, v = tid % tpg;
    const int gr0 = grp * rpg, gnr = max(0, min(rpg, nrows - gr0));

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0)
            mbar_arrive_expect_tx(bar, (uint32_t)(seg * nrows + (size_t)KC * 2));
        __syncwarp();
        for (int j = lane; j <= nrows; j += 32) {
            if (j == nrows) {
                bulk_copy_g2s(smem + lay.g, p.g + k0, (uint32_t)KC * 2, bar);
            } else {
                const int gr = r0 + j;
                const WeightView &wv = gr < p.L ? p.down : p.inject;
                const int row = gr < p.L ? gr : gr - p.L;
                const unsigned char *src = static_cast<const unsigned char *>(wv.data)
                    + (WT == 0 ? ((size_t)row * p.W + k0) * 2 : ((size_t)row * p.W + k0) / 2);
                bulk_copy_g2s(smem + lay.w + j * seg, src, (uint32_t)seg, bar);
            }
        }
    }
    // INT4: this thread's 8 inputs share one (scale, bias) group of every row, so
    // it loads one scale and one bias per row of its group now, into registers;
    // they are used after the dots, so nothing waits for them here.
    uint16_t sc_r[kRowsPerGroup], bi_r[kRowsPerGroup];
    if constexpr (WT == 1) {
        const int gi = (v * 8) >> p.down.gshift;
#pragma unroll
        for (int j = 0; j < kRowsPerGroup; ++j) {
            sc_r[j] = 0;
            bi_r[j] = 0;
            if (v < nv && j < gnr) {
                const int gr = r0 + gr0 + j;
                const WeightView &wv = gr < p.L ? p.down : p.inject;
                const int row = gr < p.L ? gr : gr - p.L;
                const size_t off = (size_t)row * (p.W >> wv.gshift) + (k0 >> wv.gshift) + gi;
                sc_r[j] = wv.scales[off];
                bi_r[j] = wv.biases[off];
            }
        }
    }

    pdl_wait();  // the residual and the previous gates come from earlier kernels

    const bool has_v = v < nv;
    uint4 rvv = make_uint4(0, 0, 0, 0), ovv = make_uint4(0, 0, 0, 0);
    float gt = 0.f;
    if (has_v) {
        rvv = *reinterpret_cast<const uint4 *>(p.raw + (size_t)(k0 / p.H) * p.raw_cstride + k0 % p.H + v * 8);
        if (p.inj_out) {
            ovv = *reinterpret_cast<const uint4 *>(p.inj_out + k0 % p.H + v * 8);
            gt = p.inj_gate[k0 / p.H];
        }
    }
    // Only now let the up kernel launch: (1) it reads the residual and the
    // previous gates before its own dependency wait, which is safe once every
    // CTA of this kernel has passed its wait (everything earlier in the
    // stream has completed); (2) its weight stream, which starts about a
    // microsecond later, then no longer competes with these residual loads.
    pdl_launch_dependents();
    const bool timed_out = !mbar_wait_bounded(bar, 0);
    if (timed_out)
        record_timeout(p.status);

    float x[8], q = 0.f;
    {
        float rf[8], gf[8];
        unpack_bf16x8(rvv, rf);
        if (p.inj_out) {
            float of[8];
            unpack_bf16x8(ovv, of);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                rf[e] = __bfloat162float(__float2bfloat16_rn(fmaf(of[e], gt, rf[e])));
        }
        unpack_bf16x8(has_v ? *reinterpret_cast<const uint4 *>(g_s + v * 8) : make_uint4(0, 0, 0, 0), gf);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            q = fmaf(rf[e], rf[e], q);
            x[e] = rf[e] * gf[e];
        }
    }

    // Even and odd inputs accumulate in the two lanes of a packed fp32 pair.
    uint64_t xp[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        xp[e] = f32x2(x[2 * e], x[2 * e + 1]);
    float xsum = 0.f;  // INT4: the group's bias multiplies the sum of the inputs
    if constexpr (WT == 1) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            xsum += x[e];
    }
    float acc[kRowsPerGroup];
#pragma unroll
    for (int j = 0; j < kRowsPerGroup; ++j) {
        acc[j] = 0.f;
        if (has_v && j < gnr) {
            const unsigned char *wr = w_s + (size_t)(gr0 + j) * seg;
            uint64_t a = 0;
            if constexpr (WT == 0) {
                const uint4 wq = *reinterpret_cast<const uint4 *>(wr + v * 16);
                a = ffma2(bf16x2_as_f32x2(wq.x), xp[0], a);
                a = ffma2(bf16x2_as_f32x2(wq.y), xp[1], a);
                a = ffma2(bf16x2_as_f32x2(wq.z), xp[2], a);
                a = ffma2(bf16x2_as_f32x2(wq.w), xp[3], a);
            } else {
                // The thread's 8 inputs share one (scale, bias) group:
                // sum (q s + b) x = s * sum q x + b * sum x.
                const uint32_t codes = *reinterpret_cast<const uint32_t *>(wr + v * 4);
                const uint32_t nlo = int4_lo_nibbles(codes), nhi = int4_hi_nibbles(codes);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    a = ffma2(int4_pair_f32x2(nlo, nhi, e), xp[e], a);
                a = f32x2(fmaf(half_bits_to_float(sc_r[j]), f32x2_sum(a), half_bits_to_float(bi_r[j]) * xsum), 0.f);
            }
            acc[j] = f32x2_sum(a);
        }
    }
    const float rsum = warp_transpose_sum8(acc, lane);
    if ((lane & 3) == 0)
        red_s[warp * (kRowsPerGroup + 1) + (lane >> 2)] = rsum;
    q = warp_sum(q);
    if (lane == 0)
        red_s[warp * (kRowsPerGroup + 1) + kRowsPerGroup] = q;
    __syncthreads();

    if (tid < nrows) {  // row tid of the block, in group tid / rpg
        const int g = tid / rpg, j = tid % rpg;
        float t = 0.f;
        for (int w = 0; w < wpg; ++w)
            t += red_s[(g * wpg + w) * (kRowsPerGroup + 1) + j];
#pragma unroll
        for (int c = 0; c < kPartCopies; ++c)
            p.part1[c * p.part1_stride + (size_t)s * p.R + r0 + tid] = t;
    }
    if (blockIdx.y == 0 && tid == blockDim.x - 1) {  // every group saw the same inputs: use group 0
        float t = 0.f;
        for (int w = 0; w < wpg; ++w)
            t += red_s[w * (kRowsPerGroup + 1) + kRowsPerGroup];
#pragma unroll
        for (int c = 0; c < kPartCopies; ++c)
            p.ssq1[c * kSsqStride + s] = t;
    }
    if (timed_out)  // do not leave with a copy into this CTA's shared memory in flight
        mbar_wait_bounded(bar, 0);
}

struct Up1Smem {
    size_t bar, w, sb, act, asum, ssq, invq, inv, total;
};

__host__ __device__ inline Up1Smem up1_layout(const UpParams &p)
{
    const size_t row = p.up.type == 0 ? (size_t)p.L * 2 : (size_t)p.L / 2;
    const int ng = p.up.type == 0 ? 0 : p.L >> p.up.gshift;
    Up1Smem s;
    s.bar = 0;
    s.w = 128;
    s.sb = round_up_sz(s.w + row * p.C * p.HB, 128);
    s.act = round_up_sz(s.sb + sizeof(float) * 2 * (size_t)ng * p.C * p.HB, 128);
    s.asum = round_up_sz(s.act + sizeof(float) * (size_t)p.L, 128);
    s.ssq = round_up_sz(s.asum + sizeof(float) * (size_t)(p.up.type == 0 ? 0 : p.L / 8), 128);
    s.invq = round_up_sz(s.ssq + sizeof(float) * kMaxCluster, 16);
    s.inv = round_up_sz(s.invq + sizeof(float) * kMaxCluster, 16);
    s.total = round_up_sz(s.inv + sizeof(float) * kMaxCluster, 128);
    return s;
}

// CC: the stream count when it is a compile-time constant (4), else 0.
template <int WT, int CC, bool PF>
__global__ void __launch_bounds__(1024, 1) hc_up1_kernel(const UpParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const Up1Smem lay = up1_layout(p);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + lay.bar);
    const unsigned char *w_s = smem + lay.w;
    float *sb_s = reinterpret_cast<float *>(smem + lay.sb);
    float *act_s = reinterpret_cast<float *>(smem + lay.act);
    float *asum_s = reinterpret_cast<float *>(smem + lay.asum);  // INT4: act summed over each 8-input word
    float *ssq_s = reinterpret_cast<float *>(smem + lay.ssq);    // sum of squares of chunk q
    float *invq_s = reinterpret_cast<float *>(smem + lay.invq);  // inv_rms of chunk q's stream
    float *inv_s = reinterpret_cast<float *>(smem + lay.inv);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int HB = p.HB, h0 = blockIdx.x * HB;
    const int hb = min(HB, p.H - h0);
    const int L = p.L;
    const size_t row_bytes = WT == 0 ? (size_t)L * 2 : (size_t)L / 2;
    const int ng = WT == 0 ? 1 : L >> p.up.gshift;

    // Thread 0 initialises the barrier and issues the weight copies at once;
    // no other thread touches the barrier before the first block-wide
    // barrier below.
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
        mbar_arrive_expect_tx(bar, (uint32_t)(row_bytes * hb * p.C));
        for (int c = 0; c < p.C; ++c)
            bulk_copy_g2s(smem + lay.w + (size_t)c * HB * row_bytes,
                          static_cast<const unsigned char *>(p.up.data) + ((size_t)c * p.H + h0) * row_bytes,
                          (uint32_t)(row_bytes * hb), bar);
    }
    if constexpr (PF) {  // the next kernel's weights, after this CTA's own (a separate instance:
        if (warp == 1)    // the branch alone slowed the one-token call by 0.1 us)
            prefetch_share_l2(p.l2_pf, p.l2_pf_bytes, lane, 32);
    }
    if constexpr (WT == 1) {
        for (int i = tid; i < p.C * hb * ng; i += blockDim.x) {
            const int c = i / (hb * ng), rem = i % (hb * ng), hl = rem / ng, gi = rem % ng;
            const size_t off = ((size_t)c * p.H + h0 + hl) * ng + gi;
            const int srow = c * HB + hl;
            sb_s[2 * (srow * ng + gi)] = half_bits_to_float(p.up.scales[off]);
            sb_s[2 * (srow * ng + gi) + 1] = half_bits_to_float(p.up.biases[off]);
        }
    }

    // Warp w owns h = h0 + w (the host launches at least hb warps); lane 4c
    // holds stream c's up row after the butterfly.
    const int hl = warp, h = h0 + hl;
    const bool h_ok = hl < hb;
    const int hc = lane >> 2;
    const bool holder = h_ok && (lane & 3) == 0 && hc < p.C;
    // Read before the dependency wait: g (a weight), and this lane's residual
    // element with the previous gate -- the down kernel lets this kernel
    // launch only after all its CTAs passed their own wait, so these are
    // final; they are read from L2 (.cg). The residual is written back only
    // after the wait, when the down kernel has finished reading it.
    float gval = 0.f, rv = 0.f, ov = 0.f, gp = 0.f;
    if (holder) {
        gval = __bfloat162float(__ushort_as_bfloat16(p.g[hc * p.H + h]));
        rv = __bfloat162float(__ushort_as_bfloat16(__ldcg(p.raw + (size_t)hc * p.raw_cstride + h)));
        if (p.inj_out) {
            ov = __bfloat162float(__ushort_as_bfloat16(__ldcg(p.inj_out + h)));
            gp = __ldcg(p.inj_gate + hc);
        }
    }

    pdl_wait();  // the partials come from the down kernel

    // One round of loads: partials (thread k owns down row k) and the chunks'
    // sums of squares (thread q < S owns chunk q).
    const int k = tid;  // the host launches at least R threads
    const int copy = blockIdx.x % kPartCopies;
    const float *part = p.part1 + copy * p.part1_stride;
    const float *ssq = p.ssq1 + copy * kSsqStride;
    float pv[kMaxCluster];
#pragma unroll
    for (int q = 0; q < kMaxCluster; ++q)
        pv[q] = (k < p.R && q < p.S) ? part[(size_t)q * p.R + k] : 0.f;
    const float sq = tid < p.S ? ssq[tid] : 0.f;
    // The next kernel's weight stream starts about a microsecond after this
    // trigger, once these loads are on their way.
    pdl_launch_dependents();
    if (tid < p.S)
        ssq_s[tid] = sq;
    __syncthreads();
    if (tid < p.S) {  // chunk q = tid: inv_rms of its stream (the stream's chunks in order)
        const int c = tid / p.sps;
        float t = 0.f;
        for (int j = 0; j < p.sps; ++j)
            t += ssq_s[c * p.sps + j];
        const float iv = rsqrtf(fmaf(t, p.inv_H, p.eps));
        invq_s[tid] = iv;
        if (tid % p.sps == 0) {
            inv_s[c] = iv;
            if (blockIdx.x == 0)
                p.inv_out[c] = iv;
        }
    }
    __syncthreads();
    float a_k = 0.f;  // act[k], 0 past L
    if (k < p.R) {
        float z = 0.f;
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q)
            if (q < p.S) z = fmaf(invq_s[q], pv[q], z);
        const float zc = z * p.inv_C;
        if (k < L) {
            const float a = zc * sigmoid_fast(zc);
            act_s[k] = a;
            a_k = a;
            if (blockIdx.x == 0)
                p.act_out[k] = a;
        } else if (blockIdx.x == 0 && p.gate) {
            p.gate[k - L] = 2.0f * sigmoid_fast(zc);
        }
    }
    if constexpr (WT == 1) {
        // The sum of each 8-input word's act values, which the dots multiply by the
        // group's bias: lanes 8w .. 8w+7 of a warp hold act[8w .. 8w+7] (L is a
        // multiple of 8), summed as ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7)).
        float t = a_k;
        t += __shfl_xor_sync(0xffffffffu, t, 1);
        t += __shfl_xor_sync(0xffffffffu, t, 2);
        t += __shfl_xor_sync(0xffffffffu, t, 4);
        if ((k & 7) == 0 && k < L)
            asum_s[k >> 3] = t;
    }
    const bool timed_out = !mbar_wait_bounded(bar, 0);
    if (timed_out)
        record_timeout(p.status);
    __syncthreads();

    // This lane's residual element (with the fused inject-add written back)
    // and its normed value, ready before the dots.
    float nvh = 0.f;
    if (holder) {
        if (p.inj_out)
            rv = __bfloat162float(__float2bfloat16_rn(fmaf(ov, gp, rv)));
        if (p.raw_out)
            p.raw_out[hc * p.H + h] = __bfloat16_as_ushort(__float2bfloat16_rn(rv));
        nvh = rv * inv_s[hc] * gval;
    }

    if (h_ok) {  // warp-uniform
        float acc[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = 0.f;
        if constexpr (WT == 0) {
            // Lane owns the bf16 pairs j = lane + 32 i of each of the C rows (the
            // lanes stay balanced for any L); the act pair is read once per j.
            constexpr int NC = CC > 0 ? CC : 8;
            uint64_t a2[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) a2[c] = 0;
            const uint32_t *wr = reinterpret_cast<const uint32_t *>(w_s) + (size_t)hl * (L / 2);
            const size_t cstride = (size_t)HB * (L / 2);  // words between streams' rows
#pragma unroll 2
            for (int j = lane; j < L / 2; j += 32) {
                const uint64_t xpair = *reinterpret_cast<const uint64_t *>(act_s + 2 * j);
#pragma unroll
                for (int c = 0; c < NC; ++c)
                    if (CC > 0 || c < p.C)
                        a2[c] = ffma2(bf16x2_as_f32x2(wr[c * cstride + j]), xpair, a2[c]);
            }
#pragma unroll
            for (int c = 0; c < NC; ++c) acc[c] = f32x2_sum(a2[c]);
        } else if constexpr (CC == 4) {
            // Lane owns stream c = lane & 3 and the code words v = lane / 4 + 8 i
            // of that row, so every lane handles the same number of words. The
            // word's 8 act values share one (scale, bias) group of the row:
            // sum (q s + b) a = s * sum q a + b * sum a.
            const int c = lane & 3;
            const int srow = c * HB + hl;
            const uint32_t *wr = reinterpret_cast<const uint32_t *>(w_s + (size_t)srow * row_bytes);
            const float *sbr = sb_s + 2 * (size_t)srow * ng;
            float a = 0.f;
#pragma unroll 5
            for (int v = lane >> 2; v < L / 8; v += 8) {
                const float4 xa = *reinterpret_cast<const float4 *>(act_s + v * 8);
                const float4 xb = *reinterpret_cast<const float4 *>(act_s + v * 8 + 4);
                const uint64_t ap[4] = {f32x2(xa.x, xa.y), f32x2(xa.z, xa.w), f32x2(xb.x, xb.y), f32x2(xb.z, xb.w)};
                const float asum = asum_s[v];
                const uint32_t codes = wr[v];
                const uint32_t nlo = int4_lo_nibbles(codes), nhi = int4_hi_nibbles(codes);
                const float *sb = sbr + 2 * ((v * 8) >> p.up.gshift);
                uint64_t dq = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dq = ffma2(int4_pair_f32x2(nlo, nhi, e), ap[e], dq);
                a += fmaf(sb[0], f32x2_sum(dq), sb[1] * asum);
            }
            // Lanes with equal lane & 3 hold parts of the same row.
            a += __shfl_xor_sync(0xffffffffu, a, 4);
            a += __shfl_xor_sync(0xffffffffu, a, 8);
            a += __shfl_xor_sync(0xffffffffu, a, 16);
            acc[0] = a;
        } else {
            for (int v = lane; v < L / 8; v += 32) {
                // The word's 8 act values share one (scale, bias) group of every
                // row: sum (q s + b) a = s * sum q a + b * sum a.
                const float4 xa = *reinterpret_cast<const float4 *>(act_s + v * 8);
                const float4 xb = *reinterpret_cast<const float4 *>(act_s + v * 8 + 4);
                const uint64_t ap[4] = {f32x2(xa.x, xa.y), f32x2(xa.z, xa.w), f32x2(xb.x, xb.y), f32x2(xb.z, xb.w)};
                const float asum = ((xa.x + xa.y) + (xa.z + xa.w)) + ((xb.x + xb.y) + (xb.z + xb.w));
                const int gi = (v * 8) >> p.up.gshift;
                constexpr int NC = CC > 0 ? CC : 8;
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    if (CC > 0 || c < p.C) {
                        const int srow = c * HB + hl;
                        const uint32_t codes =
                            *reinterpret_cast<const uint32_t *>(w_s + (size_t)srow * row_bytes + v * 4);
                        const uint32_t nlo = int4_lo_nibbles(codes), nhi = int4_hi_nibbles(codes);
                        const float *sb = sb_s + 2 * (srow * ng + gi);
                        uint64_t dq = 0;
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dq = ffma2(int4_pair_f32x2(nlo, nhi, e), ap[e], dq);
                        acc[c] += fmaf(sb[0], f32x2_sum(dq), sb[1] * asum);
                    }
                }
            }
        }
        // Lane 4c takes row c's total: from lane c in the INT4 four-stream
        // layout, else from the transposed butterfly.
        float d;
        if constexpr (WT == 1 && CC == 4)
            d = __shfl_sync(0xffffffffu, acc[0], (lane >> 2) & 3);
        else
            d = warp_transpose_sum8(acc, lane);
        const float wv = sigmoid_fast(d);
        if (p.w_out && holder)  // debug output of w
            p.w_out[hc * p.H + h] = wv;
        float term = holder ? wv * nvh : 0.f;
        term += __shfl_xor_sync(0xffffffffu, term, 4);
        term += __shfl_xor_sync(0xffffffffu, term, 8);
        term += __shfl_xor_sync(0xffffffffu, term, 16);
        if (lane == 0)
            p.mixed[h] = __bfloat16_as_ushort(__float2bfloat16_rn(term * p.inv_C));
    }
    if (timed_out)  // do not leave with a copy into this CTA's shared memory in flight
        mbar_wait_bounded(bar, 0);
}

// ---- few tokens (2 <= M <= kFewMaxTokens), bf16 weights -----------------------
//
// The one-token kernels' layout with the token loop inside: the down kernel
// streams its weight rows once and dots them with every token's chunk; the up
// kernel reduces every token's partials and loops over the tokens in its dots
// and mix. Two kernels per call, as at one token, in place of the tensor-core
// path's four. Partials: token m of chunk s at part1[copy][s][m][row], its sum of
// squares at ssq1[copy][s * M + m].

struct DownmSmem {
    size_t bar, w, g, red, total;
};

__host__ __device__ inline DownmSmem downm_layout(const DownParams &p, int nwarps)
{
    DownmSmem s;
    s.bar = 0;
    s.w = 128;
    s.g = round_up_sz(s.w + (size_t)p.KC * 2 * p.rows_per_block, 128);
    s.red = round_up_sz(s.g + (size_t)p.KC * 2, 128);
    s.total = round_up_sz(s.red + sizeof(float) * (size_t)nwarps * p.M * (kRowsPerGroup + 1), 128);
    return s;
}

__global__ void __launch_bounds__(1024, 1) hc_downm_kernel(const DownParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const int nwarps = blockDim.x >> 5;
    const DownmSmem lay = downm_layout(p, nwarps);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + lay.bar);
    const unsigned char *w_s = smem + lay.w;
    const uint16_t *g_s = reinterpret_cast<const uint16_t *>(smem + lay.g);
    float *red_s = reinterpret_cast<float *>(smem + lay.red);  // [warp][token][kRowsPerGroup + 1]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = blockIdx.x;
    const int r0 = blockIdx.y * p.rows_per_block;
    const int nrows = min(p.rows_per_block, p.R - r0);
    const int KC = p.KC, k0 = s * KC, nv = KC / 8, M = p.M;
    const size_t seg = (size_t)KC * 2;
    const int tpg = down1_group_threads(p), wpg = tpg / 32;
    const int ngroups = blockDim.x / tpg;
    const int rpg = (nrows + ngroups - 1) / ngroups;
    const int grp = tid / tpg, v = tid % tpg;
    const int gr0 = grp * rpg, gnr = max(0, min(rpg, nrows - gr0));

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0)
            mbar_arrive_expect_tx(bar, (uint32_t)(seg * nrows + (size_t)KC * 2));
        __syncwarp();
        for (int j = lane; j <= nrows; j += 32) {
            if (j == nrows) {
                bulk_copy_g2s(smem + lay.g, p.g + k0, (uint32_t)KC * 2, bar);
            } else {
                const int gr = r0 + j;
                const uint16_t *src = gr < p.L ? static_cast<const uint16_t *>(p.down.data) + (size_t)gr * p.W
                                               : static_cast<const uint16_t *>(p.inject.data) + (size_t)(gr - p.L) * p.W;
                bulk_copy_g2s(smem + lay.w + j * seg, src + k0, (uint32_t)seg, bar);
            }
        }
    }

    pdl_wait();  // the residual and the previous gates come from earlier kernels

    const bool has_v = v < nv;
    const long roff = (long)(k0 / p.H) * p.raw_cstride + k0 % p.H + v * 8;
    auto load_tok = [&](int t, uint4 &rv, uint4 &ov, float &gt) {
        rv = make_uint4(0, 0, 0, 0);
        ov = make_uint4(0, 0, 0, 0);
        gt = 0.f;
        if (has_v && t < M) {
            rv = *reinterpret_cast<const uint4 *>(p.raw + (size_t)t * p.raw_mstride + roff);
            if (p.inj_out) {
                ov = *reinterpret_cast<const uint4 *>(p.inj_out + (size_t)t * p.H + k0 % p.H + v * 8);
                gt = p.inj_gate[(size_t)t * p.inj_stride + k0 / p.H];
            }
        }
    };
    uint4 rvn, ovn;
    float gtn;
    load_tok(0, rvn, ovn, gtn);
    // The up kernel may read the residual and the previous gates before its own
    // wait once every CTA of this kernel has passed its wait.
    pdl_launch_dependents();
    const bool timed_out = !mbar_wait_bounded(bar, 0);
    if (timed_out)
        record_timeout(p.status);
    float gf[8];
    unpack_bf16x8(has_v ? *reinterpret_cast<const uint4 *>(g_s + v * 8) : make_uint4(0, 0, 0, 0), gf);

    for (int t = 0; t < M; ++t) {
        const uint4 rvv = rvn, ovv = ovn;
        const float gt = gtn;
        load_tok(t + 1, rvn, ovn, gtn);  // the next token's loads, in flight during this one
        float x[8], q = 0.f;
        {
            float rf[8];
            unpack_bf16x8(rvv, rf);
            if (p.inj_out) {
                float of[8];
                unpack_bf16x8(ovv, of);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    rf[e] = __bfloat162float(__float2bfloat16_rn(fmaf(of[e], gt, rf[e])));
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                q = fmaf(rf[e], rf[e], q);
                x[e] = rf[e] * gf[e];
            }
        }
        uint64_t xp[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            xp[e] = f32x2(x[2 * e], x[2 * e + 1]);
        float acc[kRowsPerGroup];
#pragma unroll
        for (int j = 0; j < kRowsPerGroup; ++j) {
            acc[j] = 0.f;
            if (has_v && j < gnr) {
                const uint4 wq = *reinterpret_cast<const uint4 *>(w_s + (size_t)(gr0 + j) * seg + v * 16);
                uint64_t a = 0;
                a = ffma2(bf16x2_as_f32x2(wq.x), xp[0], a);
                a = ffma2(bf16x2_as_f32x2(wq.y), xp[1], a);
                a = ffma2(bf16x2_as_f32x2(wq.z), xp[2], a);
                a = ffma2(bf16x2_as_f32x2(wq.w), xp[3], a);
                acc[j] = f32x2_sum(a);
            }
        }
        const float rsum = warp_transpose_sum8(acc, lane);
        float *rw = red_s + ((size_t)warp * M + t) * (kRowsPerGroup + 1);
        if ((lane & 3) == 0)
            rw[lane >> 2] = rsum;
        q = warp_sum(q);
        if (lane == 0)
            rw[kRowsPerGroup] = q;
    }
    __syncthreads();

    for (int i = tid; i < nrows * M; i += blockDim.x) {  // (token, row of the block)
        const int t = i / nrows, r = i % nrows;
        const int g = r / rpg, j = r % rpg;
        float sum = 0.f;
        for (int w = 0; w < wpg; ++w)
            sum += red_s[((size_t)(g * wpg + w) * M + t) * (kRowsPerGroup + 1) + j];
#pragma unroll
        for (int c = 0; c < kPartCopies; ++c)
            p.part1[c * p.part1_stride + ((size_t)s * M + t) * p.R + r0 + r] = sum;
    }
    if (blockIdx.y == 0 && tid < M) {  // every group saw the same inputs: use group 0
        float sum = 0.f;
        for (int w = 0; w < wpg; ++w)
            sum += red_s[((size_t)w * M + tid) * (kRowsPerGroup + 1) + kRowsPerGroup];
#pragma unroll
        for (int c = 0; c < kPartCopies; ++c)
            p.ssq1[c * kSsqStride + s * M + tid] = sum;
    }
    if (timed_out)
        mbar_wait_bounded(bar, 0);
}

struct UpmSmem {
    size_t bar, w, act, ssq, inv, total;
};

__host__ __device__ inline UpmSmem upm_layout(const UpParams &p)
{
    UpmSmem s;
    s.bar = 0;
    s.w = 128;
    s.act = round_up_sz(s.w + (size_t)p.L * 2 * p.C * p.HB, 128);
    s.ssq = round_up_sz(s.act + sizeof(float) * (size_t)p.M * p.L, 128);
    s.inv = round_up_sz(s.ssq + sizeof(float) * (size_t)p.M * kMaxCluster, 16);
    s.total = round_up_sz(s.inv + sizeof(float) * (size_t)p.M * kMaxCluster, 128);
    return s;
}

// CC: the stream count when it is a compile-time constant (4), else 0.
template <int CC>
__global__ void __launch_bounds__(1024, 1) hc_upm_kernel(const UpParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const UpmSmem lay = upm_layout(p);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + lay.bar);
    const unsigned char *w_s = smem + lay.w;
    float *act_s = reinterpret_cast<float *>(smem + lay.act);    // [M][L]
    float *ssq_s = reinterpret_cast<float *>(smem + lay.ssq);    // [M][S]
    float *invq_s = reinterpret_cast<float *>(smem + lay.inv);   // [M][S]: inv_rms of chunk q's stream

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int HB = p.HB, h0 = blockIdx.x * HB;
    const int hb = min(HB, p.H - h0);
    const int L = p.L, M = p.M, S = p.S;
    const size_t row_bytes = (size_t)L * 2;

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
        mbar_arrive_expect_tx(bar, (uint32_t)(row_bytes * hb * p.C));
        for (int c = 0; c < p.C; ++c)
            bulk_copy_g2s(smem + lay.w + (size_t)c * HB * row_bytes,
                          static_cast<const unsigned char *>(p.up.data) + ((size_t)c * p.H + h0) * row_bytes,
                          (uint32_t)(row_bytes * hb), bar);
    }

    const int hl = warp, h = h0 + hl;
    const bool h_ok = hl < hb;
    const int hc = lane >> 2;
    const bool holder = h_ok && (lane & 3) == 0 && hc < p.C;
    // Read before the dependency wait (the down kernel triggers after its own
    // wait): g, and each token's residual element and previous gate (.cg).
    float gval = 0.f, rv[kFewMaxTokens], ov[kFewMaxTokens], gp[kFewMaxTokens];
#pragma unroll
    for (int t = 0; t < kFewMaxTokens; ++t) {
        rv[t] = ov[t] = gp[t] = 0.f;
        if (holder && t < M) {
            rv[t] = __bfloat162float(__ushort_as_bfloat16(__ldcg(p.raw + (size_t)t * p.raw_mstride +
                                                                 (size_t)hc * p.raw_cstride + h)));
            if (p.inj_out) {
                ov[t] = __bfloat162float(__ushort_as_bfloat16(__ldcg(p.inj_out + (size_t)t * p.H + h)));
                gp[t] = __ldcg(p.inj_gate + (size_t)t * p.inj_stride + hc);
            }
        }
    }
    if (holder)
        gval = __bfloat162float(__ushort_as_bfloat16(p.g[hc * p.H + h]));

    pdl_wait();  // the partials come from the down kernel

    const int copy = blockIdx.x % kPartCopies;
    const float *part = p.part1 + copy * p.part1_stride;
    const float *ssq = p.ssq1 + copy * kSsqStride;
    for (int i = tid; i < M * S; i += blockDim.x)
        ssq_s[i] = ssq[i];  // [s][m] as written
    pdl_launch_dependents();
    __syncthreads();
    for (int i = tid; i < M * S; i += blockDim.x) {  // token m = i % M, chunk q = i / M: its stream's inv_rms
        const int m = i % M, q = i / M, c = q / p.sps;
        float t = 0.f;
        for (int j = 0; j < p.sps; ++j)
            t += ssq_s[(c * p.sps + j) * M + m];
        const float iv = rsqrtf(fmaf(t, p.inv_H, p.eps));
        invq_s[q * M + m] = iv;
        if (blockIdx.x == 0 && q % p.sps == 0)
            p.inv_out[(size_t)m * p.C + c] = iv;
    }
    __syncthreads();
    // act for every (token, row): the chunks' partials summed in order; a thread's
    // pairs two at a time, all their loads in flight together.
    constexpr int kPairs = 2;
    for (int i0 = tid; i0 < M * p.R; i0 += kPairs * blockDim.x) {
        float pv[kPairs][kMaxCluster];
#pragma unroll
        for (int u = 0; u < kPairs; ++u) {
            const int i = i0 + u * blockDim.x, m = i / p.R, k = i % p.R;
#pragma unroll
            for (int q = 0; q < kMaxCluster; ++q)
                pv[u][q] = (i < M * p.R && q < S) ? part[((size_t)q * M + m) * p.R + k] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kPairs; ++u) {
            const int i = i0 + u * blockDim.x, m = i / p.R, k = i % p.R;
            if (i >= M * p.R)
                break;
            float z = 0.f;
#pragma unroll
            for (int q = 0; q < kMaxCluster; ++q)
                if (q < S) z = fmaf(invq_s[q * M + m], pv[u][q], z);
            const float zc = z * p.inv_C;
            if (k < L) {
                const float a = zc * sigmoid_fast(zc);
                act_s[(size_t)m * L + k] = a;
                if (blockIdx.x == 0)
                    p.act_out[(size_t)m * L + k] = a;
            } else if (blockIdx.x == 0 && p.gate) {
                p.gate[(size_t)m * p.gate_stride + (k - L)] = 2.0f * sigmoid_fast(zc);
            }
        }
    }
    const bool timed_out = !mbar_wait_bounded(bar, 0);
    if (timed_out)
        record_timeout(p.status);
    __syncthreads();

    if (h_ok) {  // warp-uniform
        constexpr int NC = CC > 0 ? CC : 8;
        const uint32_t *wr = reinterpret_cast<const uint32_t *>(w_s) + (size_t)hl * (L / 2);
        const size_t cstride = (size_t)HB * (L / 2);
        for (int t = 0; t < M; ++t) {
            float nvh = 0.f, rt = rv[0], ot = ov[0], gt = gp[0];
#pragma unroll
            for (int u = 1; u < kFewMaxTokens; ++u)
                if (u == t) { rt = rv[u]; ot = ov[u]; gt = gp[u]; }
            if (holder) {
                if (p.inj_out)
                    rt = __bfloat162float(__float2bfloat16_rn(fmaf(ot, gt, rt)));
                if (p.raw_out)  // the stored residual [M][C*H], whatever view it was read through
                    p.raw_out[(size_t)t * p.W + (size_t)hc * p.H + h] = __bfloat16_as_ushort(__float2bfloat16_rn(rt));
                nvh = rt * invq_s[(hc * p.sps) * M + t] * gval;
            }
            uint64_t a2[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) a2[c] = 0;
            const float *act_t = act_s + (size_t)t * L;
#pragma unroll 2
            for (int j = lane; j < L / 2; j += 32) {
                const uint64_t xpair = *reinterpret_cast<const uint64_t *>(act_t + 2 * j);
#pragma unroll
                for (int c = 0; c < NC; ++c)
                    if (CC > 0 || c < p.C)
                        a2[c] = ffma2(bf16x2_as_f32x2(wr[c * cstride + j]), xpair, a2[c]);
            }
            float acc[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] = c < NC ? f32x2_sum(a2[c < NC ? c : 0]) : 0.f;
            const float d = warp_transpose_sum8(acc, lane);
            const float wv = sigmoid_fast(d);
            if (p.w_out && holder)
                p.w_out[(size_t)t * p.C * p.H + hc * p.H + h] = wv;
            float term = holder ? wv * nvh : 0.f;
            term += __shfl_xor_sync(0xffffffffu, term, 4);
            term += __shfl_xor_sync(0xffffffffu, term, 8);
            term += __shfl_xor_sync(0xffffffffu, term, 16);
            if (lane == 0)
                p.mixed[(size_t)t * p.H + h] = __bfloat16_as_ushort(__float2bfloat16_rn(term * p.inv_C));
        }
    }
    if (timed_out)
        mbar_wait_bounded(bar, 0);
}


__global__ void __launch_bounds__(256) hc_inject_kernel(const InjectParams p)
{
    pdl_launch_dependents();
    // The gates, and the guarantee that every reader of the old residual has
    // finished, come with the previous kernel's completion.
    pdl_wait();
    const long per_tok = p.W / 8;
    const long nvec = (long)p.M * per_tok;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < nvec; i += (long)gridDim.x * blockDim.x) {
        const long m = i / per_tok;
        const int e = (int)(i % per_tok) * 8;
        const int c = e / p.H, h = e % p.H;
        uint4 *rp = reinterpret_cast<uint4 *>(p.raw) + i;
        const uint4 rv = *rp;
        const uint4 ov = *reinterpret_cast<const uint4 *>(p.out + m * p.H + h);
        const float gt = p.gate[m * p.gate_stride + c];
        float rf[8], of[8];
        unpack_bf16x8(rv, rf);
        unpack_bf16x8(ov, of);
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(fmaf(of[2 * k], gt, rf[2 * k]),
                                                           fmaf(of[2 * k + 1], gt, rf[2 * k + 1]));
            o[k] = *reinterpret_cast<const uint32_t *>(&b);
        }
        *rp = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// raw[m][c*H + h] = emb[m][h]: one 16-byte vector of the wide row per thread.
__global__ void __launch_bounds__(256) hc_replicate_kernel(const ReplicateParams p)
{
    pdl_launch_dependents();
    pdl_wait();
    const long per_tok = (long)p.C * p.H / 8;
    const long nvec = (long)p.M * per_tok;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < nvec; i += (long)gridDim.x * blockDim.x) {
        const long m = i / per_tok;
        const int h = (int)((i % per_tok) * 8) % p.H;
        reinterpret_cast<uint4 *>(p.raw)[i] = *reinterpret_cast<const uint4 *>(p.emb + m * p.H + h);
    }
}

template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                      int cluster_x, bool pdl, Args &&...args)
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
    if (pdl) {
        attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Once per kernel and device: raises the dynamic shared-memory limit to the
// budget (which covers every launch the host logic allows) and asks for the
// largest shared-memory carveout. Consecutive kernels of a call share SMs
// (a dependent launch is resident while its predecessor runs); an SM can only
// hold CTAs of kernels whose carveouts agree and fit, so every kernel here
// asks for the same, largest one.
template <typename K>
cudaError_t allow_smem(K kernel, size_t smem)
{
    if (smem > kSmemBudget)
        return cudaErrorInvalidValue;
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
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        done.insert(key);
    return e;
}

template <int WT>
cudaError_t launch_down_wt(const DownParams &p, const LaunchCfg &cfg, cudaStream_t stream)
{
    const int mt = p.mt;
    const size_t smem = down_smem_bytes(p, mt);
    const dim3 grid(p.S, (p.R + p.rows_per_block - 1) / p.rows_per_block, 1);
    const dim3 block(down_threads(p));
    void (*k)(DownParams) = nullptr;
    switch (mt) {
    case 1: k = hc_down_kernel<WT, 1>; break;
    case 2: k = hc_down_kernel<WT, 2>; break;
    case 4: k = hc_down_kernel<WT, 4>; break;
    default: k = hc_down_kernel<WT, 8>; break;
    }
    cudaError_t e = allow_smem(k, smem);
    if (e != cudaSuccess)
        return e;
    return launch_ex(k, grid, block, smem, stream, p.S, cfg.pdl, p);
}

template <int WT>
cudaError_t launch_up_wt(const UpParams &p, const LaunchCfg &cfg, cudaStream_t stream)
{
    const int mt = p.mt;
    const size_t smem = up_smem_bytes(p, mt);
    const dim3 grid((p.H + p.HB - 1) / p.HB, 1, 1);
    const dim3 block(up_threads(p));
    void (*k)(UpParams) = nullptr;
    switch (mt) {
    case 1: k = hc_up_kernel<WT, 1>; break;
    case 2: k = hc_up_kernel<WT, 2>; break;
    case 4: k = hc_up_kernel<WT, 4>; break;
    default: k = hc_up_kernel<WT, 8>; break;
    }
    cudaError_t e = allow_smem(k, smem);
    if (e != cudaSuccess)
        return e;
    return launch_ex(k, grid, block, smem, stream, 0, cfg.pdl, p);
}

}  // namespace

cudaError_t launch_replicate(const ReplicateParams &p, const LaunchCfg &cfg, cudaStream_t stream)
{
    const long nvec = (long)p.M * p.C * p.H / 8;
    const int threads = 128;
    long blocks = std::max<long>(1, std::min<long>((nvec + threads - 1) / threads, (long)cfg.sm_count * 8));
    const cudaError_t e = allow_smem(hc_replicate_kernel, 0);
    if (e != cudaSuccess)
        return e;
    return launch_ex(hc_replicate_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream, 0, cfg.pdl, p);
}

int gemv_token_tile(int M)
{
    return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8;
}

size_t down_smem_bytes(const DownParams &p, int mt) { return down_layout(p, mt).total; }
size_t up_smem_bytes(const UpParams &p, int mt) { return up_layout(p, mt).total; }

int down_threads(const DownParams &p)
{
    const int rounds = (p.rows_per_block + 15) / 16;
    const int warps = std::max(4, (p.rows_per_block + rounds - 1) / rounds);
    return 32 * warps;
}

int up_threads(const UpParams &p)
{
    const int warps = std::min(24, std::max(2, (p.C * p.HB + 3) / 4));
    return 32 * warps;
}

cudaError_t launch_down(const DownParams &p, const LaunchCfg &cfg, cudaStream_t stream)
{
    return p.down.type == 0 ? launch_down_wt<0>(p, cfg, stream) : launch_down_wt<1>(p, cfg, stream);
}

int up1_threads(const UpParams &u) { return 32 * std::max(u.HB, (u.R + 31) / 32); }

bool one_token_ok(const DownParams &d, const UpParams &u)
{
    if (d.M != 1 || d.S > kMaxCluster || d.C > 8 || u.HB > 32 || u.R > 1024)
        return false;
    if (down1_groups(d) * down1_group_threads(d) > 1024 || up1_threads(u) > 1024)
        return false;
    return down1_layout(d).total <= kSmemBudget && up1_layout(u).total <= kSmemBudget;
}

int downm_threads(const DownParams &d) { return down1_groups(d) * down1_group_threads(d); }

bool few_tokens_ok(const DownParams &d, const UpParams &u)
{
    if (d.M < 2 || d.M > kFewMaxTokens || d.down.type != 0 || u.up.type != 0 || d.S > kMaxCluster || d.C > 8 ||
        u.HB > 32 || u.R > 1024 || d.M * d.S > kSsqStride)
        return false;
    if (downm_threads(d) > 1024 || up1_threads(u) > 1024)
        return false;
    return downm_layout(d, downm_threads(d) / 32).total <= kSmemBudget && upm_layout(u).total <= kSmemBudget;
}

cudaError_t launch_few_tokens(const DownParams &d, const UpParams &u, const LaunchCfg &cfg, cudaStream_t stream)
{
    if (!few_tokens_ok(d, u))
        return cudaErrorInvalidConfiguration;
    void (*ku)(UpParams) = u.C == 4 ? hc_upm_kernel<4> : hc_upm_kernel<0>;
    const size_t sd = downm_layout(d, downm_threads(d) / 32).total, su = upm_layout(u).total;
    cudaError_t e = allow_smem(hc_downm_kernel, sd);
    if (e == cudaSuccess)
        e = allow_smem(ku, su);
    if (e != cudaSuccess)
        return e;
    const dim3 dgrid(d.S, (d.R + d.rows_per_block - 1) / d.rows_per_block, 1);
    e = launch_ex(hc_downm_kernel, dgrid, dim3(downm_threads(d)), sd, stream, 0, cfg.pdl, d);
    if (e != cudaSuccess)
        return e;
    return launch_ex(ku, dim3((u.H + u.HB - 1) / u.HB), dim3(up1_threads(u)), su, stream, 0, cfg.pdl, u);
}

cudaError_t launch_one_token(const DownParams &d, const UpParams &u, const LaunchCfg &cfg, cudaStream_t stream)
{
    if (!one_token_ok(d, u))
        return cudaErrorInvalidConfiguration;
    void (*kd)(DownParams) = d.down.type == 0 ? hc_down1_kernel<0> : hc_down1_kernel<1>;
    void (*ku)(UpParams);
    if (u.l2_pf_bytes)
        ku = u.up.type != 0 ? (u.C == 4 ? hc_up1_kernel<1, 4, true> : hc_up1_kernel<1, 0, true>)
           : u.C == 4       ? hc_up1_kernel<0, 4, true>
                            : hc_up1_kernel<0, 0, true>;
    else
        ku = u.up.type != 0 ? (u.C == 4 ? hc_up1_kernel<1, 4, false> : hc_up1_kernel<1, 0, false>)
           : u.C == 4       ? hc_up1_kernel<0, 4, false>
                            : hc_up1_kernel<0, 0, false>;
    const size_t sd = down1_layout(d).total, su = up1_layout(u).total;
    cudaError_t e = allow_smem(kd, sd);
    if (e == cudaSuccess)
        e = allow_smem(ku, su);
    if (e != cudaSuccess)
        return e;
    const dim3 dgrid(d.S, (d.R + d.rows_per_block - 1) / d.rows_per_block, 1);
    e = launch_ex(kd, dgrid, dim3(down1_groups(d) * down1_group_threads(d)), sd, stream, 0, cfg.pdl, d);
    if (e != cudaSuccess)
        return e;
    return launch_ex(ku, dim3((u.H + u.HB - 1) / u.HB), dim3(up1_threads(u)), su, stream, 0, cfg.pdl, u);
}

cudaError_t launch_up(const UpParams &p, const LaunchCfg &cfg, cudaStream_t stream)
{
    return p.up.type == 0 ? launch_up_wt<0>(p, cfg, stream) : launch_up_wt<1>(p, cfg, stream);
}

cudaError_t launch_inject(const InjectParams &p, const LaunchCfg &cfg, cudaStream_t stream)
{
    const long nvec = (long)p.M * p.W / 8;
    const int threads = 128;
    long blocks = (nvec + threads - 1) / threads;
    blocks = std::min<long>(blocks, (long)cfg.sm_count * 8);
    blocks = std::max<long>(blocks, 1);
    const cudaError_t e = allow_smem(hc_inject_kernel, 0);
    if (e != cudaSuccess)
        return e;
    return launch_ex(hc_inject_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream, 0, cfg.pdl, p);
}

}  // namespace tshc
