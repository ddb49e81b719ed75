// hc_ple.cu -- the PLE gate on the wide residual (families/qwen4/mod.rs,
// "## PLE", layer index 1 only; the decoder adds it to the residual before that
// layer's attn_hc):
//
//   emb   = concat of the 16 table rows picked by the token's row ids
//   key   = norm_key(key_proj(emb))       value = value_proj(emb)
//   query = norm_query(hidden)
//   gate  = sigmoid(signed_sqrt((key * query).sum over h / sqrt(H)))   per stream
//   gv    = gate * value                  (value broadcast to every stream)
//   out   = gv + silu(dilated_conv(norm_conv(gv)))
//   hidden += out
//
// The three norms take the hyper-connection norm's form (groups of H, eps
// inside the root, a direct scale per element); the dilated convolution is
// depthwise and causal along the token axis (dilation 3, four taps), with the
// inputs of the nine tokens before the chunk carried in a caller-owned state.
//
// Kernels, chained with programmatic dependent launch:
//   hc_ple_gather_kernel  the 16 rows per token -> emb bf16 [M][H]; a row id out
//                         of range records TS_ERR_INVALID_ARG in the device
//                         status word and reads zeros
//   (lm_head kernel)      key_proj and value_proj rows against emb -> fp32, on
//                         the tensor cores, both weights in one launch
//   hc_ple_gate_kernel    one CTA per (stream, token): the norms' sums of
//                         squares, the gate, and the conv input
//                         x = norm_conv(gv) [M][W]
//   hc_ple_conv_kernel    one thread per channel: the causal conv over the
//                         state and the chunk, silu, gv, the residual add
//                         (rounded to bf16), and the new state.
#include <cuda_bf16.h>

#include <algorithm>

#include "hc_kernels.h"
#include "ptx.cuh"

namespace tshc {

namespace {

constexpr unsigned kStatusInvalidArg = 1u;  // TS_ERR_INVALID_ARG of ts_hc.h
constexpr int kPleThreads = 512;

__device__ __forceinline__ float bf16_at(const uint16_t *p, size_t i)
{
    return __bfloat162float(__ushort_as_bfloat16(p[i]));
}

// Grid M: token m's 16 row segments of H/16, one 16-byte vector per thread and step.
__global__ void __launch_bounds__(256) hc_ple_gather_kernel(const PleParams p)
{
    pdl_launch_dependents();
    pdl_wait();  // the rows may come from an earlier kernel
    const int m = blockIdx.x;
    const int seg = p.H / 16, nvec = seg / 8;
    for (int i = threadIdx.x; i < 16 * nvec; i += blockDim.x) {
        const int r = i / nvec, v = i % nvec;
        const int id = p.rows[(size_t)m * 16 + r];
        uint4 val = make_uint4(0, 0, 0, 0);
        if (id >= 0 && id < p.n_rows)
            val = reinterpret_cast<const uint4 *>(p.table + (size_t)id * seg)[v];
        else if (p.status)
            atomicExch(p.status, kStatusInvalidArg);
        reinterpret_cast<uint4 *>(p.emb + (size_t)m * p.H + (size_t)r * seg)[v] = val;
    }
}

// Grid (C, M): CTA (c, m) owns stream c of token m, thread t the 8-element
// chunks t, t + blockDim, ... of it. Sums of squares of the key and of the
// residual, their dot with the norms' scales applied (the norms' 1/rms factors
// are per stream, so they come after the sums), and the value's sum of squares
// (the same in every stream); one fixed-order block reduction of the four;
// then the gate and x = norm_conv(gate * value) for the stream.
__global__ void __launch_bounds__(kPleThreads) hc_ple_gate_kernel(const PleParams p)
{
    __shared__ float red[4][kPleThreads / 32];
    __shared__ float gate_rc[2];
    pdl_launch_dependents();
    pdl_wait();  // key and value come from the projection kernels
    const int c = blockIdx.x, m = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H, C = p.C, W = C * H, nch = H / 8;
    const size_t so = (size_t)c * H;
    const float *key = p.key + (size_t)m * W + so;
    const float *value = p.value + (size_t)m * H;
    const uint16_t *hid = p.hidden + (size_t)m * W + so;

    float kk = 0.f, qq = 0.f, kq = 0.f, vv = 0.f;
    for (int i = tid; i < nch; i += blockDim.x) {
        const float4 k0 = reinterpret_cast<const float4 *>(key)[2 * i], k1 = reinterpret_cast<const float4 *>(key)[2 * i + 1];
        const float4 v0 = reinterpret_cast<const float4 *>(value)[2 * i], v1 = reinterpret_cast<const float4 *>(value)[2 * i + 1];
        const uint4 q = reinterpret_cast<const uint4 *>(hid)[i];
        const uint4 gk = reinterpret_cast<const uint4 *>(p.norm_key + so)[i];
        const uint4 gq = reinterpret_cast<const uint4 *>(p.norm_query + so)[i];
        const float kf[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
        const float vf[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w}, kw[4] = {gk.x, gk.y, gk.z, gk.w}, gw[4] = {gq.x, gq.y, gq.z, gq.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float qf = (e & 1) ? bf16_hi(qw[e / 2]) : bf16_lo(qw[e / 2]);
            const float sk = (e & 1) ? bf16_hi(kw[e / 2]) : bf16_lo(kw[e / 2]);
            const float sq = (e & 1) ? bf16_hi(gw[e / 2]) : bf16_lo(gw[e / 2]);
            kk = fmaf(kf[e], kf[e], kk);
            qq = fmaf(qf, qf, qq);
            kq = fmaf(kf[e] * sk, qf * sq, kq);
            vv = fmaf(vf[e], vf[e], vv);
        }
    }
    float acc[4] = {kk, qq, kq, vv};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
        if (lane == 0)
            red[k][warp] = acc[k];
    }
    __syncthreads();
    if (tid == 0) {
        float t[4] = {0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w)  // warps in order
            for (int k = 0; k < 4; ++k)
                t[k] += red[k][w];
        const float rk = rsqrtf(fmaf(t[0], p.inv_H, p.eps)), rq = rsqrtf(fmaf(t[1], p.inv_H, p.eps));
        const float g = t[2] * rk * rq * p.inv_sqrt_H;
        const float sg = (g > 0.f) - (g < 0.f);
        const float gate = 1.0f / (1.0f + expf(-sg * sqrtf(fmaxf(fabsf(g), 1e-6f))));
        // norm_conv of gate * value: the sum over h of (gate v)^2 is gate^2 sum v^2
        gate_rc[0] = gate;
        gate_rc[1] = rsqrtf(fmaf(gate * gate * t[3], p.inv_H, p.eps));
        p.gate[(size_t)m * C + c] = gate;
    }
    __syncthreads();
    const float f = gate_rc[0] * gate_rc[1];
    float *x = p.x + (size_t)m * W + so;
    for (int i = tid; i < nch; i += blockDim.x) {
        const float4 v0 = reinterpret_cast<const float4 *>(value)[2 * i], v1 = reinterpret_cast<const float4 *>(value)[2 * i + 1];
        const uint4 gc = reinterpret_cast<const uint4 *>(p.norm_conv + so)[i];
        reinterpret_cast<float4 *>(x)[2 * i] =
            make_float4(f * v0.x * bf16_lo(gc.x), f * v0.y * bf16_hi(gc.x), f * v0.z * bf16_lo(gc.y), f * v0.w * bf16_hi(gc.y));
        reinterpret_cast<float4 *>(x)[2 * i + 1] =
            make_float4(f * v1.x * bf16_lo(gc.z), f * v1.y * bf16_hi(gc.z), f * v1.z * bf16_lo(gc.w), f * v1.w * bf16_hi(gc.w));
    }
}

// One thread per channel j: the tokens of the chunk in order, in batches of
// kConvBatch whose loads are all issued before the batch's first residual
// store; per token the causal conv over the nine earlier inputs (state, then
// the chunk's own), silu, gv and the residual add; then the last nine inputs
// become the state.
constexpr int kConvBatch = 8;
constexpr int kConvThreads = 128;

__global__ void __launch_bounds__(kConvThreads) hc_ple_conv_kernel(const PleParams p)
{
    pdl_launch_dependents();
    pdl_wait();  // x and the gates come from the gate kernel
    const int W = p.C * p.H;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= W)
        return;
    const int c = j / p.H, h = j % p.H;
    const uint2 wq = reinterpret_cast<const uint2 *>(p.conv_w)[j];  // four bf16 taps
    const float w0 = bf16_lo(wq.x), w1 = bf16_hi(wq.x), w2 = bf16_lo(wq.y), w3 = bf16_hi(wq.y);
    float win[9];  // inputs of tokens t-9 .. t-1
#pragma unroll
    for (int i = 0; i < 9; ++i)
        win[i] = p.state[(size_t)i * W + j];
    for (int t0 = 0; t0 < p.M; t0 += kConvBatch) {
        float xs[kConvBatch], gv[kConvBatch], hs[kConvBatch];
#pragma unroll
        for (int k = 0; k < kConvBatch; ++k) {
            const int t = t0 + k;
            if (t < p.M) {
                xs[k] = p.x[(size_t)t * W + j];
                gv[k] = p.gate[(size_t)t * p.C + c] * p.value[(size_t)t * p.H + h];
                hs[k] = bf16_at(p.hidden, (size_t)t * W + j);
            }
        }
#pragma unroll
        for (int k = 0; k < kConvBatch; ++k) {
            const int t = t0 + k;
            if (t < p.M) {
                const float y = fmaf(w0, win[0], fmaf(w1, win[3], fmaf(w2, win[6], w3 * xs[k])));
                const float out = gv[k] + y / (1.0f + expf(-y));
                p.hidden[(size_t)t * W + j] = __bfloat16_as_ushort(__float2bfloat16_rn(hs[k] + out));
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    win[i] = win[i + 1];
                win[8] = xs[k];
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 9; ++i)
        p.state[(size_t)i * W + j] = win[i];
}

}  // namespace

cudaError_t launch_ple(const PleParams &p, const LaunchCfg &cfg, cudaStream_t stream)
{
    auto launch = [&](auto kernel, dim3 grid, dim3 block) {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = grid;
        lc.blockDim = block;
        lc.stream = stream;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        lc.attrs = &attr;
        lc.numAttrs = cfg.pdl ? 1 : 0;
        return cudaLaunchKernelEx(&lc, kernel, p);
    };
    cudaError_t e = launch(hc_ple_gather_kernel, dim3(p.M), dim3(256));
    if (e != cudaSuccess)
        return e;
    // key = key_proj(emb) [M][W] and value = value_proj(emb) [M][H] in one launch of
    // the lm_head kernel (tensor cores; the two weights' tiles side by side), in
    // tiles of kLmHeadMaxTokens tokens.
    for (int t0 = 0; t0 < p.M; t0 += kLmHeadMaxTokens) {
        LmHeadParams g{};
        g.M = p.M - t0 < kLmHeadMaxTokens ? p.M - t0 : kLmHeadMaxTokens;
        g.H = p.H;
        g.mixed = p.emb + (size_t)t0 * p.H;
        g.w = p.key_proj;
        g.V = p.C * p.H;
        g.logits = p.key + (size_t)t0 * p.C * p.H;
        g.logits_stride = g.V;
        g.w2 = p.value_proj;
        g.V2 = p.H;
        g.logits2 = p.value + (size_t)t0 * p.H;
        g.logits2_stride = p.H;
        g.status = p.status;
        if ((e = launch_lm_head(g, cfg, stream)) != cudaSuccess)
            return e;
    }
    // The gate kernel: about one 8-element chunk of the stream per thread.
    const int gate_threads = std::min(kPleThreads, std::max(32, (p.H / 8 + 31) / 32 * 32));
    if ((e = launch(hc_ple_gate_kernel, dim3(p.C, p.M), dim3(gate_threads))) != cudaSuccess)
        return e;
    const int W = p.C * p.H;
    return launch(hc_ple_conv_kernel, dim3((W + kConvThreads - 1) / kConvThreads), dim3(kConvThreads));
}

}  // namespace tshc
