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
//   (lm_head GEMV kernel) key_proj and value_proj rows against emb -> fp32
//   hc_ple_gate_kernel    one CTA per token: the norms' sums of squares, the
//                         gate, and the conv input x = norm_conv(gv) [M][W]
//   hc_ple_conv_kernel    one thread per channel: the causal conv over the
//                         state and the chunk, silu, gv, the residual add
//                         (rounded to bf16), and the new state.
#include <cuda_bf16.h>

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

__device__ __forceinline__ float block_sum_into(float v, float *red, int tid)
{
    // Sum over the block in fixed order (warps, then the warp totals in order).
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((tid & 31) == 0)
        red[tid >> 5] = v;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
        t += red[w];
    __syncthreads();  // red may be reused
    return t;
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

// Grid M, one CTA per token. Per stream c: sums of squares of the key and of
// the residual, and their raw dot (the norms' factors are applied after the
// sums, they are per stream); the value's sum of squares (shared by the
// streams); then the gate, and x = norm_conv(gate * value).
__global__ void __launch_bounds__(kPleThreads) hc_ple_gate_kernel(const PleParams p)
{
    __shared__ float red[kPleThreads / 32];
    __shared__ float gate_s[8], rc_s[8];
    pdl_launch_dependents();
    pdl_wait();  // key and value come from the projection kernels
    const int m = blockIdx.x, tid = threadIdx.x;
    const int H = p.H, C = p.C, W = C * H;
    const float *key = p.key + (size_t)m * W;
    const float *value = p.value + (size_t)m * H;
    const uint16_t *hid = p.hidden + (size_t)m * W;

    float vv = 0.f;
    for (int h = tid; h < H; h += blockDim.x)
        vv = fmaf(value[h], value[h], vv);
    const float sum_vv = block_sum_into(vv, red, tid);

    for (int c = 0; c < C; ++c) {
        float kk = 0.f, qq = 0.f, kq = 0.f;
        for (int h = tid; h < H; h += blockDim.x) {
            const size_t j = (size_t)c * H + h;
            const float k = key[j], q = bf16_at(hid, j);
            kk = fmaf(k, k, kk);
            qq = fmaf(q, q, qq);
            kq = fmaf(k * bf16_at(p.norm_key, j), q * bf16_at(p.norm_query, j), kq);
        }
        const float skk = block_sum_into(kk, red, tid);
        const float sqq = block_sum_into(qq, red, tid);
        const float skq = block_sum_into(kq, red, tid);
        if (tid == 0) {
            const float rk = rsqrtf(fmaf(skk, p.inv_H, p.eps)), rq = rsqrtf(fmaf(sqq, p.inv_H, p.eps));
            const float g = skq * rk * rq * p.inv_sqrt_H;
            const float sg = (g > 0.f) - (g < 0.f);
            const float gate = 1.0f / (1.0f + expf(-sg * sqrtf(fmaxf(fabsf(g), 1e-6f))));
            gate_s[c] = gate;
            // norm_conv of gate * value: sum over h of (gate v)^2 = gate^2 sum v^2
            rc_s[c] = rsqrtf(fmaf(gate * gate * sum_vv, p.inv_H, p.eps));
            p.gate[(size_t)m * C + c] = gate;
        }
    }
    __syncthreads();
    for (int j = tid; j < W; j += blockDim.x) {
        const int c = j / H, h = j % H;
        p.x[(size_t)m * W + j] = gate_s[c] * value[h] * rc_s[c] * bf16_at(p.norm_conv, j);
    }
}

// One thread per channel j: for each token of the chunk in order, the causal
// conv over the nine earlier inputs (state, then the chunk's own), silu, gv
// and the residual add; then the last nine inputs become the state.
__global__ void __launch_bounds__(256) hc_ple_conv_kernel(const PleParams p)
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
    for (int t = 0; t < p.M; ++t) {
        const float xt = p.x[(size_t)t * W + j];
        const float y = fmaf(w0, win[0], fmaf(w1, win[3], fmaf(w2, win[6], w3 * xt)));
        const float gv = p.gate[(size_t)t * p.C + c] * p.value[(size_t)t * p.H + h];
        const float out = gv + y / (1.0f + expf(-y));
        const size_t o = (size_t)t * W + j;
        p.hidden[o] = __bfloat16_as_ushort(__float2bfloat16_rn(bf16_at(p.hidden, o) + out));
#pragma unroll
        for (int i = 0; i < 8; ++i)
            win[i] = win[i + 1];
        win[8] = xt;
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
    // key = key_proj(emb) [M][W], value = value_proj(emb) [M][H]: bf16 weight rows
    // against emb, the lm_head GEMV kernel, in tiles of kLmHeadMaxTokens tokens.
    for (int t0 = 0; t0 < p.M; t0 += kLmHeadMaxTokens) {
        for (int which = 0; which < 2; ++which) {
            LmHeadParams g{};
            g.M = p.M - t0 < kLmHeadMaxTokens ? p.M - t0 : kLmHeadMaxTokens;
            g.H = p.H;
            g.V = which == 0 ? p.C * p.H : p.H;
            g.mixed = p.emb + (size_t)t0 * p.H;
            g.w = which == 0 ? p.key_proj : p.value_proj;
            g.logits = which == 0 ? p.key + (size_t)t0 * p.C * p.H : p.value + (size_t)t0 * p.H;
            g.logits_stride = g.V;
            g.status = p.status;
            if (!lm_head_plan(g, cfg.sm_count))
                return cudaErrorInvalidValue;
            if ((e = launch_lm_head(g, cfg, stream)) != cudaSuccess)
                return e;
        }
    }
    if ((e = launch(hc_ple_gate_kernel, dim3(p.M), dim3(kPleThreads))) != cudaSuccess)
        return e;
    const int W = p.C * p.H;
    return launch(hc_ple_conv_kernel, dim3((W + 255) / 256), dim3(256));
}

}  // namespace tshc
