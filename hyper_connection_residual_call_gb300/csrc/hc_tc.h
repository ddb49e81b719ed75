// hc_tc.h -- launch parameters of the tensor-core (tcgen05) batched path.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "hc_kernels.h"

namespace tshc {

// The batched path starts at 2 tokens: a 16-token tile serves 2..16 tokens in
// about the time of one (absent tokens are TMA zero-fill), far faster than the
// cluster split-K kernels beyond 2 tokens.
constexpr int kTcMinTokens = 2;
constexpr size_t kTcSmemLimit = 232448;   // 227 KB opt-in shared memory per CTA
constexpr int kTcChunkCtas = 152;         // the down kernel's K split aims at about this many CTAs
constexpr int kTcMaxChunkKb = 16;         // and cuts K into chunks of at most this many 64-wide blocks
// Shared memory the reduce kernel reserves (and does not use) so that at most
// one of its CTAs runs per SM and none beside a down or up CTA: launched early
// (programmatic dependent launch), its CTAs would otherwise pile onto the few
// SMs the down kernel leaves free and run several times slower there.
constexpr size_t kTcReduceSmemReserve = 120 * 1024;

// Tiling of one call on M tokens. It depends on the shape only, not on the
// device, so the order of the split-K sums -- and every result bit -- does not
// either.
struct TcPlan {
    int NT;       // tokens per tile (multiple of 16, <= 128)
    int ntiles;   // token tiles
    int Mp;       // ntiles * NT: the padded token count of the partials
    int KBc;      // 64-wide K blocks per down CTA
    int nchunk;   // K chunks over the C*H inputs
};

__host__ __device__ inline TcPlan tc_plan(int M, int L, int C, int W)
{
    TcPlan p;
    p.NT = M >= 128 ? 128 : (M + 15) / 16 * 16;
    p.ntiles = (M + p.NT - 1) / p.NT;
    p.Mp = p.ntiles * p.NT;
    const int RT = (L + C + 127) / 128;
    const int KBT = W / 64;
    const int per = kTcChunkCtas / (RT * p.ntiles);
    const int target = per > 1 ? per : 1;
    p.KBc = (KBT + target - 1) / target;
    // A chunk's partial accumulates in one TMEM accumulator, and the error of that sum
    // grows with its length (1024 MMAs for 128 K blocks at the widest residual put act
    // past the fp32 bar); longer K is cut into more chunks, summed by the reduce kernel.
    if (p.KBc > kTcMaxChunkKb)
        p.KBc = kTcMaxChunkKb;
    p.nchunk = (KBT + p.KBc - 1) / p.KBc;
    return p;
}

// Prep: per (token, stream) the fused inject-add, inv_rms and normed = raw *
// g * inv_rms, stored as bf16 hi + lo (normed = hi + lo to ~16 significant
// bits) for the two GEMMs' TMA loads.
struct TcPrepParams {
    const uint16_t *raw;      // bf16: element (m, c, h) at raw + m*raw_mstride + c*raw_cstride + h
    long raw_mstride;         // W, or H when every stream reads one [M][H] row (entry)
    int raw_cstride;          // H, or 0 (entry)
    const uint16_t *g;        // bf16 [W]
    uint16_t *raw_out;        // bf16 [M][W]: the residual the call sees, written back; or nullptr
    const uint16_t *inj_out;  // bf16 [M][H] with a fused inject-add, else nullptr
    const float *inj_gate;    // token m's previous gates at inj_gate + m * inj_stride
    long inj_stride;
    uint16_t *x_hi, *x_lo;    // bf16 [M][W]
    float *inv_rms;           // [M][C]
    int M, H, C, W;
    float eps, inv_H;
};

struct TcDownParams {
    float *part;              // [nchunk][Mp][R]: partial z of K chunk kc
    int M, L, C, R, W, Mp;
    int has_inject;
    int KBc, nchunk;          // K blocks per chunk, chunks
    int NT, n_stages;         // tokens per tile, pipeline depth
    unsigned *status;
    // INT4-affine weights (wt == 1): producer warps dequantise the weight tiles
    // to bf16 hi + lo in place of the TMA loads of bf16 tiles (wt == 0).
    int wt;
    WeightView dw, iw;        // input_mix_weight_down, block_inject_weight
};

struct TcReduceParams {
    const float *part;
    float *act;               // [M][L] fp32
    uint16_t *act_hi;         // [M][L] bf16(act), round to nearest: the up GEMM's B operand ...
    uint16_t *act_lo;         // [M][L] bf16(act - act_hi): ... and its low part (act = hi + lo to ~16 bits)
    float *gate;              // token m's gates at gate + m * gate_stride
    long gate_stride;
    int M, L, R, Mp, nchunk;
    float inv_C;
    // Byte ranges of the up kernel's weights (data, scales, biases) that the
    // CTAs ask L2 to prefetch, split evenly over the grid; bytes == 0 if unused.
    const void *l2_next[3];
    size_t l2_next_bytes[3];
};

struct TcUpParams {
    uint16_t *mixed;          // bf16 [M][H]
    int M, H, C, L, W;
    int HBt;                  // h values per CTA (C * HBt <= 128, multiple of 8)
    int NT, n_stages;
    float inv_C;
    unsigned *status;
    int wt;                   // 1: INT4-affine up weights, dequantised by producer warps
    WeightView uw;
    float *w_out;             // optional fp32 [M][W]: w = sigmoid(up(act)) (debug output), or nullptr
};

struct TcCall {
    TcPrepParams prep;
    TcDownParams down;
    TcReduceParams red;
    TcUpParams up;
    const void *wd, *wi, *wu;  // bf16 weights
};

size_t tc_down_smem(int NT, int ns, int wt);
size_t tc_up_smem(int NT, int ns, int C, int HBt, int wt);
cudaError_t launch_tc_call(const TcCall &t, cudaStream_t stream);

}  // namespace tshc
