// hc_tc.h -- launch parameters of the tensor-core (tcgen05) batched path.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "hc_kernels.h"

namespace tshc {

constexpr int kTcMinTokens = 16;          // the batched path starts at this many tokens
constexpr size_t kTcSmemLimit = 232448;   // 227 KB opt-in shared memory per CTA

struct TcDownParams {
    const uint16_t *raw;      // bf16 [M][W]
    const uint16_t *g;        // bf16 [W]
    float *part;              // [C][R][M]: per-stream partial z (un-normalised)
    float *ssq;               // [C][M]:    per-stream sum of squares
    int M, H, C, L, R, W;
    int has_inject;
    int RT;                   // row tiles of 128
    int CS, chunk;            // CTAs per stream (cluster size), chunk width (multiple of 64)
    int NT, n_stages;         // tokens per tile (multiple of 16, <= 128), pipeline depth
    unsigned *status;
    const uint16_t *inj_out;  // fused inject-add of the previous sublayer, or nullptr
    const float *inj_gate;
    long inj_stride;
    // INT4-affine weights (wt == 1): the producers dequantise the weight tiles
    // to bf16 hi + lo in place of the TMA loads of bf16 tiles (wt == 0).
    int wt;
    WeightView dw, iw;        // input_mix_weight_down, block_inject_weight
};

struct TcReduceParams {
    const float *part;
    const float *ssq;
    float *act;               // [M][L] fp32
    uint16_t *act_hi;         // [M][L] bf16
    uint16_t *act_lo;         // [M][L] bf16
    float *inv_rms;           // [M][C]
    float *gate;              // token m's gates at gate + m * gate_stride
    long gate_stride;
    int M, H, C, L, R;
    float eps, inv_C;
};

struct TcUpParams {
    const uint16_t *raw;      // bf16 [M][W]
    const uint16_t *g;        // bf16 [W]
    const float *inv_rms;     // [M][C]
    uint16_t *mixed;          // bf16 [M][H]
    int M, H, C, L, W;
    int HBt;                  // h values per CTA (C * HBt <= 128, multiple of 8)
    int NT, n_stages;
    float inv_C;
    unsigned *status;
    uint16_t *raw_out;        // == raw when the inject-add is fused, else nullptr
    const uint16_t *inj_out;
    const float *inj_gate;
    long inj_stride;
    int wt;                   // 1: INT4-affine up weights, dequantised by producer warps
    WeightView uw;
};

struct TcCall {
    TcDownParams down;
    TcReduceParams red;
    TcUpParams up;
    const void *wd, *wi, *wu;  // bf16 weights
};

size_t tc_down_smem(int NT, int ns, int wt);
size_t tc_up_smem(int NT, int ns, int C, int HBt, int wt);
cudaError_t launch_tc_call(const TcCall &t, cudaStream_t stream);

}  // namespace tshc
