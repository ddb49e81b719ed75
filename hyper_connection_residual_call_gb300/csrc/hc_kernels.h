// hc_kernels.h -- launch parameters and launchers of the hyper-connection
// kernels (internal to the library; the public ABI is include/ts_hc.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tshc {

// A [rows][cols] weight in device memory (rows = outputs).
struct WeightView {
    int type;                 // 0 bf16, 1 INT4-affine
    int group;                // INT4 group size: 32, 64 or 128
    int gshift;               // log2(group): group indices are shifts, not divisions
    const void *data;         // bf16 [rows][cols] or uint8 [rows][cols/2]
    const uint16_t *scales;   // fp16 [rows][cols/group]
    const uint16_t *biases;   // fp16 [rows][cols/group]
};

// Split-K down projection: rows 0..L-1 are input_mix_weight_down, rows
// L..L+Ci-1 block_inject_weight (Ci = C, or 0 for the mixer). A cluster of
// S = C * sps CTAs shares one block of rows; CTA s of the cluster owns input
// columns [s*KC, (s+1)*KC), which lie inside stream s / sps.
struct DownParams {
    const uint16_t *raw;      // bf16: element (m, c, h) at raw + m*raw_mstride + c*raw_cstride + h
    long raw_mstride;         // W for a [M][W] residual; H when every stream reads one
    int raw_cstride;          // H for a [M][W] residual; 0 when every stream reads one [M][H] row (entry)
    const uint16_t *g;        // bf16 [W]
    WeightView down;          // [L][W]
    WeightView inject;        // [C][W]; data == nullptr for the mixer
    float *act;               // [M][L]  silu(z / C)
    float *inv_rms;           // [M][C]
    float *gate;              // token m's gates at gate + m * gate_stride
    long gate_stride;
    int M, H, C, L, R, W;     // R = L + Ci rows
    int sps, S, KC;           // chunks per stream, cluster size, chunk width
    int rows_per_block;
    int mt;                   // tokens per tile (1, 2, 4 or 8)
    float eps, inv_C;
    unsigned *status;
    // Optional fused inject-add of the previous sublayer: the call sees
    // raw + out * prev_gate (rounded to bf16) in place of raw. Not written here.
    // (The residual the call sees is written back by the up kernel.)
    const uint16_t *inj_out;  // bf16 [M][H], or nullptr
    const float *inj_gate;    // token m's previous gates at inj_gate + m * inj_stride
    long inj_stride;
    // One-token path (launch_one_token): per-chunk partial dots [S][R] and
    // per-chunk sums of squares [S], left in the workspace for the up kernel,
    // written kPartCopies times (copy c at part1 + c * part1_stride and at
    // ssq1 + c * kSsqStride) so that fewer up CTAs read each L2 line.
    float *part1;
    float *ssq1;
    long part1_stride;
};

// Copies of the one-token partials; up CTA b reads copy b % kPartCopies.
constexpr int kPartCopies = 8;
// The few-token path (2 <= M <= kFewMaxTokens, bf16 weights): the one-token
// kernels' layout with a token loop inside. Each token adds a serial chain to
// both kernels, so it beats the tensor-core path (about 13.6 µs per call at the
// full shape from 2 to 16 tokens) at 2 and 3 tokens (9.4 and 11.7 µs) but not at 4.
constexpr int kFewMaxTokens = 3;
constexpr long kSsqStride = 64;  // floats between the copies of the sums of squares

// Up projection + sigmoid + mean mix: CTA b owns h in [b*HB, b*HB + HB) of
// every stream, i.e. up rows {c*H + h}.
struct UpParams {
    const uint16_t *raw;      // bf16, read through the same view as DownParams::raw
    long raw_mstride;
    int raw_cstride;
    const uint16_t *g;        // bf16 [W]
    WeightView up;            // [W][L]
    const float *act;         // [M][L]
    const float *inv_rms;     // [M][C]
    uint16_t *mixed;          // bf16 [M][H]
    int M, H, C, L, W;
    int HB;
    int mt;                   // tokens per tile (1, 2, 4 or 8)
    float inv_C;
    unsigned *status;
    // Optional write-back of the residual the call sees (see DownParams): each
    // CTA owns its h-block of every stream and writes it to raw_out [M][W]
    // (raw + out * prev_gate with a fused inject-add, in place; the replicated
    // embedding row for the entry call).
    uint16_t *raw_out;        // or nullptr
    const uint16_t *inj_out;  // or nullptr (no fused inject-add)
    const float *inj_gate;
    long inj_stride;
    // One-token path (launch_one_token): every CTA forms inv_rms, act and the
    // gates itself from the down kernel's per-chunk partials (fixed order);
    // CTA 0 also writes them out (act / inv_rms to the workspace, gates).
    const float *part1;       // [S][R], kPartCopies copies part1_stride apart
    const float *ssq1;        // [S], kPartCopies copies kSsqStride apart
    long part1_stride;
    int S, sps, R;
    float eps, inv_H;
    float *act_out;           // [L]
    float *inv_out;           // [C]
    float *gate;              // gates (R > L), or nullptr; token m's at gate + m * gate_stride
    long gate_stride;
    // Optional debug output: w = sigmoid(up(act)) fp32 [M][W], or nullptr.
    float *w_out;
    // One-token path: optional L2 prefetch, before the dependency wait, of the
    // next kernel's weights (the exit's lm_head): 16-byte aligned, a multiple of
    // 16 bytes, or 0.
    const void *l2_pf;
    size_t l2_pf_bytes;
};

struct InjectParams {
    uint16_t *raw;            // bf16 [M][W], in place
    const uint16_t *out;      // bf16 [M][H]
    const float *gate;        // token m's gates at gate + m * gate_stride
    long gate_stride;
    int M, H, C, W;
};

struct ReplicateParams {
    const uint16_t *emb;      // bf16 [M][H]
    uint16_t *raw;            // bf16 [M][C*H]
    int M, H, C;
};

// lm_head after the exit mixer: logits[m][v] = sum_h w[v][h] * mixed[m][h], on
// the tensor cores (hc_tc.cu): 128-row vocabulary tiles against the token rows.
// An optional second weight w2 [V2][H] over the same tokens (V2 = 0: none) runs
// in the same launch: logits2[m][v] = sum_h w2[v][h] * mixed[m][h].
struct LmHeadParams {
    const uint16_t *mixed;    // bf16 [M][H]
    const uint16_t *w;        // bf16 [V][H]
    float *logits;            // fp32 token m's logits at logits + m * logits_stride
    long logits_stride;
    int M, H, V;              // M <= kLmHeadMaxTokens
    const uint16_t *w2;       // bf16 [V2][H], or unused when V2 == 0
    float *logits2;
    long logits2_stride;
    int V2;
    unsigned *status;
};
constexpr int kLmHeadMaxTokens = 16;

// The PLE gate on the wide residual (hc_ple.cu).
struct PleParams {
    uint16_t *hidden;            // bf16 [M][C*H], read and written
    const int32_t *rows;         // [M][16] table row ids
    const uint16_t *table;       // bf16 [n_rows][H/16]
    long n_rows;
    const uint16_t *key_proj;    // bf16 [C*H][H]
    const uint16_t *value_proj;  // bf16 [H][H]
    const uint16_t *norm_key, *norm_query, *norm_conv;  // bf16 [C*H]
    const uint16_t *conv_w;      // bf16 [C*H][4], 8-byte aligned rows
    float *state;                // fp32 [9][C*H], read and written
    uint16_t *emb;               // workspace: bf16 [M][H]
    float *key, *value, *gate, *x;  // workspace: [M][C*H], [M][H], [M][C], [M][C*H]
    int M, H, C;
    float eps, inv_H, inv_sqrt_H;
    unsigned *status;
};

struct LaunchCfg {
    int sm_count;
    bool pdl;                 // launch as a programmatic dependent of the previous kernel
};

// Token-tile width for M tokens (1, 2, 4 or 8) before shared-memory limits.
int gemv_token_tile(int M);
// Shared memory one CTA may use (leaves room for a co-resident dependent CTA).
constexpr size_t kSmemBudget = 200 * 1024;
size_t down_smem_bytes(const DownParams &p, int mt);
size_t up_smem_bytes(const UpParams &p, int mt);
int down_threads(const DownParams &p);
int up_threads(const UpParams &p);

cudaError_t launch_down(const DownParams &p, const LaunchCfg &cfg, cudaStream_t stream);
// One token (M == 1): hc_down1_kernel leaves per-chunk partials in d.part1 /
// d.ssq1 and hc_up1_kernel reduces them (u.part1 / u.ssq1 point at the same
// buffers). one_token_ok says whether a shape fits these kernels' limits.
bool one_token_ok(const DownParams &d, const UpParams &u);
bool few_tokens_ok(const DownParams &d, const UpParams &u);
cudaError_t launch_few_tokens(const DownParams &d, const UpParams &u, const LaunchCfg &cfg, cudaStream_t stream);
cudaError_t launch_one_token(const DownParams &d, const UpParams &u, const LaunchCfg &cfg, cudaStream_t stream);

cudaError_t launch_up(const UpParams &p, const LaunchCfg &cfg, cudaStream_t stream);
cudaError_t launch_inject(const InjectParams &p, const LaunchCfg &cfg, cudaStream_t stream);
// Fills rows_per_cta, rs and n_stages for M tokens; false if H is too wide for the ring.
// Shapes the lm_head kernel takes: 1 <= M <= kLmHeadMaxTokens, H a multiple of 64
// (whole K blocks), V >= 1 (and V2 >= 0).
bool lm_head_shape_ok(int M, int H, int V);
cudaError_t launch_lm_head(const LmHeadParams &p, const LaunchCfg &cfg, cudaStream_t stream);
cudaError_t launch_ple(const PleParams &p, const LaunchCfg &cfg, cudaStream_t stream);
cudaError_t launch_replicate(const ReplicateParams &p, const LaunchCfg &cfg, cudaStream_t stream);

}  // namespace tshc
