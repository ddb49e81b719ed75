/*
 * hc_oracle.c -- plain fp64 CPU oracle for the hyper-connection residual call.
 *
 * TEST INFRASTRUCTURE ONLY. This is the reference that the CUDA library is
 * checked against. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it; the product path never does. It shares no
 * code, header, table or helper with the CUDA library.
 *
 * Source of every formula: the turbospark-runtime 0.3.0 source pages
 *   [mod]  families/qwen4/mod.rs, module doc:
 *          "## The decoder layer, as pseudocode" (entry replication, the
 *          inject-add, the exit mixer), "THE INJECTION TRAP",
 *          "## Hyper-connections" (the call itself), "## PLE" (orc_ple, with
 *          its own readings), and `RMS_EPS = 1e-6`.
 *   [hc]   families/qwen4/hc.rs, `encode_hyper_connection`: step order, the
 *          weight shapes as (rows = outputs, cols = inputs), the remark that
 *          there are exactly two divisions by C, and the per-token inject row.
 *   [rf]   real_forward.rs, `RealForwardRunner` doc: weights are
 *          INT4-affine quantised (format details are not on the pages).
 *
 * Everything is evaluated in double precision on the exact values of the
 * inputs (bf16 and fp16 bit patterns are decoded exactly), with no
 * intermediate rounding, no blocking, no fusion and no reordering beyond the
 * plain definition. Loops are sequential sums in index order. OpenMP only
 * splits independent output rows across threads; it does not change any sum.
 *
 * Readings taken where the pages leave a step open:
 *   R1  RMSNorm ([mod] "grouped RMS, group=H"): r_c = 1/sqrt(mean_h x^2 + eps)
 *       with eps inside the root, the mean over the H elements of stream c.
 *   R2  The norm scale is applied directly (no 1+g) ([mod] header, [hc] doc),
 *       one scale per element of the C*H-wide vector (the norm view is
 *       C*H long in [hc]).
 *   R3  Linear weights are row-major [out][in] and carry no bias ([hc] names
 *       only `.weight` tensors and passes (rows = out, cols = in)).
 *   R4  Stream c of a wide vector is elements [c*H, (c+1)*H) (view(C, H) and
 *       flatten() of a row-major tensor, [mod]).
 *   R5  The two divisions by C are on the down output (before silu) and on
 *       the inject output (before sigmoid); the up path has none ([hc]).
 *       The mix is a mean over the C streams ([mod] "MEAN not sum").
 *   R6  silu(x) = x * sigmoid(x), sigmoid(x) = 1/(1+exp(-x)).
 *   R7  INT4-affine ([rf] names the format only): per output row, groups of
 *       `group` consecutive inputs share one fp16 scale s and one fp16 bias b;
 *       the weight is q*s + b with q in [0, 15]; element 2i sits in the low
 *       nibble of byte i, element 2i+1 in the high nibble.
 */

#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_WEIGHT_BF16 0
#define ORC_WEIGHT_INT4_AFFINE 1

/* A weight matrix in its storage format. Rows are outputs, columns inputs. */
typedef struct {
    int32_t kind;           /* ORC_WEIGHT_BF16 or ORC_WEIGHT_INT4_AFFINE */
    int32_t group;          /* INT4: inputs per (scale, bias) group */
    int64_t rows;
    int64_t cols;
    const uint16_t *bf16;   /* kind 0: bf16 bit patterns, [rows][cols] */
    const uint8_t *packed;  /* kind 1: [rows][cols/2] */
    const uint16_t *scale;  /* kind 1: fp16 bit patterns, [rows][cols/group] */
    const uint16_t *bias;   /* kind 1: fp16 bit patterns, [rows][cols/group] */
} orc_weight;

/* ---- exact decoding of the storage formats ---------------------------- */

/* bf16: 1 sign bit, 8 exponent bits (bias 127), 7 mantissa bits. */
double orc_bf16_value(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int exponent = (bits >> 7) & 0xFF;
    int mantissa = bits & 0x7F;
    double v;
    if (exponent == 0)
        v = ldexp((double)mantissa, -133);              /* subnormal: m * 2^(1-127-7) */
    else if (exponent == 0xFF)
        v = mantissa ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + mantissa), exponent - 134);  /* 1.m * 2^(e-127) */
    return sign ? -v : v;
}

/* IEEE half: 1 sign bit, 5 exponent bits (bias 15), 10 mantissa bits. */
double orc_f16_value(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int exponent = (bits >> 10) & 0x1F;
    int mantissa = bits & 0x3FF;
    double v;
    if (exponent == 0)
        v = ldexp((double)mantissa, -24);               /* subnormal: m * 2^(1-15-10) */
    else if (exponent == 0x1F)
        v = mantissa ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + mantissa), exponent - 25);  /* 1.m * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a double to the nearest bf16 value, ties to even. Used only where the
 * workload stores a tensor in bf16 (the residual carried between layers). */
double orc_round_to_bf16(double x)
{
    if (x == 0.0 || isnan(x) || isinf(x))
        return x;
    int e;
    double f = frexp(fabs(x), &e);      /* |x| = f * 2^e, f in [0.5, 1) */
    int shift = 8;                      /* 8 significant bits: 1 implicit + 7 stored */
    if (e - shift < -133)               /* below the normal range: fixed spacing 2^-133 */
        shift = e + 133;
    double scaled = ldexp(f, shift);
    double r = nearbyint(scaled);       /* default rounding mode: to nearest, ties to even */
    double v = ldexp(r, e - shift);
    if (v > ldexp(255.0, 120))          /* beyond the largest finite bf16 */
        v = INFINITY;
    return x < 0 ? -v : v;
}

void orc_round_to_bf16_array(const double *x, double *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        y[i] = orc_round_to_bf16(x[i]);
}

/* Value of weight element (o, i). */
double orc_weight_at(const orc_weight *w, int64_t o, int64_t i)
{
    if (w->kind == ORC_WEIGHT_BF16)
        return orc_bf16_value(w->bf16[o * w->cols + i]);
    uint8_t byte = w->packed[o * (w->cols / 2) + i / 2];
    int q = (i % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
    int64_t gi = o * (w->cols / w->group) + i / w->group;
    return (double)q * orc_f16_value(w->scale[gi]) + orc_f16_value(w->bias[gi]);
}

/* y = W x, y[o] = sum_i W[o, i] x[i], summed in index order. */
void orc_gemv(const orc_weight *w, const double *x, double *y, int nthreads)
{
    int64_t rows = w->rows, cols = w->cols;
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(static)
    for (int64_t o = 0; o < rows; ++o) {
        double acc = 0.0;
        for (int64_t i = 0; i < cols; ++i)
            acc += orc_weight_at(w, o, i) * x[i];
        y[o] = acc;
    }
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
static double silu(double x) { return x * sigmoid(x); }

/*
 * One hyper-connection call on M independent tokens ([mod] "## Hyper-
 * connections"; [hc] encode_hyper_connection). With `inject == NULL` this is
 * the final hyper_connection_mixer, which has no block_inject_weight and
 * returns `mixed` alone ([mod], paragraph after the pseudocode; [hc] doc).
 *
 *   raw      [M][C*H]  the wide residual, read only
 *   g        [C*H]     hc_norm.weight
 *   down     L x C*H   input_mix_weight_down.weight
 *   up       C*H x L   input_mix_weight_up.weight
 *   inject   C x C*H   block_inject_weight.weight, or NULL
 *   mixed    [M][H]    output
 *   gate     token m's C gates at gate + m*gate_stride (ignored when inject is NULL)
 *   inv_rms  [M][C], a [M][L], w [M][C*H]: optional intermediates (NULL skips)
 *
 * Returns 0, or -1 on inconsistent shapes.
 */
int orc_hc_call(int64_t M, int64_t H, int64_t C, int64_t L, double eps,
                const double *raw, const double *g,
                const orc_weight *down, const orc_weight *up, const orc_weight *inject,
                double *mixed, double *gate, int64_t gate_stride,
                double *inv_rms, double *a, double *w, int nthreads)
{
    const int64_t W = C * H;
    if (M < 0 || H < 1 || C < 1 || L < 1)
        return -1;
    if (down->rows != L || down->cols != W || up->rows != W || up->cols != L)
        return -1;
    if (inject && (inject->rows != C || inject->cols != W || gate_stride < C))
        return -1;

    for (int64_t m = 0; m < M; ++m) {
        const double *x = raw + m * W;
        double normed[W];                 /* C99 VLA: sizes here are at most a few 10^4 */
        double r[C], z[L], act[L], y[W];

        /* normed = hc_norm(raw): grouped RMS, group = H, direct scale (R1, R2). */
        for (int64_t c = 0; c < C; ++c) {
            double ss = 0.0;
            for (int64_t h = 0; h < H; ++h)
                ss += x[c * H + h] * x[c * H + h];
            r[c] = 1.0 / sqrt(ss / (double)H + eps);
            for (int64_t h = 0; h < H; ++h)
                normed[c * H + h] = x[c * H + h] * r[c] * g[c * H + h];
        }

        /* w = silu(input_mix_weight_down(normed) / C)   (R5, R6) */
        orc_gemv(down, normed, z, nthreads);
        for (int64_t k = 0; k < L; ++k)
            act[k] = silu(z[k] / (double)C);

        /* w = sigmoid(input_mix_weight_up(w)) -- no division (R5) */
        orc_gemv(up, act, y, nthreads);
        for (int64_t j = 0; j < W; ++j)
            y[j] = sigmoid(y[j]);

        /* mixed = (w.view(C,H) * normed.view(C,H)).mean(dim=C)   (R4, R5) */
        for (int64_t h = 0; h < H; ++h) {
            double s = 0.0;
            for (int64_t c = 0; c < C; ++c)
                s += y[c * H + h] * normed[c * H + h];
            mixed[m * H + h] = s / (double)C;
        }

        /* inject_w = 2 * sigmoid(block_inject_weight(normed) / C)   (R5) */
        if (inject) {
            double q[C];
            orc_gemv(inject, normed, q, nthreads);
            for (int64_t c = 0; c < C; ++c)
                gate[m * gate_stride + c] = 2.0 * sigmoid(q[c] / (double)C);
        }

        if (inv_rms)
            memcpy(inv_rms + m * C, r, sizeof(double) * (size_t)C);
        if (a)
            memcpy(a + m * L, act, sizeof(double) * (size_t)L);
        if (w)
            memcpy(w + m * W, y, sizeof(double) * (size_t)W);
    }
    return 0;
}

/*
 * The inject-add ([mod] decoder pseudocode and "THE INJECTION TRAP"):
 *   hidden = raw + (out[.., None, :] * inject_w[.., :, None]).flatten()
 * onto the UN-normalized residual `raw`, element c*H + h gaining out[h]*gate[c].
 *
 *   raw [M][C*H], out [M][H], token m's gates at gate + m*gate_stride,
 *   result [M][C*H] (may alias raw).
 */
void orc_inject_add(int64_t M, int64_t H, int64_t C, const double *raw,
                    const double *out, const double *gate, int64_t gate_stride,
                    double *result)
{
    const int64_t W = C * H;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t c = 0; c < C; ++c)
            for (int64_t h = 0; h < H; ++h)
                result[m * W + c * H + h] =
                    raw[m * W + c * H + h] + out[m * H + h] * gate[m * gate_stride + c];
}

/* Entry replication ([mod] decoder pseudocode, entry line): the embedding row
 * is repeated C times, not padded: raw[m][c*H + h] = emb[m][h]. */
void orc_replicate_entry(int64_t M, int64_t H, int64_t C, const double *emb, double *raw)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t c = 0; c < C; ++c)
            for (int64_t h = 0; h < H; ++h)
                raw[m * C * H + c * H + h] = emb[m * H + h];
}

/*
 * PLE, the per-layer embedding gate on the wide residual ([mod] "## PLE",
 * layer index 1 only; decoder pseudocode: hidden = hidden + ple(hidden, ids)
 * before that layer's attn_hc). [mod] warns that this formula, unlike the
 * hyper-connection one, was not cross-checked against the upstream source.
 * Readings taken where the section is open:
 *   P1  The 16 row ids per token (ngram_hash of the token history) are inputs:
 *       the hash is not on the pages. emb is the concatenation of the 16 table
 *       rows, each H/16 wide, in row-id order.
 *   P2  key_proj [C*H][H] and value_proj [H][H] are bias-free [out][in] weights.
 *   P3  norm_key, norm_query and norm_conv are each "grouped scaled" RMS norms
 *       of a C*H vector in the hyper-connection norm's form (R1, R2): groups of
 *       H, eps inside the root, a direct scale with one entry per element.
 *   P4  gate_c = sum_h key[c][h] * query[c][h] / sqrt(H), then the signed square
 *       root sign(g) * sqrt(max(|g|, 1e-6)) (sign(0) = 0), then sigmoid.
 *   P5  gv[c][h] = sigmoid(gate_c) * value[h] (value broadcast to every stream).
 *   P6  dilated_conv is a depthwise causal convolution along the token axis:
 *       channel j of token t is sum_{i<4} conv_w[j][i] * x[t - 3*(3 - i)][j],
 *       x = norm_conv(gv); tokens before the first come from `state` (the x of
 *       the 9 tokens before this chunk, oldest first), and state_out holds the
 *       x of the chunk's last 9 tokens (taken from state where M < 9).
 *   P7  out = gv + silu(conv); the result is hidden + out (the caller stores it).
 *
 *   hidden [M][W], rows [M][16], table [n_rows][H/16] (bf16 bits), conv_w [W][4]
 *   (bf16 bits), norm scales [W] each (values), state [9][W]; outputs: result
 *   [M][W], state_out [9][W], and optional intermediates key [M][W], value
 *   [M][H], gate [M][C] (after the sigmoid), x [M][W] (NULL skips).
 * Returns 0, or -1 on inconsistent arguments (a row id out of range included).
 */
int orc_ple(int64_t M, int64_t H, int64_t C, double eps, const double *hidden, const int32_t *rows,
            const uint16_t *table, int64_t n_rows, const orc_weight *key_proj, const orc_weight *value_proj,
            const double *norm_key, const double *norm_query, const double *norm_conv,
            const uint16_t *conv_w, const double *state, double *result, double *state_out,
            double *key_out, double *value_out, double *gate_out, double *x_out, int nthreads)
{
    const int64_t W = C * H, seg = H / 16;
    if (M < 0 || H < 16 || H % 16 != 0 || C < 1)
        return -1;
    if (key_proj->rows != W || key_proj->cols != H || value_proj->rows != H || value_proj->cols != H)
        return -1;
    double *xs = (double *)malloc(sizeof(double) * (size_t)(M + 9) * (size_t)W);  /* state, then the chunk's x */
    if (!xs)
        return -1;
    memcpy(xs, state, sizeof(double) * 9 * (size_t)W);
    for (int64_t m = 0; m < M; ++m) {
        double emb[H], key[W], value[H], query[W], gv[W];
        /* emb = concat(table[rows[h]] for h in 0..16)   (P1) */
        for (int64_t r = 0; r < 16; ++r) {
            const int64_t id = rows[m * 16 + r];
            if (id < 0 || id >= n_rows) {
                free(xs);
                return -1;
            }
            for (int64_t e = 0; e < seg; ++e)
                emb[r * seg + e] = orc_bf16_value(table[id * seg + e]);
        }
        /* key = norm_key(key_proj(emb)), value = value_proj(emb)   (P2, P3) */
        orc_gemv(key_proj, emb, key, nthreads);
        orc_gemv(value_proj, emb, value, nthreads);
        const double *hm = hidden + m * W;
        double gate[C];
        for (int64_t c = 0; c < C; ++c) {
            double sk = 0.0, sq = 0.0;
            for (int64_t h = 0; h < H; ++h) {
                sk += key[c * H + h] * key[c * H + h];
                sq += hm[c * H + h] * hm[c * H + h];
            }
            const double rk = 1.0 / sqrt(sk / (double)H + eps), rq = 1.0 / sqrt(sq / (double)H + eps);
            double dot = 0.0;
            for (int64_t h = 0; h < H; ++h) {
                const double kn = key[c * H + h] * rk * norm_key[c * H + h];
                query[c * H + h] = hm[c * H + h] * rq * norm_query[c * H + h];
                dot += kn * query[c * H + h];
                key[c * H + h] = kn;
            }
            /* gate = (key * query).sum(-1) / sqrt(H), signed square root   (P4) */
            const double g = dot / sqrt((double)H);
            const double sg = (g > 0.0) - (g < 0.0);
            gate[c] = sigmoid(sg * sqrt(fmax(fabs(g), 1e-6)));
        }
        /* gv = sigmoid(gate) * value, x = norm_conv(gv)   (P5, P3) */
        double *x = xs + (9 + m) * W;
        for (int64_t c = 0; c < C; ++c) {
            double sv = 0.0;
            for (int64_t h = 0; h < H; ++h) {
                gv[c * H + h] = gate[c] * value[h];
                sv += gv[c * H + h] * gv[c * H + h];
            }
            const double r = 1.0 / sqrt(sv / (double)H + eps);
            for (int64_t h = 0; h < H; ++h)
                x[c * H + h] = gv[c * H + h] * r * norm_conv[c * H + h];
        }
        /* out = gv + silu(dilated_conv(x)); result = hidden + out   (P6, P7) */
        for (int64_t j = 0; j < W; ++j) {
            double y = 0.0;
            for (int64_t i = 0; i < 4; ++i)
                y += orc_bf16_value(conv_w[j * 4 + i]) * xs[(9 + m - 3 * (3 - i)) * W + j];
            result[m * W + j] = hm[j] + (gv[j] + silu(y));
        }
        if (key_out)
            memcpy(key_out + m * W, key, sizeof(double) * (size_t)W);
        if (value_out)
            memcpy(value_out + m * H, value, sizeof(double) * (size_t)H);
        if (gate_out)
            memcpy(gate_out + m * C, gate, sizeof(double) * (size_t)C);
        if (x_out)
            memcpy(x_out + m * W, x, sizeof(double) * (size_t)W);
    }
    memcpy(state_out, xs + M * W, sizeof(double) * 9 * (size_t)W);
    free(xs);
    return 0;
}
