/*
 * ts_hc.h -- C ABI of the GB300 (sm_103a) hyper-connection residual call.
 *
 * The operations are those of the qwen4_exp decode flow in the
 * turbospark-runtime 0.3.0 source pages:
 *   - families/qwen4/mod.rs, module doc, "## Hyper-connections": one call maps
 *     the C*H-wide residual `raw` to the H-wide `mixed` and the C-wide gate
 *     `inject_w`;
 *   - families/qwen4/mod.rs, decoder-layer pseudocode and "THE INJECTION
 *     TRAP": the inject-add onto the un-normalized residual;
 *   - families/qwen4/mod.rs, the paragraph on the final
 *     `hyper_connection_mixer` (the call without block_inject_weight);
 *   - families/qwen4/hc.rs, `encode_hyper_connection`: step order, weight
 *     shapes (rows = outputs, cols = inputs) and the per-token inject row.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller. The library
 *     allocates nothing and keeps no state beyond per-device attributes it
 *     queries once. Every call is asynchronous on `stream` (0 = legacy default
 *     stream).
 *   - Row-major everywhere. A wide vector has C*H elements; stream c occupies
 *     elements [c*H, (c+1)*H). Linear weights are [out][in] with no bias.
 *   - bf16 tensors are 16-byte aligned; H is a multiple of 8, hc_lowrank (L)
 *     a multiple of 8 (32 for INT4 weights); 1 <= C <= 8; 8 <= L <= 1024.
 *   - M == 0 (no tokens) is a no-op for every entry point: once the shape
 *     arguments are valid it returns TS_OK without examining any pointer.
 *   - Arguments are validated on the host before anything is launched; a bad
 *     argument returns an error status without launching, and
 *     ts_hc_last_error() names it. Launch failures return TS_ERR_CUDA.
 *   - Results of the GPU path are deterministic: the same inputs give the same
 *     bits on every run (fixed-order split-K reductions, no float atomics).
 *   - A kernel that waits on an asynchronous copy gives up after about one
 *     second, records TS_ERR_TIMEOUT in a device-side status word and returns
 *     without hanging; read it with ts_hc_device_status().
 */
#ifndef TS_HC_H
#define TS_HC_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TS_OK = 0,
    TS_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad size or stride */
    TS_ERR_UNSUPPORTED = 2,   /* valid request outside what this build supports */
    TS_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    TS_ERR_WORKSPACE = 4,     /* workspace missing or smaller than ts_hc_workspace_bytes() */
    TS_ERR_TIMEOUT = 5        /* a device-side wait gave up (see ts_hc_device_status) */
} ts_status;

typedef enum {
    TS_W_BF16 = 0,            /* data: bf16 [out][in] */
    TS_W_INT4_AFFINE = 1      /* data: uint8 [out][in/2], element 2i in the low nibble of
                                 byte i; scales, biases: fp16 [out][in/group];
                                 weight = q * scale + bias, q in [0, 15] */
} ts_wtype;

/* A linear weight [out][in] in its storage format (real_forward.rs,
 * RealForwardRunner doc: projections are INT4-affine quantised or dense). */
typedef struct {
    int32_t type;             /* ts_wtype */
    int32_t group;            /* INT4: inputs per (scale, bias) group: 32, 64 or 128 */
    const void *data;
    const void *scales;       /* INT4 only, else NULL */
    const void *biases;       /* INT4 only, else NULL */
} ts_weight;

/*
 * Bytes of device workspace ts_hc_call / ts_hc_mixer need for M tokens
 * (0 for invalid shapes). The workspace is caller-owned scratch: it need not
 * be initialised, is overwritten by every call, and must not be shared by two
 * calls that can run at the same time.
 *
 * After a successful call the workspace holds two fp32 intermediates of the
 * last call, at the byte offsets ts_hc_workspace_layout() reports:
 *   inv_rms [M][C]: 1/sqrt(mean_h raw[m][c*H+h]^2 + eps), per token and stream;
 *   act     [M][L]: silu(input_mix_weight_down(normed) / C).
 */
size_t ts_hc_workspace_bytes(int M, int H, int C, int lowrank);
ts_status ts_hc_workspace_layout(int M, int H, int C, int lowrank,
                                 size_t *inv_rms_offset, size_t *act_offset);

/*
 * One hyper-connection call (attn_hc / mlp_hc) on M independent tokens
 * (families/qwen4/mod.rs "## Hyper-connections"; families/qwen4/hc.rs
 * encode_hyper_connection):
 *
 *   normed  = hc_norm(raw)                 grouped RMS, group = H, eps inside
 *                                          the root, scale applied directly
 *   act     = silu(down(normed) / C)       C*H -> L
 *   w       = sigmoid(up(act))             L -> C*H, no division
 *   mixed   = mean_c(w[c*H+h] * normed[c*H+h])
 *   gate    = 2 * sigmoid(inject(normed) / C)
 *
 *   raw        bf16 [M][C*H], read only (the caller injects separately)
 *   hc_norm_w  bf16 [C*H] (hc_norm.weight)
 *   down       [L][C*H]   (input_mix_weight_down.weight)
 *   up         [C*H][L]   (input_mix_weight_up.weight)
 *   inject     [C][C*H]   (block_inject_weight.weight)
 *   mixed      bf16 [M][H], written (rounded to nearest even)
 *   inject_w   fp32; token t's C gates are written at inject_w + t*inject_stride
 *              (inject_stride >= C; 2*C with a +C base offset for mlp_hc gives
 *              the per-token row t*C*2 of a shared micro-batch gate buffer)
 *   eps        RMS epsilon (the pages use 1e-6)
 *   workspace  >= ts_hc_workspace_bytes(M, H, C, lowrank) bytes, 256-byte aligned
 *
 * M == 0 is a no-op. Returns TS_OK or an error status (nothing launched on
 * argument errors).
 */
ts_status ts_hc_call(const void *raw, const void *hc_norm_w,
                     const ts_weight *down, const ts_weight *up, const ts_weight *inject,
                     void *mixed, float *inject_w, long inject_stride,
                     int M, int H, int C, int lowrank, float eps,
                     void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * The inject-add (families/qwen4/mod.rs decoder pseudocode and THE INJECTION
 * TRAP): raw[m][c*H+h] += out[m][h] * inject_w[m*inject_stride + c], in place
 * on the UN-normalized residual, computed in fp32 and rounded to bf16 (nearest
 * even).
 *
 *   raw       bf16 [M][C*H], read and written
 *   out       bf16 [M][H], the sublayer output
 *   inject_w  fp32, token m's gates at inject_w + m*inject_stride (inject_stride >= C)
 */
ts_status ts_hc_inject_add(void *raw, const void *out, const float *inject_w,
                           long inject_stride, int M, int H, int C, cudaStream_t stream);

/*
 * The final hyper_connection_mixer (families/qwen4/mod.rs, paragraph after the
 * hyper-connection pseudocode; families/qwen4/hc.rs, has_inject_gate = false):
 * ts_hc_call without block_inject_weight. Writes `mixed` bf16 [M][H] only.
 */
ts_status ts_hc_mixer(const void *raw, const void *hc_norm_w,
                      const ts_weight *down, const ts_weight *up,
                      void *mixed, int M, int H, int C, int lowrank, float eps,
                      void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Test and debugging aid: ts_hc_call (or, with inject == NULL, ts_hc_mixer)
 * that also writes w, the output of the up projection's sigmoid
 * (families/qwen4/mod.rs, "## Hyper-connections": w = sigmoid(up(act)), the
 * per-element mixing weight that multiplies normed before the mean over the
 * streams). The regular entry points keep w on chip.
 *
 *   w_out  fp32 [M][C*H], written: element m*C*H + c*H + h is token m's
 *          weight for stream c at h (the values the same launch mixes)
 *   inject, inject_w, inject_stride  as for ts_hc_call; inject may be NULL
 *          (the exit mixer), and then inject_w is not used
 * Every other output (mixed, the gates, the workspace intermediates) is bit
 * for bit what ts_hc_call / ts_hc_mixer writes for the same inputs: the same
 * kernels run, with one extra store per element of w.
 */
ts_status ts_hc_call_debug(const void *raw, const void *hc_norm_w,
                           const ts_weight *down, const ts_weight *up, const ts_weight *inject,
                           void *mixed, float *inject_w, long inject_stride,
                           int M, int H, int C, int lowrank, float eps,
                           void *workspace, size_t workspace_bytes, float *w_out,
                           cudaStream_t stream);

/*
 * ts_hc_call for callers that cannot allocate device memory. The pages have
 * no counterpart to this entry point; it exists for this library's users.
 *
 * Some callers cannot call cudaMalloc (or any allocator) at the point where
 * they run the call: real-time loops that must not hit the implicit
 * synchronisation an allocation can cause, and hosts that hand this library a
 * fixed memory budget and no allocator. They pass inputs and outputs
 * as for ts_hc_call but no workspace: the scratch lives in a file-scope device
 * array of TS_HC_STATIC_SCRATCH_BYTES that every GPU which loads this library
 * holds until the process exits.
 *
 *   - Shapes whose ts_hc_workspace_bytes() exceeds TS_HC_STATIC_SCRATCH_BYTES
 *     are refused with TS_ERR_WORKSPACE before anything is launched (at the
 *     full shape H=2560, C=4, lowrank=320 that allows up to 1373 tokens).
 *   - The first call on each device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind. Nothing in it needs to start at zero: each call writes every
 *     scratch byte it reads. Calls that can overlap on the GPU (other streams,
 *     other threads) race on it; serialise them.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *
 * Arguments and results as for ts_hc_call, without workspace/workspace_bytes.
 */
#define TS_HC_STATIC_SCRATCH_BYTES (64u * 1024u * 1024u)
ts_status ts_hc_call_noalloc(const void *raw, const void *hc_norm_w,
                             const ts_weight *down, const ts_weight *up, const ts_weight *inject,
                             void *mixed, float *inject_w, long inject_stride,
                             int M, int H, int C, int lowrank, float eps, cudaStream_t stream);

/*
 * The previous sublayer's inject-add fused into the next call
 * (families/qwen4/mod.rs, decoder pseudocode: each `hidden = raw + out * inject_w`
 * is immediately followed by the next attn_hc / mlp_hc, or by the exit mixer).
 * Equivalent, bit for bit, to
 *     ts_hc_inject_add(raw, out, prev_inject_w, prev_inject_stride, ...);
 *     ts_hc_call(raw, ...)            (or ts_hc_mixer when inject == NULL)
 * but with one kernel fewer on the dependency chain: the call reads
 * raw + out * prev_gate directly and writes the updated residual back to raw.
 *
 *   raw            bf16 [M][C*H], read and written (in place)
 *   out            bf16 [M][H], the sublayer output
 *   prev_inject_w  fp32, token m's previous gates at prev_inject_w + m*prev_inject_stride
 *   inject         may be NULL: then this is the exit mixer and inject_w is unused
 *   inject_w       must not share an element with prev_inject_w (two slots of a
 *                  [M][2][C] micro-batch buffer are fine); refused otherwise
 * Other arguments as for ts_hc_call.
 */
ts_status ts_hc_inject_call(void *raw, const void *out, const float *prev_inject_w, long prev_inject_stride,
                            const void *hc_norm_w, const ts_weight *down, const ts_weight *up,
                            const ts_weight *inject, void *mixed, float *inject_w, long inject_stride,
                            int M, int H, int C, int lowrank, float eps,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * The decoder's exit (families/qwen4/mod.rs, decoder pseudocode, exit lines:
 * hidden = hyper_connection_mixer(hidden); logits = lm_head(hidden), with no
 * softcap and no separate final norm), with the last sublayer's inject-add
 * fused in front when `out` is given:
 *     raw += out * prev_inject_w                    (only if out != NULL)
 *     mixed = hyper_connection_mixer(raw)           bf16 [M][H]
 *     logits[m][v] = sum_h lm_head[v][h] * mixed[m][h]   (fp32, mixed as stored)
 * lm_head runs on the tensor cores (bf16 operands, fp32 accumulation) in
 * launches of at most 16 tokens; each launches as a programmatic dependent of
 * the kernel before it and streams its first weight tiles before that kernel
 * has finished. With one token the mixer's up kernel also asks L2 to prefetch
 * the first 24 MB of lm_head while the mixer runs.
 *
 *   raw             bf16 [M][C*H]; read, and written with the fused inject-add
 *   out, prev_inject_w, prev_inject_stride   as for ts_hc_inject_call, or
 *                   out == NULL (then the other two are not used)
 *   hc_norm_w, down, up   the exit mixer's module (no inject weight)
 *   lm_head         bf16 [V][H] (lm_head.weight), 16-byte aligned
 *   mixed           bf16 [M][H], written (the lm_head reads it back)
 *   logits          fp32 [M][V], written
 * Other arguments as for ts_hc_mixer; the workspace is ts_hc_workspace_bytes(M, ...).
 * Any V >= 1 is taken; H must be a multiple of 64 (TS_ERR_UNSUPPORTED
 * otherwise), the other shape rules are those of ts_hc_mixer.
 */
ts_status ts_hc_exit_logits(void *raw, const void *out, const float *prev_inject_w, long prev_inject_stride,
                            const void *hc_norm_w, const ts_weight *down, const ts_weight *up,
                            const void *lm_head, int V, void *mixed, float *logits,
                            int M, int H, int C, int lowrank, float eps,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * PLE, the per-layer embedding gate on the wide residual (families/qwen4/mod.rs,
 * "## PLE": added to the residual before layer index 1's attn_hc, and only
 * there). For M consecutive tokens of one sequence:
 *   emb   = concat of the 16 table rows rows[m][0..16), each H/16 wide
 *   key   = norm_key(key_proj(emb))        value = value_proj(emb)
 *   query = norm_query(hidden)
 *   gate  = sigmoid(s * sqrt(max(|d|, 1e-6))), d = sum_h key[c][h] query[c][h] / sqrt(H),
 *           s the sign of d, per stream c
 *   gv    = gate * value                   (value broadcast to every stream)
 *   hidden += gv + silu(conv(norm_conv(gv)))    (rounded to bf16, in place)
 * The norms are grouped RMS norms in the hyper-connection norm's form (groups
 * of H, eps inside the root, a direct scale per element). conv is depthwise and
 * causal along the token axis: channel j of token t is
 * sum_i conv_w[j][i] * x[t - 3*(3 - i)][j], dilation 3, four taps; the inputs
 * of the 9 tokens before the chunk come from conv_state, which is updated to
 * the chunk's last 9 (zero it for a new sequence). The page notes that this
 * formula was not cross-checked upstream; the hash that picks the row ids is
 * not on the pages, so the caller supplies them.
 *
 *   hidden           bf16 [M][C*H], read and written
 *   rows             int32 [M][16], each in [0, n_rows); an id out of range reads
 *                    zeros and records TS_ERR_INVALID_ARG in the device status word
 *   table            bf16 [n_rows][H/16]
 *   key_proj         bf16 [C*H][H];  value_proj  bf16 [H][H]
 *   norm_*_w         bf16 [C*H] each
 *   conv_w           bf16 [C*H][4]
 *   conv_state       fp32 [9][C*H], oldest token first; read and written
 *   H                a multiple of 128
 *   workspace        >= ts_hc_ple_workspace_bytes(M, H, C) bytes, 256-byte
 *                    aligned; after the call it holds value fp32 [M][H], the
 *                    gates fp32 [M][C] and the conv input x fp32 [M][C*H] at the
 *                    offsets ts_hc_ple_workspace_layout() reports
 */
size_t ts_hc_ple_workspace_bytes(int M, int H, int C);
ts_status ts_hc_ple_workspace_layout(int M, int H, int C, size_t *value_offset, size_t *gate_offset,
                                     size_t *x_offset);
ts_status ts_hc_ple(void *hidden, const int32_t *rows, const void *table, long n_rows,
                    const void *key_proj, const void *value_proj, const void *norm_key_w,
                    const void *norm_query_w, const void *norm_conv_w, const void *conv_w,
                    float *conv_state, int M, int H, int C, float eps,
                    void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Entry replication fused into the stack's first call (families/qwen4/mod.rs,
 * decoder pseudocode: the entry line hidden = embed_tokens(ids).repeat(1, 1, C),
 * followed by layer 0's attn_hc). Equivalent, bit for bit, to
 *     ts_hc_replicate_entry(emb, raw, M, H, C, stream);
 *     ts_hc_call(raw, ...)            (or ts_hc_mixer when inject == NULL)
 * with one kernel fewer: the call reads every stream from the embedding row
 * and writes the replicated residual to raw.
 *
 *   emb   bf16 [M][H], read
 *   raw   bf16 [M][C*H], written (must not overlap emb; refused otherwise)
 * Other arguments as for ts_hc_call; inject may be NULL (then inject_w is not used).
 */
ts_status ts_hc_entry_call(const void *emb, void *raw, const void *hc_norm_w,
                           const ts_weight *down, const ts_weight *up, const ts_weight *inject,
                           void *mixed, float *inject_w, long inject_stride,
                           int M, int H, int C, int lowrank, float eps,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Entry replication (families/qwen4/mod.rs, decoder pseudocode, entry line:
 * the embedding row is repeated C times, not padded):
 * raw[m][c*H + h] = emb[m][h] for every stream c.
 *
 *   emb  bf16 [M][H], read
 *   raw  bf16 [M][C*H], written
 */
ts_status ts_hc_replicate_entry(const void *emb, void *raw, int M, int H, int C, cudaStream_t stream);

/*
 * The decoder stack's hyper-connection path, driven over a prompt in chunks
 * (families/qwen4/mod.rs, decoder-layer pseudocode: entry replication, per
 * layer attn_hc -> sublayer -> inject-add -> mlp_hc -> sublayer -> inject-add,
 * exit hyper_connection_mixer; real_forward.rs, the chunked-prefill driver that
 * runs a prompt through the layers a micro-batch of rows at a time).
 *
 * Tokens do not interact in this path, so the T tokens are processed in
 * chunks of at most max_chunk tokens, one after the other. For each chunk of
 * M tokens starting at token t0:
 *   raw = repeat(emb[t0 .. t0+M), C), fused into layer 0's attn_hc   ts_hc_entry_call
 *   for layer l: attn_hc(attn[l]) -> sublayer(l, 0) -> mlp_hc(mlp[l]) -> sublayer(l, 1),
 *                each inject-add fused into the call after it   ts_hc_inject_call
 *   mixed_out[t0 .. t0+M) = hyper_connection_mixer(final)   (fused with the last inject-add)
 * attn_hc writes token t's gates to slot 0 and mlp_hc to slot 1 of a
 * [M][2][C] gate buffer, i.e. at element t*C*2 and t*C*2 + C (hc.rs,
 * inject_row_offset).
 *
 * The sublayers (GDN / QSA attention, MoE) are the caller's: after every
 * hyper-connection call the driver calls
 *     sublayer(user, layer, which, t0, M, mixed, &out, stream)
 * with `mixed` the call's output (bf16 [M][H], device, valid in stream order
 * until the driver's next launch) and which = 0 after attn_hc, 1 after mlp_hc.
 * The callback may enqueue work on `stream`; it sets `out` to a 16-byte aligned
 * device buffer bf16 [M][H] holding the sublayer output, outside the workspace,
 * which must stay valid until the next hyper-connection call has read it (in
 * stream order). A status other than TS_OK, or a NULL, misaligned or
 * workspace-overlapping `out`, stops the driver, which returns an error; work
 * launched before that point stays queued.
 *
 *   emb        bf16 [T][H], the embedding rows
 *   attn, mlp  n_layers modules each; their inject weights are required
 *   final      the exit mixer's module; its inject is not read
 *   mixed_out  bf16 [T][H], written
 *   max_chunk  >= 1 tokens per chunk
 *   workspace  >= ts_hc_stack_workspace_bytes(max_chunk, H, C, lowrank) bytes,
 *              256-byte aligned; on return it begins with the last chunk's
 *              residual bf16 [M][C*H] after its last inject-add
 * Every module's tensors are validated before anything is launched. The driver
 * allocates nothing and never synchronises, so a caller may capture the whole
 * pass into a CUDA graph when its callback's work is capturable. T == 0 is a
 * no-op.
 */
typedef struct {
    const void *hc_norm_w;    /* bf16 [C*H] */
    ts_weight down;           /* [lowrank][C*H] */
    ts_weight up;             /* [C*H][lowrank] */
    ts_weight inject;         /* [C][C*H]; not read for the exit mixer */
} ts_hc_module;

/*
 * A stack's PLE module (families/qwen4/mod.rs, "## PLE"), the tensors ts_hc_ple
 * takes: table bf16 [n_rows][H/16]; key_proj bf16 [C*H][H]; value_proj bf16
 * [H][H]; norm_key_w, norm_query_w, norm_conv_w bf16 [C*H] each; conv_w bf16
 * [C*H][4]. Every pointer 16-byte aligned.
 */
typedef struct {
    const void *table;
    long n_rows;
    const void *key_proj;
    const void *value_proj;
    const void *norm_key_w;
    const void *norm_query_w;
    const void *norm_conv_w;
    const void *conv_w;
} ts_hc_ple_module;

typedef ts_status (*ts_hc_sublayer_fn)(void *user, int layer, int which, int t0, int M,
                                       const void *mixed, const void **out, cudaStream_t stream);

size_t ts_hc_stack_workspace_bytes(int max_chunk, int H, int C, int lowrank);
ts_status ts_hc_stack(const void *emb, int T, const ts_hc_module *attn, const ts_hc_module *mlp,
                      int n_layers, const ts_hc_module *final_mixer, ts_hc_sublayer_fn sublayer,
                      void *user, void *mixed_out, int max_chunk, int H, int C, int lowrank,
                      float eps, void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * ts_hc_stack with the PLE gate at layer index 1 (families/qwen4/mod.rs, decoder
 * pseudocode: `if layer_idx == 1: hidden = hidden + ple(hidden, input_ids)`
 * before that layer's attn_hc). For each chunk, layer 0's last inject-add is
 * applied on its own (ts_hc_inject_add), then ts_hc_ple on the residual, then
 * layer 1's attn_hc (ts_hc_call); every other step is as in ts_hc_stack.
 *
 *   ple             the PLE module (all of it validated before any launch)
 *   ple_rows        int32 [T][16], token t's 16 table row ids
 *   ple_conv_state  fp32 [9][C*H], the conv inputs of the 9 tokens before token 0
 *                   (zero for a new sequence); read and updated chunk by chunk, so
 *                   on return it holds the last 9 tokens' inputs
 *   n_layers        >= 2 (the PLE layer must exist)
 *   H               a multiple of 128
 *   workspace       >= ts_hc_stack_ple_workspace_bytes(max_chunk, H, C, lowrank)
 * Other arguments and results as for ts_hc_stack.
 */
size_t ts_hc_stack_ple_workspace_bytes(int max_chunk, int H, int C, int lowrank);
ts_status ts_hc_stack_ple(const void *emb, int T, const ts_hc_module *attn, const ts_hc_module *mlp,
                          int n_layers, const ts_hc_module *final_mixer, const ts_hc_ple_module *ple,
                          const int32_t *ple_rows, float *ple_conv_state, ts_hc_sublayer_fn sublayer,
                          void *user, void *mixed_out, int max_chunk, int H, int C, int lowrank,
                          float eps, void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Self-test of the failure path. Launches one thread that waits, with the same
 * bounded wait the kernels use for their asynchronous copies, on a
 * shared-memory barrier that nothing arrives at. After about one second it
 * gives up and records TS_ERR_TIMEOUT in the device status word, as a kernel
 * whose copy never completed would; ts_hc_device_status() then reports it and
 * clears it. Nothing else is read or written, and the context stays usable.
 * Returns TS_OK once launched (asynchronous on `stream`).
 */
ts_status ts_hc_selftest_timeout(cudaStream_t stream);

/* The last error message of the calling thread ("" if none). */
const char *ts_hc_last_error(void);

/*
 * Reads the device-side status word of the current device (synchronising
 * `stream`) into *status (TS_OK or TS_ERR_TIMEOUT) and clears it. Returns
 * TS_ERR_CUDA if the read itself fails.
 */
ts_status ts_hc_device_status(cudaStream_t stream, int *status);

#ifdef __cplusplus
}
#endif

#endif /* TS_HC_H */
