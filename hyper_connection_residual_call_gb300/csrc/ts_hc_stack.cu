// ts_hc_stack.cu -- the decoder stack's hyper-connection path over a prompt,
// chunk by chunk (ts_hc_stack and ts_hc_stack_ple in include/ts_hc.h). Host code only: it
// sequences the library's own entry points on one stream and allocates
// nothing.
//
// families/qwen4/mod.rs, decoder-layer pseudocode: the residual enters as the
// embedding row repeated C times, each layer reads it through attn_hc and
// mlp_hc and adds the sublayer outputs back with the inject gates, and the
// exit hyper_connection_mixer collapses it to H. real_forward.rs describes the
// chunked-prefill driver that runs a prompt through the layers one
// micro-batch of rows at a time; in this path tokens do not interact, so the
// chunks are independent and run one after the other.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>

#include "ts_hc.h"
#include "ts_hc_internal.h"

namespace {

size_t a256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace of the driver: the chunk's residual, the calls' mixed output, the
// chunk's [M][2][C] gate buffer, the calls' own workspace (the largest any
// chunk size up to max_chunk needs), then, with the PLE, its workspace.
struct StackWs {
    size_t raw, mixed, gates, call, call_bytes, ple, ple_bytes, total;
};

StackWs stack_ws(int max_chunk, int H, int C, int L, bool with_ple)
{
    StackWs w{};
    const size_t M = (size_t)max_chunk, W = (size_t)C * H;
    w.raw = 0;
    w.mixed = a256(2 * M * W);
    w.gates = w.mixed + a256(2 * M * H);
    w.call = w.gates + a256(4 * M * 2 * C);
    size_t need = 0;
    for (int m = 1; m <= max_chunk; ++m)
        need = std::max(need, ts_hc_workspace_bytes(m, H, C, L));
    w.call_bytes = a256(need);
    w.ple = w.call + w.call_bytes;
    w.ple_bytes = with_ple ? a256(ts_hc_ple_workspace_bytes(max_chunk, H, C)) : 0;  // grows with M
    w.total = w.ple + w.ple_bytes;
    return w;
}

const char *sublayer_name(int which) { return which == 0 ? "attention" : "MoE"; }

// The PLE step of a stack: module, row ids [T][16], conv state.
struct StackPle {
    const ts_hc_ple_module *mod;
    const int32_t *rows;
    float *state;
};

ts_status stack_impl(const void *emb, int T, const ts_hc_module *attn, const ts_hc_module *mlp, int n_layers,
                     const ts_hc_module *final_mixer, const StackPle *ple, ts_hc_sublayer_fn sublayer,
                     void *user, void *mixed_out, int max_chunk, int H, int C, int lowrank, float eps,
                     void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    using tshc::api_error;
    if (T < 0)
        return api_error(TS_ERR_INVALID_ARG, "T = %d must be >= 0", T);
    if (n_layers < 0)
        return api_error(TS_ERR_INVALID_ARG, "n_layers = %d must be >= 0", n_layers);
    if (max_chunk < 1)
        return api_error(TS_ERR_INVALID_ARG, "max_chunk = %d must be >= 1", max_chunk);
    ts_status st = tshc::check_shape_api(max_chunk, H, C, lowrank);
    if (st != TS_OK)
        return st;
    if (T == 0)  // nothing is read or written: pointers are not examined
        return TS_OK;

    // Everything is validated before the first launch.
    if ((st = tshc::check_ptr_api(emb, "emb", 16)) != TS_OK) return st;
    if ((st = tshc::check_ptr_api(mixed_out, "mixed_out", 16)) != TS_OK) return st;
    if (!(eps >= 0.0f) || eps > 1.0f)
        return api_error(TS_ERR_INVALID_ARG, "eps = %g must be in [0, 1]", (double)eps);
    if (n_layers > 0) {
        if (!attn || !mlp)
            return api_error(TS_ERR_INVALID_ARG, "%s is NULL with n_layers = %d", attn ? "mlp" : "attn", n_layers);
        if (!sublayer)
            return api_error(TS_ERR_INVALID_ARG, "sublayer is NULL with n_layers = %d", n_layers);
        char name[64];
        for (int l = 0; l < n_layers; ++l) {
            snprintf(name, sizeof name, "attn[%d]", l);
            if ((st = tshc::check_module(attn + l, true, H, C, lowrank, name)) != TS_OK) return st;
            snprintf(name, sizeof name, "mlp[%d]", l);
            if ((st = tshc::check_module(mlp + l, true, H, C, lowrank, name)) != TS_OK) return st;
        }
    }
    if ((st = tshc::check_module(final_mixer, false, H, C, lowrank, "final_mixer")) != TS_OK)
        return st;
    if (ple) {
        if (n_layers < 2)
            return api_error(TS_ERR_INVALID_ARG, "the PLE runs before layer 1, but n_layers = %d", n_layers);
        if ((st = tshc::check_ple_shape(H, C)) != TS_OK) return st;
        if ((st = tshc::check_ple_module(ple->mod)) != TS_OK) return st;
        if ((st = tshc::check_ptr_api(ple->rows, "ple_rows", 4)) != TS_OK) return st;
        if ((st = tshc::check_ptr_api(ple->state, "ple_conv_state", 16)) != TS_OK) return st;
    }
    const StackWs lay = stack_ws(max_chunk, H, C, lowrank, ple != nullptr);
    if (!workspace || workspace_bytes < lay.total)
        return api_error(TS_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed", workspace_bytes, lay.total);
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return api_error(TS_ERR_INVALID_ARG, "workspace is not 256-byte aligned");

    char *ws = static_cast<char *>(workspace);
    void *raw = ws + lay.raw;
    void *mixed = ws + lay.mixed;
    float *gates = reinterpret_cast<float *>(ws + lay.gates);
    void *cws = ws + lay.call;
    const long gstride = 2L * C;  // token t's slots at t*C*2 (attn_hc) and t*C*2 + C (mlp_hc)

    for (int t0 = 0; t0 < T; t0 += max_chunk) {
        const int M = std::min(max_chunk, T - t0);
        const void *emb_t = static_cast<const char *>(emb) + 2 * (size_t)t0 * H;
        if (n_layers == 0) {  // the exit mixer reads the replicated embedding directly
            st = ts_hc_replicate_entry(emb_t, raw, M, H, C, stream);
            if (st != TS_OK)
                return st;
        }
        const void *prev_out = nullptr;  // the last sublayer output, not yet injected
        const float *prev_gate = nullptr;
        for (int l = 0; l < n_layers; ++l) {
            for (int which = 0; which < 2; ++which) {
                const ts_hc_module &m = which == 0 ? attn[l] : mlp[l];
                float *slot = gates + which * C;
                if (ple && l == 1 && which == 0) {
                    // Layer 1: layer 0's last inject-add, the PLE on the residual, then attn_hc.
                    const ts_hc_ple_module &q = *ple->mod;
                    if ((st = ts_hc_inject_add(raw, prev_out, prev_gate, gstride, M, H, C, stream)) != TS_OK)
                        return st;
                    st = ts_hc_ple(raw, ple->rows + 16 * (size_t)t0, q.table, q.n_rows, q.key_proj, q.value_proj,
                                   q.norm_key_w, q.norm_query_w, q.norm_conv_w, q.conv_w, ple->state, M, H, C, eps,
                                   ws + lay.ple, lay.ple_bytes, stream);
                    if (st != TS_OK)
                        return st;
                    st = ts_hc_call(raw, m.hc_norm_w, &m.down, &m.up, &m.inject, mixed, slot, gstride, M, H, C,
                                    lowrank, eps, cws, lay.call_bytes, stream);
                } else {
                    // Layer 0's attn_hc reads the embedding row in every stream and
                    // writes the replicated residual (the entry line, fused).
                    st = l == 0 && which == 0
                             ? ts_hc_entry_call(emb_t, raw, m.hc_norm_w, &m.down, &m.up, &m.inject, mixed, slot,
                                                gstride, M, H, C, lowrank, eps, cws, lay.call_bytes, stream)
                             : ts_hc_inject_call(raw, prev_out, prev_gate, gstride, m.hc_norm_w, &m.down, &m.up,
                                                 &m.inject, mixed, slot, gstride, M, H, C, lowrank, eps, cws,
                                                 lay.call_bytes, stream);
                }
                if (st != TS_OK)
                    return st;
                const void *out = nullptr;
                st = sublayer(user, l, which, t0, M, mixed, &out, stream);
                if (st != TS_OK)
                    return api_error(st, "the %s sublayer callback of layer %d (tokens %d..%d) returned status %d",
                                     sublayer_name(which), l, t0, t0 + M - 1, (int)st);
                if (!out || reinterpret_cast<uintptr_t>(out) % 16 != 0)
                    return api_error(TS_ERR_INVALID_ARG,
                                     "the %s sublayer callback of layer %d gave %s output pointer",
                                     sublayer_name(which), l, out ? "a misaligned" : "a NULL");
                // The next call overwrites the workspace (mixed included) while it reads out.
                const char *o = static_cast<const char *>(out);
                if (o < ws + lay.total && o + 2 * (size_t)M * H > ws)
                    return api_error(TS_ERR_INVALID_ARG,
                                     "the %s sublayer callback of layer %d gave an output inside the workspace",
                                     sublayer_name(which), l);
                prev_out = out;
                prev_gate = slot;
            }
        }
        void *mo = static_cast<char *>(mixed_out) + 2 * (size_t)t0 * H;
        const ts_hc_module &f = *final_mixer;
        st = prev_out == nullptr
                 ? ts_hc_mixer(raw, f.hc_norm_w, &f.down, &f.up, mo, M, H, C, lowrank, eps, cws, lay.call_bytes,
                               stream)
                 : ts_hc_inject_call(raw, prev_out, prev_gate, gstride, f.hc_norm_w, &f.down, &f.up, nullptr,
                                     mo, nullptr, 0, M, H, C, lowrank, eps, cws, lay.call_bytes, stream);
        if (st != TS_OK)
            return st;
    }
    return TS_OK;
}

}  // namespace

extern "C" {

size_t ts_hc_stack_workspace_bytes(int max_chunk, int H, int C, int lowrank)
{
    if (max_chunk < 1 || tshc::check_shape_api(max_chunk, H, C, lowrank) != TS_OK) {
        tshc::clear_error();
        return 0;
    }
    return stack_ws(max_chunk, H, C, lowrank, false).total;
}

size_t ts_hc_stack_ple_workspace_bytes(int max_chunk, int H, int C, int lowrank)
{
    if (max_chunk < 1 || tshc::check_shape_api(max_chunk, H, C, lowrank) != TS_OK ||
        tshc::check_ple_shape(H, C) != TS_OK) {
        tshc::clear_error();
        return 0;
    }
    return stack_ws(max_chunk, H, C, lowrank, true).total;
}

ts_status ts_hc_stack(const void *emb, int T, const ts_hc_module *attn, const ts_hc_module *mlp,
                      int n_layers, const ts_hc_module *final_mixer, ts_hc_sublayer_fn sublayer,
                      void *user, void *mixed_out, int max_chunk, int H, int C, int lowrank,
                      float eps, void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    tshc::clear_error();
    return stack_impl(emb, T, attn, mlp, n_layers, final_mixer, nullptr, sublayer, user, mixed_out, max_chunk, H, C,
                      lowrank, eps, workspace, workspace_bytes, stream);
}

ts_status ts_hc_stack_ple(const void *emb, int T, const ts_hc_module *attn, const ts_hc_module *mlp,
                          int n_layers, const ts_hc_module *final_mixer, const ts_hc_ple_module *ple,
                          const int32_t *ple_rows, float *ple_conv_state, ts_hc_sublayer_fn sublayer,
                          void *user, void *mixed_out, int max_chunk, int H, int C, int lowrank,
                          float eps, void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    tshc::clear_error();
    const StackPle p{ple, ple_rows, ple_conv_state};
    return stack_impl(emb, T, attn, mlp, n_layers, final_mixer, &p, sublayer, user, mixed_out, max_chunk, H, C,
                      lowrank, eps, workspace, workspace_bytes, stream);
}

}  // extern "C"
