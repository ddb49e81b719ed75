// ts_hc_api.cu -- the C ABI of include/ts_hc.h: argument validation on the
// host, launch geometry, and the kernel launches. Allocates nothing.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "hc_kernels.h"
#include "hc_tc.h"
#include "ptx.cuh"
#include "ts_hc.h"
#include "ts_hc_internal.h"

namespace {

thread_local std::string g_last_error;

ts_status fail(ts_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

ts_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(TS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device-side status word: kernels record a timed-out wait here.
__device__ unsigned int g_device_status;

constexpr int kMaxDevices = 64;
constexpr int kMaxC = 8;
constexpr int kMaxL = 1024;
constexpr int kMaxH = 16384;

struct DeviceInfo {
    int sm_count = 0;
    unsigned *status = nullptr;
    bool ready = false;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];

ts_status device_info(DeviceInfo *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(TS_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(MultiProcessorCount)");
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_device_status);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(device status)");
        d.ready = true;
    }
    *out = d;
    return TS_OK;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

ts_status check_shape(int M, int H, int C, int L)
{
    if (M < 0)
        return fail(TS_ERR_INVALID_ARG, "M = %d must be >= 0", M);
    if (H < 8 || H % 8 != 0 || H > kMaxH)
        return fail(TS_ERR_INVALID_ARG, "H = %d must be a multiple of 8 in [8, %d]", H, kMaxH);
    if (C < 1 || C > kMaxC)
        return fail(TS_ERR_INVALID_ARG, "C = %d must be in [1, %d]", C, kMaxC);
    if (L < 8 || L % 8 != 0 || L > kMaxL)
        return fail(TS_ERR_INVALID_ARG, "lowrank = %d must be a multiple of 8 in [8, %d]", L, kMaxL);
    return TS_OK;
}

ts_status check_ptr(const void *p, const char *name, size_t align)
{
    if (!p)
        return fail(TS_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned(p, align))
        return fail(TS_ERR_INVALID_ARG, "%s is not %zu-byte aligned", name, align);
    return TS_OK;
}

ts_status check_weight(const ts_weight *w, const char *name, int rows, int cols)
{
    (void)rows;
    if (!w)
        return fail(TS_ERR_INVALID_ARG, "%s is NULL", name);
    if (w->type == TS_W_BF16) {
        if (!w->data || !aligned(w->data, 16))
            return fail(TS_ERR_INVALID_ARG, "%s.data must be a 16-byte aligned device pointer", name);
        return TS_OK;
    }
    if (w->type == TS_W_INT4_AFFINE) {
        if (w->group != 32 && w->group != 64 && w->group != 128)
            return fail(TS_ERR_UNSUPPORTED, "%s.group = %d: INT4 groups of 32, 64 or 128 are supported",
                        name, w->group);
        if (cols % w->group != 0 || cols % 32 != 0)
            return fail(TS_ERR_UNSUPPORTED, "%s: %d inputs are not a multiple of the group %d and of 32",
                        name, cols, w->group);
        if (!w->data || !aligned(w->data, 16))
            return fail(TS_ERR_INVALID_ARG, "%s.data must be a 16-byte aligned device pointer", name);
        if (!w->scales || !aligned(w->scales, 2) || !w->biases || !aligned(w->biases, 2))
            return fail(TS_ERR_INVALID_ARG, "%s.scales / %s.biases must be 2-byte aligned device pointers",
                        name, name);
        return TS_OK;
    }
    return fail(TS_ERR_INVALID_ARG, "%s.type = %d is not a ts_wtype", name, (int)w->type);
}

tshc::WeightView view(const ts_weight *w)
{
    tshc::WeightView v{};
    if (!w)
        return v;
    v.type = w->type;
    v.group = w->type == TS_W_INT4_AFFINE ? w->group : 0;
    while (v.group > 0 && (1 << v.gshift) < v.group)
        ++v.gshift;
    v.data = w->data;
    v.scales = static_cast<const uint16_t *>(w->scales);
    v.biases = static_cast<const uint16_t *>(w->biases);
    return v;
}

}  // namespace

namespace tshc {

void clear_error() { g_last_error.clear(); }

ts_status api_error(ts_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

ts_status check_shape_api(int M, int H, int C, int lowrank) { return check_shape(M, H, C, lowrank); }

ts_status check_ple_shape(int H, int C)
{
    if (H < 128 || H % 128 != 0 || H > kMaxH)
        return fail(TS_ERR_INVALID_ARG, "H = %d must be a multiple of 128 in [128, %d] (16 table segments of 8k)",
                    H, kMaxH);
    if (C < 1 || C > kMaxC)
        return fail(TS_ERR_INVALID_ARG, "C = %d must be in [1, %d]", C, kMaxC);
    return TS_OK;
}

ts_status check_ple_module(const ts_hc_ple_module *m)
{
    if (!m)
        return fail(TS_ERR_INVALID_ARG, "ple is NULL");
    if (m->n_rows < 1)
        return fail(TS_ERR_INVALID_ARG, "n_rows = %ld must be >= 1", m->n_rows);
    ts_status st;
    if ((st = check_ptr(m->table, "table", 16)) != TS_OK) return st;
    if ((st = check_ptr(m->key_proj, "key_proj", 16)) != TS_OK) return st;
    if ((st = check_ptr(m->value_proj, "value_proj", 16)) != TS_OK) return st;
    if ((st = check_ptr(m->norm_key_w, "norm_key_w", 16)) != TS_OK) return st;
    if ((st = check_ptr(m->norm_query_w, "norm_query_w", 16)) != TS_OK) return st;
    if ((st = check_ptr(m->norm_conv_w, "norm_conv_w", 16)) != TS_OK) return st;
    return check_ptr(m->conv_w, "conv_w", 16);
}

ts_status check_ptr_api(const void *p, const char *name, size_t align) { return check_ptr(p, name, align); }

ts_status check_module(const ts_hc_module *m, bool with_inject, int H, int C, int lowrank, const char *name)
{
    if (!m)
        return fail(TS_ERR_INVALID_ARG, "%s is NULL", name);
    const int W = C * H;
    char what[128];
    snprintf(what, sizeof what, "%s.hc_norm_w", name);
    ts_status st = check_ptr(m->hc_norm_w, what, 16);
    if (st != TS_OK)
        return st;
    snprintf(what, sizeof what, "%s.down", name);
    if ((st = check_weight(&m->down, what, lowrank, W)) != TS_OK)
        return st;
    snprintf(what, sizeof what, "%s.up", name);
    if ((st = check_weight(&m->up, what, W, lowrank)) != TS_OK)
        return st;
    if (with_inject) {
        snprintf(what, sizeof what, "%s.inject", name);
        if ((st = check_weight(&m->inject, what, C, W)) != TS_OK)
            return st;
        if (m->inject.type != m->down.type ||
            (m->down.type == TS_W_INT4_AFFINE && m->inject.group != m->down.group))
            return fail(TS_ERR_UNSUPPORTED, "%s: inject must have the same storage format and group as down",
                        name);
    }
    return TS_OK;
}

}  // namespace tshc

namespace {

// The batched tensor-core path: M >= kTcMinTokens, H and lowrank multiples of
// 64 (whole 64-wide K blocks), at most 8 streams.
bool tc_path_ok(int M, int H, int C, int L)
{
    return M >= tshc::kTcMinTokens && L % 64 == 0 && H % 64 == 0 && C <= 8;
}

struct WsLayout {
    size_t inv_rms, act, x_hi, x_lo, part, act_hi, act_lo, part1, ssq1, total;
};

// Per-chunk partial dots and sums of squares of the one-token path: at most
// 8 chunks (C * sps <= 8) of L + C rows.
constexpr int kPart1Chunks = 8;

WsLayout ws_layout(int M, int H, int C, int L)
{
    WsLayout w{};
    w.inv_rms = 0;
    w.act = align256(sizeof(float) * (size_t)M * C);
    w.total = w.act + align256(sizeof(float) * (size_t)M * L);
    if (M >= 1 && M <= tshc::kFewMaxTokens) {  // the down kernel leaves partials, the up kernel reduces them
        w.part1 = w.total;
        w.ssq1 = w.part1 + tshc::kPartCopies * align256(sizeof(float) * kPart1Chunks * (size_t)M * ((size_t)L + C));
        w.total = w.ssq1 + tshc::kPartCopies * sizeof(float) * tshc::kSsqStride;
    }
    if (tc_path_ok(M, H, C, L)) {  // normed hi/lo, per-chunk partials, act hi/lo
        const size_t R = (size_t)L + C, W = (size_t)C * H;
        const tshc::TcPlan pl = tshc::tc_plan(M, L, C, (int)W);
        w.x_hi = w.total;
        w.x_lo = w.x_hi + align256(2 * (size_t)M * W);
        w.part = w.x_lo + align256(2 * (size_t)M * W);
        w.act_hi = w.part + align256(sizeof(float) * (size_t)pl.nchunk * R * pl.Mp);
        w.act_lo = w.act_hi + align256(2 * (size_t)M * L);
        w.total = w.act_lo + align256(2 * (size_t)M * L);
    }
    return w;
}

// Chunks per stream for the split-K down kernel: the largest sps with
// C * sps <= 8 (one portable cluster) whose chunk H / sps is a multiple of
// `align` elements.
int choose_sps(int H, int C, int align)
{
    int best = 0;
    for (int sps = 1; C * sps <= 8; ++sps)
        if (H % sps == 0 && (H / sps) % align == 0)
            best = sps;
    return best;
}

// How a call reads and writes the residual, when not plainly ([M][C*H], read only).
//   ts_hc_inject_call: the previous sublayer's inject-add fused in (raw +
//     out * gate is what the call sees), written back in place by the up kernel;
//   ts_hc_entry_call: every stream reads one embedding row (stream stride 0),
//     and the replicated residual is written to raw_out.
struct ResidualIO {
    long mstride;             // elements between tokens of the residual the kernels read
    int cstride;              // elements between its streams (0: one row read by every stream)
    uint16_t *raw_out;        // [M][C*H] write-back of the residual the call sees
    const uint16_t *out;      // the previous sublayer's output, or nullptr
    const float *gate;        // and its gates
    long stride;
};

// The shared part of ts_hc_call, ts_hc_mixer and ts_hc_inject_call.
ts_status hc_call_impl(const void *raw, const void *hc_norm_w, const ts_weight *down,
                       const ts_weight *up, const ts_weight *inject, void *mixed, float *inject_w,
                       long inject_stride, int M, int H, int C, int L, float eps, void *workspace,
                       size_t workspace_bytes, cudaStream_t stream, const ResidualIO *fi = nullptr,
                       float *w_out = nullptr, const void *l2_pf = nullptr, size_t l2_pf_bytes = 0)
{
    ts_status st = check_shape(M, H, C, L);
    if (st != TS_OK)
        return st;
    if (M == 0)  // nothing is read or written: pointers are not examined
        return TS_OK;
    const int W = C * H;
    if ((st = check_ptr(raw, "raw", 16)) != TS_OK) return st;
    if ((st = check_ptr(hc_norm_w, "hc_norm_w", 16)) != TS_OK) return st;
    if ((st = check_ptr(mixed, "mixed", 16)) != TS_OK) return st;
    if ((st = check_weight(down, "down", L, W)) != TS_OK) return st;
    if ((st = check_weight(up, "up", W, L)) != TS_OK) return st;
    if (inject) {
        if ((st = check_weight(inject, "inject", C, W)) != TS_OK) return st;
        if (inject->type != down->type || (down->type == TS_W_INT4_AFFINE && inject->group != down->group))
            return fail(TS_ERR_UNSUPPORTED, "inject must have the same storage format and group as down");
        if ((st = check_ptr(inject_w, "inject_w", 4)) != TS_OK) return st;
        if (inject_stride < C)
            return fail(TS_ERR_INVALID_ARG, "inject_stride = %ld must be >= C = %d", inject_stride, C);
    }
    if (!(eps >= 0.0f) || eps > 1.0f)
        return fail(TS_ERR_INVALID_ARG, "eps = %g must be in [0, 1]", (double)eps);
    if (M == 0)
        return TS_OK;
    const size_t need = ts_hc_workspace_bytes(M, H, C, L);
    if (!workspace || workspace_bytes < need)
        return fail(TS_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed", workspace_bytes, need);
    if (!aligned(workspace, 256))
        return fail(TS_ERR_INVALID_ARG, "workspace is not 256-byte aligned");

    const int down_align = down->type == TS_W_BF16 ? 8 : std::max(32, down->group);
    const int sps = choose_sps(H, C, down_align);
    if (sps == 0)
        return fail(TS_ERR_UNSUPPORTED, "H = %d is not a multiple of %d (INT4 down weights)", H, down_align);

    DeviceInfo dev;
    if ((st = device_info(&dev)) != TS_OK)
        return st;

    const WsLayout wl = ws_layout(M, H, C, L);
    char *wsb = static_cast<char *>(workspace);
    float *inv_rms = reinterpret_cast<float *>(wsb + wl.inv_rms);
    float *act = reinterpret_cast<float *>(wsb + wl.act);

    const bool all_bf16 = down->type == TS_W_BF16 && up->type == TS_W_BF16 && (!inject || inject->type == TS_W_BF16);
    // INT4-affine weights on the tensor cores: dequantised per tile to bf16 hi + lo.
    const bool all_int4 = down->type == TS_W_INT4_AFFINE && up->type == TS_W_INT4_AFFINE &&
                          (!inject || inject->type == TS_W_INT4_AFFINE) && down->group % 8 == 0 &&
                          up->group % 8 == 0;
    // From 2 to kFewMaxTokens tokens bf16 calls try the few-token kernels first
    // (two kernels, no tensor cores), and take the tensor-core path when the
    // shape does not fit them.
    const bool few_first = all_bf16 && M >= 2 && M <= tshc::kFewMaxTokens;
    auto run_tc = [&]() -> ts_status {
        const tshc::TcPlan pl = tshc::tc_plan(M, L, C, W);
        tshc::TcCall t{};
        const int R = L + (inject ? C : 0);
        tshc::TcPrepParams &tp = t.prep;
        tp.raw = static_cast<const uint16_t *>(raw);
        tp.raw_mstride = fi ? fi->mstride : W;
        tp.raw_cstride = fi ? fi->cstride : H;
        tp.g = static_cast<const uint16_t *>(hc_norm_w);
        if (fi) {
            tp.raw_out = fi->raw_out;
            tp.inj_out = fi->out;
            tp.inj_gate = fi->gate;
            tp.inj_stride = fi->stride;
        }
        tp.x_hi = reinterpret_cast<uint16_t *>(wsb + wl.x_hi);
        tp.x_lo = reinterpret_cast<uint16_t *>(wsb + wl.x_lo);
        tp.inv_rms = inv_rms;
        tp.M = M; tp.H = H; tp.C = C; tp.W = W;
        tp.eps = eps; tp.inv_H = 1.0f / (float)H;
        tshc::TcDownParams &td = t.down;
        td.part = reinterpret_cast<float *>(wsb + wl.part);
        td.M = M; td.L = L; td.C = C; td.R = R; td.W = W; td.Mp = pl.Mp;
        td.has_inject = inject ? 1 : 0;
        td.KBc = pl.KBc; td.nchunk = pl.nchunk;
        td.NT = pl.NT;
        td.wt = all_int4 ? 1 : 0;
        td.dw = view(down);
        td.iw = view(inject);
        td.n_stages = 4;
        while (td.n_stages > 2 && tshc::tc_down_smem(pl.NT, td.n_stages, td.wt) > tshc::kTcSmemLimit)
            --td.n_stages;
        td.status = dev.status;
        tshc::TcReduceParams &tr = t.red;
        tr.part = td.part; tr.act = act;
        tr.act_hi = reinterpret_cast<uint16_t *>(wsb + wl.act_hi);
        tr.act_lo = reinterpret_cast<uint16_t *>(wsb + wl.act_lo);
        tr.gate = inject ? inject_w : nullptr;
        tr.gate_stride = inject ? inject_stride : 0;
        tr.M = M; tr.L = L; tr.R = R; tr.Mp = pl.Mp; tr.nchunk = pl.nchunk;
        tr.inv_C = 1.0f / (float)C;
        // L2 prefetch hint: the up weights (by the reduce kernel), rounded
        // inwards to 16-byte boundaries.
        auto hint = [](const ts_weight *w, size_t rows, size_t cols, const void **ptr, size_t *bytes) {
            const size_t wbytes = w->type == TS_W_BF16 ? rows * cols * 2 : rows * cols / 2;
            const size_t sbytes = w->type == TS_W_BF16 ? 0 : rows * (cols / w->group) * 2;
            const void *ranges[3] = {w->data, w->scales, w->biases};
            const size_t sizes[3] = {wbytes, sbytes, sbytes};
            for (int i = 0; i < 3; ++i) {
                const uintptr_t a = reinterpret_cast<uintptr_t>(ranges[i]);
                const uintptr_t lo = (a + 15) & ~uintptr_t(15), hi = (a + sizes[i]) & ~uintptr_t(15);
                ptr[i] = reinterpret_cast<const void *>(lo);
                bytes[i] = sizes[i] && hi > lo ? (size_t)(hi - lo) : 0;
            }
        };
        hint(up, (size_t)W, (size_t)L, tr.l2_next, tr.l2_next_bytes);
        tshc::TcUpParams &tu = t.up;
        tu.mixed = static_cast<uint16_t *>(mixed);
        tu.M = M; tu.H = H; tu.C = C; tu.L = L; tu.W = W;
        tu.HBt = (128 / C) / 8 * 8;
        tu.NT = pl.NT;
        tu.wt = td.wt;
        tu.uw = view(up);
        tu.n_stages = 4;
        while (tu.n_stages > 2 && tshc::tc_up_smem(pl.NT, tu.n_stages, C, tu.HBt, tu.wt) > tshc::kTcSmemLimit)
            --tu.n_stages;
        tu.inv_C = tr.inv_C;
        tu.status = dev.status;
        tu.w_out = w_out;
        t.wd = down->data;
        t.wi = inject ? inject->data : nullptr;
        t.wu = up->data;
        const cudaError_t e = tshc::launch_tc_call(t, stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "launching the tensor-core path");
        return TS_OK;
    };
    const bool tc_ok = tc_path_ok(M, H, C, L) && (all_bf16 || all_int4);
    if (tc_ok && !few_first)
        return run_tc();

    tshc::DownParams d{};
    d.raw = static_cast<const uint16_t *>(raw);
    d.raw_mstride = fi ? fi->mstride : W;
    d.raw_cstride = fi ? fi->cstride : H;
    d.g = static_cast<const uint16_t *>(hc_norm_w);
    d.down = view(down);
    d.inject = view(inject);
    d.act = act;
    d.inv_rms = inv_rms;
    d.gate = inject ? inject_w : nullptr;
    d.gate_stride = inject ? inject_stride : 0;
    d.M = M; d.H = H; d.C = C; d.L = L; d.W = W;
    d.R = L + (inject ? C : 0);
    d.sps = sps; d.S = C * sps; d.KC = H / sps;
    d.eps = eps;
    d.inv_C = 1.0f / (float)C;
    d.status = dev.status;
    if (fi) {
        d.inj_out = fi->out;
        d.inj_gate = fi->gate;
        d.inj_stride = fi->stride;
    }
    const int target_blocks = std::max(1, dev.sm_count / d.S);
    d.rows_per_block = (d.R + target_blocks - 1) / target_blocks;
    d.mt = tshc::gemv_token_tile(M);
    while (tshc::down_smem_bytes(d, d.mt) > tshc::kSmemBudget && d.mt > 1)
        d.mt /= 2;
    while (tshc::down_smem_bytes(d, d.mt) > tshc::kSmemBudget && d.rows_per_block > 1)
        d.rows_per_block = (d.rows_per_block + 1) / 2;
    if (tshc::down_smem_bytes(d, d.mt) > tshc::kSmemBudget)
        return fail(TS_ERR_UNSUPPORTED, "shape H = %d, C = %d exceeds the shared-memory budget", H, C);

    tshc::UpParams u{};
    u.raw = d.raw;
    u.raw_mstride = d.raw_mstride;
    u.raw_cstride = d.raw_cstride;
    u.g = d.g;
    u.up = view(up);
    u.act = act;
    u.inv_rms = inv_rms;
    u.mixed = static_cast<uint16_t *>(mixed);
    u.M = M; u.H = H; u.C = C; u.L = L; u.W = W;
    u.HB = (H + dev.sm_count - 1) / dev.sm_count;
    u.inv_C = d.inv_C;
    u.status = dev.status;
    u.w_out = w_out;
    u.l2_pf = l2_pf;
    u.l2_pf_bytes = l2_pf_bytes;
    if (fi) {
        u.raw_out = fi->raw_out;
        u.inj_out = fi->out;
        u.inj_gate = fi->gate;
        u.inj_stride = fi->stride;
    }
    u.mt = tshc::gemv_token_tile(M);
    while (tshc::up_smem_bytes(u, u.mt) > tshc::kSmemBudget && u.mt > 1)
        u.mt /= 2;
    while (tshc::up_smem_bytes(u, u.mt) > tshc::kSmemBudget && u.HB > 1)
        u.HB = (u.HB + 1) / 2;
    if (tshc::up_smem_bytes(u, u.mt) > tshc::kSmemBudget)
        return fail(TS_ERR_UNSUPPORTED, "shape C = %d, lowrank = %d exceeds the shared-memory budget", C, L);

    const tshc::LaunchCfg cfg{dev.sm_count, true};
    cudaError_t e;
    if (M <= tshc::kFewMaxTokens) {
        // One token (and, with bf16 weights, up to kFewMaxTokens): the down kernel
        // leaves per-chunk partials and the up kernel reduces them, so neither
        // kernel waits on another CTA.
        d.part1 = reinterpret_cast<float *>(wsb + wl.part1);
        d.ssq1 = reinterpret_cast<float *>(wsb + wl.ssq1);
        d.part1_stride = (long)(align256(sizeof(float) * kPart1Chunks * (size_t)M * ((size_t)L + C)) / sizeof(float));
        u.part1 = d.part1;
        u.ssq1 = d.ssq1;
        u.part1_stride = d.part1_stride;
        u.S = d.S;
        u.sps = d.sps;
        u.R = d.R;
        u.eps = eps;
        u.inv_H = 1.0f / (float)H;
        u.act_out = act;
        u.inv_out = inv_rms;
        u.gate = inject ? inject_w : nullptr;
        u.gate_stride = inject_stride;
        if (M == 1 && d.S <= kPart1Chunks && tshc::one_token_ok(d, u)) {
            e = tshc::launch_one_token(d, u, cfg, stream);
            if (e != cudaSuccess)
                return cuda_fail(e, "launching the one-token kernels");
            return TS_OK;
        }
        if (few_first && d.S <= kPart1Chunks && tshc::few_tokens_ok(d, u)) {
            e = tshc::launch_few_tokens(d, u, cfg, stream);
            if (e != cudaSuccess)
                return cuda_fail(e, "launching the few-token kernels");
            return TS_OK;
        }
    }
    if (tc_ok)  // the few-token kernels do not take this shape
        return run_tc();
    e = tshc::launch_down(d, cfg, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "launching the down kernel");
    e = tshc::launch_up(u, cfg, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "launching the up kernel");
    return TS_OK;
}

}  // namespace

extern "C" {

size_t ts_hc_workspace_bytes(int M, int H, int C, int lowrank)
{
    if (M < 0 || H < 1 || C < 1 || lowrank < 1)
        return 0;
    return ws_layout(M, H, C, lowrank).total;
}

ts_status ts_hc_workspace_layout(int M, int H, int C, int lowrank, size_t *inv_rms_offset,
                                 size_t *act_offset)
{
    if (M < 0 || H < 1 || C < 1 || lowrank < 1)
        return fail(TS_ERR_INVALID_ARG, "invalid shape");
    const WsLayout w = ws_layout(M, H, C, lowrank);
    if (inv_rms_offset)
        *inv_rms_offset = w.inv_rms;
    if (act_offset)
        *act_offset = w.act;
    return TS_OK;
}

ts_status ts_hc_call(const void *raw, const void *hc_norm_w, const ts_weight *down,
                     const ts_weight *up, const ts_weight *inject, void *mixed, float *inject_w,
                     long inject_stride, int M, int H, int C, int lowrank, float eps,
                     void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    g_last_error.clear();
    if (!inject)
        return fail(TS_ERR_INVALID_ARG, "inject is NULL (use ts_hc_mixer for the final mixer)");
    return hc_call_impl(raw, hc_norm_w, down, up, inject, mixed, inject_w, inject_stride, M, H, C,
                        lowrank, eps, workspace, workspace_bytes, stream);
}

ts_status ts_hc_mixer(const void *raw, const void *hc_norm_w, const ts_weight *down,
                      const ts_weight *up, void *mixed, int M, int H, int C, int lowrank, float eps,
                      void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    g_last_error.clear();
    return hc_call_impl(raw, hc_norm_w, down, up, nullptr, mixed, nullptr, 0, M, H, C, lowrank, eps,
                        workspace, workspace_bytes, stream);
}

ts_status ts_hc_call_debug(const void *raw, const void *hc_norm_w, const ts_weight *down,
                           const ts_weight *up, const ts_weight *inject, void *mixed, float *inject_w,
                           long inject_stride, int M, int H, int C, int lowrank, float eps, void *workspace,
                           size_t workspace_bytes, float *w_out, cudaStream_t stream)
{
    g_last_error.clear();
    if (M > 0) {
        const ts_status st = check_ptr(w_out, "w_out", 4);
        if (st != TS_OK)
            return st;
    }
    return hc_call_impl(raw, hc_norm_w, down, up, inject, mixed, inject ? inject_w : nullptr,
                        inject ? inject_stride : 0, M, H, C, lowrank, eps, workspace, workspace_bytes, stream,
                        nullptr, w_out);
}

}  // extern "C"

namespace {

// Whether the strided gate sets {a + m*sa + c} and {b + m*sb + c} (m < M,
// c < C, in floats) can share an element. Exact for equal strides (two slots
// of one [M][2][C] buffer are disjoint), conservative otherwise.
bool gates_overlap(const float *a, long sa, const float *b, long sb, int M, int C)
{
    const intptr_t diff = reinterpret_cast<intptr_t>(b) - reinterpret_cast<intptr_t>(a);
    const long ea = (long)(M - 1) * sa + C, eb = (long)(M - 1) * sb + C;
    if (diff >= (intptr_t)(4 * ea) || -diff >= (intptr_t)(4 * eb))
        return false;  // disjoint address ranges
    if (diff % 4 != 0 || sa != sb)
        return true;
    const long r = ((long)(diff / 4) % sa + sa) % sa;
    return !(r >= C && r <= sa - C);
}

}  // namespace

namespace {

// Bytes of lm_head that the exit's one-token mixer asks L2 to prefetch: about what
// HBM delivers beside the mixer's own weights in its ~5.5 us (12, 24 and 40 MB
// measured: 32.1, 31.95, 32.2 us per exit against 33.3). The batched mixers take
// none: 32, 48 and 80 MB from the tensor-core up kernel did not shorten an exit at
// 16 tokens (41.1 us against 41.4, 41.3, 43.3).
size_t exit_prefetch_bytes(int M) { return M == 1 ? (size_t)24 << 20 : 0; }

}  // namespace

extern "C" {

ts_status ts_hc_inject_call(void *raw, const void *out, const float *prev_inject_w, long prev_inject_stride,
                            const void *hc_norm_w, const ts_weight *down, const ts_weight *up,
                            const ts_weight *inject, void *mixed, float *inject_w, long inject_stride,
                            int M, int H, int C, int lowrank, float eps,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    g_last_error.clear();
    ts_status st = check_shape(M, H, C, lowrank);
    if (st != TS_OK)
        return st;
    if (M == 0)  // nothing is read or written: pointers are not examined
        return TS_OK;
    if ((st = check_ptr(out, "out", 16)) != TS_OK) return st;
    if ((st = check_ptr(prev_inject_w, "prev_inject_w", 4)) != TS_OK) return st;
    if (prev_inject_stride < C)
        return fail(TS_ERR_INVALID_ARG, "prev_inject_stride = %ld must be >= C = %d", prev_inject_stride, C);
    if (inject && inject_w && M > 0 && inject_stride >= C &&
        gates_overlap(prev_inject_w, prev_inject_stride, inject_w, inject_stride, M, C))
        return fail(TS_ERR_INVALID_ARG, "inject_w shares elements with prev_inject_w");
    const ResidualIO fi{(long)C * H, H, static_cast<uint16_t *>(raw), static_cast<const uint16_t *>(out),
                        prev_inject_w, prev_inject_stride};
    return hc_call_impl(raw, hc_norm_w, down, up, inject, mixed, inject_w, inject_stride, M, H, C, lowrank,
                        eps, workspace, workspace_bytes, stream, &fi);
}

ts_status ts_hc_exit_logits(void *raw, const void *out, const float *prev_inject_w, long prev_inject_stride,
                            const void *hc_norm_w, const ts_weight *down, const ts_weight *up, const void *lm_head,
                            int V, void *mixed, float *logits, int M, int H, int C, int lowrank, float eps,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    g_last_error.clear();
    ts_status st = check_shape(M, H, C, lowrank);
    if (st != TS_OK)
        return st;
    if (V < 1)
        return fail(TS_ERR_INVALID_ARG, "V = %d must be >= 1", V);
    if (M == 0)  // nothing is read or written: pointers are not examined
        return TS_OK;
    if ((st = check_ptr(lm_head, "lm_head", 16)) != TS_OK) return st;
    if ((st = check_ptr(logits, "logits", 4)) != TS_OK) return st;
    if (out) {
        if ((st = check_ptr(out, "out", 16)) != TS_OK) return st;
        if ((st = check_ptr(prev_inject_w, "prev_inject_w", 4)) != TS_OK) return st;
        if (prev_inject_stride < C)
            return fail(TS_ERR_INVALID_ARG, "prev_inject_stride = %ld must be >= C = %d", prev_inject_stride, C);
    }
    if (!tshc::lm_head_shape_ok(std::min(M, tshc::kLmHeadMaxTokens), H, V))
        return fail(TS_ERR_UNSUPPORTED, "the lm_head kernel does not take H = %d (a multiple of 64)", H);
    DeviceInfo dev;
    if ((st = device_info(&dev)) != TS_OK)
        return st;
    const ResidualIO io{(long)C * H, H, static_cast<uint16_t *>(raw), static_cast<const uint16_t *>(out),
                        prev_inject_w, prev_inject_stride};
    // While a one-token mixer runs, its up kernel asks L2 for the first part of
    // lm_head (the lm_head kernel then streams that part from L2, not HBM).
    const size_t pf = std::min(exit_prefetch_bytes(M), (size_t)V * H * 2) & ~size_t(15);
    st = hc_call_impl(raw, hc_norm_w, down, up, nullptr, mixed, nullptr, 0, M, H, C, lowrank, eps, workspace,
                      workspace_bytes, stream, out ? &io : nullptr, nullptr, lm_head, pf);
    if (st != TS_OK)
        return st;
    // lm_head over tiles of at most kLmHeadMaxTokens tokens, each a dependent of the launch before it.
    tshc::LmHeadParams lp{};
    lp.H = H;
    lp.V = V;
    for (int t0 = 0; t0 < M; t0 += tshc::kLmHeadMaxTokens) {
        lp.M = std::min(tshc::kLmHeadMaxTokens, M - t0);
        lp.mixed = static_cast<const uint16_t *>(mixed) + (size_t)t0 * H;
        lp.w = static_cast<const uint16_t *>(lm_head);
        lp.logits = logits + (size_t)t0 * V;
        lp.logits_stride = V;
        lp.status = dev.status;
        const cudaError_t e = tshc::launch_lm_head(lp, tshc::LaunchCfg{dev.sm_count, true}, stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "launching the lm_head kernel");
    }
    return TS_OK;
}

}  // extern "C"

namespace {

struct PleWs {
    size_t emb, key, value, gate, x, total;
};

PleWs ple_ws(int M, int H, int C)
{
    PleWs w{};
    const size_t m = (size_t)M, W = (size_t)C * H;
    w.emb = 0;
    w.key = align256(2 * m * H);
    w.value = w.key + align256(4 * m * W);
    w.gate = w.value + align256(4 * m * H);
    w.x = w.gate + align256(4 * m * C);
    w.total = w.x + align256(4 * m * W);
    return w;
}

}  // namespace

extern "C" {

size_t ts_hc_ple_workspace_bytes(int M, int H, int C)
{
    if (M < 0 || H < 128 || H % 128 != 0 || H > kMaxH || C < 1 || C > kMaxC)
        return 0;
    return ple_ws(M, H, C).total;
}

ts_status ts_hc_ple_workspace_layout(int M, int H, int C, size_t *value_offset, size_t *gate_offset,
                                     size_t *x_offset)
{
    if (ts_hc_ple_workspace_bytes(M, H, C) == 0 && M != 0)
        return fail(TS_ERR_INVALID_ARG, "invalid PLE shape");
    const PleWs w = ple_ws(M, H, C);
    if (value_offset) *value_offset = w.value;
    if (gate_offset) *gate_offset = w.gate;
    if (x_offset) *x_offset = w.x;
    return TS_OK;
}

ts_status ts_hc_ple(void *hidden, const int32_t *rows, const void *table, long n_rows, const void *key_proj,
                    const void *value_proj, const void *norm_key_w, const void *norm_query_w,
                    const void *norm_conv_w, const void *conv_w, float *conv_state, int M, int H, int C,
                    float eps, void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    g_last_error.clear();
    if (M < 0)
        return fail(TS_ERR_INVALID_ARG, "M = %d must be >= 0", M);
    ts_status st = tshc::check_ple_shape(H, C);
    if (st != TS_OK)
        return st;
    if (M == 0)  // nothing is read or written: pointers are not examined
        return TS_OK;
    const ts_hc_ple_module mod{table, n_rows, key_proj, value_proj, norm_key_w, norm_query_w, norm_conv_w, conv_w};
    if ((st = check_ptr(hidden, "hidden", 16)) != TS_OK) return st;
    if ((st = check_ptr(rows, "rows", 4)) != TS_OK) return st;
    if ((st = tshc::check_ple_module(&mod)) != TS_OK) return st;
    if ((st = check_ptr(conv_state, "conv_state", 16)) != TS_OK) return st;
    if (!(eps >= 0.0f) || eps > 1.0f)
        return fail(TS_ERR_INVALID_ARG, "eps = %g must be in [0, 1]", (double)eps);
    const PleWs lay = ple_ws(M, H, C);
    if (!workspace || workspace_bytes < lay.total)
        return fail(TS_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed", workspace_bytes, lay.total);
    if (!aligned(workspace, 256))
        return fail(TS_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
    DeviceInfo dev;
    if ((st = device_info(&dev)) != TS_OK)
        return st;
    if (!tshc::lm_head_shape_ok(std::min(M, tshc::kLmHeadMaxTokens), H, C * H))
        return fail(TS_ERR_UNSUPPORTED, "the projection kernel does not take H = %d", H);
    char *ws = static_cast<char *>(workspace);
    tshc::PleParams p{};
    p.hidden = static_cast<uint16_t *>(hidden);
    p.rows = rows;
    p.table = static_cast<const uint16_t *>(table);
    p.n_rows = n_rows;
    p.key_proj = static_cast<const uint16_t *>(key_proj);
    p.value_proj = static_cast<const uint16_t *>(value_proj);
    p.norm_key = static_cast<const uint16_t *>(norm_key_w);
    p.norm_query = static_cast<const uint16_t *>(norm_query_w);
    p.norm_conv = static_cast<const uint16_t *>(norm_conv_w);
    p.conv_w = static_cast<const uint16_t *>(conv_w);
    p.state = conv_state;
    p.emb = reinterpret_cast<uint16_t *>(ws + lay.emb);
    p.key = reinterpret_cast<float *>(ws + lay.key);
    p.value = reinterpret_cast<float *>(ws + lay.value);
    p.gate = reinterpret_cast<float *>(ws + lay.gate);
    p.x = reinterpret_cast<float *>(ws + lay.x);
    p.M = M; p.H = H; p.C = C;
    p.eps = eps;
    p.inv_H = 1.0f / (float)H;
    p.inv_sqrt_H = 1.0f / sqrtf((float)H);
    p.status = dev.status;
    const cudaError_t e = tshc::launch_ple(p, tshc::LaunchCfg{dev.sm_count, true}, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "launching the PLE kernels");
    return TS_OK;
}

ts_status ts_hc_entry_call(const void *emb, void *raw, const void *hc_norm_w, const ts_weight *down,
                           const ts_weight *up, const ts_weight *inject, void *mixed, float *inject_w,
                           long inject_stride, int M, int H, int C, int lowrank, float eps, void *workspace,
                           size_t workspace_bytes, cudaStream_t stream)
{
    g_last_error.clear();
    ts_status st = check_shape(M, H, C, lowrank);
    if (st != TS_OK)
        return st;
    if (M == 0)  // nothing is read or written: pointers are not examined
        return TS_OK;
    if ((st = check_ptr(emb, "emb", 16)) != TS_OK) return st;
    if ((st = check_ptr(raw, "raw", 16)) != TS_OK) return st;
    const char *e = static_cast<const char *>(emb), *r = static_cast<const char *>(raw);
    if (e < r + 2 * (size_t)M * C * H && r < e + 2 * (size_t)M * H)
        return fail(TS_ERR_INVALID_ARG, "raw overlaps emb");
    const ResidualIO io{H, 0, static_cast<uint16_t *>(raw), nullptr, nullptr, 0};
    return hc_call_impl(emb, hc_norm_w, down, up, inject, mixed, inject_w, inject_stride, M, H, C, lowrank, eps,
                        workspace, workspace_bytes, stream, &io);
}

ts_status ts_hc_inject_add(void *raw, const void *out, const float *inject_w, long inject_stride,
                           int M, int H, int C, cudaStream_t stream)
{
    g_last_error.clear();
    if (M < 0)
        return fail(TS_ERR_INVALID_ARG, "M = %d must be >= 0", M);
    if (H < 8 || H % 8 != 0 || H > kMaxH)
        return fail(TS_ERR_INVALID_ARG, "H = %d must be a multiple of 8 in [8, %d]", H, kMaxH);
    if (C < 1 || C > kMaxC)
        return fail(TS_ERR_INVALID_ARG, "C = %d must be in [1, %d]", C, kMaxC);
    if (M == 0)  // nothing is read or written: pointers are not examined
        return TS_OK;
    ts_status st;
    if ((st = check_ptr(raw, "raw", 16)) != TS_OK) return st;
    if ((st = check_ptr(out, "out", 16)) != TS_OK) return st;
    if ((st = check_ptr(inject_w, "inject_w", 4)) != TS_OK) return st;
    if (inject_stride < C)
        return fail(TS_ERR_INVALID_ARG, "inject_stride = %ld must be >= C = %d", inject_stride, C);
    if (M == 0)
        return TS_OK;
    DeviceInfo dev;
    if ((st = device_info(&dev)) != TS_OK)
        return st;
    tshc::InjectParams p{};
    p.raw = static_cast<uint16_t *>(raw);
    p.out = static_cast<const uint16_t *>(out);
    p.gate = inject_w;
    p.gate_stride = inject_stride;
    p.M = M; p.H = H; p.C = C; p.W = C * H;
    const cudaError_t e = tshc::launch_inject(p, tshc::LaunchCfg{dev.sm_count, true}, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "launching the inject-add kernel");
    return TS_OK;
}

ts_status ts_hc_replicate_entry(const void *emb, void *raw, int M, int H, int C, cudaStream_t stream)
{
    g_last_error.clear();
    if (M < 0)
        return fail(TS_ERR_INVALID_ARG, "M = %d must be >= 0", M);
    if (H < 8 || H % 8 != 0 || H > kMaxH)
        return fail(TS_ERR_INVALID_ARG, "H = %d must be a multiple of 8 in [8, %d]", H, kMaxH);
    if (C < 1 || C > kMaxC)
        return fail(TS_ERR_INVALID_ARG, "C = %d must be in [1, %d]", C, kMaxC);
    if (M == 0)  // nothing is read or written: pointers are not examined
        return TS_OK;
    ts_status st;
    if ((st = check_ptr(emb, "emb", 16)) != TS_OK) return st;
    if ((st = check_ptr(raw, "raw", 16)) != TS_OK) return st;
    if (M == 0)
        return TS_OK;
    DeviceInfo dev;
    if ((st = device_info(&dev)) != TS_OK)
        return st;
    tshc::ReplicateParams p{static_cast<const uint16_t *>(emb), static_cast<uint16_t *>(raw), M, H, C};
    const cudaError_t e = tshc::launch_replicate(p, tshc::LaunchCfg{dev.sm_count, true}, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "launching the entry-replication kernel");
    return TS_OK;
}

const char *ts_hc_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"

namespace {

// One thread waits, with the kernels' own bounded wait, on a barrier that
// nothing arrives at, and records the timeout as the kernels do.
__global__ void hc_timeout_selftest_kernel(unsigned *status)
{
    __shared__ uint64_t bar;
    tshc::mbar_init(&bar, 1);
    tshc::mbar_fence_init();
    if (!tshc::mbar_wait_bounded(&bar, 0))
        atomicExch(status, tshc::kStatusTimeout);
}

}  // namespace

extern "C" {

ts_status ts_hc_selftest_timeout(cudaStream_t stream)
{
    g_last_error.clear();
    DeviceInfo dev;
    ts_status st = device_info(&dev);
    if (st != TS_OK)
        return st;
    hc_timeout_selftest_kernel<<<1, 1, 0, stream>>>(dev.status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "launching the timeout self-test kernel");
    return TS_OK;
}

ts_status ts_hc_device_status(cudaStream_t stream, int *status)
{
    g_last_error.clear();
    if (!status)
        return fail(TS_ERR_INVALID_ARG, "status is NULL");
    unsigned v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_device_status, sizeof v, 0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "reading the device status word");
    *status = v == 0 ? TS_OK : (int)v;
    return TS_OK;
}

}  // extern "C"

// ---- ts_hc_call_noalloc: the workspace in a file-scope device array ---------

// Scratch for callers that cannot allocate. Host code only ever sees a
// host-side stand-in for this name; the device address is looked up per
// device with cudaGetSymbolAddress and passed to the kernels.
static __device__ __align__(256) unsigned char g_hc_static_scratch[TS_HC_STATIC_SCRATCH_BYTES];

namespace {

std::mutex g_static_mutex;
void *g_static_scratch[kMaxDevices];

// Device address of the array on the current device, looked up on the first
// call there (with that device current).
ts_status static_scratch(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(TS_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (!g_static_scratch[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_hc_static_scratch);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        g_static_scratch[dev] = p;
    }
    *out = g_static_scratch[dev];
    return TS_OK;
}

}  // namespace

extern "C" ts_status ts_hc_call_noalloc(const void *raw, const void *hc_norm_w, const ts_weight *down,
                                        const ts_weight *up, const ts_weight *inject, void *mixed,
                                        float *inject_w, long inject_stride, int M, int H, int C,
                                        int lowrank, float eps, cudaStream_t stream)
{
    g_last_error.clear();
    if (!inject)
        return fail(TS_ERR_INVALID_ARG, "inject is NULL (the no-allocation variant covers ts_hc_call)");
    ts_status st = check_shape(M, H, C, lowrank);
    if (st != TS_OK)
        return st;
    if (M == 0)
        return TS_OK;
    const size_t need = ts_hc_workspace_bytes(M, H, C, lowrank);
    if (need > TS_HC_STATIC_SCRATCH_BYTES)
        return fail(TS_ERR_WORKSPACE,
                    "M = %d tokens need %zu bytes of scratch; the static scratch holds %u bytes "
                    "(call ts_hc_call with a workspace, or split the tokens)",
                    M, need, (unsigned)TS_HC_STATIC_SCRATCH_BYTES);
    void *ws = nullptr;
    if ((st = static_scratch(&ws)) != TS_OK)
        return st;
    return hc_call_impl(raw, hc_norm_w, down, up, inject, mixed, inject_w, inject_stride, M, H, C, lowrank,
                        eps, ws, TS_HC_STATIC_SCRATCH_BYTES, stream);
}
