"""GPU parity: the CUDA library (called through the C ABI) against the fp64 oracle.

Covers the five workloads (tiny call, full-shape decode call, the M=128
chunked-prefill micro-batch with per-token gate rows, the 40-layer stack at
M=1 and M=16, INT4-affine weights at M=1 and M=64), plus ragged token counts
and shapes that exercise other cluster sizes, chunk widths and tile tails,
the M=0 no-op, guard regions after every output, the read-only residual,
run-to-run bit identity and the device status word.
"""
import numpy as np
import pytest
import torch

import oracle
from hyper_connection_residual_call_gb300 import binding as B
from hyper_connection_residual_call_gb300 import inputs
from gpu_common import (CHAINED_RMS_FLOOR, check_bf16, check_bf16_carried, check_fp32, guard_intact, guarded,
                        require_gpu, to_np, workspace_intermediates)

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def gpu_call(raw_d, w_d, H, C, gates=None, stride=None):
    """One ts_hc_call with sentinel guards after mixed (and after gates when owned)."""
    M = raw_d.shape[0]
    L = w_d.down.rows
    mixed, mwhole = guarded((M, H), torch.bfloat16, -77.0)
    own = gates is None
    if own:
        gates, gwhole = guarded((M, C), torch.float32, float("nan"))
        stride = C
    ws = B.workspace(M, H, C, L)
    B.hc_call(raw_d, w_d, H=H, C=C, mixed=mixed, inject_w=gates, inject_stride=stride, eps=EPS, ws=ws)
    torch.cuda.synchronize()
    assert guard_intact(mwhole, M * H, -77.0), "write past the end of mixed"
    if own:
        assert guard_intact(gwhole, M * C, float("nan")), "write past the end of inject_w"
    inv, act = workspace_intermediates(ws, M, H, C, L)
    return mixed, gates, inv, act


def check_call(res, ref, tag):
    mixed, gates, inv, act = res
    check_bf16(mixed, ref["mixed"], f"{tag} mixed")
    check_fp32(inv, ref["inv_rms"], f"{tag} inv_rms")
    check_fp32(act, ref["a"], f"{tag} act")
    if "gate" in ref and gates is not None:
        check_fp32(gates, ref["gate"], f"{tag} gate")


def call_and_inject(orc, shape, seed, kind="bf16", group=64, up_group=None):
    H, C, L, M = shape.H, shape.C, shape.L, shape.M
    w = inputs.make_hc_weights(H, C, L, seed, kind=kind, group=group, up_group=up_group)
    raw = inputs.make_residual(M, H, C, seed)
    out = inputs.make_sublayer_out(M, H, seed)
    ref = orc.hc_call(raw, w.g, w.down, w.up, w.inject, H=H, C=C, L=L, eps=EPS)
    ref_raw = orc.inject_add(raw, out, ref["gate"], H=H, C=C)
    w_d, raw_d, out_d = w.to("cuda"), raw.cuda(), out.cuda()
    raw_before = raw_d.clone()
    res = gpu_call(raw_d, w_d, H, C)
    assert torch.equal(raw_d, raw_before), "ts_hc_call wrote the residual"
    check_call(res, ref, f"{kind} M={M} H={H} C={C} L={L}")
    raw2, rwhole = guarded((M, C * H), torch.bfloat16, -5.0)
    raw2.copy_(raw_d)
    B.hc_inject_add(raw2, out_d, res[1], H=H, C=C)
    torch.cuda.synchronize()
    assert guard_intact(rwhole, M * C * H, -5.0)
    check_bf16(raw2, ref_raw, "injected residual")
    return res


def test_tiny_call(orc):
    call_and_inject(orc, inputs.TINY, inputs.SEEDS["tiny"])


def test_full_decode_call(orc):
    call_and_inject(orc, inputs.FULL_DECODE, inputs.SEEDS["full_decode"])


def test_bit_identical_runs(orc):
    s = inputs.FULL_DECODE
    w = inputs.make_hc_weights(s.H, s.C, s.L, 1).to("cuda")
    raw = inputs.make_residual(3, s.H, s.C, 1).cuda()
    a = gpu_call(raw, w, s.H, s.C)
    b = gpu_call(raw, w, s.H, s.C)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("M,H,C,L", [(3, 40, 3, 24), (5, 64, 1, 8), (9, 128, 8, 16), (17, 256, 4, 32),
                                     (2, 2560, 4, 320), (1, 8, 2, 8), (11, 96, 5, 40), (33, 512, 2, 64)])
def test_shapes_and_ragged_tokens(orc, M, H, C, L):
    call_and_inject(orc, inputs.Shape(M=M, H=H, C=C, L=L), seed=100 + M)


# The API's maxima (H = 16384, C = 8, lowrank = 1024; a wide residual of 131072): one
# token, the tensor-core path, the largest lowrank at the full shape's H.
@pytest.mark.parametrize("M,H,C,L", [(1, 16384, 8, 1024), (3, 16384, 8, 1024), (1, 2560, 8, 1024),
                                     (20, 2560, 4, 1024),
                                     # H and lowrank not multiples of 64: the cluster split-K kernels
                                     (3, 16376, 8, 1000), (1, 16376, 8, 1000)])
def test_maximum_shapes(orc, M, H, C, L):
    call_and_inject(orc, inputs.Shape(M=M, H=H, C=C, L=L), seed=150 + M)


@pytest.mark.parametrize("M", [1, 17])
def test_int4_maximum_shape(orc, M):
    call_and_inject(orc, inputs.Shape(M=M, H=16384, C=8, L=1024), seed=250 + M, kind="int4", group=128)


@pytest.mark.parametrize("M,H,C,L,group", [(3, 128, 2, 64, 32), (2, 256, 4, 64, 64), (5, 256, 1, 128, 128),
                                           (4, 128, 2, 32, 32), (7, 96, 3, 32, 32),
                                           # one token: four streams (compiled-in C) and two, groups 128 and 32
                                           (1, 256, 4, 128, 128), (1, 128, 2, 64, 32)])
def test_int4_shapes(orc, M, H, C, L, group):
    call_and_inject(orc, inputs.Shape(M=M, H=H, C=C, L=L), seed=200 + M, kind="int4", group=group)


def test_int4_tiny_up_group_32(orc):
    # the tiny shape's lowrank (32) is below the group of 64: the up weight uses groups of 32
    call_and_inject(orc, inputs.TINY, inputs.SEEDS["int4"], kind="int4", group=64, up_group=32)


@pytest.mark.parametrize("M,H,C,L,group,up_group", [(16, 2560, 4, 320, 64, None), (40, 512, 2, 64, 32, None),
                                                      (128, 1024, 8, 128, 64, 32), (8, 512, 4, 128, 128, None),
                                                      (130, 512, 4, 128, 64, None)])
def test_int4_tensor_core_path(orc, M, H, C, L, group, up_group):
    # INT4-affine weights from 2 tokens run on tcgen05: each weight tile is dequantised
    # to bf16 hi + lo and multiplied against the activation's hi + lo (three MMAs)
    call_and_inject(orc, inputs.Shape(M=M, H=H, C=C, L=L), seed=400 + M, kind="int4", group=group,
                    up_group=up_group)


@pytest.mark.parametrize("M", [1, 64])
def test_int4_full_shape(orc, M):
    s = inputs.FULL_DECODE
    call_and_inject(orc, inputs.Shape(M=M, H=s.H, C=s.C, L=s.L), inputs.SEEDS["int4"], kind="int4",
                    group=inputs.INT4_GROUP)


@pytest.mark.parametrize("M,H,C,L", [(2, 2560, 4, 320), (7, 1024, 8, 128), (15, 256, 1, 64),
                                     (16, 2560, 4, 320), (40, 2560, 4, 320),
                                     (64, 2560, 4, 320), (100, 2560, 4, 320), (130, 2560, 4, 320),
                                     (256, 2560, 4, 320), (64, 512, 2, 64), (80, 1024, 8, 128),
                                     (70, 320, 3, 64), (96, 256, 1, 128)])
def test_tensor_core_path(orc, M, H, C, L):
    # M >= 2 with bf16 weights runs on tcgen05 (tiles of up to 128 tokens)
    call_and_inject(orc, inputs.Shape(M=M, H=H, C=C, L=L), seed=300 + M)


def test_tensor_core_mixer(orc):
    s = inputs.FULL_DECODE
    M = 128
    w = inputs.make_hc_weights(s.H, s.C, s.L, 8, with_inject=False)
    raw = inputs.make_residual(M, s.H, s.C, 8)
    ref = orc.mixer(raw, w.g, w.down, w.up, H=s.H, C=s.C, L=s.L, eps=EPS)
    mixed = B.hc_mixer(raw.cuda(), w.to("cuda"), H=s.H, C=s.C, eps=EPS)
    torch.cuda.synchronize()
    check_bf16(mixed, ref["mixed"], "tensor-core mixer")


def test_mixer(orc):
    s = inputs.FULL_DECODE
    M = 3
    w = inputs.make_hc_weights(s.H, s.C, s.L, 7, with_inject=False)
    raw = inputs.make_residual(M, s.H, s.C, 7)
    ref = orc.mixer(raw, w.g, w.down, w.up, H=s.H, C=s.C, L=s.L, eps=EPS)
    w_d, raw_d = w.to("cuda"), raw.cuda()
    mixed, mwhole = guarded((M, s.H), torch.bfloat16, -77.0)
    ws = B.workspace(M, s.H, s.C, s.L)
    B.hc_mixer(raw_d, w_d, H=s.H, C=s.C, mixed=mixed, eps=EPS, ws=ws)
    torch.cuda.synchronize()
    assert guard_intact(mwhole, M * s.H, -77.0)
    inv, act = workspace_intermediates(ws, M, s.H, s.C, s.L)
    check_call((mixed, None, inv, act), ref, "mixer")


def test_mixer_equals_call_mixed():
    s = inputs.TINY
    w = inputs.make_hc_weights(s.H, s.C, s.L, 9).to("cuda")
    raw = inputs.make_residual(4, s.H, s.C, 9).cuda()
    mixed_call = gpu_call(raw, w, s.H, s.C)[0]
    mixed_mix = B.hc_mixer(raw, w, H=s.H, C=s.C, eps=EPS)
    torch.cuda.synchronize()
    assert torch.equal(mixed_call, mixed_mix)


def test_prefill_microbatch(orc):
    """attn_hc + inject, mlp_hc + inject on 128 tokens; token t's gates at
    t*C*2 (attn) and t*C*2 + C (mlp) of one buffer, none overwritten."""
    s = inputs.PREFILL
    seed = inputs.SEEDS["prefill"]
    M, H, C, L = s.M, s.H, s.C, s.L
    attn = inputs.make_hc_weights(H, C, L, seed, 0)
    mlp = inputs.make_hc_weights(H, C, L, seed, 1)
    raw = inputs.make_residual(M, H, C, seed)
    oa, om = inputs.make_sublayer_out(M, H, seed, 0), inputs.make_sublayer_out(M, H, seed, 1)
    ref = orc.prefill_pair(raw, attn, oa, mlp, om, H=H, C=C, L=L, eps=EPS, round_residual=True)

    attn_d, mlp_d = attn.to("cuda"), mlp.to("cuda")
    raw_d, oa_d, om_d = raw.cuda(), oa.cuda(), om.cuda()
    gates, gwhole = guarded((M * 2 * C,), torch.float32, float("nan"))
    mixed_a, _, inv_a, act_a = gpu_call(raw_d, attn_d, H, C, gates=gates, stride=2 * C)
    assert torch.isnan(gates.view(M, 2, C)[:, 1]).all(), "attn_hc wrote an mlp gate slot"
    B.hc_inject_add(raw_d, oa_d, gates, H=H, C=C, inject_stride=2 * C)
    raw_after_attn = raw_d.clone()
    mixed_m, _, inv_m, act_m = gpu_call(raw_d, mlp_d, H, C, gates=gates[C:], stride=2 * C)
    B.hc_inject_add(raw_d, om_d, gates[C:], H=H, C=C, inject_stride=2 * C)
    torch.cuda.synchronize()
    assert guard_intact(gwhole, M * 2 * C, float("nan")), "write past the gate buffer"
    assert not torch.isnan(gates).any(), "a gate slot was never written"
    check_fp32(gates.view(M, 2, C), ref["gates"], "gate slots")
    check_bf16(mixed_a, ref["mixed_attn"], "attn mixed")
    check_fp32(inv_a, ref["inv_rms_attn"], "attn inv_rms")
    check_fp32(act_a, ref["a_attn"], "attn act")
    check_bf16(raw_after_attn, ref["raw_after_attn"], "residual after attn inject")
    check_bf16(mixed_m, ref["mixed_mlp"], "mlp mixed")
    # mlp_hc reads the residual after a bf16-rounded inject-add (chained input)
    check_fp32(inv_m, ref["inv_rms_mlp"], "mlp inv_rms", floor=CHAINED_RMS_FLOOR)
    check_fp32(act_m, ref["a_mlp"], "mlp act", floor=CHAINED_RMS_FLOOR)
    # The second inject-add starts from a bf16 residual that may already carry a
    # legitimate rounding flip: the carried-residual bound applies.
    peak = np.maximum(np.abs(to_np(raw)), np.maximum(np.abs(ref["raw_after_attn"]), np.abs(ref["raw_after_mlp"])))
    check_bf16_carried(raw_d, ref["raw_after_mlp"], peak, "residual after mlp inject")

    # The same micro-batch as 128 single-token calls, each at its own gate row.
    raw_t = raw.cuda()
    gates_t = torch.full((M * 2 * C,), float("nan"), device="cuda")
    mixed_t = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    ws = B.workspace(1, H, C, L)
    for t in range(M):
        B.hc_call(raw_t[t:t + 1], attn_d, H=H, C=C, mixed=mixed_t[t:t + 1], inject_w=gates_t[t * 2 * C:],
                  inject_stride=2 * C, ws=ws)
        B.hc_inject_add(raw_t[t:t + 1], oa_d[t:t + 1], gates_t[t * 2 * C:], H=H, C=C, inject_stride=2 * C)
    for t in range(M):
        B.hc_call(raw_t[t:t + 1], mlp_d, H=H, C=C, mixed=mixed_t[t:t + 1],
                  inject_w=gates_t[t * 2 * C + C:], inject_stride=2 * C, ws=ws)
        B.hc_inject_add(raw_t[t:t + 1], om_d[t:t + 1], gates_t[t * 2 * C + C:], H=H, C=C, inject_stride=2 * C)
    torch.cuda.synchronize()
    check_fp32(gates_t.view(M, 2, C), ref["gates"], "per-token gate slots")
    check_bf16(mixed_t, ref["mixed_mlp"], "per-token mlp mixed")
    check_bf16_carried(raw_t, ref["raw_after_mlp"], peak, "per-token residual")


def run_stack_gpu(st, H, C):
    """entry replication, 40 x (attn_hc + inject, mlp_hc + inject), exit mixer."""
    M = st.emb.shape[0]
    L = st.final.down.rows
    raw = B.hc_replicate_entry(st.emb.cuda(), C=C)
    gates = torch.empty((M * 2 * C,), dtype=torch.float32, device="cuda")
    mixed = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    ws = B.workspace(M, H, C, L)
    for (attn, mlp), (oa, om) in zip(st.layers, st.outs):
        B.hc_call(raw, attn, H=H, C=C, mixed=mixed, inject_w=gates, inject_stride=2 * C, ws=ws)
        B.hc_inject_add(raw, oa, gates, H=H, C=C, inject_stride=2 * C)
        B.hc_call(raw, mlp, H=H, C=C, mixed=mixed, inject_w=gates[C:], inject_stride=2 * C, ws=ws)
        B.hc_inject_add(raw, om, gates[C:], H=H, C=C, inject_stride=2 * C)
    out = B.hc_mixer(raw, st.final, H=H, C=C, ws=ws)
    torch.cuda.synchronize()
    return out, raw


def run_stack_gpu_fused(st, H, C):
    """The same stack with every inject-add fused into the call that follows it."""
    M = st.emb.shape[0]
    L = st.final.down.rows
    raw = B.hc_replicate_entry(st.emb.cuda(), C=C)
    gates = torch.empty((M * 2 * C,), dtype=torch.float32, device="cuda")
    mixed = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    ws = B.workspace(M, H, C, L)
    prev_out, prev_gate = None, None
    for (attn, mlp), (oa, om) in zip(st.layers, st.outs):
        for wts, out, slot in ((attn, oa, gates), (mlp, om, gates[C:])):
            if prev_out is None:
                B.hc_call(raw, wts, H=H, C=C, mixed=mixed, inject_w=slot, inject_stride=2 * C, ws=ws)
            else:
                B.hc_inject_call(raw, prev_out, prev_gate, wts, H=H, C=C, prev_inject_stride=2 * C, mixed=mixed,
                                 inject_w=slot, inject_stride=2 * C, ws=ws)
            prev_out, prev_gate = out, slot
    out, _ = B.hc_inject_call(raw, prev_out, prev_gate, st.final, H=H, C=C, prev_inject_stride=2 * C, ws=ws)
    torch.cuda.synchronize()
    return out, raw


@pytest.mark.parametrize("M", [1, 2, 3, 128])
def test_fused_inject_call_is_bit_identical(M):
    s = inputs.FULL_DECODE
    H, C, L = s.H, s.C, s.L
    w1, w2 = inputs.make_hc_weights(H, C, L, 11, 0).to("cuda"), inputs.make_hc_weights(H, C, L, 11, 1).to("cuda")
    wm = inputs.make_hc_weights(H, C, L, 11, 2, with_inject=False).to("cuda")
    raw = inputs.make_residual(M, H, C, 11).cuda()
    o1, o2 = inputs.make_sublayer_out(M, H, 11, 0).cuda(), inputs.make_sublayer_out(M, H, 11, 1).cuda()
    ra, rb = raw.clone(), raw.clone()
    ga = torch.full((M * 2 * C,), float("nan"), device="cuda")
    gb = ga.clone()
    # separate inject-add
    B.hc_call(ra, w1, H=H, C=C, inject_w=ga, inject_stride=2 * C)
    B.hc_inject_add(ra, o1, ga, H=H, C=C, inject_stride=2 * C)
    ma, _ = B.hc_call(ra, w2, H=H, C=C, inject_w=ga[C:], inject_stride=2 * C)
    B.hc_inject_add(ra, o2, ga[C:], H=H, C=C, inject_stride=2 * C)
    xa = B.hc_mixer(ra, wm, H=H, C=C)
    # fused into the following call
    B.hc_call(rb, w1, H=H, C=C, inject_w=gb, inject_stride=2 * C)
    mb, _ = B.hc_inject_call(rb, o1, gb, w2, H=H, C=C, prev_inject_stride=2 * C, inject_w=gb[C:],
                             inject_stride=2 * C)
    xb, none = B.hc_inject_call(rb, o2, gb[C:], wm, H=H, C=C, prev_inject_stride=2 * C)
    torch.cuda.synchronize()
    assert none is None
    assert torch.equal(ma, mb) and torch.equal(xa, xb)
    assert torch.equal(ra, rb)
    assert torch.equal(ga, gb)


@pytest.mark.parametrize("M", [1, 3, 16, 40])
def test_fused_inject_reads_the_previous_gates_after_they_are_written(M):
    """A fused call starts before the previous call has finished (programmatic
    dependent launch) but must read that call's gates only once written: with
    the gate buffer refilled with NaN before every pair, each pair must equal,
    bit for bit, the same pair with a host synchronisation between the calls."""
    s = inputs.FULL_DECODE
    H, C, L = s.H, s.C, s.L
    w1, w2 = inputs.make_hc_weights(H, C, L, 12, 0).to("cuda"), inputs.make_hc_weights(H, C, L, 12, 1).to("cuda")
    raw0 = inputs.make_residual(M, H, C, 12).cuda()
    out = inputs.make_sublayer_out(M, H, 12, 0).cuda()
    ws = B.workspace(M, H, C, L)

    def pair(sync):
        raw = raw0.clone()
        gates = torch.full((M * 2 * C,), float("nan"), device="cuda")
        B.hc_call(raw, w1, H=H, C=C, inject_w=gates, inject_stride=2 * C, ws=ws)
        if sync:
            torch.cuda.synchronize()
        mixed, _ = B.hc_inject_call(raw, out, gates, w2, H=H, C=C, prev_inject_stride=2 * C,
                                    inject_w=gates[C:], inject_stride=2 * C, ws=ws)
        torch.cuda.synchronize()
        return mixed, raw, gates

    want = pair(True)
    assert all(bool(torch.isfinite(t).all()) for t in want)
    for _ in range(25):
        got = pair(False)
        assert all(torch.equal(a, b) for a, b in zip(got, want)), "a fused call read stale gates"


@pytest.mark.parametrize("M", [1, 16])
def test_full_depth_stack(orc, M):
    s = inputs.FULL_DECODE
    H, C, L = s.H, s.C, s.L
    st = inputs.make_stack(M, H, C, L, inputs.STACK_LAYERS, inputs.SEEDS["stack"])
    ref = orc.stack(st.emb, st.layers, st.outs, st.final, H=H, C=C, L=L, eps=EPS, round_residual=True)
    dev = inputs.StackInputs(st.emb, [(a.to("cuda"), m.to("cuda")) for a, m in st.layers],
                             [(a.cuda(), m.cuda()) for a, m in st.outs], st.final.to("cuda"))
    mixed, raw = run_stack_gpu(dev, H, C)
    check_bf16(mixed, ref["mixed"], f"stack mixer output M={M}")
    check_bf16_carried(raw, ref["raw"], ref["peak"], f"stack residual M={M}")
    mixed_f, raw_f = run_stack_gpu_fused(dev, H, C)
    assert torch.equal(raw_f, raw) and torch.equal(mixed_f, mixed), "fused stack differs from the unfused one"
    # The native driver (ts_hc_stack): one chunk of all M tokens runs the same
    # calls in the same order as the fused loop above, so it is bit-identical.
    mixed_d, raw_d = run_stack_driver(dev, H, C, max_chunk=M)
    assert torch.equal(raw_d, raw) and torch.equal(mixed_d, mixed), "driver differs from the fused loop"
    if M > 1:
        # Ragged chunks (5, 5, 5, 1 tokens) take other kernel paths per chunk;
        # every token's output still matches the oracle.
        mixed_c, raw_c = run_stack_driver(dev, H, C, max_chunk=5)
        check_bf16(mixed_c, ref["mixed"], f"chunked driver mixer output M={M}")
        check_bf16_carried(raw_c, ref["raw"][-raw_c.shape[0]:], ref["peak"][-raw_c.shape[0]:],
                           f"chunked driver residual (last chunk) M={M}")


def run_stack_driver(st, H, C, max_chunk):
    """The stack through ts_hc_stack; the sublayer callback hands back the stored outputs."""
    M = st.emb.shape[0]
    seen = []

    def sublayer(layer, which, t0, mixed):
        seen.append((layer, which, t0, mixed.shape[0]))
        return st.outs[layer][which][t0:t0 + mixed.shape[0]]

    mixed, raw = B.hc_stack(st.emb.cuda(), st.layers, st.final, sublayer, C=C, max_chunk=max_chunk)
    torch.cuda.synchronize()
    n = len(st.layers)
    want = [(l, w, t0, min(max_chunk, M - t0)) for t0 in range(0, M, max_chunk) for l in range(n) for w in (0, 1)]
    assert seen == want, "sublayer callbacks out of order"
    return mixed, raw.clone()


@pytest.mark.parametrize("max_chunk", [3, 4])
def test_stack_driver_feeds_mixed_to_the_sublayer(max_chunk):
    """A sublayer that reads mixed (out = bf16(0.5 * mixed + the stored output)):
    the driver equals the same library calls issued one by one, bit for bit."""
    s = inputs.TINY
    H, C, L, M, n = s.H, s.C, s.L, 7, 3
    st = inputs.make_stack(M, H, C, L, n, 21)
    dev = inputs.StackInputs(st.emb, [(a.to("cuda"), m.to("cuda")) for a, m in st.layers],
                             [(a.cuda(), m.cuda()) for a, m in st.outs], st.final.to("cuda"))

    def rule(layer, which, t0, mixed):
        stored = dev.outs[layer][which][t0:t0 + mixed.shape[0]]
        return (0.5 * mixed.float() + stored.float()).to(torch.bfloat16)

    mixed_d, raw_last = B.hc_stack(dev.emb.cuda(), dev.layers, dev.final, rule, C=C, max_chunk=max_chunk)
    torch.cuda.synchronize()
    # the same calls by hand, chunk by chunk
    ws = torch.empty(max(B.ts_hc_workspace_bytes(m, H, C, L) for m in range(1, max_chunk + 1)),
                     dtype=torch.uint8, device="cuda")
    want = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    for t0 in range(0, M, max_chunk):
        m = min(max_chunk, M - t0)
        raw = B.hc_replicate_entry(dev.emb[t0:t0 + m].cuda(), C=C)
        gates = torch.empty((m * 2 * C,), dtype=torch.float32, device="cuda")
        mixed = torch.empty((m, H), dtype=torch.bfloat16, device="cuda")
        prev = None
        for layer, (attn, mlp) in enumerate(dev.layers):
            for which, (wts, slot) in enumerate(((attn, gates), (mlp, gates[C:]))):
                if prev is None:
                    B.hc_call(raw, wts, H=H, C=C, mixed=mixed, inject_w=slot, inject_stride=2 * C, ws=ws)
                else:
                    B.hc_inject_call(raw, prev[0], prev[1], wts, H=H, C=C, prev_inject_stride=2 * C, mixed=mixed,
                                     inject_w=slot, inject_stride=2 * C, ws=ws)
                prev = (rule(layer, which, t0, mixed), slot)
        B.hc_inject_call(raw, prev[0], prev[1], dev.final, H=H, C=C, prev_inject_stride=2 * C,
                         mixed=want[t0:t0 + m], ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(mixed_d, want), "driver differs from the calls issued by hand"
    assert torch.equal(raw_last, raw), "driver's last-chunk residual differs"


def test_stack_driver_int4_matches_oracle(orc):
    """ts_hc_stack on INT4-affine modules (chunks of 4 and 1 tokens: the tensor-core
    and the one-token INT4 paths) against the oracle's stack."""
    H, C, L, M, n = 256, 4, 64, 5, 2
    st = inputs.make_stack(M, H, C, L, n, 23, kind="int4")
    ref = orc.stack(st.emb, st.layers, st.outs, st.final, H=H, C=C, L=L, eps=EPS, round_residual=True)
    dev = inputs.StackInputs(st.emb, [(a.to("cuda"), m.to("cuda")) for a, m in st.layers],
                             [(a.cuda(), m.cuda()) for a, m in st.outs], st.final.to("cuda"))
    mixed, raw = run_stack_driver(dev, H, C, max_chunk=4)
    check_bf16(mixed, ref["mixed"], "INT4 stack mixer output")
    check_bf16_carried(raw, ref["raw"][-1:], ref["peak"][-1:], "INT4 stack residual (last chunk)")


def test_stack_driver_captured_in_a_graph_is_bit_identical():
    """A whole ts_hc_stack pass captured into one CUDA graph and replayed gives the
    same bits as the pass run eagerly (the driver allocates nothing and never
    synchronises)."""
    s = inputs.FULL_DECODE
    H, C, L, M, n = s.H, s.C, s.L, 3, 2
    st = inputs.make_stack(M, H, C, L, n, 24)
    layers = [(a.to("cuda"), m.to("cuda")) for a, m in st.layers]
    outs = [(a.cuda(), m.cuda()) for a, m in st.outs]
    final = st.final.to("cuda")
    emb = st.emb.cuda()
    ws = B.stack_workspace(M, H, C, L)
    eager = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    sub = lambda l, w, t0, mixed: outs[l][w][t0:t0 + mixed.shape[0]]
    B.hc_stack(emb, layers, final, sub, C=C, mixed_out=eager, ws=ws)
    torch.cuda.synchronize()
    replayed = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        B.hc_stack(emb, layers, final, sub, C=C, mixed_out=replayed, ws=ws)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(replayed, eager), "graph replay differs from the eager pass"
    assert B.device_status() == B.TS_OK


def test_stack_driver_rejects_bad_sublayer_outputs():
    s = inputs.TINY
    H, C, L, M = s.H, s.C, s.L, 2
    st = inputs.make_stack(M, H, C, L, 1, 22)
    layers = [(a.to("cuda"), m.to("cuda")) for a, m in st.layers]
    final = st.final.to("cuda")
    emb = st.emb.cuda()
    with pytest.raises(B.HCError, match="inside the workspace"):
        B.hc_stack(emb, layers, final, lambda l, w, t0, mixed: mixed, C=C)   # aliases the driver's buffer
    with pytest.raises(ValueError, match="refused"):
        def boom(l, w, t0, mixed):
            raise ValueError("refused by the sublayer")
        B.hc_stack(emb, layers, final, boom, C=C)
    torch.cuda.synchronize()
    assert B.device_status() == B.TS_OK


@pytest.mark.parametrize("M,H,C,L,kind", [(1, 2560, 4, 320, "bf16"), (1, 256, 4, 32, "bf16"), (3, 256, 4, 32, "bf16"),
                                          (2, 2560, 4, 320, "bf16"),
                                          (16, 2560, 4, 320, "bf16"), (1, 2560, 4, 320, "int4"),
                                          (64, 2560, 4, 320, "int4"), (3, 40, 3, 24, "bf16")])
@pytest.mark.parametrize("with_inject", [True, False])
def test_entry_call_is_replicate_then_call(M, H, C, L, kind, with_inject):
    """The entry replication fused into the first call (one-token, cluster and tensor-core
    paths) equals ts_hc_replicate_entry followed by ts_hc_call / ts_hc_mixer, bit for bit."""
    w = inputs.make_hc_weights(H, C, L, 800 + M, kind=kind, with_inject=with_inject).to("cuda")
    emb = inputs.make_embedding(M, H, 800 + M).cuda()
    raw_a = B.hc_replicate_entry(emb, C=C)
    if with_inject:
        mixed_a, gates_a = B.hc_call(raw_a, w, H=H, C=C)
    else:
        mixed_a, gates_a = B.hc_mixer(raw_a, w, H=H, C=C), None
    raw_b, rwhole = guarded((M, C * H), torch.bfloat16, -3.0)
    _, mixed_b, gates_b = B.hc_entry_call(emb, w, C=C, raw=raw_b)
    torch.cuda.synchronize()
    assert guard_intact(rwhole, M * C * H, -3.0), "write past the end of raw"
    assert torch.equal(raw_b, raw_a) and torch.equal(raw_b, emb.repeat(1, C))
    assert torch.equal(mixed_b, mixed_a)
    if with_inject:
        assert torch.equal(gates_b, gates_a)
    assert B.device_status() == B.TS_OK


# The lm_head reads mixed as stored (bf16). The kernels' mixed may sit one bf16
# rounding step away from the oracle's rounded mixed in a few elements (a
# decision at a tie point); each such element moves a logit by |w[v][h]| times
# that step, so the logits keep the chained fp32 floor (1e-3 of their RMS).
EXIT_CASES = [(1, 2560, 4, 320, 1000), (1, 2560, 4, 320, 32768), (5, 2560, 4, 320, 1000), (20, 2560, 4, 320, 500),
              (3, 256, 4, 32, 777), (1, 256, 4, 32, 152), (1, 256, 4, 32, 7), (2, 2560, 4, 320, 4869),
              (1, 16384, 8, 1024, 1000), (17, 16384, 2, 128, 300)]


@pytest.mark.parametrize("M,H,C,L,V", EXIT_CASES)
def test_exit_logits(orc, M, H, C, L, V):
    """The decoder's exit: the last inject-add fused in front of the mixer, then lm_head
    (one-token, cluster and tensor-core mixers; one and two 16-token lm_head tiles;
    vocabularies below one 16-row box and ones that leave the last CTA's rows ragged)."""
    w = inputs.make_hc_weights(H, C, L, 900 + M, with_inject=False)
    lm = inputs.bf16_normal((V, H), 900 + V, std=0.02)
    raw = inputs.make_residual(M, H, C, 900 + M)
    out = inputs.make_sublayer_out(M, H, 900 + M)
    gate = torch.rand((M, C), generator=torch.Generator().manual_seed(M)) * 2
    ref_raw = orc.round_to_bf16(orc.inject_add(raw, out, gate.double().numpy(), H=H, C=C))
    ref_mixed = orc.mixer(ref_raw, w.g, w.down, w.up, H=H, C=C, L=L, eps=EPS)["mixed"]
    ref_logits = orc.lm_head(orc.round_to_bf16(ref_mixed), lm)
    w_d, lm_d = w.to("cuda"), lm.cuda()
    raw_d = raw.cuda()
    logits, lwhole = guarded((M, V), torch.float32, float("nan"))
    mixed, logits = B.hc_exit_logits(raw_d, w_d, lm_d, H=H, C=C, out=out.cuda(), prev_inject_w=gate.cuda(),
                                     logits=logits, eps=EPS)
    torch.cuda.synchronize()
    assert guard_intact(lwhole, M * V, float("nan")), "write past the end of the logits"
    check_bf16(raw_d, ref_raw, "residual after the fused inject-add")
    check_bf16(mixed, ref_mixed, "exit mixer output")
    check_fp32(logits, ref_logits, "logits", floor=CHAINED_RMS_FLOOR)
    # the same exit without the fused inject-add, on the injected residual: bit for bit
    raw2 = raw.cuda()
    B.hc_inject_add(raw2, out.cuda(), gate.cuda(), H=H, C=C)
    mixed2, logits2 = B.hc_exit_logits(raw2, w_d, lm_d, H=H, C=C, eps=EPS)
    torch.cuda.synchronize()
    assert torch.equal(raw2, raw_d) and torch.equal(mixed2, mixed) and torch.equal(logits2, logits)
    assert B.device_status() == B.TS_OK


def test_replicate_entry():
    emb = inputs.make_embedding(3, 256, 5).cuda()
    raw, whole = guarded((3, 4 * 256), torch.bfloat16, -9.0)
    B.hc_replicate_entry(emb, C=4, raw=raw)
    torch.cuda.synchronize()
    assert guard_intact(whole, 3 * 1024, -9.0)
    assert torch.equal(raw, emb.repeat(1, 4))


def test_m0_is_noop():
    s = inputs.TINY
    w = inputs.make_hc_weights(s.H, s.C, s.L, 0).to("cuda")
    raw = torch.empty((0, s.W), dtype=torch.bfloat16, device="cuda")
    mixed, gates = B.hc_call(raw, w, H=s.H, C=s.C)
    assert mixed.shape == (0, s.H)
    B.hc_inject_add(raw, torch.empty((0, s.H), dtype=torch.bfloat16, device="cuda"), gates, H=s.H, C=s.C)
    torch.cuda.synchronize()


def test_inject_add_strided_gates(orc):
    M, H, C = 3, 64, 4
    raw = inputs.make_residual(M, H, C, 31)
    out = inputs.make_sublayer_out(M, H, 31)
    gates = torch.rand(M * 7, dtype=torch.float32) * 2
    ref = orc.inject_add(raw, out, gates.double().numpy(), H=H, C=C, gate_stride=7)
    r = raw.cuda()
    B.hc_inject_add(r, out.cuda(), gates.cuda(), H=H, C=C, inject_stride=7)
    torch.cuda.synchronize()
    check_bf16(r, ref, "strided inject-add")


def test_bounded_wait_records_a_timeout_and_the_context_stays_usable(orc):
    """The kernels' bounded wait on a barrier that nothing arrives at gives up
    (after about a second) and records TS_ERR_TIMEOUT in the status word; the
    status clears once read, and a call afterwards runs and matches the oracle."""
    import time
    assert B.device_status() == B.TS_OK
    t0 = time.time()
    assert B.ts_hc_selftest_timeout(torch.cuda.current_stream().cuda_stream) == B.TS_OK
    assert B.device_status() == B.TS_ERR_TIMEOUT
    assert 0.5 < time.time() - t0 < 30
    assert B.device_status() == B.TS_OK  # cleared by the read
    res = call_and_inject(orc, inputs.TINY, inputs.SEEDS["tiny"])
    assert res[0].shape == (1, inputs.TINY.H)
    assert B.device_status() == B.TS_OK


def test_device_status_clean():
    assert B.device_status() == B.TS_OK


@pytest.mark.parametrize("M", [2, 3])
def test_few_tokens_equal_one_token_calls(M):
    """The few-token kernels keep the one-token kernels' layout and summation order, so M
    tokens in one call give, bit for bit, what M one-token calls give (tokens are
    independent: families/qwen4/mod.rs, "Chunked prefill is wired")."""
    s = inputs.FULL_DECODE
    H, C, L = s.H, s.C, s.L
    w = inputs.make_hc_weights(H, C, L, 61).to("cuda")
    raw = inputs.make_residual(M, H, C, 61).cuda()
    mixed, gates = B.hc_call(raw, w, H=H, C=C)
    for t in range(M):
        m1, g1 = B.hc_call(raw[t:t + 1].clone(), w, H=H, C=C)
        torch.cuda.synchronize()
        assert torch.equal(m1, mixed[t:t + 1]) and torch.equal(g1, gates[t:t + 1]), f"token {t}"
