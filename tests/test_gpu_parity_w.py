"""GPU parity of every intermediate of the call, including the up projection's
sigmoid output w, on every kernel path; at the workload's weight scale and at
scales that take silu and sigmoid out of their near-linear range; and on the
method's degenerate inputs.

w = sigmoid(input_mix_weight_up(act)) (families/qwen4/mod.rs,
"## Hyper-connections") never leaves the chip in the regular entry points; the
debug entry point ts_hc_call_debug writes it. Each case runs that entry point
through the C ABI, checks that its other outputs equal ts_hc_call's (or
ts_hc_mixer's) bit for bit, and compares w, act, inv_rms and the gates with
the fp64 oracle at the fp32 bar, mixed at the bf16 bar. tests/
test_parity_controls.py shows that the w check fails when the up GEMV is
skipped (w = 0.5) at these shapes, which the mixed check alone does not at the
tiny shape.
"""
import numpy as np
import pytest
import torch

import oracle
from hyper_connection_residual_call_gb300 import binding as B
from hyper_connection_residual_call_gb300 import inputs
from hyper_connection_residual_call_gb300.inputs import HCWeights, Weight, quantize_int4_affine
from gpu_common import check_bf16, check_fp32, require_gpu, workspace_intermediates

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def run_and_check(orc, raw, w, H, C, tag):
    """ts_hc_call_debug vs the oracle (every output) and vs the regular entry point (bit for bit)."""
    M, L = raw.shape[0], w.down.rows
    ref = orc.hc_call(raw, w.g, w.down, w.up, w.inject, H=H, C=C, L=L, eps=EPS, want_w=True)
    w_d, raw_d = w.to("cuda"), raw.cuda()
    ws = B.workspace(M, H, C, L)
    w_out = torch.full((M, C * H), float("nan"), dtype=torch.float32, device="cuda")
    mixed, gates, w_gpu = B.hc_call_debug(raw_d, w_d, H=H, C=C, eps=EPS, ws=ws, w_out=w_out)
    torch.cuda.synchronize()
    inv, act = workspace_intermediates(ws, M, H, C, L)
    inv, act = inv.clone(), act.clone()
    # the regular entry point: same kernels, same bits
    ws2 = B.workspace(M, H, C, L)
    if w.inject is not None:
        mixed2, gates2 = B.hc_call(raw_d, w_d, H=H, C=C, eps=EPS, ws=ws2)
    else:
        mixed2, gates2 = B.hc_mixer(raw_d, w_d, H=H, C=C, eps=EPS, ws=ws2), None
    torch.cuda.synchronize()
    inv2, act2 = workspace_intermediates(ws2, M, H, C, L)
    assert torch.equal(mixed, mixed2), f"{tag}: the debug entry point changed mixed"
    assert torch.equal(inv, inv2) and torch.equal(act, act2), f"{tag}: the debug entry point changed act / inv_rms"
    if gates is not None:
        assert torch.equal(gates, gates2), f"{tag}: the debug entry point changed the gates"
    worst = {
        "w": check_fp32(w_gpu, ref["w"], f"{tag} w"),
        "mixed": check_bf16(mixed, ref["mixed"], f"{tag} mixed"),
        "inv_rms": check_fp32(inv, ref["inv_rms"], f"{tag} inv_rms"),
        "act": check_fp32(act, ref["a"], f"{tag} act"),
    }
    if gates is not None:
        worst["gate"] = check_fp32(gates, ref["gate"], f"{tag} gate")
    assert B.device_status() == B.TS_OK
    return worst


# (M, H, C, L, kind, group): each kernel path of the library.
PATHS = {
    # one token: hc_down1_kernel + hc_up1_kernel (four streams compiled in, and any C)
    "one-token bf16 full shape": (1, 2560, 4, 320, "bf16", 0),
    "one-token bf16 tiny": (1, 256, 4, 32, "bf16", 0),
    "one-token bf16 two streams": (1, 128, 2, 64, "bf16", 0),
    "one-token int4 full shape": (1, 2560, 4, 320, "int4", 64),
    "one-token int4 group 128": (1, 256, 4, 128, "int4", 128),
    "one-token int4 two streams": (1, 128, 2, 64, "int4", 32),
    # two tokens, bf16: the few-token kernels (the one-token layout with a token loop)
    "few-token bf16 full shape": (2, 2560, 4, 320, "bf16", 0),
    "few-token bf16 eight streams": (2, 1024, 8, 128, "bf16", 0),
    "few-token bf16 one stream, odd lowrank": (2, 96, 1, 40, "bf16", 0),
    "few-token bf16 three tokens": (3, 2560, 4, 320, "bf16", 0),
    # from 2 tokens, shapes the tensor cores do not take: the cluster split-K kernels
    "cluster bf16 odd shape": (3, 40, 3, 24, "bf16", 0),
    "cluster bf16 five streams": (11, 96, 5, 40, "bf16", 0),
    "cluster bf16 one stream": (5, 64, 1, 8, "bf16", 0),
    "cluster int4": (7, 96, 3, 32, "int4", 32),
    "cluster int4 two streams": (4, 128, 2, 32, "int4", 32),
    # from 2 tokens, H and lowrank multiples of 64: tcgen05
    "tensor-core bf16 M=16": (16, 2560, 4, 320, "bf16", 0),
    "tensor-core bf16 M=128": (128, 2560, 4, 320, "bf16", 0),
    "tensor-core bf16 ragged": (70, 320, 3, 64, "bf16", 0),
    "tensor-core bf16 two tiles": (130, 512, 4, 128, "bf16", 0),
    "tensor-core int4 M=64": (64, 2560, 4, 320, "int4", 64),
    "tensor-core int4 group 32": (40, 512, 2, 64, "int4", 32),
}


def _weights(H, C, L, kind, group, seed, std=0.02, with_inject=True):
    return inputs.make_hc_weights(H, C, L, seed, kind=kind, group=group or 64, std=std, with_inject=with_inject)


@pytest.mark.parametrize("name", sorted(PATHS))
def test_w_and_every_intermediate_on_every_path(orc, name):
    M, H, C, L, kind, group = PATHS[name]
    w = _weights(H, C, L, kind, group, 700 + M)
    raw = inputs.make_residual(M, H, C, 700 + M)
    run_and_check(orc, raw, w, H, C, name)


@pytest.mark.parametrize("M", [1, 16])
def test_w_of_the_exit_mixer(orc, M):
    s = inputs.FULL_DECODE
    w = _weights(s.H, s.C, s.L, "bf16", 0, 710 + M, with_inject=False)
    raw = inputs.make_residual(M, s.H, s.C, 710 + M)
    run_and_check(orc, raw, w, s.H, s.C, f"mixer M={M}")


# Weight scales that put the pre-activations of silu and sigmoid at a few units
# (std 0.1 at the full shape) or saturate them (0.3 and more).
LARGE = [
    ("one-token bf16", 1, 2560, 4, 320, "bf16", 0, 0.1), ("one-token bf16 saturating", 1, 2560, 4, 320, "bf16", 0, 0.3),
    ("one-token int4", 1, 2560, 4, 320, "int4", 64, 0.1), ("tiny saturating", 1, 256, 4, 32, "bf16", 0, 0.3),
    ("tensor-core bf16 M=16", 16, 2560, 4, 320, "bf16", 0, 0.1),
    ("tensor-core bf16 M=128 saturating", 128, 2560, 4, 320, "bf16", 0, 0.3),
    ("tensor-core int4 M=64", 64, 2560, 4, 320, "int4", 64, 0.1),
    ("tensor-core int4 M=64 saturating", 64, 2560, 4, 320, "int4", 64, 0.3),
    ("cluster bf16", 3, 40, 3, 24, "bf16", 0, 0.5), ("cluster int4", 7, 96, 3, 32, "int4", 32, 0.5),
]


@pytest.mark.parametrize("case", LARGE, ids=[c[0] for c in LARGE])
def test_large_weights_leave_the_linear_region(orc, case):
    name, M, H, C, L, kind, group, std = case
    w = _weights(H, C, L, kind, group, 720 + M, std=std)
    raw = inputs.make_residual(M, H, C, 720 + M)
    # the case is only meaningful if the activations really are non-linear
    ref = orc.hc_call(raw[:1], w.g, w.down, w.up, w.inject, H=H, C=C, L=L, eps=EPS, want_w=True)
    assert np.abs(ref["w"] - 0.5).max() > 0.3, "w stays near sigmoid(0)"
    run_and_check(orc, raw, w, H, C, f"{name}, weight std {std}")


def _with_streams(raw, C, H, fn):
    x = raw.float().view(raw.shape[0], C, H)
    fn(x)
    return x.reshape(raw.shape[0], C * H).to(torch.bfloat16)


EDGE_SHAPES = [(1, 2560, 4, 320), (16, 2560, 4, 320), (3, 40, 3, 24)]


@pytest.mark.parametrize("M,H,C,L", EDGE_SHAPES)
def test_a_zero_stream(orc, M, H, C, L):
    """A stream of zeros: inv_rms = 1/sqrt(eps), its normed part is zero."""
    w = _weights(H, C, L, "bf16", 0, 730 + M)
    raw = _with_streams(inputs.make_residual(M, H, C, 730 + M), C, H, lambda x: x[:, 1].zero_())
    run_and_check(orc, raw, w, H, C, "zero stream")


@pytest.mark.parametrize("M,H,C,L", EDGE_SHAPES)
def test_constant_streams(orc, M, H, C, L):
    """Every stream constant: inv_rms = 1/sqrt(s^2 + eps) in closed form."""
    w = _weights(H, C, L, "bf16", 0, 740 + M)
    levels = torch.tensor([0.5, -2.0, 3.0, 1.0 / 1024, -0.75][:C])

    def fill(x):
        x.copy_(levels.view(1, C, 1).expand_as(x))

    raw = _with_streams(inputs.make_residual(M, H, C, 740 + M), C, H, fill)
    run_and_check(orc, raw, w, H, C, "constant streams")


@pytest.mark.parametrize("M,H,C,L", EDGE_SHAPES)
def test_a_residual_scaled_by_1e3(orc, M, H, C, L):
    """The norm makes the call (nearly) scale invariant; a large residual must not overflow or lose accuracy."""
    w = _weights(H, C, L, "bf16", 0, 750 + M)
    raw = (inputs.make_residual(M, H, C, 750 + M).float() * 1000.0).to(torch.bfloat16)
    run_and_check(orc, raw, w, H, C, "residual x 1e3")


def _one_hot_module(H, C, L, kind, group):
    """Down row k reads input (37 k) mod C*H, up row j reads act j mod L, inject
    row c reads input c*H + 5: each projection passes single elements through,
    so act = silu(normed_j / C), gate = 2 sigmoid(normed_j / C), w = sigmoid(act_k)."""
    W = C * H
    down = torch.zeros((L, W))
    down[torch.arange(L), (37 * torch.arange(L)) % W] = 1.0
    up = torch.zeros((W, L))
    up[torch.arange(W), torch.arange(W) % L] = 1.0
    inj = torch.zeros((C, W))
    inj[torch.arange(C), torch.arange(C) * H + 5] = 1.0
    g = inputs.bf16_normal((W,), 777, std=0.1, mean=1.0)
    mats = [t.to(torch.bfloat16) for t in (down, up, inj)]
    if kind == "bf16":
        d, u, i = (Weight("bf16", t.shape[0], t.shape[1], t) for t in mats)
    else:
        d, u, i = (quantize_int4_affine(t, group) for t in mats)
    return HCWeights(g, d, u, i)


@pytest.mark.parametrize("M,kind,group", [(1, "bf16", 0), (16, "bf16", 0), (1, "int4", 64), (64, "int4", 64)])
def test_one_hot_projections(orc, M, kind, group):
    s = inputs.FULL_DECODE
    w = _one_hot_module(s.H, s.C, s.L, kind, group)
    raw = inputs.make_residual(M, s.H, s.C, 760 + M)
    run_and_check(orc, raw, w, s.H, s.C, f"one-hot projections ({kind}, M={M})")
