"""Planted defects must fail the GPU parity checks (CPU only).

The GPU tests compare the kernels with the fp64 oracle through the tolerance
checks of ``gpu_common``. A check that cannot fail for the step it claims to
cover pins nothing, so each test here builds what a defective kernel would
return -- by planting the defect in the oracle's own computation, on the CPU --
and requires the check that the GPU tests apply to reject it:

* the up projection's sigmoid output ``w`` (families/qwen4/mod.rs,
  "## Hyper-connections": w = sigmoid(up(act))) replaced by sigmoid(0) = 0.5,
  or its pre-activation scaled by 0.8, at every shape whose ``w`` the GPU
  tests compare;
* the 40-layer stack (families/qwen4/mod.rs, decoder pseudocode) with one
  layer's gate scaled by 0.9, one inject-add skipped, or two streams swapped
  before one inject-add: the carried-residual rule must reject each;
* a correct evaluation in another precision (gates perturbed by 1e-6
  relative, the inject-add in fp32) must pass the same rule;
* a 1% error on the act of a chained call must fail the chained fp32 bar.
"""
import numpy as np
import pytest

import oracle
from hyper_connection_residual_call_gb300 import inputs
from gpu_common import CHAINED_RMS_FLOOR, carried_stats, check_bf16, check_bf16_carried, check_fp32

EPS = 1e-6


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


# The shapes (and weight scales) whose w the GPU tests compare.
W_CASES = [
    ("tiny", inputs.TINY, 0.02), ("full decode", inputs.FULL_DECODE, 0.02),
    ("small two-stream", inputs.Shape(M=1, H=128, C=2, L=64), 0.02),
    ("odd cluster shape", inputs.Shape(M=3, H=40, C=3, L=24), 0.02),
    ("full shape, large weights", inputs.FULL_DECODE, 0.1),
]


@pytest.mark.parametrize("name,shape,std", W_CASES, ids=[c[0] for c in W_CASES])
def test_up_output_defects_fail_the_w_check(orc, name, shape, std):
    H, C, L, M = shape.H, shape.C, shape.L, shape.M
    w = inputs.make_hc_weights(H, C, L, 600 + M, std=std)
    raw = inputs.make_residual(M, H, C, 600 + M)
    ref = orc.hc_call(raw, w.g, w.down, w.up, w.inject, H=H, C=C, L=L, eps=EPS, want_w=True)
    check_fp32(ref["w"], ref["w"], "the oracle against itself")
    with pytest.raises(AssertionError):  # the up GEMV skipped: w = sigmoid(0)
        check_fp32(np.full_like(ref["w"], 0.5), ref["w"], f"{name}: w = 0.5")
    logit = np.log(ref["w"]) - np.log1p(-ref["w"])
    with pytest.raises(AssertionError):  # the up pre-activation scaled by 0.8
        check_fp32(_sigmoid(0.8 * logit), ref["w"], f"{name}: 0.8 * up")


def _stack(orc, st, H, C, L, defect=None, gate_noise=0.0, fp32_inject=False, seed=0):
    """The oracle's stack loop, built from its pinned calls, with one planted
    defect (or a correct evaluation in another precision)."""
    rng = np.random.default_rng(seed)
    raw = orc.replicate_entry(st.emb, H=H, C=C)
    peak = np.abs(raw)
    M = raw.shape[0]
    for l, ((attn, mlp), (oa, om)) in enumerate(zip(st.layers, st.outs)):
        for which, (w, o) in enumerate(((attn, oa), (mlp, om))):
            gate = orc.hc_call(raw, w.g, w.down, w.up, w.inject, H=H, C=C, L=L, eps=EPS)["gate"]
            if gate_noise:
                gate = gate * (1 + gate_noise * rng.standard_normal(gate.shape))
            src = raw
            if defect == ("gate x 0.9", l, which):
                gate = 0.9 * gate
            if defect == ("swapped streams", l, which):
                src = raw.reshape(M, C, H)[:, [1, 0] + list(range(2, C)), :].reshape(M, C * H)
            if defect == ("skipped inject", l, which):
                new = src
            elif fp32_inject:
                o32 = o.float().numpy().astype(np.float32).reshape(M, 1, H)
                new = (src.astype(np.float32).reshape(M, C, H) + o32 * gate.astype(np.float32).reshape(M, C, 1))
                new = new.reshape(M, C * H).astype(np.float64)
            else:
                new = orc.inject_add(src, o, gate, H=H, C=C)
            raw = orc.round_to_bf16(new)
            peak = np.maximum(peak, np.abs(raw))
    mixed = orc.mixer(raw, st.final.g, st.final.down, st.final.up, H=H, C=C, L=L, eps=EPS)["mixed"]
    return raw, mixed, peak


@pytest.fixture(scope="module")
def stack_ref(orc):
    s = inputs.FULL_DECODE
    st = inputs.make_stack(1, s.H, s.C, s.L, inputs.STACK_LAYERS, inputs.SEEDS["stack"])
    raw, mixed, peak = _stack(orc, st, s.H, s.C, s.L)
    want = orc.stack(st.emb, st.layers, st.outs, st.final, H=s.H, C=s.C, L=s.L, eps=EPS, round_residual=True)
    # the loop above is the oracle's own stack, bit for bit
    assert np.array_equal(raw, want["raw"]) and np.array_equal(mixed, want["mixed"])
    assert np.array_equal(peak, want["peak"])
    return st, raw, mixed, peak


@pytest.mark.parametrize("defect", [("gate x 0.9", 20, 0), ("gate x 0.9", 39, 1), ("skipped inject", 20, 0),
                                    ("swapped streams", 20, 0)],
                         ids=["gate-0.9-layer-20", "gate-0.9-last-mlp", "skipped-inject", "swapped-streams"])
def test_stack_defects_fail_the_carried_residual_check(orc, stack_ref, defect):
    s = inputs.FULL_DECODE
    st, ref_raw, ref_mixed, peak = stack_ref
    raw, mixed, _ = _stack(orc, st, s.H, s.C, s.L, defect=defect)
    stats = carried_stats(raw, ref_raw, peak)
    with pytest.raises(AssertionError):
        check_bf16_carried(raw, ref_raw, peak, f"stack residual with {defect}")
    # every statistic of the rule rejects it on its own
    assert stats["max_loose"] > 1.0 and stats["rms_ulps"] > 1.25 and stats["frac_beyond_plain"] > 0.25, stats
    with pytest.raises(AssertionError):  # the exit mixer's output moves past its plain bar too
        check_bf16(mixed, ref_mixed, f"stack mixer output with {defect}")


def test_a_correct_evaluation_in_fp32_passes_the_carried_residual_check(orc, stack_ref):
    s = inputs.FULL_DECODE
    st, ref_raw, ref_mixed, peak = stack_ref
    raw, mixed, _ = _stack(orc, st, s.H, s.C, s.L, gate_noise=1e-6, fp32_inject=True, seed=1)
    stats = carried_stats(raw, ref_raw, peak)
    assert 0 < stats["frac_beyond_plain"], "the perturbation must move some rounding decisions"
    check_bf16_carried(raw, ref_raw, peak, "stack residual, correct fp32 evaluation")
    check_bf16(mixed, ref_mixed, "stack mixer output, correct fp32 evaluation")


def test_a_one_percent_act_error_fails_the_chained_fp32_bar(orc):
    s = inputs.PREFILL
    w = inputs.make_hc_weights(s.H, s.C, s.L, 2, 1)
    raw = inputs.make_residual(4, s.H, s.C, 2)
    ref = orc.hc_call(raw, w.g, w.down, w.up, w.inject, H=s.H, C=s.C, L=s.L, eps=EPS)
    check_fp32(ref["a"], ref["a"], "chained act", floor=CHAINED_RMS_FLOOR)
    with pytest.raises(AssertionError):
        check_fp32(1.01 * ref["a"], ref["a"], "chained act x 1.01", floor=CHAINED_RMS_FLOOR)
    with pytest.raises(AssertionError):
        check_fp32(1.01 * ref["inv_rms"], ref["inv_rms"], "chained inv_rms x 1.01", floor=CHAINED_RMS_FLOOR)
