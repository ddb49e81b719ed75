"""GPU parity of the PLE gate on the wide residual (families/qwen4/mod.rs,
"## PLE") against the fp64 oracle, through the C ABI.

Outputs: the residual after the add (bf16 bar) and the conv state (fp32 bar);
intermediates from the workspace: the value projection, the per-stream gates
and the conv input (fp32 bar). Also: chunks with the state handed over equal
one chunk bit for bit; a zero key projection gives the gate sigmoid(0) = 1/2
exactly; a row id out of range is recorded in the device status word.
"""
import numpy as np
import pytest
import torch

import oracle
from hyper_connection_residual_call_gb300 import binding as B
from hyper_connection_residual_call_gb300 import inputs
from gpu_common import CHAINED_RMS_FLOOR, check_bf16, check_bf16_carried, check_fp32, require_gpu

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def run_gpu(hidden, rows, w, state, C):
    h = hidden.cuda()
    st = state.cuda()
    _, ws = B.hc_ple(h, rows.cuda(), w.to("cuda"), st, C=C, eps=EPS)
    torch.cuda.synchronize()
    M, H = hidden.shape[0], w.value_proj.shape[0]
    vo, go, xo = B.ts_hc_ple_workspace_layout(M, H, C)
    f = ws.view(torch.uint8)
    value = f[vo:vo + 4 * M * H].view(torch.float32).view(M, H)
    gate = f[go:go + 4 * M * C].view(torch.float32).view(M, C)
    x = f[xo:xo + 4 * M * C * H].view(torch.float32).view(M, C * H)
    return h, st, value, gate, x


@pytest.mark.parametrize("M,H,C", [(1, 2560, 4), (5, 2560, 4), (12, 2560, 4), (20, 2560, 4), (3, 128, 4),
                                   (10, 256, 2), (3, 16384, 1)])
def test_ple_matches_oracle(orc, M, H, C):
    w = inputs.make_ple_weights(H, C, 30 + M, n_rows=2048)
    rows = inputs.make_ple_rows(M, 2048, 30 + M)
    hidden = inputs.make_residual(M, H, C, 30 + M)
    state = inputs.make_ple_state(H, C, 30 + M)
    ref = orc.ple(hidden, rows, w.table, w.key_proj, w.value_proj, w.norm_key, w.norm_query, w.norm_conv,
                  w.conv_w, state, H=H, C=C, eps=EPS)
    h, st, value, gate, x = run_gpu(hidden, rows, w, state, C)
    check_bf16(h, ref["result"], f"PLE residual M={M}")
    check_fp32(value, ref["value"], "PLE value")
    check_fp32(gate, ref["gate"], "PLE gate")
    check_fp32(x, ref["x"], "PLE conv input")
    check_fp32(st, ref["state"], "PLE conv state")
    assert B.device_status() == B.TS_OK


def test_ple_chunks_equal_one_pass():
    H, C, M = 2560, 4, 12
    w = inputs.make_ple_weights(H, C, 40, n_rows=512).to("cuda")
    rows = inputs.make_ple_rows(M, 512, 40).cuda()
    hidden = inputs.make_residual(M, H, C, 40).cuda()
    state = inputs.make_ple_state(H, C, 40).cuda()
    h1, s1 = hidden.clone(), state.clone()
    B.hc_ple(h1, rows, w, s1, C=C, eps=EPS)
    h2, s2 = hidden.clone(), state.clone()
    B.hc_ple(h2[:5], rows[:5], w, s2, C=C, eps=EPS)
    B.hc_ple(h2[5:], rows[5:], w, s2, C=C, eps=EPS)
    torch.cuda.synchronize()
    assert torch.equal(h1, h2) and torch.equal(s1, s2)


def test_ple_zero_key_gives_half_gate(orc):
    H, C, M = 256, 4, 3
    w = inputs.make_ple_weights(H, C, 41, n_rows=64)
    w.key_proj.zero_()
    rows = inputs.make_ple_rows(M, 64, 41)
    hidden = inputs.make_residual(M, H, C, 41)
    state = torch.zeros((9, C * H))
    ref = orc.ple(hidden, rows, w.table, w.key_proj, w.value_proj, w.norm_key, w.norm_query, w.norm_conv,
                  w.conv_w, state, H=H, C=C, eps=EPS)
    h, st, value, gate, x = run_gpu(hidden, rows, w, state, C)
    assert torch.all(gate == 0.5)
    check_bf16(h, ref["result"], "PLE residual, zero key")


def test_ple_row_id_out_of_range_is_reported():
    H, C, M = 128, 4, 2
    w = inputs.make_ple_weights(H, C, 42, n_rows=16).to("cuda")
    rows = inputs.make_ple_rows(M, 16, 42)
    rows[1, 3] = 16  # one past the table
    hidden = inputs.make_residual(M, H, C, 42).cuda()
    state = torch.zeros((9, C * H), device="cuda")
    assert B.device_status() == B.TS_OK
    B.hc_ple(hidden, rows.cuda(), w, state, C=C, eps=EPS)
    torch.cuda.synchronize()
    assert B.device_status() == B.TS_ERR_INVALID_ARG
    assert B.device_status() == B.TS_OK  # cleared by the read
    assert torch.isfinite(hidden.float()).all()


@pytest.mark.parametrize("max_chunk", [2, 5])
def test_stack_with_ple_matches_oracle(orc, max_chunk):
    """ts_hc_stack_ple: the PLE before layer 1's attn_hc inside the stack driver,
    chunk by chunk with the conv state carried (chunks of 2: tensor-core calls and a
    one-token tail), against the oracle's stack with the PLE on all 5 tokens at once."""
    H, C, L, M, n = 256, 4, 64, 5, 3
    st = inputs.make_stack(M, H, C, L, n, 41)
    pw = inputs.make_ple_weights(H, C, 41, n_rows=64)
    rows = inputs.make_ple_rows(M, 64, 41)
    state = inputs.make_ple_state(H, C, 41)
    ref = orc.stack(st.emb, st.layers, st.outs, st.final, H=H, C=C, L=L, eps=EPS, round_residual=True, ple=pw,
                    ple_rows=rows, ple_state=state)
    layers = [(a.to("cuda"), m.to("cuda")) for a, m in st.layers]
    outs = [(a.cuda(), m.cuda()) for a, m in st.outs]
    state_d = state.cuda()

    def sublayer(layer, which, t0, mixed):
        return outs[layer][which][t0:t0 + mixed.shape[0]]

    mixed, raw = B.hc_stack(st.emb.cuda(), layers, st.final.to("cuda"), sublayer, C=C, max_chunk=max_chunk,
                            eps=EPS, ple=pw.to("cuda"), ple_rows=rows.cuda(), ple_state=state_d)
    torch.cuda.synchronize()
    last = raw.shape[0]
    check_bf16(mixed, ref["mixed"], f"stack with PLE: mixer output (chunks of {max_chunk})")
    check_bf16_carried(raw, ref["raw"][-last:], ref["peak"][-last:], "stack with PLE: last chunk's residual")
    check_fp32(state_d, ref["ple_state"], "stack with PLE: conv state", floor=CHAINED_RMS_FLOOR)
    assert B.device_status() == B.TS_OK
