"""GPU parity on a seeded sweep of random shapes.

Each case draws a token count, a stream count, a residual width, a low rank and a
weight format, so that the cases fall on every kernel path the host picks from
(one token; two or three tokens with bf16 weights; the tensor-core path when H
and the low rank are multiples of 64; the cluster split-K kernels otherwise).
Each runs the previous sublayer's inject-add fused into a call
(`ts_hc_inject_call`: families/qwen4/mod.rs, decoder pseudocode, an inject-add
followed by the next attn_hc / mlp_hc) and then the exit mixer on the result,
and compares the residual, mixed, the gates, inv_rms and act with the fp64
oracle fed the same inputs; and the entry replication fused into a first call
(`ts_hc_entry_call`) followed by `ts_hc_call_debug`, whose up-projection output
w = sigmoid(up(act)) (mod.rs "Hyper-connections") is compared itself.
"""
import numpy as np
import pytest
import torch

import oracle
from hyper_connection_residual_call_gb300 import binding as B
from hyper_connection_residual_call_gb300 import inputs
from gpu_common import check_bf16, check_fp32, guard_intact, guarded, require_gpu, to_np, workspace_intermediates

pytestmark = pytest.mark.gpu
EPS = 1e-6


def _cases(n=28, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(rng.choice([1, 1, 2, 3, 3, 4, 5, 8, 9, 16, 17, 31, 48, 65, 129]))
        C = int(rng.integers(1, 9))
        H = int(rng.choice([8, 40, 64, 72, 128, 200, 256, 384, 512, 640]))
        L = int(rng.choice([8, 24, 32, 64, 96, 128, 192]))
        kind, group = "bf16", 64
        if H % 64 == 0 and L % 32 == 0 and rng.random() < 0.4:
            groups = [g for g in (128, 64, 32) if L % g == 0 and H % g == 0]
            kind, group = "int4", groups[sum(c[5] == "int4" for c in out) % len(groups)]
        out.append((i, M, H, C, L, kind, group))
    return out


# plus INT4 with groups of 128 on the one-token, cluster and tensor-core paths
CASES = _cases() + [(28, 1, 256, 2, 128, "int4", 128), (29, 3, 384, 3, 256, "int4", 128),
                    (30, 16, 512, 4, 128, "int4", 128)]


def test_sweep_covers_every_path():
    """The sweep must reach each kernel family the host chooses between."""
    tc = lambda M, H, L: M >= 2 and H % 64 == 0 and L % 64 == 0
    kinds = set()
    for _, M, H, C, L, kind, _ in CASES:
        if M == 1:
            kinds.add("one-token")
        elif kind == "bf16" and M <= 3:
            kinds.add("few-token")
        elif tc(M, H, L):
            kinds.add("tensor-core " + kind)
        else:
            kinds.add("cluster")
    assert kinds >= {"one-token", "few-token", "tensor-core bf16", "tensor-core int4", "cluster"}, kinds
    groups = {c[6] for c in CASES if c[5] == "int4"}
    assert groups >= {32, 64, 128}, groups


@pytest.fixture(scope="module")
def orc():
    require_gpu()
    return oracle.get()


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-M{c[1]}-H{c[2]}-C{c[3]}-L{c[4]}-{c[5]}")
def test_fused_call_then_mixer(orc, case):
    i, M, H, C, L, kind, group = case
    seed = 7000 + i
    w = inputs.make_hc_weights(H, C, L, seed, 0, kind=kind, group=group)
    wm = inputs.make_hc_weights(H, C, L, seed, 1, kind=kind, group=group, with_inject=False)
    raw = inputs.make_residual(M, H, C, seed)
    out = inputs.make_sublayer_out(M, H, seed)
    # Previous gates (values in (0, 2)) drawn as powers of two: raw + out * gate is then
    # exact in fp32, or differs from raw by less than 2^-16 of it, so the kernels' fp32
    # fused multiply-add and the oracle's fp64 sum round to the same bf16 residual, and
    # the call's inputs agree bit for bit. With other gates, one element in some tens of
    # thousands lands near a bf16 tie, rounds the other way, and moves act near zero
    # past the fp32 bar (the chained tests allow for that with a larger floor).
    prev = torch.from_numpy(2.0 ** np.random.default_rng(seed).integers(-3, 1, (M, C))).float()

    # oracle: the inject-add (rounded to bf16 as the residual is stored), the call,
    # then the exit mixer on the same residual
    inj = orc.round_to_bf16(orc.inject_add(raw, out, prev, H=H, C=C))
    ref = orc.hc_call(inj, w.g, w.down, w.up, w.inject, H=H, C=C, L=L, eps=EPS)
    ref_mix = orc.mixer(inj, wm.g, wm.down, wm.up, H=H, C=C, L=L, eps=EPS)

    w_d, wm_d = w.to("cuda"), wm.to("cuda")
    raw_d, rwhole = guarded((M, C * H), torch.bfloat16, -5.0)
    raw_d.copy_(raw.cuda())
    out_d, prev_d = out.cuda(), prev.cuda()
    mixed, mwhole = guarded((M, H), torch.bfloat16, -77.0)
    gates, gwhole = guarded((M, C), torch.float32, float("nan"))
    ws = B.workspace(M, H, C, L)
    tag = f"{kind} M={M} H={H} C={C} L={L} group={group}"
    B.hc_inject_call(raw_d, out_d, prev_d, w_d, H=H, C=C, prev_inject_stride=C, mixed=mixed, inject_w=gates,
                     inject_stride=C, eps=EPS, ws=ws)
    torch.cuda.synchronize()
    assert guard_intact(rwhole, M * C * H, -5.0), f"{tag}: write past the residual"
    assert guard_intact(mwhole, M * H, -77.0), f"{tag}: write past mixed"
    assert guard_intact(gwhole, M * C, float("nan")), f"{tag}: write past the gates"
    assert np.array_equal(to_np(raw_d), inj), f"{tag}: residual after the fused inject-add differs from the oracle's"
    check_bf16(mixed, ref["mixed"], f"{tag} mixed")
    check_fp32(gates, ref["gate"], f"{tag} gates")
    inv, act = workspace_intermediates(ws, M, H, C, L)
    check_fp32(inv, ref["inv_rms"], f"{tag} inv_rms")
    check_fp32(act, ref["a"], f"{tag} act")

    mixed2 = B.hc_mixer(raw_d, wm_d, H=H, C=C, eps=EPS)
    torch.cuda.synchronize()
    check_bf16(mixed2, ref_mix["mixed"], f"{tag} exit mixer")


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-M{c[1]}-H{c[2]}-C{c[3]}-L{c[4]}-{c[5]}")
def test_entry_call_then_w(orc, case):
    i, M, H, C, L, kind, group = case
    seed = 9000 + i
    w = inputs.make_hc_weights(H, C, L, seed, 0, kind=kind, group=group)
    emb = inputs.make_residual(M, H, 1, seed)  # [M][H]
    rep = orc.replicate_entry(emb, H=H, C=C)
    ref = orc.hc_call(rep, w.g, w.down, w.up, w.inject, H=H, C=C, L=L, eps=EPS, want_w=True)

    w_d = w.to("cuda")
    tag = f"{kind} M={M} H={H} C={C} L={L} group={group}"
    raw, mixed, gates = B.hc_entry_call(emb.cuda(), w_d, C=C, eps=EPS)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(raw), rep), f"{tag}: replicated residual"
    check_bf16(mixed, ref["mixed"], f"{tag} entry call mixed")
    check_fp32(gates, ref["gate"], f"{tag} entry call gates")

    mixed2, gates2, wv = B.hc_call_debug(raw, w_d, H=H, C=C, eps=EPS)
    torch.cuda.synchronize()
    check_bf16(mixed2, ref["mixed"], f"{tag} mixed")
    check_fp32(wv, ref["w"], f"{tag} w = sigmoid(up(act))")
