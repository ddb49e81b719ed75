"""Pins for the fp64 oracle: checks that do not retype the oracle's formula.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with something fixed independently of it:

* exact decoders and rounding versus torch / numpy's own conversions;
* closed forms of the call at special inputs (one-hot weights, constant or
  zero streams, zero projections), evaluated with scipy/torch library
  routines (expit, silu, rms_norm) -- these pin the two divisions by C and
  their order (families/qwen4/hc.rs: "exactly two, not three"), the direct
  norm scale, the mean over C (families/qwen4/mod.rs, "MEAN not sum"), the
  injection trap and the stream-major flatten order;
* invariants: scale invariance of the normalised path, stream-permutation
  equivariance, token independence, mixer == call without its gate;
* a library formulation (torch fp64 rms_norm / linear / silu / sigmoid) on
  tiny shapes C in {1,2,4}, H in {1,2,8}, L in {1,3}.

``tests/test_oracle_mutants.py`` compiles copies of the oracle with planted
mistakes and checks that at least one pin fails for each.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F
from scipy.special import expit

from hyper_connection_residual_call_gb300 import inputs
from hyper_connection_residual_call_gb300.inputs import Weight, quantize_int4_affine

EPS = 1e-6


def _bf(x) -> torch.Tensor:
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def _w(x) -> Weight:
    t = x if isinstance(x, torch.Tensor) and x.dtype == torch.bfloat16 else _bf(x)
    return Weight("bf16", t.shape[0], t.shape[1], t)


def _randn(rng, *shape, std=1.0):
    return _bf(rng.standard_normal(shape) * std)


def _close(a, b, rtol=1e-12, atol=1e-14, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    err = np.abs(a - b)
    lim = atol + rtol * np.abs(b)
    assert np.all(err <= lim), f"{what}: max err {err.max():.3e} (worst at {np.argmax(err - lim)})"


def _silu(x):
    return F.silu(torch.as_tensor(np.asarray(x, dtype=np.float64))).numpy()


# --------------------------------------------------------------- decoders

def pin_bf16_decode(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = np.array([orc.bf16_value(int(b)) for b in bits])
    ok = ~np.isnan(ref)
    assert np.all(np.isnan(got[~ok])), "bf16 NaN patterns"
    assert np.array_equal(got[ok], ref[ok]), "bf16 decode"


def pin_f16_decode(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_value(int(b)) for b in bits])
    ok = ~np.isnan(ref)
    assert np.all(np.isnan(got[~ok])), "fp16 NaN patterns"
    assert np.array_equal(got[ok], ref[ok]), "fp16 decode"


def pin_round_to_bf16(orc):
    rng = np.random.default_rng(11)
    vals = [rng.standard_normal(4000).astype(np.float32),
            (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # subnormal range
            (rng.standard_normal(2000) * 1e30).astype(np.float32)]
    # exact midpoints between neighbouring bf16 values: ties must go to even
    b = rng.integers(0x0080, 0x7F00, 3000).astype(np.uint32)
    mids = ((b << 16) | 0x8000).astype(np.uint32).view(np.float32)
    vals += [mids, -mids]
    x = np.concatenate(vals)
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    got = orc.round_to_bf16(x.astype(np.float64))
    assert np.array_equal(got, ref), f"bf16 rounding: {np.sum(got != ref)} mismatches"


def _int4_fixture():
    rows, cols, group = 3, 256, 64
    q = (np.arange(rows)[:, None] * 7 + np.arange(cols)[None, :] * 3) % 16
    s = np.array([[0.5, 0.25, 1.5, 0.0], [2.0, 0.125, 0.75, 3.0], [0.0625, 1.0, 0.5, 0.25]])
    b = np.array([[-1.25, 3.0, 0.0, 2.5], [-4.0, 0.5, 1.0, -0.375], [0.25, -2.0, 0.125, 7.0]])
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    w = Weight("int4", rows, cols, torch.from_numpy(packed),
               torch.from_numpy(s.astype(np.float16)), torch.from_numpy(b.astype(np.float16)), group)
    dense = q * np.repeat(s, group, axis=1) + np.repeat(b, group, axis=1)
    return w, dense


def pin_int4_decode(orc):
    w, dense = _int4_fixture()
    assert np.array_equal(orc.weight_values(w), dense), "INT4-affine decode"


def pin_int4_decode_every_group(orc):
    # Each supported group size (32, 64, 128 inputs per scale and bias), with
    # scales and biases exact in fp16, so the dense weight is exact in fp64.
    rows, cols = 3, 256
    q = (np.arange(rows)[:, None] * 5 + np.arange(cols)[None, :] * 11) % 16
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    for group in (32, 64, 128):
        ng = cols // group
        r, j = np.arange(rows)[:, None], np.arange(ng)[None, :]
        s = ((r * 5 + j * 3) % 8 + 1) * 0.125
        b = ((r * 3 + j * 7) % 9 - 4) * 0.25
        w = Weight("int4", rows, cols, torch.from_numpy(packed),
                   torch.from_numpy(s.astype(np.float16)), torch.from_numpy(b.astype(np.float16)), group)
        dense = q * np.repeat(s, group, axis=1) + np.repeat(b, group, axis=1)
        assert np.array_equal(orc.weight_values(w), dense), f"INT4-affine decode, group {group}"


def pin_gemv(orc):
    rng = np.random.default_rng(3)
    wt = _randn(rng, 7, 33)
    x = rng.standard_normal(33)
    _close(orc.gemv(_w(wt), x), wt.double().numpy() @ x, rtol=1e-13, atol=1e-15, what="bf16 gemv")
    w4, dense = _int4_fixture()
    x4 = rng.standard_normal(256)
    _close(orc.gemv(w4, x4), dense @ x4, rtol=1e-13, atol=1e-13, what="int4 gemv")


# --------------------------------------------------------------- the call

def pin_norm_via_zero_down(orc):
    """Wd = 0 => a = 0 => w = 0.5 => mixed = 0.5 * mean_c rms_norm(raw_c) * g_c."""
    rng = np.random.default_rng(5)
    M, C, H, L = 2, 3, 8, 5
    raw = _randn(rng, M, C * H, std=2.0)
    g = _bf(1.0 + 0.3 * rng.standard_normal(C * H))
    wd = _w(np.zeros((L, C * H)))
    wu = _w(_randn(rng, C * H, L))
    wi = _w(_randn(rng, C, C * H))
    r = orc.hc_call(raw, g, wd, wu, wi, H=H, C=C, L=L, eps=EPS, want_w=True)
    x = raw.double().view(M, C, H)
    n = torch.stack([F.rms_norm(x[:, c], (H,), weight=g.double().view(C, H)[c], eps=EPS)
                     for c in range(C)], dim=1)
    _close(r["a"], np.zeros((M, L)), what="a with zero down")
    _close(r["w"], np.full((M, C * H), 0.5), what="w with zero down")
    _close(r["mixed"], 0.5 * n.mean(dim=1).numpy(), what="mixed = 0.5 * mean_c rms_norm")


def pin_inv_rms_constant_streams(orc):
    C, H, L = 3, 8, 2
    s = [0.5, -2.0, 3.0]
    raw = _bf(np.repeat(s, H)[None, :])
    g = _bf(np.ones(C * H))
    r = orc.hc_call(raw, g, _w(np.zeros((L, C * H))), _w(np.zeros((C * H, L))), None,
                    H=H, C=C, L=L, eps=EPS)
    _close(r["inv_rms"][0], [1.0 / math.sqrt(v * v + EPS) for v in s], rtol=1e-15,
           what="inv_rms of constant streams")


def _const_stream_setup(C, H, s, g):
    raw = _bf(np.repeat(s, H)[None, :])
    n = np.repeat([v / math.sqrt(v * v + EPS) for v in s], H) * g.double().numpy()
    return raw, n


def pin_down_one_hot(orc):
    """Wd[k] = e_{j_k} => a_k = silu(n_{j_k} / C): the first /C, before silu."""
    C, H, L = 4, 8, 3
    s = [1.0, -1.5, 2.0, 0.75]
    rng = np.random.default_rng(7)
    g = _bf(3.0 + rng.standard_normal(C * H))
    raw, n = _const_stream_setup(C, H, s, g)
    picks = [1, 10, 29]
    wd = np.zeros((L, C * H))
    for k, j in enumerate(picks):
        wd[k, j] = 1.0
    r = orc.hc_call(raw, g, _w(wd), _w(np.zeros((C * H, L))), None, H=H, C=C, L=L, eps=EPS)
    _close(r["a"][0], _silu(n[picks] / C), what="a = silu(z / C)")


def pin_inject_one_hot(orc):
    """Wi[c] = e_{j_c} => gate_c = 2 sigmoid(n_{j_c} / C): the second /C and the x2."""
    C, H, L = 4, 8, 2
    s = [1.0, -1.5, 2.0, 0.75]
    rng = np.random.default_rng(8)
    g = _bf(3.0 + rng.standard_normal(C * H))
    raw, n = _const_stream_setup(C, H, s, g)
    picks = [3, 9, 22, 31]
    wi = np.zeros((C, C * H))
    for c, j in enumerate(picks):
        wi[c, j] = 1.0
    r = orc.hc_call(raw, g, _w(np.zeros((L, C * H))), _w(np.zeros((C * H, L))), _w(wi),
                    H=H, C=C, L=L, eps=EPS)
    _close(r["gate"][0], 2.0 * expit(n[picks] / C), what="gate = 2 sigmoid(q / C)")


def pin_up_one_hot_no_div(orc):
    """Wu[j] = e_{k_j} => w_j = sigmoid(a_{k_j}) (no /C on the up path); with
    streams 1.. zero, mixed[h] = w[h] * n[h] / C (the mean over C)."""
    C, H, L = 4, 6, 3
    s = [2.5, 0.0, 0.0, 0.0]
    rng = np.random.default_rng(9)
    g = _bf(2.0 + rng.standard_normal(C * H))
    raw, n = _const_stream_setup(C, H, s, g)
    n[H:] = 0.0
    picks = [0, 2, 5]
    wd = np.zeros((L, C * H))
    for k, j in enumerate(picks):
        wd[k, j] = 1.0
    ks = np.arange(C * H) % L
    wu = np.zeros((C * H, L))
    wu[np.arange(C * H), ks] = 1.0
    r = orc.hc_call(raw, g, _w(wd), _w(wu), None, H=H, C=C, L=L, eps=EPS, want_w=True)
    a = _silu(n[picks] / C)
    w = expit(a[ks])
    _close(r["w"][0], w, what="w = sigmoid(up(a))")
    _close(r["mixed"][0], w[:H] * n[:H] / C, what="mixed from one live stream")


def pin_inject_add_trap_and_layout(orc):
    """The inject lands on the UN-normalised raw, stream-major: raw'[c*H+h] =
    raw[c*H+h] + out[h] * gate[c] (families/qwen4/mod.rs, the injection trap)."""
    rng = np.random.default_rng(13)
    M, C, H, L = 2, 3, 5, 2
    raw = _randn(rng, M, C * H, std=40.0)
    out = _randn(rng, M, H)
    g = _bf(1.0 + 0.1 * rng.standard_normal(C * H))
    wi = np.zeros((C, C * H))
    wi[0, 1], wi[1, 7], wi[2, 12] = 1.0, -2.0, 0.5
    zeros_d, zeros_u = _w(np.zeros((L, C * H))), _w(np.zeros((C * H, L)))
    buf = np.full(M * 2 * C, np.nan)
    r = orc.hc_call(raw, g, zeros_d, zeros_u, _w(wi), H=H, C=C, L=L, eps=EPS,
                    gate=buf, gate_stride=2 * C)
    gates = buf.reshape(M, 2, C)[:, 0, :]
    assert not np.any(np.isnan(gates)) and np.all(np.isnan(buf.reshape(M, 2, C)[:, 1, :]))
    res = orc.inject_add(raw, out, buf, H=H, C=C, gate_stride=2 * C)
    raw64, out64 = raw.double().numpy(), out.double().numpy()
    for m in range(M):
        _close(res[m] - raw64[m], np.outer(gates[m], out64[m]).reshape(-1), rtol=1e-12,
               atol=1e-12, what="inject-add outer product, stream-major")
    r0 = orc.hc_call(raw, g, zeros_d, zeros_u, _w(np.zeros((C, C * H))), H=H, C=C, L=L, eps=EPS)
    _close(r0["gate"], np.ones((M, C)), what="gate with zero inject weight")
    res0 = orc.inject_add(raw, out, r0["gate"], H=H, C=C)
    _close(res0, raw64 + np.tile(out64, (1, C)), rtol=0, atol=0, what="plain residual add")


def pin_scale_invariance(orc):
    """With eps = 0 the call sees raw only through raw / rms(raw)."""
    rng = np.random.default_rng(17)
    M, C, H, L = 2, 4, 8, 3
    raw = _randn(rng, M, C * H)
    g = _bf(1.0 + 0.1 * rng.standard_normal(C * H))
    wd, wu, wi = _w(_randn(rng, L, C * H)), _w(_randn(rng, C * H, L)), _w(_randn(rng, C, C * H))
    r1 = orc.hc_call(raw, g, wd, wu, wi, H=H, C=C, L=L, eps=0.0)
    r2 = orc.hc_call(raw.double() * 4.0, g, wd, wu, wi, H=H, C=C, L=L, eps=0.0)
    for k in ("mixed", "gate", "a"):
        _close(r2[k], r1[k], rtol=1e-13, atol=1e-15, what=f"scale invariance of {k}")
    _close(r2["inv_rms"], r1["inv_rms"] / 4.0, rtol=1e-14, what="inv_rms scales as 1/alpha")


def pin_stream_permutation(orc):
    rng = np.random.default_rng(19)
    M, C, H, L = 2, 4, 6, 3
    W = C * H
    raw = _randn(rng, M, W)
    g = _bf(1.0 + 0.1 * rng.standard_normal(W))
    wd, wu, wi = _randn(rng, L, W), _randn(rng, W, L), _randn(rng, C, W)
    perm = [2, 0, 3, 1]
    idx = torch.from_numpy(np.concatenate([np.arange(p * H, (p + 1) * H) for p in perm]))
    r1 = orc.hc_call(raw, g, _w(wd), _w(wu), _w(wi), H=H, C=C, L=L, eps=EPS)
    r2 = orc.hc_call(raw[:, idx], g[idx], _w(wd[:, idx]), _w(wu[idx, :]), _w(wi[perm][:, idx]),
                     H=H, C=C, L=L, eps=EPS)
    _close(r2["mixed"], r1["mixed"], rtol=1e-12, atol=1e-15, what="mixed under stream permutation")
    _close(r2["a"], r1["a"], rtol=1e-12, atol=1e-15, what="a under stream permutation")
    _close(r2["gate"], r1["gate"][:, perm], rtol=1e-12, what="gates permute with streams")
    _close(r2["inv_rms"], r1["inv_rms"][:, perm], rtol=1e-14, what="inv_rms permutes")


def pin_mixer_equals_call(orc):
    rng = np.random.default_rng(23)
    M, C, H, L = 2, 4, 8, 3
    raw = _randn(rng, M, C * H)
    g = _bf(1.0 + 0.1 * rng.standard_normal(C * H))
    wd, wu, wi = _w(_randn(rng, L, C * H)), _w(_randn(rng, C * H, L)), _w(_randn(rng, C, C * H))
    call = orc.hc_call(raw, g, wd, wu, wi, H=H, C=C, L=L, eps=EPS)
    mix = orc.mixer(raw, g, wd, wu, H=H, C=C, L=L, eps=EPS)
    assert "gate" not in mix
    for k in ("mixed", "inv_rms", "a"):
        assert np.array_equal(mix[k], call[k]), f"mixer {k} differs from the call's"


def pin_token_independence(orc):
    rng = np.random.default_rng(29)
    M, C, H, L = 3, 2, 8, 3
    raw = _randn(rng, M, C * H)
    g = _bf(1.0 + 0.1 * rng.standard_normal(C * H))
    wd, wu, wi = _w(_randn(rng, L, C * H)), _w(_randn(rng, C * H, L)), _w(_randn(rng, C, C * H))
    full = orc.hc_call(raw, g, wd, wu, wi, H=H, C=C, L=L, eps=EPS)
    for m in range(M):
        one = orc.hc_call(raw[m:m + 1], g, wd, wu, wi, H=H, C=C, L=L, eps=EPS)
        for k in ("mixed", "gate", "inv_rms", "a"):
            assert np.array_equal(one[k][0], full[k][m]), f"token {m} {k}"


def _library_call(raw, g, wd, wu, wi, C, H, L, eps):
    """The call written with torch fp64 library routines."""
    M = raw.shape[0]
    x = raw.view(M, C, H)
    n = torch.stack([F.rms_norm(x[:, c], (H,), eps=eps) for c in range(C)], dim=1) * g.view(C, H)
    nf = n.reshape(M, C * H)
    a = F.silu(F.linear(nf, wd) / C)
    w = torch.sigmoid(F.linear(a, wu))
    mixed = (w.view(M, C, H) * n).mean(dim=1)
    gate = 2.0 * torch.sigmoid(F.linear(nf, wi) / C)
    return mixed.numpy(), gate.numpy(), a.numpy()


def pin_library_formulation(orc):
    rng = np.random.default_rng(31)
    for C in (1, 2, 4):
        for H in (1, 2, 8):
            for L in (1, 3):
                M = 2
                raw = _randn(rng, M, C * H)
                g = _bf(1.0 + 0.2 * rng.standard_normal(C * H))
                wd, wu, wi = _randn(rng, L, C * H), _randn(rng, C * H, L), _randn(rng, C, C * H)
                r = orc.hc_call(raw, g, _w(wd), _w(wu), _w(wi), H=H, C=C, L=L, eps=EPS)
                mixed, gate, a = _library_call(raw.double(), g.double(), wd.double(), wu.double(),
                                               wi.double(), C, H, L, EPS)
                tag = f"C={C} H={H} L={L}"
                _close(r["mixed"], mixed, atol=1e-13, what=f"mixed {tag}")
                _close(r["gate"], gate, atol=1e-13, what=f"gate {tag}")
                _close(r["a"], a, atol=1e-13, what=f"a {tag}")


def pin_int4_library_formulation(orc):
    rng = np.random.default_rng(37)
    M, C, H, L = 2, 2, 64, 64
    raw = _randn(rng, M, C * H)
    g = _bf(1.0 + 0.2 * rng.standard_normal(C * H))
    mats = [_randn(rng, L, C * H, std=0.3), _randn(rng, C * H, L, std=0.3),
            _randn(rng, C, C * H, std=0.3)]
    q = [quantize_int4_affine(m, 32) for m in mats]

    def dense(w):  # the format's definition, from the packed bytes
        p = w.data.to(torch.int64)
        nib = torch.stack([p & 0xF, p >> 4], dim=2).reshape(w.rows, w.cols).double()
        s = w.scale.double().repeat_interleave(w.group, dim=1)
        b = w.bias.double().repeat_interleave(w.group, dim=1)
        return nib * s + b

    r = orc.hc_call(raw, g, q[0], q[1], q[2], H=H, C=C, L=L, eps=EPS)
    mixed, gate, a = _library_call(raw.double(), g.double(), *[dense(w) for w in q], C, H, L, EPS)
    _close(r["mixed"], mixed, atol=1e-13, what="int4 mixed")
    _close(r["gate"], gate, atol=1e-13, what="int4 gate")
    _close(r["a"], a, atol=1e-13, what="int4 a")


# --------------------------------------------------------------- drivers

class _Mod:
    def __init__(self, g, down, up, inject):
        self.g, self.down, self.up, self.inject = g, down, up, inject


def pin_entry_replication(orc):
    rng = np.random.default_rng(41)
    emb = _randn(rng, 2, 5)
    raw = orc.replicate_entry(emb, H=5, C=3)
    assert np.array_equal(raw, np.tile(emb.double().numpy(), (1, 3))), "repeat, not pad"


def pin_prefill_gate_slots(orc):
    """Inside a micro-batch token t's attn_hc gates sit at t*C*2, its mlp_hc
    gates at t*C*2 + C; every slot is written once and none is clobbered."""
    rng = np.random.default_rng(43)
    M, C, H, L = 3, 2, 4, 2
    W = C * H

    def mod():
        return _Mod(_bf(1.0 + 0.2 * rng.standard_normal(W)), _w(_randn(rng, L, W)),
                    _w(_randn(rng, W, L)), _w(_randn(rng, C, W)))

    attn, mlp = mod(), mod()
    raw = _randn(rng, M, W)
    oa, om = _randn(rng, M, H), _randn(rng, M, H)
    r = orc.prefill_pair(raw, attn, oa, mlp, om, H=H, C=C, L=L, eps=EPS)
    assert not np.any(np.isnan(r["gates"])), "a gate slot was never written"
    for t in range(M):
        a1 = orc.hc_call(raw[t:t + 1], attn.g, attn.down, attn.up, attn.inject, H=H, C=C, L=L)
        raw_t = orc.inject_add(raw[t:t + 1], oa[t:t + 1], a1["gate"], H=H, C=C)
        m1 = orc.hc_call(raw_t, mlp.g, mlp.down, mlp.up, mlp.inject, H=H, C=C, L=L)
        assert np.array_equal(r["gates"][t, 0], a1["gate"][0]), f"token {t} attn gate slot"
        assert np.array_equal(r["gates"][t, 1], m1["gate"][0]), f"token {t} mlp gate slot"


def pin_stack_closed_form(orc):
    """All down and inject weights zero => every gate is 1 and every w is 0.5:
    the residual is emb plus every sublayer output (stored in bf16 after each
    add), the same in all C streams, and the exit mixer gives
    0.5 * rms_norm(stream) * mean_c g_c."""
    rng = np.random.default_rng(47)
    M, C, H, L, n_layers = 2, 3, 8, 2, 2
    W = C * H

    def mod(with_inject=True):
        return _Mod(_bf(1.0 + 0.2 * rng.standard_normal(W)), _w(np.zeros((L, W))),
                    _w(_randn(rng, W, L)), _w(np.zeros((C, W))) if with_inject else None)

    emb = _randn(rng, M, H)
    layers = [(mod(), mod()) for _ in range(n_layers)]
    outs = [(_randn(rng, M, H), _randn(rng, M, H)) for _ in range(n_layers)]
    final = mod(with_inject=False)
    r = orc.stack(emb, layers, outs, final, H=H, C=C, L=L, eps=EPS, round_residual=True)
    x = emb.float()
    for oa, om in outs:
        for o in (oa, om):
            s32 = x + o.float()
            assert torch.equal(s32.double(), x.double() + o.double()), "fixture needs exact fp32 sums"
            x = s32.to(torch.bfloat16).float()
    x = x.double()
    _close(r["raw"], np.tile(x.numpy(), (1, C)), rtol=0, atol=0, what="stack residual")
    gbar = final.g.double().view(C, H).mean(dim=0)
    _close(r["mixed"], 0.5 * F.rms_norm(x, (H,), weight=gbar, eps=EPS).numpy(),
           what="stack exit mixer")


def pin_lm_head(orc):
    """logits = lm_head(mixed): one-hot rows read single elements of mixed, and a
    random weight agrees with numpy's matmul."""
    rng = np.random.default_rng(11)
    H, V = 16, 7
    mixed = _randn(rng, 3, H).double().numpy()
    one_hot = torch.zeros((V, H))
    cols = [(5 * v + 2) % H for v in range(V)]
    one_hot[torch.arange(V), torch.tensor(cols)] = 1.0
    got = orc.lm_head(mixed, one_hot.to(torch.bfloat16))
    assert np.array_equal(got, mixed[:, cols]), "one-hot lm_head rows"
    w = _randn(rng, V, H, std=0.3)
    _close(orc.lm_head(mixed, w), mixed @ w.double().numpy().T, what="lm_head vs numpy")


def _ple_case(rng, M=11, H=16, C=2, n_rows=20, key_std=0.3):
    W = C * H
    return dict(hidden=_randn(rng, M, W), rows=torch.as_tensor(rng.integers(0, n_rows, (M, 16)), dtype=torch.int32),
                table=_randn(rng, n_rows, H // 16), key_proj=_randn(rng, W, H, std=key_std),
                value_proj=_randn(rng, H, H, std=0.3), norm_key=_bf(1 + 0.1 * rng.standard_normal(W)),
                norm_query=_bf(1 + 0.1 * rng.standard_normal(W)), norm_conv=_bf(1 + 0.1 * rng.standard_normal(W)),
                conv_w=_randn(rng, W, 4, std=0.5), state=torch.as_tensor(rng.standard_normal((9, W))), H=H, C=C)


def _ple_torch(hidden, rows, table, key_proj, value_proj, norm_key, norm_query, norm_conv, conv_w, state, H, C):
    """The PLE in torch fp64 library calls: indexing for the table rows, F.linear,
    F.rms_norm per stream, F.conv1d (dilation 3, one group per channel) over the
    state followed by the chunk."""
    d = lambda t: torch.as_tensor(t).double()
    M, W = hidden.shape
    hid = d(hidden)
    emb = d(table)[rows.long()].reshape(M, H)
    gnorm = lambda x, s: (F.rms_norm(x.view(-1, C, H), (H,), eps=EPS) * d(s).view(C, H)).reshape(-1, W)
    key = gnorm(F.linear(emb, d(key_proj)), norm_key).view(M, C, H)
    value = F.linear(emb, d(value_proj))
    query = gnorm(hid, norm_query).view(M, C, H)
    g = (key * query).sum(-1) / math.sqrt(H)
    gate = torch.sigmoid(torch.sign(g) * torch.sqrt(torch.clamp(g.abs(), min=1e-6)))
    gv = (gate.unsqueeze(-1) * value.unsqueeze(1)).reshape(M, W)
    x = gnorm(gv, norm_conv)
    seq = torch.cat([d(state), x], dim=0).t().unsqueeze(0)          # [1, W, 9 + M]
    y = F.conv1d(seq, d(conv_w).unsqueeze(1), dilation=3, groups=W)  # [1, W, M]
    out = gv + F.silu(y[0].t())
    return {"result": hid + out, "gate": gate, "x": x, "state": torch.cat([d(state), x])[-9:],
            "value": value, "key": key.reshape(M, W)}


def pin_ple_library_formulation(orc):
    rng = np.random.default_rng(21)
    for key_std in (0.3, 1e-9):  # the second keeps |gate| below the 1e-6 floor of the signed root
        case = _ple_case(rng, key_std=key_std)
        got = orc.ple(**case)
        want = _ple_torch(**case)
        for k in ("result", "gate", "x", "state", "value", "key"):
            _close(got[k], want[k].numpy(), rtol=1e-11, atol=1e-13, what=f"PLE {k} (key std {key_std})")


def pin_ple_zero_key_gives_half_gate(orc):
    """A zero key projection: the normed key is zero, the gate's dot is zero, the
    signed root of zero is zero and the gate is sigmoid(0) = 1/2 exactly; gv is
    value / 2 in every stream."""
    rng = np.random.default_rng(22)
    case = _ple_case(rng)
    case["key_proj"] = torch.zeros_like(case["key_proj"])
    got = orc.ple(**case)
    assert np.all(got["gate"] == 0.5), "zero key: gate = sigmoid(0)"
    H, C = case["H"], case["C"]
    value = got["value"]
    gv = np.repeat(0.5 * value[:, None, :], C, axis=1).reshape(-1, C * H)
    d = torch.as_tensor(gv)
    x = (F.rms_norm(d.view(-1, C, H), (H,), eps=EPS) * case["norm_conv"].double().view(C, H)).reshape(-1, C * H)
    _close(got["x"], x.numpy(), rtol=1e-12, atol=1e-14, what="zero key: conv input = norm_conv(value / 2)")


def pin_ple_state_carries_across_chunks(orc):
    """Tokens are one sequence: a chunk of 11 equals chunks of 4 and 7 with the
    conv state handed over."""
    rng = np.random.default_rng(23)
    case = _ple_case(rng)
    whole = orc.ple(**case)
    a = dict(case, hidden=case["hidden"][:4], rows=case["rows"][:4])
    ra = orc.ple(**a)
    b = dict(case, hidden=case["hidden"][4:], rows=case["rows"][4:], state=ra["state"])
    rb = orc.ple(**b)
    assert np.array_equal(np.concatenate([ra["result"], rb["result"]]), whole["result"])
    assert np.array_equal(rb["state"], whole["state"])


def pin_stack_ple_zero_value_adds_nothing(orc):
    """The stack with the PLE before layer 1: a PLE whose value projection and conv
    state are zero adds exactly nothing (gv = 0, every conv input and tap product is
    0, silu(0) = 0), so the stack equals the stack without it, bit for bit; with a
    non-zero value projection the stack's output changes, and the state the stack
    hands back is the PLE's own on the residual after layer 0."""
    H, C, L, M = 32, 2, 8, 3
    st = inputs.make_stack(M, H, C, L, 3, 31)
    pw = inputs.make_ple_weights(H, C, 31, n_rows=12, std=0.3)
    rows = inputs.make_ple_rows(M, 12, 31)
    zero_state = torch.zeros((9, C * H), dtype=torch.float64)
    plain = orc.stack(st.emb, st.layers, st.outs, st.final, H=H, C=C, L=L, eps=EPS)
    quiet = inputs.PleWeights(pw.table, pw.key_proj, torch.zeros_like(pw.value_proj), pw.norm_key, pw.norm_query,
                              pw.norm_conv, pw.conv_w)
    with_quiet = orc.stack(st.emb, st.layers, st.outs, st.final, H=H, C=C, L=L, eps=EPS, ple=quiet,
                           ple_rows=rows, ple_state=zero_state)
    assert np.array_equal(with_quiet["mixed"], plain["mixed"]) and np.array_equal(with_quiet["raw"], plain["raw"])
    assert not np.any(with_quiet["ple_state"]), "a zero value projection leaves a zero conv state"
    live = orc.stack(st.emb, st.layers, st.outs, st.final, H=H, C=C, L=L, eps=EPS, ple=pw, ple_rows=rows,
                     ple_state=zero_state)
    assert not np.allclose(live["mixed"], plain["mixed"], rtol=1e-6, atol=0), "the PLE changes the stack"
    after0 = orc.prefill_pair(orc.replicate_entry(st.emb, H=H, C=C), st.layers[0][0], st.outs[0][0],
                              st.layers[0][1], st.outs[0][1], H=H, C=C, L=L, eps=EPS, round_residual=True)
    own = orc.ple(after0["raw_after_mlp"], rows, pw.table, pw.key_proj, pw.value_proj, pw.norm_key, pw.norm_query,
                  pw.norm_conv, pw.conv_w, zero_state, H=H, C=C, eps=EPS)
    assert np.array_equal(live["ple_state"], own["state"]), "the PLE runs on the residual after layer 0"


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
