"""Host-side checks of the C ABI: the library loads, exports every entry point
the header declares, and rejects bad arguments before launching anything.

Every call here fails argument validation (or is an M = 0 no-op), so no CUDA
call is made: these run on a machine without a GPU.
"""
import ctypes
import os
import re

import pytest

from hyper_connection_residual_call_gb300 import binding as B
from hyper_connection_residual_call_gb300.build import INCLUDE, build

H, C, L = 2560, 4, 320
FAKE = 0x10000  # an aligned address that is never dereferenced: validation fails first


@pytest.fixture(scope="module")
def lib():
    build()
    return B.library()


def declared_symbols():
    text = open(os.path.join(INCLUDE, "ts_hc.h")).read()
    return sorted(set(re.findall(r"\b(ts_hc_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert set(names) == set(B.EXPORTS), names
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"


def test_workspace_size_and_layout(lib):
    a256 = lambda n: (n + 255) // 256 * 256
    # one token: inv_rms, act, and 8 copies of up to 8 chunks of per-row partials and of
    # the chunks' sums of squares (64-float stride)
    assert B.ts_hc_workspace_bytes(1, H, C, L) == 256 + 1280 + 8 * a256(4 * 8 * (L + C)) + 8 * 4 * 64
    # from 2 tokens the tensor-core path adds normed as bf16 hi + lo [M][C*H] x 2, the
    # down kernel's per-chunk partials [nchunk][L+C][Mp] fp32 and the activations as
    # bf16 hi + lo [M][L] x 2. The K split aims at 152 CTAs: at M=128 (one 128-token
    # tile, 3 row tiles) 160 K blocks of 64 go 4 to a chunk, 40 chunks.
    # At 2 and 3 tokens the few-token kernels' partials come first: 8 copies of up to 8
    # chunks x M tokens of per-row partials, and of the sums of squares.
    for M, nchunk, Mp in ((128, 40, 128), (2, 40, 16), (15, 40, 16), (16, 40, 16), (40, 40, 48),
                          (300, 16, 384), (8, 40, 16), (3, 40, 16)):
        tc = 2 * a256(2 * M * C * H) + a256(4 * nchunk * (L + C) * Mp) + 2 * a256(2 * M * L)
        few = 8 * a256(4 * 8 * M * (L + C)) + 8 * 4 * 64 if M <= 3 else 0
        assert B.ts_hc_workspace_bytes(M, H, C, L) == a256(4 * M * C) + a256(4 * M * L) + few + tc, M
    # shapes the tensor-core path does not take (lowrank not a multiple of 64): inv_rms, act
    assert B.ts_hc_workspace_bytes(15, H, C, 32) == a256(4 * 15 * C) + a256(4 * 15 * 32)
    assert B.ts_hc_workspace_bytes(2, H, C, 32) == (a256(4 * 2 * C) + a256(4 * 2 * 32)
                                                    + 8 * a256(4 * 8 * 2 * (32 + C)) + 8 * 4 * 64)
    assert B.ts_hc_workspace_bytes(0, H, C, L) == 0
    assert B.ts_hc_workspace_bytes(-1, H, C, L) == 0
    inv, act = B.ts_hc_workspace_layout(3, H, C, L)
    assert inv == 0 and act == 256 and act % 256 == 0


def _w(data=FAKE, typ=B.TS_W_BF16, group=0, scales=None, biases=None):
    return B.TsWeight(typ, group, data, scales, biases)


def _call(**kw):
    a = dict(raw=FAKE, g=FAKE, down=_w(), up=_w(), inject=_w(), mixed=FAKE, inject_w=FAKE, stride=C,
             M=1, H=H, C=C, L=L, eps=1e-6, ws=FAKE, ws_bytes=1 << 20, stream=None)
    a.update(kw)
    return B.ts_hc_call(a["raw"], a["g"], a["down"], a["up"], a["inject"], a["mixed"], a["inject_w"],
                        a["stride"], a["M"], a["H"], a["C"], a["L"], a["eps"], a["ws"], a["ws_bytes"],
                        a["stream"])


@pytest.mark.parametrize("kw,status,needle", [
    (dict(raw=None), B.TS_ERR_INVALID_ARG, "raw is NULL"),
    (dict(raw=FAKE + 2), B.TS_ERR_INVALID_ARG, "raw is not 16-byte aligned"),
    (dict(mixed=None), B.TS_ERR_INVALID_ARG, "mixed is NULL"),
    (dict(g=FAKE + 8), B.TS_ERR_INVALID_ARG, "hc_norm_w"),
    (dict(H=2561), B.TS_ERR_INVALID_ARG, "H = 2561"),
    (dict(C=0), B.TS_ERR_INVALID_ARG, "C = 0"),
    (dict(C=9), B.TS_ERR_INVALID_ARG, "C = 9"),
    (dict(L=4), B.TS_ERR_INVALID_ARG, "lowrank = 4"),
    (dict(M=-1), B.TS_ERR_INVALID_ARG, "M = -1"),
    (dict(stride=C - 1), B.TS_ERR_INVALID_ARG, "inject_stride"),
    (dict(inject=None), B.TS_ERR_INVALID_ARG, "ts_hc_mixer"),
    (dict(inject_w=None), B.TS_ERR_INVALID_ARG, "inject_w is NULL"),
    (dict(down=_w(data=None)), B.TS_ERR_INVALID_ARG, "down.data"),
    (dict(up=_w(typ=7)), B.TS_ERR_INVALID_ARG, "up.type"),
    (dict(down=_w(typ=B.TS_W_INT4_AFFINE, group=48, scales=FAKE, biases=FAKE)), B.TS_ERR_UNSUPPORTED, "group = 48"),
    (dict(up=_w(typ=B.TS_W_INT4_AFFINE, group=64, scales=None, biases=FAKE)), B.TS_ERR_INVALID_ARG, "scales"),
    (dict(inject=_w(typ=B.TS_W_INT4_AFFINE, group=64, scales=FAKE, biases=FAKE)), B.TS_ERR_UNSUPPORTED,
     "same storage format"),
    (dict(down=_w(typ=B.TS_W_INT4_AFFINE, group=16, scales=FAKE, biases=FAKE)), B.TS_ERR_UNSUPPORTED, "group = 16"),
    (dict(up=_w(typ=B.TS_W_INT4_AFFINE, group=256, scales=FAKE, biases=FAKE)), B.TS_ERR_UNSUPPORTED, "group = 256"),
    (dict(up=_w(typ=B.TS_W_INT4_AFFINE, group=128, scales=FAKE, biases=FAKE)), B.TS_ERR_UNSUPPORTED,
     "320 inputs are not a multiple of the group 128"),
    (dict(down=_w(typ=B.TS_W_INT4_AFFINE, group=64, scales=FAKE, biases=FAKE),
          inject=_w(typ=B.TS_W_INT4_AFFINE, group=32, scales=FAKE, biases=FAKE)), B.TS_ERR_UNSUPPORTED,
     "same storage format and group"),
    (dict(down=_w(typ=B.TS_W_INT4_AFFINE, group=64, scales=FAKE, biases=None)), B.TS_ERR_INVALID_ARG, "biases"),
    (dict(eps=-1.0), B.TS_ERR_INVALID_ARG, "eps"),
    (dict(ws_bytes=16), B.TS_ERR_WORKSPACE, "workspace of 16 bytes"),
    (dict(ws=None), B.TS_ERR_WORKSPACE, "workspace"),
    (dict(ws=FAKE + 16), B.TS_ERR_INVALID_ARG, "256-byte aligned"),
])
def test_call_rejects(lib, kw, status, needle):
    assert _call(**kw) == status
    assert needle in B.ts_hc_last_error()


def test_call_m0_is_noop(lib):
    assert _call(M=0, ws=None, ws_bytes=0) == B.TS_OK
    assert B.ts_hc_last_error() == ""


def test_call_debug_rejects_a_missing_w_buffer(lib):
    args = [FAKE, FAKE, _w(), _w(), _w(), FAKE, FAKE, C, 1, H, C, L, 1e-6, FAKE, 1 << 30]
    assert B.ts_hc_call_debug(*args, None, None) == B.TS_ERR_INVALID_ARG
    assert "w_out is NULL" in B.ts_hc_last_error()
    assert B.ts_hc_call_debug(*args, FAKE + 2, None) == B.TS_ERR_INVALID_ARG
    assert "w_out is not 4-byte aligned" in B.ts_hc_last_error()
    # the rest of the call's validation still applies
    bad = list(args)
    bad[0] = None
    assert B.ts_hc_call_debug(*bad, FAKE, None) == B.TS_ERR_INVALID_ARG
    assert "raw is NULL" in B.ts_hc_last_error()
    # M == 0: a no-op that examines no pointer
    zero = list(args)
    zero[8] = 0
    assert B.ts_hc_call_debug(*zero, None, None) == B.TS_OK


def test_entry_call_rejects(lib):
    args = dict(emb=FAKE, raw=FAKE + (1 << 20), M=2)

    def call(emb, raw, M, inject=_w()):
        return B.ts_hc_entry_call(emb, raw, FAKE, _w(), _w(), inject, FAKE, FAKE, C, M, H, C, L, 1e-6, FAKE, 1 << 30,
                                  None)

    assert call(**{**args, "emb": None}) == B.TS_ERR_INVALID_ARG and "emb is NULL" in B.ts_hc_last_error()
    assert call(**{**args, "raw": FAKE + 8}) == B.TS_ERR_INVALID_ARG and "not 16-byte aligned" in B.ts_hc_last_error()
    # the replicated residual must not overwrite the embedding rows it is built from
    assert call(**{**args, "raw": FAKE + 2 * H}) == B.TS_ERR_INVALID_ARG
    assert "raw overlaps emb" in B.ts_hc_last_error()
    assert call(**{**args, "M": 0, "emb": None, "raw": None}) == B.TS_OK


def test_exit_logits_rejects(lib):
    def call(lm_head=FAKE, V=1000, logits=FAKE, out=None, prev=None, prev_stride=C, M=1, H_=H):
        return B.ts_hc_exit_logits(FAKE, out, prev, prev_stride, FAKE, _w(), _w(), lm_head, V, FAKE, logits, M, H_,
                                   C, L, 1e-6, FAKE, 1 << 30, None)

    assert call(V=0) == B.TS_ERR_INVALID_ARG and "V = 0" in B.ts_hc_last_error()
    assert call(lm_head=None) == B.TS_ERR_INVALID_ARG and "lm_head is NULL" in B.ts_hc_last_error()
    assert call(lm_head=FAKE + 8) == B.TS_ERR_INVALID_ARG and "lm_head is not 16-byte" in B.ts_hc_last_error()
    assert call(logits=FAKE + 2) == B.TS_ERR_INVALID_ARG and "logits is not 4-byte" in B.ts_hc_last_error()
    assert call(out=FAKE, prev=None) == B.TS_ERR_INVALID_ARG and "prev_inject_w is NULL" in B.ts_hc_last_error()
    assert call(out=FAKE, prev=FAKE, prev_stride=C - 1) == B.TS_ERR_INVALID_ARG
    assert call(H_=H + 8) == B.TS_ERR_UNSUPPORTED and "multiple of 64" in B.ts_hc_last_error()
    assert call(M=0, lm_head=None, logits=None) == B.TS_OK


def test_ple_workspace_and_rejects(lib):
    a256 = lambda n: (n + 255) // 256 * 256
    M, W = 3, C * H
    assert B.ts_hc_ple_workspace_bytes(M, H, C) == (a256(2 * M * H) + a256(4 * M * W) + a256(4 * M * H)
                                                   + a256(4 * M * C) + a256(4 * M * W))
    assert B.ts_hc_ple_workspace_bytes(M, 200, C) == 0  # H not a multiple of 128

    def call(hidden=FAKE, rows=FAKE, n_rows=100, H_=H, M_=1, ws_bytes=1 << 30, conv_state=FAKE):
        return B.ts_hc_ple(hidden, rows, FAKE, n_rows, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, conv_state, M_, H_, C,
                           1e-6, FAKE, ws_bytes, None)

    assert call(H_=200) == B.TS_ERR_INVALID_ARG and "multiple of 128" in B.ts_hc_last_error()
    assert call(hidden=None) == B.TS_ERR_INVALID_ARG and "hidden is NULL" in B.ts_hc_last_error()
    assert call(rows=FAKE + 2) == B.TS_ERR_INVALID_ARG and "rows is not 4-byte" in B.ts_hc_last_error()
    assert call(n_rows=0) == B.TS_ERR_INVALID_ARG and "n_rows" in B.ts_hc_last_error()
    assert call(conv_state=FAKE + 4) == B.TS_ERR_INVALID_ARG and "conv_state" in B.ts_hc_last_error()
    assert call(ws_bytes=16) == B.TS_ERR_WORKSPACE
    assert call(M_=0, hidden=None, rows=None) == B.TS_OK


def test_mixer_rejects(lib):
    st = B.ts_hc_mixer(None, FAKE, _w(), _w(), FAKE, 1, H, C, L, 1e-6, FAKE, 1 << 20, None)
    assert st == B.TS_ERR_INVALID_ARG and "raw is NULL" in B.ts_hc_last_error()
    st = B.ts_hc_mixer(FAKE, FAKE, _w(), _w(), FAKE, 0, H, C, L, 1e-6, None, 0, None)
    assert st == B.TS_OK


@pytest.mark.parametrize("args,needle", [
    ((None, FAKE, FAKE, C, 1, H, C), "raw is NULL"),
    ((FAKE, FAKE + 4, FAKE, C, 1, H, C), "out is not 16-byte aligned"),
    ((FAKE, FAKE, FAKE + 2, C, 1, H, C), "inject_w is not 4-byte aligned"),
    ((FAKE, FAKE, FAKE, C - 1, 1, H, C), "inject_stride"),
    ((FAKE, FAKE, FAKE, C, 1, 12, C), "H = 12"),
])
def test_inject_add_rejects(lib, args, needle):
    assert B.ts_hc_inject_add(*args, None) == B.TS_ERR_INVALID_ARG
    assert needle in B.ts_hc_last_error()


def test_inject_add_m0_is_noop(lib):
    assert B.ts_hc_inject_add(FAKE, FAKE, FAKE, C, 0, H, C, None) == B.TS_OK


def test_replicate_entry_rejects(lib):
    assert B.ts_hc_replicate_entry(None, FAKE, 1, H, C, None) == B.TS_ERR_INVALID_ARG
    assert "emb is NULL" in B.ts_hc_last_error()
    assert B.ts_hc_replicate_entry(FAKE, FAKE + 8, 1, H, C, None) == B.TS_ERR_INVALID_ARG
    assert B.ts_hc_replicate_entry(FAKE, FAKE, 0, H, C, None) == B.TS_OK


def _icall(**kw):
    a = dict(raw=FAKE, out=FAKE, prev=FAKE, prev_stride=C, g=FAKE, down=_w(), up=_w(), inject=_w(),
             mixed=FAKE, inject_w=FAKE + 4096, stride=C, M=1, H=H, C=C, L=L, eps=1e-6, ws=FAKE,
             ws_bytes=1 << 20, stream=None)
    a.update(kw)
    return B.ts_hc_inject_call(a["raw"], a["out"], a["prev"], a["prev_stride"], a["g"], a["down"], a["up"],
                               a["inject"], a["mixed"], a["inject_w"], a["stride"], a["M"], a["H"], a["C"],
                               a["L"], a["eps"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,status,needle", [
    (dict(out=None), B.TS_ERR_INVALID_ARG, "out is NULL"),
    (dict(out=FAKE + 8), B.TS_ERR_INVALID_ARG, "out is not 16-byte aligned"),
    (dict(prev=None), B.TS_ERR_INVALID_ARG, "prev_inject_w is NULL"),
    (dict(prev_stride=C - 1), B.TS_ERR_INVALID_ARG, "prev_inject_stride"),
    (dict(inject_w=FAKE), B.TS_ERR_INVALID_ARG, "shares elements"),                      # same slot
    (dict(inject_w=FAKE + 8, M=3), B.TS_ERR_INVALID_ARG, "shares elements"),             # partial overlap
    (dict(inject_w=FAKE + 4 * C, prev_stride=2 * C, stride=2 * C, M=5, ws_bytes=16),     # two slots: fine,
     B.TS_ERR_WORKSPACE, "workspace"),                                                   # fails later on ws
    (dict(raw=None), B.TS_ERR_INVALID_ARG, "raw is NULL"),
    (dict(ws_bytes=16), B.TS_ERR_WORKSPACE, "workspace"),
])
def test_inject_call_rejects(lib, kw, status, needle):
    assert _icall(**kw) == status
    assert needle in B.ts_hc_last_error()


def test_inject_call_m0_is_noop(lib):
    assert _icall(M=0, ws=None, ws_bytes=0) == B.TS_OK


def test_device_status_rejects_null(lib):
    assert lib.ts_hc_device_status(None, None) == B.TS_ERR_INVALID_ARG


def test_torch_layer_requires_cuda_tensors(lib):
    import torch
    from hyper_connection_residual_call_gb300 import inputs
    w = inputs.make_hc_weights(256, 4, 32, 0)
    raw = inputs.make_residual(1, 256, 4, 0)
    with pytest.raises(B.HCError, match="CUDA tensor"):
        B.hc_call(raw, w, H=256, C=4)
    with pytest.raises(B.HCError, match="CUDA tensor"):
        B.hc_inject_add(raw, torch.zeros(1, 256, dtype=torch.bfloat16), torch.ones(1, 4), H=256, C=4)


def _module(**kw):
    m = B.TsHcModule()
    m.hc_norm_w = kw.get("g", FAKE)
    m.down, m.up = kw.get("down", _w()), kw.get("up", _w())
    m.inject = kw.get("inject", _w())
    return m


def _stack(**kw):
    n = kw.get("n_layers", 2)
    attn = kw.get("attn", (B.TsHcModule * max(n, 1))(*[_module() for _ in range(n)]))
    mlp = kw.get("mlp", (B.TsHcModule * max(n, 1))(*[_module() for _ in range(n)]))
    final = kw.get("final", _module(inject=_w(data=None)))
    fn = kw.get("fn", B.SUBLAYER_FN(lambda *a: B.TS_OK))
    return B.ts_hc_stack(kw.get("emb", FAKE), kw.get("T", 5), attn, mlp, n, final, fn, None,
                         kw.get("mixed_out", FAKE), kw.get("max_chunk", 4), H, C, L, kw.get("eps", 1e-6),
                         kw.get("ws", FAKE), kw.get("ws_bytes", 1 << 30), None)


def _ple_module(**kw):
    m = B.TsHcPleModule()
    m.table, m.n_rows = kw.get("table", FAKE), kw.get("n_rows", 100)
    m.key_proj, m.value_proj = kw.get("key_proj", FAKE), kw.get("value_proj", FAKE)
    m.norm_key_w, m.norm_query_w, m.norm_conv_w = FAKE, kw.get("norm_query_w", FAKE), FAKE
    m.conv_w = kw.get("conv_w", FAKE)
    return m


def _stack_ple(**kw):
    n = kw.get("n_layers", 2)
    attn = (B.TsHcModule * max(n, 1))(*[_module() for _ in range(n)])
    mlp = (B.TsHcModule * max(n, 1))(*[_module() for _ in range(n)])
    ple = kw.get("ple", _ple_module())
    return B.ts_hc_stack_ple(FAKE, 5, attn, mlp, n, _module(inject=_w(data=None)), ple, kw.get("rows", FAKE),
                             kw.get("state", FAKE), B.SUBLAYER_FN(lambda *a: B.TS_OK), None, FAKE, 4,
                             kw.get("H_", H), C, L, 1e-6, FAKE, kw.get("ws_bytes", 1 << 30), None)


def test_stack_ple_workspace_bytes(lib):
    a256 = lambda n: (n + 255) // 256 * 256
    for chunk in (1, 7, 16):
        assert (B.ts_hc_stack_ple_workspace_bytes(chunk, H, C, L)
                == B.ts_hc_stack_workspace_bytes(chunk, H, C, L) + a256(B.ts_hc_ple_workspace_bytes(chunk, H, C)))
    assert B.ts_hc_stack_ple_workspace_bytes(4, 2560 + 64, C, L) == 0  # H not a multiple of 128


@pytest.mark.parametrize("kw,status,needle", [
    (dict(n_layers=1), B.TS_ERR_INVALID_ARG, "n_layers = 1"),
    (dict(ple=None), B.TS_ERR_INVALID_ARG, "ple is NULL"),
    (dict(ple=_ple_module(n_rows=0)), B.TS_ERR_INVALID_ARG, "n_rows"),
    (dict(ple=_ple_module(key_proj=FAKE + 8)), B.TS_ERR_INVALID_ARG, "key_proj is not 16-byte aligned"),
    (dict(ple=_ple_module(norm_query_w=None)), B.TS_ERR_INVALID_ARG, "norm_query_w is NULL"),
    (dict(rows=FAKE + 2), B.TS_ERR_INVALID_ARG, "ple_rows is not 4-byte aligned"),
    (dict(state=None), B.TS_ERR_INVALID_ARG, "ple_conv_state is NULL"),
    (dict(H_=2560 + 64), B.TS_ERR_INVALID_ARG, "multiple of 128"),
    (dict(ws_bytes=1 << 20), B.TS_ERR_WORKSPACE, "workspace"),
])
def test_stack_ple_rejects(lib, kw, status, needle):
    assert _stack_ple(**kw) == status
    assert needle in B.ts_hc_last_error()


def test_stack_workspace_bytes(lib):
    a256 = lambda n: (n + 255) // 256 * 256
    for chunk in (1, 7, 16, 40):
        calls = max(B.ts_hc_workspace_bytes(m, H, C, L) for m in range(1, chunk + 1))
        want = a256(2 * chunk * C * H) + a256(2 * chunk * H) + a256(4 * chunk * 2 * C) + a256(calls)
        assert B.ts_hc_stack_workspace_bytes(chunk, H, C, L) == want
    assert B.ts_hc_stack_workspace_bytes(0, H, C, L) == 0
    assert B.ts_hc_stack_workspace_bytes(4, H, 0, L) == 0


def test_stack_t0_is_noop(lib):
    assert _stack(T=0, emb=None, mixed_out=None, ws=None, ws_bytes=0) == B.TS_OK


@pytest.mark.parametrize("kw,status,needle", [
    (dict(T=-1), B.TS_ERR_INVALID_ARG, "T = -1"),
    (dict(max_chunk=0), B.TS_ERR_INVALID_ARG, "max_chunk"),
    (dict(emb=None), B.TS_ERR_INVALID_ARG, "emb is NULL"),
    (dict(mixed_out=FAKE + 2), B.TS_ERR_INVALID_ARG, "mixed_out is not 16-byte aligned"),
    (dict(fn=None), B.TS_ERR_INVALID_ARG, "sublayer is NULL"),
    (dict(attn=None), B.TS_ERR_INVALID_ARG, "attn is NULL"),
    (dict(mlp=(B.TsHcModule * 2)(_module(), _module(down=_w(data=FAKE + 8)))), B.TS_ERR_INVALID_ARG,
     "mlp[1].down.data"),
    (dict(attn=(B.TsHcModule * 2)(_module(), _module(inject=_w(data=None)))), B.TS_ERR_INVALID_ARG,
     "attn[1].inject.data"),
    (dict(attn=(B.TsHcModule * 2)(_module(g=None), _module())), B.TS_ERR_INVALID_ARG, "attn[0].hc_norm_w is NULL"),
    (dict(final=None), B.TS_ERR_INVALID_ARG, "final_mixer is NULL"),
    (dict(final=_module(up=_w(typ=7))), B.TS_ERR_INVALID_ARG, "final_mixer.up.type"),
    (dict(ws_bytes=1024), B.TS_ERR_WORKSPACE, "workspace"),
    (dict(ws=FAKE + 16), B.TS_ERR_INVALID_ARG, "256-byte aligned"),
    (dict(eps=-1.0), B.TS_ERR_INVALID_ARG, "eps"),
])
def test_stack_rejects(lib, kw, status, needle):
    calls = []
    kw.setdefault("fn", B.SUBLAYER_FN(lambda *a: calls.append(a) or B.TS_OK))
    assert _stack(**kw) == status
    assert needle in B.ts_hc_last_error()
    assert not calls, "the sublayer callback ran before validation finished"
