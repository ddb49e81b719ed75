"""fp64 CPU oracle for the hyper-connection residual call -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product path (the CUDA library and its Python
binding) never imports it, and it imports nothing from the product path.

The arithmetic lives in ``hc_oracle.c`` (plain double-precision loops); this
module only compiles it, marshals arrays into it and strings the calls together
the way the turbospark-runtime 0.3.0 pages describe:

* ``hc_call`` / ``mixer``: families/qwen4/mod.rs, module doc, "## Hyper-
  connections"; families/qwen4/hc.rs, ``encode_hyper_connection``.
* ``inject_add``: families/qwen4/mod.rs, decoder-layer pseudocode and
  "THE INJECTION TRAP".
* ``prefill_pair``: families/qwen4/hc.rs, the ``inject_row_offset`` paragraph
  (token t's gates at element t*C*2 of the gate buffer inside a micro-batch),
  and families/qwen4/mod.rs, "Chunked prefill is wired".
* ``stack``: families/qwen4/mod.rs decoder-layer pseudocode (entry
  replication, two calls and two inject-adds per layer, the exit mixer).
* ``lm_head``: the same pseudocode's exit line, logits = lm_head(mixer output).
* ``ple``: families/qwen4/mod.rs, "## PLE" (layer index 1 only), with the
  readings listed beside ``orc_ple`` in ``hc_oracle.c``.

Every function is pinned by ``tests/test_oracle_pins.py`` (closed forms,
invariants, library special cases); ``tests/test_oracle_mutants.py`` plants
plausible mistakes in a copy of the C source and checks that a pin fails.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "hc_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liborc_hc.so")

RMS_EPS = 1e-6  # families/qwen4/mod.rs, `RMS_EPS`


def compile_library(src: str, out: str) -> str:
    """gcc -> shared library. ``-ffp-contract=off`` keeps every multiply and add
    separately rounded, so x86_64 and aarch64 builds agree bit for bit."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``hc_oracle.c`` into ``_build/liborc_hc.so`` if it is missing or stale."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_library(SOURCE, _LIB_PATH)


class _OrcWeight(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32),
        ("group", ctypes.c_int32),
        ("rows", ctypes.c_int64),
        ("cols", ctypes.c_int64),
        ("bf16", ctypes.c_void_p),
        ("packed", ctypes.c_void_p),
        ("scale", ctypes.c_void_p),
        ("bias", ctypes.c_void_p),
    ]


_D = ctypes.POINTER(ctypes.c_double)


def default_threads() -> int:
    if hasattr(os, "sched_getaffinity"):
        return max(1, len(os.sched_getaffinity(0)))
    return max(1, os.cpu_count() or 1)


def _np_bits(t) -> np.ndarray:
    """A torch tensor (bf16/fp16 viewed as int16) or numpy array, C-contiguous."""
    if hasattr(t, "detach"):
        import torch  # only to reinterpret 16-bit float storage as raw bits
        t = t.detach().cpu().contiguous()
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.view(torch.int16)
        t = t.numpy()
    return np.ascontiguousarray(t)


def _f64(x) -> np.ndarray:
    """Values as float64. bf16 tensors are widened by torch, an exact conversion."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _dptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(_D)


@dataclass
class _Marshalled:
    struct: _OrcWeight
    keep: tuple


def _weight(w) -> Optional[_Marshalled]:
    """Marshal a weight given by attributes kind ('bf16' | 'int4'), rows, cols,
    data, scale, bias, group (as the seeded input generators make them)."""
    if w is None:
        return None
    s = _OrcWeight()
    s.rows, s.cols = int(w.rows), int(w.cols)
    if w.kind == "bf16":
        data = _np_bits(w.data).view(np.uint16)
        assert data.shape == (s.rows, s.cols)
        s.kind, s.group = 0, 0
        s.bf16 = data.ctypes.data
        keep = (data,)
    elif w.kind == "int4":
        packed = _np_bits(w.data).view(np.uint8)
        scale = _np_bits(w.scale).view(np.uint16)
        bias = _np_bits(w.bias).view(np.uint16)
        g = int(w.group)
        assert packed.shape == (s.rows, s.cols // 2) and s.cols % g == 0
        assert scale.shape == (s.rows, s.cols // g) and bias.shape == scale.shape
        s.kind, s.group = 1, g
        s.packed, s.scale, s.bias = packed.ctypes.data, scale.ctypes.data, bias.ctypes.data
        keep = (packed, scale, bias)
    else:
        raise ValueError(f"unknown weight kind {w.kind!r}")
    return _Marshalled(s, keep)


@dataclass
class _LinearBf16:
    """A bf16 [rows][cols] weight in the form ``_weight`` marshals."""
    rows: int
    cols: int
    data: object
    kind: str = "bf16"
    scale: object = None
    bias: object = None
    group: int = 0


def _wptr(m: Optional[_Marshalled]):
    return None if m is None else ctypes.byref(m.struct)


class Oracle:
    """The oracle bound to one compiled copy of ``hc_oracle.c``."""

    def __init__(self, lib_path: Optional[str] = None):
        lib = ctypes.CDLL(lib_path or build())
        lib.orc_bf16_value.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_value.restype = ctypes.c_double
        lib.orc_f16_value.argtypes = [ctypes.c_uint16]
        lib.orc_f16_value.restype = ctypes.c_double
        lib.orc_round_to_bf16.argtypes = [ctypes.c_double]
        lib.orc_round_to_bf16.restype = ctypes.c_double
        lib.orc_round_to_bf16_array.argtypes = [_D, _D, ctypes.c_int64]
        lib.orc_weight_at.argtypes = [ctypes.POINTER(_OrcWeight), ctypes.c_int64, ctypes.c_int64]
        lib.orc_weight_at.restype = ctypes.c_double
        lib.orc_gemv.argtypes = [ctypes.POINTER(_OrcWeight), _D, _D, ctypes.c_int]
        lib.orc_hc_call.argtypes = (
            [ctypes.c_int64] * 4 + [ctypes.c_double, _D, _D]
            + [ctypes.POINTER(_OrcWeight)] * 3
            + [_D, _D, ctypes.c_int64, _D, _D, _D, ctypes.c_int])
        lib.orc_hc_call.restype = ctypes.c_int
        lib.orc_inject_add.argtypes = [ctypes.c_int64] * 3 + [_D, _D, _D, ctypes.c_int64, _D]
        lib.orc_replicate_entry.argtypes = [ctypes.c_int64] * 3 + [_D, _D]
        lib.orc_ple.argtypes = ([ctypes.c_int64] * 3 + [ctypes.c_double, _D, ctypes.c_void_p, ctypes.c_void_p,
                                                        ctypes.c_int64, ctypes.POINTER(_OrcWeight),
                                                        ctypes.POINTER(_OrcWeight), _D, _D, _D, ctypes.c_void_p, _D,
                                                        _D, _D, _D, _D, _D, _D, ctypes.c_int])
        lib.orc_ple.restype = ctypes.c_int
        self.lib = lib

    # ------------------------------------------------------------ scalars

    def bf16_value(self, bits: int) -> float:
        return self.lib.orc_bf16_value(bits & 0xFFFF)

    def f16_value(self, bits: int) -> float:
        return self.lib.orc_f16_value(bits & 0xFFFF)

    def round_to_bf16(self, x) -> np.ndarray:
        x = _f64(x)
        y = np.empty_like(x)
        self.lib.orc_round_to_bf16_array(_dptr(x.reshape(-1)), _dptr(y.reshape(-1)), x.size)
        return y

    def weight_values(self, w) -> np.ndarray:
        """Every element of a weight as float64, through the oracle's decoder."""
        m = _weight(w)
        rows, cols = m.struct.rows, m.struct.cols
        out = np.empty((rows, cols), dtype=np.float64)
        for o in range(rows):
            for i in range(cols):
                out[o, i] = self.lib.orc_weight_at(ctypes.byref(m.struct), o, i)
        return out

    def gemv(self, w, x, threads: int = 1) -> np.ndarray:
        m = _weight(w)
        x = _f64(x)
        assert x.shape == (m.struct.cols,)
        y = np.empty(m.struct.rows, dtype=np.float64)
        self.lib.orc_gemv(ctypes.byref(m.struct), _dptr(x), _dptr(y), threads)
        return y

    # ------------------------------------------------------------ the call

    def hc_call(self, raw, g, down, up, inject, *, H: int, C: int, L: int,
                eps: float = RMS_EPS, gate=None, gate_stride: Optional[int] = None,
                threads: Optional[int] = None, want_w: bool = False) -> dict:
        """One hyper-connection call on M tokens; ``inject=None`` gives the final mixer.

        raw: [M, C*H] values; g: [C*H]. Returns float64 ``mixed`` [M, H],
        ``inv_rms`` [M, C], ``a`` [M, L] (the silu output), ``w`` [M, C*H] (the
        sigmoid output) if asked, and ``gate`` [M, C] -- or, when a strided
        ``gate`` buffer is given, that buffer filled in place.
        """
        raw = _f64(raw).reshape(-1, C * H)
        M = raw.shape[0]
        g = _f64(g).reshape(C * H)
        md, mu, mi = _weight(down), _weight(up), _weight(inject)
        mixed = np.empty((M, H), dtype=np.float64)
        inv_rms = np.empty((M, C), dtype=np.float64)
        a = np.empty((M, L), dtype=np.float64)
        w = np.empty((M, C * H), dtype=np.float64) if want_w else None
        own_gate = gate is None
        if own_gate:
            gate_stride = C
            gate = np.full(max(M * C, 1), np.nan, dtype=np.float64)
        else:
            assert gate.dtype == np.float64 and gate_stride is not None
        rc = self.lib.orc_hc_call(M, H, C, L, eps, _dptr(raw), _dptr(g), _wptr(md), _wptr(mu),
                                  _wptr(mi), _dptr(mixed), _dptr(gate), int(gate_stride),
                                  _dptr(inv_rms), _dptr(a), _dptr(w), threads or default_threads())
        if rc != 0:
            raise ValueError("oracle: inconsistent shapes")
        res = {"mixed": mixed, "inv_rms": inv_rms, "a": a}
        if want_w:
            res["w"] = w
        if inject is not None:
            res["gate"] = gate[: M * C].reshape(M, C) if own_gate else gate
        return res

    def mixer(self, raw, g, down, up, **kw) -> dict:
        """The final hyper_connection_mixer: the call without block_inject_weight."""
        return self.hc_call(raw, g, down, up, None, **kw)

    def inject_add(self, raw, out, gate, *, H: int, C: int,
                   gate_stride: Optional[int] = None) -> np.ndarray:
        """raw + (out[:, None, :] * gate[:, :, None]).flatten(), onto the un-normalized raw."""
        raw = _f64(raw).reshape(-1, C * H)
        M = raw.shape[0]
        out = _f64(out).reshape(M, H)
        gate = _f64(gate).reshape(-1)
        gate_stride = C if gate_stride is None else gate_stride
        res = np.empty_like(raw)
        self.lib.orc_inject_add(M, H, C, _dptr(raw), _dptr(out), _dptr(gate), gate_stride,
                                _dptr(res))
        return res

    def lm_head(self, mixed, lm_head_w, *, threads: Optional[int] = None) -> np.ndarray:
        """logits = lm_head(mixed), one plain GEMV per token (families/qwen4/mod.rs,
        decoder pseudocode, exit lines: the mixer's output goes straight to lm_head,
        with no softcap and no separate final norm).

        ``mixed`` [M, H] values; ``lm_head_w`` bf16 [V][H] (a tensor). Returns [M, V].
        """
        mixed = _f64(mixed)
        V, H = lm_head_w.shape
        w = _LinearBf16(V, H, lm_head_w)
        return np.stack([self.gemv(w, mixed[m], threads=threads or default_threads())
                         for m in range(mixed.shape[0])])

    def ple(self, hidden, rows, table, key_proj, value_proj, norm_key, norm_query, norm_conv, conv_w, state, *,
            H: int, C: int, eps: float = RMS_EPS, threads: Optional[int] = None) -> dict:
        """The PLE gate on M consecutive tokens of one sequence (families/qwen4/mod.rs,
        "## PLE"): hidden + gv + silu(dilated_conv(norm_conv(gv))).

        hidden [M, C*H] values; rows int [M, 16]; table bf16 [n_rows, H/16];
        key_proj bf16 [C*H, H]; value_proj bf16 [H, H]; norm_key / norm_query /
        norm_conv [C*H]; conv_w bf16 [C*H, 4]; state [9, C*H] (the conv inputs of
        the 9 tokens before the chunk, oldest first). Returns float64 ``result``
        [M, C*H] (hidden + out, unrounded), ``state`` [9, C*H] after the chunk, and
        the intermediates ``key`` [M, C*H] (normed), ``value`` [M, H], ``gate``
        [M, C] (after the sigmoid), ``x`` [M, C*H] (the conv input).
        """
        W = C * H
        hidden = _f64(hidden).reshape(-1, W)
        M = hidden.shape[0]
        rows = np.ascontiguousarray(np.asarray(rows.cpu() if hasattr(rows, "cpu") else rows, dtype=np.int32))
        assert rows.shape == (M, 16)
        table_bits = _np_bits(table).view(np.uint16)
        conv_bits = _np_bits(conv_w).view(np.uint16)
        assert conv_bits.shape == (W, 4) and table_bits.shape[1] == H // 16
        mk = _weight(_LinearBf16(W, H, key_proj))
        mv = _weight(_LinearBf16(H, H, value_proj))
        nk, nq, nc = (_f64(v).reshape(W) for v in (norm_key, norm_query, norm_conv))
        state = _f64(state).reshape(9, W)
        result = np.empty((M, W))
        state_out = np.empty((9, W))
        key = np.empty((M, W))
        value = np.empty((M, H))
        gate = np.empty((M, C))
        x = np.empty((M, W))
        rc = self.lib.orc_ple(M, H, C, eps, _dptr(hidden), rows.ctypes.data, table_bits.ctypes.data,
                              table_bits.shape[0], _wptr(mk), _wptr(mv), _dptr(nk), _dptr(nq), _dptr(nc),
                              conv_bits.ctypes.data, _dptr(state), _dptr(result), _dptr(state_out), _dptr(key),
                              _dptr(value), _dptr(gate), _dptr(x), threads or default_threads())
        if rc != 0:
            raise ValueError("oracle: inconsistent PLE arguments")
        return {"result": result, "state": state_out, "key": key, "value": value, "gate": gate, "x": x}

    def replicate_entry(self, emb, *, H: int, C: int) -> np.ndarray:
        emb = _f64(emb).reshape(-1, H)
        raw = np.empty((emb.shape[0], C * H), dtype=np.float64)
        self.lib.orc_replicate_entry(emb.shape[0], H, C, _dptr(emb), _dptr(raw))
        return raw

    # ------------------------------------------------------------ drivers

    def prefill_pair(self, raw, attn, out_attn, mlp, out_mlp, *, H: int, C: int, L: int,
                     eps: float = RMS_EPS, round_residual: bool = False,
                     threads: Optional[int] = None) -> dict:
        """attn_hc + inject-add, then mlp_hc + inject-add, on an M-token micro-batch.

        ``attn`` / ``mlp`` carry attributes g, down, up, inject. Token t's
        attn_hc gates go to element t*C*2 of one gate buffer and its mlp_hc
        gates to t*C*2 + C, so no token's gate is overwritten before its
        inject-add reads it (families/qwen4/hc.rs, ``inject_row_offset``).
        ``round_residual`` stores the residual in bf16 after each inject-add.
        """
        raw = _f64(raw).reshape(-1, C * H)
        M = raw.shape[0]
        gates = np.full(M * 2 * C, np.nan, dtype=np.float64)
        r1 = self.hc_call(raw, attn.g, attn.down, attn.up, attn.inject, H=H, C=C, L=L, eps=eps,
                          gate=gates, gate_stride=2 * C, threads=threads)
        raw1 = self.inject_add(raw, out_attn, gates, H=H, C=C, gate_stride=2 * C)
        if round_residual:
            raw1 = self.round_to_bf16(raw1)
        gates_mlp = gates[C:]  # a view: its element t*2C is element t*2C + C of the buffer
        r2 = self.hc_call(raw1, mlp.g, mlp.down, mlp.up, mlp.inject, H=H, C=C, L=L, eps=eps,
                          gate=gates_mlp, gate_stride=2 * C, threads=threads)
        raw2 = self.inject_add(raw1, out_mlp, gates_mlp, H=H, C=C, gate_stride=2 * C)
        if round_residual:
            raw2 = self.round_to_bf16(raw2)
        return {"mixed_attn": r1["mixed"], "raw_after_attn": raw1, "mixed_mlp": r2["mixed"],
                "raw_after_mlp": raw2, "gates": gates.reshape(M, 2, C),
                "inv_rms_attn": r1["inv_rms"], "a_attn": r1["a"],
                "inv_rms_mlp": r2["inv_rms"], "a_mlp": r2["a"]}

    def stack(self, emb, layers: Sequence, outs: Sequence, final, *, H: int, C: int, L: int,
              eps: float = RMS_EPS, round_residual: bool = True, ple=None, ple_rows=None, ple_state=None,
              threads: Optional[int] = None) -> dict:
        """The decoder stack's hyper-connection path on M tokens (one sequence, in order).

        entry: raw = emb repeated C times; per layer l, with ``layers[l]`` =
        (attn, mlp) and ``outs[l]`` = (out_attn, out_mlp): attn_hc + inject,
        mlp_hc + inject; exit: the final mixer with ``final`` (g, down, up).
        With ``ple`` (PLE weights: table, key_proj, value_proj, norm_key,
        norm_query, norm_conv, conv_w), ``ple_rows`` [M, 16] and ``ple_state``
        [9, C*H]: raw = ple(raw) before layer 1's attn_hc (families/qwen4/mod.rs,
        decoder pseudocode, layer_idx == 1 only).

        ``round_residual``: the residual is a bf16 tensor between calls, so it
        is rounded to bf16 (ties to even) after every inject-add and after the
        PLE, as stored. Each call itself is exact in fp64.

        Also returns ``peak``: per element, the largest |raw| the residual held
        at entry, after any inject-add or after the PLE (a bf16 rounding decision
        taken at that magnitude moves the element by one ulp of it), and, with
        the PLE, ``ple_state`` after the tokens.
        """
        raw = self.replicate_entry(emb, H=H, C=C)
        peak = np.abs(raw)
        state_out = None
        for layer, ((attn, mlp), (o_attn, o_mlp)) in enumerate(zip(layers, outs)):
            if ple is not None and layer == 1:
                p = self.ple(raw, ple_rows, ple.table, ple.key_proj, ple.value_proj, ple.norm_key,
                             ple.norm_query, ple.norm_conv, ple.conv_w, ple_state, H=H, C=C, eps=eps,
                             threads=threads)
                raw = self.round_to_bf16(p["result"]) if round_residual else p["result"]
                state_out = p["state"]
                peak = np.maximum(peak, np.abs(raw))
            r = self.prefill_pair(raw, attn, o_attn, mlp, o_mlp, H=H, C=C, L=L, eps=eps,
                                  round_residual=round_residual, threads=threads)
            peak = np.maximum(peak, np.maximum(np.abs(r["raw_after_attn"]), np.abs(r["raw_after_mlp"])))
            raw = r["raw_after_mlp"]
        fin = self.mixer(raw, final.g, final.down, final.up, H=H, C=C, L=L, eps=eps,
                         threads=threads)
        out = {"mixed": fin["mixed"], "raw": raw, "peak": peak}
        if ple is not None:
            out["ple_state"] = state_out
        return out


_lock = threading.Lock()
_default: Optional[Oracle] = None


def get() -> Oracle:
    """The oracle built from the committed ``hc_oracle.c``."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle()
        return _default
