"""Seeded synthetic inputs for the hyper-connection call.

This module only draws numbers: it holds none of the call's arithmetic. It is
the one module that both the CUDA path's tests/benchmark and the CPU oracle
consume, so that both sides see bit-identical inputs.

Recipe (shapes and distributions of the qwen4_exp decode workload, H=2560,
C=4, hc_lowrank=320, as families/qwen4/mod.rs describes it; no trained
checkpoint exists, so every tensor is synthetic):

* values are drawn in fp32 from ``torch.Generator`` (CPU) and rounded to bf16,
  ties to even;
* residual ``raw`` ~ N(0, 1), its C streams drawn independently (distinct);
* ``hc_norm.weight`` g = 1 + N(0, 0.1);
* down / up / inject weights ~ N(0, 0.02);
* synthetic sublayer outputs ``out`` ~ N(0, 1), one per (layer, sublayer);
* the entry embedding row ~ N(0, 1), replicated C times by the call site;
* INT4-affine weights are quantised from the bf16 draws: per output row and
  group of ``group`` consecutive inputs, s = (max - min) / 15 and b = min, both
  rounded to fp16, q = clamp(round((w - b) / s), 0, 15) (q = 0 when s = 0);
  element 2i is the low nibble of byte i.

Every tensor has its own generator seed, derived from (config seed, weight-set
index, tensor id) by ``tensor_seed``.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import torch

G_ID, DOWN_ID, UP_ID, INJECT_ID, RAW_ID, OUT_ID, EMB_ID = range(7)
PLE_TABLE_ID, PLE_KEY_ID, PLE_VALUE_ID, PLE_NORMS_ID, PLE_CONV_ID, PLE_ROWS_ID, PLE_STATE_ID = range(7, 14)


def tensor_seed(config_seed: int, set_index: int, tensor_id: int) -> int:
    return (config_seed * 1_000_003 + set_index) * 16 + tensor_id


def bf16_normal(shape, seed: int, std: float = 1.0, mean: float = 0.0) -> torch.Tensor:
    gen = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(torch.bfloat16)


@dataclass
class Weight:
    """A [rows][cols] linear weight (rows = outputs) in its storage format.

    kind 'bf16': ``data`` bf16 [rows][cols].
    kind 'int4': ``data`` uint8 [rows][cols/2] (element 2i in the low nibble of
    byte i), ``scale`` / ``bias`` fp16 [rows][cols/group].
    """
    kind: str
    rows: int
    cols: int
    data: torch.Tensor
    scale: Optional[torch.Tensor] = None
    bias: Optional[torch.Tensor] = None
    group: int = 0

    def to(self, device) -> "Weight":
        mv = lambda t: None if t is None else t.to(device)
        return Weight(self.kind, self.rows, self.cols, mv(self.data), mv(self.scale),
                      mv(self.bias), self.group)

    @property
    def nbytes(self) -> int:
        n = self.data.numel() * self.data.element_size()
        for t in (self.scale, self.bias):
            if t is not None:
                n += t.numel() * t.element_size()
        return n


def quantize_int4_affine(w: torch.Tensor, group: int) -> Weight:
    """Min/max affine INT4 quantisation of a bf16 [rows][cols] weight (input preparation)."""
    rows, cols = w.shape
    assert cols % group == 0 and cols % 2 == 0
    wf = w.float().reshape(rows, cols // group, group)
    lo = wf.amin(dim=2)
    hi = wf.amax(dim=2)
    scale = ((hi - lo) / 15.0).to(torch.float16)
    bias = lo.to(torch.float16)
    s = scale.float().unsqueeze(2)
    b = bias.float().unsqueeze(2)
    q = torch.where(s > 0, torch.round((wf - b) / torch.where(s > 0, s, torch.ones_like(s))),
                    torch.zeros_like(wf))
    q = q.clamp(0, 15).to(torch.uint8).reshape(rows, cols)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).contiguous()
    return Weight("int4", rows, cols, packed, scale.contiguous(), bias.contiguous(), group)


@dataclass
class HCWeights:
    """The weights of one hyper-connection module (attn_hc, mlp_hc or the mixer)."""
    g: torch.Tensor                  # hc_norm.weight, bf16 [C*H]
    down: Weight                     # input_mix_weight_down.weight, [L][C*H]
    up: Weight                       # input_mix_weight_up.weight, [C*H][L]
    inject: Optional[Weight] = None  # block_inject_weight.weight, [C][C*H]; None for the mixer

    def to(self, device) -> "HCWeights":
        return HCWeights(self.g.to(device), self.down.to(device), self.up.to(device),
                         None if self.inject is None else self.inject.to(device))

    @property
    def nbytes(self) -> int:
        n = self.g.numel() * 2 + self.down.nbytes + self.up.nbytes
        return n + (self.inject.nbytes if self.inject is not None else 0)


def make_hc_weights(H: int, C: int, L: int, config_seed: int, set_index: int = 0,
                    kind: str = "bf16", with_inject: bool = True, group: int = 64,
                    up_group: Optional[int] = None, std: float = 0.02) -> HCWeights:
    """One module's weights. ``std`` is the standard deviation of the down, up and
    inject draws (0.02 in the workload; larger values put silu and sigmoid outside
    their near-linear range)."""
    W = C * H
    s = lambda tid: tensor_seed(config_seed, set_index, tid)
    g = bf16_normal((W,), s(G_ID), std=0.1, mean=1.0)
    down = bf16_normal((L, W), s(DOWN_ID), std=std)
    up = bf16_normal((W, L), s(UP_ID), std=std)
    inj = bf16_normal((C, W), s(INJECT_ID), std=std) if with_inject else None
    if kind == "bf16":
        wrap = lambda t: None if t is None else Weight("bf16", t.shape[0], t.shape[1], t)
        return HCWeights(g, wrap(down), wrap(up), wrap(inj))
    if kind == "int4":
        ug = up_group or group
        return HCWeights(g, quantize_int4_affine(down, group), quantize_int4_affine(up, ug),
                         None if inj is None else quantize_int4_affine(inj, group))
    raise ValueError(kind)


def make_residual(M: int, H: int, C: int, config_seed: int, set_index: int = 0) -> torch.Tensor:
    """raw ~ N(0,1) bf16 [M][C*H]; each stream drawn independently."""
    return bf16_normal((M, C * H), tensor_seed(config_seed, set_index, RAW_ID))


def make_sublayer_out(M: int, H: int, config_seed: int, set_index: int = 0) -> torch.Tensor:
    """Synthetic sublayer output ~ N(0,1) bf16 [M][H]."""
    return bf16_normal((M, H), tensor_seed(config_seed, set_index, OUT_ID))


def make_embedding(M: int, H: int, config_seed: int) -> torch.Tensor:
    return bf16_normal((M, H), tensor_seed(config_seed, 0, EMB_ID))


@dataclass
class Shape:
    M: int
    H: int
    C: int
    L: int

    @property
    def W(self) -> int:
        return self.C * self.H


# The five workloads. Seeds fixed per workload.
TINY = Shape(M=1, H=256, C=4, L=32)          # seed 0
FULL_DECODE = Shape(M=1, H=2560, C=4, L=320)  # seed 1
PREFILL = Shape(M=128, H=2560, C=4, L=320)    # seed 2
STACK_LAYERS = 40                             # seed 3, M = 1 and 16
INT4_GROUP = 64                               # seed 4, M = 1 and 64
SEEDS = {"tiny": 0, "full_decode": 1, "prefill": 2, "stack": 3, "int4": 4}


@dataclass
class StackInputs:
    emb: torch.Tensor
    layers: List[Tuple[HCWeights, HCWeights]]
    outs: List[Tuple[torch.Tensor, torch.Tensor]]
    final: HCWeights


def make_stack(M: int, H: int, C: int, L: int, n_layers: int, config_seed: int,
               kind: str = "bf16") -> StackInputs:
    """Entry embedding, per-layer (attn_hc, mlp_hc) weights and sublayer outputs,
    and the final mixer's weights. Weight set 2l is layer l's attn_hc, 2l+1 its
    mlp_hc, 2*n_layers the mixer."""
    emb = make_embedding(M, H, config_seed)
    layers, outs = [], []
    for l in range(n_layers):
        layers.append((make_hc_weights(H, C, L, config_seed, 2 * l, kind),
                       make_hc_weights(H, C, L, config_seed, 2 * l + 1, kind)))
        outs.append((make_sublayer_out(M, H, config_seed, 2 * l),
                     make_sublayer_out(M, H, config_seed, 2 * l + 1)))
    final = make_hc_weights(H, C, L, config_seed, 2 * n_layers, kind, with_inject=False)
    return StackInputs(emb, layers, outs, final)


@dataclass
class PleWeights:
    """The PLE module's tensors (families/qwen4/mod.rs, "## PLE"): a synthetic
    embedding table of n_rows rows of H/16, key_proj [C*H][H], value_proj [H][H],
    the three norm scales [C*H] and the depthwise conv taps [C*H][4] (bf16)."""
    table: torch.Tensor
    key_proj: torch.Tensor
    value_proj: torch.Tensor
    norm_key: torch.Tensor
    norm_query: torch.Tensor
    norm_conv: torch.Tensor
    conv_w: torch.Tensor

    def to(self, device) -> "PleWeights":
        return PleWeights(*(t.to(device) for t in (self.table, self.key_proj, self.value_proj, self.norm_key,
                                                   self.norm_query, self.norm_conv, self.conv_w)))


def make_ple_weights(H: int, C: int, config_seed: int, n_rows: int = 4096, std: float = 0.02) -> PleWeights:
    """Synthetic PLE weights: table rows N(0, 1), projections N(0, std), norm
    scales 1 + N(0, 0.1), conv taps N(0, 0.5) (bf16)."""
    W = C * H
    s = lambda tid, k=0: tensor_seed(config_seed, k, tid)
    return PleWeights(bf16_normal((n_rows, H // 16), s(PLE_TABLE_ID)),
                      bf16_normal((W, H), s(PLE_KEY_ID), std=std), bf16_normal((H, H), s(PLE_VALUE_ID), std=std),
                      bf16_normal((W,), s(PLE_NORMS_ID, 0), std=0.1, mean=1.0),
                      bf16_normal((W,), s(PLE_NORMS_ID, 1), std=0.1, mean=1.0),
                      bf16_normal((W,), s(PLE_NORMS_ID, 2), std=0.1, mean=1.0),
                      bf16_normal((W, 4), s(PLE_CONV_ID), std=0.5))


def make_ple_rows(M: int, n_rows: int, config_seed: int) -> torch.Tensor:
    """16 row ids per token, uniform in [0, n_rows) (int32 [M][16])."""
    gen = torch.Generator(device="cpu").manual_seed(tensor_seed(config_seed, 0, PLE_ROWS_ID))
    return torch.randint(0, n_rows, (M, 16), generator=gen, dtype=torch.int32)


def make_ple_state(H: int, C: int, config_seed: int) -> torch.Tensor:
    """The conv inputs of 9 earlier tokens, N(0, 1) fp32 [9][C*H]."""
    gen = torch.Generator(device="cpu").manual_seed(tensor_seed(config_seed, 0, PLE_STATE_ID))
    return torch.randn((9, C * H), generator=gen, dtype=torch.float32)
