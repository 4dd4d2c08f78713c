"""The five synthetic shard-step workloads and their input recipe.

Shapes and granularities follow the workloads the veScale-FSDP (MLSys 2026)
summary page evaluates (Llama-style dense layers, GPT-OSS-style fused experts,
DeepSeek-V3-shaped 128x128 block-quantised matrices; 实验 section and the
8-bit Adam case study) at single-layer or 1.3B scale:

  tiny        4 tensors, m=4,    g_coll=128, 3 steps
  llama_layer 9 tensors, m=8,    g_coll=128, 10 steps
  moe_layer   3 tensors, m=64,   g_coll=256, 10 steps, 2 of 32 experts zero
  dsv3_block  4 tensors, m=128,  g_coll=512, 10 steps, Student-t(3) grads
  llama_1p3b  219 tensors, m=1024, g_coll=128, 20 steps, clip at norm 1.0

Inputs: master weights N(0, 0.02) in fp32; gradients N(0, 1e-3) in bf16
(dsv3_block: 1e-3 * Student-t(3)); fresh gradients every step from the stream
(seed, step, tensor, KIND_GRAD); seed 0. Nothing here computes the method.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import (DIST_NORMAL, DIST_STUDENT_T3, KIND_GRAD, KIND_PARAM, fill_bf16, fill_f32, key,
               pick)

GRAN_ELEM, GRAN_ROWS, GRAN_TILE = 0, 1, 2


@dataclasses.dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple
    gran: int
    block_rows: int = 0
    tile_cols: int = 0
    experts: int = 0  # >0: leading dim indexes experts (zero-expert slices apply)

    @property
    def numel(self) -> int:
        return int(np.prod(self.shape, dtype=np.int64))

    @property
    def rows(self) -> int:
        return int(np.prod(self.shape[:-1], dtype=np.int64)) if len(self.shape) > 1 else 1

    @property
    def cols(self) -> int:
        return int(self.shape[-1])


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    tensors: tuple
    m: int
    g_coll: int
    steps: int
    grad_dist: int = DIST_NORMAL
    grad_scale: float = 1e-3
    param_scale: float = 0.02
    max_norm: float = math.inf
    zero_experts: int = 0
    seed: int = 0
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01

    @property
    def numel(self) -> int:
        return sum(t.numel for t in self.tensors)

    def zero_expert_ids(self) -> list[int]:
        n_exp = max((t.experts for t in self.tensors), default=0)
        if self.zero_experts == 0 or n_exp == 0:
            return []
        return pick(key(self.seed, 0, 0, 7), n_exp, self.zero_experts)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _rows(name, r, c, br):
    return TensorSpec(name, (r, c), GRAN_ROWS, block_rows=br)


def tiny() -> Workload:
    return Workload("tiny", (
        _rows("w_a", 256, 256, 32),
        TensorSpec("bias", (1024,), GRAN_ELEM),
        TensorSpec("w_b", (512, 256), GRAN_TILE, block_rows=32, tile_cols=32),
        _rows("w_c", 128, 128, 128),
    ), m=4, g_coll=128, steps=3)


def llama_layer() -> Workload:
    h, f = 4096, 11008
    return Workload("llama_layer", (
        _rows("q", h, h, 32), _rows("k", h, h, 32), _rows("v", h, h, 32), _rows("o", h, h, 32),
        _rows("gate", f, h, 32), _rows("up", f, h, 32), _rows("down", h, f, 32),
        TensorSpec("attn_norm", (h,), GRAN_ELEM), TensorSpec("ffn_norm", (h,), GRAN_ELEM),
    ), m=8, g_coll=128, steps=10)


def moe_layer() -> Workload:
    e, h, f = 32, 2880, 5760
    return Workload("moe_layer", (
        TensorSpec("gate_up", (e, f, h), GRAN_ROWS, block_rows=128, experts=e),
        TensorSpec("down", (e, h, h), GRAN_ROWS, block_rows=128, experts=e),
        TensorSpec("router", (e, h), GRAN_ELEM),
    ), m=64, g_coll=256, steps=10, zero_experts=round(0.05 * e))


def dsv3_block() -> Workload:
    h, f = 7168, 18432
    tile = dict(gran=GRAN_TILE, block_rows=128, tile_cols=128)
    return Workload("dsv3_block", (
        TensorSpec("w_in", (h, f), **tile),
        TensorSpec("w_out", (f, h), **tile),
        TensorSpec("norm_a", (h,), GRAN_ELEM),
        TensorSpec("norm_b", (h,), GRAN_ELEM),
    ), m=128, g_coll=512, steps=10, grad_dist=DIST_STUDENT_T3)


def llama_1p3b() -> Workload:
    h, f, vocab, layers = 2048, 5504, 32000, 24
    ts = [_rows("embed", vocab, h, 32)]
    for i in range(layers):
        ts += [TensorSpec(f"l{i}.attn_norm", (h,), GRAN_ELEM),
               _rows(f"l{i}.q", h, h, 32), _rows(f"l{i}.k", h, h, 32),
               _rows(f"l{i}.v", h, h, 32), _rows(f"l{i}.o", h, h, 32),
               TensorSpec(f"l{i}.ffn_norm", (h,), GRAN_ELEM),
               _rows(f"l{i}.gate", f, h, 32), _rows(f"l{i}.up", f, h, 32),
               _rows(f"l{i}.down", h, f, 32)]
    ts += [TensorSpec("final_norm", (h,), GRAN_ELEM), _rows("lm_head", vocab, h, 32)]
    return Workload("llama_1p3b", tuple(ts), m=1024, g_coll=128, steps=20, max_norm=1.0)


ALL = {w().name: w for w in (tiny, llama_layer, moe_layer, dsv3_block, llama_1p3b)}


def get(name: str) -> Workload:
    return ALL[name]()


# ---------------------------------------------------------------- inputs

def master_init(w: Workload, t: int, start: int = 0, count: int | None = None) -> np.ndarray:
    """fp32 master weights of tensor t, elements [start, start+count)."""
    n = w.tensors[t].numel - start if count is None else count
    out = np.empty(n, dtype=np.float32)
    return fill_f32(key(w.seed, 0, t, KIND_PARAM), DIST_NORMAL, w.param_scale, start, out)


def grad(w: Workload, step: int, t: int, start: int = 0, count: int | None = None,
         out: np.ndarray | None = None) -> np.ndarray:
    """bf16 gradient bits (uint16) of tensor t at `step` (1-based), elements
    [start, start+count). Zero-expert slices are zero."""
    spec = w.tensors[t]
    n = spec.numel - start if count is None else count
    if out is None:
        out = np.empty(n, dtype=np.uint16)
    fill_bf16(key(w.seed, step, t, KIND_GRAD), w.grad_dist, w.grad_scale, start, out)
    if spec.experts:
        per = spec.numel // spec.experts
        for e in w.zero_expert_ids():
            lo, hi = max(e * per, start), min((e + 1) * per, start + n)
            if lo < hi:
                out[lo - start:hi - start] = 0
    return out


def grad_f32(w: Workload, step: int, t: int, start: int = 0, count: int | None = None) -> np.ndarray:
    """fp32 gradient variant (same stream, rounded to fp32 only)."""
    spec = w.tensors[t]
    n = spec.numel - start if count is None else count
    out = np.empty(n, dtype=np.float32)
    fill_f32(key(w.seed, step, t, KIND_GRAD), w.grad_dist, w.grad_scale, start, out)
    if spec.experts:
        per = spec.numel // spec.experts
        for e in w.zero_expert_ids():
            lo, hi = max(e * per, start), min((e + 1) * per, start + n)
            if lo < hi:
                out[lo - start:hi - start] = 0
    return out
