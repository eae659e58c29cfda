"""Seeded synthetic inputs for the DFlash draft attention workloads.

This module only draws random numbers and lays out shapes: it holds none of
the layer's arithmetic.  The CUDA path, the CPU oracle, the tests and the
benchmark all take their inputs from here, so both sides always see the same
bf16 (or fp32) values.

Every tensor is drawn from its own counter-keyed stream
(``numpy.random.SeedSequence([seed, *keys])`` feeding PCG64), so one sequence
or one step of a large workload can be regenerated alone, and the values do
not depend on what else was generated before.

The shapes follow the Qwen3 draft layers the pages describe: hidden 4096,
32 query / 8 KV heads, head_dim 128, blocks of 16 (one anchor + 15 mask
tokens), rope_theta 1e6, eps 1e-6, linear weights N(0, 0.02), hidden states
N(0, 1).  No public dataset is involved; real prompts would only change the
values, not the shapes or the work.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Dict, List, Optional

import numpy as np
import torch

# --------------------------------------------------------------------------
# workload specifications
# --------------------------------------------------------------------------


@dataclass(frozen=True)
class Spec:
    name: str
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    batch: int
    dtype: str  # "bf16" | "fp32"
    n_target_layers: int = 5
    rope_theta: float = 1e6
    rms_eps: float = 1e-6
    sliding_window: int = 0
    # serving workloads: rows already in the cache before the measured step,
    # and context rows appended by that step
    prefill: int = 0
    prefill_lo: int = 0
    prefill_hi: int = 0
    n_new: int = 16
    steps: int = 1
    # packed training workload
    seq: int = 0
    n_blocks: int = 0
    max_position: int = 65536
    # layer stacks: draft layers sharing the step's projected context
    layers: int = 1
    # > 0: the whole decoder layer (norms, residual, MLP of this width)
    intermediate: int = 0
    # causal attention layer (block row t sees keys up to its own index)
    causal: bool = False
    # > 0: paged KV cache of pages of this many rows, handed out shuffled
    page_size: int = 0
    # packed layout: attention core forward + backward (training step of the
    # attention) instead of the layer forward
    backward: bool = False

    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def dtype_name(self) -> str:
        """The arithmetic type of the path, as a bench line states it."""
        return "bf16" if self.dtype == "bf16" else "f32"


SPECS: Dict[str, Spec] = {
    # tiny fp32 single layer: 112 rows prefilled, then 16 new ctx + 16 block
    "tiny_fp32": Spec("tiny_fp32", hidden=256, n_heads=4, n_kv_heads=2,
                      head_dim=64, block_size=16, batch=1, dtype="fp32",
                      n_target_layers=2, prefill=112, n_new=16,
                      max_position=4096),
    # Qwen3-8B-shaped layer, one sequence: 4096 cached + 16 new ctx + 16 block
    "qwen3_8b_single": Spec("qwen3_8b_single", hidden=4096, n_heads=32,
                            n_kv_heads=8, head_dim=128, block_size=16,
                            batch=1, dtype="bf16", prefill=4096, n_new=16),
    # serving batch: 32 sequences, cached length U[512, 8192], accept U{1..16}
    "serving_b32": Spec("serving_b32", hidden=4096, n_heads=32, n_kv_heads=8,
                        head_dim=128, block_size=16, batch=32, dtype="bf16",
                        prefill_lo=512, prefill_hi=8192, n_new=16, steps=64),
    # the same batch over a paged cache (16-row pages in shuffled order)
    "serving_b32_paged": Spec("serving_b32_paged", hidden=4096, n_heads=32,
                              n_kv_heads=8, head_dim=128, block_size=16, batch=32,
                              dtype="bf16", prefill_lo=512, prefill_hi=8192, n_new=16,
                              steps=64, page_size=16),
    # long context: 32768 cached + 16 new + 16 block, full layer
    "long_ctx_full": Spec("long_ctx_full", hidden=4096, n_heads=32,
                          n_kv_heads=8, head_dim=128, block_size=16, batch=4,
                          dtype="bf16", prefill=32768, n_new=16),
    # the same with a sliding-attention layer (window 4096, band over keys)
    "long_ctx_swa": Spec("long_ctx_swa", hidden=4096, n_heads=32,
                         n_kv_heads=8, head_dim=128, block_size=16, batch=4,
                         dtype="bf16", prefill=32768, n_new=16,
                         sliding_window=4096),
    # the whole Qwen3-8B-shaped decoder layer (attention + SwiGLU MLP of
    # width 12288), one sequence: 4096 cached + 16 new ctx + 16 block
    "decoder_8b_single": Spec("decoder_8b_single", hidden=4096, n_heads=32,
                              n_kv_heads=8, head_dim=128, block_size=16, batch=1,
                              dtype="bf16", prefill=4096, n_new=16, intermediate=12288),
    # five Qwen3-8B-shaped draft layers fed by one projected context: 4096
    # cached rows, then 16 (decode) or 512 (a long accepted run / prefill
    # chunk) new context rows and one block per layer
    "stack5_ctx16": Spec("stack5_ctx16", hidden=4096, n_heads=32, n_kv_heads=8,
                         head_dim=128, block_size=16, batch=1, dtype="bf16",
                         prefill=4096, n_new=16, layers=5),
    "stack5_ctx512": Spec("stack5_ctx512", hidden=4096, n_heads=32, n_kv_heads=8,
                          head_dim=128, block_size=16, batch=1, dtype="bf16",
                          prefill=4096, n_new=512, layers=5),
    # packed training layout: 2 x 4096 context rows, 256 anchors x 16 rows
    "packed_train": Spec("packed_train", hidden=4096, n_heads=32,
                         n_kv_heads=8, head_dim=128, block_size=16, batch=2,
                         dtype="bf16", seq=4096, n_blocks=256),
    # the same shape through the attention core forward and its backward
    # (dQ, dK, dV through the anchor mask)
    "packed_train_bwd": Spec("packed_train_bwd", hidden=4096, n_heads=32,
                             n_kv_heads=8, head_dim=128, block_size=16, batch=2,
                             dtype="bf16", seq=4096, n_blocks=256, backward=True),
}


def spec(name: str, **overrides) -> Spec:
    return replace(SPECS[name], **overrides)


# --------------------------------------------------------------------------
# random streams
# --------------------------------------------------------------------------
_KIND = {"weight": 1, "hidden": 2, "noise": 3, "layers": 4, "lengths": 5,
         "accept": 6, "anchors": 7, "gain": 8, "core": 9}


def _rng(seed: int, kind: str, *keys: int) -> np.random.Generator:
    return np.random.Generator(
        np.random.PCG64(np.random.SeedSequence([seed, _KIND[kind], *keys])))


def _normal(rng: np.random.Generator, shape, std: float, dtype: torch.dtype):
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return torch.from_numpy(a).to(dtype)


# --------------------------------------------------------------------------
# parameters
# --------------------------------------------------------------------------
def weights(sp: Spec, seed: int = 0, layer: int = 0,
            random_gains: bool = False, with_fc: bool = True) -> Dict[str, torch.Tensor]:
    """Layer parameters in nn.Linear [out, in] layout, in the spec's dtype.

    Linear weights N(0, 0.02); norm gains 1 (standard init) or, with
    ``random_gains``, 1 + N(0, 0.1).
    """
    dt = sp.torch_dtype()
    H, d = sp.hidden, sp.head_dim
    nq, nkv = sp.n_heads * d, sp.n_kv_heads * d
    w = {
        "wq": _normal(_rng(seed, "weight", layer, 0), (nq, H), 0.02, dt),
        "wk": _normal(_rng(seed, "weight", layer, 1), (nkv, H), 0.02, dt),
        "wv": _normal(_rng(seed, "weight", layer, 2), (nkv, H), 0.02, dt),
        "wo": _normal(_rng(seed, "weight", layer, 3), (H, nq), 0.02, dt),
    }
    if with_fc and sp.n_target_layers > 0:
        w["fc"] = _normal(_rng(seed, "weight", layer, 4),
                          (H, sp.n_target_layers * H), 0.02, dt)
    for i, (name, n) in enumerate((("q_norm", d), ("k_norm", d),
                                   ("hidden_norm", H))):
        if random_gains:
            g = 1.0 + 0.1 * _rng(seed, "gain", layer, i).standard_normal(
                n, dtype=np.float32)
            w[name] = torch.from_numpy(g).to(dt)
        else:
            w[name] = torch.ones(n, dtype=dt)
    return w


# --------------------------------------------------------------------------
# activations
# --------------------------------------------------------------------------
def mlp_weights(sp: Spec, seed: int, intermediate: int, layer: int = 0,
                random_gains: bool = False) -> Dict[str, torch.Tensor]:
    """Decoder-layer MLP and norm weights: gate, up [intermediate, hidden],
    down [hidden, intermediate] N(0, 0.02); norm gains 1 (or 1 + N(0, 0.1))."""
    dt = sp.torch_dtype()
    H = sp.hidden
    w = {"gate": _normal(_rng(seed, "weight", layer, 5), (intermediate, H), 0.02, dt),
         "up": _normal(_rng(seed, "weight", layer, 6), (intermediate, H), 0.02, dt),
         "down": _normal(_rng(seed, "weight", layer, 7), (H, intermediate), 0.02, dt)}
    for i, name in enumerate(("input_norm", "post_norm")):
        if random_gains:
            g = 1.0 + 0.1 * _rng(seed, "gain", layer, 3 + i).standard_normal(H, dtype=np.float32)
            w[name] = torch.from_numpy(g).to(dt)
        else:
            w[name] = torch.ones(H, dtype=dt)
    return w


def hidden_rows(sp: Spec, seed: int, kind: str, step: int, seq: int,
                rows: int) -> torch.Tensor:
    """N(0,1) rows of width hidden: ``kind`` is "hidden" (projected context,
    i.e. target_hidden) or "noise" (block embeddings)."""
    return _normal(_rng(seed, kind, step, seq), (rows, sp.hidden), 1.0,
                   sp.torch_dtype())


def target_layer_rows(sp: Spec, seed: int, step: int, seq: int,
                      rows: int) -> torch.Tensor:
    """N(0,1) rows of the concatenated target layers (fc input width)."""
    return _normal(_rng(seed, "layers", step, seq),
                   (rows, sp.n_target_layers * sp.hidden), 1.0, sp.torch_dtype())


def window_positions(start: int, n_ctx: int, q_len: int) -> torch.Tensor:
    """Positions of one sequence's window: the new context rows continue the
    cached rows (absolute row index), the block follows them."""
    return torch.arange(start, start + n_ctx + q_len, dtype=torch.int32)


# --------------------------------------------------------------------------
# serving schedule
# --------------------------------------------------------------------------
@dataclass
class ServingStep:
    n_ctx: List[int]     # new context rows per sequence
    accept: List[int]    # block tokens accepted after verification


@dataclass
class ServingSchedule:
    prefill: List[int]                      # cached rows before step 0
    steps: List[ServingStep] = field(default_factory=list)


def serving_schedule(sp: Spec, seed: int = 0,
                     steps: Optional[int] = None) -> ServingSchedule:
    """Cached lengths and per-step context counts for a serving workload.

    Fixed-length specs (``prefill`` > 0) start every sequence at ``prefill``
    rows; ragged ones draw U[prefill_lo, prefill_hi].  Step 0 appends
    ``n_new`` context rows per sequence; step s > 0 appends as many as the
    previous step accepted (U{1..block_size}).
    """
    B = sp.batch
    if sp.prefill > 0:
        pre = [sp.prefill] * B
    else:
        pre = _rng(seed, "lengths", 0).integers(
            sp.prefill_lo, sp.prefill_hi + 1, size=B).tolist()
    n_steps = sp.steps if steps is None else steps
    sched = ServingSchedule(prefill=[int(x) for x in pre])
    n_ctx = [sp.n_new] * B
    for s in range(n_steps):
        acc = _rng(seed, "accept", s).integers(
            1, sp.block_size + 1, size=B).tolist()
        sched.steps.append(ServingStep(n_ctx=list(n_ctx),
                                       accept=[int(a) for a in acc]))
        n_ctx = [int(a) for a in acc]
    return sched


# --------------------------------------------------------------------------
# packed training layout
# --------------------------------------------------------------------------
def anchors(sp: Spec, seed: int = 0) -> torch.Tensor:
    """Distinct sorted anchors per sequence, uniform in [1, seq - block_size]."""
    out = np.empty((sp.batch, sp.n_blocks), dtype=np.int32)
    for b in range(sp.batch):
        r = _rng(seed, "anchors", b)
        pick = r.choice(np.arange(1, sp.seq - sp.block_size + 1),
                        size=sp.n_blocks, replace=False)
        out[b] = np.sort(pick)
    return torch.from_numpy(out)


def core_tensors(sp: Spec, seed: int = 0) -> Dict[str, torch.Tensor]:
    """Inputs of the packed attention core and its backward, N(0,1): q and
    the output gradient d_out [B, nb*bs, n_heads, d] (per-head RMSNorm makes
    q and k unit-RMS per head, RoPE keeps that), k and v
    [B, n_kv, seq + nb*bs, d]."""
    T = sp.n_blocks * sp.block_size
    per = sp.seq + T
    shapes = {"q": (sp.batch, T, sp.n_heads, sp.head_dim),
              "k": (sp.batch, sp.n_kv_heads, per, sp.head_dim),
              "v": (sp.batch, sp.n_kv_heads, per, sp.head_dim),
              "d_out": (sp.batch, T, sp.n_heads, sp.head_dim)}
    return {name: _normal(_rng(seed, "core", i), shape, 1.0, sp.torch_dtype())
            for i, (name, shape) in enumerate(shapes.items())}

