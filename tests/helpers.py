"""Helpers shared by the GPU parity tests: build the same layer on the GPU
(through the C ABI) and in the fp64 oracle from the seeded workloads, drive
both through the same steps, and compare."""
from __future__ import annotations

import json
import os
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from block_diffusion_draft_gb300 import workloads as W
from block_diffusion_draft_gb300.dflash_attn import DFlashAttention, DraftCache
from oracle import dflash_oracle as O

# tolerances: bf16 paths max-abs and relative L2; fp32 paths relative L2
BF16_MAX_ABS, BF16_REL_L2 = 2e-2, 5e-3
FP32_REL_L2 = 1e-4


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_layer(sp: W.Spec, w: Dict[str, torch.Tensor]):
    cfg = O.LayerConfig(hidden=sp.hidden, n_heads=sp.n_heads,
                        n_kv_heads=sp.n_kv_heads, head_dim=sp.head_dim,
                        rms_eps=sp.rms_eps, rope_theta=sp.rope_theta,
                        sliding_window=sp.sliding_window,
                        n_target_layers=sp.n_target_layers, causal=sp.causal)
    lw = O.LayerWeights(wq=f64(w["wq"]), wk=f64(w["wk"]), wv=f64(w["wv"]),
                        wo=f64(w["wo"]), q_norm=f64(w["q_norm"]),
                        k_norm=f64(w["k_norm"]),
                        fc=f64(w["fc"]) if "fc" in w else None,
                        hidden_norm=f64(w["hidden_norm"]) if "fc" in w else None)
    return cfg, lw


def gpu_layer(sp: W.Spec, w: Dict[str, torch.Tensor], device="cuda") -> DFlashAttention:
    return DFlashAttention(w, hidden=sp.hidden, n_heads=sp.n_heads,
                           n_kv_heads=sp.n_kv_heads, head_dim=sp.head_dim,
                           n_target_layers=sp.n_target_layers if "fc" in w else 0,
                           rms_eps=sp.rms_eps, rope_theta=sp.rope_theta,
                           sliding_window=sp.sliding_window,
                           max_position=sp.max_position, dtype=sp.torch_dtype(),
                           device=device, causal=sp.causal)


def errors(gpu: np.ndarray, ref: np.ndarray):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), "non-finite GPU values"
    max_abs = float(np.max(np.abs(gpu - ref))) if gpu.size else 0.0
    rel = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-300))
    return max_abs, rel


def _log(what, dtype, max_abs, rel):
    path = os.environ.get("DFLASH_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", ""),
                                "what": what, "dtype": dtype, "max_abs": max_abs,
                                "rel_l2": rel}) + "\n")


def assert_close(gpu, ref, dtype: str, what: str = ""):
    max_abs, rel = errors(gpu, ref)
    _log(what, dtype, max_abs, rel)
    if dtype == "bf16":
        assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_L2, \
            f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    else:
        assert rel <= FP32_REL_L2, f"{what}: rel_l2={rel:.3e}"
    return max_abs, rel


class Scenario:
    """Drive one layer through inference steps on the GPU and in the oracle.

    ``check`` lists the sequences the oracle follows (all of them for small
    cases, a seeded sample for full-size ones: each sequence only depends on
    its own rows)."""

    def __init__(self, sp: W.Spec, seed: int, capacity: int,
                 check: Optional[Sequence[int]] = None, random_gains=False,
                 layer: int = 0, device="cuda"):
        self.sp, self.seed, self.device = sp, seed, device
        self.w = W.weights(sp, seed, layer=layer, random_gains=random_gains)
        self.cfg, self.lw = oracle_layer(sp, self.w)
        self.attn = gpu_layer(sp, self.w, device)
        self.cache = DraftCache(self.attn, sp.batch, capacity)
        self.check = list(range(sp.batch)) if check is None else list(check)
        self.ocache = O.DraftCache(sp.n_kv_heads, sp.head_dim, sp.batch)
        self.step_no = 0

    def step(self, n_ctx: List[int], q_len: Optional[int] = None):
        """One forward on both sides; returns (gpu_out, oracle_out) restricted
        to the checked sequences."""
        sp = self.sp
        q_len = sp.block_size if q_len is None else q_len
        s = self.step_no
        self.step_no += 1
        L = self.cache.lengths()
        th = [W.hidden_rows(sp, self.seed, "hidden", s, b, n_ctx[b]) for b in range(sp.batch)]
        nz = [W.hidden_rows(sp, self.seed, "noise", s, b, q_len) for b in range(sp.batch)]
        pos = [W.window_positions(L[b], n_ctx[b], q_len) for b in range(sp.batch)]
        dev = self.device
        noise = torch.stack(nz).to(dev)
        target = torch.cat(th).to(dev) if sum(n_ctx) > 0 else None
        positions = torch.cat(pos).to(dev)
        out = self.attn.forward(self.cache, noise, target, n_ctx, positions)
        torch.cuda.synchronize()
        # only the followed sequences are widened to fp64 for the oracle
        ref = O.forward(self.cfg, self.lw, self.ocache,
                        np.stack([f64(x) for x in nz]),
                        [f64(th[b]) if b in self.check else None for b in range(sp.batch)],
                        [p.numpy() for p in pos], seqs=self.check)
        got = out.to("cpu", torch.float64).numpy()
        return got[self.check], ref[self.check]

    def crop(self, keep: List[int]):
        self.cache.crop(keep)
        okeep = [keep[b] if b in self.check else 0 for b in range(self.sp.batch)]
        self.ocache.crop(okeep)

    def compare_cache(self, rows: Optional[int] = None):
        """Cached K/V rows of the checked sequences against the oracle's."""
        k, v = self.cache.read()
        k = k.to("cpu", torch.float64).numpy()
        v = v.to("cpu", torch.float64).numpy()
        res = []
        for b in self.check:
            n = self.ocache.k[b].shape[1]
            sl = slice(0, n) if rows is None else slice(max(0, n - rows), n)
            res.append((k[b][:, sl], self.ocache.k[b][:, sl],
                        v[b][:, sl], self.ocache.v[b][:, sl]))
        return res
