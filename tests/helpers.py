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
from block_diffusion_draft_gb300.dflash_attn import DFlashAttention, DraftCache, PagedCache
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


def assert_close_stream(gpu, ref, what):
    """The bf16 tolerance for outputs that are long sums (the residual stream,
    the MLP output): values reach several units (one bf16 ulp is 2^-5 at
    |r| >= 4), and every element carries the propagated rounding of the bf16
    intermediates it sums, whose size follows the output's RMS, not the
    element's own value.  So the max-abs bound applies per element relative to
    max(1, |ref|, rms(ref)); the relative L2 bound is unchanged."""
    gpu, ref = np.asarray(gpu, np.float64), np.asarray(ref, np.float64)
    assert np.all(np.isfinite(gpu))
    rms = float(np.sqrt(np.mean(ref * ref)))
    scaled = float(np.max(np.abs(gpu - ref) / np.maximum(max(1.0, rms), np.abs(ref))))
    rel = float(np.linalg.norm(gpu - ref) / np.linalg.norm(ref))
    _log(what, "bf16", scaled, rel)
    assert scaled <= BF16_MAX_ABS and rel <= BF16_REL_L2, \
        f"{what}: scaled max={scaled:.3e} rel_l2={rel:.3e}"


# The decoder-layer MLP output passes two bf16 roundings in series before
# its own (the post-norm input and the SwiGLU activation; the post norm takes
# the fp32 residual sum), and the gate x up product doubles the first.  Its
# values reach |y| ~ 10, where half a bf16 ulp is 3.1e-2, and each element's
# rounding error follows the output's RMS rather than its own value.  So the
# max-abs bound (3e-2) applies per element relative to max(1, |ref|,
# rms(ref)), as for the residual stream; the relative L2 bound is the bf16
# one (5e-3).
MLP_MAX_ABS, MLP_REL_L2 = 3e-2, 5e-3


def assert_close_mlp(gpu, ref, what):
    gpu, ref = np.asarray(gpu, np.float64), np.asarray(ref, np.float64)
    assert np.all(np.isfinite(gpu))
    rms = float(np.sqrt(np.mean(ref * ref)))
    scaled = float(np.max(np.abs(gpu - ref) / np.maximum(max(1.0, rms), np.abs(ref))))
    rel = float(np.linalg.norm(gpu - ref) / np.linalg.norm(ref))
    _log(what, "bf16-mlp", scaled, rel)
    assert scaled <= MLP_MAX_ABS and rel <= MLP_REL_L2, \
        f"{what}: scaled max={scaled:.3e} rel_l2={rel:.3e}"


class Scenario:
    """Drive one layer through inference steps on the GPU and in the oracle.

    ``check`` lists the sequences the oracle follows (all of them for small
    cases, a seeded sample for full-size ones: each sequence only depends on
    its own rows)."""

    def __init__(self, sp: W.Spec, seed: int, capacity: int,
                 check: Optional[Sequence[int]] = None, random_gains=False,
                 layer: int = 0, device="cuda", page_size: int = 0):
        self.sp, self.seed, self.device = sp, seed, device
        self.w = W.weights(sp, seed, layer=layer, random_gains=random_gains)
        self.cfg, self.lw = oracle_layer(sp, self.w)
        self.attn = gpu_layer(sp, self.w, device)
        self.page_size = page_size
        if page_size:
            # the caller's bookkeeping of a paged cache: every sequence's pages
            # from a shuffled free list, lengths on the host
            per_seq = (capacity + page_size - 1) // page_size
            rng = np.random.default_rng(seed + 99)
            self.pages = rng.permutation(sp.batch * per_seq).reshape(sp.batch, per_seq)
            self.pages = self.pages.astype(np.int32)
            self.cache = PagedCache(self.attn, sp.batch * per_seq, page_size)
            self.bt = torch.from_numpy(self.pages).to(device)
            self.lens = [0] * sp.batch
        else:
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
        L = self.lengths()
        th = [W.hidden_rows(sp, self.seed, "hidden", s, b, n_ctx[b]) for b in range(sp.batch)]
        nz = [W.hidden_rows(sp, self.seed, "noise", s, b, q_len) for b in range(sp.batch)]
        pos = [W.window_positions(L[b], n_ctx[b], q_len) for b in range(sp.batch)]
        dev = self.device
        noise = torch.stack(nz).to(dev)
        target = torch.cat(th).to(dev) if sum(n_ctx) > 0 else None
        positions = torch.cat(pos).to(dev)
        if self.page_size:
            P = self.page_size
            slots = np.concatenate([self.pages[b][k // P] * P + k % P for b in range(sp.batch)
                                    for k in [np.arange(L[b], L[b] + n_ctx[b] + q_len)]])
            out = self.attn.forward_paged(self.cache, noise, target, n_ctx, L, positions,
                                          torch.from_numpy(slots.astype(np.int32)).to(dev),
                                          self.bt)
            self.lens = [L[b] + n_ctx[b] + q_len for b in range(sp.batch)]
        else:
            out = self.attn.forward(self.cache, noise, target, n_ctx, positions)
        torch.cuda.synchronize()
        # only the followed sequences are widened to fp64 for the oracle
        ref = O.forward(self.cfg, self.lw, self.ocache,
                        np.stack([f64(x) for x in nz]),
                        [f64(th[b]) if b in self.check else None for b in range(sp.batch)],
                        [p.numpy() for p in pos], seqs=self.check)
        got = out.to("cpu", torch.float64).numpy()
        return got[self.check], ref[self.check]

    def lengths(self) -> List[int]:
        return list(self.lens) if self.page_size else self.cache.lengths()

    def crop(self, keep: List[int]):
        if self.page_size:
            self.lens = list(keep)
        else:
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
            if self.page_size:  # gather the sequence's rows through its pages
                P, idx = self.page_size, np.arange(n)[sl]
                kb = np.stack([k[self.pages[b][i // P], :, i % P] for i in idx], axis=1)
                vb = np.stack([v[self.pages[b][i // P], :, i % P] for i in idx], axis=1)
            else:
                kb, vb = k[b][:, sl], v[b][:, sl]
            res.append((kb, self.ocache.k[b][:, sl], vb, self.ocache.v[b][:, sl]))
        return res
