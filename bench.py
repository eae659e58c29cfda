#!/usr/bin/env python
"""Benchmark of the DFlash draft attention layer on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  ctx_project (fc + hidden_norm of the step's new context rows)
  -> forward (QKV projection + q/k norm + RoPE + cache append, split-KV
     attention, o_proj)
  -> crop (back to the accepted prefix).
The default workload is the serving batch of Qwen3-8B-shaped draft layers:
32 sequences with cached lengths uniform in [512, 8192], each step appending
the previous step's accepted tokens as context rows (16 at the first step)
plus a 16-row block, then cropping back to an accepted prefix of 1..16 block
rows; fc 20480 -> 4096 over the step's new context rows.  This is the
KV-read-bound configuration; `--workload` selects the others.
The metric is draft-attention blocks/s per layer (one block = one sequence's
block through one layer).  Inputs are synthetic, seeded, N(0,1) hidden
states and N(0,0.02) weights.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle, timed on the host

Prints one JSON line (rank 0).  Under torchrun (N > 1) each rank runs an
independent replica of the workload on its own GPU (the layer needs no
exchange between sequences): value = blocks of all ranks / slowest rank time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(ROOT, "block_diffusion_draft_gb300", "csrc")


def csrc_digest() -> str:
    """sha256 over the CUDA sources (names and contents, sorted by name)."""
    import hashlib
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            h.update(name.encode())
            with open(os.path.join(CSRC, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def source_digests() -> dict:
    """sha256 of each CUDA source file."""
    import hashlib
    out = {}
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, name), "rb") as f:
                out[name] = hashlib.sha256(f.read()).hexdigest()
    return out


def measured_traffic(workload: str, kernel: str):
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu
    capture in profiles/traffic.json, or None when there is none or a source
    file of that kernel (its own file, the shared headers, the launch logic)
    changed since it was taken."""
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tfile):
        return None
    tj = json.load(open(tfile))
    rec = tj.get("kernels", {}).get(f"{workload}:{kernel}")
    if not rec:
        return None
    then, now = tj.get("file_sha256", {}), source_digests()
    srcs = rec.get("sources")
    if srcs is None:  # no per-file record: every source must match
        if tj.get("csrc_sha256") != csrc_digest():
            return None
    elif any(then.get(f) is None or then.get(f) != now.get(f) for f in srcs):
        return None
    return rec.get("bytes_per_launch")

# DRAM traffic of each workload's dominant kernel, captured by ncu one kernel
# at a time (a regex on the demangled name, a few launches after set-up):
#   ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum
#       --clock-control none --kernel-name-base demangled -k regex:<kernel> -s 3 -c 3
#       --csv --log-file <dir>/traffic_<workload>.csv
#       python bench.py --workload <workload> --steps 2 --warmup 3 --no-cpu-baseline --no-clocks
# `python bench.py --ncu-traffic <dir>` turns those logs into profiles/traffic.json
# (read back by measured_traffic) and profiles/traffic.md.
_COMMON_SRC = ["dflash_api.cu", "handles.h", "internal.h", "ptx.cuh"]
TRAFFIC_CAPTURE = {
    # workload: (trace bucket, kernel regex, source files of that kernel)
    "qwen3_8b_single": ("fc", r"gemm_bf16_kernel<\(int\)1, \(int\)128>",
                        ["gemm_bf16.cu"] + _COMMON_SRC),
    "long_ctx_swa": ("fc", r"gemm_bf16_kernel<\(int\)1, \(int\)128>",
                     ["gemm_bf16.cu"] + _COMMON_SRC),
    "serving_b32": ("attn", "attn_bf16_kernel", ["attn_bf16.cu"] + _COMMON_SRC),
    "serving_b32_paged": ("attn", "attn_bf16_kernel", ["attn_bf16.cu"] + _COMMON_SRC),
    "long_ctx_full": ("attn", "attn_bf16_kernel", ["attn_bf16.cu"] + _COMMON_SRC),
    "packed_train": ("qkv", r"gemm_big_kernel<\(int\)2, \(int\)2>",
                     ["gemm_bf16.cu"] + _COMMON_SRC),
    "packed_train_bwd": ("bwd", "packed_bwd_kernel", ["attn_bwd.cu"] + _COMMON_SRC),
}


def _ncu_rows(path):
    """(launch id, kernel name, {metric: value in bytes or ns}) from an ncu --csv log."""
    import csv
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "nsecond": 1.0,
             "usecond": 1e3, "msecond": 1e6, "second": 1e9}
    launches = {}
    with open(path, newline="") as f:
        lines = [ln for ln in f if ln.startswith('"')]
    rd = csv.reader(lines)
    hdr = next(rd, None)
    if hdr is None:
        return []
    ix = {h: i for i, h in enumerate(hdr)}
    for r in rd:
        if len(r) < len(hdr) or r[ix["ID"]] == "ID":
            continue
        v = float(r[ix["Metric Value"]].replace(",", ""))
        rec = launches.setdefault(int(r[ix["ID"]]), [r[ix["Kernel Name"]], {}])
        rec[1][r[ix["Metric Name"]]] = v * scale.get(r[ix["Metric Unit"]], 1.0)
    return [(k, n, m) for k, (n, m) in sorted(launches.items())]


def launch_table(path):
    """Markdown rows (kernel, launches, total us, share) of an ncu launch list."""
    per = {}
    for _, name, m in _ncu_rows(path):
        k = name.split("(")[0].replace("void ", "").replace("df::<unnamed>::", "")
        per.setdefault(k, []).append(m.get("gpu__time_duration.sum", 0.0) / 1e3)
    tot = sum(sum(v) for v in per.values()) or 1.0
    return [f"| `{k}` | {len(v)} | {sum(v):.1f} | {100 * sum(v) / tot:.1f}% |"
            for k, v in sorted(per.items(), key=lambda kv: -sum(kv[1]))]


def write_traffic(log_dir):
    """profiles/traffic.json and traffic.md from the per-workload ncu logs."""
    kernels, md = {}, []
    for w, (bucket, kre, srcs) in TRAFFIC_CAPTURE.items():
        path = os.path.join(log_dir, f"traffic_{w}.csv")
        if not os.path.exists(path):
            continue
        rows = _ncu_rows(path)
        if not rows:
            continue
        rd = [m["dram__bytes_read.sum"] for _, _, m in rows]
        wr = [m["dram__bytes_write.sum"] for _, _, m in rows]
        us = [m["gpu__time_duration.sum"] / 1e3 for _, _, m in rows]
        tot = float(np.median(np.array(rd) + np.array(wr)))
        kernels[f"{w}:{bucket}"] = {"bytes_per_launch": tot, "launches_used": len(rows),
                                    "ncu_kernels": [kre], "sources": sorted(srcs)}
        md.append(f"| {w} | {bucket} | `{rows[0][1].split('(')[0].replace('void ', '')}` | "
                  f"{len(rows)} | {np.median(rd) / 1e6:.1f} | {np.median(wr) / 1e6:.2f} | "
                  f"{np.median(us):.1f} |")
    out = {"how": "ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,"
                  "dram__bytes_write.sum --clock-control none --kernel-name-base demangled "
                  "-k regex:<kernel> -s 3 -c 3 on the bench command of each workload; "
                  "bytes_per_launch = median over the captured launches of DRAM read + write; "
                  "an entry holds while its source files match",
           "file_sha256": source_digests(), "csrc_sha256": csrc_digest(), "kernels": kernels}
    with open(os.path.join(ROOT, "profiles", "traffic.json"), "w") as f:
        json.dump(out, f, indent=1)
    return md


sys.path.insert(0, ROOT)

METRIC = "draft-attn blocks/s per layer; achieved HBM GB/s (or tensor util) vs GB300 peak"
UNIT = "blocks/s"
L2_FLUSH_BYTES = 512 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="serving_b32")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="bound on the timed oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true",
                    help="skip the nvidia-smi sampler (for profiler runs)")
    ap.add_argument("--ncu-traffic", metavar="DIR", default=None,
                    help="no GPU work: write profiles/traffic.json from the ncu logs in DIR "
                         "and print the table rows")
    ap.add_argument("--ncu-launches", metavar="CSV", default=None,
                    help="no GPU work: print the per-kernel table of an ncu launch list")
    ap.add_argument("--read-stream", action="store_true",
                    help="measurement aid instead of the bench: time TMA read passes over "
                         "the workload's fc weight matrix (one JSON line per launch shape)")
    return ap.parse_args()


# --------------------------------------------------------------------------
# peaks and clocks
# --------------------------------------------------------------------------
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [s for t, s in self.samples if t0 - 0.05 <= t <= t1 + 0.05]
        if not rows and self.samples:  # region shorter than a sample period
            rows = [min(self.samples, key=lambda x: abs(x[0] - (t0 + t1) / 2))[1]]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[2:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
class PackedIO:
    """A step's inputs packed into one pinned host buffer and one device
    buffer (256-byte aligned slots of fixed offsets), so the step's
    host-to-device transfer is one copy, as a server that receives a request
    into one pinned region would make it."""

    def __init__(self, slots, device):
        import torch
        self.off, self.dt, off = {}, {}, 0
        for name, (numel, dt) in slots.items():
            self.off[name], self.dt[name] = off, dt
            off += (numel * torch.empty(0, dtype=dt).element_size() + 255) // 256 * 256
        self.host = torch.empty(max(off, 256), dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(max(off, 256), dtype=torch.uint8, device=device)
        self.used = 0
        self.read = None  # event: the last upload from this buffer has run

    def stage(self, tensors):
        """Host copies of the step's inputs into the pinned buffer (before the
        timed region), once the previous upload from it has been read."""
        if self.read is not None:
            self.read.synchronize()
        end = 0
        for name, t in tensors.items():
            b = t.contiguous().view(-1).view(torch_uint8())
            o = self.off[name]
            self.host[o:o + b.numel()].copy_(b)
            end = max(end, o + b.numel())
        self.used = end

    def upload(self, record=True):
        import torch
        self.dev[:self.used].copy_(self.host[:self.used], non_blocking=True)
        if record:
            self.read = torch.cuda.Event()
            self.read.record()

    def view(self, name, shape):
        import torch
        n = int(np.prod(shape)) * torch.empty(0, dtype=self.dt[name]).element_size()
        o = self.off[name]
        return self.dev[o:o + n].view(self.dt[name]).view(*shape)


def torch_uint8():
    import torch
    return torch.uint8


class ServingWorkload:
    """Inference steps of one layer: ctx_project -> forward -> crop."""

    def __init__(self, sp, seed, device, n_steps):
        import torch
        from block_diffusion_draft_gb300 import DFlashAttention, DraftCache
        from block_diffusion_draft_gb300 import workloads as W

        self.sp, self.dev = sp, device
        self.W = W
        w = W.weights(sp, seed)
        self.attn = DFlashAttention(w, hidden=sp.hidden, n_heads=sp.n_heads,
                                    n_kv_heads=sp.n_kv_heads, head_dim=sp.head_dim,
                                    n_target_layers=sp.n_target_layers,
                                    rms_eps=sp.rms_eps, rope_theta=sp.rope_theta,
                                    sliding_window=sp.sliding_window,
                                    max_position=sp.max_position, device=device)
        del w
        self.mlp = None
        if sp.intermediate > 0:
            from block_diffusion_draft_gb300 import DecoderMLP
            self.mlp = DecoderMLP(W.mlp_weights(sp, seed, sp.intermediate), sp.hidden,
                                  sp.intermediate, sp.rms_eps, device=device)
        self.fixed = sp.prefill > 0  # every step identical (crop back each time)
        sched = W.serving_schedule(sp, seed, steps=1 if self.fixed else n_steps)
        self.sched = sched
        B, q = sp.batch, sp.block_size
        pre = sched.prefill
        grow = 0 if self.fixed else sum(max(s.n_ctx) for s in sched.steps)
        self.cap = max(pre) + grow + 2 * (q + sp.block_size) + 16
        self.paged = sp.page_size > 0
        if self.paged:
            # every sequence's pages for the whole run, from a shuffled free
            # list; one block table serves every step (entries past a
            # sequence's end are not read)
            from block_diffusion_draft_gb300 import PagedCache
            P = sp.page_size
            per_seq = (self.cap + P - 1) // P
            free = np.random.default_rng(seed + 7).permutation(B * per_seq)
            self.pages = free.reshape(B, per_seq).astype(np.int32)
            self.cache = PagedCache(self.attn, B * per_seq, P)
            self.bt_h = torch.from_numpy(self.pages.copy())
            self.bt = self.bt_h.to(device)
        else:
            self.cache = DraftCache(self.attn, B, self.cap)
        # prefill: context rows at positions 0.., one block, then crop
        th = torch.cat([W.hidden_rows(sp, seed, "hidden", 1000, b, pre[b]) for b in range(B)])
        nz = torch.stack([W.hidden_rows(sp, seed, "noise", 1000, b, q) for b in range(B)])
        pos = torch.cat([W.window_positions(0, pre[b], q) for b in range(B)])
        if self.paged:
            sl = self._slots([0] * B, [pre[b] + q for b in range(B)])
            self.attn.forward_paged(self.cache, nz.to(device), th.to(device), pre, [0] * B,
                                    pos.to(device), sl.to(device), self.bt)
        else:
            self.attn.forward(self.cache, nz.to(device), th.to(device), pre, pos.to(device))
            self.cache.crop(pre)
        del th
        torch.cuda.synchronize(device)
        # per-step inputs (host copies kept pinned for the end-to-end leg)
        self.steps = []
        L = list(pre)
        for s, st in enumerate(sched.steps):
            n_ctx = st.n_ctx
            x = torch.cat([W.target_layer_rows(sp, seed, s, b, n_ctx[b]) for b in range(B)])
            nz = torch.stack([W.hidden_rows(sp, seed, "noise", s, b, q) for b in range(B)])
            pos = torch.cat([W.window_positions(L[b], n_ctx[b], q) for b in range(B)])
            keep = [L[b] + n_ctx[b] for b in range(B)] if not self.fixed else list(pre)
            st = dict(n_ctx=n_ctx, keep=keep, len_before=list(L), x_h=x, nz_h=nz, pos_h=pos,
                      x=x.to(device), nz=nz.to(device), pos=pos.to(device))
            if self.paged:
                sl = self._slots(L, [n_ctx[b] + q for b in range(B)])
                st.update(sl_h=sl, sl=sl.to(device))
            self.steps.append(st)
            if not self.fixed:
                L = keep
        rows = max(int(sum(st["n_ctx"])) for st in self.steps)
        # the context rows vary most in size from step to step: their slot
        # goes last so a step uploads only the bytes it uses
        self.io_keys = ("nz", "pos") + (("sl",) if self.paged else ()) + ("x",)
        slots = {}
        if self.paged:
            slots["bt"] = (self.bt_h.numel(), self.bt_h.dtype)
        slots.update({k: (max(st[k + "_h"].numel() for st in self.steps),
                          self.steps[0][k + "_h"].dtype) for k in self.io_keys})
        # two upload buffers taken in turn, so the host stages step i + 1
        # while step i may still be copying (eager steps); graph-replayed
        # (identical) steps use the first
        self.pios = [PackedIO(slots, device), PackedIO(slots, device)]
        # size every scratch buffer for the largest step up front, as a server
        # does at start-up (a buffer that grows mid-run synchronises the device)
        self.attn.reserve(B, B * q + rows, self.cap)
        self.th_buf = torch.empty(rows, sp.hidden, dtype=torch.bfloat16, device=device)
        self.out_buf = torch.empty(B, q, sp.hidden, dtype=torch.bfloat16, device=device)
        self.res_buf = torch.empty(B, q, sp.hidden, dtype=torch.bfloat16, device=device)
        self.out_h = torch.empty(B, q, sp.hidden, dtype=torch.bfloat16).pin_memory()
        self.blocks_per_step = B

    def _slots(self, start, count):
        """Paged cache: slots of rows start[b] .. start[b] + count[b] - 1 of
        every sequence, sequence-major (the order of the positions)."""
        import torch
        P = self.sp.page_size
        out = []
        for b, (s0, n) in enumerate(zip(start, count)):
            k = np.arange(s0, s0 + n)
            out.append(self.pages[b][k // P] * P + k % P)
        return torch.from_numpy(np.concatenate(out).astype(np.int32))

    def _inputs(self, i):
        return self.steps[i % len(self.steps)]

    def reset(self):
        """Back to the post-prefill cache state (fixed workloads stay there;
        a paged cache's lengths are the schedule's)."""
        if not self.fixed and not self.paged:
            self.cache.crop(self.sched.prefill)

    def step(self, i, inputs=None):
        """Step i from its resident device inputs (or from `inputs`, the same
        tensors as views into the packed upload buffer)."""
        st = self._inputs(i)
        d = st if inputs is None else inputs
        bt = None
        if self.paged:
            bt = self.bt if inputs is None else inputs["bt"]
        n = int(sum(st["n_ctx"]))
        th = self.th_buf[:n]
        self.attn.ctx_project(d["x"], out=th)
        if self.paged:
            self.attn.forward_paged(self.cache, d["nz"], th, st["n_ctx"], st["len_before"],
                                    d["pos"], d["sl"], bt, out=self.out_buf)
            return
        if self.mlp is None:
            self.attn.forward(self.cache, d["nz"], th, st["n_ctx"], d["pos"],
                              out=self.out_buf)
        else:
            self.mlp.layer_forward_into(self.attn, self.cache, d["nz"], None, th,
                                        st["n_ctx"], d["pos"], self.out_buf, self.res_buf)
        self.cache.crop(st["keep"])

    def stage_e2e(self, i):
        """Put step i's host inputs into the pinned upload buffer (a server
        receives each step's inputs into the same pinned memory; this runs
        before the timed region)."""
        st = self._inputs(i)
        t = {k: st[k + "_h"] for k in self.io_keys}
        if self.paged:
            t["bt"] = self.bt_h
        self._pio(i).stage(t)

    def _pio(self, i):
        return self.pios[0 if self.fixed else i % 2]

    def step_e2e(self, i):
        """The same step from the pinned upload buffer (one copy), result
        read back to host."""
        st = self._inputs(i)
        pio = self._pio(i)
        pio.upload(record=not self.fixed)
        views = {k: pio.view(k, tuple(st[k + "_h"].shape)) for k in self.io_keys}
        if self.paged:
            views["bt"] = pio.view("bt", tuple(self.bt_h.shape))
        self.step(i, views)
        self.out_h.copy_(self.out_buf, non_blocking=True)

    def io_bytes(self, i):
        st = self._inputs(i)
        h2d = sum(st[k + "_h"].numel() * st[k + "_h"].element_size() for k in self.io_keys)
        if self.paged:
            h2d += self.bt_h.numel() * self.bt_h.element_size()
        return h2d, self.out_h.numel() * self.out_h.element_size()

    def kernel_bytes(self, i):
        """Algorithmic HBM bytes of each kernel of step i (each operand read
        once, each result written once)."""
        sp, st = self.sp, self._inputs(i)
        H, d, nq, nkv, q, B = sp.hidden, sp.head_dim, sp.n_heads, sp.n_kv_heads, \
            sp.block_size, sp.batch
        n = int(sum(st["n_ctx"]))
        K = sp.n_target_layers * H
        keys = 0
        for b in range(B):
            ln = st["len_before"][b] + st["n_ctx"][b] + q
            lo = max(0, ln - q - sp.sliding_window + 1) if sp.sliding_window else 0
            keys += ln - lo
        return {
            "fc": H * K * 2 + n * K * 2 + n * H * 4,
            "norm": n * H * 4 + n * H * 2,
            "qkv": (nq + 2 * nkv) * d * H * 2 + (B * q + n) * H * 2
                   + B * q * nq * d * 2 + (B * q + n) * 2 * nkv * d * 2,
            "attn": keys * nkv * d * 2 * 2 + 2 * B * q * nq * d * 2
                    + (keys // sp.page_size * 4 if sp.page_size else 0),
            "o_proj": H * nq * d * 2 + B * q * nq * d * 2 + B * q * H * 2,
            # two add+norm passes (read 2 rows, write 2) and the SwiGLU MLP
            "mlp": (2 * 4 * B * q * H * 2 + 3 * sp.intermediate * H * 2
                    + B * q * (H + 2 * sp.intermediate + H) * 2) if sp.intermediate else 0,
        }

    def kernel_flops(self, i):
        return {}

    def config(self):
        return spec_config(self.sp)


class PackedWorkload:
    """Packed training layout forward (no cache): one call per step."""

    def __init__(self, sp, seed, device, n_steps):
        import torch
        from block_diffusion_draft_gb300 import DFlashAttention
        from block_diffusion_draft_gb300 import workloads as W

        self.sp, self.dev = sp, device
        w = W.weights(sp, seed, with_fc=False)
        self.attn = DFlashAttention(w, hidden=sp.hidden, n_heads=sp.n_heads,
                                    n_kv_heads=sp.n_kv_heads, head_dim=sp.head_dim,
                                    n_target_layers=0, rms_eps=sp.rms_eps,
                                    rope_theta=sp.rope_theta,
                                    max_position=sp.max_position, device=device)
        B, S, nb, bs = sp.batch, sp.seq, sp.n_blocks, sp.block_size
        th = torch.stack([W.hidden_rows(sp, seed, "hidden", 0, b, S) for b in range(B)])
        nz = torch.stack([W.hidden_rows(sp, seed, "noise", 0, b, nb * bs) for b in range(B)])
        an = W.anchors(sp, seed)
        self.th_h, self.nz_h, self.an_h = th.pin_memory(), nz.pin_memory(), an.pin_memory()
        self.th, self.nz, self.an = th.to(device), nz.to(device), an.to(device)
        self.out = torch.empty_like(self.nz)
        self.out_h = torch.empty_like(self.nz_h).pin_memory()
        self.blocks_per_step = B * nb
        self.anchors_np = an.numpy()
        self.fixed = True
        self.pio = PackedIO({"th": (th.numel(), th.dtype), "nz": (nz.numel(), nz.dtype),
                             "an": (an.numel(), an.dtype)}, device)

    def reset(self):
        pass

    def step(self, i, inputs=None):
        nz, th, an = (self.nz, self.th, self.an) if inputs is None else \
            (inputs["nz"], inputs["th"], inputs["an"])
        self.attn.forward_packed(nz, th, an, self.sp.block_size, out=self.out)

    def stage_e2e(self, i):
        self.pio.stage({"th": self.th_h, "nz": self.nz_h, "an": self.an_h})

    def step_e2e(self, i):
        self.pio.upload(record=False)
        self.step(i, {k: self.pio.view(k, tuple(h.shape))
                      for k, h in (("th", self.th_h), ("nz", self.nz_h), ("an", self.an_h))})
        self.out_h.copy_(self.out, non_blocking=True)

    def io_bytes(self, i):
        h2d = sum(t.numel() * t.element_size() for t in (self.th_h, self.nz_h, self.an_h))
        return h2d, self.out_h.numel() * self.out_h.element_size()

    def kernel_flops(self, i):
        sp = self.sp
        H, d, nq, nkv = sp.hidden, sp.head_dim, sp.n_heads, sp.n_kv_heads
        B, S, nb, bs = sp.batch, sp.seq, sp.n_blocks, sp.block_size
        rq, rc = B * nb * bs, B * S
        attn = 0
        for b in range(B):
            for a in self.anchors_np[b]:
                attn += 4 * nq * bs * d * (min(int(a), S) + bs)
        return {"qkv": 2 * rq * H * (nq + 2 * nkv) * d + 2 * rc * H * 2 * nkv * d,
                "attn": attn, "o_proj": 2 * rq * nq * d * H}

    def kernel_bytes(self, i):
        return {}

    def config(self):
        return spec_config(self.sp)


class PackedBwdWorkload:
    """Attention core of the packed training layout, forward (with the
    log-sum-exp) then backward (dQ, dK, dV), on Q/K/V/dO already resident."""

    def __init__(self, sp, seed, device, n_steps):
        import torch
        from block_diffusion_draft_gb300 import DFlashAttention
        from block_diffusion_draft_gb300 import workloads as W

        self.sp, self.dev = sp, device
        w = W.weights(sp, seed, with_fc=False)
        self.attn = DFlashAttention(w, hidden=sp.hidden, n_heads=sp.n_heads,
                                    n_kv_heads=sp.n_kv_heads, head_dim=sp.head_dim,
                                    n_target_layers=0, rms_eps=sp.rms_eps,
                                    rope_theta=sp.rope_theta,
                                    max_position=sp.max_position, device=device)
        del w
        x = W.core_tensors(sp, seed)
        an = W.anchors(sp, seed)
        self.h = {k: t.pin_memory() for k, t in x.items()}
        self.h["anchors"] = an.pin_memory()
        self.d = {k: t.to(device) for k, t in self.h.items()}
        self.out = torch.empty_like(self.d["q"])
        self.grads_h = {k: torch.empty_like(self.h[k]).pin_memory() for k in ("q", "k", "v")}
        self.blocks_per_step = sp.batch * sp.n_blocks
        self.anchors_np = an.numpy()
        self.fixed = True
        self.last = None
        self.pio = PackedIO({k: (t.numel(), t.dtype) for k, t in self.h.items()}, device)

    def reset(self):
        pass

    def step(self, i, inputs=None):
        d, sp = (self.d if inputs is None else inputs), self.sp
        out, lse = self.attn.packed_core(d["q"], d["k"], d["v"], d["anchors"], sp.seq,
                                         sp.block_size)
        self.last = self.attn.packed_core_backward(d["q"], d["k"], d["v"], out, lse,
                                                   d["d_out"], d["anchors"], sp.seq,
                                                   sp.block_size)

    def stage_e2e(self, i):
        self.pio.stage(self.h)

    def step_e2e(self, i):
        self.pio.upload(record=False)
        self.step(i, {k: self.pio.view(k, tuple(t.shape)) for k, t in self.h.items()})
        for g, k in zip(self.last, ("q", "k", "v")):
            self.grads_h[k].copy_(g, non_blocking=True)

    def io_bytes(self, i):
        h2d = sum(t.numel() * t.element_size() for t in self.h.values())
        return h2d, sum(t.numel() * t.element_size() for t in self.grads_h.values())

    def kernel_flops(self, i):
        """Forward attention 4 d flops per visible (query, key) pair; the
        backward's five products (S, dP, dV, dQ, dK) 10 d per pair (masked
        work and the recomputation of S and dP by the dQ CTAs not counted)."""
        sp = self.sp
        pairs = 0
        for b in range(sp.batch):
            for a in self.anchors_np[b]:
                pairs += sp.n_heads * sp.block_size * (min(int(a), sp.seq) + sp.block_size)
        return {"attn": 4 * sp.head_dim * pairs, "bwd": 10 * sp.head_dim * pairs}

    def kernel_bytes(self, i):
        return {}

    def config(self):
        return spec_config(self.sp)


class StackWorkload:
    """A stack of draft layers fed by one projected context per step:
    ctx_project (layer 0's fc) -> the context K/V of every layer from one
    grouped projection -> each layer's forward with no context rows -> crop.
    `per_layer_step` runs the same step with each layer's forward projecting
    the context rows itself (the plain schedule), timed for comparison."""

    def __init__(self, sp, seed, device, n_steps):
        import torch
        from block_diffusion_draft_gb300 import DFlashAttention, DraftCache, KVGroup
        from block_diffusion_draft_gb300 import workloads as W

        self.sp, self.dev, self.W = sp, device, W
        L, B, q, pre, n = sp.layers, sp.batch, sp.block_size, sp.prefill, sp.n_new
        self.layers, self.caches = [], []
        self.cap = pre + n + 2 * q + 16
        for l in range(L):
            w = W.weights(sp, seed, layer=l, with_fc=l == 0)
            a = DFlashAttention(w, hidden=sp.hidden, n_heads=sp.n_heads,
                                n_kv_heads=sp.n_kv_heads, head_dim=sp.head_dim,
                                n_target_layers=sp.n_target_layers if l == 0 else 0,
                                rms_eps=sp.rms_eps, rope_theta=sp.rope_theta,
                                sliding_window=sp.sliding_window,
                                max_position=sp.max_position, device=device)
            del w
            c = DraftCache(a, B, self.cap)
            th = torch.cat([W.hidden_rows(sp, seed, "hidden", 1000, b, pre) for b in range(B)])
            nz = torch.stack([W.hidden_rows(sp, seed, "noise", 1000 + l, b, q) for b in range(B)])
            pos = torch.cat([W.window_positions(0, pre, q) for b in range(B)])
            a.forward(c, nz.to(device), th.to(device), [pre] * B, pos.to(device))
            c.crop([pre] * B)
            a.reserve(B, B * q + B * n, self.cap)
            self.layers.append(a)
            self.caches.append(c)
        self.attn = self.layers[0]
        self.group = KVGroup(self.layers)
        torch.cuda.synchronize(device)
        self.x_h = torch.cat([W.target_layer_rows(sp, seed, 0, b, n) for b in range(B)])
        self.nz_h = torch.stack([torch.stack([W.hidden_rows(sp, seed, "noise", l, b, q)
                                              for b in range(B)]) for l in range(L)])
        self.pos_ctx_h = torch.cat([torch.arange(pre, pre + n, dtype=torch.int32)
                                    for b in range(B)])
        self.pos_blk_h = torch.cat([W.window_positions(pre + n, 0, q) for b in range(B)])
        self.pos_full_h = torch.cat([W.window_positions(pre, n, q) for b in range(B)])
        self.x, self.nz = self.x_h.to(device), self.nz_h.to(device)
        self.pos_ctx, self.pos_blk = self.pos_ctx_h.to(device), self.pos_blk_h.to(device)
        self.pos_full = self.pos_full_h.to(device)
        for t in ("x_h", "nz_h", "pos_ctx_h", "pos_blk_h", "pos_full_h"):
            setattr(self, t, getattr(self, t).pin_memory())
        self.th = torch.empty(B * n, sp.hidden, dtype=torch.bfloat16, device=device)
        self.out = torch.empty(L, B, q, sp.hidden, dtype=torch.bfloat16, device=device)
        self.out_h = torch.empty(L, B, q, sp.hidden, dtype=torch.bfloat16).pin_memory()
        self.fixed = True
        self.blocks_per_step = B * L  # blocks per layer-step summed over the layers
        self.io_h = {"x": self.x_h, "nz": self.nz_h, "pos_ctx": self.pos_ctx_h,
                     "pos_blk": self.pos_blk_h}
        self.pio = PackedIO({k: (t.numel(), t.dtype) for k, t in self.io_h.items()}, device)

    def handles(self):
        return self.layers

    def reset(self):
        pass

    def step(self, i=0, inputs=None):
        sp, B, n = self.sp, self.sp.batch, self.sp.n_new
        x, nz, pos_ctx, pos_blk = (self.x, self.nz, self.pos_ctx, self.pos_blk) \
            if inputs is None else (inputs["x"], inputs["nz"], inputs["pos_ctx"],
                                    inputs["pos_blk"])
        self.attn.ctx_project(x, out=self.th)
        self.group.append(self.caches, self.th, [n] * B, pos_ctx)
        for l, (a, c) in enumerate(zip(self.layers, self.caches)):
            a.forward(c, nz[l], None, [0] * B, pos_blk, out=self.out[l])
        for c in self.caches:
            c.crop([sp.prefill] * B)

    def per_layer_step(self, i=0):
        sp, B, n = self.sp, self.sp.batch, self.sp.n_new
        self.attn.ctx_project(self.x, out=self.th)
        for l, (a, c) in enumerate(zip(self.layers, self.caches)):
            a.forward(c, self.nz[l], self.th, [n] * B, self.pos_full, out=self.out[l])
        for c in self.caches:
            c.crop([sp.prefill] * B)

    def stage_e2e(self, i):
        self.pio.stage(self.io_h)

    def step_e2e(self, i):
        self.pio.upload(record=False)
        self.step(i, {k: self.pio.view(k, tuple(t.shape)) for k, t in self.io_h.items()})
        self.out_h.copy_(self.out, non_blocking=True)

    def io_bytes(self, i):
        h2d = sum(t.numel() * t.element_size()
                  for t in (self.x_h, self.nz_h, self.pos_ctx_h, self.pos_blk_h))
        return h2d, self.out_h.numel() * self.out_h.element_size()

    def kernel_bytes(self, i):
        """Algorithmic HBM bytes per trace bucket of one grouped step."""
        sp = self.sp
        H, d, nq, nkv, q, B, L = (sp.hidden, sp.head_dim, sp.n_heads, sp.n_kv_heads,
                                  sp.block_size, sp.batch, sp.layers)
        n = B * sp.n_new
        K = sp.n_target_layers * H
        keys = B * (sp.prefill + sp.n_new + q)
        return {
            "fc": H * K * 2 + n * K * 2 + n * H * 4,
            "norm": n * H * 4 + n * H * 2,
            # grouped K/V projection of the context rows, then each layer's
            # Q/K/V projection of its block rows
            "qkv": L * 2 * nkv * d * H * 2 + n * H * 2 + L * n * 2 * nkv * d * 2
                   + L * ((nq + 2 * nkv) * d * H * 2 + B * q * H * 2 + B * q * (nq + 2 * nkv) * d * 2),
            "attn": L * (keys * nkv * d * 2 * 2 + 2 * B * q * nq * d * 2),
            "o_proj": L * (H * nq * d * 2 + B * q * nq * d * 2 + B * q * H * 2),
        }

    def kernel_flops(self, i):
        return {}

    def config(self):
        return spec_config(self.sp)


def spec_config(sp):
    """The `config` of a workload's bench line (both arms)."""
    if sp.seq > 0:
        return {"workload": sp.name, "batch": sp.batch, "seq": sp.seq,
                "n_blocks": sp.n_blocks, "block_size": sp.block_size,
                "hidden": sp.hidden, "heads": f"{sp.n_heads}/{sp.n_kv_heads}",
                "head_dim": sp.head_dim,
                "step": ("packed attention core forward (with log-sum-exp) + backward "
                         "(dQ, dK, dV)") if sp.backward else "forward_packed",
                "l2": "flushed (512 MiB write) before every timed step"}
    fixed = sp.prefill > 0
    extra = {"layers": sp.layers,
             "step": "ctx_project + grouped context K/V of all layers + per-layer forward "
                     "(no context rows) + crop"} if sp.layers > 1 else {}
    if sp.intermediate > 0:
        extra = {"intermediate": sp.intermediate,
                 "step": "ctx_project + decoder layer (input norm, attention, residual, "
                         "post norm, SwiGLU MLP) + crop"}
    return {"workload": sp.name, "batch": sp.batch, "hidden": sp.hidden,
            "heads": f"{sp.n_heads}/{sp.n_kv_heads}", "head_dim": sp.head_dim,
            "block_size": sp.block_size, "fc_in": sp.n_target_layers * sp.hidden,
            "new_ctx_rows": sp.n_new if fixed else "U{1..16}",
            "cached_ctx": sp.prefill if fixed else f"U[{sp.prefill_lo},{sp.prefill_hi}]",
            "sliding_window": sp.sliding_window,
            "step": "ctx_project + forward + crop",
            **({"cache": f"paged, {sp.page_size}-row pages in shuffled order",
                "step": "ctx_project + forward over the paged cache (slot mapping and "
                        "block table per step)"} if sp.page_size else {}),
            "l2": "flushed (512 MiB write) before every timed step", **extra}


def make_workload(name, seed, device, n_steps):
    from block_diffusion_draft_gb300 import workloads as W
    sp = W.SPECS[name]
    if sp.layers > 1:
        return StackWorkload(sp, seed, device, n_steps)
    if sp.backward:
        return PackedBwdWorkload(sp, seed, device, n_steps)
    if sp.seq > 0:
        return PackedWorkload(sp, seed, device, n_steps)
    return ServingWorkload(sp, seed, device, n_steps)


# --------------------------------------------------------------------------
# CPU oracle baseline
# --------------------------------------------------------------------------
class OracleRunner:
    """The fp64 oracle on a bounded sample of the same workload.

    Serving workloads: one sequence of the batch (sequences are independent),
    prefilled once, then one oracle step = ctx_project + forward + crop of that
    sequence.  Packed workload: one oracle step = forward_packed of sequence 0
    over 8 sampled blocks (the oracle recomputes the sequence's context K/V in
    every call, as it stands)."""

    def __init__(self, name, seed):
        import torch
        from block_diffusion_draft_gb300 import workloads as W
        from oracle import dflash_oracle as O

        self.O, self.W = O, W
        self.sp = sp = W.SPECS[name]
        f64 = lambda t: t.to(torch.float64).numpy()
        w = W.weights(sp, seed, with_fc=sp.seq == 0)
        self.cfg = O.LayerConfig(hidden=sp.hidden, n_heads=sp.n_heads,
                                 n_kv_heads=sp.n_kv_heads, head_dim=sp.head_dim,
                                 rms_eps=sp.rms_eps, rope_theta=sp.rope_theta,
                                 sliding_window=sp.sliding_window,
                                 n_target_layers=sp.n_target_layers if sp.seq == 0 else 0)
        self.lw = O.LayerWeights(
            *(f64(w[k]) for k in ("wq", "wk", "wv", "wo", "q_norm", "k_norm")),
            fc=f64(w["fc"]) if "fc" in w else None,
            hidden_norm=f64(w["hidden_norm"]) if "fc" in w else None)
        del w
        q = sp.block_size
        if sp.backward:
            # one (sequence, kv head) group: its query heads over all blocks
            x = W.core_tensors(sp, seed)
            g = sp.n_heads // sp.n_kv_heads
            self.core_cfg = O.LayerConfig(hidden=sp.hidden, n_heads=g, n_kv_heads=1,
                                          head_dim=sp.head_dim, rms_eps=sp.rms_eps,
                                          rope_theta=sp.rope_theta, n_target_layers=0)
            self.cq = f64(x["q"][0, :, :g]).transpose(1, 0, 2)
            self.ck = f64(x["k"][0, :1])
            self.cv = f64(x["v"][0, :1])
            self.cdo = f64(x["d_out"][0, :, :g]).transpose(1, 0, 2)
            self.an = W.anchors(sp, seed).numpy()[0]
            self.blocks_per_step = sp.n_blocks / sp.n_kv_heads
            self.sample = (f"packed core forward + backward of sequence 0, kv head 0 ({g} query "
                           f"heads, {sp.n_blocks} blocks) per step = 1/{sp.n_kv_heads} of a "
                           "sequence's blocks")
        elif sp.seq > 0:
            self.an = W.anchors(sp, seed).numpy()[:1]
            self.th = f64(W.hidden_rows(sp, seed, "hidden", 0, 0, sp.seq))[None]
            self.nz = f64(W.hidden_rows(sp, seed, "noise", 0, 0, sp.n_blocks * q))[None]
            self.blocks = list(range(sp.n_blocks - 1, -1, -sp.n_blocks // 8))[:8]
            self.blocks_per_step = len(self.blocks)
            self.sample = (f"forward_packed of sequence 0 over {len(self.blocks)} blocks "
                           "per step (context K/V recomputed per call)")
        else:
            sched = W.serving_schedule(sp, seed, steps=1)
            self.pre = pre = sched.prefill[0]
            self.cache = O.DraftCache(sp.n_kv_heads, sp.head_dim, 1)
            th = f64(W.hidden_rows(sp, seed, "hidden", 1000, 0, pre))
            nz = f64(W.hidden_rows(sp, seed, "noise", 1000, 0, q))
            O.forward(self.cfg, self.lw, self.cache, nz[None], [th],
                      [W.window_positions(0, pre, q).numpy()])
            self.cache.crop([pre])
            n = sched.steps[0].n_ctx[0]
            self.x = f64(W.target_layer_rows(sp, seed, 0, 0, n))
            self.nzs = f64(W.hidden_rows(sp, seed, "noise", 0, 0, q))[None]
            self.pos = W.window_positions(pre, n, q).numpy()
            self.blocks_per_step = 1
            self.sample = ("ctx_project + forward + crop of one sequence per step "
                           f"({pre} cached rows, {n} new, block {q})")
            self.om = None
            if sp.intermediate > 0:
                mw = W.mlp_weights(sp, seed, sp.intermediate)
                self.om = O.MlpWeights(*(f64(mw[k]) for k in ("gate", "up", "down",
                                                               "input_norm", "post_norm")))
                self.sample = ("ctx_project + decoder layer + crop of one sequence per step "
                               f"({pre} cached rows, {n} new, block {q}, MLP {sp.intermediate})")
            # layer stack: the other layers (own weights and caches), each step
            # their per-layer forward with the context rows (the definition)
            self.more = []
            for l in range(1, sp.layers):
                wl_ = W.weights(sp, seed, layer=l, with_fc=False)
                lw = O.LayerWeights(*(f64(wl_[k]) for k in ("wq", "wk", "wv", "wo", "q_norm",
                                                             "k_norm")))
                c = O.DraftCache(sp.n_kv_heads, sp.head_dim, 1)
                O.forward(self.cfg, lw, c, nz[None], [th], [W.window_positions(0, pre, q).numpy()])
                c.crop([pre])
                self.more.append((lw, c, f64(W.hidden_rows(sp, seed, "noise", l, 0, q))[None]))
            if sp.layers > 1:
                self.blocks_per_step = sp.layers
                self.sample = (f"ctx_project + {sp.layers} per-layer forwards + crop of one "
                               f"sequence per step ({pre} cached rows, {n} new, block {q})")

    def step(self):
        O, sp = self.O, self.sp
        if sp.backward:
            O.packed_core(self.core_cfg, self.cq, self.ck, self.cv, self.an, sp.seq,
                          sp.block_size)
            O.packed_core_backward(self.core_cfg, self.cq, self.ck, self.cv, self.an, sp.seq,
                                   sp.block_size, self.cdo)
        elif sp.seq > 0:
            O.forward_packed(self.cfg, self.lw, self.nz, self.th, self.an,
                             sp.block_size, seqs=[0], blocks=self.blocks)
        else:
            t = O.ctx_project(self.cfg, self.lw, self.x)
            if self.om is None:
                O.forward(self.cfg, self.lw, self.cache, self.nzs, [t], [self.pos])
            else:
                O.decoder_layer(self.cfg, self.lw, self.om, self.cache, self.nzs, None, [t],
                                [self.pos])
            self.cache.crop([self.pre])
            for lw, c, nzs in self.more:
                O.forward(self.cfg, lw, c, nzs, [t], [self.pos])
                c.crop([self.pre])

    def time(self, steps, budget_s):
        t0 = time.perf_counter()
        n = 0
        while n < steps:
            self.step()
            n += 1
            if time.perf_counter() - t0 > budget_s:
                break
        dt = time.perf_counter() - t0
        return n, dt


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_baseline(name, seed, budget_s):
    r = OracleRunner(name, seed)
    r.step()  # warm-up
    n, dt = r.time(10 ** 6, budget_s)
    return {"value": n * r.blocks_per_step / dt, "unit": UNIT, "cores": os.cpu_count(),
            "cpu_model": host_cpu_model(), "kind": "oracle",
            "sample": f"{n} oracle steps in {dt:.1f} s: {r.sample}; fp64 numpy, BLAS "
                      "threads = all host cores"}


# --------------------------------------------------------------------------
# replicas (one process per GPU; sequences are independent, no collective on
# the data path: only the timing is reduced)
# --------------------------------------------------------------------------
def rank_env():
    """(world size, rank, local rank) from the launcher's environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica_seed(seed, rank, world):
    """Each replica draws its own sequences (weak scaling)."""
    return seed + (rank if world > 1 else 0)


def max_over_ranks(x, dist, device):
    """The slowest rank's value (the job finishes with it)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, units_per_step, ms):
    """Whole-job throughput: the units all ranks processed per second of the
    slowest rank's step time."""
    return world * units_per_step / (ms / 1000.0)


# --------------------------------------------------------------------------
# main
# --------------------------------------------------------------------------
def read_stream(args):
    """The rate at which TMA alone reads the workload's fc weight matrix
    ([hidden, n_target_layers * hidden] bf16, 168 MB for the 8B shape) in the
    boxes the GEMMs read weights in, for several CTA counts and box counts in
    flight per CTA: the read-side ceiling of the weight-streaming GEMMs at
    this size.  Each pass is one launch timed with CUDA events on the
    launching stream after a 512 MiB write (L2 flush); the median of the
    timed passes is reported, with the clocks sampled meanwhile."""
    import torch
    import __graft_entry__ as G
    G.build()
    from block_diffusion_draft_gb300 import DFlashAttention
    from block_diffusion_draft_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sp = W.SPECS[args.workload]
    w = W.weights(sp, args.seed)
    attn = DFlashAttention(w, hidden=sp.hidden, n_heads=sp.n_heads, n_kv_heads=sp.n_kv_heads,
                           head_dim=sp.head_dim, n_target_layers=sp.n_target_layers,
                           rms_eps=sp.rms_eps, rope_theta=sp.rope_theta,
                           sliding_window=sp.sliding_window, max_position=sp.max_position,
                           device=dev)
    m = w["fc"].to(dev)
    del w
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    nbytes = m.numel() * m.element_size()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = None if args.no_clocks else ClockSampler(0)
    shapes = [(c, s) for c in (64, 96, 128, sms, 2 * sms) for s in (2, 3, 4, 6, 8, 12)
              if not (c > sms and s > 6)]
    n_warm, n_time = max(1, args.warmup), 10
    res = []
    t0 = time.time()
    for ctas, stages in shapes:
        ts = []
        for r in range(n_warm + n_time):
            flush.fill_(r & 255)
            e0.record()
            attn.read_stream_probe(m, ctas, stages)
            e1.record()
            e1.synchronize()
            if r >= n_warm:
                ts.append(e0.elapsed_time(e1) * 1e3)
        us = float(np.median(ts))
        res.append({"probe": "tma_read_stream", "ctas": ctas, "stages": stages,
                    "inflight_kb_per_sm": stages * 16 * (2 if ctas > sms else 1),
                    "us": round(us, 2), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1)})
    t1 = time.time()
    if clk is not None:
        clk.stop()
    err = attn.device_error()
    if err != 0:
        raise RuntimeError(f"read-stream probe recorded device error {err}")
    for r in res:
        print(json.dumps(r))
    best = max(res, key=lambda r: r["gbs"])
    pk = peaks()
    print(json.dumps({"probe": "tma_read_stream_summary", "bytes": nbytes,
                      "matrix": list(m.shape), "box": [128, 64], "passes_timed": n_time,
                      "best": best, "copy_peak_gbs": pk["hbm_gbs"],
                      "best_frac_of_copy_peak": round(best["gbs"] / pk["hbm_gbs"], 3),
                      "clocks": clk.summary(t0, t1) if clk is not None else None}))
    return 0


def main():
    args = parse()
    if args.read_stream:
        return read_stream(args)
    if args.ncu_traffic or args.ncu_launches:
        rows = write_traffic(args.ncu_traffic) if args.ncu_traffic else \
            launch_table(args.ncu_launches)
        for row in rows:
            print(row)
        return 0
    world, rank, local = rank_env()

    if args.impl == "reference":
        if rank != 0:
            return 0
        from block_diffusion_draft_gb300 import workloads as W
        Wm = max(1, args.warmup)
        r = OracleRunner(args.workload, args.seed)
        for _ in range(Wm):
            r.step()
        n, dt = r.time(args.steps, budget_s=240.0)
        value = n * r.blocks_per_step / dt
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
                "n_gpus": args.gpus, "steps": n, "warmup": Wm,
                "ms_per_step": 1000.0 * dt / n, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded N(0,1) hidden, N(0,0.02) weights)",
                "config": dict(spec_config(W.SPECS[args.workload]),
                               parallelism=f"replicas x{world}", timing="host wall clock",
                               l2="not applicable (host cores)",
                               arm="fp64 CPU oracle"),
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(),
                                 "cpu_model": host_cpu_model(), "kind": "oracle",
                                 "sample": r.sample},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    import __graft_entry__ as G

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if rank == 0:
        G.build()
    if dist is not None:
        dist.barrier()
    G.build()

    def barrier():
        if dist is not None:
            dist.barrier()

    K, Wm = args.steps, max(3, args.warmup)
    wl = make_workload(args.workload, replica_seed(args.seed, rank, world), device, K + Wm)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)

    from block_diffusion_draft_gb300.dflash_attn import kernel_launches
    # warm-up (also sizes every scratch buffer)
    for i in range(Wm):
        wl.step(i)
    torch.cuda.synchronize(device)
    if wl.fixed:
        # identical steps: capture one into a CUDA graph to take the host out
        graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device)
        s.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(s):
            wl.step(0)
            torch.cuda.synchronize(device)
            n_cap = kernel_launches()
            with torch.cuda.graph(graph, stream=s):
                wl.step(0)
            graph_kernels = kernel_launches() - n_cap
        torch.cuda.current_stream(device).wait_stream(s)
        run = lambda i: graph.replay()
    else:
        run = wl.step
    wl.reset()
    torch.cuda.synchronize(device)

    # ---------------------------------------------------------- timed region
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    clocks = ClockSampler(device.index) if rank == 0 and not args.no_clocks else None
    # keep the GPU busy while the sampler starts
    t_load = time.time()
    while time.time() - t_load < (1.0 if clocks else 0.0):
        for i in range(20):
            run(i)
        torch.cuda.synchronize(device)
    wl.reset()
    barrier()
    torch.cuda.synchronize(device)
    n_launch0 = kernel_launches()
    t0 = time.time()
    for i in range(K):
        flush.zero_()
        ev[i][0].record()
        run(i)
        ev[i][1].record()
    torch.cuda.synchronize(device)
    barrier()
    t1 = time.time()
    # the library's own count of the kernels it launched in the timed region
    # (a graph replays the kernels launched while it was captured)
    gpu_launches = graph_kernels * K if wl.fixed else kernel_launches() - n_launch0
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = float(np.mean(step_ms))
    if clocks:
        time.sleep(0.1)
        clocks.stop()
    ms = max_over_ranks(ms, dist, device)
    value = job_value(world, wl.blocks_per_step, ms)

    # the plain per-layer schedule of a layer stack, same inputs, for comparison
    per_layer = None
    if hasattr(wl, "per_layer_step"):
        g2 = torch.cuda.CUDAGraph()
        s2 = torch.cuda.Stream(device)
        s2.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(s2):
            wl.per_layer_step(0)
            torch.cuda.synchronize(device)
            with torch.cuda.graph(g2, stream=s2):
                wl.per_layer_step(0)
        torch.cuda.current_stream(device).wait_stream(s2)
        torch.cuda.synchronize(device)
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        for i in range(K):
            flush.zero_()
            ev2[i][0].record()
            g2.replay()
            ev2[i][1].record()
        torch.cuda.synchronize(device)
        ms2 = float(np.mean([a.elapsed_time(b) for a, b in ev2]))
        per_layer = {"ms_per_step": ms2,
                     "value": world * wl.blocks_per_step / (ms2 / 1000.0),
                     "step": "ctx_project + per-layer forward with the context rows + crop"}

    # ---------------------------------------------------- per-kernel timing
    handles = wl.handles() if hasattr(wl, "handles") else [wl.attn]
    wl.reset()
    for h in handles:
        h.trace(True)
    for i in range(K):
        flush.zero_()
        wl.step(i)
    torch.cuda.synchronize(device)
    tr = {}
    for h in handles:
        for name, (t_ms, n_l) in h.trace_read().items():
            t0_, n0_ = tr.get(name, (0.0, 0))
            tr[name] = (t0_ + t_ms, n0_ + n_l)
        h.trace(False)
    kb = [wl.kernel_bytes(i) for i in range(K)]
    kf = [wl.kernel_flops(i) for i in range(K)]
    per_kernel = {}
    for name, (tot_ms, n) in tr.items():
        per_kernel[name] = {"avg_us": 1000.0 * tot_ms / n, "launches": n}
        if kb[0].get(name):
            per_kernel[name]["gbs"] = sum(k[name] for k in kb) / (tot_ms / 1000.0) / 1e9
        if kf[0].get(name):
            per_kernel[name]["tflops"] = sum(k[name] for k in kf) / (tot_ms / 1000.0) / 1e12
    # the longest-running bucket that has a roofline model (flops or bytes)
    modelled = [k for k in tr if kf[0].get(k) or kb[0].get(k)] or list(tr)
    dom = max(modelled, key=lambda k: tr[k][0])
    pk = peaks()
    tot_ms, n = tr[dom]
    if kf[0].get(dom):
        ach = sum(k[dom] for k in kf) / (tot_ms / 1000.0) / 1e12
        peak = pk["bf16_tflops_sustained"]
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": peak,
                "unit": "TFLOP/s", "frac": ach / peak,
                "peak_source": f"{pk['source']} bf16 sustained"}
    else:
        ach = sum(k[dom] for k in kb) / (tot_ms / 1000.0) / 1e9
        peak = pk["hbm_gbs"]
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peak,
                "unit": "GB/s", "frac": ach / peak, "peak_source": f"{pk['source']} hbm"}
    roof["traffic"] = measured_traffic(args.workload, dom)

    # ---------------------------------------------------- end to end (host)
    wl.reset()
    io = [wl.io_bytes(i) for i in range(K)]
    h2d = int(round(sum(b[0] for b in io) / K))
    d2h = int(round(sum(b[1] for b in io) / K))
    e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(K)]
    run_e2e = wl.step_e2e
    if wl.fixed:
        # identical steps: the copies and the library calls of one step in a
        # CUDA graph (the copies read the fixed pinned staging buffers)
        g3 = torch.cuda.CUDAGraph()
        s3 = torch.cuda.Stream(device)
        s3.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(s3):
            wl.stage_e2e(0)
            wl.step_e2e(0)
            torch.cuda.synchronize(device)
            with torch.cuda.graph(g3, stream=s3):
                wl.step_e2e(0)
        torch.cuda.current_stream(device).wait_stream(s3)
        run_e2e = lambda i: g3.replay()
    wl.reset()
    torch.cuda.synchronize(device)
    for i in range(K):
        wl.stage_e2e(i)
        flush.zero_()
        e_ev[i][0].record()
        run_e2e(i)
        e_ev[i][1].record()
        if wl.fixed:
            # one staging buffer (captured in the graph): refilled for the
            # next step only after this step's copy has read it
            e_ev[i][1].synchronize()
    torch.cuda.synchronize(device)
    e_ms = float(np.mean([a.elapsed_time(b) for a, b in e_ev]))
    e_ms = max_over_ranks(e_ms, dist, device)
    e2e = {"value": job_value(world, wl.blocks_per_step, e_ms), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}
    err = max(h.device_error() for h in handles)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": Wm, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.sp.dtype_name(),
            "data": "synthetic (seeded N(0,1) hidden, N(0,0.02) weights)",
            "config": dict(wl.config(), parallelism=f"replicas x{world}",
                           timing="CUDA graph of one step" if wl.fixed else "eager"),
            "roofline": roof, "kernels": per_kernel,
            "clocks": clocks.summary(t0, t1) if clocks else None,
            "e2e": e2e, "gpu_launches": gpu_launches,
            "device_error": err}
    if per_layer:
        line["per_layer_schedule"] = per_layer
    # algorithmic bytes of the average step (serving steps differ in length)
    step_bytes = float(np.mean([sum(k.values()) for k in kb])) if kb[0] else None
    if step_bytes:
        line["step_achieved_gbs"] = step_bytes / (ms / 1000.0) / 1e9
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(args.workload, args.seed, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
