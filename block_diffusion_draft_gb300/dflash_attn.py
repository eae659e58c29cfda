"""ctypes binding of libdflash_attn.so (include/dflash_attn.h).

Argument marshalling only: torch tensors in, their device pointers and the
current CUDA stream out to the C ABI.  Every step of the layer runs in the
library's CUDA kernels; if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from ctypes import POINTER, c_float, c_int, c_int32, c_void_p
from typing import Dict, Optional, Sequence

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libdflash_attn.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "dflash_attn.h")

DFLASH_BF16, DFLASH_FP32 = 0, 1
STATUS = {0: "OK", -1: "ERR_ARG", -2: "ERR_SHAPE", -3: "ERR_CAPACITY",
          -4: "ERR_RANGE", -5: "ERR_CUDA", -6: "ERR_DEVICE",
          -7: "ERR_UNSUPPORTED", -8: "ERR_MEMORY"}


class Config(ctypes.Structure):
    _fields_ = [("hidden", c_int32), ("n_heads", c_int32),
                ("n_kv_heads", c_int32), ("head_dim", c_int32),
                ("n_target_layers", c_int32), ("rms_eps", c_float),
                ("rope_theta", c_float), ("sliding_window", c_int32),
                ("max_position", c_int32), ("dtype", c_int32), ("causal", c_int32)]


class DFlashError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{STATUS.get(code, code)}: {message}")
        self.code = code


_LIB = None

_SIGNATURES = {
    "dflash_last_error": ([], ctypes.c_char_p),
    "dflash_abi_version": ([], c_int),
    "dflash_attn_create": ([POINTER(Config)] + [c_void_p] * 8 + [POINTER(c_void_p)], c_int),
    "dflash_attn_destroy": ([c_void_p], c_int),
    "dflash_attn_reserve": ([c_void_p, c_int, c_int, c_int], c_int),
    "dflash_cache_create": ([c_void_p, c_int, c_int, POINTER(c_void_p)], c_int),
    "dflash_cache_destroy": ([c_void_p], c_int),
    "dflash_cache_lengths": ([c_void_p, POINTER(c_int32)], c_int),
    "dflash_cache_data": ([c_void_p, POINTER(c_void_p), POINTER(c_void_p)] +
                          [POINTER(c_int32)] * 4, c_int),
    "dflash_cache_read": ([c_void_p, c_void_p, c_void_p, c_void_p], c_int),
    "dflash_cache_crop": ([c_void_p, POINTER(c_int32)], c_int),
    "dflash_ctx_project": ([c_void_p, c_void_p, c_int, c_void_p, c_void_p], c_int),
    "dflash_ctx_project_noalloc": ([c_void_p, c_void_p, c_int, c_void_p, c_void_p], c_int),
    "dflash_attn_forward": ([c_void_p, c_void_p, c_int, c_int, c_void_p, c_void_p,
                             POINTER(c_int32), c_void_p, c_void_p, c_void_p], c_int),
    "dflash_attn_forward_packed": ([c_void_p, c_int, c_int, c_int, c_int, c_void_p,
                                    c_void_p, c_void_p, c_void_p, c_void_p], c_int),
    "dflash_paged_cache_create": ([c_void_p, c_int, c_int, POINTER(c_void_p)], c_int),
    "dflash_paged_cache_destroy": ([c_void_p], c_int),
    "dflash_paged_cache_data": ([c_void_p, POINTER(c_void_p), POINTER(c_void_p)] +
                                [POINTER(c_int32)] * 4, c_int),
    "dflash_paged_cache_read": ([c_void_p, c_void_p, c_void_p, c_void_p], c_int),
    "dflash_attn_forward_paged": ([c_void_p, c_void_p, c_int, c_int, c_void_p, c_void_p,
                                   POINTER(c_int32), POINTER(c_int32), c_void_p, c_void_p,
                                   c_void_p, c_int, c_void_p, c_void_p], c_int),
    "dflash_kv_group_create": ([POINTER(c_void_p), c_int, POINTER(c_void_p)], c_int),
    "dflash_kv_group_destroy": ([c_void_p], c_int),
    "dflash_kv_group_append": ([c_void_p, POINTER(c_void_p), c_int, c_void_p,
                                POINTER(c_int32), c_void_p, c_void_p], c_int),
    "dflash_mlp_create": ([c_int, c_int, c_float] + [c_void_p] * 5 + [POINTER(c_void_p)],
                          c_int),
    "dflash_mlp_destroy": ([c_void_p], c_int),
    "dflash_decoder_layer_forward": ([c_void_p, c_void_p, c_void_p, c_int, c_int, c_void_p,
                                      c_void_p, c_void_p, POINTER(c_int32), c_void_p,
                                      c_void_p, c_void_p, c_void_p], c_int),
    "dflash_device_error": ([c_void_p, POINTER(c_int32)], c_int),
    "dflash_wait_probe": ([c_void_p, ctypes.c_int64, c_int, c_void_p], c_int),
    "dflash_read_stream_probe": ([c_void_p, c_void_p, ctypes.c_int64, ctypes.c_int64, c_int,
                                  c_int, c_void_p], c_int),
    "dflash_kernel_launches": ([POINTER(ctypes.c_uint64)], c_int),
    "dflash_packed_attn_core": ([c_void_p, c_int, c_int, c_int, c_int] + [c_void_p] * 7, c_int),
    "dflash_packed_attn_core_backward": ([c_void_p, c_int, c_int, c_int, c_int] +
                                         [c_void_p] * 11, c_int),
    "dflash_trace_enable": ([c_void_p, c_int], c_int),
    "dflash_trace_read": ([c_void_p, c_int, POINTER(ctypes.c_double), POINTER(c_int32)],
                          c_int),
}

KERNEL_KINDS = {"fc": 0, "norm": 1, "qkv": 2, "attn": 3, "o_proj": 4, "misc": 5, "mlp": 6,
                "bwd": 7}


def declared_functions() -> list:
    """Names of the functions include/dflash_attn.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_\w+)\s*\(", text)))


def lib():
    """Load the library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "block_diffusion_draft_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _LIB = L
    return _LIB


def check(rc: int) -> None:
    if rc != 0:
        raise DFlashError(rc, lib().dflash_last_error().decode())


def kernel_launches() -> int:
    """Kernels the library has launched in this process so far."""
    n = ctypes.c_uint64(0)
    check(lib().dflash_kernel_launches(ctypes.byref(n)))
    return n.value


def _p(t: Optional[torch.Tensor]):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(dev: torch.device):
    return c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _int32_array(xs: Sequence[int]):
    arr = (c_int32 * len(xs))(*[int(x) for x in xs])
    return arr


class DFlashAttention:
    """One draft attention layer held by the library.

    ``weights`` maps wq, wk, wv, wo, q_norm, k_norm and optionally fc,
    hidden_norm to tensors in nn.Linear [out, in] layout (any device; they are
    moved to ``device`` in ``dtype`` and copied into library memory).
    """

    def __init__(self, weights: Dict[str, torch.Tensor], *, hidden: int,
                 n_heads: int, n_kv_heads: int, head_dim: int = 0,
                 n_target_layers: int = 0, rms_eps: float = 1e-6,
                 rope_theta: float = 1e6, sliding_window: int = 0,
                 max_position: int = 0, dtype: torch.dtype = torch.bfloat16,
                 device: Optional[torch.device] = None, causal: bool = False):
        self.device = torch.device(device or "cuda")
        if self.device.type != "cuda":
            raise ValueError("the library runs on CUDA devices only")
        if dtype not in (torch.bfloat16, torch.float32):
            raise ValueError("dtype must be bfloat16 or float32")
        self.dtype = dtype
        self.hidden, self.n_heads, self.n_kv_heads = hidden, n_heads, n_kv_heads
        self.head_dim = head_dim or hidden // n_heads
        self.cfg = Config(hidden, n_heads, n_kv_heads, self.head_dim,
                          n_target_layers, rms_eps, rope_theta, sliding_window,
                          max_position,
                          DFLASH_BF16 if dtype == torch.bfloat16 else DFLASH_FP32,
                          1 if causal else 0)
        dev_w = {k: v.to(self.device, dtype).contiguous() for k, v in weights.items()}
        fc = dev_w.get("fc") if n_target_layers > 0 else None
        hn = dev_w.get("hidden_norm") if n_target_layers > 0 else None
        h = c_void_p()
        with torch.cuda.device(self.device):
            check(lib().dflash_attn_create(
                ctypes.byref(self.cfg), _p(dev_w["wq"]), _p(dev_w["wk"]),
                _p(dev_w["wv"]), _p(dev_w["wo"]), _p(dev_w["q_norm"]),
                _p(dev_w["k_norm"]), _p(fc), _p(hn), ctypes.byref(h)))
        self.handle = h

    # ---------------------------------------------------------------- calls
    def reserve(self, max_batch: int, max_rows: int, max_keys: int) -> None:
        with torch.cuda.device(self.device):
            check(lib().dflash_attn_reserve(self.handle, max_batch, max_rows, max_keys))

    def ctx_project(self, target_layers: torch.Tensor,
                    out: Optional[torch.Tensor] = None) -> torch.Tensor:
        rows = target_layers.shape[0]
        if out is None:
            out = torch.empty(rows, self.hidden, device=self.device, dtype=self.dtype)
        with torch.cuda.device(self.device):
            check(lib().dflash_ctx_project(self.handle, _p(target_layers.contiguous()),
                                           rows, _p(out), _stream(self.device)))
        return out

    def forward(self, cache: "DraftCache", noise: torch.Tensor,
                target_hidden: Optional[torch.Tensor], n_ctx: Sequence[int],
                positions: torch.Tensor,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
        B, q_len, _ = noise.shape
        if out is None:
            out = torch.empty_like(noise)
        th = None if target_hidden is None or target_hidden.numel() == 0 else target_hidden
        with torch.cuda.device(self.device):
            check(lib().dflash_attn_forward(
                self.handle, cache.handle, B, q_len, _p(noise), _p(th),
                _int32_array(n_ctx), _p(positions), _p(out), _stream(self.device)))
        return out

    def forward_paged(self, cache: "PagedCache", noise: torch.Tensor,
                      target_hidden: Optional[torch.Tensor], n_ctx: Sequence[int],
                      len_before: Sequence[int], positions: torch.Tensor,
                      slot_mapping: torch.Tensor, block_table: torch.Tensor,
                      out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """forward() over a paged cache: new rows go to slot_mapping's slots
        (int32, in positions order), keys are read through block_table
        (int32 [batch, bt_stride])."""
        B, q_len, _ = noise.shape
        if out is None:
            out = torch.empty_like(noise)
        th = None if target_hidden is None or target_hidden.numel() == 0 else target_hidden
        bt = block_table.contiguous()
        with torch.cuda.device(self.device):
            check(lib().dflash_attn_forward_paged(
                self.handle, cache.handle, B, q_len, _p(noise), _p(th),
                _int32_array(n_ctx), _int32_array(len_before), _p(positions),
                _p(slot_mapping), _p(bt), bt.shape[1], _p(out), _stream(self.device)))
        return out

    def forward_packed(self, noise: torch.Tensor, target_hidden: torch.Tensor,
                       anchors: torch.Tensor, block_size: int,
                       out: Optional[torch.Tensor] = None) -> torch.Tensor:
        B, q_total, _ = noise.shape
        seq = target_hidden.shape[1]
        nb = anchors.shape[1]
        if out is None:
            out = torch.empty_like(noise)
        with torch.cuda.device(self.device):
            check(lib().dflash_attn_forward_packed(
                self.handle, B, seq, nb, block_size, _p(noise), _p(target_hidden),
                _p(anchors), _p(out), _stream(self.device)))
        return out

    def packed_core(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                    anchors: torch.Tensor, seq: int, block_size: int):
        """Packed-layout attention core: q [B, T, n_heads, d], k/v
        [B, n_kv, seq + T, d] bf16, anchors [B, n_blocks] int32.  Returns
        (out like q, lse [B, T, n_heads] fp32)."""
        B, T = q.shape[0], q.shape[1]
        out = torch.empty_like(q)
        lse = torch.empty(B, T, q.shape[2], device=q.device, dtype=torch.float32)
        with torch.cuda.device(self.device):
            check(lib().dflash_packed_attn_core(
                self.handle, B, seq, T // block_size, block_size, _p(q), _p(k), _p(v),
                _p(anchors), _p(out), _p(lse), _stream(self.device)))
        return out, lse

    def packed_core_backward(self, q, k, v, out, lse, d_out, anchors, seq: int,
                             block_size: int):
        """Gradients (dq, dk, dv) of packed_core's output given d_out."""
        B, T = q.shape[0], q.shape[1]
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        with torch.cuda.device(self.device):
            check(lib().dflash_packed_attn_core_backward(
                self.handle, B, seq, T // block_size, block_size, _p(q), _p(k), _p(v),
                _p(out), _p(lse), _p(d_out), _p(anchors), _p(dq), _p(dk), _p(dv),
                _stream(self.device)))
        return dq, dk, dv

    def trace(self, enable: bool) -> None:
        """Start (fresh) or stop recording CUDA events around each launch."""
        with torch.cuda.device(self.device):
            check(lib().dflash_trace_enable(self.handle, 1 if enable else 0))

    def trace_read(self) -> dict:
        """{kernel kind: (total ms, launches)} of the current trace."""
        res = {}
        for name, kind in KERNEL_KINDS.items():
            ms, n = ctypes.c_double(0), c_int32(0)
            with torch.cuda.device(self.device):
                check(lib().dflash_trace_read(self.handle, kind, ctypes.byref(ms),
                                              ctypes.byref(n)))
            if n.value:
                res[name] = (ms.value, n.value)
        return res

    def device_error(self) -> int:
        code = c_int32(0)
        with torch.cuda.device(self.device):
            rc = lib().dflash_device_error(self.handle, ctypes.byref(code))
        if rc not in (0, -6):
            check(rc)
        return code.value

    def wait_probe(self, limit_ns: int, arrive: bool) -> None:
        """One bounded device wait of at most limit_ns on the current stream
        (arrive=False: a barrier nothing completes, so the wait runs out and
        records DFLASH_DEV_WAIT_TIMEOUT; read it with device_error())."""
        with torch.cuda.device(self.device):
            check(lib().dflash_wait_probe(self.handle, int(limit_ns), int(bool(arrive)),
                                          _stream(self.device)))

    def read_stream_probe(self, matrix: torch.Tensor, ctas: int, stages: int) -> None:
        """Enqueue one TMA read pass over a bf16 [rows, cols] matrix on the
        current stream (measurement aid: the weight boxes of the GEMMs,
        `stages` boxes in flight per CTA, data discarded)."""
        if matrix.dtype != torch.bfloat16 or matrix.dim() != 2 or not matrix.is_contiguous():
            raise ValueError("matrix must be a contiguous 2-D bf16 tensor")
        with torch.cuda.device(self.device):
            check(lib().dflash_read_stream_probe(self.handle, _p(matrix), matrix.shape[0],
                                                 matrix.shape[1], int(ctas), int(stages),
                                                 _stream(self.device)))

    def close(self) -> None:
        if getattr(self, "handle", None):
            with torch.cuda.device(self.device):
                lib().dflash_attn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DraftCache:
    """Draft KV cache held by the library ([batch][n_kv][capacity][head_dim])."""

    def __init__(self, attn: DFlashAttention, batch: int, capacity: int):
        self.attn = attn
        self.batch, self.capacity = batch, capacity
        h = c_void_p()
        with torch.cuda.device(attn.device):
            check(lib().dflash_cache_create(attn.handle, batch, capacity, ctypes.byref(h)))
        self.handle = h

    def lengths(self) -> list:
        arr = (c_int32 * self.batch)()
        check(lib().dflash_cache_lengths(self.handle, arr))
        return list(arr)

    def crop(self, keep: Sequence[int]) -> None:
        check(lib().dflash_cache_crop(self.handle, _int32_array(keep)))

    def read(self):
        """Copies of the K and V storage as [batch, n_kv, capacity, head_dim]."""
        a = self.attn
        shape = (self.batch, a.n_kv_heads, self.capacity, a.head_dim)
        k = torch.empty(shape, device=a.device, dtype=a.dtype)
        v = torch.empty(shape, device=a.device, dtype=a.dtype)
        with torch.cuda.device(a.device):
            check(lib().dflash_cache_read(self.handle, _p(k), _p(v), _stream(a.device)))
        return k, v

    def close(self) -> None:
        if getattr(self, "handle", None):
            lib().dflash_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class PagedCache:
    """Paged KV storage held by the library ([n_pages][n_kv][page_size]
    [head_dim] for K and for V); lengths and page tables are the caller's."""

    def __init__(self, attn: DFlashAttention, n_pages: int, page_size: int):
        self.attn = attn
        self.n_pages, self.page_size = n_pages, page_size
        h = c_void_p()
        with torch.cuda.device(attn.device):
            check(lib().dflash_paged_cache_create(attn.handle, n_pages, page_size,
                                                  ctypes.byref(h)))
        self.handle = h

    def read(self):
        """Copies of the K and V storage as [n_pages, n_kv, page_size, head_dim]."""
        a = self.attn
        shape = (self.n_pages, a.n_kv_heads, self.page_size, a.head_dim)
        k = torch.empty(shape, device=a.device, dtype=a.dtype)
        v = torch.empty(shape, device=a.device, dtype=a.dtype)
        with torch.cuda.device(a.device):
            check(lib().dflash_paged_cache_read(self.handle, _p(k), _p(v), _stream(a.device)))
        return k, v

    def close(self) -> None:
        if getattr(self, "handle", None):
            lib().dflash_paged_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class KVGroup:
    """Context K/V of several layers from one projection (the layers' K and V
    weights stacked); see dflash_kv_group_* in include/dflash_attn.h."""

    def __init__(self, layers: Sequence[DFlashAttention]):
        self.layers = list(layers)
        self.device = self.layers[0].device
        arr = (c_void_p * len(self.layers))(*[l.handle.value for l in self.layers])
        h = c_void_p()
        with torch.cuda.device(self.device):
            check(lib().dflash_kv_group_create(arr, len(self.layers), ctypes.byref(h)))
        self.handle = h

    def append(self, caches: Sequence["DraftCache"], target_hidden: Optional[torch.Tensor],
               n_ctx: Sequence[int], positions: Optional[torch.Tensor]) -> None:
        """Append the new context rows' K/V of every layer to its cache."""
        arr = (c_void_p * len(caches))(*[c.handle.value for c in caches])
        th = None if target_hidden is None or target_hidden.numel() == 0 else target_hidden
        with torch.cuda.device(self.device):
            check(lib().dflash_kv_group_append(self.handle, arr, len(n_ctx), _p(th),
                                               _int32_array(n_ctx), _p(positions),
                                               _stream(self.device)))

    def close(self) -> None:
        if getattr(self, "handle", None):
            with torch.cuda.device(self.device):
                lib().dflash_kv_group_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DecoderMLP:
    """Norms and Qwen3 MLP of a draft decoder layer (dflash_mlp_*): weights
    ``gate``, ``up`` [intermediate, hidden], ``down`` [hidden, intermediate],
    ``input_norm``, ``post_norm`` [hidden], all bf16."""

    def __init__(self, w: dict, hidden: int, intermediate: int, rms_eps: float = 1e-6,
                 device="cuda"):
        self.device = torch.device(device)
        self.hidden, self.intermediate = hidden, intermediate
        with torch.cuda.device(self.device):
            self._w = {k: w[k].to(self.device, torch.bfloat16).contiguous()
                       for k in ("gate", "up", "down", "input_norm", "post_norm")}
            h = c_void_p()
            check(lib().dflash_mlp_create(hidden, intermediate, rms_eps,
                                          *[_p(self._w[k]) for k in ("gate", "up", "down",
                                                                      "input_norm", "post_norm")],
                                          ctypes.byref(h)))
        self._w = None  # the library holds copies
        self.handle = h

    def layer_forward(self, attn: DFlashAttention, cache: "DraftCache", hidden: torch.Tensor,
                      residual: Optional[torch.Tensor], target_hidden: Optional[torch.Tensor],
                      n_ctx: Sequence[int], positions: torch.Tensor):
        """One decoder layer; returns (hidden_out, residual_out)."""
        B, q_len, _ = hidden.shape
        out = torch.empty_like(hidden)
        res = torch.empty_like(hidden)
        th = None if target_hidden is None or target_hidden.numel() == 0 else target_hidden
        with torch.cuda.device(self.device):
            check(lib().dflash_decoder_layer_forward(
                attn.handle, self.handle, cache.handle, B, q_len, _p(hidden), _p(residual),
                _p(th), _int32_array(n_ctx), _p(positions), _p(out), _p(res),
                _stream(self.device)))
        return out, res

    def layer_forward_into(self, attn: DFlashAttention, cache: "DraftCache",
                           hidden: torch.Tensor, residual: Optional[torch.Tensor],
                           target_hidden: Optional[torch.Tensor], n_ctx: Sequence[int],
                           positions: torch.Tensor, out: torch.Tensor,
                           residual_out: torch.Tensor) -> None:
        """layer_forward writing into caller-owned output tensors."""
        B, q_len, _ = hidden.shape
        th = None if target_hidden is None or target_hidden.numel() == 0 else target_hidden
        with torch.cuda.device(self.device):
            check(lib().dflash_decoder_layer_forward(
                attn.handle, self.handle, cache.handle, B, q_len, _p(hidden), _p(residual),
                _p(th), _int32_array(n_ctx), _p(positions), _p(out), _p(residual_out),
                _stream(self.device)))

    def close(self) -> None:
        if getattr(self, "handle", None):
            with torch.cuda.device(self.device):
                lib().dflash_mlp_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
