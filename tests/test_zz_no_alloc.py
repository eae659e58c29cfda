"""The allocation-free context projection agrees with the ordinary one and
with the oracle.

dflash_ctx_project_noalloc exists for callers that cannot let the library
allocate device memory: serving processes that fix all device memory at
start-up and treat a later allocation as a failure, and hosts whose own pool
must be the only allocator on the GPU.  It must compute what
dflash_ctx_project computes, from its fixed scratch array, call after call:
the array keeps the previous call's contents, so a second call with
different inputs is the check that nothing stale leaks through.  This file
is named to be collected last.
"""
import ctypes

import pytest
import torch

from block_diffusion_draft_gb300 import workloads as W
from block_diffusion_draft_gb300.dflash_attn import check, lib
from oracle import dflash_oracle as O

import helpers as T

pytestmark = pytest.mark.gpu


def _noalloc(attn, x, y):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib().dflash_ctx_project_noalloc(attn.handle, ctypes.c_void_p(x.data_ptr()),
                                            x.shape[0], ctypes.c_void_p(y.data_ptr()),
                                            stream)


def _small():
    return W.spec("qwen3_8b_single", hidden=1024, n_heads=8, n_kv_heads=2,
                  n_target_layers=2, max_position=4096)


@pytest.mark.parametrize("shape", ["qwen3_8b", "small", "tiny_fp32"])
def test_noalloc_matches_ctx_project_and_oracle_on_two_calls_in_a_row(shape):
    if shape == "qwen3_8b":
        sp, rows = W.SPECS["qwen3_8b_single"], (16, 7)
    elif shape == "small":
        sp, rows = _small(), (100, 33)
    else:
        sp, rows = W.SPECS["tiny_fp32"], (37, 5)
    kind = "bf16" if sp.dtype == "bf16" else "fp32"
    w = W.weights(sp, 11)
    cfg, lw = T.oracle_layer(sp, w)
    attn = T.gpu_layer(sp, w)
    for call, n in enumerate(rows):
        x = W.target_layer_rows(sp, 11, call, 0, n)
        xd = x.cuda()
        ref = attn.ctx_project(xd)
        y = torch.full_like(ref, float("nan"))
        check(_noalloc(attn, xd, y))
        torch.cuda.synchronize()
        T.assert_close(T.f64(y), T.f64(ref), kind, f"noalloc vs ctx_project, call {call}")
        T.assert_close(T.f64(y), O.ctx_project(cfg, lw, T.f64(x)), kind,
                       f"noalloc vs oracle, call {call}")
    assert attn.device_error() == 0


def test_noalloc_allocates_no_device_memory():
    sp = _small()
    attn = T.gpu_layer(sp, W.weights(sp, 13))
    xs = [W.target_layer_rows(sp, 13, c, 0, 100).cuda() for c in range(2)]
    ys = [torch.empty(100, sp.hidden, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    check(_noalloc(attn, xs[0], ys[0]))  # first call on the device: address look-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for x, y in zip(xs, ys):
        check(_noalloc(attn, x, y))
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    for x, y in zip(xs, ys):
        T.assert_close(T.f64(y), T.f64(attn.ctx_project(x)), "bf16", "noalloc rows")


def test_noalloc_row_limit_at_hidden_4096():
    # up to 384 rows the projection takes kernels with no split-K tiles: the
    # scratch is the fp32 output (384 x 4096 x 4 = 6 MiB); from 385 rows the
    # persistent kernel's split-K tiles alone fill the 16 MiB array
    sp = W.SPECS["qwen3_8b_single"]
    w = W.weights(sp, 14)
    attn = T.gpu_layer(sp, w)
    x = W.target_layer_rows(sp, 14, 0, 0, 385).cuda()
    y = torch.full((385, sp.hidden), 7.0, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(attn, x, y) == -3
    assert b"limit" in lib().dflash_last_error()
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
    check(_noalloc(attn, x[:384], y[:384]))
    ref = attn.ctx_project(x[:384])
    torch.cuda.synchronize()
    T.assert_close(T.f64(y[:384]), T.f64(ref), "bf16", "noalloc 384 rows")
    assert bool((y[384] == 7.0).all())


def test_noalloc_rejects_requests_above_its_fixed_scratch():
    sp = _small()
    attn = T.gpu_layer(sp, W.weights(sp, 12))
    rows = 8192  # 8192 x 1024 fp32 = 32 MiB of fc output alone
    x = torch.zeros(rows, 2 * sp.hidden, dtype=torch.bfloat16, device="cuda")
    y = torch.full((rows, sp.hidden), 7.0, dtype=torch.bfloat16, device="cuda")
    rc = _noalloc(attn, x, y)
    assert rc == -3
    assert b"limit" in lib().dflash_last_error()
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
