"""The allocation-free context projection agrees with the ordinary one.

dflash_ctx_project_noalloc exists for callers that cannot let the library
allocate device memory (graph capture, fixed start-up memory plans, external
pools).  It must compute what dflash_ctx_project computes, from its fixed
scratch array, call after call: the array keeps the previous call's contents,
so a second call with different inputs is the check that nothing stale leaks
through.  This file is named to be collected last.
"""
import ctypes

import pytest
import torch

from block_diffusion_draft_gb300 import workloads as W
from block_diffusion_draft_gb300.dflash_attn import check, lib

import helpers as T

pytestmark = pytest.mark.gpu


def _noalloc(attn, x, y):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib().dflash_ctx_project_noalloc(attn.handle, ctypes.c_void_p(x.data_ptr()),
                                            x.shape[0], ctypes.c_void_p(y.data_ptr()),
                                            stream)


@pytest.mark.parametrize("shape", ["qwen3_8b", "small"])
def test_noalloc_matches_ctx_project_on_two_calls_in_a_row(shape):
    if shape == "qwen3_8b":
        sp = W.SPECS["qwen3_8b_single"]
        rows = (16, 7)
    else:
        sp = W.spec("qwen3_8b_single", hidden=1024, n_heads=8, n_kv_heads=2,
                    n_target_layers=2, max_position=4096)
        rows = (100, 33)
    w = W.weights(sp, 11)
    attn = T.gpu_layer(sp, w)
    for call, n in enumerate(rows):
        x = W.target_layer_rows(sp, 11, call, 0, n).cuda()
        ref = attn.ctx_project(x)
        y = torch.full_like(ref, float("nan"))
        check(_noalloc(attn, x, y))
        torch.cuda.synchronize()
        T.assert_close(T.f64(y), T.f64(ref), "bf16", f"noalloc call {call}")
    assert attn.device_error() == 0


def test_noalloc_rejects_requests_above_its_fixed_scratch():
    sp = W.spec("qwen3_8b_single", hidden=1024, n_heads=8, n_kv_heads=2,
                n_target_layers=2, max_position=4096)
    attn = T.gpu_layer(sp, W.weights(sp, 12))
    rows = 8192  # 8192 x 1024 fp32 = 32 MiB of fc output alone
    x = torch.zeros(rows, 2 * sp.hidden, dtype=torch.bfloat16, device="cuda")
    y = torch.full((rows, sp.hidden), 7.0, dtype=torch.bfloat16, device="cuda")
    rc = _noalloc(attn, x, y)
    assert rc == -3
    assert b"limit" in lib().dflash_last_error()
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
