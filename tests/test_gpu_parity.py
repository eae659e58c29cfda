"""GPU vs oracle parity on small shapes that still span several tiles,
ragged tails, split key ranges and split-K projections.  Every call goes
through the C ABI."""
import numpy as np
import pytest
import torch

from block_diffusion_draft_gb300 import workloads as W
from oracle import dflash_oracle as O

import helpers as T

pytestmark = pytest.mark.gpu


def small_bf16(**kw):
    base = dict(hidden=1024, n_heads=8, n_kv_heads=2, head_dim=128, batch=3,
                n_target_layers=2, max_position=8192)
    base.update(kw)
    return W.spec("qwen3_8b_single", **base)


def test_tiny_fp32_workload_matches_oracle():
    # tiny fp32 layer: 112 rows prefilled through forward + crop, then a step
    # with 16 new context rows and a 16-row block (128 context rows in all)
    sp = W.SPECS["tiny_fp32"]
    sc = T.Scenario(sp, seed=0, capacity=256)
    got, ref = sc.step([sp.prefill])
    T.assert_close(got, ref, "fp32", "prefill step")
    sc.crop([sp.prefill])
    got, ref = sc.step([sp.n_new])
    T.assert_close(got, ref, "fp32", "step")
    assert sc.cache.lengths() == [sp.prefill + sp.n_new + sp.block_size]
    for k, ko, v, vo in sc.compare_cache():
        T.assert_close(k, ko, "fp32", "cache K")
        T.assert_close(v, vo, "fp32", "cache V")


@pytest.mark.parametrize("gains", [False, True])
def test_bf16_ragged_batch_two_steps(gains):
    sp = small_bf16()
    sc = T.Scenario(sp, seed=1, capacity=1024, random_gains=gains)
    # ragged prefill: 0, 1 and 300 context rows (several key tiles + tail)
    got, ref = sc.step([0, 1, 300])
    T.assert_close(got, ref, "bf16", "prefill")
    sc.crop([0, 1, 300])
    got, ref = sc.step([5, 0, 129])
    T.assert_close(got, ref, "bf16", "step 2")
    assert sc.cache.lengths() == [21, 17, 445]
    for k, ko, v, vo in sc.compare_cache():
        T.assert_close(k, ko, "bf16", "cache K")
        T.assert_close(v, vo, "bf16", "cache V")


def test_bf16_long_sequence_splits_keys_across_ctas():
    # one sequence with 2000 keys: the key range is split over several CTAs
    # and merged by the last one
    sp = small_bf16(batch=1)
    sc = T.Scenario(sp, seed=2, capacity=4096)
    got, ref = sc.step([1983])
    T.assert_close(got, ref, "bf16", "long")


def test_bf16_full_q_tile_groups8():
    # 8 query heads per kv head x 16 rows = a full 128-row Q tile
    sp = small_bf16(n_heads=8, n_kv_heads=1, batch=2)
    sc = T.Scenario(sp, seed=3, capacity=512)
    got, ref = sc.step([40, 200])
    T.assert_close(got, ref, "bf16", "g8")


@pytest.mark.parametrize("window", [0, 100])
def test_bf16_causal_layer(window):
    # causal layers ("vllm...qwen3_dflash", _dflash_layer_causal), full and
    # banded: a long prefill step split across CTAs, a crop, then a short step
    sp = small_bf16(sliding_window=window, causal=True, batch=2)
    sc = T.Scenario(sp, seed=14, capacity=1024)
    got, ref = sc.step([50, 400])
    T.assert_close(got, ref, "bf16", "causal prefill")
    sc.crop([50, 400])
    got, ref = sc.step([16, 3])
    T.assert_close(got, ref, "bf16", "causal step")


def test_fp32_causal_layer():
    sp = W.spec("tiny_fp32", causal=True)
    sc = T.Scenario(sp, seed=15, capacity=256)
    got, ref = sc.step([sp.prefill])
    T.assert_close(got, ref, "fp32", "fp32 causal")


def test_bf16_sliding_window_band():
    sp = small_bf16(sliding_window=100, batch=2)
    sc = T.Scenario(sp, seed=4, capacity=1024)
    got, ref = sc.step([50, 400])
    T.assert_close(got, ref, "bf16", "band prefill")
    sc.crop([50, 400])
    got, ref = sc.step([16, 3])
    T.assert_close(got, ref, "bf16", "band step")


def test_bf16_large_batch_persistent_gemm():
    # 40 sequences: 640 block rows and ~400 context rows take the persistent
    # 128 x 256-tile projection path
    sp = small_bf16(batch=40)
    sc = T.Scenario(sp, seed=12, capacity=256, check=[0, 17, 39])
    n = [int(x) for x in np.random.default_rng(3).integers(0, 21, size=40)]
    got, ref = sc.step(n)
    T.assert_close(got, ref, "bf16", "batch 40")
    sc.crop(n)
    got, ref = sc.step([16] * 40)
    T.assert_close(got, ref, "bf16", "batch 40 step 2")
    for k, ko, v, vo in sc.compare_cache():
        T.assert_close(k, ko, "bf16", "cache K")
        T.assert_close(v, vo, "bf16", "cache V")


def test_bf16_mid_batch_swapped_operand_o_proj():
    # 20 sequences x 16 block rows = 320 o_proj rows: the swapped-operand
    # projection kernel (two MMA chunks of 256 + 64 token rows)
    sp = small_bf16(batch=20)
    sc = T.Scenario(sp, seed=13, capacity=256, check=[0, 9, 19])
    n = [int(x) for x in np.random.default_rng(5).integers(0, 17, size=20)]
    got, ref = sc.step(n)
    T.assert_close(got, ref, "bf16", "batch 20")


def test_bf16_ctx_project_matches_oracle():
    sp = small_bf16()
    w = W.weights(sp, 5)
    cfg, lw = T.oracle_layer(sp, w)
    attn = T.gpu_layer(sp, w)
    # 129 .. 384 rows take the swapped-operand kernel (one and two MMA chunks)
    for rows in (1, 16, 129, 200, 384, 600):
        x = W.target_layer_rows(sp, 5, 0, rows, rows)
        y = attn.ctx_project(x.cuda())
        torch.cuda.synchronize()
        ref = O.ctx_project(cfg, lw, T.f64(x))
        T.assert_close(T.f64(y), ref, "bf16", f"ctx_project rows={rows}")


def test_fp32_ctx_project_matches_oracle():
    sp = W.SPECS["tiny_fp32"]
    w = W.weights(sp, 6)
    cfg, lw = T.oracle_layer(sp, w)
    attn = T.gpu_layer(sp, w)
    x = W.target_layer_rows(sp, 6, 0, 0, 37)
    y = attn.ctx_project(x.cuda())
    torch.cuda.synchronize()
    T.assert_close(T.f64(y), O.ctx_project(cfg, lw, T.f64(x)), "fp32", "fp32 ctx_project")


# bf16 cases: (query heads, blocks).  A bf16 CTA takes two Q tiles of
# 128 // (groups * 16) blocks each; the cases end on a unit with one partial
# Q tile (8, 9), with a full and a partial Q tile (8, 7), with Q tiles of 96
# rows (6, 7) and with 8-block units (4, 10).
@pytest.mark.parametrize("dtype,heads,n_blocks", [("bf16", 8, 9), ("bf16", 8, 7),
                                                  ("bf16", 6, 7), ("bf16", 4, 10),
                                                  ("fp32", 0, 5)])
def test_packed_training_layout_matches_oracle(dtype, heads, n_blocks):
    if dtype == "bf16":
        sp = small_bf16(batch=2, seq=300, n_blocks=n_blocks, n_heads=heads)
    else:
        sp = W.spec("tiny_fp32", batch=2, seq=100, n_blocks=n_blocks)
    seed = 7
    w = W.weights(sp, seed)
    cfg, lw = T.oracle_layer(sp, w)
    attn = T.gpu_layer(sp, w)
    bs = sp.block_size
    th = torch.stack([W.hidden_rows(sp, seed, "hidden", 0, b, sp.seq) for b in range(sp.batch)])
    nz = torch.stack([W.hidden_rows(sp, seed, "noise", 0, b, sp.n_blocks * bs)
                      for b in range(sp.batch)])
    anchors = W.anchors(sp, seed)
    anchors[1, -1] = sp.seq   # a block that sees the whole context
    anchors[0, 0] = 0         # and one that sees none of it
    out = attn.forward_packed(nz.cuda(), th.cuda(), anchors.cuda(), bs)
    torch.cuda.synchronize()
    ref = O.forward_packed(cfg, lw, T.f64(nz), T.f64(th), anchors.numpy(), bs)
    T.assert_close(T.f64(out), ref, dtype, "packed")
    assert attn.device_error() == 0


def test_capacity_overflow_appends_nothing():
    sp = small_bf16(batch=2)
    sc = T.Scenario(sp, seed=8, capacity=64)
    with pytest.raises(Exception, match="CAPACITY"):
        sc.attn.forward(sc.cache, torch.zeros(2, 16, sp.hidden, dtype=torch.bfloat16,
                                              device="cuda"),
                        torch.zeros(60, sp.hidden, dtype=torch.bfloat16, device="cuda"),
                        [10, 50], torch.zeros(60 + 32, dtype=torch.int32, device="cuda"))
    assert sc.cache.lengths() == [0, 0]


def test_crop_is_exact_and_rerun_reproduces_cache_bitwise():
    sp = small_bf16(batch=2)
    sc = T.Scenario(sp, seed=9, capacity=512)
    th = torch.cat([W.hidden_rows(sp, 9, "hidden", 0, b, n) for b, n in enumerate((100, 37))])
    nz = torch.stack([W.hidden_rows(sp, 9, "noise", 0, b, 16) for b in range(2)]).cuda()
    pos = torch.cat([W.window_positions(0, n, 16) for n in (100, 37)]).cuda()
    out1 = sc.attn.forward(sc.cache, nz, th.cuda(), [100, 37], pos)
    k1, v1 = sc.cache.read()
    L = sc.cache.lengths()
    assert L == [116, 53]
    with pytest.raises(Exception, match="RANGE"):
        sc.cache.crop([117, 0])
    assert sc.cache.lengths() == L
    # crop moves no data: rows below the new length are untouched
    sc.cache.crop([0, 0])
    assert sc.cache.lengths() == [0, 0]
    # the identical step again reproduces cache and output bit for bit
    out2 = sc.attn.forward(sc.cache, nz, th.cuda(), [100, 37], pos)
    k2, v2 = sc.cache.read()
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)
    for b, n in enumerate(L):
        assert torch.equal(k1[b, :, :n], k2[b, :, :n])
        assert torch.equal(v1[b, :, :n], v2[b, :, :n])
    # crop to the context rows and re-append the block alone (a different
    # launch shape): rows match within the bf16 tolerance
    sc.cache.crop([100, 37])
    pos2 = torch.cat([W.window_positions(n, 0, 16) for n in (100, 37)]).cuda()
    sc.attn.forward(sc.cache, nz, None, [0, 0], pos2)
    k3, v3 = sc.cache.read()
    torch.cuda.synchronize()
    assert sc.cache.lengths() == L
    for b, n in enumerate(L):
        assert torch.equal(k1[b, :, :n - 16], k3[b, :, :n - 16])
        T.assert_close(T.f64(k3[b, :, :n]), T.f64(k1[b, :, :n]), "bf16", "re-append K")
        T.assert_close(T.f64(v3[b, :, :n]), T.f64(v1[b, :, :n]), "bf16", "re-append V")


def test_first_call_of_fresh_layers_equals_rerun_bitwise():
    # A fresh layer's first forward (scratch allocated during the call) and
    # the identical step after crop(0), enqueued back to back with no host
    # synchronisation between them, give the same output and cache bits, on
    # 20 layers in turn.  Most CTAs of the short sequences' key clusters have
    # no keys, so this also covers the empty-unit path of the attention.
    sp = small_bf16(batch=2)
    for it in range(20):
        sc = T.Scenario(sp, seed=100 + it, capacity=512)
        n_ctx = [100, 37] if it % 2 == 0 else [3 + it, 200 - it]
        th = torch.cat([W.hidden_rows(sp, 100 + it, "hidden", 0, b, n)
                        for b, n in enumerate(n_ctx)]).cuda()
        nz = torch.stack([W.hidden_rows(sp, 100 + it, "noise", 0, b, 16)
                          for b in range(2)]).cuda()
        pos = torch.cat([W.window_positions(0, n, 16) for n in n_ctx]).cuda()
        out1 = sc.attn.forward(sc.cache, nz, th, n_ctx, pos)
        k1, v1 = sc.cache.read()
        sc.cache.crop([0, 0])
        out2 = sc.attn.forward(sc.cache, nz, th, n_ctx, pos)
        k2, v2 = sc.cache.read()
        torch.cuda.synchronize()
        diff = (out1.float() - out2.float()).abs()
        assert torch.equal(out1, out2), \
            f"layer {it}: {int((diff > 0).sum())} elements differ, max {float(diff.max()):.3e}"
        for b, n in enumerate(n_ctx):
            assert torch.equal(k1[b, :, :n + 16], k2[b, :, :n + 16])
            assert torch.equal(v1[b, :, :n + 16], v2[b, :, :n + 16])
        assert sc.attn.device_error() == 0
        sc.cache.close()
        sc.attn.close()


def test_bad_position_is_reported_not_faulted():
    sp = small_bf16(batch=1)
    sc = T.Scenario(sp, seed=10, capacity=64)
    pos = torch.full((16,), sp.max_position + 5, dtype=torch.int32, device="cuda")
    nz = torch.zeros(1, 16, sp.hidden, dtype=torch.bfloat16, device="cuda")
    sc.attn.forward(sc.cache, nz, None, [0], pos)
    assert sc.attn.device_error() == 2
    assert sc.attn.device_error() == 0
