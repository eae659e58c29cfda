"""GPU vs oracle parity at the full sizes of the benchmark workloads, in the
launch configurations the benchmark uses.  The oracle follows a seeded
sample of sequences (each sequence depends only on its own rows) or blocks;
cache lengths are checked bit-exact for every sequence."""
import numpy as np
import pytest
import torch

from block_diffusion_draft_gb300 import workloads as W
from oracle import dflash_oracle as O

import helpers as T

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _serving(name, check, steps, cap_extra=64):
    sp = W.SPECS[name]
    sched = W.serving_schedule(sp, 0, steps=steps)
    pre = sched.prefill
    cap = max(pre) + sum(max(s.n_ctx) for s in sched.steps) + 2 * sp.block_size + cap_extra
    sc = T.Scenario(sp, seed=0, capacity=cap, check=check, page_size=sp.page_size)
    # prefill: all cached rows through one forward, then crop to them
    got, ref = sc.step(pre)
    T.assert_close(got, ref, "bf16", f"{name} prefill")
    sc.crop(pre)
    L = list(pre)
    for s, st in enumerate(sched.steps):
        got, ref = sc.step(st.n_ctx)
        T.assert_close(got, ref, "bf16", f"{name} step {s}")
        assert sc.lengths() == [L[b] + st.n_ctx[b] + sp.block_size for b in range(sp.batch)]
        L = [L[b] + st.n_ctx[b] for b in range(sp.batch)]
        sc.crop(L)
        assert sc.lengths() == L
    # cached rows of the last step (context rows; the block was cropped)
    for k, ko, v, vo in sc.compare_cache(rows=64):
        T.assert_close(k, ko, "bf16", f"{name} cache K")
        T.assert_close(v, vo, "bf16", f"{name} cache V")
    assert sc.attn.device_error() == 0


def test_qwen3_8b_single_sequence():
    _serving("qwen3_8b_single", check=[0], steps=2)


def test_serving_batch_32_ragged():
    sp = W.SPECS["serving_b32"]
    pre = W.serving_schedule(sp, 0, steps=1).prefill
    check = [int(np.argmax(pre)), int(np.argmin(pre)), 5]
    _serving("serving_b32", check=check, steps=3)


def test_serving_batch_32_paged():
    # the same batch over 16-row pages handed out in shuffled order
    sp = W.SPECS["serving_b32_paged"]
    pre = W.serving_schedule(sp, 0, steps=1).prefill
    check = [int(np.argmax(pre)), int(np.argmin(pre)), 11]
    _serving("serving_b32_paged", check=check, steps=2)


@pytest.mark.parametrize("name", ["long_ctx_full", "long_ctx_swa"])
def test_long_context(name):
    _serving(name, check=[2], steps=1)


def test_packed_training_full_size():
    sp = W.SPECS["packed_train"]
    seed = 0
    w = W.weights(sp, seed, with_fc=False)
    cfg, lw = T.oracle_layer(sp, w)
    attn = T.gpu_layer(sp, w)
    bs, nb, S = sp.block_size, sp.n_blocks, sp.seq
    th = torch.stack([W.hidden_rows(sp, seed, "hidden", 0, b, S) for b in range(sp.batch)])
    nz = torch.stack([W.hidden_rows(sp, seed, "noise", 0, b, nb * bs) for b in range(sp.batch)])
    anchors = W.anchors(sp, seed)
    out = attn.forward_packed(nz.cuda(), th.cuda(), anchors.cuda(), bs)
    torch.cuda.synchronize()
    got = T.f64(out)
    blocks = [0, 1, 77, 128, 200, nb - 2, nb - 1]
    ref = O.forward_packed(cfg, lw, T.f64(nz), T.f64(th), anchors.numpy(), bs,
                           seqs=[1], blocks=blocks)
    rows = np.concatenate([np.arange(k * bs, (k + 1) * bs) for k in blocks])
    T.assert_close(got[1, rows], ref[1, rows], "bf16", "packed full size")
    assert np.all(np.isfinite(got))
    assert attn.device_error() == 0


def test_ctx_project_full_size():
    sp = W.SPECS["qwen3_8b_single"]
    w = W.weights(sp, 3)
    cfg, lw = T.oracle_layer(sp, w)
    attn = T.gpu_layer(sp, w)
    for rows in (16, 300):
        x = W.target_layer_rows(sp, 3, 0, 0, rows)
        y = attn.ctx_project(x.cuda())
        torch.cuda.synchronize()
        T.assert_close(T.f64(y), O.ctx_project(cfg, lw, T.f64(x)), "bf16",
                       f"ctx_project rows={rows}")


def test_decoder_layer_full_size():
    # the whole 8B-shaped decoder layer (SwiGLU MLP of width 12288), one
    # sequence: 4096 cached rows, then a step of 16 new context rows and a
    # block with an incoming residual stream
    from block_diffusion_draft_gb300.dflash_attn import DecoderMLP
    sp = W.SPECS["decoder_8b_single"]
    seed, q, inter = 0, sp.block_size, sp.intermediate
    w = W.weights(sp, seed)
    mw = W.mlp_weights(sp, seed, inter)
    cfg, lw = T.oracle_layer(sp, w)
    om = O.MlpWeights(*(T.f64(mw[k]) for k in ("gate", "up", "down", "input_norm",
                                                 "post_norm")))
    attn = T.gpu_layer(sp, w)
    mlp = DecoderMLP(mw, sp.hidden, inter, sp.rms_eps)
    cache = T.DraftCache(attn, 1, sp.prefill + 64)
    ocache = O.DraftCache(sp.n_kv_heads, sp.head_dim, 1)
    residual = None
    for s, n_ctx in enumerate([sp.prefill, sp.n_new]):
        L0 = cache.lengths()[0]
        th = W.hidden_rows(sp, seed, "hidden", s, 0, n_ctx)
        hid = W.hidden_rows(sp, seed, "noise", s, 0, q)[None]
        pos = W.window_positions(L0, n_ctx, q)
        out, res = mlp.layer_forward(attn, cache, hid.cuda(),
                                     None if residual is None else residual.cuda(), th.cuda(),
                                     [n_ctx], pos.cuda())
        torch.cuda.synchronize()
        ref_out, ref_res = O.decoder_layer(cfg, lw, om, ocache, T.f64(hid),
                                           None if residual is None else T.f64(residual),
                                           [T.f64(th)], [pos.numpy()])
        T.assert_close_stream(res.to("cpu", torch.float64).numpy(), ref_res, f"residual {s}")
        T.assert_close_mlp(out.to("cpu", torch.float64).numpy(), ref_out, f"mlp out {s}")
        cache.crop([L0 + n_ctx])
        ocache.crop([L0 + n_ctx])
        residual = W.hidden_rows(sp, seed, "hidden", 50 + s, 0, q)[None]
    assert attn.device_error() == 0


def test_layer_group_full_size():
    # five 8B-shaped layers fed by one projected context (the bench's
    # stack5_ctx512 step): 4096 cached rows per layer, then 512 new context
    # rows appended to all five caches by one grouped projection, and each
    # layer's block; against the oracle's per-layer forward with those rows
    from block_diffusion_draft_gb300.dflash_attn import KVGroup
    sp = W.SPECS["stack5_ctx512"]
    seed, q, pre, n = 0, sp.block_size, sp.prefill, sp.n_new
    ws = [W.weights(sp, seed, layer=l, with_fc=False) for l in range(sp.layers)]
    layers = [T.gpu_layer(sp, w) for w in ws]
    refs = [T.oracle_layer(sp, w) for w in ws]
    caches = [T.DraftCache(a, 1, pre + n + 2 * q) for a in layers]
    ocaches = [O.DraftCache(sp.n_kv_heads, sp.head_dim, 1) for _ in layers]
    th0 = W.hidden_rows(sp, seed, "hidden", 1000, 0, pre)
    for l, (a, c) in enumerate(zip(layers, caches)):
        nz = W.hidden_rows(sp, seed, "noise", 1000 + l, 0, q)[None]
        pos = W.window_positions(0, pre, q)
        a.forward(c, nz.cuda(), th0.cuda(), [pre], pos.cuda())
        cfg, lw = refs[l]
        O.forward(cfg, lw, ocaches[l], T.f64(nz), [T.f64(th0)], [pos.numpy()])
        c.crop([pre])
        ocaches[l].crop([pre])
    th = W.hidden_rows(sp, seed, "hidden", 0, 0, n)
    group = KVGroup(layers)
    group.append(caches, th.cuda(), [n], torch.arange(pre, pre + n, dtype=torch.int32).cuda())
    for l, (a, c) in enumerate(zip(layers, caches)):
        nz = W.hidden_rows(sp, seed, "noise", l, 0, q)[None]
        out = a.forward(c, nz.cuda(), None, [0], W.window_positions(pre + n, 0, q).cuda())
        torch.cuda.synchronize()
        cfg, lw = refs[l]
        ref = O.forward(cfg, lw, ocaches[l], T.f64(nz), [T.f64(th)],
                        [W.window_positions(pre, n, q).numpy()])
        T.assert_close(out.to("cpu", torch.float64).numpy(), ref, "bf16", f"layer {l}")
        k, v = c.read()
        m = ocaches[l].k[0].shape[1]
        T.assert_close(T.f64(k[0][:, m - n - q:m]), ocaches[l].k[0][:, m - n - q:m], "bf16",
                       f"layer {l} K")
        T.assert_close(T.f64(v[0][:, m - n - q:m]), ocaches[l].v[0][:, m - n - q:m], "bf16",
                       f"layer {l} V")
        assert a.device_error() == 0

