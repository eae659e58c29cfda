"""Context K/V of several layers from one projection ("vllm...qwen3_dflash",
precompute_and_store_context_kv), checked against the oracle's per-layer
forward: appending the context rows of every layer through one grouped
projection and then running each layer's forward with no context rows must
give the outputs and caches of the plain per-layer forward with those rows."""
import numpy as np
import pytest
import torch

from block_diffusion_draft_gb300 import workloads as W
from block_diffusion_draft_gb300.dflash_attn import DFlashError, DraftCache, KVGroup
from oracle import dflash_oracle as O
import helpers as T

pytestmark = pytest.mark.gpu


def small_bf16(**kw):
    base = dict(hidden=1024, n_heads=8, n_kv_heads=2, head_dim=128, batch=3,
                n_target_layers=2, max_position=8192)
    base.update(kw)
    return W.spec("qwen3_8b_single", **base)


# (layers, context rows per sequence of the first and second step): the first
# step's 177 rows take the persistent projection kernel, the second's <= 128
# rows the decode-size kernel
@pytest.mark.parametrize("n_layers,steps", [(3, ([40, 7, 130], [5, 16, 0])),
                                            (5, ([16, 16, 16], [1, 9, 3]))])
def test_kv_group_matches_per_layer_forward(n_layers, steps):
    sp = small_bf16()
    B, q, seed = sp.batch, sp.block_size, 21
    ws = [W.weights(sp, seed, layer=l) for l in range(n_layers)]
    layers = [T.gpu_layer(sp, w) for w in ws]
    refs = [T.oracle_layer(sp, w) for w in ws]
    caches = [DraftCache(a, B, 512) for a in layers]
    ocaches = [O.DraftCache(sp.n_kv_heads, sp.head_dim, B) for _ in range(n_layers)]
    group = KVGroup(layers)
    for s, n_ctx in enumerate(steps):
        L0 = caches[0].lengths()
        th = [W.hidden_rows(sp, seed, "hidden", s, b, n_ctx[b]) for b in range(B)]
        pos_ctx = torch.cat([torch.arange(L0[b], L0[b] + n_ctx[b], dtype=torch.int32)
                             for b in range(B)])
        target = torch.cat(th).cuda() if sum(n_ctx) > 0 else None
        group.append(caches, target, n_ctx, pos_ctx.cuda())
        assert caches[-1].lengths() == [L0[b] + n_ctx[b] for b in range(B)]
        for l in range(n_layers):
            nz = [W.hidden_rows(sp, seed, "noise", 100 * s + l, b, q) for b in range(B)]
            pos_blk = torch.cat([W.window_positions(L0[b] + n_ctx[b], 0, q) for b in range(B)])
            out = layers[l].forward(caches[l], torch.stack(nz).cuda(), None, [0] * B,
                                    pos_blk.cuda())
            torch.cuda.synchronize()
            cfg, lw = refs[l]
            ref = O.forward(cfg, lw, ocaches[l], np.stack([T.f64(x) for x in nz]),
                            [T.f64(x) for x in th],
                            [W.window_positions(L0[b], n_ctx[b], q).numpy() for b in range(B)])
            T.assert_close(out.to("cpu", torch.float64).numpy(), ref, "bf16",
                           f"layer {l} step {s}")
            k, v = caches[l].read()
            k = k.to("cpu", torch.float64).numpy()
            v = v.to("cpu", torch.float64).numpy()
            for b in range(B):
                n = ocaches[l].k[b].shape[1]
                T.assert_close(k[b][:, :n], ocaches[l].k[b], "bf16", f"layer {l} K")
                T.assert_close(v[b][:, :n], ocaches[l].v[b], "bf16", f"layer {l} V")
            assert layers[l].device_error() == 0
        # keep the context rows, drop the block rows (as after verification)
        keep = [L0[b] + n_ctx[b] for b in range(B)]
        for c in caches:
            c.crop(keep)
        for oc in ocaches:
            oc.crop(keep)


def test_kv_group_rejects_mismatched_caches():
    sp = small_bf16(batch=2)
    ws = [W.weights(sp, 3, layer=l) for l in range(2)]
    layers = [T.gpu_layer(sp, w) for w in ws]
    caches = [DraftCache(a, 2, 64) for a in layers]
    group = KVGroup(layers)
    th = W.hidden_rows(sp, 3, "hidden", 0, 0, 4).cuda()
    pos = torch.arange(0, 4, dtype=torch.int32).cuda()
    # different lengths across the caches
    layers[0].forward(caches[0], torch.stack([W.hidden_rows(sp, 3, "noise", 0, b, 16)
                                              for b in range(2)]).cuda(),
                      None, [0, 0], torch.arange(0, 32, dtype=torch.int32).cuda())
    with pytest.raises(DFlashError):
        group.append(caches, th, [4, 0], pos)
    caches[0].crop([0, 0])
    # a cache that would overflow: nothing is appended
    with pytest.raises(DFlashError):
        group.append(caches, W.hidden_rows(sp, 3, "hidden", 0, 0, 65).cuda(), [65, 0],
                     torch.arange(0, 65, dtype=torch.int32).cuda())
    assert caches[0].lengths() == [0, 0] and caches[1].lengths() == [0, 0]
    group.append(caches, th, [4, 0], pos)
    assert caches[1].lengths() == [4, 0]
