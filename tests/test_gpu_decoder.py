"""Draft decoder layer ("nemo_automodel...draft_qwen3", Qwen3DFlashDecoderLayer;
"vllm...qwen3_dflash", the residual-stream draft model) against the oracle:
input norm, DFlash attention, residual add, post-attention norm and the
SwiGLU MLP, with and without an incoming residual."""
import numpy as np
import pytest
import torch

from block_diffusion_draft_gb300 import workloads as W
from block_diffusion_draft_gb300.dflash_attn import DecoderMLP, DraftCache
from oracle import dflash_oracle as O
import helpers as T

pytestmark = pytest.mark.gpu


def small_bf16(**kw):
    base = dict(hidden=1024, n_heads=8, n_kv_heads=2, head_dim=128, batch=3,
                n_target_layers=2, max_position=8192)
    base.update(kw)
    return W.spec("qwen3_8b_single", **base)


assert_close_stream = T.assert_close_stream


def oracle_mlp(w):
    f = T.f64
    return O.MlpWeights(gate=f(w["gate"]), up=f(w["up"]), down=f(w["down"]),
                        input_norm=f(w["input_norm"]), post_norm=f(w["post_norm"]))


# batch 3: 48 rows (decode-size GEMMs); batch 12: 192 rows (persistent SwiGLU
# projection, swapped-operand down projection)
@pytest.mark.parametrize("batch,steps", [(3, ([40, 7, 130], [5, 16, 0])),
                                         (12, ([16] * 12, list(range(12))))])
def test_decoder_layer_matches_oracle(batch, steps):
    sp = small_bf16(batch=batch)
    B, q, seed, inter = sp.batch, sp.block_size, 31, 3072
    w = W.weights(sp, seed, random_gains=True)
    mw = W.mlp_weights(sp, seed, inter, random_gains=True)
    cfg, lw = T.oracle_layer(sp, w)
    om = oracle_mlp(mw)
    attn = T.gpu_layer(sp, w)
    mlp = DecoderMLP(mw, sp.hidden, inter, sp.rms_eps)
    cache = DraftCache(attn, B, 512)
    ocache = O.DraftCache(sp.n_kv_heads, sp.head_dim, B)
    residual = None
    for s, n_ctx in enumerate(steps):
        L0 = cache.lengths()
        th = [W.hidden_rows(sp, seed, "hidden", s, b, n_ctx[b]) for b in range(B)]
        hid = torch.stack([W.hidden_rows(sp, seed, "noise", s, b, q) for b in range(B)])
        pos = [W.window_positions(L0[b], n_ctx[b], q) for b in range(B)]
        target = torch.cat(th).cuda() if sum(n_ctx) > 0 else None
        out, res = mlp.layer_forward(attn, cache, hid.cuda(),
                                     None if residual is None else residual.cuda(), target,
                                     n_ctx, torch.cat(pos).cuda())
        torch.cuda.synchronize()
        ref_out, ref_res = O.decoder_layer(cfg, lw, om, ocache, T.f64(hid),
                                           None if residual is None else T.f64(residual),
                                           [T.f64(x) for x in th], [p.numpy() for p in pos])
        assert_close_stream(res.to("cpu", torch.float64).numpy(), ref_res, f"residual {s}")
        T.assert_close_mlp(out.to("cpu", torch.float64).numpy(), ref_out, f"mlp out {s}")
        k, v = cache.read()
        k = k.to("cpu", torch.float64).numpy()
        for b in range(B):
            n = ocache.k[b].shape[1]
            T.assert_close(k[b][:, :n], ocache.k[b], "bf16", "cache K")
        assert attn.device_error() == 0
        keep = [L0[b] + n_ctx[b] for b in range(B)]
        cache.crop(keep)
        ocache.crop(keep)
        # the next step gets a residual stream (bf16, as the GPU keeps it)
        residual = torch.stack([W.hidden_rows(sp, seed, "hidden", 50 + s, b, q)
                                for b in range(B)])
