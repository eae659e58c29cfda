"""Packed training layout: attention core forward (output and log-sum-exp) and
backward (dQ, dK, dV through the anchor mask; "nemo_automodel...draft_qwen3",
module docstring) against the oracle's fp64 core and its written-out chain
rule.

Tolerance reading for gradients: the kernels round Q' (Q times scale and
log2 e), P and dS to bf16 for the tensor cores and store bf16 results, so a
gradient element carries a relative error of a few bf16 ulps of its own
magnitude; gradient rows that sum many terms (dK, dV of early context keys,
read by every block) reach |g| of several units, where one bf16 ulp is
already 2^-7.  The max-abs bound (2e-2) is therefore applied per element
relative to max(1, |ref|); the relative L2 bound (5e-3) is the one used for
every bf16 output."""
import numpy as np
import pytest
import torch

from block_diffusion_draft_gb300 import workloads as W
from oracle import dflash_oracle as O
import helpers as T

pytestmark = pytest.mark.gpu


def assert_close_grad(gpu, ref, what):
    gpu, ref = np.asarray(gpu, np.float64), np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    scaled = float(np.max(np.abs(gpu - ref) / np.maximum(1.0, np.abs(ref))))
    rel = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-300))
    T._log(what, "bf16", scaled, rel)
    assert scaled <= T.BF16_MAX_ABS and rel <= T.BF16_REL_L2, \
        f"{what}: scaled max={scaled:.3e} rel_l2={rel:.3e}"


def core_spec(**kw):
    base = dict(hidden=1024, n_heads=8, n_kv_heads=2, head_dim=128, batch=2,
                seq=300, n_blocks=5, block_size=16)
    base.update(kw)
    return W.spec("packed_train", **base)


def oracle_cfg(sp, n_heads=None, n_kv=None):
    return O.LayerConfig(hidden=sp.hidden, n_heads=n_heads or sp.n_heads,
                         n_kv_heads=n_kv or sp.n_kv_heads, head_dim=sp.head_dim,
                         rms_eps=sp.rms_eps, rope_theta=sp.rope_theta,
                         n_target_layers=0)


def gpu_layer(sp):
    w = W.weights(sp, 3, with_fc=False)
    return T.gpu_layer(sp, w)


def run_gpu(attn, sp, x, anchors):
    q, k, v, d_o = (x[n].cuda() for n in ("q", "k", "v", "d_out"))
    an = anchors.cuda()
    out, lse = attn.packed_core(q, k, v, an, sp.seq, sp.block_size)
    dq, dk, dv = attn.packed_core_backward(q, k, v, out, lse, d_o, an, sp.seq,
                                           sp.block_size)
    torch.cuda.synchronize()
    return [t.to("cpu", torch.float64).numpy() for t in (out, lse, dq, dk, dv)]


def check_pair(sp, x, anchors, got, b, kv):
    """Compare the query heads of kv head `kv` of sequence b (and that kv
    head's dK, dV) with the oracle."""
    out, lse, dq, dk, dv = got
    g = sp.n_heads // sp.n_kv_heads
    heads = slice(kv * g, (kv + 1) * g)
    cfg = oracle_cfg(sp, n_heads=g, n_kv=1)
    q = T.f64(x["q"][b, :, heads]).transpose(1, 0, 2)
    k = T.f64(x["k"][b, kv:kv + 1])
    v = T.f64(x["v"][b, kv:kv + 1])
    d_o = T.f64(x["d_out"][b, :, heads]).transpose(1, 0, 2)
    an = anchors[b].numpy()
    o_ref, lse_ref = O.packed_core(cfg, q, k, v, an, sp.seq, sp.block_size)
    dq_ref, dk_ref, dv_ref = O.packed_core_backward(cfg, q, k, v, an, sp.seq, sp.block_size,
                                                    d_o)
    T.assert_close(out[b, :, heads].transpose(1, 0, 2), o_ref, "bf16", f"out b{b} h{kv}")
    assert_close_grad(dq[b, :, heads].transpose(1, 0, 2), dq_ref, f"dq b{b} h{kv}")
    assert_close_grad(dk[b, kv], dk_ref[0], f"dk b{b} h{kv}")
    assert_close_grad(dv[b, kv], dv_ref[0], f"dv b{b} h{kv}")
    # log-sum-exp: the scores come from q * scale * log2(e) rounded to bf16
    # (relative 2^-9 per element), which moves a score by about
    # 2^-9 * scale * sqrt(sum_d (q_d k_d)^2) ~ 2e-3 (log2 units) and the
    # log-sum-exp, a softmax-weighted mean of those shifts, by a few 1e-3
    np.testing.assert_allclose(lse[b, :, heads].T, lse_ref, rtol=0, atol=1e-2)


# seq 300: a ragged last context tile (and 64-key steps); 5 blocks: the last
# dQ unit holds one block; anchors include 0 (own block only), seq (all
# context) and unsorted values; the second case has a context tile no block
# sees (its dK, dV rows must be 0)
@pytest.mark.parametrize("seq,n_blocks,anchors", [
    (300, 5, [[0, 300, 17, 128, 129], [255, 64, 1, 299, 200]]),
    (500, 6, [[3, 60, 100, 5, 128, 64], [0, 0, 250, 1, 2, 130]]),
])
def test_packed_core_matches_oracle(seq, n_blocks, anchors):
    sp = core_spec(seq=seq, n_blocks=n_blocks)
    x = W.core_tensors(sp, seed=5)
    an = torch.tensor(anchors, dtype=torch.int32)
    attn = gpu_layer(sp)
    got = run_gpu(attn, sp, x, an)
    for b in range(sp.batch):
        for kv in range(sp.n_kv_heads):
            check_pair(sp, x, an, got, b, kv)
    # context keys at or past a sequence's largest anchor are seen by no
    # block: exactly zero gradients (for seq 500 the whole last tile)
    for b in range(sp.batch):
        top = max(anchors[b])
        assert np.all(got[3][b, :, top:seq] == 0) and np.all(got[4][b, :, top:seq] == 0)
    assert attn.device_error() == 0


def test_packed_core_backward_is_deterministic():
    sp = core_spec()
    x = W.core_tensors(sp, seed=6)
    an = torch.tensor([[0, 300, 17, 128, 129], [255, 64, 1, 299, 200]], dtype=torch.int32)
    attn = gpu_layer(sp)
    a = run_gpu(attn, sp, x, an)
    b = run_gpu(attn, sp, x, an)
    for u, w in zip(a, b):
        assert np.array_equal(u, w)


def test_packed_core_full_size_sampled():
    # the bench's training shape (2 x 4096 context rows, 256 blocks of 16,
    # 32/8 heads): one (sequence, kv head) group checked in full
    sp = W.spec("packed_train")
    x = W.core_tensors(sp, seed=0)
    an = W.anchors(sp, 0)
    attn = gpu_layer(sp)
    got = run_gpu(attn, sp, x, an)
    check_pair(sp, x, an, got, 1, 5)
    assert attn.device_error() == 0


def test_packed_core_rejects_unsupported_shapes():
    from block_diffusion_draft_gb300.dflash_attn import DFlashError
    sp = core_spec(block_size=8, n_blocks=4)
    attn = gpu_layer(sp)
    x = W.core_tensors(sp, seed=1)
    an = torch.zeros(sp.batch, sp.n_blocks, dtype=torch.int32).cuda()
    with pytest.raises(DFlashError):  # groups * block_size = 32
        attn.packed_core(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), an, sp.seq, 8)
