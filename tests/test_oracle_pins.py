"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test checks one part of the oracle against a closed form, an invariant
the pages state, a library routine, or a brute-force restatement on tiny
inputs, chosen so that a plausible slip (a dropped term, a wrong sign or
index, a transposed operand, a causal mask, the wrong GQA head, prefix
instead of suffix positions, a wrong crop) fails at least one of them.
The test ``test_pins_catch_planted_mistakes`` plants such slips in a copy of
the oracle and checks that the pins notice.
"""
import math

import numpy as np
import pytest
import torch

from oracle import dflash_oracle as O

RNG = np.random.default_rng(1234)


def tiny_cfg(**kw):
    base = dict(hidden=64, n_heads=4, n_kv_heads=2, head_dim=16,
                rms_eps=1e-6, rope_theta=1e4, n_target_layers=2)
    base.update(kw)
    return O.LayerConfig(**base)


def tiny_weights(cfg, rng=None, gains=True):
    rng = RNG if rng is None else rng
    H, d = cfg.hidden, cfg.head_dim
    g = (lambda n: 1.0 + 0.3 * rng.standard_normal(n)) if gains else np.ones
    return O.LayerWeights(
        wq=0.2 * rng.standard_normal((cfg.n_heads * d, H)),
        wk=0.2 * rng.standard_normal((cfg.n_kv_heads * d, H)),
        wv=0.2 * rng.standard_normal((cfg.n_kv_heads * d, H)),
        wo=0.2 * rng.standard_normal((H, cfg.n_heads * d)),
        q_norm=g(d), k_norm=g(d),
        fc=0.2 * rng.standard_normal((H, cfg.n_target_layers * H)),
        hidden_norm=g(H))


# --------------------------------------------------------------------------
# RMSNorm: closed forms
# --------------------------------------------------------------------------
def test_rms_norm_constant_vector_closed_form():
    # x = c * 1  ->  w * c / sqrt(c^2 + eps); a small c makes eps matter
    d = 32
    w = RNG.standard_normal(d)
    for c, eps in ((3.0, 1e-6), (-2.5, 1e-6), (1e-3, 1e-6), (0.0, 1e-6)):
        got = O.rms_norm(np.full(d, c), w, eps)
        want = w * c / math.sqrt(c * c + eps)
        np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-300)


def test_rms_norm_unit_rms_output():
    # with unit gain and eps = 0 the output has mean square exactly 1
    x = RNG.standard_normal((5, 128))
    y = O.rms_norm(x, np.ones(128), 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-13)
    # and is a positive multiple of the input row
    ratio = y / x
    np.testing.assert_allclose(ratio, ratio[:, :1] * np.ones((1, 128)), rtol=1e-12)
    assert np.all(ratio > 0)


# --------------------------------------------------------------------------
# RoPE: closed forms and invariants
# --------------------------------------------------------------------------
def _f32(x):
    return float(np.float32(x))


def test_rope_frequencies_fp32_values():
    d, theta = 128, 1e6
    f = O.rope_frequencies(d, theta)
    assert f.shape == (64,) and f[0] == 1.0
    for j in (1, 7, 31, 63):
        # the fp32 number nearest theta^(-2j/d), computed here with math.pow
        assert f[j] == _f32(math.pow(theta, -2.0 * j / d))
    assert np.all(np.diff(f) < 0)
    # every value is exactly an fp32 number
    assert np.all(f.astype(np.float32).astype(np.float64) == f)


def test_rope_basis_vectors_rotate_half_pairs():
    # NeoX rotate-half: e_j turns toward e_{j+d/2} by angle p*f_j
    d, theta = 16, 1e4
    f = O.rope_frequencies(d, theta)
    h = d // 2
    for p in (0, 1, 5, 1000):
        for j in range(h):
            ej = np.zeros((1, d)); ej[0, j] = 1.0
            ek = np.zeros((1, d)); ek[0, j + h] = 1.0
            a = p * f[j]
            rj = O.rope(ej, np.array([p]), f)[0]
            rk = O.rope(ek, np.array([p]), f)[0]
            wj = np.zeros(d); wj[j] = math.cos(a); wj[j + h] = math.sin(a)
            wk = np.zeros(d); wk[j] = -math.sin(a); wk[j + h] = math.cos(a)
            np.testing.assert_allclose(rj, wj, atol=1e-15)
            np.testing.assert_allclose(rk, wk, atol=1e-15)


def test_rope_identity_at_zero_and_norm_preserving():
    d = 32
    f = O.rope_frequencies(d, 1e6)
    x = RNG.standard_normal((7, d))
    np.testing.assert_array_equal(O.rope(x, np.zeros(7, int), f), x)
    y = O.rope(x, np.arange(7) * 977, f)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1),
                               np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rope_dot_product_depends_on_offset_only():
    d = 64
    f = O.rope_frequencies(d, 1e6)
    q, k = RNG.standard_normal((1, d)), RNG.standard_normal((1, d))
    base = (O.rope(q, np.array([40]), f) @ O.rope(k, np.array([3]), f).T)[0, 0]
    for c in (1, 1000, 30000):
        s = (O.rope(q, np.array([40 + c]), f) @ O.rope(k, np.array([3 + c]), f).T)[0, 0]
        assert abs(s - base) < 1e-9


# --------------------------------------------------------------------------
# linear: nn.Linear convention against explicit sums
# --------------------------------------------------------------------------
def test_linear_is_x_times_w_transposed():
    x = RNG.standard_normal((3, 5))
    w = RNG.standard_normal((4, 5))  # [out, in]
    y = O.linear(x, w)
    for r in range(3):
        for o in range(4):
            assert abs(y[r, o] - sum(x[r, i] * w[o, i] for i in range(5))) < 1e-13


# --------------------------------------------------------------------------
# attention core: softmax closed forms
# --------------------------------------------------------------------------
def test_attention_constant_values_give_that_constant():
    # softmax rows sum to one: if every value row is c, every output is c
    cfg = tiny_cfg()
    q = RNG.standard_normal((4, 5, 16))
    k = RNG.standard_normal((2, 9, 16))
    c = RNG.standard_normal(16)
    v = np.broadcast_to(c, (2, 9, 16)).copy()
    allowed = RNG.random((5, 9)) < 0.6
    allowed[:, 0] = True
    out = O.attention(cfg, q, k, v, allowed)
    np.testing.assert_allclose(out.reshape(5, 4, 16), np.broadcast_to(c, (5, 4, 16)),
                               rtol=1e-13, atol=1e-13)


def test_attention_equal_keys_give_mean_of_allowed_values():
    cfg = tiny_cfg()
    q = RNG.standard_normal((4, 3, 16))
    k = np.broadcast_to(RNG.standard_normal(16), (2, 6, 16)).copy()
    v = RNG.standard_normal((2, 6, 16))
    allowed = np.array([[1, 1, 1, 1, 1, 1], [1, 0, 1, 0, 1, 0], [0, 0, 0, 0, 0, 1]], bool)
    out = O.attention(cfg, q, k, v, allowed).reshape(3, 4, 16)
    for h in range(4):
        for r in range(3):
            want = v[h // 2][allowed[r]].mean(axis=0)
            np.testing.assert_allclose(out[r, h], want, rtol=1e-13, atol=1e-14)


def test_attention_matches_library_sdpa_with_repeat_kv():
    # textbook scaled-dot-product attention (torch, fp64) with KV heads
    # repeated as transformers' repeat_kv does: query head h uses kv h // g
    cfg = tiny_cfg()
    q = RNG.standard_normal((4, 6, 16))
    k = RNG.standard_normal((2, 11, 16))
    v = RNG.standard_normal((2, 11, 16))
    allowed = RNG.random((6, 11)) < 0.7
    allowed[:, 3] = True
    out = O.attention(cfg, q, k, v, allowed)
    tq = torch.from_numpy(q)[None]
    tk = torch.from_numpy(np.repeat(k, 2, axis=0))[None]
    tv = torch.from_numpy(np.repeat(v, 2, axis=0))[None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=torch.from_numpy(allowed))[0]
    ref = ref.permute(1, 0, 2).reshape(6, 64).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# masks: the pages' rules restated element by element
# --------------------------------------------------------------------------
def test_band_mask_elementwise_rule():
    for q_len, k_len, W in ((4, 10, 3), (16, 40, 7), (3, 3, 1), (5, 12, 100)):
        m = O.band_mask(q_len, k_len, W)
        for i in range(q_len):
            for j in range(k_len):
                qi = k_len - q_len + i  # query row i sits at this key index
                assert m[i, j] == (-W < j - qi < W)


def test_anchor_mask_elementwise_rule():
    S, bs, anchors = 12, 3, [1, 5, 12, 7]
    m = O.anchor_mask(S, anchors, bs)
    for qb, a in enumerate(anchors):
        for t in range(bs):
            for j in range(S + len(anchors) * bs):
                in_ctx = j < S and j < a
                own = S + qb * bs <= j < S + (qb + 1) * bs
                assert m[qb * bs + t, j] == (in_ctx or own)


# --------------------------------------------------------------------------
# the layer: brute force over the surviving history
# --------------------------------------------------------------------------
def _brute_force_step(cfg, w, history, noise_b, pos_block):
    """Output of one block given every surviving (row, position) of the
    sequence, recomputing each key/value row from its own input row.

    Independent bookkeeping: explicit key list in append order, explicit
    per-key loops, explicit repeat of KV heads, scaling = 1/sqrt(d).
    """
    d, g = cfg.head_dim, cfg.n_heads // cfg.n_kv_heads
    f = O.rope_frequencies(d, cfg.rope_theta)
    keys, vals = [], []
    for row, p in history:
        kr = O.linear(row[None], w.wk)[0].reshape(cfg.n_kv_heads, d)
        vr = O.linear(row[None], w.wv)[0].reshape(cfg.n_kv_heads, d)
        kr = np.stack([O.rope(O.rms_norm(kr[h][None], w.k_norm, cfg.rms_eps),
                              np.array([p]), f)[0] for h in range(cfg.n_kv_heads)])
        keys.append(kr); vals.append(vr)
    k_len, q_len = len(keys), noise_b.shape[0]
    out = np.zeros((q_len, cfg.n_heads * d))
    for t in range(q_len):
        qr = O.linear(noise_b[t][None], w.wq)[0].reshape(cfg.n_heads, d)
        qi = k_len - q_len + t
        for h in range(cfg.n_heads):
            qh = O.rope(O.rms_norm(qr[h][None], w.q_norm, cfg.rms_eps),
                        np.array([pos_block[t]]), f)[0]
            s = []
            for j in range(k_len):
                if cfg.sliding_window and not abs(j - qi) < cfg.sliding_window:
                    continue
                s.append((sum(qh[e] * keys[j][h // g][e] for e in range(d))
                          / math.sqrt(d), j))
            mx = max(x for x, _ in s)
            z = sum(math.exp(x - mx) for x, _ in s)
            for x, j in s:
                out[t, h * d:(h + 1) * d] += math.exp(x - mx) / z * vals[j][h // g]
    return O.linear(out, w.wo)


def _run_two_steps(cfg, w, rng, n0=5, n1=3, q_len=4, accept_crop=True):
    """Prefill step then a second step on a batch of two sequences; returns
    the oracle output of the second step and the history of seq 1."""
    B, H = 2, cfg.hidden
    cache = O.DraftCache(cfg.n_kv_heads, cfg.head_dim, B)
    hist = {b: [] for b in range(B)}
    th0 = [rng.standard_normal((n0 + b, H)) for b in range(B)]
    nz0 = rng.standard_normal((B, q_len, H))
    pos0 = [np.arange(n0 + b + q_len) for b in range(B)]
    O.forward(cfg, w, cache, nz0, th0, pos0)
    for b in range(B):
        hist[b] = [(th0[b][i], i) for i in range(n0 + b)]
        hist[b] += [(nz0[b][t], n0 + b + t) for t in range(q_len)]
    if accept_crop:
        cache.crop([n0 + b for b in range(B)])      # drop the noise rows
        for b in range(B):
            hist[b] = hist[b][:n0 + b]
    th1 = [rng.standard_normal((n1, H)) for b in range(B)]
    nz1 = rng.standard_normal((B, q_len, H))
    L = cache.lengths()
    pos1 = [np.arange(L[b], L[b] + n1 + q_len) for b in range(B)]
    out = O.forward(cfg, w, cache, nz1, th1, pos1)
    for b in range(B):
        hist[b] += [(th1[b][i], L[b] + i) for i in range(n1)]
        hist[b] += [(nz1[b][t], L[b] + n1 + t) for t in range(q_len)]
    return out, hist, nz1, pos1, n1


@pytest.mark.parametrize("window", [0, 4])
@pytest.mark.parametrize("crop", [True, False])
def test_forward_matches_brute_force(window, crop):
    rng = np.random.default_rng(7)
    cfg = tiny_cfg(hidden=32, head_dim=8, sliding_window=window)
    w = tiny_weights(cfg, rng)
    out, hist, nz1, pos1, n1 = _run_two_steps(cfg, w, rng, accept_crop=crop)
    for b in range(2):
        want = _brute_force_step(cfg, w, hist[b], nz1[b], pos1[b][n1:])
        np.testing.assert_allclose(out[b], want, rtol=1e-10, atol=1e-12)


def test_forward_is_permutation_equivariant_over_block_rows():
    # non-causal: permuting the block's rows together with their positions
    # permutes the output rows (a causal mask would break this)
    rng = np.random.default_rng(11)
    cfg = tiny_cfg()
    w = tiny_weights(cfg, rng)
    H, q_len, n = cfg.hidden, 6, 7
    th = [rng.standard_normal((n, H))]
    nz = rng.standard_normal((1, q_len, H))
    pos = [np.arange(n + q_len)]
    c1 = O.DraftCache(cfg.n_kv_heads, cfg.head_dim, 1)
    out = O.forward(cfg, w, c1, nz, th, pos)
    perm = np.array([3, 0, 5, 1, 4, 2])
    c2 = O.DraftCache(cfg.n_kv_heads, cfg.head_dim, 1)
    pos2 = [np.concatenate([pos[0][:n], pos[0][n:][perm]])]
    out2 = O.forward(cfg, w, c2, nz[:, perm], th, pos2)
    np.testing.assert_allclose(out2[0], out[0][perm], rtol=1e-12, atol=1e-13)


def test_forward_invariant_under_common_position_shift():
    rng = np.random.default_rng(13)
    cfg = tiny_cfg(rope_theta=1e6)
    w = tiny_weights(cfg, rng)
    H, q_len, n = cfg.hidden, 4, 9
    th = [rng.standard_normal((n, H))]
    nz = rng.standard_normal((1, q_len, H))
    outs = []
    for c in (0, 1, 1000):
        cache = O.DraftCache(cfg.n_kv_heads, cfg.head_dim, 1)
        outs.append(O.forward(cfg, w, cache, nz, th, [np.arange(n + q_len) + c]))
    for o in outs[1:]:
        np.testing.assert_allclose(o, outs[0], rtol=1e-9, atol=1e-10)


def test_gqa_equals_mha_with_repeated_kv_weights():
    rng = np.random.default_rng(17)
    cfg = tiny_cfg()
    w = tiny_weights(cfg, rng)
    d, g = cfg.head_dim, cfg.groups
    rep = lambda m: np.concatenate([m[(h // g) * d:(h // g + 1) * d]
                                    for h in range(cfg.n_heads)])
    cfg_mha = tiny_cfg(n_kv_heads=cfg.n_heads)
    w_mha = O.LayerWeights(wq=w.wq, wk=rep(w.wk), wv=rep(w.wv), wo=w.wo,
                           q_norm=w.q_norm, k_norm=w.k_norm)
    H, q_len, n = cfg.hidden, 4, 6
    th = [rng.standard_normal((n, H))]
    nz = rng.standard_normal((1, q_len, H))
    pos = [np.arange(n + q_len)]
    a = O.forward(cfg, w, O.DraftCache(2, d, 1), nz, th, pos)
    b = O.forward(cfg_mha, w_mha, O.DraftCache(4, d, 1), nz, th, pos)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)


def test_empty_context_is_plain_bidirectional_attention():
    # ctx_len = 0 and an empty cache: the layer is textbook non-causal
    # self-attention over the block, checked against torch SDPA (fp64)
    rng = np.random.default_rng(19)
    cfg = tiny_cfg()
    w = tiny_weights(cfg, rng)
    H, q_len = cfg.hidden, 5
    nz = rng.standard_normal((1, q_len, H))
    pos = np.arange(q_len) + 3
    out = O.forward(cfg, w, O.DraftCache(2, 16, 1), nz, [np.zeros((0, H))], [pos])
    q = O.project_q(cfg, w, nz[0], pos)
    k, v = O.project_kv(cfg, w, nz[0], pos)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x))[None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        t(q), t(np.repeat(k, 2, 0)), t(np.repeat(v, 2, 0)), is_causal=False)[0]
    ref = ref.permute(1, 0, 2).reshape(q_len, -1).numpy() @ w.wo.T
    np.testing.assert_allclose(out[0], ref, rtol=1e-12, atol=1e-13)


def test_wide_window_equals_full_attention():
    rng = np.random.default_rng(23)
    cfg_f = tiny_cfg()
    cfg_w = tiny_cfg(sliding_window=10_000)
    w = tiny_weights(cfg_f, rng)
    out_f, *_ = _run_two_steps(cfg_f, w, np.random.default_rng(5))
    out_w, *_ = _run_two_steps(cfg_w, w, np.random.default_rng(5))
    np.testing.assert_array_equal(out_f, out_w)


def test_band_hides_far_keys():
    # keys outside the band may be replaced by anything: output unchanged
    cfg = tiny_cfg(sliding_window=3)
    q = RNG.standard_normal((4, 4, 16))
    k = RNG.standard_normal((2, 12, 16))
    v = RNG.standard_normal((2, 12, 16))
    m = O.band_mask(4, 12, 3)
    a = O.attention(cfg, q, k, v, m)
    far = ~m.any(axis=0)
    assert far.any()
    k2, v2 = k.copy(), v.copy()
    k2[:, far] = 1e3 * RNG.standard_normal((2, far.sum(), 16))
    v2[:, far] = 1e3
    np.testing.assert_array_equal(a, O.attention(cfg, q, k2, v2, m))


# --------------------------------------------------------------------------
# packed training layout
# --------------------------------------------------------------------------
def test_packed_matches_explicit_anchor_mask_over_all_keys():
    rng = np.random.default_rng(29)
    cfg = tiny_cfg()
    w = tiny_weights(cfg, rng)
    S, bs, anchors = 10, 3, np.array([[1, 4, 9, 10], [2, 3, 7, 8]])
    B, nb, H = 2, 4, cfg.hidden
    th = rng.standard_normal((B, S, H))
    nz = rng.standard_normal((B, nb * bs, H))
    out = O.forward_packed(cfg, w, nz, th, anchors, bs)
    for b in range(B):
        pos_q = np.concatenate([a + np.arange(bs) for a in anchors[b]])
        kc, vc = O.project_kv(cfg, w, th[b], np.arange(S))
        kn, vn = O.project_kv(cfg, w, nz[b], pos_q)
        q = O.project_q(cfg, w, nz[b], pos_q)
        k = np.concatenate([kc, kn], 1); v = np.concatenate([vc, vn], 1)
        o = O.attention(cfg, q, k, v, O.anchor_mask(S, anchors[b], bs))
        np.testing.assert_allclose(out[b], o @ w.wo.T, rtol=1e-12, atol=1e-13)


def test_packed_single_block_at_end_equals_cache_path():
    # one block anchored at S sees every context row: the inference step with
    # those S rows as context (positions 0..S-1, block at S..S+bs-1)
    rng = np.random.default_rng(31)
    cfg = tiny_cfg()
    w = tiny_weights(cfg, rng)
    S, bs, H = 9, 4, cfg.hidden
    th = rng.standard_normal((1, S, H))
    nz = rng.standard_normal((1, bs, H))
    a = O.forward_packed(cfg, w, nz, th, np.array([[S]]), bs)
    b = O.forward(cfg, w, O.DraftCache(2, 16, 1), nz, [th[0]], [np.arange(S + bs)])
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)


# --------------------------------------------------------------------------
# cache bookkeeping
# --------------------------------------------------------------------------
def test_crop_then_reappend_reproduces_cache_bitwise():
    rng = np.random.default_rng(37)
    cfg = tiny_cfg()
    w = tiny_weights(cfg, rng)
    H = cfg.hidden
    th = [rng.standard_normal((8, H))]
    nz = rng.standard_normal((1, 4, H))
    pos = [np.arange(12)]
    c1 = O.DraftCache(2, 16, 1)
    O.forward(cfg, w, c1, nz, th, pos)
    k_full, v_full = c1.k[0].copy(), c1.v[0].copy()
    c1.crop([5])
    assert c1.lengths() == [5]
    np.testing.assert_array_equal(c1.k[0], k_full[:, :5])
    # re-append rows 5.. of the same inputs at the same positions
    kk, vv = O.project_kv(cfg, w, np.concatenate([th[0][5:], nz[0]]), np.arange(5, 12))
    c1.append(0, kk, vv)
    np.testing.assert_array_equal(c1.k[0], k_full)
    np.testing.assert_array_equal(c1.v[0], v_full)


def test_crop_out_of_range_is_an_error_and_same_length_is_noop():
    c = O.DraftCache(2, 4, 2)
    c.append(0, np.ones((2, 3, 4)), np.ones((2, 3, 4)))
    with pytest.raises(ValueError):
        c.crop([4, 0])
    with pytest.raises(ValueError):
        c.crop([-1, 0])
    c.crop([3, 0])
    assert c.lengths() == [3, 0]


# --------------------------------------------------------------------------
# context projection
# --------------------------------------------------------------------------
def test_ctx_project_is_norm_of_fc_and_checks_width():
    rng = np.random.default_rng(41)
    cfg = tiny_cfg()
    w = tiny_weights(cfg, rng)
    x = rng.standard_normal((3, 2 * cfg.hidden))
    y = O.ctx_project(cfg, w, x)
    for r in range(3):
        z = np.array([sum(x[r, i] * w.fc[o, i] for i in range(x.shape[1]))
                      for o in range(cfg.hidden)])
        want = w.hidden_norm * z / math.sqrt(sum(t * t for t in z) / len(z) + cfg.rms_eps)
        np.testing.assert_allclose(y[r], want, rtol=1e-12)
    with pytest.raises(ValueError):
        O.ctx_project(cfg, w, x[:, :-1])


# --------------------------------------------------------------------------
# the pins catch plausible slips
# --------------------------------------------------------------------------
# --------------------------------------------------------------------------
# causal layers
# --------------------------------------------------------------------------
def test_causal_mask_elementwise_rule():
    m = O.causal_mask(3, 7)
    for i in range(3):
        for j in range(7):
            assert m[i, j] == (j <= 4 + i)


def test_causal_empty_context_is_library_causal_sdpa():
    # no cached rows: a causal layer is textbook causal SDPA over the block
    cfg = tiny_cfg(causal=True)
    rng = np.random.default_rng(41)
    w = tiny_weights(cfg, rng)
    q_len = 6
    noise = rng.standard_normal((1, q_len, cfg.hidden))
    pos = np.arange(q_len)
    out = O.forward(cfg, w, O.DraftCache(cfg.n_kv_heads, cfg.head_dim, 1), noise,
                    [np.zeros((0, cfg.hidden))], [pos])
    f = O.rope_frequencies(cfg.head_dim, cfg.rope_theta)
    d, g = cfg.head_dim, cfg.groups
    def heads(wm, n, gains):
        x = (noise[0] @ wm.T).reshape(q_len, n, d).transpose(1, 0, 2)
        return np.stack([O.rope(O.rms_norm(x[h], gains, cfg.rms_eps), pos, f) for h in range(n)])
    qh = torch.from_numpy(heads(w.wq, cfg.n_heads, w.q_norm))
    kh = torch.from_numpy(heads(w.wk, cfg.n_kv_heads, w.k_norm)).repeat_interleave(g, 0)
    vh = torch.from_numpy((noise[0] @ w.wv.T).reshape(q_len, cfg.n_kv_heads, d)
                          .transpose(1, 0, 2)).repeat_interleave(g, 0)
    o = torch.nn.functional.scaled_dot_product_attention(qh[None], kh[None], vh[None],
                                                         is_causal=True)[0]
    ref = o.numpy().transpose(1, 0, 2).reshape(q_len, -1) @ w.wo.T
    np.testing.assert_allclose(out[0], ref, rtol=1e-9, atol=1e-11)


def test_causal_last_block_row_equals_non_causal():
    # the last block row sees every key either way; the first row does not
    rng = np.random.default_rng(42)
    outs = []
    for causal in (False, True):
        cfg = tiny_cfg(causal=causal)
        w = tiny_weights(cfg, np.random.default_rng(7))
        c = O.DraftCache(cfg.n_kv_heads, cfg.head_dim, 1)
        r = np.random.default_rng(8)
        th = [r.standard_normal((5, cfg.hidden))]
        noise = r.standard_normal((1, 4, cfg.hidden))
        outs.append(O.forward(cfg, w, c, noise, th, [np.arange(9)]))
    np.testing.assert_allclose(outs[0][0, -1], outs[1][0, -1], rtol=1e-12, atol=1e-13)
    assert np.abs(outs[0][0, 0] - outs[1][0, 0]).max() > 1e-6


# --------------------------------------------------------------------------
# decoder layer: SiLU, the Qwen3 MLP, norms and residuals
# --------------------------------------------------------------------------
def test_silu_closed_forms():
    x = np.linspace(-30.0, 30.0, 121)
    y = O.silu(x)
    assert O.silu(np.array([0.0]))[0] == 0.0
    # silu(x) - silu(-x) = x (sigmoid(x) + sigmoid(-x) = 1)
    np.testing.assert_allclose(y - O.silu(-x), x, rtol=0, atol=1e-12)
    # silu(1) = 1 / (1 + 1/e); large |x|: x and 0
    assert abs(O.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(y[-1] - 30.0) < 1e-11 and abs(y[0]) < 1e-11


def tiny_mlp(H, inter, rng, gains=True):
    g = (lambda n: 1.0 + 0.3 * rng.standard_normal(n)) if gains else np.ones
    return O.MlpWeights(gate=0.2 * rng.standard_normal((inter, H)),
                        up=0.2 * rng.standard_normal((inter, H)),
                        down=0.2 * rng.standard_normal((H, inter)),
                        input_norm=g(H), post_norm=g(H))


def _brute_mlp(m, y):
    """down(silu(gate y) * up y) with explicit sums and the sigmoid written out."""
    H, inter = m.gate.shape[1], m.gate.shape[0]
    out = np.zeros((y.shape[0], H))
    for r in range(y.shape[0]):
        act = []
        for j in range(inter):
            gj = sum(m.gate[j, k] * y[r, k] for k in range(H))
            uj = sum(m.up[j, k] * y[r, k] for k in range(H))
            act.append(gj / (1.0 + math.exp(-gj)) * uj)
        for i in range(H):
            out[r, i] = sum(m.down[i, j] * act[j] for j in range(inter))
    return out


def _brute_norm(x, w, eps):
    out = np.empty_like(x)
    for r in range(x.shape[0]):
        ms = sum(float(v) * float(v) for v in x[r]) / x.shape[1]
        out[r] = [w[i] * x[r, i] / math.sqrt(ms + eps) for i in range(x.shape[1])]
    return out


def test_mlp_matches_explicit_sums():
    rng = np.random.default_rng(11)
    m = tiny_mlp(8, 12, rng)
    y = rng.standard_normal((3, 8))
    np.testing.assert_allclose(O.mlp(m, y), _brute_mlp(m, y), rtol=1e-12, atol=1e-12)


def _decoder_case(seed, zero_wo=False, zero_down=False):
    rng = np.random.default_rng(seed)
    cfg = tiny_cfg()
    w = tiny_weights(cfg, rng)
    if zero_wo:
        w.wo = np.zeros_like(w.wo)
    m = tiny_mlp(cfg.hidden, 24, rng)
    if zero_down:
        m.down = np.zeros_like(m.down)
    q = 4
    hidden = rng.standard_normal((1, q, cfg.hidden))
    th = [rng.standard_normal((3, cfg.hidden))]
    pos = [np.arange(0, 3 + q)]
    return cfg, w, m, hidden, th, pos, rng


def test_decoder_layer_without_attention_is_mlp_of_post_norm():
    # wo = 0: the attention adds nothing, so r2 = hidden and the output is the
    # MLP of hidden through the post-attention norm (not the input norm)
    cfg, w, m, hidden, th, pos, _ = _decoder_case(21, zero_wo=True)
    out, r2 = O.decoder_layer(cfg, w, m, O.DraftCache(cfg.n_kv_heads, cfg.head_dim, 1),
                              hidden, None, th, pos)
    np.testing.assert_array_equal(r2, hidden)
    ref = _brute_mlp(m, _brute_norm(hidden[0], m.post_norm, cfg.rms_eps))
    np.testing.assert_allclose(out[0], ref, rtol=1e-10, atol=1e-12)


def test_decoder_layer_attention_term_reads_input_norm_rows():
    # down = 0: the MLP adds nothing; r2 - r1 is the attention of the rows
    # through the input norm (explicit loops), cache appended as by forward
    cfg, w, m, hidden, th, pos, _ = _decoder_case(22, zero_down=True)
    c1 = O.DraftCache(cfg.n_kv_heads, cfg.head_dim, 1)
    out, r2 = O.decoder_layer(cfg, w, m, c1, hidden, None, th, pos)
    assert np.all(out == 0.0)
    c2 = O.DraftCache(cfg.n_kv_heads, cfg.head_dim, 1)
    normed = _brute_norm(hidden[0], m.input_norm, cfg.rms_eps)[None]
    a = O.forward(cfg, w, c2, normed, th, pos)
    np.testing.assert_allclose(r2 - hidden, a, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(c1.k[0], c2.k[0], rtol=1e-10, atol=1e-12)


def test_decoder_layer_output_is_mlp_of_post_norm_of_the_residual():
    # both branches active: the output is the MLP (explicit sums) of the
    # returned residual r2 (pinned above as r1 + attention) through the
    # post-attention norm
    cfg, w, m, hidden, th, pos, _ = _decoder_case(24)
    out, r2 = O.decoder_layer(cfg, w, m, O.DraftCache(cfg.n_kv_heads, cfg.head_dim, 1),
                              hidden, None, th, pos)
    assert np.abs(r2 - hidden).max() > 1e-3  # the attention did contribute
    ref = _brute_mlp(m, _brute_norm(r2[0], m.post_norm, cfg.rms_eps))
    np.testing.assert_allclose(out[0], ref, rtol=1e-10, atol=1e-12)


def test_decoder_layer_residual_stream_form():
    # (hidden = a, residual = b) is the layer applied to a + b
    cfg, w, m, hidden, th, pos, rng = _decoder_case(23)
    res = rng.standard_normal(hidden.shape)
    o1, r1 = O.decoder_layer(cfg, w, m, O.DraftCache(cfg.n_kv_heads, cfg.head_dim, 1),
                             hidden - res, res, th, pos)
    o2, r2 = O.decoder_layer(cfg, w, m, O.DraftCache(cfg.n_kv_heads, cfg.head_dim, 1),
                             hidden, None, th, pos)
    np.testing.assert_allclose(o1, o2, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(r1, r2, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- packed backward
def packed_core_case(seed=7, S=7, nb=3, bs=2, d=4, heads=4, kv=2):
    rng = np.random.default_rng(seed)
    cfg = tiny_cfg(n_heads=heads, n_kv_heads=kv, head_dim=d, hidden=heads * d)
    # anchors 0 (no context) and S (all of it) included
    anchors = np.array([0, S] + list(rng.integers(1, S, nb - 2)))[:nb]
    T = nb * bs
    q = rng.standard_normal((heads, T, d))
    k = rng.standard_normal((kv, S + T, d))
    v = rng.standard_normal((kv, S + T, d))
    d_o = rng.standard_normal((heads, T, d))
    return cfg, anchors, S, bs, q, k, v, d_o


def test_packed_core_backward_matches_finite_differences():
    """Central differences of L = sum(o * dO) in every element of q, k, v."""
    cfg, anchors, S, bs, q, k, v, d_o = packed_core_case()
    dq, dk, dv = O.packed_core_backward(cfg, q, k, v, anchors, S, bs, d_o)

    def loss(q_, k_, v_):
        return float(np.sum(O.packed_core(cfg, q_, k_, v_, anchors, S, bs)[0] * d_o))

    eps = 1e-6
    for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.empty_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = xp, xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-7)


def test_packed_core_matches_torch_autograd():
    """Forward, log-sum-exp and gradients against torch SDPA + autograd in
    float64, with the anchor rule built here from its statement."""
    cfg, anchors, S, bs, q, k, v, d_o = packed_core_case(seed=11, S=40, nb=4, bs=4, d=16,
                                                         heads=4, kv=2)
    T = q.shape[1]
    allowed = torch.zeros(T, S + T, dtype=torch.bool)
    for r in range(T):
        blk = r // bs
        allowed[r, :min(int(anchors[blk]), S)] = True
        allowed[r, S + blk * bs:S + (blk + 1) * bs] = True
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    g = cfg.n_heads // cfg.n_kv_heads
    K, V = tk.repeat_interleave(g, 0), tv.repeat_interleave(g, 0)
    o = torch.nn.functional.scaled_dot_product_attention(
        tq[None], K[None], V[None], attn_mask=allowed, scale=cfg.scaling)[0]
    scores = (tq @ K.transpose(1, 2)) * cfg.scaling
    lse = torch.logsumexp(scores.masked_fill(~allowed, -math.inf), -1)
    o.backward(torch.tensor(d_o))
    o_ref, lse_ref = O.packed_core(cfg, q, k, v, anchors, S, bs)
    dq, dk, dv = O.packed_core_backward(cfg, q, k, v, anchors, S, bs, d_o)
    # both sides are float64, yet in some runs of the whole CPU suite they
    # differed by up to 7e-10 in the log-sum-exp of the heads of one kv head
    # (not reproduced in isolation); any slip in the definition moves these
    # values by 1e-3 or more, so the bounds sit between the two
    np.testing.assert_allclose(o_ref, o.detach().numpy(), rtol=1e-8, atol=1e-10)
    np.testing.assert_allclose(lse_ref, lse.detach().numpy(), rtol=1e-8, atol=1e-10)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-8, atol=1e-10)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-8, atol=1e-10)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-8, atol=1e-10)


def test_packed_core_backward_invariants():
    cfg, anchors, S, bs, q, k, v, d_o = packed_core_case(seed=3, S=9, nb=3, bs=3)
    g = cfg.groups
    dq, dk, dv = O.packed_core_backward(cfg, q, k, v, anchors, S, bs, d_o)
    # softmax rows sum to one: a KV head's dV summed over keys is its query
    # heads' dO summed over rows
    for kv in range(cfg.n_kv_heads):
        np.testing.assert_allclose(dv[kv].sum(0), d_o[kv * g:(kv + 1) * g].sum((0, 1)),
                                   rtol=1e-12, atol=1e-12)
    # equal keys: every row's scores are constant, dS rows sum to zero, dQ = 0
    k_eq = np.broadcast_to(k[:, :1], k.shape).copy()
    dq0, _, _ = O.packed_core_backward(cfg, q, k_eq, v, anchors, S, bs, d_o)
    np.testing.assert_allclose(dq0, 0.0, atol=1e-12)
    # the log-sum-exp of one row by an explicit loop over its keys
    o, lse = O.packed_core(cfg, q, k, v, anchors, S, bs)
    r, h = 4, 1
    blk = r // bs
    keys = list(range(min(int(anchors[blk]), S))) + list(range(S + blk * bs, S + (blk + 1) * bs))
    tot = sum(math.exp(cfg.scaling * float(q[h, r] @ k[h // g, j])) for j in keys)
    assert abs(lse[h, r] - math.log(tot)) < 1e-12


# ---------------------------------------------------------------- golden fixtures
GOLDEN = __import__("os").path.join(__import__("os").path.dirname(__file__), "golden")


def load_golden_matrix(name):
    rows = [ln.split() for ln in open(f"{GOLDEN}/{name}") if ln.strip() and ln[0] != "#"]
    return np.array([[int(x) for x in r] for r in rows], dtype=bool)


def test_band_mask_matches_hand_written_fixture():
    np.testing.assert_array_equal(O.band_mask(3, 7, 2),
                                  load_golden_matrix("band_mask_q3_k7_w2.txt"))


def test_anchor_mask_matches_hand_written_fixture():
    np.testing.assert_array_equal(O.anchor_mask(5, [2, 5], 2),
                                  load_golden_matrix("anchor_mask_s5_anchors_2_5_bs2.txt"))


def test_oracle_forward_matches_stored_fixture():
    """Guards the oracle against unintended changes of its arithmetic."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_oracle_golden",
                                                  f"{GOLDEN}/make_oracle_golden.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    stored = np.loadtxt(f"{GOLDEN}/oracle_forward_tiny.txt", comments="#")
    np.testing.assert_allclose(mod.compute(), stored, rtol=1e-12, atol=1e-15)


def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant slips in the oracle (CPU only) and check a pin fails for each."""
    import copy

    def broke_rope_sign(x, positions, freqs):
        half = x.shape[-1] // 2
        ang = np.asarray(positions, float)[:, None] * freqs[None, :]
        c, s = np.cos(ang), np.sin(ang)
        x1, x2 = x[..., :half], x[..., half:]
        return np.concatenate([x1 * c + x2 * s, x2 * c - x1 * s], -1)

    def broke_rope_interleaved(x, positions, freqs):
        ang = np.asarray(positions, float)[:, None] * freqs[None, :]
        c, s = np.cos(ang), np.sin(ang)
        x1, x2 = x[..., 0::2], x[..., 1::2]
        y = np.empty_like(x)
        y[..., 0::2] = x1 * c - x2 * s
        y[..., 1::2] = x2 * c + x1 * s
        return y

    def broke_norm_no_eps(x, w, eps):
        return w * x / np.sqrt(np.mean(x * x, -1, keepdims=True))

    orig_attention = O.attention

    def broke_causal(cfg, q, k, v, allowed):
        ql, kl = allowed.shape
        causal = (np.arange(kl)[None] <= (kl - ql + np.arange(ql))[:, None])
        return orig_attention(cfg, q, k, v, allowed & causal)

    def broke_gqa(cfg, q, k, v, allowed):
        # query head h reading kv head h % n_kv instead of h // groups
        perm = [h % cfg.n_kv_heads for h in range(cfg.n_heads)]
        inv = [perm.index(i) for i in range(cfg.n_kv_heads)]
        k2 = np.stack([k[perm[h]] for h in range(cfg.n_heads)])
        v2 = np.stack([v[perm[h]] for h in range(cfg.n_heads)])
        c2 = copy.copy(cfg); c2.n_kv_heads = cfg.n_heads
        return orig_attention(c2, q, k2, v2, allowed)

    orig_rms_norm = O.rms_norm

    def broke_mlp_swapped(m, y):
        return O.linear(O.silu(O.linear(y, m.up)) * O.linear(y, m.gate), m.down)

    def broke_silu_sigmoid(x):
        return 1.0 / (1.0 + np.exp(-x))

    def broke_decoder_post_on_r1(cfg, w, m, cache, hidden, residual, th, pos, seqs=None):
        r1 = hidden if residual is None else hidden + residual
        a = O.forward(cfg, w, cache, orig_rms_norm(r1, m.input_norm, cfg.rms_eps), th, pos,
                      seqs=seqs)
        return O.mlp(m, orig_rms_norm(r1, m.post_norm, cfg.rms_eps)), r1 + a

    def broke_decoder_input_gains(cfg, w, m, cache, hidden, residual, th, pos, seqs=None):
        r1 = hidden if residual is None else hidden + residual
        a = O.forward(cfg, w, cache, orig_rms_norm(r1, m.post_norm, cfg.rms_eps), th, pos,
                      seqs=seqs)
        r2 = r1 + a
        return O.mlp(m, orig_rms_norm(r2, m.post_norm, cfg.rms_eps)), r2

    def broke_causal_strict(q_len, k_len):
        qi = (k_len - q_len + np.arange(q_len))[:, None]
        return np.arange(k_len)[None, :] < qi

    def broke_bwd_no_rowsum(q, k, v, allowed, scaling, d_o):
        s = np.where(allowed, scaling * (q @ k.T), -np.inf)
        p = np.exp(s - s.max(-1, keepdims=True))
        p /= p.sum(-1, keepdims=True)
        ds = p * (d_o @ v.T)
        return scaling * (ds @ k), scaling * (ds.T @ q), p.T @ d_o

    def broke_bwd_dk_unscaled(q, k, v, allowed, scaling, d_o):
        dq, dk, dv = orig_core_bwd(q, k, v, allowed, scaling, d_o)
        return dq, dk / scaling, dv

    def broke_bwd_unmasked(q, k, v, allowed, scaling, d_o):
        return orig_core_bwd(q, k, v, np.ones_like(allowed), scaling, d_o)

    orig_core_bwd = O.attention_core_backward

    def broke_band_inclusive(q_len, k_len, window):
        qi = (k_len - q_len + np.arange(q_len))[:, None]
        return np.abs(qi - np.arange(k_len)[None, :]) <= window

    def broke_anchor_inclusive(seq, anchors, block_size):
        m = np.zeros((len(anchors) * block_size, seq + len(anchors) * block_size), bool)
        for b, a in enumerate(anchors):
            rows = slice(b * block_size, (b + 1) * block_size)
            m[rows, :min(int(a) + 1, seq)] = True
            m[rows, seq + b * block_size: seq + (b + 1) * block_size] = True
        return m

    slips = [
        ("attention_core_backward", broke_bwd_no_rowsum,
         [test_packed_core_backward_matches_finite_differences,
          test_packed_core_matches_torch_autograd]),
        ("attention_core_backward", broke_bwd_dk_unscaled,
         [test_packed_core_backward_matches_finite_differences]),
        ("attention_core_backward", broke_bwd_unmasked,
         [test_packed_core_backward_matches_finite_differences,
          test_packed_core_matches_torch_autograd]),
        ("causal_mask", broke_causal_strict, [test_causal_mask_elementwise_rule]),
        ("band_mask", broke_band_inclusive, [test_band_mask_matches_hand_written_fixture]),
        ("anchor_mask", broke_anchor_inclusive,
         [test_anchor_mask_matches_hand_written_fixture]),
        ("mlp", broke_mlp_swapped, [test_mlp_matches_explicit_sums]),
        ("silu", broke_silu_sigmoid, [test_silu_closed_forms, test_mlp_matches_explicit_sums]),
        ("decoder_layer", broke_decoder_post_on_r1,
         [test_decoder_layer_output_is_mlp_of_post_norm_of_the_residual]),
        ("decoder_layer", broke_decoder_input_gains,
         [test_decoder_layer_attention_term_reads_input_norm_rows]),
        ("rope", broke_rope_sign, [test_rope_basis_vectors_rotate_half_pairs]),
        ("rope", broke_rope_interleaved, [test_rope_basis_vectors_rotate_half_pairs]),
        ("rms_norm", broke_norm_no_eps, [test_rms_norm_constant_vector_closed_form]),
        ("attention", broke_causal, [test_forward_is_permutation_equivariant_over_block_rows]),
        ("attention", broke_gqa, [test_attention_matches_library_sdpa_with_repeat_kv]),
    ]
    for name, fn, pins in slips:
        with monkeypatch.context() as m:
            m.setattr(O, name, fn)
            for pin in pins:
                with pytest.raises(AssertionError):
                    pin()
