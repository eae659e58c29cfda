"""Plain, slow, fp64 CPU statement of the DFlash draft attention layer.

TEST INFRASTRUCTURE ONLY.  This module is the oracle that the CUDA library is
checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import or run it; the product
path (the ``block_diffusion_draft_gb300`` package and its CUDA library) never
does, and shares no code, table or constant with it.

Everything here is float64 numpy.  Inputs are whatever values the caller hands
in (the tests pass the bf16-rounded weights and activations the GPU sees,
widened exactly to float64).  No blocking, fusion or reordering beyond what the
definition states: each step is the plain formula, with ``@`` (a BLAS matmul)
as the only library primitive.

Sources (page title, then the section or symbol on that page):

* [P1] "Qwen3DFlashAttention: How It Differs from Standard Attention in the
  D-Flash Architecture" (instagit) -- "Dual-Source Key/Value Composition",
  "Per-Head RMS Normalization".
* [P2] "How DFlash Integrates with Qwen3 Rotary Embeddings for Speculative
  Decoding" (instagit) -- "Reusing Qwen3RotaryEmbedding in the Draft Model".
* [P3] "DFlash源码导读（二）：Qwen3DFlashAttention注意力实现全解析" (cf-1.com) --
  steps 1-5 of the forward walk-through and "关键设计：非因果的块扩散注意力".
* [P4] "nemo_automodel.components.speculative.dflash.draft_qwen3" (NeMo
  AutoModel API docs) -- module docstring, ``Qwen3DFlashAttention``,
  ``_sliding_window_mask``, ``apply_rotary_pos_emb``, ``Qwen3DFlashDraftModel._apply``.
* [P5] "vllm.model_executor.models.qwen3_dflash" (vLLM API docs) --
  ``DFlashQwen3Attention.__init__/forward``, ``combine_hidden_states``,
  ``precompute_and_store_context_kv``.

Readings taken where the pages are silent or disagree are listed in the
repository's design notes; the ones that shape a formula are repeated in the
docstring of the function that takes them.

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, invariants, library routines and brute force.  The absolute output of a
trained model is not pinned (parity unpinned for that): the pages print no
worked numeric example.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np


# --------------------------------------------------------------------------
# configuration and weights
# --------------------------------------------------------------------------
@dataclass
class LayerConfig:
    """Scalars of one draft attention layer.

    [P3] step 1: ``head_dim`` is the explicit config value, else
    ``hidden_size // num_attention_heads``; ``num_key_value_groups`` is
    ``num_attention_heads // num_key_value_heads``.  [P4] ``scaling`` is
    ``head_dim ** -0.5``.  [P3] step 5 / [P4] ``sliding_window``: only
    sliding-attention layers carry a window (0 here means full attention).
    """

    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int = 0
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    sliding_window: int = 0
    n_target_layers: int = 0
    # [P5] _dflash_layer_causal / _resolve_layer_attention: some checkpoints
    # make a layer causal (the sliding-attention layers, or all of them)
    causal: bool = False

    def __post_init__(self):
        if self.head_dim == 0:
            self.head_dim = self.hidden // self.n_heads
        if self.n_heads % self.n_kv_heads != 0:
            raise ValueError("n_heads must be a multiple of n_kv_heads")

    @property
    def groups(self) -> int:
        return self.n_heads // self.n_kv_heads

    @property
    def scaling(self) -> float:
        return float(self.head_dim) ** -0.5


@dataclass
class LayerWeights:
    """float64 copies of the layer's parameters, in nn.Linear [out, in] layout.

    [P4] ``Qwen3DFlashAttention``: q_proj, k_proj, v_proj, o_proj, q_norm,
    k_norm.  [P5] ``DFlashQwen3Attention``: no biases (``attention_bias=False``).
    [P5] ``DFlashQwen3Model``: ``fc`` (no bias, input = n_target_layers*hidden)
    and ``hidden_norm``.
    """

    wq: np.ndarray  # [n_heads*d, hidden]
    wk: np.ndarray  # [n_kv*d, hidden]
    wv: np.ndarray  # [n_kv*d, hidden]
    wo: np.ndarray  # [hidden, n_heads*d]
    q_norm: np.ndarray  # [d]
    k_norm: np.ndarray  # [d]
    fc: Optional[np.ndarray] = None  # [hidden, n_target_layers*hidden]
    hidden_norm: Optional[np.ndarray] = None  # [hidden]


# --------------------------------------------------------------------------
# elementary operations
# --------------------------------------------------------------------------
def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """nn.Linear without bias: ``y = x @ w.T`` with ``w`` stored [out, in]."""
    return x @ w.T


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: ``w * x / sqrt(mean(x^2) + eps)``.

    [P3] step 1 (Qwen3RMSNorm over head_dim for q_norm / k_norm, eps =
    rms_norm_eps); [P5] ``hidden_norm`` is the same norm over hidden_size.
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return w * (x / np.sqrt(ms + eps))


def rope_frequencies(head_dim: int, theta: float) -> np.ndarray:
    """Rotary frequencies ``f_j = theta^(-2j/d)`` for j < d/2, kept at fp32.

    [P4] ``Qwen3DFlashDraftModel._apply``: the frequencies (``inv_freq``) must
    be fp32 values.  Reading taken: ``f_j`` is the fp32 number nearest the
    exact ``theta^(-2j/d)``; the angle ``p * f_j`` and its sine and cosine are
    then evaluated in float64.
    """
    j = np.arange(head_dim // 2, dtype=np.float64)
    exact = np.power(float(theta), -2.0 * j / head_dim)
    return exact.astype(np.float32).astype(np.float64)


def rope(x: np.ndarray, positions: np.ndarray, freqs: np.ndarray) -> np.ndarray:
    """NeoX-style (rotate-half) rotary embedding of rows of ``x``.

    ``x`` is [..., n, d] and ``positions`` is [n].  [P5]
    ``DFlashQwen3Attention``: ``is_neox_style=True``, so element j is paired
    with element j + d/2 and both use frequency ``f_j``:
    ``x'_j = x_j cos(p f_j) - x_{j+d/2} sin(p f_j)``,
    ``x'_{j+d/2} = x_{j+d/2} cos(p f_j) + x_j sin(p f_j)``.
    """
    half = x.shape[-1] // 2
    ang = np.asarray(positions, dtype=np.float64)[:, None] * freqs[None, :]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def split_heads(y: np.ndarray, n: int, d: int) -> np.ndarray:
    """[rows, n*d] -> [n, rows, d] (head h owns columns h*d .. h*d+d-1)."""
    return y.reshape(y.shape[0], n, d).transpose(1, 0, 2)


# --------------------------------------------------------------------------
# projections of one sequence's rows
# --------------------------------------------------------------------------
def project_q(cfg: LayerConfig, w: LayerWeights, h: np.ndarray,
              positions: np.ndarray) -> np.ndarray:
    """Queries of the noise rows: q_proj -> per-head q_norm -> RoPE.

    [P5] ``DFlashQwen3Attention.forward`` order: projection, per-head RMSNorm,
    then rotary embedding.  [P4] ``apply_rotary_pos_emb``: the queries take
    the trailing q_len positions of the window; the caller passes exactly
    those.  Returns [n_heads, rows, d].
    """
    f = rope_frequencies(cfg.head_dim, cfg.rope_theta)
    q = split_heads(linear(h, w.wq), cfg.n_heads, cfg.head_dim)
    q = rms_norm(q, w.q_norm, cfg.rms_eps)
    return rope(q, positions, f)


def project_kv(cfg: LayerConfig, w: LayerWeights, h: np.ndarray,
               positions: np.ndarray):
    """Keys and values of some rows: k_proj -> k_norm -> RoPE; v_proj raw.

    [P3] step 2: the same k_proj / v_proj serve the context rows
    (``target_hidden``) and the noise rows.  [P3] step 1 and [P5]
    ``precompute_and_store_context_kv``: k_norm applies to every key, context
    keys included; V is neither normed nor rotated.  Returns two
    [n_kv, rows, d] arrays.
    """
    f = rope_frequencies(cfg.head_dim, cfg.rope_theta)
    k = split_heads(linear(h, w.wk), cfg.n_kv_heads, cfg.head_dim)
    k = rope(rms_norm(k, w.k_norm, cfg.rms_eps), positions, f)
    v = split_heads(linear(h, w.wv), cfg.n_kv_heads, cfg.head_dim)
    return k, v


# --------------------------------------------------------------------------
# masks
# --------------------------------------------------------------------------
def full_mask(q_len: int, k_len: int) -> np.ndarray:
    """Non-causal block attention: every query sees every key.

    [P3] "关键设计：非因果的块扩散注意力": ``is_causal = False`` and the mask is
    usually None, so each block token sees all context and the whole block.
    [P4] module docstring: the draft attention is not causal.
    """
    return np.ones((q_len, k_len), dtype=bool)


def band_mask(q_len: int, k_len: int, window: int) -> np.ndarray:
    """Sliding-window band over the key axis, strict on both sides.

    [P4] ``_sliding_window_mask``: query row i sits at key index
    ``k_len - q_len + i``; a key is kept when its distance to that index is
    below ``sliding_window`` (both bounds strict, symmetric band).
    """
    qi = (k_len - q_len + np.arange(q_len))[:, None]
    kj = np.arange(k_len)[None, :]
    return np.abs(qi - kj) < window


def causal_mask(q_len: int, k_len: int) -> np.ndarray:
    """Causal layers ([P5] ``_dflash_layer_causal``): query row i, at key index
    ``k_len - q_len + i``, sees the keys at or before that index -- every
    cached and context row and the block rows up to its own.  Reading taken:
    the pages resolve which layers are causal but do not print the mask; this
    is the plain causal rule over the [cache | context | block] key axis."""
    qi = (k_len - q_len + np.arange(q_len))[:, None]
    kj = np.arange(k_len)[None, :]
    return kj <= qi


def anchor_mask(seq: int, anchors: Sequence[int], block_size: int) -> np.ndarray:
    """Training-layout mask: a block sees context strictly before its anchor
    plus its own block, bidirectionally.

    [P4] module docstring: a draft block's queries attend to the projected
    context strictly before its anchor and to the other noise tokens of the
    same block.  Keys are ``[context rows 0..seq-1 | block 0 | block 1 | ...]``;
    queries are the blocks' rows in block order.
    """
    nb = len(anchors)
    q_len, k_len = nb * block_size, seq + nb * block_size
    m = np.zeros((q_len, k_len), dtype=bool)
    for b, a in enumerate(anchors):
        rows = slice(b * block_size, (b + 1) * block_size)
        m[rows, :min(int(a), seq)] = True
        m[rows, seq + b * block_size: seq + (b + 1) * block_size] = True
    return m


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
def attention(cfg: LayerConfig, q: np.ndarray, k: np.ndarray, v: np.ndarray,
              allowed: np.ndarray) -> np.ndarray:
    """Masked softmax attention with grouped KV heads.

    ``q`` [n_heads, q_len, d], ``k``/``v`` [n_kv, k_len, d], ``allowed``
    [q_len, k_len].  Query head h reads KV head ``h // groups`` ([P3] step 1:
    GQA with ``num_key_value_groups``).  Scores are ``scaling * q.k`` ([P4]
    ``scaling = head_dim ** -0.5``); disallowed keys get probability 0.
    Returns [q_len, n_heads * d] (heads concatenated, as o_proj expects).
    """
    g = cfg.groups
    out = np.empty((q.shape[1], cfg.n_heads * cfg.head_dim))
    for h in range(cfg.n_heads):
        kh, vh = k[h // g], v[h // g]
        s = cfg.scaling * (q[h] @ kh.T)
        s = np.where(allowed, s, -np.inf)
        m = np.max(s, axis=-1, keepdims=True)
        p = np.exp(s - m)
        p = p / np.sum(p, axis=-1, keepdims=True)
        out[:, h * cfg.head_dim:(h + 1) * cfg.head_dim] = p @ vh
    return out


# --------------------------------------------------------------------------
# context projection
# --------------------------------------------------------------------------
def ctx_project(cfg: LayerConfig, w: LayerWeights, x: np.ndarray) -> np.ndarray:
    """``target_hidden = hidden_norm(fc(concat of target layers))``.

    [P3] "看懂注意力数据流": the context stream is the selected target layers'
    hidden states, projected by ``fc`` and RMSNorm.  [P5]
    ``combine_hidden_states``: a width other than ``fc``'s input raises
    ValueError; ``hidden_norm`` is an RMSNorm over hidden_size.
    """
    if w.fc is None or w.hidden_norm is None:
        raise ValueError("layer has no fc / hidden_norm")
    if x.shape[-1] != w.fc.shape[1]:
        raise ValueError(
            f"expected {w.fc.shape[1]} concatenated features, got {x.shape[-1]}")
    return rms_norm(linear(x, w.fc), w.hidden_norm, cfg.rms_eps)


# --------------------------------------------------------------------------
# draft KV cache
# --------------------------------------------------------------------------
@dataclass
class DraftCache:
    """Per-sequence K/V rows kept in float64, in append order.

    [P3] step 4: each step's context + noise K/V are appended with
    ``past_key_values.update``; after verification ``crop(start)`` truncates
    the cache to the accepted prefix.  Keys are stored after k_norm and RoPE,
    values raw, exactly what the attention consumes.
    """

    n_kv_heads: int
    head_dim: int
    batch: int
    k: List[np.ndarray] = field(default_factory=list)
    v: List[np.ndarray] = field(default_factory=list)

    def __post_init__(self):
        if not self.k:
            e = np.zeros((self.n_kv_heads, 0, self.head_dim))
            self.k = [e.copy() for _ in range(self.batch)]
            self.v = [e.copy() for _ in range(self.batch)]

    def lengths(self) -> List[int]:
        return [k.shape[1] for k in self.k]

    def append(self, b: int, k: np.ndarray, v: np.ndarray) -> None:
        self.k[b] = np.concatenate([self.k[b], k], axis=1)
        self.v[b] = np.concatenate([self.v[b], v], axis=1)

    def crop(self, keep: Sequence[int]) -> None:
        """Keep the first ``keep[b]`` rows of sequence b.

        Reading taken: ``keep`` above the current length (or negative) is an
        error rather than a silent no-op; ``keep == len`` changes nothing.
        """
        for b, n in enumerate(keep):
            if n < 0 or n > self.k[b].shape[1]:
                raise ValueError(f"crop({n}) outside [0, {self.k[b].shape[1]}]")
            self.k[b] = self.k[b][:, :n]
            self.v[b] = self.v[b][:, :n]


# --------------------------------------------------------------------------
# the layer
# --------------------------------------------------------------------------
def forward(cfg: LayerConfig, w: LayerWeights, cache: DraftCache,
            noise: np.ndarray, target_hidden: Sequence[np.ndarray],
            positions: Sequence[np.ndarray],
            seqs: Optional[Sequence[int]] = None) -> np.ndarray:
    """One inference step of the layer over a batch, updating ``cache``.

    ``noise`` [B, q_len, hidden] (one anchor plus mask tokens per block);
    ``target_hidden[b]`` [n_b, hidden] (the newly accepted context rows of
    sequence b, already through ``ctx_project``); ``positions[b]`` [n_b + q_len]
    (context rows first, then the block).  Returns [B, q_len, hidden]; rows of
    sequences not in ``seqs`` (when given) are left NaN and their cache is not
    touched.

    Steps ([P3] steps 1-4, [P5] ``DFlashQwen3Attention.forward``):
    1. K_ctx, V_ctx from the new context rows, K_noise, V_noise and Q from the
       noise rows (same k_proj/v_proj for both streams, [P3] step 2);
    2. per-head q_norm / k_norm, then RoPE: context keys at their own
       positions, noise keys and the queries at the last q_len positions
       ([P3] step 3, [P4] ``apply_rotary_pos_emb``);
    3. append ``[ctx ; noise]`` K/V to the cache, attend over every cached row
       (past + new) -- non-causal, or the band of [P4] ``_sliding_window_mask``
       on sliding layers;
    4. o_proj of the heads' outputs.
    """
    B, q_len, _ = noise.shape
    out = np.full(noise.shape, np.nan)
    for b in (range(B) if seqs is None else seqs):
        pos = np.asarray(positions[b])
        n = target_hidden[b].shape[0]
        if pos.shape[0] != n + q_len:
            raise ValueError("positions must cover context rows then the block")
        kc, vc = project_kv(cfg, w, target_hidden[b], pos[:n])
        kn, vn = project_kv(cfg, w, noise[b], pos[n:])
        q = project_q(cfg, w, noise[b], pos[n:])
        cache.append(b, np.concatenate([kc, kn], axis=1),
                     np.concatenate([vc, vn], axis=1))
        k_len = cache.k[b].shape[1]
        if cfg.sliding_window > 0:
            allowed = band_mask(q_len, k_len, cfg.sliding_window)
        else:
            allowed = full_mask(q_len, k_len)
        if cfg.causal:
            allowed = allowed & causal_mask(q_len, k_len)
        o = attention(cfg, q, cache.k[b], cache.v[b], allowed)
        out[b] = linear(o, w.wo)
    return out


def forward_packed(cfg: LayerConfig, w: LayerWeights, noise: np.ndarray,
                   target_hidden: np.ndarray, anchors: np.ndarray,
                   block_size: int, seqs: Optional[Sequence[int]] = None,
                   blocks: Optional[Sequence[int]] = None) -> np.ndarray:
    """Training-layout forward: many blocks per sequence, no cache.

    ``noise`` [B, nb*bs, hidden], ``target_hidden`` [B, S, hidden] (already
    projected context), ``anchors`` [B, nb].  [P4] module docstring and
    ``assert_target_supports_rollback`` ("Training ... is a single forward
    with no cache and no rewind"): keys/values are ``[context | all blocks]``
    and block k's queries see context rows ``j < anchors[k]`` plus their own
    block.  Reading taken for the positions (silent on the pages): context row
    j is at position j, row t of block k at ``anchors[k] + t``.

    Only sequences in ``seqs`` and blocks in ``blocks`` are computed (the rest
    of ``out`` stays NaN); each needs all context K/V of its sequence.
    """
    B, q_total, _ = noise.shape
    S = target_hidden.shape[1]
    nb = anchors.shape[1]
    if q_total != nb * block_size:
        raise ValueError("noise rows must equal n_blocks * block_size")
    out = np.full(noise.shape, np.nan)
    blocks = range(nb) if blocks is None else blocks
    for b in (range(B) if seqs is None else seqs):
        kc, vc = project_kv(cfg, w, target_hidden[b], np.arange(S))
        for blk in blocks:
            a = int(anchors[b, blk])
            rows = slice(blk * block_size, (blk + 1) * block_size)
            pos = a + np.arange(block_size)
            kn, vn = project_kv(cfg, w, noise[b, rows], pos)
            q = project_q(cfg, w, noise[b, rows], pos)
            # keys visible to this block: context rows before the anchor,
            # then the block itself (other blocks are masked out entirely)
            k = np.concatenate([kc[:, :min(a, S)], kn], axis=1)
            v = np.concatenate([vc[:, :min(a, S)], vn], axis=1)
            allowed = full_mask(block_size, k.shape[1])
            o = attention(cfg, q, k, v, allowed)
            out[b, rows] = linear(o, w.wo)
    return out


# --------------------------------------------------------------------------
# packed training layout: attention core forward and backward
# --------------------------------------------------------------------------
def attention_core(q: np.ndarray, k: np.ndarray, v: np.ndarray, allowed: np.ndarray,
                   scaling: float):
    """One head of masked softmax attention, also returning the log-sum-exp.

    ``q`` [q_len, d], ``k``/``v`` [k_len, d], ``allowed`` [q_len, k_len]
    (every row must allow at least one key).  Scores ``scaling * q.k``
    ([P4] ``scaling = head_dim ** -0.5``); ``lse`` [q_len] is the natural log
    of the row's normaliser, ``log(sum over allowed keys of exp(score))``.
    """
    s = scaling * (q @ k.T)
    s = np.where(allowed, s, -np.inf)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = np.sum(e, axis=-1, keepdims=True)
    o = (e / l) @ v
    return o, (m + np.log(l))[:, 0]


def attention_core_backward(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                            allowed: np.ndarray, scaling: float, d_o: np.ndarray):
    """Gradients of one head's ``o = softmax(scaling * q k^T, masked) v`` with
    respect to q, k and v, given the gradient ``d_o`` of o.

    The chain rule written out step by step (the pages train the draft through
    autograd of this forward, [P4] module docstring): with P the softmax
    probabilities (0 where masked), ``dV = P^T dO``, ``dP = dO V^T``, each
    softmax row's Jacobian gives ``dS = P * (dP - rowsum(P * dP))``, and
    through ``S = scaling * q k^T``: ``dQ = scaling dS K``,
    ``dK = scaling dS^T Q``.
    """
    s = scaling * (q @ k.T)
    s = np.where(allowed, s, -np.inf)
    e = np.exp(s - np.max(s, axis=-1, keepdims=True))
    p = e / np.sum(e, axis=-1, keepdims=True)
    dv = p.T @ d_o
    dp = d_o @ v.T
    ds = p * (dp - np.sum(p * dp, axis=-1, keepdims=True))
    dq = scaling * (ds @ k)
    dk = scaling * (ds.T @ q)
    return dq, dk, dv


def packed_core(cfg: LayerConfig, q: np.ndarray, k: np.ndarray, v: np.ndarray,
                anchors: Sequence[int], seq: int, block_size: int):
    """Attention core of one sequence in the packed training layout.

    ``q`` [n_heads, nb*bs, d] (the blocks' rows in block order), ``k``/``v``
    [n_kv, seq + nb*bs, d] (context rows, then every block's rows); block k's
    queries see context rows before ``anchors[k]`` and their own block
    (``anchor_mask``, [P4] module docstring).  Query head h reads KV head
    ``h // groups``.  Returns ``o`` [n_heads, nb*bs, d] and ``lse``
    [n_heads, nb*bs].
    """
    allowed = anchor_mask(seq, anchors, block_size)
    o = np.empty(q.shape)
    lse = np.empty(q.shape[:2])
    for h in range(cfg.n_heads):
        o[h], lse[h] = attention_core(q[h], k[h // cfg.groups], v[h // cfg.groups],
                                      allowed, cfg.scaling)
    return o, lse


def packed_core_backward(cfg: LayerConfig, q: np.ndarray, k: np.ndarray, v: np.ndarray,
                         anchors: Sequence[int], seq: int, block_size: int,
                         d_o: np.ndarray):
    """Gradients of ``packed_core``'s output with respect to q, k and v.

    ``d_o`` [n_heads, nb*bs, d].  A KV head's gradients sum over the query
    heads that read it (GQA).  Returns ``dq`` like q, ``dk``/``dv`` like k/v.
    """
    allowed = anchor_mask(seq, anchors, block_size)
    dq = np.empty(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for h in range(cfg.n_heads):
        kv = h // cfg.groups
        dq[h], dkh, dvh = attention_core_backward(q[h], k[kv], v[kv], allowed, cfg.scaling,
                                                  d_o[h])
        dk[kv] += dkh
        dv[kv] += dvh
    return dq, dk, dv


# --------------------------------------------------------------------------
# decoder layer: norms, residuals and the MLP around the attention
# --------------------------------------------------------------------------
@dataclass
class MlpWeights:
    """The rest of a draft decoder layer.

    [P4] ``Qwen3DFlashDecoderLayer``: ``input_layernorm``, ``self_attn``,
    ``post_attention_layernorm`` and ``mlp = Qwen3MLP(config)``; [P5] stacks
    ``gate_proj`` and ``up_proj`` into one ``gate_up_proj``.  nn.Linear
    layout [out, in]: gate, up [intermediate, hidden]; down [hidden,
    intermediate]; norm gains [hidden].
    """

    gate: np.ndarray
    up: np.ndarray
    down: np.ndarray
    input_norm: np.ndarray
    post_norm: np.ndarray


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU, ``x * sigmoid(x)`` (the Qwen3 MLP activation; reading taken:
    the pages name Qwen3MLP without printing it)."""
    return x / (1.0 + np.exp(-x))


def mlp(m: MlpWeights, y: np.ndarray) -> np.ndarray:
    """Qwen3 MLP: ``down(silu(gate(y)) * up(y))``."""
    return linear(silu(linear(y, m.gate)) * linear(y, m.up), m.down)


def decoder_layer(cfg: LayerConfig, w: LayerWeights, m: MlpWeights, cache: DraftCache,
                  hidden: np.ndarray, residual: Optional[np.ndarray],
                  target_hidden: Sequence[np.ndarray], positions: Sequence[np.ndarray],
                  seqs: Optional[Sequence[int]] = None):
    """One draft decoder layer over a batch of blocks, updating ``cache``.

    Pre-norm residual block in the residual-stream form of [P5]'s draft model
    (each layer returns ``(hidden_states, residual)``; the next layer adds
    them):  ``r1 = hidden + residual`` (or ``hidden`` for the first layer),
    ``r2 = r1 + attn(input_norm(r1))``, output ``(mlp(post_norm(r2)), r2)``.
    ``hidden`` / ``residual`` [B, q_len, hidden]; the attention takes the
    normed rows as its noise rows (context K/V from ``target_hidden``).
    Reading taken: the standard Qwen3 decoder order (the pages list the parts
    of [P4] ``Qwen3DFlashDecoderLayer`` but not its forward body).
    """
    r1 = hidden if residual is None else hidden + residual
    a = forward(cfg, w, cache, rms_norm(r1, m.input_norm, cfg.rms_eps), target_hidden,
                positions, seqs=seqs)
    r2 = r1 + a
    out = mlp(m, rms_norm(r2, m.post_norm, cfg.rms_eps))
    return out, r2
