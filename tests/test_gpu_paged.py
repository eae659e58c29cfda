"""Paged draft KV cache ("vllm...qwen3_dflash", precompute_and_store_context_kv:
K/V rows inserted through a slot mapping into the layer's paged cache; the
draft attention reads the pages through the batch's block table), checked
against the oracle's contiguous cache: the outputs must match the oracle
forward, and the pages, gathered in block-table order, must hold the oracle
cache's rows.  Pages are handed out in a shuffled order so that no sequence's
pages are contiguous or ascending."""
import numpy as np
import pytest
import torch

from block_diffusion_draft_gb300 import workloads as W
from block_diffusion_draft_gb300.dflash_attn import DFlashError, PagedCache, kernel_launches
from oracle import dflash_oracle as O
import helpers as T

pytestmark = pytest.mark.gpu


def small_bf16(**kw):
    base = dict(hidden=1024, n_heads=8, n_kv_heads=2, head_dim=128, batch=3,
                n_target_layers=2, max_position=8192)
    base.update(kw)
    return W.spec("qwen3_8b_single", **base)


class PageTable:
    """The caller's bookkeeping: a shuffled free list, per-sequence page lists
    and lengths, the block table and the slot mapping of a step."""

    def __init__(self, batch, n_pages, page_size, bt_stride, seed):
        rng = np.random.default_rng(seed)
        self.free = list(rng.permutation(n_pages))
        self.P, self.stride = page_size, bt_stride
        self.pages = [[] for _ in range(batch)]
        self.len = [0] * batch

    def slots_for(self, b, n):
        """Slots of rows len[b] .. len[b] + n - 1, allocating pages as needed."""
        out = []
        for k in range(self.len[b], self.len[b] + n):
            while k // self.P >= len(self.pages[b]):
                self.pages[b].append(int(self.free.pop()))
            out.append(self.pages[b][k // self.P] * self.P + k % self.P)
        return out

    def block_table(self):
        bt = np.full((len(self.pages), self.stride), -1, np.int32)
        for b, ps in enumerate(self.pages):
            bt[b, :len(ps)] = ps
        return torch.from_numpy(bt)

    def gather(self, storage, b, n):
        """Rows 0..n-1 of sequence b from [n_pages, n_kv, P, d] storage."""
        rows = [storage[self.pages[b][k // self.P], :, k % self.P] for k in range(n)]
        return np.stack(rows, axis=1) if rows else storage[:0, :, 0][:, :0]


def run_steps(sp, page_size, n_pages, steps, seed):
    B, q = sp.batch, sp.block_size
    w = W.weights(sp, seed)
    cfg, lw = T.oracle_layer(sp, w)
    attn = T.gpu_layer(sp, w)
    cache = PagedCache(attn, n_pages, page_size)
    ocache = O.DraftCache(sp.n_kv_heads, sp.head_dim, B)
    pt = PageTable(B, n_pages, page_size, bt_stride=n_pages, seed=seed)
    for s, n_ctx in enumerate(steps):
        L0 = list(pt.len)
        th = [W.hidden_rows(sp, seed, "hidden", s, b, n_ctx[b]) for b in range(B)]
        nz = torch.stack([W.hidden_rows(sp, seed, "noise", s, b, q) for b in range(B)])
        pos = [W.window_positions(L0[b], n_ctx[b], q) for b in range(B)]
        slots = sum((pt.slots_for(b, n_ctx[b] + q) for b in range(B)), [])
        target = torch.cat(th).cuda() if sum(n_ctx) > 0 else None
        out = attn.forward_paged(cache, nz.cuda(), target, n_ctx, L0, torch.cat(pos).cuda(),
                                 torch.tensor(slots, dtype=torch.int32).cuda(),
                                 pt.block_table().cuda())
        torch.cuda.synchronize()
        ref = O.forward(cfg, lw, ocache, T.f64(nz), [T.f64(x) for x in th],
                        [p.numpy() for p in pos])
        T.assert_close(out.to("cpu", torch.float64).numpy(), ref, "bf16",
                       f"paged P={page_size} step {s}")
        k, v = (x.to("cpu", torch.float64).numpy() for x in cache.read())
        for b in range(B):
            n = ocache.k[b].shape[1]
            assert n == L0[b] + n_ctx[b] + q
            T.assert_close(pt.gather(k, b, n), ocache.k[b], "bf16", f"paged K seq {b}")
            T.assert_close(pt.gather(v, b, n), ocache.v[b], "bf16", f"paged V seq {b}")
        assert attn.device_error() == 0
        # keep the context rows, drop the block rows (the caller's lengths)
        keep = [L0[b] + n_ctx[b] for b in range(B)]
        pt.len = keep
        ocache.crop(keep)


# (page size, pages): sequences of up to ~480 rows span several 128-key tiles
# and end mid-page; the second step appends after a crop in mid-page
@pytest.mark.parametrize("page_size,n_pages", [(16, 128), (64, 40), (128, 20)])
def test_paged_forward_matches_oracle(page_size, n_pages):
    sp = small_bf16()
    run_steps(sp, page_size, n_pages, ([300, 7, 130], [5, 140, 0], [160, 0, 33]), seed=41)


@pytest.mark.parametrize("window,causal", [(100, False), (200, True)])
def test_paged_band_and_causal_layers(window, causal):
    # band layers start the key range on a 128-key tile boundary; the band
    # still cuts each row's keys
    sp = small_bf16(sliding_window=window, causal=causal)
    run_steps(sp, 32, 64, ([300, 7, 130], [61, 140, 0]), seed=43)


def test_paged_many_sequences():
    # 20 sequences of mixed lengths: the split-KV kernel with a merge pass
    sp = small_bf16(batch=20)
    lens = [int(x) for x in np.random.default_rng(5).integers(0, 260, 20)]
    run_steps(sp, 16, 700, (lens, [3] * 20), seed=47)


def test_paged_bad_slot_is_reported():
    sp = small_bf16(batch=2)
    B, q, seed = 2, sp.block_size, 51
    w = W.weights(sp, seed)
    attn = T.gpu_layer(sp, w)
    cache = PagedCache(attn, 8, 16)
    bt = torch.tensor([[0, 1, 2, -1], [3, 4, 5, -1]], dtype=torch.int32).cuda()
    nz = torch.stack([W.hidden_rows(sp, seed, "noise", 0, b, q) for b in range(B)]).cuda()
    pos = torch.cat([W.window_positions(0, 0, q) for _ in range(B)]).cuda()
    slots = list(range(0, 16)) + list(range(48, 64))
    slots[5] = 8 * 16  # one past the last slot: that row is skipped
    sl = torch.tensor(slots, dtype=torch.int32).cuda()
    n0 = kernel_launches()
    attn.forward_paged(cache, nz, None, [0, 0], [0, 0], pos, sl, bt)
    # no context rows: the QKV projection, the attention (no split at 16
    # keys) and o_proj
    assert kernel_launches() - n0 == 3
    torch.cuda.synchronize()
    assert attn.device_error() == 4  # DFLASH_DEV_SLOT
    # a block-table entry outside the cache for a page holding keys: read as
    # page 0 and reported
    slots_ok = list(range(0, 16)) + list(range(48, 64))
    bt_bad = torch.tensor([[99, 1, 2, -1], [3, 4, 5, -1]], dtype=torch.int32).cuda()
    attn.forward_paged(cache, nz, None, [0, 0], [0, 0], pos,
                       torch.tensor(slots_ok, dtype=torch.int32).cuda(), bt_bad)
    torch.cuda.synchronize()
    assert attn.device_error() == 4
    # entries past the sequences' pages may hold anything
    attn.forward_paged(cache, nz, None, [0, 0], [0, 0], pos,
                       torch.tensor(slots_ok, dtype=torch.int32).cuda(), bt)
    torch.cuda.synchronize()
    assert attn.device_error() == 0
    # host-side checks: a sequence longer than its block-table row
    with pytest.raises(DFlashError):
        attn.forward_paged(cache, nz, None, [0, 0], [60, 0], pos,
                           torch.tensor(slots, dtype=torch.int32).cuda(), bt)
    with pytest.raises(DFlashError):
        PagedCache(attn, 8, 24)
