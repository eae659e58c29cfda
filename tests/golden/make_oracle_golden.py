"""Writes oracle_forward_tiny.txt: the fp64 oracle's output for one tiny
seeded draft-attention step (two steps with a crop between them).  It calls
only the oracle; the fixture guards the oracle against unintended changes of
its arithmetic (a deliberate change regenerates it and names the passage that
justifies it).  Run from the repository root: python tests/golden/make_oracle_golden.py"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
from oracle import dflash_oracle as O  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_forward_tiny.txt")


def compute():
    rng = np.random.default_rng(20261202)
    cfg = O.LayerConfig(hidden=16, n_heads=2, n_kv_heads=1, head_dim=8, rms_eps=1e-6,
                        rope_theta=1e4, n_target_layers=2, sliding_window=5)
    H, d = 16, 8
    w = O.LayerWeights(wq=0.3 * rng.standard_normal((2 * d, H)),
                       wk=0.3 * rng.standard_normal((d, H)),
                       wv=0.3 * rng.standard_normal((d, H)),
                       wo=0.3 * rng.standard_normal((H, 2 * d)),
                       q_norm=1 + 0.1 * rng.standard_normal(d),
                       k_norm=1 + 0.1 * rng.standard_normal(d),
                       fc=0.3 * rng.standard_normal((H, 2 * H)),
                       hidden_norm=1 + 0.1 * rng.standard_normal(H))
    cache = O.DraftCache(1, d, 1)
    outs = []
    L = 0
    for n_ctx in (5, 2):
        x = rng.standard_normal((n_ctx, 2 * H))
        th = O.ctx_project(cfg, w, x)
        nz = rng.standard_normal((1, 3, H))
        pos = np.arange(L, L + n_ctx + 3)
        outs.append(O.forward(cfg, w, cache, nz, [th], [pos]))
        L += n_ctx
        cache.crop([L])
    return np.concatenate([o.reshape(-1) for o in outs])


if __name__ == "__main__":
    v = compute()
    with open(OUT, "w") as f:
        f.write("# fp64 oracle output of tests/golden/make_oracle_golden.py "
                "(written by that script, which calls only the oracle)\n")
        for x in v:
            f.write(f"{x:.17e}\n")
    print("wrote", OUT, v.size)
