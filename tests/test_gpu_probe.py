"""The TMA read-stream probe (a measurement aid): it runs to completion for
every accepted launch shape, including two CTAs per SM and a ragged share of
boxes per CTA, records no device error, and rejects bad shapes on the host."""
import pytest
import torch

from block_diffusion_draft_gb300 import workloads as W

import helpers as T

pytestmark = pytest.mark.gpu


def _layer():
    sp = W.spec("qwen3_8b_single", hidden=1024, n_heads=8, n_kv_heads=2, batch=1,
                n_target_layers=2, max_position=4096)
    return T.Scenario(sp, seed=23, capacity=256)


def test_read_stream_probe_runs_every_accepted_shape():
    sc = _layer()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    m = torch.randn(384, 4160, device="cuda").to(torch.bfloat16)  # 3 x 65 boxes
    for ctas, stages in ((1, 1), (7, 3), (sms, 4), (sms, 12), (2 * sms, 6), (195, 2)):
        sc.attn.read_stream_probe(m, ctas, stages)
    torch.cuda.synchronize()
    assert sc.attn.device_error() == 0


def test_read_stream_probe_rejects_bad_shapes():
    sc = _layer()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    m = torch.zeros(256, 128, device="cuda", dtype=torch.bfloat16)
    for ctas, stages, rows in ((1, 0, 256), (1, 13, 256), (0, 2, 256), (2 * sms + 1, 2, 256),
                               (sms + 1, 7, 256), (1, 2, 200)):
        with pytest.raises(Exception, match="ARG"):
            sc.attn.read_stream_probe(m[:rows], ctas, stages)
    assert sc.attn.device_error() == 0
