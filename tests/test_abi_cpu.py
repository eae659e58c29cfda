"""The C ABI library builds, loads and exports what the header declares.

No compute call here: every call below fails its host-side argument check
before touching CUDA, so this runs on machines without a GPU.
"""
import ctypes

import pytest

from block_diffusion_draft_gb300 import build
from block_diffusion_draft_gb300 import dflash_attn as D


@pytest.fixture(scope="module")
def L():
    build.build()
    return D.lib()


def test_every_declared_function_is_exported(L):
    names = D.declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(D._SIGNATURES), "binding and header disagree"


def test_abi_version(L):
    assert L.dflash_abi_version() == 105


def test_create_rejects_null_config(L):
    out = ctypes.c_void_p(123)
    rc = L.dflash_attn_create(None, None, None, None, None, None, None, None, None,
                              ctypes.byref(out))
    assert rc == -1 and out.value is None
    assert b"config" in L.dflash_last_error()


def test_create_rejects_bad_shapes_before_touching_the_device(L):
    fake = ctypes.c_void_p(0x1000)
    out = ctypes.c_void_p()

    def create(**kw):
        base = dict(hidden=256, n_heads=4, n_kv_heads=2, head_dim=0, n_target_layers=0,
                    rms_eps=1e-6, rope_theta=1e6, sliding_window=0, max_position=0,
                    dtype=0, causal=0)
        base.update(kw)
        cfg = D.Config(*[base[f] for f, _ in D.Config._fields_])
        return L.dflash_attn_create(ctypes.byref(cfg), fake, fake, fake, fake, fake,
                                    fake, None, None, ctypes.byref(out))

    assert create(n_heads=3, n_kv_heads=2) == -2          # groups not integral
    assert create(dtype=7) == -1                          # bad dtype
    assert create(hidden=0) == -2                         # non-positive
    assert create(head_dim=64) == -2                      # bf16 needs head_dim 128
    assert create(n_target_layers=2) == -2                # fc missing
    assert create(dtype=1, head_dim=512, hidden=2048) == -2  # fp32 head_dim limit
    assert create(causal=2) == -2                         # causal is 0 or 1


def test_calls_reject_null_handles(L):
    assert L.dflash_cache_crop(None, None) == -1
    assert L.dflash_cache_lengths(None, None) == -1
    assert L.dflash_ctx_project(None, None, 0, None, None) == -1
    assert L.dflash_attn_forward(None, None, 1, 16, None, None, None, None, None, None) == -1
    assert L.dflash_attn_forward_packed(None, 1, 1, 1, 1, None, None, None, None, None) == -1
    assert L.dflash_attn_reserve(None, 1, 1, 1) == -1
    assert L.dflash_attn_destroy(None) == 0
    assert L.dflash_cache_destroy(None) == 0


def test_later_entry_points_reject_null_arguments(L):
    # layer groups, decoder layer, paged cache, packed core: every call checks
    # its arguments on the host before any CUDA work
    out = ctypes.c_void_p()
    assert L.dflash_kv_group_create(None, 2, ctypes.byref(out)) == -1
    assert L.dflash_kv_group_append(None, None, 1, None, None, None, None) == -1
    assert L.dflash_kv_group_destroy(None) == 0
    assert L.dflash_mlp_create(4096, 12288, 1e-6, None, None, None, None, None,
                               ctypes.byref(out)) == -1
    assert L.dflash_mlp_destroy(None) == 0
    assert L.dflash_decoder_layer_forward(None, None, None, 1, 16, None, None, None, None,
                                          None, None, None, None) == -1
    assert L.dflash_paged_cache_create(None, 8, 16, ctypes.byref(out)) == -1
    assert L.dflash_paged_cache_destroy(None) == 0
    assert L.dflash_paged_cache_data(None, None, None, None, None, None, None) == -1
    assert L.dflash_paged_cache_read(None, None, None, None) == -1
    assert L.dflash_attn_forward_paged(None, None, 1, 16, None, None, None, None, None, None,
                                       None, 4, None, None) == -1
    assert L.dflash_packed_attn_core(None, 1, 64, 2, 16, None, None, None, None, None, None,
                                     None) == -1
    assert L.dflash_packed_attn_core_backward(None, 1, 64, 2, 16, None, None, None, None, None,
                                              None, None, None, None, None, None) == -1
    assert L.dflash_kernel_launches(None) == -1
    n = ctypes.c_uint64(0)
    assert L.dflash_kernel_launches(ctypes.byref(n)) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(D, "_LIB", None)
    monkeypatch.setattr(D, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        D.lib()


def test_wait_probe_checks_arguments_on_the_host(L):
    stream = ctypes.c_void_p(0)
    assert L.dflash_wait_probe(None, 1_000_000, 0, stream) == -1
    assert b"null" in L.dflash_last_error()


def test_read_stream_probe_checks_arguments_on_the_host(L):
    stream = ctypes.c_void_p(0)
    assert L.dflash_read_stream_probe(None, None, 128, 64, 1, 1, stream) == -1
    assert b"null" in L.dflash_last_error()


def test_header_is_plain_c(tmp_path):
    """The boundary header compiles as strict C99 (no C++ in the ABI)."""
    import os
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    src = tmp_path / "t.c"
    src.write_text('#include "dflash_attn.h"\nint main(void) { return dflash_abi_version() == 0; }\n')
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-fsyntax-only", "-I", inc, str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
