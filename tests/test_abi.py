"""The C-ABI library builds, loads and exports every entry point its header declares.

No GPU work: only symbol lookup and host-side argument validation that returns before any CUDA
call (invalid configurations, NULL arguments)."""
import ctypes
import re

import pytest


@pytest.fixture(scope="module")
def L():
    from speculative_pipeline_decoding_gb300 import build_ext, binding
    build_ext.build()
    return binding.lib()


def test_every_declared_symbol_is_exported(L):
    from speculative_pipeline_decoding_gb300 import binding
    names = binding.exported_symbols()
    assert len(names) >= 18
    for n in names:
        assert hasattr(L, n), n


def test_header_declares_the_boundary():
    from speculative_pipeline_decoding_gb300 import binding
    names = set(binding.exported_symbols())
    for n in ("spd_create", "spd_prefill", "spd_cycle", "spd_generate", "spd_rollback",
              "spd_generate_ar", "spd_destroy", "spd_last_error", "spd_set_draft_override",
              "spd_debug_dump"):
        assert n in names


def _cfg(**kw):
    from speculative_pipeline_decoding_gb300.binding import Config
    base = dict(n_layers=8, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64, d_ffn=512, vocab=100,
                n_stages=2, pdm_layers=1, anchors=(0, 2, 4, 6, 8), dtype="f32", max_seq=64)
    base.update(kw)
    return Config(**base)


@pytest.mark.parametrize("bad,msg", [
    (dict(n_stages=3), "must divide"),
    (dict(pdm_layers=5), "Ls <= L/n"),
    (dict(anchors=(1, 2)), "anchors[0]"),
    (dict(anchors=(0, 4, 4)), "increase"),
    (dict(anchors=(0, 9)), "<= n_layers"),
    (dict(n_kv_heads=3), "n_kv_heads"),
    (dict(head_dim=24), "head_dim"),
])
def test_create_rejects_invalid_configs_before_touching_the_gpu(L, bad, msg):
    from speculative_pipeline_decoding_gb300.binding import spd_weights
    c = _cfg(**bad).to_c()
    w = spd_weights()
    h = ctypes.c_void_p()
    rc = L.spd_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h))
    assert rc == -1
    assert h.value is None
    assert msg in L.spd_last_error(None).decode()


def test_create_rejects_null_weights(L):
    from speculative_pipeline_decoding_gb300.binding import spd_weights
    c = _cfg().to_c()
    w = spd_weights()
    h = ctypes.c_void_p()
    assert L.spd_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h)) == -1
    assert "NULL" in L.spd_last_error(None).decode()
    assert L.spd_create(None, None, None, ctypes.byref(h)) == -1


def test_null_handle_calls_are_refused(L):
    assert L.spd_rollback(None, 1, 0) == -1
    assert L.spd_cycle(None, None) == -1
    assert L.spd_dump_size(None, 0) == 0
    L.spd_destroy(None)


def test_attention_workspace_size_is_host_arithmetic(L):
    n = L.spd_attention_workspace_bytes(4, 32, 8, 128, 1000)
    chunks = -(-1000 // 128)
    assert n >= 4 * 32 * chunks * 130 * 4
    assert L.spd_attention_workspace_bytes(0, 32, 8, 128, 1000) == 0


def test_no_oracle_import_in_the_product_package():
    import os
    import speculative_pipeline_decoding_gb300 as pkg
    root = os.path.dirname(pkg.__file__)
    for dirpath, _, files in os.walk(root):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(import|from)\s+oracle", text, re.M), f
                assert "spd_inputs" not in text, f


@pytest.mark.parametrize("seed,alpha", [(2, 0.8), (2, 0.5), (2, 0.9), (7, 0.6), (2**64 - 1, 0.85),
                                        (0, 0.0), (123456789, 1.0)])
def test_library_acceptance_modes_equal_the_harness_coins(L, seed, alpha):
    """spd_acceptance_modes (C, host only) draws the same SplitMix64 coins as the seeded input module."""
    import spd_inputs as si
    from speculative_pipeline_decoding_gb300 import binding
    first, last = 514, 514 + 700
    got = binding.acceptance_modes(alpha, seed, first, last - first + 1).tolist()
    assert got == si.override_modes(seed, alpha, first, last)


def test_library_acceptance_compares_in_double_precision(L):
    """A coin exactly at alpha is a reject; one ulp above it is an accept (no float rounding of alpha)."""
    import math
    import spd_inputs as si
    from speculative_pipeline_decoding_gb300 import binding
    for q in (3, 1000, 40000):
        c = si.coin(2, q)
        assert binding.acceptance_modes(c, 2, q, 1).tolist() == [2]
        assert binding.acceptance_modes(math.nextafter(c, 2.0), 2, q, 1).tolist() == [1]


def test_acceptance_argument_checks_on_the_host(L):
    from speculative_pipeline_decoding_gb300 import binding
    with pytest.raises(binding.SpdError):
        binding.acceptance_modes(0.5, 1, -1, 4)
    assert L.spd_acceptance_modes(0.5, 1, 0, 3, None) == -1
    assert L.spd_set_acceptance(None, 0.5, 1, None, 0) == -1
