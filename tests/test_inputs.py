"""Seeded input generators: pinned to SplitMix64's published outputs and to their stated statistics."""
import math

import numpy as np
import pytest
import torch

import spd_inputs as si
from conftest import golden_rows


def test_splitmix64_matches_published_outputs():
    want = [int(r[0]) for r in golden_rows("splitmix64_seed1234567.txt")]
    assert [si.stream_py(1234567, i) for i in range(5)] == want
    got = si.stream_t(1234567, 0, 5, "cpu")
    assert [int(x) & si.MASK64 for x in got] == want


def test_torch_stream_equals_python_stream_everywhere():
    key = si.tensor_key(7, "some.tensor")
    t = si.stream_t(key, 1000, 4096, "cpu")
    assert all((int(t[i]) & si.MASK64) == si.stream_py(key, 1000 + i) for i in range(0, 4096, 7))


def test_normal_like_statistics_and_range():
    key = si.tensor_key(0, "stats")
    v = si.normal_like(key, 1 << 20, 0.02, torch.float32, "cpu").double()
    assert abs(v.mean().item()) < 1e-4
    assert abs(v.std().item() - 0.02) < 2e-4
    # Irwin-Hall(4) is bounded at sqrt(12) standard deviations
    assert v.abs().max().item() <= 0.02 * math.sqrt(12.0) * 1.0001
    # symmetric, near-normal shape: kurtosis of IH(4) is 3 - 6/(5*4) = 2.7
    z = (v - v.mean()) / v.std()
    assert abs((z ** 4).mean().item() - 2.7) < 0.03


def test_normal_like_is_chunk_invariant_and_bf16_is_rounded_f32():
    key = si.tensor_key(3, "chunks")
    a = si.normal_like(key, 10000, 0.02, torch.float32, "cpu", chunk=1 << 20)
    b = si.normal_like(key, 10000, 0.02, torch.float32, "cpu", chunk=333)
    assert torch.equal(a, b)
    c = si.normal_like(key, 10000, 0.02, torch.bfloat16, "cpu")
    assert torch.equal(c, a.to(torch.bfloat16))


def test_weight_specs_shapes():
    w = si.WORKLOADS["gqa4b_bf16_n8"]
    specs = {n: s for n, s, _ in si.weight_specs(w)}
    assert specs["layers.0.wq"] == (4096, 2560)
    assert specs["layers.31.wk"] == (1024, 2560)
    assert specs["layers.5.w_down"] == (2560, 9728)
    assert specs["pdm.fc.4"] == (2560, 5 * 2560)
    assert specs["pdm.layers.3.wo"] == (2560, 4096)
    assert "pdm.layers.4.wo" not in specs
    n_target = sum(math.prod(s) for n, s in specs.items()
                   if n.startswith("layers.") and not n.endswith("norm"))
    assert n_target * 2 == 32 * 201_850_880  # 201.9 MB of bf16 per layer


def test_prompt_tokens_in_range_and_seeded():
    w = si.WORKLOADS["dense1.5b_bf16_n8"]
    p = si.prompt_tokens(w)
    assert p.dtype == torch.int32 and p.numel() == 512
    assert int(p.min()) >= 0 and int(p.max()) < 32000
    assert torch.equal(p, si.prompt_tokens(w))
    assert len(set(p.tolist())) > 480


def test_accept_mask_rate_and_position_keying():
    m = si.accept_mask(2, 0.8, 0, 19999)
    assert abs(sum(m) / len(m) - 0.8) < 0.01
    # keyed by position only: a sub-range gives the same bits
    assert si.accept_mask(2, 0.8, 500, 599) == m[500:600]
    assert all(si.accept_mask(2, 1.0, 0, 999)) and not any(si.accept_mask(2, 0.0, 0, 999))


def test_sampling_uniforms_range_streams_and_position_keying():
    u = si.sampling_uniforms(11, 100, 4099)
    assert set(u) == set(si.SAMPLING_STREAMS)
    for name, vals in u.items():
        a = np.asarray(vals, dtype=np.float64)
        assert len(a) == 4000 and a.min() >= 0.0 and a.max() < 1.0
        assert np.float32(a.max()) < 1.0                      # representable below 1 in fp32
        assert abs(a.mean() - 0.5) < 0.02 and abs(a.var() - 1 / 12) < 0.01
        assert abs(np.corrcoef(a[:-1], a[1:])[0, 1]) < 0.05   # neighbouring positions independent
    # the four streams differ, and a position's uniform does not depend on the range asked for
    assert len({tuple(v[:8]) for v in u.values()}) == 4
    v = si.sampling_uniforms(11, 2000, 2007)
    for name in si.SAMPLING_STREAMS:
        assert v[name] == u[name][1900:1908]
    assert si.sampling_uniforms(12, 100, 107)["draft"] != u["draft"][:8]
