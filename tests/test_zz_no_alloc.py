"""The allocation-free attention entry point (spd_attention_static_scratch).

Some callers may not call cudaMalloc -- a plugin inside an application that owns the GPU's memory
budget, or a latency-critical path where an allocation could synchronise the device.  This entry
point keeps its split partials in a fixed scratch array inside the library.  Here it is checked,
through the C ABI, against the workspace-based spd_attention on the same inputs, on two calls in a
row (the array keeps the previous call's contents, so the second call shows nothing leaks over).
This file is collected last so that a failure here leaves every other test already run.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spd():
    from speculative_pipeline_decoding_gb300 import build_ext
    build_ext.build()
    import speculative_pipeline_decoding_gb300 as spd
    return spd


def _inputs(seed, R, hq, hkv, hd, max_seq, dtype):
    g = torch.Generator(device="cpu").manual_seed(seed)
    k = (torch.randn(hkv, max_seq, hd, generator=g) * 0.5).to(dtype).cuda()
    v = torch.randn(hkv, max_seq, hd, generator=g).to(dtype).cuda()
    q = (torch.randn(R, hq, hd, generator=g) * 0.5).cuda()
    pos = torch.randint(1, max_seq + 1, (R,), generator=g, dtype=torch.int32)
    pos[0] = max_seq
    return q, k, v, pos.cuda()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_static_scratch_matches_workspace_entry_point_twice(spd, dtype):
    hq, hkv, hd = 32, 8, 128
    for call, (R, max_seq, seed) in enumerate([(8, 1500, 0), (5, 700, 1)]):
        q, k, v, pos = _inputs(seed, R, hq, hkv, hd, max_seq, dtype)
        ws = torch.zeros(spd.attention_workspace_bytes(R, hq, hkv, hd, max_seq) // 4 + 1,
                         dtype=torch.int32, device="cuda")
        want = torch.full((R, hq, hd), float("nan"), device="cuda")
        got = torch.full((R, hq, hd), float("nan"), device="cuda")
        spd.attention(q, k, v, pos, want, ws)
        spd.binding.attention_static_scratch(q, k, v, pos, got)
        torch.cuda.synchronize()
        # same kernel, grid and chunk-order merge: bit-identical, and no row left at its NaN fill
        assert not torch.isnan(want).any(), f"call {call}"
        assert torch.equal(got, want), f"call {call}"


def test_static_scratch_rejects_sizes_beyond_its_array(spd):
    hq, hkv, hd, R, max_seq = 32, 8, 128, 32, 32768   # ~139 MB of partials > 16 MiB
    q = torch.zeros(R, hq, hd, device="cuda")
    k = torch.zeros(hkv, 8, hd, dtype=torch.bfloat16, device="cuda")
    pos = torch.ones(R, dtype=torch.int32, device="cuda")
    out = torch.zeros(R, hq, hd, device="cuda")
    L = spd.lib()
    rc = L.spd_attention_static_scratch(q.data_ptr(), k.data_ptr(), k.data_ptr(), 1, pos.data_ptr(),
                                        R, hq, hkv, hd, max_seq, out.data_ptr(), None)
    assert rc == -1
    assert "static scratch holds" in L.spd_last_error(None).decode()
