"""Kernel-level parity on the GPU: the grouped GEMV engine and split-K decode attention against the
oracle's own pieces (oracle.model.rmsnorm, matrix products, softmax_attend) on seeded inputs."""
import numpy as np
import pytest
import torch

import spd_inputs as si
from oracle import model as om

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spd():
    from speculative_pipeline_decoding_gb300 import build_ext
    build_ext.build()
    import speculative_pipeline_decoding_gb300 as spd
    return spd


def _normal(seed, shape, dtype, std=0.02):
    key = si.tensor_key(seed, "ops")
    return si.normal_like(key, int(np.prod(shape)), std, dtype, "cuda").view(shape)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,cols,G,norm", [(6144, 2560, 8, True), (4099, 9728, 3, False),
                                              (37, 2048, 1, True), (2560, 12800, 2, False),
                                              (300, 2056, 2, True), (129, 2080, 3, False)])
def test_grouped_gemv_matches_oracle(spd, dtype, rows, cols, G, norm):
    Ws = [_normal(10 + g, (rows, cols), dtype) for g in range(G)]
    xs = [_normal(50 + g, (cols,), torch.float32, std=1.0) for g in range(G)]
    ys = [torch.full((rows,), float("nan"), device="cuda") for _ in range(G)]
    nw = (torch.linspace(0.5, 1.5, cols, device="cuda") if norm else None)
    spd.grouped_gemv(Ws, xs, ys, norm_weight=nw, eps=1e-6)
    torch.cuda.synchronize()
    for g in range(G):
        W = Ws[g].float().cpu().numpy().astype(np.float64)
        x = xs[g].cpu().numpy()
        if norm:
            x = om.rmsnorm(x, nw.cpu().numpy(), 1e-6)
        want = W @ x.astype(np.float64)
        got = ys[g].cpu().numpy()
        err = np.max(np.abs(got - want)) / np.max(np.abs(want))
        assert err < 1e-5, (g, err)


def test_grouped_gemv_rows_do_not_depend_on_the_batch(spd):
    """A group's output is bit-identical whether it runs alone or with seven other groups."""
    rows, cols = 6144, 2560
    Ws = [_normal(100 + g, (rows, cols), torch.bfloat16) for g in range(8)]
    xs = [_normal(200 + g, (cols,), torch.float32, std=1.0) for g in range(8)]
    nw = torch.ones(cols, device="cuda")
    ys8 = [torch.empty(rows, device="cuda") for _ in range(8)]
    spd.grouped_gemv(Ws, xs, ys8, norm_weight=nw)
    for g in (0, 3, 7):
        y1 = torch.empty(rows, device="cuda")
        spd.grouped_gemv([Ws[g]], [xs[g]], [y1], norm_weight=nw)
        torch.cuda.synchronize()
        assert torch.equal(y1, ys8[g])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("hq,hkv,hd", [(32, 8, 128), (16, 16, 128), (4, 4, 64)])
def test_attention_matches_oracle(spd, dtype, hq, hkv, hd):
    max_seq = 700
    positions = [1, 2, 127, 128, 129, 300, 511, 700]
    R = len(positions)
    g = torch.Generator(device="cpu").manual_seed(0)
    k = (torch.randn(hkv, max_seq, hd, generator=g) * 0.5).to(dtype).cuda()
    v = torch.randn(hkv, max_seq, hd, generator=g).to(dtype).cuda()
    q = (torch.randn(R, hq, hd, generator=g) * 0.5).cuda()
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    out = torch.full((R, hq, hd), float("nan"), device="cuda")
    ws_bytes = spd.attention_workspace_bytes(R, hq, hkv, hd, max_seq)
    ws = torch.zeros(ws_bytes // 4 + 1, dtype=torch.int32, device="cuda")
    for rep in range(2):  # the workspace is left zeroed for the next call
        spd.attention(q, k, v, pos, out, ws)
        torch.cuda.synchronize()
        kc, vc, qc, oc = (t.float().cpu().numpy() for t in (k, v, q, out))
        gq = hq // hkv
        for r, p in enumerate(positions):
            for h in range(hq):
                want = om.softmax_attend(qc[r, h], kc[h // gq, :p], vc[h // gq, :p])
                np.testing.assert_allclose(oc[r, h], want, rtol=2e-5, atol=2e-5)


def test_attention_split_count_depends_only_on_position(spd):
    """Query r's output is bit-identical when computed alone or among other queries."""
    hq, hkv, hd, max_seq = 32, 8, 128, 1000
    g = torch.Generator(device="cpu").manual_seed(1)
    k = torch.randn(hkv, max_seq, hd, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(hkv, max_seq, hd, generator=g).to(torch.bfloat16).cuda()
    positions = [999, 998, 997, 996, 995, 994, 993, 992]
    q = torch.randn(8, hq, hd, generator=g).cuda()
    ws = torch.zeros(spd.attention_workspace_bytes(8, hq, hkv, hd, max_seq) // 4 + 1,
                     dtype=torch.int32, device="cuda")
    out8 = torch.empty(8, hq, hd, device="cuda")
    spd.attention(q, k, v, torch.tensor(positions, dtype=torch.int32, device="cuda"), out8, ws)
    for r in (0, 5):
        out1 = torch.empty(1, hq, hd, device="cuda")
        spd.attention(q[r:r + 1].contiguous(), k, v,
                      torch.tensor([positions[r]], dtype=torch.int32, device="cuda"), out1, ws)
        torch.cuda.synchronize()
        assert torch.equal(out1[0], out8[r])


def test_attention_rows_outside_the_cache_come_back_nan(spd):
    """A caller position outside 1..max_seq is not computed (no read past the cache, no partial past
    the workspace); that row reads NaN and the other rows are unaffected."""
    hq, hkv, hd, max_seq = 8, 2, 64, 300
    g = torch.Generator(device="cpu").manual_seed(2)
    k = torch.randn(hkv, max_seq, hd, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(hkv, max_seq, hd, generator=g).to(torch.bfloat16).cuda()
    positions = [5, 0, max_seq + 1, 300, -3]
    R = len(positions)
    q = torch.randn(R, hq, hd, generator=g).cuda()
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    out = torch.zeros(R, hq, hd, device="cuda")
    ws = torch.zeros(spd.attention_workspace_bytes(R, hq, hkv, hd, max_seq) // 4 + 1,
                     dtype=torch.int32, device="cuda")
    spd.attention(q, k, v, pos, out, ws)
    torch.cuda.synchronize()
    oc = out.cpu()
    for r in (1, 2, 4):
        assert torch.isnan(oc[r]).all(), r
    kc, vc, qc = (t.float().cpu().numpy() for t in (k, v, q))
    for r in (0, 3):
        p = positions[r]
        for h in range(hq):
            want = om.softmax_attend(qc[r, h], kc[h // (hq // hkv), :p], vc[h // (hq // hkv), :p])
            np.testing.assert_allclose(oc[r, h].numpy(), want, rtol=2e-5, atol=2e-5)


@pytest.mark.parametrize("hq,hkv,hd,pos0,R,max_seq", [
    (32, 8, 128, 1, 32, 300),        # first block: keys 1..32, one chunk, one split
    (32, 8, 128, 1000, 32, 1100),    # a later block: causal chunk at the diagonal
    (32, 8, 128, 8001, 32, 8200),    # long context: split over CTAs, merged in split order
    (16, 16, 128, 470, 17, 600),     # MHA, ragged block
    (8, 2, 64, 250, 32, 300),        # head size 64
    (4, 4, 64, 1, 1, 8),             # one query at position 1
])
def test_prefill_attention_matches_oracle(spd, hq, hkv, hd, pos0, R, max_seq):
    g = torch.Generator(device="cpu").manual_seed(pos0 + R)
    k = (torch.randn(hkv, max_seq, hd, generator=g) * 0.5).to(torch.bfloat16).cuda()
    v = torch.randn(hkv, max_seq, hd, generator=g).to(torch.bfloat16).cuda()
    q = (torch.randn(R, hq, hd, generator=g) * 0.5).cuda()
    out = torch.full((R, hq, hd), float("nan"), device="cuda")
    ws = torch.zeros(spd.binding.prefill_attention_workspace_bytes(hq, hkv, hd, max_seq) // 4 + 64,
                     dtype=torch.int32, device="cuda")
    for rep in range(2):  # the workspace's tickets are left zeroed for the next call
        spd.binding.prefill_attention(q, k, v, pos0, out, ws)
        torch.cuda.synchronize()
        kc, vc, qc, oc = (t.float().cpu().numpy() for t in (k, v, q, out))
        gq = hq // hkv
        for r in range(R):
            p = pos0 + r
            for h in range(hq):
                want = om.softmax_attend(qc[r, h], kc[h // gq, :p], vc[h // gq, :p])
                np.testing.assert_allclose(oc[r, h], want, rtol=1e-4, atol=1e-4, err_msg=f"rep {rep} row {r} head {h}")
