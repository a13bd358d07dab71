"""Pins of the oracle's decoder (oracle/model.py) against facts it does not define itself.

* bf16 rounding against torch's own fp32 -> bf16 conversion;
* RMSNorm against torch.nn.functional.rms_norm;
* a whole decoder layer against an independent construction from torch library
  routines (scaled_dot_product_attention with its causal mask and GQA
  expansion, rms_norm, silu) and the complex-number form of rotary embedding;
* closed forms: one cached key returns its value; a zero query averages values;
  RoPE at index 0 is the identity, preserves norms and depends only on
  relative position;
* causality and prefill == incremental decoding;
* the KV cache rejects out-of-order appends and reads past its length.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import spd_inputs as si
from oracle import model as om


def _rand(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return (g.standard_normal(shape) * scale).astype(np.float32)


def test_round_bf16_matches_torch_conversion():
    x = _rand(100000, 0, 3.0)
    # include exact ties: values halfway between two bf16 numbers
    ties = (np.arange(1, 2001, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.float32([0.0, -0.0, 1e-40, 65504.0])])
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(om.round_bf16(x), want)


def test_rmsnorm_matches_torch():
    h = _rand((5, 96), 1, 2.0)
    w = _rand(96, 2)
    got = om.rmsnorm(h, w, 1e-6)
    want = F.rms_norm(torch.from_numpy(h), (96,), torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(got, want, rtol=2e-6, atol=1e-6)


def _rope_complex(x, positions, theta):
    """RoPE as complex rotation of pairs (x_i, x_{i+hd/2}) by (pos-1)*theta^(-2i/hd)."""
    x = torch.from_numpy(x).double()
    hd = x.shape[-1]
    half = hd // 2
    z = torch.complex(x[..., :half], x[..., half:])
    inv = theta ** (-(2.0 * torch.arange(half, dtype=torch.float64)) / hd)
    ang = (torch.tensor(positions, dtype=torch.float64) - 1)[:, None] * inv[None, :]
    z = z * torch.polar(torch.ones_like(ang), ang)[:, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


def _torch_layer(p: om.LayerParams, H, positions, hq, hkv, hd, theta, eps, kv_round):
    """A decoder layer over a full causal block, built from torch library routines (fp64)."""
    T = lambda a: torch.from_numpy(np.asarray(a)).double()
    H = T(H)
    R = H.shape[0]
    X = F.rms_norm(H, (H.shape[1],), T(p.attn_norm), eps=eps)
    Q = (X @ T(p.wq).T).reshape(R, hq, hd).numpy()
    K = (X @ T(p.wk).T).reshape(R, hkv, hd).numpy()
    V = (X @ T(p.wv).T).reshape(R, hkv, hd)
    Q = _rope_complex(Q, positions, theta)
    K = _rope_complex(K, positions, theta)
    if kv_round:
        K = K.float().to(torch.bfloat16).double()
        V = V.float().to(torch.bfloat16).double()
    O = F.scaled_dot_product_attention(Q.transpose(0, 1)[None], K.transpose(0, 1)[None],
                                       V.transpose(0, 1)[None], is_causal=True,
                                       enable_gqa=True)[0].transpose(0, 1)
    H = H + O.reshape(R, hq * hd) @ T(p.wo).T
    X = F.rms_norm(H, (H.shape[1],), T(p.ffn_norm), eps=eps)
    H = H + (F.silu(X @ T(p.w_gate).T) * (X @ T(p.w_up).T)) @ T(p.w_down).T
    return H.numpy()


@pytest.mark.parametrize("dtype,hkv", [("f32", 2), ("f32", 4), ("bf16", 1)])
def test_layer_matches_torch_library_construction(dtype, hkv):
    cfg = si.small_model(n_layers=1, d_model=64, n_heads=4, n_kv_heads=hkv, head_dim=16,
                         d_ffn=96, vocab=50, dtype=dtype, init_std=0.1)
    w = si.Workload("t", cfg, 1, 1, (0, 1), 8, 4, (0.5,))
    params = si.generate_weights(w)
    params["layers.0.attn_norm"] = torch.linspace(0.5, 1.5, 64)
    params["layers.0.ffn_norm"] = torch.linspace(1.5, 0.5, 64)
    dec = om.Decoder(cfg, params)
    H = _rand((7, 64), 3)
    positions = list(range(1, 8))
    got = dec.layer(0, H, positions, dec.new_cache(8))
    want = _torch_layer(dec.layers[0], H, positions, 4, hkv, 16, cfg.rope_theta,
                        cfg.norm_eps, dtype == "bf16")
    tol = 2e-5 if dtype == "f32" else 2e-5
    np.testing.assert_allclose(got, want, rtol=tol, atol=tol * np.abs(want).max())


def test_attention_closed_forms():
    hd = 32
    v = _rand((1, hd), 4)
    q = _rand(hd, 5)
    np.testing.assert_allclose(om.softmax_attend(q, _rand((1, hd), 6), v), v[0], rtol=1e-6)
    V = _rand((9, hd), 7)
    np.testing.assert_allclose(om.softmax_attend(np.zeros(hd, np.float32), _rand((9, hd), 8), V),
                               V.mean(axis=0), rtol=1e-5, atol=1e-6)
    # permuting keys together with values leaves the output unchanged
    K = _rand((9, hd), 9)
    perm = np.random.default_rng(0).permutation(9)
    np.testing.assert_allclose(om.softmax_attend(q, K, V), om.softmax_attend(q, K[perm], V[perm]),
                               rtol=1e-5, atol=1e-6)


def test_rope_identity_norm_and_relative_position():
    hd = 64
    x = _rand((1, 3, hd), 10)
    c, s = om.rope_tables([1], hd, 10000.0)
    np.testing.assert_array_equal(om.apply_rope(x, c, s), x)
    c, s = om.rope_tables([777], hd, 10000.0)
    y = om.apply_rope(x, c, s)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-5)
    q, k = _rand((1, 1, hd), 11), _rand((1, 1, hd), 12)

    def dot(m, n):
        cm, sm = om.rope_tables([m], hd, 10000.0)
        cn, sn = om.rope_tables([n], hd, 10000.0)
        return float(np.sum(om.apply_rope(q, cm, sm) * om.apply_rope(k, cn, sn)))

    assert abs(dot(10, 3) - dot(110, 103)) < 1e-4 * abs(dot(10, 3)) + 1e-5
    assert abs(dot(10, 3) - dot(10, 4)) > 1e-4


def _small_decoder(dtype="f32", L=3):
    cfg = si.small_model(n_layers=L, d_model=64, n_heads=4, n_kv_heads=2, head_dim=16,
                         d_ffn=128, vocab=97, dtype=dtype, init_std=0.2)
    w = si.Workload("s", cfg, 1, 1, (0, L), 8, 8, (0.5,))
    return cfg, om.Decoder(cfg, si.generate_weights(w))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefill_equals_incremental_decoding(dtype):
    cfg, dec = _small_decoder(dtype)
    toks = [3, 17, 5, 60, 2, 91, 44, 8, 13]
    c1 = dec.new_cache(16)
    H, _ = dec.prefill(toks, c1)
    c2 = dec.new_cache(16)
    rows = []
    for i, t in enumerate(toks):
        h = dec.embed(t)[None]
        for l in range(dec.L):
            h = dec.layer(l, h, [i + 1], c2)
        rows.append(h[0])
    np.testing.assert_allclose(np.stack(rows), H, rtol=1e-5, atol=1e-5 * np.abs(H).max())


def test_causality_later_tokens_do_not_change_earlier_rows():
    cfg, dec = _small_decoder()
    a = [3, 17, 5, 60, 2, 91]
    b = [3, 17, 5, 1, 70, 9]
    Ha, _ = dec.prefill(a, dec.new_cache(8))
    Hb, _ = dec.prefill(b, dec.new_cache(8))
    np.testing.assert_array_equal(Ha[:3], Hb[:3])
    assert np.abs(Ha[3:] - Hb[3:]).max() > 1e-3


def test_anchor_states_are_residuals_after_b_layers():
    cfg, dec = _small_decoder(L=3)
    toks = [4, 9, 33]
    _, st = dec.prefill(toks, dec.new_cache(4), anchors=[0, 2, 3])
    np.testing.assert_array_equal(st[2][0], dec.embed(9))
    c = dec.new_cache(4)
    H = np.stack([dec.embed(t) for t in toks])
    H = dec.layer(0, H, [1, 2, 3], c)
    H = dec.layer(1, H, [1, 2, 3], c)
    np.testing.assert_array_equal(st[3][2], H[2])


def test_kv_cache_rejects_out_of_order_and_stale_reads():
    c = om.KVCache(2, 8, 1, 4, "f32")
    z = np.zeros((1, 4), np.float32)
    c.append(0, 1, z, z)
    with pytest.raises(AssertionError):
        c.append(0, 3, z, z)
    with pytest.raises(AssertionError):
        c.view(0, 2)
    c.append(0, 2, z, z)
    c.truncate(1)
    assert c.length == [1, 0]
    with pytest.raises(AssertionError):
        c.view(0, 2)


def test_greedy_ar_teacher_forcing_reproduces_free_run(tiny, tiny_ar):
    w, params, prompt, (target, _) = tiny
    forced = om.greedy_ar(target, prompt, 12, forced=tiny_ar["tokens"][:12])
    assert forced["tokens"] == tiny_ar["tokens"][:12]
    assert np.allclose(forced["gaps"], tiny_ar["gaps"][:12])


def test_top2_lowest_index_on_ties():
    x = np.float32([1.0, 3.0, 2.0, 3.0, 3.0])
    assert om.top2(x)[:2] == (1, 3)


def _head_workload(dtype):
    cfg = si.small_model(n_layers=1, d_model=64, n_heads=4, n_kv_heads=2, head_dim=16,
                         d_ffn=96, vocab=211, dtype=dtype, init_std=0.1)
    w = si.Workload("h", cfg, 1, 1, (0, 1), 4, 4, (0.5,))
    params = si.generate_weights(w)
    # non-unit, sign-changing norm weights, different for the two heads
    params["final_norm"] = torch.linspace(-1.25, 2.0, 64)
    params["pdm.norm"] = torch.linspace(1.75, 0.25, 64)
    return cfg, w, params


def _torch_head(h, norm_w, head_w, eps):
    """logits = W_lm . rms_norm(h; w), from torch's rms_norm and a float64 product."""
    T = lambda a: torch.as_tensor(np.asarray(a)).double()
    x = F.rms_norm(T(h), (h.shape[-1],), T(norm_w), eps=eps)
    return (T(head_w) @ x).numpy()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_head_logits_match_torch_norm_and_float64_product(dtype):
    """Target LM head (SPD summary step 5: the exiting token's logits) and the draft module's own
    head (step 4) = final RMSNorm with that stack's own weight, then the untied vocab matrix."""
    from oracle import spd as ospd
    cfg, w, params = _head_workload(dtype)
    target, pdm = ospd.build(w, params)
    for seed, stack, norm, head in ((21, target, "final_norm", "lm_head"),
                                    (22, pdm.stack, "pdm.norm", "pdm.lm_head")):
        h = _rand(64, seed, 3.0)
        want = _torch_head(h, params[norm], params[head].float(), cfg.norm_eps)
        got = stack.logits(h)
        assert got.shape == (cfg.vocab,)
        np.testing.assert_allclose(got, want, rtol=2e-5, atol=2e-5 * np.abs(want).max())
        # the argmax the verification uses is the float64 construction's
        assert om.top2(got)[0] == int(np.argmax(want)) or \
            np.sort(want)[-1] - np.sort(want)[-2] < 1e-4


def test_planted_head_mistakes_are_caught(monkeypatch):
    """A head that skips the final norm, or normalises with the other stack's weight, fails the pin."""
    from oracle import spd as ospd
    cfg, w, params = _head_workload("f32")
    target, pdm = ospd.build(w, params)
    h = _rand(64, 23, 3.0)
    want = _torch_head(h, params["final_norm"], params["lm_head"], cfg.norm_eps)

    def far(got):
        return np.abs(got - want).max() > 1e-2 * np.abs(want).max()

    with monkeypatch.context() as m:  # dropped final norm
        m.setattr(om, "rmsnorm", lambda x, wt, eps: x)
        assert far(target.logits(h))
    swapped = om.Decoder(cfg, params, norm_name="pdm.norm")  # the draft module's norm weight
    assert far(swapped.logits(h))
    with monkeypatch.context() as m:  # norm without its weight (all ones)
        m.setattr(target, "norm", np.ones(64, np.float32))
        assert far(target.logits(h))
    assert not far(target.logits(h))
