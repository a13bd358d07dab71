"""Oracle, part 1: the decoder that Speculative Pipeline Decoding pipelines.

TEST INFRASTRUCTURE ONLY.  Plain, slow, fp32 CPU code (numpy) that the CUDA
path is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import it; the product path
never does, and the two share no code (inputs come from ``spd_inputs``).

What is computed, and from where:

* The pages fix only the model family (Qwen3.5-4B / 9B decoders, "SPD" summary
  page, section 实验结果; v3 summary, section 4) and that the target is an
  L-layer decoder whose KV cache is kept per layer ("SPD" summary page,
  前置知识 "KV Cache与回滚").  The layer itself is the plain pre-norm decoder
  layer: RMSNorm -> Q/K/V projections -> rotary position embedding
  (rotate-half pairing i <-> i+hd/2, theta 10000, 0-based position index) ->
  causal softmax attention with grouped KV heads -> output projection and
  residual -> RMSNorm -> SwiGLU feed-forward and residual.  Final RMSNorm and an
  untied LM head give the logits; greedy decoding takes the argmax (lowest index
  on ties).  No biases, no q/k norm, eps 1e-6.
* Precision: every product, sum and activation is fp32.  Matrices and
  embeddings are stored in the model dtype (bf16 or fp32) and used exactly.
  The KV cache stores K and V rounded to the model dtype (bf16
  round-to-nearest-even for a bf16 model), which is what a bf16 model keeps.
  RoPE angles are formed in fp64 and their cos/sin rounded to fp32.
* Library primitives used as steps: ``numpy.matmul`` (a matrix product),
  ``numpy.exp``/``numpy.sqrt``/``numpy.cos``/``numpy.sin``.

Pins (tests/test_oracle_model.py) hold this file to facts that do not come
from it: torch's own scaled-dot-product attention / rms_norm / silu on the
same numbers, the complex-rotation form of RoPE, the LM heads (final norm with
the stack's own weight, then the vocab matrix) against torch's rms_norm and a
float64 product with planted mistakes caught, closed forms of special cases
(one key -> the value, zero query -> the mean value), causality, and
prefill-vs-incremental agreement.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np


# ---------------------------------------------------------------------------
# storage rounding
# ---------------------------------------------------------------------------
def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bf16 (ties to even) -> fp32, by its bit-level definition."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    r = ((u + bias) & np.uint64(0xFFFF0000)).astype(np.uint32)
    return r.view(np.float32).reshape(np.shape(x))


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    return round_bf16(x) if dtype == "bf16" else np.asarray(x, dtype=np.float32)


# ---------------------------------------------------------------------------
# elementary pieces
# ---------------------------------------------------------------------------
def rmsnorm(h: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """h / sqrt(mean(h^2) + eps) * w over the last axis, fp32."""
    h = h.astype(np.float32, copy=False)
    ms = np.mean(h * h, axis=-1, keepdims=True, dtype=np.float32)
    return (h / np.sqrt(ms + np.float32(eps))) * w


def rope_tables(positions: Sequence[int], head_dim: int, theta: float
                ) -> Tuple[np.ndarray, np.ndarray]:
    """cos, sin of angle (pos-1) * theta^(-2i/hd), i < hd/2, for 1-based positions."""
    half = head_dim // 2
    inv = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / head_dim)
    ang = (np.asarray(positions, dtype=np.float64) - 1.0)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def apply_rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate-half RoPE. x: [R, heads, hd]; cos/sin: [R, hd/2]."""
    half = x.shape[-1] // 2
    x1, x2 = x[..., :half], x[..., half:]
    c, s = cos[:, None, :], sin[:, None, :]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1).astype(np.float32)


def silu(x: np.ndarray) -> np.ndarray:
    return (x / (np.float32(1.0) + np.exp(-x))).astype(np.float32)


def softmax_attend(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """One query head over T keys: softmax(q.K^T / sqrt(hd)) V.  q [hd], K,V [T, hd]."""
    s = (K @ q) * np.float32(1.0 / np.sqrt(q.shape[-1]))
    s = s - np.max(s)
    p = np.exp(s)
    p = p / np.sum(p, dtype=np.float32)
    return (p @ V).astype(np.float32)


def top2(logits: np.ndarray) -> Tuple[int, int, float, float]:
    """(top1 index, top2 index, top1 value, top2 value); lowest index wins ties."""
    i1 = int(np.argmax(logits))
    rest = logits.copy()
    rest[i1] = -np.inf
    i2 = int(np.argmax(rest))
    return i1, i2, float(logits[i1]), float(logits[i2])


# ---------------------------------------------------------------------------
# KV cache: one list of cached positions per layer, with an explicit length
# ---------------------------------------------------------------------------
class KVCache:
    """Per-layer K/V store.  Entry p-1 of layer l holds position p.

    ``append`` insists that a position arrives exactly after its predecessor at
    the same layer, so any schedule that reads stale or missing entries fails
    loudly instead of computing something plausible.
    """

    def __init__(self, n_layers: int, max_len: int, n_kv: int, head_dim: int, dtype: str):
        self.k = np.zeros((n_layers, max_len, n_kv, head_dim), np.float32)
        self.v = np.zeros((n_layers, max_len, n_kv, head_dim), np.float32)
        self.length = [0] * n_layers
        self.dtype = dtype

    def append(self, l: int, pos: int, k: np.ndarray, v: np.ndarray) -> None:
        if self.length[l] != pos - 1:
            raise AssertionError(f"layer {l}: cache holds {self.length[l]} positions, "
                                 f"cannot append position {pos}")
        self.k[l, pos - 1] = to_storage(k, self.dtype)
        self.v[l, pos - 1] = to_storage(v, self.dtype)
        self.length[l] = pos

    def view(self, l: int, upto: int) -> Tuple[np.ndarray, np.ndarray]:
        if upto > self.length[l]:
            raise AssertionError(f"layer {l}: reading {upto} positions, cache holds {self.length[l]}")
        return self.k[l, :upto], self.v[l, :upto]

    def truncate(self, new_len: int) -> None:
        """Every layer keeps positions 1..new_len and drops the rest."""
        self.length = [min(x, new_len) for x in self.length]


# ---------------------------------------------------------------------------
# decoder
# ---------------------------------------------------------------------------
@dataclass
class LayerParams:
    attn_norm: np.ndarray
    wq: np.ndarray
    wk: np.ndarray
    wv: np.ndarray
    wo: np.ndarray
    ffn_norm: np.ndarray
    w_gate: np.ndarray
    w_up: np.ndarray
    w_down: np.ndarray


def _f32(t) -> np.ndarray:
    """torch tensor (bf16 or fp32) or array -> contiguous fp32 numpy array (exact)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to("cpu", torch.float32).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(t, dtype=np.float32)


def load_layer(params: Dict, prefix: str) -> LayerParams:
    return LayerParams(*[_f32(params[prefix + s]) for s in
                         ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm",
                          "w_gate", "w_up", "w_down")])


class Decoder:
    """The L-layer stack: embedding, decoder layers, final norm, LM head."""

    def __init__(self, cfg, params: Dict, n_layers: Optional[int] = None, prefix: str = "",
                 with_embedding: bool = True, norm_name: str = "final_norm",
                 head_name: str = "lm_head"):
        self.cfg = cfg
        self.L = cfg.n_layers if n_layers is None else n_layers
        self.d = cfg.d_model
        self.hq, self.hkv, self.hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
        self.eps, self.theta, self.dtype = cfg.norm_eps, cfg.rope_theta, cfg.dtype
        self.layers = [load_layer(params, f"{prefix}layers.{l}.") for l in range(self.L)]
        self.embed_w = _f32(params["embed"]) if with_embedding else None
        self.norm = _f32(params[prefix + norm_name])
        self.head_w = _f32(params[prefix + head_name])

    def new_cache(self, max_len: int) -> KVCache:
        return KVCache(self.L, max_len, self.hkv, self.hd, self.dtype)

    def embed(self, token: int) -> np.ndarray:
        return self.embed_w[int(token)].copy()

    def layer(self, l: int, H: np.ndarray, positions: Sequence[int], cache: KVCache) -> np.ndarray:
        """Rows H [R, d] at consecutive positions through decoder layer l.

        Each row's K/V is appended to layer l's cache; row r then attends to
        cached positions 1..positions[r] (causal).
        """
        p = self.layers[l]
        R = H.shape[0]
        hq, hkv, hd = self.hq, self.hkv, self.hd
        X = rmsnorm(H, p.attn_norm, self.eps)
        Q = (X @ p.wq.T).reshape(R, hq, hd)
        K = (X @ p.wk.T).reshape(R, hkv, hd)
        Vv = (X @ p.wv.T).reshape(R, hkv, hd)
        cos, sin = rope_tables(positions, hd, self.theta)
        Q = apply_rope(Q, cos, sin)
        K = apply_rope(K, cos, sin)
        for r, pos in enumerate(positions):
            cache.append(l, pos, K[r], Vv[r])
        group = hq // hkv
        O = np.zeros((R, hq, hd), np.float32)
        for r, pos in enumerate(positions):
            Kc, Vc = cache.view(l, pos)
            for h in range(hq):
                O[r, h] = softmax_attend(Q[r, h], Kc[:, h // group], Vc[:, h // group])
        H = H + O.reshape(R, hq * hd) @ p.wo.T
        X = rmsnorm(H, p.ffn_norm, self.eps)
        U = silu(X @ p.w_gate.T) * (X @ p.w_up.T)
        return (H + U @ p.w_down.T).astype(np.float32)

    def logits(self, h: np.ndarray) -> np.ndarray:
        return (self.head_w @ rmsnorm(h, self.norm, self.eps)).astype(np.float32)

    def prefill(self, tokens: Sequence[int], cache: KVCache, anchors: Sequence[int] = ()
                ) -> Tuple[np.ndarray, Dict[int, Dict[int, np.ndarray]]]:
        """All prompt rows through all layers; returns h^(L) rows and anchor states.

        anchor_states[pos][b] = residual of position pos after b layers, for b in anchors.
        """
        P = len(tokens)
        positions = list(range(1, P + 1))
        H = np.stack([self.embed(t) for t in tokens]).astype(np.float32)
        states: Dict[int, Dict[int, np.ndarray]] = {p: {} for p in positions}
        if 0 in anchors:
            for r, p in enumerate(positions):
                states[p][0] = H[r].copy()
        for l in range(self.L):
            H = self.layer(l, H, positions, cache)
            if (l + 1) in anchors:
                for r, p in enumerate(positions):
                    states[p][l + 1] = H[r].copy()
        return H, states


def greedy_ar(model: Decoder, prompt: Sequence[int], gen: int, max_len: Optional[int] = None,
              forced: Optional[Sequence[int]] = None) -> Dict:
    """Plain greedy autoregressive decoding of ``gen`` tokens after ``prompt``.

    With ``forced`` (a stream of ``gen`` tokens) the model is teacher-forced on it:
    each position's prediction is still reported, but the next input is forced[i].
    Returns tokens (the oracle's own predictions), top-2 gaps and top-2 ids.
    """
    P = len(prompt)
    cache = model.new_cache(max_len or (P + gen + 1))
    H, _ = model.prefill(prompt, cache)
    i1, i2, v1, v2 = top2(model.logits(H[-1]))
    preds, gaps, seconds = [i1], [v1 - v2], [i2]
    for i in range(gen - 1):
        pos = P + 1 + i
        tok = forced[i] if forced is not None else preds[-1]
        h = model.embed(tok)[None, :]
        for l in range(model.L):
            h = model.layer(l, h, [pos], cache)
        i1, i2, v1, v2 = top2(model.logits(h[0]))
        preds.append(i1)
        gaps.append(v1 - v2)
        seconds.append(i2)
    return {"tokens": preds, "gaps": gaps, "second": seconds}
