"""Seeded synthetic inputs for Speculative Pipeline Decoding workloads.

This module is shared by the CPU oracle and by the CUDA path.  It holds the
workload descriptions (model shapes, pipeline width, anchors, prompt and
generation lengths, acceptance rates) and the counter-based generators for
every input: weights, prompt token ids and the per-position acceptance coins of
the seeded-acceptance harness.  It holds none of the method's arithmetic.

Generator definitions (identical results on any device and any torch version):

* ``splitmix64`` -- the published SplitMix64 generator (Steele, Lea, Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014): state advances
  by the golden-ratio increment 0x9E3779B97F4A7C15 and each output is the
  state passed through the mix function with shifts 30/27/31 and multipliers
  0xBF58476D1CE4E5B9 / 0x94D049BB133111EB.
* weights: element ``i`` of a tensor is drawn from the ``i``-th SplitMix64
  output of a per-tensor key.  Its four 16-bit fields are summed (an
  Irwin-Hall sum of four discrete uniforms), centred and scaled to standard
  deviation ``init_std`` in one fp32 multiply, then rounded to the storage
  dtype (bf16 round-to-nearest-even, or kept fp32).  Integer arithmetic plus
  one correctly rounded multiply make CPU and GPU generation bit-identical.
* prompts: token ``i`` is the top 53 bits of the ``i``-th output modulo vocab.
* acceptance coins: ``coin(q)`` is the top 53 bits of
  ``splitmix64(seed XOR q*0x9E3779B97F4A7C15)`` divided by 2**53.
* sampling uniforms: stream s (draft, accept, resample, ar) is the coin sequence
  of the key ``splitmix64(seed XOR (s+1))``, rounded to fp32 (kept below 1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Iterable, List, Optional, Tuple

import torch

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB


# ---------------------------------------------------------------------------
# workload descriptions
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class ModelConfig:
    """Shape of one uniform decoder (target) and its draft module."""

    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_ffn: int
    vocab: int
    dtype: str  # storage type of matrices, embeddings and KV cache: "f32" | "bf16"
    rope_theta: float = 10000.0
    norm_eps: float = 1e-6
    init_std: float = 0.02


@dataclass(frozen=True)
class Workload:
    """One synthetic decode workload: model, pipeline, prompt and acceptance."""

    name: str
    model: ModelConfig
    n_stages: int          # n
    pdm_layers: int        # Ls
    anchors: Tuple[int, ...]  # B
    prompt_len: int
    gen_len: int
    alphas: Tuple[float, ...]
    weight_seed: int = 0
    prompt_seed: int = 1
    coin_seed: int = 2

    @property
    def max_seq(self) -> int:
        return self.prompt_len + self.gen_len + self.n_stages + 1


_TINY = ModelConfig(n_layers=8, d_model=256, n_heads=4, n_kv_heads=4, head_dim=64,
                    d_ffn=1024, vocab=1024, dtype="f32")
_M1P5B = ModelConfig(n_layers=32, d_model=2048, n_heads=16, n_kv_heads=16, head_dim=128,
                     d_ffn=5632, vocab=32000, dtype="bf16")
_M4B = ModelConfig(n_layers=32, d_model=2560, n_heads=32, n_kv_heads=8, head_dim=128,
                   d_ffn=9728, vocab=151936, dtype="bf16")
_M9B = ModelConfig(n_layers=32, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128,
                   d_ffn=12288, vocab=151936, dtype="bf16")
_B32 = (0, 8, 16, 24, 31)

WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_f32_n2", _TINY, 2, 1, (0, 2, 4, 6, 7), 16, 64, (0.7,)),
        Workload("dense1.5b_bf16_n8", _M1P5B, 8, 4, _B32, 512, 256, (0.8,)),
        Workload("gqa4b_bf16_n8", _M4B, 8, 4, _B32, 1024, 512, (0.6, 0.85)),
        Workload("gqa9b_bf16_n4", _M9B, 4, 8, _B32, 2048, 512, (0.5, 0.9)),
        Workload("gqa9b_bf16_n8", _M9B, 8, 4, _B32, 2048, 512, (0.5, 0.9)),
        Workload("gqa9b_bf16_n16", _M9B, 16, 2, _B32, 2048, 512, (0.5, 0.9)),
        Workload("gqa4b_bf16_n8_ctx32k", _M4B, 8, 4, _B32, 32768, 256, (0.8,)),
    ]
}


def small_model(**kw) -> ModelConfig:
    """A model shape for unit tests; keyword arguments override the defaults."""
    base = dict(n_layers=4, d_model=64, n_heads=4, n_kv_heads=2, head_dim=16,
                d_ffn=128, vocab=96, dtype="f32")
    base.update(kw)
    return ModelConfig(**base)


# ---------------------------------------------------------------------------
# SplitMix64, in Python integers and in torch int64 (wrapping) arithmetic
# ---------------------------------------------------------------------------
def mix64(z: int) -> int:
    """SplitMix64 output function on a 64-bit state (Python integers)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * _MIX1) & MASK64
    z = ((z ^ (z >> 27)) * _MIX2) & MASK64
    return z ^ (z >> 31)


def splitmix64(x: int) -> int:
    """One SplitMix64 step from state ``x``: advance by the golden increment, then mix."""
    return mix64((x + GOLDEN) & MASK64)


def _signed(u: int) -> int:
    u &= MASK64
    return u - (1 << 64) if u >= (1 << 63) else u


def _srl(x: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 lanes holding 64-bit unsigned values."""
    return (x >> k) & ((1 << (64 - k)) - 1)


def mix64_t(z: torch.Tensor) -> torch.Tensor:
    """SplitMix64 output function on int64 lanes (multiplication wraps mod 2**64)."""
    z = (z ^ _srl(z, 30)) * _signed(_MIX1)
    z = (z ^ _srl(z, 27)) * _signed(_MIX2)
    return z ^ _srl(z, 31)


def stream_t(key: int, start: int, count: int, device) -> torch.Tensor:
    """Outputs ``start .. start+count-1`` of the SplitMix64 stream seeded with ``key``.

    Output ``i`` is ``mix64(key + (i+1)*GOLDEN)``, exactly the sequence SplitMix64 yields.
    """
    idx = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    state = idx * _signed(GOLDEN) + _signed(key)
    return mix64_t(state)


def stream_py(key: int, i: int) -> int:
    return mix64((key + (i + 1) * GOLDEN) & MASK64)


def fnv1a64(s: str) -> int:
    h = 0xCBF29CE484222325
    for b in s.encode():
        h ^= b
        h = (h * 0x100000001B3) & MASK64
    return h


def tensor_key(seed: int, name: str) -> int:
    return mix64(fnv1a64(name) ^ splitmix64(seed))


# Irwin-Hall(4) of 16-bit uniforms: mean 4*32767.5, variance 4*(65536**2-1)/12
_IH_CENTER = 131070
_IH_STD = math.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0)


def normal_like(key: int, numel: int, std: float, dtype: torch.dtype, device,
                chunk: int = 1 << 24) -> torch.Tensor:
    """Approximately N(0, std) values, bit-identical on CPU and GPU (see module docstring)."""
    out = torch.empty(numel, dtype=dtype, device=device)
    scale = torch.tensor(std / _IH_STD, dtype=torch.float32, device=device)
    for s in range(0, numel, chunk):
        c = min(chunk, numel - s)
        u = stream_t(key, s, c, device)
        tot = (u & 0xFFFF) + (_srl(u, 16) & 0xFFFF) + (_srl(u, 32) & 0xFFFF) + _srl(u, 48)
        v = (tot - _IH_CENTER).to(torch.float32) * scale
        out[s:s + c] = v.to(dtype)
    return out


# ---------------------------------------------------------------------------
# weights
# ---------------------------------------------------------------------------
def torch_dtype(cfg: ModelConfig) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[cfg.dtype]


def layer_shapes(cfg: ModelConfig) -> List[Tuple[str, Tuple[int, ...], bool]]:
    """(suffix, shape, is_norm) of one decoder layer's parameters (y = W x, W is [out, in])."""
    d, hq, hkv, hd, f = cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.d_ffn
    return [
        ("attn_norm", (d,), True),
        ("wq", (hq * hd, d), False),
        ("wk", (hkv * hd, d), False),
        ("wv", (hkv * hd, d), False),
        ("wo", (d, hq * hd), False),
        ("ffn_norm", (d,), True),
        ("w_gate", (f, d), False),
        ("w_up", (f, d), False),
        ("w_down", (d, f), False),
    ]


def weight_specs(w: Workload) -> List[Tuple[str, Tuple[int, ...], bool]]:
    """Every parameter of the target decoder and of the draft module, in a fixed order."""
    cfg = w.model
    d, V = cfg.d_model, cfg.vocab
    specs: List[Tuple[str, Tuple[int, ...], bool]] = [("embed", (V, d), False)]
    for l in range(cfg.n_layers):
        specs += [(f"layers.{l}.{s}", shp, nrm) for s, shp, nrm in layer_shapes(cfg)]
    specs += [("final_norm", (d,), True), ("lm_head", (V, d), False)]
    for j in range(len(w.anchors)):
        specs.append((f"pdm.fc.{j}", (d, (j + 1) * d), False))
    for l in range(w.pdm_layers):
        specs += [(f"pdm.layers.{l}.{s}", shp, nrm) for s, shp, nrm in layer_shapes(cfg)]
    specs += [("pdm.norm", (d,), True), ("pdm.lm_head", (V, d), False)]
    return specs


def generate_weights(w: Workload, device="cpu", names: Optional[Iterable[str]] = None
                     ) -> Dict[str, torch.Tensor]:
    """All parameters of workload ``w`` on ``device``.

    Matrices and embeddings: approximately N(0, init_std) in the model dtype.
    Norm weights: ones, fp32.
    """
    cfg = w.model
    dt = torch_dtype(cfg)
    wanted = None if names is None else set(names)
    out: Dict[str, torch.Tensor] = {}
    for name, shape, is_norm in weight_specs(w):
        if wanted is not None and name not in wanted:
            continue
        if is_norm:
            out[name] = torch.ones(shape, dtype=torch.float32, device=device)
        else:
            numel = math.prod(shape)
            out[name] = normal_like(tensor_key(w.weight_seed, name), numel, cfg.init_std,
                                    dt, device).view(shape)
    return out


def prompt_tokens(w: Workload, length: Optional[int] = None, device="cpu") -> torch.Tensor:
    """Uniform-random prompt token ids (int32)."""
    n = w.prompt_len if length is None else length
    u = stream_t(tensor_key(w.prompt_seed, "prompt"), 0, n, device)
    return (_srl(u, 11) % w.model.vocab).to(torch.int32)


# ---------------------------------------------------------------------------
# seeded acceptance (harness knob: which positions get a correct draft)
# ---------------------------------------------------------------------------
def coin(seed: int, q: int) -> float:
    return (splitmix64(seed ^ ((q * GOLDEN) & MASK64)) >> 11) / float(1 << 53)


def accept_mask(seed: int, alpha: float, first: int, last: int) -> List[bool]:
    """mask[q-first] = coin(q) < alpha for positions q in [first, last]."""
    return [coin(seed, q) < alpha for q in range(first, last + 1)]


# draft-override modes per position (shared vocabulary of both sides)
DRAFT_RAW = 0          # use the draft module's top-1 as is
DRAFT_FORCE_REF = 1    # replace the draft by the reference (true greedy) token
DRAFT_FORCE_OTHER = 2  # draft module's highest-ranked token that differs from the reference


def override_modes(seed: int, alpha: float, first: int, last: int) -> List[int]:
    return [DRAFT_FORCE_REF if ok else DRAFT_FORCE_OTHER
            for ok in accept_mask(seed, alpha, first, last)]


# ---------------------------------------------------------------------------
# uniforms of sampled decoding (the random numbers the method draws are inputs)
# ---------------------------------------------------------------------------
SAMPLING_STREAMS = ("draft", "accept", "resample", "ar")


def sampling_uniforms(seed: int, first: int, last: int) -> Dict[str, List[float]]:
    """Per stream, uniforms u[q] in [0, 1) for positions q in [first, last]: stream s of seed is
    the coin sequence of the key splitmix64(seed XOR (s+1)), rounded to fp32 below 1."""
    out = {}
    for s, name in enumerate(SAMPLING_STREAMS):
        key = splitmix64(seed ^ (s + 1))
        vals = []
        for q in range(first, last + 1):
            u = coin(key, q)
            f = float(torch.tensor(u, dtype=torch.float32))
            vals.append(f if f < 1.0 else float(torch.nextafter(torch.tensor(1.0), torch.tensor(0.0))))
        out[name] = vals
    return out


__all__ = [n for n in dir() if not n.startswith("_")]
