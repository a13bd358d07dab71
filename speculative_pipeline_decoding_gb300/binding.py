"""Python binding of the SPD C ABI (include/spd.h): argument marshalling only.

Every step of the decoding path runs in the CUDA library; this module turns Python / torch
arguments into the C structs and pointers of the ABI, raises :class:`SpdError` on a non-zero
status, and refuses to work without the compiled library (there is no fallback).

Weights are passed as a dict of CUDA tensors named like the parameters of a decoder:
``embed``, ``layers.{l}.{attn_norm,wq,wk,wv,wo,ffn_norm,w_gate,w_up,w_down}``, ``final_norm``,
``lm_head``, ``pdm.fc.{j}``, ``pdm.layers.{l}.*``, ``pdm.norm``, ``pdm.lm_head``.  Matrices are
row-major [out, in] in the model dtype (bf16 or fp32), norm weights fp32.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Dict, Optional, Sequence, Tuple

import numpy as np
import torch

from . import build_ext

MAX_ANCHORS = 8
DTYPE_F32, DTYPE_BF16 = 0, 1
OPT_GRAPHS, OPT_COSCHED, OPT_TARGET_ONLY, OPT_DEBUG_LOGITS, OPT_PDL, OPT_STEP = 1, 2, 4, 8, 16, 32
OPT_POST_STEP = 64  # draft module after the target step, on its output state
OPT_DEFAULT = OPT_GRAPHS | OPT_COSCHED | OPT_PDL | OPT_STEP
DUMP_STATE, DUMP_RESID, DUMP_ANCHORS, DUMP_PDM_Z, DUMP_LOGITS, DUMP_SEQ, DUMP_TRACE, DUMP_KVLEN, DUMP_PREFILL_H = range(9)
_OPS = ["qkv", "rope_append", "attention", "o_proj", "gate_up", "down", "anchor_fc", "head",
        "control"]
KIND_NAMES = _OPS + ["draft_" + k for k in _OPS]
STATE_FIELDS = ["t", "a", "v", "pdm_len", "P", "cycles", "exits", "rejects", "err", "done",
                "max_commit", "flags", "last_exited", "last_exit_pos", "last_accept", "target_top1",
                "pdm_top1", "pdm_top2", "draft", "pushed", "err_where", "pad0", "pad1", "pad2"]
ERRORS = {-1: "SPD_EINVAL", -2: "SPD_ENOMEM", -3: "SPD_ECUDA", -4: "SPD_ESTATE", -5: "SPD_ETIMEOUT"}


class SpdError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class spd_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("d_ffn", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("n_stages", ctypes.c_int32), ("pdm_layers", ctypes.c_int32),
                ("n_anchors", ctypes.c_int32), ("anchors", ctypes.c_int32 * MAX_ANCHORS),
                ("rope_theta", ctypes.c_float), ("norm_eps", ctypes.c_float),
                ("dtype", ctypes.c_int32), ("max_seq", ctypes.c_int32)]


class spd_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")]


class spd_weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("layers", ctypes.POINTER(spd_layer_weights)),
                ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("pdm_fc", ctypes.POINTER(ctypes.c_void_p)),
                ("pdm_layers", ctypes.POINTER(spd_layer_weights)),
                ("pdm_norm", ctypes.c_void_p), ("pdm_lm_head", ctypes.c_void_p)]


class spd_cycle_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("t", "a", "v", "exited", "exit_pos", "accepted", "target_top1", "pdm_top1",
                 "pdm_top2", "draft_token", "pushed_token")]


class spd_stats(ctypes.Structure):
    _fields_ = [("cycles", ctypes.c_int64), ("exits", ctypes.c_int64), ("rejects", ctypes.c_int64),
                ("committed", ctypes.c_int64), ("device_ms", ctypes.c_double),
                ("kernel_launches", ctypes.c_int64)]


_LIB = None
_I32P = ctypes.POINTER(ctypes.c_int32)


def library_path() -> str:
    return build_ext.LIBPATH


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built (no fallback exists)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = build_ext.LIBPATH
    if not os.path.exists(path):
        raise SpdError(-3, f"SPD CUDA library missing at {path}; build it with "
                           "speculative_pipeline_decoding_gb300.build_ext.build()")
    L = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    sig = {
        "spd_create": (ctypes.c_int, [ctypes.POINTER(spd_config), ctypes.POINTER(spd_weights), vp,
                                      ctypes.POINTER(vp)]),
        "spd_destroy": (None, [vp]),
        "spd_last_error": (ctypes.c_char_p, [vp]),
        "spd_prefill": (ctypes.c_int, [vp, _I32P, i32, _I32P]),
        "spd_cycle": (ctypes.c_int, [vp, ctypes.POINTER(spd_cycle_info)]),
        "spd_generate": (ctypes.c_int, [vp, i32, vp, _I32P, ctypes.POINTER(spd_stats)]),
        "spd_generate_ar": (ctypes.c_int, [vp, i32, vp, _I32P, ctypes.POINTER(spd_stats)]),
        "spd_rollback": (ctypes.c_int, [vp, i32, i32]),
        "spd_set_draft_override": (ctypes.c_int, [vp, i32, i32, _I32P, ctypes.POINTER(ctypes.c_uint8)]),
        "spd_set_acceptance": (ctypes.c_int, [vp, ctypes.c_double, ctypes.c_uint64, _I32P, i32]),
        "spd_acceptance_modes": (ctypes.c_int, [ctypes.c_double, ctypes.c_uint64, i32, i32,
                                                ctypes.POINTER(ctypes.c_uint8)]),
        "spd_debug_wait_timeout": (ctypes.c_int, [vp, i32, ctypes.c_int64]),
        "spd_set_options": (ctypes.c_int, [vp, i32]),
        "spd_set_sampling": (ctypes.c_int, [vp, ctypes.c_float, i32, i32, i32, ctypes.POINTER(ctypes.c_float)]),
        "spd_dump_size": (sz, [vp, i32]),
        "spd_debug_dump": (ctypes.c_int, [vp, i32, vp, sz]),
        "spd_time_kernels": (ctypes.c_int, [vp, i32]),
        "spd_kernel_times": (ctypes.c_int, [vp, ctypes.POINTER(ctypes.c_int64),
                                            ctypes.POINTER(ctypes.c_double), i32]),
        "spd_cycle_bytes": (ctypes.c_int, [vp, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_double), i32]),
        "spd_attention_workspace_bytes": (sz, [i32, i32, i32, i32, i32]),
        "spd_attention": (ctypes.c_int, [vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, vp, vp, sz, vp]),
        "spd_grouped_gemv": (ctypes.c_int, [ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                                            i32, i32, i32, i32, vp, ctypes.c_float, vp]),
        "spd_attention_static_scratch": (ctypes.c_int, [vp, vp, vp, i32, vp, i32, i32, i32, i32, i32,
                                                        vp, vp]),
        "spd_prefill_attention_workspace_bytes": (sz, [i32, i32, i32, i32]),
        "spd_prefill_attention": (ctypes.c_int, [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = L
    return L


def exported_symbols() -> Sequence[str]:
    """Names of the ABI entry points declared in include/spd.h."""
    import re
    with open(os.path.join(build_ext.INCLUDE, "spd.h")) as fh:
        text = fh.read()
    return sorted(set(re.findall(r"^\s*(?:int|void|size_t|const char\*)\s+(spd_\w+)\s*\(", text, re.M)))


def _check(rc: int, h=None) -> None:
    if rc != 0:
        msg = lib().spd_last_error(h)
        raise SpdError(rc, msg.decode() if msg else "")


def _ptr(t: torch.Tensor) -> int:
    if not t.is_cuda:
        raise SpdError(-1, "tensor must live on the GPU")
    return t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        return None
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass(frozen=True)
class Config:
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_ffn: int
    vocab: int
    n_stages: int
    pdm_layers: int
    anchors: Tuple[int, ...]
    dtype: str = "bf16"
    max_seq: int = 4096
    rope_theta: float = 10000.0
    norm_eps: float = 1e-6

    @classmethod
    def from_workload(cls, w, max_seq: Optional[int] = None) -> "Config":
        m = w.model
        return cls(m.n_layers, m.d_model, m.n_heads, m.n_kv_heads, m.head_dim, m.d_ffn, m.vocab,
                   w.n_stages, w.pdm_layers, tuple(w.anchors), m.dtype,
                   max_seq if max_seq is not None else w.max_seq, m.rope_theta, m.norm_eps)

    def to_c(self) -> spd_config:
        c = spd_config()
        for f in ("n_layers", "d_model", "n_heads", "n_kv_heads", "head_dim", "d_ffn", "vocab",
                  "n_stages", "pdm_layers", "max_seq"):
            setattr(c, f, getattr(self, f))
        c.n_anchors = len(self.anchors)
        for i, b in enumerate(self.anchors):
            c.anchors[i] = b
        c.rope_theta = self.rope_theta
        c.norm_eps = self.norm_eps
        c.dtype = {"f32": DTYPE_F32, "bf16": DTYPE_BF16}[self.dtype]
        return c


_LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


class Engine:
    """One SPD handle: the caller's device weights plus the library-owned caches and graphs."""

    def __init__(self, cfg: Config, weights: Dict[str, torch.Tensor], stream=None):
        L = lib()
        self.cfg = cfg
        self._weights = weights  # borrowed by the library: keep them alive
        need = ["embed", "final_norm", "lm_head", "pdm.norm", "pdm.lm_head"]
        for k in need:
            if k not in weights:
                raise SpdError(-1, f"missing weight {k}")
        tl = (spd_layer_weights * cfg.n_layers)()
        for l in range(cfg.n_layers):
            for k in _LAYER_KEYS:
                setattr(tl[l], k, _ptr(weights[f"layers.{l}.{k}"]))
        pl = (spd_layer_weights * cfg.pdm_layers)()
        for l in range(cfg.pdm_layers):
            for k in _LAYER_KEYS:
                setattr(pl[l], k, _ptr(weights[f"pdm.layers.{l}.{k}"]))
        fc = (ctypes.c_void_p * len(cfg.anchors))()
        for j in range(len(cfg.anchors)):
            t = weights.get(f"pdm.fc.{j}")
            fc[j] = _ptr(t) if t is not None else None
        w = spd_weights()
        w.embed = _ptr(weights["embed"])
        w.layers = tl
        w.final_norm = _ptr(weights["final_norm"])
        w.lm_head = _ptr(weights["lm_head"])
        w.pdm_fc = fc
        w.pdm_layers = pl
        w.pdm_norm = _ptr(weights["pdm.norm"])
        w.pdm_lm_head = _ptr(weights["pdm.lm_head"])
        self._keep = (tl, pl, fc, w)
        c = cfg.to_c()
        h = ctypes.c_void_p()
        rc = L.spd_create(ctypes.byref(c), ctypes.byref(w), _stream_handle(stream), ctypes.byref(h))
        _check(rc, None)
        self.h = h
        self.P = 0
        self.opts = OPT_DEFAULT

    # -- lifecycle ------------------------------------------------------------
    def close(self) -> None:
        if getattr(self, "h", None):
            lib().spd_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    # -- decoding ---------------------------------------------------------------
    def prefill(self, tokens) -> int:
        arr = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        first = ctypes.c_int32()
        _check(lib().spd_prefill(self.h, arr.ctypes.data_as(_I32P), int(arr.size), ctypes.byref(first)),
               self.h)
        self.P = int(arr.size)
        return int(first.value)

    def cycle(self, info: bool = True) -> Optional[Dict[str, int]]:
        ci = spd_cycle_info()
        _check(lib().spd_cycle(self.h, ctypes.byref(ci) if info else None), self.h)
        if not info:
            return None
        return {f: int(getattr(ci, f)) for f, _ in spd_cycle_info._fields_}

    def _gen(self, fn, max_new: int, out) -> Tuple[Optional[np.ndarray], Dict[str, float]]:
        st = spd_stats()
        n_out = ctypes.c_int32()
        host = None
        if out is None:
            host = np.empty(max_new, dtype=np.int32)
            ptr = host.ctypes.data
        elif isinstance(out, torch.Tensor):
            if out.dtype != torch.int32 or out.numel() < max_new:
                raise SpdError(-1, "out must be an int32 tensor of >= max_new elements")
            ptr = out.data_ptr()
        else:
            ptr = None
        _check(fn(self.h, int(max_new), ptr, ctypes.byref(n_out), ctypes.byref(st)), self.h)
        stats = {f: getattr(st, f) for f, _ in spd_stats._fields_}
        return host, stats

    def generate(self, max_new: int, out=None):
        """SPD cycles until max_new tokens are committed; returns (tokens or None, stats)."""
        return self._gen(lib().spd_generate, max_new, out)

    def generate_ar(self, max_new: int, out=None):
        return self._gen(lib().spd_generate_ar, max_new, out)

    def rollback(self, keep_len: int, reseed: int) -> None:
        _check(lib().spd_rollback(self.h, int(keep_len), int(reseed)), self.h)

    def set_draft_override(self, first_pos: int, ref_tokens, modes) -> None:
        ref = np.ascontiguousarray(np.asarray(ref_tokens, dtype=np.int32))
        md = np.ascontiguousarray(np.asarray(modes, dtype=np.uint8))
        if ref.size != md.size:
            raise SpdError(-1, "ref_tokens and modes differ in length")
        _check(lib().spd_set_draft_override(self.h, int(first_pos), int(ref.size),
                                            ref.ctypes.data_as(_I32P),
                                            md.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))), self.h)

    def set_acceptance(self, alpha: float, seed: int, ref_tokens) -> None:
        """Seeded acceptance from (alpha, seed): ref_tokens are the reference tokens at positions
        P+1.. (the plain AR stream); alpha < 0 switches the knob off."""
        ref = np.ascontiguousarray(np.asarray(ref_tokens, dtype=np.int32))
        _check(lib().spd_set_acceptance(self.h, float(alpha), int(seed) & ((1 << 64) - 1),
                                        ref.ctypes.data_as(_I32P), int(ref.size)), self.h)

    def debug_wait_timeout(self, which: int, limit_ns: int) -> int:
        """Run one bounded device wait on a condition nothing satisfies; returns the status code
        (SPD_ETIMEOUT = -5 when the wait gave up, as it must) without raising."""
        return int(lib().spd_debug_wait_timeout(self.h, int(which), int(limit_ns)))

    def set_options(self, flags: int) -> None:
        _check(lib().spd_set_options(self.h, int(flags)), self.h)
        self.opts = int(flags)

    def set_sampling(self, temperature: float, top_k: int = 50, first_pos: int = 1, uniforms=None) -> None:
        """Sampled decoding (temperature > 0) or greedy (<= 0).  ``uniforms``: [4][count] floats in
        [0, 1) for positions first_pos.. (streams draft, accept, resample, ar)."""
        u = np.zeros((4, 0), np.float32) if uniforms is None else np.asarray(uniforms, dtype=np.float32)
        if u.ndim != 2 or u.shape[0] != 4:
            raise SpdError(-1, "uniforms must be [4][count]")
        u = np.ascontiguousarray(u)
        _check(lib().spd_set_sampling(self.h, float(temperature), int(top_k), int(first_pos), int(u.shape[1]),
                                      u.ctypes.data_as(ctypes.POINTER(ctypes.c_float))), self.h)

    # -- inspection -------------------------------------------------------------
    def dump(self, what: int) -> np.ndarray:
        n = lib().spd_dump_size(self.h, what)
        dt = np.int32 if what in (DUMP_STATE, DUMP_SEQ, DUMP_TRACE, DUMP_KVLEN) else np.float32
        buf = np.empty(n // 4, dtype=dt)
        _check(lib().spd_debug_dump(self.h, what, buf.ctypes.data, n), self.h)
        c = self.cfg
        if what == DUMP_RESID:
            return buf.reshape(c.n_stages + 1, c.d_model)
        if what == DUMP_ANCHORS:
            return buf.reshape(c.n_stages + 1, len(c.anchors), c.d_model)
        if what == DUMP_PDM_Z:
            return buf.reshape(c.n_stages + 2, c.d_model)
        if what == DUMP_LOGITS:
            return buf.reshape(2, c.vocab)
        if what == DUMP_TRACE:
            return buf.reshape(2, c.max_seq)
        if what == DUMP_PREFILL_H:
            return buf.reshape(-1, c.d_model)
        return buf

    def state(self) -> Dict[str, int]:
        s = self.dump(DUMP_STATE)
        return {k: int(v) for k, v in zip(STATE_FIELDS, s)}

    def time_kernels(self, enable: bool) -> None:
        _check(lib().spd_time_kernels(self.h, int(bool(enable))), self.h)

    def kernel_times(self) -> Dict[str, Tuple[int, float]]:
        n = len(KIND_NAMES)
        la = (ctypes.c_int64 * n)()
        ms = (ctypes.c_double * n)()
        _check(lib().spd_kernel_times(self.h, la, ms, n), self.h)
        return {KIND_NAMES[k]: (int(la[k]), float(ms[k])) for k in range(n)}

    def cycle_bytes(self, t: int, fill: int, exited: bool, with_pdm: bool) -> Dict[str, float]:
        n = len(KIND_NAMES)
        out = (ctypes.c_double * n)()
        _check(lib().spd_cycle_bytes(self.h, int(t), int(fill), int(bool(exited)), int(bool(with_pdm)),
                                     out, n), self.h)
        return {KIND_NAMES[k]: float(out[k]) for k in range(n)}


def acceptance_modes(alpha: float, seed: int, first_pos: int, count: int) -> np.ndarray:
    """The harness modes spd_set_acceptance derives (1 = reference token, 2 = another token), computed
    by the library on the host for positions first_pos .. first_pos+count-1."""
    out = np.zeros(max(0, int(count)), dtype=np.uint8)
    _check(lib().spd_acceptance_modes(float(alpha), int(seed) & ((1 << 64) - 1), int(first_pos), int(count),
                                      out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))))
    return out


# ---------------------------------------------------------------------------
# stand-alone operators
# ---------------------------------------------------------------------------
def attention_workspace_bytes(R: int, n_heads: int, n_kv_heads: int, head_dim: int, max_pos: int) -> int:
    return int(lib().spd_attention_workspace_bytes(R, n_heads, n_kv_heads, head_dim, max_pos))


def attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, pos: torch.Tensor,
              out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """out[r,h] = softmax(q[r,h] K[kv(h), :pos[r]]^T / sqrt(hd)) V.  Shapes: q,out [R,Hq,hd] fp32,
    caches [Hkv, max_seq, hd] (bf16/fp32), pos int32 [R] on the device."""
    R, hq, hd = q.shape
    hkv, max_seq, _ = k_cache.shape
    dt = DTYPE_BF16 if k_cache.dtype == torch.bfloat16 else DTYPE_F32
    _check(lib().spd_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), dt, _ptr(pos), R, hq, hkv, hd,
                               max_seq, _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream_handle(stream)))


def grouped_gemv(Ws: Sequence[torch.Tensor], xs: Sequence[torch.Tensor], ys: Sequence[torch.Tensor],
                 norm_weight: Optional[torch.Tensor] = None, eps: float = 1e-6, stream=None) -> None:
    """ys[g] = Ws[g] @ (rmsnorm(xs[g]) * norm_weight if norm_weight is given else xs[g])."""
    G = len(Ws)
    rows, cols = Ws[0].shape
    dt = DTYPE_BF16 if Ws[0].dtype == torch.bfloat16 else DTYPE_F32
    arr = lambda ts: (ctypes.c_void_p * G)(*[_ptr(t) for t in ts])
    _check(lib().spd_grouped_gemv(arr(Ws), arr(xs), arr(ys), G, rows, cols, dt,
                                  _ptr(norm_weight) if norm_weight is not None else None, eps,
                                  _stream_handle(stream)))


def attention_static_scratch(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                             pos: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """Same as :func:`attention`, for callers that cannot allocate device memory: the split
    partials live in the library's fixed 16 MiB per-GPU scratch array instead of a workspace.
    Calls that overlap on the GPU race on that array; sizes beyond it raise SpdError."""
    R, hq, hd = q.shape
    hkv, max_seq, _ = k_cache.shape
    dt = DTYPE_BF16 if k_cache.dtype == torch.bfloat16 else DTYPE_F32
    _check(lib().spd_attention_static_scratch(_ptr(q), _ptr(k_cache), _ptr(v_cache), dt, _ptr(pos), R,
                                              hq, hkv, hd, max_seq, _ptr(out), _stream_handle(stream)))


def prefill_attention_workspace_bytes(n_heads: int, n_kv_heads: int, head_dim: int, max_seq: int) -> int:
    return int(lib().spd_prefill_attention_workspace_bytes(n_heads, n_kv_heads, head_dim, max_seq))


def prefill_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, pos0: int,
                      out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """Causal attention of R = q.shape[0] rows at positions pos0..pos0+R-1 on the tensor cores.
    Shapes: q, out [R, Hq, hd] fp32; caches [Hkv, max_seq, hd] bf16."""
    R, hq, hd = q.shape
    hkv, max_seq, _ = k_cache.shape
    _check(lib().spd_prefill_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), int(pos0), R, hq, hkv, hd, max_seq,
                                       _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream_handle(stream)))
