"""Python binding of libmi_block.so (include/mi_block.h): argument marshalling only.

Every step of the block runs in the library's CUDA kernels; this module checks tensor
dtypes/devices, turns torch tensors into device pointers and the current torch stream into a
cudaStream_t, and raises MiError with the library's message when a call fails.  There is no
fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

__all__ = [
    "MiError", "lib", "library_path", "Block", "Model", "SeqLayout", "mod_rmsnorm", "gemm",
    "gemm_gated_residual", "gemm_silu_gate", "gemm_qkv_rope", "qk_norm_rope", "attention", "attention_workspace_size",
    "gated_add", "silu_gate",
    "device_error", "device_supported", "TENSORS", "TimestepModulation", "rope_tables", "time_advance",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

TENSORS = {"h": 0, "qkv": 1, "qp": 2, "kp": 3, "o": 4, "a": 5, "x1": 6, "h2": 7, "gu": 8, "m": 9, "dn": 10}


class MiError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"mi_block status {status}: {msg}")
        self.status = status


def library_path() -> str:
    return os.path.join(_HERE, "libmi_block.so")


class _BlockDesc(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int), ("n_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("mlp_inter", ctypes.c_int), ("eps", ctypes.c_float), ("fuse_epilogues", ctypes.c_int),
        ("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p), ("w_gu", ctypes.c_void_p),
        ("w_d", ctypes.c_void_p), ("q_norm_w", ctypes.c_void_p), ("k_norm_w", ctypes.c_void_p),
    ]


class SeqLayout(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("text_pad", ctypes.c_int), ("grid_h", ctypes.c_int),
                ("grid_w", ctypes.c_int)]

    @property
    def seq(self) -> int:
        return self.text_pad + self.grid_h * self.grid_w


class _TmodDesc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_blocks", ctypes.c_int), ("w_t1", ctypes.c_void_p),
                ("w_t2", ctypes.c_void_p), ("w_mod", ctypes.c_void_p)]


class _ModelDesc(ctypes.Structure):
    _fields_ = [("n_blocks", ctypes.c_int), ("blocks", ctypes.POINTER(_BlockDesc)),
                ("latent_ch", ctypes.c_int), ("w_in", ctypes.c_void_p), ("w_out", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "mi_last_error": ([], ctypes.c_char_p),
    "mi_abi_version": ([], _I),
    "mi_device_supported": ([], _I),
    "mi_device_error": ([ctypes.POINTER(_I)], _I),
    "mi_selftest_wait_timeout": ([_I, _P], _I),
    "mi_block_init": ([ctypes.POINTER(_P), ctypes.POINTER(_BlockDesc)], _I),
    "mi_block_destroy": ([_P], None),
    "mi_block_workspace_size": ([_P, _I, _I, ctypes.POINTER(_SZ)], _I),
    "mi_block_tensor_offset": ([_P, _I, _I, _I, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)], _I),
    "mi_block_forward": ([_P, ctypes.POINTER(SeqLayout), _P, _P, _P, _P, _P, _I, _P, _P, _SZ, _P], _I),
    "mi_block_forward_static_ws": ([_P, ctypes.POINTER(SeqLayout), _P, _P, _P, _P, _P, _I, _P, _P], _I),
    "mi_model_init": ([ctypes.POINTER(_P), ctypes.POINTER(_ModelDesc)], _I),
    "mi_model_destroy": ([_P], None),
    "mi_model_workspace_size": ([_P, ctypes.POINTER(SeqLayout), ctypes.POINTER(_SZ)], _I),
    "mi_model_plan": ([_P, ctypes.POINTER(SeqLayout), _I, _SZ, ctypes.POINTER(_SZ), ctypes.POINTER(ctypes.c_uint8)], _I),
    "mi_denoise_step": ([_P, ctypes.POINTER(SeqLayout), _P, _P, _P, _P, _P, _P, _I, _P, _F, _F, _P, _P, _SZ,
                         _P], _I),
    "mi_rope_tables": ([_I, _I, _I, _F, _P, _P, _P], _I),
    "mi_tmod_init": ([ctypes.POINTER(_P), ctypes.POINTER(_TmodDesc)], _I),
    "mi_tmod_destroy": ([_P], None),
    "mi_tmod_workspace_size": ([_P, _I, ctypes.POINTER(_SZ)], _I),
    "mi_timestep_modulation": ([_P, _P, _I, _P, _P, _P, _SZ, _P], _I),
    "mi_time_advance": ([_P, _I, _F, _P], _I),
    "mi_mod_rmsnorm": ([_P, _P, _I, _I, _P, _I, _I, _I, _F, _P], _I),
    "mi_gemm_bf16": ([_P, _P, _P, _I, _I, _I, _P], _I),
    "mi_gemm_bf16_gated_residual": ([_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _P], _I),
    "mi_gemm_bf16_silu_gate": ([_P, _P, _P, _I, _I, _I, _P], _I),
    "mi_gemm_bf16_qkv_rope": ([_P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _F, _P], _I),
    "mi_qk_norm_rope": ([_P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _F, _P], _I),
    "mi_attention": ([_P, _P, _P, _P, _P, _I, _I, _I, _P], _I),
    "mi_attention_workspace_size": ([_I, _I, _I, ctypes.POINTER(_SZ)], _I),
    "mi_attention_ws": ([_P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P], _I),
    "mi_gated_add": ([_P, _P, _P, _I, _P, _I, _I, _I, _P], _I),
    "mi_silu_gate": ([_P, _P, _I, _I, _P], _I),
}


def lib():
    """Load libmi_block.so (built by __graft_entry__.build()); raises if it is missing."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built: run __graft_entry__.build() first")
        L = ctypes.CDLL(path)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = L
    return _LIB


def _check(status: int):
    if status != 0:
        msg = lib().mi_last_error()
        raise MiError(status, msg.decode() if msg else "")


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor], dtype=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on the GPU")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


_BF = torch.bfloat16


def device_supported() -> bool:
    return lib().mi_device_supported() == 0


def device_error() -> int:
    """Read and clear the device error flag (synchronises the device)."""
    code = _I(0)
    _check(lib().mi_device_error(ctypes.byref(code)))
    return code.value


def selftest_wait_timeout(limit_us: int = 10000, stream=None):
    """Enqueue the bounded-wait self-test kernel (its wait runs out after limit_us)."""
    _check(lib().mi_selftest_wait_timeout(limit_us, _stream(stream)))


class Block:
    """One DiT block: weights stay owned by the caller's tensors (kept alive here)."""

    def __init__(self, w_qkv, w_o, w_gu, w_d, q_norm_w, k_norm_w, n_heads: int, eps: float = 1e-6,
                 fuse_epilogues: bool = True):
        H = w_o.shape[0]
        self._keep = (w_qkv, w_o, w_gu, w_d, q_norm_w, k_norm_w)
        self.hidden, self.n_heads, self.inter = H, n_heads, w_d.shape[1]
        self.desc = _BlockDesc(H, n_heads, 128, w_d.shape[1], eps, 1 if fuse_epilogues else 0,
                               _ptr(w_qkv, _BF), _ptr(w_o, _BF), _ptr(w_gu, _BF), _ptr(w_d, _BF),
                               _ptr(q_norm_w, _BF), _ptr(k_norm_w, _BF))
        h = _P()
        _check(lib().mi_block_init(ctypes.byref(h), ctypes.byref(self.desc)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            lib().mi_block_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace_size(self, batch: int, seq: int) -> int:
        n = _SZ(0)
        _check(lib().mi_block_workspace_size(self.handle, batch, seq, ctypes.byref(n)))
        return n.value

    def tensor_offset(self, batch: int, seq: int, name: str):
        off, nb = _SZ(0), _SZ(0)
        _check(lib().mi_block_tensor_offset(self.handle, batch, seq, TENSORS[name], ctypes.byref(off),
                                            ctypes.byref(nb)))
        return off.value, nb.value

    def forward(self, layout: SeqLayout, x, y, mod, rope_cos, rope_sin, key_mask, ws, rope_bstride: int = 0,
                stream=None):
        _check(lib().mi_block_forward(self.handle, ctypes.byref(layout), _ptr(x, _BF), _ptr(y, _BF),
                                      _ptr(mod, _BF), _ptr(rope_cos, torch.float32),
                                      _ptr(rope_sin, torch.float32), rope_bstride, _ptr(key_mask, torch.uint8),
                                      _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


class Model:
    """A stack of blocks plus the latent embedding and velocity projections."""

    def __init__(self, blocks: Sequence[dict], w_in, w_out, n_heads: int, eps: float = 1e-6,
                 fuse_epilogues: bool = True):
        n = len(blocks)
        arr = (_BlockDesc * n)()
        keep = []
        for i, b in enumerate(blocks):
            keep.append(b)
            arr[i] = _BlockDesc(b["w_o"].shape[0], n_heads, 128, b["w_d"].shape[1], eps,
                                1 if fuse_epilogues else 0, _ptr(b["w_qkv"], _BF), _ptr(b["w_o"], _BF),
                                _ptr(b["w_gu"], _BF), _ptr(b["w_d"], _BF), _ptr(b["q_norm_w"], _BF),
                                _ptr(b["k_norm_w"], _BF))
        self._keep = (keep, w_in, w_out, arr)
        self.latent_ch = w_in.shape[1]
        desc = _ModelDesc(n, arr, w_in.shape[1], _ptr(w_in, _BF), _ptr(w_out, _BF))
        h = _P()
        _check(lib().mi_model_init(ctypes.byref(h), ctypes.byref(desc)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            lib().mi_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace_size(self, layout: SeqLayout) -> int:
        n = _SZ(0)
        _check(lib().mi_model_workspace_size(self.handle, ctypes.byref(layout), ctypes.byref(n)))
        return n.value

    def plan(self, layouts: Sequence[SeqLayout], budget_bytes: int):
        """One workspace for several layouts: (bytes, served flags); MiError(status 3) when none fits."""
        n = len(layouts)
        arr = (SeqLayout * n)(*layouts)
        flags = (ctypes.c_uint8 * n)()
        nb = _SZ(0)
        _check(lib().mi_model_plan(self.handle, arr, n, budget_bytes, ctypes.byref(nb), flags))
        return nb.value, [bool(f) for f in flags]

    def denoise_step(self, layout: SeqLayout, latent, text_rows, mods, mod_final, rope_cos, rope_sin, key_mask,
                     dt: float, guidance: float, ws, skip_neg=None, rope_bstride: int = 0, stream=None):
        """skip_neg: optional host sequence of n_blocks flags (the negative element bypasses a flagged block)."""
        sk = None
        if skip_neg is not None:
            flags = [1 if bool(v) else 0 for v in (skip_neg.tolist() if hasattr(skip_neg, "tolist") else skip_neg)]
            sk = (ctypes.c_uint8 * len(flags))(*flags)
        _check(lib().mi_denoise_step(self.handle, ctypes.byref(layout), _ptr(latent, torch.float32),
                                     _ptr(text_rows, _BF),
                                     _ptr(mods, _BF), _ptr(mod_final, _BF), _ptr(rope_cos, torch.float32),
                                     _ptr(rope_sin, torch.float32), rope_bstride, _ptr(key_mask, torch.uint8),
                                     dt, guidance, ctypes.cast(sk, _P) if sk is not None else None, _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream(stream)))


class TimestepModulation:
    """Timestep -> per-block modulation on the device (weights owned by the caller's tensors)."""

    def __init__(self, w_t1, w_t2, w_mod, n_blocks: int):
        self._keep = (w_t1, w_t2, w_mod)
        self.hidden, self.n_blocks = w_t2.shape[0], n_blocks
        self.desc = _TmodDesc(w_t2.shape[0], n_blocks, _ptr(w_t1, _BF), _ptr(w_t2, _BF), _ptr(w_mod, _BF))
        h = _P()
        _check(lib().mi_tmod_init(ctypes.byref(h), ctypes.byref(self.desc)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            lib().mi_tmod_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace_size(self, batch: int) -> int:
        n = _SZ(0)
        _check(lib().mi_tmod_workspace_size(self.handle, batch, ctypes.byref(n)))
        return n.value

    def __call__(self, t, mods, mod_final, ws, stream=None):
        _check(lib().mi_timestep_modulation(self.handle, _ptr(t, torch.float32), t.numel(), _ptr(mods, _BF),
                                            _ptr(mod_final, _BF), _ptr(ws), ws.numel() * ws.element_size(),
                                            _stream(stream)))


def rope_tables(text_pad, grid_h, grid_w, rope_cos, rope_sin, theta=10000.0, stream=None):
    _check(lib().mi_rope_tables(text_pad, grid_h, grid_w, theta, _ptr(rope_cos, torch.float32),
                                _ptr(rope_sin, torch.float32), _stream(stream)))


def time_advance(t, dt, stream=None):
    _check(lib().mi_time_advance(_ptr(t, torch.float32), t.numel(), dt, _stream(stream)))


# ------------------------------------------------------------------------------- single kernels
def mod_rmsnorm(x, mod, shift_row, scale_row, out, batch, seq, eps=1e-6, stream=None):
    _check(lib().mi_mod_rmsnorm(_ptr(x, _BF), _ptr(mod, _BF), shift_row, scale_row, _ptr(out, _BF), batch, seq,
                                x.shape[-1], eps, _stream(stream)))


def gemm(a, w, c, stream=None):
    m, k = a.shape
    n = w.shape[0]
    _check(lib().mi_gemm_bf16(_ptr(a, _BF), _ptr(w, _BF), _ptr(c, _BF), m, n, k, _stream(stream)))


def gemm_gated_residual(a, w, resid, mod, gate_row, out, seq, stream=None):
    m, k = a.shape
    n = w.shape[0]
    _check(lib().mi_gemm_bf16_gated_residual(_ptr(a, _BF), _ptr(w, _BF), _ptr(resid, _BF), _ptr(mod, _BF),
                                             gate_row, _ptr(out, _BF), m, n, k, seq, _stream(stream)))


def gemm_silu_gate(a, w, m_out, stream=None):
    m, k = a.shape
    inter = w.shape[0] // 2
    _check(lib().mi_gemm_bf16_silu_gate(_ptr(a, _BF), _ptr(w, _BF), _ptr(m_out, _BF), m, inter, k,
                                        _stream(stream)))


def gemm_qkv_rope(a, w_qkv, q_norm_w, k_norm_w, rope_cos, rope_sin, qp, kp, qkv_v, batch, seq, n_heads, eps=1e-6,
                  rope_bstride=0, stream=None):
    _check(lib().mi_gemm_bf16_qkv_rope(_ptr(a, _BF), _ptr(w_qkv, _BF), _ptr(q_norm_w, _BF), _ptr(k_norm_w, _BF),
                                       _ptr(rope_cos, torch.float32), _ptr(rope_sin, torch.float32), rope_bstride,
                                       _ptr(qp, _BF), _ptr(kp, _BF), _ptr(qkv_v, _BF), batch, seq, n_heads, eps,
                                       _stream(stream)))


def qk_norm_rope(qkv, q_norm_w, k_norm_w, rope_cos, rope_sin, qp, kp, batch, seq, n_heads, eps=1e-6,
                 rope_bstride=0, stream=None):
    _check(lib().mi_qk_norm_rope(_ptr(qkv, _BF), _ptr(q_norm_w, _BF), _ptr(k_norm_w, _BF),
                                 _ptr(rope_cos, torch.float32), _ptr(rope_sin, torch.float32), rope_bstride,
                                 _ptr(qp, _BF), _ptr(kp, _BF), batch, seq, n_heads, eps, _stream(stream)))


def attention_workspace_size(batch, seq, n_heads) -> int:
    n = ctypes.c_size_t()
    _check(lib().mi_attention_workspace_size(batch, seq, n_heads, ctypes.byref(n)))
    return n.value


def attention(qp, kp, qkv, key_mask, o, batch, seq, n_heads, stream=None, ws=None):
    """Attention; with `ws` (a uint8 tensor of attention_workspace_size bytes) on the split
    one-CTA-per-SM schedule the block forward uses, without it one CTA per query-tile pair."""
    if ws is None:
        _check(lib().mi_attention(_ptr(qp, _BF), _ptr(kp, _BF), _ptr(qkv, _BF), _ptr(key_mask, torch.uint8),
                                  _ptr(o, _BF), batch, seq, n_heads, _stream(stream)))
    else:
        _check(lib().mi_attention_ws(_ptr(qp, _BF), _ptr(kp, _BF), _ptr(qkv, _BF), _ptr(key_mask, torch.uint8),
                                     _ptr(o, _BF), batch, seq, n_heads, _ptr(ws, torch.uint8) if ws.numel() else None,
                                     ws.numel(), _stream(stream)))


def gated_add(x, y, mod, gate_row, out, batch, seq, stream=None):
    _check(lib().mi_gated_add(_ptr(x, _BF), _ptr(y, _BF), _ptr(mod, _BF), gate_row, _ptr(out, _BF), batch, seq,
                              x.shape[-1], _stream(stream)))


def silu_gate(gu, m, stream=None):
    rows = gu.shape[0]
    inter = gu.shape[1] // 2
    _check(lib().mi_silu_gate(_ptr(gu, _BF), _ptr(m, _BF), rows, inter, _stream(stream)))
