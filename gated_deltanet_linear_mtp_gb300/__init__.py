"""Gated DeltaNet (GDN) decode / MTP-verify / commit on one GB300 -- Python binding of ``libgdn.so``.

Argument marshalling only: every step of the computation runs in the library's CUDA kernels
(``csrc/``); PyTorch supplies device memory and the current stream.  There is no CPU fallback: if the
library has not been built, every call raises.

    gdn_decode(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, err_word=None, scale=1.0, l2_eps=1e-6)
    gdn_decode_gated(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, norm, err_word=None, ...)
    gdn_mtp_verify(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, intermediate_states=None, ...)
    gdn_commit(state_pool, state_indices, intermediate_states, accept_len, err_word=None)
    gdn_commit_replay(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, accept_len, err_word=None, ...)
    gdn_mtp_verify_commit(prev, q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, err_word=None,
                          norm=None, ...)
    gdn_mtp_verify_gated(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, norm,
                         intermediate_states=None, err_word=None, ...)
    gdn_prefill(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, cu_seqlens, o,
                has_initial_state=None, err_word=None, ...)
    gdn_gated_rmsnorm(o, z, norm_weight, y=None, eps=1e-6)
    gdn_in_proj_conv(x, W, conv_w, conv_b, conv_state, state_indices, out, write_state, records=None,
                     err_word=None, silu=True)
    gdn_conv_commit(conv_state, state_indices, records, accept_len, err_word=None)

Shapes and semantics are those of ``include/gdn.h``: q, k ``[B,T,HK,DK]``; v, o ``[B,T,HV,DV]``; a, b
``[B,T,HV]``; A_log, dt_bias ``[HV]`` fp32; state_pool ``[num_slots,HV,DV,DK]``; state_indices, accept_len
``[B]`` int32; intermediate_states ``[B,T,HV,DV,DK]``; err_word a 1-element int32 device tensor.  Prefill takes
packed tokens: q, k ``[N,HK,DK]``; v, o ``[N,HV,DV]``; a, b ``[N,HV]``; cu_seqlens ``[B+1]`` and
has_initial_state ``[B]`` int32.  The in_proj projection takes x ``[B,T,H]`` bf16, W ``[C,H]`` bf16, conv_w
``[Cc,K]`` / conv_b ``[Cc]`` fp32, conv_state ``[num_slots,K-1,Cc]`` and records ``[B,T,Cc]``, and writes the q, k,
v, z, b, a of an ``InProjOut`` (their shapes give HK, DK, HV, DV).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from .build import LIB_PATH

__all__ = ["gdn_decode", "gdn_decode_gated", "gdn_mtp_verify", "gdn_commit", "gdn_commit_replay", "gdn_mtp_verify_commit", "ReplayTokens",
           "gdn_mtp_verify_gated", "GatedNorm",
           "gdn_prefill", "gdn_gated_rmsnorm", "gdn_in_proj_conv", "gdn_conv_commit", "InProjOut", "GdnError", "GdnDims", "lib", "STATUS", "ERRBIT_INDEX", "ERRBIT_ACCEPT_LEN", "ERRBIT_TIMEOUT",
           "ERRBIT_SEQLEN", "MAX_T", "EXPORTS"]

STATUS = {0: "GDN_OK", 1: "GDN_ERR_NULL", 2: "GDN_ERR_SHAPE", 3: "GDN_ERR_DTYPE", 4: "GDN_ERR_ALIGN",
          5: "GDN_ERR_UNSUPPORTED", 6: "GDN_ERR_CUDA", 7: "GDN_ERR_VALUE"}
ERRBIT_INDEX = 1
ERRBIT_ACCEPT_LEN = 2
ERRBIT_TIMEOUT = 4
ERRBIT_SEQLEN = 8
MAX_T = 16
F32, BF16 = 0, 1
EXPORTS = ("gdn_decode", "gdn_decode_gated", "gdn_mtp_verify", "gdn_commit", "gdn_commit_replay",
           "gdn_mtp_verify_commit", "gdn_mtp_verify_gated", "gdn_prefill",
           "gdn_gated_rmsnorm", "gdn_in_proj_conv", "gdn_conv_commit", "gdn_status_string", "gdn_last_cuda_error",
           "gdn_abi_version")


class GdnDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("HK", ctypes.c_int32), ("HV", ctypes.c_int32),
                ("DK", ctypes.c_int32), ("DV", ctypes.c_int32), ("num_slots", ctypes.c_int32),
                ("qkv_dtype", ctypes.c_int32), ("state_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("scale", ctypes.c_float), ("l2_eps", ctypes.c_float)]


class _ReplayTokensC(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("a", ctypes.c_void_p),
                ("b", ctypes.c_void_p), ("accept_len", ctypes.c_void_p)]


class ReplayTokens:
    """The k, v, a, b of an earlier ``gdn_mtp_verify`` on the same lanes (``[B, T', ...]``, T' its token count)
    and ``accept_len`` ``[B]`` int32: the tokens ``gdn_mtp_verify_commit`` commits before it verifies."""

    def __init__(self, k, v, a, b, accept_len):
        self.k, self.v, self.a, self.b, self.accept_len = k, v, a, b, accept_len


class _GatedNormC(ctypes.Structure):
    _fields_ = [("z", ctypes.c_void_p), ("z_dtype", ctypes.c_int32), ("norm_weight", ctypes.c_void_p),
                ("eps", ctypes.c_float), ("y", ctypes.c_void_p)]


class GatedNorm:
    """The gated RMSNorm of a verify's outputs into ``y``: ``z`` (the gate, o's shape, fp32 or bf16),
    ``norm_weight`` ``[DV]`` fp32, ``y`` (o's shape and dtype; may be o itself)."""

    def __init__(self, z, norm_weight, y, eps=1e-6):
        self.z, self.norm_weight, self.y, self.eps = z, norm_weight, y, eps


class _ConvDimsC(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32), ("HK", ctypes.c_int32),
                ("HV", ctypes.c_int32), ("DK", ctypes.c_int32), ("DV", ctypes.c_int32), ("K", ctypes.c_int32),
                ("num_slots", ctypes.c_int32), ("conv_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("silu", ctypes.c_int32)]


class _InProjOutC(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("z", ctypes.c_void_p),
                ("b", ctypes.c_void_p), ("a", ctypes.c_void_p)]


class InProjOut:
    """The outputs of ``gdn_in_proj_conv``: q, k ``[B,T,HK,DK]``, v, z ``[B,T,HV,DV]``, b, a ``[B,T,HV]``, one dtype."""

    def __init__(self, q, k, v, z, b, a):
        self.q, self.k, self.v, self.z, self.b, self.a = q, k, v, z, b, a


class GdnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = _lib_handle.gdn_status_string(status).decode() if _lib_handle is not None else STATUS.get(status)
        if status == 6 and _lib_handle is not None:
            msg += f" (cudaError {_lib_handle.gdn_last_cuda_error()})"
        super().__init__(f"{what}: {msg}")


_lib_handle: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded ``libgdn.so``; raises if it has not been built (no fallback exists)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m gated_deltanet_linear_mtp_gb300.build` (there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        vp, dp, ip = ctypes.c_void_p, ctypes.POINTER(GdnDims), ctypes.c_void_p
        L.gdn_decode.argtypes = [dp] + [vp] * 5 + [vp, vp, vp, ip, vp, ip, vp]
        L.gdn_decode_gated.argtypes = [dp] + [vp] * 5 + [vp, vp, vp, ip, vp, ctypes.POINTER(_GatedNormC), ip, vp]
        L.gdn_mtp_verify.argtypes = [dp] + [vp] * 5 + [vp, vp, vp, ip, vp, vp, ip, vp]
        L.gdn_commit.argtypes = [dp, vp, ip, vp, ip, ip, vp]
        L.gdn_commit_replay.argtypes = [dp] + [vp] * 5 + [vp, vp, vp, ip, ip, ip, vp]
        L.gdn_mtp_verify_commit.argtypes = ([dp, ctypes.POINTER(_ReplayTokensC)] + [vp] * 5 +
                                            [vp, vp, vp, ip, vp, ctypes.POINTER(_GatedNormC), ip, vp])
        L.gdn_mtp_verify_gated.argtypes = [dp] + [vp] * 5 + [vp, vp, vp, ip, vp, vp, ctypes.POINTER(_GatedNormC), ip, vp]
        L.gdn_prefill.argtypes = [dp, ip] + [vp] * 5 + [vp, vp, vp, ip, ip, vp, ip, vp]
        L.gdn_gated_rmsnorm.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vp, vp, vp,
                                        ctypes.c_float, vp, vp]
        cdp = ctypes.POINTER(_ConvDimsC)
        L.gdn_in_proj_conv.argtypes = [cdp, vp, vp, vp, vp, vp, ip, ctypes.c_int32, ctypes.POINTER(_InProjOutC), vp,
                                       ip, vp]
        L.gdn_conv_commit.argtypes = [cdp, vp, ip, vp, ip, ip, vp]
        for f in (L.gdn_in_proj_conv, L.gdn_conv_commit):
            f.restype = ctypes.c_int
        for f in (L.gdn_decode, L.gdn_decode_gated, L.gdn_mtp_verify, L.gdn_commit, L.gdn_commit_replay, L.gdn_mtp_verify_commit,
                  L.gdn_mtp_verify_gated, L.gdn_prefill, L.gdn_gated_rmsnorm):
            f.restype = ctypes.c_int
        L.gdn_status_string.argtypes = [ctypes.c_int]
        L.gdn_status_string.restype = ctypes.c_char_p
        L.gdn_last_cuda_error.restype = ctypes.c_int32
        L.gdn_abi_version.restype = ctypes.c_int32
        _lib_handle = L
    return _lib_handle


# ---- marshalling -------------------------------------------------------------------------------------
def _code(t, name: str) -> int:
    import torch

    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"{name}: dtype {t.dtype} (fp32 or bf16 expected)")


def _dev(t, name: str, dtype=None):
    """Pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _shape(t, want, name: str):
    if tuple(t.shape) != tuple(want):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(want)}")


def _common_device(named):
    """The one CUDA device that every given tensor (``(name, tensor)`` pairs, None skipped) lives on.

    A call launches its kernels on one GPU with raw pointers: a tensor on another GPU would be read through
    peer access or fault, so mixed devices are rejected before anything is launched."""
    dev, first = None, None
    for name, t in named:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if dev is None:
            dev, first = t.device, name
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device} but {first} is on {dev}: every tensor of one call must be "
                             "on the same GPU")
    if dev is None:
        raise ValueError("no CUDA tensor given")
    return dev


def _stream(stream, device):
    """The launch stream: the given one (which must belong to `device`) or `device`'s current stream."""
    import torch

    s = torch.cuda.current_stream(device) if stream is None else stream
    if s.device != device:
        raise ValueError(f"stream is on {s.device}, the tensors on {device}")
    return ctypes.c_void_p(s.cuda_stream)


def _io_dims(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, scale, l2_eps) -> GdnDims:
    import torch

    if q.dim() != 4 or v.dim() != 4 or state_pool.dim() != 4:
        raise ValueError("q/k and v/o are 4-D, state_pool is 4-D")
    B, T, HK, DK = q.shape
    HV, DV = v.shape[2], v.shape[3]
    _shape(k, q.shape, "k")
    _shape(v, (B, T, HV, DV), "v")
    if o is not None:
        _shape(o, (B, T, HV, DV), "o")
    _shape(a, (B, T, HV), "a")
    _shape(b, (B, T, HV), "b")
    _shape(A_log, (HV,), "A_log")
    _shape(dt_bias, (HV,), "dt_bias")
    if state_indices is not None:  # None: the caller checks the indices (prefill: one per prompt)
        _shape(state_indices, (B,), "state_indices")
    num_slots = state_pool.shape[0]
    _shape(state_pool, (num_slots, HV, DV, DK), "state_pool")
    qkv = _code(q, "q")
    for t, n in ((k, "k"), (v, "v"), (a, "a"), (b, "b")):
        if _code(t, n) != qkv:
            raise TypeError(f"{n} must have q's dtype")
    for t, n in ((A_log, "A_log"), (dt_bias, "dt_bias")):
        if t.dtype != torch.float32:
            raise TypeError(f"{n} must be fp32")
    if state_indices is not None and state_indices.dtype != torch.int32:
        raise TypeError("state_indices must be int32")
    out = _code(o, "o") if o is not None else _code(state_pool, "state_pool")
    return GdnDims(B, T, HK, HV, DK, DV, num_slots, qkv, _code(state_pool, "state_pool"), out, float(scale),
                   float(l2_eps))


def _call(status: int, what: str) -> None:
    if status != 0:
        raise GdnError(status, what)


def _launch(device, stream, fn, args, what: str) -> None:
    """One library call with `device` current, on `stream` (default: `device`'s current stream)."""
    import torch

    s = _stream(stream, device)
    with torch.cuda.device(device):
        _call(fn(*args, s), what)


def _io_named(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices):
    return [("q", q), ("k", k), ("v", v), ("a", a), ("b", b), ("A_log", A_log), ("dt_bias", dt_bias),
            ("state_pool", state_pool), ("state_indices", state_indices)]


# ---- the calls -------------------------------------------------------------------------------------------
def gdn_decode(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, err_word=None, *, scale=1.0,
               l2_eps=1e-6, stream=None) -> None:
    """T tokens (normally 1) from ``state_pool[state_indices[b]]``; the final state is written back in place."""
    L = lib()
    d = _io_dims(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, scale, l2_eps)
    device = _common_device(_io_named(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices)
                            + [("o", o), ("err_word", err_word)])
    _launch(device, stream, L.gdn_decode,
            (ctypes.byref(d), _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(a, "a"), _dev(b, "b"),
             _dev(A_log, "A_log"), _dev(dt_bias, "dt_bias"), _dev(state_pool, "state_pool"),
             _dev(state_indices, "state_indices"), _dev(o, "o"), _dev(err_word, "err_word")), "gdn_decode")


def gdn_decode_gated(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, norm, err_word=None, *,
                     scale=1.0, l2_eps=1e-6, stream=None) -> None:
    """``gdn_decode`` (o and the write-back) and the gated RMSNorm of o into ``norm.y`` (``norm``: a GatedNorm), in
    the same launch where the CTAs of a head fit one thread-block cluster."""
    L = lib()
    d = _io_dims(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, scale, l2_eps)
    nc = _norm_c(norm, o)
    device = _common_device(_io_named(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices)
                            + [("o", o), ("err_word", err_word)] + _norm_named(norm))
    _launch(device, stream, L.gdn_decode_gated,
            (ctypes.byref(d), _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(a, "a"), _dev(b, "b"),
             _dev(A_log, "A_log"), _dev(dt_bias, "dt_bias"), _dev(state_pool, "state_pool"),
             _dev(state_indices, "state_indices"), _dev(o, "o"), ctypes.byref(nc), _dev(err_word, "err_word")),
            "gdn_decode_gated")


def gdn_mtp_verify(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, intermediate_states=None,
                   err_word=None, *, scale=1.0, l2_eps=1e-6, stream=None) -> None:
    """T draft tokens from ``state_pool[state_indices[b]]`` (read only); optional per-token state cache."""
    L = lib()
    d = _io_dims(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, scale, l2_eps)
    if intermediate_states is not None:
        _shape(intermediate_states, (d.B, d.T, d.HV, d.DV, d.DK), "intermediate_states")
        if intermediate_states.dtype != state_pool.dtype:
            raise TypeError("intermediate_states must have state_pool's dtype")
    device = _common_device(_io_named(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices)
                            + [("o", o), ("intermediate_states", intermediate_states), ("err_word", err_word)])
    _launch(device, stream, L.gdn_mtp_verify,
            (ctypes.byref(d), _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(a, "a"), _dev(b, "b"),
             _dev(A_log, "A_log"), _dev(dt_bias, "dt_bias"), _dev(state_pool, "state_pool"),
             _dev(state_indices, "state_indices"), _dev(o, "o"), _dev(intermediate_states, "intermediate_states"),
             _dev(err_word, "err_word")), "gdn_mtp_verify")


def gdn_commit(state_pool, state_indices, intermediate_states, accept_len, err_word=None, *, stream=None) -> None:
    """``state_pool[state_indices[b]] = intermediate_states[b, accept_len[b] - 1]`` for active lanes."""
    import torch

    L = lib()
    if intermediate_states.dim() != 5 or state_pool.dim() != 4:
        raise ValueError("intermediate_states is [B,T,HV,DV,DK], state_pool is [num_slots,HV,DV,DK]")
    B, T, HV, DV, DK = intermediate_states.shape
    num_slots = state_pool.shape[0]
    _shape(state_pool, (num_slots, HV, DV, DK), "state_pool")
    _shape(state_indices, (B,), "state_indices")
    _shape(accept_len, (B,), "accept_len")
    if state_indices.dtype != torch.int32 or accept_len.dtype != torch.int32:
        raise TypeError("state_indices and accept_len must be int32")
    if intermediate_states.dtype != state_pool.dtype:
        raise TypeError("intermediate_states must have state_pool's dtype")
    sd = _code(state_pool, "state_pool")
    d = GdnDims(B, T, 1, HV, DK, DV, num_slots, sd, sd, sd, 1.0, 0.0)
    device = _common_device([("state_pool", state_pool), ("state_indices", state_indices),
                             ("intermediate_states", intermediate_states), ("accept_len", accept_len),
                             ("err_word", err_word)])
    _launch(device, stream, L.gdn_commit,
            (ctypes.byref(d), _dev(state_pool, "state_pool"), _dev(state_indices, "state_indices"),
             _dev(intermediate_states, "intermediate_states"), _dev(accept_len, "accept_len"),
             _dev(err_word, "err_word")), "gdn_commit")


def gdn_commit_replay(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, accept_len, err_word=None, *,
                      scale=1.0, l2_eps=1e-6, stream=None) -> None:
    """The first ``accept_len[b]`` tokens again from ``state_pool[state_indices[b]]``, final state written back
    (the verify call's inputs; no outputs).  The pool state ``gdn_commit`` leaves after a caching verify: the
    same bits for an fp32 pool or T > 8, within one bf16 ulp (the chunked tensor-core form) for a bf16 pool
    with T <= 8."""
    import torch

    L = lib()
    d = _io_dims(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, None, scale, l2_eps)
    _shape(accept_len, (d.B,), "accept_len")
    if accept_len.dtype != torch.int32:
        raise TypeError("accept_len must be int32")
    device = _common_device(_io_named(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices)
                            + [("accept_len", accept_len), ("err_word", err_word)])
    _launch(device, stream, L.gdn_commit_replay,
            (ctypes.byref(d), _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(a, "a"), _dev(b, "b"),
             _dev(A_log, "A_log"), _dev(dt_bias, "dt_bias"), _dev(state_pool, "state_pool"),
             _dev(state_indices, "state_indices"), _dev(accept_len, "accept_len"), _dev(err_word, "err_word")),
            "gdn_commit_replay")


def _norm_c(norm, o):
    """The C record of a GatedNorm for outputs o (checked: shapes, dtypes)."""
    import torch

    if norm is None:
        return None
    _shape(norm.z, o.shape, "norm.z")
    _shape(norm.y, o.shape, "norm.y")
    _shape(norm.norm_weight, (o.shape[-1],), "norm.norm_weight")
    if norm.y.dtype != o.dtype:
        raise TypeError("norm.y must have o's dtype")
    if norm.norm_weight.dtype != torch.float32:
        raise TypeError("norm.norm_weight must be fp32")
    return _GatedNormC(_dev(norm.z, "norm.z"), _code(norm.z, "norm.z"), _dev(norm.norm_weight, "norm.norm_weight"),
                       float(norm.eps), _dev(norm.y, "norm.y"))


def _norm_named(norm):
    return [] if norm is None else [("norm.z", norm.z), ("norm.norm_weight", norm.norm_weight), ("norm.y", norm.y)]


def gdn_mtp_verify_gated(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, norm, intermediate_states=None,
                         err_word=None, *, scale=1.0, l2_eps=1e-6, stream=None) -> None:
    """``gdn_mtp_verify`` (o, optional intermediate states) and the gated RMSNorm of o into ``norm.y``
    (``norm``: a GatedNorm), inside the verify kernel where one item holds a whole head."""
    L = lib()
    d = _io_dims(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, scale, l2_eps)
    if intermediate_states is not None:
        _shape(intermediate_states, (d.B, d.T, d.HV, d.DV, d.DK), "intermediate_states")
        if intermediate_states.dtype != state_pool.dtype:
            raise TypeError("intermediate_states must have state_pool's dtype")
    nc = _norm_c(norm, o)
    device = _common_device(_io_named(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices)
                            + [("o", o), ("intermediate_states", intermediate_states), ("err_word", err_word)]
                            + _norm_named(norm))
    _launch(device, stream, L.gdn_mtp_verify_gated,
            (ctypes.byref(d), _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(a, "a"), _dev(b, "b"),
             _dev(A_log, "A_log"), _dev(dt_bias, "dt_bias"), _dev(state_pool, "state_pool"),
             _dev(state_indices, "state_indices"), _dev(o, "o"), _dev(intermediate_states, "intermediate_states"),
             ctypes.byref(nc), _dev(err_word, "err_word")), "gdn_mtp_verify_gated")


def gdn_mtp_verify_commit(prev, q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, err_word=None, *,
                          norm=None, scale=1.0, l2_eps=1e-6, stream=None) -> None:
    """One speculative step in one pass: commit ``prev``'s accepted prefix (``prev``: a ``ReplayTokens``, exactly
    ``gdn_commit_replay`` of those tokens) into the slots, then verify these T tokens from the committed states
    (exactly ``gdn_mtp_verify`` without intermediate states).  ``prev`` may have another token count."""
    import torch

    L = lib()
    d = _io_dims(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, scale, l2_eps)
    if prev.k.dim() != 4:
        raise ValueError("prev.k is [B, T', HK, DK]")
    Tp = prev.k.shape[1]
    _shape(prev.k, (d.B, Tp, d.HK, d.DK), "prev.k")
    _shape(prev.v, (d.B, Tp, d.HV, d.DV), "prev.v")
    _shape(prev.a, (d.B, Tp, d.HV), "prev.a")
    _shape(prev.b, (d.B, Tp, d.HV), "prev.b")
    _shape(prev.accept_len, (d.B,), "prev.accept_len")
    for t, n in ((prev.k, "prev.k"), (prev.v, "prev.v"), (prev.a, "prev.a"), (prev.b, "prev.b")):
        if t.dtype != q.dtype:
            raise TypeError(f"{n} must have q's dtype")
    if prev.accept_len.dtype != torch.int32:
        raise TypeError("prev.accept_len must be int32")
    nc = _norm_c(norm, o)
    device = _common_device(_io_named(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices)
                            + [("o", o), ("err_word", err_word), ("prev.k", prev.k), ("prev.v", prev.v),
                               ("prev.a", prev.a), ("prev.b", prev.b), ("prev.accept_len", prev.accept_len)]
                            + _norm_named(norm))
    rt = _ReplayTokensC(Tp, _dev(prev.k, "prev.k"), _dev(prev.v, "prev.v"), _dev(prev.a, "prev.a"),
                        _dev(prev.b, "prev.b"), _dev(prev.accept_len, "prev.accept_len"))
    _launch(device, stream, L.gdn_mtp_verify_commit,
            (ctypes.byref(d), ctypes.byref(rt), _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(a, "a"),
             _dev(b, "b"), _dev(A_log, "A_log"), _dev(dt_bias, "dt_bias"), _dev(state_pool, "state_pool"),
             _dev(state_indices, "state_indices"), _dev(o, "o"), ctypes.byref(nc) if nc is not None else None,
             _dev(err_word, "err_word")),
            "gdn_mtp_verify_commit")


def gdn_prefill(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, cu_seqlens, o, has_initial_state=None,
                err_word=None, *, scale=1.0, l2_eps=1e-6, stream=None) -> None:
    """Prefill of ``len(cu_seqlens) - 1`` packed sequences: sequence b (tokens ``cu_seqlens[b]`` ..
    ``cu_seqlens[b+1]-1``) starts from ``state_pool[state_indices[b]]`` (or zero where
    ``has_initial_state[b] == 0``), writes o at its tokens and its final state into that slot."""
    import torch

    L = lib()
    if q.dim() != 3 or v.dim() != 3:
        raise ValueError("prefill takes packed tokens: q, k [N,HK,DK], v, o [N,HV,DV], a, b [N,HV]")
    N = q.shape[0]
    B = cu_seqlens.shape[0] - 1
    if cu_seqlens.dim() != 1 or B < 0:
        raise ValueError("cu_seqlens is [B+1]")
    if cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    # the [B, T] checks of the other calls, with the token axis as T of one "lane"; the indices are per prompt
    d = _io_dims(q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0), a.unsqueeze(0), b.unsqueeze(0), A_log, dt_bias,
                 state_pool, None, o.unsqueeze(0), scale, l2_eps)
    _shape(state_indices, (B,), "state_indices")
    if state_indices.dtype != torch.int32:
        raise TypeError("state_indices must be int32")
    if has_initial_state is not None:
        _shape(has_initial_state, (B,), "has_initial_state")
        if has_initial_state.dtype != torch.int32:
            raise TypeError("has_initial_state must be int32")
    d.B, d.T = B, N
    device = _common_device(_io_named(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices)
                            + [("cu_seqlens", cu_seqlens), ("o", o), ("has_initial_state", has_initial_state),
                               ("err_word", err_word)])
    _launch(device, stream, L.gdn_prefill,
            (ctypes.byref(d), _dev(cu_seqlens, "cu_seqlens"), _dev(q, "q"), _dev(k, "k"), _dev(v, "v"),
             _dev(a, "a"), _dev(b, "b"), _dev(A_log, "A_log"), _dev(dt_bias, "dt_bias"),
             _dev(state_pool, "state_pool"), _dev(state_indices, "state_indices"),
             _dev(has_initial_state, "has_initial_state"), _dev(o, "o"), _dev(err_word, "err_word")), "gdn_prefill")


def gdn_gated_rmsnorm(o, z, norm_weight, y=None, *, eps=1e-6, stream=None):
    """``y = o / sqrt(mean(o^2) + eps) * norm_weight * silu(z)`` over the last axis (DV) of o; returns y
    (a new tensor of o's shape and dtype unless given; ``y`` may be ``o`` itself)."""
    import torch

    L = lib()
    if o.dim() < 1 or tuple(z.shape) != tuple(o.shape):
        raise ValueError("z must have o's shape")
    DV = o.shape[-1]
    _shape(norm_weight, (DV,), "norm_weight")
    if norm_weight.dtype != torch.float32:
        raise TypeError("norm_weight must be fp32")
    if y is None:
        y = torch.empty_like(o)
    _shape(y, o.shape, "y")
    if y.dtype != o.dtype:
        raise TypeError("y must have o's dtype")
    rows = o.numel() // DV if DV > 0 else 0
    device = _common_device([("o", o), ("z", z), ("norm_weight", norm_weight), ("y", y)])
    _launch(device, stream, L.gdn_gated_rmsnorm,
            (rows, DV, _code(o, "o"), _code(z, "z"), _dev(o, "o"), _dev(z, "z"), _dev(norm_weight, "norm_weight"),
             float(eps), _dev(y, "y")), "gdn_gated_rmsnorm")
    return y


def _conv_dims(x, W, conv_w, conv_state, out, silu):
    """gdn_conv_dims from the tensors: x [B,T,H], W [C,H], conv_w [Cc,K], conv_state [num_slots,K-1,Cc] and the
    outputs' shapes (HK, DK from q; HV, DV from v)."""
    import torch

    if x.dim() != 3 or W.dim() != 2 or conv_w.dim() != 2 or conv_state.dim() != 3:
        raise ValueError("x is [B,T,H], W [C,H], conv_w [Cc,K], conv_state [num_slots,K-1,Cc]")
    B, T, H = x.shape
    if out.q.dim() != 4 or out.v.dim() != 4:
        raise ValueError("q and v are 4-D")
    HK, DK = out.q.shape[2], out.q.shape[3]
    HV, DV = out.v.shape[2], out.v.shape[3]
    Cc = 2 * HK * DK + HV * DV
    C = Cc + HV * DV + 2 * HV
    K = conv_w.shape[1]
    _shape(W, (C, H), "W")
    _shape(conv_w, (Cc, K), "conv_w")
    _shape(conv_state, (conv_state.shape[0], K - 1, Cc), "conv_state")
    for t, n, want in ((out.q, "q", (B, T, HK, DK)), (out.k, "k", (B, T, HK, DK)), (out.v, "v", (B, T, HV, DV)),
                       (out.z, "z", (B, T, HV, DV)), (out.b, "b", (B, T, HV)), (out.a, "a", (B, T, HV))):
        _shape(t, want, n)
    for t, n in ((x, "x"), (W, "W")):
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{n} must be bf16")
    if conv_w.dtype != torch.float32:
        raise TypeError("conv_w must be fp32")
    od = _code(out.q, "q")
    for t, n in ((out.k, "k"), (out.v, "v"), (out.z, "z"), (out.b, "b"), (out.a, "a")):
        if _code(t, n) != od:
            raise TypeError(f"{n} must have q's dtype")
    return _ConvDimsC(B, T, H, HK, HV, DK, DV, K, conv_state.shape[0], _code(conv_state, "conv_state"), od,
                      1 if silu else 0)


def gdn_in_proj_conv(x, W, conv_w, conv_b, conv_state, state_indices, out, write_state, records=None,
                     err_word=None, *, silu=True, stream=None) -> None:
    """The in_proj projection of x's rows with its causal conv1d epilogue into ``out`` (an ``InProjOut``);
    ``write_state`` (decode) moves each lane's convolution state on by its T rows, otherwise ``records``
    (``[B,T,Cc]``, conv_state's dtype) receives the pre-convolution values for ``gdn_conv_commit``."""
    import torch

    L = lib()
    d = _conv_dims(x, W, conv_w, conv_state, out, silu)
    _shape(state_indices, (d.B,), "state_indices")
    if state_indices.dtype != torch.int32:
        raise TypeError("state_indices must be int32")
    Cc = 2 * d.HK * d.DK + d.HV * d.DV
    if conv_b is not None:
        _shape(conv_b, (Cc,), "conv_b")
        if conv_b.dtype != torch.float32:
            raise TypeError("conv_b must be fp32")
    if records is not None:
        _shape(records, (d.B, d.T, Cc), "records")
        if _code(records, "records") != d.conv_dtype:
            raise TypeError("records must have conv_state's dtype")
    device = _common_device([("x", x), ("W", W), ("conv_w", conv_w), ("conv_b", conv_b), ("conv_state", conv_state),
                             ("state_indices", state_indices), ("q", out.q), ("k", out.k), ("v", out.v),
                             ("z", out.z), ("b", out.b), ("a", out.a), ("records", records), ("err_word", err_word)])
    oc = _InProjOutC(*(_dev(t, n) for t, n in ((out.q, "q"), (out.k, "k"), (out.v, "v"), (out.z, "z"),
                                                (out.b, "b"), (out.a, "a"))))
    _launch(device, stream, L.gdn_in_proj_conv,
            (ctypes.byref(d), _dev(x, "x"), _dev(W, "W"), _dev(conv_w, "conv_w"), _dev(conv_b, "conv_b"),
             _dev(conv_state, "conv_state"), _dev(state_indices, "state_indices"), 1 if write_state else 0,
             ctypes.byref(oc), _dev(records, "records"), _dev(err_word, "err_word", torch.int32)),
            "gdn_in_proj_conv")


def gdn_conv_commit(conv_state, state_indices, records, accept_len, err_word=None, *, stream=None) -> None:
    """The convolution state after each lane's first ``accept_len[b]`` verify rows, from their records."""
    import torch

    L = lib()
    if conv_state.dim() != 3 or records.dim() != 3:
        raise ValueError("conv_state is [num_slots,K-1,Cc], records [B,T,Cc]")
    B, T, Cc = records.shape
    K = conv_state.shape[1] + 1
    _shape(conv_state, (conv_state.shape[0], K - 1, Cc), "conv_state")
    _shape(state_indices, (B,), "state_indices")
    _shape(accept_len, (B,), "accept_len")
    for t, n in ((state_indices, "state_indices"), (accept_len, "accept_len")):
        if t.dtype != torch.int32:
            raise TypeError(f"{n} must be int32")
    if _code(records, "records") != _code(conv_state, "conv_state"):
        raise TypeError("records must have conv_state's dtype")
    # the commit needs only the channel count Cc = 2*HK*DK + HV*DV (at least 3): any head layout with that count
    if Cc < 3:
        raise ValueError("records: fewer than 3 channels")
    d = _ConvDimsC(B, T, 8, 1, 1, 1, Cc - 2, K, conv_state.shape[0], _code(conv_state, "conv_state"), BF16, 1)
    device = _common_device([("conv_state", conv_state), ("state_indices", state_indices), ("records", records),
                             ("accept_len", accept_len), ("err_word", err_word)])
    _launch(device, stream, L.gdn_conv_commit,
            (ctypes.byref(d), _dev(conv_state, "conv_state"), _dev(state_indices, "state_indices"),
             _dev(records, "records"), _dev(accept_len, "accept_len"), _dev(err_word, "err_word", torch.int32)),
            "gdn_conv_commit")
