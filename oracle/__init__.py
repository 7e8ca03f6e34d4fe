"""CPU oracle for the Gated DeltaNet decode / MTP-verify / commit / prefill path, its gated RMSNorm, and the
in_proj projection with its causal conv1d epilogue (and the convolution state's commit).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline`` leg
and ``--impl reference`` arm may import this package.  It shares no code with the CUDA library in
``gated_deltanet_linear_mtp_gb300`` and neither imports the other.

* ``gdn_oracle.c``  -- the loop oracle (fp64, plain loops); wrapped here through ``ctypes``.
* ``brute.py``      -- an independent NumPy product-form restatement used to pin the loop oracle.
* ``build.py``      -- compiles ``gdn_oracle.c`` with gcc into ``oracle/_build/libgdn_oracle.so``.

Arrays are passed in their storage form: fp32 as ``float32``, bf16 as ``uint16`` bit patterns, fp64 as
``float64`` (fp64 storage exists only here, for chained-call pins without storage rounding).

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py`` (closed forms, library special
cases, brute force on tiny inputs, chained-call identities); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Tuple

import numpy as np

from . import build as _build

DTYPE_CODE = {"f32": 0, "bf16": 1, "f64": 2}
NP_STORAGE = {"f32": np.float32, "bf16": np.uint16, "f64": np.float64}


class _ConvDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32), ("HK", ctypes.c_int32),
                ("HV", ctypes.c_int32), ("DK", ctypes.c_int32), ("DV", ctypes.c_int32), ("K", ctypes.c_int32),
                ("num_slots", ctypes.c_int32), ("x_dtype", ctypes.c_int32), ("conv_dtype", ctypes.c_int32),
                ("silu", ctypes.c_int32)]


def conv_channels(d: Dict) -> Tuple[int, int]:
    """(Cc, C): the convolved channels q | k | v and all in_proj channels q | k | v | z | b | a."""
    Cc = 2 * d["HK"] * d["DK"] + d["HV"] * d["DV"]
    return Cc, Cc + d["HV"] * d["DV"] + 2 * d["HV"]


def split_in_proj(d: Dict, out: np.ndarray) -> Dict[str, np.ndarray]:
    """The in_proj outputs [B, T, C] split into q, k [B,T,HK,DK], v, z [B,T,HV,DV], b, a [B,T,HV] (views)."""
    B, T = out.shape[:2]
    HK, HV, DK, DV = d["HK"], d["HV"], d["DK"], d["DV"]
    o = np.cumsum([0, HK * DK, HK * DK, HV * DV, HV * DV, HV, HV])
    return dict(q=out[..., o[0]:o[1]].reshape(B, T, HK, DK), k=out[..., o[1]:o[2]].reshape(B, T, HK, DK),
                v=out[..., o[2]:o[3]].reshape(B, T, HV, DV), z=out[..., o[3]:o[4]].reshape(B, T, HV, DV),
                b=out[..., o[4]:o[5]], a=out[..., o[5]:o[6]])


class _Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("HK", ctypes.c_int32), ("HV", ctypes.c_int32),
                ("DK", ctypes.c_int32), ("DV", ctypes.c_int32), ("num_slots", ctypes.c_int32),
                ("qkv_dtype", ctypes.c_int32), ("state_dtype", ctypes.c_int32), ("cache_dtype", ctypes.c_int32),
                ("scale", ctypes.c_double), ("l2_eps", ctypes.c_double)]


def _ptr(x: Optional[np.ndarray]):
    if x is None:
        return None
    assert x.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return x.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes handle on one build of ``gdn_oracle.c`` (the default build, or a test's variant)."""

    def __init__(self, lib_path: Optional[str] = None):
        if lib_path is None:
            lib_path = _build.library_path()
            if not os.path.exists(lib_path):
                _build.build()
        self.path = lib_path
        self.lib = ctypes.CDLL(lib_path)
        vp, dp, ip = ctypes.c_void_p, ctypes.POINTER(_Dims), ctypes.c_void_p
        self.lib.orc_verify.argtypes = [dp] + [vp] * 5 + [vp, vp, vp, ip, vp, vp]
        self.lib.orc_decode.argtypes = [dp] + [vp] * 5 + [vp, vp, vp, ip, vp]
        self.lib.orc_commit.argtypes = [dp, vp, ip, vp, ip]
        self.lib.orc_commit_replay.argtypes = [dp] + [vp] * 5 + [vp, vp, vp, ip, ip]
        self.lib.orc_prefill.argtypes = [dp, ip] + [vp] * 5 + [vp, vp, vp, ip, ip, vp]
        self.lib.orc_gated_rmsnorm.argtypes = [ctypes.c_int64, ctypes.c_int32, vp, ctypes.c_int32, vp,
                                               ctypes.c_int32, vp, ctypes.c_double, vp]
        cdp = ctypes.POINTER(_ConvDims)
        self.lib.orc_in_proj_conv.argtypes = [cdp, vp, vp, vp, vp, vp, ip, ctypes.c_int32, vp, vp]
        self.lib.orc_conv_commit.argtypes = [cdp, vp, ip, vp, ip]
        for f in (self.lib.orc_verify, self.lib.orc_decode, self.lib.orc_commit, self.lib.orc_commit_replay,
                  self.lib.orc_prefill, self.lib.orc_gated_rmsnorm, self.lib.orc_in_proj_conv,
                  self.lib.orc_conv_commit):
            f.restype = ctypes.c_int
        for name in ("orc_round_bf16", "orc_softplus", "orc_sigmoid"):
            getattr(self.lib, name).argtypes = [ctypes.c_double]
            getattr(self.lib, name).restype = ctypes.c_double
        self.lib.orc_gate.argtypes = [ctypes.c_double] * 3
        self.lib.orc_gate.restype = ctypes.c_double

    # -- scalar helpers (exported for the pins) --------------------------------------------------
    def round_bf16(self, x: float) -> float:
        return self.lib.orc_round_bf16(float(x))

    def softplus(self, x: float) -> float:
        return self.lib.orc_softplus(float(x))

    def sigmoid(self, x: float) -> float:
        return self.lib.orc_sigmoid(float(x))

    def gate(self, A_log: float, a: float, dt_bias: float) -> float:
        return self.lib.orc_gate(float(A_log), float(a), float(dt_bias))

    # -- calls -----------------------------------------------------------------------------------
    @staticmethod
    def _dims(d: Dict, B: int) -> _Dims:
        cache_dtype = d.get("cache_dtype", d["state_dtype"])
        return _Dims(B, d["T"], d["HK"], d["HV"], d["DK"], d["DV"], d["num_slots"],
                     DTYPE_CODE[d["qkv_dtype"]], DTYPE_CODE[d["state_dtype"]], DTYPE_CODE[cache_dtype],
                     float(d.get("scale", 1.0)), float(d.get("l2_eps", 1e-6)))

    @staticmethod
    def _check(x: np.ndarray, dtype: str, shape: Tuple[int, ...], name: str) -> np.ndarray:
        want = NP_STORAGE[dtype]
        if x.dtype != want or tuple(x.shape) != tuple(shape):
            raise ValueError(f"{name}: expected {want.__name__}{shape}, got {x.dtype}{x.shape}")
        return np.ascontiguousarray(x)

    def _inputs(self, d: Dict, x: Dict[str, np.ndarray], B: int):
        T, HK, HV, DK, DV = d["T"], d["HK"], d["HV"], d["DK"], d["DV"]
        qd = d["qkv_dtype"]
        q = self._check(x["q"], qd, (B, T, HK, DK), "q")
        k = self._check(x["k"], qd, (B, T, HK, DK), "k")
        v = self._check(x["v"], qd, (B, T, HV, DV), "v")
        a = self._check(x["a"], qd, (B, T, HV), "a")
        b = self._check(x["b"], qd, (B, T, HV), "b")
        A_log = self._check(x["A_log"], "f32", (HV,), "A_log")
        dt_bias = self._check(x["dt_bias"], "f32", (HV,), "dt_bias")
        idx = np.ascontiguousarray(x["indices"], dtype=np.int32)
        if idx.shape != (B,):
            raise ValueError("indices shape")
        return q, k, v, a, b, A_log, dt_bias, idx

    def verify(self, d: Dict, x: Dict[str, np.ndarray], cache: bool = True,
               o: Optional[np.ndarray] = None, cache_out: Optional[np.ndarray] = None):
        """Returns (o [B,T,HV,DV] fp64, cache [B,T,HV,DV,DK] storage or None, flag word).

        ``o`` / ``cache_out`` may be passed pre-filled (canaries): entries of skipped lanes are left as given.
        """
        B = x["q"].shape[0]
        T, HV, DV, DK = d["T"], d["HV"], d["DV"], d["DK"]
        q, k, v, a, b, A_log, dt_bias, idx = self._inputs(d, x, B)
        pool = self._check(x["pool"], d["state_dtype"], (d["num_slots"], HV, DV, DK), "pool")
        if o is None:
            o = np.zeros((B, T, HV, DV), np.float64)
        cd = d.get("cache_dtype", d["state_dtype"])
        if cache and cache_out is None:
            cache_out = np.zeros((B, T, HV, DV, DK), NP_STORAGE[cd])
        dims = self._dims(d, B)
        flags = self.lib.orc_verify(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
                                    _ptr(dt_bias), _ptr(pool), _ptr(idx), _ptr(o),
                                    _ptr(cache_out) if cache else None)
        if flags < 0:
            raise ValueError(f"oracle rejected dims ({flags})")
        return o, (cache_out if cache else None), flags

    def decode(self, d: Dict, x: Dict[str, np.ndarray], pool: np.ndarray, o: Optional[np.ndarray] = None):
        """Updates ``pool`` in place (active slots); returns (o fp64, flag word)."""
        B = x["q"].shape[0]
        q, k, v, a, b, A_log, dt_bias, idx = self._inputs(d, x, B)
        assert pool.flags["C_CONTIGUOUS"]
        self._check(pool, d["state_dtype"], (d["num_slots"], d["HV"], d["DV"], d["DK"]), "pool")
        if o is None:
            o = np.zeros((B, d["T"], d["HV"], d["DV"]), np.float64)
        dims = self._dims(d, B)
        flags = self.lib.orc_decode(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
                                    _ptr(dt_bias), _ptr(pool), _ptr(idx), _ptr(o))
        if flags < 0:
            raise ValueError(f"oracle rejected dims ({flags})")
        return o, flags

    def commit_replay(self, d: Dict, x: Dict[str, np.ndarray], pool: np.ndarray, accept_len: np.ndarray) -> int:
        """Replay commit in place: the first accept_len[b] tokens from pool[idx[b]], written back."""
        B = x["q"].shape[0]
        q, k, v, a, b, A_log, dt_bias, idx = self._inputs(d, x, B)
        assert pool.flags["C_CONTIGUOUS"]
        self._check(pool, d["state_dtype"], (d["num_slots"], d["HV"], d["DV"], d["DK"]), "pool")
        L = np.ascontiguousarray(accept_len, dtype=np.int32)
        dims = self._dims(d, B)
        flags = self.lib.orc_commit_replay(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                                           _ptr(A_log), _ptr(dt_bias), _ptr(pool), _ptr(idx), _ptr(L))
        if flags < 0:
            raise ValueError(f"oracle rejected dims ({flags})")
        return flags

    def prefill(self, d: Dict, x: Dict[str, np.ndarray], cu_seqlens: np.ndarray, pool: np.ndarray,
                has_initial_state: Optional[np.ndarray] = None, o: Optional[np.ndarray] = None):
        """Prefill of len(cu_seqlens) - 1 packed sequences; ``x`` holds q, k [N, HK, DK], v [N, HV, DV],
        a, b [N, HV], A_log, dt_bias, indices [B].  Updates ``pool`` in place (the slots of active
        sequences); returns (o [N, HV, DV] fp64, flag word).  ``o`` may be passed pre-filled (canaries)."""
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        B = cu.shape[0] - 1
        N = x["q"].shape[0]
        HK, HV, DK, DV = d["HK"], d["HV"], d["DK"], d["DV"]
        qd = d["qkv_dtype"]
        q = self._check(x["q"], qd, (N, HK, DK), "q")
        k = self._check(x["k"], qd, (N, HK, DK), "k")
        v = self._check(x["v"], qd, (N, HV, DV), "v")
        a = self._check(x["a"], qd, (N, HV), "a")
        b = self._check(x["b"], qd, (N, HV), "b")
        A_log = self._check(x["A_log"], "f32", (HV,), "A_log")
        dt_bias = self._check(x["dt_bias"], "f32", (HV,), "dt_bias")
        idx = np.ascontiguousarray(x["indices"], dtype=np.int32)
        if B < 0 or idx.shape != (B,):
            raise ValueError("indices / cu_seqlens shapes")
        assert pool.flags["C_CONTIGUOUS"]
        self._check(pool, d["state_dtype"], (d["num_slots"], HV, DV, DK), "pool")
        init = None
        if has_initial_state is not None:
            init = np.ascontiguousarray(has_initial_state, dtype=np.int32)
            if init.shape != (B,):
                raise ValueError("has_initial_state shape")
        if o is None:
            o = np.zeros((N, HV, DV), np.float64)
        if N == 0 or B == 0:
            return o, 0
        dims = self._dims(dict(d, T=N), B)
        flags = self.lib.orc_prefill(ctypes.byref(dims), _ptr(cu), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                                     _ptr(A_log), _ptr(dt_bias), _ptr(pool), _ptr(idx), _ptr(init), _ptr(o))
        if flags < 0:
            raise ValueError(f"oracle rejected dims ({flags})")
        return o, flags

    def gated_rmsnorm(self, o: np.ndarray, o_dtype: str, z: np.ndarray, z_dtype: str, w: np.ndarray,
                      eps: float) -> np.ndarray:
        """y = o / sqrt(mean(o^2) + eps) * w * silu(z) over the last axis (length DV); fp64 result."""
        o = self._check(o, o_dtype, o.shape, "o")
        z = self._check(z, z_dtype, o.shape, "z")
        DV = o.shape[-1]
        w = self._check(w, "f32", (DV,), "w")
        y = np.zeros(o.shape, np.float64)
        rows = int(np.prod(o.shape[:-1]))
        rc = self.lib.orc_gated_rmsnorm(rows, DV, _ptr(o), DTYPE_CODE[o_dtype], _ptr(z), DTYPE_CODE[z_dtype],
                                        _ptr(w), float(eps), _ptr(y))
        if rc < 0:
            raise ValueError(f"oracle rejected sizes ({rc})")
        return y

    def commit(self, d: Dict, pool: np.ndarray, indices: np.ndarray, cache: np.ndarray,
               accept_len: np.ndarray) -> int:
        """pool[idx[b]] = cache[b, L_b - 1] in place; returns the flag word."""
        B = indices.shape[0]
        assert pool.flags["C_CONTIGUOUS"] and cache.flags["C_CONTIGUOUS"]
        self._check(cache, d["state_dtype"], (B, d["T"], d["HV"], d["DV"], d["DK"]), "cache")
        idx = np.ascontiguousarray(indices, dtype=np.int32)
        L = np.ascontiguousarray(accept_len, dtype=np.int32)
        dims = self._dims(d, B)
        flags = self.lib.orc_commit(ctypes.byref(dims), _ptr(pool), _ptr(idx), _ptr(cache), _ptr(L))
        if flags < 0:
            raise ValueError(f"oracle rejected dims ({flags})")
        return flags


    # -- the in_proj projection with its causal conv1d epilogue ----------------------------------------------
    @staticmethod
    def _conv_dims(d: Dict, B: int) -> _ConvDims:
        return _ConvDims(B, d["T"], d["H"], d["HK"], d["HV"], d["DK"], d["DV"], d["K"], d["num_slots"],
                         DTYPE_CODE[d["x_dtype"]], DTYPE_CODE[d["conv_dtype"]], int(bool(d.get("silu", 1))))

    def in_proj_conv(self, d: Dict, x: np.ndarray, W: np.ndarray, conv_w: np.ndarray, conv_b: Optional[np.ndarray],
                     pool: np.ndarray, indices: np.ndarray, write_pool: bool, records: bool = True,
                     out: Optional[np.ndarray] = None):
        """x [B,T,H], W [C,H] (``x_dtype``), conv_w [Cc,K] / conv_b [Cc] fp32, pool [slots,K-1,Cc] (``conv_dtype``,
        updated in place when ``write_pool``).  Returns (out [B,T,C] fp64 in W's channel order, the recovery
        records [B,T,Cc] in ``conv_dtype`` or None, flag word).  ``out`` may be passed pre-filled (canaries):
        rows of skipped lanes are left as given."""
        B = indices.shape[0]
        T, H, K = d["T"], d["H"], d["K"]
        Cc, C = conv_channels(d)
        x = self._check(x, d["x_dtype"], (B, T, H), "x")
        W = self._check(W, d["x_dtype"], (C, H), "W")
        conv_w = self._check(conv_w, "f32", (Cc, K), "conv_w")
        if conv_b is not None:
            conv_b = self._check(conv_b, "f32", (Cc,), "conv_b")
        self._check(pool, d["conv_dtype"], (d["num_slots"], K - 1, Cc), "pool")
        assert pool.flags["C_CONTIGUOUS"]
        idx = np.ascontiguousarray(indices, dtype=np.int32)
        if out is None:
            out = np.zeros((B, T, C), np.float64)
        rec = np.zeros((B, T, Cc), NP_STORAGE[d["conv_dtype"]]) if records else None
        dims = self._conv_dims(d, B)
        flags = self.lib.orc_in_proj_conv(ctypes.byref(dims), _ptr(x), _ptr(W), _ptr(conv_w), _ptr(conv_b),
                                          _ptr(pool), _ptr(idx), int(bool(write_pool)), _ptr(out), _ptr(rec))
        if flags < 0:
            raise ValueError(f"oracle rejected dims ({flags})")
        return out, rec, flags

    def conv_commit(self, d: Dict, pool: np.ndarray, indices: np.ndarray, records: np.ndarray,
                    accept_len: np.ndarray) -> int:
        """The convolution state after each lane's first L_b rows, from its recovery records, in place."""
        B = indices.shape[0]
        Cc, _ = conv_channels(d)
        self._check(pool, d["conv_dtype"], (d["num_slots"], d["K"] - 1, Cc), "pool")
        records = self._check(records, d["conv_dtype"], (B, d["T"], Cc), "records")
        idx = np.ascontiguousarray(indices, dtype=np.int32)
        L = np.ascontiguousarray(accept_len, dtype=np.int32)
        dims = self._conv_dims(d, B)
        flags = self.lib.orc_conv_commit(ctypes.byref(dims), _ptr(pool), _ptr(idx), _ptr(records), _ptr(L))
        if flags < 0:
            raise ValueError(f"oracle rejected dims ({flags})")
        return flags


_default: Optional[Oracle] = None


def default() -> Oracle:
    """The oracle built from ``gdn_oracle.c`` as committed (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def dims_of(w) -> Dict:
    """Dims dict from a ``gdn_workloads.Workload``."""
    return dict(T=w.T, HK=w.HK, HV=w.HV, DK=w.DK, DV=w.DV, num_slots=w.num_slots, qkv_dtype=w.qkv_dtype,
                state_dtype=w.state_dtype, scale=w.scale, l2_eps=w.l2_eps)
