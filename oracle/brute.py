"""Independent NumPy restatement of the gated delta rule in product form, float64, dense matrices (decode /
verify lanes: ``lane_head``; prefill sequences: ``sequence_head``).

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).  It shares nothing with ``gdn_oracle.c`` beyond the
definition both restate: the loop oracle scales, projects and updates row by row; this module multiplies
whole matrices,

    S_t = g_t * S_{t-1} (I - beta_t kh_t kh_t^T) + beta_t v_t kh_t^T,      o_t = scale * S_t qh_t,

which equals the loop form in exact arithmetic (expand g S - beta (g S kh - v) kh^T).  softplus is
``numpy.logaddexp(0, x)`` and the sigmoid ``scipy.special.expit`` (library routines), so a slip in the
loop oracle's scalar functions also shows up as a mismatch.  Used on tiny dims only.
"""
from __future__ import annotations

from typing import Dict, List, Tuple

import numpy as np

try:
    from scipy.special import expit as _sigmoid
except ImportError:  # pragma: no cover - scipy is present on both machines, kept for safety
    def _sigmoid(x):
        return 1.0 / (1.0 + np.exp(-x))


def decode_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.asarray(x, np.float32).astype(np.float64)
    if dtype == "bf16":
        return (np.asarray(x, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == "f64":
        return np.asarray(x, np.float64)
    raise ValueError(dtype)


def lane_head(d: Dict, x: Dict[str, np.ndarray], b: int, h: int) -> Tuple[np.ndarray, List[np.ndarray]]:
    """Outputs o[b, :, h] (T x DV) and the states after each token (T arrays DV x DK) of one lane/head."""
    T, HK, HV, DK, DV = d["T"], d["HK"], d["HV"], d["DK"], d["DV"]
    qd, sd = d["qkv_dtype"], d["state_dtype"]
    eps, scale = float(d.get("l2_eps", 1e-6)), float(d.get("scale", 1.0))
    slot = int(x["indices"][b])
    hk = h // (HV // HK)
    S = decode_storage(x["pool"][slot, h], sd).reshape(DV, DK)
    I = np.eye(DK)
    outs, states = [], []
    for t in range(T):
        q = decode_storage(x["q"][b, t, hk], qd)
        k = decode_storage(x["k"][b, t, hk], qd)
        v = decode_storage(x["v"][b, t, h], qd)
        qh = q / np.sqrt(q @ q + eps)
        kh = k / np.sqrt(k @ k + eps)
        a = decode_storage(x["a"][b, t, h], qd)
        bb = decode_storage(x["b"][b, t, h], qd)
        A = float(x["A_log"][h])
        dt = float(x["dt_bias"][h])
        g = np.exp(-np.exp(A) * np.logaddexp(0.0, a + dt))
        beta = _sigmoid(bb)
        S = g * S @ (I - beta * np.outer(kh, kh)) + beta * np.outer(v, kh)
        outs.append(scale * (S @ qh))
        states.append(S.copy())
    return np.stack(outs), states


def sequence_head(d: Dict, x: Dict[str, np.ndarray], cu_seqlens, has_initial_state, b: int,
                  h: int) -> Tuple[np.ndarray, np.ndarray]:
    """Prefill of sequence b, value head h, in product form: outputs (L x DV) at token positions
    cu_seqlens[b] .. cu_seqlens[b+1]-1 of the packed arrays and the final state (DV x DK).  The start is the
    pool slot's state, or the zero matrix where has_initial_state[b] == 0."""
    HK, HV, DK, DV = d["HK"], d["HV"], d["DK"], d["DV"]
    qd, sd = d["qkv_dtype"], d["state_dtype"]
    eps, scale = float(d.get("l2_eps", 1e-6)), float(d.get("scale", 1.0))
    hk = h // (HV // HK)
    fresh = has_initial_state is not None and int(has_initial_state[b]) == 0
    S = np.zeros((DV, DK)) if fresh else decode_storage(x["pool"][int(x["indices"][b]), h], sd).reshape(DV, DK)
    I = np.eye(DK)
    outs = []
    for n in range(int(cu_seqlens[b]), int(cu_seqlens[b + 1])):
        q = decode_storage(x["q"][n, hk], qd)
        k = decode_storage(x["k"][n, hk], qd)
        v = decode_storage(x["v"][n, h], qd)
        qh = q / np.sqrt(q @ q + eps)
        kh = k / np.sqrt(k @ k + eps)
        g = np.exp(-np.exp(float(x["A_log"][h])) *
                   np.logaddexp(0.0, decode_storage(x["a"][n, h], qd) + float(x["dt_bias"][h])))
        beta = _sigmoid(decode_storage(x["b"][n, h], qd))
        S = g * S @ (I - beta * np.outer(kh, kh)) + beta * np.outer(v, kh)
        outs.append(scale * (S @ qh))
    return (np.stack(outs) if outs else np.zeros((0, DV))), S
