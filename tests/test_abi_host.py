"""libgdn.so loads, exports every function ``include/gdn.h`` declares, and rejects bad arguments on the host
with the documented status before touching CUDA (no call here reaches a kernel launch; no GPU needed)."""
import ctypes
import os
import re

import pytest

import gated_deltanet_linear_mtp_gb300 as gdn
from gated_deltanet_linear_mtp_gb300 import build as gbuild

HEADER = os.path.join(gbuild.INCLUDE, "gdn.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(gbuild.LIB_PATH):
        gbuild.build()
    return gdn.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(gdn.EXPORTS)


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_library_exports_only_the_declared_functions(L):
    """Hidden visibility: internal symbols (template statics among them) must not bind across two copies of
    the library in one process."""
    import shutil
    import subprocess

    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", gbuild.LIB_PATH], capture_output=True, text=True, check=True)
    names = {line.split()[-1] for line in out.stdout.splitlines() if line.strip()}
    assert names == set(declared_functions())


def test_status_strings_and_version(L):
    for code, name in gdn.STATUS.items():
        assert L.gdn_status_string(code).decode().startswith(name)
    assert L.gdn_status_string(99).decode() == "unknown gdn_status"
    assert L.gdn_abi_version() == 1
    assert L.gdn_last_cuda_error() == 0


# fake, aligned, never dereferenced device addresses: validation fails before any CUDA call
P = ctypes.c_void_p(0x10000)
P2 = ctypes.c_void_p(0x20000)
ODD = ctypes.c_void_p(0x10002)


def dims(**kw):
    base = dict(B=4, T=4, HK=2, HV=4, DK=128, DV=128, num_slots=8, qkv_dtype=1, state_dtype=1, out_dtype=1,
                scale=1.0, l2_eps=1e-6)
    base.update(kw)
    return gdn.GdnDims(**base)


def verify(L, d, **ptrs):
    a = dict(q=P, k=P, v=P, a=P, b=P, A_log=P, dt_bias=P, pool=P2, idx=P, o=P, cache=None, err=None)
    a.update(ptrs)
    return L.gdn_mtp_verify(ctypes.byref(d) if d is not None else None, a["q"], a["k"], a["v"], a["a"], a["b"],
                            a["A_log"], a["dt_bias"], a["pool"], a["idx"], a["o"], a["cache"], a["err"], None)


def decode(L, d, **ptrs):
    a = dict(q=P, k=P, v=P, a=P, b=P, A_log=P, dt_bias=P, pool=P2, idx=P, o=P, err=None)
    a.update(ptrs)
    return L.gdn_decode(ctypes.byref(d) if d is not None else None, a["q"], a["k"], a["v"], a["a"], a["b"],
                        a["A_log"], a["dt_bias"], a["pool"], a["idx"], a["o"], a["err"], None)


def commit(L, d, **ptrs):
    a = dict(pool=P2, idx=P, cache=P, acc=P, err=None)
    a.update(ptrs)
    return L.gdn_commit(ctypes.byref(d) if d is not None else None, a["pool"], a["idx"], a["cache"], a["acc"],
                        a["err"], None)


def replay(L, d, **ptrs):
    a = dict(q=P, k=P, v=P, a=P, b=P, A_log=P, dt_bias=P, pool=P2, idx=P, acc=P, err=None)
    a.update(ptrs)
    return L.gdn_commit_replay(ctypes.byref(d) if d is not None else None, a["q"], a["k"], a["v"], a["a"], a["b"],
                               a["A_log"], a["dt_bias"], a["pool"], a["idx"], a["acc"], a["err"], None)


@pytest.mark.parametrize("ptr", ["q", "k", "v", "a", "b", "A_log", "dt_bias", "pool", "idx", "acc"])
def test_replay_null_pointer(L, ptr):
    assert replay(L, dims(), **{ptr: None}) == 1


def test_replay_checks(L):
    assert replay(L, None) == 1
    assert replay(L, dims(T=0)) == 2
    assert replay(L, dims(DK=48)) == 5
    assert replay(L, dims(l2_eps=-1.0)) == 7
    assert replay(L, dims(), q=ODD) == 4
    assert replay(L, dims(), acc=ctypes.c_void_p(0x10002)) == 4
    z = dict(q=None, k=None, v=None, a=None, b=None, A_log=None, dt_bias=None, pool=None, idx=None, acc=None)
    assert replay(L, dims(B=0), **z) == 0


@pytest.mark.parametrize("call", [verify, decode, commit, replay])
def test_null_dims(L, call):
    assert call(L, None) == 1


@pytest.mark.parametrize("call", [verify, decode])
@pytest.mark.parametrize("ptr", ["q", "k", "v", "a", "b", "A_log", "dt_bias", "pool", "idx", "o"])
def test_null_pointer(L, call, ptr):
    assert call(L, dims(), **{ptr: None}) == 1


@pytest.mark.parametrize("ptr", ["pool", "idx", "cache", "acc"])
def test_commit_null_pointer(L, ptr):
    assert commit(L, dims(), **{ptr: None}) == 1


@pytest.mark.parametrize("kw,status", [
    (dict(T=0), 2), (dict(T=17), 2), (dict(B=-1), 2), (dict(B=65536), 2), (dict(HK=3), 2), (dict(HK=0), 2),
    (dict(HV=0), 2), (dict(DV=0), 2), (dict(num_slots=0), 2), (dict(DK=0), 2),
    (dict(DK=48), 5), (dict(DK=512), 5), (dict(DK=8), 5),
    (dict(qkv_dtype=2), 3), (dict(state_dtype=-1), 3), (dict(out_dtype=7), 3),
    (dict(l2_eps=-1.0), 7), (dict(l2_eps=float("nan")), 7), (dict(scale=float("inf")), 7),
])
def test_bad_dims(L, kw, status):
    assert verify(L, dims(**kw)) == status
    assert decode(L, dims(**kw)) == status
    assert replay(L, dims(**kw)) == status


def test_commit_ignores_io_fields_but_checks_the_rest(L):
    assert commit(L, dims(HK=3, qkv_dtype=9, l2_eps=-1.0, B=0)) == 0
    assert commit(L, dims(T=0)) == 2
    assert commit(L, dims(state_dtype=5)) == 3
    assert commit(L, dims(DK=24)) == 5


@pytest.mark.parametrize("ptr", ["q", "k", "pool"])
def test_misaligned_16(L, ptr):
    assert verify(L, dims(), **{ptr: ODD}) == 4
    assert decode(L, dims(), **{ptr: ODD}) == 4


def test_misaligned_other(L):
    assert verify(L, dims(), cache=ODD) == 4
    assert verify(L, dims(), A_log=ctypes.c_void_p(0x10002)) == 4
    assert verify(L, dims(qkv_dtype=0), v=ctypes.c_void_p(0x10002)) == 4
    assert verify(L, dims(out_dtype=0), o=ctypes.c_void_p(0x10002)) == 4
    assert verify(L, dims(), err=ctypes.c_void_p(0x10001)) == 4
    assert commit(L, dims(), cache=ODD) == 4
    assert commit(L, dims(), pool=ODD) == 4
    assert commit(L, dims(), acc=ctypes.c_void_p(0x10001)) == 4


def test_empty_batch_is_a_no_op(L):
    # B == 0: nothing is enqueued, so even NULL data pointers are accepted
    z = dict(q=None, k=None, v=None, a=None, b=None, A_log=None, dt_bias=None, pool=None, idx=None, o=None)
    assert verify(L, dims(B=0), **z) == 0
    assert decode(L, dims(B=0), **z) == 0
    assert commit(L, dims(B=0), pool=None, idx=None, cache=None, acc=None) == 0


def test_binding_refuses_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(gdn, "_lib_handle", None)
    monkeypatch.setattr(gdn, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        gdn.lib()


# ---- prefill and the gated norm: host-side checks (status before any CUDA call) --------------------------
def prefill(L, d, **ptrs):
    a = dict(cu=P, q=P, k=P, v=P, a=P, b=P, A_log=P, dt_bias=P, pool=P2, idx=P, init=None, o=P, err=None)
    a.update(ptrs)
    return L.gdn_prefill(ctypes.byref(d) if d is not None else None, a["cu"], a["q"], a["k"], a["v"], a["a"],
                         a["b"], a["A_log"], a["dt_bias"], a["pool"], a["idx"], a["init"], a["o"], a["err"], None)


def test_prefill_host_validation(L):
    assert prefill(L, None) == 1
    assert prefill(L, dims(T=-1)) == 2                      # T is the total token count: >= 0
    assert prefill(L, dims(B=0, T=100)) == 0                # no sequences: nothing enqueued
    assert prefill(L, dims(B=4, T=0)) == 0                  # no tokens: nothing enqueued
    assert prefill(L, dims(T=100), cu=None) == 1
    assert prefill(L, dims(T=100), o=None) == 1
    assert prefill(L, dims(T=100), init=ODD) == 4
    assert prefill(L, dims(T=100), cu=ODD) == 4
    assert prefill(L, dims(T=100), q=ODD) == 4
    assert prefill(L, dims(T=100, HV=3)) == 2               # HV % HK
    assert prefill(L, dims(T=100, DK=48)) == 5
    assert prefill(L, dims(T=100, qkv_dtype=7)) == 3
    assert prefill(L, dims(T=100, l2_eps=-1.0)) == 7


def norm(L, rows=16, DV=128, od=1, zd=1, o=P, z=P, w=P, eps=1e-6, y=P2):
    return L.gdn_gated_rmsnorm(rows, DV, od, zd, o, z, w, ctypes.c_float(eps), y, None)


def test_gated_rmsnorm_host_validation(L):
    assert norm(L, rows=-1) == 2
    assert norm(L, DV=0) == 2
    assert norm(L, rows=1 << 60) == 2                       # beyond the launchable row count
    assert norm(L, od=2) == 3 and norm(L, zd=-1) == 3
    assert norm(L, eps=-1e-3) == 7 and norm(L, eps=float("inf")) == 7 and norm(L, eps=float("nan")) == 7
    assert norm(L, rows=0, o=None, z=None, w=None, y=None) == 0
    assert norm(L, o=None) == 1 and norm(L, z=None) == 1 and norm(L, w=None) == 1 and norm(L, y=None) == 1
    assert norm(L, o=ctypes.c_void_p(0x10001)) == 4         # bf16 o on an odd address
    assert norm(L, od=0, o=ODD) == 4                        # fp32 o on 2 bytes
    assert norm(L, w=ODD) == 4


# ---- the Python binding rejects bad shapes and dtypes before taking any pointer (CPU tensors suffice) -----
def test_binding_prefill_and_norm_argument_checks():
    import torch

    N, HK, HV, DK, DV = 10, 2, 4, 16, 8
    bf = torch.bfloat16
    q, v, ab = torch.zeros(N, HK, DK, dtype=bf), torch.zeros(N, HV, DV, dtype=bf), torch.zeros(N, HV, dtype=bf)
    A, pool = torch.zeros(HV), torch.zeros(3, HV, DV, DK, dtype=bf)
    o, cu = torch.zeros(N, HV, DV, dtype=bf), torch.tensor([0, 4, 10], dtype=torch.int32)
    idx = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(TypeError):
        gdn.gdn_prefill(q, q, v, ab, ab, A, A, pool, idx.long(), cu, o)
    with pytest.raises(ValueError):
        gdn.gdn_prefill(q, q, v, ab, ab, A, A, pool, torch.zeros(3, dtype=torch.int32), cu, o)
    with pytest.raises(TypeError):
        gdn.gdn_prefill(q, q, v, ab, ab, A, A, pool, idx, cu.long(), o)
    with pytest.raises(ValueError):
        gdn.gdn_prefill(q.unsqueeze(0), q, v, ab, ab, A, A, pool, idx, cu, o)  # [B, T, ...] layout: not packed
    with pytest.raises(ValueError):
        gdn.gdn_prefill(q, q, v, ab, ab, A, A, pool, idx, cu, o[:5])
    with pytest.raises(TypeError):
        gdn.gdn_prefill(q, q, v, ab, ab, A, A, pool, idx, cu, o, torch.ones(2, dtype=torch.bool))
    z = torch.zeros(N * HV, DV, dtype=bf)
    with pytest.raises(ValueError):
        gdn.gdn_gated_rmsnorm(z, z[:3], torch.ones(DV))
    with pytest.raises(TypeError):
        gdn.gdn_gated_rmsnorm(z, z, torch.ones(DV, dtype=bf))
    with pytest.raises(ValueError):
        gdn.gdn_gated_rmsnorm(z, z, torch.ones(DV + 1))
    with pytest.raises(TypeError):
        gdn.gdn_gated_rmsnorm(z, z, torch.ones(DV), torch.zeros(N * HV, DV))


# ---- every tensor of a call on one GPU (checked before anything is launched; fakes stand in for GPUs) ------
class _OnDevice:
    """A CPU tensor that reports itself as living on the given CUDA device (never dereferenced: the check
    under test rejects the call first)."""

    is_cuda = True

    def __init__(self, t, device):
        import torch

        self._t, self.device = t, torch.device(device)

    def __getattr__(self, name):
        return getattr(self._t, name)


class _FakeStream:
    def __init__(self, device):
        import torch

        self.device, self.cuda_stream = torch.device(device), 0


def _verify_args(dev_of):
    import torch

    B, T, HK, HV, DK, DV = 2, 3, 1, 2, 16, 16
    bf = torch.bfloat16
    t = dict(q=torch.zeros(B, T, HK, DK, dtype=bf), k=torch.zeros(B, T, HK, DK, dtype=bf),
             v=torch.zeros(B, T, HV, DV, dtype=bf), a=torch.zeros(B, T, HV, dtype=bf),
             b=torch.zeros(B, T, HV, dtype=bf), A_log=torch.zeros(HV), dt_bias=torch.zeros(HV),
             pool=torch.zeros(4, HV, DV, DK, dtype=bf), idx=torch.zeros(B, dtype=torch.int32),
             o=torch.zeros(B, T, HV, DV, dtype=bf), acc=torch.ones(B, dtype=torch.int32),
             cache=torch.zeros(B, T, HV, DV, DK, dtype=bf))
    return {k: _OnDevice(x, dev_of(k)) for k, x in t.items()}


def test_binding_common_device_helper():
    import torch

    a, b = _OnDevice(torch.zeros(1), "cuda:0"), _OnDevice(torch.zeros(1), "cuda:1")
    assert gdn._common_device([("a", a), ("skipped", None), ("a2", a)]) == torch.device("cuda:0")
    with pytest.raises(ValueError, match="same GPU"):
        gdn._common_device([("a", a), ("b", b)])
    with pytest.raises(ValueError, match="CUDA tensor"):
        gdn._common_device([("a", a), ("cpu", torch.zeros(1))])


@pytest.mark.parametrize("odd", ["q", "v", "pool", "idx", "o", "cache", "acc"])
def test_binding_rejects_tensors_on_two_gpus(odd):
    x = _verify_args(lambda k: "cuda:1" if k == odd else "cuda:0")
    with pytest.raises(ValueError, match="same GPU"):
        if odd == "acc":
            gdn.gdn_commit(x["pool"], x["idx"], x["cache"], x["acc"])
        else:
            gdn.gdn_mtp_verify(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"], x["dt_bias"], x["pool"],
                               x["idx"], x["o"], x["cache"])
    if odd in ("pool", "idx", "acc", "cache"):
        with pytest.raises(ValueError, match="same GPU"):
            gdn.gdn_commit(x["pool"], x["idx"], x["cache"], x["acc"])


def test_binding_rejects_a_stream_of_another_gpu():
    x = _verify_args(lambda k: "cuda:0")
    with pytest.raises(ValueError, match="stream is on cuda:1"):
        gdn.gdn_mtp_verify(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"], x["dt_bias"], x["pool"], x["idx"],
                           x["o"], None, stream=_FakeStream("cuda:1"))


# ---- gdn_mtp_verify_commit: the earlier call's tokens are checked like the others ---------------------------
def verify_commit(L, d, prev_T=4, prev=True, **ptrs):
    a = dict(q=P, k=P, v=P, a=P, b=P, A_log=P, dt_bias=P, pool=P2, idx=P, o=P, err=None, pk=P, pv=P, pa=P, pb=P, acc=P)
    a.update(ptrs)
    rt = gdn._ReplayTokensC(prev_T, a["pk"], a["pv"], a["pa"], a["pb"], a["acc"])
    return L.gdn_mtp_verify_commit(ctypes.byref(d) if d is not None else None, ctypes.byref(rt) if prev else None,
                                   a["q"], a["k"], a["v"], a["a"], a["b"], a["A_log"], a["dt_bias"], a["pool"],
                                   a["idx"], a["o"], None, a["err"], None)


@pytest.mark.parametrize("ptr", ["q", "k", "v", "a", "b", "A_log", "dt_bias", "pool", "idx", "o", "pk", "pv", "pa",
                                 "pb", "acc"])
def test_verify_commit_null_pointer(L, ptr):
    assert verify_commit(L, dims(), **{ptr: None}) == 1


def test_verify_commit_checks(L):
    assert verify_commit(L, None) == 1
    assert verify_commit(L, dims(), prev=False) == 1
    assert verify_commit(L, dims(), prev_T=0) == 2
    assert verify_commit(L, dims(), prev_T=17) == 2
    assert verify_commit(L, dims(T=0)) == 2
    assert verify_commit(L, dims(DK=48)) == 5
    assert verify_commit(L, dims(), pk=ODD) == 4          # the earlier k starts on 16 bytes
    assert verify_commit(L, dims(), acc=ODD) == 4
    assert verify_commit(L, dims(qkv_dtype=0), pv=ctypes.c_void_p(0x10002)) == 4  # fp32 v on 2 bytes
    z = {k: None for k in ("q", "k", "v", "a", "b", "A_log", "dt_bias", "pool", "idx", "o", "pk", "pv", "pa", "pb",
                           "acc")}
    assert verify_commit(L, dims(B=0), **z) == 0


# ---- gdn_mtp_verify_gated: the verify's checks plus the norm record's ------------------------------------
def verify_gated(L, d, norm=True, **ptrs):
    a = dict(q=P, k=P, v=P, a=P, b=P, A_log=P, dt_bias=P, pool=P2, idx=P, o=P, cache=None, err=None, z=P, w=P, y=P,
             zd=1, eps=1e-6)
    a.update(ptrs)
    n = gdn._GatedNormC(a["z"], a["zd"], a["w"], a["eps"], a["y"])
    return L.gdn_mtp_verify_gated(ctypes.byref(d) if d is not None else None, a["q"], a["k"], a["v"], a["a"], a["b"],
                                  a["A_log"], a["dt_bias"], a["pool"], a["idx"], a["o"], a["cache"],
                                  ctypes.byref(n) if norm else None, a["err"], None)


@pytest.mark.parametrize("ptr", ["q", "k", "v", "a", "b", "A_log", "dt_bias", "pool", "idx", "o", "z", "w", "y"])
def test_verify_gated_null_pointer(L, ptr):
    assert verify_gated(L, dims(), **{ptr: None}) == 1


def test_verify_gated_checks(L):
    assert verify_gated(L, dims(), norm=False) == 1
    assert verify_gated(L, dims(), zd=7) == 3
    assert verify_gated(L, dims(), eps=-1.0) == 7
    assert verify_gated(L, dims(), eps=float("nan")) == 7
    assert verify_gated(L, dims(), y=ctypes.c_void_p(0x10001)) == 4  # bf16 y on an odd address
    assert verify_gated(L, dims(), w=ctypes.c_void_p(0x10002)) == 4
    assert verify_gated(L, dims(), zd=0, z=ctypes.c_void_p(0x10002)) == 4  # fp32 z on 2 bytes
    assert verify_gated(L, dims(T=0)) == 2
    z = {k: None for k in ("q", "k", "v", "a", "b", "A_log", "dt_bias", "pool", "idx", "o")}
    assert verify_gated(L, dims(B=0), **z) == 0


# ---- gdn_decode_gated: the decode's checks plus the norm record's ------------------------------------------
def decode_gated(L, d, norm=True, **ptrs):
    a = dict(q=P, k=P, v=P, a=P, b=P, A_log=P, dt_bias=P, pool=P2, idx=P, o=P, err=None, z=P, w=P, y=P, zd=1,
             eps=1e-6)
    a.update(ptrs)
    n = gdn._GatedNormC(a["z"], a["zd"], a["w"], a["eps"], a["y"])
    return L.gdn_decode_gated(ctypes.byref(d) if d is not None else None, a["q"], a["k"], a["v"], a["a"], a["b"],
                              a["A_log"], a["dt_bias"], a["pool"], a["idx"], a["o"],
                              ctypes.byref(n) if norm else None, a["err"], None)


@pytest.mark.parametrize("ptr", ["q", "k", "v", "a", "b", "A_log", "dt_bias", "pool", "idx", "o", "z", "w", "y"])
def test_decode_gated_null_pointer(L, ptr):
    assert decode_gated(L, dims(), **{ptr: None}) == 1


def test_decode_gated_checks(L):
    assert decode_gated(L, None) == 1
    assert decode_gated(L, dims(), norm=False) == 1
    assert decode_gated(L, dims(), zd=7) == 3
    assert decode_gated(L, dims(), eps=-1.0) == 7
    assert decode_gated(L, dims(), y=ctypes.c_void_p(0x10001)) == 4  # bf16 y on an odd address
    assert decode_gated(L, dims(), w=ctypes.c_void_p(0x10002)) == 4
    assert decode_gated(L, dims(), pool=ctypes.c_void_p(0x10008)) == 4  # the pool is read in 16-byte pieces
    assert decode_gated(L, dims(T=0)) == 2
    z = {k: None for k in ("q", "k", "v", "a", "b", "A_log", "dt_bias", "pool", "idx", "o")}
    assert decode_gated(L, dims(B=0), **z) == 0


# ---- gdn_in_proj_conv / gdn_conv_commit: host validation (nothing reaches a kernel) ---------------------------
def conv_dims(**kw):
    base = dict(B=4, T=4, H=2048, HK=16, HV=32, DK=128, DV=128, K=4, num_slots=8, conv_dtype=1, out_dtype=1, silu=1)
    base.update(kw)
    return gdn._ConvDimsC(**base)


def in_proj(L, d, out=True, **ptrs):
    a = dict(x=P2, W=P2, conv_w=P, conv_b=None, state=P, idx=P, write=1, q=P, k=P, v=P, z=P, b=P, a=P, rec=None,
             err=None)
    a.update(ptrs)
    o = gdn._InProjOutC(a["q"], a["k"], a["v"], a["z"], a["b"], a["a"])
    return L.gdn_in_proj_conv(ctypes.byref(d) if d is not None else None, a["x"], a["W"], a["conv_w"], a["conv_b"],
                              a["state"], a["idx"], a["write"], ctypes.byref(o) if out else None, a["rec"], a["err"],
                              None)


def conv_commit(L, d, **ptrs):
    a = dict(state=P, idx=P, rec=P, acc=P, err=None)
    a.update(ptrs)
    return L.gdn_conv_commit(ctypes.byref(d) if d is not None else None, a["state"], a["idx"], a["rec"], a["acc"],
                             a["err"], None)


@pytest.mark.parametrize("ptr", ["x", "W", "conv_w", "state", "idx", "q", "k", "v", "z", "b", "a"])
def test_in_proj_null_pointer(L, ptr):
    assert in_proj(L, conv_dims(), **{ptr: None}) == 1


def test_in_proj_checks(L):
    assert in_proj(L, None) == 1
    assert in_proj(L, conv_dims(), out=False) == 1
    assert in_proj(L, conv_dims(K=1)) == 2 and in_proj(L, conv_dims(K=5)) == 2
    assert in_proj(L, conv_dims(H=100)) == 2 and in_proj(L, conv_dims(H=0)) == 2  # H % 8 != 0, H < 8
    assert in_proj(L, conv_dims(T=0)) == 2 and in_proj(L, conv_dims(T=17)) == 2
    assert in_proj(L, conv_dims(HV=24, HK=16)) == 2                                # HV % HK != 0
    assert in_proj(L, conv_dims(HK=1, DK=1 << 23)) == 2                            # channels beyond the grid
    assert in_proj(L, conv_dims(conv_dtype=5)) == 3 and in_proj(L, conv_dims(out_dtype=2)) == 3
    assert in_proj(L, conv_dims(silu=2)) == 7 and in_proj(L, conv_dims(), write=3) == 7
    assert in_proj(L, conv_dims(), x=ctypes.c_void_p(0x10008)) == 4               # x and W by TMA: 16 bytes
    assert in_proj(L, conv_dims(), W=ctypes.c_void_p(0x10004)) == 4
    assert in_proj(L, conv_dims(), conv_w=ctypes.c_void_p(0x10002)) == 4
    assert in_proj(L, conv_dims(), state=ctypes.c_void_p(0x10001)) == 4           # bf16 state on an odd address
    assert in_proj(L, conv_dims(), rec=ctypes.c_void_p(0x10001)) == 4
    assert in_proj(L, conv_dims(out_dtype=0), v=ctypes.c_void_p(0x10002)) == 4    # fp32 v on 2 bytes
    z = {k: None for k in ("x", "W", "conv_w", "state", "idx", "q", "k", "v", "z", "b", "a")}
    assert in_proj(L, conv_dims(B=0), out=False, **z) == 0                        # nothing to do, nothing read


def test_conv_commit_checks(L):
    assert conv_commit(L, None) == 1
    for p in ("state", "idx", "rec", "acc"):
        assert conv_commit(L, conv_dims(), **{p: None}) == 1
    assert conv_commit(L, conv_dims(K=5)) == 2
    assert conv_commit(L, conv_dims(conv_dtype=9)) == 3
    assert conv_commit(L, conv_dims(H=3, out_dtype=9, silu=5)) != 2                # the commit reads neither
    assert conv_commit(L, conv_dims(), acc=ctypes.c_void_p(0x10002)) == 4
    assert conv_commit(L, conv_dims(B=0), state=None, idx=None, rec=None, acc=None) == 0


# ---- gdn_in_proj_conv / gdn_conv_commit bindings: shapes, dtypes and devices checked before any launch --------
def _in_proj_args(dev_of=lambda k: "cuda:0", **shape):
    import torch

    s = dict(B=2, T=3, H=64, HK=1, HV=2, DK=16, DV=16, K=4, slots=4)
    s.update(shape)
    B, T, H, HK, HV, DK, DV, K = (s[k] for k in ("B", "T", "H", "HK", "HV", "DK", "DV", "K"))
    Cc = 2 * HK * DK + HV * DV
    C = Cc + HV * DV + 2 * HV
    bf = torch.bfloat16
    t = dict(x=torch.zeros(B, T, H, dtype=bf), W=torch.zeros(C, H, dtype=bf), conv_w=torch.zeros(Cc, K),
             conv_b=torch.zeros(Cc), state=torch.zeros(s["slots"], K - 1, Cc, dtype=bf),
             idx=torch.zeros(B, dtype=torch.int32), q=torch.zeros(B, T, HK, DK, dtype=bf),
             k=torch.zeros(B, T, HK, DK, dtype=bf), v=torch.zeros(B, T, HV, DV, dtype=bf),
             z=torch.zeros(B, T, HV, DV, dtype=bf), b=torch.zeros(B, T, HV, dtype=bf), a=torch.zeros(B, T, HV, dtype=bf),
             rec=torch.zeros(B, T, Cc, dtype=bf), acc=torch.ones(B, dtype=torch.int32))
    return {k: _OnDevice(x, dev_of(k)) for k, x in t.items()}


def _in_proj(x, **kw):
    out = gdn.InProjOut(x["q"], x["k"], x["v"], x["z"], x["b"], x["a"])
    gdn.gdn_in_proj_conv(x["x"], x["W"], x["conv_w"], x["conv_b"], x["state"], x["idx"], out, False, x["rec"], **kw)


def test_in_proj_binding_checks_shapes_and_dtypes():
    import torch

    x = _in_proj_args()
    x["W"] = _OnDevice(torch.zeros(7, 64, dtype=torch.bfloat16), "cuda:0")
    with pytest.raises(ValueError, match="W: shape"):
        _in_proj(x)
    x = _in_proj_args()
    x["v"] = _OnDevice(torch.zeros(2, 3, 2, 8, dtype=torch.bfloat16), "cuda:0")  # v's DV disagrees with W's C
    with pytest.raises(ValueError, match="shape"):
        _in_proj(x)
    x = _in_proj_args()
    x["x"] = _OnDevice(torch.zeros(2, 3, 64), "cuda:0")
    with pytest.raises(TypeError, match="x must be bf16"):
        _in_proj(x)
    x = _in_proj_args()
    x["z"] = _OnDevice(torch.zeros(2, 3, 2, 16), "cuda:0")
    with pytest.raises(TypeError, match="z must have q's dtype"):
        _in_proj(x)
    x = _in_proj_args()
    x["rec"] = _OnDevice(torch.zeros(2, 3, 64), "cuda:0")
    with pytest.raises(TypeError, match="records must have conv_state's dtype"):
        _in_proj(x)
    x = _in_proj_args()
    x["state"] = _OnDevice(torch.zeros(4, 2, 64, dtype=torch.bfloat16), "cuda:0")  # K - 1 rows disagree with conv_w
    with pytest.raises(ValueError, match="conv_state: shape"):
        _in_proj(x)


@pytest.mark.parametrize("odd", ["x", "W", "state", "idx", "q", "a", "rec"])
def test_in_proj_binding_rejects_tensors_on_two_gpus(odd):
    x = _in_proj_args(lambda k: "cuda:1" if k == odd else "cuda:0")
    with pytest.raises(ValueError, match="same GPU"):
        _in_proj(x)


def test_conv_commit_binding_checks():
    import torch

    x = _in_proj_args()
    with pytest.raises(ValueError, match="same GPU"):
        gdn.gdn_conv_commit(x["state"], x["idx"], x["rec"], _OnDevice(torch.ones(2, dtype=torch.int32), "cuda:1"))
    with pytest.raises(TypeError, match="accept_len must be int32"):
        gdn.gdn_conv_commit(x["state"], x["idx"], x["rec"], _OnDevice(torch.ones(2), "cuda:0"))
    with pytest.raises(ValueError, match="conv_state: shape"):
        gdn.gdn_conv_commit(_OnDevice(torch.zeros(4, 3, 63, dtype=torch.bfloat16), "cuda:0"), x["idx"], x["rec"],
                            x["acc"])
