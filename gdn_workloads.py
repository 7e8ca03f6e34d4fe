"""Seeded synthetic inputs for the Gated DeltaNet (GDN) decode / MTP-verify state update.

This module is shared by the CPU oracle side (``oracle/``, ``tests/``) and the CUDA side (``bench.py``,
the GPU tests).  It holds NO arithmetic of the method: it only draws random numbers, casts them to the
storage types and lays them out.  Both sides receive the same bytes.

Workload shapes follow the serving setups on the pages:

* T = 4 tokens per verify (three drafted tokens plus one) -- sglang PR #23273 "[GDN] Enable FlashInfer MTP
  verify on SM100+ (Blackwell)", launch command (``--speculative-num-steps 3 --speculative-num-draft-tokens
  4``);
* T = 8 (beyond 4, with intermediate caching) -- same page, Requirements (FlashInfer #2679);
* bf16 state pool (``--mamba-ssm-dtype bfloat16``) -- same page, Throughput Benchmark server settings;
* padded lanes carry pool index -1 -- same page, Requirements (FlashInfer #2810, padding index guard);
* concurrency up to 256 requests -- same page, Mean TPOT table.

Layouts (row-major, last index contiguous):

====================  =======================  ==============================
tensor                shape                    storage
====================  =======================  ==============================
q, k                  [B, T, HK, DK]           f32 or bf16 (``qkv_dtype``)
v                     [B, T, HV, DV]           f32 or bf16
a, b                  [B, T, HV]               same as q/k/v
A_log, dt_bias        [HV]                     f32
pool                  [num_slots, HV, DV, DK]  f32 or bf16 (``state_dtype``)
indices               [B]                      int32, -1 = padded lane
accept_len            [B]                      int32 in 1..T
====================  =======================  ==============================

bf16 arrays are returned as ``uint16`` bit patterns (round-to-nearest-even from the fp32 draw, done by
``torch``'s cast).  Every tensor has its own random stream, ``numpy.random.default_rng([seed, tensor_id])``,
so that a large tensor (the pool) can be drawn or skipped without changing the others.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List, Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"
POOL_BLOCK = 16  # slots per independent pool stream

# stream ids: one independent generator per tensor
_STREAM = {"q": 1, "k": 2, "v": 3, "a": 4, "b": 5, "dt_bias": 6, "A_log": 7, "pool": 8,
           "slots": 9, "pad": 10, "accept_len": 11, "lengths": 12, "fresh": 13, "z": 14, "norm_weight": 15,
           "x": 16, "W": 17, "conv_w": 18, "conv_b": 19, "conv_state": 20, "records": 21}


def _rng(seed: int, name: str) -> np.random.Generator:
    return np.random.default_rng([int(seed), _STREAM[name]])


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even, via torch's cast."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact widening)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == BF16:
        return to_bf16_bits(x)
    raise ValueError(dtype)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic GDN workload.  ``mode`` is ``"decode"`` (write-back, no cache) or ``"verify"``."""

    name: str
    B: int
    T: int
    HK: int
    HV: int
    DK: int
    DV: int
    num_slots: int
    qkv_dtype: str
    state_dtype: str
    out_dtype: str
    mode: str
    cache: bool
    commit: bool
    seed: int
    pool_std: float = 0.05
    pad_fraction: float = 0.0
    scale: float = 1.0
    l2_eps: float = 1e-6
    pool_seed: Optional[int] = None  # None: the pool is drawn from `seed`
    commit_mode: str = "copy"        # "copy": from the cached states; "replay": re-run the accepted tokens;
    #                                  "fused": commit the previous step's accepted tokens inside this step's verify

    @property
    def n_padded(self) -> int:
        return int(round(self.pad_fraction * self.B))

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    # -- draws -----------------------------------------------------------------------------------
    def small_arrays(self) -> Dict[str, np.ndarray]:
        """Everything except the pool."""
        B, T, HK, HV, DK, DV = self.B, self.T, self.HK, self.HV, self.DK, self.DV
        s = self.seed
        out: Dict[str, np.ndarray] = {}
        f32 = np.float32
        out["q"] = _store(_rng(s, "q").standard_normal((B, T, HK, DK), dtype=f32), self.qkv_dtype)
        out["k"] = _store(_rng(s, "k").standard_normal((B, T, HK, DK), dtype=f32), self.qkv_dtype)
        out["v"] = _store(_rng(s, "v").standard_normal((B, T, HV, DV), dtype=f32), self.qkv_dtype)
        out["a"] = _store(_rng(s, "a").standard_normal((B, T, HV), dtype=f32), self.qkv_dtype)
        out["b"] = _store(_rng(s, "b").standard_normal((B, T, HV), dtype=f32), self.qkv_dtype)
        out["dt_bias"] = _rng(s, "dt_bias").standard_normal(HV, dtype=f32)
        out["A_log"] = np.log(_rng(s, "A_log").uniform(1.0, 16.0, HV)).astype(f32)
        if B > self.num_slots:
            raise ValueError("more lanes than pool slots: distinct slots are impossible")
        slots = _rng(s, "slots").permutation(self.num_slots)[:B].astype(np.int32)
        if self.n_padded:
            pad = _rng(s, "pad").permutation(B)[: self.n_padded]
            slots[pad] = -1
        out["indices"] = slots
        out["accept_len"] = _rng(s, "accept_len").integers(1, T + 1, B).astype(np.int32)
        return out

    def pool(self) -> np.ndarray:
        """Pool ~ N(0, pool_std^2); drawn in blocks of POOL_BLOCK slots, each from its own stream
        ``default_rng([seed, pool_id, block])`` so that blocks can be filled by parallel threads."""
        shape = (self.num_slots, self.HV, self.DV, self.DK)
        seed = self.seed if self.pool_seed is None else self.pool_seed
        x = np.empty(shape, np.float32)
        nblk = (self.num_slots + POOL_BLOCK - 1) // POOL_BLOCK

        def fill(i: int) -> None:
            g = np.random.default_rng([int(seed), _STREAM["pool"], i])
            blk = x[i * POOL_BLOCK:(i + 1) * POOL_BLOCK]
            g.standard_normal(out=blk, dtype=np.float32)
            blk *= np.float32(self.pool_std)

        with ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1))) as ex:
            list(ex.map(fill, range(nblk)))
        return _store(x, self.state_dtype)

    def arrays(self) -> Dict[str, np.ndarray]:
        out = self.small_arrays()
        out["pool"] = self.pool()
        return out

    def active_lanes(self, indices: Optional[np.ndarray] = None) -> int:
        if indices is None:
            indices = self.small_arrays()["indices"]
        return int((indices >= 0).sum())


def tiny() -> Workload:
    """B=2, 4 slots, HK=HV=2, DK=DV=16, T=2, all fp32, pool ~ N(0, 0.1), seed 0."""
    return Workload("tiny_B2_T2_d16_f32", B=2, T=2, HK=2, HV=2, DK=16, DV=16, num_slots=4,
                    qkv_dtype=F32, state_dtype=F32, out_dtype=F32, mode="verify", cache=True,
                    commit=True, seed=0, pool_std=0.1)


def decode_t1() -> Workload:
    """Decode T=1: B=64, HK=16, HV=32, 128x128, bf16 q/k/v, fp32 pool of 256 slots ~ N(0, 0.05)."""
    return Workload("decode_T1_B64_f32state", B=64, T=1, HK=16, HV=32, DK=128, DV=128, num_slots=256,
                    qkv_dtype=BF16, state_dtype=F32, out_dtype=BF16, mode="decode", cache=False,
                    commit=False, seed=1)


def verify_t4() -> Workload:
    """MTP verify T=4 (3 drafts + 1): B=128, bf16 state pool of 512 slots, bf16 cache, then commit."""
    return Workload("mtp_verify_T4_B128_bf16state", B=128, T=4, HK=16, HV=32, DK=128, DV=128,
                    num_slots=512, qkv_dtype=BF16, state_dtype=BF16, out_dtype=BF16, mode="verify",
                    cache=True, commit=True, seed=2)


def verify_t8() -> Workload:
    """MTP verify T=8: B=256 with 10% padded lanes (index -1), bf16 pool of 1024 slots, cache, commit."""
    return Workload("mtp_verify_T8_B256_pad10_bf16state", B=256, T=8, HK=16, HV=32, DK=128, DV=128,
                    num_slots=1024, qkv_dtype=BF16, state_dtype=BF16, out_dtype=BF16, mode="verify",
                    cache=True, commit=True, seed=3, pad_fraction=0.1)


def verify_t4_replay() -> Workload:
    """verify_t4 without intermediate caching; the accepted prefix is committed by replaying it."""
    return verify_t4().replace(name="mtp_verify_T4_B128_bf16state_replay_commit", cache=False, commit_mode="replay")


def verify_t8_replay() -> Workload:
    """verify_t8 without intermediate caching; the accepted prefix is committed by replaying it."""
    return verify_t8().replace(name="mtp_verify_T8_B256_pad10_bf16state_replay_commit", cache=False,
                               commit_mode="replay")


def verify_t4_fused() -> Workload:
    """verify_t4 as one-pass steps: each verify first commits the previous step's accepted prefix
    (gdn_mtp_verify_commit); no intermediate states."""
    return verify_t4().replace(name="mtp_verify_T4_B128_bf16state_fused_commit", cache=False, commit_mode="fused")


def verify_t8_fused() -> Workload:
    """verify_t8 as one-pass steps (gdn_mtp_verify_commit); no intermediate states."""
    return verify_t8().replace(name="mtp_verify_T8_B256_pad10_bf16state_fused_commit", cache=False,
                               commit_mode="fused")


def previous_step(w: Workload) -> Dict[str, np.ndarray]:
    """The earlier verify of a one-pass step on the same lanes: its k, v, a, b (draws of seed + 1, same shapes)
    and accept lengths U{1..T} of its own stream."""
    x = w.replace(seed=w.seed + 1).small_arrays()
    return {k: x[k] for k in ("k", "v", "a", "b", "accept_len")}


SWEEP_B = (1, 4, 16, 64, 128, 256)
SWEEP_T = (1, 2, 4, 8)
SWEEP_STATE = (F32, BF16)


def sweep() -> List[Workload]:
    """B x T x state dtype; T=1 runs as decode, T>1 as verify with caching; pool 1024 slots.

    Point i draws its inputs from seed 1000 + i; all points of one state dtype share one pool (seed 2000
    for fp32, 2001 for bf16), so the sweep needs two pool draws instead of 48."""
    pts = []
    i = 0
    for st in SWEEP_STATE:
        for T in SWEEP_T:
            for B in SWEEP_B:
                dec = T == 1
                pts.append(Workload(f"sweep_B{B}_T{T}_{st}state", B=B, T=T, HK=16, HV=32, DK=128, DV=128,
                                    num_slots=1024, qkv_dtype=BF16, state_dtype=st, out_dtype=BF16,
                                    mode="decode" if dec else "verify", cache=not dec, commit=not dec,
                                    seed=1000 + i, pool_seed=2000 + SWEEP_STATE.index(st)))
                i += 1
    return pts


def sweep_replay() -> List[Workload]:
    """The verify + replay-commit path (no intermediate states) over B x T, bf16 state, pool 1024 slots:
    point i draws its inputs from seed 3000 + i; all points share the bf16 pool of the sweep (seed 2001)."""
    pts = []
    i = 0
    for T in (2, 4, 8):
        for B in (16, 64, 128, 256):
            pts.append(Workload(f"sweep_replay_B{B}_T{T}", B=B, T=T, HK=16, HV=32, DK=128, DV=128, num_slots=1024,
                                qkv_dtype=BF16, state_dtype=BF16, out_dtype=BF16, mode="verify", cache=False,
                                commit=True, seed=3000 + i, pool_seed=2001, commit_mode="replay"))
            i += 1
    return pts


def sweep_fused() -> List[Workload]:
    """The one-pass step (gdn_mtp_verify_commit) over the grid of sweep_replay, same seeds and pool."""
    return [w.replace(name=w.name.replace("sweep_replay", "sweep_fused"), commit_mode="fused") for w in sweep_replay()]


NAMED = {"tiny": tiny, "decode": decode_t1, "verify4": verify_t4, "verify8": verify_t8,
         "verify4_replay": verify_t4_replay, "verify8_replay": verify_t8_replay,
         "verify4_fused": verify_t4_fused, "verify8_fused": verify_t8_fused}


# ---- prefill ------------------------------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    """Prefill of B packed sequences into the pool.  Lengths: ``lengths`` if given, else uniform integers in
    [min_len, max_len] (seeded).  A ``fresh_fraction`` of the sequences has no initial state
    (has_initial_state = 0: a new request) and a ``pad_fraction`` carries index -1.

    Layouts: q, k [N, HK, DK]; v [N, HV, DV]; a, b [N, HV]; cu_seqlens [B+1]; has_initial_state [B] int32."""

    name: str
    B: int
    HK: int
    HV: int
    DK: int
    DV: int
    num_slots: int
    qkv_dtype: str
    state_dtype: str
    out_dtype: str
    seed: int
    min_len: int = 1
    max_len: int = 64
    lengths: Optional[tuple] = None
    fresh_fraction: float = 0.5
    pad_fraction: float = 0.0
    pool_std: float = 0.05
    scale: float = 1.0
    l2_eps: float = 1e-6

    def replace(self, **kw) -> "PrefillWorkload":
        return dataclasses.replace(self, **kw)

    def seq_lengths(self) -> np.ndarray:
        if self.lengths is not None:
            return np.asarray(self.lengths, np.int64)
        return _rng(self.seed, "lengths").integers(self.min_len, self.max_len + 1, self.B)

    @property
    def n_tokens(self) -> int:
        return int(self.seq_lengths().sum())

    def small_arrays(self) -> Dict[str, np.ndarray]:
        lens = self.seq_lengths()
        N, B, HK, HV, DK, DV, s = int(lens.sum()), self.B, self.HK, self.HV, self.DK, self.DV, self.seed
        f32 = np.float32
        out: Dict[str, np.ndarray] = {}
        out["q"] = _store(_rng(s, "q").standard_normal((N, HK, DK), dtype=f32), self.qkv_dtype)
        out["k"] = _store(_rng(s, "k").standard_normal((N, HK, DK), dtype=f32), self.qkv_dtype)
        out["v"] = _store(_rng(s, "v").standard_normal((N, HV, DV), dtype=f32), self.qkv_dtype)
        out["a"] = _store(_rng(s, "a").standard_normal((N, HV), dtype=f32), self.qkv_dtype)
        out["b"] = _store(_rng(s, "b").standard_normal((N, HV), dtype=f32), self.qkv_dtype)
        out["dt_bias"] = _rng(s, "dt_bias").standard_normal(HV, dtype=f32)
        out["A_log"] = np.log(_rng(s, "A_log").uniform(1.0, 16.0, HV)).astype(f32)
        if B > self.num_slots:
            raise ValueError("more sequences than pool slots")
        slots = _rng(s, "slots").permutation(self.num_slots)[:B].astype(np.int32)
        n_pad = int(round(self.pad_fraction * B))
        if n_pad:
            slots[_rng(s, "pad").permutation(B)[:n_pad]] = -1
        out["indices"] = slots
        out["cu_seqlens"] = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        init = np.ones(B, np.int32)
        n_fresh = int(round(self.fresh_fraction * B))
        if n_fresh:
            init[_rng(s, "fresh").permutation(B)[:n_fresh]] = 0
        out["has_initial_state"] = init
        return out

    def pool(self) -> np.ndarray:
        return Workload(self.name, B=0, T=1, HK=self.HK, HV=self.HV, DK=self.DK, DV=self.DV,
                        num_slots=self.num_slots, qkv_dtype=self.qkv_dtype, state_dtype=self.state_dtype,
                        out_dtype=self.out_dtype, mode="decode", cache=False, commit=False, seed=self.seed,
                        pool_std=self.pool_std).pool()

    def arrays(self) -> Dict[str, np.ndarray]:
        out = self.small_arrays()
        out["pool"] = self.pool()
        return out


def prefill_8k() -> PrefillWorkload:
    """Prefill at the ISL-8K serving point: 8 prompts of 8192 tokens (65,536 tokens), HK=16, HV=32, 128x128
    bf16 state pool of 64 slots, bf16 q/k/v/o, half of the prompts new (no initial state), half continuing
    from a cached state."""
    return PrefillWorkload("prefill_ISL8K_B8_bf16state", B=8, HK=16, HV=32, DK=128, DV=128, num_slots=64,
                           qkv_dtype=BF16, state_dtype=BF16, out_dtype=BF16, seed=4, lengths=(8192,) * 8,
                           fresh_fraction=0.5)


def prefill_mix() -> PrefillWorkload:
    """Prefill of 64 prompts of mixed length, uniform in [256, 4096] tokens, otherwise as prefill_8k."""
    return PrefillWorkload("prefill_mix256to4096_B64_bf16state", B=64, HK=16, HV=32, DK=128, DV=128,
                           num_slots=128, qkv_dtype=BF16, state_dtype=BF16, out_dtype=BF16, seed=5, min_len=256,
                           max_len=4096, fresh_fraction=0.5)


# ---- gated RMSNorm of the outputs ---------------------------------------------------------------------------
def gated_norm_inputs(rows: int, DV: int, o_dtype: str, z_dtype: str, seed: int) -> Dict[str, np.ndarray]:
    """o ~ N(0, 0.3^2) (the scale of the recurrence's outputs at the workloads above), gate z ~ N(0, 1),
    norm weight ~ 1 + N(0, 0.1^2); o and z [rows, DV] in their storage types, weight fp32 [DV]."""
    f32 = np.float32
    o = _rng(seed, "v").standard_normal((rows, DV), dtype=f32) * f32(0.3)
    z = _rng(seed, "z").standard_normal((rows, DV), dtype=f32)
    w = (1.0 + 0.1 * _rng(seed, "norm_weight").standard_normal(DV)).astype(f32)
    return {"o": _store(o, o_dtype), "z": _store(z, z_dtype), "w": w}



@dataclasses.dataclass(frozen=True)
class InProjWorkload:
    """Inputs of the in_proj projection with its causal conv1d epilogue (decode or verify rows).

    x ~ N(0, 1) [B, T, H] bf16 (normalised hidden states), W ~ N(0, 1/H) [C, H] bf16 (so that every projection
    is ~ N(0, 1)), conv taps and biases ~ U(-1/sqrt(K), 1/sqrt(K)) fp32 (the usual depthwise-convolution
    initialisation, fan-in K), convolution state ~ N(0, 1) [num_slots, K-1, Cc] (earlier projections), distinct
    slots with ``pad_fraction`` of the lanes at -1, accept lengths in 1..T; C and Cc as the interface defines
    them (q | k | v | z | b | a, and q | k | v).  No method arithmetic: draws, casts and layout only."""

    name: str
    B: int
    T: int
    H: int
    HK: int
    HV: int
    DK: int
    DV: int
    K: int
    num_slots: int
    conv_dtype: str
    out_dtype: str
    seed: int
    silu: bool = True
    pad_fraction: float = 0.0

    def replace(self, **kw) -> "InProjWorkload":
        return dataclasses.replace(self, **kw)

    @property
    def Cc(self) -> int:
        return 2 * self.HK * self.DK + self.HV * self.DV

    @property
    def C(self) -> int:
        return self.Cc + self.HV * self.DV + 2 * self.HV

    def arrays(self) -> Dict[str, np.ndarray]:
        B, T, H, K, s = self.B, self.T, self.H, self.K, self.seed
        f32 = np.float32
        out: Dict[str, np.ndarray] = {}
        out["x"] = _store(_rng(s, "x").standard_normal((B, T, H), dtype=f32), BF16)
        w = _rng(s, "W").standard_normal((self.C, H), dtype=f32)
        w *= f32(1.0 / np.sqrt(H))
        out["W"] = _store(w, BF16)
        bound = f32(1.0 / np.sqrt(K))
        out["conv_w"] = _rng(s, "conv_w").uniform(-bound, bound, (self.Cc, K)).astype(f32)
        out["conv_b"] = _rng(s, "conv_b").uniform(-bound, bound, self.Cc).astype(f32)
        out["conv_state"] = _store(_rng(s, "conv_state").standard_normal((self.num_slots, K - 1, self.Cc), dtype=f32),
                                   self.conv_dtype)
        if B > self.num_slots:
            raise ValueError("more lanes than slots: distinct slots are impossible")
        slots = _rng(s, "slots").permutation(self.num_slots)[:B].astype(np.int32)
        n_pad = int(round(self.pad_fraction * B))
        if n_pad:
            slots[_rng(s, "pad").permutation(B)[:n_pad]] = -1
        out["indices"] = slots
        out["accept_len"] = _rng(s, "accept_len").integers(1, T + 1, B).astype(np.int32)
        # recovery records of an earlier verify (inputs of the commit alone): earlier projections ~ N(0, 1)
        out["records"] = _store(_rng(s, "records").standard_normal((B, T, self.Cc), dtype=f32), self.conv_dtype)
        return out


def in_proj_verify16() -> InProjWorkload:
    """16 verify rows (B = 4 lanes x T = 4, the page's largest verify row count): hidden 2048, 16 key heads and 32
    value heads of 128 (the head layout of every workload above), 4 taps, bf16 state and outputs."""
    return InProjWorkload("in_proj_conv_verify_B4_T4_H2048", B=4, T=4, H=2048, HK=16, HV=32, DK=128, DV=128, K=4,
                          num_slots=64, conv_dtype=BF16, out_dtype=BF16, seed=500)


def in_proj_decode8() -> InProjWorkload:
    """8 decode rows (the page's largest decode row count), the rest as in_proj_verify16."""
    return in_proj_verify16().replace(name="in_proj_conv_decode_B8_T1_H2048", B=8, T=1, seed=501)


def in_proj_verify512() -> InProjWorkload:
    """The verify-T4 batch of 128 lanes (512 rows): the projection becomes a GEMM with two row tiles."""
    return in_proj_verify16().replace(name="in_proj_conv_verify_B128_T4_H2048", B=128, num_slots=512, seed=502)
