"""Seeded synthetic inputs for the NVFP4 linear workloads.

This module is shared by the CUDA path's tests/benchmark and by the CPU
oracle's tests.  It holds input generation only -- shapes, distributions and
seeds -- and none of the quantisation, GEMM or epilogue arithmetic.

The shapes follow the four H3 projections the pages profile ("H3 Runtime
Current State", section "Owned Performance Kernels": QKV, attention output,
FC1, FC2) at the sizes of the synthetic workload set; the pages' real block
activations are not available, so these seeded tensors stand in for them.

Every tensor of a workload is drawn from numpy's PCG64 generator seeded with
``SeedSequence([base_seed, tensor_index])``; bf16 values are fp32 samples
rounded to nearest-even (bit patterns returned as uint16).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    N: int
    base_seed: int
    modulation: bool      # AdaLN prologue x*(1+scale)+shift
    gate_resid: bool      # epilogue out = R + g*(y + b)
    ragged: bool          # packed video+audio segments
    description: str


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 256, 512, 1024, 0, False, False, False,
                     "tiny NVFP4 linear, 0.1% x20 outliers, bias, no prologue"),
    "qkv": Workload("qkv", 8192, 3072, 9216, 1, True, False, False,
                    "QKV projection with AdaLN prologue and bias"),
    "fc1": Workload("fc1", 32768, 3072, 12288, 2, True, False, False,
                    "MLP FC1, Student-t(4) channels in 1% of columns, prologue, bias"),
    "fc2": Workload("fc2", 32768, 12288, 3072, 3, False, True, False,
                    "MLP FC2, |N(0,0.5)| input, bias + residual gate"),
    "attn_out": Workload("attn_out", 31744, 3072, 3072, 4, True, True, True,
                         "ragged video(30720)+audio(1024) attention-output projection, "
                         "per-modality shift/scale/gate, bias + residual gate"),
}

# Tensor indices inside a workload's seed space.
T_X, T_W, T_BIAS, T_SHIFT, T_SCALE, T_RESID, T_GATE, T_EXTRA = range(8)


def rng_for(base_seed: int, tensor: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([base_seed, tensor])))


def to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """fp32 samples -> bf16 bit patterns, round to nearest even (input prep)."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    u = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def segment_offsets(wl: Workload, M: int):
    """Row segments: [0, M) or, for the ragged workload, video rows then audio rows.

    At the full size the split is 30720 + 1024; reduced sizes keep the same
    audio fraction (at least one audio row) so the boundary stays ragged.
    """
    if not wl.ragged:
        return np.array([0, M], np.int64)
    audio = max(1, int(round(M * 1024 / 31744)))
    audio = min(audio, M - 1) if M > 1 else 0
    return np.array([0, M - audio, M], np.int64)


def make_x(wl: Workload, M: Optional[int] = None) -> np.ndarray:
    """Activation X [M, K] as bf16 bits."""
    M = wl.M if M is None else M
    K = wl.K
    g = rng_for(wl.base_seed, T_X)
    if wl.name == "fc2":
        x = np.abs(g.standard_normal((M, K), dtype=np.float32)) * np.float32(0.5)
    else:
        x = g.standard_normal((M, K), dtype=np.float32)
    if wl.name == "tiny":
        # exactly round(0.001*M*K) entries, without replacement, scaled by 20
        n_out = int(round(0.001 * M * K))
        idx = rng_for(wl.base_seed, T_EXTRA).choice(M * K, size=n_out, replace=False)
        x.reshape(-1)[idx] *= np.float32(20.0)
    if wl.name == "fc1":
        # heavy-tailed channels: 1% of the columns drawn from Student-t(4)
        ge = rng_for(wl.base_seed, T_EXTRA)
        ncol = int(round(0.01 * K))
        cols = np.sort(ge.choice(K, size=ncol, replace=False))
        x[:, cols] = ge.standard_t(4.0, size=(M, ncol)).astype(np.float32)
    return to_bf16_bits(x)


def make_w(wl: Workload) -> np.ndarray:
    std = 0.01 if wl.name == "fc2" else 0.02
    g = rng_for(wl.base_seed, T_W)
    return to_bf16_bits(g.standard_normal((wl.N, wl.K), dtype=np.float32) * np.float32(std))


def make_inputs(name: str, M: Optional[int] = None, with_x: bool = True) -> dict:
    """All tensors of a workload (numpy, host).  ``M`` overrides the row count.

    Returns a dict with x (bf16 bits [M,K]), w (bf16 bits [N,K]),
    bias (bf16 bits [N]), shift/scale (fp32 [nseg,K] or None),
    gate (fp32 [nseg,N] or None), resid (bf16 bits [M,N] or None),
    seg_off (int64 [nseg+1]) and the Workload record.
    """
    wl = WORKLOADS[name]
    M = wl.M if M is None else M
    seg_off = segment_offsets(wl, M)
    nseg = len(seg_off) - 1
    out = dict(workload=wl, M=M, K=wl.K, N=wl.N, seg_off=seg_off)
    out["x"] = make_x(wl, M) if with_x else None
    out["w"] = make_w(wl)
    out["bias"] = to_bf16_bits(rng_for(wl.base_seed, T_BIAS).standard_normal(wl.N, dtype=np.float32)
                               * np.float32(0.01))
    if wl.modulation:
        out["shift"] = (rng_for(wl.base_seed, T_SHIFT).standard_normal((nseg, wl.K), dtype=np.float32)
                        * np.float32(0.1))
        out["scale"] = (rng_for(wl.base_seed, T_SCALE).standard_normal((nseg, wl.K), dtype=np.float32)
                        * np.float32(0.1))
    else:
        out["shift"] = out["scale"] = None
    if wl.gate_resid:
        out["gate"] = rng_for(wl.base_seed, T_GATE).uniform(0.0, 1.0, (nseg, wl.N)).astype(np.float32)
        out["resid"] = to_bf16_bits(rng_for(wl.base_seed, T_RESID).standard_normal((M, wl.N), dtype=np.float32))
    else:
        out["gate"] = out["resid"] = None
    return out


def m_sweep_inputs(M: int) -> dict:
    """M sweep point: K = N = 3072 with the attention-output value distributions
    and a single segment."""
    base = WORKLOADS["attn_out"]
    wl = dataclasses.replace(base, name=f"sweep_{M}", M=M, ragged=False)
    seg_off = np.array([0, M], np.int64)
    g = rng_for(base.base_seed + 100, T_X)
    out = dict(workload=wl, M=M, K=3072, N=3072, seg_off=seg_off)
    out["x"] = to_bf16_bits(g.standard_normal((M, 3072), dtype=np.float32))
    out["w"] = make_w(wl)
    out["bias"] = to_bf16_bits(rng_for(base.base_seed, T_BIAS).standard_normal(3072, dtype=np.float32)
                               * np.float32(0.01))
    out["shift"] = rng_for(base.base_seed, T_SHIFT).standard_normal((1, 3072), dtype=np.float32) * np.float32(0.1)
    out["scale"] = rng_for(base.base_seed, T_SCALE).standard_normal((1, 3072), dtype=np.float32) * np.float32(0.1)
    out["gate"] = rng_for(base.base_seed, T_GATE).uniform(0.0, 1.0, (1, 3072)).astype(np.float32)
    out["resid"] = to_bf16_bits(rng_for(base.base_seed, T_RESID).standard_normal((M, 3072), dtype=np.float32))
    return out


def swiglu_fc1_inputs(M: int, N: int = 24576, K: int = 3072) -> dict:
    """FC1 feeding FC2 through SwiGLU: X [M, K] with the fc1 distributions and
    modulation vectors, W [N, K] ~ N(0, 0.02^2) whose rows are read as groups of
    256 (128 gate rows, then the 128 matching up rows), bias [N] ~ N(0, 0.01^2).
    N = 24576 gives the hidden width 12288 that the fc2 workload consumes."""
    base = WORKLOADS["fc1"]
    wl = dataclasses.replace(base, name="fc1_swiglu", M=M, N=N, K=K)
    seg_off = np.array([0, M], np.int64)
    out = dict(workload=wl, M=M, K=K, N=N, seg_off=seg_off)
    out["x"] = make_x(dataclasses.replace(base, M=M, K=K), M)   # fc1's X recipe at this K
    g = rng_for(base.base_seed + 200, T_W)
    out["w"] = to_bf16_bits(g.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    out["bias"] = to_bf16_bits(rng_for(base.base_seed + 200, T_BIAS).standard_normal(N, dtype=np.float32)
                               * np.float32(0.01))
    out["shift"] = (rng_for(base.base_seed + 200, T_SHIFT).standard_normal((1, K), dtype=np.float32)
                    * np.float32(0.1))
    out["scale"] = (rng_for(base.base_seed + 200, T_SCALE).standard_normal((1, K), dtype=np.float32)
                    * np.float32(0.1))
    out["gate"] = out["resid"] = None
    return out
