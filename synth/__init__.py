"""Seeded synthetic inputs for the routed-expert MoE FFN layer.

Both sides of every comparison (the CUDA library and the CPU oracle) draw
their inputs from here, so they see the same bytes.  Nothing in this module
computes any part of the layer: it only writes activations, router weights
and FP8 expert weights in the checkpoint format (E4M3FN codes plus one fp32
multiplier per 128x128 block) that the layer consumes.

The workload table below gives the shapes of the five layer configurations:
a tiny case, the DeepSeek-V3-shaped decode and 8K prefill layers, a
Zipf-skewed 32K prefill layer and a Kimi-K2-shaped 64K prefill layer.  Shapes
follow the KTransformers deep dive (chenxutan.com, section 1.2: 256 routed
experts + 1 shared expert, 8 selected per token) and the CPU-GPU hybrid
inference article (xingyun.xin, SLP section: 3 FP8 linear modules of
7168x2048 per expert; ring-buffer passage: 11.3 GB per DeepSeek-V3 layer and
16.9 GB per Kimi-K2 layer, i.e. 384 experts).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "_synth.so")
_lock = threading.Lock()
_handle = None

# Stream ids: one independent counter stream per tensor.
STREAM_X, STREAM_ROUTER_W, STREAM_BIAS_PERM = 1, 2, 3
STREAM_GATE, STREAM_UP, STREAM_DOWN = 10, 11, 12
STREAM_SH_GATE, STREAM_SH_UP, STREAM_SH_DOWN = 20, 21, 22


def build(force: bool = False) -> str:
    """Compile synth.c into _synth.so next to it (OpenMP when available)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", _SRC, "-o", _SO + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_SO + ".tmp", _SO)
    return _SO


def _lib():
    global _handle
    with _lock:
        if _handle is None:
            lib = ctypes.CDLL(build())
            u64, i64, i32, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p
            lib.synth_bf16_normal.argtypes = [u64, u64, i64, dbl, vp]
            lib.synth_f32_normal.argtypes = [u64, u64, i64, dbl, vp]
            lib.synth_permutation.argtypes = [u64, u64, i32, vp]
            lib.synth_fp8_blocks.argtypes = [u64, u64, i32, i32, i32, dbl, vp, vp]
            lib.synth_fp8_blocks.restype = ctypes.c_int
            _handle = lib
    return _handle


def bf16_normal(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """bf16(std * N(0,1)) as raw uint16 bit patterns."""
    out = np.empty(shape, dtype=np.uint16)
    _lib().synth_bf16_normal(seed, stream, out.size, std, out.ctypes.data)
    return out


def f32_normal(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _lib().synth_f32_normal(seed, stream, out.size, std, out.ctypes.data)
    return out


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _lib().synth_permutation(seed, stream, n, out.ctypes.data)
    return out


def fp8_blocks(seed: int, stream: int, n_mat: int, rows: int, cols: int, std: float = 0.02):
    """FP8 E4M3FN codes [n_mat][rows][cols] and fp32 block multipliers
    [n_mat][rows/128][cols/128] of W = std * N(0,1) (s = amax/448 per block)."""
    q = np.empty((n_mat, rows, cols), dtype=np.uint8)
    s = np.empty((n_mat, rows // 128, cols // 128), dtype=np.float32)
    rc = _lib().synth_fp8_blocks(seed, stream, n_mat, rows, cols, std, q.ctypes.data, s.ctypes.data)
    if rc != 0:
        raise ValueError("rows and cols must be multiples of 128")
    return q, s


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bit patterns to float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    hidden: int
    inter: int
    n_experts: int
    top_k: int
    n_shared: int = 1
    shared_inter: int = 0          # 0 -> same as inter
    router_std: float | None = None  # None -> 1/sqrt(hidden) (logits ~ N(0,1))
    zipf_s: float = 0.0            # > 0 -> per-expert bias -s*ln(rank)
    description: str = ""

    @property
    def sh_inter(self) -> int:
        return self.shared_inter or self.inter


WORKLOADS = {
    "tiny": Workload("tiny", 64, 256, 256, 8, 2, router_std=0.02,
                     description="T=64, hidden=256, 8 routed experts (inter 256), top-2, 1 shared expert"),
    "ds_decode_t1": Workload("ds_decode_t1", 1, 7168, 2048, 256, 8,
                             description="DeepSeek-V3-shaped decode layer, T=1"),
    "ds_decode_t4": Workload("ds_decode_t4", 4, 7168, 2048, 256, 8,
                             description="DeepSeek-V3-shaped decode layer, T=4"),
    "ds_decode_t16": Workload("ds_decode_t16", 16, 7168, 2048, 256, 8,
                              description="DeepSeek-V3-shaped decode layer, T=16"),
    "ds_prefill_8k": Workload("ds_prefill_8k", 8192, 7168, 2048, 256, 8,
                              description="DeepSeek-V3-shaped prefill layer, T=8192, bias 0"),
    "skew_32k": Workload("skew_32k", 32768, 7168, 2048, 256, 8, zipf_s=1.2,
                         description="DeepSeek-V3-shaped prefill layer, T=32768, Zipf(1.2) expert bias"),
    "kimi_64k": Workload("kimi_64k", 65536, 7168, 2048, 384, 8,
                         description="Kimi-K2-shaped prefill layer, T=65536, 384 experts"),
    # profiling case: DeepSeek-V3 expert shapes and ~256 rows per expert (as
    # at T=8192) with 32 experts, small enough for a full counter capture
    "ds_prefill_probe": Workload("ds_prefill_probe", 1024, 7168, 2048, 32, 8,
                                 description="DeepSeek-V3 expert shapes, 32 experts, T=1024 (profiling)"),
    "ds_decode_probe": Workload("ds_decode_probe", 16, 7168, 2048, 32, 8,
                                description="DeepSeek-V3 expert shapes, 32 experts, T=16 (profiling)"),
    "ds_decode_t1_probe": Workload("ds_decode_t1_probe", 1, 7168, 2048, 32, 8,
                                   description="DeepSeek-V3 expert shapes, 32 experts, T=1 (profiling)"),
}


def router_bias(wl: Workload, seed: int = 0) -> np.ndarray | None:
    """Per-expert router bias: none, or b_e = -s*ln(rank_e) with rank a seeded
    permutation of 1..E, so exp(b_e) = rank^-s (Zipf popularity)."""
    if wl.zipf_s <= 0:
        return None
    rank = permutation(seed, STREAM_BIAS_PERM, wl.n_experts).astype(np.float64) + 1.0
    return (-wl.zipf_s * np.log(rank)).astype(np.float32)


def make_inputs(wl: Workload, seed: int = 0, T: int | None = None, with_experts: bool = True) -> dict:
    """All inputs of one layer as host numpy arrays.

    x         uint16 [T][H]       bf16 bits, N(0,1)
    router_w  f32    [E][H]       N(0, router_std^2)
    router_b  f32    [E] or None
    w_gate/w_up uint8 [E][I][H], s_gate/s_up f32 [E][I/128][H/128]
    w_down    uint8 [E][H][I],   s_down f32 [E][H/128][I/128]
    sh_*      the same for the shared expert with E = 1 (inter = sh_inter)
    """
    T = wl.T if T is None else T
    H, I, E = wl.hidden, wl.inter, wl.n_experts
    rstd = wl.router_std if wl.router_std is not None else 1.0 / np.sqrt(H)
    d = {
        "x": bf16_normal(seed, STREAM_X, (T, H), 1.0),
        "router_w": f32_normal(seed, STREAM_ROUTER_W, (E, H), float(rstd)),
        "router_b": router_bias(wl, seed),
    }
    if with_experts:
        d["w_gate"], d["s_gate"] = fp8_blocks(seed, STREAM_GATE, E, I, H)
        d["w_up"], d["s_up"] = fp8_blocks(seed, STREAM_UP, E, I, H)
        d["w_down"], d["s_down"] = fp8_blocks(seed, STREAM_DOWN, E, H, I)
        if wl.n_shared:
            SI = wl.sh_inter
            d["sh_gate"], d["sh_s_gate"] = fp8_blocks(seed, STREAM_SH_GATE, 1, SI, H)
            d["sh_up"], d["sh_s_up"] = fp8_blocks(seed, STREAM_SH_UP, 1, SI, H)
            d["sh_down"], d["sh_s_down"] = fp8_blocks(seed, STREAM_SH_DOWN, 1, H, SI)
    return d
