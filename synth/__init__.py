"""Seeded synthetic inputs (weights, token ids, cache values, uniform draws).

A ctypes wrapper over synth.c.  Nothing here computes any part of the decoder;
both the oracle and the GPU library are fed from these functions.
"""
import ctypes
import os
import subprocess

import numpy as np

from .configs import WORKLOADS, Shape, Workload, shrink, weight_count  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force=False):
    """Compile libsynth.so next to its source (gcc, a second or two)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp,
                               "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u32, i32, i64, f32, f64, vp = (ctypes.c_uint32, ctypes.c_int32, ctypes.c_int64,
                                       ctypes.c_float, ctypes.c_double, ctypes.c_void_p)
        L.synth_hash32.argtypes = [u32]
        L.synth_hash32.restype = u32
        L.synth_uniform.argtypes = [u32, u32]
        L.synth_uniform.restype = f32
        L.synth_uniforms.argtypes = [u32, u32, i64, vp]
        L.synth_tokens.argtypes = [u32, u32, i64, i32, vp]
        L.synth_normal.argtypes = [u32, u32, i64, f64, f64, i32, vp, i32]
        L.synth_const.argtypes = [i64, f32, i32, vp]
        L.synth_model_blob.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, u32, f64, f32,
                                       vp, i32]
        L.synth_model_blob.restype = i64
        _lib = L
    return _lib


def _threads():
    return max(1, min(64, os.cpu_count() or 1))


def hash32(x: int) -> int:
    return int(lib().synth_hash32(x & 0xFFFFFFFF))


def uniform(seed: int, n: int) -> float:
    return float(lib().synth_uniform(seed & 0xFFFFFFFF, n & 0xFFFFFFFF))


def uniforms(seed: int, n0: int, count: int) -> np.ndarray:
    out = np.empty(count, np.float32)
    lib().synth_uniforms(seed, n0, count, out.ctypes.data)
    return out


def tokens(seed: int, n0: int, count: int, vocab: int) -> np.ndarray:
    out = np.empty(count, np.int32)
    lib().synth_tokens(seed, n0, count, vocab, out.ctypes.data)
    return out


def normal(seed: int, tensor_idx: int, count: int, std: float = 1.0, bf16: bool = True,
           mean: float = 0.0) -> np.ndarray:
    """N(mean, std^2) values; bf16 bit patterns (uint16) if bf16 else float32."""
    out = np.empty(count, np.uint16 if bf16 else np.float32)
    lib().synth_normal(seed, tensor_idx, count, mean, std, int(bf16), out.ctypes.data,
                       _threads())
    return out


def model_blob(shape: Shape, seed: int, wstd: float = 0.02, gain: float = 1.0,
               out: np.ndarray = None) -> np.ndarray:
    """The weight blob of a shape (uint16 bf16 bits, or float32), in loader tensor order."""
    n = weight_count(shape)
    dt = np.uint16 if shape.bf16 else np.float32
    if out is None:
        out = np.empty(n, dt)
    assert out.dtype == dt and out.size == n and out.flags.c_contiguous
    got = lib().synth_model_blob(shape.d, shape.d, shape.kvw, shape.ffn, shape.layers,
                                 shape.vocab, int(shape.tied), int(shape.bf16), seed, wstd,
                                 gain, out.ctypes.data, _threads())
    assert got == n, (got, n)
    return out


def kv_tensor_idx(layer: int, row: int, which: int, rows: int) -> int:
    """Tensor index of the synthetic keys (which=0) or values (which=1) of one cache row."""
    return (layer * rows + row) * 2 + which


def kv_values(seed: int, layer: int, row: int, rows: int, kv: int, n_pos: int, hd: int,
              bf16: bool = True, std: float = 1.0):
    """Synthetic keys and values of one (layer, row): arrays [kv][n_pos][hd]."""
    cnt = kv * n_pos * hd
    k = normal(seed, kv_tensor_idx(layer, row, 0, rows), cnt, std, bf16).reshape(kv, n_pos, hd)
    v = normal(seed, kv_tensor_idx(layer, row, 1, rows), cnt, std, bf16).reshape(kv, n_pos, hd)
    return k, v


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32)
