"""ORACLE — test infrastructure, not product code.

A ctypes wrapper over oracle.c, the plain single-threaded f32 CPU decoder that the
GPU library is checked against.  Only tests/, the smoke check and bench.py's CPU
baseline leg use it.  It never imports the GPU package and the GPU package never
imports it.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
_lib = None

OK, ERR_CONFIG, ERR_WEIGHTS_SIZE, ERR_OOM, ERR_POS_RANGE, ERR_TOKEN_RANGE, ERR_ARG = (
    0, -1, -2, -3, -4, -5, -6)


class Cfg(ctypes.Structure):
    _fields_ = [("kv", ctypes.c_int32), ("g", ctypes.c_int32), ("half", ctypes.c_int32),
                ("ffn", ctypes.c_int32), ("layers", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("eps", ctypes.c_float), ("theta", ctypes.c_float), ("tied", ctypes.c_int32),
                ("llama3", ctypes.c_int32), ("factor", ctypes.c_float),
                ("low_freq", ctypes.c_float), ("high_freq", ctypes.c_float),
                ("orig_max", ctypes.c_float), ("batch", ctypes.c_int32), ("cap", ctypes.c_int32),
                ("bf16", ctypes.c_int32), ("kv_f32", ctypes.c_int32)]


def build(force=False):
    """Compile liboracle.so next to its source (gcc, a second or two)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i32, u64, f32, vp, cp = (ctypes.c_int32, ctypes.c_uint64, ctypes.c_float,
                                 ctypes.c_void_p, ctypes.c_char_p)
        pc = ctypes.POINTER(Cfg)
        sigs = {
            "or_weight_count": ([pc], u64),
            "or_create": ([pc, vp, u64, i32, ctypes.POINTER(i32)], vp),
            "or_destroy": ([vp], None),
            "or_reset": ([vp], None),
            "or_forward": ([vp, i32, i32, i32, vp], i32),
            "or_prefill": ([vp, i32, vp, i32, i32, vp], i32),
            "or_prefill_packed": ([vp, vp, vp, vp, vp, i32, vp, i32, vp], i32),
            "or_embed": ([vp, i32], i32),
            "or_layer": ([vp, i32, i32, i32], i32),
            "or_head": ([vp, vp], None),
            "or_forward_full": ([pc, vp, u64, vp, i32, vp], i32),
            "or_attend": ([vp, i32, i32, vp, i32, vp], i32),
            "or_kv_write": ([vp, i32, i32, i32, i32, vp, vp], i32),
            "or_kv_read": ([vp, i32, i32, i32, i32, vp, vp], i32),
            "or_trace": ([vp, i32, cp, vp], i32),
            "or_tree_sum": ([vp, i32], f32),
            "or_rmsnorm": ([vp, vp, i32, f32, vp], None),
            "or_split": ([vp, i32, i32, vp, ctypes.POINTER(i32), vp, ctypes.POINTER(i32)], None),
            "or_join": ([vp, i32, vp, i32, vp], None),
            "or_gqa_kv_head": ([i32, i32], i32),
            "or_rope_head": ([vp, i32, vp, vp, vp], None),
            "or_inv_freq": ([pc, vp], None),
            "or_rope_cs": ([pc, i32, vp, vp], None),
            "or_exp_s": ([f32], f32),
            "or_f32_to_bf16": ([f32], ctypes.c_uint16),
            "or_argmax": ([vp, i32], i32),
            "or_topk": ([vp, i32, i32, vp], i32),
            "or_sample": ([vp, i32, f32, i32, f32, f32], i32),
            "or_sample_detail": ([vp, i32, f32, i32, f32, f32, vp, vp, vp], i32),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def cfg_of(shape, batch=1, cap=16, kv_f32=False) -> Cfg:
    return Cfg(shape.kv, shape.g, shape.half, shape.ffn, shape.layers, shape.vocab,
               shape.eps, shape.theta, int(shape.tied), int(shape.llama3), shape.factor,
               shape.low_freq, shape.high_freq, shape.orig_max, batch, cap, int(shape.bf16),
               int(kv_f32))


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def weight_count(cfg: Cfg) -> int:
    return int(lib().or_weight_count(ctypes.byref(cfg)))


def tree_sum(x) -> float:
    x = _f32(x)
    return float(lib().or_tree_sum(x.ctypes.data, x.size))


def rmsnorm(x, g, eps) -> np.ndarray:
    x, g = _f32(x), _f32(g)
    out = np.empty_like(x)
    lib().or_rmsnorm(x.ctypes.data, g.ctypes.data, x.size, eps, out.ctypes.data)
    return out


def split(xs, half):
    xs = _f32(xs)
    lo, hi = np.empty(max(xs.size, 1), np.float32), np.empty(max(xs.size, 1), np.float32)
    nlo, nhi = ctypes.c_int32(), ctypes.c_int32()
    lib().or_split(xs.ctypes.data, xs.size, half, lo.ctypes.data, ctypes.byref(nlo),
                   hi.ctypes.data, ctypes.byref(nhi))
    return lo[:nlo.value].copy(), hi[:nhi.value].copy()


def join(lo, hi):
    lo, hi = _f32(lo), _f32(hi)
    out = np.empty(max(lo.size + hi.size, 1), np.float32)
    lib().or_join(lo.ctypes.data, lo.size, hi.ctypes.data, hi.size, out.ctypes.data)
    return out[:lo.size + hi.size]


def gqa_kv_head(h, g) -> int:
    return int(lib().or_gqa_kv_head(h, g))


def rope_head(x, cs, sn) -> np.ndarray:
    x, cs, sn = _f32(x), _f32(cs), _f32(sn)
    out = np.empty_like(x)
    lib().or_rope_head(x.ctypes.data, x.size // 2, cs.ctypes.data, sn.ctypes.data,
                       out.ctypes.data)
    return out


def inv_freq(cfg: Cfg) -> np.ndarray:
    out = np.empty(cfg.half, np.float32)
    lib().or_inv_freq(ctypes.byref(cfg), out.ctypes.data)
    return out


def rope_cs(cfg: Cfg, t: int):
    c, s = np.empty(cfg.half, np.float32), np.empty(cfg.half, np.float32)
    lib().or_rope_cs(ctypes.byref(cfg), t, c.ctypes.data, s.ctypes.data)
    return c, s


def exp_s(x: float) -> float:
    return float(lib().or_exp_s(x))


def f32_to_bf16(x: float) -> int:
    """The bf16 bits the oracle stores for an f32 key or value (round to nearest even)."""
    return int(lib().or_f32_to_bf16(x))


def argmax(x) -> int:
    x = _f32(x)
    return int(lib().or_argmax(x.ctypes.data, x.size))


def topk(x, k) -> np.ndarray:
    x = _f32(x)
    ids = np.empty(max(min(k, x.size), 1), np.int32)
    n = lib().or_topk(x.ctypes.data, x.size, k, ids.ctypes.data)
    return ids[:n].copy()


def sample(x, temp, k, p, u) -> int:
    x = _f32(x)
    return int(lib().or_sample(x.ctypes.data, x.size, temp, k, p, u))


def sample_detail(x, temp, k, p, u):
    """(id, candidate ids in order, number kept)."""
    x = _f32(x)
    cand = np.empty(max(min(k, x.size), 1), np.int32)
    nc, nk = ctypes.c_int32(), ctypes.c_int32()
    i = lib().or_sample_detail(x.ctypes.data, x.size, temp, k, p, u, cand.ctypes.data,
                               ctypes.byref(nc), ctypes.byref(nk))
    return int(i), cand[:nc.value].copy(), int(nk.value)


def forward_full(cfg: Cfg, weights: np.ndarray, toks) -> np.ndarray:
    toks = np.ascontiguousarray(toks, dtype=np.int32)
    out = np.empty((toks.size, cfg.vocab), np.float32)
    r = lib().or_forward_full(ctypes.byref(cfg), weights.ctypes.data, weights.nbytes,
                              toks.ctypes.data, toks.size, out.ctypes.data)
    if r:
        raise RuntimeError(f"or_forward_full: {r}")
    return out


class Model:
    """The oracle decoder over a weight blob it does not own (keep `weights` alive)."""

    def __init__(self, cfg: Cfg, weights: np.ndarray, trace=False):
        self.cfg = cfg
        self.weights = weights
        err = ctypes.c_int32()
        h = lib().or_create(ctypes.byref(cfg), weights.ctypes.data, weights.nbytes, int(trace),
                            ctypes.byref(err))
        if not h:
            raise ValueError(f"or_create failed: {err.value}")
        self.h = h
        self.hd = 2 * cfg.half
        self.d = cfg.kv * cfg.g * self.hd
        self.kvw = cfg.kv * self.hd

    def close(self):
        if self.h:
            lib().or_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self):
        lib().or_reset(self.h)

    def forward(self, b, tok, t, logits=True):
        out = np.empty(self.cfg.vocab, np.float32) if logits else None
        r = lib().or_forward(self.h, b, int(tok), t, out.ctypes.data if logits else None)
        if r:
            raise ValueError(f"or_forward: {r}")
        return out

    def embed(self, tok):
        r = lib().or_embed(self.h, int(tok))
        if r:
            raise ValueError(f"or_embed: {r}")

    def layer(self, l, b, t):
        r = lib().or_layer(self.h, l, b, t)
        if r:
            raise ValueError(f"or_layer: {r}")

    def head(self):
        out = np.empty(self.cfg.vocab, np.float32)
        lib().or_head(self.h, out.ctypes.data)
        return out

    def prefill(self, b, toks, pos, logits=True):
        toks = np.ascontiguousarray(toks, dtype=np.int32)
        out = np.empty(self.cfg.vocab, np.float32) if logits else None
        r = lib().or_prefill(self.h, b, toks.ctypes.data, toks.size, pos,
                             out.ctypes.data if logits else None)
        if r:
            raise ValueError(f"or_prefill: {r}")
        return out

    def prefill_packed(self, toks, rows, positions, segments, last):
        """Prompts packed end to end: token p is position positions[p] of prompt segments[p] in
        cache row rows[p]; each attends to its own prompt's tokens up to itself.  Returns the
        logits after token last[m], [len(last)][V]."""
        arrs = [np.ascontiguousarray(a, dtype=np.int32).reshape(-1) for a in (toks, rows, positions, segments, last)]
        toks, rows, positions, segments, last = arrs
        P = toks.size
        assert rows.size == P and positions.size == P and segments.size == P
        out = np.empty((last.size, self.cfg.vocab), np.float32)
        r = lib().or_prefill_packed(self.h, toks.ctypes.data, rows.ctypes.data, positions.ctypes.data,
                                    segments.ctypes.data, P, last.ctypes.data, last.size, out.ctypes.data)
        if r:
            raise ValueError(f"or_prefill_packed: {r}")
        return out

    def attend(self, layer, b, q, t):
        q = _f32(q)
        out = np.empty(self.d, np.float32)
        r = lib().or_attend(self.h, layer, b, q.ctypes.data, t, out.ctypes.data)
        if r:
            raise ValueError(f"or_attend: {r}")
        return out

    def _cache_dtype(self):
        return np.uint16 if (self.cfg.bf16 and not self.cfg.kv_f32) else np.float32

    def kv_write(self, layer, b, pos0, k, v):
        dt = self._cache_dtype()
        k = np.ascontiguousarray(k, dtype=dt)
        v = np.ascontiguousarray(v, dtype=dt)
        n = k.shape[1]
        r = lib().or_kv_write(self.h, layer, b, pos0, n, k.ctypes.data, v.ctypes.data)
        if r:
            raise ValueError(f"or_kv_write: {r}")

    def kv_read(self, layer, b, pos0, n):
        dt = self._cache_dtype()
        k = np.empty((self.cfg.kv, n, self.hd), dt)
        v = np.empty((self.cfg.kv, n, self.hd), dt)
        r = lib().or_kv_read(self.h, layer, b, pos0, n, k.ctypes.data, v.ctypes.data)
        if r:
            raise ValueError(f"or_kv_read: {r}")
        return k, v

    def trace(self, layer, name):
        out = np.empty(max(self.d, self.cfg.ffn), np.float32)
        n = lib().or_trace(self.h, layer, name.encode(), out.ctypes.data)
        if n < 0:
            raise ValueError(f"or_trace: {n}")
        return out[:n].copy()
