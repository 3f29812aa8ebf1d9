"""Python binding of libllm (include/llm.h): argument marshalling only.

Every computation runs in the CUDA library; this module converts Python/numpy/torch
arguments to the C ABI and raises on error statuses.  If libllm.so is missing the
import of the library fails loudly: there is no CPU path.
"""
import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libllm.so")

LLM_OK, LLM_ERR_CONFIG, LLM_ERR_WEIGHTS_SIZE, LLM_ERR_OOM, LLM_ERR_POS_RANGE = 0, 1, 2, 3, 4
LLM_ERR_TOKEN_RANGE, LLM_ERR_BATCH, LLM_ERR_ARG, LLM_ERR_CUDA, LLM_ERR_DEVICE_TIMEOUT = 5, 6, 7, 8, 9
LLM_DTYPE_F32, LLM_DTYPE_BF16 = 0, 1

# every extern "C" symbol include/llm.h declares
EXPORTS = ("llm_weight_count", "llm_create", "llm_destroy", "llm_reset", "llm_prefill", "llm_decode",
           "llm_sample", "llm_step", "llm_prefill_dev", "llm_decode_dev", "llm_sample_dev",
           "llm_step_dev", "llm_synchronize", "llm_stream", "llm_logits_buffer", "llm_filled",
           "llm_last_error", "llm_status_string", "llm_kv_import", "llm_kv_export",
           "llm_debug_trace", "llm_profile_kernel", "llm_sample_noalloc",
           "llm_step_kernels", "llm_decode_rows", "llm_decode_rows_dev", "llm_step_rows",
           "llm_step_rows_dev", "llm_generate", "llm_generate_dev", "llm_decode_paged",
           "llm_decode_paged_dev", "llm_step_paged", "llm_step_paged_dev", "llm_check_wait_timeout",
           "llm_prefill_packed")


class LlmConfig(ctypes.Structure):
    _fields_ = [("kv_heads", ctypes.c_int32), ("group", ctypes.c_int32), ("half", ctypes.c_int32),
                ("ffn", ctypes.c_int32), ("layers", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("eps", ctypes.c_float), ("theta", ctypes.c_float), ("tied", ctypes.c_int32),
                ("rope_llama3", ctypes.c_int32), ("rope_factor", ctypes.c_float),
                ("rope_low_freq", ctypes.c_float), ("rope_high_freq", ctypes.c_float),
                ("rope_orig_max_pos", ctypes.c_float), ("max_batch", ctypes.c_int32),
                ("max_seq", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("debug_trace", ctypes.c_int32), ("tc_min_batch", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("step_kernel", ctypes.c_int32)]


class LlmError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{msg} (status {status})")
        self.status = status


# argument and result types of every entry point (ctypes)
_i32, _i64, _u64, _f32, _vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p
_pcfg = ctypes.POINTER(LlmConfig)
SIGNATURES = {
    "llm_weight_count": ([_pcfg], _u64),
    "llm_create": ([_pcfg, _vp, _u64, _i32, _vp, ctypes.POINTER(_vp)], _i32),
    "llm_destroy": ([_vp], _i32),
    "llm_reset": ([_vp], _i32),
    "llm_prefill": ([_vp, _vp, _i32, _i32, _i32, _vp], _i32),
    "llm_decode": ([_vp, _vp, _i32, _i32, _vp], _i32),
    "llm_sample": ([_vp, _vp, _i32, _f32, _i32, _f32, _vp, _vp], _i32),
    "llm_step": ([_vp, _vp, _i32, _i32, _f32, _i32, _f32, _vp, _vp, _vp], _i32),
    "llm_prefill_dev": ([_vp, _vp, _i32, _i32, _i32, _vp], _i32),
    "llm_decode_dev": ([_vp, _vp, _i32, _i32, _vp], _i32),
    "llm_sample_dev": ([_vp, _vp, _i32, _f32, _i32, _f32, _vp, _vp], _i32),
    "llm_step_dev": ([_vp, _vp, _i32, _i32, _f32, _i32, _f32, _vp, _vp, _vp], _i32),
    "llm_decode_rows": ([_vp, _vp, _i32, _vp, _vp], _i32),
    "llm_decode_rows_dev": ([_vp, _vp, _i32, _vp, _vp], _i32),
    "llm_step_rows": ([_vp, _vp, _i32, _vp, _f32, _i32, _f32, _vp, _vp, _vp], _i32),
    "llm_step_rows_dev": ([_vp, _vp, _i32, _vp, _f32, _i32, _f32, _vp, _vp, _vp], _i32),
    "llm_generate": ([_vp, _vp, _i32, _i32, _i32, _f32, _i32, _f32, _vp, _vp], _i32),
    "llm_generate_dev": ([_vp, _vp, _i32, _i32, _i32, _f32, _i32, _f32, _vp, _vp], _i32),
    "llm_decode_paged": ([_vp, _vp, _i32, _vp, _vp, _i32, _vp], _i32),
    "llm_decode_paged_dev": ([_vp, _vp, _i32, _vp, _vp, _i32, _vp], _i32),
    "llm_step_paged": ([_vp, _vp, _i32, _vp, _vp, _i32, _f32, _i32, _f32, _vp, _vp, _vp], _i32),
    "llm_step_paged_dev": ([_vp, _vp, _i32, _vp, _vp, _i32, _f32, _i32, _f32, _vp, _vp, _vp], _i32),
    "llm_prefill_packed": ([_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _vp], _i32),
    "llm_synchronize": ([_vp], _i32),
    "llm_stream": ([_vp], _vp),
    "llm_logits_buffer": ([_vp], _vp),
    "llm_filled": ([_vp, _i32], _i32),
    "llm_last_error": ([_vp], ctypes.c_char_p),
    "llm_status_string": ([_i32], ctypes.c_char_p),
    "llm_kv_import": ([_vp, _i32, _i32, _i32, _i32, _vp, _vp], _i32),
    "llm_kv_export": ([_vp, _i32, _i32, _i32, _i32, _vp, _vp], _i32),
    "llm_debug_trace": ([_vp, _i32, ctypes.c_char_p, _vp], _i32),
    "llm_profile_kernel": ([_vp, _i32, _i32, _i32, _i32, ctypes.POINTER(_f32)], _i32),
    "llm_sample_noalloc": ([_vp, _i32, _i32, _f32, _i32, _f32, _vp, _vp, _vp], _i32),
    "llm_step_kernels": ([_vp, _i32, _f32, _i32, ctypes.POINTER(_i32)], _i32),
    "llm_check_wait_timeout": ([_vp, _i64], _i32),
    }

_lib = None


def lib():
    """The loaded libllm.so (ctypes).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m llama_architecture_kv_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def config(shape, max_batch, max_seq, debug_trace=False, tc_min_batch=0, max_tokens=0,
           step_kernel=0) -> LlmConfig:
    """An llm_config from a shape description (fields kv, g, half, ffn, layers, vocab, eps,
    theta, tied, llama3, factor, low_freq, high_freq, orig_max, bf16)."""
    return LlmConfig(shape.kv, shape.g, shape.half, shape.ffn, shape.layers, shape.vocab,
                     shape.eps, shape.theta, int(shape.tied), int(shape.llama3), shape.factor,
                     shape.low_freq, shape.high_freq, shape.orig_max, max_batch, max_seq,
                     LLM_DTYPE_BF16 if shape.bf16 else LLM_DTYPE_F32, int(debug_trace),
                     int(tc_min_batch), int(max_tokens), int(step_kernel))


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if isinstance(a, np.ndarray):
        assert a.flags.c_contiguous
        return a.ctypes.data
    if hasattr(a, "data_ptr"):  # torch tensor
        assert a.is_contiguous()
        return a.data_ptr()
    raise TypeError(type(a))


def _check(h, status):
    if status != LLM_OK:
        msg = lib().llm_last_error(h) if h else None
        name = lib().llm_status_string(status).decode()
        raise LlmError(status, f"{name}: {msg.decode() if msg else ''}")


# ---- the C functions under their own names -------------------------------------------------

def llm_weight_count(cfg: LlmConfig) -> int:
    return int(lib().llm_weight_count(ctypes.byref(cfg)))


def llm_create(cfg: LlmConfig, weights, weights_on_device=False, stream=None):
    nbytes = weights.nbytes if isinstance(weights, np.ndarray) else weights.numel() * weights.element_size()
    h = ctypes.c_void_p()
    st = lib().llm_create(ctypes.byref(cfg), _ptr(weights), nbytes, int(weights_on_device),
                          stream, ctypes.byref(h))
    if st != LLM_OK:
        why = lib().llm_last_error(None)
        raise LlmError(st, f"llm_create: {lib().llm_status_string(st).decode()}: "
                           f"{why.decode() if why else ''}")
    return h.value


def llm_destroy(h):
    _check(None, lib().llm_destroy(h))


def llm_reset(h):
    _check(h, lib().llm_reset(h))


def llm_prefill(h, tokens, B, S, pos, logits=None):
    _check(h, lib().llm_prefill(h, _ptr(tokens), B, S, pos, _ptr(logits)))


def llm_decode(h, tokens, B, pos, logits):
    _check(h, lib().llm_decode(h, _ptr(tokens), B, pos, _ptr(logits)))


def llm_sample(h, logits, B, temp, k, p, u, ids):
    _check(h, lib().llm_sample(h, _ptr(logits), B, temp, k, p, _ptr(u), _ptr(ids)))


def llm_step(h, tokens, B, pos, temp, k, p, u, ids, logits=None):
    _check(h, lib().llm_step(h, _ptr(tokens), B, pos, temp, k, p, _ptr(u), _ptr(ids), _ptr(logits)))


def llm_prefill_dev(h, tokens, B, S, pos, logits=None):
    _check(h, lib().llm_prefill_dev(h, _ptr(tokens), B, S, pos, _ptr(logits)))


def llm_decode_dev(h, tokens, B, pos, logits):
    _check(h, lib().llm_decode_dev(h, _ptr(tokens), B, pos, _ptr(logits)))


def llm_sample_dev(h, logits, B, temp, k, p, u, ids):
    _check(h, lib().llm_sample_dev(h, _ptr(logits), B, temp, k, p, _ptr(u), _ptr(ids)))


def llm_step_dev(h, tokens, B, pos, temp, k, p, u, ids, logits=None):
    _check(h, lib().llm_step_dev(h, _ptr(tokens), B, pos, temp, k, p, _ptr(u), _ptr(ids), _ptr(logits)))


def llm_decode_rows(h, tokens, B, positions, logits):
    _check(h, lib().llm_decode_rows(h, _ptr(tokens), B, _ptr(positions), _ptr(logits)))


def llm_decode_rows_dev(h, tokens, B, positions, logits):
    _check(h, lib().llm_decode_rows_dev(h, _ptr(tokens), B, _ptr(positions), _ptr(logits)))


def llm_step_rows(h, tokens, B, positions, temp, k, p, u, ids, logits=None):
    _check(h, lib().llm_step_rows(h, _ptr(tokens), B, _ptr(positions), temp, k, p, _ptr(u), _ptr(ids),
                                  _ptr(logits)))


def llm_step_rows_dev(h, tokens, B, positions, temp, k, p, u, ids, logits=None):
    _check(h, lib().llm_step_rows_dev(h, _ptr(tokens), B, _ptr(positions), temp, k, p, _ptr(u), _ptr(ids),
                                      _ptr(logits)))


def llm_generate(h, tokens, B, pos, n_steps, temp, k, p, u, ids):
    _check(h, lib().llm_generate(h, _ptr(tokens), B, pos, n_steps, temp, k, p, _ptr(u), _ptr(ids)))


def llm_generate_dev(h, tokens, B, pos, n_steps, temp, k, p, u, ids):
    _check(h, lib().llm_generate_dev(h, _ptr(tokens), B, pos, n_steps, temp, k, p, _ptr(u), _ptr(ids)))


def llm_decode_paged(h, tokens, B, positions, table, pages_per_row, logits):
    _check(h, lib().llm_decode_paged(h, _ptr(tokens), B, _ptr(positions), _ptr(table), pages_per_row,
                                     _ptr(logits)))


def llm_decode_paged_dev(h, tokens, B, positions, table, pages_per_row, logits):
    _check(h, lib().llm_decode_paged_dev(h, _ptr(tokens), B, _ptr(positions), _ptr(table), pages_per_row,
                                         _ptr(logits)))


def llm_step_paged(h, tokens, B, positions, table, pages_per_row, temp, k, p, u, ids, logits=None):
    _check(h, lib().llm_step_paged(h, _ptr(tokens), B, _ptr(positions), _ptr(table), pages_per_row, temp, k, p,
                                   _ptr(u), _ptr(ids), _ptr(logits)))


def llm_step_paged_dev(h, tokens, B, positions, table, pages_per_row, temp, k, p, u, ids, logits=None):
    _check(h, lib().llm_step_paged_dev(h, _ptr(tokens), B, _ptr(positions), _ptr(table), pages_per_row, temp, k,
                                       p, _ptr(u), _ptr(ids), _ptr(logits)))


def llm_prefill_packed(h, tokens, rows, positions, segments, P, last, nlast, logits):
    _check(h, lib().llm_prefill_packed(h, _ptr(tokens), _ptr(rows), _ptr(positions), _ptr(segments), P,
                                       _ptr(last), nlast, _ptr(logits)))


def llm_synchronize(h):
    _check(h, lib().llm_synchronize(h))


def llm_stream(h) -> int:
    return lib().llm_stream(h) or 0


def llm_logits_buffer(h) -> int:
    return lib().llm_logits_buffer(h)


def llm_filled(h, b) -> int:
    return int(lib().llm_filled(h, b))


def llm_kv_import(h, layer, row, pos0, k, v):
    n = k.shape[1]
    _check(h, lib().llm_kv_import(h, layer, row, pos0, n, _ptr(k), _ptr(v)))


def llm_kv_export(h, layer, row, pos0, k, v):
    n = k.shape[1]
    _check(h, lib().llm_kv_export(h, layer, row, pos0, n, _ptr(k), _ptr(v)))


def llm_debug_trace(h, layer, name, dst):
    _check(h, lib().llm_debug_trace(h, layer, name.encode(), _ptr(dst)))


KERNELS = {"qkv": 0, "attention": 1, "o_proj": 2, "gate_up": 3, "down": 4, "lm_head": 5, "sampler": 6}


def llm_profile_kernel(h, which, B, pos, reps) -> float:
    ms = ctypes.c_float()
    _check(h, lib().llm_profile_kernel(h, which, B, pos, reps, ctypes.byref(ms)))
    return float(ms.value)


def llm_step_kernels(h, B, temp, k=1 << 30) -> int:
    n = ctypes.c_int32()
    _check(h, lib().llm_step_kernels(h, B, temp, k, ctypes.byref(n)))
    return int(n.value)


def llm_check_wait_timeout(h, limit_cycles):
    _check(h, lib().llm_check_wait_timeout(h, limit_cycles))


SAMPLE_NOALLOC_MAX_ELEMS = 262144


def llm_sample_noalloc(logits, B, V, temp, k, p, u, ids, stream=None):
    """Sampling on device buffers with no handle and no allocation (see include/llm.h): for
    callers that cannot allocate device memory.  B * (V rounded up to 32) <= 262144."""
    st = lib().llm_sample_noalloc(_ptr(logits), B, V, temp, k, p, _ptr(u), _ptr(ids), stream)
    if st != LLM_OK:
        raise LlmError(st, f"llm_sample_noalloc: {lib().llm_status_string(st).decode()}")


# ---- a small convenience wrapper --------------------------------------------------------

class Model:
    """One handle: host-memory entry points with numpy arrays."""

    def __init__(self, shape, weights, max_batch, max_seq, stream=None, debug_trace=False,
                 weights_on_device=False, tc_min_batch=0, max_tokens=0, step_kernel=0):
        self.shape = shape
        self.cfg = config(shape, max_batch, max_seq, debug_trace, tc_min_batch, max_tokens, step_kernel)
        self.h = llm_create(self.cfg, weights, weights_on_device, stream)
        self.V = shape.vocab
        self.cache_dtype = np.uint16 if shape.bf16 else np.float32

    def close(self):
        if self.h:
            llm_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, tokens, pos=0, logits=True):
        tokens = np.ascontiguousarray(tokens, np.int32)
        B, S = tokens.shape
        out = np.empty((B, self.V), np.float32) if logits else None
        llm_prefill(self.h, tokens, B, S, pos, out)
        return out

    def decode(self, tokens, pos):
        tokens = np.ascontiguousarray(tokens, np.int32).reshape(-1)
        out = np.empty((tokens.size, self.V), np.float32)
        llm_decode(self.h, tokens, tokens.size, pos, out)
        return out

    def decode_rows(self, tokens, positions):
        """One token per row, row b at its own position positions[b]."""
        tokens = np.ascontiguousarray(tokens, np.int32).reshape(-1)
        positions = np.ascontiguousarray(positions, np.int32).reshape(-1)
        assert positions.size == tokens.size
        out = np.empty((tokens.size, self.V), np.float32)
        llm_decode_rows(self.h, tokens, tokens.size, positions, out)
        return out

    def step_rows(self, tokens, positions, temp=0.0, k=1, p=1.0, u=None, logits=False):
        tokens = np.ascontiguousarray(tokens, np.int32).reshape(-1)
        positions = np.ascontiguousarray(positions, np.int32).reshape(-1)
        assert positions.size == tokens.size
        B = tokens.size
        ids = np.empty(B, np.int32)
        out = np.empty((B, self.V), np.float32) if logits else None
        u = None if u is None else np.ascontiguousarray(u, np.float32)
        llm_step_rows(self.h, tokens, B, positions, temp, k, p, u, ids, out)
        return (ids, out) if logits else ids

    def generate(self, tokens, pos, n_steps, temp=0.0, k=1, p=1.0, u=None):
        """n_steps chained decode + draw steps inside CUDA graphs; ids [n_steps][B]."""
        tokens = np.ascontiguousarray(tokens, np.int32).reshape(-1)
        B = tokens.size
        ids = np.empty((n_steps, B), np.int32)
        u = None if u is None else np.ascontiguousarray(u, np.float32).reshape(n_steps, B)
        llm_generate(self.h, tokens, B, pos, n_steps, temp, k, p, u, ids)
        return ids

    def decode_paged(self, tokens, positions, table):
        """One token per row at its own position, the cache read and written through the row's
        pages: table [B][pages_per_row] of pool pages (64 positions each)."""
        tokens = np.ascontiguousarray(tokens, np.int32).reshape(-1)
        positions = np.ascontiguousarray(positions, np.int32).reshape(-1)
        table = np.ascontiguousarray(table, np.int32)
        assert positions.size == tokens.size and table.shape[0] == tokens.size
        out = np.empty((tokens.size, self.V), np.float32)
        llm_decode_paged(self.h, tokens, tokens.size, positions, table, table.shape[1], out)
        return out

    def step_paged(self, tokens, positions, table, temp=0.0, k=1, p=1.0, u=None, logits=False):
        tokens = np.ascontiguousarray(tokens, np.int32).reshape(-1)
        positions = np.ascontiguousarray(positions, np.int32).reshape(-1)
        table = np.ascontiguousarray(table, np.int32)
        B = tokens.size
        ids = np.empty(B, np.int32)
        out = np.empty((B, self.V), np.float32) if logits else None
        u = None if u is None else np.ascontiguousarray(u, np.float32)
        llm_step_paged(self.h, tokens, B, positions, table, table.shape[1], temp, k, p, u, ids, out)
        return (ids, out) if logits else ids

    def prefill_packed(self, tokens, rows, positions, segments, last, logits=True):
        """Prompts packed end to end; logits [len(last)][V] after the tokens last names."""
        arrs = [np.ascontiguousarray(a, np.int32).reshape(-1) for a in (tokens, rows, positions, segments, last)]
        tokens, rows, positions, segments, last = arrs
        P = tokens.size
        assert rows.size == P and positions.size == P and segments.size == P
        out = np.empty((last.size, self.V), np.float32) if logits else None
        llm_prefill_packed(self.h, tokens, rows, positions, segments, P, last, last.size, out)
        return out

    def sample(self, logits, temp, k, p, u):
        logits = np.ascontiguousarray(logits, np.float32)
        B = logits.shape[0]
        ids = np.empty(B, np.int32)
        u = None if u is None else np.ascontiguousarray(u, np.float32)
        llm_sample(self.h, logits, B, temp, k, p, u, ids)
        return ids

    def step(self, tokens, pos, temp=0.0, k=1, p=1.0, u=None, logits=False):
        tokens = np.ascontiguousarray(tokens, np.int32).reshape(-1)
        B = tokens.size
        ids = np.empty(B, np.int32)
        out = np.empty((B, self.V), np.float32) if logits else None
        u = None if u is None else np.ascontiguousarray(u, np.float32)
        llm_step(self.h, tokens, B, pos, temp, k, p, u, ids, out)
        return (ids, out) if logits else ids

    def kv_import(self, layer, row, pos0, k, v):
        llm_kv_import(self.h, layer, row, pos0, np.ascontiguousarray(k, self.cache_dtype),
                      np.ascontiguousarray(v, self.cache_dtype))

    def kv_export(self, layer, row, pos0, n):
        k = np.empty((self.shape.kv, n, self.shape.hd), self.cache_dtype)
        v = np.empty_like(k)
        llm_kv_export(self.h, layer, row, pos0, k, v)
        return k, v

    def trace(self, layer, name):
        """One intermediate of the last traced step: [max_batch][width] (include/llm.h lists the
        names)."""
        w = {"swiglu": self.shape.ffn, "k": self.shape.kvw, "v": self.shape.kvw,
             "kr": self.shape.kvw}.get(name, self.shape.d)
        out = np.empty((self.cfg.max_batch, w), np.float32)
        llm_debug_trace(self.h, layer, name, out)
        return out

    def synchronize(self):
        llm_synchronize(self.h)

    def filled(self, b=0):
        return llm_filled(self.h, b)
