"""The C-ABI library loads and exports every entry point include/llm.h declares; host-side
argument checks that need no GPU (no compute calls here)."""
import ctypes
import os
import re

import numpy as np
import pytest

import llama_architecture_kv_gb300 as pkg
from llama_architecture_kv_gb300 import build as pkg_build
import oracle
from synth.configs import LLAMA8B, SMOL135M, SMOL1_7B, TINY

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pkg_build.build()
    return pkg.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "llm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(llm_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("llm_create", "llm_prefill", "llm_decode", "llm_sample", "llm_destroy"):
        assert n in names
    assert set(names) == set(pkg.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_weight_count_matches_the_oracle_layout(lib):
    for s in (TINY, SMOL135M, SMOL1_7B, LLAMA8B):
        c = pkg.config(s, 1, 16)
        assert pkg.llm_weight_count(c) == oracle.weight_count(oracle.cfg_of(s))


def test_status_strings(lib):
    for s in range(10):
        assert lib.llm_status_string(s)


def _create_status(cfg, nbytes):
    h = ctypes.c_void_p()
    buf = np.zeros(4, np.uint8)
    return pkg.lib().llm_create(ctypes.byref(cfg), buf.ctypes.data, nbytes, 0, None, ctypes.byref(h))


def test_create_rejects_bad_configs_before_touching_a_gpu(lib):
    good = pkg.config(TINY, 1, 16)
    n = pkg.llm_weight_count(good) * 4
    for field, val in (("kv_heads", 0), ("group", 0), ("half", 0), ("max_seq", 0), ("max_batch", 0),
                       ("dtype", 7), ("half", 12), ("group", 17)):
        c = pkg.config(TINY, 1, 16)
        setattr(c, field, val)
        assert _create_status(c, n) == pkg.LLM_ERR_CONFIG, field
    c = pkg.config(TINY, 1, 16)
    c.theta = 0.0
    assert _create_status(c, n) == pkg.LLM_ERR_CONFIG
    for delta in (-4, -2, 2, 4):
        assert _create_status(good, n + delta) == pkg.LLM_ERR_WEIGHTS_SIZE


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(pkg, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(pkg, "_lib", None)
    with pytest.raises(RuntimeError):
        pkg.lib()


def _prototypes():
    """(name, parameter count) of every function include/llm.h declares."""
    src = open(os.path.join(ROOT, "include", "llm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    out = {}
    for m in re.finditer(r"\b(llm_[a-z_]+)\s*\(([^;{)]*)\)\s*;", src):
        params = [p for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        out[m.group(1)] = len(params)
    return out


def test_binding_signatures_match_the_header():
    # a ctypes signature with the wrong number of arguments would pass garbage through the ABI
    protos = _prototypes()
    assert set(protos) == set(pkg.EXPORTS)
    for name, (argtypes, _) in pkg.SIGNATURES.items():
        assert len(argtypes) == protos[name], name


def test_header_is_plain_c(tmp_path):
    import shutil
    import subprocess
    if not shutil.which("gcc"):
        pytest.skip("no C compiler")
    src = tmp_path / "use.c"
    src.write_text('#include "llm.h"\nint main(void) { return llm_status_string(LLM_OK) == 0; }\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.join(ROOT, "include"),
                        str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_entries_refuse_a_null_handle(lib):
    # every entry that takes a handle checks it (and its buffers) before any device work
    protos = _prototypes()
    skip = {"llm_create", "llm_weight_count", "llm_status_string", "llm_last_error", "llm_stream",
            "llm_logits_buffer", "llm_filled", "llm_sample_noalloc"}
    for name in sorted(protos):
        if name in skip:
            continue
        argtypes, _ = pkg.SIGNATURES[name]
        args = [None if t in (ctypes.c_void_p, ctypes.c_char_p) or issubclass(t, ctypes._Pointer) else 0
                for t in argtypes]
        assert getattr(lib, name)(*args) == pkg.LLM_ERR_ARG, name
