"""Paged caches (Llama 3.1 8B Instruct card, "Entries": decode_paged): the caches form a pool of
64-position pages and each row reads and writes its positions through its page table.

An identity table must reproduce llm_decode_rows bit for bit; scattered tables (rows' pages
spread over the pool, crossing physical rows) must match the oracle row by row, with pages
crossed during the sequence, on every attention variant (f32 caches; bf16 head size 128 in
clusters and in the persistent split; the tensor-core projections).
"""
import numpy as np
import pytest

import llama_architecture_kv_gb300 as pkg
import oracle
import synth
from synth import WORKLOADS, shrink
from synth.configs import TINY

pytestmark = pytest.mark.gpu

F32_TOL = 1e-4
BF16_ABS = 3e-2
PAGE = 64

CASES = [
    # name, shape, B, cap (multiple of 64), tc_min_batch
    ("f32_hd32", shrink(TINY, kv=2, g=2, half=16, ffn=256, vocab=512, layers=2), 3, 256, 0),
    ("bf16_hd128_cluster", shrink(WORKLOADS["llama8b_b1"].shape, layers=2, kv=2, ffn=256, vocab=512), 2, 256, 0),
    ("bf16_hd128_persistent", shrink(WORKLOADS["llama8b_b1"].shape, layers=2, kv=2, ffn=256, vocab=512), 3, 256, 0),
    ("bf16_tensor_core", shrink(WORKLOADS["llama8b_b1"].shape, layers=2, kv=2, ffn=512, vocab=1000), 17, 192, 1),
]


def close(gl, ol, f32):
    if f32:
        return float(np.max(np.abs(gl - ol))) / float(ol.max() - ol.min()) <= F32_TOL
    return float(np.max(np.abs(gl - ol))) <= BF16_ABS


@pytest.mark.parametrize("name,shape,B,cap,tc", CASES, ids=[c[0] for c in CASES])
def test_identity_table_is_decode_rows(name, shape, B, cap, tc):
    blob = synth.model_blob(shape, 501)
    g = pkg.Model(shape, blob, max_batch=B, max_seq=cap, tc_min_batch=tc)
    P = min(cap - 1, 130)
    toks = synth.tokens(502, 0, B * (P + 1), shape.vocab).reshape(B, P + 1)
    g.prefill(toks[:, :P], 0, logits=False)
    pos = np.array([(P - 37 * b) % (P + 1) for b in range(B)], np.int32)
    cur = toks[np.arange(B), pos].astype(np.int32)
    per_row = cap // PAGE
    table = np.arange(B * per_row, dtype=np.int32).reshape(B, per_row)
    a = g.decode_paged(cur, pos, table)
    b_ = g.decode_rows(cur, pos)
    assert np.array_equal(a.view(np.uint32), b_.view(np.uint32))
    g.close()


@pytest.mark.parametrize("name,shape,B,cap,tc", CASES, ids=[c[0] for c in CASES])
def test_scattered_pages_match_oracle(name, shape, B, cap, tc):
    f32 = not shape.bf16
    blob = synth.model_blob(shape, 511, wstd=0.05 if f32 else 0.02)
    g = pkg.Model(shape, blob, max_batch=B, max_seq=cap, tc_min_batch=tc)
    S = 150  # three pages per row
    per_row = cap // PAGE
    need = (S + PAGE - 1) // PAGE
    rng = np.random.default_rng(512)
    perm = rng.permutation(B * per_row).astype(np.int32)
    table = np.zeros((B, need), np.int32)
    for b in range(B):
        table[b] = perm[b * need:(b + 1) * need]
    toks = synth.tokens(513, 0, B * S, shape.vocab).reshape(B, S)
    rows = sorted({0, B // 2, B - 1})
    refs = {b: oracle.Model(oracle.cfg_of(shape, 1, cap), blob) for b in rows}
    check_at = {0, 63, 64, 100, S - 1}
    for s in range(S):
        lg = g.decode_paged(toks[:, s], np.full(B, s, np.int32), table)
        for b in rows:
            ol = refs[b].forward(0, int(toks[b, s]), s, logits=s in check_at)
            if s in check_at:
                assert close(lg[b], ol, f32), (name, s, b)
    for r in refs.values():
        r.close()
    g.close()


def test_step_paged_ids():
    name, shape, B, cap, tc = CASES[2]
    blob = synth.model_blob(shape, 521)
    g = pkg.Model(shape, blob, max_batch=B, max_seq=cap)
    per_row = cap // PAGE
    table = np.arange(B * per_row, dtype=np.int32)[::-1].copy().reshape(B, per_row)
    toks = synth.tokens(522, 0, B * 70, shape.vocab).reshape(B, 70)
    for s in range(69):
        g.decode_paged(toks[:, s], np.full(B, s, np.int32), table)
    pos = np.full(B, 69, np.int32)
    ids, lg = g.step_paged(toks[:, 69], pos, table, logits=True)
    for b in range(B):
        assert int(ids[b]) == oracle.argmax(lg[b])
    u = synth.uniforms(523, 0, B)
    ids, lg = g.step_paged(toks[:, 69], pos, table, temp=0.9, k=30, p=0.8, u=u, logits=True)
    for b in range(B):
        assert int(ids[b]) == oracle.sample(lg[b], 0.9, 30, 0.8, float(u[b]))
    g.close()


def test_paged_errors():
    name, shape, B, cap, tc = CASES[0]
    blob = synth.model_blob(shape, 531)
    g = pkg.Model(shape, blob, max_batch=B, max_seq=cap)
    per_row = cap // PAGE
    toks = np.array([1, 2, 3], np.int32)
    ok_table = np.arange(B * per_row, dtype=np.int32).reshape(B, per_row)
    cases = [
        (np.zeros(3, np.int32), np.where(ok_table == 0, B * per_row, ok_table), pkg.LLM_ERR_ARG),  # page outside
        (np.array([0, 0, per_row * PAGE], np.int32), ok_table, pkg.LLM_ERR_POS_RANGE),
        (np.array([0, 0, 64], np.int32), ok_table[:, :1], pkg.LLM_ERR_POS_RANGE),   # past its pages
        (np.zeros(3, np.int32), np.zeros((3, per_row + 1), np.int32), pkg.LLM_ERR_ARG),  # too many pages
        (np.zeros(3, np.int32), np.full((3, per_row), -1, np.int32), pkg.LLM_ERR_ARG),
    ]
    for pos, table, code in cases:
        with pytest.raises(pkg.LlmError) as e:
            g.decode_paged(toks, pos, table)
        assert e.value.status == code, (pos, code)
    with pytest.raises(pkg.LlmError) as e:
        g.decode_paged(np.zeros(4, np.int32), np.zeros(4, np.int32), np.zeros((4, per_row), np.int32))
    assert e.value.status == pkg.LLM_ERR_BATCH
    g.close()
    h = pkg.Model(shape, blob, max_batch=B, max_seq=100)  # not a multiple of 64: no pages
    with pytest.raises(pkg.LlmError) as e:
        h.decode_paged(toks, np.zeros(3, np.int32), np.zeros((3, 1), np.int32))
    assert e.value.status == pkg.LLM_ERR_CONFIG
    h.close()
