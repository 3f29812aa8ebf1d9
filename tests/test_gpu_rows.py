"""Rows at their own positions (Llama 3.1 8B Instruct card, "Entries": decode_rows): each row
of a batch takes its token at its own position and attends over its own cache prefix.

Parity against the oracle row by row (the oracle's rows are independent single-row models), on
every attention variant: f32 caches (CUDA-core kernel), bf16 head size 128 in 8-CTA clusters
(B <= 2) and in the persistent split (B > 2), head size 64, and the tensor-core projections.
Tolerances as in test_gpu_parity.  With every position equal the step is llm_decode bit for bit.
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

CASES = [
    # name, shape, B, cap, positions of the first step, tc_min_batch (0: default)
    ("f32_hd32", shrink(TINY, kv=2, g=2, half=16, ffn=256, vocab=512, layers=2), 3, 200, [5, 150, 64], 0),
    ("bf16_hd128_cluster", shrink(WORKLOADS["llama8b_b1"].shape, layers=2, kv=2, ffn=256, vocab=512),
     2, 400, [3, 301], 0),
    ("bf16_hd128_persistent", shrink(WORKLOADS["llama8b_b1"].shape, layers=2, kv=2, ffn=256, vocab=512),
     5, 400, [0, 17, 299, 160, 33], 0),
    ("bf16_hd64_g3", shrink(WORKLOADS["smollm2_135m"].shape, layers=2, ffn=256, vocab=512),
     4, 300, [250, 1, 96, 15], 0),
    ("bf16_tensor_core", shrink(WORKLOADS["llama8b_b1"].shape, layers=2, kv=2, ffn=512, vocab=1000),
     17, 120, [(7 * b + 3) % 100 for b in range(17)], 1),
]


def close(gl, ol, f32):
    if f32:
        return float(np.max(np.abs(gl - ol))) / float(ol.max() - ol.min()) <= F32_TOL
    return float(np.max(np.abs(gl - ol))) <= BF16_ABS


@pytest.mark.parametrize("name,shape,B,cap,pos,tc", CASES, ids=[c[0] for c in CASES])
def test_decode_rows_matches_oracle_per_row(name, shape, B, cap, pos, tc):
    f32 = not shape.bf16
    blob = synth.model_blob(shape, 301, wstd=0.05 if f32 else 0.02)
    g = pkg.Model(shape, blob, max_batch=B, max_seq=cap, tc_min_batch=tc)
    P = max(pos)
    toks = synth.tokens(302, 0, B * (P + 3), shape.vocab).reshape(B, P + 3)
    if P:
        g.prefill(toks[:, :P], 0, logits=False)  # every row filled to P; each then rewinds to its own
    pos = np.array(pos, np.int32)
    rows = sorted({0, B // 2, B - 1})
    refs = {b: oracle.Model(oracle.cfg_of(shape, 1, cap), blob) for b in rows}
    for b in rows:
        if pos[b]:
            refs[b].prefill(0, toks[b, :pos[b]], 0, logits=False)
    cur = toks[np.arange(B), pos].astype(np.int32)
    for step in range(2):
        lg = g.decode_rows(cur, pos + step)
        for b in rows:
            ol = refs[b].forward(0, int(cur[b]), int(pos[b]) + step)
            assert close(lg[b], ol, f32), (name, step, b)
        for b in range(B):
            assert pkg.llm_filled(g.h, b) == int(pos[b]) + step + 1
        cur = np.argmax(lg, axis=1).astype(np.int32)
    for r in refs.values():
        r.close()
    g.close()


@pytest.mark.parametrize("name,shape,B,cap,pos,tc", CASES, ids=[c[0] for c in CASES])
def test_equal_positions_are_decode_bit_for_bit(name, shape, B, cap, pos, tc):
    blob = synth.model_blob(shape, 303)
    g = pkg.Model(shape, blob, max_batch=B, max_seq=cap, tc_min_batch=tc)
    t = min(cap - 2, 37)
    toks = synth.tokens(304, 0, B * (t + 1), shape.vocab).reshape(B, t + 1)
    g.prefill(toks[:, :t], 0, logits=False)
    a = g.decode(toks[:, t], t)
    b_ = g.decode_rows(toks[:, t], np.full(B, t, np.int32))
    assert np.array_equal(a.view(np.uint32), b_.view(np.uint32))
    g.close()


def test_step_rows_greedy_and_sampled_ids():
    name, shape, B, cap, pos, tc = CASES[2]
    blob = synth.model_blob(shape, 305)
    g = pkg.Model(shape, blob, max_batch=B, max_seq=cap)
    P = max(pos)
    toks = synth.tokens(306, 0, B * (P + 1), shape.vocab).reshape(B, P + 1)
    g.prefill(toks[:, :P], 0, logits=False)
    pos = np.array(pos, np.int32)
    cur = toks[np.arange(B), pos].astype(np.int32)
    ids, lg = g.step_rows(cur, pos, logits=True)
    for b in range(B):
        assert int(ids[b]) == oracle.argmax(lg[b])
    ref = g.decode_rows(cur, pos)  # the same step again (rewound): the same logits
    assert np.array_equal(lg.view(np.uint32), ref.view(np.uint32))
    u = synth.uniforms(307, 0, B)
    ids, lg = g.step_rows(cur, pos, temp=0.8, k=50, p=0.9, u=u, logits=True)
    for b in range(B):
        assert int(ids[b]) == oracle.sample(lg[b], 0.8, 50, 0.9, float(u[b]))
    g.close()


def test_row_position_errors():
    shape = CASES[0][1]
    blob = synth.model_blob(shape, 308)
    g = pkg.Model(shape, blob, max_batch=3, max_seq=16)
    toks = np.array([1, 2, 3], np.int32)
    g.prefill(synth.tokens(309, 0, 3 * 4, shape.vocab).reshape(3, 4), 0, logits=False)
    for bad, code in (([0, 5, 0], pkg.LLM_ERR_POS_RANGE),    # past row 1's filled length (4)
                      ([0, -1, 0], pkg.LLM_ERR_POS_RANGE),
                      ([0, 16, 0], pkg.LLM_ERR_POS_RANGE)):  # outside the cache
        with pytest.raises(pkg.LlmError) as e:
            g.decode_rows(toks, np.array(bad, np.int32))
        assert e.value.status == code
    with pytest.raises(pkg.LlmError) as e:
        g.decode_rows(np.array([1, 2, 3, 4], np.int32), np.zeros(4, np.int32))
    assert e.value.status == pkg.LLM_ERR_BATCH
    with pytest.raises(pkg.LlmError) as e:
        g.decode_rows(np.array([1, 2, shape.vocab], np.int32), np.array([4, 4, 4], np.int32))
    assert e.value.status == pkg.LLM_ERR_TOKEN_RANGE
    # a rejected call changes nothing: the rows keep their filled lengths
    assert [pkg.llm_filled(g.h, b) for b in range(3)] == [4, 4, 4]
    g.decode_rows(toks, np.array([4, 0, 2], np.int32))
    assert [pkg.llm_filled(g.h, b) for b in range(3)] == [5, 1, 3]
    g.close()
