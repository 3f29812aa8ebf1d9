"""Packed prefill (Llama 3.1 8B Instruct card, "Entries": prefill_packed): prompts packed end to
end, each token attending to its own prompt's tokens up to itself, against the oracle's
or_prefill_packed (pinned in test_oracle_pins.py).

Every case packs more tokens than one pass holds (max_tokens: several passes), interleaves the
prompts, and continues a row with a second prompt that must not see the first (its attention
starts at its own first position, inside a 16-position chunk).  Attention variants: f32 caches (CUDA-core
kernel), bf16 head size 128 in clusters and in the persistent split, and the tensor-core
projections.
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

LLAMA_LIKE = shrink(WORKLOADS["llama8b_b1"].shape, layers=2, kv=2, ffn=256, vocab=512)
CASES = [
    # name, shape, max_batch, cap, tc_min_batch
    ("f32_hd32", shrink(TINY, kv=2, g=2, half=16, ffn=256, vocab=512, layers=2), 4, 128, 0),
    ("bf16_hd128_cluster", LLAMA_LIKE, 8, 128, 0),
    ("bf16_hd128_persistent", LLAMA_LIKE, 16, 128, 0),
    ("bf16_tensor_core", shrink(WORKLOADS["llama8b_b1"].shape, layers=2, kv=2, ffn=512, vocab=1000), 17, 128, 1),
]


def pack(shape, seed):
    """Three prompts: A (row 0, positions 0..20), B (row 1, 0..36), C (row 0, 21..35: continues
    row 0 after A, starting inside a chunk); tokens interleaved, each prompt in order."""
    spans = [(0, 0, 21), (1, 0, 37), (0, 21, 15)]
    toks, rows, pos, seg = [], [], [], []
    streams = [list(range(lo, lo + n)) for _, lo, n in spans]
    k = 0
    while any(streams):
        for s, (row, lo, n) in enumerate(spans):
            if streams[s]:
                p = streams[s].pop(0)
                toks.append(int(synth.tokens(seed, k, 1, shape.vocab)[0]))
                rows.append(row)
                pos.append(p)
                seg.append(7 + s)
                k += 1
    toks, rows, pos, seg = (np.array(a, np.int32) for a in (toks, rows, pos, seg))
    last = [int(np.where((seg == 7 + s) & (pos == lo + n - 1))[0][0]) for s, (_, lo, n) in enumerate(spans)]
    return toks, rows, pos, seg, np.array(last, np.int32)


@pytest.mark.parametrize("name,shape,mb,cap,tc", CASES, ids=[c[0] for c in CASES])
def test_packed_prefill_matches_oracle(name, shape, mb, cap, tc):
    f32 = not shape.bf16
    blob = synth.model_blob(shape, 601, wstd=0.05 if f32 else 0.02)
    g = pkg.Model(shape, blob, max_batch=mb, max_seq=cap, tc_min_batch=tc, max_tokens=mb)
    toks, rows, pos, seg, last = pack(shape, 602)
    assert toks.size > mb  # several passes
    lg = g.prefill_packed(toks, rows, pos, seg, last)
    ref = oracle.Model(oracle.cfg_of(shape, mb, cap), blob)
    lo = ref.prefill_packed(toks, rows, pos, seg, last)
    ref.close()
    for m in range(len(last)):
        if f32:
            assert float(np.max(np.abs(lg[m] - lo[m]))) <= F32_TOL * float(lo[m].max() - lo[m].min()), (name, m)
        else:
            assert float(np.max(np.abs(lg[m] - lo[m]))) <= BF16_ABS, (name, m)
            assert int(np.argmax(lg[m])) == oracle.argmax(lo[m])
    assert pkg.llm_filled(g.h, 0) == 36 and pkg.llm_filled(g.h, 1) == 37
    # decoding continues each row from the packed prompts (row 0 after prompt C, row 1 after B)
    nxt = np.array([int(np.argmax(lg[2])), int(np.argmax(lg[1]))], np.int32)
    if mb >= 2:
        out = g.decode_rows(nxt, np.array([36, 37], np.int32))[:2]
        assert np.all(np.isfinite(out))
    g.close()


def test_packed_prefill_errors():
    name, shape, mb, cap, tc = CASES[0]
    blob = synth.model_blob(shape, 611)
    g = pkg.Model(shape, blob, max_batch=mb, max_seq=cap)
    t = np.array([1, 2, 3], np.int32)
    bad = [
        (([0, 0, 0], [0, 2, 3], [5, 5, 5]), pkg.LLM_ERR_ARG),          # a gap in the prompt
        (([0, 1, 0], [0, 1, 2], [5, 5, 5]), pkg.LLM_ERR_ARG),          # a prompt over two rows
        (([0, 0, 0], [0, 1, 1], [5, 5, 6]), pkg.LLM_ERR_ARG),          # two tokens in one slot
        (([0, 0, 0], [0, 1, 1], [5, 5, 6][::-1]), pkg.LLM_ERR_ARG),    # overlapping prompts
        (([0, 0, mb], [0, 1, 2], [5, 5, 5]), pkg.LLM_ERR_BATCH),
        (([0, 0, 0], [0, 1, cap], [5, 5, 5]), pkg.LLM_ERR_POS_RANGE),
    ]
    for (rows, pos, seg), code in bad:
        with pytest.raises(pkg.LlmError) as e:
            g.prefill_packed(t, rows, pos, seg, [0])
        assert e.value.status == code, (rows, pos, seg)
    with pytest.raises(pkg.LlmError) as e:
        g.prefill_packed(t, [0, 0, 0], [0, 1, 2], [5, 5, 5], [3])
    assert e.value.status == pkg.LLM_ERR_ARG
    g.close()
    # any capacity (no page size involved)
    h = pkg.Model(shape, blob, max_batch=mb, max_seq=100)
    out = h.prefill_packed(t, [0, 0, 0], [0, 1, 2], [5, 5, 5], [2])
    assert np.all(np.isfinite(out)) and h.filled(0) == 3
    h.close()
