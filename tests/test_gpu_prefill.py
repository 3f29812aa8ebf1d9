"""Prefill through passes of prompt tokens (Llama 3.1 8B Instruct card, attention.linnet
prefill<S>: token i of the prompt sees positions s <= pos + i), against the oracle's prefill
(S successive single-token steps, P1 forward_pre) — needs a GPU.

A pass is one step whose rows are prompt tokens: the projections run on the tensor cores once a
pass holds tc_min_batch tokens, every token's key and value are written before the attention
reads them, and only the last token of each row reaches the LM head.  Cases: the 8B per-head
shape (head 128, 4 query heads per kv head, llama3 RoPE, untied head) at S = 64 and 300, B = 1
and 3; one pass and several (a ragged last pass); a second prefill that continues the rows; the
weight-streaming path for the same passes; the full 8B width at S = 64; an f32 model.  Checks:
logits after the prompt within 3e-2 (f32 model: 1e-4 of the range) with the oracle's argmax,
the cache contents, and a decode step after the prompt.
"""
import numpy as np
import pytest

import llama_architecture_kv_gb300 as pkg
import oracle
import synth
from synth import WORKLOADS, shrink
from synth.configs import TINY
from tests.oracle_rows import run_rows

pytestmark = pytest.mark.gpu

BF16_ABS = 3e-2
F32_TOL = 1e-4

L8 = WORKLOADS["llama8b_b1"].shape
HEAD128 = shrink(L8, layers=2, kv=2, ffn=2048, vocab=2000)   # d 1024: the 8B head shape
WIDE8B = shrink(L8, layers=2, ffn=4096, vocab=2000)          # d 4096, 8 kv heads
F32 = shrink(TINY, kv=2, g=2, half=16, ffn=256, vocab=512, layers=2)


def _check(lg, lo, f32):
    if f32:
        assert float(np.max(np.abs(lg - lo))) <= F32_TOL * float(lo.max() - lo.min())
    else:
        assert float(np.max(np.abs(lg - lo))) <= BF16_ABS, float(np.max(np.abs(lg - lo)))
        assert int(np.argmax(lg)) == oracle.argmax(lo)


def _cache_close(gk, ok, f32, first_layer, what):
    """Cache rows against the oracle's.  bf16 caches: layer 0's keys and values come from the
    exact embeddings, so the two sides round the same f32 sums and differ only where the sum
    lies within rounding of a bf16 tie (one unit in the last place, or the f32 sum's absolute
    error for values near zero); later layers read
    attention over those cached values, so their inputs (and roundings) drift a little more.
    (The tensor cores accumulate the f32 sums in their own order and rounding, so a few per cent
    of the roundings differ by one unit even in layer 0.)"""
    if f32:
        np.testing.assert_allclose(gk, ok, rtol=0, atol=1e-5 * max(1.0, float(np.max(np.abs(ok)))))
        return
    fa, fb = synth.bf16_to_f32(gk), synth.bf16_to_f32(ok)
    same = float(np.mean(gk == ok))
    if first_layer:
        # one unit in the last place of the value, or a small absolute error of the f32 sum
        # (values near zero)
        assert np.all(np.abs(fa - fb) <= 2 ** -7 * np.abs(fb) + 1e-4 * np.max(np.abs(fb))), what
        assert same > 0.9, (what, same)
    else:
        assert np.max(np.abs(fa - fb)) <= 2 ** -6 * np.max(np.abs(fb)), (what, float(np.max(np.abs(fa - fb))))
        assert same > 0.75, (what, same)


CASES = [
    # name, shape, B, S (prompt chunks), max_tokens, tc_min_batch
    ("head128_b1_s64", HEAD128, 1, [64], 0, 0),
    ("head128_b1_s300", HEAD128, 1, [300], 0, 0),
    ("head128_b3_s300", HEAD128, 3, [300], 0, 0),
    ("head128_b3_passes_of_48", HEAD128, 3, [100], 48, 0),
    ("head128_b3_two_prompts", HEAD128, 3, [40, 57], 64, 0),
    ("head128_b3_gemv_passes", HEAD128, 3, [70], 64, 1 << 20),
    ("wide8b_b1_s64", WIDE8B, 1, [64], 0, 0),
    ("f32_b2_passes", F32, 2, [45, 20], 32, 0),
]


@pytest.mark.parametrize("name,shape,B,chunks,mt,tc", CASES, ids=[c[0] for c in CASES])
def test_prefill_passes_match_oracle(name, shape, B, chunks, mt, tc):
    f32 = not shape.bf16
    wstd = 0.05 if f32 else 0.02
    S = sum(chunks)
    cap = S + 8
    seed = 701
    toks = synth.tokens(seed + 1, 0, B * (S + 1), shape.vocab).reshape(B, S + 1)
    tasks = []
    for b in range(B):
        parts, p0 = [], 0
        for c in chunks:
            parts.append(toks[b, p0:p0 + c])
            p0 += c
        tasks.append(dict(shape=shape, seed=seed, wstd=wstd, cap=cap, prompts=parts, steps=[toks[b, S]],
                          kv=[0, shape.layers - 1]))
    refs = run_rows(tasks)  # (spawned workers; before the first GPU call of this test)
    blob = synth.model_blob(shape, seed, wstd=wstd)
    g = pkg.Model(shape, blob, max_batch=B, max_seq=cap, tc_min_batch=tc, max_tokens=mt)
    p0 = 0
    for ci, c in enumerate(chunks):
        lg = g.prefill(toks[:, p0:p0 + c], p0)
        p0 += c
        for b in range(B):
            _check(lg[b], refs[b]["prefill"][ci], f32)
    assert [g.filled(b) for b in range(B)] == [S] * B
    for layer in (0, shape.layers - 1):
        for b in range(B):
            gk, gv = g.kv_export(layer, b, 0, S)
            ok, ov = refs[b]["kv"][layer]
            _cache_close(gk, ok[:, :S], f32, layer == 0, ("keys", layer, b))
            _cache_close(gv, ov[:, :S], f32, layer == 0, ("values", layer, b))
    ids, lg = g.step(toks[:, S], S, logits=True)
    for b in range(B):
        _check(lg[b], refs[b]["steps"][0], f32)
        assert int(ids[b]) == oracle.argmax(lg[b])
    g.close()


def test_prefill_passes_equal_decode_steps_on_the_weight_streaming_path():
    # a pass of the f32 model runs the same kernels as a decode step of as many rows; the logits
    # after the prompt agree with S chained decode steps (not bit for bit: other batch shapes)
    shape = F32
    blob = synth.model_blob(shape, 711, wstd=0.05)
    toks = synth.tokens(712, 0, 2 * 20, shape.vocab).reshape(2, 20)
    a = pkg.Model(shape, blob, max_batch=2, max_seq=32, max_tokens=16)
    lg = a.prefill(toks, 0)
    b = pkg.Model(shape, blob, max_batch=2, max_seq=32)
    for i in range(20):
        lg2 = b.decode(toks[:, i], i)
    for r in range(2):
        assert float(np.max(np.abs(lg[r] - lg2[r]))) <= F32_TOL * float(lg2[r].max() - lg2[r].min())
    a.close()
    b.close()


def test_prefill_device_tokens_equal_host_tokens():
    torch = pytest.importorskip("torch")
    shape = HEAD128
    blob = synth.model_blob(shape, 721)
    toks = synth.tokens(722, 0, 3 * 50, shape.vocab).reshape(3, 50)
    g = pkg.Model(shape, blob, max_batch=3, max_seq=64, max_tokens=40)
    host = g.prefill(toks, 0)
    td = torch.from_numpy(toks).cuda()
    out = torch.empty((3, shape.vocab), dtype=torch.float32, device="cuda")
    pkg.llm_prefill_dev(g.h, td, 3, 50, 0, out)
    g.synchronize()
    assert np.array_equal(out.cpu().numpy(), host)
    g.close()
