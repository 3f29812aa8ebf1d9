"""Generation inside CUDA graphs (Llama 3.1 8B Instruct card, "Entries": generate<Steps>,
sample<Steps>): n chained decode + draw steps without host work between them.

The ids must equal those of n chained llm_step calls bit for bit (same kernels, same order),
and the oracle, replaying the generated stream, must agree with every greedy pick up to a
near-tie within the logit tolerance.
"""
import numpy as np
import pytest

import llama_architecture_kv_gb300 as pkg
import oracle
import synth
from synth import WORKLOADS, shrink
from synth.configs import TINY

pytestmark = pytest.mark.gpu

CASES = [
    # name, shape, B, cap, prompt, tc_min_batch
    ("f32_tiny", shrink(TINY, kv=2, g=2, ffn=256, vocab=512, layers=2), 2, 64, 9, 0),
    ("bf16_hd128_b1", shrink(WORKLOADS["llama8b_b1"].shape, layers=2, kv=2, ffn=256, vocab=512), 1, 64, 20, 0),
    ("bf16_hd128_b3", shrink(WORKLOADS["llama8b_b1"].shape, layers=2, kv=2, ffn=256, vocab=512), 3, 64, 20, 0),
    ("bf16_tensor_core", shrink(WORKLOADS["llama8b_b1"].shape, layers=2, kv=2, ffn=512, vocab=1000), 17, 48, 6, 1),
]
N = 11  # one graph of 8 steps, then 3 single steps


def setup(shape, B, cap, P, tc, seed):
    blob = synth.model_blob(shape, seed, wstd=0.05 if not shape.bf16 else 0.02)
    g = pkg.Model(shape, blob, max_batch=B, max_seq=cap, tc_min_batch=tc)
    toks = synth.tokens(seed + 1, 0, B * P, shape.vocab).reshape(B, P)
    lg = g.prefill(toks, 0)
    first = np.argmax(lg, axis=1).astype(np.int32)
    return blob, g, toks, first


@pytest.mark.parametrize("sampled", [False, True], ids=["greedy", "sampled"])
@pytest.mark.parametrize("name,shape,B,cap,P,tc", CASES, ids=[c[0] for c in CASES])
def test_generate_equals_chained_steps(name, shape, B, cap, P, tc, sampled):
    blob, g, toks, first = setup(shape, B, cap, P, tc, 401)
    temp, k, p = (0.8, 40, 0.9) if sampled else (0.0, 1, 1.0)
    u = synth.uniforms(403, 0, N * B).reshape(N, B) if sampled else None
    ids = g.generate(first, P, N, temp, k, p, u)
    assert [pkg.llm_filled(g.h, b) for b in range(B)] == [P + N] * B
    kv_gen = [g.kv_export(layer, b, P, N) for layer in range(shape.layers) for b in range(B)]
    # the same steps one call at a time, rewound to the prompt end
    cur = first
    for s in range(N):
        nxt = g.step(cur, P + s, temp, k, p, None if u is None else u[s])
        assert np.array_equal(nxt, ids[s]), (name, s)
        cur = nxt
    kv_step = [g.kv_export(layer, b, P, N) for layer in range(shape.layers) for b in range(B)]
    for (k1, v1), (k2, v2) in zip(kv_gen, kv_step):
        assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
    g.close()


def test_generate_oracle_replay():
    name, shape, B, cap, P, tc = CASES[0]
    blob, g, toks, first = setup(shape, B, cap, P, tc, 411)
    ids = g.generate(first, P, N)
    for b in range(B):
        ref = oracle.Model(oracle.cfg_of(shape, 1, cap), blob)
        ref.prefill(0, toks[b], 0, logits=False)
        cur = int(first[b])
        for s in range(N):
            ol = ref.forward(0, cur, P + s)
            pick = int(ids[s, b])
            tol = 1e-4 * float(ol.max() - ol.min())
            # the greedy pick is the oracle's, unless the two are tied within the tolerance
            assert pick == oracle.argmax(ol) or ol[pick] >= ol.max() - 2 * tol, (b, s)
            cur = pick
        ref.close()
    g.close()


def test_generate_dev_matches_host():
    torch = pytest.importorskip("torch")
    name, shape, B, cap, P, tc = CASES[2]
    blob, g, toks, first = setup(shape, B, cap, P, tc, 421)
    u = synth.uniforms(423, 0, N * B).reshape(N, B)
    ids_h = g.generate(first, P, N, 0.7, 1000, 0.95, u)
    dev = torch.device("cuda", 0)
    tok_d = torch.from_numpy(first).to(dev)
    u_d = torch.from_numpy(np.ascontiguousarray(u)).to(dev)
    ids_d = torch.empty((N, B), dtype=torch.int32, device=dev)
    pkg.llm_generate_dev(g.h, tok_d, B, P, N, 0.7, 1000, 0.95, u_d, ids_d)
    pkg.llm_synchronize(g.h)
    assert np.array_equal(ids_d.cpu().numpy(), ids_h)
    g.close()


def test_generate_errors():
    name, shape, B, cap, P, tc = CASES[0]
    blob, g, toks, first = setup(shape, B, cap, P, tc, 431)
    for args, code in (((first, P, 0), pkg.LLM_ERR_ARG),              # no steps
                       ((first, P, cap - P + 1), pkg.LLM_ERR_POS_RANGE),  # past the cache
                       ((first, P + 1, 2), pkg.LLM_ERR_POS_RANGE)):   # past the filled length
        with pytest.raises(pkg.LlmError) as e:
            g.generate(*args)
        assert e.value.status == code
    bad_u = np.full((2, B), 1.0, np.float32)
    with pytest.raises(pkg.LlmError) as e:
        g.generate(first, P, 2, 0.8, 10, 0.9, bad_u)
    assert e.value.status == pkg.LLM_ERR_ARG
    assert [pkg.llm_filled(g.h, b) for b in range(B)] == [P] * B
    g.close()
    t = pkg.Model(shape, blob, max_batch=B, max_seq=cap, debug_trace=True)
    t.prefill(toks, 0, logits=False)
    with pytest.raises(pkg.LlmError) as e:
        t.generate(first, P, 2)
    assert e.value.status == pkg.LLM_ERR_ARG
    t.close()
