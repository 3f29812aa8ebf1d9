"""Parity of the GPU library with the oracle, through the C ABI (needs a GPU).

Tolerances: token ids and every integer decision bit-exact; the f32
model's logits within 1e-4 of the oracle's logit range; bf16-weight models within an absolute
3e-2 with greedy argmax agreement on at least 99% of decode steps.  Decoding is teacher-forced:
the oracle replays the token stream the GPU produced, so one near-tie cannot make the two runs
diverge (bend-ml-llama's blog notes free-running streams drift apart after a few hundred tokens).
"""
import multiprocessing as mp

import numpy as np
import pytest

import llama_architecture_kv_gb300 as pkg
import oracle
import synth
from synth import WORKLOADS, shrink
from synth.configs import TINY
from tests.blob import views

pytestmark = pytest.mark.gpu

F32_TOL = 1e-4      # of the logit range, f32 model
BF16_ABS = 3e-2     # absolute, bf16-weight models
ARGMAX_AGREE = 0.99


def rel_err(a, ref):
    return float(np.max(np.abs(a - ref))) / float(ref.max() - ref.min())


def make(shape, seed, B, cap, wstd=0.02, debug_trace=False):
    blob = synth.model_blob(shape, seed, wstd=wstd)
    g = pkg.Model(shape, blob, max_batch=B, max_seq=cap, debug_trace=debug_trace)
    return blob, g


def check_bf16(gl, ol, agree):
    err = float(np.max(np.abs(gl - ol)))
    assert err <= BF16_ABS, err
    agree.append(int(np.argmax(gl)) == oracle.argmax(ol))


# ---------------------------------------------------------------------------------------
# f32 tiny model (the exact workload and shape variants)
# ---------------------------------------------------------------------------------------

def run_teacher_forced(shape, blob, gpu, prompts, steps, f32=True):
    B, S = prompts.shape
    cap = gpu.cfg.max_seq
    refs = [oracle.Model(oracle.cfg_of(shape, 1, cap), blob) for _ in range(B)]
    lg = gpu.prefill(prompts, 0)
    agree = []
    for b in range(B):
        lo = refs[b].prefill(0, prompts[b], 0)
        if f32:
            assert rel_err(lg[b], lo) <= F32_TOL
        else:
            check_bf16(lg[b], lo, agree)
    toks = np.array([np.argmax(lg[b]) for b in range(B)], np.int32)
    for t in range(S, S + steps):
        ids, lg = gpu.step(toks, t, logits=True)
        for b in range(B):
            lo = refs[b].forward(0, int(toks[b]), t)
            if f32:
                assert rel_err(lg[b], lo) <= F32_TOL, (t, b, rel_err(lg[b], lo))
            else:
                check_bf16(lg[b], lo, agree)
            assert int(ids[b]) == oracle.argmax(lg[b])  # greedy id, bit-exact on the same logits
        toks = ids
    for r in refs:
        r.close()
    return agree


def test_tiny_f32_workload():
    w = WORKLOADS["tiny_f32"]
    blob, g = make(w.shape, w.seed_weights, 1, w.cap)
    prompt = synth.tokens(w.seed_tokens, 0, w.prompt, w.shape.vocab)[None]
    run_teacher_forced(w.shape, blob, g, prompt, w.steps)
    g.close()


@pytest.mark.parametrize("name,shape", [
    ("g1", shrink(TINY, kv=4, g=1)),
    ("g4_odd_ffn", shrink(TINY, kv=1, g=4, ffn=92)),
    ("untied_llama3", shrink(TINY, tied=False, llama3=True, orig_max=64.0)),
    ("g3_hd64", shrink(TINY, kv=2, g=3, half=32, ffn=200, vocab=300)),
    ("hd128_g4", shrink(TINY, kv=2, g=4, half=64, ffn=512, vocab=1000, layers=2)),
], ids=lambda x: x if isinstance(x, str) else "")
def test_tiny_f32_variants_batched(name, shape):
    B, S, steps = 3, 7, 6
    blob, g = make(shape, 77, B, 16, wstd=0.1)
    prompts = synth.tokens(78, 0, B * S, shape.vocab).reshape(B, S)
    run_teacher_forced(shape, blob, g, prompts, steps)
    g.close()


def test_long_cache_many_splits_f32():
    # enough positions that attention uses many splits and a ragged last tile
    shape = shrink(TINY, kv=2, g=2, half=32, ffn=256, vocab=512, layers=2)
    cap = 700
    blob, g = make(shape, 91, 2, cap, wstd=0.05)
    prompts = synth.tokens(92, 0, 2 * 611, shape.vocab).reshape(2, 611)
    run_teacher_forced(shape, blob, g, prompts, 3)
    g.close()


# ---------------------------------------------------------------------------------------
# laws on the GPU
# ---------------------------------------------------------------------------------------

def test_causality_future_cache_entries_never_read():
    w = WORKLOADS["tiny_f32"]
    s = w.shape
    blob, g = make(s, w.seed_weights, 1, 16)
    toks = synth.tokens(w.seed_tokens, 0, 8, s.vocab)
    g.prefill(toks[None, :6], 0, logits=False)
    a = g.decode(toks[6:7], 6)
    junk = np.full((s.kv, 16 - 7, s.hd), np.nan, np.float32)
    for layer in range(s.layers):
        g.kv_import(layer, 0, 7, junk, junk)
    b = g.decode(toks[6:7], 6)  # rewind to 6: rewrites position 6, reads 0..6 only
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    g.close()


def test_gqa_query_heads_read_their_group():
    # one layer with W_q = W_k = 0 (every score 0: uniform weights) and W_v = 0 (the new value
    # is 0); the cache holds marker(j) = (j+1) e_j at positions 0..t-1 of kv head j, so query
    # head h's output is marker(h // g) * t / (t + 1)
    s = shrink(TINY, kv=3, g=4, half=8, layers=1)
    blob = synth.model_blob(s, 5)
    v = views(s, blob)
    for name in ("q", "k", "v"):
        v[(0, name)][...] = 0
    g = pkg.Model(s, blob, max_batch=1, max_seq=8, debug_trace=True)
    t = 5
    kk = np.zeros((s.kv, t, s.hd), np.float32)
    vv = np.zeros((s.kv, t, s.hd), np.float32)
    for j in range(s.kv):
        vv[j, :, j] = j + 1
    g.kv_import(0, 0, 0, kk, vv)
    g.decode(np.array([3], np.int32), t)
    att = g.trace(0, "attn")[0].reshape(s.heads, s.hd)
    for h in range(s.heads):
        want = np.zeros(s.hd, np.float32)
        want[h // s.g] = (h // s.g + 1) * t / (t + 1)
        np.testing.assert_allclose(att[h], want, rtol=1e-6, atol=1e-7)
    g.close()


def test_deterministic_bits():
    w = WORKLOADS["tiny_f32"]
    blob, g = make(w.shape, w.seed_weights, 2, 16)
    toks = synth.tokens(w.seed_tokens, 0, 16, w.shape.vocab).reshape(2, 8)
    a = g.prefill(toks, 0)
    b = g.prefill(toks, 0)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    g.close()


def test_kv_cache_holds_rotated_keys_rounded_like_the_oracle():
    # bf16 model: the cache row written at position t equals the oracle's (same bf16 rounding of
    # the same f32 values, up to the f32 differences of the projections)
    s = shrink(WORKLOADS["smollm2_135m"].shape, layers=2, vocab=1000)
    blob, g = make(s, 31, 1, 8)
    ref = oracle.Model(oracle.cfg_of(s, 1, 8), blob)
    toks = synth.tokens(32, 0, 5, s.vocab)
    g.prefill(toks[None], 0, logits=False)
    ref.prefill(0, toks, 0, logits=False)
    for layer in range(2):
        gk, gv = g.kv_export(layer, 0, 0, 5)
        ok, ov = ref.kv_read(layer, 0, 0, 5)
        for a, b in ((gk, ok), (gv, ov)):
            fa, fb = synth.bf16_to_f32(a), synth.bf16_to_f32(b)
            assert np.max(np.abs(fa - fb)) <= 2 ** -7 * np.max(np.abs(fb)) + 1e-6
            assert np.mean(a == b) > 0.97
    g.close()
    ref.close()


# ---------------------------------------------------------------------------------------
# the sampler: bit-exact ids on identical logits and draws
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("V", [5, 256, 49152, 128256])
def test_sampler_ids_bit_exact(V):
    s = shrink(TINY, vocab=V)
    blob, g = make(s, 3, 8, 4)
    rng = np.random.default_rng(V)
    # k <= 1024 candidates: the radix-select kernel; more: the sort of the whole row
    ks = [1, 2, 50, 1000, 1024, 1025, V, V + 10]
    for trial in range(24):
        B = int(rng.integers(1, 9))
        if trial % 4 == 0:
            logits = rng.integers(-3, 4, (B, V)).astype(np.float32)  # many ties
        else:
            logits = (rng.standard_normal((B, V)) * rng.choice([0.5, 2, 8])).astype(np.float32)
        temp = float(rng.choice([0.0, 0.3, 0.7, 0.8, 1.5])) if trial >= len(ks) else 0.8
        k = int(ks[trial]) if trial < len(ks) else int(rng.choice(ks))
        p = float(rng.choice([1e-3, 0.5, 0.9, 0.95, 1.0]))
        u = synth.uniforms(4000 + trial, 0, B)
        ids = g.sample(logits, temp, k, p, u)
        for b in range(B):
            want = oracle.argmax(logits[b]) if temp == 0 else oracle.sample(logits[b], temp, k, p, float(u[b]))
            assert int(ids[b]) == want, (trial, b, temp, k, p, float(u[b]))
    g.close()


# ---------------------------------------------------------------------------------------
# errors at the boundary
# ---------------------------------------------------------------------------------------

def test_boundary_errors():
    w = WORKLOADS["tiny_f32"]
    blob, g = make(w.shape, w.seed_weights, 2, 8)
    V = w.shape.vocab

    def status(fn):
        with pytest.raises(pkg.LlmError) as e:
            fn()
        return e.value.status

    assert status(lambda: g.decode(np.array([1], np.int32), 1)) == pkg.LLM_ERR_POS_RANGE  # past filled
    assert status(lambda: g.prefill(np.ones((1, 9), np.int32), 0)) == pkg.LLM_ERR_POS_RANGE  # > cap
    assert status(lambda: g.decode(np.array([V], np.int32), 0)) == pkg.LLM_ERR_TOKEN_RANGE
    assert status(lambda: g.decode(np.array([-1], np.int32), 0)) == pkg.LLM_ERR_TOKEN_RANGE
    assert status(lambda: g.decode(np.ones(3, np.int32), 0)) == pkg.LLM_ERR_BATCH
    lg = np.zeros((1, V), np.float32)
    assert status(lambda: g.sample(lg, -1.0, 1, 1.0, [0.5])) == pkg.LLM_ERR_ARG
    assert status(lambda: g.sample(lg, 1.0, 0, 1.0, [0.5])) == pkg.LLM_ERR_ARG
    assert status(lambda: g.sample(lg, 1.0, 5, 0.0, [0.5])) == pkg.LLM_ERR_ARG
    assert status(lambda: g.sample(lg, 1.0, 5, 1.0, [1.0])) == pkg.LLM_ERR_ARG
    # a failed call leaves the handle usable
    g.prefill(np.ones((2, 3), np.int32), 0)
    assert g.filled(0) == 3 and g.filled(1) == 3
    g.close()


def test_device_token_check_reports_on_synchronize():
    torch = pytest.importorskip("torch")
    w = WORKLOADS["tiny_f32"]
    blob, g = make(w.shape, w.seed_weights, 1, 8)
    tok = torch.tensor([w.shape.vocab + 5], dtype=torch.int32, device="cuda")
    out = torch.empty((1, w.shape.vocab), dtype=torch.float32, device="cuda")
    pkg.llm_decode_dev(g.h, tok, 1, 0, out)
    with pytest.raises(pkg.LlmError) as e:
        g.synchronize()
    assert e.value.status == pkg.LLM_ERR_TOKEN_RANGE
    g.synchronize()  # cleared
    g.close()


def test_bounded_wait_timeout_is_reported_once_and_the_handle_stays_usable():
    # a wait on a barrier that nothing arrives on runs out after a few thousand cycles; the
    # status reaches llm_synchronize once, then the handle steps normally (bit-identical logits)
    w = WORKLOADS["tiny_f32"]
    blob, g = make(w.shape, w.seed_weights, 1, 8)
    toks = synth.tokens(w.seed_tokens, 0, 3, w.shape.vocab)
    before = g.decode(toks[:1], 0)
    pkg.llm_check_wait_timeout(g.h, 5000)
    with pytest.raises(pkg.LlmError) as e:
        g.synchronize()
    assert e.value.status == pkg.LLM_ERR_DEVICE_TIMEOUT
    g.synchronize()  # reported once, then cleared
    np.testing.assert_array_equal(g.decode(toks[:1], 0), before)
    with pytest.raises(pkg.LlmError) as e:
        pkg.llm_check_wait_timeout(g.h, 0)
    assert e.value.status == pkg.LLM_ERR_ARG
    g.close()


def test_device_pointer_variants_match_host_variants():
    torch = pytest.importorskip("torch")
    w = WORKLOADS["tiny_f32"]
    blob, g = make(w.shape, w.seed_weights, 2, 16)
    toks = synth.tokens(w.seed_tokens, 0, 12, w.shape.vocab).reshape(2, 6)
    host = g.prefill(toks, 0)
    td = torch.from_numpy(toks).cuda()
    out = torch.empty((2, w.shape.vocab), dtype=torch.float32, device="cuda")
    pkg.llm_prefill_dev(g.h, td, 2, 6, 0, out)
    g.synchronize()
    assert np.array_equal(out.cpu().numpy(), host)
    ids = torch.empty(2, dtype=torch.int32, device="cuda")
    u = torch.tensor([0.25, 0.75], dtype=torch.float32, device="cuda")
    pkg.llm_step_dev(g.h, td[:, 5].contiguous(), 2, 6, 0.8, 20, 0.9, u, ids, out)
    g.synchronize()
    lg = out.cpu().numpy()
    for b in range(2):
        assert int(ids[b]) == oracle.sample(lg[b], 0.8, 20, 0.9, [0.25, 0.75][b])
    g.close()


# ---------------------------------------------------------------------------------------
# bf16 models
# ---------------------------------------------------------------------------------------

def test_smollm2_135m_short():
    w = WORKLOADS["smollm2_135m"]
    blob, g = make(w.shape, w.seed_weights, 1, 64)
    prompt = synth.tokens(w.seed_tokens, 0, 24, w.shape.vocab)[None]
    agree = run_teacher_forced(w.shape, blob, g, prompt, 12, f32=False)
    assert np.mean(agree) >= ARGMAX_AGREE
    g.close()


# ---------------------------------------------------------------------------------------
# tensor-core projections (bf16 steps of at least tc_min_batch rows)
# ---------------------------------------------------------------------------------------

TC_SHAPES = [
    # 135M-like: Q/K/V rows 960 (a ragged last 128-row tile), K = 576 (9 blocks of 64)
    ("smol135_like", shrink(WORKLOADS["smollm2_135m"].shape, layers=2, vocab=8192)),
    # 8B-like: head dim 128, g 4, untied head with a ragged vocabulary, llama3 RoPE
    ("llama_like", shrink(WORKLOADS["llama8b_b1"].shape, layers=2, kv=2, ffn=1024, vocab=3000)),
    # 1.7B-like: g 1, head dim 64, MLP width 712 (a partial last K block in down)
    ("smol17_like", shrink(WORKLOADS["smollm2_1_7b_b16"].shape, layers=2, kv=4, ffn=712, vocab=2500)),
]


@pytest.mark.parametrize("name,shape", TC_SHAPES, ids=lambda x: x if isinstance(x, str) else "")
@pytest.mark.parametrize("B", [3, 17, 40])
def test_tensor_core_path_teacher_forced(name, shape, B):
    # tc_min_batch = 1 puts every step of this handle on the tensor-core path (16-, 32- and
    # 48-column tiles for B = 3, 17, 40)
    S, steps, cap = 5, 4, 12
    blob = synth.model_blob(shape, 91)
    g = pkg.Model(shape, blob, max_batch=B, max_seq=cap, tc_min_batch=1)
    prompts = synth.tokens(92, 0, B * S, shape.vocab).reshape(B, S)
    rows = sorted({0, B // 2, B - 1})
    refs = {b: oracle.Model(oracle.cfg_of(shape, 1, cap), blob) for b in rows}
    lg = g.prefill(prompts, 0)
    agree = []
    for b in rows:
        check_bf16(lg[b], refs[b].prefill(0, prompts[b], 0), agree)
    toks = np.array([np.argmax(lg[b]) for b in range(B)], np.int32)
    for t in range(S, S + steps):
        ids, lg = g.step(toks, t, logits=True)
        for b in rows:
            check_bf16(lg[b], refs[b].forward(0, int(toks[b]), t), agree)
            assert int(ids[b]) == oracle.argmax(lg[b])
        toks = ids
    assert np.mean(agree) >= ARGMAX_AGREE
    for r in refs.values():
        r.close()
    g.close()


@pytest.mark.parametrize("ffn", [6000, 17000], ids=["mlp6000", "mlp17000"])
def test_batch1_gemv_wide_mlp_teacher_forced(ffn):
    # batch 1 on the bulk-copy GEMVs with down projection inputs of 6000 and 17000 floats (wider
    # than the inputs a thread holds in registers); 17000 also keeps the prefill passes on the
    # GEMVs (wider than the tensor-core prep kernels stage): against the oracle
    shape = shrink(WORKLOADS["llama8b_b1"].shape, layers=2, kv=2, ffn=ffn, vocab=1000)
    S, steps, cap = 4, 4, 12
    blob = synth.model_blob(shape, 95)
    g = pkg.Model(shape, blob, max_batch=1, max_seq=cap)
    ref = oracle.Model(oracle.cfg_of(shape, 1, cap), blob)
    prompt = synth.tokens(96, 0, S, shape.vocab)
    agree = []
    lg = g.prefill(prompt[None], 0)
    check_bf16(lg[0], ref.prefill(0, prompt, 0), agree)
    tok = np.array([np.argmax(lg[0])], np.int32)
    for t in range(S, S + steps):
        ids, lg = g.step(tok, t, logits=True)
        check_bf16(lg[0], ref.forward(0, int(tok[0]), t), agree)
        assert int(ids[0]) == oracle.argmax(lg[0])
        tok = ids
    assert np.mean(agree) >= ARGMAX_AGREE
    ref.close()
    g.close()


def test_tensor_core_and_gemv_paths_agree():
    shape = TC_SHAPES[1][1]
    B, S, cap = 16, 6, 10
    blob = synth.model_blob(shape, 93)
    prompts = synth.tokens(94, 0, B * S, shape.vocab).reshape(B, S)
    outs = []
    for tc_min in (1, 1 << 20):
        g = pkg.Model(shape, blob, max_batch=B, max_seq=cap, tc_min_batch=tc_min)
        lg = g.prefill(prompts, 0)
        ids, lg2 = g.step(np.argmax(lg, axis=1).astype(np.int32), S, logits=True)
        outs.append((lg, lg2, ids))
        g.close()
    # the activations reach the tensor cores as bf16 hi + lo pairs (about 2^-17 relative)
    for a, b in zip(outs[0][:2], outs[1][:2]):
        assert float(np.max(np.abs(a - b))) <= 2e-3
    rng_ = outs[1][1].max(axis=1) - outs[1][1].min(axis=1)
    assert np.all(rng_ > 0)


def test_step_kernel_counts():
    shape = TC_SHAPES[0][1]
    L = shape.layers
    blob = synth.model_blob(shape, 95)
    g = pkg.Model(shape, blob, max_batch=20, max_seq=8, tc_min_batch=16)
    greedy_gemv = pkg.llm_step_kernels(g.h, 4, 0.0)
    assert greedy_gemv == 5 * L + 4  # prologue, embedding, 5 per layer, head, argmax
    # tensor-core path, per layer: split activations + GEMM for each projection, the Q/K/V finish;
    # the head: split + GEMM, and a sum of its K splits when it has more than one
    assert pkg.llm_step_kernels(g.h, 16, 0.0) - greedy_gemv in (5 * L + 1, 5 * L + 2)
    assert pkg.llm_step_kernels(g.h, 4, 0.8) == greedy_gemv + 13  # 4 passes x 3 sort kernels + init + draw
    assert pkg.llm_step_kernels(g.h, 4, 0.8, 50) == greedy_gemv  # top-50: one selection kernel
    with pytest.raises(pkg.LlmError):
        pkg.llm_step_kernels(g.h, 21, 0.0)
    g.close()


# ---------------------------------------------------------------------------------------
# bf16 caches (the tensor-core attention kernel: head sizes 64 and 128)
# ---------------------------------------------------------------------------------------

BF16_ATTN_SHAPES = [
    ("hd128_g4", shrink(WORKLOADS["llama8b_b1"].shape, layers=1, kv=2, ffn=256, vocab=512)),
    ("hd64_g3", shrink(WORKLOADS["smollm2_135m"].shape, layers=1, ffn=256, vocab=512)),
]


def bf16_bits(x):
    return np.asarray(x, np.float32).view(np.uint32).astype(np.uint64).__rshift__(16).astype(np.uint16)


@pytest.mark.parametrize("name,shape", BF16_ATTN_SHAPES, ids=lambda x: x if isinstance(x, str) else "")
@pytest.mark.parametrize("t", [5, 70, 300])
def test_gqa_markers_bf16_cache(name, shape, t):
    # as the f32 marker test: zero Q/K/V weights make every score 0, so query head h's output
    # is marker(h // g) * t / (t + 1); t spans one chunk, a ragged third chunk and many splits
    s = shape
    blob = synth.model_blob(s, 6)
    v = views(s, blob)
    for nm in ("q", "k", "v"):
        v[(0, nm)][...] = 0
    g = pkg.Model(s, blob, max_batch=1, max_seq=t + 1, debug_trace=True)
    kk = np.zeros((s.kv, t, s.hd), np.uint16)
    vv = np.zeros((s.kv, t, s.hd), np.float32)
    for j in range(s.kv):
        vv[j, :, j] = j + 1
    g.kv_import(0, 0, 0, kk, bf16_bits(vv))
    g.decode(np.array([3], np.int32), t)
    att = g.trace(0, "attn")[0].reshape(s.heads, s.hd)
    for h in range(s.heads):
        want = np.zeros(s.hd, np.float32)
        want[h // s.g] = (h // s.g + 1) * t / (t + 1)
        np.testing.assert_allclose(att[h], want, rtol=2e-6, atol=1e-7)
    g.close()


@pytest.mark.parametrize("name,shape", BF16_ATTN_SHAPES, ids=lambda x: x if isinstance(x, str) else "")
def test_causality_bf16_cache(name, shape):
    s = shape
    B, cap, t = 2, 100, 40
    blob = synth.model_blob(s, 7)
    g = pkg.Model(s, blob, max_batch=B, max_seq=cap)
    toks = synth.tokens(8, 0, B * (t + 1), s.vocab).reshape(B, t + 1)
    g.prefill(toks[:, :t], 0, logits=False)
    a = g.decode(toks[:, t], t)
    junk = np.full((s.kv, cap - t - 1, s.hd), 0x7FC0, np.uint16)  # bf16 NaN
    for layer in range(s.layers):
        for b in range(B):
            g.kv_import(layer, b, t + 1, junk, junk)
    b_ = g.decode(toks[:, t], t)
    assert np.array_equal(a.view(np.uint32), b_.view(np.uint32))
    g.close()


# ---------------------------------------------------------------------------------------
# the divergence ladder: every intermediate of a layer against the oracle's trace
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("B", [1, 3])
def test_debug_trace_every_intermediate_matches_oracle(B):
    # one bf16 step of the 8B head shape: n1, q, k, v, qr, kr, attn, a, x1, n2, m, y of both
    # layers against the oracle's trace of the same step (bend-ml-llama "A layer", Act), each
    # within a few f32 roundings of its scale
    s = shrink(WORKLOADS["llama8b_b1"].shape, layers=2, kv=2, ffn=512, vocab=700)
    blob = synth.model_blob(s, 141)
    P = 9
    toks = synth.tokens(142, 0, B * (P + 1), s.vocab).reshape(B, P + 1)
    g = pkg.Model(s, blob, max_batch=B, max_seq=16, debug_trace=True)
    g.prefill(toks[:, :P], 0, logits=False)
    g.decode(toks[:, P], P)
    for b in range(B):
        ref = oracle.Model(oracle.cfg_of(s, 1, 16), blob, trace=True)
        ref.prefill(0, toks[b, :P], 0, logits=False)
        ref.forward(0, int(toks[b, P]), P)
        for layer in range(s.layers):
            for name in ("n1", "q", "k", "v", "qr", "kr", "attn", "a", "x1", "n2", "m", "y"):
                got = g.trace(layer, name)[b]
                want = ref.trace(layer, name)
                assert got.shape == want.shape, (name, got.shape, want.shape)
                scale = float(np.max(np.abs(want))) + 1e-30
                err = float(np.max(np.abs(got - want)))
                assert err <= 2e-3 * scale, (layer, name, b, err, scale)
        ref.close()
    g.close()
