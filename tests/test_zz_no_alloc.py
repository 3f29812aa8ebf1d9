"""The allocation-free sampler entry point, checked against the handle-based one (needs a GPU).

llm_sample_noalloc is for callers that cannot allocate device memory: code running inside an
allocator or memory-pool callback, plugins whose host application owns all device memory, or
processes that reserved every byte up front.  It keeps its sort buffers in one fixed device
array inside the library instead of a handle's allocations.  Its ids must equal llm_sample_dev's
bit for bit, including on consecutive calls that reuse that array.
"""
import numpy as np
import pytest

import llama_architecture_kv_gb300 as pkg
import synth
from synth import shrink
from synth.configs import TINY

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("V,B", [(49152, 4), (128256, 2)])
def test_noalloc_sampler_matches_handle_sampler_on_consecutive_calls(V, B):
    torch = pytest.importorskip("torch")
    s = shrink(TINY, vocab=V)
    g = pkg.Model(s, synth.model_blob(s, 9), max_batch=B, max_seq=4)
    rng = np.random.default_rng(V)
    # top-k, top-p over the whole vocabulary, greedy, and top-k again: each call reuses the
    # array the previous one left behind
    cases = [(0.8, 50, 0.9), (0.7, V, 0.95), (0.0, 1, 1.0), (1.3, 7, 0.5)]
    stream = torch.cuda.current_stream().cuda_stream
    for call, (temp, k, p) in enumerate(cases):
        logits = torch.from_numpy((rng.standard_normal((B, V)) * 2).astype(np.float32)).cuda()
        u = torch.from_numpy(synth.uniforms(4100 + call, 0, B)).cuda()
        want = torch.empty(B, dtype=torch.int32, device="cuda")
        got = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        pkg.llm_sample_dev(g.h, logits, B, temp, k, p, u, want)
        g.synchronize()
        pkg.llm_sample_noalloc(logits, B, V, temp, k, p, u, got, stream)
        torch.cuda.synchronize()
        assert torch.equal(got, want), (call, got.tolist(), want.tolist())
    g.close()


def test_noalloc_sampler_rejects_sizes_over_its_fixed_array():
    torch = pytest.importorskip("torch")
    buf = torch.zeros(8, dtype=torch.float32, device="cuda")
    ids = torch.zeros(8, dtype=torch.int32, device="cuda")
    too_many_rows = pkg.SAMPLE_NOALLOC_MAX_ELEMS // 128256 + 1
    with pytest.raises(pkg.LlmError) as e:
        pkg.llm_sample_noalloc(buf, too_many_rows, 128256, 0.8, 50, 0.9, buf, ids)
    assert e.value.status == pkg.LLM_ERR_ARG
    with pytest.raises(pkg.LlmError):
        pkg.llm_sample_noalloc(buf, 1, 16, 0.8, 0, 0.9, buf, ids)  # k < 1
