"""The allocation-free sampler entry point, checked against the handle-based one and the oracle
(needs a GPU).

llm_sample_noalloc is for callers that cannot allocate device memory: code running inside an
allocator or memory-pool callback, plugins whose host application owns all device memory, or
processes that reserved every byte up front.  It keeps its sort buffers in one fixed device
array inside the library instead of a handle's allocations.  Its ids must equal llm_sample_dev's
and the oracle sampler's bit for bit, including on consecutive calls that reuse that array, and
a call after the first must not change the device's free memory.
"""
import numpy as np
import pytest

import llama_architecture_kv_gb300 as pkg
import oracle
import synth
from synth import shrink
from synth.configs import TINY

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("V,B", [(49152, 4), (128256, 2)])
def test_noalloc_sampler_matches_handle_sampler_and_oracle_on_consecutive_calls(V, B):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(V)
    # top-k, top-p over the whole vocabulary, greedy, and top-k again: each call reuses the
    # array the previous one left behind
    cases = [(0.8, 50, 0.9), (0.7, V, 0.95), (0.0, 1, 1.0), (1.3, 7, 0.5)]
    stream = torch.cuda.current_stream().cuda_stream
    logits_h = [(rng.standard_normal((B, V)) * 2).astype(np.float32) for _ in cases]
    us = [synth.uniforms(4100 + call, 0, B) for call in range(len(cases))]
    # every device buffer exists before the first call, so the free memory can be compared
    logits = [torch.from_numpy(x).cuda() for x in logits_h]
    u = [torch.from_numpy(x).cuda() for x in us]
    got = [torch.full((B,), -1, dtype=torch.int32, device="cuda") for _ in cases]
    torch.cuda.synchronize()
    # first call on the device (in a fresh process it loads the array's module)
    temp, k, p = cases[0]
    pkg.llm_sample_noalloc(logits[0], B, V, temp, k, p, u[0], got[0], stream)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for call, (temp, k, p) in enumerate(cases):
        pkg.llm_sample_noalloc(logits[call], B, V, temp, k, p, u[call], got[call], stream)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0, "a warm call changed the free device memory"
    # the same draws through a handle, and through the oracle's sampler on the same logits
    s = shrink(TINY, vocab=V)
    g = pkg.Model(s, synth.model_blob(s, 9), max_batch=B, max_seq=4)
    for call, (temp, k, p) in enumerate(cases):
        want = torch.empty(B, dtype=torch.int32, device="cuda")
        pkg.llm_sample_dev(g.h, logits[call], B, temp, k, p, u[call], want)
        g.synchronize()
        assert torch.equal(got[call], want), (call, got[call].tolist(), want.tolist())
        ids = got[call].cpu().numpy()
        for b in range(B):
            ref = (oracle.argmax(logits_h[call][b]) if temp == 0 else
                   oracle.sample(logits_h[call][b], temp, k, p, float(us[call][b])))
            assert int(ids[b]) == ref, (call, b)
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
