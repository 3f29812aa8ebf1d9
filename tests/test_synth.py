"""The seeded input generators (no GPU).  The hash and the exact uniform are the ones of
"bend-ml-llama 0.2.1.0, main.bend", section "Sampling" (hash32: Wellons' lowbias32;
uniform: top 24 bits of hash32(hash32(seed) + n) times 2^-24)."""
import numpy as np

import synth
from synth import WORKLOADS, weight_count


def _lowbias32(x):
    x &= 0xFFFFFFFF
    x ^= x >> 16
    x = (x * 0x7FEB352D) & 0xFFFFFFFF
    x ^= x >> 15
    x = (x * 0x846CA68B) & 0xFFFFFFFF
    x ^= x >> 16
    return x


def test_hash_is_lowbias32_and_injective_on_a_sample():
    rng = np.random.default_rng(0)
    xs = [0, 1, 2, 0xFFFFFFFF] + [int(v) for v in rng.integers(0, 2**32, 2000)]
    hs = [synth.hash32(x) for x in xs]
    assert hs == [_lowbias32(x) for x in xs]
    assert synth.hash32(0) == 0
    assert len(set(hs)) == len(set(xs))


def test_uniform_is_exact_24_bit():
    u = synth.uniforms(4003, 0, 100000)
    assert u.min() >= 0 and u.max() < 1
    assert np.all((u * 2**24) == np.floor(u * 2**24))
    assert synth.uniform(4003, 17) == u[17]
    assert synth.uniform(4003, 17) == (_lowbias32(_lowbias32(4003) + 17) >> 8) / 2**24
    assert abs(u.mean() - 0.5) < 0.01


def test_tokens_in_range_and_deterministic():
    for V in (256, 49152, 128256):
        t = synth.tokens(2003, 0, 50000, V)
        assert t.min() >= 0 and t.max() < V
        assert np.array_equal(t[100:200], synth.tokens(2003, 100, 100, V))


def test_normal_statistics_and_thread_independence():
    a = synth.normal(1, 5, 400000, std=0.02, bf16=False)
    assert abs(a.mean()) < 2e-4 and abs(a.std() - 0.02) < 2e-4
    b = synth.normal(1, 5, 400000, std=0.02, bf16=True)
    f = synth.bf16_to_f32(b)
    assert np.max(np.abs(f - a)) <= np.max(np.abs(a)) * 2**-8
    lib = synth.lib()
    c = np.empty(400000, np.float32)
    lib.synth_normal(1, 5, 400000, 0.0, 0.02, 0, c.ctypes.data, 1)
    assert np.array_equal(a, c)


def test_blob_size_and_gains():
    w = WORKLOADS["tiny_f32"]
    blob = synth.model_blob(w.shape, w.seed_weights)
    assert blob.size == weight_count(w.shape) == 108864
    from tests.blob import views
    v = views(w.shape, blob)
    assert np.all(v[(0, "ln1")] == 1) and np.all(v["lnf"] == 1)
    assert abs(v["emb"].std() - 0.02) < 0.002
