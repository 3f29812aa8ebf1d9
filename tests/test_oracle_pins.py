"""Pins of the oracle to what the pages and the mathematics fix (no GPU).

Each test names the passage it pins.  Pages:
  P1 = "bend-ml-llama 0.2.1.0, main.bend"; P3 = "Llama 3.1 8B Instruct" model card.
The whole-model forward has no worked numeric example on the pages; it is pinned here by
special cases that reduce to closed forms, by invariances that a wrong index, sign or
transposed operand breaks, and by the decode == full-sequence law.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from synth import WORKLOADS, shrink
from synth.configs import LLAMA8B, SMOL135M, SMOL1_7B, TINY, Shape
from tests.blob import views

F32 = np.float32


def ulp(x):
    x = abs(float(x))
    return float(np.spacing(F32(x)))


# ---------------------------------------------------------------------------------------
# layout laws (P1 "The configuration": layout_135m / layout_360m / layout_1_7b; P3 README
# "8.03B-parameter decoder")
# ---------------------------------------------------------------------------------------

SMOL360M = Shape(kv=5, g=3, half=32, ffn=2560, layers=32, vocab=49152, eps=1e-5,
                 theta=100000.0, tied=True)


@pytest.mark.parametrize("shape,count", [(SMOL135M, 134515008), (SMOL360M, 361821120),
                                         (SMOL1_7B, 1711376384)])
def test_layout_counts_printed_on_page(shape, count):
    assert oracle.weight_count(oracle.cfg_of(shape)) == count


def test_layout_8b_matches_card():
    n = oracle.weight_count(oracle.cfg_of(LLAMA8B))
    assert n == 8030261248
    assert round(n / 1e9, 2) == 8.03


def test_config_size_laws():
    # P1 smollm2_*_sizes: hidden, query heads, head size, key width
    for s, (d, h, hd, kvw) in [(SMOL135M, (576, 9, 64, 192)), (SMOL360M, (960, 15, 64, 320)),
                               (SMOL1_7B, (2048, 32, 64, 2048))]:
        assert (s.d, s.heads, s.hd, s.kvw) == (d, h, hd, kvw)


def test_create_rejects_wrong_blob_size():
    s = TINY
    c = oracle.cfg_of(s, 1, 16)
    blob = synth.model_blob(s, 1)
    oracle.Model(c, blob).close()
    for delta in (-2, -1, 1, 2):
        n = blob.size + delta
        bad = np.zeros(max(n, 1), np.float32)[:n]
        with pytest.raises(ValueError):
            oracle.Model(c, bad)


# ---------------------------------------------------------------------------------------
# heads (P1 "Heads": law head_split)
# ---------------------------------------------------------------------------------------

def test_head_split_roundtrip_every_half():
    rng = np.random.default_rng(0)
    for n in range(0, 24):
        xs = rng.standard_normal(n).astype(F32)
        for h in range(0, n + 2):
            lo, hi = oracle.split(xs, h)
            assert lo.size == min(h, n) and hi.size == n - min(h, n)
            back = oracle.join(lo, hi)
            assert np.array_equal(back.view(np.uint32), xs.view(np.uint32))


# ---------------------------------------------------------------------------------------
# GQA mapping (P1 "Grouped-query attention": laws gqa_head, groups_len)
# ---------------------------------------------------------------------------------------

def test_gqa_head_law():
    for g in range(1, 17):
        for j in range(64):
            for i in range(g):
                assert oracle.gqa_kv_head(j * g + i, g) == j


def _model(shape, cap=8, batch=1, seed=7, blob=None, trace=False):
    c = oracle.cfg_of(shape, batch, cap)
    if blob is None:
        blob = synth.model_blob(shape, seed)
    return oracle.Model(c, blob, trace=trace), blob


def test_gqa_marker_values_reach_their_group():
    # every value of key/value head j is the marker vector (j+1) * e_j; whatever the
    # scores, the attention weights sum to one, so query head h returns marker(h // g)
    s = shrink(TINY, kv=3, g=4, half=4)
    M, _ = _model(s, cap=8)
    hd = s.hd
    rng = np.random.default_rng(1)
    for t in (0, 5):
        k = rng.standard_normal((s.kv, t + 1, hd)).astype(F32)
        v = np.zeros((s.kv, t + 1, hd), F32)
        for j in range(s.kv):
            v[j, :, j] = j + 1
        M.kv_write(0, 0, 0, k, v)
        q = rng.standard_normal(s.heads * hd).astype(F32)
        out = M.attend(0, 0, q, t).reshape(s.heads, hd)
        for h in range(s.heads):
            want = np.zeros(hd, F32)
            want[h // s.g] = h // s.g + 1
            if t == 0:
                assert np.array_equal(out[h], want)
            else:
                np.testing.assert_allclose(out[h], want, rtol=2e-6, atol=0)


# ---------------------------------------------------------------------------------------
# causality (P1 law causal; P3 attention.linnet decode: seen[s] = s <= pos)
# ---------------------------------------------------------------------------------------

def test_attention_ignores_positions_after_t():
    s = shrink(TINY, kv=2, g=2, half=4)
    M, _ = _model(s, cap=12)
    rng = np.random.default_rng(2)
    hd, t = s.hd, 6
    k = rng.standard_normal((s.kv, 12, hd)).astype(F32)
    v = rng.standard_normal((s.kv, 12, hd)).astype(F32)
    M.kv_write(0, 0, 0, k, v)
    q = rng.standard_normal(s.heads * hd).astype(F32)
    a = M.attend(0, 0, q, t)
    k2, v2 = k.copy(), v.copy()
    k2[:, t + 1:] = 1e30
    v2[:, t + 1:] = np.nan
    M.kv_write(0, 0, 0, k2, v2)
    b = M.attend(0, 0, q, t)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # and position t itself is read: changing it changes the output
    k2[:, t] += 1
    M.kv_write(0, 0, 0, k2, v2)
    c = M.attend(0, 0, q, t)
    assert not np.array_equal(a, c)


def test_model_causal_bit_identical_after_overwriting_future():
    w = WORKLOADS["tiny_f32"]
    M, blob = _model(w.shape, cap=16, seed=w.seed_weights)
    toks = synth.tokens(w.seed_tokens, 0, 10, w.shape.vocab)
    M.prefill(0, toks[:6], 0, logits=False)
    ref = M.forward(0, toks[6], 6)
    rng = np.random.default_rng(3)
    for layer in range(w.shape.layers):
        junk = rng.standard_normal((w.shape.kv, 16 - 7, w.shape.hd)).astype(F32) * 100
        M.kv_write(layer, 0, 7, junk, junk)
    again = M.forward(0, toks[6], 6)  # rewrites position 6, reads 0..6
    assert np.array_equal(ref.view(np.uint32), again.view(np.uint32))


# ---------------------------------------------------------------------------------------
# attention special cases (P1 head_att = softmax(scale * q.K) . V)
# ---------------------------------------------------------------------------------------

def test_single_position_returns_its_value():
    s = shrink(TINY, kv=2, g=3, half=4)
    M, _ = _model(s, cap=4)
    rng = np.random.default_rng(4)
    k = rng.standard_normal((s.kv, 1, s.hd)).astype(F32)
    v = rng.standard_normal((s.kv, 1, s.hd)).astype(F32)
    M.kv_write(0, 0, 0, k, v)
    q = rng.standard_normal(s.heads * s.hd).astype(F32) * 10
    out = M.attend(0, 0, q, 0).reshape(s.heads, s.hd)
    for h in range(s.heads):
        assert np.array_equal(out[h], v[h // s.g, 0])


def test_equal_scores_average_values():
    s = shrink(TINY, kv=1, g=2, half=4)
    M, _ = _model(s, cap=8)
    rng = np.random.default_rng(5)
    t = 7
    k = np.zeros((1, t + 1, s.hd), F32)
    v = rng.standard_normal((1, t + 1, s.hd)).astype(F32)
    M.kv_write(0, 0, 0, k, v)
    out = M.attend(0, 0, rng.standard_normal(s.heads * s.hd).astype(F32), t)
    np.testing.assert_allclose(out.reshape(s.heads, s.hd)[0], v[0].astype(np.float64).mean(0),
                               rtol=0, atol=1e-6)


def test_scores_scaled_by_inverse_sqrt_head():
    # two positions: keys 0 and e_0, query a * e_0: weights are softmax([0, a / sqrt(hd)])
    s = shrink(TINY, kv=1, g=1, half=8)
    M, _ = _model(s, cap=4)
    hd = s.hd
    k = np.zeros((1, 2, hd), F32)
    k[0, 1, 0] = 1
    v = np.zeros((1, 2, hd), F32)
    v[0, 0, 0] = 1  # output[0] = weight of position 0
    M.kv_write(0, 0, 0, k, v)
    a = 3.0
    q = np.zeros(hd, F32)
    q[0] = a
    out = M.attend(0, 0, q, 1)
    want = 1.0 / (1.0 + math.exp(a / math.sqrt(hd)))
    assert abs(out[0] - want) < 1e-6


# ---------------------------------------------------------------------------------------
# RMSNorm (P1 rmsnorm, squares, pair_sums, tree_sum)
# ---------------------------------------------------------------------------------------

def test_tree_sum_is_pairwise_not_running():
    e = 2.0 ** -24
    # pairs: (1 + e) -> 1 (tie to even), (e + e) = 2e; then 1 + 2e exactly.  A running sum
    # from the left loses every e and gives 1.
    assert oracle.tree_sum([1.0, e, e, e]) == 1.0 + 2 * e
    # odd tail carried to the next round: [a, b, c] -> [a+b, c] -> a+b+c
    assert oracle.tree_sum([1.0, 2.0, 4.0]) == 7.0
    assert oracle.tree_sum([]) == 0.0
    assert oracle.tree_sum([3.5]) == 3.5


def test_tree_sum_exact_on_integers_and_error_bound():
    rng = np.random.default_rng(6)
    ints = rng.integers(-1000, 1000, 777).astype(F32)
    assert oracle.tree_sum(ints) == float(ints.astype(np.int64).sum())
    for n in (5, 64, 576, 4097):
        x = rng.standard_normal(n).astype(F32)
        exact = math.fsum(float(v) for v in x)
        bound = math.ceil(math.log2(n)) * 2.0 ** -24 * float(np.abs(x).astype(np.float64).sum())
        assert abs(oracle.tree_sum(x) - exact) <= bound


def test_rmsnorm_constant_vector_closed_form():
    for n in (64, 576, 4096):
        for c in (0.5, 3.0, 0.001):
            x = np.full(n, c, F32)
            g = np.linspace(0.5, 2.0, n).astype(F32)
            out = oracle.rmsnorm(x, g, 1e-5)
            want = g.astype(np.float64) * (c / math.sqrt(c * c + 1e-5))
            np.testing.assert_allclose(out, want, rtol=4e-7, atol=0)


def test_rmsnorm_scale_invariance_and_gain():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(576).astype(F32)
    g = rng.standard_normal(576).astype(F32)
    a = oracle.rmsnorm(x, g, 0.0)
    b = oracle.rmsnorm(x * F32(4.0), g, 0.0)  # power of two: every step scales exactly
    assert np.array_equal(a, b)
    rms = oracle.rmsnorm(x, np.ones_like(x), 0.0)
    assert abs(float(np.mean(rms.astype(np.float64) ** 2)) - 1.0) < 1e-5


# ---------------------------------------------------------------------------------------
# RoPE (P1 inv_freq, rot_at, rot_lo / rot_hi: q*cos + rotate_half(q)*sin)
# ---------------------------------------------------------------------------------------

def test_rope_identity_at_position_zero():
    for s in (TINY, SMOL135M, LLAMA8B):
        c = oracle.cfg_of(s)
        cs, sn = oracle.rope_cs(c, 0)
        assert np.all(cs == 1.0) and np.all(sn == 0.0)
        x = np.random.default_rng(8).standard_normal(s.hd).astype(F32)
        assert np.array_equal(oracle.rope_head(x, cs, sn), x)


def test_rope_rotation_direction():
    # the pair (lo_i, hi_i) turns by +angle: (1, 0) -> (cos a, sin a); (0, 1) -> (-sin a, cos a)
    s = shrink(TINY, half=4)
    c = oracle.cfg_of(s)
    cs, sn = oracle.rope_cs(c, 1)
    assert cs[0] == F32(math.cos(1.0)) and sn[0] == F32(math.sin(1.0))  # inv[0] = 1
    x = np.zeros(8, F32)
    x[0] = 1
    y = oracle.rope_head(x, cs, sn)
    assert y[0] == cs[0] and y[4] == sn[0]
    x = np.zeros(8, F32)
    x[4] = 1
    y = oracle.rope_head(x, cs, sn)
    assert y[0] == -sn[0] and y[4] == cs[0]


def test_rope_preserves_pair_norms_and_relative_scores():
    s = SMOL135M
    c = oracle.cfg_of(s)
    rng = np.random.default_rng(9)
    q = rng.standard_normal(s.hd).astype(F32)
    k = rng.standard_normal(s.hd).astype(F32)
    h = s.half

    def rot(x, t):
        cs, sn = oracle.rope_cs(c, t)
        return oracle.rope_head(x, cs, sn).astype(np.float64)

    for t in (1, 17, 200):
        y = rot(q, t)
        np.testing.assert_allclose(y[:h] ** 2 + y[h:] ** 2,
                                   q[:h].astype(np.float64) ** 2 + q[h:].astype(np.float64) ** 2,
                                   rtol=1e-5, atol=1e-6)
    # q at t and k at s score like q at t+D and k at s+D
    a = rot(q, 40) @ rot(k, 13)
    b = rot(q, 40 + 50) @ rot(k, 13 + 50)
    assert abs(a - b) < 1e-4


def test_inv_freq_plain():
    for s in (TINY, SMOL135M, SMOL1_7B):
        inv = oracle.inv_freq(oracle.cfg_of(s))
        assert inv[0] == 1.0
        want = 1.0 / np.power(np.float64(s.theta), np.arange(s.half) * 2.0 / s.hd)
        np.testing.assert_allclose(inv, want, rtol=2 ** -23)
        assert np.all(np.diff(inv) < 0)


def test_llama3_bands_on_the_8b_card():
    # P3 README "Validation": the smooth band is frequency indices 29-34 of 64; shorter
    # wavelengths (< 2048) unchanged, longer ones (> 8192) divided by 8
    c8 = oracle.cfg_of(LLAMA8B)
    plain = oracle.inv_freq(oracle.cfg_of(shrink(LLAMA8B, llama3=False)))
    inv = oracle.inv_freq(c8)
    wl = 2 * math.pi / plain.astype(np.float64)
    mid = [i for i in range(64) if not (inv[i] == plain[i] or inv[i] == plain[i] / F32(8))]
    assert mid == list(range(29, 35))
    for i in range(64):
        if wl[i] < 2048 * 0.999:
            assert inv[i] == plain[i]
        elif wl[i] > 8192 * 1.001:
            assert inv[i] == plain[i] / F32(8)
        else:
            assert plain[i] / 8 < inv[i] < plain[i]
    assert np.all(np.diff(inv) < 0)


@pytest.mark.parametrize("edge", ["high", "low"])
def test_llama3_blend_is_continuous_at_band_edges(edge):
    # put a band edge exactly on the wavelength of frequency i: at the high-frequency edge
    # (wavelen == orig/high) the blend must equal the unscaled frequency, at the
    # low-frequency edge (wavelen == orig/low) the frequency divided by factor (P3 rope.linnet:
    # smooth == 1 / smooth == 0; the swapped blend the card reports fails the first)
    base = shrink(LLAMA8B, llama3=False)
    plain = oracle.inv_freq(oracle.cfg_of(base))
    for i in (20, 30, 40):
        wl = F32(F32(2.0) * F32(3.14159265)) / plain[i]
        if edge == "high":
            s = shrink(LLAMA8B, orig_max=float(wl * F32(4)), low_freq=1.0, high_freq=4.0)
            want = plain[i]
        else:
            s = shrink(LLAMA8B, orig_max=float(wl), low_freq=1.0, high_freq=4.0)
            want = plain[i] / F32(8)
        inv = oracle.inv_freq(oracle.cfg_of(s))
        assert inv[i] == want, (i, inv[i], want)


# ---------------------------------------------------------------------------------------
# the model: special cases and invariances (P1 block, forward, head_of; P3 DecoderLayer)
# ---------------------------------------------------------------------------------------

def _zero_layers(shape, blob):
    v = views(shape, blob)
    for i in range(shape.layers):
        for name in ("q", "k", "v", "o", "gate", "up", "down"):
            v[(i, name)][...] = 0
    return v


@pytest.mark.parametrize("tied", [True, False])
def test_zero_layers_give_head_of_normed_embedding(tied):
    # with every layer matrix zero, attention reads zero values and the MLP adds zero, so
    # logits = head . rmsnorm(emb[tok], lnf) (head = emb when tied)
    s = shrink(TINY, tied=tied, vocab=40, layers=2)
    blob = synth.model_blob(s, 11)
    v = _zero_layers(s, blob)
    rng = np.random.default_rng(10)
    v["lnf"][...] = rng.uniform(0.5, 1.5, s.d)
    M, _ = _model(s, cap=8, blob=blob)
    for t, tok in enumerate([3, 17, 39]):
        lg = M.forward(0, tok, t).astype(np.float64)
        x = v["emb"][tok].astype(np.float64)
        nf = v["lnf"] * x / math.sqrt(np.mean(x * x) + s.eps)
        head = v["emb"] if tied else v["lm_head"]
        np.testing.assert_allclose(lg, head.astype(np.float64) @ nf, rtol=0, atol=1e-6)


def test_attention_only_layer_matches_hand_computation_at_t0():
    # at position 0 attention returns V[0] = W_v n1 (one weight of 1), so with a zero MLP
    # one layer is x + W_o W_v rmsnorm(x): q, k and RoPE drop out
    s = shrink(TINY, layers=1, vocab=30)
    blob = synth.model_blob(s, 12)
    v = views(s, blob)
    v[(0, "gate")][...] = 0
    v[(0, "up")][...] = 0
    v[(0, "down")][...] = 0
    M, _ = _model(s, cap=4, blob=blob, trace=True)
    tok = 5
    M.forward(0, tok, 0)
    x = v["emb"][tok].astype(np.float64)
    n1 = x / math.sqrt(np.mean(x * x) + s.eps)
    val = v[(0, "v")].astype(np.float64) @ n1            # [kvw]
    att = np.concatenate([val[(h // s.g) * s.hd:(h // s.g + 1) * s.hd] for h in range(s.heads)])
    y = x + v[(0, "o")].astype(np.float64) @ att
    np.testing.assert_allclose(M.trace(0, "y"), y, rtol=0, atol=2e-6)


def test_mlp_only_layer_matches_hand_computation():
    # with zero attention projections the layer is x + W_down (silu(W_g n2) * (W_u n2))
    s = shrink(TINY, layers=1, vocab=30)
    blob = synth.model_blob(s, 13)
    v = views(s, blob)
    for name in ("q", "k", "v", "o"):
        v[(0, name)][...] = 0
    M, _ = _model(s, cap=4, blob=blob, trace=True)
    M.forward(0, 9, 2)
    x = v["emb"][9].astype(np.float64)
    n2 = x / math.sqrt(np.mean(x * x) + s.eps)
    g = v[(0, "gate")].astype(np.float64) @ n2
    u = v[(0, "up")].astype(np.float64) @ n2
    y = x + v[(0, "down")].astype(np.float64) @ (g / (1 + np.exp(-g)) * u)
    np.testing.assert_allclose(M.trace(0, "y"), y, rtol=0, atol=2e-6)


def test_permuting_mlp_inner_units_changes_nothing():
    # rows of gate and up and columns of down permuted together: same function
    s = shrink(TINY, layers=2)
    blob = synth.model_blob(s, 14)
    toks = [1, 50, 200, 7, 7]
    M, _ = _model(s, cap=8, blob=blob.copy())
    ref = M.prefill(0, toks, 0)
    perm = np.random.default_rng(11).permutation(s.ffn)
    v = views(s, blob)
    for i in range(s.layers):
        v[(i, "gate")][...] = v[(i, "gate")][perm]
        v[(i, "up")][...] = v[(i, "up")][perm]
        v[(i, "down")][...] = v[(i, "down")][:, perm]
    M2, _ = _model(s, cap=8, blob=blob)
    np.testing.assert_allclose(M2.prefill(0, toks, 0), ref, rtol=0, atol=2e-6)


def test_permuting_kv_groups_changes_nothing():
    # key/value head j and its query heads j*g..j*g+g-1 moved together to another slot
    s = shrink(TINY, kv=3, g=2, half=4, layers=2)
    blob = synth.model_blob(s, 15)
    toks = [3, 9, 27, 81, 243 % s.vocab]
    M, _ = _model(s, cap=8, blob=blob.copy())
    ref = M.prefill(0, toks, 0)
    pj = np.array([2, 0, 1])
    hd = s.hd
    qrows = np.concatenate([np.arange(hd) + (pj[h // s.g] * s.g + h % s.g) * hd
                            for h in range(s.heads)])
    kvrows = np.concatenate([np.arange(hd) + pj[j] * hd for j in range(s.kv)])
    v = views(s, blob)
    for i in range(s.layers):
        v[(i, "q")][...] = v[(i, "q")][qrows]
        v[(i, "k")][...] = v[(i, "k")][kvrows]
        v[(i, "v")][...] = v[(i, "v")][kvrows]
        v[(i, "o")][...] = v[(i, "o")][:, qrows]
    M2, _ = _model(s, cap=8, blob=blob)
    np.testing.assert_allclose(M2.prefill(0, toks, 0), ref, rtol=0, atol=2e-6)


def test_query_head_uses_its_own_group_not_neighbours():
    # zeroing the values of key/value head 1 changes exactly query heads g..2g-1
    s = shrink(TINY, kv=3, g=2, half=4)
    M, _ = _model(s, cap=4)
    rng = np.random.default_rng(12)
    k = rng.standard_normal((s.kv, 3, s.hd)).astype(F32)
    v = rng.standard_normal((s.kv, 3, s.hd)).astype(F32)
    q = rng.standard_normal(s.heads * s.hd).astype(F32)
    M.kv_write(0, 0, 0, k, v)
    a = M.attend(0, 0, q, 2).reshape(s.heads, s.hd)
    v[1] = 0
    M.kv_write(0, 0, 0, k, v)
    b = M.attend(0, 0, q, 2).reshape(s.heads, s.hd)
    for h in range(s.heads):
        assert np.array_equal(a[h], b[h]) == (h // s.g != 1)


def _c1_variants():
    yield "tiny_f32", TINY, WORKLOADS["tiny_f32"].seed_weights
    yield "g1", shrink(TINY, kv=4, g=1), 21
    yield "g4_odd_ffn", shrink(TINY, kv=1, g=4, ffn=90), 22
    yield "untied_llama3", shrink(TINY, tied=False, llama3=True, orig_max=64.0), 23


@pytest.mark.parametrize("name,shape,seed", list(_c1_variants()), ids=lambda x: str(x)[:12])
def test_decode_token_by_token_equals_full_sequence(name, shape, seed):
    # P3 attention.linnet: forward (causal mask over a whole sequence) and decode (one
    # position at a time through the cache) compute the same logits
    S = 10
    blob = synth.model_blob(shape, seed, wstd=0.1)
    toks = synth.tokens(seed + 1, 0, S, shape.vocab)
    full = oracle.forward_full(oracle.cfg_of(shape, 1, S), blob, toks)
    M, _ = _model(shape, cap=S, blob=blob)
    for t in range(S):
        lg = M.forward(0, toks[t], t)
        rng_ = float(full[t].max() - full[t].min())
        assert np.max(np.abs(lg - full[t])) <= 1e-6 * rng_, (t, np.max(np.abs(lg - full[t])))


def test_prefill_equals_forward_pre_then_forward():
    w = WORKLOADS["tiny_f32"]
    blob = synth.model_blob(w.shape, w.seed_weights)
    toks = synth.tokens(w.seed_tokens, 0, 8, w.shape.vocab)
    A, _ = _model(w.shape, cap=16, blob=blob)
    B, _ = _model(w.shape, cap=16, blob=blob)
    a = A.prefill(0, toks, 0)
    for t in range(7):
        B.forward(0, toks[t], t, logits=False)
    b = B.forward(0, toks[7], 7)
    assert np.array_equal(a, b)


def test_rows_of_a_batch_are_independent():
    w = WORKLOADS["tiny_f32"]
    blob = synth.model_blob(w.shape, w.seed_weights)
    M, _ = _model(w.shape, cap=8, batch=3, blob=blob)
    S, _ = _model(w.shape, cap=8, batch=1, blob=blob)
    t1 = [5, 6, 7, 8]
    t2 = [100, 3, 3, 9]
    M.prefill(0, t1, 0, logits=False)
    a = M.prefill(2, t2, 0)
    b = S.prefill(0, t2, 0)
    assert np.array_equal(a, b)


def test_position_and_token_range_errors():
    w = WORKLOADS["tiny_f32"]
    M, _ = _model(w.shape, cap=4, seed=w.seed_weights)
    with pytest.raises(ValueError):
        M.forward(0, 3, 4)  # t >= cap (P1 KV.push needs t < cap)
    with pytest.raises(ValueError):
        M.forward(0, w.shape.vocab, 0)
    with pytest.raises(ValueError):
        M.forward(1, 3, 0)


# ---------------------------------------------------------------------------------------
# greedy and sampling (P1 argmax, "Sampling": topk, kept, pick, sample; law sample_below)
# ---------------------------------------------------------------------------------------

def test_argmax_first_of_ties():
    assert oracle.argmax([1, 3, 3, 2]) == 1
    assert oracle.argmax([-1, -1]) == 0
    assert oracle.argmax([0, 0, 5]) == 2


def test_exp_s_accuracy_and_exact_points():
    assert oracle.exp_s(0.0) == 1.0
    assert oracle.exp_s(-200.0) == 0.0
    xs = np.concatenate([np.linspace(-104, 0, 200001), -np.logspace(-8, 2, 2000)]).astype(F32)
    worst = 0.0
    for x in xs[::7]:
        e = math.exp(float(x))
        got = oracle.exp_s(float(x))
        if e < 1.2e-38:  # subnormal range: absolute error within one subnormal step
            assert abs(got - e) <= 2 ** -149
            continue
        worst = max(worst, abs(got - e) / ulp(e))
    assert worst <= 2.0, worst


def _p1_sampler(xs, temp, k, p, u):
    """The sampler of P1 "Sampling", restated step by step for tiny inputs: one-pass
    insertion top-k (a value enters if there is room or it is above the smallest kept;
    it goes before the first candidate that is strictly smaller), weights by exp_s, the
    kept count and the draw."""
    xs = [F32(x) for x in xs]
    temp, p, u = F32(temp), F32(p), F32(u)
    cs = []
    for i, h in enumerate(xs):
        room = len(cs) < k
        lo = cs[-1][0] if cs else F32(0)
        if not (room or h > lo):
            continue
        pos = next((j for j, (cv, _) in enumerate(cs) if cv < h), len(cs))
        cs = (cs[:pos] + [(h, i)] + cs[pos:])[:k]
    top = cs[0][0]

    def wt(v):
        return F32(oracle.exp_s(float(F32(F32(v / temp) - F32(top / temp)))))

    Z = F32(0)
    for v, _ in cs:
        Z = F32(Z + wt(v))
    lim = F32(p * Z)
    acc, n = F32(0), 0
    for v, _ in cs:
        acc = F32(acc + wt(v))
        n += 1
        if not acc < lim:
            break
    target = F32(u * acc)
    a = F32(0)
    for j in range(n):
        a2 = F32(a + wt(cs[j][0]))
        if j == n - 1 or target < a2:
            return cs[j][1], [i for _, i in cs], n
        a = a2


def test_sampler_matches_page_algorithm_on_tiny_inputs():
    rng = np.random.default_rng(13)
    for trial in range(3000):
        V = int(rng.integers(1, 9))
        if trial % 3 == 0:
            xs = rng.integers(-2, 3, V).astype(F32)  # many ties
        else:
            xs = (rng.standard_normal(V) * 3).astype(F32)
        temp = float(rng.choice([0.3, 0.8, 1.0, 2.5]))
        k = int(rng.integers(1, V + 3))
        p = float(rng.choice([1e-6, 0.3, 0.9, 1.0]))
        u = float(F32(rng.random()))
        want = _p1_sampler(xs, temp, k, p, u)
        got = oracle.sample_detail(xs, temp, k, p, u)
        assert got[0] == want[0] and list(got[1]) == want[1] and got[2] == want[2], (
            xs, temp, k, p, u, got, want)


def test_sample_below_and_membership():
    rng = np.random.default_rng(14)
    for _ in range(20000):
        V = int(rng.integers(1, 70))
        xs = (rng.standard_normal(V) * rng.choice([0.1, 1, 10])).astype(F32)
        temp = float(rng.uniform(0.05, 3))
        k = int(rng.integers(1, V + 5))
        p = float(rng.uniform(1e-4, 1))
        u = float(F32(rng.random()))
        i, cand, n = oracle.sample_detail(xs, temp, k, p, u)
        assert 0 <= i < V
        assert len(cand) == min(k, V)
        assert 1 <= n <= len(cand)
        assert i in cand[:n]
        # the candidates are the k largest (ties by lower id)
        order = sorted(range(V), key=lambda j: (-float(xs[j]), j))[:min(k, V)]
        assert list(cand) == order


def test_sampler_special_cases():
    rng = np.random.default_rng(15)
    for _ in range(500):
        V = int(rng.integers(2, 300))
        xs = rng.standard_normal(V).astype(F32)
        a = oracle.argmax(xs)
        u = float(F32(rng.random()))
        assert oracle.sample(xs, 0.7, 1, 0.9, u) == a              # k = 1: the top logit
        assert oracle.sample(xs, 0.7, V, 1e-9, u) == a             # p -> 0: the first kept only
        assert oracle.sample(xs, 0.7, V, 0.9, 0.0) == a            # u = 0: the first candidate


def test_sampler_draws_in_proportion_to_weights():
    # with k = V and p = 1 the draw is the inverse of the cumulative weights: over a grid of
    # u each id is drawn a share equal to its weight / Z
    xs = np.array([0.0, -0.5, 1.0, 0.25, -2.0], F32)
    temp = 0.9
    N = 20000
    counts = np.zeros(xs.size)
    for i in range(N):
        counts[oracle.sample(xs, temp, xs.size, 1.0, (i + 0.5) / N)] += 1
    w = np.exp(xs.astype(np.float64) / temp)
    np.testing.assert_allclose(counts / N, w / w.sum(), atol=2.0 / N)


def test_draw_is_strict_at_an_exact_boundary():
    # two equal logits weigh 1 each (Z = Zp = 2); u = 1/2 puts the target on the first
    # cumulative weight exactly, and "above the target" is strict, so the second is drawn
    xs = [0.25, 0.25]
    assert oracle.sample(xs, 1.0, 2, 1.0, 0.5) == 1
    assert oracle.sample(xs, 1.0, 2, 1.0, float(np.nextafter(F32(0.5), F32(0)))) == 0
    # top-p: the second candidate is kept only while the weight before it (1) is below p*Z
    assert oracle.sample_detail(xs, 1.0, 2, 0.5, 0.9)[2] == 1   # p*Z = 1: not below
    assert oracle.sample_detail(xs, 1.0, 2, 0.51, 0.9)[2] == 2


def test_rotation_is_identity_at_position_zero_in_the_model():
    # P1 rot_at(0): every angle is 0, so the rotated heads equal the projected ones, and the
    # rotation at t=1 turns by exactly inv[i] radians (absolute positions, not shifted)
    s = shrink(TINY, layers=1)
    M, _ = _model(s, cap=4, trace=True)
    M.forward(0, 3, 0)
    assert np.array_equal(M.trace(0, "qr"), M.trace(0, "q"))
    assert np.array_equal(M.trace(0, "kr"), M.trace(0, "k"))
    M.forward(0, 3, 1)
    k, kr = M.trace(0, "k"), M.trace(0, "kr")
    h = s.half
    a = np.arctan2(kr[h:2 * h].astype(np.float64), kr[:h]) - np.arctan2(k[h:2 * h].astype(np.float64), k[:h])
    a = (a + np.pi) % (2 * np.pi) - np.pi
    want = 1.0 / np.power(np.float64(s.theta), np.arange(h) * 2.0 / s.hd)
    np.testing.assert_allclose(a, want, atol=1e-5)


# ---------------------------------------------------------------------------------------
# packed prefill (Llama 3.1 8B Instruct card, "Entries": prefill_packed; lib.linnet)
# ---------------------------------------------------------------------------------------

PACK_SHAPES = [shrink(TINY, kv=2, g=2, layers=2), shrink(SMOL135M, layers=1, ffn=64, vocab=96)]


@pytest.mark.parametrize("shape", PACK_SHAPES, ids=["f32", "bf16"])
def test_packed_single_prompt_is_prefill(shape):
    # one prompt at positions 0..S-1: token t attends to positions 0..t of its row, exactly as
    # S decode steps do, in the same order -- bit for bit, logits and cache
    S = 7
    toks = synth.tokens(901, 0, S, shape.vocab)
    a, blob = _model(shape, cap=16, batch=2, seed=902)
    b, _ = _model(shape, cap=16, batch=2, blob=blob)
    la = a.prefill_packed(toks, np.ones(S), np.arange(S), np.zeros(S), [S - 1])[0]
    lb = b.prefill(1, toks, 0)
    assert np.array_equal(la.view(np.uint32), lb.view(np.uint32))
    for layer in range(shape.layers):
        ka, va = a.kv_read(layer, 1, 0, S)
        kb, vb = b.kv_read(layer, 1, 0, S)
        assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    a.close()
    b.close()


@pytest.mark.parametrize("shape", PACK_SHAPES, ids=["f32", "bf16"])
def test_packed_prompts_do_not_see_each_other(shape):
    # two prompts packed end to end, then interleaved: each gives what it gives alone
    t0 = synth.tokens(903, 0, 5, shape.vocab)
    t1 = synth.tokens(904, 0, 3, shape.vocab)
    alone = []
    for r, t in ((0, t0), (1, t1)):
        m, blob = _model(shape, cap=8, batch=2, seed=905)
        alone.append(m.prefill(r, t, 0))
        m.close()
    toks = np.concatenate([t0, t1])
    rows = np.array([0] * 5 + [1] * 3)
    pos = np.array(list(range(5)) + list(range(3)))
    seg = np.array([0] * 5 + [1] * 3)
    m, blob = _model(shape, cap=8, batch=2, seed=905)
    end_to_end = m.prefill_packed(toks, rows, pos, seg, [4, 7])
    m.close()
    order = [0, 5, 1, 6, 2, 7, 3, 4]  # alternate the prompts' tokens, each prompt still in order
    m, blob = _model(shape, cap=8, batch=2, seed=905)
    inter = m.prefill_packed(toks[order], rows[order], pos[order], seg[order], [order.index(4), order.index(7)])
    m.close()
    for k in range(2):
        assert np.array_equal(end_to_end[k].view(np.uint32), alone[k].view(np.uint32))
        assert np.array_equal(inter[k].view(np.uint32), alone[k].view(np.uint32))


def test_packed_prompt_sees_only_itself_not_its_rows_older_cache():
    # a prompt at positions 5..9 of a row whose cache already holds positions 0..4: the pass
    # ignores them (a decode-style prefill at position 5 would not), and attention being
    # relative, the result is the same prompt's at positions 0..4 up to RoPE rounding
    shape = PACK_SHAPES[0]
    toks = synth.tokens(906, 0, 5, shape.vocab)
    seg = np.zeros(5)
    m, blob = _model(shape, cap=16, batch=1, seed=907)
    m.prefill(0, synth.tokens(908, 0, 5, shape.vocab), 0, logits=False)
    a = m.prefill_packed(toks, np.zeros(5), np.arange(5, 10), seg, [4])[0]
    m.prefill(0, synth.tokens(909, 0, 5, shape.vocab), 0, logits=False)  # other older content
    b = m.prefill_packed(toks, np.zeros(5), np.arange(5, 10), seg, [4])[0]
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    m.prefill(0, synth.tokens(908, 0, 5, shape.vocab), 0, logits=False)
    c = m.prefill(0, toks, 5)  # decode-style: reads positions 0..4 as well
    assert not np.array_equal(a.view(np.uint32), c.view(np.uint32))
    m.close()
    z, _ = _model(shape, cap=16, batch=1, blob=blob)
    at0 = z.prefill_packed(toks, np.zeros(5), np.arange(5), seg, [4])[0]
    z.close()
    assert float(np.max(np.abs(a - at0))) <= 1e-4 * float(at0.max() - at0.min())


def test_packed_rejects_shared_slots_and_bad_indices():
    shape = PACK_SHAPES[0]
    m, _ = _model(shape, cap=8, batch=2, seed=910)
    toks = np.array([1, 2, 3])
    with pytest.raises(ValueError):  # two tokens in one (row, position) slot
        m.prefill_packed(toks, [0, 0, 1], [0, 0, 0], [0, 1, 2], [0])
    with pytest.raises(ValueError):  # last names no token
        m.prefill_packed(toks, [0, 0, 0], [0, 1, 2], [0, 0, 0], [3])
    with pytest.raises(ValueError):  # row outside the cache
        m.prefill_packed(toks, [0, 0, 2], [0, 1, 2], [0, 0, 0], [2])
    with pytest.raises(ValueError):  # position outside the cache
        m.prefill_packed(toks, [0, 0, 0], [0, 1, 8], [0, 0, 0], [2])
    m.close()


# ---- bf16 cache rounding (Llama 3.1 8B Instruct card, attention.linnet decode: a cache of
# element type T = bf16; the f32 value of a key or value is rounded to the nearest bf16, ties to
# the even significand, as IEEE 754 round-to-nearest-even fixes) ----

def _bits(x: float) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0])


def _f32(bits: int) -> float:
    return float(np.array([bits], np.uint32).view(np.float32)[0])


def _rne_bf16_exact(bits: int) -> int:
    """Nearest bf16 to the f32 value with these bits, by exact comparison of the two
    neighbouring bf16 values (distances in exact rationals); ties go to the even one."""
    from fractions import Fraction
    x = _f32(bits)
    if math.isnan(x):
        return None
    if math.isinf(x):
        return bits >> 16
    lo = bits >> 16                       # truncation: the neighbour toward zero
    hi = lo + 1                           # the neighbour away from zero (may be an infinity)
    xv = Fraction(x)
    lv = Fraction(_f32(lo << 16))
    hx = _f32(hi << 16)
    if math.isinf(hx):
        # above the largest finite bf16 the next value up is 2^128 for rounding purposes
        hv = Fraction(2) ** 128 * (1 if x > 0 else -1)
    else:
        hv = Fraction(hx)
    dl, dh = abs(xv - lv), abs(xv - hv)
    if dl < dh:
        return lo
    if dh < dl:
        return hi
    return lo if (lo & 1) == 0 else hi


@pytest.mark.parametrize("bits, want", [
    (0x3F808000, 0x3F80),  # 1 + 2^-8: tie, the even neighbour is 1
    (0x3F818000, 0x3F82),  # 1 + 3*2^-8: tie, the even neighbour is 1 + 2^-6
    (0x3F808001, 0x3F81),  # just above a tie
    (0x3F807FFF, 0x3F80),  # just below a tie
    (0x3F817FFF, 0x3F81),
    (0xBF808000, 0xBF80),  # negative ties
    (0xBF818000, 0xBF82),
    (0xBF808001, 0xBF81),
    (0x7F7FFFFF, 0x7F80),  # the largest finite f32 rounds to +infinity
    (0x7F7F8000, 0x7F80),  # tie between the largest finite bf16 and infinity: even is infinity
    (0x7F7F7FFF, 0x7F7F),
    (0xFF7FFFFF, 0xFF80),
    (0x7F800000, 0x7F80),  # infinities stay
    (0xFF800000, 0xFF80),
    (0x00000000, 0x0000),  # signed zeros stay
    (0x80000000, 0x8000),
    (0x00000001, 0x0000),  # subnormals round like any other value
    (0x00008000, 0x0000),
    (0x00018000, 0x0002),
    (0x00008001, 0x0001),
    (0x807F8000, 0x8080),  # largest negative subnormal tie rounds up to the smallest normal
])
def test_bf16_cache_rounding_fixed_cases(bits, want):
    assert oracle.f32_to_bf16(_f32(bits)) == want


@pytest.mark.parametrize("bits", [0x7FC00000, 0xFFC00000, 0x7F800001, 0x7F810000, 0xFFFFFFFF])
def test_bf16_cache_rounding_keeps_nan(bits):
    got = oracle.f32_to_bf16(_f32(bits))
    assert (got & 0x7F80) == 0x7F80 and (got & 0x7F) != 0, hex(got)
    assert (got >> 15) == (bits >> 31)


def test_bf16_cache_rounding_matches_exact_nearest_even():
    rng = np.random.default_rng(21)
    # random bit patterns, plus values a few ulps around every tie of a range of exponents
    pats = [int(b) for b in rng.integers(0, 2 ** 32, 20000, dtype=np.uint64)]
    for e in range(0, 255, 7):
        for m in rng.integers(0, 2 ** 7, 8):
            tie = (e << 23) | (int(m) << 16) | 0x8000
            pats += [tie + dd for dd in (-2, -1, 0, 1, 2)] + [(tie | 0x80000000) + dd for dd in (-1, 0, 1)]
    n = 0
    for b in pats:
        want = _rne_bf16_exact(b & 0xFFFFFFFF)
        if want is None:
            continue
        assert oracle.f32_to_bf16(_f32(b & 0xFFFFFFFF)) == want, hex(b)
        n += 1
    assert n > 20000


def test_cache_holds_the_rounded_rotated_keys():
    # the bf16 cache of a forward step holds exactly the rounding of the rotated keys and of the
    # values the layer computed (kr and v of the trace)
    s = shrink(SMOL135M, layers=1, vocab=64, ffn=64)
    blob = synth.model_blob(s, 31)
    M = oracle.Model(oracle.cfg_of(s, 1, 8), blob, trace=True)
    M.forward(0, 11, 3)
    k, v = M.kv_read(0, 0, 3, 1)
    kr, vv = M.trace(0, "kr"), M.trace(0, "v")
    want_k = np.array([oracle.f32_to_bf16(float(x)) for x in kr], np.uint16).reshape(s.kv, 1, s.hd)
    want_v = np.array([oracle.f32_to_bf16(float(x)) for x in vv], np.uint16).reshape(s.kv, 1, s.hd)
    np.testing.assert_array_equal(k, want_k)
    np.testing.assert_array_equal(v, want_v)
    M.close()
