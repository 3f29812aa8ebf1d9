"""The stored full-size oracle results (tests/golden/fullsize_*.json) against the current input
generators and against themselves: the files were written offline from seeded inputs, so a change
to the generators (or a damaged file) would otherwise surface only as a GPU test failure.

Checked without running the oracle: the fixed logit indices, every step's fed token (the row's
first decode token from the token generator, then the previous step's argmax or draw), the draws
u from the uniform generator, positions counting up from the prompt's end (or the filled cache),
and each digest's own consistency (the 16 largest sorted by value, then id; the argmax first).
"""
import glob
import importlib.util
import json
import os

import numpy as np
import pytest

import synth
from synth import WORKLOADS

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
FILES = sorted(glob.glob(os.path.join(GOLDEN, "fullsize_*.json")))


def _writer():
    spec = importlib.util.spec_from_file_location("make_fullsize", os.path.join(GOLDEN, "make_fullsize.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _check_digest(rec, idx, vocab):
    top_ids, top_vals = rec["top_ids"], rec["top_vals"]
    assert len(top_ids) == 16 and len(top_vals) == 16 and len(rec["vals"]) == len(idx)
    assert all(0 <= i < vocab for i in top_ids) and len(set(top_ids)) == 16
    # sorted by value descending, equal values by id ascending (a stable sort of -logits)
    for a in range(15):
        assert (top_vals[a] > top_vals[a + 1]) or (top_vals[a] == top_vals[a + 1] and top_ids[a] < top_ids[a + 1])
    assert rec["argmax"] == top_ids[0]
    # a stored index that is also among the largest carries the same value
    pos = {int(i): k for k, i in enumerate(idx)}
    for i, v in zip(top_ids, top_vals):
        if i in pos:
            assert rec["vals"][pos[i]] == v
    assert all(np.isfinite(rec["vals"])) and all(np.isfinite(top_vals))


def _check_steps(steps, w, row, t0, first):
    s = w.shape
    tok = first
    for i, rec in enumerate(steps):
        assert rec["t"] == t0 + i
        assert rec["tok"] == tok
        if w.temp > 0:
            u = float(synth.uniforms(w.seed_uniform, i * w.batch + row, 1)[0])
            assert rec["u"] == u
            assert 0 <= rec["id"] < s.vocab
            tok = rec["id"]
        else:
            assert "id" not in rec
            tok = rec["argmax"]


def test_every_job_has_its_file():
    jobs = _writer().JOBS
    names = {os.path.basename(p)[len("fullsize_"):-len(".json")] for p in FILES}
    assert names == set(jobs), (names, set(jobs))


@pytest.mark.parametrize("path", FILES, ids=lambda p: os.path.basename(p))
def test_stored_results_follow_the_generators(path):
    mk = _writer()
    with open(path) as f:
        d = json.load(f)
    name, row, nsteps, extra = mk.JOBS[d["job"]]
    w = WORKLOADS[name]
    s = w.shape
    assert (d["workload"], d["row"], d["batch"], d["prompt"], d["fill"]) == (name, row, w.batch, w.prompt, w.fill)
    idx = d["idx"]
    assert idx == [int(i) for i in mk.sample_indices(s.vocab)]
    P = w.prompt
    if P > 0:
        _check_digest(d["prefill"], idx, s.vocab)
        assert d["prefill_seconds"] > 0
    else:
        assert "prefill" not in d
    t0 = max(P, w.fill)
    first = int(synth.tokens(w.seed_tokens, w.batch * P, w.batch, s.vocab)[row])
    assert len(d["steps"]) == nsteps
    for rec in d["steps"]:
        _check_digest(rec, idx, s.vocab)
    _check_steps(d["steps"], w, row, t0, first)
    if extra:
        w2 = WORKLOADS[extra[0]]
        steps2 = d["steps_" + extra[0]]
        assert len(steps2) == extra[1]
        for rec in steps2:
            _check_digest(rec, idx, s.vocab)
        first2 = int(synth.tokens(w2.seed_tokens, w2.batch * P, w2.batch, s.vocab)[row])
        _check_steps(steps2, w2, row, t0, first2)
