"""Write the stored oracle results that the full-size parity tests compare against.

Only the oracle (oracle/) and the seeded input generators (synth/) run here.  An 8B-shaped
oracle position takes seconds on one core, so a 2048-token prompt is hours of CPU work: these
files are written once, offline, and committed; the GPU tests then replay the same seeded
inputs and compare.

Each job runs one cache row of one workload, as the benchmark builds it:
  * the row's prompt (synthetic tokens; prompt b of a batch is tokens[b*P:(b+1)*P]) through the
    oracle's prefill, then decode steps from the row's first decode token (tokens[B*P + b]);
    each later step feeds the oracle's own choice (greedy argmax, or the sampler with the draw
    u = uniform(seed_u, s*B + b));
  * the long-context presets instead fill the cache with synthetic keys and values (positions
    0..fill-1) and decode from there.
For every step the file keeps the fed token and position, the oracle's argmax and (sampled
workloads) its draw, the 16 largest logits with their ids, and the logits at 256 fixed indices.

usage: python tests/golden/make_fullsize.py JOB [JOB ...]     (jobs: see JOBS)
"""
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402
from synth import WORKLOADS  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
N_IDX = 256
N_TOP = 16

# job -> (workload, row, decode steps, extra: a second decode run from the prompt's end with the
# first tokens of another batch size of the same seeds)
JOBS = {
    "llama8b_row0": ("llama8b_b1", 0, 16, ("llama8b_b32", 4)),
    "llama8b_row31": ("llama8b_b32", 31, 4, None),
    "smollm2_1_7b_row0": ("smollm2_1_7b_b16", 0, 16, None),
    "smollm2_1_7b_row7": ("smollm2_1_7b_b16", 7, 16, None),
    "smollm2_1_7b_row15": ("smollm2_1_7b_b16", 15, 16, None),
    "llama8b_long_b1_row0": ("llama8b_long_b1", 0, 4, None),
    "llama8b_long_b8_row0": ("llama8b_long_b8", 0, 2, None),
    "llama8b_long_b8_row7": ("llama8b_long_b8", 7, 2, None),
}


def sample_indices(vocab):
    return np.sort(np.random.default_rng(12345).choice(vocab, N_IDX, replace=False)).astype(np.int64)


def digest(lo, idx):
    top = np.argsort(-lo, kind="stable")[:N_TOP]
    return {"argmax": oracle.argmax(lo), "top_ids": [int(i) for i in top],
            "top_vals": [float(lo[i]) for i in top], "vals": [float(v) for v in lo[idx]]}


def decode(ref, w, row, t0, tok, steps, idx, log):
    out = []
    s = w.shape
    k = w.top_k or s.vocab
    for i in range(steps):
        t = t0 + i
        lo = ref.forward(0, int(tok), t)
        rec = {"t": t, "tok": int(tok), **digest(lo, idx)}
        if w.temp > 0:
            u = float(synth.uniforms(w.seed_uniform, i * w.batch + row, 1)[0])
            rec["u"] = u
            rec["id"] = oracle.sample(lo, w.temp, k, w.top_p, u)
            tok = rec["id"]
        else:
            tok = rec["argmax"]
        out.append(rec)
        log(f"step {i} t={t} -> {tok}")
    return out


def run(job):
    name, row, steps, extra = JOBS[job]
    w = WORKLOADS[name]
    s = w.shape
    t_start = time.time()

    def log(msg):
        print(f"[{job} {time.time() - t_start:8.1f}s] {msg}", flush=True)

    blob = synth.model_blob(s, w.seed_weights)
    log("weights ready")
    P = w.prompt
    cap = max(P, w.fill) + steps + 1
    ref = oracle.Model(oracle.cfg_of(s, 1, cap), blob)
    idx = sample_indices(s.vocab)
    res = {"job": job, "workload": name, "row": row, "batch": w.batch, "prompt": P, "fill": w.fill,
           "idx": [int(i) for i in idx]}
    if P > 0:
        prompt = synth.tokens(w.seed_tokens, row * P, P, s.vocab)
        t0 = time.time()
        lo = ref.prefill(0, prompt, 0)
        log(f"prefill of {P} positions: {time.time() - t0:.1f} s")
        res["prefill"] = digest(lo, idx)
        res["prefill_seconds"] = time.time() - t0
    else:
        for layer in range(s.layers):
            k, v = synth.kv_values(w.seed_kv, layer, row, w.batch, s.kv, w.fill, s.hd, bf16=s.bf16)
            ref.kv_write(layer, 0, 0, k, v)
        log(f"cache filled to {w.fill}")
    t0 = max(P, w.fill)
    first = int(synth.tokens(w.seed_tokens, w.batch * P, w.batch, s.vocab)[row])
    t1 = time.time()
    res["steps"] = decode(ref, w, row, t0, first, steps, idx, log)
    res["decode_seconds_per_step"] = (time.time() - t1) / steps
    if extra:
        w2 = WORKLOADS[extra[0]]
        first2 = int(synth.tokens(w2.seed_tokens, w2.batch * P, w2.batch, s.vocab)[row])
        res["steps_" + extra[0]] = decode(ref, w2, row, t0, first2, extra[1], idx, log)
    ref.close()
    path = os.path.join(HERE, f"fullsize_{job}.json")
    with open(path + ".tmp", "w") as f:
        json.dump(res, f)
    os.replace(path + ".tmp", path)
    log(f"wrote {path}")


if __name__ == "__main__":
    for j in sys.argv[1:]:
        run(j)
