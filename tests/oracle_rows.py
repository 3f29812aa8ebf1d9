"""Oracle runs of independent cache rows in worker processes (test infrastructure).

Each task rebuilds the seeded weight blob and runs one row through the oracle: a prompt through
or_prefill (logits after its last token, and the row's cache), then decode steps from given
tokens.  Rows are independent, so the workers of a spawn pool run them side by side; the pool is
created with the spawn method, so no worker inherits a CUDA context.
"""
import multiprocessing as mp

import numpy as np

import oracle
import synth


def run_row(task):
    """task: dict(shape, seed, wstd, cap, prompt, pos0, steps=[tokens], kv=[layers]).
    Returns dict(prefill=logits, steps=[logits], kv={layer: (k, v)} of positions 0..end)."""
    s = task["shape"]
    blob = synth.model_blob(s, task["seed"], wstd=task.get("wstd", 0.02))
    ref = oracle.Model(oracle.cfg_of(s, 1, task["cap"]), blob)
    out = {"steps": [], "kv": {}}
    pos = task.get("pos0", 0)
    for chunk in task["prompts"]:
        lo = ref.prefill(0, np.asarray(chunk, np.int32), pos)
        pos += len(chunk)
        out.setdefault("prefill", []).append(lo)
    for tok in task.get("steps", []):
        out["steps"].append(ref.forward(0, int(tok), pos))
        pos += 1
    for layer in task.get("kv", []):
        out["kv"][layer] = ref.kv_read(layer, 0, 0, pos)
    ref.close()
    return out


def run_rows(tasks, workers=None):
    ctx = mp.get_context("spawn")
    with ctx.Pool(processes=workers or min(len(tasks), 8)) as pool:
        return pool.map(run_row, tasks)
