#!/usr/bin/env python
"""Decode throughput of the KV-cached Llama decoder step on GB300.

A step is one pass of the whole hot path for a batch: embedding, every layer (norm, Q/K/V,
RoPE, KV write, attention, o_proj, norm, SwiGLU MLP), final norm, LM head and the sampler,
run as `llm_step_dev` on device-resident inputs.  The default workload is the Llama-3.1-8B
shape (hidden 4096, 32 layers, 32/8 heads of 128, MLP 14336, vocabulary 128256, untied head,
llama3 RoPE) at batch 1 with a 2048-position cache prefilled from synthetic tokens, greedy.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle (the plain f32
decoder under oracle/) on the same workload instead, on a bounded sample per step.
"""
import argparse
import dataclasses
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402
from synth import WORKLOADS  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
GATEUP = 3  # kernel id of the norm + gate/up + SwiGLU GEMV (llm_profile_kernel)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama8b_b1", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-steps", type=int, default=2, help="oracle decode steps for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-layers", type=int, default=2,
                    help="reference arm: layers of the model run per timed step")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling)")
    ap.add_argument("--prompt", type=int, default=-1, help="override the prompt length (profiling)")
    ap.add_argument("--generate", action="store_true",
                    help="time llm_generate_dev: the K steps as CUDA graphs of 8 chained steps")
    ap.add_argument("--rows", action="store_true",
                    help="rows at their own positions (decode_rows): row b at P - b * (P // 2B)")
    ap.add_argument("--kernels", action="store_true",
                    help="print each kernel's isolated launch time (CUDA events) and exit")
    ap.add_argument("--max-tokens", type=int, default=0,
                    help="prompt tokens per prefill pass (0: the library default)")
    ap.add_argument("--b32-steps", type=int, default=64,
                    help="default workload: also time this many batch-32 steps (0: skip)")
    ap.add_argument("--step-kernel", type=int, default=0, choices=[0, 1],
                    help="batch 1: 1 runs each step as one persistent kernel")
    ap.add_argument("--tc-min-batch", type=int, default=0,
                    help="rows from which a step runs its projections on the tensor cores (0: library default)")
    return ap.parse_args()


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, under_load_from=0):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines[under_load_from:]:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_function_text(src, name):
    """The definition of function `name` in source text src: from its name through the closing
    brace of its body (None if src does not define it)."""
    for m in re.finditer(r"\b%s\s*\(" % re.escape(name), src):
        i, depth = m.end(), 1
        while depth and i < len(src):
            depth += {"(": 1, ")": -1}.get(src[i], 0)
            i += 1
        while i < len(src) and src[i] in " \t\n":
            i += 1
        if i < len(src) and src[i] == "{":
            depth = 0
            for k in range(i, len(src)):
                depth += {"{": 1, "}": -1}.get(src[k], 0)
                if depth == 0:
                    return src[m.start():k + 1]
    return None


def traffic_from_profile(kernel_file, profile_name):
    """dram bytes per launch from the committed ncu summary, if taken on the current source: the
    profiled kernel's own definition (kernel_function / kernel_function_sha256_16) when the
    summary names it, else the whole file (kernel_source_sha256_16)."""
    path = os.path.join(ROOT, "profiles", profile_name)
    src = os.path.join(ROOT, "llama_architecture_kv_gb300", "csrc", kernel_file)
    try:
        text = open(path).read()
        code = open(src, "rb").read()
        m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
        m_fn = re.search(r"kernel_function:\s*(\w+)", text)
        m_fsha = re.search(r"kernel_function_sha256_16:\s*([0-9a-f]+)", text)
        if m_fn and m_fsha:
            body = kernel_function_text(code.decode(), m_fn.group(1))
            ok = body is not None and hashlib.sha256(body.encode()).hexdigest()[:16] == m_fsha.group(1)
        else:
            m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
            ok = m_sha is not None and m_sha.group(1) == hashlib.sha256(code).hexdigest()[:16]
        if ok and m_tr:
            return float(m_tr.group(1))
    except OSError:
        pass
    return None


NOMINAL_HBM_GBS = 8000.0  # nominal HBM3e bandwidth of the part, reported beside the measured copy rate


def step_roofline(step_bytes, B, peak_gbs, per_gpu_tok_s, K, elapsed):
    """The whole step against HBM: B tokens per step_bytes streamed, at the measured copy rate
    and at the nominal 8 TB/s."""
    roof = B * peak_gbs * 1e9 / step_bytes
    roof_nominal = B * NOMINAL_HBM_GBS * 1e9 / step_bytes
    return {"bytes_per_step": step_bytes, "roofline_tok_s": roof, "frac_of_roofline": per_gpu_tok_s / roof,
            "roofline_tok_s_nominal_8tbs": roof_nominal, "frac_of_nominal_8tbs": per_gpu_tok_s / roof_nominal,
            "hbm_gbs_achieved": step_bytes * K / elapsed / 1e9}


def max_over_ranks(x, device):
    """The largest of every rank's x: the job takes as long as its slowest replica."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world, B, K, elapsed):
    """Tokens per second of the whole job: every replica's B rows x K steps over the slowest time."""
    return world * B * K / elapsed


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ---------------------------------------------------------------------------------------
# the CPU oracle (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------------------

def oracle_for(w, blob, cap):
    import oracle
    m = oracle.Model(oracle.cfg_of(w.shape, 1, cap), blob)
    s = w.shape
    if w.prompt:  # a synthetic cache of the prompt's length (values do not change the cost)
        for layer in range(s.layers):
            k, v = synth.kv_values(w.seed_kv, layer, 0, 1, s.kv, w.prompt, s.hd, bf16=s.bf16)
            m.kv_write(layer, 0, 0, k, v)
    return m


def blob_step_bytes(w, blob):
    """The weight bytes a decode step reads, from the weight blob: every weight but the embedding
    table (a tied head reads that table in full)."""
    s = w.shape
    es = 2 if s.bf16 else 4
    return blob.nbytes - (0 if s.tied else s.vocab * s.d * es)


def workload_config(w, args, world, wbytes):
    """The `config` of a bench line (both arms): the workload as the GPU arm runs it."""
    s, B, P = w.shape, w.batch, w.prompt
    pos0 = P if P else w.fill
    temp, k_, p_ = w.temp, (w.top_k or s.vocab), w.top_p
    rows = getattr(args, "rows", False)
    return {"workload": w.name, "batch": B, "prompt": P, "cache_positions": pos0,
            "weights": "bf16" if s.bf16 else "f32", "kv_cache": "bf16" if s.bf16 else "f32",
            "sampling": "greedy" if temp == 0 else f"temp {temp} top-k {k_} top-p {p_}",
            "positions": ("own per row (decode_rows): row b at %d - %d b" % (pos0, pos0 // (2 * B))
                          if rows else "shared"),
            "loop": "llm_generate_dev (graphs of 8 chained steps)" if args.generate else "llm_step_dev per step",
            "l2": "inputs larger than L2 (weights %.1f GB per step)" % (wbytes / 1e9),
            "parallelism": f"replicas x{world}"}


def time_oracle_layers(m, w, pos, nl, steps, warmup):
    """Per timed step: one token's embedding plus `nl` consecutive layers (rotating through the
    model), and the final norm + LM head on every (L / nl)-th step, so that L / nl steps do
    exactly one token's work.  Returns (seconds per token = the mean step time x L / nl, the mean
    step time, steps timed)."""
    L = w.shape.layers
    per_token = max(1, L // nl)
    times = []
    for i in range(warmup + steps):
        t0 = time.perf_counter()
        m.embed(1)
        l0 = (i * nl) % L
        for l in range(l0, min(L, l0 + nl)):
            m.layer(l, 0, pos)
        if i % per_token == per_token - 1:
            m.head()
        if i >= warmup:
            times.append(time.perf_counter() - t0)
    return float(np.mean(times)) * per_token, float(np.mean(times)), len(times)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    blob = synth.model_blob(w.shape, w.seed_weights)
    cap = w.prompt + 2
    m = oracle_for(w, blob, cap)
    nl = max(1, min(args.ref_layers, w.shape.layers))
    t0 = time.perf_counter()
    sec_per_tok, sec_per_step, n = time_oracle_layers(m, w, w.prompt, nl, args.steps, args.warmup)
    wall = time.perf_counter() - t0
    value = w.batch / (sec_per_tok * w.batch)  # one row at a time: tokens per second of one row
    sample = (f"row 0 of batch {w.batch} at position {w.prompt} over a synthetic {w.prompt}-position "
              f"cache; each step runs {nl} of {w.shape.layers} layers (the LM head every "
              f"{max(1, w.shape.layers // nl)} steps), step time scaled by {w.shape.layers // nl}")
    line = {
        "impl": "reference", "metric": "decode tok/s", "value": value, "unit": "tok/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        # ms_per_step: a timed step as it ran (the sample); ms_per_token: the scaled full token
        "ms_per_step": sec_per_step * 1e3, "ms_per_token": sec_per_tok * 1e3,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, args, world, blob_step_bytes(w, blob)),
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": wall,
    }
    print(json.dumps(line), flush=True)
    m.close()


# ---------------------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------------------

def kernel_table(pkg, h, w, B, pos):
    """Each kernel of the step timed alone (llm_profile_kernel), with its algorithmic bytes."""
    s = w.shape
    es = 2 if s.bf16 else 4
    kvb = B * 2 * s.kv * s.hd * es * (pos + 1)
    nbytes = {"qkv": (s.d + 2 * s.kvw) * s.d * es, "attention": kvb, "o_proj": s.d * s.d * es,
              "gate_up": 2 * s.ffn * s.d * es, "down": s.d * s.ffn * es,
              "lm_head": s.vocab * s.d * es, "sampler": B * s.vocab * 4}
    peak, _ = peaks()
    rows = {}
    for name, kid in pkg.KERNELS.items():
        ms = pkg.llm_profile_kernel(h, kid, B, pos, 2 * s.layers)
        gbs = nbytes[name] / (ms / 1e3) / 1e9
        rows[name] = {"us": ms * 1e3, "bytes": nbytes[name], "GB/s": gbs, "frac": gbs / peak}
    per_step = sum(rows[k]["us"] * (s.layers if k in ("qkv", "attention", "o_proj", "gate_up", "down") else 1)
                   for k in rows)
    print(json.dumps({"workload": w.name, "layers": s.layers, "batch": B, "pos": pos,
                      "kernels": rows, "sum_isolated_us_per_step": per_step}), flush=True)


def host_cpu():
    """The host CPU's model name (lscpu, else /proc/cpuinfo) and its logical core count."""
    name = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                name = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not name:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu model")):
                    name = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return name or "unknown", os.cpu_count()


def step_bytes_of(pkg, cfg, s, B, mean_pos):
    """Algorithmic bytes of one decode step: every weight but the embedding table (the tied head
    reads that table in full), plus the keys and values of positions 0..t of every row."""
    es = 2 if s.bf16 else 4
    wbytes = (pkg.llm_weight_count(cfg) - s.vocab * s.d) * es
    if s.tied:
        wbytes += s.vocab * s.d * es
    kv_bytes = B * 2 * s.layers * s.kv * s.hd * es * (mean_pos + 1)
    return wbytes, wbytes + kv_bytes


def fill_cache(model, w, torch, stream, gpu_index):
    """The workload's cache: its prompt through llm_prefill (timed: a first call captures the pass
    graphs, the second is timed with CUDA events), or synthetic keys and values."""
    s, B, P = w.shape, w.batch, w.prompt
    if not P:
        for layer in range(s.layers):
            for b in range(B):
                k, v = synth.kv_values(w.seed_kv, layer, b, B, s.kv, w.fill, s.hd, bf16=s.bf16)
                model.kv_import(layer, b, 0, k, v)
        return None
    prompt = synth.tokens(w.seed_tokens, 0, B * P, s.vocab).reshape(B, P)
    model.prefill(prompt, 0, logits=False)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index) as clocks:
        torch.cuda.nvtx.range_push(f"prefill_b{B}")  # (a profiler can select the timed region)
        e0.record(stream)
        t0 = time.perf_counter()
        model.prefill(prompt, 0, logits=True)
        wall = time.perf_counter() - t0
        e1.record(stream)
        e1.synchronize()
        torch.cuda.nvtx.range_pop()
    ms = e0.elapsed_time(e1)
    return {"tokens": B * P, "batch": B, "prompt": P, "ms": ms, "tok_s": B * P / (ms / 1e3),
            "wall_ms": wall * 1e3, "max_tokens": int(model.cfg.max_tokens) or 512,
            "what": "llm_prefill of the whole prompt (passes of prompt tokens; logits of the last)",
            "clocks": clocks.summary()}


def time_steps(pkg, torch, h, w, B, pos0, K, W, dev, stream, local, world, first, rowpos=None, generate=False):
    """W warm-up steps rewinding to pos0, then K timed steps of llm_step_dev (or one
    llm_generate_dev call) bracketed by CUDA events on the handle's stream, clocks sampled."""
    s = w.shape
    tok = [torch.from_numpy(first).to(dev), torch.empty(B, dtype=torch.int32, device=dev)]
    u_all = synth.uniforms(w.seed_uniform, 0, B * (W + K)).reshape(W + K, B)
    u_dev = torch.from_numpy(u_all).to(dev)
    temp, k_, p_ = w.temp, (w.top_k or s.vocab), w.top_p

    def step_dev(tk, i, u, ids):
        if rowpos is None:
            pkg.llm_step_dev(h, tk, B, pos0 + i, temp, k_, p_, u, ids)
        else:
            pkg.llm_step_rows_dev(h, tk, B, rowpos + i, temp, k_, p_, u, ids)

    # generation warm-up: 9 steps capture both generation graphs (8 steps, then a single step)
    GW = 9
    gen_ids = torch.empty((max(GW, K), B), dtype=torch.int32, device=dev) if generate else None
    u_gw = (torch.from_numpy(synth.uniforms(w.seed_uniform, B * (W + K), B * GW).reshape(GW, B)).to(dev)
            if generate else None)
    with torch.cuda.stream(stream):
        for i in range(W):  # warm-up: rewind to the prompt end every time
            step_dev(tok[0], 0, u_dev[i], tok[1])
        if generate:
            pkg.llm_generate_dev(h, tok[0], B, pos0, GW, temp, k_, p_, u_gw, gen_ids[:GW])
        pkg.llm_synchronize(h)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clocks:
            torch.cuda.nvtx.range_push(f"decode_b{B}")  # (a profiler can select the timed region)
            e0.record(stream)
            if generate:
                pkg.llm_generate_dev(h, tok[0], B, pos0, K, temp, k_, p_, u_dev[W:W + K], gen_ids[:K])
            else:
                for i in range(K):
                    step_dev(tok[i % 2], i, u_dev[W + i], tok[(i + 1) % 2])
            e1.record(stream)
            e1.synchronize()
            torch.cuda.nvtx.range_pop()
        pkg.llm_synchronize(h)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    return ms, clocks.summary(), u_all


def run_ours(args):
    import torch

    import llama_architecture_kv_gb300 as pkg

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    w = WORKLOADS[args.workload]
    if args.layers > 0:
        w = dataclasses.replace(w, shape=dataclasses.replace(w.shape, layers=args.layers))
    if args.prompt >= 0:
        w = dataclasses.replace(w, prompt=args.prompt)
    s, B, P = w.shape, w.batch, w.prompt
    K, W = args.steps, args.warmup
    cap = max(w.cap, P + max(W + K, 9) + 1)  # (9: the generation warm-up)
    stream = torch.cuda.Stream()

    t0 = time.perf_counter()
    blob = synth.model_blob(s, w.seed_weights)
    log(f"[bench] weights generated: {blob.nbytes / 1e9:.2f} GB in {time.perf_counter() - t0:.1f} s")
    t0 = time.perf_counter()
    model = pkg.Model(s, blob, max_batch=B, max_seq=cap, stream=stream.cuda_stream, max_tokens=args.max_tokens,
                      step_kernel=args.step_kernel, tc_min_batch=args.tc_min_batch)
    h = model.h
    log(f"[bench] model created in {time.perf_counter() - t0:.1f} s")
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        prefill = fill_cache(model, w, torch, stream, local)
    pos0 = P if P else w.fill
    log(f"[bench] cache filled to {pos0} positions in {time.perf_counter() - t0:.1f} s"
        + (f" (timed prefill {prefill['ms']:.1f} ms, {prefill['tok_s']:.0f} tok/s)" if prefill else ""))

    if args.kernels:
        kernel_table(pkg, h, w, B, pos0)
        model.close()
        return
    dev = torch.device("cuda", local)
    first = synth.tokens(w.seed_tokens, B * P, B, s.vocab)
    temp, k_, p_ = w.temp, (w.top_k or s.vocab), w.top_p
    # rows at their own positions: spread over the upper half of the cache
    rowpos = (pos0 - np.arange(B, dtype=np.int32) * (pos0 // (2 * B))).astype(np.int32) if args.rows else None
    ms, clk, u_all = time_steps(pkg, torch, h, w, B, pos0, K, W, dev, stream, local, world, first, rowpos,
                                args.generate)
    elapsed = ms / 1e3
    if world > 1:
        elapsed = max_over_ranks(elapsed, dev)
        torch.distributed.barrier()
    value = whole_job_value(world, B, K, elapsed)

    # end to end through the public host API: tokens in from pinned host memory, ids out
    tok_h = torch.from_numpy(first.copy()).pin_memory()
    ids_h = torch.empty(B, dtype=torch.int32).pin_memory()
    u_h = torch.from_numpy(u_all[:1].reshape(-1).copy()).pin_memory()
    E = min(K, 100)
    gen_h = torch.empty((E, B), dtype=torch.int32).pin_memory() if args.generate else None
    u_e = torch.from_numpy(np.ascontiguousarray(u_all[:E])).pin_memory() if args.generate else None
    torch.cuda.synchronize()
    te = time.perf_counter()
    if args.generate:
        pkg.llm_generate(h, tok_h, B, pos0, E, temp, k_, p_, u_e if temp > 0 else None, gen_h)
    for i in range(0 if args.generate else E):
        if rowpos is None:
            pkg.llm_step(h, tok_h if i == 0 else ids_h, B, pos0 + i, temp, k_, p_,
                         u_h if temp > 0 else None, ids_h)
        else:
            pkg.llm_step_rows(h, tok_h if i == 0 else ids_h, B, rowpos + i, temp, k_, p_,
                              u_h if temp > 0 else None, ids_h)
    e2e_s = time.perf_counter() - te
    e2e = {"value": B * E / e2e_s, "unit": "tok/s",
           "h2d_bytes_per_step": (4 * B / E if args.generate else 4 * B) + (4 * B if temp > 0 else 0),
           "d2h_bytes_per_step": 4 * B}

    # the dominant kernel, timed alone (consecutive launches walk the layers: weights from HBM);
    # five timings of 4 x layers launches each, the median reported
    reps = 4 * s.layers
    # (at a position every row has reached: rows at their own positions sit at or above their minimum)
    kpos = int(rowpos.min()) if rowpos is not None else pos0
    kms_all = [pkg.llm_profile_kernel(h, GATEUP, B, kpos, reps) for _ in range(5)]
    kms = float(np.median(kms_all))
    bytes_gu = 2 * s.ffn * s.d * (2 if s.bf16 else 4)  # algorithmic: the gate and up weights
    achieved = bytes_gu / (kms / 1e3) / 1e9
    peak, peak_kind = peaks()
    tc = s.bf16 and B >= (args.tc_min_batch or 2)  # the handle's tensor-core threshold
    if tc:
        kname = "tc_gemm_kernel (gate/up, timed with its tc_prep_kernel: x1 = x + o_proj, norm, bf16 split)"
        traffic = traffic_from_profile("gemm.cu", "tc_gemm_gate_up_llama8b_b32.md") if w.name == "llama8b_b32" else None
    else:
        kname = ("gemv_tma_kernel<EPI_SWIGLU> (norm + gate/up + SwiGLU, bulk-copy rings)" if s.bf16 and B == 1
                 else "gemv_kernel<EPI_SWIGLU> (norm + gate/up + SwiGLU)")
        traffic = traffic_from_profile("gemv.cu", "gate_up_gemv_llama8b_b1.md") if w.name == "llama8b_b1" else None
    roofline = {"bound": "hbm", "kernel": kname,
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_kind": peak_kind, "traffic": traffic, "ms_per_launch": kms,
                "ms_per_launch_runs": kms_all,
                "algorithmic_bytes_per_launch": bytes_gu}
    mean_pos = (float(np.mean(rowpos)) if rowpos is not None else pos0) + (K - 1) / 2
    wbytes, step_bytes = step_bytes_of(pkg, model.cfg, s, B, mean_pos)
    step_roof = step_roofline(step_bytes, B, peak, value / world, K, elapsed)
    launches = (K * (pkg.llm_step_kernels(h, B, temp, k_) + 1) + K // 8 + K % 8 if args.generate
                else K * pkg.llm_step_kernels(h, B, temp, k_))
    model.close()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        t0 = time.perf_counter()
        m = oracle_for(w, blob, pos0 + 2)
        n = max(1, args.cpu_steps)
        ts = []
        for i in range(n):
            t1 = time.perf_counter()
            m.forward(0, int(first[0]), pos0 + (i % 2), logits=True)
            ts.append(time.perf_counter() - t1)
        m.close()
        cpu_name, nproc = host_cpu()
        cpu = {"value": 1.0 / float(np.mean(ts)), "unit": "tok/s", "cores": 1, "kind": "oracle",
               "cpu_model": cpu_name, "nproc": nproc,
               "sample": f"{n} full decode steps of row 0 at position {pos0} over a synthetic "
                         f"{pos0}-position cache, single-threaded f32 C on one of {nproc} cores ({cpu_name})"}
        log(f"[bench] cpu baseline in {time.perf_counter() - t0:.1f} s")

    # the batch-32 half of the metric, in the same run (same weights, its own handle)
    b32 = None
    if (w.name == "llama8b_b1" and args.b32_steps > 0 and world == 1 and not args.rows and not args.generate
            and args.layers <= 0 and args.prompt < 0):
        w32 = WORKLOADS["llama8b_b32"]
        K32, W32 = args.b32_steps, 3
        cap32 = max(w32.cap, w32.prompt + W32 + K32 + 1)
        m32 = pkg.Model(s, blob, max_batch=w32.batch, max_seq=cap32, stream=stream.cuda_stream,
                        max_tokens=args.max_tokens)
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            pf32 = fill_cache(m32, w32, torch, stream, local)
        log(f"[bench] batch 32: cache filled in {time.perf_counter() - t0:.1f} s")
        first32 = synth.tokens(w32.seed_tokens, w32.batch * w32.prompt, w32.batch, s.vocab)
        ms32, clk32, _ = time_steps(pkg, torch, m32.h, w32, w32.batch, w32.prompt, K32, W32, dev, stream, local,
                                    world, first32)
        v32 = w32.batch * K32 / (ms32 / 1e3)
        _, sb32 = step_bytes_of(pkg, m32.cfg, s, w32.batch, w32.prompt + (K32 - 1) / 2)
        b32 = {"workload": w32.name, "batch": w32.batch, "value": v32, "unit": "tok/s", "steps": K32,
               "warmup": W32, "ms_per_step": ms32 / K32,
               "step_roofline": step_roofline(sb32, w32.batch, peak, v32, K32, ms32 / 1e3),
               "clocks": clk32, "prefill": pf32,
               "gpu_launches": K32 * pkg.llm_step_kernels(m32.h, w32.batch, 0.0)}
        m32.close()

    line = {
        "metric": "decode tok/s", "value": value, "unit": "tok/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, args, world, wbytes),
        "roofline": roofline, "step_roofline": step_roof, "cpu_baseline": cpu, "e2e": e2e,
        "clocks": clk, "prefill": prefill, "batch32": b32,
        # a generation step replaces the prologue by its own and ends with one copy of its draws;
        # each graph launch (8 steps, then single steps) is preceded by one state update
        "gpu_launches": launches,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
