"""Benchmark: sampled-token logprobs/s at diff = 0 on the dense-decoder workload.

One step = one RL data step of the 4-layer d=512 dense decoder (8 heads x 64,
SwiGLU 1408, vocab 32000, RoPE), batch 16, prompts 128-512 tokens, 256 greedy
tokens: the rollout (packed prefill of the prompts + 255 decode steps replayed
from a CUDA graph) and the training-side recompute (one packed chunked prefill
over prompt + response) of all 4096 sampled tokens' logprobs.  value = sampled
tokens whose logprob was produced by both sides and checked bit-equal, per second.
The same step in BI_FAST mode (split-K, batch-dependent attention split, vocab
split) is timed for the "% of non-invariant path" ratio.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the only reference this method has) on
a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sampled-token logprobs/s on 1 GB300 at diff=0; % of non-invariant path; % roofline"
UNIT = "logprobs/s"
WORKLOAD = ("dense decoder 4 layers, d=512, 8 heads x 64, SwiGLU 1408, vocab 32000, RoPE, bf16 weights N(0,0.02); "
            "batch 16, prompts 128-512 tokens (uniform), 256 greedy tokens; step = rollout (prefill + CUDA-graph "
            "decode) + training recompute (packed prefill, chunk 2048) of all 4096 sampled-token logprobs")


def _flat_numbers(d, prefix=""):
    """(dotted key, number) pairs of a JSON object, nested objects included."""
    out = []
    if isinstance(d, dict):
        for k, v in d.items():
            out += _flat_numbers(v, f"{prefix}.{k}" if prefix else str(k))
    elif isinstance(d, (int, float)) and not isinstance(d, bool):
        out.append((prefix.lower(), float(d)))
    return out


def parse_peaks(d):
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained) from the measured-peaks
    record, or None.  Keys are matched by what they name (hbm / bf16 / sustained),
    flat or nested (a "value" leaf under the named key counts), TB/s and PFLOP/s
    converted."""
    nums = _flat_numbers(d)

    def pick(want, avoid=()):
        for k, v in nums:
            if all(w in k for w in want) and not any(a in k for a in avoid) and v > 0:
                return k, v
        return None, None

    kh, hbm = pick(("hbm",), ("clock", "mhz", "util", "pct", "frac"))
    kb, bf = pick(("bf16",), ("sustain", "clock", "mhz", "util", "pct", "frac"))
    ks, bs = pick(("bf16", "sustain"), ("clock", "mhz", "util", "pct", "frac"))
    if hbm is None or bf is None:
        return None
    if "tb" in kh or hbm < 100:          # TB/s
        hbm *= 1000.0
    if "pflop" in kb or bf < 50:         # PFLOP/s
        bf *= 1000.0
    if bs is None:
        bs = bf
    elif "pflop" in ks or bs < 50:
        bs *= 1000.0
    return hbm, bf, bs


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            got = parse_peaks(json.load(open(p)))
            if got:
                return got[0], got[1], got[2], "measured"
        except Exception:
            pass
    return 6800.0, 1900.0, 1700.0, "fallback"


class Clocks:
    """Samples nvidia-smi during the timed region."""

    def __init__(self, path):
        self.path = path
        self.proc = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "200",
                                          "-i", str(int(os.environ.get("LOCAL_RANK", "0")))], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        try:
            rows = [r.split(",") for r in open(self.path).read().strip().splitlines() if r.strip()]
        except Exception:
            return None
        if not rows:
            return None
        sm = [float(r[1]) for r in rows]
        mx = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": reasons, "samples": len(rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    return ws, rank


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise maximum of per-rank timings (the slowest replica sets the job's time).
    `dist` is torch.distributed (or None for a single process)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_rate(n_replicas, units_per_replica, ms):
    """Units every replica processed in one step, divided by the step time (ms)."""
    return n_replicas * units_per_replica / (ms / 1000.0)


def _cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 0) for i in threadpool_info()), default=0)
        if n:
            return n
    except Exception:
        pass
    return os.cpu_count()


def oracle_sample(budget_s=12.0, gens=None, seed_extra=0):
    """Time the CPU oracle scoring sampled tokens of the workload, sequence by sequence,
    until the budget is used.  Returns (logprobs/s, n_logprobs, seconds, lp list)."""
    from oracle import model as omodel
    from synthetic import C2, make_decoder_weights, make_prompts
    cfg = C2
    shape = cfg["shape"]
    wb = make_decoder_weights(shape, seed=cfg["seed"], w_std=cfg["w_std"])
    prompts = make_prompts(cfg["batch"], cfg["prompt_min"], cfg["prompt_max"], shape.vocab, cfg["seed"])
    W = omodel.weights_to_f32(wb)
    rng = np.random.default_rng(99 + seed_extra)
    n, t0, out = 0, time.perf_counter(), []
    b = 0
    while True:
        g = gens[b] if gens is not None else rng.integers(0, shape.vocab, cfg["gen"]).astype(np.int32)
        _, lp, _ = omodel.score_generation(W, shape, prompts[b], g)
        out.append((b, lp))
        n += len(lp)
        b = (b + 1) % len(prompts)
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return n / dt, n, dt, out


def _cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine()


def oracle_config_rates(small: bool):
    """The CPU oracle on a bounded sample of each workload, in the configuration
    table's units.  `small` (the one-thread run) takes smaller samples of the
    workloads whose rows are independent.  Returns {config: {value, unit, sample, s}}."""
    from oracle import model as omodel
    from oracle import moe as omoe
    from synthetic import (C1, C2, C3, C4, C5, bits_to_f32, make_c5_prompt_lengths, make_decoder_weights,
                           make_logprob_head, make_moe_layer, make_prompts)
    res = {}

    def put(name, units, unit, dt, sample):
        res[name] = {"value": round(units / dt, 2), "unit": unit, "s": round(dt, 2), "sample": sample}

    # logprob head, all 512 rows
    h = make_logprob_head(C1["n_seq"] * C1["seq_len"], C1["d"], C1["vocab"], C1["w_std"], C1["seed"])
    hf, gf, wf = bits_to_f32(h["h"]), bits_to_f32(h["gain"]), bits_to_f32(h["w"])
    t0 = time.perf_counter()
    omodel.logprob_head(hf, gf, wf, h["ids"])
    put("logprob_head_512x256x4096", len(h["ids"]), "logprobs/s", time.perf_counter() - t0, "all 512 rows")
    # dense decoder: whole sequences, 256 teacher-forced logprobs each (seeded ids)
    shape = C2["shape"]
    W = omodel.weights_to_f32(make_decoder_weights(shape, seed=C2["seed"], w_std=C2["w_std"]))
    prompts = make_prompts(C2["batch"], C2["prompt_min"], C2["prompt_max"], shape.vocab, C2["seed"])
    rng = np.random.default_rng(99)
    n_seq = 1 if small else 4
    t0 = time.perf_counter()
    for b in range(n_seq):
        omodel.score_generation(W, shape, prompts[b], rng.integers(0, shape.vocab, C2["gen"]))
    put("dense_decoder_16x256", n_seq * C2["gen"], "logprobs/s", time.perf_counter() - t0,
        f"{n_seq} of 16 sequences, {C2['gen']} sampled-token logprobs each")
    del W
    # MoE layer: a token subset (tokens are independent)
    m = make_moe_layer(C3["n_tokens"], C3["d"], C3["ffn"], C3["n_experts"], C3["w_std"], C3["seed"])
    n_tok = 64 if small else 512
    x, lg = bits_to_f32(m["x"][:n_tok]), m["router_logits"][:n_tok]
    w13, w2 = bits_to_f32(m["w13"]), bits_to_f32(m["w2"])
    t0 = time.perf_counter()
    omoe.moe_layer(x, lg, w13, w2, C3["top_k"])
    put("moe_layer_4096x2048_e64_top8", n_tok, "tokens/s", time.perf_counter() - t0,
        f"{n_tok} of 4096 tokens (rows are independent)")
    del m, w13, w2
    # large-vocab logprob: a row subset
    n_row = 32 if small else 256
    rng4 = np.random.default_rng(C4["seed"])
    from synthetic import normal_bf16
    h4 = bits_to_f32(normal_bf16(rng4, (n_row, C4["d"]), 1.0))
    w4 = bits_to_f32(normal_bf16(rng4, (C4["vocab"], C4["d"]), C4["w_std"]))
    ids4 = rng4.integers(0, C4["vocab"], n_row)
    t0 = time.perf_counter()
    omodel.logprob_head(h4, None, w4, ids4, norm=False)
    put("large_vocab_logprob_16384x4096x129280", n_row, "logprobs/s", time.perf_counter() - t0,
        f"{n_row} of 16384 rows (rows are independent)")
    del w4
    # long-context GQA: the shortest sequence, 8 teacher-forced decode tokens
    shape5 = C5["shape"]
    W5 = omodel.weights_to_f32(make_decoder_weights(shape5, seed=C5["seed"], w_std=C5["w_std"]))
    lens = make_c5_prompt_lengths(C5["batch"], C5["ctx_min"], C5["ctx_max"], C5["seed"])
    rng5 = np.random.default_rng(C5["seed"] + 3)
    prompts5 = [rng5.integers(0, shape5.vocab, int(n)).astype(np.int32) for n in lens]
    b = int(np.argmin(lens))
    t0 = time.perf_counter()
    omodel.score_generation(W5, shape5, prompts5[b], np.random.default_rng(5).integers(0, shape5.vocab, 8))
    put("long_context_gqa_decode_step_64seq", 8, "logprobs/s", time.perf_counter() - t0,
        f"the shortest of the 64 sequences ({int(lens[b])} prompt tokens), 8 teacher-forced logprobs")
    return res


def _oracle_rates_subprocess(one_thread: bool, timeout_s=600):
    """Run oracle_config_rates in a fresh interpreter (BLAS thread counts are fixed
    at import); one_thread sets every BLAS/OpenMP pool to one thread."""
    import subprocess
    env = dict(os.environ)
    if one_thread:
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
            env[k] = "1"
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-rates"] + (["--one-thread"] if one_thread else [])
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=timeout_s)
        lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
        return json.loads(lines[-1]) if r.returncode == 0 and lines else {"error": r.stderr[-300:]}
    except Exception as e:   # the baseline is reported, never required
        return {"error": str(e)[:300]}


def run_reference(args):
    ws, rank = _dist()
    if rank != 0:
        return
    for i in range(args.warmup):
        oracle_sample(budget_s=0.1, seed_extra=i)
    vals, ns, dts = [], 0, 0.0
    for i in range(args.steps):
        v, n, dt, _ = oracle_sample(budget_s=2.0, seed_extra=100 + i)
        vals.append(v)
        ns += n
        dts += dt
    value = ns / dts
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dts / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "reference": "CPU oracle (numpy fp32, fp64 logsumexp)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": _cpu_cores(), "kind": "oracle",
                             "sample": "per step: teacher-forced oracle scoring of whole sequences (256 "
                                       "logprobs each) for ~2 s"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import invariant_forward_policy_gb300 as bi
    from invariant_forward_policy_gb300.decoder import Decoder, Episode
    from synthetic import C2, make_decoder_weights, make_prompts

    ws_n, rank = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    cfg = C2
    shape = cfg["shape"]
    wb = make_decoder_weights(shape, seed=cfg["seed"], w_std=cfg["w_std"])
    prompts = make_prompts(cfg["batch"], cfg["prompt_min"], cfg["prompt_max"], shape.vocab, cfg["seed"])
    B, G = len(prompts), cfg["gen"]
    dec = Decoder(shape, wb, max_pos=1024, device=dev)
    lens = [len(p) for p in prompts]
    prompt_host = torch.from_numpy(np.concatenate(prompts).astype(np.int32)).pin_memory()
    prompt_dev = prompt_host.to(dev)
    ep = Episode(dec, lens, G, mode=bi.BI_INVARIANT)
    ep_fast = Episode(dec, lens, G, mode=bi.BI_FAST)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # > L2 (129 MB)
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def timed(e, k, keep, tag):
        times = []
        for i in range(k):
            flush.zero_()
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            if i == 0:
                torch.cuda.nvtx.range_push(f"step_{tag}")   # lets ncu capture one whole step
            s0.record(stream)
            ids, lp_r, lp_t = e.run(prompt_dev)
            s1.record(stream)
            if i == 0:
                torch.cuda.nvtx.range_pop()
            if keep is not None:
                keep.append((ids.clone(), lp_r.clone(), lp_t.clone()))
            times.append((s0, s1))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in times]

    for _ in range(max(args.warmup, 3)):
        ep.run(prompt_dev)
        ep_fast.run(prompt_dev)
    barrier()
    n0 = bi.bi_launch_count()
    ep.run(prompt_dev)
    torch.cuda.synchronize()
    launches_eager_part = bi.bi_launch_count() - n0     # host-issued launches (prefill, recompute, first step)
    # decode launches replayed per graph replay = launches issued by one eager decode step
    n1 = bi.bi_launch_count()
    ep._decode_step()
    torch.cuda.synchronize()
    per_decode = bi.bi_launch_count() - n1
    gpu_launches = launches_eager_part + per_decode * (G - 1)
    ep.run(prompt_dev)   # restore a consistent state after the probe step

    results = []
    barrier()
    clocks_path = args.clocks_csv
    if not clocks_path:
        fd, clocks_path = tempfile.mkstemp(prefix="clocks_bench_", suffix=".csv")
        os.close(fd)
    with Clocks(clocks_path) as ck:
        t_inv = timed(ep, args.steps, results, "invariant")
        t_fast = timed(ep_fast, args.steps, None, "fast")
    barrier()
    clocks = ck.summary()
    ms_inv = sum(t_inv) / len(t_inv)
    ms_fast = sum(t_fast) / len(t_fast)
    ms_inv, ms_fast = max_over_ranks([ms_inv, ms_fast], dist, device=dev)
    tokens = B * G
    value = whole_job_rate(ws_n, tokens, ms_inv)
    fast_value = whole_job_rate(ws_n, tokens, ms_fast)

    # diff = 0 in every timed step (rollout vs recompute) and identical across steps
    from oracle.ops import diff_stats  # host-side acceptance statistics
    diffs = [diff_stats(r[1].cpu().numpy().ravel(), r[2].cpu().numpy().ravel()) for r in results]
    bitwise = all(torch.equal(r[1].view(torch.int32), r[2].view(torch.int32)) for r in results)
    same_across = all(torch.equal(r[0], results[0][0]) and torch.equal(r[1].view(torch.int32),
                                                                         results[0][1].view(torch.int32)) for r in results)
    worst = {k: max(d[k] for d in diffs) for k in diffs[0]}

    # end to end through the public API with host buffers: H2D prompts, D2H ids + both logprob sets
    e2e_t = []
    out_ids = torch.empty((B, G), dtype=torch.int32).pin_memory()
    out_lr = torch.empty((B, G), dtype=torch.float32).pin_memory()
    out_lt = torch.empty((B, G), dtype=torch.float32).pin_memory()
    # the first device-to-host copy into pinned memory carries a one-time set-up
    # (~0.6 s on GB300): warm-up steps of this path are untimed, like the device ones
    for i in range(max(args.warmup, 3) + args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        pd = prompt_host.to(dev, non_blocking=True)
        ids, lr, lt = ep.run(pd)
        out_ids.copy_(ids, non_blocking=True)
        out_lr.copy_(lr, non_blocking=True)
        out_lt.copy_(lt, non_blocking=True)
        torch.cuda.synchronize()
        if i >= max(args.warmup, 3):
            e2e_t.append(time.perf_counter() - t0)
    e2e_val = ws_n * tokens / (sum(e2e_t) / len(e2e_t))

    # roofline of the dominant kernel (timed live, same shapes as in the step)
    roof = roofline_probe(dec, ep, args)
    kernels = kernel_table(args) if not args.no_kernels else None
    configs = config_table(args) if not args.no_configs else None

    # CPU oracle baseline on a bounded sample (rank 0, N = 1 only), also a parity spot check
    cpu = None
    parity = None
    if rank == 0 and ws_n == 1 and not args.no_cpu:
        gens = results[0][0].cpu().numpy()
        v, n, dt, outs = oracle_sample(budget_s=args.cpu_budget, gens=gens)
        cpu = {"value": v, "unit": UNIT, "cores": _cpu_cores(), "kind": "oracle",
               "sample": f"teacher-forced oracle scoring of {len(outs)} sequences, cycling over the {B} of the "
                         f"workload with the GPU's sampled ids ({n} sampled-token logprobs) in {dt:.1f} s"}
        lr0 = results[0][1].cpu().numpy()
        errs = np.concatenate([np.abs(lr0[b] - lp) for b, lp in outs])
        parity = {"max": float(errs.max()), "mean": float(errs.mean()), "p99": float(np.quantile(errs, 0.99)),
                  "n": int(errs.size), "bound_max": 2e-2, "bound_mean": 5e-3,
                  "floor": "max 1.1e-2 / mean 2.8e-3 (oracle vs its own fp64 and bf16-P variants)"}
        # the oracle on every workload's sample, all cores and one thread (fresh interpreters)
        cpu["configs"] = {"all_cores": _oracle_rates_subprocess(False), "one_thread": _oracle_rates_subprocess(True)}
        cpu["cpu_model"] = _cpu_model()

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_n, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_inv, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": WORKLOAD, "l2": "flushed (256 MB write) between timed steps",
                           "parallelism": f"replicas x{ws_n}" if ws_n > 1 else "1 GPU",
                           "invariant_fraction_of_non_invariant": round(value / fast_value, 4)},
                "diff": {**worst, "bitwise_all_steps": bitwise, "identical_across_steps": same_across},
                "non_invariant": {"value": fast_value, "ms_per_step": ms_fast,
                                  "invariant_fraction": value / fast_value},
                "roofline": roof,
                "kernels": kernels,
                "configs": configs,
                "cpu_baseline": cpu,
                "oracle_err": parity,
                "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": int(prompt_host.numel() * 4),
                        "d2h_bytes_per_step": int(B * G * 12)},
                "gpu_launches": int(gpu_launches),
                "clocks": clocks}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def _graph_us(fn, n=20, reps=10):
    """Per-launch device time of `fn` replayed from a CUDA graph of n launches (CUDA events)."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(n):
            fn()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1000.0 / (n * reps)


def roofline_probe(dec, ep, args):
    """Roofline of the step's dominant kernel class, the decode-size GEMMs (QKV, O,
    gate/up+SwiGLU, down of every layer on the mma.sync rows schedule, and the
    fused lm_head+logprob on the tcgen05 tile schedule with its LSE epilogue):
    each is launched at its decode shape (M = 16) from a CUDA graph, the way the
    decode step runs it, and timed with CUDA events.  achieved = the algorithmic
    bytes of one decode step's GEMMs (weights + activations in + out) / their
    summed launch time.  The weights are L2-resident across decode steps (the
    58.5 MB model fits the 129 MB L2): these launches are latency-bound."""
    import torch
    import invariant_forward_policy_gb300 as bi
    hbm, tf, tf_s, src = _peaks()
    s = dec.shape
    B, d, F, V = ep.B, s.d, s.ffn, s.vocab
    nqkv = (s.n_heads_q + 2 * s.n_heads_kv) * s.head_dim
    hq = s.n_heads_q * s.head_dim
    dev = dec.device
    lw = dec.layers[0]
    x = (0.5 * torch.randn((B, max(d, hq, F)), device=dev)).to(torch.bfloat16)
    outs = torch.empty((B, max(nqkv, d, F)), dtype=torch.bfloat16, device=dev)
    lp = torch.empty(B, dtype=torch.float32, device=dev)
    am = torch.empty(B, dtype=torch.int32, device=dev)
    wsh = torch.empty(bi.bi_lm_head_logprob_workspace_size(B, V, d), dtype=torch.uint8, device=dev)
    xd, xh, xf = x[:, :d].contiguous(), x[:, :hq].contiguous(), x[:, :F].contiguous()
    shapes = [
        ("qkv", lambda: bi.bi_gemm(xd, B, d, lw["wqkv"], nqkv, outs), nqkv * d * 2 + B * d * 2 + B * nqkv * 2),
        ("o", lambda: bi.bi_gemm(xh, B, hq, lw["wo"], d, outs), d * hq * 2 + B * hq * 2 + B * d * 2),
        ("gate_up_swiglu", lambda: bi.bi_gemm(xd, B, d, lw["w13"], 2 * F, outs, bi.BI_DTYPE_BF16, bi.BI_EPI_SWIGLU),
         2 * F * d * 2 + B * d * 2 + B * F * 2),
        ("down", lambda: bi.bi_gemm(xf, B, F, lw["w2"], d, outs), d * F * 2 + B * F * 2 + B * d * 2),
    ]
    per_step_us, per_step_bytes, detail = 0.0, 0, {}
    for name, fn, nbytes in shapes:
        us = _graph_us(fn)
        detail[name] = round(us, 2)
        per_step_us += s.n_layers * us
        per_step_bytes += s.n_layers * nbytes
    us = _graph_us(lambda: bi.bi_lm_head_logprob(xd, B, d, dec.w["lm_head"], V, None, lp, am, bi.BI_INVARIANT, wsh))
    detail["lm_head_logprob_fused"] = round(us, 2)
    per_step_us += us
    per_step_bytes += V * d * 2 + B * d * 2 + B * 8
    achieved = per_step_bytes / (per_step_us * 1e-6) / 1e9
    return {"kernel": "decode-size GEMM launches of one decode step (M 16): gemm_rows_kernel for QKV, O, "
                      "gate/up+SwiGLU and down per layer; gemm_tc_kernel<EPI_LSE> for the fused lm_head + log-softmax",
            "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "traffic": None, "us_per_decode_step": round(per_step_us, 2), "us_per_launch": detail,
            "algorithmic_bytes_per_decode_step": per_step_bytes, "peak_source": src,
            "note": "weights L2-resident across decode steps; launches are latency-bound (a few us each, "
                    "16 rows); frac of the HBM copy peak"}


def kernel_table(args):
    """Achieved rates of the other kernels at their workload shapes (CUDA events,
    warm L2 unless stated): decode attention of the long-context decoder (HBM),
    vocab-wide logprob (HBM), RMSNorm (HBM), and the large GEMMs (tensor)."""
    import torch
    import invariant_forward_policy_gb300 as bi
    from synthetic import C5, make_c5_prompt_lengths
    hbm, tf, tf_s, src = _peaks()
    dev = torch.device("cuda")
    out = {}
    # decode attention, long-context GQA shape: 64 sequences, contexts 1K-32K log-uniform, 4 kv heads x 128
    lens = make_c5_prompt_lengths(C5["batch"], C5["ctx_min"], C5["ctx_max"], C5["seed"])
    B, Hq, Hkv, hd = len(lens), 16, 4, 128
    mb = int(-(-lens.max() // 64))
    nblk = int(sum(-(-int(n) // 64) for n in lens))
    kc = (0.5 * torch.randn((nblk, Hkv, 64, hd), device=dev)).to(torch.bfloat16)
    vc = (0.5 * torch.randn((nblk, Hkv, 64, hd), device=dev)).to(torch.bfloat16)
    tab = torch.full((B, mb), -1, dtype=torch.int32)
    o = 0
    for b, n in enumerate(lens):
        k = -(-int(n) // 64)
        tab[b, :k] = torch.arange(o, o + k, dtype=torch.int32)
        o += k
    bt = tab.to(dev)
    q = (0.5 * torch.randn((B, Hq, hd), device=dev)).to(torch.bfloat16)
    seq = torch.arange(B, dtype=torch.int32, device=dev)
    row0 = torch.arange(B + 1, dtype=torch.int32, device=dev)
    pos0 = torch.from_numpy((lens - 1).astype("int32")).to(dev)
    ao = torch.empty((B, Hq * hd), dtype=torch.bfloat16, device=dev)
    max_ctx = int(lens.max())
    ws = torch.empty(bi.bi_attention_workspace_size(B, Hq, hd, max_ctx, 512), dtype=torch.uint8, device=dev)
    us = _graph_us(lambda: bi.bi_attention(q, B, seq, row0, pos0, B, 1, Hq, Hkv, hd, kc, vc, bt, mb, nblk, max_ctx, 512,
                                           hd ** -0.5, ws, ao), n=5, reps=5)
    nbytes = int(lens.sum()) * Hkv * hd * 2 * 2
    out["attention_decode_long_context"] = {"shape": f"64 seqs, ctx {int(lens.min())}-{max_ctx} (sum {int(lens.sum())}), "
                                            "16/4 heads x 128, split 512", "us": round(us, 1),
                                            "GB/s": round(nbytes / us / 1e3, 1), "frac": round(nbytes / us / 1e3 / hbm, 3),
                                            "bound": "hbm", "note": "KV (1.2 GB) exceeds L2"}
    # the same decode through an FP8 KV cache: attention reads the codes and scales
    # directly (the drivers' path), and the pages' literal form (dequantise-and-gather
    # into a bf16 workspace, then the bf16 attention) for comparison
    k8 = torch.randint(0, 0x7E, (nblk, Hkv, 64, hd), dtype=torch.uint8, device=dev)
    v8 = torch.randint(0, 0x7E, (nblk, Hkv, 64, hd), dtype=torch.uint8, device=dev)
    ks8 = torch.full((nblk, Hkv, 64), 2.0 ** -8, device=dev)
    vs8 = torch.full_like(ks8, 2.0 ** -8)
    kw = torch.empty((B * mb, Hkv, 64, hd), dtype=torch.bfloat16, device=dev)
    vw = torch.empty_like(kw)
    wbt = torch.empty((B, mb), dtype=torch.int32, device=dev)
    b8 = int(lens.sum()) * Hkv * (hd + 4) * 2
    us8 = _graph_us(lambda: bi.bi_attention_fp8(q, B, seq, row0, pos0, B, 1, Hq, Hkv, hd, k8, v8, ks8, vs8, bt, mb,
                                                nblk, max_ctx, 512, hd ** -0.5, ws, ao), n=5, reps=5)

    def gather_step():
        bi.bi_kv_fp8_gather(k8, v8, ks8, vs8, nblk, seq, row0, pos0, B, Hkv, hd, bt, mb, kw, vw, wbt)
        bi.bi_attention(q, B, seq, row0, pos0, B, 1, Hq, Hkv, hd, kw, vw, wbt, mb, B * mb, max_ctx, 512, hd ** -0.5,
                        ws, ao)
    usg = _graph_us(gather_step, n=5, reps=5)
    out["attention_decode_long_context_fp8_kv"] = {
        "us": round(us8, 1), "GB/s": round(b8 / us8 / 1e3, 1), "frac": round(b8 / us8 / 1e3 / hbm, 3), "bound": "hbm",
        "gather_path_us": round(usg, 1),
        "note": "algorithmic bytes = the FP8 cache (codes + scales) read once; pages expanded to bf16 in shared "
                "memory (bound by that expansion, not by HBM); gather_path_us = dequantise-and-gather + bf16 attention"}
    del kc, vc, k8, v8, kw, vw
    # vocab-wide logprob, large-vocab shape (8.47 GB of fp32 logits, > L2)
    T, Vv = 16384, 129280
    logits = torch.randn((T, Vv), device=dev)
    lp = torch.empty(T, device=dev)
    ids = torch.randint(0, Vv, (T,), dtype=torch.int32, device=dev)
    us = _graph_us(lambda: bi.bi_logprob_gather(logits, ids, T, Vv, lp), n=2, reps=3)
    out["logprob_16384x129280"] = {"us": round(us, 1), "GB/s": round(T * Vv * 4 / us / 1e3, 1),
                                   "frac": round(T * Vv * 4 / us / 1e3 / hbm, 3), "bound": "hbm"}
    del logits
    # RMSNorm with residual add, 65536 rows x 2048 (read x, residual, write residual, y: 4 x 268 MB)
    Rr, dd = 65536, 2048
    xx = torch.randn((Rr, dd), device=dev).to(torch.bfloat16)
    rr = torch.randn((Rr, dd), device=dev).to(torch.bfloat16)
    yy = torch.empty_like(xx)
    gg = torch.ones(dd, device=dev).to(torch.bfloat16)
    us = _graph_us(lambda: bi.bi_rmsnorm(xx, rr, gg, yy, Rr, dd), n=5, reps=5)
    out["rmsnorm_residual_65536x2048"] = {"us": round(us, 1), "GB/s": round(4 * Rr * dd * 2 / us / 1e3, 1),
                                          "frac": round(4 * Rr * dd * 2 / us / 1e3 / hbm, 3), "bound": "hbm"}
    del xx, rr, yy
    # deterministic Top-K (sparse-attention indexer budget K = 2048): one decode step of the
    # long-context batch (64 rows, contexts 1K-32K) and one 2048-row prefill chunk at 30K-32K
    for tag, nv in (("topk_decode_64rows_ctx1k-32k_k2048", lens.astype(np.int32)),
                    ("topk_prefill_2048rows_ctx30k-32k_k2048", np.arange(30721, 32769, dtype=np.int32))):
        T, ld = len(nv), int(nv.max())
        S = torch.randn((T, ld), device=dev)
        nvd = torch.from_numpy(nv).to(dev)
        idx = torch.empty((T, 2048), dtype=torch.int32, device=dev)
        us_i = _graph_us(lambda: bi.bi_topk(S, T, ld, nvd, 2048, idx, bi.BI_INVARIANT), n=5, reps=5)
        us_f = _graph_us(lambda: bi.bi_topk(S, T, ld, nvd, 2048, idx, bi.BI_FAST), n=5, reps=5)
        nbytes = float(nv.astype(np.int64).sum()) * 4
        out[tag] = {"us": round(us_i, 1), "GB/s": round(nbytes / us_i / 1e3, 1),
                    "frac": round(nbytes / us_i / 1e3 / hbm, 3), "bound": "hbm",
                    "non_invariant_us": round(us_f, 1), "invariant_fraction": round(us_f / us_i, 3),
                    "note": "algorithmic bytes = the scores read once; 4 radix passes + 1 ordered pass re-read them"}
        del S
    # Mamba-2 chunked scan (32 heads x 64, state 128, 8 B/C groups, chunk 64): a prefill
    # of 16 sequences x 2048 and a decode step of 64 sequences at mid-chunk positions.
    Hs, Gs, Ps, Ns, Qs = 32, 8, 64, 128, 64
    alu_peak = 152 * 128 * 2 * 2.07e9 / 1e12      # fp32 FMA lanes x 2 FLOP x max SM clock, TFLOP/s
    for tag, n_seq, per in (("ssd_prefill_16x2048", 16, 2048), ("ssd_decode_64seq", 64, 1)):
        T = n_seq * per
        xs = torch.randn((T, Hs, Ps), device=dev).to(torch.bfloat16)
        Bs = (torch.randn((T, Gs, Ns), device=dev) * Ns ** -0.5).to(torch.bfloat16)
        Cs = (torch.randn((T, Gs, Ns), device=dev) * Ns ** -0.5).to(torch.bfloat16)
        la = -torch.rand((T, Hs), device=dev) * 0.2
        st = torch.zeros((n_seq, bi.bi_ssd_state_bytes(Hs, Gs, Ps, Ns, Qs) // 4), device=dev)
        ys = torch.empty((T, Hs, Ps), device=dev)
        sq = torch.arange(n_seq, dtype=torch.int32, device=dev)
        r0 = torch.arange(0, T + 1, per, dtype=torch.int32, device=dev)
        p0 = torch.full((n_seq,), 0 if per > 1 else 40, dtype=torch.int32, device=dev)
        us = _graph_us(lambda: bi.bi_ssd_chunk_scan(xs, Bs, Cs, la, sq, r0, p0, n_seq, per, Hs, Gs, Ps, Ns, Qs, st,
                                                    n_seq, ys), n=3, reps=3)
        if per > 1:   # every chunk complete: rows + exit states
            fma = n_seq * Hs * (per // Qs) * (Qs * (Qs + 1) / 2 * Ns + Qs * Ps * (Ns + (Qs + 1) / 2) + Ns * Ps * Qs)
        else:         # one row at offset 40: its chunk row and no exit state
            fma = n_seq * Hs * (41 * Ns + Ps * (Ns + 41))
        out[tag] = {"us": round(us, 1), "TFLOP/s": round(2 * fma / us / 1e6, 2),
                    "frac": round(2 * fma / us / 1e6 / alu_peak, 3), "bound": "alu",
                    "peak": round(alu_peak, 1), "peak_note": "fp32 FMA: 152 SMs x 128 lanes x 2 x 2.07 GHz"}
        del xs, Bs, Cs, la, st, ys
    # block-FP8 W8A8 GEMM (activation quantisation separate), prefill FFN shape
    Mf, Nf, Kf = 8192, 11264, 2048
    Af = torch.randn((Mf, Kf), device=dev).to(torch.bfloat16)
    Wf = (0.02 * torch.randn((Nf, Kf), device=dev)).to(torch.bfloat16)
    qa = torch.empty((Mf, Kf), dtype=torch.uint8, device=dev)
    sa = torch.empty((Mf, Kf // 128), device=dev)
    qw = torch.empty((Nf, Kf), dtype=torch.uint8, device=dev)
    sw = torch.empty((Nf // 128, Kf // 128), device=dev)
    bi.bi_quantize_fp8(Wf, Nf, Kf, 128, qw, sw)
    bi.bi_quantize_fp8(Af, Mf, Kf, 1, qa, sa)
    Cf = torch.empty((Mf, Nf), dtype=torch.bfloat16, device=dev)
    us = _graph_us(lambda: bi.bi_gemm_fp8(qa, sa, Mf, Kf, qw, sw, Nf, Cf), n=3, reps=3)
    fl = 2.0 * Mf * Nf * Kf
    out["gemm_fp8_8192x11264x2048"] = {"us": round(us, 1), "TFLOP/s": round(fl / us / 1e6, 1),
                                       "frac": round(fl / us / 1e6 / (2 * tf), 3), "bound": "tensor",
                                       "peak_note": "fp8 peak = 2 x the bf16 peak (nominal ratio)"}
    us_q = _graph_us(lambda: bi.bi_quantize_fp8(Af, Mf, Kf, 1, qa, sa), n=3, reps=3)
    qbytes = Mf * Kf * 2 + Mf * Kf + Mf * (Kf // 128) * 4
    out["quantize_fp8_act_8192x2048"] = {"us": round(us_q, 1), "GB/s": round(qbytes / us_q / 1e3, 1),
                                         "frac": round(qbytes / us_q / 1e3 / hbm, 3), "bound": "hbm"}
    del Af, Wf, qa, qw, Cf
    # tensor-bound GEMMs: fused large-vocab lm_head + log-softmax, prefill FFN
    def gemm_rate(M, N, K, fn_builder, tag):
        fn, flops = fn_builder(M, N, K)
        us = _graph_us(fn, n=2, reps=3)
        out[tag] = {"us": round(us, 1), "TFLOP/s": round(flops / us / 1e6, 1), "frac": round(flops / us / 1e6 / tf, 3),
                    "bound": "tensor"}

    def fused_head(M, N, K):
        X = torch.randn((M, K), device=dev).to(torch.bfloat16)
        W = (0.01 * torch.randn((N, K), device=dev)).to(torch.bfloat16)
        I = torch.randint(0, N, (M,), dtype=torch.int32, device=dev)
        L = torch.empty(M, device=dev)
        Wk = torch.empty(bi.bi_lm_head_logprob_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
        return (lambda: bi.bi_lm_head_logprob(X, M, K, W, N, I, L, None, bi.BI_INVARIANT, Wk)), 2.0 * M * N * K

    def ffn_gate_up(M, N, K):
        X = torch.randn((M, K), device=dev).to(torch.bfloat16)
        W = (0.02 * torch.randn((N, K), device=dev)).to(torch.bfloat16)
        C = torch.empty((M, N // 2), device=dev, dtype=torch.bfloat16)
        return (lambda: bi.bi_gemm(X, M, K, W, N, C, bi.BI_DTYPE_BF16, bi.BI_EPI_SWIGLU)), 2.0 * M * N * K

    gemm_rate(16384, 129280, 4096, fused_head, "lm_head_logprob_fused_16384x129280x4096")
    gemm_rate(16384, 11264, 2048, ffn_gate_up, "gate_up_swiglu_16384x11264x2048")
    out["peak_source"] = src
    return out


def _c5_recompute(dec, shape, lens, prompts, tf_peak):
    """Training-side recompute of the long-context workload: one packed prefill
    (chunk 2048, up to 16384 rows a pass) over prompt + 127 fed-back tokens of all
    64 sequences, scoring 128 tokens each (teacher forced on seeded ids; the
    arithmetic does not depend on which ids).  Returns row() arguments."""
    import torch
    from invariant_forward_policy_gb300.decoder import recompute_pack
    from synthetic import C5
    B, n_gen = len(lens), C5["gen"]
    gens = [np.random.default_rng(C5["seed"] + 9 + b).integers(0, shape.vocab, n_gen).astype(np.int32)
            for b in range(B)]
    seqs, tg, lf = recompute_pack(prompts, gens, range(B))
    tot = [len(x) for x in seqs]
    max_ctx = max(tot)
    mb = -(-max_ctx // 64)
    bt, nb = dec.paged_block_table(tot, mb, seed=7)
    cache = dec.alloc_cache(nb)
    import invariant_forward_policy_gb300 as bi
    from invariant_forward_policy_gb300 import _lib as L
    dev = dec.device
    tok = torch.from_numpy(np.concatenate(seqs).astype(np.int32)).to(dev)
    tgt = torch.from_numpy(np.concatenate(tg).astype(np.int32)).to(dev)
    cu = np.concatenate([[0], np.cumsum(tot)]).astype(np.int64)
    lp = torch.empty(int(cu[-1]), dtype=torch.float32, device=dev)
    ws = {m: dec.workspace(16384, min(B, 128), max_ctx, 2048, m) for m in (bi.BI_INVARIANT, bi.BI_FAST)}

    def call(mode):
        L.bi_forward_prefill(dec.handle, tok, tgt, cu, [0] * B, lf, B, C5["chunk"], bt, bt.shape[1], cache.k, cache.v,
                             cache.n_blocks, lp, None, ws[mode], 16384, max_ctx, 2048, mode)

    # one call lasts about a second: eager launches, CUDA events, the two arms alternating
    ts = {"invariant": [], "non_invariant": []}
    for _ in range(3):
        for mode, tag in ((bi.BI_INVARIANT, "invariant"), (bi.BI_FAST, "non_invariant")):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            call(mode)
            e1.record()
            torch.cuda.synchronize()
            ts[tag].append(e0.elapsed_time(e1) * 1000.0)
    t = {tag: float(np.median(v[1:])) for tag, v in ts.items()}     # the first round is a warm-up
    s = shape
    per_tok = 2.0 * s.n_layers * s.d * ((s.n_heads_q + 2 * s.n_heads_kv) * s.head_dim + s.n_heads_q * s.head_dim
                                       + 3 * s.ffn)
    lin = per_tok * sum(tot) + 2.0 * s.d * s.vocab * B * n_gen
    att = 4.0 * s.head_dim * s.n_heads_q * s.n_layers * sum(n * (n + 1) / 2.0 for n in tot)
    fl = lin + att
    del cache
    torch.cuda.empty_cache()
    return (B * n_gen, "logprobs/s", t,
            {"bound": "tensor", "prefill_tokens_per_s": round(sum(tot) / (t["invariant"] * 1e-6), 1),
             "TFLOP/s": round(fl / t["invariant"] / 1e6, 1), "frac": round(fl / t["invariant"] / 1e6 / tf_peak, 3),
             "linear_TFLOP": round(lin / 1e12, 1), "attention_TFLOP": round(att / 1e12, 1),
             "peak": "bf16 sustained",
             "note": f"{sum(tot)} packed tokens (prompts 1K-32K + 127 generated), chunk 2048, eager launches"})


def config_table(args):
    """Timed unit of each other configuration of the scope table, invariant and
    non-invariant (BI_FAST, the same kernels with batch-dependent choices), with
    the roofline of its dominant work.  CUDA events around CUDA-graph replays.
      logprob head: 512 rows x 256 -> RMSNorm -> lm_head 4096 -> log-softmax + gather
        (latency-bound; inputs fit L2);
      MoE layer: 4096 tokens x 2048, 64 experts top-8, F 1024: route, permute,
        grouped gate/up + SwiGLU and down GEMMs, slot-order combine (805 MB of
        expert weights > L2);
      large-vocab logprob: 16384 x 4096 -> lm_head 129280 -> log-softmax + gather,
        fused (1.06 GB of weights > L2);
      long-context GQA decode: one decode step of the 8-layer d 2048 model over 64
        sequences with contexts 1K-32K (KV 8.6 GB > L2), replayed at fixed positions.
    Inputs of the MoE and large-vocab cases are drawn on the device with torch's
    seeded normal generator (the recipe's distributions); the others come from
    the seeded numpy generators."""
    import torch
    import invariant_forward_policy_gb300 as bi
    from invariant_forward_policy_gb300.decoder import Decoder
    from synthetic import C1, C3, C4, C5, make_c5_prompt_lengths, make_decoder_weights, make_logprob_head
    hbm, tf, tf_s, src = _peaks()
    dev = torch.device("cuda")
    out = {"peak_source": src}

    def both(build, n, reps, rounds=3):
        # the two arms alternate and each reports its median, so clock and
        # power drift over the measurement favour neither
        fns = {tag: build(mode) for mode, tag in ((bi.BI_INVARIANT, "invariant"), (bi.BI_FAST, "non_invariant"))}
        ts = {tag: [] for tag in fns}
        for _ in range(rounds):
            for tag, fn in fns.items():
                ts[tag].append(_graph_us(fn, n=n, reps=reps))
        return {tag: float(np.median(v)) for tag, v in ts.items()}

    def row(name, units, unit, t, extra):
        v_inv, v_fast = units / (t["invariant"] * 1e-6), units / (t["non_invariant"] * 1e-6)
        out[name] = {"value": round(v_inv, 1), "unit": unit, "us": round(t["invariant"], 1),
                     "non_invariant": round(v_fast, 1), "invariant_fraction": round(v_inv / v_fast, 3), **extra}

    # logprob head
    h = make_logprob_head(C1["n_seq"] * C1["seq_len"], C1["d"], C1["vocab"], C1["w_std"], C1["seed"])
    R, d, V = h["h"].shape[0], C1["d"], C1["vocab"]
    X = torch.from_numpy(h["h"].view(np.int16)).to(dev).view(torch.bfloat16)
    W = torch.from_numpy(h["w"].view(np.int16)).to(dev).view(torch.bfloat16)
    g = torch.from_numpy(h["gain"].view(np.int16)).to(dev).view(torch.bfloat16)
    ids = torch.from_numpy(h["ids"]).to(dev)
    Y = torch.empty_like(X)
    lp = torch.empty(R, device=dev)

    def head(mode):
        ws = torch.empty(bi.bi_lm_head_logprob_workspace_size(R, V, d, mode), dtype=torch.uint8, device=dev)
        return lambda: (bi.bi_rmsnorm(X, None, g, Y, R, d, 1e-6, mode),
                        bi.bi_lm_head_logprob(Y, R, d, W, V, ids, lp, None, mode, ws))
    t = both(head, 20, 10)
    row("logprob_head_512x256x4096", R, "logprobs/s", t, {"bound": "latency", "note": "2 launches, inputs in L2"})
    del X, W, Y

    # MoE layer
    gen = torch.Generator(device=dev)
    gen.manual_seed(C3["seed"])
    T, dm, E, k, F = C3["n_tokens"], C3["d"], C3["n_experts"], C3["top_k"], C3["ffn"]
    x = torch.randn((T, dm), device=dev, generator=gen).to(torch.bfloat16)
    lg = torch.randn((T, E), device=dev, generator=gen)
    w13 = (C3["w_std"] * torch.randn((E, 2 * F, dm), device=dev, generator=gen)).to(torch.bfloat16)
    w2 = (C3["w_std"] * torch.randn((E, dm, F), device=dev, generator=gen)).to(torch.bfloat16)
    y = torch.empty((T, dm), dtype=torch.bfloat16, device=dev)

    def moe(mode):
        ws = torch.empty(bi.bi_moe_layer_workspace_size(T, dm, E, k, F, mode), dtype=torch.uint8, device=dev)
        return lambda: bi.bi_moe_layer(x, lg, T, dm, E, k, F, w13, w2, y, mode, ws)
    t = both(moe, 3, 5)
    fl = 2.0 * T * k * (2 * F * dm + dm * F)
    row("moe_layer_4096x2048_e64_top8", T, "tokens/s", t,
        {"bound": "tensor", "TFLOP/s": round(fl / t["invariant"] / 1e6, 1),
         "frac": round(fl / t["invariant"] / 1e6 / tf, 3)})
    del x, lg, w13, w2, y

    # large-vocab logprob
    gen.manual_seed(C4["seed"])
    T4, d4, V4 = C4["n_tokens"], C4["d"], C4["vocab"]
    H4 = torch.randn((T4, d4), device=dev, generator=gen).to(torch.bfloat16)
    W4 = (C4["w_std"] * torch.randn((V4, d4), device=dev, generator=gen)).to(torch.bfloat16)
    I4 = torch.randint(0, V4, (T4,), dtype=torch.int32, device=dev, generator=gen)
    L4 = torch.empty(T4, device=dev)

    def big(mode):
        ws = torch.empty(bi.bi_lm_head_logprob_workspace_size(T4, V4, d4, mode), dtype=torch.uint8, device=dev)
        return lambda: bi.bi_lm_head_logprob(H4, T4, d4, W4, V4, I4, L4, None, mode, ws)
    t = both(big, 2, 3)
    fl = 2.0 * T4 * V4 * d4
    row("large_vocab_logprob_16384x4096x129280", T4, "logprobs/s", t,
        {"bound": "tensor", "TFLOP/s": round(fl / t["invariant"] / 1e6, 1),
         "frac": round(fl / t["invariant"] / 1e6 / tf, 3)})
    del H4, W4, I4, L4
    torch.cuda.empty_cache()

    # long-context GQA decode step, bf16 model, then the block-FP8 model (W8A8 linear
    # layers, FP8 KV cache: half the weight and KV bytes)
    shape = C5["shape"]
    lens = make_c5_prompt_lengths(C5["batch"], C5["ctx_min"], C5["ctx_max"], C5["seed"])
    B = len(lens)
    wb = make_decoder_weights(shape, seed=C5["seed"], w_std=C5["w_std"])
    max_ctx = int(lens.max()) + 1
    rng = np.random.default_rng(C5["seed"] + 3)
    prompts = [rng.integers(0, shape.vocab, int(n)).astype(np.int32) for n in lens]
    for fp8 in (False, True):
        # positions up to the longest prompt + the generated tokens (the recompute leg needs them)
        dec = Decoder(shape, wb, max_pos=int(lens.max()) + C5["gen"] + 64, fp8=fp8)
        mb = -(-max_ctx // 64)
        bt, nb = dec.paged_block_table([int(n) + 1 for n in lens], mb, seed=5)
        cache = dec.alloc_cache(nb)
        _, sm, cu = dec.prefill(prompts, cache, bt, logit_from=[int(n) - 1 for n in lens], chunk=C5["chunk"],
                                max_tokens=16384, max_ctx=max_ctx, max_logit_rows=B)
        tok = sm[torch.from_numpy(cu[1:] - 1).to(dev)].contiguous()
        pos = torch.from_numpy(lens.astype(np.int32)).to(dev)
        smp = torch.empty(B, dtype=torch.int32, device=dev)
        lpd = torch.empty(B, device=dev)

        def step(mode):
            ws = dec.workspace(B, B, max_ctx, B, mode)
            return lambda: dec.decode(tok, pos, cache, bt, max_ctx, smp, lpd, ws, mode)
        t = both(step, 3, 5)
        per_kv = 2 * (shape.head_dim + 4) if fp8 else 2 * shape.head_dim * 2   # K and V bytes per token and kv head
        kv = float(sum(int(n) + 1 for n in lens)) * shape.n_layers * shape.n_heads_kv * per_kv
        if fp8:
            wbytes = sum(lw[k + "8"].numel() + lw[k + "_s"].numel() * 4 for lw in dec.layers
                         for k in ("wqkv", "wo", "w13", "w2"))
            wbytes += sum(lw[k].numel() * 2 for lw in dec.layers for k in ("attn_norm", "ffn_norm"))
            wbytes += wb["lm_head"].nbytes + wb["final_norm"].nbytes
        else:
            wbytes = sum(a.nbytes for lw in wb["layers"] for a in lw.values()) + wb["lm_head"].nbytes + \
                wb["final_norm"].nbytes
        name = "long_context_gqa_decode_step_64seq" + ("_fp8" if fp8 else "")
        row(name, B, "logprobs/s", t,
            {"bound": "hbm", "GB/s": round((kv + wbytes) / t["invariant"] / 1e3, 1),
             "frac": round((kv + wbytes) / t["invariant"] / 1e3 / hbm, 3),
             "bytes_per_step": int(kv + wbytes),
             "note": ("FP8 codes + scales of the KV cache and of the linear weights (bf16 lm_head) read once per "
                      "step; bound in practice by the in-shared-memory expansion of the FP8 pages" if fp8 else
                      "KV of every context + all layer and lm_head weights read once per step (embedding rows "
                      "excluded)")})
        if not fp8:
            row("long_context_gqa_recompute_64seq", *_c5_recompute(dec, shape, lens, prompts, tf_s))
        dec.close()
        del cache
        torch.cuda.empty_cache()

    # block-FP8 dense decoder: the default workload's whole episode (prefill, 255
    # graph-replayed decode steps, recompute) with W8A8 linear layers and the FP8
    # KV cache; the bf16 model's episode is timed alongside for the ratio
    from invariant_forward_policy_gb300.decoder import Episode
    from synthetic import C2, make_prompts
    shape2 = C2["shape"]
    wb2 = make_decoder_weights(shape2, seed=C2["seed"], w_std=C2["w_std"])
    prompts2 = make_prompts(C2["batch"], C2["prompt_min"], C2["prompt_max"], shape2.vocab, C2["seed"])
    lens2 = [len(p) for p in prompts2]
    pd2 = torch.from_numpy(np.concatenate(prompts2).astype(np.int32)).to(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    dec8 = Decoder(shape2, wb2, max_pos=1024, fp8=True)
    dec16 = Decoder(shape2, wb2, max_pos=1024)
    eps = {"invariant": Episode(dec8, lens2, C2["gen"], mode=bi.BI_INVARIANT),
           "non_invariant": Episode(dec8, lens2, C2["gen"], mode=bi.BI_FAST),
           "bf16_model": Episode(dec16, lens2, C2["gen"], mode=bi.BI_INVARIANT)}
    for e in eps.values():
        for _ in range(2):
            e.run(pd2)
    ts = {tag: [] for tag in eps}
    diff0 = True
    for _ in range(3):
        for tag, e in eps.items():
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            _, lr, lt = e.run(pd2)
            e1.record()
            torch.cuda.synchronize()
            ts[tag].append(e0.elapsed_time(e1) * 1000.0)
            if tag == "invariant":
                diff0 = diff0 and bool(torch.equal(lr.view(torch.int32), lt.view(torch.int32)))
    t = {tag: float(np.median(v)) for tag, v in ts.items()}
    toks = C2["batch"] * C2["gen"]
    row("fp8_dense_decoder_episode_16x256", toks, "tokens/s", t,
        {"bound": "latency", "bf16_model_tokens_per_s": round(toks / (t["bf16_model"] * 1e-6), 1),
         "fp8_over_bf16": round(t["bf16_model"] / t["invariant"], 3), "rollout_equals_recompute": diff0,
         "note": "W8A8 block-FP8 linear layers + FP8 KV cache (codes + per-(token, head) scales); L2 flushed"})
    del eps, dec8, dec16, flush
    torch.cuda.empty_cache()
    return out


def run_kernel_case(name: str, reps: int):
    """Launch one kernel of the step at its step shape `reps` times (profiling aid)."""
    import torch
    import invariant_forward_policy_gb300 as bi
    torch.manual_seed(0)
    dev = torch.device("cuda")
    if name in ("gemm_decode_qkv", "gemm_decode_down", "gemm_decode_lm_head", "gemm_prefill"):
        M, N, K, dt = {"gemm_decode_qkv": (16, 1536, 512, bi.BI_DTYPE_BF16),
                       "gemm_decode_down": (16, 512, 1408, bi.BI_DTYPE_BF16),
                       "gemm_decode_lm_head": (16, 32000, 512, bi.BI_DTYPE_FP32),
                       "gemm_prefill": (8192, 5632 * 2, 2048, bi.BI_DTYPE_BF16)}[name]
        A = (0.5 * torch.randn((M, K), device=dev)).to(torch.bfloat16)
        W = (0.02 * torch.randn((N, K), device=dev)).to(torch.bfloat16)
        C = torch.empty((M, N), device=dev, dtype=torch.float32 if dt == bi.BI_DTYPE_FP32 else torch.bfloat16)
        for _ in range(reps):
            bi.bi_gemm(A, M, K, W, N, C, dt)
    elif name == "attention_decode":
        B, Hq, Hkv, hd, ctx = 16, 8, 8, 64, 700
        max_blk = -(-ctx // 64)
        kc = (0.5 * torch.randn((B * max_blk, Hkv, 64, hd), device=dev)).to(torch.bfloat16)
        vc = (0.5 * torch.randn((B * max_blk, Hkv, 64, hd), device=dev)).to(torch.bfloat16)
        bt = torch.arange(B * max_blk, dtype=torch.int32, device=dev).view(B, max_blk)
        q = (0.5 * torch.randn((B, Hq, hd), device=dev)).to(torch.bfloat16)
        seq = torch.arange(B, dtype=torch.int32, device=dev)
        row0 = torch.arange(B + 1, dtype=torch.int32, device=dev)
        pos0 = torch.full((B,), ctx - 1, dtype=torch.int32, device=dev)
        out = torch.empty((B, Hq * hd), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(bi.bi_attention_workspace_size(B, Hq, hd, ctx, 512), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            bi.bi_attention(q, B, seq, row0, pos0, B, 1, Hq, Hkv, hd, kc, vc, bt, max_blk, B * max_blk, ctx, 512, 0.125,
                            ws, out)
    elif name in ("step", "fp8_step"):
        # the timed unit of the default run: rollout + recompute of the dense-decoder workload
        # (fp8_step: the same episode with W8A8 block-FP8 layers and the FP8 KV cache)
        from invariant_forward_policy_gb300.decoder import Decoder, Episode
        from synthetic import C2, make_decoder_weights, make_prompts
        shape = C2["shape"]
        wb = make_decoder_weights(shape, seed=C2["seed"], w_std=C2["w_std"])
        prompts = make_prompts(C2["batch"], C2["prompt_min"], C2["prompt_max"], shape.vocab, C2["seed"])
        dec = Decoder(shape, wb, max_pos=1024, device=dev, fp8=name == "fp8_step")
        ep = Episode(dec, [len(p) for p in prompts], C2["gen"], mode=bi.BI_INVARIANT)
        pd = torch.from_numpy(np.concatenate(prompts).astype(np.int32)).to(dev)
        for _ in range(reps):
            ep.run(pd)
    elif name in ("c5_decode", "c5_decode_fp8"):
        # long-context GQA decode steps (8 layers, d 2048, 64 sequences, contexts 1K-32K) after an
        # untimed prefill; the decode launches sit in the NVTX range "decode" (c5_decode_fp8: W8A8
        # block-FP8 layers and the FP8 KV cache)
        from invariant_forward_policy_gb300.decoder import Decoder
        from synthetic import C5, make_c5_prompt_lengths, make_decoder_weights
        shape = C5["shape"]
        lens = make_c5_prompt_lengths(C5["batch"], C5["ctx_min"], C5["ctx_max"], C5["seed"])
        B = len(lens)
        wb = make_decoder_weights(shape, seed=C5["seed"], w_std=C5["w_std"])
        max_ctx = int(lens.max()) + 1
        rng = np.random.default_rng(C5["seed"] + 3)
        prompts = [rng.integers(0, shape.vocab, int(n)).astype(np.int32) for n in lens]
        dec = Decoder(shape, wb, max_pos=max_ctx + 64, device=dev, fp8=name == "c5_decode_fp8")
        mb = -(-max_ctx // 64)
        bt, nb = dec.paged_block_table([int(n) + 1 for n in lens], mb, seed=5)
        cache = dec.alloc_cache(nb)
        _, sm, cu = dec.prefill(prompts, cache, bt, logit_from=[int(n) - 1 for n in lens], chunk=C5["chunk"],
                                max_tokens=16384, max_ctx=max_ctx, max_logit_rows=B)
        tok = sm[torch.from_numpy(cu[1:] - 1).to(dev)].contiguous()
        pos = torch.from_numpy(lens.astype(np.int32)).to(dev)
        smp = torch.empty(B, dtype=torch.int32, device=dev)
        lpd = torch.empty(B, device=dev)
        ws = dec.workspace(B, B, max_ctx, B)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("decode")
        for _ in range(reps):
            dec.decode(tok, pos, cache, bt, max_ctx, smp, lpd, ws)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    elif name == "c5_recompute":
        # training-side recompute of the long-context workload: one packed chunk-2048 prefill over
        # prompt + 127 fed-back tokens of all 64 sequences (the bench's recompute row)
        from invariant_forward_policy_gb300 import _lib as L
        from invariant_forward_policy_gb300.decoder import Decoder, recompute_pack
        from synthetic import C5, make_c5_prompt_lengths, make_decoder_weights
        shape = C5["shape"]
        lens = make_c5_prompt_lengths(C5["batch"], C5["ctx_min"], C5["ctx_max"], C5["seed"])
        B, n_gen = len(lens), C5["gen"]
        wb = make_decoder_weights(shape, seed=C5["seed"], w_std=C5["w_std"])
        rng = np.random.default_rng(C5["seed"] + 3)
        prompts = [rng.integers(0, shape.vocab, int(n)).astype(np.int32) for n in lens]
        gens = [np.random.default_rng(C5["seed"] + 9 + b).integers(0, shape.vocab, n_gen).astype(np.int32)
                for b in range(B)]
        seqs, tg, lf = recompute_pack(prompts, gens, range(B))
        tot = [len(x) for x in seqs]
        max_ctx = max(tot)
        dec = Decoder(shape, wb, max_pos=max_ctx + 64, device=dev)
        bt, nb = dec.paged_block_table(tot, -(-max_ctx // 64), seed=7)
        cache = dec.alloc_cache(nb)
        tok = torch.from_numpy(np.concatenate(seqs).astype(np.int32)).to(dev)
        tgt = torch.from_numpy(np.concatenate(tg).astype(np.int32)).to(dev)
        cu = np.concatenate([[0], np.cumsum(tot)]).astype(np.int64)
        lp = torch.empty(int(cu[-1]), dtype=torch.float32, device=dev)
        ws = dec.workspace(16384, min(B, 128), max_ctx, 2048, bi.BI_INVARIANT)
        for _ in range(reps):
            L.bi_forward_prefill(dec.handle, tok, tgt, cu, [0] * B, lf, B, C5["chunk"], bt, bt.shape[1], cache.k,
                                 cache.v, cache.n_blocks, lp, None, ws, 16384, max_ctx, 2048, bi.BI_INVARIANT)
    elif name == "gemm_fp8":
        # block-FP8 W8A8 GEMM at a prefill FFN shape (operands quantised once, untimed)
        M, N, K = 8192, 11264, 2048
        A = torch.randn((M, K), device=dev).to(torch.bfloat16)
        W = (0.02 * torch.randn((N, K), device=dev)).to(torch.bfloat16)
        qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
        sa = torch.empty((M, K // 128), device=dev)
        qw = torch.empty((N, K), dtype=torch.uint8, device=dev)
        sw = torch.empty((N // 128, K // 128), device=dev)
        bi.bi_quantize_fp8(A, M, K, 1, qa, sa)
        bi.bi_quantize_fp8(W, N, K, 128, qw, sw)
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        for _ in range(reps):
            bi.bi_gemm_fp8(qa, sa, M, K, qw, sw, N, C)
    elif name == "topk_decode":
        # deterministic Top-K, K = 2048, one decode step of 64 rows with contexts 1K-32K
        from synthetic import C5, make_c5_prompt_lengths
        nv = make_c5_prompt_lengths(C5["batch"], C5["ctx_min"], C5["ctx_max"], C5["seed"]).astype(np.int32)
        T, ld = len(nv), int(nv.max())
        S = torch.randn((T, ld), device=dev)
        idx = torch.empty((T, 2048), dtype=torch.int32, device=dev)
        nvd = torch.from_numpy(nv).to(dev)
        for _ in range(reps):
            bi.bi_topk(S, T, ld, nvd, 2048, idx)
    elif name == "topk_prefill":
        # deterministic Top-K, K = 2048, a 2048-row prefill chunk at positions 30K-32K (one CTA per row)
        nv = np.arange(30721, 32769, dtype=np.int32)
        T, ld = len(nv), int(nv.max())
        S = torch.randn((T, ld), device=dev)
        idx = torch.empty((T, 2048), dtype=torch.int32, device=dev)
        nvd = torch.from_numpy(nv).to(dev)
        for _ in range(reps):
            bi.bi_topk(S, T, ld, nvd, 2048, idx)
    elif name == "ssd_prefill":
        # Mamba-2 chunked scan: 16 sequences x 2048, 32 heads x 64, state 128, 8 groups, chunk 64
        n_seq, per, Hs, Gs, Ps, Ns, Qs = 16, 2048, 32, 8, 64, 128, 64
        T = n_seq * per
        xs = torch.randn((T, Hs, Ps), device=dev).to(torch.bfloat16)
        Bs = (torch.randn((T, Gs, Ns), device=dev) * Ns ** -0.5).to(torch.bfloat16)
        Cs = (torch.randn((T, Gs, Ns), device=dev) * Ns ** -0.5).to(torch.bfloat16)
        la = -torch.rand((T, Hs), device=dev) * 0.2
        st = torch.zeros((n_seq, bi.bi_ssd_state_bytes(Hs, Gs, Ps, Ns, Qs) // 4), device=dev)
        ys = torch.empty((T, Hs, Ps), device=dev)
        sq = torch.arange(n_seq, dtype=torch.int32, device=dev)
        r0 = torch.arange(0, T + 1, per, dtype=torch.int32, device=dev)
        p0 = torch.zeros(n_seq, dtype=torch.int32, device=dev)
        for _ in range(reps):
            st.zero_()
            bi.bi_ssd_chunk_scan(xs, Bs, Cs, la, sq, r0, p0, n_seq, per, Hs, Gs, Ps, Ns, Qs, st, n_seq, ys)
    elif name == "kv_fp8_gather":
        # FP8 KV read path: 16 sequences x 8192 context, 4 kv heads x 128 (0.27 GB of codes)
        B, Hkv, hd, ctx = 16, 4, 128, 8192
        mb = ctx // 64
        k8 = torch.randint(0, 0x7E, (B * mb, Hkv, 64, hd), dtype=torch.uint8, device=dev)
        v8 = torch.randint(0, 0x7E, (B * mb, Hkv, 64, hd), dtype=torch.uint8, device=dev)
        ks = torch.full((B * mb, Hkv, 64), 2.0 ** -8, device=dev)
        vs = torch.full_like(ks, 2.0 ** -8)
        bt = torch.arange(B * mb, dtype=torch.int32, device=dev).view(B, mb)
        kw = torch.empty((B * mb, Hkv, 64, hd), dtype=torch.bfloat16, device=dev)
        vw = torch.empty_like(kw)
        wbt = torch.empty((B, mb), dtype=torch.int32, device=dev)
        seq = torch.arange(B, dtype=torch.int32, device=dev)
        row0 = torch.arange(B + 1, dtype=torch.int32, device=dev)
        pos0 = torch.full((B,), ctx - 1, dtype=torch.int32, device=dev)
        for _ in range(reps):
            bi.bi_kv_fp8_gather(k8, v8, ks, vs, B * mb, seq, row0, pos0, B, Hkv, hd, bt, mb, kw, vw, wbt)
    elif name == "attention_decode_long_fp8":
        # persistent decode schedule over an FP8 cache: 32 sequences x 4096 context, 16/4 heads x 128
        # (134 MB of codes + 2 MB of scales > L2)
        B, Hq, Hkv, hd, ctx = 32, 16, 4, 128, 4096
        max_blk = ctx // 64
        k8 = torch.randint(0, 0x7E, (B * max_blk, Hkv, 64, hd), dtype=torch.uint8, device=dev)
        v8 = torch.randint(0, 0x7E, (B * max_blk, Hkv, 64, hd), dtype=torch.uint8, device=dev)
        ks = torch.full((B * max_blk, Hkv, 64), 2.0 ** -8, device=dev)
        vs = torch.full_like(ks, 2.0 ** -8)
        bt = torch.arange(B * max_blk, dtype=torch.int32, device=dev).view(B, max_blk)
        q = (0.5 * torch.randn((B, Hq, hd), device=dev)).to(torch.bfloat16)
        seq = torch.arange(B, dtype=torch.int32, device=dev)
        row0 = torch.arange(B + 1, dtype=torch.int32, device=dev)
        pos0 = torch.full((B,), ctx - 1, dtype=torch.int32, device=dev)
        out = torch.empty((B, Hq * hd), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(bi.bi_attention_workspace_size(B, Hq, hd, ctx, 512), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            bi.bi_attention_fp8(q, B, seq, row0, pos0, B, 1, Hq, Hkv, hd, k8, v8, ks, vs, bt, max_blk, B * max_blk,
                                ctx, 512, hd ** -0.5, ws, out)
    elif name == "attention_decode_long":
        # persistent decode schedule: 32 sequences x 4096 context, 16/4 heads x 128 (268 MB of KV > L2)
        B, Hq, Hkv, hd, ctx = 32, 16, 4, 128, 4096
        max_blk = ctx // 64
        kc = (0.5 * torch.randn((B * max_blk, Hkv, 64, hd), device=dev)).to(torch.bfloat16)
        vc = (0.5 * torch.randn((B * max_blk, Hkv, 64, hd), device=dev)).to(torch.bfloat16)
        bt = torch.arange(B * max_blk, dtype=torch.int32, device=dev).view(B, max_blk)
        q = (0.5 * torch.randn((B, Hq, hd), device=dev)).to(torch.bfloat16)
        seq = torch.arange(B, dtype=torch.int32, device=dev)
        row0 = torch.arange(B + 1, dtype=torch.int32, device=dev)
        pos0 = torch.full((B,), ctx - 1, dtype=torch.int32, device=dev)
        out = torch.empty((B, Hq * hd), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(bi.bi_attention_workspace_size(B, Hq, hd, ctx, 512), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            bi.bi_attention(q, B, seq, row0, pos0, B, 1, Hq, Hkv, hd, kc, vc, bt, max_blk, B * max_blk, ctx, 512,
                            hd ** -0.5, ws, out)
    elif name == "attention_prefill_long":
        # row-parallel prefill schedule: one 2048-row chunk at positions 30720..32767 of a
        # 32768-token sequence, 16/4 heads x 128 (64 splits of 512, then the split merge)
        Hq, Hkv, hd, ctx, ch = 16, 4, 128, 32768, 2048
        max_blk = ctx // 64
        kc = (0.5 * torch.randn((max_blk, Hkv, 64, hd), device=dev)).to(torch.bfloat16)
        vc = (0.5 * torch.randn((max_blk, Hkv, 64, hd), device=dev)).to(torch.bfloat16)
        bt = torch.arange(max_blk, dtype=torch.int32, device=dev).view(1, max_blk)
        q = (0.5 * torch.randn((ch, Hq, hd), device=dev)).to(torch.bfloat16)
        seq = torch.zeros(1, dtype=torch.int32, device=dev)
        row0 = torch.tensor([0, ch], dtype=torch.int32, device=dev)
        pos0 = torch.tensor([ctx - ch], dtype=torch.int32, device=dev)
        out = torch.empty((ch, Hq * hd), dtype=torch.bfloat16, device=dev)
        # the invariant call's partials only (the size query also covers BI_FAST's smaller splits)
        ws = torch.empty(ch * Hq * (ctx // 512) * (hd + 2) * 4 + 256, dtype=torch.uint8, device=dev)
        for _ in range(reps):
            bi.bi_attention(q, ch, seq, row0, pos0, 1, ch, Hq, Hkv, hd, kc, vc, bt, max_blk, max_blk, ctx, 512,
                            hd ** -0.5, ws, out)
    elif name == "rmsnorm":
        # residual add + norm, 16384 rows x 2048 (4 x 67 MB: above L2)
        R, d = 16384, 2048
        x = torch.randn((R, d), device=dev).to(torch.bfloat16)
        r = torch.randn((R, d), device=dev).to(torch.bfloat16)
        y = torch.empty_like(x)
        g = torch.ones(d, device=dev).to(torch.bfloat16)
        for _ in range(reps):
            bi.bi_rmsnorm(x, r, g, y, R, d)
    elif name == "logprob":
        # vocab-wide log-softmax + gather, 2048 rows x 129280 (1.06 GB of fp32 logits)
        T, V = 2048, 129280
        logits = torch.randn((T, V), device=dev)
        lp = torch.empty(T, device=dev)
        ids = torch.randint(0, V, (T,), dtype=torch.int32, device=dev)
        for _ in range(reps):
            bi.bi_logprob_gather(logits, ids, T, V, lp)
    elif name == "lm_head_fused_decode":
        # the dense decoder's decode-step head: 16 rows x 512 -> 32000, fused log-softmax records + merge
        T, d, V = 16, 512, 32000
        H = torch.randn((T, d), device=dev).to(torch.bfloat16)
        W = (0.02 * torch.randn((V, d), device=dev)).to(torch.bfloat16)
        lp = torch.empty(T, device=dev)
        am = torch.empty(T, dtype=torch.int32, device=dev)
        ws = torch.empty(bi.bi_lm_head_logprob_workspace_size(T, V, d, bi.BI_INVARIANT), dtype=torch.uint8,
                         device=dev)
        for _ in range(reps):
            bi.bi_lm_head_logprob(H, T, d, W, V, None, lp, am, bi.BI_INVARIANT, ws)
    elif name == "lm_head_fused":
        # fused lm_head + log-softmax records + merge, 2048 rows x 4096 -> 129280
        T, d, V = 2048, 4096, 129280
        H = torch.randn((T, d), device=dev).to(torch.bfloat16)
        W = (0.01 * torch.randn((V, d), device=dev)).to(torch.bfloat16)
        ids = torch.randint(0, V, (T,), dtype=torch.int32, device=dev)
        lp = torch.empty(T, device=dev)
        ws = torch.empty(bi.bi_lm_head_logprob_workspace_size(T, V, d, bi.BI_INVARIANT), dtype=torch.uint8,
                         device=dev)
        for _ in range(reps):
            bi.bi_lm_head_logprob(H, T, d, W, V, ids, lp, None, bi.BI_INVARIANT, ws)
    elif name == "moe_layer":
        # MoE layer: router top-8, permutation, grouped expert GEMMs, slot-order combine (4096 x 2048, 64 experts)
        T, dm, E, k, F = 4096, 2048, 64, 8, 1024
        x = torch.randn((T, dm), device=dev).to(torch.bfloat16)
        lg = torch.randn((T, E), device=dev)
        w13 = (0.02 * torch.randn((E, 2 * F, dm), device=dev)).to(torch.bfloat16)
        w2 = (0.02 * torch.randn((E, dm, F), device=dev)).to(torch.bfloat16)
        y = torch.empty((T, dm), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(bi.bi_moe_layer_workspace_size(T, dm, E, k, F, bi.BI_INVARIANT), dtype=torch.uint8,
                         device=dev)
        for _ in range(reps):
            bi.bi_moe_layer(x, lg, T, dm, E, k, F, w13, w2, y, bi.BI_INVARIANT, ws)
    else:
        raise SystemExit(f"unknown kernel case {name}")
    torch.cuda.synchronize()
    assert bi.bi_device_status() == 0
    print(json.dumps({"kernel_case": name, "reps": reps, "ok": True}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel-case", default=None,
                    help="run one kernel at its step shape (gemm_decode_qkv, gemm_decode_down, gemm_decode_lm_head, "
                         "lm_head_fused_decode, gemm_prefill, "
                         "attention_decode, attention_decode_long, attention_decode_long_fp8, gemm_fp8, topk_decode, ssd_prefill, "
                         "kv_fp8_gather, c5_decode, c5_decode_fp8, c5_recompute, topk_prefill, attention_prefill_long, rmsnorm, "
                         "logprob, lm_head_fused, "
                         "moe_layer) or "
                         "the whole step (step, or fp8_step with the block-FP8 model) and exit; for profiling")
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-kernels", action="store_true", help="skip the per-kernel rate table")
    ap.add_argument("--no-configs", action="store_true", help="skip the other configurations' timed units")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--clocks-csv", default=None,
                    help="keep the nvidia-smi samples of the timed region in this file (default: a temporary file)")
    ap.add_argument("--oracle-rates", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--one-thread", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_rates:
        # child of the CPU-baseline leg: the oracle on each workload's sample, in this interpreter's threads
        rates = oracle_config_rates(small=args.one_thread)
        print(json.dumps({"cores": 1 if args.one_thread else _cpu_cores(), "rates": rates}), flush=True)
        return
    if args.kernel_case:
        run_kernel_case(args.kernel_case, args.reps)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
