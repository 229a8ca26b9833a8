#!/usr/bin/env python
"""SwiftKV prefill benchmark on GB300.

One step = one swiftkv_prefill of a packed batch of prompts: layers 1..l for every
prompt token, the boundary RMSNorm + wide KV GEMM into every skipped cache, the
last-token tail through layers l+1..L, and the LM head. Default workload:
Llama-3.1-8B shape (bf16, random-init N(0, 0.02)), l = 16, no AcrossKV, 16 prompts
with lengths U[500, 1000], token ids U[0, V), 16-token pages.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0). Multi-GPU runs (torchrun) are independent replicas:
every rank prefills its own prompts (weak scaling); the only collectives are the
timing barrier and the max-over-ranks of the elapsed time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "prefill tokens/s and dense-equiv TFLOP/s (% of bf16 peak), 1×GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], 0.0, set()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = max(mx, float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(self.REASONS, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- workload

def workload_batch(w, rank: int, reserve_tokens: int = 0):
    """Each replica prefills its own prompts (weak scaling): the input seed depends on the rank."""
    if w.mixed:
        return synth.mixed_batch(w.shape.vocab, w.mix_chunks, w.mix_decode, w.mix_decode_ctx[0],
                                 w.mix_decode_ctx[1], w.page_size, seed=synth.SEED_INPUTS + 1000 * rank)
    return synth.prompt_batch(w.shape.vocab, w.num_prompts, w.len_lo, w.len_hi, w.page_size,
                              reserve_tokens=reserve_tokens, seed=synth.SEED_INPUTS + 1000 * rank)


def replica_barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value over all ranks (the timing rule: the slowest replica sets the time)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def whole_job_throughput(units_all_ranks: float, steps: int, seconds: float) -> float:
    """Units all ranks processed (per step, summed over ranks) divided by the max-over-ranks
    elapsed time."""
    return units_all_ranks * steps / seconds


def gen_weights(w, keep_raw: bool):
    """Seeded synthetic weights, layer by layer (input generation, not timed)."""
    raw = {}
    for j in range(w.shape.L):
        rep = j < w.l or (j - w.l) % w.g == 0
        kinds = None if rep else ("wq", "wo", "wg", "wu", "wd", "gamma_attn", "gamma_mlp", "bq")
        lw = synth.layer_weights(w.shape, j, kinds=kinds)
        yield ("layer", j, lw)
        if keep_raw:
            raw[j] = lw
    g = synth.global_weights(w.shape)
    yield ("globals", None, g)


def oracle_weights(w, raw_layers, raw_globals):
    """Oracle view of already generated weights (float32 copies of the bf16 values)."""
    import oracle
    f32 = synth.bf16_bits_to_f32
    cache = {}

    def layer_fn(j):
        if j not in cache:
            r = raw_layers[j] if raw_layers is not None and j in raw_layers else \
                synth.layer_weights(w.shape, j)
            cache[j] = oracle.Layer(gamma_attn=r["gamma_attn"], wq=f32(r["wq"]),
                                    wk=f32(r["wk"]) if "wk" in r else None,
                                    wv=f32(r["wv"]) if "wv" in r else None, wo=f32(r["wo"]),
                                    gamma_mlp=r["gamma_mlp"], wg=f32(r["wg"]), wu=f32(r["wu"]),
                                    wd=f32(r["wd"]), bq=r.get("bq"), bk=r.get("bk"), bv=r.get("bv"))
        return cache[j]

    g = raw_globals if raw_globals is not None else synth.global_weights(w.shape, kinds=("gamma_final", "lm_head"))
    emb = g.get("embed")

    def embed_fn(tokens):
        if emb is not None:
            return f32(emb[np.asarray(tokens)])
        return f32(synth.embed_rows(w.shape, tokens))

    return oracle.Weights(layer_fn, embed_fn, g["gamma_final"], f32(g["lm_head"]))


def oracle_sample_time(w, weights, tokens):
    """Times the oracle's prefill-skipping path on one prompt (seconds)."""
    import oracle
    from oracle import model as OM
    cfg = oracle.config_of(w.shape)
    t0 = time.perf_counter()
    OM.swiftkv_prefill_one(cfg, weights, tokens, w.l, w.g)
    return time.perf_counter() - t0


L2_BYTES = 129e6  # GB300 L2
PROFILED_PASS_NOTE = ("per-launch CUDA events on the launch stream over a second pass of the same K steps, "
                      "right after the uninstrumented timed region that gives `value`")


def l2_note(shape) -> str:
    """Whether a step's inputs exceed L2 (the timing rule needs that or an L2 flush): the bf16
    weights, all of which a step reads once."""
    s = shape
    per_layer = s.d * (s.n_q + 2 * s.n_kv) * s.d_h + s.n_q * s.d_h * s.d + 3 * s.d * s.ffn
    weight_bytes = 2 * (s.L * per_layer + 2 * s.vocab * s.d)
    if weight_bytes > L2_BYTES:
        return f"inputs larger than L2 (~{weight_bytes / 1e9:.1f} GB of bf16 weights read from HBM every step)"
    return f"weights {weight_bytes / 1e6:.1f} MB fit in L2: a parity configuration, not a timing one"


def workload_config(w, batch, norm_fusion=0):
    if w.mixed:
        chunks = ", ".join(f"{n}@{c}" for c, n in w.mix_chunks)
        return {
            "workload": f"{w.name}: {w.shape.name} shape bf16 random-init N(0,0.02), SwiftKV l={w.l}, "
                        f"AcrossKV g={w.g}, one serving step: prompt chunks (tokens@cached) {chunks} + "
                        f"{w.mix_decode} decode tokens with cached context U[{w.mix_decode_ctx[0]},"
                        f"{w.mix_decode_ctx[1]}], 16-token pages",
            "chunks": len(w.mix_chunks), "decode_tokens": int(w.mix_decode),
            "tokens_per_step": int(batch.cu_seqlens[-1]), "cached_tokens": int(batch.extra["ctx"].sum()),
            "l": w.l, "g": w.g, "L": w.shape.L, "kv_cache": w.kv_dtype,
            "l2": l2_note(w.shape),
            "parallelism": "replicas (one independent serving step per GPU)",
            "norm_fusion": norm_fusion,
        }
    return {
        "workload": f"{w.name}: {w.shape.name} shape bf16 random-init N(0,0.02), SwiftKV l={w.l}, "
                    f"AcrossKV g={w.g}, {w.num_prompts} prompts U[{w.len_lo},{w.len_hi}] packed varlen, "
                    f"16-token pages",
        "prompts": int(w.num_prompts), "tokens_per_step": int(batch.cu_seqlens[-1]),
        "l": w.l, "g": w.g, "L": w.shape.L, "kv_cache": w.kv_dtype,
        "l2": l2_note(w.shape),
        "parallelism": "replicas (one independent prefill per GPU)",
        "norm_fusion": norm_fusion,
    }


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, w, rank, world):
    if rank != 0:
        return 0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    batch = workload_batch(w, 0)
    sample_len = args.ref_sample_tokens
    log(f"[reference] generating weights for {w.name} ...")
    t0 = time.time()
    weights = oracle_weights(w, None, None)
    log(f"[reference] oracle weights ready (lazy) in {time.time() - t0:.1f}s")

    def sample(step):
        s = step % len(batch.lens)
        a = int(batch.cu_seqlens[s])
        return batch.tokens[a:a + min(sample_len, int(batch.lens[s]))]

    for i in range(args.warmup):
        oracle_sample_time(w, weights, sample(i))
    tot_tok, tot_s = 0, 0.0
    for k in range(args.steps):
        toks = sample(args.warmup + k)
        tot_s += oracle_sample_time(w, weights, toks)
        tot_tok += len(toks)
    value = tot_tok / tot_s
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; no dataset)", "config": workload_config(w, batch),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: first {sample_len} tokens of one prompt of the workload, "
                                   f"full SwiftKV prefill path (layers 1..l, wide KV, last-token tail, "
                                   f"LM head) in float64 NumPy"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm

def run_ours(args, w, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from swiftkv_prefill_skipping_gb300 import api, binding
    from swiftkv_prefill_skipping_gb300 import flops as FL

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks, peak_src = load_peaks()
    n_dec_req = 0 if w.mixed else (args.decode_steps if args.decode_steps is not None else w.decode_steps)
    # decode steps: one warm-up, the timed ones, and up to five profiled ones
    batch = workload_batch(w, rank, reserve_tokens=n_dec_req + 6 if n_dec_req > 0 else 0)
    T, P = int(batch.cu_seqlens[-1]), int(len(batch.lens))
    want_cpu = (rank == 0 and world == 1 and not args.no_cpu_baseline)

    t0 = time.time()
    model = api.Model(w.shape, w.l, w.g)
    raw_layers, raw_globals = ({}, None) if want_cpu else (None, None)
    for kind, j, wts in gen_weights(w, keep_raw=False):
        if kind == "layer":
            model.load_layer(j, wts)
            if want_cpu:
                raw_layers[j] = wts
        else:
            model.load_globals(wts)
            if want_cpu:
                raw_globals = wts
    binding.check(binding.lib().swiftkv_set_norm_fusion(model.handle, args.norm_fusion))
    log(f"[ours] rank {rank}: weights generated + loaded in {time.time() - t0:.1f}s "
        f"({model.memory()[0] / 2**30:.1f} GiB on device)")
    kv = api.KVCache(model, batch.num_pages, batch.block_table, device=dev, dtype=w.kv_dtype)
    tokens = torch.as_tensor(batch.tokens, device=dev)
    logits = torch.empty((P, w.shape.vocab), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    ctx_lens = None
    if w.mixed:
        # the cached prefixes of the step's sequences, filled once before timing; every
        # timed step then rewrites the same cache rows with the same values
        ctx_lens = [int(c) for c in batch.extra["ctx"]]
        t0 = time.time()
        fill_prefixes(model, kv, batch, stream, dev)
        torch.cuda.synchronize()
        log(f"[ours] rank {rank}: {sum(ctx_lens)} cached prefix tokens prefilled in {time.time() - t0:.1f}s")

    def step():
        if ctx_lens is not None:
            api.forward(model, tokens, batch.cu_seqlens, ctx_lens, kv, logits=logits, stream=stream)
        else:
            api.prefill(model, tokens, batch.cu_seqlens, kv, logits=logits, stream=stream)

    def barrier():
        replica_barrier(world)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    st = model.status()
    if st != 0:
        raise RuntimeError(f"device status word {st} after warm-up")

    sampler = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else
                           int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local_rank]))
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.4)
    # the timed region: K steps with no instrumentation
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_per_step = ms / args.steps
    T_all = sum_over_ranks(T, world, dev)
    value = whole_job_throughput(T_all, args.steps, ms / 1e3)

    # where the time goes: the same K steps again, every launch bracketed by CUDA events on
    # its own stream (swiftkv_profile_begin/end); only the per-kernel breakdown and the
    # roofline come from this pass, never `value`
    binding.check(binding.lib().swiftkv_profile_begin(model.handle))
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(args.steps):
        step()
    p1.record(stream)
    torch.cuda.synchronize()
    entries = (binding.ProfileEntry * 64)()
    n_ent = binding.check(binding.lib().swiftkv_profile_end(model.handle, entries, 64))
    ms_profiled = p0.elapsed_time(p1) / args.steps
    st = model.status()
    if st != 0:
        raise RuntimeError(f"device status word {st} after the timed steps")

    prof = {}
    for i in range(n_ent):
        e = entries[i]
        prof[e.name.decode()] = {"calls": e.calls, "kernels": e.kernels, "ms": e.ms, "flops": e.flops,
                                 "bytes": e.bytes}
    launches = sum(v["kernels"] for v in prof.values())

    fl = FL.prefill_flops(w.shape, batch.lens, w.l, w.g, ctx=ctx_lens)
    dense_tflops = sum_over_ranks(fl["dense_equiv"], world, dev) * args.steps / (ms / 1e3) / 1e12
    exec_tflops = sum_over_ranks(fl["executed"], world, dev) * args.steps / (ms / 1e3) / 1e12
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))

    # dominant kernel class: the one with most device time
    dom_name = max(prof, key=lambda k: prof[k]["ms"]) if prof else None
    roofline = None
    if dom_name:
        d = prof[dom_name]
        tensor_bound = d["flops"] > 0 and (d["flops"] / max(d["bytes"], 1.0)) > 300
        if tensor_bound:
            ach = d["flops"] / (d["ms"] / 1e3) / 1e12
            roofline = {"kernel": dom_name, "bound": "tensor", "achieved": ach, "peak": peak_sus,
                        "unit": "TFLOP/s", "frac": ach / peak_sus,
                        "peak_source": f"{peak_src} bf16_tflops_sustained (kernel timed inside a long step)",
                        "traffic": traffic_per_launch(dom_name), "launch_avg_ms": d["ms"] / d["calls"],
                        "algorithmic_flops_per_launch": d["flops"] / d["calls"],
                        "timing": PROFILED_PASS_NOTE}
        else:
            ach = d["bytes"] / (d["ms"] / 1e3) / 1e9
            roofline = {"kernel": dom_name, "bound": "hbm", "achieved": ach, "peak": float(peaks["hbm_gbs"]),
                        "unit": "GB/s", "frac": ach / float(peaks["hbm_gbs"]),
                        "peak_source": f"{peak_src} hbm_gbs", "traffic": traffic_per_launch(dom_name),
                        "launch_avg_ms": d["ms"] / d["calls"], "algorithmic_bytes_per_launch": d["bytes"] / d["calls"],
                        "timing": PROFILED_PASS_NOTE}

    # end to end through the C ABI with host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e and ctx_lens is not None:
        # public Python API with pinned host buffers: token copy in, forward, logits copy out
        h_tok = torch.empty(T, dtype=torch.int32, pin_memory=True)
        h_tok.copy_(torch.as_tensor(batch.tokens))
        h_log = torch.empty((P, w.shape.vocab), dtype=torch.float32, pin_memory=True)
        d_tok = torch.empty(T, dtype=torch.int32, device=dev)

        def e2e_step():
            d_tok.copy_(h_tok, non_blocking=True)
            api.forward(model, d_tok, batch.cu_seqlens, ctx_lens, kv, logits=logits, stream=stream)
            h_log.copy_(logits, non_blocking=True)
            stream.synchronize()

        e2e_step()
        barrier()
        t1 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        el = max_over_ranks(time.perf_counter() - t1, world, dev)
        e2e = {"value": whole_job_throughput(T_all, args.steps, el), "unit": "tokens/s",
               "h2d_bytes_per_step": T * 4 + (2 * P + 1) * 4, "d2h_bytes_per_step": P * w.shape.vocab * 4,
               "ms_per_step": 1e3 * el / args.steps}
    elif not args.no_e2e:
        h_tok = torch.empty(T, dtype=torch.int32, pin_memory=True)
        h_tok.copy_(torch.as_tensor(batch.tokens))
        h_log = torch.empty((P, w.shape.vocab), dtype=torch.float32, pin_memory=True)
        h_tok_np, h_log_np = h_tok.numpy(), h_log.numpy()
        api.prefill_host(model, h_tok_np, batch.cu_seqlens, kv, logits=h_log_np, stream=stream)
        barrier()
        t1 = time.perf_counter()
        for _ in range(args.steps):
            api.prefill_host(model, h_tok_np, batch.cu_seqlens, kv, logits=h_log_np, stream=stream)
        el = max_over_ranks(time.perf_counter() - t1, world, dev)
        e2e = {"value": whole_job_throughput(T_all, args.steps, el), "unit": "tokens/s",
               "h2d_bytes_per_step": T * 4 + (P + 1) * 4, "d2h_bytes_per_step": P * w.shape.vocab * 4,
               "ms_per_step": 1e3 * el / args.steps}

    # decode from the filled caches (greedy, every sequence one token per step): TPOT
    decode = None
    n_dec = n_dec_req
    if n_dec > 0:
        if batch.block_table.shape[1] * 16 < int(batch.lens.max()) + n_dec:
            raise RuntimeError("block table too small for the decode steps")
        api.prefill(model, tokens, batch.cu_seqlens, kv, logits=logits, stream=stream)
        nxt = torch.argmax(logits, dim=-1).to(torch.int32)
        lens = [int(x) for x in batch.lens]
        api.decode_step(model, nxt, lens, kv, stream=stream)           # warm-up step
        lens = [x + 1 for x in lens]
        torch.cuda.synchronize()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(n_dec):
            _, nxt = api.decode_step(model, nxt, lens, kv, stream=stream)
            lens = [x + 1 for x in lens]
        d1.record(stream)
        torch.cuda.synchronize()
        tpot = max_over_ranks(d0.elapsed_time(d1) / n_dec, world, dev)
        # one more profiled pass of a few steps: where a decode step's time goes
        n_prof = min(n_dec, 5)
        binding.check(binding.lib().swiftkv_profile_begin(model.handle))
        for _ in range(n_prof):
            _, nxt = api.decode_step(model, nxt, lens, kv, stream=stream)
            lens = [x + 1 for x in lens]
        torch.cuda.synchronize()
        n_ent = binding.check(binding.lib().swiftkv_profile_end(model.handle, entries, 64))
        dk = {}
        for i in range(n_ent):
            e = entries[i]
            dk[e.name.decode()] = {"ms_per_step": e.ms / n_prof, "calls_per_step": e.calls / n_prof,
                                   "gbs": (e.bytes / (e.ms / 1e3) / 1e9) if e.bytes else None}
        decode = {"steps": n_dec, "batch": P, "tpot_ms": tpot, "ttft_ms": ms_per_step,
                  "decode_tokens_per_s": P * 1e3 / tpot,
                  "kernels_profiled": dict(sorted(dk.items(), key=lambda kv_: -kv_[1]["ms_per_step"]))}

    cpu = None
    if want_cpu:
        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        ow = oracle_weights(w, raw_layers, raw_globals)
        a = int(batch.cu_seqlens[0])
        n = min(args.cpu_sample_tokens, int(batch.lens[0]))
        sample = batch.tokens[a:a + n]
        secs = oracle_sample_time(w, ow, sample)
        cpu = {"value": n / secs, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"first {n} tokens of prompt 0 of this workload through the oracle's full "
                         f"SwiftKV prefill path (float64 NumPy), {secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded random-init weights and token ids; no dataset)",
            "config": workload_config(w, batch, args.norm_fusion),
            "dense_equiv_tflops": dense_tflops,
            "dense_equiv_frac_of_peak": {"burst": dense_tflops / peak_burst, "sustained": dense_tflops / peak_sus,
                                         "peak_source": peak_src},
            "executed_tflops": exec_tflops,
            "executed_frac_of_peak": {"burst": exec_tflops / peak_burst, "sustained": exec_tflops / peak_sus},
            "roofline": roofline,
            "step_roofline": step_roofline(prof, args.steps, ms_per_step, peak_sus,
                                           float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))),
            "ms_per_step_profiled": ms_profiled,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "kv_cache": kv_cache_info(model, w),
            "decode": decode,
            "clocks": clocks,
            "kernels": {k: {"ms_per_step": v["ms"] / args.steps, "calls_per_step": v["calls"] / args.steps,
                            "tflops": (v["flops"] / (v["ms"] / 1e3) / 1e12) if v["flops"] else None,
                            "gbs": (v["bytes"] / (v["ms"] / 1e3) / 1e9) if v["bytes"] else None}
                        for k, v in sorted(prof.items(), key=lambda kv_: -kv_[1]["ms"])},
        }
        print(json.dumps(line), flush=True)
    model.free()
    return 0


def step_roofline(prof: dict, steps: int, ms_per_step: float, peak_tflops: float, hbm_gbs: float) -> dict:
    """End-to-end roofline of one step: the sum over kernel classes of
    max(FLOPs / bf16 peak, bytes / HBM bandwidth), from the algorithmic FLOPs and bytes each
    class records, against the measured (uninstrumented) step time. Classes that record
    neither (plan, host uploads) count zero; attention classes record both their FLOPs and
    the K/V, Q and output bytes they must move."""
    t = 0.0
    per = {}
    for name, v in prof.items():
        tf = (v["flops"] or 0.0) / (peak_tflops * 1e12)
        tb = (v["bytes"] or 0.0) / (hbm_gbs * 1e9)
        per[name] = 1e3 * max(tf, tb) / steps
        t += per[name]
    return {"t_roofline_ms": t, "ms_per_step": ms_per_step, "frac": t / ms_per_step if ms_per_step > 0 else None,
            "peak_tflops": peak_tflops, "hbm_gbs": hbm_gbs,
            "per_class_ms": dict(sorted(per.items(), key=lambda kv_: -kv_[1]))}


def kv_cache_info(model, w) -> dict:
    """KV-cache bytes per token (all caches, K and V, scales included) and the reduction
    against an ordinary model's bf16 cache (L caches)."""
    sh = w.shape
    per_head = sh.d_h * (1 if w.kv_dtype == "fp8" else 2) + (4 if w.kv_dtype == "fp8" else 0)
    per_token = model.num_caches * 2 * sh.n_kv * per_head
    ordinary = sh.L * 2 * sh.n_kv * sh.d_h * 2
    return {"dtype": w.kv_dtype, "caches": model.num_caches, "bytes_per_token": per_token,
            "reduction_vs_ordinary_bf16": 1.0 - per_token / ordinary}


def fill_prefixes(model, kv, batch, stream, dev, max_tokens: int = 16384) -> None:
    """Prefills the cached prefix of every sequence of a serving-step batch (ctx > 0) in
    groups of at most max_tokens tokens (a longer prefix gets a group of its own)."""
    import torch
    from swiftkv_prefill_skipping_gb300 import api
    ctx, pcu, ptok = batch.extra["ctx"], batch.extra["prefix_cu"], batch.extra["prefix_tokens"]
    rows = [s for s in range(len(ctx)) if ctx[s] > 0]
    group, n = [], 0

    def run(group):
        toks = np.concatenate([ptok[pcu[s]:pcu[s + 1]] for s in group])
        cu = np.concatenate([[0], np.cumsum([int(ctx[s]) for s in group])]).astype(np.int32)
        api.prefill(model, torch.as_tensor(toks, device=dev), cu, kv.view(group), stream=stream)

    for s in rows:
        if group and n + int(ctx[s]) > max_tokens:
            run(group)
            group, n = [], 0
        group.append(s)
        n += int(ctx[s])
    if group:
        run(group)


def traffic_per_launch(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None when the
    summary is absent or was taken on a different build of the kernel's sources."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.md")
    if not os.path.exists(p):
        return None
    import hashlib
    rows = {}
    with open(p) as f:
        for line in f:
            if line.startswith("traffic|"):
                _, name, srcs, digest, bytes_ = line.strip().split("|")
                rows[name] = (srcs.split("+"), digest, float(bytes_))
    if kernel not in rows:
        return None
    srcs, digest, b = rows[kernel]
    h = hashlib.sha256()
    for src in srcs:
        path = os.path.join(ROOT, src)
        if not os.path.exists(path):
            return None
        with open(path, "rb") as f:
            h.update(f.read())
    return b if h.hexdigest()[:16] == digest else None


def relaunch_ranks(n: int) -> int:
    """`bench.py --gpus N` outside torchrun: start N ranks on this node (one per GPU) through
    torch.distributed.run on 127.0.0.1 and return its exit status."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="llama8b_l16", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=512)
    ap.add_argument("--ref-sample-tokens", type=int, default=128)
    ap.add_argument("--norm-fusion", type=int, choices=(0, 1), default=0,
                    help="prompt rows' RMSNorm inside the GEMM epilogues (1) or as its own pass (0, default)")
    ap.add_argument("--decode-steps", type=int, default=None,
                    help="greedy decode steps timed after the prefill (default: the workload's own)")
    args = ap.parse_args()
    w = synth.WORKLOADS[args.workload]
    if args.gpus < 1:
        log(f"--gpus {args.gpus}: need at least one GPU")
        return 2
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return relaunch_ranks(args.gpus)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        log(f"--gpus {args.gpus} does not match WORLD_SIZE={world}: launch one rank per GPU "
            f"(torchrun --nproc-per-node {args.gpus}) or pass --gpus {world}")
        return 2
    if args.impl == "reference":
        return run_reference(args, w, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        return run_ours(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
