"""Single-kernel timing and profiling driver (CUDA events on the launch stream).

  python -m swiftkv_prefill_skipping_gb300.kernel_bench gemm --impl 0 --M 11703 --N 6144 --K 4096
  python -m swiftkv_prefill_skipping_gb300.kernel_bench prefill --layers 2 --l 1 --prompts 16
  python -m swiftkv_prefill_skipping_gb300.kernel_bench decode --batch 24 --ctx 1000 --kv fp8

`gemm` runs the C-ABI GEMM self-test entry (impl 0 tcgen05, 1 mma.sync tiles; impl 2 is
the skinny split-K kernel through swiftkv_gemm_skinny_noalloc, so no allocation is timed)
on seeded bf16 operands and reports TFLOP/s and GB/s of operand traffic. `prefill` runs a SwiftKV prefill of a
reduced-depth model with the Llama-3.1-8B layer shape (same per-layer kernels as the
full model, a few GB on the device) and prints the per-kernel-class breakdown; it is
the small case for profiling the attention and norm kernels. `decode` prefills `batch`
sequences of `ctx` tokens through a reduced-depth model with the Qwen2.5-14B layer shape
(40 query heads, 8 KV heads, d_head 128) and times greedy decode steps from its bf16 or
FP8 cache: the small case for the single-row attention and the skinny GEMMs (`--rows-impl 1`: one launch
per GEMM and norm instead of the chained launch per layer).
"""
from __future__ import annotations

import argparse
import ctypes as C
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def gemm(args):
    import torch
    from swiftkv_prefill_skipping_gb300 import binding as B
    lib = B.lib()
    g = torch.Generator(device="cuda").manual_seed(0)
    A = (torch.randn(args.M, args.K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    W = (torch.randn(args.N, args.K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    out = torch.empty(args.M, args.N, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream()

    def run():
        if args.impl == 2:   # skinny split-K through the entry that allocates nothing per call
            B.check(lib.swiftkv_gemm_skinny_noalloc(A.data_ptr(), W.data_ptr(), out.data_ptr(), args.M, args.N,
                                                    args.K, C.c_void_p(s.cuda_stream)))
        else:
            B.check(lib.swiftkv_gemm_bf16(A.data_ptr(), W.data_ptr(), out.data_ptr(), args.M, args.N, args.K,
                                          args.impl, st.data_ptr(), C.c_void_p(s.cuda_stream)))

    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(args.iters):
        run()
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / max(args.iters, 1)
    tf = 2.0 * args.M * args.N * args.K / (ms / 1e3) / 1e12
    gbs = 2.0 * (args.M + args.N) * args.K / (ms / 1e3) / 1e9
    print(json.dumps({"kernel": "gemm", "impl": args.impl, "M": args.M, "N": args.N, "K": args.K,
                      "ms": ms, "tflops": tf, "operand_gbs": gbs, "status": int(st.item())}))


def prefill(args):
    import dataclasses

    import torch

    import synth
    from swiftkv_prefill_skipping_gb300 import api, binding
    shape = dataclasses.replace(synth.LLAMA8B, L=args.layers, name=f"llama3.1-8b-width-{args.layers}layers")
    batch = synth.prompt_batch(shape.vocab, args.prompts, args.len_lo, args.len_hi)
    m = api.load_synthetic(shape, args.l, args.g)
    kv = api.KVCache(m, batch.num_pages, batch.block_table)
    tok = torch.as_tensor(batch.tokens, device="cuda")
    for _ in range(args.warmup):
        api.prefill(m, tok, batch.cu_seqlens, kv)
    torch.cuda.synchronize()
    binding.check(binding.lib().swiftkv_profile_begin(m.handle))
    for _ in range(args.iters):
        api.prefill(m, tok, batch.cu_seqlens, kv)
    torch.cuda.synchronize()
    ents = (binding.ProfileEntry * 64)()
    n = binding.check(binding.lib().swiftkv_profile_end(m.handle, ents, 64))
    res = {}
    for i in range(n):
        e = ents[i]
        res[e.name.decode()] = {"ms_per_iter": e.ms / args.iters, "calls": e.calls // args.iters,
                                "tflops": e.flops / (e.ms / 1e3) / 1e12 if e.flops else None,
                                "gbs": e.bytes / (e.ms / 1e3) / 1e9 if e.bytes else None}
    print(json.dumps({"kernel": "prefill", "tokens": int(batch.cu_seqlens[-1]), "layers": args.layers,
                      "l": args.l, "classes": res}))
    assert m.status() == 0


def decode(args):
    import dataclasses

    import torch

    import synth
    from swiftkv_prefill_skipping_gb300 import api, binding
    shape = dataclasses.replace(synth.QWEN14B, L=args.layers, name=f"qwen2.5-14b-width-{args.layers}layers")
    batch = synth.prompt_batch(shape.vocab, args.batch, args.ctx, args.ctx,
                               reserve_tokens=args.warmup + 2 * args.iters)  # timed and profiled passes
    m = api.load_synthetic(shape, args.l, args.g)
    binding.check(binding.lib().swiftkv_set_rows_impl(m.handle, args.rows_impl))
    kv = api.KVCache(m, batch.num_pages, batch.block_table, dtype=args.kv)
    lg = api.prefill(m, torch.as_tensor(batch.tokens, device="cuda"), batch.cu_seqlens, kv)
    nxt = torch.argmax(lg, dim=-1).to(torch.int32)
    lens = [int(x) for x in batch.lens]
    for _ in range(args.warmup):
        _, nxt = api.decode_step(m, nxt, lens, kv)
        lens = [x + 1 for x in lens]
    torch.cuda.synchronize()
    # whole steps without per-launch events, then the same number with them (breakdown)
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(args.iters):
        _, nxt = api.decode_step(m, nxt, lens, kv)
        lens = [x + 1 for x in lens]
    e1.record(s)
    torch.cuda.synchronize()
    step_ms = e0.elapsed_time(e1) / args.iters
    binding.check(binding.lib().swiftkv_profile_begin(m.handle))
    for _ in range(args.iters):
        _, nxt = api.decode_step(m, nxt, lens, kv)
        lens = [x + 1 for x in lens]
    torch.cuda.synchronize()
    ents = (binding.ProfileEntry * 64)()
    n = binding.check(binding.lib().swiftkv_profile_end(m.handle, ents, 64))
    res = {}
    for i in range(n):
        e = ents[i]
        res[e.name.decode()] = {"ms_per_step": e.ms / args.iters, "calls": e.calls // args.iters,
                                "gbs": e.bytes / (e.ms / 1e3) / 1e9 if e.bytes else None}
    print(json.dumps({"kernel": "decode", "batch": args.batch, "ctx": args.ctx, "kv": args.kv,
                      "layers": args.layers, "rows_impl": args.rows_impl, "step_ms": step_ms, "classes": res}))
    assert m.status() == 0


def main():
    ap = argparse.ArgumentParser()
    sub = ap.add_subparsers(dest="cmd", required=True)
    g = sub.add_parser("gemm")
    g.add_argument("--impl", type=int, default=0)
    g.add_argument("--M", type=int, default=11703)
    g.add_argument("--N", type=int, default=6144)
    g.add_argument("--K", type=int, default=4096)
    g.add_argument("--iters", type=int, default=10)
    g.add_argument("--warmup", type=int, default=3)
    p = sub.add_parser("prefill")
    p.add_argument("--layers", type=int, default=2)
    p.add_argument("--l", type=int, default=1)
    p.add_argument("--g", type=int, default=1)
    p.add_argument("--prompts", type=int, default=16)
    p.add_argument("--len-lo", type=int, default=500)
    p.add_argument("--len-hi", type=int, default=1000)
    p.add_argument("--iters", type=int, default=5)
    p.add_argument("--warmup", type=int, default=2)
    d = sub.add_parser("decode")
    d.add_argument("--layers", type=int, default=2)
    d.add_argument("--l", type=int, default=1)
    d.add_argument("--g", type=int, default=1)
    d.add_argument("--batch", type=int, default=24)
    d.add_argument("--ctx", type=int, default=1000)
    d.add_argument("--kv", choices=("bf16", "fp8"), default="bf16")
    d.add_argument("--rows-impl", type=int, choices=(0, 1), default=0)
    d.add_argument("--iters", type=int, default=3)
    d.add_argument("--warmup", type=int, default=2)
    args = ap.parse_args()
    {"gemm": gemm, "prefill": prefill, "decode": decode}[args.cmd](args)


if __name__ == "__main__":
    main()
