"""Benchmark of the Dory looped nGPT token forward on GB300.

Default workload: the 2B-shaped bf16 model (hidden 2048, 16 q / 4 kv heads of 128, ffn
5632, vocab 32000, 2/4/2 attention+MLP pairs, loops 4, sliding window 512, last_loop f32
KV): a 4096-token seeded prompt in 64-row chunks, then batch-1 decode steps with
teacher-forced seeded ids. One step = one decode token through the whole forward.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line. Under torchrun each rank runs its own replica (batch-1 decode does
not shard), ranks meet at a barrier around the timed region, and the slowest rank's time
counts. `--impl reference` times the CPU oracle on the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode tokens/s at batch 1/64 (loops=4) + fraction of HBM roofline; prefill tok/s"
SEED = 1236  # seed = 1234 + config index (the 2B decode workload is the second config)
PROMPT = 4096
DECODE = 256


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return j["hbm_gbs"], j["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


class Clocks:
    """nvidia-smi samples of the SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev: int):
        self.dev = dev
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.p:
            self.p.terminate()
            try:
                self.out, _ = self.p.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = max(mx, float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# DRAM bytes (read + write) per algorithmic byte of the persistent decode kernel, from the
# ncu capture of the reduced 3-pass case (429.4 + 4.8 MB for 427.3 MB of weights and KV);
# the kernel streams every weight once per token, so the ratio carries to the full model.
MEGA_TRAFFIC_PER_BYTE = (429.4 + 4.8) / 427.3


def roofline_decode(st, bytes_step, achieved, hbm, src):
    """The batch-1 decode step is one launch of the persistent kernel, after one memset of
    its counters and tagged words (652 KB for the 2B shape, about a microsecond), so the
    step's CUDA-event time is that kernel's launch duration (and a little more)."""
    one = int(st["launches"]) == 1
    return {"bound": "hbm", "kernel": "mega_decode_kernel" if one else "fused decode kernels",
            "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
            "traffic": round(bytes_step * MEGA_TRAFFIC_PER_BYTE) if one else None,
            "note": f"algorithmic bytes per launch {bytes_step} (bf16 weights once + f32 KV rows read and "
                    f"written) / launch time from CUDA events on the launching stream; traffic = ncu dram "
                    f"read+write per algorithmic byte of the same kernel (reduced 3-pass case) x these "
                    f"bytes; peak {src}"}


def workload_config():
    return synth.dory2b(max_batch=1, max_seqs=1, max_context=PROMPT + DECODE + 64)


def profile_case(args):
    """Small cases for ncu captures (each prints one JSON line; none is a bench line):
    decode-3pass: batch-1 decode of the 2B shape cut to one input, one recurrent and one
    output pair at loops 1 (427 MB of weights per token, still larger than L2, about 1 GB on
    the device); prefill: 64-row chunks of a prompt of --prompt tokens on the 2B model;
    prefill-whole: the same prompt in one dory_prefill call;
    batch64: the batch-64 decode line with 4 timed steps (in an NVTX range "decode")."""
    import torch

    from looped_normalized_gpt_gb300 import Dory, build

    build()
    if args.profile_case == "batch64":
        w = synth.weights(synth.dory2b(), SEED)
        out = bench_batch(Dory, torch, w, int(os.environ.get("LOCAL_RANK", "0")), steps=4, nvtx=True)
        return {"case": "batch64", **out, "note": "profiling case, not a bench line"}
    if args.profile_case == "context-small":
        # the long-context lines on fewer sequences (a few GB on the device), the timed decode
        # steps inside an NVTX range "decode" (ncu --nvtx --nvtx-include decode/)
        w = synth.weights(synth.dory2b(), SEED)
        dev = int(os.environ.get("LOCAL_RANK", "0"))
        # (6 and 8 rows: the steps of 5+ rows of the bench lines, tensor-core projections)
        pl = synth.dory2b(rec_kinds="S*S*", kv_mode="per_loop", max_loops=8, loops=8, full_window=8192,
                          max_batch=6, max_seqs=6, max_context=8192 + 64)
        q8 = synth.dory2b(rec_kinds="S*S*", kv_mode="last_loop", kv_quant="q8_2f", loops=16, max_loops=16,
                          full_window=8192, max_batch=8, max_seqs=8, max_context=8192 + 64)
        return {"case": "context-small",
                "per_loop_batch6": bench_context_decode(Dory, torch, w, dev, pl, 6, 8192, [2, 4, 8, 4], 1, SEED + 1,
                                                        nvtx=True),
                "q8_batch8": bench_context_decode(Dory, torch, w, dev, q8, 8, 8192, [16, 16], 1, SEED + 3, nvtx=True),
                "note": "profiling case, not a bench line"}
    if args.profile_case in ("context-per-loop", "context-q8"):  # one long-context batch line alone
        w = synth.weights(synth.dory2b(), SEED)
        dev = int(os.environ.get("LOCAL_RANK", "0"))
        fn = bench_per_loop16 if args.profile_case == "context-per-loop" else bench_q8_batch64
        return {"case": args.profile_case, "line": fn(Dory, torch, w, dev, nvtx=True),
                "note": "profiling case, not a bench line"}
    if args.profile_case == "context":  # the two long-context batch lines alone (timed steps in NVTX "decode")
        w = synth.weights(synth.dory2b(), SEED)
        dev = int(os.environ.get("LOCAL_RANK", "0"))
        return {"case": "context", "per_loop_batch16": bench_per_loop16(Dory, torch, w, dev, nvtx=True),
                "q8_batch64": bench_q8_batch64(Dory, torch, w, dev, nvtx=True), "note": "profiling case, not a bench line"}
    if args.profile_case in ("prefill", "prefill-whole"):
        cfg = synth.dory2b(max_batch=1, max_seqs=1, max_context=args.prompt + 64, prompt_loops=2)
        g = Dory(cfg, synth.weights(cfg, SEED))
        ids = synth.token_ids(SEED, 0, args.prompt, cfg.vocab)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        if args.profile_case == "prefill-whole":
            g.prefill(0, ids, 0, cfg.loops, "none")
        else:
            for a0 in range(0, args.prompt, 64):
                g.prefill_chunk(0, ids[a0:a0 + 64], a0, cfg.loops, "none")
        torch.cuda.synchronize()
        ms = (time.perf_counter() - t0) * 1e3
        g.close()
        return {"case": "prefill", "tokens": args.prompt, "ms_host": round(ms, 3),
                "note": "profiling case, not a bench line"}
    pat, a, b, c = synth.pattern_of("S", "S", "S")
    cfg = synth.dory2b(pattern=pat, n_in=a, n_rec=b, n_out=c, loops=1, max_batch=1, max_seqs=1,
                       max_context=args.prompt + DECODE + 64)
    w = synth.weights(cfg, SEED)
    g = Dory(cfg, w)
    ids = synth.token_ids(SEED, 0, args.prompt + DECODE, cfg.vocab)
    for a0 in range(0, args.prompt, 64):
        g.prefill_chunk(0, ids[a0:a0 + 64], a0, cfg.loops, "none")
    dec = ids[args.prompt:]
    for i in range(args.warmup):
        g.decode_step([int(dec[i])], [0], cfg.loops)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.warmup, args.warmup + args.steps):
        g.decode_step([int(dec[i])], [0], cfg.loops)
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / max(args.steps, 1)
    st = g.stats()
    g.close()
    return {"case": "decode-2b-3pass", "ms_per_step_host": round(ms, 4), "launches_per_step": st["launches"],
            "weight_bytes_per_step": st["weight_bytes"], "note": "profiling case, not a bench line"}


def bench_ours(args, rank, world):
    global PROMPT
    PROMPT = args.prompt
    import torch

    from looped_normalized_gpt_gb300 import Dory, build
    from looped_normalized_gpt_gb300.shard import job_throughput, slowest

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    build()
    cfg = workload_config()
    t0 = time.time()
    w = synth.weights(cfg, SEED)
    t_gen = time.time() - t0
    stream = torch.cuda.current_stream()
    g = Dory(cfg, w, stream=stream.cuda_stream)
    ids = synth.token_ids(SEED, 0, PROMPT + DECODE, cfg.vocab)
    prompt, dec = ids[:PROMPT], ids[PROMPT:]
    for a in range(0, PROMPT, 64):
        g.prefill_chunk(0, prompt[a:a + 64], a, cfg.loops, "last" if a + 64 >= PROMPT else "none")
    torch.cuda.synchronize()
    dec_dev = torch.from_numpy(dec.astype(np.int32)).to(f"cuda:{dev}")
    K, W = args.steps, args.warmup
    assert W + K <= DECODE, "warmup + steps must fit the 256 decode tokens"
    for i in range(W):
        g.decode_step(dec_dev[i:i + 1], [0], cfg.loops)
    st = g.stats()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(dev) as clk:
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(W, W + K):
            g.decode_step(dec_dev[i:i + 1], [0], cfg.loops)
        e1.record(stream)
        torch.cuda.synchronize()
    ms = slowest(e0.elapsed_time(e1))  # the slowest rank's time (one replica per rank)
    if world > 1:
        torch.distributed.barrier()
    value = job_throughput(K, ms, world)

    # end to end: host ids from pinned memory in, logits back to host, every step
    g2_ids = torch.from_numpy(dec.astype(np.int32)).pin_memory()
    host_logits = torch.empty(cfg.vocab, dtype=torch.float32).pin_memory()
    g.reset(0)
    for a in range(0, PROMPT, 64):
        g.prefill_chunk(0, prompt[a:a + 64], a, cfg.loops, "last" if a + 64 >= PROMPT else "none")
    for i in range(W):
        g.decode_step(g2_ids[i:i + 1], [0], cfg.loops)
        g.logits(0, out=host_logits)
    torch.cuda.synchronize()
    t_a = time.perf_counter()
    for i in range(W, W + K):
        g.decode_step(g2_ids[i:i + 1], [0], cfg.loops)
        g.logits(0, out=host_logits)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t_a
    e2e = world * K / e2e_s

    hbm, tf, src = peaks()
    bytes_step = st["weight_bytes"] + st["kv_read_bytes"] + st["kv_write_bytes"]
    achieved = bytes_step / (ms / 1e3 / K) / 1e9
    clocks = clk.summary()
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms / K, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 weights, f32 activations and KV",
        "data": "synthetic: seeded unit-row random weights, seeded uniform token ids",
        "config": {"workload": f"Dory-2B-shape batch-1 decode after a {PROMPT}-token prompt, loops 4, "
                               "sliding window 512, last_loop f32 KV",
                   "batch": 1, "loops": 4, "prompt": PROMPT, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (2.1 GB of weights streamed per token)"},
        "e2e": {"value": round(e2e, 2), "unit": "tokens/s", "h2d_bytes_per_step": 4 + 16,
                "d2h_bytes_per_step": cfg.vocab * 4},
        "gpu_launches": int(st["launches"]) * K,
        "roofline": roofline_decode(st, bytes_step, achieved, hbm, src),
        "clocks": clocks,
        "weights_gen_s": round(t_gen, 1),
    }
    return out, g, cfg, w


def bench_context_decode(g_cls, torch, w, dev, cfg, nseq: int, ctx: int, sched, warmup: int, seed: int,
                         nvtx: bool = False):
    """Batch decode at a long synthetic context: `nseq` sequences with `ctx` unit-norm K/V rows
    in every slot (drawn on the GPU, written through the append path, so q8 rings quantise
    and freeze as in a forward), then len(sched) timed steps, step i at sched[i] loops. The
    algorithmic bytes are the weights once per step plus the K/V rows read and written,
    summed over the timed steps. The weights are the main line's 2B set (the values do not
    change the bytes moved)."""
    stream = torch.cuda.current_stream()
    g = g_cls(cfg, w, stream=stream.cuda_stream)
    try:
        gen = torch.Generator(device=f"cuda:{dev}")
        gen.manual_seed(seed)
        for s_ in range(nseq):
            for o in range(cfg.attn_layers):
                _, slots, _ = g.slot_info(o)
                for sl in range(slots):
                    k = torch.randn(ctx, cfg.nk, cfg.hd, device=f"cuda:{dev}", generator=gen)
                    v = torch.randn(ctx, cfg.nk, cfg.hd, device=f"cuda:{dev}", generator=gen)
                    k /= k.norm(dim=2, keepdim=True)
                    v /= v.norm(dim=2, keepdim=True)
                    g.write_kv_rows(s_, o, sl, 0, k.contiguous(), v.contiguous())
            g.set_position(s_, ctx)
        steps = len(sched)
        ids = torch.from_numpy(synth.token_ids(seed, 7, nseq * (steps + warmup), cfg.vocab)).to(f"cuda:{dev}")
        seqs = list(range(nseq))
        for i in range(warmup):
            g.decode_step(ids[i * nseq:(i + 1) * nseq], seqs, int(sched[i % steps]))
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b = 0
        if nvtx:
            torch.cuda.nvtx.range_push("decode")
        e0.record(stream)
        for i in range(steps):
            j = warmup + i
            g.decode_step(ids[j * nseq:(j + 1) * nseq], seqs, int(sched[i]))
            st = g.stats()
            b += st["weight_bytes"] + st["kv_read_bytes"] + st["kv_write_bytes"]
        e1.record(stream)
        if nvtx:
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        s_total = e0.elapsed_time(e1) / 1e3
        hbm, _, _ = peaks()
        return {"value": round(nseq * steps / s_total, 1), "unit": "tokens/s", "ms_per_step": round(s_total * 1e3 / steps, 4),
                "batch": nseq, "context": ctx, "loops": sorted({int(x) for x in sched}), "kv": cfg.kv_quant,
                "kv_mode": cfg.kv_mode,
                "roofline": {"bound": "hbm", "achieved": round(b / s_total / 1e9, 1), "peak": hbm, "unit": "GB/s",
                             "frac": round(b / s_total / 1e9 / hbm, 4), "bytes_per_step": round(b / steps)}}
    finally:
        g.close()


def bench_per_loop16(g_cls, torch, w, dev, steps: int = 16, warmup: int = 3, nvtx: bool = False):
    """per_loop KV, batch 16 at context 8192, every second recurrent attention layer full
    (full_window 8192), loops drawn per step from {2, 4, 8}."""
    cfg = synth.dory2b(rec_kinds="S*S*", kv_mode="per_loop", max_loops=8, loops=8, full_window=8192,
                       max_batch=16, max_seqs=16, max_context=8192 + steps + warmup + 64)
    return bench_context_decode(g_cls, torch, w, dev, cfg, 16, 8192, synth.loop_schedule(SEED + 1, steps), warmup,
                                SEED + 1, nvtx=nvtx)


def bench_q8_batch64(g_cls, torch, w, dev, steps: int = 8, warmup: int = 3, nvtx: bool = False):
    """q8_2f KV (last_loop), batch 64 at context 8192, loops 16, full layers capped at 8192."""
    cfg = synth.dory2b(rec_kinds="S*S*", kv_mode="last_loop", kv_quant="q8_2f", loops=16, max_loops=16,
                       full_window=8192, max_batch=64, max_seqs=64, max_context=8192 + steps + warmup + 64)
    return bench_context_decode(g_cls, torch, w, dev, cfg, 64, 8192, [16] * steps, warmup, SEED + 3, nvtx=nvtx)


def bench_batch(g_cls, torch, w, dev, batch: int = 64, ctx: int = 1024, steps: int = 16, warmup: int = 3,
                nvtx: bool = False):
    """Batch decode on the same model: `batch` sequences, each with `ctx` positions of
    synthetic unit-norm K/V rows in every slot, then `steps` decode steps at loops 4 (inside
    an NVTX range "decode" with `nvtx`)."""
    cfg = synth.dory2b(max_batch=batch, max_seqs=batch, max_context=ctx + steps + warmup + 64)
    stream = torch.cuda.current_stream()
    g = g_cls(cfg, w, stream=stream.cuda_stream)
    try:
        gen = torch.Generator(device=f"cuda:{dev}")
        gen.manual_seed(SEED + 100)
        n_attn = cfg.attn_layers
        for s_ in range(batch):
            for o in range(n_attn):
                k = torch.randn(ctx, cfg.nk, cfg.hd, device=f"cuda:{dev}", generator=gen)
                v = torch.randn(ctx, cfg.nk, cfg.hd, device=f"cuda:{dev}", generator=gen)
                k /= k.norm(dim=2, keepdim=True)
                v /= v.norm(dim=2, keepdim=True)
                g.write_kv_rows(s_, o, 0, 0, k.contiguous(), v.contiguous())
            g.set_position(s_, ctx)
        ids = torch.from_numpy(synth.token_ids(SEED, 7, batch * (steps + warmup), cfg.vocab)).to(f"cuda:{dev}")
        seqs = list(range(batch))
        for i in range(warmup):
            g.decode_step(ids[i * batch:(i + 1) * batch], seqs, cfg.loops)
        st = g.stats()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if nvtx:
            torch.cuda.nvtx.range_push("decode")
        for i in range(warmup, warmup + steps):
            g.decode_step(ids[i * batch:(i + 1) * batch], seqs, cfg.loops)
        if nvtx:
            torch.cuda.nvtx.range_pop()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        hbm, _, _ = peaks()
        b = st["weight_bytes"] + st["kv_read_bytes"] + st["kv_write_bytes"]
        return {"value": round(batch / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
                "batch": batch, "context": ctx, "loops": cfg.loops,
                "roofline": {"bound": "hbm", "achieved": round(b / (ms / 1e3) / 1e9, 1), "peak": hbm, "unit": "GB/s",
                             "frac": round(b / (ms / 1e3) / 1e9 / hbm, 4), "bytes_per_step": b}}
    finally:
        g.close()


def bench_prefill(g_cls, torch, w, n_tokens: int = 16384, prompt_loops: int = 2, whole: bool = True):
    """Prefill of an n-token seeded prompt at loops 4 (prompt_loops for the chunks whose logits
    are unread, the last chunk reads its last row). whole: one dory_prefill call (input and
    output blocks over 512 rows at once, the recurrent block in 64-row chunks); else one
    dory_prefill_chunk call per 64 rows. Reports the HBM roofline (weights streamed per step)
    and the bf16 tensor roofline (algorithmic projection FLOPs, 2 x weights x rows)."""
    cfg = synth.dory2b(max_batch=1, max_seqs=1, max_context=n_tokens + 64, prompt_loops=prompt_loops)
    stream = torch.cuda.current_stream()
    g = g_cls(cfg, w, stream=stream.cuda_stream)
    try:
        ids = synth.token_ids(SEED + 2, 0, n_tokens, cfg.vocab)
        dids = torch.from_numpy(ids).to("cuda")

        def run():
            g.reset(0)
            if whole:
                g.prefill(0, dids, 0, cfg.loops, "last")
                st = g.stats()
                return st["weight_bytes"], st["flops"]
            wb = fl = 0
            for a in range(0, n_tokens, 64):
                g.prefill_chunk(0, dids[a:a + 64], a, cfg.loops, "last" if a + 64 >= n_tokens else "none")
                st = g.stats()
                wb += st["weight_bytes"]
                fl += st["flops"]
            return wb, fl
        run()  # warm-up: captures the step graphs
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        wb, fl = run()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        hbm, tf, src = peaks()
        return {"value": round(n_tokens / (ms / 1e3), 1), "unit": "tokens/s", "ms": round(ms, 2),
                "tokens": n_tokens, "call": "dory_prefill" if whole else "dory_prefill_chunk x 64 rows",
                "loops": cfg.loops, "prompt_loops": prompt_loops,
                "roofline": {"bound": "hbm", "achieved": round(wb / (ms / 1e3) / 1e9, 1), "peak": hbm,
                             "unit": "GB/s", "frac": round(wb / (ms / 1e3) / 1e9 / hbm, 4), "weight_bytes": wb},
                "tensor": {"achieved": round(fl / (ms / 1e3) / 1e12, 1), "peak": tf, "unit": "TFLOP/s",
                           "frac": round(fl / (ms / 1e3) / 1e12 / tf, 4), "flops": fl,
                           "note": f"algorithmic projection and head FLOPs (2 x weights x rows) over the call; "
                                   f"peak: bf16 dense, {src}"}}
    finally:
        g.close()


def cpu_baseline(cfg, w, steps: int = 6):
    """The oracle as it stands, on this host's cores: a 64-token prompt, then `steps` timed
    decode tokens of the same model."""
    from oracle import dory_oracle as O

    o = O.DoryOracle(cfg, w)
    st = O.SeqState()
    ids = synth.token_ids(SEED, 0, 64 + steps + 1, cfg.vocab)
    o.forward_chunk(st, ids[:64], 0, cfg.loops, "last")
    o.forward_chunk(st, ids[64:65], 64, cfg.loops, "last")
    t = time.perf_counter()
    for i in ids[65:65 + steps]:
        o.forward_chunk(st, [int(i)], st.pos, cfg.loops, "last")
    s = time.perf_counter() - t
    return {"value": round(steps / s, 3), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{steps} batch-1 decode tokens after a 64-token prompt, same model, float64 NumPy"}


def bench_reference(args, rank, world):
    if rank != 0:
        return None
    cfg = workload_config()
    w = synth.weights(cfg, SEED)
    from oracle import dory_oracle as O

    o = O.DoryOracle(cfg, w)
    st = O.SeqState()
    ids = synth.token_ids(SEED, 0, 64 + args.warmup + args.steps, cfg.vocab)
    o.forward_chunk(st, ids[:64], 0, cfg.loops, "last")
    for i in ids[64:64 + args.warmup]:
        o.forward_chunk(st, [int(i)], st.pos, cfg.loops, "last")
    t = time.perf_counter()
    for i in ids[64 + args.warmup:]:
        o.forward_chunk(st, [int(i)], st.pos, cfg.loops, "last")
    s = time.perf_counter() - t
    v = args.steps / s
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * s / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded unit-row random weights, seeded uniform token ids",
        "config": {"workload": "Dory-2B-shape batch-1 decode after a 64-token prompt (bounded CPU sample), loops 4, "
                               "sliding window 512, last_loop f32 KV", "batch": 1, "loops": 4},
        "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"{args.steps} decode tokens after a 64-token prompt"},
        "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the batch-64 decode and prefill lines")
    ap.add_argument("--prompt", type=int, default=PROMPT, help="prompt tokens before the decode steps")
    ap.add_argument("--profile-case", choices=["decode-3pass", "prefill", "prefill-whole", "batch64", "context",
                                               "context-small", "context-per-loop", "context-q8"],
                    help="run a small case for ncu captures instead of the bench")
    args = ap.parse_args()
    if args.profile_case:
        print(json.dumps(profile_case(args)), flush=True)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        out = bench_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        import torch

        torch.distributed.init_process_group("nccl")
    out, g, cfg, w = bench_ours(args, rank, world)
    g.close()
    if not args.no_extra:
        import torch

        from looped_normalized_gpt_gb300 import Dory

        dev = int(os.environ.get("LOCAL_RANK", "0"))
        out["extra"] = {"decode_batch64": bench_batch(Dory, torch, w, dev),
                        "prefill_16k": bench_prefill(Dory, torch, w),
                        "prefill_16k_chunks": bench_prefill(Dory, torch, w, whole=False),
                        "decode_per_loop_batch16_ctx8192": bench_per_loop16(Dory, torch, w, dev),
                        "decode_q8_batch64_ctx8192": bench_q8_batch64(Dory, torch, w, dev)}
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(cfg, w)
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch

        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
