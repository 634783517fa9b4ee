"""Benchmark of libfattn on one GB300 (or N independent replicas under torchrun).

Primary line: config 2, causal prefill B=4 T=2048 Hq=12 Hkv=2 d=128 (bf16
inputs, fp32 accumulation) -> algorithmic TFLOP/s (4*d per unmasked
query/key pair).  Secondary entries: config 3 paged decode (KV GB/s),
config 4 long masked prefill, config 5 chunked prefill over the paged cache.

Timing: W warm-up steps, then exactly K timed steps; each step's kernel work
is bracketed by CUDA events on the launching stream and the L2 cache is
flushed before every step, outside the events (a 2x-L2 buffer is overwritten,
then a second one is read, leaving only clean lines).  Barrier + synchronize on both sides of the timed region; the max over
ranks is taken.  `e2e` repeats the primary step through the host-buffer entry
point fa_prefill_host with the inputs in pinned host memory: the host->device
copies of q/k/v, the kernels and the device->host copy of the output are all
inside the timed region (overlapped one sequence at a time by the library).

`--impl reference` times the fp64 CPU oracle (the only other implementation
of this method here) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "prefill attn TFLOP/s & paged-decode KV GB/s on 1 GB300, % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# the sources the profiled kernels (attn_tc_kernel, paged_decode_kernel, mask_classify_kernel) are built from
PROFILED_SOURCES = ("attn_tc.cu", "paged.cu", "cache_ops.cu", "common.cuh", "host_common.cuh")


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in PROFILED_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_tiled_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic():
    """Per-launch DRAM bytes from committed ncu summaries (lines 'traffic <kernel-key> <bytes>'),
    used only while the kernel sources are the ones the counters were taken on."""
    out, src = {}, None
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if os.path.exists(path):
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) == 2 and parts[0] == "source":
                    src = parts[1]
                if len(parts) == 3 and parts[0] == "traffic":
                    out[parts[1]] = float(parts[2])
    return out if src == kernel_source_hash() else {}


# ------------------------------------------------------------ distributed ---
def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, ws: int) -> float:
    if ws <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks ---
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------ timing ---
class Timer:
    """Per-step CUDA-event timing on the current stream with an L2 flush before each step."""

    def __init__(self, flush_bytes: int):
        # L2 flush: overwrite one 2x-L2 buffer, then read a second one, so the L2
        # holds only clean lines of neither operand when the step starts (a
        # write alone would leave dirty lines whose write-back the timed step
        # would pay for)
        self.flush = torch.empty(flush_bytes // 4, dtype=torch.float32, device="cuda")
        self.flush_rd = torch.ones(flush_bytes // 4, dtype=torch.float32, device="cuda")

    def flush_l2(self, i: int):
        # ~100+ us of GPU work: it also keeps the GPU busy while the host
        # enqueues the step, so no host-side gap falls between the events
        self.flush.fill_(float(i))
        self.flush_rd.sum()
        self.flush_rd.sum()

    def run(self, step, steps: int, warmup: int, ws: int, sampler: ClockSampler | None = None,
            min_warm_s: float = 0.0):
        from paged_kv_cache_tiled_gb300 import fattn as F
        t0 = time.time()
        i = 0
        while i < warmup or (time.time() - t0) < min_warm_s:
            self.flush_l2(i)
            step()
            i += 1
        torch.cuda.synchronize()
        if F.fa_get_error() != F.FA_OK:
            raise RuntimeError("device error during warm-up")
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        launches = 0
        barrier(ws)
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for i in range(steps):
            self.flush_l2(i)
            starts[i].record()
            step()
            ends[i].record()
            launches += F.fa_last_launch_count()
        torch.cuda.synchronize()
        barrier(ws)
        wall = time.perf_counter() - wall0
        if F.fa_get_error() != F.FA_OK:
            raise RuntimeError("device error during timed steps")
        times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        return float(np.mean(times)), launches, wall, times


def steady_state(steps, rounds: int, warmup: int, ws: int) -> float:
    """Mean time per step of back-to-back steps cycling over `steps` -- the
    same workload on distinct input sets whose total exceeds L2, so no step
    finds its inputs in L2 -- with one CUDA-event pair around all of them
    (rounds * len(steps) steps).  This is how a model runs attention layer
    after layer; it leaves out the fixed cost of an event pair around each
    single step, which the isolated per-step timing includes."""
    for _ in range(max(warmup, 3)):
        for st in steps:
            st()
    torch.cuda.synchronize()
    barrier(ws)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(rounds):
        for st in steps:
            st()
    b.record()
    b.synchronize()
    barrier(ws)
    return reduce_max(a.elapsed_time(b) / (rounds * len(steps)), ws)


# ---------------------------------------------------------------- workloads ---
def prefill_setup(case):
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    out = torch.empty_like(q)
    return q, k, v, out


def bench_prefill(F, timer, case, steps, warmup, ws, peaks, sampler=None, masked=False, min_warm_s=0.0,
                  causal=None):
    """`causal` overrides the case's flag (config 4 carries its causality in M)."""
    causal = case.causal if causal is None else causal
    q, k, v, out = prefill_setup(case)
    flops = W.attention_flops(case.T, case.T, case.d, case.B * case.Hq, True)
    if masked:
        M = case.mask.cuda()
        wsb = torch.empty(F.fa_prefill_masked_workspace_size(case.T), dtype=torch.uint8, device="cuda")

        def step():
            F.fa_prefill_masked(q, k, v, M, causal=False, scale=case.scale, out=out, ws=wsb)
    else:
        def step():
            F.fa_prefill(q, k, v, causal=causal, scale=case.scale, out=out)
    if sampler:
        sampler.start()
    ms, launches, wall, _ = timer.run(step, steps, warmup, ws, min_warm_s=min_warm_s)
    clocks = sampler.stop() if sampler else None
    ms = reduce_max(ms, ws)
    tflops = flops / (ms * 1e-3) / 1e12
    return dict(ms=ms, tflops=tflops, flops=flops, launches=launches, clocks=clocks, wall=wall,
                tensors=(q, k, v, out), step=step)


def paged_setup(F, p):
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    F.fa_cache_append(p.k_new.cuda(), p.v_new.cuda(), kc, vc, p.slot_mapping.cuda())
    torch.cuda.synchronize()
    return dict(q=p.q.cuda(), kc=kc, vc=vc, bt=p.block_table.cuda(), ctx=p.ctx_lens.cuda(), ql=p.q_lens.cuda(),
                out=torch.empty(p.total_q, p.Hq, p.d, dtype=torch.bfloat16, device="cuda"),
                ws=torch.empty(F.fa_paged_attn_workspace_size(p.num_seqs, p.max_blocks_per_seq, p.Hq, p.Hkv, p.d,
                                                              p.total_q), dtype=torch.uint8, device="cuda"))


def paged_bytes(p):
    """Algorithmic bytes: every cached K/V element of every context read once
    (per kv head), queries read once, outputs written once, block-table
    entries and lengths read once."""
    ctx = p.ctx_lens.numpy().astype(np.int64)
    kv = int(ctx.sum()) * p.Hkv * p.d * 2 * 2
    qo = 2 * p.total_q * p.Hq * p.d * 2
    tables = int(((ctx + 15) // 16).sum()) * 4 + 8 * p.num_seqs
    return kv + qo + tables, kv


def paged_flops(p):
    ctx = p.ctx_lens.numpy().astype(np.int64)
    ql = p.q_lens.numpy().astype(np.int64)
    tot = 0.0
    for c, q in zip(ctx, ql):
        tot += W.attention_flops(int(q), int(c), p.d, p.Hq, p.causal)
    return tot


def paged_issued_flops(p):
    """MMA work the chunked-prefill launch issues for the chunks that take the
    tensor-core path (whole 128x128 score tiles for both products), next to the
    decode rows' algorithmic work: each work entry covers 2*128/g tokens of one
    kv head when g = Hq/Hkv divides 128 (packed tiles), else 128 tokens of a
    head pair or 256 tokens of one head; it scans the 128-key tiles up to its
    last token's position."""
    g = p.Hq // p.Hkv
    pack = g in (2, 4, 8, 16)
    ent = 2 * (128 // g) if pack else (128 if g % 2 == 0 else 256)
    per_entry_rows = 2 * 128  # two 128-row slots per unit
    units_per_entry = p.Hkv if pack else (p.Hkv * (g // 2) if g % 2 == 0 else p.Hq)
    tot = 0.0
    for c, q in zip(p.ctx_lens.numpy().astype(np.int64), p.q_lens.numpy().astype(np.int64)):
        if q * g <= 16:
            tot += W.attention_flops(int(q), int(c), p.d, p.Hq, p.causal)
            continue
        for t0 in range(0, int(q), ent):
            last = min(int(q), t0 + ent)
            n_kt = -(-(int(c) - int(q) + last) // 128) if p.causal else -(-int(c) // 128)
            tot += units_per_entry * n_kt * 4.0 * per_entry_rows * 128 * p.d
    return tot


def bench_paged(F, timer, p, steps, warmup, ws, with_append=False):
    t = paged_setup(F, p)
    max_q = int(p.q_lens.max())
    if with_append:
        kn, vn, sm = p.k_new.cuda(), p.v_new.cuda(), p.slot_mapping.cuda()

    def step():
        if with_append:
            F.fa_cache_append(kn, vn, t["kc"], t["vc"], sm)
        F.fa_paged_attn(t["q"], t["kc"], t["vc"], t["bt"], t["ctx"], t["ql"], causal=p.causal, scale=p.scale,
                        out=t["out"], max_q_len=max_q, ws=t["ws"])
    ms, launches, wall, _ = timer.run(step, steps, warmup, ws)
    ms = reduce_max(ms, ws)
    return dict(ms=ms, launches=launches, wall=wall)


def bench_paged_fp8(F, timer, p, steps, warmup, ws, k_scale=0.0625, v_scale=0.03125):
    """Decode over the 8-bit cache: the case's context and new tokens are
    quantised into E4M3 caches first (outside the timed region)."""
    nb, Hkv, _, d = p.k_cache.shape
    kc = torch.zeros(nb, Hkv, 16, d, dtype=torch.uint8, device="cuda")
    vc = torch.zeros(nb, Hkv, d, 16, dtype=torch.uint8, device="cuda")
    used = np.unique(p.block_table.numpy()[p.block_table.numpy() >= 0])
    slots = torch.from_numpy((used[:, None] * 16 + np.arange(16)[None, :]).ravel().astype(np.int32)).cuda()
    ui = torch.from_numpy(used).long()
    F.fa_cache_append_fp8(p.k_cache[ui].permute(0, 2, 1, 3).reshape(-1, Hkv, d).cuda(),
                          p.v_cache[ui].permute(0, 2, 1, 3).reshape(-1, Hkv, d).cuda(), kc, vc, slots, k_scale, v_scale)
    F.fa_cache_append_fp8(p.k_new.cuda(), p.v_new.cuda(), kc, vc, p.slot_mapping.cuda(), k_scale, v_scale)
    q, bt, ctx, ql = p.q.cuda(), p.block_table.cuda(), p.ctx_lens.cuda(), p.q_lens.cuda()
    out = torch.empty_like(q)
    wsb = torch.empty(F.fa_paged_attn_workspace_size(p.num_seqs, p.max_blocks_per_seq, p.Hq, p.Hkv, p.d, p.total_q),
                      dtype=torch.uint8, device="cuda")
    mq = int(p.q_lens.max())

    def step():
        F.fa_paged_attn_fp8(q, kc, vc, k_scale, v_scale, bt, ctx, ql, causal=True, scale=p.scale, out=out,
                            max_q_len=mq, ws=wsb)
    ms, launches, wall, _ = timer.run(step, steps, warmup, ws)
    kv = int(p.ctx_lens.numpy().astype(np.int64).sum()) * p.Hkv * p.d * 2
    return dict(ms=reduce_max(ms, ws), launches=launches, wall=wall), kv


def bench_decode_graph(F, p, warmup, n_steps=200):
    """Host submission cost of a decode step: n_steps steps issued back to
    back (no L2 flush: this measures launch overhead, not bandwidth), once as
    eager calls through the binding (Python + C ABI + three kernel launches
    per step) and once as replays of the step captured by fa_decode_graph_*.
    Wall time per step (host clock around the loop, synchronised) and device
    time per step (CUDA events around the loop)."""
    t = paged_setup(F, p)
    kn, vn, sm = p.k_new.cuda(), p.v_new.cuda(), p.slot_mapping.cuda()
    mq = int(p.q_lens.max())

    def eager():
        F.fa_cache_append(kn, vn, t["kc"], t["vc"], sm)
        F.fa_paged_attn(t["q"], t["kc"], t["vc"], t["bt"], t["ctx"], t["ql"], causal=True, scale=p.scale,
                        out=t["out"], max_q_len=mq, ws=t["ws"])
    eager()
    g = F.DecodeGraph(t["q"], t["kc"], t["vc"], t["bt"], t["ctx"], t["ql"], t["out"], t["ws"], k_new=kn, v_new=vn,
                      slot_mapping=sm, scale=p.scale, max_q_len=mq)
    res = {}
    for name, fn in (("eager", eager), ("graph", g.replay)):
        for _ in range(max(3, warmup)):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        a.record()
        for _ in range(n_steps):
            fn()
        b.record()
        b.synchronize()
        wall = (time.perf_counter() - t0) / n_steps * 1e6
        res[name] = (wall, a.elapsed_time(b) / n_steps * 1e3)
    assert F.fa_get_error() == F.FA_OK
    kernels = g.kernel_count
    g.close()
    return {"workload": "config 3 decode step: append of the 64 new tokens + paged attention, "
                        f"{n_steps} steps submitted back to back (L2 not flushed)",
            "metric": "decode step wall time", "unit": "us", "higher_is_better": False,
            "value": res["graph"][0], "eager_wall_us": res["eager"][0], "graph_wall_us": res["graph"][0],
            "eager_device_us": res["eager"][1], "graph_device_us": res["graph"][1],
            "launch_overhead_share": (res["eager"][0] - res["graph"][0]) / res["eager"][0],
            "kernels_per_step": kernels}


def host_link(hq, hk, hv, hout, q, k, v, out, steps, ws):
    """The host link alone on the same buffers, no kernels: pinned host->device
    copies of q, k, v; the device->host copy of the output; and both
    directions issued at once on two streams -- the copy floor of the
    end-to-end step.  CUDA events, mean of `steps` repetitions after 3 warm-ups."""
    def timed(fn):
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(steps):
            fn()
        b.record()
        b.synchronize()
        return reduce_max(a.elapsed_time(b) / steps, ws)

    def h2d():
        for dst, src in ((q, hq), (k, hk), (v, hv)):
            dst.copy_(src, non_blocking=True)

    def d2h():
        hout.copy_(out, non_blocking=True)

    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def both():  # the two directions on two streams at once, joined back to the current stream
        cur = torch.cuda.current_stream()
        s_in.wait_stream(cur)
        s_out.wait_stream(cur)
        with torch.cuda.stream(s_in):
            h2d()
        with torch.cuda.stream(s_out):
            d2h()
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)
    nin = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    nout = hout.numel() * hout.element_size()
    t_in, t_out, t_both = timed(h2d), timed(d2h), timed(both)
    return {"h2d_gbs": nin / (t_in * 1e-3) / 1e9, "d2h_gbs": nout / (t_out * 1e-3) / 1e9, "floor_ms": t_both,
            "floor": "bare pinned copies of the same bytes, inputs in and output out concurrently on two streams, "
                     "no kernels"}


# ----------------------------------------------------------- cpu baseline ---
def oracle_sample_c2(batches: int = 1):
    """Bounded sample of config 2 for the CPU oracle: the first `batches`
    batch entries, all 12 heads, full T=2048 causal."""
    case = W.config2()
    q, k, v = case.q[:batches].contiguous(), case.k[:batches].contiguous(), case.v[:batches].contiguous()
    flops = W.attention_flops(case.T, case.T, case.d, batches * case.Hq, True)
    return case, q, k, v, flops


def time_oracle(q, k, v, case, threads):
    import oracle
    t0 = time.perf_counter()
    oracle.attention(q, k, v, True, case.scale, nthreads=threads)
    return time.perf_counter() - t0


def cpu_baseline(batches=1):
    case, q, k, v, flops = oracle_sample_c2(batches)
    threads = os.cpu_count() or 1
    dt = time_oracle(q, k, v, case, threads)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"config 2 rows of batch entries 0..{batches - 1} (all 12 heads, T=2048, causal): "
                      f"{flops / 1e9:.2f} GFLOP algorithmic in {dt:.2f} s on {threads} threads"}


def run_reference(args, ws, rank):
    if rank != 0:
        return
    case, q, k, v, flops = oracle_sample_c2(1)
    threads = os.cpu_count() or 1
    for _ in range(args.warmup):
        time_oracle(q, k, v, case, threads)
    times = [time_oracle(q, k, v, case, threads) for _ in range(args.steps)]
    ms = float(np.mean(times)) * 1e3
    val = flops / (ms * 1e-3) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "config 2 causal prefill B=4 T=2048 Hq=12 Hkv=2 d=128; each step = batch entry 0 "
                                   "(1/4 of the workload) through the fp64 CPU oracle"},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": "batch entry 0 of config 2 per step"},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile(F, args):
    """Only the chosen workload's step, args.warmup + args.steps times."""
    name = args.profile
    if name in ("c2", "c4", "c4causal", "c1"):
        if name == "c1":
            case, _ = W.config1()
            case = W.PrefillCase("c1", case.q.to(torch.bfloat16), case.k.to(torch.bfloat16),
                                 case.v.to(torch.bfloat16), True, case.scale)
        else:
            case = W.config2() if name == "c2" else W.config4()
        q, k, v, out = prefill_setup(case)
        if name == "c4":
            M = case.mask.cuda()
            wsb = torch.empty(F.fa_prefill_masked_workspace_size(case.T), dtype=torch.uint8, device="cuda")

            def step():
                F.fa_prefill_masked(q, k, v, M, causal=False, scale=case.scale, out=out, ws=wsb)
        else:
            def step():
                F.fa_prefill(q, k, v, causal=True, scale=case.scale, out=out)
    else:
        p = W.config3() if name == "c3" else W.config5()
        t = paged_setup(F, p)
        max_q = int(p.q_lens.max())

        def step():
            F.fa_paged_attn(t["q"], t["kc"], t["vc"], t["bt"], t["ctx"], t["ql"], causal=p.causal, scale=p.scale,
                            out=t["out"], max_q_len=max_q, ws=t["ws"])
    for _ in range(args.warmup + args.steps):
        step()
    torch.cuda.synchronize()
    st = F.fa_get_error()
    print(f"profile {name}: {args.warmup + args.steps} steps, status {F.status_string(st)}", flush=True)
    if st != F.FA_OK:
        sys.exit(1)


# -------------------------------------------------------------------- main ---
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--min-warm-s", type=float, default=1.5,
                    help="minimum warm-up time of the primary workload (clock sampling starts with it)")
    ap.add_argument("--profile", choices=["c1", "c2", "c3", "c4", "c4causal", "c5"], default=None,
                    help="run only this workload's step (warm-up + steps, no L2 flush, no JSON) for ncu captures")
    args = ap.parse_args()
    ws, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return

    torch.cuda.set_device(local)
    from paged_kv_cache_tiled_gb300 import build
    build.build()
    from paged_kv_cache_tiled_gb300 import fattn as F

    if args.profile:
        run_profile(F, args)
        return

    peaks, peak_src = load_peaks()
    traffic = profile_traffic()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    timer = Timer(max(2 * l2, 256 << 20))
    sampler = ClockSampler(local)

    # ---------------- primary: config 2 prefill
    c2 = W.config2()
    res = bench_prefill(F, timer, c2, args.steps, args.warmup, ws, peaks, sampler=sampler,
                        min_warm_s=args.min_warm_s)
    tc_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    roof = {"bound": "tensor", "achieved": res["tflops"], "peak": tc_peak, "unit": "TFLOP/s",
            "frac": res["tflops"] / tc_peak, "traffic": traffic.get("attn_tc_dense_c2"),
            "kernel": "attn_tc_kernel<128, dense>", "peak_source": f"{peak_src} bf16 burst",
            "algorithmic_flops_per_launch": res["flops"]}

    # ---------------- steady state: back-to-back steps over 4 distinct input sets (4 x 58.7 MB > L2)
    c2_sets = [prefill_setup(c2) for _ in range(4)]

    def c2_step(t):
        return lambda: F.fa_prefill(t[0], t[1], t[2], causal=True, scale=c2.scale, out=t[3])
    ss_ms = steady_state([c2_step(t) for t in c2_sets], max(1, args.steps // 4), args.warmup, ws)
    ss_tflops = res["flops"] / (ss_ms * 1e-3) / 1e12
    steady = {"ms_per_step": ss_ms, "value": ss_tflops, "unit": "TFLOP/s", "frac": ss_tflops / tc_peak,
              "how": "back-to-back steps cycling over 4 distinct input sets (235 MB, more than L2), one CUDA-event "
                     "pair around all of them; no L2 flush needed"}
    del c2_sets

    # ---------------- e2e through host buffers
    q, k, v, out = res["tensors"]
    hq, hk, hv = (t.cpu().pin_memory() for t in (c2.q, c2.k, c2.v))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e_step():  # host-buffer entry point: per-sequence copies overlapped with the kernels
        F.fa_prefill_host(hq, hk, hv, hout, q, k, v, out, causal=True, scale=c2.scale)
    e_ms, _, _, _ = timer.run(e2e_step, args.steps, args.warmup, ws)
    e_ms = reduce_max(e_ms, ws)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = hout.numel() * hout.element_size()
    link = host_link(hq, hk, hv, hout, q, k, v, out, args.steps, ws)
    e2e = {"value": res["flops"] / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e_ms, "api": "fa_prefill_host (pinned host buffers)",
           **link, "frac_of_floor": link["floor_ms"] / e_ms}

    line = {"metric": METRIC, "value": res["tflops"] * ws, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: seeded N(0,1) bf16 inputs with the shapes of config 2 (no weights needed)",
            "config": {"workload": "config 2: causal prefill B=4 T=2048 Hq=12 Hkv=2 d=128 bf16, scale 1/sqrt(128)",
                       "l2": "flushed before every timed step, outside the events: a 2x-L2 buffer is overwritten, then a second 2x-L2 buffer is read (clean L2)",
                       "replicas": ws},
            "roofline": roof, "steady_state": steady, "e2e": e2e, "gpu_launches": res["launches"],
            "clocks": res["clocks"]}

    # ---------------- secondary workloads
    if not args.no_secondary:
        sec = []
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        # config 3: paged decode
        c3 = W.config3()
        r3 = bench_paged(F, timer, c3, args.steps, args.warmup, ws)
        b3, kv3 = paged_bytes(c3)
        gbs = b3 / (r3["ms"] * 1e-3) / 1e9
        # steady state: 4 copies of the cache pool (each step reads 128 MB of a different copy)
        t3 = paged_setup(F, c3)
        pools = [(t3["kc"], t3["vc"])] + [(t3["kc"].clone(), t3["vc"].clone()) for _ in range(3)]

        def c3_step(kc, vc):
            return lambda: F.fa_paged_attn(t3["q"], kc, vc, t3["bt"], t3["ctx"], t3["ql"], causal=True, scale=c3.scale,
                                           out=t3["out"], max_q_len=1, ws=t3["ws"])
        ss3_ms = steady_state([c3_step(*pp) for pp in pools], max(1, args.steps // 4), args.warmup, ws)
        ss3_gbs = b3 / (ss3_ms * 1e-3) / 1e9
        del pools, t3
        sec.append({"workload": "config 3: paged decode, 64 seqs ctx U[128,4096], Hq=12 Hkv=2 d=128, 16-token blocks",
                    "metric": "paged-decode KV GB/s", "value": gbs, "unit": "GB/s", "ms_per_step": r3["ms"],
                    "kv_bytes": kv3, "algorithmic_bytes": b3, "gpu_launches": r3["launches"],
                    "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                                 "traffic": traffic.get("paged_decode_c3"), "peak_source": f"{peak_src} hbm copy",
                                 "kernel": "paged_decode_kernel<128> + paged_merge_kernel<128>"},
                    "steady_state": {"ms_per_step": ss3_ms, "value": ss3_gbs, "unit": "GB/s", "frac": ss3_gbs / hbm,
                                     "how": "back-to-back decode calls cycling over 4 copies of the cache pool "
                                            "(each call reads 128 MB of a different copy), one CUDA-event pair "
                                            "around all of them"}})
        del c3
        # config 4: long masked prefill (and the same problem through the causal flag)
        steps4 = max(3, min(args.steps, 10))
        c4 = W.config4()
        r4 = bench_prefill(F, timer, c4, steps4, min(args.warmup, 3), ws, peaks, masked=True)
        r4c = bench_prefill(F, timer, c4, steps4, min(args.warmup, 3), ws, peaks, causal=True)
        tc_sus = float(peaks.get("bf16_tflops_sustained", tc_peak))
        for r, name, tkey in ((r4, "additive mask M (-inf above diagonal) via fa_prefill_masked", "attn_tc_masked_c4"),
                              (r4c, "causal flag via fa_prefill", "attn_tc_dense_c4")):
            sec.append({"workload": f"config 4: long prefill B=1 T=16384 Hq=32 Hkv=8 d=128, {name}",
                        "metric": "prefill attn TFLOP/s", "value": r["tflops"], "unit": "TFLOP/s",
                        "ms_per_step": r["ms"], "gpu_launches": r["launches"],
                        "roofline": {"bound": "tensor", "achieved": r["tflops"], "peak": tc_peak, "unit": "TFLOP/s",
                                     "frac": r["tflops"] / tc_peak,
                                     "traffic": traffic.get(tkey) if tkey else None,
                                     "peak_source": f"{peak_src} bf16 burst (the launch is timed alone)",
                                     "frac_of_sustained_peak": r["tflops"] / tc_sus}})
        # the mask-class pass alone: one read of the 1.07 GB mask
        M4 = c4.mask.cuda()
        cls4 = torch.empty(((c4.T + 127) // 128, (c4.T + 127) // 128), dtype=torch.uint8, device="cuda")

        def mask_step():
            F.fa_mask_tile_classes(M4, out=cls4)
        mms, ml, _, _ = timer.run(mask_step, steps4, min(args.warmup, 3), ws)
        mms = reduce_max(mms, ws)
        mbytes = M4.numel() * 4 + cls4.numel()
        mgbs = mbytes / (mms * 1e-3) / 1e9
        sec.append({"workload": "config 4 mask-class pass alone: fp32 M [16384, 16384] -> 128x128 tile classes",
                    "metric": "mask pass GB/s", "value": mgbs, "unit": "GB/s", "ms_per_step": mms,
                    "gpu_launches": ml, "algorithmic_bytes": mbytes,
                    "roofline": {"bound": "hbm", "achieved": mgbs, "peak": float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
                                 "unit": "GB/s", "frac": mgbs / float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
                                 "traffic": traffic.get("mask_classify_c4"), "peak_source": f"{peak_src} hbm copy",
                                 "kernel": "mask_classify_kernel"}})
        del c4, r4, r4c, M4, cls4
        torch.cuda.empty_cache()
        # config 5: append + chunked prefill over the paged cache
        c5 = W.config5()
        r5 = bench_paged(F, timer, c5, args.steps, args.warmup, ws, with_append=True)
        f5 = paged_flops(c5)
        b5, kv5 = paged_bytes(c5)
        tf5 = f5 / (r5["ms"] * 1e-3) / 1e12
        t_bound = max(f5 / (tc_peak * 1e12), b5 / (hbm * 1e9))
        sec.append({"workload": "config 5: append + chunked prefill, 16 seqs ctx U[0,8192] + chunk U[1,512], "
                                "Hq=32 Hkv=8 d=128",
                    "metric": "prefill attn TFLOP/s", "value": tf5, "unit": "TFLOP/s", "ms_per_step": r5["ms"],
                    "gpu_launches": r5["launches"], "algorithmic_flops": f5, "algorithmic_bytes": b5,
                    "issued_over_algorithmic_flops": paged_issued_flops(c5) / f5,
                    "roofline": {"bound": "tensor" if f5 / (tc_peak * 1e12) > b5 / (hbm * 1e9) else "hbm",
                                 "achieved": tf5, "peak": tc_peak, "unit": "TFLOP/s",
                                 "frac": t_bound / (r5["ms"] * 1e-3), "traffic": traffic.get("attn_tc_paged_c5"),
                                 "kernel": "attn_tc_kernel<128, paged> (traffic: that launch alone)",
                                 "note": "frac = max(F/P_tc, B/BW) / measured time"}})
        # rotary embedding fused with the append, at config 5's chunk size
        rc = W.rope_case(21, 4096, 32, 8, 128, num_blocks=20000, max_pos=8704)
        rq, rk, rv = rc.q.cuda(), rc.k.cuda(), rc.v.cuda()
        rpos, rcs, rsm = rc.positions.cuda(), rc.cos_sin.cuda(), rc.slot_mapping.cuda()
        rkc = torch.zeros(rc.num_blocks, 8, 16, 128, dtype=torch.bfloat16, device="cuda")
        rvc, rqo = torch.zeros_like(rkc), torch.empty_like(rq)

        def rope_step():
            F.fa_cache_append_rope(rq, rk, rv, rpos, rcs, rkc, rvc, rsm, q_out=rqo)
        rms, rl, _, _ = timer.run(rope_step, args.steps, args.warmup, ws)
        rms = reduce_max(rms, ws)
        rbytes = 2 * rq.numel() * 2 + 2 * (rk.numel() + rv.numel()) * 2 + rc.N * (128 * 4 + 8)
        rgbs = rbytes / (rms * 1e-3) / 1e9
        sec.append({"workload": "rotary embedding of q and k fused with the cache append: 4096 tokens, Hq=32 Hkv=8 "
                                "d=128, positions U[0,8704), slots in a 20000-block pool",
                    "metric": "fused append GB/s", "value": rgbs, "unit": "GB/s", "ms_per_step": rms,
                    "gpu_launches": rl, "algorithmic_bytes": rbytes,
                    "roofline": {"bound": "hbm", "achieved": rgbs, "peak": hbm, "unit": "GB/s", "frac": rgbs / hbm,
                                 "traffic": None, "peak_source": f"{peak_src} hbm copy",
                                 "kernel": "rope_append_kernel<false>"}})
        del rq, rk, rv, rkc, rvc, rqo
        # config 3 over the 8-bit (E4M3) cache: half the KV bytes
        c3 = W.config3()
        r8, kv8 = bench_paged_fp8(F, timer, c3, args.steps, args.warmup, ws)
        gbs8 = kv8 / (r8["ms"] * 1e-3) / 1e9
        sec.append({"workload": "config 3 over the 8-bit E4M3 cache (k_scale 1/16, v_scale 1/32): paged decode, 64 seqs "
                                "ctx U[128,4096], Hq=12 Hkv=2 d=128",
                    "metric": "paged-decode KV GB/s", "value": gbs8, "unit": "GB/s", "ms_per_step": r8["ms"],
                    "kv_bytes": kv8, "gpu_launches": r8["launches"],
                    "roofline": {"bound": "hbm", "achieved": gbs8, "peak": hbm, "unit": "GB/s", "frac": gbs8 / hbm,
                                 "traffic": None, "peak_source": f"{peak_src} hbm copy",
                                 "kernel": "paged_decode_kernel<128, true> + paged_merge_kernel<128>"}})
        del c3
        # config 3 decode step (append of each sequence's new token + paged
        # attention), submitted back to back: eager calls vs one CUDA-graph replay
        sec.append(bench_decode_graph(F, W.config3(), args.warmup))
        line["secondary"] = sec

    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(1)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
