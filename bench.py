"""Benchmark: one decode step of a paged-KV GQA attention layer, Qwen3-4B shape.

A step is the whole hot path on one batch, as one call:
``pkv_decode_append_attention`` writes the 64 new tokens' K/V through the page
table and runs the split-KV decode over the pages including them, then the
LSE merge (two kernels). The two-call step (``pkv_append``, then
``pkv_decode_attention``) and the decode call alone are timed beside it.
Workload: B=64, Hq=32, Hkv=8, D=128,
page 128, keys attended uniform in [512, 1024], sequential pages (a fresh
batch's allocation, the contiguous fast path); a second line of numbers is
taken with randomly permuted pages, and the packed document-causal prefill
(64 documents, lengths uniform in [64, 1024]) is timed alongside.

Inputs are seeded synthetic tensors (the pages measured real prompts of a
public math dataset; these stand in with the same shapes and lengths).
Timing: CUDA events on the launching stream; the K timed steps rotate over
enough independent pool sets that the KV read each step (~201 MB) comes from
HBM, not L2. Prints one JSON line on rank 0.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn KV GB/s & % of HBM peak; tokens/s/layer at B=64 Qwen3-4B shape"
UNIT = "GB/s"
WORKLOAD = ("qwen3_b64_decode: B=64, Hq=32, Hkv=8, D=128, page_size=128, keys U[512,1024], "
            "sequential pages, seed 0; step = one fused call: append 64 tokens + split-KV "
            "decode + merge")
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 126 * 1024 * 1024


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def captured_traffic(key: str):
    """DRAM bytes per call from the committed ncu capture (profiles/traffic.json),
    or None when any source the kernels are built from has changed since that
    capture (sha256 over the listed sources, in order)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[key]
        m = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                m.update(f.read())
        if m.hexdigest() != rec["sources_sha256"]:
            return None
        return int(rec["dram_bytes_per_call"])
    except Exception:
        return None


def step_bytes(case) -> int:
    """Algorithmic bytes of one fused decode step: the decode launch's bytes
    plus the append's (each live row's new K and V read once and written
    once into the pool)."""
    live = int((case.batch_idx != 0).sum())
    return decode_bytes(case) + live * case.num_kv_heads * case.head_dim * 2 * 2 * 2


def decode_bytes(case) -> int:
    """Algorithmic bytes of one decode launch: K and V rows of every attended
    key (all kv heads), q in, out and lse out, the page-table entries walked,
    batch_idx and seq_lens."""
    d = case.head_dim
    hkv, hq, B = case.num_kv_heads, case.num_q_heads, case.batch
    live = case.batch_idx != 0
    lens = case.seq_lens[live].long()
    kv = int(lens.sum()) * hkv * d * 2 * 2
    pages = int(((lens + case.page_size - 1) // case.page_size).sum()) * 4
    return kv + B * hq * d * 2 * 2 + B * hq * 4 + pages + B * 8


def append_bytes(case) -> int:
    n = int((case.batch_idx != 0).sum())
    return n * case.num_kv_heads * case.head_dim * 2 * 2 * 2 + case.batch * 8 + n * 4


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


_ORACLE_CHILD = """
import json, multiprocessing as mp, os, statistics, sys, time
sys.path.insert(0, ROOT)
import oracle.paged_attention as orc
from paged_kv_gqa_pkv_gb300 import workloads as W
from paged_kv_gqa_pkv_gb300.workloads import bf16_bits
c = (W.long_context_decode(0) if WORKLOAD == "long_context_decode"
     else W.qwen3_b64_decode(0, permute=False))
kb, vb = bf16_bits(c.k_pool), bf16_bits(c.v_pool)
tab, bi, ip, sl = (c.page_table.numpy(), c.batch_idx.numpy(), c.input_pos.numpy(),
                   c.seq_lens.numpy())
kn, vn, q = bf16_bits(c.k_new), bf16_bits(c.v_new), bf16_bits(c.q)
row_kv = [int(n) * c.num_kv_heads * c.head_dim * 4 for n in sl]
res = {"host_cpu_count": os.cpu_count()}
if MODE == "full":
    # whole step on one core: append of the new tokens, then decode of all rows
    times = []
    for _ in range(REPS):
        t0 = time.perf_counter()
        k2, v2, _ = orc.append(kb, vb, tab, kn, vn, bi, ip, c.page_size)
        orc.decode_attention(q, k2, v2, tab, bi, sl, c.page_size, c.scale)
        times.append(time.perf_counter() - t0)
    res.update(seconds=statistics.median(times), kv_bytes=sum(row_kv), cores=1)
else:
    # decode rows spread over a pool of processes, one row per task; the
    # pools already hold the appended tokens (the append is done once, untimed)
    k2, v2, _ = orc.append(kb, vb, tab, kn, vn, bi, ip, c.page_size)

    def one_row(r):
        orc.decode_attention(q, k2, v2, tab, bi, sl, c.page_size, c.scale, rows=[r])
        return None

    # this process has never touched a GPU (CUDA_VISIBLE_DEVICES is empty):
    # fork shares the pools with the workers without copying them
    procs = NPROC or os.cpu_count() or 1
    with mp.get_context("fork").Pool(procs) as pool:
        pool.map(one_row, ROWS[:procs], chunksize=1)        # warm the workers
        if MODE == "parallel":
            times = []
            for _ in range(REPS):
                t0 = time.perf_counter()
                pool.map(one_row, ROWS, chunksize=1)
                times.append(time.perf_counter() - t0)
            res.update(seconds=statistics.median(times),
                       kv_bytes=sum(row_kv[r] for r in ROWS), cores=procs)
        else:
            # reference arm: STEPS timed steps after WARMUP, each the decode of
            # PER_STEP rows (a block of rows, in turn)
            tot_t, tot_b = 0.0, 0
            for i in range(WARMUP + STEPS):
                blk = [ROWS[(i * PER_STEP + j) % len(ROWS)] for j in range(PER_STEP)]
                t0 = time.perf_counter()
                pool.map(one_row, blk, chunksize=1)
                dt = time.perf_counter() - t0
                if i >= WARMUP:
                    tot_t += dt
                    tot_b += sum(row_kv[r] for r in blk)
            res.update(seconds=tot_t, kv_bytes=tot_b, steps=STEPS, cores=procs)
print(json.dumps(res))
"""


def run_oracle_child(mode: str, workload: str = "qwen3_b64_decode", reps: int = 5,
                     rows=None, nproc: int = 0, steps: int = 0, warmup: int = 0,
                     per_step: int = 0):
    """Runs the oracle, as it stands, in a child process started by
    subprocess (never forked from a process that touched CUDA) with one BLAS
    thread per process. ``full``: the whole step on one core. ``parallel``:
    decode of ``rows`` over a pool of ``nproc`` processes (0: all host
    cores). ``steps``: the reference arm's timed steps."""
    code = (f"ROOT={ROOT!r}\nMODE={mode!r}\nWORKLOAD={workload!r}\nREPS={reps}\n"
            f"ROWS={list(rows or [])!r}\nNPROC={nproc}\nSTEPS={steps}\nWARMUP={warmup}\n"
            f"PER_STEP={per_step}\n") + _ORACLE_CHILD
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1",
               MKL_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=3600)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return d["kv_bytes"] / d["seconds"] / 1e9, d


def run_reference(args):
    """Reference arm: the float64 CPU oracle on the same workload, metric and
    unit, on all host cores (one process per core, one row per task). Each
    step decodes a block of rows of the 64 (all 64 when the run is short;
    16 per step for runs of more than 1000 steps, so the default run stays
    within minutes); the append is done once before timing."""
    world, rank, _ = _dist()
    if rank != 0:
        return
    per_step = 64 if args.steps + args.warmup <= 1000 else 16
    value, d = run_oracle_child("steps", rows=list(range(64)), steps=args.steps,
                                warmup=args.warmup, per_step=per_step)
    sample = (f"decode of {per_step} of the 64 rows per step (blocks in turn), one row per "
              f"task on {d['cores']} processes; append done once before timing")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": d["seconds"] / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": d["cores"], "kind": "oracle",
                             "sample": sample, "host_cpu_count": d["host_cpu_count"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_pkv(args):
    import torch
    from paged_kv_gqa_pkv_gb300 import binding
    from paged_kv_gqa_pkv_gb300 import build as _b
    from paged_kv_gqa_pkv_gb300 import workloads as W

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        _b.build()
    if world > 1:
        dist.barrier()
    binding.load_library()
    hbm_peak, bf16_peak, peak_kind = _peaks()

    def make_sets(case, n_sets):
        sets = []
        for _ in range(n_sets):
            sets.append(dict(
                kp=case.k_pool.to(dev), vp=case.v_pool.to(dev), pt=case.page_table.to(dev),
                q=case.q.to(dev), kn=case.k_new.to(dev), vn=case.v_new.to(dev),
                bi=case.batch_idx.to(dev), ip=case.input_pos.to(dev),
                sl=case.seq_lens.to(dev)))
        return sets

    def kv_set_bytes(case):
        return 2 * case.k_pool.numel() * 2

    def decode_rig(case, warmup):
        """Device copies of `case` (enough pool sets that each step's KV comes
        from HBM), the call bodies (append, decode, fused step) on set i mod
        n_sets, and a graph-capture helper; the calls are run eagerly first."""
        import types
        n_sets = max(2, math.ceil(2 * L2_BYTES / kv_set_bytes(case)) + 1)
        sets = make_sets(case, n_sets)
        B, hq = case.batch, case.num_q_heads
        ws_bytes = binding.pkv_decode_workspace_size(sets[0]["kp"], sets[0]["pt"],
                                                     case.page_size, B, hq)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        out = torch.empty((B, hq, 128), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, hq), dtype=torch.float32, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)

        def append(i):
            s = sets[i % n_sets]
            binding.pkv_append(s["kp"], s["vp"], s["pt"], s["kn"], s["vn"], s["bi"], s["ip"],
                               case.page_size, dev_err=err)

        def decode(i):
            s = sets[i % n_sets]
            binding.pkv_decode_attention(s["kp"], s["vp"], s["pt"], s["q"], s["bi"], s["sl"],
                                         case.page_size, case.scale, out=out, lse=lse,
                                         workspace=ws, dev_err=err)

        def fused(i):
            s = sets[i % n_sets]
            binding.pkv_decode_append_attention(s["kp"], s["vp"], s["pt"], s["q"], s["kn"],
                                                s["vn"], s["bi"], s["sl"], case.page_size,
                                                case.scale, out=out, lse=lse, workspace=ws,
                                                dev_err=err)

        def capture(n, body):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(n):
                    body(i)
            return g

        for i in range(max(warmup, n_sets)):   # eager warm-up (first-call set-up)
            append(i)
            decode(i)
            fused(i)
        torch.cuda.synchronize()
        return types.SimpleNamespace(n_sets=n_sets, sets=sets, append=append, decode=decode,
                                     fused=fused, capture=capture, err=err)

    def check_err(err, what):
        if int(err.item()) != 0:
            raise RuntimeError(f"device error bits {int(err.item()):#x} in {what}")

    def device_lead_in():
        """About half a millisecond of device work ahead of a start event: by
        the time the event fires, the host has submitted the graph launches
        that follow, so the timed region holds the steps' device time and not
        the host's submission of a graph of ~100-200 kernels (~50 us on an
        idle GPU). A serving loop submits the next replay while the current
        one runs; the end-to-end figure keeps the host's share."""
        torch.cuda._sleep(1_000_000)

    def replay_ms(g, n_calls, reps):
        """Median per-call ms over `reps` timed replays of graph g (n_calls
        calls each); the graph has been launched before."""
        ms = []
        for _ in range(reps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            device_lead_in()
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b) / n_calls)
        return ms

    def timed_decode_config(case, reps=7):
        """The fused step and the decode call alone on `case`, each from
        replays of a graph of 48-odd calls over rotating pool sets (KV from
        HBM); each graph is launched once untimed; medians of `reps`."""
        rig = decode_rig(case, 3)
        per_graph = rig.n_sets * max(1, 48 // rig.n_sets)
        step_g = rig.capture(per_graph, rig.fused)
        dec_g = rig.capture(per_graph, rig.decode)
        step_g.replay()
        dec_g.replay()
        torch.cuda.synchronize()
        step_ms = statistics.median(replay_ms(step_g, per_graph, reps))
        dec_ms = statistics.median(replay_ms(dec_g, per_graph, reps))
        check_err(rig.err, case.name)
        del step_g, dec_g, rig
        torch.cuda.empty_cache()
        live = int((case.batch_idx != 0).sum())
        db, sb = decode_bytes(case), step_bytes(case)
        return {"workload": case.name, "batch": case.batch, "live_rows": live,
                "kv_tokens": int(case.seq_lens[case.batch_idx != 0].long().sum()),
                "step_us": step_ms * 1e3, "step_gbs": sb / (step_ms * 1e-3) / 1e9,
                "decode_call_us": dec_ms * 1e3,
                "decode_call_gbs": db / (dec_ms * 1e-3) / 1e9,
                "frac_of_measured": db / (dec_ms * 1e-3) / 1e9 / hbm_peak,
                "frac_of_nominal_8TBs": db / (dec_ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
                "tokens_per_s_per_layer": live / (step_ms * 1e-3)}

    def timed_decode(case, steps, warmup):
        """Times `steps` decode steps (the fused append + decode call) replayed
        from CUDA graphs, rotating over pool sets so each step's KV comes from
        HBM; a second graph of decode calls alone gives the decode call's
        duration, and a third the two-call step (append, then decode)."""
        rig = decode_rig(case, warmup)
        n_sets, append, decode, fused, capture, err = (rig.n_sets, rig.append, rig.decode,
                                                       rig.fused, rig.capture, rig.err)

        per_graph = n_sets * max(1, 96 // n_sets)
        step_g = capture(per_graph, fused)
        tail = steps % per_graph
        tail_g = capture(tail, fused) if tail else None
        dec_g = capture(per_graph, decode)
        two_g = capture(per_graph, lambda i: (append(i), decode(i)))
        # every graph the timed region replays is launched untimed first, so
        # no first launch of a freshly instantiated graph is timed
        for _ in range(max(1, warmup // per_graph)):
            step_g.replay()
            if tail_g is not None:
                tail_g.replay()
            dec_g.replay()
            two_g.replay()
        torch.cuda.synchronize()

        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        with ClockSampler(local) as clk:
            device_lead_in()
            t0.record()
            for _ in range(steps // per_graph):
                step_g.replay()
            if tail_g is not None:
                tail_g.replay()
            t1.record()
            torch.cuda.synchronize()
        total_ms = t0.elapsed_time(t1)

        # decode calls alone and the two-call step, same graph shape; several
        # timed replays each
        reps = max(3, min(50, steps // per_graph))
        dec_ms, two_ms = [], []
        for _ in range(reps):
            dec_ms += replay_ms(dec_g, per_graph, 1)
            two_ms += replay_ms(two_g, per_graph, 1)
        check_err(err, "the decode step")
        del step_g, tail_g, dec_g, two_g, rig
        torch.cuda.empty_cache()
        dec_sorted = sorted(dec_ms)
        return dict(total_ms=total_ms, dec_ms=statistics.median(dec_ms),
                    two_call_ms=statistics.median(two_ms),
                    dec_p10=dec_sorted[len(dec_ms) // 10],
                    dec_p90=dec_sorted[(9 * len(dec_ms)) // 10],
                    clocks=clk.summary(), n_sets=n_sets, set_bytes=kv_set_bytes(case),
                    per_graph=per_graph)

    def e2e_decode(case, steps, warmup, staged=True, zero_copy=False):
        """Same step through the public binding with pinned host buffers: each
        step copies its inputs host->device and brings the result to the host.
        With zero_copy the step's inputs are not copied: the fused call reads
        them from the pinned host buffer over the host link (q's rows by
        cp.async, the rest by plain loads), and the page table, cache state
        like the pools, stays on the device.
        The inputs are laid out the way a serving loop would: q, the new K/V,
        batch_idx, seq_lens and the page table in one pinned host buffer and
        one device buffer (each tensor a 256-byte aligned view). A step is one
        host->device copy of that buffer (``staged``: pkv_stage_from_host, the
        SMs' own loads; else a copy-engine copy) and the fused call, which
        writes out and lse straight into one pinned host buffer (the decode
        entry points allow host memory for them); captured once as a CUDA
        graph and replayed, then a stream sync on the host."""
        s = make_sets(case, 1)[0]
        B, hq = case.batch, case.num_q_heads

        def staged(parts, device, pin=False):
            offs, n = {}, 0
            for k, t in parts:
                offs[k] = n
                n += (t.numel() * t.element_size() + 255) // 256 * 256
            buf = torch.zeros(n, dtype=torch.uint8, device=device)
            if pin:
                buf = buf.pin_memory()
            views = {k: buf[offs[k]:offs[k] + t.numel() * t.element_size()].view(t.dtype)
                     .view(t.shape) for k, t in parts}
            return buf, views

        ins = [("q", case.q), ("kn", case.k_new), ("vn", case.v_new),
               ("bi", case.batch_idx), ("sl", case.seq_lens), ("pt", case.page_table)]
        if zero_copy:
            # the page table is cache state that stays on the device; the
            # step's inputs stay in pinned host memory and the kernels read
            # them over the host link
            ins = ins[:-1]
        host_in, hv = staged(ins, "cpu", pin=True)
        for k, t in ins:
            hv[k].copy_(t)
        dev_in, dv = staged(ins, dev)
        if zero_copy:
            dv = dict(hv)
            dv["pt"] = case.page_table.to(dev)
        outs = [("out", torch.empty((B, hq, 128), dtype=torch.bfloat16)),
                ("lse", torch.empty((B, hq), dtype=torch.float32))]
        host_out, ov = staged(outs, "cpu", pin=True)
        ws = torch.empty(binding.pkv_decode_workspace_size(s["kp"], dv["pt"], case.page_size,
                                                           B, hq),
                         dtype=torch.uint8, device=dev)
        h2d = host_in.numel()
        d2h = host_out.numel()

        es = torch.cuda.Stream(device=dev)

        def body():
            if zero_copy:
                pass
            elif staged:
                binding.pkv_stage_from_host(dev_in, host_in)
            else:
                dev_in.copy_(host_in, non_blocking=True)
            binding.pkv_decode_append_attention(s["kp"], s["vp"], dv["pt"], dv["q"], dv["kn"],
                                                dv["vn"], dv["bi"], dv["sl"], case.page_size,
                                                case.scale, out=ov["out"], lse=ov["lse"],
                                                workspace=ws)

        # the step (copy in, fused call, copy out) is captured once as a graph,
        # as a serving loop replays its decode step; every replay still moves
        # the inputs and the result across and the host waits for them
        torch.cuda.synchronize()
        with torch.cuda.stream(es):
            for _ in range(3):
                body()
            es.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=es):
                body()
        torch.cuda.synchronize()

        def step():
            g.replay()
            es.synchronize()

        with torch.cuda.stream(es):
            for _ in range(warmup):
                step()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            t0.record(es)
            for _ in range(steps):
                step()
            t1.record(es)
            torch.cuda.synchronize()
        return t0.elapsed_time(t1) / steps, h2d, d2h

    def timed_prefill(reps):
        """Packed prefill of the 64-document workload: the append of its k/v
        into the pages and the tcgen05 attention, each timed with CUDA events
        over `reps` back-to-back calls (the inputs, ~430 MB, exceed L2)."""
        c = W.packed_prefill(0)
        q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
        bi, ip = c.batch_idx.to(dev), c.input_pos.to(dev)
        kp, vp, pt = c.k_pool.to(dev), c.v_pool.to(dev), c.page_table.to(dev)
        out = torch.empty_like(q)
        lse = torch.empty((c.n_tokens, c.num_q_heads), dtype=torch.float32, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        for _ in range(3):
            binding.pkv_append(kp, vp, pt, k, v, bi, ip, c.page_size, dev_err=err)
            binding.pkv_prefill_attention(q, k, v, bi, ip, c.scale, out=out, lse=lse,
                                          dev_err=err)
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record()
        for _ in range(reps):
            binding.pkv_append(kp, vp, pt, k, v, bi, ip, c.page_size, dev_err=err)
        ev[1].record()
        for _ in range(reps):
            binding.pkv_prefill_attention(q, k, v, bi, ip, c.scale, out=out, lse=lse,
                                          dev_err=err)
        ev[2].record()
        torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise RuntimeError(f"device error bits {int(err.item()):#x} in prefill")
        app_us = ev[0].elapsed_time(ev[1]) / reps * 1e3
        att_us = ev[1].elapsed_time(ev[2]) / reps * 1e3
        # the same append with k_norm and the rotary embedding applied to K
        # (Qwen3's rope theta 1e6; a seeded k_norm weight)
        cos, sin = W.rope_tables(int(c.input_pos.max()) + 1)
        cos, sin = cos.to(dev), sin.to(dev)
        knw = (torch.rand(c.head_dim, generator=torch.Generator().manual_seed(0)) * 1.75
               + 0.25).to(dev)
        for _ in range(3):
            binding.pkv_append_rope(kp, vp, pt, k, v, bi, ip, c.page_size, cos, sin,
                                    k_norm_weight=knw, dev_err=err)
        torch.cuda.synchronize()
        er = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        er[0].record()
        for _ in range(reps):
            binding.pkv_append_rope(kp, vp, pt, k, v, bi, ip, c.page_size, cos, sin,
                                    k_norm_weight=knw, dev_err=err)
        er[1].record()
        torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise RuntimeError(f"device error bits {int(err.item()):#x} in the rope append")
        rope_us = er[0].elapsed_time(er[1]) / reps * 1e3
        flops = 4.0 * c.head_dim * c.num_q_heads * c.info["pairs"]
        tf = flops / (att_us * 1e-6) / 1e12
        return {"workload": f"packed_prefill: 64 documents, lengths U[64,1024], "
                            f"T={c.n_tokens}, Hq=32, Hkv=8, D=128, seed 0",
                "attention_call_us": att_us, "algorithmic_flops": flops,
                "tflops": tf, "bound": "tensor", "peak_tflops": bf16_peak,
                "frac": tf / bf16_peak, "peak_kind": peak_kind,
                "traffic": captured_traffic("prefill_call"),
                "append_call_us": app_us,
                "append_gbs": (c.n_tokens * c.num_kv_heads * c.head_dim * 2 * 4)
                / (app_us * 1e-6) / 1e9,
                "append_rope_knorm_call_us": rope_us,
                "append_rope_knorm_traffic": captured_traffic("append_rope_call"),
                "append_rope_knorm_gbs": (c.n_tokens * c.num_kv_heads * c.head_dim * 2 * 4)
                / (rope_us * 1e-6) / 1e9}

    def timed_chunked_prefill(reps, n_decode=0, page_size=128):
        """Chunked prefill over the paged cache: 16 chunks of 512 tokens over
        prefixes U[512, 4096] (T=8192), pages permuted, plus `n_decode` decode
        tokens for a mixed step. The chunk K/V are appended once; the tcgen05
        paged attention is timed with CUDA events over `reps` back-to-back
        calls (the pools, ~450 MB, exceed L2)."""
        c = W.chunked_prefill(0, n_decode=n_decode, page_size=page_size)
        q, bi, ip = c.q.to(dev), c.batch_idx.to(dev), c.input_pos.to(dev)
        kp, vp, pt = c.k_pool.to(dev), c.v_pool.to(dev), c.page_table.to(dev)
        out = torch.empty_like(q)
        lse = torch.empty((c.n_tokens, c.num_q_heads), dtype=torch.float32, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        binding.pkv_append(kp, vp, pt, c.k_new.to(dev), c.v_new.to(dev), bi, ip, c.page_size,
                           dev_err=err)
        for _ in range(3):
            binding.pkv_prefill_paged_attention(kp, vp, pt, q, bi, ip, c.page_size, c.scale,
                                                out=out, lse=lse, dev_err=err)
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record()
        for _ in range(reps):
            binding.pkv_prefill_paged_attention(kp, vp, pt, q, bi, ip, c.page_size, c.scale,
                                                out=out, lse=lse, dev_err=err)
        ev[1].record()
        torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise RuntimeError(f"device error bits {int(err.item()):#x} in chunked prefill")
        att_us = ev[0].elapsed_time(ev[1]) / reps * 1e3
        flops = 4.0 * c.head_dim * c.num_q_heads * c.info["pairs"]
        tf = flops / (att_us * 1e-6) / 1e12
        return {"workload": f"chunked_prefill: 16 chunks of 512 over prefixes U[512,4096] + "
                            f"{n_decode} decode tokens, T={c.n_tokens}, Hq=32, Hkv=8, D=128, "
                            f"page {page_size}, permuted pages, seed 0",
                "attention_call_us": att_us, "algorithmic_flops": flops, "tflops": tf,
                "bound": "tensor", "peak_tflops": bf16_peak, "frac": tf / bf16_peak,
                "peak_kind": peak_kind,
                "traffic": (captured_traffic("chunked_prefill_call")
                            if n_decode == 0 and page_size == 128 else None)}

    def timed_mixed_one_call(reps, n_decode=48):
        """The mixed step (16 chunks of 512 plus `n_decode` decode tokens,
        shuffled) through pkv_mixed_attention: one call, the decode tokens
        routed to the split-KV decode kernels; CUDA events over `reps`
        back-to-back calls (the K/V of the step appended once beforehand)."""
        c = W.chunked_prefill(0, n_decode=n_decode)
        q, bi, ip = c.q.to(dev), c.batch_idx.to(dev), c.input_pos.to(dev)
        kp, vp, pt = c.k_pool.to(dev), c.v_pool.to(dev), c.page_table.to(dev)
        out = torch.empty_like(q)
        lse = torch.empty((c.n_tokens, c.num_q_heads), dtype=torch.float32, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = torch.empty(binding.pkv_mixed_workspace_size(kp, pt, c.page_size, c.n_tokens,
                                                          c.num_q_heads),
                         dtype=torch.uint8, device=dev)
        binding.pkv_append(kp, vp, pt, c.k_new.to(dev), c.v_new.to(dev), bi, ip, c.page_size,
                           dev_err=err)

        def call():
            binding.pkv_mixed_attention(kp, vp, pt, q, bi, ip, c.page_size, c.scale, out=out,
                                        lse=lse, workspace=ws, dev_err=err)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record()
        for _ in range(reps):
            call()
        ev[1].record()
        torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise RuntimeError(f"device error bits {int(err.item()):#x} in the one-call mixed step")
        us = ev[0].elapsed_time(ev[1]) / reps * 1e3
        flops = 4.0 * c.head_dim * c.num_q_heads * c.info["pairs"]
        tf = flops / (us * 1e-6) / 1e12
        return {"call_us": us, "tflops": tf, "frac": tf / bf16_peak,
                "calls": "pkv_mixed_attention: routing, chunked prefill on the chunks' tokens, "
                         f"split-KV decode + merge on the {n_decode} decode tokens"}

    def timed_mixed_split(reps, n_decode=48):
        """The same mixed step (16 chunks of 512 plus `n_decode` one-token
        decodes, shuffled) served as two calls: the chunks' tokens through the
        paged prefill (their K/V appended once beforehand), and the decode
        tokens through the fused append + split-KV decode. Each call and the
        pair are timed with CUDA events over `reps` back-to-back repetitions."""
        c = W.chunked_prefill(0, n_decode=n_decode)
        slot_len = {s + 1: n for s, n in enumerate(c.chunk_lens)}
        is_dec = torch.tensor([slot_len.get(int(b), 0) == 1 for b in c.batch_idx.tolist()])
        ci = (~is_dec).nonzero().flatten()
        di = is_dec.nonzero().flatten()
        kp, vp, pt = c.k_pool.to(dev), c.v_pool.to(dev), c.page_table.to(dev)
        q_c, bi_c, ip_c = c.q[ci].to(dev), c.batch_idx[ci].to(dev), c.input_pos[ci].to(dev)
        q_d, bi_d = c.q[di].to(dev), c.batch_idx[di].to(dev)
        sl_d = (c.input_pos[di] + 1).to(dev)
        kn_d, vn_d = c.k_new[di].to(dev), c.v_new[di].to(dev)
        nd = int(di.numel())
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        binding.pkv_append(kp, vp, pt, c.k_new[ci].to(dev), c.v_new[ci].to(dev), bi_c, ip_c,
                           c.page_size, dev_err=err)
        out_c = torch.empty_like(q_c)
        lse_c = torch.empty((q_c.shape[0], c.num_q_heads), dtype=torch.float32, device=dev)
        out_d = torch.empty_like(q_d)
        lse_d = torch.empty((nd, c.num_q_heads), dtype=torch.float32, device=dev)
        ws = torch.empty(binding.pkv_decode_workspace_size(kp, pt, c.page_size, nd,
                                                           c.num_q_heads),
                         dtype=torch.uint8, device=dev)

        def pre():
            binding.pkv_prefill_paged_attention(kp, vp, pt, q_c, bi_c, ip_c, c.page_size,
                                                c.scale, out=out_c, lse=lse_c, dev_err=err)

        def dec():
            binding.pkv_decode_append_attention(kp, vp, pt, q_d, kn_d, vn_d, bi_d, sl_d,
                                                c.page_size, c.scale, out=out_d, lse=lse_d,
                                                workspace=ws, dev_err=err)
        for _ in range(3):
            pre()
            dec()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        ev[0].record()
        for _ in range(reps):
            pre()
        ev[1].record()
        for _ in range(reps):
            dec()
        ev[2].record()
        for _ in range(reps):
            pre()
            dec()
        ev[3].record()
        torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise RuntimeError(f"device error bits {int(err.item()):#x} in the split mixed step")
        both_us = ev[2].elapsed_time(ev[3]) / reps * 1e3
        flops = 4.0 * c.head_dim * c.num_q_heads * c.info["pairs"]
        tf = flops / (both_us * 1e-6) / 1e12
        return {"prefill_call_us": ev[0].elapsed_time(ev[1]) / reps * 1e3,
                "decode_call_us": ev[1].elapsed_time(ev[2]) / reps * 1e3,
                "step_us": both_us, "tflops": tf, "frac": tf / bf16_peak,
                "calls": "pkv_prefill_paged_attention on the chunks' tokens, then "
                         f"pkv_decode_append_attention on the {nd} decode tokens"}

    from paged_kv_gqa_pkv_gb300 import sharding
    # each rank serves its own shard of independent sequences (weak scaling)
    case = W.qwen3_b64_decode(sharding.shard_seed(rank), permute=False)
    bytes_dec = decode_bytes(case)
    kv_only = int(case.seq_lens.long().sum()) * case.num_kv_heads * case.head_dim * 4
    r = timed_decode(case, args.steps, args.warmup)
    ms_step = sharding.max_over_ranks(r["total_ms"] / args.steps, device=dev)
    value = sharding.whole_job_rate(kv_only, world, ms_step * 1e-3) / 1e9

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    achieved = step_bytes(case) / (ms_step * 1e-3) / 1e9
    dec_gbs = bytes_dec / (r["dec_ms"] * 1e-3) / 1e9
    perm = W.qwen3_b64_decode(0, permute=True)
    rp = timed_decode(perm, max(args.steps // 4, 10), args.warmup)
    perm256 = W.qwen3_b64_decode(0, permute=True, page_size=256)
    rp256 = timed_decode(perm256, max(args.steps // 4, 10), args.warmup)
    e2e_ms, h2d, d2h = e2e_decode(case, max(args.steps // 10, 10), args.warmup, zero_copy=True)
    e2e_ce_ms, h2d_ce, _ = e2e_decode(case, max(args.steps // 10, 10), args.warmup,
                                      staged=False)
    e2e_st_ms, _, _ = e2e_decode(case, max(args.steps // 10, 10), args.warmup, staged=True)
    # the other decode workloads, and the batch sweep at the Qwen3-4B shape
    configs = {"padded_bucket": timed_decode_config(W.padded_bucket_decode(0)),
               "long_context_b256": timed_decode_config(W.long_context_decode(0))}
    sweep = [timed_decode_config(W.qwen3_b64_decode(0, permute=False, batch=b))
             for b in (8, 16, 32, 64, 128, 256)]
    prefill = timed_prefill(20)
    chunked = timed_chunked_prefill(20)
    mixed = timed_chunked_prefill(20, n_decode=48)
    chunked256 = timed_chunked_prefill(20, page_size=256)
    chunked["mixed_step_with_48_decode_tokens"] = {
        "attention_call_us": mixed["attention_call_us"], "tflops": mixed["tflops"],
        "frac": mixed["frac"], "split": timed_mixed_split(20),
        "one_call": timed_mixed_one_call(20)}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": "replicas" if world > 1 else "single",
                   "l2": f"inputs larger than L2: {r['n_sets']} rotating pool sets of "
                         f"{r['set_bytes'] / 1e6:.0f} MB"},
        "tokens_per_s_per_layer": world * case.batch / (ms_step * 1e-3),
        "decode_call_us": r["dec_ms"] * 1e3, "decode_call_us_p10_p90": [r["dec_p10"] * 1e3,
                                                                         r["dec_p90"] * 1e3],
        "decode_call_gbs": dec_gbs, "decode_call_frac": dec_gbs / hbm_peak,
        "two_call_step_us": r["two_call_ms"] * 1e3,
        "timing": f"CUDA-graph replay of {r['per_graph']}-step graphs; decode call = replay "
                  f"of {r['per_graph']} decode calls / {r['per_graph']}; each timed region "
                  f"starts behind ~0.5 ms of device work, so the host's graph submission "
                  f"is not timed",
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": captured_traffic("decode_step"),
                     "traffic_unit": "bytes per step (ncu dram read+write, both kernels)",
                     "kernel": "pkv_decode_append_attention (split-KV pass with the fused "
                               "append, then the LSE merge): the timed step",
                     "algorithmic_bytes": step_bytes(case),
                     "peak_kind": peak_kind, "frac_of_nominal_8TBs": achieved / NOMINAL_HBM_GBS},
        "page_size_256": {
            "decode_call_us": rp256["dec_ms"] * 1e3,
            "decode_frac": decode_bytes(perm256) / (rp256["dec_ms"] * 1e-3) / 1e9 / hbm_peak,
            "chunked_prefill_call_us": chunked256["attention_call_us"],
            "chunked_prefill_frac": chunked256["frac"],
            "workloads": "qwen3_b64_decode and chunked_prefill as above, page 256, "
                         "permuted pages"},
        "permuted_pages": {"decode_call_us": rp["dec_ms"] * 1e3,
                           "achieved_gbs": decode_bytes(perm) / (rp["dec_ms"] * 1e-3) / 1e9,
                           "frac": decode_bytes(perm) / (rp["dec_ms"] * 1e-3) / 1e9 / hbm_peak},
        "e2e": {"value": kv_only / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms,
                "transfers": "inputs (q, k_new, v_new, batch_idx, seq_lens) read by the fused "
                             "call from one pinned host buffer over the host link, no copy; "
                             "results: out and lse written by the kernels into pinned host "
                             "memory; the page table stays on the device",
                "copy_engine_ms_per_step": e2e_ce_ms,
                "copy_engine": f"the same step with its inputs and the page table ({h2d_ce} "
                               f"bytes) copied to the device by the copy engine first",
                "staged_ms_per_step": e2e_st_ms,
                "staged": "the same step with the inputs copied by pkv_stage_from_host (the "
                          "SMs' own loads over the host link) instead of the copy engine"},
        "decode_configs": configs,
        "batch_sweep": {"workload": "qwen3_b64_decode shape at batch B: Hq=32, Hkv=8, D=128, "
                                    "page 128, keys U[512,1024], sequential pages, seed 0",
                        "rows": sweep},
        "prefill": prefill,
        "chunked_prefill": chunked,
        "gpu_launches": 2 * args.steps,
        "clocks": r["clocks"],
    }
    if not args.no_cpu_baseline:
        # the oracle as it stands on the host cores: all 64 rows of the step
        # over one process per core, then the whole step on one core, then a
        # seeded sample of 64 of the 256 long-context rows over all cores
        gbs, d = run_oracle_child("parallel", rows=list(range(64)), reps=5)
        gbs1, d1 = run_oracle_child("full", reps=3)
        long_rows = sorted(int(x) for x in
                           torch.randperm(256, generator=torch.Generator().manual_seed(0))[:64])
        gbsl, dl = run_oracle_child("parallel", workload="long_context_decode", rows=long_rows,
                                    reps=3)
        line["cpu_baseline"] = {
            "value": gbs, "unit": UNIT, "cores": d["cores"], "kind": "oracle",
            "sample": f"decode of all 64 rows of the step, one row per task on {d['cores']} "
                      "processes (one BLAS thread each), append done once before timing; "
                      "median of 5",
            "host_cpu_count": d["host_cpu_count"], "seconds_per_step": d["seconds"],
            "single_core": {"value": gbs1, "cores": 1, "seconds_per_step": d1["seconds"],
                            "sample": "the full step (append 64 tokens + decode all 64 rows) "
                                      "on one core, median of 3"},
            "long_context_b256": {"value": gbsl, "cores": dl["cores"],
                                  "seconds": dl["seconds"],
                                  "sample": "decode of 64 seeded rows of the 256, one row per "
                                            "task on all cores, median of 3"}}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_pkv(args)


if __name__ == "__main__":
    main()
