"""Benchmark of the attention-over-KV-cache hot path on GB300.

Headline workload (one "step"): the decode batch -- 64 sequences, 1 query and
1 appended token each, Hq=32, Hkv=8, D=128, bf16 paged cache (page 16,
seeded page permutation), cache lengths U[512, 4096].  One step = one
pkv_attn_varlen_kvcache_fwd call: KV append + persistent attention kernel +
split-KV combine.  value = algorithmic bytes of the step / device time, GB/s.

The other workloads (prefill with a cached prefix, the mixed batch, the fp8
cache) are measured the same way and reported under "workloads".

Timing: W warm-up steps, then the call is captured into a CUDA graph and K
replays are timed, each with CUDA events on the launching stream (the eager,
uncaptured call is timed too and reported beside it); L2 is flushed (256 MB
write, then a 256 MB read of another buffer so that the write's dirty lines
drain outside the timed region) before every timed step and before every
timed kernel.  --impl reference times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time


def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _set_blas_threads(n: int) -> None:
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = str(n)


# BLAS threads are fixed before numpy loads: the oracle child legs run with
# the count they are given, the reference arm with every core of the host
if "--oracle-leg-child" in sys.argv:
    _set_blas_threads(int(sys.argv[sys.argv.index("--oracle-threads") + 1]))
elif "--impl" in sys.argv and "reference" in sys.argv:
    _set_blas_threads(_host_cores())
else:
    _set_blas_threads(1)

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "decode KV GB/s & prefill attn TFLOP/s on 1 GB300, % of roofline"
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


# --------------------------------------------------------------------------- ncu traffic
def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments, trailing blanks and empty lines
    (string and character literals are kept as they are)."""
    out, i, n, quote = [], 0, len(text), None
    while i < n:
        c = text[i]
        if quote:
            out.append(c)
            if c == "\\" and i + 1 < n:
                out.append(text[i + 1])
                i += 2
                continue
            if c == quote:
                quote = None
            i += 1
        elif c in "\"'":
            quote = c
            out.append(c)
            i += 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(l.rstrip() for l in "".join(out).splitlines() if l.strip())


def kernel_source_hash() -> str:
    """Hash of the CUDA sources' code (comments and blank lines left out): a
    stored ncu traffic figure is used only for the kernel it was measured on."""
    import hashlib
    csrc = os.path.join(ROOT, "paged_kv_variable_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def stored_traffic(name: str):
    """dram bytes (read + write) per launch from profiles/<name>.txt, or None if
    that capture was taken on other kernel sources."""
    try:
        kv = {}
        with open(os.path.join(ROOT, "profiles", name + ".txt")) as f:
            for line in f:
                if "=" in line and not line.startswith("#"):
                    k, v = line.split("=", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_hash") != kernel_source_hash():
            return None
        return int(float(kv["dram_bytes_read_per_launch"]) + float(kv["dram_bytes_write_per_launch"]))
    except Exception:
        return None


# --------------------------------------------------------------------------- algorithmic work
def step_work(spec, with_new=True):
    """Bytes and flops one call must move / compute (valid tokens, unmasked pairs)."""
    es = 2 if spec.cache_dtype == "bf16" else 1
    lk = spec.kv_lens.astype(np.int64)
    lq = spec.q_lens.astype(np.int64)
    kv = int(lk.sum()) * spec.hkv * spec.d * 2 * es
    qo = int(lq.sum()) * spec.hq * spec.d * 2 * 2
    bt = int(sum((int(n) + spec.page_size - 1) // spec.page_size for n in lk)) * 4 if spec.page_size else 0
    new = int(spec.new_lens.sum()) * spec.hkv * spec.d * 2 * (2 + es) if with_new else 0
    pairs = 0
    for a, k in zip(lq, lk):
        a, k = int(a), int(k)
        if spec.causal:
            i = np.arange(a)
            pairs += int(np.clip(i + 1 + k - a, 0, k).sum())
        else:
            pairs += a * k
    return {"attn_bytes": kv + qo + bt, "append_bytes": new, "bytes": kv + qo + bt + new,
            "flops": 4 * spec.d * spec.hq * pairs}


# --------------------------------------------------------------------------- ranks
def aggregate_over_ranks(t_step_ms: float, units_per_rank: float, world: int, device=None):
    """Whole-job throughput of `world` replicas: every rank processed
    `units_per_rank` in its own t_step_ms; the job takes the slowest rank's
    time.  Returns (max step ms over ranks, job units per second)."""
    import torch
    import torch.distributed as dist
    t = t_step_ms
    if world > 1:
        ten = torch.tensor([t_step_ms], dtype=torch.float64, device=device)
        dist.all_reduce(ten, op=dist.ReduceOp.MAX)
        t = float(ten.item())
    return t, units_per_rank * world / (t * 1e-3)


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples (every 50 ms) while the timed region runs.

    One `nvidia-smi -lms 50` child streams the samples; only those taken between
    mark_start() and mark_end() are summarised (all of them if none fell there)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []   # (time, fields)
        self.window = (None, None)
        self._proc = None
        self._t = None

    def _read(self):
        for line in self._proc.stdout:
            f = [x.strip() for x in line.strip().split(",")]
            if len(f) >= 3:
                self.samples.append((time.perf_counter(), f))

    def __enter__(self):
        try:
            self._proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                           "--format=csv,noheader,nounits", "-lms", "50"],
                                          stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self._proc = None
            return self
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        t0 = time.perf_counter()
        while not self.samples and time.perf_counter() - t0 < 5.0 and self._proc.poll() is None:
            time.sleep(0.01)
        return self

    def mark_start(self):
        self.window = (time.perf_counter(), None)

    def mark_end(self):
        self.window = (self.window[0], time.perf_counter())

    def __exit__(self, *a):
        if self._proc is not None:
            time.sleep(0.06)  # one more sample after the region
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
                self._proc.wait(timeout=5)
        if self._t:
            self._t.join(timeout=5)

    def summary(self):
        t0, t1 = self.window
        inside = [f for t, f in self.samples if t0 is not None and t1 is not None and t0 <= t <= t1]
        rows = inside or [f for _, f in self.samples]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(s[1]) for s in rows if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in rows if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for s in rows for k in range(4) if len(s) > 5 + k and
                          s[5 + k].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "samples_in_timed_region": len(inside)}


# --------------------------------------------------------------------------- GPU arm
class Workload:
    """A case resident on the device, runnable as one library call per step."""

    def __init__(self, name, case, device):
        import torch
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        from tests import harness as H
        self.name, self.case = name, case
        self.g = H.GpuCase(case, device=device)
        self.g.write_prefix()
        self.work = step_work(case.spec, with_new=case.k_new is not None)
        self.torch = torch
        self.nsplit = self.g.plan.stats()["num_split_units"]

    def launches_per_step(self):
        return (1 if self.case.k_new is not None else 0) + 1 + (1 if self.nsplit else 0)

    def step(self, stream=None):
        self.g.run(stream)


def time_workload(wl, steps, warmup, flush, stream, graph=True):
    """Per-step device times (whole call, attention kernel) over `steps` steps.

    graph=True: the library call is captured once into a CUDA graph and each
    step is one replay, as a serving loop runs a fixed-shape decode step (no
    host launch gaps between the append, attention and combine kernels).
    graph=False: each step is an eager call from Python."""
    import torch
    import paged_kv_variable_gb300 as pkv
    for _ in range(warmup):
        wl.step()
    torch.cuda.synchronize()
    step_ms, kern_ms = [], []
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def capture(profiled):
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        if profiled:
            pkv.set_profile_events(k0, k1)
        with torch.cuda.graph(g, stream=cap):
            wl.step(cap)
        pkv.set_profile_events(None, None)
        torch.cuda.synchronize()
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        return g

    # The step is timed without the kernel events (with them the library keeps
    # the kernels strictly in order); the attention kernel in a second replay
    # of the same call captured with its events.
    g_step = capture(False) if graph else None
    g_prof = capture(True) if graph else None
    for _ in range(steps):
        flush_l2(flush)
        s0.record(stream)
        if graph:
            g_step.replay()
        else:
            wl.step()
        s1.record(stream)
        flush_l2(flush)
        if graph:
            g_prof.replay()
        else:
            pkv.set_profile_events(k0, k1)
            wl.step()
            pkv.set_profile_events(None, None)
        torch.cuda.synchronize()
        step_ms.append(s0.elapsed_time(s1))
        kern_ms.append(k0.elapsed_time(k1))
    assert wl.g.status() == 0, wl.g.pkv.last_error()
    del g_step, g_prof
    return step_ms, kern_ms


def flush_l2(bufs):
    """Evict L2 before a timed step: write one buffer twice the size of L2, then
    read another, so that the dirty lines of the write are written back here
    and not inside the timed region."""
    bufs[0].zero_()
    bufs[1].sum()


# what each --workload runs (the default is the headline decode batch; the
# others exist for profiler captures)
WORKLOAD_NAMES = {
    "decode": "decode: B=64, 1 query + 1 appended token each, Hq=32, Hkv=8, D=128, bf16 paged cache page 16 "
              "(seeded permutation), cache lens U[512,4096]",
    "decode-small": "decode: 16 sequences of the B=64 decode batch (profiler captures)",
    "prefill": "prefill: B=8, 512 new tokens on a 1536-token cached prefix, Hq=32, Hkv=8, D=128, bf16 "
               "contiguous cache, causal (profiler captures)",
    "fp8-decode": "decode at kv length 2048 on the fp8 cache of the B=64 fp8 prefill (profiler captures)",
    "fp8-prefill-small": "fp8 cache: causal prefill of 2048 tokens into an empty cache, B=4, Hq=32, Hkv=8, D=128, "
                         "page 16 (profiler captures)",
    "mixed": "mixed: 60 decode requests (cache U[1024,8192]) + 4 prefill requests (2048 tokens on U[0,2048]), "
             "Hq=32, Hkv=8, D=128, bf16 paged cache page 16, one launch (profiler captures)",
}


def e2e_decode(case, steps, warmup, device, mode="graph"):
    """The same step through the public API from HOST buffers, wall-clock timed:
    pinned-host -> device copies of the step's inputs (q, new K/V, lengths,
    cu_seqlens), the call, and the device -> host copy of the output, then a
    stream synchronisation, all inside the timed region.

    mode="graph": the serving-loop form -- a plan made once and the call
    captured once in a CUDA graph; each step copies its inputs in and replays
    the graph.  For a decode batch the plan is pkv_plan_decode_dynamic's (the
    lengths are read on the device at every call); a batch with prefill rows
    takes a plan for its own lengths.  mode="host_plan": each step also makes
    the plan on the host and uploads it before an eager call."""
    import torch
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from tests import harness as H
    import paged_kv_variable_gb300 as pkv
    g = H.GpuCase(case, device=device)
    spec = case.spec
    # the step's inputs (q, new K/V, cu_seqlens, lengths) sit in one pinned host
    # buffer and one device buffer, 256-byte aligned segments of each: one
    # host -> device copy a step, the call's arguments pointing into the device
    # buffer
    src = {
        "q": torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16),
        "k_new": torch.from_numpy(case.k_new.view(np.int16)).view(torch.bfloat16),
        "v_new": torch.from_numpy(case.v_new.view(np.int16)).view(torch.bfloat16),
        "cu_q": torch.from_numpy(np.ascontiguousarray(spec.cu_q, dtype=np.int32)),
        "cu_new": torch.from_numpy(np.ascontiguousarray(spec.cu_new, dtype=np.int32)),
        "lens": torch.from_numpy(np.ascontiguousarray(spec.cache_lens, dtype=np.int32)),
    }
    offs, off = {}, 0
    for k, t in src.items():
        offs[k] = off
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    hpack = torch.empty(off, dtype=torch.uint8).pin_memory()
    dpack = torch.empty(off, dtype=torch.uint8, device=device)

    def seg(buf, k):
        t = src[k]
        return buf[offs[k]:offs[k] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

    for k, t in src.items():
        seg(hpack, k).copy_(t)
    g.q, g.k_new, g.v_new = seg(dpack, "q"), seg(dpack, "k_new"), seg(dpack, "v_new")
    g.cu_q, g.cu_new, g.cache_lens = seg(dpack, "cu_q"), seg(dpack, "cu_new"), seg(dpack, "lens")
    dpack.copy_(hpack)
    out_h = torch.empty(g.out.shape, dtype=torch.bfloat16).pin_memory()
    h2d = hpack.numel()
    d2h = out_h.numel() * out_h.element_size()
    nsms = torch.cuda.get_device_properties(device).multi_processor_count
    stream = torch.cuda.current_stream()

    if mode == "graph":
        decode_only = bool(np.all(spec.q_lens * (spec.hq // spec.hkv) <= 16))
        if decode_only:
            pl = pkv.plan_decode_dynamic(g.problem, spec.q_lens, spec.cache_lens, spec.new_lens, nsms)
        else:
            pl = pkv.plan(g.problem, spec.q_lens, spec.cache_lens, spec.new_lens, nsms)
        ws = pkv.workspace_tensor(pl.workspace_bytes, device)
        pl.upload(ws)
        args = g.args()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        pkv.attn_varlen_kvcache_fwd(g.problem, args, pl, ws, stream=cap)
        cap.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            pkv.attn_varlen_kvcache_fwd(g.problem, args, pl, ws, stream=cap)
        torch.cuda.synchronize()

        def one():
            dpack.copy_(hpack, non_blocking=True)
            graph.replay()
            out_h.copy_(g.out, non_blocking=True)
            stream.synchronize()
    else:
        def one():
            pl = pkv.plan(g.problem, spec.q_lens, spec.cache_lens, spec.new_lens, nsms)
            dpack.copy_(hpack, non_blocking=True)
            pl.upload(g.workspace)
            pkv.attn_varlen_kvcache_fwd(g.problem, g.args(), pl, g.workspace)
            out_h.copy_(g.out, non_blocking=True)
            stream.synchronize()
            pl.close()

    for _ in range(warmup):
        one()
    ts = []
    for _ in range(steps):
        t0 = time.perf_counter()
        one()
        ts.append(time.perf_counter() - t0)
    if mode == "graph":
        assert pkv.get_status(ws) == 0, pkv.last_error()
        return statistics.median(ts) * 1e3, h2d, d2h
    return statistics.median(ts) * 1e3, h2d + int(g.plan.stats()["upload_bytes"]), d2h


def cpu_model() -> str:
    """The host CPU's model name (x86 'model name', or lscpu's 'Model name' on Arm)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_sample_seconds(case, seqs):
    """One bounded sample: the oracle on the given sequences of the workload."""
    import oracle
    sub = synth.subset_case(case, seqs)
    t0 = time.perf_counter()
    oracle.forward(sub)
    return time.perf_counter() - t0, step_work(sub.spec)["bytes"]


def _oracle_leg_child(budget_s: float) -> None:
    """Child process of the CPU leg (BLAS threads fixed by the parent): the
    oracle on whole sequences of the decode batch, three repeats of about
    budget_s / 3 each; prints the median throughput as JSON."""
    case = synth.config2()
    spec = case.spec
    vals, seqs_total, t_total = [], 0, 0.0
    nxt = 0
    for _ in range(3):
        t = b = 0.0
        n = 0
        while t < budget_s / 3:
            dt, by = oracle_sample_seconds(case, [nxt % spec.batch])
            nxt += 1
            t += dt
            b += by
            n += 1
        vals.append(b / t / 1e9)
        seqs_total += n
        t_total += t
    print(json.dumps({"value": statistics.median(vals), "repeats": vals, "sequences": seqs_total,
                      "seconds": t_total}))


def cpu_oracle_leg(budget_s=12.0):
    """The oracle as it stands, on bounded samples of the decode batch, timed
    on the host cores twice: BLAS threads = every core of the process's
    affinity set, and 1 thread (child processes, so the thread count is fixed
    before numpy loads).  Median of 3 repeats each."""
    cores = _host_cores()
    legs = {}
    for n in (cores, 1):
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-leg-child", "--oracle-threads",
                            str(n), "--oracle-budget", str(budget_s)], capture_output=True, text=True,
                           timeout=30 + 20 * budget_s)
        legs[n] = json.loads(r.stdout.strip().splitlines()[-1])
    allc, one = legs[cores], legs[1]
    return {"value": round(allc["value"], 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"whole sequences of the decode batch (B=64, Hq=32, Hkv=8, D=128), {allc['sequences']} "
                      f"sequences in {allc['seconds']:.1f} s at BLAS threads = {cores}; median of 3 repeats; "
                      "fp64 NumPy",
            "single_thread": {"value": round(one["value"], 4), "cores": 1,
                              "sample": f"{one['sequences']} sequences in {one['seconds']:.1f} s, median of 3"}}


def decode_variant(d=128, page_size=16):
    """The decode batch (B=64, one query and one appended token each, Hq=32,
    Hkv=8, cache lengths U[512,4096], the same seed, so the same lengths) at
    another head dim or page size."""
    import math
    rng = np.random.Generator(np.random.PCG64(1002))
    B = 64
    lc = rng.integers(512, 4096, size=B, endpoint=True).astype(np.int32)
    ones = np.ones(B, np.int32)
    width = (4097 + page_size - 1) // page_size
    spec = synth.Spec(batch=B, hq=32, hkv=8, d=d, page_size=page_size, causal=True,
                      softmax_scale=float(np.float32(1.0 / math.sqrt(d))), cache_dtype="bf16", q_lens=ones,
                      cache_lens=lc, new_lens=ones.copy(), capacity=width * page_size,
                      name=f"decode-d{d}-p{page_size}")
    return synth.make_case(spec, rng, block_table_width=width)


def use_ragged_page_list(wl):
    """Address the workload's paged cache through a ragged page list (each
    sequence's used pages concatenated, page_indptr offsets) in place of the
    padded block table."""
    import torch
    case, g = wl.case, wl.g
    spec = case.spec
    P = spec.page_size
    counts = [(int(n) + P - 1) // P for n in spec.kv_lens]
    flat = np.concatenate([case.block_table[b, :counts[b]] for b in range(spec.batch)]).astype(np.int32)
    indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    flat_t = torch.from_numpy(flat).to(g.q.device)
    indptr_t = torch.from_numpy(indptr).to(g.q.device)

    def args(with_new=True):
        return g.pkv.make_args(q=g.q, out=g.out, lse=g.lse, cu_seqlens_q=g.cu_q,
                               max_seqlen_q=int(spec.q_lens.max()), k_cache=g.k_cache, v_cache=g.v_cache,
                               cache_seqlens=g.cache_lens, k_new=g.k_new if with_new else None,
                               v_new=g.v_new if with_new else None,
                               cu_seqlens_knew=g.cu_new if with_new else None, block_table=flat_t,
                               page_indptr=indptr_t)
    g.args = args
    return wl


def with_q_scale(case):
    """The fp8 workload with quantised queries: per-tensor q_scale = amax(|q|)/448
    (fp32), the same rule as the cache scales."""
    import dataclasses
    amax = np.float32(np.abs(synth.bf16_bits_to_f32(case.q)).max())
    return dataclasses.replace(case, q_scale=float(np.float32(amax) / np.float32(448.0)))


def gpu_arm(args):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    peaks = _peaks()

    decode_case = synth.config2()
    cpu_base = cpu_oracle_leg(12.0 if args.cpu_leg else 1.5) if rank == 0 and not args.quick else None

    from paged_kv_variable_gb300 import build
    build.build()
    stream = torch.cuda.current_stream()
    flush = (torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device),
             torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device))

    if args.workload == "decode-small":
        # 16 sequences of the decode batch (about 150 MB of KV, above L2): profiler captures
        main = Workload("decode-small", synth.subset_case(decode_case, list(range(16))), device)
    elif args.workload == "prefill":
        # the contiguous-cache causal prefill (profiler captures of the tensor-core tile)
        main = Workload("prefill", synth.config3(True), device)
    elif args.workload == "fp8-decode":
        # decode token 2049 on the fp8 cache written by the fp8 prefill (profiler captures)
        pre_case, dec_case = synth.config5()
        main = Workload("fp8-decode", dec_case, device)
        pre = Workload("fp8-prefill", pre_case, device)
        pre.step()
        main.g.k_cache.copy_(pre.g.k_cache)
        main.g.v_cache.copy_(pre.g.v_cache)
        del pre
        torch.cuda.synchronize()
        torch.cuda.empty_cache()   # only the decode step's buffers stay on the device
    elif args.workload == "fp8-prefill-small":
        main = Workload("fp8-prefill-small", synth.config5(batch=4)[0], device)
    elif args.workload == "mixed":
        main = Workload("mixed", synth.config4(), device)
    else:
        main = Workload("decode", decode_case, device)
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        clk.mark_start()
        step_ms, kern_ms = time_workload(main, args.steps, args.warmup, flush, stream)
        torch.cuda.synchronize()
        clk.mark_end()
        if world > 1:
            dist.barrier()
        t_wall = time.perf_counter() - t_wall
    clocks = clk.summary()
    if args.quick:
        # profiler runs: the timed graph replays only
        if rank == 0:
            print(json.dumps({"workload": args.workload, "ms_per_step": round(statistics.median(step_ms), 5),
                              "attn_kernel_ms": round(statistics.median(kern_ms), 5), "quick": True}))
        return
    eager_ms, eager_kern_ms = time_workload(main, max(10, args.steps // 4), 3, flush, stream, graph=False)
    t_step, job_bytes_per_s = aggregate_over_ranks(statistics.median(step_ms), main.work["bytes"], world, device)
    t_kern = statistics.median(kern_ms)
    value = job_bytes_per_s / 1e9
    achieved = main.work["attn_bytes"] / (t_kern * 1e-3) / 1e9

    e2e_ms, h2d, d2h = e2e_decode(main.case, max(3, args.steps // 2), 3, device)
    e2e_hp_ms, h2d_hp, _ = e2e_decode(main.case, max(3, args.steps // 4), 3, device, mode="host_plan")
    e2e_val = main.work["bytes"] * world / (e2e_ms * 1e-3) / 1e9

    extra = {}
    if args.secondary and rank == 0:
        secondary = [("prefill_cached_prefix_causal", lambda: synth.config3(True), "tensor"),
                     ("prefill_cached_prefix_noncausal", lambda: synth.config3(False), "tensor"),
                     ("mixed_prefill_decode", synth.config4, "mixed"),
                     ("fp8_prefill", lambda: synth.config5()[0], "tensor"),
                     ("fp8_prefill_quantised_q", lambda: with_q_scale(synth.config5()[0]), "fp8tensor"),
                     ("fp8_decode", lambda: synth.config5()[1], "hbm"),
                     ("decode_head_dim_64", lambda: decode_variant(d=64), "hbm"),
                     ("decode_head_dim_256", lambda: decode_variant(d=256), "hbm"),
                     ("decode_page_size_4", lambda: decode_variant(page_size=4), "hbm"),
                     ("decode_ragged_page_list", synth.config2, "hbm")]
        n_sec = max(30, args.steps)
        for name, mk, bound in secondary:
            case = mk()
            wl = Workload(name, case, device)
            if name == "decode_ragged_page_list":
                use_ragged_page_list(wl)
            if name == "fp8_decode":
                pre = Workload("fp8_prefill_for_decode", synth.config5()[0], device)
                pre.step()
                wl.g.k_cache.copy_(pre.g.k_cache)
                wl.g.v_cache.copy_(pre.g.v_cache)
                del pre
            sm, km = time_workload(wl, n_sec, 3, flush, stream)
            ts, tk = statistics.median(sm), statistics.median(km)
            ent = {"ms_per_call": round(ts, 4), "attn_kernel_ms": round(tk, 4), "timed_calls": len(sm),
                   "stat": "median",
                   "tflops": round(wl.work["flops"] / (ts * 1e-3) / 1e12, 1),
                   "gbs": round(wl.work["bytes"] / (ts * 1e-3) / 1e9, 1)}
            if bound == "tensor":
                ent["attn_tflops"] = round(wl.work["flops"] / (tk * 1e-3) / 1e12, 1)
                ent["frac_of_bf16_peak"] = round(ent["attn_tflops"] / peaks["bf16_tflops"], 3)
            elif bound == "fp8tensor":
                # Q.K^T on e4m3 tensor cores (half of the flops), P.V on f16: the
                # pair's peak is the harmonic mix of the fp8 and bf16 dense rates
                fp8_peak = 2.0 * peaks["bf16_tflops"]
                ent["attn_tflops"] = round(wl.work["flops"] / (tk * 1e-3) / 1e12, 1)
                ent["frac_of_bf16_peak"] = round(ent["attn_tflops"] / peaks["bf16_tflops"], 3)
                ent["fp8_peak_tflops_derived"] = round(fp8_peak, 1)
                ent["mixed_peak_tflops_derived"] = round(2.0 / (1.0 / fp8_peak + 1.0 / peaks["bf16_tflops"]), 1)
                ent["frac_of_mixed_peak"] = round(ent["attn_tflops"] / ent["mixed_peak_tflops_derived"], 3)
                ent["peak_note"] = ("fp8 dense peak derived as 2 x the measured bf16 peak (no measured fp8 figure); "
                                    "Q.K^T runs on e4m3, P.V on f16, so the mixed peak is their harmonic mean")
            elif bound == "hbm":
                ent["attn_gbs"] = round(wl.work["attn_bytes"] / (tk * 1e-3) / 1e9, 1)
                ent["frac_of_hbm_peak"] = round(ent["attn_gbs"] / peaks["hbm_gbs"], 3)
            else:
                # decode part bound by HBM, prefill part by the tensor cores
                sp = wl.case.spec
                dec = [b for b in range(sp.batch) if sp.q_lens[b] * sp.g <= 16]
                pre = [b for b in range(sp.batch) if sp.q_lens[b] * sp.g > 16]
                wd = step_work(synth.subset_case(wl.case, dec).spec) if dec else {"attn_bytes": 0}
                wp = step_work(synth.subset_case(wl.case, pre).spec) if pre else {"flops": 0}
                t_dec = wd["attn_bytes"] / (peaks["hbm_gbs"] * 1e9)
                t_pre = wp["flops"] / (peaks["bf16_tflops"] * 1e12)
                ent["bound_ms_serial"] = round((t_dec + t_pre) * 1e3, 4)
                ent["bound_ms_overlap"] = round(max(t_dec, t_pre) * 1e3, 4)
                ent["target_ms"] = round((t_dec / 0.7 + t_pre / 0.5) * 1e3, 4)
                ent["meets_target"] = bool(ts <= ent["target_ms"])
                ent["overlap_frac"] = round(ent["bound_ms_overlap"] / ts, 3)
                ent["serial_frac"] = round(ent["bound_ms_serial"] / ts, 3)
            extra[name] = ent
            del wl
            torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAMES.get(args.workload, args.workload),
                       "step": "kv append + persistent attention + split-KV combine (one library call)",
                       "launch": "CUDA graph replay of the captured library call, one per step",
                       "l2": "flushed before every timed step (256 MB write, then a 256 MB read of another "
                             "buffer so no dirty line is written back inside the timed events)",
                       "parallelism": f"replicas x{world}", "split_units": main.nsplit},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "traffic": stored_traffic("attn_kernel_decode_batch64_traffic"),
                         "algorithmic_bytes": main.work["attn_bytes"], "source_hash": kernel_source_hash(),
                         "kernel": "attn_kernel (persistent attention)", "peak_src": peaks["src"],
                         "attn_kernel_ms": round(t_kern, 5)},
            "cpu_baseline": cpu_base,
            "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 4),
                    "form": "host buffers -> copies in, replay of the captured call (plan made once: "
                            "pkv_plan_decode_dynamic for a decode batch, else a plan for its lengths), copy out, "
                            "synchronise; wall clock",
                    "host_plan_each_step": {
                        "value": round(main.work["bytes"] * world / (e2e_hp_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                        "ms_per_step": round(e2e_hp_ms, 4), "h2d_bytes_per_step": int(h2d_hp)}},
            "gpu_launches": main.launches_per_step() * args.steps,
            "eager": {"ms_per_step": round(statistics.median(eager_ms), 5),
                      "attn_kernel_ms": round(statistics.median(eager_kern_ms), 5),
                      "note": "the same step as separate eager calls from Python"},
            "clocks": clocks,
            "wall_s_timed_region": round(t_wall, 4),
            "workloads": extra,
        }
        print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    case = synth.config2()
    work = step_work(case.spec)
    cores = _host_cores()
    per = []
    for i in range(args.warmup + args.steps):
        # each step: the oracle on a bounded sample (4 sequences) of the decode batch
        dt, by = oracle_sample_seconds(case, [(4 * i + k) % case.spec.batch for k in range(4)])
        if i >= args.warmup:
            per.append((dt, by))
    tot_t = sum(t for t, _ in per)
    tot_b = sum(b for _, b in per)
    value = tot_b / tot_t / 1e9
    sample = f"4 sequences of the decode batch per step, fp64 NumPy, BLAS threads = {cores}"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.median([t for t, _ in per]) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAMES["decode"], "sample": "4 sequences of the batch per step"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "work_bytes_full_step": work["bytes"]}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-secondary", dest="secondary", action="store_false")
    ap.add_argument("--workload", default="decode", choices=sorted(WORKLOAD_NAMES))
    ap.add_argument("--quick", action="store_true",
                    help="profiler runs: time the graph replays of the workload only (no CPU, eager, e2e or "
                         "secondary legs)")
    ap.add_argument("--no-cpu-leg", dest="cpu_leg", action="store_false")
    ap.add_argument("--oracle-leg-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--oracle-threads", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-budget", type=float, default=12.0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_leg_child:
        _oracle_leg_child(args.oracle_budget)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
