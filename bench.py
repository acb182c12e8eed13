"""Benchmark of the weight-absorbed MLA decode path on one GB300.

A step is one decode step of the large V3 workload: 64 sequences, 128 heads,
context lengths drawn uniformly from [1024, 16384], page 64, random block
table; bf16 storage, fp32 accumulation. One step runs every stage of the path
through the C ABI: absorb (W_UK fold) -> q concat and cache write of the new
rows (one launch) -> split-KV decode with the W_UV un-projection (schedule,
split kernel, LSE combine fused with v_up).
Inputs are resident in HBM before the timed region; the latent cache (about
0.56 GB) is larger than L2 (129 MB), so no flush is needed between steps.

Printed (rank 0, one JSON line): value = latent-KV GB/s, i.e. the decode
stage's algorithmic bytes (cache rows read, q_cat read, o_lat written, block
table and lengths read) per step over the step time; queries/s beside it; the
roofline of the decode-and-un-project call (timed live with CUDA events on its
stream, with that call's own algorithmic bytes and flops); the
end-to-end figure through the same API with host buffers; the float64 oracle
timed on a bounded sample on the host cores; and the SM clocks sampled during
the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode latent-KV HBM GB/s (% roofline); queries/s at 128 heads"
UNIT = "GB/s"
WORKLOAD = "v3_bf16_decode_b64_ctx1k-16k"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# --------------------------------------------------------------------------- helpers

def _peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=FALLBACK_HBM_GBS, bf16_tflops=FALLBACK_BF16_TFLOPS,
                bf16_tflops_sustained=1700.0, source="fallback")


def decode_algorithmic_bytes(seq_lens, B, H, L, R, max_blocks, es=2, cache_es=None) -> int:
    """Bytes the decode stage must move: every cached row once (cache_es bytes an element,
    1 for an e4m3 cache), q_cat in, o_lat out, the block-table entries in use and the lengths."""
    E = L + R
    ce = es if cache_es is None else cache_es
    rows = int(sum(int(n) for n in seq_lens))
    pages = int(sum((int(n) + 63) // 64 for n in seq_lens))
    return rows * E * ce + B * H * E * es + B * H * L * es + pages * 4 + B * 4


def decode_algorithmic_flops(seq_lens, H, L, R) -> int:
    return int(sum(int(n) for n in seq_lens)) * H * 2 * ((L + R) + L)


def decode_v_up_algorithmic(seq_lens, B, H, L, R, V, es=2) -> tuple[int, int]:
    """Bytes and flops of the decode with its un-projection as one call: the decode's, less
    the o_lat it no longer writes, plus W_UV read and out written; plus the un-projection's
    2*B*H*L*V flops."""
    nbytes = decode_algorithmic_bytes(seq_lens, B, H, L, R, 0, es) - B * H * L * es + H * L * V * es + B * H * V * es
    return nbytes, decode_algorithmic_flops(seq_lens, H, L, R) + 2 * B * H * L * V


def roofline(nbytes: float, flops: float, ms: float, peaks: dict, sustained: bool = False) -> dict:
    """Roofline figures of one launch against the tighter of its two bounds: HBM bytes at the
    measured copy rate, or bf16 tensor flops at the measured GEMM rate (burst for a kernel timed
    alone, sustained for one timed inside a long step)."""
    tc_peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (tc_peak * 1e12)
    sec = ms * 1e-3
    if t_hbm >= t_tc:
        r = {"bound": "hbm", "achieved": nbytes / sec / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        r = {"bound": "tensor", "achieved": flops / sec / 1e12, "peak": tc_peak, "unit": "TFLOP/s"}
    r["frac"] = r["achieved"] / r["peak"]
    return r


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        # the busiest samples are the ones under load
        loaded = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


TRAFFIC_SOURCES = ("attn_tc.cu", "attn_simt.cu", "combine_vup.cu")


def _sources_sha(names) -> str:
    h = hashlib.sha256()
    for n in names:
        h.update(open(os.path.join(ROOT, "mla_latent_kv_11_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:16]


def _traffic_for(names=TRAFFIC_SOURCES) -> float | None:
    """ncu DRAM bytes per call recorded for the current sources of its kernels, else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    entry = d.get("decode")
    if not entry:
        return None
    try:
        if _sources_sha(names) != entry.get("source_sha"):
            return None
    except OSError:
        return None
    return float(entry["bytes_per_launch"])


# --------------------------------------------------------------------------- the workload

class DecodeStep:
    """Device-resident inputs of one decode step and the three calls that run it."""

    def __init__(self, mla, w, device, rank_seed=0):
        import numpy as np
        import torch
        self.mla, self.w = mla, w
        g = w.geom
        self.B, self.H, self.P, self.R, self.V, self.L = w.batch, g.n_head, g.d_nope, g.d_rope, g.d_v, g.kv_rank
        self.E = self.L + self.R
        dt = torch.bfloat16

        def dev(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(dt)

        self.dev = dev
        self.q_nope = dev(w.q_nope)
        self.q_pe = dev(w.q_pe)
        self.w_uk = dev(w.w_uk)
        self.w_uv = dev(w.w_uv)
        self.new_kv_c = dev(w.new_kv_c)
        self.new_k_pe = dev(w.new_k_pe)
        self.slots = torch.from_numpy(w.slots).to(device)
        self.table = torch.from_numpy(w.block_table).to(device)
        self.lens = torch.from_numpy(w.seq_lens).to(device)
        self.cache = dev(w.full_cache())
        B, H, L, E, V = self.B, self.H, self.L, self.E, self.V
        self.q_cat = torch.empty((B, H, E), dtype=dt, device=device)
        self.out = torch.empty((B, H, V), dtype=dt, device=device)
        self.ws = torch.empty(mla.mla_decode_v_up_workspace_size(B, H, L, 0), dtype=torch.uint8, device=device)
        # absorb (1) + concat and cache write (1) + decode with v_up (schedule, split, combine
        # with the un-projection: 3)
        self.launches_per_step = 5

    def run(self, ev_decode=None, q_nope=None, q_pe=None, kv_c=None, k_pe=None, slots=None,
            table=None, lens=None, out=None):
        m = self.mla
        out = self.out if out is None else out
        q_nope = self.q_nope if q_nope is None else q_nope
        # one call for steps 1 to 3: the absorb writes q_lat straight into q_cat's first L
        # columns, and the rope columns of q_cat and the cache write of the new rows run in one
        # launch alongside it
        m.mla_absorb_concat_cache_write(self.q_cat, q_nope.transpose(0, 1), self.w_uk,
                                        self.q_pe if q_pe is None else q_pe, self.cache,
                                        self.new_kv_c if kv_c is None else kv_c,
                                        self.new_k_pe if k_pe is None else k_pe, self.slots if slots is None else slots)
        if ev_decode is not None:
            ev_decode[0].record()
        m.mla_decode_v_up(out, self.q_cat, self.cache, self.table if table is None else table,
                          self.lens if lens is None else lens, self.L, self.R, self.w.scale, self.w_uv,
                          workspace=self.ws)
        if ev_decode is not None:
            ev_decode[1].record()


def _smi_id(local: int) -> str:
    """nvidia-smi's name for torch device ``local`` (its UUID: CUDA_VISIBLE_DEVICES renumbers)."""
    import torch
    u = getattr(torch.cuda.get_device_properties(local), "uuid", None)
    if u is None:
        return str(local)
    u = str(u)
    return u if u.startswith("GPU-") else "GPU-" + u


def _dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(value: float, group=None) -> float:
    """The maximum of a per-rank float over all ranks (identity on one rank)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return value
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def sum_over_ranks(value: float, group=None) -> float:
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return value
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return float(t.item())


def job_throughput(bytes_per_rank_step: float, ms_step_slowest: float, world: int) -> float:
    """Whole-job GB/s: the bytes every rank processed in a step over the slowest rank's step time
    (weak scaling: each rank runs its own batch)."""
    return bytes_per_rank_step * world / (ms_step_slowest * 1e-3) / 1e9


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# --------------------------------------------------------------------------- CPU oracle leg

def oracle_sample(w, n_seq: int, start: int = 0):
    """A bounded sample of the workload for the oracle: sequences [start, start+n_seq)
    with their own blocks only (block ids renumbered), in float64."""
    import numpy as np
    import mla_inputs as mi
    ids = [(start + i) % w.batch for i in range(n_seq)]
    lens = w.seq_lens[ids]
    page, E = w.page, w.geom.entry
    need = [(int(n) + page - 1) // page for n in lens]
    old_blocks = np.concatenate([w.block_table[b, :k] for b, k in zip(ids, need)])
    table = np.zeros((n_seq, max(need)), np.int64)
    k = 0
    for i, n in enumerate(need):
        table[i, :n] = np.arange(k, k + n)
        k += n
    storage = mi.decode_f64(w.cache_rows(old_blocks).reshape(-1), w.dtype)
    # slots of the appended rows, renumbered into the sample's blocks
    slots = np.array([table[i, (int(lens[i]) - 1) // page] * page + (int(lens[i]) - 1) % page
                      for i in range(n_seq)], np.int64)
    f = lambda a: mi.decode_f64(a, w.dtype)
    return dict(q_nope=f(w.q_nope[ids]), q_pe=f(w.q_pe[ids]), w_uk=f(w.w_uk), w_uv=f(w.w_uv),
                new_kv_c=f(w.new_kv_c[ids]), new_k_pe=f(w.new_k_pe[ids]), slots=slots,
                storage=storage, offset=0, page=page, strides=(page * E, E, 1), block_table=table,
                seq_lens=lens, scale=w.scale), lens


def _blas_threads() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_oracle_leg(w, budget_s: float = 12.0) -> dict:
    """Time the float64 oracle's decode step on a bounded sample of the workload."""
    from oracle import mla_oracle as orc
    g = w.geom
    n_total, t_total, bytes_total = 0, 0.0, 0
    start = 0
    while t_total < budget_s and n_total < w.batch:
        n = 2
        args, lens = oracle_sample(w, n, start)
        t0 = time.perf_counter()
        orc.decode_step(**args)
        t_total += time.perf_counter() - t0
        bytes_total += decode_algorithmic_bytes(lens, n, g.n_head, g.kv_rank, g.d_rope, 0)
        n_total += n
        start += n
    return {"value": bytes_total / t_total / 1e9, "unit": UNIT, "cores": _blas_threads(),
            "kind": "oracle",
            "queries_per_s": n_total / t_total,
            "sample": f"{n_total} of {w.batch} sequences of the same workload (their own blocks), "
                      f"one decode step each, float64 numpy oracle; {t_total:.1f} s"}


# --------------------------------------------------------------------------- the arms

def run_reference(args) -> None:
    """The oracle on the host cores, each step a bounded sample (one sequence, rotating)."""
    rank, world, _ = _dist_env()
    if rank != 0:
        return
    import mla_inputs as mi
    from oracle import mla_oracle as orc
    w = mi.v3_decode_large(materialize_cache=False)
    g = w.geom
    for i in range(args.warmup):
        a, _ = oracle_sample(w, 1, i)
        orc.decode_step(**a)
    t_total, bytes_total, n = 0.0, 0, 0
    for i in range(args.steps):
        a, lens = oracle_sample(w, 1, args.warmup + i)
        t0 = time.perf_counter()
        orc.decode_step(**a)
        t_total += time.perf_counter() - t0
        bytes_total += decode_algorithmic_bytes(lens, 1, g.n_head, g.kv_rank, g.d_rope, 0)
        n += 1
    value = bytes_total / t_total / 1e9
    cores = _blas_threads()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / max(n, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "queries_per_s": n / t_total,
        "config": {"workload": WORKLOAD, "batch": w.batch, "heads": g.n_head, "page": w.page,
                   "sample_per_step": "one sequence of the batch (rotating), its own blocks"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{n} sequences, one per step, float64 numpy oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_ours(args) -> None:
    import numpy as np
    import torch
    import torch.distributed as dist

    rank, world, local = _dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"

    import mla_latent_kv_11_gb300 as mla
    from mla_latent_kv_11_gb300 import build as mla_build
    import mla_inputs as mi
    if rank == 0:
        mla_build.build()
    barrier()
    mla.lib()

    # Every rank runs its own batch of 64 sequences: weak scaling, no data-path collective.
    w = mi.v3_decode_large(materialize_cache=True)
    g = w.geom
    step = DecodeStep(mla, w, device)
    stream = torch.cuda.current_stream()
    B, H, L, R = step.B, step.H, step.L, step.R
    bytes_step = decode_algorithmic_bytes(w.seq_lens, B, H, L, R, 0)
    call_bytes, call_flops = decode_v_up_algorithmic(w.seq_lens, B, H, L, R, step.V)

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()

    # The timed steps go to the GPU as one CUDA graph of all K steps, as a serving loop launches
    # them (the C-ABI calls captured once). An event node between two kernels of a graph costs the
    # step about 4 us (it takes the place of the programmatic launch edge), so the step is timed
    # over a graph of the K steps with no event inside, and the decode call's duration over a
    # second replay of the same K steps captured with an event pair around each call. Where
    # torch cannot capture external events, both are timed over one eager loop with the events.
    graphs_t, timed_launch = None, "eager"
    try:
        evs = [(torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True)) for _ in range(args.steps)]
        g_plain, g_ev = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_plain):
            for i in range(args.steps):
                step.run()
        with torch.cuda.graph(g_ev):
            for i in range(args.steps):
                step.run(ev_decode=evs[i])
        g_plain.replay()                               # warm replays of the captured steps
        g_ev.replay()
        torch.cuda.synchronize()
        graphs_t, timed_launch = (g_plain, g_ev), "cuda_graph"
    except (TypeError, RuntimeError) as exc:
        torch.cuda.synchronize()
        timed_launch = f"eager ({type(exc).__name__})"
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(_smi_id(local)) as clk:
        barrier()
        torch.cuda.synchronize()
        clk.mark_start()
        t_start.record(stream)
        if graphs_t is not None:
            graphs_t[0].replay()
        else:
            for i in range(args.steps):
                step.run(ev_decode=evs[i])
        t_end.record(stream)
        if graphs_t is not None:
            graphs_t[1].replay()                       # the same K steps, the call's events inside
        torch.cuda.synchronize()
        clk.mark_end()
        barrier()
    ms_total = t_start.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total)
    ms_step = ms_total / args.steps
    decode_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in evs))
    clocks = clk.summary()

    # end to end through the same calls with host buffers: every step copies its inputs in from
    # pinned host memory, runs the three calls and copies its output back; like a serving loop,
    # the copies of neighbouring steps run on two copy streams under the compute (two sets of
    # device buffers, ordered by events), and the timed region ends when the last output is back
    def pinned(t):
        return t.detach().cpu().pin_memory()

    # the step's inputs sit in one pinned staging buffer (each at a 256-byte-aligned offset), so
    # a step's input transfer is one host-to-device copy into one device buffer of the same layout
    names = ("q_nope", "q_pe", "new_kv_c", "new_k_pe", "slots", "table", "lens")
    offs, o = {}, 0
    for k in names:
        t = getattr(step, k)
        offs[k] = (o, t.numel() * t.element_size())
        o = (o + offs[k][1] + 255) // 256 * 256
    host_buf = torch.empty(o, dtype=torch.uint8).pin_memory()
    for k in names:
        t = pinned(getattr(step, k)).contiguous()
        a, n = offs[k]
        host_buf[a:a + n].copy_(t.view(-1).view(torch.uint8))
    dev_buf = [torch.empty(o, dtype=torch.uint8, device=device) for _ in range(2)]

    def carve(buf, k):
        a, n = offs[k]
        t = getattr(step, k)
        return buf[a:a + n].view(t.dtype).view(t.shape)

    dev_in = [{k: carve(dev_buf[b], k) for k in names} for b in range(2)]
    dev_out = [torch.empty_like(step.out) for _ in range(2)]
    out_host = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    h2d = o
    d2h = out_host[0].numel() * out_host[0].element_size()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "done", "out")}

    def h2d_copy(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev["done"][b])        # step i-2 has finished reading these buffers
            dev_buf[b].copy_(host_buf, non_blocking=True)
            ev["in"][b].record(s_in)

    def run_on(b):
        d = dev_in[b]
        step.run(q_nope=d["q_nope"], q_pe=d["q_pe"], kv_c=d["new_kv_c"], k_pe=d["new_k_pe"],
                 slots=d["slots"], table=d["table"], lens=d["lens"], out=dev_out[b])

    # like a serving loop, the step goes to the GPU as one CUDA graph per input buffer set: the
    # three calls (five kernels) are captured once through the
    # same C ABI and replayed, so the host's per-call marshalling is paid once, not every step
    for b in range(2):                                 # the first eager runs read real inputs
        dev_buf[b].copy_(host_buf)
    torch.cuda.synchronize()
    graphs, launch = [], "cuda_graph"
    try:
        for b in range(2):
            run_on(b)                                  # eager once: lazy host set-up happens here
            torch.cuda.synchronize()
            gph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gph):
                run_on(b)
            graphs.append(gph)
    except Exception as exc:                          # capture unavailable: launch eagerly
        torch.cuda.synchronize()
        graphs, launch = [], f"eager ({type(exc).__name__})"

    def e2e_run(i):
        b = i % 2
        stream.wait_event(ev["in"][b])
        if i >= 2:
            stream.wait_event(ev["out"][b])           # step i-2's output has left this buffer
        if graphs:
            graphs[b].replay()
        else:
            run_on(b)
        ev["done"][b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["done"][b])
            out_host[b].copy_(dev_out[b], non_blocking=True)
            ev["out"][b].record(s_out)

    def e2e_loop(n):
        s_in.wait_stream(stream)      # the copies start after everything queued so far (the
        s_out.wait_stream(stream)     # timing event included)
        h2d_copy(0)
        for i in range(n):
            if i + 1 < n:
                h2d_copy(i + 1)
            e2e_run(i)
        stream.wait_stream(s_out)
        stream.wait_stream(s_in)

    e2e_loop(args.warmup)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_loop(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1)) / args.steps
    barrier()
    # the end-to-end output is the eager step's, bit for bit (same inputs, same kernels)
    step.run()
    torch.cuda.synchronize()
    if not torch.equal(out_host[(args.steps - 1) % 2].to(device).view(torch.int16), step.out.view(torch.int16)):
        raise RuntimeError("end-to-end output differs from the eager step's")

    # component figures on their own workloads (not part of the step's value)
    components = component_figures(mla, mi, device) if rank == 0 and not args.no_components else {}

    cpu = cpu_oracle_leg(w) if rank == 0 and world == 1 and not args.no_cpu else None

    if rank != 0:
        return
    peaks = _peaks()
    value = job_throughput(bytes_step, ms_step, world)
    rl = roofline(call_bytes, call_flops, decode_ms, peaks, sustained=True)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "queries_per_s": B * world / (ms_step * 1e-3),
        "config": {"workload": WORKLOAD, "batch_per_gpu": B, "heads": H, "kv_lora_rank": L,
                   "rope_dim": R, "page": w.page, "context": "U[1024,16384] per sequence",
                   "cached_rows": int(w.seq_lens.sum()), "l2": "inputs larger than L2 (no flush)",
                   "parallelism": f"replicas x{world} (sequences sharded, no collective)",
                   "launch": timed_launch},
        "roofline": {"kernel": "mla_decode_v_up (schedule + split + combine with the W_UV un-projection)", **rl,
                     "traffic": _traffic_for(),
                     "timing": ("CUDA events around each call, captured in a second replay of the K timed steps"
                                if graphs_t is not None else "CUDA events around each call in the timed loop"),
                     "peak_source": peaks["source"], "ms_per_launch": decode_ms,
                     "bytes_per_launch": call_bytes, "flops_per_launch": call_flops,
                     "hbm_frac": call_bytes / (decode_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                     "tensor_frac": call_flops / (decode_ms * 1e-3) / (peaks["bf16_tflops_sustained"] * 1e12)},
        "e2e": {"value": job_throughput(bytes_step, e2e_ms, world), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "launch": launch},
        "gpu_launches": step.launches_per_step * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "components": components,
    }
    print(json.dumps(line), flush=True)


def component_figures(mla, mi, device, only=None) -> dict:
    """Per-stage figures on the other workloads, each against the tighter of its rooflines:
    NoPE prefill, decode at a fixed 8192 context (bf16 and e4m3 cache, 128 heads; bf16 at 64
    heads), and the copy kernels. The copies run far shorter than a host call, so they are
    timed as device time: many launches captured in one CUDA graph, replayed between events,
    cycling through enough input sets to exceed L2."""
    import numpy as np
    import torch
    out = {}
    peaks = _peaks()
    torch.manual_seed(1234)
    l2_bytes = 129 * 2 ** 20

    def timed(fn, reps=10, warm=3):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    def device_timed(fns, per_graph=64, reps=5):
        """Mean device time of one call: per_graph calls (cycling through fns) in one graph."""
        for f in fns:
            f()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(per_graph):
                fns[i % len(fns)]()
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (reps * per_graph)

    def dev(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(device).view(torch.bfloat16)

    def want(group):
        return only is None or group in only

    if want("prefill"):
        prefill_figures(mla, mi, device, out, peaks, timed)
    if want("decode"):
        decode_figures(mla, mi, device, out, peaks, timed)
    if want("decode") or want("sparse"):
        sparse_figures(mla, mi, device, out, peaks, timed)
    if want("copy"):
        copy_figures(mla, mi, device, out, peaks, dev, device_timed, l2_bytes)
    return out


def prefill_figures(mla, mi, device, out, peaks, timed) -> None:
    """NoPE causal prefill, 64 heads, 4 x 2048."""
    import numpy as np
    import torch
    H, L, page, n_seq, S = 64, 512, 64, 4, 2048
    T = n_seq * S
    q = torch.randn((T, H, L), device=device, dtype=torch.bfloat16) * 0.7
    nb = T // page
    cache = torch.randn((nb, page, L), device=device, dtype=torch.bfloat16)
    table = torch.from_numpy(mi.permutation(4077, nb).astype(np.int32).reshape(n_seq, S // page)).to(device)
    cu = torch.arange(0, T + 1, S, dtype=torch.int32, device=device)
    kv = torch.full((n_seq,), S, dtype=torch.int32, device=device)
    o = torch.empty((T, H, L), dtype=torch.bfloat16, device=device)
    ms = timed(lambda: mla.mla_prefill(o, q, cache, table, cu, kv, S, L, 0, 1.0 / 16.0), reps=3, warm=1)
    flops = n_seq * (S * (S + 1) // 2) * H * 2 * (L + L)
    nbytes = (2 * T * H * L + T * L) * 2
    out["prefill_nope_h64_4x2048"] = {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12,
                                      "frac_of_bf16_peak": flops / (ms * 1e-3) / (peaks["bf16_tflops"] * 1e12),
                                      "roofline": roofline(nbytes, flops, ms, peaks)}
    del q, cache, o


def decode_figures(mla, mi, device, out, peaks, timed) -> None:
    """Decode at a fixed 8192-token context: 64 sequences, page 64, a seeded block permutation
    (the "batch 64 x 8K context" reading of the large decode); 128 heads with a 64-wide rope
    part (bf16 and e4m3 cache), and the 64-head NoPE geometry (no rope part)."""
    import numpy as np
    import torch
    B, L, page, ctx = 64, 512, 64, 8192
    nbl = ctx // page
    table = torch.from_numpy(mi.permutation(8192, B * nbl).astype(np.int32).reshape(B, nbl)).to(device)
    lens = torch.full((B,), ctx, dtype=torch.int32, device=device)
    for H, R, name in ((128, 64, "decode_b64_ctx8192_fixed"), (64, 0, "decode_h64_nope_b64_ctx8192_fixed")):
        E = L + R
        cache = torch.randn((B * nbl, page, E), device=device, dtype=torch.bfloat16) * 0.1
        q = torch.randn((B, H, E), device=device, dtype=torch.bfloat16) * 0.1
        o = torch.empty((B, H, L), dtype=torch.bfloat16, device=device)
        ws = torch.empty(mla.mla_decode_workspace_size(B, H, L, 0), dtype=torch.uint8, device=device)
        ms = timed(lambda: mla.mla_decode(o, q, cache, table, lens, L, R, 1.0 / math.sqrt(192), workspace=ws),
                   reps=20)
        nbytes = decode_algorithmic_bytes([ctx] * B, B, H, L, R, nbl)
        flops = decode_algorithmic_flops([ctx] * B, H, L, R)
        out[name] = {"ms": ms, "heads": H, "rope_dim": R, "gbs": nbytes / (ms * 1e-3) / 1e9,
                     "frac_of_hbm_peak": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                     "queries_per_s": B / (ms * 1e-3), "roofline": roofline(nbytes, flops, ms, peaks)}
        if H == 128:
            # the same rows in an e4m3 cache (scale 1/16), 576-byte rows
            scale = torch.full((1,), 1.0 / 16.0, dtype=torch.float32, device=device)
            rows = cache.view(-1, E)
            cache8 = torch.empty((B * nbl, page, E), dtype=torch.uint8, device=device)
            slots = torch.arange(rows.shape[0], dtype=torch.int64, device=device)
            mla.mla_cache_write_fp8(cache8, rows[:, :L], rows[:, L:], slots, scale)
            ms8 = timed(lambda: mla.mla_decode_fp8(o, q, cache8, table, lens, L, R, 1.0 / math.sqrt(192),
                                                   descale_k=scale, workspace=ws), reps=3, warm=1)
            nbytes8 = decode_algorithmic_bytes([ctx] * B, B, H, L, R, nbl, cache_es=1)
            out["decode_fp8_b64_ctx8192_fixed"] = {
                "ms": ms8, "gbs": nbytes8 / (ms8 * 1e-3) / 1e9, "queries_per_s": B / (ms8 * 1e-3),
                "path": "tensor cores (e4m3 pages loaded by TMA, converted to bf16 in shared memory)",
                "roofline": roofline(nbytes8, flops, ms8, peaks)}
            del cache8, rows, slots
        del cache, q, o, ws
    del table, lens


def sparse_figures(mla, mi, device, out, peaks, timed) -> None:
    """Sparse top-2048 decode over an fp8 ds_mla cache."""
    import numpy as np
    import torch
    # sparse top-2048 decode over an fp8 ds_mla cache: 64 queries of 128 heads, distinct slots
    # scattered over 4096 blocks of 64 entries (172 MB), every slot list full
    nrows = 4096 * 64
    codes = torch.randint(0, 0x70, (nrows, 512), dtype=torch.uint8, device=device)
    codes |= torch.randint(0, 2, (nrows, 512), dtype=torch.uint8, device=device) << 7
    scales = (torch.rand((nrows, 4), device=device) * (1.0 / 32 - 1.0 / 128) + 1.0 / 128).view(torch.uint8)
    rope = (torch.randn((nrows, 64), device=device) * 0.1).to(torch.bfloat16).view(torch.uint8)
    view = torch.cat([codes, scales, rope], dim=1).view(4096, 64, 656)
    del codes, scales, rope
    idx = mi.permutation(8193, nrows)[: 64 * 2048].astype(np.int32).reshape(64, 2048)
    qs = torch.randn((64, 128, 576), device=device).mul_(0.1).to(torch.bfloat16)
    os_ = torch.empty((64, 128, 512), dtype=torch.bfloat16, device=device)
    ind = torch.from_numpy(idx).to(device)
    ms = timed(lambda: mla.mla_decode_sparse_fp8(os_, qs, view, ind, 576 ** -0.5), reps=10)
    nbytes = 64 * 2048 * 656 + 64 * 128 * 576 * 2 + 64 * 128 * 512 * 2 + 64 * 2048 * 4
    flops = 64 * 2048 * 128 * 2 * (576 + 512)
    out["decode_sparse_fp8_b64_top2048"] = {"ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9,
                                            "queries_per_s": 64 / (ms * 1e-3),
                                            "roofline": roofline(nbytes, flops, ms, peaks)}
    del view, qs, os_, ind


def copy_figures(mla, mi, device, out, peaks, dev, device_timed, l2_bytes) -> None:
    """Concat and cache write, unified-slot workload (64 tokens x 128 heads; 200 new rows into
    the middle layer of a 3-layer cache); the concat inputs come in enough copies to exceed L2."""
    import torch
    w = mi.write_concat_workload()
    Nh, Bq, Lq = w.q_nope_storage.shape
    Rq = w.q_pe.shape[2]
    q_bytes = 2 * Bq * Nh * (Lq + Rq) * 2
    n_sets = max(2, -(-2 * l2_bytes // q_bytes))
    sets = []
    for _ in range(n_sets):
        store = dev(w.q_nope_storage)
        sets.append((store.as_strided((Bq, Nh, Lq), (Lq, Bq * Lq, 1)), dev(w.q_pe),
                     torch.empty((Bq, Nh, Lq + Rq), dtype=torch.bfloat16, device=device)))
    ms = device_timed([lambda s=s: mla.mla_concat_q(s[2], s[0], s[1]) for s in sets])
    out["concat_q_64x128"] = {"ms": ms, "gbs": q_bytes / (ms * 1e-3) / 1e9,
                              "roofline": roofline(q_bytes, 0, ms, peaks), "timing": f"device ({n_sets} input sets)"}
    E = w.entry
    big = torch.zeros((w.num_blocks, w.n_layers * w.page * E), dtype=torch.bfloat16, device=device)
    view = big.view(-1).as_strided((w.num_blocks, w.page, E), (w.n_layers * w.page * E, E, 1),
                                   w.layer * w.page * E)
    kv_c, k_pe = dev(w.kv_c), dev(w.k_pe)
    slots = torch.from_numpy(w.slots).to(device)
    ms = device_timed([lambda: mla.mla_cache_write(view, kv_c, k_pe, slots)])
    c_bytes = 2 * w.kv_c.shape[0] * E * 2 + w.slots.size * 8
    out["cache_write_200tok_unified_view"] = {"ms": ms, "gbs": c_bytes / (ms * 1e-3) / 1e9,
                                              "timing": "device (200 rows: launch-latency bound)"}
    # both in one launch, the step's form: rope columns into q_cat after an in-place absorb
    fused = []
    for s in sets:
        q_cat = s[2]
        fused.append(lambda q_cat=q_cat, r=s[1]: mla.mla_concat_q_cache_write(
            q_cat, q_cat[:, :, :Lq], r, view, kv_c, k_pe, slots))
    ms = device_timed(fused)
    f_bytes = 2 * Bq * Nh * Rq * 2 + c_bytes
    out["concat_rope_and_cache_write_one_launch"] = {"ms": ms, "gbs": f_bytes / (ms * 1e-3) / 1e9,
                                                     "timing": f"device ({n_sets} input sets)"}


def run_components(only) -> None:
    """The chosen per-stage figures alone on this process's GPU (for profiling one kernel)."""
    import torch
    import mla_latent_kv_11_gb300 as mla
    from mla_latent_kv_11_gb300 import build as mla_build
    import mla_inputs as mi
    mla_build.build()
    mla.lib()
    torch.cuda.set_device(0)
    print(json.dumps({"components": component_figures(mla, mi, "cuda:0", only=set(only))}), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle leg")
    ap.add_argument("--no-components", action="store_true", help="skip the per-stage figures")
    ap.add_argument("--component", action="append", choices=["prefill", "decode", "sparse", "copy"],
                    help="run only these per-stage figures (no decode step) and print them")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.component:
        run_components(args.component)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
