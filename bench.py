#!/usr/bin/env python3
"""Benchmark of paged relative-bias attention on GB300.

One step = one relattn_decode call on the Inkling-Small local-layer decode
workload (16 sequences, 32/8 heads, d = 128, window = rel_extent = 512,
lengths uniform in [4096, 32768], 128-token blocks from a 4096-block pool):
the window-aware walk, the split-KV kernel and the split-combine, all in one
kernel launch.  Cold caches come from inputs larger than L2: the steps rotate
over input sets that stand for the layers of a model -- each with its own KV
pool, queries and rel, all sharing one sequence-length vector and one block
table, as per-layer caches do -- until one pass over them touches more than
twice the L2, with no flush in between.  One pass over the sets (one decode call per set, back to back) is
captured as a CUDA graph, the way a serving step runs its kernels; each
replay is timed with CUDA events on the launching stream and divided by the
calls in it.

The JSON line reports decode HBM GB/s of algorithmic bytes (window keys at
token granularity, q, the used part of rel, out, block-table entries), the
decode kernel's roofline against the measured HBM copy peak, an end-to-end
figure through the C ABI with host buffers, the float64 oracle timed on the
host cores, and -- under "secondary" -- the other decode workloads and the
chunked prefill's TFLOP/s.

--impl reference times the oracle itself (on host cores) on the same
workload and metric.  --gpus N runs N independent replicas (one per rank);
the path does not shard.
"""

import os

# The oracle legs run with one BLAS thread; the count is reported.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from paged_relative_bias_gb300 import inputs as I  # noqa: E402

METRIC = ("relattn decode HBM GB/s (% of peak) + ms/step; "
          "prefill TFLOP/s (% BF16 peak)")
BLOCK = 128


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------

def decode_work(wl, seq_lens):
    """Algorithmic bytes of one decode call and of each (sequence, KV head).

    With k query tokens per sequence (positions L - k .. L - 1) the keys
    counted are those any of them sees, once; q, the rel entries each token
    uses and out count per token and head."""
    g = wl.num_q_heads // wl.num_kv_heads
    k = max(1, wl.query_tokens)
    res = 2 if wl.rel_dtype == "bf16" else 4
    kes = 1 if wl.kv_dtype == "fp8" else 2
    total = 0
    per_group = []
    for L in seq_lens:
        lo = max(0, L - k - wl.window + 1) if wl.window > 0 else 0
        P = L - 1
        blocks = P // BLOCK - lo // BLOCK + 1
        kv = (P - lo + 1) * (wl.d_qk + wl.d_v) * kes
        head = 0
        for Pi in range(L - k, L):
            n = min(wl.window, Pi + 1) if wl.window > 0 else Pi + 1
            head += wl.d_qk * 2 + min(wl.rel_extent, n) * res + wl.d_v * 2
        grp = kv + g * head
        per_group.append(grp)
        total += wl.num_kv_heads * grp + blocks * 4 + 4
    return total, per_group


def prefill_work(wl):
    """(flops, bytes) of one chunked-prefill call, visible pairs only."""
    flops = 0
    rel = 0
    kv_prefix = 0
    for n, ctx in zip(wl.new_tokens, wl.ctx_lens):
        for t in range(n):
            P = ctx + t
            vis = min(wl.window, P + 1) if wl.window > 0 else P + 1
            flops += vis
            rel += min(wl.rel_extent, vis)
        lo = max(0, ctx - wl.window + 1) if wl.window > 0 else 0
        kv_prefix += max(0, ctx - lo)
    T = sum(wl.new_tokens)
    Hq, Hkv = wl.num_q_heads, wl.num_kv_heads
    kvrow = Hkv * (wl.d_qk + wl.d_v) * 2  # a new token's bf16 key and value rows
    kvc = kvrow // 2 if wl.kv_dtype == "fp8" else kvrow  # ... as cached
    flops *= Hq * 2 * (wl.d_qk + wl.d_v)
    res = 2 if wl.rel_dtype == "bf16" else 4
    nbytes = (rel * Hq * res + T * Hq * (wl.d_qk + wl.d_v) * 2 + T * kvrow + T * kvc
              + kv_prefix * kvc)
    return flops, nbytes


def describe(wl):
    """One-line description of a workload (sizes and element types)."""
    if isinstance(wl, I.DecodeWorkload):
        lens = {"fixed": lambda s: f"L={s[1]}", "uniform": lambda s: f"L~U[{s[1]},{s[2]}]",
                "loguniform": lambda s: f"L~logU[{s[1]},{s[2]}]"}[wl.lengths[0]](wl.lengths)
        win = f"W={wl.window}" if wl.window > 0 else "global"
        kind = f"{wl.query_tokens}-token decode" if wl.query_tokens > 0 else "decode"
        return (f"{wl.name}: {kind} B={wl.batch} {wl.num_q_heads}/{wl.num_kv_heads} "
                f"d={wl.d_qk}/{wl.d_v} {win} E={wl.rel_extent} {lens} {wl.rel_dtype} rel "
                f"{'e4m3' if wl.kv_dtype == 'fp8' else 'bf16'} KV")
    win = f"W={wl.window}" if wl.window > 0 else "global"
    return (f"{wl.name}: prefill {len(wl.new_tokens)}x{wl.new_tokens[0]} after "
            f"{wl.ctx_lens[0]} cached, {wl.num_q_heads}/{wl.num_kv_heads} d={wl.d_qk} {win} "
            f"E={wl.rel_extent} {wl.rel_dtype} rel {'e4m3' if wl.kv_dtype == 'fp8' else 'bf16'} KV")


# The other spec workloads, timed after the headline and reported
# under "secondary" by short key (the sizes of each key are in describe()).
SECONDARY_DECODE = (  # key, workload, rel type, cache type
    ("cfg3a_global_b1", "global_decode_b1", "f32", "bf16"),
    ("cfg3b_global_b8", "global_decode_b8", "f32", "bf16"),
    ("cfg5_diffhead", "diffhead_decode", "f32", "bf16"),
    ("verify_k8", "verify_decode", "f32", "bf16"),
    ("cfg2_bf16rel", "local_decode", "bf16", "bf16"),
    ("cfg3b_e4m3", "global_decode_b8", "f32", "fp8"),
    ("cfg3a_e4m3", "global_decode_b1", "f32", "fp8"),
)
SECONDARY_PREFILL = (  # key, rel type, cache type (the chunked-prefill workload)
    ("cfg4", "f32", "bf16"),
    ("cfg4_bf16rel", "bf16", "bf16"),
    ("cfg4_e4m3", "f32", "fp8"),
)


# ---------------------------------------------------------------------------
# environment
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock/throttle samples every 100 ms while running."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        ident = str(device_index)
        try:
            u = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", ident], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        self.windows = []

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append(dict(ts=ts, sm=float(f[1]), smax=float(f[2]),
                                 hw=f[5], hwt=f[6], swt=f[7], swp=f[8]))
            except ValueError:
                continue
        inside = [r for r in rows if any(a - 1 <= r["ts"] <= b + 1 for a, b in self.windows)]
        use = inside if len(inside) >= 3 else rows
        reasons = set()
        for r in use:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(r["sm"] for r in use),
                "sm_max_mhz": max(r["smax"] for r in use),
                "reasons": sorted(reasons), "samples": len(use)}


class Dist:
    """The replicas of a torchrun launch (one rank per GPU, env:// rendezvous):
    a barrier and the max over ranks of the timed seconds.  No data-path
    collective: the path does not shard.  backend "gloo" runs the same logic
    on host tensors (tests)."""

    def __init__(self, backend: str = "nccl"):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.dev = "cpu"
        if self.world > 1:
            import torch.distributed as dist
            if backend == "nccl":
                torch.cuda.set_device(self.local)
                self.dev = f"cuda:{self.local}"
                dist.init_process_group("nccl", device_id=torch.device("cuda", self.local))
            else:
                dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=self.dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# timing
# ---------------------------------------------------------------------------

def timed_steps(fn, steps, warmup, flush, dist, sampler):
    """Per-step device times (ms) of fn(k) for steps k = 0, 1, ...; flush (if
    any) runs before every step, outside the timed region."""
    for k in range(warmup):
        if flush is not None:
            flush()
        fn(k)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    t0 = time.time()
    for k, (a, b) in enumerate(ev):
        if flush is not None:
            flush()
        a.record()
        fn(k)
        b.record()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    sampler.mark(t0, time.time())
    return [a.elapsed_time(b) for a, b in ev]


def roofline(bound, achieved, peak, unit, traffic):
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic}


def committed_traffic(kernel_tag):
    """dram bytes per launch from a committed ncu summary, if still current.

    profiles/<tag>.traffic holds `<bytes> <sha256 of the kernel source>`; the
    number is used only while the source is unchanged since the capture.
    """
    import hashlib
    path = os.path.join(ROOT, "profiles", kernel_tag + ".traffic")
    if not os.path.exists(path):
        return None
    try:
        nbytes, digest = open(path).read().split()[:2]
    except ValueError:
        return None
    src = os.path.join(ROOT, "paged_relative_bias_gb300", "csrc",
                       {"decode": "relattn_decode.cu", "prefill": "relattn_prefill.cu"}[
                           kernel_tag.split("_")[0]])
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return int(float(nbytes)) if h == digest else None


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def decode_sets(wl, device, l2, shared_pool=False):
    """Per-layer input sets, enough that one pass over them reads more than
    twice the L2 (a single set when one step already does).  Every set has its
    own KV pool, queries and rel; all share the first set's sequence lengths
    and block table tensors, like the layers of one decode step.

    shared_pool: the sets share the first set's KV pool instead, each with
    its own renumbered block table (the same bytes per call from a footprint
    of one pool: the small case for profiler captures)."""
    first = I.make_decode(wl, device)
    alg0, _ = decode_work(wl, first["seq_lens"].cpu().tolist())
    n = 1 if alg0 >= 2 * l2 else min(16, -(-2 * l2 // alg0))
    sets = [first]
    for s in range(1, n):
        if shared_pool:
            sets.append(I.relayout_decode(first, seed=100 + s))
            continue
        c = I.make_decode(wl, device, seed_data=s)  # same layout seed: same lengths and tables
        assert torch.equal(c["block_table"], first["block_table"])
        c["block_table"], c["seq_lens"] = first["block_table"], first["seq_lens"]
        sets.append(c)
    algs = [alg0] * n
    return sets, algs


def run_decode(R, wl, device, steps, warmup, dist, sampler, l2, shared_pool=False):
    """Graph-replayed decode steps rotating over the input sets."""
    sets, algs = decode_sets(wl, device, l2, shared_pool)
    tok = (wl.query_tokens,) if wl.query_tokens > 0 else ()
    fn = R.relattn_decode_multi if wl.query_tokens > 0 else R.relattn_decode
    wss, outs = [], []
    for case in sets:
        dims = R.Dims(wl.batch, wl.num_q_heads, case["block_table"].shape[1], 0, 0, 0)
        wss.append(R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                                       case["v_cache"])),
                                   device))
        outs.append(torch.empty((wl.batch, *tok, wl.num_q_heads, wl.d_v), dtype=torch.bfloat16,
                                device=device))

    def call(i):
        c = sets[i]
        fn(c["q"], c["rel"], c["k_cache"], c["v_cache"], c["block_table"], c["seq_lens"],
           wl.window, wl.rel_extent, out=outs[i], workspace=wss[i], k_scale=c.get("k_scale"),
           v_scale=c.get("v_scale"))

    # graphs[r]: calls for sets 0..r-1 back to back (r = len(sets) is one
    # full pass; shorter ones time the remainder of steps)
    n = len(sets)
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    graphs = {}
    with torch.cuda.stream(side):
        for i in range(n):  # first calls outside capture (lazy module loading)
            call(i)
        torch.cuda.synchronize(device)
        for r in sorted({n, steps % n, warmup % n} - {0}):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for i in range(r):
                    call(i)
            graphs[r] = g
    torch.cuda.current_stream(device).wait_stream(side)
    torch.cuda.synchronize(device)

    def chunks(total):  # graph replays covering exactly `total` calls
        return [n] * (total // n) + ([total % n] if total % n else [])

    def replay(k):
        graphs[plan[k]].replay()

    for r in chunks(warmup):
        graphs[r].replay()
    plan = chunks(steps)
    times = timed_steps(replay, len(plan), 0, None, dist, sampler)
    for ws in wss:
        if R.read_status(ws) != 0:
            raise RuntimeError("decode reported a device status")
    step_bytes = [algs[k % n] for k in range(steps)]
    # per-call times: each replay's time spread over its calls
    per_call = [t / r for t, r in zip(times, plan) for _ in range(r)]
    return sets, step_bytes, per_call, wss


def run_decode_e2e(R, sets, wl, wss, device, steps, warmup, dist, sampler):
    """The public call with host inputs: every step copies its inputs from
    pinned host memory and its output back, inside the timed region, rotating
    over the same input sets (their KV pools stay resident, like a serving
    cache).  Steps are pipelined the way a serving loop runs them: two device
    input buffers and two output buffers, and three streams ordered by events
    -- step k+1's inputs are copied in while step k's kernel runs, and step
    k's output is copied out while step k+1's runs.  One pass over the sets
    (per step: the input copy, the C-ABI call, the output copy) is captured as
    a CUDA graph, as a serving step's work is, and replayed; the timed region
    runs from before the first step's input copy to the end of the last
    step's output copy."""
    keys = ("q", "rel", "seq_lens", "block_table")
    # one pinned staging buffer per set holding the step's inputs back to
    # back (256-byte aligned pieces), so each step is one H2D copy; a device
    # buffer's pieces are the call's input tensors
    offs, size = {}, 0
    for k in keys:
        offs[k] = size
        size += (sets[0][k].numel() * sets[0][k].element_size() + 255) // 256 * 256
    host = []
    for c in sets:
        buf = torch.empty(size, dtype=torch.uint8).pin_memory()
        for k in keys:
            nb = c[k].numel() * c[k].element_size()
            buf[offs[k]:offs[k] + nb].copy_(c[k].cpu().contiguous().view(-1).view(torch.uint8))
        host.append(buf)
    NBUF = 2
    dbufs = [torch.empty(size, dtype=torch.uint8, device=device) for _ in range(NBUF)]

    def views(dbuf):
        return {k: dbuf[offs[k]:offs[k] + sets[0][k].numel() * sets[0][k].element_size()]
                .view(sets[0][k].dtype).view(sets[0][k].shape) for k in keys}
    devs = [views(d) for d in dbufs]
    tok = (wl.query_tokens,) if wl.query_tokens > 0 else ()
    oshape = (wl.batch, *tok, wl.num_q_heads, wl.d_v)
    out_h = [torch.empty(oshape, dtype=torch.bfloat16).pin_memory() for _ in range(NBUF)]
    out_d = [torch.empty(oshape, dtype=torch.bfloat16, device=device) for _ in range(NBUF)]

    # the C-ABI call of each (set, buffer), checked and marshalled once (its
    # buffers stay in place; only their contents change from step to step)
    runs = [[R.bind_decode(d["q"], d["rel"], c["k_cache"], c["v_cache"], d["block_table"],
                           d["seq_lens"], wl.window, wl.rel_extent, od, wss[i],
                           k_scale=c.get("k_scale"), v_scale=c.get("v_scale"))
             for d, od in zip(devs, out_d)] for i, c in enumerate(sets)]
    s_h2d, s_comp, s_d2h = (torch.cuda.Stream(device) for _ in range(3))
    ev_h2d, ev_kern, ev_d2h = ([torch.cuda.Event() for _ in range(NBUF)] for _ in range(3))

    def enqueue(k):
        b, i = k % NBUF, k % len(sets)
        with torch.cuda.stream(s_h2d):
            if k >= NBUF:
                s_h2d.wait_event(ev_kern[b])  # step k - 2's kernel has read buffer b
            dbufs[b].copy_(host[i], non_blocking=True)
            ev_h2d[b].record(s_h2d)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev_h2d[b])
            if k >= NBUF:
                s_comp.wait_event(ev_d2h[b])  # step k - 2's output has been copied out
            runs[i][b]()
            ev_kern[b].record(s_comp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev_kern[b])
            out_h[b].copy_(out_d[b], non_blocking=True)
            ev_d2h[b].record(s_d2h)

    cur = torch.cuda.current_stream(device)
    for st in (s_h2d, s_comp, s_d2h):
        st.wait_stream(cur)
    n = len(sets)
    for k in range(n):  # first calls outside capture
        enqueue(k)
    torch.cuda.synchronize(device)

    def capture(r):  # steps 0 .. r - 1 of a pass
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s_comp):
            s_h2d.wait_stream(s_comp)
            s_d2h.wait_stream(s_comp)
            for k in range(r):
                enqueue(k)
            s_comp.wait_stream(s_h2d)
            s_comp.wait_stream(s_d2h)
        return g
    graphs = {r: capture(r) for r in sorted({n, steps % n} - {0})}
    torch.cuda.synchronize(device)
    plan = [n] * (steps // n) + ([steps % n] if steps % n else [])
    with torch.cuda.stream(s_comp):
        for _ in range(max(1, warmup // n)):
            graphs[n].replay()
    torch.cuda.synchronize(device)
    dist.barrier()
    torch.cuda.synchronize(device)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    with torch.cuda.stream(s_comp):
        t_start.record(s_comp)
        for r in plan:
            graphs[r].replay()
        t_end.record(s_comp)
    torch.cuda.synchronize(device)
    dist.barrier()
    torch.cuda.synchronize(device)
    sampler.mark(w0, time.time())
    total = t_start.elapsed_time(t_end)
    times = [total / steps] * steps
    # the staged pieces are the set's inputs
    dbufs[0].copy_(host[0])
    torch.cuda.synchronize(device)
    for k in keys:
        if not torch.equal(devs[0][k], sets[0][k]):
            raise RuntimeError(f"e2e staging of {k} does not match its input")
    h2d = size  # the whole staging buffer (the four inputs and their padding)
    d2h = out_h[0].numel() * out_h[0].element_size()
    return times, h2d, d2h


def run_prefill(R, wl, device, steps, warmup, dist, sampler, case=None):
    case = case if case is not None else I.make_prefill(wl, device)
    dims = R.prefill_dims(case["q"], case["block_table"], case["ctx_lens"], case["max_q_len"])
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                             case["v_cache"])), device)
    out = torch.empty((case["num_tokens"], wl.num_q_heads, wl.d_v), dtype=torch.bfloat16,
                      device=device)

    def step(k):
        R.relattn_prefill(case["q"], case["k"], case["v"], case["rel"], case["cu_seqlens"],
                          case["k_cache"], case["v_cache"], case["block_table"],
                          case["ctx_lens"], wl.window, wl.rel_extent, case["max_q_len"],
                          out=out, workspace=ws, k_scale=case.get("k_scale"),
                          v_scale=case.get("v_scale"))

    # a step reads several GB (rel alone is T * Hq * E * 4 bytes), far more
    # than the L2: no flush is needed between steps
    times = timed_steps(step, steps, warmup, None, dist, sampler)
    if R.read_status(ws) != 0:
        raise RuntimeError("prefill reported a device status")
    return times


def run_prefill_graph(R, wl, device, calls, dist, sampler, per_replay=20):
    """Per-call device times (ms) of a small prefill: `per_replay` calls back to
    back captured in one CUDA graph, each replay timed with events and divided
    by its calls (a single call is shorter than an event pair's overhead).
    The calls rewrite the same cache entries with the same values."""
    case = I.make_prefill(wl, device)
    dims = R.prefill_dims(case["q"], case["block_table"], case["ctx_lens"], case["max_q_len"])
    ws = R.new_workspace(R.workspace_size(dims, R.cache_desc(case["k_cache"],
                                                             case["v_cache"])), device)
    out = torch.empty((case["num_tokens"], wl.num_q_heads, wl.d_v), dtype=torch.bfloat16,
                      device=device)

    def call():
        R.relattn_prefill(case["q"], case["k"], case["v"], case["rel"], case["cu_seqlens"],
                          case["k_cache"], case["v_cache"], case["block_table"],
                          case["ctx_lens"], wl.window, wl.rel_extent, case["max_q_len"],
                          out=out, workspace=ws)

    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        call()
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for _ in range(per_replay):
                call()
    torch.cuda.current_stream(device).wait_stream(side)
    torch.cuda.synchronize(device)
    reps = max(1, calls // per_replay)
    times = timed_steps(lambda k: g.replay(), reps, 3, None, dist, sampler)
    if R.read_status(ws) != 0:
        raise RuntimeError("prefill reported a device status")
    return [t / per_replay for t in times]


def prefill_entry(key, wl, times, peaks):
    """A compact secondary entry for a prefill workload: TFLOP/s of visible
    pairs, its HBM roofline and both bf16 tensor fractions."""
    flops, pbytes = prefill_work(wl)
    ms = sum(times) / len(times)
    tflops = flops / (ms / 1e3) / 1e12
    return {"workload": key, "value": round(tflops, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 5),
            "roofline": {"bound": "hbm", "frac": round(pbytes / (ms / 1e3) / 1e9 / peaks["hbm"], 4)},
            "frac_bf16": round(tflops / peaks["bf16"], 4),
            "frac_bf16_sustained": round(tflops / peaks["bf16_sustained"], 4)}


def group_blocks(O, wl, L, table_row):
    """[(logical, physical)] blocks holding any key the sequence's query
    tokens see: the oracle's walk for the newest token, widened back to the
    first visible key of the oldest one when there are several."""
    k = max(1, wl.query_tokens)
    blocks = O.decode_blocks(L, wl.window, table_row)
    lo, _ = O.visible_keys(L - k, wl.window)
    first = lo // BLOCK
    return [(lb, int(table_row[lb])) for lb in range(first, blocks[0][0])] + blocks


def cache_bits(t):
    """Host copy of KV cache blocks for the oracle ([n, 128, Hkv, d]): bf16
    bit patterns, or those of a head-major e4m3 cache ([n, Hkv, 128, d])."""
    from paged_relative_bias_gb300.inputs import bf16_bits
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).transpose(1, 2).contiguous().cpu().numpy()
    return bf16_bits(t)


def oracle_group(O, wl, q, rel, b, kc, vc, sub, L, heads, k_scale=1.0, v_scale=1.0):
    """The oracle on one (sequence, KV head) group over its gathered blocks."""
    fn = O.decode_multi if wl.query_tokens > 0 else O.decode
    fn(q[b:b + 1], rel[b:b + 1], kc, vc, sub, np.array([L]), wl.window, wl.rel_extent,
       heads=heads, k_scale=k_scale, v_scale=v_scale)


def oracle_decode_sample(case, wl, budget_s):
    """Time the float64 oracle on the workload's (sequence, KV head) groups:
    whole passes over all groups, repeated until ~budget_s of CPU time (at
    least one pass).  Returns (GB/s of algorithmic bytes, groups done, groups
    per pass, seconds)."""
    from oracle import relattn_oracle as O
    from paged_relative_bias_gb300.inputs import bf16_bits
    lens = case["seq_lens"].cpu().tolist()
    _, per_group = decode_work(wl, lens)
    g = wl.num_q_heads // wl.num_kv_heads
    q = bf16_bits(case["q"])
    rel = (bf16_bits(case["rel"]) if case["rel"].dtype == torch.bfloat16
           else case["rel"].cpu().numpy())
    table = case["block_table"].cpu().numpy()
    # each sequence's blocks, gathered once (host copies; not timed)
    per_seq = []
    for b in range(wl.batch):
        blocks = group_blocks(O, wl, lens[b], table[b])
        ids = torch.tensor([p for _, p in blocks], device=case["k_cache"].device)
        sub = np.full((1, table.shape[1]), -1, dtype=np.int64)
        for i, (lblk, _) in enumerate(blocks):
            sub[0, lblk] = i
        per_seq.append((cache_bits(case["k_cache"].index_select(0, ids)),
                        cache_bits(case["v_cache"].index_select(0, ids)), sub))
    groups = [(b, kvh) for b in range(wl.batch) for kvh in range(wl.num_kv_heads)]
    pool_data = dict(wl=wl, q=q, rel=rel, per_seq=per_seq, lens=lens, g=g,
                     k_scale=case.get("k_scale", 1.0), v_scale=case.get("v_scale", 1.0))
    done, nbytes, elapsed = 0, 0, 0.0
    while elapsed < budget_s or done == 0:
        for b, kvh in groups:
            kc, vc, sub = per_seq[b]
            heads = list(range(kvh * g, (kvh + 1) * g))
            t0 = time.perf_counter()
            oracle_group(O, wl, q, rel, b, kc, vc, sub, lens[b], heads,
                         case.get("k_scale", 1.0), case.get("v_scale", 1.0))
            elapsed += time.perf_counter() - t0
            done += 1
            nbytes += per_group[b]
            if elapsed >= budget_s and done >= len(groups):
                break
    pass_bytes = wl.num_kv_heads * sum(per_group)  # one pass: every (sequence, KV head)
    return nbytes / elapsed / 1e9, done, len(groups), elapsed, pool_data, pass_bytes


def cores_used():
    return int(os.environ.get("OMP_NUM_THREADS", "1"))


# --- the same oracle on every host core: one worker process per core, each
# taking (sequence, KV head) groups, one BLAS thread each
_POOL = None


def _pool_init(data):
    global _POOL
    _POOL = data


def _pool_group(bk):
    from oracle import relattn_oracle as O
    b, kvh = bk
    d = _POOL
    kc, vc, sub = d["per_seq"][b]
    heads = list(range(kvh * d["g"], (kvh + 1) * d["g"]))
    oracle_group(O, d["wl"], d["q"], d["rel"], b, kc, vc, sub, d["lens"][b], heads,
                 d["k_scale"], d["v_scale"])
    return b


def oracle_decode_all_cores(data, bytes_per_pass, budget_s):
    """Wall-clock GB/s of the oracle over whole passes of the workload, its
    (sequence, KV head) groups spread over a spawned pool of one process per
    host core.  Returns (GB/s, passes, cores, seconds)."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    groups = [(b, kvh) for b in range(len(data["lens"])) for kvh in range(data["wl"].num_kv_heads)]
    chunk = max(1, len(groups) // (4 * cores))
    with mp.get_context("spawn").Pool(cores, initializer=_pool_init, initargs=(data,)) as pool:
        pool.map(_pool_group, groups, chunksize=chunk)  # warm the workers
        passes, t0 = 0, time.perf_counter()
        while passes == 0 or time.perf_counter() - t0 < budget_s:
            pool.map(_pool_group, groups, chunksize=chunk)
            passes += 1
        el = time.perf_counter() - t0
    return passes * bytes_per_pass / el / 1e9, passes, cores, el


def prefill_workload(args):
    wl = I.WORKLOADS["chunked_prefill"]
    if args.rel == "bf16":
        wl = I.variant(wl, rel_dtype="bf16")
    if args.kv == "fp8":
        wl = I.variant(wl, kv_dtype="fp8")
    nseq = args.prefill_seqs or len(wl.new_tokens)
    new = args.prefill_new_tokens or wl.new_tokens[0]
    if (nseq, new) != (len(wl.new_tokens), wl.new_tokens[0]):
        wl = I.variant(wl, new_tokens=(new,) * nseq, ctx_lens=wl.ctx_lens[:1] * nseq)
    return wl


def ours_prefill(args, R, dist, device, peaks, sampler):
    """Chunked prefill as the timed step (TFLOP/s of visible pairs)."""
    wl = prefill_workload(args)
    flops, pbytes = prefill_work(wl)
    times = run_prefill(R, wl, device, args.steps, args.warmup, dist, sampler)
    t_ms = sum(times) / len(times)
    t_max = dist.max(sum(times))
    value = flops * dist.world * args.steps / (t_max / 1e3) / 1e12
    clocks = sampler.stop()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if wl.kv_dtype == "fp8" else "bf16",
        "data": f"synthetic (seeded N(0,1) q/k/v bf16, rel {wl.rel_dtype})",
        "config": {"workload": describe(wl),
                   "l2": "inputs larger than L2 (a step reads several GB), no flush",
                   "parallelism": f"replicas x{dist.world} (the path does not shard)"},
        "roofline": roofline("hbm", pbytes / (t_ms / 1e3) / 1e9, peaks["hbm"], "GB/s", None),
        "tensor_frac_of_bf16_peak": round(flops / (t_ms / 1e3) / 1e12 / peaks["bf16"], 4),
        "tensor_frac_of_bf16_sustained": round(
            flops / (t_ms / 1e3) / 1e12 / peaks["bf16_sustained"], 4),
        "peak_source": peaks["source"], "gpu_launches": 2 * args.steps, "clocks": clocks,
        "note": "step = cache write + attention kernels"}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


def ours(args):
    from paged_relative_bias_gb300 import build as B
    from paged_relative_bias_gb300 import relattn as R
    B.build()
    R.lib()
    dist = Dist()
    device = torch.device("cuda", dist.local)
    torch.cuda.set_device(device)
    peaks = load_peaks()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size

    sampler = ClockSampler(device.index)
    if args.workload == "chunked_prefill":
        return ours_prefill(args, R, dist, device, peaks, sampler)
    wl = I.WORKLOADS[args.workload]
    if args.rel == "bf16":
        wl = I.variant(wl, rel_dtype="bf16")
    if args.kv == "fp8":
        wl = I.variant(wl, kv_dtype="fp8")
    sets, step_bytes, times, wss = run_decode(R, wl, device, args.steps, args.warmup, dist,
                                              sampler, l2, args.pool == "shared")
    case = sets[0]
    t_ms = sum(times) / len(times)
    t_max = dist.max(sum(times))
    value = sum(step_bytes) * dist.world / (t_max / 1e3) / 1e9
    kernel_gbs = sum(step_bytes) / (sum(times) / 1e3) / 1e9
    e2e_times, h2d, d2h = run_decode_e2e(R, sets, wl, wss, device, args.steps, args.warmup,
                                         dist, sampler)
    e2e_max = dist.max(sum(e2e_times))
    e2e_value = sum(step_bytes) * dist.world / (e2e_max / 1e3) / 1e9
    n_sets = len(sets)
    l2_note = (f"inputs > L2: {n_sets} rotating sets x "
               f"{sum(step_bytes) / len(step_bytes) / 1e6:.1f} MB vs {l2 / 1e6:.0f} MB L2, "
               f"no flush; a graph replays the {n_sets} calls back to back")
    del sets

    secondary = []
    if not args.no_secondary:
        for key, name, rdt, kvd in SECONDARY_DECODE:
            w2 = I.variant(I.WORKLOADS[name], rel_dtype=rdt, kv_dtype=kvd)
            c2, b2, t2, _ = run_decode(R, w2, device, args.secondary_steps, 3, dist, sampler, l2)
            gbs = sum(b2) / (sum(t2) / 1e3) / 1e9
            secondary.append({
                "workload": key, "value": round(gbs, 1), "unit": "GB/s",
                "ms_per_step": round(sum(t2) / len(t2), 5),
                "roofline": {"bound": "hbm", "frac": round(gbs / peaks["hbm"], 4)}})
            del c2
            torch.cuda.empty_cache()
        wp0 = prefill_workload(args)
        for key, rdt, kvd in SECONDARY_PREFILL:
            wp = I.variant(wp0, rel_dtype=rdt, kv_dtype=kvd)
            secondary.append(prefill_entry(key, wp, run_prefill(
                R, wp, device, max(3, args.secondary_steps // 4), 2, dist, sampler), peaks))
            torch.cuda.empty_cache()
        wt = I.WORKLOADS["tiny_prefill"]
        secondary.append(prefill_entry("cfg1_tiny", wt, run_prefill_graph(
            R, wt, device, args.secondary_steps, dist, sampler), peaks))
    clocks = sampler.stop()

    cpu = None
    if dist.world == 1 and not args.no_cpu_baseline:
        gbs, done, total, el, pool_data, pass_bytes = oracle_decode_sample(case, wl,
                                                                           args.cpu_budget)
        cpu = {"value": round(gbs, 6), "unit": "GB/s", "cores": cores_used(), "kind": "oracle",
               "sample": f"{done} (sequence, KV head) groups, {done / total:.1f} passes over "
                         f"the workload's {total}, float64 numpy, {el:.2f} s of CPU time"}
        if args.cpu_all_cores > 0:
            gall, passes, ncores, el2 = oracle_decode_all_cores(pool_data, pass_bytes,
                                                                args.cpu_all_cores)
            cpu["all_cores"] = {
                "value": round(gall, 6), "unit": "GB/s", "cores": ncores,
                "sample": f"{passes} whole passes over the workload's {total} groups, "
                          f"spread over {ncores} spawned processes (one BLAS thread "
                          f"each), {el2:.2f} s wall"}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v bf16, rel fp32)",
        "config": {"workload": describe(wl), "l2": l2_note,
                   "layers": ("a set per layer: own KV pool, q, rel; shared seq_lens and "
                              "block table" if args.pool == "per-set" else
                              "sets share one KV pool, own q, rel, renumbered table"),
                   "parallelism": f"replicas x{dist.world} (the path does not shard)"},
        "roofline": roofline("hbm", kernel_gbs, peaks["hbm"], "GB/s",
                             committed_traffic("decode_" + args.workload)),
        "peak_source": peaks["source"],
        "frac_of_nominal_8000": round(kernel_gbs / 8000.0, 4),
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(sum(e2e_times) / len(e2e_times), 5),
                "pipeline": "2 input and 2 output buffers; H2D, kernel, D2H streams; "
                            "a pass of steps replayed as a CUDA graph"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "secondary": secondary,
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


# ---------------------------------------------------------------------------
# reference arm: the oracle on host cores
# ---------------------------------------------------------------------------

def reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import relattn_oracle as O
    from paged_relative_bias_gb300.inputs import bf16_bits
    wl = I.WORKLOADS[args.workload]
    if args.rel == "bf16":
        wl = I.variant(wl, rel_dtype="bf16")
    if args.kv == "fp8":
        wl = I.variant(wl, kv_dtype="fp8")
    device = "cuda" if torch.cuda.is_available() else "cpu"
    case = I.make_decode(wl, device)
    lens = case["seq_lens"].cpu().tolist()
    _, per_group = decode_work(wl, lens)
    g = wl.num_q_heads // wl.num_kv_heads
    q = bf16_bits(case["q"])
    rel = (bf16_bits(case["rel"]) if case["rel"].dtype == torch.bfloat16
           else case["rel"].cpu().numpy())
    table = case["block_table"].cpu().numpy()
    groups = [(b, kvh) for b in range(wl.batch) for kvh in range(wl.num_kv_heads)]
    prepared = []
    for b in range(wl.batch):
        blocks = group_blocks(O, wl, lens[b], table[b])
        ids = torch.tensor([p for _, p in blocks], device=case["k_cache"].device)
        sub = np.full((1, table.shape[1]), -1, dtype=np.int64)
        for i, (lblk, _) in enumerate(blocks):
            sub[0, lblk] = i
        prepared.append((cache_bits(case["k_cache"].index_select(0, ids)),
                         cache_bits(case["v_cache"].index_select(0, ids)), sub))

    def step(i):
        b, kvh = groups[i % len(groups)]
        kc, vc, sub = prepared[b]
        oracle_group(O, wl, q, rel, b, kc, vc, sub, lens[b], list(range(kvh * g, (kvh + 1) * g)),
                     case.get("k_scale", 1.0), case.get("v_scale", 1.0))
        return per_group[b]

    for i in range(args.warmup):
        step(i)
    nbytes = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        nbytes += step(args.warmup + i)
    el = time.perf_counter() - t0
    value = nbytes / el / 1e9
    sample = (f"each step: one (sequence, KV head) group of the workload "
              f"({g} query heads over its window), float64 numpy oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(wl), "l2": "n/a (host)", "parallelism": "host"},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": cores_used(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="local_decode",
                    choices=["local_decode", "global_decode_b1", "global_decode_b8",
                             "diffhead_decode", "verify_decode", "chunked_prefill"])
    ap.add_argument("--prefill-new-tokens", type=int, default=0,
                    help="new tokens per sequence of the chunked prefill (default 8192)")
    ap.add_argument("--prefill-seqs", type=int, default=0,
                    help="sequences of the chunked prefill (default 4)")
    ap.add_argument("--rel", choices=["f32", "bf16"], default="f32",
                    help="element type of the rel input of the timed workload")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="element type of the KV cache of the timed workload (decode or "
                         "prefill)")
    ap.add_argument("--pool", choices=["per-set", "shared"], default="per-set",
                    help="decode input sets: one KV pool each (default), or one shared pool "
                         "with renumbered block tables (small device footprint, for ncu)")
    ap.add_argument("--secondary-steps", type=int, default=50)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--cpu-all-cores", type=float, default=8.0,
                    help="seconds of wall time for the oracle on every host core (0: skip)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        reference(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
