"""Benchmark: paged split-KV GQA decode attention on GB300.

One step is one pass of the whole decode hot path over one batch of
synthetic input, as a Gemma-4-31B-shaped decode step runs it:
  * the global-layer decode (32 query heads on 4 KV heads, head dim 512,
    bf16 K/V in shuffled pages of 256) at each of the contexts 10,602,
    40,002, 81,653 and 163,336: the step's new K/V row is written into its
    page by the decode's own partial kernel, which then computes the
    split-KV partials, and the two-level merge combines them;
  * the sliding-window decode (32 query heads on 16 KV heads, head dim 256,
    window 1,024, pages of 64, resident length window + one page), the
    same way.
value = algorithmic bytes (K and V of every attended key) / step time, GB/s.

Timing: W untimed warm-up steps, then K steps between CUDA events on the
launching stream, with a barrier and a device synchronize on both sides;
consecutive steps read three rotating copies of the pools (2.4 GB of K/V a
step, far beyond the 129 MB L2), so no call finds its data in L2.  The timed
steps are replays of CUDA graphs captured once (one per pool copy) from the
same library calls, as a decode engine runs its step.  The partial kernels'
durations for the roofline come from a further pass of K eager steps with
CUDA events recorded around each partial launch.  Per call, with a cold L2
(a 256 MB read before every call): microseconds -- one graph of ten (read,
call) pairs less ten reads alone, per call; and the call's own graph replayed
alone between two events (us_iso, which adds an idle GPU's event and launch
latency) -- GB/s, the fraction of 8 TB/s and of the measured copy bandwidth,
and the time per call back to back (a graph of calls over pool copies that
hold more than twice the L2); the split count swept over 8..256 at every
global context with the best one reported.  e2e: the same step through the library's C entry
points (eager calls, no graphs), with each step's inputs copied in from
pinned host memory and its outputs copied back inside the timed region.

--impl reference times the CPU oracle (an fp64 direct softmax over the
paged pool, run on the host's cores) on the same workload: the pages this
method comes from ship no runnable code, so the oracle is the only
reference implementation there is.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "decode attn µs/call & effective HBM GB/s (% of 8 TB/s) at 10.6K–163K ctx"
FALLBACK_HBM_GBS = 6800.0
DEFAULT_CONTEXTS = (10602, 40002, 81653, 163336)
DEFAULT_SWEEP = (8, 16, 32, 64, 128, 256)
NOMINAL_HBM_GBS = 8000.0  # the metric's denominator (GB300 HBM3e, nominal)
WINDOW_RESIDENCY = W.WINDOW + 64
ROTATE = 3
PARTIAL_SOURCES = ("paged_split_kv_attn_gb300/csrc/partial_kernel.cuh",
                   "paged_split_kv_attn_gb300/csrc/partial_mma.cuh",
                   "paged_split_kv_attn_gb300/csrc/partial_mma.cu",
                   "paged_split_kv_attn_gb300/csrc/pskv_internal.cuh")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "partial_mma_d512_ctx40002.md")


def partial_kernel_hash() -> str:
    """Hash of the partial kernel's code (comments and blank space left out, so
    that editing a comment keeps the recorded counters valid)."""
    import re
    h = hashlib.sha256()
    for rel in PARTIAL_SOURCES:
        with open(os.path.join(ROOT, rel)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak() -> float:
    """Dense bf16 TFLOP/s from the measured-peaks file (burst), else the fallback figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def recorded_traffic():
    """DRAM bytes per key of the partial kernel from the committed ncu summary,
    or None when the kernel source changed since the counters were taken."""
    rec = {}
    try:
        with open(TRAFFIC_FILE) as f:
            for line in f:
                key, _, val = line.strip().partition(":")
                if key in ("dram_bytes_per_key", "source_hash"):
                    rec[key] = val.strip()
    except OSError:
        return None
    if rec.get("source_hash") != partial_kernel_hash() or "dram_bytes_per_key" not in rec:
        return None
    return float(rec["dram_bytes_per_key"])


# ---- distributed plumbing (replicas only: every rank runs the same step) ----------

class Dist:
    """Rank bookkeeping for `--gpus N` under torchrun: N independent replicas of
    the step, a barrier around the timed region and the max time over ranks.
    NCCL on GPUs; gloo when `backend="gloo"` (the CPU tests use it)."""

    def __init__(self, backend: str | None = None):
        import torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.backend = backend or "nccl"
        if self.world > 1:
            import torch.distributed as dist
            if self.backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(self.backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64,
                         device="cuda" if self.backend == "nccl" else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def whole_job_gbps(step_bytes: int, world: int, ms_per_step_max: float) -> float:
    """Whole-job throughput: the bytes all ranks processed per step over the
    slowest rank's step time (every rank runs the same step)."""
    return step_bytes * world / (ms_per_step_max * 1e-3) / 1e9


# ---- clocks --------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"pskv_clocks_rank{device_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
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
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ---- the workload ----------------------------------------------------------------

_CASES: dict = {}


def global_case(ctx: int, seed: int | None = None):
    """The global-layer decode case at `ctx` keys (made once per process)."""
    seed = ctx if seed is None else seed
    key = ("global", ctx, seed)
    if key not in _CASES:
        _CASES[key] = W.global_case(ctx, seed=seed)
    return _CASES[key]


def window_case():
    """The sliding-window decode case at residency window + one page."""
    key = ("window", WINDOW_RESIDENCY)
    if key not in _CASES:
        _CASES[key] = W.window_case(WINDOW_RESIDENCY, seed=7)
    return _CASES[key]


class Call:
    """One decode call of the step: a pool (and rotating copies), its inputs and outputs.

    With ``prep`` the step's new tokens arrive as projection rows: the fused
    K/V prep normalises and rotates them, writes K and V into their pages and
    the prepared queries into ``q`` (one launch); without it the K/V rows are
    copied into the pages as they are (kv_append_rows) and ``q`` is given."""

    def __init__(self, name, case, windowed, splits, dev, rotate, tokens=1, prep=False,
                 fused=False, tree=False):
        import torch
        import paged_split_kv_attn_gb300 as pskv
        self.name, self.case, self.windowed = name, case, windowed
        self.tokens = tokens  # query tokens per row: > 1 is a verify window (multi-row decode)
        self.splits = splits
        self.prep = prep
        self.fused = fused and tokens == 1 and not prep  # the append inside the decode
        bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
            torch.bfloat16).to(dev)
        f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
        k0, v0 = bf(case.k_pool), bf(case.v_pool)
        self.k = [k0] + [k0.clone() for _ in range(rotate - 1)]
        self.v = [v0] + [v0.clone() for _ in range(rotate - 1)]
        self.status = torch.zeros(4, dtype=torch.int32, device=dev)
        self.layouts = [pskv.paged_kv_layout_create(k, v, self.status)
                        for k, v in zip(self.k, self.v)]
        self.q = bf(case.q if tokens == 1 else W.window_queries(case, tokens))
        # a drafted tree over the window (one seeded tree per row), else a causal window
        self.tree_mask = None if not tree else torch.from_numpy(np.ascontiguousarray(np.stack(
            [W.tree_masks(W.random_tree_parents(b, tokens)) for b in range(case.batch)]))
            .view(np.int64)).to(dev)
        self.tables = torch.from_numpy(case.page_tables).to(dev)
        self.lens = torch.from_numpy(case.seq_lens).to(dev)
        self.lens_host = case.seq_lens.copy()
        self.pages_of_row = torch.from_numpy(case.pages_of_row).to(dev)
        self.first_pos = None if case.first_pos is None else torch.from_numpy(case.first_pos).to(dev)
        self.window_lo = None if case.window_lo is None else torch.from_numpy(case.window_lo).to(dev)
        b, hq, d = case.q.shape
        hkv = case.num_kv_heads
        # the step's new tokens: the last `tokens` positions of each row
        self.rows = [r for r in range(b) for _ in range(tokens)]
        self.pos = [int(case.seq_lens[r]) - tokens + t for r in range(b) for t in range(tokens)]
        self.row_of = torch.tensor(self.rows, dtype=torch.int32, device=dev)
        self.pos_of = torch.tensor(self.pos, dtype=torch.int32, device=dev)
        ps = case.page_size
        self.k_new = torch.stack([k0[int(case.page_tables[r, p // ps]), :, p % ps]
                                  for r, p in zip(self.rows, self.pos)]).contiguous()
        self.v_new = torch.stack([v0[int(case.page_tables[r, p // ps]), :, p % ps]
                                  for r, p in zip(self.rows, self.pos)]).contiguous()
        if prep:
            # global layers: K and V from one projection row, the first quarter
            # rotated; sliding layers: separate bands, the whole head rotated
            fp = 0 if case.first_pos is None else int(case.first_pos.max())
            rot = d if windowed else case.k_pool.shape[3] if case.folded else d // 4
            self.prep_in = W.make_prep_inputs(len(self.rows) + hq, len(self.rows), hq, hkv, d, rot,
                                              fp + int(case.seq_lens.max()),
                                              shared_kv=not windowed)
            pi = self.prep_in
            self.x = bf(pi.x)
            self.w_q, self.w_k = f32(pi.w_q), f32(pi.w_k)
            self.rope_cos, self.rope_sin = f32(pi.rope_cos), f32(pi.rope_sin)
        self.out = torch.empty(tuple(self.q.shape[:-1]) + (d,), dtype=torch.bfloat16, device=dev)
        self.ws = pskv.workspace(b * tokens, hq, d, splits, dev)
        self.bytes = case.kv_bytes()
        self.partial_bytes_per_launch = self.bytes
        self.hkv = hkv

    def step_inputs(self) -> dict:
        """The tensors a decode step brings from the host (rebound by pack())."""
        if self.prep:
            return {"x": self.x, "pos_of": self.pos_of}
        return {"q": self.q, "k_new": self.k_new, "v_new": self.v_new, "pos_of": self.pos_of}

    def run(self, it: int, events=None):
        import paged_split_kv_attn_gb300 as pskv
        layout = self.layouts[it % len(self.layouts)]
        if self.prep:
            pi = self.prep_in
            n, hq, d = len(self.rows), self.q.shape[-2], self.q.shape[-1]
            pskv.kv_prep_append(layout, self.x, pi.q_col, pi.k_col, pi.v_col, hq, self.row_of,
                                self.pos_of, self.tables, self.pages_of_row, pi.rot, pi.eps,
                                w_q=self.w_q, w_k=self.w_k, rope_cos=self.rope_cos,
                                rope_sin=self.rope_sin, first_pos=self.first_pos,
                                q_out=self.q.view(n, hq, d))
        elif not self.fused:
            pskv.kv_append_rows(layout, self.k_new, self.v_new, self.row_of, self.pos_of,
                                self.tables, self.pages_of_row)
        app = (self.k_new, self.v_new, self.pages_of_row) if self.fused else None
        if self.tree_mask is not None:
            pskv.decode_attn_tree(layout, self.q, self.tables, self.lens, self.lens_host,
                                  self.tree_mask, self.case.scale, num_splits=self.splits,
                                  workspace=self.ws, out=self.out, events=events)
        elif self.tokens > 1:
            pskv.decode_attn_multirow(layout, self.q, self.tables, self.lens, self.lens_host,
                                      self.case.scale, num_splits=self.splits, workspace=self.ws,
                                      out=self.out, events=events)
        elif self.windowed:
            pskv.decode_attn_windowed(layout, self.q, self.tables, self.lens, self.lens_host,
                                      self.first_pos, self.window_lo, self.case.scale,
                                      num_splits=self.splits, workspace=self.ws, out=self.out,
                                      events=events, append=app)
        else:
            pskv.decode_attn_splitkv(layout, self.q, self.tables, self.lens, self.lens_host,
                                     self.case.scale, num_splits=self.splits, workspace=self.ws,
                                     out=self.out, events=events, append=app)



class Packed:
    """The step's small per-step tensors (queries, new K/V rows, positions; and
    the outputs) packed into one device buffer each way, with pinned host
    twins, so the end-to-end step moves them with one copy in and one out.

    Two sets of device buffers alternate between steps, so that step i+1's
    inputs can be copied in while step i computes and step i's outputs are
    copied out while step i+1 computes (a copy stream each way)."""

    def __init__(self, calls, dev):
        import torch
        def pack(items):
            offs, total = [], 0
            for t in items:
                offs.append(total)
                total += (t.numel() * t.element_size() + 255) // 256 * 256
            buf = torch.empty(total, dtype=torch.uint8, device=dev)
            views = []
            for t, off in zip(items, offs):
                n = t.numel() * t.element_size()
                v = buf[off:off + n].view(t.dtype).view(t.shape)
                v.copy_(t)
                views.append(v)
            return buf, views
        self.calls = calls
        ins = [(c, k, t) for c in calls for k, t in c.step_inputs().items()]
        self.keys = [(c, k) for c, k, _ in ins]
        self.dev_in, self.in_views, self.dev_out, self.out_views = [], [], [], []
        for _ in range(2):
            buf, views = pack([t for _, _, t in ins])
            self.dev_in.append(buf)
            self.in_views.append(views)
            buf, views = pack([c.out for c in calls])
            self.dev_out.append(buf)
            self.out_views.append(views)
        self.bind(0)
        torch.cuda.synchronize()
        self.host_in = self.dev_in[0].cpu().pin_memory()
        self.host_out = [torch.empty_like(self.dev_out[0], device="cpu").pin_memory()
                         for _ in range(2)]
        self.h2d_stream, self.d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
        self.h2d_done = [torch.cuda.Event() for _ in range(2)]
        self.computed = [torch.cuda.Event() for _ in range(2)]
        self.d2h_done = [torch.cuda.Event() for _ in range(2)]

    def bind(self, parity: int):
        """Point the calls' step tensors at buffer set `parity`."""
        for (c, k), v in zip(self.keys, self.in_views[parity]):
            setattr(c, k, v)
        for c, v in zip(self.calls, self.out_views[parity]):
            c.out = v

    def step_e2e(self, it: int, run_step, started):
        """Copy step `it`'s inputs in, run it (run_step(it, parity)), copy its
        outputs out; `started` is an event recorded where the timed region starts."""
        import torch
        p = it % 2
        compute = torch.cuda.current_stream()
        with torch.cuda.stream(self.h2d_stream):
            self.h2d_stream.wait_event(started)
            if it >= 2:
                self.h2d_stream.wait_event(self.computed[p])  # step it-2 has used these inputs
            self.dev_in[p].copy_(self.host_in, non_blocking=True)
            self.h2d_done[p].record(self.h2d_stream)
        compute.wait_event(self.h2d_done[p])
        if it >= 2:
            compute.wait_event(self.d2h_done[p])  # step it-2's outputs have left this buffer
        run_step(it, p)
        self.computed[p].record(compute)
        with torch.cuda.stream(self.d2h_stream):
            self.d2h_stream.wait_event(self.computed[p])
            self.host_out[p].copy_(self.dev_out[p], non_blocking=True)
            self.d2h_done[p].record(self.d2h_stream)

    def finish(self, it_last: int):
        """Make the compute stream wait for the last outputs to reach the host."""
        import torch
        torch.cuda.current_stream().wait_event(self.d2h_done[it_last % 2])


class PrefillCall:
    """A paged prefill timed beside the step: each row's last `chunk` keys are
    its new tokens (already in the pool), each attending keys up to itself
    (within `window` keys when > 0)."""

    def __init__(self, name, case, chunk, window, dev):
        import torch
        import paged_split_kv_attn_gb300 as pskv
        self.name, self.case, self.chunk, self.window = name, case, chunk, window
        bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
            torch.bfloat16).to(dev)
        self.status = torch.zeros(4, dtype=torch.int32, device=dev)
        self.k, self.v = bf(case.k_pool), bf(case.v_pool)
        self.layout = pskv.paged_kv_layout_create(self.k, self.v, self.status)
        b, hq, d = case.q.shape
        counts = [min(chunk, int(n)) for n in case.seq_lens]
        self.cu_host = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        self.cu = torch.from_numpy(self.cu_host).to(dev)
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([chunk, 11])))
        self.q = bf(W.bf16_bits(rng.standard_normal((int(self.cu_host[-1]), hq, d),
                                                    dtype=np.float32)))
        self.tables = torch.from_numpy(case.page_tables).to(dev)
        self.lens = torch.from_numpy(case.seq_lens).to(dev)
        self.lens_host = case.seq_lens.copy()
        self.out = torch.empty_like(self.q)
        self.tokens = int(self.cu_host[-1])
        # algorithmic FLOPs: 2 D (scores) + 2 D (values) per visible (token, key, q head)
        vis = 0
        for L, T in zip(case.seq_lens, counts):
            own = np.arange(int(L) - T, int(L), dtype=np.int64)
            seen = own + 1 if window == 0 else np.minimum(own + 1, window)
            vis += int(seen.sum())
        self.flops = 4 * hq * d * vis

    def run(self, it: int, events=None):
        import paged_split_kv_attn_gb300 as pskv
        pskv.prefill_attn_paged(self.layout, self.q, self.cu, self.cu_host, self.tables,
                                self.lens, self.lens_host, self.case.scale, window=self.window,
                                out=self.out, events=events)


def make_prefill_calls(args, dev):
    """--prefill specs: family:context:chunk[:window]."""
    calls = []
    for spec in args.prefill:
        fam, ctx, chunk, *rest = spec.split(":")
        ctx, chunk, window = int(ctx), int(chunk), int(rest[0]) if rest else 0
        shape = W.GLOBAL_SHAPE if fam == "global" else W.WINDOW_SHAPE
        case = W.make_paged_case(ctx + chunk, [ctx], dtype="bf16", **shape)
        calls.append(PrefillCall(f"prefill_{fam}_{ctx}x{chunk}" + (f"_w{window}" if window else ""),
                                 case, chunk, window, dev))
    return calls


def make_extra_calls(args, dev):
    """Calls measured one at a time beside the step: the folded format, verify
    windows of the global shape (multi-row decode) and a ragged batch."""
    prep, fused = args.append == "prep", args.append == "fused"
    calls = [Call(f"folded_{ctx}", W.folded_case(ctx, seed=ctx + 1), False, args.splits, dev,
                  ROTATE, prep=prep, fused=fused) for ctx in args.folded_contexts]
    for t in args.verify_tokens:
        ctx = args.verify_context
        calls.append(Call(f"verify_{ctx}x{t}", global_case(ctx, ctx + 2), False,
                          args.splits, dev, ROTATE, tokens=t, prep=prep))
    for t in args.tree_tokens:
        ctx = args.verify_context
        calls.append(Call(f"tree_{ctx}x{t}", global_case(ctx, ctx + 3), False,
                          args.splits, dev, ROTATE, tokens=t, prep=prep, tree=True))
    if not args.no_ragged:
        calls.append(Call("ragged16", W.ragged_case(0), False, args.splits, dev, ROTATE,
                          prep=prep, fused=fused))
    return calls


def make_calls(args, dev):
    calls, prep, fused = [], args.append == "prep", args.append == "fused"
    for ctx in args.contexts:
        calls.append(Call(f"global_{ctx}", global_case(ctx), False, args.splits, dev,
                          ROTATE, prep=prep, fused=fused))
    if not args.no_window:
        calls.append(Call(f"window_{WINDOW_RESIDENCY}", window_case(),
                          True, args.window_splits, dev, ROTATE, prep=prep, fused=fused))
    return calls


# ---- CPU baseline: the oracle on a bounded sample ----------------------------------

def cpu_baseline(cases, budget_s: float):
    import oracle
    done_bytes, reps, t0 = 0, 0, time.perf_counter()
    while True:
        for c in cases:
            oracle.decode_direct(c.q, c.k_pool, c.v_pool, c.page_tables, c.seq_lens, c.scale,
                                 c.first_pos, c.window_lo)
            done_bytes += c.kv_bytes()
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": done_bytes / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{reps} passes of the step's {len(cases)} calls "
                      f"({'/'.join(str(int(c.seq_lens.sum())) for c in cases)} keys), "
                      f"fp64 direct softmax, {dt:.1f} s"}


# ---- main ----------------------------------------------------------------------------

def parse():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--contexts", type=int, nargs="+", default=list(DEFAULT_CONTEXTS))
    ap.add_argument("--splits", type=int, default=0, help="global-layer split count (0 = auto)")
    ap.add_argument("--window-splits", type=int, default=0)
    ap.add_argument("--no-window", action="store_true")
    ap.add_argument("--no-ragged", action="store_true",
                    help="skip the 16-row ragged batch timed beside the step")
    ap.add_argument("--append", choices=["fused", "copy", "prep"], default="fused",
                    help="new tokens of the step: K/V rows written by the decode itself, "
                         "copied into the pages by a separate launch, or projection rows "
                         "through the fused K/V prep")
    ap.add_argument("--no-prep-step", action="store_true",
                    help="skip timing the step with the fused K/V prep beside the headline step")
    ap.add_argument("--folded-contexts", type=int, nargs="*", default=[40002],
                    help="contexts of the folded-format decode timed beside the step")
    ap.add_argument("--verify-tokens", type=int, nargs="*", default=[2, 4, 8],
                    help="verify-window lengths of the multi-row decode timed beside the step")
    ap.add_argument("--tree-tokens", type=int, nargs="*", default=[8],
                    help="drafted-tree sizes (tree attention) timed beside the step")
    ap.add_argument("--verify-context", type=int, default=40002,
                    help="context of those verify windows (global-layer shape)")
    ap.add_argument("--prefill", nargs="*",
                    default=["global:10602:512", "global:4096:4096", "sliding:4096:4096:1024"],
                    help="paged prefills timed beside the step: family:context:chunk[:window]")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="time eager stream launches instead of CUDA graph replays")
    ap.add_argument("--sweep", type=int, nargs="*", default=list(DEFAULT_SWEEP),
                    help="split counts each global context is also timed at alone "
                         "(the automatic plan is always added); none to skip")
    ap.add_argument("--detail", default=None,
                    help="also write every per-call figure (unrounded) to this JSON file")
    return ap.parse_args()


def reference_arm(args):
    """The CPU oracle on the same workload, each step a full pass (bounded by K)."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import oracle
    cases = [global_case(ctx) for ctx in args.contexts]
    if not args.no_window:
        cases.append(window_case())
    nbytes = sum(c.kv_bytes() for c in cases)
    for _ in range(min(args.warmup, 1)):
        for c in cases:
            oracle.decode_direct(c.q, c.k_pool, c.v_pool, c.page_tables, c.seq_lens, c.scale,
                                 c.first_pos, c.window_lo)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for c in cases:
            oracle.decode_direct(c.q, c.k_pool, c.v_pool, c.page_tables, c.seq_lens, c.scale,
                                 c.first_pos, c.window_lo)
    dt = (time.perf_counter() - t0) / args.steps
    value = nbytes / dt / 1e9
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": config_dict(args),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": f"{args.steps} full step(s) of the workload"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(args):
    """The workload, named by what it is (kept short: the line must fit a log tail)."""
    wl = ("gemma4-31b decode step: global layer (32q/4kv, hd512, pages 256) at "
          + "/".join(str(c) for c in args.contexts)
          + ("" if args.no_window else
             f" + sliding layer (32q/16kv, hd256, W{W.WINDOW}, pages 64) at {WINDOW_RESIDENCY}"))
    return {"workload": wl, "batch": 1, "splits": args.splits or "auto",
            "new_tokens": {"prep": "fused K/V prep (norm, rotation, page write) per call",
                           "copy": "kv_append_rows per call",
                           "fused": "row written by the decode's own partial kernel"}[args.append],
            "kv": "bf16, f32 accumulate, bf16 out",
            "l2": f"inputs larger than L2: {ROTATE} rotating pool copies",
            "parallelism": "replicas"}


def r1(x):
    """Round for the printed line (full precision goes to --detail)."""
    return None if x is None else round(float(x), 1)


LINE_BUDGET = 2900  # characters of the printed line: a log tail keeps about 3,000


def make_line(args, world, value, ms, launches, roofline, e2e, clock_info, step_ms, detail,
              sweep, prefill) -> dict:
    """The printed JSON line: the contract's keys, then the per-call figures in
    compact rows (cold L2: us from a sequence of reads and calls, us of the call
    alone between events, GB/s, % of 8 TB/s, % of the measured copy peak, splits,
    partial-kernel us; then us per call back to back), the split
    sweep (us at each count, then the best count) and prefill TFLOP/s."""
    per_call = {"cols": ["us", "us_iso", "GBps", "pct_8TBs", "pct_meas", "P", "partial_us",
                         "us_b2b"]}
    for name, d in detail.items():
        per_call[name] = [r1(d["us_per_call"]), r1(d["us_isolated"]), round(d["GBps_per_call"]),
                          r1(100 * d["frac_of_8TBs"]), r1(100 * d["frac_of_measured"]),
                          d["splits"], r1(d["partial_us"]), r1(d["us_stream"])]
    line = {"metric": METRIC, "value": r1(value), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": config_dict(args), "gpu_launches": int(launches),
            "roofline": roofline, "e2e": e2e, "clocks": clock_info, "step_ms": step_ms,
            "per_call": per_call}
    if sweep:
        line["sweep_us"] = {"P": list(args.sweep)}
        for name, sw in sweep.items():
            line["sweep_us"][name] = [r1(sw["us"][p]) for p in args.sweep] + [sw["best_splits"]]
    if prefill:
        line["prefill_tflops"] = {k.replace("prefill_", ""): round(v["tflops"]) for k, v in
                                  prefill.items()}
    return line


def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
        return
    import torch
    import paged_split_kv_attn_gb300 as pskv
    from paged_split_kv_attn_gb300 import build as lib_build

    dist = Dist()
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    lib_build.build()
    pskv.load_library()
    calls = make_calls(args, dev)
    packed = Packed(calls, dev)
    stream = torch.cuda.current_stream()
    step_bytes = sum(c.bytes for c in calls)
    peak, peak_kind = measured_peak()

    # per-call partial-kernel events (recorded by the library around the partial launch)
    ev = {c.name: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)] for c in calls}
    for c in calls:
        for b, e in ev[c.name]:
            b.record()
            e.record()
    for it in range(args.warmup):
        for c in calls:
            c.run(it)
    torch.cuda.synchronize()
    for c in calls:
        if c.status[0].item() != 0:
            raise RuntimeError(f"{c.name}: device fault word {c.status[0].item()}")

    def capture(step_calls):
        """One CUDA graph per pool copy of the given calls, captured once; returns
        (graphs, library launches per replay)."""
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for c in step_calls:  # warm the capture path (plans, attributes) outside capture
                c.run(0)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        n0 = pskv.pskv_kernel_launches()
        gs = []
        for r in range(ROTATE):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for c in step_calls:
                    c.run(r)
            gs.append(g)
        per = (pskv.pskv_kernel_launches() - n0) / ROTATE
        for g in gs:
            g.replay()
        torch.cuda.synchronize()
        return gs, per

    # ---- the step as CUDA graphs: one graph per pool copy, captured once
    graphs = None
    if not args.eager:
        graphs, launches_per_step = capture(calls)

    def timed(run_step, steps=None):
        """K steps between events on the stream, barrier and synchronize on both sides."""
        steps = args.steps if steps is None else steps
        dist.barrier()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for it in range(steps):
            run_step(it)
        t1.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        return dist.max(t0.elapsed_time(t1) / steps)

    def eager_step(it):
        for c in calls:
            c.run(it)

    def keep_busy(seconds: float):
        """Replay the step for about `seconds`, so that the clock samples taken
        around the timed region see the GPU under this load."""
        t_end = time.perf_counter() + seconds
        it = 0
        while time.perf_counter() < t_end:
            for _ in range(16):
                if graphs is not None:
                    graphs[it % ROTATE].replay()
                else:
                    eager_step(it)
                it += 1
            torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    keep_busy(0.4)
    launches0 = pskv.pskv_kernel_launches()
    if graphs is not None:
        ms = timed(lambda it: graphs[it % ROTATE].replay())
        launches = int(round(launches_per_step * args.steps))
    else:
        ms = timed(eager_step)
        launches = pskv.pskv_kernel_launches() - launches0
    keep_busy(0.2)
    clock_info = clocks.stop()
    clock_info["window"] = "every 100 ms: 0.4 s before the timed steps, them, 0.2 s after"
    value = whole_job_gbps(step_bytes, dist.world, ms)
    eager_ms = ms if graphs is None else timed(eager_step)

    # ---- end to end through the C entry points: eager library calls each step
    # (no graphs), each step's inputs copied in from pinned host memory (one
    # packed copy) and its outputs copied back (one copy), inside the timed
    # region; the copies of neighbouring steps overlap the step in between
    def run_e2e(it, parity):
        packed.bind(parity)
        for c in calls:
            c.run(it)

    def timed_e2e(steps):
        dist.barrier()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for it in range(steps):
            packed.step_e2e(it, run_e2e, t0)
        packed.finish(steps - 1)
        t1.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        return dist.max(t0.elapsed_time(t1) / steps)

    timed_e2e(max(args.warmup, 2))
    e2e_ms = timed_e2e(args.steps)
    packed.bind(0)
    for c in calls:
        if c.status[0].item() != 0:
            raise RuntimeError(f"{c.name}: device fault word {c.status[0].item()}")

    # ---- the partial kernels' durations: a pass of K eager steps with CUDA
    # events recorded by the library right around each partial launch
    for it in range(args.steps):
        for c in calls:
            c.run(it, events=ev[c.name][it])
    torch.cuda.synchronize()
    detail = {}
    for c in calls:
        part = statistics.mean([b.elapsed_time(e) for b, e in ev[c.name]])
        detail[c.name] = {"kv_bytes": c.bytes, "partial_us": 1e3 * part,
                          "partial_GBps": c.bytes / (part * 1e-3) / 1e9}

    # ---- calls timed beside the step (not in value): partial kernel alone by events
    extra = make_extra_calls(args, dev)
    for c in extra:
        pe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for it in range(args.warmup):
            c.run(it)
        for it in range(args.steps):
            c.run(it, events=pe[it])
        torch.cuda.synchronize()
        part = statistics.mean([b.elapsed_time(e) for b, e in pe])
        detail[c.name] = {"kv_bytes": c.bytes, "partial_us": 1e3 * part,
                          "partial_GBps": c.bytes / (part * 1e-3) / 1e9}

    # ---- each call alone, replayed from its own graphs with a cold L2 (a 256 MB
    # buffer is READ between calls: reads leave no dirty lines to write back)
    flush = torch.ones(int(256e6) // 4, dtype=torch.float32, device=dev)

    def graph_of(fn):
        """fn() captured once as a CUDA graph (after one run outside capture)."""
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        g.replay()
        torch.cuda.synchronize()
        return g

    def replay_us(g, reps=7):
        """Median duration of a graph replay between events on the stream."""
        ts = []
        for _ in range(reps):
            b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b.record(stream)
            g.replay()
            e.record(stream)
            torch.cuda.synchronize()
            ts.append(b.elapsed_time(e) * 1e3)
        return statistics.median(ts)

    SEQ = 10  # (read, call) pairs per graph in the cold per-call figure
    g_reads = graph_of(lambda: [flush.sum() for _ in range(SEQ)])
    read_us = replay_us(g_reads) / SEQ  # one 256 MB read, as it runs inside the sequence

    def per_call_us(c, reps, seq=SEQ):
        """One call at a time with a cold L2, two ways.

        us: one graph of `seq` (256 MB read, call) pairs over the rotating pool
        copies, its replay time less that of `seq` reads alone, per call -- the
        call's device time with a cold L2 and cold code, its launches queued as
        an engine queues them.
        us_iso: the call's own graph replayed alone after a 256 MB read, between
        two events (mean of `reps`; the event clock ticks in ~1 us steps); this
        adds the event and graph-launch latency of an idle GPU (a graph of one
        trivial kernel measures ~5-7 us this way)."""
        g = graph_of(lambda: [(flush.sum(), c.run(r % ROTATE)) for r in range(seq)])
        us_seq = (replay_us(g) - read_us * seq) / seq
        del g
        cg, _ = capture([c])
        times = []
        for it in range(reps):
            flush.sum()
            b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b.record(stream)
            cg[it % ROTATE].replay()
            e.record(stream)
            torch.cuda.synchronize()
            times.append(b.elapsed_time(e) * 1e3)
        del cg
        return us_seq, statistics.mean(times)

    l2_bytes = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 << 20

    def stream_us(c):
        """The call back to back, as a decode engine issues it: one graph of n
        calls over n pool copies (n copies hold more than twice the L2, so each
        call finds its pool cold), replayed; time per call."""
        n = max(ROTATE, -(-2 * l2_bytes // c.bytes) + 1)
        cc = c if n <= len(c.layouts) else Call(c.name, c.case, c.windowed, c.splits, dev, n,
                                                 tokens=c.tokens, fused=c.fused,
                                                 tree=c.tree_mask is not None)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            cc.run(0)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for r in range(n):
                cc.run(r)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = 10
        b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b.record(stream)
        for _ in range(reps):
            g.replay()
        e.record(stream)
        torch.cuda.synchronize()
        del g, cc
        return b.elapsed_time(e) * 1e3 / (reps * n)

    reps = max(20, min(args.steps, 50))
    for c in calls + extra:
        us, us_iso = per_call_us(c, reps)
        us_s = stream_us(c)
        gbps = c.bytes / (us * 1e-6) / 1e9
        detail[c.name].update({
            "us_stream": us_s, "GBps_stream": c.bytes / (us_s * 1e-6) / 1e9,
            "us_per_call": us, "GBps_per_call": gbps, "us_isolated": us_iso,
            "frac_of_8TBs": gbps / NOMINAL_HBM_GBS, "frac_of_measured": gbps / peak,
            "splits": c.splits or (pskv.pskv_plan_splits(c.layouts[0], c.case.num_q_heads,
                                                         c.lens_host)
                                   if c.tokens == 1 else "auto")})

    # ---- the split-count sweep of every global context (each call alone, cold L2)
    sweep = {}
    if args.sweep:
        for c in calls:
            if c.windowed:
                continue
            res = {}
            ws0, s0 = c.ws, c.splits  # the step's graphs point at this workspace: keep it alive
            for p in args.sweep:
                c.splits = p
                c.ws = pskv.workspace(1, 32, 512, p, dev)
                res[p] = per_call_us(c, 20, seq=6)[0]
            c.splits, c.ws = s0, ws0
            best = min(res, key=res.get)
            sweep[c.name] = {"us": res, "best_splits": best, "best_us": res[best],
                             "auto_splits": detail[c.name]["splits"],
                             "auto_us": detail[c.name]["us_per_call"]}
    del flush

    # ---- the same step with the fused K/V prep in place of the row copy
    # (projection rows in, normalised and rotated K/V written into the pages,
    # queries out)
    prep_ms = None
    if args.append != "prep" and not args.no_prep_step and graphs is not None:
        pargs = argparse.Namespace(**{**vars(args), "append": "prep"})
        pcalls = make_calls(pargs, dev)
        for it in range(args.warmup):
            for c in pcalls:
                c.run(it)
        pgraphs, _ = capture(pcalls)
        prep_ms = timed(lambda it: pgraphs[it % ROTATE].replay())
        for c in pcalls:
            if c.status[0].item() != 0:
                raise RuntimeError(f"{c.name}: device fault word {c.status[0].item()}")
        del pgraphs, pcalls

    # ---- paged prefills beside the step, last (tensor-core work: FLOP/s against
    # the bf16 peak; heavy enough to move the clocks, so nothing is timed after them)
    prefill = {}
    for c in make_prefill_calls(args, dev):
        cg, _ = capture([c])
        times = []
        for it in range(5):
            b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b.record(stream)
            cg[it % ROTATE].replay()
            e.record(stream)
            torch.cuda.synchronize()
            times.append(b.elapsed_time(e) * 1e3)
        if c.status[0].item() != 0:
            raise RuntimeError(f"{c.name}: device fault word {c.status[0].item()}")
        us = statistics.median(times)
        tf = c.flops / (us * 1e-6) / 1e12
        prefill[c.name] = {"tokens": c.tokens, "us": us, "tflops": tf,
                           "frac_of_bf16_peak": tf / measured_tensor_peak()}
        del cg, c

    glob = [c for c in calls if not c.windowed]
    part_bytes = sum(c.bytes for c in glob)
    part_s = sum(detail[c.name]["partial_us"] * 1e-6 for c in glob)
    achieved = part_bytes / part_s / 1e9
    traffic_per_key = recorded_traffic()
    keys_per_launch = statistics.mean(int(c.case.seq_lens.sum()) for c in glob)
    roofline = {"bound": "hbm", "kernel": "pskv_partial_kernel<MmaConsumer<512, 8>>",
                "achieved": r1(achieved), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "peak_source": "measured hbm_gbs" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": part_bytes / len(glob),
                "traffic": None if traffic_per_key is None
                else round(traffic_per_key * keys_per_launch)}

    line = make_line(args, dist.world, value, ms, launches, roofline,
                     {"value": r1(whole_job_gbps(step_bytes, dist.world, e2e_ms)), "unit": "GB/s",
                      "ms_per_step": round(e2e_ms, 5),
                      "h2d_bytes_per_step": packed.host_in.numel(),
                      "d2h_bytes_per_step": packed.host_out[0].numel(),
                      "how": "eager C-ABI calls; one packed copy in, one out per step"},
                     clock_info, {"graph": round(ms, 5), "eager": round(eager_ms, 5),
                                  "prep": None if prep_ms is None else round(prep_ms, 5)},
                     detail, sweep, prefill)
    if dist.rank == 0 and not args.no_cpu_baseline:
        cb = cpu_baseline([c.case for c in calls], args.cpu_seconds)
        cb["value"] = round(cb["value"], 3)
        line["cpu_baseline"] = cb
    if dist.rank == 0:
        if args.detail:
            with open(args.detail, "w") as f:
                json.dump({"line": line, "calls": detail, "sweep": sweep, "prefill": prefill,
                           "prep_step_ms": prep_ms, "eager_ms": eager_ms}, f, indent=1)
        print(json.dumps(line, separators=(",", ":"), ensure_ascii=False), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
