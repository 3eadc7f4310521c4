"""Benchmark of the paged-KV decode step on one GB300 (or N independent replicas).

A step is one Qwen3-0.6B-shaped decode step at batch 16: for each of 28
layers, append the new token's K/V rows and run decode attention over the
paged cache, as one pkv_decode_append_attn launch (--unfused: pkv_append
then pkv_decode_attn; the other variant is timed as an extra). Request lengths are
U{300..3000} (short clips plus prompt), pages randomly placed, every layer has
its own KV pool (about 3 GB in total, far larger than the 129 MB L2, so no L2
flush is needed between steps). The step's launches are captured once in a
CUDA graph and replayed.

Printed: one JSON line (rank 0). `value` is decode steps/s over all ranks.
`roofline` is for the decode kernel: algorithmic bytes per launch (every
cached K/V row of the layer once, the appended rows, q, out, block table and
lengths) over its mean duration in the timed region (CUDA events on the launch
stream around the graph replays; the step is nothing but these launches). The
duration of an isolated launch (events around each launch, no overlap with a
neighbour) is reported beside it. `e2e` runs the same step through the
Python API with the step's inputs copied from pinned host memory and the
attention output copied back, synchronising every step. `cpu_baseline` times
the fp64 CPU oracle on a bounded sample of the same workload.

`--impl reference` times the oracle alone (on the host cores) on samples of
the same workload and prints the same line with "impl": "reference".
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn KV GB/s & % HBM peak; decode steps/s at bs16 (1×GB300)"
UNIT = "steps/s"
WORKLOAD = ("qwen3-0.6b decode step: 28 layers x bs16, 16q/8kv heads, d128, page 16, seq U{300..3000}; "
            "per layer one fused KV-append + decode-attention launch (early prefetch)")


# DRAM traffic of one decode launch on this workload's per-layer pool, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), valid only for the decode kernel source it was
# measured on (sha256 prefix of csrc/decode_kernel.cuh followed by csrc/pkv_mma.cuh); any other source
# reports null.
NCU_DECODE_TRAFFIC = {"f60bafc4eddad24d": 107_560_448 + 3_036_928}


def _decode_traffic():
    import hashlib

    h = hashlib.sha256()
    for f in ("decode_kernel.cuh", "pkv_mma.cuh"):
        h.update(open(os.path.join(ROOT, "paged_kv_decode_gb300", "csrc", f), "rb").read())
    return NCU_DECODE_TRAFFIC.get(h.hexdigest()[:16])


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1954.7)), "measured"
    return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------ workload
class DecodeStep:
    """Device-resident 28-layer decode step (all layers share one block table)."""

    def __init__(self, device, seq_lens, layers: int, seed: int, fused: bool = True, early: bool = True,
                 rope: bool = False, producer: bool = False):
        import torch

        import paged_kv_decode_gb300 as pkv
        from paged_kv_decode_gb300 import workloads as W

        self.torch, self.pkv = torch, pkv
        case = W.decode_case(seed, seq_lens, layers=layers, device=device, pending_append=True, poison=True)
        self.case = case
        self.layers = layers
        self.B = case.batch
        self.scale = case.geom.scale
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
        self.q, self.k_pages, self.v_pages = case.q, case.k_pages, case.v_pages
        self.k_new, self.v_new = case.k_new, case.v_new
        self.block_table = i32(case.block_table)
        self.seq_lens = i32(case.seq_lens)
        self.slot_mapping = i32(case.slot_mapping)
        self.out = torch.empty_like(self.q)
        nbytes = pkv.decode_workspace_bytes(self.B, case.max_pages, case.num_pages)
        self.ws = pkv.Workspace(nbytes, device)
        self.graph = None
        self.fused = fused
        self.early = early and fused  # each layer's predecessor writes only other layers' pools
        # rotary embedding of the new token fused in (theta 1e6: "Fun-ASR-Nano Native Runtime Design")
        self.cos_sin = pkv.rope_cos_sin(1e6, int(np.max(seq_lens)) + 1, device=device) if (rope and fused) else None
        # producer: before each layer's attention, one kernel writes that layer's q / k_new / v_new (a copy
        # into one [q | k_new | v_new] buffer per layer), standing in for the QKV projection that precedes
        # attention in a decoder layer; the attention launch then follows a kernel that is not attention
        self.producer = producer
        if producer:
            g = case.geom
            nq, nk = self.B * g.n_q_heads * g.head_dim, self.B * g.n_kv_heads * g.head_dim
            self.qkv = torch.empty(layers, nq + 2 * nk, dtype=torch.bfloat16, device=device)
            qs, ks, vs = [], [], []
            for l in range(layers):
                buf = self.qkv[l]
                qs.append(buf[:nq].view(self.q[l].shape))
                ks.append(buf[nq:nq + nk].view(self.k_new[l].shape))
                vs.append(buf[nq + nk:].view(self.v_new[l].shape))
                qs[l].copy_(self.q[l])
                ks[l].copy_(self.k_new[l])
                vs[l].copy_(self.v_new[l])
            self.qkv_src = self.qkv.clone()
            self.q, self.k_new, self.v_new = qs, ks, vs

    def produce(self, l):
        """The stand-in producer kernel of layer l: writes the layer's q, k_new and v_new."""
        self.qkv[l].copy_(self.qkv_src[l])
    # algorithmic bytes of one decode launch (one layer)
    def decode_bytes(self) -> int:
        c = self.case
        kv = int(c.seq_lens.astype(np.int64).sum()) * c.geom.n_kv_heads * c.geom.head_dim * 2 * 2
        qo = 2 * self.B * c.geom.n_q_heads * c.geom.head_dim * 2
        meta = self.block_table.numel() * 4 + self.B * 4
        new_rows = self.append_bytes() if self.fused else 0  # k_new / v_new read and written into the pool
        return kv + qo + meta + new_rows

    def append_bytes(self) -> int:
        c = self.case
        return 2 * 2 * self.B * c.geom.n_kv_heads * c.geom.head_dim * 2 + self.B * 4

    def layer(self, l):
        pkv = self.pkv
        if self.producer:
            self.produce(l)
        if self.fused and self.cos_sin is not None:
            pkv.decode_append_rope_attn(self.q[l], self.k_new[l], self.v_new[l], self.k_pages[l], self.v_pages[l],
                                        self.block_table, self.seq_lens, self.cos_sin, self.out[l], self.scale,
                                        self.ws, early_prefetch=self.early)
            return
        if self.fused:
            pkv.decode_append_attn(self.q[l], self.k_new[l], self.v_new[l], self.k_pages[l], self.v_pages[l],
                                   self.block_table, self.seq_lens, self.out[l], self.scale, self.ws,
                                   early_prefetch=self.early)
            return
        pkv.append(self.k_new[l], self.v_new[l], self.slot_mapping, self.k_pages[l], self.v_pages[l], self.ws)
        pkv.decode_attn(self.q[l], self.k_pages[l], self.v_pages[l], self.block_table, self.seq_lens, self.out[l],
                        self.scale, self.ws)

    def decode_launch(self, l):
        """The launch the roofline times: the step's decode kernel for layer l."""
        if self.fused:
            self.layer(l)
        else:
            self.pkv.decode_attn(self.q[l], self.k_pages[l], self.v_pages[l], self.block_table, self.seq_lens,
                                 self.out[l], self.scale, self.ws)

    def step_eager(self):
        for l in range(self.layers):
            self.layer(l)

    def producers_only(self):
        for l in range(self.layers):
            self.produce(l)

    def capture(self, body=None):
        torch = self.torch
        body = body or self.step_eager
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            body()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            body()
        torch.cuda.synchronize()
        self.graph = g
        return g


def _barrier(dist_on):
    if dist_on:
        import torch.distributed as dist

        dist.barrier()


def _max_over_ranks(x: float, dist_on: bool) -> float:
    """Slowest rank's value (the tensor lives where the process group's backend wants it)."""
    if not dist_on:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_rate(local_total: float, units_per_rank: int, world: int, dist_on: bool):
    """Whole-job rate of N independent replicas: all ranks' units over the slowest rank's time.

    local_total is this rank's time for its units (any time unit); returns (slowest time, units / time unit).
    """
    slowest = _max_over_ranks(local_total, dist_on)
    return slowest, world * units_per_rank / slowest


def time_graph(step, steps, warmup, dist_on):
    torch = step.torch
    g = step.graph
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    _barrier(dist_on)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(steps):
        g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    _barrier(dist_on)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)  # ms


def time_decode_launches(step, reps):
    """Mean duration (ms) of the decode kernel: per-launch CUDA events on the launch stream,
    with the stream kept busy so that launch latency does not enter the intervals."""
    torch, pkv = step.torch, step.pkv
    st = torch.cuda.current_stream()
    durs = []
    n = step.layers
    for _ in range(reps):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda._sleep(int(2e7))  # ~10 ms of GPU work queued ahead of the launches
        for l in range(n):
            evs[l][0].record(st)
            step.decode_launch(l)
            evs[l][1].record(st)
        torch.cuda.synchronize()
        durs += [a.elapsed_time(b) for a, b in evs]
    return float(np.mean(durs)), len(durs)


class PrefillStep:
    """Workload 4: one 4096-token chunk after `prefix` cached tokens plus 15 concurrent decode requests."""

    def __init__(self, device, prefix, seed=4):
        import torch

        import paged_kv_decode_gb300 as pkv
        from paged_kv_decode_gb300 import workloads as W

        self.torch, self.pkv = torch, pkv
        c = W.prefill_case(seed, [prefix], [W.PREFILL_CHUNK], dec_seq_lens=W.mixed_decode_lens(seed), device=device,
                           poison=True)
        self.case = c
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
        self.q, self.k_new, self.v_new = c.q[0], c.k_new[0], c.v_new[0]
        self.k_pages, self.v_pages = c.k_pages[0], c.v_pages[0]
        self.slots, self.bt = i32(c.slot_mapping), i32(c.block_table)
        self.prefix, self.cu = i32(c.prefix_lens), i32(c.cu_q_lens)
        self.out = torch.empty_like(self.q)
        self.dq, self.dk, self.dv = c.dec_q[0], c.dec_k_new[0], c.dec_v_new[0]
        self.dslots, self.dbt, self.dlens = i32(c.dec_slot_mapping), i32(c.dec_block_table), i32(c.dec_seq_lens)
        self.dout = torch.empty_like(self.dq)
        # one workspace per kind of attention call (decode and prefill keep their counters apart)
        self.ws = pkv.Workspace(
            pkv.decode_workspace_bytes(len(c.dec_seq_lens), c.dec_block_table.shape[1], c.num_pages), device)
        self.pws = pkv.Workspace(pkv.prefill_workspace_bytes(1, W.PREFILL_CHUNK, c.num_pages), device)
        self.mws = pkv.Workspace(pkv.mixed_workspace_bytes(1, W.PREFILL_CHUNK, len(c.dec_seq_lens),
                                                           c.dec_block_table.shape[1], c.num_pages), device)
        self.scale = c.geom.scale
        P, L = int(prefix), W.PREFILL_CHUNK
        self.pairs = L * P + L * (L + 1) // 2
        self.flops = 4 * c.geom.head_dim * c.geom.n_q_heads * self.pairs

    def prefill(self):
        self.pkv.prefill_chunk_attn(self.q, self.k_pages, self.v_pages, self.bt, self.prefix, self.cu, self.out,
                                    self.scale, self.case.q_lens.max(), self.pws)

    def mixed(self):
        pkv = self.pkv
        pkv.append(self.k_new, self.v_new, self.slots, self.k_pages, self.v_pages, self.ws)
        pkv.append(self.dk, self.dv, self.dslots, self.k_pages, self.v_pages, self.ws)
        self.prefill()
        pkv.decode_attn(self.dq, self.k_pages, self.v_pages, self.dbt, self.dlens, self.dout, self.scale, self.ws)

    def mixed_branches(self):
        """The mixed step as two branches: the chunk (append, prefill) on the current stream and the
        decode requests (append, attention) on a side stream. They touch disjoint slots and separate
        workspaces, so a graph of this runs them concurrently where SMs are free."""
        torch, pkv = self.torch, self.pkv
        main = torch.cuda.current_stream()
        if not hasattr(self, "side"):
            self.side = torch.cuda.Stream()
        self.side.wait_stream(main)
        pkv.append(self.k_new, self.v_new, self.slots, self.k_pages, self.v_pages, self.pws)
        self.prefill()
        with torch.cuda.stream(self.side):
            pkv.append(self.dk, self.dv, self.dslots, self.k_pages, self.v_pages, self.ws)
            pkv.decode_attn(self.dq, self.k_pages, self.v_pages, self.dbt, self.dlens, self.dout, self.scale,
                            self.ws)
        main.wait_stream(self.side)

    def mixed_one_launch(self):
        """The mixed step with both attentions in one launch (pkv_mixed_step_attn) after the two appends."""
        pkv = self.pkv
        pkv.append(self.k_new, self.v_new, self.slots, self.k_pages, self.v_pages, self.mws)
        pkv.append(self.dk, self.dv, self.dslots, self.k_pages, self.v_pages, self.mws)
        pkv.mixed_step_attn(self.q, self.k_pages, self.v_pages, self.bt, self.prefix, self.cu, self.out,
                            self.case.q_lens.max(), self.dq, self.dbt, self.dlens, self.dout, self.scale, self.mws)

    def capture_mixed(self, body=None):
        """One CUDA graph of the mixed step (default: two branches)."""
        torch = self.torch
        body = body or self.mixed_branches
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            body()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            body()
        torch.cuda.synchronize()
        return g


def time_launches(torch, fn, reps):
    """Mean duration (ms) of fn's GPU work, bracketed by events with the stream kept busy."""
    st = torch.cuda.current_stream()
    durs = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(int(2e7))
        e0.record(st)
        fn()
        e1.record(st)
        torch.cuda.synchronize()
        durs.append(e0.elapsed_time(e1))
    return float(np.mean(durs))


class GenericDecodeStep:
    """Decode attention over `layers` distinct pools of another cache geometry: the decode kernel with
    run-time head counts (1 to 8 query heads per KV head, head_dim 64 or 128). fused: each layer is one fused
    append + decode launch with early prefetch (the decode step); otherwise decode attention alone."""

    def __init__(self, device, seq_lens, geom, layers: int, seed: int, fused: bool = False):
        import torch

        import paged_kv_decode_gb300 as pkv
        from paged_kv_decode_gb300 import workloads as W

        self.torch, self.pkv, self.layers, self.geom, self.fused = torch, pkv, layers, geom, fused
        case = W.decode_case(seed, seq_lens, geom=geom, layers=layers, device=device, pending_append=fused,
                             poison=True)
        self.case = case
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
        self.block_table, self.seq_lens = i32(case.block_table), i32(case.seq_lens)
        self.out = torch.empty_like(case.q)
        self.ws = pkv.Workspace(pkv.decode_workspace_bytes(case.batch, case.max_pages, case.num_pages, geom.n_q_heads,
                                                           geom.n_kv_heads, geom.head_dim), device)
        self.graph = None

    def decode_bytes(self) -> int:
        c, g = self.case, self.geom
        kv = int(c.seq_lens.astype(np.int64).sum()) * g.n_kv_heads * g.head_dim * 2 * 2
        new_rows = 2 * 2 * c.batch * g.n_kv_heads * g.head_dim * 2 if self.fused else 0  # read and written
        return kv + 2 * c.batch * g.n_q_heads * g.head_dim * 2 + self.block_table.numel() * 4 + c.batch * 4 + new_rows

    def step_eager(self):
        c = self.case
        for l in range(self.layers):
            if self.fused:  # each layer's predecessor writes only another layer's pool: early prefetch holds
                self.pkv.decode_append_attn(c.q[l], c.k_new[l], c.v_new[l], c.k_pages[l], c.v_pages[l],
                                            self.block_table, self.seq_lens, self.out[l], self.geom.scale, self.ws,
                                            early_prefetch=True)
            else:
                self.pkv.decode_attn(c.q[l], c.k_pages[l], c.v_pages[l], self.block_table, self.seq_lens,
                                     self.out[l], self.geom.scale, self.ws)

    capture = DecodeStep.capture


def measure_shapes(device, hbm, layers=8, steps=30, warmup=5):
    """Other decoder geometries (run-time head counts), bs16 U{300..3000} (one case a single
    40000-token request): per-layer time and bandwidth (the pages name these backbones without head
    counts; the shapes are examples)."""
    from paged_kv_decode_gb300 import workloads as W

    res = {}
    bs16 = W.config_seq_lens(2)
    for name, g, lens in (("32q_8kv_d128", W.Geometry(32, 8, 128), bs16),
                          ("32q_32kv_d128", W.Geometry(32, 32, 128), bs16),
                          ("32q_32kv_d64", W.Geometry(32, 32, 64), bs16),
                          ("64q_8kv_d128", W.Geometry(64, 8, 128), bs16),
                          ("16q_8kv_d64", W.Geometry(16, 8, 64), bs16),
                          ("32q_8kv_d128_40k", W.Geometry(32, 8, 128), [40000])):
        import torch

        res[name] = {"layers_in_graph": layers}
        for key, fused in (("", False), ("fused_early_", True)):
            st = GenericDecodeStep(device, lens, g, layers, seed=31, fused=fused)
            st.capture()
            ms = time_graph(st, steps, warmup, False) / steps
            us = ms * 1e3 / layers
            gbps = st.decode_bytes() / (us * 1e-6) / 1e9
            res[name].update({f"{key}us_per_layer": us, f"{key}gbps": gbps, f"{key}frac_of_measured_hbm": gbps / hbm,
                              f"{key}bytes_per_layer": st.decode_bytes()})
            del st
            torch.cuda.empty_cache()
    return res


def run_geometry(args, device):
    """One other geometry alone (bs16, decode attention only, `layers` pools in a graph)."""
    from paged_kv_decode_gb300 import workloads as W

    q, kv, d = (int(x) for x in args.geometry.split(","))
    st = GenericDecodeStep(device, W.config_seq_lens(2), W.Geometry(q, kv, d), args.layers, seed=31,
                           fused=args.geometry_fused)
    st.capture()
    ms = time_graph(st, args.steps, args.warmup, False) / args.steps
    us = ms * 1e3 / args.layers
    hbm = _peaks()[0]
    gbps = st.decode_bytes() / (us * 1e-6) / 1e9
    what = "fused append + decode (early prefetch)" if args.geometry_fused else "decode attention"
    print(json.dumps({"workload": f"{what}, {q}q/{kv}kv/d{d}, bs16 U{{300..3000}}, "
                                  f"{args.layers} layers per graph", "us_per_layer": us, "gbps": gbps,
                      "frac_of_measured_hbm": gbps / hbm, "bytes_per_layer": st.decode_bytes(),
                      "steps": args.steps, "warmup": args.warmup}), flush=True)


def run_prefill_geometry(args, device):
    """Chunked prefill alone on another cache geometry: a 4096-row chunk after 0 / 8192 / 32768 cached tokens
    (the prefill kernel on pairs of query heads), TFLOP/s of the causal flops."""
    import torch

    import paged_kv_decode_gb300 as pkv
    from paged_kv_decode_gb300 import workloads as W

    q, kv, d = (int(x) for x in args.prefill_geometry.split(","))
    g = W.Geometry(q, kv, d)
    bf16 = _peaks()[1]
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
    res = {}
    for P in (0, 8192, 32768):
        c = W.prefill_case(4, [P], [W.PREFILL_CHUNK], geom=g, device=device, poison=True)
        kp, vp, qq = c.k_pages[0], c.v_pages[0], c.q[0]
        out = torch.empty_like(qq)
        ws = pkv.Workspace(pkv.prefill_workspace_bytes(1, W.PREFILL_CHUNK, c.num_pages, q, kv, d), device)
        pkv.append(c.k_new[0], c.v_new[0], i32(c.slot_mapping), kp, vp, ws)
        bt, pl, cu = i32(c.block_table), i32(c.prefix_lens), i32(c.cu_q_lens)
        fn = lambda: pkv.prefill_chunk_attn(qq, kp, vp, bt, pl, cu, out, g.scale, W.PREFILL_CHUNK, ws)
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        ms = time_launches(torch, fn, max(3, args.steps))
        flops = 4 * d * q * (W.PREFILL_CHUNK * P + W.PREFILL_CHUNK * (W.PREFILL_CHUNK + 1) // 2)
        tf = flops / (ms * 1e-3) / 1e12
        res[f"prefix_{P}"] = {"prefill_us": ms * 1e3, "tflops": tf, "frac_of_measured_bf16": tf / bf16}
        del c, kp, vp, qq, out, ws
        torch.cuda.empty_cache()
    print(json.dumps({"workload": f"chunked prefill, {q}q/{kv}kv/d{d}, 4096-row chunk after 0/8192/32768 cached "
                                  f"tokens", **res, "steps": args.steps, "warmup": args.warmup}), flush=True)


def measure_prefill(device, bf16_peak, reps=10):
    import torch

    res = {}
    for prefix in (0, 8192, 32768):
        ps = PrefillStep(device, prefix)
        ps.mixed()
        torch.cuda.synchronize()
        ms = time_launches(torch, ps.prefill, reps)
        mixed_ms = time_launches(torch, ps.mixed, reps)
        g = ps.capture_mixed()
        graph_ms = time_launches(torch, g.replay, reps)
        g1 = ps.capture_mixed(ps.mixed_one_launch)
        one_ms = time_launches(torch, g1.replay, reps)
        tf = ps.flops / (ms * 1e-3) / 1e12
        res[f"prefix_{prefix}"] = {"chunk": 4096, "prefill_us": ms * 1e3, "tflops": tf,
                                   "frac_of_measured_bf16": tf / bf16_peak, "gflop": ps.flops / 1e9,
                                   "mixed_step_us": mixed_ms * 1e3,
                                   # the same step as one CUDA graph, decode requests on a parallel branch
                                   "mixed_step_graph_us": graph_ms * 1e3,
                                   # the appends and one pkv_mixed_step_attn launch, as one CUDA graph
                                   "mixed_step_one_launch_us": one_ms * 1e3}
        del g, g1
        del ps
        torch.cuda.empty_cache()
    return res


def stage_inputs(step, align=256):
    """One device buffer and one pinned host buffer holding all of a step's inputs: slots, lengths and
    block table, then q, k_new and v_new of each layer, each 256-byte aligned. The step's tensors become
    views of the device buffer, so a step's inputs arrive in one host-to-device copy."""
    torch = step.torch
    shared = [("slot_mapping", step.slot_mapping), ("seq_lens", step.seq_lens), ("block_table", step.block_table)]
    per_layer = [("q", step.q), ("k_new", step.k_new), ("v_new", step.v_new)]
    parts, off = [], 0
    for name, t in shared:
        parts.append((name, None, off, t))
        off += (t.numel() * t.element_size() + align - 1) // align * align
    layer_off = []
    for l in range(step.layers):
        layer_off.append(off)
        for name, t in per_layer:
            parts.append((name, l, off, t[l]))
            off += (t[l].numel() * t[l].element_size() + align - 1) // align * align
    step.staging_layer_off = layer_off  # offset of each layer's inputs in the staging buffers
    dev = torch.empty(off, dtype=torch.uint8, device=step.out.device)
    host = torch.empty(off, dtype=torch.uint8, pin_memory=True)
    layered = {name: [None] * step.layers for name, _ in per_layer}
    for name, l, o, t in parts:
        nb = t.numel() * t.element_size()
        view = dev[o:o + nb].view(t.dtype).view(t.shape)
        view.copy_(t)
        host[o:o + nb].copy_(t.detach().cpu().contiguous().view(-1).view(torch.uint8))
        if l is None:
            setattr(step, name, view)
        else:
            layered[name][l] = view
    for name, views in layered.items():
        setattr(step, name, views)
    return dev, host


def time_e2e(step, steps, warmup, dist_on, overlap=True):
    """Steps/s through the Python API with host buffers: H2D of q, k_new, v_new, slots, lengths and
    block table from pinned memory (one staging buffer), the step, D2H of the attention output (all in
    one CUDA graph), then a synchronize, every step.

    overlap: the lengths, block table and layer 0's inputs are copied first; the other layers' inputs
    follow on a side stream that only layer 1 waits for, and each layer's output is copied back on a
    second side stream right after the layer. Kernel-to-kernel edges stay programmatic (no copy feeds a
    later layer except layer 1's inputs), so the layers keep their overlap."""
    torch = step.torch
    dev, host = stage_inputs(step)
    hout = torch.empty(step.out.shape, dtype=step.out.dtype, pin_memory=True)
    h2d = host.numel()
    d2h = hout.numel() * hout.element_size()
    split = step.staging_layer_off[1] if step.layers > 1 else host.numel()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def body():
        if not overlap:
            dev.copy_(host, non_blocking=True)
            step.step_eager()
            hout.copy_(step.out, non_blocking=True)
            return
        main = torch.cuda.current_stream()
        s_in.wait_stream(main)
        s_out.wait_stream(main)
        dev[:split].copy_(host[:split], non_blocking=True)
        with torch.cuda.stream(s_in):
            dev[split:].copy_(host[split:], non_blocking=True)
        for l in range(step.layers):
            if l == 1:
                main.wait_stream(s_in)
            step.layer(l)
            s_out.wait_stream(main)
            with torch.cuda.stream(s_out):
                hout[l].copy_(step.out[l], non_blocking=True)
        main.wait_stream(s_in)
        main.wait_stream(s_out)

    # one CUDA graph per step: the host->device copy of the step's inputs from pinned memory,
    # the layers, and the device->host copy of the output; a replay and a synchronize per step
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        body()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        body()
    torch.cuda.synchronize()

    def one():
        g.replay()
        torch.cuda.current_stream().synchronize()

    for _ in range(warmup):
        one()
    _barrier(dist_on)
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    dt = time.perf_counter() - t0
    _barrier(dist_on)
    return dt, h2d, d2h


# ------------------------------------------------------------------------------ CPU oracle
def _cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample_case(seed):
    from paged_kv_decode_gb300 import workloads as W

    return W.decode_case(seed, W.config_seq_lens(2, seed), layers=1, device="cpu", pending_append=False,
                         poison=True)


def cpu_baseline(seed, budget_s=10.0):
    """Oracle on whole layers of the workload (all 16 requests), as many as fit the budget."""
    import oracle

    case = oracle_sample_case(seed)
    cores = _cpu_cores()
    layers = 0
    t = 0.0
    while layers < 1 or t < budget_s:
        t0 = time.perf_counter()
        oracle.decode(case.q[0], case.k_pages[0], case.v_pages[0], case.block_table, case.seq_lens, case.geom.scale,
                      n_threads=cores)
        t += time.perf_counter() - t0
        layers += 1
        if layers >= 5000:
            break
    steps_per_s = layers / t / 28.0
    return {"value": steps_per_s, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{layers} full layers (bs16, all heads) of the same workload, fp64 C oracle, "
                      f"{t:.1f} s; steps/s = layers/s / 28"}


# ------------------------------------------------------------------------------ main
def _rounded(x, digits=4):
    """Floats to `digits` significant digits, recursively (keeps the summary short)."""
    if isinstance(x, dict):
        return {k: _rounded(v, digits) for k, v in x.items()}
    if isinstance(x, float):
        return float(f"{x:.{digits}g}")
    return x


def oracle_step(case, layers, cores):
    """One decode step of the workload on the oracle: `layers` calls over the whole bs16 layer (all 16
    requests, all heads). The calls reuse one layer's pool: the oracle's work per layer does not depend
    on which layer's values it reads, and 28 pools (3 GB) would not add anything but generation time."""
    import oracle

    for _ in range(layers):
        oracle.decode(case.q[0], case.k_pages[0], case.v_pages[0], case.block_table, case.seq_lens, case.geom.scale,
                      n_threads=cores)


def run_reference(args, rank, world):
    if rank != 0:
        return
    case = oracle_sample_case(2)
    cores = _cpu_cores()
    layers = args.layers
    for _ in range(args.warmup):
        oracle_step(case, 1, cores)  # warm-up: one layer each
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(case, layers, cores)
    t = time.perf_counter() - t0
    steps_per_s = args.steps / t
    line = {
        "impl": "reference", "metric": METRIC, "value": steps_per_s, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / steps_per_s, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": 16, "layers": 28, "seq_len": "U{300..3000}",
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": steps_per_s, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each timed step = one whole decode step of the workload: {layers} oracle "
                                   f"calls over a full bs16 layer (16 requests, all heads; one layer's pool "
                                   f"reused); {args.steps} steps in {t:.2f} s"},
        "e2e": {"value": steps_per_s, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=28)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the 40k-context and prefill measurements")
    ap.add_argument("--geometry", default=None, metavar="Q,KV,D",
                    help="time only the decode path on that cache geometry (bs16 U{300..3000}) and exit")
    ap.add_argument("--prefill-geometry", default=None, metavar="Q,KV,D",
                    help="time only chunked prefill on that cache geometry (4096 rows after 0/8192/32768) and exit")
    ap.add_argument("--geometry-fused", action="store_true",
                    help="with --geometry: time the fused append + decode call with early prefetch")
    ap.add_argument("--unfused", action="store_true",
                    help="time the step as separate pkv_append + pkv_decode_attn launches")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch

    from paged_kv_decode_gb300.build import build_library
    from paged_kv_decode_gb300 import workloads as W

    if rank == 0 or world == 1:
        build_library()
    dist_on = world > 1
    if dist_on:
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
        if rank != 0:
            build_library()
    device = torch.device("cuda", local_rank if dist_on else 0)
    torch.cuda.set_device(device)
    if args.geometry:
        run_geometry(args, device)
        return
    if args.prefill_geometry:
        run_prefill_geometry(args, device)
        return

    # each replica runs its own copy of the workload (replicas only: requests are independent)
    step = DecodeStep(device, W.config_seq_lens(2), args.layers, seed=2 + rank, fused=not args.unfused)
    step.capture()
    launches_per_step = args.layers if step.fused else 2 * args.layers

    clocks = ClockSampler(device.index)
    clocks.start()
    ms_total = time_graph(step, args.steps, args.warmup, dist_on)
    dec_ms, dec_n = time_decode_launches(step, reps=max(3, min(20, args.steps // 50)))
    clk = clocks.stop()

    ms_total, steps_per_ms = replica_rate(ms_total, args.steps, world, dist_on)
    ms_per_step = ms_total / args.steps
    steps_per_s = steps_per_ms * 1e3

    e2e_steps = max(10, args.steps // 10)
    e2e_dt, h2d, d2h = time_e2e(step, e2e_steps, args.warmup, dist_on)
    e2e_dt, e2e_value = replica_rate(e2e_dt, e2e_steps, world, dist_on)

    hbm, bf16, peak_kind = _peaks()
    main_fused = step.fused
    dec_bytes = step.decode_bytes()
    isolated = dec_bytes / (dec_ms * 1e-3) / 1e9
    if step.fused:
        # the timed step is nothing but the 28 decode launches (append fused in): their mean
        # duration over the timed region is the step time / 28, launches overlapping through PDL
        launch_us = ms_per_step * 1e3 / args.layers
        achieved = dec_bytes / (launch_us * 1e-6) / 1e9
    else:
        launch_us = dec_ms * 1e3
        achieved = isolated
    step_bytes = args.layers * (dec_bytes + (0 if step.fused else step.append_bytes()))
    pool_bytes = 2 * step.k_pages.numel() * step.k_pages.element_size()
    step_tokens = float(np.asarray(step.case.seq_lens, dtype=np.int64).sum())

    extra = {}
    if not args.no_extra:
        variants = [("separate_append_and_decode", False, False, False), ("fused_no_early_prefetch", True, False, False),
                    ("fused_early_prefetch", True, True, False), ("fused_rope_early_prefetch", True, True, True)]
        for name, fused, early, rope in variants:
            if fused == step.fused and early == step.early and not rope:
                continue
            other = DecodeStep(device, W.config_seq_lens(2), args.layers, seed=2 + rank, fused=fused, early=early,
                               rope=rope)
            other.capture()
            n_o = max(50, args.steps // 4)
            ot = time_graph(other, n_o, args.warmup, dist_on) / n_o
            extra["step_" + name] = {"ms_per_step": ot, "steps_per_s": 1e3 / ot,
                                     "launches_per_step": args.layers * (1 if fused else 2)}
            del other
            torch.cuda.empty_cache()
        long_step = None
        del step
        torch.cuda.empty_cache()
        long_step = DecodeStep(device, W.config_seq_lens(3, context=40000), args.layers, seed=3 + rank,
                               fused=not args.unfused)
        long_step.capture()
        lt = time_graph(long_step, max(20, args.steps // 4), args.warmup, dist_on) / max(20, args.steps // 4)
        ld_ms, _ = time_decode_launches(long_step, reps=5)
        lb = long_step.decode_bytes()
        extra["long_context_40k"] = {
            "workload": "long-audio decode: 28 layers x bs1, context 40000, same geometry",
            "ms_per_step": lt, "steps_per_s": 1e3 / lt,
            # in the step, like the headline roofline: step time / layers per launch
            "launch_us_in_step": lt * 1e3 / args.layers,
            "gbps_in_step": lb / (lt * 1e-3 / args.layers) / 1e9,
            "frac_of_measured_hbm_in_step": lb / (lt * 1e-3 / args.layers) / 1e9 / hbm,
            # one launch at a time, events around it
            "decode_kernel_us": ld_ms * 1e3, "decode_gbps": lb / (ld_ms * 1e-3) / 1e9,
            "frac_of_measured_hbm": lb / (ld_ms * 1e-3) / 1e9 / hbm,
        }
        del long_step
        torch.cuda.empty_cache()

        def in_step(lens, seed, name):
            st = DecodeStep(device, lens, args.layers, seed=seed, fused=not args.unfused)
            st.capture()
            n = max(20, args.steps // 4)
            t = time_graph(st, n, args.warmup, dist_on) / n
            b = st.decode_bytes()
            tok = int(np.asarray(lens, dtype=np.int64).sum())
            res = {"workload": name, "ms_per_step": t, "steps_per_s": 1e3 / t, "launch_us_in_step": t * 1e3 / args.layers,
                   "gbps_in_step": b / (t * 1e-3 / args.layers) / 1e9,
                   "frac_of_measured_hbm_in_step": b / (t * 1e-3 / args.layers) / 1e9 / hbm,
                   "kv_token_layers_per_s": tok * args.layers / (t * 1e-3)}
            del st
            torch.cuda.empty_cache()
            return res

        def after_producer(lens, seed, name):
            """Each layer's fused attention launch follows the stand-in producer of that layer's q / k_new /
            v_new. The attention's share of the step = (step - the producers alone) / layers."""
            st = DecodeStep(device, lens, args.layers, seed=seed, fused=True, early=True, producer=True)
            n = max(20, args.steps // 4)
            st.capture()
            t_all = time_graph(st, n, args.warmup, dist_on) / n
            st.capture(st.producers_only)
            t_prod = time_graph(st, n, args.warmup, dist_on) / n
            b = st.decode_bytes()
            us = (t_all - t_prod) * 1e3 / args.layers
            res = {"workload": name, "ms_per_step": t_all, "producers_alone_ms": t_prod, "attention_us_per_layer": us,
                   "attention_gbps": b / (us * 1e-6) / 1e9, "attention_frac_of_measured_hbm": b / (us * 1e-6) / 1e9 / hbm,
                   "attention_frac_of_nominal_8tbs": b / (us * 1e-6) / 1e9 / 8000.0}
            del st
            torch.cuda.empty_cache()
            return res

        extra["after_producer"] = {
            "what": "every layer's fused append + decode launch (early prefetch) follows one kernel that writes "
                    "that layer's q / k_new / v_new (a copy into the layer's [q | k_new | v_new] buffer), standing "
                    "in for the QKV projection before attention; attention time = (step - producers alone) / 28",
            "bs16": after_producer(W.config_seq_lens(2), 2 + rank, "bs16 U{300..3000}"),
            "long_40k": after_producer(W.config_seq_lens(3, context=40000), 3 + rank, "bs1, context 40000")}

        # the long-audio sweep of workload 3 and the CFG-paired batch of workload 5
        extra["context_sweep"] = {
            f"context_{c}": in_step(W.config_seq_lens(3, context=c), 3 + rank,
                                    f"long-audio decode: 28 layers x bs1, context {c}")
            for c in (4096, 16384, 65536)}
        extra["cfg_pairs_bs32"] = in_step(
            W.config_seq_lens(5), 5 + rank,
            "CFG-paired decode: 28 layers x bs32 (16 conditional U{1000..8000} + 16 companions U{8..64} + g)")
        extra["other_geometries_bs16"] = {
            "workload": "other geometries (run-time head counts), bs16 U{300..3000} (the _40k case: one "
                        "40000-token request), 8 layers per graph: decode attention alone, and (fused_early_*) one "
                        "fused append + decode launch per layer with early prefetch",
            **measure_shapes(device, hbm)}
        extra["chunked_prefill"] = {
            "workload": "4096-token chunk (1 request) after 0/8192/32768 cached tokens; mixed step adds the chunk "
                        "append, 15 decode appends and decode attention over U{500..5000}",
            **measure_prefill(device, bf16)}

    if rank != 0:
        if dist_on:
            import torch.distributed as dist

            dist.destroy_process_group()
        return

    line = {
        "metric": METRIC, "value": steps_per_s, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": 16 * world, "layers": args.layers,
                   "seq_len": "U{300..3000}", "parallelism": "replicas" if world > 1 else "single",
                   "l2": "no flush: %d distinct layer pools of %.2f GB in total exceed the 129 MB L2" % (
                       args.layers, pool_bytes / 1e9)},
        "kv_gbps_step": step_bytes / (ms_per_step * 1e-3) / 1e9 * world,
        # attended (KV token, layer) pairs per second: each cached token of each layer read once
        "kv_token_layers_per_s": step_tokens * args.layers
        / (ms_per_step * 1e-3) * world,
        "roofline": {"bound": "hbm", "kernel": "pkv::decode_kernel", "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": _decode_traffic(), "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": dec_bytes, "launch_us": launch_us,
                     "launch_us_basis": "timed region / launches" if main_fused else "per-launch events",
                     "isolated_launch_us": dec_ms * 1e3, "isolated_achieved": isolated,
                     "isolated_launches_timed": dec_n, "frac_of_nominal_8tbs": achieved / 8000.0},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if extra:
        line["extra"] = extra
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(2)
    # the decode and prefill targets in a few keys at the end of the line
    summary = {"hbm_peak_gbps": hbm, "bf16_peak_tflops": bf16,
               "decode_bs16": {"in_step_gbps": achieved, "frac_measured": achieved / hbm,
                               "frac_8tbs": achieved / 8000.0, "isolated_frac_measured": isolated / hbm}}
    if extra:
        lc = extra["long_context_40k"]
        summary["decode_40k"] = {"in_step_gbps": lc["gbps_in_step"], "frac_measured": lc["gbps_in_step"] / hbm,
                                 "frac_8tbs": lc["gbps_in_step"] / 8000.0,
                                 "isolated_frac_measured": lc["frac_of_measured_hbm"]}
        for key, name in (("bs16", "decode_bs16"), ("long_40k", "decode_40k")):
            ap = extra["after_producer"][key]
            summary[name]["after_producer_frac_measured"] = ap["attention_frac_of_measured_hbm"]
            summary[name]["after_producer_frac_8tbs"] = ap["attention_frac_of_nominal_8tbs"]
        cp = extra["chunked_prefill"]
        summary["prefill_4096"] = {f"P{P}": {"tflops": cp[f"prefix_{P}"]["tflops"],
                                             "frac_measured": cp[f"prefix_{P}"]["frac_of_measured_bf16"],
                                             "mixed_graph_us": cp[f"prefix_{P}"]["mixed_step_graph_us"],
                                             "mixed_one_launch_us": cp[f"prefix_{P}"]["mixed_step_one_launch_us"]}
                                   for P in (0, 8192, 32768)}
    line["summary"] = _rounded(summary)
    print(json.dumps(line), flush=True)
    if dist_on:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
