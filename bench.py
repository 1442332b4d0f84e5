#!/usr/bin/env python3
"""Benchmark of the WKV-7 state-slot hot path on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mixed|decode12|prefill|sweep|verify|hibernate] [--batch B] [--graph]

Default workload ("mixed", one step = every part of the hot path): on a
4096-slot pool of 32 heads x 64 (1 layer) -- create 64 fresh slots, snapshot
64 slots, decode 1024 slots at permuted ids, chunked prefill of 64 ragged
sequences (lengths uniform on 1..2048) into the fresh slots, fork 64 slots,
restore the 64 snapshots.  Throughput = (decode tokens + prefill tokens) per
second; one decode slot-step and one prefill token are each one token through
one layer.  Other workloads: "decode12" (12 layers x 12 heads, 256 of 1024
slots), "prefill" (8 x 4096 tokens, 32 heads), "sweep" (32 layers x 64 heads,
--batch of a 4096-slot pool).

Prints ONE JSON line (rank 0).  Timing: W untimed steps, then K steps between
CUDA events on the launching stream, bracketed by a barrier and a device
synchronisation, max over ranks.  Each step moves more bytes than the 129 MB L2
holds (inputs larger than L2), so no explicit flush is used.
--impl reference times the CPU oracle (the only reference this method has) on
a bounded sample of the same workload per step.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "WKV-7 decode slot-steps/s + GB/s (% HBM peak); prefill tokens/s (% roofline)"
HEAD_BYTES_STATE = 64 * 64 * 4
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# --------------------------------------------------------------------------- env
def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["mixed", "decode12", "prefill", "sweep", "verify",
                                          "hibernate", "decode_mixed"],
                   default="mixed")
    p.add_argument("--batch", type=int, default=4096, help="sweep batch size")
    p.add_argument("--graph", action="store_true", help="replay each step as a CUDA graph")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--checkpoints", action="store_true",
                   help="prefill workload: also keep the state at every 64-token boundary")
    p.add_argument("--verify-k", type=int, default=5,
                   help="verify workload: tokens per slot per call (K drafts + 1)")
    p.add_argument("--no-rollback", action="store_true",
                   help="verify workload: no per-token rollback states")
    p.add_argument("--state-dtype", choices=["f32", "bf16"], default="f32",
                   help="mixed and sweep workloads: state storage (bf16 halves the state bytes)")
    p.add_argument("--out-dtype", choices=["f32", "bf16"], default="f32",
                   help="mixed workload: output dtype (bf16: each readout rounded to bf16, half the "
                        "output bytes)")
    p.add_argument("--no-targets", action="store_true",
                   help="mixed workload: skip the 8 x 4096 prefill and the 32-layer sweep lines")
    p.add_argument("--min-timed-s", type=float, default=0.6,
                   help="repeat the K-step timed region until at least this long (clock samples)")
    return p.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS)


# kernel -> (committed ncu summary, the workloads whose launch of that kernel it
# profiles, the sources it was taken on)
KERNEL_SOURCES = {
    "prefill": ("prefill_chunk_kernel.mixed_prefill_64seq.md", ("mixed",),
                ["prefill_chunk.cu", "sm100_ptx.cuh", "device_common.cuh", "wkv7_internal.h",
                 "prefill_seq_unit.cuh"]),
    "decode": ("decode_kernel.mixed_decode_1024of4096.md", ("mixed", "decode_mixed"),
               ["decode.cu", "device_common.cuh", "wkv7_internal.h", "row_sums.cuh"]),
}


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if that summary
    was taken on this workload's launch shape and the kernel's sources are
    unchanged since; else None."""
    import hashlib
    if kernel not in KERNEL_SOURCES or workload not in KERNEL_SOURCES[kernel][1]:
        return None
    fname, _, sources = KERNEL_SOURCES[kernel]
    try:
        text = open(os.path.join(ROOT, "profiles", fname)).read()
        m = hashlib.sha256()
        for f in sources:
            with open(os.path.join(ROOT, "rwkv_wkv_gb300", "csrc", f), "rb") as fh:
                m.update(fh.read())
    except OSError:
        return None
    fields = dict(line.strip().split(": ", 1) for line in text.splitlines()
                  if line.strip().startswith(("dram_bytes_per_launch:", "source_sha256:")))
    if fields.get("source_sha256") != m.hexdigest()[:16]:
        return None
    return int(fields["dram_bytes_per_launch"])


def aggregate(elapsed_s: float, units: float, world: int, device=None, op: str = "sum"):
    """Whole-job figures over ranks: max of the elapsed times, sum (or max) of the units."""
    if world <= 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM if op == "sum" else dist.ReduceOp.MAX)
    return float(t.item()), float(u.item())


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", gpu_id], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def wait_first(self, timeout=5.0):
        t0 = time.time()
        while self.proc and not self.samples and time.time() - t0 < timeout:
            time.sleep(0.02)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [s for ts, s in self.samples if t0 <= ts <= t1 + 0.05 and len(s) >= 9]
        if not rows:
            rows = [s for _, s in self.samples if len(s) >= 9][-3:]
        if not rows:
            return None
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = sorted({name for r in rows for name, val in zip(self.REASONS, r[5:9])
                          if val.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------- workloads
class Workload:
    """One benchmark workload on one GPU.  Subclasses set self.phases (ordered
    names), self.phase_bytes (algorithmic bytes per phase per step),
    self.tokens_per_step, self.dominant and implement setup/step/host_io."""
    name = ""
    description = ""
    dominant = ""

    def config(self) -> dict:
        return {}


class Mixed(Workload):
    name = wl.MIXED.name

    def __init__(self, torch, device, seed=wl.MIXED.seed, state_dtype="f32", out_dtype="f32"):
        from rwkv_wkv_gb300 import Pool
        W = wl.MIXED
        self.state_dtype, self.out_dtype = state_dtype, out_dtype
        self.out_elem_bytes = 2 if out_dtype == "bf16" else 4
        self.state_head_bytes = HEAD_BYTES_STATE // (2 if state_dtype == "bf16" else 1)
        self.torch, self.device = torch, device
        self.H, self.N = W.H, W.N
        plan = wl.mixed_plan(seed)
        self.plan = plan
        self.lengths = plan["lengths"].astype(np.int64)
        self.total = int(self.lengths.sum())
        self.pool = Pool(1, W.H, W.n_slots, n_snapshots=wl.MIXED_VERB_N, device=device,
                         state_dtype=state_dtype, out_dtype=out_dtype)
        g = torch.Generator(device=device).manual_seed(seed)
        self.pool.states.normal_(0.0, 0.1, generator=g)
        # slot table: every id in use except the prefill targets, which each
        # step creates (zeroed) and returns at the end.
        self.pool.alloc(W.n_slots)
        self.pool.free(list(plan["prefill"][::-1]))
        self.snap_ids_host = self.pool.snapshot_alloc(wl.MIXED_VERB_N)
        i32 = lambda x: torch.as_tensor(np.asarray(x, dtype=np.int32), device=device)  # noqa: E731
        self.dec_ids = i32(plan["decode"])
        self.pre_ids = i32(plan["prefill"])
        self.cu = i32(wl.cu_seqlens(self.lengths))
        self.fork_src, self.fork_dst = i32(plan["fork_src"]), i32(plan["fork_dst"])
        self.snap_src, self.snap_ids = i32(plan["snap_src"]), i32(self.snap_ids_host)
        B = wl.MIXED_DECODE_B
        self.dec_in = wl.token_inputs_device(seed, B, W.H, W.N, device, generator_offset=1)
        self.pre_in = wl.token_inputs_device(seed, self.total, W.H, W.N, device,
                                             generator_offset=2)
        odt = self.pool.o_torch_dtype
        self.o_dec = torch.empty(B, W.H, W.N, dtype=odt, device=device)
        self.o_pre = torch.empty(self.total, W.H, W.N, dtype=odt, device=device)
        slot_bytes = self.pool.slot_bytes
        nv = wl.MIXED_VERB_N
        in_row = W.H * W.N * 2 * 6
        out_row = W.H * W.N * self.out_elem_bytes
        self.phases = ["create", "snapshot", "decode", "prefill", "fork", "restore"]
        self.phase_bytes = {
            "create": wl.MIXED_PREFILL_SEQS * slot_bytes,
            "snapshot": 2 * nv * slot_bytes,
            "decode": B * (W.H * 2 * self.state_head_bytes + in_row + out_row),
            "prefill": self.total * (in_row + out_row)
            + wl.MIXED_PREFILL_SEQS * W.H * 2 * self.state_head_bytes,
            "fork": 2 * nv * slot_bytes,
            "restore": 2 * nv * slot_bytes,
        }
        self.tokens_per_step = B + self.total
        self.dominant = "prefill"
        self.launches_per_step = 6
        self.check_ids = True

    def step(self, ev=None):
        pool = self.pool
        rec = (lambda name: ev[name].record()) if ev else (lambda name: None)
        rec("start")
        created = pool.create(wl.MIXED_PREFILL_SEQS)
        if self.check_ids:
            assert created == [int(x) for x in self.plan["prefill"]], "slot table order"
            self.check_ids = False
        rec("create")
        pool.snapshot(self.snap_src, self.snap_ids)
        rec("snapshot")
        pool.decode_step(0, self.dec_ids, *self.dec_in, o=self.o_dec)
        rec("decode")
        pool.prefill(0, self.pre_ids, self.cu, *self.pre_in, o=self.o_pre,
                     max_seqlen=wl.MIXED_MAX_LEN)
        rec("prefill")
        pool.fork(self.fork_src, self.fork_dst)
        rec("fork")
        pool.restore(self.snap_ids, self.snap_src)
        rec("restore")
        pool.free(created[::-1])

    def verb_ceiling(self):
        """GB/s of the device's own contiguous copy (torch copy_, a cudaMemcpyAsync)
        and fill (zero_, a cudaMemsetAsync) of the same bytes as one verb call (64
        slots), timed with CUDA events in this run: at 32-64 MB per call, the
        ramp-up and tail of any transfer are a visible share of its time, so this,
        not the large-copy peak, is what a verb of this size can reach."""
        torch = self.torch
        nbytes = wl.MIXED_VERB_N * self.pool.slot_bytes
        a = torch.empty(nbytes, dtype=torch.uint8, device=self.pool.device)
        b = torch.empty(nbytes, dtype=torch.uint8, device=self.pool.device)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=self.pool.device)
        out = {}
        for name, fn, moved in (("copy", lambda: b.copy_(a), 2 * nbytes), ("fill", lambda: b.zero_(), nbytes)):
            ts = []
            for r in range(23):
                flush.fill_(r & 0xFF)
                s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s0.record()
                fn()
                s1.record()
                torch.cuda.synchronize()
                if r >= 3:
                    ts.append(s0.elapsed_time(s1))
            out[name] = moved / (statistics.median(ts) / 1e3) / 1e9
        del a, b, flush
        return out

    def host_io(self):
        """(inputs to upload each step, outputs to read back each step)."""
        ins = [self.dec_ids, self.pre_ids, self.cu, self.fork_src, self.fork_dst,
               self.snap_src, self.snap_ids] + self.dec_in + self.pre_in
        return ins, [self.o_dec, self.o_pre]

    def config(self):
        return {"workload": wl.MIXED.description
                + ("; bf16 state storage" if self.state_dtype == "bf16" else "")
                + ("; bf16 outputs" if self.out_dtype == "bf16" else ""),
                "pool_slots": wl.MIXED.n_slots,
                "layers": 1, "heads": self.H, "head_size": self.N,
                "decode_slots": wl.MIXED_DECODE_B, "prefill_seqs": wl.MIXED_PREFILL_SEQS,
                "prefill_tokens": self.total, "verb_slots": wl.MIXED_VERB_N,
                "state_dtype": self.state_dtype, "input_dtype": "bf16", "output_dtype": self.out_dtype}

    def oracle_sample(self, frac_target: float):
        """Sample of the step for the CPU oracle: every decode row and prefill
        sequence on a subset of the (independent) heads; below one head, also
        the first rows and sequences only."""
        return _head_sample(self.H, frac_target, wl.MIXED_DECODE_B, self.lengths,
                            self.tokens_per_step)


def _head_sample(H, frac_target, n_rows, lengths, tokens_per_step, layers=1):
    n_heads = int(min(H, max(1, round(frac_target * H))))
    sub = min(1.0, frac_target * H) if n_heads == 1 else 1.0
    n_dec = int(max(1 if n_rows else 0, round(n_rows * sub))) if n_rows else 0
    lens = np.asarray(lengths if lengths is not None else [], dtype=np.int64)
    if len(lens) and sub < 1.0:
        budget = max(1.0, lens.sum() * sub)
        csum = np.cumsum(lens)
        n_seq = max(1, int(np.searchsorted(csum, budget, side="right")))
        lens = lens[:n_seq]
    toks = n_dec * layers + int(lens.sum())
    frac = (toks / float(tokens_per_step)) * (n_heads / float(H))
    desc = (f"{n_heads} of {H} heads; {n_dec} of {n_rows} decode rows"
            + (f" x {layers} layers" if layers > 1 else "")
            + (f"; {len(lens)} prefill sequences ({int(lens.sum())} tokens)" if len(lens) else "")
            + f"; step time scaled by the work fraction {frac:.5f}")
    return {"heads": n_heads, "decode_rows": n_dec, "layers": layers,
            "prefill_lengths": lens, "frac": frac, "desc": desc}


class Decode12(Workload):
    name = wl.DECODE_12L.name

    def __init__(self, torch, device):
        from rwkv_wkv_gb300 import Pool
        W = wl.DECODE_12L
        self.torch, self.W = torch, W
        self.H, self.N, self.L = W.H, W.N, W.n_layers
        self.B = 256
        self.pool = Pool(W.n_layers, W.H, W.n_slots, device=device)
        g = torch.Generator(device=device).manual_seed(W.seed)
        self.pool.states.normal_(0.0, 0.1, generator=g)
        slots = wl.distinct_slots(W.seed, "decode/slots", self.B, W.n_slots)
        self.ids = torch.as_tensor(slots.astype(np.int32), device=device)
        self.ins = [wl.token_inputs_device(W.seed, self.B, W.H, W.N, device, generator_offset=l)
                    for l in range(self.L)]
        self.o = [torch.empty(self.B, W.H, W.N, dtype=torch.float32, device=device)
                  for _ in range(self.L)]
        self.phases = ["decode"]
        row = W.H * (2 * HEAD_BYTES_STATE + W.N * 2 * 6 + W.N * 4)
        self.phase_bytes = {"decode": self.L * self.B * row}
        self.tokens_per_step = self.L * self.B  # slot-steps (one slot, one layer)
        self.dominant = "decode"
        self.launches_per_step = self.L

    def step(self, ev=None):
        if ev:
            ev["start"].record()
        for l in range(self.L):
            self.pool.decode_step(l, self.ids, *self.ins[l], o=self.o[l])
        if ev:
            ev["decode"].record()

    def host_io(self):
        return [self.ids] + [t for x in self.ins for t in x], list(self.o)

    def config(self):
        return {"workload": self.W.description, "pool_slots": self.W.n_slots, "layers": self.L,
                "heads": self.H, "head_size": self.N, "decode_slots": self.B,
                "state_dtype": "f32", "input_dtype": "bf16", "output_dtype": "f32"}

    def oracle_sample(self, frac_target):
        return _head_sample(self.H, frac_target, self.B, None, self.tokens_per_step,
                            layers=self.L)


class Sweep(Workload):
    name = wl.SWEEP_32L.name

    def __init__(self, torch, device, batch, state_dtype="f32"):
        from rwkv_wkv_gb300 import Pool
        W = wl.SWEEP_32L
        self.torch, self.W = torch, W
        self.H, self.N, self.L, self.B = W.H, W.N, W.n_layers, batch
        self.state_dtype = state_dtype
        self.state_head_bytes = HEAD_BYTES_STATE // (2 if state_dtype == "bf16" else 1)
        self.pool = Pool(W.n_layers, W.H, W.n_slots, device=device, state_dtype=state_dtype)
        g = torch.Generator(device=device).manual_seed(W.seed)
        for l0 in range(0, W.n_slots, 256):  # in pieces: no float32 temporary of a bf16 pool
            self.pool.states[l0:l0 + 256].normal_(0.0, 0.1, generator=g)
        slots = wl.distinct_slots(W.seed, f"sweep/slots{batch}", batch, W.n_slots)
        self.ids = torch.as_tensor(slots.astype(np.int32), device=device)
        self.ins = wl.token_inputs_device(W.seed, batch, W.H, W.N, device)
        self.o = torch.empty(batch, W.H, W.N, dtype=torch.float32, device=device)
        self.phases = ["decode"]
        row = W.H * (2 * self.state_head_bytes + W.N * 2 * 6 + W.N * 4)
        self.phase_bytes = {"decode": self.L * self.B * row}
        self.tokens_per_step = self.L * self.B
        self.dominant = "decode"
        self.launches_per_step = self.L

    def step(self, ev=None):
        if ev:
            ev["start"].record()
        for l in range(self.L):
            self.pool.decode_step(l, self.ids, *self.ins, o=self.o)
        if ev:
            ev["decode"].record()

    def host_io(self):
        return [self.ids] + list(self.ins), [self.o]

    def config(self):
        return {"workload": self.W.description + f"; batch {self.B}"
                + ("; bf16 state storage" if self.state_dtype == "bf16" else ""),
                "pool_slots": self.W.n_slots,
                "layers": self.L, "heads": self.H, "head_size": self.N, "decode_slots": self.B,
                "state_bytes_per_slot_layer": self.H * self.state_head_bytes,
                "state_dtype": self.state_dtype, "input_dtype": "bf16", "output_dtype": "f32"}

    def oracle_sample(self, frac_target):
        return _head_sample(self.H, frac_target, self.B, None, self.tokens_per_step,
                            layers=self.L)


class Prefill(Workload):
    name = wl.PREFILL_8x4096.name

    def __init__(self, torch, device, checkpoints=False):
        from rwkv_wkv_gb300 import Pool
        W = wl.PREFILL_8x4096
        self.torch, self.W = torch, W
        self.H, self.N = W.H, W.N
        self.S, self.T = 8, 4096
        self.total = self.S * self.T
        self.checkpoints = checkpoints
        n_ck = self.S * (self.T // 64) if checkpoints else 0
        self.pool = Pool(1, W.H, W.n_slots, n_snapshots=n_ck, device=device)
        self.ck = None
        if checkpoints:  # the state after every 64th token of every sequence
            i32 = lambda x: torch.as_tensor(np.asarray(x, dtype=np.int32), device=device)  # noqa: E731
            self.ck = (i32(np.arange(self.S + 1) * (self.T // 64)), i32(np.arange(n_ck)))
        self.pool.alloc(W.n_slots)
        self.pool.free(list(range(W.n_slots))[::-1])
        self.ids = torch.arange(self.S, dtype=torch.int32, device=device)
        self.cu = torch.as_tensor(wl.cu_seqlens([self.T] * self.S), device=device)
        self.ins = wl.token_inputs_device(W.seed, self.total, W.H, W.N, device)
        self.o = torch.empty(self.total, W.H, W.N, dtype=torch.float32, device=device)
        self.phases = ["create", "prefill"]
        self.phase_bytes = {"create": self.S * self.pool.slot_bytes,
                            "prefill": self.total * W.H * (W.N * 2 * 6 + W.N * 4)
                            + self.S * W.H * 2 * HEAD_BYTES_STATE
                            + n_ck * W.H * HEAD_BYTES_STATE}
        self.tokens_per_step = self.total
        self.dominant = "prefill"
        self.launches_per_step = 2

    def step(self, ev=None):
        rec = (lambda name: ev[name].record()) if ev else (lambda name: None)
        rec("start")
        created = self.pool.create(self.S)
        rec("create")
        if self.ck is None:
            self.pool.prefill(0, self.ids, self.cu, *self.ins, o=self.o, max_seqlen=self.T)
        else:
            self.pool.prefill(0, self.ids, self.cu, *self.ins, o=self.o, max_seqlen=self.T,
                              cu_ckpt=self.ck[0], ckpt_ids=self.ck[1])
        rec("prefill")
        self.pool.free(created[::-1])

    def host_io(self):
        meta = [self.ids, self.cu] + (list(self.ck) if self.ck is not None else [])
        return meta + list(self.ins), [self.o]

    def config(self):
        return {"workload": self.W.description
                + (" + state checkpoint every 64 tokens" if self.checkpoints else ""),
                "layers": 1, "heads": self.H,
                "head_size": self.N, "prefill_seqs": self.S, "prefill_tokens": self.total,
                "chunk": 64, "state_dtype": "f32", "input_dtype": "bf16", "output_dtype": "f32",
                "checkpoints": self.S * (self.T // 64) if self.checkpoints else 0}

    def oracle_sample(self, frac_target):
        return _head_sample(self.H, frac_target, 0, np.array([self.T] * self.S),
                            self.tokens_per_step)


class Verify(Workload):
    """Speculative-verify step on slots: K consecutive tokens for each of 1024
    slots of a 4096-slot, 32-head pool in one call, keeping (by default) the
    state after every token for rollback."""
    name = "verify"

    def __init__(self, torch, device, K=5, rollback=True):
        from rwkv_wkv_gb300 import Pool
        W = wl.MIXED
        self.torch, self.W = torch, W
        self.H, self.N, self.K, self.B = W.H, W.N, K, wl.MIXED_DECODE_B
        self.rollback = rollback
        self.pool = Pool(1, W.H, W.n_slots, n_snapshots=self.B * K if rollback else 0,
                         device=device)
        g = torch.Generator(device=device).manual_seed(W.seed)
        self.pool.states.normal_(0.0, 0.1, generator=g)
        slots = wl.distinct_slots(W.seed, "verify/slots", self.B, W.n_slots)
        self.ids = torch.as_tensor(slots.astype(np.int32), device=device)
        self.snaps = (torch.arange(self.B * K, dtype=torch.int32, device=device)
                      if rollback else None)
        flat = wl.token_inputs_device(W.seed, self.B * K, W.H, W.N, device, generator_offset=5)
        self.ins = [x.view(self.B, K, W.H, W.N) for x in flat]
        self.o = torch.empty(self.B, K, W.H, W.N, dtype=torch.float32, device=device)
        per_head = 2 * HEAD_BYTES_STATE + K * (W.N * 2 * 6 + W.N * 4)
        if rollback:
            per_head += K * HEAD_BYTES_STATE
        self.phases = ["verify"]
        self.phase_bytes = {"verify": self.B * W.H * per_head}
        self.tokens_per_step = self.B * K
        self.dominant = "verify"
        self.launches_per_step = 1

    def step(self, ev=None):
        rec = (lambda name: ev[name].record()) if ev else (lambda name: None)
        rec("start")
        self.pool.decode_multi(0, self.ids, *self.ins, o=self.o, step_snap_ids=self.snaps)
        rec("verify")

    def host_io(self):
        meta = [self.ids] + ([self.snaps] if self.snaps is not None else [])
        return meta + list(self.ins), [self.o]

    def config(self):
        return {"workload": f"speculative verify: {self.K} tokens on each of {self.B} slots of a "
                f"{self.W.n_slots}-slot pool, 32 heads x 64, 1 layer"
                + (", state after every token kept for rollback" if self.rollback else ""),
                "pool_slots": self.W.n_slots, "layers": 1, "heads": self.H, "head_size": self.N,
                "rows": self.B, "tokens_per_row": self.K, "rollback_states": self.rollback,
                "state_dtype": "f32", "input_dtype": "bf16", "output_dtype": "f32"}

    def oracle_sample(self, frac_target):
        # each row is a K-token run of the recurrence: the oracle's prefill form
        return _head_sample(self.H, frac_target, 0, np.array([self.K] * self.B),
                            self.tokens_per_step)


class Hibernate(Workload):
    """Hibernate 1024 slots of the mixed step's pool (4096 slots x 32 heads, 512 KiB
    each) to pinned host memory and resume them, one call each per step.  The bound
    is the device's link to host memory, so the roofline peak is a contiguous
    pinned copy of the same bytes measured in the same run."""
    name = "hibernate_1024_of_4096"
    unit = "slots/s"

    def __init__(self, torch, device, batch=1024):
        from rwkv_wkv_gb300 import Pool
        W = wl.MIXED
        self.torch, self.device = torch, device
        self.H, self.N, self.B = W.H, W.N, batch
        self.pool = Pool(1, W.H, W.n_slots, device=device)
        g = torch.Generator(device=device).manual_seed(W.seed)
        self.pool.states.normal_(0.0, 0.1, generator=g)
        plan = wl.mixed_plan()
        self.ids = torch.as_tensor(plan["decode"][:batch].astype(np.int32), device=device)
        self.host = torch.empty(batch * self.pool.slot_bytes, dtype=torch.uint8, pin_memory=True)
        self.phases = ["hibernate", "resume"]
        link = batch * self.pool.slot_bytes
        self.phase_bytes = {"hibernate": link, "resume": link}
        self.tokens_per_step = 2 * batch
        self.dominant = "hibernate"
        self.launches_per_step = 2
        self.no_e2e = True

    def step(self, ev=None):
        rec = (lambda name: ev[name].record()) if ev else (lambda name: None)
        rec("start")
        self.pool.hibernate(self.ids, self.host)
        rec("hibernate")
        self.pool.resume(self.host, self.ids)
        rec("resume")

    def link_peak(self):
        """GB/s of contiguous pinned copies of the same bytes, device->host and back."""
        torch = self.torch
        dev = torch.empty(self.host.numel(), dtype=torch.uint8, device=self.device)
        out = {}
        for name, fn in (("d2h", lambda: self.host.copy_(dev, non_blocking=True)),
                         ("h2d", lambda: dev.copy_(self.host, non_blocking=True))):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            for _ in range(10):
                fn()
            e.record()
            torch.cuda.synchronize()
            out[name] = self.host.numel() * 10 / (s.elapsed_time(e) / 1e3) / 1e9
        del dev
        return out

    def host_io(self):
        return [self.ids], []

    def config(self):
        return {"workload": "hibernate + resume of 1024 slots (32 heads x 64, 1 layer, "
                            "512 KiB per slot) of a 4096-slot pool to pinned host memory",
                "pool_slots": wl.MIXED.n_slots, "layers": 1, "heads": self.H,
                "head_size": self.N, "verb_slots": self.B, "state_dtype": "f32"}

    def oracle_sample(self, frac_target):
        return None


class DecodeMixed(Workload):
    """The mixed serving step's decode call alone: 1024 slots at permuted ids of its
    4096-slot, 32-head pool (the same launch, about 2.2 GB on the device)."""
    name = "decode_1024_of_4096_32H"

    def __init__(self, torch, device):
        from rwkv_wkv_gb300 import Pool
        W = wl.MIXED
        self.torch, self.H, self.N = torch, W.H, W.N
        self.pool = Pool(1, W.H, W.n_slots, device=device)
        g = torch.Generator(device=device).manual_seed(W.seed)
        self.pool.states.normal_(0.0, 0.1, generator=g)
        plan = wl.mixed_plan(W.seed)
        self.ids = torch.as_tensor(plan["decode"].astype(np.int32), device=device)
        B = wl.MIXED_DECODE_B
        self.ins = wl.token_inputs_device(W.seed, B, W.H, W.N, device, generator_offset=1)
        self.o = torch.empty(B, W.H, W.N, dtype=torch.float32, device=device)
        self.phases = ["decode"]
        self.phase_bytes = {"decode": B * W.H * (2 * HEAD_BYTES_STATE + W.N * 2 * 6 + W.N * 4)}
        self.tokens_per_step = B
        self.dominant = "decode"
        self.launches_per_step = 1

    def step(self, ev=None):
        if ev:
            ev["start"].record()
        self.pool.decode_step(0, self.ids, *self.ins, o=self.o)
        if ev:
            ev["decode"].record()

    def host_io(self):
        return [self.ids] + list(self.ins), [self.o]

    def config(self):
        return {"workload": "the mixed step's decode call: 1024 of 4096 slots, 32 heads x 64, 1 layer",
                "pool_slots": wl.MIXED.n_slots, "layers": 1, "heads": self.H, "head_size": self.N,
                "decode_slots": wl.MIXED_DECODE_B, "state_dtype": "f32", "input_dtype": "bf16",
                "output_dtype": "f32"}

    def oracle_sample(self, frac_target):
        return _head_sample(self.H, frac_target, wl.MIXED_DECODE_B, None, self.tokens_per_step)


def make_workload(args, torch, device):
    if args.workload == "mixed":
        return Mixed(torch, device, state_dtype=args.state_dtype, out_dtype=args.out_dtype)
    if args.workload == "decode_mixed":
        return DecodeMixed(torch, device)
    if args.workload == "decode12":
        return Decode12(torch, device)
    if args.workload == "prefill":
        return Prefill(torch, device, checkpoints=args.checkpoints)
    if args.workload == "verify":
        return Verify(torch, device, K=args.verify_k, rollback=not args.no_rollback)
    if args.workload == "hibernate":
        return Hibernate(torch, device)
    return Sweep(torch, device, args.batch, args.state_dtype)


# ------------------------------------------------------------- oracle timing
def prepare_oracle_sample(wk, sample, seed=12345):
    """Seeded host inputs of one oracle sample (drawn once, reused per step)."""
    H, N, nh = wk.H, wk.N, sample["heads"]
    heads = list(range(nh))
    work = []
    n = sample.get("decode_rows", 0)
    for l in range(sample.get("layers", 1) if n else 0):
        ins = wl.token_inputs(seed, f"oracle/dec{l}", n, H, N, dtype="bf16", heads=heads)
        st = wl.slot_states(seed, "oracle/state", range(n), 1, nh, N)[:, 0]
        work.append(("decode", st, [ins[k].astype(np.float64) for k in wl.INPUT_NAMES]))
    lens = sample.get("prefill_lengths")
    if lens is not None and len(lens):
        cu = wl.cu_seqlens(lens)
        ins = wl.token_inputs(seed, "oracle/pre", int(cu[-1]), H, N, dtype="bf16", heads=heads)
        work.append(("prefill", cu, [ins[k].astype(np.float64) for k in wl.INPUT_NAMES],
                     np.zeros((len(lens), nh, N, N))))
    return work


def time_oracle_sample(work, keep=None):
    """Time the CPU oracle on one prepared sample; returns (seconds, threads).
    With a list `keep`, the oracle's (o, final states) of each item are appended."""
    import oracle
    n_threads = os.cpu_count() or 1
    t_total = 0.0
    for item in work:
        t0 = time.perf_counter()
        if item[0] == "decode":
            res = oracle.decode_step(item[1], *item[2], n_threads=n_threads)
        else:
            res = oracle.prefill(item[3], item[1], *item[2], n_threads=n_threads)
        t_total += time.perf_counter() - t0
        if keep is not None:
            keep.append(res)
    return t_total, n_threads


def _default_dtypes(wk) -> bool:
    """Float32 states and outputs: the launch shapes the committed profiles cover."""
    return getattr(wk, "state_dtype", "f32") == "f32" and getattr(wk, "out_dtype", "f32") == "f32"


def gpu_parity(work, refs, out_dtype="f32"):
    """The library on the oracle sample's own inputs (a pool of the sample's heads),
    against the oracle's results: the normwise-max relative error of o and of the
    states, its worst (row or sequence, head) slice (denominators floored at 1% of
    the median slice scale), and the elementwise median |x - y| / (|y| + 1e-6
    max|y|).  Part of the CPU-baseline leg.  With bf16 outputs the tolerance grows by
    half a bf16 unit (2^-8)."""
    import oracle
    import torch
    from rwkv_wkv_gb300 import Pool
    dev = torch.device("cuda", torch.cuda.current_device())
    out = {}
    for item, (o_ref, S_ref) in zip(work, refs):
        ins = [torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev).to(torch.bfloat16)
               for x in item[2]]
        if item[0] == "decode":
            st = item[1]
            n, nh = st.shape[0], st.shape[1]
            with Pool(1, nh, n, device=dev, out_dtype=out_dtype) as pool:
                pool.states[:, 0] = torch.from_numpy(np.ascontiguousarray(st, dtype=np.float32)).to(dev)
                o = pool.decode_step(0, torch.arange(n, dtype=torch.int32, device=dev), *ins)
                status = pool.device_status()
                o, S = o.float().cpu().numpy(), pool.states[:, 0].cpu().numpy()
            slices_o = oracle.rel_err_slices(o, o_ref, 2, floor_frac=1e-2)
            tol = 1e-4
        else:
            cu = item[1]
            st = item[3]
            n, nh = st.shape[0], st.shape[1]
            with Pool(1, nh, n, device=dev, out_dtype=out_dtype) as pool:
                pool.states.zero_()
                o = pool.prefill(0, torch.arange(n, dtype=torch.int32, device=dev),
                                 torch.as_tensor(cu, device=dev), *ins,
                                 max_seqlen=int(np.max(np.diff(cu))))
                status = pool.device_status()
                o, S = o.float().cpu().numpy(), pool.states[:, 0].cpu().numpy()
            slices_o = oracle.rel_err_segments(o, o_ref, cu, floor_frac=1e-2)
            tol = 2e-2
        if out_dtype == "bf16":
            tol += 2.0 ** -8
        out[item[0]] = {"o_normwise": float(f"{oracle.rel_err(o, o_ref):.3e}"),
                        "o_worst_slice": float(f"{float(np.max(slices_o)):.3e}"),
                        "o_elem_median": float(f"{float(np.median(oracle.elementwise_rel(o, o_ref))):.3e}"),
                        "state_normwise": float(f"{oracle.rel_err(S, S_ref):.3e}"),
                        "state_worst_slice": float(f"{float(oracle.rel_err_slices(S, S_ref, 2, floor_frac=1e-2).max()):.3e}"),
                        "tolerance": tol, "device_status": int(status)}
        out[item[0]]["within_tolerance"] = bool(
            status == 0 and max(out[item[0]]["o_normwise"], out[item[0]]["o_worst_slice"],
                                out[item[0]]["state_normwise"], out[item[0]]["state_worst_slice"]) < tol)
    return out


def sized_sample(wk, seconds):
    """A sample whose oracle time is about `seconds` (from a one-head probe)."""
    probe = wk.oracle_sample(1.0 / wk.H)
    t, _ = time_oracle_sample(prepare_oracle_sample(wk, probe))
    frac = min(1.0, probe["frac"] * seconds / max(t, 1e-3))
    sample = wk.oracle_sample(frac)
    return sample, prepare_oracle_sample(wk, sample)


# ------------------------------------------------------------------ our arm
def run_ours(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import rwkv_wkv_gb300 as rw
    rw.load_library()
    wk = make_workload(args, torch, device)
    stream = torch.cuda.current_stream(device)
    peaks = load_peaks()

    graph = None
    if args.graph:
        if args.workload not in ("decode12", "sweep"):
            raise SystemExit("--graph is offered for the decode-only workloads")
        wk.step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            wk.step()
        torch.cuda.synchronize()

    def one_step(ev=None):
        if graph is not None:
            if ev:
                ev["start"].record()
            graph.replay()
            if ev:
                ev[wk.phases[-1]].record()
        else:
            wk.step(ev)

    for _ in range(max(3, args.warmup)):
        one_step()
    torch.cuda.synchronize()

    props = torch.cuda.get_device_properties(device)
    uuid = str(getattr(props, "uuid", "") or "")
    gpu_id = uuid if uuid.startswith("GPU-") else (f"GPU-{uuid}" if uuid else str(local))
    clocks = ClockSampler(gpu_id)
    clocks.wait_first()

    names = ["start"] + wk.phases
    events = [{n: torch.cuda.Event(enable_timing=True) for n in names}
              for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    # The timed region is exactly K steps between a barrier and a device sync on both
    # sides.  It is repeated R times (R >= 3, enough repeats to cover --min-timed-s, the
    # same R on every rank) so that the clock sampler sees the GPU under this load; the
    # reported time is the median repeat.
    reps, phase_samples = [], {n: [] for n in wk.phases}
    n_rep = None
    launches0 = rw.launch_count()
    t_wall0 = time.time()
    while n_rep is None or len(reps) < n_rep:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for k in range(args.steps):
            one_step(events[k])
        end.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        reps.append(start.elapsed_time(end) / 1e3)
        prev = "start"
        for n in wk.phases:
            src = "start" if graph is not None else prev
            phase_samples[n].extend(e[src].elapsed_time(e[n]) for e in events)
            prev = n
        if n_rep is None:
            want = max(3, min(50, int(np.ceil(args.min_timed_s / max(reps[0], 1e-6)))))
            n_rep = int(aggregate(0.0, float(want), world, device, op="max")[1]) if world > 1 else want
    t_wall1 = time.time()
    launches = (rw.launch_count() - launches0) // n_rep
    if graph is not None:
        launches = wk.launches_per_step * args.steps
    clk = clocks.summary(t_wall0, t_wall1)
    clocks.stop()
    elapsed = statistics.median(reps)
    phase_ms = {n: statistics.mean(v) for n, v in phase_samples.items()}
    if graph is not None:
        phase_ms = {wk.phases[-1]: phase_ms[wk.phases[-1]]}
    units = wk.tokens_per_step * args.steps
    elapsed_max, units_all = aggregate(elapsed, units, world, device)
    value = units_all / elapsed_max

    hbm = peaks["hbm_gbs"]
    dom = wk.dominant
    dom_ms = phase_ms.get(dom, elapsed * 1e3 / args.steps)
    achieved = wk.phase_bytes[dom] / (dom_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "peak_source": peaks["source"] + " (hbm copy)",
                "bytes_per_launch": wk.phase_bytes[dom], "ms_per_launch": round(dom_ms, 4),
                "traffic": profiled_traffic(dom, args.workload) if _default_dtypes(wk) else None,
                "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)"}
    phases = {}
    for n in wk.phases:
        ms = phase_ms.get(n)
        if ms is None:
            continue
        gbs = wk.phase_bytes[n] / (ms / 1e3) / 1e9
        phases[n] = {"ms": round(ms, 4), "GB_per_s": round(gbs, 1),
                     "hbm_frac": round(gbs / hbm, 4)}
    if hasattr(wk, "link_peak"):  # bound by the link to host memory, not by HBM
        link = wk.link_peak()
        for n, direction in (("hibernate", "d2h"), ("resume", "h2d")):
            phases[n] = {"ms": phases[n]["ms"], "GB_per_s": phases[n]["GB_per_s"],
                         "link_frac": round(phases[n]["GB_per_s"] / link[direction], 4),
                         "link_peak_GB_per_s": round(link[direction], 1)}
        roofline = {"bound": "host link", "kernel": "slot_copy_kernel (hibernate)",
                    "achieved": phases["hibernate"]["GB_per_s"], "peak": round(link["d2h"], 1),
                    "unit": "GB/s", "frac": phases["hibernate"]["link_frac"],
                    "peak_source": "measured in this run: contiguous pinned device->host copy "
                                   "of the same bytes (cudaMemcpyAsync through torch)",
                    "bytes_per_launch": wk.phase_bytes["hibernate"],
                    "ms_per_launch": phases["hibernate"]["ms"], "traffic": None}
    if hasattr(wk, "verb_ceiling"):  # small copies: also against a same-size device copy
        ceil = wk.verb_ceiling()
        for n in ("create", "snapshot", "fork", "restore"):
            if n in phases:
                ref = ceil["fill"] if n == "create" else ceil["copy"]
                phases[n]["same_size_device_copy_GB_per_s"] = round(ref, 1)
                phases[n]["frac_of_same_size_device_copy"] = round(phases[n]["GB_per_s"] / ref, 4)
    extra = {}
    if "decode" in phase_ms:
        rows = wk.phase_bytes["decode"]
        per_row = wk.H * (2 * getattr(wk, "state_head_bytes", HEAD_BYTES_STATE) + wk.N * 2 * 6
                          + wk.N * getattr(wk, "out_elem_bytes", 4))
        n_slot_steps = rows // per_row
        extra["decode"] = {"slot_steps_per_s": round(n_slot_steps / (phase_ms["decode"] / 1e3), 1),
                           "GB_per_s": phases["decode"]["GB_per_s"],
                           "hbm_frac": phases["decode"]["hbm_frac"],
                           "traffic": profiled_traffic("decode", args.workload)
                           if _default_dtypes(wk) else None}
    if "verify" in phase_ms:
        extra["verify"] = {"slot_token_steps_per_s": round(wk.tokens_per_step
                                                           / (phase_ms["verify"] / 1e3), 1),
                           "GB_per_s": phases["verify"]["GB_per_s"],
                           "hbm_frac": phases["verify"]["hbm_frac"]}
    if "prefill" in phase_ms:
        extra["prefill"] = {"tokens_per_s": round(wk.total / (phase_ms["prefill"] / 1e3), 1),
                            "GB_per_s": phases["prefill"]["GB_per_s"],
                            "roofline_frac": phases["prefill"]["hbm_frac"],
                            "bound": "hbm"}

    cfg = wk.config()
    state_dtype = getattr(wk, "state_dtype", "f32")
    out_dtype = getattr(wk, "out_dtype", "f32")

    unit = getattr(wk, "unit", "tokens/s")

    e2e = None
    if not args.no_e2e and graph is None and not getattr(wk, "no_e2e", False):
        e2e = run_e2e(torch, wk, args, world, device)

    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and wk.oracle_sample(0.01):
        cpu_base = cpu_baseline(wk, target_seconds=8.0)

    targets = None
    if (args.workload == "mixed" and world == 1 and not args.no_targets and _default_dtypes(wk)):
        del wk  # free the mixed step's pool before the next workloads are built
        torch.cuda.empty_cache()
        targets = run_targets(torch, device, args, peaks)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(elapsed_max * 1e3 / args.steps, 4),
        "repeats": n_rep,
        "ms_per_step_repeats": {"median": round(statistics.median(reps) * 1e3 / args.steps, 4),
                                "min": round(min(reps) * 1e3 / args.steps, 4),
                                "max": round(max(reps) * 1e3 / args.steps, 4)},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 state, f32 arithmetic" if state_dtype == "bf16"
                 else "f32+bf16", "data": "synthetic",
        "config": full_config(cfg, world, bool(graph)),
        "roofline": roofline, "phases": phases, **extra,
        "targets": targets,
        "e2e": e2e, "gpu_launches": int(launches), "clocks": clk,
        "cpu_baseline": cpu_base,
        "dtype_note": ("state stored in bf16 (each step computed in float32, the new state rounded "
                       "to bf16); decode arithmetic and outputs float32; inputs bf16"
                       if state_dtype == "bf16" else
                       "state, decode arithmetic and outputs float32; prefill contractions "
                       "bf16 tensor-core operands with float32 accumulation; inputs bf16")
                      + ("; outputs rounded to bf16 as stored" if out_dtype == "bf16" else ""),
    }
    if world > 1:
        torch.distributed.destroy_process_group()
    return line if rank == 0 else None


def full_config(cfg: dict, world: int, graph: bool) -> dict:
    """The line's config: the workload's own keys plus how it was run (the same
    keys for both arms)."""
    return dict(cfg, parallelism=f"replicas x{world}" if world > 1 else "1 gpu",
                l2="inputs larger than L2 (every step moves > 129 MB)", graph=bool(graph))


def _time_phase(torch, step, phase, steps, warmup, reps=3):
    """Median over `reps` repeats of the mean CUDA-event time (ms) of `phase`
    over `steps` steps, after `warmup` untimed steps."""
    for _ in range(warmup):
        step(None)
    torch.cuda.synchronize()
    means = []
    for _ in range(reps):
        evs = [{n: torch.cuda.Event(enable_timing=True) for n in ("start", phase)}
               for _ in range(steps)]
        for e in evs:
            step(e)
        torch.cuda.synchronize()
        means.append(statistics.mean(e["start"].elapsed_time(e[phase]) for e in evs))
    return statistics.median(means)


def run_targets(torch, device, args, peaks):
    """The two figures the method statement sets targets on, measured in the same
    process after the mixed step (each pool freed before the next is built):
    the chunked prefill of 8 sequences x 4096 tokens x 32 heads (prefill >= 50% of
    its HBM roofline) and the 32-layer x 64-head decode sweep at B = 1024 and
    B = 4096 slots (decode >= 70% of HBM at >= 1024 slots), the sweep replayed as
    a CUDA graph of its 32 layer calls."""
    hbm = peaks["hbm_gbs"]
    out = {}
    wk = Prefill(torch, device)

    def pstep(ev):
        if ev:
            ev["start"].record()
        wk.pool.prefill(0, wk.ids, wk.cu, *wk.ins, o=wk.o, max_seqlen=wk.T)
        if ev:
            ev["prefill"].record()
    ms = _time_phase(torch, pstep, "prefill", steps=10, warmup=3)
    nbytes = wk.phase_bytes["prefill"]
    gbs = nbytes / (ms / 1e3) / 1e9
    out["prefill_8x4096"] = {
        "workload": wk.W.description, "ms": round(ms, 4),
        "tokens_per_s": round(wk.total / (ms / 1e3), 1),
        "roofline": {"bound": "hbm", "kernel": "prefill_chunk_kernel", "achieved": round(gbs, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                     "bytes_per_launch": nbytes, "ms_per_launch": round(ms, 4),
                     "peak_source": peaks["source"] + " (hbm copy)"},
        "target_frac": 0.5}
    del wk, pstep
    torch.cuda.empty_cache()
    sweep = {}
    for B in (1024, 4096):
        wk = Sweep(torch, device, B)
        wk.step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            wk.step()
        torch.cuda.synchronize()

        def sstep(ev):
            if ev:
                ev["start"].record()
            g.replay()
            if ev:
                ev["decode"].record()
        ms = _time_phase(torch, sstep, "decode", steps=5, warmup=3)
        nbytes = wk.phase_bytes["decode"]
        gbs = nbytes / (ms / 1e3) / 1e9
        sweep[f"B{B}"] = {"ms_per_sweep": round(ms, 3),
                          "slot_steps_per_s": round(wk.tokens_per_step / (ms / 1e3), 1),
                          "GB_per_s": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4)}
        del g, wk, sstep
        torch.cuda.empty_cache()
    out["sweep_32L_64H"] = dict(sweep, workload=wl.SWEEP_32L.description
                                + "; 32 layer calls replayed as one CUDA graph",
                                bytes_per_slot_step=2 * 64 * 64 * 64 * 4 + 64 * 64 * (6 * 2 + 4),
                                target_hbm_frac=0.7)
    return out


def run_e2e(torch, wk, args, world, device):
    """Same steps through the public API with pinned host buffers: every step
    uploads its inputs host->device and reads its outputs back device->host, all
    inside the timed region.  Steps whose copies are large enough to be bound by
    the link (over 256 MB) are pipelined as a serving loop would: the copies run on
    their own streams (the link is full duplex), so while step k computes, step
    k+1's inputs go up and step k-1's outputs come down; each per-step tensor has
    two device buffers and the workload's tensors are pointed at buffer k % 2
    before step k (the library reads device pointers at call time).  Smaller steps
    are bound by the host-side cost of their many small copies, which the extra
    bookkeeping would only add to, and run copy-in, step, copy-out in order."""
    ins, outs = wk.host_io()
    h_ins = [t.cpu().pin_memory() for t in ins]
    h_outs = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs] for _ in range(2)]
    buf_in = [[t.clone() for t in ins] for _ in range(2)]
    buf_out = [[torch.empty_like(t) for t in outs] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    steps = max(3, min(args.steps, 20))
    pipelined = h2d + d2h > (256 << 20)
    compute = torch.cuda.current_stream(device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):  # every buffer starts free
        done[b].record(compute)
        out_free[b].record(compute)

    def step_in_order(k):
        for d, h in zip(ins, h_ins):
            d.copy_(h, non_blocking=True)
        wk.step()
        for h, d in zip(h_outs[0], outs):
            h.copy_(d, non_blocking=True)

    def step_pipelined(k):
        b = k % 2
        with torch.cuda.stream(s_in):  # upload step k's inputs once step k-2 has consumed buffer b
            s_in.wait_event(done[b])
            for d, h in zip(buf_in[b], h_ins):
                d.copy_(h, non_blocking=True)
            in_ready[b].record(s_in)
        compute.wait_event(in_ready[b])
        compute.wait_event(out_free[b])  # step k-2's outputs have been read back
        for t, d in zip(ins, buf_in[b]):
            t.set_(d)
        for t, d in zip(outs, buf_out[b]):
            t.set_(d)
        wk.step()
        done[b].record(compute)
        with torch.cuda.stream(s_out):  # read step k's outputs back
            s_out.wait_event(done[b])
            for h, d in zip(h_outs[b], buf_out[b]):
                h.copy_(d, non_blocking=True)
            out_free[b].record(s_out)

    step = step_pipelined if pipelined else step_in_order
    for k in range(2):
        step(k)
    torch.cuda.synchronize()
    # Three timed runs of `steps` steps each; the host link's rate varies between runs
    # (other tenants share it), so the line carries the median run and the spread.
    runs = []
    for _ in range(3):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(compute)
        s_in.wait_stream(compute)
        s_out.wait_stream(compute)
        for k in range(steps):
            step(k)
        compute.wait_stream(s_in)
        compute.wait_stream(s_out)
        e.record(compute)
        torch.cuda.synchronize()
        elapsed_max, units = aggregate(s.elapsed_time(e) / 1e3, wk.tokens_per_step * steps, world,
                                       device)
        runs.append(units / elapsed_max)
    value = statistics.median(runs)
    return {"value": round(value, 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": steps, "ms_per_step": round(1e3 * wk.tokens_per_step * world / value, 3),
            "runs": 3, "value_min": round(min(runs), 1), "value_max": round(max(runs), 1),
            "copies": "own streams, overlapping neighbouring steps (double-buffered)" if pipelined
                      else "in order around each step"}


def cpu_baseline(wk, target_seconds=12.0, parity=True):
    """The oracle timed on the host cores on a bounded sample of the workload; with
    `parity`, the library is also run on the same sample and compared with it."""
    sample, work = sized_sample(wk, target_seconds)
    refs = []
    t, threads = time_oracle_sample(work, keep=refs)
    step_s = t / sample["frac"]
    out = {"value": round(wk.tokens_per_step / step_s, 1), "unit": "tokens/s",
           "cores": threads, "kind": "oracle", "seconds": round(t, 2),
           "sample": sample["desc"]}
    if parity:
        out["parity_on_sample"] = gpu_parity(work, refs, getattr(wk, "out_dtype", "f32"))
    return out


# ------------------------------------------------------------ reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    if args.workload == "hibernate":
        return {"impl": "reference", "unavailable": "the oracle computes the recurrence only; "
                "a slot copy to host memory has no CPU reference computation"}
    # The oracle needs the workload's shapes only: built without a GPU.
    wk = _shapes_only(args)
    per_step = min(5.0, 90.0 / max(1, args.steps + args.warmup))
    sample, work = sized_sample(wk, per_step)
    for _ in range(args.warmup):
        time_oracle_sample(work)
    runs = [time_oracle_sample(work) for _ in range(args.steps)]
    times = [t for t, _ in runs]
    threads = runs[0][1] if runs else (os.cpu_count() or 1)
    step_s = statistics.mean(times) / sample["frac"]
    value = wk.tokens_per_step / step_s
    cfg = wk.config()
    return {"impl": "reference", "metric": METRIC, "value": round(value, 1),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": full_config(cfg, world, args.graph),
            "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": threads,
                             "kind": "oracle", "sample": sample["desc"]},
            "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def _shapes_only(args):
    """A workload object carrying shapes and sample plans, with no device state;
    its config() is the GPU arm's own (the same method on the same attributes)."""
    class S(Workload):
        pass
    s = S()
    s.state_dtype = args.state_dtype
    s.state_head_bytes = HEAD_BYTES_STATE // (2 if args.state_dtype == "bf16" else 1)
    s.out_dtype = args.out_dtype if args.workload == "mixed" else "f32"
    if args.workload == "mixed":
        plan = wl.mixed_plan()
        s.H, s.N = wl.MIXED.H, wl.MIXED.N
        s.lengths = plan["lengths"].astype(np.int64)
        s.total = int(s.lengths.sum())
        s.tokens_per_step = wl.MIXED_DECODE_B + s.total
        cls = Mixed
    elif args.workload == "decode12":
        W = wl.DECODE_12L
        s.H, s.N, s.L, s.B, s.W = W.H, W.N, W.n_layers, 256, W
        s.tokens_per_step = s.L * s.B
        cls = Decode12
    elif args.workload == "prefill":
        W = wl.PREFILL_8x4096
        s.H, s.N, s.S, s.T, s.W = W.H, W.N, 8, 4096, W
        s.total = s.S * s.T
        s.checkpoints = args.checkpoints
        s.tokens_per_step = s.total
        cls = Prefill
    elif args.workload == "decode_mixed":
        s.H, s.N = wl.MIXED.H, wl.MIXED.N
        s.tokens_per_step = wl.MIXED_DECODE_B
        cls = DecodeMixed
    elif args.workload == "verify":
        W = wl.MIXED
        s.H, s.N, s.K, s.B, s.W = W.H, W.N, args.verify_k, wl.MIXED_DECODE_B, W
        s.rollback = not args.no_rollback
        s.tokens_per_step = s.B * s.K
        cls = Verify
    else:
        W = wl.SWEEP_32L
        s.H, s.N, s.L, s.B, s.W = W.H, W.N, W.n_layers, args.batch, W
        s.tokens_per_step = s.L * s.B
        cls = Sweep
    s.oracle_sample = lambda f: cls.oracle_sample(s, f)
    s.config = lambda: cls.config(s)
    return s


def main(argv=None):
    args = parse_args(argv)
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
