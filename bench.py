#!/usr/bin/env python3
"""Benchmark of the paged GQA attention hot path (libpagedattn) on GB300.

The metric is paged-GQA decode KV GB/s.  The headline step is one pass of the decode calls
over their workloads, inputs resident in HBM:
  1. pa_append_decode          append of 64 new tokens fused with the batched decode (64 seqs,
                               ctx ~U[1024,1152], 32q/8kv/128): pa_kv_append + pa_decode in one launch
  2. pa_decode_splitkv         4 x 8192, P in 8..32 (Qwen3-32B-shaped 64q/8kv/128), then
     pa_combine                its log-sum-exp merge
  3. pa_decode_splitkv         1 x 32768, P in 8..32, then pa_combine
value = the KV bytes those calls must read (each (block, kv head) tile once) / step time.
The full hot path adds the chunked prefill's workload to the step ("full_step"):
  4. pa_kv_append              8 x 256 chunk tokens
  5. pa_prefill_chunked        8 x 256-token causal chunks over a shared 768-token prefix, 32q/8kv/128
whose KV bytes count the shared prefix once.  The workloads are independent requests on
separate pools, so a step runs each on a stream of its own, forked from and joined back into
one stream; it is captured once as a CUDA graph with those parallel branches and replayed, as a
serving loop replays its step.  The same calls one after another on one stream are timed too
("step_serial_us").  L2 is flushed (a 512 MB buffer is read) before every timed replay, outside
the timed interval.

Every call is also timed on its own ("per_call"; the split-KV partitions and their combine as
one unit): a graph of [L2 flush, event, call, event] is replayed and the interval between the
two event nodes is "us_isolated" (it carries the call's launch latency: about 5 us even for
an empty kernel on this harness).  "us" is the marginal cost of one more launch in a stream:
the same graph with the call run a second time on a second, untouched copy of its inputs
(L2-cold as well), minus the isolated time (median, p10, p90).  Fractions use "us", against
the measured HBM copy peak and the nominal 8 TB/s, or the measured bf16 peak.

The end-to-end numbers ("e2e" for the decode step, "full_step.e2e" for the full path) run the
step through the public API with host buffers, the copies inside the timed interval: each
workload's inputs are staged in one pinned host buffer; they go up on a copy stream, piece by
piece (each decode workload whole, then the chunked prefill in two groups of sequences); each
piece's calls run on a compute stream of their own once its inputs have arrived, and its output
comes back on a copy stream of its own as soon as it is done.  That step is captured as one
CUDA graph (copies included) and replayed; "eager_value" issues it from Python call by call
(host-bound).  The e2e outputs are checked bit for bit against the step's.  The two
latency-bound decode shapes (1 seq x 37 tokens, 4q/1kv/64; 1 seq x 1152 tokens, 32q/8kv/128)
and a speculative-verify shape are reported under "latency".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--serial-step]

--impl reference times the CPU fp64 oracle (the reference arm of this comparison) on a
bounded sample of the decode step, on all host cores.  Under torchrun (N > 1) every rank runs
the full step on its own GPU (independent replicas, weak scaling); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import tempfile
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "paged GQA decode: KV GB/s & frac of GB300 HBM peak; µs/call per batch×ctx"
WORKLOAD = ("decode step: fused append(64)+decode 64x~1088 (32q/8kv/128) + split-KV 4x8192 and 1x32768 "
            "(P in 8..32) with their log-sum-exp combine (64q/8kv/128); block 16; bf16 N(0,1)")
FULL_WORKLOAD = WORKLOAD.replace("decode step", "full hot path") + (
    " + append(2048) + chunked prefill 8x256 over a shared 768-token prefix (32q/8kv/128)")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal
DECODE_WORKLOADS = ("batched_decode", "splitkv_4x8192", "splitkv_1x32768")
FULL_WORKLOADS = ("chunked_prefill",) + DECODE_WORKLOADS  # longest chain first
KERNEL_SOURCES = {
    "decode": ["pa_decode.cu", "pa_block_attn.cuh", "pa_device.cuh"],
    "splitkv": ["pa_decode.cu", "pa_block_attn.cuh", "pa_device.cuh"],
    "prefill": ["pa_prefill_tc2.cu", "pa_device.cuh"],  # the tcgen05 kernel the profile covers
    "append": ["pa_append.cu", "pa_device.cuh"],
    "combine": ["pa_decode.cu", "pa_device.cuh"],
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------- peaks, clocks, profiles
def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text: str) -> str:
    """A source without its comments, blank lines and layout whitespace: what a change to the
    kernel changes."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    lines = (" ".join(line.split("//", 1)[0].split()) for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def source_sha(kind: str) -> str:
    """Hash of the kernel sources a profile's counters were taken on, comments aside."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        h.update(_code_only((ROOT / "paged_kv_gqa_slot_gb300" / "csrc" / f).read_text()).encode())
    return h.hexdigest()[:12]


def profiled_traffic(kind: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if its sources still match."""
    pat = re.compile(r"^traffic:\s+kernel=(\S+)\s+workload=(\S+)\s+dram_bytes_per_launch=(\d+)\s+source_sha=(\S+)")
    for f in sorted((ROOT / "profiles").glob("*.md")):
        for line in f.read_text().splitlines():
            m = pat.match(line.strip())
            if m and m.group(1) == kind and m.group(2) == workload:
                return int(m.group(3)) if m.group(4) == source_sha(kind) else None
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU is under load."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.NamedTemporaryFile(mode="w", prefix="pa_clocks_", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in Path(self.out.name).read_text().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        try:
            os.unlink(self.out.name)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- work per call
def causal_flops(case) -> float:
    """QK^T and PV multiply-adds of the chunked prefill, causal-exact (2 flops each)."""
    keys = 0
    for L, C in zip(case.seq_lens.tolist(), case.q_lens):
        pre = L - C
        keys += C * pre + C * (C + 1) // 2
    return float(keys) * case.num_heads * case.head_dim * 4


def unique_kv_bytes(case) -> int:
    """Bytes of K and V the attention must read: every (pool slot, kv head) row that some
    sequence attends to, counted once (a prefix shared by several sequences counts once)."""
    bs = case.block_size
    slots = []
    bt = case.block_tables.numpy()
    for s, L in enumerate(case.seq_lens.tolist()):
        t = np.arange(L)
        slots.append(bt[s, t // bs].astype(np.int64) * bs + t % bs)
    n = np.unique(np.concatenate(slots)).size if slots else 0
    return int(n) * case.num_kv_heads * case.head_dim * 2 * 2


def attn_bytes(case) -> int:
    """Algorithmic bytes of one attention call: its unique K/V rows plus q and out."""
    return unique_kv_bytes(case) + 2 * case.q.numel() * 2


class Call:
    """One unit of the step's work as timed on its own: one or more launches of one workload
    (the split-KV partitions and their merge together), with its algorithmic work."""

    def __init__(self, name, kind, fns, units, unit_kind, workload):
        self.name, self.kind, self.fns, self.units, self.unit_kind, self.workload = (name, kind, fns, units, unit_kind,
                                                                                    workload)

    def fn(self):
        for f in self.fns:
            f()


class Step:
    """Device-resident inputs of the benchmark's workloads and the calls that make a step.
    With copies=2 every workload also has a second, independent set of device buffers
    (calls_alt), for timing a call as the marginal cost of one more launch on cold inputs."""

    GROUPS = {"decode": ("c3",), "splitkv": ("c4a", "c4b"), "prefill": ("c5",), "decode_step": ("c3", "c4a", "c4b")}

    def __init__(self, device, only=None, copies=1):
        import paged_kv_gqa_slot_gb300 as pa
        import workloads as W
        self.pa = pa
        groups = set(self.GROUPS[only]) if only else {"c3", "c4a", "c4b", "c5"}
        t0 = time.time()
        self.c3 = W.batched_decode() if "c3" in groups else None
        self.c4a = W.splitkv_decode(1004, 4, 8192) if "c4a" in groups else None
        self.c4b = W.splitkv_decode(1004, 1, 32768) if "c4b" in groups else None
        self.c5 = W.chunked_prefill() if "c5" in groups else None
        log(f"[bench] workloads drawn in {time.time() - t0:.1f}s")
        self.dev = device
        # partitions as the library suggests, kept within the workload's 8..32
        self.P4a = min(32, max(8, pa.pa_splitkv_num_partitions(4, 8, 512))) if self.c4a is not None else 8
        self.P4b = min(32, max(8, pa.pa_splitkv_num_partitions(1, 8, 2048))) if self.c4b is not None else 32
        self.copies = [self._upload() for _ in range(copies)]
        self.calls = self._calls(self.copies[0])
        self.calls_alt = self._calls(self.copies[1]) if copies > 1 else None
        g3, g4a, g4b, g5 = (self.copies[0][k] for k in ("c3", "c4a", "c4b", "c5"))
        self.by_name = {"batched_decode": (g3, self.c3), "splitkv_4x8192": (g4a, self.c4a),
                        "splitkv_1x32768": (g4b, self.c4b), "chunked_prefill": (g5, self.c5)}
        self.available = tuple(w for w in FULL_WORKLOADS if self.by_name[w][1] is not None)
        self.streams = {w: torch.cuda.Stream(device=device) for w in self.available}

    def _upload(self):
        """One set of device buffers for every workload: {"c3": g, ...}."""
        pa, d = self.pa, self.dev

        def up(c, P=None):
            """A workload's pool, and its per-step inputs packed into one device buffer (views
            at 256-byte aligned offsets, the small tables first, then the new K and V rows and
            q) with a pinned host copy of the same layout: a serving loop stages a step's
            inputs like this, so that they go up in few copies."""
            if c is None:
                return None
            g = {"k": c.k_cache.to(d), "v": c.v_cache.to(d)}
            g["pool"] = pa.PaPool(g["k"], g["v"])
            ins = {"bt": c.block_tables, "sl": c.seq_lens, "cu": c.cu_q_lens, "slots": c.slot_mapping}
            if c is self.c5:  # the prefill groups' cu_q_lens, rebased to 0, for the e2e pipeline
                for i, (b0, b1) in enumerate(prefill_groups(c)):
                    ins[f"cu{i}"] = c.cu_q_lens[b0:b1 + 1] - c.cu_q_lens[b0]
            ins.update({"k_new": c.k_new, "v_new": c.v_new, "q": c.q})
            layout, off = {}, 0
            for key, t in ins.items():
                off = (off + 255) // 256 * 256
                layout[key] = off
                off += t.numel() * t.element_size()
            host = torch.empty(max(off, 1), dtype=torch.uint8).pin_memory()
            dev = torch.empty(max(off, 1), dtype=torch.uint8, device=d)
            for key, t in ins.items():
                nb = t.numel() * t.element_size()
                host[layout[key]:layout[key] + nb].copy_(t.contiguous().view(-1).view(torch.uint8))
                g[key] = dev[layout[key]:layout[key] + nb].view(t.dtype).view(t.shape)
            dev.copy_(host)
            g["in_host"], g["in_dev"], g["in_layout"] = host, dev, layout
            g["out"] = torch.empty_like(g["q"])
            if P is not None:
                g["ws_o"] = torch.empty((c.batch, c.num_heads, P, c.head_dim), dtype=torch.float32, device=d)
                g["ws_lse"] = torch.empty((c.batch, c.num_heads, P), dtype=torch.float32, device=d)
            return g

        return {"c3": up(self.c3), "c4a": up(self.c4a, self.P4a), "c4b": up(self.c4b, self.P4b), "c5": up(self.c5)}

    def _calls(self, gs):
        pa = self.pa
        c3, c4a, c4b, c5 = self.c3, self.c4a, self.c4b, self.c5
        g3, g4a, g4b, g5 = gs["c3"], gs["c4a"], gs["c4b"], gs["c5"]
        app_bytes = lambda c: 2 * 2 * c.k_new.numel() * 2  # read new rows, write pool rows, K and V
        calls = []
        if g3 is not None:
            # the decode step's append and attention in one launch (pa_append_decode)
            calls.append(Call(
                "append_decode[batched_decode,64x~1088]", "decode",
                [lambda: pa.pa_append_decode(g3["pool"], g3["k_new"], g3["v_new"], g3["slots"], g3["q"], g3["bt"],
                                             g3["sl"], c3.scale, g3["out"])],
                attn_bytes(c3) + app_bytes(c3), "bytes", "batched_decode"))
        for g, c, P, wl, tag in ((g4a, c4a, self.P4a, "splitkv_4x8192", "4x8192"),
                                 (g4b, c4b, self.P4b, "splitkv_1x32768", "1x32768")):
            if g is None:
                continue
            calls.append(Call(
                f"decode_splitkv+combine[{tag},P={P}]", "splitkv",
                [lambda g=g, c=c, P=P: pa.pa_decode_splitkv(g["pool"], g["q"], g["bt"], g["sl"], c.scale, P,
                                                            g["ws_o"], g["ws_lse"]),
                 lambda g=g: pa.pa_combine(g["ws_o"], g["ws_lse"], g["out"])],
                attn_bytes(c), "bytes", wl))
        if g5 is not None:
            mx5 = max(c5.q_lens)
            calls += [
                Call("kv_append[chunked_prefill,2048]", "append",
                     [lambda: pa.pa_kv_append(g5["pool"], g5["k_new"], g5["v_new"], g5["slots"])], app_bytes(c5),
                     "bytes", "chunked_prefill"),
                Call("prefill_chunked[8x256 over 768]", "prefill",
                     [lambda: pa.pa_prefill_chunked(g5["pool"], g5["q"], g5["cu"], g5["bt"], g5["sl"], c5.scale, mx5,
                                                    g5["out"])], causal_flops(c5), "flops", "chunked_prefill")]
        return calls

    def kv_bytes(self, workloads) -> int:
        """KV bytes the attention calls of these workloads must read (unique rows)."""
        return sum(unique_kv_bytes(self.by_name[w][1]) for w in workloads if w in self.available)

    def calls_of(self, workloads):
        return [c for c in self.calls if c.workload in workloads]

    def launches(self, workloads) -> int:
        return sum(len(c.fns) for c in self.calls_of(workloads))

    def run(self, workloads):
        """The workloads' calls one after another on the current stream."""
        for c in self.calls_of(workloads):
            c.fn()

    def run_parallel(self, workloads):
        """Every workload on a stream of its own, forked from the current stream and joined
        back into it: the workloads are independent requests on separate pools, and one
        workload's latency-bound stretches (a kernel's start, its last wave) leave SMs and
        HBM bandwidth that another's calls can use."""
        main = torch.cuda.current_stream(self.dev)
        ws = [w for w in FULL_WORKLOADS if w in workloads and w in self.available]
        for w in ws:
            self.streams[w].wait_stream(main)
        for w in ws:
            with torch.cuda.stream(self.streams[w]):
                for c in self.calls_of((w,)):
                    c.fn()
        for w in ws:
            main.wait_stream(self.streams[w])


# groups of prefill sequences in the e2e pipeline (1, 2, 3 and 4 measured; 2 and 3 best)
E2E_PREFILL_GROUPS = 2


def prefill_groups(c):
    """The e2e pipeline's groups of prefill sequences: [(b0, b1), ...]."""
    n = max(1, min(E2E_PREFILL_GROUPS, c.batch))
    edges = [c.batch * i // n for i in range(n + 1)]
    return [(b0, b1) for b0, b1 in zip(edges[:-1], edges[1:]) if b1 > b0]


class E2E:
    """One step of the given workloads as a serving loop runs it with its inputs in pinned host
    memory: every piece's inputs go up on one copy stream as early as possible, its calls run on
    a compute stream of their own once they have arrived, and its output comes back on another
    copy stream as soon as its last call is done (one copy stream per piece, so that none waits
    behind another's output), while later pieces are still going up or computing.

    The pieces, in upload order: each decode workload whole (its inputs in one copy), then the
    chunked prefill in groups of sequences (the first group also brings the workload's small
    tables; each group its rows of new K, new V and q, three copies).  A prefill group is an
    append and a prefill over its own sequences (views of the workload's tensors, cu_q_lens
    rebased to 0): the same per-sequence arithmetic as the one-launch prefill, so the same
    bits."""

    def __init__(self, step: Step, workloads):
        pa = step.pa
        self.step = step
        self.dev = step.dev
        self.workloads = [w for w in DECODE_WORKLOADS + ("chunked_prefill",) if w in workloads and w in step.available]
        self.pieces = []
        for w in self.workloads:
            g, c = step.by_name[w]
            if w != "chunked_prefill":
                d2h = [(torch.empty_like(g["out"], device="cpu").pin_memory(), g["out"])]
                fns = [f for call in step.calls_of((w,)) for f in call.fns]
                self.pieces.append(([(g["in_host"], g["in_dev"])], d2h, fns, w))
                continue
            assert c.k_new.shape[0] == sum(c.q_lens), "prefill workload: one appended row per chunk query"
            cu = c.cu_q_lens.tolist()
            lay, hb, db = g["in_layout"], g["in_host"], g["in_dev"]
            row = c.k_new[0].numel() * 2  # bytes of one new K (or V) row
            qrow = c.q[0].numel() * 2
            for i, (b0, b1) in enumerate(prefill_groups(c)):
                r0, r1 = cu[b0], cu[b1]
                h2d = [(hb[lay["bt"]:lay["k_new"]], db[lay["bt"]:lay["k_new"]])] if i == 0 else []
                for key, rb in (("k_new", row), ("v_new", row), ("q", qrow)):
                    h2d.append((hb[lay[key] + r0 * rb:lay[key] + r1 * rb], db[lay[key] + r0 * rb:lay[key] + r1 * rb]))
                dv = {"q": g["q"][r0:r1], "k_new": g["k_new"][r0:r1], "v_new": g["v_new"][r0:r1],
                      "slots": g["slots"][r0:r1], "bt": g["bt"][b0:b1], "sl": g["sl"][b0:b1], "cu": g[f"cu{i}"],
                      "out": g["out"][r0:r1]}
                d2h = [(torch.empty_like(dv["out"], device="cpu").pin_memory(), dv["out"])]
                mx = max(c.q_lens[b0:b1])
                fns = [lambda dv=dv, g=g: pa.pa_kv_append(g["pool"], dv["k_new"], dv["v_new"], dv["slots"]),
                       lambda dv=dv, g=g, c=c, mx=mx: pa.pa_prefill_chunked(g["pool"], dv["q"], dv["cu"], dv["bt"],
                                                                           dv["sl"], c.scale, mx, dv["out"])]
                self.pieces.append((h2d, d2h, fns, w))
        self.h2d_bytes = sum(h.numel() * h.element_size() for pc in self.pieces for h, _ in pc[0])
        self.d2h_bytes = sum(h.numel() * h.element_size() for pc in self.pieces for h, _ in pc[1])
        # the prefill groups' calls on high-priority streams: the copies of their large output
        # wait for them, so their CTAs take SMs ahead of the decodes' as SMs free up
        lo, hi = torch.cuda.Stream.priority_range()
        self.s_in = torch.cuda.Stream(device=self.dev)
        self.s_comp = [torch.cuda.Stream(device=self.dev, priority=hi if label == "chunked_prefill" else 0)
                       for _, _, _, label in self.pieces]
        self.s_out = [torch.cuda.Stream(device=self.dev) for _ in self.pieces]

    def run(self):
        main = torch.cuda.current_stream(self.dev)
        self.s_in.wait_stream(main)
        ready = []
        with torch.cuda.stream(self.s_in):
            for h2d, _, _, _ in self.pieces:
                for h, dv in h2d:
                    dv.copy_(h, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(self.s_in)
                ready.append(ev)
        done = []
        for (_, _, fns, _), ev, sc in zip(self.pieces, ready, self.s_comp):
            sc.wait_event(ev)
            with torch.cuda.stream(sc):
                for fn in fns:
                    fn()
            ev2 = torch.cuda.Event()
            ev2.record(sc)
            done.append(ev2)
        for (_, d2h, _, _), ev2, so in zip(self.pieces, done, self.s_out):
            so.wait_event(ev2)
            with torch.cuda.stream(so):
                for h, dv in d2h:
                    h.copy_(dv, non_blocking=True)
            main.wait_stream(so)

    def outputs(self):
        """Host copies of every workload's output after an e2e step: {workload: tensor}, the
        prefill groups joined in sequence order."""
        outs = {}
        for _, d2h, _, label in self.pieces:
            outs.setdefault(label, []).extend(h for h, _ in d2h)
        return {k: torch.cat(v) for k, v in outs.items()}


# ----------------------------------------------------------------------------- timing
def flush_l2(buf):
    # reading a buffer larger than L2 leaves it full of clean lines of that buffer
    return buf.sum()


def capture_graph(fn, dev):
    """fn's launches as one CUDA graph (captured on a side stream after one eager run)."""
    st = torch.cuda.Stream(device=dev)
    st.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        fn()
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(graph, stream=st):
            fn()
    torch.cuda.current_stream(dev).wait_stream(st)
    torch.cuda.synchronize(dev)
    return graph


def time_graph(graph, reps, flush_buf):
    """Device time (us) of `reps` replays, each after an L2 flush that stays outside the
    interval; the interval includes the graph's launch latency."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for s, e in ev:
        flush_l2(flush_buf)
        s.record()
        graph.replay()
        e.record()
    torch.cuda.synchronize()
    return np.array([s.elapsed_time(e) * 1e3 for s, e in ev])


def _external_events():
    """Timing events that become event-record nodes when captured in a CUDA graph, or None."""
    try:
        return (torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True))
    except TypeError:
        return None


def time_in_graph(fn, reps, flush_buf, dev):
    """Device time (us) of fn with a cold L2, `reps` times: one graph of [L2 flush, event, fn,
    event] is replayed, and the interval between its two event nodes is fn's device time,
    without the graph's launch latency.  None where events cannot be graph nodes."""
    evs = _external_events()
    if evs is None:
        return None
    s, e = evs
    st = torch.cuda.Stream(device=dev)
    st.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        fn()
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(graph, stream=st):
            flush_l2(flush_buf)
            s.record(st)
            fn()
            e.record(st)
    torch.cuda.current_stream(dev).wait_stream(st)
    torch.cuda.synchronize(dev)
    out = []
    try:
        for i in range(reps + 2):
            graph.replay()
            torch.cuda.synchronize(dev)
            if i >= 2:
                out.append(s.elapsed_time(e) * 1e3)
    except RuntimeError as err:  # the events did not become timing nodes of the graph
        log(f"[bench] in-graph event timing unavailable ({err}); timing calls with their launch")
        return None
    finally:
        del graph
    return np.array(out)


def stats(us):
    us = np.asarray(us, dtype=np.float64)
    return {"median": round(float(np.median(us)), 2), "p10": round(float(np.percentile(us, 10)), 2),
            "p90": round(float(np.percentile(us, 90)), 2), "mean": round(float(us.mean()), 2)}


def time_step(step, workloads, steps, warmup, flush_buf, dev, serial=False):
    """The step over `workloads`, replayed as one CUDA graph (as a serving loop replays its
    step): `steps` timed replays after `warmup` untimed ones, L2 flushed before each."""
    graph = capture_graph((lambda: step.run(workloads)) if serial else (lambda: step.run_parallel(workloads)), dev)
    for _ in range(warmup):
        flush_l2(flush_buf)
        graph.replay()
    torch.cuda.synchronize()
    us = time_graph(graph, steps, flush_buf)
    del graph
    return us


def time_calls(step, steps, flush_buf, dev):
    """Every call unit of the step on its own, L2 cold: (marginal, isolated) device times (us).
    isolated: the unit alone after an L2 flush, between event nodes of one graph (it carries
    the unit's launch latency, about 5 us on this harness even for an empty kernel).
    marginal: what one more launch of the unit costs in a stream -- the same graph with the
    unit run a second time on the second, untouched copy of its inputs, minus the isolated
    graph; the second launch's start overlaps the first one's tail, as in a serving loop."""
    res = {}
    for c, c2 in zip(step.calls, step.calls_alt or step.calls):
        one = time_in_graph(c.fn, steps, flush_buf, dev)
        if one is None:  # no event nodes in graphs: whole-replay timing
            g1 = capture_graph(c.fn, dev)
            time_graph(g1, 2, flush_buf)
            one = time_graph(g1, steps, flush_buf)
            del g1
            res[c.name] = (one, one)
            continue
        if step.calls_alt is None:
            res[c.name] = (one, one)
            continue
        two = time_in_graph(lambda: (c.fn(), c2.fn()), steps, flush_buf, dev)
        res[c.name] = (two - np.median(one), one)
    return res


def time_e2e(step, workloads, steps, flush_buf):
    """End-to-end step time (us) through the public API: the e2e step (uploads, calls,
    downloads) replayed as one CUDA graph, the copies on every replay.  Also the same step
    issued eagerly from Python (host-bound).  Returns (graph us, eager us, E2E)."""
    e2e = E2E(step, workloads)
    torch.cuda.synchronize()
    for _ in range(2):  # warm the copies
        e2e.run()
    torch.cuda.synchronize()
    eager = []
    for _ in range(steps):
        flush_l2(flush_buf)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        e2e.run()
        e.record()
        e.synchronize()
        eager.append(s.elapsed_time(e) * 1e3)
    graph = capture_graph(e2e.run, step.dev)
    time_graph(graph, 2, flush_buf)
    replay = time_graph(graph, steps, flush_buf)
    torch.cuda.synchronize()
    # The pipelined pieces must give the very bits of the step's calls.  Poison every output
    # first (so that a row the pieces fail to write cannot pass on an earlier step's value),
    # replay the e2e step once, then run the step's calls (one prefill launch) on the same
    # inputs and compare every workload's output; the device status must stay clean.
    import paged_kv_gqa_slot_gb300 as pa
    pa.pa_device_status(clear=True)
    for w in e2e.workloads:
        step.by_name[w][0]["out"].fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    got = {k: v.clone() for k, v in e2e.outputs().items()}
    del graph
    step.run(e2e.workloads)
    torch.cuda.synchronize()
    status = pa.pa_device_status(clear=True)
    if status:
        raise RuntimeError(f"device status {status:#x} after the e2e step")
    for w in e2e.workloads:
        if not torch.equal(got[w], step.by_name[w][0]["out"].cpu()):
            raise RuntimeError(f"e2e output of {w} differs from the step's")
    return replay, np.array(eager), e2e


def hbm_fracs(gbs, peaks):
    return {"frac_hbm": round(gbs / peaks["hbm_gbs"], 3), "frac_hbm_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 3)}


def latency_configs(flush_buf, peaks, reps=30):
    """The latency-bound decode shapes: cold (L2 flushed; in-graph event interval, and with the
    launch) and CUDA-graph-warm (100 back-to-back calls in one graph)."""
    import paged_kv_gqa_slot_gb300 as pa
    import workloads as W
    res = {}
    dev = torch.device("cuda", torch.cuda.current_device())
    for name, make in (("tiny_decode[1x37,4q/1kv/64]", W.tiny_decode),
                       ("qwen3_4b_decode[1x1152,32q/8kv/128]", W.qwen3_4b_decode)):
        c = make()
        k, v = c.k_cache.cuda(), c.v_cache.cuda()
        pool = pa.PaPool(k, v)
        q, bt, sl = c.q.cuda(), c.block_tables.cuda(), c.seq_lens.cuda()
        out = torch.empty_like(q)
        fn = lambda: pa.pa_decode(pool, q, bt, sl, c.scale, out)
        for _ in range(5):
            fn()
        cold = time_in_graph(fn, reps, flush_buf, dev)
        g1 = capture_graph(fn, dev)
        cold_launch = time_graph(g1, reps, flush_buf)
        del g1
        if cold is None:
            cold = cold_launch
        # warm: 100 calls replayed from one CUDA graph
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(st):
            fn()
            torch.cuda.synchronize()
            with torch.cuda.graph(graph, stream=st):
                for _ in range(100):
                    fn()
        torch.cuda.current_stream().wait_stream(st)
        graph.replay()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(5):
            graph.replay()
        e.record()
        e.synchronize()
        warm = s.elapsed_time(e) * 1e3 / 500
        del graph
        kvb = attn_bytes(c)
        gbs = kvb / float(np.median(cold)) / 1e3
        res[name] = {"us_cold": stats(cold), "us_cold_launch": stats(cold_launch),
                     "us_per_call_graph_warm": round(warm, 2), "bytes": int(kvb), "kv_gbs_cold": round(gbs, 1),
                     **hbm_fracs(gbs, peaks), "hbm_floor_us": round(kvb / peaks["hbm_gbs"] / 1e3, 3),
                     "decode_splits": pa.pa_decode_num_splits(c.batch, c.num_kv_heads, c.max_blocks)}
    # multi-query decode: 64 sequences x 4 draft tokens (a speculative-decoding verify)
    c = W.spec_verify()
    k, v = c.k_cache.cuda(), c.v_cache.cuda()
    pool = pa.PaPool(k, v)
    pa.pa_kv_append(pool, c.k_new.cuda(), c.v_new.cuda(), c.slot_mapping.cuda())
    q, bt, sl, cu = c.q.cuda(), c.block_tables.cuda(), c.seq_lens.cuda(), c.cu_q_lens.cuda()
    out = torch.empty_like(q)
    fn = lambda: pa.pa_prefill_chunked(pool, q, cu, bt, sl, c.scale, 4, out)
    fn()
    torch.cuda.synchronize()
    us = time_in_graph(fn, 20, flush_buf, dev)
    if us is None:
        us = time_graph(capture_graph(fn, dev), 20, flush_buf)
    gbs = attn_bytes(c) / float(np.median(us)) / 1e3
    res["spec_verify[64x~1088,C=4,32q/8kv/128]"] = {"us": stats(us), "kv_gbs": round(gbs, 1), **hbm_fracs(gbs, peaks)}
    return res


# ----------------------------------------------------------------------------- CPU oracle baseline
class OracleSample:
    """A bounded sample of the decode step for the fp64 CPU oracle: the append + decode of the
    first `decode_seqs` batched-decode sequences and both split-KV workloads with their merge;
    with `prefill_stride`, also the chunked prefill on every prefill_stride-th (token, head)
    row (the full-path sample).  `parts` are the split-KV partition counts of the two
    workloads: the step's own, or 16 for both (the library's count for these shapes on 152
    SMs) where no GPU is there to ask."""

    def __init__(self, decode_seqs=None, prefill_stride=None, parts=(16, 16)):
        import oracle
        import workloads as W
        from workloads import u16
        self.orc = oracle.load()
        self.u16 = u16
        self.parts = tuple(int(p) for p in parts)
        self.c3 = W.batched_decode()
        if decode_seqs is not None:
            self.c3 = self._first_seqs(self.c3, decode_seqs)
        self.c4a = W.splitkv_decode(1004, 4, 8192)
        self.c4b = W.splitkv_decode(1004, 1, 32768)
        self.kv_bytes = unique_kv_bytes(self.c3) + unique_kv_bytes(self.c4a) + unique_kv_bytes(self.c4b)
        self.c5 = None
        self.prefill_frac = 0.0
        if prefill_stride:
            self.c5 = W.chunked_prefill()
            T, H = self.c5.q.shape[0], self.c5.num_heads
            idx = np.arange(0, T * H, prefill_stride)
            self.rows_t = (idx // H).astype(np.int32)
            self.rows_h = (idx % H).astype(np.int32)
            self.prefill_frac = len(idx) / (T * H)
            self.kv_bytes += unique_kv_bytes(self.c5) * self.prefill_frac
        self.pools = {}
        for name, c in (("c3", self.c3), ("c4a", self.c4a), ("c4b", self.c4b), ("c5", self.c5)):
            if c is not None:
                self.pools[name] = (u16(c.k_cache).copy(), u16(c.v_cache).copy())

    @staticmethod
    def _first_seqs(c, n):
        """The first n sequences of a decode case (one appended token per sequence)."""
        import workloads as W
        return W.PagedCase(**{**c.__dict__, "q": c.q[:n], "block_tables": c.block_tables[:n],
                              "seq_lens": c.seq_lens[:n], "q_lens": c.q_lens[:n], "cu_q_lens": c.cu_q_lens[:n + 1],
                              "k_new": c.k_new[:n], "v_new": c.v_new[:n], "slot_mapping": c.slot_mapping[:n],
                              "k_seq": c.k_seq[:n], "v_seq": c.v_seq[:n]})

    def run(self):
        o, u16 = self.orc, self.u16
        k, v = self.pools["c3"]
        c = self.c3
        o.kv_append(k, v, u16(c.k_new), u16(c.v_new), c.slot_mapping.numpy())
        o.decode(k, v, u16(c.q), c.block_tables.numpy(), c.seq_lens.numpy(), c.scale)
        for name, c, P in (("c4a", self.c4a, self.parts[0]), ("c4b", self.c4b, self.parts[1])):
            k, v = self.pools[name]
            op, lse = o.decode_partitions(k, v, u16(c.q), c.block_tables.numpy(), c.seq_lens.numpy(), c.scale, P)
            o.combine(op, lse)
        if self.c5 is not None:
            k, v = self.pools["c5"]
            c = self.c5
            o.kv_append(k, v, u16(c.k_new), u16(c.v_new), c.slot_mapping.numpy())
            o.prefill_rows(k, v, u16(c.q), c.cu_q_lens.numpy(), c.block_tables.numpy(), c.seq_lens.numpy(), c.scale,
                           self.rows_t, self.rows_h)

    def describe(self) -> str:
        s = (f"append + decode of {self.c3.batch} batched-decode sequences, split-KV 4x8192 (P={self.parts[0]}) and "
             f"1x32768 (P={self.parts[1]}) with their merge")
        if self.c5 is not None:
            s += f", append + chunked prefill on {self.prefill_frac:.4f} of its (token, head) rows"
        return s + f"; {self.kv_bytes / 1e6:.1f} MB of KV"

    def time(self, threads, reps=1):
        """(GB/s, seconds per sample, threads used) on `threads` host threads."""
        used = self.orc.set_threads(threads)
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            self.run()
            ts.append(time.perf_counter() - t0)
        dt = float(np.mean(ts))
        return self.kv_bytes / dt / 1e9, dt, used


# ----------------------------------------------------------------------------- main
def max_over_ranks(x: float, device) -> float:
    """The largest x over all ranks (the job is as slow as its slowest replica)."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value_gbs(step_kv_bytes: int, world_size: int, step_us: float) -> float:
    """Whole-job throughput: every replica reads its own step's KV bytes in step_us."""
    return world_size * step_kv_bytes / step_us / 1e3


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def base_config(serial=False):
    form = ("its calls one after another on one stream" if serial else
            "its workloads (independent requests on separate pools) as parallel branches")
    return {"workload": WORKLOAD, "l2": "flushed before every timed step (512 MB buffer read)",
            "timing": f"CUDA events around each replay of the step captured as one CUDA graph, {form}; "
                      "per-call times from event nodes inside one graph per call, around the call"}


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    sample = OracleSample(decode_seqs=16)
    threads = os.cpu_count() or 1
    for _ in range(args.warmup):
        sample.time(threads)
    ts = []
    used = 1
    for _ in range(args.steps):
        _, dt, used = sample.time(threads)
        ts.append(dt)
    mean_s = float(np.mean(ts))
    value = sample.kv_bytes / mean_s / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_s * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {**base_config(), "l2": "not applicable (host CPU)",
                       "timing": f"host wall clock (time.perf_counter) around each oracle step, {used} threads"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
                             "sample": sample.describe(), "host_cpu_count": os.cpu_count()},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def call_entry(call, kern_us, launch_us, peaks, peak_src):
    """Per-call record: marginal device time in a stream (median, p10, p90), the isolated
    time with its launch latency, and the achieved rate against the peaks."""
    st = stats(kern_us)
    med = st["median"]
    e = {"launches": len(call.fns), "us": st, "us_isolated": stats(launch_us)}
    if call.unit_kind == "bytes":
        gbs = call.units / med / 1e3
        e.update({"bytes": int(call.units), "GB/s": round(gbs, 1), **hbm_fracs(gbs, peaks)})
    else:
        tf = call.units / med / 1e6
        e.update({"flops": int(call.units), "TFLOP/s": round(tf, 1), "frac_bf16": round(tf / peaks["bf16_tflops"], 3)})
    return e


def roofline_of(call, kern_us, peaks, peak_src):
    med = float(np.median(kern_us))
    traffic = profiled_traffic(call.kind, call.workload)
    if call.unit_kind == "bytes":
        ach = call.units / med / 1e3
        return {"kernel": call.name, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 3),
                "frac_nominal_8tbs": round(ach / NOMINAL_HBM_GBS, 3), "traffic": traffic,
                "algorithmic_bytes_per_launch": int(call.units), "us": round(med, 2),
                "peak_source": f"{peak_src} (HBM copy)"}
    ach = call.units / med / 1e6
    return {"kernel": call.name, "bound": "tensor", "achieved": round(ach, 1), "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 3), "traffic": traffic,
            "algorithmic_flops_per_launch": int(call.units), "us": round(med, 2),
            "peak_source": f"{peak_src} (bf16 burst)"}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--serial-step", action="store_true",
                    help="headline the calls one after another on one stream instead of the parallel branches")
    ap.add_argument("--only", choices=sorted(Step.GROUPS),
                    help="time only this part of the step (for profiling); skips the extras")
    args = ap.parse_args(argv)
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    assert args.warmup >= 3, "at least 3 warm-up steps"

    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_gqa_slot_gb300 as pa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks, peak_src = load_peaks()
    step = Step(dev, args.only, copies=2)
    extras = args.only is None
    headline = tuple(w for w in DECODE_WORKLOADS if w in step.available) or step.available
    full = step.available
    flush_buf = torch.ones(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    pa.pa_device_status(clear=True)

    # clocks are sampled over a sustained stretch of steps and the timed steps
    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    sampler.start()
    t_end = time.time() + (1.5 if extras else 0.0)
    while time.time() < t_end:
        flush_l2(flush_buf)
        step.run_parallel(full)
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    step_us = time_step(step, headline, args.steps, args.warmup, flush_buf, dev, args.serial_step)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    wall = time.time() - wall0
    other_us = time_step(step, headline, args.steps, 2, flush_buf, dev, not args.serial_step)
    full_us = time_step(step, full, args.steps, 2, flush_buf, dev, args.serial_step) if full != headline else None
    calls_t = time_calls(step, args.steps, flush_buf, dev)
    clocks = sampler.stop()
    status = pa.pa_device_status(clear=True)
    if status:
        raise RuntimeError(f"device status {status:#x} after the timed steps")

    mean_step_us = max_over_ranks(float(step_us.mean()), dev)
    kv_head = step.kv_bytes(headline)
    value = job_value_gbs(kv_head, ws, mean_step_us)  # GB/s

    calls = {c.name: call_entry(c, *calls_t[c.name], peaks, peak_src) for c in step.calls}
    head_calls = step.calls_of(headline)
    dom = max(head_calls, key=lambda c: float(np.median(calls_t[c.name][0])))
    roof = roofline_of(dom, calls_t[dom.name][0], peaks, peak_src)
    rooflines = {c.name: roofline_of(c, calls_t[c.name][0], peaks, peak_src) for c in step.calls}
    tot = sum(float(np.median(calls_t[c.name][0])) for c in step.calls)
    for c in step.calls:
        calls[c.name]["share_of_serial_sum"] = round(float(np.median(calls_t[c.name][0])) / tot, 3)

    # end to end through the public API with host buffers
    e2e, full_e2e, lat = None, None, {}
    if extras:
        n_e2e = max(5, min(args.steps, 20))
        rep, eager, ee = time_e2e(step, headline, n_e2e, flush_buf)
        e2e = {"value": round(kv_head / float(rep.mean()) / 1e3, 1), "unit": "GB/s",
               "h2d_bytes_per_step": int(ee.h2d_bytes), "d2h_bytes_per_step": int(ee.d2h_bytes),
               "us_per_step": stats(rep), "timing": "the e2e step replayed as one CUDA graph",
               "eager_value": round(kv_head / float(eager.mean()) / 1e3, 1)}
        if full != headline:
            rep_f, eager_f, ef = time_e2e(step, full, n_e2e, flush_buf)
            kv_full = step.kv_bytes(full)
            full_e2e = {"value": round(kv_full / float(rep_f.mean()) / 1e3, 1), "unit": "GB/s",
                        "h2d_bytes_per_step": int(ef.h2d_bytes), "d2h_bytes_per_step": int(ef.d2h_bytes),
                        "us_per_step": stats(rep_f), "eager_value": round(kv_full / float(eager_f.mean()) / 1e3, 1)}
        lat = latency_configs(flush_buf, peaks) if rank == 0 else {}

    cpu = None
    if rank == 0 and ws == 1 and extras and not args.no_cpu_baseline:
        sample = OracleSample(decode_seqs=16, parts=(step.P4a, step.P4b))
        v1, dt1, _ = sample.time(1)
        vall, dtall, used = sample.time(os.cpu_count() or 1, reps=3)
        cpu = {"value": round(vall, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
               "single_thread_value": round(v1, 4), "host_cpu_count": os.cpu_count(),
               "sample": sample.describe() + f"; {dt1:.1f}s on 1 thread, {dtall:.2f}s on {used} threads "
                                             "(OpenMP over (sequence, head) rows)"}

    if rank == 0:
        full_step = None
        if full_us is not None:
            kv_full = step.kv_bytes(full)
            full_step = {"workload": FULL_WORKLOAD, "us": stats(full_us), "kv_bytes": int(kv_full),
                         "kv_gbs": round(kv_full / float(full_us.mean()) / 1e3, 1), "e2e": full_e2e}
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(mean_step_us / 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": (base_config(args.serial_step) if extras else
                       {**base_config(args.serial_step), "workload": f"only {args.only}"}),
            "step_kv_bytes": int(kv_head), "step_us": stats(step_us),
            "frac_hbm": round(value / ws / peaks["hbm_gbs"], 3),
            "frac_hbm_nominal_8tbs": round(value / ws / NOMINAL_HBM_GBS, 3),
            ("step_parallel_us" if args.serial_step else "step_serial_us"): stats(other_us),
            "full_step": full_step, "roofline": roof, "rooflines": rooflines, "per_call": calls, "latency": lat,
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": step.launches(headline) * args.steps, "clocks": clocks,
            "wall_s_timed": round(wall, 3),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
