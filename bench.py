#!/usr/bin/env python3
"""Benchmark of the paged GQA attention hot path (libpagedattn) on GB300.

One step = one pass of every call of the hot path over its workload, inputs resident
in HBM:
  1-2. pa_append_decode  append of 64 new tokens fused with the batched decode (64 seqs,
                         ctx ~U[1024,1152], 32q/8kv/128): pa_kv_append + pa_decode in one launch
  3. pa_decode_splitkv   4 x 8192, P in 8..32 + pa_combine   (Qwen3-32B-shaped 64q/8kv/128)
  4. pa_decode_splitkv   1 x 32768, P in 8..32 + pa_combine
  5. pa_kv_append        8 x 256 chunk tokens     (chunked prefill over a shared 768-token prefix)
  6. pa_prefill_chunked  8 x 256-token causal chunks, 32q/8kv/128
The workloads are independent requests on separate pools, so the step runs each on a stream
of its own (the prefill chain first, then the decodes), forked from and joined back into one
stream; it is captured once as a CUDA graph with those parallel branches and replayed, as a
serving loop replays its step.  The same calls one after another on one stream are timed too
("step_serial_us").  value = KV bytes the attention calls must read per step / step time (GB/s),
L2 flushed (a 512 MB buffer is read) before every timed replay, outside the timed interval.
Each call is also captured and timed on its own and reported under "per_call".  The
end-to-end number ("e2e") runs the step through the public API with host buffers, the
copies inside the timed interval: each workload's inputs are staged in one pinned host
buffer; they are copied up on a copy stream, piece by piece (each decode workload whole,
then the chunked prefill in two groups of sequences); each piece's calls run on a compute
stream of their own once its inputs have arrived, and its output is copied back on a copy
stream of its own as soon as it is done, while later pieces still go up or compute.  That
e2e step is captured as one CUDA graph (copies included) and replayed, as a serving loop
replays its step; "eager_value" issues the same step from Python call by call (host-bound).
The e2e outputs are checked bit for bit against the step's.  The two latency-bound decode
shapes (1 seq x 37 tokens, 4q/1kv/64; 1 seq x 1152 tokens, 32q/8kv/128) are reported
under "latency" (cold and CUDA-graph-replayed).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--serial-step]

--serial-step makes the serial step the headline value (the parallel one is then reported as
"step_parallel_us").

--impl reference times the CPU fp64 oracle (the reference arm of this comparison) on a
bounded sample of the same step.  Under torchrun (N > 1) every rank runs the full step on
its own GPU (independent replicas, weak scaling); rank 0 prints one JSON line.
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
WORKLOAD = ("serving step: fused append(64)+decode 64x~1088 (32q/8kv/128) + split-KV 4x8192 and 1x32768 (P in 8..32) "
            "with combine (64q/8kv/128) + append(2048) + chunked prefill 8x256 over a shared 768-token "
            "prefix (32q/8kv/128); block 16; bf16 N(0,1)")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {
    "decode": ["pa_decode.cu", "pa_block_attn.cuh", "pa_device.cuh"],
    "splitkv": ["pa_decode.cu", "pa_block_attn.cuh", "pa_device.cuh"],
    "prefill": ["pa_prefill.cu", "pa_prefill_tc.cu", "pa_block_attn.cuh", "pa_device.cuh"],
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


def source_sha(kind: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        h.update((ROOT / "paged_kv_gqa_slot_gb300" / "csrc" / f).read_bytes())
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


# ----------------------------------------------------------------------------- workload
def causal_flops(case) -> float:
    """QK^T and PV multiply-adds of the chunked prefill, causal-exact (2 flops each)."""
    keys = 0
    for L, C in zip(case.seq_lens.tolist(), case.q_lens):
        pre = L - C
        keys += C * pre + C * (C + 1) // 2
    return float(keys) * case.num_heads * case.head_dim * 4


def attn_bytes(case, extra_q_out=True) -> int:
    """Algorithmic bytes of one attention call: K and V once per kv head, plus q and out."""
    b = case.kv_bytes()
    if extra_q_out:
        b += 2 * case.q.numel() * 2
    return b


class Step:
    """Device-resident inputs of one step and the calls that make it."""

    GROUPS = {"decode": ("c3",), "splitkv": ("c4a", "c4b"), "prefill": ("c5",), "tiny_decode": ("c1",),
              "qwen3_4b_decode": ("c2",)}

    def __init__(self, device, only=None):
        import paged_kv_gqa_slot_gb300 as pa
        import workloads as W
        self.pa = pa
        groups = set(self.GROUPS[only]) if only else {"c3", "c4a", "c4b", "c5"}
        t0 = time.time()
        self.c1 = W.tiny_decode() if "c1" in groups else None
        self.c2 = W.qwen3_4b_decode() if "c2" in groups else None
        self.c3 = W.batched_decode() if "c3" in groups else None
        self.c4a = W.splitkv_decode(1004, 4, 8192) if "c4a" in groups else None
        self.c4b = W.splitkv_decode(1004, 1, 32768) if "c4b" in groups else None
        self.c5 = W.chunked_prefill() if "c5" in groups else None
        log(f"[bench] workloads drawn in {time.time() - t0:.1f}s")
        self.dev = device
        d = device

        def up(c):
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
                for i, (b0, b1) in enumerate(self.prefill_groups(c)):
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
            return g

        self.g1, self.g2 = up(self.c1), up(self.c2)
        self.g3, self.g4a, self.g4b, self.g5 = up(self.c3), up(self.c4a), up(self.c4b), up(self.c5)
        # partitions as the library suggests, kept within the workload's 8..32
        self.P4a = min(32, max(8, pa.pa_splitkv_num_partitions(4, 8, 512))) if self.c4a is not None else 8
        self.P4b = min(32, max(8, pa.pa_splitkv_num_partitions(1, 8, 2048))) if self.c4b is not None else 32
        for g, c, P in ((self.g4a, self.c4a, self.P4a), (self.g4b, self.c4b, self.P4b)):
            if g is None:
                continue
            g["ws_o"] = torch.empty((c.batch, c.num_heads, P, c.head_dim), dtype=torch.float32, device=d)
            g["ws_lse"] = torch.empty((c.batch, c.num_heads, P), dtype=torch.float32, device=d)
        c3, c4a, c4b, c5 = self.c3, self.c4a, self.c4b, self.c5
        g3, g4a, g4b, g5 = self.g3, self.g4a, self.g4b, self.g5
        app_bytes = lambda c: 2 * 2 * c.k_new.numel() * 2  # read new rows, write pool rows, K and V
        ws_bytes = lambda g: g["ws_o"].numel() * 4 + g["ws_lse"].numel() * 4 + g["out"].numel() * 2
        # (name, kind, fn, units, unit_kind)
        self.calls = []
        for g, c, nm in ((self.g1, self.c1, "decode[tiny,1x37,4q/1kv/64]"),
                         (self.g2, self.c2, "decode[qwen3_4b,1x1152,32q/8kv/128]")):
            if g is not None:
                self.calls.append((nm, "decode", (lambda g=g, c=c: pa.pa_decode(g["pool"], g["q"], g["bt"], g["sl"],
                                                                               c.scale, g["out"])),
                                   attn_bytes(c), "bytes"))
        if g3 is not None:
            # the decode step's append and attention in one launch (pa_append_decode)
            self.calls += [
                ("append_decode[batched_decode,64x~1088]", "decode",
                 lambda: pa.pa_append_decode(g3["pool"], g3["k_new"], g3["v_new"], g3["slots"], g3["q"], g3["bt"],
                                             g3["sl"], c3.scale, g3["out"]),
                 attn_bytes(c3) + app_bytes(c3), "bytes")]
        if g4a is not None:
            self.calls += [
                (f"decode_splitkv[4x8192,P={self.P4a}]", "splitkv",
                 lambda: pa.pa_decode_splitkv(g4a["pool"], g4a["q"], g4a["bt"], g4a["sl"], c4a.scale, self.P4a,
                                              g4a["ws_o"], g4a["ws_lse"]), attn_bytes(c4a), "bytes"),
                (f"combine[4x8192,P={self.P4a}]", "combine", lambda: pa.pa_combine(g4a["ws_o"], g4a["ws_lse"], g4a["out"]),
                 ws_bytes(g4a), "bytes")]
        if g4b is not None:
            self.calls += [
                (f"decode_splitkv[1x32768,P={self.P4b}]", "splitkv",
                 lambda: pa.pa_decode_splitkv(g4b["pool"], g4b["q"], g4b["bt"], g4b["sl"], c4b.scale, self.P4b,
                                              g4b["ws_o"], g4b["ws_lse"]), attn_bytes(c4b), "bytes"),
                (f"combine[1x32768,P={self.P4b}]", "combine", lambda: pa.pa_combine(g4b["ws_o"], g4b["ws_lse"], g4b["out"]),
                 ws_bytes(g4b), "bytes")]
        if g5 is not None:
            mx5 = max(c5.q_lens)
            self.calls += [
                ("kv_append[chunked_prefill,2048]", "append",
                 lambda: pa.pa_kv_append(g5["pool"], g5["k_new"], g5["v_new"], g5["slots"]), app_bytes(c5), "bytes"),
                ("prefill_chunked[8x256 over 768]", "prefill",
                 lambda: pa.pa_prefill_chunked(g5["pool"], g5["q"], g5["cu"], g5["bt"], g5["sl"], c5.scale, mx5,
                                               g5["out"]), causal_flops(c5), "flops")]
        # the step's metric: KV bytes the attention calls must read
        cases = ((self.g1, self.c1), (self.g2, self.c2), (g3, c3), (g4a, c4a), (g4b, c4b), (g5, c5))
        self.step_kv_bytes = sum(c.kv_bytes() for _, c in cases if c is not None)
        self.cases = [(g, c) for g, c in cases if c is not None]
        # parallel branches: one per workload, the longest chain (append + prefill) first
        order = ["chunked_prefill", "batched_decode", "splitkv_4x8192", "splitkv_1x32768", "qwen3_4b_decode",
                 "tiny_decode"]
        self.branches = []
        for label in order:
            idx = [i for i, (name, _, _, _, _) in enumerate(self.calls) if call_workload(name) == label]
            if idx:
                self.branches.append(idx)
        assert sorted(i for b in self.branches for i in b) == list(range(len(self.calls)))
        self.branch_streams = [torch.cuda.Stream(device=d) for _ in self.branches]

    def run(self, events=None):
        """The calls one after another on the current stream."""
        for i, (_, _, fn, _, _) in enumerate(self.calls):
            fn()
            if events is not None:
                events[i + 1].record()

    def run_parallel(self):
        """Every workload on a stream of its own, forked from the current stream and joined
        back into it: the workloads are independent requests on separate pools, and one
        workload's latency-bound stretches (a kernel's start, its last wave) leave SMs and
        HBM bandwidth that another's calls can use."""
        main = torch.cuda.current_stream(self.dev)
        for st in self.branch_streams:
            st.wait_stream(main)
        for st, idx in zip(self.branch_streams, self.branches):
            with torch.cuda.stream(st):
                for i in idx:
                    self.calls[i][2]()
        for st in self.branch_streams:
            main.wait_stream(st)

    # ---- end-to-end: inputs from pinned host memory, outputs back to pinned host memory
    # groups of prefill sequences in the e2e pipeline (1, 2, 3 and 4 measured; 2 and 3 best)
    E2E_PREFILL_GROUPS = 2

    def prefill_groups(self, c):
        """The e2e pipeline's groups of prefill sequences: [(b0, b1), ...]."""
        n = max(1, min(self.E2E_PREFILL_GROUPS, c.batch))
        edges = [c.batch * i // n for i in range(n + 1)]
        return [(b0, b1) for b0, b1 in zip(edges[:-1], edges[1:]) if b1 > b0]

    def e2e_setup(self):
        """The step's pieces, in upload order: each decode workload whole (its inputs in one
        copy), then the chunked prefill in groups of sequences (the first group also brings
        the workload's small tables; each group its rows of new K, new V and q, three
        copies).  A piece is its host-to-device copies, its device-to-host copies and its
        calls.  A prefill group is an append and a prefill over its own sequences (views of
        the workload's tensors, cu_q_lens rebased to 0): the same per-sequence arithmetic as
        the one-launch prefill, so the same bits."""
        pa = self.pa
        self.e2e_pieces = []
        for g, c in self.cases:
            if c is self.c5:
                continue
            d2h = [(torch.empty_like(g["out"], device="cpu").pin_memory(), g["out"])]
            fns = [fn for (name, _, fn, _, _) in self.calls if call_workload(name) == c.name]
            self.e2e_pieces.append(([(g["in_host"], g["in_dev"])], d2h, fns, c.name))
        if self.c5 is not None:
            g, c = self.g5, self.c5
            assert c.k_new.shape[0] == sum(c.q_lens), "prefill workload: one appended row per chunk query"
            cu = c.cu_q_lens.tolist()
            lay, hb, db = g["in_layout"], g["in_host"], g["in_dev"]
            row = c.k_new[0].numel() * 2  # bytes of one new K (or V) row
            qrow = c.q[0].numel() * 2
            for i, (b0, b1) in enumerate(self.prefill_groups(c)):
                r0, r1 = cu[b0], cu[b1]
                h2d = [(hb[lay["bt"]:lay["k_new"]], db[lay["bt"]:lay["k_new"]])] if i == 0 else []
                for key, rb in (("k_new", row), ("v_new", row), ("q", qrow)):
                    h2d.append((hb[lay[key] + r0 * rb:lay[key] + r1 * rb], db[lay[key] + r0 * rb:lay[key] + r1 * rb]))
                dv = {"q": g["q"][r0:r1], "k_new": g["k_new"][r0:r1], "v_new": g["v_new"][r0:r1],
                      "slots": g["slots"][r0:r1], "bt": g["bt"][b0:b1], "sl": g["sl"][b0:b1], "cu": g[f"cu{i}"],
                      "out": g["out"][r0:r1]}
                d2h = [(torch.empty_like(dv["out"], device="cpu").pin_memory(), dv["out"])]
                mx = max(c.q_lens[b0:b1])
                fns = [lambda dv=dv: pa.pa_kv_append(g["pool"], dv["k_new"], dv["v_new"], dv["slots"]),
                       lambda dv=dv, mx=mx: pa.pa_prefill_chunked(g["pool"], dv["q"], dv["cu"], dv["bt"], dv["sl"],
                                                                 c.scale, mx, dv["out"])]
                self.e2e_pieces.append((h2d, d2h, fns, c.name))
        self.h2d_bytes = sum(h.numel() * h.element_size() for pc in self.e2e_pieces for h, _ in pc[0])
        self.d2h_bytes = sum(h.numel() * h.element_size() for pc in self.e2e_pieces for h, _ in pc[1])
        # the prefill groups' calls on high-priority streams: the copies of their large output
        # wait for them, so their CTAs take SMs ahead of the decodes' as SMs free up
        lo, hi = torch.cuda.Stream.priority_range()
        self.s_in = torch.cuda.Stream(device=self.dev)
        self.s_comp = [torch.cuda.Stream(device=self.dev, priority=hi if label == "chunked_prefill" else 0)
                       for _, _, _, label in self.e2e_pieces]
        self.s_out = [torch.cuda.Stream(device=self.dev) for _ in self.e2e_pieces]

    def e2e_run(self):
        """One step as a serving loop runs it: every piece's inputs go up on one copy stream as
        early as possible, its calls run on a compute stream of its own once they have
        arrived, and its output comes back on another copy stream as soon as its last call is
        done (one copy stream per piece, so that none waits behind another's output), while
        later pieces are still going up or computing."""
        main = torch.cuda.current_stream(self.dev)
        self.s_in.wait_stream(main)
        ready = []
        with torch.cuda.stream(self.s_in):
            for h2d, _, _, _ in self.e2e_pieces:
                for h, dv in h2d:
                    dv.copy_(h, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(self.s_in)
                ready.append(ev)
        done = []
        for (_, _, fns, _), ev, sc in zip(self.e2e_pieces, ready, self.s_comp):
            sc.wait_event(ev)
            with torch.cuda.stream(sc):
                for fn in fns:
                    fn()
            ev2 = torch.cuda.Event()
            ev2.record(sc)
            done.append(ev2)
        for (_, d2h, _, _), ev2, so in zip(self.e2e_pieces, done, self.s_out):
            so.wait_event(ev2)
            with torch.cuda.stream(so):
                for h, dv in d2h:
                    h.copy_(dv, non_blocking=True)
            main.wait_stream(so)

    def e2e_outputs(self):
        """Host copies of every workload's output after an e2e step: {workload: tensor}, the
        prefill groups joined in sequence order."""
        outs = {}
        for _, d2h, _, label in self.e2e_pieces:
            outs.setdefault(label, []).extend(h for h, _ in d2h)
        return {k: torch.cat(v) for k, v in outs.items()}


def call_workload(name: str) -> str:
    """Workload label of a call, as used by the traffic lines of the profile summaries."""
    for key, label in (("tiny", "tiny_decode"), ("qwen3_4b", "qwen3_4b_decode"), ("batched", "batched_decode"),
                       ("4x8192", "splitkv_4x8192"), ("1x32768", "splitkv_1x32768"), ("chunked", "chunked_prefill"),
                       ("8x256", "chunked_prefill")):
        if key in name:
            return label
    return "unknown"


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
    """Device time of `reps` replays, each after an L2 flush that stays outside the interval."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for s, e in ev:
        flush_l2(flush_buf)
        s.record()
        graph.replay()
        e.record()
    torch.cuda.synchronize()
    return np.array([s.elapsed_time(e) * 1e3 for s, e in ev])  # us


def time_steps(step, steps, warmup, flush_buf, dev, serial=False):
    """The step is replayed as one CUDA graph (as a serving loop replays its step): `steps`
    timed replays after `warmup` untimed ones, with the workloads as parallel branches (or
    the calls one after another: `serial`).  The other form is timed the same way and
    returned as `other_us`.  Per-call times come from one graph per call, timed the same
    way."""
    graph = capture_graph(step.run if serial else step.run_parallel, dev)
    for _ in range(warmup):
        flush_l2(flush_buf)
        graph.replay()
    torch.cuda.synchronize()
    step_us = time_graph(graph, steps, flush_buf)
    other = capture_graph(step.run_parallel if serial else step.run, dev)
    time_graph(other, 2, flush_buf)
    other_us = time_graph(other, steps, flush_buf)
    del other
    per_call = np.zeros((steps, len(step.calls)))
    for i, (_, _, fn, _, _) in enumerate(step.calls):
        g1 = capture_graph(fn, dev)
        time_graph(g1, 2, flush_buf)
        per_call[:, i] = time_graph(g1, steps, flush_buf)
        del g1
    del graph
    return step_us, other_us, per_call


def time_e2e(step, steps, flush_buf):
    """End-to-end step time (us): the e2e step (uploads, calls, downloads) replayed as one
    CUDA graph, as a serving loop replays its step with inputs staged in fixed pinned
    buffers; the copies run on every replay.  Also the same step issued eagerly from Python
    (host-bound: every copy and call is a few microseconds of host work)."""
    step.e2e_setup()
    torch.cuda.synchronize()
    for _ in range(2):  # warm the copies
        step.e2e_run()
    torch.cuda.synchronize()
    eager = []
    for _ in range(steps):
        flush_l2(flush_buf)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        step.e2e_run()
        e.record()
        e.synchronize()
        eager.append(s.elapsed_time(e) * 1e3)
    graph = capture_graph(step.e2e_run, step.dev)
    time_graph(graph, 2, flush_buf)
    replay = time_graph(graph, steps, flush_buf)
    torch.cuda.synchronize()
    # The pipelined pieces must give the very bits of the step's calls.  Poison every output
    # first (so that a row the pieces fail to write cannot pass on an earlier step's value),
    # replay the e2e step once, then run the step's calls (one prefill launch) on the same
    # inputs and compare every workload's output; the device status must stay clean.
    import paged_kv_gqa_slot_gb300 as pa
    pa.pa_device_status(clear=True)
    for g, _ in step.cases:
        g["out"].fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    got = {k: v.clone() for k, v in step.e2e_outputs().items()}
    del graph
    step.run()
    torch.cuda.synchronize()
    status = pa.pa_device_status(clear=True)
    if status:
        raise RuntimeError(f"device status {status:#x} after the e2e step")
    for g, c in step.cases:
        if not torch.equal(got[c.name], g["out"].cpu()):
            raise RuntimeError(f"e2e output of {c.name} differs from the step's")
    return float(np.mean(replay)), float(np.mean(eager))


def latency_configs(flush_buf):
    import paged_kv_gqa_slot_gb300 as pa
    import workloads as W
    res = {}
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
        cold = []
        for _ in range(30):
            flush_l2(flush_buf)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            fn()
            e.record()
            e.synchronize()
            cold.append(s.elapsed_time(e) * 1e3)
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
        kvb = attn_bytes(c)
        res[name] = {"us_per_call_cold": round(float(np.median(cold)), 2), "us_per_call_graph_warm": round(warm, 2),
                     "kv_gbs_cold": round(kvb / float(np.median(cold)) / 1e3, 1),
                     "decode_splits": pa.pa_decode_num_splits(c.batch, c.num_kv_heads, c.max_blocks)}
        del graph
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
    us = float(np.median(time_graph(capture_graph(fn, q.device), 20, flush_buf)))
    res["spec_verify[64x~1088,C=4,32q/8kv/128]"] = {"us_per_call": round(us, 2),
                                                   "kv_gbs": round(c.kv_bytes() / us / 1e3, 1)}
    return res


# ----------------------------------------------------------------------------- CPU oracle baseline
class OracleSample:
    """A bounded sample of the step for the fp64 CPU oracle: the decode and split-KV calls
    whole, the chunked prefill on every `prefill_stride`-th (token, head) row."""

    def __init__(self, prefill_stride=16, decode_seqs=None):
        import oracle
        import workloads as W
        from workloads import u16
        self.orc = oracle.load()
        self.u16 = u16
        self.c3 = W.batched_decode()
        if decode_seqs is not None:
            self.c3 = self._first_seqs(self.c3, decode_seqs)
        self.c4a = W.splitkv_decode(1004, 4, 8192)
        self.c4b = W.splitkv_decode(1004, 1, 32768)
        self.c5 = W.chunked_prefill()
        T, H = self.c5.q.shape[0], self.c5.num_heads
        idx = np.arange(0, T * H, prefill_stride)
        self.rows_t = (idx // H).astype(np.int32)
        self.rows_h = (idx % H).astype(np.int32)
        self.prefill_frac = len(idx) / (T * H)
        self.kv_bytes = (self.c3.kv_bytes() + self.c4a.kv_bytes() + self.c4b.kv_bytes()
                         + self.c5.kv_bytes() * self.prefill_frac)
        self.pools = {}
        for name, c in (("c3", self.c3), ("c4a", self.c4a), ("c4b", self.c4b), ("c5", self.c5)):
            k, v = u16(c.k_cache).copy(), u16(c.v_cache).copy()
            self.pools[name] = (k, v)

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
        for name, c, P in (("c4a", self.c4a, 8), ("c4b", self.c4b, 32)):
            k, v = self.pools[name]
            op, lse = o.decode_partitions(k, v, u16(c.q), c.block_tables.numpy(), c.seq_lens.numpy(), c.scale, P)
            o.combine(op, lse)
        k, v = self.pools["c5"]
        c = self.c5
        o.kv_append(k, v, u16(c.k_new), u16(c.v_new), c.slot_mapping.numpy())
        o.prefill_rows(k, v, u16(c.q), c.cu_q_lens.numpy(), c.block_tables.numpy(), c.seq_lens.numpy(), c.scale,
                       self.rows_t, self.rows_h)


def describe_sample(s: OracleSample) -> str:
    return (f"append + decode of {s.c3.batch} batched-decode sequences, split-KV 4x8192 (P=8) and 1x32768 (P=32) "
            f"with combine, append + chunked prefill on {s.prefill_frac:.4f} of its (token, head) rows; "
            f"{s.kv_bytes / 1e6:.1f} MB of KV-equivalent work")


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
                      "per-call times from one graph per call, timed the same way"}


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    sample = OracleSample(prefill_stride=64, decode_seqs=16)
    for _ in range(args.warmup):
        sample.run()
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        sample.run()
        ts.append(time.perf_counter() - t0)
    mean_s = float(np.mean(ts))
    value = sample.kv_bytes / mean_s / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_s * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {**base_config(), "l2": "not applicable (host CPU)",
                       "timing": "host wall clock (time.perf_counter) around each oracle step, one thread"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": describe_sample(sample)},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


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
    step = Step(dev, args.only)
    extras = args.only is None
    flush_buf = torch.ones(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    pa.pa_device_status(clear=True)

    # clocks are sampled over a sustained stretch of steps and the timed steps
    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    sampler.start()
    t_end = time.time() + (1.5 if extras else 0.0)
    while time.time() < t_end:
        flush_l2(flush_buf)
        (step.run if args.serial_step else step.run_parallel)()
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    step_us, other_us, per_call = time_steps(step, args.steps, args.warmup, flush_buf, dev, args.serial_step)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    wall = time.time() - wall0
    clocks = sampler.stop()
    status = pa.pa_device_status(clear=True)
    if status:
        raise RuntimeError(f"device status {status:#x} after the timed steps")

    mean_step_us = max_over_ranks(float(step_us.mean()), dev)
    value = job_value_gbs(step.step_kv_bytes, ws, mean_step_us)  # GB/s

    # per call
    calls = {}
    means = per_call.mean(axis=0)
    for (name, kind, _, units, ukind), us in zip(step.calls, means):
        if ukind == "bytes":
            ach = units / us / 1e3
            calls[name] = {"us": round(float(us), 2), "GB/s": round(ach, 1),
                           "frac_hbm": round(ach / peaks["hbm_gbs"], 3), "share": round(float(us) / means.sum(), 3)}
        else:
            ach = units / us / 1e6
            calls[name] = {"us": round(float(us), 2), "TFLOP/s": round(ach, 1),
                           "frac_bf16": round(ach / peaks["bf16_tflops"], 3), "share": round(float(us) / means.sum(), 3)}
    # dominant kernel of the step
    di = int(np.argmax(means))
    dname, dkind, _, dunits, dukind = step.calls[di]
    wl = call_workload(dname)
    if dukind == "bytes":
        ach = dunits / means[di] / 1e3
        roof = {"kernel": dname, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 3), "traffic": profiled_traffic(dkind, wl),
                "algorithmic_bytes_per_launch": int(dunits), "peak_source": peak_src}
    else:
        ach = dunits / means[di] / 1e6
        roof = {"kernel": dname, "bound": "tensor", "achieved": round(ach, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 3), "traffic": profiled_traffic(dkind, wl),
                "algorithmic_flops_per_launch": int(dunits), "peak_source": peak_src}

    # end to end through the public API with host buffers
    e2e, lat = None, {}
    if extras:
        e2e_us, eager_us = time_e2e(step, max(5, min(args.steps, 20)), flush_buf)
        e2e = {"value": round(step.step_kv_bytes / e2e_us / 1e3, 1), "unit": "GB/s",
               "h2d_bytes_per_step": int(step.h2d_bytes), "d2h_bytes_per_step": int(step.d2h_bytes),
               "us_per_step": round(e2e_us, 1), "timing": "the e2e step replayed as one CUDA graph",
               "eager_value": round(step.step_kv_bytes / eager_us / 1e3, 1)}
        lat = latency_configs(flush_buf) if rank == 0 else {}

    cpu = None
    if rank == 0 and ws == 1 and extras and not args.no_cpu_baseline:
        sample = OracleSample(prefill_stride=4)
        t0 = time.perf_counter()
        sample.run()
        dt = time.perf_counter() - t0
        cpu = {"value": round(sample.kv_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": describe_sample(sample) + f"; {dt:.1f}s single-threaded on the host"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(mean_step_us / 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": (base_config(args.serial_step) if extras else
                       {**base_config(args.serial_step), "workload": f"only {args.only}"}),
            "step_kv_bytes": int(step.step_kv_bytes),
            ("step_parallel_us" if args.serial_step else "step_serial_us"): round(float(other_us.mean()), 2),
            "roofline": roof, "per_call": calls, "latency": lat, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": len(step.calls) * args.steps, "clocks": clocks,
            "wall_s_timed": round(wall, 3),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
