"""Benchmark of the compressed-KV decode hot path (one JSON line on stdout).

Metric: decode-attention layer-steps/s, with the achieved HBM bandwidth of the
dominant kernel against the measured copy bandwidth of this GPU.

A step is one decode step of one layer for the whole batch on a synthetic
workload (see compressed_kv_sparse_append_gb300/workloads.py):
  * CSA workloads (default: csa_128k = batch 8, 131072-token context, 32768
    compressed entries, 128 heads, 64 indexer heads, top-512, mixed
    FP8-nope/BF16-rope main KV, FP4 indexer keys): kv_append_quant_multi of
    the step's new compressed entry and indexer key (one launch for both
    planes), csa_index_topk, csa_sparse_attn;
  * hca_1m: kv_append_quant + hca_attn;
  * csa2_group: one csa2_group_decode call (six layer-steps).
Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream, with a 1 GiB L2 flush (outside the events) before
every step; barrier + max over ranks when launched with torchrun (each rank
runs its own replica: batch sharding needs no collective).
"""

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

METRIC = "decode attn layer-steps/s at 128k/1M ctx; achieved HBM GB/s vs ~8 TB/s peak"
UNIT = "layer-steps/s"
ALL_SOURCES = ["append.cu", "indexer.cu", "indexer_umma.cu", "attention.cu", "api.cu",
               "common.cuh", "select.cuh", "topk_merge.cuh", "indexer.cuh", "attention.cuh",
               "tmap.cuh", "hadamard.cuh"]
# The sources that decide each library call's kernels and their DRAM traffic
# (the kernel code, the headers it includes, the host code that sizes the
# launch).  Keyed by the call's tag in a step's call list.
_ATTN = ["attention.cu", "attention.cuh", "common.cuh", "tmap.cuh", "api.cu"]
KERNEL_SOURCES = {
    "csa_index_topk": ["indexer_umma.cu", "indexer.cu", "topk_merge.cuh", "select.cuh",
                       "indexer.cuh", "common.cuh", "tmap.cuh", "hadamard.cuh", "api.cu"],
    "csa_sparse_attn": _ATTN,
    "hca_attn": _ATTN,
    "kv_append_quant": ["append.cu", "common.cuh", "hadamard.cuh", "api.cu"],
}
TRAFFIC_MD = os.path.join(ROOT, "profiles", "traffic.md")


def _strip_comments(text):
    """C/C++ source without comments and with whitespace runs collapsed, so
    that a comment-only edit leaves a source key unchanged."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_key(tag=None):
    """16 hex digits of SHA-256 over the comment-stripped sources of a call's
    kernels (all sources for an unknown tag).  A traffic figure is valid
    only while its row's key equals this."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(tag, ALL_SOURCES):
        path = os.path.join(ROOT, "compressed_kv_sparse_append_gb300", "csrc", f)
        if os.path.exists(path):
            with open(path, encoding="utf-8") as fh:
                h.update(f.encode() + b"\0" + _strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def _traffic_rows():
    rows = []
    if os.path.exists(TRAFFIC_MD):
        for line in open(TRAFFIC_MD, encoding="utf-8"):
            parts = [p.strip() for p in line.strip().strip("|").split("|")]
            if len(parts) >= 4 and ":" in parts[0] and not parts[0].startswith("-"):
                rows.append(parts)
    return rows


def profiled_traffic(tag, workload):
    """Per-launch DRAM bytes of call `tag` on `workload` from the committed
    table, if it was captured on the current sources (else None)."""
    cur = source_key(tag)
    for parts in _traffic_rows():
        if parts[0] == "%s:%s" % (tag, workload) and parts[1] == cur:
            try:
                return float(parts[2])
            except ValueError:
                return None
    return None


def record_traffic(csv_path, tag, workload, scale=1.0, note=""):
    """Reads an `ncu --csv --page raw --metrics dram__bytes_read.sum,
    dram__bytes_write.sum` log, averages read + write bytes over its launches
    (every captured launch must be of the call's kernels), multiplies by
    `scale` (units processed by a full launch / by a captured one, for a
    capture on a smaller case) and writes the row of `tag:workload` in
    profiles/traffic.md under the current source key."""
    import csv
    unit_mult = {"byte": 1.0, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9,
                 "kibyte": 1024.0, "mibyte": 1024.0 ** 2, "gibyte": 1024.0 ** 3}
    with open(csv_path, encoding="utf-8", errors="replace") as f:
        lines = [l for l in f if l.startswith('"')]
    rows = list(csv.reader(lines))
    head = rows[0]
    ir, iw = head.index("dram__bytes_read.sum"), head.index("dram__bytes_write.sum")
    units = rows[1]
    per = []
    for r in rows[2:]:
        if len(r) <= max(ir, iw):
            continue
        v = float(r[ir].replace(",", "")) * unit_mult[units[ir].lower()] + \
            float(r[iw].replace(",", "")) * unit_mult[units[iw].lower()]
        per.append(v)
    if not per:
        raise SystemExit("no launches in %s" % csv_path)
    value = statistics.mean(per) * scale
    key = "%s:%s" % (tag, workload)
    new_row = "| %s | %s | %.0f | %s |" % (key, source_key(tag), value,
                                          note or "%d launch(es), scale %g" % (len(per), scale))
    text = open(TRAFFIC_MD, encoding="utf-8").read() if os.path.exists(TRAFFIC_MD) else ""
    out, done = [], False
    for line in text.splitlines():
        parts = [p.strip() for p in line.strip().strip("|").split("|")]
        if parts and parts[0] == key:
            out.append(new_row)
            done = True
        else:
            out.append(line)
    if not done:
        out.append(new_row)
    with open(TRAFFIC_MD, "w", encoding="utf-8") as f:
        f.write("\n".join(out) + "\n")
    print(new_row)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="csa_128k")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="timed oracle work of the cpu_baseline sample")
    p.add_argument("--ref-seconds", type=float, default=60.0,
                   help="--impl reference: timed oracle work of the whole run (split over its steps)")
    p.add_argument("--record-traffic", metavar="NCU_CSV",
                   help="write the DRAM traffic row of --call on --workload into profiles/traffic.md "
                        "from an ncu raw CSV log, and exit")
    p.add_argument("--call", default="csa_index_topk", help="call tag for --record-traffic")
    p.add_argument("--traffic-scale", type=float, default=1.0,
                   help="full-launch units / captured-launch units (--record-traffic)")
    p.add_argument("--traffic-note", default="")
    p.add_argument("--no-sub", dest="sub", action="store_false",
                   help="time only --workload (by default the 1M-context CSA and HCA workloads are "
                        "timed too and reported under 'sub')")
    return p.parse_args()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is None:
            self.result = None
            return False
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        self.result = None if not sm else {
            "sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
            "samples": len(sm)}
        return False


# ------------------------------------------------------------------ setup --

def setup_csa(wl, dev, ckv, wlmod):
    """Cache planes of a CSA layer, filled through kv_append_quant."""
    import torch
    B, n = wl.B, wl.n_comp
    cap = n + 8                     # room for the step's appended entry
    kv = ckv.Plane(wl.main_fmt, 512, B, cap, dev, nope_block=wl.nope_block)
    win = ckv.Plane(wl.main_fmt, 512, B, wl.W, dev, nope_block=wl.nope_block)
    keys = ckv.Plane(wl.idx_fmt, 128, B, cap, dev)
    ws = ckv.new_workspace(256, dev)
    for b in range(B):
        kvr, kr, wr = wlmod.sequence_rows(wl, b, n, dev)
        base = torch.arange(n, dtype=torch.int64, device=dev) + b * cap
        ckv.kv_append_quant(kv, kvr, base, ws=ws)
        ckv.kv_append_quant(keys, kr, base, ws=ws)
        ckv.kv_append_quant(win, wr, torch.arange(wl.W, dtype=torch.int64, device=dev) + b * wl.W, ws=ws)
        if wl.ties:
            # ~5 % exact ties crowded at the top-k boundary: rank this
            # sequence's entries with the kernel's own scores, copy donors
            q, qi, w = wlmod.step_queries(wl, 0, dev, batch=[b])
            dbg = torch.zeros((1, n), device=dev)
            one = ckv.Plane(wl.idx_fmt, 128, 1, cap, dev, data=keys.data[b:b + 1], scale=keys.scale[b:b + 1])
            ckv.csa_index_topk(one, torch.tensor([n], dtype=torch.int32, device=dev), n, qi, w, wl.topk,
                               dbg_scores=dbg)
            order = torch.argsort(dbg[0], descending=True, stable=True).cpu()
            kr2 = wlmod.inject_ties(kr, order, seed=wl.seed + b)
            ckv.kv_append_quant(keys, kr2, base, ws=ws)
        del kvr, kr, wr
    torch.cuda.synchronize()
    assert ckv.read_device_status(ws) == 0
    return kv, win, keys, cap


def packed(tensors, dev):
    """The same tensors as views of one device buffer (256-byte aligned
    offsets), so that a step's inputs or outputs move in one copy."""
    import torch
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(total, dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(tensors, offs):
        v = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return buf, views


class Step:
    """One decode step of a workload: ``run(marks)`` enqueues the step's
    library calls in order; with ``marks`` (len(calls) + 1 CUDA events) it
    records an event before every call and one after the last.  ``calls``
    lists (tag, algorithmic bytes per launch) in call order; ``launches``
    counts the kernels one step launches; ``layers`` its layer-steps."""

    def __init__(self, run, calls, launches, layers, host, ws):
        self.run, self.calls, self.launches, self.layers = run, calls, launches, layers
        self.host, self.ws = host, ws

    @property
    def step_bytes(self):
        return sum(b for _, b in self.calls)


def _marked(marks, i):
    if marks is not None:
        marks[i].record()


def make_step(wl, dev, ckv, wlmod):
    import torch
    B = wl.B
    n = wl.n_comp
    tau = wl.tau
    n_comp = torch.full((B,), n, dtype=torch.int32, device=dev)
    win_len = torch.full((B,), wl.W, dtype=torch.int32, device=dev)
    q, qi, w = wlmod.step_queries(wl, 0, dev)
    main_row = {"bf16": 1024, "mixed": 576 + 4 * (448 // wl.nope_block), "fp4": 288}[wl.main_fmt]
    if wl.kind == "csa":
        kv, win, keys, cap = setup_csa(wl, dev, ckv, wlmod)
        new_kv = wlmod.append_rows(wl, B, 512, 0, dev)
        new_key = wlmod.append_rows(wl, B, 128, 1, dev)
        in_buf, (q, qi, w, new_kv, new_key) = packed((q, qi, w, new_kv, new_key), dev)
        slot = torch.arange(B, dtype=torch.int64, device=dev) * cap + n
        idx = torch.empty((B, wl.topk), dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        lse = torch.empty((B, wl.H), device=dev)
        ws = ckv.new_workspace(max(ckv.workspace_bytes(ckv.OP_INDEX_TOPK, B, wl.H, wl.HI, n, wl.topk, 0),
                                   ckv.workspace_bytes(ckv.OP_SPARSE_ATTN, B)), dev)
        ent = {"bf16": 256, "fp4": 72}[wl.idx_fmt]
        key_row = {"bf16": 256, "fp4": 72}[wl.idx_fmt]
        calls = [
            ("kv_append_quant", B * (1024 + main_row) + B * (256 + key_row)),
            ("csa_index_topk", B * n * ent + qi.numel() * 2 + w.numel() * 4 + idx.numel() * 4),
            ("csa_sparse_attn", B * (wl.topk + wl.W) * main_row + idx.numel() * 4
             + q.numel() * 2 + out.numel() * 2 + lse.numel() * 4),
        ]

        def run(marks=None):
            # the new main-KV and indexer-key rows, one launch for both planes
            _marked(marks, 0)
            ckv.kv_append_quant_multi([kv, keys], [new_kv, new_key], [slot, slot], ws=ws)
            _marked(marks, 1)
            ckv.csa_index_topk(keys, n_comp, n, qi, w, wl.topk, out_idx=idx, ws=ws)
            _marked(marks, 2)
            ckv.csa_sparse_attn(kv, win, win_len, idx, q, tau, out=out, lse=lse, ws=ws)
            _marked(marks, 3)
            return out

        return Step(run, calls, 3, 1, {"inputs": in_buf, "outputs": out}, ws)
    if wl.kind == "hca":
        cap = n + 8
        kv = ckv.Plane("bf16", 512, B, cap, dev)
        win = ckv.Plane("bf16", 512, B, wl.W, dev)
        ws = ckv.new_workspace(ckv.workspace_bytes(ckv.OP_HCA_ATTN, B), dev)
        for b in range(B):
            kvr, _, wr = wlmod.sequence_rows(wl, b, n, dev)
            ckv.kv_append_quant(kv, kvr, torch.arange(n, dtype=torch.int64, device=dev) + b * cap, ws=ws)
            ckv.kv_append_quant(win, wr, torch.arange(wl.W, dtype=torch.int64, device=dev) + b * wl.W, ws=ws)
        new_kv = wlmod.append_rows(wl, B, 512, 0, dev)
        in_buf, (q, new_kv) = packed((q, new_kv), dev)
        slot = torch.arange(B, dtype=torch.int64, device=dev) * cap + n
        out = torch.empty_like(q)
        lse = torch.empty((B, wl.H), device=dev)
        calls = [
            ("kv_append_quant", B * (1024 + 1024)),
            ("hca_attn", B * (n + wl.W) * 1024 + q.numel() * 2 + out.numel() * 2 + lse.numel() * 4),
        ]

        def run(marks=None):
            _marked(marks, 0)
            ckv.kv_append_quant(kv, new_kv, slot, ws=ws)
            _marked(marks, 1)
            ckv.hca_attn(kv, n_comp, n, win, win_len, q, tau, out=out, lse=lse, ws=ws)
            _marked(marks, 2)
            return out

        return Step(run, calls, 2, 1, {"inputs": in_buf, "outputs": out}, ws)
    # csa2 group
    L = wl.n_layers
    cap = n + 16
    keys = ckv.Plane("fp4", 128, B, cap, dev)
    kvs = [ckv.Plane("fp4", 512, B, cap, dev) for _ in range(L)]
    wins = [ckv.Plane("fp4", 512, B, wl.W, dev) for _ in range(L)]
    ws0 = ckv.new_workspace(256, dev)
    for l in range(L):
        for b in range(B):
            kvr, kr, wr = wlmod.sequence_rows(wl, b, n, dev, layer=l)
            base = torch.arange(n, dtype=torch.int64, device=dev) + b * cap
            ckv.kv_append_quant(kvs[l], kvr, base, ws=ws0)
            ckv.kv_append_quant(wins[l], wr, torch.arange(wl.W, dtype=torch.int64, device=dev) + b * wl.W, ws=ws0)
            if l == 0:
                ckv.kv_append_quant(keys, kr, base, ws=ws0)
    qs, qis, ws_ = [], [], []
    for l in range(L):
        ql, qil, wl_ = wlmod.step_queries(wl, 0, dev, layer=l)
        qs.append(ql)
        qis.append(qil if l < 2 else None)
        ws_.append(wl_ if l < 2 else None)
    app = wlmod.append_rows(wl, wl.n_append, 512, 0, dev)
    # the step's inputs in one buffer, its L outputs in another
    in_buf, views = packed(qs + qis[:2] + ws_[:2] + [app], dev)
    qs, qis[:2], ws_[:2], app = views[:L], views[L:L + 2], views[L + 2:L + 4], views[L + 4]
    out_buf, outs = packed([torch.empty_like(qs[0]) for _ in range(L)], dev)
    roles = [ckv.CSA2_FULL, ckv.CSA2_REINDEX] + [ckv.CSA2_REUSE] * (L - 2)
    g = ckv.make_group(roles, [0, 0] + list(range(2, L)), [0, 0] + [0] * (L - 2), kvs, wins, keys, qs,
                       qis, ws_, outs, pool_len=wl.pool_len)
    per = wl.n_append // B
    app_slot = (torch.arange(B, device=dev)[:, None] * cap + n + torch.arange(per, device=dev)[None]).flatten().to(torch.int64)
    ws = ckv.new_workspace(ckv.workspace_bytes(ckv.OP_CSA2, B, wl.H, wl.HI, n, wl.topk, wl.pool_len), dev)
    calls = [("csa2_group_decode",
              B * n * 72 + B * wl.pool_len * 72 + L * B * (wl.topk + wl.W) * 288
              + L * 2 * qs[0].numel() * 2 + wl.n_append * (1024 + 288))]

    def run(marks=None):
        _marked(marks, 0)
        ckv.csa2_group_decode(g, n_comp, n, win_len, B, wl.H, wl.HI, wl.topk, tau, append_dst=kvs[0],
                              append_src=app, append_slot=app_slot, ws=ws)
        _marked(marks, 1)
        return outs[0]

    # launches: append + Full index + Reindex index + the attention, four
    # layers at most per launch
    return Step(run, calls, 3 + (L + 3) // 4, L, {"inputs": in_buf, "outputs": out_buf}, ws)


# ------------------------------------------------------------------ timing --

FLUSH_BYTES = 1 << 30   # > L2 (129 MB); ~150 us of GPU time that also hides host enqueue


def time_steps(step, K, W, dev):
    """K steps, each after an L2 flush.  The flush keeps the GPU busy while
    the host enqueues the step's launches, so the events bracket device time
    only; the host enqueue time is returned for checking that assumption.
    The step's kernels are launched with programmatic dependent launch, and
    events between them would serialise them: the step times come from a
    pass with events around whole steps only, each call's launch duration
    from a second pass with events between the calls."""
    import torch
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(W):
        flush.zero_()
        step.run()
    torch.cuda.synchronize()
    new_ev = lambda: torch.cuda.Event(enable_timing=True)
    ev = [(new_ev(), new_ev()) for _ in range(K)]
    marks = [[new_ev() for _ in range(len(step.calls) + 1)] for _ in range(K)]
    fl = [(new_ev(), new_ev()) for _ in range(K)]
    host_us = []
    for i in range(K):
        fl[i][0].record()
        flush.zero_()
        fl[i][1].record()
        t0 = time.perf_counter()
        ev[i][0].record()
        step.run()
        ev[i][1].record()
        host_us.append((time.perf_counter() - t0) * 1e6)
    for i in range(K):
        flush.zero_()
        step.run(marks[i])
    torch.cuda.synchronize()
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    call_ms = [[m[c].elapsed_time(m[c + 1]) for m in marks] for c in range(len(step.calls))]
    flush_us = [f[0].elapsed_time(f[1]) * 1000.0 for f in fl]
    return step_ms, call_ms, statistics.median(host_us), statistics.median(flush_us)


def time_e2e(step, K, W, dev):
    """Same steps through the public API, with every step's inputs (queries,
    indexer queries, head weights, new rows) copied from pinned host memory
    into the device tensors the step reads, and the outputs copied back to
    pinned host memory, inside the timed region.  The step's inputs are views
    of one device buffer and its outputs of another, so each direction is a
    single copy."""
    import torch
    d_in, d_out = step.host["inputs"], step.host["outputs"]
    h_in = d_in.cpu().pin_memory()
    h_out = torch.empty(d_out.shape, dtype=d_out.dtype).pin_memory()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def one():
        d_in.copy_(h_in, non_blocking=True)
        step.run()
        h_out.copy_(d_out, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(W):
        flush.zero_()
        one()
    tot = 0.0
    for _ in range(K):
        flush.zero_()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        one()
        e1.record()
        torch.cuda.synchronize()
        tot += e0.elapsed_time(e1)
    bi = h_in.numel() * h_in.element_size()
    bo = h_out.numel() * h_out.element_size()
    return tot / K, bi, bo


# ------------------------------------------------------------ CPU oracle --

def cpu_oracle_sample(wl, budget_s, max_seqs=2):
    """Times the oracle (as it stands) on a bounded sample of the workload:
    layer-steps of up to ``max_seqs`` sequences, generated on the host with
    the same recipe and repeated until ``budget_s`` seconds of timed work.
    Each sequence's cache (main KV, window, indexer keys) is quantised before
    the timer starts, as a decode step finds it resident; the timed work is
    the step's own: the append of its new entries, the indexer query, scores
    and top-k, and the attention.  Returns (layer-steps/s, cores, sample
    description, seconds)."""
    import numpy as np
    from compressed_kv_sparse_append_gb300 import workloads as wlmod
    from oracle import attention as oa, fp_formats as ff, indexer as oi, csa2 as oc

    f = lambda t: t.float().numpy()
    n = wl.n_comp
    L = wl.n_layers

    def prepare(b):
        kv, keys, win = wlmod.sequence_rows(wl, b, n, "cpu")
        q, qi, w = wlmod.step_queries(wl, 0, "cpu", batch=[b])
        kvf, winf = f(kv), f(win)
        c = {"q": f(q[0])}
        if wl.kind == "hca":
            c["new"] = [(f(wlmod.append_rows(wl, 1, 512, 0, "cpu")), "bf16")]
            c["kv"] = ff.quantize_entries(kvf, "bf16")
            c["win"] = ff.quantize_entries(winf, "bf16")
        elif wl.kind == "csa":
            c["new"] = [(f(wlmod.append_rows(wl, 1, 512, 0, "cpu")), wl.main_fmt),
                        (f(wlmod.append_rows(wl, 1, 128, 1, "cpu")), wl.idx_fmt)]
            c["kv"] = ff.quantize_entries(kvf, wl.main_fmt, wl.nope_block)
            c["win"] = ff.quantize_entries(winf, wl.main_fmt, wl.nope_block)
            c["keys"] = ff.quantize_entries(f(keys), wl.idx_fmt)
            c["qi"], c["w"] = f(qi[0]), f(w[0]).astype(np.float64)
        else:
            c["new"] = [(f(wlmod.append_rows(wl, max(1, wl.n_append // wl.B), 512, 0, "cpu")), "fp4")]
            c["kv"] = ff.fp4_quantize(kvf)
            c["win"] = ff.fp4_quantize(winf)
            c["keys"] = ff.fp4_quantize(f(keys))
            c["qi"], c["w"] = f(qi[0]), f(w[0]).astype(np.float64)
        return c

    def step(c):
        for rows, fmt in c["new"]:                    # the step's append
            ff.quantize_entries(rows, fmt, wl.nope_block)
        kd, ks = c["kv"]
        wd, wsc = c["win"]
        if wl.kind == "hca":
            oa.hca_attention(c["q"], kd, ks, "bf16", n, wd, wsc, wl.W, wl.tau)
        elif wl.kind == "csa":
            kvals = ff.dequantize_entries(c["keys"][0], c["keys"][1], wl.idx_fmt)
            qv = oi.indexer_query(c["qi"], wl.idx_fmt == "fp4")
            idx = oi.topk_set(oi.index_scores(qv, c["w"], kvals), wl.topk)
            oa.csa_sparse_attention(c["q"], kd, ks, wl.main_fmt, idx, wd, wsc, wl.W, wl.tau,
                                    nope_block=wl.nope_block)
        else:
            kvals = ff.fp4_dequantize(*c["keys"])
            roles = [oc.FULL, oc.REINDEX] + [oc.REUSE] * (L - 2)
            oc.csa2_group_sequence(roles, [0] * L, [0] * L, kvals, n, [c["qi"]] * L, [c["w"]] * L, True,
                                   wl.topk, wl.pool_len, [c["q"]] * L, [(kd, ks, "fp4")] * L,
                                   [(wd, wsc)] * L, wl.W, wl.tau)

    cache = [prepare(b) for b in range(min(max_seqs, wl.B))]
    t_total, steps = 0.0, 0
    while t_total < budget_s or steps == 0:
        c = cache[steps % len(cache)]
        t0 = time.perf_counter()
        step(c)
        t_total += time.perf_counter() - t0
        steps += 1
    layers = L if wl.kind == "csa2" else 1
    per_layer_step = t_total / steps * wl.B / layers   # whole batch, one layer
    desc = ("%d sequence-step(s) (cycling over %d of the batch's %d sequences) of %s, cache quantised "
            "before the timer, oracle float64 NumPy, %.1f s timed" % (steps, len(cache), wl.B, wl.name,
                                                                      t_total))
    return 1.0 / per_layer_step, os.cpu_count(), desc, t_total


# ------------------------------------------------------------------- main --

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, None
    import torch.distributed as dist
    dist.init_process_group("gloo")
    return dist.get_rank(), ws, dist


def max_over_ranks(x, dist):
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, wl, rank, world, dist):
    if rank != 0:
        return
    budget = max(0.5, args.ref_seconds / max(1, args.steps + args.warmup))
    vals = []
    for i in range(args.warmup + args.steps):
        v, cores, desc, secs = cpu_oracle_sample(wl, budget)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def workload_config(wl):
    return {"workload": wl.name, "kind": wl.kind, "batch": wl.B, "context_tokens": wl.T,
            "compressed_entries": wl.n_comp, "heads": wl.H, "indexer_heads": wl.HI, "topk": wl.topk,
            "window": wl.W, "main_kv": wl.main_fmt, "indexer_keys": wl.idx_fmt or None,
            "fp8_scale_block": wl.nope_block if wl.main_fmt == "mixed" else None,
            "layers_per_step": wl.n_layers, "l2": "flushed (1 GiB write) before every step"}


def measure(wl, args, dev, local, ckv, wlmod, dist, world, e2e=True):
    """Times one workload; returns its record (the JSON line's fields)."""
    import torch
    step = make_step(wl, dev, ckv, wlmod)
    if dist:
        dist.barrier()
    with ClockSampler(local) as clk:
        step_ms, call_ms, host_us, flush_us = time_steps(step, args.steps, args.warmup, dev)
    status = ckv.read_device_status(step.ws)
    if status != 0:
        raise RuntimeError("device status %d after the timed steps of %s" % (status, wl.name))
    total_ms = max_over_ranks(sum(step_ms), dist)
    ms_per_step = total_ms / args.steps
    value = world * step.layers * args.steps / (total_ms / 1000.0)
    peak, peak_kind = measured_peaks()
    per_call = {}
    for (tag, nbytes), ms in zip(step.calls, call_ms):
        avg_ms = max_over_ranks(statistics.mean(ms), dist)
        per_call[tag] = {"avg_launch_us": avg_ms * 1000.0, "algorithmic_bytes": nbytes,
                         "achieved_gbs": nbytes / (avg_ms / 1000.0) / 1e9,
                         "frac": nbytes / (avg_ms / 1000.0) / 1e9 / peak}
    dom_tag = max(per_call, key=lambda t: per_call[t]["avg_launch_us"])
    dom = per_call[dom_tag]
    rec = {"value": value, "ms_per_step": ms_per_step,
           "roofline": {"bound": "hbm", "kernel": dom_tag, "achieved": dom["achieved_gbs"], "peak": peak,
                        "peak_kind": peak_kind, "unit": "GB/s", "frac": dom["frac"],
                        "traffic": profiled_traffic(dom_tag, wl.name),
                        "algorithmic_bytes": dom["algorithmic_bytes"],
                        "avg_launch_us": dom["avg_launch_us"]},
           "calls": per_call,
           "step_frac": step.step_bytes / (ms_per_step / 1000.0) / 1e9 / peak,
           "gpu_launches": step.launches * args.steps,
           "clocks": clk.result,
           "step_ms_median": statistics.median(step_ms),
           "host_enqueue_us": host_us, "flush_us": flush_us}
    if e2e:
        e2e_ms, bi, bo = time_e2e(step, max(3, args.steps // 2), max(3, args.warmup), dev)
        e2e_ms = max_over_ranks(e2e_ms, dist)
        rec["e2e"] = {"value": world * step.layers / (e2e_ms / 1000.0), "unit": UNIT,
                      "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo}
    del step
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


# The configurations that carry the 70 %-of-HBM target, timed after the
# headline workload and reported beside it.
SUB_WORKLOADS = ("csa_1m", "hca_1m")


def main():
    args = parse()
    if args.record_traffic:
        record_traffic(args.record_traffic, args.call, args.workload, args.traffic_scale, args.traffic_note)
        return
    from compressed_kv_sparse_append_gb300 import workloads as wlmod
    wl = wlmod.WORKLOADS[args.workload]
    rank, world, dist = dist_setup()
    if args.impl == "reference":
        run_reference(args, wl, rank, world, dist)
        return
    import torch
    from compressed_kv_sparse_append_gb300 import binding as ckv
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = "cuda:%d" % local
    rec = measure(wl, args, dev, local, ckv, wlmod, dist, world)
    line = {"metric": METRIC, "value": rec.pop("value"), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec.pop("ms_per_step"),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp4/fp8/bf16 in, f32 accumulate", "data": "synthetic",
            "config": dict(workload_config(wl), launch="eager calls")}
    line.update(rec)
    if args.sub and args.workload not in SUB_WORKLOADS:
        sub_args = argparse.Namespace(**vars(args))
        sub_args.steps = min(args.steps, 20)
        line["sub"] = {}
        for name in SUB_WORKLOADS:
            r = measure(wlmod.WORKLOADS[name], sub_args, dev, local, ckv, wlmod, dist, world, e2e=False)
            line["sub"][name] = {"value": r["value"], "unit": UNIT, "ms_per_step": r["ms_per_step"],
                                 "steps": sub_args.steps, "roofline": r["roofline"], "calls": r["calls"],
                                 "step_frac": r["step_frac"], "clocks": r["clocks"],
                                 "config": workload_config(wlmod.WORKLOADS[name])}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, desc, _ = cpu_oracle_sample(wl, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
