#!/usr/bin/env python
"""Benchmark of the per-rank hot path of context-parallel causal attention
over packed THD (libcpthd on one GB300).

One *step* runs the whole path for one packed workload: for every strategy
the workload names and every context-parallel rank (sequentially, on one
GPU): partition index -> reorder of the Q slice and of the int64
input_ids / labels / position_ids, with the attention plan (row-group
metadata) beside it on a side stream -> the planned causal THD attention
kernel.

The headline metric is attention TFLOPS over unmasked pairs only
(4 * d * pairs * Hq per step, pairs counted from the rank's index list)
divided by the device time of the step, measured with CUDA events on the
launching stream. The step's library calls are captured once into a CUDA
graph and replayed, so host launch overhead does not enter the device time.
L2 (129 MB) is flushed between timed steps by writing a 256 MB buffer
outside the timed region. Each (strategy, rank) part is also replayed alone
to report per-rank attention times, and the attention kernel is replayed
alone (its plan, the row-group metadata, replayed outside the events) for
the roofline. The
end-to-end figure adds, every step, the host-to-device copy of all inputs
from pinned memory and the device-to-host copy of every output and LSE.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the float64 CPU oracle, timed on host cores

Under torchrun (N > 1) every rank runs an independent replica of the step
(weak scaling; the path has no collective), the slowest rank's time counts,
and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "causal-THD attn fwd TFLOPS (unmasked pairs) & % BF16 peak; reorder GB/s"
DEFAULT_WORKLOAD = "long131072_h8"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20

# DRAM bytes per launch of the attention kernel on the default workload
# (dram__bytes_read.sum + dram__bytes_write.sum from one ncu capture of the 32
# rank-slice launches of one step, averaged over them). The figure holds for
# the kernel sources that hash to ATTN_TRAFFIC["source_sha256"]; once they
# change, the line reports null until it is captured again.
ATTN_SOURCES = ("csrc/attn_fwd.cu", "csrc/attn_plan.cuh", "csrc/attn_common.cuh", "csrc/attn_meta.cuh",
                "csrc/sm100.cuh", "csrc/common.cuh")
ATTN_TRAFFIC = {"workload": "long131072_h8", "bytes_per_launch": 1061359112,
                "source_sha256": "2641be9ab235f1febf48f65e008aaf9a7e39d82ae703fb56cb015a130604a122"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    """(world_size, rank, local_rank) from the torchrun environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, device) -> float:
    """The largest value of ``x`` over all ranks (a time: the slowest replica
    counts). Identity without an initialised process group."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(units_per_replica: float, world: int, seconds: float) -> float:
    """Whole-job throughput of ``world`` replicas that each did the same work
    in at most ``seconds`` (weak scaling)."""
    return world * units_per_replica / seconds


def attn_source_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ATTN_SOURCES:
        with open(os.path.join(ROOT, "context_packed_thd_gb300", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(workload: str, subset: bool):
    """Per-launch DRAM bytes of the attention kernel (ATTN_TRAFFIC), or None
    when the workload differs, only part of the step runs, or the kernel
    sources changed since the capture."""
    if subset or workload != ATTN_TRAFFIC["workload"] or ATTN_TRAFFIC["bytes_per_launch"] is None:
        return None
    return ATTN_TRAFFIC["bytes_per_launch"] if attn_source_sha() == ATTN_TRAFFIC["source_sha256"] else None


def rank_pairs(idx: np.ndarray, lay: W.Layout) -> int:
    """Unmasked (query, key) pairs of one rank's slice, per head: a row at
    position pos of a document sees pos + 1 keys; pad rows see none."""
    cup = lay.cu_seqlens_padded.astype(np.int64)
    j = np.searchsorted(cup, idx, side="right") - 1
    pos = idx - cup[j]
    valid = pos < lay.lengths[j]
    return int((pos[valid] + 1).sum())


def attn_tiles(idx: np.ndarray, lay: W.Layout):
    """Query tiles (first row, rows) the attention plan cuts one slice into:
    at every change of document, a run's rows go into 128-row tiles aligned
    to the run's end with the remainder first, and runs shorter than a tile
    are packed together while they fit (the library's rule, restated here
    for reporting)."""
    cup = lay.cu_seqlens_padded.astype(np.int64)
    j = np.searchsorted(cup, idx, side="right") - 1
    n = len(idx)
    starts = np.r_[0, np.nonzero(np.diff(j) != 0)[0] + 1]
    ends = np.r_[starts[1:], n]
    tiles, cur0, curh = [], 0, 0
    for s, e in zip(starts.tolist(), ends.tolist()):
        head, full = (e - s) % 128, (e - s) // 128
        if head:
            if curh and curh + head <= 128:
                curh += head
            else:
                if curh:
                    tiles.append((cur0, curh))
                cur0, curh = s, head
        if full:
            if curh:
                tiles.append((cur0, curh))
                curh = 0
            tiles += [(s + head + 128 * f, 128) for f in range(full)]
    if curh:
        tiles.append((cur0, curh))
    return tiles


def kernel_pairs(idx: np.ndarray, lay: W.Layout, hq: int, hkv: int) -> int:
    """(query row, key) products per head that the attention kernel computes
    for one slice: every 128-row tile (two tiles per CTA item, sharing their
    key blocks, when the GQA group size is odd; one tile under two heads
    otherwise) walks, for every document among its group's real rows, the
    128-key blocks from the document start to the group's largest slot in it.
    Useful pairs / this = the fraction of the tensor work that is unmasked."""
    head_pairs = (hq // hkv) % 2 == 0
    cup = lay.cu_seqlens_padded.astype(np.int64)
    jj = np.searchsorted(cup, idx, side="right") - 1
    pos = idx - cup[jj]
    valid = pos < lay.lengths[jj]
    tiles = attn_tiles(idx, lay)
    if head_pairs:
        groups = [(a, a + h) for a, h in tiles]
    else:  # consecutive tiles in pairs: rows from the first tile's start to the second's end
        groups = [(tiles[i][0], sum(tiles[min(i + 1, len(tiles) - 1)])) for i in range(0, len(tiles), 2)]
    tiles_per_group = 1 if head_pairs else 2
    total = 0
    for a, b in groups:
        m = valid[a:b]
        if not m.any():
            continue
        dj, dp = jj[a:b][m], pos[a:b][m]
        for d in np.unique(dj):
            total += (int(dp[dj == d].max()) + 128) // 128
    return total * 128 * 128 * tiles_per_group


# ----------------------------------------------------------------------------
# clocks sampling (nvidia-smi during the timed region)
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# the CUDA path
# ----------------------------------------------------------------------------
class Strategy:
    """Device-resident inputs, outputs and workspaces of one strategy."""

    def __init__(self, cp, cfg, strategy, dev):
        self.name = strategy
        self.cfg = cfg
        inp = W.make_attn_inputs(cfg, strategy)
        lay = inp.layout
        self.lay = lay
        self.T = lay.T
        self.cpsize = cfg.cp
        self.t_local = cp.cp_local_tokens(strategy, lay.T, cfg.cp)
        ids, labels, pos = W.make_ids_logical(cfg.seed, lay)
        host = {
            "q": inp.q, "k": inp.k, "v": inp.v,
            "cu": torch.from_numpy(lay.cu_seqlens), "cup": torch.from_numpy(lay.cu_seqlens_padded),
            "ids": W.to_physical(ids, lay, -1), "labels": W.to_physical(labels, lay, -1),
            "pos": W.to_physical(pos, lay, -1),
        }
        self.host = {k: v.contiguous().pin_memory() for k, v in host.items()}
        self.dev = {k: v.to(dev) for k, v in self.host.items()}
        tl, hq, d = self.t_local, cfg.hq, cfg.d
        self.idx = [torch.empty(tl, dtype=torch.int32, device=dev) for _ in range(cfg.cp)]
        self.q_loc = [torch.empty((tl, hq, d), dtype=torch.bfloat16, device=dev) for _ in range(cfg.cp)]
        self.ids_loc = [[torch.empty(tl, dtype=torch.int64, device=dev) for _ in range(3)] for _ in range(cfg.cp)]
        self.out = [torch.empty((tl, hq, d), dtype=torch.bfloat16, device=dev) for _ in range(cfg.cp)]
        self.lse = [torch.empty((hq, tl), dtype=torch.float32, device=dev) for _ in range(cfg.cp)]
        self.ws = torch.empty(cp.thd_causal_attn_workspace_size(tl, hq, cfg.hkv, d), dtype=torch.uint8, device=dev)
        self.err = torch.zeros(2, dtype=torch.int32, device=dev)
        self.side = torch.cuda.Stream(device=dev)
        self.out_host = [torch.empty_like(o, device="cpu").pin_memory() for o in self.out]
        self.lse_host = [torch.empty_like(x, device="cpu").pin_memory() for x in self.lse]
        # algorithmic work, from the index lists the library itself returns
        self.pairs, self.kpairs = [], []
        for r in range(cfg.cp):
            cp.cp_partition_index(strategy, self.dev["cup"], self.T, cfg.cp, r, out=self.idx[r], err=self.err)
            idx_h = self.idx[r].cpu().numpy().astype(np.int64)
            self.pairs.append(rank_pairs(idx_h, lay))
            self.kpairs.append(kernel_pairs(idx_h, lay, hq, cfg.hkv))
        self.flops = [4.0 * d * p * hq for p in self.pairs]
        # reorder bytes per rank: read + write of every gathered row, plus the index list
        rb = hq * d * 2 + 3 * 8
        self.reorder_bytes = tl * (2 * rb + 4)
        # launches per rank: partition index 1, one gather of Q and the three
        # id tensors 1, the attention plan 2 (rows; groups with their tiles
        # and order), the attention kernel 1
        self.launches_per_rank = 5

    def run_prep(self, cp, r):
        # The rank's index list, then one gather of Q and the three id
        # tensors. (cp_partition_reorder_multi does both in one launch and is
        # faster alone, but the step of all ranks back to back runs 2.5%
        # slower with it on GB300: the two small launches chain better.)
        d = self.dev
        cp.cp_partition_index(self.name, d["cup"], self.T, self.cpsize, r, out=self.idx[r], err=self.err)
        cp.cp_reorder_multi([d["q"], d["ids"], d["labels"], d["pos"]], self.idx[r],
                            outs=[self.q_loc[r]] + self.ids_loc[r], err=self.err)

    def run_attn(self, cp, r):
        d = self.dev
        cp.thd_causal_attn_fwd(self.idx[r], self.q_loc[r], d["k"], d["v"], d["cu"], d["cup"], out=self.out[r],
                               lse=self.lse[r], workspace=self.ws, err=self.err)

    def run_plan(self, cp, r):
        d = self.dev
        cp.thd_causal_attn_plan(self.idx[r], self.T, d["cu"], d["cup"], self.cfg.hq, self.cfg.hkv, workspace=self.ws,
                                err=self.err)

    def run_kernel(self, cp, r):
        """The attention kernel alone, against the plan run_plan wrote."""
        d = self.dev
        cp.thd_causal_attn_fwd_planned(self.q_loc[r], d["k"], d["v"], self.ws, out=self.out[r], lse=self.lse[r],
                                       err=self.err)

    def run_rank(self, cp, r):
        """One rank slice as a caller would run it: the plan (row-group
        metadata) needs only the partition index, so it runs on a side
        stream while the gather runs on the current one, and the attention
        kernel waits for both."""
        d = self.dev
        main = torch.cuda.current_stream()
        cp.cp_partition_index(self.name, d["cup"], self.T, self.cpsize, r, out=self.idx[r], err=self.err)
        self.side.wait_stream(main)
        with torch.cuda.stream(self.side):
            self.run_plan(cp, r)
        cp.cp_reorder_multi([d["q"], d["ids"], d["labels"], d["pos"]], self.idx[r],
                            outs=[self.q_loc[r]] + self.ids_loc[r], err=self.err)
        main.wait_stream(self.side)
        self.run_kernel(cp, r)


def _graph_ms(fn, flush, reps=5):
    """Median device time of ``fn`` captured as a CUDA graph (L2 flushed before each replay)."""
    fn()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ms = []
    for _ in range(reps):
        flush.zero_()
        ev0.record(stream)
        g.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms.append(ev0.elapsed_time(ev1))
    return statistics.median(ms)


def other_workloads(cp, current, dev, flush, peak, peak_sustained, hbm_peak):
    """Attention throughput of every other multi-rank workload: all ranks of
    all its strategies in one CUDA graph (L2 flushed before each replay), so
    that the line also carries the long-context and many-document figures;
    the attention kernel alone per slice (plan written first, as for the
    headline's roofline); then the backward of every rank slice, each timed
    alone.
    Fractions are given of the burst and of the sustained bf16 peak: the
    long workload's graph runs tens of milliseconds of tensor work, long
    enough for the power cap to lower the clocks as in the sustained
    measurement."""
    out = {}
    for cfg in W.CONFIGS:
        if cfg.name in (current, "tiny"):
            continue
        sts = [Strategy(cp, cfg, s, dev) for s in cfg.strategies]
        for st in sts:
            for r in range(cfg.cp):
                st.run_prep(cp, r)

        def attn_all():
            for st in sts:
                for r in range(cfg.cp):
                    st.run_attn(cp, r)

        ms = _graph_ms(attn_all, flush, reps=3)
        # the attention kernel alone per slice (its plan written beforehand,
        # outside the timed graph), as the headline's roofline figure is
        kern_ms = {}
        for st in sts:
            kern_ms[st.name] = []
            for r in range(cfg.cp):
                st.run_plan(cp, r)
                kern_ms[st.name].append(_graph_ms(lambda st=st, r=r: st.run_kernel(cp, r), flush, reps=3))
        # each strategy's slices alone as well: DualChunkSwap balances the
        # ranks, NO_LOAD_BALANCE leaves them as uneven as the pack makes them
        by_strategy = {}
        if len(sts) > 1:
            for st in sts:
                ms_s = _graph_ms(lambda st=st: [st.run_attn(cp, r) for r in range(cfg.cp)], flush, reps=3)
                tf_s = sum(st.flops) / (ms_s * 1e-3) / 1e12
                tk_s = sum(st.flops) / (sum(kern_ms[st.name]) * 1e-3) / 1e12
                by_strategy[st.name] = {"attn_tflops": round(tf_s, 3), "frac_of_peak": round(tf_s / peak, 4),
                                        "frac_of_sustained_peak": round(tf_s / peak_sustained, 4),
                                        "ms": round(ms_s, 4), "kernel_tflops": round(tk_s, 3),
                                        "kernel_frac_of_peak": round(tk_s / peak, 4),
                                        "kernel_ms_per_rank_max": round(max(kern_ms[st.name]), 5),
                                        "kernel_ms_per_rank_min": round(min(kern_ms[st.name]), 5),
                                        "useful_pair_frac": round(sum(st.pairs) / sum(st.kpairs), 4)}
        dcs = [st for st in sts if st.name == W.DUAL_CHUNK_SWAP]
        restore = kv_restore(cp, cfg, dcs[0], flush, hbm_peak) if dcs else None
        bwd = backward(cp, cfg, sts, range(cfg.cp), flush, peak, peak_sustained)
        for st in sts:
            e = st.err.cpu().tolist()
            if e[0] != 0:
                raise RuntimeError(f"device check failed on {cfg.name}: {cp.cpthd_status_string(e[0])} ({e})")
        flops = sum(sum(st.flops) for st in sts)
        tf = flops / (ms * 1e-3) / 1e12
        tk = flops / (sum(sum(v) for v in kern_ms.values()) * 1e-3) / 1e12
        useful = sum(sum(st.pairs) for st in sts) / sum(sum(st.kpairs) for st in sts)
        out[cfg.name] = {"attn_tflops": round(tf, 3), "frac_of_peak": round(tf / peak, 4),
                         "frac_of_sustained_peak": round(tf / peak_sustained, 4), "ms": round(ms, 4),
                         "kernel_tflops": round(tk, 3), "kernel_frac_of_peak": round(tk / peak, 4),
                         "rank_slices": cfg.cp * len(sts), "strategies": list(cfg.strategies),
                         "useful_pair_frac": round(useful, 4),
                         "per_strategy": by_strategy or None, "kv_restore": restore, "backward": bwd}
        del sts
        torch.cuda.empty_cache()
    return out


def kv_restore(cp, cfg, st, flush, hbm_peak):
    """Restore of all-gathered K and V (rank-major) to token order: the
    gathered buffers are simulated on one GPU, the restore is one reorder
    launch of both tensors through cp_restore_index."""
    d = st.dev
    idx_all = cp.cp_partition_index(st.name, d["cup"], st.T, cfg.cp, -1)
    kg, vg = cp.cp_reorder(d["k"], idx_all), cp.cp_reorder(d["v"], idx_all)
    restore = cp.cp_restore_index(st.name, d["cup"], st.T, cfg.cp)
    ko, vo = torch.empty_like(kg), torch.empty_like(vg)
    ms = _graph_ms(lambda: cp.cp_reorder_multi([kg, vg], restore, outs=[ko, vo], err=st.err), flush)
    ok = torch.equal(ko.view(torch.int16), d["k"].view(torch.int16)) and torch.equal(vo.view(torch.int16),
                                                                                     d["v"].view(torch.int16))
    row = cfg.hkv * cfg.d * 2
    nbytes = st.T * (2 * 2 * row + 4)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"strategy": st.name, "GB/s": round(gbs, 1), "peak_GB/s": hbm_peak, "frac": round(gbs / hbm_peak, 4),
            "ms": round(ms, 5), "bytes": nbytes, "bit_exact": bool(ok)}


def dcs_two_launch(cp, cfg, st, ranks, flush):
    """Matched-input comparison: a DualChunkSwap rank's attention as one launch
    over its whole slice against two launches, one per owned chunk (the two
    attention steps the pages describe), on the same inputs. The two
    launches' outputs, put back in slice order, are compared with the one
    launch's (max |difference|), and the device checks are read."""
    d = st.dev
    lay = st.lay
    lcu = lay.cu_seqlens_padded.astype(np.int64) // cfg.cp
    halves = [[], []]
    for j in range(lay.num_docs):
        c = (lcu[j + 1] - lcu[j]) // 2
        halves[0].append(np.arange(lcu[j], lcu[j] + c))
        halves[1].append(np.arange(lcu[j] + c, lcu[j + 1]))
    rows = [np.concatenate(h).astype(np.int64) for h in halves]
    fused, split, max_diff, identical = [], [], 0.0, True
    for r in ranks:
        rows_d = [torch.from_numpy(x).to(st.idx[r].device) for x in rows]
        idx_h = [st.idx[r][x].contiguous() for x in rows_d]
        q_h = [st.q_loc[r][x].contiguous() for x in rows_d]
        out_h = [torch.empty_like(q) for q in q_h]
        lse_h = [torch.empty((cfg.hq, q.shape[0]), dtype=torch.float32, device=q.device) for q in q_h]
        ws_h = [torch.empty(cp.thd_causal_attn_workspace_size(q.shape[0], cfg.hq, cfg.hkv, cfg.d), dtype=torch.uint8,
                            device=q.device) for q in q_h]

        def two():
            for h in range(2):
                cp.thd_causal_attn_fwd(idx_h[h], q_h[h], d["k"], d["v"], d["cu"], d["cup"], out=out_h[h],
                                       lse=lse_h[h], workspace=ws_h[h], err=st.err)
        fused.append(_graph_ms(lambda: st.run_attn(cp, r), flush, reps=3))
        split.append(_graph_ms(two, flush, reps=3))
        torch.cuda.synchronize()
        e = st.err.cpu().tolist()
        if e[0] != 0:
            raise RuntimeError(f"device check failed in the two-launch run: {cp.cpthd_status_string(e[0])} ({e})")
        out_one, lse_one = st.out[r], st.lse[r]
        for h in range(2):
            do = (out_h[h].float() - out_one[rows_d[h]].float()).abs().max().item()
            fin = torch.isfinite(lse_one[:, rows_d[h]])
            if not torch.equal(fin, torch.isfinite(lse_h[h])):
                raise RuntimeError("two-launch run: pad rows differ from the one-launch run")
            dl = (lse_h[h][fin] - lse_one[:, rows_d[h]][fin]).abs().max().item() if fin.any() else 0.0
            max_diff = max(max_diff, do, dl)
            identical = identical and torch.equal(out_h[h], out_one[rows_d[h]]) and torch.equal(
                lse_h[h][fin], lse_one[:, rows_d[h]][fin])
    if max_diff > 2e-2:
        raise RuntimeError(f"two-launch outputs differ from the one-launch outputs by {max_diff}")
    return {"attn_ms_one_launch": round(sum(fused), 5), "attn_ms_two_launches": round(sum(split), 5),
            "two_over_one": round(sum(split) / sum(fused), 3), "ranks": len(ranks),
            "max_abs_diff_vs_one_launch": max_diff, "bit_identical_to_one_launch": bool(identical)}


def backward(cp, cfg, strategies, ranks, flush, peak, peak_sustained=None):
    """The attention backward of every (strategy, rank) slice of the step,
    timed alone (graph replays, L2 flushed before each). Algorithmic work is
    the usual 2.5x the forward: 10 * d * pairs * Hq (the S recompute, dP, dS V,
    dQ, dK, dV products counted once). It runs after the timed step, for tens
    of milliseconds of tensor work, so it is given as a fraction of both the
    burst and the sustained peak."""
    res = {}
    tot_f, tot_ms = 0.0, 0.0
    for st in strategies:
        d = st.dev
        dev = d["q"].device
        tl = st.t_local
        dout = W.randn_bf16(cfg.seed, 6, (tl, cfg.hq, cfg.d)).to(dev)
        dq = torch.empty((tl, cfg.hq, cfg.d), dtype=torch.float32, device=dev)
        dk = torch.empty((st.T, cfg.hkv, cfg.d), dtype=torch.float32, device=dev)
        dv = torch.empty_like(dk)
        ws = torch.empty(cp.thd_causal_attn_bwd_workspace_size(tl, cfg.hq, cfg.hkv, cfg.d), dtype=torch.uint8,
                         device=dev)
        ms, fl = [], []
        for r in ranks:
            st.run_rank(cp, r)
            ms.append(_graph_ms(lambda: cp.thd_causal_attn_bwd(
                st.idx[r], st.q_loc[r], d["k"], d["v"], st.out[r], dout, st.lse[r], d["cu"], d["cup"], dq=dq, dk=dk,
                dv=dv, workspace=ws, err=st.err), flush, reps=3))
            fl.append(2.5 * st.flops[r])
        res[st.name] = {"ms_per_rank_max": round(max(ms), 5), "ms_per_rank_min": round(min(ms), 5),
                        "tflops": round(sum(fl) / (sum(ms) * 1e-3) / 1e12, 3)}
        tot_f += sum(fl)
        tot_ms += sum(ms)
        del dq, dk, dv, ws
    tf = tot_f / (tot_ms * 1e-3) / 1e12
    res["all"] = {"tflops": round(tf, 3), "frac_of_peak": round(tf / peak, 4),
                  "flops": "10 * d * unmasked pairs * Hq per slice"}
    if peak_sustained:
        res["all"]["frac_of_sustained_peak"] = round(tf / peak_sustained, 4)
    return res


def activation_reorder(cp, cfg, st, ranks, flush, dev, hbm_peak):
    """Reorder of the workload's [T, width] bf16 activations into every rank's
    token order (graph replays, L2 flushed before each)."""
    act = W.make_activations(cfg.seed, st.T, cfg.act_width, device=str(dev))
    out = torch.empty((st.t_local, cfg.act_width), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    times = []
    for r in ranks:
        cp.cp_reorder(act, st.idx[r], out=out, err=st.err)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cp.cp_reorder(act, st.idx[r], out=out, err=st.err)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ms = []
        for _ in range(5):
            flush.zero_()
            ev0.record(stream)
            g.replay()
            ev1.record(stream)
            torch.cuda.synchronize()
            ms.append(ev0.elapsed_time(ev1))
        times.append(statistics.median(ms))
    row = cfg.act_width * 2
    per_rank_bytes = st.t_local * (2 * row + 4)
    gbs = per_rank_bytes * len(ranks) / (sum(times) * 1e-3) / 1e9
    del act, out
    return {"GB/s": round(gbs, 1), "peak_GB/s": hbm_peak, "frac": round(gbs / hbm_peak, 4),
            "bytes_per_rank": per_rank_bytes, "ms_per_rank_max": round(max(times), 5),
            "shape": f"[{st.T}, {cfg.act_width}] bf16 -> [{st.t_local}, {cfg.act_width}] per rank, {st.name}"}


def run_cuda(args):
    import context_packed_thd_gb300 as cp

    world, rank, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = W.CONFIG_BY_NAME[args.workload]
    names = [s for s in cfg.strategies if args.strategy in (None, s)]
    if args.strategy == W.PACKED_MIRRORED:
        names = [W.PACKED_MIRRORED]
    if not names:
        raise SystemExit(f"workload {cfg.name} does not run strategy {args.strategy}")
    strategies = [Strategy(cp, cfg, s, dev) for s in names]
    ranks = list(range(cfg.cp)) if args.rank is None else [args.rank]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        for st in strategies:
            for r in ranks:
                st.run_rank(cp, r)

    n_ranks = len(ranks) * len(strategies)
    for _ in range(args.warmup):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    for st in strategies:
        e = st.err.cpu().tolist()
        if e[0] != 0:
            raise RuntimeError(f"device check failed during warm-up: {cp.cpthd_status_string(e[0])} ({e})")

    # ---- CUDA graphs: the whole step, and every (strategy, rank) part alone ---
    # The library's calls are plain kernel launches on the current stream, so
    # a step is captured once and replayed; this removes the host-side launch
    # gaps that would otherwise dominate the small workloads.
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        step()
    g_prep, g_attn, g_plan, g_kern = [], [], [], []
    for st in strategies:
        for r in ranks:
            gp, ga, gl, gk = (torch.cuda.CUDAGraph() for _ in range(4))
            with torch.cuda.graph(gp):
                st.run_prep(cp, r)
            with torch.cuda.graph(ga):
                st.run_attn(cp, r)
            with torch.cuda.graph(gl):
                st.run_plan(cp, r)
            with torch.cuda.graph(gk):
                st.run_kernel(cp, r)
            g_prep.append(gp)
            g_attn.append(ga)
            g_plan.append(gl)
            g_kern.append(gk)
    torch.cuda.synchronize()
    for _ in range(2):
        g_step.replay()
    torch.cuda.synchronize()

    # ---- device-timed region -------------------------------------------------
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush.zero_()
        step_ev[i][0].record(stream)
        g_step.replay()
        step_ev[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()

    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    total_ms = sum(step_ms)
    flops_step = sum(st.flops[r] for st in strategies for r in ranks)
    total_ms = max_over_ranks(total_ms, dev)
    value = replica_value(flops_step * args.steps, world, total_ms * 1e-3) / 1e12

    # ---- end to end: pinned host inputs -> step -> host results --------------
    # Measured right after the device-timed region, before the extras (which
    # allocate and free gigabytes of pinned memory), after two untimed
    # iterations, with Python's collector held off; the median step counts.
    # Copies and compute overlap per strategy the way a caller would overlap
    # them: the inputs go up on one copy stream, each strategy's ranks run
    # once its inputs are in, and its outputs go down on a second copy stream
    # while the next strategy runs.
    e2e_steps = max(3, min(args.steps, 10))
    h2d = sum(sum(t.numel() * t.element_size() for t in st.host.values()) for st in strategies)
    d2h = sum(st.out[r].numel() * st.out[r].element_size() + st.lse[r].numel() * st.lse[r].element_size()
              for st in strategies for r in ranks)
    g_rank = []
    for st in strategies:
        gs = []
        for r in ranks:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                st.run_rank(cp, r)
            gs.append(g)
        g_rank.append(gs)
    up_stream, down_stream = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_step():
        inputs_in = []
        with torch.cuda.stream(up_stream):
            for st in strategies:
                for key, h in st.host.items():
                    st.dev[key].copy_(h, non_blocking=True)
                inputs_in.append(up_stream.record_event())
        for k, st in enumerate(strategies):
            stream.wait_event(inputs_in[k])
            for i, r in enumerate(ranks):
                g_rank[k][i].replay()
                computed = stream.record_event()
                # each rank's results go down while the next rank computes
                with torch.cuda.stream(down_stream):
                    down_stream.wait_event(computed)
                    st.out_host[r].copy_(st.out[r], non_blocking=True)
                    st.lse_host[r].copy_(st.lse[r], non_blocking=True)
        torch.cuda.synchronize()

    gc.collect()
    gc.disable()
    try:
        for _ in range(2):
            e2e_step()
        e2e_times = []
        for _ in range(e2e_steps):
            t0 = time.perf_counter()
            e2e_step()
            e2e_times.append(time.perf_counter() - t0)
    finally:
        gc.enable()
    e2e_s = max_over_ranks(statistics.median(e2e_times), dev)
    e2e_value = replica_value(flops_step, world, e2e_s) / 1e12

    # ---- each part of the step alone (graph replays, L2 flushed before each) --
    reps = 20  # median of 20 replays per (strategy, rank) part
    # The attention kernel is timed alone for the roofline: the plan (row-
    # group metadata, group order) is replayed outside the events, then the
    # planned attention launch between them.
    attn_ms = [[0.0] * reps for _ in range(n_ranks)]
    prep_ms = [[0.0] * reps for _ in range(n_ranks)]
    kern_ms = [[0.0] * reps for _ in range(n_ranks)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for k in range(n_ranks):
        for i in range(reps):
            flush.zero_()
            ev[0].record(stream)
            g_prep[k].replay()
            ev[1].record(stream)
            flush.zero_()
            ev[2].record(stream)
            g_attn[k].replay()
            ev[3].record(stream)
            g_plan[k].replay()
            flush.zero_()
            ev[4].record(stream)
            g_kern[k].replay()
            ev[5].record(stream)
            torch.cuda.synchronize()
            prep_ms[k][i] = ev[0].elapsed_time(ev[1])
            attn_ms[k][i] = ev[2].elapsed_time(ev[3])
            kern_ms[k][i] = ev[4].elapsed_time(ev[5])

    # per-rank attention times (median over replays) and the dominant-kernel roofline
    med_attn = [statistics.median(x) for x in attn_ms]
    med_kern = [statistics.median(x) for x in kern_ms]
    med_prep = [statistics.median(x) for x in prep_ms]
    per_strategy = {}
    k = 0
    for st in strategies:
        ms = med_attn[k:k + len(ranks)]
        kms = med_kern[k:k + len(ranks)]
        fl = [st.flops[r] for r in ranks]
        pr = [st.pairs[r] for r in ranks]
        kp = [st.kpairs[r] for r in ranks]
        per_strategy[st.name] = {
            "attn_ms_per_rank_max": round(max(ms), 5), "attn_ms_per_rank_min": round(min(ms), 5),
            "kernel_ms_per_rank_max": round(max(kms), 5), "kernel_ms_per_rank_min": round(min(kms), 5),
            "kernel_ms_max_over_min": round(max(kms) / min(kms), 3),
            "rank_of_max": ranks[kms.index(max(kms))], "rank_of_min": ranks[kms.index(min(kms))],
            "kernel_ms_per_rank": [round(x, 5) for x in kms],
            "attn_tflops": round(sum(fl) / (sum(ms) * 1e-3) / 1e12, 3),
            "kernel_tflops": round(sum(fl) / (sum(kms) * 1e-3) / 1e12, 3),
            "pairs_per_rank_max": max(pr), "pairs_per_rank_min": min(pr),
            "pairs_max_over_min": round(max(pr) / min(pr), 3),
            "useful_pair_frac": round(sum(pr) / sum(kp), 4),
        }
        k += len(ranks)
    achieved = flops_step / (sum(med_kern) * 1e-3) / 1e12
    call_tflops = flops_step / (sum(med_attn) * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    peak_sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    reorder_bytes = sum(st.reorder_bytes * len(ranks) for st in strategies)
    prep_total_ms = sum(med_prep)
    act = activation_reorder(cp, cfg, strategies[0], ranks, flush, dev, hbm_peak) if cfg.act_width else None
    dcs_st = [st for st in strategies if st.name == W.DUAL_CHUNK_SWAP]
    extras = set() if args.no_extras else set(args.extras.split(","))
    restore = kv_restore(cp, cfg, dcs_st[0], flush, hbm_peak) if dcs_st and "restore" in extras else None
    two = dcs_two_launch(cp, cfg, dcs_st[0], ranks, flush) if dcs_st and "two_launch" in extras else None
    bwd = backward(cp, cfg, strategies, ranks, flush, peak, peak_sustained) if "backward" in extras else None
    others = other_workloads(cp, cfg.name, dev, flush, peak, peak_sustained, hbm_peak) if "others" in extras else None


    for st in strategies:
        e = st.err.cpu().tolist()
        if e[0] != 0:
            raise RuntimeError(f"device check failed: {cp.cpthd_status_string(e[0])} ({e})")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": cfg.name, "T": int(sum(cfg.lengths)), "docs": len(cfg.lengths), "Hq": cfg.hq,
                       "Hkv": cfg.hkv, "d": cfg.d, "cp_size": cfg.cp, "strategies": list(cfg.strategies),
                       "ranks_per_step": n_ranks, "flops_per_step": flops_step,
                       "subset": None if (args.strategy is None and args.rank is None)
                       else {"strategy": args.strategy, "rank": args.rank},
                       "l2": "flushed between timed steps (256 MB write, untimed); K/V and Q exceed L2",
                       "launch": "one CUDA graph per step (the library calls, captured once)",
                       "parallelism": f"replicas{world}"},
            "per_strategy": per_strategy,
            "reorder": {"GB/s": round(reorder_bytes / (prep_total_ms * 1e-3) / 1e9, 2),
                        "bytes_per_step": reorder_bytes,
                        "note": "partition index + one gather launch of Q and the int64 ids, timed together per rank"},
            "reorder_activations": act,
            "kv_restore": restore,
            "dcs_one_vs_two_launches": two,
            "backward": bwd,
            "attention_other_workloads": others,
            "useful_pair_frac": round(sum(sum(st.pairs) for st in strategies)
                                      / sum(sum(st.kpairs) for st in strategies), 4),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4),
                         "frac_of_sustained_peak": round(achieved / peak_sustained, 4),
                         "traffic": measured_traffic(cfg.name, args.strategy is not None or args.rank is not None),
                         "kernel": "attn_fwd_tc_kernel (thd_causal_attn_fwd_planned, timed per launch; the plan "
                                   "is replayed outside the events)",
                         "launch_us_mean": round(sum(med_kern) / len(med_kern) * 1e3, 3),
                         "whole_call_tflops": round(call_tflops, 3),
                         "peak_source": f"{peak_src} bf16_tflops (burst); sustained = {peak_src} "
                                        "bf16_tflops_sustained"},
            "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 4),
                    "timing": f"wall clock, median of {e2e_steps} steps after 2 untimed ones; uploads per "
                              "strategy, compute, and downloads per rank slice overlapped on three streams"},
            "gpu_launches": sum(st.launches_per_rank for st in strategies) * len(ranks) * args.steps,
            "gpu_launches_note": "library kernels inside the timed step replays; the L2 flush between steps is a torch fill",
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ----------------------------------------------------------------------------
# the float64 oracle on host cores
# ----------------------------------------------------------------------------
class OracleSlices:
    """The oracle's inputs and partitions of one workload, built once (not
    timed), and the oracle's forward of one rank slice, timed: the partition
    index, the gather of the Q slice and the attention of all its rows, or of
    ``n_rows`` evenly spaced rows."""

    def __init__(self, cfg):
        from oracle import partition as P
        self.cfg = cfg
        self.inputs = {s: W.make_attn_inputs(cfg, s) for s in cfg.strategies}
        self.pairs = {}
        for s in cfg.strategies:
            lay = self.inputs[s].layout
            for r in range(cfg.cp):
                idx = np.asarray(P.partition_index(s, lay.cu_seqlens_padded.tolist(), cfg.cp, r), dtype=np.int64)
                self.pairs[(s, r)] = rank_pairs(idx, lay)

    def flops(self, key) -> float:
        return 4.0 * self.cfg.d * self.cfg.hq * self.pairs[key]

    def run(self, strategy, r, n_rows=None):
        """Returns (seconds, unmasked-pair FLOPs computed, rows computed)."""
        from oracle import attention as A
        from oracle import partition as P
        cfg = self.cfg
        inp = self.inputs[strategy]
        lay = inp.layout
        t0 = time.perf_counter()
        idx = np.asarray(P.partition_index(strategy, lay.cu_seqlens_padded.tolist(), cfg.cp, r), dtype=np.int64)
        q_loc = inp.q[torch.from_numpy(idx)]
        rows = None
        if n_rows is not None and n_rows < len(idx):
            rows = np.unique(np.linspace(0, len(idx) - 1, max(int(n_rows), 1)).round().astype(np.int64))
        A.attention_fwd(q_loc, inp.k, inp.v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, rows=rows)
        dt = time.perf_counter() - t0
        sel = idx if rows is None else idx[rows]
        return dt, 4.0 * cfg.d * cfg.hq * rank_pairs(sel, lay), len(sel)


def cpu_model() -> str:
    """Host CPU model name (best effort; Arm hosts report it through lscpu)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(cfg, seconds):
    """Time the oracle as it stands on a bounded sample of the workload (about
    ``seconds`` of CPU work): whole rank slices from the cheapest up while
    they fit, then evenly spaced rows of each strategy's costliest slice not
    yet timed, sized by the rate measured so far to fill the rest."""
    orc = OracleSlices(cfg)
    order = sorted(orc.pairs, key=lambda k: (orc.pairs[k], k))
    t_sum, f_sum, done = 0.0, 0.0, []
    timed = set()
    for key in order:
        if t_sum > 0 and orc.flops(key) / (f_sum / t_sum) > seconds - t_sum:
            break
        dt, f, _ = orc.run(*key)
        t_sum, f_sum = t_sum + dt, f_sum + f
        done.append(f"{key[0]}:{key[1]} (all rows)")
        timed.add(key)
        if t_sum >= seconds:
            break
    rest = [k for k in order if k not in timed]
    costliest = []
    for s in cfg.strategies:
        ks = [k for k in rest if k[0] == s]
        if ks:
            costliest.append(ks[-1])
    for i, key in enumerate(costliest):
        left = seconds - t_sum
        if left <= 0.5:
            break
        share = left / (len(costliest) - i)
        t_local = W.layout_for(cfg, key[0]).T // cfg.cp
        n = max(16, int(t_local * share * (f_sum / t_sum) / orc.flops(key)))
        dt, f, rows = orc.run(*key, n_rows=n)
        t_sum, f_sum = t_sum + dt, f_sum + f
        done.append(f"{key[0]}:{key[1]} ({rows} evenly spaced rows of {W.layout_for(cfg, key[0]).T // cfg.cp})")
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(f_sum / t_sum / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{cfg.name}: rank slices {', '.join(done)}; all heads, float64 numpy, partition + Q gather "
                      f"+ attention timed, {t_sum:.1f} s"}


# FLOPs of oracle work per reference-arm step: a whole rank slice when it is
# smaller, else this many FLOPs' worth of its rows (evenly spaced).
REFERENCE_STEP_FLOPS = 4e10


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    cfg = W.CONFIG_BY_NAME[args.workload]
    orc = OracleSlices(cfg)
    order = [(s, r) for s in cfg.strategies for r in range(cfg.cp)]
    t_local = {s: W.layout_for(cfg, s).T // cfg.cp for s in cfg.strategies}

    def one(i):
        key = order[i % len(order)]
        f_slice = orc.flops(key)
        n = None if f_slice <= REFERENCE_STEP_FLOPS else max(16, int(t_local[key[0]] * REFERENCE_STEP_FLOPS / f_slice))
        return orc.run(*key, n_rows=n)

    for i in range(args.warmup):
        one(i)
    t_sum, f_sum = 0.0, 0.0
    for i in range(args.steps):
        dt, f, _ = one(i)
        t_sum += dt
        f_sum += f
    value = f_sum / t_sum / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = (f"{cfg.name}: one rank slice per step, cycling the {len(order)} (strategy, rank) slices; a slice of "
              f"more than {REFERENCE_STEP_FLOPS:.0e} unmasked-pair FLOP is cut to that many FLOPs' worth of evenly "
              "spaced rows; partition + Q gather + attention in float64 numpy")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t_sum / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "T": int(sum(cfg.lengths)), "Hq": cfg.hq, "Hkv": cfg.hkv, "d": cfg.d,
                   "cp_size": cfg.cp, "strategies": list(cfg.strategies)},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.CONFIG_BY_NAME))
    ap.add_argument("--cpu-seconds", type=float, default=20.0, help="CPU-oracle sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the K/V restore, one-vs-two-launch, backward and other-workload measurements")
    ap.add_argument("--extras", default="restore,two_launch,backward,others",
                    help="comma-separated extras to run (restore, two_launch, backward, others)")
    ap.add_argument("--strategy", choices=list(W.ALL_STRATEGIES), default=None,
                    help="time one strategy only (profiling); the headline runs every strategy")
    ap.add_argument("--rank", type=int, default=None,
                    help="time one context-parallel rank only (profiling); the headline runs every rank")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "cuda":
        print("note: --warmup below 3 is not a valid measurement", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_cuda(args)


if __name__ == "__main__":
    main()
