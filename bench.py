"""Benchmark of indexer-selected block-sparse attention on GB300 (one JSON line on stdout).

A step is one pass of the whole method over one batch of queries: pool the index-key blocks
that this step's tokens complete, score every visible block, keep the top-k blocks plus the
tail, and attend over the kept cells (sfa_pool_index_keys -> sfa_index_scores ->
sfa_topk_blocks -> sfa_gather_attend).  Inputs are seeded synthetic tensors resident in HBM;
L2 is flushed before every timed step, outside the timed events: 512 MB are written, then a
separate 256 MB buffer is read, so that no dirty line of the flush is written back inside the
timed step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

--impl reference times the CPU oracle (the plain fp64 C implementation) on the host cores on
a bounded sample of the same workload.  Under torchrun each rank runs its own replica of the
workload on its own GPU (weak scaling, no collective on the data path); rank 0 prints.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import indexer_selected_sparse_block_gb300 as sfa  # noqa: E402
from indexer_selected_sparse_block_gb300 import _binding as B  # noqa: E402

METRIC = "sparse-attn tokens/s (decode, pp2048) at depth; gathered-KV HBM GB/s vs peak"
DEFAULT_WORKLOAD = "decode_32x131072"
SECOND_WORKLOAD = "pp2048_131072"
PAGE_CELLS = 64
Q8_CACHE = ("q8_0 rows (blocks of 32 int8 codes with a binary16 scale; 624 B per 576-wide row), "
            "attention on binary16 tensor-core operands")
WINDOW = 128   # positions of the dense window in the dense-window + sparse companion line
PAGED_LAYOUT = (f"paged: {PAGE_CELLS}-cell pages dealt from a seeded shuffled page table, "
                "one spare page per sequence")
L2_FLUSH_BYTES = 512 << 20
HOLD_CYCLES = 400_000          # ~0.2 ms GPU spin that covers the host's enqueue of one step
CSRC = os.path.join(ROOT, "indexer_selected_sparse_block_gb300", "csrc")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def src_hash(name):
    with open(os.path.join(CSRC, name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel, workload, source):
    """dram bytes per launch from a committed ncu summary, if taken on the current source of
    the kernel that runs (source: its file)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(f"{kernel}@{workload}")
    except Exception:
        return None
    if not rec or rec.get("source") != source or rec.get("src_sha256_16") != src_hash(source):
        return None
    return rec["dram_bytes_per_launch"]


# ------------------------------------------------------------------ algorithmic work per step
def algorithmic(w, attended, bounded=None, kv="bf16"):
    """Bytes / FLOPs each stage must move / do for one step of workload w (one rank).

    attended[i] = |A_i|, the number of cells query i attends (kept blocks * cr + tail).
    Pooled keys are 4*d_idx bytes per block (bf16 hi + lo halves); a query tile of one
    sequence reads that sequence's pooled keys once, so decode reads them once per query and
    a prefill ubatch once per sequence.  bounded: the bound pass of the bounded selection --
    "i8" reads d_idx bytes of codes and 8 of scale and bound factor per block, "hi" (or True)
    2*d_idx bytes of hi halves and a 4-byte bound factor; None / False: the exact scores.
    """
    cr = w.compress_ratio
    nb = [(w.depth + j + 1) // cr for j in range(w.n_q_per_seq)] * w.n_seq
    if kv == "q8_0":   # q8_0 cache rows: codes, binary16 scales, padding
        kv_row = w.h_kv * (B.sfa_q8_0_row_bytes(w.dkq) + (0 if w.v_is_k else B.sfa_q8_0_row_bytes(w.dv)))
    else:
        kv_row = w.h_kv * (w.dkq + (0 if w.v_is_k else w.dv)) * 2
    if bounded == "i8":   # codes + (scale, bound factor)
        per_blk = w.d_idx + 8
    elif bounded:         # hi halves + bound factor
        per_blk = 2 * w.d_idx + 4
    else:
        per_blk = 4 * w.d_idx
    if w.kind == "decode":
        kbar_bytes = sum(b * per_blk for b in nb)
    else:
        kbar_bytes = w.n_seq * max(nb) * per_blk
    return {
        "kbar_bytes": kbar_bytes,
        "score_bytes": sum(b * (8 if bounded else 4) for b in nb),   # + the bounds
        "score_flops": sum(b * 2 * w.h_idx * w.d_idx for b in nb),
        "gathered_kv_bytes": sum(a * kv_row for a in attended),
        "attend_flops": sum(a * 2 * w.h_q * (w.dkq + w.dv) for a in attended),
    }


# ------------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 10 ms while the steps run; summary() keeps the samples taken
    between mark_start() and mark_end() (warm-up and timed steps: the GPU under load)."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "10"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)   # let the sampler start before the load does
        self.t0 = self.t1 = None
        return self

    def mark_start(self):
        self.t0 = datetime.datetime.now()

    def mark_end(self):
        self.t1 = datetime.datetime.now()

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                ts = None
            if ts is not None and self.t0 is not None and self.t1 is not None and \
                    not (self.t0 <= ts <= self.t1):
                continue
            try:
                sm.append(float(f[2]))
                mx = max(mx, float(f[3]))
            except ValueError:
                continue
            for name, v in zip(names, f[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------ GPU arm
class Workbench:
    """Inputs, buffers and one step of the method for workload w on the current device."""

    def __init__(self, w, dev, bounded=None, paged=False, kv="bf16", window=0,
                 window_mode="single", bound_pass=None):
        self.w, self.dev, self.paged, self.kv = w, dev, paged, kv
        self.case = sfa.make_case(w, device=dev)
        self.n_blk_max = w.n_tok // w.compress_ratio
        # the drawn bf16 rows, per sequence: the host source of the end-to-end step's new rows
        self.seq_rows = {n: self.case[n] for n in ("X", "K", "V") if self.case[n] is not None}
        if kv == "q8_0":   # K and V as q8_0 cache rows (the index keys X stay bf16)
            for n in ("K", "V"):
                t = self.case[n]
                if t is not None:
                    rb = B.sfa_q8_0_row_bytes(t.shape[-1])
                    y = torch.empty(t.shape[:-1] + (rb,), dtype=torch.uint8, device=dev)
                    B.sfa_quantize_kv_q8_0(t.view(t.shape[0], -1, t.shape[-1]),
                                           y.view(t.shape[0], -1, rb))
                    self.case[n] = y
        self.cell_of = None
        if paged:
            # a paged cache: the same rows in 64-cell pages dealt from a seeded shuffled page
            # table (one spare page per sequence)
            self.cell_of, n_cells = sfa.make_cell_map(w.n_seq, w.n_tok, page=PAGE_CELLS,
                                                      spare_pages=w.n_seq, seed=w.seed,
                                                      device=dev)
            for n in ("X", "K", "V"):
                if self.case[n] is not None:
                    self.case[n] = sfa.to_cells(self.case[n], self.cell_of, n_cells)
        self.step = sfa.SfaStep(n_seq=w.n_seq, n_tok_cap=w.n_tok, n_q=w.n_q, h_q=w.h_q,
                                h_kv=w.h_kv, dkq=w.dkq, dv=w.dv, h_idx=w.h_idx, d_idx=w.d_idx,
                                compress_ratio=w.compress_ratio,
                                indexer_top_k=w.indexer_top_k, n_blk_max=self.n_blk_max,
                                q_group=w.n_q_per_seq, bounded=bounded, cell_of=self.cell_of,
                                window=window, window_mode=window_mode, bound_pass=bound_pass,
                                device=dev)
        # the cache state before the step: every block completed by earlier tokens is pooled
        self.first_new_blk = w.depth // w.compress_ratio
        self.step.pool(self.case["X"], 0, self.first_new_blk)
        # blocks completed by this step's tokens (depth .. depth + n_q_per_seq - 1)
        self.new_blocks = (self.first_new_blk, self.n_blk_max)
        torch.cuda.synchronize()

    def launches_per_step(self):
        w, st = self.w, self.step
        n = 1 if self.new_blocks[1] > self.new_blocks[0] else 0
        if n and st.bound_pass == "i8":
            n += 1  # the 8-bit copy of the new pooled rows
        if not st.dense:
            n += 1  # scores
            if st.bounded:
                n += 1  # the cluster selection kernel
            else:
                n += 1 + (B.sfa_topk_workspace_bytes(w.n_q, self.n_blk_max, w.indexer_top_k) > 0)
            n_kv = w.indexer_top_k * w.compress_ratio + w.compress_ratio - 1
        else:
            n_kv = st.n_kv_dense
        dt = B.SFA_Q8_0 if self.kv == "q8_0" else B.SFA_BF16
        n += B.sfa_attend_plan(dt, w.n_q, w.h_kv, w.dkq, not w.v_is_k, n_kv, w.compress_ratio,
                               st.dense)[1]
        return n

    def run_step(self, events=None, before_attend=None):
        c, st, w = self.case, self.step, self.w
        ev = events or {}
        if "pool" in ev:
            ev["pool"][0].record()
        st.pool(c["X"], *self.new_blocks)
        if "pool" in ev:
            ev["pool"][1].record()
        if not st.dense:
            if "scores" in ev:
                ev["scores"][0].record()
            st.score(c["q_idx"], c["w"], c["q_seq"], c["q_pos"])
            if "scores" in ev:
                ev["scores"][1].record()
                ev["topk"][0].record()
            st.topk(c["q_idx"], c["w"], c["q_seq"], c["q_pos"])
            if "topk" in ev:
                ev["topk"][1].record()
        if before_attend is not None:
            before_attend()
        if "attend" in ev:
            ev["attend"][0].record()
        st.attend(c["Q"], c["K"], c["V"], c["q_seq"], c["q_pos"], w.scale)
        if "attend" in ev:
            ev["attend"][1].record()


def flush_l2(flush):
    """Evicts L2: writes the 512 MB flush buffer, then reads a clean 256 MB one, so that the
    flush leaves clean lines only (nothing of it is written back inside a timed step)."""
    flush[0].zero_()
    flush[1].sum()


def measure(wb, steps, warmup, flush, per_stage=True, clk=None):
    """Device time of `steps` steps (L2 flushed before each), plus per-stage averages.

    Before each timed step the stream is held by a short GPU spin (outside the timed events)
    so that the host has enqueued the whole step before the first timed event runs: the
    events then see GPU execution only, not host launch latency."""
    if clk is not None:
        clk.mark_start()
    for _ in range(warmup):
        flush_l2(flush)
        wb.run_step()
    torch.cuda.synchronize()
    stages = ["pool", "scores", "topk", "attend"]
    step_ms, stage_ms = [], {s: [] for s in stages}
    for _ in range(steps):
        flush_l2(flush)
        torch.cuda._sleep(HOLD_CYCLES)
        ev = {s: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for s in stages} if per_stage else {}
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        wb.run_step(ev)
        e1.record()
        torch.cuda.synchronize()
        step_ms.append(e0.elapsed_time(e1))
        for s, (a, b) in ev.items():
            try:
                stage_ms[s].append(a.elapsed_time(b))
            except (RuntimeError, ValueError):   # a stage this workload does not run
                pass
    if clk is not None:
        clk.mark_end()
    return step_ms, {s: (sum(v) / len(v) if v else 0.0) for s, v in stage_ms.items()}


def read_floor(nbytes, flush, dev, reps=10):
    """Device time of a plain contiguous read of nbytes (a torch sum over a bf16 buffer, L2
    flushed first): the shortest time any kernel needs to stream that many bytes once on this
    GPU, launch, ramp-up and tail included.  A reference for the gathered-KV attention of the
    same size, not part of the method."""
    buf = torch.ones(max(nbytes // 2, 1), dtype=torch.bfloat16, device=dev)
    best = None
    for _ in range(reps + 3):
        flush_l2(flush)
        torch.cuda._sleep(HOLD_CYCLES)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        buf.sum(dtype=torch.float32)
        b.record()
        torch.cuda.synchronize()
        t = a.elapsed_time(b)
        best = t if best is None else min(best, t)
    del buf
    return best


def gather_ceiling(wb, flush, reps=10):
    """Device time of sfa_gather_kv_bandwidth on the step's own kept lists (L2 flushed before
    each rep, as before the timed steps): the K/V rows the attention gathers, moved into shared
    memory with nothing computed -- the attention's data-movement ceiling on these lists."""
    w, st, c = wb.w, wb.step, wb.case
    if w.dkq not in (576, 512) or wb.kv != "bf16" or wb.paged or st.dense:
        return None
    chk = torch.zeros(1, dtype=torch.int32, device=wb.dev)
    ts = []
    for r in range(reps + 2):
        flush_l2(flush)
        torch.cuda._sleep(HOLD_CYCLES)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        B.sfa_gather_kv_bandwidth(c["K"], c["V"], c["q_seq"], c["q_pos"], st.blk_idx, st.n_sel,
                                  st.top_k, w.compress_ratio, w.dkq, w.dv, chk,
                                  dev_status=st.status)
        e1.record()
        torch.cuda.synchronize()
        if r >= 2:
            ts.append(e0.elapsed_time(e1))
    return sum(ts) / len(ts)


def measure_e2e(wb, steps, warmup):
    """Same step through the public API with host inputs: each step copies this step's query
    inputs and new cache rows from pinned host memory, runs, and has O in host memory at its
    end.  The query inputs travel in one pinned host arena mirrored by one device arena, and
    the new cache rows go from the same host arena straight into their cache slots, in one copy
    kernel reading the pinned host memory (sfa_copy_cache_rows_multi).  A large Q (prefill:
    9.4 MB at 512 queries) goes instead by the copy engine on a side stream, concurrently with
    the scoring and the selection, and the attention waits for it (prefill_512x8192 end to end
    425 -> 392 us); a decode step's 0.6 MB measured faster through the kernel (88.3 against
    90.1 us: the join costs more than the copy).  q8_0 caches quantize the new rows on the
    device first, and a paged cache places them into their cells.  The attention writes O into
    pinned host memory directly (SfaStep.set_output)."""
    c, w = wb.case, wb.w
    sl = slice(w.depth, w.n_tok)   # the step's new cache rows (positions depth .. n_tok - 1)
    new_rows = {n: t[:, sl] for n, t in wb.seq_rows.items()}   # bf16, from the host
    # paged: the new rows go to their cells (the page table is known before the step)
    new_cells = wb.cell_of[:, sl].reshape(-1).long() if wb.paged else None
    # new rows through the device: q8_0 caches quantize them there; a paged cache scatters them
    via_dev = wb.kv == "q8_0" or wb.paged
    staging = {}
    if wb.kv == "q8_0":
        for n in ("K", "V"):
            if n in new_rows:
                t = new_rows[n]
                rb = B.sfa_q8_0_row_bytes(t.shape[-1])
                staging[n] = torch.empty(t.shape[:-1] + (rb,), dtype=torch.uint8, device=t.device)
    names = ["Q", "q_idx", "w", "q_seq", "q_pos"]
    parts = {n: c[n] for n in names}
    parts.update({f"{n}_new": t for n, t in new_rows.items()})
    offs, total = {}, 0
    for n, t in parts.items():
        offs[n] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    n_dev = total if via_dev else offs[f"{next(iter(new_rows))}_new"]   # bytes the arena copies
    dev_arena = torch.empty(total, dtype=torch.uint8, device=c["Q"].device)
    host_arena = torch.empty(total, dtype=torch.uint8).pin_memory()
    dv, hv, saved = {}, {}, {n: c[n] for n in names}
    for n, t in parts.items():
        nbytes = t.numel() * t.element_size()
        hv[n] = host_arena[offs[n]:offs[n] + nbytes].view(t.dtype).view(t.shape)
        hv[n].copy_(t.cpu())
        dv[n] = dev_arena[offs[n]:offs[n] + nbytes].view(t.dtype).view(t.shape)
    for n in names:
        c[n] = dv[n]
    out = torch.empty(wb.step.O.shape, dtype=torch.float32).pin_memory()
    dev_O = wb.step.set_output(out)   # the attention writes O into host memory
    h2d = total
    d2h = out.numel() * out.element_size()

    # the arena starts with Q; a large one goes by the copy engine on a side stream
    n_q = offs["q_idx"] if offs["q_idx"] >= (4 << 20) else 0
    side = torch.cuda.Stream() if n_q else None

    def join_q():
        if side is not None:
            torch.cuda.current_stream().wait_stream(side)

    def one():
        if side is not None:
            side.wait_stream(torch.cuda.current_stream())   # the last step is done with Q
            with torch.cuda.stream(side):
                dev_arena[:n_q].copy_(host_arena[:n_q], non_blocking=True)
        copies = [(dev_arena[n_q:n_dev].view(1, -1), host_arena[n_q:n_dev].view(1, -1))]
        if not via_dev:   # host rows straight into the cache slots, in the same launch
            copies += [(c[n][:, sl], hv[f"{n}_new"]) for n in new_rows]
        B.sfa_copy_cache_rows_multi(copies)
        for n in new_rows:
            if not via_dev:
                continue
            src = dv[f"{n}_new"]
            if n in staging:
                stg = staging[n]
                B.sfa_quantize_kv_q8_0(src.view(src.shape[0], -1, src.shape[-1]),
                                       stg.view(stg.shape[0], -1, stg.shape[-1]))
                src = stg
            if new_cells is None:
                c[n][:, sl].copy_(src)
            else:
                c[n].index_copy_(0, new_cells, src.reshape((-1,) + tuple(c[n].shape[1:])))
        wb.run_step(before_attend=join_q)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1) / steps
    # the same step captured once as a CUDA graph (copies, launches), replayed
    graph = sfa.SfaStep.graphed(one)
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    # the host copy of O is the device result: the same bits
    wb.step.set_output(dev_O)
    wb.run_step()
    torch.cuda.synchronize()
    same = bool(torch.equal(out, dev_O.cpu()))
    c.update(saved)
    q_path = ("Q by the copy engine on a side stream, overlapping scores and selection"
              if side is not None else "Q with the other inputs, by the copy kernel")
    return e0.elapsed_time(e1) / steps, eager_ms, h2d, d2h, same, q_path


def oracle_sample(w, dev_case, n_queries, n_threads):
    """Host copies of a bounded sample (the first n_queries queries) for the CPU oracle."""
    import numpy as np

    qi = list(range(min(n_queries, w.n_q)))
    seqs = sorted({int(dev_case["q_seq"][i]) for i in qi})
    remap = {s: k for k, s in enumerate(seqs)}
    npf = lambda t: t.float().cpu().numpy()  # noqa: E731
    st = torch.tensor(seqs, device=dev_case["X"].device)
    X = npf(dev_case["X"].index_select(0, st))
    K = npf(dev_case["K"].index_select(0, st))
    V = None if dev_case["V"] is None else npf(dev_case["V"].index_select(0, st))
    sel = torch.tensor(qi, device=dev_case["X"].device)
    q = {n: dev_case[n].index_select(0, sel) for n in ["Q", "q_idx", "w", "q_pos", "q_seq"]}
    q_seq = np.array([remap[int(s)] for s in q["q_seq"].cpu()], np.int32)
    return dict(X=X, q_idx=npf(q["q_idx"]), w=npf(q["w"]), Q=npf(q["Q"]), K=K, V=V,
                q_seq=q_seq, q_pos=q["q_pos"].cpu().numpy().astype(np.int32)), len(qi)


def time_oracle(w, sample, n_q, n_threads, min_seconds=3.0, max_reps=50):
    import oracle
    oracle.build()
    reps, t0 = 0, time.perf_counter()
    while True:
        out = oracle.run(sample["X"], sample["q_idx"], sample["w"], sample["Q"], sample["K"],
                         sample["V"], sample["q_seq"], sample["q_pos"], cr=w.compress_ratio,
                         top_k=w.indexer_top_k, scale=w.scale, dv=w.dv, n_threads=n_threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    return n_q * reps / el, out["threads"], el


def job_throughput(local_ms_total, local_units, steps, dist=None, device="cpu"):
    """Whole-job throughput of weak-scaled replicas.  The job takes as long as its slowest
    rank (the timed totals reduce to their maximum) and processes the units of every rank
    (they sum).  Returns (units per second, milliseconds per step).  `dist` is
    torch.distributed when several ranks run (NCCL wants `device` on the GPU, gloo the CPU)."""
    ms = torch.tensor([float(local_ms_total)], dtype=torch.float64, device=device)
    units = torch.tensor([float(local_units)], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(ms, op=dist.ReduceOp.MAX)
        dist.all_reduce(units, op=dist.ReduceOp.SUM)
    ms_per_step = float(ms.item()) / steps
    return float(units.item()) / (ms_per_step / 1000.0), ms_per_step


def run_reference(args, w, rank, world):
    """--impl reference: the CPU oracle on the host cores, on bounded samples of w."""
    if rank != 0:
        return
    import numpy as np  # noqa: F401
    cores = os.cpu_count() or 1
    dev = torch.device("cuda:0") if torch.cuda.is_available() else torch.device("cpu")
    case = sfa.make_case(w, device=dev)
    sample, nq = oracle_sample(w, case, min(cores, w.n_q), cores)
    del case
    vals, used = [], 1
    for _ in range(args.warmup):
        time_oracle(w, sample, nq, cores, min_seconds=0.0, max_reps=1)
    t_all = time.perf_counter()
    for _ in range(args.steps):
        v, used, _ = time_oracle(w, sample, nq, cores, min_seconds=0.0, max_reps=1)
        vals.append(v)
    el = time.perf_counter() - t_all
    value = nq * args.steps / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "queries_per_step_sample": nq},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                             "sample": f"first {nq} of {w.n_q} queries of {w.name}, whole "
                                       "method (pool, score, sort, mask, attend) per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(sfa.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-second", action="store_true", help="skip the pp2048 companion line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--exact", action="store_true",
                    help="decode: exact scores + select instead of the bounded selection")
    ap.add_argument("--bounded", action="store_true",
                    help="decode: the bounded selection even below its default size (captures)")
    ap.add_argument("--bound-pass", default=None, choices=["i8", "hi"],
                    help="the bounded selection's bound pass (default: i8 up to a budget of 1024)")
    ap.add_argument("--seqs", type=int, default=0,
                    help="override the number of sequences (smaller runs for ncu captures)")
    ap.add_argument("--paged", action="store_true",
                    help="time the paged cache layout (shuffled 64-cell pages) as the main line")
    ap.add_argument("--no-paged", action="store_true", help="skip the paged companion line")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "q8_0"],
                    help="KV cache type of the main line (q8_0: quantized rows)")
    ap.add_argument("--no-q8", action="store_true", help="skip the q8_0-cache companion line")
    ap.add_argument("--no-window", action="store_true",
                    help="skip the dense-window + sparse companion line (decode workloads)")
    ap.add_argument("--depth", type=int, default=0,
                    help="override the cache depth (smaller runs for ncu captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.exact and args.bounded:
        ap.error("--exact and --bounded exclude each other")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = sfa.WORKLOADS[args.workload]
    if args.seqs:
        w = w.with_(n_seq=args.seqs, name=f"{w.name}[seqs={args.seqs}]")
    if args.depth:
        w = w.with_(depth=args.depth, name=f"{w.name}[depth={args.depth}]")
    if args.impl == "reference":
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
        run_reference(args, w, rank, world)
        return

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        dist.barrier()
        __graft_entry__.build()
    hbm_peak, tf_peak, peak_kind = peaks()
    flush = (torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev),
             torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.float32, device=dev))

    sel_mode = False if args.exact else (True if args.bounded else None)
    wb = Workbench(w, dev, bounded=sel_mode, paged=args.paged, kv=args.kv,
                   bound_pass=args.bound_pass)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # the timed steps run back to back with no event between their kernels (an event
        # there would hold each kernel until the one before it has fully drained); the
        # per-stage split comes from a separate, shorter pass with events between stages
        step_ms, _ = measure(wb, args.steps, args.warmup, flush, per_stage=False, clk=clk)
        _, stage_ms = measure(wb, max(3, args.steps // 2), 3, flush, per_stage=True)
        value, ms_per_step = job_throughput(sum(step_ms), w.n_q, args.steps, dist, dev)
    torch.cuda.synchronize()
    status = B.sfa_read_device_status(wb.step.status)
    n_q_total = w.n_q * world

    n_sel = wb.step.n_sel.cpu()
    tail = [(int(p) + 1) % w.compress_ratio for p in wb.case["q_pos"].cpu()]
    attended = [int(n) * w.compress_ratio + t for n, t in zip(n_sel, tail)] if not wb.step.dense \
        else [int(p) + 1 for p in wb.case["q_pos"].cpu()]
    alg = algorithmic(w, attended, wb.step.bound_pass, kv=args.kv)
    kernels = {}
    for name, ms in stage_ms.items():
        if ms <= 0 or (name == "pool" and wb.new_blocks[1] <= wb.new_blocks[0]):
            continue
        if name in ("scores", "topk") and wb.step.dense:
            continue
        k = {"ms": ms}
        if name == "scores":
            k.update(bound="hbm", bytes=alg["kbar_bytes"] + alg["score_bytes"])
        elif name == "attend":
            k.update(bound="hbm" if w.kind == "decode" else "tensor", bytes=alg["gathered_kv_bytes"],
                     flops=alg["attend_flops"])
        elif name == "topk":
            k.update(bound="hbm", bytes=alg["score_bytes"])
        elif name == "pool":
            nb = wb.new_blocks[1] - wb.new_blocks[0]
            k.update(bound="hbm", bytes=w.n_seq * nb * (w.compress_ratio * 2 + 4) * w.d_idx)
        if "bytes" in k:
            k["GBps"] = k["bytes"] / (ms * 1e6)
            k["hbm_frac"] = k["GBps"] / hbm_peak
        if "flops" in k:
            k["TFLOPs"] = k["flops"] / (ms * 1e9)
            k["tensor_frac"] = k["TFLOPs"] / tf_peak
            k["bound"] = "tensor" if k["tensor_frac"] > k.get("hbm_frac", 0.0) else "hbm"
        kernels[name] = k
    dom = max(kernels, key=lambda n: kernels[n]["ms"])
    dk = kernels[dom]
    src = {"scores": "scores_i8.cu" if wb.step.bound_pass == "i8" else "scores.cu",
           "attend": "attend.cu", "topk": "topk.cu", "pool": "pool.cu"}[dom]
    # the kernel's bound is the resource it uses the larger fraction of
    if dk.get("tensor_frac", 0.0) > dk.get("hbm_frac", 0.0):
        roof = {"bound": "tensor", "achieved": dk["TFLOPs"], "peak": tf_peak, "unit": "TFLOP/s",
                "frac": dk["TFLOPs"] / tf_peak}
    else:
        roof = {"bound": "hbm", "achieved": dk["GBps"], "peak": hbm_peak, "unit": "GB/s",
                "frac": dk["GBps"] / hbm_peak}
    roof["kernel"] = dom
    roof["peak_source"] = f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured" \
        else "fallback"
    roof["traffic"] = recorded_traffic(dom, w.name, src)
    roof["source"] = src

    e2e_ms, e2e_eager_ms, h2d, d2h, e2e_same, q_path = measure_e2e(wb, max(3, args.steps // 2), 3)
    floor = None
    if "attend" in kernels and w.kind == "decode":
        fb = kernels["attend"]["bytes"]
        fms = read_floor(fb, flush, dev)
        floor = {"bytes": fb, "ms": fms, "GBps": fb / (fms * 1e6), "hbm_frac": fb / (fms * 1e6) / hbm_peak,
                 "attend_over_floor": kernels["attend"]["ms"] / fms,
                 "what": "plain contiguous read of the gathered-KV byte count (torch sum), L2 flushed"}
    gms = gather_ceiling(wb, flush) if "attend" in kernels else None
    gather = None
    if gms:
        gb = kernels["attend"]["bytes"]
        gather = {"ms": gms, "GBps": gb / (gms * 1e6), "hbm_frac": gb / (gms * 1e6) / hbm_peak,
                  "attend_over_gather": kernels["attend"]["ms"] / gms,
                  "what": "sfa_gather_kv_bandwidth on the step's kept lists: the attended K/V "
                          "rows moved into shared memory (one bulk copy per 4-row run, four "
                          "issuing warps per SM), nothing computed; L2 flushed"}
    launches = wb.launches_per_step() * args.steps

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if args.kv == "bf16" else "f16 (q8_0 KV)",
            "data": "synthetic (seeded N(0,1) K/Q/index keys, U(0,1) head weights)",
            "config": {"workload": w.name, "kind": w.kind, "n_seq": w.n_seq,
                       "queries_per_step": w.n_q, "depth": w.depth, "h_q": w.h_q,
                       "h_kv": w.h_kv, "dkq": w.dkq, "dv": w.dv, "v_is_k": w.v_is_k,
                       "h_idx": w.h_idx, "d_idx": w.d_idx, "compress_ratio": w.compress_ratio,
                       "indexer_top_k": w.indexer_top_k,
                       "selection": (f"bounded ({wb.step.bound_pass} bound pass)"
                                     if wb.step.bounded else "exact"),
                       "cache_layout": PAGED_LAYOUT if wb.paged else "contiguous per sequence",
                       "kv_cache": Q8_CACHE if args.kv == "q8_0" else "bf16",
                       "l2": "flushed before every timed "
                       "step outside the timed events (512 MB written, then 256 MB of another "
                       "buffer read)"},
            "gathered_kv_GBps": kernels.get("attend", {}).get("GBps"),
            "gathered_kv_read_floor": floor,
            "gather_ceiling": gather,
            "gathered_kv_hbm_frac": kernels.get("attend", {}).get("hbm_frac"),
            "roofline": roof, "kernels": kernels,
            "e2e": {"value": n_q_total / (e2e_ms / 1000.0), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "launch": "one CUDA graph per step (SfaStep.graphed)",
                    "eager_value": n_q_total / (e2e_eager_ms / 1000.0),
                    "output": "O written by the attention into pinned host memory",
                    "inputs": q_path, "host_O_equals_device_O": e2e_same},
            "gpu_launches": launches, "clocks": clk.summary(), "device_status": status}
    if wb.step.bounded:   # candidates per query the bounds could not rule out
        nb = max(wb.n_blk_max, 1)
        cn = wb.step.refine_ws.view(torch.int32)[2 * w.n_q * nb: 2 * w.n_q * nb + w.n_q].cpu()
        cn = [int(x) for x in cn if int(x) >= 0]
        line["bounded_selection"] = {"candidates_per_query_mean": (sum(cn) / len(cn)) if cn else 0,
                                     "candidates_per_query_max": max(cn) if cn else 0}
    wb_sel = (wb.step.n_sel.clone(), wb.step.O.clone(), wb.step.blk_idx.clone())
    del wb
    torch.cuda.empty_cache()

    if not args.no_paged and not args.paged and rank == 0 and world == 1:
        # the same workload on a paged cache: the pool and the attention read through the map
        wbp = Workbench(w, dev, bounded=sel_mode, paged=True, kv=args.kv)
        sp, _ = measure(wbp, max(3, args.steps // 2), 3, flush, per_stage=False)
        _, stp = measure(wbp, 3, 3, flush, per_stage=True)
        msp = sum(sp) / len(sp)
        same = bool(torch.equal(wbp.step.n_sel, wb_sel[0]) and torch.equal(wbp.step.O, wb_sel[1]))
        line["paged"] = {"cache_layout": PAGED_LAYOUT, "value": w.n_q / (msp / 1000.0),
                         "unit": "tokens/s", "ms_per_step": msp, "stage_ms": stp,
                         "same_output_as_contiguous": same,
                         "device_status": B.sfa_read_device_status(wbp.step.status)}
        del wbp
        torch.cuda.empty_cache()

    if not args.no_q8 and args.kv == "bf16" and rank == 0 and world == 1:
        # the same workload on q8_0 K/V caches: the attention gathers the quantized rows
        wbq = Workbench(w, dev, bounded=sel_mode, paged=args.paged, kv="q8_0")
        sq, _ = measure(wbq, max(3, args.steps // 2), 3, flush, per_stage=False)
        _, stq = measure(wbq, 3, 3, flush, per_stage=True)
        msq = sum(sq) / len(sq)
        aq = algorithmic(w, attended, wbq.step.bound_pass, kv="q8_0")
        same = bool(torch.equal(wbq.step.n_sel, wb_sel[0]) and torch.equal(wbq.step.blk_idx, wb_sel[2]))
        ref = wb_sel[1]
        dev_rel = ((wbq.step.O - ref).abs().amax(-1) / ref.abs().amax(-1).clamp_min(1e-30)).max()
        att_ms = stq.get("attend", 0.0)
        line["kv_q8_0"] = {"kv_cache": Q8_CACHE, "value": w.n_q / (msq / 1000.0),
                           "unit": "tokens/s", "ms_per_step": msq, "stage_ms": stq,
                           "gathered_kv_bytes": aq["gathered_kv_bytes"],
                           "gathered_kv_GBps": aq["gathered_kv_bytes"] / (att_ms * 1e6) if att_ms else None,
                           "same_selection_as_bf16": same,
                           "max_rel_diff_vs_bf16_cache": float(dev_rel),
                           "device_status": B.sfa_read_device_status(wbq.step.status)}
        del wbq
        torch.cuda.empty_cache()

    if not args.no_window and args.kv == "bf16" and not args.paged and w.kind == "decode" \
            and rank == 0 and world == 1:
        # the dense window of the WINDOW most recent positions beside the kept blocks, in one
        # pass and as the two parts combined by their log-sum-exp
        res, outs = {}, {}
        for mode in ("single", "split"):
            wbw = Workbench(w, dev, bounded=sel_mode, window=WINDOW,
                            window_mode=mode)
            sw, _ = measure(wbw, max(3, args.steps // 2), 3, flush, per_stage=False)
            _, stw = measure(wbw, 3, 3, flush, per_stage=True)
            msw = sum(sw) / len(sw)
            res[mode] = {"value": w.n_q / (msw / 1000.0), "unit": "tokens/s", "ms_per_step": msw,
                         "stage_ms": stw,
                         "device_status": B.sfa_read_device_status(wbw.step.status)}
            outs[mode] = wbw.step.O.clone()
            if mode == "single":   # the attended cells: kept tokens before the suffix + suffix
                sel = wbw.step.blk_idx.cpu()
                ns = wbw.step.n_sel.cpu()
                cells = 0
                for i, p in enumerate(wbw.case["q_pos"].cpu().tolist()):
                    s0 = min(((p + 1) // w.compress_ratio) * w.compress_ratio,
                             max(0, p - WINDOW + 1))
                    kept = sel[i, : int(ns[i])].long() * w.compress_ratio
                    kept_cells = int(((s0 - kept).clamp(0, w.compress_ratio)).sum())
                    cells += kept_cells + (p + 1 - s0)
                row_b = w.h_kv * (w.dkq + (0 if w.v_is_k else w.dv)) * 2
                res["gathered_kv_bytes"] = cells * row_b
            del wbw
            torch.cuda.empty_cache()
        a, b = outs["single"], outs["split"]
        res["max_rel_diff_single_vs_split"] = float(
            ((a - b).abs().amax(-1) / a.abs().amax(-1).clamp_min(1e-30)).max())
        for mode in ("single", "split"):
            att = res[mode]["stage_ms"].get("attend", 0.0)
            res[mode]["gathered_kv_GBps"] = res["gathered_kv_bytes"] / (att * 1e6) if att else None
        line["window"] = {"window": WINDOW,
                          "what": "attention over the kept blocks, the tail and the WINDOW most "
                                  "recent positions: one pass (single) vs the kept part and the "
                                  "window part apart + sfa_combine_attention (split)", **res}
        del outs

    if not args.no_second and rank == 0 and world == 1:
        w2 = sfa.WORKLOADS[SECOND_WORKLOAD]
        wb2 = Workbench(w2, dev)
        s2, _ = measure(wb2, max(3, args.steps // 4), 3, flush, per_stage=False)
        _, st2 = measure(wb2, 3, 3, flush, per_stage=True)
        ms2 = sum(s2) / len(s2)
        n_sel2 = wb2.step.n_sel.cpu()
        att2 = [int(n) * w2.compress_ratio + (int(p) + 1) % w2.compress_ratio
                for n, p in zip(n_sel2, wb2.case["q_pos"].cpu())]
        a2 = algorithmic(w2, att2, wb2.step.bound_pass)
        g2 = gather_ceiling(wb2, flush, reps=5)
        line["pp2048"] = {
            "gather_ceiling": None if not g2 else {
                "ms": g2, "GBps": a2["gathered_kv_bytes"] / (g2 * 1e6),
                "attend_over_gather": st2["attend"] / g2,
                "what": "sfa_gather_kv_bandwidth on the step's kept lists (mostly L2 -> shared "
                        "memory; L2 flushed before each rep)"},
            "workload": w2.name, "value": w2.n_q / (ms2 / 1000.0), "unit": "tokens/s",
            "ms_per_step": ms2, "stage_ms": st2,
            "attend_TFLOPs": a2["attend_flops"] / (st2["attend"] * 1e9),
            "attend_tensor_frac": a2["attend_flops"] / (st2["attend"] * 1e9) / tf_peak,
            "scores_TFLOPs": a2["score_flops"] / (st2["scores"] * 1e9),
            "scores_tensor_frac": a2["score_flops"] / (st2["scores"] * 1e9) / tf_peak}
        del wb2
        torch.cuda.empty_cache()

    if rank == 0 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        case = sfa.make_case(w, device=dev)
        sample, nq = oracle_sample(w, case, min(cores, w.n_q), cores)
        del case
        v, used, el = time_oracle(w, sample, nq, cores)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": used, "kind": "oracle",
                                "sample": f"first {nq} of {w.n_q} queries of {w.name} "
                                          f"(whole method per query), repeated for {el:.1f} s"}
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
