"""Benchmark: paged-attention KV GB/s (fraction of HBM peak) and verified tokens/s.

One step = one pass of the decode hot path over the Llama3-8B-shaped batch
(64 sequences, 32 q / 8 KV heads, head_dim 128, contexts U[512,1024] in a
64k-token pool of 256-token pages): kv_append of the 64 new tokens' K/V
through the block tables, then paged_attn (split-K page streaming + combine).
`value` counts the step's algorithmic bytes (paged_attn: each distinct cached
K/V token once, plus q, out, tables and lengths; kv_append: the new rows read
and written) over the step's device time, the two calls launched back to back
as a decode loop runs them; inputs are resident in HBM and L2 is flushed
between steps. The roofline block times paged_attn on its own. A second block reports
the speculative-verification step (16 sequences, q_len 6 causal, then greedy
accept over [16, 6, 128256] fp32 logits) as verified tokens/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own independently seeded batch on
its own GPU (no collective on the data path; weak scaling) and rank 0 prints
one JSON line with the max-over-ranks time. `--impl reference` times the CPU
fp64 oracle on a bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "paged-attn KV GB/s (frac of HBM peak); verified tokens/s at 1 GB300"
DECODE_CFG = 1   # Llama3-8B-shaped decode batch
VERIFY_CFG = 3   # speculative verification batch
DEDUP_CFG = 2    # 100 sequences sharing a 16-page prefix
TINY_CFG = 0     # 4 sequences, 8 q / 2 KV heads
FRAG_CFG = 4     # 8 x 8192-token contexts on a churned pool, q_len 1 or 6
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def attention_flops(w: wl.Workload) -> int:
    """Algorithmic FLOPs of one paged_attn call: 2 d per visible key for
    q.k and 2 d for p.v, over every (new token, query head) row."""
    n, T = w.q_lens.astype(np.int64), w.seq_lens.astype(np.int64)
    visible = sum(int((T[b] - n[b]) * n[b] + n[b] * (n[b] + 1) // 2) for b in range(len(n)))
    return 4 * w.head_dim * w.num_q_heads * visible


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def counted_bytes(w: wl.Workload, with_logits=False) -> int:
    """Algorithmic bytes of one paged_attn call: distinct K/V tokens once,
    q and out (bf16), block table, seq_lens and q_lens (+ logits)."""
    n = w.unique_kv_bytes() + 2 * w.q.nbytes + w.block_table.nbytes + w.seq_lens.nbytes \
        + w.q_lens.nbytes
    if with_logits and w.logits is not None:
        n += w.logits.nbytes
    return int(n)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.2)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i] == "Active"})
        loaded = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------- our arm
class GpuBatch:
    """A workload resident on the GPU plus everything one step needs."""

    def __init__(self, w: wl.Workload, device, use_plan=False):
        import torch

        import speculative_decode_gb300 as sa
        self.w, self.sa, self.torch = w, sa, torch

        def T(a):
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                a = a.view(np.int16)
            return torch.from_numpy(a).to(device)

        self.T = T
        self.dims = sa.dims_for(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.num_pages,
                                w.max_pages_per_seq, w.total_q, int(w.q_lens.max()))
        self.kp, self.vp = T(w.k_pages), T(w.v_pages)
        self.bt, self.sl, self.ql = T(w.block_table), T(w.seq_lens), T(w.q_lens)
        self.q, self.k_new, self.v_new = T(w.q), T(w.k_new), T(w.v_new)
        self.out = torch.zeros_like(self.q)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.plan = sa.Plan(self.dims, w.block_table, w.seq_lens, w.q_lens) if use_plan else None
        self.ws = torch.zeros(sa.paged_attn_workspace_size(self.dims, self.plan), dtype=torch.uint8,
                              device=device)
        self.kernels_attn = sa.paged_attn_kernel_count(self.dims, self.plan)
        self.verify = w.logits is not None
        if self.verify:
            B, k1, V = w.logits.shape
            self.logits, self.cand, self.ncand = T(w.logits), T(w.candidates), T(w.n_cand)
            self.window0 = T(w.window)
            self.window = self.window0.clone()
            self.acc = torch.zeros(B, dtype=torch.int32, device=device)
            self.nxt = torch.zeros_like(self.acc)
            self.vws = torch.zeros(sa.spec_verify_workspace_size(B, k1 - 1, V),
                                   dtype=torch.uint8, device=device)

    def append(self):
        self.sa.kv_append(self.dims, self.k_new, self.v_new, self.kp, self.vp, self.bt, self.sl,
                          self.ql, err_flag=self.err)

    def attend(self):
        self.sa.paged_attn(self.dims, self.q, self.kp, self.vp, self.bt, self.sl, self.ql,
                           self.w.scale, self.out, self.ws, plan=self.plan, err_flag=self.err)

    def accept(self):
        self.sa.spec_verify_greedy(self.logits, self.cand, self.ncand, self.acc, self.nxt,
                                   self.vws, window=self.window, err_flag=self.err)

    def prepare_defrag(self):
        """Compaction plan of this batch's pool (host, not timed); its moves on the device."""
        new, moves, n_live = self.sa.defrag_moves(self.dims, self.w.block_table, self.w.seq_lens)
        self.moves = self.T(moves.reshape(-1, 2))
        self.n_moves, self.n_live = len(moves), n_live
        return new

    def defrag(self):
        # the moves copy pages (sources stay), so repeating them copies the same bytes again
        self.sa.defrag_apply(self.dims, self.kp, self.vp, self.moves, self.n_moves, err_flag=self.err)

    def launches_per_step(self):
        return 1 + self.kernels_attn + (1 if self.verify else 0)


def timed_steps(batch: GpuBatch, steps: int, warmup: int, flush, parts):
    """Run warmup + steps; per step record device time of each named part with
    CUDA events on the launching stream, flushing L2 before every step."""
    torch = batch.torch
    stream = torch.cuda.current_stream()
    fns = {"append": batch.append, "attend": batch.attend, "accept": batch.accept, "defrag": batch.defrag}
    for _ in range(warmup):
        flush()
        for p in parts:
            fns[p]()
    torch.cuda.synchronize()
    if int(batch.err.item()) != 0:
        raise SystemExit(f"device error flag {int(batch.err.item())} after warm-up; not timing")
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in parts] for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(steps):
        flush()
        for i, p in enumerate(parts):
            ev[s][i][0].record(stream)
            fns[p]()
            ev[s][i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - t0
    per_part = {p: [ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(steps)]
                for i, p in enumerate(parts)}
    return per_part, wall


# DRAM bytes (read + written) of one decode-batch launch of the attention
# kernel (stream_attn_kernel<4, 16>), from one ncu capture of this build
# (dram__bytes_read.sum 200.367616 MB + dram__bytes_write.sum 3.497984 MB);
# None whenever the kernel changes until it is captured again.
DECODE_TRAFFIC_BYTES = 203865600


def timed_sequence(batch: GpuBatch, steps: int, warmup: int, flush, parts):
    """Run warmup + steps of the named parts launched back to back (no event
    between them, so a kernel may start while its predecessor finishes); per
    step one pair of CUDA events around all of them, L2 flushed before."""
    torch = batch.torch
    stream = torch.cuda.current_stream()
    fns = {"append": batch.append, "attend": batch.attend, "accept": batch.accept, "defrag": batch.defrag}
    for _ in range(warmup):
        flush()
        for p in parts:
            fns[p]()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    for s in range(steps):
        flush()
        ev[s][0].record(stream)
        for p in parts:
            fns[p]()
        ev[s][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    return [a.elapsed_time(b) for a, b in ev]


def append_bytes(w: wl.Workload) -> int:
    """kv_append's algorithmic bytes: the new K and V rows read, then written."""
    return 2 * 2 * int(w.q_lens.sum()) * w.num_kv_heads * w.head_dim * 2


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(cfg: int, rank: int) -> int:
    """Seed of rank's batch of workload cfg: rank 0 uses the workload's own
    seed, every other rank an independent batch of the same shapes."""
    return 1000 + cfg + 1 + 7919 * rank


def quant_block(batch: GpuBatch, w: wl.Workload, dev, steps: int, warmup: int, flush, bits: int):
    """paged_attn over int8 (bits 8) or int4 (bits 4) pages for the decode
    batch: codes uniform over [-127, 127] (int8) or [-7, 7] (int4, as nibbles
    1..15) and per-row scales near those of N(0,1) rows (synthetic, seeded);
    counted bytes = distinct cached tokens x heads x (128 codes of `bits` bits
    + 4-byte scale) x 2, plus q, out and the tables."""
    torch, sa = batch.torch, batch.sa
    rng = np.random.default_rng(2024 + bits)
    shape = w.k_pages.shape
    cmax = 127 if bits == 8 else 7
    if bits == 8:
        codes = lambda: rng.integers(-127, 128, size=shape, dtype=np.int8)
    else:
        codes = lambda: (rng.integers(1, 16, size=shape[:-1] + (64,), dtype=np.uint8)
                         | (rng.integers(1, 16, size=shape[:-1] + (64,), dtype=np.uint8) << 4))
    kc = torch.from_numpy(codes()).to(dev)
    vc = torch.from_numpy(codes()).to(dev)
    ks = torch.from_numpy((rng.uniform(2.5, 3.5, size=shape[:-1]) / cmax).astype(np.float32)).to(dev)
    vs = torch.from_numpy((rng.uniform(2.5, 3.5, size=shape[:-1]) / cmax).astype(np.float32)).to(dev)
    ws = torch.zeros(sa.paged_attn_workspace_size(batch.dims), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    attn = sa.paged_attn_q8 if bits == 8 else sa.paged_attn_q4

    def call():
        attn(batch.dims, batch.q, kc, vc, ks, vs, batch.bt, batch.sl, batch.ql, w.scale,
             batch.out, ws, err_flag=batch.err)

    for _ in range(warmup):
        flush()
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    for e0, e1 in ev:
        flush()
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    assert int(batch.err.item()) == 0, "device error flag set"
    t = max_over_ranks(statistics.median(a.elapsed_time(b) for a, b in ev))
    tokens_heads = sum(int(T) for T in w.seq_lens) * w.num_kv_heads
    q_bytes = (tokens_heads * (128 * bits // 8 + 4) * 2 + 2 * w.q.nbytes + w.block_table.nbytes
               + w.seq_lens.nbytes + w.q_lens.nbytes)
    return {"workload": w.name + (" int8 pages" if bits == 8 else " int4 pages"), "paged_attn_ms": round(t, 5),
            "counted_bytes": int(q_bytes), "GBps": round(q_bytes / (t * 1e-3) / 1e9, 1),
            "cached_tokens_per_s": round(sum(int(T) for T in w.seq_lens) / (t * 1e-3), 1)}


def e2e_steps(batch: GpuBatch, steps: int, warmup: int):
    """The same decode step through the public API with host buffers: every
    step copies its inputs host->device from pinned memory and reads the
    attention output back device->host; timed with events around all of it.
    The inputs (q, k_new, v_new, tables, lengths) sit in one pinned staging
    buffer and go over in one copy into one device buffer, of which the
    kernels read 256-byte-aligned views, as a serving loop would stage them."""
    torch = batch.torch
    stream = torch.cuda.current_stream()
    names = ["q", "k_new", "v_new", "bt", "sl", "ql"]
    srcs = [getattr(batch, n) for n in names]
    sizes = [t.numel() * t.element_size() for t in srcs]
    offs, total = [], 0
    for n in sizes:
        offs.append(total)
        total += (n + 255) // 256 * 256
    host_buf = torch.zeros(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=srcs[0].device)
    saved = {}
    for name, t, o, n in zip(names, srcs, offs, sizes):
        host_buf[o:o + n].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
        saved[name] = t
        setattr(batch, name, dev_buf[o:o + n].view(t.dtype).view(t.shape))
    out_host = torch.empty(batch.out.shape, dtype=batch.out.dtype).pin_memory()
    h2d = sum(sizes)
    d2h = out_host.numel() * out_host.element_size()

    def step():
        dev_buf.copy_(host_buf, non_blocking=True)
        batch.append()
        batch.attend()
        out_host.copy_(batch.out, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    for name, t in saved.items():
        setattr(batch, name, t)
    return e0.elapsed_time(e1) / steps, h2d, d2h


def run_ours(args):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    # a stream of our own (not the legacy default stream), on which the
    # combine pass can start as a programmatic dependent of the split kernel
    torch.cuda.set_stream(torch.cuda.Stream(device=torch.device("cuda", local)))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    barrier()
    dev = torch.device("cuda", local)

    # L2 flush before every timed step: write a buffer twice the L2 size, then
    # read another one of the same size. The write evicts everything; the read
    # leaves the L2 holding clean lines of unrelated data, so the timed kernels
    # neither find their inputs cached nor pay for writing back the flush's own
    # dirty lines.
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nflush = max(2 * l2, 1 << 20) // 8 * 8
    flush_w = torch.empty(nflush, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(nflush, dtype=torch.uint8, device=dev)

    def flush():
        flush_w.zero_()
        flush_r.view(torch.int64).sum()

    # ---- headline: decode step on the Llama3-8B-shaped batch
    w = wl.config(DECODE_CFG, seed=rank_seed(DECODE_CFG, rank))
    batch = GpuBatch(w, dev)
    cbytes = counted_bytes(w)
    sbytes = cbytes + append_bytes(w)
    with ClockSampler(local) as clk:
        # the step as a decode loop runs it: kv_append, then paged_attn, back to back
        steps_ms = timed_sequence(batch, args.steps, args.warmup, flush, ["append", "attend"])
        # each kernel call timed on its own (events between them) for the roofline
        parts, wall = timed_steps(batch, args.steps, args.warmup, flush, ["append", "attend"])
    clocks = clk.summary()
    t_attn = statistics.median(parts["attend"])      # ms
    t_step = statistics.median(steps_ms)
    t_attn_max = max_over_ranks(t_attn)
    # CUDA events on this GPU count in ticks of 2.048 us, so a median moves in
    # whole ticks; the roofline takes the average launch duration, the mean
    t_attn_mean_max = max_over_ranks(statistics.mean(parts["attend"]))
    t_step_max = max_over_ranks(t_step)
    t_append_max = max_over_ranks(statistics.median(parts["append"]))
    assert int(batch.err.item()) == 0, "device error flag set"

    e2e_ms, h2d, d2h = e2e_steps(batch, max(10, args.steps // 10), args.warmup)
    e2e_ms = max_over_ranks(e2e_ms)

    # ---- second block: speculative verification step
    wv = wl.config(VERIFY_CFG, seed=rank_seed(VERIFY_CFG, rank))
    vb = GpuBatch(wv, dev)
    vsteps = max(3, args.steps // 4)
    vparts, _ = timed_steps(vb, vsteps, args.warmup, flush, ["append", "attend", "accept"])
    tv_attn = max_over_ranks(statistics.median(vparts["attend"]))
    tv_acc = max_over_ranks(statistics.median(vparts["accept"]))
    tv_step = max_over_ranks(statistics.median(
        [a + b + c for a, b, c in zip(vparts["append"], vparts["attend"], vparts["accept"])]))
    torch.cuda.synchronize()
    emitted = int((vb.acc.cpu().numpy() + 1).sum())
    vq = int(wv.q_lens.sum())
    vbytes = counted_bytes(wv)

    # ---- third block: the dedup batch (100 sequences sharing a 4096-token
    # prefix), paged_attn with the shared-run plan and without it
    wd = wl.config(DEDUP_CFG, seed=rank_seed(DEDUP_CFG, rank))
    dsteps = max(3, args.steps // 4)
    dedup = {"workload": wd.name, "unique_bytes": counted_bytes(wd)}
    for label, use_plan in (("with_plan", True), ("without_plan", False)):
        db = GpuBatch(wd, dev, use_plan=use_plan)
        dparts, _ = timed_steps(db, dsteps, args.warmup, flush, ["attend"])
        t = max_over_ranks(statistics.median(dparts["attend"]))
        dedup[label] = {"paged_attn_ms": round(t, 5),
                        "GBps_unique": round(dedup["unique_bytes"] / (t * 1e-3) / 1e9, 1)}
        if use_plan:
            dedup["plan"] = db.plan.stats()
        del db

    # ---- fourth block: compaction of the spec-verify batch's fragmented pool
    # (512 pages, 8 KV heads): the host plan once, the page copies timed
    vb.prepare_defrag()
    fparts, _ = timed_steps(vb, vsteps, args.warmup, flush, ["defrag"])
    tf = max_over_ranks(statistics.median(fparts["defrag"]))
    moved = vb.n_moves * 2 * wv.num_kv_heads * wl.PAGE_SIZE * 128 * 2  # K and V bytes of the moved pages
    defrag = {"workload": f"{wv.name} pool ({wv.num_pages} pages)", "live_pages": vb.n_live,
              "moved_pages": vb.n_moves, "moved_bytes": moved, "ms": round(tf, 5),
              "GBps": round(2 * moved / (tf * 1e-3) / 1e9, 1),
              "counts": "bytes read + bytes written / device time of sa_defrag_apply"}
    del vb

    # ---- fifth block: chunked prefill through the pages (8 sequences append a
    # 512-token chunk after 3584 cached tokens; the tensor cores attend it)
    wp = wl.prefill_chunk(seed=1100 + rank)
    pb = GpuBatch(wp, dev)
    pparts, _ = timed_steps(pb, vsteps, args.warmup, flush, ["append", "attend"])
    tp = max_over_ranks(statistics.median(pparts["attend"]))
    tpa = max_over_ranks(statistics.median(pparts["append"]))
    pflops = attention_flops(wp)
    tpeak, tpeak_kind = bf16_peak()
    prefill = {"workload": wp.name, "paged_attn_ms": round(tp, 5), "kv_append_ms": round(tpa, 5),
               "flops": pflops, "TFLOPs": round(pflops / (tp * 1e-3) / 1e12, 1),
               "frac_of_bf16_peak": round(pflops / (tp * 1e-3) / 1e12 / tpeak, 4),
               "peak_source": f"{tpeak_kind} bf16_tflops",
               "tokens_per_s": round(world * int(wp.q_lens.sum()) / (tp * 1e-3), 1),
               "counts": "4 x 128 x visible keys per (new token, query head) row / paged_attn device time"}
    del pb

    # ---- the tiny decode batch and the fragmented long-context batch,
    # paged_attn only (KV bytes over device time, as for the headline)
    extra = {}
    for label, cfg in (("tiny", TINY_CFG), ("fragmented", FRAG_CFG)):
        we = wl.config(cfg, seed=rank_seed(cfg, rank))
        eb = GpuBatch(we, dev)
        eparts, _ = timed_steps(eb, vsteps, args.warmup, flush, ["attend"])
        t = max_over_ranks(statistics.median(eparts["attend"]))
        eby = counted_bytes(we)
        extra[label] = {"workload": we.name, "paged_attn_ms": round(t, 5), "bytes": eby,
                        "GBps": round(eby / (t * 1e-3) / 1e9, 1), "kernels": eb.kernels_attn}
        assert int(eb.err.item()) == 0, "device error flag set"
        del eb

    # ---- sixth block: the decode batch over int8 and int4 pages (synthetic
    # seeded codes and per-row scales of the same shapes), attention only
    q8 = quant_block(batch, w, dev, vsteps, args.warmup, flush, 8)
    q4 = quant_block(batch, w, dev, vsteps, args.warmup, flush, 4)
    q8["bf16_paged_attn_ms"] = q4["bf16_paged_attn_ms"] = round(t_attn_max, 5)

    peak, peak_kind = hbm_peak()
    achieved = cbytes / (t_attn_mean_max * 1e-3) / 1e9
    defrag["frac_of_hbm_peak"] = round(defrag["GBps"] / peak, 4)
    for v in extra.values():
        v["frac_of_hbm_peak"] = round(v["GBps"] / peak, 4)
    line = {
        "metric": METRIC,
        "value": round(world * sbytes / (t_step_max * 1e-3) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_step_max, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "accumulate": "f32",
        "data": "synthetic (seeded bf16 N(0,1) q/k/v, random non-contiguous block tables)",
        "config": {
            "workload": w.name,
            "seqs": w.num_seqs, "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
            "head_dim": 128, "page_size": 256, "pool_pages": w.num_pages,
            "ctx": "uniform[512,1024]", "q_len": 1,
            "step": "kv_append + paged_attn",
            "value_counts": "step algorithmic bytes (paged_attn: each distinct cached K/V token once "
                            "+ q + out + tables; kv_append: new K/V rows read and written) / step device "
                            "time (one event pair around kv_append + paged_attn launched back to back)",
            "l2": "flushed before every step: 2x L2 written, then 2x L2 of other data read",
            "timing": "median over the timed steps of each block's CUDA-event times (which tick in "
                      "2.048 us); the roofline block takes the mean",
            "parallelism": f"replicas x{world} (independent batches, no collective)",
        },
        "counted_bytes_per_step": sbytes,
        "paged_attn_bytes": cbytes,
        "paged_attn_ms": round(t_attn_max, 5),
        "paged_attn_ms_mean": round(t_attn_mean_max, 5),
        "kv_append_ms": round(t_append_max, 5),
        "frac_of_hbm_peak": round(cbytes / (t_attn_max * 1e-3) / 1e9 / peak, 4),
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": DECODE_TRAFFIC_BYTES,
            "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of stream_attn_kernel<4, 16>, "
                              "one capture of this build",
            "kernel": "paged_attn call (stream_attn_kernel<4, 16>, one launch)",
            "duration": "mean of the timed calls' CUDA-event times (events tick in 2.048 us)",
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s",
        },
        "verify": {
            "workload": wv.name,
            "query_tokens_per_s": round(world * vq / (tv_attn * 1e-3), 1),
            "emitted_tokens_per_s": round(world * emitted / ((tv_attn + tv_acc) * 1e-3), 1),
            "emitted_per_step": emitted,
            "paged_attn_ms": round(tv_attn, 5),
            "paged_attn_GBps": round(vbytes / (tv_attn * 1e-3) / 1e9, 1),
            "spec_verify_ms": round(tv_acc, 5),
            "spec_verify_GBps": round(wv.logits.nbytes / (tv_acc * 1e-3) / 1e9, 1),
            "step_ms": round(tv_step, 5),
            "note": "per attention layer: one layer's attention + one greedy accept",
        },
        "tiny": extra["tiny"],
        "fragmented": extra["fragmented"],
        "dedup": dedup,
        "defrag": defrag,
        "prefill": prefill,
        "q8": q8,
        "q4": q4,
        "e2e": {"value": round(world * sbytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_ms, 5)},
        "gpu_launches": int(args.steps * batch.launches_per_step()),
        "clocks": clocks,
    }
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(w) if (world == 1 and not args.no_cpu_baseline) else None
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------ oracle timing
def oracle_sample(w: wl.Workload, seqs):
    """Counted bytes of the attention of the listed sequences (all heads)."""
    sub = {}
    P = w.page_size
    for b in seqs:
        T = int(w.seq_lens[b])
        for j in range(-(-T // P)):
            pid = int(w.block_table[b, j])
            sub[pid] = max(sub.get(pid, 0), min(P, T - j * P))
    kv = sum(sub.values()) * w.num_kv_heads * w.head_dim * 4
    qrows = int(sum(w.q_lens[b] for b in seqs))
    return kv + 2 * qrows * w.num_q_heads * w.head_dim * 2


def time_oracle_sequences(w: wl.Workload, seqs, n_threads=0):
    import oracle
    qstart = np.concatenate([[0], np.cumsum(w.q_lens)])
    toks, heads = [], []
    for b in seqs:
        for i in range(int(w.q_lens[b])):
            for h in range(w.num_q_heads):
                toks.append(int(qstart[b]) + i)
                heads.append(h)
    t0 = time.perf_counter()
    oracle.attention_rows(w.q, w.k_pages, w.v_pages, w.block_table, w.seq_lens, w.q_lens, w.scale,
                          toks, heads, n_threads=n_threads)
    return time.perf_counter() - t0


def cpu_baseline(w: wl.Workload):
    import oracle
    oracle.build()
    cores = oracle.num_threads()
    seqs = list(range(w.num_seqs))
    time_oracle_sequences(w, seqs[:2])                      # warm (library load, caches)
    reps, t = 0, 0.0
    while reps < 3 and t < 15.0:
        t += time_oracle_sequences(w, seqs)
        reps += 1
    nbytes = oracle_sample(w, seqs) * reps
    one = time_oracle_sequences(w, seqs[:4], n_threads=1)
    return {"value": round(nbytes / t / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"full decode batch ({w.num_seqs} seqs x {w.num_q_heads} heads) x {reps}, "
                      "attention only, fp64",
            "value_1core": round(oracle_sample(w, seqs[:4]) / one / 1e9, 5)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    cores = oracle.num_threads()
    w = wl.config(DECODE_CFG)
    # bounded sample per step: one sequence of the decode batch (all its heads)
    for s in range(args.warmup):
        time_oracle_sequences(w, [s % w.num_seqs])
    times, nbytes = [], 0
    t_start = time.perf_counter()
    for s in range(args.steps):
        b = s % w.num_seqs
        times.append(time_oracle_sequences(w, [b]))
        nbytes += oracle_sample(w, [b])
        if time.perf_counter() - t_start > 120.0:        # keep the run within minutes
            break
    t = sum(times)
    value = nbytes / t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": len(times),
        "warmup": args.warmup, "ms_per_step": round(1e3 * t / len(times), 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded decode batch)",
        "config": {"workload": w.name, "step": "oracle attention of one sequence (all heads)"},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": "one sequence of the decode batch per step"},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
