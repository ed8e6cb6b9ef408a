#!/usr/bin/env python
"""Benchmark of the attention-scored sparse KV path on GB300.

Default workload (the headline metric "KV tokens scored+compacted/s"): the
Llama-3.1-8B-shaped layer at the end of prefill -- 4 sequences x 32,768
tokens, 32 query / 8 KV heads, d=128, bf16, SnapKV window of 64 queries,
pooling 7, budget 2048 per KV head.  One step = the whole path on one batch:
window scoring -> pooled top-k -> compaction into fresh pages and decode
attention over the retained entries (the two side by side on two streams,
as the pipeline runs them).  Inputs are synthetic (seeded N(0,1) with
1% of keys offset by 3 sigma along a random direction) and resident in HBM;
the KV cache (570 MB) is larger than L2, so no flush is needed between steps.
Before each step the cache's metadata (block table, slot map, lengths, free
list, refcounts) is restored so that every step compresses the same input;
the restore sits outside the device-timed region (it does not touch K/V: the
compaction writes only fresh pages).

Other workloads (--workload): snapkv_tiny, quest_decode, h2o_decode,
kara_prune, kara_schedule -- each prints its own line with its own dominant
kernel.

--impl reference times the CPU oracle (the slow, plain fp64 reference) on a
bounded sample of the same workload on the host cores.
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
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        out = {}
        for k in FALLBACK_PEAKS:
            v = d.get(k)
            if isinstance(v, dict):
                v = v.get("value")
            out[k] = float(v) if v is not None else None
        if all(v is not None for v in out.values()):
            return out, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline / reference arm)
# ---------------------------------------------------------------------------


def oracle_prepare(workload: str, groups: int):
    """Builds a bounded sample of the workload for the oracle; returns a
    function that runs the oracle once on a fresh copy of it and reports
    (token-equivalents processed, seconds, description)."""
    import numpy as np
    import se_workloads as W
    from oracle import attention as oattn
    from oracle import cache as ocache
    from oracle import pipelines as opipe
    from oracle import quest as oquest
    from oracle import scoring as oscore
    from oracle import selection as osel

    if workload in ("snapkv_llama8b", "snapkv_tiny"):
        full = W.WORKLOADS[workload]()
        shape = W.WORKLOADS[workload](B=1)
        inp = W.snapkv_inputs(shape, "cpu")
        c0 = ocache.from_tensors(inp["cache"])
        heads = list(range(min(groups, shape.Hkv)))
        q_pos = inp["q_pos"].numpy()
        q_dec = opipe.to_f64(inp["q_dec"])
        desc = (f"1 of {full.B} sequences, {len(heads)} of {shape.Hkv} KV heads ({shape.ctx} "
                "tokens): score + pool/top-k + compact + decode")

        def run():
            c = c0.copy()
            t0 = time.perf_counter()
            s = oscore.score_window(c, inp["q_win"], q_pos, [0], [shape.ctx], [0],
                                    [shape.scored], True, groups=[(0, h) for h in heads])
            keep = [[osel.topk_keep(s[(0, h)], 0, shape.keep_topk, shape.pool_kernel,
                                    shape.scored, shape.ctx) if h in heads
                     else np.arange(shape.ctx - shape.budget, shape.ctx)
                     for h in range(shape.Hkv)]]
            ocache.compact(c, keep, [0])
            oattn.decode_attention(c, q_dec, "dense", groups=[(0, h) for h in heads])
            return shape.ctx * len(heads) / shape.Hkv, time.perf_counter() - t0, desc
        return run
    if workload == "quest_decode":
        shape = W.quest_decode(B=1, ctx=16 * 1024)
        inp = W.quest_inputs(shape, "cpu")
        c = ocache.from_tensors(inp["cache"])
        kmin, kmax = oquest.build_meta(c)
        g = [(0, h) for h in range(min(groups, shape.Hkv))]
        desc = (f"1 sequence, {len(g)} KV heads, 16384-token context (1023 candidate pages): "
                "page bound + top-128 + decode")

        def run():
            t0 = time.perf_counter()
            opipe.quest_step(c, kmin, kmax, inp["q_steps"][0], shape.top_pages, groups=g)
            return len(g) / shape.Hkv, time.perf_counter() - t0, desc
        return run
    if workload == "h2o_decode":
        shape = W.h2o_decode(B=1, ctx=1152)
        inp = W.h2o_inputs(shape, "cpu", steps=2)
        c0 = ocache.from_tensors(inp["cache"])
        acc0 = np.random.default_rng(0).random(c0.slot_map.shape)
        desc = "1 sequence at the 1152-token budget: append + attention + acc + evict"

        def run():
            c, acc = c0.copy(), acc0.copy()
            t0 = time.perf_counter()
            opipe.h2o_step(c, acc, inp["q_steps"][0], inp["k_steps"][0], inp["v_steps"][0], shape)
            return 1.0, time.perf_counter() - t0, desc
        return run
    if workload == "kara_prune":
        shape = W.kara_prune(B=1)
        inp = W.kara_inputs(shape, "cpu")
        c0 = ocache.from_tensors(inp["cache"])
        q_pos = inp["q_pos"].numpy()
        mask = inp["prune_mask"].numpy()
        desc = "1 of 128 sequences (16384 tokens): Kara compress + prune"

        def run():
            c = c0.copy()
            t0 = time.perf_counter()
            r = opipe.kara_compress(c, inp["q_win"], q_pos, shape)
            ocache.compact(c, r["keep"], r["first_slot"])
            ocache.prune(c, [shape.prune_L], [shape.prune_R], mask)
            return shape.ctx, time.perf_counter() - t0, desc
        return run
    if workload == "kara_schedule":
        shape = W.kara_schedule(B=2)
        inp = W.kara_schedule_inputs(shape, "cpu", steps=4)
        c0 = ocache.from_tensors(inp["cache"])
        # sequence 1 fills its window at the first step: one compression per call
        win0 = [shape.ctx - shape.fill(0), shape.ctx - (shape.window - 1)]
        desc = ("2 sequences (2304 resident tokens) for one decode step in which one of "
                "them compresses its window")

        def run():
            c, ring, win = c0.copy(), inp["q_ring"].clone(), list(win0)
            t0 = time.perf_counter()
            opipe.kara_schedule_step(c, inp["q_steps"][0], inp["k_steps"][0],
                                     inp["v_steps"][0], ring, win, shape)
            return 2.0, time.perf_counter() - t0, desc
        return run
    raise ValueError(workload)


def oracle_runs(workload: str, groups: int, n: int):
    run = oracle_prepare(workload, groups)
    return [run() for _ in range(n)]


_UNIT_STATE = {}


def _oracle_unit_init(workload):
    """Worker set-up: one sequence of the workload (seeded, the same for every
    worker) in the oracle's cache form."""
    import se_workloads as W
    from oracle import cache as ocache
    shape = W.WORKLOADS[workload](B=1)
    inp = W.snapkv_inputs(shape, "cpu")
    _UNIT_STATE.update(shape=shape, inp=inp, c=ocache.from_tensors(inp["cache"]),
                       q_pos=inp["q_pos"].numpy())


def _oracle_unit(h):
    """One (sequence, KV head) unit of the SnapKV oracle: window scores,
    pooled top-k, decode attention over the kept entries."""
    from oracle import attention as oattn
    from oracle import pipelines as opipe
    from oracle import scoring as oscore
    from oracle import selection as osel
    st = _UNIT_STATE
    shape, inp, c = st["shape"], st["inp"], st["c"]
    h = h % shape.Hkv
    s = oscore.score_window(c, inp["q_win"], st["q_pos"], [0], [shape.ctx], [0], [shape.scored],
                            True, groups=[(0, h)])
    keep = osel.topk_keep(s[(0, h)], 0, shape.keep_topk, shape.pool_kernel, shape.scored, shape.ctx)
    G = shape.G
    oattn.attend(opipe.to_f64(inp["q_dec"])[0, h * G:(h + 1) * G], c.keys(0, h, keep),
                 c.vals(0, h, keep))
    return h


def oracle_all_cores(workload: str):
    """The SnapKV oracle over as many (sequence, KV head) units as the
    workload has, on all host cores (one single-threaded worker per core,
    spawned); returns (token-equivalents, seconds, cores, description)."""
    import multiprocessing as mp
    import se_workloads as W
    full = W.WORKLOADS[workload]()
    cores = os.cpu_count() or 1
    n_units = full.B * full.Hkv
    workers = min(cores, n_units)
    ctx = mp.get_context("spawn")
    with ctx.Pool(processes=workers, initializer=_oracle_unit_init, initargs=(workload,)) as pool:
        pool.map(_oracle_unit, range(workers), chunksize=1)            # warm the workers
        t0 = time.perf_counter()
        pool.map(_oracle_unit, range(n_units), chunksize=1)
        dt = time.perf_counter() - t0
    desc = (f"{n_units} (sequence, KV head) units of {full.ctx} tokens (the workload's count; "
            f"each a head of one seeded sequence), one single-threaded worker per core on "
            f"{workers} of {cores} host cores: score + pool/top-k + decode over the kept entries")
    return full.B * full.ctx, dt, workers, desc


def oracle_subprocess(workload: str, groups: int, n: int = 1, all_cores: bool = False):
    """Oracle samples in a child process pinned to one BLAS / OpenMP thread
    (all_cores: the whole SnapKV batch over a pool of such workers)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    call = (f"bench.oracle_all_cores({workload!r})" if all_cores
            else f"bench.oracle_runs({workload!r}, {groups}, {n})")
    code = (f"import sys, json; sys.path.insert(0, {ROOT!r}); import bench; "
            f"print(json.dumps({call}))")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


# ---------------------------------------------------------------------------
# GPU workloads
# ---------------------------------------------------------------------------

METRIC = "KV tokens scored+compacted/s"


class Events:
    def __init__(self, torch, names):
        self.torch = torch
        self.names = names
        self.ev = {n: [] for n in names}

    def mark(self, name):
        e = self.torch.cuda.Event(enable_timing=True)
        e.record()
        self.ev[name].append(e)

    def durations(self, a, b):
        return [x.elapsed_time(y) for x, y in zip(self.ev[a], self.ev[b])]


def run_snapkv(args, torch, rank, world):
    import se_workloads as W
    from attention_scored_sparse_gb300 import pipelines as P
    shape = W.WORKLOADS[args.workload](**batch_kw(args))
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = W.snapkv_inputs(shape, dev)
    pc = inp["cache"]
    pipe = P.SnapKV(pc, shape.Hq, ctx=shape.ctx, window=shape.window, budget=shape.budget,
                    pool_kernel=shape.pool_kernel)
    o = torch.empty_like(inp["q_dec"])
    meta = {n: getattr(pc, n).clone() for n in
            ["block_table", "slot_map", "ctx_len", "free_list", "free_top", "page_refcount"]}

    def restore():
        for n, t in meta.items():
            getattr(pc, n).copy_(t)

    stages = ["s0", "s1", "s2", "s3"]
    ev = Events(torch, stages)

    # the step as the pipeline runs it: compaction and decode attention in
    # one pass over the kept entries (se_compact_decode)
    def step(timed):
        restore()
        if timed: ev.mark("s0")
        pipe.score(inp["q_win"], inp["q_pos"])
        if timed: ev.mark("s1")
        pipe.select()
        if timed: ev.mark("s2")
        pipe.compact_decode_fused(inp["q_dec"], o)
        if timed: ev.mark("s3")

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    assert int(pc.status.item()) == 0
    t_wall, clocks = timed_loop(args, torch, rank, world, lambda: step(True), lambda: step(False))
    score_ms = ev.durations("s0", "s1")
    sel_ms = ev.durations("s1", "s2")
    cd_ms = ev.durations("s2", "s3")
    step_ms = [a + b + c for a, b, c in zip(score_ms, sel_ms, cd_ms)]
    ms = statistics.mean(step_ms)
    # breakdown only (not the step time): compaction, then decode attention
    # over the compacted cache, one after the other
    sq = Events(torch, ["c0", "c1", "c2"])
    for _ in range(20):
        restore()
        pipe.score(inp["q_win"], inp["q_pos"])
        pipe.select()
        sq.mark("c0")
        pipe.compact()
        sq.mark("c1")
        pipe.decode(inp["q_dec"], o)
        sq.mark("c2")
    torch.cuda.synchronize()
    comp_ms = sq.durations("c0", "c1")
    dec_ms = sq.durations("c1", "c2")
    G, D, B, Hkv = shape.G, shape.D, shape.B, shape.Hkv
    rows = shape.window * G
    flops = 2.0 * D * rows * shape.ctx * B * Hkv          # one sweep over the attention range
    entry = 2 * D * (2 if shape.dtype == torch.bfloat16 else 4)  # K + V bytes of one entry
    comp_bytes = 2.0 * B * Hkv * shape.budget * entry            # read + write
    dec_bytes = B * Hkv * shape.budget * entry
    tokens = B * shape.ctx
    # e2e: host buffers, copies inside the timed region
    e2e = run_e2e_snapkv(torch, pipe, inp, restore, args.steps)
    detail = {
        "score_ms": statistics.mean(score_ms), "select_ms": statistics.mean(sel_ms),
        "compact_and_decode_ms": statistics.mean(cd_ms),
        "compact_ms": statistics.mean(comp_ms), "decode_ms": statistics.mean(dec_ms),
        "score_tflops": flops / (statistics.mean(score_ms) * 1e-3) / 1e12,
        "compact_gbs": comp_bytes / (statistics.mean(comp_ms) * 1e-3) / 1e9,
        "decode_gbs": dec_bytes / (statistics.mean(dec_ms) * 1e-3) / 1e9,
    }
    hbm = peaks()[0]["hbm_gbs"]
    # the step's one pass over the kept entries: each read once, written once
    detail["compact_and_decode_gbs"] = comp_bytes / (statistics.mean(cd_ms) * 1e-3) / 1e9
    detail["compact_and_decode_frac_of_hbm"] = detail["compact_and_decode_gbs"] / hbm
    detail["compact_frac_of_hbm"] = detail["compact_gbs"] / hbm
    detail["decode_frac_of_hbm"] = detail["decode_gbs"] / hbm
    # DRAM bytes of one se_score_window call: none measured on the current
    # scorer kernels (the last ncu capture, 275.99 + 3.33 MB and 278.70 +
    # 2.75 MB for the two passes, predates a change to pass 1)
    roof = dict(bound="tensor", achieved=detail["score_tflops"], unit="TFLOP/s",
                kernel="se_score_window", per_launch=f"{flops:.4g} FLOP (one QK^T sweep)",
                traffic=None)
    launches = 2 + 1 + 3         # score (2), select, compaction plan + compaction/decode + commit
    cfg = {"workload": f"{shape.name}: B={B} x {shape.ctx} tokens, Hq={shape.Hq}/Hkv={Hkv}, "
                       f"d={D}, window {shape.window}, pool {shape.pool_kernel}, budget "
                       f"{shape.budget}", "l2": "inputs larger than L2 (KV cache 570 MB)"}
    return dict(tokens=tokens, ms=ms, wall=t_wall, clocks=clocks, detail=detail, roof=roof,
                launches=launches, cfg=cfg, e2e=e2e, dtype="bf16" if shape.dtype == torch.bfloat16 else "f32")


def run_e2e_snapkv(torch, pipe, inp, restore, steps):
    """Same metric through the public API with host-resident per-step inputs,
    as a serving loop runs it: the pipeline step is captured once per input
    buffer in a CUDA graph (two device input buffers); while step i computes
    from one buffer, a second stream copies the next step's q_win, q_pos,
    q_dec from pinned host memory into the other, and after the step its
    decode output and kept indices are read back.  Each timed step holds the
    graph, one host-to-device copy of a step's inputs (the step's end waits
    for it) and the device-to-host read of its own results; steps are
    enqueued without host synchronisation between them."""
    hq = {k: inp[k].cpu().pin_memory() for k in ("q_win", "q_pos", "q_dec")}
    dq = [{k: torch.empty_like(inp[k]) for k in hq} for _ in range(2)]
    outs = [torch.empty_like(inp["q_dec"]) for _ in range(2)]
    ho = torch.empty(outs[0].shape, dtype=outs[0].dtype, pin_memory=True)
    hk = torch.empty(pipe.keep.shape, dtype=pipe.keep.dtype, pin_memory=True)
    for j in range(2):
        for k in hq:
            dq[j][k].copy_(hq[k])
    graphs = []
    for j in range(2):
        restore()
        pipe.step(dq[j]["q_win"], dq[j]["q_pos"], dq[j]["q_dec"], outs[j])      # warm
        torch.cuda.synchronize()
        restore()
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_):
            pipe.step(dq[j]["q_win"], dq[j]["q_pos"], dq[j]["q_dec"], outs[j])
        graphs.append(g_)
    torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    # steps are enqueued back to back (no host synchronisation between them,
    # as a serving loop runs); buffer 1 - j is refilled only after the step
    # that read it last has ended
    ev = []
    ends = [None, None]
    for i in range(steps + 2):
        j = i % 2
        restore()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        h2d = torch.cuda.Event()
        e0.record(main)
        if ends[1 - j] is not None:
            side.wait_event(ends[1 - j])
        side.wait_event(e0)
        with torch.cuda.stream(side):
            for k in hq:
                dq[1 - j][k].copy_(hq[k], non_blocking=True)   # the next step's inputs
            h2d.record(side)
        graphs[j].replay()
        ho.copy_(outs[j], non_blocking=True)
        hk.copy_(pipe.keep, non_blocking=True)
        main.wait_event(h2d)
        e1.record(main)
        ends[j] = e1
        ev.append((e0, e1))
    torch.cuda.synchronize()
    total = [x.elapsed_time(y) for x, y in ev[2:]]
    bi = sum(t.numel() * t.element_size() for t in hq.values())
    bo = ho.numel() * ho.element_size() + hk.numel() * hk.element_size()
    return statistics.mean(total), bi, bo


def run_quest(args, torch, rank, world):
    import se_workloads as W
    from attention_scored_sparse_gb300 import pipelines as P
    shape = W.quest_decode(**batch_kw(args))
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = W.quest_inputs(shape, dev)
    pipe = P.QuestDecode(inp["cache"], shape.Hq, ctx=shape.ctx, top_pages=shape.top_pages)
    pipe.build_meta()                    # warm
    m0 = torch.cuda.Event(enable_timing=True)
    m1 = torch.cuda.Event(enable_timing=True)
    m0.record()
    pipe.build_meta()
    m1.record()
    torch.cuda.synchronize()
    meta_ms = m0.elapsed_time(m1)
    # metadata build reads every resident key once and writes 2 x D per (page, head)
    meta_build_bytes = shape.B * shape.ctx * shape.Hkv * shape.D * 2 + \
        shape.B * (shape.ctx // shape.page_size) * shape.Hkv * 2 * shape.D * 2
    o = torch.empty_like(inp["q_steps"][0])
    sq = torch.empty_like(inp["q_steps"][0])
    sq.copy_(inp["q_steps"][0])
    # the per-step working set (page bounds 67 MB + selected K/V 17 MB) fits in
    # L2, so L2 is flushed by a 256 MB write before every timed step
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    # the step as a serving loop replays it (page selection, then attention,
    # captured together), its two halves for the breakdown, and the same step
    # as one cluster launch
    parts = {"step": lambda q: pipe.step(q, o), "select": pipe.select,
             "decode": lambda q: pipe.decode(q, o), "fused": lambda q: pipe.step_fused(q, o)}
    graphs = {}
    for name, fn in parts.items():
        fn(sq)
        torch.cuda.synchronize()
        if not args.no_graph:
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_):
                fn(sq)
            graphs[name] = g_
    torch.cuda.synchronize()

    def run(name):
        if name in graphs:
            graphs[name].replay()
        else:
            parts[name](sq)

    ev = Events(torch, ["s0", "s1", "f0", "f1"])
    it = [0]

    def step(timed):
        q = inp["q_steps"][it[0] % shape.steps]
        it[0] += 1
        sq.copy_(q)
        flush.fill_(it[0] & 255)
        if timed: ev.mark("s0")
        run("step")                        # page selection, then attention
        if timed: ev.mark("s1")
        flush.fill_((it[0] + 1) & 255)
        if timed: ev.mark("f0")
        run("fused")                       # the same step as one cluster launch
        if timed: ev.mark("f1")

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    t_wall, clocks = timed_loop(args, torch, rank, world, lambda: step(True), lambda: step(False))
    fused = ev.durations("f0", "f1")
    two_call = statistics.mean(ev.durations("s0", "s1"))
    ms = two_call
    # breakdown only (not the step time): the two halves replayed one after
    # the other, L2 flushed before each pair
    bq = Events(torch, ["b0", "b1", "b2"])
    for i in range(20):
        sq.copy_(inp["q_steps"][i % shape.steps])
        flush.fill_(i & 255)
        bq.mark("b0")
        run("select")
        bq.mark("b1")
        run("decode")
        bq.mark("b2")
    torch.cuda.synchronize()
    sel = bq.durations("b0", "b1")
    dec = bq.durations("b1", "b2")
    nb = shape.ctx // shape.page_size
    meta_bytes = shape.B * shape.Hkv * (nb - 1) * 2 * shape.D * 2
    kv_bytes = shape.B * shape.Hkv * (shape.top_pages + 1) * shape.page_size * 2 * shape.D * 2
    detail = {"meta_build_ms": meta_ms, "meta_build_gbs": meta_build_bytes / (meta_ms * 1e-3) / 1e9,
              "fused_step_ms": statistics.mean(fused), "two_call_step_ms": two_call,
              "select_ms": statistics.mean(sel), "decode_ms": statistics.mean(dec),
              "select_gbs": meta_bytes / (statistics.mean(sel) * 1e-3) / 1e9,
              "decode_gbs": kv_bytes / (statistics.mean(dec) * 1e-3) / 1e9,
              "step_gbs": (meta_bytes + kv_bytes) / (ms * 1e-3) / 1e9}
    roof = dict(bound="hbm", achieved=detail["step_gbs"], unit="GB/s",
                kernel="quest step (bound + top-k + decode attention)",
                per_launch=f"{meta_bytes + kv_bytes:.4g} B")
    return dict(tokens=shape.B, ms=ms, wall=t_wall, clocks=clocks, detail=detail, roof=roof,
                launches=2 + 1 + 1, metric="decode tokens/s", e2e=None,
                cfg={"workload": f"quest_decode: B={shape.B} x 131072 tokens, top 128 pages + current, "
                                 "32/8 heads, d=128, bf16",
                     "l2": "L2 flushed (256 MB write) before every timed step",
                     "launch": "step replayed from one CUDA graph (page bound, top-k, attention)"},
                dtype="bf16")


def run_h2o(args, torch, rank, world):
    import se_workloads as W
    from attention_scored_sparse_gb300 import pipelines as P
    shape = W.h2o_decode(**batch_kw(args))
    dev = torch.device("cuda", torch.cuda.current_device())
    nsteps = max(args.steps + args.warmup + 2, 16)
    inp = W.h2o_inputs(shape, dev, steps=nsteps)
    pipe = P.H2O(inp["cache"], shape.Hq, prompt=shape.ctx, heavy=shape.heavy, recent=shape.recent)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    pipe.prefill(inp["q_prompt"], inp["q_pos"])
    t1.record()
    torch.cuda.synchronize()
    prefill_ms = t0.elapsed_time(t1)
    o = torch.empty_like(inp["q_steps"][0])
    # the step (append, attention + running scores, evict-one, move-last) is
    # captured once in a CUDA graph over static input buffers; each step
    # copies its q, k, v in and replays the graph
    sq = torch.empty_like(inp["q_steps"][0])
    sk = torch.empty_like(inp["k_steps"][0])
    sv = torch.empty_like(inp["v_steps"][0])
    sq.copy_(inp["q_steps"][0]); sk.copy_(inp["k_steps"][0]); sv.copy_(inp["v_steps"][0])
    graph = None
    if not args.no_graph:
        s_cap = torch.cuda.Stream()
        s_cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s_cap):
            pipe.step(sq, sk, sv, o)          # warm: kernel attributes, first launches
        torch.cuda.current_stream().wait_stream(s_cap)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            pipe.step(sq, sk, sv, o)
        torch.cuda.synchronize()
    ev = Events(torch, ["s0", "s1"])
    it = [0]

    def step(timed):
        t = it[0] % nsteps
        it[0] += 1
        if timed: ev.mark("s0")
        sq.copy_(inp["q_steps"][t]); sk.copy_(inp["k_steps"][t]); sv.copy_(inp["v_steps"][t])
        if graph is not None:
            graph.replay()
        else:
            pipe.step(sq, sk, sv, o)
        if timed: ev.mark("s1")

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    t_wall, clocks = timed_loop(args, torch, rank, world, lambda: step(True), lambda: step(False))
    ms = statistics.mean(ev.durations("s0", "s1"))
    kv_bytes = shape.B * shape.Hkv * (shape.budget + 1) * 2 * shape.D * 2
    detail = {"prefill_ms": prefill_ms, "step_gbs": kv_bytes / (ms * 1e-3) / 1e9}
    detail.update(time_h2o_chunked(torch, shape, 512, dev))
    roof = dict(bound="hbm", achieved=detail["step_gbs"], unit="GB/s", kernel="h2o step",
                per_launch=f"{kv_bytes:.4g} B")
    return dict(tokens=shape.B, ms=ms, wall=t_wall, clocks=clocks, detail=detail, roof=roof,
                launches=1 + 1 + 1 + 1, metric="decode tokens/s", e2e=None,   # append, decode, evict-one, move-last
                cfg={"workload": f"h2o_decode: B={shape.B}, 4096-token prompt, budget 1024+128, "
                                 "32/8 heads, d=128, bf16", "l2": "inputs larger than L2"},
                dtype="bf16")


def time_h2o_chunked(torch, shape, chunk, dev, reps=3):
    """Chunk-wise H2O prefill eviction of the same prompt shape (chunks of
    ``chunk`` tokens appended, scored into the running scores, evicted to the
    budget); the cache metadata is restored between runs, outside the events."""
    import se_workloads as W
    from attention_scored_sparse_gb300 import pipelines as P
    inp = W.h2o_chunked_inputs(shape, chunk, dev)
    pc = inp["cache"]
    meta = ["block_table", "slot_map", "ctx_len", "logical_len", "free_list", "free_top",
            "page_refcount", "status"]
    snap = {m: getattr(pc, m).clone() for m in meta}
    pipe = P.H2OChunkedPrefill(pc, shape.Hq, chunk=chunk, heavy=shape.heavy, recent=shape.recent)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    times = []
    for r in range(reps + 1):
        for m in meta:
            getattr(pc, m).copy_(snap[m])
        torch.cuda.synchronize()
        t0.record()
        pipe.run(inp["q_chunks"], inp["q_pos"], inp["k_chunks"], inp["v_chunks"])
        t1.record()
        torch.cuda.synchronize()
        if r > 0:
            times.append(t0.elapsed_time(t1))
    if int(pc.status.item()) != 0:
        raise RuntimeError(f"chunked prefill failed with device status {int(pc.status.item())}")
    del inp, pipe
    return {"chunked_prefill_ms": statistics.mean(times), "chunked_prefill_chunk": chunk}


def run_kara(args, torch, rank, world):
    import se_workloads as W
    from attention_scored_sparse_gb300 import pipelines as P
    shape = W.kara_prune(**batch_kw(args))
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = W.kara_inputs(shape, dev)
    pc = inp["cache"]
    pipe = P.Kara(pc, shape.Hq, ctx=shape.ctx, window=shape.window, protected=shape.protected,
                  candidates=shape.candidates, budget=shape.budget, chunk_coef=shape.chunk_coef)
    meta = {n: getattr(pc, n).clone() for n in
            ["block_table", "slot_map", "ctx_len", "free_list", "free_top", "page_refcount"]}
    L = torch.full((shape.B,), shape.prune_L, dtype=torch.int32, device=dev)
    R = torch.full((shape.B,), shape.prune_R, dtype=torch.int32, device=dev)
    o = torch.empty_like(inp["q_dec"])
    new_ctx = shape.prune_L + shape.prune_keep + (shape.ctx - shape.window - shape.prune_R) + \
        shape.budget + shape.protected

    def restore():
        for n, t in meta.items():
            getattr(pc, n).copy_(t)

    ev = Events(torch, ["s0", "s1", "s2", "s3"])

    def step(timed):
        restore()
        if timed: ev.mark("s0")
        pipe.compress(inp["q_win"], inp["q_pos"])
        if timed: ev.mark("s1")
        pipe.prune(L, R, inp["prune_mask"])
        if timed: ev.mark("s2")
        pipe.decode(inp["q_dec"], o, max_entries=new_ctx)
        if timed: ev.mark("s3")

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    assert int(pc.status.item()) == 0
    t_wall, clocks = timed_loop(args, torch, rank, world, lambda: step(True), lambda: step(False))
    comp = ev.durations("s0", "s1")
    prn = ev.durations("s1", "s2")
    dec = ev.durations("s2", "s3")
    ms = statistics.mean([a + b + c for a, b, c in zip(comp, prn, dec)])
    entry = 2 * shape.D * 2
    moved = shape.prune_keep + (shape.ctx - shape.window - shape.prune_R) + shape.budget + shape.protected
    prune_bytes = 2.0 * shape.B * shape.Hkv * moved * entry
    dec_bytes = shape.B * shape.Hkv * new_ctx * entry
    detail = {"compress_ms": statistics.mean(comp), "prune_ms": statistics.mean(prn),
              "decode_ms": statistics.mean(dec),
              "prune_gbs": prune_bytes / (statistics.mean(prn) * 1e-3) / 1e9,
              "decode_gbs": dec_bytes / (statistics.mean(dec) * 1e-3) / 1e9}
    roof = dict(bound="hbm", achieved=detail["prune_gbs"], unit="GB/s", kernel="se_prune_span",
                per_launch=f"{prune_bytes:.4g} B (moved entries, read + write)")
    return dict(tokens=shape.B * shape.ctx, ms=ms, wall=t_wall, clocks=clocks, detail=detail,
                roof=roof, launches=3 + 1 + 3 + 5 + 1, e2e=None,
                cfg={"workload": f"kara_prune: B={shape.B} x 16384 tokens, window 256 (32 protected), "
                                 "chunk budget 64, prune [2048,6144) keep 20%",
                     "l2": "inputs larger than L2"}, dtype="bf16")


def batch_kw(args):
    """--batch: a smaller batch of the same workload (profiling captures)."""
    return {"B": args.batch} if getattr(args, "batch", None) else {}


def timed_loop(args, torch, rank, world, fn, warm=None):
    """Times args.steps calls of fn.  The clock sampler starts first; `warm`
    (untimed steps) keeps the GPU busy for at least 0.3 s while it starts, so
    that the clock record holds samples under load even for short runs."""
    import torch.distributed as dist
    with ClockSampler(torch.cuda.current_device()) as cs:
        if warm is not None:
            t_w = time.perf_counter()
            while time.perf_counter() - t_w < 0.3:
                for _ in range(8):
                    warm()
                torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            fn()
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        # a few more samples at the same load after the timed region
        if warm is not None:
            t_w = time.perf_counter()
            while time.perf_counter() - t_w < 0.05:
                warm()
            torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    return t1 - t0, cs.summary()


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's step time (every rank runs its own replica)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Units processed by all ranks per second of the slowest rank."""
    return units_per_rank * world / (ms * 1e-3)


def run_kara_schedule(args, torch, rank, world):
    import se_workloads as W
    from attention_scored_sparse_gb300 import pipelines as P
    n_steps = args.warmup + args.steps
    shape = W.kara_schedule(steps=n_steps, **batch_kw(args))
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = W.kara_schedule_inputs(shape, dev)
    fills = [shape.fill(b) for b in range(shape.B)]
    pipe = P.KaraSchedule(inp["cache"], shape.Hq, ctx=shape.ctx, fills=fills,
                          window=shape.window, protected=shape.protected,
                          candidates=shape.candidates, budget=shape.budget,
                          chunk_coef=shape.chunk_coef, max_ctx=shape.ctx + n_steps)
    o = torch.empty_like(inp["q_steps"][0])
    ring = inp["q_ring"]
    ev = Events(torch, ["s0", "s1"])
    it = [0]
    resident = []                        # entries attended per step (for the GB/s)

    def step(timed):
        t = it[0]
        it[0] += 1
        resident.append(sum(pipe.ctx) + shape.B)
        if timed: ev.mark("s0")
        pipe.step(inp["q_steps"][t], inp["k_steps"][t], inp["v_steps"][t], o, ring)
        if timed: ev.mark("s1")

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    c0 = pipe.compressions
    t_wall, clocks = timed_loop(args, torch, rank, world, lambda: step(True))
    if int(inp["cache"].status.item()) != 0:
        raise RuntimeError(f"device status {int(inp['cache'].status.item())}")
    ms = statistics.mean(ev.durations("s0", "s1"))
    entry = 2 * shape.D * 2 * shape.Hkv
    kv_bytes = statistics.mean(resident[args.warmup:]) * entry
    detail = {"compressions_per_step": (pipe.compressions - c0) / args.steps,
              "decode_gbs": kv_bytes / (ms * 1e-3) / 1e9}
    roof = dict(bound="hbm", achieved=detail["decode_gbs"], unit="GB/s",
                kernel="kara schedule step (append + decode + staggered compression)",
                per_launch=f"{kv_bytes:.4g} B (resident K/V attended per step)")
    return dict(tokens=shape.B, ms=ms, wall=t_wall, clocks=clocks, detail=detail, roof=roof,
                launches=1 + 1 + (3 + 1 + 3) * detail["compressions_per_step"],   # append, decode, compressions
                metric="decode tokens/s", e2e=None,
                cfg={"workload": f"kara_schedule: B={shape.B} decoding over 2304 resident tokens, "
                                 "Kara window 256 (32 protected, 32 candidates, chunk budget 64) "
                                 "compressed when full, staggered over the 160-step period; "
                                 "32/8 heads, d=128, bf16",
                     "l2": "inputs larger than L2 (1.2 GB attended per step)"},
                dtype="bf16")


def other_workloads(args, torch, rank, world):
    """Step time and roofline fraction of the Quest, H2O and Kara workloads
    (20 timed steps each after 3 warm-up steps), measured in this run."""
    import copy
    pk, src = peaks()
    out = {}
    for name in ("quest_decode", "h2o_decode", "kara_prune"):
        a2 = copy.copy(args)
        a2.workload, a2.steps, a2.warmup = name, 20, 3
        try:
            r = RUNNERS[name](a2, torch, rank, world)
        except Exception as exc:  # reported, not hidden
            out[name] = {"error": str(exc)[-300:]}
            continue
        peak = pk["bf16_tflops"] if r["roof"]["bound"] == "tensor" else pk["hbm_gbs"]
        keep = {k: v for k, v in r["detail"].items() if k.endswith(("_ms", "_gbs"))}
        out[name] = {"ms_per_step": r["ms"], "value": r["tokens"] / (r["ms"] * 1e-3),
                     "unit": "KV tokens/s" if r.get("metric", METRIC) == METRIC else "decode tokens/s",
                     "kernel": r["roof"]["kernel"], "achieved": r["roof"]["achieved"],
                     "unit_roof": r["roof"]["unit"], "frac": r["roof"]["achieved"] / peak,
                     "l2": r["cfg"].get("l2"), "detail": keep}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


RUNNERS = {"snapkv_llama8b": run_snapkv, "snapkv_tiny": run_snapkv, "quest_decode": run_quest,
           "h2o_decode": run_h2o, "kara_prune": run_kara, "kara_schedule": run_kara_schedule}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="snapkv_llama8b", choices=sorted(RUNNERS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch decode steps eagerly")
    ap.add_argument("--batch", type=int, default=None,
                    help="sequences of the workload (default: the workload's own; for profiling)")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the short runs of the other workloads reported in detail")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))

    if args.impl == "reference":
        if rank != 0:
            return
        runs = oracle_subprocess(args.workload, 1, args.warmup + args.steps)[args.warmup:]
        per = [r[0] for r in runs]
        times = [r[1] for r in runs]
        desc = runs[0][2]
        value = sum(per) / sum(times)
        unit = ("KV tokens/s" if args.workload.startswith("snapkv") or args.workload == "kara_prune"
                else "decode tokens/s")
        line = {"impl": "reference", "metric": METRIC if unit == "KV tokens/s" else "decode tokens/s",
                "value": value, "unit": unit, "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic",
                "config": {"workload": args.workload, "sample": desc},
                "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    import attention_scored_sparse_gb300  # noqa: F401  (fails loudly without the library)

    r = RUNNERS[args.workload](args, torch, rank, world)
    ms = max_over_ranks(r["ms"], world, "cuda")
    value = whole_job_rate(r["tokens"], world, ms)
    pk, src = peaks()
    peak = pk["bf16_tflops"] if r["roof"]["bound"] == "tensor" else pk["hbm_gbs"]
    metric = r.get("metric", METRIC)
    unit = "KV tokens/s" if metric == METRIC else "decode tokens/s"
    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": r["dtype"], "data": "synthetic",
        "config": dict(r["cfg"], parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        "roofline": {"bound": r["roof"]["bound"], "achieved": r["roof"]["achieved"], "peak": peak,
                     "unit": r["roof"]["unit"], "frac": r["roof"]["achieved"] / peak,
                     "traffic": r["roof"].get("traffic"), "kernel": r["roof"]["kernel"],
                     "per_launch": r["roof"]["per_launch"], "peak_source": src},
        "clocks": r["clocks"], "gpu_launches": int(round(r["launches"] * args.steps)), "detail": r["detail"],
        "wall_s_timed_region": r["wall"],
    }
    if r.get("e2e"):
        e2e_ms, bi, bo = r["e2e"]
        e2e_ms = max_over_ranks(e2e_ms, world, "cuda")     # the slowest rank, like the step time
        line["e2e"] = {"value": r["tokens"] * world / (e2e_ms * 1e-3), "unit": unit,
                       "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo}
    if world == 1 and args.workload == "snapkv_llama8b" and not args.no_others:
        # short runs of the other workloads (their own inputs and step), for
        # the decode / compaction / Quest fractions beside the headline
        line["detail"]["other_workloads"] = other_workloads(args, torch, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            tokens, dt, desc = oracle_subprocess(args.workload, 2)[0]
            base = {"value": tokens / dt, "unit": unit, "cores": 1, "kind": "oracle",
                    "sample": desc, "host_cores": os.cpu_count()}
            if args.workload == "snapkv_llama8b":
                tok_all, dt_all, cores, desc_all = oracle_subprocess(args.workload, 0, all_cores=True)
                base = {"value": tok_all / dt_all, "unit": unit, "cores": cores, "kind": "oracle",
                        "sample": desc_all, "host_cores": os.cpu_count(),
                        "one_core": {"value": tokens / dt, "cores": 1, "sample": desc}}
            line["cpu_baseline"] = base
        except Exception as exc:  # reported, not hidden
            line["cpu_baseline"] = {"value": None, "error": str(exc)[-300:]}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
