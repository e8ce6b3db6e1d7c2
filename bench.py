#!/usr/bin/env python
"""Benchmark of the CSA2 FP4 sparse-decode hot path on B300.

Workload (one "step"): a decode step of a three-layer CSA2 group FULL -> REINDEX ->
REUSE for 32 sequences at 128K context (32768 compressed entries each), 64 query
heads, latent 512 + rope 64 in FP4 (E2M1 + E4M3 per 16), indexer 8 x 64 in bf16,
top-K 2048, sliding window 128. Per layer one csa2_decode_layer call: the indexer and
top-K selection, then the attention over the selected entries and the window
(csa2_decode_attention); REUSE skips the indexer.
--attn fused times csa2_index_topk + csa2_decode_attention instead, --attn two-call
csa2_index_topk + csa2_sparse_decode + csa2_swa_merge. The KV caches and keys are resident in HBM (written before timing); each
timed step re-reads them, and L2 is flushed between steps.

Prints one JSON line. The GPU arm runs on one GPU only (--gpus 1, no torchrun ranks):
the attention and CED kernels use TMA cluster multicast, which this library runs in
single-GPU calls only, so more ranks get an "unavailable" line and launch nothing.
--impl reference times the CPU oracle on the same workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import csa2_inputs as ci  # noqa: E402

METRIC = "CSA2 FP4 decode steps/s + HBM GB/s vs 8 TB/s; CED KV-proj TFLOP/s"
CFG = ci.DECODE_128K
ENTRY_BYTES = 288 + 36   # per entry as the method stores it (the 60 bytes padding each 384-byte row not counted)
KEY_BYTES = 64 * 2
SWA_ROW_BYTES = 576 * 2
TARGET_HBM_GBS = 8000.0


def algorithmic_bytes_per_step(cfg=CFG) -> int:
    """Indexer keys (FULL, REINDEX) + K selected entries + SWA window, per sequence per layer."""
    per_seq = 0
    for m in cfg.modes:
        if m != ci.REUSE:
            per_seq += cfg.N * KEY_BYTES
        per_seq += cfg.K * ENTRY_BYTES + cfg.W * SWA_ROW_BYTES
    return per_seq * cfg.B


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, src="fallback")


def ncu_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu record, or None when the
    kernel's source has changed since that capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        rec = json.load(open(p))[kernel]
        src = open(os.path.join(ROOT, rec["source"]), "rb").read()
        if hashlib.sha256(src).hexdigest() != rec["sha256"]:
            return None
        return int(rec["bytes_per_launch"])
    except Exception:
        return None


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def aggregate_over_ranks(total_s: float, steps: int, world: int, device=None):
    """Every rank times its own replica of the workload (no collective on the data path);
    the job's time is the slowest rank's, and its value is world x steps / that time.
    Returns (seconds, whole-job steps/s)."""
    if world > 1:
        import torch
        t = torch.tensor([total_s], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_s = float(t.item())
    return total_s, world * steps / total_s


# ---------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
# The FP4 cache exists before a decode step (written by the FULL layer's encode or the
# appends), so encoding it is set-up: it runs in a spawn process pool, untimed. The timed
# oracle work of a layer is the indexer and top-K (FULL, REINDEX), the dequantisation of
# the selected entries, the sparse attention, the SWA branch and the merge, in the main
# process (NumPy, float64; BLAS threads as configured).
def _encode_rows_task(task):
    """Spawn-pool task: FP4 codes / scales of rows [r0, r1) of a sequence's latent KV."""
    name, layer, b, r0, r1 = task
    from oracle import fp4
    cfg = ci.CONFIGS[name]
    X = ci.latent_rows(cfg, layer, b, np.arange(r0, r1))
    return b, r0, fp4.encode(X)


_POOL = None


def oracle_pool():
    """Process pool (spawn: safe after CUDA was initialised) for the cache set-up."""
    global _POOL
    if _POOL is None:
        import multiprocessing as mp
        _POOL = mp.get_context("spawn").Pool(max(1, min(16, cpu_cores())))
    return _POOL


def oracle_caches(cfg, seqs, chunk=65536):
    """FP4 cache (codes, scales) of the FULL layer for each sequence in seqs (set-up)."""
    tasks = [(cfg.name, 0, b, r0, min(r0 + chunk, cfg.N)) for b in seqs for r0 in range(0, cfg.N, chunk)]
    parts = {}
    for b, r0, (c, sc) in oracle_pool().imap_unordered(_encode_rows_task, tasks):
        parts.setdefault(b, []).append((r0, c, sc))
    out = {}
    for b, lst in parts.items():
        lst.sort(key=lambda x: x[0])
        out[b] = (np.concatenate([x[1] for x in lst]), np.concatenate([x[2] for x in lst]))
    return out


def oracle_layer_seconds(cfg, inp, li, b, cache, prev_idx=None, tokens=None):
    """Timed oracle work of layer li for sequence b (query tokens `tokens`, default all).
    Returns (seconds, idx [T', K]) where idx feeds a following REUSE layer."""
    from oracle import attention, fp4, indexer
    L = inp.layers[li]
    codes, scales = cache
    f64 = lambda a: ci.bf16_bits_to_f32(a).astype(np.float64)
    ts = list(range(cfg.T)) if tokens is None else list(tokens)
    t0 = time.perf_counter()
    if L.mode != ci.REUSE:
        I = indexer.scores(f64(L.q_idx[b][ts]), L.w_idx[b][ts], f64(L.z[b]))
        idx = np.stack([indexer.topk(I[k], int(inp.n_visible[b * cfg.T + t]), cfg.K) for k, t in enumerate(ts)])
    else:
        idx = prev_idx
    for k, t in enumerate(ts):
        qi = b * cfg.T + t
        sel = idx[k][idx[k] >= 0]
        rows = fp4.decode(codes[sel], scales[sel])
        q = f64(L.q[b, t])
        og, lg = attention.attend(q, rows, cfg.d_v, cfg.softmax_scale)
        os_, ls = attention.swa_branch(q, f64(L.swa[b]), int(inp.win_start[qi]), int(inp.win_len[qi]), cfg.d_v,
                                       cfg.softmax_scale)
        attention.merge(og, lg, os_, ls)
    return time.perf_counter() - t0, idx


def oracle_step_seconds(cfg, inp, caches, seqs=None, tokens=None):
    """One oracle step: every layer of the group for every sequence in seqs (default all),
    over the query tokens `tokens` (default all). Returns (seconds, per-layer seconds)."""
    seqs = range(cfg.B) if seqs is None else seqs
    per_layer = [0.0] * len(cfg.modes)
    for b in seqs:
        prev = None
        for li in range(len(cfg.modes)):
            dt, prev = oracle_layer_seconds(cfg, inp, li, b, caches[b], prev, tokens)
            per_layer[li] += dt
    return sum(per_layer), per_layer


def cpu_cores() -> int:
    return len(os.sched_getaffinity(0))


def blas_threads() -> str:
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k):
            return f"{k}={os.environ[k]}"
    return "BLAS default (all cores)"


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    inp = ci.make_decode_inputs(CFG, with_x=False)
    wall0 = time.perf_counter()
    caches = oracle_caches(CFG, range(CFG.B))
    setup_s = time.perf_counter() - wall0
    for _ in range(args.warmup):
        oracle_step_seconds(CFG, inp, caches)
    times, per_layer = [], None
    for _ in range(args.steps):
        dt, per_layer = oracle_step_seconds(CFG, inp, caches)
        times.append(dt)
    step_s = sum(times) / len(times)
    value = 1.0 / step_s
    sample = (f"every step is the full workload: {CFG.B} sequences x {len(CFG.modes)} layers (indexer, top-K, "
              f"dequantisation of the selected entries, attention, SWA, merge), FP64 NumPy; last step's per-layer "
              f"seconds {[round(x, 3) for x in per_layer]}; the FP4 caches ({CFG.B} x {CFG.N} entries) were encoded "
              f"before timing ({setup_s:.1f} s in a {min(16, cpu_cores())}-process pool)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(),
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample, "blas": blas_threads()},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def cpu_baselines(bench_inp=None):
    """The oracle timed on the host cores for every workload of the bench (a reported
    baseline, not a target): the three decode workloads in full, the prefill chunk on 64
    evenly spaced query tokens (first and last included) and the CED projection on 256
    sampled rows x all 20 layers, both extrapolated linearly."""
    out = {}
    cores = cpu_cores()

    def entry(value, unit, sample):
        return {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample,
                "blas": blas_threads()}

    # 128K decode group: one full step
    cfg = ci.DECODE_128K
    inp = bench_inp if bench_inp is not None else ci.make_decode_inputs(cfg, with_x=False)
    caches = oracle_caches(cfg, range(cfg.B))
    step_s, per_layer = oracle_step_seconds(cfg, inp, caches)
    out[cfg.name] = entry(1.0 / step_s, "steps/s",
                          f"one full step: {cfg.B} sequences x {len(cfg.modes)} layers, per-layer seconds "
                          f"{[round(x, 3) for x in per_layer]}; FP4 caches encoded before timing")
    del caches
    # tiny decode step: full, mean of 20 calls
    cfg = ci.TINY
    inp = ci.make_decode_inputs(cfg, with_x=False)
    caches = oracle_caches(cfg, range(cfg.B))
    ts = [oracle_step_seconds(cfg, inp, caches)[0] for _ in range(20)]
    out[cfg.name] = entry(statistics.mean(ts) * 1e6, "us/call", "the full tiny step (one FULL layer), mean of 20")
    # 1M decode: full
    cfg = ci.DECODE_1M
    inp = ci.make_decode_inputs(cfg, with_x=False)
    caches = oracle_caches(cfg, range(cfg.B))
    step_s, _ = oracle_step_seconds(cfg, inp, caches)
    out[cfg.name] = entry(1.0 / step_s, "calls/s", f"the full call: {cfg.B} sequences x {cfg.N} entries")
    del caches, inp
    # prefill chunk: 64 evenly spaced tokens, extrapolated to 4096
    cfg = ci.PREFILL_CHUNK
    inp = ci.make_decode_inputs(cfg, with_x=False)
    caches = oracle_caches(cfg, range(cfg.B))
    toks = sorted(set(np.linspace(0, cfg.T - 1, 64).round().astype(int).tolist()))
    dt, _ = oracle_step_seconds(cfg, inp, caches, tokens=toks)
    call_s = dt / len(toks) * cfg.T
    flop = 2.0 * cfg.T * cfg.H * (cfg.K + cfg.W) * (576 + cfg.d_v) + 2.0 * cfg.T * cfg.N * cfg.H_I * 64
    out[cfg.name] = entry(1.0 / call_s, "calls/s",
                          f"{len(toks)} evenly spaced query tokens of {cfg.T} ({dt:.2f} s), extrapolated x"
                          f"{cfg.T / len(toks):.0f}; {flop / call_s / 1e12:.6f} TFLOP/s")
    del caches, inp
    # CED projection: 256 sampled rows x 20 layers, extrapolated to 32768 rows
    from oracle import ced
    cc = ci.CED_PROJ
    cin = ci.make_ced_inputs(cc)
    rows = np.linspace(0, cc.rows - 1, 256).round().astype(int)
    f32 = lambda a: ci.bf16_bits_to_f32(a)
    Hs = f32(cin.H[rows])
    t0 = time.perf_counter()
    for l in range(cc.n_layers):
        ced.project_and_encode(Hs, f32(cin.W_kv[l]), f32(cin.W_z[l]))
    dt = time.perf_counter() - t0
    full_s = dt * cc.rows / len(rows)
    flops = 2.0 * cc.rows * cc.d_model * cc.n_layers * (576 + 64)
    out[cc.name] = entry(flops / full_s / 1e12, "TFLOP/s",
                         f"256 evenly spaced rows x {cc.n_layers} layers ({dt:.2f} s: FP64 products, fp32 rounding, "
                         f"FP4 encode of C, bf16 of Z), extrapolated x{cc.rows // 256} to {cc.rows} rows")
    return out


def config_block():
    return {"workload": "csa2_decode_group_b32_ctx128k_full_reindex_reuse", "batch": CFG.B,
            "entries": CFG.N, "context_tokens": CFG.ctx, "heads": CFG.H, "indexer_heads": CFG.H_I,
            "top_k": CFG.K, "n_win": CFG.W, "layers": "FULL,REINDEX,REUSE",
            "kv_format": "e2m1 + e4m3/16 (324 B/entry)", "l2": "flushed between timed steps (256 MiB write)"}


# ---------------------------------------------------------------------------
# Clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        self.gpu_id = gpu_id

    def start(self):
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
ONE_GPU_ONLY = ("one GPU per process and one process per job: the attention and CED kernels load "
                "through TMA cluster multicast, which this library runs in single-GPU calls only")


def run_ours(args):
    rank, _, world = dist_env()
    if world > 1 or args.gpus != 1:
        # refused before CUDA is touched: no kernel of this library runs under more than one rank
        if rank == 0:
            print(json.dumps({"metric": METRIC, "n_gpus": max(world, args.gpus), "unavailable": ONE_GPU_ONLY}),
                  flush=True)
        print(f"bench.py: --gpus {args.gpus} / WORLD_SIZE {world} refused: {ONE_GPU_ONLY}", file=sys.stderr)
        return 0
    world = 1
    import torch
    from cuda.bindings import driver as cu

    import sparse_attention_kv_decode_b300 as csa2

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    L = csa2.lib()
    cfg = CFG
    inp = ci.make_decode_inputs(cfg)
    b16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    t32 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    X = t32(inp.layers[0].X)
    codes, scales = csa2.csa2_encode_kv(X)
    del X
    inp.layers[0].X = None
    nvis, wst, wln = t32(inp.n_visible), t32(inp.win_start), t32(inp.win_len)
    dl = []
    for Lr in inp.layers:
        d = dict(mode=Lr.mode, q=b16(Lr.q), swa=b16(Lr.swa))
        if Lr.mode != ci.REUSE:
            d.update(q_idx=b16(Lr.q_idx), w=t32(Lr.w_idx), z=b16(Lr.z))
        d["o"] = torch.empty((cfg.B, cfg.T, cfg.H, cfg.d_v), dtype=torch.float32, device=dev)
        d["lse"] = torch.empty((cfg.B, cfg.T, cfg.H), dtype=torch.float32, device=dev)
        dl.append(d)
    idx_bufs = [torch.empty((cfg.B, cfg.T, cfg.K), dtype=torch.int32, device=dev) for _ in range(2)]
    ws = csa2.csa2_workspace(cfg.B, cfg.T, cfg.H, cfg.N, cfg.K, device=dev)
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream
    scale = ctypes.c_float(cfg.softmax_scale)
    P = lambda t: t.data_ptr()
    wsp, wsn = P(ws), ws.numel()

    # the step as a list of (name, kind, thunk) C-ABI calls on `stream`: `calls` for the
    # per-call breakdown, `step_calls` for the timed step (with --attn layer one
    # csa2_decode_layer per layer, which is csa2_index_topk + csa2_decode_attention)
    calls, step_calls = [], []
    cur = None
    layer = args.attn == "layer"
    for li, d in enumerate(dl):
        mode = d["mode"]
        if mode != ci.REUSE:
            cur = idx_bufs[li % 2]
            calls.append((f"index_topk[{ci.MODE_NAMES[mode]}]", "index",
                          (lambda d=d, cur=cur, mode=mode: L.csa2_index_topk(
                              mode, cfg.B, cfg.T, cfg.H_I, P(d["q_idx"]), P(d["w"]), P(d["z"]), cfg.N, P(nvis),
                              cfg.K, None, P(cur), None, wsp, wsn, sp))))
        else:
            calls.append(("index_topk[REUSE]", "reuse",
                          (lambda cur=cur: L.csa2_index_topk(2, cfg.B, cfg.T, 0, None, None, None, 0, None,
                                                             cfg.K, P(cur), P(cur), None, None, 0, sp))))
        if layer:
            step_calls.append((f"decode_layer[{ci.MODE_NAMES[mode]}]", "layer",
                               (lambda d=d, cur=cur, mode=mode: L.csa2_decode_layer(
                                   mode, cfg.B, cfg.T, cfg.H, cfg.H_I, P(d["q"]),
                                   P(d["q_idx"]) if mode != ci.REUSE else None,
                                   P(d["w"]) if mode != ci.REUSE else None,
                                   P(d["z"]) if mode != ci.REUSE else None, P(codes), P(scales), cfg.N,
                                   P(nvis) if mode != ci.REUSE else None, cfg.K,
                                   P(cur) if mode == ci.REUSE else None, P(cur), P(d["swa"]), cfg.S, P(wst),
                                   P(wln), cfg.W, cfg.d_v, scale, P(d["o"]), P(d["lse"]), wsp, wsn, sp))))
        if args.attn in ("fused", "layer"):
            calls.append((f"decode_attention[{ci.MODE_NAMES[mode]}]", "attn",
                          (lambda d=d, cur=cur: L.csa2_decode_attention(
                              cfg.B, cfg.T, cfg.H, P(d["q"]), P(codes), P(scales), cfg.N, P(cur), cfg.K,
                              P(d["swa"]), cfg.S, P(wst), P(wln), cfg.W, cfg.d_v, scale, P(d["o"]), P(d["lse"]),
                              wsp, wsn, sp))))
        else:
            calls.append((f"sparse_decode[{ci.MODE_NAMES[mode]}]", "sparse",
                          (lambda d=d, cur=cur: L.csa2_sparse_decode(
                              cfg.B, cfg.T, cfg.H, P(d["q"]), P(codes), P(scales), cfg.N, P(cur), cfg.K, cfg.d_v,
                              scale, P(d["o"]), P(d["lse"]), wsp, wsn, sp))))
            calls.append((f"swa_merge[{ci.MODE_NAMES[mode]}]", "swa",
                          (lambda d=d: L.csa2_swa_merge(
                              cfg.B, cfg.T, cfg.H, P(d["q"]), P(d["swa"]), cfg.S, P(wst), P(wln), cfg.W, cfg.d_v,
                              scale, P(d["o"]), P(d["lse"]), P(d["o"]), P(d["lse"]), wsp, wsn, sp))))
    if not layer:
        step_calls = calls
    launches_per_call = {"index": 2, "reuse": 0, "attn": 1, "sparse": 1, "swa": 1}

    def cuchk(r):
        err = r[0] if isinstance(r, tuple) else r
        if int(err) != 0:
            raise RuntimeError(f"CUDA driver error {err}")
        return r[1] if isinstance(r, tuple) and len(r) > 1 else None

    events = [cuchk(cu.cuEventCreate(0)) for _ in range(len(calls) + 1)]

    def enqueue_step(record=True):
        for i, (name, _, fn) in enumerate(calls if record else step_calls):
            if record:
                cuchk(cu.cuEventRecordWithFlags(events[i], sp, cu.CUevent_record_flags.CU_EVENT_RECORD_EXTERNAL))
            st = fn()
            if st != 0:
                raise RuntimeError(f"{name} returned {st}")
        if record:
            cuchk(cu.cuEventRecordWithFlags(events[-1], sp, cu.CUevent_record_flags.CU_EVENT_RECORD_EXTERNAL))

    # warm once eagerly (sets kernel attributes), then capture the step as a CUDA graph
    with torch.cuda.stream(stream):
        enqueue_step(record=False)
    stream.synchronize()
    st, flags = csa2.csa2_read_device_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags}")
    # the timed graph has no event nodes between the kernels (each kernel may then
    # start while its predecessor drains: programmatic dependent launch); a second
    # graph with an event around every call gives the per-call breakdown
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        enqueue_step(record=False)
    graph_calls = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_calls, stream=stream):
        enqueue_step(record=True)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            flush.fill_(1)
            graph.replay()
            flush.fill_(1)
            graph_calls.replay()
    torch.cuda.synchronize()

    gpu_uuid = None
    try:
        gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if not gpu_uuid.startswith("GPU-"):
            gpu_uuid = "GPU-" + gpu_uuid
    except Exception:
        gpu_uuid = None
    clocks = ClockSampler(gpu_uuid)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for e0, e1 in ev:
            flush.fill_(1)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
    stream.synchronize()
    wall = time.perf_counter() - wall0
    step_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    clk = clocks.stop()
    # per-call breakdown (separate pass, events between the calls)
    per_call = [[] for _ in calls]
    for _ in range(min(args.steps, 200)):
        with torch.cuda.stream(stream):
            flush.fill_(1)
            graph_calls.replay()
        stream.synchronize()
        for i in range(len(calls)):
            per_call[i].append(cuchk(cu.cuEventElapsedTime(events[i], events[i + 1])))
    torch.cuda.synchronize()

    total_s, value = aggregate_over_ranks(sum(step_ms) / 1e3, args.steps, world, dev)
    ms_per_step = total_s * 1e3 / args.steps
    peaks = load_peaks()
    bytes_step = algorithmic_bytes_per_step(cfg)

    # per-call breakdown and roofline of the dominant call
    kinds = {}
    breakdown = []
    for (name, kind, _), ts in zip(calls, per_call):
        avg = statistics.mean(ts) * 1e-3
        breakdown.append({"call": name, "us": round(avg * 1e6, 2)})
        k = kinds.setdefault(kind, [0.0, 0])
        k[0] += avg
        k[1] += 1
    Q = cfg.B * cfg.T
    flops_sparse = 2.0 * Q * cfg.H * cfg.K * (576 + cfg.d_v)
    flops_swa = 2.0 * Q * cfg.H * cfg.W * (576 + cfg.d_v)
    models = {
        "index": ("hbm", Q * cfg.N * KEY_BYTES, "GB/s", peaks["hbm"]),
        "attn": ("tensor", flops_sparse + flops_swa, "TFLOP/s", peaks["bf16"]),
        "sparse": ("tensor", flops_sparse, "TFLOP/s", peaks["bf16"]),
        "swa": ("tensor", flops_swa, "TFLOP/s", peaks["bf16"]),
    }
    dom = max((k for k in kinds if k in models), key=lambda k: kinds[k][0])
    bound, work, unit, peak = models[dom]
    t_launch = kinds[dom][0] / kinds[dom][1]
    achieved = work / t_launch / (1e9 if unit == "GB/s" else 1e12)
    rows = {}
    for k, (b, w, u, pk) in models.items():
        if k in kinds:
            tl = kinds[k][0] / kinds[k][1]
            a = w / tl / (1e9 if u == "GB/s" else 1e12)
            rows[k] = {"bound": b, "achieved": round(a, 2), "peak": pk, "unit": u, "frac": round(a / pk, 4),
                       "us_per_call": round(tl * 1e6, 2)}
    roofline = {"kernel": {"index": "csa2_index_topk (indexer score + top-K select kernels)",
                           "attn": "csa2_decode_attention (attn_tc_kernel, FP4 entries + window)",
                           "sparse": "csa2_sparse_decode (attn_tc_kernel)",
                           "swa": "csa2_swa_merge (attn_tc_kernel)"}[dom],
                "bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "peak_source": peaks["src"],
                "traffic": ncu_traffic({"index": "index_score_kernel<1>", "attn": "attn_tc_kernel<2>",
                                        "sparse": "attn_tc_kernel<0>", "swa": "attn_tc_kernel<1>"}[dom]),
                "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)"}

    pool = None
    if not args.no_pool:
        try:
            pool = run_pool_indexer(args, torch, L, cfg, dl, codes, scales, nvis, idx_bufs, ws, dev, peaks, stream,
                                    flush)
        except Exception as ex:  # reported, not hidden
            pool = {"error": repr(ex)}
    app = None
    if not args.no_pool:
        try:
            app = run_cache_append(args, torch, csa2, cfg, dev, stream, flush)
        except Exception as ex:  # reported, not hidden
            app = {"error": repr(ex)}
    variants = None
    if not args.no_pool:
        try:
            variants = run_step_variants(args, torch, csa2, L, cfg, dl, codes, scales, nvis, wst, wln, idx_bufs,
                                         ws, stream, flush)
        except Exception as ex:  # reported, not hidden
            variants = {"error": repr(ex)}
    others = None
    if not args.no_configs:
        try:
            others = run_other_configs(args, torch, csa2, dev, peaks, flush)
        except Exception as ex:  # reported, not hidden
            others = {"error": repr(ex)}
    ced = None
    if not args.no_ced:
        try:
            ced = run_ced(args, torch, csa2, dev, peaks)
        except Exception as ex:  # reported, not hidden
            ced = {"error": repr(ex)}
    e2e = None if args.no_e2e else run_e2e(args, torch, csa2, L, cfg, dl, codes, scales, nvis, wst, wln, idx_bufs,
                                           ws, world, dev)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        inp.layers[0].X = None
        baselines = cpu_baselines(inp)
        cpu = baselines.pop(cfg.name)
        if others is not None and "error" not in others:
            for name, row in others.items():
                if name in baselines:
                    row["cpu_baseline"] = baselines[name]
        if ced is not None and "error" not in ced:
            ced["cpu_baseline"] = baselines.get(ci.CED_PROJ.name)

    n_launch = sum(launches_per_call[k] for _, k, _ in calls) * args.steps
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16/fp16 mma, fp32 acc (fp4 e2m1+e4m3 cache)", "data": "synthetic",
            "config": config_block(),
            "hbm_gbs_step": round(bytes_step / (ms_per_step * 1e-3) / 1e9, 1),
            "frac_of_8tbs": round(bytes_step / (ms_per_step * 1e-3) / 1e9 / TARGET_HBM_GBS, 4),
            "frac_of_measured_hbm": round(bytes_step / (ms_per_step * 1e-3) / 1e9 / peaks["hbm"], 4),
            "bytes_per_step": bytes_step,
            "roofline": roofline, "roofline_by_call": rows, "calls": breakdown,
            "calls_note": "per-call means from a separate pass with an event between calls",
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clk, "gpu_launches": n_launch,
            "wall_s_timed_loop": round(wall, 3),
            "ced_projection": ced,
            "hierarchical_indexer": pool,
            "cache_append": app,
            "step_variants": variants,
            "other_configs": others,
        }
        print(json.dumps(line), flush=True)
    return 0


def run_pool_indexer(args, torch, L, cfg, dl, codes, scales, nvis, idx_bufs, ws, dev, peaks, stream, flush):
    """The REINDEX layer's selection two ways on the same inputs: the full scan
    (CSA2_MODE_REINDEX) and the hierarchical indexer (CSA2_MODE_REINDEX_POOL), which scores
    only the aligned 8-position blocks of the FULL layer's selection. Device time per call
    (CUDA graph of the one call, events on its stream, L2 flushed between replays) and the
    pool's key bytes as an HBM roofline."""
    li_full = next((i for i, d in enumerate(dl) if d["mode"] == ci.FULL), None)
    li_re = next((i for i, d in enumerate(dl) if d["mode"] == ci.REINDEX), None)
    if li_full is None or li_re is None:
        return None
    d = dl[li_re]
    full_sel = idx_bufs[li_full % 2].clone()
    outs = [torch.empty_like(full_sel) for _ in range(2)]
    sp = stream.cuda_stream
    P = lambda t: t.data_ptr()
    pf = False   # as in csa2_decode_layer

    def call(mode, prev, out):
        if pf:
            return L.csa2_index_topk_prefetch(mode, cfg.B, cfg.T, cfg.H_I, P(d["q_idx"]), P(d["w"]), P(d["z"]), cfg.N,
                                              P(nvis), cfg.K, prev, P(out), None, P(codes), P(scales),
                                              P(ws), ws.numel(), sp)
        return L.csa2_index_topk(mode, cfg.B, cfg.T, cfg.H_I, P(d["q_idx"]), P(d["w"]), P(d["z"]), cfg.N, P(nvis),
                                 cfg.K, prev, P(out), None, P(ws), ws.numel(), sp)

    variants = [("REINDEX", lambda: call(ci.REINDEX, None, outs[0])),
                ("REINDEX_POOL", lambda: call(ci.REINDEX_POOL, P(full_sel), outs[1]))]
    times = {}
    for name, fn in variants:
        with torch.cuda.stream(stream):
            if fn() != 0:
                raise RuntimeError(f"index_topk[{name}] failed")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        ts = []
        n = min(args.steps, 200)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n + 3)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                flush.fill_(1)
                e0.record(stream)
                g.replay()
                e1.record(stream)
        stream.synchronize()
        ts = [e0.elapsed_time(e1) for e0, e1 in evs[3:]]
        times[name] = statistics.mean(ts) * 1e-3
    from sparse_attention_kv_decode_b300 import csa2_read_device_status
    st, flags = csa2_read_device_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags}")

    # pool size per query from the FULL selection: distinct 8-position blocks, visible positions in them
    sel = full_sel.reshape(-1, cfg.K).cpu().numpy()
    nv = nvis.reshape(-1).cpu().numpy().astype(np.int64)
    pooled = 0
    for r in range(sel.shape[0]):
        blk = np.unique(sel[r][sel[r] >= 0] >> 3).astype(np.int64)
        pooled += int(np.clip(nv[r] - 8 * blk, 0, 8).sum())
    Q = cfg.B * cfg.T
    full_bytes = Q * cfg.N * KEY_BYTES
    pool_bytes = pooled * KEY_BYTES
    t_full, t_pool = times["REINDEX"], times["REINDEX_POOL"]
    a_full = full_bytes / t_full / 1e9
    a_pool = pool_bytes / t_pool / 1e9
    return {"call": "csa2_index_topk_prefetch" if pf else "csa2_index_topk",
            "reindex_us": round(t_full * 1e6, 2), "reindex_pool_us": round(t_pool * 1e6, 2),
            "speedup": round(t_full / t_pool, 3),
            "pool_positions_mean": round(pooled / Q, 1), "positions_full_scan": cfg.N,
            "reindex_key_gbs": round(a_full, 1), "reindex_pool_key_gbs": round(a_pool, 1),
            "reindex_pool_frac": round(a_pool / peaks["hbm"], 4), "peak_gbs": peaks["hbm"],
            "launches": {"REINDEX": 2, "REINDEX_POOL": 3},
            "note": "pool = aligned 8-position blocks holding an entry of the FULL layer's selection; "
                    "bytes = pooled visible positions x 128-byte keys"}


def run_cache_append(args, torch, csa2, cfg, dev, stream, flush):
    """csa2_cache_append for the bench's sequences: the FULL layer's append of one token
    (window ring row, the FP4 entry the token completes, its indexer key, n_visible and
    the window bounds), CUDA graph of the one call, L2 flushed between replays. Every
    sequence sits at a token that completes an entry (the costlier of the two kinds of
    step); n_tokens is not advanced so that each replay does the same work."""
    B, N, W = cfg.B, cfg.N, cfg.W
    g = torch.Generator(device=dev).manual_seed(7)
    swa = torch.zeros((B, 2 * W, 576), dtype=torch.bfloat16, device=dev)
    codes, scales = csa2.csa2_kv_cache((B, N), device=dev)
    z = torch.zeros((B, N, 64), dtype=torch.bfloat16, device=dev)
    row = torch.randn((B, 576), generator=g, device=dev).to(torch.bfloat16)
    ent = torch.randn((B, 576), generator=g, device=dev)
    zk = torch.randn((B, 64), generator=g, device=dev).to(torch.bfloat16)
    n_tok = torch.full((B,), 4 * (N // 2) - 1, dtype=torch.int32, device=dev)
    nvis, wst, wln = (torch.zeros(B, dtype=torch.int32, device=dev) for _ in range(3))
    ws = csa2.csa2_workspace(B, 1, 1, 0, 1, device=dev)

    def call():
        csa2.csa2_cache_append(n_tok, swa_row=row, swa_kv=swa, n_win=W, entry_kv=ent, entry_z=zk, kv_codes=codes,
                               kv_scales=scales, z=z, n_visible=nvis, win_start=wst, win_len=wln, advance=False,
                               ws=ws, stream=stream)

    with torch.cuda.stream(stream):
        call()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    n = min(args.steps, 200)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n + 3)]
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            flush.fill_(1)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
    stream.synchronize()
    us = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs[3:]) * 1e3
    st, flags = csa2.csa2_read_device_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags}")
    # per sequence: window row in + 2 rows out, fp32 entry in + 288 + 36 B out, key in + out,
    # n_tokens in, n_visible / win_start / win_len out
    bytes_call = B * (1152 * 3 + 2304 + 324 + 128 * 2 + 4 + 12)
    return {"call": "csa2_cache_append", "sequences": B, "us": round(us, 2), "bytes": bytes_call,
            "gbs": round(bytes_call / (us * 1e-6) / 1e9, 2), "launches": 1,
            "note": "one token per sequence completing an FP4 entry; a few KB per sequence, launch-bound"}


def run_step_variants(args, torch, csa2, L, cfg, dl, codes, scales, nvis, wst, wln, idx_bufs, ws, stream, flush):
    """The timed decode step in two more forms, each as one CUDA graph timed like the step:
    (1) step_with_pool: the REINDEX layer ranks only the FULL layer's candidate pool
        (CSA2_MODE_REINDEX_POOL); (2) step_with_append: before each layer its cache append of
        the step's token (FULL: window row, the FP4 entry the token completes and its key;
        REINDEX: window row and key; REUSE: window row), the layers reading n_visible and
        the window bounds the appends write. The token is 4N-1, the last one of the cache, so
        the layers see the same N entries and W window rows as the step; n_tokens is not
        advanced, so every replay does the same work."""
    P = lambda t: t.data_ptr() if t is not None else None
    sp = stream.cuda_stream
    scale = ctypes.c_float(cfg.softmax_scale)
    wsp, wsn = P(ws), ws.numel()
    B, W = cfg.B, cfg.W

    def layer(d, mode, prev, out, nv, ws_, wl_, swa, s_stride):
        reuse = mode == ci.REUSE
        return L.csa2_decode_layer(mode, cfg.B, cfg.T, cfg.H, cfg.H_I, P(d["q"]),
                                   None if reuse else P(d["q_idx"]), None if reuse else P(d["w"]),
                                   None if reuse else P(d["z"]), P(codes), P(scales), cfg.N,
                                   None if reuse else P(nv), cfg.K, P(prev), P(out), P(swa), s_stride,
                                   P(ws_), P(wl_), W, cfg.d_v, scale, P(d["o"]), P(d["lse"]), wsp, wsn, sp)

    def timed(thunks):
        with torch.cuda.stream(stream):
            for fn in thunks:
                if fn() != 0:
                    raise RuntimeError("step variant call failed")
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for fn in thunks:
                fn()
        n = min(args.steps, 500)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n + 3)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                flush.fill_(1)
                e0.record(stream)
                g.replay()
                e1.record(stream)
        stream.synchronize()
        st, flags = csa2.csa2_read_device_status(ws, stream)
        if st != 0:
            raise RuntimeError(f"device status {st} flags {flags}")
        us = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs[3:]) * 1e3
        return {"us_per_step": round(us, 2), "steps_per_s": round(1e6 / us, 1)}

    modes = [d["mode"] for d in dl]
    out = {}
    if modes == [ci.FULL, ci.REINDEX, ci.REUSE]:
        full_sel, re_sel = idx_bufs[0], idx_bufs[1]
        thunks = [lambda: layer(dl[0], ci.FULL, None, full_sel, nvis, wst, wln, dl[0]["swa"], cfg.S),
                  lambda: layer(dl[1], ci.REINDEX_POOL, full_sel, re_sel, nvis, wst, wln, dl[1]["swa"], cfg.S),
                  lambda: layer(dl[2], ci.REUSE, re_sel, re_sel, nvis, wst, wln, dl[2]["swa"], cfg.S)]
        out["step_with_pool"] = dict(timed(thunks), launches=3 + 3 + 1,
                                     note="FULL -> REINDEX_POOL -> REUSE, csa2_decode_layer per layer")

        g = torch.Generator(device=stream.device).manual_seed(11)
        rings = [torch.zeros((B, 2 * W, 576), dtype=torch.bfloat16, device=stream.device) for _ in dl]
        rows = [torch.randn((B, 576), generator=g, device=stream.device).to(torch.bfloat16) for _ in dl]
        ent = torch.randn((B, 576), generator=g, device=stream.device)
        keys = [torch.randn((B, 64), generator=g, device=stream.device).to(torch.bfloat16) for _ in dl]
        n_tok = torch.full((B,), 4 * cfg.N - 1, dtype=torch.int32, device=stream.device)
        a_nv, a_ws, a_wl = (torch.zeros(B, dtype=torch.int32, device=stream.device) for _ in range(3))

        def app(li, with_entry, with_key):
            return L.csa2_cache_append(B, P(n_tok), 0, 4, P(rows[li]), P(rings[li]), 2 * W, W,
                                       P(ent) if with_entry else None, csa2.F32,
                                       P(keys[li]) if with_key else None, P(codes), P(scales),
                                       P(dl[li]["z"]) if with_key else None, cfg.N, P(a_nv), P(a_ws), P(a_wl),
                                       wsp, wsn, sp)
        thunks = [lambda: app(0, True, True),
                  lambda: layer(dl[0], ci.FULL, None, full_sel, a_nv, a_ws, a_wl, rings[0], 2 * W),
                  lambda: app(1, False, True),
                  lambda: layer(dl[1], ci.REINDEX, None, re_sel, a_nv, a_ws, a_wl, rings[1], 2 * W),
                  lambda: app(2, False, False),
                  lambda: layer(dl[2], ci.REUSE, re_sel, re_sel, a_nv, a_ws, a_wl, rings[2], 2 * W)]
        out["step_with_append"] = dict(timed(thunks), launches=3 + 2 + 2 + 1,
                                       note="csa2_cache_append before each csa2_decode_layer (token 4N-1)")
    return out


def run_other_configs(args, torch, csa2, dev, peaks, flush):
    """The other decode workloads, one csa2_decode_layer(FULL) call each as a CUDA graph
    (inputs resident, L2 flushed between replays): the tiny step (one sequence, 1024
    entries, 16 heads, K = 128; reported in microseconds per call), 4 sequences at 1M
    tokens (262,144 entries), reported against HBM (keys + selected entries + window), and a
    4096-token prefill chunk over 32,768 entries (causal), reported in TFLOP/s (attention
    over the selected entries and the window, plus the indexer, as stated for that
    workload)."""
    out = {}
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream
    L = csa2.lib()
    P = lambda t: t.data_ptr() if t is not None else None
    b16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    t32 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    chosen = [c for c in (args.configs or "").split(",") if c]
    for cfg, steps in ((ci.TINY, min(args.steps, 200)), (ci.DECODE_1M, min(args.steps, 200)),
                       (ci.PREFILL_CHUNK, min(args.steps, 20))):
        if chosen and cfg.name not in chosen:
            continue
        inp = ci.make_decode_inputs(cfg)
        Lr = inp.layers[0]
        X = t32(Lr.X)
        codes, scales = csa2.csa2_encode_kv(X)
        del X
        Lr.X = None
        q, qi, w, z, swa = b16(Lr.q), b16(Lr.q_idx), t32(Lr.w_idx), b16(Lr.z), b16(Lr.swa)
        nvis, wst, wln = t32(inp.n_visible), t32(inp.win_start), t32(inp.win_len)
        idx = torch.empty((cfg.B, cfg.T, cfg.K), dtype=torch.int32, device=dev)
        o = torch.empty((cfg.B, cfg.T, cfg.H, cfg.d_v), dtype=torch.float32, device=dev)
        lse = torch.empty((cfg.B, cfg.T, cfg.H), dtype=torch.float32, device=dev)
        ws = csa2.csa2_workspace(cfg.B, cfg.T, cfg.H, cfg.N, cfg.K, device=dev)
        scale = ctypes.c_float(cfg.softmax_scale)

        def call():
            return L.csa2_decode_layer(ci.FULL, cfg.B, cfg.T, cfg.H, cfg.H_I, P(q), P(qi), P(w), P(z), P(codes),
                                       P(scales), cfg.N, P(nvis), cfg.K, None, P(idx), P(swa), cfg.S, P(wst), P(wln),
                                       cfg.W, cfg.d_v, scale, P(o), P(lse), P(ws), ws.numel(), sp)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            if call() != 0:
                raise RuntimeError(f"{cfg.name}: csa2_decode_layer failed")
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            call()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps + 3)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                flush.fill_(1)
                e0.record(stream)
                g.replay()
                e1.record(stream)
        stream.synchronize()
        st, flags = csa2.csa2_read_device_status(ws, stream)
        if st != 0:
            raise RuntimeError(f"{cfg.name}: device status {st} flags {flags}")
        us = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs[3:]) * 1e3
        row = {"sequences": cfg.B, "query_tokens": cfg.T, "entries": cfg.N, "top_k": cfg.K, "n_win": cfg.W,
               "us_per_call": round(us, 2), "calls_per_s": round(1e6 / us, 1), "timed_calls": steps,
               "launches_per_call": 3}
        if cfg.T == 1:
            byt = algorithmic_bytes_per_step(cfg)
            gbs = byt / (us * 1e-6) / 1e9
            row.update(bytes=byt, gbs=round(gbs, 1), frac_of_8tbs=round(gbs / TARGET_HBM_GBS, 4),
                       frac_of_measured_hbm=round(gbs / peaks["hbm"], 4))
        else:
            Qn = cfg.B * cfg.T
            flop = 2.0 * Qn * cfg.H * (cfg.K + cfg.W) * (576 + cfg.d_v) + 2.0 * Qn * cfg.N * cfg.H_I * 64
            tf = flop / (us * 1e-6) / 1e12
            row.update(flop=flop, tflops=round(tf, 1), frac_of_bf16_peak=round(tf / peaks["bf16"], 4),
                       flop_note="attention over K entries + window (2 Q H (K+W) 1088) + indexer over all "
                                 "N entries (2 Q N H_I 64), as stated for this workload")
        out[cfg.name] = row
        del codes, scales, q, qi, w, z, swa, idx, o, lse, ws, g, inp
        torch.cuda.empty_cache()
    return out


def run_ced(args, torch, csa2, dev, peaks):
    """CED projection, Eq. (1), with the fused FP4 cache write: 32768 x 4096 against
    20 layers x (576 + 64) columns. Timed alone with CUDA events (inputs > L2)."""
    cfg = ci.CED_PROJ
    inp = ci.make_ced_inputs(cfg)
    b16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    h, wkv, wz = b16(inp.H), b16(inp.W_kv), b16(inp.W_z)
    del inp
    codes, scales = csa2.csa2_kv_cache((cfg.n_layers, cfg.rows), device=dev)
    z = torch.empty((cfg.n_layers, cfg.rows, 64), dtype=torch.bfloat16, device=dev)
    ws = csa2.csa2_workspace(0, 0, 0, 0, 0, device=dev)
    stream = torch.cuda.Stream(device=dev)
    L = csa2.lib()
    args_c = (h.data_ptr(), csa2.BF16, cfg.rows, cfg.d_model, wkv.data_ptr(), wz.data_ptr(), cfg.n_layers,
              codes.data_ptr(), scales.data_ptr(), z.data_ptr(), ws.data_ptr(), ws.numel(), stream.cuda_stream)
    for _ in range(3):
        r = L.csa2_encode_kv(*args_c)
        if r != 0:
            return {"error": f"csa2_encode_kv returned {r}"}
    st, flags = csa2.csa2_read_device_status(ws, stream)
    if st != 0:
        return {"error": f"device status {st} flags {flags}"}
    n = 20
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    times = []
    for i in range(n):
        ev[i].record(stream)
        L.csa2_encode_kv(*args_c)
        ev[i + 1].record(stream)
    stream.synchronize()
    times = [ev[i].elapsed_time(ev[i + 1]) * 1e-3 for i in range(n)]
    t = statistics.mean(times)
    flops = 2.0 * cfg.rows * cfg.d_model * cfg.n_layers * (576 + 64)
    tf = flops / t / 1e12
    return {"config": {"workload": cfg.name, "rows": cfg.rows, "d_model": cfg.d_model, "n_layers": cfg.n_layers},
            "value": round(tf, 1), "unit": "TFLOP/s", "ms_per_launch": round(t * 1e3, 4), "launches": n,
            "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16"], "unit": "TFLOP/s",
                         "frac": round(tf / peaks["bf16"], 4), "peak_source": peaks["src"] + " bf16 burst",
                         "frac_of_sustained": round(tf / peaks["bf16_sus"], 4), "traffic": ncu_traffic("ced_proj_kernel")}}


def run_e2e(args, torch, csa2, L, cfg, dl, codes, scales, nvis, wst, wln, idx_bufs, ws, world, dev):
    """Same step through the C ABI with host buffers, as a serving loop runs it: per step,
    one H2D copy of the step's queries (every layer's q, q_idx, w packed in one pinned
    buffer) and one D2H copy of every layer's output (O and LSE packed likewise), no graph,
    one ctypes call per layer with its arguments prepared once. The copies run on their own
    streams with two sets of device I/O buffers, so step i+1's upload and step i-1's
    download overlap step i's kernels."""
    comp = torch.cuda.Stream(device=dev)
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)
    sp = comp.cuda_stream
    scale = ctypes.c_float(cfg.softmax_scale)
    P = lambda t: t.data_ptr()

    def packed(likes):
        """One pinned host buffer and one device buffer holding tensors shaped like `likes`
        (each at a 256-byte offset); returns both buffers and the per-tensor views."""
        offs, total = [], 0
        for t in likes:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        hb = torch.empty(total, dtype=torch.uint8, pin_memory=True)
        db = torch.empty(total, dtype=torch.uint8, device=dev)
        view = lambda buf, o, t: buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        return hb, db, [view(hb, o, t) for o, t in zip(offs, likes)], [view(db, o, t) for o, t in zip(offs, likes)]

    in_keys = [(li, k) for li, d in enumerate(dl) for k in ("q", "q_idx", "w") if k in d]
    out_keys = [(li, k) for li, d in enumerate(dl) for k in ("o", "lse")]
    sets = []   # per buffer set: (host in, device in, host out, device out, per-layer ctypes args)
    for sidx in range(2):
        hi, di, hviews, dviews = packed([dl[li][k] for li, k in in_keys])
        for (li, k), h in zip(in_keys, hviews):
            h.copy_(dl[li][k].cpu())
        ho, do, _, oviews = packed([dl[li][k] for li, k in out_keys])
        dev_of = {key: v for key, v in zip(in_keys + out_keys, dviews + oviews)}
        calls, cur = [], None
        for li, d in enumerate(dl):
            reuse = d["mode"] == ci.REUSE
            if not reuse:
                cur = idx_bufs[li % 2]
            calls.append((d["mode"], cfg.B, cfg.T, cfg.H, cfg.H_I, P(dev_of[li, "q"]),
                          None if reuse else P(dev_of[li, "q_idx"]), None if reuse else P(dev_of[li, "w"]),
                          None if reuse else P(d["z"]), P(codes), P(scales), cfg.N,
                          None if reuse else P(nvis), cfg.K, P(cur) if reuse else None, P(cur),
                          P(d["swa"]), cfg.S, P(wst), P(wln), cfg.W, cfg.d_v, scale, P(dev_of[li, "o"]),
                          P(dev_of[li, "lse"]), P(ws), ws.numel(), sp))
        sets.append((hi, di, ho, do, calls))
    h2d, d2h = sets[0][0].numel(), sets[0][2].numel()
    ev = lambda: torch.cuda.Event()
    # per set: inputs landed / kernels done / outputs copied out
    up_done, comp_done, down_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    started = [False, False]

    def step(i):
        s = i & 1
        hi, di, ho, do, calls = sets[s]
        with torch.cuda.stream(up):
            if started[s]:
                up.wait_event(comp_done[s])      # the kernels of step i-2 have read this set's inputs
            di.copy_(hi, non_blocking=True)
            up_done[s].record(up)
        comp.wait_event(up_done[s])
        if started[s]:
            comp.wait_event(down_done[s])        # step i-2's outputs have left this set
        for a in calls:
            r = L.csa2_decode_layer(*a)
            assert r == 0
        comp_done[s].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(comp_done[s])
            ho.copy_(do, non_blocking=True)
            down_done[s].record(down)
        started[s] = True

    for i in range(max(3, args.warmup // 4)):
        step(i)
    torch.cuda.synchronize(dev)
    n = max(500, args.steps // 4)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # the timed region starts before the first upload and ends after the last download
    e0.record(up)
    comp.wait_stream(up)
    down.wait_stream(up)
    for i in range(n):
        step(i)
    down.wait_stream(comp)
    e1.record(down)
    torch.cuda.synchronize(dev)
    total, value = aggregate_over_ranks(e0.elapsed_time(e1) / 1e3, n, world, dev)
    return {"value": value, "unit": "steps/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n, "note": "csa2_decode_layer calls without a graph; every step one copy of the packed pinned "
                                "host inputs (q, q_idx, w of every layer) and one copy of the packed outputs (O, LSE "
                                "of every layer) on copy streams, two device I/O buffer sets (upload of step i+1 and "
                                "download of step i-1 overlap step i)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-ced", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the 1M-context decode and the prefill-chunk measurements")
    ap.add_argument("--configs", default="",
                    help="comma-separated subset of the other workloads to run (names as in other_configs; "
                         "default: all)")
    ap.add_argument("--no-pool", action="store_true",
                    help="skip the side measurements (REINDEX vs REINDEX_POOL, csa2_cache_append)")
    ap.add_argument("--attn", choices=["layer", "fused", "two-call"], default="layer",
                    help="per layer: one csa2_decode_layer call (the selection, then the attention); "
                         "csa2_index_topk + csa2_decode_attention; or "
                         "csa2_index_topk + csa2_sparse_decode + csa2_swa_merge")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    try:
        if args.impl == "reference":
            return run_reference(args)
        return run_ours(args)
    finally:
        if _POOL is not None:
            _POOL.terminate()


if __name__ == "__main__":
    sys.exit(main())
