"""Benchmark of the paged K16/V8 decode hot path on GB300 (one JSON line on rank 0).

Default workload: asymmetric-KV decode at the pages' shape -- batch 32, context
8192 + U{0..127}, 32 query / 8 KV heads, head dim 128, page size 16, NHD pages, K FP16,
V FP8 E4M3 with a per-layer scale, 36 layers per step (36 distinct layer pools, 29 GB,
so every layer call streams from HBM: inputs larger than L2, no flush needed).
A step is one decode call per layer (one kernel launch each: split work + fused merge).

value        KV GB/s: algorithmic bytes of all layer calls / device time (CUDA events)
e2e          the same metric through the C ABI with the per-step inputs (q, block
             tables, seq_lens) copied host->device from pinned memory and the outputs
             copied back inside the timed region (the KV cache is resident state); one
             packed copy per layer on a copy stream, overlapping the other layers' decode
roofline     split kernel's algorithmic bytes / its own event-timed duration, against
             the measured HBM copy peak
cpu_baseline the float64 oracle on the host cores, on a sample of the same workload
decode_workloads  the mixed-fidelity batch, its all-FP16 control, the TARGET/BASE mix
             and high concurrency, each on its own pools (per layer under programmatic
             launch, and per launch alone)
companions   gather, demotion (E4M3, BASE), promotion, append and FP16 prefill on their
             workloads (32 x 8192-token prompts; 8 x 8192 for prefill)

--impl reference times the float64 oracle (there is no other reference program) on the
host cores, on bounded samples of the same workload.
"""

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

WORKLOADS = {
    "pages_shape": dict(desc="asymmetric-KV decode at the pages' shape", batch=32, q_heads=32,
                        kv_heads=8, head_dim=128, layers=36, v_format="e4m3", scale_mode=0,
                        context="8192+U{0..127}"),
    "high_concurrency": dict(desc="high-concurrency decode", batch=256, q_heads=32, kv_heads=4,
                             head_dim=128, layers=48, v_format="e4m3", scale_mode=0,
                             context="20% U[1,63], rest ceil(LogNormal(ln 2048, 1)) <= 32768"),
    "mixed": dict(desc="mixed-fidelity batch", batch=64, q_heads=32, kv_heads=8, head_dim=128,
                  layers=2, v_format="mixed", scale_mode=1, context="U[512, 32768]"),
    "mixed_fp16_control": dict(desc="mixed-fidelity batch, all-FP16 control", batch=64, q_heads=32,
                               kv_heads=8, head_dim=128, layers=2, v_format="fp16", scale_mode=0,
                               context="U[512, 32768]"),
    "mixed_base": dict(desc="mixed-fidelity batch, ElasticKV TARGET/BASE pages", batch=64, q_heads=32,
                       kv_heads=8, head_dim=128, layers=2, v_format="mixed", scale_mode=1,
                       context="U[512, 32768]", p_compact=0.0, p_base=0.5),
}


def lens_for(name):
    from mixed_precision_paged_gb300 import workloads as wl
    if name == "pages_shape":
        return wl.pages_shape_lens()
    if name == "high_concurrency":
        return wl.high_concurrency_lens()
    return wl.mixed_lens()


def load_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def _production_source(data):
    """Source text as the production library compiles it: blocks that only the tests'
    library builds (#ifdef EKV_TEST_WAIT_TIMEOUT ... #endif) are dropped with the blank
    line after them; where such a block has an #else branch, that branch is kept."""
    out, state, drop_blank = [], 0, False
    for line in data.decode().splitlines(keepends=True):
        if line.startswith("#ifdef EKV_TEST_WAIT_TIMEOUT"):
            state = 1
            continue
        if state:
            if line.startswith("#else"):
                state = 2
            elif line.startswith("#endif"):
                state, drop_blank = 0, state == 1
            elif state == 2:
                out.append(line)
            continue
        if drop_blank and line.strip() == "":
            drop_blank = False
            continue
        drop_blank = False
        out.append(line)
    return "".join(out).encode()


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ["decode_mma.cu", "pipeline.cuh", "decode.cuh", "common.cuh", "pool_maps.h", "decode_simt.cu"]:
        h.update(_production_source(open(os.path.join(ROOT, "mixed_precision_paged_gb300", "csrc", f), "rb").read()))
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per split launch from profiles/traffic.json (written from the committed
    ncu summaries), when it was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))["decode_split_mma"][workload]
    except (OSError, ValueError, KeyError):
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return float(rec["traffic_bytes_per_launch"])
    except (KeyError, TypeError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------- oracle (CPU)

def _oracle_unit(args):
    """One sequence through the float64 oracle (runs in a single-threaded worker)."""
    from oracle import decode as od
    q, k, v, scales, scale_mode, modes, uniform_mode, L = args
    n = k.shape[0]
    bt = np.arange(n, dtype=np.int32)[None, :]
    out, lse = od.paged_decode(q[None], k, v, scales, scale_mode, modes, uniform_mode, bt,
                               np.array([L], dtype=np.int32))
    return out[0]


def _init_worker():
    os.environ["OMP_NUM_THREADS"] = "1"


def oracle_pool(cores):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    pool = ctx.Pool(cores, initializer=_init_worker)
    os.environ.clear()
    os.environ.update(env)
    return pool


def host_units(case_np, seqs):
    """Per-sequence oracle inputs with the sequence's pages renumbered 0..n-1."""
    units = []
    for b in seqs:
        L = int(case_np.seq_lens[b])
        n = (L + 15) // 16
        pages = case_np.block_table[b, :n]
        scales = case_np.v_scales if case_np.scale_mode == 0 else case_np.v_scales[pages]
        modes = None if case_np.page_mode is None else case_np.page_mode[pages]
        units.append((case_np.q[b], case_np.k_pages[pages], case_np.v_pages[pages], scales,
                      case_np.scale_mode, modes, case_np.uniform_mode, L))
    return units


def device_case_to_host(case, seqs):
    """Host copies of the arrays the oracle needs for sequences `seqs` only."""
    from mixed_precision_paged_gb300 import workloads as wl
    import torch
    bt = case.block_table.cpu().numpy()
    lens = case.seq_lens.cpu().numpy()
    need = sorted({int(p) for b in seqs for p in bt[b, : (int(lens[b]) + 15) // 16]})
    remap = np.full(case.num_pages, -1, dtype=np.int64)
    remap[need] = np.arange(len(need))
    idx = torch.as_tensor(need, device=case.k_pages.device)
    k = case.k_pages.index_select(0, idx).cpu().numpy()
    v = case.v_pages.index_select(0, idx).cpu().numpy()
    sc = case.v_scales.cpu().numpy() if case.scale_mode == 0 else case.v_scales.index_select(0, idx).cpu().numpy()
    pm = None if case.page_mode is None else case.page_mode.index_select(0, idx).cpu().numpy()
    bt2 = np.where(bt >= 0, remap[np.clip(bt, 0, case.num_pages - 1)], 0).astype(np.int32)
    return wl.DecodeCase(q=case.q.cpu().numpy(), k_pages=k, v_pages=v, v_scales=sc,
                         scale_mode=case.scale_mode, page_mode=pm, uniform_mode=case.uniform_mode,
                         block_table=bt2, seq_lens=lens, num_q_heads=case.num_q_heads,
                         num_kv_heads=case.num_kv_heads, head_dim=case.head_dim)


def cpu_baseline(cases, wk, target_s=15.0):
    """Time the oracle on whole sequences of the first layers until ~target_s of CPU
    work has been sampled (one single-threaded spawn worker per host core)."""
    from mixed_precision_paged_gb300 import roofline as rf
    cores = os.cpu_count() or 1
    pool = oracle_pool(cores)
    try:
        # calibrate on one sequence
        c0 = device_case_to_host(cases[0], [0])
        t0 = time.perf_counter()
        pool.map(_oracle_unit, host_units(c0, [0]))
        per_seq = time.perf_counter() - t0
        n_seq_total = max(1, int(target_s / max(per_seq, 1e-3)))
        units, lens = [], []
        li = 0
        while len(units) < n_seq_total and li < len(cases):
            B = cases[li].batch
            take = list(range(min(B, n_seq_total - len(units))))
            hc = device_case_to_host(cases[li], take)
            units += host_units(hc, take)
            lens += [int(hc.seq_lens[b]) for b in take]
            li += 1
        t0 = time.perf_counter()
        pool.map(_oracle_unit, units, chunksize=1)
        wall = time.perf_counter() - t0
    finally:
        pool.close()
        pool.join()
    vb = 1 if wk["v_format"] == "e4m3" else 2
    nbytes = rf.decode_bytes(lens, wk["q_heads"], wk["kv_heads"], wk["head_dim"], vb,
                             per_page_scales=False)["total"] if wk["v_format"] != "mixed" else None
    if nbytes is None:
        nbytes = sum(l * wk["kv_heads"] * wk["head_dim"] * 3 for l in lens)
    return {"value": nbytes / wall / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(units)} whole sequences (layers 0..{li - 1}), float64 numpy oracle, "
                      f"{cores} single-threaded spawn workers, {wall:.2f} s wall"}


# ----------------------------------------------------------------- reference arm

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from mixed_precision_paged_gb300 import roofline as rf
    from mixed_precision_paged_gb300 import workloads as wl
    wk = WORKLOADS[args.workload]
    cores = os.cpu_count() or 1
    lens_all = lens_for(args.workload)
    n = min(len(lens_all), cores)
    lens = lens_all[:n]
    case = wl.make_decode_case(lens, wk["q_heads"], wk["kv_heads"], wk["head_dim"],
                               v_format=wk["v_format"], scale_mode=wk["scale_mode"],
                               seed=args.seed, poison=False)
    units = host_units(case, range(n))
    vb = 1 if wk["v_format"] == "e4m3" else 2
    nbytes = rf.decode_bytes(lens, wk["q_heads"], wk["kv_heads"], wk["head_dim"], vb,
                             per_page_scales=False)["total"]
    pool = oracle_pool(cores)
    try:
        for _ in range(args.warmup):
            pool.map(_oracle_unit, units, chunksize=1)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            pool.map(_oracle_unit, units, chunksize=1)
        wall = time.perf_counter() - t0
    finally:
        pool.close()
        pool.join()
    value = nbytes * args.steps / wall / 1e9
    sample = (f"each step: {n} of the workload's sequences (one layer), float64 numpy oracle, "
              f"{cores} single-threaded spawn workers")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": wall / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(args, wk),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


METRIC = "paged K16/V8 decode attention: KV GB/s and % of GB300 HBM peak; tokens/s"


def config_of(args, wk):
    return {"workload": wk["desc"], "batch": wk["batch"], "context": wk["context"],
            "q_heads": wk["q_heads"], "kv_heads": wk["kv_heads"], "head_dim": wk["head_dim"],
            "page_size": 16, "layers": args.layers or wk["layers"],
            "kv_format": {"e4m3": "K fp16 / V e4m3, per-layer scale",
                          "fp16": "K fp16 / V fp16",
                          "mixed": "K fp16 / V per page fp16 or e4m3 (p=0.5), per-(page, head) scale"}[wk["v_format"]],
            "l2": "inputs larger than L2: distinct layer pools streamed in turn"
                  if (args.layers or wk["layers"]) > 1 else "L2 flushed (1 GiB read) between steps",
            "parallelism": f"dp{args.gpus} (independent batches per GPU, no collective)",
            "launch": ("programmatic dependent launch: each layer call's prologue and first page fills "
                       "overlap the previous call's tail" if args.pdl and args.variant == 0
                       else "plain stream order")}


# ---------------------------------------------------------------------- companions

def companions(ekv, torch, peaks):
    """Gather (4 chunks of 8 prompts into a 4,096-page workspace) and demotion of 50% of
    16,384 FP16 value pages, on the 32 x 8192-token gather/demote workload."""
    from mixed_precision_paged_gb300 import roofline as rf
    from mixed_precision_paged_gb300 import workloads as wl
    H, D, S = 8, 128, 16
    gd = wl.device_gather_demote_case(seed=1004)
    P = gd.k_pages.shape[0]
    k, v8, sc, bt = gd.k_pages, gd.v8_pages, gd.v_scales, gd.block_table
    ws_k = torch.empty((gd.ws_pages, S, H, D), dtype=torch.float16, device="cuda")
    ws_v = torch.empty_like(ws_k)
    idx = torch.empty((gd.ws_pages,), dtype=torch.int32, device="cuda")
    ctx = ekv.Context(H, H, D, 1)
    chunks = gd.chunks

    gctx = ekv.Context(H, H, D, 1, pdl=True)         # the chunks of an admission back to back

    def gather_all(c):
        for pr in chunks:
            ekv.ekv_gather_prefill(c.handle, k, v8, v8.shape[1], P, sc, 1, None, 1, bt, bt.shape[1], bt.shape[0],
                                   pr, ws_k, ws_v, idx, gd.ws_pages)
    reps = 10
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_gather = {}
    for name, c in (("pdl", gctx), ("plain", ctx)):
        for _ in range(3):
            gather_all(c)
        torch.cuda.synchronize()
        s.record()
        for _ in range(reps):
            gather_all(c)
        e.record()
        torch.cuda.synchronize()
        t_gather[name] = s.elapsed_time(e) / reps
    gerr = gctx.error()
    gctx.close()
    t_g = t_gather["pdl"]
    gb = rf.gather_bytes(P, P, H, D, per_page_scales=True)
    # demotion: FP16 pool N(0, 2), half of the pages
    v16b = gd.v16_pages
    work = torch.empty_like(v16b)
    mode = torch.zeros(P, dtype=torch.uint8, device="cuda")
    scale_out = torch.zeros((P, H), dtype=torch.float32, device="cuda")
    ids = gd.demote_ids
    g = torch.Generator(device="cuda")
    g.manual_seed(1005)
    flush = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    ts = []
    for rep in range(8):
        # fresh FP16 pages, then a 1 GiB read so that none of them is left in L2; no
        # host synchronisation before the start event, so the stream is busy when the
        # demotion is enqueued and the host's launch time is not counted
        work.copy_(v16b)
        mode.zero_()
        flush.sum()
        s.record()
        ekv.ekv_demote_pages(ctx.handle, work, work.shape[1], P, ids, P // 2, mode, scale_out)
        e.record()
        torch.cuda.synchronize()
        if rep >= 3:
            ts.append(s.elapsed_time(e))
    t_d = float(np.median(ts))
    # BASE: demote the same pages to BASE with a low-byte backing, then promote back
    low = torch.empty((P // 2, S * H * D), dtype=torch.uint8, device="cuda")
    tb, tp = [], []
    for rep in range(8):
        work.copy_(v16b)
        mode.zero_()
        flush.sum()
        s.record()
        ekv.ekv_demote_pages_base(ctx.handle, work, work.shape[1], P, ids, P // 2, mode, low)
        e.record()
        flush.sum()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record()
        ekv.ekv_promote_pages(ctx.handle, work, work.shape[1], P, ids, P // 2, mode, low)
        e2.record()
        torch.cuda.synchronize()
        if rep >= 3:
            tb.append(s.elapsed_time(e))
            tp.append(s2.elapsed_time(e2))
    exact = bool(torch.equal(work, v16b))
    # FP16 causal prefill over the last gathered chunk (8 prompts x 8192 tokens in the
    # 4,096-page workspace), random FP16 queries
    n_pr, L_pr = 8, 512 * S
    qp = torch.randn((n_pr * L_pr, H * 4, D), generator=g, device="cuda").to(torch.float16)
    outp = torch.empty_like(qp)
    cu_p = torch.arange(0, (n_pr + 1) * L_pr, L_pr, dtype=torch.int32, device="cuda")
    po_p = torch.arange(0, n_pr * 512, 512, dtype=torch.int32, device="cuda")
    t_pf, perr, outs = {}, {}, {}
    for variant, name in ((0, "tcgen05"), (1, "mma_sync")):
        pctx = ekv.Context(H * 4, H, D, 1, variant=variant)
        ekv.ekv_prefill_attention(pctx.handle, qp, ws_k, ws_v, 4096, cu_p, po_p, n_pr, L_pr, 0.0, outp)
        torch.cuda.synchronize()
        tps = []
        for _ in range(3):
            flush.sum()                                  # the GPU is busy while the call is submitted
            s.record()
            ekv.ekv_prefill_attention(pctx.handle, qp, ws_k, ws_v, 4096, cu_p, po_p, n_pr, L_pr, 0.0, outp)
            e.record()
            torch.cuda.synchronize()
            tps.append(s.elapsed_time(e))
        t_pf[name] = float(np.median(tps))
        perr[name] = list(pctx.error())
        outs[name] = outp.clone()
        pctx.close()
    pf_flop = rf.prefill_flops([L_pr] * n_pr, H * 4, D)
    pf_agree = float((outs["tcgen05"].float() - outs["mma_sync"].float()).abs().max())
    del outs
    del qp, outp
    # cache writer: one new token for each of the 32 sequences per call (latency-bound)
    k_new = torch.randn((32, H, D), generator=g, device="cuda").to(torch.float16)
    v_new = torch.randn((32, H, D), generator=g, device="cuda").to(torch.float16)
    pos = torch.full((32,), 512 * 16 - 1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        ekv.ekv_append_kv(ctx.handle, k_new, v_new, k, v8, v8.shape[1], P, sc, 1, None, 1, bt, 512, pos, 32)
    torch.cuda.synchronize()
    s.record()
    for _ in range(100):
        ekv.ekv_append_kv(ctx.handle, k_new, v_new, k, v8, v8.shape[1], P, sc, 1, None, 1, bt, 512, pos, 32)
    e.record()
    torch.cuda.synchronize()
    t_a_host = s.elapsed_time(e) / 100               # bound by the Python call rate
    # the device time per call: 100 calls captured in one CUDA graph and replayed
    t_a = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(100):
                ekv.ekv_append_kv(ctx.handle, k_new, v_new, k, v8, v8.shape[1], P, sc, 1, None, 1, bt, 512, pos, 32)
        graph.replay()
        torch.cuda.synchronize()
        s.record()
        graph.replay()
        e.record()
        torch.cuda.synchronize()
        t_a = s.elapsed_time(e) / 100
    except Exception:
        t_a = None
    t_b, t_p = float(np.median(tb)), float(np.median(tp))
    bb = rf.base_transition_bytes(P // 2, H, D)
    del flush, low
    db = rf.demote_bytes(P // 2, H, D)
    err = ctx.error()
    hbm = peaks["hbm_gbs"]
    out = {"workload": "32 prompts x 8192 tokens (16,384 pages, 8 KV heads, D 128)",
           "gather": {"ms": t_g, "GB/s": gb / t_g / 1e6, "frac_of_measured_hbm": gb / t_g / 1e6 / hbm,
                      "bytes": gb, "what": "16,384 pages in 4 chunks of 4,096 into the FP16 workspace, the "
                                           "chunk calls back to back under programmatic dependent launch",
                      "plain_stream_order": {"ms": t_gather["plain"], "GB/s": gb / t_gather["plain"] / 1e6,
                                             "frac_of_measured_hbm": gb / t_gather["plain"] / 1e6 / hbm},
                      "device_error": list(gerr)},
           "demote": {"ms": t_d, "GB/s": db / t_d / 1e6, "frac_of_measured_hbm": db / t_d / 1e6 / hbm,
                      "bytes": db, "what": "8,192 of 16,384 FP16 value pages -> E4M3 + scales"},
           "demote_base": {"ms": t_b, "GB/s": bb / t_b / 1e6, "frac_of_measured_hbm": bb / t_b / 1e6 / hbm,
                           "bytes": bb, "what": "the same 8,192 pages -> BASE high bytes + low-byte backing"},
           "promote": {"ms": t_p, "GB/s": bb / t_p / 1e6, "frac_of_measured_hbm": bb / t_p / 1e6 / hbm,
                       "bytes": bb, "what": "BASE -> TARGET from the backing", "exact_round_trip": exact},
           "prefill": {"ms": t_pf["tcgen05"], "TFLOP/s": pf_flop / t_pf["tcgen05"] / 1e9, "flop": pf_flop,
                       "frac_of_measured_bf16": pf_flop / t_pf["tcgen05"] / 1e9 / peaks["bf16_tflops"],
                       "what": "causal FP16 prefill, 8 prompts x 8192 tokens, 32/8 heads, D 128, over the "
                               "4,096-page workspace (tcgen05 MMA, TMEM accumulators, TMA)",
                       "mma_sync": {"ms": t_pf["mma_sync"], "TFLOP/s": pf_flop / t_pf["mma_sync"] / 1e9},
                       "max_abs_diff_between_kernels": pf_agree, "device_error": perr},
           "append": {"us": None if t_a is None else t_a * 1e3,
                      "GB/s": None if t_a is None else rf.append_bytes(32, H, D, 1) / t_a / 1e6,
                      "us_python_loop": t_a_host * 1e3, "bytes": rf.append_bytes(32, H, D, 1),
                      "what": "one token for each of 32 sequences into E4M3 pages; us = device time per call "
                              "(100 calls replayed from one CUDA graph), us_python_loop = back-to-back calls "
                              "from Python (host-bound)"},
           "device_error": list(err)}
    ctx.close()
    return out


# ------------------------------------------------------------ other decode workloads

def layer_bytes(wk, lens, cases):
    """Algorithmic bytes of each layer call of a workload (roofline.decode_bytes)."""
    from mixed_precision_paged_gb300 import roofline as rf
    Hq, Hkv, D = wk["q_heads"], wk["kv_heads"], wk["head_dim"]
    per_call = []
    for c in cases:
        if wk["v_format"] == "mixed":
            modes = c.page_mode.cpu().numpy()
            bt = c.block_table.cpu().numpy()
            code = {0: 2, 1: 1, 2: -1}                  # TARGET, E4M3, BASE (see decode_bytes)
            vbp = [[code[int(modes[bt[b, j]])] for j in range((l + 15) // 16)] for b, l in enumerate(lens)]
            per_call.append(rf.decode_bytes(lens, Hq, Hkv, D, vbp, per_page_scales=True))
        else:
            per_call.append(rf.decode_bytes(lens, Hq, Hkv, D, 1 if wk["v_format"] == "e4m3" else 2,
                                            per_page_scales=False))
    return per_call


def decode_workloads(ekv, torch, peaks, steps, warmup, seed):
    """The other decode configurations, each on its own layer pools drawn with the seeds
    the full-size parity tests check: the mixed-fidelity batch (p = 0.5 TARGET / E4M3),
    its all-FP16 control, the TARGET / BASE mix (2 layers each, 3.8-4.4 GB per layer) and
    high concurrency (48 layers, 51 GB). Per workload: the step of all layer calls under
    programmatic dependent launch (us per layer, GB/s, tokens/s), and each call alone in
    plain stream order (the library's per-launch events)."""
    from mixed_precision_paged_gb300 import workloads as wl
    hbm = float(peaks["hbm_gbs"])
    res = {}
    for name in ("mixed", "mixed_fp16_control", "mixed_base", "high_concurrency"):
        wk = WORKLOADS[name]
        lens = lens_for(name)
        B, Hq, Hkv, D, layers = len(lens), wk["q_heads"], wk["kv_heads"], wk["head_dim"], wk["layers"]
        cases = [wl.device_decode_case(lens, Hq, Hkv, D, v_format=wk["v_format"], scale_mode=wk["scale_mode"],
                                       seed=seed + 7919 * l, p_compact=wk.get("p_compact", 0.5),
                                       p_base=wk.get("p_base", 0.0)) for l in range(layers)]
        per_call = layer_bytes(wk, lens, cases)
        step_bytes = sum(x["total"] for x in per_call)
        split_bytes = float(np.mean([x["split"] for x in per_call]))
        ctx = ekv.Context(Hq, Hkv, D, B, pdl=True)
        outs = [torch.empty((B, Hq, D), dtype=torch.float16, device="cuda") for _ in range(layers)]
        stream = torch.cuda.current_stream()

        def step():
            for l in range(layers):
                ctx.decode(cases[l], outs[l], stream=stream)
        n_steps = max(steps, 10) if layers > 2 else max(steps, 20)
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(n_steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        ms_step = t0.elapsed_time(t1) / n_steps
        ekv.ekv_set_pdl(ctx.handle, 0)                   # each launch alone, between its events
        ekv.ekv_profile_enable(ctx.handle, True)
        ekv.ekv_profile_read(ctx.handle)
        for _ in range(max(1, 40 // layers)):
            step()
        torch.cuda.synchronize()
        split_ms, split_n = ekv.ekv_profile_read(ctx.handle)
        err = ctx.error()
        ctx.close()
        gbs = step_bytes / (ms_step / 1e3) / 1e9
        launch_ms = split_ms / split_n
        res[name] = {
            "workload": wk["desc"], "batch": B, "context": wk["context"], "q_heads": Hq, "kv_heads": Hkv,
            "head_dim": D, "layers": layers, "kv_format": wk["v_format"], "steps": n_steps,
            "us_per_layer": ms_step / layers * 1e3, "GB/s": gbs, "frac_of_measured_hbm": gbs / hbm,
            "frac_of_8tbs_spec": gbs / 8000.0,
            "tokens_per_s": B / (ms_step / 1e3) if layers > 2 else B / (ms_step / layers / 1e3),
            "tokens_per_s_unit": (f"sequences / s, one step = {layers} layer calls" if layers > 2
                                  else "sequences / s per layer call"),
            "per_launch_plain_order": {"us": launch_ms * 1e3, "GB/s": split_bytes / (launch_ms / 1e3) / 1e9,
                                       "frac_of_measured_hbm": split_bytes / (launch_ms / 1e3) / 1e9 / hbm},
            "traffic_bytes_per_launch": profiled_traffic(name),
            "device_error": list(err)}
        del cases, outs
        torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- main

def run_prefill_only(args):
    """The FP16 causal prefill alone (32/8 heads, D 128) on PROMPTS x TOKENS over a
    workspace of exactly their pages; prints one JSON line (ms per call, TFLOP/s)."""
    import torch
    from mixed_precision_paged_gb300 import build
    build.ensure_built()
    from mixed_precision_paged_gb300 import ekv
    from mixed_precision_paged_gb300 import roofline as rf
    n, L = args.prefill_only
    Hq, Hkv, D = 32, 8, 128
    g = torch.Generator(device="cuda")
    g.manual_seed(args.seed)
    pages = (L + 15) // 16
    ws_k = torch.randn((n * pages, 16, Hkv, D), generator=g, device="cuda").to(torch.float16)
    ws_v = torch.randn((n * pages, 16, Hkv, D), generator=g, device="cuda").to(torch.float16)
    q = torch.randn((n * L, Hq, D), generator=g, device="cuda").to(torch.float16)
    out = torch.empty_like(q)
    cu = torch.arange(0, (n + 1) * L, L, dtype=torch.int32, device="cuda")
    po = torch.arange(0, n * pages, pages, dtype=torch.int32, device="cuda")
    ctx = ekv.Context(Hq, Hkv, D, 1, variant=args.variant)
    for _ in range(args.warmup):
        ekv.ekv_prefill_attention(ctx.handle, q, ws_k, ws_v, n * pages, cu, po, n, L, 0.0, out)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.steps):
        ekv.ekv_prefill_attention(ctx.handle, q, ws_k, ws_v, n * pages, cu, po, n, L, 0.0, out)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / args.steps
    flop = rf.prefill_flops([L] * n, Hq, D)
    peaks, src = load_peaks()
    print(json.dumps({"prefill_only": f"{n} x {L}", "variant": args.variant, "ms": ms,
                      "TFLOP/s": flop / ms / 1e9, "frac_of_bf16": flop / ms / 1e9 / peaks["bf16_tflops"],
                      "peak_source": src, "device_error": list(ctx.error())}))
    ctx.close()


def run_gather_only(args):
    """The compact-prefill gather alone on the gather/demotion workload (16,384 pages in 4
    chunks of 4,096 into one workspace, chunk calls back to back under programmatic
    dependent launch, then in plain stream order); one JSON line (ms per 4 chunks, GB/s)."""
    import torch
    from mixed_precision_paged_gb300 import build
    build.ensure_built()
    from mixed_precision_paged_gb300 import ekv
    from mixed_precision_paged_gb300 import roofline as rf
    from mixed_precision_paged_gb300 import workloads as wl
    gd = wl.device_gather_demote_case(seed=1004)
    P, S, H, D = gd.k_pages.shape
    ws_k = torch.empty((gd.ws_pages, S, H, D), dtype=torch.float16, device="cuda")
    ws_v = torch.empty_like(ws_k)
    idx = torch.empty((gd.ws_pages,), dtype=torch.int32, device="cuda")
    bt = gd.block_table
    res = {}
    for name, pdl in (("pdl", True), ("plain", False)):
        ctx = ekv.Context(H, H, D, 1, pdl=pdl)

        def gather_all():
            for pr in gd.chunks:
                ekv.ekv_gather_prefill(ctx.handle, gd.k_pages, gd.v8_pages, gd.v8_pages.shape[1], P, gd.v_scales, 1,
                                       None, 1, bt, bt.shape[1], bt.shape[0], pr, ws_k, ws_v, idx, gd.ws_pages)
        for _ in range(args.warmup):
            gather_all()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(args.steps):
            gather_all()
        e.record()
        torch.cuda.synchronize()
        res[name] = s.elapsed_time(e) / args.steps
        res[name + "_device_error"] = list(ctx.error())
        ctx.close()
    gb = rf.gather_bytes(P, P, H, D, per_page_scales=True)
    peaks, src = load_peaks()
    print(json.dumps({"gather_only": "16,384 pages in 4 chunks of 4,096", "bytes": gb,
                      "ms_pdl": res["pdl"], "GB/s_pdl": gb / res["pdl"] / 1e6,
                      "ms_plain": res["plain"], "GB/s_plain": gb / res["plain"] / 1e6,
                      "frac_of_measured_hbm_pdl": gb / res["pdl"] / 1e6 / peaks["hbm_gbs"], "peak_source": src,
                      "device_error": [res["pdl_device_error"], res["plain_device_error"]]}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ekv", choices=["ekv", "reference"])
    ap.add_argument("--workload", default="pages_shape", choices=sorted(WORKLOADS))
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling)")
    ap.add_argument("--variant", type=int, default=0, help="0 tensor-core, 1 CUDA-core consumer")
    ap.add_argument("--pdl", type=int, default=1, choices=[0, 1],
                    help="programmatic dependent launch between the layer calls (tensor-core consumer)")
    ap.add_argument("--seed", type=int, default=1002)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-companions", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--prefill-only", type=int, nargs=2, metavar=("PROMPTS", "TOKENS"),
                    help="time only the FP16 causal prefill on PROMPTS x TOKENS (profiling)")
    ap.add_argument("--gather-only", action="store_true",
                    help="time only the compact-prefill gather on its workload (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.prefill_only:
        return run_prefill_only(args)
    if args.gather_only:
        return run_gather_only(args)

    import torch
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from mixed_precision_paged_gb300 import build
    if rank == 0:
        build.ensure_built()
    if world > 1:
        dist.barrier()
    from mixed_precision_paged_gb300 import ekv
    from mixed_precision_paged_gb300 import roofline as rf
    from mixed_precision_paged_gb300 import workloads as wl

    wk = WORKLOADS[args.workload]
    layers = args.layers or wk["layers"]
    lens = lens_for(args.workload)
    B, Hq, Hkv, D = len(lens), wk["q_heads"], wk["kv_heads"], wk["head_dim"]
    cases = [wl.device_decode_case(lens, Hq, Hkv, D, v_format=wk["v_format"], scale_mode=wk["scale_mode"],
                                   seed=args.seed + 7919 * (rank * 1000 + l), p_compact=wk.get("p_compact", 0.5),
                                   p_base=wk.get("p_base", 0.0)) for l in range(layers)]
    torch.cuda.synchronize()
    # algorithmic bytes per layer call
    per_call = layer_bytes(wk, lens, cases)
    step_bytes = sum(x["total"] for x in per_call)
    split_bytes = float(np.mean([x["split"] for x in per_call]))

    pdl = bool(args.pdl) and args.variant == 0
    ctx = ekv.Context(Hq, Hkv, D, B, variant=args.variant, pdl=pdl)
    outs = [torch.empty((B, Hq, D), dtype=torch.float16, device="cuda") for _ in range(layers)]
    stream = torch.cuda.current_stream()
    # one-layer runs evict L2 between steps by reading 1 GiB (a read leaves no dirty
    # lines whose write-back would land inside the next timed decode)
    flush = torch.ones(1 << 28, dtype=torch.int32, device="cuda") if layers == 1 else None

    def step():
        if flush is not None:
            flush.sum()
        for l in range(layers):
            ctx.decode(cases[l], outs[l], stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("ekv_timed")
    t_start.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clock_rec = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    if flush is not None:       # the flush writes are not decode work: time them alone
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(args.steps):
            flush.sum()
        f1.record(stream)
        torch.cuda.synchronize()
        elapsed_ms -= f0.elapsed_time(f1)
    # the split kernel's own duration for the roofline: a separate pass with the library's
    # CUDA events around each split launch (kept out of the timed region above), each
    # launch in plain stream order so that its events bracket it alone
    ekv.ekv_set_pdl(ctx.handle, 0)
    ekv.ekv_profile_enable(ctx.handle, True)
    ekv.ekv_profile_read(ctx.handle)
    for _ in range(min(args.steps, 20)):
        step()
    torch.cuda.synchronize()
    split_ms, split_n = ekv.ekv_profile_read(ctx.handle)
    ekv.ekv_profile_enable(ctx.handle, False)
    # the same launches back to back in plain stream order with no events between them:
    # no programmatic overlap, and no event pair inside each launch's time
    plain_ms = None
    if flush is None:
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        plain_steps = min(args.steps, 20)
        p0.record(stream)
        for _ in range(plain_steps):
            step()
        p1.record(stream)
        torch.cuda.synchronize()
        plain_ms = p0.elapsed_time(p1) / (plain_steps * layers)
    ekv.ekv_set_pdl(ctx.handle, int(pdl))
    # what the same events cost around an empty launch of the split kernel's shape
    floor_ms = ekv.ekv_profile_launch_floor(ctx.handle, 64, stream)
    err = ctx.error()
    if world > 1:
        t = torch.tensor([elapsed_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())

    # end to end through the C ABI: per-step inputs from pinned host memory, outputs back.
    # The layers go in chunks (a first chunk of one layer, then up to seven): each chunk's
    # inputs (q, block tables, seq_lens of its layers) are one contiguous pinned buffer and
    # one H2D copy on a copy stream, and each chunk's outputs go back in one copy on that
    # stream while the next chunk decodes. Events order every copy against the kernels that
    # use it; inside a chunk the layer calls follow each other directly in the stream.
    bounds = [0, 1] + list(range(8, layers, 7)) + [layers] if layers > 1 else [0, 1]
    chunks = [list(range(a, b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]

    def packed(ls):
        parts = []
        for l in ls:
            c = cases[l]
            parts += [c.q.contiguous().view(torch.uint8).reshape(-1),
                      c.block_table.contiguous().view(torch.uint8).reshape(-1),
                      c.seq_lens.contiguous().view(torch.uint8).reshape(-1)]
        return torch.cat(parts).cpu().pin_memory(), [p.numel() for p in parts]
    in_h, sizes = zip(*[packed(ls) for ls in chunks])
    in_d = [torch.empty_like(h, device="cuda") for h in in_h]
    views = {}
    for ci, ls in enumerate(chunks):
        off = 0
        for i, l in enumerate(ls):
            nq, nbt, nsl = sizes[ci][3 * i:3 * i + 3]
            c = cases[l]
            views[l] = (in_d[ci][off:off + nq].view(torch.float16).view(c.q.shape),
                        in_d[ci][off + nq:off + nq + nbt].view(torch.int32).view(c.block_table.shape),
                        in_d[ci][off + nq + nbt:off + nq + nbt + nsl].view(torch.int32))
            off += nq + nbt + nsl
    out_d = [torch.empty((len(ls), B, Hq, D), dtype=torch.float16, device="cuda") for ls in chunks]
    out_h = [torch.empty((len(ls), B, Hq, D), dtype=torch.float16).pin_memory() for ls in chunks]
    h2d = sum(h.numel() for h in in_h)
    d2h = sum(o.numel() * 2 for o in out_h)
    copy = torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in chunks]
    ev_out = [torch.cuda.Event() for _ in chunks]
    ev_done = torch.cuda.Event()

    def e2e_step():
        copy.wait_stream(stream)                     # the previous step's kernels have used the buffers
        for ci in range(len(chunks)):
            with torch.cuda.stream(copy):
                in_d[ci].copy_(in_h[ci], non_blocking=True)
                ev_in[ci].record(copy)
        for ci, ls in enumerate(chunks):
            stream.wait_event(ev_in[ci])
            for i, l in enumerate(ls):
                c = cases[l]
                q_l, bt_l, sl_l = views[l]
                ekv.ekv_paged_decode(ctx.handle, q_l, c.k_pages, c.v_pages, c.v_page_stride, c.num_pages,
                                     c.v_scales, c.scale_mode, c.page_mode, c.uniform_mode, bt_l,
                                     int(c.block_table.shape[1]), sl_l, B, 0.0, out_d[ci][i], None, stream)
            ev_out[ci].record(stream)
            copy.wait_event(ev_out[ci])
            with torch.cuda.stream(copy):
                out_h[ci].copy_(out_d[ci], non_blocking=True)
        ev_done.record(copy)
        stream.wait_event(ev_done)                   # the step ends when its last output is home

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    # the outputs that came home equal the device-timed calls' outputs bit for bit
    e2e_same = all(torch.equal(out_h[ci][i], outs[l].cpu()) for ci, ls in enumerate(chunks)
                   for i, l in enumerate(ls))
    if world > 1:
        t = torch.tensor([e2e_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())

    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    value = step_bytes * args.steps * world / (elapsed_ms / 1e3) / 1e9
    e2e_value = step_bytes * args.e2e_steps * world / (e2e_ms / 1e3) / 1e9
    ms_step = elapsed_ms / args.steps
    achieved = split_bytes / (split_ms / split_n / 1e3) / 1e9 if split_n else None
    # the same kernel inside the timed stream: each step is its layer calls alone, so the
    # timed region divided by its launches is the kernel's time per launch in the stream
    stream_ms = elapsed_ms / (args.steps * layers) if flush is None else None
    stream_achieved = split_bytes / (stream_ms / 1e3) / 1e9 if stream_ms else None
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": config_of(args, wk),
        "tokens_per_s": B * world / (ms_step / 1e3),
        "hbm_frac_of_measured": value / world / hbm, "hbm_frac_of_8tbs_spec": value / world / 8000.0,
        "roofline": {"bound": "hbm", "achieved": stream_achieved if stream_achieved else achieved, "peak": hbm,
                     "unit": "GB/s",
                     "frac": (stream_achieved if stream_achieved else achieved) / hbm if (stream_achieved or achieved)
                     else None,
                     "traffic": profiled_traffic(args.workload),
                     "kernel": "decode_split_mma" if args.variant == 0 else "decode_split_simt",
                     "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": split_bytes,
                     "avg_launch_ms": stream_ms if stream_ms else (split_ms / split_n if split_n else None),
                     "launch_mode": ("the timed region's launches, layer calls back to back"
                                     + (" under programmatic dependent launch" if pdl else " in plain stream order")
                                     + ": CUDA events around the timed region / launches (the region holds "
                                       "these launches only)") if stream_ms else
                                    "each launch alone between the library's CUDA events",
                     "isolated_launch": {"avg_launch_ms": split_ms / split_n if split_n else None,
                                         "achieved": achieved, "frac": achieved / hbm if achieved else None,
                                         "launch_mode": "each launch alone in plain stream order, between the "
                                                        "library's CUDA events on the launching stream (a "
                                                        "separate pass after the timed region)",
                                         "plain_order_stream": (
                                             {"avg_launch_ms": plain_ms,
                                              "achieved": split_bytes / (plain_ms / 1e3) / 1e9,
                                              "frac": split_bytes / (plain_ms / 1e3) / 1e9 / hbm,
                                              "launch_mode": "the layer calls back to back in plain stream "
                                                             "order (no programmatic launch), CUDA events "
                                                             "around the pass only"}
                                             if plain_ms else None),
                                         "launch_floor_ms": floor_ms,
                                         "launch_floor": "an empty kernel with the split kernel's grid, block, "
                                                         "shared memory and parameters, between the same "
                                                         "events, the stream kept busy so that the launches "
                                                         "queue (ekv_profile_launch_floor)"}},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": args.e2e_steps, "ms_per_step": e2e_ms / args.e2e_steps,
                "layer_chunks": [len(ls) for ls in chunks], "outputs_equal_device_run": e2e_same},
        "gpu_launches": layers * args.steps,
        "clocks": clock_rec,
        "kv_dtype": "K f16, V e4m3 (compact) / f16 (TARGET); f32 accumulation",
        "device_error": list(err),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cases, wk)
    del cases
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_companions and args.workload == "pages_shape":
        line["decode_workloads"] = decode_workloads(ekv, torch, peaks, min(args.steps, 20), args.warmup,
                                                    args.seed)
        line["companions"] = companions(ekv, torch, peaks)
    if rank == 0:
        print(json.dumps(line))
    ctx.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
