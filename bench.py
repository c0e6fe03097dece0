#!/usr/bin/env python
"""Benchmark of indexer-selected sparse attention decode on GB300.

Workload: steady-state decode, batch 32, each sequence with a 32768-token
prefix, ratio 4, budget 2048 (K = 512 blocks, inert bound 2051), indexer
64 heads x 128, main attention 32 q / 4 kv heads x 128, bf16 paged KV (64-token
pages, randomly permuted page table). One step = one fused qsa_decode call
(append, index score, top-K select, gather attention, split merge, counter
commit) for the 32 rows, replayed as a CUDA graph.

L2: six independent batches of 32 sequences rotate step by step, so the
202 MB a step reads come from HBM (1.2 GB between two uses of a batch, L2 is
129 MB). Positions advance on the device each step; prefixes start below
32768 so that the mean prefix over the run is 32768.

One JSON line (rank 0): value = query rows/s over all ranks; roofline of the
dominant kernel (per-stage CUDA-event timing); e2e through host buffers;
cpu_baseline = the CPU oracle on a bounded sample; nvidia-smi clocks sampled
during the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode query-rows/sec and achieved HBM GB/s (% of roofline) at batch×prefix"
WORKLOAD_ID = 2            # steady-state decode, batch 32 x 32k prefix
N_BATCHES = 6              # default rotating independent batches (L2 defeat)
KERNELS_PER_STEP = 5       # append, score, select, attention, merge (+ commit)
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=30)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--breakdown-steps", type=int, default=600)
    ap.add_argument("--e2e-steps", type=int, default=600)
    ap.add_argument("--oracle-rows", type=int, default=64, help="rows per CPU worker in the cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--n-batches", type=int, default=N_BATCHES,
                    help="rotating batches of 32 sequences (fewer: smaller device footprint, for profiling)")
    ap.add_argument("--legs", default="decode,prefill,ragged,verify",
                    help="comma list of legs to run: decode (the headline), prefill (chunked-prefill "
                         "index scoring against the bf16 tensor peak, and the fused prefill step), ragged "
                         "(batch 64, log-uniform prefixes), verify (R = 3 verify, rewind, 4 decode steps)")
    ap.add_argument("--prefill-steps", type=int, default=10)
    ap.add_argument("--reuse-steps", type=int, default=300,
                    help="decode steps with a reused selection (MTP draft steps); 0 skips the leg")
    ap.add_argument("--pre-steps", type=int, default=300,
                    help="decode steps through the pre-indexer (norm + RoPE of queries and keys); 0 skips")
    ap.add_argument("--mxfp8-steps", type=int, default=600,
                    help="decode steps with the MXFP8 index plane (own cache); 0 skips")
    ap.add_argument("--mxfp4-steps", type=int, default=600,
                    help="decode steps with the MXFP4 index plane (own cache); 0 skips")
    ap.add_argument("--attn-steps", type=int, default=300,
                    help="decode steps with the main-attention options (q/k norm + RoPE, output gate; own "
                         "cache); 0 skips")
    ap.add_argument("--window-steps", type=int, default=300,
                    help="decode steps with a 128-token always-kept local window; 0 skips")
    ap.add_argument("--prefill-warmup", type=int, default=3)
    ap.add_argument("--ragged-steps", type=int, default=200, help="timed steps of the ragged-decode leg")
    ap.add_argument("--ragged-warmup", type=int, default=5)
    ap.add_argument("--verify-cycles", type=int, default=50, help="timed cycles of the verify + rewind leg")
    ap.add_argument("--verify-warmup", type=int, default=3)
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------
# algorithmic bytes / flops (per row), from the method's definition
# ---------------------------------------------------------------------------

def key_bytes(sh, fmt):
    """Bytes of one stored compressed key: bf16, or MX elements + one scale byte per 32."""
    return {"bf16": 2 * sh.idx_dim, "mxfp8": sh.idx_dim + sh.idx_dim // 32,
            "mxfp4": sh.idx_dim // 2 + sh.idx_dim // 32}[fmt]


def row_work(sh, visible, fmt="bf16"):
    n_blk = visible // sh.ratio
    tail = visible - n_blk * sh.ratio
    active = n_blk > sh.topk
    n_tok = min(n_blk, sh.topk) * sh.ratio + tail
    key_b = key_bytes(sh, fmt)
    score_b = (n_blk * key_b + sh.n_idx_heads * sh.idx_dim * 2 + 4 * sh.n_idx_heads) if active else 0
    attn_b = n_tok * sh.n_kv_heads * sh.head_dim * 2 * 2 + 2 * sh.n_q_heads * sh.head_dim * 2
    append_b = (2 * sh.n_kv_heads * sh.head_dim + sh.idx_dim) * 2
    score_f = 2 * sh.n_idx_heads * sh.idx_dim * n_blk if active else 0
    attn_f = 4 * sh.n_q_heads * sh.head_dim * n_tok
    return dict(score_bytes=score_b, attn_bytes=attn_b, append_bytes=append_b,
                score_flops=score_f, attn_flops=attn_f, n_tok=n_tok, n_blk=n_blk)


def sum_work(sh, visibles, fmt="bf16"):
    tot = {}
    for v in visibles:
        for k, x in row_work(sh, v, fmt).items():
            tot[k] = tot.get(k, 0) + x
    return tot


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, t0, t1):
        """Samples whose host timestamp falls in [t0, t1] (wall clock)."""
        import datetime
        sm, mx, reasons, n_all = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 10:
                continue
            n_all += 1
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if not (t0 - 0.05 <= ts <= t1 + 0.05):
                continue
            try:
                sm.append(float(parts[2])); mx.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_total": n_all}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

# ---------------------------------------------------------------------------
# replicas (one process per GPU, no data-path collective): host-side pieces
# ---------------------------------------------------------------------------

def rank_env():
    """(world, rank, local rank) from the launcher's environment (torchrun sets
    all three; a plain run is one rank)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica_seed(seed, rank):
    """Each replica pages its own cache with its own seeded page table."""
    return seed + 1000 * rank


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x, device):
    """The largest x over all ranks (x itself without a process group): the
    slowest replica sets the step time of the whole job."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(rows_per_rank, world, ms):
    """Rows per second of the whole job: every rank's rows over the slowest
    rank's step time (weak scaling: the rows per rank stay fixed as N grows)."""
    return rows_per_rank * world / (ms * 1e-3)


STICKY_CUDA = ("illegal memory access", "illegal instruction", "misaligned address", "unspecified launch failure",
               "hardware stack error", "device-side assert", "launch timed out", "invalid program counter")


def guarded(fn, dist, torch):
    """Run one secondary leg. On a single rank its failure is reported in the
    line (the device-timed headline still prints), with "ok": false; a sticky
    CUDA error (the context is lost) is re-raised, and so is any failure when
    several ranks run, since the other ranks would wait in mismatched
    collectives."""
    try:
        return fn()
    except Exception as e:
        msg = f"{type(e).__name__}: {e}"
        if dist is not None or any(k in msg.lower() for k in STICKY_CUDA):
            raise
        try:
            torch.cuda.synchronize()
        except Exception:
            raise e
        return {"ok": False, "error": msg}


def traffic_for(kernel_key):
    """ncu DRAM bytes per launch for a kernel, if the committed counters were
    taken on the kernel source as it is now."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(kernel_key)
    if not ent:
        return None
    src = os.path.join(ROOT, ent["source"])
    if not os.path.exists(src):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if h != ent.get("sha256"):
        return None
    return ent["bytes_per_launch_full_size"]


def run_gpu(args):
    import torch

    from indexer_selected_sparse_gb300 import qsa as Q
    from indexer_selected_sparse_gb300 import synth as S

    world, rank, local = rank_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    NB = args.n_batches
    wl = S.workload(WORKLOAD_ID)
    sh = wl.shapes
    cfg = Q.Config.of(sh)
    B = wl.n_seq
    K, W = args.steps, args.warmup
    total_steps = W + K + args.breakdown_steps + args.e2e_steps + 4
    adv_per_batch = (math.ceil((W + K + min(K, 600) + args.e2e_steps + NB + 4) / NB) + (62 if args.reuse_steps > 0 else 0)
                     + (math.ceil(args.pre_steps / NB) + 2 if args.pre_steps > 0 else 0)
                     + (math.ceil(args.window_steps / NB) + 2 if args.window_steps > 0 else 0)
                     + max([math.ceil(n / NB) + 2 for n in (args.mxfp8_steps, args.mxfp4_steps, args.attn_steps)
                            if n > 0] or [0]))
    # center the prefixes of the main timed region on 32768
    start = wl.prefixes[0] - W // NB - K // (2 * NB)
    start = max(start, 8)
    n_slots = B * NB
    P = sh.page_size
    max_pages = math.ceil((start + adv_per_batch + 8) / P)
    pt = S.page_table(replica_seed(wl.seed, rank), n_slots, max_pages, contiguous=False)
    cache = Q.PagedCache(cfg, pt, n_slots * max_pages, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    # prefix: every sequence filled through the library's own append
    t_setup = time.time()
    chunk = 8192
    for s in range(n_slots):
        a = 0
        while a < start:
            m = min(chunk, start - a)
            k, v, ix = S.token_rows(sh, wl.seed, s, torch.arange(a, a + m), device=dev)
            rows = Q.Rows(torch.tensor([s], device=dev), torch.tensor([a], device=dev, dtype=torch.int32), m)
            Q.qsa_append(cfg, rows, cache, k, v, ix, status)
            a += m
    torch.cuda.synchronize()
    assert int(status.item()) == 0, Q.qsa_strerror(int(status.item()))
    setup_s = time.time() - t_setup

    # per batch: step inputs (one set per batch, re-appended at advancing positions)
    ws = Q.workspace(cfg, B, cache.max_blocks, device=dev)
    batches = []
    for b in range(NB):
        ids = torch.arange(b * B, (b + 1) * B, dtype=torch.int32, device=dev)
        pos0 = torch.full((B,), start, dtype=torch.int32, device=dev)
        ks, vs, iis, qs, qis, wss = [], [], [], [], [], []
        for s in range(b * B, (b + 1) * B):
            k, v, ix = S.token_rows(sh, wl.seed, s, torch.tensor([start]), device=dev)
            q, qi, w = S.query_rows(sh, wl.seed, s, torch.tensor([start]), device=dev)
            ks.append(k); vs.append(v); iis.append(ix); qs.append(q); qis.append(qi); wss.append(w)
        cat = lambda xs: torch.cat(xs).contiguous()
        batches.append(dict(ids=ids, pos0=pos0, k=cat(ks), v=cat(vs), idx=cat(iis), q=cat(qs),
                            q_idx=cat(qis), w=cat(wss),
                            out=torch.empty(B, sh.n_q_heads, sh.head_dim, dtype=torch.bfloat16, device=dev)))

    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def decode_call(bt, advance=True):
        rows = Q.Rows(bt["ids"], bt["pos0"], 1, advance=advance)
        Q.qsa_decode(cfg, rows, cache, bt["k"], bt["v"], bt["idx"], bt["q_idx"], bt["w"], bt["q"],
                     bt["out"], ws, status)

    # one graph per batch (one step), and one graph holding a whole rotation:
    # the NB batches' steps back to back, as the op runs inside a larger graph
    # (a model step) where its first kernel follows another kernel rather than
    # a graph launch
    graphs = []
    for bt in batches:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            decode_call(bt)
        graphs.append(g)
    rotation = torch.cuda.CUDAGraph()
    with torch.cuda.graph(rotation, stream=stream):
        for bt in batches:
            decode_call(bt)
    torch.cuda.synchronize()

    # host-side mirror of the positions (for the exact algorithmic bytes)
    hpos = [start] * NB

    def replay(b):
        graphs[b].replay()
        hpos[b] += 1

    def replay_rotation():
        rotation.replay()
        for b in range(NB):
            hpos[b] += 1

    with torch.cuda.stream(stream):
        for i in range(W):
            replay(i % NB)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, Q.qsa_strerror(int(status.item()))

    # ---- timed region: K fused steps (K // NB rotations, then K % NB single steps)
    n_rot, n_rest = K // NB, K % NB
    order = [b for _ in range(n_rot) for b in range(NB)] + list(range(n_rest))
    # exact visible counts of every row of every timed step
    sim = list(hpos)
    visibles = []
    for b in order:
        visibles += [sim[b] + 1] * B
        sim[b] += 1
    vis_dev = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    smi_id = vis_dev.split(",")[local].strip() if vis_dev else str(local)
    clk = ClockSampler(smi_id)
    time.sleep(0.5)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(n_rot):
            replay_rotation()
        for b in range(n_rest):
            replay(b)
        ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(dist)
    clk.stop()
    clocks = clk.summary(t0, t1)
    ms = max_over_ranks(dist, ev0.elapsed_time(ev1) / K, dev)
    st = int(status.item())
    assert st == 0, f"device status {st}: {Q.qsa_strerror(st)}"
    # the same steps with one graph launch per step (not the headline: the
    # launch gap between graphs is included)
    KS = min(K, 600)
    es0 = torch.cuda.Event(enable_timing=True)
    es1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        es0.record(stream)
        for i in range(KS):
            replay(i % NB)
        es1.record(stream)
    torch.cuda.synchronize()
    ms_single = es0.elapsed_time(es1) / KS
    assert int(status.item()) == 0, Q.qsa_strerror(int(status.item()))
    rows_per_step = B * world
    value = whole_job_rate(B, world, ms)
    work = sum_work(sh, visibles)
    step_bytes = (work["score_bytes"] + work["attn_bytes"] + work["append_bytes"]) / K
    hbm_gbs, tf_peak, peak_kind = measured_peaks()
    step_gbs = step_bytes / (ms * 1e-3) / 1e9

    # ---- per-stage timing (same workload, stage entry points, events between)
    roofline, stage_ms, stage_bytes, stage_flops = None, {}, {}, {}
    if args.breakdown_steps > 0:
        roofline, stage_ms, stage_bytes, stage_flops = stage_breakdown(
            args, Q, torch, cfg, sh, cache, batches, ws, status, stream, hpos, NB, B, hbm_gbs, peak_kind)

    out_e2e = guarded(lambda: run_e2e(args, Q, torch, cfg, cache, batches, ws, status, stream, NB, B,
                                      rows_per_step, decode_call, dist, dev), dist, torch)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    out = make_line(wl, sh, B, K, W, world, value, ms, visibles, step_bytes, step_gbs, hbm_gbs, NB,
                    roofline, stage_ms, stage_bytes, stage_flops, out_e2e, clocks, setup_s)
    out["ms_per_step_one_graph_per_step"] = round(ms_single, 5)
    if args.reuse_steps > 0:
        out["reuse"] = run_reuse(args, Q, torch, cfg, sh, cache, batches, ws, status, stream, NB, B, hbm_gbs)
    if args.pre_steps > 0:
        out["pre_indexer"] = run_pre(args, Q, S, torch, cfg, sh, cache, batches, status, stream, NB, B, hbm_gbs,
                                     ms)
    if args.window_steps > 0:
        out["local_window"] = run_window(args, Q, torch, sh, cache, batches, status, stream, NB, B, ms)
    for fmt, steps in (("mxfp8", args.mxfp8_steps), ("mxfp4", args.mxfp4_steps)):
        if steps > 0:
            out[fmt] = run_mx(args, Q, S, torch, wl, sh, pt, max_pages, start, batches, stream, NB, B, hbm_gbs,
                              ms, fmt, steps)
    late = None
    if args.attn_steps > 0:
        # run last of all GPU work (after the prefill leg), so that nothing else depends on it
        def late():
            return run_attn_options(args, Q, S, torch, wl, sh, pt, max_pages, start, batches, stream, NB, B, ms)
    return out, rank, world, late


def run_attn_options(args, Q, S, torch, wl, sh, pt, max_pages, start, batches, stream, NB, B, ms_plain):
    """The decode workload with the main-attention options on (qsa_attn_options):
    q and k heads GemmaRMSNormed (gain 1 + gamma) and NeoX-roped over 64 dims
    (keys as they are appended, the step's queries inside the step) and a
    sigmoid output gate, one bf16 gate value per output element. Its own cache,
    filled through qsa_append_ex with the same prefixes; the decode leg's step
    inputs plus a gate per batch; one rotation graph of the NB batches."""
    dev = batches[0]["k"].device
    cfg = Q.Config.of(sh)
    n_slots = B * NB
    cache_a = Q.PagedCache(cfg, pt, n_slots * max_pages, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    gen = torch.Generator().manual_seed(wl.seed + 77)
    gq = (0.2 * torch.randn(sh.head_dim, generator=gen)).to(dev)
    gk = (0.2 * torch.randn(sh.head_dim, generator=gen)).to(dev)
    fill = Q.AttnOptions(None, gk, 1e-6, 1e4, 64)
    chunk = 8192
    for s_ in range(n_slots):
        a = 0
        while a < start:
            m = min(chunk, start - a)
            k, v, ix = S.token_rows(sh, wl.seed, s_, torch.arange(a, a + m), device=dev)
            Q.qsa_append_ex(cfg, None, fill, Q.Rows(torch.tensor([s_], device=dev),
                                                   torch.tensor([a], device=dev, dtype=torch.int32), m),
                            cache_a, k, v, ix, status)
            a += m
    gates = [(2 * torch.randn(B, sh.n_q_heads, sh.head_dim, generator=gen)).to(torch.bfloat16).to(dev)
             for _ in range(NB)]
    opts = [Q.AttnOptions(gq, gk, 1e-6, 1e4, 64, gate=gates[b]) for b in range(NB)]
    ws_a = Q.workspace_ex(cfg, B, cache_a.max_blocks, device=dev)
    pos_a = [torch.full((B,), start, dtype=torch.int32, device=dev) for _ in range(NB)]
    rot = torch.cuda.CUDAGraph()
    with torch.cuda.graph(rot, stream=stream):
        for b, bt in enumerate(batches):
            Q.qsa_decode_ex(cfg, None, opts[b], Q.Rows(bt["ids"], pos_a[b], 1, advance=True), cache_a, bt["k"],
                            bt["v"], bt["idx"], bt["q_idx"], bt["w"], bt["q"], bt["out"], ws_a, status,
                            stream=stream)
    torch.cuda.synchronize()
    n_rot = max(1, math.ceil(args.attn_steps / NB))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        rot.replay()  # warm-up rotation
        e0.record(stream)
        for _ in range(n_rot):
            rot.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st == 0, f"device status {st}: {Q.qsa_strerror(st)}"
    steps = n_rot * NB
    ms = e0.elapsed_time(e1) / steps
    del rot, cache_a
    return {"what": "decode step with the main-attention options: q/k GemmaRMSNorm + NeoX RoPE (64 dims) and a "
                    "sigmoid output gate, batch 32 x 32k",
            "steps": steps, "ms_per_step": round(ms, 5), "rows_per_s": round(B / (ms * 1e-3), 1),
            "overhead_vs_plain_ms": round(ms - ms_plain, 5),
            "extra_bytes_per_row": sh.n_q_heads * sh.head_dim * 2}


def run_window(args, Q, torch, sh, cache, batches, status, stream, NB, B, ms_plain, window=128):
    """The decode step with an always-kept local window (local_window = 128: every
    row also attends to its last 128 tokens, a union with the top-k set), on the
    decode leg's cache and inputs: one rotation graph of the NB batches."""
    dev = cache.k_pool.device
    cfg_w = Q.Config.of(sh, Q.QSA_INDEX_BF16, window)
    ws = Q.workspace(cfg_w, B, cache.max_blocks, device=dev)
    rot = torch.cuda.CUDAGraph()
    with torch.cuda.graph(rot, stream=stream):
        for bt in batches:
            Q.qsa_decode(cfg_w, Q.Rows(bt["ids"], bt["pos0"], 1, advance=True), cache, bt["k"], bt["v"], bt["idx"],
                         bt["q_idx"], bt["w"], bt["q"], bt["out"], ws, status, stream=stream)
    torch.cuda.synchronize()
    n_rot = max(1, math.ceil(args.window_steps / NB))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        rot.replay()  # warm-up rotation
        e0.record(stream)
        for _ in range(n_rot):
            rot.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st == 0, f"device status {st}: {Q.qsa_strerror(st)}"
    steps = n_rot * NB
    ms = e0.elapsed_time(e1) / steps
    return {"what": f"decode step with a {window}-token always-kept local window (union with the top-k set), "
                    "batch 32 x 32k", "window": window,
            "steps": steps, "ms_per_step": round(ms, 5), "rows_per_s": round(B / (ms * 1e-3), 1),
            "overhead_vs_plain_ms": round(ms - ms_plain, 5),
            "tokens_per_row": "selected tokens before the run + the last 128 (at most budget + 128 + ratio - 1)"}


MX_LEGS = {
    "mxfp8": ("QSA_INDEX_MXFP8", "E4M3"),
    "mxfp4": ("QSA_INDEX_MXFP4", "E2M1"),
}


def run_mx(args, Q, S, torch, wl, sh, pt, max_pages, start, batches, stream, NB, B, hbm_gbs, ms_plain, fmt,
           n_steps):
    """The same decode workload with an MX index plane (index_format
    QSA_INDEX_MXFP8 or QSA_INDEX_MXFP4): compressed keys stored as E4M3 or E2M1
    elements + one E8M0 scale per 32 values (132 or 68 bytes per key instead of
    256), index queries MX-rounded inside the step. Its own cache, filled through
    qsa_append with the same prefixes (the positions the decode leg started
    from); the same step inputs; one rotation graph of the NB batches, timed
    with CUDA events."""
    dev = batches[0]["k"].device
    const, elem = MX_LEGS[fmt]
    cfg8 = Q.Config.of(sh, getattr(Q, const))
    n_slots = B * NB
    cache8 = Q.PagedCache(cfg8, pt, n_slots * max_pages, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    chunk = 8192
    for s_ in range(n_slots):
        a = 0
        while a < start:
            m = min(chunk, start - a)
            k, v, ix = S.token_rows(sh, wl.seed, s_, torch.arange(a, a + m), device=dev)
            Q.qsa_append(cfg8, Q.Rows(torch.tensor([s_], device=dev), torch.tensor([a], device=dev,
                                                                                 dtype=torch.int32), m),
                         cache8, k, v, ix, status)
            a += m
    ws8 = Q.workspace(cfg8, B, cache8.max_blocks, device=dev)
    pos8 = [torch.full((B,), start, dtype=torch.int32, device=dev) for _ in range(NB)]
    rot = torch.cuda.CUDAGraph()
    with torch.cuda.graph(rot, stream=stream):
        for b, bt in enumerate(batches):
            Q.qsa_decode(cfg8, Q.Rows(bt["ids"], pos8[b], 1, advance=True), cache8, bt["k"], bt["v"], bt["idx"],
                         bt["q_idx"], bt["w"], bt["q"], bt["out"], ws8, status, stream=stream)
    torch.cuda.synchronize()
    n_rot = max(1, math.ceil(n_steps / NB))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        rot.replay()  # warm-up rotation
        e0.record(stream)
        for _ in range(n_rot):
            rot.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st == 0, f"device status {st}: {Q.qsa_strerror(st)}"
    steps = n_rot * NB
    ms = e0.elapsed_time(e1) / steps
    # timed rows: every batch at positions start + 1 .. start + n_rot (one warm-up step each before)
    visibles = [start + 1 + r + 1 for r in range(1, n_rot + 1) for _ in range(NB) for _ in range(B)]
    work = sum_work(sh, visibles, fmt)
    step_bytes = (work["score_bytes"] + work["attn_bytes"] + work["append_bytes"]) / steps
    gbs = step_bytes / (ms * 1e-3) / 1e9
    stages = None
    if args.breakdown_steps > 0:
        # per-stage graphs on this cache, at the positions the timed rotations reached
        bts = [dict(bt, pos0=pos8[b]) for b, bt in enumerate(batches)]
        _, stage_ms, _, _ = stage_breakdown(args, Q, torch, cfg8, sh, cache8, bts, ws8, status, stream,
                                            [start + n_rot + 1] * NB, NB, B, hbm_gbs, "")
        stages = {k_: round(v_, 5) for k_, v_ in stage_ms.items()}
    del cache8
    return {"what": f"the decode workload (batch 32 x 32k) with the {fmt.upper()} index plane: compressed keys "
                    f"as {elem} + one E8M0 scale per 32 values, index queries {fmt.upper()}-rounded in the step",
            "steps": steps, "ms_per_step": round(ms, 5), "rows_per_s": round(B / (ms * 1e-3), 1),
            "speedup_vs_bf16_plane": round(ms_plain / ms, 3), "bytes_per_step": int(step_bytes),
            "stages_ms": stages,
            "achieved_gbs": round(gbs, 1), "hbm_roofline_frac": round(gbs / hbm_gbs, 4),
            "bytes": f"{fmt.upper()} keys ({key_bytes(sh, fmt)} B per block), bf16 q_idx, w, K+V of the selected "
                     "tokens, q, o, appends"}


def run_pre(args, Q, S, torch, cfg, sh, cache, batches, status, stream, NB, B, hbm_gbs, ms_plain):
    """The fused decode step through the pre-indexer (qsa_decode_pre): the step's
    index queries get Gemma RMSNorm + NeoX RoPE, a block completed by the step
    is pooled, normed and roped, then score, select, attend as in the plain step.
    Timed on the decode leg's cache (its older blocks were pooled without the
    pre-indexer, which changes the values scored, not the work done)."""
    dev = cache.k_pool.device
    d = sh.idx_dim
    u = S.uniform01(7, 101, torch.arange(2 * d, dtype=torch.int64)).to(torch.float32)
    pre = Q.PreIndexer((0.4 * (u[:d] - 0.5)).to(dev), (0.4 * (u[d:] - 0.5)).to(dev), 1e-6, 1e4, 64)
    ws = Q.workspace_pre(cfg, B, cache.max_blocks, device=dev)
    rot = torch.cuda.CUDAGraph()
    with torch.cuda.graph(rot, stream=stream):
        for bt in batches:
            Q.qsa_decode_pre(cfg, pre, Q.Rows(bt["ids"], bt["pos0"], 1, advance=True), cache, bt["k"], bt["v"],
                             bt["idx"], bt["q_idx"], bt["w"], bt["q"], bt["out"], ws, status, stream=stream)
    torch.cuda.synchronize()
    n_rot = max(1, math.ceil(args.pre_steps / NB))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        rot.replay()  # warm-up rotation
        e0.record(stream)
        for _ in range(n_rot):
            rot.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st == 0, f"device status {st}: {Q.qsa_strerror(st)}"
    steps = n_rot * NB
    ms = e0.elapsed_time(e1) / steps
    return {"what": "fused decode step through the pre-indexer (qsa_decode_pre: query norm + RoPE, "
                    "completed-block norm + RoPE, score, select, attend), batch 32 x 32k",
            "steps": steps, "ms_per_step": round(ms, 5), "rows_per_s": round(B / (ms * 1e-3), 1),
            "overhead_vs_plain_ms": round(ms - ms_plain, 5)}


def run_reuse(args, Q, torch, cfg, sh, cache, batches, ws, status, stream, NB, B, hbm_gbs):
    """Decode steps that reuse the step-0 selection (MTP draft steps): append,
    then attention over the reused blocks plus the tail since; no scoring or
    selection. Each batch selects once (untimed), then takes up to 60 reuse
    steps: the token set grows by one per step and must stay within the split
    plan (qsa_max_attend_tokens)."""
    dev = cache.k_pool.device
    per_batch = min(60, max(1, args.reuse_steps // NB))
    limit = Q.qsa_max_attend_tokens(cfg) - sh.topk * sh.ratio - sh.ratio
    per_batch = max(1, min(per_batch, limit))
    torch.cuda.synchronize()
    cur = [int(bt["pos0"][0].item()) for bt in batches]  # every sequence of a batch is at one position
    sels, nsels, selpos = [], [], []
    for b, bt in enumerate(batches):
        sel = torch.empty(B, cfg.topk, dtype=torch.int32, device=dev)
        nsel = torch.empty(B, dtype=torch.int32, device=dev)
        selpos.append(torch.full((B,), cur[b], dtype=torch.int32, device=dev))
        rows = Q.Rows(bt["ids"], bt["pos0"], 1, advance=True)
        with torch.cuda.stream(stream):
            Q.qsa_decode(cfg, rows, cache, bt["k"], bt["v"], bt["idx"], bt["q_idx"], bt["w"], bt["q"],
                         bt["out"], ws, status, sel_out=sel, n_sel_out=nsel, stream=stream)
        sels.append(sel); nsels.append(nsel)
    rot = torch.cuda.CUDAGraph()
    with torch.cuda.graph(rot, stream=stream):
        for b, bt in enumerate(batches):
            Q.qsa_decode_reuse(cfg, Q.Rows(bt["ids"], bt["pos0"], 1, advance=True), cache, bt["k"], bt["v"],
                               bt["idx"], bt["q"], sels[b], nsels[b], selpos[b], bt["out"], ws, status,
                               stream=stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        rot.replay()  # warm-up rotation
        e0.record(stream)
        for _ in range(per_batch - 1):
            rot.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st == 0, f"device status {st}: {Q.qsa_strerror(st)}"
    steps = (per_batch - 1) * NB
    ms = e0.elapsed_time(e1) / steps
    # algorithmic bytes: the reused token set (K + V of every KV head), q, o, appends
    # timed rows: batch b at positions cur[b] + 2 .. cur[b] + per_batch
    tot = 0
    for r in range(per_batch - 1):
        for b in range(NB):
            V = cur[b] + 2 + r + 1
            tail = V - ((cur[b] + 1) // sh.ratio) * sh.ratio
            n_tok = sh.topk * sh.ratio + tail
            tot += B * (n_tok * sh.n_kv_heads * sh.head_dim * 4 + 2 * sh.n_q_heads * sh.head_dim * 2
                        + (2 * sh.n_kv_heads * sh.head_dim + sh.idx_dim) * 2)
    gbs = tot / steps / (ms * 1e-3) / 1e9
    return {"what": "decode steps reusing the step-0 selection (MTP draft steps): append + attention "
                    "over the reused blocks and the tail since, no scoring or selection",
            "steps": steps, "ms_per_step": round(ms, 5), "rows_per_s": round(B / (ms * 1e-3), 1),
            "achieved_gbs": round(gbs, 1), "hbm_roofline_frac": round(gbs / hbm_gbs, 4),
            "bytes": "reused token set K+V, q, o, appended rows"}


def stage_breakdown(args, Q, torch, cfg, sh, cache, batches, ws, status, stream, hpos, NB, B, hbm_gbs,
                    peak_kind):
    """Per-stage device time of the decode step: each stage is one CUDA graph
    holding that stage's calls for all NB rotating batches back to back (so a
    graph launch is spread over NB launches and the batches' data, NB x the
    step's bytes, does not fit in L2), timed with CUDA events around each replay
    and divided by NB. Stages run in step order (every batch's append, then every
    batch's scoring, ...); each batch has its own score rows and selection."""
    dev = cache.k_pool.device
    ld = (cache.max_blocks + 3) // 4 * 4
    scores = [torch.empty(B, ld, dtype=torch.float32, device=dev) for _ in batches]
    sel = [torch.empty(B, cfg.topk, dtype=torch.int32, device=dev) for _ in batches]
    nsel = [torch.empty(B, dtype=torch.int32, device=dev) for _ in batches]
    one = torch.ones(B, dtype=torch.int32, device=dev)
    calls = []
    for b, bt in enumerate(batches):
        rows = Q.Rows(bt["ids"], bt["pos0"], 1)
        calls.append((
            lambda bt=bt, rows=rows: Q.qsa_append(cfg, rows, cache, bt["k"], bt["v"], bt["idx"], status),
            lambda bt=bt, rows=rows, b=b: Q.qsa_index_score(cfg, rows, cache, bt["q_idx"], bt["w"], scores[b], ld,
                                                            status),
            lambda rows=rows, b=b: Q.qsa_topk_select(cfg, rows, scores[b], ld, sel[b], nsel[b], status),
            lambda bt=bt, rows=rows, b=b: Q.qsa_gather_attn(cfg, rows, cache, bt["q"], sel[b], nsel[b], bt["out"],
                                                            ws, status),
            lambda bt=bt: Q.qsa_rewind(cfg, bt["ids"], one, cache.ingested, status)))
    stage_graphs = []
    for j in range(5):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for c in calls:
                c[j]()
        stage_graphs.append(g)
    torch.cuda.synchronize()
    KB = max(1, math.ceil(args.breakdown_steps / NB))  # rotations
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(KB)]
    with torch.cuda.stream(stream):
        for i in range(KB):
            e = evs[i]
            for j in range(4):
                e[j].record(stream)
                stage_graphs[j].replay()
            e[4].record(stream)
            stage_graphs[4].replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, Q.qsa_strerror(int(status.item()))
    names = ["append", "index_score", "topk_select", "gather_attn"]
    stage_ms = {n: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(KB)) / (KB * NB)
                for j, n in enumerate(names)}
    bvis = []
    for b in range(NB):
        bvis += [hpos[b] + 1] * B
    bw = sum_work(sh, bvis)
    stage_bytes = {"append": bw["append_bytes"] / NB, "index_score": bw["score_bytes"] / NB,
                   "gather_attn": bw["attn_bytes"] / NB, "topk_select": 0}
    stage_flops = {"index_score": bw["score_flops"] / NB, "gather_attn": bw["attn_flops"] / NB}
    dominant = max(stage_ms, key=lambda n: stage_ms[n])
    if dominant == "topk_select":
        dominant = "gather_attn" if stage_ms["gather_attn"] >= stage_ms["index_score"] else "index_score"
    ach = stage_bytes[dominant] / (stage_ms[dominant] * 1e-3) / 1e9
    roofline = {"kernel": {"gather_attn": "attn_kernel<4> + merge_kernel", "index_score": "score_tc_kernel<128>",
                           "append": "append_kernel"}[dominant],
                "bound": "hbm", "achieved": round(ach, 1), "peak": hbm_gbs, "unit": "GB/s",
                "frac": round(ach / hbm_gbs, 4), "peak_kind": peak_kind + " (hbm_gbs, copy)",
                "traffic": traffic_for(dominant),
                "algorithmic_bytes_per_launch": int(stage_bytes[dominant]),
                "launch_ms": round(stage_ms[dominant], 5)}
    return roofline, stage_ms, stage_bytes, stage_flops


STEP_INPUTS = ("k", "v", "idx", "q_idx", "w", "q")


def packed(torch, tensors, device, pin=False):
    """One byte buffer holding the tensors back to back, each at a 256-byte
    boundary (the C ABI wants 16), and a view of each tensor's shape and dtype
    into it: a step's inputs then cross to the device in one copy."""
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(total, dtype=torch.uint8, device=device, pin_memory=pin)
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
    return buf, views


def run_e2e(args, Q, torch, cfg, cache, batches, ws, status, stream, NB, B, rows_per_step, decode_call,
            dist, dev):
    # ---- end to end: host buffers, H2D inputs + fused step + D2H output per step.
    # A step's six inputs sit packed in one pinned host buffer and cross in one
    # copy to one device buffer, whose views the step reads. One CUDA graph holds a
    # rotation of the NB independent batches: each step's H2D copy runs on a copy
    # stream ahead of its step, and each output's D2H copy on a second copy stream
    # after it, so copies overlap the neighbouring steps; every step still moves
    # its own inputs and output inside the timed region.
    e2e = None
    KE = args.e2e_steps
    if KE > 0:
        keep = []
        h2d = d2h = h2d_copied = 0
        for bt in batches:
            ins = [bt[k] for k in STEP_INPUTS]
            dbuf, dviews = packed(torch, ins, dev)
            hbuf, hviews = packed(torch, ins, "cpu", pin=True)
            for hv, t in zip(hviews, ins):
                hv.copy_(t.cpu())
            hout = torch.empty_like(bt["out"], device="cpu").pin_memory()
            ebt = dict(bt)
            ebt.update(zip(STEP_INPUTS, dviews))
            keep.append((dbuf, hbuf, hout, ebt))
            h2d = sum(t.numel() * t.element_size() for t in ins)   # the inputs' own bytes
            h2d_copied = hbuf.numel()                               # with the 256-byte alignment gaps
            d2h = hout.numel() * hout.element_size()
        d2h_stream = torch.cuda.Stream(device=dev)
        ev_fork = torch.cuda.Event()
        ev_step = [torch.cuda.Event() for _ in range(NB)]
        ev_join = torch.cuda.Event()
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            ev_fork.record(stream)
            d2h_stream.wait_event(ev_fork)
            for b, (dbuf, hbuf, hout, ebt) in enumerate(keep):
                # the inputs cross by qsa_stage_in, a copy kernel in the step's own
                # programmatic chain (a copy-engine node would break the chain)
                Q.qsa_stage_in(dbuf, hbuf, stream=stream)
                decode_call(ebt)
                ev_step[b].record(stream)
                with torch.cuda.stream(d2h_stream):
                    d2h_stream.wait_event(ev_step[b])
                    hout.copy_(batches[b]["out"], non_blocking=True)
            ev_join.record(d2h_stream)
            stream.wait_event(ev_join)
        torch.cuda.synchronize()
        n_rot = max(1, math.ceil(KE / NB))
        with torch.cuda.stream(stream):
            g.replay()  # warm-up rotation
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
        barrier(dist)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n_rot):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        steps = n_rot * NB
        ems = max_over_ranks(dist, e0.elapsed_time(e1) / steps, dev)
        assert int(status.item()) == 0, Q.qsa_strerror(int(status.item()))
        e2e = {"value": round(rows_per_step / (ems * 1e-3), 1), "unit": "rows/s",  # rows of all ranks
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "h2d_bytes_copied_per_step": h2d_copied,
               "ms_per_step": round(ems, 5), "steps": steps,
               "path": "per step: pinned host inputs (one packed buffer) -> qsa_stage_in (a copy kernel in the "
                       "step's programmatic launch chain, overlapping the previous step's last kernel) -> "
                       f"qsa_decode -> D2H of the output; one CUDA graph per rotation of the {NB} independent "
                       "batches, the D2H copies on a copy stream after their steps"}
    return e2e


def make_line(wl, sh, B, K, W, world, value, ms, visibles, step_bytes, step_gbs, hbm_gbs, NB,
              roofline, stage_ms, stage_bytes, stage_flops, e2e, clocks, setup_s):
    vmin, vmax = min(visibles), max(visibles)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "batch": B, "prefix": wl.prefixes[0],
                   "prefix_range_timed": [vmin - 1, vmax - 1],
                   "mean_prefix_timed": round(sum(visibles) / len(visibles) - 1, 1),
                   "ratio": sh.ratio, "budget": sh.budget, "topk": sh.topk, "idx_heads": sh.n_idx_heads,
                   "idx_dim": sh.idx_dim, "q_heads": sh.n_q_heads, "kv_heads": sh.n_kv_heads,
                   "head_dim": sh.head_dim, "page_size": sh.page_size,
                   "l2": f"inputs larger than L2: {NB} rotating batches of {B} sequences, "
                         f"{step_bytes / 1e6:.1f} MB per step, {NB * step_bytes / 1e9:.2f} GB per rotation",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "graph": f"one CUDA graph per rotation of the {NB} batches ({NB} steps back to back), "
                            "positions advanced on the device"},
        "achieved_gbs": round(step_gbs, 1),
        "hbm_roofline_frac": round(step_gbs / hbm_gbs, 4),
        "roofline": roofline,
        "stages_ms": {k: round(v, 5) for k, v in stage_ms.items()},
        "stages_gbs": {k: round(stage_bytes[k] / (stage_ms[k] * 1e-3) / 1e9, 1) for k in stage_ms if stage_bytes.get(k)},
        "stages_tflops": {k: round(stage_flops[k] / (stage_ms[k] * 1e-3) / 1e12, 1) for k in stage_flops},
        "e2e": e2e,
        "gpu_launches": KERNELS_PER_STEP * K,
        "clocks": clocks,
        "setup_s": round(setup_s, 1),
    }
    return out


# ---------------------------------------------------------------------------
# chunked-prefill leg: index scoring on the tensor cores, and the fused step
# ---------------------------------------------------------------------------

PREFILL_WORKLOAD_ID = 5    # one sequence, 8193-token chunk appended to a 24576-token prefix


def run_prefill(args, dev):
    """Chunked prefill: one sequence, an 8193-row chunk on a 24576-token prefix
    (ratio 4, budget 2048, indexer 64 x 128). Every chunk row scores all blocks
    visible to it (6144..8192), which is a causal 8192-block x (8193 x 64) x 128
    bf16 contraction plus the ReLU * w epilogue. The compressed keys of the
    sequence (2 MB) are L2-resident by the nature of the workload (every row
    reads them); the score rows written (269 MB) exceed L2.

    Times qsa_index_score alone (the tensor-core kernel, against the bf16
    peak), the other stage entry points, and the whole fused step
    (qsa_decode of the 8193 rows, the chunk rewound between steps)."""
    import torch

    from indexer_selected_sparse_gb300 import qsa as Q
    from indexer_selected_sparse_gb300 import synth as S

    wl = S.workload(PREFILL_WORKLOAD_ID)
    sh = wl.shapes
    cfg = Q.Config.of(sh)
    p, C = wl.prefixes[0], wl.rows_per_seq
    max_pages = math.ceil((p + C + 8) / sh.page_size)
    cache = Q.PagedCache(cfg, S.page_table(wl.seed, 1, max_pages, contiguous=False), max_pages, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    seq = torch.zeros(1, dtype=torch.int32, device=dev)
    a = 0
    while a < p:
        m = min(8192, p - a)
        k, v, ix = S.token_rows(sh, wl.seed, 0, torch.arange(a, a + m), device=dev)
        Q.qsa_append(cfg, Q.Rows(seq, torch.tensor([a], dtype=torch.int32, device=dev), m), cache, k, v, ix, status)
        a += m
    pos = torch.arange(p, p + C)
    k, v, ix = S.token_rows(sh, wl.seed, 0, pos, device=dev)
    q, qi, w = S.query_rows(sh, wl.seed, 0, pos, device=dev)
    rows = Q.Rows(seq, torch.tensor([p], dtype=torch.int32, device=dev), C)
    ws = Q.workspace(cfg, C, cache.max_blocks, device=dev)
    out = torch.empty(C, sh.n_q_heads, sh.head_dim, dtype=torch.bfloat16, device=dev)
    drop = torch.tensor([C], dtype=torch.int32, device=dev)
    ld = (cache.max_blocks + 3) // 4 * 4
    scores = torch.empty(C, ld, dtype=torch.float32, device=dev)
    sel = torch.empty(C, cfg.topk, dtype=torch.int32, device=dev)
    nsel = torch.empty(C, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def fused():
        Q.qsa_decode(cfg, rows, cache, k, v, ix, qi, w, q, out, ws, status, stream=stream)

    def rewind():
        Q.qsa_rewind(cfg, seq, drop, cache.ingested, status, stream=stream)

    def timed(fn, n, after=None):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                e0.record(stream)
                fn()
                e1.record(stream)
                if after is not None:
                    after()
        torch.cuda.synchronize()
        return sum(e0.elapsed_time(e1) for e0, e1 in evs) / n

    W, K = max(args.prefill_warmup, 1), max(args.prefill_steps, 1)
    with torch.cuda.stream(stream):
        for _ in range(W):
            fused()
            rewind()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, Q.qsa_strerror(int(status.item()))
    step_ms = timed(fused, K, after=rewind)
    with torch.cuda.stream(stream):
        fused()  # leave the chunk appended for the stage entry points
    torch.cuda.synchronize()
    score_fn = lambda: Q.qsa_index_score(cfg, rows, cache, qi, w, scores, ld, status, stream=stream)
    select_fn = lambda: Q.qsa_topk_select(cfg, rows, scores, ld, sel, nsel, status, stream=stream)
    attn_fn = lambda: Q.qsa_gather_attn(cfg, rows, cache, q, sel, nsel, out, ws, status, stream=stream)
    stage_ms = {}
    for name, fn in (("index_score", score_fn), ("topk_select", select_fn), ("gather_attn", attn_fn)):
        with torch.cuda.stream(stream):
            for _ in range(W):
                fn()
        stage_ms[name] = timed(fn, K)
    assert int(status.item()) == 0, Q.qsa_strerror(int(status.item()))

    visibles = [p + j + 1 for j in range(C)]
    work = sum_work(sh, visibles)
    _, tf_burst, peak_kind = measured_peaks()
    score_tflops = work["score_flops"] / (stage_ms["index_score"] * 1e-3) / 1e12
    attn_tflops = work["attn_flops"] / (stage_ms["gather_attn"] * 1e-3) / 1e12
    return {
        "workload": wl.name, "rows": C, "prefix": p,
        "index_score": {"kernel": "score_tc_kernel<128>", "bound": "tensor",
                        "achieved": round(score_tflops, 1), "peak": tf_burst, "unit": "TFLOP/s",
                        "frac": round(score_tflops / tf_burst, 4),
                        "peak_kind": peak_kind + " (bf16_tflops, burst: the kernel is timed alone)",
                        "flops_per_launch": int(work["score_flops"]),
                        "launch_ms": round(stage_ms["index_score"], 4)},
        "stages_ms": {k_: round(v_, 4) for k_, v_ in stage_ms.items()},
        "gather_attn_tflops": round(attn_tflops, 1),
        "fused_step_ms": round(step_ms, 4),
        "rows_per_s": round(C / (step_ms * 1e-3), 1),
        "timing": f"{K} launches after {W} warm-up, CUDA events on the launching stream; "
                  "fused step = qsa_decode of the chunk (append, score, select, attend, merge), "
                  "rewound between steps outside the events",
    }


# ---------------------------------------------------------------------------
# ragged decode (batch 64, log-uniform prefixes) and verify + rewind legs
# ---------------------------------------------------------------------------

def fill_prefixes(Q, S, torch, cfg, sh, wl, cache, prefixes, status, dev, seqs=None):
    """Every sequence's prefix through the library's own append (8192 tokens a call)."""
    seqs = list(range(len(prefixes))) if seqs is None else seqs
    for s_, n in zip(seqs, prefixes):
        a = 0
        while a < n:
            m = min(8192, n - a)
            k, v, ix = S.token_rows(sh, wl.seed, s_, torch.arange(a, a + m), device=dev)
            Q.qsa_append(cfg, Q.Rows(torch.tensor([s_], device=dev), torch.tensor([a], device=dev, dtype=torch.int32),
                                     m), cache, k, v, ix, status)
            a += m


def run_ragged(args, dev):
    """Ragged decode (batch 64, prefixes log-uniform in [512, 131072] with the
    inert-bound boundary 2050 / 2051 / 2052 and dense prefixes forced in): one
    fused qsa_decode of the 64 rows per step, a CUDA graph replayed with the
    positions advancing on the device. A step reads about 0.34 GB (more than L2),
    so the data comes from HBM. Bytes per row from the method's definition
    (keys only for rows past the inert bound)."""
    import torch

    from indexer_selected_sparse_gb300 import qsa as Q
    from indexer_selected_sparse_gb300 import synth as S

    wl = S.workload(3)
    sh = wl.shapes
    cfg = Q.Config.of(sh)
    B = wl.n_seq
    W, K = max(args.ragged_warmup, 3), max(args.ragged_steps, 1)
    max_pages = math.ceil((max(wl.prefixes) + W + K + 8) / sh.page_size)
    cache = Q.PagedCache(cfg, S.page_table(wl.seed, B, max_pages, contiguous=False), B * max_pages, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    fill_prefixes(Q, S, torch, cfg, sh, wl, cache, wl.prefixes, status, dev)
    ids = torch.arange(B, dtype=torch.int32, device=dev)
    pos0 = torch.tensor(wl.prefixes, dtype=torch.int32, device=dev)
    k, v, ix = zip(*[S.token_rows(sh, wl.seed, s_, torch.tensor([p]), device=dev) for s_, p in enumerate(wl.prefixes)])
    q, qi, w = zip(*[S.query_rows(sh, wl.seed, s_, torch.tensor([p]), device=dev) for s_, p in enumerate(wl.prefixes)])
    cat = lambda xs: torch.cat(xs).contiguous()
    k, v, ix, q, qi, w = map(cat, (k, v, ix, q, qi, w))
    out = torch.empty(B, sh.n_q_heads, sh.head_dim, dtype=torch.bfloat16, device=dev)
    ws = Q.workspace(cfg, B, cache.max_blocks, device=dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        Q.qsa_decode(cfg, Q.Rows(ids, pos0, 1, advance=True), cache, k, v, ix, qi, w, q, out, ws, status,
                     stream=stream)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(W):
            g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(K):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st == 0, f"device status {st}: {Q.qsa_strerror(st)}"
    ms = e0.elapsed_time(e1) / K
    # timed rows: every sequence at prefixes + W .. prefixes + W + K - 1 (visible one more)
    visibles = [p + W + t + 1 for t in range(K) for p in wl.prefixes]
    work = sum_work(sh, visibles)
    step_bytes = (work["score_bytes"] + work["attn_bytes"] + work["append_bytes"]) / K
    hbm_gbs, _, peak_kind = measured_peaks()
    gbs = step_bytes / (ms * 1e-3) / 1e9
    dense = sum(1 for p in wl.prefixes if (p + W + 1) // sh.ratio <= sh.topk)
    return {"workload": wl.name, "batch": B, "steps": K, "warmup": W, "ms_per_step": round(ms, 5),
            "rows_per_s": round(B / (ms * 1e-3), 1), "bytes_per_step": int(step_bytes),
            "achieved_gbs": round(gbs, 1), "hbm_roofline_frac": round(gbs / hbm_gbs, 4),
            "peak_kind": peak_kind + " (hbm_gbs, copy)",
            "rows_dense": dense, "prefix_range": [min(wl.prefixes), max(wl.prefixes)],
            "bytes": "per row: compressed keys (rows past the inert bound), q_idx, w, K+V of the token set, q, o, "
                     "appended rows",
            "timing": f"{K} steps after {W} warm-up, one CUDA graph per step, positions advanced on the device; "
                      f"{step_bytes / 1e9:.2f} GB per step (more than L2)"}


def token_count(sel_rows, visibles, ratio):
    """Distinct tokens of a sequence's rows: each row's selected blocks (expanded
    to their ratio tokens) plus its tail [n_blk * ratio, visible)."""
    toks = set()
    for sel, vis in zip(sel_rows, visibles):
        n_blk = vis // ratio
        for b in sel:
            if b >= 0:
                toks.update(range(b * ratio, b * ratio + ratio))
        toks.update(range(n_blk * ratio, vis))
    return len(toks)


def run_verify(args, dev):
    """Speculative verify + rewind (batch 16, prefix 65536): a cycle is one fused
    qsa_decode of R = 3 causal rows per sequence (2 drafts + 1), the rewind of
    the rejected rows (0..2 per sequence, seeded), 4 decode steps on fresh rows
    at the re-used positions, and a rewind back to the start so the cycle repeats
    on the same data; one CUDA graph per cycle. Algorithmic bytes of the verify rows:
    a sequence's compressed keys once for its 3 verify rows, K+V once per distinct
    token of their sets (the union, from the step's own selections), plus the
    decode rows as in the decode leg."""
    import torch

    from indexer_selected_sparse_gb300 import qsa as Q
    from indexer_selected_sparse_gb300 import synth as S

    wl = S.workload(4)
    sh = wl.shapes
    cfg = Q.Config.of(sh)
    B, R, p = wl.n_seq, wl.rows_per_seq, wl.prefixes[0]
    D = wl.extra["decode_after"]
    rej = S.reject_counts(wl.seed, B)
    max_pages = math.ceil((p + R + D + 8) / sh.page_size)
    cache = Q.PagedCache(cfg, S.page_table(wl.seed, B, max_pages, contiguous=False), B * max_pages, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    fill_prefixes(Q, S, torch, cfg, sh, wl, cache, wl.prefixes, status, dev)
    ids = torch.arange(B, dtype=torch.int32, device=dev)
    cat = lambda xs: torch.cat(xs).contiguous()

    def inputs(positions, epoch):
        rows = [S.token_rows(sh, wl.seed, s_, torch.tensor(ps), epoch=epoch, device=dev) for s_, ps in positions]
        qs = [S.query_rows(sh, wl.seed, s_, torch.tensor(ps), epoch=epoch, device=dev) for s_, ps in positions]
        k, v, ix = (cat([r[i] for r in rows]) for i in range(3))
        q, qi, w = (cat([x[i] for x in qs]) for i in range(3))
        return dict(k=k, v=v, idx=ix, q=q, q_idx=qi, w=w)

    ver = inputs([(s_, list(range(p, p + R))) for s_ in range(B)], 0)
    acc = [R - r for r in rej]
    dec = [inputs([(s_, [p + acc[s_] + j]) for s_ in range(B)], 1) for j in range(D)]
    pos_v = torch.full((B,), p, dtype=torch.int32, device=dev)
    pos_d = [torch.tensor([p + a + j for a in acc], dtype=torch.int32, device=dev) for j in range(D)]
    drop_rej = torch.tensor(rej, dtype=torch.int32, device=dev)
    drop_all = torch.tensor([a + D for a in acc], dtype=torch.int32, device=dev)
    out_v = torch.empty(B * R, sh.n_q_heads, sh.head_dim, dtype=torch.bfloat16, device=dev)
    out_d = torch.empty(B, sh.n_q_heads, sh.head_dim, dtype=torch.bfloat16, device=dev)
    sel_v = torch.empty(B * R, cfg.topk, dtype=torch.int32, device=dev)
    nsel_v = torch.empty(B * R, dtype=torch.int32, device=dev)
    ws = Q.workspace(cfg, B * R, cache.max_blocks, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def cycle():
        Q.qsa_decode(cfg, Q.Rows(ids, pos_v, R), cache, ver["k"], ver["v"], ver["idx"], ver["q_idx"], ver["w"],
                     ver["q"], out_v, ws, status, sel_out=sel_v, n_sel_out=nsel_v, stream=stream)
        Q.qsa_rewind(cfg, ids, drop_rej, cache.ingested, status, stream=stream)
        for j in range(D):
            d = dec[j]
            Q.qsa_decode(cfg, Q.Rows(ids, pos_d[j], 1), cache, d["k"], d["v"], d["idx"], d["q_idx"], d["w"], d["q"],
                         out_d, ws, status, stream=stream)
        Q.qsa_rewind(cfg, ids, drop_all, cache.ingested, status, stream=stream)

    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        cycle()
    torch.cuda.synchronize()
    W, K = max(args.verify_warmup, 3), max(args.verify_cycles, 1)
    with torch.cuda.stream(stream):
        for _ in range(W):
            g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(K):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st == 0, f"device status {st}: {Q.qsa_strerror(st)}"
    assert cache.ingested.cpu().tolist() == [p] * B
    ms = e0.elapsed_time(e1) / K
    # bytes of a cycle: the verify rows (keys once per sequence, K+V once per
    # distinct selected token), then the decode rows
    sel_h = sel_v.cpu().tolist()
    kb = key_bytes(sh, "bf16")
    ver_bytes = 0
    for s_ in range(B):
        vis = [p + j + 1 for j in range(R)]
        n_blk_last = vis[-1] // sh.ratio
        ver_bytes += n_blk_last * kb if n_blk_last > sh.topk else 0
        ver_bytes += R * (sh.n_idx_heads * sh.idx_dim * 2 + 4 * sh.n_idx_heads)
        ver_bytes += token_count(sel_h[s_ * R:(s_ + 1) * R], vis, sh.ratio) * sh.n_kv_heads * sh.head_dim * 4
        ver_bytes += R * (2 * sh.n_q_heads * sh.head_dim * 2 + (2 * sh.n_kv_heads * sh.head_dim + sh.idx_dim) * 2)
    dw = sum_work(sh, [p + acc[s_] + j + 1 for j in range(D) for s_ in range(B)])
    cyc_bytes = ver_bytes + dw["score_bytes"] + dw["attn_bytes"] + dw["append_bytes"]
    hbm_gbs, _, peak_kind = measured_peaks()
    rows = B * R + B * D
    gbs = cyc_bytes / (ms * 1e-3) / 1e9
    return {"workload": wl.name, "cycles": K, "warmup": W, "ms_per_cycle": round(ms, 5),
            "rows_per_cycle": rows, "rows_per_s": round(rows / (ms * 1e-3), 1), "bytes_per_cycle": int(cyc_bytes),
            "achieved_gbs": round(gbs, 1), "hbm_roofline_frac": round(gbs / hbm_gbs, 4),
            "peak_kind": peak_kind + " (hbm_gbs, copy)", "rejected": rej,
            "cycle": f"verify ({B} x {R} causal rows) -> rewind rejected -> {D} decode steps -> rewind to the start; "
                     "one CUDA graph per cycle",
            "bytes": "verify: keys once per sequence, K+V once per distinct token of its rows (union), q_idx, w, q, "
                     "o and appends per row; decode rows as in the decode leg"}


# ---------------------------------------------------------------------------
# CPU oracle (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------

def _oracle_worker(job):
    """Runs in a spawned process: builds one sequence's oracle state at the
    workload's prefix from the seeded generator (untimed), then times `rows`
    decode rows (append the token, score, select, attend, then rewind so every
    row sees the same prefix)."""
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["OMP_NUM_THREADS"] = "1"
    os.environ["MKL_NUM_THREADS"] = "1"
    import numpy as np
    import torch
    torch.set_num_threads(1)
    from indexer_selected_sparse_gb300 import synth as S
    from oracle import qsa_oracle as O

    seq, prefix, n_warm, n_rows, wl_id = job
    wl = S.workload(wl_id)
    sh = wl.shapes

    def b(t):
        return t.contiguous().view(torch.int16).numpy().astype(np.uint16)

    # index keys for every position; K/V rows only where the row attends (the
    # row is the same every time, so its token set is fixed): the oracle's
    # state holds zeros for K/V rows it never reads
    pos = torch.arange(prefix + 1)
    _, _, ix = S.token_rows(S.Shapes(sh.ratio, sh.budget, sh.n_idx_heads, sh.idx_dim, 1, 1, 8),
                            wl.seed, seq, pos)
    q, qi, w = S.query_rows(sh, wl.seed, seq, pos[prefix:])
    qb, qib, wn = b(q[0]), b(qi[0]), w[0].numpy()
    st = O.SeqState(sh.ratio, sh.n_kv_heads, sh.head_dim, sh.idx_dim, prefix + 1)
    z = np.zeros((prefix, sh.n_kv_heads, sh.head_dim), np.uint16)
    st.append(0, z, z, b(ix[:prefix]))
    kn, vn, _ = S.token_rows(sh, wl.seed, seq, pos[prefix:])
    kb, vb, ib = b(kn), b(vn), b(ix[prefix:])
    st.append(prefix, kb, vb, ib)
    toks = O.attend_row(st, prefix, qib, wn, qb, sh.topk)["tokens"]
    st.rewind(1)
    need = torch.from_numpy(toks[toks < prefix])
    kt, vt, _ = S.token_rows(sh, wl.seed, seq, need)
    st.K[need.numpy()] = b(kt)
    st.V[need.numpy()] = b(vt)
    times = []
    for r in range(n_warm + n_rows):
        t0 = time.perf_counter()
        st.append(prefix, kb, vb, ib)
        O.attend_row(st, prefix, qib, wn, qb, sh.topk)
        st.rewind(1)
        t1 = time.perf_counter()
        if r >= n_warm:
            times.append((t0, t1))
    return times


def _prefill_oracle_worker(job):
    """Runs in a spawned process: the chunked-prefill sequence (prefix + chunk,
    every token appended, as the fused step appends the chunk before any row
    attends) built from the seeded generator (untimed), then the oracle row by
    row for the rows given (score, select, attend), each timed."""
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["OMP_NUM_THREADS"] = "1"
    os.environ["MKL_NUM_THREADS"] = "1"
    import numpy as np
    import torch
    torch.set_num_threads(1)
    from indexer_selected_sparse_gb300 import synth as S
    from oracle import qsa_oracle as O

    rows, wl_id = job
    wl = S.workload(wl_id)
    sh = wl.shapes
    p, C = wl.prefixes[0], wl.rows_per_seq
    n = p + C

    def b(t):
        return t.contiguous().view(torch.int16).numpy().astype(np.uint16)

    k, v, ix = S.token_rows(sh, wl.seed, 0, torch.arange(n))
    st = O.SeqState(sh.ratio, sh.n_kv_heads, sh.head_dim, sh.idx_dim, n)
    st.append(0, b(k), b(v), b(ix))
    q, qi, w = S.query_rows(sh, wl.seed, 0, torch.tensor([p + j for j in rows]))
    times = []
    for r, j in enumerate(rows):
        t0 = time.perf_counter()
        O.attend_row(st, p + j, b(qi[r]), w[r].numpy(), b(q[r]), sh.topk)
        times.append((t0, time.perf_counter()))
    return times


def prefill_cpu_baseline(stride=16):
    """The oracle on every stride-th row of the chunked-prefill workload, over up
    to 16 single-thread worker processes; rows/s as for the decode baseline."""
    import multiprocessing as mp
    wl = __import__("indexer_selected_sparse_gb300.synth", fromlist=["synth"]).workload(PREFILL_WORKLOAD_ID)
    rows = list(range(0, wl.rows_per_seq, stride))
    n = min(os.cpu_count() or 1, 16, len(rows))
    jobs = [(rows[i::n], PREFILL_WORKLOAD_ID) for i in range(n)]
    with mp.get_context("spawn").Pool(n) as pool:
        res = pool.map(_prefill_oracle_worker, jobs)
    per_row = statistics.median([t1 - t0 for r in res for (t0, t1) in r])
    return {"value": round(pool_rate(res), 2), "unit": "rows/s", "cores": n, "kind": "oracle",
            "sample": f"a 1/{stride} subsample: rows 0, {stride}, 2*{stride}, ... of the 8193-row chunk "
                      f"({len(rows)} rows) over {n} worker processes (1 BLAS thread each); each row = score, "
                      "select, attend over the whole appended chunk; rate = sum of the workers' own rates",
            "single_thread_rows_per_s": round(1.0 / per_row, 2), "cpu": cpu_model()}


def oracle_pool_run(n_workers, prefix, n_warm, rows_per_worker):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    jobs = [(s, prefix, n_warm, rows_per_worker, WORKLOAD_ID) for s in range(n_workers)]
    with ctx.Pool(n_workers) as pool:
        res = pool.map(_oracle_worker, jobs)
    return res


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for l in f:
                if l.lower().startswith(("model name", "cpu part")):
                    return l.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def pool_rate(res):
    """Rows per second of the worker pool: the sum over workers of each worker's
    own rate (its rows over the span from its first row's start to its last
    row's end). The workers' set-up times differ, so a span from the earliest
    start to the latest end would count their start skew as work time."""
    rate = 0.0
    for r in res:
        span = r[-1][1] - r[0][0]
        rate += len(r) / span if span > 0 else 0.0
    return rate


def cpu_baseline(rows_per_worker):
    n = min(os.cpu_count() or 1, 16)
    res = oracle_pool_run(n, 32768, 1, rows_per_worker)
    rows = sum(len(r) for r in res)
    per_row = statistics.median([t1 - t0 for r in res for (t0, t1) in r])
    return {"value": round(pool_rate(res), 2), "unit": "rows/s", "cores": n, "kind": "oracle",
            "sample": f"{rows} decode rows: {n} worker processes x {rows_per_worker} rows each (1 BLAS thread "
                      f"each), one sequence per worker at prefix 32768 of the batch-32 x 32k workload; each row = "
                      f"append + score + select + attend, then rewind; rate = sum of the workers' own rates",
            "single_thread_rows_per_s": round(1.0 / per_row, 2), "cpu": cpu_model()}


def run_reference(args):
    world, rank, _ = rank_env()
    if rank != 0:
        return  # the oracle runs once, on rank 0's host cores
    n = min(os.cpu_count() or 1, 16)
    K, W = args.steps, args.warmup
    # a step = one decode row (of the batch's 32) on the CPU; the K steps are
    # spread over n worker processes that run in parallel
    res = oracle_pool_run(n, 32768, max(1, math.ceil(W / n)), math.ceil(K / n))
    rows = sum(len(r) for r in res)
    value = pool_rate(res)   # the same method as the GPU arm's cpu_baseline
    wall = rows / value
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "rows/s",
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(wall / K * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "steady-decode b32 prefix32768 r4 B2048 HI64xdI128 Hq32/Hkv4",
                       "sample": f"each step: one decode row; {rows} rows over {n} CPU worker processes"},
            "cpu_baseline": {"value": round(value, 2), "unit": "rows/s", "cores": n, "kind": "oracle",
                             "sample": f"{rows} decode rows at prefix 32768: {n} workers x {math.ceil(K / n)} rows "
                                       "each; rate = sum of the workers' own rates (as the GPU arm's cpu_baseline)",
                             "cpu": cpu_model()},
            "e2e": {"value": round(value, 2), "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    legs = {x.strip() for x in args.legs.split(",") if x.strip()}
    if "decode" not in legs:
        # prefill leg alone (profiling): one line with the prefill object only
        import torch
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        pre = run_prefill(args, torch.device("cuda", local))
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps({"prefill": pre}), flush=True)
        return
    out, rank, world, late = run_gpu(args)
    import torch
    ldev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    if "prefill" in legs:
        out["prefill"] = run_prefill(args, ldev)
    if "ragged" in legs:
        out["ragged"] = guarded(lambda: run_ragged(args, ldev), None if world == 1 else True, torch)
    if "verify" in legs:
        out["verify"] = guarded(lambda: run_verify(args, ldev), None if world == 1 else True, torch)
    if late is not None:
        import torch
        out["attn_options"] = guarded(late, None if world == 1 else True, torch)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(args.oracle_rows)
            if "prefill" in out:
                out["prefill"]["cpu_baseline"] = prefill_cpu_baseline()
        else:
            out["cpu_baseline"] = None
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
