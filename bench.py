#!/usr/bin/env python
"""Throughput of the fused sparse attention step (index scores -> top-k ->
windowed + sparse MQA) on GB300, as one JSON line.

Default workload: ragged long-context decode, batch 128, lengths
U[8192, 131072] (query at L-1), r=4, index 64x128 fp8 keys + per-position
scale, topk 2048, attention 64x128, window 128 -- the largest decode workload
with an HBM-roofline target; ``--workload`` picks another.  One step = one
sa_fused_decode call over the whole batch with its inputs resident in HBM.
Three copies of every input rotate between steps, so each step reads data
evicted from L2 by the two before it.  The line also carries the decode
batch-64 workload and the 4096-token prefill chunk as extra fields
(``workloads``), timed the same way.

``--impl reference`` times the float64 CPU oracle on the host cores instead
(the baseline arm); it never touches the GPU.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "query-tokens/s of fused indexer+top-k+sparse attn; % of HBM roofline"
UNIT = "query-tokens/s"
STAGES = ("idx_score", "idx_topk", "sparse_mqa")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="c4", choices=("c0", "c1", "c2", "c3", "c4"))
    ap.add_argument("--extra", default="c2,c3",
                    help="other workloads timed the same way and reported as extra fields ('' for none)")
    ap.add_argument("--copies", type=int, default=3)
    ap.add_argument("--soak-seconds", type=float, default=1.5)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-two-level", action="store_true", help="skip the two-level top-k measurement")
    ap.add_argument("--no-v41", action="store_true", help="skip the V4.1-shape measurement")
    ap.add_argument("--v41-only", action="store_true", help="print only the V4.1-shape measurement")
    ap.add_argument("--producer-only", action="store_true", help="print only the index-producer measurement")
    ap.add_argument("--compressor-only", action="store_true", help="print only the compressor measurement")
    return ap.parse_args()


def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's value (a job's time is its slowest rank's);
    the value itself without an initialised process group of several ranks."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


# ------------------------------------------------------------- accounting ---

def algorithmic_bytes(w):
    """Per-step algorithmic bytes of each stage (the roofline numerators)."""
    pos = w.q_pos.astype(np.int64)
    nv = np.minimum((pos + 1) // w.r, w.N_c)
    kb = 1 if w.k_dtype == 1 else 2
    key_row = w.D_I * kb + (4 if w.k_scale is not None else 0)
    n_w = np.minimum(w.W, pos + 1)
    k_eff = np.minimum(w.K, nv)
    kv_row = 2 * w.D * 2  # K and V rows, bf16
    return {
        "idx_score": int(np.sum(nv) * key_row),
        "idx_topk": int(np.sum(nv) * 4 + w.T * w.K * 4),
        "sparse_mqa": int(np.sum(n_w + k_eff) * kv_row),
        "step": int(np.sum(nv) * key_row + np.sum(n_w + k_eff) * kv_row),
    }


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


STAGE_SOURCES = {"idx_score": ("idx_score.cu", "idx_score_umma.cu", "umma.cuh", "common.cuh"),
                 "idx_topk": ("idx_topk.cu", "common.cuh"),
                 "level_one": ("idx_candidates.cu", "common.cuh"),
                 "level_two": ("idx_topk.cu", "common.cuh"),
                 "index_producer": ("idx_producer.cu", "common.cuh"),
                 "sparse_mqa": ("sparse_mqa.cu", "sparse_mqa_umma.cu", "sparse_mqa_umma512.cu", "umma.cuh",
                                "common.cuh")}


def _code_only(text):
    """Source text without comments, blank lines or trailing blanks: an edit to
    a comment leaves the hash (and so a recorded capture) unchanged."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash(stage):
    h = hashlib.sha256()
    for src in STAGE_SOURCES[stage]:
        with open(os.path.join(ROOT, "indexer_selected_sparse_score_gb300", "csrc", src)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(stage, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of that kernel (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(f"{stage}:{workload}")
    except Exception:
        return None
    if not rec or rec.get("source_sha256_16") != kernel_source_hash(stage):
        return None
    return rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------- clocks ---

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.rows = []
        self.proc = None
        sel = []
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            if vis:
                sel = ["-i", vis.split(",")[device_index]]
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "200", *sel]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 7:
                self.rows.append((time.time(), parts))

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [p for (ts, p) in self.rows if t0 <= ts <= t1]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(p[0]) for p in rows if p[0].replace(".", "", 1).isdigit()]
        mx = [float(p[1]) for p in rows if p[1].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in rows for i in range(4) if p[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------- reference arm ---

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from indexer_selected_sparse_score_gb300 import workloads as wl
    oracle.build()
    threads = os.cpu_count() or 1
    oracle.set_threads(threads)
    w = wl.generate(wl.CONFIGS[args.workload])
    p = oracle.Problem(**w.problem_fields())
    # size each step's sample so that the whole run stays within ~150 s
    t0 = time.perf_counter()
    oracle.fused(p, w.K, rows=[0])
    one = time.perf_counter() - t0
    per_step_budget = 150.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(w.T, math.floor(per_step_budget * threads / max(one, 1e-6)))))
    cursor = 0

    def step():
        nonlocal cursor
        rows = [(cursor + i) % w.T for i in range(n)]
        cursor = (cursor + n) % w.T
        oracle.fused(p, w.K, rows=rows)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = n * args.steps / el
    sample = f"{n} of the {w.T} query tokens per step (rotating), float64 oracle, {threads} threads"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{w.spec.name}: {w.spec.description}",
                                          "global_batch": n, "seed": w.seed},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ---------------------------------------------------------------- our arm ---

def cpu_baseline(w, seconds):
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    oracle.set_threads(threads)
    p = oracle.Problem(**w.problem_fields())
    t0 = time.perf_counter()
    oracle.fused(p, w.K, rows=[0])
    one = time.perf_counter() - t0
    n = int(max(1, min(w.T, math.floor(seconds * threads / max(one, 1e-6)))))
    rows = list(range(n))
    t0 = time.perf_counter()
    oracle.fused(p, w.K, rows=rows)
    el = time.perf_counter() - t0
    return {"value": n / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"query tokens 0..{n - 1} of the {w.T}-token batch (same seeded workload), "
                      f"float64 oracle, one OpenMP thread per host core, {el:.1f} s"}


CAND_BLOCK, CAND_BLOCKS = 8, 2048  # candidate blocks of 8 positions, 2048 of them kept


def two_level_topk(binding, torch, wl, steps, peak):
    """Device time of the two-level top-k: level one (sa_candidate_blocks, 2048
    blocks of 8 kept) and level two (sa_topk_candidates), with the one-level
    sa_topk beside them, on rows shaped like the ragged long-context decode
    workload (128 tokens, N_c 32768, lengths U[8192, 131072], r 4; N(0,1)
    scores, -inf past each token's visible end).  L2 is flushed before every
    timed launch; each launch is bracketed by its own CUDA events."""
    spec = wl.CONFIGS["c4"]
    q_seq, q_pos = wl.draw_positions(spec, wl.SEEDS["c4"])
    nv = np.minimum((q_pos.astype(np.int64) + 1) // spec.r, spec.N_c)
    T, N_c, K = spec.T, spec.N_c, spec.K
    gen = torch.Generator(device="cuda").manual_seed(7)
    scores = torch.randn((T, N_c), device="cuda", generator=gen)
    d_nv = torch.from_numpy(nv).cuda()
    scores[torch.arange(N_c, device="cuda")[None, :] >= d_nv[:, None]] = float("-inf")
    d_seq = torch.from_numpy(q_seq).cuda()
    d_pos = torch.from_numpy(q_pos).cuda()
    ia = binding.IndexArgs(spec.B, T, spec.H_I, spec.D_I, N_c, spec.r, d_seq.data_ptr(), d_pos.data_ptr(),
                           None, 0, None, None, None, 0, None)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    binding.sa_workspace_init(ws)
    words = binding.sa_candidate_words(N_c, CAND_BLOCK)
    cand = torch.empty((T, words), dtype=torch.int32, device="cuda")
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")  # twice L2
    calls = {
        "level_one": lambda: binding.sa_candidate_blocks(scores, ia, CAND_BLOCK, CAND_BLOCKS, cand, ws),
        "level_two": lambda: binding.sa_topk_candidates(scores, ia, K, cand, CAND_BLOCK, idx, ws),
        "one_level_topk": lambda: binding.sa_topk(scores, ia, K, idx, ws),
    }
    for f in calls.values():  # warm-up (and the mask level two reads)
        for _ in range(3):
            f()
    calls["level_one"]()
    n = max(5, steps)
    ms = {}
    for name, f in calls.items():
        if name == "level_two":
            calls["level_one"]()
        tot = 0.0
        for _ in range(n):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            f()
            e1.record()
            torch.cuda.synchronize()
            tot += e0.elapsed_time(e1)
        ms[name] = tot / n
    if binding.sa_check_device_status(ws) != binding.SA_OK:
        raise RuntimeError("device status not OK after the two-level top-k")
    nb = (nv + CAND_BLOCK - 1) // CAND_BLOCK
    # level two reads the scores of the kept visible positions (blocks of 8 are
    # compacted), counted from level one's mask
    bits = np.unpackbits(cand.cpu().numpy().view(np.uint8), axis=1, bitorder="little")
    kept_vis = 0
    for t in range(T):
        kb = np.nonzero(bits[t, :nb[t]])[0]
        c = len(kb) * CAND_BLOCK
        if len(kb) and kb[-1] == nb[t] - 1:
            c -= int(nb[t]) * CAND_BLOCK - int(nv[t])
        kept_vis += c
    alg = {"level_one": int(nv.sum() * 4 + T * words * 4),          # visible scores read, mask written
           "level_two": int(kept_vis * 4 + T * words * 4 + T * K * 4),  # kept scores and mask read, indices written
           "one_level_topk": int(nv.sum() * 4 + T * K * 4)}
    res = {"workload": "128 tokens, N_c 32768, lengths U[8192,131072], r 4 (the ragged long-context decode "
                       "geometry); N(0,1) fp32 scores; blocks of 8, 2048 kept; K 2048; L2 flushed per launch",
           "rows_with_selection": int(np.sum(nb > CAND_BLOCKS))}
    for name, v in ms.items():
        gbs = alg[name] / (v / 1000.0) / 1e9
        res[name] = {"us": round(v * 1000.0, 2), "algorithmic_bytes": alg[name], "GB_s": round(gbs, 1),
                     "frac_of_hbm_peak": round(gbs / peak, 4),
                     "traffic": recorded_traffic(name if name != "one_level_topk" else "idx_topk", "c4_two_level")}
    return res


def v41_decode(binding, torch, steps, peak):
    """The fused step on the released V4.1 attention shape: decode batch 64 at
    positions U[32768, 65535], r 2 (N_c 32768), index 32 x 128 with bf16 queries and
    fp8 keys + per-position scale U(0.5, 2), w U(0,1)/32, top-k 512, window 128,
    64 query heads of dim 512 over one kv tensor used as K and V, a per-head sink,
    scale 512^-0.5.  Inputs are drawn on the device (seeded N(0,1)), three copies
    rotate between steps; CUDA-graph replay of sa_fused_decode, plus the stage
    times from sa_fused_decode_staged."""
    B = T = 64
    r, N_c, H_I, D_I, K, W, R, H, D = 2, 32768, 32, 128, 512, 128, 128, 64, 512
    q_pos = np.random.default_rng(41).integers(32768, 65535, size=T, endpoint=True).astype(np.int32)
    q_seq = np.arange(T, dtype=np.int32)
    gen = torch.Generator(device="cuda").manual_seed(41)
    bf = torch.bfloat16

    def normal(shape, dtype=bf):
        return torch.empty(shape, dtype=dtype, device="cuda").normal_(generator=gen)

    copies = []
    for _ in range(3):
        d = {"q_seq": torch.from_numpy(q_seq).cuda(), "q_pos": torch.from_numpy(q_pos).cuda(),
             "q_I": normal((T, H_I, D_I)), "w": torch.rand((T, H_I), device="cuda", generator=gen) / 32,
             "k_I": normal((B, N_c, D_I)).to(torch.float8_e4m3fn),
             "k_scale": torch.rand((B, N_c), device="cuda", generator=gen) * 1.5 + 0.5,
             "Q": normal((T, H, D)), "KVw": normal((B, R, D)), "KVc": normal((B, N_c, D)),
             "sink": normal((H,), torch.float32)}
        ia = binding.IndexArgs(B, T, H_I, D_I, N_c, r, d["q_seq"].data_ptr(), d["q_pos"].data_ptr(),
                               d["q_I"].data_ptr(), 0, None, d["w"].data_ptr(), d["k_I"].data_ptr(), 1,
                               d["k_scale"].data_ptr())
        aa = binding.AttnArgs(H, D, W, R, d["Q"].data_ptr(), d["KVw"].data_ptr(), d["KVw"].data_ptr(),
                              d["KVc"].data_ptr(), d["KVc"].data_ptr(), d["sink"].data_ptr(), float(D) ** -0.5)
        copies.append((d, ia, aa))
    n = binding.sa_workspace_size(copies[0][1], copies[0][2], K)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    binding.sa_workspace_init(ws)
    out = torch.empty((T, H, D), dtype=bf, device="cuda")
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    for _, ia, aa in copies:
        binding.sa_fused_decode(ia, aa, K, idx, out, ws)
    torch.cuda.synchronize()
    graphs = []
    for _, ia, aa in copies:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            binding.sa_fused_decode(ia, aa, K, idx, out, ws)
        graphs.append(g)
    for i in range(6):
        graphs[i % 3].replay()
    torch.cuda.synchronize()
    n_steps = max(10, steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(n_steps):
        graphs[i % 3].replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n_steps
    # stage times: one staged graph per copy (events between the stages), each
    # replayed right after the previous copy's step
    stage_events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in copies]
    for row in stage_events:
        for e in row:
            e.record()  # materialise the CUDA event handles
    torch.cuda.synchronize()
    staged = []
    for (_, ia, aa), evs in zip(copies, stage_events):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            binding.sa_fused_decode_staged(ia, aa, K, idx, out, ws, [e.cuda_event for e in evs])
        staged.append(g)
    sums = [0.0, 0.0, 0.0]
    for i in range(n_steps):
        k = i % 3
        staged[(k - 1) % 3].replay()
        staged[k].replay()
        torch.cuda.synchronize()
        for j in range(3):
            sums[j] += stage_events[k][j].elapsed_time(stage_events[k][j + 1])
    if binding.sa_check_device_status(ws) != binding.SA_OK:
        raise RuntimeError("device status not OK after the V4.1-shape steps")
    nv = np.minimum((q_pos.astype(np.int64) + 1) // r, N_c)
    n_w = np.minimum(W, q_pos.astype(np.int64) + 1)
    idx_bytes = int(np.sum(nv) * (D_I + 4))
    attn_bytes = int(np.sum(n_w + np.minimum(K, nv)) * D * 2)  # one kv row serves as K and V
    step_bytes = idx_bytes + attn_bytes
    st = dict(zip(("idx_score", "idx_topk", "sparse_mqa"), (v / n_steps for v in sums)))
    attn_flop = float(np.sum(n_w + np.minimum(K, nv))) * H * D * 4  # Q.K and P.V
    return {"workload": "V4.1 released attention shape: decode batch 64, positions U[32768,65535], r 2, "
                        "index 32x128 fp8 keys + scale, topk 512, window 128, 64 heads x dim 512, one kv "
                        "tensor as K and V, sink; device-drawn N(0,1) inputs, 3 rotating copies",
            "ms_per_step": round(ms, 5), "value": round(T / (ms / 1000.0), 1), "unit": "query-tokens/s",
            "step_bytes": step_bytes, "frac_of_hbm_peak": round(step_bytes / (ms / 1000.0) / 1e9 / peak, 4),
            "stages_ms": {k: round(v, 5) for k, v in st.items()},
            "idx_score_GB_s": round(idx_bytes / (st["idx_score"] / 1000.0) / 1e9, 1),
            "sparse_mqa_GB_s": round(attn_bytes / (st["sparse_mqa"] / 1000.0) / 1e9, 1),
            "sparse_mqa_TFLOP_s": round(attn_flop / (st["sparse_mqa"] / 1000.0) / 1e12, 2),
            "sparse_mqa_traffic": recorded_traffic("sparse_mqa", "v41"),
            "note": "attention at head dim 512 runs on the tcgen05 kernel (sparse_mqa_umma512): one token per 2-CTA cluster, the parts merged over distributed shared memory"}


def index_producer(binding, torch, steps, peak):
    """Device time of sa_rotate_quant (the V3.2 index producer: Hadamard
    rotation and e4m3 block quantisation) on the rows of a 4096-token prefill
    chunk: 64 query heads + 1 key per token = 266,240 rows of 128 bf16 values
    (device-drawn N(0,1)); L2 flushed before each launch."""
    rows = 4096 * 65
    gen = torch.Generator(device="cuda").manual_seed(32)
    x = torch.empty((rows, 128), dtype=torch.bfloat16, device="cuda").normal_(generator=gen)
    codes = torch.empty((rows, 128), dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, dtype=torch.float32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    binding.sa_workspace_init(ws)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        binding.sa_rotate_quant(x, rows, codes, scales, ws)
    n, tot = max(5, steps), 0.0
    for _ in range(n):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        binding.sa_rotate_quant(x, rows, codes, scales, ws)
        e1.record()
        torch.cuda.synchronize()
        tot += e0.elapsed_time(e1)
    if binding.sa_check_device_status(ws) != binding.SA_OK:
        raise RuntimeError("device status not OK after the index producer")
    us = tot / n * 1000.0
    alg = rows * (128 * 2 + 128 + 4)
    gbs = alg / (us / 1e6) / 1e9
    return {"workload": "rows of a 4096-token prefill chunk: 64 query heads + 1 key, 128 bf16 each "
                        "(266,240 rows); L2 flushed per launch",
            "us": round(us, 2), "algorithmic_bytes": alg, "GB_s": round(gbs, 1),
            "frac_of_hbm_peak": round(gbs / peak, 4), "traffic": recorded_traffic("index_producer", "prefill")}


def time_workload(binding, torch, w, n_copies, steps, warmup, before_timed=None, after_timed=None):
    """Device time of the fused step on workload ``w``: ``n_copies`` device
    copies of the inputs rotate between steps; one CUDA graph per copy holds
    one sa_fused_decode call.  Returns the time of exactly ``steps`` graph
    replays between CUDA events on the launching stream (after ``warmup``
    untimed replays), the same steps launched eagerly, and per-stage times from
    staged graphs (events between the stages), each measured step replayed
    right after the previous copy's step so that it starts on a busy GPU, as in
    the timed loop."""
    copies = [binding.upload(w, device="cuda") for _ in range(max(1, n_copies))]
    K = w.K
    ws = binding.new_workspace(copies[0])
    out = torch.empty((w.T, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((w.T, max(K, 1)), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    launches_per_step = binding.sa_fused_decode_launch_count(copies[0].ia, copies[0].aa, K)

    def eager_step(i):
        dp = copies[i % len(copies)]
        binding.sa_fused_decode(dp.ia, dp.aa, K, idx, out, ws, stream)

    for i in range(warmup):
        eager_step(i)
    torch.cuda.synchronize()
    if binding.sa_check_device_status(ws) != binding.SA_OK:
        raise RuntimeError("device status not OK after warm-up")
    graphs = []
    for dp in copies:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            binding.sa_fused_decode(dp.ia, dp.aa, K, idx, out, ws)
        graphs.append(g)
    stage_events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in copies]
    for row in stage_events:
        for e in row:
            e.record(stream)  # materialise the CUDA event handles
    torch.cuda.synchronize()
    staged_graphs = []
    for dp, evs in zip(copies, stage_events):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            binding.sa_fused_decode_staged(dp.ia, dp.aa, K, idx, out, ws, [e.cuda_event for e in evs])
        staged_graphs.append(g)
    for i in range(max(3, warmup)):
        graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()

    def step(i):
        graphs[i % len(graphs)].replay()

    if before_timed:
        before_timed(step)
    # ---- timed region: exactly `steps` graph replays
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    if after_timed:
        after_timed()
    ms_total = ev0.elapsed_time(ev1)
    # ---- the same steps launched eagerly through the C ABI (no graph)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        eager_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    eager_ms_per_step = e0.elapsed_time(e1) / steps
    # ---- per-stage device time from the staged graphs
    sums = {s_: 0.0 for s_ in STAGES}
    for i in range(steps):
        k = i % len(staged_graphs)
        staged_graphs[(k - 1) % len(staged_graphs)].replay()
        staged_graphs[k].replay()
        torch.cuda.synchronize()
        evs = stage_events[k]
        for j, s_ in enumerate(STAGES):
            sums[s_] += evs[j].elapsed_time(evs[j + 1])
    stage_ms = {s_: sums[s_] / steps for s_ in STAGES}
    if binding.sa_check_device_status(ws) != binding.SA_OK:
        raise RuntimeError("device status not OK after the timed steps")
    return {"copies": copies, "ws": ws, "out": out, "idx": idx, "stream": stream,
            "launches_per_step": launches_per_step, "ms_total": ms_total,
            "eager_ms_per_step": eager_ms_per_step, "stage_ms": stage_ms}


def workload_field(binding, torch, wl, name, steps, warmup, n_copies, peak):
    """One extra workload, timed like the headline line: query-tokens/s, the
    step's HBM-roofline fraction, and per-stage times, bytes and traffic."""
    spec = wl.CONFIGS[name]
    w = wl.generate(spec)
    tw = time_workload(binding, torch, w, n_copies, steps, warmup)
    ms = tw["ms_total"] / steps
    nbytes = algorithmic_bytes(w)
    res = {"workload": f"{spec.name}: {spec.description}", "ms_per_step": round(ms, 5),
           "value": round(w.T / (ms / 1000.0), 1), "unit": UNIT, "step_bytes": nbytes["step"],
           "frac_of_hbm_peak": round(nbytes["step"] / (ms / 1000.0) / 1e9 / peak, 4),
           "frac_of_8TBps": round(nbytes["step"] / (ms / 1000.0) / 8e12, 4),
           "eager_ms_per_step": round(tw["eager_ms_per_step"], 5),
           "stages": {s: {"ms": round(tw["stage_ms"][s], 5), "algorithmic_bytes": nbytes[s],
                          "GB_s": round(nbytes[s] / (tw["stage_ms"][s] / 1000.0) / 1e9, 1),
                          "traffic": recorded_traffic(s, name)} for s in STAGES}}
    if name == "c3":
        res["note"] = ("prefill: 4096 queries share one sequence's keys, so the per-query bytes of the metric "
                       "are mostly L2 hits; the stage is tensor-bound (index ~0.52 TFLOP fp8, attention "
                       "~0.29 TFLOP bf16)")
        res["tensor_tflops"] = {
            "idx_score": round(2.0 * float(np.sum(np.minimum((w.q_pos.astype(np.int64) + 1) // w.r, w.N_c)))
                               * w.H_I * w.D_I / (tw["stage_ms"]["idx_score"] / 1000.0) / 1e12, 1),
            "sparse_mqa": round(4.0 * float(np.sum(np.minimum(w.W, w.q_pos.astype(np.int64) + 1)
                                                   + np.minimum(w.K, (w.q_pos.astype(np.int64) + 1) // w.r)))
                                * w.H * w.D / (tw["stage_ms"]["sparse_mqa"] / 1000.0) / 1e12, 1)}
    del tw
    torch.cuda.empty_cache()
    return res


def compressor_field(binding, torch, steps, peak):
    """Device time of the V4.1 compressor (row f3) on synthetic inputs, L2
    flushed before each launch: the prefill of a 4096-token chunk (D 512,
    r 4: 1024 groups), one decode step of 128 sequences whose groups all
    complete, and the index-key producer on the chunk's 1024 compressed rows
    and on the decode step's 128."""
    gen = torch.Generator(device="cuda").manual_seed(44)
    D, r, S = 512, 4, 4096
    G = S // r
    kv = torch.randn((1, S, D), device="cuda", generator=gen)
    sc = torch.randn((1, S, D), device="cuda", generator=gen)
    w = torch.rand(D, device="cuda", generator=gen) + 0.5
    latent = torch.empty((1, G, D), dtype=torch.bfloat16, device="cuda")
    B = 128
    kv_d = torch.randn((B, D), device="cuda", generator=gen)
    sc_d = torch.randn((B, D), device="cuda", generator=gen)
    kvs = torch.randn((B, r, D), device="cuda", generator=gen)
    scs = torch.randn((B, r, D), device="cuda", generator=gen)
    pos = torch.full((B,), 4 * 8191 + 3, dtype=torch.int32, device="cuda")  # every group completes
    out_d = torch.empty((B, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    binding.sa_workspace_init(ws)
    rope = binding.RopeArgs(64, 160000.0, 16.0, 65536, 32.0, 1.0)
    kn = torch.rand(128, device="cuda", generator=gen) + 0.5
    kproj = torch.randn((G, 128), device="cuda", generator=gen).bfloat16()
    kI = torch.empty((B, 32768, 128), dtype=torch.uint8, device="cuda")
    ks = torch.empty((B, 32768), dtype=torch.float32, device="cuda")
    seq_p = torch.zeros(G, dtype=torch.int32, device="cuda")
    grp_p = torch.arange(G, dtype=torch.int32, device="cuda")
    seq_d = torch.arange(B, dtype=torch.int32, device="cuda")
    grp_d = torch.full((B,), 8191, dtype=torch.int32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    calls = {
        "prefill_4096x512": (lambda: binding.sa_compress_prefill(kv, sc, 1, S, D, r, w, 1e-6, latent),
                             2 * S * D * 4 + G * D * 2),
        "decode_b128x512": (lambda: binding.sa_compress_decode(kv_d, sc_d, pos, B, D, r, kvs, scs, w, 1e-6, out_d, ws),
                            B * (2 * D * 4 + 2 * D * 4 + 2 * r * D * 4 + D * 2)),
        "index_keys_1024_rows": (lambda: binding.sa_index_key_publish(kproj, G, seq_p, grp_p, r, kn, 1e-6, rope, kI,
                                                                      ks, B, 32768, ws),
                                 G * (128 * 2 + 128 + 4 + 8)),
        "index_keys_128_rows": (lambda: binding.sa_index_key_publish(kproj[:B], B, seq_d, grp_d, r, kn, 1e-6, rope, kI,
                                                                     ks, B, 32768, ws),
                                B * (128 * 2 + 128 + 4 + 8)),
    }
    res = {"workload": "prefill chunk of 4096 tokens (D 512, r 4); decode step of 128 sequences whose groups all "
                       "complete; index keys (128 values, rope 64, YaRN) for 1024 and 128 rows; N(0,1) inputs; "
                       "L2 flushed per launch"}
    for name, (f, alg) in calls.items():
        for _ in range(3):
            f()
        tot, n = 0.0, max(5, steps)
        for _ in range(n):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            f()
            e1.record()
            torch.cuda.synchronize()
            tot += e0.elapsed_time(e1)
        us = tot / n * 1000.0
        gbs = alg / (us / 1e6) / 1e9
        res[name] = {"us": round(us, 2), "algorithmic_bytes": alg, "GB_s": round(gbs, 1),
                     "frac_of_hbm_peak": round(gbs / peak, 4)}
    if binding.sa_check_device_status(ws) != binding.SA_OK:
        raise RuntimeError("device status not OK after the compressor")
    return res


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    from indexer_selected_sparse_score_gb300 import binding, build
    from indexer_selected_sparse_score_gb300 import workloads as wl

    if local_rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    binding.load()

    if args.producer_only:
        if rank == 0:
            print(json.dumps({"index_producer": index_producer(binding, torch, args.steps, peaks()[0])}), flush=True)
        return
    if args.compressor_only:
        if rank == 0:
            print(json.dumps({"compressor": compressor_field(binding, torch, args.steps, peaks()[0])}), flush=True)
        return
    if args.v41_only:
        if rank == 0:
            print(json.dumps({"v41_decode": v41_decode(binding, torch, args.steps, peaks()[0])}), flush=True)
        return
    spec = wl.CONFIGS[args.workload]
    w = wl.generate(spec, seed=wl.SEEDS[spec.name] + 1000 * rank)
    sampler = ClockSampler(local_rank)
    soak = {}

    def clock_soak(step):
        sampler.start()
        soak["t0"] = time.time()
        i = 0
        while time.time() - soak["t0"] < args.soak_seconds:  # same steps, untimed, to read clocks under load
            step(i)
            i += 1
            if i % 64 == 0:
                torch.cuda.synchronize()
        if world > 1:
            dist.barrier()

    def after_timed():
        if world > 1:
            dist.barrier()
        soak["t1"] = time.time()
        sampler.stop()

    tw = time_workload(binding, torch, w, args.copies, args.steps, args.warmup,
                       before_timed=clock_soak, after_timed=after_timed)
    copies, ws, out, idx, K, stream = tw["copies"], tw["ws"], tw["out"], tw["idx"], w.K, tw["stream"]
    launches_per_step = tw["launches_per_step"]
    ms = max_over_ranks(tw["ms_total"], "cuda")
    ms_per_step = ms / args.steps
    value = w.T * world * args.steps / (ms / 1000.0)
    eager_ms_per_step = tw["eager_ms_per_step"]
    stage_ms = tw["stage_ms"]

    # ---- end to end through the C ABI with host buffers: every step copies its
    # query inputs from one pinned host staging buffer (one H2D copy), runs the
    # fused call on them, and reads out + idx back (one D2H copy)
    names = ("q_seq", "q_pos", "q_I", "q_scale", "w", "Q")
    host = {n: np.ascontiguousarray(getattr(w, n)) for n in names if getattr(w, n) is not None}
    offs, off = {}, 0
    for n, a in host.items():
        off = (off + 255) & ~255
        offs[n] = off
        off += a.nbytes
    h_in = torch.empty(off, dtype=torch.uint8).pin_memory()
    h_in_np = h_in.numpy()
    for n, a in host.items():
        h_in_np[offs[n]:offs[n] + a.nbytes] = a.reshape(-1).view(np.uint8)
    h2d = off
    ob = out.numel() * out.element_size()
    ib_off = (ob + 255) & ~255
    # two output buffers (device and pinned host), alternating per step
    d_outs = [torch.empty(ib_off + idx.numel() * idx.element_size(), dtype=torch.uint8, device="cuda")
              for _ in range(2)]
    outs_v = [(d[:ob].view(out.dtype).view(out.shape), d[ib_off:].view(idx.dtype).view(idx.shape)) for d in d_outs]
    h_outs = [torch.empty(d.numel(), dtype=torch.uint8).pin_memory() for d in d_outs]
    d2h = d_outs[0].numel()
    e2e_args = []  # per input copy: device staging buffer and argument structs pointing into it
    for dp in copies:
        d_in = torch.empty(off, dtype=torch.uint8, device="cuda")
        ia = binding.IndexArgs(*[getattr(dp.ia, f_) for f_, _ in binding.IndexArgs._fields_])
        aa = binding.AttnArgs(*[getattr(dp.aa, f_) for f_, _ in binding.AttnArgs._fields_])
        base = d_in.data_ptr()
        for n in host:
            if n == "Q":
                aa.Q = base + offs[n]
            else:
                setattr(ia, n, base + offs[n])
        e2e_args.append((d_in, ia, aa))
    # A serving loop's pipeline: step i's inputs go up on one copy stream while
    # step i-1 computes, and step i-1's outputs come back on another while step
    # i computes; events order every reuse of a buffer.
    up_stream, down_stream = torch.cuda.Stream(), torch.cuda.Stream()
    nsteps_total = args.steps + 2
    ev_up = [torch.cuda.Event() for _ in range(nsteps_total)]
    ev_comp = [torch.cuda.Event() for _ in range(nsteps_total)]
    ev_down = [torch.cuda.Event() for _ in range(nsteps_total)]

    def e2e_step(i, g):
        d_in, ia, aa = e2e_args[i % len(e2e_args)]
        with torch.cuda.stream(up_stream):
            if g >= len(e2e_args):  # the staging buffer was read by step g - 3
                up_stream.wait_event(ev_comp[g - len(e2e_args)])
            d_in.copy_(h_in, non_blocking=True)
            ev_up[g].record(up_stream)
        stream.wait_event(ev_up[g])
        if g >= 2:  # the output buffer was read back by step g - 2
            stream.wait_event(ev_down[g - 2])
        out_v, idx_v = outs_v[g % 2]
        binding.sa_fused_decode(ia, aa, K, idx_v, out_v, ws, stream)
        ev_comp[g].record(stream)
        with torch.cuda.stream(down_stream):
            down_stream.wait_event(ev_comp[g])
            h_outs[g % 2].copy_(d_outs[g % 2], non_blocking=True)
            ev_down[g].record(down_stream)

    for i in range(2):
        e2e_step(i, i)
    torch.cuda.synchronize()
    ev_up = [torch.cuda.Event() for _ in range(nsteps_total)]
    ev_comp = [torch.cuda.Event() for _ in range(nsteps_total)]
    ev_down = [torch.cuda.Event() for _ in range(nsteps_total)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up_stream.wait_stream(stream)
    down_stream.wait_stream(stream)
    for i in range(args.steps):
        e2e_step(i, i)
    stream.wait_stream(up_stream)
    stream.wait_stream(down_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), "cuda")
    e2e_value = w.T * world * args.steps / (e2e_ms / 1000.0)

    # ---- roofline of the dominant kernel
    nbytes = algorithmic_bytes(w)
    peak, peak_src = peaks()
    dom = max(STAGES, key=lambda s: stage_ms[s])
    achieved = nbytes[dom] / (stage_ms[dom] / 1000.0) / 1e9
    traffic = recorded_traffic(dom, spec.name)
    stages = {s: {"ms": round(stage_ms[s], 5), "algorithmic_bytes": nbytes[s],
                  "GB_s": round(nbytes[s] / (stage_ms[s] / 1000.0) / 1e9, 1) if stage_ms[s] > 0 else None}
              for s in STAGES}
    step_frac = nbytes["step"] / (ms_per_step / 1000.0) / 1e9 / peak

    clocks = sampler.summary(soak["t0"], soak["t1"])
    two_level = None if args.no_two_level else two_level_topk(binding, torch, wl, args.steps, peak)
    v41 = None if args.no_v41 else v41_decode(binding, torch, args.steps, peak)
    producer = index_producer(binding, torch, args.steps, peak)
    compressor = compressor_field(binding, torch, args.steps, peak)
    extra = {}
    for name in [x for x in args.extra.split(",") if x and x != spec.name]:
        extra[name] = workload_field(binding, torch, wl, name, args.steps, args.warmup, args.copies, peak)
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8/bf16 in, fp32 accumulate",
        "data": "synthetic (seeded, shapes and distributions of the workload)",
        "config": {"workload": f"{spec.name}: {spec.description}", "global_batch": w.T * world,
                   "per_gpu_batch": w.T, "seed": w.seed,
                   "l2": f"{len(copies)} rotating input copies; each step's {nbytes['step'] / 1e6:.1f} MB "
                         f"is evicted by the others (L2 129 MB)",
                   "parallelism": f"replicas x{world}"},
        "hbm_roofline": {"step_bytes": nbytes["step"], "frac_of_peak": round(step_frac, 4),
                         "frac_of_8TBps": round(nbytes["step"] / (ms_per_step / 1000.0) / 8e12, 4)},
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else peak_src,
                     "algorithmic_bytes_per_launch": nbytes[dom]},
        "stages": stages,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "every step copies its query inputs from pinned host memory (one copy) and reads out + idx "
                        "back (one copy); the copies run on their own streams, overlapped with the neighbouring "
                        "steps' compute; index/KV caches resident"},
        "gpu_launches": launches_per_step * args.steps,
        "launch": "CUDA graph replay of one sa_fused_decode call per step",
        "eager": {"ms_per_step": round(eager_ms_per_step, 5),
                  "value": w.T * world / (eager_ms_per_step / 1000.0),
                  "note": "the same steps launched through the C ABI without a graph"},
        "clocks": clocks,
        "two_level_topk": two_level,
        "v41_decode": v41,
        "index_producer": producer,
        "compressor": compressor,
        "workloads": extra,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
