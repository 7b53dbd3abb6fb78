#!/usr/bin/env python3
"""Benchmark of the speculative-sampling verify step on GB300.

One step = one spec_verify call over one batch of a workload.  The headline
line is the largest single-GPU workload (B=512, ragged gamma_b in 1..8,
V=152064, bf16, T=0.7, top-k 100 then top-p 0.9); the same measurement runs
on the other target workloads and goes into ``per_config``:

  1  B=64,   gamma=4, V=50304,  fp32, T=1,   top-k 50 then top-p 0.9
  2  B=256,  gamma=8, V=128256, bf16, T=0.8, top-p 0.95
  3  B=4096, gamma=4, V=1024,   fp32, T=1,   Dirichlet(0.3) laws

Inputs are seeded and synthetic, resident in HBM, and rotated over enough
distinct sets that the bytes the kernel reads between two uses of a set
exceed 3x the L2 size.  The timed region replays a captured CUDA graph of
exactly K launches; per-launch CUDA events on the same stream give the
kernel duration for the roofline.

Per workload the line reports:
  * value: verified draft positions/s (sum of gamma_b per call / time);
  * roofline.frac: nominal bytes (both logit tensors read once over the
    valid positions, sum_b (2 gamma_b + 1) V s) / kernel time / measured
    HBM peak; frac_early_exit: the same with the bytes the method must read
    given where each row stopped; traffic: DRAM bytes per launch from the
    committed ncu summary of the current kernel source (else null);
  * e2e: the same metric with every step's inputs copied from pinned host
    memory and the outputs copied back inside the timed region;
  * cpu_baseline (rank 0, one GPU): the fp64 oracle on the host cores over
    a bounded sample of rows of the first timed input set, and on the same
    rows the GPU/oracle parity counts (rows, draws, draws near a boundary,
    disagreements, hard disagreements): the oracle draws these rows' draft
    tokens itself with its own sampler, the GPU verifies the whole set with
    those tokens, and the sampled rows are compared.

``--impl reference`` times the fp64 CPU oracle as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_verify_03_gb300 import workloads as W  # noqa: E402

METRIC = "verified draft positions/sec (BxgammaxV logits) and achieved HBM GB/s vs peak"
UNIT = "positions/s"
PROFILES = os.path.join(ROOT, "profiles")
HEADLINE = 4
PER_CONFIG = (1, 2, 3)
EPS_BOUNDARY = 1e-6  # a draw this close to a decision or CDF boundary is exempt


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", type=int, default=HEADLINE, help="workload of the headline line")
    ap.add_argument("--per-config", default=",".join(map(str, PER_CONFIG)),
                    help="comma-separated workloads measured into per_config ('' = none)")
    ap.add_argument("--seed", type=int, default=1000)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cluster-size", type=int, default=0)
    ap.add_argument("--sets", type=int, default=0, help="input sets to rotate (0 = auto)")
    ap.add_argument("--no-workspace", action="store_true",
                    help="pass no workspace (the cluster-per-row kernel)")
    ap.add_argument("--levels", type=int, default=3, help="cascade leg: levels incl. the target")
    ap.add_argument("--leg", default="verify", choices=["verify", "commit", "law", "sample", "cascade"],
                    help="commit: time the post-verify step (token bookkeeping and the "
                         "draft-length controller) on the workload's shape; law: time the "
                         "emitted-token law (scoring) over the workload's draft positions; "
                         "sample: the draft sampler over the workload's draft rows; cascade: "
                         "the multi-stage draft cascade with --levels levels")
    return ap.parse_args(argv)


def aggregate(total_ms: float, positions: float, world: int, dev=None):
    """Whole-job figures of weak-scaled replicas: every rank verified its own
    batches; the job took the slowest rank's time.  Returns (job time in ms,
    positions of all ranks, positions/s).  With world > 1 the process group
    must be initialised (NCCL on the GPU machine, gloo in the CPU tests)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        p = torch.tensor([float(positions)], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(p, op=dist.ReduceOp.SUM)
        total_ms, positions = float(t.item()), float(p.item())
    return total_ms, positions, positions / (total_ms * 1e-3)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# The sources each kernel is compiled from: its translation unit and the
# headers of the library that it includes.
KERNEL_SOURCES = {
    "strip_kernel": ("spec_strip.cu", "sv_core.cuh", "sv_common.cuh", "sv_strip.h"),
    "row_kernel": ("spec_row.cu", "sv_core.cuh", "sv_common.cuh", "sv_row.h"),
    "row_cta_kernel": ("spec_row.cu", "sv_core.cuh", "sv_common.cuh", "sv_row.h"),
    "verify_kernel": ("spec_verify.cu", "sv_core.cuh", "sv_common.cuh", "sv_row.h", "sv_strip.h",
                      "sv_verify.h"),
    "law_kernel": ("spec_law.cu", "sv_common.cuh"),
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the sources a kernel is built from (a profile taken on other
    sources no longer describes it)."""
    h = hashlib.sha256()
    cdir = os.path.join(ROOT, "speculative_decoding_verify_03_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        h.update(f.encode())
        h.update(open(os.path.join(cdir, f), "rb").read())
    return h.hexdigest()[:16]


def profile_summary(kernel: str, w: W.Workload) -> str:
    return os.path.join(PROFILES, f"{kernel}_{w.name}.txt")


def profiled_traffic(path: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel's current sources (else None)."""
    try:
        kv = {}
        for line in open(path):
            if ":" in line:
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("kernel_source_hash") != kernel_source_hash(kernel):
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def measured_peak():
    try:
        mp = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(mp["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def nominal_bytes(w: W.Workload, gam) -> int:
    """Both logit tensors read once over the valid positions:
    sum_b (2 gamma_b + 1) V s (greedy reads the target only)."""
    es = 4 if w.dtype == "f32" else 2
    g = np.full(w.B, w.gamma_max, np.int64) if gam is None else np.asarray(gam, np.int64)
    per = (g + 1) if w.temperature == 0.0 else (2 * g + 1)
    return int((per * w.V * es).sum())


def bytes_read(acc, gam, s, V, greedy):
    """Early-exit bytes of one call: the logit rows the method must read given
    where each row stopped (positions 0..accepted_len of the target; the draft
    rows of the tested positions)."""
    tgt_rows = acc + 1
    drf_rows = 0 if greedy else np.minimum(acc + 1, gam)
    return int(((tgt_rows + drf_rows) * V * s).sum())


# ------------------------------------------------------------ the oracle legs
def _oracle_tokens(w: W.Workload, b: dict, rows, threads: int):
    """Draft tokens of the given rows drawn by the oracle's sampler from the
    filtered draft law q, for the valid positions (i < gamma_b; 0 elsewhere)."""
    import oracle
    G = w.gamma_max
    gam = b["gamma_per_row"]
    tok = np.zeros((len(rows), G), np.int32)
    if G == 0:
        return tok
    d = b["draft"]
    sel = [(j, i) for j, r in enumerate(rows) for i in range(int(gam[r]) if gam is not None else G)]
    flat = np.empty((len(sel), w.V), d.dtype)
    uu = np.empty(len(sel), np.float32)
    for n, (j, i) in enumerate(sel):
        flat[n] = d[rows[j], i, : w.V]
        uu[n] = b["draft_uniforms"][rows[j], i]
    got = oracle.sample(flat, w.temperature, w.top_k, w.top_p, uu, threads=threads)
    for n, (j, i) in enumerate(sel):
        tok[j, i] = got[n]
    return tok


def _sub_batch(w: W.Workload, b: dict, rows):
    if len(rows) == b["target"].shape[0] and np.array_equal(rows, np.arange(len(rows))):
        return {"target": b["target"][:, :, : w.V], "draft": b["draft"][:, :, : w.V],
                "uniforms": b["uniforms"], "gamma_per_row": b["gamma_per_row"]}
    return {"target": b["target"][rows][:, :, : w.V], "draft": b["draft"][rows][:, :, : w.V],
            "uniforms": b["uniforms"][rows],
            "gamma_per_row": None if b["gamma_per_row"] is None else b["gamma_per_row"][rows]}


def _oracle_verify(w: W.Workload, sb: dict, tok, threads: int):
    import oracle
    return oracle.verify(sb["target"], sb["draft"], tok, sb["uniforms"], w.temperature, w.top_k,
                         w.top_p, gamma_per_row=sb["gamma_per_row"], threads=threads)


def parity_counts(o: dict, acc, nxt):
    """GPU/oracle agreement on the sampled rows: token ids and accepted
    lengths must match, except on rows whose oracle decision path passes
    within EPS_BOUNDARY of a decision boundary (acceptance ratio, CDF
    boundary, top-p mass).  Draws = acceptance tests + inverse-CDF draws."""
    d = o["diag"]
    near = ((d["accept_margin"] < EPS_BOUNDARY) | (d["cdf_margin"] < EPS_BOUNDARY) |
            (d["topp_margin"] < EPS_BOUNDARY))
    mism = (o["accepted_len"] != acc) | (o["next_token"] != nxt)
    draws = int(d["n_tests"].sum() + d["n_draws"].sum())
    return {"rows": int(len(acc)), "draws": draws, "near_boundary": int(near.sum()),
            "disagree": int(mism.sum()), "hard": int((mism & ~near).sum()),
            "disagree_frac": float(mism.sum()) / max(1, draws)}


def cpu_leg(w: W.Workload, host: dict, verify_fn, seed: int, max_rows: int = 512,
            budget_s: float = 1.5):
    """The oracle, as it stands, on a bounded sample of the first timed set's
    rows: draft tokens from the oracle's sampler, then the verify step timed
    on all host cores (repeated passes until ~budget_s of wall time) and on
    one thread (an eighth of the rows).  The GPU verifies the whole set with
    those tokens on the sampled rows (verify_fn(rows, tokens) -> (acc, nxt)
    of the sampled rows), and the two are compared (parity_counts)."""
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(seed)
    n = min(w.B, max_rows)
    rows = np.sort(rng.choice(w.B, size=n, replace=False)) if n < w.B else np.arange(w.B)
    tok = _oracle_tokens(w, host, rows, cores)
    sb = _sub_batch(w, host, rows)
    gam = sb["gamma_per_row"]
    pos = int(gam.sum()) if gam is not None else n * w.gamma_max
    passes, elapsed, o = 0, 0.0, None
    while passes == 0 or elapsed < budget_s:
        t0 = time.perf_counter()
        o = _oracle_verify(w, sb, tok, cores)
        elapsed += time.perf_counter() - t0
        passes += 1
    n1 = max(1, n // 8)
    sb1 = _sub_batch(w, host, rows[:n1])
    t0 = time.perf_counter()
    _oracle_verify(w, sb1, tok[:n1], 1)
    el1 = time.perf_counter() - t0
    pos1 = int(sb1["gamma_per_row"].sum()) if gam is not None else n1 * w.gamma_max
    acc, nxt = verify_fn(rows, tok)
    return ({"value": passes * pos / elapsed, "unit": UNIT, "cores": cores, "kind": "oracle",
             "value_1_thread": pos1 / el1,
             "sample": f"{n} rows of the first timed input set ({pos} draft positions), "
                       f"{passes} pass(es) on {cores} threads in {elapsed:.2f} s; one thread: "
                       f"{n1} rows in {el1:.2f} s"},
            parity_counts(o, acc, nxt))


def reference_arm(w: W.Workload, seed: int, steps: int, warmup: int):
    """--impl reference: the fp64 oracle on the host cores; each step verifies
    one row per host thread (a bounded sample of the workload's batch), with
    draft tokens from the oracle's own sampler."""
    cores = os.cpu_count() or 1
    n = min(w.B, 4 * cores)
    host = W.make_batch(w, seed, rows=np.arange(n))
    host["workload"] = w
    tok = _oracle_tokens(w, host, np.arange(n), cores)
    sb_all = _sub_batch(w, host, np.arange(n))

    def one(j):
        rows = (np.arange(cores) + j * cores) % n
        sb = {k: (v[rows] if v is not None else None) for k, v in sb_all.items()}
        _oracle_verify(w, sb, tok[rows], cores)
        g = sb["gamma_per_row"]
        return int(g.sum()) if g is not None else len(rows) * w.gamma_max

    for j in range(warmup):
        one(j)
    t0 = time.perf_counter()
    pos = sum(one(j) for j in range(steps))
    el = time.perf_counter() - t0
    v = pos / el
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1,
            "steps": steps, "warmup": warmup, "ms_per_step": el / max(1, steps) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "rows_per_step": cores},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{steps} steps of {cores} rows from a pool of {n} rows"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


class ClockSampler:
    def __init__(self, index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                       "-i", str(index), "-lms", "50"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        for line in self.f:
            c = [x.strip() for x in line.split(",")]
            if len(c) < 10:
                continue
            try:
                sm.append(float(c[2]))
                mx.append(float(c[3]))
            except ValueError:
                continue
            for name, col in (("hw_slowdown", 6), ("hw_thermal_slowdown", 7),
                              ("sw_thermal_slowdown", 8), ("sw_power_cap", 9)):
                if c[col].lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.f.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- other legs
def commit_leg(args, w, sv, torch, dev):
    """The post-verify step on the workload's shape: a CUDA graph of K calls
    (the sequences grow by at most gamma_max + 1 tokens a call; capacity for
    every call), events around the whole graph.  Bytes moved per call: the
    four int32 row inputs, the accepted drafts read, the tokens written and
    the three int32 row outputs (a few hundred bytes a row): launch-bound."""
    rng = np.random.default_rng(args.seed)
    B, gm = w.B, w.gamma_max
    K, Wm = args.steps, max(3, args.warmup)
    cap = (K + Wm + 2) * (gm + 1) + 8  # the warm-ups and one graph replay
    acc = torch.from_numpy(rng.integers(0, gm + 1, size=B).astype(np.int32)).to(dev)
    nxt = torch.from_numpy(rng.integers(0, w.V, size=B).astype(np.int32)).to(dev)
    tok = torch.from_numpy(rng.integers(0, w.V, size=(B, gm)).astype(np.int32)).to(dev)
    gam = torch.full((B,), gm, dtype=torch.int32, device=dev)
    seq = torch.zeros((B, cap), dtype=torch.int32, device=dev)
    slen = torch.zeros(B, dtype=torch.int32, device=dev)
    aimd = (1, gm, 1, 0.5)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for _ in range(Wm):
            sv.spec_commit(acc, nxt, tok, seq, slen, gamma_per_row=gam, aimd=aimd)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(K):
                sv.spec_commit(acc, nxt, tok, seq, slen, gamma_per_row=gam, aimd=aimd)
        slen.zero_()
        g.replay()  # warm replay
        slen.zero_()
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    a_h = acc.cpu().numpy().astype(np.int64)
    moved = B * 4 * 4 + int(a_h.sum()) * 4 + int((a_h + 1).sum()) * 4 + B * 3 * 4
    return {"leg": "commit", "metric": "committed rows/s", "value": B * K / (ms * 1e-3),
            "unit": "rows/s", "n_gpus": 1, "steps": K, "warmup": Wm,
            "ms_per_step": ms / K, "higher_is_better": True, "data": "synthetic",
            "config": {"workload": w.name, "B": B, "gamma": gm, "aimd": list(aimd),
                       "timing": "CUDA graph of K calls, events around the graph"},
            "bytes_per_step": moved, "gbs": moved / (ms / K * 1e-3) / 1e9,
            "bound": "launch", "gpu_launches": K}


def calls_launches(kernel: str) -> int:
    """Kernels one call launches on the path that runs `kernel`: the strip
    path a counter clear and the kernel; the row path with a workspace a
    counter clear, the row kernel and the second kernel for the rows it
    defers; the others one."""
    return {"strip_kernel": 2, "row_cta_kernel": 3}.get(kernel, 1)


def sample_leg(args, w, sv, torch, dev):
    """spec_sample (the draft model's per-step sampler) over the workload's
    draft rows: B * gamma_max rows of V with its temperature and filters, a
    uniform each; rotated input sets beyond L2, a CUDA graph of K calls,
    events around the graph.  Algorithmic bytes: each row read once."""
    rng = np.random.default_rng(args.seed)
    n, V = w.B * w.gamma_max, w.V
    es = 4 if w.dtype == "f32" else 2
    n_sets = max(3, int(np.ceil(3 * 136e6 / (n * V * es))))
    sets = []
    for k in range(n_sets):
        b = W.make_batch(w, args.seed + 29 * k)
        dr = np.ascontiguousarray(b["draft"][:, :, :V]).reshape(n, V)
        conv = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)) \
            if w.dtype == "bf16" else torch.from_numpy
        u = torch.from_numpy(rng.random(n, dtype=np.float32))
        sets.append((conv(dr).to(dev), u.to(dev)))
    K, Wm = args.steps, max(3, args.warmup)
    T, kw = w.temperature, dict(top_k=w.top_k, top_p=w.top_p)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for j in range(Wm):
            sv.spec_sample(*sets[j % n_sets], T, **kw)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(K):
                sv.spec_sample(*sets[j % n_sets], T, **kw)
        g.replay()
        stream.synchronize()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b_.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b_)
    peak, kind = measured_peak()
    achieved = n * V * es / (ms / K * 1e-3) / 1e9
    # the kernel the library selects with its cached workspace (a row is a
    # sequence with no drafts)
    filt = 0 < w.top_k < V or w.top_p < 1
    if V <= 1024 and (T == 0 or not filt):
        kernel = "row_kernel" if T == 0 else "row_cta_kernel"
    else:
        kernel = "strip_kernel" if (T == 0 or filt) else "verify_kernel"
    return {"leg": "sample", "metric": "sampled tokens/s", "value": n * K / (ms * 1e-3),
            "unit": "tokens/s", "n_gpus": 1, "steps": K, "warmup": Wm, "ms_per_step": ms / K,
            "higher_is_better": True, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "rows": n, "V": V, "temperature": T,
                       "top_k": w.top_k, "top_p": w.top_p, "l2": f"{n_sets} rotated input sets",
                       "timing": "CUDA graph of K calls, events around the graph"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": kind, "kernel": kernel,
                         "algorithmic_bytes_per_launch": n * V * es},
            "gpu_launches": K * calls_launches(kernel)}


def cascade_leg(args, w, sv, torch, dev):
    """spec_cascade_verify on the workload with args.levels levels (target,
    intermediate levels between target and draft, the draft): rotated input
    sets beyond L2, a CUDA graph of K calls, events around the graph.  The
    metric counts the drafted positions, sum gamma_b, as the verify line does;
    nominal bytes: every stage reading both its tensors once over the valid
    positions, (levels - 1) sum_b (2 gamma_b + 1) V s."""
    L = args.levels - 1
    es = 4 if w.dtype == "f32" else 2
    K, Wm = args.steps, max(3, args.warmup)
    sets, pos, nom = [], [], []
    per_set = (L + 1) * w.B * (w.gamma_max + 1) * (w.V + w.pos_pad) * es
    n_sets = max(2, int(np.ceil(3 * 136e6 / per_set)))
    for k in range(n_sets):
        b = W.make_batch(w, args.seed + 31 * k)
        c = W.cascade_levels(b, L + 1, args.seed + 31 * k + 1)

        def to_dev(a):
            if a.dtype == np.uint16:
                return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        lv = [to_dev(x)[:, :, : w.V] for x in c["levels"]]
        G = w.gamma_max
        du = torch.from_numpy(b["draft_uniforms"]).to(dev)
        tok = sv.spec_sample(lv[-1].reshape(-1, w.V), du.reshape(-1), w.temperature, w.top_k,
                             w.top_p).reshape(w.B, G).contiguous()
        gam = torch.from_numpy(b["gamma_per_row"]).to(dev) if b["gamma_per_row"] is not None else None
        gh = b["gamma_per_row"] if b["gamma_per_row"] is not None else np.full(w.B, G, np.int32)
        sets.append((lv, tok, torch.from_numpy(c["uniforms"]).to(dev), gam))
        pos.append(int(gh.sum()))
        nom.append(L * nominal_bytes(w, gh))
    P0 = sv.cascade_params(sets[0][0], w.temperature, w.top_k, w.top_p, sets[0][3])
    ws = torch.zeros(max(sv.cascade_workspace_bytes(P0, L + 1), 256), dtype=torch.uint8, device=dev)

    def step(j):
        lv, tok, uni, gam = sets[j % n_sets]
        sv.spec_cascade_verify(lv, tok, uni, w.temperature, w.top_k, w.top_p, gamma_per_row=gam,
                               workspace=ws)

    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for j in range(Wm):
            step(j)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(K):
                step(j)
        g.replay()
        stream.synchronize()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b_.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b_)
    peak, kind = measured_peak()
    positions = sum(pos[j % n_sets] for j in range(K))
    nominal = float(np.mean([nom[j % n_sets] for j in range(K)]))
    achieved = nominal / (ms / K * 1e-3) / 1e9
    kernel = kernel_name(sv, w, P0, ws.numel(), 0)
    return {"leg": "cascade", "metric": "verified draft positions/sec", "unit": "positions/s",
            "value": positions / (ms * 1e-3), "n_gpus": 1, "steps": K, "warmup": Wm,
            "ms_per_step": ms / K, "higher_is_better": True, "dtype": w.dtype,
            "data": "synthetic", "config": {"workload": w.name, "levels": L + 1,
                                            "l2": f"{n_sets} rotated input sets",
                                            "timing": "CUDA graph of K calls, events around the graph"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": kind,
                         "bytes": "nominal: each stage reads both its tensors once over the valid "
                                  "positions, (levels - 1) sum_b (2 gamma_b + 1) V s",
                         "nominal_bytes_per_launch": nominal, "kernel": kernel},
            # per call: the state's initialisation, then per stage the verify
            # step's launches and the update kernel
            "gpu_launches": K * (1 + L * (calls_launches(kernel) + 1))}


def law_leg(args, w, sv, torch, dev):
    """spec_law over the workload's draft positions (one row per position:
    B * gamma_max rows of V, with the workload's temperature and filters),
    the token of each row a draft token; rotated input sets beyond L2, a CUDA
    graph of K calls, events around the graph.  Algorithmic bytes: both rows
    read once."""
    rng = np.random.default_rng(args.seed)
    n, V = w.B * w.gamma_max, w.V
    es = 4 if w.dtype == "f32" else 2
    row_bytes = 2 * V * es
    n_sets = max(3, int(np.ceil(3 * 136e6 / (n * row_bytes))))
    sets = []
    for k in range(n_sets):
        b = W.make_batch(w, args.seed + 17 * k)
        tg = np.ascontiguousarray(b["target"][:, :-1, :V]).reshape(n, V)
        dr = np.ascontiguousarray(b["draft"][:, :, :V]).reshape(n, V)
        conv = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)) \
            if w.dtype == "bf16" else torch.from_numpy
        tok = torch.from_numpy(rng.integers(0, V, size=n).astype(np.int32))
        sets.append((conv(tg).to(dev), conv(dr).to(dev), tok.to(dev)))
    K, Wm = args.steps, max(3, args.warmup)
    T = w.temperature if w.temperature > 0 else 1.0
    # filtered laws run on the strip-parallel kernel with one workspace for
    # every call (two launches a call: its counter clear, the kernel)
    prm = sv.SpecParams(B=n, gamma_max=0, V=V, dtype=sv.SPEC_F32 if w.dtype == "f32" else sv.SPEC_BF16,
                        temperature=T, top_p=w.top_p, top_k=w.top_k, flags=0,
                        target_pos_stride=V, target_row_stride=V, draft_pos_stride=V,
                        draft_row_stride=V, gamma_per_row=None, cluster_size=0, list_capacity=0)
    ws_bytes = sv.law_workspace_bytes(prm)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    kernel = "strip_kernel (law)" if ws is not None else (
        "law_filt_kernel" if (0 < w.top_k < V or w.top_p < 1.0) else "law_kernel")
    kw = dict(top_k=w.top_k, top_p=w.top_p, workspace=ws)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for j in range(Wm):
            sv.spec_law(*sets[j % n_sets], T, **kw)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(K):
                sv.spec_law(*sets[j % n_sets], T, **kw)
        g.replay()
        stream.synchronize()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b_.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b_)
    peak, kind = measured_peak()
    achieved = n * row_bytes / (ms / K * 1e-3) / 1e9
    return {"leg": "law", "metric": "scored tokens/s", "value": n * K / (ms * 1e-3),
            "unit": "tokens/s", "n_gpus": 1, "steps": K, "warmup": Wm, "ms_per_step": ms / K,
            "higher_is_better": True, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "rows": n, "V": V, "temperature": T,
                       "top_k": w.top_k, "top_p": w.top_p,
                       "l2": f"{n_sets} rotated input sets",
                       "timing": "CUDA graph of K calls, events around the graph"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": kind, "kernel": kernel,
                         "algorithmic_bytes_per_launch": n * row_bytes},
            "gpu_launches": K * (2 if ws is not None else 1)}


# --------------------------------------------------------------- verify leg
def kernel_name(sv, w: W.Workload, prm, ws_bytes: int, cluster_size: int) -> str:
    """The kernel the library selects for this problem (the same rule as its
    dispatcher)."""
    k_on, p_on = 0 < w.top_k < w.V, w.top_p < 1.0
    if w.V <= 1024 and cluster_size == 0 and (w.temperature == 0 or not (k_on or p_on)):
        # sampling with the deferred-row list: a CTA per row, uncertain rows
        # to a second kernel; else a warp per row
        if w.temperature > 0 and ws_bytes >= sv.workspace_bytes(prm):
            return "row_cta_kernel"
        return "row_kernel"
    if ws_bytes > sv.workspace_bytes() and ws_bytes >= sv.workspace_bytes(prm):
        return "strip_kernel"
    return "verify_kernel"


def run_config(args, w: W.Workload, sv, torch, dev, rank: int, world: int) -> dict:
    """Time spec_verify on one workload; returns its line (without the
    top-level contract keys that only the headline carries)."""
    es = 4 if w.dtype == "f32" else 2
    greedy = w.temperature == 0.0
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    seed = args.seed + 1000 * w_id(w) + 7919 * rank

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def make_set(k, keep_host):
        b = W.make_batch(w, seed + k)
        b["workload"] = w
        tgt = to_dev(b["target"])[:, :, : w.V]
        drf = to_dev(b["draft"])[:, :, : w.V]
        uni = to_dev(b["uniforms"])
        gam = to_dev(b["gamma_per_row"]) if b["gamma_per_row"] is not None else None
        du = to_dev(b["draft_uniforms"])
        G = w.gamma_max
        flat = drf.reshape(-1, w.V) if G else None
        tok = (sv.spec_sample(flat, du.reshape(-1), w.temperature, w.top_k, w.top_p)
               .reshape(w.B, G) if G else torch.zeros((w.B, 0), dtype=torch.int32, device=dev))
        gh = b["gamma_per_row"] if b["gamma_per_row"] is not None else np.full(w.B, w.gamma_max,
                                                                                np.int32)
        return {"tgt": tgt, "drf": drf, "uni": uni, "gam": gam, "tok": tok.contiguous(),
                "gam_host": gh, "host": b if keep_host else None}

    alloc_per_set = (w.B * (2 * w.gamma_max + 1) * (w.V + w.pos_pad)) * es
    first = make_set(0, True)
    prm = sv.make_params(first["tgt"], first["drf"], w.temperature, w.top_k, w.top_p,
                         first["gam"], args.cluster_size)
    ws_bytes = sv.workspace_bytes(prm) if not args.no_workspace else 0
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev) if ws_bytes else None
    kernel = kernel_name(sv, w, prm, ws_bytes, args.cluster_size)
    acc0, _ = sv.spec_verify(first["tgt"], first["drf"], first["tok"], first["uni"],
                             w.temperature, w.top_k, w.top_p, gamma_per_row=first["gam"],
                             cluster_size=args.cluster_size, workspace=ws)
    torch.cuda.synchronize()
    read0 = bytes_read(acc0.cpu().numpy(), first["gam_host"], es, w.V, greedy)
    n_sets = args.sets or max(2, math.ceil(3 * l2 / max(1, min(read0, alloc_per_set))))
    n_sets = min(n_sets, max(2, int(0.25 * torch.cuda.mem_get_info(dev)[0] // alloc_per_set)))
    sets = [first] + [make_set(k, False) for k in range(1, n_sets)]
    outs = [(torch.empty(w.B, dtype=torch.int32, device=dev),
             torch.empty(w.B, dtype=torch.int32, device=dev)) for _ in range(n_sets)]

    def step(j):
        s = sets[j % n_sets]
        sv.spec_verify(s["tgt"], s["drf"], s["tok"], s["uni"], w.temperature, w.top_k, w.top_p,
                       gamma_per_row=s["gam"], cluster_size=args.cluster_size,
                       out=outs[j % n_sets], workspace=ws)

    # early-exit bytes per set (outputs are deterministic per set)
    for j in range(n_sets):
        step(j)
    torch.cuda.synchronize()
    read_per_set = [bytes_read(outs[j][0].cpu().numpy(), sets[j]["gam_host"], es, w.V, greedy)
                    for j in range(n_sets)]
    pos_per_set = [int(s["gam_host"].sum()) for s in sets]
    nom_per_set = [nominal_bytes(w, s["gam_host"]) for s in sets]

    stream = torch.cuda.Stream(dev)
    K, Wm = args.steps, max(3, args.warmup)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for j in range(Wm):
            step(j)
    stream.synchronize()

    # capture exactly K launches, each bracketed by timing events
    def timing_event():
        try:  # an event-record node when captured in a graph
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return torch.cuda.Event(enable_timing=True)

    ev = [(timing_event(), timing_event()) for _ in range(K)]
    graph = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for j in range(K):
                ev[j][0].record(stream)
                step(j)
                ev[j][1].record(stream)
    except Exception as e:  # fall back to eager launches
        print(f"[bench] graph capture failed ({e}); timing eager launches", file=sys.stderr)
        graph = None
    torch.cuda.synchronize()
    if graph is not None:  # warm replay
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(dev.index or 0)
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    if graph is not None:
        with torch.cuda.stream(stream):
            graph.replay()
    else:
        with torch.cuda.stream(stream):
            for j in range(K):
                ev[j][0].record(stream)
                step(j)
                ev[j][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.stop()
    total_ms = t0.elapsed_time(t1)
    try:
        launch_ms = np.array([a.elapsed_time(b) for a, b in ev])
        launch_timing = "CUDA events around each call (all of its launches)"
    except Exception:  # captured events not timeable: graph average (includes gaps)
        torch.cuda.synchronize()
        launch_ms = np.full(K, total_ms / K)
        launch_timing = "graph time / K (includes inter-launch gaps)"
    positions = sum(pos_per_set[j % n_sets] for j in range(K))
    total_ms, _, value = aggregate(total_ms, positions, world, dev)
    ee_bytes = float(np.mean([read_per_set[j % n_sets] for j in range(K)]))
    nominal = float(np.mean([nom_per_set[j % n_sets] for j in range(K)]))
    mean_launch_s = float(launch_ms.mean()) * 1e-3
    peak, peak_kind = measured_peak()
    traffic = profiled_traffic(profile_summary(kernel, w), kernel)
    launches_per_call = calls_launches(kernel)

    line = {
        "workload": w.name, "value": value, "unit": UNIT, "steps": K, "warmup": Wm,
        "ms_per_step": total_ms / K, "dtype": w.dtype,
        "config": {"workload": w.name, "B": w.B, "gamma": w.gamma_max, "V": w.V,
                   "ragged_gamma": w.ragged, "temperature": w.temperature, "top_k": w.top_k,
                   "top_p": w.top_p,
                   "l2": f"{n_sets} rotated input sets ({n_sets * alloc_per_set / 1e9:.2f} GB; "
                         f"{n_sets * float(np.mean(read_per_set)) / 1e6:.0f} MB read per "
                         f"rotation vs L2 {l2 / 1e6:.0f} MB)",
                   "timing": "CUDA graph of K launches, events per launch"},
        "roofline": {"bound": "hbm", "achieved": nominal / mean_launch_s / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": nominal / mean_launch_s / 1e9 / peak,
                     "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs (burst copy)",
                     "bytes": "nominal: both logit tensors read once over the valid positions, "
                              "sum_b (2 gamma_b + 1) V s",
                     "nominal_bytes_per_launch": nominal,
                     "early_exit_bytes_per_launch": ee_bytes,
                     "frac_early_exit": ee_bytes / mean_launch_s / 1e9 / peak,
                     "traffic_gbs": traffic / mean_launch_s / 1e9 if traffic else None,
                     "kernel": kernel, "kernel_us": mean_launch_s * 1e6,
                     "kernel_us_p10_p50_p90": [float(x) * 1e3 for x in
                                               np.percentile(launch_ms, [10, 50, 90])],
                     "kernel_timing": launch_timing},
        "gpu_launches": K * launches_per_call,
        "clocks": clocks,
    }

    # ---- end to end through the public API with host buffers
    if not args.no_e2e:
        line["e2e"] = e2e_leg(args, w, sv, torch, dev, sets, ws, stream, pos_per_set, world)

    # ---- the oracle: CPU baseline and parity counts on the first set
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = first["host"]

        def verify_rows(rows, tok_rows):
            tok = first["tok"].clone()
            tok[torch.from_numpy(rows).to(dev)] = torch.from_numpy(tok_rows).to(dev)
            acc, nxt = sv.spec_verify(first["tgt"], first["drf"], tok, first["uni"],
                                      w.temperature, w.top_k, w.top_p,
                                      gamma_per_row=first["gam"],
                                      cluster_size=args.cluster_size, workspace=ws)
            torch.cuda.synchronize()
            return acc.cpu().numpy()[rows], nxt.cpu().numpy()[rows]

        cb, par = cpu_leg(w, host, verify_rows, seed)
        line["cpu_baseline"] = cb
        line["parity"] = par
    first["host"] = None
    del sets, outs, ws, first
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


def w_id(w: W.Workload) -> int:
    for k, v in W.WORKLOADS.items():
        if v.name == w.name:
            return k
    return 0


def e2e_leg(args, w, sv, torch, dev, sets, ws, stream, pos_per_set, world):
    """The same metric through the public API with host buffers: every
    step's inputs are copied from pinned host memory (the padded tensors as
    the caller holds them), the outputs copied back, inside the timed
    region.  Two device input sets: the copies of step j + 1 (four copy
    streams, each logit tensor in two halves of rows) overlap the verify
    call of step j."""
    b = sets[0]["host"]
    h = {}
    for key, name in (("tgt", "target"), ("drf", "draft")):
        base = np.ascontiguousarray(b[name])  # padded tensor = the input
        h[key] = torch.from_numpy(base.view(np.int16) if base.dtype == np.uint16
                                  else base).pin_memory()
    h["tok"] = sets[0]["tok"].cpu().pin_memory()
    h["uni"] = sets[0]["uni"].cpu().pin_memory()
    hsets = [h]
    dbufs = []
    for _ in range(2):
        d = {}
        for key in ("tgt", "drf"):
            d[key] = torch.empty(hsets[0][key].shape, dtype=hsets[0][key].dtype, device=dev)
        d["tok"] = torch.empty_like(sets[0]["tok"])
        d["uni"] = torch.empty_like(sets[0]["uni"])
        dbufs.append(d)
    hacc = torch.empty(w.B, dtype=torch.int32).pin_memory()
    hnxt = torch.empty(w.B, dtype=torch.int32).pin_memory()
    dacc = torch.empty(w.B, dtype=torch.int32, device=dev)
    dnxt = torch.empty(w.B, dtype=torch.int32, device=dev)
    gam_dev = sets[0]["gam"]
    h2d = sum(hsets[0][k].numel() * hsets[0][k].element_size() for k in hsets[0])
    d2h = 2 * w.B * 4
    Ke = max(10, min(args.steps, 50))
    cs = [torch.cuda.Stream(dev) for _ in range(4)]
    done = [None, None]  # the verify call that last read each input set
    half = (w.B + 1) // 2

    def e2e_copy(j):
        h, d = hsets[j % len(hsets)], dbufs[j % 2]
        parts = [[("tok", slice(None))], [("uni", slice(None))], [], []]
        for n, key in enumerate(("tgt", "drf")):
            parts[2 * n].append((key, slice(0, half)))
            parts[2 * n + 1].append((key, slice(half, None)))
        ev = []
        for c, items in zip(cs, parts):
            if done[j % 2] is not None:
                c.wait_event(done[j % 2])
            with torch.cuda.stream(c):
                for key, sl in items:
                    d[key][sl].copy_(h[key][sl], non_blocking=True)
                e = torch.cuda.Event()
                e.record(c)
                ev.append(e)
        return ev

    def e2e_run(j, ev):
        d = dbufs[j % 2]
        for e in ev:
            stream.wait_event(e)
        with torch.cuda.stream(stream):
            tg = d["tgt"].view(torch.bfloat16) if w.dtype == "bf16" else d["tgt"]
            dr = d["drf"].view(torch.bfloat16) if w.dtype == "bf16" else d["drf"]
            sv.spec_verify(tg[:, :, : w.V], dr[:, :, : w.V], d["tok"], d["uni"],
                           w.temperature, w.top_k, w.top_p, gamma_per_row=gam_dev,
                           cluster_size=args.cluster_size, out=(dacc, dnxt), workspace=ws)
            hacc.copy_(dacc, non_blocking=True)
            hnxt.copy_(dnxt, non_blocking=True)
            e = torch.cuda.Event()
            e.record(stream)
            done[j % 2] = e

    def e2e_steps(n):
        ev = e2e_copy(0)
        for j in range(n):
            nxt = e2e_copy(j + 1) if j + 1 < n else None
            e2e_run(j, ev)
            ev = nxt

    e2e_steps(3)
    torch.cuda.synchronize()
    a, bb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for c in cs:
        c.wait_stream(stream)
    a.record(cs[0])
    for c in cs[1:] + [stream]:
        c.wait_event(a)
    e2e_steps(Ke)
    for c in cs:
        stream.wait_stream(c)
    bb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(bb)
    e2e_pos = sum(pos_per_set[j % len(hsets)] for j in range(Ke))
    _, _, e2e_value = aggregate(e2e_ms, e2e_pos, world, dev)
    del dbufs, hsets
    return {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": Ke,
            "h2d_gbs": h2d * Ke / (e2e_ms * 1e-3) / 1e9}


def main(argv=None):
    args = parse(argv)
    rank, world, local = dist_env()
    w = W.WORKLOADS[args.config]
    if args.impl == "reference":
        if rank != 0:
            return
        line = reference_arm(w, args.seed, args.steps, args.warmup)
        line["n_gpus"] = args.gpus
        print(json.dumps(line))
        return

    import torch
    import speculative_decoding_verify_03_gb300 as sv

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    sv.build() if rank == 0 or world == 1 else None
    if args.leg in ("commit", "law", "sample", "cascade"):
        if rank == 0:
            fn = {"commit": commit_leg, "law": law_leg, "sample": sample_leg,
                  "cascade": cascade_leg}[args.leg]
            print(json.dumps(fn(args, w, sv, torch, dev)))
        return
    if world > 1:
        torch.distributed.barrier()
    sv.lib()

    head = run_config(args, w, sv, torch, dev, rank, world)
    others = [int(x) for x in args.per_config.split(",") if x.strip() != ""]
    per = {}
    for c in others:
        if c == args.config:
            continue
        per[W.WORKLOADS[c].name] = run_config(args, W.WORKLOADS[c], sv, torch, dev, rank, world)

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
            "steps": head["steps"], "warmup": head["warmup"], "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": head["dtype"], "data": "synthetic (seeded)",
            "config": dict(head["config"],
                           parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
            "roofline": head["roofline"],
            "gpu_launches": head["gpu_launches"],
            "clocks": head["clocks"],
            "e2e": head.get("e2e"),
            "cpu_baseline": head.get("cpu_baseline"),
            "parity": head.get("parity"),
            "per_config": per,
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
