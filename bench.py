#!/usr/bin/env python3
"""Indexer hot-path benchmark (one JSON line on rank 0).

Default workload: the large prefill -- 2 sequences of 32768 query rows from start_pos 0
(8192 compressed positions each at ratio 4), 64 fp4 index heads, top-2048, offset 8192,
5 % of the rows with head weights x8. One step is the whole hot path for that batch:
publish the keys of the step's groups, then query prep + scores + causal mask + top-k
(indexer_forward_publish). The decode, prefill, two-level decode and tiny prefill
workloads are measured in the same run and reported under "per_config".

  value        queries/s over all ranks, inputs resident in HBM, CUDA-graph
               replay of the steps, CUDA events on the launching stream.
               Inputs larger than L2 (1.07 GB of q per step) or rotating copies.
  e2e          the same metric through the public C-ABI call with pinned HOST
               buffers: per step the inputs host->device, the call, the top-k
               device->host, all inside the timed region.
  roofline     the dominant kernel (scores): algorithmic flops (or bytes) per
               launch / its average duration, from CUDA events around a graph
               of back-to-back launches of that kernel alone (its own entry
               point), against the measured peak in MEASURED_PEAKS.json.
  step_roofline the whole step against the same peak (the step's algorithmic
               work / the step's time).
  cpu_baseline the CPU oracle, as it stands, on a bounded sample of the same
               workload, one process per host core (rank 0, N=1).

--impl reference times that oracle as the reference arm.
Multi-GPU (torchrun): every rank runs its own replica of the workload (the path
shards by sequence and query row, no data-path collective); the time is the max
over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import MIXED, ROPE, WORKLOADS, MixedBatch, Workload, normal_bf16  # noqa: E402

METRIC = "indexer score+top-k queries/s and key-scores/s; % of HBM / FP4-MMA roofline"
UNIT = "queries/s"
FP4_OVER_BF16 = 13.5 / 2.25          # nominal dense fp4 / bf16 tensor ratio of the part
FP8_OVER_BF16 = 4.5 / 2.25           # nominal dense fp8 / bf16 tensor ratio of the part


def fmt_of(wl) -> dict:
    """Row format of a workload: MXFP4 (68-byte rows) or FP8 (132-byte rows)."""
    if getattr(wl, "key_format", 0) == 1:
        return {"name": "fp8", "row": 132, "dtype": "e4m3 x e4m3 -> f32", "ratio": FP8_OVER_BF16, "label": "fp8"}
    return {"name": "mxfp4", "row": 68, "dtype": "e2m1 x e2m1 -> f32", "ratio": FP4_OVER_BF16, "label": "fp4"}
ROTATE = 16


HEADLINE = "large_prefill"
# timed steps of each workload when --steps is not given (each run a fraction of a second)
DEFAULT_STEPS = {"large_prefill": 40, "prefill": 400, "prefill_fp8": 400, "prefill_qproj": 200, "decode": 5000,
                 "decode_fp8": 5000, "two_level_decode": 2000, "tiny_prefill": 5000}
# the other configurations, measured in the same run as the headline and reported under per_config
PER_CONFIG = ("tiny_prefill", "decode", "prefill", "two_level_decode")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=None)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS) + sorted(MIXED))
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle sample budget for cpu_baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-config", action="store_true", help="skip the other configurations' sub-records")
    p.add_argument("--profile-kernel", default=None, choices=["publish", "prep_q", "scores", "topk", "candidates"],
                   help="run the workload's kernels once through the split entry points, then this kernel three "
                        "times, and exit (a short, small-footprint command for ncu captures)")
    p.add_argument("--batch", type=int, default=None,
                   help="override the workload's batch (a smaller case of the same kernels, for ncu captures)")
    a = p.parse_args()
    if a.steps is None:
        a.steps = DEFAULT_STEPS.get(a.workload, 1000)
    if a.warmup is None:
        a.warmup = max(3, a.steps // 10)
    return a


# ----------------------------------------------------------------------------- distributed
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            if torch.cuda.is_available():
                self.pg.barrier(device_ids=[self.local])
            else:
                self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (50 ms) of SM clock and throttle reasons around the timed region."""
    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.uuid = str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            self.uuid = ""
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = self.t1 = None

    def region(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = []
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, parts))
            except Exception:
                continue
        os.unlink(self.file.name)
        if self.uuid:
            mine = [r for r in rows if self.uuid in r[1][1]]
            rows = mine or rows
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.05 <= r[0] <= self.t1 + 0.05]
        window = "timed" if inside else "warmup+timed"
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1][2]) for r in use if r[1][2].replace(".", "").isdigit()]
        smax = [float(r[1][3]) for r in use if r[1][3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[1][6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(use), "window": window}


# ----------------------------------------------------------------------------- roofline inputs
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def profile_traffic(kernel_tag: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the kernel
    source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(path):
        return None
    src = open(os.path.join(ROOT, "sparse_attention_top_indexer_gb300", "csrc", "kernel_score.cu"), "rb").read()
    digest = hashlib.sha256(src).hexdigest()[:16]
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != digest:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------------------- our arm
class Setup:
    """Device tensors of one workload: RoPE table, weights, rotating caches and inputs."""

    def __init__(self, wl: Workload, dev, rotate: int):
        import sparse_attention_top_indexer_gb300 as X
        self.X = X
        self.wl = wl
        self.dev = dev
        X.load_library()
        self.dims = X.make_dims(n_heads=wl.H, ratio=wl.ratio, index_topk=wl.topk, offset=wl.offset,
                                rope_dim=wl.rope_dim, head_dim=wl.D, cand_topk_blocks=wl.cand_topk_blocks,
                                cand_block_size=wl.cand_block_size, norm_eps=wl.norm_eps, key_format=wl.key_format)
        self.table = torch.empty((wl.max_pos, wl.rope_dim // 2, 2), dtype=torch.float32, device=dev)
        X.indexer_rope_table(X.IndexerYarn(ROPE.theta, ROPE.factor, ROPE.original_seq_len, ROPE.beta_fast,
                                           ROPE.beta_slow), wl.rope_dim, wl.max_pos, self.table)
        self.wk, self.knw = wl.wk(dev), wl.k_norm_w(dev)
        self.decode = wl.S == 1 and wl.start_pos > 0
        self.rotate = rotate
        if self.decode:
            base = X.new_key_cache(wl.B, wl.T_cap, device=dev, key_format=wl.key_format)
            X.indexer_publish_k(self.dims, wl.latent(dev), self.wk, self.knw, self.table, 0, base)
            self.caches = [base] + [base.clone() for _ in range(rotate - 1)]
            self.lat = [normal_bf16(wl.seed, f"{wl.name}/latent_step/{i}", (wl.B, 1, wl.D), device=dev)
                        for i in range(rotate)]
        else:
            self.caches = [X.new_key_cache(wl.B, wl.T_cap, device=dev, key_format=wl.key_format)
                           for _ in range(rotate)]
            self.lat = [normal_bf16(wl.seed, f"{wl.name}/latent/{i}", (wl.B, wl.T, wl.D), device=dev)
                        for i in range(rotate)]
        tags = ["q1", "q2"] if wl.two_level else ["q"]
        self.q = {t: [normal_bf16(wl.seed, f"{wl.name}/{t}/{i}", (wl.B, wl.S, wl.H, wl.D), device=dev)
                      for i in range(rotate)] for t in tags}
        self.w = {t: [normal_bf16(wl.seed, f"{wl.name}/w{t[1:]}/{i}", (wl.B, wl.S, wl.H), device=dev)
                      for i in range(rotate)] for t in tags}
        if wl.fused_q:   # the query latent and wq_b in place of q
            self.qr = [wl.qr(dev, tag=f"qr/{i}") for i in range(rotate)]
            self.wq = wl.wq_b(dev)
        self.ws_bytes = X.indexer_workspace_size(self.dims, wl.B, wl.S, wl.start_pos)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        X.indexer_workspace_init(self.ws)
        self.top = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device=dev)
        self.top1 = torch.empty_like(self.top)
        self.cand = (torch.empty((wl.B, wl.S, wl.cand_topk_blocks), dtype=torch.int32, device=dev)
                     if wl.two_level else None)
        # split-entry buffers for the per-kernel breakdown
        self.q_rows = torch.empty((wl.B, wl.S, wl.H, X.row_bytes(wl.key_format)), dtype=torch.uint8, device=dev)
        self.w_prime = torch.empty((wl.B, wl.S, wl.H), dtype=torch.float32, device=dev)
        self.scores = torch.empty((wl.B, wl.S, wl.T), dtype=torch.float32, device=dev)

    def publish(self, i):
        wl = self.wl
        self.X.indexer_publish_k(self.dims, self.lat[i], self.wk, self.knw, self.table,
                                 wl.start_pos if self.decode else 0, self.caches[i])

    def step(self, i):
        """One pass of the whole hot path over batch i: the step's key publish and the forward
        in one call (indexer_forward_publish); a two-level step's consumer layer follows."""
        X, wl = self.X, self.wl
        sp = wl.start_pos if self.decode else 0
        if wl.fused_q:   # key publish, the fused query projection + prep, scores, top-k
            X.indexer_publish_k(self.dims, self.lat[i], self.wk, self.knw, self.table, sp, self.caches[i])
            X.indexer_prep_q_proj(self.dims, self.qr[i], self.wq, self.w["q"][i], wl.start_pos, self.table,
                                  self.q_rows, self.w_prime, self.ws)
            X.indexer_scores(self.dims, self.q_rows, self.w_prime, wl.start_pos, self.caches[i], self.scores, self.ws)
            X.indexer_topk(self.dims, self.scores, wl.start_pos, self.top)
            return
        if wl.two_level:
            X.indexer_forward_publish(self.dims, self.lat[i], self.wk, self.knw, self.q["q1"][i], self.w["q1"][i], sp,
                                      self.table, self.caches[i], self.top1, self.ws, cand_out=self.cand)
            X.indexer_forward(self.dims, self.q["q2"][i], self.w["q2"][i], wl.start_pos, self.table, self.caches[i],
                              self.top, self.ws, cand_in=self.cand)
        else:
            X.indexer_forward_publish(self.dims, self.lat[i], self.wk, self.knw, self.q["q"][i], self.w["q"][i], sp,
                                      self.table, self.caches[i], self.top, self.ws)

    def launches_per_step(self) -> int:
        # decode: publish + query prep in one launch, scores, top-k (level one: candidate
        # blocks and top-k in one launch); prefill: separate publish and query prep launches;
        # a two-level step's consumer layer: query prep, scores, top-k
        small = self.decode and self.wl.B * self.wl.S * self.wl.H <= 16384
        if self.wl.fused_q:
            return 4
        return (3 if small else 4) + (3 if self.wl.two_level else 0)

    def kernel_kinds(self):
        """One launch of each kernel of the step through its own entry point, on batch i."""
        X, wl = self.X, self.wl
        tag = "q2" if wl.two_level else "q"
        kinds = {
            "publish": lambda i: self.publish(i),
            "prep_q": lambda i: X.indexer_prep_q(self.dims, self.q[tag][i], self.w[tag][i], wl.start_pos, self.table,
                                                 self.q_rows, self.w_prime),
            "scores": lambda i: X.indexer_scores(self.dims, self.q_rows, self.w_prime, wl.start_pos, self.caches[i],
                                                 self.scores, self.ws),
            "topk": lambda i: X.indexer_topk(self.dims, self.scores, wl.start_pos, self.top),
        }
        if wl.two_level:
            kinds["candidates"] = lambda i: X.indexer_select_candidate_blocks(self.dims, self.scores, wl.start_pos,
                                                                              self.cand)
        if wl.fused_q:
            kinds["prep_q_proj"] = lambda i: X.indexer_prep_q_proj(self.dims, self.qr[i], self.wq, self.w[tag][i],
                                                                   wl.start_pos, self.table, self.q_rows,
                                                                   self.w_prime, self.ws)
        return kinds


def visible_pairs(wl: Workload) -> int:
    vis = [min(wl.T, (wl.start_pos + s + 1) // wl.ratio) for s in range(wl.S)]
    return wl.B * int(sum(vis))


def score_units(wl: Workload):
    """Algorithmic work of one scores launch: HBM bytes and tensor flops."""
    pairs = visible_pairs(wl)
    rb = 132 if wl.key_format == 1 else 68   # bytes per key / query-head row
    # every key of a sequence is read once (prefill: they stay in L2 across query groups)
    key_bytes = wl.B * wl.T * rb
    q_bytes = wl.B * wl.S * wl.H * (rb + 4)
    out_bytes = pairs * 4
    flops = pairs * wl.H * wl.D * 2
    return {"bytes": key_bytes + q_bytes + out_bytes, "flops": flops, "pairs": pairs}


def capture(fn, n: int):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            fn(i)
    return g


def step_units(wl: Workload):
    """Algorithmic work of one whole step (key publish, query prep, scores, top-k): HBM bytes
    (keys read once, bf16 q and w in, the step's latents in, indices out) and tensor flops."""
    u = score_units(wl)
    rb = fmt_of(wl)["row"]
    keys_pub = wl.B * (1 if (wl.S == 1 and wl.start_pos > 0) else wl.T)
    nvec = wl.B * wl.S * wl.H
    by = (wl.B * wl.T * rb + keys_pub * (wl.D * 2 + rb) + nvec * (wl.D * 2 + 2) + wl.B * wl.S * wl.topk * 4)
    return {"bytes": by, "flops": u["flops"], "pairs": u["pairs"]}


def run_ours(args, dist: Dist, name=None, steps=None, warmup=None, with_e2e=True):
    name = name or args.workload
    steps = steps or args.steps
    warmup = args.warmup if warmup is None else warmup
    wl = WORKLOADS[name]
    if args.batch and name == args.workload:
        wl = dataclasses.replace(wl, B=args.batch)
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    big_inputs = wl.B * wl.S * wl.H * wl.D * 2 > 256 * 1024 * 1024
    rotate = 1 if big_inputs else ROTATE
    st = Setup(wl, dev, rotate)
    for i in range(rotate):            # eager warm-up (also sets the kernels' attributes)
        st.step(i)
    torch.cuda.synchronize()
    X = st.X
    X.indexer_status(st.ws)

    # graphs of `rotate` steps (+ remainders) replayed for the warm-up and the timed region
    g_full = capture(st.step, rotate)
    rem = steps % rotate
    g_rem = capture(st.step, rem) if rem else None
    n_full = steps // rotate
    for _ in range(max(1, math.ceil(warmup / rotate))):
        g_full.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(dist.local)
    time.sleep(0.15)
    dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    e0.record()
    for _ in range(n_full):
        g_full.replay()
    if g_rem is not None:
        g_rem.replay()
    e1.record()
    torch.cuda.synchronize()
    w1 = time.time()
    dist.barrier()
    sampler.region(w0, w1)
    time.sleep(0.1)
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1)
    ms_max = dist.max(ms)
    X.indexer_status(st.ws)
    del g_full, g_rem

    queries = dist.world * wl.B * wl.S * steps
    value = queries / (ms_max / 1e3)
    units = score_units(wl)
    key_scores = dist.world * units["pairs"] * steps / (ms_max / 1e3)

    # per-kernel breakdown (split entry points, events between kernels, graph replay)
    kernel_ms = breakdown(st, rotate)

    # end to end through the public API with pinned host buffers
    e2e = run_e2e(st, steps, dist) if with_e2e else None

    peaks = measured_peaks()
    score_ms = kernel_ms.get("scores")
    fm = fmt_of(wl)
    step_ms = ms_max / steps
    su = step_units(wl)
    if wl.S == 1:
        achieved = units["bytes"] / (score_ms / 1e3) / 1e9 if score_ms else None
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak if achieved else None,
                "traffic": profile_traffic(f"scores_{wl.name}"),
                "algorithmic_bytes_per_launch": units["bytes"], "kernel": f"score_kernel<{wl.H},1,1,{fm['name']}>",
                "kernel_ms": score_ms, "peak_source": f"{peaks['source']} hbm_gbs"}
        sa = su["bytes"] / (step_ms / 1e3) / 1e9
        step_roof = {"bound": "hbm", "achieved": sa, "peak": peak, "unit": "GB/s", "frac": sa / peak,
                     "algorithmic_bytes_per_step": su["bytes"], "step_ms": step_ms}
        st_ms = (kernel_ms.get("scores") or 0) + (kernel_ms.get("topk") or 0)
        if st_ms:   # scoring + top-k, the two kernels the decode target names
            step_roof["scores_topk"] = {"ms": st_ms, "achieved": units["bytes"] / (st_ms / 1e3) / 1e9,
                                        "frac": units["bytes"] / (st_ms / 1e3) / 1e9 / peak}
    else:
        achieved = units["flops"] / (score_ms / 1e3) / 1e12 if score_ms else None
        peak = peaks["bf16_tflops"] * fm["ratio"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak if achieved else None,
                "traffic": profile_traffic(f"scores_{wl.name}"),
                "algorithmic_flops_per_launch": units["flops"], "kernel": "score_rows_kernel",
                "kernel_ms": score_ms,
                "peak_source": f"{peaks['source']} bf16_tflops x {fm['ratio']:g} (nominal {fm['label']}/bf16)"}
        sa = su["flops"] / (step_ms / 1e3) / 1e12
        step_roof = {"bound": "tensor", "achieved": sa, "peak": peak, "unit": "TFLOP/s", "frac": sa / peak,
                     "algorithmic_flops_per_step": su["flops"], "step_ms": step_ms}

    # the HBM-bound helper kernels against the same peak: algorithmic bytes per launch
    rb = fm["row"]
    nvec = wl.B * wl.S * wl.H
    keys = wl.B * (1 if st.decode else wl.T)
    helper_bytes = {"prep_q": nvec * (wl.D * 2 + 2 + rb + 4),
                    "publish": keys * (wl.D * 2 + rb) + wl.D * wl.D * 2 + wl.D * 2,
                    "topk": units["pairs"] * 4 + wl.B * wl.S * wl.topk * 4}
    helpers = {k: {"bytes": b, "GB/s": b / (kernel_ms[k] / 1e3) / 1e9,
                   "frac": b / (kernel_ms[k] / 1e3) / 1e9 / peaks["hbm_gbs"]}
               for k, b in helper_bytes.items() if kernel_ms.get(k)}
    if kernel_ms.get("prep_q_proj"):   # the bf16 projection on the tensor cores
        pf = 2.0 * wl.B * wl.S * wl.q_lora_rank * wl.H * wl.D
        pa = pf / (kernel_ms["prep_q_proj"] / 1e3) / 1e12
        helpers["prep_q_proj"] = {"flops": pf, "TFLOP/s": pa, "frac": pa / peaks["bf16_tflops"],
                                  "peak_source": f"{peaks['source']} bf16_tflops"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": steps,
        "warmup": warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": fm["dtype"], "data": "synthetic",
        "config": {"workload": describe(wl), "B": wl.B, "S": wl.S, "start_pos": wl.start_pos, "T": wl.T,
                   "H": wl.H, "topk": wl.topk, "ratio": wl.ratio,
                   "l2": (f"{rotate} rotating key caches / inputs "
                          f"({rotate * wl.B * wl.T_cap * rb / 1e6:.0f} MB of keys)"
                          if rotate > 1 else
                          f"inputs larger than L2 ({wl.B * wl.S * wl.H * wl.D * 2 / 1e9:.2f} GB of q per step)"),
                   "timing": "CUDA-graph replay, CUDA events on the launching stream"},
        "key_scores_per_s": key_scores,
        "kernel_ms": kernel_ms,
        "roofline": roof,
        "step_roofline": step_roof,
        "helper_rooflines": helpers,
        "e2e": e2e,
        "gpu_launches": st.launches_per_step() * steps,
        "clocks": clocks,
    }
    del st
    torch.cuda.empty_cache()
    return line, wl


def measure_producers(wl: Workload, dev, reps: int = 3) -> dict:
    """The upstream producers on the workload's tokens (indexer_compress_weights: the
    Compressor's latent and its fp4/e4m3 copy, and weights_proj, from hidden states of size
    wl.dim): CUDA-event time of a graph of back-to-back launches, against the larger of the
    HBM time of its algorithmic bytes and the bf16 tensor time of its flops."""
    import sparse_attention_top_indexer_gb300 as X
    d = X.make_dims(n_heads=wl.H, ratio=wl.ratio, index_topk=wl.topk, norm_eps=wl.norm_eps)
    x = wl.x(dev)
    wkv, wg, nw, wp = wl.wkv(dev), wl.wgate(dev), wl.c_norm_w(dev), wl.wproj(dev)
    G = wl.S // wl.ratio
    lat = torch.empty((wl.B, G, wl.D), dtype=torch.bfloat16, device=dev)
    latq = torch.empty_like(lat)
    w = torch.empty((wl.B, wl.S, wl.H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(X.STATUS_BYTES, dtype=torch.uint8, device=dev)
    X.indexer_workspace_init(ws)
    fn = lambda i: X.indexer_compress_weights(d, x, wkv, wg, nw, wp, lat, w, ws, latent_q=latq)
    fn(0)
    torch.cuda.synchronize()
    g = capture(fn, reps)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    X.indexer_status(ws)
    ms = e0.elapsed_time(e1) / (reps * reps)
    R = wl.B * wl.S
    n_out = 2 * wl.D + wl.H
    flops = 2.0 * R * wl.dim * n_out
    byts = R * wl.dim * 2 + n_out * wl.dim * 2 + 2 * R // wl.ratio * wl.D * 2 + R * wl.H * 2
    peaks = measured_peaks()
    t_hbm = byts / (peaks["hbm_gbs"] * 1e9) * 1e3
    t_mma = flops / (peaks["bf16_tflops"] * 1e12) * 1e3
    del x, g
    torch.cuda.empty_cache()
    return {"kernel": "compress_kernel (indexer_compress_weights)", "ms": ms, "rows": R, "dim": wl.dim,
            "outputs_per_row": n_out, "flops": flops, "bytes": byts, "TFLOP/s": flops / (ms / 1e3) / 1e12,
            "GB/s": byts / (ms / 1e3) / 1e9, "bound": "hbm" if t_hbm >= t_mma else "tensor",
            "frac": max(t_hbm, t_mma) / ms,
            "peak_source": f"{peaks['source']} hbm_gbs and bf16_tflops (the larger of the two times)"}


def per_config_records(args, dist: Dist) -> dict:
    """The other configurations, measured in the same run: value, step time, kernel times,
    the dominant kernel's roofline and the whole step's, and e2e through the host-buffer call."""
    out = {}
    for name in PER_CONFIG:
        if name == args.workload:
            continue
        steps = DEFAULT_STEPS[name]
        line, _ = run_ours(args, dist, name=name, steps=steps, warmup=max(3, steps // 10))
        out[name] = {k: line[k] for k in ("value", "unit", "ms_per_step", "steps", "warmup", "key_scores_per_s",
                                          "kernel_ms", "roofline", "step_roofline", "e2e", "gpu_launches",
                                          "clocks")}
        out[name]["workload"] = line["config"]["workload"]
        out[name]["l2"] = line["config"]["l2"]
    return out


# ----------------------------------------------------------------------------- mixed batches
class MixedSetup:
    """A server step over a page pool: every sequence's keys before this step are
    published once; a step publishes the keys its rows complete (slot mapping) and runs
    indexer_forward_paged over the whole batch. `rotate` pool copies and inputs."""

    def __init__(self, m: MixedBatch, dev, rotate: int):
        import sparse_attention_top_indexer_gb300 as X
        self.X, self.m, self.dev, self.rotate = X, m, dev, rotate
        X.load_library()
        self.dims = X.make_dims(n_heads=m.H, ratio=m.ratio, index_topk=m.topk, offset=m.offset,
                                rope_dim=m.rope_dim, head_dim=m.D, cand_topk_blocks=m.cand_topk_blocks,
                                cand_block_size=m.cand_block_size, norm_eps=m.norm_eps)
        self.table = torch.empty((m.max_pos, m.rope_dim // 2, 2), dtype=torch.float32, device=dev)
        X.indexer_rope_table(X.IndexerYarn(ROPE.theta, ROPE.factor, ROPE.original_seq_len, ROPE.beta_fast,
                                           ROPE.beta_slow), m.rope_dim, m.max_pos, self.table)
        self.wk, self.knw = m.wk(dev), m.k_norm_w(dev)
        bt = m.block_table()
        self.bt = bt.to(dev)
        # keys before the step (published once) and the keys the step's rows complete
        old_pos, old_slot, new_pos, new_slot = [], [], [], []
        for b, (sp, S) in enumerate(m.seqs):
            t_old, t_new = sp // m.ratio, m.T_list[b]
            for lo, hi, pos, slot in ((0, t_old, old_pos, old_slot), (t_old, t_new, new_pos, new_slot)):
                j = torch.arange(lo, hi)
                pos.append(j * m.ratio)
                slot.append(bt[b, j // 64].long() * 64 + j % 64)
        i32 = lambda xs: torch.cat(xs).to(torch.int32).to(dev)
        self.old_pos, self.old_slot = i32(old_pos), i32(old_slot)
        self.new_pos, self.new_slot = i32(new_pos), i32(new_slot)
        self.n_new = int(self.new_pos.numel())
        self.status = torch.empty(X.STATUS_BYTES, dtype=torch.uint8, device=dev)
        X.indexer_workspace_init(self.status)
        base = X.new_key_pool(m.num_pages, device=dev)
        n_old = int(self.old_pos.numel())
        lat_old = normal_bf16(m.seed, f"{m.name}/latent_old", (n_old, m.D), device=dev)
        X.indexer_publish_k_paged(self.dims, lat_old, self.wk, self.knw, self.table, self.old_pos, self.old_slot,
                                  base, self.status)
        self.pools = [base] + [base.clone() for _ in range(rotate - 1)]
        self.lat = [normal_bf16(m.seed, f"{m.name}/latent_new/{i}", (self.n_new, m.D), device=dev)
                    for i in range(rotate)]
        self.q = [normal_bf16(m.seed, f"{m.name}/q/{i}", (m.Q, m.H, m.D), device=dev) for i in range(rotate)]
        self.w = [normal_bf16(m.seed, f"{m.name}/w/{i}", (m.Q, m.H), device=dev) for i in range(rotate)]
        self.seq_pos = torch.tensor([sp for sp, _ in m.seqs], dtype=torch.int32, device=dev)
        self.q_start = torch.tensor(m.q_start, dtype=torch.int32, device=dev)
        self.ws = torch.empty(X.indexer_workspace_size_paged(self.dims, m.Q, m.n_seq, m.T_max), dtype=torch.uint8,
                              device=dev)
        X.indexer_workspace_init(self.ws)
        self.top = torch.empty((m.Q, m.topk), dtype=torch.int32, device=dev)

    def publish(self, i):
        self.X.indexer_publish_k_paged(self.dims, self.lat[i], self.wk, self.knw, self.table, self.new_pos,
                                       self.new_slot, self.pools[i], self.status)

    def forward(self, i):
        m = self.m
        self.X.indexer_forward_paged(self.dims, self.q[i], self.w[i], self.seq_pos, self.q_start, m.T_max,
                                     self.table, self.pools[i], self.bt, self.top, self.ws)

    def step(self, i):
        self.publish(i)
        self.forward(i)


def mixed_units(m: MixedBatch):
    """Algorithmic work of one forward over the batch: every key of a sequence read once,
    query rows in, indices out; tensor flops of every visible (row, key) pair."""
    pairs = 0
    for (sp, S), T in zip(m.seqs, m.T_list):
        pairs += sum(min(T, (sp + s + 1) // m.ratio) for s in range(S))
    key_bytes = sum(m.T_list) * 68
    q_bytes = m.Q * m.H * (m.D * 2 + 2)
    out_bytes = m.Q * m.topk * 4
    return {"bytes": key_bytes + q_bytes + out_bytes, "flops": pairs * m.H * m.D * 2, "pairs": pairs}


def run_mixed(args, dist: Dist):
    m = MIXED[args.workload]
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    rotate = ROTATE
    st = MixedSetup(m, dev, rotate)
    for i in range(rotate):
        st.step(i)
    torch.cuda.synchronize()
    X = st.X
    X.indexer_status(st.ws)
    X.indexer_status(st.status)
    g_full = capture(st.step, rotate)
    n_full = max(1, args.steps // rotate)
    steps = n_full * rotate
    for _ in range(max(1, math.ceil(args.warmup / rotate))):
        g_full.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(dist.local)
    time.sleep(0.15)
    dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    e0.record()
    for _ in range(n_full):
        g_full.replay()
    e1.record()
    torch.cuda.synchronize()
    w1 = time.time()
    dist.barrier()
    sampler.region(w0, w1)
    time.sleep(0.1)
    clocks = sampler.stop()
    ms_max = dist.max(e0.elapsed_time(e1))
    X.indexer_status(st.ws)
    X.indexer_status(st.status)
    # the step's two calls alone (graphs of back-to-back launches, events around them)
    kernel_ms = {}
    for name, fn in (("publish_paged", st.publish), ("forward_paged", st.forward)):
        g = capture(fn, rotate)
        g.replay()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        for _ in range(10):
            g.replay()
        a1.record()
        torch.cuda.synchronize()
        kernel_ms[name] = a0.elapsed_time(a1) / (10 * rotate)
    units = mixed_units(m)
    peaks = measured_peaks()
    fwd = kernel_ms["forward_paged"]
    t_hbm = units["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_mma = units["flops"] / (peaks["bf16_tflops"] * FP4_OVER_BF16 * 1e12)
    if t_hbm >= t_mma:
        achieved = units["bytes"] / (fwd / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                "algorithmic_bytes_per_launch": units["bytes"],
                "kernel": "indexer_forward_paged (plan, query prep, scores, top-k)", "kernel_ms": fwd,
                "peak_source": f"{peaks['source']} hbm_gbs"}
    else:
        achieved = units["flops"] / (fwd / 1e3) / 1e12
        peak = peaks["bf16_tflops"] * FP4_OVER_BF16
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": None, "algorithmic_flops_per_launch": units["flops"],
                "kernel": "indexer_forward_paged (plan, query prep, scores, top-k)", "kernel_ms": fwd,
                "peak_source": f"{peaks['source']} bf16_tflops x {FP4_OVER_BF16:g} (nominal fp4/bf16)"}
    n_dec = sum(1 for _, S in m.seqs if S == 1)
    line = {
        "metric": METRIC, "value": dist.world * m.Q * steps / (ms_max / 1e3), "unit": UNIT, "n_gpus": dist.world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms_max / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e2m1 x e2m1 -> f32", "data": "synthetic",
        "config": {"workload": (f"{m.name}: mixed batch of {m.n_seq} sequences ({n_dec} decode rows, "
                                f"{m.n_seq - n_dec} prefill chunks), {m.Q} query rows, T_max {m.T_max}, H{m.H}, "
                                f"top-{m.topk}, keys in a pool of {m.num_pages} 64-key pages"),
                   "Q": m.Q, "n_seq": m.n_seq, "T_max": m.T_max, "H": m.H, "topk": m.topk, "ratio": m.ratio,
                   "l2": f"{rotate} rotating page pools / inputs ({rotate * m.num_pages * 4352 / 1e6:.0f} MB)",
                   "timing": "CUDA-graph replay, CUDA events on the launching stream"},
        "key_scores_per_s": dist.world * units["pairs"] * steps / (ms_max / 1e3),
        "kernel_ms": kernel_ms,
        "roofline": roof,
        "gpu_launches": 5 * steps,
        "clocks": clocks,
    }
    return line


def breakdown(st: Setup, rotate: int, reps: int = 20):
    """Average device time of each kernel of the step: a CUDA graph of `rotate`
    back-to-back launches of that kernel alone (rotating inputs), replayed `reps` times
    between CUDA events on the launching stream."""
    out = {}
    kinds = st.kernel_kinds()
    for name in ["publish", "prep_q", "prep_q_proj", "scores", "candidates", "topk"]:
        if name not in kinds:
            continue
        g = capture(kinds[name], rotate)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        out[name] = e0.elapsed_time(e1) / (reps * rotate)
    st.X.indexer_status(st.ws)
    return out


def run_e2e(st: Setup, n_steps: int, dist: Dist):
    wl, X = st.wl, st.X
    R = st.rotate
    tag = "q2" if wl.two_level else "q"
    qh = [t.cpu().pin_memory() for t in st.q[tag]]
    wh = [t.cpu().pin_memory() for t in st.w[tag]]
    lh = [t.cpu().pin_memory() for t in st.lat]
    outh = [torch.empty(st.top.shape, dtype=torch.int32).pin_memory() for _ in range(R)]
    qd, wd, ld = torch.empty_like(st.q[tag][0]), torch.empty_like(st.w[tag][0]), torch.empty_like(st.lat[0])
    q1 = st.q.get("q1")
    steps = n_steps if wl.S == 1 else min(n_steps, 64)

    if wl.fused_q:   # the query latent crosses the bus instead of q
        qh = [t.cpu().pin_memory() for t in st.qr]
        qd = torch.empty_like(st.qr[0])
    host_call = not wl.fused_q and not wl.two_level   # one C call takes the host buffers itself
    if host_call:
        # consecutive steps alternate between two streams, each with its own workspace, output
        # buffer and key cache (where the workload rotates fewer than two), so that one step's
        # host copies overlap the kernels of the step before, as a serving loop would run them
        streams = [torch.cuda.Stream(device=st.dev) for _ in range(2)]
        ws_h = []
        for _ in range(2):
            w_ = torch.empty(X.indexer_workspace_size_host(st.dims, wl.B, wl.S, wl.start_pos, lh[0].shape[1],
                                                           lh[0].shape[2]), dtype=torch.uint8, device=st.dev)
            X.indexer_workspace_init(w_)
            ws_h.append(w_)
        caches = st.caches if R >= 2 else [st.caches[0], st.caches[0].clone()]
        outs = outh if R >= 2 else [outh[0], torch.empty_like(outh[0]).pin_memory()]

    def one(i):
        j = i % R
        if host_call:
            sp = wl.start_pos if st.decode else 0
            k = i % 2
            c = j if R >= 2 else k
            X.indexer_forward_publish_host(st.dims, lh[j], st.wk, st.knw, qh[j], wh[j], sp, st.table, caches[c],
                                           outs[c], ws_h[k], stream=streams[k])
            return
        qd.copy_(qh[j], non_blocking=True)
        wd.copy_(wh[j], non_blocking=True)
        ld.copy_(lh[j], non_blocking=True)
        sp = wl.start_pos if st.decode else 0
        if wl.fused_q:
            X.indexer_publish_k(st.dims, ld, st.wk, st.knw, st.table, sp, st.caches[j])
            X.indexer_prep_q_proj(st.dims, qd, st.wq, wd, wl.start_pos, st.table, st.q_rows, st.w_prime, st.ws)
            X.indexer_scores(st.dims, st.q_rows, st.w_prime, wl.start_pos, st.caches[j], st.scores, st.ws)
            X.indexer_topk(st.dims, st.scores, wl.start_pos, st.top)
        elif wl.two_level:
            X.indexer_forward_publish(st.dims, ld, st.wk, st.knw, q1[j], st.w["q1"][j], sp, st.table, st.caches[j],
                                      st.top1, st.ws, cand_out=st.cand)
            X.indexer_forward(st.dims, qd, wd, wl.start_pos, st.table, st.caches[j], st.top, st.ws, cand_in=st.cand)
        else:
            X.indexer_forward_publish(st.dims, ld, st.wk, st.knw, qd, wd, sp, st.table, st.caches[j], st.top, st.ws)
        outh[j].copy_(st.top, non_blocking=True)

    for i in range(min(8, steps)):
        one(i)
    torch.cuda.synchronize()
    dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    if host_call:
        for s_ in streams:
            s_.wait_event(e0)
    for i in range(steps):
        one(i)
    if host_call:
        for s_ in streams:
            torch.cuda.current_stream().wait_stream(s_)
    e1.record()
    torch.cuda.synchronize()
    ms = dist.max(e0.elapsed_time(e1))
    if host_call:
        for w_ in ws_h:
            X.indexer_status(w_)
    h2d = qh[0].numel() * 2 + wh[0].numel() * 2 + lh[0].numel() * 2
    d2h = outh[0].numel() * 4
    return {"value": dist.world * wl.B * wl.S * steps / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": ms / steps,
            "api": ("indexer_publish_k, indexer_prep_q_proj, indexer_scores, indexer_topk" if wl.fused_q
                    else "indexer_forward_publish_host" if host_call else "indexer_forward_publish")
                   + " (eager Python/ctypes calls, pinned host buffers"
                   + ("; consecutive steps on two streams, each step's copies overlapping the step before)"
                      if host_call else ")")}


def describe(wl: Workload) -> str:
    kind = "decode" if wl.S == 1 else "prefill"
    extra = f", two-level {wl.cand_topk_blocks}x{wl.cand_block_size} candidate blocks" if wl.two_level else ""
    if wl.fused_q:
        extra += f", queries from qr through wq_b (q_lora_rank {wl.q_lora_rank}) fused into the query prep"
    return (f"{wl.name}: {kind} B{wl.B} S{wl.S} start_pos {wl.start_pos}, ratio {wl.ratio} -> {wl.T} compressed "
            f"positions, H{wl.H} {fmt_of(wl)['label']} heads, top-{wl.topk}, offset {wl.offset}{extra}")


# ----------------------------------------------------------------------------- oracle arm / baseline
class OracleSample:
    """The CPU oracle on one sequence of the workload (its keys published once, untimed).
    A decode step is the sequence's query row with the publish of the key its token
    completes; a prefill step is a set of query rows sampled across the sequence (rows are
    independent given the keys), each generated on its own from the seeded streams."""

    def __init__(self, wl: Workload, b: int = 0):
        import oracle as O
        self.O, self.wl, self.b = O, wl, b
        from tests import cases as C
        self.C = C
        self.cos, self.sin = C.oracle_table(wl.max_pos, wl.rope_dim)
        self.wk, self.knw = C.bits(wl.wk()), C.bits(wl.k_norm_w())
        self.fmt = fmt_of(wl)
        lat = C.bits(wl.latent()[b:b + 1])
        slots, rows, _ = O.publish_keys(lat, self.wk, self.knw, self.cos, self.sin, 0, wl.ratio, wl.rope_dim,
                                        wl.norm_eps, fmt=self.fmt["name"])
        self.cache = np.zeros((1, wl.T_cap, self.fmt["row"]), np.uint8)
        self.cache[0, slots] = rows[0]
        self.w = C.bits(wl.w()[b])                                   # [S, H], heavy rows included
        if wl.fused_q:   # queries from the query latent through wq_b, inside the timed step
            self.qr, self.wq = C.bits(wl.qr()[b]), C.bits(wl.wq_b())
        self.dl = C.bits(wl.decode_latent()[b:b + 1]) if wl.S == 1 and wl.start_pos > 0 else None

    def run(self, rows) -> int:
        """One oracle step over the given query rows of the sequence (publish of the step's key
        for decode, query prep, scores, causal mask, top-k); returns the rows done."""
        O, wl, C = self.O, self.wl, self.C
        rows = np.asarray(rows)
        if self.dl is not None:
            slots, krows, _ = O.publish_keys(self.dl, self.wk, self.knw, self.cos, self.sin, wl.start_pos,
                                             wl.ratio, wl.rope_dim, wl.norm_eps, fmt=self.fmt["name"])
            self.cache[0, slots] = krows[0]
        flat = [self.b * wl.S + int(r) for r in rows]
        if wl.fused_q:
            q = O.project_queries(self.qr[rows][None], self.wq, wl.H)
        else:
            q = C.bits(wl.q_rows(flat))[None]                       # [1, R, H, D]
        pos = wl.start_pos + rows
        q_rows, wprime, _ = O.prep_queries(q, self.w[rows][None], self.cos, self.sin, wl.start_pos, wl.rope_dim,
                                           wl.H, row_positions=pos, fmt=self.fmt["name"])
        vis = O.visible_lens(wl.start_pos, len(rows), wl.ratio, row_positions=pos)
        sc = O.index_scores(q_rows, wprime, self.cache, wl.T, vis)
        O.topk_positions(sc[0], vis, wl.topk, wl.offset, wl.T)
        return len(rows)


def _oracle_worker(job):
    """One host process of the oracle baseline: an OracleSample of one sequence, then steps of
    `rows_per_step` sampled rows until `seconds` have passed (or exactly `n_steps` steps).
    Returns (rows done, wall seconds, CPU seconds)."""
    name, worker, seconds, n_steps, n_warm, rows_per_step = job
    wl = WORKLOADS[name]
    samp = OracleSample(wl, b=worker % wl.B)
    rng = np.random.default_rng(1000 + worker)
    pick = lambda: np.sort(rng.choice(wl.S, size=min(rows_per_step, wl.S), replace=False))
    for _ in range(n_warm):
        samp.run(pick())
    n = 0
    c0, t0 = time.process_time(), time.perf_counter()
    k = 0
    while True:
        n += samp.run(pick())
        k += 1
        if (n_steps and k >= n_steps) or (not n_steps and time.perf_counter() - t0 >= seconds):
            break
    return n, time.perf_counter() - t0, time.process_time() - c0


def _oracle_pool_run(name: str, seconds: float, n_steps: int, n_warm: int, rows_per_step: int):
    """Runs _oracle_worker in one spawned process per host core (single-threaded numpy each)."""
    import multiprocessing as mp
    n = max(1, os.cpu_count() or 1)
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            res = pool.map(_oracle_worker, [(name, i, seconds, n_steps, n_warm, rows_per_step) for i in range(n)])
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    rows = sum(r[0] for r in res)
    wall = max(r[1] for r in res)
    cpu = sum(r[2] for r in res)
    return rows, wall, cpu, n


def _rows_per_step(wl: Workload) -> int:
    return 1 if wl.S == 1 else 2


def cpu_baseline(wl: Workload, seconds: float):
    rps = _rows_per_step(wl)
    rows, wall, cpu, n = _oracle_pool_run(wl.name, seconds, 0, 1, rps)
    return {"value": rows / wall, "unit": UNIT, "cores": n, "nproc": os.cpu_count(), "kind": "oracle",
            "cpu_seconds_per_wall_second": cpu / wall,
            "sample": (f"{n} processes (one per host core, single-threaded numpy f64), each on one sequence of "
                       f"{describe(wl)}: steps of {rps} query row(s) drawn uniformly over the sequence's rows "
                       f"(decode: the step's key publish too), {rows} rows in {wall:.1f} s wall; keys published "
                       f"untimed")}


def run_reference(args, dist: Dist):
    if args.workload in MIXED:
        return ({"impl": "reference", "unavailable": "the oracle reference arm times the uniform workloads; "
                 "mixed page-pool batches are compared with the oracle per sequence in the tests"}
                if dist.rank == 0 else None), None
    wl = WORKLOADS[args.workload]
    if dist.rank != 0:
        return None, wl
    rps = _rows_per_step(wl)
    rows, wall, cpu, n = _oracle_pool_run(wl.name, 0.0, args.steps, args.warmup, rps)
    value = rows / wall
    sample = (f"each step: every one of {n} processes (one per host core, single-threaded numpy f64) runs {rps} "
              f"query row(s) of one sequence of {describe(wl)}, drawn uniformly over its rows (decode: with the "
              f"step's key publish); keys published untimed")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": wall * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": describe(wl), "B": wl.B, "S": wl.S, "start_pos": wl.start_pos, "T": wl.T, "H": wl.H,
                   "topk": wl.topk, "ratio": wl.ratio},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": n, "nproc": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line, wl


def profile_kernel(args):
    """The workload's kernels once each through the split entry points (so every input of the
    named kernel is real), then the named kernel three more times; prints one short line."""
    wl = WORKLOADS[args.workload]
    if args.batch:
        wl = dataclasses.replace(wl, B=args.batch)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    st = Setup(wl, dev, 1)
    kinds = st.kernel_kinds()
    order = ["publish", "prep_q", "scores"] + (["candidates"] if wl.two_level else []) + ["topk"]
    for k in order:
        kinds[k](0)
    torch.cuda.synchronize()
    for _ in range(3):
        kinds[args.profile_kernel](0)
    torch.cuda.synchronize()
    st.X.indexer_status(st.ws)
    print(json.dumps({"profile_kernel": args.profile_kernel, "workload": describe(wl)}), flush=True)


def main():
    args = parse_args()
    if args.profile_kernel:
        profile_kernel(args)
        return
    dist = Dist()
    try:
        if args.impl == "reference":
            line, _ = run_reference(args, dist)
        elif args.workload in MIXED:
            line = run_mixed(args, dist)
        else:
            line, wl = run_ours(args, dist)
            if args.workload == HEADLINE and not args.no_per_config:
                line["per_config"] = per_config_records(args, dist)
                line["upstream_producers"] = measure_producers(wl, torch.device("cuda", dist.local))
            if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
        if dist.rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
