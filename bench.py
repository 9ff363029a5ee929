#!/usr/bin/env python3
"""Benchmark of the PowerSGD hook step on GB300.

Metric: PowerSGD step throughput as gradient GB/s (W replica buckets of N
fp32 elements consumed per step, W * N * 4 bytes / step time), with the HBM
roofline fraction of the dominant kernel.  One step = one psgd_step call in
the compressed phase (warm-started Q): error feedback + unscale + replica
mean + P = M Q, Gram-Schmidt, Q = M^T P, decompression, on every tensor of
the bucket.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Multi-GPU: the path simulates its W data-parallel replicas inside one GPU and
does not shard, so N GPUs run N independent replicas of the workload
(weak scaling); the time is the max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

# The bucket-group rows run on up to 16 streams; CUDA's default of 8 hardware
# work queues makes streams 9-16 share queues with 1-8 (false dependencies
# between independent buckets: GPT-2-XL's 290 buckets on 16 streams 9.9 ms
# against 9.4 ms with 16 queues).  Process-local, read when CUDA starts.
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "16")

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "PowerSGD step throughput, gradient GB/s and % of HBM roofline (1 GB300)"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="bert-large",
                    choices=["bert-large", "gpt2-xl", "resnet50", "rank-sweep", "fp16-scaled"])
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--extra", default="gpt2-xl,bert-large:bf16,gpt2-xl:bf16,fp16-scaled",
                    help="comma-separated workloads also measured and reported under 'workloads' "
                         "(NAME or NAME:DTYPE; fp16-scaled = the 8192 x 8192 rank-4 matrix in fp16 "
                         "pre-scaled by 65536 and unscaled by 2^-16 in pass 1; 'none' for none)")
    ap.add_argument("--grad-dtype", default="f32", choices=["f32", "f16", "bf16"],
                    help="type of the replica gradient buckets of the main workload (the pages' "
                         "fp16/bf16 compress wrappers hand the hook 16-bit buckets)")
    ap.add_argument("--rank", type=int, default=None, help="rank of the rank-sweep workload")
    ap.add_argument("--replicas", type=int, default=None,
                    help="replica count W of the main workload instead of its own (e.g. 3 or 6 on "
                         "the BERT-large bucket)")
    ap.add_argument("--layers", type=int, default=None,
                    help="profiling cases: only this many transformer layers, no embeddings")
    ap.add_argument("--batched", dest="batched", action="store_true", default=True,
                    help="also time batched_powerSGD_hook on the workload's bucket (one padded square; default)")
    ap.add_argument("--no-batched", dest="batched", action="store_false")
    ap.add_argument("--buckets", type=float, default=25.0,
                    help="also time the workload split into DDP-style buckets of at most this many MB "
                         "(tensors in reverse order), stepped on one stream, on --bucket-streams, and on "
                         "--bucket-streams with CUDA-graph replay (default 25, DDP's bucket_cap_mb; 0: off)")
    ap.add_argument("--bucket-streams", type=int, default=16,
                    help="streams of the overlapped bucket-group runs (--buckets)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
GSIZE = {"f32": 4, "f16": 2, "bf16": 2}
LOSS_SCALE = 65536.0   # GradScaler's default initial scale


def workload_spec(name, rank_override=None, layers=None, dtype="f32", replicas=None):
    """A workload: the bucket's tensor shapes, replicas, rank and input
    recipe; `dtype` is the type of the replica buckets (f32, f16, bf16).
    fp16-scaled is the 8192 x 8192 rank-4 matrix whose N(0, 1e-3) gradients
    are multiplied by 65536 and stored in fp16, as GradScaler-scaled
    half-precision training produces them; pass 1 unscales by 2^-16."""
    from powersgd_rank_gradient_gb300 import workloads as wl

    if name == "rank-sweep":
        spec = dict(name=f"rank-sweep-8192-r{rank_override or 8}", shapes=[(8192, 8192)], world_size=1,
                    rank=rank_override or 8, mcr=2.0, std=1.0, heavy=0.0, batch_same_shape=False)
    elif name == "fp16-scaled":
        spec = dict(name="fp16-scaled-8192-r4", shapes=[(8192, 8192)], world_size=1, rank=4, mcr=2.0,
                    std=1e-3, heavy=0.0, batch_same_shape=False)
        dtype = "f16"
        spec["loss_scale"] = LOSS_SCALE
    else:
        w = wl.WORKLOADS[name]
        if layers is not None and name in ("bert-large", "gpt2-xl"):
            shapes = w["shapes"](layers=layers, embeddings=False)
            name = f"{name}-{layers}layers"
        else:
            shapes = w["shapes"]()
        spec = dict(name=name, shapes=shapes, world_size=w["world_size"], rank=w["rank"],
                    mcr=w["mcr"], std=w["std"], heavy=w["heavy"], batch_same_shape=w["batch_same_shape"])
    spec.setdefault("loss_scale", 1.0)
    if replicas is not None and replicas != spec["world_size"]:
        spec["world_size"] = replicas
        spec["name"] = f"{spec['name']}-W{replicas}"
    spec["dtype"] = dtype
    if dtype != "f32" and not spec["name"].endswith(dtype) and name != "fp16-scaled":
        spec["name"] = f"{spec['name']}-{dtype}"
    return spec


def make_bucket(spec, seed, device):
    """One replica's bucket of the workload, in its gradient type."""
    import torch

    from powersgd_rank_gradient_gb300 import workloads as wl

    g = wl.gaussian_bucket_torch(spec["shapes"], spec["std"], seed, device, heavy_fraction=spec["heavy"])
    if spec["loss_scale"] != 1.0:
        g.mul_(spec["loss_scale"])
    if spec["dtype"] == "f16":
        return g.half()
    if spec["dtype"] == "bf16":
        return g.bfloat16()
    return g


def torch_dtype(spec):
    import torch

    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[spec["dtype"]]


def plan_counts(spec):
    from powersgd_rank_gradient_gb300 import _lib

    comp, ranks, rows, cols = _lib.plan(spec["shapes"], spec["rank"], spec["mcr"])
    numels = []
    for s in spec["shapes"]:
        n = 1
        for d in s:
            n *= d
        numels.append(n)
    nc = sum(n for n, c in zip(numels, comp) if c)
    return dict(N=sum(numels), Nc=nc, Nunc=sum(numels) - nc, compressed=sum(comp),
                tensors=len(numels),
                pq=sum((r + c) * k for r, c, k, cc in zip(rows, cols, ranks, comp) if cc))


def step_bytes(spec, counts):
    """Bytes one step must move.  'design' is this implementation's
    three-pass schedule with the factored residual; 'survey_min' is the
    explicit-residual minimum per compressed element, the smaller of the
    scheme that overwrites e_w with M_w in pass 1 (W s_g + 20 W + 4) and the
    one that re-reads g and e in pass 3 (2 W s_g + 12 W + 12) -- the bound
    the targets are quoted against (for fp32, min(6W+1, 5W+3) * 4)."""
    W = spec["world_size"]
    gsz = GSIZE[spec["dtype"]]
    nc, nu = counts["Nc"], counts["Nunc"]
    reread = W * 4
    mbar = reread > 8
    p1 = W * (gsz + 8) + (4 if mbar else 0)
    p2 = 4 if mbar else reread
    design = nc * (p1 + p2 + 4) + nu * (W * gsz + 4)
    per_el = min(W * gsz + 20 * W + 4, 2 * W * gsz + 12 * W + 12)
    survey = nc * per_el + nu * (W * gsz + 4) + (W + 1) * counts["pq"] * 4
    # pass 1 of the explicit-residual scheme: read g_w and e_w, write M_w
    survey_pass1 = nc * W * (gsz + 8)
    return dict(design=design, survey_min=survey, survey_pass1=survey_pass1)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_src_hash():
    """Hash of the sources the captured pass kernels (the chunk-stationary
    pass 1 of ranks up to 8, passes 2 and 3) are compiled from: their device
    code, tiling constants and launchers.  Host code and the other kernels
    (the Gram-Schmidt stage, the rank-16/32 tensor-core kernels) do not change
    their counters."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "powersgd_rank_gradient_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if not (f in ("psgd_kernels.cuh", "psgd_internal.h", "psgd_launch_rp.cuh")
                or (f.startswith("kern_rp") and f.endswith(".cu"))):
            continue
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it
    was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("src_hash") != kernel_src_hash():
        return None
    ent = d.get("workloads", {}).get(workload, {}).get(kernel)
    return None if ent is None else float(ent)


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]),
                                     hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            if r["hw"].lower().startswith("active"):
                reasons.add("hw_slowdown")
            if r["hwt"].lower().startswith("active"):
                reasons.add("hw_thermal_slowdown")
            if r["swt"].lower().startswith("active"):
                reasons.add("sw_thermal_slowdown")
            if r["pcap"].lower().startswith("active"):
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


# ---------------------------------------------------------------------------
# multi-rank aggregation (one independent replica of the workload per GPU)
# ---------------------------------------------------------------------------
def reduce_max(x, dist, device=None):
    """Max of a float over all ranks (identity without a process group)."""
    if dist is None:
        return float(x)
    import torch

    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step, steps, ranks, max_ms):
    """Whole-job GB/s: every rank processed `steps` steps of
    `bytes_per_rank_step` bytes; the job took the slowest rank's time."""
    return bytes_per_rank_step * steps * ranks / (max_ms / 1e3) / 1e9


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------
def run_native(spec, args, dist, rank_id, world, device, light=False):
    """Times the workload's warm-started compressed step.  light: the step
    alone (no vanilla/first-call rows, batched hook, bucket groups or e2e)."""
    import torch

    from powersgd_rank_gradient_gb300 import PowerSGDState, workloads as wl

    W = spec["world_size"]
    counts = plan_counts(spec)
    N = counts["N"]
    gsz = GSIZE[spec["dtype"]]
    inv_scale = 1.0 / spec["loss_scale"]
    st = PowerSGDState(spec["shapes"], W, matrix_approximation_rank=spec["rank"], start_powerSGD_iter=0,
                       min_compression_rate=spec["mcr"], use_error_feedback=True, warm_start=True,
                       batch_tensors_with_same_shape=spec["batch_same_shape"], random_seed=0,
                       grad_dtype=torch_dtype(spec), device=device)
    # two resident input sets (W replica buckets each), alternated step to step
    sets = []
    for k in range(2):
        sets.append([make_bucket(spec, wl.replica_seed(w, k), device) for w in range(W)])
    out = torch.empty(N, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    # the clock sampler runs from the warm-up through the timed region
    clocks = Clocks(device.index)
    if rank_id == 0:
        clocks.start()
    for i in range(args.warmup):
        st.step(sets[i % 2], out=out, inv_loss_scale=inv_scale)
    if st.status():
        raise RuntimeError("warm-up step was skipped (non-finite input)")
    torch.cuda.synchronize(device)
    st.profile_read()  # discard warm-up records
    # the per-kernel breakdown: the same steps with an event pair around every
    # kernel (those events cost the small buckets several percent of a step,
    # so they stay out of the timed region)
    st.profile(True)
    for i in range(args.steps):
        st.step(sets[i % 2], out=out, inv_loss_scale=inv_scale)
    torch.cuda.synchronize(device)
    st.profile(False)
    prof_all = st.profile_read()
    kern = max((k for k in prof_all if prof_all[k][0] > 0), key=lambda k: prof_all[k][1])   # dominant
    launches_per_step = sum(v[0] for v in prof_all.values()) / args.steps
    # the timed region: events around the dominant kernel only
    st.profile_select([kern])
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        st.step(sets[i % 2], out=out, inv_loss_scale=inv_scale)
    e1.record(stream)
    torch.cuda.synchronize(device)
    if dist is not None:
        dist.barrier()
    clk = clocks.stop() if rank_id == 0 else None
    st.profile(False)
    ms = reduce_max(e0.elapsed_time(e1), dist, device)
    if st.status():
        raise RuntimeError("timed step was skipped (non-finite input)")
    prof = st.profile_read()
    ms_step = ms / args.steps
    grad_bytes = W * N * gsz
    value = job_throughput(grad_bytes, args.steps, world, ms)
    launches = int(round(launches_per_step * args.steps))
    n_l, tot_ms, bpl = prof[kern]
    peak, peak_kind = load_peaks()
    launch_s = tot_ms / n_l / 1e3 if n_l else None
    achieved = bpl / launch_s / 1e9 if n_l and bpl else None
    kernels = {k: {"launches": v[0], "avg_us": (v[1] / v[0] * 1e3) if v[0] else None,
                   "share": v[1] / max(1e-12, sum(x[1] for x in prof_all.values())),
                   "algo_bytes_per_launch": v[2] or None,
                   "gbs": (v[2] / (v[1] / v[0] / 1e3) / 1e9) if v[0] and v[2] else None}
               for k, v in prof_all.items() if v[0]}
    sb = step_bytes(spec, counts)
    roof = {"bound": "hbm", "kernel": kern, "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": (achieved / peak) if achieved else None, "peak_source": peak_kind,
            "traffic": ncu_traffic(spec["name"], kern),
            "bytes_basis": "the kernel's own algorithmic bytes per launch",
            "timing": "CUDA events around this kernel's launches inside the timed region (the "
                      "region records no other kernel's events); kernels[...] come from a "
                      "profiled pass over the same steps just before it"}
    roof["frac_design"] = roof["frac"]
    if kern == "pass1" and launch_s:
        # the explicit-residual scheme's pass 1 (read g_w and e_w, write M_w:
        # W (s_g + 8) bytes per compressed element), on the same launch time
        roof["achieved_survey_pass1"] = sb["survey_pass1"] / launch_s / 1e9
        roof["frac_survey_pass1"] = roof["achieved_survey_pass1"] / peak
    step_gbs = sb["design"] / (ms_step / 1e3) / 1e9
    survey_gbs = sb["survey_min"] / (ms_step / 1e3) / 1e9
    res = dict(
        value=value, ms_per_step=ms_step, grad_bytes=grad_bytes, launches=launches, clocks=clk,
        roofline=roof,
        step_roofline={"design_bytes": sb["design"], "design_gbs": step_gbs,
                       "design_frac_of_measured": step_gbs / peak,
                       "survey_min_bytes": sb["survey_min"],
                       "survey_min_note": "explicit-residual equivalent: the bytes a design that writes "
                                          "e_w would move; the factored residual moves fewer, so this "
                                          "fraction can exceed 1",
                       "survey_min_frac_of_nominal_8tbs": survey_gbs / NOMINAL_HBM_GBS,
                       "survey_min_frac_of_measured": survey_gbs / peak},
        kernels=kernels, counts=counts, dtype=spec["dtype"], loss_scale=spec["loss_scale"])
    if not light:
        res["rows"] = run_rows(spec, args, dist, device, sets, out, W, N)
        res["rows"]["steady_step_graph"] = run_graph(st, spec, args, dist, device, sets[0], out, W, N)
        try:
            res["rows"]["dp_split_one_process"] = run_dp(spec, args, dist, device, sets[0][0], out, N)
        except Exception as e:   # a row, not the headline: report it and go on
            res["rows"]["dp_split_one_process"] = {"error": str(e)}
        if args.batched:
            res["rows"]["next_batched_hook"] = run_batched(spec, args, dist, device, sets, out, W, N)
        if args.buckets > 0:
            res["rows"]["next_bucket_overlap"] = run_buckets(spec, args, dist, device, sets, W, N)
    del sets
    torch.cuda.empty_cache()
    if not args.no_e2e and not light:
        res["e2e"] = run_e2e(st, spec, args, dist, device, N, W)
    st.close()
    return res


def run_graph(st, spec, args, dist, device, grads, out, W, N):
    """The same steady step replayed as one CUDA graph (psgd_set_graph), against
    the launched step on the same inputs: what launch gaps cost.  The graph is
    keyed by the buffers' addresses, so both runs step one resident input set
    (far larger than L2).  No per-kernel events inside a graph: step time only."""
    import torch

    stream = torch.cuda.current_stream(device)
    inv_scale = 1.0 / spec["loss_scale"]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    res = {}
    for label, graph in (("launched_ms_per_step", False), ("graph_ms_per_step", True)):
        st.set_graph(graph)
        for _ in range(3):
            st.step(grads, out=out, inv_loss_scale=inv_scale)
        torch.cuda.synchronize(device)
        e0.record(stream)
        for _ in range(args.steps):
            st.step(grads, out=out, inv_loss_scale=inv_scale)
        e1.record(stream)
        torch.cuda.synchronize(device)
        res[label] = reduce_max(e0.elapsed_time(e1), dist, device) / args.steps
    caps, reps = st.graph_stats()
    st.set_graph(False)
    if st.status():
        raise RuntimeError("graph-replayed step was skipped (non-finite input)")
    res["graph_gradient_gbs"] = W * N * GSIZE[spec["dtype"]] / (res["graph_ms_per_step"] / 1e3) / 1e9
    res["graph_captures"] = caps
    res["graph_replays"] = reps
    return res


def run_dp(spec, args, dist, device, grad, out, N):
    """The data-parallel split (one replica per process: begin, project,
    finish) in a one-process world, where its two exchanges are identities,
    against the fused step of a one-replica state on the same bucket: what the
    split costs a process besides its collectives."""
    import torch

    from powersgd_rank_gradient_gb300 import DataParallelPowerSGDState, PowerSGDState

    stream = torch.cuda.current_stream(device)
    inv_scale = 1.0 / spec["loss_scale"]
    kw = dict(matrix_approximation_rank=spec["rank"], start_powerSGD_iter=0, min_compression_rate=spec["mcr"],
              batch_tensors_with_same_shape=spec["batch_same_shape"], grad_dtype=torch_dtype(spec), device=device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    res = {"replicas_per_process": 1}
    dp = DataParallelPowerSGDState(spec["shapes"], world_size=1, **kw)

    def dp_step():
        dp.begin(grad, out, inv_scale)
        dp.project()
        dp.finish()

    fused = PowerSGDState(spec["shapes"], 1, **kw)
    for label, fn in (("split_ms_per_step", dp_step),
                      ("fused_ms_per_step", lambda: fused.step([grad], out=out, inv_loss_scale=inv_scale))):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(device)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(device)
        res[label] = reduce_max(e0.elapsed_time(e1), dist, device) / args.steps
    if fused.status():
        raise RuntimeError("one-replica step was skipped (non-finite input)")
    res["split_gradient_gbs"] = N * GSIZE[spec["dtype"]] / (res["split_ms_per_step"] / 1e3) / 1e9
    dp.close()
    fused.close()
    return res


def run_rows(spec, args, dist, device, sets, out, W, N):
    """The survey's other hot-path rows on the same resident inputs:
    A1, the vanilla phase (every call before start_powerSGD_iter is the plain
    replica mean of the whole bucket), and A3, the first compressed call
    (draw Q, orthogonalise it, then the step) against a warm-started one."""
    import torch

    from powersgd_rank_gradient_gb300 import PowerSGDState

    stream = torch.cuda.current_stream(device)
    rows = {}
    gsz = GSIZE[spec["dtype"]]
    inv_scale = 1.0 / spec["loss_scale"]
    van = PowerSGDState(spec["shapes"], W, matrix_approximation_rank=spec["rank"],
                        start_powerSGD_iter=1 << 60, min_compression_rate=spec["mcr"],
                        use_error_feedback=False, grad_dtype=torch_dtype(spec), device=device)
    for i in range(3):
        van.step(sets[i % 2], out=out, inv_loss_scale=inv_scale)
    torch.cuda.synchronize(device)
    van.profile(True)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        van.step(sets[i % 2], out=out, inv_loss_scale=inv_scale)
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = reduce_max(e0.elapsed_time(e1), dist, device) / args.steps
    prof = van.profile_read()
    n_l, tot_ms, _ = prof["mean"]
    mean_bytes = N * (W * gsz + 4)
    peak, _ = load_peaks()
    rows["A1_vanilla_phase"] = {
        "ms_per_step": ms, "gradient_gbs": W * N * gsz / (ms / 1e3) / 1e9,
        "kernel": "mean", "algo_bytes_per_launch": mean_bytes,
        "achieved_gbs": mean_bytes / (tot_ms / n_l / 1e3) / 1e9,
        "frac_of_measured": mean_bytes / (tot_ms / n_l / 1e3) / 1e9 / peak}
    van.close()
    # A3: a fresh state's first compressed call (Q draw + orthogonalisation)
    fresh = PowerSGDState(spec["shapes"], W, matrix_approximation_rank=spec["rank"], start_powerSGD_iter=0,
                          min_compression_rate=spec["mcr"],
                          batch_tensors_with_same_shape=spec["batch_same_shape"],
                          grad_dtype=torch_dtype(spec), device=device)
    times = []
    for i in range(3):
        e0.record(stream)
        fresh.step(sets[i % 2], out=out, inv_loss_scale=inv_scale)
        e1.record(stream)
        torch.cuda.synchronize(device)
        times.append(e0.elapsed_time(e1))
    fresh.close()
    rows["A3_first_compressed_call"] = {"ms": times[0], "next_calls_ms": times[1:],
                                        "q_init_overhead_ms": times[0] - min(times[1:])}
    return rows


def run_batched(spec, args, dist, device, sets, out, W, N):
    """batched_powerSGD_hook on the same bucket: one zero-padded square of
    side ceil(sqrt(N)), warm-started steps."""
    import torch

    from powersgd_rank_gradient_gb300 import BatchedPowerSGDState

    stream = torch.cuda.current_stream(device)
    gsz = GSIZE[spec["dtype"]]
    inv_scale = 1.0 / spec["loss_scale"]
    st = BatchedPowerSGDState(N, W, matrix_approximation_rank=spec["rank"], start_powerSGD_iter=0,
                              grad_dtype=torch_dtype(spec), device=device)
    for i in range(3):
        st.step(sets[i % 2], out=out, inv_loss_scale=inv_scale)
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        st.step(sets[i % 2], out=out, inv_loss_scale=inv_scale)
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = reduce_max(e0.elapsed_time(e1), dist, device) / args.steps
    # per-kind kernel times on separate (profiled) steps
    st.profile(True)
    st.profile_read()
    for i in range(args.steps):
        st.step(sets[i % 2], out=out, inv_loss_scale=inv_scale)
    torch.cuda.synchronize(device)
    kinds = {k: round(v[1] / args.steps, 4) for k, v in st.profile_read().items() if v[0]}
    st.profile(False)
    side = st.side
    st.close()
    return {"side": side, "vector_path": side % 4 == 0, "ms_per_step": ms,
            "gradient_gbs": W * N * gsz / (ms / 1e3) / 1e9, "kernel_ms_per_step": kinds}


def ddp_buckets(shapes, cap_mb, elem_bytes=4):
    """Tensor indices per bucket, DDP-style: tensors in reverse order, a new
    bucket whenever the next tensor would take the current one past cap_mb."""
    from powersgd_rank_gradient_gb300 import workloads as wl

    cap = cap_mb * 2**20
    buckets, cur, used = [], [], 0
    for i in reversed(range(len(shapes))):
        nb = wl.numel(shapes[i]) * elem_bytes
        if cur and used + nb > cap:
            buckets.append(cur)
            cur, used = [], 0
        cur.append(i)
        used += nb
    if cur:
        buckets.append(cur)
    return buckets


def run_buckets(spec, args, dist, device, sets, W, N):
    """The same iteration with the bucket split into DDP-style buckets, each
    its own hook call: a PowerSGDGroup on one stream, on S, and on S with
    each bucket's steady step replayed as a CUDA graph."""
    import torch

    from powersgd_rank_gradient_gb300 import PowerSGDGroup, workloads as wl

    shapes = spec["shapes"]
    idx = ddp_buckets(shapes, args.buckets, GSIZE[spec["dtype"]])
    off = [0]
    for s_ in shapes:
        off.append(off[-1] + wl.numel(s_))
    bucket_shapes = [[shapes[i] for i in b] for b in idx]
    # each bucket's replica inputs: the values of input set 0, in fresh tensors
    grads = [[torch.cat([sets[0][w][off[i]:off[i + 1]] for i in b]) for w in range(W)] for b in idx]
    outs = [torch.empty(g[0].numel(), dtype=torch.float32, device=device) for g in grads]
    stream = torch.cuda.current_stream(device)
    gsz = GSIZE[spec["dtype"]]
    inv_scale = 1.0 / spec["loss_scale"]
    res = {"cap_mb": args.buckets, "n_buckets": len(idx),
           "largest_bucket_mb": max(g[0].numel() for g in grads) * gsz / 2**20}
    S = args.bucket_streams
    for label, n_streams, graphs in (("serial", 1, False), (f"streams_{S}", S, False),
                                     (f"streams_{S}_graphs", S, True)):
        grp = PowerSGDGroup(bucket_shapes, W, matrix_approximation_rank=spec["rank"], start_powerSGD_iter=0,
                            min_compression_rate=spec["mcr"],
                            batch_tensors_with_same_shape=spec["batch_same_shape"], n_streams=n_streams,
                            graphs=graphs, grad_dtype=torch_dtype(spec), device=device)

        def iteration():
            for b in range(len(idx)):
                grp.step(b, grads[b], out=outs[b], inv_loss_scale=inv_scale)
            grp.wait()

        for _ in range(max(3, args.warmup)):
            iteration()
        if grp.status():
            raise RuntimeError("bucket group step was skipped (non-finite input)")
        torch.cuda.synchronize(device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            iteration()
        e1.record(stream)
        torch.cuda.synchronize(device)
        ms = reduce_max(e0.elapsed_time(e1), dist, device) / args.steps
        res[label] = {"ms_per_step": ms, "gradient_gbs": W * N * gsz / (ms / 1e3) / 1e9}
        grp.close()
    del grads, outs
    torch.cuda.empty_cache()
    return res


def run_e2e(st, spec, args, dist, device, N, W):
    """Same metric through psgd_step_host: every step copies the W pinned host
    buckets to the device and reads the result back."""
    import torch

    from powersgd_rank_gradient_gb300 import workloads as wl

    gsz = GSIZE[spec["dtype"]]
    inv_scale = 1.0 / spec["loss_scale"]
    host = []
    for w in range(W):
        g = make_bucket(spec, wl.replica_seed(w, 7), device)
        h = torch.empty(N, dtype=g.dtype, pin_memory=True)
        h.copy_(g)
        host.append(h)
        del g
    host_out = torch.empty(N, dtype=torch.float32, pin_memory=True)
    stream = torch.cuda.current_stream(device)
    st.step_host(host, host_out, inv_loss_scale=inv_scale)  # allocates the staging buffers
    torch.cuda.synchronize(device)
    k = max(3, min(args.steps, 10))
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(k):
        st.step_host(host, host_out, inv_loss_scale=inv_scale)
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = reduce_max(e0.elapsed_time(e1), dist, device)
    ws = dist.get_world_size() if dist is not None else 1
    return {"value": job_throughput(W * N * gsz, k, ws, ms), "unit": UNIT,
            "h2d_bytes_per_step": W * N * gsz, "d2h_bytes_per_step": N * 4, "ms_per_step": ms / k}


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline / reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(spec, budget):
    """The first tensor of each distinct shape, in bucket order, up to `budget`
    elements (a tensor larger than the budget is skipped): every kind of layer
    matrix and vector of the bucket, once."""
    sel, seen = [], set()
    tot = 0
    for s in spec["shapes"]:
        key = tuple(s)
        if key in seen:
            continue
        n = 1
        for d in s:
            n *= d
        if n > budget or tot + n > budget:
            continue
        seen.add(key)
        sel.append(s)
        tot += n
    return sel, tot


def time_oracle(spec, steps, budget=None, target_s=None, warmup=1):
    import numpy as np

    import oracle
    from powersgd_rank_gradient_gb300 import workloads as wl

    W = spec["world_size"]
    if budget is None:
        budget = 10_500_000 if W >= 8 else (13_000_000 if W >= 4 else 32_000_000)
    shapes, n = oracle_sample(spec, budget)
    if not shapes:
        shapes, n = spec["shapes"][:1], 1
        for d in spec["shapes"][0]:
            n *= d
    o = oracle.PowerSGDOracle(shapes=shapes, world_size=W, matrix_approximation_rank=spec["rank"],
                              start_powerSGD_iter=0, min_compression_rate=spec["mcr"])
    grads = [wl.gaussian_bucket_np(shapes, spec["std"], wl.replica_seed(w, 0),
                                   heavy_fraction=spec["heavy"]) for w in range(W)]
    for _ in range(max(1, warmup)):
        o.step(grads)  # untimed (the first one draws Q)
    times = []
    t_start = time.perf_counter()
    for i in range(steps):
        t0 = time.perf_counter()
        o.step(grads)
        times.append(time.perf_counter() - t0)
        if target_s is not None and time.perf_counter() - t_start > target_s:
            break
    t = statistics.median(times)
    return dict(value=W * n * GSIZE[spec["dtype"]] / t / 1e9, unit=UNIT, cores=os.cpu_count(), kind="oracle",
                sample=f"{len(shapes)} tensors, the first of each distinct shape ({n} elements per replica, "
                       f"W={W}) of the {spec['name']} bucket, fp64 NumPy, median of {len(times)} steps",
                s_per_step=t)


# ---------------------------------------------------------------------------
def main():
    args = parse()
    rank_id = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    spec = workload_spec(args.workload, rank_override=args.rank, layers=args.layers, dtype=args.grad_dtype,
                         replicas=args.replicas)
    base_cfg = {"workload": spec["name"], "world_size_W": spec["world_size"],
                "matrix_approximation_rank": spec["rank"], "min_compression_rate": spec["mcr"],
                "start_powerSGD_iter": 0, "use_error_feedback": True, "warm_start": True,
                "batch_tensors_with_same_shape": spec["batch_same_shape"],
                "gradients": f"N(0,{spec['std']}) {spec['dtype']}" + (f", {spec['heavy']:.0%} heavy rows x100" if spec["heavy"] else "")
                             + (f", x{spec['loss_scale']:g} (unscaled in pass 1)" if spec["loss_scale"] != 1.0 else ""),
                "l2": "inputs larger than L2 (each step reads >10 GB)" if spec["name"] != "resnet50" else "inputs larger than L2",
                "parallelism": f"replicas x{world}"}

    if args.impl == "reference":
        if rank_id != 0:
            return
        cb = time_oracle(spec, args.steps, warmup=args.warmup, target_s=120.0)
        line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": cb["s_per_step"] * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": base_cfg,
                "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
                "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch

    dist = None
    if world > 1:
        import torch.distributed as tdist

        tdist.init_process_group("nccl")
        dist = tdist
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from powersgd_rank_gradient_gb300 import _lib

    _lib.lib()

    res = run_native(spec, args, dist, rank_id, world, device)
    extras = {}
    for item in [x for x in args.extra.split(",") if x and x != "none"]:
        name, _, dt = item.partition(":")
        sp = workload_spec(name, layers=args.layers, dtype=dt or "f32")
        if sp["name"] == spec["name"]:
            continue
        # the main workload's fp32 companions get every row; 16-bit lines the step alone
        r = run_native(sp, args, dist, rank_id, world, device, light=sp["dtype"] != "f32")
        extras[sp["name"]] = {"metric": METRIC, "value": r["value"], "unit": UNIT,
                              "ms_per_step": r["ms_per_step"], "dtype": sp["dtype"],
                              "loss_scale": sp["loss_scale"], "gpu_launches": r["launches"],
                              "config": {"workload": sp["name"], "world_size_W": sp["world_size"],
                                         "matrix_approximation_rank": sp["rank"],
                                         "gradients": f"N(0,{sp['std']}) {sp['dtype']}"
                                         + (f" x{sp['loss_scale']:g}" if sp["loss_scale"] != 1.0 else "")},
                              "roofline": r["roofline"], "step_roofline": r["step_roofline"],
                              "e2e": r.get("e2e"), "clocks": r["clocks"],
                              "kernels": r["kernels"], "rows": r.get("rows")}
    cpu = None
    if rank_id == 0 and world == 1 and not args.no_cpu:
        cb = time_oracle(spec, 50, target_s=15.0)
        cpu = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
    if dist is not None:
        dist.barrier()
    if rank_id == 0:
        line = {"metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "grad_dtype": spec["dtype"],
                "data": "synthetic",
                "config": base_cfg, "clocks": res["clocks"], "gpu_launches": res["launches"],
                "roofline": res["roofline"], "step_roofline": res["step_roofline"],
                "e2e": res.get("e2e"), "cpu_baseline": cpu, "kernels": res["kernels"],
                "rows": res.get("rows"),
                "workloads": extras}
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
