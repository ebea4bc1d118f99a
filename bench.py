"""Benchmark: ReplaySSM decode of a Nemotron-shaped Mamba-2 layer on GB300.

Workload (per GPU): batch 256, 128 heads, headdim 64, dstate 128, 8 groups, bf16 inputs,
FP32 checkpoint, window L = 16; synthetic seeded inputs of the layer's distributions.
One bench step = one window of L decode tokens for the whole batch (15 non-flush steps and
one flush), i.e. batch * L tokens. The 1 GiB checkpoint is larger than the 129 MB L2, so no
L2 flush is needed between steps.

``python bench.py [--gpus N --steps K --warmup W]`` prints one JSON line. Under torchrun
every rank decodes its own batch (weak scaling, no collective on the data path); value is
all ranks' tokens over the slowest rank's time. ``--impl reference`` times the FP64 oracle
on the host cores on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import pathlib
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = pathlib.Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import synthgen as sg  # noqa: E402

METRIC = "replay decode tokens/s & achieved HBM GB/s (vs ~8 TB/s), batch 256, L=16"
UNIT = "tokens/s"
WORKLOAD = dict(batch=256, nheads=128, headdim=64, dstate=128, ngroups=8, dtype="bf16", L=16)
PROFILE_TRAFFIC = ROOT / "profiles" / "replay_step_nemotron_b256.md"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ algorithmic bytes
def record_bytes(w, esz):
    """Bytes of one input record (x, B, dt) of one sequence."""
    return (w["nheads"] * w["headdim"] + w["ngroups"] * w["dstate"] + w["nheads"]) * esz


# Read-copy bytes per state element (NVFP4: half a byte of code plus one E4M3 scale per 16)
# and whether the copy has an FP32 scale per slab.
RC_BYTES = {"bf16": (2, False), "e4m3": (1, True), "fp16": (2, False), "nvfp4": (0.5 + 1 / 16, True)}


def step_bytes(w, n_prior: int, flush: bool, esz=2, state_bytes=4, rc_bytes=0, shared=False, slab_scale=False):
    """Algorithmic HBM bytes of one replay_step launch over the batch.

    Reads: the checkpoint (FP32, or the read copy on a non-flush step), the n_prior
    buffered records, this token's inputs (x, B, C, dt). Writes: y (FP32) and either the
    appended record (non-flush) or the new checkpoint (+ read copy) (flush). With a shared
    checkpoint the copy is the only state: a flush reads and writes just the copy.
    """
    b, H, P, N, G = w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"]
    S = b * H * P * N
    rec = b * record_bytes(w, esz)
    inputs = b * (H * P + 2 * G * N + H) * esz
    y = b * H * P * 4
    copy = S * rc_bytes + (b * H * 4 if slab_scale else 0)
    if flush:
        if shared:
            return 2 * copy + n_prior * rec + inputs + y
        return S * state_bytes + n_prior * rec + inputs + y + S * state_bytes + copy
    read = copy if rc_bytes else S * state_bytes
    return read + n_prior * rec + inputs + y + rec


def conv_bytes(w, esz=2, state_bytes=4):
    b, H, P, N, G = w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"]
    S = b * H * P * N
    return 2 * S * state_bytes + b * (H * P + 2 * G * N + H) * esz + b * H * P * 4


# ------------------------------------------------------------------ peaks and clocks
def hbm_peak():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return float(json.loads(p.read_text())["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_sources_sha():
    """Hash of the CUDA sources' code: comments and blank lines do not count, so a comment
    edit keeps the recorded ncu traffic valid."""
    h = hashlib.sha256()
    csrc = ROOT / "hybrid_model_ssm_mamba_gb300" / "csrc"
    for p in sorted(csrc.glob("*")):
        if p.suffix in (".cu", ".cuh", ".h"):
            text = re.sub(r"/\*.*?\*/", "", p.read_text(), flags=re.S)
            lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
            h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch from the committed ncu summary, if taken on these sources."""
    if not PROFILE_TRAFFIC.exists():
        return None
    vals = {}
    for line in PROFILE_TRAFFIC.read_text().splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            m = re.search(r"`([^`]*)`", v)
            vals[k.strip()] = m.group(1) if m else v.strip()
    if vals.get("kernel_sources_sha256") != kernel_sources_sha():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of this GPU's clocks during the timed region."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [s.strip() for s in line.split(",")]
            if len(f) < 8 or (self.uuid and self.uuid not in f[0]):
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ distributed plumbing
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ the replay arm
def window_inputs(shape, seed, L, torch):
    """L tokens of inputs on the device (one per position in the window) + pinned copies."""
    d = sg.token_inputs(shape, seed, np.arange(L))
    dev, host = [], []
    for t in range(L):
        ins = []
        for k in ("x", "B", "C", "dt"):
            a = np.ascontiguousarray(d[k].store[:, t])
            ht = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
            host.append(ht)
            ins.append(ht.to("cuda", non_blocking=False))
        dev.append(ins)
    return dev, [host[4 * t: 4 * t + 4] for t in range(L)]


def run_replay(args, rank, world, local_rank):
    import torch
    from hybrid_model_ssm_mamba_gb300 import replay as R

    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    w = dict(WORKLOAD)
    if args.kernels_only and args.batch:      # diagnostics: a smaller batch for profiler runs
        w["batch"] = args.batch
    L = w["L"]
    shape = sg.LayerShape(w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"], w["dtype"])
    A, D = sg.head_params(w["nheads"], 0)
    rc_code = {"none": R.REPLAY_RC_NONE, "bf16": R.REPLAY_RC_BF16, "e4m3": R.REPLAY_RC_FP8E4M3,
               "fp16": R.REPLAY_RC_FP16, "nvfp4": R.REPLAY_RC_NVFP4}[args.read_copy]
    cfg = R.ReplayConfig(w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"], L, 0,
                         R.REPLAY_BF16, rc_code, int(args.shared_checkpoint),
                         R.REPLAY_CKPT_F16_SR if args.fp16_checkpoint else R.REPLAY_CKPT_F32)
    st = R.ReplayStore(cfg, torch.from_numpy(A), torch.from_numpy(D))
    dev, host = window_inputs(shape, rank, L, torch)
    y = torch.empty(w["batch"], w["nheads"], w["headdim"], device="cuda")
    stream = torch.cuda.current_stream()

    def window(events=None):
        for t in range(L):
            if events is not None:
                events[t][0].record(stream)
            st.step(*dev[t], y)
            if events is not None:
                events[t][1].record(stream)

    for _ in range(args.warmup):
        window()
    torch.cuda.synchronize()
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(L)]
          for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = str(getattr(torch.cuda.get_device_properties(local_rank), "uuid", ""))
    barrier(world)
    torch.cuda.synchronize()
    # The timed region holds the steps alone: an event recorded between two steps would keep
    # a step's prep kernel from starting during the previous step (read copies).
    with ClockSampler(uuid) as clk:
        t0.record(stream)
        for k in range(args.steps):
            window()
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    elapsed = t0.elapsed_time(t1) / 1e3
    # Per-call durations (non-flush and flush calls), from a diagnostic pass after the timed
    # region with an event pair around every call.
    diag = min(args.steps, 20)
    for k in range(diag):
        window(ev[k])
    torch.cuda.synchronize()
    launch_s = np.array([[ev[k][t][0].elapsed_time(ev[k][t][1]) / 1e3 for t in range(L)] for k in range(diag)])
    assert st.status() == 0
    elapsed_max = max_over_ranks(elapsed, world, "cuda")
    tokens = world * w["batch"] * L * args.steps

    # roofline of replay_step: the algorithmic bytes of every call in the timed region / the
    # region's event-timed duration (calls run back to back: the window-average call)
    rcb, slab_scale = RC_BYTES[args.read_copy] if args.read_copy != "none" else (0, False)
    per_pos = [step_bytes(w, t, flush=(t == L - 1), rc_bytes=rcb, shared=args.shared_checkpoint,
                          slab_scale=slab_scale) for t in range(L)]
    alg_bytes = sum(per_pos) * args.steps
    peak, peak_kind = hbm_peak()
    achieved = alg_bytes / elapsed / 1e9
    nf_bytes = sum(per_pos[:-1]) * diag
    nf_s = launch_s[:, :-1].sum()
    traffic = recorded_traffic()
    if args.kernels_only:   # a short diagnostic line for profiling runs, not the benchmark line
        return {"mode": "kernels-only", "read_copy": args.read_copy, "shared_checkpoint": args.shared_checkpoint,
                "tokens_per_s": tokens / elapsed_max, "achieved_gbs": achieved,
                "nonflush_launch_us": float(launch_s[:, :-1].mean() * 1e6),
                "flush_launch_us": float(launch_s[:, -1].mean() * 1e6)}

    # e2e: every token's inputs come from pinned host memory and its y goes back to pinned
    # host memory, through the public call. Copies run on their own streams, double-buffered,
    # so token t+1's inputs travel while token t decodes and y_t returns meanwhile.
    y_host = [torch.empty(w["batch"], w["nheads"], w["headdim"], pin_memory=True) for _ in range(L)]
    stage = [[torch.empty_like(t) for t in dev[0]] for _ in range(2)]
    ybuf = [torch.empty_like(y) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731

    def e2e_window(prev):
        """prev: events of the previous window's last two tokens (buffer reuse)."""
        done_in, done_step, done_out = {}, dict(prev["step"]), dict(prev["out"])
        for t in range(L):
            slot = t % 2
            with torch.cuda.stream(s_in):
                if (t - 2) in done_step:
                    s_in.wait_event(done_step[t - 2])        # the step that read this buffer
                for dst, src in zip(stage[slot], host[t]):
                    dst.copy_(src, non_blocking=True)
                done_in[t] = ev()
                done_in[t].record(s_in)
            stream.wait_event(done_in[t])
            if (t - 2) in done_out:
                stream.wait_event(done_out[t - 2])           # y buffer copied out
            st.step(*stage[slot], ybuf[slot], stream)
            done_step[t] = ev()
            done_step[t].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_step[t])
                y_host[t].copy_(ybuf[slot], non_blocking=True)
                done_out[t] = ev()
                done_out[t].record(s_out)
        return {"step": {t - L: done_step[t] for t in (L - 2, L - 1)},
                "out": {t - L: done_out[t] for t in (L - 2, L - 1)}}

    prev = {"step": {}, "out": {}}
    for _ in range(2):
        prev = e2e_window(prev)
    e_steps = max(1, min(args.steps, 50))
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    prev = {"step": {}, "out": {}}
    for _ in range(e_steps):
        prev = e2e_window(prev)
    for e in prev["out"].values():
        stream.wait_event(e)
    e1.record(stream)
    torch.cuda.synchronize()
    e_el = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, "cuda")
    h2d = sum(t.numel() * t.element_size() for ins in host for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in y_host)

    # the conventional load-update-store baseline on the same workload
    state = torch.zeros(w["batch"], w["nheads"], w["headdim"], w["dstate"], device="cuda")
    for t in range(L):
        R.conv_step(cfg, state, R.REPLAY_F32, st.A, st.D, *dev[t], y)
    c_steps = max(1, min(args.steps, 20))
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    c0.record(stream)
    for _ in range(c_steps):
        for t in range(L):
            R.conv_step(cfg, state, R.REPLAY_F32, st.A, st.D, *dev[t], y)
    c1.record(stream)
    torch.cuda.synchronize()
    conv_s = c0.elapsed_time(c1) / 1e3 / (c_steps * L)
    conv_tps = w["batch"] / conv_s
    del state
    extra = {}
    if not args.no_extra:
        extra["read_copy"] = run_read_copies(torch, R, dev)
        fp32_nf_us = float(launch_s[:, :-1].mean() * 1e6)
        fp32_window_us = elapsed / args.steps * 1e6
        fp32_nf_window_us = (fp32_window_us - float(launch_s[:, -1].mean() * 1e6)) / (L - 1)
        for v in extra["read_copy"].values():   # the post's "non-flush kernel N x faster" figure
            v["nonflush_speedup_vs_fp32"] = fp32_nf_us / v["nonflush_launch_us"]
            v["nonflush_speedup_vs_fp32_in_window"] = fp32_nf_window_us / v["nonflush_us_in_window"]
            v["window_speedup_vs_fp32"] = fp32_window_us / v["window_us"]
        extra["speculative"] = run_speculative(torch, R)
        keep = ("replay_verify_commit_us", "snapshot_verify_commit_us", "conventional_step_us",
                "replay_speedup_vs_snapshot", "replay_vs_standard_step")
        extra["speculative"]["by_drafts"] = {
            f"T{T}": {k: round(v, 3) for k, v in run_speculative(torch, R, T=T).items() if k in keep}
            for T in (1, 8)}
        # the batch x window sweep of the small layer (fewer tokens than --sweep) and the
        # 40-layer stack, compact: speed-up of replay over the conventional step per config
        sw = run_sweep(torch, R, tokens=128)
        extra["sweep"] = {"workload": "tiny-layer shape (8 heads, FP32 inputs), L2 flushed before every token; "
                                      "speedup = conventional us / replay us per token",
                          "speedup": {f"b{r['batch']}_L{r['window_L']}": round(r["speedup"], 3)
                                      for r in sw if "batch" in r},
                          "stack_40_layers": {k: v for k, v in sw[-1].items() if k != "sweep"}}

    result = {
        "metric": METRIC, "value": tokens / elapsed_max, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_max / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "Nemotron-shaped Mamba-2 layer decode, ReplaySSM window",
                   "batch_per_gpu": w["batch"], "nheads": w["nheads"], "headdim": w["headdim"],
                   "dstate": w["dstate"], "ngroups": w["ngroups"], "window_L": L,
                   "inputs": "bf16 x/B/C/dt, FP32 checkpoint, FP32 y",
                   "step": f"one window = {L} decode tokens x batch (15 non-flush + 1 flush)",
                   "l2": "1 GiB checkpoint > 129 MB L2: no flush needed",
                   "parallelism": f"dp{world} (independent batches)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": "replay_step (prep + main kernel per token, window average)",
                     "achieved_from": "algorithmic bytes of the timed region's calls / its event-timed duration",
                     "algorithmic_bytes_per_launch": alg_bytes / (args.steps * L),
                     "nonflush_achieved": nf_bytes / nf_s / 1e9,
                     "nonflush_frac": nf_bytes / nf_s / 1e9 / peak,
                     "nonflush_launch_us": float(launch_s[:, :-1].mean() * 1e6),
                     "flush_launch_us": float(launch_s[:, -1].mean() * 1e6),
                     "per_call_from": f"event pairs around each call, {diag} windows after the timed region"},
        "e2e": {"value": world * w["batch"] * L * e_steps / e_el, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * L * 2,
        "baselines": {"conv_step_tokens_per_s": conv_tps,
                      "conv_step_achieved_gbs": conv_bytes(w) / conv_s / 1e9,
                      "replay_speedup_vs_conv": (w["batch"] * L * args.steps / elapsed) / conv_tps},
        "clocks": clk.summary(),
        "extra": extra,
    }
    if rank == 0:
        result["cpu_baseline"] = cpu_baseline(args.cpu_sample_seqs, args.cpu_sample_tokens)
    st.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result if rank == 0 else None


# ------------------------------------------------------------------ secondary workloads
SPEC = dict(batch=512, nheads=8, headdim=64, dstate=128, ngroups=1, dtype="f32", L=16, T=4)


def l2_flusher(torch):
    """A buffer at least twice the L2 size; writing it evicts earlier data from L2."""
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    buf = torch.empty(max(2 * l2, 1 << 28) // 4, dtype=torch.float32, device="cuda")
    return lambda: buf.fill_(1.0)


def run_speculative(torch, R, calls=64, distinct=16, T=None):
    """Speculative verify on the tiny layer's shape at batch 512, T = 4 (or T), accept ~ U{0..T}:
    ReplaySSM verify + commit against snapshot-per-draft verify + commit, and against one
    conventional decode step of the same shape; L2 is flushed before every timed call."""
    w = SPEC
    T, L = T or w["T"], w["L"]
    shape = sg.LayerShape(w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"], w["dtype"])
    A, D = sg.head_params(w["nheads"], 0)
    cfg = R.ReplayConfig(w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"], L, T,
                         R.REPLAY_F32, R.REPLAY_RC_NONE)
    st = R.ReplayStore(cfg, torch.from_numpy(A), torch.from_numpy(D))
    drafts = []
    for c in range(distinct):
        d = sg.draft_inputs(shape, 0, c, T)
        drafts.append([torch.from_numpy(d[k].store).cuda() for k in ("x", "B", "C", "dt")])
    accepts = [torch.from_numpy(sg.accept_lengths(w["batch"], T, 0, c)).cuda() for c in range(calls)]
    y = torch.empty(w["batch"], T, w["nheads"], w["headdim"], device="cuda")
    snaps = torch.zeros(w["batch"], T + 1, w["nheads"], w["headdim"], w["dstate"], device="cuda")
    cur = torch.zeros(w["batch"], dtype=torch.int32, device="cuda")
    state = torch.zeros(w["batch"], w["nheads"], w["headdim"], w["dstate"], device="cuda")
    y1 = torch.empty(w["batch"], w["nheads"], w["headdim"], device="cuda")
    first = [[t[:, 0].contiguous() for t in dr] for dr in drafts]
    flush = l2_flusher(torch)

    def timed(fn):
        ts = []
        for c in range(calls):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn(c)
            e1.record()
            ts.append((e0, e1))
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in ts])) * 1e3

    def replay(c):
        st.verify(T, *drafts[c % distinct], y)
        st.commit(accepts[c])

    def snapshot(c):
        R.conv_verify_snapshot(cfg, T, snaps, cur, st.A, st.D, *drafts[c % distinct], y)
        R.conv_commit(w["batch"], T, cur, accepts[c])

    def standard(c):
        R.conv_step(cfg, state, R.REPLAY_F32, st.A, st.D, *first[c % distinct], y1)

    for fn in (replay, snapshot, standard):
        fn(0)
    r_us, s_us, c_us = timed(replay), timed(snapshot), timed(standard)
    assert st.status() == 0
    st.close()
    return {"workload": f"tiny-layer shape at batch 512, 8 heads, T={T}, accept ~ U{{0..{T}}}, L2 flushed per call",
            "replay_verify_commit_us": r_us, "snapshot_verify_commit_us": s_us,
            "conventional_step_us": c_us, "replay_speedup_vs_snapshot": s_us / r_us,
            "snapshot_vs_standard_step": s_us / c_us, "replay_vs_standard_step": r_us / c_us,
            "calls": calls}


def run_read_copies(torch, R, dev, steps=10):
    """The headline window with a bf16, E4M3, FP16 or NVFP4 read copy of the FP32 checkpoint,
    with a shared bf16, E4M3, FP16 (stochastically rounded) or NVFP4 checkpoint, and with an
    FP16 stochastically rounded checkpoint beside an NVFP4 read copy."""
    w = WORKLOAD
    L = w["L"]
    A, D = sg.head_params(w["nheads"], 0)
    y = torch.empty(w["batch"], w["nheads"], w["headdim"], device="cuda")
    out = {}
    for name, rc, fmt, shared, ckpt in (
            ("bf16", R.REPLAY_RC_BF16, "bf16", 0, 0), ("e4m3", R.REPLAY_RC_FP8E4M3, "e4m3", 0, 0),
            ("fp16", R.REPLAY_RC_FP16, "fp16", 0, 0), ("nvfp4", R.REPLAY_RC_NVFP4, "nvfp4", 0, 0),
            ("shared_bf16", R.REPLAY_RC_BF16, "bf16", 1, 0), ("shared_e4m3", R.REPLAY_RC_FP8E4M3, "e4m3", 1, 0),
            ("shared_fp16_sr", R.REPLAY_RC_FP16, "fp16", 1, 0), ("shared_nvfp4", R.REPLAY_RC_NVFP4, "nvfp4", 1, 0),
            ("fp16_sr_ckpt_nvfp4", R.REPLAY_RC_NVFP4, "nvfp4", 0, R.REPLAY_CKPT_F16_SR)):
        rcb, slab_scale = RC_BYTES[fmt]
        cfg = R.ReplayConfig(w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"], L, 0,
                             R.REPLAY_BF16, rc, shared, ckpt)
        st = R.ReplayStore(cfg, torch.from_numpy(A), torch.from_numpy(D))
        for _ in range(2):
            for t in range(L):
                st.step(*dev[t], y)
        # whole windows, nothing between the steps; then per-call durations with events
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        w0.record()
        for k in range(steps):
            for t in range(L):
                st.step(*dev[t], y)
        w1.record()
        torch.cuda.synchronize()
        window_us = w0.elapsed_time(w1) * 1e3 / steps
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps * L)]
        torch.cuda.synchronize()
        for k in range(steps):
            for t in range(L):
                ev[k * L + t][0].record()
                st.step(*dev[t], y)
                ev[k * L + t][1].record()
        torch.cuda.synchronize()
        us = np.array([a.elapsed_time(b) for a, b in ev]).reshape(steps, L) * 1e3
        nf_bytes = sum(step_bytes(w, t, False, rc_bytes=rcb, slab_scale=slab_scale) for t in range(L - 1))
        fl_bytes = step_bytes(w, L - 1, True, rc_bytes=rcb, shared=bool(shared), slab_scale=slab_scale,
                              state_bytes=2 if ckpt else 4)
        # back to back in a window the next call's prep overlaps this call's kernel, which an
        # event pair around each call prevents: the window's non-flush calls on average
        nf_window_us = (window_us - float(us[:, -1].mean())) / (L - 1)
        out[name] = {"tokens_per_s": w["batch"] * L / (window_us * 1e-6),
                     "window_us": window_us,
                     "nonflush_launch_us": float(us[:, :-1].mean()),
                     "flush_launch_us": float(us[:, -1].mean()),
                     "nonflush_us_in_window": nf_window_us,
                     "nonflush_achieved_gbs": nf_bytes / (us[:, :-1].sum(axis=1).mean() * 1e-6) / 1e9,
                     "nonflush_achieved_gbs_in_window": nf_bytes / ((L - 1) * nf_window_us * 1e-6) / 1e9,
                     "flush_achieved_gbs": fl_bytes / (us[:, -1].mean() * 1e-6) / 1e9}
        assert st.status() == 0
        st.close()
        del st
    return out


def run_sweep(torch, R, tokens=512, distinct=32, batches=(1, 16, 64, 256, 512), windows=(4, 8, 16, 32)):
    """Batch x window sweep on the tiny layer's shape (8 heads, FP32 inputs), replay vs the
    conventional step, L2 flushed before every token (each token timed alone), plus a
    40-layer stack at batch 256 (2.5 GiB of state, no flush needed). One JSON line each."""
    out = []
    shape_of = lambda b: sg.LayerShape(b, 8, 64, 128, 1, "f32")  # noqa: E731
    A, D = sg.head_params(8, 0)
    flush = l2_flusher(torch)

    def inputs(b):
        d = sg.token_inputs(shape_of(b), 0, np.arange(distinct))
        return [[torch.from_numpy(np.ascontiguousarray(d[k].store[:, t])).cuda() for k in ("x", "B", "C", "dt")]
                for t in range(distinct)]

    def per_token_us(fn, n):
        ev = []
        for t in range(n):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn(t)
            e1.record()
            ev.append((e0, e1))
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in ev])) * 1e3

    for b in batches:
        ins = inputs(b)
        y = torch.empty(b, 8, 64, device="cuda")
        state = torch.zeros(b, 8, 64, 128, device="cuda")
        cfg0 = R.ReplayConfig(b, 8, 64, 128, 1, 16, 0, R.REPLAY_F32, R.REPLAY_RC_NONE)
        Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
        conv = lambda t: R.conv_step(cfg0, state, R.REPLAY_F32, Ad, Dd, *ins[t % distinct], y)  # noqa: E731
        conv(0)
        c_us = per_token_us(conv, tokens)
        for L in windows:
            cfg = R.ReplayConfig(b, 8, 64, 128, 1, L, 0, R.REPLAY_F32, R.REPLAY_RC_NONE)
            st = R.ReplayStore(cfg, torch.from_numpy(A), torch.from_numpy(D))
            step = lambda t: st.step(*ins[t % distinct], y)  # noqa: E731
            for t in range(L):
                step(t)
            r_us = per_token_us(step, tokens)
            assert st.status() == 0
            st.close()
            out.append({"sweep": "tiny-layer shape, L2 flushed per token", "batch": b, "window_L": L,
                        "tokens": tokens, "replay_us_per_token": r_us, "conv_us_per_token": c_us,
                        "replay_tokens_per_s": b / (r_us * 1e-6), "conv_tokens_per_s": b / (c_us * 1e-6),
                        "speedup": c_us / r_us})
    # 40 independent layers at batch 256: every token runs all 40 layers' steps
    b, layers, L = 256, 40, 16
    ins = inputs(b)
    y = torch.empty(b, 8, 64, device="cuda")
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    cfg = R.ReplayConfig(b, 8, 64, 128, 1, L, 0, R.REPLAY_F32, R.REPLAY_RC_NONE)
    stores = [R.ReplayStore(cfg, Ad, Dd) for _ in range(layers)]
    states = [torch.zeros(b, 8, 64, 128, device="cuda") for _ in range(layers)]

    def timed_stack(fn, n):
        for t in range(L):
            fn(t)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for t in range(n):
            fn(t)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / n

    r_stack = timed_stack(lambda t: [s.step(*ins[t % distinct], y) for s in stores], 64)
    c_stack = timed_stack(lambda t: [R.conv_step(cfg, s, R.REPLAY_F32, Ad, Dd, *ins[t % distinct], y)
                                     for s in states], 64)
    # The same stack with every token's 40 layer steps replayed from a CUDA graph (one graph per
    # window position for the replay arm, whose kernels depend on the position; one per token
    # of the window for the conventional arm), so the host's launch rate no longer bounds it.
    r_graphs, c_graphs = [], []
    for t in range(L):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for s in stores:
                s.step(*ins[t % distinct], y)
        r_graphs.append(g)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for s in states:
                R.conv_step(cfg, s, R.REPLAY_F32, Ad, Dd, *ins[t % distinct], y)
        c_graphs.append(g)
    r_graph = timed_stack(lambda t: r_graphs[t % L].replay(), 64)
    c_graph = timed_stack(lambda t: c_graphs[t % L].replay(), 64)
    layer_bytes = sum(step_bytes(dict(batch=b, nheads=8, headdim=64, dstate=128, ngroups=1), t, t == L - 1, esz=4)
                      for t in range(L)) / L
    for s in stores:
        assert s.status() == 0
        s.close()
    out.append({"sweep": "40-layer stack, tiny-layer shape, batch 256, L 16 (2.5 GiB of state)",
                "replay_us_per_token_all_layers": r_stack, "conv_us_per_token_all_layers": c_stack,
                "replay_tokens_per_s": b / (r_stack * 1e-6), "conv_tokens_per_s": b / (c_stack * 1e-6),
                "speedup": c_stack / r_stack,
                "graph_replay_us_per_token": r_graph, "graph_conv_us_per_token": c_graph,
                "graph_speedup": c_graph / r_graph,
                "graph_replay_achieved_gbs": layers * layer_bytes / (r_graph * 1e-6) / 1e9,
                "graph_conv_achieved_gbs": layers * conv_bytes(dict(batch=b, nheads=8, headdim=64, dstate=128,
                                                                     ngroups=1), esz=4) / (c_graph * 1e-6) / 1e9})
    return out


# ------------------------------------------------------------------ the oracle (CPU)
def oracle_tokens_per_s(n_seqs: int, n_tokens: int, seed: int = 0):
    """Time the FP64 oracle decoding n_tokens of n_seqs sequences of the workload (all
    heads); inputs are drawn before the clock starts."""
    from oracle.mamba2 import Mamba2Decoder
    w = WORKLOAD
    shape = sg.LayerShape(w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"], w["dtype"])
    A, D = sg.head_params(w["nheads"], 0)
    seqs = np.arange(n_seqs)
    d = sg.token_inputs(shape, seed, np.arange(n_tokens), seqs)
    orc = Mamba2Decoder(A.astype(np.float64), D.astype(np.float64), w["ngroups"],
                        np.zeros((n_seqs, w["nheads"], w["headdim"], w["dstate"])))
    t0 = time.perf_counter()
    for t in range(n_tokens):
        orc.step(d["x"].f64[:, t], d["B"].f64[:, t], d["C"].f64[:, t], d["dt"].f64[:, t])
    return n_seqs * n_tokens / (time.perf_counter() - t0)


def _oracle_worker(job):
    """One process of the all-cores oracle run: decode its own sequences, report its span."""
    first, n_seqs, n_tokens = job
    from oracle.mamba2 import Mamba2Decoder
    w = WORKLOAD
    shape = sg.LayerShape(w["batch"], w["nheads"], w["headdim"], w["dstate"], w["ngroups"], w["dtype"])
    A, D = sg.head_params(w["nheads"], 0)
    d = sg.token_inputs(shape, 0, np.arange(n_tokens), np.arange(first, first + n_seqs))
    orc = Mamba2Decoder(A.astype(np.float64), D.astype(np.float64), w["ngroups"],
                        np.zeros((n_seqs, w["nheads"], w["headdim"], w["dstate"])))
    t0 = time.time()
    for t in range(n_tokens):
        orc.step(d["x"].f64[:, t], d["B"].f64[:, t], d["C"].f64[:, t], d["dt"].f64[:, t])
    return t0, time.time(), n_seqs * n_tokens


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_all_cores(cores, seqs_per_core, n_tokens):
    """The oracle on every host core: one process per core, each decoding its own sequences
    (the (sequence, head) units are independent). Processes are spawned, not forked (the
    parent holds a CUDA context), with one BLAS/OpenMP thread each. Tokens over the span from
    the first process's start to the last one's end."""
    import multiprocessing as mp
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    jobs = [((c * seqs_per_core) % WORKLOAD["batch"], seqs_per_core, n_tokens) for c in range(cores)]
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_oracle_worker, jobs, chunksize=1)
    return sum(r[2] for r in res) / (max(r[1] for r in res) - min(r[0] for r in res))


def cpu_baseline(n_seqs, n_tokens):
    one = oracle_tokens_per_s(n_seqs, n_tokens)
    cores = host_cores()
    per_core = max(1, n_seqs // 2)
    try:
        allc = oracle_all_cores(cores, per_core, n_tokens)
    except Exception as e:  # noqa: BLE001 -- the baseline is reported, never the product
        allc, cores = None, 1
        print(f"all-cores oracle run failed: {e!r}", file=sys.stderr)
    value = allc if allc is not None else one
    return {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
            "one_thread_value": one, "all_cores_value": allc, "host_cores": host_cores(),
            "sample": (f"one thread: {n_seqs} of 256 sequences x {n_tokens} tokens; all cores: {cores} "
                       f"processes x {per_core} sequences x {n_tokens} tokens; all 128 heads, numpy FP64")}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    for _ in range(args.warmup):
        oracle_tokens_per_s(1, 2)
    t0 = time.perf_counter()
    n_seqs, n_tokens = 2, 4
    for _ in range(args.steps):
        oracle_tokens_per_s(n_seqs, n_tokens, seed=1)
    el = time.perf_counter() - t0
    v = args.steps * n_seqs * n_tokens / el
    sample = f"per step {n_seqs} sequences x {n_tokens} tokens, all 128 heads (numpy FP64, one thread)"
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "Nemotron-shaped Mamba-2 layer decode, FP64 oracle on host cores",
                       "batch_per_gpu": WORKLOAD["batch"], "window_L": WORKLOAD["L"]},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="replayssm", choices=["replayssm", "reference"])
    ap.add_argument("--cpu-sample-seqs", type=int, default=8)
    ap.add_argument("--cpu-sample-tokens", type=int, default=48)
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the secondary workloads (read copies, speculative verify)")
    ap.add_argument("--read-copy", default="none", choices=["none", "bf16", "e4m3", "fp16", "nvfp4"],
                    help="diagnostics: give the timed store this read copy (the benchmark line is 'none')")
    ap.add_argument("--shared-checkpoint", action="store_true",
                    help="diagnostics: the read copy is the checkpoint (needs --read-copy)")
    ap.add_argument("--fp16-checkpoint", action="store_true",
                    help="diagnostics: keep the checkpoint in FP16 with stochastic rounding (needs --read-copy)")
    ap.add_argument("--batch", type=int, default=0,
                    help="diagnostics with --kernels-only: sequences per GPU (default: the workload's 256)")
    ap.add_argument("--kernels-only", action="store_true",
                    help="diagnostics: time only the replay windows and print a short line (for ncu runs)")
    ap.add_argument("--verify-only", action="store_true",
                    help="diagnostics: run only the speculative verify workload and print its line")
    ap.add_argument("--drafts", type=int, default=0,
                    help="diagnostics with --verify-only: draft count T (default 4)")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the benchmark line: batch x window sweep and 40-layer stack, "
                         "one JSON line per configuration")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)      # at least 3 untimed warm-up steps
    rank, world, local_rank = dist_env()
    if args.sweep or args.verify_only:
        import torch
        from hybrid_model_ssm_mamba_gb300 import replay as R
        torch.cuda.set_device(local_rank)
        lines = run_sweep(torch, R) if args.sweep else [run_speculative(torch, R, calls=args.steps, T=args.drafts)]
        for line in lines:
            print(json.dumps(line), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_replay(args, rank, world, local_rank)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
