"""Benchmark: attention-backward TFLOP/s on one GB300 (and % of dense-BF16 peak).

One step = one whole backward (attn_bwd_preprocess + attn_bwd) over the
GQA 4:1 causal workload (B=2, Hq=16, Hk=4, Sq=Sk=1024, D=128, bf16 N(0,1)
inputs, seed 1) with inputs resident in HBM. FLOPs counted: 10 * B * Hq * D *
(live (i, j) entries per (b, h)). The whole working set is smaller than L2,
so L2 is flushed (a 256 MiB write, then a 256 MiB read that forces the
flush's dirty lines out) between timed steps, outside the timed events. O and LSE inputs come from the library's own forward.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]

Under torchrun each rank runs an independent copy of the workload on its GPU
(weak scaling, no data-path collective); value = all ranks' FLOPs / the
slowest rank's time. --impl reference times the float64 CPU oracle on a
bounded sample of the same workload on the host cores.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import WORKLOADS, make_workload  # noqa: E402

METRIC = "attention-backward TFLOP/s on 1 GB300 and % of dense-BF16 tensor peak"
DEFAULT_WORKLOAD = "gqa4_causal_s1024_d128"
L2_FLUSH_BYTES = 256 << 20


def live_entries(w) -> int:
    """Live (i, j) pairs per (batch, head) under the workload's mask."""
    if w.__class__.__name__ == "SparseWorkload":
        pos = (w.n_ori - w.Sq) + np.arange(w.Sq)
        lo = np.maximum(pos - w.ori_win_left if w.ori_win_left >= 0 else 0, 0)
        hi = np.minimum(pos + w.ori_win_right if w.ori_win_right >= 0 else w.n_ori - 1,
                        w.n_ori - 1)
        ori = int(np.maximum(hi - lo + 1, 0).sum())
        cmp = int((w.cmp_idx[:, 0, :] >= 0).sum()) if w.cmp_idx is not None else 0
        return ori + cmp
    i = np.arange(w.Sq)[:, None]
    j = np.arange(w.Sk)[None, :]
    inside = np.ones((w.Sq, w.Sk), dtype=bool)
    if w.window_left >= 0:
        inside &= j >= i - w.window_left
    if w.window_right >= 0:
        inside &= j <= i + w.window_right
    return int((inside | (j < w.num_sink)).sum())


def flops_of(w) -> float:
    B = getattr(w, "B", 1)
    return 10.0 * B * w.Hq * w.D * live_entries(w)


def algorithmic_bytes(w) -> float:
    """Each input read once and each output written once (bf16 in, fp32 out)."""
    if w.__class__.__name__ == "SparseWorkload":
        n = w.Sq * w.Hq * w.D
        kv = (w.n_ori + w.n_cmp) * w.Hk * w.D
        return 2 * 3 * n + 2 * kv + 4 * n + 4 * kv + 8 * w.Sq * w.Hq + 4 * w.cmp_idx.size
    nq = w.B * w.Sq * w.Hq * w.D
    nk = w.B * w.Sk * w.Hk * w.D
    b = 2 * (3 * nq + 2 * nk) + 4 * nq + 4 * 2 * nk + 8 * w.B * w.Hq * w.Sq
    if w.bias is not None:
        b += 4 * w.bias.size
    if w.want_dbias:
        b += 4 * w.Hq * w.Sq * w.Sk
    return float(b)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background during timing."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def reduce_max(values, device):
    """Element-wise max of a list of floats over all ranks (any backend)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def overrides_of(args):
    out = {}
    for kv in args.override:
        key, _, val = kv.partition("=")
        out[key] = int(val)
    return out


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_ours(args):
    import torch
    import torch.distributed as dist
    import attention_backward_attn_gb300 as ab

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = make_workload(args.workload, **overrides_of(args))
    sparse = w.__class__.__name__ == "SparseWorkload"

    def up_bf16(x):
        return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev).to(torch.bfloat16)

    # ---- inputs resident in HBM; O / LSE from the library forward ----
    if sparse:
        q, do = up_bf16(w.q[None]), up_bf16(w.do[None])
        okv = up_bf16(w.ori_kv)
        ckv = up_bf16(w.cmp_kv) if w.cmp_kv is not None else None
        idx = torch.from_numpy(w.cmp_idx).to(dev) if w.cmp_idx is not None else None
        o = torch.empty_like(q)
        lse = torch.empty((1, w.Hq, w.Sq), dtype=torch.float32, device=dev)
        sp = ab.sparse_from(okv, ckv, idx, w.ori_win_left, w.ori_win_right)
        prob = ab.problem_from(q, None, None, o, do, w.scale, Sk=0, Hk=w.Hk)
        ab.attn_fwd_lse(prob, None, sp, q, None, None, None, o, lse)
        plan = ab.BackwardPlan(q, None, None, o, do, lse, w.scale, ori_kv=okv, cmp_kv=ckv,
                               cmp_idx=idx, ori_win_left=w.ori_win_left,
                               ori_win_right=w.ori_win_right, deterministic=args.deterministic)
        bias = None
    else:
        q, k, v, do = (up_bf16(x) for x in (w.q, w.k, w.v, w.do))
        bias = (torch.from_numpy(w.bias).to(dev) if w.bias is not None else None)
        mask = ab.mask_from(w.window_left, w.window_right, w.num_sink)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
        prob = ab.problem_from(q, k, v, o, do, w.scale)
        ab.attn_fwd_lse(prob, mask, None, q, k, v, bias, o, lse)
        plan = ab.BackwardPlan(q, k, v, o, do, lse, w.scale, mask=mask, bias=bias,
                               want_dbias=w.want_dbias, deterministic=args.deterministic)
    torch.cuda.synchronize()

    def second_plan():
        # a second set of per-step buffers (inputs, gradients, workspace) for
        # the pipelined end-to-end leg; read-only tensors (bias, the sparse KV
        # rows and indices) are shared
        if sparse:
            return ab.BackwardPlan(q.clone(), None, None, o.clone(), do.clone(), lse.clone(),
                                   w.scale, ori_kv=okv, cmp_kv=ckv, cmp_idx=idx,
                                   ori_win_left=w.ori_win_left, ori_win_right=w.ori_win_right,
                                   deterministic=args.deterministic)
        return ab.BackwardPlan(q.clone(), k.clone(), v.clone(), o.clone(), do.clone(),
                               lse.clone(), w.scale, mask=mask, bias=bias,
                               want_dbias=w.want_dbias, deterministic=args.deterministic)

    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    evict = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    scratch = torch.empty((), dtype=torch.float32, device=dev)
    flops = flops_of(w)

    # warm-up (also performs the one-time per-kernel set-up before any capture)
    for _ in range(args.warmup):
        plan.run()
    torch.cuda.synchronize()
    code, detail = plan.device_status()
    if code != 0:
        raise RuntimeError(f"device status {ab.status_string(code)} ({detail})")

    # The two C-ABI calls of a step, captured once into CUDA graphs and replayed
    # per step, so that host-side enqueue time (ctypes, tensor-map encoding)
    # never shows up as GPU idle time inside the timed events.
    def call_pre():
        ab.attn_bwd_preprocess(plan.prob, plan.sparse, plan.q, plan.k, plan.v, plan.o, plan.do,
                               plan.delta, plan.dbias, plan.dk, plan.dv, plan.workspace,
                               plan.ws_bytes)

    def call_bwd():
        ab.attn_bwd(plan.prob, plan.mask, plan.sparse, plan.q, plan.k, plan.v, plan.do,
                    plan.lse, plan.delta, plan.bias, plan.dq, plan.dk, plan.dv, plan.dbias,
                    plan.workspace, plan.ws_bytes)

    # g_step is the timed step (the backward kernel is launched as a programmatic
    # dependent of the pre-pass, so it may start its set-up while the pre-pass
    # drains); g_pre / g_bwd time the backward call on its own.
    g_step, g_pre, g_bwd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        call_pre()
        call_bwd()
    with torch.cuda.graph(g_pre):
        call_pre()
    with torch.cuda.graph(g_bwd):
        call_bwd()
    for _ in range(args.warmup):
        g_step.replay()
        g_pre.replay()
        g_bwd.replay()
    torch.cuda.synchronize()

    def flush_l2(s):
        # L2 flush (not timed): write a buffer larger than L2, then read another
        # one so that the flush's own dirty lines are written back before the
        # step starts instead of inside it
        flush.fill_(float(s))
        torch.sum(evict, dim=0, out=scratch)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    bends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for s in range(args.steps):
        flush_l2(s)
        starts[s].record(stream)
        g_step.replay()
        ends[s].record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    # the backward call alone (after an untimed pre-pass), for the roofline
    for s in range(args.steps):
        flush_l2(s)
        g_pre.replay()
        mids[s].record(stream)
        g_bwd.replay()
        bends[s].record(stream)
    torch.cuda.synchronize()
    time.sleep(0.2)
    clocks = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    bwd_ms = [a.elapsed_time(b) for a, b in zip(mids, bends)]
    code, detail = plan.device_status()
    if code != 0:
        raise RuntimeError(f"device status {ab.status_string(code)} ({detail})")

    total_ms = float(sum(step_ms))
    mean_bwd_ms = float(sum(bwd_ms) / len(bwd_ms))
    # slowest rank defines the job's time (weak scaling: every rank ran a replica)
    total_ms, mean_bwd_ms = reduce_max([total_ms, mean_bwd_ms], dev)

    # ---- end to end through the public API: pinned host in, result out ----
    e2e = run_e2e(args, ab, plan, second_plan(), sparse, flops)

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    peaks, peaks_src = measured_peaks()
    path = "tcgen05" if plan.path == 1 else "simt"
    # kernels per step: the fused pre-pass, then one tcgen05 kernel (key-major and
    # query-major CTAs in one launch) or two SIMT kernels
    if path == "tcgen05":
        roof = {"bound": "tensor", "achieved": flops / (mean_bwd_ms * 1e-3) / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
        launches_per_step = 2
        if args.deterministic and sparse:
            launches_per_step = 4  # + compressed-row slot table + ordered row sums
        elif args.deterministic and w.want_dbias and w.B > 1:
            launches_per_step = 3  # + the batch-ordered sum of the per-batch dbias slices
    else:
        roof = {"bound": "alu", "achieved": flops / (mean_bwd_ms * 1e-3) / 1e12,
                "peak": SIMT_FP32_PEAK_TFLOPS, "unit": "TFLOP/s"}
        launches_per_step = 3
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = (NCU_TRAFFIC.get(args.workload)
                       if not overrides_of(args) and not args.deterministic else None)
    roof["peak_source"] = peaks_src
    roof["kernel"] = "attn_bwd (" + path + ")"
    value = ws * flops * args.steps / (total_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16" if path == "tcgen05" else "f32",
        "data": "synthetic (seeded bf16 N(0,1); O/LSE from the library forward)",
        "config": {"workload": args.workload, "overrides": overrides_of(args) or None,
                   "flops_per_step": flops,
                   "algorithmic_bytes_per_step": algorithmic_bytes(w),
                   "path": path, "deterministic": bool(args.deterministic), "l2": "flushed between steps (256 MiB write + 256 MiB read, untimed)",
                   "launch": "attn_bwd_preprocess + attn_bwd captured once into one CUDA graph (the backward a programmatic dependent of the pre-pass), replayed per step",
                   "parallelism": f"replicas x{ws}"},
        "pct_of_peak": round(100.0 * value / ws / peaks["bf16_tflops"], 2),
        "bwd_only_ms": round(mean_bwd_ms, 5),
        "roofline": roof,
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
        "e2e": e2e,
        "wall_s": round(wall, 3),
    }
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    print(json.dumps(line))
    if ws > 1:
        dist.destroy_process_group()


# dram__bytes_read.sum + dram__bytes_write.sum of the dominant kernel, per launch, from
# the ncu captures summarised in profiles/. Three are smaller captures scaled to the full
# launch by the units processed, since their DRAM bytes grow in proportion: the sparse
# one has 1024 of the 4096 tokens (Q, dO, dQ are linear in Sq), the ALiBi one 8 of the 16
# heads (every tensor is per head), the windowed one S = 4096 of 8192 (fixed window: live
# entries, CTAs and bytes linear in S). An entry goes back to None when its kernel changes.
NCU_TRAFFIC = {
    "gqa4_causal_s1024_d128": 25.5168e6 + 12.288e3,
    "mha_alibi_dbias_s2048_d64": 2 * (366.990336e6 + 176.617728e6),
    "gqa4_window1024_sink4_s8192_d128": 2 * (158.30016e6 + 66.37824e6),
    "sparse_scfa_s4096_h64_d512": 4 * (140.928e6 + 82.918912e6),
}

# CUDA-core fp32 FMA rate for the SIMT fallback's roofline: 152 SMs x 128
# FP32 lanes x 2 FLOP x 2.07 GHz.
SIMT_FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def run_e2e(args, ab, plan, second_plan, sparse, flops):
    """Same metric through the public API, with per-step H2D of the inputs from
    pinned host memory and D2H of the gradients inside the timed region.

    Steps run as a pipeline over two sets of device buffers (two plans): the
    H2D copies of step k, the backward of step k - 1 and the D2H copies of
    step k - 2 overlap on three streams, ordered by events (a slot's inputs
    are overwritten only after its previous backward read them, its outputs
    only after they were copied out)."""
    import torch

    def ins_of(pl):
        return [pl.q, pl.o, pl.do, pl.lse] + ([] if sparse else [pl.k, pl.v])

    def outs_of(pl):
        o = [pl.dq] + ([pl.d_ori] + ([pl.d_cmp] if pl.d_cmp is not None else [])
                       if sparse else [pl.dk, pl.dv])
        return o + ([pl.dbias] if pl.dbias is not None else [])

    plans = [plan, second_plan]
    h_in = [t.cpu().pin_memory() for t in ins_of(plan)]
    h_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs_of(plan)]
             for _ in range(2)]
    s_in, s_cp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "cp", "out")}

    def step(k):
        sl = k & 1
        pl = plans[sl]
        if k >= 2:
            s_in.wait_event(ev["cp"][sl])   # the slot's inputs were read by step k - 2
        with torch.cuda.stream(s_in):
            for h, d in zip(h_in, ins_of(pl)):
                d.copy_(h, non_blocking=True)
        ev["in"][sl].record(s_in)
        s_cp.wait_event(ev["in"][sl])
        if k >= 2:
            s_cp.wait_event(ev["out"][sl])  # the slot's outputs of step k - 2 were copied out
        pl.run(stream=s_cp)
        ev["cp"][sl].record(s_cp)
        s_out.wait_event(ev["cp"][sl])
        with torch.cuda.stream(s_out):
            for h, d in zip(h_out[sl], outs_of(pl)):
                h.copy_(d, non_blocking=True)
        ev["out"][sl].record(s_out)

    steps = max(3, min(args.steps, 20))
    for k in range(4):
        step(k)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for k in range(steps):
        step(k)
    s_in.wait_stream(s_out)  # the last D2H is inside the timed region
    b.record(s_in)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return {"value": round(flops / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in ins_of(plan))),
            "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in outs_of(plan))),
            "ms_per_step": round(ms, 5),
            "pipeline": "2 buffer slots; H2D, backward and D2H of consecutive steps overlap"}


# ------------------------------------------------------ CPU oracle legs ----

def _oracle_sample(w):
    """A bounded sample of the workload for the float64 oracle: one batch and
    one KV-head group (dense), or the first Sq/16 tokens (sparse). Returns
    (callable, flops of the sample, description)."""
    import oracle
    from workloads import bf16_round
    if w.__class__.__name__ == "SparseWorkload":
        n = max(1, w.Sq // 16)
        q = np.asarray(w.q, np.float64)
        okv = np.asarray(w.ori_kv, np.float64)
        ckv = None if w.cmp_kv is None else np.asarray(w.cmp_kv, np.float64)
        # tokens of the sample sit at the end of the sequence (all windows full)
        sl = slice(w.Sq - n, w.Sq)
        idx = w.cmp_idx[sl] if w.cmp_idx is not None else None
        O, L = oracle.sparse_forward(q[sl], okv, ckv, idx, w.scale, w.ori_win_left, w.ori_win_right)
        O = bf16_round(O.astype(np.float32)).astype(np.float64)
        L = L.astype(np.float32).astype(np.float64)
        do = np.asarray(w.do[sl], np.float64)
        live = n * min(w.ori_win_left + 1, w.n_ori) + (int((idx[:, 0] >= 0).sum()) if idx is not None else 0)
        fl = 10.0 * w.Hq * w.D * live

        def fn():
            oracle.sparse_backward(q[sl], okv, ckv, idx, O, do, L, w.scale, w.ori_win_left,
                                   w.ori_win_right)
        return fn, fl, f"last {n} of {w.Sq} tokens, all {w.Hq} heads"
    r = w.Hq // w.Hk
    tr = lambda x: np.ascontiguousarray(np.asarray(x, np.float64).transpose(0, 2, 1, 3))
    Q, K, V, dO = tr(w.q[:1, :, :r]), tr(w.k[:1, :, :1]), tr(w.v[:1, :, :1]), tr(w.do[:1, :, :r])
    m = None
    if w.window_left >= 0 or w.window_right >= 0 or w.num_sink:
        m = oracle.live_mask(w.Sq, w.Sk, w.window_left, w.window_right, w.num_sink)
    bias = None if w.bias is None else w.bias[:r].astype(np.float64)
    O, L = oracle.forward(Q, K, V, w.scale, m, bias)
    O = bf16_round(O.astype(np.float32)).astype(np.float64)
    L = L.astype(np.float32).astype(np.float64)
    fl = 10.0 * r * w.D * live_entries(w)

    def fn():
        oracle.backward(Q, K, V, O, dO, L, w.scale, m, bias)
    return fn, fl, f"batch 0, KV head 0 with its {r} query heads (1/{w.B * w.Hk} of the workload)"


def _cores():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def cpu_baseline(w, budget_s=20.0):
    fn, fl, desc = _oracle_sample(w)
    fn()  # warm
    t0 = time.perf_counter()
    reps = 0
    while True:
        fn()
        reps += 1
        if time.perf_counter() - t0 > budget_s or reps >= 50:
            break
    dt = (time.perf_counter() - t0) / reps
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": _cores(),
            "kind": "oracle", "sample": f"{desc}; {reps} reps, {dt:.3f} s each"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    w = make_workload(args.workload)
    fn, fl, desc = _oracle_sample(w)
    for _ in range(args.warmup):
        fn()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn()
    dt = (time.perf_counter() - t0) / args.steps
    value = fl / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded bf16 N(0,1))",
        "config": {"workload": args.workload, "sample": desc},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": _cores(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--deterministic", action="store_true",
                    help="time the bitwise-reproducible mode (ATTN_FLAG_DETERMINISTIC)")
    ap.add_argument("--override", nargs="*", default=[], metavar="KEY=INT",
                    help="shrink the workload (e.g. Sq=1024 n_ori=1024 n_cmp=256) for a "
                         "profiler capture; the JSON line then records the overrides")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
