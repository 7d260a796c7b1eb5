"""Benchmark of the MoE-layer forward (moe_forward) on GB300.

One step = one full forward of the layer over one batch of synthetic tokens:
router -> grouping -> gate/up GEMM (rows gathered in-kernel) + SwiGLU -> down GEMM + routing
weight -> combine, i.e. every kernel moe_forward launches. Default workload: the
Mixtral-shaped layer (T=4096, d=4096, E=8, K=2, n=14336, bf16, fp32 accumulate).

Prints ONE JSON line on rank 0:
  value       useful TFLOP/s (2*T*K*3*d*n per step) of all ranks together, device
              timed with CUDA events around K forwards exactly as a user calls them
              (no events inside a step), inputs resident in HBM
  e2e         same metric from pinned host memory, host<->device copies of every
              step inside the timed region (moe_forward_host_stream: the copies of
              neighbouring batches overlap the layer)
  roofline    the dominant kernel (gate/up GEMM) against the measured bf16 peak; its
              duration comes from a second region of K forwards right after the
              timed one, with an event between every two stages
  gpu_launches  kernels per step x K, as the library counts them (moe_forward_launches:
              6 on the Mixtral-shaped layer with its CTA-pair row gather, 5 on the tiny one)
  cpu_baseline  the CPU oracle on a bounded token sample (rank 0, N=1 only)
  clocks      nvidia-smi SM clocks / throttle reasons sampled during the timed region
  extra       tokens/s, per-stage times (from the second region), router and combine
              GB/s, % of peak, routing statistics (tile padding, rows per expert), and
              `sustained`: back-to-back forwards over about 2 s against the sustained
              bf16 peak (the K-step `value` is a burst figure), and `backward`: the
              layer's backward (pre-activations, dH with dS, dX, weight gradients,
              router) timed per call after the forward regions (--no-backward skips it)

--routing rounded runs the layer under Token Rounding (moe_forward_rounded: each
expert's top-K count rounded to a multiple of the 128-row tile); its value
counts the rows the rounded routing computes, and extra.topk_rows_equiv_tflops
the top-K rows, T*K, over the same time.

--impl reference times the CPU oracle (the only reference this layer has) on the
same workload and metric. Under torchrun every rank runs its own replica (tokens
are independent: weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

STAGES = ["route", "permute", "gemm_gate_up", "gemm_down", "combine"]
# Token Rounding (--routing rounded): the grouping step is the rounding step
STAGES_ROUNDED = ["route", "round", "gemm_gate_up", "gemm_down", "combine"]
METRIC = "MoE layer fwd useful TFLOPS and % of GB300 BF16 tensor peak; router GB/s"
# ncu: dram__bytes_read.sum + dram__bytes_write.sum of one gate/up GEMM launch on
# the Mixtral-shaped workload (profiles/traffic_gemm_mixtral.md). Set back to None
# whenever the kernel changes, until it is captured again.
GEMM1_TRAFFIC_BYTES = {"mixtral": 2.341297e9 + 0.230692e9}


def workload_desc(name, c, routing="topk"):
    return (f"{name}-shaped MoE layer forward T={c['T']} d={c['d']} E={c['E']} K={c['K']} "
            f"n={c['n']}" + (" zipf-bias" if c.get("zipf") else "")
            + (" token-rounding M=128" if routing == "rounded" else ""))


def useful_flops(c, tokens=None):
    T = c["T"] if tokens is None else tokens
    return 2.0 * T * c["K"] * 3 * c["d"] * c["n"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm=j["hbm_gbs"], bf16=j["bf16_tflops"],
                    bf16_sustained=j.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        time.sleep(0.25)
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
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v == "Active"})
        mhz = sorted(r[0] for r in rows)
        loaded = [r for r in rows if r[2] > 250.0] or rows
        lm = sorted(r[0] for r in loaded)
        return {"sm_mhz": lm[len(lm) // 2], "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "sm_mhz_min": mhz[0],
                "power_w_max": max(r[2] for r in rows)}


def dist_setup():
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(value_per_rank_units: float, seconds_max: float, world: int) -> float:
    """Whole-job throughput: units every rank processed / slowest rank's time."""
    return value_per_rank_units * world / seconds_max


def oracle_sample_tflops(inp_np, c, tokens):
    """Time the CPU oracle (token-by-token definition) on `tokens`; TFLOP/s."""
    import oracle
    X, Wr, bias, W1, W3, W2 = inp_np
    t0 = time.perf_counter()
    oracle.forward_tokens(X, Wr, bias, W1, W3, W2, c["K"], tokens)
    dt = time.perf_counter() - t0
    return useful_flops(c, len(tokens)) / dt / 1e12, dt


def host_inputs(inp):
    from top_routing_grouped_02_gb300 import synth
    bias = inp["bias"]
    return (synth.bf16_bits(inp["X"]), inp["Wr"].cpu().numpy(),
            None if bias is None else bias.cpu().numpy(), synth.bf16_bits(inp["W1"]),
            synth.bf16_bits(inp["W3"]), synth.bf16_bits(inp["W2"]))


def calibrate_sample(inp_np, c, seconds: float, rng_seed=0):
    """Token count whose oracle run takes about `seconds`, and its TFLOP/s."""
    import numpy as np
    rng = np.random.default_rng(rng_seed)
    n = 4
    while True:
        toks = np.sort(rng.choice(c["T"], size=min(n, c["T"]), replace=False))
        tf, dt = oracle_sample_tflops(inp_np, c, toks)
        if dt >= seconds * 0.5 or n >= c["T"]:
            return n, tf, dt
        n = min(c["T"], max(n * 2, int(n * seconds / max(dt, 1e-3))))


def run_reference(args, c, world, rank):
    """The reference arm: the CPU oracle as it stands, on rank 0 only."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    from top_routing_grouped_02_gb300 import synth
    oracle.build()
    inp = synth.layer_inputs(device="cuda" if _has_cuda() else "cpu", **c)
    inp_np = host_inputs(inp)
    budget = 150.0 / max(1, args.steps + args.warmup)
    n, _, _ = calibrate_sample(inp_np, c, budget)
    rng = np.random.default_rng(1)
    for _ in range(args.warmup):
        toks = np.sort(rng.choice(c["T"], size=n, replace=False))
        oracle_sample_tflops(inp_np, c, toks)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        toks = np.sort(rng.choice(c["T"], size=n, replace=False))
        oracle.forward_tokens(*inp_np, c["K"], toks)
    dt = time.perf_counter() - t0
    value = useful_flops(c, n) * args.steps / dt / 1e12
    sample = f"{n} of {c['T']} tokens per step (token-by-token oracle, routing included)"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(args.workload, c), **{k: c[k] for k in "TdEKn"}},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _has_cuda():
    import torch
    return torch.cuda.is_available()


def measure_backward(args, c, inp, stream, dev):
    """The layer's backward (top-K choice held fixed) on the same inputs: the
    five calls a training step makes after the forward's routing and grouping,
    timed on the launch stream with an event between every two calls, over
    `args.steps` passes after 2 untimed ones. The routing and grouping are the
    forward's (computed once, outside the timed passes); dY is synthetic
    N(0,1). Returns the per-call times and each GEMM's rate against the bf16
    peak."""
    import numpy as np
    import torch
    from top_routing_grouped_02_gb300 import moe, synth

    T, d, E, K, n = c["T"], c["d"], c["E"], c["K"], c["n"]
    R = T * K
    ws = moe.workspace(T, d, E, K, n, dev)
    dY = synth.normal("dY", (T, d), 1.0, torch.bfloat16, dev, seed=args.seed + 7)
    names = ["gate_up_train", "dh", "dx", "dw", "router"]
    with torch.cuda.stream(stream):
        logits = torch.empty((T, E), dtype=torch.float32, device=dev)
        idx, w, counts = moe.moe_route(inp["X"], inp["Wr"], K, inp["bias"], logits=logits,
                                       stream=stream)
        g = moe.moe_permute(idx, E, counts=counts, ws=ws, stream=stream)
        scratch = torch.zeros(int(moe.lib().moe_backward_dw_scratch_bytes(T, d, E, K)),
                              dtype=torch.uint8, device=dev)
        wv = w.view(-1)

        def one_pass(ev=None):
            rec = (lambda j: ev[j].record(stream)) if ev is not None else (lambda j: None)
            rec(0)
            H, A1, A3 = moe.moe_gemm_gate_up_train(inp["X"], inp["W1"], inp["W3"],
                                                   g["perm_token"], g["offsets"], K, ws=ws,
                                                   stream=stream)
            rec(1)
            dA1, dA3, dS = moe.moe_backward_dh(dY, inp["W2"], A1, A3, wv, g["perm_token"],
                                               g["perm_slot"], g["offsets"], K, ws=ws,
                                               stream=stream)
            rec(2)
            dXg, _ = moe.moe_backward_dx(dA1, dA3, inp["W1"], inp["W3"], g["offsets"],
                                         g["row_of_slot"], K, ws=ws, stream=stream)
            rec(3)
            moe.moe_backward_dw(inp["X"], dY, H, dA1, dA3, wv, g["perm_token"], g["perm_slot"],
                                g["offsets"], K, scratch=scratch, stream=stream)
            rec(4)
            moe.moe_backward_router(inp["X"], inp["Wr"], logits, idx, dS, g["row_of_slot"], dXg,
                                    ws=ws, stream=stream)
            rec(5)

        for _ in range(2):
            one_pass()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
               for _ in range(args.steps)]
        torch.cuda.synchronize()
        for i in range(args.steps):
            one_pass(evs[i])
        torch.cuda.synchronize()
    st, word = moe.moe_sync_check(ws)
    if st != 0:
        raise RuntimeError(f"device error word {word:#x} in the backward region")
    st, word = moe.moe_sync_check(scratch)
    if st != 0:
        raise RuntimeError(f"device error word {word:#x} in the weight-gradient scratch")
    ms = {s: float(np.mean([evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps)]))
          for j, s in enumerate(names)}
    total = float(np.mean([evs[i][0].elapsed_time(evs[i][-1]) for i in range(args.steps)]))
    peak = load_peaks()["bf16"]
    gemm_flops = {"gate_up_train": 4.0 * R * d * n, "dh": 2.0 * R * d * n,
                  "dx": 4.0 * R * d * n, "dw": 6.0 * R * d * n}
    rates = {k: f / (ms[k] / 1e3) / 1e12 for k, f in gemm_flops.items()}
    # the router's share: X and dXg read, the fp32 router share of dX written
    # and read back, dX written (the dL, dWr, dbias terms are E-wide, small)
    router_bytes = T * d * 2 + R * d * 2 + 2 * T * d * 4 + T * d * 2
    useful = 12.0 * R * d * n  # dX and the weight gradients of both GEMMs
    return {
        "passes": args.steps, "ms_per_pass": round(total, 4),
        "stage_ms": {k: round(v, 4) for k, v in ms.items()},
        "gemm_tflops": {k: round(v, 2) for k, v in rates.items()},
        "gemm_frac_bf16_peak": {k: round(v / peak, 4) for k, v in rates.items()},
        "router_GBps": round(router_bytes / (ms["router"] / 1e3) / 1e9, 1),
        "useful_tflops": round(useful / (total / 1e3) / 1e12, 2),
        "useful_flops_per_pass": useful,
        "note": "gradients with the top-K choice fixed; the pass recomputes the gate/up "
                "pre-activations (4*R*d*n flops, counted in gemm_tflops, not in useful)",
    }


def run_gpu(args, c, world, rank, local):
    import numpy as np
    import torch
    from top_routing_grouped_02_gb300 import moe, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    T, d, E, K, n = c["T"], c["d"], c["E"], c["K"], c["n"]
    inp = synth.layer_inputs(device=dev, seed=args.seed + rank, **c)
    rounded = args.routing == "rounded"
    stages = STAGES_ROUNDED if rounded else STAGES
    ws = (moe.workspace_rounded if rounded else moe.workspace)(T, d, E, K, n, dev)
    Y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    row_map = torch.empty((T, E), dtype=torch.int32, device=dev) if rounded else None
    stream = torch.cuda.Stream(device=dev)  # a capturable (non-legacy) stream

    def step(events=None):
        if rounded:
            moe.moe_forward_rounded(inp["X"], inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K,
                                    inp["bias"], ws=ws, Y=Y, row_map=row_map, stream=stream,
                                    events=events)
        else:
            moe.moe_forward(inp["X"], inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K, inp["bias"],
                            ws=ws, Y=Y, stream=stream, events=events)

    for _ in range(args.warmup):
        step()
    st, word = moe.moe_sync_check(ws)
    if st != 0:
        raise RuntimeError(f"device error word {word:#x} during warm-up")
    # rows the expert GEMMs compute: T*K for top-K routing; Token Rounding's
    # rounded total (the same in every step: the inputs do not change)
    R = int((row_map >= 0).sum().item()) if rounded else T * K

    # Timed region: K forwards as a user runs them (no events inside a step, so
    # every kernel boundary keeps its programmatic dependent launch). Direct calls
    # by default; --graph captures the K steps once as a CUDA graph and replays it.
    graph, launch = None, "direct calls"
    if args.graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for i in range(args.steps):
                    step()
            torch.cuda.synchronize()
            launch = "one CUDA graph of the K steps"
        except RuntimeError as exc:  # capture unsupported here: time direct calls
            graph, launch = None, f"direct calls (graph capture failed: {exc})"[:200]
            torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        if graph is not None:
            with torch.cuda.stream(stream):
                graph.replay()
        else:
            for i in range(args.steps):
                step()
        stop.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    st, word = moe.moe_sync_check(ws)
    if st != 0:
        raise RuntimeError(f"device error word {word:#x} in the timed region")
    ms_total = start.elapsed_time(stop)
    ms_max = max_over_ranks(ms_total, world)

    # Stage region right after it: the same K forwards with an event between
    # every two stages (the traced forward records them on the launch stream),
    # for the per-kernel times and the roofline of the dominant kernel.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize()
    st, word = moe.moe_sync_check(ws)
    if st != 0:
        raise RuntimeError(f"device error word {word:#x} in the stage region")
    stage_ms = {s: float(np.mean([evs[i][j].elapsed_time(evs[i][j + 1])
                                  for i in range(args.steps)])) for j, s in enumerate(stages)}
    # kernels per forward, as the library reports them; the expert GEMMs take 1
    # launch when fused, 2 apart, 3 on CTA pairs (the row gather)
    launches = moe.forward_launches(T, d, E, K, n, rounded)
    fused = moe.forward_launches(T, d, E, K, n, rounded, part="expert_mlp") == 1
    if fused:  # one launch holds both GEMMs: the gate/up interval (down is empty)
        stage_ms = {("expert_mlp_fused" if k == "gemm_gate_up" else k):
                    (v + stage_ms["gemm_down"] if k == "gemm_gate_up" else v)
                    for k, v in stage_ms.items() if k != "gemm_down"}
    ms_step = ms_max / args.steps
    flops = 2.0 * R * 3 * d * n
    value = aggregate(flops * args.steps, ms_max / 1e3, world) / 1e12

    # Sustained region: back-to-back forwards for about --sustained-seconds, long
    # enough for the power cap to settle, against the sustained bf16 peak (the
    # K-step `value` above is a burst figure for the short window it times).
    sustained = None
    if args.sustained_seconds > 0:
        n_sus = max(args.steps, int(math.ceil(args.sustained_seconds * 1e3 / ms_step)))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clk_sus:
            barrier(world)
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(n_sus):
                step()
            b.record(stream)
            torch.cuda.synchronize()
            barrier(world)
        st, word = moe.moe_sync_check(ws)
        if st != 0:
            raise RuntimeError(f"device error word {word:#x} in the sustained region")
        ms_sus = max_over_ranks(a.elapsed_time(b), world)
        sus_value = aggregate(flops * n_sus, ms_sus / 1e3, world) / 1e12
        sus_peak = load_peaks()["bf16_sustained"]
        csum = clk_sus.summary()
        sustained = {"steps": n_sus, "seconds": round(ms_sus / 1e3, 3),
                     "ms_per_step": round(ms_sus / n_sus, 4), "value": round(sus_value, 3),
                     "unit": "TFLOP/s", "peak_sustained": sus_peak,
                     "frac_of_sustained_peak": None if not sus_peak
                     else round(sus_value / world / sus_peak, 4),
                     "clocks": {k: csum.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons",
                                                         "power_w_max")}}

    # end to end from pinned host memory: every step copies its batch in and its
    # output out. Top-K routing goes through moe_forward_host_stream, which
    # overlaps the copies of neighbouring batches with the layer.
    # (at most about 1 GB of pinned host batches for X, the same for Y)
    e2e_steps = max(3, min(args.steps, 20, int(1e9 // (T * d * 2))))
    Xh = inp["X"].cpu().pin_memory()
    Yh = torch.empty_like(Xh).pin_memory()
    Xd = torch.empty_like(inp["X"])
    Yd = torch.empty_like(inp["X"])
    Xhs = Xh.unsqueeze(0).repeat(e2e_steps, 1, 1).pin_memory()
    Yhs = torch.empty_like(Xhs).pin_memory()
    Xd2 = torch.empty((2, T, d), dtype=torch.bfloat16, device=dev)
    Yd2 = torch.empty_like(Xd2)
    s_comp, s_in, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))

    def host_step():
        if rounded:
            # same sequence as moe_forward_host: copy in, layer, copy out, wait
            Xd.copy_(Xh, non_blocking=True)
            moe.moe_forward_rounded(Xd, inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K,
                                    inp["bias"], ws=ws, Y=Yd, stream=stream)
            Yh.copy_(Yd, non_blocking=True)
            stream.synchronize()
        else:
            moe.moe_forward_host(Xh, Yh, Xd, Yd, inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K,
                                 inp["bias"], ws=ws, stream=stream)

    def host_run():
        if rounded:
            for _ in range(e2e_steps):
                host_step()
        else:
            moe.moe_forward_host_stream(Xhs, Yhs, Xd2, Yd2, inp["Wr"], inp["W1"], inp["W3"],
                                        inp["W2"], K, inp["bias"], ws=ws, stream=s_comp,
                                        h2d_stream=s_in, d2h_stream=s_out)

    for _ in range(2):
        host_step()
    host_run()
    barrier(world)
    t0 = time.perf_counter()
    host_run()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    barrier(world)
    e2e_value = aggregate(flops * e2e_steps, e2e_s, world) / 1e12

    # routing statistics (outside the timed region): tile padding and expert load
    if rounded:
        cnt = (row_map >= 0).sum(dim=0).cpu().numpy()
    else:
        _, _, cnt_t = moe.moe_route(inp["X"], inp["Wr"], K, inp["bias"])
        cnt = cnt_t.cpu().numpy()
    tiles_used = int(np.sum((cnt + 127) // 128))
    routing_stats = {
        "active_experts": int((cnt > 0).sum()), "rows_per_expert_max": int(cnt.max()),
        "rows_per_expert_min": int(cnt.min()), "rows_per_expert_var": round(float(cnt.var()), 1),
        "tiles_128": tiles_used,
        "padded_rows_pct": round(100.0 * (tiles_used * 128 - int(cnt.sum())) / max(1, tiles_used * 128), 2),
    }

    peaks = load_peaks()
    # the roofline object: the gate/up GEMM, or the fused launch of both GEMMs
    if fused:
        g1_name, g1_flops = "expert_mlp_fused (tcgen05 gate/up + SwiGLU and down, one launch)", flops
        g1_tflops = g1_flops / (stage_ms["expert_mlp_fused"] / 1e3) / 1e12
        g2_tflops = None
    else:
        g1_name, g1_flops = "gemm_gate_up (tcgen05 grouped GEMM + SwiGLU)", 4.0 * R * d * n
        g1_tflops = g1_flops / (stage_ms["gemm_gate_up"] / 1e3) / 1e12
        g2_tflops = 2.0 * R * n * d / (stage_ms["gemm_down"] / 1e3) / 1e12
    router_bytes = T * d * 2 + d * E * 4 + R * 8 + E * 4
    combine_bytes = (R + T) * d * 2
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload_desc(args.workload, c, args.routing),
                   **{k: c[k] for k in "TdEKn"}, "routing": args.routing, "rows": R,
                   "seed": args.seed, "launch": launch,
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "l2": "inputs larger than L2: expert weights "
                         f"{3 * E * d * n * 2 / 1e9:.2f} GB per step, no flush"},
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": T * d * 2, "d2h_bytes_per_step": T * d * 2},
        "roofline": {"kernel": g1_name, "bound": "tensor",
                     "achieved": round(g1_tflops, 2), "peak": peaks["bf16"], "unit": "TFLOP/s",
                     "frac": round(g1_tflops / peaks["bf16"], 4),
                     "traffic": None if rounded or fused
                     else (GEMM1_TRAFFIC_BYTES or {}).get(args.workload),
                     "peak_source": f"{peaks['source']} bf16 burst (cuBLAS)",
                     "algorithmic_flops_per_launch": g1_flops},
        "gpu_launches": launches * args.steps,
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "extra": {
            "tokens_per_s": round(T * world / (ms_step / 1e3), 1),
            "pct_bf16_peak_layer": round(value / world / peaks["bf16"] * 100, 2),
            "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
            "topk_rows_equiv_tflops": round(useful_flops(c) * world / (ms_step / 1e3) / 1e12, 3),
            "routing": routing_stats,
            "gemm_down_tflops": None if g2_tflops is None else round(g2_tflops, 2),
            "router_GBps": round(router_bytes / (stage_ms["route"] / 1e3) / 1e9, 1),
            "router_frac_hbm": round(router_bytes / (stage_ms["route"] / 1e3) / 1e9 / peaks["hbm"], 4),
            "combine_GBps": round(combine_bytes / (stage_ms["combine"] / 1e3) / 1e9, 1),
            "hbm_peak_GBps": peaks["hbm"], "clock_samples": clocks.get("samples"),
            "power_w_max": clocks.get("power_w_max"),
            "sustained": sustained,
        },
    }
    if not args.no_backward and not rounded:
        line["extra"]["backward"] = measure_backward(args, c, inp, stream, dev)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not rounded:
        import oracle
        oracle.build()
        inp_np = host_inputs(inp)
        ntok, tf, dt = calibrate_sample(inp_np, c, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s",
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": f"{ntok} of {T} tokens, token-by-token oracle "
                                          f"(routing included), {dt:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_router_only(args, world, rank, local):
    """The router-only workload: given logits [T,8] fp32, softmax + top-2 +
    counts (moe_route_logits), T in {256, 512, 1024, 2048}; microseconds per call."""
    import torch
    from top_routing_grouped_02_gb300 import moe, synth
    torch.cuda.set_device(local)
    stream = torch.cuda.current_stream()
    per_t = {}
    import ctypes
    lib = moe.lib()
    for T in synth.ROUTER_T:
        logits = synth.router_logits_input(T, device="cuda")
        K, E = synth.ROUTER_K, synth.ROUTER_E
        idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
        w = torch.empty((T, K), dtype=torch.float32, device="cuda")
        counts = torch.empty(E, dtype=torch.int32, device="cuda")
        ptrs = [ctypes.c_void_p(t.data_ptr()) for t in (logits, idx, w, counts)]

        def call(st):
            rc = lib.moe_route_logits(ptrs[0], T, E, K, 1, ptrs[1], ptrs[2], ptrs[3],
                                      ctypes.c_void_p(st.cuda_stream))
            if rc != 0:
                raise moe.MoeError("moe_route_logits", rc)

        for _ in range(args.warmup):
            call(stream)
        torch.cuda.synchronize()
        # device time: the calls are captured once in a CUDA graph and replayed, so
        # host launch overhead does not sit between them
        side = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for _ in range(args.steps):
                    call(side)
        graph.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / args.steps
        nbytes = T * synth.ROUTER_E * 4 + T * synth.ROUTER_K * 8 + synth.ROUTER_E * 4
        per_t[T] = {"us": round(us, 3), "GBps": round(nbytes / (us * 1e-6) / 1e9, 2)}
    # Supplementary sweep (not the metric): the same call at 2^20 .. 2^23 tokens,
    # where the traffic is large enough to compare with HBM bandwidth. Logits of
    # 2^22 tokens and more exceed L2; the smaller ones may partly stay in it.
    peaks = load_peaks()
    sweep = {}
    for T in (1 << 20, 1 << 21, 1 << 22, 1 << 23):
        K, E = synth.ROUTER_K, synth.ROUTER_E
        logits = synth.router_logits_input(T, device="cuda")
        idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
        w = torch.empty((T, K), dtype=torch.float32, device="cuda")
        counts = torch.empty(E, dtype=torch.int32, device="cuda")
        ptrs = [ctypes.c_void_p(t.data_ptr()) for t in (logits, idx, w, counts)]

        def call_big(st, T=T, ptrs=ptrs):
            rc = lib.moe_route_logits(ptrs[0], T, E, K, 1, ptrs[1], ptrs[2], ptrs[3],
                                      ctypes.c_void_p(st.cuda_stream))
            if rc != 0:
                raise moe.MoeError("moe_route_logits", rc)

        reps = 20
        for _ in range(3):
            call_big(stream)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            call_big(stream)
        b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / reps
        nbytes = T * E * 4 + T * K * 8 + E * 4
        sweep[T] = {"us": round(us, 2), "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
                    "frac_hbm": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm"], 3),
                    "bytes": nbytes}
        del logits, idx, w, counts
    total_tokens = sum(synth.ROUTER_T)
    total_us = sum(v["us"] for v in per_t.values())
    if rank == 0:
        print(json.dumps({
            "metric": "router-only fused gating (softmax + top-2 + counts) time per call",
            "value": round(total_tokens / (total_us * 1e-6), 1), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_us / 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "router-only logits [T,8] fp32, K=2, T in 256..2048"},
            "gpu_launches": len(synth.ROUTER_T) * args.steps,
            "extra": {"per_T": per_t,
                      "supplementary_sweep": {"note": "same call at large T, direct calls "
                                              "(memset + one kernel each); logits exceed L2 "
                                              "from T = 2^22; HBM peak " + peaks["source"],
                                              "hbm_peak_GBps": peaks["hbm"], "per_T": sweep}}}),
              flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixtral",
                    choices=["tiny", "mixtral", "dsv3", "sonic", "router"])
    ap.add_argument("--routing", choices=["topk", "rounded"], default="topk",
                    help="rounded: Token Rounding of the top-K counts to multiples of 128")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sustained-seconds", type=float, default=2.0,
                    help="length of the sustained region reported in extra.sustained (0: skip)")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the backward region reported in extra.backward")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's token count T (0: the workload's own)")
    ap.add_argument("--graph", action="store_true",
                    help="time one CUDA graph of the K steps instead of direct calls")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from top_routing_grouped_02_gb300 import synth
    world, rank, local = dist_setup()
    if args.workload == "router":
        run_router_only(args, world, rank, local)
        return
    c = dict(synth.WORKLOADS[args.workload])
    if args.tokens:  # a smaller (or larger) case of the same layer, e.g. for ncu captures
        c["T"] = args.tokens
    if args.impl == "reference":
        run_reference(args, c, world, rank)
    else:
        run_gpu(args, c, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
