"""Benchmark: weight-streaming throughput of the whole decode step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--n-tok T] [--impl kq|reference]

One step = the weight GEMVs of one decode step of the 52-layer decoder
(per layer: q/k/v, o, gate/up in Q4_K and down in Q6_K; hidden 5120,
intermediate 32768) plus a Q6_K LM head 200000 x 5120 -- 19.1 GB of packed
weights streamed once -- captured as one CUDA graph.  The metric is weight
GB/s (packed bytes streamed per second); microseconds per step and the
equivalent tokens/s are reported beside it.  Inputs are synthetic (seeded);
the 19.1 GB working set is far larger than L2, so no flush is needed.

N > 1 (torchrun): every rank runs an independent replica on its own GPU
(the path has no exchange step); value = total bytes of all ranks / the
slowest rank's time.  --impl reference times the CPU oracle on a bounded
sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "K-quant GEMV weight GB/s (% of B300 HBM peak) at 1/8 tokens; us per decode step"
# single launches of one decoder layer (layer 0's weights), for profiling:
# the matrices that share the launch
CASES = {"qkv": ("q", "k", "v"), "o": ("o",), "gate_up": ("gate", "up"), "down": ("down",),
         "lm_head": ("lm_head",)}
WORKLOAD = "decode_step_52L_h5120_i32768_q4k_q6k_lmhead200000"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--n-tok", type=int, default=1)
    p.add_argument("--impl", default="kq", choices=["kq", "reference"])
    p.add_argument("--layers", type=int, default=wl.LAYERS)
    p.add_argument("--no-extra", action="store_true", help="skip the n_tok=8 line and e2e")
    p.add_argument("--case", default="step", choices=["step"] + sorted(CASES),
                   help="one launch of the decode step instead of the whole step (for profiling)")
    p.add_argument("--path", default="bf16", choices=["bf16", "q8"],
                   help="--case: the bf16-activation kernels, or the int8-activation dp4a "
                        "kernel (one launch per matrix)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return rank, local, world


def init_dist(world):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("gloo")
        return dist
    return None


def max_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def replica_throughput(dist, bytes_this_rank: float, seconds_this_rank: float):
    """Whole-job throughput of independent replicas: the bytes every rank
    streamed divided by the slowest rank's time.  Returns (GB/s, slowest
    seconds, total bytes)."""
    t_max = max_over_ranks(dist, seconds_this_rank)
    total = sum_over_ranks(dist, float(bytes_this_rank))
    return total / t_max / 1e9, t_max, total


NOMINAL_HBM_GBS = 7700.0   # B300 HBM3e, nominal (context only; the roofline uses the measured peak)


def cpu_model() -> str:
    """The host CPU's model name (Linux /proc/cpuinfo), for the oracle baseline."""
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh), "measured"
    except OSError:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_sha() -> str:
    """Hash of the kernel sources' code: comments and blank space are left
    out, so a comment edit does not void the recorded DRAM traffic (no
    string literal in the sources holds a comment marker)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quant_weight_gemv_dequant_b300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), encoding="utf-8") as fh:
                code = re.sub(r"/\*.*?\*/", " ", fh.read(), flags=re.S)
            code = re.sub(r"//[^\n]*", "", code)
            code = "\n".join(" ".join(line.split()) for line in code.splitlines() if line.strip())
            h.update(name.encode() + code.encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
    except (OSError, ValueError):
        return None
    e = d.get(kernel)
    if not e or e.get("kernel_src_sha") != kernel_source_sha():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ inputs

def build_pools_library(device):
    """Pools of N(0, 0.02) super-blocks quantised by the library's host
    quantiser (identical bytes to the oracle's, tested)."""
    import torch
    import quant_weight_gemv_dequant_b300 as kq
    pw = wl.pool_weights(wl.derive_seed(900), wl.POOL_BLOCKS)
    return {f: torch.from_numpy(kq.kq_quantize(f, pw, wl.POOL_BLOCKS, 256)).to(device)
            for f in (wl.Q4_K, wl.Q5_K, wl.Q6_K)}


def build_step(pools_dev, n_tok, layers, device, spec=None, head_spec=None, base=5):
    """The decode step of `layers` layers of `spec` (default: the benchmark
    layer) plus `head_spec`, tiled from the pools; returns (step, pinned
    host copy of all its activation inputs)."""
    import torch
    from quant_weight_gemv_dequant_b300.decode_step import DecodeStep
    spec = wl.DECODE_LAYER if spec is None else spec
    h = wl.LM_HEAD if head_spec is None else head_spec
    Ls = []
    for l in range(layers):
        L = {}
        for i, m in enumerate(spec):
            seed = wl.derive_seed(base, l, i)
            L[m.name] = (m.fmt, wl.tile_matrix_device(pools_dev[m.fmt], m.fmt, seed, m.N, m.K), m.N, m.K)
        Ls.append(L)
    head = (h.fmt, wl.tile_matrix_device(pools_dev[h.fmt], h.fmt, wl.derive_seed(base, 999), h.N, h.K), h.N, h.K)
    step = DecodeStep(Ls, head, n_tok, device=device)
    # the step's activation inputs, in the order of step.x_all (layer by layer:
    # x_attn, x_o, x_ffn, x_down; then the head), in one pinned host buffer
    parts = []
    for l in range(layers):
        for j, key in enumerate(("x_attn", "x_o", "x_ffn", "x_down")):
            parts.append(wl.activations_bf16(wl.derive_seed(base, l, 100 + j), n_tok, step.x[l][key].shape[1]))
    parts.append(wl.activations_bf16(wl.derive_seed(base, 998), n_tok, h.K))
    flat = np.concatenate([p_.reshape(-1) for p_ in parts])
    host_x = torch.from_numpy(flat.view(np.int16)).view(torch.bfloat16).pin_memory()
    step.x_all.copy_(host_x)
    torch.cuda.synchronize()
    return step, host_x


def io_bytes(step):
    xb = sum(t.numel() * 2 for xs in step.x for t in xs.values()) + step.x_head.numel() * 2
    yb = sum(t.numel() * 4 for ys in step.y for t in ys.values()) + step.y_head.numel() * 4
    return xb, yb


def time_graph(g, stream, steps, warmup, dist):
    """Seconds per replay: events recorded on the stream the graph is
    launched on (CUDAGraph.replay launches on the current stream)."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    return e0.elapsed_time(e1) / 1e3 / steps


def dominant_kernel_timing(step, steps, warmup, stream):
    """Average duration of the dominant launch (the grouped gate/up Q4_K GEMV
    of each layer): a graph of the step's own gate/up launches, timed with
    events on the launching stream."""
    import torch
    import quant_weight_gemv_dequant_b300 as kq
    g = torch.cuda.CUDAGraph()
    lay = step.layers

    def run():
        for l, L in enumerate(lay):
            f, Wg, N, K = L["gate"]
            kq.kq_gemv_multi(f, [Wg, L["up"][1]], [step.y[l]["gate"], step.y[l]["up"]], [N, L["up"][2]],
                             step.x[l]["x_ffn"], K, step.n_tok, stream)

    with torch.cuda.stream(stream):
        run()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        run()
    dur_total = time_graph(g, stream, steps, warmup, None)
    launches = len(lay)
    dur = dur_total / launches
    L0 = lay[0]
    nbytes = (L0["gate"][1].numel() + L0["up"][1].numel() + step.x[0]["x_ffn"].numel() * 2
              + (L0["gate"][2] + L0["up"][2]) * 4 * step.n_tok)
    return dur, nbytes, "gemv_q4k_gate_up"


# ------------------------------------------- per-config and per-launch lines

L2_BYTES = 126e6   # B300 L2


def graph_time(launch, n_launch, stream, reps=5):
    """Seconds per launch of launch(i) for i < n_launch, captured in one CUDA
    graph and replayed `reps` times; CUDA events on the launching stream."""
    import torch
    for i in range(min(n_launch, 8)):      # shapes seen once outside capture
        launch(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n_launch):
            launch(i)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / (reps * n_launch)


def copies_for(nbytes: int) -> int:
    """Weight copies to rotate through so that one round streams >= 4x L2."""
    return max(1, int(np.ceil(4 * L2_BYTES / nbytes)))


def time_group(groups, T, K, stream, heavy=False, seed=0):
    """Per-launch seconds of one grouped launch (fmt, [W], [N]) rotated over
    the copies in `groups` (a list of (fmt, [W], [N]) with the same shapes)."""
    import torch
    import quant_weight_gemv_dequant_b300 as kq
    dev = groups[0][1][0].device
    x = torch.from_numpy(wl.activations_bf16(wl.derive_seed(60, seed, T), T, K, heavy=heavy)
                         .view(np.int16)).to(dev).view(torch.bfloat16)
    ys = [torch.empty((T, n), dtype=torch.float32, device=dev) for n in groups[0][2]]
    R = len(groups)

    def launch(i):
        f, Ws, Ns = groups[i % R]
        kq.kq_gemv_multi(f, Ws, ys, Ns, x, K, T, stream)

    return graph_time(launch, max(2 * R, 24), stream)


def rate_line(nbytes, seconds, hbm):
    return {"us": seconds * 1e6, "weight_gb_s": nbytes / seconds / 1e9,
            "frac_of_hbm_peak": nbytes / seconds / 1e9 / hbm}


def measure_configs(pools, device, stream, hbm):
    """The other workloads, each timed as graph replays of its launches over
    rotated weight copies (>= 4x L2 per round): C1 single Q4_K 4096x4096 at
    1 and 8 tokens; C2 attention projections (q/k/v grouped, o) plus q in the
    merged group-128 layout; C3 the SwiGLU FFN with heavy-tailed x; C4 one
    Q5_K layer (seven projections, four launches) at n_tok 1, 2, 4, 8, 16."""
    import torch
    import quant_weight_gemv_dequant_b300 as kq
    out = {}

    def host_quant(fmt, m, seed):
        w = wl.weights_f32(wl.derive_seed(61, seed), m.N, m.K)
        return torch.from_numpy(kq.kq_quantize(fmt, w, m.N, m.K)).to(device)

    # C1
    m = wl.SINGLE_Q4K[0]
    W = host_quant(m.fmt, m, 1)
    R = copies_for(m.nbytes)
    groups = [(m.fmt, [W.clone()], [m.N]) for _ in range(R)]
    c1 = {"workload": "single_q4k_4096x4096", "weight_bytes": m.nbytes, "copies": R}
    for T in (1, 8):
        c1[f"n_tok_{T}"] = rate_line(m.nbytes, time_group(groups, T, m.K, stream, seed=1), hbm)
    out["C1"] = c1
    del groups, W

    # C2
    q, k, v, o, qg = wl.ATTN_Q4K
    Wq, Wk, Wv, Wo = (host_quant(mm.fmt, mm, 20 + i) for i, mm in enumerate((q, k, v, o)))
    Wqg = torch.from_numpy(kq.kq_quantize(wl.Q4_G128, wl.weights_f32(wl.derive_seed(61, 20), q.N, q.K),
                                          q.N, q.K)).to(device)
    qkv_bytes = q.nbytes + k.nbytes + v.nbytes
    c2 = {"workload": "attention_q4k_h5120_q4096_kv256_plus_q_g128",
          "weight_bytes": qkv_bytes + o.nbytes, "q_g128_bytes": qg.nbytes}
    R = copies_for(qkv_bytes)
    t_qkv = time_group([(q.fmt, [Wq.clone(), Wk.clone(), Wv.clone()], [q.N, k.N, v.N]) for _ in range(R)],
                       1, q.K, stream, seed=2)
    R = copies_for(o.nbytes)
    t_o = time_group([(o.fmt, [Wo.clone()], [o.N]) for _ in range(R)], 1, o.K, stream, seed=3)
    R = copies_for(qg.nbytes)
    t_qg = time_group([(qg.fmt, [Wqg.clone()], [qg.N]) for _ in range(R)], 1, qg.K, stream, seed=2)
    c2["n_tok_1"] = {"qkv": rate_line(qkv_bytes, t_qkv, hbm), "o": rate_line(o.nbytes, t_o, hbm),
                     "q_g128": rate_line(qg.nbytes, t_qg, hbm),
                     "attention_total": rate_line(qkv_bytes + o.nbytes, t_qkv + t_o, hbm)}
    out["C2"] = c2
    del Wq, Wk, Wv, Wo, Wqg

    # C3
    gate, up, down = wl.FFN_Q4K_Q6K
    gu_bytes = gate.nbytes + up.nbytes
    R = copies_for(gu_bytes)
    gu = [(gate.fmt, [wl.tile_matrix_device(pools[gate.fmt], gate.fmt, wl.derive_seed(62, r, 0), gate.N, gate.K),
                      wl.tile_matrix_device(pools[up.fmt], up.fmt, wl.derive_seed(62, r, 1), up.N, up.K)],
           [gate.N, up.N]) for r in range(R)]
    t_gu = time_group(gu, 1, gate.K, stream, heavy=True, seed=4)
    del gu
    R = copies_for(down.nbytes)
    dn = [(down.fmt, [wl.tile_matrix_device(pools[down.fmt], down.fmt, wl.derive_seed(62, r, 2), down.N, down.K)],
           [down.N]) for r in range(R)]
    t_dn = time_group(dn, 1, down.K, stream, heavy=True, seed=5)
    del dn
    out["C3"] = {"workload": "ffn_q4k_gate_up_2x32768x5120_q6k_down_5120x32768_heavy_tailed_x",
                 "weight_bytes": gu_bytes + down.nbytes,
                 "n_tok_1": {"gate_up": rate_line(gu_bytes, t_gu, hbm), "down": rate_line(down.nbytes, t_dn, hbm),
                             "ffn_total": rate_line(gu_bytes + down.nbytes, t_gu + t_dn, hbm)}}

    # C4
    lay = wl.LAYER_Q5K
    lay_bytes = sum(mm.nbytes for mm in lay)
    R = copies_for(lay_bytes)
    mats = [{mm.name: wl.tile_matrix_device(pools[wl.Q5_K], wl.Q5_K, wl.derive_seed(63, r, i), mm.N, mm.K)
             for i, mm in enumerate(lay)} for r in range(R)]
    by = {mm.name: mm for mm in lay}
    launches = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))
    c4 = {"workload": "q5k_layer_h5120_i32768_seven_projections", "weight_bytes": lay_bytes, "copies": R}
    for T in (1, 2, 4, 8, 16):
        xs = {K: torch.from_numpy(wl.activations_bf16(wl.derive_seed(64, T, K), T, K).view(np.int16))
              .to(device).view(torch.bfloat16) for K in {mm.K for mm in lay}}
        ys = {mm.name: torch.empty((T, mm.N), dtype=torch.float32, device=device) for mm in lay}

        def step(i, T=T, xs=xs, ys=ys):
            Ws = mats[i % R]
            for grp in launches:
                K = by[grp[0]].K
                kq.kq_gemv_multi(wl.Q5_K, [Ws[n] for n in grp], [ys[n] for n in grp],
                                 [by[n].N for n in grp], xs[K], K, T, stream)

        t = graph_time(step, max(2 * R, 8), stream)
        c4[f"n_tok_{T}"] = {**rate_line(lay_bytes, t, hbm), "us_per_token": t * 1e6 / T}
    out["C4"] = c4
    del mats
    torch.cuda.empty_cache()
    return out


def step_launch_table(pools, device, stream, hbm, n_toks=(1, 8)):
    """Per-launch time of each launch type of the decode step (layer-0
    shapes, rotated copies >= 4x L2) at the given widths, with its share of
    a step (52 layers + head); the largest share per width is the dominant
    kernel of that width."""
    table = {}
    for T in n_toks:
        row = {}
        for case, names in CASES.items():
            mats = [wl.LM_HEAD] if names == ("lm_head",) else [m for m in wl.DECODE_LAYER if m.name in names]
            nbytes = sum(m.nbytes for m in mats)
            R = copies_for(nbytes)
            groups = [(mats[0].fmt, [wl.tile_matrix_device(pools[m.fmt], m.fmt, wl.derive_seed(65, r, i), m.N, m.K)
                                     for i, m in enumerate(mats)], [m.N for m in mats]) for r in range(R)]
            t = time_group(groups, T, mats[0].K, stream, seed=6)
            del groups
            per_step = 1 if case == "lm_head" else wl.LAYERS
            row[case] = {**rate_line(nbytes, t, hbm), "bytes_per_launch": nbytes, "launches_per_step": per_step,
                         "us_per_step": t * 1e6 * per_step}
        tot = sum(r["us_per_step"] for r in row.values())
        for r in row.values():
            r["share"] = r["us_per_step"] / tot
        table[f"n_tok_{T}"] = row
    return table


# ------------------------------------------------------------- CPU oracle

def oracle_samples(pools_host, rounds: int, n_tok: int = 1):
    """Inputs for the oracle timing: per round, 2 sampled rows of each of the
    7 layer matrices (layer = round index) and of the LM head, same tiling
    and activations as the GPU step."""
    mats = list(enumerate(wl.DECODE_LAYER)) + [(999, wl.LM_HEAD)]
    xs = {}
    out = []
    for r in range(rounds):
        for i, m in mats:
            seed = wl.derive_seed(5, r % wl.LAYERS, i) if i != 999 else wl.derive_seed(5, 999)
            rows = (wl.splitmix64(seed, np.arange(2, dtype=np.uint64)) % np.uint64(m.N)).astype(np.int64)
            sub = wl.tiled_rows(pools_host[m.fmt], m.fmt, seed, m.N, m.K, rows)
            if m.K not in xs:
                xs[m.K] = wl.activations_bf16(wl.derive_seed(5, 0, 100), n_tok, m.K)
            out.append((m.fmt, sub, len(rows), m.K, xs[m.K]))
    return out


def oracle_sample_rate(samples, budget_s: float):
    """Weight GB/s of the single-threaded fp64 oracle over the samples,
    cycling through them for about budget_s seconds (only oracle calls are
    inside the timed region)."""
    import oracle
    done_bytes, el, k = 0, 0.0, 0
    while el < budget_s:
        fmt, sub, n, K, x = samples[k % len(samples)]
        t0 = time.perf_counter()
        oracle.gemv(fmt, sub, n, K, x)
        el += time.perf_counter() - t0
        done_bytes += sub.size
        k += 1
    return done_bytes / el / 1e9, el, done_bytes


def oracle_pools():
    import oracle
    pw = wl.pool_weights(wl.derive_seed(900), wl.POOL_BLOCKS)
    return {f: oracle.quantize(f, pw, wl.POOL_BLOCKS, 256) for f in (wl.Q4_K, wl.Q6_K)}


# ------------------------------------------------------------------- arms

def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    samples = oracle_samples(oracle_pools(), 8, args.n_tok)
    step_bytes = wl.decode_step_bytes(args.layers)
    per_step = []
    for _ in range(args.warmup):
        oracle_sample_rate(samples, 0.2)
    for _ in range(args.steps):
        gbs, el, nb = oracle_sample_rate(samples, 1.0)
        per_step.append((gbs, el, nb))
    tot_b = sum(p[2] for p in per_step)
    tot_t = sum(p[1] for p in per_step)
    value = tot_b / tot_t / 1e9
    ms = step_bytes / (value * 1e9) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "n_tok": args.n_tok, "layers": args.layers,
                   "weight_bytes_per_step": step_bytes},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "cpu_model": cpu_model(), "host_cpus": os.cpu_count(),
                         "sample": f"2 sampled rows of each of the 7 matrices of 8 layers and of the LM head, "
                                   f"cycled for ~1 s of single-threaded fp64 oracle per step; {tot_b} packed "
                                   f"bytes total; ms_per_step extrapolates to the full 19.1 GB step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_kq(args):
    import torch
    rank, local, world = dist_env()
    dist = init_dist(world)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import quant_weight_gemv_dequant_b300 as kq
    kq.lib()

    pools = build_pools_library(device)
    step, host_x = build_step(pools, args.n_tok, args.layers, device)
    stream = torch.cuda.Stream(device=device)
    g = step.capture(stream)
    wbytes = step.weight_bytes()
    xb, yb = io_bytes(step)

    with ClockSampler(local) as clk:
        t_step = time_graph(g, stream, args.steps, max(3, args.warmup), dist)
    value, t_max, total_bytes = replica_throughput(dist, wbytes, t_step)
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])

    extra = {}
    if not args.no_extra and args.n_tok == 1:
        # n_tok = 8 (speculative verify) on the same weights
        s8 = type(step)(step.layers, step.lm_head, 8, device=device)
        for l in range(args.layers):
            for j, key in enumerate(("x_attn", "x_o", "x_ffn", "x_down")):
                xb8 = wl.activations_bf16(wl.derive_seed(5, l, 200 + j), 8, s8.x[l][key].shape[1])
                s8.x[l][key].copy_(torch.from_numpy(xb8.view(np.int16)).view(torch.bfloat16))
        g8 = s8.capture(stream)
        t8 = max_over_ranks(dist, time_graph(g8, stream, args.steps, 3, dist))
        del g8, s8
        # the CUDA-core path at this width: two 4-token passes over the same
        # weights (what the library falls back to without the tensor-core
        # kernel), i.e. twice the n_tok = 4 step
        s4 = type(step)(step.layers, step.lm_head, 4, device=device)
        for l in range(args.layers):
            for j, key in enumerate(("x_attn", "x_o", "x_ffn", "x_down")):
                xb4 = wl.activations_bf16(wl.derive_seed(5, l, 200 + j), 4, s4.x[l][key].shape[1])
                s4.x[l][key].copy_(torch.from_numpy(xb4.view(np.int16)).view(torch.bfloat16))
        g4 = s4.capture(stream)
        t4 = max_over_ranks(dist, time_graph(g4, stream, max(10, args.steps // 4), 3, dist))
        del g4, s4
        extra["n_tok_8"] = {"ms_per_step": t8 * 1e3, "weight_gb_s": wbytes / t8 / 1e9 * world,
                            "pct_of_hbm_peak": 100 * wbytes / t8 / 1e9 / hbm,
                            "tok_per_s": 8 / t8 * world, "path": "tensor cores (mma.sync bf16)",
                            "cuda_core_ms_per_step": 2 * t4 * 1e3,
                            "cuda_core_path": "two n_tok=4 passes (CUDA cores)",
                            "n_tok_4_ms_per_step": t4 * 1e3}

    # the same step with the SwiGLU chain fused: each layer's gate/up launch
    # writes h = bf16(silu(gate) * up) and its down projection reads h
    if not args.no_extra and args.n_tok == 1:
        sf = type(step)(step.layers, step.lm_head, 1, device=device, fused_ffn=True)
        sf.x_all.copy_(step.x_all)
        gf = sf.capture(stream)
        tf = max_over_ranks(dist, time_graph(gf, stream, args.steps, 3, dist))
        extra["fused_ffn"] = {"ms_per_step": tf * 1e3, "weight_gb_s": wbytes / tf / 1e9 * world,
                              "pct_of_hbm_peak": 100 * wbytes / tf / 1e9 / hbm,
                              "launches_per_step": sf.launches(),
                              "path": "per layer: q/k/v, o, gate/up writing bf16 silu(gate)*up, down reading it"}
        del gf, sf

    # the pages' own shapes (hidden 6656, intermediate 19968, vocab 202048;
    # q, k, v and the attention's sigmoid gate in one launch): a second
    # 52-layer step of 17.0 GB
    if not args.no_extra and args.n_tok == 1:
        sp, _ = build_step(pools, 1, args.layers, device, spec=wl.GLIMMER_LAYER,
                           head_spec=wl.GLIMMER_HEAD, base=7)
        gp = sp.capture(stream)
        tp = max_over_ranks(dist, time_graph(gp, stream, args.steps, 3, dist))
        pb = sp.weight_bytes()
        extra["pages_shapes"] = {"workload": "decode_step_52L_h6656_i19968_qkvg_q4k_q6k_lmhead202048",
                                 "weight_bytes_per_step": pb, "ms_per_step": tp * 1e3,
                                 "weight_gb_s": pb / tp / 1e9 * world,
                                 "pct_of_hbm_peak": 100 * pb / tp / 1e9 / hbm,
                                 "tok_per_s": 1 / tp * world, "launches_per_step": sp.launches()}
        del gp, sp
        torch.cuda.empty_cache()

    # dominant kernel: grouped gate/up Q4_K GEMV launches
    dur, kbytes, kname = dominant_kernel_timing(step, args.steps, 3, stream)
    achieved = kbytes / dur / 1e9

    # the other workloads, and every launch type of the step at 1 and 8 tokens
    configs, table, roofline_n8 = None, None, None
    if not args.no_extra and rank == 0:
        configs = measure_configs(pools, device, stream, hbm)
        table = step_launch_table(pools, device, stream, hbm)
        dom = max(table["n_tok_8"].items(), key=lambda kv: kv[1]["share"])
        roofline_n8 = {"bound": "hbm", "kernel": f"{dom[0]} at n_tok 8", "achieved": dom[1]["weight_gb_s"],
                       "peak": hbm, "peak_kind": peak_kind, "unit": "GB/s",
                       "frac": dom[1]["weight_gb_s"] / hbm, "traffic": None,
                       "bytes_per_launch": dom[1]["bytes_per_launch"], "launch_us": dom[1]["us"],
                       "share_of_step": dom[1]["share"]}

    # end to end through the public API with host buffers: per step, H2D of
    # every activation input from pinned memory, the layers, D2H of the
    # logits.  The step is captured with its input copies (DecodeStep.capture
    # with host_x: layer by layer on a second stream, each layer waiting for
    # its own inputs), so one replay copies every input of the step.
    e2e = None
    if not args.no_extra:
        y_host = torch.empty(step.y_head.shape, dtype=torch.float32).pin_memory()
        h2d = host_x.numel() * 2
        d2h = y_host.numel() * 4
        ge = step.capture(stream, host_x=host_x)

        def e2e_step():
            with torch.cuda.stream(stream):
                ge.replay()
                y_host.copy_(step.y_head, non_blocking=True)
            stream.synchronize()

        for _ in range(3):
            e2e_step()
        barrier(dist)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        te = max_over_ranks(dist, (time.perf_counter() - t0) / args.steps)
        e2e = {"value": total_bytes / te / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": te * 1e3}

    cpu = None
    if rank == 0 and not args.no_extra:
        gbs, el, nb = oracle_sample_rate(oracle_samples(oracle_pools(), 8, args.n_tok), 12.0)
        cpu = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "cpu_model": cpu_model(), "host_cpus": os.cpu_count(),
               "sample": f"single-threaded fp64 oracle on 2 sampled rows of each of the 7 matrices of 8 "
                         f"layers and of the LM head, cycled for {el:.1f} s ({nb} packed bytes)"}

    if rank == 0:
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": t_max * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "n_tok": args.n_tok, "layers": args.layers,
                       "weight_bytes_per_step": wbytes, "x_bytes": xb, "y_bytes": yb,
                       "l2": "inputs larger than L2 (19.1 GB weights per step)",
                       "graph": "one CUDA graph per step", "parallelism": f"replicas x{world}"},
            "us_per_step": t_max * 1e6, "tok_per_s": args.n_tok / t_max * world,
            "pct_of_hbm_peak": 100 * value / world / hbm,
            "pct_of_nominal_hbm": 100 * value / world / NOMINAL_HBM_GBS,
            "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": hbm,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": profiled_traffic(kname), "bytes_per_launch": kbytes,
                         "launch_us": dur * 1e6},
            "roofline_n8": roofline_n8, "configs": configs, "launch_table": table,
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": step.launches() * args.steps,
            "clocks": clocks, **extra,
        }
        print(json.dumps(line), flush=True)
    barrier(dist)


def run_case(args):
    """--case NAME: warm-up + `steps` launches of one grouped launch of the
    decode step on its full-size matrices (the same weights every launch;
    q/k/v and o fit in L2), timed with CUDA events; one JSON line."""
    import torch
    import quant_weight_gemv_dequant_b300 as kq
    _, local, _ = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    kq.lib()
    pools = build_pools_library(device)
    names = CASES[args.case]
    mats = [wl.LM_HEAD] if names == ("lm_head",) else [m for m in wl.DECODE_LAYER if m.name in names]
    Ws = [wl.tile_matrix_device(pools[m.fmt], m.fmt, wl.derive_seed(5, 0, i), m.N, m.K)
          for i, m in enumerate(mats)]
    fmt, K, T = mats[0].fmt, mats[0].K, args.n_tok
    xb = wl.activations_bf16(wl.derive_seed(5, 0, 100), T, K)
    x = torch.from_numpy(xb.view(np.int16)).to(device).view(torch.bfloat16)
    ys = [torch.empty((T, m.N), dtype=torch.float32, device=device) for m in mats]
    Ns = [m.N for m in mats]
    stream = torch.cuda.current_stream(device)

    def launch():
        if args.path == "q8":
            for W, y, N in zip(Ws, ys, Ns):
                kq.kq_gemv_q8(fmt, W, x, y, N, K, T)
        else:
            kq.kq_gemv_multi(fmt, Ws, ys, Ns, x, K, T)

    for _ in range(max(3, args.warmup)):
        launch()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        launch()
    e1.record(stream)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / args.steps
    nbytes = sum(m.nbytes for m in mats)
    print(json.dumps({"case": args.case, "path": args.path,
                      "matrices": [f"{m.name} {m.N}x{m.K} fmt {m.fmt}" for m in mats],
                      "n_tok": T, "launches": args.steps, "us_per_launch": t * 1e6,
                      "weight_gb_s": nbytes / t / 1e9,
                      "l2": "weights resident in L2" if nbytes < 100e6 else "weights larger than L2",
                      "status": kq.kq_device_status(check=False)}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.case != "step":
        run_case(args)
    else:
        run_kq(args)


if __name__ == "__main__":
    main()
