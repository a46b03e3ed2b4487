"""Benchmark of the pi0 action-expert denoise chunk (18 blocks x 10 Euler steps,
64 query tokens over a 512-token prefix KV) on one GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one lat_denoise_chunk (the whole hot path: state token, 10 x
[embedding, 18 x block, head + Euler]).  The metric is milliseconds per
denoised chunk (lower is better); microseconds per block and tokens/s are
reported alongside.  Every step streams all 623 MB of folded block weights
from HBM (L2 is 129 MB), so no flush is needed between steps.

The headline line also carries config.dense: every dense configuration
(prefix prefill B = 1 / 8, the DiT 1.3B stage, its interleaved schedule, the
DiT 14B block with 1 / 4 / 8 chunks) timed with CUDA events in the same run,
with its useful TFLOP/s against the measured bf16 peak (--no-dense skips it).

--impl reference times the CPU oracle (float64 numpy) on the same workload on
the host cores, one whole denoise step per step; under torchrun only rank 0
runs it.
Multi-GPU: replicas only (one independent chunk per GPU per step, no
collective on the data path); value = whole-job chunks per step time.
"""
import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "pi0_ae"
PAGES_AE_MS = 11.001   # pages' action-expert time, 2 views, RTX 4090 (context)
# DRAM bytes (read + write) of one step-kernel launch from the last ncu capture
# of the kernel as it stands (dram__bytes_read.sum + dram__bytes_write.sum);
# None when the kernel has changed since
STEP_TRAFFIC = None


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-dense", action="store_true",
                   help="skip timing the dense configurations in the headline run")
    p.add_argument("--layers", type=int, default=0,
                   help="dense workloads: run this many blocks instead of the configuration's "
                        "(same per-block shapes; for small profiler captures)")
    p.add_argument("--workload", default=WORKLOAD, choices=[WORKLOAD, "pi0_cycle"] + list(DENSE_WORKLOADS),
                   help="pi0_ae (default: the headline line) or one dense configuration")
    return p.parse_args()


# dense configurations (parity cases of the dense path; timed on request):
# name -> (config, batch, metric, unit)
DENSE_WORKLOADS = {
    "prefill_b1": ("prefill", 1, "ms per prefix prefill", "ms"),
    "prefill_b8": ("prefill", 8, "ms per prefix prefill", "ms"),
    "dit_1p3b": ("dit_1p3b", 4, "ms per denoised chunk", "ms"),
    # steady state of the interleaved schedule through lat_dit_pipeline_push: one
    # push admits a chunk, runs latent in/out + 30 blocks for the 4 chunks in
    # flight (steps 0..3) and completes one chunk
    "dit_1p3b_pipeline": ("dit_1p3b", 4, "ms per denoised chunk", "ms"),
    "dit_14b_n1": ("dit_14b", 1, "us per block", "us"),
    "dit_14b_n4": ("dit_14b", 4, "us per block", "us"),
    "dit_14b_n8": ("dit_14b", 8, "us per block", "us"),
    # the 1.3B chunk with the Wan-class options: 3-D RoPE over one 30 x 52 frame
    # per chunk, cross-attention to 512 text tokens, rings in pages of 256 tokens
    "dit_1p3b_wan": ("dit_1p3b", 4, "ms per denoised chunk", "ms",
                     dict(grid_h=30, grid_w=52, text_len=512, page_tokens=256)),
}


def dist_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def aggregate(elapsed_ms, units_per_rank, world, reduce_max):
    """Whole-job numbers: max time over ranks, units summed over ranks."""
    t = reduce_max(elapsed_ms)
    return t, units_per_rank * world


def job_ms_per_chunk(elapsed_ms, steps, world, reduce_max):
    """Replicas: every rank denoises `steps` chunks of its own; the job's time is
    the slowest rank's, so the whole-job time per chunk is max_t / (steps * world).
    Returns (ms per step on the slowest rank, whole-job ms per chunk)."""
    t_max, chunks = aggregate(elapsed_ms, steps, world, reduce_max)
    return t_max / steps, t_max / chunks


def algorithmic_bytes(cfg):
    """Bytes per block-step and per chunk (weights read once + KV read once)."""
    D, F, Hq, Hkv, dh, L, S = cfg["D"], cfg["F"], cfg["Hq"], cfg["Hkv"], cfg["dh"], cfg["L"], cfg["S"]
    Tkv = cfg["T_prefix"] + cfg["T_q"]
    w_block = 2 * (D * (Hq + 2 * Hkv) * dh + Hq * dh * D + D * 2 * F + F * D)
    kv_block = 2 * 2 * Tkv * Hkv * dh
    A = cfg["act_dim"]
    per_step_extra = 2 * D * D + 4 * (A * D + D * A)          # W2 (bf16), W' and W_out (fp32)
    return w_block, kv_block, L * S * (w_block + kv_block) + S * per_step_extra


def macs(cfg):
    D, F, Hq, Hkv, dh, L, S, T = cfg["D"], cfg["F"], cfg["Hq"], cfg["Hkv"], cfg["dh"], cfg["L"], cfg["S"], cfg["T_q"]
    Tkv = cfg["T_prefix"] + T
    per_block = T * (D * (Hq + 2 * Hkv) * dh + Hq * dh * D + D * 2 * F + F * D) + 2 * T * Hq * Tkv * dh
    return per_block, per_block * L * S


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)), "samples": len(sm),
                "reasons": sorted(reasons)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def cpu_baseline(cfg, wb, ib):
    """The oracle as it stands, one full denoised chunk on the host cores."""
    from oracle import pi0
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1)))
    blocks = [pi0.method_block(pi0.decode_tree(b)) for b in wb["blocks"]]
    t0 = time.perf_counter()
    pi0.denoise(ib["noise"], ib["state"], ib["kv"], wb, cfg, blocks=blocks)
    ms = (time.perf_counter() - t0) * 1e3
    return {"value": round(ms, 3), "unit": "ms", "cores": cores, "kind": "oracle",
            "sample": "one full chunk (18 blocks x 10 steps), float64 numpy, weights pre-decoded"}


def run_reference(args):
    """The oracle as it stands on the host cores: every step is one whole
    denoise step of the chunk (state row + embedding, all 18 blocks, head and
    Euler update), steps cycling through the chunk's 10 denoise steps and
    starting a new chunk after the last; ms_per_step x steps is the timed time
    and the value, ms per chunk, is ms_per_step x 10."""
    rank, _, world = dist_info()
    if rank != 0:
        return
    from latency_transformer_block_gb300 import synth
    from oracle import bf16, pi0
    cfg = synth.config(WORKLOAD)
    wb = synth.pi0_weights(cfg, 0)
    ib = synth.pi0_inputs(cfg, 0)
    blocks = [pi0.method_block(pi0.decode_tree(b)) for b in wb["blocks"]]
    W = pi0.decode_tree({k: v for k, v in wb.items() if k != "blocks"})
    kv = bf16.decode(ib["kv"])
    Tp, Tq, S, L, D = cfg["T_prefix"], cfg["T_q"], cfg["S"], cfg["L"], cfg["D"]
    pos = Tp + np.arange(Tq)
    times = pi0.times(cfg)
    st = pi0.state_token(ib["state"].astype(np.float64), W)
    state = {"x": ib["noise"].astype(np.float64), "s": 0}

    def one():
        s = state["s"]
        x = state["x"] if s > 0 else ib["noise"].astype(np.float64)
        h = np.vstack([st[None, :], pi0.embed(x, times[s], W, D)])
        for l in range(L):
            h, _, _ = pi0.block(h, kv[l, 0, :Tp], kv[l, 1, :Tp], pos, blocks[l], cfg)
        state["x"] = x + (1.0 / S) * pi0.head(h[1:], W, cfg["eps"])
        state["s"] = (s + 1) % S

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    ms_step = (time.perf_counter() - t0) * 1e3 / args.steps
    value = ms_step * S
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1)))
    line = {
        "impl": "reference", "metric": "ms per denoised chunk", "value": round(value, 3), "unit": "ms",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) inputs, N(0,0.02) bf16 weights)",
        "config": {"workload": WORKLOAD, "blocks": L, "steps": S, "tokens": Tq, "prefix_kv": Tp,
                   "step_unit": "one denoise step of the chunk (18 blocks + embedding + head); value = 10 steps",
                   "us_per_block": round(ms_step * 1e3 / L, 1)},
        "cpu_baseline": {"value": round(value, 3), "unit": "ms", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} timed denoise steps of pi0_ae chunks (each 18 blocks + "
                                   f"embedding + head, float64 numpy), x{S} per chunk"},
        "e2e": {"value": round(value, 3), "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    rank, local_rank, world = dist_info()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    from latency_transformer_block_gb300 import build as B
    B.build()
    from latency_transformer_block_gb300 import synth
    from latency_transformer_block_gb300.models import Pi0ActionExpert

    cfg = synth.config(WORKLOAD)
    wb = synth.pi0_weights(cfg, 0)
    ib = synth.pi0_inputs(cfg, 0)
    m = Pi0ActionExpert(cfg, wb, device=dev)
    kv = m.kv_from_bits(ib["kv"])
    state = torch.from_numpy(ib["state"]).to(dev)
    noise = torch.from_numpy(ib["noise"]).to(dev)
    x = noise.clone()
    stream = torch.cuda.Stream(dev)

    def step():
        x.copy_(noise, non_blocking=True)
        m.denoise(kv, state, x, stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
    stream.synchronize()
    m.ctx.sync()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def reduce_max(v):
        if world == 1:
            return v
        t = torch.tensor([v], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())

    clocks = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    m.ctx.sync()
    elapsed = e0.elapsed_time(e1)
    ms_per_step, value = job_ms_per_chunk(elapsed, args.steps, world, reduce_max)

    # --- end to end through the C ABI with host buffers (pinned), copies timed ---
    h_noise = torch.from_numpy(ib["noise"]).pin_memory()
    h_state = torch.from_numpy(ib["state"]).pin_memory()
    h_out = torch.empty_like(h_noise).pin_memory()
    with torch.cuda.stream(stream):
        for _ in range(3):
            x.copy_(h_noise, non_blocking=True)
            state.copy_(h_state, non_blocking=True)
            m.denoise(kv, state, x, stream)
            h_out.copy_(x, non_blocking=True)
        stream.synchronize()
        t0 = time.perf_counter()
        ee0, ee1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ee0.record(stream)
        for _ in range(args.steps):
            x.copy_(h_noise, non_blocking=True)
            state.copy_(h_state, non_blocking=True)
            m.denoise(kv, state, x, stream)
            h_out.copy_(x, non_blocking=True)
        ee1.record(stream)
        stream.synchronize()
        host_ms = (time.perf_counter() - t0) * 1e3
    e2e_ms = reduce_max(max(ee0.elapsed_time(ee1), host_ms)) / args.steps

    # --- dominant kernel alone: the persistent step kernel, one launch per
    #     chunk (embedding, W2, every block and the head of all denoise steps),
    #     timed back to back with events on its stream; each chunk starts from
    #     the previous one's actions (a second buffer, so no copy in between;
    #     the captured graph holds the launch and its 128-byte barrier clear) ---
    peak_gbs, peak_tf, peak_src = measured_peaks()
    w_block, kv_block, bytes_chunk = algorithmic_bytes(cfg)
    mac_block, mac_chunk = macs(cfg)
    reps = 10
    x2 = noise.clone()
    with torch.cuda.stream(stream):
        for _ in range(3):
            m.denoise(kv, state, x2, stream)
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record(stream)
        for _ in range(reps):
            m.denoise(kv, state, x2, stream)
        k1.record(stream)
        stream.synchronize()
    m.ctx.sync()
    launch_us = k0.elapsed_time(k1) * 1e3 / reps
    launch_gbs = bytes_chunk / launch_us / 1e3
    path_gbs = bytes_chunk / (ms_per_step * 1e-3) / 1e9
    # our kernels per chunk: the one step-kernel launch
    launches_per_chunk = 1

    line = {
        "metric": "ms per denoised chunk", "value": round(value, 4), "unit": "ms", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": False, "scaling": "weak",
        "vs_baseline": round(value / PAGES_AE_MS, 4), "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) inputs and prefix KV, N(0,0.02) bf16 weights)",
        "config": {"workload": WORKLOAD, "blocks": cfg["L"], "steps": cfg["S"], "tokens": cfg["T_q"],
                   "prefix_kv": cfg["T_prefix"], "width": cfg["D"], "ffn": cfg["F"],
                   "us_per_block": round(ms_per_step * 1e3 / (cfg["L"] * cfg["S"]), 3),
                   "tokens_per_s": round(cfg["T_q"] * 1e3 / ms_per_step, 1),
                   "l2": "inputs larger than L2: 623 MB of block weights streamed per step",
                   "path_roofline_ms": round(bytes_chunk / (peak_gbs * 1e9) * 1e3, 4),
                   "path_hbm_gbs": round(path_gbs, 1), "path_frac": round(path_gbs / peak_gbs, 4),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm",
                     "kernel": f"pi0_step_kernel (the whole chunk: {cfg['S']} steps x {cfg['L']} blocks, one launch)",
                     "achieved": round(launch_gbs, 1), "peak": peak_gbs, "unit": "GB/s",
                     "frac": round(launch_gbs / peak_gbs, 4), "traffic": STEP_TRAFFIC,
                     "algorithmic_bytes": bytes_chunk, "us_per_launch": round(launch_us, 2),
                     "peak_source": f"{peak_src} hbm_gbs (burst copy)"},
        "clocks": clk,
        "e2e": {"value": round(e2e_ms, 4), "unit": "ms",
                "h2d_bytes_per_step": int(h_noise.numel() * 4 + h_state.numel() * 4),
                "d2h_bytes_per_step": int(h_out.numel() * 4)},
        "gpu_launches": launches_per_chunk * args.steps,
    }
    if rank == 0 and not args.no_dense:
        # the dense configurations, each timed with CUDA events in this same run
        # (one model at a time; device memory freed in between)
        del m, kv
        torch.cuda.empty_cache()
        line["config"]["dense"] = {}
        for name in DENSE_WORKLOADS:
            r = dense_measure(name, max(3, min(args.steps, 10)), 3, dev)
            line["config"]["dense"][name] = r["summary"]
            torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, wb, ib)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def dense_flops(cfg, nb, descs=None):
    """Useful FLOPs of one step of a dense workload (2 per multiply-add): the
    method's projections and its dense attention; for the prefix model the last
    layer computes K and V only."""
    D, F, Hq, Hkv, dh, L = cfg["D"], cfg["F"], cfg["Hq"], cfg.get("Hkv", cfg["Hq"]), cfg["dh"], cfg["L"]
    if cfg["kind"] == "prefill":
        tok = nb * cfg["T_prefix"]
        qd, kvd = Hq * dh, Hkv * dh
        proj = D * (qd + 2 * kvd) + qd * D + D * 2 * F + F * D
        attn = 2 * nb * Hq * cfg["T_prefix"] * cfg["T_prefix"] * dh
        macs = tok * cfg["patch_dim"] * D + (L - 1) * (tok * proj + attn) + tok * D * 2 * kvd
        return 2 * macs
    T, nh = cfg["T_chunk"], cfg["n_hist"]
    per_chunk_proj = T * (D * 3 * D + D * D + D * F + F * D)
    tl = cfg.get("text_len", 0)
    per_chunk_cross = T * 2 * D * D + 2 * T * tl * D if tl else 0   # q, o projections; scores and P V
    macs = 0
    for (_, c, _) in descs:
        macs += per_chunk_proj + 2 * T * T * (1 + min(c, nh)) * D + per_chunk_cross
    return 2 * macs * L


def device_weights(make, cfg, dev, seed=0):
    """Synthetic weights of the architecture for timing only, drawn on the
    device with the generator's layout and distributions (N(0, 0.02) bf16,
    norm scales 1 + N(0, 0.02)): the host generator would spend minutes on the
    gigabytes of prefix and DiT weights.  Parity runs use the host generator."""
    import torch
    tmpl = make(dict(cfg, L=1), seed)          # one block: names and shapes
    g = torch.Generator(device=dev)
    g.manual_seed(seed)

    def draw(name, a):
        t = torch.randn(a.shape, generator=g, device=dev) * 0.02
        if name.startswith("g_"):
            t += 1.0
        return t.to(torch.bfloat16)
    out = {k: draw(k, v) for k, v in tmpl.items() if k != "blocks"}
    blk = tmpl["blocks"][0]
    out["blocks"] = [{k: draw(k, v) for k, v in blk.items()} for _ in range(cfg["L"])]
    return out


def dense_measure(workload, steps, warmup, dev, layers=0):
    """Time one dense configuration (CUDA events on its stream) and the dense
    GEMM alone on its FFN-in projection; returns the full line and a summary.
    layers > 0 runs that many blocks instead of the configuration's."""
    import torch
    from latency_transformer_block_gb300 import build as B
    B.build()
    from latency_transformer_block_gb300 import synth
    from latency_transformer_block_gb300.models import DitStage, Pi0Prefix
    name, nb, metric, unit = DENSE_WORKLOADS[workload][:4]
    over = dict(DENSE_WORKLOADS[workload][4]) if len(DENSE_WORKLOADS[workload]) > 4 else {}
    if layers > 0:
        over["L"] = layers
    cfg = synth.config(name, **over)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    stream = torch.cuda.Stream(dev)
    if cfg["kind"] == "prefill":
        m = Pi0Prefix(cfg, device_weights(synth.prefill_weights, cfg, dev), max_batch=nb, device=dev)
        pe = torch.randn(nb, cfg["T_prefix"], cfg["patch_dim"], generator=gen, device=dev).to(torch.bfloat16)
        kv = m.new_kv(nb)
        flops = dense_flops(cfg, nb)
        rows = nb * cfg["T_prefix"]
        ffn_n, ffn_k = 2 * cfg["F"], cfg["D"]

        def step():
            m.prefill(pe, kv, stream)
        blocks = cfg["L"]
    elif workload.endswith("_pipeline"):
        m = DitStage(cfg, device_weights(synth.dit_weights, cfg, dev), max_batch=nb, n_streams=1, device=dev)
        ring = torch.randn(1, cfg["L"], cfg["S"], cfg["n_hist"] + 1, 2, cfg["T_chunk"], cfg["D"],
                           generator=gen, device=dev).to(torch.bfloat16)
        noise = torch.randn(cfg["T_chunk"], cfg["lat_dim"], generator=gen, device=dev)
        done = torch.empty_like(noise)
        cfg["Hkv"] = cfg["H"]
        cfg["Hq"] = cfg["H"]
        descs = synth.dit_chunk_descs(cfg, nb, first_chunk=nb + 3)
        rows = nb * cfg["T_chunk"]
        flops = dense_flops(cfg, nb, descs) + 2 * 2.0 * rows * cfg["lat_dim"] * cfg["D"]
        ffn_n, ffn_k = cfg["F"], cfg["D"]
        for _ in range(cfg["S"] - 1):   # fill the pipeline: from here on every push completes a chunk
            m.push(ring, 0, noise, done, stream)

        def step():
            m.push(ring, 0, noise, done, stream)
        blocks = cfg["L"]
    else:
        descs = synth.dit_chunk_descs(cfg, nb)
        streams = (nb + cfg["S"] - 1) // cfg["S"]
        m = DitStage(cfg, device_weights(synth.dit_weights, cfg, dev), max_batch=nb, n_streams=streams,
                     device=dev)
        if cfg.get("page_tokens", 0):   # the rings in a pool of pages, a seeded permutation of it
            table, n_pool = synth.dit_page_table(cfg, streams, cfg["L"])
            ring = torch.randn(n_pool, 2, cfg["page_tokens"], cfg["D"], generator=gen, device=dev).to(torch.bfloat16)
            m.bind_pages(table)
        else:
            ring = torch.randn(streams, cfg["L"], cfg["S"], cfg["n_hist"] + 1, 2, cfg["T_chunk"], cfg["D"],
                               generator=gen, device=dev).to(torch.bfloat16)
        for st in range(streams if cfg.get("text_len", 0) else 0):   # each stream's text context
            m.set_text(st, torch.randn(cfg["text_len"], cfg["D"], generator=gen, device=dev).to(torch.bfloat16))
        x = torch.randn(nb, cfg["T_chunk"], cfg["D"], generator=gen, device=dev)
        cfg["Hkv"] = cfg["H"]
        cfg["Hq"] = cfg["H"]
        flops = dense_flops(cfg, nb, descs)
        rows = nb * cfg["T_chunk"]
        ffn_n, ffn_k = cfg["F"], cfg["D"]

        def step():
            for l in range(cfg["L"]):
                m.block(l, x, descs, ring, stream)
        blocks = cfg["L"]
    with torch.cuda.stream(stream):
        for _ in range(max(3, warmup)):
            step()
    stream.synchronize()
    m.ctx.sync()
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    stream.synchronize()
    clk = clocks.stop()
    m.ctx.sync()
    ms = e0.elapsed_time(e1) / steps
    peak_gbs, peak_tf, peak_src = measured_peaks()
    tflops = flops / (ms * 1e-3) / 1e12
    # dominant kernel alone: the dense tcgen05 GEMM on the FFN-in projection with
    # the path's two fp16 planes of the activation (the executed tensor work is
    # twice the useful work)
    terms = 2
    act = torch.randn(rows, terms * ffn_k, generator=gen, device=dev).to(torch.float16)
    out = torch.empty(rows, ffn_n, device=dev, dtype=torch.float32)
    reps = 10
    with torch.cuda.stream(stream):
        m.ctx.debug_dense_gemm(2, 0, act, rows, terms, out, stream)
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record(stream)
        for _ in range(reps):
            m.ctx.debug_dense_gemm(2, 0, act, rows, terms, out, stream)
        k1.record(stream)
    stream.synchronize()
    m.ctx.sync()
    g_us = k0.elapsed_time(k1) * 1e3 / reps
    g_useful = 2.0 * rows * ffn_n * ffn_k / (g_us * 1e-6) / 1e12
    value = ms if unit == "ms" else ms * 1e3 / blocks
    line = {
        "metric": metric, "value": round(value, 4), "unit": unit, "n_gpus": 1, "steps": steps,
        "warmup": warmup, "ms_per_step": round(ms, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) inputs and history, N(0,0.02) bf16 weights drawn on the device)",
        "config": {"workload": workload, "batch": nb, "blocks": blocks, **over,
                   "us_per_block": round(ms * 1e3 / blocks, 2), "useful_tflop_per_step": round(flops / 1e12, 3),
                   "path_tflops": round(tflops, 1), "path_frac": round(tflops / peak_tf, 4),
                   "l2": "inputs larger than L2 (weights and KV streamed per step)"},
        "roofline": {"bound": "tensor", "kernel": "dense_gemm_kernel (FFN-in projection, M = %d, %d planes)" % (rows, terms),
                     "achieved": round(g_useful, 1), "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": round(g_useful / peak_tf, 4), "executed_frac": round(terms * g_useful / peak_tf, 4),
                     "traffic": None, "us_per_launch": round(g_us, 1),
                     "peak_source": f"{peak_src} bf16_tflops (burst cuBLAS)"},
        "clocks": clk, "e2e": None, "gpu_launches": None,
    }
    summary = {"metric": metric, "value": round(value, 4), "unit": unit, "ms_per_step": round(ms, 4),
               "steps": steps, "us_per_block": round(ms * 1e3 / blocks, 2),
               "useful_tflops": round(tflops, 1), "path_frac_of_bf16_peak": round(tflops / peak_tf, 4),
               "ffn_in_gemm_useful_tflops": round(g_useful, 1),
               "ffn_in_gemm_frac": round(g_useful / peak_tf, 4), "sm_mhz": clk.get("sm_mhz"),
               "clock_reasons": clk.get("reasons")}
    del m
    return {"line": line, "summary": summary}


def run_dense(args):
    rank, local_rank, world = dist_info()
    if rank != 0:
        return
    import torch
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    r = dense_measure(args.workload, args.steps, args.warmup, dev, args.layers)
    if args.layers > 0:
        r["line"]["config"]["blocks_run"] = args.layers
        r["line"]["config"]["note"] = "fewer blocks than the configuration (profiling run)"
    print(json.dumps(r["line"]), flush=True)


def run_cycle(args):
    """Control cycle of the pi0 pipeline: prefill of a new observation's prefix
    KV (B = 1) and one denoised action chunk.  Sequential: both on one stream.
    Concurrent (the reading note's two-stream scheme): the prefill writes the
    next cache on one stream while the action expert works from the previous
    cache on another; the two caches swap every cycle."""
    import torch
    rank, local_rank, world = dist_info()
    if rank != 0:
        return
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from latency_transformer_block_gb300 import build as B
    B.build()
    from latency_transformer_block_gb300 import synth
    from latency_transformer_block_gb300.models import Pi0ActionExpert, Pi0Prefix

    cp, ca = synth.config("prefill"), synth.config(WORKLOAD)
    pre = Pi0Prefix(cp, synth.prefill_weights(cp, 0), max_batch=1, device=dev)
    ae = Pi0ActionExpert(ca, synth.pi0_weights(ca, 0), device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    pe = torch.randn(1, cp["T_prefix"], cp["patch_dim"], generator=gen, device=dev).to(torch.bfloat16)
    kvs = [pre.new_kv(1)[:, 0] for _ in range(2)]       # [L][2][T_prefix + T_q][Hkv dh] each
    ib = synth.pi0_inputs(ca, 0)
    state = torch.from_numpy(ib["state"]).to(dev)
    noise = torch.from_numpy(ib["noise"]).to(dev)
    x = noise.clone()
    sa, sb = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    for k in kvs:
        pre.prefill(pe, k.unsqueeze(1), sa)
    sa.synchronize()

    def cycle(i, concurrent):
        s2 = sb if concurrent else sa
        pre.prefill(pe, kvs[i % 2].unsqueeze(1), sa)
        with torch.cuda.stream(s2):
            x.copy_(noise, non_blocking=True)
        ae.denoise(kvs[(i + 1) % 2], state, x, s2)
        if concurrent:             # the cycle ends when both are done
            ea, eb = torch.cuda.Event(), torch.cuda.Event()
            ea.record(sa)
            eb.record(sb)
            sa.wait_event(eb)
            sb.wait_event(ea)

    def timed(concurrent):
        for i in range(max(3, args.warmup)):
            cycle(i, concurrent)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(sa)
        for i in range(args.steps):
            cycle(i, concurrent)
        e1.record(sa)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    seq_ms = timed(False)
    conc_ms = timed(True)
    clk = clocks.stop()
    ae.ctx.sync()
    pre.ctx.sync()
    line = {
        "metric": "ms per control cycle (prefix prefill B=1 + one denoised action chunk)",
        "value": round(conc_ms, 4), "unit": "ms", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(conc_ms, 4), "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) inputs, N(0,0.02) bf16 weights)",
        "config": {"workload": "pi0_cycle", "sequential_ms": round(seq_ms, 4), "concurrent_ms": round(conc_ms, 4),
                   "streams": 2, "caches": 2,
                   "l2": "inputs larger than L2 (4.0 GB prefix weights + 623 MB expert weights per cycle)"},
        "roofline": None, "clocks": clk, "e2e": None, "gpu_launches": None,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "pi0_cycle":
        run_cycle(args)
    elif args.workload != WORKLOAD:
        run_dense(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
