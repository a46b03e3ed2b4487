"""Phase table of the persistent step kernel (pi0 action expert) from its
device timestamps (lat_debug_trace).

  python -m latency_transformer_block_gb300.step_trace [--workload pi0_ae] [--chunks 3]

Runs `--chunks` denoised chunks with the trace enabled (one launch each; every
denoise step writes the same slots, so the buffer holds the last step of the
last chunk) and prints, per phase of a block, the median over the blocks of
one denoise step of
  work    = last CTA finishing the phase - first CTA starting it,
  barrier = first CTA starting the next phase - last CTA finishing this one,
plus the sub-steps of the projection phases (median over the CTAs that take
part): first activation tile, operand built, accumulator complete, epilogue
done, each relative to the CTA's own phase start.

Timestamps are the GPU's global timer (ns) written by thread 0 of each CTA's
math warps; the trace changes nothing in the kernel's work but the writes.
"""
import argparse
import sys

import numpy as np

# trace slots (the kernel's layout: 64 per CTA per block)
PHASES = [  # (name, start slot, end slot)
    ("QKV projection + head-group finalize", 1, 2),
    ("attention", 5, 6),
    ("combine", 7, 8),
    ("O projection + residual", 9, 10),
    ("gate/up projection + GeGLU tiles", 11, 12),
    ("down projection + residual", 15, 16),
]
PROJ_SLOTS = {"QKV": (1, 20), "O": (9, 24), "gate/up": (11, 28), "down": (15, 32)}
SUB = ["first tile", "operand built", "accumulator complete", "epilogue done"]


def phase_table(tr: np.ndarray):
    """tr: int64 [blocks][grid][64] timestamps (0 = not written)."""
    L, G, _ = tr.shape
    work = np.zeros((L, len(PHASES)))
    bar = np.full((L, len(PHASES)), np.nan)
    for l in range(L):
        for i, (_, s, e) in enumerate(PHASES):
            st = tr[l, :, s].astype(np.float64)
            en = tr[l, :, e].astype(np.float64)
            work[l, i] = (en.max() - st[st > 0].min()) / 1e3
            if i + 1 < len(PHASES):
                nxt = tr[l, :, PHASES[i + 1][1]].astype(np.float64)
            elif l + 1 < L:
                nxt = tr[l + 1, :, PHASES[0][1]].astype(np.float64)
            else:
                continue
            bar[l, i] = (nxt[nxt > 0].min() - en.max()) / 1e3
    sub = {}
    for name, (s0, base) in PROJ_SLOTS.items():
        vals = []
        for l in range(L):
            st = tr[l, :, s0].astype(np.float64)
            rows = tr[l, :, base:base + 4].astype(np.float64)
            ok = (rows > 0).all(axis=1)
            if ok.any():
                vals.append(np.median((rows[ok] - st[ok, None]) / 1e3, axis=0))
        sub[name] = np.median(np.array(vals), axis=0) if vals else None
    return work, bar, sub


def spread(tr: np.ndarray):
    """Per projection, percentiles over (block, CTA) of the sub-steps and of
    the CTA's own end of the phase, relative to the first CTA starting it."""
    res = {}
    ends = {"QKV": 2, "O": 10, "gate/up": 12, "down": 16}
    xrecv = {"QKV": 38, "O": 39, "gate/up": 40, "down": 41}
    for name, (s0, base) in PROJ_SLOTS.items():
        vals = []
        for l in range(tr.shape[0]):
            st = tr[l, :, s0].astype(np.float64)
            t0 = st[st > 0].min()
            rows = tr[l, :, base:base + 4].astype(np.float64)
            ok = (rows > 0).all(axis=1)
            if ok.any():
                xr = tr[l, ok, xrecv[name]][:, None].astype(np.float64)
                xr = np.where(xr > 0, xr, np.nan)
                v = np.concatenate([rows[ok], xr, tr[l, ok, ends[name]][:, None].astype(np.float64)], axis=1)
                vals.append((v - t0) / 1e3)
        if vals:
            v = np.concatenate(vals)
            res[name] = np.nanpercentile(v, [10, 50, 90, 100], axis=0)
    return res


STEP_EDGES = [  # (name, trace row: 0 = first block, -1 = last block, start slot, end slot)
    ("head of the previous step + embedding", 0, 42, 43),
    ("W2 projection (embedding)", 0, 44, 49),
    ("head of the last step", -1, 50, 51),
]


def step_edges(tr: np.ndarray):
    """The chunk's per-step phases around the blocks: work (last CTA end -
    first CTA start) and the barrier to the next phase, us."""
    res = []
    nxt_slot = {42: (0, 44), 44: (0, 1)}
    for name, row, s0, s1 in STEP_EDGES:
        st = tr[row, :, s0].astype(np.float64)
        en = tr[row, :, s1].astype(np.float64)
        if not (st > 0).any():
            continue
        work = (en[en > 0].max() - st[st > 0].min()) / 1e3
        bar = float("nan")
        if s0 in nxt_slot:
            r, ns = nxt_slot[s0]
            nx = tr[r, :, ns].astype(np.float64)
            if (nx > 0).any():
                bar = (nx[nx > 0].min() - en[en > 0].max()) / 1e3
        res.append((name, work, bar))
    return res


HEAD = [("actions loaded", 52), ("row loaded, sum of squares", 53), ("W_out in shared memory", 54),
        ("head dot products", 55), ("actions updated", 56), ("embedding stored", 57)]


def head_spread(tr: np.ndarray):
    """Sub-steps of the head + embedding phase (first block's row) and of the
    last head (last block's row): percentiles over the CTAs that run them, us
    from the first CTA's phase start."""
    res = {}
    for name, row, s0, marks in (("head of the previous step + embedding", 0, 42, HEAD),
                                 ("head of the last step", -1, 50, HEAD[:5])):
        st = tr[row, :, s0].astype(np.float64)
        if not (st > 0).any():
            continue
        t0 = st[st > 0].min()
        cols = tr[row, :, [m for _, m in marks]].T.astype(np.float64)
        ok = (cols > 0).all(axis=1)
        if ok.any():
            res[name] = (marks, np.percentile((cols[ok] - t0) / 1e3, [10, 50, 90, 100], axis=0))
    return res


ATTN = [("q and key tiles loaded", 17), ("own-key lo planes loaded", 18), ("P V done", 19), ("partials stored", 6)]
COMB = [("weights of the rows", 36), ("merged, planes stored", 37)]


def attention_spread(tr: np.ndarray):
    """Attention and combine sub-steps: percentiles over (block, CTA) of each
    mark, us from the first CTA's phase start."""
    res = {}
    for name, s0, marks in (("attention", 5, ATTN), ("combine", 7, COMB)):
        vals = []
        for l in range(tr.shape[0]):
            st = tr[l, :, s0].astype(np.float64)
            t0 = st[st > 0].min()
            cols = tr[l, :, [m for _, m in marks]].T.astype(np.float64)
            ok = (cols > 0).all(axis=1)
            if ok.any():
                vals.append((cols[ok] - t0) / 1e3)
        if vals:
            res[name] = (marks, np.percentile(np.concatenate(vals), [10, 50, 90, 100], axis=0))
    return res


def report(tr: np.ndarray, out=sys.stdout):
    work, bar, sub = phase_table(tr)
    mw = np.median(work, axis=0)
    # the last phase of the last block has no next phase: its column may be all NaN
    mb = np.array([np.nanmedian(c) if np.isfinite(c).any() else np.nan for c in bar.T])
    print("| phase | work us | barrier us |", file=out)
    print("|---|---|---|", file=out)
    for i, (name, _, _) in enumerate(PHASES):
        print(f"| {name} | {mw[i]:.2f} | {mb[i]:.2f} |", file=out)
    per_block = np.median(work.sum(axis=1) + np.nan_to_num(bar).sum(axis=1))
    print(f"| total | {mw.sum():.2f} | {np.nansum(mb):.2f} ({per_block:.1f} us per block) |", file=out)
    edges = step_edges(tr)
    if edges:
        print("", file=out)
        print("| per-step phase | work us | barrier us |", file=out)
        print("|---|---|---|", file=out)
        for name, w, b in edges:
            print(f"| {name} | {w:.2f} | {b:.2f} |", file=out)
    print("", file=out)
    print("| projection | " + " | ".join(SUB) + " |", file=out)
    print("|---|" + "---|" * len(SUB), file=out)
    for name, v in sub.items():
        if v is not None:
            print(f"| {name} | " + " | ".join(f"{x:.2f}" for x in v) + " |", file=out)
    print("", file=out)
    print("Spread over CTAs (us from the first CTA's phase start; p10 / p50 / p90 / max):", file=out)
    print("", file=out)
    print("| projection | " + " | ".join(SUB) + " | cluster exchange received | CTA's phase end |", file=out)
    print("|---|" + "---|" * (len(SUB) + 2), file=out)
    for name, q in spread(tr).items():
        print(f"| {name} | " + " | ".join(" / ".join(f"{q[i, j]:.2f}" for i in range(4)) for j in range(q.shape[1]))
              + " |", file=out)
    print("", file=out)
    for name, (marks, q) in list(attention_spread(tr).items()) + list(head_spread(tr).items()):
        print(f"{name} (us from the first CTA's phase start; p10 / p50 / p90 / max):", file=out)
        for j, (label, _) in enumerate(marks):
            print(f"  {label}: " + " / ".join(f"{q[i, j]:.2f}" for i in range(4)), file=out)


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--workload", default="pi0_ae")
    p.add_argument("--chunks", type=int, default=3)
    args = p.parse_args()
    import torch

    from latency_transformer_block_gb300 import synth
    from latency_transformer_block_gb300.models import Pi0ActionExpert

    cfg = synth.config(args.workload)
    wb = synth.pi0_weights(cfg, 0)
    ib = synth.pi0_inputs(cfg, 0)
    m = Pi0ActionExpert(cfg, wb, device="cuda:0")
    kv = m.kv_from_bits(ib["kv"])
    state = torch.from_numpy(ib["state"]).cuda()
    noise = torch.from_numpy(ib["noise"]).cuda()
    x = noise.clone()
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros(cfg["L"] * grid * 64, dtype=torch.int64, device="cuda")
    m.ctx.debug_trace(buf)
    for _ in range(args.chunks):
        x.copy_(noise)
        buf.zero_()
        m.denoise(kv, state, x)
    m.ctx.sync()
    m.ctx.debug_trace(None)
    # every step of the chunk's launch writes the same slots: the last one stays
    tr = buf.view(cfg["L"], grid, 64).cpu().numpy()
    ctas = int((tr[0] != 0).any(axis=1).sum())   # the buffer has a row per SM; the launch uses fewer CTAs
    print(f"step kernel phases, workload {args.workload}: {cfg['L']} blocks of the last denoise step, "
          f"{ctas} CTAs")
    report(tr)


if __name__ == "__main__":
    main()
