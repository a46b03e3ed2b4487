"""One DiT block stage of chunked autoregressive denoising, float64.

Source: PhysisServe article (AREX feed, 2026-10-15), section on cutting the
pipeline into "one block at one denoise step": each chunk starts from noise and
runs several denoise steps; the next chunk does not wait for the previous one
to finish, it reads the *noisy* KV that the earlier chunks left at the current
step; a stage is one transformer block at one denoise step and the KV stays
where it was produced.  Section on one GPU running several stages: tasks of
different chunks on the same block are merged into one batch.

Readings where the pages are silent (listed in the design notes):
* Block (Wan/DiT style, adaLN): m = A[s] split into (shift1, scale1, gate1,
  shift2, scale2, gate2), each of width D;
  h  = x + gate1 * Attn(LN(x) (1 + scale1) + shift1)
  x' = h + gate2 * (GELU_tanh(u W1) W2),  u = LN(h) (1 + scale2) + shift2.
  Attention is full multi-head, no biases, RoPE (rotate-half, 1-D) on Q and K.
* A[s] = SiLU(e(t_s)) Wmod + bmod with e(t) = SiLU(temb256(t) Wt1 + bt1) Wt2 + bt2,
  t_s = s / S, shared by all blocks.
* Ring: one ring of n_hist + 1 = 5 chunk slots per (stream, block, step);
  chunk c lives in slot c mod 5.  Chunk c at step s attends to its own tokens
  and to chunks c-1 .. c-n_hist (those >= 0) of the same stream at the same
  step.  Token j of chunk c has RoPE position c * T_chunk + j.
* A batched call first writes every chunk's own K/V into its slot (bf16, the
  ring's format), then runs attention for every chunk.  A chunk's history keys
  are the ring's bf16 values; its own keys enter its attention as computed.
  Two chunks of one call may not share a (stream, step, slot).
* Latent in/out and the denoise step (the pages are silent; the plainest
  reading): a chunk's latent z [T, A] enters the stage as x = z W_in + b_in, the
  L blocks run at its step s, v = x W_out + b_out, and z <- z + dt v with
  dt = 1 / S (the same grid t_s = s / S as the adaLN table).
* Interleaved schedule (the article's steady state of one stream: the chunks
  in flight sit at different denoise steps and run through every block as one
  batch): interval i admits chunk i at step 0 and advances every chunk in
  flight by one step; chunk c leaves after interval c + S - 1.
* Wan-class options (the article names Wan backbones but specifies neither;
  cfg keys, 0 / absent = off):
  - grid_h, grid_w: 3-D RoPE.  A chunk is T / (grid_h grid_w) latent frames of
    grid_h x grid_w patches; token j of chunk c sits at (frame, y, x) =
    (c F_c + j // (grid_h grid_w), (j // grid_w) % grid_h, j % grid_w).
  - text_len: text cross-attention between self-attention and the FFN,
    h' = h + Attn(LN(h) g_c + b_c) W_o^c with q from it, k, v from the stream's
    text context ctx [text_len, D]: k = ctx W_k^c, v = ctx W_v^c; no RoPE, no
    mask, no adaLN gate.  The context's K/V are kept at full precision (not a
    bf16 cache).
  - page_tokens: the ring lives in pages of a pool through a page table; only
    addresses change (``ring_to_pool`` / ``pool_to_ring``).
"""
import numpy as np

from . import bf16
from .ops import attention, gelu_tanh, layernorm, rope, rope3d, silu, timestep_embedding


def adaln_table(W, cfg):
    """A[s] for s < S: float64 [S, 6D]."""
    S, td = cfg["S"], cfg["t_dim"]
    rows = []
    for s in range(S):
        e = silu(timestep_embedding(s / S, td) @ W["wt1"] + W["bt1"]) @ W["wt2"] + W["bt2"]
        rows.append(silu(e) @ W["wmod"] + W["bmod"])
    return np.stack(rows)


def ring_slot(c: int, n_hist: int) -> int:
    return c % (n_hist + 1)


def history_chunks(c: int, n_hist: int) -> list:
    """Earlier chunks visible to chunk c, oldest first."""
    return [c - k for k in range(n_hist, 0, -1) if c - k >= 0]


def positions(c: int, T: int) -> np.ndarray:
    return c * T + np.arange(T)


def positions3(c: int, cfg: dict) -> np.ndarray:
    """(frame, y, x) of the tokens of chunk c: int64 [T, 3]."""
    T, gh, gw = cfg["T_chunk"], cfg["grid_h"], cfg["grid_w"]
    fc = T // (gh * gw)
    j = np.arange(T)
    return np.stack([c * fc + j // (gh * gw), (j // gw) % gh, j % gw], axis=1)


def _rope_qk(y, c, cfg, rows=None):
    """RoPE of the q or k projection y[T', H, dh] of chunk c (rows: token indices
    of y's rows, all tokens when None)."""
    T, base = cfg["T_chunk"], cfg["rope_base"]
    if cfg.get("grid_h", 0):
        pos = positions3(c, cfg)
        return rope3d(y, pos if rows is None else pos[rows], base)
    pos = positions(c, T)
    return rope(y, pos if rows is None else pos[rows], base)


def _cross(h, w, ctx, cfg):
    """The text cross-attention sublayer: h + Attn(LN(h) g_c + b_c, ctx) W_o^c."""
    H, dh, eps = cfg["H"], cfg["dh"], cfg["eps"]
    u = layernorm(h, eps) * w["g_c"] + w["b_c"]
    q = (u @ w["cq"]).reshape(len(h), H, dh)
    k = (ctx @ w["ck"]).reshape(len(ctx), H, dh)
    v = (ctx @ w["cv"]).reshape(len(ctx), H, dh)
    o = attention(q, k, v, 1.0 / np.sqrt(dh)).reshape(len(h), H * dh)
    return h + o @ w["co"]


def pages_per_ring(cfg: dict) -> int:
    P = cfg["page_tokens"]
    return -(-(cfg["n_hist"] + 1) * cfg["T_chunk"] // P)


def ring_to_pool(ring, table, cfg, n_pool):
    """Scatter rings [streams, L, S, n_hist+1, 2, T, D] into a page pool
    [n_pool, 2, P, D] through table [streams, L, S, pages]: ring row r of
    (stream, block, step) = slot * T + j lives in page table[..., r // P] at
    offset r % P.  Unused pool rows are 0."""
    st, L, S, R, _, T, D = ring.shape
    P = cfg["page_tokens"]
    pool = np.zeros((n_pool, 2, P, D), dtype=ring.dtype)
    for a in range(st):
        for l in range(L):
            for s in range(S):
                flat = ring[a, l, s].transpose(1, 0, 2, 3).reshape(2, R * T, D)
                for r in range(R * T):
                    pool[table[a, l, s, r // P], :, r % P] = flat[:, r]
    return pool


def pool_to_ring(pool, table, cfg, streams, L):
    """The inverse of ``ring_to_pool``."""
    S, R, T, P = cfg["S"], cfg["n_hist"] + 1, cfg["T_chunk"], cfg["page_tokens"]
    D = pool.shape[-1]
    ring = np.zeros((streams, L, S, R, 2, T, D), dtype=pool.dtype)
    for a in range(streams):
        for l in range(L):
            for s in range(S):
                for r in range(R * T):
                    ring[a, l, s, r // T, :, r % T] = pool[table[a, l, s, r // P], :, r % P]
    return ring


def _split6(a, D):
    return [a[i * D:(i + 1) * D] for i in range(6)]


def block_batch(xs, descs, ring, table, w, cfg, text=None):
    """One DiT block for a batch of chunks.

    xs[n, T, D] residual streams (fp32/fp64); descs: list of (stream, chunk, step);
    ring: float64 [streams, S, n_hist+1, 2, T, D] for this block, modified in
    place (own K/V written, bf16-rounded); table[S, 6D]; w: block weights
    (float64); text[stream]: the text contexts [text_len, D] (cfg text_len > 0).
    Returns x'[n, T, D].
    """
    D, H, dh, T, nh = cfg["D"], cfg["H"], cfg["dh"], cfg["T_chunk"], cfg["n_hist"]
    eps = cfg["eps"]
    n = len(descs)
    seen = set()
    for (st, c, s) in descs:
        key = (st, s, ring_slot(c, nh))
        assert key not in seen, "two chunks of one call share a ring slot"
        seen.add(key)
    qs, mods, own = [], [], []
    # phase 1: norm + modulation + QKV + RoPE; own K/V into the ring
    for b, (st, c, s) in enumerate(descs):
        sh1, sc1, g1, sh2, sc2, g2 = _split6(table[s], D)
        mods.append((sh1, sc1, g1, sh2, sc2, g2))
        u = layernorm(np.asarray(xs[b], np.float64), eps) * (1.0 + sc1) + sh1
        q = _rope_qk((u @ w["wq"]).reshape(T, H, dh), c, cfg)
        k = _rope_qk((u @ w["wk"]).reshape(T, H, dh), c, cfg)
        v = (u @ w["wv"]).reshape(T, H, dh)
        ring[st, s, ring_slot(c, nh), 0] = bf16.round_rne(k.reshape(T, D))
        ring[st, s, ring_slot(c, nh), 1] = bf16.round_rne(v.reshape(T, D))
        qs.append(q)
        own.append((k.reshape(T, D), v.reshape(T, D)))
    # phase 2: attention over history + own, then the rest of the block
    out = np.empty((n, T, D))
    for b, (st, c, s) in enumerate(descs):
        sh1, sc1, g1, sh2, sc2, g2 = mods[b]
        hist = history_chunks(c, nh)
        K = np.concatenate([ring[st, s, ring_slot(cc, nh), 0] for cc in hist] + [own[b][0]])
        V = np.concatenate([ring[st, s, ring_slot(cc, nh), 1] for cc in hist] + [own[b][1]])
        o = attention(qs[b], K.reshape(-1, H, dh), V.reshape(-1, H, dh),
                      1.0 / np.sqrt(dh)).reshape(T, D)
        h = np.asarray(xs[b], np.float64) + g1 * (o @ w["wo"])
        if cfg.get("text_len", 0):
            h = _cross(h, w, np.asarray(text[st], np.float64), cfg)
        u2 = layernorm(h, eps) * (1.0 + sc2) + sh2
        out[b] = h + g2 * (gelu_tanh(u2 @ w["w1"]) @ w["w2"])
    return out


def block_batch_rows(xs, descs, ring, table, w, cfg, rows, text=None):
    """Same block, but only output rows ``rows`` (token indices) of every chunk.

    K/V of every token are still computed (attention needs all of them); the
    query-side work is done for the sampled rows only.  Returns x'[n, len(rows), D]
    and updates ``ring`` like ``block_batch``.
    """
    D, H, dh, T, nh = cfg["D"], cfg["H"], cfg["dh"], cfg["T_chunk"], cfg["n_hist"]
    eps = cfg["eps"]
    rows = np.asarray(rows)
    qs, mods, own = [], [], []
    for b, (st, c, s) in enumerate(descs):
        sh1, sc1, g1, sh2, sc2, g2 = _split6(table[s], D)
        mods.append((sh1, sc1, g1, sh2, sc2, g2))
        u = layernorm(np.asarray(xs[b], np.float64), eps) * (1.0 + sc1) + sh1
        k = _rope_qk((u @ w["wk"]).reshape(T, H, dh), c, cfg)
        v = (u @ w["wv"]).reshape(T, H, dh)
        ring[st, s, ring_slot(c, nh), 0] = bf16.round_rne(k.reshape(T, D))
        ring[st, s, ring_slot(c, nh), 1] = bf16.round_rne(v.reshape(T, D))
        own.append((k.reshape(T, D), v.reshape(T, D)))
        qs.append(_rope_qk((u[rows] @ w["wq"]).reshape(len(rows), H, dh), c, cfg, rows))
    out = np.empty((len(descs), len(rows), D))
    for b, (st, c, s) in enumerate(descs):
        sh1, sc1, g1, sh2, sc2, g2 = mods[b]
        hist = history_chunks(c, nh)
        K = np.concatenate([ring[st, s, ring_slot(cc, nh), 0] for cc in hist] + [own[b][0]])
        V = np.concatenate([ring[st, s, ring_slot(cc, nh), 1] for cc in hist] + [own[b][1]])
        o = attention(qs[b], K.reshape(-1, H, dh), V.reshape(-1, H, dh),
                      1.0 / np.sqrt(dh)).reshape(len(rows), D)
        h = np.asarray(xs[b], np.float64)[rows] + g1 * (o @ w["wo"])
        if cfg.get("text_len", 0):
            h = _cross(h, w, np.asarray(text[st], np.float64), cfg)
        u2 = layernorm(h, eps) * (1.0 + sc2) + sh2
        out[b] = h + g2 * (gelu_tanh(u2 @ w["w1"]) @ w["w2"])
    return out


def stage_interval(lats, descs, rings, table, W, cfg, text=None):
    """One interval: chunk b of the batch (stream, chunk, step) = descs[b] runs
    x = z W_in + b_in, all L blocks at its step, v = x W_out + b_out and the
    Euler update z + dt v.

    lats: list of [T, A] latents; rings: float64 [streams, L, S, n_hist+1, 2, T, D]
    (modified in place, one ring per block as in ``block_batch``); table: the
    adaLN table [S, 6D]; W: weights with "blocks", "w_in", "b_in", "w_out", "b_out".
    Returns the updated latents.
    """
    dt = 1.0 / cfg["S"]
    xs = np.stack([np.asarray(z, np.float64) @ W["w_in"] + W["b_in"] for z in lats])
    for l, wl in enumerate(W["blocks"]):
        xs = block_batch(xs, descs, rings[:, l], table, wl, cfg, text)
    return [np.asarray(lats[b], np.float64) + dt * (xs[b] @ W["w_out"] + W["b_out"])
            for b in range(len(descs))]


def interval_descs(i: int, n_chunks: int, S: int, stream: int = 0) -> list:
    """Chunks in flight during interval i of one stream, as (stream, chunk, step):
    chunk c is at step i - c; ordered by chunk slot c mod S."""
    chunks = [c for c in range(max(0, i - S + 1), min(i, n_chunks - 1) + 1)]
    return sorted(((stream, c, i - c) for c in chunks), key=lambda d: d[1] % S)


def pipeline(noises, rings, table, W, cfg, stream=0, text=None):
    """Interleaved schedule over a stream of chunks; returns their final latents
    in chunk order (chunk c is done after interval c + S - 1)."""
    S, n = cfg["S"], len(noises)
    live = {}
    done = [None] * n
    for i in range(n + S - 1):
        if i < n:
            live[i] = np.asarray(noises[i], np.float64)
        descs = interval_descs(i, n, S, stream)
        new = stage_interval([live[c] for (_, c, _) in descs], descs, rings, table, W, cfg, text)
        for (_, c, _), z in zip(descs, new):
            live[c] = z
        if i - (S - 1) >= 0:
            done[i - (S - 1)] = live.pop(i - (S - 1))
    return done


def sequential(noises, rings, table, W, cfg, stream=0, text=None):
    """The plain order: every step of chunk c before chunk c + 1."""
    out = []
    for c, z in enumerate(noises):
        z = np.asarray(z, np.float64)
        for s in range(cfg["S"]):
            z = stage_interval([z], [(stream, c, s)], rings, table, W, cfg, text)[0]
        out.append(z)
    return out

