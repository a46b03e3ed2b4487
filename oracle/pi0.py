"""pi0 action expert and its prefix prefill, float64.

Source: "Running VLAs at Real-time Speed" (reading note on arXiv 2510.26742),
section 2 and Fig. 4 (63 action tokens + 1 state token = 64 positions, actions
and state padded to 32 dims, 10 flow-matching steps, a vision/language prefix
whose KV cache is computed once and reused by every denoise step of the action
expert), section 4 (folds; the last prefix layer only needs its K and V) and
section 9 (same inputs and same initial noise when comparing).

Readings where the pages are silent (listed in the design notes):
* Blocks are pre-norm: h = x + Attn(RMSNorm_g1(x)); x' = h + FFN(RMSNorm_g2(h)),
  FFN(u) = (GELU_tanh(u Wg) * (u Wu)) Wd, no biases inside blocks.
* Attention is bidirectional over [prefix cache | own 64 tokens], multi-query
  (all q heads share the single KV head).  K is stored after RoPE.  The own
  tokens' K and V are written into cache slots T_prefix .. T_prefix+63 in the
  cache's bf16 format for later readers; the block's own attention uses them as
  computed (the prefix keys are the cache's bf16 values).
* Positions: prefix token i -> i; query token j (j = 0 is the state token) ->
  T_prefix + j.
* Time grid t_s = s / S, dt = 1 / S; x_{s+1} = x_s + dt * v(x_s, t_s).
* Embedding of action rows: SiLU([x W_in + b_in ; temb(t)] W1 + b1) W2 + b2
  (temb of width D); state row: state W_state + b_state (independent of t).
* Head: v = RMSNorm_gf(h[1:]) W_out + b_out on the 63 action rows.

The block weights used by the method are the folded, bf16-stored ones
(``fold.fold_scale``); ``method_block`` builds them, ``block`` runs the block
for any (g, W) pair, so the same code checks the fold identity.
"""
import numpy as np

from . import bf16
from .fold import fold_scale, merge_columns, time_fold
from .ops import attention, gelu_tanh, rmsnorm, rope, silu, timestep_embedding


def decode_tree(bits):
    if isinstance(bits, dict):
        return {k: decode_tree(v) for k, v in bits.items()}
    if isinstance(bits, list):
        return [decode_tree(v) for v in bits]
    if isinstance(bits, np.ndarray) and bits.dtype == np.uint16:
        return bf16.decode(bits)
    return bits


def method_block(blk: dict) -> dict:
    """Stored weights of one block after the RMSNorm-scale fold (g -> 1)."""
    D = blk["wq"].shape[0]
    one = np.ones(D)
    return {
        "g_attn": one,
        "wq": fold_scale(blk["g_attn"], blk["wq"]),
        "wk": fold_scale(blk["g_attn"], blk["wk"]),
        "wv": fold_scale(blk["g_attn"], blk["wv"]),
        "wo": blk["wo"],
        "g_ffn": one,
        "wg": fold_scale(blk["g_ffn"], blk["wg"]),
        "wu": fold_scale(blk["g_ffn"], blk["wu"]),
        "wd": blk["wd"],
    }


def qkv(x, w, cfg):
    """Merged projection of the normed input; returns q[T,Hq,dh], k, v[T,Hkv,dh]."""
    T = x.shape[0]
    Hq, Hkv, dh = cfg["Hq"], cfg["Hkv"], cfg["dh"]
    xn = rmsnorm(x, cfg["eps"]) * w["g_attn"]
    y = xn @ merge_columns(w["wq"], w["wk"], w["wv"])
    q = y[:, : Hq * dh].reshape(T, Hq, dh)
    k = y[:, Hq * dh: (Hq + Hkv) * dh].reshape(T, Hkv, dh)
    v = y[:, (Hq + Hkv) * dh:].reshape(T, Hkv, dh)
    return q, k, v


def chunk_mask(T, Tp, cfg):
    """Which keys [prefix | own] each query token of the chunk sees: all of
    them (default, bidirectional), or with cfg["prefix_lm"] the block mask of the
    pi0 model, where the state token (query 0) sees the prefix and itself only
    and the action tokens see everything.  None when nothing is masked."""
    if not cfg.get("prefix_lm"):
        return None
    allow = np.ones((T, Tp + T), dtype=bool)
    allow[0, Tp + 1:] = False
    return allow


def block(x, k_prefix, v_prefix, pos, w, cfg, kv_only=False):
    """One pre-norm block over [prefix KV | own tokens].

    x[T, D] residual stream; k_prefix/v_prefix[Tp, Hkv*dh] cached (post-RoPE);
    pos[T] positions of the own tokens.  Returns (x', k_own, v_own), k_own and
    v_own being the bf16 values written to the cache (post-RoPE K); the
    attention inside the block uses the unrounded own K and V.
    """
    T = x.shape[0]
    Hq, Hkv, dh = cfg["Hq"], cfg["Hkv"], cfg["dh"]
    base = cfg["rope_base"]
    q, k, v = qkv(x, w, cfg)
    q = rope(q, pos, base)
    k = rope(k, pos, base)
    k = k.reshape(T, Hkv * dh)
    v = v.reshape(T, Hkv * dh)
    k_own = bf16.round_rne(k)          # what the cache stores
    v_own = bf16.round_rne(v)
    if kv_only:
        return None, k_own, v_own
    K = np.concatenate([k_prefix, k]).reshape(-1, Hkv, dh)
    V = np.concatenate([v_prefix, v]).reshape(-1, Hkv, dh)
    o = attention(q, K, V, 1.0 / np.sqrt(dh), allow=chunk_mask(T, k_prefix.shape[0], cfg)).reshape(T, Hq * dh)
    h = x + o @ w["wo"]
    hn = rmsnorm(h, cfg["eps"]) * w["g_ffn"]
    f = (gelu_tanh(hn @ w["wg"]) * (hn @ w["wu"])) @ w["wd"]
    return h + f, k_own, v_own


def state_token(state, W):
    return state @ W["w_state"] + W["b_state"]


def embed(x, t, W, D):
    """Action rows, unfolded: SiLU([x W_in + b_in ; temb(t)] W1 + b1) W2 + b2."""
    a = x @ W["w_in"] + W["b_in"]
    te = np.broadcast_to(timestep_embedding(t, D), a.shape)
    z = np.concatenate([a, te], axis=1) @ W["w1"] + W["b1"]
    return silu(z) @ W["w2"] + W["b2"]


def embed_folded(x, s, w_fold, table, W):
    """Action rows, folded: SiLU(x W' + T[s]) W2 + b2."""
    return silu(x @ w_fold + table[s]) @ W["w2"] + W["b2"]


def head(h, W, eps):
    """v = RMSNorm_gf(h) W_out + b_out."""
    return (rmsnorm(h, eps) * W["g_final"]) @ W["w_out"] + W["b_out"]


def times(cfg):
    S = cfg["S"]
    return [s / S for s in range(S)]


def denoise(noise, state, kv_bits, weight_bits, cfg, blocks=None, return_trace=False):
    """Full action-expert chunk: S Euler steps of the L-block stack.

    noise[Tq-1, A], state[A] (fp32 inputs), kv_bits[L, 2, Tp+Tq, Hkv*dh] bf16.
    Returns (actions[Tq-1, A] float64, kv_bits after the run (own slots written)).
    ``blocks`` may pass pre-built method weights (list of dicts) to save decoding.
    """
    D, L, S, Tp, Tq = cfg["D"], cfg["L"], cfg["S"], cfg["T_prefix"], cfg["T_q"]
    W = decode_tree({k: v for k, v in weight_bits.items() if k != "blocks"})
    if blocks is None:
        blocks = [method_block(decode_tree(b)) for b in weight_bits["blocks"]]
    kv = bf16.decode(kv_bits)
    pos = Tp + np.arange(Tq)
    dt = 1.0 / S
    x = np.asarray(noise, dtype=np.float64)
    st = state_token(np.asarray(state, dtype=np.float64), W)
    trace = []
    for s, t in enumerate(times(cfg)):
        h = np.vstack([st[None, :], embed(x, t, W, D)])
        for l in range(L):
            h, k_own, v_own = block(h, kv[l, 0, :Tp], kv[l, 1, :Tp], pos, blocks[l], cfg)
            kv[l, 0, Tp:] = k_own
            kv[l, 1, Tp:] = v_own
        v = head(h[1:], W, cfg["eps"])
        x = x + dt * v
        if return_trace:
            trace.append(x.copy())
    out = (x, bf16.encode(kv))
    return out + (trace,) if return_trace else out


def block_step(x, kv_bits_layer, weight_block_bits, cfg):
    """One block on a residual stream x[Tq, D] at the query positions.

    kv_bits_layer[2, Tp+Tq, Hkv*dh]; returns (x', k_own bits, v_own bits).
    """
    Tp, Tq = cfg["T_prefix"], cfg["T_q"]
    kv = bf16.decode(kv_bits_layer)
    w = method_block(decode_tree(weight_block_bits))
    x2, k_own, v_own = block(np.asarray(x, np.float64), kv[0, :Tp], kv[1, :Tp],
                             Tp + np.arange(Tq), w, cfg)
    return x2, bf16.encode(k_own), bf16.encode(v_own)


def prefill(patch_emb_bits, weight_bits, cfg, skip_last=True, blocks=None):
    """Prefix KV cache from patch embeddings.

    patch_emb_bits[B, Tp, P] bf16.  Patch projection h = e W_patch + b_patch,
    then L bidirectional blocks over the Tp prefix tokens at positions 0..Tp-1.
    Returns kv bits [L, B, 2, Tp+Tq, Hkv*dh] with slots >= Tp left zero.  With
    skip_last, the last block stops after its K and V (section 4.3 of the note).
    """
    L, Tp, Tq, Hkv, dh = cfg["L"], cfg["T_prefix"], cfg["T_q"], cfg["Hkv"], cfg["dh"]
    B = patch_emb_bits.shape[0]
    wp = bf16.decode(weight_bits["w_patch"])
    bp = bf16.decode(weight_bits["b_patch"])
    if blocks is None:
        blocks = [method_block(decode_tree(b)) for b in weight_bits["blocks"]]
    kv = np.zeros((L, B, 2, Tp + Tq, Hkv * dh))
    pos = np.arange(Tp)
    empty = np.zeros((0, Hkv * dh))
    for b in range(B):
        h = bf16.decode(patch_emb_bits[b]) @ wp + bp
        for l in range(L):
            last = l == L - 1
            h, k_own, v_own = block(h, empty, empty, pos, blocks[l], cfg,
                                    kv_only=(last and skip_last))
            kv[l, b, 0, :Tp] = k_own
            kv[l, b, 1, :Tp] = v_own
    return bf16.encode(kv)


def fold_tables(weight_bits, cfg):
    """Folded embedding quantities of the method: (W' [A, D], T [S, D])."""
    W = decode_tree({k: v for k, v in weight_bits.items() if k != "blocks"})
    return time_fold(W["w_in"], W["b_in"], W["w1"], W["b1"], times(cfg), cfg["D"])
