"""Seeded synthetic inputs for the low-latency transformer-block path.

This module only *draws data*: model shapes, weights, caches, noise and chunk
descriptors.  It holds none of the method's arithmetic (no norm, projection,
attention, fold or integration step), so both the CUDA path and the CPU oracle
may read it without sharing any computation.

Every tensor is drawn from its own counter-based Philox stream, keyed by
``(seed, tensor name, block index)``, in fixed blocks of ``_CHUNK`` elements, so
the values do not depend on the number of threads used to draw them.
Floating-point tensors that the model stores in bf16 are returned as raw bf16
bit patterns (``uint16``); fp32 tensors (residual stream, actions, noise) are
returned as ``float32``.

Weight matrices use the math convention ``y = x @ W``: shape ``[K_in, N_out]``,
row-major.

The shapes are the workloads of the pages (pi0 action expert over a 512-token
vision prefix, its prefix prefill, and chunked autoregressive DiT stages of a
1.3B-class and a 14B-class video model); sizes the pages leave open are fixed
here and listed in the design notes.
"""
from __future__ import annotations

import hashlib
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_CHUNK = 1 << 20

# ----------------------------------------------------------------------------
# Model shapes.  kind = "pi0" (RMSNorm + GeGLU, MQA, denoise loop with time
# embedding), "prefill" (the prefix model producing the pi0 KV cache) or "dit"
# (LayerNorm + adaLN, MHA, chunked AR diffusion stage).
# ----------------------------------------------------------------------------
CONFIGS = {
    # 1 block, width 256, 4 q heads x 64, 1 kv head, GeGLU 1024, 64 query tokens
    # over a 128-token prefix, 2 Euler steps on 32-dim actions.
    "tiny": dict(kind="pi0", D=256, Hq=4, Hkv=1, dh=64, F=1024, L=1, S=2,
                 T_prefix=128, T_q=64, act_dim=32, rope_base=10000.0, eps=1e-6),
    # pi0 action expert: 18 blocks, width 1024, 8 q heads x 256, 1 kv head x 256,
    # GeGLU 4096, 63 actions + 1 state over a 512-token vision prefix, 10 steps.
    "pi0_ae": dict(kind="pi0", D=1024, Hq=8, Hkv=1, dh=256, F=4096, L=18, S=10,
                   T_prefix=512, T_q=64, act_dim=32, rope_base=10000.0, eps=1e-6),
    # prefix prefill that produces the pi0 KV cache: 18 blocks, width 2048,
    # GeGLU 16384, 512 tokens from 1152-dim patch embeddings.
    "prefill": dict(kind="prefill", D=2048, Hq=8, Hkv=1, dh=256, F=16384, L=18,
                    T_prefix=512, T_q=64, patch_dim=1152, rope_base=10000.0,
                    eps=1e-6, batches=(1, 8)),
    # chunked AR-diffusion DiT stage, 1.3B class: 30 blocks, width 1536,
    # 12 heads x 128, GELU-tanh FFN 8960, chunk 1560 over 4 history chunks,
    # 4 denoise steps, 4 chunks (one per step) batched per block.
    # Latent tokens of 64 channels enter / leave the stage through linear
    # projections (lat_dim; the interleaved-schedule interval).
    "dit_1p3b": dict(kind="dit", D=1536, H=12, dh=128, F=8960, L=30, S=4,
                     T_chunk=1560, n_hist=4, t_dim=256, rope_base=10000.0,
                     eps=1e-6, batches=(4,), lat_dim=64,
                     grid_h=0, grid_w=0, text_len=0, page_tokens=0),
    # one 14B-class DiT block: width 5120, 40 heads x 128, FFN 13824.
    "dit_14b": dict(kind="dit", D=5120, H=40, dh=128, F=13824, L=1, S=4,
                    T_chunk=1560, n_hist=4, t_dim=256, rope_base=10000.0,
                    eps=1e-6, batches=(1, 4, 8), lat_dim=64,
                    grid_h=0, grid_w=0, text_len=0, page_tokens=0),
}

WEIGHT_STD = 0.02
SCALE_STD = 0.02  # norm scales g = 1 + N(0, SCALE_STD)


def config(name: str, **overrides) -> dict:
    cfg = dict(CONFIGS[name])
    cfg["name"] = name
    cfg.update(overrides)
    return cfg


# ----------------------------------------------------------------------------
# Raw draws
# ----------------------------------------------------------------------------
def _key(seed: int, name: str, block: int) -> int:
    h = hashlib.blake2b(f"{seed}/{name}/{block}".encode(), digest_size=16)
    return int.from_bytes(h.digest(), "little")


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def _draw(seed: int, name: str, n: int, out: np.ndarray, post) -> np.ndarray:
    """Fill ``out`` (n elements) block by block: N(0,1) float32 -> ``post``."""
    nblk = (n + _CHUNK - 1) // _CHUNK

    def fill(b):
        lo, hi = b * _CHUNK, min(n, (b + 1) * _CHUNK)
        g = np.random.Generator(np.random.Philox(key=_key(seed, name, b)))
        out[lo:hi] = post(g.standard_normal(hi - lo, dtype=np.float32))

    if nblk <= 1:
        for b in range(nblk):
            fill(b)
    else:
        list(_pool().map(fill, range(nblk)))
    return out


def standard_normal(seed: int, name: str, n: int) -> np.ndarray:
    """``n`` N(0,1) float32 draws for tensor ``name``."""
    return _draw(seed, name, n, np.empty(n, dtype=np.float32), lambda z: z)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, round to nearest even (data encoding)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def normal_bf16(seed, name, shape, std=1.0, mean=0.0) -> np.ndarray:
    n = int(np.prod(shape))
    sd, mu = np.float32(std), np.float32(mean)

    def post(z):
        if std != 1.0:
            z *= sd
        if mean != 0.0:
            z += mu
        return bf16_bits(z)

    return _draw(seed, name, n, np.empty(n, dtype=np.uint16), post).reshape(shape)


def normal_f32(seed, name, shape, std=1.0) -> np.ndarray:
    z = standard_normal(seed, name, int(np.prod(shape))).reshape(shape)
    if std != 1.0:
        z *= np.float32(std)
    return z


def zeros_bf16(shape) -> np.ndarray:
    return np.zeros(shape, dtype=np.uint16)


# ----------------------------------------------------------------------------
# pi0-style block stack (action expert and prefix prefill share the block)
# ----------------------------------------------------------------------------
def block_weights_rms(cfg: dict, seed: int, layer: int, prefix: str = "blk") -> dict:
    D, Hq, Hkv, dh, F = cfg["D"], cfg["Hq"], cfg["Hkv"], cfg["dh"], cfg["F"]
    p = f"{prefix}{layer}."
    w = WEIGHT_STD
    return {
        "g_attn": normal_bf16(seed, p + "g_attn", (D,), SCALE_STD, 1.0),
        "wq": normal_bf16(seed, p + "wq", (D, Hq * dh), w),
        "wk": normal_bf16(seed, p + "wk", (D, Hkv * dh), w),
        "wv": normal_bf16(seed, p + "wv", (D, Hkv * dh), w),
        "wo": normal_bf16(seed, p + "wo", (Hq * dh, D), w),
        "g_ffn": normal_bf16(seed, p + "g_ffn", (D,), SCALE_STD, 1.0),
        "wg": normal_bf16(seed, p + "wg", (D, F), w),
        "wu": normal_bf16(seed, p + "wu", (D, F), w),
        "wd": normal_bf16(seed, p + "wd", (F, D), w),
    }


def pi0_weights(cfg: dict, seed: int = 0) -> dict:
    """Action-expert weights: L blocks plus the action/time embedding and head."""
    D, A = cfg["D"], cfg["act_dim"]
    w = WEIGHT_STD
    return {
        "blocks": [block_weights_rms(cfg, seed, l) for l in range(cfg["L"])],
        "w_in": normal_bf16(seed, "w_in", (A, D), w),       # action -> D
        "b_in": normal_bf16(seed, "b_in", (D,), w),
        "w1": normal_bf16(seed, "w1", (2 * D, D), w),       # [action emb ; time emb] -> D
        "b1": normal_bf16(seed, "b1", (D,), w),
        "w2": normal_bf16(seed, "w2", (D, D), w),
        "b2": normal_bf16(seed, "b2", (D,), w),
        "w_state": normal_bf16(seed, "w_state", (A, D), w),
        "b_state": normal_bf16(seed, "b_state", (D,), w),
        "g_final": normal_bf16(seed, "g_final", (D,), SCALE_STD, 1.0),
        "w_out": normal_bf16(seed, "w_out", (D, A), w),
        "b_out": normal_bf16(seed, "b_out", (A,), w),
    }


def pi0_inputs(cfg: dict, seed: int = 0) -> dict:
    """Prefix KV (N(0,1) bf16; own-token slots zero), noise and state (N(0,1) fp32).

    KV layout: [L][2][T_prefix + T_q][Hkv * dh] (plane 0 = K, plane 1 = V).
    """
    L, Tp, Tq, Hkv, dh, A = (cfg["L"], cfg["T_prefix"], cfg["T_q"], cfg["Hkv"],
                             cfg["dh"], cfg["act_dim"])
    kv = np.zeros((L, 2, Tp + Tq, Hkv * dh), dtype=np.uint16)
    kv[:, :, :Tp, :] = normal_bf16(seed, "kv_prefix", (L, 2, Tp, Hkv * dh))
    return {
        "kv": kv,
        "noise": normal_f32(seed, "noise", (Tq - 1, A)),
        "state": normal_f32(seed, "state", (A,)),
    }


def residual_stream(cfg: dict, seed: int = 0, std: float = 0.5, tag: str = "xres") -> np.ndarray:
    """A residual-stream input for one block, N(0, std^2) fp32 [T_q][D]."""
    return normal_f32(seed, tag, (cfg["T_q"], cfg["D"]), std)


def attention_inputs(T_q, T_kv, Hq, Hkv, dh, seed=0, q_std=0.6):
    """q fp32 [T_q][Hq*dh] ~ N(0, q_std^2); k, v bf16 [T_kv][Hkv*dh] ~ N(0,1)."""
    return {
        "q": normal_f32(seed, "attn_q", (T_q, Hq * dh), q_std),
        "k": normal_bf16(seed, "attn_k", (T_kv, Hkv * dh)),
        "v": normal_bf16(seed, "attn_v", (T_kv, Hkv * dh)),
    }


def prefill_weights(cfg: dict, seed: int = 0) -> dict:
    D, P = cfg["D"], cfg["patch_dim"]
    w = WEIGHT_STD
    return {
        "blocks": [block_weights_rms(cfg, seed, l, prefix="vlm") for l in range(cfg["L"])],
        "w_patch": normal_bf16(seed, "w_patch", (P, D), w),
        "b_patch": normal_bf16(seed, "b_patch", (D,), w),
    }


def prefill_inputs(cfg: dict, B: int, seed: int = 0) -> dict:
    return {"patch_emb": normal_bf16(seed, f"patch_emb", (B, cfg["T_prefix"], cfg["patch_dim"]))}


# ----------------------------------------------------------------------------
# DiT stage (LayerNorm + adaLN, GELU-tanh FFN, MHA over a ring of noisy KV)
# ----------------------------------------------------------------------------
def dit_weights(cfg: dict, seed: int = 0, layers=None) -> dict:
    D, F, td = cfg["D"], cfg["F"], cfg["t_dim"]
    w = WEIGHT_STD
    layers = range(cfg["L"]) if layers is None else layers
    blocks = []
    for l in layers:
        p = f"dit{l}."
        blocks.append({
            "wq": normal_bf16(seed, p + "wq", (D, D), w),
            "wk": normal_bf16(seed, p + "wk", (D, D), w),
            "wv": normal_bf16(seed, p + "wv", (D, D), w),
            "wo": normal_bf16(seed, p + "wo", (D, D), w),
            "w1": normal_bf16(seed, p + "w1", (D, F), w),
            "w2": normal_bf16(seed, p + "w2", (F, D), w),
        })
        if cfg.get("text_len", 0):   # text cross-attention: LayerNorm affine, q / k / v / o
            blocks[-1].update({
                "g_c": normal_bf16(seed, p + "g_c", (D,), SCALE_STD, 1.0),
                "b_c": normal_bf16(seed, p + "b_c", (D,), w),
                "cq": normal_bf16(seed, p + "cq", (D, D), w),
                "ck": normal_bf16(seed, p + "ck", (D, D), w),
                "cv": normal_bf16(seed, p + "cv", (D, D), w),
                "co": normal_bf16(seed, p + "co", (D, D), w),
            })
    return {
        "blocks": blocks,
        # timestep MLP: sinusoid(t_dim) -> D -> SiLU -> D, then SiLU -> 6D
        "wt1": normal_bf16(seed, "wt1", (td, D), w),
        "bt1": normal_bf16(seed, "bt1", (D,), w),
        "wt2": normal_bf16(seed, "wt2", (D, D), w),
        "bt2": normal_bf16(seed, "bt2", (D,), w),
        "wmod": normal_bf16(seed, "wmod", (D, 6 * D), w),
        "bmod": normal_bf16(seed, "bmod", (6 * D,), w),
        # latent in / out projections of the stage (lat_dim channels)
        "w_in": normal_bf16(seed, "dit.w_in", (cfg["lat_dim"], D), w),
        "b_in": normal_bf16(seed, "dit.b_in", (D,), w),
        "w_out": normal_bf16(seed, "dit.w_out", (D, cfg["lat_dim"]), w),
        "b_out": normal_bf16(seed, "dit.b_out", (cfg["lat_dim"],), w),
    }


def dit_ring(cfg: dict, seed: int = 0, streams: int = 1, layers: int = 1,
             tag: str = "ring") -> np.ndarray:
    """Noisy history KV rings, N(0,1) bf16.

    Layout [streams][layers][S][n_hist+1][2][T_chunk][D]: one ring of
    ``n_hist + 1`` chunk slots per (stream, block, denoise step); plane 0 = K,
    plane 1 = V.
    """
    shape = (streams, layers, cfg["S"], cfg["n_hist"] + 1, 2, cfg["T_chunk"], cfg["D"])
    return normal_bf16(seed, tag, shape)


def dit_text(cfg: dict, streams: int = 1, seed: int = 0, tag: str = "text") -> np.ndarray:
    """Text contexts of the streams (already in the model width), N(0,1) bf16:
    [streams][text_len][D]."""
    return normal_bf16(seed, tag, (streams, cfg["text_len"], cfg["D"]))


def dit_page_table(cfg: dict, streams: int = 1, layers: int = 1, seed: int = 0,
                   spare: int = 3) -> tuple:
    """A page table for rings kept in pages of cfg["page_tokens"] tokens: every
    (stream, block, step) ring of (n_hist + 1) * T_chunk tokens gets
    ceil(.../page_tokens) pages, drawn as a seeded permutation of a pool with
    ``spare`` pages more than needed.  Returns (table int32 [streams][layers][S]
    [pages], pool size)."""
    S = cfg["S"]
    per = -(-(cfg["n_hist"] + 1) * cfg["T_chunk"] // cfg["page_tokens"])
    n = streams * layers * S * per
    perm = np.random.Generator(np.random.Philox(key=_key(seed, "page_table", 0))).permutation(n + spare)
    return perm[:n].astype(np.int32).reshape(streams, layers, S, per), n + spare


def dit_latents(cfg: dict, n: int, seed: int = 0, tag: str = "x") -> np.ndarray:
    """Residual-stream latents of n chunks, N(0,1) fp32: [n][T_chunk][D]."""
    return normal_f32(seed, tag, (n, cfg["T_chunk"], cfg["D"]))


def dit_noise(cfg: dict, n: int, seed: int = 0, tag: str = "noise") -> np.ndarray:
    """Starting latents of n chunks, N(0,1) fp32: [n][T_chunk][lat_dim]."""
    return normal_f32(seed, tag, (n, cfg["T_chunk"], cfg["lat_dim"]))


def dit_chunk_descs(cfg: dict, n: int, first_chunk: int = 7) -> list:
    """Steady-state batch of (stream, chunk, step) triples.

    Within a stream, chunk c is at step 0, c-1 at step 1, ... (one chunk per
    denoise step, as in a pipelined stream); n > S fills further streams.
    """
    S = cfg["S"]
    return [(b // S, first_chunk - (b % S), b % S) for b in range(n)]


def to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit pattern -> float32 (exact widening; data decoding only)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
