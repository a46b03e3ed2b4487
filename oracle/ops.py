"""Elementary operations of the transformer block, float64, from their definitions.

Readings where the pages are silent (each listed in the design notes):
* RMSNorm / LayerNorm epsilon 1e-6; LayerNorm has no affine part (the adaLN
  modulation supplies it).
* RoPE is the rotate-half form: dimension i pairs with i + dh/2,
  theta_i = base**(-2i/dh), angle = position * theta_i.  3-D RoPE (video
  tokens at (frame, y, x)): three bands of the head, each such a RoPE of its own
  width at its own coordinate.
* Attention scale 1/sqrt(dh); no mask (every query sees every key given).
* GELU is the tanh form of Hendrycks & Gimpel.
* Timestep embedding: [sin(1000 t w_i), cos(1000 t w_i)], w_i = 10000**(-i/(d/2)).
"""
import numpy as np


def rmsnorm(x: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x**2) + eps) over the last axis (no learnable scale)."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps)


def layernorm(x: np.ndarray, eps: float) -> np.ndarray:
    """(x - mean) / sqrt(var + eps) over the last axis, biased variance, no affine."""
    mu = np.mean(x, axis=-1, keepdims=True)
    d = x - mu
    var = np.mean(d * d, axis=-1, keepdims=True)
    return d / np.sqrt(var + eps)


def rope_angles(pos: np.ndarray, dh: int, base: float) -> np.ndarray:
    """angle[t, i] = pos[t] * base**(-2i/dh), i < dh/2."""
    i = np.arange(dh // 2, dtype=np.float64)
    theta = base ** (-2.0 * i / dh)
    return np.asarray(pos, dtype=np.float64)[:, None] * theta[None, :]


def rope(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """Rotate-half RoPE of x[T, H, dh] at positions pos[T].

    For i < dh/2 the pair (x_i, x_{i+dh/2}) is rotated by the angle pos*theta_i:
    (a, b) -> (a cos - b sin, b cos + a sin).
    """
    T, H, dh = x.shape
    half = dh // 2
    ang = rope_angles(pos, dh, base)            # [T, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def rope_bands(dh: int) -> list:
    """3-D RoPE bands of a head (frame, height, width): (offset, width) each.
    Frame d_f = dh - 4 floor(dh/6), height and width 2 floor(dh/6) each."""
    dhw = 2 * (dh // 6)
    df = dh - 2 * dhw
    return [(0, df), (df, dhw), (df + dhw, dhw)]


def rope3d(x: np.ndarray, pos3: np.ndarray, base: float) -> np.ndarray:
    """3-D RoPE of x[T, H, dh] at positions pos3[T, 3] = (frame, y, x): band b
    (rope_bands) is a rotate-half RoPE of its own width at coordinate pos3[:, b]."""
    out = np.array(x, dtype=np.float64, copy=True)
    for b, (o, d) in enumerate(rope_bands(x.shape[2])):
        out[..., o:o + d] = rope(x[..., o:o + d], pos3[:, b], base)
    return out


def softmax(z: np.ndarray, axis: int = -1) -> np.ndarray:
    z = z - np.max(z, axis=axis, keepdims=True)
    e = np.exp(z)
    return e / np.sum(e, axis=axis, keepdims=True)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, allow=None) -> np.ndarray:
    """softmax(q k^T * scale) v per head; with `allow` (bool [Tq, Tk]) the
    scores of disallowed (query, key) pairs are -inf before the softmax.

    q[Tq, Hq, dh], k/v[Tk, Hkv, dh]; query head h reads kv head h // (Hq/Hkv)
    (Hkv = 1 is multi-query attention, Hkv = Hq multi-head).
    """
    Tq, Hq, dh = q.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    out = np.empty((Tq, Hq, v.shape[2]), dtype=np.float64)
    for h in range(Hq):
        j = h // group
        z = (q[:, h, :] @ k[:, j, :].T) * scale
        if allow is not None:
            z = np.where(allow, z, -np.inf)
        p = softmax(z, axis=-1)
        out[:, h, :] = p @ v[:, j, :]
    return out


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x)."""
    return x / (1.0 + np.exp(-x))


def timestep_embedding(t: float, d: int) -> np.ndarray:
    """[sin(1000 t w_i) for i < d/2] ++ [cos(1000 t w_i) for i < d/2], w_i = 1e4**(-i/(d/2))."""
    half = d // 2
    w = 10000.0 ** (-np.arange(half, dtype=np.float64) / half)
    a = 1000.0 * float(t) * w
    return np.concatenate([np.sin(a), np.cos(a)])
