"""Offline graph transforms of the method, float64 ("Running VLAs at Real-time
Speed", reading note on arXiv 2510.26742, section 4 / paper section 3.2, Fig. 3).

* RMSNorm scale fold (section 4.1): (x_hat * g) W = x_hat [diag(g) W].  Only the
  fixed per-dimension scale g folds; the normalisation stays input-dependent.
  The folded block weights are streamed from HBM in bf16, so the method stores
  diag(g) W rounded to bf16; ``fold_scale`` does exactly that.  (g W of two bf16
  numbers has at most 16 significant bits, so the only rounding is the final
  bf16 store.)
* Action/time-embedding fold (section 4.2): the action projection feeds a
  linear layer through a concatenation with the time encoding and no
  nonlinearity in between, so the two weights pre-multiply, and the time branch
  for the fixed denoise times becomes a per-step bias table added before SiLU.
  These folded quantities are small and stored in fp32; here they are exact.
* Merged QKV (section 4.3): one projection with [Wq | Wk | Wv] split by columns.
"""
import numpy as np

from . import bf16
from .ops import timestep_embedding


def fold_scale(g: np.ndarray, w: np.ndarray) -> np.ndarray:
    """diag(g) W rounded to the bf16 storage of the streamed weights."""
    return bf16.round_rne(g[:, None] * w)


def fold_scale_exact(g: np.ndarray, w: np.ndarray) -> np.ndarray:
    """diag(g) W without the storage rounding (for the identity check)."""
    return g[:, None] * w


def merge_columns(*ws: np.ndarray) -> np.ndarray:
    """[W_1 | W_2 | ...] along the output dimension."""
    return np.concatenate(ws, axis=1)


def time_fold(w_in, b_in, w1, b1, times, d_emb):
    """Folded action/time embedding.

    Unfolded: z = [x W_in + b_in ; temb(t)] W1 + b1, with W1 = [W1_a ; W1_t]
    stacked by rows (first D rows act on the action embedding).
    Folded:   z = x W' + T[s],  W' = W_in W1_a,
              T[s] = temb(t_s) W1_t + b_in W1_a + b1.
    Returns (W' [A, D], T [S, D]).
    """
    D = w_in.shape[1]
    w1a, w1t = w1[:D], w1[D:]
    w_fold = w_in @ w1a
    table = np.stack([timestep_embedding(t, d_emb) @ w1t + b_in @ w1a + b1 for t in times])
    return w_fold, table
