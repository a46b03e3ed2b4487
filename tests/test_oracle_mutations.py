"""Plant plausible mistakes in the oracle (on the CPU) and check a pin fails.

Each mutation replaces one oracle function by a subtly wrong version (a wrong
sign, a swapped pairing, a dropped term, an off-by-one) and runs the pin tests
that should catch it.  A mutation no pin catches would mean the oracle is not
pinned at that point.
"""
import numpy as np
import pytest

import oracle.bf16 as bf16
import oracle.ops as ops
import oracle.dit as dit
import oracle.pi0 as pi0
import oracle.fold as fold
import tests.test_oracle_pins as pins


def _rope_wrong_sign(x, pos, base):
    T, H, dh = x.shape
    half = dh // 2
    ang = ops.rope_angles(pos, dh, base)
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c + b * s, b * c - a * s], axis=-1)


def _rope_interleaved(x, pos, base):
    T, H, dh = x.shape
    ang = ops.rope_angles(pos, dh, base)
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = b * c + a * s
    return out


def _attention_no_scale(q, k, v, scale):
    return _orig_attention(q, k, v, 1.0)


def _rmsnorm_var(x, eps):
    return x / np.sqrt(np.var(x, axis=-1, keepdims=True) + eps)


def _gelu_wrong_const(x):
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.0447 * x ** 3)))


def _temb_swapped(t, d):
    half = d // 2
    w = 10000.0 ** (-np.arange(half, dtype=np.float64) / half)
    a = 1000.0 * float(t) * w
    return np.concatenate([np.cos(a), np.sin(a)])


def _history_off_by_one(c, n_hist):
    return [c - k for k in range(n_hist + 1, 0, -1) if c - k >= 0]


def _fold_no_round(g, w):
    return g[:, None] * w * (1 + 2.0 ** -7)


def _times_wrong(cfg):
    S = cfg["S"]
    return [(s + 1) / S for s in range(S)]


def _descs_step_off_by_one(i, n_chunks, S, stream=0):
    chunks = [c for c in range(max(0, i - S + 1), min(i, n_chunks - 1) + 1)]
    return sorted(((stream, c, min(S - 1, i - c + 1)) for c in chunks), key=lambda d: d[1] % S)


def _mask_wrong_row(T, Tp, cfg):
    if not cfg.get("prefix_lm"):
        return None
    allow = np.ones((T, Tp + T), dtype=bool)
    allow[T - 1, Tp + 1:] = False
    return allow


def _layernorm_no_center(x, eps):
    return x / np.sqrt(np.var(x, axis=-1, keepdims=True) + eps)


def _silu_sigmoid_approx(x):
    return x / (1.0 + np.exp(-1.702 * x))


def _round_half_away(x):
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    r = np.sign(m) * np.floor(np.abs(np.ldexp(m, 8)) + 0.5)
    return np.ldexp(r, e - 8)


def _ring_slot_mod_nhist(c, n_hist):
    return c % n_hist


def _positions_shifted(c, T):
    return c * T + np.arange(T) + 1


def _softmax_over_queries(z, axis=-1):
    z = z - np.max(z, axis=-2, keepdims=True)
    e = np.exp(z)
    return e / np.sum(e, axis=-2, keepdims=True)


def _rope_angles_half_rate(pos, dh, base):
    i = np.arange(dh // 2, dtype=np.float64)
    return np.asarray(pos, dtype=np.float64)[:, None] * (base ** (-i / dh))[None, :]


def _embed_no_silu(x, t, W, D):
    a = x @ W["w_in"] + W["b_in"]
    te = np.broadcast_to(ops.timestep_embedding(t, D), a.shape)
    z = np.concatenate([a, te], axis=1) @ W["w1"] + W["b1"]
    return z @ W["w2"] + W["b2"]


def _split6_swap_first(a, D):
    sh1, sc1, g1, sh2, sc2, g2 = [a[i * D:(i + 1) * D] for i in range(6)]
    return [sc1, sh1, g1, sh2, sc2, g2]


def _split6_swap_second(a, D):
    sh1, sc1, g1, sh2, sc2, g2 = [a[i * D:(i + 1) * D] for i in range(6)]
    return [sh1, sc1, g1, sc2, sh2, g2]


def _head_no_gfinal(h, W, eps):
    return ops.rmsnorm(h, eps) @ W["w_out"] + W["b_out"]


def _head_no_norm(h, W, eps):
    return (h * W["g_final"]) @ W["w_out"] + W["b_out"]


def _adaln_no_inner_silu(W, cfg):
    S, td = cfg["S"], cfg["t_dim"]
    rows = []
    for s in range(S):
        e = (ops.timestep_embedding(s / S, td) @ W["wt1"] + W["bt1"]) @ W["wt2"] + W["bt2"]
        rows.append(ops.silu(e) @ W["wmod"] + W["bmod"])
    return np.stack(rows)


def _adaln_grid_shifted(W, cfg):
    S, td = cfg["S"], cfg["t_dim"]
    rows = []
    for s in range(S):
        e = ops.silu(ops.timestep_embedding((s + 1) / S, td) @ W["wt1"] + W["bt1"]) @ W["wt2"] + W["bt2"]
        rows.append(ops.silu(e) @ W["wmod"] + W["bmod"])
    return np.stack(rows)


def _state_token_no_bias(state, W):
    return state @ W["w_state"]


def _prefill_no_patch_bias(patch_emb_bits, weight_bits, cfg, skip_last=True, blocks=None):
    wb = dict(weight_bits)
    wb["b_patch"] = np.zeros_like(wb["b_patch"])
    return _orig_prefill(patch_emb_bits, wb, cfg, skip_last=skip_last, blocks=blocks)


def _bands_equal_thirds(dh):
    w = 2 * (dh // 6)
    return [(0, w), (w, w), (2 * w, dh - 2 * w)]


def _positions3_yx_swapped(c, cfg):
    T, gh, gw = cfg["T_chunk"], cfg["grid_h"], cfg["grid_w"]
    j = np.arange(T)
    return np.stack([c * (T // (gh * gw)) + j // (gh * gw), j % gw, (j // gw) % gh], axis=1)


def _rope3d_one_band(x, pos3, base):
    return ops.rope(x, pos3[:, 0], base)


def _cross_no_affine(h, w, ctx, cfg):
    return _orig_cross(h, dict(w, g_c=np.ones_like(w["g_c"]), b_c=np.zeros_like(w["b_c"])), ctx, cfg)


def _cross_k_from_h(h, w, ctx, cfg):
    H, dh, eps = cfg["H"], cfg["dh"], cfg["eps"]
    u = ops.layernorm(h, eps) * w["g_c"] + w["b_c"]
    q = (u @ w["cq"]).reshape(len(h), H, dh)
    k = (u @ w["ck"]).reshape(len(h), H, dh)
    v = (ctx @ w["cv"]).reshape(len(ctx), H, dh)[:len(h)] if len(ctx) >= len(h) else (u @ w["cv"]).reshape(len(h), H, dh)
    o = ops.attention(q, k, v, 1.0 / np.sqrt(dh)).reshape(len(h), H * dh)
    return h + o @ w["co"]


def _pool_row_off_by_one(ring, table, cfg, n_pool):
    st, L, S, R, _, T, D = ring.shape
    P = cfg["page_tokens"]
    pool = np.zeros((n_pool, 2, P, D), dtype=ring.dtype)
    for a in range(st):
        for l in range(L):
            for s in range(S):
                flat = ring[a, l, s].transpose(1, 0, 2, 3).reshape(2, R * T, D)
                for r in range(R * T):
                    pool[table[a, l, s, r // P], :, (r + 1) % P] = flat[:, r]
    return pool


_orig_attention = ops.attention
_orig_cross = dit._cross
_orig_prefill = pi0.prefill

MUTATIONS = [
    # (module, attribute, replacement, pins that must catch it)
    ((ops, pi0, dit), "rope", _rope_wrong_sign, ["test_rope_hand_case", "test_rope_is_complex_rotation"]),
    ((ops, pi0, dit), "rope", _rope_interleaved, ["test_rope_hand_case", "test_rope_is_complex_rotation"]),
    ((ops, pi0, dit), "attention", _attention_no_scale, ["test_attention_brute_force"]),
    ((ops, pi0), "rmsnorm", _rmsnorm_var, ["test_rmsnorm_closed_forms"]),
    ((ops, pi0, dit), "gelu_tanh", _gelu_wrong_const, ["test_gelu_tanh_against_erf_gelu"]),
    ((ops, pi0, dit, fold), "timestep_embedding", _temb_swapped, ["test_timestep_embedding_closed_forms"]),
    ((dit,), "history_chunks", _history_off_by_one, ["test_ring_slot_matches_fifo_simulation"]),
    ((fold, pi0), "fold_scale", _fold_no_round, ["test_rmsnorm_scale_fold_identity"]),
    ((pi0,), "times", _times_wrong, ["test_time_grid"]),
    ((pi0,), "chunk_mask", _mask_wrong_row, ["test_pi0_prefix_lm_mask"]),
    ((dit,), "interval_descs", _descs_step_off_by_one,
     ["test_dit_interleaved_schedule", "test_dit_pipeline_equals_sequential"]),
    ((ops, dit), "layernorm", _layernorm_no_center, ["test_layernorm_closed_forms"]),
    ((ops, pi0, dit), "silu", _silu_sigmoid_approx, ["test_silu_library"]),
    ((bf16,), "round_rne", _round_half_away, ["test_bf16_ties_to_even_and_decode"]),
    ((dit,), "ring_slot", _ring_slot_mod_nhist, ["test_ring_slot_matches_fifo_simulation"]),
    ((dit,), "positions", _positions_shifted, ["test_ring_slot_matches_fifo_simulation"]),
    ((ops,), "softmax", _softmax_over_queries, ["test_attention_brute_force"]),
    ((ops,), "rope_angles", _rope_angles_half_rate, ["test_rope_hand_case", "test_rope_is_complex_rotation"]),
    ((pi0,), "embed", _embed_no_silu, ["test_time_embedding_fold"]),
    ((dit,), "_split6", _split6_swap_first, ["test_dit_zero_gates_is_identity_and_history_set"]),
    ((dit,), "_split6", _split6_swap_second, ["test_dit_ffn_branch_closed_form"]),
    ((pi0,), "head", _head_no_gfinal, ["test_head_closed_form", "test_denoise_wiring_with_identity_blocks"]),
    ((pi0,), "head", _head_no_norm, ["test_head_closed_form", "test_denoise_wiring_with_identity_blocks"]),
    ((dit,), "adaln_table", _adaln_no_inner_silu, ["test_adaln_table_closed_form"]),
    ((dit,), "adaln_table", _adaln_grid_shifted, ["test_adaln_table_closed_form"]),
    ((pi0,), "state_token", _state_token_no_bias, ["test_state_token_closed_form"]),
    ((pi0,), "prefill", _prefill_no_patch_bias, ["test_prefill_patch_projection"]),
    ((ops,), "rope_bands", _bands_equal_thirds, ["test_rope_bands_split"]),
    ((dit,), "positions3", _positions3_yx_swapped, ["test_positions3_hand_cases"]),
    ((ops, dit), "rope3d", _rope3d_one_band,
     ["test_rope3d_reduces_to_rope_per_band", "test_dit_wan_block_rows_and_batch"]),
    ((dit,), "_cross", _cross_no_affine, ["test_dit_cross_attention_closed_forms"]),
    ((dit,), "_cross", _cross_k_from_h, ["test_dit_cross_attention_closed_forms"]),
    ((dit,), "ring_to_pool", _pool_row_off_by_one, ["test_page_pool_round_trip_and_hand_case"]),
]


def _run_pin(name):
    fn = getattr(pins, name)
    if name == "test_attention_brute_force":
        fn(4, 1)
    else:
        fn()


@pytest.mark.parametrize("mods,attr,repl,catchers", MUTATIONS,
                         ids=[f"{m[1]}:{m[2].__name__}" for m in MUTATIONS])
def test_mutation_is_caught(monkeypatch, mods, attr, repl, catchers):
    for m in mods:
        if hasattr(m, attr):
            monkeypatch.setattr(m, attr, repl)
    caught = False
    for name in catchers:
        try:
            _run_pin(name)
        except AssertionError:
            caught = True
    assert caught, f"mutation {repl.__name__} of {attr} not caught by {catchers}"
