"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against something it does not compute itself: a
library routine, a closed form, an invariant of the mathematics, brute force on
tiny inputs, or a special case whose answer is known.  Together they are meant
to catch a dropped term, a wrong sign or index, or a transposed operand
anywhere in ``oracle/``.
"""
import math

import numpy as np
import pytest
import torch

from latency_transformer_block_gb300 import synth
from oracle import bf16, dit, fold, ops, pi0

RNG = np.random.default_rng(1234)


# ----------------------------------------------------------------------------
# bf16 storage
# ----------------------------------------------------------------------------
def test_bf16_round_matches_torch_conversion():
    x = (RNG.standard_normal(200_000) * np.exp(RNG.uniform(-20, 20, 200_000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(bf16.round_rne(x.astype(np.float64)), ref)
    ref_bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16.encode(x.astype(np.float64)), ref_bits)


def test_bf16_round_paths_agree():
    # values that are exact float32 take the bit path, others the frexp path;
    # adding 2^-40 relative moves a value off float32 without crossing a bf16
    # rounding boundary (except exact ties, which the offset breaks upward)
    x = (RNG.standard_normal(100_000) * np.exp(RNG.uniform(-10, 10, 100_000))).astype(np.float32)
    x = x.astype(np.float64)
    a = bf16.round_rne(x)
    b = bf16.round_rne(x * (1 + 2.0 ** -40))
    tie = np.abs(x - a) == 0.5 * bf16.ulp(a)
    assert np.array_equal(a[~tie], b[~tie])


def test_bf16_ties_to_even_and_decode():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to the even mantissa (1.0)
    assert bf16.round_rne(np.array([1 + 2.0 ** -8]))[0] == 1.0
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert bf16.round_rne(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert bf16.round_rne(np.array([-(1 + 3 * 2.0 ** -8)]))[0] == -(1 + 2.0 ** -6)
    bits = np.array([0x3F80, 0xC000, 0x3E80, 0x0000], dtype=np.uint16)
    assert list(bf16.decode(bits)) == [1.0, -2.0, 0.25, 0.0]
    assert bf16.ulp(np.array([1.0]))[0] == 2.0 ** -7


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------
def _attention_loops(q, k, v, scale):
    """Brute force with Python loops and math.exp."""
    Tq, Hq, dh = q.shape
    Tk, Hkv, _ = k.shape
    group = Hq // Hkv
    out = np.zeros((Tq, Hq, v.shape[2]))
    for i in range(Tq):
        for h in range(Hq):
            j = h // group
            s = [sum(q[i, h, d] * k[t, j, d] for d in range(dh)) * scale for t in range(Tk)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = sum(e)
            for d in range(v.shape[2]):
                out[i, h, d] = sum(e[t] * v[t, j, d] for t in range(Tk)) / z
    return out


@pytest.mark.parametrize("Hq,Hkv", [(4, 1), (2, 2), (4, 2)])
def test_attention_brute_force(Hq, Hkv):
    q = RNG.standard_normal((5, Hq, 4))
    k = RNG.standard_normal((7, Hkv, 4))
    v = RNG.standard_normal((7, Hkv, 3))
    got = ops.attention(q, k, v, 0.5)
    assert np.allclose(got, _attention_loops(q, k, v, 0.5), rtol=1e-13, atol=1e-14)


def test_attention_special_cases():
    q = RNG.standard_normal((6, 2, 8))
    v = RNG.standard_normal((9, 1, 8))
    k_same = np.repeat(RNG.standard_normal((1, 1, 8)), 9, axis=0)
    # all keys equal -> output is the mean of V
    got = ops.attention(q, k_same, v, 0.3)
    assert np.allclose(got, np.broadcast_to(v.mean(axis=0), got.shape), atol=1e-14)
    # a single key -> output is that V row
    got1 = ops.attention(q, k_same[:1], v[:1], 0.3)
    assert np.allclose(got1, np.broadcast_to(v[0], got1.shape), atol=1e-15)
    # adding one vector to every key shifts each query's scores by a constant
    k = RNG.standard_normal((9, 1, 8))
    delta = RNG.standard_normal((1, 1, 8)) * 3
    assert np.allclose(ops.attention(q, k, v, 0.3), ops.attention(q, k + delta, v, 0.3),
                       rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------
# norms
# ----------------------------------------------------------------------------
def test_rmsnorm_closed_forms():
    eps = 1e-6
    for c in (3.0, -0.5, 1e-4):
        x = np.full((1, 16), c)
        assert np.allclose(ops.rmsnorm(x, eps), c / np.sqrt(c * c + eps), rtol=1e-15)
    x = RNG.standard_normal((4, 64))
    y = ops.rmsnorm(x, 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-14)
    assert np.allclose(ops.rmsnorm(7.0 * x, 0.0), y, rtol=1e-14)  # scale invariance
    ms = np.mean(x * x, axis=-1)
    y = ops.rmsnorm(x, eps)
    assert np.allclose(np.mean(y * y, axis=-1), ms / (ms + eps), rtol=1e-13)


def test_layernorm_closed_forms():
    eps = 1e-6
    x = RNG.standard_normal((5, 128)) * 3 + 2
    y = ops.layernorm(x, eps)
    var = x.var(axis=-1)
    assert np.allclose(y.mean(axis=-1), 0.0, atol=1e-14)
    assert np.allclose(y.var(axis=-1), var / (var + eps), rtol=1e-13)
    assert np.allclose(ops.layernorm(x + 11.0, eps), y, rtol=1e-10, atol=1e-12)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (128,), eps=eps).numpy()
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------
def test_rope_hand_case():
    # dh = 4: pairs (0, 2) with theta 1 and (1, 3) with theta 1e4**-0.5 = 0.01
    x = np.zeros((1, 1, 4)); x[0, 0, 0] = 1.0
    y = ops.rope(x, np.array([1]), 10000.0)
    assert np.allclose(y[0, 0], [math.cos(1.0), 0.0, math.sin(1.0), 0.0], atol=1e-16)
    x = np.zeros((1, 1, 4)); x[0, 0, 3] = 1.0
    y = ops.rope(x, np.array([2]), 10000.0)
    assert np.allclose(y[0, 0], [0.0, -math.sin(0.02), 0.0, math.cos(0.02)], atol=1e-16)


def test_rope_is_complex_rotation():
    dh, base = 64, 10000.0
    x = RNG.standard_normal((9, 3, dh))
    pos = RNG.integers(0, 200_000, 9)
    z = x[..., : dh // 2] + 1j * x[..., dh // 2:]
    theta = base ** (-np.arange(dh // 2) * 2.0 / dh)
    zr = z * np.exp(1j * pos[:, None, None] * theta[None, None, :])
    y = ops.rope(x, pos, base)
    assert np.allclose(y[..., : dh // 2], zr.real, rtol=1e-11, atol=1e-11)
    assert np.allclose(y[..., dh // 2:], zr.imag, rtol=1e-11, atol=1e-11)


def test_rope_invariants():
    dh = 32
    q = RNG.standard_normal((1, 1, dh))
    k = RNG.standard_normal((1, 1, dh))
    assert np.array_equal(ops.rope(q, np.array([0]), 1e4), q)
    assert np.isclose(np.linalg.norm(ops.rope(q, np.array([77]), 1e4)), np.linalg.norm(q))

    def dot(m, n):
        return float(np.sum(ops.rope(q, np.array([m]), 1e4) * ops.rope(k, np.array([n]), 1e4)))

    assert np.isclose(dot(5, 3), dot(105, 103), rtol=1e-11)
    assert np.isclose(dot(0, 9), dot(600, 609), rtol=1e-11)


# ----------------------------------------------------------------------------
# activations and timestep embedding
# ----------------------------------------------------------------------------
def test_gelu_tanh_against_erf_gelu():
    x = np.linspace(-8, 8, 20001)
    erf_gelu = 0.5 * x * (1 + np.array([math.erf(v / math.sqrt(2)) for v in x]))
    dev = np.max(np.abs(ops.gelu_tanh(x) - erf_gelu))
    assert dev < 5e-4  # the tanh form's known max deviation is about 4.7e-4 (|x| ~ 2.1)
    assert ops.gelu_tanh(np.array([0.0]))[0] == 0.0
    assert np.isclose(ops.gelu_tanh(np.array([12.0]))[0], 12.0)
    assert abs(ops.gelu_tanh(np.array([-12.0]))[0]) < 1e-12
    tg = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.allclose(ops.gelu_tanh(x), tg, rtol=1e-12, atol=1e-13)


def test_silu_library():
    x = np.linspace(-30, 30, 1001)
    assert np.allclose(ops.silu(x), torch.nn.functional.silu(torch.from_numpy(x)).numpy(),
                       rtol=1e-13, atol=1e-15)


def test_timestep_embedding_closed_forms():
    e0 = ops.timestep_embedding(0.0, 8)
    assert np.array_equal(e0, [0, 0, 0, 0, 1, 1, 1, 1])
    e = ops.timestep_embedding(0.25, 8)
    w = 10000.0 ** (-np.arange(4) / 4)
    assert np.isclose(e[0], math.sin(250.0))           # lowest index: frequency 1
    assert np.isclose(e[3], math.sin(250.0 * w[3]))
    assert np.isclose(e[7], math.cos(250.0 * w[3]))
    assert np.allclose(e[:4] ** 2 + e[4:] ** 2, 1.0)


# ----------------------------------------------------------------------------
# folds (section 4 of the reading note)
# ----------------------------------------------------------------------------
def _tiny_cfg():
    return synth.config("tiny", D=32, Hq=2, Hkv=1, dh=16, F=48, T_prefix=8, T_q=6, act_dim=4)


def _tiny_pi0(seed=3):
    cfg = _tiny_cfg()
    wb = synth.pi0_weights(cfg, seed)
    ib = synth.pi0_inputs(cfg, seed)
    return cfg, wb, ib


def test_rmsnorm_scale_fold_identity():
    cfg, wb, ib = _tiny_pi0()
    blk = pi0.decode_tree(wb["blocks"][0])
    kv = bf16.decode(ib["kv"][0])
    x = RNG.standard_normal((cfg["T_q"], cfg["D"]))
    pos = cfg["T_prefix"] + np.arange(cfg["T_q"])
    Tp = cfg["T_prefix"]
    unfused, _, _ = pi0.block(x, kv[0, :Tp], kv[1, :Tp], pos, blk, cfg)
    exact = dict(blk)
    one = np.ones(cfg["D"])
    exact.update(g_attn=one, g_ffn=one,
                 wq=fold.fold_scale_exact(blk["g_attn"], blk["wq"]),
                 wk=fold.fold_scale_exact(blk["g_attn"], blk["wk"]),
                 wv=fold.fold_scale_exact(blk["g_attn"], blk["wv"]),
                 wg=fold.fold_scale_exact(blk["g_ffn"], blk["wg"]),
                 wu=fold.fold_scale_exact(blk["g_ffn"], blk["wu"]))
    folded, _, _ = pi0.block(x, kv[0, :Tp], kv[1, :Tp], pos, exact, cfg)
    # the cache write rounds K/V to bf16 and both sides see the same rounding
    # unless a value sits on a tie; compare on the residual stream
    assert np.allclose(folded, unfused, rtol=1e-12, atol=1e-12)
    # the stored fold is the exact product rounded once to bf16
    st = fold.fold_scale(blk["g_attn"], blk["wq"])
    ex = fold.fold_scale_exact(blk["g_attn"], blk["wq"])
    assert np.all(np.abs(st - ex) <= 2.0 ** -8 * np.abs(ex))
    assert np.array_equal(st, bf16.round_rne(ex))


def test_merged_qkv_equals_separate():
    cfg, wb, _ = _tiny_pi0()
    w = pi0.method_block(pi0.decode_tree(wb["blocks"][0]))
    x = RNG.standard_normal((cfg["T_q"], cfg["D"]))
    q, k, v = pi0.qkv(x, w, cfg)
    xn = ops.rmsnorm(x, cfg["eps"])
    assert np.allclose(q.reshape(len(x), -1), xn @ w["wq"], rtol=1e-14, atol=1e-15)
    assert np.allclose(k.reshape(len(x), -1), xn @ w["wk"], rtol=1e-14, atol=1e-15)
    assert np.allclose(v.reshape(len(x), -1), xn @ w["wv"], rtol=1e-14, atol=1e-15)


def test_time_embedding_fold():
    cfg, wb, ib = _tiny_pi0()
    W = pi0.decode_tree({k: v for k, v in wb.items() if k != "blocks"})
    w_fold, table = pi0.fold_tables(wb, cfg)
    x = np.asarray(ib["noise"], np.float64)
    for s, t in enumerate(pi0.times(cfg)):
        a = pi0.embed(x, t, W, cfg["D"])
        b = pi0.embed_folded(x, s, w_fold, table, W)
        assert np.allclose(a, b, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------
# Euler integration and block wiring
# ----------------------------------------------------------------------------
def test_time_grid():
    assert pi0.times(synth.config("pi0_ae")) == [s / 10 for s in range(10)]


def test_constant_velocity_field_integrates_exactly():
    """W_out = 0, b_out = c  =>  v = c at every step  =>  x_S = x_0 + S dt c = x_0 + c."""
    cfg, wb, ib = _tiny_pi0()
    cfg = dict(cfg, S=5)
    wb = dict(wb)
    wb["w_out"] = np.zeros_like(wb["w_out"])
    c = bf16.round_rne(RNG.standard_normal(cfg["act_dim"]))
    wb["b_out"] = bf16.encode(c)
    x, _ = pi0.denoise(ib["noise"], ib["state"], ib["kv"], wb, cfg)
    assert np.allclose(x, ib["noise"] + c[None, :], rtol=0, atol=1e-14)


def test_linear_velocity_euler_closed_form():
    """x_{s+1} = x_s + dt (a x_s + c) has x_S = (1+a dt)^S x0 + c dt sum_k (1+a dt)^k."""
    a, c, S = -0.7, 0.3, 10
    dt = 1.0 / S
    x0 = RNG.standard_normal(5)
    x = x0.copy()
    for _ in range(S):
        x = x + dt * (a * x + c)
    r = 1 + a * dt
    assert np.allclose(x, r ** S * x0 + c * dt * sum(r ** k for k in range(S)), rtol=1e-14)


def test_block_identity_and_wiring():
    cfg, wb, ib = _tiny_pi0()
    blk = pi0.decode_tree(wb["blocks"][0])
    Tp, T = cfg["T_prefix"], cfg["T_q"]
    kv = bf16.decode(ib["kv"][0])
    x = RNG.standard_normal((T, cfg["D"]))
    pos = Tp + np.arange(T)
    zero = dict(blk, wo=np.zeros_like(blk["wo"]), wd=np.zeros_like(blk["wd"]))
    y, k_own, v_own = pi0.block(x, kv[0, :Tp], kv[1, :Tp], pos, zero, cfg)
    assert np.array_equal(y, x)
    # q = 0 -> uniform attention over [prefix | own]: o = mean of all V rows,
    # the prefix from the cache, the own rows as computed
    unif = dict(blk, wq=np.zeros_like(blk["wq"]), wd=np.zeros_like(blk["wd"]))
    y, k_own, v_own = pi0.block(x, kv[0, :Tp], kv[1, :Tp], pos, unif, cfg)
    xn = ops.rmsnorm(x, cfg["eps"]) * blk["g_attn"]
    v_exact = xn @ blk["wv"]
    vmean = np.concatenate([kv[1, :Tp], v_exact]).mean(axis=0)          # [Hkv*dh]
    o = np.tile(vmean, cfg["Hq"] // cfg["Hkv"])                          # every q head
    assert np.allclose(y, x + o[None, :] @ blk["wo"], rtol=1e-12, atol=1e-13)
    # the cache receives the bf16 of the projected (un-rotated) values
    assert np.array_equal(v_own, bf16.round_rne(v_exact))
    # with attention removed the FFN sees the *normed* residual (pre-norm)
    noatt = dict(blk, wo=np.zeros_like(blk["wo"]))
    y, _, _ = pi0.block(x, kv[0, :Tp], kv[1, :Tp], pos, noatt, cfg)
    hn = ops.rmsnorm(x, cfg["eps"]) * blk["g_ffn"]
    ffn = (ops.gelu_tanh(hn @ blk["wg"]) * (hn @ blk["wu"])) @ blk["wd"]
    assert np.allclose(y, x + ffn, rtol=1e-12, atol=1e-13)


def test_prefill_last_layer_skip_leaves_kv_unchanged():
    cfg = synth.config("prefill", D=32, Hq=2, Hkv=1, dh=16, F=48, L=3, T_prefix=8,
                       T_q=4, patch_dim=12)
    wb = synth.prefill_weights(cfg, 5)
    pe = synth.prefill_inputs(cfg, 2, 5)["patch_emb"]
    a = pi0.prefill(pe, wb, cfg, skip_last=True)
    b = pi0.prefill(pe, wb, cfg, skip_last=False)
    assert np.array_equal(a, b)
    assert not np.any(a[:, :, :, cfg["T_prefix"]:])   # own-token slots untouched
    # batch elements are independent
    a1 = pi0.prefill(pe[1:2], wb, cfg)
    assert np.array_equal(a[:, 1:2], a1)


# ----------------------------------------------------------------------------
# DiT stage: ring, batching, adaLN wiring
# ----------------------------------------------------------------------------
def test_ring_slot_matches_fifo_simulation():
    nh = 4
    slots = [None] * (nh + 1)      # slot -> chunk living there
    where = {}
    for c in range(40):
        if c >= nh + 1:            # the chunk that leaves the window frees its slot
            free = where.pop(c - nh - 1)
        else:
            free = slots.index(None)
        slots[free] = c
        where[c] = free
        assert free == dit.ring_slot(c, nh)
        visible = sorted(ch for ch in slots if ch is not None and ch != c)
        assert visible == dit.history_chunks(c, nh)
    assert list(dit.positions(3, 1560)[[0, -1]]) == [4680, 6239]


def _tiny_dit(seed=2):
    cfg = synth.config("dit_1p3b", D=32, H=2, dh=16, F=40, L=1, T_chunk=6, t_dim=16)
    wb = synth.dit_weights(cfg, seed)
    W = pi0.decode_tree({k: v for k, v in wb.items() if k != "blocks"})
    w = pi0.decode_tree(wb["blocks"][0])
    table = dit.adaln_table(W, cfg)
    ring = bf16.decode(synth.dit_ring(cfg, seed, streams=2))[:, 0]
    return cfg, w, W, table, ring


def test_dit_batch_equals_separate_calls():
    cfg, w, _, table, ring = _tiny_dit()
    descs = [(0, 9, 0), (0, 8, 1), (0, 7, 2), (1, 2, 3)]
    xs = synth.dit_latents(cfg, len(descs), 4)
    r_batch = ring.copy()
    out = dit.block_batch(xs, descs, r_batch, table, w, cfg)
    r_sep = ring.copy()
    for b, d in enumerate(descs):
        ob = dit.block_batch(xs[b:b + 1], [d], r_sep, table, w, cfg)
        assert np.array_equal(ob[0], out[b])
    assert np.array_equal(r_sep, r_batch)
    rows = [0, 3, 5]
    r_rows = ring.copy()
    part = dit.block_batch_rows(xs, descs, r_rows, table, w, cfg, rows)
    assert np.allclose(part, out[:, rows], rtol=1e-12, atol=1e-12)
    assert np.array_equal(r_rows, r_batch)


def test_dit_zero_gates_is_identity_and_history_set():
    cfg, w, W, table, ring = _tiny_dit()
    D = cfg["D"]
    W0 = dict(W, wmod=np.zeros_like(W["wmod"]))
    bm = RNG.standard_normal(6 * D)
    bm[2 * D:3 * D] = 0.0          # gate1
    bm[5 * D:6 * D] = 0.0          # gate2
    W0["bmod"] = bm
    t0 = dit.adaln_table(W0, cfg)
    assert np.allclose(t0, bm[None, :])
    xs = synth.dit_latents(cfg, 1, 8)
    out = dit.block_batch(xs, [(0, 6, 1)], ring.copy(), t0, w, cfg)
    assert np.array_equal(out[0], xs[0].astype(np.float64))
    # q = 0 -> uniform attention: o = mean of V over history chunks + own chunk
    bm2 = RNG.standard_normal(6 * D) * 0.1
    t2 = np.broadcast_to(bm2, (cfg["S"], 6 * D)).copy()
    wz = dict(w, wq=np.zeros_like(w["wq"]), w2=np.zeros_like(w["w2"]))
    u = ops.layernorm(xs[0].astype(np.float64), cfg["eps"]) * (1 + bm2[D:2 * D]) + bm2[:D]
    v_own = u @ w["wv"]
    for c in (0, 2, 9):
        r = ring.copy()
        out = dit.block_batch(xs, [(0, c, 1)], r, t2, wz, cfg)
        hist = [cc for cc in range(c - 4, c) if cc >= 0]
        V = np.concatenate([r[0, 1, cc % 5, 1] for cc in hist] + [v_own])
        assert np.array_equal(r[0, 1, c % 5, 1], bf16.round_rne(v_own))
        o = V.mean(axis=0)
        expect = xs[0] + bm2[2 * D:3 * D] * (o[None, :] @ w["wo"])
        assert np.allclose(out[0], expect, rtol=1e-12, atol=1e-12)


def test_dit_ffn_branch_closed_form():
    # gate1 = 0 leaves h = x; scale2 = -1 turns LN(h)(1 + scale2) + shift2 into
    # the shift row for every token, so the block is
    # x + gate2 * (GELU(shift2 W1) W2): the second modulation triple's order, its
    # "1 +" and the FFN wiring, against matrix products and the pinned GELU
    cfg, w, W, table, ring = _tiny_dit()
    D = cfg["D"]
    bm = RNG.standard_normal(6 * D) * 0.5
    bm[2 * D:3 * D] = 0.0          # gate1
    bm[4 * D:5 * D] = -1.0         # scale2
    t = np.broadcast_to(bm, (cfg["S"], 6 * D)).copy()
    xs = synth.dit_latents(cfg, 1, 9)
    out = dit.block_batch(xs, [(0, 5, 2)], ring.copy(), t, w, cfg)
    sh2, g2 = bm[3 * D:4 * D], bm[5 * D:6 * D]
    f = ops.gelu_tanh(sh2[None, :] @ w["w1"]) @ w["w2"]
    expect = xs[0].astype(np.float64) + g2 * f
    assert np.allclose(out[0], expect, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# Interleaved stage schedule of chunked AR diffusion (latent in/out + Euler)
# ---------------------------------------------------------------------------
def _pipe_dit(seed=3, L=2, S=4):
    cfg = synth.config("dit_1p3b", D=32, H=2, dh=16, F=40, L=L, S=S, T_chunk=6, t_dim=16, lat_dim=8)
    wb = synth.dit_weights(cfg, seed)
    W = pi0.decode_tree({k: v for k, v in wb.items() if k != "blocks"})
    W["blocks"] = [pi0.decode_tree(b) for b in wb["blocks"]]
    table = dit.adaln_table(W, cfg)
    rings = np.zeros((1, L, S, cfg["n_hist"] + 1, 2, cfg["T_chunk"], cfg["D"]))
    return cfg, W, table, rings


def test_dit_interleaved_schedule():
    """Chunk c is at step s during interval c + s; one chunk per step and slot."""
    S, n = 4, 7
    seen = {}
    for i in range(n + S - 1):
        ds = dit.interval_descs(i, n, S)
        steps = [s for (_, _, s) in ds]
        assert len(set(steps)) == len(steps) and all(0 <= s < S for s in steps)
        slots = [c % S for (_, c, _) in ds]
        assert slots == sorted(slots) and len(set(slots)) == len(slots)
        for (_, c, s) in ds:
            seen.setdefault(c, []).append((i, s))
    assert sorted(seen) == list(range(n))
    for c in range(n):
        assert seen[c] == [(c + s, s) for s in range(S)]


def test_dit_pipeline_equals_sequential():
    """The interleaved order reads exactly the history KV the plain order reads."""
    cfg, W, table, rings = _pipe_dit()
    noises = synth.dit_noise(cfg, 6, 5)
    r_pipe, r_seq = rings.copy(), rings.copy()
    a = dit.pipeline(list(noises), r_pipe, table, W, cfg)
    b = dit.sequential(list(noises), r_seq, table, W, cfg)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert np.array_equal(r_pipe, r_seq)
    assert not np.array_equal(a[0], np.asarray(noises[0], np.float64))


def test_dit_pipeline_linear_field_closed_form():
    """Identity blocks (zero adaLN gates): z <- z + dt ((z W_in + b_in) W_out + b_out)
    is linear, so after S steps z_S = z_0 P^S + dt k sum_{j<S} P^j with
    P = I + dt W_in W_out and k = b_in W_out + b_out."""
    cfg, W, _, rings = _pipe_dit()
    D, S = cfg["D"], cfg["S"]
    dt = 1.0 / S
    bm = RNG.standard_normal(6 * D)
    bm[2 * D:3 * D] = 0.0
    bm[5 * D:6 * D] = 0.0
    W0 = dict(W, wmod=np.zeros_like(W["wmod"]), bmod=bm)
    table = dit.adaln_table(W0, cfg)
    noises = synth.dit_noise(cfg, 3, 7)
    out = dit.pipeline(list(noises), rings.copy(), table, W0, cfg)
    P = np.eye(cfg["lat_dim"]) + dt * (W["w_in"] @ W["w_out"])
    k = W["b_in"] @ W["w_out"] + W["b_out"]
    geo = sum(np.linalg.matrix_power(P, j) for j in range(S))
    for z0, z in zip(noises, out):
        ref = np.asarray(z0, np.float64) @ np.linalg.matrix_power(P, S) + dt * (k @ geo)
        assert np.allclose(z, ref, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------------------
# pi0 block mask variant (state token sees the prefix and itself only)
# ---------------------------------------------------------------------------
def test_masked_attention_is_attention_over_the_allowed_keys():
    q = RNG.standard_normal((5, 2, 4))
    k = RNG.standard_normal((7, 1, 4))
    v = RNG.standard_normal((7, 1, 3))
    allow = RNG.random((5, 7)) < 0.6
    allow[:, 2] = True                              # every row sees at least one key
    got = ops.attention(q, k, v, 0.5, allow=allow)
    for t in range(5):
        keys = np.flatnonzero(allow[t])
        ref = _attention_loops(q[t:t + 1], k[keys], v[keys], 0.5)
        assert np.allclose(got[t:t + 1], ref, rtol=1e-13, atol=1e-14)


def test_pi0_prefix_lm_mask():
    """With the block mask the state token's row equals a block run on the state
    token alone (it sees the prefix and itself), and the action rows equal the
    unmasked block's (they see every key either way)."""
    cfg, wb, ib = _tiny_pi0()
    blk = pi0.decode_tree(wb["blocks"][0])
    kv = bf16.decode(ib["kv"][0])
    x = RNG.standard_normal((cfg["T_q"], cfg["D"]))
    Tp = cfg["T_prefix"]
    pos = Tp + np.arange(cfg["T_q"])
    full, _, _ = pi0.block(x, kv[0, :Tp], kv[1, :Tp], pos, blk, cfg)
    cm = dict(cfg, prefix_lm=1)
    masked, k_m, v_m = pi0.block(x, kv[0, :Tp], kv[1, :Tp], pos, blk, cm)
    alone, _, _ = pi0.block(x[:1], kv[0, :Tp], kv[1, :Tp], pos[:1], blk, cm)
    assert np.allclose(masked[0], alone[0], rtol=1e-12, atol=1e-13)
    assert np.array_equal(masked[1:], full[1:])
    assert not np.allclose(masked[0], full[0])


# ----------------------------------------------------------------------------
# action head, state token, adaLN table, prefix patch projection: closed forms
# on hand-built weights (each would miss a dropped term with random weights
# that the network-level pins zero out)
# ----------------------------------------------------------------------------
def test_head_closed_form():
    """Rows h_r = a_r u with u a +-1 vector: mean(h_r^2) = a_r^2, so RMSNorm
    gives a_r u / sqrt(a_r^2 + eps); W_out picks the first A dimensions, so the
    velocity is that row times g_final on those dimensions, plus b_out."""
    D, A, eps = 16, 4, 1e-6
    u = np.where(RNG.standard_normal(D) > 0, 1.0, -1.0)
    a = np.array([3.0, -0.5, 7.25])
    h = a[:, None] * u[None, :]
    g = 1.5 + 0.25 * np.arange(D)
    w_out = np.zeros((D, A))
    w_out[np.arange(A), np.arange(A)] = 1.0
    b = np.array([0.5, -1.0, 2.0, 0.0])
    v = pi0.head(h, {"g_final": g, "w_out": w_out, "b_out": b}, eps)
    expect = (a / np.sqrt(a * a + eps))[:, None] * (u[:A] * g[:A])[None, :] + b[None, :]
    assert np.allclose(v, expect, rtol=1e-14, atol=1e-15)


def test_denoise_wiring_with_identity_blocks():
    """Blocks with W_o = W_d = 0 are the identity, so each Euler step is
    x <- x + dt head(embed(x, t_s)) on the action rows (the state row is not
    integrated): the loop's order of embedding, head, rows and time grid."""
    cfg, wb, ib = _tiny_pi0()
    cfg = dict(cfg, S=3)
    wb = dict(wb)
    blocks = []
    for b in wb["blocks"]:
        b = dict(b)
        b["wo"] = bf16.encode(np.zeros(b["wo"].shape))
        b["wd"] = bf16.encode(np.zeros(b["wd"].shape))
        blocks.append(b)
    wb["blocks"] = blocks
    W = pi0.decode_tree({k: v for k, v in wb.items() if k != "blocks"})
    x, _ = pi0.denoise(ib["noise"], ib["state"], ib["kv"], wb, cfg)
    ref = np.asarray(ib["noise"], np.float64)
    for s in range(cfg["S"]):
        ref = ref + (1.0 / cfg["S"]) * pi0.head(pi0.embed(ref, s / cfg["S"], W, cfg["D"]), W, cfg["eps"])
    assert np.allclose(x, ref, rtol=1e-12, atol=1e-13)


def test_state_token_closed_form():
    state = np.array([1.0, -2.0, 0.5, 3.0])
    w = np.zeros((4, 8))
    w[0, 0], w[1, 3], w[3, 7] = 2.0, 1.0, -1.0
    b = 0.5 * np.arange(8) + 0.25
    got = pi0.state_token(state, {"w_state": w, "b_state": b})
    expect = b.copy()
    expect[0] += 2.0
    expect[3] += -2.0
    expect[7] += -3.0
    assert np.array_equal(got, expect)


def test_adaln_table_closed_form():
    """Wt1 routes cos(1000 t) (the embedding's first cosine, frequency 1) to
    every hidden unit, Wt2 is the identity and Wmod repeats its input six
    times, so A[s][kD + j] = SiLU(SiLU(cos(1000 t_s) + bt1_j) + bt2_j) + bmod_{kD+j}
    with t_s = s / S; SiLU from the library."""
    D, td, S = 4, 16, 4
    wt1 = np.zeros((td, D))
    wt1[td // 2, :] = 1.0
    bt1 = np.array([0.5, -1.0, 0.0, 2.0])
    bt2 = np.array([0.0, 0.25, -0.5, 1.0])
    bmod = np.linspace(-1.0, 1.0, 6 * D)
    W = {"wt1": wt1, "bt1": bt1, "wt2": np.eye(D), "bt2": bt2, "wmod": np.tile(np.eye(D), (1, 6)), "bmod": bmod}
    A = dit.adaln_table(W, {"S": S, "t_dim": td})
    silu = torch.nn.functional.silu
    for s in range(S):
        z = torch.tensor(math.cos(1000.0 * s / S) + bt1, dtype=torch.float64)
        e = silu(z) + torch.from_numpy(bt2)
        expect = np.tile(silu(e).numpy(), 6) + bmod
        assert np.allclose(A[s], expect, rtol=1e-13, atol=1e-14)


def test_prefill_patch_projection():
    """One-hot patch embeddings pick rows of W_patch, so layer 0's K/V are the
    first block's K/V of h_i = W_patch[j_i] + b_patch at positions 0..Tp-1."""
    cfg = synth.config("prefill", D=32, Hq=2, Hkv=1, dh=16, F=48, L=2, T_prefix=8, T_q=4, patch_dim=12)
    wb = synth.prefill_weights(cfg, 7)
    Tp, P = cfg["T_prefix"], cfg["patch_dim"]
    idx = np.array([3, 0, 11, 5, 5, 7, 1, 2])
    pe = np.zeros((1, Tp, P))
    pe[0, np.arange(Tp), idx] = 1.0
    kv = bf16.decode(pi0.prefill(bf16.encode(pe), wb, cfg))
    wp, bp = bf16.decode(wb["w_patch"]), bf16.decode(wb["b_patch"])
    assert np.count_nonzero(bp) > cfg["D"] // 2
    h = wp[idx] + bp
    w0 = pi0.method_block(pi0.decode_tree(wb["blocks"][0]))
    empty = np.zeros((0, cfg["Hkv"] * cfg["dh"]))
    _, k, v = pi0.block(h, empty, empty, np.arange(Tp), w0, cfg, kv_only=True)
    assert np.array_equal(kv[0, 0, 0, :Tp], k)
    assert np.array_equal(kv[0, 0, 1, :Tp], v)


# ---------------------------------------------------------------------------
# Wan-class options of the DiT block: 3-D RoPE, text cross-attention, pages
# ---------------------------------------------------------------------------
def test_rope_bands_split():
    # frame d - 4 floor(d/6), height and width 2 floor(d/6): contiguous, even widths
    assert ops.rope_bands(128) == [(0, 44), (44, 42), (86, 42)]
    assert ops.rope_bands(64) == [(0, 24), (24, 20), (44, 20)]
    for dh in (16, 32, 96, 128, 256):
        b = ops.rope_bands(dh)
        assert b[0][0] == 0 and b[1][0] == b[0][1] and b[2][0] == b[1][0] + b[1][1]
        assert sum(w for _, w in b) == dh and all(w % 2 == 0 for _, w in b)


def test_positions3_hand_cases():
    cfg = synth.config("dit_1p3b", T_chunk=24, grid_h=4, grid_w=3)   # 2 frames of 4 x 3
    p = dit.positions3(5, cfg)
    assert p.shape == (24, 3)
    assert list(p[0]) == [10, 0, 0] and list(p[2]) == [10, 0, 2] and list(p[3]) == [10, 1, 0]
    assert list(p[11]) == [10, 3, 2] and list(p[12]) == [11, 0, 0] and list(p[23]) == [11, 3, 2]
    # one frame's (y, x) are all distinct; the configs' chunk is one 30 x 52 frame
    assert len({(y, x) for _, y, x in p[:12]}) == 12
    big = synth.config("dit_1p3b", grid_h=30, grid_w=52)
    q = dit.positions3(3, big)
    assert q[0].tolist() == [3, 0, 0] and q[-1].tolist() == [3, 29, 51] and q[52].tolist() == [3, 1, 0]


def test_rope3d_reduces_to_rope_per_band():
    dh, base = 32, 10000.0
    x = RNG.standard_normal((7, 2, dh))
    pos = RNG.integers(0, 500, (7, 3))
    y = ops.rope3d(x, pos, base)
    for b, (o, w) in enumerate(ops.rope_bands(dh)):
        assert np.allclose(y[..., o:o + w], ops.rope(x[..., o:o + w], pos[:, b], base), rtol=1e-13, atol=1e-13)
        # a vector living on band b turns with coordinate b only
        xb = np.zeros_like(x)
        xb[..., o:o + w] = x[..., o:o + w]
        moved = pos.copy()
        moved[:, [i for i in range(3) if i != b]] += 17
        assert np.allclose(ops.rope3d(xb, pos, base), ops.rope3d(xb, moved, base), rtol=1e-13, atol=1e-13)


def test_rope3d_scores_depend_on_relative_position_only():
    dh, base = 48, 10000.0
    q = RNG.standard_normal((1, 1, dh))
    k = RNG.standard_normal((1, 1, dh))

    def dot(a, b):
        return float(np.sum(ops.rope3d(q, np.array([a]), base) * ops.rope3d(k, np.array([b]), base)))

    a, b, shift = np.array([3, 1, 4]), np.array([1, 5, 9]), np.array([40, 7, 11])
    assert np.isclose(dot(a, b), dot(a + shift, b + shift), rtol=1e-11)
    assert not np.isclose(dot(a, b), dot(a, b + np.array([0, 1, 0])), rtol=1e-6)


def _tiny_wan(seed=4, **over):
    cfg = synth.config("dit_1p3b", D=32, H=2, dh=16, F=40, L=1, T_chunk=12, t_dim=16,
                       grid_h=2, grid_w=3, text_len=5, **over)
    wb = synth.dit_weights(cfg, seed)
    W = pi0.decode_tree({k: v for k, v in wb.items() if k != "blocks"})
    w = pi0.decode_tree(wb["blocks"][0])
    table = dit.adaln_table(W, cfg)
    ring = bf16.decode(synth.dit_ring(cfg, seed, streams=2))[:, 0]
    text = bf16.decode(synth.dit_text(cfg, 2, seed))
    return cfg, w, table, ring, text


def test_dit_cross_attention_closed_forms():
    cfg, w, table, ring, text = _tiny_wan()
    D, eps = cfg["D"], cfg["eps"]
    xs = synth.dit_latents(cfg, 1, 5)
    desc = [(1, 6, 2)]
    # W_o^c = 0: the block without its cross-attention sublayer
    off = dit.block_batch(xs, desc, ring.copy(), table, dict(w, co=np.zeros_like(w["co"])), dict(cfg, text_len=0))
    on0 = dit.block_batch(xs, desc, ring.copy(), table, dict(w, co=np.zeros_like(w["co"])), cfg, text)
    assert np.array_equal(off, on0)
    # gate1 = gate2 = 0 isolates the sublayer: x' = x + cross(x)
    tz = table.copy()
    tz[:, 2 * D:3 * D] = 0.0
    tz[:, 5 * D:6 * D] = 0.0
    x0 = xs[0].astype(np.float64)
    # one text token: softmax = 1, every row gets (ctx W_v^c) W_o^c
    one = dict(cfg, text_len=1)
    ctx1 = text[:, :1]
    out = dit.block_batch(xs, desc, ring.copy(), tz, w, one, ctx1)
    expect = x0 + (ctx1[1] @ w["cv"]) @ w["co"]
    assert np.allclose(out[0], expect, rtol=1e-12, atol=1e-12)
    # g_c = b_c = 0: q = 0, uniform weights, every row gets mean(ctx W_v^c) W_o^c;
    # LN affine pinned with b_c alone (g_c = 0): q = b_c W_q^c for every row
    wz = dict(w, g_c=np.zeros(D), b_c=np.zeros(D))
    out = dit.block_batch(xs, desc, ring.copy(), tz, wz, cfg, text)
    expect = x0 + (text[1] @ w["cv"]).mean(axis=0) @ w["co"]
    assert np.allclose(out[0], expect, rtol=1e-12, atol=1e-12)
    wb_ = dict(w, g_c=np.zeros(D))
    out = dit.block_batch(xs, desc, ring.copy(), tz, wb_, cfg, text)
    H, dh = cfg["H"], cfg["dh"]
    q = (w["b_c"] @ w["cq"]).reshape(H, dh)
    k = (text[1] @ w["ck"]).reshape(-1, H, dh)
    v = (text[1] @ w["cv"]).reshape(-1, H, dh)
    o = np.empty(D)
    for h in range(H):
        z = k[:, h] @ q[h] / math.sqrt(dh)
        p = np.exp(z - z.max())
        o[h * dh:(h + 1) * dh] = (p / p.sum()) @ v[:, h]
    assert np.allclose(out[0], x0 + o @ w["co"], rtol=1e-12, atol=1e-12)
    # with the affine: rows see LN(h) g_c + b_c (brute force on one row)
    out = dit.block_batch(xs, desc, ring.copy(), tz, w, cfg, text)
    r = 4
    u = ops.layernorm(x0[r:r + 1], eps)[0] * w["g_c"] + w["b_c"]
    qr = (u @ w["cq"]).reshape(H, dh)
    for h in range(H):
        z = k[:, h] @ qr[h] / math.sqrt(dh)
        p = np.exp(z - z.max())
        o[h * dh:(h + 1) * dh] = (p / p.sum()) @ v[:, h]
    assert np.allclose(out[0, r], x0[r] + o @ w["co"], rtol=1e-12, atol=1e-12)


def test_dit_wan_block_rows_and_batch():
    cfg, w, table, ring, text = _tiny_wan()
    descs = [(0, 9, 0), (1, 3, 2)]
    xs = synth.dit_latents(cfg, 2, 6)
    r_batch = ring.copy()
    out = dit.block_batch(xs, descs, r_batch, table, w, cfg, text)
    rows = [0, 5, 11]
    r_rows = ring.copy()
    part = dit.block_batch_rows(xs, descs, r_rows, table, w, cfg, rows, text)
    assert np.allclose(part, out[:, rows], rtol=1e-12, atol=1e-12)
    assert np.array_equal(r_rows, r_batch)
    # 3-D RoPE in the block: k written to the ring is the 3-D rotation of u W_k
    D, T = cfg["D"], cfg["T_chunk"]
    sh1, sc1 = table[0, :D], table[0, D:2 * D]
    u = ops.layernorm(xs[0].astype(np.float64), cfg["eps"]) * (1 + sc1) + sh1
    k = ops.rope3d((u @ w["wk"]).reshape(T, cfg["H"], cfg["dh"]), dit.positions3(9, cfg), cfg["rope_base"])
    assert np.array_equal(r_batch[0, 0, 9 % 5, 0], bf16.round_rne(k.reshape(T, D)))


def test_page_pool_round_trip_and_hand_case():
    cfg = synth.config("dit_1p3b", D=8, T_chunk=24, page_tokens=10)
    assert dit.pages_per_ring(cfg) == 12            # 5 slots x 24 tokens = 120 = 12 pages
    table, n_pool = synth.dit_page_table(cfg, streams=2, layers=3)
    assert table.shape == (2, 3, cfg["S"], 12) and n_pool == 2 * 3 * cfg["S"] * 12 + 3
    assert len(np.unique(table)) == table.size and table.min() >= 0 and table.max() < n_pool
    ring = RNG.standard_normal((2, 3, cfg["S"], 5, 2, 24, 8))
    pool = dit.ring_to_pool(ring, table, cfg, n_pool)
    # ring row r = slot * T + j lives at page table[r // P], offset r % P:
    # slot 1, token 23 is row 47 -> page table[4], offset 7 (a chunk boundary inside a page)
    assert np.array_equal(pool[table[1, 2, 3, 4], :, 7], ring[1, 2, 3, 1, :, 23])
    assert np.array_equal(pool[table[0, 1, 0, 2], :, 3], ring[0, 1, 0, 0, :, 23])
    assert np.array_equal(pool[table[0, 1, 0, 2], :, 4], ring[0, 1, 0, 1, :, 0])
    assert np.array_equal(dit.pool_to_ring(pool, table, cfg, 2, 3), ring)
