"""GPU parity of the pi0 action-expert path against the CPU oracle.

All calls go through the C ABI (liblat.so via ctypes).  Inputs come from the
seeded generator only; expected values come from ``oracle/`` only.
"""
import ctypes

import numpy as np
import pytest
import torch

from latency_transformer_block_gb300 import lat, synth
from latency_transformer_block_gb300.models import Pi0ActionExpert, bits_of
from oracle import bf16, pi0
from tests.parity import BLOCK_TOL, FINAL_TOL, assert_bf16_close, assert_rel, assert_scale_rel

pytestmark = pytest.mark.gpu

_CACHE = {}


def _model(name, **over):
    key = (name, tuple(sorted(over.items())))
    if key not in _CACHE:
        cfg = synth.config(name, **over)
        wb = synth.pi0_weights(cfg, 0)
        _CACHE[key] = (cfg, wb, Pi0ActionExpert(cfg, wb))
    return _CACHE[key]


def _run_block(name, layer=0, seed=0, **over):
    cfg, wb, m = _model(name, **over)
    ib = synth.pi0_inputs(cfg, seed)
    x = synth.residual_stream(cfg, seed)
    kv_l = ib["kv"][layer]
    xd = torch.from_numpy(x).cuda()
    kvd = m.kv_from_bits(kv_l)
    m.block(layer, xd, kvd)
    m.ctx.sync()
    got_x = xd.cpu().numpy()
    got_kv = bits_of(kvd)
    ref_x, k_own, v_own = pi0.block_step(x, kv_l, wb["blocks"][layer], cfg)
    Tp = cfg["T_prefix"]
    return cfg, got_x, ref_x, got_kv, kv_l, k_own, v_own, Tp


@pytest.mark.parametrize("name,over,layer", [
    ("tiny", {}, 0),
    ("tiny", {"T_q": 40, "T_prefix": 100}, 0),     # ragged tokens and key blocks
    ("tiny", {"T_q": 2, "T_prefix": 0}, 0),        # degenerate: state + 1 action, no prefix
    ("pi0_ae", {}, 0),
    ("pi0_ae", {}, 17),
    ("tiny", {"prefix_lm": 1}, 0),                 # block mask: the state token sees prefix + itself
    ("pi0_ae", {"prefix_lm": 1}, 0),
])
def test_block_parity(name, over, layer):
    cfg, got_x, ref_x, got_kv, kv_in, k_own, v_own, Tp = _run_block(name, layer, **over)
    assert_rel(got_x, ref_x, BLOCK_TOL, f"{name} block {layer} residual")
    assert_bf16_close(got_kv[0, Tp:], k_own, f"{name} own K")
    assert_bf16_close(got_kv[1, Tp:], v_own, f"{name} own V")
    assert np.array_equal(got_kv[:, :Tp], kv_in[:, :Tp]), "prefix slots must not change"


@pytest.mark.parametrize("name,over", [("tiny", {}), ("tiny", {"T_q": 33, "T_prefix": 70, "S": 3}),
                                       ("tiny", {"prefix_lm": 1}), ("pi0_ae", {})])
def test_denoise_parity(name, over):
    cfg, wb, m = _model(name, **over)
    ib = synth.pi0_inputs(cfg, 1)
    kv = m.kv_from_bits(ib["kv"])
    state = torch.from_numpy(ib["state"]).cuda()
    x = torch.from_numpy(ib["noise"]).cuda()
    m.denoise(kv, state, x)
    m.ctx.sync()
    got = x.cpu().numpy()
    ref, ref_kv = pi0.denoise(ib["noise"], ib["state"], ib["kv"], wb, cfg)
    assert_rel(got, ref, FINAL_TOL, f"{name} actions")
    Tp = cfg["T_prefix"]
    got_kv = bits_of(kv)
    assert np.array_equal(got_kv[:, :, :Tp], ib["kv"][:, :, :Tp])
    # own slots hold the last step's K/V, bf16 values that sit at the end of the
    # whole chain; near the 1e-3 floor one bf16 ulp alone is up to 0.8 %, so they
    # are held to the final tolerance relative to their RMS (scale-relative)
    assert_scale_rel(bf16.decode(got_kv[:, :, Tp:]), bf16.decode(ref_kv[:, :, Tp:]), FINAL_TOL,
                     f"{name} final own KV")


def test_constant_velocity_field_is_exact():
    """W_out = 0, b_out = c  =>  actions = noise + c (up to fp32 rounding of S additions)."""
    cfg = synth.config("tiny", S=4)
    wb = dict(synth.pi0_weights(cfg, 7))
    wb["w_out"] = np.zeros_like(wb["w_out"])
    c = np.linspace(-1, 1, cfg["act_dim"])
    wb["b_out"] = bf16.encode(c)
    m = Pi0ActionExpert(cfg, wb)
    ib = synth.pi0_inputs(cfg, 7)
    x = torch.from_numpy(ib["noise"]).cuda()
    m.denoise(m.kv_from_bits(ib["kv"]), torch.from_numpy(ib["state"]).cuda(), x)
    m.ctx.sync()
    expect = ib["noise"].astype(np.float64) + bf16.round_rne(c)[None, :]
    assert np.max(np.abs(x.cpu().numpy() - expect)) < 4e-6


def test_graph_replay_and_recapture():
    cfg, wb, m = _model("tiny")
    ib = synth.pi0_inputs(cfg, 3)
    outs = []
    for rep in range(3):
        kv = m.kv_from_bits(ib["kv"])              # new addresses on rep 0 and 1 -> re-capture
        x = torch.from_numpy(ib["noise"]).cuda()
        state = torch.from_numpy(ib["state"]).cuda()
        m.denoise(kv, state, x)
        m.ctx.sync()
        outs.append(x.cpu().numpy())
        if rep == 2:                                # same buffers again: replay
            x.copy_(torch.from_numpy(ib["noise"]))
            kv.copy_(m.kv_from_bits(ib["kv"]))
            m.denoise(kv, state, x)
            m.ctx.sync()
            outs.append(x.cpu().numpy())
    for o in outs[1:]:
        assert np.allclose(o, outs[0], rtol=1e-5, atol=1e-6)


def test_indices_exact():
    cfg, wb, m = _model("pi0_ae")
    slots, pos = m.ctx.debug_indices(n=cfg["T_q"])
    expect = list(cfg["T_prefix"] + np.arange(cfg["T_q"]))
    assert slots == expect and pos == expect


def test_abi_errors():
    cfg, wb, m = _model("tiny")
    ib = synth.pi0_inputs(cfg, 0)
    x = torch.zeros(cfg["T_q"] * cfg["D"] + 4, device="cuda")
    kv = m.kv_from_bits(ib["kv"][0])
    with pytest.raises(lat.LatError) as e:
        m.ctx.block_forward(5, x, kv)
    assert e.value.code == 1   # LAT_ERR_ARG
    bad = ctypes.c_void_p(x.data_ptr() + 4)
    assert lat.lib().lat_block_forward(m.ctx.handle, 0, bad, None, 1, lat.ptr(kv), None) == 3  # LAT_ERR_ALIGN
    assert lat.lib().lat_block_forward(m.ctx.handle, 0, None, None, 1, lat.ptr(kv), None) == 1  # NULL
    with pytest.raises(lat.LatError) as e:
        m.ctx.prefill_kv(x, 1, kv)
    assert e.value.code == 7   # LAT_ERR_STATE
    with pytest.raises(lat.LatError) as e:
        m.ctx.set_schedule([0.0, 0.5])
    assert e.value.code == 2   # LAT_ERR_SHAPE
    m.ctx.sync()


def test_set_schedule_matches_oracle_time_grid():
    cfg = synth.config("tiny", S=3)
    wb = synth.pi0_weights(cfg, 11)
    m = Pi0ActionExpert(cfg, wb)
    t = [0.0, 0.2, 0.55, 1.0]
    m.ctx.set_schedule(t)
    ib = synth.pi0_inputs(cfg, 11)
    x = torch.from_numpy(ib["noise"]).cuda()
    m.denoise(m.kv_from_bits(ib["kv"]), torch.from_numpy(ib["state"]).cuda(), x)
    m.ctx.sync()
    # oracle with the same grid: patch times() and the per-step dt
    ref = _oracle_denoise_with_grid(ib, wb, cfg, t)
    assert_rel(x.cpu().numpy(), ref, FINAL_TOL, "scheduled actions")


def _oracle_denoise_with_grid(ib, wb, cfg, t):
    W = pi0.decode_tree({k: v for k, v in wb.items() if k != "blocks"})
    blocks = [pi0.method_block(pi0.decode_tree(b)) for b in wb["blocks"]]
    kv = bf16.decode(ib["kv"])
    Tp, Tq = cfg["T_prefix"], cfg["T_q"]
    pos = Tp + np.arange(Tq)
    x = ib["noise"].astype(np.float64)
    st = pi0.state_token(ib["state"].astype(np.float64), W)
    for s in range(cfg["S"]):
        h = np.vstack([st[None, :], pi0.embed(x, t[s], W, cfg["D"])])
        for l in range(cfg["L"]):
            h, k_own, v_own = pi0.block(h, kv[l, 0, :Tp], kv[l, 1, :Tp], pos, blocks[l], cfg)
            kv[l, 0, Tp:] = k_own
            kv[l, 1, Tp:] = v_own
        x = x + (t[s + 1] - t[s]) * pi0.head(h[1:], W, cfg["eps"])
    return x


def test_two_streams_stale_cache():
    """The two-stream scheme of the reading note: the prefix model fills the next
    cache on one stream while the action expert denoises from the previous cache
    on another.  The actions match the oracle on the cache they read, and the
    new cache matches a prefill run alone (the prefill path is deterministic)."""
    from latency_transformer_block_gb300.models import Pi0Prefix
    ca = synth.config("tiny", Hq=2, Hkv=1, dh=256, L=2)
    cp = synth.config("prefill", D=256, Hq=2, Hkv=1, dh=256, F=512, L=2, T_prefix=ca["T_prefix"],
                      T_q=ca["T_q"], patch_dim=64)
    wa = synth.pi0_weights(ca, 4)
    pre = Pi0Prefix(cp, synth.prefill_weights(cp, 4), max_batch=1)
    ae = Pi0ActionExpert(ca, wa)
    pe0 = _dev_pe(synth.prefill_inputs(cp, 1, 5)["patch_emb"])
    pe1 = _dev_pe(synth.prefill_inputs(cp, 1, 6)["patch_emb"])
    kv0, kv1, kv1_alone = pre.new_kv(1), pre.new_kv(1), pre.new_kv(1)
    pre.prefill(pe0, kv0)
    pre.prefill(pe1, kv1_alone)
    torch.cuda.synchronize()
    ib = synth.pi0_inputs(ca, 4)
    kv0_bits = bits_of(kv0)[:, 0]
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    state = torch.from_numpy(ib["state"]).cuda()
    x = torch.from_numpy(ib["noise"]).cuda()
    pre.prefill(pe1, kv1, sa)                       # next observation, stream A
    ae.denoise(kv0[:, 0], state, x, sb)             # actions from the previous cache, stream B
    torch.cuda.synchronize()
    ae.ctx.sync()
    pre.ctx.sync()
    # the residual GEMMs may split K (fp32 reductions in any order): cache codes
    # within one bf16 ulp of a prefill run alone
    Tp = cp["T_prefix"]
    assert_bf16_close(bits_of(kv1)[:, 0, :, :Tp], bits_of(kv1_alone)[:, 0, :, :Tp], "two-stream new cache")
    ref, _ = pi0.denoise(ib["noise"], ib["state"], kv0_bits, wa, ca)
    assert_rel(x.cpu().numpy(), ref, FINAL_TOL, "two-stream actions")


def _dev_pe(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
