"""Kernel-level GPU parity: single kernels of the path against the oracle's
matching piece (through the C ABI's measurement hooks)."""
import numpy as np
import pytest
import torch

from latency_transformer_block_gb300 import synth
from latency_transformer_block_gb300.models import Pi0ActionExpert, _dev_bf16
from oracle import bf16, ops
from tests.parity import BLOCK_TOL, assert_rel

pytestmark = pytest.mark.gpu

_CTX = {}


def _ctx(name):
    if name not in _CTX:
        cfg = synth.config(name)
        _CTX[name] = (cfg, Pi0ActionExpert(cfg, synth.pi0_weights(cfg, 0)))
    return _CTX[name]


def run_attention(m, cfg, T_q, T_kv, seed):
    Hq, Hkv, dh = cfg["Hq"], cfg["Hkv"], cfg["dh"]
    a = synth.attention_inputs(T_q, T_kv, Hq, Hkv, dh, seed)
    q = torch.from_numpy(a["q"]).cuda()
    k = _dev_bf16(a["k"], "cuda")
    v = _dev_bf16(a["v"], "cuda")
    out = torch.full((T_q, Hq * dh), float("nan"), device="cuda")
    m.ctx.debug_attention(q, k, v, out, T_q, T_kv)
    m.ctx.sync()
    ref = ops.attention(a["q"].astype(np.float64).reshape(T_q, Hq, dh),
                        bf16.decode(a["k"]).reshape(T_kv, Hkv, dh),
                        bf16.decode(a["v"]).reshape(T_kv, Hkv, dh), 1.0 / np.sqrt(dh))
    return out.cpu().numpy(), ref.reshape(T_q, Hq * dh)


@pytest.mark.parametrize("name,T_q,T_kv", [("tiny", 64, 192), ("pi0_ae", 64, 576), ("pi0_ae", 37, 100),
                                           ("pi0_ae", 5, 1), ("tiny", 1, 129)])
def test_attention_kernel(name, T_q, T_kv):
    cfg, m = _ctx(name)
    got, ref = run_attention(m, cfg, T_q, T_kv, seed=T_q * 1000 + T_kv)
    assert_rel(got, ref, BLOCK_TOL, f"attention {name} {T_q}x{T_kv}")


def test_device_wait_timeout_is_reported_and_cleared():
    """Failure detection without a GPU fault: a bounded wait that nothing
    completes gives up (~0.5 s), lat_sync reports LAT_ERR_TIMEOUT, and after
    lat_clear_error the same context computes correct results again."""
    from latency_transformer_block_gb300 import lat
    cfg = synth.config("tiny")
    m = Pi0ActionExpert(cfg, synth.pi0_weights(cfg, 0))
    m.ctx.debug_timeout()
    with pytest.raises(lat.LatError) as e:
        m.ctx.sync()
    assert e.value.code == 6                       # LAT_ERR_TIMEOUT
    m.ctx.clear_error()
    m.ctx.sync()
    got, ref = run_attention(m, cfg, 64, 192, seed=5)
    assert_rel(got, ref, BLOCK_TOL, "attention after a cleared timeout")


@pytest.mark.parametrize("mode", ["one_step", "whole_chunk"])
@pytest.mark.parametrize("which", [1, 2, 3], ids=["grid_barrier", "qkv_cluster_exchange", "gate_up_cluster_exchange"])
def test_step_kernel_wait_timeout_is_reported_and_cleared(which, mode):
    """Failure detection of the persistent step kernel's own waits, without a
    GPU fault: one wait of the first block expects an arrival that never comes,
    gives up (~0.5 s), every later wait of the launch returns at once, lat_sync
    reports LAT_ERR_TIMEOUT; with the skew off and the error cleared the same
    context denoises a chunk that matches the oracle.  `one_step`: the blocks
    of one denoise step; `whole_chunk`: the launch that runs every step of a
    chunk with its embedding and head."""
    from latency_transformer_block_gb300 import lat
    from oracle import pi0
    from tests.parity import FINAL_TOL
    cfg = synth.config("tiny")
    wb = synth.pi0_weights(cfg, 0)
    m = Pi0ActionExpert(cfg, wb)
    ib = synth.pi0_inputs(cfg, 2)
    kv = m.kv_from_bits(ib["kv"])
    m.ctx.debug_wait_skew(which, 1)
    if mode == "one_step":
        m.ctx.debug_step(kv, 1)
    else:
        x = torch.from_numpy(ib["noise"]).cuda()
        m.denoise(kv, torch.from_numpy(ib["state"]).cuda(), x)
    with pytest.raises(lat.LatError) as e:
        m.ctx.sync()
    assert e.value.code == 6                       # LAT_ERR_TIMEOUT
    m.ctx.debug_wait_skew(0, 0)
    m.ctx.clear_error()
    m.ctx.sync()
    kv = m.kv_from_bits(ib["kv"])
    x = torch.from_numpy(ib["noise"]).cuda()
    m.denoise(kv, torch.from_numpy(ib["state"]).cuda(), x)
    m.ctx.sync()
    ref, _ = pi0.denoise(ib["noise"], ib["state"], ib["kv"], wb, cfg)
    assert_rel(x.cpu().numpy(), ref, FINAL_TOL, "actions after a cleared step-kernel timeout")
