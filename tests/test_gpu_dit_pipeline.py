"""GPU parity of the interleaved stage schedule of chunked AR diffusion.

lat_dit_interval (latent in-projection, every block of the stage at each
chunk's own denoise step, out-projection, Euler update) and the scheduler
lat_dit_pipeline_push are compared with the oracle's ``stage_interval`` and
``pipeline`` on the same seeded inputs.  All calls go through the C ABI.
"""
import numpy as np
import pytest
import torch

from latency_transformer_block_gb300 import lat, synth
from latency_transformer_block_gb300.models import DitStage, bits_of
from oracle import bf16, dit, pi0
from tests.parity import FINAL_TOL, assert_rel

pytestmark = pytest.mark.gpu

# two blocks of width 256 (2 heads x 128), ragged chunk of 100 tokens, 16 latent channels
PIPE_DIT = dict(D=256, H=2, dh=128, F=512, L=2, T_chunk=100, t_dim=64, lat_dim=16)


def _oracle_weights(wb):
    W = pi0.decode_tree({k: v for k, v in wb.items() if k != "blocks"})
    W["blocks"] = [pi0.decode_tree(b) for b in wb["blocks"]]
    return W


def _dev_ring(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)


def test_dit_interval_parity():
    """A steady-state batch (chunks 7..4 at steps 0..3) over a seeded history."""
    cfg = synth.config("dit_1p3b", **PIPE_DIT)
    wb = synth.dit_weights(cfg, 1)
    m = DitStage(cfg, wb, max_batch=4, n_streams=1)
    descs = synth.dit_chunk_descs(cfg, 4)
    ring_bits = synth.dit_ring(cfg, 1, streams=1, layers=cfg["L"])
    z0 = synth.dit_noise(cfg, 4, 1)
    z = torch.from_numpy(z0).cuda()
    ring = _dev_ring(ring_bits)
    m.interval(ring, z, descs)
    m.ctx.sync()
    W = _oracle_weights(wb)
    table = dit.adaln_table(W, cfg)
    rings = bf16.decode(ring_bits)
    ref = dit.stage_interval(list(z0), descs, rings, table, W, cfg)
    assert_rel(z.cpu().numpy(), np.stack(ref), FINAL_TOL, "dit interval latents")
    # every block's ring got the chunks' own K/V (bf16 codes within one ulp)
    got = bf16.decode(bits_of(ring))
    for (st, c, s) in descs:
        sl = c % (cfg["n_hist"] + 1)
        assert_rel(got[st, :, s, sl], rings[st, :, s, sl], FINAL_TOL, f"dit interval own KV chunk {c}")


def test_dit_pipeline_parity():
    """Six chunks through the scheduler (three draining pushes) against the
    oracle's interleaved schedule, which equals the plain sequential order."""
    cfg = synth.config("dit_1p3b", **PIPE_DIT)
    wb = synth.dit_weights(cfg, 2)
    m = DitStage(cfg, wb, max_batch=4, n_streams=2)
    S, n = cfg["S"], 6
    noises = synth.dit_noise(cfg, n, 2)
    rings0 = np.zeros((2, cfg["L"], S, cfg["n_hist"] + 1, 2, cfg["T_chunk"], cfg["D"]), np.float64)
    ring = torch.zeros(rings0.shape, dtype=torch.bfloat16, device="cuda")
    done = torch.zeros(cfg["T_chunk"], cfg["lat_dim"], device="cuda")
    got, order = {}, []
    for i in range(n + S - 1):
        noise = torch.from_numpy(noises[i]).cuda() if i < n else None
        c = m.push(ring, 1, noise, done)   # stream 1 of 2
        order.append(c)
        if c >= 0:
            got[c] = done.cpu().numpy()
    m.ctx.sync()
    assert order == [-1] * (S - 1) + list(range(n))
    W = _oracle_weights(wb)
    table = dit.adaln_table(W, cfg)
    ref = dit.pipeline(list(noises), rings0[1:2], table, W, cfg)
    for c in range(n):
        assert_rel(got[c], ref[c], FINAL_TOL, f"dit pipeline chunk {c}")
    # stream 0 was never touched
    assert not bits_of(ring)[0].any()
    # after a reset the stream starts again at chunk 0
    m.ctx.dit_pipeline_reset(1)
    assert m.push(ring, 1, torch.from_numpy(noises[0]).cuda(), done) == -1


def test_dit_pipeline_constant_velocity_field_is_exact():
    """W_out = 0, b_out = c: every step adds dt c, so a chunk leaves as noise + c
    (S = 4, dt = 1/4: exact up to fp32 rounding of four additions)."""
    cfg = synth.config("dit_1p3b", **PIPE_DIT)
    wb = dict(synth.dit_weights(cfg, 3))
    wb["w_out"] = np.zeros_like(wb["w_out"])
    c = np.linspace(-1, 1, cfg["lat_dim"])
    wb["b_out"] = bf16.encode(c)
    cq = bf16.decode(wb["b_out"])
    m = DitStage(cfg, wb, max_batch=4, n_streams=1)
    noises = synth.dit_noise(cfg, 2, 3)
    ring = torch.zeros((1, cfg["L"], cfg["S"], cfg["n_hist"] + 1, 2, cfg["T_chunk"], cfg["D"]),
                       dtype=torch.bfloat16, device="cuda")
    done = torch.zeros(cfg["T_chunk"], cfg["lat_dim"], device="cuda")
    outs = {}
    for i in range(2 + cfg["S"] - 1):
        k = m.push(ring, 0, torch.from_numpy(noises[i]).cuda() if i < 2 else None, done)
        if k >= 0:
            outs[k] = done.cpu().numpy().astype(np.float64)
    for k in range(2):
        np.testing.assert_allclose(outs[k], noises[k].astype(np.float64) + cq, rtol=0, atol=4e-6)


def test_dit_pipeline_errors():
    cfg = synth.config("dit_1p3b", **PIPE_DIT)
    wb = synth.dit_weights(cfg, 0)
    m = DitStage(cfg, wb, max_batch=4, n_streams=1)
    ring = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lat.LatError) as e:
        m.push(ring, 1)                      # stream out of range
    assert e.value.code == 1
    small = DitStage(cfg, wb, max_batch=2, n_streams=1)
    with pytest.raises(lat.LatError) as e:
        small.push(ring, 0)                  # S = 4 chunks in flight need max_batch >= 4
    assert e.value.code == 2
    no_io = DitStage(dict(cfg, lat_dim=0), wb, max_batch=4, n_streams=1)
    with pytest.raises(lat.LatError) as e:
        no_io.push(ring, 0)
    assert e.value.code == 7
    z = torch.zeros(4, cfg["T_chunk"], cfg["lat_dim"], device="cuda")
    with pytest.raises(lat.LatError) as e:
        m.interval(ring, z, [(0, 5, 0), (0, 10, 0)])   # same stream, step and slot
    assert e.value.code == 1
