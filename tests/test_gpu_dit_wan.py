"""GPU parity of the DiT stage's Wan-class options against the oracle: 3-D
video RoPE (grid_h x grid_w patches per frame), text cross-attention
(lat_dit_set_text) and rings kept in pages of a pool (lat_dit_bind_pages), at
a small size over several ragged tiles and at the 1.3B size on sampled rows.
All calls go through the C ABI.
"""
import numpy as np
import pytest
import torch

from latency_transformer_block_gb300 import lat, synth
from latency_transformer_block_gb300.models import DitStage, _dev_bf16, bits_of
from oracle import bf16, dit, ops, pi0
from tests.parity import BLOCK_TOL, FINAL_TOL, assert_bf16_close, assert_rel

pytestmark = pytest.mark.gpu

# two blocks of width 256 (2 heads x 128); a chunk is 2 frames of 5 x 10 patches;
# 64 text tokens; pages of 48 tokens (a chunk of 100 tokens spans page boundaries)
SMALL_WAN = dict(D=256, H=2, dh=128, F=512, L=2, T_chunk=100, t_dim=64, lat_dim=16,
                 grid_h=5, grid_w=10, text_len=64)


def _band_pair_order(dh):
    """For each dim k of a head in the ring's order (3-D RoPE: the bands' first
    halves, then their second halves), the model's dim (band offset + i, or
    + i + width / 2)."""
    bands = ops.rope_bands(dh)
    pairs = []
    for o, w in bands:
        pairs += [(o, w, i) for i in range(w // 2)]
    return np.array([o + i for o, w, i in pairs] + [o + i + w // 2 for o, w, i in pairs])


def _k_to_model_order(k_bits, cfg):
    """Ring K rows [.., D] from the ring's band-pair order back to the model's."""
    dh, H = cfg["dh"], cfg["H"]
    perm = _band_pair_order(dh)
    out = np.empty_like(k_bits)
    for h in range(H):
        out[..., h * dh + perm] = k_bits[..., h * dh:(h + 1) * dh]
    return out


def _k_to_ring_order(k_bits, cfg):
    """The inverse of ``_k_to_model_order``."""
    dh, H = cfg["dh"], cfg["H"]
    perm = _band_pair_order(dh)
    out = np.empty_like(k_bits)
    for h in range(H):
        out[..., h * dh:(h + 1) * dh] = k_bits[..., h * dh + perm]
    return out


def _device_ring(ring_bits, cfg):
    """The rings as the library holds them: with 3-D RoPE, K in band-pair order."""
    r = ring_bits.copy()
    if cfg.get("grid_h", 0):
        r[..., 0, :, :] = _k_to_ring_order(r[..., 0, :, :], cfg)
    return r


def _wan_case(cfg, descs, seed=0, streams=1, layer=0, rows=None, paged=False):
    """One block through lat_block_forward; returns (got_x, ref_x, got_ring, ref_ring,
    ring_in), rings as bf16 codes [streams, S, slots, 2, T, D] of the block, K
    in the model's dim order."""
    wb = synth.dit_weights(cfg, seed)
    n = len(descs)
    m = DitStage(cfg, wb, max_batch=max(n, 1), n_streams=streams)
    text_bits = synth.dit_text(cfg, streams, seed) if cfg.get("text_len", 0) else None
    if text_bits is not None:
        for st in range(streams):
            m.set_text(st, text_bits[st])
    ring_bits = synth.dit_ring(cfg, seed, streams=streams, layers=cfg["L"])
    xs = synth.dit_latents(cfg, n, seed)
    x = torch.from_numpy(xs).cuda()
    if paged:
        table, n_pool = synth.dit_page_table(cfg, streams, cfg["L"], seed)
        pool = _dev_bf16(dit.ring_to_pool(_device_ring(ring_bits, cfg), table, cfg, n_pool), "cuda")
        m.bind_pages(table)
        m.block(layer, x, descs, pool)
        m.ctx.sync()
        got_ring = dit.pool_to_ring(bits_of(pool), table, cfg, streams, cfg["L"])
    else:
        ring = _dev_bf16(_device_ring(ring_bits, cfg), "cuda")
        m.block(layer, x, descs, ring)
        m.ctx.sync()
        got_ring = bits_of(ring)
    got_x = x.cpu().numpy()
    got_ring = got_ring[:, layer].copy()
    if cfg.get("grid_h", 0):
        got_ring[..., 0, :, :] = _k_to_model_order(got_ring[..., 0, :, :], cfg)
    W = pi0.decode_tree({k: v for k, v in wb.items() if k != "blocks"})
    table_a = dit.adaln_table(W, cfg)
    w = pi0.decode_tree(wb["blocks"][layer])
    r = bf16.decode(ring_bits[:, layer])
    text = bf16.decode(text_bits) if text_bits is not None else None
    if rows is None:
        ref_x = dit.block_batch(xs, descs, r, table_a, w, cfg, text)
    else:
        ref_x = dit.block_batch_rows(xs, descs, r, table_a, w, cfg, rows, text)
        got_x = got_x[:, rows]
    return got_x, ref_x, got_ring, bf16.encode(r), ring_bits[:, layer]


def _check_ring(cfg, descs, streams, got_ring, ref_ring, ring_in, what):
    nh = cfg["n_hist"]
    touched = {(st, s, c % (nh + 1)) for (st, c, s) in descs}
    for (st, c, s) in descs:
        sl = c % (nh + 1)
        assert_bf16_close(got_ring[st, s, sl], ref_ring[st, s, sl], f"{what} own KV chunk {c}")
    for st in range(streams):
        for s in range(cfg["S"]):
            for sl in range(nh + 1):
                if (st, s, sl) not in touched:
                    assert np.array_equal(got_ring[st, s, sl], ring_in[st, s, sl])


@pytest.mark.parametrize("descs,streams,layer,paged", [
    ([(0, 7, 0), (0, 6, 1), (0, 5, 2), (0, 4, 3)], 1, 1, False),     # steady state, 4 chunks at steps 0..3
    ([(0, 0, 0), (1, 2, 0), (1, 9, 3)], 2, 0, False),                 # no history, two streams (two texts)
    ([(0, 7, 0), (0, 6, 1), (0, 5, 2), (0, 4, 3)], 1, 1, True),      # the same through pages of 48 tokens
    ([(0, 0, 0), (1, 2, 0), (1, 9, 3)], 2, 0, True),
])
def test_dit_wan_small_parity(descs, streams, layer, paged):
    cfg = synth.config("dit_1p3b", **SMALL_WAN, page_tokens=48 if paged else 0)
    got_x, ref_x, got_ring, ref_ring, ring_in = _wan_case(cfg, descs, streams=streams, layer=layer, paged=paged)
    assert_rel(got_x, ref_x, BLOCK_TOL, "dit (3-D RoPE, text cross-attention) block residual")
    _check_ring(cfg, descs, streams, got_ring, ref_ring, ring_in, "dit wan")


@pytest.mark.parametrize("wan", [False, True], ids=["plain", "3d_rope_text"])
def test_dit_pages_equal_contiguous_ring(wan):
    """Pages change addresses only: the same chunks through a page pool (pages of
    48 tokens, a seeded permutation of pool pages) give bit-identical outputs,
    and the pool read back through the table is the contiguous ring."""
    base = dict(SMALL_WAN) if wan else dict(D=256, H=2, dh=128, F=512, L=2, T_chunk=100, t_dim=64)
    descs = [(0, 7, 0), (0, 6, 1), (1, 5, 2), (0, 4, 3)]
    out = {}
    for paged in (False, True):
        cfg = synth.config("dit_1p3b", **base, page_tokens=48 if paged else 0)
        out[paged] = _wan_case(cfg, descs, streams=2, layer=1, paged=paged)
    assert np.array_equal(out[False][0], out[True][0]), "paged block output differs from the contiguous ring's"
    assert np.array_equal(out[False][2], out[True][2]), "paged ring contents differ from the contiguous ring's"


@pytest.mark.parametrize("grid,paged", [(None, False), (None, True), ((2, 5), True)],
                         ids=["1d", "1d_pages8", "3d_pages8"])
def test_dit_short_chunks_parity(grid, paged):
    """Chunks of 20 tokens: a 32-row group of the QKV epilogue spans two or three
    chunks (the per-row rotation table's fallback for a third chunk, the chunk walk
    of the cache stores), and pages of 8 tokens put several page boundaries inside
    one warp's rows; 3-D RoPE over two 2 x 5 frames per chunk."""
    base = dict(D=256, H=2, dh=128, F=512, L=2, T_chunk=20, t_dim=64)
    if grid:
        base.update(grid_h=grid[0], grid_w=grid[1], text_len=16, lat_dim=16)
    cfg = synth.config("dit_1p3b", **base, page_tokens=8 if paged else 0)
    descs = [(0, 7, 0), (0, 6, 1), (0, 5, 2), (0, 4, 3), (1, 2, 0)]   # 100 rows, 5 chunks
    got_x, ref_x, got_ring, ref_ring, ring_in = _wan_case(cfg, descs, streams=2, layer=1, paged=paged)
    assert_rel(got_x, ref_x, BLOCK_TOL, "dit short chunks block residual")
    _check_ring(cfg, descs, 2, got_ring, ref_ring, ring_in, "dit short chunks")


def test_dit_wan_1p3b_sampled_rows():
    """The 1.3B block with one 30 x 52 frame per chunk, 512 text tokens and
    pages of 256 tokens: the steady-state batch of four chunks on sampled rows
    (first, middle and the ragged last query tile)."""
    cfg = synth.config("dit_1p3b", L=1, grid_h=30, grid_w=52, text_len=512, page_tokens=256)
    descs = synth.dit_chunk_descs(cfg, 4)
    rows = np.r_[0:8, 700:708, 1530:1560]
    got_x, ref_x, got_ring, ref_ring, ring_in = _wan_case(cfg, descs, rows=rows, paged=True)
    assert_rel(got_x, ref_x, BLOCK_TOL, "dit 1.3B (3-D RoPE, text, pages) block residual (sampled rows)")
    for (st, c, s) in descs:
        sl = c % 5
        assert_bf16_close(got_ring[st, s, sl], ref_ring[st, s, sl], f"dit 1.3B wan own KV chunk {c}")


def test_dit_wan_interval_parity():
    """lat_dit_interval with every option on: latent in, both blocks, latent out,
    Euler update, against the oracle's stage interval."""
    cfg = synth.config("dit_1p3b", **SMALL_WAN, page_tokens=48)
    wb = synth.dit_weights(cfg, 1)
    m = DitStage(cfg, wb, max_batch=4, n_streams=1)
    text_bits = synth.dit_text(cfg, 1, 1)
    m.set_text(0, text_bits[0])
    descs = synth.dit_chunk_descs(cfg, 4)
    ring_bits = synth.dit_ring(cfg, 1, streams=1, layers=cfg["L"])
    table, n_pool = synth.dit_page_table(cfg, 1, cfg["L"], 1)
    pool = _dev_bf16(dit.ring_to_pool(_device_ring(ring_bits, cfg), table, cfg, n_pool), "cuda")
    m.bind_pages(table)
    z0 = synth.dit_noise(cfg, 4, 1)
    z = torch.from_numpy(z0).cuda()
    m.interval(pool, z, descs)
    m.ctx.sync()
    W = pi0.decode_tree({k: v for k, v in wb.items() if k != "blocks"})
    W["blocks"] = [pi0.decode_tree(b) for b in wb["blocks"]]
    ref = dit.stage_interval(list(z0), descs, bf16.decode(ring_bits), dit.adaln_table(W, cfg), W, cfg,
                             bf16.decode(text_bits))
    assert_rel(z.cpu().numpy(), np.stack(ref), FINAL_TOL, "dit wan interval latents")


def test_dit_wan_state_errors():
    """A stream without a text context, or pages without a table: LAT_ERR_STATE
    before anything is enqueued; the options on a context without them:
    LAT_ERR_STATE; a bad stream index: LAT_ERR_ARG."""
    cfg = synth.config("dit_1p3b", **SMALL_WAN, page_tokens=48)
    wb = synth.dit_weights(cfg, 0)
    m = DitStage(cfg, wb, max_batch=1, n_streams=2)
    x = torch.zeros(1, cfg["T_chunk"], cfg["D"], device="cuda")
    pool = torch.zeros(64, 2, 48, cfg["D"], dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lat.LatError) as e:
        m.block(0, x, [(0, 1, 0)], pool)
    assert e.value.code == 7                           # LAT_ERR_STATE: no text context
    text = synth.dit_text(cfg, 2, 0)
    m.set_text(0, text[0])
    with pytest.raises(lat.LatError) as e:
        m.block(0, x, [(0, 1, 0)], pool)
    assert e.value.code == 7                           # no page table bound
    with pytest.raises(lat.LatError) as e:
        m.set_text(2, text[0])
    assert e.value.code == 1                           # LAT_ERR_ARG
    plain = DitStage(synth.config("dit_1p3b", D=256, H=2, dh=128, F=512, L=1, T_chunk=100, t_dim=64),
                     synth.dit_weights(synth.config("dit_1p3b", D=256, H=2, dh=128, F=512, L=1, T_chunk=100,
                                                    t_dim=64), 0), max_batch=1)
    with pytest.raises(lat.LatError) as e:
        plain.set_text(0, text[0])
    assert e.value.code == 7
