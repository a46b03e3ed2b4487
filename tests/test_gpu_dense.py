"""GPU parity of the dense path (prefix prefill and DiT stage) against the oracle."""
import numpy as np
import pytest
import torch

from latency_transformer_block_gb300 import lat, synth
from latency_transformer_block_gb300.models import DitStage, Pi0Prefix, _dev_bf16, bits_of
from oracle import bf16, dit, pi0
from tests.parity import BLOCK_TOL, FINAL_TOL, assert_bf16_close, assert_rel

pytestmark = pytest.mark.gpu


# ----------------------------------------------------------------------------
# prefix prefill
# ----------------------------------------------------------------------------
def _prefill(cfg, B, seed=0, max_batch=None, model=None):
    wb = synth.prefill_weights(cfg, seed)
    pe = synth.prefill_inputs(cfg, B, seed)["patch_emb"]
    m = model or Pi0Prefix(cfg, wb, max_batch=max_batch or B)
    kv = m.new_kv(B)
    m.prefill(_dev_bf16(pe, "cuda"), kv)
    m.ctx.sync()
    return wb, pe, bits_of(kv), m


SMALL_PREFIX = dict(D=512, Hq=2, Hkv=1, dh=256, F=1024, L=3, T_prefix=100, T_q=8, patch_dim=192)


def test_prefill_small_parity():
    cfg = synth.config("prefill", **SMALL_PREFIX)
    wb, pe, got, _ = _prefill(cfg, 2)
    ref = pi0.prefill(pe, wb, cfg)
    Tp = cfg["T_prefix"]
    # layer 0: one block from exact inputs -> cache values within one bf16 ulp
    assert_bf16_close(got[0, :, :, :Tp], ref[0, :, :, :Tp], "prefill layer 0 KV")
    assert_rel(bf16.decode(got[:, :, :, :Tp]), bf16.decode(ref[:, :, :, :Tp]), FINAL_TOL, "prefill KV all layers")
    assert not np.any(got[:, :, :, Tp:]), "own-token slots must stay untouched"


def test_prefill_full_b8_every_element_and_batch_independence():
    """Full size, B = 8: every element's layer-0 K/V against the oracle (one
    block from exact inputs: cache codes within one ulp), the whole 18-layer
    cache of elements 0 and 5 against the oracle (final tolerance), and element
    3 of the batch against a B = 1 run of the same input (GPU against GPU)."""
    cfg = synth.config("prefill")
    wb = synth.prefill_weights(cfg, 0)
    m = Pi0Prefix(cfg, wb, max_batch=8)
    pe8 = synth.prefill_inputs(cfg, 8, 0)["patch_emb"]
    kv8 = m.new_kv(8)
    m.prefill(_dev_bf16(pe8, "cuda"), kv8)
    kv1 = m.new_kv(1)
    m.prefill(_dev_bf16(pe8[3:4], "cuda"), kv1)
    m.ctx.sync()
    got8, got1 = bits_of(kv8), bits_of(kv1)
    Tp = cfg["T_prefix"]
    # layer 0 of every element: a one-layer prefill is the patch projection and
    # the first block's K/V only
    cfg1 = dict(cfg, L=1)
    wb1 = dict(wb, blocks=wb["blocks"][:1])
    blocks1 = [pi0.method_block(pi0.decode_tree(wb["blocks"][0]))]
    for b in range(8):
        ref0 = pi0.prefill(pe8[b:b + 1], wb1, cfg1, blocks=blocks1)
        assert_bf16_close(got8[0, b:b + 1, :, :Tp], ref0[0, :, :, :Tp], f"prefill B=8 element {b} layer 0 KV")
    blocks = [pi0.method_block(pi0.decode_tree(bl)) for bl in wb["blocks"]]
    for b in (0, 5):
        ref = pi0.prefill(pe8[b:b + 1], wb, cfg, blocks=blocks)
        assert_rel(bf16.decode(got8[:, b:b + 1, :, :Tp]), bf16.decode(ref[:, :, :, :Tp]), FINAL_TOL,
                   f"prefill B=8 element {b} KV, all 18 layers")
    assert not np.any(got8[:, :, :, Tp:]), "own-token slots must stay untouched"
    # batch elements are independent: with one element the residual GEMMs split
    # K (fp32 partial sums added in another order), so codes agree to rounding
    assert_bf16_close(got8[:, 3:4, :, :Tp], got1[:, :, :, :Tp], "prefill batch independence", max_ulp=2)


# ----------------------------------------------------------------------------
# DiT stage
# ----------------------------------------------------------------------------
def _dit_case(cfg, descs, seed=0, streams=1, layer=0, rows=None):
    wb = synth.dit_weights(cfg, seed)
    n = len(descs)
    m = DitStage(cfg, wb, max_batch=n, n_streams=streams)
    ring_bits = synth.dit_ring(cfg, seed, streams=streams, layers=cfg["L"])
    xs = synth.dit_latents(cfg, n, seed)
    x = torch.from_numpy(xs).cuda()
    ring = _dev_bf16(ring_bits, "cuda")
    m.block(layer, x, descs, ring)
    m.ctx.sync()
    got_x, got_ring = x.cpu().numpy(), bits_of(ring)
    W = pi0.decode_tree({k: v for k, v in wb.items() if k != "blocks"})
    table = dit.adaln_table(W, cfg)
    w = pi0.decode_tree(wb["blocks"][layer])
    r = bf16.decode(ring_bits[:, layer])
    if rows is None:
        ref_x = dit.block_batch(xs, descs, r, table, w, cfg)
    else:
        ref_x = dit.block_batch_rows(xs, descs, r, table, w, cfg, rows)
        got_x = got_x[:, rows]
    return got_x, ref_x, got_ring[:, layer], bf16.encode(r), ring_bits[:, layer]


SMALL_DIT = dict(D=256, H=2, dh=128, F=512, L=2, T_chunk=100, t_dim=64)


@pytest.mark.parametrize("descs,streams,layer", [
    ([(0, 7, 0), (0, 6, 1), (0, 5, 2), (0, 4, 3)], 1, 1),     # steady state, 4 chunks at steps 0..3
    ([(0, 0, 0), (1, 2, 0), (1, 9, 3)], 2, 0),                 # first chunk (no history), two streams
    ([(0, 3, 2)], 1, 0),                                       # single chunk, partial history
])
def test_dit_small_parity(descs, streams, layer):
    cfg = synth.config("dit_1p3b", **SMALL_DIT)
    got_x, ref_x, got_ring, ref_ring, ring_in = _dit_case(cfg, descs, streams=streams, layer=layer)
    assert_rel(got_x, ref_x, BLOCK_TOL, "dit small block residual")
    nh = cfg["n_hist"]
    for (st, c, s) in descs:
        slot = c % (nh + 1)
        assert_bf16_close(got_ring[st, s, slot], ref_ring[st, s, slot], f"dit own KV chunk {c}")
    # every other slot is untouched
    touched = {(st, s, c % (nh + 1)) for (st, c, s) in descs}
    for st in range(streams):
        for s in range(cfg["S"]):
            for sl in range(nh + 1):
                if (st, s, sl) not in touched:
                    assert np.array_equal(got_ring[st, s, sl], ring_in[st, s, sl])


def test_dit_1p3b_full_block_sampled_rows():
    cfg = synth.config("dit_1p3b", L=1)
    descs = synth.dit_chunk_descs(cfg, 4)
    rows = np.r_[0:8, 700:708, 1530:1560]          # includes the ragged last tile
    got_x, ref_x, got_ring, ref_ring, _ = _dit_case(cfg, descs, rows=rows)
    assert_rel(got_x, ref_x, BLOCK_TOL, "dit 1.3B block residual (sampled rows)")
    for (st, c, s) in descs:
        sl = c % 5
        assert_bf16_close(got_ring[st, s, sl], ref_ring[st, s, sl], f"dit 1.3B own KV chunk {c}")


def test_dit_1p3b_mixed_history_sampled_rows():
    # three chunks with 0, 2 and 4 history chunks (25, 51 and 77 key blocks):
    # 468 attention tiles, so the 12 tiles past the third wave (query tiles
    # 1..12 of the last head of the chunk with 4 history chunks) are cut into
    # 12 key ranges each, a count bounded by the chunk with only its own keys;
    # the sampled rows 1400.. and 1540.. lie in split tiles
    cfg = synth.config("dit_1p3b", L=1)
    descs = [(0, 0, 0), (0, 2, 1), (0, 9, 2)]
    rows = np.r_[0:4, 1400:1404, 1540:1560]        # the last query tiles are the split ones
    got_x, ref_x, got_ring, ref_ring, _ = _dit_case(cfg, descs, rows=rows)
    assert_rel(got_x, ref_x, BLOCK_TOL, "dit 1.3B mixed-history block residual (sampled rows)")
    for (st, c, s) in descs:
        sl = c % 5
        assert_bf16_close(got_ring[st, s, sl], ref_ring[st, s, sl], f"dit 1.3B own KV chunk {c}")


def test_dit_14b_block_batch8_sampled_rows():
    cfg = synth.config("dit_14b")
    descs = synth.dit_chunk_descs(cfg, 8)
    rows = np.r_[0:4, 777:781, 1556:1560]
    got_x, ref_x, got_ring, ref_ring, _ = _dit_case(cfg, descs, streams=2, rows=rows)
    assert_rel(got_x, ref_x, BLOCK_TOL, "dit 14B block residual (sampled rows)")
    for (st, c, s) in descs:
        sl = c % 5
        assert_bf16_close(got_ring[st, s, sl], ref_ring[st, s, sl], f"dit 14B own KV chunk {c}")


@pytest.mark.parametrize("n", [1, 4])
def test_dit_14b_block_sampled_rows(n):
    """14B block with one chunk (its last wave's tail tiles split into key
    ranges) and with four chunks at steps 0..3 (104 tail tiles, run whole)."""
    cfg = synth.config("dit_14b")
    descs = synth.dit_chunk_descs(cfg, n)
    rows = np.r_[0:4, 640:644, 1400:1404, 1536:1560]   # the last query tiles: split / ragged
    got_x, ref_x, got_ring, ref_ring, _ = _dit_case(cfg, descs, streams=1, rows=rows)
    assert_rel(got_x, ref_x, BLOCK_TOL, f"dit 14B block n={n} residual (sampled rows)")
    for (st, c, s) in descs:
        sl = c % 5
        assert_bf16_close(got_ring[st, s, sl], ref_ring[st, s, sl], f"dit 14B n={n} own KV chunk {c}")


def test_dit_1p3b_whole_stage_interval():
    """The full 1.3B stage: latent in-projection, all 30 blocks at each chunk's
    own step, out-projection and Euler update for four chunks at steps 0..3
    (chunks 3, 2, 1, 0: the interval that admits chunk 3), against the oracle's
    stage interval at the final tolerance.  History slots the chunks read are
    seeded; the others stay zero on both sides."""
    cfg = synth.config("dit_1p3b")
    wb = synth.dit_weights(cfg, 4)
    m = DitStage(cfg, wb, max_batch=4, n_streams=1)
    descs = synth.dit_chunk_descs(cfg, 4, first_chunk=3)
    S, nh, L = cfg["S"], cfg["n_hist"], cfg["L"]
    shape = (1, L, S, nh + 1, 2, cfg["T_chunk"], cfg["D"])
    ring_bits = np.zeros(shape, np.uint16)
    for (st, c, s) in descs:
        for cc in dit.history_chunks(c, nh):
            ring_bits[st, :, s, cc % (nh + 1)] = synth.normal_bf16(4, f"ring.{s}.{cc}", (L, 2, cfg["T_chunk"], cfg["D"]))
    z0 = synth.dit_noise(cfg, 4, 4)
    z = torch.from_numpy(z0).cuda()
    ring = torch.from_numpy(ring_bits.view(np.int16)).cuda().view(torch.bfloat16)
    m.interval(ring, z, descs)
    m.ctx.sync()
    got = z.cpu().numpy()
    del ring
    W = pi0.decode_tree({k: v for k, v in wb.items() if k != "blocks"})
    W["blocks"] = [pi0.decode_tree(b) for b in wb["blocks"]]
    table = dit.adaln_table(W, cfg)
    # bf16 values are exact in float32; the oracle widens them to float64 as it reads
    rings = synth.to_f32(ring_bits)
    ref = dit.stage_interval(list(z0), descs, rings, table, W, cfg)
    assert_rel(got, np.stack(ref), FINAL_TOL, "dit 1.3B whole-stage interval latents")


def test_dit_indices_and_errors():
    cfg = synth.config("dit_1p3b", **SMALL_DIT)
    wb = synth.dit_weights(cfg, 0)
    m = DitStage(cfg, wb, max_batch=4, n_streams=2)
    chunks = [(0, c, 0) for c in range(13)] + [(1, 123456, 2)]
    slots, pos = m.ctx.debug_indices(chunks=chunks)
    assert slots == [dit.ring_slot(c, cfg["n_hist"]) for (_, c, _) in chunks]
    assert pos == [int(dit.positions(c, cfg["T_chunk"])[0]) for (_, c, _) in chunks]
    ring = torch.zeros(1, device="cuda", dtype=torch.bfloat16)
    x = torch.zeros(16, device="cuda")
    for bad in ([(0, 5, 0), (0, 10, 0)],       # same stream, step and slot
                [(0, 5, 4)],                    # step out of range
                [(2, 5, 0)],                    # stream out of range
                [(0, -1, 0)],
                [(0, c, 0) for c in range(5)]):  # more than max_batch
        with pytest.raises(lat.LatError) as e:
            m.block(0, x, bad, ring)
        assert e.value.code == 1


# ----------------------------------------------------------------------------
# precision study: one fp16 plane of the activation instead of two
# ----------------------------------------------------------------------------
def _dense_case_output(case, terms):
    """One block of a dense configuration (sampled rows for the DiT) with the
    projections multiplying `terms` fp16 planes of their activation; returns
    (GPU output, oracle output)."""
    if case == "prefill":
        cfg = synth.config("prefill", L=1)
        wb = synth.prefill_weights(cfg, 0)
        pe = synth.prefill_inputs(cfg, 1, 0)["patch_emb"]
        m = Pi0Prefix(cfg, wb, max_batch=1)
        m.ctx.debug_act_terms(terms)
        kv = m.new_kv(1)
        m.prefill(_dev_bf16(pe, "cuda"), kv)
        m.ctx.sync()
        Tp = cfg["T_prefix"]
        return bf16.decode(bits_of(kv)[0, :, :, :Tp]), bf16.decode(pi0.prefill(pe, wb, cfg)[0, :, :, :Tp])
    cfg = synth.config(case, L=1)
    descs = synth.dit_chunk_descs(cfg, 1)
    rows = np.r_[0:8, 700:708, 1540:1560]
    wb = synth.dit_weights(cfg, 0)
    m = DitStage(cfg, wb, max_batch=1, n_streams=1)
    m.ctx.debug_act_terms(terms)
    ring_bits = synth.dit_ring(cfg, 0, streams=1, layers=1)
    xs = synth.dit_latents(cfg, 1, 0)
    x = torch.from_numpy(xs).cuda()
    m.block(0, x, descs, _dev_bf16(ring_bits, "cuda"))
    m.ctx.sync()
    W = pi0.decode_tree({k: v for k, v in wb.items() if k != "blocks"})
    ref = dit.block_batch_rows(xs, descs, bf16.decode(ring_bits[:, 0]), dit.adaln_table(W, cfg),
                               pi0.decode_tree(wb["blocks"][0]), cfg, rows)
    return x.cpu().numpy()[:, rows], ref


@pytest.mark.parametrize("case", ["dit_1p3b", "dit_14b", "prefill"])
def test_one_activation_plane_error_is_measured(case):
    """The dense projections multiply two fp16 planes of their activation (hi +
    lo, 22 bits); one plane (hi, 11 bits) would halve the tensor work.  On the
    block of each dense configuration: two planes meet the block tolerance,
    one plane's error is measured and recorded in the parity report (it is the
    figure the choice of two planes rests on: measured above the tolerance),
    and it is larger than two planes' (the flag takes effect)."""
    from tests.parity import REPORT, max_rel_err
    got2, ref = _dense_case_output(case, 2)
    got1, _ = _dense_case_output(case, 1)
    if case == "prefill":
        # cache codes (bf16): one ulp is up to 7.8e-3 of a value, so the codes
        # are held to one ulp and the error is reported relative to their RMS
        assert_bf16_close(bf16.encode(got2), bf16.encode(ref), "prefill layer 0 KV, two fp16 activation planes")
        rms = np.sqrt(np.mean(ref * ref))
        e2, e1 = (float(np.max(np.abs(g - ref)) / rms) for g in (got2, got1))
        what = "max error / RMS"
    else:
        e2 = assert_rel(got2, ref, BLOCK_TOL, f"{case} block, two fp16 activation planes")
        e1 = max_rel_err(got1, ref)
        what = "max relative error"
    REPORT.append((f"{case} block with ONE fp16 activation plane ({what}; precision study, not a bound)", e1,
                   BLOCK_TOL))
    print(f"{case}: {what} one plane {e1:.3e}, two planes {e2:.3e} (block tolerance {BLOCK_TOL:.0e})")
    assert np.isfinite(e1) and e1 > e2
