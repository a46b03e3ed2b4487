"""lat_chunk_attention_noalloc against the context's attention (GPU).

The no-allocation entry point serves callers that cannot call cudaMalloc (an
engine owning all device memory through its own pool, a real-time loop that
forbids allocation): it takes its key-range scratch from a static device array
instead of a context's workspace.  It must give the same attention as the
context path, on consecutive calls that share that array.  This file is
collected last so that a failure here leaves every other test already run.
"""
import numpy as np
import pytest
import torch

from latency_transformer_block_gb300 import lat, synth
from latency_transformer_block_gb300.models import Pi0ActionExpert, _dev_bf16
from tests.parity import BLOCK_TOL, assert_rel

pytestmark = pytest.mark.gpu


def test_noalloc_attention_matches_context_attention_on_two_calls():
    cfg = synth.config("pi0_ae", L=1)
    m = Pi0ActionExpert(cfg, synth.pi0_weights(cfg, 0))
    Hq, Hkv, dh = cfg["Hq"], cfg["Hkv"], cfg["dh"]
    # two calls in a row with different shapes: the second must not see the
    # first call's leftovers in the shared scratch
    for call, (T_q, T_kv) in enumerate([(64, 576), (40, 300)]):
        a = synth.attention_inputs(T_q, T_kv, Hq, Hkv, dh, seed=100 + call)
        q = torch.from_numpy(a["q"]).cuda()
        k = _dev_bf16(a["k"], "cuda")
        v = _dev_bf16(a["v"], "cuda")
        ref = torch.full((T_q, Hq * dh), float("nan"), device="cuda")
        got = torch.full((T_q, Hq * dh), float("nan"), device="cuda")
        m.ctx.debug_attention(q, k, v, ref, T_q, T_kv)
        lat.chunk_attention_noalloc(q, k, v, got, T_q, T_kv, Hq, Hkv, dh)
        m.ctx.sync()
        assert_rel(got.cpu().numpy(), ref.cpu().numpy(), BLOCK_TOL, f"noalloc call {call}")
    # a size beyond the static scratch is refused before any work
    big = torch.zeros(16, device="cuda")
    with pytest.raises(lat.LatError) as e:
        lat.chunk_attention_noalloc(big, big, big, big, 4096, 64, 32, 1, 256)
    assert e.value.code == 2
