"""lat_chunk_attention_noalloc against the oracle and the context's attention (GPU).

The no-allocation entry point serves callers that cannot call cudaMalloc (an
engine owning all device memory through its own pool, a real-time loop that
forbids allocation): it takes its key-range scratch from a static device array
instead of a context's workspace.  It must give the attention of the oracle
(and the same as the context path) on consecutive calls that share that
array, for every head dimension and head grouping it accepts, including the
shapes where the array holds a single key range (the kernel then writes the
output directly, no merge).  This file is collected last so that a failure
here leaves every other test already run.
"""
import numpy as np
import pytest
import torch

from latency_transformer_block_gb300 import lat, synth
from latency_transformer_block_gb300.models import Pi0ActionExpert, _dev_bf16
from oracle import bf16, ops
from tests.parity import BLOCK_TOL, assert_rel

pytestmark = pytest.mark.gpu


def _inputs(T_q, T_kv, Hq, Hkv, dh, seed):
    a = synth.attention_inputs(T_q, T_kv, Hq, Hkv, dh, seed)
    q = torch.from_numpy(a["q"]).cuda()
    k = _dev_bf16(a["k"], "cuda")
    v = _dev_bf16(a["v"], "cuda")
    ref = ops.attention(a["q"].astype(np.float64).reshape(T_q, Hq, dh),
                        bf16.decode(a["k"]).reshape(T_kv, Hkv, dh),
                        bf16.decode(a["v"]).reshape(T_kv, Hkv, dh), 1.0 / np.sqrt(dh))
    return q, k, v, ref.reshape(T_q, Hq * dh)


# (T_q, T_kv, Hq, Hkv, dh): MQA, MHA (Hkv = Hq) and grouped (1 < Hkv < Hq) heads;
# dh 64 / 128 / 256; T_kv not a multiple of 32; Hq = 32, T_q = 64, dh = 256
# leaves room for one key range only (32 * 64 * 258 > 1048576 / 2)
CASES = [
    (64, 576, 8, 1, 256),
    (40, 301, 4, 4, 64),
    (17, 95, 8, 2, 128),
    (64, 200, 16, 16, 128),
    (33, 1000, 6, 3, 64),
    (64, 129, 32, 1, 256),
]


@pytest.mark.parametrize("T_q,T_kv,Hq,Hkv,dh", CASES, ids=[f"{c[0]}x{c[1]}_h{c[2]}kv{c[3]}_d{c[4]}" for c in CASES])
def test_noalloc_attention_matches_oracle_on_two_calls(T_q, T_kv, Hq, Hkv, dh):
    # two calls in a row, the second with other inputs and fewer keys: it must
    # not see the first call's leftovers in the shared array
    for call, tkv in enumerate([T_kv, max(1, T_kv - 37)]):
        q, k, v, ref = _inputs(T_q, tkv, Hq, Hkv, dh, seed=1000 * call + T_q + tkv + dh)
        got = torch.full((T_q, Hq * dh), float("nan"), device="cuda")
        lat.chunk_attention_noalloc(q, k, v, got, T_q, tkv, Hq, Hkv, dh)
        torch.cuda.synchronize()
        assert_rel(got.cpu().numpy(), ref, BLOCK_TOL, f"noalloc call {call} {T_q}x{tkv} h{Hq}/{Hkv} d{dh}")


def test_noalloc_attention_matches_context_attention_on_two_calls():
    cfg = synth.config("pi0_ae", L=1)
    m = Pi0ActionExpert(cfg, synth.pi0_weights(cfg, 0))
    Hq, Hkv, dh = cfg["Hq"], cfg["Hkv"], cfg["dh"]
    for call, (T_q, T_kv) in enumerate([(64, 576), (40, 300)]):
        q, k, v, _ = _inputs(T_q, T_kv, Hq, Hkv, dh, seed=100 + call)
        ref = torch.full((T_q, Hq * dh), float("nan"), device="cuda")
        got = torch.full((T_q, Hq * dh), float("nan"), device="cuda")
        m.ctx.debug_attention(q, k, v, ref, T_q, T_kv)
        lat.chunk_attention_noalloc(q, k, v, got, T_q, T_kv, Hq, Hkv, dh)
        m.ctx.sync()
        assert_rel(got.cpu().numpy(), ref.cpu().numpy(), BLOCK_TOL, f"noalloc vs context, call {call}")
    # a size beyond the static scratch is refused before any work
    big = torch.zeros(16, device="cuda")
    with pytest.raises(lat.LatError) as e:
        lat.chunk_attention_noalloc(big, big, big, big, 4096, 64, 32, 1, 256)
    assert e.value.code == 2
