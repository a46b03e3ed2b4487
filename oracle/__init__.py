"""CPU oracle for the low-latency transformer-block path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run anything in this package.
The product path (``include/lat.h`` and the CUDA library behind it) never calls
it, and it shares no code with that path: the two meet only in the seeded input
generator ``latency_transformer_block_gb300.synth``, which draws data and holds
none of the method's arithmetic.

What it computes, and where the pages define it:

* ``ops``   -- the elementary operations (RMSNorm, LayerNorm, rotate-half RoPE,
  softmax attention, GELU-tanh, SiLU, sinusoidal timestep embedding), written
  out from their textbook definitions in float64.
* ``fold``  -- the offline graph transforms of "Running VLAs at Real-time Speed"
  (reading note on arXiv 2510.26742), section 4: the RMSNorm scale fold
  (x_hat * g) W = x_hat [diag(g) W] (section 4.1), the action/time-embedding
  fold with a precomputed time table (section 4.2) and the merged QKV
  projection (section 4.3).
* ``pi0``   -- the pi0 action expert (Fig. 4 of that note: 63 action tokens +
  1 state token over a 512-token vision prefix KV, 18 blocks x 10 flow-matching
  steps) and the prefix prefill that produces its KV cache, including the
  skipped attention/FFN of the last prefix layer (section 4.3).
* ``dit``   -- one DiT block stage of chunked autoregressive denoising over
  noisy history KV, with same-block batching of chunks at different denoise
  steps (PhysisServe article, sections on stage pipelining and on one GPU
  running several stages).

Precision.  All arithmetic is float64.  The pages fix the storage precision
(BF16 weights and KV cache) but not the arithmetic; the oracle therefore keeps
bf16 exactly where the method *stores* bf16 -- weights, folded weights that the
method stores as bf16, and K/V written into the cache -- and rounds there with
round-to-nearest-even, and is exact (float64) everywhere else.
"""
