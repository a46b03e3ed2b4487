/*
 * lat.h -- C ABI of the low-latency transformer-block library (GB300, sm_103a).
 *
 * The hot path: a small chunk of query tokens runs through a stack of
 * transformer blocks, attending to a cached prefix / history KV, and the stack
 * is repeated over a fixed number of flow-matching (Euler) denoise steps.  Two
 * model families take this path:
 *
 *  - LAT_PI0_ACTION_EXPERT: the pi0 action expert ("Running VLAs at Real-time
 *    Speed", reading note on arXiv 2510.26742, section 2 and Fig. 4): 63 action
 *    tokens + 1 state token over a per-layer prefix KV of 512 vision tokens,
 *    18 blocks x 10 Euler steps.  RMSNorm with its scale folded into the next
 *    weight (section 4.1), folded action/time embedding with a precomputed time
 *    table (section 4.2), merged QKV with RoPE (section 4.3), gated FFN
 *    (section 5).
 *  - LAT_PI0_PREFIX: the prefix model whose per-layer K/V is that cache; the
 *    last layer stops after K and V (section 4.3).
 *  - LAT_DIT: one DiT block stage of chunked autoregressive denoising
 *    (PhysisServe article, sections on pipelining by "one block at one denoise
 *    step" and on batching chunks of one block): a chunk attends to its own
 *    tokens and to the noisy KV that the previous chunks left at the same
 *    denoise step; LayerNorm + adaLN shift/scale/gate, GELU-tanh FFN.
 *
 * Conventions for every call
 *  - Pointers named "device" are CUDA device pointers owned by the caller; the
 *    library borrows them for the duration of the work it enqueues.  Pointers
 *    named "host" are read before the call returns.
 *  - All device pointers must be 16-byte aligned (LAT_ERR_ALIGN otherwise).
 *  - bf16 = IEEE bfloat16 bit patterns; fp32 = IEEE float.
 *  - Weight matrices passed to lat_create use the math convention y = x W:
 *    bf16 [K_in][N_out], row-major.
 *  - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Work is enqueued asynchronously; argument errors are detected on the host
 *    and returned before anything is enqueued.  A device-side wait that gives
 *    up (bounded spin) records LAT_ERR_TIMEOUT in the context; it is returned
 *    by lat_sync(); lat_clear_error() makes the context usable again.
 *  - No call allocates device memory except lat_create (weights, tables,
 *    workspace) and the first lat_denoise_chunk on a new set of buffer
 *    addresses (graph instantiation).
 *  - A context is not thread-safe: calls on one context must be serialised by
 *    the caller and enqueued on one stream at a time.
 */
#ifndef LAT_H
#define LAT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LAT_OK = 0,
  LAT_ERR_ARG = 1,        /* null pointer, index out of range, bad enum          */
  LAT_ERR_SHAPE = 2,      /* a size the kernels do not support                   */
  LAT_ERR_ALIGN = 3,      /* a device pointer not 16-byte aligned                */
  LAT_ERR_CUDA = 4,       /* a CUDA runtime/driver call failed (see lat_last_error) */
  LAT_ERR_OOM = 5,        /* device allocation failed in lat_create              */
  LAT_ERR_TIMEOUT = 6,    /* a bounded device-side wait gave up                  */
  LAT_ERR_STATE = 7,      /* call not valid for this context kind / state        */
  LAT_ERR_UNSUPPORTED = 8, /* no kernel for this device (needs sm_103)           */
  LAT_ERR_RANGE = 9       /* an activation reached |x| >= 65504 (or was not finite):
                             the fp16 operand planes of the action expert's
                             projections cannot hold it; results meaningless   */
} lat_status;

typedef enum {
  LAT_PI0_ACTION_EXPERT = 0,
  LAT_PI0_PREFIX = 1,
  LAT_DIT = 2
} lat_model_kind;

/* Model shape.  Fields not used by a kind must be 0. */
typedef struct {
  int kind;        /* lat_model_kind                                              */
  int D;           /* residual width                                             */
  int Hq, Hkv, dh; /* query heads, KV heads, head dim (DiT: Hq == Hkv)           */
  int F;           /* FFN width                                                   */
  int L;           /* blocks                                                      */
  int S;           /* denoise steps (action expert, DiT)                          */
  int T_prefix;    /* pi0: prefix tokens in the cache                             */
  int T_q;         /* pi0: query tokens (state + actions); DiT: tokens per chunk  */
  int act_dim;     /* action expert: action/state width; DiT: latent channels of */
                   /* the stage's latent in/out projections (0 = none)            */
  int n_hist;      /* DiT: history chunks visible to a chunk (ring = n_hist+1)    */
  int t_dim;       /* DiT: sinusoidal timestep width of the adaLN MLP             */
  int patch_dim;   /* prefix: patch-embedding width                               */
  int max_batch;   /* prefix: max B; DiT: max chunks per lat_block_forward call   */
  int n_streams;   /* DiT: number of independent rings in the kv buffer           */
  float rope_base; /* RoPE base (10000)                                           */
  float eps;       /* norm epsilon (1e-6)                                         */
  int prefix_lm;   /* action expert: 0 = the chunk's tokens all see each other;   */
                   /* 1 = the pi0 model's block mask: the state token (token 0)   */
                   /* sees the prefix and itself only, the action tokens every key */
  /* DiT, Wan-class options (0 = off; see lat_dit_set_text / lat_dit_bind_pages): */
  int grid_h, grid_w; /* 3-D RoPE: a chunk is T_q / (grid_h grid_w) latent frames  */
                   /* of grid_h x grid_w patches                                  */
  int text_len;    /* text cross-attention over a context of text_len tokens      */
  int page_tokens; /* rings kept in pages of page_tokens tokens of a page pool    */
} lat_model_desc;

/* One block's weights (device, bf16, [K_in][N_out] row-major; vectors [D]). */
typedef struct {
  const void *g_attn;  /* pi0: RMSNorm scale before attention [D]               */
  const void *wq;      /* [D][Hq*dh]                                             */
  const void *wk;      /* [D][Hkv*dh]                                            */
  const void *wv;      /* [D][Hkv*dh]                                            */
  const void *wo;      /* [Hq*dh][D]                                             */
  const void *g_ffn;   /* pi0: RMSNorm scale before the FFN [D]                  */
  const void *wg;      /* pi0: gate projection [D][F]                            */
  const void *wu;      /* pi0: up projection [D][F]                              */
  const void *wd;      /* pi0: down projection [F][D]                            */
  const void *w1;      /* DiT: FFN in [D][F]                                     */
  const void *w2;      /* DiT: FFN out [F][D]                                    */
  /* DiT with text_len > 0: the cross-attention sublayer                         */
  const void *g_cross, *b_cross; /* LayerNorm affine [D], [D]                     */
  const void *cq, *ck, *cv, *co; /* [D][D] each                                    */
} lat_block_weights;

typedef struct {
  const lat_block_weights *blocks; /* host array of L                              */
  /* action expert: action/time embedding, state token and head                  */
  const void *w_in, *b_in;         /* [act_dim][D], [D]                           */
  const void *w1, *b1;             /* [2D][D] (rows 0..D-1: action emb, D..: time emb), [D] */
  const void *w2, *b2;             /* [D][D], [D]                                 */
  const void *w_state, *b_state;   /* [act_dim][D], [D]                           */
  const void *g_final;             /* [D]                                         */
  const void *w_out, *b_out;       /* [D][act_dim], [act_dim]                     */
  /* DiT with act_dim > 0: w_in, b_in and w_out, b_out are the stage's latent in- */
  /* and out-projections (same shapes as above); the other fields above are unused */
  /* prefix: patch projection                                                     */
  const void *w_patch, *b_patch;   /* [patch_dim][D], [D]                         */
  /* DiT: timestep MLP producing the adaLN table                                   */
  const void *wt1, *bt1;           /* [t_dim][D], [D]                             */
  const void *wt2, *bt2;           /* [D][D], [D]                                 */
  const void *wmod, *bmod;         /* [D][6D], [6D]                               */
} lat_weights;

/* One chunk of a DiT batch. */
typedef struct {
  int stream;  /* ring index, 0 <= stream < n_streams                             */
  int chunk;   /* chunk index c >= 0 (RoPE position of token j: c*T_q + j; with   */
               /* grid_h > 0: frame c*T_q/(grid_h grid_w) + j/(grid_h grid_w),   */
               /* row (j/grid_w) mod grid_h, column j mod grid_w)                 */
  int step;    /* denoise step 0 <= step < S                                      */
} lat_chunk_desc;

typedef struct lat_ctx lat_ctx;

/*
 * lat_create -- fold and copy the weights, build the tables, allocate workspace.
 *
 * Offline transforms ("Running VLAs at Real-time Speed", section 4):
 *  - RMSNorm scale fold (4.1): diag(g) W for the QKV and gate/up projections,
 *    stored as bf16 (one rounding of the exact product); the head's
 *    diag(g_final) W_out is stored in fp32.
 *  - Action/time fold (4.2): W' = W_in W1[0:D] (fp32 [act_dim][D]) and the time
 *    table T[s] = temb(t_s) W1[D:2D] + b_in W1[0:D] + b1 (fp32 [S][D]).
 *  - Merged QKV (4.3): one [Wq|Wk|Wv] projection.
 *  - DiT: adaLN table A[s] = SiLU(e(t_s)) Wmod + bmod (fp32 [S][6D]),
 *    e(t) = SiLU(temb_t_dim(t) Wt1 + bt1) Wt2 + bt2.
 * The default schedule is t_s = s/S, dt = 1/S.  The caller's weight buffers are
 * not referenced after lat_create returns.  Synchronous.
 * Errors: LAT_ERR_ARG / LAT_ERR_SHAPE for descriptors the kernels do not cover,
 * LAT_ERR_OOM, LAT_ERR_CUDA, LAT_ERR_UNSUPPORTED (no sm_103 device).
 */
lat_status lat_create(const lat_model_desc *desc, const lat_weights *w, lat_ctx **out);

/*
 * lat_set_schedule -- replace the denoise time grid: t (host, S+1 values,
 * t[0] < t[1] < ... < t[S]).  Step s evaluates the model at t[s] and moves x by
 * (t[s+1] - t[s]) * v.  Rebuilds the time table / adaLN table (section 4.2: a
 * schedule change needs the precomputed table recomputed).  Synchronous.
 */
lat_status lat_set_schedule(lat_ctx *ctx, const float *t, int n);

/*
 * lat_prefill_kv -- LAT_PI0_PREFIX: per-layer K/V of the prefix tokens.
 *  patch_emb: device bf16 [B][T_prefix][patch_dim], 1 <= B <= max_batch.
 *  kv:        device bf16 [L][B][2][T_prefix + T_q][Hkv*dh]; slots
 *             0..T_prefix-1 of plane 0 (K, after RoPE at positions 0..) and
 *             plane 1 (V) are written; slots >= T_prefix are not touched.
 * The last layer computes only its K and V.
 */
lat_status lat_prefill_kv(lat_ctx *ctx, const void *patch_emb, int B, void *kv, void *stream);

/*
 * lat_block_forward -- one block, in place on the residual stream.
 * Defined by: for the pi0 models, the reading note's Fig. 4 (a pre-norm block
 * of the action expert over [prefix KV | own tokens]) with the folds of its
 * section 4; for LAT_DIT, the PhysisServe article's stage, "one transformer
 * block at one denoise step", where a chunk reads the noisy KV that earlier
 * chunks left at the same step and chunks of the same block at different
 * steps are merged into one batch (its sections on the stage cut and on one
 * GPU serving several stages).
 *  LAT_PI0_ACTION_EXPERT / LAT_PI0_PREFIX (chunks = NULL, n = 1):
 *    x:  device fp32 [T_q][D] (action expert) -- query tokens at positions
 *        T_prefix + j;
 *    kv: device bf16 [2][T_prefix + T_q][Hkv*dh] of this layer; own K/V are
 *        written to slots T_prefix.. and attention runs over all slots.
 *  LAT_DIT:
 *    x:  device fp32 [n][T_q][D], one chunk per chunks[i] (host array, n <= max_batch);
 *    kv: device bf16 rings [n_streams][L][S][n_hist+1][2][T_q][D]; chunk c at
 *        step s writes its K/V into slot c mod (n_hist+1) of ring
 *        (stream, layer, s), then attends to that slot and to the slots of
 *        chunks c-1..c-n_hist (those >= 0).  Two chunks of one call may not
 *        share (stream, step, slot): LAT_ERR_ARG.  With grid_h > 0 (3-D RoPE)
 *        each head's K in the ring has its dh dims in band-pair order: the
 *        first halves of the frame, height and width bands, then their second
 *        halves (every score is unchanged: q uses the same order).  With
 *        page_tokens > 0, kv is the page pool (lat_dit_bind_pages).
 */
lat_status lat_block_forward(lat_ctx *ctx, int layer, float *x, const lat_chunk_desc *chunks,
                             int n, void *kv, void *stream);

/*
 * lat_denoise_chunk -- LAT_PI0_ACTION_EXPERT: the full S-step x L-block loop.
 * Defined by: the reading note's section 2 (the expert reuses the prefix KV
 * cache over 10 flow-matching steps of 18 blocks each, 63 action + 1 state
 * token), section 4.2 (the time embedding folded into a per-step table) and
 * section 3 (launch gaps are what the expert's time is lost to); each step
 * ends in the Euler update x <- x + dt * v.  The whole chunk -- state token,
 * then per step the embedding, W2, the L blocks and the head with its Euler
 * update -- is ONE launch of the persistent step kernel (grid barriers between
 * its phases), preceded by a 128-byte clear of its barrier counter.
 *  kv:    device bf16 [L][2][T_prefix + T_q][Hkv*dh] (slots >= T_prefix are
 *         overwritten with the query tokens' K/V at every step);
 *  state: device fp32 [act_dim];
 *  x:     device fp32 [T_q - 1][act_dim]: the initial noise in, the actions out
 *         (written once, after the last step; the steps in between keep the
 *         actions in the context's own buffers).
 * The first call for a given (kv, state, x, stream) captures the clear and the
 * launch in a CUDA graph; later calls replay it.  The context keeps the graphs of up to 4
 * such tuples (e.g. two caches used in turn while the next one is prefilled on
 * another stream); a fifth replaces the least recently used one.
 */
lat_status lat_denoise_chunk(lat_ctx *ctx, void *kv, const float *state, float *x, void *stream);

/*
 * lat_dit_interval -- LAT_DIT with latent I/O (act_dim > 0): one interval of
 * the interleaved stage schedule of chunked autoregressive denoising
 * (PhysisServe article: chunks at different denoise steps share the stage as
 * one batch per block; a chunk reads the noisy KV that earlier chunks left at
 * the same step).  Every chunk b of the batch, at its own step s_b, runs
 *   x = z W_in + b_in,  the L blocks (lat_block_forward's math, all chunks
 *   batched per block),  v = x W_out + b_out,  z <- z + dt[s_b] v
 * with dt[s] = t_{s+1} - t_s of the context's schedule.
 *  lat:    device fp32 [n][T_q][act_dim], the chunks' latents z, updated in place;
 *  chunks: host [n], 1 <= n <= max_batch, the same rules as lat_block_forward
 *          (no two chunks share (stream, step, ring slot): LAT_ERR_ARG);
 *  kv:     the rings, as for lat_block_forward (every block's ring is written).
 * Errors: LAT_ERR_STATE without latent I/O weights; LAT_ERR_ARG / LAT_ERR_ALIGN
 * for bad arguments, detected before anything is enqueued.
 */
lat_status lat_dit_interval(lat_ctx *ctx, void *kv, float *lat, const lat_chunk_desc *chunks, int n,
                            void *stream);

/*
 * lat_dit_pipeline_push -- the scheduler of one stream's steady state (same
 * article): admit a new chunk and run one interval over every chunk in flight.
 * The context keeps, per stream, the latents of the chunks in flight (at most
 * S, one per denoise step) and the index of the next chunk.  A push
 *  - with noise != NULL admits chunk c = (chunks admitted so far) at step 0,
 *    its latent copied from noise (device fp32 [T_q][act_dim]);
 *  - runs lat_dit_interval on the chunks in flight (chunk c' at the number of
 *    intervals it has been through), then
 *  - if a chunk has completed its S steps: copies its latent to done (device
 *    fp32 [T_q][act_dim], may be NULL) and stores its index in *done_chunk
 *    (host), else *done_chunk = -1.
 * A push with noise == NULL only advances (drains) the chunks in flight.  In the
 * steady state a push admits chunk c and completes chunk c - S + 1.  Requires
 * S <= max_batch.  Asynchronous like every call; *done_chunk is known on return.
 */
lat_status lat_dit_pipeline_push(lat_ctx *ctx, void *kv, int stream_id, const float *noise, float *done,
                                 int *done_chunk, void *stream);

/*
 * lat_dit_set_text -- LAT_DIT with text_len > 0: the text context of one stream
 * ring (its chunks' cross-attention keys and values).
 * Defined by: none of the pages (the PhysisServe article names Wan-class
 * backbones, which attend to a text context; the reading): a sublayer between
 * self-attention and the FFN, x += Attn(LN(x) g_cross + b_cross, ctx) co with
 * q = (..) cq, k = ctx ck, v = ctx cv per head, no RoPE, no mask, no gate.
 *  text: device bf16 [text_len][D], already in the model width; read during the
 *        call (stream-ordered).
 * Computes every block's K/V of the context once, into the context's own
 * buffer (fp32 values kept as two fp16 planes), used by every later chunk of
 * that stream until the next call.  A chunk of a stream without a context
 * fails with LAT_ERR_STATE.
 */
lat_status lat_dit_set_text(lat_ctx *ctx, int stream_id, const void *text, void *stream);

/*
 * lat_dit_bind_pages -- LAT_DIT with page_tokens > 0: the page table of the
 * rings.  Defined by: none of the pages (M*'s serving layer integrates paged
 * attention; the reading): the (n_hist+1) * T_q tokens of each (stream, block,
 * step) ring -- chunk c's token j at ring row (c mod (n_hist+1)) * T_q + j --
 * live in pages of page_tokens tokens (a page size need not divide T_q).
 *  table: device int32 [n_streams][L][S][ceil((n_hist+1) T_q / page_tokens)],
 *         page indices into the pool; borrowed until the next call.
 * With pages bound, the kv argument of lat_block_forward / lat_dit_interval /
 * lat_dit_pipeline_push is the pool, device bf16 [pages][2][page_tokens][D]
 * (plane 0 K, plane 1 V); every value written and read is the one the
 * contiguous ring would hold at that row.  The caller keeps every page index
 * below the pool's size (not checked on the device).
 */
lat_status lat_dit_bind_pages(lat_ctx *ctx, const int *table);

/* lat_dit_pipeline_reset -- forget the chunks in flight of one stream and start
 * its chunk count at 0 again (host state only). */
lat_status lat_dit_pipeline_reset(lat_ctx *ctx, int stream_id);

/*
 * lat_debug_indices -- the integer maps the kernels use, computed by the same
 * device code: for chunk i (DiT) ring slot slot_out[i] and RoPE position of its
 * first token pos_out[i]; for the pi0 kinds (chunks = NULL, n = T_q) the cache
 * slot and position of query token i.  Host output arrays of n ints.
 * Synchronous; allocates and frees small temporary device buffers.
 */
lat_status lat_debug_indices(lat_ctx *ctx, const lat_chunk_desc *chunks, int n, int *slot_out,
                             int *pos_out);

/*
 * lat_debug_gemm -- measurement hook for the action expert: enqueue `reps`
 * back-to-back launches of one streamed projection (which: 0 = merged QKV,
 * 1 = attention output, 2 = gate/up, 3 = down) of blocks layer, layer+1, ...
 * (mod L, so successive launches stream different weights from HBM) on the
 * context's own workspace.  Used to time the weight-streaming kernel alone with
 * events on `stream`.  The block projections are held in the layout of the
 * persistent step kernel (fp16 = 2^s x the folded weight, QKV rows permuted),
 * which this bf16 kernel streams as bytes: its outputs are not meaningful,
 * only its time.  The workspace accumulators are left dirty: call
 * lat_debug_clear before the next lat_denoise_chunk / lat_block_forward.
 */
lat_status lat_debug_gemm(lat_ctx *ctx, int which, int layer, int reps, void *stream);
lat_status lat_debug_clear(lat_ctx *ctx, void *stream);

/*
 * lat_debug_step -- measurement hook for the action expert: enqueue `reps`
 * launches of the persistent step kernel (all L blocks of one denoise step,
 * each launch preceded by the clear of its barrier counter and statistics) on
 * the context's own residual stream, with the caller's cache `kv` (device,
 * [L][2][T_prefix + T_q][Hkv dh] bf16; own-token slots are overwritten).  Used
 * to time the kernel alone with events on `stream`; the residual stream is left
 * with meaningless values (the next lat_denoise_chunk overwrites it).
 */
lat_status lat_debug_step(lat_ctx *ctx, void *kv, int reps, void *stream);

/*
 * lat_debug_trace -- measurement hook for the action expert's persistent step
 * kernel: with buf != NULL (device, caller-owned, 8-byte aligned, at least
 * num_SMs * L * 64 entries) later launches record %globaltimer nanoseconds at
 * the phase boundaries of every block, buf[(layer * grid + cta) * 64 + event]
 * (event 0: block start; 2p + 1 / 2p + 2: phase p = 0..7 begins (after its grid
 * barrier) / ends; 17..19 inside the attention phase; 20 + 4 g .. 23 + 4 g for
 * projection g: first activation tile in, operand built, accumulator ready,
 * epilogue issued; 36, 37 inside the combine).  Each launch overwrites the
 * entries of its layers.  buf = NULL turns recording off.  Drops the captured
 * denoise graph (the next lat_denoise_chunk re-captures).  LAT_ERR_SHAPE if the
 * buffer is too small.  For a LAT_DIT context (dh = 128) later block calls record
 * the tensor-core attention of CTA (0, 0, 0) instead: buf[(role * 32 + block) * 8
 * + event] for the first 32 key blocks (role 0 MMA issue, 1 a row thread, 2 a
 * loader thread), at least 768 entries.
 */
lat_status lat_debug_trace(lat_ctx *ctx, unsigned long long *buf, long long n);

/*
 * lat_debug_dense_gemm -- one dense projection of a LAT_PI0_PREFIX or LAT_DIT
 * context alone (kernel-level parity and timing):
 *   out[m][n] = sum_t sum_k act[m][t*K + k] * W[n][k]
 * for the folded K-major weight W of block `layer` (which: 0 = merged QKV,
 * 1 = attention output, 2 = FFN in (prefix: gate/up interleaved in tiles of 64
 * gate + 64 up rows), 3 = FFN out).
 *  act: device fp16 [M][terms*K] (terms fp16 planes of one activation);
 *  out: device fp32 [M][N].  1 <= M <= the context's workspace rows, terms 1..2.
 *  W is held as fp16 = 2^s W (exact) and the result scaled back by 2^-s.
 */
lat_status lat_debug_dense_gemm(lat_ctx *ctx, int which, int layer, const void *act, int M, int terms,
                                float *out, void *stream);

/*
 * lat_debug_attention -- the chunk attention of an action-expert context
 * alone (kernel-level parity and timing): out = softmax(q k^T / sqrt(dh)) v,
 * no mask, query head h reading KV head h / (Hq / Hkv), using the context's
 * head layout and its workspace for the key-range partials.
 *  q:   device fp32 [T_q][Hq*dh] (RoPE already applied);
 *  k,v: device bf16 [T_kv][Hkv*dh];
 *  out: device fp32 [T_q][Hq*dh].
 * 1 <= T_q <= the context's T_q, 1 <= T_kv <= T_prefix + T_q of the context.
 * Reuses the context's workspace: not concurrent with other calls on it.
 */
lat_status lat_debug_attention(lat_ctx *ctx, const float *q, const void *k, const void *v, float *out, int T_q,
                               int T_kv, void *stream);

/*
 * lat_chunk_attention_noalloc -- the chunk attention for callers that cannot
 * allocate device memory.  (No counterpart on the pages: it is a packaging of
 * the attention step for such callers.)
 *
 * Who needs it: code that owns every byte of device memory itself -- an
 * inference engine with its own memory pool, or a real-time control loop that
 * forbids allocation once it runs -- can neither call cudaMalloc nor create a
 * context (lat_create allocates weights and workspace).  This call needs no
 * context and allocates nothing: the key-range partials it merges live in one
 * static device array of 4 MiB (1048576 floats) inside the library, which every
 * GPU that loads the library holds until the process exits.
 *
 *  out = softmax(q k^T / sqrt(dh)) v per query head, no mask, query head h
 *  reading KV head h / (Hq / Hkv).
 *  q:   device fp32 [T_q][Hq*dh];  k, v: device bf16 [T_kv][Hkv*dh];
 *  out: device fp32 [T_q][Hq*dh].  dh in {64, 128, 256}.
 * Limit: Hq * T_q * (dh + 2) <= 1048576 (one key range of partials), else
 * LAT_ERR_SHAPE; larger T_kv only means fewer, longer key ranges.
 * Speed: the keys are split into as many ranges as the array holds partials
 * for (at most 32, one per 32-key block at least), where a context's
 * attention sizes its ranges by the SM count; at shapes where the array holds
 * fewer ranges the call runs on fewer CTAs and is slower than the context's.
 * The first call on a device (with that device current) looks up the array's
 * device address and sets the kernels' shared-memory limit, and so does the
 * first call after the device's context changed (e.g. after cudaDeviceReset,
 * which unloads the library's module); make that first
 * call before any stream capture.  Every call shares the one array: calls that
 * overlap on the GPU (different streams, or different host threads) race on
 * it and must be serialised by the caller.  Nothing in it needs clearing: a
 * call writes every partial it reads.
 */
lat_status lat_chunk_attention_noalloc(const float *q, const void *k, const void *v, float *out, int T_q,
                                       int T_kv, int Hq, int Hkv, int dh, void *stream);

/* Wait for all work of the context and report a recorded device-side error. */
lat_status lat_sync(lat_ctx *ctx);

/*
 * lat_clear_error -- after lat_sync has returned LAT_ERR_TIMEOUT: wait for the
 * device, then clear the context's device error word so that its waits work
 * again.  (While the word is set, every bounded wait of the context's kernels
 * gives up at once and the results are meaningless.)  Synchronous.
 */
lat_status lat_clear_error(lat_ctx *ctx);

/*
 * lat_debug_timeout -- failure-detection check: enqueue one kernel whose
 * bounded wait (on an mbarrier that nothing arrives on) gives up after the
 * spin budget (~0.5 s) and records the error like any other wait of the path.
 * The next lat_sync returns LAT_ERR_TIMEOUT; no GPU fault is involved.
 */
lat_status lat_debug_timeout(lat_ctx *ctx, void *stream);

/*
 * lat_debug_wait_skew -- failure-detection check of the persistent step
 * kernel's own bounded waits (action-expert contexts).  From the next launch
 * on, one wait of the launch's first block expects `extra` more arrivals than
 * will ever come: which = 1 the first grid barrier (between the QKV and the
 * attention phase; `extra` arrivals too many), 2 the first QKV and 3 the
 * first gate/up exchange of split-K partial sums inside a thread-block
 * cluster (`extra` phases of the exchange barrier too many); which = 0 or
 * extra = 0 switches it off.  The wait gives up after the
 * spin budget (~0.5 s) and records LAT_ERR_TIMEOUT; every later wait of the
 * launch sees the error and returns at once, the launch runs to its end with
 * meaningless results and leaves no copy in flight.  The next lat_sync
 * reports the timeout; after lat_clear_error (and the skew switched off) the
 * context computes correct results again.  No GPU fault is involved.
 * Captured denoise graphs are dropped (they hold the old arguments).
 */
lat_status lat_debug_wait_skew(lat_ctx *ctx, int which, int extra);

/*
 * lat_debug_act_terms -- precision study of the dense path (LAT_PI0_PREFIX,
 * LAT_DIT): the block projections multiply `terms` fp16 planes of their
 * activation (2, the default: hi + lo, 22 significant bits; 1: hi only, 11
 * bits, half the tensor work).  For measuring the error of one plane against
 * the oracle; not meant for production use.
 */
lat_status lat_debug_act_terms(lat_ctx *ctx, int terms);

/* Human-readable name of a status; message of the last failure on this thread. */
const char *lat_status_str(lat_status s);
const char *lat_last_error(void);

void lat_destroy(lat_ctx *ctx);

#ifdef __cplusplus
}
#endif
#endif /* LAT_H */
