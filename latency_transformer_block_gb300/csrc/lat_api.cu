// C ABI of the low-latency transformer-block library (declared in include/lat.h).
//
// Host side: argument validation, offline folds, tensor maps, workspace, the
// per-block kernel sequence and the CUDA-graph capture of the denoise loop
// ("Running VLAs at Real-time Speed", reading note, section 3: CUDA Graph
// replay of a fixed kernel sequence with fixed buffers).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <utility>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/lat.h"
#include "attention.cuh"
#include "attention_tc.cuh"
#include "common.cuh"
#include "dense_gemm.cuh"
#include "dense_kernels.cuh"
#include "pi0_step.cuh"
#include "skinny_gemm.cuh"
#include "small_kernels.cuh"

using namespace lat;
typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// errors
// ---------------------------------------------------------------------------
static thread_local std::string g_last_error;

lat_status lat_internal_fail(lat_status s, const char* msg) {
  g_last_error = msg;
  return s;
}

static lat_status fail(lat_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

#define CUDA_TRY(expr)                                                                        \
  do {                                                                                        \
    cudaError_t e_ = (expr);                                                                  \
    if (e_ != cudaSuccess)                                                                    \
      return fail(e_ == cudaErrorMemoryAllocation ? LAT_ERR_OOM : LAT_ERR_CUDA, "%s: %s (%s:%d)", \
                  #expr, cudaGetErrorString(e_), __FILE__, __LINE__);                         \
  } while (0)

#define LAT_TRY(expr)              \
  do {                             \
    lat_status s_ = (expr);        \
    if (s_ != LAT_OK) return s_;   \
  } while (0)

static inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------
// tensor maps (driver entry point fetched through the runtime)
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static lat_status get_encode(EncodeTiledFn* fn) {
  static EncodeTiledFn cached = nullptr;
  if (!cached) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    CUDA_TRY(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q));
    if (q != cudaDriverEntryPointSuccess || !p) return fail(LAT_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cached = reinterpret_cast<EncodeTiledFn>(p);
  }
  *fn = cached;
  return LAT_OK;
}

// K-major bf16 matrix [rows][K] -> tiles of 128 rows x 64 K, 128-byte swizzle.
static lat_status make_kmajor_map(CUtensorMap* map, const void* base, int rows, int K, int box_rows) {
  EncodeTiledFn enc;
  LAT_TRY(get_encode(&enc));
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(LAT_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return LAT_OK;
}

// ---------------------------------------------------------------------------
// context
// ---------------------------------------------------------------------------
struct GemmPlan {
  int w_row0_per_layer;  // rows of one layer inside the stacked tensor
  int N_out, K, splits;
};

struct lat_ctx {
  lat_model_desc d{};
  int num_sms = 0;
  std::vector<void*> allocs;

  // streamed block weights, K-major bf16, stacked over layers
  bf16 *wqkv = nullptr, *wo = nullptr, *wgu = nullptr, *wd = nullptr, *w2 = nullptr;
  CUtensorMap map_qkv, map_o, map_gu, map_d, map_w2;
  int nqkv = 0;
  GemmPlan g_qkv{}, g_o{}, g_gu{}, g_d{};

  // action-expert tables (fp32)
  float *wfold = nullptr, *ttab = nullptr, *b2 = nullptr, *gfin = nullptr, *bout = nullptr, *dt = nullptr;
  bf16 *w_state = nullptr, *b_state = nullptr, *w1_keep = nullptr, *b1_keep = nullptr, *w_in_keep = nullptr,
       *b_in_keep = nullptr, *w_out = nullptr;
  float* cos_t = nullptr;
  float* sin_t = nullptr;

  // workspace
  bf16 *planes_x = nullptr, *planes_o = nullptr, *planes_h = nullptr;   // [3][64][K] activation planes
  CUtensorMap bmap_x, bmap_o, bmap_h, pmap_o, pmap_h, pmap_e;
  float *xres = nullptr, *qkv_acc = nullptr, *gu_acc = nullptr, *q = nullptr, *o = nullptr, *r1 = nullptr,
        *r2 = nullptr, *z = nullptr, *pm = nullptr, *pl = nullptr, *po = nullptr, *state_emb = nullptr,
        *temb = nullptr;
  int attn_split = 1;
  DevErr* err = nullptr;

  // persistent step kernel: arguments, zero-at-entry block
  MkArgs mk{};
  int step_grid = 0;   // CTAs of one step-kernel launch: co-resident clusters x 4
  void* mk_zero = nullptr;
  size_t mk_zero_bytes = 0;

  // dense path (prefix prefill, DiT)
  bf16 *wup = nullptr, *wdown = nullptr, *wpatch = nullptr;
  CUtensorMap map_up, map_down, map_patch;
  float *bpatch = nullptr, *adaln = nullptr, *cos_j = nullptr, *sin_j = nullptr, *qkvbuf = nullptr,
        *qbuf = nullptr;
  float* adaln_tmp = nullptr;   // scratch of the adaLN table build: [S][t_dim], [S][D], [S][D]
  // prefix attention split over key ranges: partial outputs and (max, sum), at
  // most num_sms CTAs x 64 rows
  float *seg_part_o = nullptr, *seg_part_ml = nullptr;
  float *tc_part_o = nullptr, *tc_part_ml = nullptr;   // DiT attention: key ranges of the split tiles
  double* theta = nullptr;
  __half *kown = nullptr, *vown = nullptr;   // own tokens' K/V as computed, two fp16 planes [2][m_max][kvd] (prefill)
  __half* kvown16 = nullptr;   // the same as fp16 planes [M][K hi | K lo | V hi | V lo] (DiT)
  float4* rope_rot = nullptr;  // DiT: each row's rotation, [m_max / 32][2][16][32] float4 (rope_rows_kernel)
  __half* hist16 = nullptr;    // fp16 copy of one call's history K/V planes, [planes][T_q][D] (DiT)
  int hist_rows = 0;
  __half *act2 = nullptr, *act2f = nullptr;   // fp16 activation planes [M][kActTerms * K]
  int act_terms = kActTerms;   // planes of the activation the block projections multiply (1: hi only)
  // the four block projections (merged QKV, output, FFN in, FFN out) of the dense
  // path are held as fp16 = 2^s x folded bf16 weight; wscale = 2^-s per matrix
  float wscale[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};   // indexed by WSel
  CUtensorMap map_act_d, map_act_o, map_act_f;
  int m_max = 0;
  bf16 *wt1 = nullptr, *bt1 = nullptr, *wt2 = nullptr, *bt2 = nullptr, *wmod = nullptr, *bmod = nullptr;

  unsigned long long* attn_trace = nullptr;   // DiT: timestamps of the attention (measurement hook)

  // DiT, Wan-class options
  int frames_per_chunk = 0;        // 3-D RoPE: T_q / (grid_h grid_w)
  bf16 *wcq = nullptr, *wco = nullptr, *wckv = nullptr;   // cross-attention, K-major fp16 (2^s): [L][D][D],
  CUtensorMap map_cq, map_co, map_ckv;                      //   [L][D][D], [L][2D][D] (K rows, then V rows)
  float* cross_ln = nullptr;       // [L][2][D]: b_cross (shift), g_cross - 1 (scale)
  __half* text_kv = nullptr;       // [n_streams][L][text_len][K hi | K lo | V hi | V lo]
  std::vector<char> text_set;      // per stream: lat_dit_set_text was called
  const int* page_table = nullptr; // [n_streams][L][S][pages_per_ring] (lat_dit_bind_pages)
  int pages_per_ring = 0;

  // DiT latent I/O (act_dim > 0) and the interleaved schedule
  bf16 *wlin = nullptr, *blin = nullptr, *wlout = nullptr, *blout = nullptr;   // [A][D], [D], [D][A], [A]
  float *dit_x = nullptr, *dit_z = nullptr, *dit_v = nullptr;   // [m_max][D], [m_max][A], [m_max][A]
  float* pipe_lat = nullptr;                   // [n_streams][S][T_q][A]: latents in flight, slot c mod S
  std::vector<int> pipe_next, pipe_done;       // per stream: chunks admitted / completed so far
  std::vector<int> pipe_step;                  // [n_streams][S]: steps done by the chunk in each slot

  // captured denoise loop
  // captured denoise loops, one per (kv, state, x, stream), least recently used replaced
  struct Graph {
    cudaGraphExec_t exec = nullptr;
    void* kv = nullptr;
    const float* state = nullptr;
    float* x = nullptr;
    void* stream = nullptr;
    unsigned long long used = 0;
  };
  static constexpr int kGraphs = 4;
  Graph graphs[kGraphs];
  unsigned long long graph_clock = 0;
  void drop_graphs() {
    for (Graph& g : graphs) {
      if (g.exec) cudaGraphExecDestroy(g.exec);
      g = Graph{};
    }
  }

  template <class T>
  lat_status alloc(T** p, size_t count) {
    void* v = nullptr;
    cudaError_t e = cudaMalloc(&v, count * sizeof(T) + 16);
    if (e != cudaSuccess) return fail(LAT_ERR_OOM, "cudaMalloc(%zu): %s", count * sizeof(T), cudaGetErrorString(e));
    allocs.push_back(v);
    *p = reinterpret_cast<T*>(v);
    return LAT_OK;
  }
  ~lat_ctx() {
    drop_graphs();
    for (void* p : allocs) cudaFree(p);
  }
};

static constexpr int kStages = 4;
static constexpr int kMaxKeySplits = 32;   // partials the combine kernel merges

static lat_status launch_check(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(LAT_ERR_CUDA, "launch %s: %s", what, cudaGetErrorString(e));
  return LAT_OK;
}

static GemmPlan plan_gemm(int N_out, int K, int num_sms) {
  GemmPlan p;
  p.w_row0_per_layer = N_out;
  p.N_out = N_out;
  p.K = K;
  const int m_tiles = N_out / 128, kb = K / 64;
  int s = num_sms / m_tiles;
  if (s < 1) s = 1;
  if (s > kb) s = kb;
  p.splits = s;
  return p;
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel on the stream finishes; it orders itself with
// griddepcontrol.wait before touching that kernel's results.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

#define PDL_TRY(what, expr)                                                              \
  do {                                                                                   \
    cudaError_t e_ = (expr);                                                             \
    if (e_ != cudaSuccess) return fail(LAT_ERR_CUDA, "launch %s: %s", what, cudaGetErrorString(e_)); \
  } while (0)

static lat_status enqueue_skinny(const lat_ctx* c, const CUtensorMap& map, const CUtensorMap& bmap,
                                 const GemmPlan& g, int layer, SkinnyArgs a, cudaStream_t st) {
  a.w_row0 = layer * g.w_row0_per_layer;
  a.N_out = g.N_out;
  a.K = g.K;
  a.splits = g.splits;
  a.err = c->err;
  const int grid = (g.N_out / 128) * g.splits;
  PDL_TRY("skinny_gemm", launch_pdl(skinny_gemm_kernel<kStages>, dim3(grid), dim3(192),
                                    (size_t)skinny_smem_bytes(kStages), st, map, bmap, a));
  return LAT_OK;
}

// planes [3 * 64][K] bf16 read by TMA in 192 x 64 boxes
static lat_status make_planes_map(CUtensorMap* map, const void* base, int K) {
  return make_kmajor_map(map, base, 192, K, 192);
}

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------
static lat_status check_desc(const lat_model_desc* d) {
  if (!d) return fail(LAT_ERR_ARG, "desc is NULL");
  if (d->kind != LAT_PI0_ACTION_EXPERT && d->kind != LAT_PI0_PREFIX && d->kind != LAT_DIT)
    return fail(LAT_ERR_UNSUPPORTED, "model kind %d not built into this library", d->kind);
  if (d->Hq <= 0 || d->Hkv <= 0 || d->Hq % d->Hkv) return fail(LAT_ERR_SHAPE, "Hq must be a multiple of Hkv");
  if (d->L <= 0) return fail(LAT_ERR_SHAPE, "L must be positive");
  if (!(d->eps > 0.f) || !(d->rope_base > 1.f)) return fail(LAT_ERR_ARG, "eps / rope_base out of range");
  if (d->F <= 0) return fail(LAT_ERR_SHAPE, "F must be positive");
  if (d->kind == LAT_PI0_ACTION_EXPERT) {
    if (d->D <= 0 || d->D % 128 || d->D > 8192) return fail(LAT_ERR_SHAPE, "D must be a multiple of 128 in [128, 8192]");
    if (d->dh != 64 && d->dh != 128 && d->dh != 256) return fail(LAT_ERR_SHAPE, "dh must be 64, 128 or 256");
    if (((d->Hq + 2 * d->Hkv) * d->dh) % 128) return fail(LAT_ERR_SHAPE, "(Hq + 2 Hkv) dh must be a multiple of 128");
    if ((d->Hq * d->dh) % 64) return fail(LAT_ERR_SHAPE, "Hq dh must be a multiple of 64");
    if (d->F % 64) return fail(LAT_ERR_SHAPE, "F must be a multiple of 64");
    if (d->S <= 0) return fail(LAT_ERR_SHAPE, "S must be positive");
    if (d->T_q < 2 || d->T_q > 64) return fail(LAT_ERR_SHAPE, "T_q must be in [2, 64]");
    if (d->T_prefix < 0) return fail(LAT_ERR_SHAPE, "T_prefix must be >= 0");
    if (d->act_dim <= 0) return fail(LAT_ERR_SHAPE, "act_dim must be positive");
    if (d->prefix_lm != 0 && d->prefix_lm != 1) return fail(LAT_ERR_ARG, "prefix_lm must be 0 or 1");
    return LAT_OK;
  }
  // dense kinds: 128 x 256 x 64 tiles (every projection width a multiple of 256)
  if (d->dh != 128 && d->dh != 256) return fail(LAT_ERR_SHAPE, "dh must be 128 or 256 for the dense path");
  if (d->D <= 0 || d->D % 256 || d->D > 8192) return fail(LAT_ERR_SHAPE, "D must be a multiple of 256 in [256, 8192]");
  if (d->prefix_lm) return fail(LAT_ERR_ARG, "prefix_lm applies to the action expert only");
  if ((d->Hq * d->dh) % 256) return fail(LAT_ERR_SHAPE, "Hq dh must be a multiple of 256");
  if (d->max_batch < 1 || d->max_batch > kMaxChunks) return fail(LAT_ERR_SHAPE, "max_batch must be in [1, 16]");
  if (d->kind == LAT_PI0_PREFIX) {
    if (d->dh != 256) return fail(LAT_ERR_SHAPE, "prefix model: dh must be 256");
    if (((d->Hq + 2 * d->Hkv) * d->dh) % 256 || (2 * d->Hkv * d->dh) % 256)
      return fail(LAT_ERR_SHAPE, "QKV and KV widths must be multiples of 256");
    if (d->F % 128) return fail(LAT_ERR_SHAPE, "F must be a multiple of 128");
    if (d->patch_dim <= 0 || d->patch_dim % 64) return fail(LAT_ERR_SHAPE, "patch_dim must be a multiple of 64");
    if (d->T_prefix < 1 || d->T_q < 0) return fail(LAT_ERR_SHAPE, "T_prefix must be >= 1");
    return LAT_OK;
  }
  if (d->Hq != d->Hkv || d->Hq * d->dh != d->D) return fail(LAT_ERR_SHAPE, "DiT: Hq == Hkv and Hq dh == D");
  if (d->dh != 128) return fail(LAT_ERR_SHAPE, "DiT: dh must be 128 (tensor-core attention)");
  if (d->F % 256) return fail(LAT_ERR_SHAPE, "F must be a multiple of 256");
  if (d->S <= 0 || d->T_q < 1 || d->n_hist < 0 || d->n_streams < 1 || d->t_dim <= 0 || d->t_dim % 2)
    return fail(LAT_ERR_SHAPE, "DiT: S, T_q, n_streams, t_dim must be positive (t_dim even), n_hist >= 0");
  if (d->n_hist + 1 > kMaxSeg) return fail(LAT_ERR_SHAPE, "n_hist must be <= 4");
  if (d->act_dim < 0) return fail(LAT_ERR_SHAPE, "DiT: act_dim (latent channels) must be >= 0");
  if (d->grid_h < 0 || d->grid_w < 0 || (d->grid_h > 0) != (d->grid_w > 0))
    return fail(LAT_ERR_SHAPE, "DiT: grid_h and grid_w both positive (3-D RoPE) or both 0");
  if (d->grid_h > 0 && d->T_q % (d->grid_h * d->grid_w))
    return fail(LAT_ERR_SHAPE, "DiT: T_q must be whole frames of grid_h x grid_w tokens");
  if (d->text_len < 0 || d->text_len > d->max_batch * d->T_q)
    return fail(LAT_ERR_SHAPE, "DiT: text_len must be in [0, max_batch * T_q]");
  if (d->page_tokens < 0 || (d->page_tokens > 0 && d->page_tokens > (d->n_hist + 1) * d->T_q))
    return fail(LAT_ERR_SHAPE, "DiT: page_tokens must be in [0, (n_hist + 1) T_q]");
  return LAT_OK;
}
// ring rows of one (stream, block, step) and pages per ring
static int ring_pages(const lat_model_desc& d) {
  return d.page_tokens > 0 ? ((d.n_hist + 1) * d.T_q + d.page_tokens - 1) / d.page_tokens : 0;
}

// ---------------------------------------------------------------------------
// offline folds
// ---------------------------------------------------------------------------
static float bf16_bits_to_float(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

static lat_status fold_t(const void* W, const void* g, bf16* out, int K, int N, int il = 0, int il_off = 0) {
  if (!W || !aligned16(W)) return fail(LAT_ERR_ALIGN, "weight pointer NULL or not 16-byte aligned");
  dim3 grid((N + 31) / 32, (K + 31) / 32), block(32, 8);
  fold_transpose_kernel<<<grid, block>>>(reinterpret_cast<const bf16*>(W), reinterpret_cast<const bf16*>(g), out,
                                         K, N, il, il_off);
  return launch_check("fold_transpose");
}

// Hold a folded bf16 weight (n values) as fp16 = 2^s w in place, s chosen so
// that max |w| 2^s lies in [2^14, 2^15): the conversion is exact except for
// values below 2^(-14-s), which keep fp16's subnormal spacing (an absolute
// error <= 2^(-25-s), ~1e-13 for N(0, 0.02) weights).  *inv = 2^-s.
static lat_status to_f16_scaled(bf16* w, size_t n, float* inv) {
  unsigned* dmax = nullptr;
  CUDA_TRY(cudaMalloc(&dmax, sizeof(unsigned)));
  unsigned hm = 0;
  cudaError_t e = cudaMemset(dmax, 0, sizeof(unsigned));
  if (e == cudaSuccess) {
    absmax_bf16_kernel<<<1024, 256>>>(w, n, dmax);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpy(&hm, dmax, sizeof(unsigned), cudaMemcpyDeviceToHost);
  cudaFree(dmax);
  if (e != cudaSuccess) return fail(LAT_ERR_CUDA, "weight scan: %s", cudaGetErrorString(e));
  float m;
  std::memcpy(&m, &hm, sizeof(float));
  if (!std::isfinite(m)) return fail(LAT_ERR_ARG, "non-finite weight");
  int ex = 0;
  if (m > 0.f) std::frexp(m, &ex);          // m < 2^ex
  const int s = m > 0.f ? std::min(15 - ex, 100) : 0;
  *inv = std::ldexp(1.f, -s);
  const size_t blocks = std::min<size_t>((n + 255) / 256, 65536);
  bf16_to_f16_scaled_kernel<<<(unsigned)blocks, 256>>>(reinterpret_cast<uint16_t*>(w), n, std::ldexp(1.f, s));
  return launch_check("to_f16_scaled");
}

static lat_status small_gemm(const void* A, bool a_bf16, int lda, const void* B, bool b_bf16, int ldb,
                             const void* bias, bool bias_bf16, float* C, int ldc, int M, int N, int K, int act,
                             cudaStream_t st = 0) {
  SmallGemmArgs a{A, a_bf16, lda, B, b_bf16, ldb, bias, bias_bf16, C, ldc, M, N, K, act};
  dim3 grid((N + 127) / 128, M);
  small_gemm_kernel<<<grid, 128, 0, st>>>(a);
  return launch_check("small_gemm");
}

static void timestep_embedding_host(double t, int d, std::vector<float>& out) {
  const int half = d / 2;
  out.resize(d);
  for (int i = 0; i < half; ++i) {
    const double w = std::pow(10000.0, -(double)i / half);
    out[i] = (float)std::sin(1000.0 * t * w);
    out[half + i] = (float)std::cos(1000.0 * t * w);
  }
}

static lat_status build_schedule(lat_ctx* c, const std::vector<double>& t) {
  const lat_model_desc& d = c->d;
  // time table T[s] = temb(t_s) W1[D:2D] + b_in W1[0:D] + b1, and dt[s]
  std::vector<float> emb((size_t)d.S * d.D), tmp;
  for (int s = 0; s < d.S; ++s) {
    timestep_embedding_host(t[s], d.D, tmp);
    std::memcpy(&emb[(size_t)s * d.D], tmp.data(), d.D * sizeof(float));
  }
  std::vector<float> dts(d.S);
  for (int s = 0; s < d.S; ++s) dts[s] = (float)(t[s + 1] - t[s]);
  CUDA_TRY(cudaMemcpy(c->temb, emb.data(), emb.size() * sizeof(float), cudaMemcpyHostToDevice));
  CUDA_TRY(cudaMemcpy(c->dt, dts.data(), dts.size() * sizeof(float), cudaMemcpyHostToDevice));
  // bias row c0 = b_in W1[0:D] + b1  (into ttab row 0 temporarily via z scratch)
  float* c0 = c->z;  // [D] scratch
  LAT_TRY(small_gemm(c->b_in_keep, true, d.D, c->w1_keep, true, d.D, c->b1_keep, true, c0, d.D, 1, d.D, d.D, 0));
  // T[s] = temb(t_s) W1_t + c0
  LAT_TRY(small_gemm(c->temb, false, d.D, c->w1_keep + (size_t)d.D * d.D, true, d.D, c0, false, c->ttab, d.D, d.S,
                     d.D, d.D, 0));
  CUDA_TRY(cudaDeviceSynchronize());
  return LAT_OK;
}

// the step kernel for a head dimension: the blocks of one step, or a whole chunk
static const void* step_kernel(int dh, bool chunk) {
  if (dh == 64) return chunk ? (const void*)pi0_step_kernel<64, true> : (const void*)pi0_step_kernel<64, false>;
  if (dh == 128) return chunk ? (const void*)pi0_step_kernel<128, true> : (const void*)pi0_step_kernel<128, false>;
  return chunk ? (const void*)pi0_step_kernel<256, true> : (const void*)pi0_step_kernel<256, false>;
}

// Grid of the persistent step kernel: as many clusters of kMkCluster CTAs
// (one CTA per SM) as can be resident at once, which its grid barriers need.
static lat_status step_grid(lat_ctx* c) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kMkCluster);
  cfg.blockDim = dim3(kMkThreads);
  cfg.dynamicSmemBytes = mk_smem_bytes();
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kMkCluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  cudaError_t e;
  e = cudaOccupancyMaxActiveClusters(&n, step_kernel(c->d.dh, true), &cfg);
  if (e != cudaSuccess) return fail(LAT_ERR_CUDA, "cudaOccupancyMaxActiveClusters: %s", cudaGetErrorString(e));
  n = std::min(n, c->num_sms / kMkCluster);
  if (n < 1) return fail(LAT_ERR_UNSUPPORTED, "no cluster of %d step-kernel CTAs fits on this device", kMkCluster);
  c->step_grid = n * kMkCluster;
  return LAT_OK;
}

static lat_status create_pi0(lat_ctx* c, const lat_weights* w) {
  const lat_model_desc& d = c->d;
  const int D = d.D, F = d.F, L = d.L, A = d.act_dim;
  const int qd = d.Hq * d.dh, kvd = d.Hkv * d.dh;
  c->nqkv = (d.Hq + 2 * d.Hkv) * d.dh;
  if (!w || !w->blocks) return fail(LAT_ERR_ARG, "weights / blocks NULL");
  const void* vecs[] = {w->w_in, w->b_in, w->w1, w->b1, w->w2, w->b2, w->w_state, w->b_state, w->g_final, w->w_out,
                        w->b_out};
  for (const void* p : vecs)
    if (!p || !aligned16(p)) return fail(LAT_ERR_ALIGN, "embedding/head weight NULL or not 16-byte aligned");
  for (int l = 0; l < L; ++l) {
    const lat_block_weights& b = w->blocks[l];
    const void* bp[] = {b.g_attn, b.wq, b.wk, b.wv, b.wo, b.g_ffn, b.wg, b.wu, b.wd};
    for (const void* p : bp)
      if (!p || !aligned16(p)) return fail(LAT_ERR_ALIGN, "block %d weight NULL or not 16-byte aligned", l);
  }
  // --- streamed weights: fold + transpose to K-major, stacked over layers ---
  LAT_TRY(c->alloc(&c->wqkv, (size_t)L * c->nqkv * D));
  LAT_TRY(c->alloc(&c->wo, (size_t)L * D * qd));
  LAT_TRY(c->alloc(&c->wgu, (size_t)L * 2 * F * D));
  LAT_TRY(c->alloc(&c->wd, (size_t)L * D * F));
  LAT_TRY(c->alloc(&c->w2, (size_t)D * D));
  // merged QKV rows permuted for the step kernel: in each 128-row tile, row
  // 32 j + c holds the first element of rotary pair 16 j + c of the tile and
  // row 32 j + 16 + c its partner dh / 2 further on, so that the quarter of a
  // tile one CTA finalizes holds whole pairs (the pairs of the heads q.., k..,
  // v.. in order; v rows are not rotated but move the same way)
  if (c->nqkv % 128) return fail(LAT_ERR_SHAPE, "(Hq + 2 Hkv) * dh must be a multiple of 128");
  std::vector<int> perm(c->nqkv);
  {
    const int pph = d.dh / 2;
    for (int u = 0; u < c->nqkv / 128; ++u)
      for (int j = 0; j < 4; ++j)
        for (int h = 0; h < 2; ++h)
          for (int cc = 0; cc < 16; ++cc) {
            const int P = 64 * u + 16 * j + cc;
            perm[128 * u + 32 * j + 16 * h + cc] = (P / pph) * d.dh + P % pph + h * pph;
          }
  }
  int* dperm = nullptr;
  bf16* qkv_tmp = nullptr;
  LAT_TRY(c->alloc(&dperm, (size_t)c->nqkv));
  LAT_TRY(c->alloc(&qkv_tmp, (size_t)c->nqkv * D));
  CUDA_TRY(cudaMemcpy(dperm, perm.data(), perm.size() * sizeof(int), cudaMemcpyHostToDevice));
  for (int l = 0; l < L; ++l) {
    const lat_block_weights& b = w->blocks[l];
    bf16* q0 = c->wqkv + (size_t)l * c->nqkv * D;
    LAT_TRY(fold_t(b.wq, b.g_attn, qkv_tmp, D, qd));
    LAT_TRY(fold_t(b.wk, b.g_attn, qkv_tmp + (size_t)qd * D, D, kvd));
    LAT_TRY(fold_t(b.wv, b.g_attn, qkv_tmp + (size_t)(qd + kvd) * D, D, kvd));
    gather_rows_kernel<<<c->nqkv, 256>>>(qkv_tmp, dperm, q0, c->nqkv, D);
    LAT_TRY(launch_check("gather_rows"));
    LAT_TRY(fold_t(b.wo, nullptr, c->wo + (size_t)l * D * qd, qd, D));
    // gate/up rows interleaved in 128-row tiles: 64 gate rows, then the 64 up
    // rows of the same FFN columns (one tile holds both inputs of its GeGLU)
    bf16* gu0 = c->wgu + (size_t)l * 2 * F * D;
    LAT_TRY(fold_t(b.wg, b.g_ffn, gu0, D, F, 64, 0));
    LAT_TRY(fold_t(b.wu, b.g_ffn, gu0, D, F, 64, 64));
    LAT_TRY(fold_t(b.wd, nullptr, c->wd + (size_t)l * D * F, F, D));
  }
  LAT_TRY(fold_t(w->w2, nullptr, c->w2, D, D));
  // the step kernel multiplies the block projections with two fp16 planes of
  // the activation: each family is held as fp16 = 2^s x the folded bf16 weight
  // (exact), 2^-s applied in the epilogue
  LAT_TRY(to_f16_scaled(c->wqkv, (size_t)L * c->nqkv * D, &c->mk.wsc[0]));
  LAT_TRY(to_f16_scaled(c->wo, (size_t)L * D * qd, &c->mk.wsc[1]));
  LAT_TRY(to_f16_scaled(c->wgu, (size_t)L * 2 * F * D, &c->mk.wsc[2]));
  LAT_TRY(to_f16_scaled(c->wd, (size_t)L * D * F, &c->mk.wsc[3]));
  LAT_TRY(to_f16_scaled(c->w2, (size_t)D * D, &c->mk.wsc[4]));
  LAT_TRY(make_kmajor_map(&c->map_qkv, c->wqkv, L * c->nqkv, D, 128));
  LAT_TRY(make_kmajor_map(&c->map_o, c->wo, L * D, qd, 128));
  LAT_TRY(make_kmajor_map(&c->map_gu, c->wgu, L * 2 * F, D, 128));
  LAT_TRY(make_kmajor_map(&c->map_d, c->wd, L * D, F, 128));
  LAT_TRY(make_kmajor_map(&c->map_w2, c->w2, D, D, 128));
  c->g_qkv = plan_gemm(c->nqkv, D, c->num_sms);
  c->g_o = plan_gemm(D, qd, c->num_sms);
  c->g_gu = plan_gemm(2 * F, D, c->num_sms);
  c->g_d = plan_gemm(D, F, c->num_sms);

  // --- embedding / head (fp32 folds) ---
  LAT_TRY(c->alloc(&c->w_in_keep, (size_t)A * D));
  LAT_TRY(c->alloc(&c->b_in_keep, (size_t)D));
  LAT_TRY(c->alloc(&c->w1_keep, (size_t)2 * D * D));
  LAT_TRY(c->alloc(&c->b1_keep, (size_t)D));
  LAT_TRY(c->alloc(&c->w_state, (size_t)A * D));
  LAT_TRY(c->alloc(&c->b_state, (size_t)D));
  CUDA_TRY(cudaMemcpy(c->w_in_keep, w->w_in, (size_t)A * D * 2, cudaMemcpyDeviceToDevice));
  CUDA_TRY(cudaMemcpy(c->b_in_keep, w->b_in, (size_t)D * 2, cudaMemcpyDeviceToDevice));
  CUDA_TRY(cudaMemcpy(c->w1_keep, w->w1, (size_t)2 * D * D * 2, cudaMemcpyDeviceToDevice));
  CUDA_TRY(cudaMemcpy(c->b1_keep, w->b1, (size_t)D * 2, cudaMemcpyDeviceToDevice));
  CUDA_TRY(cudaMemcpy(c->w_state, w->w_state, (size_t)A * D * 2, cudaMemcpyDeviceToDevice));
  CUDA_TRY(cudaMemcpy(c->b_state, w->b_state, (size_t)D * 2, cudaMemcpyDeviceToDevice));
  LAT_TRY(c->alloc(&c->wfold, (size_t)A * D));
  LAT_TRY(c->alloc(&c->ttab, (size_t)d.S * D));
  LAT_TRY(c->alloc(&c->temb, (size_t)d.S * D));
  LAT_TRY(c->alloc(&c->dt, (size_t)d.S));
  LAT_TRY(c->alloc(&c->b2, (size_t)D));
  LAT_TRY(c->alloc(&c->gfin, (size_t)D));
  LAT_TRY(c->alloc(&c->w_out, (size_t)D * A));
  LAT_TRY(c->alloc(&c->bout, (size_t)A));
  // W' = W_in W1[0:D]
  LAT_TRY(small_gemm(w->w_in, true, D, w->w1, true, D, nullptr, false, c->wfold, D, A, D, D, 0));
  bf16_to_f32_kernel<<<(D + 255) / 256, 256>>>(reinterpret_cast<const bf16*>(w->b2), c->b2, D);
  LAT_TRY(launch_check("b2"));
  bf16_to_f32_kernel<<<(A + 255) / 256, 256>>>(reinterpret_cast<const bf16*>(w->b_out), c->bout, A);
  LAT_TRY(launch_check("bout"));
  bf16_to_f32_kernel<<<(D + 255) / 256, 256>>>(reinterpret_cast<const bf16*>(w->g_final), c->gfin, D);
  LAT_TRY(launch_check("g_final"));
  CUDA_TRY(cudaMemcpy(c->w_out, w->w_out, (size_t)D * A * 2, cudaMemcpyDeviceToDevice));

  // --- RoPE tables for the query positions (float64 -> fp32) ---
  const int half = d.dh / 2;
  std::vector<float> ct((size_t)d.T_q * half), stt((size_t)d.T_q * half);
  for (int t = 0; t < d.T_q; ++t)
    for (int i = 0; i < half; ++i) {
      const double theta = std::pow((double)d.rope_base, -2.0 * i / d.dh);
      const double ang = (double)query_pos(d.T_prefix, t) * theta;
      ct[(size_t)t * half + i] = (float)std::cos(ang);
      stt[(size_t)t * half + i] = (float)std::sin(ang);
    }
  LAT_TRY(c->alloc(&c->cos_t, ct.size()));
  LAT_TRY(c->alloc(&c->sin_t, stt.size()));
  CUDA_TRY(cudaMemcpy(c->cos_t, ct.data(), ct.size() * 4, cudaMemcpyHostToDevice));
  CUDA_TRY(cudaMemcpy(c->sin_t, stt.data(), stt.size() * 4, cudaMemcpyHostToDevice));
  // the same angles in the step kernel's q-fragment order: [warp][dh / 64][4][lane]
  // x {cos i, cos i+1, sin i, sin i+1}, warp = row tile (w & 3) x dim half (w >> 2)
  {
    const int ksh = d.dh / 64, q4 = d.dh / 4;
    std::vector<float> rf((size_t)8 * ksh * 4 * 32 * 4, 0.f);
    for (int w = 0; w < 8; ++w)
      for (int ks = 0; ks < ksh; ++ks)
        for (int e = 0; e < 4; ++e)
          for (int ln = 0; ln < 32; ++ln) {
            const int row = (w & 3) * 16 + (ln >> 2) + (e & 1) * 8;
            const int i = (w >> 2) * q4 + ks * 16 + 2 * (ln & 3) + (e >> 1) * 8;
            if (row >= d.T_q) continue;
            float* o = &rf[((((size_t)w * ksh + ks) * 4 + e) * 32 + ln) * 4];
            o[0] = ct[(size_t)row * half + i];
            o[1] = ct[(size_t)row * half + i + 1];
            o[2] = stt[(size_t)row * half + i];
            o[3] = stt[(size_t)row * half + i + 1];
          }
    float* dev = nullptr;
    LAT_TRY(c->alloc(&dev, rf.size()));
    CUDA_TRY(cudaMemcpy(dev, rf.data(), rf.size() * 4, cudaMemcpyHostToDevice));
    c->mk.rope_frag = reinterpret_cast<const float4*>(dev);
  }

  // --- workspace ---
  const int T = d.T_q;
  const int T_kv = d.T_prefix + d.T_q;
  const int nkb = attn_key_blocks(T_kv);
  c->attn_split = nkb < kMaxKeySplits ? nkb : kMaxKeySplits;
  LAT_TRY(c->alloc(&c->xres, (size_t)64 * D));   // 64 rows: the step kernel reads 64 x 64 tiles
  LAT_TRY(c->alloc(&c->qkv_acc, (size_t)T * c->nqkv));
  LAT_TRY(c->alloc(&c->gu_acc, (size_t)T * 2 * F));
  LAT_TRY(c->alloc(&c->z, (size_t)T * D));
  LAT_TRY(c->alloc(&c->pm, (size_t)c->attn_split * d.Hq * T));
  LAT_TRY(c->alloc(&c->pl, (size_t)c->attn_split * d.Hq * T));
  LAT_TRY(c->alloc(&c->po, (size_t)c->attn_split * d.Hq * T * d.dh));
  LAT_TRY(c->alloc(&c->state_emb, (size_t)D));
  LAT_TRY(c->alloc(&c->planes_x, (size_t)192 * D));
  LAT_TRY(c->alloc(&c->planes_o, (size_t)192 * qd));
  LAT_TRY(c->alloc(&c->planes_h, (size_t)192 * F));
  CUDA_TRY(cudaMemset(c->planes_x, 0, (size_t)192 * D * 2));
  CUDA_TRY(cudaMemset(c->planes_o, 0, (size_t)192 * qd * 2));
  CUDA_TRY(cudaMemset(c->planes_h, 0, (size_t)192 * F * 2));
  LAT_TRY(make_planes_map(&c->bmap_x, c->planes_x, D));
  LAT_TRY(make_planes_map(&c->bmap_o, c->planes_o, qd));
  LAT_TRY(make_planes_map(&c->bmap_h, c->planes_h, F));
  // the step kernel's operands of the O / down projections: [2][64][K] fp16
  LAT_TRY(make_kmajor_map(&c->pmap_o, c->planes_o, 128, qd, 128));
  LAT_TRY(make_kmajor_map(&c->pmap_h, c->planes_h, 128, F, 128));
  LAT_TRY(c->alloc(&c->err, 1));
  CUDA_TRY(cudaMemset(c->qkv_acc, 0, (size_t)T * c->nqkv * 4));
  CUDA_TRY(cudaMemset(c->gu_acc, 0, (size_t)T * 2 * F * 4));
  CUDA_TRY(cudaMemset(c->err, 0, sizeof(DevErr)));
  CUDA_TRY(cudaMemset(c->xres, 0, (size_t)64 * D * 4));

  // --- persistent step kernel: barrier counter (cleared before every launch),
  //     key-block partials, maps, cluster plans ---
  {
    c->mk_zero_bytes = 128;
    uint8_t* z = nullptr;
    LAT_TRY(c->alloc(&z, c->mk_zero_bytes));
    CUDA_TRY(cudaMemset(z, 0, c->mk_zero_bytes));
    c->mk_zero = z;
    MkArgs& m = c->mk;
    m.bar = reinterpret_cast<unsigned*>(z);
    bf16 *qpl = nullptr, *kvo = nullptr;
    LAT_TRY(c->alloc(&qpl, (size_t)2 * 64 * qd));
    LAT_TRY(c->alloc(&kvo, (size_t)4 * 64 * kvd));
    CUDA_TRY(cudaMemset(qpl, 0, (size_t)2 * 64 * qd * 2));
    CUDA_TRY(cudaMemset(kvo, 0, (size_t)4 * 64 * kvd * 2));
    m.q_planes = qpl;
    m.kv_own = kvo;
    float *pm = nullptr, *pl = nullptr, *po = nullptr;
    LAT_TRY(c->alloc(&pm, (size_t)nkb * d.Hq * T));
    LAT_TRY(c->alloc(&pl, (size_t)nkb * d.Hq * T));
    LAT_TRY(c->alloc(&po, (size_t)nkb * d.Hq * 64 * d.dh));   // fragment order covers 64 rows
    m.part_m = pm;
    m.part_l = pl;
    m.part_o = po;
    m.x = c->xres;
    m.o_planes = reinterpret_cast<__half*>(c->planes_o);
    m.h_planes = reinterpret_cast<__half*>(c->planes_h);
    m.cos_t = c->cos_t;
    m.sin_t = c->sin_t;
    m.err = c->err;
    m.D = D;
    m.F = F;
    m.Hq = d.Hq;
    m.Hkv = d.Hkv;
    m.T_q = T;
    m.T_prefix = d.T_prefix;
    m.T_kv = T_kv;
    m.nqkv = c->nqkv;
    m.prefix_lm = d.prefix_lm;
    m.eps = d.eps;
    m.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d.dh));
    m.trace_stride = c->num_sms;
    // grid: as many clusters of 4 as are co-resident with one CTA per SM
    LAT_TRY(step_grid(c));
    const int NC = c->step_grid / kMkCluster;
    // QKV and gate/up: split-K partial sums meet in the cluster (distributed
    // shared memory) and are finalized there; O and down: every CTA adds its
    // K range's partial sums into the residual stream itself
    MkGemm& gq = m.g[0];
    gq = MkGemm{c->nqkv / 128, D / 64, c->nqkv, 0, 1, 0, 0};
    MkGemm& go = m.g[1];
    go = MkGemm{D / 128, qd / 64, D, 0, 0, 1, 0};
    go.splits = std::min(c->step_grid / go.MT, go.KT);
    MkGemm& gu = m.g[2];
    gu = MkGemm{2 * F / 128, D / 64, 2 * F, 1, 0, 0, 0};
    MkGemm& gd = m.g[3];
    gd = MkGemm{D / 128, F / 64, D, 0, 0, 1, 0};
    gd.splits = std::min(c->step_grid / gd.MT, gd.KT);
    if (gq.MT > NC || gq.KT < kMkCluster) return fail(LAT_ERR_SHAPE, "QKV tiles exceed the co-resident clusters");
    if (go.splits < 1 || gd.splits < 1) return fail(LAT_ERR_SHAPE, "O / down projections exceed the grid");
    if (gu.MT % 2 || gu.MT / 2 > NC || gu.KT < 2)
      return fail(LAT_ERR_SHAPE, "gate/up tiles (2F / 128 = %d) exceed twice the co-resident clusters (%d)",
                  gu.MT, NC);
    // a whole chunk in one launch: W2 (the embedding's second projection) adds
    // its K ranges into the residual rows like O and down; the head and the
    // embedding take one CTA per action row
    MkGemm& g2 = m.g[4];
    g2 = MkGemm{D / 128, D / 64, D, 0, 0, 1, 0};
    g2.splits = std::min(c->step_grid / g2.MT, g2.KT);
    if (g2.splits < 1) return fail(LAT_ERR_SHAPE, "W2 projection exceeds the grid");
    // the head and embedding: a pair of CTAs per action row, one for the state row
    if (2 * (T - 1) + 1 > c->step_grid)
      return fail(LAT_ERR_SHAPE, "%d action rows need %d step-kernel CTAs (%d)", T - 1, 2 * (T - 1) + 1, c->step_grid);
    if (A % 4 || 1024 % A || A > 256)
      return fail(LAT_ERR_SHAPE, "act_dim %d: the fused head needs a multiple of 4 dividing 1024", A);
    if ((size_t)D * A * 2 > (size_t)kMkXOff || (size_t)(D + 1024 + D / 2 + A + 16) * 4 > (size_t)(kMkRegion - kMkXOff))
      return fail(LAT_ERR_SHAPE, "width %d x act_dim %d: the fused head exceeds the step kernel's shared memory", D, A);
    float* ab = nullptr;
    LAT_TRY(c->alloc(&ab, (size_t)2 * (T - 1) * A));
    m.act_buf = ab;
    bf16* ep = nullptr;   // [2][64][D] fp16 planes of the embedding
    LAT_TRY(c->alloc(&ep, (size_t)2 * 64 * D));
    CUDA_TRY(cudaMemset(ep, 0, (size_t)2 * 64 * D * 2));   // row 0 (the state token) and rows >= T_q stay 0
    LAT_TRY(make_kmajor_map(&c->pmap_e, ep, 128, D, 128));
    m.e_planes = reinterpret_cast<__half*>(ep);
    m.A = A;
    m.w_state = c->w_state;
    m.b_state = c->b_state;
    m.state_emb = c->state_emb;
    m.wfold = c->wfold;
    m.ttab = c->ttab;
    m.b2 = c->b2;
    m.w_out = reinterpret_cast<const __nv_bfloat16*>(c->w_out);
    m.g_final = c->gfin;
    m.bout = c->bout;
    m.dt = c->dt;
  }

  std::vector<double> t(d.S + 1);
  for (int s = 0; s <= d.S; ++s) t[s] = (double)s / d.S;
  LAT_TRY(build_schedule(c, t));
  CUDA_TRY(cudaDeviceSynchronize());
  return LAT_OK;
}

// ---------------------------------------------------------------------------
// chunk attention: key-range partials (n_split > 1) merged by the combine kernel
// ---------------------------------------------------------------------------
static lat_status enqueue_attention(const lat_model_desc& d, const float* q, int q_ld, const bf16* k, const bf16* v,
                                    int kv_ld, int T_q, int T_kv, int n_split, float* out, int out_ld, float* pm,
                                    float* pl, float* po, cudaStream_t st, const float* k_own = nullptr,
                                    const float* v_own = nullptr, int own0 = 0) {
  AttnArgs a{};
  a.k_own = k_own; a.v_own = v_own; a.own0 = k_own ? own0 : T_kv; a.own_ld = kv_ld;
  a.q = q; a.q_ld = q_ld; a.k = k; a.v = v; a.kv_ld = kv_ld;
  a.T_q = T_q; a.T_kv = T_kv; a.Hq = d.Hq; a.Hkv = d.Hkv;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d.dh));
  a.n_split = n_split;
  a.out = out; a.out_ld = out_ld; a.part_m = pm; a.part_l = pl; a.part_o = po;
  cudaError_t e = launch_chunk_attention(a, d.dh, st);
  if (e != cudaSuccess) return fail(LAT_ERR_CUDA, "launch attention: %s", cudaGetErrorString(e));
  return LAT_OK;
}

// ---------------------------------------------------------------------------
// Persistent step kernel, one launch in clusters of 4 (cooperative: every CTA
// is resident, which the grid barriers need).  steps == 0: layers [l0, l1) of
// one denoise step on ctx->xres.  steps > 0: the whole chunk of `steps`
// denoise steps on the actions x (noise in, actions out) with the robot state.
// ---------------------------------------------------------------------------
static lat_status enqueue_pi0_step(lat_ctx* c, int l0, int l1, bf16* kv, long long kv_stride, cudaStream_t st,
                                   int steps = 0, float* x = nullptr, const float* state = nullptr) {
  CUDA_TRY(cudaMemsetAsync(c->mk_zero, 0, c->mk_zero_bytes, st));
  MkArgs a = c->mk;
  a.l0 = l0;
  a.l1 = l1;
  a.kv = kv;
  a.kv_stride = kv_stride;
  a.steps = steps;
  a.act = x;
  a.state = state;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c->step_grid);
  cfg.blockDim = dim3(kMkThreads);
  cfg.dynamicSmemBytes = mk_smem_bytes();
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kMkCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  void* args[] = {&c->map_qkv, &c->map_o, &c->map_gu, &c->map_d, &c->pmap_o, &c->pmap_h, &c->map_w2, &c->pmap_e, &a};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, step_kernel(c->d.dh, steps > 0), args);
  if (e != cudaSuccess) return fail(LAT_ERR_CUDA, "launch pi0_step: %s", cudaGetErrorString(e));
  return LAT_OK;
}

// one denoised chunk: state token, then per step the embedding, W2, every
// block and the head + Euler update, all inside one step-kernel launch
static lat_status enqueue_denoise(lat_ctx* c, bf16* kv, const float* state, float* x, cudaStream_t st) {
  const lat_model_desc& d = c->d;
  const size_t layer_elems = (size_t)2 * (d.T_prefix + d.T_q) * d.Hkv * d.dh;
  return enqueue_pi0_step(c, 0, d.L, kv, (long long)layer_elems, st, d.S, x, state);
}


// ---------------------------------------------------------------------------
// dense path: prefix prefill and DiT stage
// ---------------------------------------------------------------------------
// three pipeline slots of two activation planes + one 256-row weight tile (64 KB each)
static constexpr int kDStages = 3;

// weight of a dense projection: the four fp16 block projections, or the bf16
// patch embedding (prefix prefill, one plain bf16 activation plane)
enum WSel : int { W_QKV = 0, W_O = 1, W_UP = 2, W_DOWN = 3, W_PATCH = 4, W_CQ = 5, W_CO = 6, W_CKV = 7 };

static lat_status enqueue_dense(const lat_ctx* c, const CUtensorMap& amap, int wsel, DenseArgs a, cudaStream_t st) {
  const CUtensorMap* wm[8] = {&c->map_qkv, &c->map_o, &c->map_up, &c->map_down, &c->map_patch,
                              &c->map_cq, &c->map_co, &c->map_ckv};
  a.err = c->err;
  // DiT projections with a long epilogue (RoPE + cache stores, GELU + plane
  // split): longer chunks, so that the MMAs run on through it
  a.chunk_mma = c->d.kind == LAT_DIT && (a.epi == E_ROPE_KV || a.epi == E_GELU_SPLIT) ? kChunkMMALong : kChunkMMA;
  a.f16 = wsel != W_PATCH;
  a.out_scale = wsel != W_PATCH ? c->wscale[wsel] : 1.f;
  if (a.N % 256 || a.K % 64 || a.terms < 1 || a.terms > kActTerms) return fail(LAT_ERR_SHAPE, "dense GEMM shape");
  const int mn = ((a.M + 127) / 128) * (a.N / 256);
  // fewer output tiles than SMs (few tokens, narrow output): split K so that
  // every SM gets work, keeping at least 8 K-blocks per range; only the linear
  // epilogues can take partial sums (residual ones add into x, a plain store
  // adds into a zeroed output)
  a.ksplit = 1;
  if ((a.epi == E_RESID || a.epi == E_RESID_GATE || a.epi == E_STORE) && mn < c->num_sms)
    a.ksplit = std::max(1, std::min(c->num_sms / mn, (a.K / 64) / 8));
  if (a.ksplit > 1 && a.epi == E_STORE)
    CUDA_TRY(cudaMemsetAsync(a.out, 0, (size_t)a.M * a.ldo * sizeof(float), st));
  const int tiles = mn * a.ksplit;
  const int grid = tiles < c->num_sms ? tiles : c->num_sms;   // persistent over the tiles
  if (a.epi == E_ROPE_KV)
    dense_gemm_kernel<kDStages, kActTerms, true>
        <<<grid, kDThreads, dense_smem_bytes(kDStages, kActTerms), st>>>(amap, *wm[wsel], a);
  else
    dense_gemm_kernel<kDStages, kActTerms, false>
        <<<grid, kDThreads, dense_smem_bytes(kDStages, kActTerms), st>>>(amap, *wm[wsel], a);
  return launch_check("dense_gemm");
}

// norm prologue of M rows: one warp per row up to D = 2048, else one CTA per row
static lat_status enqueue_norm(const NormArgs& na, int M, cudaStream_t st) {
  const unsigned g = (unsigned)((M + 7) / 8);
  const int nv = (na.D + 127) / 128;   // float4 per lane
  if (nv <= 4) norm_split_warp_kernel<4><<<g, 256, 0, st>>>(na, M);
  else if (nv <= 8) norm_split_warp_kernel<8><<<g, 256, 0, st>>>(na, M);
  else if (nv <= 12) norm_split_warp_kernel<12><<<g, 256, 0, st>>>(na, M);
  else if (nv <= 16) norm_split_warp_kernel<16><<<g, 256, 0, st>>>(na, M);
  else norm_split_kernel<<<M, 256, 0, st>>>(na);
  return launch_check("norm_split");
}

// tensor map of a row-major bf16 activation [rows][cols] read in 128 x 64 tiles
static lat_status make_act_map(CUtensorMap* map, const void* base, int rows, int cols) {
  return make_kmajor_map(map, base, rows, cols, 128);
}

static lat_status build_rope_tables(lat_ctx* c, int T) {
  const lat_model_desc& d = c->d;
  const int half = d.dh / 2;
  std::vector<float> ct((size_t)T * half), stt((size_t)T * half);
  std::vector<double> th(half);
  for (int i = 0; i < half; ++i) th[i] = std::pow((double)d.rope_base, -2.0 * i / d.dh);
  for (int t = 0; t < T; ++t)
    for (int i = 0; i < half; ++i) {
      const double ang = (double)t * th[i];
      ct[(size_t)t * half + i] = (float)std::cos(ang);
      stt[(size_t)t * half + i] = (float)std::sin(ang);
    }
  LAT_TRY(c->alloc(&c->cos_j, ct.size()));
  LAT_TRY(c->alloc(&c->sin_j, stt.size()));
  LAT_TRY(c->alloc(&c->theta, th.size()));
  CUDA_TRY(cudaMemcpy(c->cos_j, ct.data(), ct.size() * 4, cudaMemcpyHostToDevice));
  CUDA_TRY(cudaMemcpy(c->sin_j, stt.data(), stt.size() * 4, cudaMemcpyHostToDevice));
  CUDA_TRY(cudaMemcpy(c->theta, th.data(), th.size() * 8, cudaMemcpyHostToDevice));
  return LAT_OK;
}

// 3-D RoPE ("frame, height, width" bands of each head; the DiT context's
// reading of Wan-class video tokens).  The kernel rotates pair (p, p + dh/2)
// of a head; the bands' own pairs (o_b + i, o_b + i + d_b/2) are put there by
// a permutation of the q and k dims (rows of the folded Wq, Wk): kernel pair p
// is band b's pair i = p - P_b, P_b = the pairs of the bands before it.
struct Rope3d {
  int off[3], width[3], pair0[4];
  explicit Rope3d(int dh) {
    const int hw = 2 * (dh / 6);
    width[0] = dh - 2 * hw;
    width[1] = width[2] = hw;
    off[0] = 0;
    off[1] = width[0];
    off[2] = width[0] + hw;
    pair0[0] = 0;
    for (int b = 0; b < 3; ++b) pair0[b + 1] = pair0[b] + width[b] / 2;
  }
  int band(int p) const { return p < pair0[1] ? 0 : p < pair0[2] ? 1 : 2; }
  // model dim of kernel dim k (< dh)
  int model_dim(int k, int dh) const {
    const int p = k < dh / 2 ? k : k - dh / 2, b = band(p), i = p - pair0[b];
    return off[b] + i + (k < dh / 2 ? 0 : width[b] / 2);
  }
};

// cos / sin of each token's angles within its chunk (frame within the chunk,
// row, column) and the per-pair frequency the chunk's frame offset turns by
// (frame band only); the kernel composes them as for 1-D RoPE
static lat_status build_rope_tables_3d(lat_ctx* c) {
  const lat_model_desc& d = c->d;
  const int half = d.dh / 2, T = d.T_q, gh = d.grid_h, gw = d.grid_w;
  const Rope3d r(d.dh);
  std::vector<float> ct((size_t)T * half), stt((size_t)T * half);
  std::vector<double> th(half), thp(half);
  for (int p = 0; p < half; ++p) {
    const int b = r.band(p), i = p - r.pair0[b];
    th[p] = std::pow((double)d.rope_base, -2.0 * i / r.width[b]);
    thp[p] = b == 0 ? th[p] : 0.0;
  }
  for (int j = 0; j < T; ++j) {
    const int coord[3] = {j / (gh * gw), (j / gw) % gh, j % gw};
    for (int p = 0; p < half; ++p) {
      const double ang = (double)coord[r.band(p)] * th[p];
      ct[(size_t)j * half + p] = (float)std::cos(ang);
      stt[(size_t)j * half + p] = (float)std::sin(ang);
    }
  }
  LAT_TRY(c->alloc(&c->cos_j, ct.size()));
  LAT_TRY(c->alloc(&c->sin_j, stt.size()));
  LAT_TRY(c->alloc(&c->theta, thp.size()));
  CUDA_TRY(cudaMemcpy(c->cos_j, ct.data(), ct.size() * 4, cudaMemcpyHostToDevice));
  CUDA_TRY(cudaMemcpy(c->sin_j, stt.data(), stt.size() * 4, cudaMemcpyHostToDevice));
  CUDA_TRY(cudaMemcpy(c->theta, thp.data(), thp.size() * 8, cudaMemcpyHostToDevice));
  c->frames_per_chunk = T / (gh * gw);
  return LAT_OK;
}

static lat_status alloc_dense_workspace(lat_ctx* c, int rows_per_group) {
  const lat_model_desc& d = c->d;
  const int qd = d.Hq * d.dh;
  c->m_max = d.max_batch * rows_per_group;
  const int terms = kActTerms;
  const int wact = d.D > qd ? d.D : qd;
  LAT_TRY(c->alloc(&c->act2, (size_t)c->m_max * terms * wact));
  LAT_TRY(c->alloc(&c->act2f, (size_t)c->m_max * terms * d.F));
  // fp32 [q | k | v] of the prefill's QKV projection; a DiT block rotates and
  // stores in the projection's epilogue, and uses it only to encode the text
  if (d.kind != LAT_DIT) LAT_TRY(c->alloc(&c->qkvbuf, (size_t)c->m_max * c->nqkv));
  else if (d.text_len > 0) LAT_TRY(c->alloc(&c->qkvbuf, (size_t)d.text_len * 2 * d.D));
  LAT_TRY(c->alloc(&c->qbuf, (size_t)c->m_max * qd));
  if (d.kind == LAT_DIT) {
    LAT_TRY(c->alloc(&c->kvown16, (size_t)c->m_max * 4 * d.Hkv * d.dh));
    LAT_TRY(c->alloc(&c->rope_rot, (size_t)(c->m_max + 31) / 32 * 1024));
    const int planes = std::max(1, 2 * d.max_batch * d.n_hist);
    if (planes > kMaxHistPlanes) return fail(LAT_ERR_SHAPE, "max_batch x n_hist must be <= %d", kMaxHistPlanes / 2);
    if ((size_t)planes * d.T_q > 0x7fffffffu) return fail(LAT_ERR_SHAPE, "history copy too large for one tensor map");
    c->hist_rows = planes * d.T_q;
    LAT_TRY(c->alloc(&c->hist16, (size_t)c->hist_rows * d.D));
    CUDA_TRY(cudaMemset(c->hist16, 0, (size_t)c->hist_rows * d.D * 2));   // rows never written stay finite
    // at most one key range per SM (enqueue_attention_seg), 128 rows x dh each
    LAT_TRY(c->alloc(&c->tc_part_o, (size_t)c->num_sms * 128 * d.dh));
    LAT_TRY(c->alloc(&c->tc_part_ml, (size_t)c->num_sms * 128 * 2));
  } else {
    LAT_TRY(c->alloc(&c->kown, (size_t)2 * c->m_max * d.Hkv * d.dh));
    LAT_TRY(c->alloc(&c->vown, (size_t)2 * c->m_max * d.Hkv * d.dh));
    LAT_TRY(c->alloc(&c->seg_part_o, (size_t)c->num_sms * 64 * d.dh));
    LAT_TRY(c->alloc(&c->seg_part_ml, (size_t)c->num_sms * 64 * 2));
  }
  LAT_TRY(make_act_map(&c->map_act_d, c->act2, c->m_max, terms * d.D));
  LAT_TRY(make_act_map(&c->map_act_o, c->act2, c->m_max, terms * qd));
  LAT_TRY(make_act_map(&c->map_act_f, c->act2f, c->m_max, terms * d.F));
  LAT_TRY(c->alloc(&c->err, 1));
  CUDA_TRY(cudaMemset(c->err, 0, sizeof(DevErr)));
  return LAT_OK;
}

static lat_status create_prefix(lat_ctx* c, const lat_weights* w) {
  const lat_model_desc& d = c->d;
  const int D = d.D, F = d.F, L = d.L;
  const int qd = d.Hq * d.dh, kvd = d.Hkv * d.dh;
  c->nqkv = qd + 2 * kvd;
  if (!w || !w->blocks) return fail(LAT_ERR_ARG, "weights / blocks NULL");
  if (!w->w_patch || !w->b_patch || !aligned16(w->w_patch) || !aligned16(w->b_patch))
    return fail(LAT_ERR_ALIGN, "patch weights NULL or not 16-byte aligned");
  for (int l = 0; l < L; ++l) {
    const lat_block_weights& b = w->blocks[l];
    const void* bp[] = {b.g_attn, b.wq, b.wk, b.wv, b.wo, b.g_ffn, b.wg, b.wu, b.wd};
    for (const void* p : bp)
      if (!p || !aligned16(p)) return fail(LAT_ERR_ALIGN, "block %d weight NULL or not 16-byte aligned", l);
  }
  LAT_TRY(c->alloc(&c->wqkv, (size_t)L * c->nqkv * D));
  LAT_TRY(c->alloc(&c->wo, (size_t)L * D * qd));
  LAT_TRY(c->alloc(&c->wup, (size_t)L * 2 * F * D));
  LAT_TRY(c->alloc(&c->wdown, (size_t)L * D * F));
  LAT_TRY(c->alloc(&c->wpatch, (size_t)D * d.patch_dim));
  for (int l = 0; l < L; ++l) {
    const lat_block_weights& b = w->blocks[l];
    bf16* q0 = c->wqkv + (size_t)l * c->nqkv * D;
    LAT_TRY(fold_t(b.wq, b.g_attn, q0, D, qd));
    LAT_TRY(fold_t(b.wk, b.g_attn, q0 + (size_t)qd * D, D, kvd));
    LAT_TRY(fold_t(b.wv, b.g_attn, q0 + (size_t)(qd + kvd) * D, D, kvd));
    LAT_TRY(fold_t(b.wo, nullptr, c->wo + (size_t)l * D * qd, qd, D));
    bf16* gu0 = c->wup + (size_t)l * 2 * F * D;   // tiles of [64 gate | 64 up] rows
    LAT_TRY(fold_t(b.wg, b.g_ffn, gu0, D, F, 64, 0));
    LAT_TRY(fold_t(b.wu, b.g_ffn, gu0, D, F, 64, 64));
    LAT_TRY(fold_t(b.wd, nullptr, c->wdown + (size_t)l * D * F, F, D));
  }
  LAT_TRY(to_f16_scaled(c->wqkv, (size_t)L * c->nqkv * D, &c->wscale[W_QKV]));
  LAT_TRY(to_f16_scaled(c->wo, (size_t)L * D * qd, &c->wscale[W_O]));
  LAT_TRY(to_f16_scaled(c->wup, (size_t)L * 2 * F * D, &c->wscale[W_UP]));
  LAT_TRY(to_f16_scaled(c->wdown, (size_t)L * D * F, &c->wscale[W_DOWN]));
  LAT_TRY(fold_t(w->w_patch, nullptr, c->wpatch, d.patch_dim, D));
  LAT_TRY(c->alloc(&c->bpatch, (size_t)D));
  bf16_to_f32_kernel<<<(D + 255) / 256, 256>>>(reinterpret_cast<const bf16*>(w->b_patch), c->bpatch, D);
  LAT_TRY(launch_check("bpatch"));
  LAT_TRY(make_kmajor_map(&c->map_qkv, c->wqkv, L * c->nqkv, D, 128));
  LAT_TRY(make_kmajor_map(&c->map_o, c->wo, L * D, qd, 128));
  LAT_TRY(make_kmajor_map(&c->map_up, c->wup, L * 2 * F, D, 128));
  LAT_TRY(make_kmajor_map(&c->map_down, c->wdown, L * D, F, 128));
  LAT_TRY(make_kmajor_map(&c->map_patch, c->wpatch, D, d.patch_dim, 128));
  LAT_TRY(c->alloc(&c->xres, (size_t)d.max_batch * d.T_prefix * D));
  LAT_TRY(alloc_dense_workspace(c, d.T_prefix));
  LAT_TRY(build_rope_tables(c, d.T_prefix));
  CUDA_TRY(cudaDeviceSynchronize());
  return LAT_OK;
}

static lat_status build_adaln(lat_ctx* c, const std::vector<double>& t) {
  const lat_model_desc& d = c->d;
  const int D = d.D, S = d.S, td = d.t_dim;
  std::vector<float> emb((size_t)S * td), tmp;
  for (int s = 0; s < S; ++s) {
    timestep_embedding_host(t[s], td, tmp);
    std::memcpy(&emb[(size_t)s * td], tmp.data(), td * sizeof(float));
  }
  // scratch owned by the context (allocated with it: a schedule change allocates nothing)
  float* e0 = c->adaln_tmp;
  float* e1 = e0 + (size_t)S * td;
  float* e2 = e1 + (size_t)S * D;
  CUDA_TRY(cudaMemcpy(e0, emb.data(), emb.size() * 4, cudaMemcpyHostToDevice));
  // e(t) = SiLU(temb Wt1 + bt1) Wt2 + bt2 ; A = SiLU(e) Wmod + bmod
  lat_status st = small_gemm(e0, false, td, c->wt1, true, D, c->bt1, true, e1, D, S, D, td, 1);
  if (st == LAT_OK) st = small_gemm(e1, false, D, c->wt2, true, D, c->bt2, true, e2, D, S, D, D, 1);
  if (st == LAT_OK) st = small_gemm(e2, false, D, c->wmod, true, 6 * D, c->bmod, true, c->adaln, 6 * D, S, 6 * D, D, 0);
  cudaError_t e = cudaDeviceSynchronize();
  if (st != LAT_OK) return st;
  if (e != cudaSuccess) return fail(LAT_ERR_CUDA, "adaLN table: %s", cudaGetErrorString(e));
  std::vector<float> dts(S);   // Euler step sizes of the latent update
  for (int s = 0; s < S; ++s) dts[s] = (float)(t[s + 1] - t[s]);
  CUDA_TRY(cudaMemcpy(c->dt, dts.data(), dts.size() * sizeof(float), cudaMemcpyHostToDevice));
  return LAT_OK;
}

static lat_status create_dit(lat_ctx* c, const lat_weights* w) {
  const lat_model_desc& d = c->d;
  const int D = d.D, F = d.F, L = d.L;
  c->nqkv = 3 * D;
  if (!w || !w->blocks) return fail(LAT_ERR_ARG, "weights / blocks NULL");
  const void* vecs[] = {w->wt1, w->bt1, w->wt2, w->bt2, w->wmod, w->bmod};
  for (const void* p : vecs)
    if (!p || !aligned16(p)) return fail(LAT_ERR_ALIGN, "timestep MLP weight NULL or not 16-byte aligned");
  for (int l = 0; l < L; ++l) {
    const lat_block_weights& b = w->blocks[l];
    const void* bp[] = {b.wq, b.wk, b.wv, b.wo, b.w1, b.w2};
    for (const void* p : bp)
      if (!p || !aligned16(p)) return fail(LAT_ERR_ALIGN, "block %d weight NULL or not 16-byte aligned", l);
  }
  LAT_TRY(c->alloc(&c->wqkv, (size_t)L * 3 * D * D));
  LAT_TRY(c->alloc(&c->wo, (size_t)L * D * D));
  LAT_TRY(c->alloc(&c->wup, (size_t)L * F * D));
  LAT_TRY(c->alloc(&c->wdown, (size_t)L * D * F));
  for (int l = 0; l < L; ++l) {
    const lat_block_weights& b = w->blocks[l];
    bf16* q0 = c->wqkv + (size_t)l * 3 * D * D;
    LAT_TRY(fold_t(b.wq, nullptr, q0, D, D));
    LAT_TRY(fold_t(b.wk, nullptr, q0 + (size_t)D * D, D, D));
    LAT_TRY(fold_t(b.wv, nullptr, q0 + (size_t)2 * D * D, D, D));
    LAT_TRY(fold_t(b.wo, nullptr, c->wo + (size_t)l * D * D, D, D));
    LAT_TRY(fold_t(b.w1, nullptr, c->wup + (size_t)l * F * D, D, F));
    LAT_TRY(fold_t(b.w2, nullptr, c->wdown + (size_t)l * D * F, F, D));
  }
  if (d.grid_h > 0) {   // 3-D RoPE: each head's q and k dims in band-pair order (rows of Wq, Wk)
    const Rope3d r(d.dh);
    std::vector<int> perm((size_t)3 * D);
    for (int row = 0; row < 3 * D; ++row) {
      const int part = row / D, h = (row % D) / d.dh, k = row % d.dh;
      perm[row] = part < 2 ? part * D + h * d.dh + r.model_dim(k, d.dh) : row;
    }
    int* dperm = nullptr;
    bf16* tmp = nullptr;
    CUDA_TRY(cudaMalloc(&dperm, perm.size() * sizeof(int)));
    cudaError_t e = cudaMalloc(&tmp, (size_t)3 * D * D * sizeof(bf16));
    if (e == cudaSuccess) e = cudaMemcpy(dperm, perm.data(), perm.size() * sizeof(int), cudaMemcpyHostToDevice);
    for (int l = 0; l < L && e == cudaSuccess; ++l) {
      bf16* q0 = c->wqkv + (size_t)l * 3 * D * D;
      e = cudaMemcpy(tmp, q0, (size_t)3 * D * D * sizeof(bf16), cudaMemcpyDeviceToDevice);
      if (e == cudaSuccess) {
        gather_rows_kernel<<<3 * D, 256>>>(tmp, dperm, q0, 3 * D, D);
        e = cudaGetLastError();
      }
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    cudaFree(dperm);
    cudaFree(tmp);
    if (e != cudaSuccess) return fail(LAT_ERR_CUDA, "3-D RoPE weight permutation: %s", cudaGetErrorString(e));
  }
  if (d.text_len > 0) {   // cross-attention: q, o and the context's k | v, folded like the block's
    LAT_TRY(c->alloc(&c->wcq, (size_t)L * D * D));
    LAT_TRY(c->alloc(&c->wco, (size_t)L * D * D));
    LAT_TRY(c->alloc(&c->wckv, (size_t)L * 2 * D * D));
    LAT_TRY(c->alloc(&c->cross_ln, (size_t)L * 2 * D));
    std::vector<uint16_t> gb(2 * (size_t)D);
    std::vector<float> ln((size_t)L * 2 * D);
    for (int l = 0; l < L; ++l) {
      const lat_block_weights& b = w->blocks[l];
      const void* cp[] = {b.g_cross, b.b_cross, b.cq, b.ck, b.cv, b.co};
      for (const void* p : cp)
        if (!p || !aligned16(p)) return fail(LAT_ERR_ALIGN, "block %d cross-attention weight NULL or not 16-byte aligned", l);
      LAT_TRY(fold_t(b.cq, nullptr, c->wcq + (size_t)l * D * D, D, D));
      LAT_TRY(fold_t(b.co, nullptr, c->wco + (size_t)l * D * D, D, D));
      LAT_TRY(fold_t(b.ck, nullptr, c->wckv + (size_t)l * 2 * D * D, D, D));
      LAT_TRY(fold_t(b.cv, nullptr, c->wckv + (size_t)l * 2 * D * D + (size_t)D * D, D, D));
      CUDA_TRY(cudaMemcpy(gb.data(), b.b_cross, (size_t)D * 2, cudaMemcpyDeviceToHost));
      CUDA_TRY(cudaMemcpy(gb.data() + D, b.g_cross, (size_t)D * 2, cudaMemcpyDeviceToHost));
      for (int i = 0; i < D; ++i) {
        ln[(size_t)l * 2 * D + i] = bf16_bits_to_float(gb[i]);                 // shift = b
        ln[(size_t)l * 2 * D + D + i] = bf16_bits_to_float(gb[D + i]) - 1.f;   // scale = g - 1 (exact)
      }
    }
    CUDA_TRY(cudaMemcpy(c->cross_ln, ln.data(), ln.size() * 4, cudaMemcpyHostToDevice));
    LAT_TRY(to_f16_scaled(c->wcq, (size_t)L * D * D, &c->wscale[W_CQ]));
    LAT_TRY(to_f16_scaled(c->wco, (size_t)L * D * D, &c->wscale[W_CO]));
    LAT_TRY(to_f16_scaled(c->wckv, (size_t)L * 2 * D * D, &c->wscale[W_CKV]));
    LAT_TRY(make_kmajor_map(&c->map_cq, c->wcq, L * D, D, 128));
    LAT_TRY(make_kmajor_map(&c->map_co, c->wco, L * D, D, 128));
    LAT_TRY(make_kmajor_map(&c->map_ckv, c->wckv, L * 2 * D, D, 128));
    LAT_TRY(c->alloc(&c->text_kv, (size_t)d.n_streams * L * d.text_len * 4 * D));
    c->text_set.assign(d.n_streams, 0);
  }
  c->pages_per_ring = ring_pages(d);
  LAT_TRY(to_f16_scaled(c->wqkv, (size_t)L * 3 * D * D, &c->wscale[W_QKV]));
  LAT_TRY(to_f16_scaled(c->wo, (size_t)L * D * D, &c->wscale[W_O]));
  LAT_TRY(to_f16_scaled(c->wup, (size_t)L * F * D, &c->wscale[W_UP]));
  LAT_TRY(to_f16_scaled(c->wdown, (size_t)L * D * F, &c->wscale[W_DOWN]));
  LAT_TRY(make_kmajor_map(&c->map_qkv, c->wqkv, L * 3 * D, D, 128));
  LAT_TRY(make_kmajor_map(&c->map_o, c->wo, L * D, D, 128));
  LAT_TRY(make_kmajor_map(&c->map_up, c->wup, L * F, D, 128));
  LAT_TRY(make_kmajor_map(&c->map_down, c->wdown, L * D, F, 128));
  // timestep MLP weights are kept for schedule changes
  const int td = d.t_dim;
  LAT_TRY(c->alloc(&c->wt1, (size_t)td * D));
  LAT_TRY(c->alloc(&c->bt1, (size_t)D));
  LAT_TRY(c->alloc(&c->wt2, (size_t)D * D));
  LAT_TRY(c->alloc(&c->bt2, (size_t)D));
  LAT_TRY(c->alloc(&c->wmod, (size_t)D * 6 * D));
  LAT_TRY(c->alloc(&c->bmod, (size_t)6 * D));
  CUDA_TRY(cudaMemcpy(c->wt1, w->wt1, (size_t)td * D * 2, cudaMemcpyDeviceToDevice));
  CUDA_TRY(cudaMemcpy(c->bt1, w->bt1, (size_t)D * 2, cudaMemcpyDeviceToDevice));
  CUDA_TRY(cudaMemcpy(c->wt2, w->wt2, (size_t)D * D * 2, cudaMemcpyDeviceToDevice));
  CUDA_TRY(cudaMemcpy(c->bt2, w->bt2, (size_t)D * 2, cudaMemcpyDeviceToDevice));
  CUDA_TRY(cudaMemcpy(c->wmod, w->wmod, (size_t)D * 6 * D * 2, cudaMemcpyDeviceToDevice));
  CUDA_TRY(cudaMemcpy(c->bmod, w->bmod, (size_t)6 * D * 2, cudaMemcpyDeviceToDevice));
  LAT_TRY(c->alloc(&c->adaln, (size_t)d.S * 6 * D));
  LAT_TRY(c->alloc(&c->adaln_tmp, (size_t)d.S * (td + 2 * D)));
  LAT_TRY(c->alloc(&c->dt, (size_t)d.S));
  std::vector<double> t(d.S + 1);
  for (int s = 0; s <= d.S; ++s) t[s] = (double)s / d.S;
  LAT_TRY(build_adaln(c, t));
  LAT_TRY(alloc_dense_workspace(c, d.T_q));
  if (d.act_dim > 0) {   // latent in/out projections (kept as bf16 [K][N]) and the schedule's state
    const int A = d.act_dim;
    const void* io[] = {w->w_in, w->b_in, w->w_out, w->b_out};
    for (const void* p : io)
      if (!p || !aligned16(p)) return fail(LAT_ERR_ALIGN, "latent in/out weight NULL or not 16-byte aligned");
    LAT_TRY(c->alloc(&c->wlin, (size_t)A * D));
    LAT_TRY(c->alloc(&c->blin, (size_t)D));
    LAT_TRY(c->alloc(&c->wlout, (size_t)D * A));
    LAT_TRY(c->alloc(&c->blout, (size_t)A));
    CUDA_TRY(cudaMemcpy(c->wlin, w->w_in, (size_t)A * D * 2, cudaMemcpyDeviceToDevice));
    CUDA_TRY(cudaMemcpy(c->blin, w->b_in, (size_t)D * 2, cudaMemcpyDeviceToDevice));
    CUDA_TRY(cudaMemcpy(c->wlout, w->w_out, (size_t)D * A * 2, cudaMemcpyDeviceToDevice));
    CUDA_TRY(cudaMemcpy(c->blout, w->b_out, (size_t)A * 2, cudaMemcpyDeviceToDevice));
    LAT_TRY(c->alloc(&c->dit_x, (size_t)c->m_max * D));
    LAT_TRY(c->alloc(&c->dit_z, (size_t)c->m_max * A));
    LAT_TRY(c->alloc(&c->dit_v, (size_t)c->m_max * A));
    LAT_TRY(c->alloc(&c->pipe_lat, (size_t)d.n_streams * d.S * d.T_q * A));
    c->pipe_next.assign(d.n_streams, 0);
    c->pipe_done.assign(d.n_streams, 0);
    c->pipe_step.assign((size_t)d.n_streams * d.S, 0);
  }
  if (d.grid_h > 0) LAT_TRY(build_rope_tables_3d(c));
  else LAT_TRY(build_rope_tables(c, d.T_q));
  CUDA_TRY(cudaDeviceSynchronize());
  return LAT_OK;
}

static lat_status enqueue_attention_seg(const lat_ctx* c, const SegAttnArgs& a, int groups, cudaStream_t st) {
  const int dh = c->d.dh;
  if (dh == 128) {   // tensor-core attention: one CTA per (128 rows, head, group)
    const lat_model_desc& d = c->d;
    if (!a.hist16 || !a.own16) return fail(LAT_ERR_STATE, "tensor-core attention needs the fp16 history copy");
    CUtensorMap ring_map, own_map;
    LAT_TRY(make_kmajor_map(&ring_map, a.hist16, a.hist_rows, a.kv_ld, 128));
    LAT_TRY(make_kmajor_map(&own_map, a.own16, a.own_rows > 0 ? a.own_rows : c->m_max, 4 * a.kv_ld, 64));
    // One CTA per SM (TMEM), so the tiles run in waves of num_sms.  The tiles
    // of a last, partly filled wave are cut into key ranges of at least
    // kTcMinRangeBlocks blocks, as many per tile as fill the SMs once, and a
    // combine kernel merges them: the tail takes a fraction of a whole tile's
    // time instead of all of it.
    const int nqt = (a.T_rows + 127) / 128, tiles = nqt * d.Hq * groups;
    SegAttnArgs b = a;
    b.tc_whole = tiles;
    b.tc_pieces = 1;
    b.tc_part_o = c->tc_part_o;
    b.tc_part_ml = c->tc_part_ml;
    const int tail = tiles % c->num_sms;
    if (tail > 0 && c->tc_part_o) {
      int nblk_min = INT_MAX;   // key blocks of each group, counted as the kernel does
      for (int g = 0; g < groups; ++g) {
        int nb = 0;
        for (int s = 0; s < a.grp[g].nseg; ++s) {
          const AttnSeg& sg = a.grp[g].seg[s];
          nb += sg.k16 ? (sg.n + kTcKBO - 1) / kTcKBO : (sg.n + kTcKB - 1) / kTcKB;
        }
        nblk_min = std::min(nblk_min, nb);
      }
      const int pieces = std::min(c->num_sms / tail, nblk_min / kTcMinRangeBlocks);
      if (pieces >= 2) {   // tail * pieces <= num_sms: fits the scratch
        b.tc_whole = tiles - tail;
        b.tc_pieces = pieces;
      }
    }
    const int items = b.tc_whole + (tiles - b.tc_whole) * b.tc_pieces;
    attention_tc_kernel<<<items, kTcThreads, attn_tc_smem_bytes(), st>>>(b, ring_map, own_map, c->err);
    LAT_TRY(launch_check("attention_tc"));
    if (b.tc_pieces > 1) {
      attention_tc_combine_kernel<<<dim3(tiles - b.tc_whole, 128), 128, 0, st>>>(b);
      LAT_TRY(launch_check("attention_tc_combine"));
    }
    return LAT_OK;
  }
  if (dh != 256) return fail(LAT_ERR_SHAPE, "dense-path attention: dh 128 or 256");
  // fewer CTAs than SMs (few groups): split the keys into ranges (at least two
  // 64-key blocks each), merged by the combine kernel
  SegAttnArgs b = a;
  const int ctas = c->d.Hq * ((a.T_rows + 63) / 64) * groups;
  int nkb_max = 1;
  for (int g = 0; g < groups; ++g)
    for (int s = 0; s < a.grp[g].nseg; ++s) nkb_max = std::max(nkb_max, (a.grp[g].seg[s].n + 63) / 64);
  b.kv_split = 1;
  if (ctas < c->num_sms && c->seg_part_o)
    b.kv_split = std::max(1, std::min(std::min(4, c->num_sms / ctas), nkb_max / 2));
  b.part_o = c->seg_part_o;
  b.part_ml = c->seg_part_ml;
  dim3 grid(c->d.Hq, (a.T_rows + 63) / 64, groups * b.kv_split);
  if ((long long)grid.x * grid.y * grid.z > c->num_sms)   // two CTAs a SM: 16-key blocks
    attention_seg_kernel<256, 16><<<grid, 128, seg_attn_smem_bytes(dh, 16), st>>>(b);
  else
    attention_seg_kernel<256, 32><<<grid, 128, seg_attn_smem_bytes(dh, 32), st>>>(b);
  LAT_TRY(launch_check("attention_seg"));
  if (b.kv_split > 1) {
    attention_seg_combine_kernel<<<dim3(a.T_rows, c->d.Hq, groups), dh, 0, st>>>(b, dh);
    LAT_TRY(launch_check("attention_seg_combine"));
  }
  return LAT_OK;
}

static lat_status enqueue_prefill(lat_ctx* c, const bf16* pe, int B, bf16* kv, cudaStream_t st) {
  const lat_model_desc& d = c->d;
  const int D = d.D, F = d.F, L = d.L, T = d.T_prefix, M = B * T;
  const int qd = d.Hq * d.dh, kvd = d.Hkv * d.dh, T_kv = d.T_prefix + d.T_q;
  CUtensorMap pmap;
  LAT_TRY(make_act_map(&pmap, pe, M, d.patch_dim));
  {  // patch projection
    DenseArgs a{};
    a.M = M; a.N = D; a.K = d.patch_dim; a.terms = 1; a.w_row0 = 0; a.epi = E_STORE;
    a.out = c->xres; a.ldo = D; a.bias = c->bpatch;
    LAT_TRY(enqueue_dense(c, pmap, W_PATCH, a, st));
  }
  for (int l = 0; l < L; ++l) {
    const bool last = (l == L - 1);
    NormArgs na{};
    na.x = c->xres; na.D = D; na.mode = NORM_RMS; na.eps = d.eps; na.act2 = c->act2;
    LAT_TRY(enqueue_norm(na, M, st));
    {
      DenseArgs a{};
      a.M = M; a.K = D; a.terms = c->act_terms; a.epi = E_STORE; a.out = c->qkvbuf;
      if (last) { a.N = 2 * kvd; a.w_row0 = l * c->nqkv + qd; a.ldo = 2 * kvd; }
      else { a.N = c->nqkv; a.w_row0 = l * c->nqkv; a.ldo = c->nqkv; }
      LAT_TRY(enqueue_dense(c, c->map_act_d, W_QKV, a, st));
    }
    RopeKvArgs ra{};
    ra.qkv = c->qkvbuf; ra.ld_qkv = last ? 2 * kvd : c->nqkv; ra.q_cols = last ? 0 : qd; ra.kv_cols = kvd;
    ra.dh = d.dh; ra.T = T; ra.cos_j = c->cos_j; ra.sin_j = c->sin_j; ra.theta = c->theta;
    ra.q_out = c->qbuf; ra.kv_ld = kvd; ra.kb2 = c->kown; ra.vb2 = c->vown;
    ra.lo_off = (long long)c->m_max * kvd;
    SegAttnArgs sa{};
    for (int b = 0; b < B; ++b) {
      bf16* kb = kv + (((size_t)l * B + b) * 2 + 0) * T_kv * kvd;
      ra.pos0[b] = 0;
      ra.kdst[b] = kb;
      ra.vdst[b] = kb + (size_t)T_kv * kvd;
      sa.grp[b].nseg = 1;   // the prefix tokens attend to their own K/V as computed
      AttnSeg sg{nullptr, nullptr, c->kown + (size_t)b * T * kvd, c->vown + (size_t)b * T * kvd, T};
      sg.lo_off = (long long)c->m_max * kvd;
      sa.grp[b].seg[0] = sg;
    }
    rope_kv_kernel<<<M, 128, 0, st>>>(ra);
    LAT_TRY(launch_check("rope_kv"));
    if (last) break;   // the last layer only needs its K and V
    sa.q = c->qbuf; sa.q_ld = qd; sa.T_rows = T; sa.Hq = d.Hq; sa.Hkv = d.Hkv; sa.kv_ld = kvd;
    sa.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d.dh));
    sa.out = c->act2; sa.ldh = qd;
    LAT_TRY(enqueue_attention_seg(c, sa, B, st));
    {
      DenseArgs a{};
      a.M = M; a.N = D; a.K = qd; a.terms = c->act_terms; a.w_row0 = l * D; a.epi = E_RESID; a.out = c->xres; a.ldo = D;
      LAT_TRY(enqueue_dense(c, c->map_act_o, W_O, a, st));
    }
    LAT_TRY(enqueue_norm(na, M, st));
    {
      DenseArgs a{};
      a.M = M; a.N = 2 * F; a.K = D; a.terms = c->act_terms; a.w_row0 = l * 2 * F; a.epi = E_GEGLU_SPLIT;
      a.act2 = c->act2f; a.ldh = F;
      LAT_TRY(enqueue_dense(c, c->map_act_d, W_UP, a, st));
    }
    {
      DenseArgs a{};
      a.M = M; a.N = D; a.K = F; a.terms = c->act_terms; a.w_row0 = l * D; a.epi = E_RESID; a.out = c->xres; a.ldo = D;
      LAT_TRY(enqueue_dense(c, c->map_act_f, W_DOWN, a, st));
    }
  }
  return LAT_OK;
}

static bf16* ring_ptr(const lat_ctx* c, bf16* kv, int stream, int layer, int step, int slot, int plane) {
  const lat_model_desc& d = c->d;
  const size_t R = d.n_hist + 1;
  const size_t idx = ((((size_t)stream * d.L + layer) * d.S + step) * R + slot) * 2 + plane;
  return kv + idx * d.T_q * d.D;
}

// One DiT block on a batch of chunks: adaLN norm, QKV, RoPE (1-D or 3-D) with
// the own K/V into the ring (or its pages), the history's fp16 copy, attention,
// O (x gate); with text_len > 0 the text cross-attention sublayer; the FFN.
static lat_status enqueue_dit_block(lat_ctx* c, int l, float* x, const lat_chunk_desc* ch, int n, bf16* kv,
                                    cudaStream_t st) {
  const lat_model_desc& d = c->d;
  const int D = d.D, F = d.F, T = d.T_q, M = n * T;
  const int R = d.n_hist + 1, P = d.page_tokens;
  NormArgs na{};
  na.x = x; na.D = D; na.mode = NORM_LN_MOD; na.eps = d.eps; na.table = c->adaln; na.rows_per_chunk = T;
  na.act2 = c->act2;
  for (int b = 0; b < n; ++b) {
    na.shift_off[b] = ch[b].step * 6 * D + 0 * D;
    na.scale_off[b] = ch[b].step * 6 * D + 1 * D;
  }
  LAT_TRY(enqueue_norm(na, M, st));
  // the QKV projection turns q and k and stores q, the ring rows and the fp16
  // planes of the own K / V in its epilogue, from each row's rotation
  RopeRowsArgs rr{};
  rr.M = M; rr.T = T; rr.n = n; rr.cos_j = c->cos_j; rr.sin_j = c->sin_j; rr.theta = c->theta; rr.rot = c->rope_rot;
  DenseArgs qa{};
  qa.M = M; qa.N = 3 * D; qa.K = D; qa.terms = c->act_terms; qa.w_row0 = l * 3 * D; qa.epi = E_ROPE_KV;
  RopeEpi& ra = qa.rope;
  ra.rot = c->rope_rot; ra.heads = d.Hq; ra.T = T; ra.q_out = c->qbuf; ra.own16 = c->kvown16;
  ra.ring.ld = D;
  if (P > 0) {
    ra.ring.page_tokens = P;
    ra.ring.pool = kv;
  }
  // the page list of ring (stream, layer, step)
  auto pages = [&](int stream, int step) {
    return c->page_table + (((size_t)stream * d.L + l) * d.S + step) * c->pages_per_ring;
  };
  SegAttnArgs sa{};
  HistCvtArgs hc{};   // every distinct history segment of the call, once, into the fp16 copy
  hc.rows = T;
  hc.cols = D;
  if (P > 0) {
    hc.page_tokens = P;
    hc.pool = kv;
  }
  long long hkey[kMaxHistPlanes / 2];   // (stream, step, slot) of each copied segment
  for (int b = 0; b < n; ++b) {
    const int cb = ch[b].chunk, sb = ch[b].step, stb = ch[b].stream;
    rr.pos0[b] = d.grid_h > 0 ? (long long)cb * c->frames_per_chunk : chunk_pos0(cb, T);
    if (P > 0) {
      ra.ring.ptab[b] = pages(stb, sb);
      ra.ring.row0[b] = ring_slot_of(cb, d.n_hist) * T;
    } else {
      ra.ring.kdst[b] = ring_ptr(c, kv, stb, l, sb, ring_slot_of(cb, d.n_hist), 0);
      ra.ring.vdst[b] = ring_ptr(c, kv, stb, l, sb, ring_slot_of(cb, d.n_hist), 1);
    }
    int ns = 0;
    for (int k = d.n_hist; k >= 1; --k) {       // history, oldest first
      const int cc = cb - k;
      if (cc < 0) continue;
      const int slot = ring_slot_of(cc, d.n_hist);
      const long long key = ((long long)stb * d.S + sb) * R + slot;
      int q = 0;
      while (2 * q < hc.planes && hkey[q] != key) ++q;
      if (2 * q == hc.planes) {
        if (2 * q + 2 > kMaxHistPlanes || (2 * q + 2) * T > c->hist_rows)
          return fail(LAT_ERR_SHAPE, "history copy overflow");
        hkey[q] = key;
        if (P > 0) {
          hc.ptab[q] = pages(stb, sb);
          hc.row0[q] = slot * T;
        } else {
          hc.src[2 * q] = ring_ptr(c, kv, stb, l, sb, slot, 0);
          hc.src[2 * q + 1] = ring_ptr(c, kv, stb, l, sb, slot, 1);
        }
        hc.dst[2 * q] = c->hist16 + (size_t)(2 * q) * T * D;
        hc.dst[2 * q + 1] = c->hist16 + (size_t)(2 * q + 1) * T * D;
        hc.planes = 2 * q + 2;
      }
      AttnSeg sg{nullptr, nullptr, nullptr, nullptr, T};
      sg.kh = hc.dst[2 * q];
      sg.vh = hc.dst[2 * q + 1];
      sa.grp[b].seg[ns++] = sg;
    }
    // own keys as computed (fp16 hi/lo planes of the fp32 values); the ring slot holds their bf16 copy
    const __half* own = c->kvown16 + (size_t)b * T * 4 * D;
    sa.grp[b].seg[ns++] = AttnSeg{nullptr, nullptr, nullptr, nullptr, T, own, own + 2 * D};
    sa.grp[b].nseg = ns;
  }
  rope_rows_kernel<<<(M + 31) / 32, 256, 0, st>>>(rr);
  LAT_TRY(launch_check("rope_rows"));
  LAT_TRY(enqueue_dense(c, c->map_act_d, W_QKV, qa, st));
  if (hc.planes > 0) {   // after the ring rows are written: a chunk of this call may be another's history
    // contiguous: 256 chunks of 8 values a CTA; pages: one warp per (plane, row), 8 a CTA
    const size_t work = P > 0 ? ((size_t)hc.planes * T + 7) / 8 : ((size_t)hc.planes * T * D / 8 + 255) / 256;
    const unsigned grid = (unsigned)std::min<size_t>(work, (size_t)c->num_sms * 8);
    hist_to_f16_kernel<<<grid, 256, 0, st>>>(hc);
    LAT_TRY(launch_check("hist_to_f16"));
  }
  sa.q = c->qbuf; sa.q_ld = D; sa.T_rows = T; sa.Hq = d.Hq; sa.Hkv = d.Hkv; sa.kv_ld = D;
  sa.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d.dh));
  sa.out = c->act2; sa.ldh = D;
  sa.trace = c->attn_trace;
  sa.hist16 = c->hist16; sa.hist_rows = c->hist_rows; sa.own16 = c->kvown16;
  LAT_TRY(enqueue_attention_seg(c, sa, n, st));
  {
    DenseArgs a{};
    a.M = M; a.N = D; a.K = D; a.terms = c->act_terms; a.w_row0 = l * D; a.epi = E_RESID_GATE; a.out = x; a.ldo = D;
    a.gate = c->adaln; a.rows_per_chunk = T;
    for (int b = 0; b < n; ++b) a.gate_off[b] = ch[b].step * 6 * D + 2 * D;
    LAT_TRY(enqueue_dense(c, c->map_act_o, W_O, a, st));
  }
  if (d.text_len > 0) {   // x += Attn(LN(x) g + b, text) Wo^c: q from x, the stream's K/V of the text
    NormArgs nc = na;
    for (int b = 0; b < n; ++b) {
      nc.shift_off[b] = l * 2 * D;
      nc.scale_off[b] = l * 2 * D + D;
    }
    nc.table = c->cross_ln;
    LAT_TRY(enqueue_norm(nc, M, st));
    {
      DenseArgs a{};
      a.M = M; a.N = D; a.K = D; a.terms = c->act_terms; a.w_row0 = l * D; a.epi = E_STORE; a.out = c->qbuf;
      a.ldo = D;
      LAT_TRY(enqueue_dense(c, c->map_act_d, W_CQ, a, st));
    }
    SegAttnArgs ca = sa;
    for (int b = 0; b < n; ++b) {
      const __half* tk = c->text_kv + ((size_t)ch[b].stream * d.L + l) * d.text_len * 4 * D;
      ca.grp[b].nseg = 1;
      ca.grp[b].seg[0] = AttnSeg{nullptr, nullptr, nullptr, nullptr, d.text_len, tk, tk + 2 * D};
    }
    ca.own16 = c->text_kv;
    ca.own_rows = d.n_streams * d.L * d.text_len;
    ca.trace = nullptr;
    LAT_TRY(enqueue_attention_seg(c, ca, n, st));
    DenseArgs a{};
    a.M = M; a.N = D; a.K = D; a.terms = c->act_terms; a.w_row0 = l * D; a.epi = E_RESID; a.out = x; a.ldo = D;
    LAT_TRY(enqueue_dense(c, c->map_act_o, W_CO, a, st));
  }
  for (int b = 0; b < n; ++b) {
    na.shift_off[b] = ch[b].step * 6 * D + 3 * D;
    na.scale_off[b] = ch[b].step * 6 * D + 4 * D;
  }
  LAT_TRY(enqueue_norm(na, M, st));
  {
    DenseArgs a{};
    a.M = M; a.N = F; a.K = D; a.terms = c->act_terms; a.w_row0 = l * F; a.epi = E_GELU_SPLIT; a.act2 = c->act2f; a.ldh = F;
    LAT_TRY(enqueue_dense(c, c->map_act_d, W_UP, a, st));
  }
  {
    DenseArgs a{};
    a.M = M; a.N = D; a.K = F; a.terms = c->act_terms; a.w_row0 = l * D; a.epi = E_RESID_GATE; a.out = x; a.ldo = D;
    a.gate = c->adaln; a.rows_per_chunk = T;
    for (int b = 0; b < n; ++b) a.gate_off[b] = ch[b].step * 6 * D + 5 * D;
    LAT_TRY(enqueue_dense(c, c->map_act_f, W_DOWN, a, st));
  }
  return LAT_OK;
}

// One interval of the interleaved stage schedule for n chunks whose latents
// sit at the device addresses lat[b] (gathered into one buffer for the
// projections): x = z W_in + b_in, the L blocks, v = x W_out + b_out,
// z += dt[step] v, scattered back.
static lat_status enqueue_dit_interval(lat_ctx* c, bf16* kv, float* const* lat, const lat_chunk_desc* ch, int n,
                                       cudaStream_t st) {
  const lat_model_desc& d = c->d;
  const int T = d.T_q, A = d.act_dim, D = d.D, M = n * T;
  const size_t zb = (size_t)T * A * 4;
  for (int b = 0; b < n; ++b)
    if (lat[b] != c->dit_z + (size_t)b * T * A)
      CUDA_TRY(cudaMemcpyAsync(c->dit_z + (size_t)b * T * A, lat[b], zb, cudaMemcpyDeviceToDevice, st));
  LAT_TRY(small_gemm(c->dit_z, false, A, c->wlin, true, D, c->blin, true, c->dit_x, D, M, D, A, 0, st));
  for (int l = 0; l < d.L; ++l) LAT_TRY(enqueue_dit_block(c, l, c->dit_x, ch, n, kv, st));
  LAT_TRY(small_gemm(c->dit_x, false, D, c->wlout, true, A, c->blout, true, c->dit_v, A, M, A, D, 0, st));
  DitEulerArgs e{};
  e.z = c->dit_z;
  e.v = c->dit_v;
  e.dt = c->dt;
  for (int b = 0; b < n; ++b) e.step[b] = ch[b].step;
  e.T = T;
  e.A = A;
  e.n = n;
  const size_t total = (size_t)M * A;
  dit_euler_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(e);
  LAT_TRY(launch_check("dit_euler"));
  for (int b = 0; b < n; ++b)
    if (lat[b] != c->dit_z + (size_t)b * T * A)
      CUDA_TRY(cudaMemcpyAsync(lat[b], c->dit_z + (size_t)b * T * A, zb, cudaMemcpyDeviceToDevice, st));
  return LAT_OK;
}

// ---------------------------------------------------------------------------
// ABI
// ---------------------------------------------------------------------------
extern "C" {

const char* lat_status_str(lat_status s) {
  switch (s) {
    case LAT_OK: return "LAT_OK";
    case LAT_ERR_ARG: return "LAT_ERR_ARG";
    case LAT_ERR_SHAPE: return "LAT_ERR_SHAPE";
    case LAT_ERR_ALIGN: return "LAT_ERR_ALIGN";
    case LAT_ERR_CUDA: return "LAT_ERR_CUDA";
    case LAT_ERR_OOM: return "LAT_ERR_OOM";
    case LAT_ERR_TIMEOUT: return "LAT_ERR_TIMEOUT";
    case LAT_ERR_RANGE: return "LAT_ERR_RANGE";
    case LAT_ERR_STATE: return "LAT_ERR_STATE";
    case LAT_ERR_UNSUPPORTED: return "LAT_ERR_UNSUPPORTED";
  }
  return "LAT_ERR_?";
}

const char* lat_last_error(void) { return g_last_error.c_str(); }

lat_status lat_create(const lat_model_desc* desc, const lat_weights* w, lat_ctx** out) {
  if (!out) return fail(LAT_ERR_ARG, "out is NULL");
  *out = nullptr;
  LAT_TRY(check_desc(desc));
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  CUDA_TRY(cudaGetDeviceProperties(&prop, dev));
  if (prop.major != 10 || prop.minor != 3)
    return fail(LAT_ERR_UNSUPPORTED, "needs an sm_103 device, found sm_%d%d", prop.major, prop.minor);
  lat_ctx* c = new lat_ctx();
  c->d = *desc;
  c->num_sms = prop.multiProcessorCount;
  static bool attr_done = false;
  if (!attr_done) {
    cudaFuncSetAttribute(skinny_gemm_kernel<kStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         skinny_smem_bytes(kStages));
    set_attention_smem_limits();
    for (auto k : {dense_gemm_kernel<kDStages, kActTerms, false>, dense_gemm_kernel<kDStages, kActTerms, true>})
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dense_smem_bytes(kDStages, kActTerms));
    cudaFuncSetAttribute(attention_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, attn_tc_smem_bytes());
    for (int dh : {64, 128, 256})
      for (bool chunk : {false, true})
        cudaFuncSetAttribute(step_kernel(dh, chunk), cudaFuncAttributeMaxDynamicSharedMemorySize, mk_smem_bytes());
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
      delete c;
      return fail(LAT_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    }
    attr_done = true;
  }
  lat_status s = desc->kind == LAT_PI0_ACTION_EXPERT ? create_pi0(c, w)
                 : desc->kind == LAT_PI0_PREFIX        ? create_prefix(c, w)
                                                       : create_dit(c, w);
  if (s != LAT_OK) {
    std::string msg = g_last_error;
    cudaDeviceSynchronize();
    delete c;
    g_last_error = msg;
    return s;
  }
  *out = c;
  return LAT_OK;
}

lat_status lat_set_schedule(lat_ctx* c, const float* t, int n) {
  if (!c || !t) return fail(LAT_ERR_ARG, "NULL argument");
  if (n != c->d.S + 1) return fail(LAT_ERR_SHAPE, "schedule needs S + 1 = %d values", c->d.S + 1);
  for (int i = 0; i < c->d.S; ++i)
    if (!(t[i + 1] > t[i])) return fail(LAT_ERR_ARG, "schedule must be increasing");
  std::vector<double> tt(t, t + n);
  CUDA_TRY(cudaDeviceSynchronize());
  if (c->d.kind == LAT_DIT) return build_adaln(c, tt);
  if (c->d.kind != LAT_PI0_ACTION_EXPERT) return fail(LAT_ERR_STATE, "the prefix model has no schedule");
  return build_schedule(c, tt);
}

lat_status lat_prefill_kv(lat_ctx* c, const void* patch_emb, int B, void* kv, void* stream) {
  if (!c || !patch_emb || !kv) return fail(LAT_ERR_ARG, "NULL argument");
  if (c->d.kind != LAT_PI0_PREFIX) return fail(LAT_ERR_STATE, "lat_prefill_kv needs a LAT_PI0_PREFIX context");
  if (B < 1 || B > c->d.max_batch) return fail(LAT_ERR_SHAPE, "B = %d outside [1, max_batch = %d]", B, c->d.max_batch);
  if (!aligned16(patch_emb) || !aligned16(kv)) return fail(LAT_ERR_ALIGN, "pointer not 16-byte aligned");
  return enqueue_prefill(c, reinterpret_cast<const bf16*>(patch_emb), B, reinterpret_cast<bf16*>(kv),
                         reinterpret_cast<cudaStream_t>(stream));
}

static lat_status check_dev_err(lat_ctx* c) {
  DevErr e{};
  CUDA_TRY(cudaMemcpy(&e, c->err, sizeof(e), cudaMemcpyDeviceToHost));
  if (e.code & kErrLaunch)
    return fail(LAT_ERR_CUDA, "the step kernel ran without its clusters of %d CTAs (site %u)", kMkCluster, e.where);
  // a wait that gave up comes first: the values computed after it are not
  // meaningful, so a range error recorded with it is a consequence
  if (e.code & ~kErrRange) return fail(LAT_ERR_TIMEOUT, "device wait gave up (code %u, site %u)", e.code, e.where);
  if (e.code & kErrRange)
    return fail(LAT_ERR_RANGE, "an activation left the fp16 operand range (code %u, site %u)", e.code, e.where);
  return LAT_OK;
}

// A DiT batch: 1 <= n <= max_batch chunks with indices in range, no two
// sharing (stream, step, ring slot).
// the Wan-class options a DiT stream needs before its chunks run
static lat_status check_stream_ready(const lat_ctx* c, int stream) {
  if (c->d.text_len > 0 && !c->text_set[stream])
    return fail(LAT_ERR_STATE, "stream %d has no text context (lat_dit_set_text)", stream);
  if (c->d.page_tokens > 0 && !c->page_table) return fail(LAT_ERR_STATE, "no page table bound (lat_dit_bind_pages)");
  return LAT_OK;
}

static lat_status check_chunks(const lat_ctx* c, const lat_chunk_desc* chunks, int n) {
  if (!chunks || n < 1 || n > c->d.max_batch) return fail(LAT_ERR_ARG, "DiT: need 1 <= n <= max_batch chunks");
  for (int i = 0; i < n; ++i) {
    const lat_chunk_desc& a = chunks[i];
    if (a.chunk < 0 || a.step < 0 || a.step >= c->d.S || a.stream < 0 || a.stream >= c->d.n_streams)
      return fail(LAT_ERR_ARG, "chunk %d: index out of range", i);
    if ((long long)a.chunk * c->d.T_q > 0x7fffffffLL) return fail(LAT_ERR_ARG, "chunk %d: position overflow", i);
    for (int j = 0; j < i; ++j)
      if (chunks[j].stream == a.stream && chunks[j].step == a.step &&
          ring_slot_of(chunks[j].chunk, c->d.n_hist) == ring_slot_of(a.chunk, c->d.n_hist))
        return fail(LAT_ERR_ARG, "chunks %d and %d share a ring slot", j, i);
    LAT_TRY(check_stream_ready(c, a.stream));
  }
  return LAT_OK;
}

lat_status lat_block_forward(lat_ctx* c, int layer, float* x, const lat_chunk_desc* chunks, int n, void* kv,
                             void* stream) {
  if (!c || !x || !kv) return fail(LAT_ERR_ARG, "NULL argument");
  if (layer < 0 || layer >= c->d.L) return fail(LAT_ERR_ARG, "layer %d out of range", layer);
  if (!aligned16(x) || !aligned16(kv)) return fail(LAT_ERR_ALIGN, "x / kv not 16-byte aligned");
  if (c->d.kind == LAT_PI0_ACTION_EXPERT) {
    if (chunks != nullptr || n != 1) return fail(LAT_ERR_ARG, "pi0 block: chunks must be NULL and n == 1");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t xb = (size_t)c->d.T_q * c->d.D * 4;
    CUDA_TRY(cudaMemcpyAsync(c->xres, x, xb, cudaMemcpyDeviceToDevice, st));
    LAT_TRY(enqueue_pi0_step(c, layer, layer + 1, reinterpret_cast<bf16*>(kv), 0, st));
    CUDA_TRY(cudaMemcpyAsync(x, c->xres, xb, cudaMemcpyDeviceToDevice, st));
    return LAT_OK;
  }
  if (c->d.kind != LAT_DIT) return fail(LAT_ERR_STATE, "lat_block_forward: the prefix model runs via lat_prefill_kv");
  LAT_TRY(check_chunks(c, chunks, n));
  return enqueue_dit_block(c, layer, x, chunks, n, reinterpret_cast<bf16*>(kv), reinterpret_cast<cudaStream_t>(stream));
}

lat_status lat_denoise_chunk(lat_ctx* c, void* kv, const float* state, float* x, void* stream) {
  if (!c || !kv || !state || !x) return fail(LAT_ERR_ARG, "NULL argument");
  if (c->d.kind != LAT_PI0_ACTION_EXPERT) return fail(LAT_ERR_STATE, "lat_denoise_chunk needs an action-expert context");
  if (!aligned16(kv) || !aligned16(state) || !aligned16(x)) return fail(LAT_ERR_ALIGN, "pointer not 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  lat_ctx::Graph* gr = nullptr;
  for (lat_ctx::Graph& g : c->graphs)
    if (g.exec && g.kv == kv && g.state == state && g.x == x && g.stream == stream) gr = &g;
  if (!gr) {
    gr = &c->graphs[0];   // a free slot, else the least recently used one
    for (lat_ctx::Graph& g : c->graphs)
      if (!g.exec || (gr->exec && g.used < gr->used)) gr = &g;
    if (gr->exec) {
      cudaGraphExecDestroy(gr->exec);
      *gr = lat_ctx::Graph{};
    }
    cudaStream_t cap = st;
    bool own = false;
    if (cap == nullptr) {  // the legacy stream cannot be captured: capture on a private one
      CUDA_TRY(cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking));
      own = true;
    }
    CUDA_TRY(cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal));
    lat_status s = enqueue_denoise(c, reinterpret_cast<bf16*>(kv), state, x, cap);
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamEndCapture(cap, &g);
    if (own) cudaStreamDestroy(cap);
    if (s != LAT_OK) {
      if (g) cudaGraphDestroy(g);
      return s;
    }
    if (e != cudaSuccess) return fail(LAT_ERR_CUDA, "graph capture: %s", cudaGetErrorString(e));
    e = cudaGraphInstantiate(&gr->exec, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      gr->exec = nullptr;
      return fail(LAT_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(e));
    }
    gr->kv = kv;
    gr->state = state;
    gr->x = x;
    gr->stream = stream;
  }
  gr->used = ++c->graph_clock;
  CUDA_TRY(cudaGraphLaunch(gr->exec, st));
  return LAT_OK;
}

static lat_status check_latent_io(const lat_ctx* c) {
  if (c->d.kind != LAT_DIT) return fail(LAT_ERR_STATE, "needs a LAT_DIT context");
  if (c->d.act_dim <= 0 || !c->wlin) return fail(LAT_ERR_STATE, "the DiT context has no latent in/out projections");
  return LAT_OK;
}

lat_status lat_dit_interval(lat_ctx* c, void* kv, float* lat, const lat_chunk_desc* chunks, int n, void* stream) {
  if (!c || !kv || !lat) return fail(LAT_ERR_ARG, "NULL argument");
  LAT_TRY(check_latent_io(c));
  if (!aligned16(kv) || !aligned16(lat)) return fail(LAT_ERR_ALIGN, "kv / lat not 16-byte aligned");
  LAT_TRY(check_chunks(c, chunks, n));
  float* ptrs[kMaxChunks];
  for (int b = 0; b < n; ++b) ptrs[b] = lat + (size_t)b * c->d.T_q * c->d.act_dim;
  return enqueue_dit_interval(c, reinterpret_cast<bf16*>(kv), ptrs, chunks, n, reinterpret_cast<cudaStream_t>(stream));
}

lat_status lat_dit_pipeline_push(lat_ctx* c, void* kv, int sid, const float* noise, float* done, int* done_chunk,
                                 void* stream) {
  if (!c || !kv || !done_chunk) return fail(LAT_ERR_ARG, "NULL argument");
  *done_chunk = -1;
  LAT_TRY(check_latent_io(c));
  const lat_model_desc& d = c->d;
  if (sid < 0 || sid >= d.n_streams) return fail(LAT_ERR_ARG, "stream_id %d out of range", sid);
  if (d.S > d.max_batch) return fail(LAT_ERR_SHAPE, "the schedule needs S <= max_batch");
  LAT_TRY(check_stream_ready(c, sid));
  if (!aligned16(kv) || (noise && !aligned16(noise)) || (done && !aligned16(done)))
    return fail(LAT_ERR_ALIGN, "pointer not 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int S = d.S, T = d.T_q, A = d.act_dim;
  int& next = c->pipe_next[sid];
  int& fin = c->pipe_done[sid];
  int* steps = &c->pipe_step[(size_t)sid * S];
  auto slot = [&](int ch) { return c->pipe_lat + ((size_t)sid * S + ch % S) * T * A; };
  if (noise) {
    if ((long long)next * T > 0x7fffffffLL) return fail(LAT_ERR_ARG, "chunk position overflow: reset the stream");
    CUDA_TRY(cudaMemcpyAsync(slot(next), noise, (size_t)T * A * 4, cudaMemcpyDeviceToDevice, st));
    steps[next % S] = 0;
    ++next;
  }
  const int n = next - fin;   // chunks in flight, fin .. next - 1
  if (n == 0) return LAT_OK;
  lat_chunk_desc ch[kMaxChunks];
  float* ptrs[kMaxChunks];
  for (int b = 0; b < n; ++b) {
    const int cc = fin + b;
    ch[b] = lat_chunk_desc{sid, cc, steps[cc % S]};
    ptrs[b] = slot(cc);
  }
  LAT_TRY(check_chunks(c, ch, n));
  LAT_TRY(enqueue_dit_interval(c, reinterpret_cast<bf16*>(kv), ptrs, ch, n, st));
  for (int b = 0; b < n; ++b) ++steps[(fin + b) % S];
  if (steps[fin % S] == S) {   // the oldest chunk has run its S steps
    if (done) CUDA_TRY(cudaMemcpyAsync(done, slot(fin), (size_t)T * A * 4, cudaMemcpyDeviceToDevice, st));
    *done_chunk = fin;
    ++fin;
  }
  return LAT_OK;
}

lat_status lat_dit_set_text(lat_ctx* c, int sid, const void* text, void* stream) {
  if (!c || !text) return fail(LAT_ERR_ARG, "NULL argument");
  const lat_model_desc& d = c->d;
  if (d.kind != LAT_DIT || d.text_len <= 0) return fail(LAT_ERR_STATE, "needs a DiT context with text_len > 0");
  if (sid < 0 || sid >= d.n_streams) return fail(LAT_ERR_ARG, "stream_id %d out of range", sid);
  if (!aligned16(text)) return fail(LAT_ERR_ALIGN, "text not 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int D = d.D, Tt = d.text_len;
  // the context as fp32 rows, then as the two fp16 planes the projections multiply
  bf16_to_f32_kernel<<<(Tt * D + 255) / 256, 256, 0, st>>>(reinterpret_cast<const bf16*>(text), c->qkvbuf, Tt * D);
  LAT_TRY(launch_check("text bf16 -> fp32"));
  NormArgs na{};
  na.x = c->qkvbuf; na.D = D; na.mode = NORM_NONE; na.eps = d.eps; na.rows_per_chunk = Tt; na.act2 = c->act2;
  LAT_TRY(enqueue_norm(na, Tt, st));
  for (int l = 0; l < d.L; ++l) {   // k | v of every block, fp32, then their fp16 planes
    DenseArgs a{};
    a.M = Tt; a.N = 2 * D; a.K = D; a.terms = kActTerms; a.w_row0 = l * 2 * D; a.epi = E_STORE; a.out = c->qkvbuf;
    a.ldo = 2 * D;
    LAT_TRY(enqueue_dense(c, c->map_act_d, W_CKV, a, st));
    __half* out = c->text_kv + ((size_t)sid * d.L + l) * Tt * 4 * D;
    const size_t n4 = (size_t)Tt * 2 * D / 4;
    kv_planes_kernel<<<(unsigned)std::min<size_t>((n4 + 255) / 256, (size_t)c->num_sms * 8), 256, 0, st>>>(
        c->qkvbuf, Tt, D, out);
    LAT_TRY(launch_check("kv_planes"));
  }
  c->text_set[sid] = 1;
  return LAT_OK;
}

lat_status lat_dit_bind_pages(lat_ctx* c, const int* table) {
  if (!c || !table) return fail(LAT_ERR_ARG, "NULL argument");
  if (c->d.kind != LAT_DIT || c->d.page_tokens <= 0) return fail(LAT_ERR_STATE, "needs a DiT context with page_tokens > 0");
  if (!aligned16(table)) return fail(LAT_ERR_ALIGN, "page table not 16-byte aligned");
  c->page_table = table;
  return LAT_OK;
}

lat_status lat_dit_pipeline_reset(lat_ctx* c, int sid) {
  if (!c) return fail(LAT_ERR_ARG, "NULL argument");
  LAT_TRY(check_latent_io(c));
  if (sid < 0 || sid >= c->d.n_streams) return fail(LAT_ERR_ARG, "stream_id %d out of range", sid);
  c->pipe_next[sid] = c->pipe_done[sid] = 0;
  for (int s = 0; s < c->d.S; ++s) c->pipe_step[(size_t)sid * c->d.S + s] = 0;
  return LAT_OK;
}

lat_status lat_debug_indices(lat_ctx* c, const lat_chunk_desc* chunks, int n, int* slot_out, int* pos_out) {
  if (!c || !slot_out || !pos_out || n <= 0) return fail(LAT_ERR_ARG, "bad argument");
  std::vector<int> ch(n, 0);
  if (c->d.kind == LAT_DIT) {
    if (!chunks) return fail(LAT_ERR_ARG, "chunks NULL");
    for (int i = 0; i < n; ++i) {
      if (chunks[i].chunk < 0) return fail(LAT_ERR_ARG, "negative chunk index");
      ch[i] = chunks[i].chunk;
    }
  } else if (n > c->d.T_q) {
    return fail(LAT_ERR_ARG, "n > T_q");
  }
  int *dch = nullptr, *ds = nullptr, *dp = nullptr;
  CUDA_TRY(cudaMalloc(&dch, n * sizeof(int)));
  CUDA_TRY(cudaMalloc(&ds, n * sizeof(int)));
  CUDA_TRY(cudaMalloc(&dp, n * sizeof(int)));
  cudaMemcpy(dch, ch.data(), n * sizeof(int), cudaMemcpyHostToDevice);
  debug_indices_kernel<<<(n + 127) / 128, 128>>>(dch, n, c->d.kind, c->d.T_prefix, c->d.T_q, c->d.n_hist, ds, dp);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpy(slot_out, ds, n * sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(pos_out, dp, n * sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(dch);
  cudaFree(ds);
  cudaFree(dp);
  if (e != cudaSuccess) return fail(LAT_ERR_CUDA, "debug_indices: %s", cudaGetErrorString(e));
  return LAT_OK;
}

lat_status lat_debug_gemm(lat_ctx* c, int which, int layer, int reps, void* stream) {
  if (!c) return fail(LAT_ERR_ARG, "ctx is NULL");
  if (c->d.kind != LAT_PI0_ACTION_EXPERT) return fail(LAT_ERR_STATE, "needs an action-expert context");
  if (which < 0 || which > 3 || layer < 0 || layer >= c->d.L || reps < 0) return fail(LAT_ERR_ARG, "bad argument");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const lat_model_desc& d = c->d;
  const int T = d.T_q, D = d.D, F = d.F, qd = d.Hq * d.dh;
  for (int r = 0; r < reps; ++r) {
    const int l = (layer + r) % d.L;   // successive launches read different layers' weights (HBM, not L2)
    SkinnyArgs a{};
    a.n_tok = T;
    if (which == 0) {
      a.out = c->qkv_acc; a.out_ld = c->nqkv;
      LAT_TRY(enqueue_skinny(c, c->map_qkv, c->bmap_x, c->g_qkv, l, a, st));
    } else if (which == 1) {
      a.out = c->xres; a.out_ld = D;
      LAT_TRY(enqueue_skinny(c, c->map_o, c->bmap_o, c->g_o, l, a, st));
    } else if (which == 2) {
      a.out = c->gu_acc; a.out_ld = 2 * F;
      LAT_TRY(enqueue_skinny(c, c->map_gu, c->bmap_x, c->g_gu, l, a, st));
    } else {
      a.out = c->xres; a.out_ld = D;
      LAT_TRY(enqueue_skinny(c, c->map_d, c->bmap_h, c->g_d, l, a, st));
    }
  }
  (void)qd;
  return LAT_OK;
}

lat_status lat_debug_attention(lat_ctx* c, const float* q, const void* k, const void* v, float* out, int T_q,
                               int T_kv, void* stream) {
  if (!c || !q || !k || !v || !out) return fail(LAT_ERR_ARG, "NULL argument");
  if (c->d.kind != LAT_PI0_ACTION_EXPERT) return fail(LAT_ERR_STATE, "needs an action-expert context");
  const lat_model_desc& d = c->d;
  if (T_q < 1 || T_q > d.T_q || T_kv < 1 || T_kv > d.T_prefix + d.T_q)
    return fail(LAT_ERR_SHAPE, "T_q / T_kv out of the context's range");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(LAT_ERR_ALIGN, "pointer not 16-byte aligned");
  const int nkb = attn_key_blocks(T_kv);
  const int n_split = nkb < kMaxKeySplits ? nkb : kMaxKeySplits;
  return enqueue_attention(d, q, d.Hq * d.dh, reinterpret_cast<const bf16*>(k), reinterpret_cast<const bf16*>(v),
                           d.Hkv * d.dh, T_q, T_kv, n_split, out, d.Hq * d.dh, c->pm, c->pl, c->po,
                           reinterpret_cast<cudaStream_t>(stream));
}

lat_status lat_debug_dense_gemm(lat_ctx* c, int which, int layer, const void* act, int M, int terms, float* out,
                                void* stream) {
  if (!c || !act || !out) return fail(LAT_ERR_ARG, "NULL argument");
  if (c->d.kind != LAT_PI0_PREFIX && c->d.kind != LAT_DIT) return fail(LAT_ERR_STATE, "needs a dense context");
  const lat_model_desc& d = c->d;
  if (which < 0 || which > 3 || layer < 0 || layer >= d.L || M < 1 || M > c->m_max || terms < 1 || terms > kActTerms)
    return fail(LAT_ERR_ARG, "bad argument");
  if (!aligned16(act) || !aligned16(out)) return fail(LAT_ERR_ALIGN, "pointer not 16-byte aligned");
  const int qd = d.Hq * d.dh;
  const int ffn_rows = d.kind == LAT_PI0_PREFIX ? 2 * d.F : d.F;
  const int N[4] = {c->nqkv, d.D, ffn_rows, d.D};
  const int K[4] = {d.D, qd, d.D, d.F};
  CUtensorMap amap;
  LAT_TRY(make_act_map(&amap, act, M, terms * K[which]));
  DenseArgs a{};
  a.M = M; a.N = N[which]; a.K = K[which]; a.terms = terms; a.w_row0 = layer * N[which];
  a.epi = E_STORE; a.out = out; a.ldo = N[which];
  return enqueue_dense(c, amap, which, a, reinterpret_cast<cudaStream_t>(stream));
}

lat_status lat_debug_step(lat_ctx* c, void* kv, int reps, void* stream) {
  if (!c || !kv) return fail(LAT_ERR_ARG, "NULL argument");
  if (c->d.kind != LAT_PI0_ACTION_EXPERT) return fail(LAT_ERR_STATE, "step kernel: action-expert contexts only");
  if (reps < 1) return fail(LAT_ERR_ARG, "reps must be positive");
  if (!aligned16(kv)) return fail(LAT_ERR_ALIGN, "kv not 16-byte aligned");
  const size_t layer_elems = (size_t)2 * (c->d.T_prefix + c->d.T_q) * c->d.Hkv * c->d.dh;
  for (int r = 0; r < reps; ++r)
    LAT_TRY(enqueue_pi0_step(c, 0, c->d.L, reinterpret_cast<bf16*>(kv), (long long)layer_elems,
                             reinterpret_cast<cudaStream_t>(stream)));
  return LAT_OK;
}

lat_status lat_debug_trace(lat_ctx* c, unsigned long long* buf, long long n) {
  if (!c) return fail(LAT_ERR_ARG, "ctx is NULL");
  if (c->d.kind == LAT_DIT) {   // the tensor-core attention of the DiT block: 3 x 32 x 8 entries
    if (buf && n < 3 * 32 * 8) return fail(LAT_ERR_SHAPE, "trace buffer too small");
    c->attn_trace = buf;
    return LAT_OK;
  }
  if (c->d.kind != LAT_PI0_ACTION_EXPERT) return fail(LAT_ERR_STATE, "trace: action-expert and DiT contexts only");
  if (buf && n < (long long)c->num_sms * c->d.L * 64) return fail(LAT_ERR_SHAPE, "trace buffer too small");
  if (buf && (reinterpret_cast<uintptr_t>(buf) & 7u)) return fail(LAT_ERR_ALIGN, "trace buffer not 8-byte aligned");
  c->mk.trace = buf;
  c->drop_graphs();   // the captured graphs hold the old arguments
  return LAT_OK;
}

lat_status lat_debug_clear(lat_ctx* c, void* stream) {
  if (!c) return fail(LAT_ERR_ARG, "ctx is NULL");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const lat_model_desc& d = c->d;
  CUDA_TRY(cudaMemsetAsync(c->qkv_acc, 0, (size_t)d.T_q * c->nqkv * 4, st));
  CUDA_TRY(cudaMemsetAsync(c->gu_acc, 0, (size_t)d.T_q * 2 * d.F * 4, st));
  return LAT_OK;
}

lat_status lat_sync(lat_ctx* c) {
  if (!c) return fail(LAT_ERR_ARG, "ctx is NULL");
  CUDA_TRY(cudaDeviceSynchronize());
  return check_dev_err(c);
}

lat_status lat_clear_error(lat_ctx* c) {
  if (!c) return fail(LAT_ERR_ARG, "ctx is NULL");
  CUDA_TRY(cudaDeviceSynchronize());
  CUDA_TRY(cudaMemset(c->err, 0, sizeof(DevErr)));
  return LAT_OK;
}

lat_status lat_debug_act_terms(lat_ctx* c, int terms) {
  if (!c) return fail(LAT_ERR_ARG, "ctx is NULL");
  if (c->d.kind != LAT_PI0_PREFIX && c->d.kind != LAT_DIT) return fail(LAT_ERR_STATE, "dense contexts only");
  if (terms < 1 || terms > kActTerms) return fail(LAT_ERR_ARG, "terms must be 1 or 2");
  c->act_terms = terms;
  return LAT_OK;
}

lat_status lat_debug_wait_skew(lat_ctx* c, int which, int extra) {
  if (!c) return fail(LAT_ERR_ARG, "ctx is NULL");
  if (c->d.kind != LAT_PI0_ACTION_EXPERT) return fail(LAT_ERR_STATE, "wait skew: action-expert contexts only");
  if (which < 0 || which > 3 || extra < 0) return fail(LAT_ERR_ARG, "which must be 0..3 and extra >= 0");
  c->mk.skew_where = extra > 0 ? which : 0;
  c->mk.skew = which > 0 ? (unsigned)extra : 0u;
  c->drop_graphs();   // the captured graphs hold the old arguments
  return LAT_OK;
}

lat_status lat_debug_timeout(lat_ctx* c, void* stream) {
  if (!c) return fail(LAT_ERR_ARG, "ctx is NULL");
  debug_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(c->err, 999);
  return launch_check("debug_timeout");
}

void lat_destroy(lat_ctx* c) {
  if (!c) return;
  cudaDeviceSynchronize();
  delete c;
}

}  // extern "C"
