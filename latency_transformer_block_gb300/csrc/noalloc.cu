// lat_chunk_attention_noalloc: the chunk attention for callers that cannot
// allocate device memory.
//
// The attention splits the keys into ranges and merges per-range partial
// results (running max, running sum, unnormalised output), which needs scratch
// memory.  lat_create's context keeps that scratch in its cudaMalloc'd
// workspace; this entry point instead uses one file-scope device array, so it
// needs no context and calls no allocator at all.  It is for code that owns
// every device byte itself (an engine with its own memory pool, or a real-time
// loop that forbids allocation once it runs) and therefore can neither call
// cudaMalloc nor let a library do it for them.
//
// The array is part of the library image: every GPU that loads liblat.so holds
// it (4 MiB) until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/lat.h"
#include "attention.cuh"

lat_status lat_internal_fail(lat_status s, const char* msg);

namespace {

constexpr int kNoAllocScratchFloats = 1 << 20;   // 4 MiB of fp32 partials
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

// Device address of g_noalloc_scratch, per device, and the id of the device
// context it was looked up in.  In host code the symbol name is only a
// host-side stand-in; a kernel must be given the address that
// cudaGetSymbolAddress returns with the device current.  A new context on the
// device (after cudaDeviceReset the module is loaded again, at a new address,
// and the kernels' shared-memory limits are back at their defaults) repeats
// the set-up.
float* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_ctx_id[kMaxDevices] = {};
std::mutex g_setup_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// id of the current device context (0 if the driver cannot tell)
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked = false;
  if (!looked) {
    looked = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  }
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_cur && get_id && get_cur(&c) == CUDA_SUCCESS && c && get_id(c, &id) == CUDA_SUCCESS) return id;
  return 0;
}

lat_status setup_device(int dev, float** out) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  const unsigned long long id = current_ctx_id();
  if (!g_scratch_addr[dev] || id != g_ctx_id[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return lat_internal_fail(LAT_ERR_CUDA, "cudaGetSymbolAddress(noalloc scratch) failed");
    e = lat::set_attention_smem_limits();
    if (e != cudaSuccess) return lat_internal_fail(LAT_ERR_CUDA, "cudaFuncSetAttribute(attention) failed");
    g_scratch_addr[dev] = static_cast<float*>(p);
    g_ctx_id[dev] = id;
  }
  *out = g_scratch_addr[dev];
  return LAT_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" lat_status lat_chunk_attention_noalloc(const float* q, const void* k, const void* v, float* out,
                                                  int T_q, int T_kv, int Hq, int Hkv, int dh, void* stream) {
  if (!q || !k || !v || !out) return lat_internal_fail(LAT_ERR_ARG, "NULL argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return lat_internal_fail(LAT_ERR_ALIGN, "pointer not 16-byte aligned");
  if (T_q < 1 || T_kv < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv)
    return lat_internal_fail(LAT_ERR_SHAPE, "need T_q, T_kv, Hq, Hkv >= 1 and Hq a multiple of Hkv");
  if (dh != 64 && dh != 128 && dh != 256) return lat_internal_fail(LAT_ERR_SHAPE, "dh must be 64, 128 or 256");
  // one key range needs Hq * T_q * (dh + 2) floats of partials (output, max, sum)
  const long long per_split = (long long)Hq * T_q * (dh + 2);
  if (per_split > kNoAllocScratchFloats)
    return lat_internal_fail(LAT_ERR_SHAPE,
                             "Hq * T_q * (dh + 2) exceeds the static scratch (1048576 floats, 4 MiB)");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return lat_internal_fail(LAT_ERR_CUDA, "no usable current device");
  float* scratch = nullptr;
  lat_status s = setup_device(dev, &scratch);
  if (s != LAT_OK) return s;

  // as many key ranges as the array holds partials for (at most 32, at most
  // one per 32-key block); a context sizes its ranges by the SM count instead,
  // so at shapes where the array holds fewer ranges this call has fewer CTAs
  const int nkb = lat::attn_key_blocks(T_kv);
  int n_split = (int)(kNoAllocScratchFloats / per_split);
  if (n_split > nkb) n_split = nkb;
  if (n_split > 32) n_split = 32;   // partials the combine kernel merges
  if (n_split < 1) n_split = 1;

  lat::AttnArgs a{};
  a.q = q;
  a.q_ld = Hq * dh;
  a.k = reinterpret_cast<const __nv_bfloat16*>(k);
  a.v = reinterpret_cast<const __nv_bfloat16*>(v);
  a.kv_ld = Hkv * dh;
  a.T_q = T_q;
  a.T_kv = T_kv;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)dh));
  a.n_split = n_split;
  a.out = out;
  a.out_ld = Hq * dh;
  // partials: [n_split][Hq][T_q] max, then sum, then [n_split][Hq][T_q][dh]
  // output.  Every element the merge reads is written by this call first, so
  // nothing needs clearing between calls.
  const size_t nrow = (size_t)n_split * Hq * T_q;
  a.part_m = scratch;
  a.part_l = scratch + nrow;
  a.part_o = scratch + 2 * nrow;
  cudaError_t e = lat::launch_chunk_attention(a, dh, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return lat_internal_fail(LAT_ERR_CUDA, cudaGetErrorString(e));
  return LAT_OK;
}
