// Weight-streaming GEMM for a skinny activation (<= 64 tokens) on tcgen05.
//
//   out[t][f] (+)= sum_k act(t, k) * W[f][k]        (t < 64 tokens, f < N_out)
//
// The pages' action expert is memory bound: every block streams its weights
// once per denoise step while only 64 tokens use them ("Running VLAs at
// Real-time Speed", reading note, section 5: GEMM tiles per shape, partial
// split-K for tail blocks, section 6.2: roofline 2KM/B_mem).  The layout here:
//
//  * A operand = a 128 x 64 tile of the K-major weight matrix, moved by TMA
//    (128-byte swizzle) through a ring of STAGES shared-memory slots with an
//    L2 evict-first hint (weights are read once per step).
//  * B operand = the activation, written by the kernel that produces it as
//    three bf16 planes (hi, mid, lo: 24 significant bits) stacked as 192
//    K-major rows [3][64 tokens][K]; its 192 x 64 tile of the same K range
//    arrives by TMA in the same stage.  (The action expert's blocks run in the
//    persistent step kernel; this kernel serves the embedding projection and
//    the standalone weight-streaming measurement.)
//  * One tcgen05.mma per 16-wide K step: M = 128 features, N = 192, fp32
//    accumulator in TMEM.  The epilogue adds the three terms of each token and
//    reduces split-K partial sums with fp32 atomics.
//  * Grid = (N_out / 128) m-tiles x `splits` K ranges.  Warp 0 issues TMA,
//    warp 1 issues MMAs, warps 2..5 run the epilogue.
//  * Programmatic dependent launch: the weight tiles of the first stages are
//    requested before griddepcontrol.wait (they do not depend on the previous
//    kernel), so the weight stream starts while the previous kernel finishes.
#pragma once
#include "common.cuh"

namespace lat {

struct SkinnyArgs {
  int w_row0;            // first row of this matrix inside the stacked weight tensor
  int N_out;             // multiple of 128
  int K;                 // multiple of 64
  int splits;            // K ranges (1 <= splits <= K / 64)
  int n_tok;             // <= 64 (rows of the output)
  float* out;            // fp32 [n_tok][out_ld], accumulated atomically
  int out_ld;
  const float* bias;     // fp32 [N_out], added once (split 0), may be null
  DevErr* err;
};

constexpr int kSkW = 128 * 64 * 2;   // weight tile bytes
constexpr int kSkB = 192 * 64 * 2;   // activation tile bytes (3 planes x 64 tokens)

__host__ __device__ constexpr int skinny_smem_bytes(int stages) {
  return 1024 + stages * (kSkW + kSkB) + 8 * (2 * stages + 1) + 16;
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <int STAGES>
__global__ void __launch_bounds__(192, 1) skinny_gemm_kernel(const __grid_constant__ CUtensorMap wmap,
                                                             const __grid_constant__ CUtensorMap bmap,
                                                             SkinnyArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;
  uint8_t* sB = smem + STAGES * kSkW;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * kSkB);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = a.N_out / 128;
  const int m = blockIdx.x % m_tiles;
  const int split = blockIdx.x / m_tiles;
  const int kb_total = a.K / 64;
  const int kb0 = split * kb_total / a.splits;
  const int nkb = (split + 1) * kb_total / a.splits - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch();

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&wmap);
      tma_prefetch_desc(&bmap);
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_b = l2_policy_evict_last();
      const int npre = nkb < STAGES ? nkb : STAGES;
      // weights first: independent of the previous kernel
      for (int i = 0; i < npre; ++i) {
        mbar_arrive_expect_tx(&full[i], kSkW + kSkB);
        tma_load_2d(sW + i * kSkW, &wmap, &full[i], (kb0 + i) * 64, a.w_row0 + m * 128, pol_w);
      }
      griddep_wait();
      for (int i = 0; i < npre; ++i) tma_load_2d(sB + i * kSkB, &bmap, &full[i], (kb0 + i) * 64, 0, pol_b);
      int issued = npre;
      for (int i = npre; i < nkb; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, a.err, 10)) break;
        mbar_arrive_expect_tx(&full[s], kSkW + kSkB);
        tma_load_2d(sW + s * kSkW, &wmap, &full[s], (kb0 + i) * 64, a.w_row0 + m * 128, pol_w);
        tma_load_2d(sB + s * kSkB, &bmap, &full[s], (kb0 + i) * 64, 0, pol_b);
        ++issued;
      }
      // drain: never leave a copy in flight into this CTA's shared memory
      for (int i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
        mbar_wait(&full[i % STAGES], (i / STAGES) & 1, a.err, 13);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 192);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!mbar_wait(&full[s], ph, a.err, 11)) break;
        tc_fence_after();
        const uint32_t aa = smem_u32(sW + s * kSkW), bb = smem_u32(sB + s * kSkB);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16_ss(tmem, desc_k_sw128(aa + k * 32), desc_k_sw128(bb + k * 32), idesc, (i | k) != 0);
        mma_commit(&empty[s]);
      }
      mma_commit(acc_full);
    }
  } else {
    griddep_wait();   // `out` may be read/written by the previous kernel
    if (mbar_wait(acc_full, 0, a.err, 15)) {
      tc_fence_after();
      const int quad = warp & 3;
      const int f = m * 128 + quad * 32 + lane;
      const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16);
      float acc[64];
      float v[32];
      tmem_ld32(tbase + 0, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = v[j];
      tmem_ld32(tbase + 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[32 + j] = v[j];
#pragma unroll
      for (int c = 2; c < 6; ++c) {
        tmem_ld32(tbase + c * 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[((c & 1) * 32) + j] += v[j];
      }
      const float bias = (split == 0 && a.bias) ? a.bias[f] : 0.f;
#pragma unroll
      for (int tok = 0; tok < 64; ++tok)
        if (tok < a.n_tok) atomicAdd(&a.out[(size_t)tok * a.out_ld + f], acc[tok] + bias);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// tanh from the exponential (no cancellation concern here: the callers use
// 1 + tanh), accurate to a few fp32 ulps of 1
__device__ __forceinline__ float gelu_tanh_fast(float x) {
  const float k0 = 0.7978845608028654f;
  const float y = k0 * (x + 0.044715f * x * x * x);
  const float e = __expf(2.f * y);
  const float t = 1.f - 2.f / (1.f + e);
  return 0.5f * x * (1.f + t);
}

}  // namespace lat
