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
//  * B operand = the activations of the same 64 K-columns, split into three
//    bf16 terms (hi, mid, lo: 24 significant bits) stacked as 192 rows, written
//    to shared memory by the CTA's own threads in the same swizzled layout.
//    The transform of the source (plain, GeGLU with the RMS row scale, SiLU)
//    happens while splitting.
//  * One tcgen05.mma per 16-wide K step: M = 128 features, N = 192, fp32
//    accumulator in TMEM (192 columns).  The epilogue adds the three terms of
//    each token and reduces split-K partial sums with fp32 atomics.
//  * Grid = (N_out / 128) m-tiles x `splits` K ranges.  Warp 0 issues TMA,
//    warp 1 issues MMAs, warps 2..5 prepare B tiles and run the epilogue.
#pragma once
#include "common.cuh"

namespace lat {

enum BMode : int { B_PLAIN = 0, B_GEGLU = 1, B_SILU = 2 };

struct SkinnyArgs {
  int w_row0;            // first row of this matrix inside the stacked weight tensor
  int N_out;             // multiple of 128
  int K;                 // multiple of 64
  int splits;            // K ranges (1 <= splits <= K / 64)
  const float* src;      // activations fp32 [n_tok][src_ld]
  int src_ld;
  int src2_off;          // B_GEGLU: offset of the up half inside a row
  const float* row_scale;  // B_GEGLU: per-token RMS factor
  int mode;
  int n_tok;             // <= 64
  float* out;            // fp32 [n_tok][out_ld], accumulated atomically
  int out_ld;
  const float* bias;     // fp32 [N_out], added once (split 0), may be null
  const float* stat_src; // optional side job: stat_out[t] = rsqrt(mean(stat_src[t]^2) + eps)
  int stat_len;
  float* stat_out;
  float eps;
  DevErr* err;
};

constexpr int kSkW = 128 * 64 * 2;   // weight tile bytes
constexpr int kSkB = 192 * 64 * 2;   // activation tile bytes (3 terms x 64 tokens)

__host__ __device__ constexpr int skinny_smem_bytes(int stages) {
  return 1024 + stages * (kSkW + kSkB) + 8 * (3 * stages + 1) + 16;
}

// Prepare the B tile (3 x 64 rows x 64 K) for K columns [k0, k0 + 64).
// Thread t of 128 handles token row t/2 and 32 consecutive columns.
__device__ __forceinline__ void skinny_prep_b(uint8_t* b, const SkinnyArgs& a, int k0, int t) {
  const int row = t >> 1, half = t & 1;
  const int kc = k0 + half * 32;
  float v[32];
  if (row < a.n_tok) {
    const float4* p = reinterpret_cast<const float4*>(a.src + (size_t)row * a.src_ld + kc);
    if (a.mode == B_GEGLU) {
      const float4* q = reinterpret_cast<const float4*>(a.src + (size_t)row * a.src_ld + a.src2_off + kc);
      const float r = a.row_scale[row];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float4 g = p[j], u = q[j];
        v[4 * j + 0] = gelu_tanh(r * g.x) * (r * u.x);
        v[4 * j + 1] = gelu_tanh(r * g.y) * (r * u.y);
        v[4 * j + 2] = gelu_tanh(r * g.z) * (r * u.z);
        v[4 * j + 3] = gelu_tanh(r * g.w) * (r * u.w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float4 g = p[j];
        v[4 * j + 0] = g.x; v[4 * j + 1] = g.y; v[4 * j + 2] = g.z; v[4 * j + 3] = g.w;
      }
      if (a.mode == B_SILU) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = silu(v[j]);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = 0.f;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t wh[4], wm[4], wl[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      Split3 s0 = split3(v[c * 8 + 2 * e]), s1 = split3(v[c * 8 + 2 * e + 1]);
      wh[e] = pack_bf16(s0.hi, s1.hi);
      wm[e] = pack_bf16(s0.mid, s1.mid);
      wl[e] = pack_bf16(s0.lo, s1.lo);
    }
    const int kk = half * 32 + c * 8;
    *reinterpret_cast<uint4*>(b + sw128_offset(row, kk)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
    *reinterpret_cast<uint4*>(b + sw128_offset(64 + row, kk)) = make_uint4(wm[0], wm[1], wm[2], wm[3]);
    *reinterpret_cast<uint4*>(b + sw128_offset(128 + row, kk)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
  }
}

template <int STAGES>
__global__ void __launch_bounds__(192, 1) skinny_gemm_kernel(const __grid_constant__ CUtensorMap wmap,
                                                             SkinnyArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;
  uint8_t* sB = smem + STAGES * kSkW;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * kSkB);
  uint64_t* full_w = bars;
  uint64_t* full_b = bars + STAGES;
  uint64_t* empty = bars + 2 * STAGES;
  uint64_t* acc_full = bars + 3 * STAGES;
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
      mbar_init(&full_w[s], 1);
      mbar_init(&full_b[s], 128);
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

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&wmap);
      const uint64_t pol = l2_policy_evict_first();
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, a.err, 10)) break;
        mbar_arrive_expect_tx(&full_w[s], kSkW);
        tma_load_2d(sW + s * kSkW, &wmap, &full_w[s], (kb0 + i) * 64, a.w_row0 + m * 128, pol);
        ++issued;
      }
      // drain: never leave a copy in flight into this CTA's shared memory
      for (int i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
        mbar_wait(&full_w[i % STAGES], (i / STAGES) & 1, a.err, 13);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 192);
      bool ok = true;
      for (int i = 0; i < nkb && ok; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        ok = mbar_wait(&full_w[s], ph, a.err, 11) && mbar_wait(&full_b[s], ph, a.err, 12);
        if (!ok) break;
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
    const int t = threadIdx.x - 64;  // 0..127
    // optional side job: RMS statistics of one token row per CTA
    if (a.stat_out) {
      __shared__ float red[4];
      for (int row = blockIdx.x; row < a.n_tok; row += gridDim.x) {
        const float* xr = a.stat_src + (size_t)row * a.stat_len;
        float ss = 0.f;
        for (int j = t; j < a.stat_len; j += 128) ss += xr[j] * xr[j];
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) red[warp - 2] = ss;
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (t == 0) a.stat_out[row] = rsqrtf((red[0] + red[1] + red[2] + red[3]) / a.stat_len + a.eps);
        asm volatile("bar.sync 1, 128;" ::: "memory");
      }
    }
    for (int i = 0; i < nkb; ++i) {
      const int s = i % STAGES;
      const uint32_t ph = (i / STAGES) & 1;
      if (!mbar_wait(&empty[s], ph ^ 1, a.err, 14)) break;
      skinny_prep_b(sB + s * kSkB, a, (kb0 + i) * 64, t);
      fence_proxy_async_smem();
      mbar_arrive(&full_b[s]);
    }
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

}  // namespace lat
