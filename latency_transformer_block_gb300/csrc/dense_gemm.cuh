// Dense GEMM on tcgen05 for many tokens (prefix prefill, batched DiT chunks):
//
//   acc[m][n] = sum_k A[m][k] W[n][k]
//
// A is an activation stored as `terms` bf16 planes side by side ([M][terms*K],
// plane t holding the t-th term of the fp32 value's split, so sum_t A_t = A to
// 8 * terms significant bits); the K loop runs over terms*K and reuses the
// weight tile of column k mod K for every plane.  Products of bf16 pairs are
// exact on the tensor cores and accumulate in fp32 in TMEM.
//
// Tile 128 (tokens) x 128 (features) x 64, both operands moved by TMA with a
// 128-byte swizzle through STAGES slots; a slot holds one weight tile and the
// `terms` activation tiles of the same K range, so each weight tile crosses
// from L2 once (per-SM L2 bandwidth, ~120 GB/s, is what bounds this GEMM);
// one tcgen05.mma (M=128, N=128, K=16) per 16-wide K step and plane; warp 0
// issues TMA, warp 1 MMAs, warps 2..5 accumulate and run the fused epilogue
// (bias, residual, per-chunk gate, GELU / GeGLU followed by the split of the
// next GEMM's activation).
//
// Accumulation in two levels: the tensor core sums one chunk of at most 32
// MMAs (8 / terms K-blocks of all planes) into a TMEM accumulator; the epilogue warps add each
// finished chunk into fp32 registers (round to nearest) while the tensor core
// fills the other TMEM accumulator.  Measured on this hardware, an fp32 TMEM
// accumulator run over thousands of MMAs drifts by about one unit of its last
// place per MMA in one direction (K = 13824 x 2 terms gave 2e-4 relative
// error); chunks of 32 MMAs bound that drift to ~4e-6.
#pragma once
#include "common.cuh"

namespace lat {

enum DenseEpi : int {
  E_STORE = 0,        // out[m][n] = acc (+ bias[n])
  E_RESID = 1,        // out[m][n] += acc
  E_RESID_GATE = 2,   // out[m][n] += gate[chunk(m)][n] * acc
  E_GELU_SPLIT = 3,   // act planes <- exact split of GELU_tanh(acc)
  E_GEGLU_SPLIT = 4,  // tile = [64 gate | 64 up] -> act planes <- exact split of GELU(g) * u
};

constexpr int kMaxChunks = 16;
constexpr int kChunkMMA = 32;   // MMAs (of K = 16) per TMEM accumulation chunk, at most

struct DenseArgs {
  int M, N, K;           // K = reduction length of one term
  int terms;             // planes in A (1, 2 or 3)
  int w_row0;            // first weight row of this matrix in the stacked tensor
  int epi;
  float* out;            // fp32 [M][ldo] (E_STORE / E_RESID / E_RESID_GATE)
  int ldo;
  const float* bias;     // E_STORE: fp32 [N] or null
  // E_RESID_GATE: gate row of chunk b = gate + gate_off[b]; chunk(m) = m / rows_per_chunk
  const float* gate;
  int gate_off[kMaxChunks];
  int rows_per_chunk;
  // E_*_SPLIT: bf16 planes [M][3 * ldh] (hi at column c, mid at ldh + c, lo at 2 ldh + c)
  __nv_bfloat16* act2;
  int ldh;
  DevErr* err;
};

constexpr int kDA = 128 * 64 * 2;   // A tile bytes (one plane)
constexpr int kDB = 128 * 64 * 2;   // B tile bytes
constexpr int kDSlot = 3 * kDA + kDB;   // one slot: up to three planes of A + B

__host__ __device__ constexpr int dense_smem_bytes(int stages) {
  return 1024 + stages * kDSlot + 8 * (2 * stages + 4) + 16;
}

// 8 values -> three planes of 8 bf16 (hi, mid, lo: the exact split of the fp32 value)
__device__ __forceinline__ void store_split3(__nv_bfloat16* hi, int plane, const float* v) {
  uint32_t wh[4], wm[4], wl[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) split_pair_exact(v[2 * e], v[2 * e + 1], wh[e], wm[e], wl[e]);
  *reinterpret_cast<uint4*>(hi) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
  *reinterpret_cast<uint4*>(hi + plane) = make_uint4(wm[0], wm[1], wm[2], wm[3]);
  *reinterpret_cast<uint4*>(hi + 2 * plane) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
}

// Epilogue of one tile row: 128 accumulated columns of token `row`, feature
// tile tn.
__device__ __forceinline__ void dense_epilogue(const DenseArgs& a, const float (&acc)[128], int row, int tn) {
  if (a.epi == E_GEGLU_SPLIT) {
    // columns 0..63 gate, 64..127 up of features tn*64 + j
    __nv_bfloat16* hi = a.act2 + (size_t)row * 3 * a.ldh + tn * 64;
#pragma unroll
    for (int j = 0; j < 64; j += 8) {
      float h[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) h[e] = gelu_tanh(acc[j + e]) * acc[64 + j + e];
      store_split3(hi + j, a.ldh, h);
    }
  } else if (a.epi == E_GELU_SPLIT) {
    __nv_bfloat16* hi = a.act2 + (size_t)row * 3 * a.ldh + tn * 128;
#pragma unroll
    for (int j = 0; j < 128; j += 8) {
      float h[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) h[e] = gelu_tanh(acc[j + e]);
      store_split3(hi + j, a.ldh, h);
    }
  } else {
    const int n0 = tn * 128;
    float* o = a.out + (size_t)row * a.ldo + n0;
    const float* gate = (a.epi == E_RESID_GATE) ? a.gate + a.gate_off[row / a.rows_per_chunk] + n0 : nullptr;
#pragma unroll
    for (int j = 0; j < 128; j += 4) {
      float4 r = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
      if (a.epi == E_STORE) {
        if (a.bias) {
          const float4 b = *reinterpret_cast<const float4*>(a.bias + n0 + j);
          r.x += b.x; r.y += b.y; r.z += b.z; r.w += b.w;
        }
      } else {
        const float4 x = *reinterpret_cast<const float4*>(o + j);
        if (a.epi == E_RESID_GATE) {
          const float4 gg = *reinterpret_cast<const float4*>(gate + j);
          r.x = x.x + gg.x * r.x; r.y = x.y + gg.y * r.y; r.z = x.z + gg.z * r.z; r.w = x.w + gg.w * r.w;
        } else {
          r.x += x.x; r.y += x.y; r.z += x.z; r.w += x.w;
        }
      }
      *reinterpret_cast<float4*>(o + j) = r;
    }
  }
}

template <int STAGES>
__global__ void __launch_bounds__(192, 1) dense_gemm_kernel(const __grid_constant__ CUtensorMap amap,
                                                            const __grid_constant__ CUtensorMap wmap, DenseArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * kDSlot);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;    // [2]
  uint64_t* acc_empty = bars + 2 * STAGES + 2;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = a.N / 128;
  const int tiles = ((a.M + 127) / 128) * n_tiles;
  const int nkb = a.K / 64;                                   // K-blocks of one plane
  const int chunk_kb = kChunkMMA / (4 * a.terms);             // K-blocks per accumulation chunk
  const int nchunk = (nkb + chunk_kb - 1) / chunk_kb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&acc_full[0], 1);
    mbar_init(&acc_full[1], 1);
    mbar_init(&acc_empty[0], 128);
    mbar_init(&acc_empty[1], 128);
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

  // persistent: CTA b takes tiles b, b + grid, ...; the slot ring and the two
  // accumulators carry on across tiles, so a tile's epilogue overlaps the next
  // tile's MMAs (counters it / gch run over all tiles of the CTA)
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&amap);
      tma_prefetch_desc(&wmap);
      const uint64_t pol_w = l2_policy_evict_last();   // weight tiles are re-read by every m-tile
      const uint64_t pol_a = l2_policy_evict_first();
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        const int tm = tile / n_tiles, tn = tile % n_tiles;
        for (int i = 0; i < nkb; ++i, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, a.err, 20)) { ok = false; break; }
          uint8_t* slot = smem + s * kDSlot;
          mbar_arrive_expect_tx(&full[s], a.terms * kDA + kDB);
          for (int t = 0; t < a.terms; ++t)
            tma_load_2d(slot + t * kDA, &amap, &full[s], t * a.K + i * 64, tm * 128, pol_a);
          tma_load_2d(slot + 3 * kDA, &wmap, &full[s], i * 64, a.w_row0 + tn * 128, pol_w);
        }
      }
      for (uint32_t i = (it > (uint32_t)STAGES ? it - STAGES : 0); i < it; ++i)
        mbar_wait(&full[i % STAGES], (i / STAGES) & 1, a.err, 21);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 128);
      bool ok = true;
      uint32_t it = 0, gch = 0;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        for (int ch = 0; ch < nchunk && ok; ++ch, ++gch) {
          const int buf = gch & 1;
          // the epilogue has drained this accumulator (use gch - 2)
          if (!mbar_wait(&acc_empty[buf], ((gch >> 1) & 1) ^ 1, a.err, 24)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(buf * 128);
          const int i0 = ch * chunk_kb, i1 = min(nkb, i0 + chunk_kb);
          for (int i = i0; i < i1; ++i, ++it) {
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            if (!mbar_wait(&full[s], ph, a.err, 22)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + s * kDSlot), bb = sa + 3 * kDA;
            for (int t = 0; t < a.terms; ++t) {
              const uint32_t aa = sa + t * kDA;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_bf16_ss(d, desc_k_sw128(aa + k * 32), desc_k_sw128(bb + k * 32), idesc,
                            (i > i0) || (t > 0) || (k > 0));
            }
            mma_commit(&empty[s]);
          }
          mma_commit(&acc_full[buf]);
        }
      }
    }
  } else {
    const int quad = warp & 3;
    uint32_t gch = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
      const int tm = tile / n_tiles, tn = tile % n_tiles;
      const int row = tm * 128 + quad * 32 + lane;
      const bool valid = row < a.M;
      float acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.f;
      for (int ch = 0; ch < nchunk; ++ch, ++gch) {
        const int buf = gch & 1;
        if (!mbar_wait(&acc_full[buf], (gch >> 1) & 1, a.err, 23)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tb = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * 128);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[32];
          tmem_ld32(tb + c * 32, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[c * 32 + j] += v[j];
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
      }
      if (ok && valid) dense_epilogue(a, acc, row, tn);
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
