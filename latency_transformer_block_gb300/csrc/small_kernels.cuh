// Small kernels of the action-expert path and the offline folds.
#pragma once
#include "common.cuh"

namespace lat {

// The integer maps used by the kernels, exposed for exact checks.
//  pi0: query token t lives in cache slot T_prefix + t and has RoPE position
//       T_prefix + t (the prefix occupies slots / positions 0..T_prefix-1).
//  DiT: chunk c lives in ring slot c mod (n_hist + 1); its token j has RoPE
//       position c * T_chunk + j.
__host__ __device__ __forceinline__ int query_slot(int T_prefix, int t) { return T_prefix + t; }
__host__ __device__ __forceinline__ int query_pos(int T_prefix, int t) { return T_prefix + t; }
__host__ __device__ __forceinline__ int ring_slot_of(int chunk, int n_hist) { return chunk % (n_hist + 1); }
__host__ __device__ __forceinline__ long long chunk_pos0(int chunk, int T) { return (long long)chunk * T; }



// ---------------------------------------------------------------------------
// Offline folds
// ---------------------------------------------------------------------------
// out[orow(n)][k] = bf16( g[k] * W[k][n] )  -- transpose to K-major with the
// RMSNorm scale folded (g may be null: plain transpose).  W: bf16 [K][N]
// row-major; out row stride = K.  With il > 0 the output rows interleave blocks
// of il rows: orow(n) = (n / il) * 2 il + il_off + n mod il (gate and up
// projections share 2*il-row tiles).  32 x 32 tiles, blockDim (32, 8).
static __global__ void fold_transpose_kernel(const __nv_bfloat16* W, const __nv_bfloat16* g, __nv_bfloat16* out,
                                             int K, int N, int il, int il_off) {
  __shared__ float tile[32][33];
  const int k0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int k = k0 + i, n = n0 + threadIdx.x;
    float v = 0.f;
    if (k < K && n < N) {
      v = __bfloat162float(W[(size_t)k * N + n]);
      if (g) v *= __bfloat162float(g[k]);   // exact in fp32: 8 x 8 significant bits
    }
    tile[i][threadIdx.x] = v;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int n = n0 + i, k = k0 + threadIdx.x;
    if (n < N && k < K) {
      const size_t orow = il > 0 ? (size_t)(n / il) * 2 * il + il_off + n % il : (size_t)n;
      out[orow * K + k] = __float2bfloat16_rn(tile[threadIdx.x][i]);
    }
  }
}

// out[r][k] = in[perm[r]][k]: a row permutation of a row-major [rows][K] bf16 matrix
static __global__ void gather_rows_kernel(const __nv_bfloat16* in, const int* perm, __nv_bfloat16* out, int rows,
                                          int K) {
  const int r = blockIdx.x;
  if (r >= rows) return;
  const __nv_bfloat16* src = in + (size_t)perm[r] * K;
  __nv_bfloat16* dst = out + (size_t)r * K;
  for (int k = threadIdx.x; k < K; k += blockDim.x) dst[k] = src[k];
}

// max |w| over n bf16 values into *out (as fp32 bits: non-negative floats
// order like their bit patterns).  *out must start at 0.
static __global__ void absmax_bf16_kernel(const __nv_bfloat16* w, size_t n, unsigned* out) {
  float m = 0.f;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    m = fmaxf(m, fabsf(__bfloat162float(w[i])));
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(out, __float_as_uint(m));
}

// In place: bf16 bit patterns w -> fp16 bit patterns of w * scale (scale a power of two).
static __global__ void bf16_to_f16_scaled_kernel(uint16_t* w, size_t n, float scale) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float v = __bfloat162float(__ushort_as_bfloat16(w[i])) * scale;
    w[i] = __half_as_ushort(__float2half_rn(v));
  }
}

// Generic small fp32 GEMM for the offline tables (CUDA cores, fp32 accumulate):
//   C[m][n] = act( sum_k A[m][k] B[k][n] + bias[n] )
// A, B, bias each either bf16 or fp32 (flags).  act: 0 none, 1 SiLU.
struct SmallGemmArgs {
  const void* A; int a_bf16; int lda;
  const void* B; int b_bf16; int ldb;
  const void* bias; int bias_bf16;
  float* C; int ldc;
  int M, N, K, act;
};

__device__ __forceinline__ float ld_any(const void* p, int is_bf16, size_t i) {
  return is_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i])
                 : reinterpret_cast<const float*>(p)[i];
}

static __global__ void small_gemm_kernel(SmallGemmArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const int m = blockIdx.y;
  if (n >= a.N) return;
  float acc = 0.f;
  for (int k = 0; k < a.K; ++k)
    acc = fmaf(ld_any(a.A, a.a_bf16, (size_t)m * a.lda + k), ld_any(a.B, a.b_bf16, (size_t)k * a.ldb + n), acc);
  if (a.bias) acc += ld_any(a.bias, a.bias_bf16, n);
  if (a.act == 1) acc = silu(acc);
  a.C[(size_t)m * a.ldc + n] = acc;
}

// Euler step of the DiT latents of n chunks (T rows each): z[m][a] += dt[s_b] * v[m][a]
// for row m of chunk b = m / T at its denoise step s_b.
struct DitEulerArgs {
  float* z;
  const float* v;
  const float* dt;
  int step[16];
  int T, A, n;
};

static __global__ void dit_euler_kernel(DitEulerArgs a) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)a.n * a.T * a.A) return;
  const int b = (int)(i / ((size_t)a.T * a.A));
  a.z[i] += a.dt[a.step[b]] * a.v[i];
}

// Failure-detection check: one thread waits on an mbarrier that nothing
// arrives on; the bounded wait gives up after the spin budget and records the
// error in the context's error word (site `where`), as every wait of the path does.
static __global__ void debug_timeout_kernel(DevErr* err, unsigned where) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, err, where);
}

static __global__ void bf16_to_f32_kernel(const __nv_bfloat16* in, float* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = __bfloat162float(in[i]);
}

static __global__ void debug_indices_kernel(const int* chunks, int n, int kind, int T_prefix, int T_q, int n_hist,
                                     int* slot_out, int* pos_out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  if (kind == 2) {
    slot_out[i] = ring_slot_of(chunks[i], n_hist);
    pos_out[i] = (int)chunk_pos0(chunks[i], T_q);
  } else {
    slot_out[i] = query_slot(T_prefix, i);
    pos_out[i] = query_pos(T_prefix, i);
  }
}

}  // namespace lat
