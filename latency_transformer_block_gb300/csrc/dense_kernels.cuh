// Prologue / epilogue kernels of the dense path (prefix prefill, DiT stage).
#pragma once
#include "common.cuh"
#include "dense_gemm.cuh"

namespace lat {

// ---------------------------------------------------------------------------
// Norm prologue with the split of the next GEMM's activation into two fp16 planes:
//   RMS:    u = x * rsqrt(mean(x^2) + eps)              (scale g folded into W)
//   LN_MOD: u = LN(x) * (1 + scale_b) + shift_b          (adaLN of chunk b)
//   act[m][c] = fp16(u), act[m][D + c] = fp16(u - act[m][c])
// One CTA of 256 threads per row.
// ---------------------------------------------------------------------------
enum NormMode : int { NORM_RMS = 0, NORM_LN_MOD = 1 };

struct NormArgs {
  const float* x;
  int D;
  int mode;
  float eps;
  const float* table;      // LN_MOD: adaLN table [S][6D]
  int shift_off[kMaxChunks];  // LN_MOD: table offset of chunk b's shift row
  int scale_off[kMaxChunks];
  int rows_per_chunk;
  __half* act2;            // [M][kActTerms * D]
};

static __global__ void __launch_bounds__(256) norm_split_kernel(NormArgs a) {
  const int m = blockIdx.x;
  const float* xr = a.x + (size_t)m * a.D;
  __shared__ float red[8];
  __shared__ float stat[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto block_sum = [&](float v) {
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float s = 0.f;
    if (threadIdx.x == 0) {
      for (int w = 0; w < 8; ++w) s += red[w];
      stat[0] = s;
    }
    __syncthreads();
    s = stat[0];
    __syncthreads();
    return s;
  };
  float mu = 0.f, rs;
  if (a.mode == NORM_LN_MOD) {
    float s = 0.f;
    for (int c = threadIdx.x; c < a.D; c += 256) s += xr[c];
    mu = block_sum(s) / a.D;
    float v = 0.f;
    for (int c = threadIdx.x; c < a.D; c += 256) {
      const float d = xr[c] - mu;
      v += d * d;
    }
    rs = rsqrtf(block_sum(v) / a.D + a.eps);
  } else {
    float s = 0.f;
    for (int c = threadIdx.x; c < a.D; c += 256) s += xr[c] * xr[c];
    rs = rsqrtf(block_sum(s) / a.D + a.eps);
  }
  const float* sh = nullptr;
  const float* sc = nullptr;
  if (a.mode == NORM_LN_MOD) {
    const int b = m / a.rows_per_chunk;
    sh = a.table + a.shift_off[b];
    sc = a.table + a.scale_off[b];
  }
  __half* hi = a.act2 + (size_t)m * kActTerms * a.D;
  for (int c = threadIdx.x; c < a.D; c += 256) {
    float u = (xr[c] - mu) * rs;
    if (a.mode == NORM_LN_MOD) u = u * (1.f + sc[c]) + sh[c];
    const __half h = __float2half_rn(u);
    hi[c] = h;
    hi[a.D + c] = __float2half_rn(u - __half2float(h));
  }
}

// ---------------------------------------------------------------------------
// RoPE + K/V into the cache.  Input qkv fp32 [M][ld_qkv] = [q (Hq*dh) | k | v]
// (or [k | v] when q_cols == 0).  Row m belongs to group b = m / T (a chunk or a
// batch element) at token j = m % T, position pos0[b] + j.
//   cos/sin(pos * theta_i) = rotation of j (fp32 table built from float64)
//   composed with the rotation of pos0[b] (float64 on the device, per CTA).
// q -> fp32 q_out [M][Hq*dh]; k, v -> bf16 rows j of kdst[b], vdst[b].
// Grid M, blockDim 128.
// ---------------------------------------------------------------------------
struct RopeKvArgs {
  const float* qkv;
  int ld_qkv;
  int q_cols;               // Hq * dh (0: no q)
  int kv_cols;              // Hkv * dh
  int dh;
  int T;
  const float* cos_j;       // [T][dh/2]
  const float* sin_j;
  const double* theta;      // [dh/2] base^(-2i/dh) in float64
  long long pos0[kMaxChunks];
  float* q_out;
  __nv_bfloat16* kdst[kMaxChunks];
  __nv_bfloat16* vdst[kMaxChunks];
  int kv_ld;                // row stride of kdst / vdst (elements)
  float* k32;               // fp32 K (after RoPE) and V as computed, [M][kv_cols], or
  float* v32;
  __half* k16;              // the same as two fp16 planes (hi at column c, lo at kv_cols + c)
  __half* v16;              // of rows ld16 apart
  int ld16;
};

static __global__ void __launch_bounds__(128) rope_kv_kernel(RopeKvArgs a) {
  const int m = blockIdx.x;
  const int b = m / a.T, j = m % a.T;
  const int half = a.dh / 2;
  __shared__ float cb[128], sb[128];   // rotation of pos0[b], dh/2 <= 128
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    if (a.pos0[b] == 0) {
      cb[i] = 1.f;
      sb[i] = 0.f;
    } else {
      double s, c;
      sincos((double)a.pos0[b] * a.theta[i], &s, &c);
      cb[i] = (float)c;
      sb[i] = (float)s;
    }
  }
  __syncthreads();
  const float* row = a.qkv + (size_t)m * a.ld_qkv;
  const float* cj = a.cos_j + (size_t)j * half;
  const float* sj = a.sin_j + (size_t)j * half;
  const int nq = a.q_cols / a.dh, nk = a.kv_cols / a.dh;
  for (int p = threadIdx.x; p < (nq + nk) * half; p += blockDim.x) {
    const int head = p / half, i = p % half;
    const float c = cj[i] * cb[i] - sj[i] * sb[i];
    const float s = sj[i] * cb[i] + cj[i] * sb[i];
    const int col = head * a.dh + i;   // within q, or within k when head >= nq
    const float x0 = row[col], x1 = row[col + half];
    const float y0 = x0 * c - x1 * s, y1 = x1 * c + x0 * s;
    if (head < nq) {
      float* qo = a.q_out + (size_t)m * a.q_cols + col;
      qo[0] = y0;
      qo[half] = y1;
    } else {
      __nv_bfloat16* kr = a.kdst[b] + (size_t)j * a.kv_ld + (col - a.q_cols);
      kr[0] = __float2bfloat16_rn(y0);
      kr[half] = __float2bfloat16_rn(y1);
      if (a.k16) {
        __half* k16 = a.k16 + (size_t)m * a.ld16 + (col - a.q_cols);
        const __half h0 = __float2half_rn(y0), h1 = __float2half_rn(y1);
        k16[0] = h0;
        k16[half] = h1;
        k16[a.kv_cols] = __float2half_rn(y0 - __half2float(h0));
        k16[a.kv_cols + half] = __float2half_rn(y1 - __half2float(h1));
      } else {
        float* k32 = a.k32 + (size_t)m * a.kv_cols + (col - a.q_cols);
        k32[0] = y0;
        k32[half] = y1;
      }
    }
  }
  const float* vr = row + a.q_cols + a.kv_cols;
  for (int c = threadIdx.x; c < a.kv_cols; c += blockDim.x) {
    a.vdst[b][(size_t)j * a.kv_ld + c] = __float2bfloat16_rn(vr[c]);
    if (a.v16) {
      __half* v16 = a.v16 + (size_t)m * a.ld16 + c;
      const __half h = __float2half_rn(vr[c]);
      v16[0] = h;
      v16[a.kv_cols] = __float2half_rn(vr[c] - __half2float(h));
    } else {
      a.v32[(size_t)m * a.kv_cols + c] = vr[c];
    }
  }
}

}  // namespace lat
