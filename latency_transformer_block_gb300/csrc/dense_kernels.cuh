// Prologue / epilogue kernels of the dense path (prefix prefill, DiT stage).
#pragma once
#include "common.cuh"
#include "dense_gemm.cuh"

namespace lat {

// ---------------------------------------------------------------------------
// Norm prologue with the split of the next GEMM's activation into two fp16 planes:
//   RMS:    u = x * rsqrt(mean(x^2) + eps)              (scale g folded into W)
//   LN_MOD: u = LN(x) * (1 + scale_b) + shift_b          (adaLN of chunk b, or a
//           LayerNorm affine: scale = g - 1, shift = b, the same for every b)
//   NONE:   u = x                                        (the planes alone)
//   act[m][c] = fp16(u), act[m][D + c] = fp16(u - act[m][c])
// One CTA of 256 threads per row (norm_split_kernel), or one warp per row for
// D <= 2048 (norm_split_warp_kernel).
// ---------------------------------------------------------------------------
enum NormMode : int { NORM_RMS = 0, NORM_LN_MOD = 1, NORM_NONE = 2 };

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

// The row stays in registers (float4, up to kNormV per thread: D <= 8192) and
// is read once; the planes are written 4 values (8 bytes) at a time.
constexpr int kNormV = 8;

__device__ __forceinline__ uint2 pack_half4(float a, float b, float c, float d) {
  const __half2 x = __floats2half2_rn(a, b), y = __floats2half2_rn(c, d);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&x), *reinterpret_cast<const uint32_t*>(&y));
}

// Columns 4c .. 4c + 3 of a row: normalised (mean mu, factor rs), the adaLN /
// affine rows applied (LN_MOD), stored as the two fp16 planes.
__device__ __forceinline__ void norm_store4(const NormArgs& a, __half* hi, int c, float4 x, float mu, float rs,
                                            const float4* sh, const float4* sc) {
  float w[4] = {(x.x - mu) * rs, (x.y - mu) * rs, (x.z - mu) * rs, (x.w - mu) * rs};
  if (a.mode == NORM_LN_MOD) {
    const float4 k = __ldg(sc + c), t = __ldg(sh + c);
    w[0] = w[0] * (1.f + k.x) + t.x;
    w[1] = w[1] * (1.f + k.y) + t.y;
    w[2] = w[2] * (1.f + k.z) + t.z;
    w[3] = w[3] * (1.f + k.w) + t.w;
  }
  const uint2 h = pack_half4(w[0], w[1], w[2], w[3]);
  const __half2 h01 = *reinterpret_cast<const __half2*>(&h.x), h23 = *reinterpret_cast<const __half2*>(&h.y);
  const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
  *reinterpret_cast<uint2*>(hi + 4 * c) = h;
  *reinterpret_cast<uint2*>(hi + a.D + 4 * c) = pack_half4(w[0] - f01.x, w[1] - f01.y, w[2] - f23.x, w[3] - f23.y);
}

static __global__ void __launch_bounds__(256) norm_split_kernel(NormArgs a) {
  const int m = blockIdx.x;
  const int n4 = a.D / 4;
  const float4* xr = reinterpret_cast<const float4*>(a.x + (size_t)m * a.D);
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
  float4 v[kNormV];
#pragma unroll
  for (int u = 0; u < kNormV; ++u) {
    const int c = threadIdx.x + 256 * u;
    v[u] = c < n4 ? __ldg(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float mu = 0.f, rs;
  if (a.mode == NORM_LN_MOD) {
    float s = 0.f;
#pragma unroll
    for (int u = 0; u < kNormV; ++u) s += (v[u].x + v[u].y) + (v[u].z + v[u].w);
    mu = block_sum(s) / a.D;
    float q = 0.f;
#pragma unroll
    for (int u = 0; u < kNormV; ++u)
      if (threadIdx.x + 256 * u < n4) {
        const float d0 = v[u].x - mu, d1 = v[u].y - mu, d2 = v[u].z - mu, d3 = v[u].w - mu;
        q += (d0 * d0 + d1 * d1) + (d2 * d2 + d3 * d3);
      }
    rs = rsqrtf(block_sum(q) / a.D + a.eps);
  } else if (a.mode == NORM_RMS) {
    float q = 0.f;
#pragma unroll
    for (int u = 0; u < kNormV; ++u) q += (v[u].x * v[u].x + v[u].y * v[u].y) + (v[u].z * v[u].z + v[u].w * v[u].w);
    rs = rsqrtf(block_sum(q) / a.D + a.eps);
  } else {
    rs = 1.f;
  }
  const float4* sh = nullptr;
  const float4* sc = nullptr;
  if (a.mode == NORM_LN_MOD) {
    const int b = m / a.rows_per_chunk;
    sh = reinterpret_cast<const float4*>(a.table + a.shift_off[b]);
    sc = reinterpret_cast<const float4*>(a.table + a.scale_off[b]);
  }
  __half* hi = a.act2 + (size_t)m * kActTerms * a.D;
#pragma unroll
  for (int u = 0; u < kNormV; ++u) {
    const int c = threadIdx.x + 256 * u;
    if (c < n4) norm_store4(a, hi, c, v[u], mu, rs, sh, sc);
  }
}

// The same for rows of D <= 32 * 4 * NV: one warp per row (eight a CTA), the
// row in registers, the sums by warp shuffles alone.  Grid ceil(M / 8).
template <int NV>
static __global__ void __launch_bounds__(256) norm_split_warp_kernel(NormArgs a, int M) {
  const int m = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (m >= M) return;   // whole warps; nothing below synchronises the CTA
  const int n4 = a.D / 4;
  const float4* xr = reinterpret_cast<const float4*>(a.x + (size_t)m * a.D);
  auto warp_sum = [](float v) {
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
  };
  float4 v[NV];
#pragma unroll
  for (int u = 0; u < NV; ++u) {
    const int c = lane + 32 * u;
    v[u] = c < n4 ? __ldg(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float mu = 0.f, rs = 1.f;
  if (a.mode == NORM_LN_MOD) {
    float s = 0.f;
#pragma unroll
    for (int u = 0; u < NV; ++u) s += (v[u].x + v[u].y) + (v[u].z + v[u].w);
    mu = warp_sum(s) / a.D;
    float q = 0.f;
#pragma unroll
    for (int u = 0; u < NV; ++u)
      if (lane + 32 * u < n4) {
        const float d0 = v[u].x - mu, d1 = v[u].y - mu, d2 = v[u].z - mu, d3 = v[u].w - mu;
        q += (d0 * d0 + d1 * d1) + (d2 * d2 + d3 * d3);
      }
    rs = rsqrtf(warp_sum(q) / a.D + a.eps);
  } else if (a.mode == NORM_RMS) {
    float q = 0.f;
#pragma unroll
    for (int u = 0; u < NV; ++u) q += (v[u].x * v[u].x + v[u].y * v[u].y) + (v[u].z * v[u].z + v[u].w * v[u].w);
    rs = rsqrtf(warp_sum(q) / a.D + a.eps);
  }
  const float4* sh = nullptr;
  const float4* sc = nullptr;
  if (a.mode == NORM_LN_MOD) {
    const int b = m / a.rows_per_chunk;
    sh = reinterpret_cast<const float4*>(a.table + a.shift_off[b]);
    sc = reinterpret_cast<const float4*>(a.table + a.scale_off[b]);
  }
  __half* hi = a.act2 + (size_t)m * kActTerms * a.D;
#pragma unroll
  for (int u = 0; u < NV; ++u) {
    const int c = lane + 32 * u;
    if (c < n4) norm_store4(a, hi, c, v[u], mu, rs, sh, sc);
  }
}

// ---------------------------------------------------------------------------
// RoPE + K/V into the cache (prefix prefill).  Input qkv fp32 [M][ld_qkv] =
// [q (Hq*dh) | k | v] (or [k | v] when q_cols == 0).  Row m belongs to batch
// element b = m / T at token j = m % T, position pos0[b] + j.
//   cos/sin(pos * theta_i) = rotation of j (fp32 table built from float64)
//   composed with the rotation of pos0[b] (float64 on the device, per CTA).
// q -> fp32 q_out [M][Hq*dh]; k, v -> bf16 rows j of kdst[b], vdst[b] and the
// two fp16 planes of the values as computed.
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
  __half* kb2;              // K (after RoPE) and V as computed, as two fp16 planes
  __half* vb2;              //   [M][kv_cols] (hi), then lo lo_off elements later
  long long lo_off;
};

// cos / sin of pos0 * theta_i in float64, rounded to fp32 (1, 0 at pos0 = 0)
__device__ __forceinline__ void base_rotation(long long pos0, double theta, float& c, float& s) {
  if (pos0 == 0) {
    c = 1.f;
    s = 0.f;
  } else {
    double sd, cd;
    sincos((double)pos0 * theta, &sd, &cd);
    c = (float)cd;
    s = (float)sd;
  }
}

static __global__ void __launch_bounds__(128) rope_kv_kernel(RopeKvArgs a) {
  const int m = blockIdx.x;
  const int b = m / a.T, j = m % a.T;
  const int half = a.dh / 2;
  __shared__ float cb[128], sb[128];   // rotation of pos0[b], dh/2 <= 128
  for (int i = threadIdx.x; i < half; i += blockDim.x) base_rotation(a.pos0[b], a.theta[i], cb[i], sb[i]);
  __syncthreads();
  const float* row = a.qkv + (size_t)m * a.ld_qkv;
  __nv_bfloat16* krow = a.kdst[b] + (size_t)j * a.kv_ld;   // this token's K and V rows in the cache
  __nv_bfloat16* vrow = a.vdst[b] + (size_t)j * a.kv_ld;
  const float* cj = a.cos_j + (size_t)j * half;
  const float* sj = a.sin_j + (size_t)j * half;
  const int nq = a.q_cols / a.dh, nk = a.kv_cols / a.dh;
  const int h4 = half / 4;
  auto bf4 = [](const float (&y)[4]) {
    const __nv_bfloat162 x = __floats2bfloat162_rn(y[0], y[1]), z = __floats2bfloat162_rn(y[2], y[3]);
    return make_uint2(*reinterpret_cast<const uint32_t*>(&x), *reinterpret_cast<const uint32_t*>(&z));
  };
  // 4 RoPE pairs (i .. i+3, i+half .. i+half+3) of one head per item: float4
  // loads, 8- or 16-byte stores
  for (int p = threadIdx.x; p < (nq + nk) * h4; p += blockDim.x) {
    const int head = p / h4, i = (p % h4) * 4;
    const int col = head * a.dh + i;   // within q, or within k when head >= nq
    const float4 cv = *reinterpret_cast<const float4*>(cj + i), sv = *reinterpret_cast<const float4*>(sj + i);
    const float4 v0 = *reinterpret_cast<const float4*>(row + col);
    const float4 v1 = *reinterpret_cast<const float4*>(row + col + half);
    const float cjj[4] = {cv.x, cv.y, cv.z, cv.w}, sjj[4] = {sv.x, sv.y, sv.z, sv.w};
    const float x0[4] = {v0.x, v0.y, v0.z, v0.w}, x1[4] = {v1.x, v1.y, v1.z, v1.w};
    float y0[4], y1[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float c = cjj[e] * cb[i + e] - sjj[e] * sb[i + e];
      const float s = sjj[e] * cb[i + e] + cjj[e] * sb[i + e];
      y0[e] = x0[e] * c - x1[e] * s;
      y1[e] = x1[e] * c + x0[e] * s;
    }
    if (head < nq) {
      float* qo = a.q_out + (size_t)m * a.q_cols + col;
      *reinterpret_cast<float4*>(qo) = make_float4(y0[0], y0[1], y0[2], y0[3]);
      *reinterpret_cast<float4*>(qo + half) = make_float4(y1[0], y1[1], y1[2], y1[3]);
    } else {
      __nv_bfloat16* kr = krow + (col - a.q_cols);
      *reinterpret_cast<uint2*>(kr) = bf4(y0);
      *reinterpret_cast<uint2*>(kr + half) = bf4(y1);
      __half* kp = a.kb2 + (size_t)m * a.kv_cols + (col - a.q_cols);
      uint2 h, l;
      split_pair_h2(y0[0], y0[1], h.x, l.x);
      split_pair_h2(y0[2], y0[3], h.y, l.y);
      *reinterpret_cast<uint2*>(kp) = h;
      *reinterpret_cast<uint2*>(kp + a.lo_off) = l;
      split_pair_h2(y1[0], y1[1], h.x, l.x);
      split_pair_h2(y1[2], y1[3], h.y, l.y);
      *reinterpret_cast<uint2*>(kp + half) = h;
      *reinterpret_cast<uint2*>(kp + half + a.lo_off) = l;
    }
  }
  const float* vr = row + a.q_cols + a.kv_cols;
  for (int c = 4 * threadIdx.x; c < a.kv_cols; c += 4 * blockDim.x) {
    const float4 t = *reinterpret_cast<const float4*>(vr + c);
    const float y[4] = {t.x, t.y, t.z, t.w};
    *reinterpret_cast<uint2*>(vrow + c) = bf4(y);
    __half* vp = a.vb2 + (size_t)m * a.kv_cols + c;
    uint2 h, l;
    split_pair_h2(y[0], y[1], h.x, l.x);
    split_pair_h2(y[2], y[3], h.y, l.y);
    *reinterpret_cast<uint2*>(vp) = h;
    *reinterpret_cast<uint2*>(vp + a.lo_off) = l;
  }
}

// ---------------------------------------------------------------------------
// Rotation of every row of a DiT call (dh = 128), the table the E_ROPE_KV
// epilogue of the QKV projection reads: row m (token j = m % T of chunk
// b = m / T) turns pair i by cos/sin(pos0[b] theta_i) (float64 on the device)
// composed with the token's own cos_j / sin_j (the 1-D position j, or the
// frame-within-chunk, row and column of a video token).  Output per 32-row
// group g: [2][16][32] float4, (cos | sin) of pairs 4i .. 4i + 3 of row 32g + r,
// so that a warp holding rows 32g .. 32g + 31 reads each float4 row coalesced.
// Rows m >= M of the last group repeat row M - 1.  Grid ceil(M / 32), blockDim 256.
// ---------------------------------------------------------------------------
struct RopeRowsArgs {
  int M, T, n;              // rows, rows per chunk, chunks
  const float* cos_j;       // [T][64]
  const float* sin_j;
  const double* theta;      // [64] the per-pair frequency the chunk's base position turns by
  long long pos0[kMaxChunks];
  float4* rot;
};

static __global__ void __launch_bounds__(256) rope_rows_kernel(RopeRowsArgs a) {
  const int m0 = blockIdx.x * 32, b0 = m0 / a.T;
  __shared__ float cb[2][64], sb[2][64];   // base rotations of chunks b0, b0 + 1
  if (threadIdx.x < 128) {
    const int k = threadIdx.x >> 6, i = threadIdx.x & 63, b = min(b0 + k, a.n - 1);
    base_rotation(a.pos0[b], a.theta[i], cb[k][i], sb[k][i]);
  }
  __syncthreads();
  float4* out = a.rot + (size_t)blockIdx.x * 1024;
  for (int it = threadIdx.x; it < 512; it += blockDim.x) {
    const int r = it & 31, i = 4 * (it >> 5);
    const int m = min(m0 + r, a.M - 1), b = m / a.T, j = m - b * a.T;
    const float4 cv = *reinterpret_cast<const float4*>(a.cos_j + (size_t)j * 64 + i);
    const float4 sv = *reinterpret_cast<const float4*>(a.sin_j + (size_t)j * 64 + i);
    const float cjj[4] = {cv.x, cv.y, cv.z, cv.w}, sjj[4] = {sv.x, sv.y, sv.z, sv.w};
    float c[4], s[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float bc, bs;
      if (b - b0 < 2) {
        bc = cb[b - b0][i + e];
        bs = sb[b - b0][i + e];
      } else {   // chunks shorter than 32 rows: a group spans more than two
        base_rotation(a.pos0[b], a.theta[i + e], bc, bs);
      }
      c[e] = cjj[e] * bc - sjj[e] * bs;
      s[e] = sjj[e] * bc + cjj[e] * bs;
    }
    out[(it >> 5) * 32 + r] = make_float4(c[0], c[1], c[2], c[3]);
    out[512 + (it >> 5) * 32 + r] = make_float4(s[0], s[1], s[2], s[3]);
  }
}

// K | V rows as computed (fp32 [rows][2 cols]) -> [rows][K hi | K lo | V hi | V lo]
// fp16 planes, the layout the tensor-core attention reads its non-cached keys in
// (the text context's keys and values of a cross-attention).
static __global__ void __launch_bounds__(256) kv_planes_kernel(const float* kv, int rows, int cols, __half* out) {
  const size_t n4 = (size_t)rows * 2 * cols / 4;
  for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < n4; i += (size_t)gridDim.x * 256) {
    const size_t e = 4 * i, r = e / (2 * cols), c = e % (2 * cols);
    const float4 v = *reinterpret_cast<const float4*>(kv + e);
    const uint2 h = pack_half4(v.x, v.y, v.z, v.w);
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
    const size_t o = r * 4 * cols + (c < (size_t)cols ? c : cols + c);   // K at 0.., V at 2 cols..
    *reinterpret_cast<uint2*>(out + o) = h;
    *reinterpret_cast<uint2*>(out + o + cols) = pack_half4(v.x - f0.x, v.y - f0.y, v.z - f1.x, v.w - f1.y);
  }
}

}  // namespace lat
