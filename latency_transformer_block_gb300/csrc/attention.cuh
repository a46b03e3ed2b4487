// Chunk-over-cached-KV attention: softmax(Q K^T / sqrt(dh)) V, no mask, with
// grouped KV heads (Hkv = 1 is the pi0 multi-query case: all query heads read
// the one cached head).  "Running VLAs at Real-time Speed" (reading note,
// section 5) keeps a library attention here; this is a hand-written one.
//
// Each CTA runs 4 warps x 16 query rows of one query head against a range of
// 64-key blocks with an online softmax (running max / sum per row, rescaling
// the output accumulator).  Q (fp32) and P (fp32) enter the warp-level bf16
// tensor-core MMA as three-term splits; cached K and V are bf16 values; the
// block's own keys (index >= own0) come in fp32 as computed and are split into
// two bf16 planes (hi, lo) in shared memory; accumulation is fp32.  With
// several key ranges (flash-decoding) each CTA writes its partial (max, sum,
// unnormalised output) and a combine kernel merges them.
#pragma once
#include "common.cuh"

namespace lat {

struct AttnArgs {
  const float* q;            // fp32 [T_q][q_ld], head h at column h*dh
  int q_ld;
  const __nv_bfloat16* k;    // bf16 keys [T_kv][kv_ld], kv head j at column j*dh
  const __nv_bfloat16* v;
  int kv_ld;
  int T_q, T_kv, Hq, Hkv;
  float scale_log2;          // log2(e) / sqrt(dh)
  int n_split;               // key ranges
  float* out;                // n_split == 1: fp32 [T_q][out_ld] (head h at h*dh)
  int out_ld;
  float* part_m;             // n_split > 1: [n_split][Hq][T_q]
  float* part_l;
  float* part_o;             // [n_split][Hq][T_q][dh]
  const float* k_own;        // fp32 keys own0.. [T_kv - own0][own_ld] (null: none)
  const float* v_own;
  int own0;
  int own_ld;
  int force_partials;        // write partials even with one key range (combine follows)
};

// 8 fp32 values -> 8 bf16 hi and 8 bf16 lo (two-term split)
__device__ __forceinline__ void split8_to(const float* src, uint4& hi, uint4& lo) {
  const float4 a = *reinterpret_cast<const float4*>(src);
  const float4 b = *reinterpret_cast<const float4*>(src + 4);
  uint32_t h[4], l[4];
  split_pair2(a.x, a.y, h[0], l[0]);
  split_pair2(a.z, a.w, h[1], l[1]);
  split_pair2(b.x, b.y, h[2], l[2]);
  split_pair2(b.z, b.w, h[3], l[3]);
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// 16-byte async copy global -> shared; src_bytes = 0 fills zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Keys per block of the chunk attention (and per key range when every range
// holds one block).
constexpr int kAttnKB = 32;
__host__ __device__ constexpr int attn_key_blocks(int T_kv) { return (T_kv + kAttnKB - 1) / kAttnKB; }

// Eight warps per CTA: warp w takes query rows (w & 3) * 16 .. +15 of the CTA's
// 64 and half (w >> 2) of the head dimension.  Scores are summed over the two
// halves through shared memory, so both warps of a row tile hold the same S and
// the same P; each accumulates the output columns of its half.
//   S = (q_hi + q_lo) k              cached keys (bf16 values)
//   S = (q_hi + q_lo) k_hi + q_hi k_lo   own keys (fp32 as computed, two planes)
//   O += (p_hi + p_lo) v  /  (p_hi + p_lo) v_hi + p_hi v_lo
// The dropped products (q_lo k_lo, p_lo v_lo) are below 2^-16 of the kept ones.
template <int DH>
static __global__ void __launch_bounds__(256) attention_kernel(AttnArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int KB = kAttnKB;
  constexpr int LD = DH + 8;      // padded smem row (bf16): conflict-free ldmatrix
  constexpr int HD = DH / 2;      // dims per warp
  constexpr int KS = HD / 16;     // k-steps of S per warp
  constexpr int NT = HD / 8;      // output n-tiles per warp
  constexpr int SLD = KB + 2;     // partial-score row (fp32)
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(smem_raw);   // [2 planes][KB][LD]
  __nv_bfloat16* sV = sK + 2 * KB * LD;
  float* sS = reinterpret_cast<float*>(sV + 2 * KB * LD);            // [8 warps][16][SLD]

  const int h = blockIdx.x;
  const int qt = blockIdx.y;
  const int split = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int rt = warp & 3, half = warp >> 2;
  const int d0 = half * HD;
  const int kvh = h / (a.Hq / a.Hkv);
  const int nkb = attn_key_blocks(a.T_kv);
  const int kb0 = split * nkb / a.n_split, kb1 = (split + 1) * nkb / a.n_split;

  const int r0 = qt * 64 + rt * 16 + g;   // this thread's two query rows: r0, r0 + 8
  const int r1 = r0 + 8;
  const bool v0 = r0 < a.T_q, v1 = r1 < a.T_q;

  // Q fragments of this warp's rows and dims, split once (rows past T_q are 0)
  uint32_t qh[KS][4], ql[KS][4];
  {
    const float* q0 = a.q + (size_t)(v0 ? r0 : 0) * a.q_ld + h * DH + d0 + 2 * tq;
    const float* q1 = a.q + (size_t)(v1 ? r1 : 0) * a.q_ld + h * DH + d0 + 2 * tq;
    float2 x[KS][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      x[ks][0] = v0 ? *reinterpret_cast<const float2*>(q0 + ks * 16) : make_float2(0.f, 0.f);
      x[ks][1] = v1 ? *reinterpret_cast<const float2*>(q1 + ks * 16) : make_float2(0.f, 0.f);
      x[ks][2] = v0 ? *reinterpret_cast<const float2*>(q0 + ks * 16 + 8) : make_float2(0.f, 0.f);
      x[ks][3] = v1 ? *reinterpret_cast<const float2*>(q1 + ks * 16 + 8) : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int e = 0; e < 4; ++e) split_pair2(x[ks][e].x, x[ks][e].y, qh[ks][e], ql[ks][e]);
  }

  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  const uint32_t sKa = smem_u32(sK), sVa = smem_u32(sV);
  const uint32_t LO = (uint32_t)(KB * LD * 2);   // byte offset of the lo plane
  float* myS = sS + warp * 16 * SLD;
  const float* peerS = sS + (warp ^ 4) * 16 * SLD;

  for (int kb = kb0; kb < kb1; ++kb) {
    // ---- stage K and V blocks (zero-filled past T_kv); own keys as hi + lo ----
    const bool has_lo = a.k_own != nullptr && (kb + 1) * KB > a.own0 && a.own0 < a.T_kv;
    __syncthreads();
    for (int idx = threadIdx.x; idx < KB * (DH / 8); idx += 256) {
      const int row = idx / (DH / 8), c8 = idx % (DH / 8);
      const int key = kb * KB + row;
      const bool own = a.k_own != nullptr && key >= a.own0 && key < a.T_kv;
      if (!own) {   // cache keys (and zero fill past T_kv) by async copy
        const bool in = key < a.T_kv;
        const size_t off = (size_t)(in ? key : 0) * a.kv_ld + kvh * DH + c8 * 8;
        cp_async16(sK + row * LD + c8 * 8, a.k + off, in ? 16 : 0);
        cp_async16(sV + row * LD + c8 * 8, a.v + off, in ? 16 : 0);
        if (has_lo) {
          *reinterpret_cast<uint4*>(sK + KB * LD + row * LD + c8 * 8) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(sV + KB * LD + row * LD + c8 * 8) = make_uint4(0, 0, 0, 0);
        }
      } else {      // own keys as computed: hi and lo planes
        const size_t off = (size_t)(key - a.own0) * a.own_ld + kvh * DH + c8 * 8;
        uint4 kk, kl, vv, vl;
        split8_to(a.k_own + off, kk, kl);
        split8_to(a.v_own + off, vv, vl);
        *reinterpret_cast<uint4*>(sK + row * LD + c8 * 8) = kk;
        *reinterpret_cast<uint4*>(sK + KB * LD + row * LD + c8 * 8) = kl;
        *reinterpret_cast<uint4*>(sV + row * LD + c8 * 8) = vv;
        *reinterpret_cast<uint4*>(sV + KB * LD + row * LD + c8 * 8) = vl;
      }
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- partial S over this warp's dims: 16 rows x 32 keys (4 n-tiles) ----
    float sa[4][4], sb[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) sa[j][e] = sb[j][e] = 0.f;
    const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t b[4][2];
#pragma unroll
      for (int jp = 0; jp < 2; ++jp) {
        const int key = jp * 16 + ((mi >> 1) << 3) + rr;
        const int col = d0 + ks * 16 + ((mi & 1) << 3);
        ldsm_x4(sKa + (uint32_t)(key * LD + col) * 2u, b[2 * jp][0], b[2 * jp][1], b[2 * jp + 1][0],
                b[2 * jp + 1][1]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) mma_16816(sa[j], qh[ks], b[j][0], b[j][1]);
#pragma unroll
      for (int j = 0; j < 4; ++j) mma_16816(sb[j], ql[ks], b[j][0], b[j][1]);
      if (has_lo) {
#pragma unroll
        for (int jp = 0; jp < 2; ++jp) {
          const int key = jp * 16 + ((mi >> 1) << 3) + rr;
          const int col = d0 + ks * 16 + ((mi & 1) << 3);
          ldsm_x4(sKa + LO + (uint32_t)(key * LD + col) * 2u, b[2 * jp][0], b[2 * jp][1], b[2 * jp + 1][0],
                  b[2 * jp + 1][1]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_16816(sb[j], qh[ks], b[j][0], b[j][1]);
      }
    }
    // ---- exchange partial scores with the warp of the other half ----
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = j * 8 + 2 * tq;
      *reinterpret_cast<float2*>(myS + g * SLD + c) = make_float2(sa[j][0] + sb[j][0], sa[j][1] + sb[j][1]);
      *reinterpret_cast<float2*>(myS + (g + 8) * SLD + c) = make_float2(sa[j][2] + sb[j][2], sa[j][3] + sb[j][3]);
    }
    __syncthreads();
    float s[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = j * 8 + 2 * tq;
      const float2 p0 = *reinterpret_cast<const float2*>(peerS + g * SLD + c);
      const float2 p1 = *reinterpret_cast<const float2*>(peerS + (g + 8) * SLD + c);
      // a + b == b + a: both warps of the pair get bit-identical scores
      s[j][0] = (sa[j][0] + sb[j][0]) + p0.x;
      s[j][1] = (sa[j][1] + sb[j][1]) + p0.y;
      s[j][2] = (sa[j][2] + sb[j][2]) + p1.x;
      s[j][3] = (sa[j][3] + sb[j][3]) + p1.y;
    }

    // ---- online softmax (base 2) ----
    float mx0 = m0, mx1 = m1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int key = kb * KB + j * 8 + 2 * tq;
      s[j][0] = (key < a.T_kv) ? s[j][0] * a.scale_log2 : -INFINITY;
      s[j][1] = (key + 1 < a.T_kv) ? s[j][1] * a.scale_log2 : -INFINITY;
      s[j][2] = (key < a.T_kv) ? s[j][2] * a.scale_log2 : -INFINITY;
      s[j][3] = (key + 1 < a.T_kv) ? s[j][3] * a.scale_log2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][1]));
      mx1 = fmaxf(mx1, fmaxf(s[j][2], s[j][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float al0 = exp2f(m0 - mx0), al1 = exp2f(m1 - mx1);
    m0 = mx0;
    m1 = mx1;
    float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      s[j][0] = exp2f(s[j][0] - mx0);
      s[j][1] = exp2f(s[j][1] - mx0);
      s[j][2] = exp2f(s[j][2] - mx1);
      s[j][3] = exp2f(s[j][3] - mx1);
      sum0 += s[j][0] + s[j][1];
      sum1 += s[j][2] + s[j][3];
    }
    sum0 += __shfl_xor_sync(0xffffffffu, sum0, 1);
    sum0 += __shfl_xor_sync(0xffffffffu, sum0, 2);
    sum1 += __shfl_xor_sync(0xffffffffu, sum1, 1);
    sum1 += __shfl_xor_sync(0xffffffffu, sum1, 2);
    l0 = l0 * al0 + sum0;
    l1 = l1 * al1 + sum1;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      o[j][0] *= al0;
      o[j][1] *= al0;
      o[j][2] *= al1;
      o[j][3] *= al1;
    }

    // ---- O += P V over this warp's output columns ----
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint32_t ph[4], pl[4];
      split_pair2(s[2 * kk][0], s[2 * kk][1], ph[0], pl[0]);
      split_pair2(s[2 * kk][2], s[2 * kk][3], ph[1], pl[1]);
      split_pair2(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pl[2]);
      split_pair2(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pl[3]);
      const int key = kk * 16 + ((mi & 1) << 3) + rr;
      uint32_t b[NT][2];
#pragma unroll
      for (int jp = 0; jp < NT / 2; ++jp) {
        const int col = d0 + jp * 16 + ((mi >> 1) << 3);
        ldsm_x4_t(sVa + (uint32_t)(key * LD + col) * 2u, b[2 * jp][0], b[2 * jp][1], b[2 * jp + 1][0],
                  b[2 * jp + 1][1]);
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) mma_16816(o[j], ph, b[j][0], b[j][1]);
#pragma unroll
      for (int j = 0; j < NT; ++j) mma_16816(o[j], pl, b[j][0], b[j][1]);
      if (has_lo) {
#pragma unroll
        for (int jp = 0; jp < NT / 2; ++jp) {
          const int col = d0 + jp * 16 + ((mi >> 1) << 3);
          ldsm_x4_t(sVa + LO + (uint32_t)(key * LD + col) * 2u, b[2 * jp][0], b[2 * jp][1], b[2 * jp + 1][0],
                    b[2 * jp + 1][1]);
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_16816(o[j], ph, b[j][0], b[j][1]);
      }
    }
  }

  // ---- write out ----
  if (a.n_split == 1 && !a.force_partials) {
    const float i0 = (l0 > 0.f) ? 1.f / l0 : 0.f, i1 = (l1 > 0.f) ? 1.f / l1 : 0.f;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int c = h * DH + d0 + j * 8 + 2 * tq;
      if (v0) *reinterpret_cast<float2*>(a.out + (size_t)r0 * a.out_ld + c) = make_float2(o[j][0] * i0, o[j][1] * i0);
      if (v1) *reinterpret_cast<float2*>(a.out + (size_t)r1 * a.out_ld + c) = make_float2(o[j][2] * i1, o[j][3] * i1);
    }
  } else {
    const size_t base = ((size_t)split * a.Hq + h) * a.T_q;
    if (tq == 0 && half == 0) {
      if (v0) { a.part_m[base + r0] = m0; a.part_l[base + r0] = l0; }
      if (v1) { a.part_m[base + r1] = m1; a.part_l[base + r1] = l1; }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int c = d0 + j * 8 + 2 * tq;
      if (v0) *reinterpret_cast<float2*>(a.part_o + (base + r0) * DH + c) = make_float2(o[j][0], o[j][1]);
      if (v1) *reinterpret_cast<float2*>(a.part_o + (base + r1) * DH + c) = make_float2(o[j][2], o[j][3]);
    }
  }
}

// Merge key-range partials: o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
// Grid (T_q, Hq), blockDim = dh.  With planes != null the result is written as
// the three bf16 planes [3][64][Hq*dh] of the output projection's activation.
static __global__ void attention_combine_kernel(AttnArgs a, int dh, __nv_bfloat16* planes) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  constexpr int MAXS = 32;
  __shared__ float sw[MAXS];
  __shared__ float sL;
  // every partial's output value is requested before any is used
  float ov[MAXS];
#pragma unroll
  for (int s = 0; s < MAXS; ++s) {
    const int sc = s < a.n_split ? s : 0;
    ov[s] = __ldcg(a.part_o + (((size_t)sc * a.Hq + h) * a.T_q + t) * dh + d);
  }
  if (d < 32) {   // weights 2^(m_s - M) of the key ranges, and L
    const bool in = d < a.n_split;
    const size_t i = ((size_t)(in ? d : 0) * a.Hq + h) * a.T_q + t;
    const float mv = in ? __ldcg(a.part_m + i) : -INFINITY;
    const float lv = in ? __ldcg(a.part_l + i) : 0.f;
    float M = mv;
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = (mv == -INFINITY) ? 0.f : exp2f(mv - M);
    float L = w * lv;
    for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    sw[d] = w;
    if (d == 0) sL = L;
  }
  __syncthreads();
  float acc = 0.f;
#pragma unroll
  for (int s = 0; s < MAXS; ++s)
    if (s < a.n_split) acc += sw[s] * ov[s];
  const float o = acc / sL;
  if (planes) {
    const int K = a.Hq * dh, c = h * dh + d;
    const Split3 s3 = split3(o);
    planes[(size_t)t * K + c] = s3.hi;
    planes[(size_t)(64 + t) * K + c] = s3.mid;
    planes[(size_t)(128 + t) * K + c] = s3.lo;
  } else {
    a.out[(size_t)t * a.out_ld + h * dh + d] = o;
  }
}


// ---------------------------------------------------------------------------
// Segmented attention for the dense path.  Group b (a DiT chunk or a prefill
// batch element) has T_rows query rows starting at row b * T_rows of q and up
// to kMaxSeg key segments (ring slots of the noisy history plus its own slot,
// or the prefix cache); keys of a segment are rows 0..n-1 of k/v with stride
// kv_ld.  Q and P enter the MMA as TERMS-term bf16 splits; fp32 segments (the
// group's own keys as computed) as two bf16 planes.  The output of row r, head
// h, dim d goes to the two fp16 planes out[r][t*ldh + h*DH + d] (hi, lo of the
// fp32 value) -- the split activation of the output projection.
// Grid (Hq, ceil(T_rows / 64), groups).
// ---------------------------------------------------------------------------
constexpr int kMaxSeg = 5;

struct AttnSeg {
  const __nv_bfloat16* k;    // bf16 keys (cache; tensor-core kernel: their fp16 copy kh / vh), or
  const __nv_bfloat16* v;
  const __half* kb2;         // keys as computed (own tokens) as two fp16 planes (hi, then lo
  const __half* vb2;         //   lo_off elements later; rows of kv_ld), or
  int n;
  const __half* k16;         // the same as two fp16 planes per key row (hi at column c,
  const __half* v16;         // lo at kv_ld + c; row stride 4 kv_ld): tensor-core kernel
  const __half* kh;          // cached keys / values converted to fp16 (rows of kv_ld),
  const __half* vh;          //   read by the tensor-core kernel
  long long lo_off;          // kb2 / vb2: elements from the hi plane to the lo plane
};

struct SegGroup {
  int nseg;
  AttnSeg seg[kMaxSeg];
};

struct SegAttnArgs {
  const float* q;            // fp32 [groups * T_rows][q_ld]
  int q_ld;
  int T_rows;
  int Hq, Hkv, kv_ld;
  float scale_log2;
  __half* out;               // fp16 planes [groups * T_rows][kActTerms * ldh]
  int ldh;
  unsigned long long* trace; // null, or per-block timestamps of CTA (0, 0, 0) (tensor-core kernel)
  const __half* hist16;      // tensor-core kernel: base of the fp16 history copy (kh / vh are rows of it),
  int hist_rows;             //   its rows,
  const __half* own16;       //   and the base of the own fp16 planes
  int own_rows;              //   its rows (0: the context's dense-path workspace rows)
  // prefix attention with kv_split > 1 key ranges per (head, query tile, group):
  // blockIdx.z = group * kv_split + range; each range leaves its unnormalised
  // output and row (max, sum) in part_o [z][Hq][T_rows][dh] / part_ml [z][Hq][T_rows][2]
  int kv_split;
  float* part_o;
  float* part_ml;
  // tensor-core kernel: a 1-D grid of work items over the tiles (query tile
  // fastest, then head, then group).  Tiles 0 .. tc_whole - 1 run whole; each
  // later tile is cut into tc_pieces key ranges (one item each) that leave
  // their unnormalised output and row (max, sum) in tc_part_o [piece][128][128]
  // / tc_part_ml [piece][128][2], piece = item - tc_whole, for the combine.
  int tc_whole, tc_pieces;
  float* tc_part_o;
  float* tc_part_ml;
  SegGroup grp[16];
};

// fp16 operands, fp32 accumulation
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Attention of the prefix tokens over their own K/V (prefix prefill; the
// segments of a group must be own-key segments, kb2 / vb2 set), warp MMA
// m16n8k16 with fp16 operands and fp32 accumulation.  Operands as two fp16
// terms: q and P (hi = fp16(x), lo = fp16(x - hi)) and the own K / V as the
// two fp16 planes the RoPE kernel wrote:
//   S = q_hi K_hi + q_lo K_hi + q_hi K_lo,   O = P_hi V_hi + P_lo V_hi + P_hi V_lo
// (the dropped lo x lo products are below 2^-22 of the kept ones).  One CTA =
// one (head, 64-row query tile, group), 4 warps of 16 rows; keys in blocks of
// KB, both planes of K and V by async copies.  The K/V tiles are all of the
// shared memory: with KB = 32 (67.6 KB for dh = 256) two CTAs share an SM (255
// registers a thread: two CTAs fill the register file) and hide each other's
// latency; KB = 64 (135 KB, one CTA per SM) syncs half as often, for grids
// that have no more CTAs than SMs.
template <int DH, int KB>
static __global__ void __launch_bounds__(128) attention_seg_kernel(const __grid_constant__ SegAttnArgs a) {
  constexpr int LD = DH + 8;
  constexpr int NT = DH / 8;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __half* sK = reinterpret_cast<__half*>(smem_raw);   // [2 planes][KB][LD]
  __half* sV = sK + 2 * KB * LD;
  __half* sQ = sV + 2 * KB * LD;                      // the CTA's 64 q rows as [2 planes][64][LD]
  const uint32_t LO = (uint32_t)(KB * LD * 2);
  const int h = blockIdx.x, qt = blockIdx.y, b = blockIdx.z / a.kv_split, kr = blockIdx.z % a.kv_split;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int kvh = h / (a.Hq / a.Hkv);
  const int rl0 = qt * 64 + warp * 16 + g, rl1 = rl0 + 8;     // rows within the group
  const bool v0 = rl0 < a.T_rows, v1 = rl1 < a.T_rows;
  const size_t row0 = (size_t)b * a.T_rows + (v0 ? rl0 : 0), row1 = (size_t)b * a.T_rows + (v1 ? rl1 : 0);

  // the q rows of this CTA, once: two fp16 planes (hi = fp16(q), lo = fp16(q - hi))
  for (int idx = threadIdx.x; idx < 64 * (DH / 4); idx += 128) {
    const int row = idx / (DH / 4), c4 = (idx % (DH / 4)) * 4;
    const int rl = qt * 64 + row;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (rl < a.T_rows) v = *reinterpret_cast<const float4*>(a.q + ((size_t)b * a.T_rows + rl) * a.q_ld + h * DH + c4);
    uint32_t h0, l0, h1, l1;
    split_pair_h2(v.x, v.y, h0, l0);
    split_pair_h2(v.z, v.w, h1, l1);
    *reinterpret_cast<uint2*>(sQ + row * LD + c4) = make_uint2(h0, h1);
    *reinterpret_cast<uint2*>(sQ + 64 * LD + row * LD + c4) = make_uint2(l0, l1);
  }
  const uint32_t sQa = smem_u32(sQ);
  // q fragments of k-step ks as two fp16 terms [term][4], by ldmatrix
  auto q_frag = [&](int ks, uint32_t (&af)[2][4]) {
    const uint32_t ad = sQa + (uint32_t)((warp * 16 + (lane & 15)) * LD + ks * 16 + ((lane >> 4) << 3)) * 2u;
    ldsm_x4(ad, af[0][0], af[0][1], af[0][2], af[0][3]);
    ldsm_x4(ad + (uint32_t)(64 * LD * 2), af[1][0], af[1][1], af[1][2], af[1][3]);
  };
  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const uint32_t sKa = smem_u32(sK), sVa = smem_u32(sV);
  const SegGroup& G = a.grp[b];

  for (int si = 0; si < G.nseg; ++si) {
    const AttnSeg sg = G.seg[si];
    if (!sg.kb2) continue;   // own-key segments only (the host passes nothing else)
    const int nkb = (sg.n + KB - 1) / KB;
    // this CTA's key blocks: range kr of kv_split
    for (int kb = kr * nkb / a.kv_split; kb < (kr + 1) * nkb / a.kv_split; ++kb) {
      __syncthreads();
      for (int idx = threadIdx.x; idx < KB * (DH / 8); idx += 128) {
        const int row = idx / (DH / 8), c8 = idx % (DH / 8);
        const int key = kb * KB + row;
        const bool in = key < sg.n;
        const size_t o = (size_t)(in ? key : 0) * a.kv_ld + kvh * DH + c8 * 8;
        cp_async16(sK + row * LD + c8 * 8, sg.kb2 + o, in ? 16 : 0);
        cp_async16(sV + row * LD + c8 * 8, sg.vb2 + o, in ? 16 : 0);
        cp_async16(sK + KB * LD + row * LD + c8 * 8, sg.kb2 + sg.lo_off + o, in ? 16 : 0);
        cp_async16(sV + KB * LD + row * LD + c8 * 8, sg.vb2 + sg.lo_off + o, in ? 16 : 0);
      }
      cp_async_wait_all();
      __syncthreads();
      float s[KB / 8][4];
#pragma unroll
      for (int j = 0; j < KB / 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll 4
      for (int ks = 0; ks < DH / 16; ++ks) {
        uint32_t af[2][4];
        q_frag(ks, af);
#pragma unroll
        for (int jp = 0; jp < KB / 16; ++jp) {
          const int mi = lane >> 3, rr = lane & 7;
          const int key = jp * 16 + ((mi >> 1) << 3) + rr;
          const int col = ks * 16 + ((mi & 1) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(sKa + (uint32_t)(key * LD + col) * 2u, b0, b1, b2, b3);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            mma_16816_f16(s[2 * jp], af[t], b0, b1);
            mma_16816_f16(s[2 * jp + 1], af[t], b2, b3);
          }
          ldsm_x4(sKa + LO + (uint32_t)(key * LD + col) * 2u, b0, b1, b2, b3);
          mma_16816_f16(s[2 * jp], af[0], b0, b1);
          mma_16816_f16(s[2 * jp + 1], af[0], b2, b3);
        }
      }
      float mx0 = m0, mx1 = m1;
#pragma unroll
      for (int j = 0; j < KB / 8; ++j) {
        const int key = kb * KB + j * 8 + 2 * tq;
        s[j][0] = (key < sg.n) ? s[j][0] * a.scale_log2 : -INFINITY;
        s[j][1] = (key + 1 < sg.n) ? s[j][1] * a.scale_log2 : -INFINITY;
        s[j][2] = (key < sg.n) ? s[j][2] * a.scale_log2 : -INFINITY;
        s[j][3] = (key + 1 < sg.n) ? s[j][3] * a.scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][1]));
        mx1 = fmaxf(mx1, fmaxf(s[j][2], s[j][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float al0 = exp2f(m0 - mx0), al1 = exp2f(m1 - mx1);
      m0 = mx0;
      m1 = mx1;
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int j = 0; j < KB / 8; ++j) {
        s[j][0] = exp2f(s[j][0] - mx0);
        s[j][1] = exp2f(s[j][1] - mx0);
        s[j][2] = exp2f(s[j][2] - mx1);
        s[j][3] = exp2f(s[j][3] - mx1);
        sum0 += s[j][0] + s[j][1];
        sum1 += s[j][2] + s[j][3];
      }
      sum0 += __shfl_xor_sync(0xffffffffu, sum0, 1);
      sum0 += __shfl_xor_sync(0xffffffffu, sum0, 2);
      sum1 += __shfl_xor_sync(0xffffffffu, sum1, 1);
      sum1 += __shfl_xor_sync(0xffffffffu, sum1, 2);
      l0 = l0 * al0 + sum0;
      l1 = l1 * al1 + sum1;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        o[j][0] *= al0;
        o[j][1] *= al0;
        o[j][2] *= al1;
        o[j][3] *= al1;
      }
#pragma unroll
      for (int kk = 0; kk < KB / 16; ++kk) {
        uint32_t pf[2][4];
        split_pair_h2(s[2 * kk][0], s[2 * kk][1], pf[0][0], pf[1][0]);
        split_pair_h2(s[2 * kk][2], s[2 * kk][3], pf[0][1], pf[1][1]);
        split_pair_h2(s[2 * kk + 1][0], s[2 * kk + 1][1], pf[0][2], pf[1][2]);
        split_pair_h2(s[2 * kk + 1][2], s[2 * kk + 1][3], pf[0][3], pf[1][3]);
#pragma unroll
        for (int jp = 0; jp < NT / 2; ++jp) {
          const int mi = lane >> 3, rr = lane & 7;
          const int key = kk * 16 + ((mi & 1) << 3) + rr;
          const int col = jp * 16 + ((mi >> 1) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sVa + (uint32_t)(key * LD + col) * 2u, b0, b1, b2, b3);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            mma_16816_f16(o[2 * jp], pf[t], b0, b1);
            mma_16816_f16(o[2 * jp + 1], pf[t], b2, b3);
          }
          ldsm_x4_t(sVa + LO + (uint32_t)(key * LD + col) * 2u, b0, b1, b2, b3);
          mma_16816_f16(o[2 * jp], pf[0], b0, b1);
          mma_16816_f16(o[2 * jp + 1], pf[0], b2, b3);
        }
      }
    }
  }
  if (a.kv_split > 1) {   // partial of one key range: unnormalised output, row max and sum
    const size_t base = ((size_t)blockIdx.z * a.Hq + h) * a.T_rows;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int c = j * 8 + 2 * tq;
      if (v0) *reinterpret_cast<float2*>(a.part_o + (base + rl0) * DH + c) = make_float2(o[j][0], o[j][1]);
      if (v1) *reinterpret_cast<float2*>(a.part_o + (base + rl1) * DH + c) = make_float2(o[j][2], o[j][3]);
    }
    if (tq == 0) {
      if (v0) *reinterpret_cast<float2*>(a.part_ml + (base + rl0) * 2) = make_float2(m0, l0);
      if (v1) *reinterpret_cast<float2*>(a.part_ml + (base + rl1) * 2) = make_float2(m1, l1);
    }
    return;
  }
  const float i0 = (l0 > 0.f) ? 1.f / l0 : 0.f, i1 = (l1 > 0.f) ? 1.f / l1 : 0.f;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int c = h * DH + j * 8 + 2 * tq;
    if (v0) {
      uint32_t hh, ll;
      split_pair_h2(o[j][0] * i0, o[j][1] * i0, hh, ll);
      __half* p = a.out + row0 * kActTerms * a.ldh + c;
      *reinterpret_cast<uint32_t*>(p) = hh;
      *reinterpret_cast<uint32_t*>(p + a.ldh) = ll;
    }
    if (v1) {
      uint32_t hh, ll;
      split_pair_h2(o[j][2] * i1, o[j][3] * i1, hh, ll);
      __half* p = a.out + row1 * kActTerms * a.ldh + c;
      *reinterpret_cast<uint32_t*>(p) = hh;
      *reinterpret_cast<uint32_t*>(p + a.ldh) = ll;
    }
  }
}

// Merge of the prefix attention's key ranges: per (row, head) of group b,
// M = max_r m_r, o = sum_r 2^(m_r - M) O_r / sum_r 2^(m_r - M) l_r, written as
// the two fp16 planes of the output projection's operand.  Grid (T_rows, Hq,
// groups), one thread per head dimension.
static __global__ void attention_seg_combine_kernel(const __grid_constant__ SegAttnArgs a, int dh) {
  const int row = blockIdx.x, h = blockIdx.y, b = blockIdx.z, c = threadIdx.x;
  float M = -INFINITY;
  for (int r = 0; r < a.kv_split; ++r) {
    const size_t z = (size_t)b * a.kv_split + r;
    M = fmaxf(M, a.part_ml[((z * a.Hq + h) * a.T_rows + row) * 2]);
  }
  float num = 0.f, den = 0.f;
  for (int r = 0; r < a.kv_split; ++r) {
    const size_t z = (size_t)b * a.kv_split + r;
    const size_t i = (z * a.Hq + h) * a.T_rows + row;
    const float m = a.part_ml[i * 2], w = m == -INFINITY ? 0.f : exp2f(m - M);
    num += w * a.part_o[i * dh + c];
    den += w * a.part_ml[i * 2 + 1];
  }
  const float v = den > 0.f ? num / den : 0.f;
  const __half hv = __float2half_rn(v);
  __half* p = a.out + ((size_t)b * a.T_rows + row) * kActTerms * a.ldh + h * dh + c;
  p[0] = hv;
  p[a.ldh] = __float2half_rn(v - __half2float(hv));
}

// Launch the attention (and the combine when there are several key ranges).
// The kernels need more than 48 KB of dynamic shared memory for dh = 256:
// call set_attention_smem_limits() once per device first.
// segment attention: K and V blocks of kb keys in two planes each, rows padded to dh + 8
static inline int seg_attn_smem_bytes(int dh, int kb) { return (4 * kb + 2 * 64) * (dh + 8) * 2; }
// chunk attention: K and V blocks in two planes each, plus the partial scores
static inline int chunk_attn_smem_bytes(int dh) { return 4 * kAttnKB * (dh + 8) * 2 + 8 * 16 * (kAttnKB + 2) * 4; }

// Each attribute call's own status (the first failure), so that an error an
// earlier, unrelated launch left behind is neither reported here nor cleared.
static inline cudaError_t set_attention_smem_limits() {
  const cudaFuncAttribute A = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(attention_seg_kernel<256, 16>, A, seg_attn_smem_bytes(256, 16))) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(attention_seg_kernel<256, 32>, A, seg_attn_smem_bytes(256, 32))) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(attention_kernel<64>, A, chunk_attn_smem_bytes(64))) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(attention_kernel<128>, A, chunk_attn_smem_bytes(128))) != cudaSuccess) return e;
  return cudaFuncSetAttribute(attention_kernel<256>, A, chunk_attn_smem_bytes(256));
}

// Launches report their own status (cudaLaunchKernelEx), not the sticky last
// error of the thread.
static inline cudaError_t launch_chunk_attention(const AttnArgs& a, int dh, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hq, (a.T_q + 63) / 64, a.n_split);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = chunk_attn_smem_bytes(dh);
  cfg.stream = st;
  cudaError_t e;
  if (dh == 64) e = cudaLaunchKernelEx(&cfg, attention_kernel<64>, a);
  else if (dh == 128) e = cudaLaunchKernelEx(&cfg, attention_kernel<128>, a);
  else e = cudaLaunchKernelEx(&cfg, attention_kernel<256>, a);
  if (e != cudaSuccess || a.n_split == 1) return e;
  cudaLaunchConfig_t cc = {};
  cc.gridDim = dim3(a.T_q, a.Hq);
  cc.blockDim = dim3(dh);
  cc.stream = st;
  return cudaLaunchKernelEx(&cc, attention_combine_kernel, a, dh, (__nv_bfloat16*)nullptr);
}

}  // namespace lat
