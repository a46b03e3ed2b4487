// Persistent kernel for the pi0 action expert: all blocks of one denoise step
// in one launch.
//
// "Running VLAs at Real-time Speed" (reading note, sections 3 and 6) puts the
// action expert's time into launch gaps and into streaming every block's
// weights once per step; the TileRT page describes a persistent engine that
// keeps weight loads running while compute waits on its dependencies.  Here one
// CTA per SM lives for the whole step:
//
//  * warp 0 streams this CTA's share of every block's weights (128 x 64 bf16
//    tiles, TMA, 128-byte swizzle) through a ring of shared-memory slots.  The
//    weights do not depend on activations, so the stream runs ahead across
//    phase boundaries and is throttled only by the ring.
//  * warp 1 issues tcgen05 MMAs (M = 128 weight rows, N = 192 = three bf16
//    planes x 64 tokens, fp32 accumulator in TMEM, two buffers).
//  * warps 4..11 ("math") do everything that depends on activations: they
//    load the fp32 residual stream from global memory (several k-tiles in
//    flight, in registers) and split it into three bf16 planes in the MMA's
//    swizzled layout (warp 2 brings the other operands' planes by TMA), run
//    the split-K epilogues (vector reductions into fp32 sums at L2), the
//    attention and the combine of key-range partials.
//  * Per weight tile the shared memory moves ~80 KB (MMA reads of the 24 KB
//    operand and 16 KB weight tile, the operand's 24 KB of stores, the weight
//    tile's 16 KB TMA write); at ~128 B per clock that, not the tensor core
//    (96 cycles per M = 128, N = 192 MMA), paces a projection's k-tiles.
//
// Per block six phases, separated by a grid barrier (bounded spin):
//   1 QKV projection of x (sums of squares of x on the side, each head
//     group from its own K ranges); the CTAs of
//     each head group (its m-tiles, all K ranges) then wait for one another
//     on a group counter and finalize the group's q / own k, v: RMS factor,
//     RoPE, two-term bf16 planes, own k / v to the cache as bf16
//   2 attention: per (head, 32-key block), partial (max, sum, output)
//   3 combine of the key-block partials into the exact bf16 planes of o;
//     clears the QKV sums for the next block
//   4 x += o Wo (operand planes by TMA)
//   5 gate/up projection of x (gate and up rows of the same 64 FFN columns
//     in one 128-row tile; sums of squares on the side); the CTAs of each
//     tile wait for one another and write h = GELU(r g) * (r u) as exact
//     bf16 planes
//   6 x += h Wd (operand planes by TMA); clears the gate/up sums
// The RMSNorm scales are folded into the weights; the per-token factor
// r = rsqrt(mean(x^2) + eps) multiplies the projection sums (the projection is
// linear in its input), as in the pages' fold (section 4.1).
#pragma once
#include "attention.cuh"
#include "common.cuh"
#include "skinny_gemm.cuh"

namespace lat {

constexpr int kMkThreads = 384;                 // 12 warps
constexpr int kMkNW = 6;                        // weight ring slots
constexpr int kMkNB = 4;                        // activation-plane ring slots
constexpr int kMkPre = 4;                       // k-tiles of x the math warps hold in flight (registers)
constexpr int kMkWBytes = 128 * 64 * 2;         // one weight tile
constexpr int kMkBBytes = 192 * 64 * 2;         // one activation tile, three planes
constexpr int kMkRegion = 99 * 1024;            // the operand slots, also the attention's tiles
constexpr int kMkBars = 2 * kMkNW + 3 * kMkNB + 3;
static_assert(kMkNB * kMkBBytes <= kMkRegion, "operand slots must fit in the activation region");

__host__ __device__ constexpr int mk_smem_bytes() { return 1024 + kMkNW * kMkWBytes + kMkRegion + 8 * kMkBars + 16; }

// attention tiles: K hi, V hi, K lo, V lo ([32 keys][dh + 8] bf16 each), the
// exchanged scores [8][16][34] fp32; the q planes [2][64][dh + 8] bf16 overlay
// everything after the two hi planes (they are consumed before it is needed)
template <int DH>
__host__ __device__ constexpr int mk_attn_smem() {
  return 4 * kAttnKB * (DH + 8) * 2 + 8 * 16 * (kAttnKB + 2) * 4;
}
template <int DH>
__host__ __device__ constexpr int mk_attn_q_end() {
  return 2 * kAttnKB * (DH + 8) * 2 + 2 * 64 * (DH + 8) * 2;
}
static_assert(mk_attn_smem<256>() <= kMkRegion && mk_attn_q_end<256>() <= kMkRegion,
              "attention tiles must fit in the activation region");

// One projection: MT tiles of 128 output rows, KT tiles of 64 inputs, K split
// into `splits` ranges; CTA b < MT * splits takes m-tile b % MT and K range
// b / MT.  N = rows of one layer's matrix in the stacked weight tensor.
struct MkGemm {
  int MT, KT, splits, N;
};

struct MkArgs {
  MkGemm g[4];              // 0 QKV, 1 O, 2 gate/up, 3 down
  int l0, l1;               // layers [l0, l1) of this launch
  int D, F, Hq, Hkv, T_q, T_prefix, T_kv, nqkv;
  int prefix_lm;            // 1: the state token (query row 0) sees the prefix and itself only
  float eps, scale_log2;
  float* x;                 // fp32 [64][D] residual stream (rows >= T_q stay 0)
  float* qkv;               // fp32 [64][nqkv] QKV sums (vector reductions of every K range; 0 at entry,
                            // cleared again in the GeGLU phase for the next block)
  float* gu;                // fp32 [64][2F] gate/up sums in weight-row order (each 128-row tile = 64 gate
                            // rows, then the 64 up rows of the same FFN columns); 0 at entry, cleared
                            // again in the down phase for the next block
  __nv_bfloat16* o_planes;  // [3][64][Hq dh] attention output as exact bf16 planes (rows >= T_q stay 0)
  __nv_bfloat16* h_planes;  // [3][64][F] GeGLU output as exact bf16 planes (rows >= T_q stay 0)
  __nv_bfloat16* q_planes;  // [2][64][Hq dh] q after RoPE, two-term bf16 (hi, lo)
  __nv_bfloat16* kv_own;    // [k hi, k lo, v hi, v lo][64][Hkv dh] own keys / values, two-term bf16
  float* ss;                // fp32 [L][2][64] sums of squares of x (0 at entry)
  float* part_m;            // [n_kb][Hq][T_q]
  float* part_l;
  float* part_o;            // [n_kb][Hq][8 warps][dh / 16 n-tiles][32 lanes] x float4
  const float* cos_t;       // [T_q][dh / 2] RoPE tables of the query positions
  const float* sin_t;
  const float4* rope_frag;  // the same angles in the attention's q-fragment order:
                            // [8 warps][dh / 32 k-steps][4][32 lanes] x {cos i, cos i+1, sin i, sin i+1}
  __nv_bfloat16* kv;        // cache of layer l0: [2][T_kv][Hkv dh]
  long long kv_stride;      // elements from one layer's cache to the next
  unsigned* bar;            // grid barrier counter (0 at entry)
  unsigned* grp_cnt;        // dataflow counters, kCntWords words (0 at entry)
  DevErr* err;
  int skew_where;           // failure-detection hook: 0 off; 1 the first grid barrier, 2 the first QKV
                            // head-group wait, 3 the first gate/up tile wait of the launch waits for
  unsigned skew;            // this many arrivals more than will ever come (the wait runs out, the
                            // error word records a timeout and every later wait returns at once)
  unsigned long long* trace;   // null, or [layers][grid][64] phase timestamps (ns): 0..14 block
                               // start and the ends of each phase / barrier, 16..18 attention,
                               // 20 + 4 g .. 23 + 4 g projection g
};

struct MkRange {
  int m, k0, k1;
  bool active;
};

__device__ __forceinline__ MkRange mk_range(const MkGemm& g, int b) {
  MkRange r;
  r.active = b < g.MT * g.splits;
  r.m = b % g.MT;
  const int s = b / g.MT;
  r.k0 = s * g.KT / g.splits;
  r.k1 = (s + 1) * g.KT / g.splits;
  return r;
}

__device__ __forceinline__ bool mk_aborted(DevErr* e) { return *reinterpret_cast<volatile unsigned*>(&e->code) != 0; }

// Bounded mbarrier wait that also gives up as soon as any CTA has recorded an
// error: after a failure every wait returns at once and the kernel runs to its
// end with meaningless results (the host reports the error).
__device__ __forceinline__ bool mk_wait(uint64_t* bar, uint32_t parity, DevErr* err, unsigned where) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (int i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63) {
      if (mk_aborted(err)) return false;
      if (clock64() - t0 > kSpinBudget) {
        record_error(err, 1u, where);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mk_mark(unsigned long long* tr, int ev) {
  if (tr) tr[ev] = global_ns();
}

__device__ __forceinline__ float2 ldcg2(const float* p) { return __ldcg(reinterpret_cast<const float2*>(p)); }

// 4 x 4 transpose among the lanes k = lane % 4 of each lane quad: on entry
// lane k holds row k (a0..a3), on exit it holds column k.  Two exchange rounds
// (partner lane k ^ 1, then k ^ 2), two shuffles each.
__device__ __forceinline__ void quad_transpose(float& a0, float& a1, float& a2, float& a3, int k) {
  const bool c = k & 1, d = (k >> 1) & 1;
  const float x0 = __shfl_xor_sync(0xffffffffu, c ? a0 : a1, 1);
  const float x1 = __shfl_xor_sync(0xffffffffu, c ? a2 : a3, 1);
  if (c) { a0 = x0; a2 = x1; } else { a1 = x0; a3 = x1; }
  const float y0 = __shfl_xor_sync(0xffffffffu, d ? a0 : a2, 2);
  const float y1 = __shfl_xor_sync(0xffffffffu, d ? a1 : a3, 2);
  if (d) { a0 = y0; a1 = y1; } else { a2 = y0; a3 = y1; }
}

// n4 float4 of p = 0, spread over the grid's math threads
__device__ __forceinline__ void mk_zero_f4(float* p, int n4, int mt) {
  float4* z = reinterpret_cast<float4*>(p);
  for (int i = blockIdx.x * 256 + mt; i < n4; i += gridDim.x * 256) __stcg(z + i, make_float4(0.f, 0.f, 0.f, 0.f));
}



// 8 fp32 values (registers) -> 8 bf16 hi and 8 bf16 lo (two-term split)
__device__ __forceinline__ void split8_regs(const float (&v)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) split_pair2(v[2 * e], v[2 * e + 1], h[e], l[e]);
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Grid barrier among the math warps of all CTAs (barrier n waits for n * grid
// arrivals).  Generic-proxy writes before it become visible to TMA reads after it.
__device__ __forceinline__ void mk_grid_sync(unsigned* ctr, unsigned target, DevErr* err, int mt) {
  fence_proxy_async_global();
  named_sync(1, 256);
  if (mt == 0) {
    __threadfence();
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(ctr), "r"(1u) : "memory");
    const long long t0 = clock64();
    for (int i = 0;; ++i) {
      if (ld_acquire_u32(ctr) >= target) break;
      if ((i & 15) == 15) {
        if (mk_aborted(err)) break;
        if (clock64() - t0 > kSpinBudget) {
          record_error(err, 2u, 900);
          break;
        }
      }
    }
    fence_proxy_async_global();
  }
  named_sync(1, 256);
}

// Shared state of the math warps.
struct MkMath {
  uint8_t* sB;
  uint64_t* bfull;
  uint64_t* bempty;
  uint64_t* accfull;
  uint64_t* go;
  uint32_t tmem;
  uint32_t bt, gc;
  int mt;
};

// Math side of one projection.  Projections of the residual stream x (QKV,
// gate/up): the math warps load their rows of x straight from global memory,
// kMkPre k-tiles in flight in registers, and write the exact bf16 planes into
// the operand slots; for the others (act == nullptr) the loader brings the
// planes by TMA.  Then the split-K epilogue: every K range adds its partial
// sums into `out` (vector reductions at L2).  `stats`, when given, receives
// this K range's per-token sums of squares of x (atomic adds).
// 16 bytes from global memory through L2 (not L1: other SMs write x), issued
// where it stands so that several k-tiles are in flight at once
__device__ __forceinline__ float4 mk_ldcg4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void mk_load_tile(const float* act, int ld, int kt, const int (&rows)[2], int p,
                                             float4 (&v)[4]) {
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) v[2 * i + hh] = mk_ldcg4(act + (size_t)rows[i] * ld + kt * 64 + hh * 32 + 4 * p);
}

__device__ __forceinline__ void mk_gemm_math(MkMath& s, const MkGemm& g, const float* act, int act_ld, float* stats,
                                             float* out, int ld, int T_q, DevErr* err, unsigned long long* tr) {
  const MkRange r = mk_range(g, blockIdx.x);
  if (!r.active) return;
  const int nk = r.k1 - r.k0;
  const int mw = s.mt >> 5, lane = s.mt & 31;
  if (!act) {   // the loader brings this projection's operand planes by TMA
    s.bt += nk;
    if (tr) tr[0] = tr[1] = global_ns();
  }
  // conversion layout: per k-tile each thread takes two rows, 8 columns of each
  // (cols 4p..4p+3 and 32+4p..+3); rows ordered so a warp's 8-byte stores of
  // one pass touch both halves of the 128-byte swizzled rows (conflict-free)
  const int rq = lane >> 3, p = lane & 7;
  int rows[2];
  float sq[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    rows[i] = mw * 8 + i + (rq & 1) * 4 + (rq >> 1) * 2;
    sq[i] = 0.f;
  }
  if (act) {
    float4 xv[kMkPre][4];
#pragma unroll
    for (int u = 0; u < kMkPre; ++u)
      if (u < nk) mk_load_tile(act, act_ld, r.k0 + u, rows, p, xv[u]);
    mk_mark(tr, 0);
    for (int j0 = 0; j0 < nk; j0 += kMkPre) {
#pragma unroll
      for (int u = 0; u < kMkPre; ++u) {
        const int j = j0 + u;
        if (j < nk) {
          const uint32_t b = s.bt % kMkNB;
          mk_wait(&s.bempty[b], ((s.bt / kMkNB) & 1) ^ 1, err, 31);
          uint8_t* dst = s.sB + b * kMkBBytes;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int t = rows[i];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int col = hh * 32 + 4 * p;
              const float4 v = xv[u][2 * i + hh];
              if (stats) sq[i] += (v.x * v.x + v.y * v.y) + (v.z * v.z + v.w * v.w);
              uint32_t h0, m0, l0, h1, m1, l1;
              split_pair_exact(v.x, v.y, h0, m0, l0);
              split_pair_exact(v.z, v.w, h1, m1, l1);
              const uint32_t off = (uint32_t)(t * 128 + ((((col >> 3) ^ t) & 7) << 4) + ((p & 1) << 3));
              *reinterpret_cast<uint2*>(dst + off) = make_uint2(h0, h1);
              *reinterpret_cast<uint2*>(dst + 8192 + off) = make_uint2(m0, m1);
              *reinterpret_cast<uint2*>(dst + 16384 + off) = make_uint2(l0, l1);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.bfull[b]);   // this warp's rows of the operand are written
          ++s.bt;
          if (j + kMkPre < nk) mk_load_tile(act, act_ld, r.k0 + j + kMkPre, rows, p, xv[u]);
        }
      }
    }
  }
  if (stats) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float v = sq[i];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      if (p == 0) atomicAdd(stats + rows[i], v);
    }
  }
  // epilogue: warp (4 + mw) reads TMEM lanes 32 (mw % 4) .. +31 = output rows,
  // tokens 32 (mw / 4) .. +31 of each plane; the planes are summed hi + mid + lo
  if (act) mk_mark(tr, 1);
  mk_wait(s.accfull, s.gc & 1, err, 32);
  mk_mark(tr, 2);
  tc_fence_after();
  const uint32_t acc = s.tmem + (s.gc & 1) * 256;
  ++s.gc;
  const int q = mw & 3, ch = mw >> 2;
  const int f = r.m * 128 + q * 32 + lane;
  const uint32_t tb = acc + ((uint32_t)(q * 32) << 16) + (uint32_t)(ch * 32);
  float v[32], w[32], z[32];
  tmem_ld32x3(tb, tb + 64, tb + 128, v, w, z);
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = (v[j] + w[j]) + z[j];
  tc_fence_before();
  // each lane quad transposes 4 tokens x its 4 outputs, so a lane adds 4
  // consecutive outputs of one token: one vector reduction
  const int k4 = lane & 3;
  const int fb = f - k4;
#pragma unroll
  for (int j0 = 0; j0 < 32; j0 += 4) {
    float a0 = v[j0], a1 = v[j0 + 1], a2 = v[j0 + 2], a3 = v[j0 + 3];
    quad_transpose(a0, a1, a2, a3, k4);
    const int t = ch * 32 + j0 + k4;
    if (t < T_q) red_add_v4(out + (size_t)t * ld + fb, a0, a1, a2, a3);
  }
  mk_mark(tr, 3);
}

// q, own k and own v of one head group, from the finished QKV sums: every CTA
// of the projection adds its K range into a.qkv (vector reductions); the CTA
// that completes a group (all K ranges of its m-tiles) runs this for the
// group's heads.  r = rsqrt(mean(x^2) + eps), RoPE (rotate-half pairs
// (i, i + dh/2)) on q and k heads, two-term bf16 splits into q_planes /
// kv_own, and the bf16 cache copy (nearest) of own k / v at slots T_prefix + t.
template <int DH>
__device__ __forceinline__ void mk_qkv_finalize_group(const MkArgs& a, int h0, int nhd, int part, int parts,
                                                      const float* ss1, __nv_bfloat16* kc, __nv_bfloat16* vc,
                                                      float invD, int mt) {
  constexpr int HD = DH / 2;
  const int nh = a.Hq + a.Hkv, kvd = a.Hkv * DH, qd = a.Hq * DH;
  const size_t qpl = (size_t)64 * qd, kpl = (size_t)64 * kvd;
  for (int hd = h0; hd < h0 + nhd; ++hd) {
    if (hd < nh) {   // q or k head: 4 RoPE pairs per item
      const int n = a.T_q * (HD / 4);
      for (int it = part * n / parts + mt; it < (part + 1) * n / parts; it += 256) {
        const int t = it / (HD / 4), i = (it % (HD / 4)) * 4;
        const float* p0 = a.qkv + (size_t)t * a.nqkv + hd * DH + i;
        const float4 x0 = __ldcg(reinterpret_cast<const float4*>(p0));
        const float4 x1 = __ldcg(reinterpret_cast<const float4*>(p0 + HD));
        const float rv = rsqrtf(__ldcg(ss1 + t) * invD + a.eps);
        const float4 c = __ldg(reinterpret_cast<const float4*>(a.cos_t + (size_t)t * HD + i));
        const float4 sn = __ldg(reinterpret_cast<const float4*>(a.sin_t + (size_t)t * HD + i));
        const float a0[4] = {rv * x0.x, rv * x0.y, rv * x0.z, rv * x0.w};
        const float a1[4] = {rv * x1.x, rv * x1.y, rv * x1.z, rv * x1.w};
        const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {sn.x, sn.y, sn.z, sn.w};
        float y0[4], y1[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          y0[e] = a0[e] * cc[e] - a1[e] * ss[e];
          y1[e] = a1[e] * cc[e] + a0[e] * ss[e];
        }
        uint32_t h0w[2], l0w[2], h1w[2], l1w[2];
        split_pair2(y0[0], y0[1], h0w[0], l0w[0]);
        split_pair2(y0[2], y0[3], h0w[1], l0w[1]);
        split_pair2(y1[0], y1[1], h1w[0], l1w[0]);
        split_pair2(y1[2], y1[3], h1w[1], l1w[1]);
        if (hd < a.Hq) {
          uint2* q = reinterpret_cast<uint2*>(a.q_planes + (size_t)t * qd + hd * DH + i);
          q[0] = make_uint2(h0w[0], h0w[1]);
          q[HD / 4] = make_uint2(h1w[0], h1w[1]);
          q[qpl / 4] = make_uint2(l0w[0], l0w[1]);
          q[qpl / 4 + HD / 4] = make_uint2(l1w[0], l1w[1]);
        } else {
          const int kh = hd - a.Hq;
          uint2* k = reinterpret_cast<uint2*>(a.kv_own + (size_t)t * kvd + kh * DH + i);
          k[0] = make_uint2(h0w[0], h0w[1]);
          k[HD / 4] = make_uint2(h1w[0], h1w[1]);
          k[kpl / 4] = make_uint2(l0w[0], l0w[1]);
          k[kpl / 4 + HD / 4] = make_uint2(l1w[0], l1w[1]);
          float tx, ty;
          uint2* ck = reinterpret_cast<uint2*>(kc + (size_t)(a.T_prefix + t) * kvd + kh * DH + i);
          ck[0] = make_uint2(rn_pair(y0[0], y0[1], tx, ty), rn_pair(y0[2], y0[3], tx, ty));
          ck[HD / 4] = make_uint2(rn_pair(y1[0], y1[1], tx, ty), rn_pair(y1[2], y1[3], tx, ty));
        }
      }
    } else {   // v head: 4 values per item
      const int n = a.T_q * (DH / 4), j0 = (hd - nh) * DH;
      for (int it = part * n / parts + mt; it < (part + 1) * n / parts; it += 256) {
        const int t = it / (DH / 4), j = j0 + (it % (DH / 4)) * 4;
        float4 x = __ldcg(reinterpret_cast<const float4*>(a.qkv + (size_t)t * a.nqkv + nh * DH + j));
        const float rv = rsqrtf(__ldcg(ss1 + t) * invD + a.eps);
        x.x *= rv; x.y *= rv; x.z *= rv; x.w *= rv;
        uint32_t hh[2], ll[2];
        split_pair2(x.x, x.y, hh[0], ll[0]);
        split_pair2(x.z, x.w, hh[1], ll[1]);
        uint2* v = reinterpret_cast<uint2*>(a.kv_own + 2 * kpl + (size_t)t * kvd + j);
        v[0] = make_uint2(hh[0], hh[1]);
        v[kpl / 4] = make_uint2(ll[0], ll[1]);
        float tx, ty;
        *reinterpret_cast<uint2*>(vc + (size_t)(a.T_prefix + t) * kvd + j) =
            make_uint2(rn_pair(x.x, x.y, tx, ty), rn_pair(x.z, x.w, tx, ty));
      }
    }
  }
}

// Counters after the grid barrier word (MkArgs::grp_cnt), 0 at launch entry;
// each grows by one group's arrivals per block.
constexpr int kCntQkvArr = 0;      // [32] QKV head groups: CTAs past their epilogue
constexpr int kCntGuArr = 32;      // [192] gate/up tiles: CTAs past their epilogue
constexpr int kCntWords = 224;
// Per-token sums of squares of the projection input (MkArgs::ss), one row of
// 64 per QKV head group, then one per gate/up tile: each group's own K ranges
// add into its row, so a group needs no other group's statistics.
constexpr int kSsQkv = 0;
constexpr int kSsGu = 32;
constexpr int kSsRows = 224;

// Count this CTA into group counter `cnt`, then wait until the group has all
// `target` arrivals.  Bounded: gives up (error recorded) after the spin budget
// or when another CTA has failed.  The counters grow by one group's arrivals
// per block and start at 0 with each launch.
__device__ __forceinline__ void mk_group_wait(unsigned* cnt, unsigned target, DevErr* err, unsigned where, int mt) {
  __threadfence();   // this thread's reductions are performed before the arrival
  named_sync(2, 256);
  if (mt == 0) {
    atomicAdd(cnt, 1u);
    const long long t0 = clock64();
    for (int i = 0; ld_acquire_u32(cnt) < target; ++i)
      if ((i & 15) == 15 && (mk_aborted(err) || clock64() - t0 > kSpinBudget)) {
        if (!mk_aborted(err)) record_error(err, 2u, where);
        break;
      }
    __threadfence();
  }
  named_sync(2, 256);
}

// After the QKV epilogue: every CTA of a head group (the m-tiles of whole
// heads, all K ranges) waits for the group, then finalizes its share of the
// group's heads.  `lr` = block index within the launch.
template <int DH>
struct MkQkvGroups {
  static constexpr int MPG = DH >= 128 ? DH / 128 : 1;   // m-tiles per group
  static constexpr int HPG = DH >= 128 ? 1 : 128 / DH;   // heads per group
};

template <int DH>
__device__ __forceinline__ void mk_qkv_arrive(const MkArgs& a, int lr, __nv_bfloat16* kc, __nv_bfloat16* vc,
                                              float invD, int mt) {
  const MkGemm& g = a.g[0];
  const MkRange r = mk_range(g, blockIdx.x);
  if (!r.active) return;
  constexpr int MPG = MkQkvGroups<DH>::MPG, HPG = MkQkvGroups<DH>::HPG;
  const int grp = r.m / MPG;
  const int per = MPG * g.splits;
  const int part = (r.m % MPG) * g.splits + (int)blockIdx.x / g.MT;
  const unsigned extra = (lr == 0 && a.skew_where == 2) ? a.skew : 0u;
  mk_group_wait(a.grp_cnt + kCntQkvArr + grp, (unsigned)((lr + 1) * per) + extra, a.err, 901, mt);
  mk_qkv_finalize_group<DH>(a, grp * HPG, HPG, part, per, a.ss + (kSsQkv + grp) * 64, kc, vc, invD, mt);
}

// Phase 3: attention of the chunk over [cache | own], one (head, 32-key block)
// per unit, partial (max, sum, unnormalised output) per unit.  Same arithmetic
// as attention_kernel (two-term q and p, own keys as computed in two planes);
// warp half h owns head dims [h dh/4, +dh/4) and [dh/2 + h dh/4, +dh/4).  q and
// the own keys arrive as planes from phase 2, cache keys from the cache.
template <int DH>
__device__ __forceinline__ void mk_attention(const MkArgs& a, __nv_bfloat16* kc, __nv_bfloat16* vc, uint8_t* sR,
                                             int mt, unsigned long long* tr) {
  constexpr int KB = kAttnKB;
  constexpr int LD = DH + 8;
  constexpr int HD = DH / 2;
  constexpr int KS = HD / 16;
  constexpr int NT = HD / 8;
  constexpr int SLD = KB + 2;
  constexpr int Q4 = DH / 4;
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(sR);       // hi plane; lo plane at + 2 KB LD
  __nv_bfloat16* sV = sK + KB * LD;
  float* sS = reinterpret_cast<float*>(sK + 4 * KB * LD);
  __nv_bfloat16* sQ = sK + 2 * KB * LD;                            // q hi plane; lo plane at + 64 LD
  const int warp = mt >> 5, lane = mt & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int rt = warp & 3, half = warp >> 2;
  const int nkb = attn_key_blocks(a.T_kv);
  const int units = a.Hq * nkb;
  const int kvd = a.Hkv * DH, group = a.Hq / a.Hkv, qd = a.Hq * DH;
  const int own0 = a.T_prefix;
  const int r0 = rt * 16 + g, r1 = r0 + 8;
  const bool v0 = r0 < a.T_q, v1 = r1 < a.T_q;
  const uint32_t sKa = smem_u32(sK), sVa = smem_u32(sV), sQa = smem_u32(sQ);
  const uint32_t LO = (uint32_t)(2 * KB * LD * 2);
  const size_t kpl = (size_t)64 * kvd, qpl = (size_t)64 * qd;
  float* myS = sS + warp * 16 * SLD;
  const float* peerS = sS + (warp ^ 4) * 16 * SLD;
  const int mi = lane >> 3, rr = lane & 7;

  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int h = u / nkb, kb = u % nkb, kvh = h / group;
    const bool has_lo = (kb + 1) * KB > own0 && own0 < a.T_kv;
    named_sync(3, 256);   // the previous unit is done with the tiles
    // ---- async copies: hi planes of the key block (cache keys, then own
    //      keys), q planes ----
    auto kv_copies = [&](bool own_pass) {
      for (int idx = mt; idx < KB * (DH / 8); idx += 256) {
        const int row = idx / (DH / 8), c8 = idx % (DH / 8);
        const int key = kb * KB + row;
        const bool own = key >= own0 && key < a.T_kv;
        const bool in = key < a.T_kv;
        if (own != own_pass) continue;
        const __nv_bfloat16* ks;
        const __nv_bfloat16* vs;
        if (own) {
          const size_t off = (size_t)(key - own0) * kvd + kvh * DH + c8 * 8;
          ks = a.kv_own + off;
          vs = a.kv_own + 2 * kpl + off;
        } else {
          const size_t off = (size_t)(in ? key : 0) * kvd + kvh * DH + c8 * 8;
          ks = kc + off;
          vs = vc + off;
        }
        cp_async16(sK + row * LD + c8 * 8, ks, in ? 16 : 0);
        cp_async16(sV + row * LD + c8 * 8, vs, in ? 16 : 0);
      }
    };
    kv_copies(false);
    if (has_lo) kv_copies(true);
    for (int idx = mt; idx < 2 * 64 * (DH / 8); idx += 256) {
      const int pr = idx / (DH / 8), c8 = idx % (DH / 8);   // plane-row: plane pr / 64, row pr % 64
      const int row = pr & 63;
      const bool in = row < a.T_q;
      const __nv_bfloat16* src = a.q_planes + (pr >> 6) * qpl + (size_t)(in ? row : 0) * qd + h * DH + c8 * 8;
      cp_async16(sQ + pr * LD + c8 * 8, src, in ? 16 : 0);
    }
    cp_async_wait_all();
    named_sync(3, 256);
    // ---- q fragments by ldmatrix: rows rt*16.., this warp's dims ----
    uint32_t qh[KS][4], ql[KS][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int db = (ks < KS / 2) ? half * Q4 + ks * 16 : HD + half * Q4 + (ks - KS / 2) * 16;
      const uint32_t ad = sQa + (uint32_t)((rt * 16 + (lane & 15)) * LD + db + ((lane >> 4) << 3)) * 2u;
      ldsm_x4(ad, qh[ks][0], qh[ks][1], qh[ks][2], qh[ks][3]);
      ldsm_x4(ad + (uint32_t)(64 * LD * 2), ql[ks][0], ql[ks][1], ql[ks][2], ql[ks][3]);
    }
    named_sync(3, 256);   // the q tiles are consumed: their bytes hold the lo planes and scores next
    mk_mark(tr, 17);
    // ---- lo planes: own keys from phase 2, zero for cache keys ----
    if (has_lo) {
      for (int idx = mt; idx < KB * (DH / 8); idx += 256) {
        const int row = idx / (DH / 8), c8 = idx % (DH / 8);
        const int key = kb * KB + row;
        if (key >= own0 && key < a.T_kv) {
          const size_t off = (size_t)(key - own0) * kvd + kvh * DH + c8 * 8;
          cp_async16(sK + 2 * KB * LD + row * LD + c8 * 8, a.kv_own + kpl + off, 16);
          cp_async16(sV + 2 * KB * LD + row * LD + c8 * 8, a.kv_own + 3 * kpl + off, 16);
        } else {
          *reinterpret_cast<uint4*>(sK + 2 * KB * LD + row * LD + c8 * 8) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(sV + 2 * KB * LD + row * LD + c8 * 8) = make_uint4(0, 0, 0, 0);
        }
      }
      cp_async_wait_all();
    }
    named_sync(3, 256);
    mk_mark(tr, 18);

    // ---- partial scores over this warp's dims: 16 rows x 32 keys ----
    float sa[4][4], sb[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) sa[j][e] = sb[j][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int db = (ks < KS / 2) ? half * Q4 + ks * 16 : HD + half * Q4 + (ks - KS / 2) * 16;
      uint32_t b[4][2];
#pragma unroll
      for (int jp = 0; jp < 2; ++jp) {
        const int key = jp * 16 + ((mi >> 1) << 3) + rr;
        const int col = db + ((mi & 1) << 3);
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
          const int col = db + ((mi & 1) << 3);
          ldsm_x4(sKa + LO + (uint32_t)(key * LD + col) * 2u, b[2 * jp][0], b[2 * jp][1], b[2 * jp + 1][0],
                  b[2 * jp + 1][1]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_16816(sb[j], qh[ks], b[j][0], b[j][1]);
      }
    }
    // ---- exchange partial scores with the other half ----
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = j * 8 + 2 * tq;
      *reinterpret_cast<float2*>(myS + g * SLD + c) = make_float2(sa[j][0] + sb[j][0], sa[j][1] + sb[j][1]);
      *reinterpret_cast<float2*>(myS + (g + 8) * SLD + c) = make_float2(sa[j][2] + sb[j][2], sa[j][3] + sb[j][3]);
    }
    named_sync(3, 256);
    float s[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = j * 8 + 2 * tq;
      const float2 p0 = *reinterpret_cast<const float2*>(peerS + g * SLD + c);
      const float2 p1 = *reinterpret_cast<const float2*>(peerS + (g + 8) * SLD + c);
      s[j][0] = (sa[j][0] + sb[j][0]) + p0.x;
      s[j][1] = (sa[j][1] + sb[j][1]) + p0.y;
      s[j][2] = (sa[j][2] + sb[j][2]) + p1.x;
      s[j][3] = (sa[j][3] + sb[j][3]) + p1.y;
    }
    // ---- softmax of this key block (base 2) ----
    // keys a row may see: all T_kv, or with the block mask the state token
    // (row 0) only the prefix and itself (keys < T_prefix + 1)
    const int lim0 = (a.prefix_lm && r0 == 0) ? a.T_prefix + 1 : a.T_kv;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int key = kb * KB + j * 8 + 2 * tq;
      s[j][0] = (key < lim0) ? s[j][0] * a.scale_log2 : -INFINITY;
      s[j][1] = (key + 1 < lim0) ? s[j][1] * a.scale_log2 : -INFINITY;
      s[j][2] = (key < a.T_kv) ? s[j][2] * a.scale_log2 : -INFINITY;
      s[j][3] = (key + 1 < a.T_kv) ? s[j][3] * a.scale_log2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][1]));
      mx1 = fmaxf(mx1, fmaxf(s[j][2], s[j][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    // a row with every key of the block masked keeps max -inf (weight 0 in the
    // combine); its exponentials are taken against 0 so that they are 0, not NaN
    const float e0 = mx0 == -INFINITY ? 0.f : mx0, e1 = mx1 == -INFINITY ? 0.f : mx1;
    float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      s[j][0] = exp2f(s[j][0] - e0);
      s[j][1] = exp2f(s[j][1] - e0);
      s[j][2] = exp2f(s[j][2] - e1);
      s[j][3] = exp2f(s[j][3] - e1);
      sum0 += s[j][0] + s[j][1];
      sum1 += s[j][2] + s[j][3];
    }
    sum0 += __shfl_xor_sync(0xffffffffu, sum0, 1);
    sum0 += __shfl_xor_sync(0xffffffffu, sum0, 2);
    sum1 += __shfl_xor_sync(0xffffffffu, sum1, 1);
    sum1 += __shfl_xor_sync(0xffffffffu, sum1, 2);

    // ---- O = P V over this warp's output dims ----
    float o[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
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
        const int j8 = 2 * jp;
        const int col = ((j8 < NT / 2) ? half * Q4 + j8 * 8 : HD + half * Q4 + (j8 - NT / 2) * 8) + ((mi >> 1) << 3);
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
          const int j8 = 2 * jp;
          const int col =
              ((j8 < NT / 2) ? half * Q4 + j8 * 8 : HD + half * Q4 + (j8 - NT / 2) * 8) + ((mi >> 1) << 3);
          ldsm_x4_t(sVa + LO + (uint32_t)(key * LD + col) * 2u, b[2 * jp][0], b[2 * jp][1], b[2 * jp + 1][0],
                    b[2 * jp + 1][1]);
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_16816(o[j], ph, b[j][0], b[j][1]);
      }
    }

    mk_mark(tr, 19);
    // ---- partials of this key block: (max, sum) per row; the unnormalised
    //      output in fragment order, [warp][n-tile][lane] x float4 (rows r0 | r1) ----
    const size_t base = ((size_t)kb * a.Hq + h) * a.T_q;
    if (tq == 0 && half == 0) {
      if (v0) { a.part_m[base + r0] = mx0; a.part_l[base + r0] = sum0; }
      if (v1) { a.part_m[base + r1] = mx1; a.part_l[base + r1] = sum1; }
    }
    float4* po = reinterpret_cast<float4*>(a.part_o) + (((size_t)kb * a.Hq + h) * 8 + warp) * NT * 32 + lane;
#pragma unroll
    for (int j = 0; j < NT; ++j) __stcg(po + j * 32, make_float4(o[j][0], o[j][1], o[j][2], o[j][3]));
  }
  fence_proxy_async_smem();   // the tiles' bytes are reused by TMA in the next phase
}

// Phase 4: o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s per (token,
// head), written as the exact bf16 planes of the output projection's operand.  Work comes in
// chunks of 256 fragments (the attention's output order); for the <= 2 (head,
// warp) groups of a chunk the per-row weights 2^(m_s - M) / L go to shared
// memory first, then each thread merges one fragment over all key blocks.
template <int DH>
__device__ __forceinline__ void mk_combine(const MkArgs& a, int mt, float* sw, unsigned long long* tr) {
  constexpr int HD = DH / 2, NT = HD / 8, Q4 = DH / 4;
  constexpr int PER_HW = NT * 32;   // fragments of one (head, warp)
  const int nkb = attn_key_blocks(a.T_kv);
  const int qd = a.Hq * DH;
  const int items = a.Hq * 8 * PER_HW;
  const size_t ml_stride = (size_t)a.Hq * a.T_q;
  const size_t o_stride = (size_t)a.Hq * 8 * PER_HW;
  const size_t pl = (size_t)64 * qd;   // one plane
  for (int c0 = blockIdx.x * 256; c0 < items; c0 += gridDim.x * 256) {
    const int g0 = c0 / PER_HW;
    // this thread's fragment of every key block, loaded before the weights so
    // that both passes wait on one L2 round trip (up to kCombPre key blocks)
    constexpr int kCombPre = 24;
    const int it = c0 + mt;
    const bool has_it = it < items;
    const float4* po = reinterpret_cast<const float4*>(a.part_o) + (has_it ? it : 0);
    float4 ov[kCombPre];
#pragma unroll
    for (int e = 0; e < kCombPre; ++e)
      ov[e] = (has_it && e < nkb) ? __ldcg(po + (size_t)e * o_stride) : make_float4(0.f, 0.f, 0.f, 0.f);
    // pass 1: weights of the rows of groups g0, g0 + 1 (16 rows each): thread
    // (row mt / 8, lane-group part mt % 8) takes key blocks part, part + 8, ...
    {
      const int row = mt >> 3, part = mt & 7;
      const int gg = g0 + (row >> 4), rr = row & 15;
      const int h = gg / 8, t = (gg % 8 & 3) * 16 + rr;
      const bool valid = h < a.Hq && t < a.T_q;
      const size_t i0 = (size_t)(valid ? h : 0) * a.T_q + (valid ? t : 0);
      constexpr int MAXP = 4;   // key blocks per thread held in registers (n_kb <= 32)
      float mv[MAXP], lv[MAXP];
#pragma unroll
      for (int e = 0; e < MAXP; ++e) {
        const int kb = part + 8 * e;
        const bool in = valid && kb < nkb;
        mv[e] = in ? __ldcg(a.part_m + (size_t)kb * ml_stride + i0) : -INFINITY;
        lv[e] = in ? __ldcg(a.part_l + (size_t)kb * ml_stride + i0) : 0.f;
      }
      float M = -INFINITY;
#pragma unroll
      for (int e = 0; e < MAXP; ++e) M = fmaxf(M, mv[e]);
      for (int kb = part + 8 * MAXP; kb < nkb; kb += 8)   // longer caches
        if (valid) M = fmaxf(M, __ldcg(a.part_m + (size_t)kb * ml_stride + i0));
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 1));
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 4));
      float wv[MAXP], L = 0.f;
#pragma unroll
      for (int e = 0; e < MAXP; ++e) {
        wv[e] = (mv[e] == -INFINITY) ? 0.f : exp2f(mv[e] - M);
        L += wv[e] * lv[e];
      }
      for (int kb = part + 8 * MAXP; kb < nkb; kb += 8)
        if (valid) {
          const float m = __ldcg(a.part_m + (size_t)kb * ml_stride + i0);
          L += exp2f(m - M) * __ldcg(a.part_l + (size_t)kb * ml_stride + i0);
        }
      L += __shfl_xor_sync(0xffffffffu, L, 1);
      L += __shfl_xor_sync(0xffffffffu, L, 2);
      L += __shfl_xor_sync(0xffffffffu, L, 4);
      const float il = valid ? 1.f / L : 0.f;
#pragma unroll
      for (int e = 0; e < MAXP; ++e)
        if (part + 8 * e < nkb) sw[row * nkb + part + 8 * e] = wv[e] * il;
      for (int kb = part + 8 * MAXP; kb < nkb; kb += 8)
        sw[row * nkb + kb] = valid ? exp2f(__ldcg(a.part_m + (size_t)kb * ml_stride + i0) - M) * il : 0.f;
    }
    named_sync(3, 256);
    mk_mark(tr, 36);
    // pass 2: one fragment per thread
    if (has_it) {
      const int lane = it & 31, j = (it >> 5) % NT, gg = it / PER_HW;
      const int h = gg / 8, w = gg % 8;
      const int rt = w & 3, half = w >> 2, g = lane >> 2, tq = lane & 3;
      const int r0 = rt * 16 + g, r1 = r0 + 8;
      const int c = ((j < NT / 2) ? half * Q4 + j * 8 : HD + half * Q4 + (j - NT / 2) * 8) + 2 * tq;
      const float* w0 = sw + ((gg - g0) * 16 + g) * nkb;
      const float* w1 = w0 + 8 * nkb;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int e = 0; e < kCombPre; ++e) {
        if (e < nkb) {
          const float a0 = w0[e], a1 = w1[e];
          acc.x += a0 * ov[e].x;
          acc.y += a0 * ov[e].y;
          acc.z += a1 * ov[e].z;
          acc.w += a1 * ov[e].w;
        }
      }
      for (int e = kCombPre; e < nkb; ++e) {   // longer caches
        const float4 z = __ldcg(po + (size_t)e * o_stride);
        const float a0 = w0[e], a1 = w1[e];
        acc.x += a0 * z.x;
        acc.y += a0 * z.y;
        acc.z += a1 * z.z;
        acc.w += a1 * z.w;
      }
      uint32_t hi, mid, lo;
      const size_t col = (size_t)h * DH + c;
      if (r0 < a.T_q) {
        split_pair_exact(acc.x, acc.y, hi, mid, lo);
        uint32_t* d = reinterpret_cast<uint32_t*>(a.o_planes + (size_t)r0 * qd + col);
        d[0] = hi;
        d[pl / 2] = mid;
        d[pl] = lo;
      }
      if (r1 < a.T_q) {
        split_pair_exact(acc.z, acc.w, hi, mid, lo);
        uint32_t* d = reinterpret_cast<uint32_t*>(a.o_planes + (size_t)r1 * qd + col);
        d[0] = hi;
        d[pl / 2] = mid;
        d[pl] = lo;
      }
    }
    named_sync(3, 256);   // sw is reused by the next chunk
    mk_mark(tr, 37);
  }
  fence_proxy_async_smem();   // sw's bytes are reused by TMA in the next phase
}

// h = GELU(r g) * (r u) for the 64 FFN columns of gate/up tile m and every
// token, as the exact bf16 planes of the down projection's operand; g and u
// are the finished gate/up sums, r = rsqrt(mean(x^2) + eps) of the FFN input.
__device__ __forceinline__ void mk_geglu_tile(const MkArgs& a, int m, int part, int parts, const float* ss2,
                                              float invD, int mt) {
  const int F = a.F;
  const size_t pl = (size_t)64 * F;
  const int n = a.T_q * 16;
  for (int it = part * n / parts + mt; it < (part + 1) * n / parts; it += 256) {
    const int t = it >> 4, i = (it & 15) * 4;
    const float* gp = a.gu + (size_t)t * 2 * F + m * 128 + i;
    const float4 g = __ldcg(reinterpret_cast<const float4*>(gp));
    const float4 u = __ldcg(reinterpret_cast<const float4*>(gp + 64));
    const float rv = rsqrtf(__ldcg(ss2 + t) * invD + a.eps);
    const float h0 = gelu_tanh_fast(rv * g.x) * (rv * u.x), h1 = gelu_tanh_fast(rv * g.y) * (rv * u.y);
    const float h2 = gelu_tanh_fast(rv * g.z) * (rv * u.z), h3 = gelu_tanh_fast(rv * g.w) * (rv * u.w);
    uint32_t a0, b0, c0, a1, b1, c1;
    split_pair_exact(h0, h1, a0, b0, c0);
    split_pair_exact(h2, h3, a1, b1, c1);
    uint2* d = reinterpret_cast<uint2*>(a.h_planes + (size_t)t * F + m * 64 + i);
    d[0] = make_uint2(a0, a1);
    d[pl / 4] = make_uint2(b0, b1);
    d[pl / 2] = make_uint2(c0, c1);
  }
}

// After the gate/up epilogue: every CTA of a tile (all K ranges) waits for
// the tile, then writes its share of the tile's GeGLU planes.
__device__ __forceinline__ void mk_gu_arrive(const MkArgs& a, int lr, float invD, int mt) {
  const MkGemm& g = a.g[2];
  const MkRange r = mk_range(g, blockIdx.x);
  if (!r.active) return;
  const unsigned extra = (lr == 0 && a.skew_where == 3) ? a.skew : 0u;
  mk_group_wait(a.grp_cnt + kCntGuArr + r.m, (unsigned)((lr + 1) * g.splits) + extra, a.err, 902, mt);
  mk_geglu_tile(a, r.m, (int)blockIdx.x / g.MT, g.splits, a.ss + (kSsGu + r.m) * 64, invD, mt);
}

template <int DH>
__global__ void __launch_bounds__(kMkThreads, 1)
    pi0_step_kernel(const __grid_constant__ CUtensorMap w_qkv, const __grid_constant__ CUtensorMap w_o,
                    const __grid_constant__ CUtensorMap w_gu, const __grid_constant__ CUtensorMap w_d,
                    const __grid_constant__ CUtensorMap act_op, const __grid_constant__ CUtensorMap act_hp,
                    const MkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;
  uint8_t* sR = smem + kMkNW * kMkWBytes;
  uint8_t* sB = sR;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sR + kMkRegion);
  uint64_t* wfull = bars;                  // weight tile landed
  uint64_t* wempty = wfull + kMkNW;        // weight slot free (MMA done)
  uint64_t* bfull = wempty + kMkNW;        // operand tile built by the math warps (8 arrivals)
  uint64_t* bfullt = bfull + kMkNB;        // operand tile landed by TMA (O and down projections)
  uint64_t* bempty = bfullt + kMkNB;       // operand slot free (MMA done)
  uint64_t* accfull = bempty + kMkNB;      // accumulator complete
  uint64_t* mdone = accfull + 1;           // every MMA complete (teardown)
  uint64_t* go = mdone + 1;                // grid barrier passed before a projection phase
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(go + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kMkNW; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], 1);
    }
    for (int i = 0; i < kMkNB; ++i) {
      mbar_init(&bfull[i], 8);
      mbar_init(&bfullt[i], 1);
      mbar_init(&bempty[i], 1);
    }
    mbar_init(accfull, 1);
    mbar_init(mdone, 1);
    mbar_init(go, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;");
    if (warp == 0 && lane == 0) {
      // ---------------- weight stream ----------------
      tma_prefetch_desc(&w_qkv);
      tma_prefetch_desc(&w_o);
      tma_prefetch_desc(&w_gu);
      tma_prefetch_desc(&w_d);
      const uint64_t pol = l2_policy_evict_first();
      uint32_t wt = 0;
      bool ok = true;
      for (int l = a.l0; l < a.l1 && ok; ++l)
        for (int gi = 0; gi < 4 && ok; ++gi) {
          const MkRange r = mk_range(a.g[gi], blockIdx.x);
          if (!r.active) continue;
          const CUtensorMap* map = gi == 0 ? &w_qkv : gi == 1 ? &w_o : gi == 2 ? &w_gu : &w_d;
          const int row = l * a.g[gi].N + r.m * 128;
          for (int k = r.k0; k < r.k1; ++k) {
            const uint32_t s = wt % kMkNW;
            if (!mk_wait(&wempty[s], ((wt / kMkNW) & 1) ^ 1, a.err, 20)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&wfull[s], kMkWBytes);
            tma_load_2d(sW + s * kMkWBytes, map, &wfull[s], k * 64, row, pol);
            ++wt;
          }
        }
      // never leave a copy in flight into this CTA's shared memory
      for (uint32_t i = wt > (uint32_t)kMkNW ? wt - kMkNW : 0; i < wt; ++i)
        mbar_wait(&wfull[i % kMkNW], (i / kMkNW) & 1, nullptr, 0);
    } else if (warp == 1 && lane == 0) {
      // ---------------- MMA issue ----------------
      const uint32_t idesc = idesc_bf16_f32(128, 192);
      uint32_t wt = 0, bt = 0, gc = 0, pf = 0, pt = 0;   // pf / pt: per-slot parities of bfull / bfullt
      bool ok = true;
      for (int l = a.l0; l < a.l1 && ok; ++l)
        for (int gi = 0; gi < 4 && ok; ++gi) {
          const MkRange r = mk_range(a.g[gi], blockIdx.x);
          if (!r.active) continue;
          const uint32_t acc = tmem + (gc & 1) * 256;
          for (int k = r.k0; k < r.k1; ++k) {
            const uint32_t b = bt % kMkNB, s = wt % kMkNW;
            const bool tma_b = gi == 1 || gi == 3;
            uint64_t* bf = tma_b ? &bfullt[b] : &bfull[b];
            const uint32_t par = ((tma_b ? pt : pf) >> b) & 1u;
            if (!mk_wait(bf, par, a.err, 21) || !mk_wait(&wfull[s], (wt / kMkNW) & 1, a.err, 22)) {
              ok = false;
              break;
            }
            if (tma_b) pt ^= 1u << b;
            else pf ^= 1u << b;
            tc_fence_after();
            const uint32_t wa = smem_u32(sW + s * kMkWBytes), ba = smem_u32(sB + b * kMkBBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_ss(acc, desc_k_sw128(wa + kk * 32), desc_k_sw128(ba + kk * 32), idesc,
                          (k != r.k0 || kk != 0) ? 1u : 0u);
            mma_commit(&wempty[s]);
            mma_commit(&bempty[b]);
            ++wt;
            ++bt;
          }
          if (!ok) break;
          mma_commit(accfull);
          ++gc;
        }
      mma_commit(mdone);   // every MMA of this CTA has completed before TMEM is freed
      mbar_wait(mdone, 0, nullptr, 0);
    } else if (warp == 2 && lane == 0) {
      // ---------------- activation loader ----------------
      // after each grid barrier that opens the output or the down projection:
      // the operand planes straight into the operand slots (the math warps
      // build the QKV and gate/up operands from x themselves)
      tma_prefetch_desc(&act_op);
      tma_prefetch_desc(&act_hp);
      const uint64_t pol = l2_policy_evict_last();
      uint32_t bt = 0, gop = 0;
      uint32_t bout = 0;            // operand copies issued, by slot (bit)
      uint32_t pt = 0;              // per-slot parity of bfullt
      bool ok = true;
      for (int l = a.l0; l < a.l1 && ok; ++l)
        for (int gi = 0; gi < 4 && ok; ++gi) {
          if (!mk_wait(go, gop & 1, a.err, 40)) {
            ok = false;
            break;
          }
          ++gop;
          fence_proxy_async_global();
          fence_proxy_async_smem();
          const MkRange r = mk_range(a.g[gi], blockIdx.x);
          if (!r.active) continue;
          const int nk = r.k1 - r.k0;
          if (gi == 1 || gi == 3) {   // operand planes straight into the operand slots
            const CUtensorMap* map = gi == 1 ? &act_op : &act_hp;
            for (int j = 0; j < nk; ++j) {
              const uint32_t b = bt % kMkNB;
              if (!mk_wait(&bempty[b], ((bt / kMkNB) & 1) ^ 1, a.err, 41)) {
                ok = false;
                break;
              }
              fence_proxy_async_smem();
              mbar_arrive_expect_tx(&bfullt[b], kMkBBytes);
              tma_load_2d(sB + b * kMkBBytes, map, &bfullt[b], (r.k0 + j) * 64, 0, pol);
              bout |= 1u << b;
              pt ^= 1u << b;
              ++bt;
            }
          } else {                    // built by the math warps
            bt += nk;
          }
        }
      // never leave a copy in flight: every operand copy has landed
      for (int i = 0; i < kMkNB; ++i)
        if ((bout >> i) & 1u) mbar_wait(&bfullt[i], ((pt >> i) & 1u) ^ 1u, nullptr, 0);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 224;");
    // ---------------- math warps ----------------
    MkMath s;
    s.sB = sB;
    s.bfull = bfull;
    s.bempty = bempty;
    s.accfull = accfull;
    s.go = go;
    s.tmem = tmem;
    s.bt = s.gc = 0;
    s.mt = threadIdx.x - 128;
    const int mt = s.mt;
    const unsigned G = gridDim.x;
    unsigned nbar = 0;
    const float invD = 1.f / (float)a.D;
    const int kvd = a.Hkv * DH;
    for (int l = a.l0; l < a.l1; ++l) {
      __nv_bfloat16* kc = a.kv + (size_t)(l - a.l0) * a.kv_stride;
      __nv_bfloat16* vc = kc + (size_t)a.T_kv * kvd;
      unsigned long long* tr =
          (a.trace && mt == 0) ? a.trace + ((size_t)(l - a.l0) * gridDim.x + blockIdx.x) * 64 : nullptr;
      mk_mark(tr, 0);
      // phases: 0 QKV (+ q / own k, v), 2 attention, 3 combine, 4 O, 5 gate/up
      // (+ GeGLU planes), 7 down; a grid barrier before each (the first one of
      // a launch has none).  Indices 1 and 6 (former separate finalize phases)
      // are skipped so trace slots keep their meaning.
      const int lr = l - a.l0;
      for (int ph = 0; ph < 8; ++ph) {
        if (ph == 1 || ph == 6) continue;   // finalized inside the QKV and gate/up phases
        if (ph > 0 || l > a.l0) {
          ++nbar;
          const unsigned extra = (nbar == 1 && a.skew_where == 1) ? a.skew : 0u;
          mk_grid_sync(a.bar, nbar * G + extra, a.err, mt);
        }
        const bool proj = ph == 0 || ph == 4 || ph == 5 || ph == 7;
        if (proj && mt == 0) mbar_arrive(go);   // the loader may fetch this phase's operand
        mk_mark(tr, 2 * ph + 1);
        if (ph == 2) {
          mk_attention<DH>(a, kc, vc, sR, mt, tr);
        } else if (ph == 3) {
          mk_combine<DH>(a, mt, reinterpret_cast<float*>(sR), tr);
          // the QKV sums and statistics of the next block start from zero
          // (every finalizer of this block is done before the barrier that
          // opened phase 2)
          mk_zero_f4(a.qkv, 16 * a.nqkv, mt);
          mk_zero_f4(a.ss + kSsQkv * 64, 16 * (kSsGu - kSsQkv), mt);
        } else {
          const int gi = ph == 0 ? 0 : ph == 4 ? 1 : ph == 5 ? 2 : 3;
          float* out = ph == 0 ? a.qkv : ph == 5 ? a.gu : a.x;
          const int ld = ph == 0 ? a.nqkv : ph == 5 ? 2 * a.F : a.D;
          const MkRange r = mk_range(a.g[gi], blockIdx.x);
          float* stats = nullptr;   // this K range's sums of squares of x, into its group's row
          if (ph == 0 && r.m % MkQkvGroups<DH>::MPG == 0) stats = a.ss + (kSsQkv + r.m / MkQkvGroups<DH>::MPG) * 64;
          if (ph == 5) stats = a.ss + (kSsGu + r.m) * 64;
          mk_gemm_math(s, a.g[gi], ph == 0 || ph == 5 ? a.x : nullptr, a.D, stats, out, ld, a.T_q, a.err,
                       tr ? tr + 20 + 4 * gi : nullptr);
          if (ph == 0) mk_qkv_arrive<DH>(a, lr, kc, vc, invD, mt);
          if (ph == 5) mk_gu_arrive(a, lr, invD, mt);
          // the gate/up sums and statistics of the next block start from zero
          // (every GeGLU tile of this block was written before the barrier that
          // opened phase 7)
          if (ph == 7) {
            mk_zero_f4(a.gu, 32 * a.F, mt);
            mk_zero_f4(a.ss + kSsGu * 64, 16 * (kSsRows - kSsGu), mt);
          }
        }
        mk_mark(tr, 2 * ph + 2);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace lat
