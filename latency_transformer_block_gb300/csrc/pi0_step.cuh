// Persistent kernel for the pi0 action expert: the blocks of one denoise step,
// or (chunk kernel) a whole denoised chunk -- every step's embedding, W2
// projection, blocks and head -- in one launch.
//
// "Running VLAs at Real-time Speed" (reading note, sections 3 and 6) puts the
// action expert's time into launch gaps and into streaming every block's
// weights once per step; the TileRT page describes a persistent engine that
// keeps weight loads running while compute waits on its dependencies.  Here one
// CTA per SM lives for the whole launch, in thread-block clusters of 4
// (cooperative launch: every CTA is resident, which the grid barriers need):
//
//  * warp 0 streams this CTA's share of every projection's weights (128 x 64
//    fp16 tiles, TMA, 128-byte swizzle) through a ring of shared-memory slots.
//    The weights do not depend on activations, so the stream runs ahead
//    across phase (and step) boundaries and is throttled only by the ring.
//  * warp 1 issues tcgen05 MMAs (M = 128 weight rows, N = 128 = two fp16
//    planes x 64 tokens, fp32 accumulator in TMEM, two buffers).
//  * warp 2 brings the operand planes of the O, down and W2 projections by
//    TMA once the grid barrier before them has passed.
//  * warps 4..11 ("math") do everything that depends on activations: they
//    load the fp32 residual stream (several k-tiles in flight, in registers)
//    and split it into two fp16 planes (hi = fp16(x), lo = fp16(x - hi)) in
//    the MMA's swizzled layout, run the split-K epilogues, the attention, the
//    combine of key-range partials and (chunk kernel) the head and embedding.
//  * Weights are held as fp16 = 2^s x the folded bf16 weight (exact); the
//    epilogue multiplies by 2^-s.
//
// Per block six phases, separated by a grid barrier (bounded spin):
//   QKV projection of x: the 4 CTAs of a cluster take the 4 K ranges of one
//     128-row tile; their partial sums (and the per-token sums of squares of
//     x) meet in the cluster by bulk copies into the finalizing CTA's shared
//     memory; each CTA finalizes a quarter of the tile's rows (whole rotary
//     pairs: RMS factor, RoPE, q planes, own k / v into the cache)
//   attention: per (head, 32-key block), partial (max, sum, output)
//   combine of the key-block partials into the fp16 planes of o
//   x += o Wo: every CTA adds its K range's partial sums into x (vector
//     reductions at L2)
//   gate/up projection of x (gate and up rows of the same 64 FFN columns in
//     one 128-row tile; two tiles x two K ranges per cluster, exchanged like
//     QKV); h = GELU(r g) * (r u) as fp16 planes
//   x += h Wd, like O
// The RMSNorm scales are folded into the weights; the per-token factor
// r = rsqrt(mean(x^2) + eps) multiplies the projection sums (the projection is
// linear in its input), as in the pages' fold (section 4.1).
#pragma once
#include "attention.cuh"
#include "common.cuh"
#include "skinny_gemm.cuh"

namespace lat {

constexpr int kMkThreads = 384;                 // 12 warps
constexpr int kMkCluster = 4;                   // CTAs per thread-block cluster
constexpr int kMkNW = 6;                        // weight ring slots
constexpr int kMkNB = 4;                        // activation-plane ring slots
constexpr int kMkPre = 5;   // k-tiles of x the math warps hold in flight (registers)
constexpr int kMkWBytes = 128 * 64 * 2;         // one weight tile
constexpr int kMkBBytes = 128 * 64 * 2;         // one activation tile, two fp16 planes
// cluster exchange area (after the operand slots): 4 slots of split-K partial
// sums [64 tokens][32 rows] fp32, written by the CTAs of the cluster into the
// CTA that finalizes those rows, then 4 x 64 per-token sums of squares of x
constexpr int kMkXSlot = 64 * 32 * 4;
constexpr int kMkXOff = kMkNB * kMkBBytes;
constexpr int kMkXBytes = 4 * kMkXSlot + 4 * 64 * 4;
constexpr int kMkRegion = 99 * 1024;            // also the attention's tiles (its own phase)
static_assert(kMkXOff + kMkXBytes <= kMkRegion, "operand slots and exchange area fit in the region");
constexpr int kMkBars = 2 * kMkNW + 3 * kMkNB + 6;
static_assert(kMkRegion % 1024 == 0, "the weight ring after the region stays 1024-byte aligned");

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

// One projection: MT tiles of 128 output rows (N rows of one layer's matrix
// in the stacked weight tensor), KT tiles of 64 inputs.  CTA b is rank
// b % 4 of cluster c = b / 4.
//  pair = 0: cpm clusters per tile split its K into 4 cpm ranges (cluster c
//            takes tile c / cpm; its ranks take 4 consecutive ranges); the 4
//            partial sums of each row meet in the cluster: rank j finalizes
//            rows 32 j .. 32 j + 31 of the tile.
//  pair = 1: cluster c takes tiles 2 c and 2 c + 1, each split into 2 K
//            ranges (ranks 2 i, 2 i + 1 of tile 2 c + i).
//  direct = 1: no exchange; CTA b takes tile b % MT and K range b / MT of
//            `splits` and adds its partial sums into the output itself.
struct MkGemm {
  int MT, KT, N, pair, cpm, direct, splits;
};

struct MkArgs {
  MkGemm g[5];              // 0 QKV, 1 O, 2 gate/up, 3 down, 4 W2 (the embedding's second projection)
  int l0, l1;               // layers [l0, l1) of this launch
  int steps;                // 0: the blocks once (one denoise step, or one block); > 0: a whole chunk of
                            // `steps` denoise steps, each embedding + W2 + every block, then the head
  int D, F, Hq, Hkv, T_q, T_prefix, T_kv, nqkv;
  int prefix_lm;            // 1: the state token (query row 0) sees the prefix and itself only
  float eps, scale_log2;
  float* x;                 // fp32 [64][D] residual stream (rows >= T_q stay 0)
  __half* o_planes;         // [2][64][Hq dh] attention output as two fp16 planes (rows >= T_q stay 0)
  __half* h_planes;         // [2][64][F] GeGLU output as two fp16 planes (rows >= T_q stay 0)
  float wsc[5];             // 2^-s of each projection's weights (held as fp16 = 2^s w, exact)
  // chunk mode: the embedding and head around the blocks (all fp32 unless noted)
  float* act;               // [T_q - 1][A] actions: the noise in, the actions out (x <- x + dt v)
  float* act_buf;           // [2][T_q - 1][A] the actions between steps (step s writes buffer s mod 2)
  const float* state;       // [A]
  const __nv_bfloat16* w_state;   // bf16 [A][D]
  const __nv_bfloat16* b_state;   // bf16 [D]
  float* state_emb;         // [D] state row, written at step 0
  const float* wfold;       // [A][D] W' = W_in W1_a
  const float* ttab;        // [S][D] T[s]
  const float* b2;          // [D]
  __half* e_planes;         // [2][64][D] SiLU(x W' + T[s]) of the action rows (row 1 + t) as two fp16
                            // planes, the W2 operand (row 0 and rows >= T_q stay 0)
  const __nv_bfloat16* w_out;   // bf16 [D][A] (the head's weight; copied whole into shared memory)
  const float* g_final;     // [D] the final RMSNorm scale
  const float* bout;        // [A]
  const float* dt;          // [S]
  int A;
  __nv_bfloat16* q_planes;  // [2][64][Hq dh] q after RoPE, two-term bf16 (hi, lo)
  __nv_bfloat16* kv_own;    // [k hi, k lo, v hi, v lo][64][Hkv dh] own keys / values, two-term bf16
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
  DevErr* err;
  int skew_where;           // failure-detection hook: 0 off; 1 the first grid barrier, 2 the first QKV
                            // exchange, 3 the first gate/up exchange of the launch waits for
  unsigned skew;            // this many phases more than will ever complete (the wait runs out, the
                            // error word records a timeout and every later wait returns at once)
  unsigned long long* trace;   // null, or [layers][trace_stride][64] phase timestamps (ns): 0..14 block
                               // start and the ends of each phase / barrier, 16..18 attention,
                               // 20 + 4 g .. 23 + 4 g projection g, 38 + g its cluster exchange received
  int trace_stride;
};

struct MkRange {
  int m, k0, k1;
  bool active;
};

__device__ __forceinline__ MkRange mk_range(const MkGemm& g, int b) {
  MkRange r;
  const int c = b / kMkCluster, q = b % kMkCluster;
  int s, S;
  if (g.direct) {
    r.active = b < g.MT * g.splits;
    r.m = b % g.MT;
    s = b / g.MT;
    S = g.splits;
  } else if (g.pair) {
    r.active = c < g.MT / 2;
    r.m = 2 * c + (q >> 1);
    s = q & 1;
    S = 2;
  } else {
    r.active = c < g.MT * g.cpm;
    r.m = c / g.cpm;
    s = (c % g.cpm) * kMkCluster + q;
    S = kMkCluster * g.cpm;
  }
  r.k0 = s * g.KT / S;
  r.k1 = (s + 1) * g.KT / S;
  return r;
}

// Position in a launch's order of projections: per denoise step (chunk mode)
// W2, then per block QKV, O, gate/up, down.
struct MkPos {
  int s, l, gi;
  bool valid;
};

__device__ __forceinline__ MkPos mk_seq_first(const MkArgs& a) {
  MkPos p;
  p.s = 0;
  p.l = a.l0;
  p.gi = a.steps > 0 ? 4 : 0;
  p.valid = a.l1 > a.l0;
  return p;
}

__device__ __forceinline__ void mk_seq_next(const MkArgs& a, MkPos& p) {
  if (p.gi == 4) {
    p.gi = 0;
    p.l = a.l0;
    return;
  }
  if (++p.gi < 4) return;
  p.gi = 0;
  if (++p.l < a.l1) return;
  if (a.steps > 0 && ++p.s < a.steps) {
    p.gi = 4;
    return;
  }
  p.valid = false;
}

__device__ __forceinline__ bool mk_aborted(DevErr* e) { return *reinterpret_cast<volatile unsigned*>(&e->code) != 0; }

// An activation outside the fp16 operand planes' range.  Not recorded once
// the launch has given up on a wait: the math warps then run on to the end
// over values that no longer mean anything.
__device__ __forceinline__ void mk_range_error(DevErr* e, unsigned where) {
  if (!mk_aborted(e)) record_error(e, kErrRange, where);
}

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

// The same for an mbarrier completed by copies from other CTAs of the cluster
// (acquire at cluster scope).  It does not give up early when another CTA has
// failed: every CTA of an active cluster always sends its partial sums, so the
// bytes always come, and no copy may still be on its way into this CTA when it
// leaves; only the spin budget ends it.
__device__ __forceinline__ bool mk_wait_cluster(uint64_t* bar, uint32_t parity, DevErr* err, unsigned where) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  for (int i = 0;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 63) == 63 && clock64() - t0 > kSpinBudget) {
      record_error(err, 1u, where);
      return false;
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

// Shared state of the math warps.  Every shared-memory address is a fixed
// offset from the (1024-byte aligned) base, so only the base is kept:
//   [weight slots kMkNW x kMkWBytes][region kMkRegion: operand slots, exchange
//   slots and statistics][mbarriers: wfull[NW] wempty[NW] bfull[NB] bfullt[NB]
//   bempty[NB] accfull mdone go xfull never hfull][TMEM address, re-arm table]
struct MkMath {
  uint8_t* base;
  uint32_t tmem;
  uint32_t bt, gc, xuse;
  bool xbroken;       // an exchange wait ran out: no further arming or waiting
  int mt;
  __device__ __forceinline__ uint8_t* sB() const { return base + kMkNW * kMkWBytes; }   // operand slots
  // cluster exchange slots [4][64 tokens][32 rows] and [4][64] sums of squares of x, by source K range
  __device__ __forceinline__ float* xbuf() const { return reinterpret_cast<float*>(sB() + kMkXOff); }
  __device__ __forceinline__ float* xss() const { return xbuf() + kMkCluster * (kMkXSlot / 4); }
  __device__ __forceinline__ uint64_t* bars() const { return reinterpret_cast<uint64_t*>(sB() + kMkRegion); }
  __device__ __forceinline__ uint64_t* bfull() const { return bars() + 2 * kMkNW; }
  __device__ __forceinline__ uint64_t* bempty() const { return bars() + 2 * kMkNW + 2 * kMkNB; }
  __device__ __forceinline__ uint64_t* accfull() const { return bars() + 2 * kMkNW + 3 * kMkNB; }
  __device__ __forceinline__ uint64_t* go() const { return accfull() + 2; }
  // exchange complete: armed by this CTA with the bytes it will receive
  __device__ __forceinline__ uint64_t* xfull() const { return accfull() + 3; }
  // an mbarrier nothing arrives on (failure hook)
  __device__ __forceinline__ uint64_t* never() const { return accfull() + 4; }
  // the head's weight landed in the operand slots (chunk mode)
  __device__ __forceinline__ uint64_t* hfull() const { return accfull() + 5; }
  // after the barriers: the TMEM address, then the re-arm table (mk_xtable)
  __device__ __forceinline__ const uint32_t* xtable() const {
    return reinterpret_cast<const uint32_t*>(bars() + kMkBars) + 1;
  }
};

// does cluster c take part in the exchange of this projection
__device__ __forceinline__ bool mk_cluster_active(const MkGemm& g, int c) {
  if (g.direct) return false;
  return g.pair ? c < g.MT / 2 : c < g.MT * g.cpm;
}

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

// bytes a CTA receives in the exchange of projection gi: the 4 slots of
// partial sums, plus the sums of squares of x (QKV: 4 K ranges; gate/up: 2)
__device__ __forceinline__ uint32_t mk_xbytes(int gi) {
  return 4 * kMkXSlot + (gi == 0 ? 4 * 256 : gi == 2 ? 2 * 256 : 0);
}

// The exchanges of cluster c: QKV (gi 0) and gate/up (gi 2) of every block,
// where the cluster holds tiles of them (O, down and W2 add their partial sums
// into x directly).  Bytes of the cluster's first exchange of the launch, and
// of the one after its exchange in projection gi at position p (0 after the
// last one).
__device__ __forceinline__ uint32_t mk_first_xbytes(const MkArgs& a, int c) {
  if (a.l1 <= a.l0) return 0;
  return mk_cluster_active(a.g[0], c) ? mk_xbytes(0) : mk_cluster_active(a.g[2], c) ? mk_xbytes(2) : 0;
}

// The table the math warps re-arm from (set up once per launch, in shared
// memory): [0] bytes after a QKV exchange, [1] after a gate/up exchange.
__device__ __forceinline__ void mk_xtable(const MkArgs& a, int c, uint32_t* t) {
  const bool q_on = mk_cluster_active(a.g[0], c), u_on = mk_cluster_active(a.g[2], c);
  t[0] = mk_xbytes(u_on ? 2 : 0);
  t[1] = mk_xbytes(q_on ? 0 : 2);
}

// Math side of one projection.  Projections of the residual stream x (QKV,
// gate/up): the math warps load their rows of x straight from global memory,
// PRE k-tiles in flight in registers, and write the exact bf16 planes into
// the operand slots; for the others (act == nullptr) the loader brings the
// planes by TMA.  Then the split-K epilogue: each warp sums the three planes
// of its quarter of the tile's rows and stores them, through distributed
// shared memory, into the exchange slot of the cluster rank that finalizes
// those rows; with `stats` the per-token sums of squares of this K range go
// to the ranks that need them.  Every warp then arrives on every rank's
// exchange barrier.
// 16 bytes from global memory through L2 (not L1: other SMs write x), issued
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

template <int PRE>
__device__ __forceinline__ void mk_gemm_math(MkMath& s, const MkGemm& g, const float* act, int act_ld, bool stats,
                                             float wsc, float* out, int ld, int T_q, DevErr* err,
                                             unsigned long long* tr) {
  const MkRange r = mk_range(g, blockIdx.x);
  if (!r.active) return;
  const int nk = r.k1 - r.k0;
  const int mw = s.mt >> 5, lane = s.mt & 31;
  const uint32_t rank = blockIdx.x % kMkCluster;
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
    float amax = 0.f;   // largest |x| converted (fp16 planes hold |x| < 65504)
    float4 xv[PRE][4];
#pragma unroll
    for (int u = 0; u < PRE; ++u)
      if (u < nk) mk_load_tile(act, act_ld, r.k0 + u, rows, p, xv[u]);
    mk_mark(tr, 0);
    for (int j0 = 0; j0 < nk; j0 += PRE) {
#pragma unroll
      for (int u = 0; u < PRE; ++u) {
        const int j = j0 + u;
        if (j < nk) {
          const uint32_t b = s.bt % kMkNB;
          mk_wait(&s.bempty()[b], ((s.bt / kMkNB) & 1) ^ 1, err, 31);
          uint8_t* dst = s.sB() + b * kMkBBytes;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int t = rows[i];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int col = hh * 32 + 4 * p;
              const float4 v = xv[u][2 * i + hh];
              if (stats) sq[i] += (v.x * v.x + v.y * v.y) + (v.z * v.z + v.w * v.w);
              amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
              uint32_t h0, l0, h1, l1;
              split_pair_h2(v.x, v.y, h0, l0);
              split_pair_h2(v.z, v.w, h1, l1);
              const uint32_t off = (uint32_t)(t * 128 + ((((col >> 3) ^ t) & 7) << 4) + ((p & 1) << 3));
              *reinterpret_cast<uint2*>(dst + off) = make_uint2(h0, h1);
              *reinterpret_cast<uint2*>(dst + 8192 + off) = make_uint2(l0, l1);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.bfull()[b]);   // this warp's rows of the operand are written
          ++s.bt;
          if (j + PRE < nk) mk_load_tile(act, act_ld, r.k0 + j + PRE, rows, p, xv[u]);
        }
      }
    }
    if (!(amax < kF16Max)) mk_range_error(err, 33);
  }
  // this K range's per-token sums of squares of x (lanes p == 0 hold rows[i])
  float ssq[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float v = sq[i];
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    ssq[i] = v;
  }
  // epilogue: warp (4 + mw) reads TMEM lanes 32 q .. +31 = rows of the tile,
  // tokens 32 ch .. +31 of each plane, sums the planes hi + lo and undoes the
  // weights' power-of-two scale
  if (act) mk_mark(tr, 1);
  mk_wait(s.accfull(), s.gc & 1, err, 32);
  mk_mark(tr, 2);
  tc_fence_after();
  const uint32_t acc = s.tmem + (s.gc & 1) * 256;
  ++s.gc;
  const int q = mw & 3, ch = mw >> 2;
  const uint32_t tb = acc + ((uint32_t)(q * 32) << 16) + (uint32_t)(ch * 32);
  float v[32], w[32];
  tmem_ld32x2(tb, tb + 64, v, w);
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = (v[j] + w[j]) * wsc;
  tc_fence_before();
  if (g.direct) {
    // each lane quad transposes 4 tokens x its 4 rows, so a lane adds 4
    // consecutive outputs of one token: one vector reduction into `out`
    const int k4 = lane & 3;
    const int fb = r.m * 128 + q * 32 + lane - k4;
#pragma unroll
    for (int j0 = 0; j0 < 32; j0 += 4) {
      float a0 = v[j0], a1 = v[j0 + 1], a2 = v[j0 + 2], a3 = v[j0 + 3];
      quad_transpose(a0, a1, a2, a3, k4);
      const int t = ch * 32 + j0 + k4;
      if (t < T_q) red_add_v4(out + (size_t)t * ld + fb, a0, a1, a2, a3);
    }
    mk_mark(tr, 3);
    return;
  }
  // every MMA of the projection is complete, so the operand slots are free:
  // stage this warp's block, [token][row] (32 x 32 fp32), and the statistics
  float* stg = reinterpret_cast<float*>(s.sB()) + mw * 1024;
#pragma unroll
  for (int j = 0; j < 32; ++j) stg[j * 32 + lane] = v[j];
  float* sst = reinterpret_cast<float*>(s.sB()) + 8 * 1024;
  if (stats && p == 0) {
    sst[rows[0]] = ssq[0];
    sst[rows[1]] = ssq[1];
  }
  fence_proxy_async_smem();
  __syncwarp();
  // the block goes to the rank that finalizes these rows, into the slot of
  // this K range (tokens 32 ch ..): one bulk copy, completing on its barrier
  uint32_t dest, slot;
  if (g.pair) {
    dest = (rank & 2) | (uint32_t)(q & 1);       // the K range (q & 1) of this tile finalizes its half
    slot = (rank & 1) * 2 + (uint32_t)(q >> 1);  // [source K range][gate | up]
  } else {
    dest = (uint32_t)q;
    slot = rank;
  }
  if (lane == 0)
    bulk_copy_to_cluster(cluster_map(smem_u32(s.xbuf() + slot * (kMkXSlot / 4) + ch * 1024), dest), smem_u32(stg),
                         4096u, cluster_map(smem_u32(s.xfull()), dest));
  if (stats) {
    // the sums of squares of this K range: to every rank (QKV) or to the two
    // ranks of this tile (gate/up), in the row of this K range
    named_sync(2, 256);
    if (s.mt == 0) {
      const uint32_t src = g.pair ? (rank & 1) : rank;
      const uint32_t at = smem_u32(s.xss() + src * 64);
      for (uint32_t d = 0; d < kMkCluster; ++d)
        if (!g.pair || (d & 2) == (rank & 2))
          bulk_copy_to_cluster(cluster_map(at, d), smem_u32(sst), 256u, cluster_map(smem_u32(s.xfull()), d));
    }
  }
  mk_mark(tr, 3);
}

// Wait until this CTA has received every byte of the exchange of projection
// gi (its partial sums and statistics from the cluster), then arm the barrier
// with the bytes of its next exchange; with `skew` first a wait that nothing
// completes.
__device__ __forceinline__ void mk_exchange_wait(MkMath& s, const MkArgs& a, int gi, bool skew, unsigned where) {
  if (skew) mk_wait(s.never(), 0, a.err, where + 100);
  if (s.xbroken) return;
  const bool ok = mk_wait_cluster(s.xfull(), s.xuse & 1, a.err, where);
  ++s.xuse;
  if (!ok) {
    s.xbroken = true;
    return;
  }
  // armed for the next exchange even after the last one: a barrier left
  // expecting bytes at exit is harmless (nothing is in flight to this CTA)
  if (s.mt == 0) mbar_arrive_expect_tx(s.xfull(), s.xtable()[gi >> 1]);
}

// QKV: rank j of the cluster of tile u finalizes the tile's rows 32 j .. +31,
// which hold 16 rotary pairs (the weight rows are permuted at fold time: row
// 32 j + c holds the first element of pair 16 j + c of the tile, row
// 32 j + 16 + c its partner dh / 2 further on).  Per token: the sum of the 4 K
// ranges times r = rsqrt(mean(x^2) + eps), RoPE on q and k heads, two-term
// bf16 planes into q_planes / kv_own, and k, v (nearest bf16) into the cache
// at slot T_prefix + t.
// The rotation angles of a thread's (at most 4) items, loaded before the
// exchange wait so that their latency overlaps it.
struct MkRot {
  float c[4], s[4];
};

template <int DH>
__device__ __forceinline__ MkRot mk_qkv_angles(const MkArgs& a, int u, int j, int mt) {
  constexpr int PPH = DH / 2;
  MkRot rot;
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    const int it = mt + 256 * n;
    rot.c[n] = 1.f;
    rot.s[n] = 0.f;
    if (it < a.T_q * 16) {
      const int t = it >> 4, c = it & 15;
      const int P = 64 * u + 16 * j + c;
      if (P / PPH < a.Hq + a.Hkv) {
        rot.c[n] = __ldg(a.cos_t + (size_t)t * PPH + P % PPH);
        rot.s[n] = __ldg(a.sin_t + (size_t)t * PPH + P % PPH);
      }
    }
  }
  return rot;
}

template <int DH>
__device__ __forceinline__ void mk_qkv_finalize(const MkArgs& a, int u, int j, const float* xbuf, const float* xss,
                                                __nv_bfloat16* kc, __nv_bfloat16* vc, float invD, const MkRot& rot,
                                                int mt) {
  constexpr int PPH = DH / 2;   // rotary pairs per head
  const int qd = a.Hq * DH, kvd = a.Hkv * DH;
  const size_t qpl = (size_t)64 * qd, kpl = (size_t)64 * kvd;
#pragma unroll
  for (int n = 0; n < 4; ++n) {   // T_q <= 64: at most 4 items of 16 pairs x T_q tokens per thread
    const int it = mt + 256 * n;
    if (it >= a.T_q * 16) break;
    const int t = it >> 4, c = it & 15;
    float x0 = 0.f, x1 = 0.f;
#pragma unroll
    for (int src = 0; src < kMkCluster; ++src) {
      x0 += xbuf[src * 2048 + t * 32 + c];
      x1 += xbuf[src * 2048 + t * 32 + 16 + c];
    }
    const float ss = (xss[t] + xss[64 + t]) + (xss[128 + t] + xss[192 + t]);
    const float rv = rsqrtf(ss * invD + a.eps);
    x0 *= rv;
    x1 *= rv;
    const int P = 64 * u + 16 * j + c;
    const int head = P / PPH, i = P % PPH;
    // q and k heads are rotated (v heads carry cos 1, sin 0)
    const float y0 = x0 * rot.c[n] - x1 * rot.s[n];
    const float y1 = x1 * rot.c[n] + x0 * rot.s[n];
    const __nv_bfloat16 h0 = __float2bfloat16_rn(y0), h1 = __float2bfloat16_rn(y1);
    const __nv_bfloat16 l0 = __float2bfloat16_rn(y0 - __bfloat162float(h0));
    const __nv_bfloat16 l1 = __float2bfloat16_rn(y1 - __bfloat162float(h1));
    if (head < a.Hq) {
      __nv_bfloat16* q = a.q_planes + (size_t)t * qd + head * DH + i;
      q[0] = h0;
      q[PPH] = h1;
      q[qpl] = l0;
      q[qpl + PPH] = l1;
    } else {
      const bool isk = head < a.Hq + a.Hkv;
      const int kh = isk ? head - a.Hq : head - a.Hq - a.Hkv;
      __nv_bfloat16* o = a.kv_own + (isk ? 0 : 2 * kpl) + (size_t)t * kvd + kh * DH + i;
      o[0] = h0;
      o[PPH] = h1;
      o[kpl] = l0;
      o[kpl + PPH] = l1;
      __nv_bfloat16* cache = (isk ? kc : vc) + (size_t)(a.T_prefix + t) * kvd + kh * DH + i;
      cache[0] = h0;   // the nearest bf16 of the value
      cache[PPH] = h1;
    }
  }
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
// head), written as the two fp16 planes of the output projection's operand
// (o is a weighted mean of cached values, far inside fp16's range).  Work comes in
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
      uint32_t hi, lo;
      const size_t col = (size_t)h * DH + c;
      if (!(fmaxf(r0 < a.T_q ? fmaxf(fabsf(acc.x), fabsf(acc.y)) : 0.f,
                  r1 < a.T_q ? fmaxf(fabsf(acc.z), fabsf(acc.w)) : 0.f) < kF16Max))
        mk_range_error(a.err, 37);
      if (r0 < a.T_q) {
        split_pair_h2(acc.x, acc.y, hi, lo);
        uint32_t* d = reinterpret_cast<uint32_t*>(a.o_planes + (size_t)r0 * qd + col);
        d[0] = hi;
        d[pl / 2] = lo;
      }
      if (r1 < a.T_q) {
        split_pair_h2(acc.z, acc.w, hi, lo);
        uint32_t* d = reinterpret_cast<uint32_t*>(a.o_planes + (size_t)r1 * qd + col);
        d[0] = hi;
        d[pl / 2] = lo;
      }
    }
    named_sync(3, 256);   // sw is reused by the next chunk
    mk_mark(tr, 37);
  }
  fence_proxy_async_smem();   // sw's bytes are reused by TMA in the next phase
}

// gate/up: rank (i, k) of the cluster (tile 2 c + i, K range k) finalizes the
// FFN columns 64 m + 32 k .. +31 of its tile m: g and u are the sums of the
// two K ranges' partials, r = rsqrt(mean(x^2) + eps) of the FFN input, and
// h = GELU(r g) * (r u) goes out as the two fp16 planes of the down
// projection's operand.
__device__ __forceinline__ void mk_gu_finalize(const MkArgs& a, int m, int k, const float* xbuf, const float* xss,
                                               float invD, int mt) {
  const int F = a.F;
  const size_t pl = (size_t)64 * F;
  for (int it = mt; it < a.T_q * 8; it += 256) {
    const int t = it >> 3, c4 = (it & 7) * 4;
    const float4 g0 = *reinterpret_cast<const float4*>(xbuf + 0 * 2048 + t * 32 + c4);
    const float4 u0 = *reinterpret_cast<const float4*>(xbuf + 1 * 2048 + t * 32 + c4);
    const float4 g1 = *reinterpret_cast<const float4*>(xbuf + 2 * 2048 + t * 32 + c4);
    const float4 u1 = *reinterpret_cast<const float4*>(xbuf + 3 * 2048 + t * 32 + c4);
    const float rv = rsqrtf((xss[t] + xss[64 + t]) * invD + a.eps);
    const float h0 = gelu_tanh_fast(rv * (g0.x + g1.x)) * (rv * (u0.x + u1.x));
    const float h1 = gelu_tanh_fast(rv * (g0.y + g1.y)) * (rv * (u0.y + u1.y));
    const float h2 = gelu_tanh_fast(rv * (g0.z + g1.z)) * (rv * (u0.z + u1.z));
    const float h3 = gelu_tanh_fast(rv * (g0.w + g1.w)) * (rv * (u0.w + u1.w));
    if (!(fmaxf(fmaxf(fabsf(h0), fabsf(h1)), fmaxf(fabsf(h2), fabsf(h3))) < kF16Max)) mk_range_error(a.err, 34);
    uint32_t a0, b0, a1, b1;
    split_pair_h2(h0, h1, a0, b0);
    split_pair_h2(h2, h3, a1, b1);
    uint2* d = reinterpret_cast<uint2*>(a.h_planes + (size_t)t * F + m * 64 + k * 32 + c4);
    d[0] = make_uint2(a0, a1);
    d[pl / 4] = make_uint2(b0, b1);
  }
}

// Chunk mode: the action rows' head of the previous denoise step and the
// embedding of this one ("Running VLAs at Real-time Speed", the action
// expert's input and output projections, in the folded form of its
// section 4.2).  Action row t has the pair of CTAs 2t, 2t + 1; each computes
// the row's head (the same values) and half of its embedding columns:
//   head (step s - 1):  v[a] = r(h) sum_n g[n] h[n] W_out[n][a] + b_out[a],
//                       h = x[1 + t], r(h) = 1 / sqrt(mean(h^2) + eps),
//                       act_s[t][a] = act_{s-1}[t][a] + dt[s - 1] v[a]
//                       (written by CTA 2t: into act_buf[s mod 2], after the
//                       last step into the caller's actions; act_0, the
//                       noise, is first copied to act_buf[0], so no phase
//                       reads what it writes)
//   embedding (step s): emb[1 + t][n] = SiLU(sum_a act[t][a] W'[a][n] + T[s][n])
//                       x[1 + t][n] = b2[n]   (the W2 projection adds onto it)
// and CTA 2 (T_q - 1) the state row: x[0] = state_emb = state W_state +
// b_state (computed at step 0).  The embedding goes out as the two fp16
// planes the W2 projection's loader brings by TMA (an activation outside
// fp16's range records LAT_ERR_RANGE).  W_out was copied into the operand
// slots before the grid barrier (mk_head_prefetch, barrier `hfull`); the
// scratch lives in the exchange area.  Every read of the residual stream
// bypasses L1 (other SMs wrote it).
__device__ __forceinline__ void mk_head_embed(const MkArgs& a, int s, bool head, bool embed, uint8_t* sB,
                                              uint64_t* hfull, int mt, unsigned long long* tr) {
  const int D = a.D, A = a.A, T1 = a.T_q - 1;
  const int b = blockIdx.x;
  if (b == 2 * T1 && embed) {
    float* x0 = a.x;
    for (int n = mt; n < D; n += 256) {
      float v;
      if (s == 0) {
        v = __bfloat162float(a.b_state[n]);
        for (int j = 0; j < A; ++j) v = fmaf(a.state[j], __bfloat162float(a.w_state[(size_t)j * D + n]), v);
        a.state_emb[n] = v;
      } else {
        v = a.state_emb[n];   // written by this CTA at step 0
      }
      x0[n] = v;
    }
    return;
  }
  if (b >= 2 * T1) return;
  const int t = b >> 1, half = b & 1;
  float* sh = reinterpret_cast<float*>(sB + kMkXOff);   // [D] g (.) h
  float* part = sh + D;                                 // [256] partial sums
  float* zp = part + 256 * 4;                           // [D / 2] embedding partials
  float* xa = zp + D / 2;                               // [A] this row's actions
  float* red = xa + A;                                  // [8] + 1
  float* hrow = a.x + (size_t)(1 + t) * D;
  const size_t ra = (size_t)t * A + mt, nb = (size_t)T1 * A;
  if (mt < A) xa[mt] = __ldcg((s == 0 ? a.act : a.act_buf + ((s - 1) & 1) * nb) + ra);   // CTA 2t wrote it
  if (s == 0 && half == 0 && mt < A) a.act_buf[ra] = xa[mt];
  mk_mark(tr, 0);
  // loads that wait on nothing, issued before the ones the steps depend on
  const float bo = head && mt < A ? a.bout[mt] : 0.f;
  const float dts = head ? a.dt[s - 1] : 0.f;
  if (head) {
    float ss = 0.f;
    for (int n = 4 * mt; n < D; n += 1024) {
      const float4 v = mk_ldcg4(hrow + n);
      const float4 g = *reinterpret_cast<const float4*>(a.g_final + n);
      *reinterpret_cast<float4*>(sh + n) = make_float4(g.x * v.x, g.y * v.y, g.z * v.z, g.w * v.w);
      ss += (v.x * v.x + v.y * v.y) + (v.z * v.z + v.w * v.w);
    }
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((mt & 31) == 0) red[mt >> 5] = ss;
    mk_mark(tr, 1);
    mk_wait(hfull, (uint32_t)(s - 1) & 1u, a.err, 36);   // W_out in the operand slots
    mk_mark(tr, 2);
    named_sync(4, 256);
    if (mt == 0) {
      float tot = 0.f;
      for (int w = 0; w < 8; ++w) tot += red[w];
      red[8] = rsqrtf(tot / (float)D + a.eps);
    }
    // thread mt: column pair cp (columns 2 cp, 2 cp + 1), rows n = rp mod RP
    const int A2 = A >> 1, RP = 256 / A2;
    const int cp = mt % A2, rp = mt / A2;
    const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(sB);
    float2 acc = make_float2(0.f, 0.f);
    const int n_it = D / RP;
    for (int i0 = 0; i0 < n_it; i0 += 8) {   // 8 rows' loads in flight, then their FMAs
      __nv_bfloat162 w[8];
      float hv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int n = rp + (i0 + u < n_it ? i0 + u : 0) * RP;
        w[u] = w2[n * A2 + cp];
        hv[u] = i0 + u < n_it ? sh[n] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float2 wf = __bfloat1622float2(w[u]);
        acc.x = fmaf(hv[u], wf.x, acc.x);
        acc.y = fmaf(hv[u], wf.y, acc.y);
      }
    }
    part[rp * A + 2 * cp] = acc.x;
    part[rp * A + 2 * cp + 1] = acc.y;
    named_sync(4, 256);
    mk_mark(tr, 3);
    if (mt < A) {
      float v = 0.f;
      for (int i = 0; i < RP; ++i) v += part[i * A + mt];
      v = red[8] * v + bo;
      const float nx = xa[mt] + dts * v;
      xa[mt] = nx;
      if (half == 0) (s == a.steps ? a.act : a.act_buf + (s & 1) * nb)[ra] = nx;
    }
  }
  named_sync(4, 256);   // xa complete; every read of the row h is done
  mk_mark(tr, 4);
  if (!embed) return;
  // this CTA's half of the columns, n0 .. n0 + D / 2: thread (jh, q) sums the
  // actions jh A / 2 .. of column quad q; the second half of the actions
  // meets the first in shared memory
  const int n0 = half * (D >> 1), jh = mt >> 7, q = mt & 127;
  const int A_h = A >> 1;
  const float* tt = a.ttab + (size_t)s * D;
  __half* ehi = a.e_planes + (size_t)(1 + t) * D;
  __half* elo = ehi + (size_t)64 * D;
  for (int c0 = 0; c0 < (D >> 1); c0 += 512) {   // the same trip count in every thread (named barrier)
    const int c = c0 + 4 * q;
    const bool on = c < (D >> 1);
    const int n = n0 + (on ? c : 0);
    float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 tv = z, bv = z;
    if (jh == 0 && on) {
      tv = *reinterpret_cast<const float4*>(tt + n);
      bv = *reinterpret_cast<const float4*>(a.b2 + n);
    }
    const float* wf = a.wfold + (size_t)(jh * A_h) * D + n;
#pragma unroll 16
    for (int j = 0; j < (on ? A_h : 0); ++j) {
      const float4 w = *reinterpret_cast<const float4*>(wf + (size_t)j * D);
      const float xj = xa[jh * A_h + j];
      z.x = fmaf(xj, w.x, z.x);
      z.y = fmaf(xj, w.y, z.y);
      z.z = fmaf(xj, w.z, z.z);
      z.w = fmaf(xj, w.w, z.w);
    }
    if (jh == 1 && on) *reinterpret_cast<float4*>(zp + c) = z;
    named_sync(4, 256);
    if (jh == 0 && on) {
      const float4 z1 = *reinterpret_cast<const float4*>(zp + c);
      const float e0 = silu(z.x + z1.x + tv.x), e1 = silu(z.y + z1.y + tv.y);
      const float e2 = silu(z.z + z1.z + tv.z), e3 = silu(z.w + z1.w + tv.w);
      if (!(fmaxf(fmaxf(fabsf(e0), fabsf(e1)), fmaxf(fabsf(e2), fabsf(e3))) < kF16Max))
        mk_range_error(a.err, 35);
      uint32_t h0, l0, h1, l1;
      split_pair_h2(e0, e1, h0, l0);
      split_pair_h2(e2, e3, h1, l1);
      *reinterpret_cast<uint2*>(ehi + n) = make_uint2(h0, h1);
      *reinterpret_cast<uint2*>(elo + n) = make_uint2(l0, l1);
      *reinterpret_cast<float4*>(hrow + n) = bv;
    }
    named_sync(4, 256);   // zp is reused by the next columns
  }
  // the scratch (generic writes) is next written by peers' bulk copies
  fence_proxy_async_smem();
  mk_mark(tr, 5);
}

// Chunk mode, after the last block's down projection of a step: the CTAs of
// the action rows copy W_out (bf16 [D][A]) whole into their operand slots,
// which no projection uses until W2 of the next step, so that the head after
// the grid barrier reads it from shared memory.
__device__ __forceinline__ void mk_head_prefetch(const MkArgs& a, uint8_t* sB, uint64_t* hfull, int mt) {
  if ((int)blockIdx.x >= 2 * (a.T_q - 1)) return;
  named_sync(4, 256);   // every math warp is past its reads of the slots
  if (mt == 0) {
    fence_proxy_async_smem();
    const uint32_t bytes = (uint32_t)(a.D * a.A * 2);
    mbar_arrive_expect_tx(hfull, bytes);
    bulk_copy_g2s(smem_u32(sB), a.w_out, bytes, smem_u32(hfull));
  }
}

template <int DH, bool CHUNK>
__global__ void __launch_bounds__(kMkThreads, 1)
    pi0_step_kernel(const __grid_constant__ CUtensorMap w_qkv, const __grid_constant__ CUtensorMap w_o,
                    const __grid_constant__ CUtensorMap w_gu, const __grid_constant__ CUtensorMap w_d,
                    const __grid_constant__ CUtensorMap act_op, const __grid_constant__ CUtensorMap act_hp,
                    const __grid_constant__ CUtensorMap w_w2, const __grid_constant__ CUtensorMap act_ep,
                    const MkArgs a) {
  // the CTAs exchange partial sums with the other CTAs of their cluster of 4:
  // launched any other way (a replay by a tool that drops the cluster shape)
  // every CTA records the error and returns before any barrier, TMEM or
  // distributed shared-memory access
  if (cluster_size() != (uint32_t)kMkCluster || gridDim.x % kMkCluster != 0) {
    if (threadIdx.x == 0) record_error(a.err, kErrLaunch, 950);
    return;
  }
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
  uint64_t* xfull = go + 1;                // cluster exchange received (bytes, armed by this CTA)
  uint64_t* never = xfull + 1;             // nothing arrives (failure hook)
  uint64_t* hfull = never + 1;             // the head's weight landed (chunk mode)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(hfull + 1);
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
    mbar_init(xfull, 1);
    mbar_init(never, 1);
    mbar_init(hfull, 1);
    fence_mbar_init();
    // armed with the bytes of this CTA's first exchange before any peer can
    // send (the cluster barrier below)
    const uint32_t nb = mk_first_xbytes(a, (int)blockIdx.x / kMkCluster);
    if (nb) mbar_arrive_expect_tx(xfull, nb);
    mk_xtable(a, (int)blockIdx.x / kMkCluster, tmem_slot + 1);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the cluster's barriers are initialised before any CTA of it arrives on a
  // peer's barrier or stores into a peer's exchange area
  cluster_sync_all();

  // register split of the launch's 384 x 168 = 64512 registers: the four
  // producer warps keep 40 each (128 x 40 = 5120), the eight math warps take
  // 232 (256 x 232 = 59392); 5120 + 59392 = 64512
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 40;");
    if (warp == 0 && lane == 0) {
      // ---------------- weight stream ----------------
      tma_prefetch_desc(&w_qkv);
      tma_prefetch_desc(&w_o);
      tma_prefetch_desc(&w_gu);
      tma_prefetch_desc(&w_d);
      if (a.steps > 0) tma_prefetch_desc(&w_w2);
      const uint64_t pol = l2_policy_evict_first();
      uint32_t wt = 0;
      bool ok = true;
      for (MkPos ps = mk_seq_first(a); ps.valid && ok; mk_seq_next(a, ps)) {
          const int gi = ps.gi;
          const MkRange r = mk_range(a.g[gi], blockIdx.x);
          if (!r.active) continue;
          const CUtensorMap* map = gi == 0 ? &w_qkv : gi == 1 ? &w_o : gi == 2 ? &w_gu : gi == 3 ? &w_d : &w_w2;
          const int row = (gi == 4 ? 0 : ps.l * a.g[gi].N) + r.m * 128;
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
      const uint32_t idesc = idesc_f16_f32(128, 128);   // M = 128 weight rows, N = 2 fp16 planes x 64 tokens
      uint32_t wt = 0, bt = 0, gc = 0, pf = 0, pt = 0;   // pf / pt: per-slot parities of bfull / bfullt
      bool ok = true;
      for (MkPos ps = mk_seq_first(a); ps.valid && ok; mk_seq_next(a, ps)) {
          const int gi = ps.gi;
          const MkRange r = mk_range(a.g[gi], blockIdx.x);
          if (!r.active) continue;
          const uint32_t acc = tmem + (gc & 1) * 256;
          for (int k = r.k0; k < r.k1; ++k) {
            const uint32_t b = bt % kMkNB, s = wt % kMkNW;
            const bool tma_b = gi == 1 || gi == 3 || gi == 4;
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
      // after each grid barrier that opens the output, the down or the W2
      // projection: the operand planes straight into the operand slots (the
      // math warps build the QKV and gate/up operands from x themselves)
      tma_prefetch_desc(&act_op);
      tma_prefetch_desc(&act_hp);
      if (a.steps > 0) tma_prefetch_desc(&act_ep);
      const uint64_t pol = l2_policy_evict_last();
      uint32_t bt = 0, gop = 0;
      uint32_t bout = 0;            // operand copies issued, by slot (bit)
      uint32_t pt = 0;              // per-slot parity of bfullt
      bool ok = true;
      for (MkPos ps = mk_seq_first(a); ps.valid && ok; mk_seq_next(a, ps)) {
          const int gi = ps.gi;
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
          if (gi == 1 || gi == 3 || gi == 4) {   // operand planes straight into the operand slots
            const CUtensorMap* map = gi == 1 ? &act_op : gi == 3 ? &act_hp : &act_ep;
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
    asm volatile("setmaxnreg.inc.sync.aligned.u32 232;");
    // ---------------- math warps ----------------
    MkMath s;
    s.base = smem;
    s.xbroken = false;
    s.tmem = tmem;
    s.bt = s.gc = s.xuse = 0;
    s.mt = threadIdx.x - 128;
    const int mt = s.mt;
    const unsigned G = gridDim.x;
    unsigned nbar = 0;
    const float invD = 1.f / (float)a.D;
    const int kvd = a.Hkv * DH;
    constexpr bool chunk = CHUNK;   // a whole chunk (a.steps > 0) or the blocks once
    const int cl = (int)blockIdx.x / kMkCluster, rk = (int)blockIdx.x % kMkCluster;
    for (int st = 0; st < (chunk ? a.steps : 1); ++st) {
      if constexpr (chunk) {
        // before the first block of each step, after a grid barrier (none
        // before the launch's first phase): the head of the previous step and
        // the embedding (trace slots 42, 43, sub-steps 52..), then W2 (44..49)
        unsigned long long* tr0 = (a.trace && mt == 0) ? a.trace + (size_t)blockIdx.x * 64 : nullptr;
        if (st > 0) {
          ++nbar;
          mk_grid_sync(a.bar, nbar * G, a.err, mt);
        }
        mk_mark(tr0, 42);
        mk_head_embed(a, st, st > 0, true, s.sB(), s.hfull(), mt, tr0 ? tr0 + 52 : nullptr);
        mk_mark(tr0, 43);
        ++nbar;
        mk_grid_sync(a.bar, nbar * G + ((nbar == 1 && a.skew_where == 1) ? a.skew : 0u), a.err, mt);
        if (mt == 0) mbar_arrive(s.go());   // the loader may fetch the embedding planes
        mk_mark(tr0, 44);
        mk_gemm_math<kMkPre>(s, a.g[4], nullptr, a.D, false, a.wsc[4], a.x, a.D, a.T_q, a.err,
                             tr0 ? tr0 + 45 : nullptr);
        mk_mark(tr0, 49);
      }
      for (int l = a.l0; l < a.l1; ++l) {
        __nv_bfloat16* kc = a.kv + (size_t)(l - a.l0) * a.kv_stride;
        __nv_bfloat16* vc = kc + (size_t)a.T_kv * kvd;
        unsigned long long* tr =
            (a.trace && mt == 0) ? a.trace + ((size_t)(l - a.l0) * a.trace_stride + blockIdx.x) * 64 : nullptr;
        mk_mark(tr, 0);
        // phases: 0 QKV (+ q / own k, v), 2 attention, 3 combine, 4 O, 5 gate/up
        // (+ GeGLU planes), 7 down; a grid barrier before each (the first one of
        // a launch has none).  Indices 1 and 6 (former separate finalize phases)
        // are skipped so trace slots keep their meaning.
        for (int ph = 0; ph < 8; ++ph) {
          if (ph == 1 || ph == 6) continue;   // finalized inside the QKV and gate/up phases
          if (ph > 0 || l > a.l0 || chunk) {
            ++nbar;
            const unsigned extra = (nbar == 1 && a.skew_where == 1) ? a.skew : 0u;
            mk_grid_sync(a.bar, nbar * G + extra, a.err, mt);
          }
          const bool proj = ph == 0 || ph == 4 || ph == 5 || ph == 7;
          if (proj && mt == 0) mbar_arrive(s.go());   // the loader may fetch this phase's operand
          mk_mark(tr, 2 * ph + 1);
          if (ph == 2) {
            mk_attention<DH>(a, kc, vc, s.sB(), mt, tr);
          } else if (ph == 3) {
            mk_combine<DH>(a, mt, reinterpret_cast<float*>(s.sB()), tr);
          } else {
            const int gi = ph == 0 ? 0 : ph == 4 ? 1 : ph == 5 ? 2 : 3;
            const MkGemm& g = a.g[gi];
            const MkRange r = mk_range(g, blockIdx.x);
            mk_gemm_math<kMkPre>(s, g, ph == 0 || ph == 5 ? a.x : nullptr, a.D, ph == 0 || ph == 5, a.wsc[gi], a.x,
                                 a.D, a.T_q, a.err, tr ? tr + 20 + 4 * gi : nullptr);
            if (r.active && !g.direct) {   // QKV and gate/up: the whole cluster is active or idle
              const bool skew = a.skew > 0 && st == 0 && l == a.l0 &&
                                ((a.skew_where == 2 && ph == 0) || (a.skew_where == 3 && ph == 5));
              MkRot rot;
              if (ph == 0) rot = mk_qkv_angles<DH>(a, cl, rk, mt);
              mk_exchange_wait(s, a, gi, skew, 903 + gi);
              mk_mark(tr, 38 + gi);   // exchange received
              if (ph == 0) mk_qkv_finalize<DH>(a, cl, rk, s.xbuf(), s.xss(), kc, vc, invD, rot, mt);
              else mk_gu_finalize(a, r.m, rk & 1, s.xbuf(), s.xss(), invD, mt);
            }
          }
          if (chunk && ph == 7 && l == a.l1 - 1) mk_head_prefetch(a, s.sB(), s.hfull(), mt);
          mk_mark(tr, 2 * ph + 2);
        }
      }
    }
    if constexpr (chunk) {   // the last step's head
      unsigned long long* trl =
          (a.trace && mt == 0) ? a.trace + ((size_t)(a.l1 - 1 - a.l0) * a.trace_stride + blockIdx.x) * 64 : nullptr;
      ++nbar;
      mk_grid_sync(a.bar, nbar * G, a.err, mt);
      mk_mark(trl, 50);
      mk_head_embed(a, a.steps, true, false, s.sB(), s.hfull(), mt, trl ? trl + 52 : nullptr);
      mk_mark(trl, 51);
    }
  }
  tc_fence_before();
  __syncthreads();
  // no CTA leaves while a peer of its cluster may still store into it
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace lat
