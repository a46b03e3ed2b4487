// Dense GEMM on tcgen05 for many tokens (prefix prefill, batched DiT chunks):
//
//   acc[m][n] = sum_k A[m][k] W[n][k]
//
// A is an activation stored as `terms` 16-bit planes side by side
// ([M][terms*K]): for the block projections two fp16 planes (hi, lo: 22
// significant bits of the fp32 value) against the weight held as fp16 =
// 2^s W (exact), for the patch embedding one plain bf16 plane; the K loop runs
// over terms*K and reuses the weight tile of column k mod K for every plane.
// Products are exact on the tensor cores and accumulate in fp32 in TMEM.
//
// Tile 128 (tokens) x 256 (features) x 64, both operands moved by TMA with a
// 128-byte swizzle through STAGES slots; a slot holds one weight tile and the
// `terms` activation tiles of the same K range, so each weight tile crosses
// from L2 once.  One tcgen05.mma (M=128, N=256, K=16) per 16-wide K step and
// plane: on this hardware an M=128 MMA takes the same ~152 cycles for N = 64,
// 128 or 256, so only N = 256 runs the tensor core at its rate.  Warp 0 issues
// TMA, warp 1 MMAs, warps 4..11 accumulate and run the fused epilogue (bias,
// residual, per-chunk gate, GELU / GeGLU followed by the split of the next
// GEMM's activation).
//
// Accumulation in two levels: the tensor core sums one chunk of at most 32
// (or 64) MMAs into a TMEM accumulator; the epilogue warps add each finished
// chunk into fp32 registers (round to nearest) while the tensor core fills the
// other TMEM accumulator.  Measured on this hardware, an fp32 TMEM accumulator
// run over thousands of MMAs drifts by about one unit of its last place per
// MMA in one direction (K = 13824 x 2 terms gave 2e-4 relative error); chunks
// of 32 MMAs bound that drift to ~4e-6, chunks of 64 to ~8e-6.  The chunk
// length also sets how far the tensor core runs into the next tile (two
// accumulators of one chunk each) while the epilogue warps finish the last
// one: the DiT block's QKV and FFN-in projections take chunks of 64, so that
// their MMAs do not wait on the longer epilogues (RoPE and the cache stores,
// GELU and the plane split).  The residual projections (short epilogues, the
// longest K) and the prefix prefill (whose K/V error compounds over its 18
// blocks) keep chunks of 32.
#pragma once
#include "common.cuh"

namespace lat {

enum DenseEpi : int {
  E_STORE = 0,        // out[m][n] = acc (+ bias[n])
  E_RESID = 1,        // out[m][n] += acc
  E_RESID_GATE = 2,   // out[m][n] += gate[chunk(m)][n] * acc
  E_GELU_SPLIT = 3,   // act planes <- split of GELU_tanh(acc)
  E_GEGLU_SPLIT = 4,  // tile = [64 gate | 64 up] -> act planes <- split of GELU(g) * u
  E_ROPE_KV = 5,      // [q | k | v] heads of 128: rotary on q and k; q -> fp32, k and v -> ring + fp16 planes
};

constexpr int kMaxChunks = 16;
constexpr int kChunkMMA = 32;       // MMAs (of K = 16) per TMEM accumulation chunk, at most (default)
constexpr int kChunkMMALong = 64;   // the same for the DiT QKV and FFN-in projections

// The K / V ring rows of the chunks of a call: chunk b's token j is row j of
// kdst[b] / vdst[b] (rows ld elements apart), or with page_tokens > 0 ring row
// row0[b] + j, which lives in page ptab[b][row / page_tokens] of the pool
// [pages][2][page_tokens][ld] (plane 0 K, 1 V) at row % page_tokens.
struct RingRows {
  __nv_bfloat16* kdst[kMaxChunks];
  __nv_bfloat16* vdst[kMaxChunks];
  int ld;
  int page_tokens;
  const int* ptab[kMaxChunks];
  int row0[kMaxChunks];
  __nv_bfloat16* pool;
};

__device__ __forceinline__ __nv_bfloat16* ring_row(const RingRows& g, int b, int j, int plane) {
  if (g.page_tokens > 0) {
    const int r = g.row0[b] + j, P = g.page_tokens;
    return g.pool + ((size_t)g.ptab[b][r / P] * 2 * P + (size_t)plane * P + r % P) * g.ld;
  }
  return (plane ? g.vdst[b] : g.kdst[b]) + (size_t)j * g.ld;
}

// E_ROPE_KV: the QKV projection of a DiT block (dh = 128, as many k and v
// heads as q heads).  Output column n is part n / D (q, k, v) of head
// (n % D) / 128; row m is token m % T of chunk m / T.  Pair (i, i + 64) of a
// q or k head turns by the row's rotation rot (rope_rows_kernel: the chunk's
// base position composed with the token's angles).
struct RopeEpi {
  const float4* rot;   // per 32-row group g: [2][16][32] float4, (cos | sin) of pairs 4i .. 4i + 3 of row 32 g + r
  int heads;           // heads per part (D = 128 heads)
  int T;
  float* q_out;        // fp32 [M][D]
  __half* own16;       // [M][4 D]: K hi | K lo | V hi | V lo (fp16 planes of the values as computed)
  RingRows ring;       // the bf16 K / V rows of the cache
};

struct DenseArgs {
  int M, N, K;           // K = reduction length of one term
  int terms;             // planes in A (1..PLANES)
  int f16;               // operands fp16 (activation planes, scaled fp16 weights) instead of bf16
  float out_scale;       // acc *= out_scale before the epilogue (2^-s of weights held as 2^s W)
  int w_row0;            // first weight row of this matrix in the stacked tensor
  int epi;
  int chunk_mma;         // MMAs per TMEM accumulation chunk: kChunkMMA or kChunkMMALong
  int ksplit;            // K ranges per output tile (> 1 only for E_STORE (out zeroed before, the
                         // first range adds the bias), E_RESID and E_RESID_GATE: each range adds
                         // its partial product into out with vector reductions)
  float* out;            // fp32 [M][ldo] (E_STORE / E_RESID / E_RESID_GATE)
  int ldo;
  const float* bias;     // E_STORE: fp32 [N] or null
  // E_RESID_GATE: gate row of chunk b = gate + gate_off[b]; chunk(m) = m / rows_per_chunk
  const float* gate;
  int gate_off[kMaxChunks];
  int rows_per_chunk;
  // E_*_SPLIT: fp16 planes [M][kActTerms * ldh] (hi of column c at c, lo at ldh + c)
  __half* act2;
  int ldh;
  RopeEpi rope;          // E_ROPE_KV
  DevErr* err;
};

// Tile order: groups of `group` m-tiles, m fastest within a group and the
// group's n-tiles in turn.  A wave of CTAs then covers a block of about
// `group` m-tiles x (grid / group) n-tiles: each weight tile crosses from HBM
// once per group (its readers run together) and the group's activation rows
// stay in L2 while the group sweeps the n-tiles.  With at most kDGroupAll
// m-tiles (activation planes of ~42 MB) one group takes them all, so every
// weight tile crosses from HBM once; more m-tiles go in groups of kDGroupM.
constexpr int kDGroupM = 8;
constexpr int kDGroupAll = 16;
__device__ __forceinline__ void dense_tile(int t, int m_tiles, int n_tiles, int& tm, int& tn) {
  const int group = m_tiles <= kDGroupAll ? m_tiles : kDGroupM;
  const int grp = t / (group * n_tiles);
  const int m0 = grp * group, gm = min(group, m_tiles - m0);
  const int r = t - grp * group * n_tiles;
  tm = m0 + r % gm;
  tn = r / gm;
}

constexpr int kDA = 128 * 64 * 2;   // A tile bytes (one plane, 128 tokens x 64)
constexpr int kDB = 256 * 64 * 2;   // B tile bytes (256 weight rows x 64)
// one pipeline slot: up to PLANES activation tiles + one weight tile
__host__ __device__ constexpr int dense_slot_bytes(int planes) { return planes * kDA + kDB; }

// Epilogue: eight warps; warp 4 + e reads TMEM lanes 32 (e % 4) .. + 31 (the
// rows of its quadrant) and columns 128 (e / 4) .. + 127 of the 256-wide
// accumulator (E_ROPE_KV: pairs 32 (e / 4) .. + 31 of the tile's two heads,
// see rope_rot_load).  Each passes its 32 rows x 128 columns through a 4 KB buffer
// [32 rows][8 float4] in four 32-column quarters, float4 chunk c of row r at
// position c ^ (r & 7) (conflict-free both for a lane writing its own row and
// for 8 lanes reading one row), so that global reads and writes run along rows
// (a lane holding a whole row would touch 32 rows per warp access).
constexpr int kDEpiWarps = 8;
constexpr int kDThreads = 128 + 32 * kDEpiWarps;        // warpgroup 0: TMA, MMA; 1-2: epilogue
constexpr int kDStageBytes = kDEpiWarps * 32 * 32 * 4;   // 32 KB
// registers per thread after setmaxnreg: producer warpgroup / epilogue warpgroups
// (128 x 56 + 256 x 224 = 64512 = 384 x 168, the registers given at launch)
constexpr int kDRegsProd = 56, kDRegsEpi = 224;

__host__ __device__ constexpr int dense_smem_bytes(int stages, int planes) {
  return 1024 + stages * dense_slot_bytes(planes) + kDStageBytes + 8 * (2 * stages + 4) + 16;
}

__device__ __forceinline__ void stage_put(float4* st, int lane, const float* v, float scale) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    st[lane * 8 + (c ^ (lane & 7))] =
        make_float4(v[4 * c] * scale, v[4 * c + 1] * scale, v[4 * c + 2] * scale, v[4 * c + 3] * scale);
}

// One staged 32-column quarter of the warp's rows row0 .. row0 + 31: output
// columns n0 .. n0 + 31 (feature columns of the split planes for the
// E_*_SPLIT epilogues).  Lane l takes float4 chunk l & 7 of rows 4i + (l >> 3);
// the loads of 8 rows are issued before their stores.
__device__ __forceinline__ void epi_quarter(const DenseArgs& a, const float4* st, int row0, int n0, int lane,
                                            bool first_range) {
  const int c = lane & 7, rsub = lane >> 3;
  const int col = n0 + 4 * c;
  float4 bias = make_float4(0.f, 0.f, 0.f, 0.f);
  if (a.epi == E_STORE && a.bias && first_range) bias = *reinterpret_cast<const float4*>(a.bias + col);
#pragma unroll 1
  for (int i0 = 0; i0 < 32; i0 += 8) {
    float4 x[2], g[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int row = row0 + i0 + 4 * u + rsub;
      x[u] = g[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row < a.M && (a.epi == E_RESID || a.epi == E_RESID_GATE) && a.ksplit == 1)
        x[u] = *reinterpret_cast<const float4*>(a.out + (size_t)row * a.ldo + col);
      if (row < a.M && a.epi == E_RESID_GATE)
        g[u] = *reinterpret_cast<const float4*>(a.gate + a.gate_off[row / a.rows_per_chunk] + col);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r0 = i0 + 4 * u + rsub, row = row0 + r0;
      if (row >= a.M) continue;
      float4 r = st[r0 * 8 + (c ^ (r0 & 7))];
      if (a.epi == E_GELU_SPLIT || a.epi == E_GEGLU_SPLIT) {
        if (a.epi == E_GELU_SPLIT) {
          r.x = gelu_tanh(r.x); r.y = gelu_tanh(r.y); r.z = gelu_tanh(r.z); r.w = gelu_tanh(r.w);
        }
        uint2 hv, lv;
        split_pair_h2(r.x, r.y, hv.x, lv.x);
        split_pair_h2(r.z, r.w, hv.y, lv.y);
        __half* hp = a.act2 + (size_t)row * kActTerms * a.ldh + col;
        *reinterpret_cast<uint2*>(hp) = hv;
        *reinterpret_cast<uint2*>(hp + a.ldh) = lv;
        continue;
      }
      if (a.ksplit > 1) {   // one K range of several: add the partial product
        if (a.epi == E_RESID_GATE) {
          r.x *= g[u].x; r.y *= g[u].y; r.z *= g[u].z; r.w *= g[u].w;
        } else if (a.epi == E_STORE) {
          r.x += bias.x; r.y += bias.y; r.z += bias.z; r.w += bias.w;
        }
        red_add_v4(a.out + (size_t)row * a.ldo + col, r.x, r.y, r.z, r.w);
        continue;
      }
      if (a.epi == E_STORE) {
        r.x += bias.x; r.y += bias.y; r.z += bias.z; r.w += bias.w;
      } else if (a.epi == E_RESID_GATE) {
        r.x = x[u].x + g[u].x * r.x; r.y = x[u].y + g[u].y * r.y;
        r.z = x[u].z + g[u].z * r.z; r.w = x[u].w + g[u].w * r.w;
      } else {
        r.x += x[u].x; r.y += x[u].y; r.z += x[u].z; r.w += x[u].w;
      }
      *reinterpret_cast<float4*>(a.out + (size_t)row * a.ldo + col) = r;
    }
  }
}

// One staged 32-column quarter (columns col0 .. col0 + 31 of part `part`) of
// the E_ROPE_KV epilogue: q rows as fp32, k / v rows as bf16 into the ring and
// as two fp16 planes.  Lane l takes float4 chunk l & 7 of rows 4i + (l >> 3).
__device__ __forceinline__ void rope_quarter(const DenseArgs& a, const float4* st, int row0, int part, int col0,
                                             int lane, int b0) {
  const RopeEpi& r = a.rope;
  const int c = lane & 7, rsub = lane >> 3, col = col0 + 4 * c, D = r.heads * 128;
#pragma unroll 2
  for (int i = 0; i < 32; i += 4) {
    const int r0 = i + rsub, row = row0 + r0;
    if (row >= a.M) continue;
    const float4 v = st[r0 * 8 + (c ^ (r0 & 7))];
    if (part == 0) {
      *reinterpret_cast<float4*>(r.q_out + (size_t)row * D + col) = v;
      continue;
    }
    int b = b0, j = row - b0 * r.T;   // b0 = row0 / T: chunks of at least 32 rows step once at most
    while (j >= r.T) {
      j -= r.T;
      ++b;
    }
    const __nv_bfloat162 x = __floats2bfloat162_rn(v.x, v.y), z = __floats2bfloat162_rn(v.z, v.w);
    *reinterpret_cast<uint2*>(ring_row(r.ring, b, j, part - 1) + col) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&x), *reinterpret_cast<const uint32_t*>(&z));
    uint2 h, l;
    split_pair_h2(v.x, v.y, h.x, l.x);
    split_pair_h2(v.z, v.w, h.y, l.y);
    __half* p = r.own16 + (size_t)row * 4 * D + (size_t)(part - 1) * 2 * D + col;
    *reinterpret_cast<uint2*>(p) = h;
    *reinterpret_cast<uint2*>(p + D) = l;
  }
}

// E_ROPE_KV: the 256 columns of a tile are two heads of one part (q, k or
// v); epilogue warp hc takes pairs 32 hc .. 32 hc + 31 of both, so lane l
// holds acc[32 k + t] = tile column 32 hc + 64 k + t of row row0 + l (k = 0, 1:
// the pair's first and second members in head 0, k = 2, 3 in head 1) and
// needs the rotation of 32 pairs of its row only.  rope_rot_load fetches that
// of 16 pairs (cos and sin of pairs 32 hc + 16 h .. + 15: 8 float4, coalesced
// over the warp's 32 rows); the first half is issued before the last
// accumulation chunk lands, so that its L2 latency overlaps the MMAs.
__device__ __forceinline__ void rope_rot_load(const DenseArgs& a, int row0, int hc, int h, int lane,
                                              float4 (&rv)[8]) {
  const float4* rc = a.rope.rot + (size_t)(row0 >> 5) * 1024 + (hc * 8 + h * 4) * 32 + lane;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    rv[u] = __ldg(rc + u * 32);            // cos of pairs 32 hc + 16 h + 4u .. + 3
    rv[4 + u] = __ldg(rc + 512 + u * 32);  // sin
  }
}

// Turn pairs t = 16 h .. 16 h + 15 (of the warp's 32) of both heads by rv,
// the weight scale sc folded into cos and sin (a power of two: exact).
__device__ __forceinline__ void rope_turn(float (&acc)[128], const float4 (&rv)[8], int h, float sc) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float cc[4] = {rv[u].x * sc, rv[u].y * sc, rv[u].z * sc, rv[u].w * sc};
    const float ss[4] = {rv[4 + u].x * sc, rv[4 + u].y * sc, rv[4 + u].z * sc, rv[4 + u].w * sc};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int t = 64 * g + 16 * h + 4 * u + e;
        const float x0 = acc[t], x1 = acc[32 + t];
        acc[t] = x0 * cc[e] - x1 * ss[e];
        acc[32 + t] = x1 * cc[e] + x0 * ss[e];
      }
    }
  }
}

// E_ROPE_KV epilogue of one tile for the warp's 32 rows (layout above): q and
// k heads turn each pair by the row's rotation (rv0: pairs 0 .. 15 of the
// warp's, loaded during the last chunk), then every quarter passes through
// the staging buffer to its stores.
__device__ __forceinline__ void rope_epilogue(const DenseArgs& a, float (&acc)[128], int row0, int n0, float4* st,
                                              int lane, const float4 (&rv0)[8]) {
  const RopeEpi& r = a.rope;
  const int D = r.heads * 128, hc = (n0 >> 7) & 1, t0 = n0 - hc * 128;
  const int part = t0 / D, col0 = t0 - part * D + hc * 32, b0 = row0 / r.T;
  float sc = a.out_scale;
  if (part < 2 && row0 < a.M) {   // warp-uniform: a warp wholly past M stores nothing
    rope_turn(acc, rv0, 0, sc);
    float4 rv1[8];
    rope_rot_load(a, row0, hc, 1, lane, rv1);
    rope_turn(acc, rv1, 1, sc);
    sc = 1.f;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    stage_put(st, lane, acc + 32 * k, sc);
    __syncwarp();
    rope_quarter(a, st, row0, part, col0 + (k >> 1) * 128 + (k & 1) * 64, lane, b0);
    __syncwarp();
  }
}

// Epilogue of one tile for the warp's 32 rows (lane l holds the 128
// accumulated columns of row row0 + l): output columns n0 .. n0 + 127, or for
// the gate/up tile of E_GEGLU_SPLIT ([64 gate | 64 up] of features f0 ..
// f0 + 63) those features.  The accumulators are scaled by a.out_scale (a
// power of two: exact) on the way.  All lanes take part.
__device__ __forceinline__ void dense_epilogue(const DenseArgs& a, float (&acc)[128], int row0, int n0, int f0,
                                               float4* st, int lane, bool first_range) {
  if (a.epi == E_GEGLU_SPLIT) {
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = gelu_tanh(acc[j] * a.out_scale) * (acc[64 + j] * a.out_scale);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      stage_put(st, lane, acc + 32 * q, 1.f);
      __syncwarp();
      epi_quarter(a, st, row0, f0 + 32 * q, lane, true);
      __syncwarp();
    }
    return;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    stage_put(st, lane, acc + 32 * q, a.out_scale);
    __syncwarp();
    epi_quarter(a, st, row0, n0 + 32 * q, lane, first_range);
    __syncwarp();
  }
}

// ROPE: the E_ROPE_KV instantiation (its own column assignment and epilogue;
// the other epilogues run in the instantiation without them).
template <int STAGES, int PLANES, bool ROPE>
__global__ void __launch_bounds__(kDThreads, 1) dense_gemm_kernel(const __grid_constant__ CUtensorMap amap,
                                                                  const __grid_constant__ CUtensorMap wmap,
                                                                  const __grid_constant__ DenseArgs a) {
  constexpr int kSlot = dense_slot_bytes(PLANES);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float4* stage = reinterpret_cast<float4*>(smem + STAGES * kSlot);   // epilogue staging, 4 KB per warp
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * kSlot + kDStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;       // [2]
  uint64_t* acc_empty = bars + 2 * STAGES + 2;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = a.N / 256, m_tiles = (a.M + 127) / 128, mn = m_tiles * n_tiles;
  const int tiles = mn * a.ksplit;                            // tile t: K range t / mn of output tile t % mn
  const int nkb = a.K / 64;                                   // K-blocks of one plane
  const int chunk_kb = a.chunk_mma / (4 * a.terms);           // K-blocks per accumulation chunk
  // K-blocks [kb0, kb1) of tile t and their accumulation chunks
  auto krange = [&](int t, int& kb0, int& kb1) {
    const int ks = t / mn;
    kb0 = ks * nkb / a.ksplit;
    kb1 = (ks + 1) * nkb / a.ksplit;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&acc_full[0], 1);
    mbar_init(&acc_full[1], 1);
    mbar_init(&acc_empty[0], 32 * kDEpiWarps);
    mbar_init(&acc_empty[1], 32 * kDEpiWarps);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);   // two 256-column accumulators
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // persistent: CTA b takes tiles b, b + grid, ...; the slot ring and the two
  // accumulators carry on across tiles, so a tile's epilogue overlaps the next
  // tile's MMAs (counters it / gch run over all tiles of the CTA)
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kDRegsProd));
    if (warp == 0 && lane == 0) {
      tma_prefetch_desc(&amap);
      tma_prefetch_desc(&wmap);
      const uint64_t pol_w = l2_policy_evict_last();   // weight tiles are re-read by every m-tile
      const uint64_t pol_a = l2_policy_evict_first();
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        int tm, tn;
        dense_tile(tile % mn, m_tiles, n_tiles, tm, tn);
        int kb0, kb1;
        krange(tile, kb0, kb1);
        for (int i = kb0; i < kb1; ++i, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, a.err, 20)) { ok = false; break; }
          uint8_t* slot = smem + s * kSlot;
          mbar_arrive_expect_tx(&full[s], a.terms * kDA + kDB);
          for (int t = 0; t < a.terms; ++t)
            tma_load_2d(slot + t * kDA, &amap, &full[s], t * a.K + i * 64, tm * 128, pol_a);
          // the weight tile's 256 rows in two 128-row boxes (contiguous in the swizzled layout)
          tma_load_2d(slot + PLANES * kDA, &wmap, &full[s], i * 64, a.w_row0 + tn * 256, pol_w);
          tma_load_2d(slot + PLANES * kDA + kDB / 2, &wmap, &full[s], i * 64, a.w_row0 + tn * 256 + 128, pol_w);
        }
      }
      for (uint32_t i = (it > (uint32_t)STAGES ? it - STAGES : 0); i < it; ++i)
        mbar_wait(&full[i % STAGES], (i / STAGES) & 1, a.err, 21);
    } else if (warp == 1 && lane == 0) {
      const uint32_t idesc = a.f16 ? idesc_f16_f32(128, 256) : idesc_bf16_f32(128, 256);
      bool ok = true;
      uint32_t it = 0, gch = 0;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        int kb0, kb1;
        krange(tile, kb0, kb1);
        const int nchunk = (kb1 - kb0 + chunk_kb - 1) / chunk_kb;
        for (int ch = 0; ch < nchunk && ok; ++ch, ++gch) {
          const int buf = gch & 1;
          // the epilogue has drained this accumulator (use gch - 2)
          if (!mbar_wait(&acc_empty[buf], ((gch >> 1) & 1) ^ 1, a.err, 24)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(buf * 256);
          const int i0 = kb0 + ch * chunk_kb, i1 = min(kb1, i0 + chunk_kb);
          for (int i = i0; i < i1; ++i, ++it) {
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            if (!mbar_wait(&full[s], ph, a.err, 22)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + s * kSlot), bb = sa + PLANES * kDA;
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
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kDRegsEpi));
    const int ew = warp - 4;
    const int quad = warp & 3, hc = ew >> 2;   // TMEM lane quadrant, column half
    constexpr bool rope = ROPE;
    float4* st = stage + ew * 32 * 8;
    uint32_t gch = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
      int tm, tn;
      dense_tile(tile % mn, m_tiles, n_tiles, tm, tn);
      int kb0, kb1;
      krange(tile, kb0, kb1);
      const int nchunk = (kb1 - kb0 + chunk_kb - 1) / chunk_kb;
      const int row0 = tm * 128 + quad * 32;
      float acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.f;
      // the warp's 128 accumulator columns: 16-column pieces c at col(c) =
      // base + (c / 2) pstride + (c % 2) 16 (E_ROPE_KV: pairs 32 hc .. of both heads)
      const int cbase = rope ? hc * 32 : hc * 128;
      constexpr int pstride = rope ? 64 : 32;
      float4 rv[8];   // E_ROPE_KV: the rotation of the first 16 pairs
      for (int ch = 0; ch < nchunk; ++ch, ++gch) {
        const int buf = gch & 1;
        if constexpr (rope) {
          if (ch == nchunk - 1 && row0 < a.M) rope_rot_load(a, row0, hc, 0, lane, rv);
        }
        // warp-uniform outcome: the TMEM loads below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (gch >> 1) & 1, a.err, 23))) { ok = false; break; }
        tc_fence_after();
        const uint32_t tb = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * 256 + cbase);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float v[16];
          tmem_ld16(tb + (c >> 1) * pstride + (c & 1) * 16, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[c * 16 + j] += v[j];
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
      }
      if (!ok) break;
      if constexpr (rope) rope_epilogue(a, acc, row0, tn * 256 + hc * 128, st, lane, rv);
      else dense_epilogue(a, acc, row0, tn * 256 + hc * 128, tn * 128 + hc * 64, st, lane, tile < mn);
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
