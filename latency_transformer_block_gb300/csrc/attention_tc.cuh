// Segmented attention on the 5th-generation tensor cores (tcgen05, TMEM) for
// the dense path's MHA with dh = 128 (the DiT stage): a chunk of query rows
// attends to its noisy history segments (bf16 ring slots) and to its own keys
// as computed (fp32, two bf16 planes).  Same inputs, outputs and arithmetic
// as attention_seg_kernel (exact three-term q and P, own keys in two planes,
// online softmax in base 2, fp32 accumulation), with the products on tcgen05:
//
//   S  = sum_t Q_t K^T          M = 128 query rows, N = 64 keys, K = 128 dims
//   O += sum_t P_t V            M = 128 query rows, N = 128 dims, K = 64 keys
//                               (V as an MN-major operand: dims contiguous, as stored)
//
// One CTA = one (head, group, 128-row tile).  Warp 0 (lane 0) issues the MMAs;
// warps 1..3 load each key block (K and V by cp.async into the swizzled layout,
// own keys split into two planes); warps 4..11 hold the rows:
// warp w reads TMEM lanes 32 (w % 4).., half (w - 4) / 4 of the keys of S and
// of the columns of O.  The product of one key block lands in TMEM and is
// added to the running output in fp32 registers, so no TMEM accumulation chain
// is longer than 20 MMAs.
#pragma once
#include "attention.cuh"
#include "common.cuh"
#include "pi0_step.cuh"   // named_sync

namespace lat {

constexpr int kTcThreads = 384;
constexpr int kTcKB = 64;                       // keys per block
constexpr int kTcQT = 16384;                    // one [128 rows][64] bf16 tile
constexpr int kTcKT = 8192;                     // one [64 keys][64] bf16 tile
// shared memory: Q [3 terms][2 k-tiles], K [hi, lo][2 k-tiles], V^T [hi, lo],
// P [3 terms], row exchange, barriers
constexpr int kTcOffQ = 0;
constexpr int kTcOffK = kTcOffQ + 6 * kTcQT;    // 96 KB
constexpr int kTcOffV = kTcOffK + 4 * kTcKT;    // +32 KB
constexpr int kTcOffP = kTcOffV + 2 * kTcQT;    // +32 KB
constexpr int kTcOffX = kTcOffP + 3 * kTcQT;    // +48 KB
constexpr int kTcOffBar = kTcOffX + 4 * 128 * 4;   // exchange: [2 parities][2 halves][128 rows]
constexpr int kTcSmem = 1024 + kTcOffBar + 16 * 8 + 16;

__host__ __device__ constexpr int attn_tc_smem_bytes() { return kTcSmem; }

// Shared-memory descriptor of an MN-major operand with 128-byte swizzle: rows
// of 128 bytes run along N (64 elements), 8 rows (8 consecutive K) form one
// 1024-byte swizzle atom; `lbo` = bytes between atoms adjacent along N (the
// next 64 elements of N), `sbo` = bytes between atoms adjacent along K.
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;   // descriptor version
  d |= (uint64_t)2 << 61;   // SWIZZLE_128B
  return d;
}

// byte offset of element (row r, column c < 64) in a K-major 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)(r * 128 + ((((c >> 3) ^ r) & 7) << 4) + ((c & 7) << 1));
}

// Bounded wait that also returns at once after any recorded error, so a
// failed launch ends quickly instead of every later wait using its budget.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, DevErr* err, unsigned where) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (int i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63) {
      if (*reinterpret_cast<volatile unsigned*>(&err->code) != 0) return false;
      if (clock64() - t0 > kSpinBudget) {
        record_error(err, 1u, where);
        return false;
      }
    }
  }
}

// timestamp of (role, block, event) for CTA (0, 0, 0) when tracing
__device__ __forceinline__ void tc_mark(unsigned long long* tr, int role, int j, int ev) {
  if (tr && j < 32 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    tr[(role * 32 + j) * 8 + ev] = t;
  }
}

// key block j of a group -> (segment, block within the segment)
__device__ __forceinline__ void tc_block(const SegGroup& G, int j, int& si, int& kb) {
  si = 0;
  kb = j;
  while (si < G.nseg - 1) {
    const int nb = (G.seg[si].n + kTcKB - 1) / kTcKB;
    if (kb < nb) break;
    kb -= nb;
    ++si;
  }
}

static __global__ void __launch_bounds__(kTcThreads, 1)
    attention_tc_kernel(const __grid_constant__ SegAttnArgs a, DevErr* err) {
  constexpr int DH = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + kTcOffQ;
  uint8_t* sK = sm + kTcOffK;   // [hi k-tile 0, hi k-tile 1, lo k-tile 0, lo k-tile 1]
  uint8_t* sV = sm + kTcOffV;   // V [hi, lo] x [2 halves of 64 dims][64 keys][64 dims]
  uint8_t* sP = sm + kTcOffP;   // [3 terms][128 rows][64 keys]
  float* sX = reinterpret_cast<float*>(sm + kTcOffX);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kTcOffBar);
  uint64_t* q_full = bar + 0;   // Q planes built (256 arrivals)
  uint64_t* k_full = bar + 1;   // K block loaded (96)
  uint64_t* v_full = bar + 2;   // V block loaded (96)
  uint64_t* k_free = bar + 3;   // S MMAs done with K (commit)
  uint64_t* v_free = bar + 4;   // PV MMAs done with V and P (commit)
  uint64_t* s_full = bar + 5;   // S in TMEM (commit)
  uint64_t* s_free = bar + 6;   // S read by the row warps (256)
  uint64_t* p_full = bar + 7;   // P written, previous O read (256)
  uint64_t* o_full = bar + 8;   // O of the block in TMEM (commit)
  uint64_t* mdone = bar + 9;    // every MMA complete (teardown)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 10);

  const int h = blockIdx.x, qt = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = h / (a.Hq / a.Hkv);
  const SegGroup& G = a.grp[b];
  int nblk = 0;
  for (int si = 0; si < G.nseg; ++si) nblk += (G.seg[si].n + kTcKB - 1) / kTcKB;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 256);
    mbar_init(k_full, 96);
    mbar_init(v_full, 96);
    mbar_init(k_free, 1);
    mbar_init(v_free, 1);
    mbar_init(s_full, 1);
    mbar_init(s_free, 256);
    mbar_init(p_full, 256);
    mbar_init(o_full, 1);
    mbar_init(mdone, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);   // S at columns [0, 64), O of a block at [128, 256)
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- MMA issue: S(0), then per block PV(j), S(j + 1) ----------------
      const uint32_t idS = idesc_bf16_f32(128, kTcKB), idO = idesc_bf16_f32(128, DH) | (1u << 16);   // B MN-major
      const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK), va = smem_u32(sV), pa = smem_u32(sP);
      bool ok = tc_wait(q_full, 0, err, 60);
      auto issue_s = [&](int j) {
        int si, kb;
        tc_block(G, j, si, kb);
        const bool own = G.seg[si].k32 != nullptr;
        if (!tc_wait(k_full, j & 1, err, 61)) return false;
        tc_mark(a.trace, 0, j, 0);
        if (j > 0 && !tc_wait(s_free, (j - 1) & 1, err, 62)) return false;
        tc_mark(a.trace, 0, j, 1);
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < DH / 16; ++ks) {
          const int kt = ks >> 2;
          const uint32_t off = (uint32_t)((ks & 3) * 32);
#pragma unroll
          for (int t = 0; t < 3; ++t)
            mma_bf16_ss(tmem, desc_k_sw128(qa + (t * 2 + kt) * kTcQT + off), desc_k_sw128(ka + kt * kTcKT + off), idS,
                        (ks | t) != 0 ? 1u : 0u);
          if (own)
#pragma unroll
            for (int t = 0; t < 2; ++t)
              mma_bf16_ss(tmem, desc_k_sw128(qa + (t * 2 + kt) * kTcQT + off),
                          desc_k_sw128(ka + (2 + kt) * kTcKT + off), idS, 1u);
        }
        mma_commit(k_free);
        mma_commit(s_full);
        tc_mark(a.trace, 0, j, 2);
        return true;
      };
      if (ok && nblk > 0) ok = issue_s(0);
      for (int j = 0; j < nblk && ok; ++j) {
        int si, kb;
        tc_block(G, j, si, kb);
        const bool own = G.seg[si].k32 != nullptr;
        if (!tc_wait(p_full, j & 1, err, 63)) {
          ok = false;
          break;
        }
        tc_mark(a.trace, 0, j, 3);
        if (!tc_wait(v_full, j & 1, err, 64)) {
          ok = false;
          break;
        }
        tc_mark(a.trace, 0, j, 4);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTcKB / 16; ++kk) {
          const uint32_t off = (uint32_t)(kk * 32);
          const uint32_t voff = (uint32_t)(kk * 2048);   // 16 keys = two 8-key atoms
#pragma unroll
          for (int t = 0; t < 3; ++t)
            mma_bf16_ss(tmem + 128, desc_k_sw128(pa + t * kTcQT + off), desc_mn_sw128(va + voff, kTcKT, 1024), idO,
                        (kk | t) != 0 ? 1u : 0u);
          if (own)
#pragma unroll
            for (int t = 0; t < 2; ++t)
              mma_bf16_ss(tmem + 128, desc_k_sw128(pa + t * kTcQT + off),
                          desc_mn_sw128(va + kTcQT + voff, kTcKT, 1024), idO, 1u);
        }
        mma_commit(v_free);
        mma_commit(o_full);
        // S of the next block: its K was loaded while the rows ran block j
        if (j + 1 < nblk && !issue_s(j + 1)) {
          ok = false;
          break;
        }
      }
      mma_commit(mdone);
      mbar_wait(mdone, 0, nullptr, 0);
    }
  } else if (warp < 4) {
    // ---------------- loaders: K and V of each key block ----------------
    const int lt = threadIdx.x - 32;
    bool ok = true;
    for (int j = 0; j < nblk && ok; ++j) {
      int si, kb;
      tc_block(G, j, si, kb);
      const AttnSeg sg = G.seg[si];
      const bool own = sg.k32 != nullptr;
      const int k0 = kb * kTcKB;
      if (j > 0 && !tc_wait(k_free, (j - 1) & 1, err, 65)) {
        ok = false;
        break;
      }
      if (lt == 0) tc_mark(a.trace, 2, j, 0);
      fence_proxy_async_smem();
      for (int it = lt; it < kTcKB * (DH / 8); it += 96) {
        const int r = it >> 4, c = it & 15;       // key row, 8-dim chunk
        const int key = k0 + r;
        const bool in = key < sg.n;
        const size_t off = (size_t)(in ? key : 0) * a.kv_ld + kvh * DH + c * 8;
        uint8_t* dst = sK + (c >> 3) * kTcKT + r * 128 + ((((c & 7) ^ r) & 7) << 4);
        if (!own) {
          cp_async16(dst, sg.k + off, in ? 16 : 0);
        } else {
          uint4 hi = make_uint4(0, 0, 0, 0), lo = hi;
          if (in) split8_to(sg.k32 + off, hi, lo);
          *reinterpret_cast<uint4*>(dst) = hi;
          *reinterpret_cast<uint4*>(dst + 2 * kTcKT) = lo;
        }
      }
      cp_async_wait_all();
      fence_proxy_async_smem();
      if (lt == 0) tc_mark(a.trace, 2, j, 1);
      mbar_arrive(k_full);
      if (j > 0 && !tc_wait(v_free, (j - 1) & 1, err, 66)) {
        ok = false;
        break;
      }
      if (lt == 0) tc_mark(a.trace, 2, j, 2);
      fence_proxy_async_smem();
      for (int it = lt; it < kTcKB * (DH / 8); it += 96) {
        const int r = it >> 4, c = it & 15;       // key row, 8-dim chunk
        const int key = k0 + r;
        const bool in = key < sg.n;
        const size_t off = (size_t)(in ? key : 0) * a.kv_ld + kvh * DH + c * 8;
        uint8_t* dst = sV + (c >> 3) * kTcKT + r * 128 + ((((c & 7) ^ r) & 7) << 4);
        if (!own) {
          cp_async16(dst, sg.v + off, in ? 16 : 0);
        } else {
          uint4 hi = make_uint4(0, 0, 0, 0), lo = hi;
          if (in) split8_to(sg.v32 + off, hi, lo);
          *reinterpret_cast<uint4*>(dst) = hi;
          *reinterpret_cast<uint4*>(dst + kTcQT) = lo;
        }
      }
      cp_async_wait_all();
      fence_proxy_async_smem();
      if (lt == 0) tc_mark(a.trace, 2, j, 3);
      mbar_arrive(v_full);
    }
  } else {
    // ---------------- row warps ----------------
    const int st = threadIdx.x - 128;
    const int qd = warp & 3, half = (warp - 4) >> 2;
    const int r = qd * 32 + lane;                    // row of the tile = TMEM lane
    const int rg = qt * 128 + r;                     // row within the group
    // Q planes (exact three-term split) for the tile's 128 rows
    for (int it = st; it < 128 * (DH / 8); it += 256) {
      const int rr = it >> 4, c = it & 15;
      const int rq = qt * 128 + rr;
      uint4 hv = make_uint4(0, 0, 0, 0), mv = hv, lv = hv;
      if (rq < a.T_rows) {
        const float* src = a.q + ((size_t)b * a.T_rows + rq) * a.q_ld + h * DH + c * 8;
        const float4 x0 = *reinterpret_cast<const float4*>(src);
        const float4 x1 = *reinterpret_cast<const float4*>(src + 4);
        split_pair_exact(x0.x, x0.y, hv.x, mv.x, lv.x);
        split_pair_exact(x0.z, x0.w, hv.y, mv.y, lv.y);
        split_pair_exact(x1.x, x1.y, hv.z, mv.z, lv.z);
        split_pair_exact(x1.z, x1.w, hv.w, mv.w, lv.w);
      }
      const uint32_t o = (uint32_t)((c >> 3) * kTcQT + rr * 128 + ((((c & 7) ^ rr) & 7) << 4));
      *reinterpret_cast<uint4*>(sQ + o) = hv;
      *reinterpret_cast<uint4*>(sQ + 2 * kTcQT + o) = mv;
      *reinterpret_cast<uint4*>(sQ + 4 * kTcQT + o) = lv;
    }
    fence_proxy_async_smem();
    mbar_arrive(q_full);

    float o[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) o[i] = 0.f;
    float m = -INFINITY, l = 0.f, alpha_prev = 0.f;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    for (int j = 0; j < nblk; ++j) {
      int si, kb;
      tc_block(G, j, si, kb);
      const int n = G.seg[si].n, k0 = kb * kTcKB;
      tc_wait(s_full, j & 1, err, 67);
      if (st == 0) tc_mark(a.trace, 1, j, 0);
      tc_fence_after();
      float sv[32];
      tmem_ld32(trow + (uint32_t)(half * 32), sv);
      tc_fence_before();
      mbar_arrive(s_free);
      float mloc = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        sv[i] = (k0 + half * 32 + i < n) ? sv[i] * a.scale_log2 : -INFINITY;
        mloc = fmaxf(mloc, sv[i]);
      }
      float* xb = sX + (j & 1) * 256;
      xb[half * 128 + r] = mloc;
      named_sync(4, 256);
      if (st == 0) tc_mark(a.trace, 1, j, 1);
      const float mnew = fmaxf(m, fmaxf(mloc, xb[(half ^ 1) * 128 + r]));
      const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - mnew);
      float lsum = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        sv[i] = exp2f(sv[i] - mnew);
        lsum += sv[i];
      }
      l = l * alpha + lsum;
      m = mnew;
      if (j > 0) {   // O of block j - 1 into the running output (frees P and the O columns)
        tc_wait(o_full, (j - 1) & 1, err, 68);
        if (st == 0) tc_mark(a.trace, 1, j, 2);
        tc_fence_after();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          float t[32];
          tmem_ld32(trow + 128u + (uint32_t)(half * 64 + c2 * 32), t);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[c2 * 32 + i] = o[c2 * 32 + i] * alpha_prev + t[i];
        }
      }
      alpha_prev = alpha;
      // P of this block: exact three-term split, keys half*32 .. +31 of row r
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint4 hv, mv, lv;
        split_pair_exact(sv[8 * c4 + 0], sv[8 * c4 + 1], hv.x, mv.x, lv.x);
        split_pair_exact(sv[8 * c4 + 2], sv[8 * c4 + 3], hv.y, mv.y, lv.y);
        split_pair_exact(sv[8 * c4 + 4], sv[8 * c4 + 5], hv.z, mv.z, lv.z);
        split_pair_exact(sv[8 * c4 + 6], sv[8 * c4 + 7], hv.w, mv.w, lv.w);
        const uint32_t off = (uint32_t)(r * 128 + ((((half * 4 + c4) ^ r) & 7) << 4));
        *reinterpret_cast<uint4*>(sP + off) = hv;
        *reinterpret_cast<uint4*>(sP + kTcQT + off) = mv;
        *reinterpret_cast<uint4*>(sP + 2 * kTcQT + off) = lv;
      }
      tc_fence_before();
      fence_proxy_async_smem();
      if (st == 0) tc_mark(a.trace, 1, j, 3);
      mbar_arrive(p_full);
    }
    if (nblk > 0) {
      tc_wait(o_full, (nblk - 1) & 1, err, 69);
      tc_fence_after();
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        float t[32];
        tmem_ld32(trow + 128u + (uint32_t)(half * 64 + c2 * 32), t);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[c2 * 32 + i] = o[c2 * 32 + i] * alpha_prev + t[i];
      }
      tc_fence_before();
    }
    // the row's sum over both halves of the keys
    float* xl = sX + (nblk & 1) * 256;
    xl[half * 128 + r] = l;
    named_sync(4, 256);
    const float lt = l + xl[(half ^ 1) * 128 + r];
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    if (rg < a.T_rows) {
      // the two fp16 planes of the output projection's activation
#pragma unroll
      for (int i = 0; i < 64; ++i) o[i] *= inv;
      store_planes<64>(a.out + ((size_t)b * a.T_rows + rg) * kActTerms * a.ldh + h * DH + half * 64, a.ldh, o);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace lat
