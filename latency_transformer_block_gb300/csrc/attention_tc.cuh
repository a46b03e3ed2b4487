// Segmented attention on the 5th-generation tensor cores (tcgen05, TMEM) for
// the dense path's MHA with dh = 128 (the DiT stage): a chunk of query rows
// attends to its noisy history segments (bf16 ring slots) and to its own keys
// as computed (fp32).  Online softmax in base 2, fp32 accumulation; the
// operands enter the tensor cores in fp16:
//
//   q, P       two fp16 planes (hi = fp16(x), lo = fp16(x - hi): 22 bits)
//   cached K/V the ring's bf16 values converted to fp16 (exact for
//              2^-14 <= |x| < 65504; below, fp16's subnormal spacing 2^-24)
//              once per call by hist_to_f16_kernel, into a copy that every
//              query tile and head then reads by TMA
//   own K/V    two fp16 planes of the fp32 values
//
//   S  = (Q_hi + Q_lo) K^T  (own keys: (Q_hi + Q_lo) (K_hi + K_lo)^T, with
//        K_hi and K_lo as the two 64-row halves of one N = 128 operand, so
//        each 16-dim step is two MMAs as for cached keys; the row warps add
//        the two 64-column halves of S)
//   O  = (P_hi + P_lo) V    (+ P_hi V_lo for own keys)
//
// The dropped cross term P_lo V_lo is below 2^-22 of the kept ones.  One CTA =
// one (128-row query tile, head, group), or one key range of such a tile when
// the launch splits the tiles of its last, partly filled wave
// (attention_tc_combine_kernel merges the ranges).  Keys run in blocks:
// 128 cached keys (history segments concatenated, N = 128 for S) or 64 own
// keys (hi and lo planes in the same buffers).  On this hardware an M = 128
// MMA costs the same ~152 cycles for N up to 256, so wide blocks matter.
//
// Roles: warp 0 (lane 0) issues the MMAs in the order S(0), S(1), PV(0),
// S(2), PV(1), ... so the tensor core computes S(j+1) while the row warps run
// the softmax of block j; warp 1 (lane 0) moves K and V of each block by TMA
// into one of two buffers each; warps 4..11 hold the rows: warp w reads TMEM
// lanes 32 (w % 4) .. + 31, half (w - 4) / 4 of each block's keys and of the
// output columns.  The row warps also release each landed K/V block to the
// MMA warp, zeroing the rows past the valid keys of a partial own block
// first (cached blocks need nothing: scores past the valid keys are masked,
// and the rows after them in the fp16 copy are finite): K(j+1) before the
// softmax of block j, V(j) right after writing its P.
//
// TMEM (512 columns): S of block j in columns 128 (j % 2) ..; the row warps
// write P of the block back over its own S columns as packed fp16 (per
// 32-key chunk: 16 columns of P_hi, then 16 of P_lo) and the PV MMA reads it
// there as its A operand.  The product of one key block, P V, lands in
// columns 256 + 128 (j % 2) .. and is added to the running output in fp32
// registers, so no TMEM accumulation chain is longer than 16 MMAs.
#pragma once
#include "attention.cuh"
#include "common.cuh"
#include "pi0_step.cuh"   // named_sync

namespace lat {

constexpr int kTcThreads = 384;
constexpr int kTcKB = 128;                      // cached keys per block
constexpr int kTcKBO = 64;                      // own keys per block
constexpr int kTcMinRangeBlocks = 2;            // key blocks of a split tile's key range, at least
constexpr int kTcQT = 16384;                    // one [128 rows][64] 16-bit tile
constexpr int kTcBuf = 32768;                   // one K or V buffer
// shared memory: Q [2 planes][2 k-tiles], K [2 buffers], V [2 buffers], row
// exchange [2 parities][2 halves][128 rows] fp32, barriers
constexpr int kTcOffQ = 0;
constexpr int kTcOffK = kTcOffQ + 4 * kTcQT;    // 64 KB
constexpr int kTcOffV = kTcOffK + 2 * kTcBuf;   // +64 KB
constexpr int kTcOffX = kTcOffV + 2 * kTcBuf;   // +64 KB
constexpr int kTcOffBar = kTcOffX + 4 * 128 * 4;
constexpr int kTcNBar = 24;
constexpr int kTcOffTab = kTcOffBar + kTcNBar * 8;   // TcSegTab
constexpr int kTcSmem = 1024 + kTcOffTab + 128 + 16;
// registers per thread after setmaxnreg: MMA/TMA warpgroup, row warpgroups
// (128 x 56 + 256 x 224 = 64512 = 384 x 168, the registers given at launch)
constexpr int kTcRegsLoad = 56, kTcRegsRow = 224;

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

// D[tmem] (+)= A[tmem] * B[smem desc]: A (M = 128 lanes x K = 16) read from
// TMEM, 16-bit elements packed two per 32-bit column.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 bit, 32 consecutive columns per thread, then wait for the store.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bit, 64 consecutive columns per thread in one instruction,
// then wait for the load.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
      "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 32 bit, 64 consecutive columns per thread in one instruction,
// then wait for the store.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {"
      "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,"
      "%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
      "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n\t"
      "tcgen05.wait::st.sync.aligned;"
      :
      : "r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]),
        "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]),
        "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]),
        "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]),
        "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
      : "memory");
}

// 2^x by the special-function unit (ex2.approx; results below 2^-126 flush to
// zero).  The softmax weights it produces lie in [0, 1], where a flushed value
// is negligible against the row sum.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 8 bf16 (one uint4) -> 8 fp16
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  auto cv = [](uint32_t w) {
    const __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    return *reinterpret_cast<const uint32_t*>(&h);
  };
  return make_uint4(cv(v.x), cv(v.y), cv(v.z), cv(v.w));
}

// 8 fp32 -> fp16 hi (8) and lo (8)
__device__ __forceinline__ void f32x8_to_h2planes(const float4 a, const float4 b, uint4& hi, uint4& lo) {
  split_pair_h2(a.x, a.y, hi.x, lo.x);
  split_pair_h2(a.z, a.w, hi.y, lo.y);
  split_pair_h2(b.x, b.y, hi.z, lo.z);
  split_pair_h2(b.z, b.w, hi.w, lo.w);
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

// The key blocks of a group: each cached segment (those without k16) cut
// into blocks of kTcKB keys, then the own keys (the segment with k16: fp16
// hi/lo planes) in blocks of kTcKBO.  A block never spans two segments, so
// each K or V block is one or two TMA boxes.  The per-segment table lives in
// shared memory (filled by one thread).
struct TcSegTab {
  int krow[kMaxSeg];       // first ring row of cached segment s, K plane
  int vrow[kMaxSeg];       // ... V plane
  int n[kMaxSeg];          // its keys
  int blk0[kMaxSeg + 1];   // its first block
  int own_row;             // first row of the own keys in the own-plane buffer
};

struct TcKeys {
  int nseg_c;              // cached segments
  int own_seg;             // index of the own segment (-1: none)
  int n_o;                 // own keys
  int nb_c, nblk;          // cached blocks, all blocks
  // tab: filled when not null (one thread)
  __device__ void init(const SegAttnArgs& a, const SegGroup& G, TcSegTab* tab) {
    nseg_c = 0;
    n_o = 0;
    own_seg = -1;
    nb_c = 0;
    for (int s = 0; s < G.nseg; ++s) {
      if (G.seg[s].k16) {
        own_seg = s;
        n_o = G.seg[s].n;
        if (tab) tab->own_row = (int)((G.seg[s].k16 - a.own16) / (4 * (size_t)a.kv_ld));
      } else {
        if (tab) {
          tab->krow[nseg_c] = (int)((G.seg[s].kh - a.hist16) / (size_t)a.kv_ld);
          tab->vrow[nseg_c] = (int)((G.seg[s].vh - a.hist16) / (size_t)a.kv_ld);
          tab->n[nseg_c] = G.seg[s].n;
          tab->blk0[nseg_c] = nb_c;
        }
        ++nseg_c;
        nb_c += (G.seg[s].n + kTcKB - 1) / kTcKB;
      }
    }
    if (tab) tab->blk0[nseg_c] = nb_c;
    nblk = nb_c + (n_o + kTcKBO - 1) / kTcKBO;
  }
  __device__ bool own(int j) const { return j >= nb_c; }
  // cached block j: its segment, first key within the segment and valid keys
  __device__ void cached(const TcSegTab* tab, int j, int& s, int& k0, int& nv) const {
    s = 0;
    while (s + 1 < nseg_c && j >= tab->blk0[s + 1]) ++s;
    k0 = (j - tab->blk0[s]) * kTcKB;
    nv = min(kTcKB, tab->n[s] - k0);
  }
  // valid keys of block j
  __device__ int valid(const TcSegTab* tab, int j) const {
    if (own(j)) return min(kTcKBO, n_o - (j - nb_c) * kTcKBO);
    int s, k0, nv;
    cached(tab, j, s, k0, nv);
    return nv;
  }
};

// ring_map: the fp16 history copy as rows of kv_ld (box 64 x 128, 128-byte swizzle);
// own_map: the own fp16 planes as rows of 4 kv_ld, [K hi | K lo | V hi | V lo]
// (box 64 x 64, same swizzle).
static __global__ void __launch_bounds__(kTcThreads, 1)
    attention_tc_kernel(const __grid_constant__ SegAttnArgs a, const __grid_constant__ CUtensorMap ring_map,
                        const __grid_constant__ CUtensorMap own_map, DevErr* err) {
  constexpr int DH = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + kTcOffQ;   // [plane][k-tile] of [128 rows][64 dims], K-major, swizzled
  uint8_t* sK = sm + kTcOffK;   // buffer: cached [k-tile][128 keys][64]; own hi [k-tile][64 keys][64], lo at +16 KB
  uint8_t* sV = sm + kTcOffV;   // buffer: cached [64-dim half][128 keys][64]; own hi [half][64 keys][64], lo at +16 KB
  float* sX = reinterpret_cast<float*>(sm + kTcOffX);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kTcOffBar);
  uint64_t* q_full = bar + 0;    // Q planes built (256 arrivals)
  uint64_t* k_full = bar + 1;    // [2] K block in fp16 (256: row warps)
  uint64_t* k_free = bar + 3;    // [2] S MMAs done with the K buffer (commit)
  uint64_t* v_full = bar + 5;    // [2] V block in fp16 (256)
  uint64_t* v_free = bar + 7;    // [2] PV MMAs done with the V buffer (commit)
  uint64_t* s_full = bar + 9;    // [2] S in TMEM (commit)
  uint64_t* p_full = bar + 11;   // [2] P written over S (256)
  uint64_t* o_full = bar + 13;   // [2] P V of the block in TMEM (commit)
  uint64_t* o_free = bar + 15;   // [2] P V read by the row warps (256)
  uint64_t* mdone = bar + 17;    // every MMA complete (teardown)
  uint64_t* kt_full = bar + 18;  // [2] TMA of the K block landed (1 + bytes)
  uint64_t* vt_full = bar + 20;  // [2] TMA of the V block landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 22);
  TcSegTab* tab = reinterpret_cast<TcSegTab*>(sm + kTcOffTab);

  // work item -> tile (and key range).  Query tile fastest: the tiles of one
  // head run together and share its K/V in L2.
  const int nqt = (a.T_rows + 127) / 128;
  const int item = blockIdx.x;
  const int tile = item < a.tc_whole ? item : a.tc_whole + (item - a.tc_whole) / a.tc_pieces;
  const int piece = item < a.tc_whole ? -1 : (item - a.tc_whole) % a.tc_pieces;
  const int qt = tile % nqt, h = (tile / nqt) % a.Hq, b = tile / (nqt * a.Hq);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = h / (a.Hq / a.Hkv);
  const SegGroup& G = a.grp[b];
  TcKeys kk;
  kk.init(a, G, threadIdx.x == 0 ? tab : nullptr);
  // key blocks j0 .. j0 + nblk - 1 of the group; below, j counts within the
  // range (buffers and parities) and j0 + j names the block
  const int j0 = piece < 0 ? 0 : piece * kk.nblk / a.tc_pieces;
  const int nblk = (piece < 0 ? kk.nblk : (piece + 1) * kk.nblk / a.tc_pieces) - j0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 256);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 256);
      mbar_init(&k_free[i], 1);
      mbar_init(&v_full[i], 256);
      mbar_init(&v_free[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 256);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_free[i], 256);
      mbar_init(&kt_full[i], 1);
      mbar_init(&vt_full[i], 1);
    }
    mbar_init(mdone, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);   // S/P [2 x 128], P V [2 x 128]
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kTcRegsLoad));
    if (warp == 0) {
      if (lane == 0) {
        // ---------------- MMA issue: S(0), S(1), PV(0), S(2), PV(1), ... ----------------
        const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK), va = smem_u32(sV);
        const uint32_t idO = idesc_f16_f32(128, DH) | (1u << 16);   // B (V) MN-major
        auto issue_s = [&](int j) -> bool {
          const int bf = j & 1;
          if (!tc_wait(&k_full[bf], (j >> 1) & 1, err, 61)) return false;
          tc_mark(a.trace, 0, j, 0);
          tc_fence_after();
          // 128 B-operand rows per k-tile: 128 cached keys, or the 64 own keys'
          // hi plane then their lo plane (S columns 0..63: (Q_hi + Q_lo) K_hi,
          // 64..127: (Q_hi + Q_lo) K_lo, summed by the row warps)
          const uint32_t kb = ka + (uint32_t)(bf * kTcBuf);
          const uint32_t idS = idesc_f16_f32(128, 128);
          const uint32_t d = tmem + (uint32_t)(bf * 128);
#pragma unroll
          for (int s = 0; s < DH / 16; ++s) {   // dims 16 s .. 16 s + 15
            const uint32_t kt = (uint32_t)(s >> 2), off = (uint32_t)((s & 3) * 32);
            const uint64_t bk = desc_k_sw128(kb + kt * 16384u + off);
            mma_bf16_ss(d, desc_k_sw128(qa + kt * kTcQT + off), bk, idS, s != 0 ? 1u : 0u);   // Q_hi K
            mma_bf16_ss(d, desc_k_sw128(qa + (2 + kt) * kTcQT + off), bk, idS, 1u);          // Q_lo K
          }
          mma_commit(&k_free[bf]);
          mma_commit(&s_full[bf]);
          return true;
        };
        auto issue_pv = [&](int j) -> bool {
          const int bf = j & 1;
          const uint32_t par = (uint32_t)(j >> 1) & 1u;
          if (!tc_wait(&p_full[bf], par, err, 62) || !tc_wait(&v_full[bf], par, err, 63)) return false;
          if (j >= 2 && !tc_wait(&o_free[bf], par ^ 1u, err, 64)) return false;
          tc_mark(a.trace, 0, j, 1);
          tc_fence_after();
          const bool own = kk.own(j0 + j);
          const int nk = own ? kTcKBO : kTcKB;
          const uint32_t vb = va + (uint32_t)(bf * kTcBuf);
          const uint32_t lbo = own ? 8192u : 16384u;   // bytes between the two 64-dim halves of V
          const uint32_t ps = tmem + (uint32_t)(bf * 128);
          const uint32_t d = tmem + 256u + (uint32_t)(bf * 128);
          for (int i = 0; i < nk / 16; ++i) {   // keys 16 i .. 16 i + 15
            const uint32_t ph = ps + (uint32_t)(32 * (i >> 1) + 8 * (i & 1));   // P_hi; P_lo at + 16
            const uint64_t bv = desc_mn_sw128(vb + (uint32_t)i * 2048u, lbo, 1024);
            mma_f16_ts(d, ph, bv, idO, i != 0 ? 1u : 0u);   // P_hi V
            mma_f16_ts(d, ph + 16u, bv, idO, 1u);           // P_lo V
            if (own)                                         // P_hi V_lo
              mma_f16_ts(d, ph, desc_mn_sw128(vb + 16384u + (uint32_t)i * 2048u, lbo, 1024), idO, 1u);
          }
          mma_commit(&v_free[bf]);
          mma_commit(&o_full[bf]);
          return true;
        };
        bool ok = tc_wait(q_full, 0, err, 60);
        for (int j = 0; j <= nblk && ok; ++j) {
          if (j < nblk) ok = issue_s(j);
          if (ok && j >= 1) ok = issue_pv(j - 1);
        }
        mma_commit(mdone);
        mbar_wait(mdone, 0, nullptr, 0);
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------- TMA: K and V of each block ----------------
      // cached: two 128-row boxes of fp16 history rows; own: two 64-row boxes of
      // each fp16 plane, into the swizzled operand layout
      tma_prefetch_desc(&ring_map);
      tma_prefetch_desc(&own_map);
      const uint64_t pol = l2_policy_evict_last();   // every query tile of the head re-reads the block
      bool ok = true;
      for (int j = 0; j < nblk && ok; ++j) {
        const int bf = j & 1;
        const uint32_t par = (uint32_t)(j >> 1) & 1u;
        for (int isv = 0; isv < 2 && ok; ++isv) {
          if (j >= 2 && !tc_wait(isv ? &v_free[bf] : &k_free[bf], par ^ 1u, err, isv ? 66 : 65)) {
            ok = false;
            break;
          }
          tc_mark(a.trace, 2, j, isv ? 2 : 0);
          uint8_t* dst = (isv ? sV : sK) + bf * kTcBuf;
          uint64_t* tb = isv ? &vt_full[bf] : &kt_full[bf];
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(tb, kTcBuf);
          if (!kk.own(j0 + j)) {
            int sgi, k0, nv;
            kk.cached(tab, j0 + j, sgi, k0, nv);
            const int row = (isv ? tab->vrow[sgi] : tab->krow[sgi]) + k0;
            tma_load_2d(dst, &ring_map, tb, kvh * DH, row, pol);
            tma_load_2d(dst + 16384, &ring_map, tb, kvh * DH + 64, row, pol);
          } else {
            // own-plane rows: [K hi | K lo | V hi | V lo], kv_ld columns each
            // K: [k-tile][hi 64 rows | lo 64 rows]; V: [plane][64-dim half][64 keys]
            const int row = tab->own_row + (j0 + j - kk.nb_c) * kTcKBO;
            const int xh = (isv ? 2 * a.kv_ld : 0) + kvh * DH, xl = xh + a.kv_ld;
            const int o1 = isv ? 8192 : 16384, ol = isv ? 16384 : 8192;   // second k-tile / half, lo plane
            tma_load_2d(dst, &own_map, tb, xh, row, pol);
            tma_load_2d(dst + o1, &own_map, tb, xh + 64, row, pol);
            tma_load_2d(dst + ol, &own_map, tb, xl, row, pol);
            tma_load_2d(dst + ol + o1, &own_map, tb, xl + 64, row, pol);
          }
        }
      }
      // never leave a copy in flight into this CTA's shared memory
      for (int j = (nblk > 2 ? nblk - 2 : 0); j < nblk; ++j) {
        tc_wait(&kt_full[j & 1], (uint32_t)(j >> 1) & 1u, err, 71);
        tc_wait(&vt_full[j & 1], (uint32_t)(j >> 1) & 1u, err, 72);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kTcRegsRow));
    // ---------------- row warps ----------------
    const int st = threadIdx.x - 128;
    const int quad = warp & 3, half = (warp - 4) >> 2;
    const int r = quad * 32 + lane;                  // row of the tile = TMEM lane
    const int rg = qt * 128 + r;                     // row within the group
    // Q planes (fp16 hi, lo) for the tile's 128 rows
    for (int it = st; it < 128 * (DH / 8); it += 256) {
      const int rr = it >> 4, c = it & 15;
      const int rq = qt * 128 + rr;
      uint4 hv = make_uint4(0, 0, 0, 0), lv = hv;
      if (rq < a.T_rows) {
        const float* src = a.q + ((size_t)b * a.T_rows + rq) * a.q_ld + h * DH + c * 8;
        f32x8_to_h2planes(__ldg(reinterpret_cast<const float4*>(src)), __ldg(reinterpret_cast<const float4*>(src + 4)),
                          hv, lv);
      }
      const int o = (c >> 3) * kTcQT + rr * 128 + (((c & 7) ^ (rr & 7)) << 4);
      *reinterpret_cast<uint4*>(sQ + o) = hv;
      *reinterpret_cast<uint4*>(sQ + 2 * kTcQT + o) = lv;
    }
    fence_proxy_async_smem();
    mbar_arrive(q_full);

    // a landed K or V block: own blocks get the rows past their valid keys
    // zeroed (the own planes after a group's keys may hold anything)
    auto prep = [&](int j, bool isv) {
      const int bf = j & 1;
      tc_wait(isv ? &vt_full[bf] : &kt_full[bf], (uint32_t)(j >> 1) & 1u, err, isv ? 70 : 69);
      uint8_t* dst = (isv ? sV : sK) + bf * kTcBuf;
      const int nv = kk.valid(tab, j0 + j);
      if (kk.own(j0 + j) && nv < kTcKBO) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int it = st + 256 * u, r = it >> 4, c = it & 15;
          if (r < nv) continue;
          const int o1 = isv ? 8192 : 16384, ol = isv ? 16384 : 8192;   // as the TMA placed them
          const int off = (c >> 3) * o1 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(dst + off) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(dst + ol + off) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(isv ? &v_full[bf] : &k_full[bf]);
    };

    float o[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) o[i] = 0.f;
    float m = -INFINITY, l = 0.f, alpha_prev = 0.f;
    const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
    // P V of block jb into the running output (then the columns are free again)
    auto add_o = [&](int jb) {
      const int bf = jb & 1;
      tc_wait(&o_full[bf], (uint32_t)(jb >> 1) & 1u, err, 68);
      tc_fence_after();
      float t[64];
      tmem_ld64(trow + 256u + (uint32_t)(bf * 128 + half * 64), t);
#pragma unroll
      for (int i = 0; i < 64; ++i) o[i] = o[i] * alpha_prev + t[i];
      tc_fence_before();
      mbar_arrive(&o_free[bf]);
    };
    if (nblk > 0) prep(0, false);
    for (int j = 0; j < nblk; ++j) {
      const int bf = j & 1;
      const bool own = kk.own(j0 + j);
      if (j + 1 < nblk) prep(j + 1, false);   // K of the next block: its S overlaps this softmax
      const int nh = (own ? kTcKBO : kTcKB) / 2;     // keys of this thread's half
      const int k0 = half * nh, nv = kk.valid(tab, j0 + j);
      tc_wait(&s_full[bf], (uint32_t)(j >> 1) & 1u, err, 67);
      if (st == 0) tc_mark(a.trace, 1, j, 0);
      tc_fence_after();
      const uint32_t sb = trow + (uint32_t)(bf * 128 + k0);   // S (then P) columns of my keys
      // raw scores of my keys (an own block has 32 per half: the K_hi and K_lo
      // parts, 64 columns apart)
      float s[64];
      if (own) {
        float t[32], u[32];
        tmem_ld32x2(sb, sb + 64u, t, u);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = t[i] + u[i];
      } else {
        tmem_ld64(sb, s);
      }
      float mloc = -INFINITY;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        s[i] = (i < nh && k0 + i < nv) ? s[i] : -INFINITY;
        mloc = fmaxf(mloc, s[i]);
      }
      mloc *= a.scale_log2;   // the scale is positive: the maximum commutes with it
      float* xb = sX + (j & 1) * 256;
      xb[half * 128 + r] = mloc;
      named_sync(4, 256);
      // every block has a valid key, so mnew is finite from the first block on
      const float mnew = fmaxf(m, fmaxf(mloc, xb[(half ^ 1) * 128 + r]));
      const float alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - mnew);
      float lsum = 0.f;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        s[i] = ex2_approx(fmaf(s[i], a.scale_log2, -mnew));   // masked keys: 2^-inf = 0
        lsum += s[i];
      }
      l = l * alpha + lsum;
      m = mnew;
      if (st == 0) tc_mark(a.trace, 1, j, 1);
      // P over the S columns: per 32-key chunk 16 columns of P_hi, 16 of P_lo
      if (own) {
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 16; ++e) split_pair_h2(s[2 * e], s[2 * e + 1], w[e], w[16 + e]);
        tmem_st32(sb, w);
      } else {
        uint32_t w[64];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
#pragma unroll
          for (int e = 0; e < 16; ++e)
            split_pair_h2(s[32 * ch + 2 * e], s[32 * ch + 2 * e + 1], w[32 * ch + e], w[32 * ch + 16 + e]);
        tmem_st64(sb, w);
      }
      tc_fence_before();
      mbar_arrive(&p_full[bf]);
      prep(j, true);   // V of this block
      if (st == 0) tc_mark(a.trace, 1, j, 2);
      if (j > 0) add_o(j - 1);
      if (st == 0) tc_mark(a.trace, 1, j, 3);
      alpha_prev = alpha;
    }
    if (nblk > 0) add_o(nblk - 1);
    // the row's sum over both halves of the keys
    float* xl = sX + (nblk & 1) * 256;
    xl[half * 128 + r] = l;
    named_sync(4, 256);
    const float lt = l + xl[(half ^ 1) * 128 + r];
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    if (rg < a.T_rows && piece < 0) {
#pragma unroll
      for (int i = 0; i < 64; ++i) o[i] *= inv;
      // the two fp16 planes of the output projection's activation
      store_planes<64>(a.out + ((size_t)b * a.T_rows + rg) * kActTerms * a.ldh + h * DH + half * 64, a.ldh, o);
    } else if (rg < a.T_rows) {
      // one key range of a split tile: unnormalised output (relative to 2^m)
      // and the row's (m, sum) for attention_tc_combine_kernel
      const size_t pr = (size_t)(item - a.tc_whole) * 128 + r;
      float4* po = reinterpret_cast<float4*>(a.tc_part_o + pr * DH + half * 64);
#pragma unroll
      for (int i = 0; i < 16; ++i) po[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
      if (half == 0) *reinterpret_cast<float2*>(a.tc_part_ml + pr * 2) = make_float2(m, lt);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge the key ranges of the split tiles: per row, the ranges' outputs
// weighted by 2^(m_p - max m) over the weighted sums, written as the two fp16
// planes a whole tile writes.  Grid (split tiles, 128 rows), one thread per
// head dim.  A range without keys has m = -inf and weight 0.
static __global__ void __launch_bounds__(128) attention_tc_combine_kernel(const __grid_constant__ SegAttnArgs a) {
  constexpr int DH = 128;
  const int nqt = (a.T_rows + 127) / 128;
  const int tile = a.tc_whole + blockIdx.x, r = blockIdx.y, c = threadIdx.x;
  const int qt = tile % nqt, h = (tile / nqt) % a.Hq, b = tile / (nqt * a.Hq);
  const int rg = qt * 128 + r;
  if (rg >= a.T_rows) return;
  const size_t p0 = (size_t)blockIdx.x * a.tc_pieces;
  float M = -INFINITY;
  for (int p = 0; p < a.tc_pieces; ++p) M = fmaxf(M, a.tc_part_ml[((p0 + p) * 128 + r) * 2]);
  float num = 0.f, den = 0.f;
  for (int p = 0; p < a.tc_pieces; ++p) {
    const size_t i = (p0 + p) * 128 + r;
    const float m = a.tc_part_ml[i * 2], w = m == -INFINITY ? 0.f : exp2f(m - M);
    num += w * a.tc_part_o[i * DH + c];
    den += w * a.tc_part_ml[i * 2 + 1];
  }
  const float v = den > 0.f ? num / den : 0.f;
  const __half hv = __float2half_rn(v);
  __half* o = a.out + ((size_t)b * a.T_rows + rg) * kActTerms * a.ldh + h * DH + c;
  o[0] = hv;
  o[a.ldh] = __float2half_rn(v - __half2float(hv));
}

// The history K/V segments of one call (bf16 ring rows) -> their fp16 copy,
// planes of `rows` x `cols`; the same conversion per value as bf16x8_to_f16x8.
constexpr int kMaxHistPlanes = 128;
struct HistCvtArgs {
  const __nv_bfloat16* src[kMaxHistPlanes];
  __half* dst[kMaxHistPlanes];
  int planes, rows, cols;
  // page_tokens > 0: planes 2q (K) and 2q + 1 (V) are ring rows row0[q] ..
  // + rows - 1 of one ring, kept in the pool [pages][2][page_tokens][cols]
  // through its page list ptab[q] (src unused)
  int page_tokens;
  const int* ptab[kMaxHistPlanes / 2];
  int row0[kMaxHistPlanes / 2];
  const __nv_bfloat16* pool;
};

// Contiguous rings: a grid-stride loop over 8-value chunks.  Pages: one warp
// per (plane, row), the row's pool address resolved once through the page
// table and its cols / 8 chunks taken by the lanes in turn (grid-stride over
// planes x rows, 8 warps a CTA).
static __global__ void __launch_bounds__(256) hist_to_f16_kernel(const __grid_constant__ HistCvtArgs a) {
  if (a.page_tokens == 0) {
    const size_t per = (size_t)a.rows * a.cols / 8;   // 8-value chunks per plane
    const size_t n = per * a.planes;
    for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (size_t)gridDim.x * 256) {
      const int p = (int)(i / per);
      const size_t j = i - (size_t)p * per;
      reinterpret_cast<uint4*>(a.dst[p])[j] = bf16x8_to_f16x8(__ldcs(reinterpret_cast<const uint4*>(a.src[p]) + j));
    }
    return;
  }
  const int lane = threadIdx.x & 31, c8 = a.cols / 8;   // cols is a multiple of 8
  const long long tasks = (long long)a.planes * a.rows;
  for (long long t = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); t < tasks; t += (long long)gridDim.x * 8) {
    const int p = (int)(t / a.rows), row = (int)(t - (long long)p * a.rows);
    const int r = a.row0[p >> 1] + row, P = a.page_tokens;
    const uint4* src = reinterpret_cast<const uint4*>(
        a.pool + (((size_t)a.ptab[p >> 1][r / P] * 2 + (p & 1)) * P + r % P) * (size_t)a.cols);
    uint4* dst = reinterpret_cast<uint4*>(a.dst[p] + (size_t)row * a.cols);
#pragma unroll 4
    for (int c = lane; c < c8; c += 32) dst[c] = bf16x8_to_f16x8(__ldcs(src + c));
  }
}

}  // namespace lat
