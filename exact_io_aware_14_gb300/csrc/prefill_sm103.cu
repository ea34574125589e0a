// Exact attention forward, prefill / training shapes, for sm_103a.
//
// One CTA computes two 128-row query tiles that share every K/V tile: two
// consecutive row tiles of one head, or -- when the GQA group size is even --
// the same row tile of two query heads that read the same KV head (equal
// causal extents).  Twelve warps:
//   warp 0        TMA producer: per work unit Q_0, Q_1, then its K/V tiles
//                 into one ring of shared-memory slots in the order the MMA
//                 thread uses them
//   warp 1        TMEM allocator and MMA issuer (one thread), per key tile j:
//                   O_0 += P_0 V_{j-1};  S_0 = Q_0 K_j^T;
//                   O_1 += P_1 V_{j-1};  S_1 = Q_1 K_j^T
//                 so the tensor core works on one tile while the softmax
//                 warpgroup of the other tile runs (ping-pong); a commit
//                 after the last MMA that reads a ring slot frees it.
//   warps 4-7     softmax of tile 0, warps 8-11 softmax of tile 1: one
//                 thread owns one query row (one TMEM lane); it reads its
//                 128 scores, forms p under the row's exponent reference m
//                 (taking the tile max only where m is first set or must
//                 move), adds to the sum l, rescales its O row in TMEM only
//                 if m moved, and writes P (bf16) back into TMEM over the
//                 scores; the P.V MMA reads P from TMEM as its A operand.
//                 At the end: O / l and the LSE.
//
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+d),
// O_1 [384,384+d); P_t is packed bf16x2 in the first 64 columns of S_t.
//
// The method is the tiled online softmax of "FlashAttention: Part 2"
// (chizkidd.github.io), section 6.2: per score tile, update (m, l, a) with
// alpha = exp(m - m') and discard the tile.  Normalisation is deferred to the
// epilogue and the rescale is skipped when the max did not move ("Trace
// FlashAttention's evolution through plain PyTorch code", FA2 and FA4
// paragraphs); the two-tile ping-pong follows the FA3 schedule of section 1.5.
// Scores are handled in base 2: p = 2^(s*c - m*c) with c = scale*log2(e) folded
// into one FMA, and LSE = (m*c + log2 l) * ln 2.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "exp2_poly.cuh"
#include "launch.h"
#include "ptx.cuh"

// Build switch: ATTN_EXP2_POLY = K > 0 computes every K-th pair of a row's
// exponentials with the software exp2 of exp2_poly.cuh (on the FMA and
// integer pipes) instead of the MUFU unit, as FA4 does on Blackwell; 0 (the
// default build) uses MUFU for all of them.  K divides 16.
#ifndef ATTN_EXP2_POLY
#define ATTN_EXP2_POLY 0
#endif

namespace attn {
namespace {

constexpr int kPolyEvery = ATTN_EXP2_POLY;
static_assert(kPolyEvery == 0 || (kPolyEvery > 0 && 16 % kPolyEvery == 0), "ATTN_EXP2_POLY must divide 16");

// 2^x for the pair of a row's exponentials with pair index i (the index
// within its 64-column half): MUFU, or the software form for every
// kPolyEvery-th pair.
__device__ __forceinline__ float2 exp2_pair(float2 x, int i) {
  if (kPolyEvery > 0 && (i % (kPolyEvery > 0 ? kPolyEvery : 1)) == kPolyEvery - 1) return exp2_poly2(x);
  return make_float2(ex2_approx(x.x), ex2_approx(x.y));
}

__device__ uint32_t g_prefill_status;

constexpr int BM = 128;  // query rows per tile (MMA M, TMEM lanes)
constexpr int BN = 128;  // keys per K/V tile (MMA N of QK^T, K of PV)
constexpr int kThreads = 384;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: no legitimate wait comes close
constexpr uint32_t kTmemCols = 512;

template <int D>
struct Layout {
  // one ring of K and V tiles, filled in the order the MMA thread uses them
  static constexpr int kSlots = (D == 64) ? 10 : 5;
  static constexpr int kHalf = 128 * 128;  // one 64-column block of a 128-row tile
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kOffQ = 0;  // Q_0, Q_1
  static constexpr int kOffRing = kOffQ + 2 * kTile;
  static constexpr int kOffBar = kOffRing + kSlots * kTile;
  static constexpr int kNumBars = 2 * kSlots + 6 * 2 + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 B
};

__device__ __forceinline__ void record(uint32_t site, uint32_t code) {
  atomicCAS(&g_prefill_status, 0u, (site << 8) | code);
}

// warp-uniform bounded wait
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         uint32_t site) {
  bool ok = mbar_wait(bar, parity, abort_flag, kWaitLimitNs);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) record(site, kDevTimeout);
  return ok;
}
// single-thread bounded wait
__device__ __forceinline__ bool wait_one(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         uint32_t site) {
  bool ok = mbar_wait(bar, parity, abort_flag, kWaitLimitNs);
  if (!ok) record(site, kDevTimeout);
  return ok;
}

// Ring order of the K/V tiles of a unit with n key tiles: K_0, then K_m,
// V_{m-1} for m = 1 .. n-1, then V_{n-1}; MMA step j uses K_j and V_{j-1}.
// K_j is loaded two steps ahead of its use, V_{j-1} one step ahead.
__device__ __forceinline__ int k_item(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int v_item(int j, int n) { return j == n - 1 ? 2 * n - 1 : 2 * j + 2; }

struct TileInfo {
  int hq;    // query head
  int row0;  // first query row
  int n_kt;  // key tiles this tile visits (0: inactive)
};

// Where a tile's max is taken (a row's first visible scores, or a warp's rare
// fix-up), the row's exponent reference is moved (and O, l rescaled) only when
// that max exceeds it by more than this many powers of two.  Between moves p
// stays small enough (2^8 here, 2^16 under the one-pass form's sum check
// below) for bf16 P, fp32 l and the fp32 O accumulator to hold it with full
// relative precision, and O / l and the LSE come out the same.
constexpr float kRescaleLog2 = 8.f;

// One 64-column half h of this lane's scores, read from TMEM.  Masked tiles
// keep columns [lo, lim) (kLo) or [0, lim); kNeg: the scale is negative and
// the kernel works on -s.
__device__ __forceinline__ void load_half(uint32_t tS, int h, uint32_t (&u)[2][32]) {
  tmem_ld32(tS + 64 * h, u[0]);
  tmem_ld32(tS + 64 * h + 32, u[1]);
  tmem_wait_ld();
}

template <bool kMasked, bool kNeg, bool kLo>
__device__ __forceinline__ float half_max(const uint32_t (&u)[2][32], int h, int lo, int lim) {
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int i = 0; i < 64; i += 4) {
    float v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[k] = __uint_as_float(u[(i + k) >> 5][(i + k) & 31]);
      if (kNeg) v[k] = -v[k];
      if (kMasked) v[k] = (64 * h + i + k < lim && (!kLo || 64 * h + i + k >= lo)) ? v[k] : -INFINITY;
    }
    mx0 = fmax3(mx0, v[0], v[1]);
    mx1 = fmax3(mx1, v[2], v[3]);
  }
  return fmaxf(mx0, mx1);
}

// p = 2^(s*c - mc) for half h, packed as bf16 pairs into pk and summed into
// acc0 / acc1.
template <bool kMasked, bool kNeg, bool kLo>
__device__ __forceinline__ void half_exp(const uint32_t (&u)[2][32], int h, int lo, int lim, float c, float mc,
                                         float2& acc0, float2& acc1, uint32_t (&pk)[32]) {
  const float2 c2 = make_float2(c, c), nmc2 = make_float2(-mc, -mc);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float v0 = __uint_as_float(u[i >> 4][(2 * i) & 31]);
    float v1 = __uint_as_float(u[i >> 4][(2 * i + 1) & 31]);
    if (kNeg) {
      v0 = -v0;
      v1 = -v1;
    }
    const float2 x = ffma2(make_float2(v0, v1), c2, nmc2);
    const float2 e = exp2_pair(x, i);
    float p0 = e.x;
    float p1 = e.y;
    if (kMasked) {  // also right for c == 0, where -inf * 0 would not give 0
      p0 = (64 * h + 2 * i < lim && (!kLo || 64 * h + 2 * i >= lo)) ? p0 : 0.f;
      p1 = (64 * h + 2 * i + 1 < lim && (!kLo || 64 * h + 2 * i + 1 >= lo)) ? p1 : 0.f;
    }
    if (i & 1)
      acc1 = fadd2(acc1, make_float2(p0, p1));
    else
      acc0 = fadd2(acc0, make_float2(p0, p1));
    pk[i] = pack_bf16x2(p0, p1);
  }
}

__device__ __forceinline__ float acc_sum(float2 a0, float2 a1) { return (a0.x + a0.y) + (a1.x + a1.y); }

// half_exp for one 32-column quarter q of the scores (uq: its raw values),
// writing pairs (q & 1) * 16 .. + 15 of the half's packed P.  Two quarters in
// order give the same operations in the same order as half_exp.
template <bool kMasked, bool kNeg, bool kLo>
__device__ __forceinline__ void quarter_exp(const uint32_t (&uq)[32], int q, int lo, int lim, float c, float mc,
                                            float2& acc0, float2& acc1, uint32_t (&pk)[32]) {
  const float2 c2 = make_float2(c, c), nmc2 = make_float2(-mc, -mc);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float v0 = __uint_as_float(uq[2 * i]);
    float v1 = __uint_as_float(uq[2 * i + 1]);
    if (kNeg) {
      v0 = -v0;
      v1 = -v1;
    }
    const float2 x = ffma2(make_float2(v0, v1), c2, nmc2);
    const float2 e = exp2_pair(x, (q & 1) * 16 + i);
    float p0 = e.x;
    float p1 = e.y;
    if (kMasked) {
      p0 = (32 * q + 2 * i < lim && (!kLo || 32 * q + 2 * i >= lo)) ? p0 : 0.f;
      p1 = (32 * q + 2 * i + 1 < lim && (!kLo || 32 * q + 2 * i + 1 >= lo)) ? p1 : 0.f;
    }
    if (i & 1)
      acc1 = fadd2(acc1, make_float2(p0, p1));
    else
      acc0 = fadd2(acc0, make_float2(p0, p1));
    pk[(q & 1) * 16 + i] = pack_bf16x2(p0, p1);
  }
}

// Row max of one 128-column score tile (this thread's lane).
template <bool kMasked, bool kNeg, bool kLo = false>
__device__ __forceinline__ float score_tile_max(uint32_t tS, int lo, int lim) {
  float mx = -INFINITY;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t u[2][32];
    load_half(tS, h, u);
    mx = fmaxf(mx, half_max<kMasked, kNeg, kLo>(u, h, lo, lim));
  }
  return mx;
}

// p = 2^(s*c - mc) for the 128 scores of this lane, written back as bf16
// pairs over the first 64 columns (half h of P only overwrites scores already
// consumed).  Returns the row sum of the fp32 p.
template <bool kMasked, bool kNeg, bool kLo = false>
__device__ __forceinline__ float score_tile_exp(uint32_t tS, int lo, int lim, float c, float mc) {
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    uint32_t u[2][32], pk[32];
    load_half(tS, h, u);
    half_exp<kMasked, kNeg, kLo>(u, h, lo, lim, c, mc, acc0, acc1, pk);
    tmem_st32(tS + 32 * h, pk);
  }
  return acc_sum(acc0, acc1);
}

// A half's p sum above this means one of its p passed it; below it every
// p <= 2^16, which bf16 P and the fp32 row sum and O accumulator hold with
// full relative precision.
constexpr float kSumLimit = 65536.f;

struct HalfFix {
  float sum;  // the half's (or the tile's) row sum after the fix
  float m;    // the lane's exponent reference after the fix
};

// Rare path of the one-pass softmax, half 0: some lane's half-0 sum passed
// kSumLimit (flag ov) before its P was stored, so its scores are still in
// TMEM.  Every lane of the warp calls this together (TMEM accesses are
// warp-wide); a lane with ov moves its reference to the half's max, the
// others recompute the same P.  Stores half 0's P.
template <bool kMasked, bool kNeg, bool kLo>
__device__ __noinline__ HalfFix fix_half0(uint32_t tS, int lo, int lim, float c, float m, bool ov) {
  uint32_t u[2][32], pk[32];
  float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
  load_half(tS, 0, u);
  if (ov) m = fmaxf(m, half_max<kMasked, kNeg, kLo>(u, 0, lo, lim));
  half_exp<kMasked, kNeg, kLo>(u, 0, lo, lim, c, m * c, a0, a1, pk);
  tmem_st32(tS, pk);
  return {acc_sum(a0, a1), m};
}

// Rare path, half 1: some lane's half-1 sum passed kSumLimit; half 1's
// scores are still in TMEM, half 0's P went out under the reference m.  A
// lane with ov moves its reference to the half's max and rescales its stored
// half-0 P (and sum t0) by 2^(m*c - m_new*c); every lane recomputes and
// stores half 1's P.  Returns the tile's row sum.
template <bool kMasked, bool kNeg, bool kLo>
__device__ __noinline__ HalfFix fix_half1(uint32_t tS, int lo, int lim, float c, float m, float t0, bool ov) {
  uint32_t u[2][32], pk[32];
  float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
  load_half(tS, 1, u);
  float a01 = 1.f;
  if (ov) {
    const float m_new = fmaxf(m, half_max<kMasked, kNeg, kLo>(u, 1, lo, lim));
    a01 = ex2_approx(m * c - m_new * c);
    m = m_new;
  }
  half_exp<kMasked, kNeg, kLo>(u, 1, lo, lim, c, m * c, a0, a1, pk);
  tmem_st32(tS + 32, pk);
  tmem_wait_st();  // half 0's P was stored by the caller just before
  tmem_ld32(tS, u[0]);
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float lo_f = __uint_as_float(u[0][i] << 16), hi_f = __uint_as_float(u[0][i] & 0xffff0000u);
    u[0][i] = (a01 != 1.f) ? pack_bf16x2(lo_f * a01, hi_f * a01) : u[0][i];
  }
  tmem_st32(tS, u[0]);
  return {t0 * a01 + acc_sum(a0, a1), m};
}

// One pass over the tile for rows whose exponent reference m is set (every
// row of the warp has seen scores): p = 2^(s*c - m*c) under the current
// reference, each score read once and no max formed; a half whose p sum
// passes kSumLimit sends the warp through fix_half0 / fix_half1, which move
// that row's reference.  Keeps the two-pass form's summation order, so the
// result is the same whenever the reference does not move.  Returns the row
// sum in units of the updated reference m.
template <bool kMasked, bool kNeg, bool kLo = false>
__device__ __forceinline__ float score_tile_onepass(uint32_t tS, int lo, int lim, float c, float& m) {
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
  uint32_t ua[32], ub[32], pk[32];
  // each quarter's load is issued before the previous quarter's arithmetic
  // and awaited after it; no call and no use of a register in flight comes
  // between a load and its wait
  tmem_ld32(tS, ua);
  tmem_wait_ld();
  tmem_ld32(tS + 32, ub);
  quarter_exp<kMasked, kNeg, kLo>(ua, 0, lo, lim, c, m * c, acc0, acc1, pk);
  tmem_wait_ld();
  tmem_ld32(tS + 64, ua);
  quarter_exp<kMasked, kNeg, kLo>(ub, 1, lo, lim, c, m * c, acc0, acc1, pk);
  tmem_wait_ld();
  float t0 = acc_sum(acc0, acc1);
  const bool ov0 = !(t0 <= kSumLimit);
  if (__any_sync(0xffffffffu, ov0)) {
    const HalfFix f = fix_half0<kMasked, kNeg, kLo>(tS, lo, lim, c, m, ov0);
    if (ov0) {
      m = f.m;
      t0 = f.sum;
      acc0 = make_float2(t0, 0.f);  // later sums build on the fixed half-0 sum
      acc1 = make_float2(0.f, 0.f);
    }
  } else {
    tmem_st32(tS, pk);
  }
  tmem_ld32(tS + 96, ub);
  quarter_exp<kMasked, kNeg, kLo>(ua, 2, lo, lim, c, m * c, acc0, acc1, pk);
  tmem_wait_ld();
  quarter_exp<kMasked, kNeg, kLo>(ub, 3, lo, lim, c, m * c, acc0, acc1, pk);
  float total = acc_sum(acc0, acc1);
  const bool ov1 = !(total - t0 <= kSumLimit);
  if (__any_sync(0xffffffffu, ov1)) {
    const HalfFix f = fix_half1<kMasked, kNeg, kLo>(tS, lo, lim, c, m, t0, ov1);
    if (ov1) {
      m = f.m;
      total = f.sum;
    }
  } else {
    tmem_st32(tS + 32, pk);
  }
  return total;
}

// Work unit U -> (batch, KV head, the two query tiles).  Units are numbered
// (u_rev, head slot, batch) with u_rev slowest, so units whose rows see a
// right-bounded key range (causal, or a window's right side) come longest
// first and every round holds units of about one length, which the zig-zag
// balances.  kSlotMajor (the instance for no mask, where all units of a slot
// are equally long) numbers them (head slot, batch, u_rev) with u_rev
// fastest instead: the CTAs of a round then share a few heads' K and V,
// which come from L2 after their first read.  Keys of the unit's sequence: nk (Nk, or its cache length when
// seqlens is given); key j is visible to row i iff j < nk, j <= i + coff and,
// in the general form, j >= i + lo.  causal 1 aligns top-left (coff = 0), 2
// bottom-right (coff = nk - Nq); a local window (wl, wr) is aligned
// bottom-right: row i sits at key position i + nk - Nq and sees wl keys
// before it and wr after it (negative: that side unbounded).  The unit's key
// tiles are kt0 .. kt0 + n_kt - 1; tile t visits the first ti[t].n_kt of them
// in the order key_tile gives.
struct Unit {
  int b, hkv, n_kt;
  int nk, coff, lo, kt0;
  bool rot;  // visit kt0 last (key_tile)
  TileInfo ti[2];
};
template <bool kGeneral, bool kSlotMajor = false>
__device__ __forceinline__ Unit decode_unit(int U, int B, int Hq, int Hkv, int Nq, int Nk, int causal, int wl, int wr,
                                            const int* __restrict__ seqlens, int pair_heads, int units_per_bh) {
  Unit u;
  const int hslots = pair_heads ? Hq / 2 : Hq;
  const int bh_count = B * hslots;
  int u_rev, bh;
  if (kSlotMajor) {
    bh = U / units_per_bh;
    u_rev = U % units_per_bh;
  } else {
    u_rev = U / bh_count;
    bh = U % bh_count;
  }
  const bool rev = (causal != 0) || (kGeneral && wr >= 0);
  const int unit = rev ? (units_per_bh - 1 - u_rev) : u_rev;
  u.b = bh / hslots;
  const int hs = bh % hslots;
  if (pair_heads) {
    u.ti[0].hq = 2 * hs;
    u.ti[1].hq = 2 * hs + 1;
    u.ti[0].row0 = u.ti[1].row0 = unit * BM;
  } else {
    u.ti[0].hq = u.ti[1].hq = hs;
    u.ti[0].row0 = (2 * unit) * BM;
    u.ti[1].row0 = (2 * unit + 1) * BM;
  }
  u.hkv = u.ti[0].hq / (Hq / Hkv);  // both heads of a pair share the KV head
  u.nk = seqlens ? min(max(seqlens[u.b], 0), Nk) : Nk;
  if (!kGeneral) {
    u.coff = (causal == 2) ? u.nk - Nq : 0;
    u.lo = 0;
    u.kt0 = 0;
    u.rot = false;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int kend = causal ? max(0, min(u.nk, u.ti[t].row0 + BM + u.coff)) : u.nk;
      u.ti[t].n_kt = (u.ti[t].row0 < Nq) ? (kend + BN - 1) / BN : 0;
    }
  } else {
    const int pos0 = u.nk - Nq;  // key position of query row 0
    int hi = u.nk;               // no right bound
    if (causal) hi = (causal == 2) ? pos0 : 0;
    if (wr >= 0) hi = min(hi, pos0 + wr);
    u.coff = hi;
    u.lo = (wl >= 0) ? pos0 - wl : -(Nq + BM);  // -(Nq + BM): no left bound for any row of a tile
    int kend[2], first = u.nk;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      // keys some row of the tile sees: [row0 + lo, row0 + BM - 1 + hi] within [0, nk)
      const int kbeg = max(0, u.ti[t].row0 + u.lo);
      kend[t] = min(u.nk, u.ti[t].row0 + BM + hi);
      if (u.ti[t].row0 >= Nq || kend[t] <= kbeg)
        kend[t] = 0;
      else
        first = min(first, kbeg);
    }
    u.kt0 = first / BN;
#pragma unroll
    for (int t = 0; t < 2; ++t) u.ti[t].n_kt = kend[t] > 0 ? (kend[t] + BN - 1) / BN - u.kt0 : 0;
    // Under a left window bound the first key tile is usually a staircase
    // that some rows see only in part.  A row's first visited tile is the one
    // where its max is taken in two passes, which on a masked tile costs about
    // twice an unmasked one and sits on the critical path of the unit's start;
    // when both query tiles visit the same key tiles (a head pair) and a full
    // tile follows, kt0 is visited last instead.  Visiting order does not
    // change what is computed, only the rounding order of the sums.
    u.rot = pair_heads && u.ti[0].n_kt >= 3 && u.ti[1].n_kt == u.ti[0].n_kt &&
            u.kt0 * BN < u.ti[0].row0 + BM - 1 + u.lo;
  }
  u.n_kt = max(u.ti[0].n_kt, u.ti[1].n_kt);
  return u;
}

// Key tile visited at step j of a unit: kt0 + j, or with u.rot kt0 + 1,
// kt0 + 2, ..., kt0 + n_kt - 1 and then kt0.
template <bool kGeneral>
__device__ __forceinline__ int key_tile(const Unit& u, int j) {
  if (!kGeneral) return j;  // kt0 = 0, no rotation
  return u.kt0 + (u.rot ? (j + 1 < u.n_kt ? j + 1 : 0) : j);
}

// Unit of round r for this CTA: zig-zag over the CTAs (c, then G-1-c, ...),
// which balances the longest-first causal units across CTAs.  -1: none.
__device__ __forceinline__ int unit_of_round(int r, int total_units) {
  const int G = gridDim.x, c = blockIdx.x;
  const int U = r * G + ((r & 1) ? (G - 1 - c) : c);
  return U < total_units ? U : -1;
}

// Persistent: each CTA walks the units of rounds r = 0, 1, ... (unit_of_round).
// Barrier phases run on across units: per-unit barriers by the unit count
// `uc`, score / P barriers by the running key-tile count of each query tile,
// ring slots by the running item count.
// kGeneral: keys per sequence may come from seqlens (attn_fwd_kvcache) and
// the mask may have a local window; otherwise every sequence has Nk keys,
// seqlens is not read and the mask is at most causal.
template <int D, bool kNeg, bool kGeneral, bool kSlotMajor>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ out,
                       float* __restrict__ lse_out, int B, int Hq, int Hkv, int Nq, int Nk, int causal,
                       int wl, int wr, const int* __restrict__ seqlens,
                       float scale_log2, int pair_heads, int units_per_bh, int total_units) {
  using L = Layout<D>;
  constexpr int NS = L::kSlots;
  const int* const lens = kGeneral ? seqlens : nullptr;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (TMA's 128-byte swizzle), taken as an offset into
  // the shared array itself: pointers derived from it stay in the shared
  // space, so the compiler emits shared loads and stores and needs no
  // generic-to-shared conversion for every barrier operation
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* bar_full = bars;              // [NS] ring slot loaded
  uint64_t* bar_empty = bar_full + NS;    // [NS] ring slot released
  uint64_t* bar_sfull = bar_empty + NS;   // [2] S_t complete
  uint64_t* bar_pfull = bar_sfull + 2;    // [2] P_t written (4 softmax warps)
  uint64_t* bar_odone = bar_pfull + 2;    // [2] last P.V of the unit into O_t complete
  uint64_t* bar_qfull = bar_odone + 2;    // [2] Q_t loaded
  uint64_t* bar_qfree = bar_qfull + 2;    // [2] last QK^T of the unit read Q_t
  uint64_t* bar_ofree = bar_qfree + 2;    // [2] epilogue read O_t out of TMEM (4 softmax warps)
  uint64_t* bar_vfix = bar_ofree + 2;     // last V tile of a cache row landed (producer only)
  uint64_t* bar_drain = bar_vfix + 1;     // after an abort: the MMAs issued so far completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_full + s, 1);
      mbar_init(bar_empty + s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_sfull + t, 1);
      mbar_init(bar_pfull + t, 4);  // one arrival per softmax warp
      mbar_init(bar_odone + t, 1);
      mbar_init(bar_qfull + t, 1);
      mbar_init(bar_qfree + t, 1);
      mbar_init(bar_ofree + t, 4);
    }
    mbar_init(bar_vfix, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  uint8_t* sQ = smem + L::kOffQ;
  uint8_t* sRing = smem + L::kOffRing;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t item_base = 0, vfix_uses = 0;
      uint32_t issued = 0;         // ring items issued so far
      int q_issued[2] = {0, 0};    // Q loads issued per tile
      bool vfix_pending = false;   // the last item's load completes on bar_vfix and was not awaited
      int uc = 0;
      bool ok = true;
      for (int rnd = 0; ok && rnd * static_cast<int>(gridDim.x) < total_units; ++rnd) {
        const int U = unit_of_round(rnd, total_units);
        if (U < 0) continue;
        const Unit u = decode_unit<kGeneral, kSlotMajor>(U, B, Hq, Hkv, Nq, Nk, causal, wl, wr, lens, pair_heads,
                                                          units_per_bh);
        if (kGeneral && lens && (lens[u.b] < 0 || lens[u.b] > Nk) && u.ti[0].hq == 0) record(11, kDevBadSeqlen);
        for (int t = 0; t < 2; ++t) {
          // Q_t of the previous unit must have been read by its last QK^T
          if (uc >= 1 && !wait_one(bar_qfree + t, (uc - 1) & 1, abort_flag, 1)) { ok = false; break; }
          mbar_arrive_expect_tx(bar_qfull + t, L::kTile);
          for (int h = 0; h < D / 64; ++h)
            tma_load_4d(sQ + t * L::kTile + h * L::kHalf, &tm_q, bar_qfull + t, h * 64, u.ti[t].hq, u.ti[t].row0,
                        u.b);
          q_issued[t] = uc + 1;
        }
        for (int item = 0; ok && item < 2 * u.n_kt; ++item) {
          const uint32_t gi = item_base + item;
          const int slot = gi % NS;
          if (gi >= NS && !wait_one(bar_empty + slot, ((gi / NS) - 1) & 1, abort_flag, 2)) { ok = false; break; }
          // item -> (K or V, key tile), the inverse of k_item / v_item
          const bool is_v = (item == 2 * u.n_kt - 1) || (item > 0 && (item & 1) == 0);
          const int kt = (item == 2 * u.n_kt - 1) ? u.n_kt - 1 : (is_v ? item / 2 - 1 : (item + 1) / 2);
          // A cache's last V tile may run past the cache length into rows that
          // hold anything, NaN included (and P = 0 times NaN is not 0): it is
          // loaded against a private barrier and those rows are cleared before
          // the MMA thread is told the tile is there.
          const int ktile = key_tile<kGeneral>(u, kt);
          const int valid = u.nk - ktile * BN;
          const bool fix = kGeneral && lens && is_v && valid < BN;
          uint64_t* done = fix ? bar_vfix : bar_full + slot;
          mbar_arrive_expect_tx(done, L::kTile);
          for (int h = 0; h < D / 64; ++h)
            tma_load_4d(sRing + slot * L::kTile + h * L::kHalf, is_v ? &tm_v : &tm_k, done, h * 64, u.hkv,
                        ktile * BN, u.b);
          issued = gi + 1;
          if (fix) {
            if (!wait_one(bar_vfix, vfix_uses & 1, abort_flag, 12)) {
              vfix_pending = true;
              ok = false;
              break;
            }
            ++vfix_uses;
            for (int h = 0; h < D / 64; ++h) {
              uint8_t* base = sRing + slot * L::kTile + h * L::kHalf;
              for (int off = max(valid, 0) * 128; off < BN * 128; off += 16)
                *reinterpret_cast<uint4*>(base + off) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();  // the generic stores before the tensor core's reads
            mbar_arrive(bar_full + slot);
          }
        }
        item_base += 2 * u.n_kt;
        ++uc;
      }
      if (!ok) {
        // after an abort, loads already issued may still be in flight: they
        // land before the CTA may exit (bounded, not abortable).  Only the
        // last item of each ring slot can be pending.
        volatile int no_abort = 0;
        for (int t = 0; t < 2; ++t)
          if (q_issued[t] > 0) mbar_wait(bar_qfull + t, (q_issued[t] - 1) & 1, &no_abort, kWaitLimitNs);
        for (int s = 0; s < NS && static_cast<uint32_t>(s) < issued; ++s) {
          const uint32_t last = s + NS * ((issued - 1 - s) / NS);
          if (vfix_pending && last == issued - 1) continue;  // completes on bar_vfix instead
          mbar_wait(bar_full + s, (last / NS) & 1, &no_abort, kWaitLimitNs);
        }
        if (vfix_pending) mbar_wait(bar_vfix, vfix_uses & 1, &no_abort, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, 1);
      // Descriptors are built once; an offset of X bytes is X >> 4 added to
      // the start-address field (no carry: shared addresses stay below 2^18).
      const uint64_t dQ = sdesc_sw128(smem_u32(sQ), 16, 1024);          // Q_t, K tiles: K-major
      const uint64_t dK = sdesc_sw128(smem_u32(sRing), 16, 1024);
      const uint64_t dV = sdesc_sw128(smem_u32(sRing), L::kHalf, 1024);  // V tiles: MN-major
      uint32_t item_base = 0;
      int kc[2] = {0, 0};  // key tiles done per query tile (score / P barrier phases)
      int uc = 0;
      bool ok = true;
      for (int rnd = 0; ok && rnd * static_cast<int>(gridDim.x) < total_units; ++rnd) {
        const int U = unit_of_round(rnd, total_units);
        if (U < 0) continue;
        const Unit u = decode_unit<kGeneral, kSlotMajor>(U, B, Hq, Hkv, Nq, Nk, causal, wl, wr, lens, pair_heads,
                                                          units_per_bh);
        const int n_kt = u.n_kt;
        for (int t = 0; t < 2 && ok; ++t) {
          ok = wait_one(bar_qfull + t, uc & 1, abort_flag, 3);
          if (ok && u.ti[t].n_kt == 0) {
            // nothing to compute for this tile: hand its per-unit barriers on
            if (uc >= 1) ok = wait_one(bar_ofree + t, (uc - 1) & 1, abort_flag, 9);
            mma_commit(bar_qfree + t);
            mma_commit(bar_odone + t);
          }
        }
        if (ok && n_kt > 0) ok = wait_one(bar_full + item_base % NS, (item_base / NS) & 1, abort_flag, 4);  // K_0
        // Steps 2 .. n_both-2, where both tiles do P.V and QK^T and no per-unit
        // barrier is due, run in a branch-free loop (below); the others in the
        // general form.  Every instruction of this thread between two MMA
        // batches leaves the tensor core idle, so the loop keeps ring positions
        // and barrier parities incrementally and probes the barriers it will
        // wait on next (K_{j+1}, P_1, then the next step's V_j and P_0) right
        // after issuing a batch, while the queued MMAs still run; a barrier
        // found complete is not waited on again.
        const int n_both = min(u.ti[0].n_kt, u.ti[1].n_kt);
        const int j_steady_end = n_both - 2;
        for (int j = 0; ok && j <= n_kt;) {
          if (j >= 2 && j <= j_steady_end) {
            // ring items: K_j = g, V_{j-1} = g+1, K_{j+1} = g+2, V_j = g+3.
            // V_{j-1} was loaded only after S_1(j-2) was complete, so it is
            // awaited right before its first use, a step after the general
            // form would; K_{j+1} is awaited after tile 0's MMAs.
            const uint32_t g = item_base + 2 * j - 1;
            int s0 = static_cast<int>(g % NS);
            uint32_t ph0 = (g / NS) & 1u;
            uint32_t pp0 = static_cast<uint32_t>(kc[0] + j - 1) & 1u;
            uint32_t pp1 = static_cast<uint32_t>(kc[1] + j - 1) & 1u;
            bool v_ready = false, p0_ready = false;  // probed during the previous step
            for (; j <= j_steady_end; ++j) {
              int s1 = s0 + 1;
              uint32_t ph1 = ph0;
              if (s1 >= NS) { s1 -= NS; ph1 ^= 1u; }
              int s2 = s1 + 1;
              uint32_t ph2 = ph1;
              if (s2 >= NS) { s2 -= NS; ph2 ^= 1u; }
              int s3 = s2 + 1;
              uint32_t ph3 = ph2;
              if (s3 >= NS) { s3 -= NS; ph3 ^= 1u; }
              const uint64_t dv = dV + static_cast<uint64_t>((s1 * L::kTile) >> 4);
              const uint64_t db = dK + static_cast<uint64_t>((s0 * L::kTile) >> 4);
              if (!v_ready && !wait_one(bar_full + s1, ph1, abort_flag, 5)) { ok = false; break; }
              if (!p0_ready && !wait_one(bar_pfull + 0, pp0, abort_flag, 6)) { ok = false; break; }
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < BN / 16; ++kk)
                mma_bf16_ts(tmem + 256, tmem + kk * 8, dv + ((kk * 16 * 128) >> 4), idesc_pv, 1u);
              const bool k_ready = mbar_test_wait(bar_full + s2, ph2);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * L::kHalf + (kk & 3) * 32) >> 4;
                mma_bf16_ss(tmem, dQ + off, db + off, idesc_qk, kk > 0 ? 1u : 0u);
              }
              mma_commit(bar_sfull + 0);
              const bool p1_ready = mbar_test_wait(bar_pfull + 1, pp1);
              if (!k_ready && !wait_one(bar_full + s2, ph2, abort_flag, 4)) { ok = false; break; }
              if (!p1_ready && !wait_one(bar_pfull + 1, pp1, abort_flag, 6)) { ok = false; break; }
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < BN / 16; ++kk)
                mma_bf16_ts(tmem + 384, tmem + 128 + kk * 8, dv + ((kk * 16 * 128) >> 4), idesc_pv, 1u);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * L::kHalf + (kk & 3) * 32) >> 4;
                mma_bf16_ss(tmem + 128, dQ + ((L::kTile) >> 4) + off, db + off, idesc_qk, kk > 0 ? 1u : 0u);
              }
              mma_commit(bar_sfull + 1);
              mma_commit(bar_empty + s1);  // V_{j-1}: both P.V done
              mma_commit(bar_empty + s0);  // K_j: both QK^T done
              v_ready = mbar_test_wait(bar_full + s3, ph3);
              p0_ready = mbar_test_wait(bar_pfull + 0, pp0 ^ 1u);
              s0 = s2;
              ph0 = ph2;
              pp0 ^= 1u;
              pp1 ^= 1u;
            }
            if (ok) {
              // the general form expects V_{j-1} (the item after K_j) to have
              // been awaited in step j-1
              int s1 = s0 + 1;
              uint32_t ph1 = ph0;
              if (s1 >= NS) { s1 -= NS; ph1 ^= 1u; }
              ok = wait_one(bar_full + s1, ph1, abort_flag, 5);
            }
            continue;
          }
          const uint32_t ki = item_base + k_item(j), vi = item_base + (j >= 1 ? v_item(j - 1, n_kt) : 0);
          const int ks = ki % NS, vs = vi % NS;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int n_t = u.ti[t].n_kt;
            const uint32_t tS = tmem + t * 128;
            const uint32_t tO = tmem + 256 + t * 128;
            if (j >= 1 && j - 1 < n_t) {
              // O_t += P_t V_{j-1}; P_t sits in the first 64 columns of S_t
              if (!wait_one(bar_pfull + t, (kc[t] + j - 1) & 1, abort_flag, 6)) { ok = false; break; }
              // the first P.V of a unit overwrites O_t: the previous epilogue must have read it
              if (j == 1 && uc >= 1 && !wait_one(bar_ofree + t, (uc - 1) & 1, abort_flag, 9)) { ok = false; break; }
              tc_fence_after();
              const uint64_t dv = dV + static_cast<uint64_t>((vs * L::kTile) >> 4);
#pragma unroll
              for (int kk = 0; kk < BN / 16; ++kk)
                mma_bf16_ts(tO, tS + kk * 8, dv + ((kk * 16 * 128) >> 4), idesc_pv, (j - 1 > 0 || kk > 0) ? 1u : 0u);
              if (j == n_t) mma_commit(bar_odone + t);
              // the last P.V of the step: V_{j-1}'s slot is free once it completes
              if (t == 1 || j - 1 >= u.ti[1].n_kt) mma_commit(bar_empty + vs);
            }
            if (j < n_t) {
              // S_t = Q_t K_j^T (after the P.V that read P_t: MMAs run in issue order)
              const uint64_t da = dQ + static_cast<uint64_t>((t * L::kTile) >> 4);
              const uint64_t db = dK + static_cast<uint64_t>((ks * L::kTile) >> 4);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * L::kHalf + (kk & 3) * 32) >> 4;
                mma_bf16_ss(tS, da + off, db + off, idesc_qk, kk > 0 ? 1u : 0u);
              }
              mma_commit(bar_sfull + t);
              if (j == n_t - 1) mma_commit(bar_qfree + t);
              // the last QK^T of the step: K_j's slot is free once it completes
              if (t == 1 || j >= u.ti[1].n_kt) mma_commit(bar_empty + ks);
            }
            if (t == 0) {
              // the operands of step j+1 (K_{j+1}, V_j), awaited while the tensor
              // core still has this step's tile-0 MMAs queued
              if (j + 1 < n_kt) {
                const uint32_t kn = item_base + k_item(j + 1);
                if (!wait_one(bar_full + kn % NS, (kn / NS) & 1, abort_flag, 4)) { ok = false; break; }
              }
              if (j < n_kt) {
                const uint32_t vn = item_base + v_item(j, n_kt);
                if (!wait_one(bar_full + vn % NS, (vn / NS) & 1, abort_flag, 5)) { ok = false; break; }
              }
            }
          }
          ++j;
        }
        kc[0] += u.ti[0].n_kt;
        kc[1] += u.ti[1].n_kt;
        item_base += 2 * n_kt;
        ++uc;
      }
      if (!ok) {
        // after an abort, the MMAs issued so far complete before TMEM is freed
        volatile int no_abort = 0;
        mma_commit(bar_drain);
        mbar_wait(bar_drain, 0, &no_abort, kWaitLimitNs);
      }
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax + epilogue
    const int t = (warp - 4) >> 2;  // query tile of this warpgroup
    const int quarter = warp & 3;  // TMEM lanes this warp may touch: 32*quarter .. +31
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + t * 128 + lane_off;
    const uint32_t tO = tmem + 256 + t * 128 + lane_off;
    // with a negative scale the kernel works on -s with |c| (kNeg), so the
    // max logic is the same
    const float c = kNeg ? -scale_log2 : scale_log2;
    const bool o_32b_aligned = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
    int kc = 0, uc = 0;
    bool ok = true;
    for (int rnd = 0; ok && rnd * static_cast<int>(gridDim.x) < total_units; ++rnd) {
      const int U = unit_of_round(rnd, total_units);
      if (U < 0) continue;
      const Unit u = decode_unit<kGeneral, kSlotMajor>(U, B, Hq, Hkv, Nq, Nk, causal, wl, wr, lens, pair_heads,
                                                          units_per_bh);
      const TileInfo me = t ? u.ti[1] : u.ti[0];
      const int grow = me.row0 + r;
      const int my_kt = me.n_kt;
      float m = -INFINITY;  // exponent reference of this row (sign-adjusted raw score units)
      float l = 0.f;        // running sum of 2^(s*c - m*c)
      for (int j = 0; j < my_kt; ++j) {
        if (!wait_all(bar_sfull + t, (kc + j) & 1, abort_flag, 7)) { ok = false; break; }
        tc_fence_after();
        const int kbase = key_tile<kGeneral>(u, j) * BN;
        bool masked;
        int lim = BN, lo = 0;  // columns outside [lo, lim) of this tile are masked for this row
        if (kGeneral) {
          masked = (kbase + BN > u.nk) || (kbase + BN - 1 > me.row0 + u.coff) || (kbase < me.row0 + BM - 1 + u.lo);
          if (masked) {
            lim = min(u.nk - kbase, grow + u.coff - kbase + 1);
            lo = grow + u.lo - kbase;
          }
        } else {
          masked = (kbase + BN > u.nk) || (causal && kbase + BN - 1 > me.row0 + u.coff);
          if (masked) {
            lim = u.nk - kbase;
            if (causal) lim = min(lim, grow + u.coff - kbase + 1);
          }
        }
        bool need;
        float m_new, alpha;
        if (__any_sync(0xffffffffu, m == -INFINITY)) {
          // some row of the warp sees its first scores: the tile max sets the
          // reference, which then moves only when a tile max is more than
          // 2^kRescaleLog2 above it
          const float mt = masked ? score_tile_max<true, kNeg, kGeneral>(tS, lo, lim)
                                  : score_tile_max<false, kNeg>(tS, lo, lim);
          need = (m == -INFINITY) || ((mt - m) * c > kRescaleLog2);
          m_new = need ? fmaxf(m, mt) : m;
          const float mc = (m_new == -INFINITY) ? 0.f : m_new * c;
          alpha = (m == -INFINITY) ? 0.f : (need ? ex2_approx(fmaf(m, c, -mc)) : 1.f);
          const float rowsum = masked ? score_tile_exp<true, kNeg, kGeneral>(tS, lo, lim, c, mc)
                                      : score_tile_exp<false, kNeg>(tS, lo, lim, c, mc);
          l = l * alpha + rowsum;
        } else {
          // no max between the scores and the exponentials on the path to P
          m_new = m;
          const float rowsum = masked ? score_tile_onepass<true, kNeg, kGeneral>(tS, lo, lim, c, m_new)
                                      : score_tile_onepass<false, kNeg>(tS, lo, lim, c, m_new);
          need = m_new != m;
          alpha = need ? ex2_approx(fmaf(m, c, -m_new * c)) : 1.f;
          l = l * alpha + rowsum;
        }

        // O_t holds the sum through tile j-1 (P.V of j-1 completed before S_j was
        // written): rescale it now if this row's reference moved.
        if (j > 0 && __any_sync(0xffffffffu, need && m != -INFINITY)) {
          const float a = (need && m != -INFINITY) ? alpha : 1.f;
          const float2 a2 = make_float2(a, a);
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t w[32];
            tmem_ld32(tO + cc * 32, w);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 x = fmul2(make_float2(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1])), a2);
              w[2 * i] = __float_as_uint(x.x);
              w[2 * i + 1] = __float_as_uint(x.y);
            }
            tmem_st32(tO + cc * 32, w);
          }
        }
        m = m_new;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_pfull + t);
      }
      if (!ok) break;

      // ---------------------------------------------------------------- epilogue
      if (!wait_all(bar_odone + t, uc & 1, abort_flag, 8)) { ok = false; break; }
      tc_fence_after();
      const bool store = me.row0 < Nq && grow < Nq;
      __nv_bfloat16* orow = out + ((static_cast<size_t>(u.b) * Nq + grow) * Hq + me.hq) * D;
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t w32[32];
        if (my_kt > 0) {
          tmem_ld32(tO + cc * 32, w32);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) w32[i] = 0u;
        }
        if (cc == D / 32 - 1) {
          // O_t has been read out of TMEM: the next unit's first P.V may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_ofree + t);
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(w32[2 * i]) * inv_l, __uint_as_float(w32[2 * i + 1]) * inv_l);
        if (store) {
          if (o_32b_aligned) {  // 32-byte stores: a warp writes 32 full sectors per instruction
            st_global_v8(orow + cc * 32, w);
            st_global_v8(orow + cc * 32 + 16, w + 8);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
      }
      if (store) {
        const float lse = (l > 0.f) ? (m * c + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        lse_out[(static_cast<size_t>(u.b) * Hq + me.hq) * Nq + grow] = lse;
      }
      kc += my_kt;
      ++uc;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_d(const PrefillParams& p, cudaStream_t stream) {
  using L = Layout<D>;
  const int n_qtiles = (p.Nq + BM - 1) / BM;
  const int G = p.Hq / p.Hkv;
  const int pair_heads = (G % 2 == 0) ? 1 : 0;
  const int units_per_bh = pair_heads ? n_qtiles : (n_qtiles + 1) / 2;
  const int hslots = pair_heads ? p.Hq / 2 : p.Hq;
  const long long total = static_cast<long long>(units_per_bh) * p.B * hslots;
  if (total == 0) return cudaSuccess;
  if (total > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  int dev = 0, n_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(total < n_sm ? total : n_sm);  // one persistent CTA per SM
  const bool general = p.seqlens || p.window_left >= 0 || p.window_right >= 0;
  const bool neg = p.scale_log2 < 0.f;
  auto kern = general        ? (neg ? prefill_fwd_kernel<D, true, true, false> : prefill_fwd_kernel<D, false, true, false>)
              : p.causal == 0 ? (neg ? prefill_fwd_kernel<D, true, false, true> : prefill_fwd_kernel<D, false, false, true>)
                              : (neg ? prefill_fwd_kernel<D, true, false, false> : prefill_fwd_kernel<D, false, false, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, L::kAlloc, stream>>>(p.tm_q, p.tm_k, p.tm_v, static_cast<__nv_bfloat16*>(p.o), p.lse, p.B,
                                              p.Hq, p.Hkv, p.Nq, p.Nk, p.causal, p.window_left, p.window_right,
                                              p.seqlens, p.scale_log2, pair_heads,
                                              units_per_bh, static_cast<int>(total));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream) {
  if (p.d == 64) return launch_d<64>(p, stream);
  if (p.d == 128) return launch_d<128>(p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t fetch_status_prefill(cudaStream_t stream, uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_prefill_status, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_prefill_status, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

}  // namespace attn
