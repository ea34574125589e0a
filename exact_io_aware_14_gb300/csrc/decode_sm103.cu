// Query-length-one decode against a KV cache, split over the key axis, for
// sm_103a (pyshine.com flash-attention tour, "Why You Need This": with one
// query the cache is split across thread blocks and the partial results are
// combined).
//
// Split kernel: one CTA (8 warps) per (split of `chunk` keys, KV head, block
// of up to 4 query heads of that KV head's group, batch).  K/V tiles of 64
// keys stream through a 3-stage TMA ring; each K and V byte is read once per
// CTA and serves every query head of the block.  The warps are specialised
// and hand tiles over through mbarriers (no block-wide barrier in the loop),
// so the scores of tile t+1 overlap the P.V of tile t:
//   warps 0-3  scores: 8 threads per key, each owning 16 of the 128 head dims
//              of the 4 query heads (q held in registers), packed fp32x2 FMAs
//              and a 3-level shuffle reduction; then one warp per head runs
//              the online softmax (exponent reference moved only when the max
//              rises by more than 2^8, as in the prefill kernel) and writes
//              P.
//   warps 4-7  P.V: each thread owns 4 output dims of the 4 heads for a
//              quarter of the keys, packed fp32x2 FMAs.  Lane 0 of warp 4
//              issues the TMA loads, refilling a stage as soon as its P.V is
//              done.
// The CTA writes its split's normalised partial output and natural-log LSE.
// Decode is memory-bound ("FlashAttention: Part 2", section 4.1): the kernel
// exists to keep ~128 KB of loads in flight per SM with few instructions per
// byte.
//
// Combine kernel: LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s;
// launched as a programmatic dependent of the split kernel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace {

__device__ uint32_t g_decode_status;

constexpr int KT = 64;        // keys per tile
constexpr int HPC = 4;        // query heads per CTA
constexpr int kThreads = 256;
constexpr int kScoreThreads = 128;  // warps 0-3
constexpr int kStages = 3;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kRescaleLog2 = 8.f;  // see the prefill kernel

template <int D>
struct DLayout {
  static constexpr int kHalf = KT * 128;  // one 64-column box: 64 rows x 128 B
  static constexpr int kTile = KT * D * 2;
  static constexpr int kDQ = D / 4;                       // 4-dim groups per row (P.V role)
  static constexpr int kNG = 128 / kDQ;                   // key groups in the P.V role
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kStages * kTile;
  static constexpr int kOffS = kOffV + kStages * kTile;   // float [2][HPC][KT]
  static constexpr int kOffP = kOffS + 2 * HPC * KT * 4;  // float [2][KT][HPC]
  static constexpr int kOffA = kOffP + 2 * KT * HPC * 4;  // float [2][HPC] alpha
  static constexpr int kOffRed = kOffA + 2 * HPC * 4;     // float [kNG][HPC][D]
  static constexpr int kOffML = kOffRed + kNG * HPC * D * 4;  // float m[HPC], l[HPC], abort flag
  static constexpr int kOffBar = kOffML + 2 * HPC * 4 + 16;   // full[kStages], pfull[2], pfree[2]
  static constexpr int kBytes = kOffBar + (kStages + 4) * 8 + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

__device__ __forceinline__ void record(uint32_t site, uint32_t code) {
  atomicCAS(&g_decode_status, 0u, (site << 8) | code);
}

// warp-uniform bounded wait
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  bool ok = mbar_wait(bar, parity, abort_flag, kWaitLimitNs);
  return __all_sync(0xffffffffu, ok);
}

// barrier over the score warps (named barrier 1) that also ORs a flag
__device__ __forceinline__ bool score_bar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(kScoreThreads)
      : "memory");
  return r != 0;
}

// Work order for up to kRankB sequences: the CTAs (in launch order) take
// every sequence's full splits first and the shorter last splits after them,
// longest first, so the last CTAs to start are the shortest.  Warp 0 lists
// the splits from seqlens (lanes hold sequences lane and lane+32) and picks
// item i; returns (b, split), or b = -1 when i is past the last split.
constexpr int kRankB = 64;
__device__ __forceinline__ int2 pick_item(const int* __restrict__ seqlens, int B, int max_seqlen, int chunk, int i,
                                          int lane) {
  int nf[2], rem[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int b = lane + 32 * k;
    int v = b < B ? seqlens[b] : 0;
    v = v < 0 ? 0 : (v > max_seqlen ? max_seqlen : v);
    nf[k] = v / chunk;
    rem[k] = v % chunk;
  }
  // full splits, sequence after sequence: exclusive prefix of nf over b
  int incl0 = nf[0], incl1 = nf[1];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y0 = __shfl_up_sync(0xffffffffu, incl0, o), y1 = __shfl_up_sync(0xffffffffu, incl1, o);
    if (lane >= o) {
      incl0 += y0;
      incl1 += y1;
    }
  }
  const int tot0 = __shfl_sync(0xffffffffu, incl0, 31);
  incl1 += tot0;
  const int n_full = __shfl_sync(0xffffffffu, incl1, 31);
  int2 r = make_int2(-1, 0);
  if (i < n_full) {
    if (incl0 - nf[0] <= i && i < incl0) r = make_int2(lane, i - (incl0 - nf[0]));
    if (incl1 - nf[1] <= i && i < incl1) r = make_int2(lane + 32, i - (incl1 - nf[1]));
  } else {
    // last splits shorter than the chunk, ranked by length (longest first), then b
    const int j = i - n_full;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      int rank = 0;
      for (int b2 = 0; b2 < B; ++b2) {
        const int r2 = __shfl_sync(0xffffffffu, rem[b2 >> 5], b2 & 31);
        rank += (r2 > rem[k] || (r2 == rem[k] && b2 < lane + 32 * k)) ? 1 : 0;
      }
      if (rem[k] > 0 && rank == j) r = make_int2(lane + 32 * k, nf[k]);
    }
  }
  // the (single) lane that found the item broadcasts it
  const unsigned found = __ballot_sync(0xffffffffu, r.x >= 0);
  if (found == 0u) return make_int2(-1, 0);
  const int src = __ffs(found) - 1;
  return make_int2(__shfl_sync(0xffffffffu, r.x, src), __shfl_sync(0xffffffffu, r.y, src));
}

// Paged cache: the pages of one split, at most this many.
constexpr int kMaxSplitPages = 128;

// kPaged: K/V live in pages [num_pages, page_size, Hkv, d]; key k of sequence
// b is row k % page_size of page block_table[b * max_blocks + k / page_size]
// (page_size a multiple of the 64-key tile, so a tile never spans pages).
template <int D, bool kPaged>
__global__ void __launch_bounds__(kThreads, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const __nv_bfloat16* __restrict__ q, const int* __restrict__ seqlens, int max_seqlen,
                        int Hq, int Hkv, int chunk, int n_split, float scale_log2, float* __restrict__ o_part,
                        float* __restrict__ lse_part, const int* __restrict__ block_table, int max_blocks,
                        int page_size, int num_pages) {
  using L = DLayout<D>;
  constexpr int NCH = D / 64;  // 16-byte chunks per key that one score thread reads
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (TMA's 128-byte swizzle), taken as an offset into
  // the shared array itself: pointers derived from it stay in the shared
  // space, so the compiler emits shared loads and stores and needs no
  // generic-to-shared conversion for every barrier operation
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  // grid (KV head x head block, batch, split).  Up to kRankB sequences the
  // CTA with linear item index (z, y) takes the item pick_item lists there;
  // beyond that, splits are launched highest first (only long sequences
  // have high splits, and every sequence's low splits are full chunks).
  const int G = Hq / Hkv;
  const int n_hblk = (G + HPC - 1) / HPC;
  const int hkv = blockIdx.x / n_hblk;
  const int hb = blockIdx.x % n_hblk;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // the combine kernel may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int B = gridDim.y;
  int b = blockIdx.y, split = n_split - 1 - blockIdx.z;
  if (B <= kRankB) {
    __shared__ int2 s_item;
    if (warp == 0) {
      const int2 it = pick_item(seqlens, B, max_seqlen, chunk, blockIdx.z * B + blockIdx.y, lane);
      if (lane == 0) s_item = it;
    }
    __syncthreads();
    b = s_item.x;
    split = s_item.y;
    if (b < 0) return;  // past the last split
  }
  int Lb = seqlens[b];
  if (Lb < 0 || Lb > max_seqlen) {
    if (tid == 0 && blockIdx.x == 0) record(1, kDevBadSeqlen);
    Lb = Lb < 0 ? 0 : max_seqlen;
  }
  const int k0 = split * chunk;
  if (k0 >= Lb) return;  // empty split: the combine never reads it
  const int kn = min(chunk, Lb - k0);
  const int n_t = (kn + KT - 1) / KT;
  const int hq0 = hkv * G + hb * HPC;
  const int nh = min(HPC, G - hb * HPC);

  float* sS = reinterpret_cast<float*>(smem + L::kOffS);
  float* sP = reinterpret_cast<float*>(smem + L::kOffP);
  float* sAlpha = reinterpret_cast<float*>(smem + L::kOffA);
  float* sRed = reinterpret_cast<float*>(smem + L::kOffRed);
  float* sM = reinterpret_cast<float*>(smem + L::kOffML);
  float* sL = sM + HPC;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffML + 2 * HPC * 4);
  uint64_t* bar_full = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* bar_pfull = bar_full + kStages;  // [2] P of a tile written (4 score warps)
  uint64_t* bar_pfree = bar_pfull + 2;       // [2] P.V of a tile done (4 P.V warps)
  uint8_t* sK = smem + L::kOffK;
  uint8_t* sV = smem + L::kOffV;

  // pages of this split (paged cache): read once, before the barrier below
  __shared__ int s_pages[kPaged ? kMaxSplitPages : 1];
  const int p0 = kPaged ? k0 / page_size : 0;
  if (kPaged) {
    const int n_pg = (k0 + kn - 1) / page_size - p0 + 1;  // <= kMaxSplitPages (checked on the host)
    for (int i = tid; i < n_pg; i += kThreads) {
      int pg = block_table[static_cast<size_t>(b) * max_blocks + p0 + i];
      if (pg < 0 || pg >= num_pages) {
        record(6, kDevBadPage);
        pg = 0;  // keep every load inside the page pool; the result is flagged
      }
      s_pages[i] = pg;
    }
  }

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bar_full + s, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_pfull + i, 4);
      mbar_init(bar_pfree + i, 4);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();

  const bool negate = scale_log2 < 0.f;
  const float c = negate ? -scale_log2 : scale_log2;

  // Loads are issued by lane 0 of warp 4 (the first P.V warp): the first
  // kStages tiles now, then each stage again as soon as its P.V is done.
  auto issue = [&](int t) {
    const int s = t % kStages;
    const int key = k0 + t * KT;
    // (row, outer index) of the tile: (key, b), or (row in page, page) when paged
    const int row = kPaged ? key % page_size : key;
    const int outer = kPaged ? s_pages[key / page_size - p0] : b;
    mbar_arrive_expect_tx(bar_full + s, 2 * L::kTile);
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      tma_load_4d(sK + s * L::kTile + h * L::kHalf, &tm_k, bar_full + s, h * 64, hkv, row, outer);
      tma_load_4d(sV + s * L::kTile + h * L::kHalf, &tm_v, bar_full + s, h * 64, hkv, row, outer);
    }
  };
  const bool loader = (tid == kScoreThreads);
  int n_issued = 0;  // meaningful in the loader only
  if (loader) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    for (int t = 0; t < n_t && t < kStages; ++t) issue(t);
    n_issued = min(n_t, kStages);
  }

  if (warp < 4) {
    // ================================================================ scores + softmax
    // key slot ks (keys ks, ks+16, ks+32, ks+48), 16-byte chunk dseg of each
    // 64-column half of the key row
    const int ks = tid >> 3;
    const int dseg = tid & 7;
    float qf[HPC][NCH * 8];  // this thread's dims of the 4 query heads (0 for missing heads)
#pragma unroll
    for (int h = 0; h < HPC; ++h) {
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        uint4 raw = make_uint4(0u, 0u, 0u, 0u);
        if (h < nh)
          raw = *reinterpret_cast<const uint4*>(q + (static_cast<size_t>(b) * Hq + hq0 + h) * D + 64 * cc + 8 * dseg);
        qf[h][8 * cc + 0] = bf16lo(raw.x); qf[h][8 * cc + 1] = bf16hi(raw.x);
        qf[h][8 * cc + 2] = bf16lo(raw.y); qf[h][8 * cc + 3] = bf16hi(raw.y);
        qf[h][8 * cc + 4] = bf16lo(raw.z); qf[h][8 * cc + 5] = bf16hi(raw.z);
        qf[h][8 * cc + 6] = bf16lo(raw.w); qf[h][8 * cc + 7] = bf16hi(raw.w);
      }
    }
    float m = -INFINITY, l = 0.f;  // reference of head `warp`; this lane's part of its sum
    for (int t = 0; t < n_t; ++t) {
      const int s = t % kStages;
      const int buf = t & 1;
      const bool got = wait_all(bar_full + s, (t / kStages) & 1, abort_flag);
      const int valid = min(KT, kn - t * KT);
      const uint32_t kbase = smem_u32(sK + s * L::kTile);
      const uint32_t vbase = smem_u32(sV + s * L::kTile);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int key = ks + 16 * kk;
        float2 a[HPC];
#pragma unroll
        for (int h = 0; h < HPC; ++h) a[h] = make_float2(0.f, 0.f);
#pragma unroll
        for (int cc = 0; cc < NCH; ++cc) {
          const uint4 kv = ld_shared_v4(kbase + cc * L::kHalf + key * 128 + ((dseg ^ (key & 7)) << 4));
          const float2 k01 = make_float2(bf16lo(kv.x), bf16hi(kv.x)), k23 = make_float2(bf16lo(kv.y), bf16hi(kv.y));
          const float2 k45 = make_float2(bf16lo(kv.z), bf16hi(kv.z)), k67 = make_float2(bf16lo(kv.w), bf16hi(kv.w));
#pragma unroll
          for (int h = 0; h < HPC; ++h) {
            a[h] = ffma2(make_float2(qf[h][8 * cc + 0], qf[h][8 * cc + 1]), k01, a[h]);
            a[h] = ffma2(make_float2(qf[h][8 * cc + 2], qf[h][8 * cc + 3]), k23, a[h]);
            a[h] = ffma2(make_float2(qf[h][8 * cc + 4], qf[h][8 * cc + 5]), k45, a[h]);
            a[h] = ffma2(make_float2(qf[h][8 * cc + 6], qf[h][8 * cc + 7]), k67, a[h]);
          }
        }
        float v[HPC];
#pragma unroll
        for (int h = 0; h < HPC; ++h) v[h] = a[h].x + a[h].y;
        // reduce the 4 head sums over the 8 threads of this key: after the
        // first two levels lane bit 2 selects heads {0,1}/{2,3} and bit 1 the head
        const bool hi2 = dseg & 4;
        const float s0 = hi2 ? v[0] : v[2], s1 = hi2 ? v[1] : v[3];
        const float r0 = __shfl_xor_sync(0xffffffffu, s0, 4), r1 = __shfl_xor_sync(0xffffffffu, s1, 4);
        const float w0 = (hi2 ? v[2] : v[0]) + r0, w1 = (hi2 ? v[3] : v[1]) + r1;
        const bool hi1 = dseg & 2;
        const float r2 = __shfl_xor_sync(0xffffffffu, hi1 ? w0 : w1, 2);
        float w = (hi1 ? w1 : w0) + r2;
        w += __shfl_xor_sync(0xffffffffu, w, 1);
        if ((dseg & 1) == 0) {
          const int head = ((dseg >> 2) & 1) * 2 + ((dseg >> 1) & 1);
          sS[(buf * HPC + head) * KT + key] = (key < valid) ? (negate ? -w : w) : -INFINITY;
        }
      }
      // all scores of the tile written; the abort decision is made together
      if (score_bar_or(!got || *abort_flag)) {
        if (tid == 0) record(2, kDevTimeout);
        *abort_flag = 1;
        break;
      }
      // P buffer `buf` is free once the P.V of tile t-2 is done.  A failed
      // wait only raises the flag: the score warps leave the loop together at
      // the next score barrier, so none is left waiting there.
      if (t >= 2 && !wait_all(bar_pfree + buf, ((t - 2) >> 1) & 1, abort_flag)) {
        if (lane == 0) record(3, kDevTimeout);
      }
      // online softmax of head `warp` over this tile's 64 scores.  The
      // reference only has to move when a score exceeds it by more than
      // 2^kRescaleLog2, which each lane checks for its own two scores (one
      // vote); only then is the tile max formed.  Each lane keeps its own part
      // of the sum l; the parts are added once, at the end of the split.
      {
        const float x0 = sS[(buf * HPC + warp) * KT + lane], x1 = sS[(buf * HPC + warp) * KT + lane + 32];
        const float mc_old = (m == -INFINITY) ? 0.f : m * c;
        const bool big = (m == -INFINITY) || (fmaf(x0, c, -mc_old) > kRescaleLog2) ||
                         (fmaf(x1, c, -mc_old) > kRescaleLog2);
        float alpha = 1.f;
        float mc = mc_old;
        if (__any_sync(0xffffffffu, big)) {
          float mt = fmaxf(x0, x1);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
          const bool need = (m == -INFINITY) || ((mt - m) * c > kRescaleLog2);
          const float m_new = need ? fmaxf(m, mt) : m;
          mc = (m_new == -INFINITY) ? 0.f : m_new * c;
          alpha = (m == -INFINITY) ? 0.f : (need ? ex2_approx(fmaf(m, c, -mc)) : 1.f);
          l *= alpha;
          m = m_new;
        }
        float p0 = ex2_approx(fmaf(x0, c, -mc)), p1 = ex2_approx(fmaf(x1, c, -mc));
        p0 = (lane < valid) ? p0 : 0.f;  // also right for c == 0
        p1 = (lane + 32 < valid) ? p1 : 0.f;
        l += p0 + p1;
        sP[(buf * KT + lane) * HPC + warp] = p0;
        sP[(buf * KT + lane + 32) * HPC + warp] = p1;
        if (lane == 0) sAlpha[buf * HPC + warp] = alpha;
      }
      if (valid < KT) {
        // rows past the cache length may hold anything (NaN): zero them in V so
        // that p = 0 contributes exactly nothing
        for (int idx = tid; idx < (KT - valid) * (D / 8); idx += kScoreThreads) {
          const int row = valid + idx / (D / 8), cc = idx % (D / 8);
          st_shared_v4(vbase + (cc >> 3) * L::kHalf + row * 128 + (((cc & 7) ^ (row & 7)) << 4), 0u, 0u, 0u, 0u);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pfull + buf);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) {
      sM[warp] = m;
      sL[warp] = l;
    }
  } else {
    // ================================================================ P.V
    const int ptid = tid - kScoreThreads;
    const int dq = ptid % L::kDQ;  // dims 4dq .. 4dq+3
    const int grp = ptid / L::kDQ;  // keys grp, grp + kNG, ...
    const int col = 4 * dq;
    const int cbyte = (col & 63) * 2;  // byte offset inside a 128-B half row (8-byte aligned)
    float2 acc[HPC][2];
#pragma unroll
    for (int h = 0; h < HPC; ++h) acc[h][0] = acc[h][1] = make_float2(0.f, 0.f);
    for (int t = 0; t < n_t; ++t) {
      const int s = t % kStages;
      const int buf = t & 1;
      if (!wait_all(bar_pfull + buf, (t >> 1) & 1, abort_flag)) break;
      const float4 al = *reinterpret_cast<const float4*>(sAlpha + buf * HPC);
      if (al.x != 1.f || al.y != 1.f || al.z != 1.f || al.w != 1.f) {
        const float alv[HPC] = {al.x, al.y, al.z, al.w};
#pragma unroll
        for (int h = 0; h < HPC; ++h) {
          acc[h][0] = fmul2(acc[h][0], make_float2(alv[h], alv[h]));
          acc[h][1] = fmul2(acc[h][1], make_float2(alv[h], alv[h]));
        }
      }
      const uint32_t vcol = smem_u32(sV + s * L::kTile) + (col >> 6) * L::kHalf + (cbyte & 15);
#pragma unroll
      for (int jj = 0; jj < KT / L::kNG; ++jj) {
        const int j = jj * L::kNG + grp;
        uint32_t v0, v1;
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                     : "=r"(v0), "=r"(v1)
                     : "r"(vcol + j * 128 + ((((cbyte >> 4) ^ (j & 7))) << 4)));
        const float2 va = make_float2(bf16lo(v0), bf16hi(v0)), vb = make_float2(bf16lo(v1), bf16hi(v1));
        const float4 p = *reinterpret_cast<const float4*>(sP + (buf * KT + j) * HPC);
        const float pv[HPC] = {p.x, p.y, p.z, p.w};
#pragma unroll
        for (int h = 0; h < HPC; ++h) {
          acc[h][0] = ffma2(make_float2(pv[h], pv[h]), va, acc[h][0]);
          acc[h][1] = ffma2(make_float2(pv[h], pv[h]), vb, acc[h][1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pfree + buf);
      // refill this tile's stage once all four P.V warps are done with it (the
      // score warps finished with its K before marking P ready)
      if (warp == 4 && t + kStages < n_t) {
        if (!wait_all(bar_pfree + buf, (t >> 1) & 1, abort_flag)) {
          if (lane == 0) record(4, kDevTimeout);
          break;
        }
        if (lane == 0) {
          issue(t + kStages);
          n_issued = t + kStages + 1;
        }
      }
    }
    if (loader && *abort_flag) {
      // every issued load must land before the CTA may exit (bounded, not abortable)
      volatile int no_abort = 0;
      for (int t = n_issued > kStages ? n_issued - kStages : 0; t < n_issued; ++t)
        if (!mbar_wait(bar_full + (t % kStages), (t / kStages) & 1, &no_abort, kWaitLimitNs)) break;
    }
#pragma unroll
    for (int h = 0; h < HPC; ++h) {
      float* dst = sRed + (grp * HPC + h) * D + col;
      *reinterpret_cast<float4*>(dst) = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
    }
  }

  __syncthreads();
  if (*abort_flag) return;
  // merge the key groups, then write the split's normalised output and LSE
  for (int idx = tid; idx < nh * D; idx += kThreads) {
    const int h = idx / D, dd = idx % D;
    float sum = 0.f;
#pragma unroll
    for (int g = 0; g < L::kNG; ++g) sum += sRed[(g * HPC + h) * D + dd];
    const float lh = sL[h];
    const size_t row = (static_cast<size_t>(b) * Hq + hq0 + h) * n_split + split;
    o_part[row * D + dd] = sum / lh;
    if (dd == 0) lse_part[row] = (sM[h] * c + __log2f(lh)) * 0.6931471805599453f;
  }
}

// One CTA per (b, hq), one thread per output dim.  It runs after the split
// grid, on the critical path of the step, so its loads are issued together:
// the split LSEs spread over the threads for a block-wide max, then the
// weighted sum eight splits at a time (independent loads, one L2 round trip
// per eight splits instead of one per split).
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const float* __restrict__ o_part,
                                                           const float* __restrict__ lse_part,
                                                           const int* __restrict__ seqlens, int max_seqlen, int Hq,
                                                           int chunk, int n_split, __nv_bfloat16* __restrict__ out,
                                                           float* __restrict__ lse_out) {
  constexpr int kWarps = D / 32;
  __shared__ float s_red[kWarps];
  const int b = blockIdx.x / Hq;
  const int hq = blockIdx.x % Hq;
  const int dd = threadIdx.x;
  // launched as a programmatic dependent of the split kernel: wait until all
  // of its partials are written and visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int Lb = seqlens[b];
  Lb = Lb < 0 ? 0 : (Lb > max_seqlen ? max_seqlen : Lb);
  const int ns = (Lb + chunk - 1) / chunk;
  const size_t row = static_cast<size_t>(b) * Hq + hq;
  if (ns == 0) {
    out[row * D + dd] = __float2bfloat16_rn(0.f);
    if (dd == 0) lse_out[row] = -INFINITY;
    return;
  }
  const float* lp = lse_part + row * n_split;
  float mx = -INFINITY;
  for (int s = dd; s < ns; s += D) mx = fmaxf(mx, lp[s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((dd & 31) == 0) s_red[dd >> 5] = mx;
  __syncthreads();
  mx = s_red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) mx = fmaxf(mx, s_red[w]);
  const float* op = o_part + row * n_split * D + dd;
  float tot = 0.f, acc = 0.f;
  int s = 0;
  for (; s + 8 <= ns; s += 8) {
    float l8[8], o8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      l8[i] = lp[s + i];
      o8[i] = op[static_cast<size_t>(s + i) * D];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float w = expf(l8[i] - mx);
      tot += w;
      acc = fmaf(w, o8[i], acc);
    }
  }
  for (; s < ns; ++s) {
    const float w = expf(lp[s] - mx);
    tot += w;
    acc = fmaf(w, op[static_cast<size_t>(s) * D], acc);
  }
  out[row * D + dd] = __float2bfloat16_rn(acc / tot);
  if (dd == 0) lse_out[row] = mx + logf(tot);
}

template <int D>
cudaError_t launch_d(const DecodeParams& p, cudaStream_t stream) {
  using L = DLayout<D>;
  const int G = p.Hq / p.Hkv;
  const int n_hblk = (G + HPC - 1) / HPC;
  auto kern = p.block_table ? decode_split_kernel<D, true> : decode_split_kernel<D, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  dim3 grid(p.Hkv * n_hblk, p.B, p.n_split);
  kern<<<grid, kThreads, L::kAlloc, stream>>>(p.tm_k, p.tm_v, static_cast<const __nv_bfloat16*>(p.q), p.seqlens,
                                               p.max_seqlen, p.Hq, p.Hkv, p.chunk, p.n_split, p.scale_log2,
                                               p.o_part, p.lse_part, p.block_table, p.max_blocks, p.page_size,
                                               p.num_pages);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the combine grid is set up while the split
  // grid drains, instead of after it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.B * p.Hq);
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, static_cast<const float*>(p.o_part),
                            static_cast<const float*>(p.lse_part), p.seqlens, p.max_seqlen, p.Hq, p.chunk, p.n_split,
                            static_cast<__nv_bfloat16*>(p.o), p.lse);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.d == 64) return launch_d<64>(p, stream);
  if (p.d == 128) return launch_d<128>(p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t fetch_status_decode(cudaStream_t stream, uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_decode_status, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_decode_status, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

}  // namespace attn
