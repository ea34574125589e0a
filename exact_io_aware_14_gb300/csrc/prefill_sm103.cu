// Exact attention forward, prefill / training shapes, for sm_103a.
//
// One CTA computes one 128-row query tile of one (batch, query head):
//   warp 0      TMA producer: Q once, then K_j / V_j tiles into a ring
//   warp 1      TMEM allocator and MMA issuer (one thread):
//                 S_j = Q K_j^T  -> TMEM (two S buffers, so QK^T of tile j+1
//                                   overlaps the softmax of tile j)
//                 O  += P_j V_j  -> TMEM
//   warps 2-5   softmax: one thread owns one query row (TMEM lane), keeps
//               the running max m and sum l in registers, writes P_j (bf16)
//               to shared memory, rescales its O row only when m moved,
//               and at the end writes O / l and the row's LSE.
//
// The method is the tiled online softmax of "FlashAttention: Part 2"
// (chizkidd.github.io), section 6.2: per score tile, update (m, l, a) with
// alpha = exp(m - m') and discard the tile.  Normalisation is deferred to the
// epilogue and the rescale is skipped when the max did not move ("Trace
// FlashAttention's evolution through plain PyTorch code", FA2 and FA4
// paragraphs).  Scores are handled in base 2: t = s * scale * log2(e), so
// p = 2^(t - m) and LSE = (m + log2 l) * ln 2.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace {

__device__ uint32_t g_prefill_status;

constexpr int BM = 128;  // query rows per tile (MMA M, TMEM lanes)
constexpr int BN = 128;  // keys per K/V tile (MMA N of QK^T, K of PV)
constexpr int kThreads = 192;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: no legitimate wait comes close
constexpr uint32_t kTmemCols = 512;               // S0 [0,128) S1 [128,256) O [256, 256+d)

template <int D>
struct Layout {
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static constexpr int kHalf = BM * 128;            // one 64-column block of a 128-row tile
  static constexpr int kQBytes = BM * D * 2;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int kPBytes = BM * BN * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKVBytes;
  static constexpr int kOffP = kOffV + kStages * kKVBytes;
  static constexpr int kOffBar = kOffP + kPBytes;
  static constexpr int kNumBars = 1 + 3 * kStages + 2 + 2 + 1 + 1;
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ out,
                       float* __restrict__ lse_out, int B, int Hq, int Hkv, int Nq, int Nk, int causal,
                       float scale_log2, int n_qtiles) {
  using L = Layout<D>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* bar_q = bars;
  uint64_t* bar_kfull = bars + 1;
  uint64_t* bar_vfull = bar_kfull + S;
  uint64_t* bar_kvempty = bar_vfull + S;
  uint64_t* bar_sfull = bar_kvempty + S;  // [2]
  uint64_t* bar_sfree = bar_sfull + 2;    // [2]
  uint64_t* bar_pfull = bar_sfree + 2;
  uint64_t* bar_odone = bar_pfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: longest causal tiles first (the block scheduler issues low ids first).
  const int bh_count = B * Hq;
  const int qt_rev = blockIdx.x / bh_count;
  const int bh = blockIdx.x % bh_count;
  const int qt = causal ? (n_qtiles - 1 - qt_rev) : qt_rev;
  const int b = bh / Hq;
  const int hq = bh % Hq;
  const int hkv = hq / (Hq / Hkv);
  const int row0 = qt * BM;
  const int kend = causal ? min(Nk, row0 + BM) : Nk;
  const int n_kt = (kend + BN - 1) / BN;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_kfull + s, 1);
      mbar_init(bar_vfull + s, 1);
      mbar_init(bar_kvempty + s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_sfull + i, 1);
      mbar_init(bar_sfree + i, 128);
    }
    mbar_init(bar_pfull, 128);
    mbar_init(bar_odone, 1);
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
  const uint32_t tS0 = tmem, tS1 = tmem + 128, tO = tmem + 256;

  uint8_t* sQ = smem + L::kOffQ;
  uint8_t* sK = smem + L::kOffK;
  uint8_t* sV = smem + L::kOffV;
  uint8_t* sP = smem + L::kOffP;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && n_kt > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar_q, L::kQBytes);
      for (int h = 0; h < D / 64; ++h) tma_load_4d(sQ + h * L::kHalf, &tm_q, bar_q, h * 64, hq, row0, b);
      for (int j = 0; j < n_kt; ++j) {
        const int s = j % S;
        if (j >= S && !wait_one(bar_kvempty + s, ((j / S) - 1) & 1, abort_flag, 1)) break;
        mbar_arrive_expect_tx(bar_kfull + s, L::kKVBytes);
        for (int h = 0; h < D / 64; ++h)
          tma_load_4d(sK + s * L::kKVBytes + h * L::kHalf, &tm_k, bar_kfull + s, h * 64, hkv, j * BN, b);
        mbar_arrive_expect_tx(bar_vfull + s, L::kKVBytes);
        for (int h = 0; h < D / 64; ++h)
          tma_load_4d(sV + s * L::kKVBytes + h * L::kHalf, &tm_v, bar_vfull + s, h * 64, hkv, j * BN, b);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_kt > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, 1);
      const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV), aP = smem_u32(sP);
      bool ok = wait_one(bar_q, 0, abort_flag, 2);
      auto issue_pv = [&](int t) -> bool {
        const int s = t % S;
        if (!wait_one(bar_pfull, t & 1, abort_flag, 3)) return false;
        if (!wait_one(bar_vfull + s, (t / S) & 1, abort_flag, 4)) return false;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          const uint64_t da = sdesc_sw128(aP + (ks >> 2) * L::kHalf + (ks & 3) * 32, 16, 1024);
          const uint64_t db = sdesc_sw128(aV + s * L::kKVBytes + ks * 16 * 128, L::kHalf, 1024);
          mma_bf16_ss(tO, da, db, idesc_pv, (t > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(bar_odone);
        mma_commit(bar_kvempty + s);
        return true;
      };
      for (int j = 0; ok && j < n_kt; ++j) {
        const int s = j % S;
        if (!wait_one(bar_kfull + s, (j / S) & 1, abort_flag, 5)) { ok = false; break; }
        if (j >= 2 && !wait_one(bar_sfree + (j & 1), ((j >> 1) - 1) & 1, abort_flag, 6)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tS = (j & 1) ? tS1 : tS0;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t da = sdesc_sw128(aQ + (ks >> 2) * L::kHalf + (ks & 3) * 32, 16, 1024);
          const uint64_t db = sdesc_sw128(aK + s * L::kKVBytes + (ks >> 2) * L::kHalf + (ks & 3) * 32, 16, 1024);
          mma_bf16_ss(tS, da, db, idesc_qk, ks > 0 ? 1u : 0u);
        }
        mma_commit(bar_sfull + (j & 1));
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(n_kt - 1);
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int quarter = warp & 3;  // TMEM lanes this warp may touch: 32*quarter .. +31
    const int r = quarter * 32 + lane;
    const int grow = row0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t sP_row = smem_u32(sP) + r * 128;
    float m = -INFINITY;  // running max, base-2 scaled units
    float l = 0.f;        // running sum of 2^(t - m)
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      if (!wait_all(bar_sfull + (j & 1), (j >> 1) & 1, abort_flag, 7)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tS = ((j & 1) ? tS1 : tS0) + lane_off;
      float t[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tS + c * 32, u);
#pragma unroll
        for (int i = 0; i < 32; ++i) t[c * 32 + i] = __uint_as_float(u[i]);
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar_sfree + (j & 1));

      const int kbase = j * BN;
      float mt = -INFINITY;
      if (kbase + BN > Nk || (causal && kbase + BN - 1 > row0)) {
        int lim = Nk - kbase;
        if (causal) lim = min(lim, grow - kbase + 1);
#pragma unroll
        for (int i = 0; i < BN; ++i) {
          t[i] = (i < lim) ? t[i] * scale_log2 : -INFINITY;
          mt = fmaxf(mt, t[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < BN; ++i) {
          t[i] *= scale_log2;
          mt = fmaxf(mt, t[i]);
        }
      }
      const float m_new = fmaxf(m, mt);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      float rsum = 0.f;
#pragma unroll
      for (int i = 0; i < BN; ++i) {
        t[i] = ex2_approx(t[i] - m_use);
        rsum += t[i];
      }
      const float alpha = ex2_approx(m - m_use);  // m = -inf -> 0
      l = l * alpha + rsum;

      if (j > 0) {
        // O holds the sum through tile j-1 once PV_{j-1} completes; P's buffer is free then too
        if (!wait_all(bar_odone, (j - 1) & 1, abort_flag, 8)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, m_new != m)) {
          const float a = (m_new != m) ? alpha : 1.f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t u[32];
            tmem_ld32(tO + lane_off + c * 32, u);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * a);
            tmem_st32(tO + lane_off + c * 32, u);
          }
          tmem_wait_st();
        }
      }
      m = m_new;

      // P row -> shared memory, K-major with the 128-B swizzle the MMA descriptor expects
#pragma unroll
      for (int c = 0; c < BN / 8; ++c) {
        const uint32_t addr = sP_row + (c >> 3) * L::kHalf + ((((c & 7) ^ (r & 7))) << 4);
        st_shared_v4(addr, pack_bf16x2(t[8 * c + 0], t[8 * c + 1]), pack_bf16x2(t[8 * c + 2], t[8 * c + 3]),
                     pack_bf16x2(t[8 * c + 4], t[8 * c + 5]), pack_bf16x2(t[8 * c + 6], t[8 * c + 7]));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_pfull);
    }

    // ---------------------------------------------------------------- epilogue
    if (ok && n_kt > 0) ok = wait_all(bar_odone, (n_kt - 1) & 1, abort_flag, 9);
    if (ok) {
      tc_fence_after();
      const bool store = grow < Nq;
      __nv_bfloat16* orow = out + ((static_cast<size_t>(b) * Nq + grow) * Hq + hq) * D;
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        if (n_kt > 0) {
          tmem_ld32(tO + lane_off + c * 32, u);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(u[2 * i]) * inv_l, __uint_as_float(u[2 * i + 1]) * inv_l);
        if (store) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (store) {
        const float lse = (l > 0.f) ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        lse_out[(static_cast<size_t>(b) * Hq + hq) * Nq + grow] = lse;
      }
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
  const long long blocks = static_cast<long long>(n_qtiles) * p.B * p.Hq;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(prefill_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  prefill_fwd_kernel<D><<<static_cast<unsigned>(blocks), kThreads, L::kAlloc, stream>>>(
      p.tm_q, p.tm_k, p.tm_v, static_cast<__nv_bfloat16*>(p.o), p.lse, p.B, p.Hq, p.Hkv, p.Nq, p.Nk, p.causal,
      p.scale_log2, n_qtiles);
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
