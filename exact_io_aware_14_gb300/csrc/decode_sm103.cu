// Query-length-one decode against a KV cache, split over the key axis, for
// sm_103a (pyshine.com flash-attention tour, "Why You Need This": with one
// query the cache is split across thread blocks and the partial results are
// combined).
//
// Split kernel: one CTA per (split of `chunk` keys, KV head, block of up to 4
// query heads of that KV head's group, batch).  K/V tiles of 64 keys stream
// through a 2-stage TMA ring; each K and V byte is read once per CTA and
// serves every query head of the group.  Per tile: scores on CUDA cores ->
// online softmax (running max m, sum l, rescale only when m moved) -> P V
// accumulation in registers.  The CTA writes its split's normalised partial
// output and natural-log LSE.  Decode is memory-bound ("FlashAttention:
// Part 2", section 4.1), so the kernel is built to keep HBM busy: three
// CTAs per SM, up to 64 KB of loads in flight per CTA.
//
// Combine kernel: LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace {

__device__ uint32_t g_decode_status;

constexpr int KT = 64;        // keys per tile
constexpr int HPC = 4;        // query heads per CTA
constexpr int kThreads = 128;
constexpr int kStages = 2;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

template <int D>
struct DLayout {
  static constexpr int kHalf = KT * 128;  // one 64-column box: 64 rows x 128 B
  static constexpr int kTile = KT * D * 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kStages * kTile;
  static constexpr int kOffQ = kOffV + kStages * kTile;        // float [HPC][D]
  static constexpr int kOffS = kOffQ + HPC * D * 4;            // float [HPC][KT]
  static constexpr int kOffP = kOffS + HPC * KT * 4;           // float [KT][HPC]
  static constexpr int kNG = kThreads / (D / 2);               // key groups in the PV phase
  static constexpr int kOffRed = kOffP + KT * HPC * 4;         // float [kNG][HPC][D]
  static constexpr int kOffA = kOffRed + kNG * HPC * D * 4;    // float alpha[HPC], m[HPC], l[HPC]
  static constexpr int kOffBar = kOffA + 3 * HPC * 4 + 16;
  static constexpr int kBytes = kOffBar + kStages * 8 + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

__device__ __forceinline__ void record(uint32_t site, uint32_t code) {
  atomicCAS(&g_decode_status, 0u, (site << 8) | code);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 3)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const __nv_bfloat16* __restrict__ q, const int* __restrict__ seqlens, int max_seqlen,
                        int Hq, int Hkv, int chunk, int n_split, float scale_log2, float* __restrict__ o_part,
                        float* __restrict__ lse_part) {
  using L = DLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int split = blockIdx.x;
  const int G = Hq / Hkv;
  const int n_hblk = (G + HPC - 1) / HPC;
  const int hkv = blockIdx.y / n_hblk;
  const int hb = blockIdx.y % n_hblk;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  int Lb = seqlens[b];
  if (Lb < 0 || Lb > max_seqlen) {
    if (tid == 0 && split == 0 && blockIdx.y == 0) record(1, kDevBadSeqlen);
    Lb = Lb < 0 ? 0 : max_seqlen;
  }
  const int k0 = split * chunk;
  if (k0 >= Lb) return;  // empty split: the combine never reads it
  const int kn = min(chunk, Lb - k0);
  const int n_t = (kn + KT - 1) / KT;
  const int hq0 = hkv * G + hb * HPC;
  const int nh = min(HPC, G - hb * HPC);

  float* sQ = reinterpret_cast<float*>(smem + L::kOffQ);
  float* sS = reinterpret_cast<float*>(smem + L::kOffS);
  float* sP = reinterpret_cast<float*>(smem + L::kOffP);
  float* sRed = reinterpret_cast<float*>(smem + L::kOffRed);
  float* sAlpha = reinterpret_cast<float*>(smem + L::kOffA);
  float* sM = sAlpha + HPC;
  float* sL = sM + HPC;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffA + 3 * HPC * 4);
  uint64_t* bar_full = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint8_t* sK = smem + L::kOffK;
  uint8_t* sV = smem + L::kOffV;

  // query heads of this CTA -> fp32 in shared memory (missing heads read as 0)
  for (int idx = tid; idx < HPC * D; idx += kThreads) {
    const int h = idx / D, dd = idx % D;
    float x = 0.f;
    if (h < nh) x = __bfloat162float(q[(static_cast<size_t>(b) * Hq + hq0 + h) * D + dd]);
    sQ[idx] = x;
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bar_full + s, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();

  auto issue = [&](int t) {
    const int s = t % kStages;
    const int key = k0 + t * KT;
    mbar_arrive_expect_tx(bar_full + s, 2 * L::kTile);
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      tma_load_4d(sK + s * L::kTile + h * L::kHalf, &tm_k, bar_full + s, h * 64, hkv, key, b);
      tma_load_4d(sV + s * L::kTile + h * L::kHalf, &tm_v, bar_full + s, h * 64, hkv, key, b);
    }
  };
  int n_issued = 0;  // meaningful in thread 0 only
  if (tid == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    for (int t = 0; t < n_t && t < kStages; ++t) issue(t);
    n_issued = min(n_t, kStages);
  }

  // running state of head `warp` (every lane of that warp holds it)
  float m = -INFINITY, l = 0.f;
  constexpr int NDP = D / 2;          // dimension pairs
  constexpr int NG = L::kNG;          // key groups in the PV phase
  const int dp = tid % NDP;
  const int grp = tid / NDP;
  float2 acc[HPC];  // dims (2dp, 2dp+1) of each head
#pragma unroll
  for (int h = 0; h < HPC; ++h) acc[h] = make_float2(0.f, 0.f);

  const int qk_key = tid % KT;
  const int qk_hp = tid / KT;  // heads 2*qk_hp, 2*qk_hp + 1
  bool ok = true;

  int t_stop = n_t;
  for (int t = 0; t < n_t; ++t) {
    const int s = t % kStages;
    bool got = mbar_wait(bar_full + s, (t / kStages) & 1, abort_flag, kWaitLimitNs);
    if (!__syncthreads_and(got)) {
      if (tid == 0) record(2, kDevTimeout);
      ok = false;
      t_stop = t;
      break;
    }
    const int valid = min(KT, kn - t * KT);
    const uint32_t kbase = smem_u32(sK + s * L::kTile);
    const uint32_t vbase = smem_u32(sV + s * L::kTile);
    if (valid < KT) {
      // rows past the cache length may hold anything (NaN): zero them in V so
      // that p = 0 contributes exactly nothing
      for (int idx = tid; idx < (KT - valid) * (D / 8); idx += kThreads) {
        const int row = valid + idx / (D / 8), c = idx % (D / 8);
        st_shared_v4(vbase + (c >> 3) * L::kHalf + row * 128 + (((c & 7) ^ (row & 7)) << 4), 0u, 0u, 0u, 0u);
      }
    }

    // scores of key qk_key for heads 2*qk_hp and 2*qk_hp+1 (packed fp32x2 FMAs,
    // four independent partial sums per head)
    {
      float2 a0 = make_float2(0.f, 0.f), a0b = a0, a1 = a0, a1b = a0;
      const float* q0 = sQ + (2 * qk_hp) * D;
      const float* q1 = q0 + D;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 kv = ld_shared_v4(kbase + (c >> 3) * L::kHalf + qk_key * 128 + (((c & 7) ^ (qk_key & 7)) << 4));
        const float4 x0 = *reinterpret_cast<const float4*>(q0 + 8 * c);
        const float4 x1 = *reinterpret_cast<const float4*>(q0 + 8 * c + 4);
        const float4 y0 = *reinterpret_cast<const float4*>(q1 + 8 * c);
        const float4 y1 = *reinterpret_cast<const float4*>(q1 + 8 * c + 4);
        const float2 k01 = make_float2(bf16lo(kv.x), bf16hi(kv.x)), k23 = make_float2(bf16lo(kv.y), bf16hi(kv.y));
        const float2 k45 = make_float2(bf16lo(kv.z), bf16hi(kv.z)), k67 = make_float2(bf16lo(kv.w), bf16hi(kv.w));
        a0 = ffma2(make_float2(x0.x, x0.y), k01, a0);
        a0b = ffma2(make_float2(x0.z, x0.w), k23, a0b);
        a0 = ffma2(make_float2(x1.x, x1.y), k45, a0);
        a0b = ffma2(make_float2(x1.z, x1.w), k67, a0b);
        a1 = ffma2(make_float2(y0.x, y0.y), k01, a1);
        a1b = ffma2(make_float2(y0.z, y0.w), k23, a1b);
        a1 = ffma2(make_float2(y1.x, y1.y), k45, a1);
        a1b = ffma2(make_float2(y1.z, y1.w), k67, a1b);
      }
      const float d0 = (a0.x + a0.y) + (a0b.x + a0b.y);
      const float d1 = (a1.x + a1.y) + (a1b.x + a1b.y);
      const bool vis = qk_key < valid;
      sS[(2 * qk_hp) * KT + qk_key] = vis ? d0 * scale_log2 : -INFINITY;
      sS[(2 * qk_hp + 1) * KT + qk_key] = vis ? d1 * scale_log2 : -INFINITY;
    }
    __syncthreads();

    // online softmax of head `warp` over this tile's 64 scores
    {
      const float x0 = sS[warp * KT + lane], x1 = sS[warp * KT + lane + 32];
      float mt = fmaxf(x0, x1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      const float m_new = fmaxf(m, mt);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float p0 = ex2_approx(x0 - m_use), p1 = ex2_approx(x1 - m_use);
      float ps = p0 + p1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      const float alpha = (m_new == m) ? 1.f : ex2_approx(m - m_use);
      l = l * alpha + ps;
      m = m_new;
      sP[lane * HPC + warp] = p0;
      sP[(lane + 32) * HPC + warp] = p1;
      if (lane == 0) sAlpha[warp] = alpha;
    }
    __syncthreads();

    // O += P V for dims (2dp, 2dp+1), keys grp, grp+NG, ...
    {
      const float4 al = *reinterpret_cast<const float4*>(sAlpha);
      if (al.x != 1.f || al.y != 1.f || al.z != 1.f || al.w != 1.f) {
        acc[0] = fmul2(acc[0], make_float2(al.x, al.x));
        acc[1] = fmul2(acc[1], make_float2(al.y, al.y));
        acc[2] = fmul2(acc[2], make_float2(al.z, al.z));
        acc[3] = fmul2(acc[3], make_float2(al.w, al.w));
      }
      const int col = 2 * dp;
      const uint32_t vcol = vbase + (col >> 6) * L::kHalf;
      const int cbyte = (col & 63) * 2;
#pragma unroll 8
      for (int jj = 0; jj < KT / NG; ++jj) {
        const int j = jj * NG + grp;
        uint32_t vv;
        asm volatile("ld.shared.b32 %0, [%1];"
                     : "=r"(vv)
                     : "r"(vcol + j * 128 + ((((cbyte >> 4) ^ (j & 7))) << 4) + (cbyte & 15)));
        const float2 v = make_float2(bf16lo(vv), bf16hi(vv));
        const float4 p = *reinterpret_cast<const float4*>(sP + j * HPC);
        acc[0] = ffma2(make_float2(p.x, p.x), v, acc[0]);
        acc[1] = ffma2(make_float2(p.y, p.y), v, acc[1]);
        acc[2] = ffma2(make_float2(p.z, p.z), v, acc[2]);
        acc[3] = ffma2(make_float2(p.w, p.w), v, acc[3]);
      }
    }
    __syncthreads();  // stage s, sS and sP are free again
    if (tid == 0 && t + kStages < n_t) {
      issue(t + kStages);
      n_issued = t + kStages + 1;
    }
  }

  // every issued load must land before the CTA may exit (bounded, not abortable)
  if (!ok) {
    if (tid == 0) {
      volatile int no_abort = 0;
      for (int t = t_stop; t < n_issued; ++t)
        if (!mbar_wait(bar_full + (t % kStages), (t / kStages) & 1, &no_abort, kWaitLimitNs)) break;
    }
    return;
  }

  // merge the NG key groups, then write the split's normalised output and LSE
#pragma unroll
  for (int h = 0; h < HPC; ++h) {
    sRed[(grp * HPC + h) * D + 2 * dp] = acc[h].x;
    sRed[(grp * HPC + h) * D + 2 * dp + 1] = acc[h].y;
  }
  if (lane == 0) {
    sM[warp] = m;
    sL[warp] = l;
  }
  __syncthreads();
  for (int idx = tid; idx < nh * D; idx += kThreads) {
    const int h = idx / D, dd = idx % D;
    float sum = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g) sum += sRed[(g * HPC + h) * D + dd];
    const float lh = sL[h];
    const size_t row = (static_cast<size_t>(b) * Hq + hq0 + h) * n_split + split;
    o_part[row * D + dd] = sum / lh;
    if (dd == 0) lse_part[row] = (sM[h] + __log2f(lh)) * 0.6931471805599453f;
  }
}

template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const float* __restrict__ o_part,
                                                           const float* __restrict__ lse_part,
                                                           const int* __restrict__ seqlens, int max_seqlen, int Hq,
                                                           int chunk, int n_split, __nv_bfloat16* __restrict__ out,
                                                           float* __restrict__ lse_out) {
  const int b = blockIdx.x / Hq;
  const int hq = blockIdx.x % Hq;
  const int dd = threadIdx.x;
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
  for (int s = 0; s < ns; ++s) mx = fmaxf(mx, lp[s]);
  float tot = 0.f, acc = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float w = expf(lp[s] - mx);
    tot += w;
    acc = fmaf(w, o_part[(row * n_split + s) * D + dd], acc);
  }
  out[row * D + dd] = __float2bfloat16_rn(acc / tot);
  if (dd == 0) lse_out[row] = mx + logf(tot);
}

template <int D>
cudaError_t launch_d(const DecodeParams& p, cudaStream_t stream) {
  using L = DLayout<D>;
  const int G = p.Hq / p.Hkv;
  const int n_hblk = (G + HPC - 1) / HPC;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_split, p.Hkv * n_hblk, p.B);
  decode_split_kernel<D><<<grid, kThreads, L::kAlloc, stream>>>(
      p.tm_k, p.tm_v, static_cast<const __nv_bfloat16*>(p.q), p.seqlens, p.max_seqlen, p.Hq, p.Hkv, p.chunk,
      p.n_split, p.scale_log2, p.o_part, p.lse_part);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<D><<<p.B * p.Hq, D, 0, stream>>>(p.o_part, p.lse_part, p.seqlens, p.max_seqlen, p.Hq,
                                                         p.chunk, p.n_split, static_cast<__nv_bfloat16*>(p.o),
                                                         p.lse);
  return cudaGetLastError();
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
