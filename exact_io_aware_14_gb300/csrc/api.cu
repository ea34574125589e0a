// extern "C" boundary of the library: argument checks, TMA descriptor
// encoding and dispatch to the kernel units.  Declared in include/attn.h.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "launch.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 4-D view {d, H, N, B} of a dense BSHD bf16 tensor; box {64, 1, rows, 1},
// 128-byte swizzle (one box row = 64 bf16 = 128 B).
bool make_map(CUtensorMap* m, const void* base, int B, int N, int H, int d, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t nn = N > 0 ? (cuuint64_t)N : 1u;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, nn, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2, nn * H * d * 2};
  const cuuint32_t box[4] = {64u, 1u, (cuuint32_t)box_rows, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr double kLog2e = 1.4426950408889634;

size_t splitkv_part_elems(int B, int Hq, int n_split) {
  return static_cast<size_t>(B) * Hq * n_split;
}
size_t round16(size_t x) { return (x + 15) & ~size_t(15); }

}  // namespace

extern "C" {

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case ATTN_ERR_LAUNCH: return "CUDA launch or runtime error";
    case ATTN_ERR_TIMEOUT: return "device pipeline wait timed out";
    case ATTN_ERR_DEVICE_ARG: return "cache length or page index out of range";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

}  // extern "C"

namespace {

// A window side of Nq + Nk or more bounds nothing: it is made unbounded (-1),
// which also keeps every position sum inside int range.
int normalise_window(int w, int Nq, int Nk) {
  if (w < 0) return -1;
  return static_cast<long long>(w) >= static_cast<long long>(Nq) + Nk ? -1 : w;
}

// Shared by attn_fwd, attn_fwd_window and attn_fwd_kvcache.  Nk is the
// allocated key length (max_seqlen for a cache); seqlens is null or a device
// array of per-sequence key counts.
attn_status prefill(const void* q, const void* k, const void* v, const int* seqlens, void* o, float* lse, int B,
                    int Hq, int Hkv, int Nq, int Nk, int d, int causal, int window_left, int window_right,
                    float scale, void* stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 0 || Nk < 0 || (Hq % Hkv) != 0) return ATTN_ERR_INVALID_ARG;
  if (causal < 0 || causal > 2) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  // 32-bit TMA coordinates and grid: keep rows and tiles well inside int range
  if (static_cast<long long>(Nq) + Nk + 256 > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>((Nq + 127) / 128) * B * Hq > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if (Nq == 0) return ATTN_OK;
  if (!q || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (Nk > 0 && (!k || !v)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_MISALIGNED;
  if (Nk > 0 && (!aligned16(k) || !aligned16(v))) return ATTN_ERR_MISALIGNED;
  if (seqlens && (reinterpret_cast<uintptr_t>(seqlens) & 3u)) return ATTN_ERR_MISALIGNED;

  attn::PrefillParams p;
  std::memset(&p, 0, sizeof p);
  // With no keys nothing is loaded from K/V; the maps then describe q (never used).
  const void* kb = Nk > 0 ? k : q;
  const void* vb = Nk > 0 ? v : q;
  const int nk_map = Nk > 0 ? Nk : Nq;
  const int hkv_map = Nk > 0 ? Hkv : Hq;
  if (!make_map(&p.tm_q, q, B, Nq, Hq, d, 128) || !make_map(&p.tm_k, kb, B, nk_map, hkv_map, d, 128) ||
      !make_map(&p.tm_v, vb, B, nk_map, hkv_map, d, 128))
    return ATTN_ERR_LAUNCH;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.d = d;
  p.causal = causal;
  p.seqlens = seqlens;
  p.window_left = normalise_window(window_left, Nq, Nk);
  p.window_right = normalise_window(window_right, Nq, Nk);
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * kLog2e);
  return attn::launch_prefill(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace

extern "C" {

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Nq, int Nk, int d, int causal, float scale, void* stream) {
  return prefill(q, k, v, nullptr, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, -1, -1, scale, stream);
}

attn_status attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                            int Hkv, int Nq, int Nk, int d, int causal, int window_left, int window_right, float scale,
                            void* stream) {
  return prefill(q, k, v, nullptr, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, window_left, window_right, scale, stream);
}

attn_status attn_fwd_kvcache(const void* q, const void* k_cache, const void* v_cache, const int* seqlens,
                             int max_seqlen, void* o, float* lse, int B, int Hq, int Hkv, int Nq, int d, int causal,
                             int window_left, int window_right, float scale, void* stream) {
  if (max_seqlen < 1) return ATTN_ERR_INVALID_ARG;
  if (Nq > 0 && (!k_cache || !v_cache || !seqlens)) return ATTN_ERR_INVALID_ARG;
  return prefill(q, k_cache, v_cache, seqlens, o, lse, B, Hq, Hkv, Nq, max_seqlen, d, causal, window_left,
                 window_right, scale, stream);
}

size_t attn_splitkv_workspace_size(int B, int Hq, int max_seqlen, int d, int chunk) {
  if (B < 1 || Hq < 1 || max_seqlen < 1 || d < 1 || chunk < 64 || (chunk % 64) != 0) return 0;
  const int n_split = (max_seqlen + chunk - 1) / chunk;
  const size_t parts = splitkv_part_elems(B, Hq, n_split);
  return round16(parts * d * sizeof(float)) + round16(parts * sizeof(float));
}

}  // extern "C"

namespace attn {

attn_status check_splitkv_args(const void* q, const void* k, const void* v, const int* seqlens, int max_seqlen,
                               const int* block_table, int page_size, const void* o, const float* lse, int B, int Hq,
                               int Hkv, int d, float scale, int chunk) {
  if (B < 1 || Hq < 1 || Hkv < 1 || (Hq % Hkv) != 0 || max_seqlen < 1) return ATTN_ERR_INVALID_ARG;
  if (chunk < 64 || (chunk % 64) != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (B > 65535) return ATTN_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if (static_cast<long long>(Hkv) * ((G + 3) / 4) > 65535) return ATTN_ERR_UNSUPPORTED;
  if ((max_seqlen + static_cast<long long>(chunk) - 1) / chunk > 65535) return ATTN_ERR_UNSUPPORTED;  // grid z
  if (!q || !k || !v || !seqlens || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(seqlens) & 3u))
    return ATTN_ERR_MISALIGNED;
  if (block_table) {
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u)) return ATTN_ERR_MISALIGNED;
    // the pages of one split must fit the kernel's list of them
    if (chunk / page_size + 2 > 128) return ATTN_ERR_UNSUPPORTED;
  }
  return ATTN_OK;
}

}  // namespace attn

namespace {

// Shared by the contiguous and the paged split-KV calls.  Paged: block_table
// non-null, k/v are page pools [num_pages, page_size, Hkv, d] and the
// logical cache capacity is max_blocks * page_size.
attn_status splitkv(const void* q, const void* k, const void* v, const int* seqlens, int max_seqlen,
                    const int* block_table, int max_blocks, int page_size, int num_pages, void* o, float* lse,
                    int B, int Hq, int Hkv, int d, float scale, int chunk, void* workspace, size_t workspace_bytes,
                    void* stream) {
  const attn_status st =
      attn::check_splitkv_args(q, k, v, seqlens, max_seqlen, block_table, page_size, o, lse, B, Hq, Hkv, d, scale,
                               chunk);
  if (st != ATTN_OK) return st;
  const size_t need = attn_splitkv_workspace_size(B, Hq, max_seqlen, d, chunk);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;

  attn::DecodeParams p;

  std::memset(&p, 0, sizeof p);
  const bool ok_maps = block_table ? (make_map(&p.tm_k, k, num_pages, page_size, Hkv, d, 64) &&
                                      make_map(&p.tm_v, v, num_pages, page_size, Hkv, d, 64))
                                   : (make_map(&p.tm_k, k, B, max_seqlen, Hkv, d, 64) &&
                                      make_map(&p.tm_v, v, B, max_seqlen, Hkv, d, 64));
  if (!ok_maps) return ATTN_ERR_LAUNCH;
  p.n_split = (max_seqlen + chunk - 1) / chunk;
  const size_t parts = splitkv_part_elems(B, Hq, p.n_split);
  p.o_part = static_cast<float*>(workspace);
  p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + round16(parts * d * sizeof(float)));
  p.q = q;
  p.seqlens = seqlens;
  p.o = o;
  p.lse = lse;
  p.block_table = block_table;
  p.max_blocks = max_blocks;
  p.page_size = page_size;
  p.num_pages = num_pages;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.d = d;
  p.max_seqlen = max_seqlen;
  p.chunk = chunk;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * kLog2e);
  return attn::launch_decode(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace

extern "C" {

attn_status attn_fwd_splitkv(const void* q, const void* k_cache, const void* v_cache, const int* seqlens,
                             int max_seqlen, void* o, float* lse, int B, int Hq, int Hkv, int d, float scale,
                             int chunk, void* workspace, size_t workspace_bytes, void* stream) {
  return splitkv(q, k_cache, v_cache, seqlens, max_seqlen, nullptr, 0, 0, 0, o, lse, B, Hq, Hkv, d, scale, chunk,
                 workspace, workspace_bytes, stream);
}

attn_status attn_fwd_splitkv_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                                   int max_blocks, int page_size, int num_pages, const int* seqlens, void* o,
                                   float* lse, int B, int Hq, int Hkv, int d, float scale, int chunk, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (!block_table || max_blocks < 1 || num_pages < 1 || page_size < 64 || (page_size % 64) != 0)
    return ATTN_ERR_INVALID_ARG;
  const long long cap = static_cast<long long>(max_blocks) * page_size;
  if (cap > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  return splitkv(q, k_pages, v_pages, seqlens, static_cast<int>(cap), block_table, max_blocks, page_size, num_pages,
                 o, lse, B, Hq, Hkv, d, scale, chunk, workspace, workspace_bytes, stream);
}

attn_status attn_selftest_wait_timeout(unsigned long long limit_ns, void* stream) {
  if (limit_ns < 1000ull) limit_ns = 1000ull;
  if (limit_ns > 2000000000ull) limit_ns = 2000000000ull;
  return attn::launch_selftest_wait_timeout(limit_ns, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_LAUNCH;
}

attn_status attn_selftest_exp2_poly(const float* x, float* y, long long n, void* stream) {
  if (n < 0) return ATTN_ERR_INVALID_ARG;
  if (n == 0) return ATTN_OK;
  if (!x || !y) return ATTN_ERR_INVALID_ARG;
  if (n > (1LL << 38)) return ATTN_ERR_UNSUPPORTED;  // grid of 256-thread blocks, one pair per thread
  if ((reinterpret_cast<uintptr_t>(x) & 3u) || (reinterpret_cast<uintptr_t>(y) & 3u)) return ATTN_ERR_MISALIGNED;
  return attn::launch_selftest_exp2_poly(x, y, n, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_LAUNCH;
}

attn_status attn_probe_read_bandwidth(const void* buf, size_t bytes, unsigned long long* sink, void* stream) {
  if (bytes == 0) return ATTN_OK;
  if (!buf || !sink) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(buf) || (bytes & 15u) || (reinterpret_cast<uintptr_t>(sink) & 7u)) return ATTN_ERR_MISALIGNED;
  return attn::launch_read_probe(buf, static_cast<long long>(bytes / 16), sink, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_LAUNCH;
}

attn_status attn_get_device_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_LAUNCH;
  uint32_t w_prefill = 0, w_decode = 0, w_selftest = 0;
  if (attn::fetch_status_prefill(s, &w_prefill) != cudaSuccess) return ATTN_ERR_LAUNCH;
  if (attn::fetch_status_decode(s, &w_decode) != cudaSuccess) return ATTN_ERR_LAUNCH;
  if (attn::fetch_status_selftest(s, &w_selftest) != cudaSuccess) return ATTN_ERR_LAUNCH;
  const uint32_t w = w_prefill ? w_prefill : (w_decode ? w_decode : w_selftest);
  switch (w & 0xffu) {
    case 0: return ATTN_OK;
    case attn::kDevTimeout: return ATTN_ERR_TIMEOUT;
    case attn::kDevBadSeqlen:
    case attn::kDevBadPage: return ATTN_ERR_DEVICE_ARG;
    default: return ATTN_ERR_LAUNCH;
  }
}

}  // extern "C"
