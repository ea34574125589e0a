// Host-side interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Internal to the library.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn.h"

namespace attn {

// Device status codes.  Kernels never trap: a wait that runs out of time
// records (site << 8) | code in the unit's status word and the kernel unwinds.
enum DeviceCode : uint32_t { kDevOk = 0, kDevTimeout = 5, kDevBadSeqlen = 6, kDevBadPage = 7 };

struct PrefillParams {
  CUtensorMap tm_q, tm_k, tm_v;  // 4-D maps {d, H, N, B}, box {64, 1, 128, 1}, 128-B swizzle
  void* o;
  float* lse;
  int B, Hq, Hkv, Nq, Nk, d;
  int causal;            // 0 none, 1 aligned top-left, 2 aligned bottom-right
  const int* seqlens;    // null, or keys per sequence (cache lengths <= Nk) on the device
  int window_left, window_right;  // local window aligned bottom-right; -1: that side unbounded
  float scale_log2;      // scale * log2(e)
};
cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream);

struct DecodeParams {
  CUtensorMap tm_k, tm_v;  // 4-D maps {d, Hkv, max_seqlen, B}, box {64, 1, 64, 1}, 128-B swizzle
  const void* q;
  const int* seqlens;
  void* o;
  float* lse;
  float* o_part;    // [B, Hq, n_split, d]
  float* lse_part;  // [B, Hq, n_split]
  // paged cache (block_table non-null): maps are {d, Hkv, page_size, num_pages}
  const int* block_table;  // [B, max_blocks]
  int max_blocks, page_size, num_pages;
  int B, Hq, Hkv, d, max_seqlen, chunk, n_split;
  float scale_log2;
};
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);

// Host checks of the split-KV decode arguments other than the workspace, in
// the order the entry points report them (no CUDA call).  block_table is
// null for a contiguous cache.
attn_status check_splitkv_args(const void* q, const void* k, const void* v, const int* seqlens, int max_seqlen,
                               const int* block_table, int page_size, const void* o, const float* lse, int B, int Hq,
                               int Hkv, int d, float scale, int chunk);

// Reads and clears the device status word of each kernel unit (stream-ordered,
// then synchronises the stream).  Returns the first non-zero word, or 0.
cudaError_t fetch_status_prefill(cudaStream_t stream, uint32_t* out);
cudaError_t fetch_status_decode(cudaStream_t stream, uint32_t* out);
cudaError_t launch_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_selftest_exp2_poly(const float* x, float* y, long long n, cudaStream_t stream);
cudaError_t launch_read_probe(const void* buf, long long n16, unsigned long long* sink, cudaStream_t stream);
cudaError_t fetch_status_selftest(cudaStream_t stream, uint32_t* out);

}  // namespace attn
