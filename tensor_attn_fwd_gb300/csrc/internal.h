// internal.h -- declarations shared by the library's translation units (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

#include "../../include/attn.h"

namespace attn {

// Device address of the library's status word on the current device (the
// word kernels write ATTN_ERR_TIMEOUT into).  nullptr on failure.
int* status_word_device_ptr();

// Streaming-multiprocessor count of the current device (cached per device).
int sm_count();

// Raise the kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device).
cudaError_t ensure_smem_attr(const void* kernel, int bytes);

// Tiled TMA map of a contiguous [planes, rows, D] bf16 tensor with boxes of
// [1, box_rows, 64] elements and 128-byte swizzle (rows past `rows` read as
// zero).  False if the driver entry point is unavailable or rejects the map.
bool encode_bf16_map(CUtensorMap* map, const void* base, int D, int rows, int planes,
                     int box_rows);

// Launch `kernel` on `stream` as a programmatic dependent of the previous
// kernel in the stream: its CTAs may start (and run their set-up) while that
// kernel finishes; the kernel itself executes griddepcontrol.wait before it
// touches global memory, so it still sees all of that kernel's writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Kernel launchers; arguments are already validated.  Return cudaError_t of
// the launch.
// o: fp32 [B,Hq,Sq,D], or bf16 when o_bf16 != 0.
cudaError_t launch_attn_fwd(const void* q, const void* k, const void* v, void* o, int o_bf16,
                            float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                            float scale, cudaStream_t stream, int* status);

// Paged KV cache: k, v are [num_pages, Hkv, page_size, D]; key t of sequence b
// is row t % page_size of page block_table[b * max_pages + t / page_size].
struct PagedKV {
  const int* block_table;  // device int32 [B, max_pages]
  int page_size;           // a multiple of 32
  int max_pages;
  int num_pages;
};

// Head dimension 256 (one query tile per CTA, double-buffered S); called by
// launch_attn_fwd.
// Work items of the D 64/128 prefill per KV split: pairs of 128-row query tiles,
// either of one head (rows 256i..256i+255) or, when Sq <= 128 and the KV groups
// have an even number of query heads, of two heads of one group.
inline int fwd_head_pairs(int Hq, int Hkv, int Sq) {
  return (Sq <= 128 && (Hq / Hkv) % 2 == 0) ? 1 : 0;
}
inline long long fwd_items_per_split(long long B, int Hq, int Hkv, int Sq) {
  return fwd_head_pairs(Hq, Hkv, Sq) ? B * Hq / 2 : B * Hq * ((Sq + 255) / 256);
}

// The prefill kernels' work-item orders (each a separate kernel instantiation):
// 0 longest first; 1 KV head by KV head (no causal mask; at D = 256 only when all
// K/V exceed 96 MB); 2 longest first within chunks of KV heads whose K/V fit in
// L2 (D = 256 under the causal mask, all K/V beyond 96 MB, Sq <= 4096).  Measured: see the item lookups in attn_fwd.cu and
// attn_fwd_d256.cu.
constexpr long long kFwdKvChunkBytes = 48ll << 20;
inline long long fwd_kv_head_bytes(int Sk, int D) { return 4ll * Sk * D; }  // K + V, bf16
inline int fwd_kv_chunk(int Sk, int D) {
  const long long c = kFwdKvChunkBytes / fwd_kv_head_bytes(Sk, D);
  return c < 1 ? 1 : (c > (1 << 30) ? (1 << 30) : static_cast<int>(c));
}
inline int fwd_item_order(long long B, int Hq, int Hkv, int Sq, int Sk, int D, int causal) {
  if (D != 256 && fwd_head_pairs(Hq, Hkv, Sq)) return 0;
  const bool big_kv = B * Hkv * fwd_kv_head_bytes(Sk, D) > 2 * kFwdKvChunkBytes;
  if (!causal) {
    if (D == 256) return big_kv ? 1 : 0;
    return static_cast<long long>(Hq / Hkv) * ((Sq + 255) / 256) <= 32 ? 1 : 0;
  }
  return D == 256 && Sq <= 4096 && big_kv ? 2 : 0;
}

// Prefill over KV splits (D 64 or 128): split s covers KV tiles
// [s*t, (s+1)*t), t = ceil(ceil(Sk/128) / num_splits), and writes its partial O
// (fp32, normalised by its own row sum) and LSE at o_part / lse_part + s * the
// size of one full output; rows a split leaves empty get O = 0, LSE = -inf.
cudaError_t launch_attn_fwd_splitkv(const void* q, const void* k, const void* v, float* o_part,
                                    float* lse_part, int B, int Hq, int Hkv, int Sq, int Sk,
                                    int D, int causal, int num_splits, float scale,
                                    cudaStream_t stream, int* status);
cudaError_t launch_attn_fwd_d256(const void* q, const void* k, const void* v, void* o, int o_bf16,
                                 float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int causal,
                                 float scale, cudaStream_t stream, int* status);

// QKV projection + rotary embedding (qkv_rope.cu).
cudaError_t launch_rope_table(float* table, int max_pos, int D, double base, cudaStream_t stream);
cudaError_t launch_qkv_rope(const void* x, const void* w, const float* rope, const int* positions,
                            void* q, void* k, void* v, int B, int S, int hidden, int Hq, int Hkv,
                            int D, int max_pos, int style, cudaStream_t stream, int* status);

// The argument checks every split-KV decode entry point shares (inputs, sizes,
// split count, scale, head dimension, input alignment); `paged` skips the
// contiguous-cache size limit.  ATTN_OK or the status to return.
int decode_check_args(const void* q, const void* k, const void* v, int B, int Hq, int Hkv,
                      int Sk, int D, int num_splits, float scale, bool paged);

// seqlens: optional device int32 [B] of per-sequence key counts (nullptr: Sk).
// paged: optional page layout (then Sk = max_pages * page_size, the capacity).
// fused: when counters != nullptr, the CTA that completes a (batch, KV head,
// 16-head slice) group last also combines the group's partials into o / lse
// (counters: int32 [B * Hkv * ceil((Hq/Hkv)/16)], zero on entry, zero again after).
struct FusedCombine {
  float* o;
  float* lse;
  int* counters;
};
cudaError_t launch_decode_splitkv(const void* q, const void* k, const void* v, float* o_part,
                                  float* lse_part, int B, int Hq, int Hkv, int Sk, int D,
                                  int num_splits, float scale, cudaStream_t stream, int* status,
                                  const int* seqlens = nullptr, const PagedKV* paged = nullptr,
                                  const FusedCombine* fused = nullptr);

// Backward: Delta into `delta` ([B,Hq,Sq]), then dK/dV and dQ kernels.
cudaError_t launch_attn_bwd(const void* q, const void* k, const void* v, const float* o,
                            const float* lse, const void* dout, float* dq, float* dk, float* dv,
                            float* delta, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                            int causal, float scale, cudaStream_t stream, int* status);

cudaError_t launch_wait_selftest(uint64_t limit_ns, int* status, uint64_t* waited_ns,
                                 cudaStream_t stream);
cudaError_t launch_combine(const float* o_part, const float* lse_part, float* o, float* lse,
                           int rows, int D, int num_splits, cudaStream_t stream);

}  // namespace attn
