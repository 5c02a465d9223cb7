// api.cu -- the C ABI of libattn.so: argument validation, status codes and the
// per-device state (SM count, kernel attributes, device status word).  Every
// entry point validates before launching; nothing here allocates device
// memory or synchronises, except attn_debug_status().
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"

namespace attn {
namespace {

constexpr int kMaxDevices = 64;

// Written by kernels whose bounded wait expired (ATTN_ERR_TIMEOUT).
__device__ int g_status_word = 0;

std::mutex g_mutex;
int g_sm_count[kMaxDevices] = {0};
int* g_status_ptr[kMaxDevices] = {nullptr};

struct AttrEntry {
  const void* kernel;
  int bytes;
  uint64_t device_mask;
};
constexpr int kAttrSlots = 32;  // one per kernel instantiation that sets its shared memory size
AttrEntry g_attr[kAttrSlots];
int g_attr_n = 0;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Sizes are int on the ABI; keep every product the kernels form in range.
constexpr long long kMaxElems = 1ll << 40;
constexpr int kMaxSeq = 1 << 30;

}  // namespace

int sm_count() {
  const int dev = current_device();
  if (dev < 0) return 1;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

int* status_word_device_ptr() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

cudaError_t ensure_smem_attr(const void* kernel, int bytes) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  AttrEntry* e = nullptr;
  for (int i = 0; i < g_attr_n; ++i)
    if (g_attr[i].kernel == kernel) e = &g_attr[i];
  if (e != nullptr && e->bytes >= bytes && (e->device_mask >> dev & 1u)) return cudaSuccess;
  const cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err != cudaSuccess) return err;
  if (e == nullptr) {
    if (g_attr_n >= kAttrSlots) return cudaSuccess;  // table full: set again next time
    e = &g_attr[g_attr_n++];
    e->kernel = kernel;
    e->bytes = bytes;
    e->device_mask = 0;
  }
  e->bytes = bytes;
  e->device_mask |= uint64_t(1) << dev;
  return cudaSuccess;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qres;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &qres) == cudaSuccess &&
        qres == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

bool encode_bf16_map(CUtensorMap* map, const void* base, int D, int rows, int planes,
                     int box_rows) {
  auto fn = get_encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(rows), cuuint64_t(planes)};
  const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(D) * 2 * cuuint64_t(rows)};
  const cuuint32_t box[3] = {64, cuuint32_t(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace attn

using namespace attn;

extern "C" {

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG: invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED: unsupported configuration";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED: pointer not 16-byte aligned";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: CUDA runtime error";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: a kernel wait expired";
    case ATTN_ERR_BOUNDS: return "ATTN_ERR_BOUNDS: a kernel store fell outside its output (debug build)";
    default: return "unknown attn status";
  }
}

int attn_version(void) { return (1 << 16) | 0; }

namespace {

int fwd_common(const void* q, const void* k, const void* v, void* o, int o_bf16, float* lse,
               int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
               void* stream) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (Sq > kMaxSeq || Sk > kMaxSeq) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq * Sq * D > kMaxElems ||
      static_cast<long long>(B) * Hkv * Sk * D > kMaxElems)
    return ATTN_ERR_UNSUPPORTED;
  // Work items (B*Hq*ceil(Sq/256), or ceil(Sq/128) at D = 256) are indexed with int.
  if (static_cast<long long>(B) * Hq * ((Sq + 127) / 128) > (1ll << 30)) return ATTN_ERR_UNSUPPORTED;
  if (D != 64 && D != 128 && D != 256) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_MISALIGNED;
  int* status = status_word_device_ptr();
  if (status == nullptr) return ATTN_ERR_CUDA;
  const cudaError_t e = launch_attn_fwd(q, k, v, o, o_bf16, lse, B, Hq, Hkv, Sq, Sk, D, causal,
                                        scale, static_cast<cudaStream_t>(stream), status);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

int attn_fwd(const void* q, const void* k, const void* v, float* o, float* lse, int B, int Hq,
             int Hkv, int Sq, int Sk, int D, int causal, float scale, void* stream) {
  return fwd_common(q, k, v, o, 0, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, stream);
}

int attn_fwd_bf16o(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                   void* stream) {
  return fwd_common(q, k, v, o, 1, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, stream);
}

int attn_fwd_splitkv(const void* q, const void* k, const void* v, float* o_part,
                     float* lse_part, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                     int num_splits, float scale, void* stream) {
  if (!q || !k || !v || !o_part || !lse_part) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (Sq > kMaxSeq || Sk > kMaxSeq) return ATTN_ERR_UNSUPPORTED;
  // Every split covers at least one 128-key tile.
  if (num_splits < 1 || num_splits > (Sk + 127) / 128) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_splits) * B * Hq * Sq * D > kMaxElems ||
      static_cast<long long>(B) * Hkv * Sk * D > kMaxElems)
    return ATTN_ERR_UNSUPPORTED;
  // Work items B*Hq*ceil(Sq/256)*num_splits are indexed with int.
  if (static_cast<long long>(B) * Hq * ((Sq + 255) / 256) * num_splits > (1ll << 30))
    return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_part) ||
      !aligned16(lse_part))
    return ATTN_ERR_MISALIGNED;
  int* status = status_word_device_ptr();
  if (status == nullptr) return ATTN_ERR_CUDA;
  const cudaError_t e =
      launch_attn_fwd_splitkv(q, k, v, o_part, lse_part, B, Hq, Hkv, Sq, Sk, D, causal,
                              num_splits, scale, static_cast<cudaStream_t>(stream), status);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_fwd_num_splits(int B, int Hq, int Hkv, int Sq, int Sk, int D, int* num_splits) {
  if (num_splits == nullptr) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || D <= 0 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  const int n_sm = sm_count();
  if (n_sm <= 0) return ATTN_ERR_CUDA;
  long long ns = 1;
  if (D == 64 || D == 128) {
    // Work items without splitting (two 128-row query tiles each).
    const long long base = fwd_items_per_split(B, Hq, Hkv, Sq);
    const long long kv_tiles = (Sk + 127) / 128;
    // Splitting pays when it removes more KV steps from every item than the
    // combine and the partials cost: a cache long against the chunk
    // (Sk > 2 Sq) or at least 16 KV tiles.  Measured counter-examples: causal
    // or not, B1 H16 S1024 D64 (one pass 14.0 us, 2 splits 14.8) and B1 Hq32
    // Hkv8 Sq512 Sk1024 (16.2 vs 18.2).
    const bool worth = Sk > 2ll * Sq || kv_tiles >= 16;
    if (worth && base * 5 < static_cast<long long>(n_sm) * 4) {
      // Too few to fill the GPU: as many splits as still fit every item in one
      // round on the SMs (a second round would cost as much as it saves), each
      // split keeping at least four 128-key tiles.
      ns = n_sm / base > 1 ? n_sm / base : 1;
      const long long cap = kv_tiles / 4 > 1 ? kv_tiles / 4 : 1;
      if (ns > cap) ns = cap;
    }
  }
  *num_splits = static_cast<int>(ns);
  return ATTN_OK;
}

}  // extern "C"

int attn::decode_check_args(const void* q, const void* k, const void* v, int B, int Hq, int Hkv,
                            int Sk, int D, int num_splits, float scale, bool paged) {
  if (!q || !k || !v) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sk <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (num_splits < 1 || num_splits > Sk) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  // The kernels split [0, Sk) with int arithmetic.
  if (Sk > kMaxSeq) return ATTN_ERR_UNSUPPORTED;
  if (!paged && static_cast<long long>(B) * Hkv * Sk * D > kMaxElems) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_splits) * B * Hq * D > kMaxElems) return ATTN_ERR_UNSUPPORTED;
  // Output rows (and tensor-map planes) are indexed with int.
  if (static_cast<long long>(B) * Hq > (1ll << 30)) return ATTN_ERR_UNSUPPORTED;
  const int head_slices = (Hq / Hkv + 15) / 16;  // query heads per decode CTA: 16
  if (B > 65535 || static_cast<long long>(Hkv) * head_slices > 65535)
    return ATTN_ERR_UNSUPPORTED;
  if (D != 64 && D != 128 && D != 256) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return ATTN_ERR_MISALIGNED;
  return ATTN_OK;
}

extern "C" {

namespace {

int decode_common(const void* q, const void* k, const void* v, const int* seqlens,
                  float* o_part, float* lse_part, int B, int Hq, int Hkv, int Sk, int D,
                  int num_splits, float scale, void* stream, const PagedKV* paged = nullptr) {
  if (!o_part || !lse_part) return ATTN_ERR_INVALID_ARG;
  const int chk = decode_check_args(q, k, v, B, Hq, Hkv, Sk, D, num_splits, scale,
                                    paged != nullptr);
  if (chk != ATTN_OK) return chk;
  if (!aligned16(o_part) || !aligned16(lse_part)) return ATTN_ERR_MISALIGNED;
  int* status = status_word_device_ptr();
  if (status == nullptr) return ATTN_ERR_CUDA;
  const cudaError_t e =
      launch_decode_splitkv(q, k, v, o_part, lse_part, B, Hq, Hkv, Sk, D, num_splits, scale,
                            static_cast<cudaStream_t>(stream), status, seqlens, paged);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

int attn_decode_splitkv(const void* q, const void* k, const void* v, float* o_part,
                        float* lse_part, int B, int Hq, int Hkv, int Sk, int D, int num_splits,
                        float scale, void* stream) {
  return decode_common(q, k, v, nullptr, o_part, lse_part, B, Hq, Hkv, Sk, D, num_splits, scale,
                       stream);
}

int attn_decode_splitkv_varlen(const void* q, const void* k, const void* v, const int* seqlens,
                               float* o_part, float* lse_part, int B, int Hq, int Hkv, int Sk,
                               int D, int num_splits, float scale, void* stream) {
  if (!seqlens) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(seqlens) & 3u) != 0) return ATTN_ERR_MISALIGNED;
  return decode_common(q, k, v, seqlens, o_part, lse_part, B, Hq, Hkv, Sk, D, num_splits, scale,
                       stream);
}

int attn_decode_fused(const void* q, const void* k, const void* v, const int* seqlens, float* o,
                      float* lse, float* o_part, float* lse_part, int* counters, int B, int Hq,
                      int Hkv, int Sk, int D, int num_splits, float scale, void* stream) {
  if (!o_part || !lse_part || !o || !lse || !counters) return ATTN_ERR_INVALID_ARG;
  const int chk = decode_check_args(q, k, v, B, Hq, Hkv, Sk, D, num_splits, scale, false);
  if (chk != ATTN_OK) return chk;
  if (!aligned16(o_part) || !aligned16(lse_part) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(counters) & 3u) != 0) return ATTN_ERR_MISALIGNED;
  if (seqlens != nullptr && (reinterpret_cast<uintptr_t>(seqlens) & 3u) != 0)
    return ATTN_ERR_MISALIGNED;
  int* status = status_word_device_ptr();
  if (status == nullptr) return ATTN_ERR_CUDA;
  const FusedCombine fused{o, lse, counters};
  const cudaError_t e =
      launch_decode_splitkv(q, k, v, o_part, lse_part, B, Hq, Hkv, Sk, D, num_splits, scale,
                            static_cast<cudaStream_t>(stream), status, seqlens, nullptr, &fused);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_decode_fused_counters(int B, int Hq, int Hkv, int* count) {
  if (count == nullptr) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  const long long n = static_cast<long long>(B) * Hkv * ((Hq / Hkv + 15) / 16);
  if (n > (1ll << 31) - 1) return ATTN_ERR_UNSUPPORTED;
  *count = static_cast<int>(n);
  return ATTN_OK;
}

namespace {

// The paged decode entry points' checks of the cache description; ATTN_OK or
// the status to return.  On success *paged describes the cache and *capacity is
// max_pages * page_size.
int paged_check_args(const int* block_table, const int* seqlens, int Hkv, int num_pages,
                     int page_size, int max_pages, int D, int B, PagedKV* paged, int* capacity) {
  if (!block_table || !seqlens) return ATTN_ERR_INVALID_ARG;
  if (num_pages <= 0 || page_size <= 0 || max_pages <= 0) return ATTN_ERR_INVALID_ARG;
  if (page_size % 32 != 0) return ATTN_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(block_table) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(seqlens) & 3u) != 0)
    return ATTN_ERR_MISALIGNED;
  const long long cap = static_cast<long long>(max_pages) * page_size;
  if (cap > kMaxSeq) return ATTN_ERR_UNSUPPORTED;
  if (Hkv > 0 && static_cast<long long>(num_pages) * Hkv > (1ll << 30)) return ATTN_ERR_UNSUPPORTED;
  if (Hkv > 0 && D > 0 &&
      static_cast<long long>(num_pages) * Hkv * page_size * D > kMaxElems)
    return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * max_pages > (1ll << 31) - 1) return ATTN_ERR_UNSUPPORTED;
  *paged = PagedKV{block_table, page_size, max_pages, num_pages};
  *capacity = static_cast<int>(cap);
  return ATTN_OK;
}

}  // namespace

int attn_decode_fused_paged(const void* q, const void* k_cache, const void* v_cache,
                            const int* block_table, const int* seqlens, float* o, float* lse,
                            float* o_part, float* lse_part, int* counters, int B, int Hq, int Hkv,
                            int num_pages, int page_size, int max_pages, int D, int num_splits,
                            float scale, void* stream) {
  PagedKV paged;
  int capacity = 0;
  const int pchk = paged_check_args(block_table, seqlens, Hkv, num_pages, page_size, max_pages,
                                    D, B, &paged, &capacity);
  if (pchk != ATTN_OK) return pchk;
  if (!o_part || !lse_part || !o || !lse || !counters) return ATTN_ERR_INVALID_ARG;
  // The contiguous-size checks apply to the capacity; the cache itself is
  // num_pages pages, checked above.
  const int chk = decode_check_args(q, k_cache, v_cache, B, Hq, Hkv, capacity, D, num_splits,
                                    scale, true);
  if (chk != ATTN_OK) return chk;
  if (!aligned16(o_part) || !aligned16(lse_part) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(counters) & 3u) != 0) return ATTN_ERR_MISALIGNED;
  int* status = status_word_device_ptr();
  if (status == nullptr) return ATTN_ERR_CUDA;
  const FusedCombine fused{o, lse, counters};
  const cudaError_t e = launch_decode_splitkv(q, k_cache, v_cache, o_part, lse_part, B, Hq, Hkv,
                                              capacity, D, num_splits, scale,
                                              static_cast<cudaStream_t>(stream), status, seqlens,
                                              &paged, &fused);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_decode_splitkv_paged(const void* q, const void* k_cache, const void* v_cache,
                              const int* block_table, const int* seqlens, float* o_part,
                              float* lse_part, int B, int Hq, int Hkv, int num_pages,
                              int page_size, int max_pages, int D, int num_splits, float scale,
                              void* stream) {
  PagedKV paged;
  int capacity = 0;
  const int pchk = paged_check_args(block_table, seqlens, Hkv, num_pages, page_size, max_pages,
                                    D, B, &paged, &capacity);
  if (pchk != ATTN_OK) return pchk;
  // The contiguous-size checks of decode_common apply to the capacity; the
  // cache itself is num_pages pages, checked above.
  return decode_common(q, k_cache, v_cache, seqlens, o_part, lse_part, B, Hq, Hkv, capacity, D,
                       num_splits, scale, stream, &paged);
}

int attn_bwd(const void* q, const void* k, const void* v, const float* o, const float* lse,
             const void* dout, float* dq, float* dk, float* dv, float* delta_ws, int B, int Hq,
             int Hkv, int Sq, int Sk, int D, int causal, float scale, void* stream) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !delta_ws)
    return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (Sq > kMaxSeq || Sk > kMaxSeq) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq * Sq * D > kMaxElems ||
      static_cast<long long>(B) * Hkv * Sk * D > kMaxElems)
    return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq * ((Sq + 127) / 128) > (1ll << 30) ||
      static_cast<long long>(B) * Hkv * ((Sk + 127) / 128) > (1ll << 30))
    return ATTN_ERR_UNSUPPORTED;
  // Delta rows are indexed with int.
  if (static_cast<long long>(B) * Hq * Sq > (1ll << 30)) return ATTN_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(delta_ws))
    return ATTN_ERR_MISALIGNED;
  int* status = status_word_device_ptr();
  if (status == nullptr) return ATTN_ERR_CUDA;
  const cudaError_t e =
      launch_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, delta_ws, B, Hq, Hkv, Sq, Sk, D, causal,
                      scale, static_cast<cudaStream_t>(stream), status);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_rope_table(float* table, int max_pos, int D, float base, void* stream) {
  if (!table) return ATTN_ERR_INVALID_ARG;
  if (max_pos <= 0 || D <= 0 || D % 2 != 0) return ATTN_ERR_INVALID_ARG;
  if (!(base > 1.f) || !std::isfinite(base)) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(max_pos) * D > kMaxElems) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(table)) return ATTN_ERR_MISALIGNED;
  const cudaError_t e = launch_rope_table(table, max_pos, D, static_cast<double>(base),
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_qkv_rope(const void* x, const void* w, const float* rope_table, const int* positions,
                  void* q, void* k, void* v, int B, int S, int hidden, int Hq, int Hkv, int D,
                  int max_pos, int style, void* stream) {
  if (!x || !w || !rope_table || !q || !k || !v) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || S <= 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_pos <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (style != 0 && style != 1) return ATTN_ERR_INVALID_ARG;
  if (positions == nullptr && max_pos < S) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256) return ATTN_ERR_UNSUPPORTED;
  if (hidden % 8 != 0) return ATTN_ERR_UNSUPPORTED;  // TMA row pitch: a multiple of 16 bytes
  const long long T = static_cast<long long>(B) * S;
  const long long N = static_cast<long long>(Hq + 2ll * Hkv) * D;
  if (T > (1ll << 30) || N > (1ll << 30)) return ATTN_ERR_UNSUPPORTED;
  if (T * hidden > kMaxElems || N * hidden > kMaxElems || T * N > kMaxElems)
    return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w) || !aligned16(rope_table) || !aligned16(q) ||
      !aligned16(k) || !aligned16(v))
    return ATTN_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(positions) & 3u) != 0) return ATTN_ERR_MISALIGNED;
  int* status = status_word_device_ptr();
  if (status == nullptr) return ATTN_ERR_CUDA;
  const cudaError_t e = launch_qkv_rope(x, w, rope_table, positions, q, k, v, B, S, hidden, Hq,
                                        Hkv, D, max_pos, style,
                                        static_cast<cudaStream_t>(stream), status);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_decode_num_splits(int B, int Hq, int Hkv, int Sk, int D, int* num_splits) {
  if (num_splits == nullptr) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sk <= 0 || D <= 0 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  const int n_sm = sm_count();
  if (n_sm <= 0) return ATTN_ERR_CUDA;
  // CTAs without splitting: (batch, KV head, 16-head slice of the group).
  const long long base = static_cast<long long>(B) * Hkv * ((Hq / Hkv + 15) / 16);
  long long ns = 1;
  if (base * 5 < static_cast<long long>(n_sm) * 4) {
    // Too few to stream at full bandwidth.  At D = 256 a decode CTA takes a
    // whole SM, so the CTAs must fit in one wave: floor(SMs / base).  Otherwise
    // about one CTA per SM (two at D = 64, whose CTAs are lighter), rounded to
    // the nearest power of two: with power-of-two caches the splits then cut the
    // keys into whole 128-key groups (four warps x 32 keys), and the measured
    // optimum sat there (B1 Hq32 Hkv8 Sk32768: 16 splits 27.5 us, 19 splits
    // 28.2; B4 Hq32 Hkv4 Sk32768 D64: 16 splits 28.9, 10 splits 30.4).
    if (D == 256) {
      ns = n_sm / base > 1 ? n_sm / base : 1;
    } else {
      const long long ctas = (D == 64 ? 2ll : 1ll) * n_sm;
      const double t = static_cast<double>((ctas + base - 1) / base);
      ns = 1ll << std::lround(std::log2(t));
    }
    // Each split keeps at least 128 KB of K and V per KV head (128 keys at
    // D = 256, 256 at D = 128, 512 at D = 64): single-sequence B1 Hq32 Hkv8 Sk4096 gets 16
    // splits, 8.9 us against the 13.4 of an earlier 1024-key floor, and
    // B1 Hq32 Hkv8 Sk8192 D64 16 splits (11.1 us; 32 splits 13.9).  At most 32
    // splits, the combine's one pass over a warp of partials: with one or two
    // CTAs per split more only lengthen the combine's serial loop over them
    // (B1 Hq8 Hkv1 Sk16384: 64 splits 16.7 us, 32 13.4).
    if (ns > 32) ns = 32;
    const long long min_keys = 32768 / D;
    const long long cap = Sk / min_keys > 1 ? Sk / min_keys : 1;
    if (ns > cap) ns = cap;
  }
  *num_splits = static_cast<int>(ns);
  return ATTN_OK;
}

int attn_combine(const float* o_part, const float* lse_part, float* o, float* lse, int B, int Hq,
                 int D, int num_splits, void* stream) {
  if (!o_part || !lse_part || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || D <= 0 || num_splits < 1) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(num_splits) * B * Hq * D > kMaxElems ||
      static_cast<long long>(B) * Hq > (1ll << 30))
    return ATTN_ERR_UNSUPPORTED;
  if (D != 64 && D != 128 && D != 256) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(o_part) || !aligned16(lse_part) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_MISALIGNED;
  const cudaError_t e = launch_combine(o_part, lse_part, o, lse, B * Hq, D, num_splits,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_wait_selftest(unsigned long long limit_ns, unsigned long long* waited_ns, void* stream) {
  if (limit_ns < 1000ull || limit_ns > 1000000000ull) return ATTN_ERR_INVALID_ARG;
  if (waited_ns != nullptr && (reinterpret_cast<uintptr_t>(waited_ns) & 7u) != 0)
    return ATTN_ERR_MISALIGNED;
  int* status = status_word_device_ptr();
  if (status == nullptr) return ATTN_ERR_CUDA;
  const cudaError_t e =
      launch_wait_selftest(limit_ns, status, reinterpret_cast<uint64_t*>(waited_ns),
                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_debug_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  int value = 0;
  if (cudaMemcpyFromSymbol(&value, g_status_word, sizeof(int)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  return value;
}

}  // extern "C"
