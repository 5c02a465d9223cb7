// attn_decode.cu -- split-KV decode (one query row per head) and the
// log-sum-exp combine of its partials.
//
// Source: "A Thread-Register Decoupled GPU Execution Model for Efficient Tensor
// Computation", Methodology and Evaluation: decode attention (FlashDecoding) is
// GEMV plus softmax, highly memory bound, and does not use the tensor cores.
// The kernel therefore streams K and V once from HBM through shared memory with
// bulk copies and does the arithmetic on the CUDA cores in fp32.
//
// decode kernel, one CTA per (split, KV head, batch) [x 4-head slice of the
// query group when the group is wider than 4]:
//   * the CTA's 4 query heads share every K/V byte it reads (GQA);
//   * each of its 4 warps owns every 4th block of 32 keys of the split and
//     keeps its own online-softmax state; each warp has a private ring of
//     shared-memory slots filled by cp.async.bulk (K block, V block, K, V, ...),
//     so warps never wait on each other while streaming;
//   * inside a warp, lanes form 4 groups of 8; a group works on one key at a
//     time, each lane holding D/8 dimensions: QK partial dot products are
//     reduced across the 8 lanes with a reduce-scatter (3 shuffle rounds), so
//     afterwards lane `sub` of group `grp` owns the scores of key 4*sub+grp;
//   * P*V accumulates into per-lane registers (4 heads x D/8 dims); the warps'
//     states are merged through shared memory at the end.
// Scores are kept in the log2 domain: q is pre-multiplied by scale*log2(e).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int kHeads = 4;    // query heads per CTA
constexpr int kBlk = 32;     // keys per block
constexpr int kWarps = 4;    // warps per CTA
constexpr int kSlots = 3;    // ring slots per warp
constexpr float kLn2 = 0.69314718055994531f;

template <int D>
struct DecodeSmem {
  alignas(128) uint8_t ring[kWarps][kSlots][kBlk * D * 2];
  alignas(16) float p[kWarps][kBlk][kHeads];   // this block's softmax numerators
  alignas(16) float red_o[kWarps][kHeads][D];  // per-warp partial outputs
  float red_m[kWarps][kHeads];
  float red_l[kWarps][kHeads];
  alignas(8) uint64_t full[kWarps][kSlots];
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void record_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32, 2)
    decode_splitkv_kernel(const __nv_bfloat16* __restrict__ q,
                          const __nv_bfloat16* __restrict__ k,
                          const __nv_bfloat16* __restrict__ v, float* __restrict__ o_part,
                          float* __restrict__ lse_part, int B, int Hq, int Hkv, int Sk,
                          int chunk, int head_slices, float qscale, int* status) {
  constexpr int NCH = D / 64;           // 16-byte chunks per lane per row
  constexpr int DL = 8 * NCH;           // dimensions per lane
  constexpr uint32_t kRowBytes = D * 2;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecodeSmem<D>& sm = *reinterpret_cast<DecodeSmem<D>*>(smem_raw);

  const int split = blockIdx.x;
  const int g = blockIdx.y / head_slices;
  const int slice = blockIdx.y % head_slices;
  const int b = blockIdx.z;
  const int G = Hq / Hkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grp = lane >> 3;
  const int sub = lane & 7;

  const long long kb64 = static_cast<long long>(split) * chunk;
  const int key_begin = kb64 < Sk ? static_cast<int>(kb64) : Sk;
  const int key_end = min(key_begin + chunk, Sk);
  const int nkeys = key_end - key_begin;
  const int nblk = (nkeys + kBlk - 1) / kBlk;
  const int my_nblk = warp < nblk ? (nblk - warp + kWarps - 1) / kWarps : 0;
  const int nloads = 2 * my_nblk;

  const size_t kv_off = (static_cast<size_t>(b) * Hkv + g) * static_cast<size_t>(Sk) * D;
  const __nv_bfloat16* kbase = k + kv_off;
  const __nv_bfloat16* vbase = v + kv_off;

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kSlots; ++s) mbar_init(&sm.full[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const uint64_t policy = policy_evict_first();
  // Load number li of this warp: even = K block, odd = V block of its (li/2)-th block.
  auto issue = [&](int li) {
    const int blk = warp + (li >> 1) * kWarps;
    const int key0 = key_begin + blk * kBlk;
    const int rows = min(kBlk, key_end - key0);
    const __nv_bfloat16* src = ((li & 1) ? vbase : kbase) + static_cast<size_t>(key0) * D;
    const int slot = li % kSlots;
    const uint32_t bytes = static_cast<uint32_t>(rows) * kRowBytes;
    mbar_arrive_expect_tx(&sm.full[warp][slot], bytes);
    bulk_load(sm.ring[warp][slot], src, bytes, &sm.full[warp][slot], policy);
  };
  int issued = 0;
  if (lane == 0) {
    for (; issued < kSlots && issued < nloads; ++issued) issue(issued);
  }

  // This CTA's query heads: slice*4 + t of the group, t < 4.
  float qf[kHeads][DL];
#pragma unroll
  for (int t = 0; t < kHeads; ++t) {
    const int hl = slice * kHeads + t;
    if (hl < G) {
      const int hq = g * G + hl;
      const uint4* qrow =
          reinterpret_cast<const uint4*>(q + (static_cast<size_t>(b) * Hq + hq) * D);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        float f[8];
        bf16x8_to_f32(__ldg(qrow + c * 8 + sub), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) qf[t][c * 8 + e] = f[e] * qscale;
      }
    } else {
#pragma unroll
      for (int d = 0; d < DL; ++d) qf[t][d] = 0.f;
    }
  }

  float m_run[kHeads], l_lane[kHeads], acc[kHeads][DL];
#pragma unroll
  for (int t = 0; t < kHeads; ++t) {
    m_run[t] = -INFINITY;
    l_lane[t] = 0.f;
#pragma unroll
    for (int d = 0; d < DL; ++d) acc[t][d] = 0.f;
  }

  bool ok = true;
  int consumed = 0;
  for (int i = 0; i < my_nblk && ok; ++i) {
    const int blk = warp + i * kWarps;
    const int key0 = key_begin + blk * kBlk;
    const int nvalid = min(kBlk, key_end - key0);

    // ---------------- K block: scores for 32 keys x 4 heads
    {
      const int li = 2 * i;
      const int slot = li % kSlots;
      ok = mbar_wait(&sm.full[warp][slot], (li / kSlots) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      consumed = li + 1;
      const uint8_t* kb = sm.ring[warp][slot];
      float part[32];  // index 4*t + head, key 4*t + grp
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const uint4* row = reinterpret_cast<const uint4*>(kb + (4 * t + grp) * kRowBytes);
        float kf[DL];
#pragma unroll
        for (int c = 0; c < NCH; ++c) bf16x8_to_f32(row[c * 8 + sub], kf + c * 8);
#pragma unroll
        for (int h = 0; h < kHeads; ++h) {
          float s = 0.f;
#pragma unroll
          for (int d = 0; d < DL; ++d) s = fmaf(qf[h][d], kf[d], s);
          part[4 * t + h] = s;
        }
      }
      // Reduce-scatter across the 8 lanes of the group.
#pragma unroll
      for (int i2 = 0; i2 < 16; ++i2) {
        const bool up = lane & 4;
        const float send = up ? part[i2] : part[i2 + 16];
        const float keep = up ? part[i2 + 16] : part[i2];
        part[i2] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
      }
#pragma unroll
      for (int i2 = 0; i2 < 8; ++i2) {
        const bool up = lane & 2;
        const float send = up ? part[i2] : part[i2 + 8];
        const float keep = up ? part[i2 + 8] : part[i2];
        part[i2] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
      }
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2) {
        const bool up = lane & 1;
        const float send = up ? part[i2] : part[i2 + 4];
        const float keep = up ? part[i2 + 4] : part[i2];
        part[i2] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
      }
      const int jj = 4 * sub + grp;  // the key whose scores this lane now owns
      const bool valid = jj < nvalid;
      float pv[kHeads];
#pragma unroll
      for (int h = 0; h < kHeads; ++h) {
        const float sc = valid ? part[h] : -INFINITY;
        float mb = sc;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
          mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
        const float mn = fmaxf(m_run[h], mb);
        const float base = (mn == -INFINITY) ? 0.f : mn;
        const float alpha = ex2(m_run[h] - base);
        pv[h] = ex2(sc - base);
        m_run[h] = mn;
        l_lane[h] = fmaf(l_lane[h], alpha, pv[h]);
        if (alpha != 1.f) {  // warp-uniform: m_run and base are uniform
#pragma unroll
          for (int d = 0; d < DL; ++d) acc[h][d] *= alpha;
        }
      }
      *reinterpret_cast<float4*>(&sm.p[warp][jj][0]) = make_float4(pv[0], pv[1], pv[2], pv[3]);
      __syncwarp();
      if (lane == 0 && li + kSlots < nloads) {
        fence_proxy_async_smem();
        issue(li + kSlots);
        ++issued;
      }
    }

    // ---------------- V block: acc += p * V
    {
      const int li = 2 * i + 1;
      const int slot = li % kSlots;
      ok = mbar_wait(&sm.full[warp][slot], (li / kSlots) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      consumed = li + 1;
      const uint8_t* vb = sm.ring[warp][slot];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int j = 4 * t + grp;
        if (j < nvalid) {
          const float4 pp = *reinterpret_cast<const float4*>(&sm.p[warp][j][0]);
          const float ph[4] = {pp.x, pp.y, pp.z, pp.w};
          const uint4* row = reinterpret_cast<const uint4*>(vb + j * kRowBytes);
          float vf[DL];
#pragma unroll
          for (int c = 0; c < NCH; ++c) bf16x8_to_f32(row[c * 8 + sub], vf + c * 8);
#pragma unroll
          for (int h = 0; h < kHeads; ++h)
#pragma unroll
            for (int d = 0; d < DL; ++d) acc[h][d] = fmaf(ph[h], vf[d], acc[h][d]);
        }
      }
      __syncwarp();
      if (lane == 0 && li + kSlots < nloads) {
        fence_proxy_async_smem();
        issue(li + kSlots);
        ++issued;
      }
    }
  }

  if (!ok) {
    // A wait expired: report it, let this warp's copies in flight land, and
    // finish without further use of the ring.
    record_status(status, ATTN_ERR_TIMEOUT);
    if (lane == 0) {
      for (int li = consumed; li < issued; ++li)
        (void)mbar_wait(&sm.full[warp][li % kSlots], (li / kSlots) & 1);
    }
    __syncwarp();
  }

  // ---------------- merge: lanes of a warp, then the warps of the CTA
#pragma unroll
  for (int h = 0; h < kHeads; ++h) {
    float l = l_lane[h];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    l_lane[h] = l;
#pragma unroll
    for (int d = 0; d < DL; ++d) {
      float a = acc[h][d];
      a += __shfl_xor_sync(0xffffffffu, a, 8);
      a += __shfl_xor_sync(0xffffffffu, a, 16);
      acc[h][d] = a;
    }
  }
  if (grp == 0) {
#pragma unroll
    for (int h = 0; h < kHeads; ++h)
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        float4* dst = reinterpret_cast<float4*>(&sm.red_o[warp][h][c * 64 + sub * 8]);
        dst[0] = make_float4(acc[h][c * 8 + 0], acc[h][c * 8 + 1], acc[h][c * 8 + 2],
                             acc[h][c * 8 + 3]);
        dst[1] = make_float4(acc[h][c * 8 + 4], acc[h][c * 8 + 5], acc[h][c * 8 + 6],
                             acc[h][c * 8 + 7]);
      }
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < kHeads; ++h) {
      sm.red_m[warp][h] = m_run[h];
      sm.red_l[warp][h] = l_lane[h];
    }
  }
  __syncthreads();

  // Thread layout for the final merge: head h = warp, D/32 dims per lane.
  {
    const int h = warp;
    const int hl = slice * kHeads + h;
    if (hl < G) {
      const int hq = g * G + hl;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.red_m[w][h]);
      constexpr int DPL = D / 32;
      float out[DPL];
      float lse;
      if (M == -INFINITY) {
#pragma unroll
        for (int e = 0; e < DPL; ++e) out[e] = 0.f;
        lse = -INFINITY;
      } else {
        float L = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) out[e] = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float wt = ex2(sm.red_m[w][h] - M);
          L = fmaf(wt, sm.red_l[w][h], L);
#pragma unroll
          for (int e = 0; e < DPL; ++e) out[e] = fmaf(wt, sm.red_o[w][h][lane * DPL + e], out[e]);
        }
        const float inv = 1.f / L;
#pragma unroll
        for (int e = 0; e < DPL; ++e) out[e] *= inv;
        lse = (M + log2f(L)) * kLn2;
      }
      const size_t row = (static_cast<size_t>(split) * B + b) * Hq + hq;
      float* dst = o_part + row * D + lane * DPL;
      if constexpr (DPL == 4) {
        *reinterpret_cast<float4*>(dst) = make_float4(out[0], out[1], out[2], out[3]);
      } else {
        *reinterpret_cast<float2*>(dst) = make_float2(out[0], out[1]);
      }
      if (lane == 0) lse_part[row] = lse;
    }
  }
}

// One warp per output row: lse = ln sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s.
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ o_part,
                                                      const float* __restrict__ lse_part,
                                                      float* __restrict__ o,
                                                      float* __restrict__ lse, int rows,
                                                      int num_splits) {
  constexpr int DPL = D / 32;
  constexpr float kLog2e = 1.4426950408889634f;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float M = -INFINITY;
  for (int s = 0; s < num_splits; ++s)
    M = fmaxf(M, __ldg(lse_part + static_cast<size_t>(s) * rows + row));
  float out[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) out[e] = 0.f;
  float L;
  if (M == -INFINITY) {
    L = -INFINITY;
  } else {
    float W = 0.f;
    for (int s = 0; s < num_splits; ++s) {
      const size_t r = static_cast<size_t>(s) * rows + row;
      const float w = ex2((__ldg(lse_part + r) - M) * kLog2e);
      W += w;
      const float* src = o_part + r * D + lane * DPL;
      if constexpr (DPL == 4) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(src));
        out[0] = fmaf(w, x.x, out[0]);
        out[1] = fmaf(w, x.y, out[1]);
        out[2] = fmaf(w, x.z, out[2]);
        out[3] = fmaf(w, x.w, out[3]);
      } else {
        const float2 x = __ldg(reinterpret_cast<const float2*>(src));
        out[0] = fmaf(w, x.x, out[0]);
        out[1] = fmaf(w, x.y, out[1]);
      }
    }
    const float inv = 1.f / W;
#pragma unroll
    for (int e = 0; e < DPL; ++e) out[e] *= inv;
    L = M + logf(W);
  }
  float* dst = o + static_cast<size_t>(row) * D + lane * DPL;
  if constexpr (DPL == 4) {
    *reinterpret_cast<float4*>(dst) = make_float4(out[0], out[1], out[2], out[3]);
  } else {
    *reinterpret_cast<float2*>(dst) = make_float2(out[0], out[1]);
  }
  if (lane == 0) lse[row] = L;
}

template <int D>
cudaError_t launch_decode_impl(const void* q, const void* k, const void* v, float* o_part,
                               float* lse_part, int B, int Hq, int Hkv, int Sk, int num_splits,
                               float scale, cudaStream_t stream, int* status) {
  const int G = Hq / Hkv;
  const int head_slices = (G + kHeads - 1) / kHeads;
  const int chunk = (Sk + num_splits - 1) / num_splits;
  const size_t smem = sizeof(DecodeSmem<D>);
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(decode_splitkv_kernel<D>),
                                   static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid(num_splits, Hkv * head_slices, B);
  const float qscale = scale * 1.4426950408889634f;
  decode_splitkv_kernel<D><<<grid, kWarps * 32, smem, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), o_part, lse_part, B, Hq, Hkv, Sk, chunk,
      head_slices, qscale, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_splitkv(const void* q, const void* k, const void* v, float* o_part,
                                  float* lse_part, int B, int Hq, int Hkv, int Sk, int D,
                                  int num_splits, float scale, cudaStream_t stream,
                                  int* status) {
  if (D == 128)
    return launch_decode_impl<128>(q, k, v, o_part, lse_part, B, Hq, Hkv, Sk, num_splits,
                                   scale, stream, status);
  return launch_decode_impl<64>(q, k, v, o_part, lse_part, B, Hq, Hkv, Sk, num_splits, scale,
                                stream, status);
}

cudaError_t launch_combine(const float* o_part, const float* lse_part, float* o, float* lse,
                           int rows, int D, int num_splits, cudaStream_t stream) {
  const dim3 grid((rows + 7) / 8);
  if (D == 128)
    combine_kernel<128><<<grid, 256, 0, stream>>>(o_part, lse_part, o, lse, rows, num_splits);
  else
    combine_kernel<64><<<grid, 256, 0, stream>>>(o_part, lse_part, o, lse, rows, num_splits);
  return cudaGetLastError();
}

}  // namespace attn

// ---------------------------------------------------------------------------
// attn_decode_noalloc: the decode above with its partials kept in a static
// device array instead of caller-supplied workspace, for callers that cannot
// allocate device memory when they call in.  The kernels are the same; only
// where the partials live differs.
// ---------------------------------------------------------------------------
#include <mutex>

namespace attn {
namespace {

// Scratch for the per-split partials: o_part [ns,B,Hq,D] then lse_part
// [ns,B,Hq].  Part of the module image, so every device that loads the
// library reserves it until the process exits.  In host code this name is
// only a host-side stand-in: kernels get the device address looked up below.
static __device__ __align__(256) float g_decode_scratch[ATTN_NOALLOC_SCRATCH_FLOATS];

constexpr int kScratchMaxDevices = 64;
std::mutex g_scratch_mutex;
float* g_scratch_dev_ptr[kScratchMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device, looked up once
// per device (with that device current) and cached.  nullptr on failure.
float* decode_scratch_ptr() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kScratchMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_dev_ptr[dev] == nullptr) {
    float* p = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_decode_scratch) != cudaSuccess)
      return nullptr;
    g_scratch_dev_ptr[dev] = p;
  }
  return g_scratch_dev_ptr[dev];
}

bool aligned16_ptr(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace attn

extern "C" int attn_decode_noalloc(const void* q, const void* k, const void* v, float* o,
                                   float* lse, int B, int Hq, int Hkv, int Sk, int D,
                                   int num_splits, float scale, void* stream) {
  using namespace attn;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sk <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (num_splits < 1 || num_splits > Sk) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hkv * Sk * D > (1ll << 40)) return ATTN_ERR_UNSUPPORTED;
  const int head_slices = (Hq / Hkv + 3) / 4;
  if (B > 65535 || static_cast<long long>(Hkv) * head_slices > 65535) return ATTN_ERR_UNSUPPORTED;
  // The partials must fit the static scratch array.
  const long long part_floats = static_cast<long long>(num_splits) * B * Hq * D;
  const long long lse_floats = static_cast<long long>(num_splits) * B * Hq;
  if (part_floats + lse_floats > static_cast<long long>(ATTN_NOALLOC_SCRATCH_FLOATS))
    return ATTN_ERR_UNSUPPORTED;
  if (!aligned16_ptr(q) || !aligned16_ptr(k) || !aligned16_ptr(v) || !aligned16_ptr(o) ||
      !aligned16_ptr(lse))
    return ATTN_ERR_MISALIGNED;
  float* scratch = decode_scratch_ptr();
  int* status = status_word_device_ptr();
  if (scratch == nullptr || status == nullptr) return ATTN_ERR_CUDA;
  float* o_part = scratch;                // D is a multiple of 64: lse_part stays 256-byte aligned
  float* lse_part = scratch + part_floats;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_decode_splitkv(q, k, v, o_part, lse_part, B, Hq, Hkv, Sk, D, num_splits,
                                        scale, s, status);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  e = launch_combine(o_part, lse_part, o, lse, B * Hq, D, num_splits, s);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
