// qkv_rope.cu -- QKV projection with the rotary embedding fused into its
// epilogue, writing Q, K and V in the attention kernels' [B, H, S, D] layout.
//
// Source: "A Thread-Register Decoupled GPU Execution Model for Efficient Tensor
// Computation", Background (a linear projection of the hidden states gives Q,
// K and V, each a GEMM with its weight matrix; RoPE is one of the vector
// operations around it) and "VDCores: Resource Decoupled Programming and
// Execution for Asynchronous GPUs", Evaluation (QKV-Projection + RoPE as a
// fused pattern).  The rotary embedding is the standard one:
//   theta_i = base^(-2i/D), angle = pos * theta_i,
//   (a, b) -> (a cos - b sin, a sin + b cos)
// on dims (2i, 2i+1) (style 0) or (i, i + D/2) (style 1), for Q and K heads.
//
// GEMM  Y[T, N] = X[T, hidden] W[N, hidden]^T,  N = (Hq + 2 Hkv) D, on tcgen05:
//   tile 128 tokens x 256 features, K in steps of 64 (one 128B-swizzled box),
//   4-stage TMA ring (A 16 KB + B 32 KB per stage), fp32 accumulator in TMEM,
//   two accumulator buffers (2 x 256 columns) so that the epilogue of one tile
//   overlaps the MMAs of the next.  Persistent grid, one CTA per SM.
// Roles (192 threads): warp 0 TMA (one thread), warp 1 MMA (one thread),
// warps 2-5 epilogue (thread = token row = TMEM lane): tcgen05.ld of the
// accumulator, rotation with a (cos, sin) table, bf16 rounding, store into
// Q / K / V.  Rows past T, and features past N, are loaded as zeros by TMA and
// never stored.  All waits are bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kGStages = 4;
constexpr int kGThreads = 192;
constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kBBytes = kBN * kBK * 2;  // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr size_t kGSmem = 1024 + size_t(kGStages) * kStageBytes + 256;
static_assert(kGSmem <= 232448, "shared memory per CTA");
constexpr uint32_t kIdescG = idesc_bf16_f32(kBM, kBN, false, false);

struct GBars {
  uint64_t full[kGStages], empty[kGStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(GBars) <= 256, "barrier block too large");

struct QkvParams {
  const float* rope;     // [max_pos, D/2, 2] (cos, sin)
  const int* positions;  // [T] or null (position = s)
  __nv_bfloat16* q;      // [B, Hq, S, D]
  __nv_bfloat16* k;      // [B, Hkv, S, D]
  __nv_bfloat16* v;      // [B, Hkv, S, D]
  int* status;
  int T, S, hidden, Hq, Hkv, D, N, max_pos, style;
  int mt, nt, kb;        // tiles along T and N, K blocks
};

__device__ __forceinline__ void gnote(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ bool gwait(uint64_t* bar, uint32_t parity, GBars* bars) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&bars->abort)) return false;
    if (globaltimer() - t0 > ATTN_WAIT_NS) {
      *reinterpret_cast<volatile int*>(&bars->abort) = 1;
      return false;
    }
  }
}

__device__ void g_load(const CUtensorMap* tmX, const CUtensorMap* tmW, const QkvParams& p,
                       uint8_t* ring, GBars* bars) {
  uint32_t ctr = 0;
  bool ok = true;
  const int total = p.mt * p.nt;
  for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
    const int m0 = (t / p.nt) * kBM, n0 = (t % p.nt) * kBN;
    for (int kb = 0; kb < p.kb; ++kb) {
      const uint32_t st = ctr % kGStages;
      if (ctr >= uint32_t(kGStages) &&
          !(ok = gwait(&bars->empty[st], ((ctr / kGStages) - 1) & 1, bars)))
        break;
      uint8_t* sA = ring + st * kStageBytes;
      mbar_arrive_expect_tx(&bars->full[st], kStageBytes);
      tma_load_3d(sA, tmX, &bars->full[st], kb * kBK, m0, 0);
      tma_load_3d(sA + kABytes, tmW, &bars->full[st], kb * kBK, n0, 0);
      ++ctr;
    }
  }
  if (!ok) gnote(p.status, ATTN_ERR_TIMEOUT);
  for (uint32_t c = (ctr > uint32_t(kGStages) ? ctr - kGStages : 0); c < ctr; ++c)
    (void)mbar_wait(&bars->full[c % kGStages], (c / kGStages) & 1);
}

__device__ void g_mma(const QkvParams& p, uint8_t* ring, GBars* bars, uint32_t tmem) {
  constexpr uint64_t kDesc = sdesc_sw128(0, 16, 1024);  // K-major, 128B swizzle
  constexpr uint32_t kHi = static_cast<uint32_t>(kDesc >> 32);
  const uint32_t lo0 = static_cast<uint32_t>(kDesc) + (smem_u32(ring) >> 4);
  uint32_t ctr = 0, i = 0;
  bool ok = true;
  const int total = p.mt * p.nt;
  for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++i) {
    const uint32_t a = i & 1;
    if (i >= 2 && !(ok = gwait(&bars->acc_empty[a], ((i >> 1) - 1) & 1, bars))) break;
    tc_fence_after();
    const uint32_t d = tmem + a * kBN;
    for (int kb = 0; kb < p.kb; ++kb) {
      const uint32_t st = ctr % kGStages;
      if (!(ok = gwait(&bars->full[st], (ctr / kGStages) & 1, bars))) break;
      tc_fence_after();
      const uint32_t sa = lo0 + ((st * kStageBytes) >> 4);
      const uint32_t sb = sa + (kABytes >> 4);
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint64_t ad = desc_from_words(sa + ((kk * 32) >> 4), kHi);
        const uint64_t bd = desc_from_words(sb + ((kk * 32) >> 4), kHi);
        if (kb == 0 && kk == 0)
          mma_ss_c<0>(d, ad, bd, kIdescG);
        else
          mma_ss_c<1>(d, ad, bd, kIdescG);
      }
      tc_commit(&bars->empty[st]);
      ++ctr;
    }
    if (!ok) break;
    tc_commit(&bars->acc_full[a]);
  }
  if (!ok) gnote(p.status, ATTN_ERR_TIMEOUT);
  tc_commit(&bars->mma_done);
  (void)mbar_wait(&bars->mma_done, 0);
}

// Store 32 fp32 values as bf16 (64 bytes) at dst.
__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst, const float* x) {
#pragma unroll
  for (int e = 0; e < 32; e += 8) {
    uint4 w;
    w.x = pack_bf16x2(x[e], x[e + 1]);
    w.y = pack_bf16x2(x[e + 2], x[e + 3]);
    w.z = pack_bf16x2(x[e + 4], x[e + 5]);
    w.w = pack_bf16x2(x[e + 6], x[e + 7]);
    *reinterpret_cast<uint4*>(dst + e) = w;
  }
}

__device__ void g_epilogue(const QkvParams& p, GBars* bars, uint32_t tmem, int warp, int lane) {
  const int quarter = warp & 3;  // TMEM lanes this warp may access
  const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
  const int half = p.D / 2;
  uint32_t i = 0;
  bool ok = true;
  const int total = p.mt * p.nt;
  for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++i) {
    const uint32_t a = i & 1;
    ok = __all_sync(0xffffffffu, gwait(&bars->acc_full[a], (i >> 1) & 1, bars));
    if (!ok) break;
    tc_fence_after();
    const int m0 = (t / p.nt) * kBM, n0 = (t % p.nt) * kBN;
    const int row = m0 + quarter * 32 + lane;
    const bool valid = row < p.T;
    int b = 0, s = 0, pos = 0;
    if (valid) {
      b = row / p.S;
      s = row - b * p.S;
      pos = p.positions != nullptr ? __ldg(p.positions + row) : s;
      if (pos < 0 || pos >= p.max_pos) {
        gnote(p.status, ATTN_ERR_INVALID_ARG);
        pos = min(max(pos, 0), p.max_pos - 1);
      }
    }
    const float2* cs_row = reinterpret_cast<const float2*>(p.rope) + static_cast<size_t>(pos) * half;
    for (int hh = 0; hh < kBN / p.D; ++hh) {
      const int n_h = n0 + hh * p.D;
      if (n_h >= p.N) break;
      const int head = n_h / p.D;
      __nv_bfloat16* base;
      int h, H;
      if (head < p.Hq) {
        base = p.q; h = head; H = p.Hq;
      } else if (head < p.Hq + p.Hkv) {
        base = p.k; h = head - p.Hq; H = p.Hkv;
      } else {
        base = p.v; h = head - p.Hq - p.Hkv; H = p.Hkv;
      }
      const bool rotate = head < p.Hq + p.Hkv;
      __nv_bfloat16* dst = base + ((static_cast<size_t>(b) * H + h) * p.S + s) * p.D;
      const uint32_t col0 = tmem + lane_addr + a * kBN + hh * p.D;
      if (!rotate || p.style == 0) {
        for (int c = 0; c < p.D; c += 32) {
          uint32_t r[32];
          tmem_ld32(col0 + c, r);
          float x[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(r[e]);
          if (rotate && valid) {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              // pairs (c+e, c+e+1) and (c+e+2, c+e+3): frequencies (c+e)/2, (c+e)/2+1
              const float4 cs = __ldg(reinterpret_cast<const float4*>(cs_row + (c + e) / 2));
              const float a0 = x[e], b0 = x[e + 1], a1 = x[e + 2], b1 = x[e + 3];
              x[e] = a0 * cs.x - b0 * cs.y;
              x[e + 1] = a0 * cs.y + b0 * cs.x;
              x[e + 2] = a1 * cs.z - b1 * cs.w;
              x[e + 3] = a1 * cs.w + b1 * cs.z;
            }
          }
          if (valid) store32_bf16(dst + c, x);
        }
      } else {
        for (int c = 0; c < half; c += 32) {
          uint32_t rl[32], rh[32];
          tmem_ld32(col0 + c, rl);
          tmem_ld32(col0 + half + c, rh);
          float lo[32], hi[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            lo[e] = __uint_as_float(rl[e]);
            hi[e] = __uint_as_float(rh[e]);
          }
          if (valid) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float4 cs = __ldg(reinterpret_cast<const float4*>(cs_row + c + e));
              const float a0 = lo[e], b0 = hi[e], a1 = lo[e + 1], b1 = hi[e + 1];
              lo[e] = a0 * cs.x - b0 * cs.y;
              hi[e] = a0 * cs.y + b0 * cs.x;
              lo[e + 1] = a1 * cs.z - b1 * cs.w;
              hi[e + 1] = a1 * cs.w + b1 * cs.z;
            }
            store32_bf16(dst + c, lo);
            store32_bf16(dst + half + c, hi);
          }
        }
      }
    }
    // Every tcgen05.ld of this buffer has completed (each waits); the MMA
    // warp may reuse it.
    tc_fence_before();
    mbar_arrive(&bars->acc_empty[a]);
  }
  if (!ok) gnote(p.status, ATTN_ERR_TIMEOUT);
}

__global__ void __launch_bounds__(kGThreads, 1)
    qkv_rope_kernel(const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmW, const QkvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  GBars* bars = reinterpret_cast<GBars*>(ring + kGStages * kStageBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->acc_full[a], 1);
      mbar_init(&bars->acc_empty[a], 128);
    }
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  if (warp == 0) {
    if (lane == 0) g_load(&tmX, &tmW, p, ring, bars);
  } else if (warp == 1) {
    if (lane == 0) g_mma(p, ring, bars, tmem);
  } else {
    g_epilogue(p, bars, tmem, warp, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// (cos, sin) of pos * base^(-2i/D) for pos < max_pos, i < D/2, computed in
// double precision and rounded to fp32.
__global__ void rope_table_kernel(float* table, int max_pos, int D, double log_base) {
  const long long n = static_cast<long long>(max_pos) * (D / 2);
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(idx % (D / 2));
    const long long pos = idx / (D / 2);
    const double theta = exp(-2.0 * i / D * log_base);
    double sn, cs;
    sincos(static_cast<double>(pos) * theta, &sn, &cs);
    table[2 * idx] = static_cast<float>(cs);
    table[2 * idx + 1] = static_cast<float>(sn);
  }
}

}  // namespace

cudaError_t launch_rope_table(float* table, int max_pos, int D, double base, cudaStream_t stream) {
  const long long n = static_cast<long long>(max_pos) * (D / 2);
  const int blocks = static_cast<int>(n / 256 + 1 < 4096 ? n / 256 + 1 : 4096);
  rope_table_kernel<<<blocks, 256, 0, stream>>>(table, max_pos, D, std::log(base));
  return cudaGetLastError();
}

cudaError_t launch_qkv_rope(const void* x, const void* w, const float* rope, const int* positions,
                            void* q, void* k, void* v, int B, int S, int hidden, int Hq, int Hkv,
                            int D, int max_pos, int style, cudaStream_t stream, int* status) {
  QkvParams p;
  p.rope = rope;
  p.positions = positions;
  p.q = static_cast<__nv_bfloat16*>(q);
  p.k = static_cast<__nv_bfloat16*>(k);
  p.v = static_cast<__nv_bfloat16*>(v);
  p.status = status;
  p.T = B * S;
  p.S = S;
  p.hidden = hidden;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.N = (Hq + 2 * Hkv) * D;
  p.max_pos = max_pos;
  p.style = style;
  p.mt = (p.T + kBM - 1) / kBM;
  p.nt = (p.N + kBN - 1) / kBN;
  p.kb = (hidden + kBK - 1) / kBK;
  CUtensorMap tmX, tmW;
  if (!encode_bf16_map(&tmX, x, hidden, p.T, 1, kBM) ||
      !encode_bf16_map(&tmW, w, hidden, p.N, 1, kBN))
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(qkv_rope_kernel),
                                   static_cast<int>(kGSmem));
  if (e != cudaSuccess) return e;
  const int total = p.mt * p.nt;
  const int grid = total < sm_count() ? total : sm_count();
  qkv_rope_kernel<<<grid, kGThreads, kGSmem, stream>>>(tmX, tmW, p);
  return cudaGetLastError();
}

}  // namespace attn
