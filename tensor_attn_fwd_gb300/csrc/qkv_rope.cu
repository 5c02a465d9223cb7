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
// GEMM  Y[T, N] = X[T, hidden] W[N, hidden]^T,  N = (Hq + 2 Hkv) D, on tcgen05,
// K in steps of 64 (one 128B-swizzled box), fp32 accumulator in TMEM, two
// accumulator buffers (2 x 256 columns) so that the epilogue of one tile
// overlaps the MMAs of the next.  Persistent grid, one CTA per SM.  Two forms:
//   single  tile 128 tokens x 256 features per CTA; 4-stage ring of
//           A 16 KB + B 32 KB (K = 64 per stage).
//   pair    a cluster of two CTAs on neighbouring SMs computes 256 tokens x
//           256 features with tcgen05.mma.cta_group::2 (M = 256) issued by the
//           even CTA: each CTA stages its own 128 token rows of X and half of
//           the 256 weight rows (N is split across the pair), so K = 64 costs
//           A 16 KB + B 16 KB per SM for the same work per SM -- a third less
//           shared-memory fill per FLOP.  A stage holds K = 128 (3 stages of
//           64 KB), i.e. 8 MMAs per barrier wait and commit.  Full barriers live in
//           the even CTA and count both CTAs' copies; MMA completions are
//           multicast to both CTAs; both CTAs' epilogue threads release an
//           accumulator buffer on the even CTA's barrier.
// Roles (192 threads): warp 0 TMA, warp 1 MMA (each a whole warp; one elected
// lane issues),
// warps 2-5 epilogue (thread = token row = TMEM lane): tcgen05.ld of the
// accumulator, rotation with a (cos, sin) table, bf16 rounding, store into
// Q / K / V.  Rows past T, and features past N, are loaded as zeros by TMA and
// never stored.  All waits are bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int kBM = 128, kBN = 256, kBK = 64;  // rows per CTA, features per tile, TMA box K
constexpr int kGThreads = 192;
constexpr uint32_t kASub = kBM * kBK * 2;  // one [128 rows x 64] A box: 16 KB

template <bool kPair>
struct GCfg {
  static constexpr uint32_t kBRows = kPair ? kBN / 2 : kBN;  // weight rows staged per CTA
  // K per stage: two 64-wide boxes per operand in the pair form (8 MMAs per
  // barrier wait and commit), one in the single form.
  static constexpr int kSubK = kPair ? 2 : 1;
  static constexpr int kStageK = kSubK * kBK;
  static constexpr uint32_t kBSub = kBRows * kBK * 2;
  static constexpr uint32_t kABytes = kSubK * kASub;
  static constexpr uint32_t kBBytes = kSubK * kBSub;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = kPair ? 3 : 4;
  static constexpr size_t kSmem = 1024 + size_t(kStages) * kStageBytes + 256;
  static_assert(kSmem <= 232448, "shared memory per CTA");
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kPair ? 2 * kBM : kBM, kBN, false, false);
};
constexpr int kGMaxStages = 6;

struct GBars {
  uint64_t full[kGMaxStages], empty[kGMaxStages];
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

// Bounded wait; in the pair form barriers are also signalled from the peer
// CTA, so the wait acquires at cluster scope.
template <bool kPair>
__device__ __forceinline__ bool gwait(uint64_t* bar, uint32_t parity, GBars* bars) {
  const uint32_t a = smem_u32(bar);
  auto probe = [&] { return kPair ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity); };
  if (probe()) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (probe()) return true;
    if (*reinterpret_cast<volatile int*>(&bars->abort)) return false;
    if (globaltimer() - t0 > ATTN_WAIT_NS) {
      *reinterpret_cast<volatile int*>(&bars->abort) = 1;
      return false;
    }
  }
}

// The wait for a whole converged warp (the TMA and MMA roles run as whole warps
// and issue from one elected lane); the vote keeps the outcome uniform.  Used
// once per output tile.  Per K stage those warps wait without a vote: each lane
// keeps its outcome, issue continues with in-bounds addresses, and one vote per
// tile makes the stop decision uniform; a lane still polling is waited for by
// the next elect.sync.
template <bool kPair>
__device__ __forceinline__ bool gwait_w(uint64_t* bar, uint32_t parity, GBars* bars) {
  return __all_sync(0xffffffffu, gwait<kPair>(bar, parity, bars));
}

// Work slots: one per CTA (single) or one per CTA pair.
template <bool kPair>
__device__ __forceinline__ int g_slot() {
  return kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
}
template <bool kPair>
__device__ __forceinline__ int g_slots() {
  return kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
}

template <bool kPair>
__device__ void g_load(const CUtensorMap* tmX, const CUtensorMap* tmW, const QkvParams& p,
                       uint8_t* ring, GBars* bars) {
  using C = GCfg<kPair>;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  uint32_t ctr = 0;
  bool ok = true;
  const int total = p.mt * p.nt;
  for (int t = g_slot<kPair>(); t < total && ok; t += g_slots<kPair>()) {
    const int m0 = (t / p.nt) * (kPair ? 2 * kBM : kBM) + int(rank) * kBM;
    const int n0 = (t % p.nt) * kBN + int(rank) * int(C::kBRows);
    bool good = true;
    for (int kb = 0; kb < p.kb; ++kb) {
      const uint32_t st = ctr % C::kStages;
      if (ctr >= uint32_t(C::kStages))
        good &= gwait<kPair>(&bars->empty[st], ((ctr / C::kStages) - 1) & 1, bars);
      uint8_t* sA = ring + st * C::kStageBytes;
      // Boxes past `hidden` are zero-filled by TMA and still deliver their bytes.
      if (elect_one()) {
        if constexpr (kPair) {
          // The even CTA's barrier counts both CTAs' bytes.
          if (rank == 0) mbar_arrive_expect_tx(&bars->full[st], 2 * C::kStageBytes);
          const uint32_t fb = mapa_shared(smem_u32(&bars->full[st]), 0);
#pragma unroll
          for (int sub = 0; sub < C::kSubK; ++sub) {
            const int x = kb * C::kStageK + sub * kBK;
            tma_load_3d_pair(sA + sub * kASub, tmX, fb, x, m0, 0);
            tma_load_3d_pair(sA + C::kABytes + sub * C::kBSub, tmW, fb, x, n0, 0);
          }
        } else {
          mbar_arrive_expect_tx(&bars->full[st], C::kStageBytes);
#pragma unroll
          for (int sub = 0; sub < C::kSubK; ++sub) {
            const int x = kb * C::kStageK + sub * kBK;
            tma_load_3d(sA + sub * kASub, tmX, &bars->full[st], x, m0, 0);
            tma_load_3d(sA + C::kABytes + sub * C::kBSub, tmW, &bars->full[st], x, n0, 0);
          }
        }
      }
      __syncwarp();
      ++ctr;
    }
    ok = __all_sync(0xffffffffu, good);
  }
  if (!ok) gnote(p.status, ATTN_ERR_TIMEOUT);
  // Let every copy issued land before the CTA can exit (in the pair form the
  // even CTA's barriers count both CTAs' copies, and the closing cluster
  // barrier keeps the odd CTA alive until then).
  if (rank == 0)
    for (uint32_t c = (ctr > uint32_t(C::kStages) ? ctr - C::kStages : 0); c < ctr; ++c)
      (void)mbar_wait(&bars->full[c % C::kStages], (c / C::kStages) & 1);
}

template <bool kPair>
__device__ void g_mma(const QkvParams& p, uint8_t* ring, GBars* bars, uint32_t tmem) {
  using C = GCfg<kPair>;
  constexpr uint64_t kDesc = sdesc_sw128(0, 16, 1024);  // K-major, 128B swizzle
  constexpr uint32_t kHi = static_cast<uint32_t>(kDesc >> 32);
  const uint32_t lo0 = static_cast<uint32_t>(kDesc) + (smem_u32(ring) >> 4);
  auto commit = [&](uint64_t* bar) {  // completion to both CTAs of a pair
    if constexpr (kPair)
      tc_commit_pair_mc_w(smem_u32(bar), 0x3);
    else
      tc_commit_w(bar);
  };
  uint32_t ctr = 0, i = 0;
  bool ok = true;
  const int total = p.mt * p.nt;
  for (int t = g_slot<kPair>(); t < total && ok; t += g_slots<kPair>(), ++i) {
    const uint32_t a = i & 1;
    if (i >= 2 && !(ok = gwait_w<kPair>(&bars->acc_empty[a], ((i >> 1) - 1) & 1, bars))) break;
    tc_fence_after();
    const uint32_t d = tmem + a * kBN;
    bool good = true;
    for (int kb = 0; kb < p.kb; ++kb) {
      const uint32_t st = ctr % C::kStages;
      good &= gwait<kPair>(&bars->full[st], (ctr / C::kStages) & 1, bars);
      tc_fence_after();
      const uint32_t sa = lo0 + ((st * C::kStageBytes) >> 4);
      const uint32_t sb = sa + (C::kABytes >> 4);
#pragma unroll
      for (int kk = 0; kk < C::kStageK / 16; ++kk) {
        const int sub = kk >> 2;
        const uint64_t ad = desc_from_words(sa + ((sub * kASub + (kk & 3) * 32) >> 4), kHi);
        const uint64_t bd = desc_from_words(sb + ((sub * C::kBSub + (kk & 3) * 32) >> 4), kHi);
        if constexpr (kPair) {
          if (kb == 0 && kk == 0)
            mma_ss_pair_w<0>(d, ad, bd, C::kIdesc);
          else
            mma_ss_pair_w<1>(d, ad, bd, C::kIdesc);
        } else {
          if (kb == 0 && kk == 0)
            mma_ss_w<0>(d, ad, bd, C::kIdesc);
          else
            mma_ss_w<1>(d, ad, bd, C::kIdesc);
        }
      }
      commit(&bars->empty[st]);
      ++ctr;
    }
    if (!(ok = __all_sync(0xffffffffu, good))) break;
    commit(&bars->acc_full[a]);
  }
  if (!ok) gnote(p.status, ATTN_ERR_TIMEOUT);
  if constexpr (kPair)
    tc_commit_pair_mc_w(smem_u32(&bars->mma_done), 0x1);
  else
    tc_commit_w(&bars->mma_done);
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

template <bool kPair>
__device__ void g_epilogue(const QkvParams& p, GBars* bars, uint32_t tmem, int warp, int lane) {
  const int quarter = warp & 3;  // TMEM lanes this warp may access
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
  const int half = p.D / 2;
  uint32_t i = 0;
  bool ok = true;
  const int total = p.mt * p.nt;
  for (int t = g_slot<kPair>(); t < total && ok; t += g_slots<kPair>(), ++i) {
    const uint32_t a = i & 1;
    ok = __all_sync(0xffffffffu, gwait<kPair>(&bars->acc_full[a], (i >> 1) & 1, bars));
    if (!ok) break;
    tc_fence_after();
    const int m0 = (t / p.nt) * (kPair ? 2 * kBM : kBM) + int(rank) * kBM;
    const int n0 = (t % p.nt) * kBN;
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
    // warp may reuse it (in the pair form: the even CTA's barrier).
    tc_fence_before();
    if constexpr (kPair)
      mbar_arrive_cluster(mapa_shared(smem_u32(&bars->acc_empty[a]), 0));
    else
      mbar_arrive(&bars->acc_empty[a]);
  }
  if (!ok) gnote(p.status, ATTN_ERR_TIMEOUT);
}

template <bool kPair>
__global__ void __launch_bounds__(kGThreads, 1)
    qkv_rope_kernel(const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmW, const QkvParams p) {
  using C = GCfg<kPair>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  GBars* bars = reinterpret_cast<GBars*>(ring + C::kStages * C::kStageBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool mma_cta = !kPair || cluster_ctarank() == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->acc_full[a], 1);
      mbar_init(&bars->acc_empty[a], kPair ? 256 : 128);  // every epilogue thread (of the pair)
    }
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(&bars->tmem_base, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&bars->tmem_base, 512);
      tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  }
  tc_fence_before();
  if constexpr (kPair)
    cluster_sync();  // both CTAs' barriers are initialised before any remote use
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  if (warp == 0) {
    g_load<kPair>(&tmX, &tmW, p, ring, bars);
  } else if (warp == 1) {
    if (mma_cta) g_mma<kPair>(p, ring, bars, tmem);
  } else {
    g_epilogue<kPair>(p, bars, tmem, warp, lane);
  }
  tc_fence_before();
  if constexpr (kPair)
    cluster_sync();  // no CTA leaves while its peer may still signal its barriers
  else
    __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem, 512);
    else
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
  p.nt = (p.N + kBN - 1) / kBN;
  // CTA pairs once there are at least 512 tokens (two 256-row tiles).
  const bool pair = p.T >= 4 * kBM;
  const int stage_k = pair ? GCfg<true>::kStageK : GCfg<false>::kStageK;
  p.kb = (hidden + stage_k - 1) / stage_k;
  CUtensorMap tmX, tmW;
  if (!encode_bf16_map(&tmX, x, hidden, p.T, 1, kBM) ||
      !encode_bf16_map(&tmW, w, hidden, p.N, 1, pair ? kBN / 2 : kBN))
    return cudaErrorInvalidValue;
  if (!pair) {
    p.mt = (p.T + kBM - 1) / kBM;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(qkv_rope_kernel<false>),
                                     static_cast<int>(GCfg<false>::kSmem));
    if (e != cudaSuccess) return e;
    const int total = p.mt * p.nt;
    const int grid = total < sm_count() ? total : sm_count();
    qkv_rope_kernel<false><<<grid, kGThreads, GCfg<false>::kSmem, stream>>>(tmX, tmW, p);
    return cudaGetLastError();
  }
  p.mt = (p.T + 2 * kBM - 1) / (2 * kBM);
  const void* kernel = reinterpret_cast<const void*>(qkv_rope_kernel<true>);
  cudaError_t e = ensure_smem_attr(kernel, static_cast<int>(GCfg<true>::kSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(kGThreads, 1, 1);
  cfg.dynamicSmemBytes = GCfg<true>::kSmem;
  cfg.stream = stream;
  // Clusters of two resident at once, per device (computed once; concurrent
  // first calls store the same value).
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int resident = max_clusters[dev].load(std::memory_order_relaxed);
  if (resident == 0) {
    cfg.gridDim = dim3(2, 1, 1);
    if (cudaOccupancyMaxActiveClusters(&resident, kernel, &cfg) != cudaSuccess || resident <= 0)
      resident = sm_count() / 2;
    max_clusters[dev].store(resident, std::memory_order_relaxed);
  }
  const int total = p.mt * p.nt;
  const int clusters = total < resident ? total : resident;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  e = cudaLaunchKernelEx(&cfg, qkv_rope_kernel<true>, tmX, tmW, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace attn
