// attn_bwd.cu -- attention backward (dQ, dK, dV) on sm_103a tensor cores.
//
// Source: "A Thread-Register Decoupled GPU Execution Model for Efficient Tensor
// Computation", Methodology and Evaluation (the FlashAttention backward: more
// GEMMs than the forward, more live tensors, operand transposes and score
// recomputation).  For O = softmax(S) V with S = scale * Q K^T (+ mask) and an
// upstream gradient dO:
//   P = exp(S - LSE)   Delta_i = sum_d dO_id O_id   dP = dO V^T
//   dS = P * (dP - Delta)   dV = P^T dO   dK = scale * dS^T Q   dQ = scale * dS K
// (dK and dV sum over the query heads that share a KV head).
//
// Three kernels, enqueued in order on the caller's stream:
//   delta kernel  Delta = rowsum(dO * O) into caller workspace.
//   dK/dV kernel  one CTA per 128-key tile of one KV head.  It loops over every
//                 (query head of the group, 128-row query tile) that sees those
//                 keys: S^T = K Q^T and dP^T = V dO^T (smem x smem) into TMEM;
//                 the gradient warps (one thread per key) turn them into P^T
//                 and dS^T (bf16, written back into TMEM over S^T / dP^T); then
//                 dV += P^T dO and dK += dS^T Q accumulate in TMEM.  No atomics.
//                 Per step the MMA warp issues dV(s) as soon as P^T(s) is in
//                 TMEM and S^T(s+1) right behind it (it overwrites P^T(s) only
//                 after dV has read it), so the gradient warps' dS^T(s) overlaps
//                 dV(s) and S^T(s+1); then dK(s) once dS^T(s) is in TMEM and
//                 dP^T(s+1), which overlap the exponentials of step s+1.
//   dQ kernel     persistent (one CTA per SM) over the 128-row query tiles,
//                 highest first: S = Q K^T and dP = dO V^T recomputed for each
//                 visible KV tile, dS written into TMEM, dQ += dS K accumulated
//                 in one of two TMEM buffers (a tile's epilogue overlaps the
//                 next tile's products; its Q and dO load once the current
//                 tile's last S and dP are done).  S(s+1) is issued as soon as
//                 the gradient warps have read S(s), so it overlaps their work
//                 on step s; K and V stream through separate rings (K is
//                 needed until dQ(s), V only until dP(s)).
// Roles (320 threads): warps 0-7 gradient math (two warpgroups, each owning 64
// of a tile's 128 columns: the backward needs no row reductions, so the split
// is free), warp 8 MMA issue, warp 9 TMA.  Each warpgroup writes its bf16
// P / dS values into its own half of the S / dP columns, so neither can
// overwrite scores the other has not read yet.
// The Q/dO (dK/dV kernel) or K/V (dQ kernel) tiles stream through a two-stage
// ring; the fixed operand tiles are loaded once.  All waits are bounded.
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

constexpr int kBwdThreads = 320;
constexpr int kBwdMmaWarp = 8;
constexpr int kBwdLoadWarp = 9;
constexpr int kGradThreads = 256;
constexpr int kStages = 2;
constexpr uint32_t kSub = 128 * 128;  // [128 rows x 64 bf16] 128B-swizzled sub-tile
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kKStages = 3;  // dQ kernel: K ring
constexpr int kVStages = 2;  // dQ kernel: V ring

template <int D>
struct BwdCfg {
  static constexpr uint32_t kTile = (D / 64) * kSub;  // one 128 x D bf16 tile
  // dK/dV smem: two fixed tiles, kStages x (two streamed tiles), then scalars/barriers
  static constexpr uint32_t kFixed = 2 * kTile;
  static constexpr uint32_t kRing = kStages * 2 * kTile;
  // Per gradient warp: -LSE2 and -Delta of its 64 columns for the current step.
  static constexpr uint32_t kScalars = 8 * 2 * 64 * 4;
  static constexpr uint32_t kBarBytes = 256;
  static constexpr size_t kSmem = 1024 + kFixed + kRing + kScalars + kBarBytes;
  // dQ smem: Q and dO fixed, a K ring and a V ring, barriers.
  static constexpr size_t kSmemDq =
      1024 + kFixed + size_t(kKStages + kVStages) * kTile + kBarBytes;
  static_assert(kSmem <= 232448 && kSmemDq <= 232448, "shared memory per CTA");
  static constexpr uint32_t kColS = 0, kColDP = 128, kColA0 = 256, kColA1 = 256 + D;
  static constexpr uint32_t kIdescSS = idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t kIdescTS = idesc_bf16_f32(128, D, false, true);
};

struct BwdBars {
  uint64_t fixed_full;
  uint64_t full[kKStages], empty[kKStages];     // dK/dV: Q+dO stages; dQ: K stages
  uint64_t full_v[kVStages], empty_v[kVStages];  // dQ: V stages
  uint64_t s_full;    // S (or S^T) of the current step is in TMEM
  uint64_t dp_full;   // dP (or dP^T) of the current step is in TMEM
  uint64_t p_ready;   // dK/dV: P^T written; dQ: S read (its columns are free)
  uint64_t ds_full;   // dS (or dS^T) written
  uint64_t acc_full;  // all accumulating MMAs have completed
  uint64_t mma_done;
  // persistent dQ kernel: Q/dO buffer reusable; dQ accumulator b complete / read out
  uint64_t q_empty, acc_full2[2], acc_free[2];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(BwdBars) <= 256, "barrier block too large");

struct BwdParams {
  const float* lse;    // [B,Hq,Sq] natural log
  const float* delta;  // [B,Hq,Sq]
  float* out0;         // dkdv: dK [B,Hkv,Sk,D]; dq: dQ [B,Hq,Sq,D]
  float* out1;         // dkdv: dV
  int* status;
  int B, Hq, Hkv, Sq, Sk, causal;
  float scale, scale_log2;
};

// Read-only global load issued where it stands in the program.
__device__ __forceinline__ float ld_nc_f32(const float* ptr) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(ptr) : "memory");
  return v;
}

__device__ __forceinline__ void bwd_record(int* status) {
  if (status != nullptr) atomicCAS(status, 0, ATTN_ERR_TIMEOUT);
}

__device__ __forceinline__ bool bwd_wait(uint64_t* bar, uint32_t parity, BwdBars* bars);

// The wait for a whole converged warp (the TMA and MMA roles run as whole warps
// and issue from one elected lane); the vote keeps the outcome uniform.  Used
// once per work item.  Inside a step those warps wait without a vote (a vote
// per wait costs several per cent): each lane keeps its outcome, issue
// continues with in-bounds addresses, and one vote per step makes the stop
// decision uniform; a lane still polling is waited for by the next elect.sync.
__device__ __forceinline__ bool bwd_wait_w(uint64_t* bar, uint32_t parity, BwdBars* bars) {
  return __all_sync(0xffffffffu, bwd_wait(bar, parity, bars));
}

__device__ __forceinline__ bool bwd_wait(uint64_t* bar, uint32_t parity, BwdBars* bars) {
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

// First 128-row query tile that can see key tile n (bottom-right causal).
__device__ __forceinline__ int first_q_tile(const BwdParams& p, int n) {
  if (!p.causal) return 0;
  const int row = 128 * n - (p.Sk - p.Sq);
  return row <= 0 ? 0 : row / 128;
}

// KV tiles a query tile needs (as in the forward).
__device__ __forceinline__ int kv_tiles_for(const BwdParams& p, int m) {
  const int row_first = 128 * m;
  if (row_first >= p.Sq) return 0;
  int nvis = p.Sk;
  if (p.causal) {
    const int row_last = min(row_first + 127, p.Sq - 1);
    nvis = min(p.Sk, row_last + p.Sk - p.Sq + 1);
    if (nvis <= 0) return 0;
  }
  return (nvis + 127) / 128;
}

// ------------------------------------------------------------------ Delta
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16* __restrict__ dout,
                                                        const float* __restrict__ o,
                                                        float* __restrict__ delta, int rows) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  constexpr int DPL = D / 32;
  const __nv_bfloat16* dr = dout + static_cast<size_t>(row) * D + lane * DPL;
  const float* orow = o + static_cast<size_t>(row) * D + lane * DPL;
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < DPL; ++e) acc = fmaf(__bfloat162float(dr[e]), orow[e], acc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) delta[row] = acc;
}

// ------------------------------------------------------------------ shared pieces
template <int D>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                          int row0, int plane) {
#pragma unroll
  for (int s = 0; s < D / 64; ++s) tma_load_3d(dst + s * kSub, map, bar, s * 64, row0, plane);
}

// One 128x128 SS product into TMEM column d_col (called by the whole MMA warp): a b^T (K-major tiles, D deep).
template <int D>
__device__ __forceinline__ void mma_ss_tile(uint32_t tmem, uint32_t d_col, uint32_t a_smem,
                                            uint32_t b_smem) {
  using C = BwdCfg<D>;
  constexpr uint64_t kDesc = sdesc_sw128(0, 16, 1024);
  constexpr uint32_t kHi = static_cast<uint32_t>(kDesc >> 32);
  constexpr uint32_t kLo = static_cast<uint32_t>(kDesc);
  const uint32_t a = kLo + (a_smem >> 4);
  const uint32_t b = kLo + (b_smem >> 4);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * kSub + (kk & 3) * 32) >> 4;
    const uint64_t ad = desc_from_words(a + off, kHi);
    const uint64_t bd = desc_from_words(b + off, kHi);
    if (kk == 0)
      mma_ss_w<0>(tmem + d_col, ad, bd, C::kIdescSS);
    else
      mma_ss_w<1>(tmem + d_col, ad, bd, C::kIdescSS);
  }
}

// acc (+)= A(tmem, 128 x 128 bf16 at column a_col) x B(smem tile, MN-major)
// (called by the whole MMA warp).
template <int D>
__device__ __forceinline__ void mma_ts_acc(uint32_t tmem, uint32_t acc_col, uint32_t a_col,
                                           uint32_t b_smem, bool first) {
  using C = BwdCfg<D>;
  constexpr uint64_t kDesc = sdesc_sw128(0, kSub, 1024);
  constexpr uint32_t kHi = static_cast<uint32_t>(kDesc >> 32);
  constexpr uint32_t kLo = static_cast<uint32_t>(kDesc);
  const uint32_t b = kLo + (b_smem >> 4);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint64_t bd = desc_from_words(b + kk * (2048 >> 4), kHi);
    // bf16 A: rows 0-63 packed at columns [0,32), rows 64-127 at [64,96).
    const uint32_t ac = a_col + kk * 8 + (kk >= 4 ? 32 : 0);
    if (first && kk == 0)
      mma_ts_w<0>(tmem + acc_col, tmem + ac, bd, C::kIdescTS);
    else
      mma_ts_w<1>(tmem + acc_col, tmem + ac, bd, C::kIdescTS);
  }
}

// Read columns [c_begin, c_end) of this thread's fp32 accumulator row from
// TMEM, scale them and store them to global memory (valid rows only).  Rows
// are D floats apart and lane l holds row l of its warp's 32; lane pairs swap
// half their segments (pair_transpose8) so that each store writes 64
// contiguous bytes of one row.  All 32 lanes must call it.
template <int D>
__device__ __forceinline__ void store_acc_row(uint32_t taddr, float* dst, float mul, bool valid,
                                              int c_begin, int c_end, int lane, const float* base,
                                              size_t bytes, int* status) {
  const int pb = lane & 1;
  const bool partner_valid = __shfl_xor_sync(0xffffffffu, valid, 1);
  const bool even_valid = pb ? partner_valid : valid, odd_valid = pb ? valid : partner_valid;
  float* even_row = dst - pb * D;
  const bool v8 = (reinterpret_cast<uintptr_t>(dst) & 31u) == 0;
#pragma unroll 1
  for (int c = c_begin; c < c_end; c += 32) {
    uint32_t w[32];
    tmem_ld32(taddr + c, w);
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * mul);
    pair_transpose8(w, lane);
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      float* e = even_row + c + 8 * (2 * m + pb);
      float* o = even_row + D + c + 8 * (2 * m + pb);
      if (even_valid && store_in_bounds(e, 32, base, bytes, status)) st_global_8w(e, &w[16 * m], v8);
      if (odd_valid && store_in_bounds(o, 32, base, bytes, status)) st_global_8w(o, &w[16 * m + 8], v8);
    }
  }
}

// ------------------------------------------------------------------ dK / dV
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmDO, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::kTile;
  uint8_t* sRing = smem + C::kFixed;  // stage st: Q at +0, dO at +kTile
  float* sScal = reinterpret_cast<float*>(smem + C::kFixed + C::kRing);  // [st][2][128]
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::kFixed + C::kRing + C::kScalars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Work: key tile n of KV head (b, g); CTAs are numbered n-major so the
  // largest work (low n under a causal mask) is scheduled first.
  const int n = blockIdx.x / (p.B * p.Hkv);
  const int bg = blockIdx.x % (p.B * p.Hkv);
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int group = p.Hq / p.Hkv;
  const int mtiles = (p.Sq + 127) / 128;
  const int m0 = min(first_q_tile(p, n), mtiles);
  const int per_head = mtiles - m0;
  const int nsteps = group * per_head;

  if (threadIdx.x == 0) {
    mbar_init(&bars->fixed_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_ready, kGradThreads / 32);  // one arrival per gradient warp
    mbar_init(&bars->ds_full, kGradThreads / 32);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kBwdMmaWarp) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  bool ok = true;

  if (warp == kBwdLoadWarp) {
    if (nsteps > 0) {
      if (elect_one()) {
        mbar_arrive_expect_tx(&bars->fixed_full, 2 * C::kTile);
        load_tile<D>(sK, &tmK, &bars->fixed_full, 128 * n, bg);
        load_tile<D>(sV, &tmV, &bars->fixed_full, 128 * n, bg);
      }
      __syncwarp();
      for (int s = 0; s < nsteps && ok; ++s) {
        const int st = s % kStages;
        bool good = true;
        if (s >= kStages) good = bwd_wait(&bars->empty[st], ((s / kStages) - 1) & 1, bars);
        const int h = g * group + s / per_head;
        const int m = m0 + s % per_head;
        uint8_t* dst = sRing + st * 2 * C::kTile;
        if (elect_one()) {
          mbar_arrive_expect_tx(&bars->full[st], 2 * C::kTile);
          load_tile<D>(dst, &tmQ, &bars->full[st], 128 * m, b * p.Hq + h);
          load_tile<D>(dst + C::kTile, &tmDO, &bars->full[st], 128 * m, b * p.Hq + h);
        }
        __syncwarp();
        ok = __all_sync(0xffffffffu, good);
      }
      if (!ok) bwd_record(p.status);
      for (int s = max(0, nsteps - kStages); s < nsteps; ++s)
        (void)mbar_wait(&bars->full[s % kStages], (s / kStages) & 1);
      (void)mbar_wait(&bars->fixed_full, 0);
    }
  } else if (warp == kBwdMmaWarp) {
    if (nsteps > 0) {
      ok = bwd_wait_w(&bars->fixed_full, 0, bars);
      const uint32_t k_addr = smem_u32(sK), v_addr = smem_u32(sV);
      // S^T = K Q^T of step s (its Q/dO stage must have landed) and dP^T = V dO^T.
      auto issue_s = [&](int s) -> bool {  // this lane's wait outcome
        const int st = s % kStages;
        const bool got = bwd_wait(&bars->full[st], (s / kStages) & 1, bars);
        mma_ss_tile<D>(tmem, C::kColS, k_addr, smem_u32(sRing + st * 2 * C::kTile));
        tc_commit_w(&bars->s_full);
        return got;
      };
      auto issue_dp = [&](int s) {  // after issue_s(s), which waited for the stage
        const int st = s % kStages;
        mma_ss_tile<D>(tmem, C::kColDP, v_addr, smem_u32(sRing + st * 2 * C::kTile) + C::kTile);
        tc_commit_w(&bars->dp_full);
      };
      if (ok) {
        const bool got = issue_s(0);
        issue_dp(0);
        ok = __all_sync(0xffffffffu, got);
      }
      // One vote after the loop: after a timed-out wait the abort flag makes
      // every later wait give up after a few polls (operands stay in bounds).
      bool good = true;
      for (int s = 0; s < nsteps && ok; ++s) {
        const int st = s % kStages;
        const uint32_t q_addr = smem_u32(sRing + st * 2 * C::kTile);
        const uint32_t do_addr = q_addr + C::kTile;
        // dV += P^T dO as soon as P^T is in TMEM (B operands MN-major: their
        // rows are the K dimension), then at once S^T(s+1): it overwrites P^T(s)
        // only after dV has read it (same-thread tcgen05 order), and the
        // gradient warps need S^T(s) no more; they compute dS^T(s) meanwhile.
        good &= bwd_wait(&bars->p_ready, s & 1, bars);
        tc_fence_after();
        mma_ts_acc<D>(tmem, C::kColA1, C::kColS, do_addr, s == 0);
        if (s + 1 < nsteps) good &= issue_s(s + 1);
        // dK += dS^T Q once dS^T is in TMEM; then the stage is free, and
        // dP^T(s+1) may overwrite dS^T(s).
        good &= bwd_wait(&bars->ds_full, s & 1, bars);
        tc_fence_after();
        mma_ts_acc<D>(tmem, C::kColA0, C::kColDP, q_addr, s == 0);
        tc_commit_w(&bars->empty[st]);
        if (s + 1 < nsteps) issue_dp(s + 1);
      }
      ok = ok && __all_sync(0xffffffffu, good);
      if (ok) tc_commit_w(&bars->acc_full);
      if (!ok) bwd_record(p.status);
      tc_commit_w(&bars->mma_done);
      (void)mbar_wait(&bars->mma_done, 0);
    }
  } else {
    // Gradient warps: thread r owns key 128n + r (TMEM lane r); warpgroup
    // `half` handles columns [64*half, 64*half + 64).
    const int quad = warp & 3;
    const int half = warp >> 2;
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const int key = 128 * n + r;
    const bool key_valid = key < p.Sk;
    // LSE and Delta of a step's 64 columns (2 per lane), loaded one step ahead:
    // the loads stay in flight through the previous step's work (volatile asm
    // keeps them ahead of that work's tcgen05 operations).  Rows past Sq load
    // row Sq - 1 (in bounds) and are zeroed when staged.
    float pre_l[2] = {0.f, 0.f}, pre_d[2] = {0.f, 0.f};
    auto fetch = [&](int s) {
      const int h = g * group + s / per_head;
      const int m = m0 + s % per_head;
      const size_t base = static_cast<size_t>(b * p.Hq + h) * p.Sq;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int row = min(128 * m + 64 * half + 32 * u + lane, p.Sq - 1);
        pre_l[u] = ld_nc_f32(p.lse + base + row);
        pre_d[u] = ld_nc_f32(p.delta + base + row);
      }
    };
    if (nsteps > 0) fetch(0);
    for (int s = 0; s < nsteps && ok; ++s) {
      const int m = m0 + s % per_head;
      // This step's -LSE (log2 domain) and -Delta for the warpgroup's 64
      // columns, in the warp's own buffer (no cross-warp barrier, so an
      // aborting warp cannot strand others); read back as broadcast float4.
      float* nl2 = sScal + warp * 128;
      float* ndl = nl2 + 64;
      __syncwarp();  // every lane is done with the previous step's values
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const bool rv = 128 * m + 64 * half + 32 * u + lane < p.Sq;
        nl2[32 * u + lane] = rv ? -pre_l[u] * kLog2e : 0.f;
        ndl[32 * u + lane] = rv ? -pre_d[u] : 0.f;
      }
      __syncwarp();
      if (s + 1 < nsteps) fetch(s + 1);
      // Visible columns (query rows 128m + col) of this key: [c_lo, c_hi) --
      // row >= key - (Sk - Sq) under the causal mask, row < Sq.
      const int row_lo = p.causal ? key - (p.Sk - p.Sq) : -0x40000000;
      const int c_lo = max(row_lo - 128 * m, 0);
      const int c_hi = key_valid ? min(p.Sq - 128 * m, 128) : 0;
      const bool need_mask = __any_sync(0xffffffffu, c_lo > 64 * half || c_hi < 64 * half + 64);
      ok = __all_sync(0xffffffffu, bwd_wait(&bars->s_full, s & 1, bars));
      if (!ok) break;
      tc_fence_after();
      // P^T for this warpgroup's 64 columns: kept in registers for dS^T and
      // written (bf16) into its own half of the S^T columns.
      const uint64_t sl2 = f2_pack(p.scale_log2, p.scale_log2);
      float pv[64];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * half + cc;
        uint32_t sr[32];
        tmem_ld32(tmem + lane_addr + C::kColS + 32 * c, sr);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 nl = *reinterpret_cast<const float4*>(nl2 + 32 * cc + e);
          float x[4];
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sl2,
                           f2_pack(nl.x, nl.y)),
                    x[0], x[1]);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), sl2,
                           f2_pack(nl.z, nl.w)),
                    x[2], x[3]);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float pu = ex2(x[u]);
            if (need_mask) {
              const int col = 32 * c + e + u;
              pu = (col >= c_lo && col < c_hi) ? pu : 0.f;
            }
            pv[32 * cc + e + u] = pu;
          }
          pk[e >> 1] = pack_bf16x2(pv[32 * cc + e], pv[32 * cc + e + 1]);
          pk[(e >> 1) + 1] = pack_bf16x2(pv[32 * cc + e + 2], pv[32 * cc + e + 3]);
        }
        tmem_st16(tmem + lane_addr + C::kColS + 64 * half + 16 * cc, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&bars->p_ready);
      // dS^T = P^T (dP^T - Delta), into this warpgroup's half of the dP^T columns.
      ok = __all_sync(0xffffffffu, bwd_wait(&bars->dp_full, s & 1, bars));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * half + cc;
        uint32_t dr[32];
        tmem_ld32(tmem + lane_addr + C::kColDP + 32 * c, dr);
        uint32_t dk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 nd = *reinterpret_cast<const float4*>(ndl + 32 * cc + e);
          float d[4];
          f2_unpack(f2_mul(f2_pack(pv[32 * cc + e], pv[32 * cc + e + 1]),
                           f2_add(f2_pack(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])),
                                  f2_pack(nd.x, nd.y))),
                    d[0], d[1]);
          f2_unpack(f2_mul(f2_pack(pv[32 * cc + e + 2], pv[32 * cc + e + 3]),
                           f2_add(f2_pack(__uint_as_float(dr[e + 2]), __uint_as_float(dr[e + 3])),
                                  f2_pack(nd.z, nd.w))),
                    d[2], d[3]);
          dk[e >> 1] = pack_bf16x2(d[0], d[1]);
          dk[(e >> 1) + 1] = pack_bf16x2(d[2], d[3]);
        }
        tmem_st16(tmem + lane_addr + C::kColDP + 64 * half + 16 * cc, dk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&bars->ds_full);
    }
    if (ok) {
      float* dk_row = p.out0 + (static_cast<size_t>(bg) * p.Sk + key) * D;
      float* dv_row = p.out1 + (static_cast<size_t>(bg) * p.Sk + key) * D;
      const size_t kv_bytes = static_cast<size_t>(p.B) * p.Hkv * p.Sk * D * sizeof(float);
      if (nsteps == 0) {
        // No query row sees these keys: their gradients are zero.
        if (key_valid && store_in_bounds(dk_row, D * 4, p.out0, kv_bytes, p.status) &&
            store_in_bounds(dv_row, D * 4, p.out1, kv_bytes, p.status)) {
          for (int c = half * D / 2; c < (half + 1) * D / 2; c += 4) {
            *reinterpret_cast<float4*>(dk_row + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(dv_row + c) = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      } else {
        ok = __all_sync(0xffffffffu, bwd_wait(&bars->acc_full, 0, bars));
        if (ok) {
          tc_fence_after();
          store_acc_row<D>(tmem + lane_addr + C::kColA0, dk_row, p.scale, key_valid,
                           half * D / 2, (half + 1) * D / 2, lane, p.out0, kv_bytes, p.status);
          store_acc_row<D>(tmem + lane_addr + C::kColA1, dv_row, 1.f, key_valid,
                           half * D / 2, (half + 1) * D / 2, lane, p.out1, kv_bytes, p.status);
        }
      }
    }
    if (!ok) bwd_record(p.status);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ dQ
// Persistent: min(#query tiles, #SMs) CTAs, each walking the query tiles
// (highest tile first, i.e. longest under a causal mask) in the order c,
// 2G-1-c, 2G+c, ... (G CTAs), which balances a descending cost list.  Across
// its tiles a CTA keeps one TMEM allocation and its barrier phases; the next
// tile's Q and dO load as soon as the current tile's last S and dP products
// are done, and the dQ accumulator alternates between two TMEM buffers so that
// one tile's epilogue overlaps the next tile's products.
__device__ __forceinline__ int dq_tile_index(int round, int cta, int grid) {
  return round * grid + ((round & 1) ? (grid - 1 - cta) : cta);
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmDO, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sDO = smem + C::kTile;
  uint8_t* sK = smem + C::kFixed;                // K ring: kKStages tiles
  uint8_t* sV = sK + kKStages * C::kTile;        // V ring: kVStages tiles
  BwdBars* bars = reinterpret_cast<BwdBars*>(sV + kVStages * C::kTile);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Work: query tile m of head (b, h), numbered m-major with the highest m first.
  const int BH = p.B * p.Hq;
  const int mtiles = (p.Sq + 127) / 128;
  const int total = BH * mtiles;
  const int group = p.Hq / p.Hkv;

  if (threadIdx.x == 0) {
    mbar_init(&bars->fixed_full, 1);  // this tile's Q and dO have landed
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars->full_v[s], 1);
      mbar_init(&bars->empty_v[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_ready, kGradThreads / 32);  // one arrival per gradient warp
    mbar_init(&bars->ds_full, kGradThreads / 32);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->acc_full2[b], 1);
      mbar_init(&bars->acc_free[b], kGradThreads / 32);
    }
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kBwdMmaWarp) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  bool ok = true;

  if (warp == kBwdLoadWarp) {
    uint32_t G = 0;   // first global step of the current tile
    uint32_t gl = 0;  // steps whose K and V copies were issued
    int kt = 0;       // tiles with work so far (Q/dO loads issued)
    for (int rnd = 0; ok; ++rnd) {
      const int idx = dq_tile_index(rnd, blockIdx.x, gridDim.x);
      if (idx >= total) break;
      const int m = mtiles - 1 - idx / BH, bh = idx % BH;
      const int nsteps = kv_tiles_for(p, m);
      if (nsteps == 0) continue;
      const int bkv = (bh / p.Hq) * p.Hkv + (bh % p.Hq) / group;
      // Q and dO of this tile once the previous tile's last S and dP are done.
      if (kt > 0 && !(ok = __all_sync(0xffffffffu, bwd_wait(&bars->q_empty, (kt - 1) & 1, bars))))
        break;
      if (elect_one()) {
        mbar_arrive_expect_tx(&bars->fixed_full, 2 * C::kTile);
        load_tile<D>(sQ, &tmQ, &bars->fixed_full, 128 * m, bh);
        load_tile<D>(sDO, &tmDO, &bars->fixed_full, 128 * m, bh);
      }
      __syncwarp();
      ++kt;
      // K(s) and V(s) in use order; K(s) is held until dQ(s), V(s) until dP(s).
      for (int s = 0; s < nsteps && ok; ++s) {
        const uint32_t g = G + s;
        const int sk = g % kKStages, sv = g % kVStages;
        bool good = true;
        if (g >= uint32_t(kKStages))
          good = bwd_wait(&bars->empty[sk], ((g / kKStages) - 1) & 1, bars);
        if (elect_one()) {
          mbar_arrive_expect_tx(&bars->full[sk], C::kTile);
          load_tile<D>(sK + sk * C::kTile, &tmK, &bars->full[sk], 128 * s, bkv);
        }
        __syncwarp();
        if (g >= uint32_t(kVStages))
          good &= bwd_wait(&bars->empty_v[sv], ((g / kVStages) - 1) & 1, bars);
        if (elect_one()) {
          mbar_arrive_expect_tx(&bars->full_v[sv], C::kTile);
          load_tile<D>(sV + sv * C::kTile, &tmV, &bars->full_v[sv], 128 * s, bkv);
        }
        __syncwarp();
        gl = g + 1;
        ok = __all_sync(0xffffffffu, good);
      }
      G += nsteps;
    }
    if (!ok) bwd_record(p.status);
    // Every copy this warp issued lands before the CTA can exit (older copies
    // have landed: their slots were released after their use).
    for (uint32_t g = (gl > uint32_t(kKStages) ? gl - kKStages : 0); g < gl; ++g)
      (void)mbar_wait(&bars->full[g % kKStages], (g / kKStages) & 1);
    for (uint32_t g = (gl > uint32_t(kVStages) ? gl - kVStages : 0); g < gl; ++g)
      (void)mbar_wait(&bars->full_v[g % kVStages], (g / kVStages) & 1);
    if (kt > 0) (void)mbar_wait(&bars->fixed_full, (kt - 1) & 1);
  } else if (warp == kBwdMmaWarp) {
    const uint32_t q_addr = smem_u32(sQ), do_addr = smem_u32(sDO);
    const uint32_t k_base = smem_u32(sK), v_base = smem_u32(sV);
    auto issue_s = [&](uint32_t g) -> bool {  // S = Q K^T; this lane's wait outcome
      const int sk = g % kKStages;
      const bool got = bwd_wait(&bars->full[sk], (g / kKStages) & 1, bars);
      mma_ss_tile<D>(tmem, C::kColS, q_addr, k_base + sk * C::kTile);
      tc_commit_w(&bars->s_full);
      return got;
    };
    auto issue_dp = [&](uint32_t g) -> bool {  // dP = dO V^T; V(g) is free afterwards
      const int sv = g % kVStages;
      const bool got = bwd_wait(&bars->full_v[sv], (g / kVStages) & 1, bars);
      mma_ss_tile<D>(tmem, C::kColDP, do_addr, v_base + sv * C::kTile);
      tc_commit_w(&bars->dp_full);
      tc_commit_w(&bars->empty_v[sv]);
      return got;
    };
    uint32_t G = 0;  // first global step of the current tile
    int kt = 0;      // tiles with work so far
    bool good = true;  // one vote per tile, as in the dK/dV kernel's loop
    for (int rnd = 0; ok; ++rnd) {
      const int idx = dq_tile_index(rnd, blockIdx.x, gridDim.x);
      if (idx >= total) break;
      const int nsteps = kv_tiles_for(p, mtiles - 1 - idx / BH);
      if (nsteps == 0) continue;
      const int buf = kt & 1;
      const uint32_t acc_col = buf ? C::kColA1 : C::kColA0;
      good &= bwd_wait(&bars->fixed_full, kt & 1, bars);  // this tile's Q and dO
      // The epilogue of tile kt-2 has read this accumulator buffer.
      if (kt >= 2) good &= bwd_wait(&bars->acc_free[buf], ((kt >> 1) - 1) & 1, bars);
      // S(G) overwrites the S columns once the previous step's S has been read.
      if (G > 0) good &= bwd_wait(&bars->p_ready, (G - 1) & 1, bars);
      tc_fence_after();
      good &= issue_s(G);
      good &= issue_dp(G);
      if (nsteps == 1) tc_commit_w(&bars->q_empty);  // last S and dP of the tile issued
      for (int s = 0; s < nsteps; ++s) {
        const uint32_t g = G + s;
        // S(g+1) as soon as the gradient warps have read S(g) ...
        if (s + 1 < nsteps) {
          good &= bwd_wait(&bars->p_ready, g & 1, bars);
          tc_fence_after();
          good &= issue_s(g + 1);
        }
        // ... dQ += dS K once dS(g) is in TMEM (K MN-major: its rows are the K dim) ...
        good &= bwd_wait(&bars->ds_full, g & 1, bars);
        tc_fence_after();
        mma_ts_acc<D>(tmem, acc_col, C::kColDP, k_base + (g % kKStages) * C::kTile, s == 0);
        tc_commit_w(&bars->empty[g % kKStages]);
        // ... then dP(g+1), which overwrites dS(g) after dQ has read it.  After
        // the tile's last dP, Q and dO may be replaced by the next tile's.
        if (s + 1 < nsteps) {
          good &= issue_dp(g + 1);
          if (s + 2 == nsteps) tc_commit_w(&bars->q_empty);
        }
      }
      tc_commit_w(&bars->acc_full2[buf]);
      G += nsteps;
      ++kt;
      ok = __all_sync(0xffffffffu, good);
    }
    if (!ok) bwd_record(p.status);
    // Every MMA this warp issued completes before TMEM is released.
    tc_commit_w(&bars->mma_done);
    (void)mbar_wait(&bars->mma_done, 0);
  } else {
    // Gradient warps: thread r owns query row 128m + r (TMEM lane r); warpgroup
    // `half` handles keys [64*half, 64*half + 64) of each tile.
    const int quad = warp & 3;
    const int half = warp >> 2;
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const uint64_t sl2 = f2_pack(p.scale_log2, p.scale_log2);
    const size_t q_bytes = static_cast<size_t>(p.B) * p.Hq * p.Sq * D * sizeof(float);
    uint32_t G = 0;  // first global step of the current tile
    int kt = 0;      // tiles with work so far
    for (int rnd = 0; ok; ++rnd) {
      const int idx = dq_tile_index(rnd, blockIdx.x, gridDim.x);
      if (idx >= total) break;
      const int m = mtiles - 1 - idx / BH, bh = idx % BH;
      const int nsteps = kv_tiles_for(p, m);
      const int row = 128 * m + r;
      const bool row_valid = row < p.Sq;
      float* dq_row = p.out0 + (static_cast<size_t>(bh) * p.Sq + row) * D;
      if (nsteps == 0) {
        // No key is visible to these rows: their gradient is zero.
        if (row_valid && store_in_bounds(dq_row, D * 4, p.out0, q_bytes, p.status))
          for (int c = half * D / 2; c < (half + 1) * D / 2; c += 4)
            *reinterpret_cast<float4*>(dq_row + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      const float lse2 = row_valid ? __ldg(p.lse + static_cast<size_t>(bh) * p.Sq + row) * kLog2e
                                   : 0.f;
      const float dlt = row_valid ? __ldg(p.delta + static_cast<size_t>(bh) * p.Sq + row) : 0.f;
      const uint64_t nl2 = f2_pack(-lse2, -lse2);
      const uint64_t ndl = f2_pack(-dlt, -dlt);
      const int key_hi = p.causal ? min(p.Sk - 1, row + p.Sk - p.Sq) : p.Sk - 1;
      for (int s = 0; s < nsteps && ok; ++s) {
        const uint32_t g = G + s;
        ok = __all_sync(0xffffffffu, bwd_wait(&bars->s_full, g & 1, bars));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld32(tmem + lane_addr + C::kColS + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(sr));
        tmem_ld32(tmem + lane_addr + C::kColS + 64 * half + 32,
                  *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
        // S(g) is in registers: its columns may be overwritten by S(g+1).
        tc_fence_before();
        mbar_arrive_warp(&bars->p_ready);
        // Keys 128s + 64*half + e are visible for e < n_vis (causal limit, Sk).
        const int n_vis = row_valid ? min(max(key_hi - (128 * s + 64 * half) + 1, 0), 64) : 0;
        const bool need_mask = __any_sync(0xffffffffu, n_vis < 64);
        float pv[64];
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sl2, nl2),
                    x0, x1);
          float p0 = ex2(x0), p1 = ex2(x1);
          if (need_mask) {
            p0 = e < n_vis ? p0 : 0.f;
            p1 = e + 1 < n_vis ? p1 : 0.f;
          }
          pv[e] = p0;
          pv[e + 1] = p1;
        }
        ok = __all_sync(0xffffffffu, bwd_wait(&bars->dp_full, g & 1, bars));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t dr[32];
          tmem_ld32(tmem + lane_addr + C::kColDP + 64 * half + 32 * cc, dr);
          uint32_t dk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float d0, d1;
            f2_unpack(f2_mul(f2_pack(pv[32 * cc + e], pv[32 * cc + e + 1]),
                             f2_add(f2_pack(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])),
                                    ndl)),
                      d0, d1);
            dk[e >> 1] = pack_bf16x2(d0, d1);
          }
          tmem_st16(tmem + lane_addr + C::kColDP + 64 * half + 16 * cc, dk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&bars->ds_full);
      }
      if (!ok) break;
      // Epilogue: dQ * scale from this tile's accumulator buffer, which the
      // MMA warp may reuse for tile kt+2 once every gradient warp has read it.
      const int buf = kt & 1;
      ok = __all_sync(0xffffffffu, bwd_wait(&bars->acc_full2[buf], (kt >> 1) & 1, bars));
      if (!ok) break;
      tc_fence_after();
      store_acc_row<D>(tmem + lane_addr + (buf ? C::kColA1 : C::kColA0), dq_row, p.scale,
                       row_valid, half * D / 2, (half + 1) * D / 2, lane, p.out0, q_bytes,
                       p.status);
      tc_fence_before();
      mbar_arrive_warp(&bars->acc_free[buf]);
      G += nsteps;
      ++kt;
    }
    if (!ok) bwd_record(p.status);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_bwd_impl(const void* q, const void* k, const void* v, const float* o,
                            const float* lse, const void* dout, float* dq, float* dk, float* dv,
                            float* delta, int B, int Hq, int Hkv, int Sq, int Sk, int causal,
                            float scale, cudaStream_t stream, int* status) {
  using C = BwdCfg<D>;
  const int rows = B * Hq * Sq;
  bwd_delta_kernel<D><<<(rows + 7) / 8, 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(dout), o, delta, rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap tmQ, tmK, tmV, tmDO;
  if (!encode_bf16_map(&tmQ, q, D, Sq, B * Hq, 128) ||
      !encode_bf16_map(&tmK, k, D, Sk, B * Hkv, 128) ||
      !encode_bf16_map(&tmV, v, D, Sk, B * Hkv, 128) ||
      !encode_bf16_map(&tmDO, dout, D, Sq, B * Hq, 128))
    return cudaErrorInvalidValue;
  if ((e = ensure_smem_attr(reinterpret_cast<const void*>(bwd_dkdv_kernel<D>),
                            static_cast<int>(C::kSmem))) != cudaSuccess)
    return e;
  if ((e = ensure_smem_attr(reinterpret_cast<const void*>(bwd_dq_kernel<D>),
                            static_cast<int>(C::kSmemDq))) != cudaSuccess)
    return e;
  BwdParams p;
  p.lse = lse;
  p.delta = delta;
  p.status = status;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.causal = causal;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.out0 = dk;
  p.out1 = dv;
  const int kv_ctas = B * Hkv * ((Sk + 127) / 128);
  bwd_dkdv_kernel<D><<<kv_ctas, kBwdThreads, C::kSmem, stream>>>(tmQ, tmK, tmV, tmDO, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  p.out0 = dq;
  p.out1 = nullptr;
  const int q_tiles = B * Hq * ((Sq + 127) / 128);
  const int q_ctas = q_tiles < sm_count() ? q_tiles : sm_count();
  bwd_dq_kernel<D><<<q_ctas, kBwdThreads, C::kSmemDq, stream>>>(tmQ, tmK, tmV, tmDO, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd(const void* q, const void* k, const void* v, const float* o,
                            const float* lse, const void* dout, float* dq, float* dk, float* dv,
                            float* delta, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                            int causal, float scale, cudaStream_t stream, int* status) {
  if (D == 128)
    return launch_bwd_impl<128>(q, k, v, o, lse, dout, dq, dk, dv, delta, B, Hq, Hkv, Sq, Sk,
                                causal, scale, stream, status);
  return launch_bwd_impl<64>(q, k, v, o, lse, dout, dq, dk, dv, delta, B, Hq, Hkv, Sq, Sk, causal,
                             scale, stream, status);
}

}  // namespace attn
