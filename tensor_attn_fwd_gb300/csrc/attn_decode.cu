// attn_decode.cu -- split-KV decode (one query row per head) and the
// log-sum-exp combine of its partials.
//
// Source: "A Thread-Register Decoupled GPU Execution Model for Efficient Tensor
// Computation", Methodology and Evaluation: decode attention (FlashDecoding) is
// GEMV plus softmax and highly memory bound.  The kernel streams every K and V
// byte exactly once from HBM with TMA and keeps the arithmetic far below the
// memory time.
//
// decode kernel, one CTA per (split, KV head, batch) [x 16-head slice of the
// query group when the group is wider than 16]:
//   * the CTA's query heads (up to 16, the M rows of an m16n8k16 MMA) share
//     every K/V byte it reads (GQA);
//   * each of its 4 warps owns every 4th block of 32 keys of the split, keeps
//     its own online-softmax state and has a private ring of shared-memory
//     slots filled by 128-byte-swizzled TMA copies (K block, V block, ...), so
//     warps never wait on each other while streaming;
//   * S = Q K^T and O += P V run on mma.sync (bf16 in, fp32 accumulate) with
//     ldmatrix / ldmatrix.trans fragments; the online softmax works directly on
//     the accumulator fragments; P is rounded to bf16 for the second MMA;
//   * the warps' states are merged through shared memory at the end.
// Scores are kept in the log2 domain (scaled by scale * log2 e).  The running
// maximum is moved lazily (only when it grows by more than 8) so the O
// fragments are rarely rescaled; O and l always share one reference maximum.
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

constexpr int kRows = 16;    // query heads per CTA: the M rows of the MMA
constexpr int kBlk = 32;     // keys per block
constexpr int kWarps = 4;    // warps per CTA
constexpr int kSlots = 3;    // ring slots per warp
constexpr int kPidBlocks = 32;  // paged: page ids looked up ahead per warp (one per lane)
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLazyRescale = 8.0f;

template <int D>
struct DecCfg {
  static constexpr int kSub = D / 64;                       // 64-dim swizzled sub-tiles
  static constexpr uint32_t kSubBytes = kBlk * 128;         // [32 keys x 64 dims] bf16
  static constexpr uint32_t kSlotBytes = kSub * kSubBytes;  // one K or V block
  static constexpr size_t kRingBytes = size_t(kWarps) * kSlots * kSlotBytes;
  static constexpr size_t kStatBytes = 2 * kWarps * kRows * sizeof(float);
  // Paged caches: the page ids of each warp's first kPidBlocks blocks.
  static constexpr size_t kPidBytes = size_t(kWarps) * kPidBlocks * sizeof(int);
  static constexpr size_t kSmemBytes =
      1024 + kRingBytes + kStatBytes + kWarps * kSlots * sizeof(uint64_t) + kPidBytes;
  // The per-warp partial outputs reuse the ring once streaming is over.
  static_assert(size_t(kWarps) * kRows * D * sizeof(float) <= kRingBytes, "ring reuse");
};

__device__ __forceinline__ void record_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// c += a * b, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared address of 16-byte chunk `cidx` (dims 8*cidx..8*cidx+7) of key row
// `key` in a block stored as 64-dim sub-tiles with the TMA 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(uint32_t base, int key, int cidx) {
  return base + (cidx >> 3) * (kBlk * 128) + key * 128 + ((((cidx & 7) ^ (key & 7))) << 4);
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32, 2)
    decode_splitkv_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __nv_bfloat16* __restrict__ q, float* __restrict__ o_part,
                          float* __restrict__ lse_part, const int* __restrict__ seqlens,
                          const int* __restrict__ block_table, int page_size, int max_pages,
                          int num_pages, int B, int Hq, int Hkv, int Sk, int num_splits,
                          int head_slices, float scale_log2, int* status,
                          float* __restrict__ o_final, float* __restrict__ lse_final,
                          int* __restrict__ counters) {
  using C = DecCfg<D>;
  constexpr int KS = D / 16;  // k-steps of S = Q K^T
  constexpr int NT = D / 8;   // n-tiles of O += P V
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  float* red_m = reinterpret_cast<float*>(smem + C::kRingBytes);  // [warp][row]
  float* red_l = red_m + kWarps * kRows;                           // [warp][row]
  uint64_t* full = reinterpret_cast<uint64_t*>(red_l + kWarps * kRows);  // [warp][slot]
  int* pids = reinterpret_cast<int*>(full + kWarps * kSlots);              // [warp][block]
  float* red_o = reinterpret_cast<float*>(ring);                   // [warp][row][D], after streaming

  // Launched as a programmatic dependent: nothing in global memory (inputs,
  // the sequence lengths, the partials a previous combine may still read) is
  // touched before the previous kernel in the stream has completed.
  grid_dependency_wait();

  const int split = blockIdx.x;
  const int g = blockIdx.y / head_slices;
  const int slice = blockIdx.y % head_slices;
  const int b = blockIdx.z;
  const int G = Hq / Hkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grp = lane >> 2;  // MMA group: rows grp and grp + 8
  const int tq = lane & 3;    // thread in group

  // This sequence's keys: all Sk, or its own length (clamped to [0, Sk]).
  const int len = seqlens != nullptr ? min(max(__ldg(seqlens + b), 0), Sk) : Sk;
  int chunk = (len + num_splits - 1) / num_splits;
  // Paged: whole 32-key blocks per split, so no block straddles two pages.
  if (block_table != nullptr) chunk = (chunk + kBlk - 1) / kBlk * kBlk;
  const long long kb64 = static_cast<long long>(split) * chunk;
  const int key_begin = kb64 < len ? static_cast<int>(kb64) : len;
  const int key_end = min(key_begin + chunk, len);
  const int nkeys = key_end - key_begin;
  const int nblk = (nkeys + kBlk - 1) / kBlk;
  const int my_nblk = warp < nblk ? (nblk - warp + kWarps - 1) / kWarps : 0;
  const int nloads = 2 * my_nblk;
  const int bkv = b * Hkv + g;

  uint64_t* my_full = full + warp * kSlots;
  uint8_t* my_ring = ring + size_t(warp) * kSlots * C::kSlotBytes;
  int* my_pids = pids + warp * kPidBlocks;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kSlots; ++s) mbar_init(&my_full[s], 1);
    fence_mbar_init();
  }
  // Page id of a block (key0 is a multiple of 32 and page_size of 32: the
  // block lies inside one page); a bad table entry is reported and page 0 read.
  auto page_of = [&](int key0) -> int {
    int pid = __ldg(block_table + static_cast<size_t>(b) * max_pages + key0 / page_size);
    if (pid < 0 || pid >= num_pages) {
      record_status(status, ATTN_ERR_INVALID_ARG);
      pid = 0;
    }
    return pid;
  };
  // The warp looks up its first kPidBlocks page ids at once (a lane each), so
  // the issuing lane does not wait on a table load in front of every copy.
  if (block_table != nullptr && lane < my_nblk)
    my_pids[lane] = page_of(key_begin + (warp + lane * kWarps) * kBlk);
  __syncwarp();

  // Load number li of this warp: even = K block, odd = V block of its (li/2)-th block.
  auto issue = [&](int li) {
    const int key0 = key_begin + (warp + (li >> 1) * kWarps) * kBlk;
    const int slot = li % kSlots;
    uint8_t* dst = my_ring + slot * C::kSlotBytes;
    int plane = bkv, row = key0;
    if (block_table != nullptr) {
      const int blk = li >> 1;
      const int pid = blk < kPidBlocks ? my_pids[blk] : page_of(key0);
      plane = pid * Hkv + g;
      row = key0 - (key0 / page_size) * page_size;
    }
    mbar_arrive_expect_tx(&my_full[slot], C::kSlotBytes);
#pragma unroll
    for (int s = 0; s < C::kSub; ++s)
      tma_load_3d(dst + s * C::kSubBytes, (li & 1) ? &tmV : &tmK, &my_full[slot], s * 64, row,
                  plane);
  };
  int issued = 0;
  if (lane == 0) {
    for (; issued < kSlots && issued < nloads; ++issued) issue(issued);
  }

  // Q as the A operand: rows grp (regs 0, 2) and grp + 8 (regs 1, 3).
  uint32_t qa[KS][4];
  {
    const int h0 = slice * kRows + grp, h1 = h0 + 8;
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(
        q + (static_cast<size_t>(b) * Hq + g * G + min(h0, G - 1)) * D);
    const uint32_t* q1 = reinterpret_cast<const uint32_t*>(
        q + (static_cast<size_t>(b) * Hq + g * G + min(h1, G - 1)) * D);
    const bool v0 = h0 < G, v1 = h1 < G;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = v0 ? __ldg(q0 + 8 * ks + tq) : 0u;
      qa[ks][1] = v1 ? __ldg(q1 + 8 * ks + tq) : 0u;
      qa[ks][2] = v0 ? __ldg(q0 + 8 * ks + 4 + tq) : 0u;
      qa[ks][3] = v1 ? __ldg(q1 + 8 * ks + 4 + tq) : 0u;
    }
  }

  float o[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};  // rows grp, grp + 8 (log2 domain)
  float l_run[2] = {0.f, 0.f};              // this lane's part of the row sums

  bool ok = true;
  int consumed = 0;
  for (int i = 0; i < my_nblk && ok; ++i) {
    const int key0 = key_begin + (warp + i * kWarps) * kBlk;
    const int nvalid = min(kBlk, key_end - key0);

    // ---------------- K block: S = Q K^T for 32 keys (4 n-tiles of 8 keys)
    float s[4][4];
    {
      const int li = 2 * i;
      const int slot = li % kSlots;
      ok = __all_sync(0xffffffffu, mbar_wait(&my_full[slot], (li / kSlots) & 1));
      if (!ok) break;
      consumed = li + 1;
      const uint32_t kb = smem_u32(my_ring + slot * C::kSlotBytes);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        const int key = 8 * nt + (lane & 7);
#pragma unroll
        for (int kp = 0; kp < KS / 2; ++kp) {
          uint32_t r[4];
          ldsm_x4(swz(kb, key, 4 * kp + (lane >> 3)), r);
          mma_16816(s[nt], qa[2 * kp], r[0], r[1]);
          mma_16816(s[nt], qa[2 * kp + 1], r[2], r[3]);
        }
      }
      __syncwarp();
      if (lane == 0 && li + kSlots < nloads) {
        fence_proxy_async_smem();
        issue(li + kSlots);
        ++issued;
      }
    }

    // ---------------- online softmax on the S fragments
    uint32_t pa[2][4];  // P as the A operand of the two 16-key steps
    {
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = 8 * nt + 2 * tq + (e & 1);
          const float x = key < nvalid ? s[nt][e] * scale_log2 : -INFINITY;
          s[nt][e] = x;
          mx[e >> 1] = fmaxf(mx[e >> 1], x);
        }
      float alpha[2];
      bool need = false;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        alpha[r] = 1.f;
        if (m_run[r] == -INFINITY || mx[r] > m_run[r] + kLazyRescale) {
          alpha[r] = ex2(m_run[r] - mx[r]);  // 0 on the first block
          m_run[r] = mx[r];
          l_run[r] *= alpha[r];
          need = true;
        }
      }
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          o[nt][0] *= alpha[0];
          o[nt][1] *= alpha[0];
          o[nt][2] *= alpha[1];
          o[nt][3] *= alpha[1];
        }
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float pv = ex2(s[nt][e] - m_run[e >> 1]);
          s[nt][e] = pv;
          l_run[e >> 1] += pv;
        }
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        pa[kk][0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
        pa[kk][1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
        pa[kk][2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        pa[kk][3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      }
    }

    // ---------------- V block: O += P V (two 16-key steps x D/8 n-tiles)
    {
      const int li = 2 * i + 1;
      const int slot = li % kSlots;
      ok = __all_sync(0xffffffffu, mbar_wait(&my_full[slot], (li / kSlots) & 1));
      if (!ok) break;
      consumed = li + 1;
      const uint32_t vb = smem_u32(my_ring + slot * C::kSlotBytes);
      if (nvalid < kBlk) {
        // Rows past the block's last key are real keys of another split, zero
        // fill past Sk, or (with per-sequence lengths) unwritten cache memory
        // that may hold NaN/Inf: zero them so that p = 0 contributes nothing.
        uint8_t* vrow = my_ring + slot * C::kSlotBytes;
        for (int idx = lane; idx < (kBlk - nvalid) * 8 * C::kSub; idx += 32) {
          const int r = nvalid + idx / (8 * C::kSub);
          const int c = idx % (8 * C::kSub);  // 16-byte chunk across the sub-tiles
          *reinterpret_cast<uint4*>(vrow + (c >> 3) * C::kSubBytes + r * 128 + (c & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
      }
      const int mat = lane >> 3;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int key = 16 * kk + (mat & 1) * 8 + (lane & 7);
#pragma unroll
        for (int ndp = 0; ndp < NT / 2; ++ndp) {
          uint32_t r[4];
          ldsm_x4_t(swz(vb, key, 2 * ndp + (mat >> 1)), r);
          mma_16816(o[2 * ndp], pa[kk], r[0], r[1]);
          mma_16816(o[2 * ndp + 1], pa[kk], r[2], r[3]);
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
        (void)mbar_wait(&my_full[li % kSlots], (li / kSlots) & 1);
    }
    __syncwarp();
  }

  // ---------------- merge: the 4 lanes of a row, then the warps of the CTA
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
  }
  __syncthreads();  // every warp is done with the ring: reuse it for red_o
  {
    float* mine = red_o + size_t(warp) * kRows * D;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      *reinterpret_cast<float2*>(mine + grp * D + 8 * nt + 2 * tq) = make_float2(o[nt][0], o[nt][1]);
      *reinterpret_cast<float2*>(mine + (grp + 8) * D + 8 * nt + 2 * tq) =
          make_float2(o[nt][2], o[nt][3]);
    }
    if (tq == 0) {
      red_m[warp * kRows + grp] = m_run[0];
      red_m[warp * kRows + grp + 8] = m_run[1];
      red_l[warp * kRows + grp] = l_run[0];
      red_l[warp * kRows + grp + 8] = l_run[1];
    }
  }
  __syncthreads();

  // 128 threads: row r = tid / 8 (16 rows), D/8 dims each.
  {
    const int r = threadIdx.x >> 3;
    const int part = threadIdx.x & 7;
    const int hl = slice * kRows + r;
    if (hl < G) {
      const int hq = g * G + hl;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * kRows + r]);
      constexpr int DPT = D / 8;
      float out[DPT];
#pragma unroll
      for (int e = 0; e < DPT; ++e) out[e] = 0.f;
      float lse;
      if (M == -INFINITY) {
        lse = -INFINITY;
      } else {
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float wt = ex2(red_m[w * kRows + r] - M);
          L = fmaf(wt, red_l[w * kRows + r], L);
          const float* src = red_o + (size_t(w) * kRows + r) * D + part * DPT;
#pragma unroll
          for (int e = 0; e < DPT; ++e) out[e] = fmaf(wt, src[e], out[e]);
        }
        const float inv = 1.f / L;
#pragma unroll
        for (int e = 0; e < DPT; ++e) out[e] *= inv;
        lse = (M + log2f(L)) * kLn2;
      }
      const size_t row = (static_cast<size_t>(split) * B + b) * Hq + hq;
      const size_t rows = static_cast<size_t>(num_splits) * B * Hq;  // debug bounds checks
      float* dst = o_part + row * D + part * DPT;
      if (store_in_bounds(dst, DPT * 4, o_part, rows * D * sizeof(float), status)) {
#pragma unroll
        for (int e = 0; e < DPT; e += 4)
          *reinterpret_cast<float4*>(dst + e) = make_float4(out[e], out[e + 1], out[e + 2], out[e + 3]);
      }
      if (part == 0 && store_in_bounds(lse_part + row, 4, lse_part, rows * sizeof(float), status))
        lse_part[row] = lse;
    }
  }

  // Fused combine (counters != nullptr): the CTA that completes a (batch, KV
  // head, head slice) group last merges the group's partials and resets the
  // group's counter for the next call.  After the CTA barrier one thread counts
  // the CTA in with an acquire-release atomic at GPU scope: the release
  // publishes every thread's partial stores (ordered before it by the
  // barrier), the acquire in the last CTA makes every other CTA's visible.
  // The merge is combine_kernel's, warp by warp over the rows (lanes over the
  // splits), so both paths give the same bits; it reads through L2 (ld.cg).
  if (counters != nullptr) {
    __shared__ int s_last;
    __syncthreads();
    int* counter = counters + blockIdx.z * gridDim.y + blockIdx.y;
    if (threadIdx.x == 0) {
      int prev;
      asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                   : "=r"(prev) : "l"(counter) : "memory");
      s_last = prev == num_splits - 1;
    }
    __syncthreads();
    if (s_last) {
      // Warp w merges rows w, w + 4, w + 8, w + 12 of the slice together (their
      // loads in flight at once), each in combine_kernel's order.
      constexpr int DPL = D / 32;
      constexpr int RPW = kRows / kWarps;
      constexpr float kLog2e = 1.4426950408889634f;
      const size_t split_rows = static_cast<size_t>(B) * Hq;  // rows per split
      bool valid[RPW];
      size_t row0[RPW];  // split 0's row
      float M[RPW], W[RPW], out[RPW][DPL];
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        const int hl = slice * kRows + warp + kWarps * i;
        valid[i] = hl < G;
        row0[i] = static_cast<size_t>(b) * Hq + g * G + (valid[i] ? hl : 0);
        M[i] = -INFINITY;
        W[i] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) out[i][e] = 0.f;
      }
      for (int s = lane; s < num_splits; s += 32)
#pragma unroll
        for (int i = 0; i < RPW; ++i)
          if (valid[i]) M[i] = fmaxf(M[i], __ldcg(lse_part + s * split_rows + row0[i]));
#pragma unroll
      for (int i = 0; i < RPW; ++i)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
          M[i] = fmaxf(M[i], __shfl_xor_sync(0xffffffffu, M[i], off));
      for (int c0 = 0; c0 < num_splits; c0 += 32) {
        const int s_lane = c0 + lane;
        float w_lane[RPW];
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
          w_lane[i] = valid[i] && M[i] != -INFINITY && s_lane < num_splits
                          ? ex2((__ldcg(lse_part + s_lane * split_rows + row0[i]) - M[i]) * kLog2e)
                          : 0.f;
          W[i] += w_lane[i];
        }
        const int cnt = min(32, num_splits - c0);
#pragma unroll 4
        for (int kk = 0; kk < cnt; ++kk) {
#pragma unroll
          for (int i = 0; i < RPW; ++i) {
            const float w = __shfl_sync(0xffffffffu, w_lane[i], kk);
            if (!valid[i] || M[i] == -INFINITY) continue;
            const float* src = o_part + ((c0 + kk) * split_rows + row0[i]) * D + lane * DPL;
            if constexpr (DPL >= 4) {
#pragma unroll
              for (int e = 0; e < DPL; e += 4) {
                const float4 x = __ldcg(reinterpret_cast<const float4*>(src + e));
                out[i][e] = fmaf(w, x.x, out[i][e]);
                out[i][e + 1] = fmaf(w, x.y, out[i][e + 1]);
                out[i][e + 2] = fmaf(w, x.z, out[i][e + 2]);
                out[i][e + 3] = fmaf(w, x.w, out[i][e + 3]);
              }
            } else {
              const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
              out[i][0] = fmaf(w, x.x, out[i][0]);
              out[i][1] = fmaf(w, x.y, out[i][1]);
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        if (!valid[i]) continue;  // uniform in the warp
        float L = -INFINITY;
        if (M[i] != -INFINITY) {
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) W[i] += __shfl_xor_sync(0xffffffffu, W[i], off);
          const float inv = 1.f / W[i];
#pragma unroll
          for (int e = 0; e < DPL; ++e) out[i][e] *= inv;
          L = M[i] + logf(W[i]);
        }
        float* dst = o_final + row0[i] * D + lane * DPL;
        if (store_in_bounds(dst, DPL * 4, o_final, split_rows * D * sizeof(float), status)) {
          if constexpr (DPL >= 4) {
#pragma unroll
            for (int e = 0; e < DPL; e += 4)
              *reinterpret_cast<float4*>(dst + e) =
                  make_float4(out[i][e], out[i][e + 1], out[i][e + 2], out[i][e + 3]);
          } else {
            *reinterpret_cast<float2*>(dst) = make_float2(out[i][0], out[i][1]);
          }
        }
        if (lane == 0 && store_in_bounds(lse_final + row0[i], 4, lse_final,
                                         split_rows * sizeof(float), status))
          lse_final[row0[i]] = L;
      }
      if (threadIdx.x == 0) *counter = 0;
    }
  }
  // The next kernel in the stream (the combine, when not fused) may now be
  // scheduled; it waits for this grid to finish.
  grid_launch_dependents();
}

// One warp per output row: lse = ln sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s.
// Splits are handled 32 at a time: lane s holds split s's LSE and weight, the
// max and sum are warp reductions, and the O loads of all splits of a chunk are
// independent (lane-parallel over D, unrolled over splits).
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
  // Launched as a dependent of the split kernel: its partials are complete
  // and visible once this returns.
  grid_dependency_wait();
  if (row >= rows) return;
  float M = -INFINITY;
  for (int s = lane; s < num_splits; s += 32)
    M = fmaxf(M, __ldg(lse_part + static_cast<size_t>(s) * rows + row));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float out[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) out[e] = 0.f;
  float L = -INFINITY;
  if (M != -INFINITY) {
    float W = 0.f;
    for (int c0 = 0; c0 < num_splits; c0 += 32) {
      const int s_lane = c0 + lane;
      const float w_lane =
          s_lane < num_splits
              ? ex2((__ldg(lse_part + static_cast<size_t>(s_lane) * rows + row) - M) * kLog2e)
              : 0.f;
      W += w_lane;
      const int cnt = min(32, num_splits - c0);
#pragma unroll 8
      for (int k = 0; k < cnt; ++k) {
        const float w = __shfl_sync(0xffffffffu, w_lane, k);
        const float* src = o_part + (static_cast<size_t>(c0 + k) * rows + row) * D + lane * DPL;
        if constexpr (DPL >= 4) {
#pragma unroll
          for (int e = 0; e < DPL; e += 4) {
            const float4 x = __ldg(reinterpret_cast<const float4*>(src + e));
            out[e] = fmaf(w, x.x, out[e]);
            out[e + 1] = fmaf(w, x.y, out[e + 1]);
            out[e + 2] = fmaf(w, x.z, out[e + 2]);
            out[e + 3] = fmaf(w, x.w, out[e + 3]);
          }
        } else {
          const float2 x = __ldg(reinterpret_cast<const float2*>(src));
          out[0] = fmaf(w, x.x, out[0]);
          out[1] = fmaf(w, x.y, out[1]);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
    const float inv = 1.f / W;
#pragma unroll
    for (int e = 0; e < DPL; ++e) out[e] *= inv;
    L = M + logf(W);
  }
  float* dst = o + static_cast<size_t>(row) * D + lane * DPL;
  if constexpr (DPL >= 4) {
#pragma unroll
    for (int e = 0; e < DPL; e += 4)
      *reinterpret_cast<float4*>(dst + e) = make_float4(out[e], out[e + 1], out[e + 2], out[e + 3]);
  } else {
    *reinterpret_cast<float2*>(dst) = make_float2(out[0], out[1]);
  }
  if (lane == 0) lse[row] = L;
}

template <int D>
cudaError_t launch_decode_impl(const void* q, const void* k, const void* v, const int* seqlens,
                               const PagedKV* paged, float* o_part, float* lse_part, int B,
                               int Hq, int Hkv, int Sk, int num_splits, float scale,
                               cudaStream_t stream, int* status, const FusedCombine* fused) {
  using C = DecCfg<D>;
  const int G = Hq / Hkv;
  const int head_slices = (G + kRows - 1) / kRows;
  // Contiguous: planes are (b, kv head) with Sk rows.  Paged: planes are
  // (page, kv head) with page_size rows.
  const int rows = paged != nullptr ? paged->page_size : Sk;
  const int planes = paged != nullptr ? paged->num_pages * Hkv : B * Hkv;
  CUtensorMap tmK, tmV;
  if (!encode_bf16_map(&tmK, k, D, rows, planes, kBlk) ||
      !encode_bf16_map(&tmV, v, D, rows, planes, kBlk))
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(decode_splitkv_kernel<D>),
                                   static_cast<int>(C::kSmemBytes));
  if (e != cudaSuccess) return e;
  const dim3 grid(num_splits, Hkv * head_slices, B);
  const float scale_log2 = scale * 1.4426950408889634f;
  return launch_programmatic(
      decode_splitkv_kernel<D>, grid, dim3(kWarps * 32), C::kSmemBytes, stream, tmK, tmV,
      static_cast<const __nv_bfloat16*>(q), o_part, lse_part, seqlens,
      paged != nullptr ? paged->block_table : nullptr, paged != nullptr ? paged->page_size : 0,
      paged != nullptr ? paged->max_pages : 0, paged != nullptr ? paged->num_pages : 0, B, Hq, Hkv,
      Sk, num_splits, head_slices, scale_log2, status, fused != nullptr ? fused->o : nullptr,
      fused != nullptr ? fused->lse : nullptr, fused != nullptr ? fused->counters : nullptr);
}

}  // namespace

cudaError_t launch_decode_splitkv(const void* q, const void* k, const void* v, float* o_part,
                                  float* lse_part, int B, int Hq, int Hkv, int Sk, int D,
                                  int num_splits, float scale, cudaStream_t stream, int* status,
                                  const int* seqlens, const PagedKV* paged,
                                  const FusedCombine* fused) {
  if (D == 256)
    return launch_decode_impl<256>(q, k, v, seqlens, paged, o_part, lse_part, B, Hq, Hkv, Sk,
                                   num_splits, scale, stream, status, fused);
  if (D == 128)
    return launch_decode_impl<128>(q, k, v, seqlens, paged, o_part, lse_part, B, Hq, Hkv, Sk,
                                   num_splits, scale, stream, status, fused);
  return launch_decode_impl<64>(q, k, v, seqlens, paged, o_part, lse_part, B, Hq, Hkv, Sk,
                                num_splits, scale, stream, status, fused);
}

cudaError_t launch_combine(const float* o_part, const float* lse_part, float* o, float* lse,
                           int rows, int D, int num_splits, cudaStream_t stream) {
  // Programmatic stream serialisation: the combine grid is scheduled while the
  // preceding split kernel drains and waits for it on the device.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((rows + 7) / 8, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (D == 256)
    e = cudaLaunchKernelEx(&cfg, combine_kernel<256>, o_part, lse_part, o, lse, rows, num_splits);
  else if (D == 128)
    e = cudaLaunchKernelEx(&cfg, combine_kernel<128>, o_part, lse_part, o, lse, rows, num_splits);
  else
    e = cudaLaunchKernelEx(&cfg, combine_kernel<64>, o_part, lse_part, o, lse, rows, num_splits);
  if (e != cudaSuccess) return e;
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
  if (!o || !lse) return ATTN_ERR_INVALID_ARG;
  // The same checks as attn_decode_splitkv (including the sequence-length cap).
  const int chk = decode_check_args(q, k, v, B, Hq, Hkv, Sk, D, num_splits, scale, false);
  if (chk != ATTN_OK) return chk;
  // The partials must fit the static scratch array.
  const long long part_floats = static_cast<long long>(num_splits) * B * Hq * D;
  const long long lse_floats = static_cast<long long>(num_splits) * B * Hq;
  if (part_floats + lse_floats > static_cast<long long>(ATTN_NOALLOC_SCRATCH_FLOATS))
    return ATTN_ERR_UNSUPPORTED;
  if (!aligned16_ptr(o) || !aligned16_ptr(lse)) return ATTN_ERR_MISALIGNED;
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
