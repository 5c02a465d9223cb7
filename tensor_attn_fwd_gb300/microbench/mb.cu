// Microbenchmarks of the sm_103a mechanisms the attention kernels are built
// around.  Each prints one JSON object per line:
//   mma_cycles      cycles per tcgen05.mma (kind::f16, bf16 -> fp32) issued back
//                   to back by one converged warp (elect.sync), one CTA per SM
//   wait_latency    cycles of a dependent mbarrier.try_wait on a completed phase
//   step_sequence   cycles per KV step of the prefill MMA warp's issue sequence
//                   (32 MMAs, 5 waits, 4 commits) with every barrier complete,
//                   and the same with each wait repeated four times
//   ex2_rate        ex2.approx.f32 results per clock per SM (MUFU)
//   tmem_bw         bytes per clock per SM that tcgen05.ld / tcgen05.st move
//                   between TMEM and registers (32x32b shapes, as the softmax
//                   and epilogue use them), with 4 and 8 warps per CTA
//   tma_ring_bw     a TMA producer feeding a ring of 32 KB stages (two 128 x 64
//                   bf16 boxes, 128B swizzle, the prefill K/V tile) and a
//                   consumer that only releases them: GB/s over all SMs, from
//                   HBM (1 GiB streamed) and from L2 (a 38 MiB set re-read)
// Every wait is bounded; every TMEM and shared-memory address is in bounds.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <vector>

#include "../csrc/ptx.cuh"

using namespace attn::ptx;

namespace {

constexpr int kGrid = 152;
constexpr int kSmem = 200 * 1024;  // one CTA per SM

struct Bars {
  uint64_t done, sink[8], fin;
  int abort;
};

__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait(bar, parity);
}

// Shared prologue: zeroed operand tiles, 512 TMEM columns, barriers.
__device__ uint8_t* setup(uint8_t* smem_raw, Bars* bars, uint32_t* tbase) {
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  for (int i = threadIdx.x; i < (196608) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x < 32) {
    tmem_alloc(tbase, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&bars->done, 1);
    for (int i = 0; i < 8; ++i) mbar_init(&bars->sink[i], 1);
    mbar_init(&bars->fin, 1);
    bars->abort = 0;
    fence_mbar_init();
    mbar_arrive(&bars->done);  // phase 0 complete: every wait on it succeeds
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return sm;
}

__device__ void teardown(Bars* bars, uint32_t tbase, int* status) {
  if (threadIdx.x < 32) {
    tc_commit_w(&bars->fin);  // every MMA of warp 0 done before TMEM goes
    if (!bounded_wait(&bars->fin, 0)) atomicExch(status, 1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(tbase, 512);
}

// MODE 0: SS M128 N128 K16; 1: SS M128 N256; 2: TS M128 N128 (A from TMEM);
// 3: SS M64 N256 (A: 64 rows of the same tile); 4: SS M128 N64; 5: TS M128 N64
// (the D = 64 forward's PV shape).
template <int MODE>
__global__ void __launch_bounds__(128, 1) mma_cycles(long long* out, int iters, int* status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  __shared__ uint32_t tbase;
  uint8_t* sm = setup(smem_raw, &bars, &tbase);
  if (threadIdx.x < 32) {
    constexpr int N = (MODE == 1 || MODE == 3) ? 256 : MODE >= 4 ? 64 : 128;
    constexpr int M = MODE == 3 ? 64 : 128;
    constexpr uint32_t idesc = idesc_bf16_f32(M, N, false, false);
    const uint64_t a0 = sdesc_sw128(smem_u32(sm), 16, 1024);
    const uint64_t b0 = sdesc_sw128(smem_u32(sm + 16384), 16, 1024);
    const long long t0 = clock64();
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t a = a0 + ((kk * 32) >> 4), b = b0 + ((kk * 32) >> 4);
        if (MODE == 2 || MODE == 5)
          mma_ts_w<1>(tbase, tbase + 256 + kk * 8, b, idesc);
        else
          mma_ss_w<1>(tbase, a, b, idesc);
      }
    }
    tc_commit_w(&bars.sink[0]);
    if (!bounded_wait(&bars.sink[0], 0)) atomicExch(status, 1);
    const long long t1 = clock64();
    if (threadIdx.x == 0) out[blockIdx.x] = t1 - t0;
  }
  teardown(&bars, tbase, status);
}

__global__ void wait_latency(long long* out, int n) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive(&bar);
  }
  __syncthreads();
  const uint32_t a = smem_u32(&bar);
  uint32_t acc = 0;
  const long long t0 = clock64();
#pragma unroll 1
  for (int i = 0; i < n; ++i) {
    if (!mbar_try_wait(a, 0)) acc += 7;  // a branch on the result, as in a wait loop
    ++acc;
  }
  const long long t1 = clock64();
  if (threadIdx.x == 0) {
    out[0] = t1 - t0;
    out[1] = acc;
  }
}

// The prefill MMA warp's KV step: per tile, wait for each half of P and issue
// its 4 PV MMAs, then the 8 MMAs of the next S and a commit; a K/V acquire per
// step and two release commits.  WREP repeats every wait.
template <int WREP>
__global__ void __launch_bounds__(128, 1) step_sequence(long long* out, int steps, int* status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  __shared__ uint32_t tbase;
  uint8_t* sm = setup(smem_raw, &bars, &tbase);
  if (threadIdx.x < 32) {
    constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);
    constexpr uint64_t kDescK = sdesc_sw128(0, 16, 1024);
    constexpr uint64_t kDescV = sdesc_sw128(0, 16384, 1024);
    constexpr uint32_t kHi = static_cast<uint32_t>(kDescK >> 32);
    const uint32_t q_lo = static_cast<uint32_t>(kDescK) + (smem_u32(sm) >> 4);
    const uint32_t k_lo = static_cast<uint32_t>(kDescK) + (smem_u32(sm + 65536) >> 4);
    const uint32_t v_lo = static_cast<uint32_t>(kDescV) + (smem_u32(sm + 98304) >> 4);
    constexpr uint32_t kTile16 = 32768 >> 4;
    bool good = true;
    auto W = [&]() {
#pragma unroll 1
      for (int i = 0; i < WREP; ++i) good &= mbar_try_wait(smem_u32(&bars.done), 0);
      tc_fence_after();
    };
    auto S = [&](int t) {
      const uint32_t d = tbase + (t ? 128 : 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
        const uint64_t a = desc_from_words(q_lo + t * kTile16 + off, kHi);
        const uint64_t b = desc_from_words(k_lo + off, kHi);
        mma_ss_w<1>(d, a, b, kIdescQK);
      }
    };
    auto PV = [&](int t, int half) {
      const uint32_t d = tbase + (t ? 384 : 256), a = tbase + (t ? 128 : 0);
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const int kk = half * 4 + k4;
        mma_ts_w<1>(d, a + kk * 8, desc_from_words(v_lo + kk * (2048 >> 4), kHi), kIdescPV);
      }
    };
    const long long t0 = clock64();
#pragma unroll 1
    for (int j = 0; j < steps; ++j) {
      W();  // K/V acquire
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        W();
        PV(t, 0);
        W();
        PV(t, 1);
        S(t);
        tc_commit_w(&bars.sink[t]);
      }
      tc_commit_w(&bars.sink[2 + (j & 1)]);
      tc_commit_w(&bars.sink[4 + (j & 1)]);
    }
    tc_commit_w(&bars.sink[7]);
    const long long t1 = clock64();  // the issue loop's time, as the MMA warp sees it
    if (!__all_sync(0xffffffffu, good)) atomicExch(status, 1);
    if (threadIdx.x == 0) out[blockIdx.x] = t1 - t0;
  }
  teardown(&bars, tbase, status);
}

__global__ void __launch_bounds__(1024, 1) ex2_rate(long long* out, float* sink, int iters) {
  float x[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = -0.001f * static_cast<float>(threadIdx.x + i);
  __syncthreads();
  const long long t0 = clock64();
#pragma unroll 1
  for (int it = 0; it < iters; ++it)
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = ex2(x[i]) - 1.0f;
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += x[i];
  if (s == 12345.f) sink[threadIdx.x] = s;  // keeps the loop
  if (threadIdx.x == 0) out[blockIdx.x] = t1 - t0;
}

// TMEM bandwidth.  Warp w reads (or writes) the columns [c0, c0 + 256) of its
// lane quarter (w % 4) in 64-column loads (two 32x32b.x32 under one wait) or
// 32-column stores; with 8 warps, warps w and w + 4 take the two column
// halves.  clock64 around the loop of the slowest warp.
template <bool STORE>
__global__ void __launch_bounds__(256, 1) tmem_bw(long long* out, int sweeps, int* status) {
  __shared__ uint32_t tbase;
  __shared__ __align__(8) uint64_t fin;
  if (threadIdx.x < 32) {
    tmem_alloc(&tbase, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&fin, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const uint32_t cols = nwarps > 4 ? 256u : 512u;
  const uint32_t c0 = (nwarps > 4 && warp >= 4) ? 256u : 0u;
  const uint32_t base = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16) + c0;
  uint32_t acc = 0;
  uint32_t r[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) r[i] = threadIdx.x * 64 + i;
  __syncthreads();
  const long long t0 = clock64();
#pragma unroll 1
  for (int sw = 0; sw < sweeps; ++sw) {
    if (STORE) {
#pragma unroll 1
      for (uint32_t c = 0; c < cols; c += 64) {
        tmem_st32(base + c, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_st32(base + c + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
      }
      tmem_st_wait();
    } else {
#pragma unroll 1
      for (uint32_t c = 0; c < cols; c += 64) {
        tmem_ld64(base + c, r);
#pragma unroll
        for (int i = 0; i < 64; i += 8) acc ^= r[i];
      }
    }
  }
  const long long t1 = clock64();
  __syncthreads();
  if (acc == 0x9e3779b9u) out[255] = acc;  // keeps the loads
  if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned long long*>(&out[blockIdx.x]),
                                         static_cast<unsigned long long>(t1 - t0));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(tbase, 512);
  (void)status;
  (void)fin;
}

// TMA ring.  CTA b streams `tiles` 128-row tiles of plane b (rows wrap around
// `rows`) into kRing stages; warp 0 produces, warp 1 waits for each stage and
// releases it.  Each stage is two [128 x 64] bf16 boxes (32 KB).
constexpr int kRing = 6;
constexpr uint32_t kStageBytes = 32768;

__global__ void __launch_bounds__(64, 1) tma_ring(const __grid_constant__ CUtensorMap map,
                                                  long long* out, int tiles, int rows,
                                                  int* status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kRing], empty[kRing];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    fence_mbar_init();
    prefetch_tmap(&map);
  }
  __syncthreads();
  const int tiles_per_plane = rows / 128;
  bool ok = true;
  const long long t0 = clock64();
  if (threadIdx.x < 32) {
    for (int i = 0; i < tiles && ok; ++i) {
      const int st = i % kRing;
      if (i >= kRing) ok = mbar_wait(&empty[st], ((i / kRing) - 1) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (ok && elect_one()) {
        mbar_arrive_expect_tx(&full[st], kStageBytes);
        const int row = (i % tiles_per_plane) * 128;
        tma_load_3d(sm + st * kStageBytes, &map, &full[st], 0, row, blockIdx.x);
        tma_load_3d(sm + st * kStageBytes + 16384, &map, &full[st], 64, row, blockIdx.x);
      }
      __syncwarp();
    }
    // every issued copy lands before the CTA can exit
    for (int i = (tiles > kRing ? tiles - kRing : 0); i < tiles; ++i)
      if (!mbar_wait(&full[i % kRing], (i / kRing) & 1)) ok = false;
  } else {
    for (int i = 0; i < tiles && ok; ++i) {
      const int st = i % kRing;
      ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (i / kRing) & 1));
      if (ok && elect_one()) mbar_arrive(&empty[st]);
      __syncwarp();
    }
  }
  const long long t1 = clock64();
  if (!ok) atomicExch(status, 1);
  if (threadIdx.x == 32) out[blockIdx.x] = t1 - t0;
}

bool encode_ring_map(CUtensorMap* map, void* base, int rows, int planes) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return false;
  const cuuint64_t dims[3] = {128, cuuint64_t(rows), cuuint64_t(planes)};
  const cuuint64_t strides[2] = {256, 256 * cuuint64_t(rows)};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn)(
             map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

double median(std::vector<long long> v) {
  std::sort(v.begin(), v.end());
  return static_cast<double>(v[v.size() / 2]);
}

template <typename K>
bool launch_cta_per_sm(K kernel, long long* d_out, int arg, int* d_st, std::vector<long long>& h) {
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  for (int rep = 0; rep < 2; ++rep) kernel<<<kGrid, 128, kSmem>>>(d_out, arg, d_st);
  if (cudaDeviceSynchronize() != cudaSuccess) return false;
  h.assign(kGrid, 0);
  cudaMemcpy(h.data(), d_out, kGrid * sizeof(long long), cudaMemcpyDeviceToHost);
  int st = 0;
  cudaMemcpy(&st, d_st, sizeof(int), cudaMemcpyDeviceToHost);
  return st == 0;
}

}  // namespace

int main() {
  long long* d_out;
  int* d_st;
  float* d_sink;
  cudaMalloc(&d_out, 256 * sizeof(long long));
  cudaMalloc(&d_st, sizeof(int));
  cudaMalloc(&d_sink, 1024 * sizeof(float));
  cudaMemset(d_st, 0, sizeof(int));
  std::vector<long long> h;
  bool ok = true;

  const int iters = 2000;
  const char* names[6] = {"SS M128 N128 K16", "SS M128 N256 K16", "TS M128 N128 K16",
                          "SS M64 N256 K16",  "SS M128 N64 K16",  "TS M128 N64 K16"};
  for (int mode = 0; mode < 6 && ok; ++mode) {
    if (mode == 0) ok = launch_cta_per_sm(mma_cycles<0>, d_out, iters, d_st, h);
    if (mode == 1) ok = launch_cta_per_sm(mma_cycles<1>, d_out, iters, d_st, h);
    if (mode == 2) ok = launch_cta_per_sm(mma_cycles<2>, d_out, iters, d_st, h);
    if (mode == 3) ok = launch_cta_per_sm(mma_cycles<3>, d_out, iters, d_st, h);
    if (mode == 4) ok = launch_cta_per_sm(mma_cycles<4>, d_out, iters, d_st, h);
    if (mode == 5) ok = launch_cta_per_sm(mma_cycles<5>, d_out, iters, d_st, h);
    if (ok)
      printf("{\"bench\": \"mma_cycles\", \"shape\": \"%s\", \"cycles_per_mma\": %.1f}\n",
             names[mode], median(h) / (iters * 4.0));
  }

  if (ok) {
    const int n = 10000;
    for (int rep = 0; rep < 2; ++rep) wait_latency<<<1, 32>>>(d_out, n);
    ok = cudaDeviceSynchronize() == cudaSuccess;
    long long w[2] = {0, 0};
    cudaMemcpy(w, d_out, sizeof(w), cudaMemcpyDeviceToHost);
    if (ok)
      printf("{\"bench\": \"wait_latency\", \"cycles_per_try_wait\": %.1f}\n",
             static_cast<double>(w[0]) / n);
  }

  if (ok) {
    const int steps = 400;
    ok = launch_cta_per_sm(step_sequence<1>, d_out, steps, d_st, h);
    const double c1 = ok ? median(h) / steps : 0.0;
    if (ok) ok = launch_cta_per_sm(step_sequence<4>, d_out, steps, d_st, h);
    const double c4 = ok ? median(h) / steps : 0.0;
    if (ok)
      printf("{\"bench\": \"step_sequence\", \"mma_cycles_per_step\": 2048, "
             "\"cycles_per_step\": %.1f, \"cycles_per_step_waits_x4\": %.1f, "
             "\"cycles_per_extra_wait\": %.1f}\n",
             c1, c4, (c4 - c1) / 15.0);
  }

  if (ok) {
    const int it = 4096;
    for (int rep = 0; rep < 2; ++rep) ex2_rate<<<kGrid, 1024>>>(d_out, d_sink, it);
    ok = cudaDeviceSynchronize() == cudaSuccess;
    h.assign(kGrid, 0);
    cudaMemcpy(h.data(), d_out, kGrid * sizeof(long long), cudaMemcpyDeviceToHost);
    if (ok)
      printf("{\"bench\": \"ex2_rate\", \"results_per_clock_per_sm\": %.1f}\n",
             1024.0 * 8.0 * it / median(h));
  }

  // TMEM bandwidth: 4 and 8 warps, loads and stores.
  for (int nw = 4; nw <= 8 && ok; nw += 4) {
    for (int store = 0; store < 2 && ok; ++store) {
      const int sweeps = 2000;
      // kSmem of dynamic shared memory keeps one CTA (and one TMEM allocation) per SM
      cudaFuncSetAttribute(tmem_bw<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
      cudaFuncSetAttribute(tmem_bw<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
      for (int rep = 0; rep < 2 && ok; ++rep) {
        cudaMemset(d_out, 0, 256 * sizeof(long long));
        if (store)
          tmem_bw<true><<<kGrid, nw * 32, kSmem>>>(d_out, sweeps, d_st);
        else
          tmem_bw<false><<<kGrid, nw * 32, kSmem>>>(d_out, sweeps, d_st);
        ok = cudaDeviceSynchronize() == cudaSuccess;
      }
      h.assign(kGrid, 0);
      cudaMemcpy(h.data(), d_out, kGrid * sizeof(long long), cudaMemcpyDeviceToHost);
      // 128 lanes x 512 columns x 4 bytes per sweep
      if (ok)
        printf("{\"bench\": \"tmem_bw\", \"op\": \"%s\", \"warps\": %d, "
               "\"bytes_per_clock_per_sm\": %.1f}\n",
               store ? "st 32x32b.x32" : "ld 32x32b.x32 (x2 per wait)", nw,
               128.0 * 512 * 4 * sweeps / median(h));
    }
  }

  // TMA ring: 1 GiB streamed from HBM once, then a 38 MiB set re-read from L2.
  if (ok) {
    const int rows_hbm = 27520;  // 152 planes x 27520 rows x 256 B = 1.07 GB
    void* buf = nullptr;
    ok = cudaMalloc(&buf, size_t(kGrid) * rows_hbm * 256) == cudaSuccess;
    if (ok) cudaMemset(buf, 0, size_t(kGrid) * rows_hbm * 256);
    const int smem = kRing * kStageBytes + 1024;
    cudaFuncSetAttribute(tma_ring, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    const struct { const char* src; int rows; int tiles; } cases[2] = {
        {"hbm", rows_hbm, rows_hbm / 128}, {"l2", 1024, 8 * 32}};
    for (int c = 0; c < 2 && ok; ++c) {
      CUtensorMap map;
      ok = encode_ring_map(&map, buf, cases[c].rows, kGrid);
      if (!ok) break;
      cudaEvent_t a, b;
      cudaEventCreate(&a);
      cudaEventCreate(&b);
      float best = 1e30f;
      for (int rep = 0; rep < 3 && ok; ++rep) {
        if (c == 0) cudaMemset(buf, rep, size_t(kGrid) * rows_hbm * 256);  // evicts L2
        cudaEventRecord(a);
        tma_ring<<<kGrid, 64, smem>>>(map, d_out, cases[c].tiles, cases[c].rows, d_st);
        cudaEventRecord(b);
        ok = cudaEventSynchronize(b) == cudaSuccess;
        float ms = 0.f;
        cudaEventElapsedTime(&ms, a, b);
        best = std::min(best, ms);
      }
      h.assign(kGrid, 0);
      cudaMemcpy(h.data(), d_out, kGrid * sizeof(long long), cudaMemcpyDeviceToHost);
      int st = 0;
      cudaMemcpy(&st, d_st, sizeof(int), cudaMemcpyDeviceToHost);
      ok = ok && st == 0;
      const double bytes = double(kGrid) * cases[c].tiles * kStageBytes;
      if (ok)
        printf("{\"bench\": \"tma_ring_bw\", \"source\": \"%s\", \"stages\": %d, "
               "\"gb_per_s\": %.1f, \"bytes_per_clock_per_sm\": %.1f}\n",
               cases[c].src, kRing, bytes / (best * 1e-3) / 1e9,
               double(cases[c].tiles) * kStageBytes / median(h));
      cudaEventDestroy(a);
      cudaEventDestroy(b);
    }
    if (buf) cudaFree(buf);
  }

  const cudaError_t e = cudaGetLastError();
  if (!ok || e != cudaSuccess) {
    printf("{\"error\": \"%s\"}\n", ok ? cudaGetErrorString(e) : "a measurement failed");
    return 1;
  }
  return 0;
}
