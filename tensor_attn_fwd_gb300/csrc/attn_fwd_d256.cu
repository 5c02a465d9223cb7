// attn_fwd_d256.cu -- fused attention forward for head dimension 256.
//
// Source: "A Thread-Register Decoupled GPU Execution Model for Efficient Tensor
// Computation", Background (Equ. 1, fused FlashAttention-style attention with
// its softmax phase between the two GEMMs; tensor cores fed from shared and
// tensor memory) and Methodology (GQA/MQA).  Same computation, masks, LSE and
// lazy rescale as the D = 64 / 128 kernel; only the tiling differs.
//
// At D = 256 one 128-row query tile needs 256 TMEM columns for O, so two tiles
// (the D <= 128 kernel's ping-pong) do not fit in 512 columns.  Here a CTA
// owns one query tile at a time and double-buffers S instead:
//   TMEM  S_0 [0,128)  S_1 [128,256)  O [256,512)   (P bf16 over S's first 64)
// The MMA warp issues S(g+1) before O += P(g) V(g), where g counts the CTA's
// (item, KV tile) steps across items, so the tensor core computes the next
// scores while the softmax warps work on the current ones.
//
// K and V tiles (128 keys x 256 dims) are moved as two halves of 128 dims
// each; a half has the shape and shared-memory layout of a D = 128 tile, so
//   S   = Q[:, :128] K_lo^T + Q[:, 128:] K_hi^T
//   O_lo += P V_lo   (O columns 256..383),   O_hi += P V_hi   (384..511)
// use the D = 128 descriptors.  The ring holds five halves (160 KB) next to
// the 64 KB Q tile.
//
// Roles (192 threads): warps 0-3 softmax (thread r owns row / TMEM lane r) and
// epilogue, warp 4 MMA issue, warp 5 TMA (each a whole warp; one elected lane
// issues).
//
// O rescale hazard: S(g) completes before O += P(g-1) V(g-1) has run, so a
// softmax thread that must rescale O at step g first waits for that product.
// pv_done[g % 2] completes when the product of step g has: when S(g) is
// complete, so is the product of step g-2, hence a waiter for step g-1 (or,
// in the epilogue, for step g) is never more than one phase of that barrier
// behind -- with a single barrier it could be two, and a parity wait would
// pass early.  All waits are bounded.
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

constexpr int kD = 256;
constexpr int kThreads256 = 192;
constexpr int kMmaWarp256 = 4;
constexpr int kLoadWarp256 = 5;
constexpr uint32_t kSub = 128 * 128;            // [128 rows x 64 bf16] swizzled sub-tile
constexpr uint32_t kQBytes = 4 * kSub;          // 128 x 256 bf16
constexpr uint32_t kHalfBytes = 2 * kSub;       // 128 x 128 bf16 (half of a K or V tile)
constexpr int kStages256 = 5;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
constexpr float kRescale = 8.0f;
constexpr float kLn2f = 0.69314718055994531f;
constexpr size_t kSmem256 = 1024 + size_t(kQBytes) + size_t(kStages256) * kHalfBytes + 256;
static_assert(kSmem256 <= 232448, "shared memory per CTA");
constexpr uint32_t kIdescQK256 = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV256 = idesc_bf16_f32(128, 128, false, true);
// O (all 256 columns) += P V in one MMA per 16 keys, when V's two halves sit
// in consecutive ring slots: their four 64-column sub-tiles are then evenly
// spaced (the descriptor's 16 KB leading-byte offset) from the first slot.
constexpr uint32_t kIdescPVWide = idesc_bf16_f32(128, 256, false, true);

struct Bars256 {
  uint64_t q_full, q_empty;
  uint64_t kv_full[kStages256], kv_empty[kStages256];
  uint64_t s_full[2], p_full[2][2];
  uint64_t pv_done[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars256) <= 256, "barrier block too large");

struct Params256 {
  void* o;  // fp32, or bf16 when o_bf16
  int o_bf16;
  int o_v8;  // o is 32-byte aligned: 32-byte stores
  size_t o_bytes, lse_bytes;  // output extents (bounds checks of debug builds)
  float* lse;
  int* status;
  int B, Hq, Hkv, Sq, Sk, causal;
  float scale_log2;
  int num_tiles;    // ceil(Sq / 128)
  int total_items;  // B * Hq * num_tiles
  int kv_chunk;     // ORDER 2: KV heads per chunk
};

struct Item256 {
  int bh;
  int row0;  // first query row
  int n;     // KV tiles to visit (0: nothing visible)
};

__device__ __forceinline__ int kv_tiles(const Params256& p, int row_first) {
  if (row_first >= p.Sq) return 0;
  int nvis = p.Sk;
  if (p.causal) {
    const int row_last = min(row_first + 127, p.Sq - 1);
    nvis = min(p.Sk, row_last + p.Sk - p.Sq + 1);
    if (nvis <= 0) return 0;
  }
  return (nvis + 127) / 128;
}

// Longest first (highest query tiles under the causal mask), boustrophedon
// over the persistent CTAs, as in the D <= 128 kernel (see item_at for the
// order without the mask).
__device__ __forceinline__ int item_idx(int round, int cta, int grid) {
  return round * grid + ((round & 1) ? (grid - 1 - cta) : cta);
}

// Within the launch one of three orders, each its own instantiation (so that
// the default order's code is compiled as it was):
//   ORDER 0  highest query tiles first (longest first under the causal mask).
//   ORDER 1  KV head by KV head (its query heads fastest, then its row tiles),
//            so that the items sharing a KV head's K/V run at the same time and
//            read them from L2; without the causal mask (every item then has
//            the same length, so the order costs no balance) when all K/V exceed
//            96 MB.  With one query tile per CTA this kernel streams twice the K/V
//            per tensor cycle of the D <= 128 kernel, and the order gained on
//            every such shape measured (multi-head B8 H16 S2048 +43 %, GQA B4
//            Hq32 Hkv8 S4096 +9 %, B16 Hq32 Hkv8 S1024 +7 %); with K/V that fit
//            in L2 it measured 0.6-2.3 % slower.
//   ORDER 2  chunks of kv_chunk KV heads (48 MB of K/V), each in ORDER 0: under
//            the causal mask when all K/V exceed twice that and Sq <= 4096, so
//            that the heads in flight keep their K/V in L2 while longest first
//            within a chunk keeps the CTAs balanced (multi-head B8 H16 S2048
//            +29 %, B4 H16 S4096 +8 %, GQA B4 Hq32 Hkv8 S4096 +6.5 %).  At
//            S = 8192 the chunks' longest-first lists no longer balance across
//            the CTAs (multi-head D = 128 B4 H32 S8192: -5 to -8 %).
template <int ORDER>
__device__ __forceinline__ Item256 item_at(const Params256& p, int idx) {
  const int BH = p.B * p.Hq;
  Item256 it;
  if (ORDER == 0) {
    it.bh = idx % BH;
    it.row0 = (p.num_tiles - 1 - idx / BH) * 128;
  } else if (ORDER == 2) {
    const int group = p.Hq / p.Hkv;
    const int full = p.kv_chunk * group * p.num_tiles;  // items of a full chunk
    const int c = idx / full, rc = idx % full;
    const int qh_in = min(p.kv_chunk, p.B * p.Hkv - c * p.kv_chunk) * group;
    it.bh = c * p.kv_chunk * group + rc % qh_in;  // KV heads' query heads are contiguous
    it.row0 = (p.num_tiles - 1 - rc / qh_in) * 128;
  } else {
    const int group = p.Hq / p.Hkv;
    const int rest = idx / group;
    const int bg = rest / p.num_tiles;  // b * Hkv + KV head
    it.bh = (bg / p.Hkv) * p.Hq + (bg % p.Hkv) * group + idx % group;
    it.row0 = (rest % p.num_tiles) * 128;
  }
  it.n = kv_tiles(p, it.row0);
  return it;
}

// Next item of this CTA with work, starting at round r (r is advanced past it).
template <int ORDER>
__device__ __forceinline__ bool next_work(const Params256& p, int& r, Item256& it) {
  while (true) {
    const int idx = item_idx(r, blockIdx.x, gridDim.x);
    if (idx >= p.total_items) return false;
    ++r;
    it = item_at<ORDER>(p, idx);
    if (it.n > 0) return true;
  }
}

__device__ __forceinline__ void note_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Bars256* bars) {
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

// The same wait for a whole converged warp (the TMA and MMA roles run as whole
// warps and issue from one elected lane); the vote keeps the outcome uniform.
// Used once per work item.  Inside a KV step those warps wait without a vote
// (a vote per wait costs several per cent): each lane keeps its outcome, issue
// continues with in-bounds addresses, and one vote per step makes the stop
// decision uniform; a lane still polling is waited for by the next elect.sync.
__device__ __forceinline__ bool wait_bar_w(uint64_t* bar, uint32_t parity, Bars256* bars) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, bars));
}

// ------------------------------------------------------------------ producer
// Load order (= the MMA warp's use order):
//   Q(i0) K_0(i0) | K_1 V_0 | K_2 V_1 | ... | K_{n-1} V_{n-2} | Q(i1) K_0(i1) V_{n-1} | ...
// i.e. per step j the next scores' K (or the next item's Q and K_0), then V_j.
struct Ring {
  uint32_t ctr = 0;
};

__device__ __forceinline__ bool load_half(const CUtensorMap* map, int half, int key0, int plane,
                                          uint8_t* sKV, Bars256* bars, Ring& ring) {
  const uint32_t st = ring.ctr % kStages256;
  bool got = true;
  if (ring.ctr >= uint32_t(kStages256))
    got = wait_bar(&bars->kv_empty[st], ((ring.ctr / kStages256) - 1) & 1, bars);
  if (elect_one()) {
    mbar_arrive_expect_tx(&bars->kv_full[st], kHalfBytes);
#pragma unroll
    for (int s = 0; s < 2; ++s)
      tma_load_3d(sKV + st * kHalfBytes + s * kSub, map, &bars->kv_full[st],
                  half * 128 + s * 64, key0, plane);
  }
  __syncwarp();
  ++ring.ctr;
  return got;  // this lane's outcome
}

template <int ORDER>
__device__ void load_role256(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                             const CUtensorMap* tmV, const Params256& p, uint8_t* sQ,
                             uint8_t* sKV, Bars256* bars) {
  const int group = p.Hq / p.Hkv;
  Ring ring;
  uint32_t q_ctr = 0;
  bool ok = true;
  int r = 0;
  Item256 it;
  if (!next_work<ORDER>(p, r, it)) return;
  auto load_q_k0 = [&](const Item256& x) -> bool {
    if (q_ctr > 0 && !wait_bar_w(&bars->q_empty, (q_ctr - 1) & 1, bars)) return false;
    if (elect_one()) {
      mbar_arrive_expect_tx(&bars->q_full, kQBytes);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        tma_load_3d(sQ + s * kSub, tmQ, &bars->q_full, s * 64, x.row0, x.bh);
    }
    __syncwarp();
    ++q_ctr;
    const int bkv = (x.bh / p.Hq) * p.Hkv + (x.bh % p.Hq) / group;
    bool g = load_half(tmK, 0, 0, bkv, sKV, bars, ring);
    g &= load_half(tmK, 1, 0, bkv, sKV, bars, ring);
    return __all_sync(0xffffffffu, g);
  };
  ok = load_q_k0(it);
  while (ok) {
    const int bkv = (it.bh / p.Hq) * p.Hkv + (it.bh % p.Hq) / group;
    Item256 nxt;
    bool have_next = false;
    for (int j = 0; j < it.n && ok; ++j) {
      bool g = true;
      if (j + 1 < it.n) {
        g &= load_half(tmK, 0, (j + 1) * 128, bkv, sKV, bars, ring);
        g &= load_half(tmK, 1, (j + 1) * 128, bkv, sKV, bars, ring);
      } else {
        have_next = next_work<ORDER>(p, r, nxt);
        if (have_next) g &= load_q_k0(nxt);
      }
      g &= load_half(tmV, 0, j * 128, bkv, sKV, bars, ring);
      g &= load_half(tmV, 1, j * 128, bkv, sKV, bars, ring);
      ok = __all_sync(0xffffffffu, g);
    }
    if (!ok || !have_next) break;
    it = nxt;
  }
  if (!ok) note_status(p.status, ATTN_ERR_TIMEOUT);
  // Let every copy this thread issued land before the CTA can exit.
  const uint32_t last = ring.ctr;
  for (uint32_t c = (last > uint32_t(kStages256) ? last - kStages256 : 0); c < last; ++c)
    (void)mbar_wait(&bars->kv_full[c % kStages256], (c / kStages256) & 1);
  if (q_ctr > 0) (void)mbar_wait(&bars->q_full, (q_ctr - 1) & 1);
}

// ------------------------------------------------------------------ MMA issuer
template <int ORDER>
__device__ void mma_role256(const Params256& p, uint8_t* sQ, uint8_t* sKV, Bars256* bars,
                            uint32_t tmem) {
  constexpr uint64_t kDescK = sdesc_sw128(0, 16, 1024);    // Q and K: K-major
  constexpr uint64_t kDescV = sdesc_sw128(0, kSub, 1024);  // V: MN-major
  constexpr uint32_t kHi = static_cast<uint32_t>(kDescK >> 32);
  static_assert(static_cast<uint32_t>(kDescV >> 32) == kHi, "same SBO/swizzle words");
  constexpr uint32_t kLoK = static_cast<uint32_t>(kDescK);
  constexpr uint32_t kLoV = static_cast<uint32_t>(kDescV);
  constexpr uint32_t kHalf16 = kHalfBytes >> 4;
  const uint32_t q_lo = kLoK + (smem_u32(sQ) >> 4);
  const uint32_t k_lo = kLoK + (smem_u32(sKV) >> 4);
  const uint32_t v_lo = kLoV + (smem_u32(sKV) >> 4);
  uint32_t kv_ctr = 0, q_ctr = 0;
  uint32_t g_s = 0, g_pv = 0;  // steps whose S / PV have been issued
  bool ok = true;

  // Per-lane outcomes (no vote); see the note above wait_bar_w.
  auto acquire = [&](uint32_t& st) -> bool {
    st = kv_ctr % kStages256;
    const bool got = wait_bar(&bars->kv_full[st], (kv_ctr / kStages256) & 1, bars);
    ++kv_ctr;
    return got;
  };
  // S(g) = Q K^T into buffer g % 2; releases the two K halves afterwards.
  auto issue_s = [&]() -> bool {
    uint32_t st0, st1;
    bool got = acquire(st0);
    got &= acquire(st1);
    tc_fence_after();
    const uint32_t d = tmem + ((g_s & 1) ? kColS1 : kColS0);
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      const int sub = kk >> 2;  // Q sub-tile 0..3; K half sub >> 1, its sub-tile sub & 1
      const uint32_t qoff = (sub * kSub + (kk & 3) * 32) >> 4;
      const uint32_t koff = (((sub & 1) * kSub + (kk & 3) * 32) >> 4) + ((sub >> 1) ? st1 : st0) * kHalf16;
      const uint64_t a = desc_from_words(q_lo + qoff, kHi);
      const uint64_t b = desc_from_words(k_lo + koff, kHi);
      if (kk == 0)
        mma_ss_w<0>(d, a, b, kIdescQK256);
      else
        mma_ss_w<1>(d, a, b, kIdescQK256);
    }
    tc_commit_w(&bars->s_full[g_s & 1]);
    tc_commit_w(&bars->kv_empty[st0]);
    tc_commit_w(&bars->kv_empty[st1]);
    ++g_s;
    return got;
  };

  int r = 0;
  Item256 it;
  if (!next_work<ORDER>(p, r, it)) return;
  if (!(ok = wait_bar_w(&bars->q_full, q_ctr & 1, bars))) goto done;
  ++q_ctr;
  if (!(ok = __all_sync(0xffffffffu, issue_s()))) goto done;
  if (it.n == 1) tc_commit_w(&bars->q_empty);
  while (true) {
    Item256 nxt;
    bool have_next = false;
    for (int j = 0; j < it.n; ++j) {
      bool good = true;
      // Scores of the next step first: this item's tile j+1, or the next item's tile 0.
      if (j + 1 < it.n) {
        good &= issue_s();
        if (j + 2 == it.n) tc_commit_w(&bars->q_empty);  // the item's last S is issued
      } else {
        have_next = next_work<ORDER>(p, r, nxt);
        if (have_next) {
          if (!(ok = wait_bar_w(&bars->q_full, q_ctr & 1, bars))) goto done;
          ++q_ctr;
          good &= issue_s();
          if (nxt.n == 1) tc_commit_w(&bars->q_empty);
        }
      }
      // O += P(g) V(g), in two key halves as P arrives.
      uint32_t v0, v1;
      good &= acquire(v0);
      good &= acquire(v1);
      const uint32_t buf = g_pv & 1;
      const uint32_t a = tmem + (buf ? kColS1 : kColS0);
      const uint32_t par = (g_pv >> 1) & 1;
      const bool wide = v1 == v0 + 1;  // no wrap between the halves
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        good &= wait_bar(&bars->p_full[buf][half], par, bars);
        tc_fence_after();
        if (wide) {
          const uint32_t b0 = v_lo + v0 * kHalf16;
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = half * 4 + k4;
            const uint64_t bd = desc_from_words(b0 + kk * (2048 >> 4), kHi);
            if (j == 0 && kk == 0)
              mma_ts_w<0>(tmem + kColO, a + kk * 8, bd, kIdescPVWide);
            else
              mma_ts_w<1>(tmem + kColO, a + kk * 8, bd, kIdescPVWide);
          }
        } else {
#pragma unroll
          for (int vh = 0; vh < 2; ++vh) {
            const uint32_t b0 = v_lo + (vh ? v1 : v0) * kHalf16;
            const uint32_t d = tmem + kColO + vh * 128;
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const int kk = half * 4 + k4;
              const uint64_t bd = desc_from_words(b0 + kk * (2048 >> 4), kHi);
              if (j == 0 && kk == 0)
                mma_ts_w<0>(d, a + kk * 8, bd, kIdescPV256);
              else
                mma_ts_w<1>(d, a + kk * 8, bd, kIdescPV256);
            }
          }
        }
      }
      tc_commit_w(&bars->pv_done[g_pv & 1]);
      tc_commit_w(&bars->kv_empty[v0]);
      tc_commit_w(&bars->kv_empty[v1]);
      ++g_pv;
      if (!(ok = __all_sync(0xffffffffu, good))) goto done;
    }
    if (!have_next) break;
    it = nxt;
  }
done:
  if (!ok) note_status(p.status, ATTN_ERR_TIMEOUT);
  // Every MMA this thread issued must finish before TMEM is released.
  tc_commit_w(&bars->mma_done);
  (void)mbar_wait(&bars->mma_done, 0);
}

// ------------------------------------------------------------------ softmax + epilogue
template <int ORDER>
__device__ void softmax_role256(const Params256& p, Bars256* bars, uint32_t tmem, int warp,
                                int lane) {
  const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t tO = tmem + lane_addr + kColO;
  const float sl2 = p.scale_log2;
  uint32_t g = 0;  // steps processed by this CTA (same count as the MMA warp's)
  bool ok = true;

  for (int r = 0; ok; ++r) {
    const int idx = item_idx(r, blockIdx.x, gridDim.x);
    if (idx >= p.total_items) break;
    const Item256 it = item_at<ORDER>(p, idx);
    const int row = it.row0 + warp * 32 + lane;
    const bool row_valid = row < p.Sq;
    const size_t o_off = (static_cast<size_t>(it.bh) * p.Sq + row) * kD;
    float* o_row = static_cast<float*>(p.o) + o_off;
    __nv_bfloat16* o_row16 = static_cast<__nv_bfloat16*>(p.o) + o_off;
    float* lse_ptr = p.lse + static_cast<size_t>(it.bh) * p.Sq + row;
    if (it.n == 0) {
      if (row_valid &&
          store_in_bounds(p.o_bf16 ? static_cast<const void*>(o_row16) : o_row,
                          kD * (p.o_bf16 ? 2 : 4), p.o, p.o_bytes, p.status) &&
          store_in_bounds(lse_ptr, 4, p.lse, p.lse_bytes, p.status)) {
        if (p.o_bf16) {
#pragma unroll 4
          for (int c = 0; c < kD; c += 8)
            *reinterpret_cast<uint4*>(o_row16 + c) = make_uint4(0u, 0u, 0u, 0u);
        } else {
#pragma unroll 4
          for (int c = 0; c < kD; c += 4)
            *reinterpret_cast<float4*>(o_row + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        *lse_ptr = -INFINITY;
      }
      continue;
    }
    const int limit = p.causal ? min(row + p.Sk - p.Sq, p.Sk - 1) : p.Sk - 1;
    float m = -INFINITY;
    float l = 0.f;

    for (int j = 0; j < it.n; ++j, ++g) {
      const uint32_t buf = g & 1;
      const uint32_t tS = tmem + lane_addr + (buf ? kColS1 : kColS0);
      ok = __all_sync(0xffffffffu, wait_bar(&bars->s_full[buf], (g >> 1) & 1, bars));
      if (!ok) break;
      tc_fence_after();
      uint32_t sa[64], sb[64];
      tmem_ld64(tS, sa);
      tmem_ld64_nowait(tS + 64, sb);
      const int key0 = j * 128;
      const bool need_mask = __any_sync(0xffffffffu, key0 + 127 > limit);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (key0 + c > limit) sa[c] = __float_as_uint(-INFINITY);
      }
      float ch[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 64; c += 8)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          ch[e] = max3(ch[e], __uint_as_float(sa[c + e]), __uint_as_float(sa[c + 4 + e]));
      tmem_ld_wait64(sb);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (key0 + 64 + c > limit) sb[c] = __float_as_uint(-INFINITY);
      }
#pragma unroll
      for (int c = 0; c < 64; c += 8)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          ch[e] = max3(ch[e], __uint_as_float(sb[c + e]), __uint_as_float(sb[c + 4 + e]));
      const float m_tile = max3(ch[0], ch[1], fmaxf(ch[2], ch[3])) * sl2;

      bool rescale = false;
      float alpha = 1.f;
      if (j == 0) {
        m = m_tile;
      } else if (m_tile - m > kRescale) {  // false when both are -inf
        alpha = ex2(m - m_tile);
        m = m_tile;
        l *= alpha;
        rescale = true;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O must hold P(g-1) V(g-1) before it is scaled.
        const uint32_t gp = g - 1;
        ok = __all_sync(0xffffffffu, wait_bar(&bars->pv_done[gp & 1], (gp >> 1) & 1, bars));
        if (!ok) break;
        tc_fence_after();
        const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
        for (int c = 0; c < kD; c += 32) {
          uint32_t orow[32];
          tmem_ld32(tO + c, orow);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float x0, x1;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(orow[e]), __uint_as_float(orow[e + 1])), a2),
                      x0, x1);
            orow[e] = __float_as_uint(x0);
            orow[e + 1] = __float_as_uint(x1);
          }
          tmem_st32(tO + c, orow);
        }
      }
      const float base = (m == -INFINITY) ? 0.f : m;
      const uint64_t sc2 = f2_pack(sl2, sl2);
      const uint64_t nb2 = f2_pack(-base, -base);
      uint64_t acc2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) acc2[e] = f2_pack(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t* src = c < 2 ? &sa[32 * c] : &sb[32 * (c - 2)];
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(src[2 * e]), __uint_as_float(src[2 * e + 1])),
                           sc2, nb2),
                    x0, x1);
          const float p0 = ex2(x0);
          const float p1 = ex2(x1);
          acc2[e & 3] = f2_add(acc2[e & 3], f2_pack(p0, p1));
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tS + 16 * c, pk);
        if (c & 1) {
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars->p_full[buf][c >> 1]);
        }
      }
      float rsum = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float a, b;
        f2_unpack(acc2[e], a, b);
        rsum += a + b;
      }
      l += rsum;
    }
    if (!ok) break;

    // Epilogue once the item's last product O += P V has completed.
    const uint32_t gl = g - 1;  // the item's last step
    ok = __all_sync(0xffffffffu, wait_bar(&bars->pv_done[gl & 1], (gl >> 1) & 1, bars));
    if (!ok) break;
    tc_fence_after();
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    // Lane pairs swap half their segments so that each store writes 64
    // contiguous bytes of a row (as in the D = 64/128 kernel's epilogue).
    const int pb = lane & 1;
    const bool even_valid = row - pb < p.Sq, odd_valid = row - pb + 1 < p.Sq;
    if (p.o_bf16) {
#pragma unroll 1
      for (int c = 0; c < kD; c += 32) {
        uint32_t w[16];
        {
          uint32_t orow[32];
          tmem_ld32(tO + c, orow);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(orow[2 * i]) * inv_l,
                               __uint_as_float(orow[2 * i + 1]) * inv_l);
        }
        pair_transpose8(w, lane);
        __nv_bfloat16* e16 = o_row16 + (0 - pb) * kD + c + 16 * pb;
        __nv_bfloat16* d16 = o_row16 + (1 - pb) * kD + c + 16 * pb;
        if (even_valid && store_in_bounds(e16, 32, p.o, p.o_bytes, p.status))
          st_global_8w(e16, &w[0], p.o_v8);
        if (odd_valid && store_in_bounds(d16, 32, p.o, p.o_bytes, p.status))
          st_global_8w(d16, &w[8], p.o_v8);
      }
    } else {
#pragma unroll 1
      for (int c = 0; c < kD; c += 32) {
        uint32_t w[32];
        tmem_ld32(tO + c, w);
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * inv_l);
        pair_transpose8(w, lane);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          float* e32 = o_row + (0 - pb) * kD + c + 8 * (2 * m + pb);
          float* d32 = o_row + (1 - pb) * kD + c + 8 * (2 * m + pb);
          if (even_valid && store_in_bounds(e32, 32, p.o, p.o_bytes, p.status))
            st_global_8w(e32, &w[16 * m], p.o_v8);
          if (odd_valid && store_in_bounds(d32, 32, p.o, p.o_bytes, p.status))
            st_global_8w(d32, &w[16 * m + 8], p.o_v8);
        }
      }
    }
    // The TMEM loads of O have completed (tcgen05.wait::ld inside tmem_ld32)
    // before the next item's first product may overwrite O: that product
    // waits for P of the next step, which these threads write after this.
    if (row_valid && store_in_bounds(lse_ptr, 4, p.lse, p.lse_bytes, p.status))
      *lse_ptr = l > 0.f ? (m + log2f(l)) * kLn2f : -INFINITY;
  }
  if (!ok) note_status(p.status, ATTN_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ kernel
template <int ORDER>
__global__ void __launch_bounds__(kThreads256, 1)
    attn_fwd_d256_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const Params256 p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + kQBytes;
  Bars256* bars = reinterpret_cast<Bars256*>(sKV + kStages256 * kHalfBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < kStages256; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->p_full[b][0], 128);
      mbar_init(&bars->p_full[b][1], 128);
    }
    mbar_init(&bars->pv_done[0], 1);
    mbar_init(&bars->pv_done[1], 1);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp256) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == kLoadWarp256 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // Programmatic dependent: global memory is touched only after the previous
  // kernel in the stream has completed (see attn_fwd_kernel).
  grid_dependency_wait();
  grid_launch_dependents();

  if (warp < 4) {
    softmax_role256<ORDER>(p, bars, tmem, warp, lane);
  } else if (warp == kMmaWarp256) {
    mma_role256<ORDER>(p, sQ, sKV, bars, tmem);
  } else if (warp == kLoadWarp256) {
    load_role256<ORDER>(&tmQ, &tmK, &tmV, p, sQ, sKV, bars);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp256) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_attn_fwd_d256(const void* q, const void* k, const void* v, void* o, int o_bf16,
                                 float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int causal,
                                 float scale, cudaStream_t stream, int* status) {
  CUtensorMap tmQ, tmK, tmV;
  if (!encode_bf16_map(&tmQ, q, kD, Sq, B * Hq, 128) ||
      !encode_bf16_map(&tmK, k, kD, Sk, B * Hkv, 128) ||
      !encode_bf16_map(&tmV, v, kD, Sk, B * Hkv, 128))
    return cudaErrorInvalidValue;
  const int order = fwd_item_order(B, Hq, Hkv, Sq, Sk, kD, causal);  // see item_at
  auto kernel = order == 1 ? attn_fwd_d256_kernel<1>
                           : (order == 2 ? attn_fwd_d256_kernel<2> : attn_fwd_d256_kernel<0>);
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kernel),
                                   static_cast<int>(kSmem256));
  if (e != cudaSuccess) return e;
  Params256 p;
  p.o = o;
  p.o_bf16 = o_bf16;
  p.o_v8 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
  p.o_bytes = static_cast<size_t>(B) * Hq * Sq * kD * (o_bf16 ? 2 : 4);
  p.lse_bytes = static_cast<size_t>(B) * Hq * Sq * sizeof(float);
  p.lse = lse;
  p.status = status;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.causal = causal;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.num_tiles = (Sq + 127) / 128;
  p.total_items = B * Hq * p.num_tiles;
  p.kv_chunk = fwd_kv_chunk(Sk, kD);
  const int grid = p.total_items < sm_count() ? p.total_items : sm_count();
  return launch_programmatic(kernel, dim3(grid), dim3(kThreads256), kSmem256,
                             stream, tmQ, tmK, tmV, p);
}

}  // namespace attn
