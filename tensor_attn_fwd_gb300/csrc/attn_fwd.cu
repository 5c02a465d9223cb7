// attn_fwd.cu -- fused one-pass attention forward on sm_103a tensor cores.
//
// Source: "A Thread-Register Decoupled GPU Execution Model for Efficient Tensor
// Computation": Background (Equ. 1, fused FlashAttention-style attention; the
// softmax phase -- row max, exp, row sum, rescale -- runs on the SIMD/SFU pipes
// between the two GEMMs; warp specialisation with mbarrier producer/consumer
// synchronisation; Blackwell's tensor cores take operands from shared and
// tensor memory instead of registers, Fig. 2) and Methodology (GQA/MQA).
//
// Work item: two 128-row query tiles (256 rows) of one (batch, query head).
// One persistent CTA per SM walks a static longest-first list of items.
//
// Roles (384 threads):
//   warps 0-3  softmax for query tile 0  (thread r owns TMEM lane / row r)
//   warps 4-7  softmax for query tile 1
//   warp  8    MMA issuer (whole warp, one elected lane issues): S_t = Q_t K_j^T
//              and O_t += P_t V_j
//   warp  9    TMA producer (whole warp, one elected lane issues): Q tiles and a
//              K/V stage ring; V_j and K_j+1 complete on one barrier
//   warps 10-11 idle
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   S_0 [0,128)  S_1 [128,256)  O_0 [256,256+D)  O_1 [256+D,256+2D)
//   P_t (bf16, two per column) overwrites the first 64 columns of S_t.
//
// Per KV tile j and query tile t the MMA warp issues S_t(j) (smem x smem),
// waits for the softmax warps to turn S_t(j) into P_t(j), then issues
// O_t += P_t(j) V_j (tmem x smem) followed by S_t(j+1).  While the softmax
// warps of one tile work, the tensor core runs the other tile's GEMMs.
// tcgen05 operations issued by one thread execute in order, so S_t(j+1) never
// overwrites P_t(j) before O_t += P_t(j) V_j has read it.
//
// Online softmax (per row, log2 domain, x = s * scale * log2 e):
//   m' = max(m, max_j x_j); p_j = 2^(x_j - m'); l = l * 2^(m - m') + sum p_j.
// The rescale of O and l is lazy: the running maximum is only moved (and O
// rescaled in TMEM) when the new maximum exceeds it by more than 8, so p stays
// below 2^8; O and l always share the same reference maximum, which keeps the
// result exact up to rounding.
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

constexpr int kThreads = 384;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kRowsPerItem = 256;
constexpr uint32_t kSubBytes = 128 * 128;  // one [128 rows x 64 bf16] swizzled sub-tile
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kLaunchRegs = 168;  // 65536 / 384, rounded down to a multiple of 8
constexpr uint32_t kRegsSoftmax = 200;
constexpr uint32_t kRegsOther = 104;
static_assert(256 * kRegsSoftmax + 128 * kRegsOther == kThreads * kLaunchRegs,
              "register split must use exactly the launch allocation");
constexpr float kLn2 = 0.69314718055994531f;

template <int D>
struct Cfg {
  static constexpr int kSub = D / 64;
  static constexpr uint32_t kTileBytes = kSub * kSubBytes;  // 128 x D bf16
  static constexpr int kStages = (D == 128) ? 5 : 9;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128;
  static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kBarBytes = 256;
  static constexpr size_t kSmemBytes =
      1024 + 2 * size_t(kTileBytes) + size_t(kStages) * kTileBytes + kBarBytes;
  // MMA instruction descriptors.
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
};

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t kv_full[10], kv_empty[10];
  uint64_t s_full[2], p_full[2][2], o_full[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block too large");

struct FwdParams {
  void* o;           // fp32, or bf16 when o_bf16; split s writes at o + s * split_stride_o
  int o_bf16;
  int o_v8;          // o is 32-byte aligned: 32-byte stores
  size_t o_bytes, lse_bytes;  // output extents (bounds checks of debug builds)
  float* lse;        // split s writes at lse + s * split_stride_lse
  int* status;
  int B, Hq, Hkv, Sq, Sk;
  int causal;
  float scale_log2;  // scale * log2(e)
  int num_pairs;     // ceil(Sq / 256)
  int head_pairs;    // 1: an item is rows [0,128) of two query heads of one KV group
  int num_splits;    // KV splits (1: plain forward)
  int split_tiles;   // KV tiles per split
  size_t split_stride_o, split_stride_lse;
  int total_items;   // B * Hq * num_pairs * num_splits (B * Hq / 2 * num_splits in pairs)
};

// A work item is two 128-row query tiles that stream the same K/V: rows
// [256i, 256i+128) and [256i+128, 256i+256) of one query head, or, when
// Sq <= 128 and the KV groups have an even number of heads, rows [0,128) of
// query heads 2k and 2k+1 (the same KV head), so that both tiles have rows.
struct Item {
  int bh;      // b * Hq + h of query tile 0; tile 1's is bh + head_pairs
  int q_row0;  // first query row of tile 0; tile 1's is q_row0 + 128 (0 in head pairs)
  int split;   // KV split
  int j0;      // first KV tile of the split
  int n[2];    // end (exclusive) of query tile 0 / 1's KV tiles in the split;
               // n[t] <= j0: nothing to compute for tile t
};

// Number of leading keys that query tile t of an item needs, in KV tiles.
__device__ __forceinline__ int tile_kv_count(const FwdParams& p, int row_first) {
  if (row_first >= p.Sq) return 0;
  int nvis = p.Sk;
  if (p.causal) {
    const int row_last = min(row_first + 127, p.Sq - 1);
    nvis = min(p.Sk, row_last + p.Sk - p.Sq + 1);
    if (nvis <= 0) return 0;
  }
  return (nvis + 127) / 128;
}

// Items are ordered longest first (highest query rows first under the causal
// mask); CTA c takes indices c, 2G-1-c, 2G+c, ... (boustrophedon), which
// balances the per-CTA totals of a descending cost list.
__device__ __forceinline__ int item_index(int round, int cta, int grid) {
  return round * grid + ((round & 1) ? (grid - 1 - cta) : cta);
}

__device__ __forceinline__ int tile_row0(const FwdParams& p, const Item& it, int t) {
  return it.q_row0 + (p.head_pairs ? 0 : 128 * t);
}
__device__ __forceinline__ int tile_bh(const FwdParams& p, const Item& it, int t) {
  return it.bh + (p.head_pairs ? t : 0);
}

// Split-major order: every item of split 0 (the longest) first, then split 1, ...;
// within a split one of two orders, each its own instantiation of the kernel
// (a runtime branch in this shared lookup cost the default order ~1 % on
// causal launches whose path had not changed):
//   ORDER 0  highest query rows first (longest first under the causal mask).
//   ORDER 1  KV head by KV head: its query heads fastest, then its row pairs, so
//            that the items sharing a KV head's K/V run at the same time and
//            find them in L2.  The host (fwd_item_order) takes it only without
//            the causal mask (every item then has the same length, so the order
//            costs no balance) and when a KV head has at most 32 items; then
//            ORDER 0 spreads them over as many rounds and re-reads K/V from DRAM
//            once all K/V exceed L2 (multi-head B8 H16 S2048: +10 %).  With more
//            (B1 H16 S16384, GQA B2 Hq32 S8192) each round already streams every
//            KV head's K/V in step across several CTAs, and ORDER 1 measured
//            1.5-2.5 % slower.  Under the causal mask, chunking the KV heads so
//            that the heads in flight stay in L2 (the D = 256 kernel's ORDER 2)
//            measured -3 to +3 % here, so causal launches keep ORDER 0.
template <int ORDER>
__device__ __forceinline__ Item get_item(const FwdParams& p, int idx) {
  const int BH = p.B * p.Hq;
  Item it;
  if (p.head_pairs) {
    const int per_split = BH / 2;
    it.split = idx / per_split;
    it.bh = 2 * (idx % per_split);
    it.q_row0 = 0;
  } else if (ORDER == 0) {
    const int per_split = BH * p.num_pairs;
    it.split = idx / per_split;
    const int r = idx % per_split;
    it.bh = r % BH;
    it.q_row0 = (p.num_pairs - 1 - r / BH) * kRowsPerItem;
  } else {
    const int per_split = BH * p.num_pairs;
    it.split = idx / per_split;
    const int r = idx % per_split;
    const int group = p.Hq / p.Hkv;
    const int rest = r / group;
    const int bg = rest / p.num_pairs;  // b * Hkv + KV head
    it.bh = (bg / p.Hkv) * p.Hq + (bg % p.Hkv) * group + r % group;
    it.q_row0 = (rest % p.num_pairs) * kRowsPerItem;
  }
  it.j0 = it.split * p.split_tiles;
  const int j_end = it.j0 + p.split_tiles;
  it.n[0] = min(tile_kv_count(p, it.q_row0), j_end);
  it.n[1] = min(tile_kv_count(p, tile_row0(p, it, 1)), j_end);
  return it;
}

__device__ __forceinline__ void record_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Bars* bars) {
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

// The same wait for a whole converged warp; the vote keeps the lanes together
// and the outcome uniform.  Used where a wait happens once per work item.
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, Bars* bars) {
  return __all_sync(0xffffffffu, wait_or_abort(bar, parity, bars));
}
// Inside a KV step the TMA and MMA warps wait without a vote (a vote after
// every wait costs ~5 % of the step): each lane keeps its own outcome, the warp
// carries on issuing with in-bounds addresses whatever it is, and one vote per
// step (TMA warp) or per work item (MMA warp) makes the decision to stop
// uniform.  A lane that is still polling is waited for by the next
// elect.sync, so the warp reconverges by itself.

// ------------------------------------------------------------------ producer
template <int D, int ORDER>
__device__ void load_role(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                          const FwdParams& p, uint8_t* sQ, uint8_t* sKV, Bars* bars) {
  using C = Cfg<D>;
  const int group = p.Hq / p.Hkv;
  uint32_t kv_ctr = 0, q_ctr = 0;
  bool ok = true;
  // L2 priorities: every query tile is read by one item, every K/V tile by
  // all items of its KV head (Hq/Hkv heads x the head's query tiles), so K/V
  // are kept and Q (and, in the softmax role, O) are let go first.
  const uint64_t pol_q = policy_evict_first();
  const uint64_t pol_kv = policy_evict_last();
  for (int r = 0; ok; ++r) {
    const int idx = item_index(r, blockIdx.x, gridDim.x);
    if (idx >= p.total_items) break;
    const Item it = get_item<ORDER>(p, idx);
    const int n = max(it.n[0], it.n[1]);  // end of the item's KV tiles
    if (n <= it.j0) continue;
    const int b = it.bh / p.Hq, h = it.bh % p.Hq;  // both tiles' KV head
    const int bkv = b * p.Hkv + h / group;
    if (q_ctr > 0 && !(ok = wait_warp(&bars->q_empty, (q_ctr - 1) & 1, bars))) break;
    if (elect_one()) {
      mbar_arrive_expect_tx(&bars->q_full, 2 * C::kTileBytes);
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int s = 0; s < C::kSub; ++s)
          tma_load_3d_hint(sQ + t * C::kTileBytes + s * kSubBytes, tmQ, &bars->q_full, s * 64,
                           tile_row0(p, it, t), tile_bh(p, it, t), pol_q);
    }
    __syncwarp();
    ++q_ctr;
    // Load order: K_0 alone, then (V_j, K_j+1) as one pair per step, V_n-1 alone.
    // A pair's two copies complete on V_j's barrier, so the MMA warp waits once
    // per step for both; K_j+1's own barrier gets a plain arrive, which keeps
    // every stage at one completed phase per use (a stage alternates between K
    // and V as the ring wraps).
    auto take_stage = [&](uint32_t& st) -> bool {
      st = kv_ctr % C::kStages;
      bool g = true;
      if (kv_ctr >= uint32_t(C::kStages))
        g = wait_or_abort(&bars->kv_empty[st], ((kv_ctr / C::kStages) - 1) & 1, bars);
      ++kv_ctr;
      return g;
    };
    {
      uint32_t st;
      const bool g = take_stage(st);
      if (elect_one()) {
        mbar_arrive_expect_tx(&bars->kv_full[st], C::kTileBytes);
#pragma unroll
        for (int s = 0; s < C::kSub; ++s)
          tma_load_3d_hint(sKV + st * C::kTileBytes + s * kSubBytes, tmK, &bars->kv_full[st],
                           s * 64, it.j0 * 128, bkv, pol_kv);
      }
      __syncwarp();
      ok = __all_sync(0xffffffffu, g);
    }
    for (int j = it.j0; j < n && ok; ++j) {
      uint32_t sv, sk = 0;
      const bool pair = j + 1 < n;
      bool good = take_stage(sv);
      if (pair) good &= take_stage(sk);
      if (elect_one()) {
        mbar_arrive_expect_tx(&bars->kv_full[sv], pair ? 2 * C::kTileBytes : C::kTileBytes);
#pragma unroll
        for (int s = 0; s < C::kSub; ++s)
          tma_load_3d_hint(sKV + sv * C::kTileBytes + s * kSubBytes, tmV, &bars->kv_full[sv],
                           s * 64, j * 128, bkv, pol_kv);
        if (pair) {
#pragma unroll
          for (int s = 0; s < C::kSub; ++s)
            tma_load_3d_hint(sKV + sk * C::kTileBytes + s * kSubBytes, tmK, &bars->kv_full[sv],
                             s * 64, (j + 1) * 128, bkv, pol_kv);
          mbar_arrive(&bars->kv_full[sk]);
        }
      }
      __syncwarp();
      ok = __all_sync(0xffffffffu, good);
    }
  }
  if (!ok) record_status(p.status, ATTN_ERR_TIMEOUT);
  // Let every copy this thread issued land before the CTA can exit.  Copies of
  // slots reused since have landed already (their slot was released by the MMA
  // warp after it saw them).  Each item takes an even number of slots (K_0, then
  // V/K pairs, then V_n-1) and kStages is odd, so the last kStages uses start
  // with the first slot of a pair: the barrier that counts a K_j+1 is waited here
  // whenever K_j+1 is.
  static_assert(C::kStages % 2 == 1, "drain window must start on a pair's first slot");
  const uint32_t last = kv_ctr;
  for (uint32_t c = (last > uint32_t(C::kStages) ? last - C::kStages : 0); c < last; ++c)
    (void)mbar_wait(&bars->kv_full[c % C::kStages], (c / C::kStages) & 1);
  if (q_ctr > 0) (void)mbar_wait(&bars->q_full, (q_ctr - 1) & 1);
}

// ------------------------------------------------------------------ MMA issuer
template <int D, int ORDER>
__device__ void mma_role(const FwdParams& p, uint8_t* sQ, uint8_t* sKV, Bars* bars,
                         uint32_t tmem) {
  using C = Cfg<D>;
  // Descriptor words: the high word is fixed per operand kind, the low word is
  // (smem address >> 4) plus the leading-byte-offset field, so each MMA only
  // adds a compile-time offset to a base.
  constexpr uint64_t kDescK = sdesc_sw128(0, 16, 1024);         // Q and K: K-major
  constexpr uint64_t kDescV = sdesc_sw128(0, kSubBytes, 1024);  // V: MN-major
  constexpr uint32_t kHi = static_cast<uint32_t>(kDescK >> 32);
  static_assert(static_cast<uint32_t>(kDescV >> 32) == kHi, "same SBO/swizzle words");
  constexpr uint32_t kLoK = static_cast<uint32_t>(kDescK);
  constexpr uint32_t kLoV = static_cast<uint32_t>(kDescV);
  constexpr uint32_t kTile16 = C::kTileBytes >> 4;
  const uint32_t q_lo = kLoK + (smem_u32(sQ) >> 4);
  const uint32_t k_lo = kLoK + (smem_u32(sKV) >> 4);
  const uint32_t v_lo = kLoV + (smem_u32(sKV) >> 4);
  uint32_t kv_ctr = 0, q_ctr = 0;
  uint32_t p_phase[2] = {0, 0};
  bool ok = true;

  // S_t = Q_t K^T over D in steps of 16 (K-major operands, 128B swizzle).
  auto issue_s = [&](int t, uint32_t kst) {
    const uint32_t a0 = q_lo + t * kTile16;
    const uint32_t b0 = k_lo + kst * kTile16;
    const uint32_t d = tmem + (t ? C::kColS1 : C::kColS0);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = ((kk >> 2) * kSubBytes + (kk & 3) * 32) >> 4;
      const uint64_t a = desc_from_words(a0 + off, kHi);
      const uint64_t b = desc_from_words(b0 + off, kHi);
      if (kk == 0)
        mma_ss_w<0>(d, a, b, C::kIdescQK);
      else
        mma_ss_w<1>(d, a, b, C::kIdescQK);
    }
  };
  // O_t (+)= P_t V for key steps [kk0, kk0+4) (P from TMEM, V MN-major).
  auto issue_pv_half = [&](int t, uint32_t vst, int half, bool first) {
    const uint32_t b0 = v_lo + vst * kTile16;
    const uint32_t d = tmem + (t ? C::kColO1 : C::kColO0);
    const uint32_t a = tmem + (t ? C::kColS1 : C::kColS0);
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      const int kk = half * 4 + k4;
      const uint64_t bd = desc_from_words(b0 + kk * (2048 >> 4), kHi);
      if (first && kk == 0)
        mma_ts_w<0>(d, a + kk * 8, bd, C::kIdescPV);
      else
        mma_ts_w<1>(d, a + kk * 8, bd, C::kIdescPV);
    }
  };
  // Per-lane outcome (no vote); see the note above wait_warp.
  auto acquire_kv = [&](uint32_t& st) -> bool {
    st = kv_ctr % C::kStages;
    const bool got = wait_or_abort(&bars->kv_full[st], (kv_ctr / C::kStages) & 1, bars);
    ++kv_ctr;
    return got;
  };

  for (int r = 0; ok; ++r) {
    const int idx = item_index(r, blockIdx.x, gridDim.x);
    if (idx >= p.total_items) break;
    const Item it = get_item<ORDER>(p, idx);
    const int n = max(it.n[0], it.n[1]);  // end of the item's KV tiles
    if (n <= it.j0) continue;
    if (!(ok = wait_warp(&bars->q_full, q_ctr & 1, bars))) break;
    ++q_ctr;

    // Q may be overwritten once the item's last S MMA has completed.
    int s_left = max(it.n[0] - it.j0, 0) + max(it.n[1] - it.j0, 0);
    auto issue_s_counted = [&](int t, uint32_t st) {
      issue_s(t, st);
      tc_commit_w(&bars->s_full[t]);
      if (--s_left == 0) tc_commit_w(&bars->q_empty);
    };
    uint32_t kst;
    if (!(ok = __all_sync(0xffffffffu, acquire_kv(kst)))) break;
    tc_fence_after();
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (it.n[t] > it.j0) issue_s_counted(t, kst);
    }
    tc_commit_w(&bars->kv_empty[kst]);

    // One vote per item: after a timed-out wait the abort flag makes every
    // later wait of the item give up after a few polls, and the MMAs keep
    // in-bounds operands, so the item runs out quickly and the vote ends it.
    bool good = true;
    for (int j = it.j0; j < n; ++j) {
      // Both operand tiles of this step are acquired before any P wait, so
      // their (usually already satisfied) waits overlap queued MMAs.
      uint32_t vst, nkst = 0;
      const bool has_next = j + 1 < n;
      good &= acquire_kv(vst);
      if (has_next) {  // landed with V_j: counted on V_j's barrier
        nkst = kv_ctr % C::kStages;
        ++kv_ctr;
      }
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (j >= it.n[t]) continue;
        // P arrives in two halves (keys 0-63, 64-127): start on the first
        // while the softmax warps are still producing the second.
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          good &= wait_or_abort(&bars->p_full[t][half], p_phase[t], bars);
          tc_fence_after();
          issue_pv_half(t, vst, half, j == it.j0);
        }
        p_phase[t] ^= 1;
        if (j == it.n[t] - 1)
          tc_commit_w(&bars->o_full[t]);
        else
          issue_s_counted(t, nkst);
      }
      tc_commit_w(&bars->kv_empty[vst]);
      if (has_next) tc_commit_w(&bars->kv_empty[nkst]);
    }
    ok = __all_sync(0xffffffffu, good);
    if (!ok) break;
  }
  if (!ok) record_status(p.status, ATTN_ERR_TIMEOUT);
  // Every MMA this thread issued must finish before TMEM is released.
  tc_commit_w(&bars->mma_done);
  (void)mbar_wait(&bars->mma_done, 0);
}

// ------------------------------------------------------------------ softmax
template <int D, int ORDER>
__device__ void softmax_role(const FwdParams& p, Bars* bars, uint32_t tmem, int warp, int lane) {
  using C = Cfg<D>;
  const int t = warp >> 2;
  const int quad = warp & 3;
  const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t tS = tmem + lane_addr + (t ? C::kColS1 : C::kColS0);
  const uint32_t tO = tmem + lane_addr + (t ? C::kColO1 : C::kColO0);
  const float sl2 = p.scale_log2;
  const uint64_t pol_o = policy_evict_first();  // output rows are written once
  uint32_t s_phase = 0, o_phase = 0;
  bool ok = true;

  for (int r = 0; ok; ++r) {
    const int idx = item_index(r, blockIdx.x, gridDim.x);
    if (idx >= p.total_items) break;
    const Item it = get_item<ORDER>(p, idx);
    // This warpgroup's tile (t is a runtime value: select, do not index, so the
    // item stays in registers).
    const int nt = t ? it.n[1] : it.n[0];  // end of this tile's KV tiles in the split
    const int bh = tile_bh(p, it, t);
    const int row = tile_row0(p, it, t) + quad * 32 + lane;
    const bool row_valid = row < p.Sq;
    const size_t o_off = (static_cast<size_t>(bh) * p.Sq + row) * D +
                         static_cast<size_t>(it.split) * p.split_stride_o;
    float* o_row = static_cast<float*>(p.o) + o_off;
    __nv_bfloat16* o_row16 = static_cast<__nv_bfloat16*>(p.o) + o_off;
    float* lse_ptr = p.lse + static_cast<size_t>(bh) * p.Sq + row +
                     static_cast<size_t>(it.split) * p.split_stride_lse;
    if (nt <= it.j0) {
      // No key of the split visible to any row of this tile (or the tile is
      // past Sq): O = 0, LSE = -inf (a split a combine weighs with 0).
      if (row_valid &&
          store_in_bounds(p.o_bf16 ? static_cast<const void*>(o_row16) : o_row,
                          D * (p.o_bf16 ? 2 : 4), p.o, p.o_bytes, p.status) &&
          store_in_bounds(lse_ptr, 4, p.lse, p.lse_bytes, p.status)) {
        if (p.o_bf16) {
#pragma unroll 4
          for (int c = 0; c < D; c += 8)
            *reinterpret_cast<uint4*>(o_row16 + c) = make_uint4(0u, 0u, 0u, 0u);
        } else {
#pragma unroll 4
          for (int c = 0; c < D; c += 4)
            *reinterpret_cast<float4*>(o_row + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        *lse_ptr = -INFINITY;
      }
      continue;
    }
    // Largest key index this row may see.
    const int limit = p.causal ? min(row + p.Sk - p.Sq, p.Sk - 1) : p.Sk - 1;
    float m = -INFINITY;  // reference maximum (log2 domain)
    float l = 0.f;

    for (int j = it.j0; j < nt; ++j) {
      ok = __all_sync(0xffffffffu, wait_or_abort(&bars->s_full[t], s_phase, bars));
      if (!ok) break;
      s_phase ^= 1;
      tc_fence_after();

      // S row: columns 0..63 are loaded and waited for, 64..127 stay in
      // flight while the first half is masked and reduced.
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
      // Row maximum: 4 independent chains of 3-input max.
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
      if (j == it.j0) {
        m = m_tile;
      } else if (m_tile - m > kRescaleThreshold) {  // false when both are -inf
        alpha = ex2(m - m_tile);
        m = m_tile;
        l *= alpha;
        rescale = true;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O_t(j-1) is complete: S_t(j) was committed after O_t += P_t(j-1) V.
        const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
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
      // p = 2^(s * scale * log2 e - m), two columns per paired FMA/ADD.
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
          // Keys [64*(c/2), 64*(c/2)+64) of P (and any O rescale) are in TMEM.
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive_warp(&bars->p_full[t][c >> 1]);
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

    // Epilogue: O = O / l, LSE = ln 2 * (m + log2 l).
    ok = __all_sync(0xffffffffu, wait_or_abort(&bars->o_full[t], o_phase, bars));
    if (!ok) break;
    o_phase ^= 1;
    tc_fence_after();
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    // Lane pairs swap half their segments (pair_transpose8), so each store
    // writes 64 contiguous bytes of a row: 16 rows per warp store instead of
    // 32, halving the L1 wavefronts that the per-row layout of TMEM costs.
    const int pb = lane & 1;
    const bool even_valid = row - pb < p.Sq, odd_valid = row - pb + 1 < p.Sq;
    if (p.o_bf16) {
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
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
        __nv_bfloat16* e16 = o_row16 + (0 - pb) * D + c + 16 * pb;
        __nv_bfloat16* d16 = o_row16 + (1 - pb) * D + c + 16 * pb;
        if (even_valid && store_in_bounds(e16, 32, p.o, p.o_bytes, p.status))
          st_global_8w_hint(e16, &w[0], p.o_v8, pol_o);
        if (odd_valid && store_in_bounds(d16, 32, p.o, p.o_bytes, p.status))
          st_global_8w_hint(d16, &w[8], p.o_v8, pol_o);
      }
    } else {
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t w[32];
        tmem_ld32(tO + c, w);
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * inv_l);
        pair_transpose8(w, lane);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          float* e32 = o_row + (0 - pb) * D + c + 8 * (2 * m + pb);
          float* d32 = o_row + (1 - pb) * D + c + 8 * (2 * m + pb);
          if (even_valid && store_in_bounds(e32, 32, p.o, p.o_bytes, p.status))
            st_global_8w_hint(e32, &w[16 * m], p.o_v8, pol_o);
          if (odd_valid && store_in_bounds(d32, 32, p.o, p.o_bytes, p.status))
            st_global_8w_hint(d32, &w[16 * m + 8], p.o_v8, pol_o);
        }
      }
    }
    if (row_valid && store_in_bounds(lse_ptr, 4, p.lse, p.lse_bytes, p.status))
      *lse_ptr = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
  }
  if (!ok) record_status(p.status, ATTN_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ kernel
template <int D, int ORDER>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + 2 * C::kTileBytes;
  Bars* bars = reinterpret_cast<Bars*>(sKV + C::kStages * C::kTileBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t][0], 4);  // one arrival per softmax warp of the tile
      mbar_init(&bars->p_full[t][1], 4);
      mbar_init(&bars->o_full[t], 1);
    }
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == kLoadWarp && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // Launched as a programmatic dependent: the set-up above may overlap the end
  // of the previous kernel in the stream; nothing is read or written in
  // global memory before that kernel has completed and its writes are visible.
  grid_dependency_wait();
  grid_launch_dependents();  // the next kernel may start its own set-up

  // Register split: the softmax warpgroups hold a full S row; the MMA/TMA
  // warpgroup needs few.  256*kRegsSoftmax + 128*kRegsOther equals the
  // launch allocation of 384 threads x 168 registers (checked at build time).
  if (warp < 8) {
    setmaxnreg_inc<kRegsSoftmax>();
    softmax_role<D, ORDER>(p, bars, tmem, warp, lane);
  } else {
    setmaxnreg_dec<kRegsOther>();
    if (warp == kMmaWarp) {
      mma_role<D, ORDER>(p, sQ, sKV, bars, tmem);
    } else if (warp == kLoadWarp) {
      load_role<D, ORDER>(&tmQ, &tmK, &tmV, p, sQ, sKV, bars);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
template <int D>
cudaError_t launch_fwd_impl(const void* q, const void* k, const void* v, void* o, int o_bf16,
                            float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int causal,
                            int num_splits, float scale, cudaStream_t stream, int* status) {
  using C = Cfg<D>;
  CUtensorMap tmQ, tmK, tmV;
  if (!encode_bf16_map(&tmQ, q, D, Sq, B * Hq, 128) || !encode_bf16_map(&tmK, k, D, Sk, B * Hkv, 128) ||
      !encode_bf16_map(&tmV, v, D, Sk, B * Hkv, 128))
    return cudaErrorInvalidValue;
  // Item order: see get_item.
  const int order = fwd_item_order(B, Hq, Hkv, Sq, Sk, D, causal);
  auto kernel = order == 1 ? attn_fwd_kernel<D, 1> : attn_fwd_kernel<D, 0>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kernel),
                                   static_cast<int>(C::kSmemBytes));
  if (e != cudaSuccess) return e;
  FwdParams p;
  p.o = o;
  p.o_bf16 = o_bf16;
  p.o_v8 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
  p.o_bytes = static_cast<size_t>(num_splits) * B * Hq * Sq * D * (o_bf16 ? 2 : 4);
  p.lse_bytes = static_cast<size_t>(num_splits) * B * Hq * Sq * sizeof(float);
  p.lse = lse;
  p.status = status;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.causal = causal;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.num_pairs = (Sq + kRowsPerItem - 1) / kRowsPerItem;
  p.head_pairs = fwd_head_pairs(Hq, Hkv, Sq);
  const int kv_tiles = (Sk + 127) / 128;
  p.num_splits = num_splits;
  p.split_tiles = (kv_tiles + num_splits - 1) / num_splits;
  p.split_stride_o = static_cast<size_t>(B) * Hq * Sq * D;
  p.split_stride_lse = static_cast<size_t>(B) * Hq * Sq;
  p.total_items = static_cast<int>(fwd_items_per_split(B, Hq, Hkv, Sq) * num_splits);
  const int grid = p.total_items < sm_count() ? p.total_items : sm_count();
  return launch_programmatic(kernel, dim3(grid), dim3(kThreads), C::kSmemBytes, stream, tmQ,
                             tmK, tmV, p);
}

}  // namespace

cudaError_t launch_attn_fwd(const void* q, const void* k, const void* v, void* o, int o_bf16,
                            float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                            float scale, cudaStream_t stream, int* status) {
  if (D == 256)
    return launch_attn_fwd_d256(q, k, v, o, o_bf16, lse, B, Hq, Hkv, Sq, Sk, causal, scale,
                                stream, status);
  if (D == 128)
    return launch_fwd_impl<128>(q, k, v, o, o_bf16, lse, B, Hq, Hkv, Sq, Sk, causal, 1, scale,
                                stream, status);
  return launch_fwd_impl<64>(q, k, v, o, o_bf16, lse, B, Hq, Hkv, Sq, Sk, causal, 1, scale,
                             stream, status);
}

cudaError_t launch_attn_fwd_splitkv(const void* q, const void* k, const void* v, float* o_part,
                                    float* lse_part, int B, int Hq, int Hkv, int Sq, int Sk,
                                    int D, int causal, int num_splits, float scale,
                                    cudaStream_t stream, int* status) {
  if (D == 128)
    return launch_fwd_impl<128>(q, k, v, o_part, 0, lse_part, B, Hq, Hkv, Sq, Sk, causal,
                                num_splits, scale, stream, status);
  return launch_fwd_impl<64>(q, k, v, o_part, 0, lse_part, B, Hq, Hkv, Sq, Sk, causal,
                             num_splits, scale, stream, status);
}

}  // namespace attn
