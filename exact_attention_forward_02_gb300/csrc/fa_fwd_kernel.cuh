// fa_fwd_kernel.cuh -- the forward attention kernel (device code). Included by fa_fwd.cu.
//
// What it computes (CS336 lecture 5 "05_flash_attention.py", part 2, flash_attention_forward;
// "Flash Attention" (blog.cyberangel.work), sections "Online Softmax" and "平行化"):
// for each query tile Q_i and each key/value tile (K_j, V_j), in order of j,
//     S    = tau * Q_i K_j^T            (masked to -inf where a key is not visible)
//     m'   = max(m, rowmax(S))
//     P    = exp(S - m')
//     l    = exp(m - m') l + rowsum(P)
//     O~   = exp(m - m') O~ + P V_j
// and finally O = O~ / l, L = m + ln l. The scores never leave the SM.
//
// With dropout ("Flash Attention" page, "Algorithm 2") the P fed to the second product is
// masked by the Philox mask of philox.cuh, l stays the sum of the undropped P, and the
// epilogue divides by l (1 - p).
//
// GB300 mapping (one persistent CTA per SM, 12 warps):
//   warp 8      TMA producer: loads the two 128-row Q tiles of a work item once, then
//               streams K_j, V_j through a ring of shared-memory slots (mbarrier pipeline).
//   warp 9      MMA issuer for both Q tiles (warp-converged, one elected lane): issues
//               tcgen05.mma for S = Q K^T (both operands K-major in shared memory, fp32
//               accumulator in Tensor Memory) and O~ += P V (P read from Tensor Memory,
//               V MN-major in shared memory), and signals completion with tcgen05.commit.
//   warps 10,11 store warps, one per Q tile: the softmax warps hand each finished slice of
//               O (or of a stream-K partial state) over in a shared-memory stage, and the
//               store warp copies it to global memory with TMA while they go on.
//   warps 0-7   two softmax warpgroups, one per Q tile (ping-pong): thread r owns query
//               row r of its tile (TMEM lane r), reads its 128 scores with tcgen05.ld,
//               applies the mask, keeps (m, l) in registers in base-2 units (the scale is
//               folded with log2(e)), writes P as 16-bit values over its scores in Tensor
//               Memory, rescales O~ in TMEM when the running max grows by more than 2^8,
//               and runs the epilogue.
// Work items are (batch*head, 256-row query block); causal items run heaviest first.
#pragma once

#include <cuda.h>
#include <math.h>
#include <stdint.h>

#include "fa_fwd.h"
#include "philox.cuh"
#include "sm103_ptx.cuh"

// Device-side status word (one per device that loads the library; this header is compiled
// once, as part of fa_fwd.cu).
__device__ int g_fa_status;

namespace fa {

constexpr int BM = 128;                  // query rows per tile = TMEM lanes
constexpr int BN = 128;                  // keys per K/V tile
constexpr int NUM_WARPS = 12;            // three warpgroups: softmax 0, softmax 1, load/MMA
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int WARP_LOAD = 8;
constexpr int WARP_MMA = 9;              // issues every MMA and owns the TMEM allocation
constexpr int WARP_STORE0 = 10;          // warps 10 and 11: TMA stores of Q tile 0 and 1
// Register split (launch: 384 threads x 168): the load/MMA warpgroup gives registers
// to the two softmax warpgroups: 2*128*200 + 128*104 = 64512 = 384*168.
constexpr uint32_t REGS_SOFTMAX = 200;
constexpr uint32_t REGS_OTHER = 104;
constexpr uint32_t TMEM_COLS = 512;      // S0 | S1 | O0 | O1, 128 columns each
constexpr uint32_t TMEM_S0 = 0, TMEM_O0 = 256;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units: rescale O~ only when m grows > 2^8
constexpr int SMEM_LIMIT = 232448;       // 227 KB opt-in dynamic shared memory per CTA
// Columns of one stream-K partial state (O~[d], m, l), each stored for the 128 rows of a
// Q tile; the host sizes the workspace with the same function.
__host__ __device__ constexpr int part_cols(int d) { return d + 2; }
constexpr int MAX_SLOTS = 8;
// Epilogue stage of one Q tile: one 64-column box of O in 16 bits (128 rows x 128 bytes,
// 128-byte swizzled as the O tensor map expects) or 32 fp32 columns of a partial state.
constexpr int STAGE_BYTES = 16384;
enum StageKind : int {
  STAGE_O_BOX = 0,      // box (x, y, z) of O
  STAGE_PART = 1,       // `bytes` of a partial state to `dst`
  STAGE_PART_LAST = 2,  // m and l of a partial state; then count the piece (and merge if last)
  STAGE_EXIT = 3,       // no more stores
};
struct StageCmd {
  int kind;
  int x, y, z;     // STAGE_O_BOX: box coordinates (column, row, head); z is also the head
  float* dst;      // STAGE_PART*: destination
  uint32_t bytes;
  int item, n_kv;  // STAGE_PART_LAST: the piece
  int q0;          //                  and its first query row
};

struct Barriers {
  uint64_t q_full, q_empty;
  uint64_t kv_full[MAX_SLOTS];
  uint64_t kv_release[MAX_SLOTS];  // release unit m = {V of tile m-1, K of tile m}
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t mma_drain;
  uint64_t stage_full[2], stage_empty[2];  // per Q tile: stage written / copied out
  uint64_t decided[2];                      // per Q tile: merge_now holds this piece's choice
  StageCmd cmd[2];
  int merge_now[2];
  uint32_t tmem_base;
  int abort_flag;
};

// ESZ: bytes per input element (2 for fp16/bf16, 1 for E4M3)
template <int D, int ESZ = 2>
struct Layout {
  static constexpr int TILE_BYTES = BM * D * ESZ;     // one Q, K or V tile (V^T for E4M3)
  static constexpr int CHUNK_BYTES = BM * 128;        // 128 rows x one 128-byte swizzle span
  static constexpr int CHUNKS = D * ESZ / 128;        // 128-byte spans per row
  static constexpr int CHUNK_ELEMS = 128 / ESZ;       // elements per span
  static constexpr int FIXED = 2 * TILE_BYTES + 2 * STAGE_BYTES + 1024 /*align*/ + 512 /*bars*/;
  static constexpr int SLOTS_FIT = (SMEM_LIMIT - FIXED) / TILE_BYTES;
  static constexpr int KV_SLOTS = SLOTS_FIT > MAX_SLOTS ? MAX_SLOTS : SLOTS_FIT;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + 2 * TILE_BYTES;
  static constexpr int OFF_STAGE = OFF_KV + KV_SLOTS * TILE_BYTES;  // 1024-byte aligned
  static constexpr int OFF_BAR = OFF_STAGE + 2 * STAGE_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + (int)sizeof(Barriers) + 1024;
  static_assert(KV_SLOTS >= 2, "need at least two K/V slots");
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
};

struct Params {
  void* O;
  float* L;
  int BH, Nq, Nk;
  int n_qblk;      // ceil(Nq / 256)
  int n_items;     // n_qblk * BH
  int n_kv_all;    // ceil(Nk / 128)
  float c;         // scale * log2(e)
  unsigned long long wait_limit_ns;
  // dropout (kernels instantiated with DROP only)
  uint32_t drop_bias;    // (0x100 - t) * 0x00010001 for the 8-bit threshold t
  uint32_t drop_offset;  // counter word 3
  float drop_rscale;     // 256 / (256 - t)
  PhiloxKeys drop_keys;  // round keys of the seed
  float o_scale;         // extra factor on O (the V descale of E4M3 inputs; 1 otherwise)
  // stream-K split of the key range (full attention with a workspace): the flattened
  // (item, K/V tile) sequence is cut into gridDim.x equal contiguous ranges
  int streamk;
  float* ws_part;  // partial states: [CTA][slot 2][Q tile 2][D + 2][128 rows] fp32 (O~, m, l),
                   // stored column by column so that a warp's accesses are coalesced
  int* ws_cnt;     // per (item, Q tile): K/V tiles accounted for; back to 0 after use
  long long ws_part_len, ws_cnt_len;  // their lengths in elements (checked by debug builds)
};

// Debug builds (FA_DEBUG) check every stream-K workspace access against the workspace's
// layout: an index outside it records FA_ERR_BOUNDS in the status word and the access is
// skipped or redirected to the workspace's start (never a trap). Release builds compile the
// checks out.
__device__ __forceinline__ bool ws_in_range(long long first, long long count, long long len) {
#ifdef FA_DEBUG
  if (first < 0 || count < 0 || first + count > len) {
    atomicCAS(&g_fa_status, 0, FA_ERR_BOUNDS);
    return false;
  }
#else
  (void)first;
  (void)count;
  (void)len;
#endif
  return true;
}

// Debug builds also check the coordinates of every TMA tile copy against the tensor's
// extents (x the innermost, in elements): x on a 16-byte boundary and the tile's first
// element inside the tensor. A load outside is recorded only (TMA fills what lies outside,
// and the load's barrier still expects its bytes); a store outside is recorded and skipped.
__device__ __forceinline__ bool tile_in_range(int x, int y, int z, int xdim, int ydim, int zdim,
                                              int esz) {
#ifdef FA_DEBUG
  if (x < 0 || (x * esz) % 16 != 0 || x >= xdim || y < 0 || y >= ydim || z < 0 || z >= zdim) {
    atomicCAS(&g_fa_status, 0, FA_ERR_BOUNDS);
    return false;
  }
#else
  (void)x, (void)y, (void)z, (void)xdim, (void)ydim, (void)zdim, (void)esz;
#endif
  return true;
}

// ----------------------------------------------------------------------------- waits
__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       unsigned long long limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicCAS(&g_fa_status, 0, FA_ERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}
// Drain wait used on the way out after an abort: ignores the abort flag, still bounded.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicCAS(&g_fa_status, 0, FA_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}
// Bounded wait: true when the phase of `parity` completed; false when the wait gave up
// (the status word then holds FA_ERR_TIMEOUT) or another role already gave up.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, abort_flag, limit_ns);
}

struct Item {
  int bh, q0;
  int j0, n_kv;    // this piece covers K/V tiles [j0, j0 + n_kv) of the item
  int n_kv0;       // of which the first n_kv0 reach Q tile 0 (causal: one fewer, the last
                   // tile lies wholly above tile 0's diagonal)
  bool has1;       // the second 128-row tile holds at least one valid query row
  bool partial;    // the piece covers only part of the item's key range
  int item;        // linear item index
  int slot;        // partial-row slot of this CTA: 0 = first piece of its range, 1 = last
};

// The r-th work item of this CTA. Items are ordered by decreasing cost (causal) and
// dealt out boustrophedon: CTA b takes b, 2G-1-b, 2G+b, 4G-1-b, ... so that every CTA
// gets one item from each "row" of G items, alternating heavy and light ends.
__device__ __forceinline__ int item_of(int r, const Params& p) {
  const int G = gridDim.x, b = blockIdx.x;
  const int base = r * G;
  return base + ((r & 1) ? (G - 1 - b) : b);
}

template <bool CAUSAL>
__device__ __forceinline__ Item decode_item(int t, const Params& p) {
  Item it;
  int qblk;
  if (CAUSAL) {  // heaviest (last) query blocks first
    qblk = p.n_qblk - 1 - t / p.BH;
    it.bh = t % p.BH;
  } else {       // consecutive items share a head's K/V in L2
    it.bh = t / p.n_qblk;
    qblk = t % p.n_qblk;
  }
  it.q0 = qblk * 2 * BM;
  it.has1 = it.q0 + BM < p.Nq;
  if (CAUSAL) {
    const int last_row = min(it.q0 + 2 * BM, p.Nq) - 1;
    it.n_kv = min(p.n_kv_all, last_row / BN + 1);
    const int last_row0 = min(it.q0 + BM, p.Nq) - 1;
    it.n_kv0 = min(p.n_kv_all, last_row0 / BN + 1);
  } else {
    it.n_kv = p.n_kv_all;
    it.n_kv0 = it.n_kv;
  }
  it.j0 = 0;
  it.partial = false;
  it.item = t;
  it.slot = 0;
  return it;
}

// Stream-K range boundaries: CTA c owns units [bound(c), bound(c+1)) of the flattened
// (item, K/V tile) sequence of W units.
__device__ __forceinline__ long long sk_bound(long long c, long long W, long long G) {
  return (c * W) / G;
}
// the CTA whose range contains unit u
__device__ __forceinline__ int sk_owner(long long u, long long W, long long G) {
  long long c = (u * G) / W;
  while (c + 1 < G && sk_bound(c + 1, W, G) <= u) ++c;
  return (int)c;
}

// Per-thread iterator over this CTA's pieces; every role walks the same sequence.
struct Sched {
  long long u, u1;  // stream-K: next unit, end of range
  int r;            // otherwise: round of the item deal
  bool first;
};

__device__ __forceinline__ Sched sched_begin(const Params& p) {
  Sched s;
  s.r = 0;
  s.first = true;
  s.u = s.u1 = 0;
  if (p.streamk) {
    const long long W = (long long)p.n_items * p.n_kv_all;
    s.u = sk_bound(blockIdx.x, W, gridDim.x);
    s.u1 = sk_bound(blockIdx.x + 1, W, gridDim.x);
  }
  return s;
}

template <bool CAUSAL>
__device__ __forceinline__ bool sched_next(Sched& s, Item& it, const Params& p) {
  if (!CAUSAL && p.streamk) {
    if (s.u >= s.u1) return false;
    const long long n = p.n_kv_all;
    const int t = (int)(s.u / n);
    const long long e = min(s.u1, (long long)(t + 1) * n);
    it = decode_item<false>(t, p);
    it.j0 = (int)(s.u - (long long)t * n);
    it.n_kv = (int)(e - s.u);
    it.n_kv0 = it.n_kv;
    it.partial = it.n_kv != p.n_kv_all;
    it.slot = s.first ? 0 : 1;
    s.first = false;
    s.u = e;
    return true;
  }
  const int t = item_of(s.r, p);
  if (t >= p.n_items) return false;
  ++s.r;
  it = decode_item<CAUSAL>(t, p);
  return true;
}

// Maximum of the N values of t as a balanced tree of three-input maxima; t is consumed.
template <int N>
__device__ __forceinline__ float tree_max(float* t) {
  if constexpr (N == 1) {
    return t[0];
  } else {
    constexpr int M = (N + 2) / 3;
#pragma unroll
    for (int i = 0; i < M; ++i) {
      const float y = 3 * i + 1 < N ? t[3 * i + 1] : -INFINITY;
      const float z = 3 * i + 2 < N ? t[3 * i + 2] : -INFINITY;
      t[i] = max3(t[3 * i], y, z);
    }
    return tree_max<M>(t);
  }
}

// ----------------------------------------------------------------------------- kernel
// BF16: type of O (and of Q, K, V unless FP8). FP8: Q, K are E4M3 [BH, N, D] and tmV maps
// V^T, E4M3 [BH, D, ldvt] (keys contiguous), so that V is a K-major operand of P V.
template <int D, bool BF16, bool CAUSAL, bool DROP, bool FP8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const Params p) {
  static_assert(!(FP8 && DROP), "dropout is not combined with E4M3 inputs");
  static_assert(!FP8 || D == 128, "E4M3 inputs need d = 128 (one 128-byte row per tile row)");
  using LY = Layout<D, FP8 ? 1 : 2>;
  constexpr int PART_COLS = part_cols(D);  // O~[D], m, l of a row, each stored for 128 rows
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle atoms
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Barriers* bars = reinterpret_cast<Barriers*>(smem + LY::OFF_BAR);
  const uint32_t sQ = smem_u32(smem + LY::OFF_Q);
  const uint32_t sKV = smem_u32(smem + LY::OFF_KV);
  const uint32_t sStage = smem_u32(smem + LY::OFF_STAGE);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->q_full), 1);
    mbar_init(smem_u32(&bars->q_empty), 1);
    for (int s = 0; s < LY::KV_SLOTS; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), 1);
      mbar_init(smem_u32(&bars->kv_release[s]), 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(smem_u32(&bars->s_full[g]), 1);
      mbar_init(smem_u32(&bars->p_full[g]), 4);    // one arrival per softmax warp
      mbar_init(smem_u32(&bars->o_done[g]), 1);
      mbar_init(smem_u32(&bars->stage_full[g]), 4);  // one arrival per softmax warp
      mbar_init(smem_u32(&bars->stage_empty[g]), 1);
      mbar_init(smem_u32(&bars->decided[g]), 1);
    }
    mbar_init(smem_u32(&bars->mma_drain), 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == WARP_LOAD && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(&bars->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const unsigned long long lim = p.wait_limit_ns;
  if (warp >= WARP_LOAD) {
  regs_dec<REGS_OTHER>();
  if (warp == WARP_LOAD) {
    // ======================================================================= producer
    if (lane == 0) {
      const uint64_t pol_kv = l2_policy_evict_last();
      const uint64_t pol_q = l2_policy_evict_first();
      // K/V loads are numbered globally (K_0 V_0 K_1 V_1 ... over all items of this CTA);
      // load i goes to slot i mod KV_SLOTS. The slot's previous occupant (load i - KV_SLOTS)
      // belongs to release unit u = (i - KV_SLOTS + 1) / 2, whose barrier is kv_release[u mod
      // KV_SLOTS] at phase u / KV_SLOTS.
      uint32_t ld = 0, q_ph = 0;
      uint32_t issued_mask = 0, last_par = 0;  // for draining on abort
      bool q_issued = false;
      bool ok = true;
      auto load_kv = [&](const CUtensorMap* tm, int bh, int row0, bool is_v) -> bool {
        const uint32_t slot = ld % LY::KV_SLOTS;
        const uint32_t par = (ld / LY::KV_SLOTS) & 1u;
        if (ld >= (uint32_t)LY::KV_SLOTS) {
          const uint32_t u = (ld - LY::KV_SLOTS + 1) >> 1;
          if (!wait_bar(smem_u32(&bars->kv_release[u % LY::KV_SLOTS]), (u / LY::KV_SLOTS) & 1u,
                        abort_flag, lim))
            return false;
        }
        const uint32_t full = smem_u32(&bars->kv_full[slot]);
        mbar_arrive_expect_tx(full, LY::TILE_BYTES);
        const uint32_t dst = sKV + slot * LY::TILE_BYTES;
        if (FP8 && is_v) {  // V^T tile: D rows (head dims) x 128 keys starting at key row0
          tile_in_range(row0, 0, bh, p.Nk, D, p.BH, 1);
          tma_load_3d_hint(dst, tm, full, row0, 0, bh, pol_kv);
        } else {
          tile_in_range(0, row0, bh, D, p.Nk, p.BH, 128 / LY::CHUNK_ELEMS);
#pragma unroll
          for (int c = 0; c < LY::CHUNKS; ++c)
            tma_load_3d_hint(dst + c * LY::CHUNK_BYTES, tm, full, c * LY::CHUNK_ELEMS, row0, bh,
                             pol_kv);
        }
        issued_mask |= 1u << slot;
        last_par = (last_par & ~(1u << slot)) | (par << slot);
        ++ld;
        return true;
      };
      Sched sch = sched_begin(p);
      Item it;
      for (int r = 0; ok && sched_next<CAUSAL>(sch, it, p); ++r) {
        ok = load_kv(&tmK, it.bh, it.j0 * BN, false);
        if (!ok) break;
        ok = wait_bar(smem_u32(&bars->q_empty), q_ph ^ 1, abort_flag, lim);
        if (!ok) break;
        q_ph ^= 1;
        const uint32_t qf = smem_u32(&bars->q_full);
        mbar_arrive_expect_tx(qf, (it.has1 ? 2 : 1) * LY::TILE_BYTES);
        tile_in_range(0, it.q0 + (it.has1 ? BM : 0), it.bh, D, p.Nq, p.BH, 128 / LY::CHUNK_ELEMS);
#pragma unroll
        for (int c = 0; c < LY::CHUNKS; ++c)
          tma_load_3d_hint(sQ + c * LY::CHUNK_BYTES, &tmQ, qf, c * LY::CHUNK_ELEMS, it.q0, it.bh,
                           pol_q);
        if (it.has1) {
#pragma unroll
          for (int c = 0; c < LY::CHUNKS; ++c)
            tma_load_3d_hint(sQ + LY::TILE_BYTES + c * LY::CHUNK_BYTES, &tmQ, qf,
                             c * LY::CHUNK_ELEMS, it.q0 + BM, it.bh, pol_q);
        }
        q_issued = true;
        ok = load_kv(&tmV, it.bh, it.j0 * BN, true);
        for (int j = 1; j < it.n_kv && ok; ++j) {
          ok = load_kv(&tmK, it.bh, (it.j0 + j) * BN, false);
          if (ok) ok = load_kv(&tmV, it.bh, (it.j0 + j) * BN, true);
        }
      }
      if (!ok) {
        // drain: every issued copy must land before the CTA may exit
        for (int s = 0; s < LY::KV_SLOTS; ++s)
          if (issued_mask & (1u << s))
            wait_drain(smem_u32(&bars->kv_full[s]), (last_par >> s) & 1u, lim);
        if (q_issued) wait_drain(smem_u32(&bars->q_full), q_ph ^ 1, lim);
      }
    }
  } else if (warp == WARP_MMA) {
    // ======================================================================= MMA issuer
    // The whole warp runs this loop converged, so descriptors and counters stay
    // warp-uniform; one elected lane issues each tcgen05.mma / commit.
    {
      // E4M3: both operands of both products K-major (V^T tiles), type code 0 = E4M3
      constexpr uint32_t ID_S = umma_idesc_f16(FP8 ? 0 : (BF16 ? 1 : 0), 0, 0, BM, BN);
      constexpr uint32_t ID_O = umma_idesc_f16(FP8 ? 0 : (BF16 ? 1 : 0), 0, FP8 ? 0 : 1, BM, D);
      // descriptors are built once; per k-step and per slot only the start-address field
      // (bits 0-13, in 16-byte units) advances, which never carries out of its field
      const uint64_t dQ0 = umma_smem_desc(sQ, 16, 1024);
      const uint64_t dK = umma_smem_desc(sKV, 16, 1024);
      const uint64_t dV = FP8 ? umma_smem_desc(sKV, 16, 1024) : umma_smem_desc(sKV, LY::CHUNK_BYTES, 1024);
      uint32_t m = 0;  // global K/V tile counter: K_m is load 2m, V_m is load 2m+1
      uint32_t q_ph = 0;
      uint32_t p_ph[2] = {0, 0};
      bool ok = true;
      auto wait_all = [&](uint32_t bar, uint32_t par) -> bool {
        return __all_sync(0xffffffffu, wait_bar(bar, par, abort_flag, lim));
      };
      auto kv_wait = [&](uint32_t ld, uint32_t& slot) -> bool {
        slot = ld % LY::KV_SLOTS;
        return wait_all(smem_u32(&bars->kv_full[slot]), (ld / LY::KV_SLOTS) & 1u);
      };
      auto commit = [&](uint64_t* bar) {
        if (elect_one()) umma_commit(smem_u32(bar));
        __syncwarp();
      };
      // S_g = Q_g K^T : M=128 rows, N=128 keys, K=D (32 bytes per instruction: 16
      // elements of 16 bits, or 32 of E4M3)
      auto issue_s = [&](int g, uint32_t kslot) {
        const uint64_t dq = dQ0 + ((g * LY::TILE_BYTES) >> 4);
        const uint64_t dk = dK + ((kslot * LY::TILE_BYTES) >> 4);
        if (elect_one()) {
#pragma unroll
          for (int ks = 0; ks < D * (FP8 ? 1 : 2) / 32; ++ks) {
            const uint32_t off = ((ks >> 2) * LY::CHUNK_BYTES + (ks & 3) * 32) >> 4;
            if constexpr (FP8)
              umma_ss_f8(tmem + TMEM_S0 + g * 128, dq + off, dk + off, ID_S, ks > 0 ? 1u : 0u);
            else
              umma_ss(tmem + TMEM_S0 + g * 128, dq + off, dk + off, ID_S, ks > 0 ? 1u : 0u);
          }
        }
        __syncwarp();
      };
      // O_g += P_g V : M=128 rows, N=D, K=128 keys; P is read from Tensor Memory
      // (E4M3: P holds four keys per TMEM column, V^T is K-major: 32 keys per instruction,
      // 8 TMEM columns and 32 bytes of every V^T row)
      auto issue_pv = [&](int g, uint32_t vslot, bool acc) {
        const uint64_t dv = dV + ((vslot * LY::TILE_BYTES) >> 4);
        if (elect_one()) {
          if constexpr (FP8) {
#pragma unroll
            for (int ks = 0; ks < BN / 32; ++ks)
              umma_ts_f8(tmem + TMEM_O0 + g * 128, tmem + TMEM_S0 + g * 128 + ks * 8,
                         dv + ((ks * 32) >> 4), ID_O, (acc || ks > 0) ? 1u : 0u);
          } else {
#pragma unroll
            for (int ks = 0; ks < BN / 16; ++ks)
              umma_ts(tmem + TMEM_O0 + g * 128, tmem + TMEM_S0 + g * 128 + ks * 8,
                      dv + ((ks * 16 * 128) >> 4), ID_O, (acc || ks > 0) ? 1u : 0u);
          }
        }
        __syncwarp();
      };
      Sched sch = sched_begin(p);
      Item it;
      for (int r = 0; ok && sched_next<CAUSAL>(sch, it, p); ++r) {
        uint32_t sK;
        ok = kv_wait(2 * m, sK) && wait_all(smem_u32(&bars->q_full), q_ph);
        if (!ok) break;
        q_ph ^= 1;
        tc_fence_after();
        issue_s(0, sK);
        commit(&bars->s_full[0]);
        if (it.has1) {
          issue_s(1, sK);
          commit(&bars->s_full[1]);
        }
        commit(&bars->kv_release[m % LY::KV_SLOTS]);
        // Q is read by the S products only: its buffer is free for the next item's Q once
        // the item's last S products complete, a K/V tile before the item ends
        if (it.n_kv == 1) commit(&bars->q_empty);
        for (int j = 0; j < it.n_kv; ++j) {
          const uint32_t mj = m + j;
          const bool has_next = j + 1 < it.n_kv;
          uint32_t sV, sKn = 0;
          bool have_kn = false;
          auto wait_kn = [&]() -> bool {  // K_(j+1), before the first S product that reads it
            if (!have_kn) {
              if (!kv_wait(2 * mj + 2, sKn)) return false;
              have_kn = true;
              tc_fence_after();
            }
            return true;
          };
          if (j < it.n_kv0) {
            ok = kv_wait(2 * mj + 1, sV) && wait_all(smem_u32(&bars->p_full[0]), p_ph[0]);
            if (!ok) break;
            p_ph[0] ^= 1;
            tc_fence_after();
            issue_pv(0, sV, j > 0);
            if (j + 1 < it.n_kv0) {
              // S_g(j+1) is issued after PV_g(j): its commit also tells the softmax warps
              // that O_g is up to date (tcgen05 ops of one thread complete in issue order)
              ok = wait_kn();
              if (!ok) break;
              issue_s(0, sKn);
              commit(&bars->s_full[0]);
            } else {
              commit(&bars->o_done[0]);
            }
          } else {
            ok = kv_wait(2 * mj + 1, sV);
            if (!ok) break;
          }
          if (it.has1) {
            ok = wait_all(smem_u32(&bars->p_full[1]), p_ph[1]);
            if (!ok) break;
            p_ph[1] ^= 1;
            tc_fence_after();
            issue_pv(1, sV, j > 0);
            if (has_next) {
              ok = wait_kn();
              if (!ok) break;
              issue_s(1, sKn);
              commit(&bars->s_full[1]);
            } else {
              commit(&bars->o_done[1]);
            }
          }
          // unit mj+1 = {V_mj, K_mj+1}: both are consumed once the MMAs above complete
          if (has_next) commit(&bars->kv_release[(mj + 1) % LY::KV_SLOTS]);
          if (j + 2 == it.n_kv) commit(&bars->q_empty);  // the item's last S products
        }
        m += it.n_kv;
      }
      // every issued MMA must finish before TMEM can be released
      commit(&bars->mma_drain);
      wait_drain(smem_u32(&bars->mma_drain), 0, lim);
      __syncwarp();
    }
  } else {
    // ======================================================================= store warps
    // Warp 10 + g copies out what softmax warpgroup g leaves in its stage, one command at a
    // time: a box of O (TMA tensor store, clipped at the end of the sequence) or a slice of
    // a partial state (bulk copy). After a partial state's last slice it waits for the
    // copies to complete, adds the piece's K/V tile count to the tile's counter, and merges
    // the item's pieces from the workspace if that completed the count.
    const int g = warp - WARP_STORE0;
    const uint32_t stg = sStage + g * STAGE_BYTES;
    // Merge of every piece of (item, Q tile g) from the workspace, four rows per lane. The
    // arithmetic and its order are those of the softmax warps' merge, so the result does
    // not depend on which piece completes the count: l is summed with explicit
    // non-contracted products and sums (an FMA contraction chosen differently in two
    // places would round differently), O~ with explicit fmaf.
    auto merge_from_workspace = [&](int item, int bh, int q0) {
      const long long W = (long long)p.n_items * p.n_kv_all;
      const long long G = gridDim.x;
      const long long ub = (long long)item * p.n_kv_all;
      const int c0 = sk_owner(ub, W, G), c1 = sk_owner(ub + p.n_kv_all - 1, W, G);
      const int slot0 = sk_bound(c0, W, G) < ub ? 1 : 0;
      const float oscale = (DROP ? p.drop_rscale : 1.f) * (FP8 ? p.o_scale : 1.f);
#pragma unroll 1
      for (int rq = 0; rq < BM / 32; ++rq) {
        const int r = rq * 32 + lane;
        const int row = q0 + g * BM + r;
        const bool valid = row < p.Nq;
        auto piece = [&](int cc) -> const float* {
          const long long base = (((long long)cc * 2 + (cc == c0 ? slot0 : 0)) * 2 + g) * PART_COLS * BM;
          return p.ws_part + (ws_in_range(base, PART_COLS * BM, p.ws_part_len) ? base : 0) + r;
        };
        uint8_t* orow = reinterpret_cast<uint8_t*>(p.O) +
                        ((size_t)bh * p.Nq + (size_t)(valid ? row : 0)) * D * 2;
        float m, l;
        if (c1 - c0 == 1) {
          const float* p0 = piece(c0);
          const float* p1 = piece(c1);
          const float m0 = __ldcg(p0 + D * BM), l0 = __ldcg(p0 + (D + 1) * BM);
          const float m1 = __ldcg(p1 + D * BM), l1 = __ldcg(p1 + (D + 1) * BM);
          m = fmaxf(m0, m1);
          const float w0 = ex2_approx(m0 - m), w1 = ex2_approx(m1 - m);
          l = __fadd_rn(__fmul_rn(l0, w0), __fmul_rn(l1, w1));
          const float inv_l = (l > 0.f ? 1.f / l : 0.f) * oscale;
          const float a0 = w0 * inv_l, a1 = w1 * inv_l;
#pragma unroll 1
          for (int q = 0; q < D / 16; ++q) {
            float x0[16], x1[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              x0[k] = __ldcg(p0 + (q * 16 + k) * BM);
              x1[k] = __ldcg(p1 + (q * 16 + k) * BM);
            }
            uint32_t w16[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              w16[k] = pack2<BF16>(fmaf(x1[2 * k], a1, x0[2 * k] * a0),
                                   fmaf(x1[2 * k + 1], a1, x0[2 * k + 1] * a0));
            if (valid) {
              uint4* dst = reinterpret_cast<uint4*>(orow + q * 32);
              dst[0] = make_uint4(w16[0], w16[1], w16[2], w16[3]);
              dst[1] = make_uint4(w16[4], w16[5], w16[6], w16[7]);
            }
          }
        } else {
          m = -INFINITY;
          for (int cc = c0; cc <= c1; ++cc) m = fmaxf(m, __ldcg(piece(cc) + D * BM));
          l = 0.f;
          for (int cc = c0; cc <= c1; ++cc) {
            const float* pc = piece(cc);
            l = __fadd_rn(l, __fmul_rn(__ldcg(pc + (D + 1) * BM), ex2_approx(__ldcg(pc + D * BM) - m)));
          }
          const float inv_l = (l > 0.f ? 1.f / l : 0.f) * oscale;
#pragma unroll 1
          for (int q = 0; q < D / 16; ++q) {
            float acc[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) acc[k] = 0.f;
            for (int cc = c0; cc <= c1; ++cc) {
              const float* pc = piece(cc);
              const float wgt = ex2_approx(__ldcg(pc + D * BM) - m) * inv_l;
#pragma unroll
              for (int k = 0; k < 16; ++k) acc[k] = fmaf(__ldcg(pc + (q * 16 + k) * BM), wgt, acc[k]);
            }
            uint32_t w16[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) w16[k] = pack2<BF16>(acc[2 * k], acc[2 * k + 1]);
            if (valid) {
              uint4* dst = reinterpret_cast<uint4*>(orow + q * 32);
              dst[0] = make_uint4(w16[0], w16[1], w16[2], w16[3]);
              dst[1] = make_uint4(w16[4], w16[5], w16[6], w16[7]);
            }
          }
        }
        if (valid) p.L[(size_t)bh * p.Nq + row] = (m + log2f(l)) * 0.69314718055994531f;
      }
    };
    uint32_t f_ph = 0;
    while (true) {
      if (!__all_sync(0xffffffffu, wait_bar(smem_u32(&bars->stage_full[g]), f_ph, abort_flag, lim)))
        break;
      f_ph ^= 1;
      const StageCmd c = bars->cmd[g];
      if (c.kind == STAGE_EXIT) break;
      if (lane == 0) {
        if (c.kind == STAGE_O_BOX) {
          if (tile_in_range(c.x, c.y, c.z, D, p.Nq, p.BH, 2)) tma_store_3d(&tmO, stg, c.x, c.y, c.z);
        }
        else if (ws_in_range(c.dst - p.ws_part, c.bytes / 4, p.ws_part_len))
          bulk_store_s2g(c.dst, stg, c.bytes);
        bulk_commit();
        bulk_wait_read0();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->stage_empty[g]));
      if (c.kind == STAGE_PART_LAST) {
        int last = 0;
        if (lane == 0) {
          bulk_wait0();  // the piece's whole state is in global memory
          fence_proxy_async_global();
          __threadfence();
          int* cnt = p.ws_cnt + (size_t)c.item * 2 + g;
          last = ws_in_range((long long)c.item * 2 + g, 1, p.ws_cnt_len) &&
                 atomicAdd(cnt, c.n_kv) + c.n_kv == p.n_kv_all;
          if (last) {
            atomicExch(cnt, 0);  // every piece is in: ready for the next call
            __threadfence();
          }
        }
        if (__shfl_sync(0xffffffffu, last, 0)) merge_from_workspace(c.item, c.z, c.q0);
      }
    }
    if (lane == 0) bulk_wait0();  // no copy of this warp is still in flight at exit
    __syncwarp();
  }
  // exit: every role of the CTA has finished with Tensor Memory
  tc_fence_before();
  named_bar_sync(1, NUM_THREADS);
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
  } else {
    regs_inc<REGS_SOFTMAX>();
    // ======================================================================= softmax
    const int g = warp >> 2;         // which Q tile / warpgroup
    const int wq = warp & 3;         // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;    // row within the tile
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + TMEM_S0 + g * 128;
    const uint32_t tO = tmem + lane_off + TMEM_O0 + g * 128;
    const float c = p.c;
    uint32_t s_ph = 0, o_ph = 0;
    // this tile's epilogue stage: before fill n, the store warp has copied out fill n - 1
    const uint32_t stg = sStage + g * STAGE_BYTES;
    uint32_t n_fill = 0, dec_ph = 0;
    auto stage_acquire = [&]() -> bool {
      const bool w2 = wait_bar(smem_u32(&bars->stage_empty[g]), (n_fill & 1u) ^ 1u, abort_flag, lim);
      ++n_fill;
      return __all_sync(0xffffffffu, w2);
    };
    // hand the stage to the store warp; `it` is the current piece
    Item it = {};
    auto stage_release = [&](int kind, int x, float* dst, uint32_t bytes) {
      fence_proxy_async_smem();  // this thread's stage writes -> visible to the TMA copy
      if (r == 0) {
        StageCmd& c = bars->cmd[g];
        c.kind = kind;
        c.x = x;
        c.y = it.q0 + g * BM;
        c.z = it.bh;
        c.dst = dst;
        c.bytes = bytes;
        c.item = it.item;
        c.n_kv = it.n_kv;
        c.q0 = it.q0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->stage_full[g]));
    };
    bool ok = true;
    Sched sch = sched_begin(p);
    for (int rr = 0; ok && sched_next<CAUSAL>(sch, it, p); ++rr) {
      if (g == 1 && !it.has1) continue;
      const int row = it.q0 + g * BM + r;
      const int kv_lim = CAUSAL ? min(row + 1, p.Nk) : p.Nk;  // keys [0, kv_lim) visible
      float m_run = -INFINITY, l_run = 0.f;
      const int n_kv_g = g == 0 ? it.n_kv0 : it.n_kv;  // K/V tiles that reach this Q tile
      for (int j = 0; j < n_kv_g; ++j) {
        // dropout: the keep bits of this row for K/V tile j, drawn before S_g(j) is ready
        // (they do not depend on it), so the generator runs while this warpgroup would
        // otherwise wait for the tensor core
        uint32_t kbits[4] = {0, 0, 0, 0};
        if constexpr (DROP)
          dropout_row_bits((uint32_t)(it.j0 + j) * (BN / 16), (uint32_t)row, (uint32_t)it.bh,
                           p.drop_offset, p.drop_keys, p.drop_bias, kbits);
        // S_g(j) ready; for j > 0 this also means PV_g(j-1) has completed
        ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->s_full[g]), s_ph, abort_flag, lim));
        if (!ok) break;
        s_ph ^= 1;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, sr[q]);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q) reg_fence(sr[q]);

        const int vis = kv_lim - (it.j0 + j) * BN;
        const bool full = vis >= BN;
        auto sv = [&](int k) { return __uint_as_float(sr[k >> 5][k & 31]); };
        // raw row max over the visible keys: a balanced tree of three-input maxima (depth 5
        // for 128 keys, against 16 for four running chains). The E4M3 instantiation keeps
        // the four chains: with its products at half the 16-bit tensor time, the tree
        // measured 1 % slower there (causal B=2, H=8, N=8192: 185.0 against 182.9 us).
        float mt;
        if constexpr (FP8) {
          float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          if (full) {
#pragma unroll
            for (int k = 0; k < 64; ++k) mx[k & 3] = max3(mx[k & 3], sv(2 * k), sv(2 * k + 1));
          } else {
#pragma unroll
            for (int k = 0; k < 64; ++k)
              mx[k & 3] = max3(mx[k & 3], 2 * k < vis ? sv(2 * k) : -INFINITY,
                               2 * k + 1 < vis ? sv(2 * k + 1) : -INFINITY);
          }
          mt = fmaxf(max3(mx[0], mx[1], mx[2]), mx[3]);
        } else {
          float t[43];
          if (full) {
#pragma unroll
            for (int i = 0; i < 42; ++i) t[i] = max3(sv(3 * i), sv(3 * i + 1), sv(3 * i + 2));
            t[42] = fmaxf(sv(126), sv(127));
          } else {
            auto mv = [&](int e) { return e < vis ? sv(e) : -INFINITY; };
#pragma unroll
            for (int i = 0; i < 42; ++i) t[i] = max3(mv(3 * i), mv(3 * i + 1), mv(3 * i + 2));
            t[42] = fmaxf(mv(126), mv(127));
          }
          mt = tree_max<43>(t);
        }
        const float m_tile = (mt == -INFINITY) ? -INFINITY : mt * c;
        float m_new = m_run, alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          m_new = m_tile;
        } else if (m_tile > m_run + RESCALE_THRESHOLD) {
          m_new = m_tile;
          alpha = ex2_approx(m_run - m_new);
          rescale = true;
        }
        const float nb = (m_new == -INFINITY) ? 0.f : -m_new;
        // P = exp2(S*c - m): the scaling in packed pairs, the exponentials on the MUFU,
        // the row sum in packed pairs; P is packed to 16-bit pairs (key 2k in the low
        // half, key 2k+1 in the high half) for the second product
        const uint64_t c2 = f2(c, c), nb2 = f2(nb, nb);
        uint64_t acc[4] = {0, 0, 0, 0};
        uint32_t pk[2][32];
        // dropout: l keeps the undropped sum; only the 16-bit P of the second product is
        // masked, pair k by the bits (k & 15, 16 + (k & 15)) of kbits[k >> 4]
        auto drop_pair = [&](int k, uint32_t w) -> uint32_t {
          if constexpr (DROP) {
            return w & pair_mask(kbits[k >> 4], k & 15);
          } else {
            return w;
          }
        };
        // P of key pair k (keys 2k, 2k+1) into the packed words of the second product:
        // two 16-bit values per word, or (E4M3) four 8-bit values per word, lowest key in
        // the lowest bits; k is a compile-time constant in the unrolled loops below
        float pe0 = 0.f, pe1 = 0.f;
        auto emit = [&](int k, float p0, float p1) {
          if constexpr (FP8) {
            if ((k & 1) == 0) {
              pe0 = p0;
              pe1 = p1;
            } else {
              pk[(k >> 1) >> 5][(k >> 1) & 31] = pack4_e4m3(pe0, pe1, p0, p1);
            }
          } else {
            pk[k >> 5][k & 31] = drop_pair(k, pack2<BF16>(p0, p1));
          }
        };
        // two branch-free copies of the loop (full tile / masked tile) so that the
        // scheduler can overlap the exponentials of many iterations
        if (full) {
#pragma unroll
          for (int k = 0; k < 64; ++k) {
            float t0, t1;
            f2_split(f2_fma(f2(sv(2 * k), sv(2 * k + 1)), c2, nb2), t0, t1);
            const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
            acc[k & 3] = f2_add(acc[k & 3], f2(p0, p1));
            emit(k, p0, p1);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 64; ++k) {
            float t0, t1;
            f2_split(f2_fma(f2(sv(2 * k), sv(2 * k + 1)), c2, nb2), t0, t1);
            const float p0 = 2 * k < vis ? ex2_approx(t0) : 0.f;
            const float p1 = 2 * k + 1 < vis ? ex2_approx(t1) : 0.f;
            acc[k & 3] = f2_add(acc[k & 3], f2(p0, p1));
            emit(k, p0, p1);
          }
        }
        float ls;
        {
          float a0, a1, b0, b1;
          f2_split(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
          (void)b0; (void)b1;
          ls = a0 + a1;
        }

        // rescale O~ (in TMEM) when this row's max grew past the threshold
        if (__any_sync(0xffffffffu, rescale)) {
          const uint64_t al2 = f2(alpha, alpha);
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            tmem_ld32(tO + q * 32, o);
            tmem_wait_ld();
            reg_fence(o);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              float x0, x1;
              f2_split(f2_mul(f2(__uint_as_float(o[2 * k]), __uint_as_float(o[2 * k + 1])), al2), x0, x1);
              o[2 * k] = __float_as_uint(x0);
              o[2 * k + 1] = __float_as_uint(x1);
            }
            tmem_st32(tO + q * 32, o);
          }
        }
        l_run = l_run * alpha + ls;
        m_run = m_new;

        // P overwrites the first 64 (E4M3: 32) columns of this tile's S region (the A
        // operand of PV)
        tmem_st32(tS, pk[0]);
        if constexpr (!FP8) tmem_st32(tS + 32, pk[1]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[g]));
      }
      if (!ok) break;
      // ------------------------------------------------------------------ epilogue
      // O leaves through this tile's shared-memory stage: the warps write one slice (a
      // 64-column box of 16-bit O, or 32 fp32 columns of a partial state), and the store warp
      // copies it out with TMA while the warpgroup goes on to its next piece.
      {
        const bool w = wait_bar(smem_u32(&bars->o_done[g]), o_ph, abort_flag, lim);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        o_ph ^= 1;
        tc_fence_after();
        const bool valid = row < p.Nq;
        // this row's 32 values of box half h (bf16 or fp16 pairs), 128-byte swizzled: the
        // 16-byte chunk j of row r sits at chunk position j ^ (r mod 8)
        auto st_box_half = [&](int h, const uint32_t (&w16)[16]) {
          const uint32_t rowb = stg + (uint32_t)r * 128u;
#pragma unroll
          for (int v = 0; v < 4; ++v)
            st_shared_v4(rowb + ((uint32_t)((4 * h + v) ^ (r & 7)) << 4), w16[4 * v], w16[4 * v + 1],
                         w16[4 * v + 2], w16[4 * v + 3]);
        };
        if (!it.partial) {
          // O = O~ / l (with dropout O~ / (l (1 - p))), L = (m + log2 l) ln 2
          float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
          if constexpr (DROP) inv_l *= p.drop_rscale;
          if constexpr (FP8) inv_l *= p.o_scale;
          const uint64_t il2 = f2(inv_l, inv_l);
          for (int b = 0; b < D / 64; ++b) {
            ok = stage_acquire();
            if (!ok) break;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t o[32];
              tmem_ld32(tO + (2 * b + h) * 32, o);
              tmem_wait_ld();
              reg_fence(o);
              uint32_t w16[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                float x0, x1;
                f2_split(f2_mul(f2(__uint_as_float(o[2 * k]), __uint_as_float(o[2 * k + 1])), il2), x0, x1);
                w16[k] = pack2<BF16>(x0, x1);
              }
              st_box_half(h, w16);
            }
            stage_release(STAGE_O_BOX, 64 * b, nullptr, 0);
          }
          if (!ok) break;
          if (valid) p.L[(size_t)it.bh * p.Nq + row] = (m_run + log2f(l_run)) * 0.69314718055994531f;
          tc_fence_before();
        } else {
          // Part of the key range only ("Flash Attention" page, section "平行化": partial
          // states (m, l, O~) merge with the associative operator). One counter per (item,
          // Q tile) holds the K/V tiles of the pieces stored so far. If row 0's thread finds
          // all other pieces counted, the warpgroup merges at once from its Tensor Memory O~
          // and its (m, l); otherwise it stores its state through the stage and the store
          // warp counts the piece (and merges if that completes the count).
          int* cnt = p.ws_cnt + (size_t)it.item * 2 + g;
          if (r == 0) {
            bars->merge_now[g] = ws_in_range((long long)it.item * 2 + g, 1, p.ws_cnt_len) &&
                                 ld_acquire_gpu(cnt) + it.n_kv == p.n_kv_all;
            mbar_arrive(smem_u32(&bars->decided[g]));
          }
          ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->decided[g]), dec_ph, abort_flag, lim));
          if (!ok) break;
          dec_ph ^= 1;
          const bool merge = *reinterpret_cast<volatile int*>(&bars->merge_now[g]) != 0;
          if (!merge) {
            float* dst = p.ws_part + (((size_t)blockIdx.x * 2 + it.slot) * 2 + g) * PART_COLS * BM;
            for (int f = 0; f < D / 32; ++f) {
              ok = stage_acquire();
              if (!ok) break;
              uint32_t o[32];
              tmem_ld32(tO + f * 32, o);
              tmem_wait_ld();
              reg_fence(o);
              // column-major: column k of the slice holds the 128 rows in order
#pragma unroll
              for (int k = 0; k < 32; ++k) st_shared_u32(stg + (uint32_t)(k * BM + r) * 4u, o[k]);
              stage_release(STAGE_PART, 0, dst + f * 32 * BM, 32 * BM * 4);
            }
            if (!ok) break;
            ok = stage_acquire();
            if (!ok) break;
            st_shared_u32(stg + (uint32_t)r * 4u, __float_as_uint(m_run));
            st_shared_u32(stg + (uint32_t)(BM + r) * 4u, __float_as_uint(l_run));
            stage_release(STAGE_PART_LAST, 0, dst + D * BM, 2 * BM * 4);
          } else {
            if (r == 0) atomicExch(cnt, 0);  // every piece is in: ready for the next call
            const long long W = (long long)p.n_items * p.n_kv_all;
            const long long G = gridDim.x;
            const long long ub = (long long)it.item * p.n_kv_all;
            const int c0 = sk_owner(ub, W, G), c1 = sk_owner(ub + p.n_kv_all - 1, W, G);
            // the first piece is its CTA's last one (slot 1) unless that CTA's range starts
            // with this item; every later piece is its CTA's first (slot 0)
            const int slot0 = sk_bound(c0, W, G) < ub ? 1 : 0;
            auto piece = [&](int cc) -> const float* {
              const long long base = (((long long)cc * 2 + (cc == c0 ? slot0 : 0)) * 2 + g) * PART_COLS * BM;
              return p.ws_part + (ws_in_range(base, PART_COLS * BM, p.ws_part_len) ? base : 0) + r;
            };
            const int me = blockIdx.x;
            const float oscale = (DROP ? p.drop_rscale : 1.f) * (FP8 ? p.o_scale : 1.f);
            // The pieces are combined in the order of their CTAs (c0 first), whichever piece
            // merges, so that the result does not depend on which one finished last.
            float m, l;
            if (c1 - c0 == 1) {
              // one other piece (an item spans two CTAs): its m, l and the first half of
              // its O~ are loaded together, the rest while the first half is combined
              const bool first = c0 == me;
              const float* po = piece(first ? c1 : c0);
              const float mo = __ldcg(po + D * BM), lo = __ldcg(po + (D + 1) * BM);
              float x[2][32];
#pragma unroll
              for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int k = 0; k < 32; ++k) x[hh][k] = __ldcg(po + (hh * 32 + k) * BM);
              m = fmaxf(m_run, mo);
              const float w_own = ex2_approx(m_run - m), w_o = ex2_approx(mo - m);
              l = first ? __fadd_rn(__fmul_rn(l_run, w_own), __fmul_rn(lo, w_o))
                        : __fadd_rn(__fmul_rn(lo, w_o), __fmul_rn(l_run, w_own));
              const float inv_l = (l > 0.f ? 1.f / l : 0.f) * oscale;
              const float a_own = w_own * inv_l, a_o = w_o * inv_l;
              const float a0 = first ? a_own : a_o, a1 = first ? a_o : a_own;
              for (int b = 0; b < D / 64; ++b) {
                ok = stage_acquire();
                if (!ok) break;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int q = 2 * b + h;
                  uint32_t o[32];
                  tmem_ld32(tO + q * 32, o);
                  tmem_wait_ld();
                  reg_fence(o);
                  uint32_t w16[16];
#pragma unroll
                  for (int k = 0; k < 16; ++k) {
                    float acc2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                      const float own = __uint_as_float(o[2 * k + e]);
                      const float xo = x[h][2 * k + e];
                      const float x0 = first ? own : xo, x1 = first ? xo : own;
                      acc2[e] = fmaf(x1, a1, x0 * a0);
                    }
                    w16[k] = pack2<BF16>(acc2[0], acc2[1]);
                  }
                  st_box_half(h, w16);
                  if (q + 2 < D / 32) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) x[h][k] = __ldcg(po + ((q + 2) * 32 + k) * BM);
                  }
                }
                stage_release(STAGE_O_BOX, 64 * b, nullptr, 0);
              }
              if (!ok) break;
            } else {
              // three or more pieces (short ranges): one chunk of one piece at a time
              m = m_run;
              for (int cc = c0; cc <= c1; ++cc)
                if (cc != me) m = fmaxf(m, __ldcg(piece(cc) + D * BM));
              l = 0.f;
              for (int cc = c0; cc <= c1; ++cc) {
                const float* pc = piece(cc);
                const float lc = cc == me ? l_run : __ldcg(pc + (D + 1) * BM);
                const float mc = cc == me ? m_run : __ldcg(pc + D * BM);
                l = __fadd_rn(l, __fmul_rn(lc, ex2_approx(mc - m)));
              }
              const float inv_l = (l > 0.f ? 1.f / l : 0.f) * oscale;
              const float a_own = ex2_approx(m_run - m) * inv_l;
              for (int b = 0; b < D / 64; ++b) {
                ok = stage_acquire();
                if (!ok) break;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  uint32_t o[32];
                  tmem_ld32(tO + (2 * b + h) * 32, o);
                  tmem_wait_ld();
                  reg_fence(o);
                  float acc[32];
#pragma unroll
                  for (int k = 0; k < 32; ++k) acc[k] = 0.f;
                  for (int cc = c0; cc <= c1; ++cc) {
                    if (cc == me) {
#pragma unroll
                      for (int k = 0; k < 32; ++k) acc[k] = fmaf(__uint_as_float(o[k]), a_own, acc[k]);
                      continue;
                    }
                    const float* pc = piece(cc);
                    float xx[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) xx[k] = __ldcg(pc + ((2 * b + h) * 32 + k) * BM);
                    const float wgt = ex2_approx(__ldcg(pc + D * BM) - m) * inv_l;
#pragma unroll
                    for (int k = 0; k < 32; ++k) acc[k] = fmaf(xx[k], wgt, acc[k]);
                  }
                  uint32_t w16[16];
#pragma unroll
                  for (int k = 0; k < 16; ++k) w16[k] = pack2<BF16>(acc[2 * k], acc[2 * k + 1]);
                  st_box_half(h, w16);
                }
                stage_release(STAGE_O_BOX, 64 * b, nullptr, 0);
              }
              if (!ok) break;
            }
            if (valid) p.L[(size_t)it.bh * p.Nq + row] = (m + log2f(l)) * 0.69314718055994531f;
          }
          tc_fence_before();
        }
      }
    }
    // the store warp of this tile stops after the copies handed to it so far
    if (ok && stage_acquire()) stage_release(STAGE_EXIT, 0, nullptr, 0);
    // exit: the load/MMA warpgroup releases Tensor Memory after this barrier
    tc_fence_before();
    named_bar_sync(1, NUM_THREADS);
  }
}

// Bounded-wait self test: one barrier that nothing ever signals.
__global__ void fa_wait_selftest_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)wait_bar(smem_u32(&bar), 0, &abort_flag, limit_ns);
  __syncthreads();
}

}  // namespace fa
