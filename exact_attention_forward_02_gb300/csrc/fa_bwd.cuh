// fa_bwd.cuh -- attention backward (dQ, dK, dV) for GB300 (sm_103a). Included by fa_fwd.cu.
//
// What it computes (CS336 lecture 5 "05_flash_attention.py", part 3, flash_attention_backward;
// "Flash Attention" page, "Algorithm 4: backward pass" and its derivation): with
// S = tau Q K^T (masked), P = exp(S - L) recomputed from the forward's logsumexp L,
//     dV = P^T dO,  dP = dO V^T,  D_i = rowsum(dO_i o O_i),  dS = P o (dP - D),
//     dQ = tau dS K,  dK = tau dS^T Q.
// Two kernels, so that every accumulator fits Tensor Memory and nothing is accumulated
// with atomics:
//   fa_bwd_dq_kernel  one 128-row query tile per CTA, looping over key tiles: computes
//                     D (stored for the second kernel) and dQ; TMEM: S | dP | dQ.
//   fa_bwd_dkv_kernel one 128-key tile per CTA, looping over query tiles: the transposed
//                     products S^T = K Q^T and dP^T = V dO^T, then dV += P^T dO and
//                     dK += dS^T Q; TMEM: S^T | dP^T | dK | dV.
// Roles per CTA (10 warps): warps 0-7 elementwise work in two warpgroups that split the
// tile's 128 columns in halves (thread r of either warpgroup owns TMEM lane r, warpgroup h
// columns [64h, 64h + 64)), warp 8 TMA producer, warp 9 MMA issuer (warp-converged, one
// elected lane issues). The 16-bit operands do not overwrite the scores of the next
// product: dS has its own columns in the dQ kernel, and P^T, dS^T share S^T's columns in
// the dK/dV kernel, so that the next tile's (dQ kernel: both, dK/dV kernel: dP^T) score
// products run while the elementwise warps work.
#pragma once

namespace fa {

constexpr int BW_EW_WARPS = 8;  // elementwise warps (two warpgroups)
constexpr int BW_WARPS = BW_EW_WARPS + 2;
constexpr int BW_THREADS = BW_WARPS * 32;
constexpr int BW_WARP_LOAD = 8;
constexpr int BW_WARP_MMA = 9;
constexpr int BW_MAX_SLOTS = 8;


struct BwdParams {
  const void* O;      // dq kernel: forward output (16-bit), for D
  const void* dO;     // dq kernel: upstream gradient rows (16-bit), for D
  const float* L;     // forward logsumexp (natural log), [BH, Nq]
  float* Dws;         // D = rowsum(dO o O), [BH, Nq] fp32 (written by the dq kernel)
  void* dQ;           // outputs (16-bit)
  void* dK;
  void* dV;
  int BH, Nq, Nk;
  int n_qt, n_kt;     // ceil(Nq/128), ceil(Nk/128)
  int n_items;
  float c;            // scale * log2(e)
  float scale;
  unsigned long long wait_limit_ns;
  // dropout (kernels instantiated with DROP): the mask of the forward's (seed, offset)
  uint32_t drop_bias;     // (0x100 - t) * 0x00010001 for the 8-bit threshold t
  uint32_t drop_offset;
  float drop_rscale;      // 256 / (256 - t)
  PhiloxKeys drop_keys;
};

struct BwdBars {
  uint64_t a_full, a_empty;            // the CTA's resident tiles (Q+dO, or K+V)
  uint64_t full[BW_MAX_SLOTS];         // streamed tile pairs (dQ kernel: K tiles)
  uint64_t release[BW_MAX_SLOTS];
  uint64_t vfull[BW_MAX_SLOTS];        // dQ kernel: V tiles, a ring of their own
  uint64_t vrelease[BW_MAX_SLOTS];
  uint64_t s_full;                      // both score products of the current tile in TMEM
  uint64_t sdp_free;                    // the elementwise warps hold the scores in registers
  uint64_t op_done;                     // the previous tile's accumulating products completed
  uint64_t pt_full;                     // dK/dV kernel: P^T written back (dV may start)
  uint64_t dp_full, dp_read;            // dK/dV kernel: dP^T computed / read by every EW warp
  uint64_t p_full;                      // 16-bit operands written back to TMEM
  uint64_t done;                        // accumulators final for the current item
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
struct BwdLayout {
  static constexpr int TILE_BYTES = BM * D * 2;
  static constexpr int CHUNK_BYTES = BM * 128;
  static constexpr int CHUNKS = D / 64;
  static constexpr int PAIR_BYTES = 2 * TILE_BYTES;   // a streamed pair of tiles
  static constexpr int FIXED = 2 * TILE_BYTES + 1024 + 1024;
  static constexpr int SLOTS_FIT = (SMEM_LIMIT - FIXED) / PAIR_BYTES;
  static constexpr int SLOTS = SLOTS_FIT > BW_MAX_SLOTS ? BW_MAX_SLOTS : SLOTS_FIT;
  static constexpr int OFF_A = 0;                     // resident pair
  static constexpr int OFF_S = 2 * TILE_BYTES;        // streamed pairs
  static constexpr int OFF_LD = OFF_S + SLOTS * PAIR_BYTES;  // 2 x 128 floats (L, D of a tile)
  static constexpr int OFF_BAR = OFF_LD + 1024;
  static constexpr int SMEM_BYTES = OFF_BAR + (int)sizeof(BwdBars) + 1024;
  static_assert(SLOTS >= 2, "need two streamed slots");
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
};

// dQ kernel: K and V stream through rings of their own, because V_j is read only by the
// dP product and can leave long before K_j, which the dQ product still reads: a deeper
// K ring then lets the next tiles' loads start early enough to hide their latency.
template <int D>
struct DqLayout {
  static constexpr int TILE_BYTES = BM * D * 2;
  static constexpr int CHUNK_BYTES = BM * 128;
  static constexpr int CHUNKS = D / 64;
  static constexpr int FIXED = 2 * TILE_BYTES + 1024 + 1024;
  static constexpr int V_SLOTS = 2;
  static constexpr int K_FIT = (SMEM_LIMIT - FIXED - V_SLOTS * TILE_BYTES) / TILE_BYTES;
  static constexpr int K_SLOTS = K_FIT > BW_MAX_SLOTS ? BW_MAX_SLOTS : K_FIT;
  static constexpr int OFF_A = 0;                           // Q, dO (resident)
  static constexpr int OFF_K = 2 * TILE_BYTES;              // K ring
  static constexpr int OFF_V = OFF_K + K_SLOTS * TILE_BYTES;  // V ring
  static constexpr int OFF_BAR = OFF_V + V_SLOTS * TILE_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + (int)sizeof(BwdBars) + 1024;
  static_assert(K_SLOTS >= 3, "need three K slots");
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
};

// the r-th item of this CTA: boustrophedon deal (b, 2G-1-b, 2G+b, ...) of items sorted
// by decreasing cost
__device__ __forceinline__ int bw_item_of(int r) {
  const int G = gridDim.x, b = blockIdx.x;
  return r * G + ((r & 1) ? (G - 1 - b) : b);
}

__device__ __forceinline__ void store_row16(void* base, size_t row, int d_cols, int q32,
                                            const uint32_t (&w16)[16]) {
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(base) + row * d_cols * 2 + q32 * 64);
#pragma unroll
  for (int v = 0; v < 4; ++v) dst[v] = make_uint4(w16[4 * v], w16[4 * v + 1], w16[4 * v + 2], w16[4 * v + 3]);
}

// ============================================================================ dQ kernel
// CTA item: (bh, query tile qt). Streams K_j, V_j; per key tile:
//   S = Q K_j^T, dP = dO V_j^T  (TMEM)  ->  dS = P o (dP - D)  (16-bit, over S)  ->  dQ += dS K_j
template <int D, bool BF16, bool CAUSAL, bool DROP>
__global__ void __launch_bounds__(BW_THREADS, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                     const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const BwdParams p) {
  using LY = DqLayout<D>;
  // dS gets its own 64 columns, so that S and dP are free as soon as the elementwise warps
  // have read them: the next tile's score products then overlap the elementwise pass
  constexpr uint32_t T_S = 0, T_DP = 128, T_DQ = 256, T_DS = 384, T_COLS = 512;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + LY::OFF_BAR);
  const uint32_t sA = smem_u32(smem + LY::OFF_A);   // Q tile, then dO tile
  const uint32_t sK = smem_u32(smem + LY::OFF_K);   // K ring
  const uint32_t sV = smem_u32(smem + LY::OFF_V);   // V ring
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_kv_all = p.n_kt;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->a_full), 1);
    mbar_init(smem_u32(&bars->a_empty), 1);
    for (int s = 0; s < LY::K_SLOTS; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->release[s]), 1);
    }
    for (int s = 0; s < LY::V_SLOTS; ++s) {
      mbar_init(smem_u32(&bars->vfull[s]), 1);
      mbar_init(smem_u32(&bars->vrelease[s]), 1);
    }
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->sdp_free), BW_EW_WARPS);
    mbar_init(smem_u32(&bars->op_done), 1);
    mbar_init(smem_u32(&bars->p_full), BW_EW_WARPS);  // one arrival per elementwise warp
    mbar_init(smem_u32(&bars->done), 1);
    mbar_init(smem_u32(&bars->mma_drain), 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == BW_WARP_MMA) {
    tmem_alloc(smem_u32(&bars->tmem_base), T_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const unsigned long long lim = p.wait_limit_ns;

  // causal: heaviest (last) query tiles first; full: head by head (K/V reuse in L2)
  auto item_tiles = [&](int t, int& bh, int& q0, int& n_kv) {
    if (CAUSAL) {
      bh = t % p.BH;
      q0 = (p.n_qt - 1 - t / p.BH) * BM;
    } else {
      bh = t / p.n_qt;
      q0 = (t % p.n_qt) * BM;
    }
    n_kv = CAUSAL ? min(n_kv_all, (min(q0 + BM, p.Nq) - 1) / BN + 1) : n_kv_all;
  };

  if (warp == BW_WARP_LOAD) {
    if (lane == 0) {
      // streamed tiles are read by every CTA working on the same head: keep them in L2;
      // the CTA's resident tiles are read once
      const uint64_t pol_reuse = l2_policy_evict_last();
      const uint64_t pol_once = l2_policy_evict_first();
      uint32_t j_glob = 0, a_ph = 0;
      bool ok = true;
      uint32_t issued = 0, last_par = 0, vissued = 0, vlast_par = 0;
      bool a_issued = false;
      for (int rr_ = 0, t = bw_item_of(0); t < p.n_items && ok; t = bw_item_of(++rr_)) {
        int bh, q0, n_kv;
        item_tiles(t, bh, q0, n_kv);
        ok = wait_bar(smem_u32(&bars->a_empty), a_ph ^ 1, abort_flag, lim);
        if (!ok) break;
        a_ph ^= 1;
        const uint32_t af = smem_u32(&bars->a_full);
        mbar_arrive_expect_tx(af, 2 * LY::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < LY::CHUNKS; ++c) {
          tma_load_3d_hint(sA + c * LY::CHUNK_BYTES, &tmQ, af, c * 64, q0, bh, pol_once);
          tma_load_3d_hint(sA + LY::TILE_BYTES + c * LY::CHUNK_BYTES, &tmdO, af, c * 64, q0, bh, pol_once);
        }
        a_issued = true;
        for (int j = 0; j < n_kv && ok; ++j, ++j_glob) {
          // K_j into K slot j_glob mod K_SLOTS, V_j into V slot j_glob mod V_SLOTS, each
          // once the slot's previous tile has been released
          const uint32_t ks = j_glob % LY::K_SLOTS, kpar = (j_glob / LY::K_SLOTS) & 1u;
          if (j_glob >= (uint32_t)LY::K_SLOTS) {
            const uint32_t u = j_glob - LY::K_SLOTS;
            ok = wait_bar(smem_u32(&bars->release[u % LY::K_SLOTS]), (u / LY::K_SLOTS) & 1u, abort_flag, lim);
            if (!ok) break;
          }
          const uint32_t fk = smem_u32(&bars->full[ks]);
          mbar_arrive_expect_tx(fk, LY::TILE_BYTES);
#pragma unroll
          for (int c = 0; c < LY::CHUNKS; ++c)
            tma_load_3d_hint(sK + ks * LY::TILE_BYTES + c * LY::CHUNK_BYTES, &tmK, fk, c * 64, j * BN, bh,
                             pol_reuse);
          issued |= 1u << ks;
          last_par = (last_par & ~(1u << ks)) | (kpar << ks);
          const uint32_t vs = j_glob % LY::V_SLOTS, vpar = (j_glob / LY::V_SLOTS) & 1u;
          if (j_glob >= (uint32_t)LY::V_SLOTS) {
            const uint32_t u = j_glob - LY::V_SLOTS;
            ok = wait_bar(smem_u32(&bars->vrelease[u % LY::V_SLOTS]), (u / LY::V_SLOTS) & 1u, abort_flag, lim);
            if (!ok) break;
          }
          const uint32_t fv = smem_u32(&bars->vfull[vs]);
          mbar_arrive_expect_tx(fv, LY::TILE_BYTES);
#pragma unroll
          for (int c = 0; c < LY::CHUNKS; ++c)
            tma_load_3d_hint(sV + vs * LY::TILE_BYTES + c * LY::CHUNK_BYTES, &tmV, fv, c * 64, j * BN, bh,
                             pol_reuse);
          vissued |= 1u << vs;
          vlast_par = (vlast_par & ~(1u << vs)) | (vpar << vs);
        }
      }
      if (!ok) {
        for (int s = 0; s < LY::K_SLOTS; ++s)
          if (issued & (1u << s)) wait_drain(smem_u32(&bars->full[s]), (last_par >> s) & 1u, lim);
        for (int s = 0; s < LY::V_SLOTS; ++s)
          if (vissued & (1u << s)) wait_drain(smem_u32(&bars->vfull[s]), (vlast_par >> s) & 1u, lim);
        if (a_issued) wait_drain(smem_u32(&bars->a_full), a_ph ^ 1, lim);
      }
    }
  } else if (warp == BW_WARP_MMA) {
    constexpr uint32_t ID_S = umma_idesc_f16(BF16 ? 1 : 0, 0, 0, BM, BN);  // S, dP: K-major x K-major
    constexpr uint32_t ID_Q = umma_idesc_f16(BF16 ? 1 : 0, 0, 1, BM, D);   // dQ: A in TMEM, K MN-major
    const uint64_t dA = umma_smem_desc(sA, 16, 1024);
    const uint64_t dKd = umma_smem_desc(sK, 16, 1024);
    const uint64_t dVd = umma_smem_desc(sV, 16, 1024);
    const uint64_t dBmn = umma_smem_desc(sK, LY::CHUNK_BYTES, 1024);
    uint32_t j_glob = 0, a_ph = 0, p_ph = 0;
    bool ok = true;
    auto wait_all = [&](uint32_t bar, uint32_t par) {
      return __all_sync(0xffffffffu, wait_bar(bar, par, abort_flag, lim));
    };
    auto kv_wait = [&](uint32_t g) {
      return wait_all(smem_u32(&bars->full[g % LY::K_SLOTS]), (g / LY::K_SLOTS) & 1u) &&
             wait_all(smem_u32(&bars->vfull[g % LY::V_SLOTS]), (g / LY::V_SLOTS) & 1u);
    };
    // S = Q K^T into T_S, dP = dO V^T into T_DP (K = D per product) for K/V load g; V_g
    // has no reader after dP and leaves its slot then
    auto issue_scores = [&](uint32_t g) {
      if (elect_one()) {
        const uint64_t dk = dKd + (((g % LY::K_SLOTS) * LY::TILE_BYTES) >> 4);
        const uint64_t dv = dVd + (((g % LY::V_SLOTS) * LY::TILE_BYTES) >> 4);
        const uint64_t ddo = dA + (LY::TILE_BYTES >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * LY::CHUNK_BYTES + (ks & 3) * 32) >> 4;
          umma_ss(tmem + T_S, dA + off, dk + off, ID_S, ks > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * LY::CHUNK_BYTES + (ks & 3) * 32) >> 4;
          umma_ss(tmem + T_DP, ddo + off, dv + off, ID_S, ks > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&bars->s_full));
        umma_commit(smem_u32(&bars->vrelease[g % LY::V_SLOTS]));
      }
      __syncwarp();
    };
    auto n_kv_of = [&](int t) {
      int bh, q0, n;
      item_tiles(t, bh, q0, n);
      return n;
    };
    // The CTA's tiles in order (items, then key tiles), one tile of lookahead: the scores
    // of tile g+1 are issued once the elementwise warps hold tile g's in registers, and
    // dQ += dS_g K_g once they have written dS_g. g numbers the K/V slot loads.
    uint32_t f_ph = 0;
    int rr_ = 0, t = bw_item_of(0);
    if (t < p.n_items) {
      ok = wait_all(smem_u32(&bars->a_full), a_ph) && kv_wait(0);
      if (ok) {
        a_ph ^= 1;
        tc_fence_after();
        issue_scores(0);
        if (n_kv_of(t) == 1 && elect_one()) umma_commit(smem_u32(&bars->a_empty));
        __syncwarp();
      }
    }
    for (; t < p.n_items && ok; t = bw_item_of(++rr_)) {
      const int n_kv = n_kv_of(t);
      const int t_next = bw_item_of(rr_ + 1);
      for (int j = 0; j < n_kv; ++j, ++j_glob) {
        const uint32_t slot = j_glob % LY::K_SLOTS;
        const bool last_in_item = j + 1 == n_kv;
        ok = wait_all(smem_u32(&bars->sdp_free), f_ph);
        if (!ok) break;
        f_ph ^= 1;
        if (!last_in_item || t_next < p.n_items) {
          if (last_in_item) {  // the next item's Q, dO
            ok = wait_all(smem_u32(&bars->a_full), a_ph);
            if (!ok) break;
            a_ph ^= 1;
          }
          ok = kv_wait(j_glob + 1);
          if (!ok) break;
          tc_fence_after();
          issue_scores(j_glob + 1);
          // the scores of an item's last tile are the last reads of its Q, dO
          const int j_next = last_in_item ? 0 : j + 1;
          const int n_next = last_in_item ? n_kv_of(t_next) : n_kv;
          if (j_next + 1 == n_next && elect_one()) umma_commit(smem_u32(&bars->a_empty));
          __syncwarp();
        }
        ok = wait_all(smem_u32(&bars->p_full), p_ph);
        if (!ok) break;
        p_ph ^= 1;
        tc_fence_after();
        // dQ += dS K_j : M=128 queries, N=D, K=128 keys; dS from TMEM, K_j MN-major
        if (elect_one()) {
          const uint64_t dk = dBmn + ((slot * LY::TILE_BYTES) >> 4);
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks)
            umma_ts(tmem + T_DQ, tmem + T_DS + ks * 8, dk + ((ks * 16 * 128) >> 4), ID_Q,
                    (j > 0 || ks > 0) ? 1u : 0u);
          umma_commit(smem_u32(&bars->op_done));
          umma_commit(smem_u32(&bars->release[slot]));  // K_j: no further reader
          if (last_in_item) umma_commit(smem_u32(&bars->done));
        }
        __syncwarp();
      }
    }
    if (elect_one()) umma_commit(smem_u32(&bars->mma_drain));
    __syncwarp();
    wait_drain(smem_u32(&bars->mma_drain), 0, lim);
    __syncwarp();
  } else {
    // ------------------------------------------------------------------- elementwise
    const int wq = warp & 3;
    const int hf = warp >> 2;  // column half: keys [64 hf, 64 hf + 64) of every key tile
    const int r = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + T_S + hf * 64, tDP = tmem + lane_off + T_DP + hf * 64;
    const uint32_t tDS = tmem + lane_off + T_DS + hf * 32;
    const uint32_t tQ = tmem + lane_off + T_DQ;
    uint32_t s_ph = 0, d_ph = 0, o_ph = 0;
    bool first_tile = true;
    bool ok = true;
    for (int rr_ = 0, t = bw_item_of(0); t < p.n_items && ok; t = bw_item_of(++rr_)) {
      int bh, q0, n_kv;
      item_tiles(t, bh, q0, n_kv);
      const int row = q0 + r;
      const bool valid = row < p.Nq;
      const size_t grow = (size_t)bh * p.Nq + (valid ? row : 0);
      // D = rowsum(dO o O) in fp32 from the 16-bit rows (both halves compute it; the
      // second read of the row hits L2); half 0 stores it for the dK/dV kernel
      float Drow = 0.f, L2 = INFINITY;
      if (valid) {
        const uint4* o4 = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.O) + grow * D * 2);
        const uint4* g4 = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.dO) + grow * D * 2);
        float acc2[2] = {0.f, 0.f};
#pragma unroll 4
        for (int v = 0; v < D / 8; ++v) {
          const uint4 a = o4[v], b = g4[v];
          const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float a0, a1, b0, b1;
            unpack2<BF16>(aw[e], a0, a1);
            unpack2<BF16>(bw[e], b0, b1);
            acc2[e & 1] = fmaf(a0, b0, fmaf(a1, b1, acc2[e & 1]));
          }
        }
        Drow = acc2[0] + acc2[1];
        if (hf == 0) p.Dws[grow] = Drow;
        L2 = p.L[grow] * 1.4426950408889634f;
      }
      const int kv_lim = CAUSAL ? min(row + 1, p.Nk) : p.Nk;
      for (int j = 0; j < n_kv; ++j) {
        // dropout ("Algorithm 4": dP = dP_dropped o Z): this row's keep bits for the half's
        // 64 keys, drawn before the scores are ready
        uint32_t kb[2] = {0, 0};
        if constexpr (DROP)
          dropout_row_bits<2>((uint32_t)(j * (BN / 16) + hf * 4), (uint32_t)row, (uint32_t)bh,
                              p.drop_offset, p.drop_keys, p.drop_bias, kb);
        ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->s_full), s_ph, abort_flag, lim));
        if (!ok) break;
        s_ph ^= 1;
        tc_fence_after();
        const int vis = kv_lim - j * BN;
        // this half's 64 keys: P = exp2(S c - L log2 e), dS = P (dP - D) -> 16-bit pairs
        // over the first 32 columns of the half
        uint32_t sr[2][32], dr[2][32];
        tmem_ld32(tS, sr[0]);
        tmem_ld32(tS + 32, sr[1]);
        tmem_ld32(tDP, dr[0]);
        tmem_ld32(tDP + 32, dr[1]);
        tmem_wait_ld();
        reg_fence(sr[0]); reg_fence(sr[1]); reg_fence(dr[0]); reg_fence(dr[1]);
        // S and dP are in registers: their columns may take the next tile's scores
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->sdp_free));
        // in phases over all 64 values (exponent arguments, exponentials, products), so
        // that the exponentials issue back to back instead of one dependent chain per pair
        const uint64_t c2 = f2(p.c, p.c), nl2 = f2(-L2, -L2), nd2 = f2(-Drow, -Drow);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          float t0, t1;
          f2_split(f2_fma(f2(__uint_as_float(sr[k >> 4][(2 * k) & 31]),
                             __uint_as_float(sr[k >> 4][(2 * k + 1) & 31])), c2, nl2), t0, t1);
          sr[k >> 4][(2 * k) & 31] = __float_as_uint(t0);
          sr[k >> 4][(2 * k + 1) & 31] = __float_as_uint(t1);
        }
        if (vis >= hf * 64 + 64) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            sr[e >> 5][e & 31] = __float_as_uint(ex2_approx(__uint_as_float(sr[e >> 5][e & 31])));
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            sr[e >> 5][e & 31] = __float_as_uint(
                hf * 64 + e < vis ? ex2_approx(__uint_as_float(sr[e >> 5][e & 31])) : 0.f);
        }
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const uint64_t g2 = f2(__uint_as_float(dr[k >> 4][(2 * k) & 31]),
                                 __uint_as_float(dr[k >> 4][(2 * k + 1) & 31]));
          uint64_t gd;  // dP - D, with dP = dP_dropped * Z under dropout
          if constexpr (DROP) {
            const float m0 = row_bit(kb, 2 * k) ? p.drop_rscale : 0.f;
            const float m1 = row_bit(kb, 2 * k + 1) ? p.drop_rscale : 0.f;
            gd = f2_fma(g2, f2(m0, m1), nd2);
          } else {
            gd = f2_add(g2, nd2);
          }
          float a0, a1;
          f2_split(f2_mul(f2(__uint_as_float(sr[k >> 4][(2 * k) & 31]),
                             __uint_as_float(sr[k >> 4][(2 * k + 1) & 31])), gd),
                   a0, a1);
          pk[k] = pack2<BF16>(a0, a1);
        }
        // the previous tile's dQ product reads the dS columns until it completes
        if (!first_tile) {
          ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->op_done), o_ph, abort_flag, lim));
          if (!ok) break;
          o_ph ^= 1;
          tc_fence_after();
        }
        first_tile = false;
        tmem_st32(tDS, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->p_full));
      }
      if (!ok) break;
      // dQ = scale * (dS K) -> 16-bit; this half stores columns [D/2 hf, D/2 (hf + 1))
      ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->done), d_ph, abort_flag, lim));
      if (!ok) break;
      d_ph ^= 1;
      tc_fence_after();
#pragma unroll
      for (int qq = 0; qq < D / 64; ++qq) {
        const int q = hf * (D / 64) + qq;
        uint32_t o[32];
        tmem_ld32(tQ + q * 32, o);
        tmem_wait_ld();
        reg_fence(o);
        uint32_t w16[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          w16[k] = pack2<BF16>(__uint_as_float(o[2 * k]) * p.scale, __uint_as_float(o[2 * k + 1]) * p.scale);
        if (valid) store_row16(p.dQ, grow, D, q, w16);
      }
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == BW_WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, T_COLS);
  }
}

// ============================================================================ dK, dV kernel
// CTA item: (bh, key tile kt). Streams Q_i, dO_i; per query tile:
//   S^T = K Q_i^T, dP^T = V dO_i^T  (TMEM)  ->  P^T, dS^T (16-bit, over S^T)
//   ->  dV += P^T dO_i,  dK += dS^T Q_i
// TMEM: two 128-column score regions that swap roles every query tile, then dK and dV.
template <int D, bool BF16, bool CAUSAL, bool DROP>
__global__ void __launch_bounds__(BW_THREADS, 1)
    fa_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                      const BwdParams p) {
  using LY = BwdLayout<D>;
  // score regions [0, 128) and [128, 256): query tile g (counted over the CTA's items)
  // takes S^T in region g & 1 and dP^T in the other one
  constexpr uint32_t T_DK = 256, T_DV = 256 + D, T_COLS = 512;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + LY::OFF_BAR);
  const uint32_t sA = smem_u32(smem + LY::OFF_A);   // K tile, then V tile
  const uint32_t sS = smem_u32(smem + LY::OFF_S);   // Q_i, dO_i pairs
  float* sLD = reinterpret_cast<float*>(smem + LY::OFF_LD);  // [0,128): L log2e, [128,256): D
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->a_full), 1);
    mbar_init(smem_u32(&bars->a_empty), 1);
    for (int s = 0; s < LY::SLOTS; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->release[s]), 1);
    }
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->op_done), 1);
    mbar_init(smem_u32(&bars->pt_full), BW_EW_WARPS);
    mbar_init(smem_u32(&bars->dp_full), 1);
    mbar_init(smem_u32(&bars->dp_read), BW_EW_WARPS);
    mbar_init(smem_u32(&bars->p_full), BW_EW_WARPS);  // one arrival per elementwise warp
    mbar_init(smem_u32(&bars->done), 1);
    mbar_init(smem_u32(&bars->mma_drain), 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == BW_WARP_MMA) {
    tmem_alloc(smem_u32(&bars->tmem_base), T_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const unsigned long long lim = p.wait_limit_ns;

  // query tiles [i0, n_qt) meet key tile kt (causal: only tiles with a query >= the tile's first key)
  // causal: heaviest (first) key tiles first; full: head by head (Q/dO reuse in L2)
  auto item_tiles = [&](int t, int& bh, int& k0, int& i0, int& n_q) {
    if (CAUSAL) {
      bh = t % p.BH;
      k0 = (t / p.BH) * BN;
    } else {
      bh = t / p.n_kt;
      k0 = (t % p.n_kt) * BN;
    }
    i0 = CAUSAL ? k0 / BM : 0;
    n_q = p.n_qt - i0;
  };

  if (warp == BW_WARP_LOAD) {
    if (lane == 0) {
      // streamed tiles are read by every CTA working on the same head: keep them in L2;
      // the CTA's resident tiles are read once
      const uint64_t pol_reuse = l2_policy_evict_last();
      const uint64_t pol_once = l2_policy_evict_first();
      uint32_t i_glob = 0, a_ph = 0;
      bool ok = true;
      uint32_t issued = 0, last_par = 0;
      bool a_issued = false;
      for (int rr_ = 0, t = bw_item_of(0); t < p.n_items && ok; t = bw_item_of(++rr_)) {
        int bh, k0, i0, n_q;
        item_tiles(t, bh, k0, i0, n_q);
        ok = wait_bar(smem_u32(&bars->a_empty), a_ph ^ 1, abort_flag, lim);
        if (!ok) break;
        a_ph ^= 1;
        const uint32_t af = smem_u32(&bars->a_full);
        mbar_arrive_expect_tx(af, 2 * LY::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < LY::CHUNKS; ++c) {
          tma_load_3d_hint(sA + c * LY::CHUNK_BYTES, &tmK, af, c * 64, k0, bh, pol_once);
          tma_load_3d_hint(sA + LY::TILE_BYTES + c * LY::CHUNK_BYTES, &tmV, af, c * 64, k0, bh, pol_once);
        }
        a_issued = true;
        for (int i = 0; i < n_q && ok; ++i, ++i_glob) {
          const uint32_t slot = i_glob % LY::SLOTS, par = (i_glob / LY::SLOTS) & 1u;
          if (i_glob >= (uint32_t)LY::SLOTS) {
            const uint32_t u = i_glob - LY::SLOTS;
            ok = wait_bar(smem_u32(&bars->release[u % LY::SLOTS]), (u / LY::SLOTS) & 1u, abort_flag, lim);
            if (!ok) break;
          }
          const uint32_t f = smem_u32(&bars->full[slot]);
          mbar_arrive_expect_tx(f, 2 * LY::TILE_BYTES);
          const uint32_t dst = sS + slot * LY::PAIR_BYTES;
#pragma unroll
          for (int c = 0; c < LY::CHUNKS; ++c) {
            tma_load_3d_hint(dst + c * LY::CHUNK_BYTES, &tmQ, f, c * 64, (i0 + i) * BM, bh, pol_reuse);
            tma_load_3d_hint(dst + LY::TILE_BYTES + c * LY::CHUNK_BYTES, &tmdO, f, c * 64, (i0 + i) * BM, bh,
                             pol_reuse);
          }
          issued |= 1u << slot;
          last_par = (last_par & ~(1u << slot)) | (par << slot);
        }
      }
      if (!ok) {
        for (int s = 0; s < LY::SLOTS; ++s)
          if (issued & (1u << s)) wait_drain(smem_u32(&bars->full[s]), (last_par >> s) & 1u, lim);
        if (a_issued) wait_drain(smem_u32(&bars->a_full), a_ph ^ 1, lim);
      }
    }
  } else if (warp == BW_WARP_MMA) {
    constexpr uint32_t ID_S = umma_idesc_f16(BF16 ? 1 : 0, 0, 0, BN, BM);  // S^T, dP^T
    constexpr uint32_t ID_G = umma_idesc_f16(BF16 ? 1 : 0, 0, 1, BN, D);   // dV, dK: B MN-major
    const uint64_t dA = umma_smem_desc(sA, 16, 1024);
    const uint64_t dB = umma_smem_desc(sS, 16, 1024);
    const uint64_t dBmn = umma_smem_desc(sS, LY::CHUNK_BYTES, 1024);
    uint32_t i_glob = 0, a_ph = 0, p_ph = 0, pt_ph = 0, r_ph = 0;
    bool ok = true;
    auto wait_all = [&](uint32_t bar, uint32_t par) {
      return __all_sync(0xffffffffu, wait_bar(bar, par, abort_flag, lim));
    };
    // dP^T = V dO_i^T into score region `reg` (K = D per product)
    auto issue_dpt = [&](uint32_t slot, uint32_t reg) {
      if (elect_one()) {
        const uint64_t ddo = dB + ((slot * LY::PAIR_BYTES) >> 4) + (LY::TILE_BYTES >> 4);
        const uint64_t dv = dA + (LY::TILE_BYTES >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * LY::CHUNK_BYTES + (ks & 3) * 32) >> 4;
          umma_ss(tmem + reg, dv + off, ddo + off, ID_S, ks > 0 ? 1u : 0u);  // V dO^T
        }
        umma_commit(smem_u32(&bars->dp_full));
      }
      __syncwarp();
    };
    // S^T = K Q_i^T into score region `reg`
    auto issue_st = [&](uint32_t slot, uint32_t reg) {
      if (elect_one()) {
        const uint64_t dq = dB + ((slot * LY::PAIR_BYTES) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * LY::CHUNK_BYTES + (ks & 3) * 32) >> 4;
          umma_ss(tmem + reg, dA + off, dq + off, ID_S, ks > 0 ? 1u : 0u);   // K Q^T
        }
        umma_commit(smem_u32(&bars->s_full));
      }
      __syncwarp();
    };
    // Per query tile g: P^T and dS^T go back over S^T(g), so S^T(g+1) is computed into the
    // region of dP^T(g) as soon as the elementwise warps have read dP^T(g), which they do
    // after storing P^T(g): the next tile's scores are ready when they finish tile g. Then
    // dV(g) (P^T(g) stored), dK(g) (dS^T(g) stored), and dP^T(g+1) into S^T(g)'s region,
    // which dK(g) has read (tcgen05 ops of one thread run in issue order).
    // Under dropout the elementwise warps take S^T and dP^T together, in one pass that
    // keeps the keep bits live once (a pass split around the dP^T read spills and is
    // slower): the regions stay fixed (S^T in [0, 128), dP^T in [128, 256)), dP^T(g+1) is
    // issued once they have read tile g, and S^T(g+1) after dK(g).
    for (int rr_ = 0, t = bw_item_of(0); t < p.n_items && ok; t = bw_item_of(++rr_)) {
      int bh, k0, i0, n_q;
      item_tiles(t, bh, k0, i0, n_q);
      (void)bh; (void)k0;
      ok = wait_all(smem_u32(&bars->a_full), a_ph) &&
           wait_all(smem_u32(&bars->full[i_glob % LY::SLOTS]), (i_glob / LY::SLOTS) & 1u);
      if (!ok) break;
      a_ph ^= 1;
      tc_fence_after();
      if constexpr (DROP) {
        issue_dpt(i_glob % LY::SLOTS, 128u);
        issue_st(i_glob % LY::SLOTS, 0u);  // its commit also covers dP^T
      } else {
        issue_st(i_glob % LY::SLOTS, (i_glob & 1u) * 128u);
        issue_dpt(i_glob % LY::SLOTS, ((i_glob & 1u) ^ 1u) * 128u);
      }
      for (int i = 0; i < n_q; ++i) {
        const uint32_t g = i_glob + i;
        const uint32_t reg_s = DROP ? 0u : (g & 1u) * 128u, reg_dp = reg_s ^ 128u;
        const uint32_t slot = g % LY::SLOTS;
        const uint32_t nslot = (g + 1) % LY::SLOTS;
        const bool has_next = i + 1 < n_q;
        ok = wait_all(smem_u32(&bars->dp_read), r_ph);
        if (!ok) break;
        r_ph ^= 1;
        if (has_next) {
          ok = wait_all(smem_u32(&bars->full[nslot]), ((g + 1) / LY::SLOTS) & 1u);
          if (!ok) break;
          tc_fence_after();
          if constexpr (DROP)
            issue_dpt(nslot, reg_dp);
          else
            issue_st(nslot, reg_dp);
        }
        const uint64_t dq = dBmn + ((slot * LY::PAIR_BYTES) >> 4);
        ok = wait_all(smem_u32(&bars->pt_full), pt_ph);
        if (!ok) break;
        pt_ph ^= 1;
        tc_fence_after();
        if (elect_one()) {
          const uint64_t ddo = dq + (LY::TILE_BYTES >> 4);
#pragma unroll
          for (int ks = 0; ks < BM / 16; ++ks) {  // dV += P^T dO_i (K = 128 queries)
            umma_ts(tmem + T_DV, tmem + reg_s + ks * 8, ddo + ((ks * 16 * 128) >> 4), ID_G,
                    (i > 0 || ks > 0) ? 1u : 0u);
          }
        }
        __syncwarp();
        ok = wait_all(smem_u32(&bars->p_full), p_ph);
        if (!ok) break;
        p_ph ^= 1;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int ks = 0; ks < BM / 16; ++ks) {  // dK += dS^T Q_i
            umma_ts(tmem + T_DK, tmem + reg_s + 64 + ks * 8, dq + ((ks * 16 * 128) >> 4), ID_G,
                    (i > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(smem_u32(&bars->release[slot]));  // Q_i, dO_i: no further reader
          if (!has_next) {
            umma_commit(smem_u32(&bars->done));
            umma_commit(smem_u32(&bars->a_empty));
          }
        }
        __syncwarp();
        if (has_next) {
          if constexpr (DROP)
            issue_st(nslot, reg_s);
          else
            issue_dpt(nslot, reg_s);
        }
      }
      i_glob += n_q;
    }
    if (elect_one()) umma_commit(smem_u32(&bars->mma_drain));
    __syncwarp();
    wait_drain(smem_u32(&bars->mma_drain), 0, lim);
    __syncwarp();
  } else {
    // ------------------------------------------------------------------- elementwise
    const int wq = warp & 3;
    const int hf = warp >> 2;         // column half: queries [64 hf, 64 hf + 64) of each tile
    const int r = wq * 32 + lane;     // key row of the tile (TMEM lane)
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tK = tmem + lane_off + T_DK, tV = tmem + lane_off + T_DV;
    uint32_t s_ph = 0, dp_ph = 0, d_ph = 0;
    uint32_t gq = 0;  // query tiles processed by this CTA (selects the score regions)
    bool ok = true;
    for (int rr_ = 0, t = bw_item_of(0); t < p.n_items && ok; t = bw_item_of(++rr_)) {
      int bh, k0, i0, n_q;
      item_tiles(t, bh, k0, i0, n_q);
      const int key = k0 + r;
      for (int i = 0; i < n_q; ++i, ++gq) {
        const int q0 = (i0 + i) * BM;
        // this half's scores: S^T columns [64 hf, 64 hf + 64) of region gq & 1, dP^T the same
        // columns of the other region; the 16-bit P^T goes to columns [32 hf, 32 hf + 32) of
        // S^T's region and dS^T 64 columns further
        const uint32_t reg_s = DROP ? 0u : (gq & 1u) * 128u, reg_dp = reg_s ^ 128u;
        const uint32_t tS = tmem + lane_off + reg_s + hf * 64, tDP = tmem + lane_off + reg_dp + hf * 64;
        const uint32_t tPT = tmem + lane_off + reg_s + hf * 32;
        // dropout: bit (c & 31) of zb[c >> 5] is the keep bit of query
        // q0 + 64 hf + c (c < 64) for this thread's key. Each lane of a 16-key group draws the
        // call of one query row for its group; a shuffle hands the group's 16-bit mask on.
        uint32_t zb[2] = {0, 0};
        if constexpr (DROP) {
          const uint32_t grp = (uint32_t)((k0 + wq * 32) >> 4) + (uint32_t)(lane >> 4);
#pragma unroll
          for (int blk = 0; blk < 4; ++blk) {
            const uint32_t qrow = (uint32_t)(q0 + hf * 64 + blk * 16 + (lane & 15));
            const uint32_t m16 = keep16(dropout_words(grp, qrow, (uint32_t)bh, p.drop_offset,
                                                      p.drop_keys), p.drop_bias);
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) {
              const uint32_t v = __shfl_sync(0xffffffffu, m16, (lane & 16) | ii);
              const int c = blk * 16 + ii;
              zb[c >> 5] |= ((v >> (lane & 15)) & 1u) << (c & 31);
            }
          }
        }
        // this query tile's L log2(e) (staged by half 0) and D (by half 1), one value per
        // thread (rows past Nq: L = +inf so that P = 0); the previous tile's readers
        // finished at the barrier that ended its iteration
        {
          const int qrow = q0 + r;
          const bool qv = qrow < p.Nq;
          const size_t g = (size_t)bh * p.Nq + (qv ? qrow : 0);
          if (hf == 0)
            sLD[r] = qv ? p.L[g] * 1.4426950408889634f : INFINITY;
          else
            sLD[128 + r] = qv ? p.Dws[g] : 0.f;
        }
        // one barrier both publishes sLD and makes the wait's outcome the same in all
        // elementwise warps (so that a timeout ends the loop everywhere, never at a barrier)
        ok = named_bar_red_and(2, BW_EW_WARPS * 32,
                               wait_bar(smem_u32(&bars->s_full), s_ph, abort_flag, lim));
        if (!ok) break;
        s_ph ^= 1;
        tc_fence_after();
        // causal: query q sees this key iff q >= key; first visible query of the tile:
        const int qfirst = CAUSAL ? key - q0 : 0;
        uint32_t sr[2][32], dr[2][32];
        tmem_ld32(tS, sr[0]);
        tmem_ld32(tS + 32, sr[1]);
        if constexpr (DROP) {  // dP^T is ready with S^T (see the MMA warp)
          tmem_ld32(tDP, dr[0]);
          tmem_ld32(tDP + 32, dr[1]);
        }
        tmem_wait_ld();
        reg_fence(sr[0]); reg_fence(sr[1]);
        if constexpr (DROP) {
          reg_fence(dr[0]); reg_fence(dr[1]);
        }
        // both halves hold their scores in registers: S^T's columns may now take P^T, dS^T
        tc_fence_before();
        named_bar_sync(3, BW_EW_WARPS * 32);
        if constexpr (DROP) {
          if (lane == 0) mbar_arrive(smem_u32(&bars->dp_read));
        }
        // in phases over all 64 values (exponent arguments, exponentials, products), so
        // that the exponentials issue back to back instead of one dependent chain per pair
        const uint64_t c2 = f2(p.c, p.c);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float2 l2 = *reinterpret_cast<const float2*>(sLD + hf * 64 + 2 * k);
          float t0, t1;
          f2_split(f2_fma(f2(__uint_as_float(sr[k >> 4][(2 * k) & 31]),
                             __uint_as_float(sr[k >> 4][(2 * k + 1) & 31])), c2, f2(-l2.x, -l2.y)),
                   t0, t1);
          sr[k >> 4][(2 * k) & 31] = __float_as_uint(t0);
          sr[k >> 4][(2 * k + 1) & 31] = __float_as_uint(t1);
        }
        if (qfirst <= hf * 64) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            sr[e >> 5][e & 31] = __float_as_uint(ex2_approx(__uint_as_float(sr[e >> 5][e & 31])));
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            sr[e >> 5][e & 31] = __float_as_uint(
                hf * 64 + e >= qfirst ? ex2_approx(__uint_as_float(sr[e >> 5][e & 31])) : 0.f);
        }
        if constexpr (!DROP) {
          // P^T first
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pp[16];
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              pp[kk] = pack2<BF16>(__uint_as_float(sr[c][2 * kk]), __uint_as_float(sr[c][2 * kk + 1]));
            tmem_st16(tPT + c * 16, pp);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->pt_full));
          // then dP^T: the same outcome in every elementwise warp (a timeout ends the loop
          // everywhere, never at a barrier); once read, its region may take S^T(g+1)
          ok = named_bar_red_and(4, BW_EW_WARPS * 32,
                                 wait_bar(smem_u32(&bars->dp_full), dp_ph, abort_flag, lim));
          if (!ok) break;
          dp_ph ^= 1;
          tc_fence_after();
          tmem_ld32(tDP, dr[0]);
          tmem_ld32(tDP + 32, dr[1]);
          tmem_wait_ld();
          reg_fence(dr[0]); reg_fence(dr[1]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->dp_read));
          // dS^T = P^T o (dP^T - D)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pd[16];
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
              const float2 dd = *reinterpret_cast<const float2*>(sLD + 128 + hf * 64 + c * 32 + 2 * kk);
              const uint64_t p2 = f2(__uint_as_float(sr[c][2 * kk]), __uint_as_float(sr[c][2 * kk + 1]));
              const uint64_t g2 = f2(__uint_as_float(dr[c][2 * kk]), __uint_as_float(dr[c][2 * kk + 1]));
              float a0, a1;
              f2_split(f2_mul(p2, f2_add(g2, f2(-dd.x, -dd.y))), a0, a1);
              pd[kk] = pack2<BF16>(a0, a1);
            }
            tmem_st16(tPT + 64 + c * 16, pd);
          }
        } else {
          // one pass builds both operands: P^T o Z and dS^T = P^T o (dP^T o Z - D) (Z's
          // 1/(1-p) is applied to dV at the end)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pp[16], pd[16];
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
              const float2 dd = *reinterpret_cast<const float2*>(sLD + 128 + hf * 64 + c * 32 + 2 * kk);
              const float p0 = __uint_as_float(sr[c][2 * kk]), p1 = __uint_as_float(sr[c][2 * kk + 1]);
              const uint64_t g2 = f2(__uint_as_float(dr[c][2 * kk]), __uint_as_float(dr[c][2 * kk + 1]));
              const uint32_t z0 = (zb[c] >> (2 * kk)) & 1u, z1 = (zb[c] >> (2 * kk + 1)) & 1u;
              float a0, a1;
              f2_split(f2_mul(f2(p0, p1), f2_fma(g2, f2(z0 ? p.drop_rscale : 0.f, z1 ? p.drop_rscale : 0.f),
                                                 f2(-dd.x, -dd.y))),
                       a0, a1);
              pp[kk] = pack2<BF16>(z0 ? p0 : 0.f, z1 ? p1 : 0.f);
              pd[kk] = pack2<BF16>(a0, a1);
            }
            tmem_st16(tPT + c * 16, pp);
            tmem_st16(tPT + 64 + c * 16, pd);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if constexpr (DROP) {
          if (lane == 0) mbar_arrive(smem_u32(&bars->pt_full));
        }
        if (lane == 0) mbar_arrive(smem_u32(&bars->p_full));
        named_bar_sync(2, BW_EW_WARPS * 32);  // every thread is done reading sLD
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->done), d_ph, abort_flag, lim));
      if (!ok) break;
      d_ph ^= 1;
      tc_fence_after();
      const bool valid = key < p.Nk;
      const size_t grow = (size_t)bh * p.Nk + (valid ? key : 0);
      // this half stores columns [D/2 hf, D/2 (hf + 1)) of dK and dV
#pragma unroll
      for (int qq = 0; qq < D / 64; ++qq) {
        const int q = hf * (D / 64) + qq;
        uint32_t o[32];
        uint32_t w16[16];
        tmem_ld32(tK + q * 32, o);
        tmem_wait_ld();
        reg_fence(o);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          w16[k] = pack2<BF16>(__uint_as_float(o[2 * k]) * p.scale, __uint_as_float(o[2 * k + 1]) * p.scale);
        if (valid) store_row16(p.dK, grow, D, q, w16);
        tmem_ld32(tV + q * 32, o);
        tmem_wait_ld();
        reg_fence(o);
        const float vs = DROP ? p.drop_rscale : 1.f;
#pragma unroll
        for (int k = 0; k < 16; ++k)
          w16[k] = pack2<BF16>(__uint_as_float(o[2 * k]) * vs, __uint_as_float(o[2 * k + 1]) * vs);
        if (valid) store_row16(p.dV, grow, D, q, w16);
      }
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == BW_WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, T_COLS);
  }
}

}  // namespace fa
