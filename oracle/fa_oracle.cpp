// fa_oracle.cpp -- plain float64 CPU oracle for the exact attention forward pass.
//
// TEST INFRASTRUCTURE ONLY. This file is the definition the CUDA path is checked
// against; it is built by the test harness and is called only by the tests, by
// the smoke check and by the benchmark's CPU-baseline leg. No product code path
// links, loads or calls it, and it shares no code, header or constant with the
// CUDA library.
//
// Everything is computed in IEEE double from inputs that the caller has already
// widened (exactly) from fp16/bf16. Nothing is blocked, fused or reordered
// beyond what each cited definition states.
//
// Sources (web pages, cited by title and section):
//   [CS336] CS336 lecture 5 code "05_flash_attention.py":
//           part 1 "在线 softmax" (online_softmax_stats) and
//           part 2 "FlashAttention 前向" (standard_attention, flash_attention_forward).
//   [CA]    "Flash Attention" (blog.cyberangel.work): sections "Online Softmax"
//           (safe softmax, 3 passes) and "平行化" (the (m, d) and (m, d, o~) merge).
//   [HW]    "手写 Flash Attention：从算法原理到高性能实现": section 2.2 "Online Softmax"
//           (the worked row [2,1,5,3] with block 2).
//   [CS336-3] the same CS336 page, part 3 "FlashAttention 反向" (the gradient formulas
//           dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = dS K tau, dK = dS^T Q tau).
//   [CA-2]  the "Flash Attention" page, "Algorithm 2" (mask and dropout: P_dropped =
//           dropout(P, p), O = P_dropped V; the forward also returns the generator
//           state R) and "Algorithm 4" (the backward regenerates the mask Z from R:
//           dV += (P o Z)^T dO, dP = dP_dropped o Z).
//   [PHILOX] J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel Random
//           Numbers: As Easy as 1, 2, 3" (SC'11), section 3.3: the Philox-4x32 bijection
//           with 10 rounds. The pages name no generator; this published counter-based
//           one is implemented here and, separately, in the CUDA library.
//
// Pins (what fixes each function other than itself) live in tests/test_oracle_pins.py.
// Every exported function is pinned; none is "parity unpinned".

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

const double NEG_INF = -std::numeric_limits<double>::infinity();

// One output row of attention by the plain definition ([CS336] part 2,
// standard_attention; [CA] "Why Flash Attention"):
//   s_j = scale * <q, k_j>            for every key j (the whole row is materialised)
//   s_j = -inf  if causal and j > i   (query i sees key j iff j <= i; top-left aligned,
//                                      the triu(1) mask of standard_attention)
//   p   = safe softmax of s           ([CA] "Safe softmax (3 遍掃描)": max, sum, divide)
//   o   = sum_j p_j v_j
//   L   = m + ln(sum_j exp(s_j - m))  (logsumexp, [CS336] part 2 "L_i = m_i + log(l_i)")
void attention_row(const double* q, const double* K, const double* V,
                   int Nk, int d, double scale, bool causal, int64_t i,
                   double* s /* scratch [Nk] */, double* o /* [d] */, double* L) {
    // scores
    for (int j = 0; j < Nk; ++j) {
        if (causal && (int64_t)j > i) { s[j] = NEG_INF; continue; }
        const double* k = K + (int64_t)j * d;
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += q[c] * k[c];
        s[j] = scale * acc;
    }
    // pass 1: row max
    double m = NEG_INF;
    for (int j = 0; j < Nk; ++j) m = std::max(m, s[j]);
    // pass 2: denominator
    double den = 0.0;
    for (int j = 0; j < Nk; ++j) den += std::exp(s[j] - m);
    // pass 3: normalised probabilities, written over the scores (P row materialised)
    for (int j = 0; j < Nk; ++j) s[j] = std::exp(s[j] - m) / den;
    *L = m + std::log(den);
    if (V == nullptr) return;  // the caller wants the probabilities only
    // o = P V
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int j = 0; j < Nk; ++j) {
        const double p = s[j];
        if (p == 0.0) continue;
        const double* v = V + (int64_t)j * d;
        for (int c = 0; c < d; ++c) o[c] += p * v[c];
    }
}

// Philox-4x32-10 ([PHILOX] section 3.3). One round maps the counter (c0, c1, c2, c3)
// under the round key (k0, k1) to
//   (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))
// with the 32x32->64-bit products split into high and low words and the multipliers
// M0 = 0xD2511F53, M1 = 0xCD9E8D57. The key is bumped by the Weyl constants
// (0x9E3779B9, 0xBB67AE85) between rounds.
void philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        const uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// The dropout mask Z of [CA-2]. The pages fix dropout(P, p) (each probability kept with
// probability 1 - p and then divided by 1 - p, so that E[P_dropped] = P) but name no
// generator or counter layout; this is the library's definition of both:
//   threshold t = floor(p * 256 + 0.5), an 8-bit integer (p is used to 1/256);
//   for element (bh, i, j) = (b*H + h, query row, key):
//     words = Philox-4x32-10(counter = (j >> 4, i, bh, offset),
//                            key = (seed mod 2^32, seed div 2^32))
//     w = words[(j >> 2) & 3]; the four keys 4m .. 4m+3 of w take, in order, byte 0,
//     byte 2, byte 1 and byte 3 of w (the low bytes of its two 16-bit halves serve the
//     first key pair, the high bytes the second): x = byte ((j & 1) * 2 + ((j >> 1) & 1))
//     keep = (x >= t);  Z_ij = keep ? 256 / (256 - t) : 0
// so one call of the generator serves sixteen consecutive keys of one query row, and the
// kept fraction is exactly (256 - t) / 256 in expectation.
struct Dropout {
    uint32_t t;
    uint32_t key[2];
    uint32_t offset;
    double z_keep;  // 256 / (256 - t)
};

bool dropout_threshold(double p, uint32_t* t) {
    if (!(p >= 0.0) || !std::isfinite(p)) return false;
    const double tt = std::floor(p * 256.0 + 0.5);
    if (tt >= 256.0) return false;
    *t = (uint32_t)tt;
    return true;
}

Dropout make_dropout(uint32_t t, uint64_t seed, uint32_t offset) {
    Dropout dr;
    dr.t = t;
    dr.key[0] = (uint32_t)(seed & 0xFFFFFFFFu);
    dr.key[1] = (uint32_t)(seed >> 32);
    dr.offset = offset;
    dr.z_keep = 256.0 / (256.0 - (double)t);
    return dr;
}

bool dropout_keep(const Dropout& dr, int64_t bh, int64_t i, int64_t j) {
    const uint32_t ctr[4] = {(uint32_t)(j >> 4), (uint32_t)i, (uint32_t)bh, dr.offset};
    uint32_t w[4];
    philox4x32_10(ctr, dr.key, w);
    const uint32_t word = w[(j >> 2) & 3];
    const int byte = (int)((j & 1) * 2 + ((j >> 1) & 1));
    const uint32_t x = (word >> (8 * byte)) & 0xFFu;
    return x >= dr.t;
}

template <class F>
void parallel_for(int64_t n, int nthreads, F&& f) {
    if (nthreads <= 0) nthreads = (int)std::max(1u, std::thread::hardware_concurrency());
    if (nthreads > n) nthreads = (int)std::max<int64_t>(1, n);
    if (nthreads == 1) { f(0, n); return; }
    std::vector<std::thread> th;
    th.reserve(nthreads);
    // interleaved chunks so that causal rows (whose cost grows with i) balance
    const int64_t chunk = 16;
    for (int t = 0; t < nthreads; ++t) {
        th.emplace_back([&, t]() {
            for (int64_t c0 = (int64_t)t * chunk; c0 < n; c0 += (int64_t)nthreads * chunk)
                f(c0, std::min(n, c0 + chunk));
        });
    }
    for (auto& x : th) x.join();
}

// One output row of attention with dropout ([CA-2]): P_i by the plain definition
// (attention_row), then o = sum_j P_ij Z_ij v_j with Z from the mask definition above.
// L is the logsumexp of the undropped scores, as without dropout (Algorithm 2 returns
// the statistics of the softmax, which dropout does not change).
void dropout_attention_row(const double* q, const double* K, const double* V, int Nk, int d,
                           double scale, bool causal, int64_t bh, int64_t i,
                           const Dropout& dr, double* s, double* o, double* L) {
    attention_row(q, K, nullptr, Nk, d, scale, causal, i, s, o, L);
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int j = 0; j < Nk; ++j) {
        const double p = s[j];
        if (p == 0.0 || !dropout_keep(dr, bh, i, j)) continue;
        const double pz = p * dr.z_keep;
        const double* v = V + (int64_t)j * d;
        for (int c = 0; c < d; ++c) o[c] += pz * v[c];
    }
}

}  // namespace

extern "C" {

// Number of threads the oracle uses when asked for 0 (all host cores).
int fa_oracle_hw_threads(void) {
    return (int)std::max(1u, std::thread::hardware_concurrency());
}

// Full attention forward by the plain definition (see attention_row).
// Q, O: [B,H,Nq,d]; K, V: [B,H,Nk,d]; L: [B,H,Nq]; all float64, row-major, dense.
// nthreads <= 0 uses every host core. Returns the number of threads used.
int fa_oracle_attention(const double* Q, const double* K, const double* V,
                        int B, int H, int Nq, int Nk, int d, double scale, int causal,
                        double* O, double* L, int nthreads) {
    const int64_t rows = (int64_t)B * H * Nq;
    if (nthreads <= 0) nthreads = fa_oracle_hw_threads();
    parallel_for(rows, nthreads, [&](int64_t r0, int64_t r1) {
        std::vector<double> s((size_t)std::max(Nk, 1));
        for (int64_t r = r0; r < r1; ++r) {
            const int64_t bh = r / Nq, i = r % Nq;
            attention_row(Q + r * d, K + bh * (int64_t)Nk * d, V + bh * (int64_t)Nk * d,
                          Nk, d, scale, causal != 0, i, s.data(), O + r * d, L + r);
        }
    });
    return nthreads;
}

// The same definition evaluated only on selected rows. rows[t] is a flat row index
// b*H*Nq + h*Nq + i; O_rows is [nrows, d], L_rows is [nrows]. Q is [B,H,Nq,d],
// K and V are [B,H,Nk,d] (the full tensors).
int fa_oracle_attention_rows(const double* Q, const double* K, const double* V,
                             int B, int H, int Nq, int Nk, int d, double scale, int causal,
                             const int64_t* rows, int64_t nrows,
                             double* O_rows, double* L_rows, int nthreads) {
    (void)B; (void)H;
    if (nthreads <= 0) nthreads = fa_oracle_hw_threads();
    parallel_for(nrows, nthreads, [&](int64_t t0, int64_t t1) {
        std::vector<double> s((size_t)std::max(Nk, 1));
        for (int64_t t = t0; t < t1; ++t) {
            const int64_t r = rows[t];
            const int64_t bh = r / Nq, i = r % Nq;
            attention_row(Q + r * d, K + bh * (int64_t)Nk * d, V + bh * (int64_t)Nk * d,
                          Nk, d, scale, causal != 0, i, s.data(), O_rows + t * d, L_rows + t);
        }
    });
    return nthreads;
}

// The probability matrix P of one head by the same definition: P is [Nq, Nk].
// Q is [Nq,d], K is [Nk,d]. Used by the invariant pins (rows sum to one).
void fa_oracle_probs(const double* Q, const double* K, int Nq, int Nk, int d,
                     double scale, int causal, double* P) {
    std::vector<double> o((size_t)d), vdummy((size_t)Nk * d, 0.0);
    for (int64_t i = 0; i < Nq; ++i) {
        double Lr;
        // attention_row leaves the normalised probabilities in its scratch row.
        attention_row(Q + i * d, K, vdummy.data(), Nk, d, scale, causal != 0, i,
                      P + i * (int64_t)Nk, o.data(), &Lr);
    }
}

// Online softmax statistics ([CS336] part 1, online_softmax_stats; [CA] "Online
// softmax (2 遍掃描)"): read x in chunks of `block`; keep m = running max and
// l = sum exp(x - m); when a chunk raises the max to m_new, re-base the old sum:
//   m_new = max(m, max(chunk));  l = l * exp(m - m_new) + sum_chunk exp(x - m_new).
// The state after every chunk is written to m_trace[c], l_trace[c] when those are
// non-null (the worked example on the [HW] page prints these intermediates).
// Returns the number of chunks.
int fa_oracle_online_softmax(const double* x, int n, int block,
                             double* m_out, double* l_out,
                             double* m_trace, double* l_trace) {
    double m = NEG_INF, l = 0.0;
    int c = 0;
    for (int s = 0; s < n; s += block, ++c) {
        const int e = std::min(n, s + block);
        double cmax = NEG_INF;
        for (int t = s; t < e; ++t) cmax = std::max(cmax, x[t]);
        const double m_new = std::max(m, cmax);
        double add = 0.0;
        for (int t = s; t < e; ++t) add += std::exp(x[t] - m_new);
        // exp(m - m_new) with m = -inf and a finite m_new is exp(-inf) = 0.
        l = l * std::exp(m - m_new) + add;
        m = m_new;
        if (m_trace) m_trace[c] = m;
        if (l_trace) l_trace[c] = l;
    }
    *m_out = m;
    *l_out = l;
    return c;
}

// The merge operator on partial states ([CA] "平行化"): for states (m_a, d_a, o_a) and
// (m_b, d_b, o_b) with o of length dv (dv may be 0 for the (m, d) pair),
//   m = max(m_a, m_b)
//   d = d_a e^{m_a - m} + d_b e^{m_b - m}
//   o = o_a e^{m_a - m} + o_b e^{m_b - m}
// An empty state (m = -inf, d = 0, o = 0) is the identity: its weight e^{-inf - m} is 0.
void fa_oracle_merge(double m_a, double d_a, const double* o_a,
                     double m_b, double d_b, const double* o_b, int dv,
                     double* m_out, double* d_out, double* o_out) {
    const double m = std::max(m_a, m_b);
    const double wa = (m_a == NEG_INF) ? 0.0 : std::exp(m_a - m);
    const double wb = (m_b == NEG_INF) ? 0.0 : std::exp(m_b - m);
    *m_out = m;
    *d_out = d_a * wa + d_b * wb;
    for (int c = 0; c < dv; ++c) o_out[c] = o_a[c] * wa + o_b[c] * wb;
}

// The state (m, d, o~) of one key block for one query row ([CA] "平行化": the
// per-element state (x_k, 1, v_k) merged over the block): s_j = scale*<q,k_j>
// (masked to -inf when causal and j > i), m = max_j s_j, d = sum_j e^{s_j - m},
// o~ = sum_j e^{s_j - m} v_j. Keys j in [j0, j1). A block with every key masked
// returns the identity state (-inf, 0, 0).
void fa_oracle_block_state(const double* q, const double* K, const double* V, int d,
                           int64_t i, int j0, int j1, double scale, int causal,
                           double* m_out, double* d_out, double* o_out) {
    std::vector<double> s((size_t)std::max(j1 - j0, 1));
    double m = NEG_INF;
    for (int j = j0; j < j1; ++j) {
        double v;
        if (causal && (int64_t)j > i) v = NEG_INF;
        else {
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += q[c] * K[(int64_t)j * d + c];
            v = scale * acc;
        }
        s[(size_t)(j - j0)] = v;
        m = std::max(m, v);
    }
    for (int c = 0; c < d; ++c) o_out[c] = 0.0;
    double den = 0.0;
    if (m != NEG_INF) {
        for (int j = j0; j < j1; ++j) {
            const double w = std::exp(s[(size_t)(j - j0)] - m);
            den += w;
            for (int c = 0; c < d; ++c) o_out[c] += w * V[(int64_t)j * d + c];
        }
    }
    *m_out = m;
    *d_out = den;
}

// Gradients of the attention forward with respect to Q, K and V for an upstream gradient
// dO ([CS336-3]; "Flash Attention" page, "Algorithm 4: backward pass" and its derivation),
// with the dropout mask Z of [CA-2] when `dr` is non-null (Z_ij = 1 otherwise).
// For each (b, h) the probability matrix is materialised one row at a time by the plain
// definition (attention_row: scores, mask, safe softmax), then, row i:
//   dP_ij = Z_ij <dO_i, V_j>                   (Algorithm 4: dP = dP_dropped o Z)
//   D_i   = sum_j P_ij dP_ij                    (the softmax Jacobian contracted with dP)
//   dS_ij = P_ij (dP_ij - D_i)
//   dQ_i  = scale * sum_j dS_ij K_j
//   dK_j += scale * dS_ij Q_i,   dV_j += P_ij Z_ij dO_i
// All arrays float64 and dense: Q, dO, dQ are [B,H,Nq,d]; K, V, dK, dV are [B,H,Nk,d].
// Parallel over (b, h). Returns the number of threads used.
static int attention_bwd(const double* Q, const double* K, const double* V, const double* dO,
                         int B, int H, int Nq, int Nk, int d, double scale, int causal,
                         const Dropout* dr, double* dQ, double* dK, double* dV, int nthreads) {
  const int64_t heads = (int64_t)B * H;
  if (nthreads <= 0) nthreads = fa_oracle_hw_threads();
  std::vector<std::thread> th;
  const int nt = (int)std::min<int64_t>(std::max(1, nthreads), std::max<int64_t>(1, heads));
  for (int t = 0; t < nt; ++t) {
    th.emplace_back([&, t]() {
      std::vector<double> prow((size_t)std::max(Nk, 1)), dprow((size_t)std::max(Nk, 1)),
          zrow((size_t)std::max(Nk, 1), 1.0), o((size_t)d);
      for (int64_t bh = t; bh < heads; bh += nt) {
        const double* q = Q + bh * (int64_t)Nq * d;
        const double* k = K + bh * (int64_t)Nk * d;
        const double* v = V + bh * (int64_t)Nk * d;
        const double* go = dO + bh * (int64_t)Nq * d;
        double* gq = dQ + bh * (int64_t)Nq * d;
        double* gk = dK + bh * (int64_t)Nk * d;
        double* gv = dV + bh * (int64_t)Nk * d;
        for (int64_t x = 0; x < (int64_t)Nk * d; ++x) { gk[x] = 0.0; gv[x] = 0.0; }
        for (int64_t i = 0; i < Nq; ++i) {
          double Lr;
          attention_row(q + i * d, k, v, Nk, d, scale, causal != 0, i, prow.data(), o.data(), &Lr);
          if (dr)
            for (int j = 0; j < Nk; ++j) zrow[(size_t)j] = dropout_keep(*dr, bh, i, j) ? dr->z_keep : 0.0;
          double Di = 0.0;
          for (int j = 0; j < Nk; ++j) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += go[i * d + c] * v[(int64_t)j * d + c];
            dprow[(size_t)j] = acc * zrow[(size_t)j];
            Di += prow[(size_t)j] * dprow[(size_t)j];
          }
          for (int c = 0; c < d; ++c) gq[i * d + c] = 0.0;
          for (int j = 0; j < Nk; ++j) {
            const double pij = prow[(size_t)j];
            if (pij == 0.0) continue;
            const double ds = pij * (dprow[(size_t)j] - Di);
            const double pz = pij * zrow[(size_t)j];
            for (int c = 0; c < d; ++c) {
              gq[i * d + c] += scale * ds * k[(int64_t)j * d + c];
              gk[(int64_t)j * d + c] += scale * ds * q[i * d + c];
              gv[(int64_t)j * d + c] += pz * go[i * d + c];
            }
          }
        }
      }
    });
  }
  for (auto& x : th) x.join();
  return nt;
}

// The backward pass without dropout (Z = 1 everywhere; see attention_bwd).
int fa_oracle_attention_bwd(const double* Q, const double* K, const double* V, const double* dO,
                            int B, int H, int Nq, int Nk, int d, double scale, int causal,
                            double* dQ, double* dK, double* dV, int nthreads) {
  return attention_bwd(Q, K, V, dO, B, H, Nq, Nk, d, scale, causal, nullptr, dQ, dK, dV, nthreads);
}

// The backward pass with the dropout mask of seed/offset and probability p_drop
// ([CA-2]; see attention_bwd). Returns -1 for a p_drop outside [0, 1 - 2^-9).
int fa_oracle_attention_bwd_dropout(const double* Q, const double* K, const double* V,
                                    const double* dO, int B, int H, int Nq, int Nk, int d,
                                    double scale, int causal, double p_drop, uint64_t seed,
                                    uint32_t offset, double* dQ, double* dK, double* dV,
                                    int nthreads) {
  uint32_t t;
  if (!dropout_threshold(p_drop, &t)) return -1;
  const Dropout dr = make_dropout(t, seed, offset);
  return attention_bwd(Q, K, V, dO, B, H, Nq, Nk, d, scale, causal, &dr, dQ, dK, dV, nthreads);
}

// Philox-4x32-10 of one counter under one key ([PHILOX]; see philox4x32_10).
void fa_oracle_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
  philox4x32_10(ctr, key, out);
}

// The 8-bit dropout threshold t of p_drop (see Dropout), or -1 when p_drop is negative,
// not finite, or so close to 1 that t would be 256.
int fa_oracle_dropout_threshold(double p_drop) {
  uint32_t t;
  return dropout_threshold(p_drop, &t) ? (int)t : -1;
}

// The keep mask of [CA-2] for every (b, h, i, j): keep is [B,H,Nq,Nk] bytes, 1 = kept.
// Returns 0, or -1 for an invalid p_drop.
int fa_oracle_dropout_keep(int B, int H, int Nq, int Nk, double p_drop, uint64_t seed,
                           uint32_t offset, uint8_t* keep) {
  uint32_t t;
  if (!dropout_threshold(p_drop, &t)) return -1;
  const Dropout dr = make_dropout(t, seed, offset);
  for (int64_t bh = 0; bh < (int64_t)B * H; ++bh)
    for (int64_t i = 0; i < Nq; ++i)
      for (int64_t j = 0; j < Nk; ++j)
        keep[(bh * Nq + i) * Nk + j] = dropout_keep(dr, bh, i, j) ? 1 : 0;
  return 0;
}

// Attention forward with dropout ([CA-2]) on selected rows: rows[t] is a flat row index
// b*H*Nq + h*Nq + i; O_rows is [nrows, d], L_rows [nrows]; Q [B,H,Nq,d], K and V
// [B,H,Nk,d]. Returns the number of threads used, or -1 for an invalid p_drop.
int fa_oracle_attention_dropout_rows(const double* Q, const double* K, const double* V,
                                     int B, int H, int Nq, int Nk, int d, double scale,
                                     int causal, double p_drop, uint64_t seed, uint32_t offset,
                                     const int64_t* rows, int64_t nrows,
                                     double* O_rows, double* L_rows, int nthreads) {
  (void)B; (void)H;
  uint32_t t;
  if (!dropout_threshold(p_drop, &t)) return -1;
  const Dropout dr = make_dropout(t, seed, offset);
  if (nthreads <= 0) nthreads = fa_oracle_hw_threads();
  parallel_for(nrows, nthreads, [&](int64_t t0, int64_t t1) {
    std::vector<double> s((size_t)std::max(Nk, 1));
    for (int64_t x = t0; x < t1; ++x) {
      const int64_t r = rows[x];
      const int64_t bh = r / Nq, i = r % Nq;
      dropout_attention_row(Q + r * d, K + bh * (int64_t)Nk * d, V + bh * (int64_t)Nk * d, Nk,
                            d, scale, causal != 0, bh, i, dr, s.data(), O_rows + x * d,
                            L_rows + x);
    }
  });
  return nthreads;
}

// Attention forward with dropout ([CA-2]) on every row; arrays as fa_oracle_attention.
int fa_oracle_attention_dropout(const double* Q, const double* K, const double* V,
                                int B, int H, int Nq, int Nk, int d, double scale, int causal,
                                double p_drop, uint64_t seed, uint32_t offset,
                                double* O, double* L, int nthreads) {
  const int64_t n = (int64_t)B * H * Nq;
  std::vector<int64_t> rows((size_t)n);
  for (int64_t r = 0; r < n; ++r) rows[(size_t)r] = r;
  return fa_oracle_attention_dropout_rows(Q, K, V, B, H, Nq, Nk, d, scale, causal, p_drop, seed,
                                          offset, rows.data(), n, O, L, nthreads);
}

}  // extern "C"
