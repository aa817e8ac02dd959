// SDM oracle: a plain, slow CPU statement of what the Sparse Delta Memory layer
// computes, forward and backward.  TEST INFRASTRUCTURE ONLY: the tests, the smoke
// check and the CPU baseline of the benchmark call it; the product library never
// links, loads or calls anything in this directory.
//
// Source: "Sparse Delta Memory (SDM)" technical summary, gist.science/it/paper/2607.07386,
// section "Meccanismo Core" (its Japanese twin, gist.science/ja/paper/2607.07386,
// "コアメカニズム", states the same formulas):
//   item 1  explicit memory table M_t in R^{N x d_v}
//   item 2  k', q' split in two halves; their outer sum scores the N slots; top-W
//           (write) and top-R (read) slots via topk(s1 (+) s2) = topk(topk(s1) (+) topk(s2))
//   item 3  forget gate  M~_t[i] = alpha_t * M_{t-1}[i]
//           delta update M_t[i]  = M~_t[i] + beta_t * k_t^(i) * (v_t - M~_t[i])
//           unselected slots are left unchanged
//   item 4  the output is a weighted sum of the R selected read slots
//
// Readings where the pages are silent (each one is listed in the design notes):
//   * the halves' entries are the sub-scores themselves; flat slot = i*S + j with
//     i indexing the first half (S = sqrt(N));
//   * inner top-k uses k = min(K, S); order is (value desc, index asc); the outer
//     top-K over the k x k grid is ordered by (fp32 sum desc, flat asc);
//   * the pair sums are formed in fp32 (the precision the selection is reported in);
//   * k_t^(i) = softmax over the W selected write scores, read weights = softmax
//     over the R selected read scores (temperature 1, max-subtracted);
//   * the read sees M_t, i.e. it comes after the write of the same token;
//   * alpha_t, beta_t are one scalar per (sequence, head, token).
// State and all scan arithmetic are fp64.
//
// Backward pass (oracle_scan_backward): reverse-mode derivative of the same scan for the
// loss L = sum_t <dO_t, o_t> + <dM_T, M_T>, with the selected slots held fixed (they are
// discrete).  It recomputes the forward, keeping every token's write rows before the update
// and read rows after it, then walks the tokens backwards with the adjoint G = dL/dM_t:
//   read   o_t = sum_j r_j M_t[ir_j]:   G[ir_j] += r_j dO_t,  dr_j = <dO_t, M_t[ir_j]>
//   write  M_t[i] = a M_{t-1}[i] + b k_i (v_t - a M_{t-1}[i]), with G after the read:
//          dv_t += b k_i G[i];  da_t += (1 - b k_i) <G[i], M_{t-1}[i]>;
//          db_t += k_i <G[i], v_t - a M_{t-1}[i]>;  dk_i = b <G[i], v_t - a M_{t-1}[i]>;
//          then G[i] <- a (1 - b k_i) G[i]
//   softmax  ds_i = w_i (dw_i - sum_l w_l dw_l) for both k (write) and r (read)
// and dL/dM_0 is G after token 0.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <thread>
#include <vector>

namespace {

struct Scored {
  float v;
  int32_t i;
};

// Ranking used everywhere in the selection: higher score first, then lower index.
// Comparing floats with != / > treats -0 and +0 as equal, so they tie on value.
inline bool ranks_before(const Scored& a, const Scored& b) {
  if (a.v != b.v) return a.v > b.v;
  return a.i < b.i;
}

// The kk best entries of one half (S sub-scores), best first.
void top_of_half(const float* x, int S, int kk, std::vector<Scored>& out) {
  std::vector<Scored> all(S);
  for (int j = 0; j < S; ++j) all[j] = Scored{x[j], j};
  std::partial_sort(all.begin(), all.begin() + kk, all.end(), ranks_before);
  out.assign(all.begin(), all.begin() + kk);
}

// Product-key selection for one (sequence, head, token) and one of k' / q':
// topk( topk(s1) (+) topk(s2) ), written out literally: both inner lists, the
// full kk x kk grid of fp32 sums, and a top-K of that grid.
void select_one(const float* half0, const float* half1, int S, int K, int32_t* idx, float* sc) {
  const int kk = std::min(K, S);
  std::vector<Scored> a, b;
  top_of_half(half0, S, kk, a);
  top_of_half(half1, S, kk, b);
  std::vector<Scored> grid;
  grid.reserve(size_t(kk) * kk);
  for (int p = 0; p < kk; ++p)
    for (int q = 0; q < kk; ++q) {
      const float s = a[p].v + b[q].v;  // fp32 sum
      grid.push_back(Scored{s, a[p].i * S + b[q].i});
    }
  std::partial_sort(grid.begin(), grid.begin() + K, grid.end(), ranks_before);
  for (int r = 0; r < K; ++r) {
    idx[r] = grid[r].i;
    sc[r] = grid[r].v;
  }
}

// Run f(i) for i in [0, n) over up to n_threads std::threads.
template <class F>
void parallel_for(long long n, int n_threads, F f) {
  if (n_threads <= 1 || n <= 1) {
    for (long long i = 0; i < n; ++i) f(i);
    return;
  }
  const int nt = int(std::min<long long>(n_threads, n));
  std::vector<std::thread> pool;
  for (int w = 0; w < nt; ++w)
    pool.emplace_back([=]() {
      for (long long i = w; i < n; i += nt) f(i);
    });
  for (auto& th : pool) th.join();
}

// Softmax of n scores in fp64, max-subtracted.
void softmax64(const float* s, int n, double* w) {
  double mx = s[0];
  for (int i = 1; i < n; ++i) mx = std::max(mx, double(s[i]));
  double z = 0.0;
  for (int i = 0; i < n; ++i) {
    w[i] = std::exp(double(s[i]) - mx);
    z += w[i];
  }
  for (int i = 0; i < n; ++i) w[i] /= z;
}

// Recurrent scan of one (sequence, head) over T tokens, state M[N][d_v] in fp64.
void scan_one(double* M, long long N, int dv, int T, int W, int R, const int32_t* idx_w,
              const float* sc_w, const int32_t* idx_r, const float* sc_r, const float* v,
              const float* alpha, const float* beta, double* o) {
  (void)N;
  std::vector<double> kw(W), rw(R);
  for (int t = 0; t < T; ++t) {
    // item 3: gated delta update of the W write slots (distinct rows).
    softmax64(sc_w + size_t(t) * W, W, kw.data());
    const double a = alpha[t], b = beta[t];
    const float* vt = v + size_t(t) * dv;
    for (int i = 0; i < W; ++i) {
      double* row = M + size_t(idx_w[size_t(t) * W + i]) * dv;
      for (int c = 0; c < dv; ++c) {
        const double mt = a * row[c];                     // forget gate
        row[c] = mt + b * kw[i] * (double(vt[c]) - mt);   // delta update
      }
    }
    // item 4: weighted read of the R read slots from the updated table.
    softmax64(sc_r + size_t(t) * R, R, rw.data());
    double* ot = o + size_t(t) * dv;
    for (int c = 0; c < dv; ++c) ot[c] = 0.0;
    for (int i = 0; i < R; ++i) {
      const double* row = M + size_t(idx_r[size_t(t) * R + i]) * dv;
      for (int c = 0; c < dv; ++c) ot[c] += rw[i] * row[c];
    }
  }
}

// Softmax backward: ds_i = w_i (dw_i - sum_l w_l dw_l).
void softmax64_backward(const double* w, const double* dw, int n, double* ds) {
  double dot = 0.0;
  for (int i = 0; i < n; ++i) dot += w[i] * dw[i];
  for (int i = 0; i < n; ++i) ds[i] = w[i] * (dw[i] - dot);
}

// Reverse-mode pass of scan_one for one (sequence, head).  M: state before token 0 (fp64,
// not modified); dO [T][dv]; G: in dL/dM_T (zeros if the final state carries no gradient),
// out dL/dM_0.  Outputs dv [T][dv], da [T], db [T], dsw [T][W], dsr [T][R].
void scan_backward_one(const double* M_in, long long N, int dv, int T, int W, int R,
                       const int32_t* idx_w, const float* sc_w, const int32_t* idx_r,
                       const float* sc_r, const float* v, const float* alpha, const float* beta,
                       const double* dO, double* G, double* dvv, double* da, double* db,
                       double* dsw, double* dsr) {
  // Forward again, keeping the rows the backward needs.
  std::vector<double> M(M_in, M_in + size_t(N) * dv);
  std::vector<double> w_prev(size_t(T) * W * dv), r_after(size_t(T) * R * dv);
  std::vector<double> kw(size_t(T) * W), rw(size_t(T) * R);
  for (int t = 0; t < T; ++t) {
    softmax64(sc_w + size_t(t) * W, W, kw.data() + size_t(t) * W);
    softmax64(sc_r + size_t(t) * R, R, rw.data() + size_t(t) * R);
    const double a = alpha[t], b = beta[t];
    const float* vt = v + size_t(t) * dv;
    for (int i = 0; i < W; ++i) {
      double* row = M.data() + size_t(idx_w[size_t(t) * W + i]) * dv;
      double* keep = w_prev.data() + (size_t(t) * W + i) * dv;
      const double k = kw[size_t(t) * W + i];
      for (int c = 0; c < dv; ++c) {
        keep[c] = row[c];
        const double mt = a * row[c];
        row[c] = mt + b * k * (double(vt[c]) - mt);
      }
    }
    for (int j = 0; j < R; ++j) {
      const double* row = M.data() + size_t(idx_r[size_t(t) * R + j]) * dv;
      std::copy(row, row + dv, r_after.data() + (size_t(t) * R + j) * dv);
    }
  }
  // Backwards over the tokens.
  std::vector<double> dk(W), dr(R);
  for (int t = T - 1; t >= 0; --t) {
    const double* dot = dO + size_t(t) * dv;
    const double* r = rw.data() + size_t(t) * R;
    for (int j = 0; j < R; ++j) {
      const double* mr = r_after.data() + (size_t(t) * R + j) * dv;
      double s = 0.0;
      for (int c = 0; c < dv; ++c) s += dot[c] * mr[c];
      dr[j] = s;
      double* g = G + size_t(idx_r[size_t(t) * R + j]) * dv;
      for (int c = 0; c < dv; ++c) g[c] += r[j] * dot[c];
    }
    softmax64_backward(r, dr.data(), R, dsr + size_t(t) * R);
    const double a = alpha[t], b = beta[t];
    const float* vt = v + size_t(t) * dv;
    const double* k = kw.data() + size_t(t) * W;
    double* dvt = dvv + size_t(t) * dv;
    for (int c = 0; c < dv; ++c) dvt[c] = 0.0;
    double sa = 0.0, sb = 0.0;
    for (int i = 0; i < W; ++i) {
      const double* mp = w_prev.data() + (size_t(t) * W + i) * dv;
      double* g = G + size_t(idx_w[size_t(t) * W + i]) * dv;
      double ge = 0.0, gm = 0.0;  // <G, v - a M_prev>, <G, M_prev>
      for (int c = 0; c < dv; ++c) {
        ge += g[c] * (double(vt[c]) - a * mp[c]);
        gm += g[c] * mp[c];
        dvt[c] += b * k[i] * g[c];
      }
      dk[i] = b * ge;
      sa += (1.0 - b * k[i]) * gm;
      sb += k[i] * ge;
      for (int c = 0; c < dv; ++c) g[c] *= a * (1.0 - b * k[i]);
    }
    da[t] = sa;
    db[t] = sb;
    softmax64_backward(k, dk.data(), W, dsw + size_t(t) * W);
  }
}

}  // namespace

extern "C" {

// Product-key selection for n independent items.  halves: [n][2][S] fp32
// (half 0 then half 1).  Outputs idx[n][K] (flat slot index) and sc[n][K] (fp32
// pair sum), best first.  Returns 0, or -1 on bad sizes.
int oracle_select(const float* halves, long long n, int S, int K, int32_t* idx, float* sc,
                  int n_threads) {
  if (n < 0 || S < 1 || K < 1 || (long long)K > (long long)S * S) return -1;
  parallel_for(n, n_threads, [=](long long it) {
    const float* h = halves + size_t(it) * 2 * S;
    select_one(h, h + S, S, K, idx + size_t(it) * K, sc + size_t(it) * K);
  });
  return 0;
}

// Scan of nh independent (sequence, head) pairs.  M: [nh][N][d_v] fp64, in: the
// state before token 0, out: after token T-1.  idx_w/sc_w: [nh][T][W];
// idx_r/sc_r: [nh][T][R]; v: [nh][T][d_v] fp32; alpha, beta: [nh][T];
// o: [nh][T][d_v] fp64.  Returns 0, or -1 on bad sizes / out-of-range indices.
int oracle_scan(double* M, int nh, long long N, int dv, int T, int W, int R,
                const int32_t* idx_w, const float* sc_w, const int32_t* idx_r, const float* sc_r,
                const float* v, const float* alpha, const float* beta, double* o, int n_threads) {
  if (nh < 0 || N < 1 || dv < 1 || T < 0 || W < 1 || R < 1) return -1;
  const long long nw = (long long)nh * T * W, nr = (long long)nh * T * R;
  for (long long i = 0; i < nw; ++i)
    if (idx_w[i] < 0 || idx_w[i] >= N) return -1;
  for (long long i = 0; i < nr; ++i)
    if (idx_r[i] < 0 || idx_r[i] >= N) return -1;
  parallel_for(nh, n_threads, [=](long long h) {
    scan_one(M + size_t(h) * N * dv, N, dv, T, W, R, idx_w + size_t(h) * T * W,
             sc_w + size_t(h) * T * W, idx_r + size_t(h) * T * R, sc_r + size_t(h) * T * R,
             v + size_t(h) * T * dv, alpha + size_t(h) * T, beta + size_t(h) * T,
             o + size_t(h) * T * dv);
  });
  return 0;
}

// Backward of oracle_scan for nh (sequence, head) pairs, loss sum_t <dO_t, o_t> + <dMT, M_T>.
// M: [nh][N][d_v] fp64 state before token 0 (not modified); dO: [nh][T][d_v] fp64;
// G: [nh][N][d_v] fp64, in dL/dM_T, out dL/dM_0.  Outputs (fp64): dv [nh][T][d_v],
// dalpha, dbeta [nh][T], dsc_w [nh][T][W], dsc_r [nh][T][R].  Returns 0 or -1.
int oracle_scan_backward(const double* M, int nh, long long N, int dv, int T, int W, int R,
                         const int32_t* idx_w, const float* sc_w, const int32_t* idx_r,
                         const float* sc_r, const float* v, const float* alpha, const float* beta,
                         const double* dO, double* G, double* dvv, double* dalpha, double* dbeta,
                         double* dsc_w, double* dsc_r, int n_threads) {
  if (nh < 0 || N < 1 || dv < 1 || T < 0 || W < 1 || R < 1) return -1;
  const long long nw = (long long)nh * T * W, nr = (long long)nh * T * R;
  for (long long i = 0; i < nw; ++i)
    if (idx_w[i] < 0 || idx_w[i] >= N) return -1;
  for (long long i = 0; i < nr; ++i)
    if (idx_r[i] < 0 || idx_r[i] >= N) return -1;
  parallel_for(nh, n_threads, [=](long long h) {
    scan_backward_one(M + size_t(h) * N * dv, N, dv, T, W, R, idx_w + size_t(h) * T * W,
                      sc_w + size_t(h) * T * W, idx_r + size_t(h) * T * R,
                      sc_r + size_t(h) * T * R, v + size_t(h) * T * dv, alpha + size_t(h) * T,
                      beta + size_t(h) * T, dO + size_t(h) * T * dv, G + size_t(h) * N * dv,
                      dvv + size_t(h) * T * dv, dalpha + size_t(h) * T, dbeta + size_t(h) * T,
                      dsc_w + size_t(h) * T * W, dsc_r + size_t(h) * T * R);
  });
  return 0;
}

}  // extern "C"
