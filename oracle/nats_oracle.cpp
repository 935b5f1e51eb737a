// nats_oracle.cpp - plain, slow, float64 CPU oracle of the NAtS-L hybrid
// attention layer forward (prefill).
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
// benchmark's CPU-baseline leg may load this library.  It shares no code,
// header, table or helper with the CUDA path and must never be used to
// produce a product result.
//
// Source of every step: "Neural Attention Search Linear (NAtS-L)", technical
// summary (Dutch and German versions of the same page), section
// "Kernmechanismen":
//   item 1 (token-level hybridisation): the sequence is cut into chunks; an
//          Attention Score Layer (mean pooling followed by a linear layer)
//          maps each chunk to one score per operation type (softmax attention,
//          Gated DeltaNet); the operation with the highest score gets the chunk.
//   item 3 (chunk-wise computation): inside a chunk both the softmax and the
//          linear correlations are computed; both hidden states (the retained
//          KV set and the Gated DeltaNet state) are pseudo-updated for every
//          new chunk, and for the operation that was not selected the state
//          is reset / rolled back to the beginning of the chunk.
//   item 4 (output merging): both branch outputs are RMS-normalised
//          separately and combined by a weighted sum whose weights come from
//          the query projections.
// Readings where the pages are silent (named CONV-n):
//   CONV-1  Gated DeltaNet: S_t = a_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
//           read out after the update: o_t = S_t (scale * q_t).
//   CONV-2  score input: mean over the chunk's tokens of [q_t ; k_t] (unscaled q),
//           per-head weights W_s[h] (2 x 2dk) and bias b_s[h] (2); row 0 = softmax.
//   CONV-3  argmax ties go to row 0 (softmax).
//   CONV-4  the softmax branch of every token attends to all tokens of earlier
//           softmax-selected chunks plus its own chunk causally (diagonal
//           included), whatever its own chunk's selection.
//   CONV-5  rollback restores the state exactly as it was at the chunk start.
//   CONV-6  initial state S = 0, empty KV set.
//   CONV-7  scale = 1/sqrt(dk) unless given.
//   CONV-8  RMSNorm per token over dv: x / sqrt(mean(x^2) + eps) * w.
//   CONV-9  merge: w_t = sigmoid(q_t . W_g[h] + b_g[h]); out = w N_soft + (1 - w) N_lin.
//   CONV-12 a last partial chunk pools over the tokens it has.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

extern "C" {

typedef struct {
  int32_t B, H, L, dk, dv, chunk;
  double scale;  // <= 0 selects 1/sqrt(dk)
  double eps;
} nats_oracle_dims;

}  // extern "C"

namespace {

struct HeadView {
  const float* q;  // [L, dk]
  const float* k;  // [L, dk]
  const float* v;  // [L, dv]
  const float* g;  // [L]
  const float* beta;
  int b, h;
};

double scale_of(const nats_oracle_dims& d) {
  return d.scale > 0 ? d.scale : 1.0 / std::sqrt((double)d.dk);
}

// Kernmechanismen 1: mean-pool the chunk's [q ; k], one linear score per
// operation, argmax (CONV-2, CONV-3).
void select_head(const nats_oracle_dims& d, const HeadView& hv, const float* w_s,
                 const float* b_s, uint8_t* sel, double* scores) {
  const int C = d.chunk, N = (d.L + C - 1) / C, dk = d.dk;
  const float* W = w_s + (size_t)hv.h * 2 * 2 * dk;
  std::vector<double> p(2 * dk);
  for (int c = 0; c < N; ++c) {
    const int t0 = c * C, t1 = std::min(d.L, t0 + C);
    std::fill(p.begin(), p.end(), 0.0);
    for (int t = t0; t < t1; ++t) {
      for (int j = 0; j < dk; ++j) {
        p[j] += hv.q[(size_t)t * dk + j];
        p[dk + j] += hv.k[(size_t)t * dk + j];
      }
    }
    for (double& x : p) x /= (double)(t1 - t0);
    double s[2];
    for (int o = 0; o < 2; ++o) {
      double acc = b_s ? (double)b_s[hv.h * 2 + o] : 0.0;
      for (int j = 0; j < 2 * dk; ++j) acc += (double)W[o * 2 * dk + j] * p[j];
      s[o] = acc;
    }
    sel[c] = (s[0] >= s[1]) ? 0 : 1;
    if (scores) {
      scores[2 * c] = s[0];
      scores[2 * c + 1] = s[1];
    }
  }
}

// Kernmechanismen 3, softmax side (CONV-4, CONV-6, CONV-7): explicit softmax
// over the retained KV set.  After chunk c, its tokens join the retained set
// only if the chunk chose softmax; otherwise the set is rolled back.
void softmax_branch(const nats_oracle_dims& d, const HeadView& hv, const uint8_t* sel,
                    const uint8_t* rows, double* o_s) {
  const int C = d.chunk, N = (d.L + C - 1) / C, dk = d.dk, dv = d.dv;
  const double scale = scale_of(d);
  std::vector<int> kv;  // retained token indices
  kv.reserve(d.L);
  std::vector<double> logit;
  std::vector<int> J;
  for (int c = 0; c < N; ++c) {
    const int t0 = c * C, t1 = std::min(d.L, t0 + C);
    for (int t = t0; t < t1; ++t) {
      if (rows && !rows[t]) continue;
      J.assign(kv.begin(), kv.end());
      for (int j = t0; j <= t; ++j) J.push_back(j);
      logit.resize(J.size());
      double m = -INFINITY;
      for (size_t n = 0; n < J.size(); ++n) {
        double acc = 0.0;
        const float* qt = hv.q + (size_t)t * dk;
        const float* kj = hv.k + (size_t)J[n] * dk;
        for (int i = 0; i < dk; ++i) acc += (double)qt[i] * (double)kj[i];
        logit[n] = acc * scale;
        m = std::max(m, logit[n]);
      }
      double Z = 0.0;
      for (double& x : logit) {
        x = std::exp(x - m);
        Z += x;
      }
      double* o = o_s + (size_t)t * dv;
      for (int i = 0; i < dv; ++i) o[i] = 0.0;
      for (size_t n = 0; n < J.size(); ++n) {
        const double p = logit[n] / Z;
        const float* vj = hv.v + (size_t)J[n] * dv;
        for (int i = 0; i < dv; ++i) o[i] += p * (double)vj[i];
      }
    }
    if (sel[c] == 0)
      for (int j = t0; j < t1; ++j) kv.push_back(j);
  }
}

// Kernmechanismen 3, linear side (CONV-1, CONV-5, CONV-6): the Gated DeltaNet
// recurrence token by token; the state is pseudo-updated through every chunk
// and restored to the chunk-start copy when the chunk chose softmax.
void gdn_branch(const nats_oracle_dims& d, const HeadView& hv, const uint8_t* sel,
                double* o_l, double* state_out) {
  const int C = d.chunk, N = (d.L + C - 1) / C, dk = d.dk, dv = d.dv;
  const double scale = scale_of(d);
  std::vector<double> S((size_t)dv * dk, 0.0), S0, Sk(dv);
  for (int c = 0; c < N; ++c) {
    const int t0 = c * C, t1 = std::min(d.L, t0 + C);
    S0 = S;
    for (int t = t0; t < t1; ++t) {
      const double a = std::exp((double)hv.g[t]);
      const double b = hv.beta[t];
      const float* kt = hv.k + (size_t)t * dk;
      const float* vt = hv.v + (size_t)t * dv;
      const float* qt = hv.q + (size_t)t * dk;
      // S k_t with the pre-update state
      for (int r = 0; r < dv; ++r) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += S[(size_t)r * dk + i] * (double)kt[i];
        Sk[r] = acc;
      }
      // S <- a S (I - b k k^T) + b v k^T  =  a S - a b (S k) k^T + b v k^T
      for (int r = 0; r < dv; ++r) {
        const double coef = b * (double)vt[r] - a * b * Sk[r];
        for (int i = 0; i < dk; ++i)
          S[(size_t)r * dk + i] = a * S[(size_t)r * dk + i] + coef * (double)kt[i];
      }
      if (o_l) {
        double* o = o_l + (size_t)t * dv;
        for (int r = 0; r < dv; ++r) {
          double acc = 0.0;
          for (int i = 0; i < dk; ++i) acc += S[(size_t)r * dk + i] * (double)qt[i];
          o[r] = acc * scale;
        }
      }
    }
    if (sel[c] == 0) S = S0;  // rollback: the chunk belongs to the softmax branch
  }
  if (state_out) std::copy(S.begin(), S.end(), state_out);
}

// Kernmechanismen 4 (CONV-8, CONV-9): RMSNorm per branch, query-gated sum.
void norm_merge(const nats_oracle_dims& d, const HeadView& hv, const float* w_g,
                const float* b_g, const float* nw_s, const float* nw_l, const uint8_t* rows,
                const double* o_s, const double* o_l, double* out) {
  const int dk = d.dk, dv = d.dv;
  for (int t = 0; t < d.L; ++t) {
    if (rows && !rows[t]) continue;
    const double* xs = o_s + (size_t)t * dv;
    const double* xl = o_l + (size_t)t * dv;
    double ms = 0.0, ml = 0.0;
    for (int i = 0; i < dv; ++i) {
      ms += xs[i] * xs[i];
      ml += xl[i] * xl[i];
    }
    const double rs = 1.0 / std::sqrt(ms / dv + d.eps);
    const double rl = 1.0 / std::sqrt(ml / dv + d.eps);
    double z = b_g ? (double)b_g[hv.h] : 0.0;
    const float* qt = hv.q + (size_t)t * dk;
    for (int i = 0; i < dk; ++i) z += (double)qt[i] * (double)w_g[(size_t)hv.h * dk + i];
    const double w = 1.0 / (1.0 + std::exp(-z));
    double* o = out + (size_t)t * dv;
    for (int i = 0; i < dv; ++i) {
      const double ns = xs[i] * rs * (nw_s ? (double)nw_s[i] : 1.0);
      const double nl = xl[i] * rl * (nw_l ? (double)nw_l[i] : 1.0);
      o[i] = w * ns + (1.0 - w) * nl;
    }
  }
}

bool dims_ok(const nats_oracle_dims* d) {
  return d && d->B >= 0 && d->H >= 0 && d->L >= 0 && d->dk > 0 && d->dv > 0 && d->chunk > 0;
}

HeadView view_of(const nats_oracle_dims& d, const float* q, const float* k, const float* v,
                 const float* g, const float* beta, int flat) {
  HeadView hv;
  hv.b = flat / d.H;
  hv.h = flat % d.H;
  hv.q = q + (size_t)flat * d.L * d.dk;
  hv.k = k + (size_t)flat * d.L * d.dk;
  hv.v = v ? v + (size_t)flat * d.L * d.dv : nullptr;
  hv.g = g ? g + (size_t)flat * d.L : nullptr;
  hv.beta = beta ? beta + (size_t)flat * d.L : nullptr;
  return hv;
}

template <class F>
int run_parallel(int n_items, int threads, F&& fn) {
  int nt = threads > 0 ? threads : (int)std::thread::hardware_concurrency();
  nt = std::max(1, std::min(nt, std::max(1, n_items)));
  std::atomic<int> next{0};
  auto worker = [&]() {
    for (int i = next.fetch_add(1); i < n_items; i = next.fetch_add(1)) fn(i);
  };
  if (nt == 1) {
    worker();
  } else {
    std::vector<std::thread> pool;
    for (int i = 0; i < nt; ++i) pool.emplace_back(worker);
    for (auto& th : pool) th.join();
  }
  return nt;
}

}  // namespace

extern "C" {

// Selection only, for every (b, h).  sel: [B*H, N] (0 softmax, 1 Gated
// DeltaNet); scores: [B*H, N, 2] or NULL.  Returns 0 on success.
int nats_oracle_select(const nats_oracle_dims* dims, const float* q, const float* k,
                       const float* w_s, const float* b_s, uint8_t* sel, double* scores,
                       int32_t threads) {
  if (!dims_ok(dims) || !q || !k || !w_s || !sel) return 1;
  const nats_oracle_dims d = *dims;
  const int N = (d.L + d.chunk - 1) / d.chunk;
  run_parallel(d.B * d.H, threads, [&](int flat) {
    HeadView hv = view_of(d, q, k, nullptr, nullptr, nullptr, flat);
    select_head(d, hv, w_s, b_s, sel + (size_t)flat * N, scores ? scores + (size_t)flat * N * 2 : nullptr);
  });
  return 0;
}

// Full layer forward for the heads listed in `heads` (flat b*H+h; NULL means
// all B*H heads in order).  Outputs are packed per listed head:
//   sel [n, N], scores [n, N, 2], o_s / o_l / out [n, L, dv], state [n, dv, dk];
// any output may be NULL.  `rows` ([L] bytes or NULL = all) limits the rows of
// o_s and out that are computed; other rows are left untouched.  The Gated
// DeltaNet branch always runs over every row (its state needs them).
// sel_in ([B*H, N] or NULL) overrides the score layer's choice.
int nats_oracle_forward(const nats_oracle_dims* dims, const float* q, const float* k,
                        const float* v, const float* g, const float* beta, const float* w_s,
                        const float* b_s, const float* w_g, const float* b_g,
                        const float* norm_w_soft, const float* norm_w_lin, const uint8_t* sel_in,
                        const int32_t* heads, int32_t n_heads, const uint8_t* rows,
                        uint8_t* sel, double* scores, double* o_s, double* o_l, double* out,
                        double* state, int32_t threads, int32_t* threads_used) {
  if (!dims_ok(dims) || !q || !k || !v || !g || !beta || !w_g) return 1;
  if (!sel_in && !w_s) return 1;
  const nats_oracle_dims d = *dims;
  const int N = (d.L + d.chunk - 1) / d.chunk;
  const int n = heads ? n_heads : d.B * d.H;
  for (int i = 0; heads && i < n; ++i)
    if (heads[i] < 0 || heads[i] >= d.B * d.H) return 2;
  const int used = run_parallel(n, threads, [&](int i) {
    const int flat = heads ? heads[i] : i;
    HeadView hv = view_of(d, q, k, v, g, beta, flat);
    std::vector<uint8_t> s(N);
    if (sel_in) {
      std::copy(sel_in + (size_t)flat * N, sel_in + (size_t)(flat + 1) * N, s.begin());
      if (scores) std::fill(scores + (size_t)i * N * 2, scores + (size_t)(i + 1) * N * 2, 0.0);
    } else {
      select_head(d, hv, w_s, b_s, s.data(), scores ? scores + (size_t)i * N * 2 : nullptr);
    }
    if (sel) std::copy(s.begin(), s.end(), sel + (size_t)i * N);
    std::vector<double> os, ol;
    double* ps = o_s ? o_s + (size_t)i * d.L * d.dv : nullptr;
    double* pl = o_l ? o_l + (size_t)i * d.L * d.dv : nullptr;
    if (out && !ps) {
      os.assign((size_t)d.L * d.dv, 0.0);
      ps = os.data();
    }
    if (out && !pl) {
      ol.assign((size_t)d.L * d.dv, 0.0);
      pl = ol.data();
    }
    if (ps) softmax_branch(d, hv, s.data(), rows, ps);
    if (pl || state) gdn_branch(d, hv, s.data(), pl, state ? state + (size_t)i * d.dv * d.dk : nullptr);
    if (out)
      norm_merge(d, hv, w_g, b_g, norm_w_soft, norm_w_lin, rows, ps, pl, out + (size_t)i * d.L * d.dv);
  });
  if (threads_used) *threads_used = used;
  return 0;
}

}  // extern "C"
