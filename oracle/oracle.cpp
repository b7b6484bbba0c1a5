// CPU oracle for the DominoTree drafting-round tree builder.
//
// TEST INFRASTRUCTURE. Only the test suite, the smoke check and the bench's CPU-baseline leg load this library.
// The CUDA product path never calls it, and the two share no code: this file has its own bf16 decoding, its own
// GRU, its own correction and softmax, its own heap.
//
// Plain and slow on purpose: fp64 everywhere, one loop per formula, library sort and heap, no blocking or fusion.
// Inputs are read in their storage form (fp32, or bf16 bit patterns) and widened exactly to double.
//
// What it computes follows three web pages about the paper "DominoTree: Conditional Tree-Structured Drafting with
// Domino for Speculative Decoding" (arXiv 2607.08642):
//   [S] blog.captcha.la summary      - "Methodology — deep read", "Technical innovations", "Key findings"
//   [Z] zhichai.top blog (Chinese)   - "两条路线的困境", "DominoTree 的破局"
//   [G] gist.science explainer (fr)  - "Résumé Technique / Méthodologie / Composants Clés", "Vérification"
// Where the pages are silent the reading taken is stated next to the code it governs.
//
// Parity status of each function (what pins it, all in the CPU test suite):
//   orc_topm        - pinned: full lexicographic sort of every row (brute force).
//   orc_gru_step    - pinned: torch.nn.GRUCell in fp64 on the same weights.
//   orc_child_logp  - pinned: with M = V equals torch.log_softmax of the full-vocabulary corrected row.
//   orc_build_trees - pinned: brute-force enumeration of the depth-limited M-ary tree on tiny inputs; the
//                     W_c = 0 factorised closed form; the M = 1 / max_depth = 1 / n = 1 special cases.
//   orc_rescore     - pinned: must reproduce orc_build_trees' own scores on its own trees, and the brute-force
//                     path scores.
//   orc_accept_paths - pinned: the longest path, among all root-to-node paths enumerated, whose tokens agree with
//                     the target's next tokens along it; special cases (all rejected, a whole chain accepted).
//   orc_lmhead_topm - pinned: numpy's fp64 matmul of the widened inputs followed by a full lexicographic sort; a
//                     one-hot head whose logits are the hidden values themselves; duplicated head rows (ties go
//                     to the lower id).
//   orc_tree_attention - pinned: torch's scaled_dot_product_attention in fp64 with the same boolean mask and the
//                     key/value heads repeated for the grouped query heads; a diagonal mask with no prefix (every
//                     node sees only itself: out = its own v); equal scores (out = the mean of the visible v).
//   orc_build_trees_marginal - pinned: brute-force enumeration of the depth-limited tree under the product of the
//                     marginals (log-softmax by torch), and equality with orc_build_trees at W_c = 0.
//   The GRU gate layout (rows r|z|n, PyTorch convention) and the order "add correction, then divide by T" are
//   readings; against the real Domino checkpoint the semantics are parity unpinned (no equations on the pages).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <numeric>
#include <queue>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };  // ORC_F64: the oracle's own fp64 intermediates

enum {
  ORC_OK = 0,
  ORC_ERR_ARG = 1,      // inconsistent sizes or a null pointer
  ORC_ERR_NAN = 2,      // a NaN among the logits
  ORC_ERR_BUDGET = 3,   // fewer than n nodes exist within max_depth
  ORC_ERR_TREE = 4,     // orc_rescore: the given tree is not a valid draft tree over the candidates
};

// Exact widening of one stored element to double.
double load(const void* base, int dtype, size_t i) {
  if (dtype == ORC_F64) return static_cast<const double*>(base)[i];
  if (dtype == ORC_F32) return static_cast<double>(static_cast<const float*>(base)[i]);
  const uint32_t bits = static_cast<uint32_t>(static_cast<const uint16_t*>(base)[i]) << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return static_cast<double>(f);
}

struct Weights {
  int H, E, dtype;
  const void* emb;   // [V,E]
  const void* w_ih;  // [3H,E], gate rows r|z|n
  const void* w_hh;  // [3H,H], gate rows r|z|n
  const void* b_ih;  // [3H] or null (zero)
  const void* b_hh;  // [3H] or null (zero)
  const void* w_c;   // [V,H] correction rows
};

double bias(const void* b, int dtype, size_t i) { return b ? load(b, dtype, i) : 0.0; }

// ---------------------------------------------------------------------------------------------------------------
// Top-M candidate restriction. [S] "Methodology — deep read" and "Technical innovations": at every block position
// the children may only be the M tokens with the highest marginal logit. [G] "Composants Clés — Restriction de
// Candidats". Order: value descending, then id ascending (so -0.0 and +0.0 tie and the id decides).
int topm_row(const void* logits, int dtype, size_t row_off, int V, int M, int32_t* ids, double* vals) {
  std::vector<double> v(static_cast<size_t>(V));
  for (int i = 0; i < V; ++i) {
    v[i] = load(logits, dtype, row_off + static_cast<size_t>(i));
    if (std::isnan(v[i])) return ORC_ERR_NAN;
  }
  std::vector<int> order(static_cast<size_t>(V));
  std::iota(order.begin(), order.end(), 0);
  std::partial_sort(order.begin(), order.begin() + M, order.end(), [&](int a, int b) {
    if (v[a] != v[b]) return v[a] > v[b];
    return a < b;
  });
  for (int m = 0; m < M; ++m) {
    ids[m] = order[m];
    vals[m] = v[order[m]];
  }
  return ORC_OK;
}

// ---------------------------------------------------------------------------------------------------------------
// One step of the Domino GRU along a draft path. [S] "Methodology — deep read": the hidden state is carried and
// updated along each candidate path. [G] "Composants Clés": only the light GRU correction is recomputed per node.
// Reading: the pages give no equations, so the cell is PyTorch's GRUCell with gate rows r|z|n:
//   r = sigmoid(W_ir x + b_ir + W_hr h + b_hr)
//   u = sigmoid(W_iz x + b_iz + W_hz h + b_hz)          (the update gate, "z" in PyTorch's notation)
//   g = tanh(W_in x + b_in + r * (W_hn h + b_hn))
//   h' = (1 - u) * g + u * h
void gru_step(const Weights& w, const double* x, const double* h, double* out) {
  const int H = w.H, E = w.E;
  for (int k = 0; k < H; ++k) {
    double in_side[3], hid_side[3];
    for (int gate = 0; gate < 3; ++gate) {
      const size_t row = static_cast<size_t>(gate) * H + k;
      double a = bias(w.b_ih, w.dtype, row);
      for (int e = 0; e < E; ++e) a += load(w.w_ih, w.dtype, row * E + e) * x[e];
      double c = bias(w.b_hh, w.dtype, row);
      for (int j = 0; j < H; ++j) c += load(w.w_hh, w.dtype, row * H + j) * h[j];
      in_side[gate] = a;
      hid_side[gate] = c;
    }
    const double r = 1.0 / (1.0 + std::exp(-(in_side[0] + hid_side[0])));
    const double u = 1.0 / (1.0 + std::exp(-(in_side[1] + hid_side[1])));
    const double g = std::tanh(in_side[2] + r * hid_side[2]);
    out[k] = (1.0 - u) * g + u * h[k];
  }
}

// ---------------------------------------------------------------------------------------------------------------
// Conditional log-probabilities of the M candidates of one block position, given the hidden state h of the node
// being expanded. [S] "Methodology — deep read": the correction is applied only to the top-M slice, by fetching
// the matching rows of the correction matrix and of the base logits. [G] "Composants Clés": the base marginal
// logit L_base is corrected by Delta L (the GRU head's output) on that slice.
// Reading: Delta L_m = W_c[ids_m] . h; the corrected logit is divided by the temperature (T_eff = 1 when T = 0,
// greedy decoding, where a softmax is undefined), then log-softmax over the M candidates only.
void child_logp(const Weights& w, const int32_t* ids, const double* base, int M, double T_eff, const double* h,
                double* logp) {
  const int H = w.H;
  std::vector<double> z(static_cast<size_t>(M));
  for (int m = 0; m < M; ++m) {
    double s = 0.0;
    for (int k = 0; k < H; ++k) s += load(w.w_c, w.dtype, static_cast<size_t>(ids[m]) * H + k) * h[k];
    z[m] = (base[m] + s) / T_eff;
  }
  double mx = z[0];
  for (int m = 1; m < M; ++m) mx = std::max(mx, z[m]);
  double sum = 0.0;
  for (int m = 0; m < M; ++m) sum += std::exp(z[m] - mx);
  const double lse = std::log(sum);
  for (int m = 0; m < M; ++m) logp[m] = (z[m] - mx) - lse;
}

// ---------------------------------------------------------------------------------------------------------------
// Best-first tree growth. [S] "Methodology — deep read": DDTree's best-first search with a max-priority queue keyed
// by the cumulative conditional log-probability, expanded until the node budget n (or the depth limit) is reached;
// the tree is prefix-closed. [G] "Tas de Recherche de Premier Choix à Score Conditionnel".
// Readings: the root is the last accepted token, has score 0 and hidden state h0 (no GRU step); its children sit
// at depth 1 and use block position 0, and in general a node at depth d expands into block position d. The budget
// counts draft nodes only. Ties in the queue: higher score first, then lower token id, then earlier insertion
// (children are inserted in candidate order m = 0..M-1, the root's first). The n-th pop is not expanded.
struct Cand {
  double score;
  int token;
  int parent;  // index of the parent among the popped nodes, -1 for a child of the root
  int depth;
  long long seq;
};
struct RanksBelow {  // a ranks below b in the queue
  bool operator()(const Cand& a, const Cand& b) const {
    if (a.score != b.score) return a.score < b.score;
    if (a.token != b.token) return a.token > b.token;
    return a.seq > b.seq;
  }
};

// Number of nodes of the depth-limited M-ary tree, saturated at `cap`.
long long tree_size(int M, int max_depth, long long cap) {
  long long total = 0, level = 1;
  for (int d = 1; d <= max_depth; ++d) {
    level = (level > cap / std::max(M, 1)) ? cap : level * M;
    total = std::min(cap, total + level);
  }
  return total;
}

int build_one(const Weights& w, const int32_t* ids, const double* vals, int M, int n, int max_depth, double T,
              const double* h0, int32_t* tokens, int32_t* parents, int32_t* depth, double* scores, uint8_t* mask,
              double* gaps) {
  const int H = w.H, E = w.E;
  const double T_eff = T > 0.0 ? T : 1.0;
  std::priority_queue<Cand, std::vector<Cand>, RanksBelow> frontier;
  std::vector<double> hs(static_cast<size_t>(n) * H);  // hidden state of every popped, expanded node
  std::vector<double> logp(static_cast<size_t>(M)), x(static_cast<size_t>(E));
  long long seq = 0;

  auto expand = [&](const double* h, int parent, int d, double score) {
    child_logp(w, ids + static_cast<size_t>(d) * M, vals + static_cast<size_t>(d) * M, M, T_eff, h, logp.data());
    for (int m = 0; m < M; ++m)
      frontier.push(Cand{score + logp[m], ids[static_cast<size_t>(d) * M + m], parent, d + 1, seq++});
  };

  expand(h0, -1, 0, 0.0);
  for (int i = 0; i < n; ++i) {
    if (frontier.empty()) return ORC_ERR_BUDGET;
    const Cand u = frontier.top();
    frontier.pop();
    gaps[i] = frontier.empty() ? std::numeric_limits<double>::infinity() : u.score - frontier.top().score;
    tokens[i] = u.token;
    parents[i] = u.parent;
    depth[i] = u.depth;
    scores[i] = u.score;
    if (i + 1 < n && u.depth < max_depth) {
      const double* hp = u.parent < 0 ? h0 : &hs[static_cast<size_t>(u.parent) * H];
      for (int e = 0; e < E; ++e) x[e] = load(w.emb, w.dtype, static_cast<size_t>(u.token) * E + e);
      gru_step(w, x.data(), hp, &hs[static_cast<size_t>(i) * H]);
      expand(&hs[static_cast<size_t>(i) * H], i, u.depth, u.score);
    }
  }
  // Ancestor-only attention mask ([S] "Methodology — deep read"; [G] "Vérification"): row i sees itself and its
  // ancestors. The root (the accepted prefix) is always visible and has no column.
  for (int i = 0; i < n; ++i) {
    for (int j = 0; j < n; ++j) mask[static_cast<size_t>(i) * n + j] = 0;
    for (int j = i; j >= 0; j = parents[j]) mask[static_cast<size_t>(i) * n + j] = 1;
  }
  return ORC_OK;
}

// Scores of a given tree (for instance one built elsewhere), recomputed along each node's path.
int rescore_one(const Weights& w, const int32_t* ids, const double* vals, int M, int n, int max_depth, double T,
                const double* h0, const int32_t* tokens, const int32_t* parents, const int32_t* depth,
                double* scores) {
  const int H = w.H, E = w.E;
  const double T_eff = T > 0.0 ? T : 1.0;
  std::vector<double> hs(static_cast<size_t>(n) * H);
  std::vector<char> has_h(static_cast<size_t>(n), 0);
  std::vector<double> logp(static_cast<size_t>(M)), x(static_cast<size_t>(E));
  for (int i = 0; i < n; ++i) {
    const int p = parents[i];
    if (p < -1 || p >= i) return ORC_ERR_TREE;
    const int d = depth[i];
    if (d != (p < 0 ? 1 : depth[p] + 1) || d < 1 || d > max_depth) return ORC_ERR_TREE;
    const double* hp = h0;
    double base_score = 0.0;
    if (p >= 0) {
      if (!has_h[p]) {
        const double* hpp = parents[p] < 0 ? h0 : &hs[static_cast<size_t>(parents[p]) * H];
        for (int e = 0; e < E; ++e) x[e] = load(w.emb, w.dtype, static_cast<size_t>(tokens[p]) * E + e);
        gru_step(w, x.data(), hpp, &hs[static_cast<size_t>(p) * H]);
        has_h[p] = 1;
      }
      hp = &hs[static_cast<size_t>(p) * H];
      base_score = scores[p];
    }
    const size_t pos = static_cast<size_t>(d - 1) * M;
    child_logp(w, ids + pos, vals + pos, M, T_eff, hp, logp.data());
    int found = -1;
    for (int m = 0; m < M; ++m)
      if (ids[pos + m] == tokens[i]) { found = m; break; }
    if (found < 0) return ORC_ERR_TREE;
    scores[i] = base_score + logp[found];
  }
  return ORC_OK;
}

// ---------------------------------------------------------------------------------------------------------------
// The factorised (marginal) scoring of DDTree, the baseline DominoTree is ablated against. [S] "Methodology — deep
// read": DDTree scores tree nodes by factorized marginal log-probabilities; [S] "Key findings": conditional scoring
// gains +9.2% throughput over marginal scoring at matched budget and verifier; [G] "Énoncé du Problème": in the
// factorised formulations a token's score depends only on its position, not on the path that reached it.
// Reading: the marginal log-probability of candidate m at block position d is the log-softmax of the top-M base
// logits of that position divided by the temperature (T_eff = 1 when T = 0), restricted to those M; a node's score
// is the sum along its path; the same best-first search, ties and budget as build_one.
int build_one_marginal(const int32_t* ids, const double* vals, int M, int n, int max_depth, double T,
                       int32_t* tokens, int32_t* parents, int32_t* depth, double* scores, uint8_t* mask,
                       double* gaps) {
  const double T_eff = T > 0.0 ? T : 1.0;
  // per-position marginal log-probabilities over the M candidates
  std::vector<double> marg(static_cast<size_t>(max_depth) * M);
  for (int d = 0; d < max_depth; ++d) {
    const double* v = vals + static_cast<size_t>(d) * M;
    double mx = v[0] / T_eff;
    for (int m = 1; m < M; ++m) mx = std::max(mx, v[m] / T_eff);
    double sum = 0.0;
    for (int m = 0; m < M; ++m) sum += std::exp(v[m] / T_eff - mx);
    const double lse = std::log(sum);
    for (int m = 0; m < M; ++m) marg[static_cast<size_t>(d) * M + m] = (v[m] / T_eff - mx) - lse;
  }
  std::priority_queue<Cand, std::vector<Cand>, RanksBelow> frontier;
  long long seq = 0;
  auto expand = [&](int parent, int d, double score) {
    for (int m = 0; m < M; ++m)
      frontier.push(Cand{score + marg[static_cast<size_t>(d) * M + m], ids[static_cast<size_t>(d) * M + m], parent,
                         d + 1, seq++});
  };
  expand(-1, 0, 0.0);
  for (int i = 0; i < n; ++i) {
    if (frontier.empty()) return ORC_ERR_BUDGET;
    const Cand u = frontier.top();
    frontier.pop();
    gaps[i] = frontier.empty() ? std::numeric_limits<double>::infinity() : u.score - frontier.top().score;
    tokens[i] = u.token;
    parents[i] = u.parent;
    depth[i] = u.depth;
    scores[i] = u.score;
    if (i + 1 < n && u.depth < max_depth) expand(i, u.depth, u.score);
  }
  for (int i = 0; i < n; ++i) {
    for (int j = 0; j < n; ++j) mask[static_cast<size_t>(i) * n + j] = 0;
    for (int j = i; j >= 0; j = parents[j]) mask[static_cast<size_t>(i) * n + j] = 1;
  }
  return ORC_OK;
}

// ---------------------------------------------------------------------------------------------------------------
// Acceptance of a verified tree. [S] "Methodology — deep read": one target forward pass over the tree (ancestor-only
// mask) verifies it and the longest accepted root-to-leaf path is kept; [S] "Threat model" and [G] "Résultats
// Expérimentaux": lossless, the output equals serial greedy decoding. Reading (greedy verification): target_next[0]
// is the target's next token after the accepted prefix, target_next[1 + i] its next token after node i; a path
// v1 .. vk is accepted when token(v1) = target_next[0] and token(v_{j+1}) = target_next[1 + v_j]; the bonus token is
// the target's next token after the last accepted node. If two children of a node carry the same token, the earlier
// pop is taken. Returns ORC_ERR_TREE unless every parent precedes its child.
int accept_one(int n, const int32_t* tokens, const int32_t* parents, const int32_t* target_next, int32_t* accept_len,
               int32_t* path, int32_t* bonus) {
  for (int i = 0; i < n; ++i)
    if (parents[i] < -1 || parents[i] >= i) return ORC_ERR_TREE;
  int cur = -1, len = 0, want = target_next[0];
  while (true) {
    int next = -1;
    for (int i = 0; i < n; ++i)
      if (parents[i] == cur && tokens[i] == want) {
        next = i;
        break;
      }
    if (next < 0) break;
    path[len++] = next;
    cur = next;
    want = target_next[1 + next];
  }
  for (int i = len; i < n; ++i) path[i] = -1;
  *accept_len = len;
  *bonus = want;
  return ORC_OK;
}

int threads_or_default(int threads) {
#ifdef _OPENMP
  return threads > 0 ? threads : omp_get_max_threads();
#else
  (void)threads;
  return 1;
#endif
}

}  // namespace

extern "C" {

// Top-M of every row of logits [B,K,V] -> ids [B,K,M], vals [B,K,M] (fp64, exact widening of the stored value).
int orc_topm(const void* logits, int dtype, int B, int K, int V, int M, int32_t* ids, double* vals, int threads) {
  if (!logits || !ids || !vals || B < 0 || K < 1 || V < 1 || M < 1 || M > V) return ORC_ERR_ARG;
  const long long rows = static_cast<long long>(B) * K;
  int status = ORC_OK;
#pragma omp parallel for schedule(dynamic) num_threads(threads_or_default(threads))
  for (long long r = 0; r < rows; ++r) {
    const int s = topm_row(logits, dtype, static_cast<size_t>(r) * V, V, M, ids + r * M, vals + r * M);
    if (s != ORC_OK) {
#pragma omp critical
      status = s;
    }
  }
  return status;
}

// Top-M of the full-vocabulary projection: logits[r][v] = sum_k hidden[r][k] * w_head[v][k] (fp64 from the exactly
// widened inputs, the plain dot product, no bias), then the M largest of every row with ties to the lower id, as in
// orc_topm. [S] "Methodology — deep read" and [G] "Composants Clés — Restriction de Candidats": the drafter's base
// logits come from the costly projection over the whole vocabulary (W2), of which only the top-M are kept.
// hidden [R,D], w_head [V,D], each fp32 or bf16 (dtype code as for the weights); ids [R,M], vals [R,M].
int orc_lmhead_topm(int R, int D, int V, int M, const void* hidden, int hdtype, const void* w_head, int wdtype,
                    int32_t* ids, double* vals, int threads) {
  if (!hidden || !w_head || !ids || !vals || R < 0 || D < 1 || V < 1 || M < 1 || M > V) return ORC_ERR_ARG;
  int status = ORC_OK;
#pragma omp parallel for schedule(dynamic) num_threads(threads_or_default(threads))
  for (int r = 0; r < R; ++r) {
    std::vector<double> h(static_cast<size_t>(D));
    for (int k = 0; k < D; ++k) h[k] = load(hidden, hdtype, static_cast<size_t>(r) * D + k);
    std::vector<double> logits(static_cast<size_t>(V));
    for (int v = 0; v < V; ++v) {
      double acc = 0.0;
      for (int k = 0; k < D; ++k) acc += h[k] * load(w_head, wdtype, static_cast<size_t>(v) * D + k);
      logits[v] = acc;
    }
    const int s = topm_row(logits.data(), ORC_F64, 0, V, M, ids + static_cast<size_t>(r) * M,
                           vals + static_cast<size_t>(r) * M);
    if (s != ORC_OK) {
#pragma omp critical
      status = s;
    }
  }
  return status;
}

// Tree attention of the verify pass. [S] "Methodology — deep read": the tree is verified in one target forward pass
// with an ancestor-only causal mask; [G] "Composants Clés — Vérification": standard tree attention, unchanged.
// Reading: for request b, query head h and tree node i, the keys are the L prefix positions (all visible) and the n
// tree positions L + t with mask[b][i][t] = 1 (its ancestors and itself); grouped-query heads: query head h reads
// key/value head h / (Hq / Hkv). out = softmax_j(scale * q . k_j) v_j over the visible keys, in fp64.
// q [B][n][Hq][d], k and v [B][Hkv][L + n][d] (fp32 or bf16), mask [B][n][n] uint8, out [B][n][Hq][d] fp64.
int orc_tree_attention(int B, int n, int L, int Hq, int Hkv, int d, const void* q, const void* k, const void* v,
                       int dtype, const uint8_t* mask, double scale, double* out, int threads) {
  if (!q || !k || !v || !mask || !out || B < 0 || n < 1 || L < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || d < 1)
    return ORC_ERR_ARG;
  const int G = Hq / Hkv, T = L + n;
#pragma omp parallel for collapse(2) schedule(dynamic) num_threads(threads_or_default(threads))
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hq; ++h) {
      const int kvh = h / G;
      const size_t kv0 = (static_cast<size_t>(b) * Hkv + kvh) * T;
      std::vector<double> sc(static_cast<size_t>(T));
      for (int i = 0; i < n; ++i) {
        const size_t q0 = ((static_cast<size_t>(b) * n + i) * Hq + h) * d;
        double mx = -std::numeric_limits<double>::infinity();
        for (int j = 0; j < T; ++j) {
          const bool visible = j < L || mask[(static_cast<size_t>(b) * n + i) * n + (j - L)] != 0;
          if (!visible) {
            sc[j] = -std::numeric_limits<double>::infinity();
            continue;
          }
          double dot = 0.0;
          for (int e = 0; e < d; ++e) dot += load(q, dtype, q0 + e) * load(k, dtype, (kv0 + j) * d + e);
          sc[j] = scale * dot;
          mx = std::max(mx, sc[j]);
        }
        double den = 0.0;
        for (int j = 0; j < T; ++j) den += std::isinf(sc[j]) && sc[j] < 0 ? 0.0 : std::exp(sc[j] - mx);
        double* o = out + q0;
        for (int e = 0; e < d; ++e) o[e] = 0.0;
        for (int j = 0; j < T; ++j) {
          if (std::isinf(sc[j]) && sc[j] < 0) continue;
          const double w = std::exp(sc[j] - mx) / den;
          for (int e = 0; e < d; ++e) o[e] += w * load(v, dtype, (kv0 + j) * d + e);
        }
      }
    }
  return ORC_OK;
}

int orc_gru_step(int H, int E, int wdtype, const void* w_ih, const void* w_hh, const void* b_ih, const void* b_hh,
                 const double* x, const double* h, double* out) {
  if (!w_ih || !w_hh || !x || !h || !out || H < 1 || E < 1) return ORC_ERR_ARG;
  const Weights w{H, E, wdtype, nullptr, w_ih, w_hh, b_ih, b_hh, nullptr};
  gru_step(w, x, h, out);
  return ORC_OK;
}

int orc_child_logp(int H, int wdtype, const void* w_c, const int32_t* ids, const double* base, int M, double T,
                   const double* h, double* logp) {
  if (!w_c || !ids || !base || !h || !logp || H < 1 || M < 1 || !(T >= 0.0)) return ORC_ERR_ARG;
  const Weights w{H, 0, wdtype, nullptr, nullptr, nullptr, nullptr, nullptr, w_c};
  child_logp(w, ids, base, M, T > 0.0 ? T : 1.0, h, logp);
  return ORC_OK;
}

// Best-first conditional trees for B independent requests. ids/vals are the top-M per position ([B,K,M]),
// h0 is [B,H] (fp64). Outputs: tokens/parents/depth [B,n], scores [B,n], mask [B,n,n], and gaps [B,n] = the popped
// node's score minus the best remaining frontier score at the time of that pop (+inf if the frontier is empty).
int orc_build_trees(int B, int K, int M, int n, int max_depth, double T, const int32_t* ids, const double* vals,
                    const double* h0, int H, int E, int wdtype, const void* emb, const void* w_ih, const void* w_hh,
                    const void* b_ih, const void* b_hh, const void* w_c, int32_t* tokens, int32_t* parents,
                    int32_t* depth, double* scores, uint8_t* mask, double* gaps, int threads) {
  if (!ids || !vals || !h0 || !emb || !w_ih || !w_hh || !w_c || !tokens || !parents || !depth || !scores || !mask ||
      !gaps || B < 0 || K < 1 || M < 1 || n < 1 || max_depth < 1 || max_depth > K || H < 1 || E < 1 || !(T >= 0.0))
    return ORC_ERR_ARG;
  if (tree_size(M, max_depth, n) < n) return ORC_ERR_BUDGET;
  const Weights w{H, E, wdtype, emb, w_ih, w_hh, b_ih, b_hh, w_c};
  int status = ORC_OK;
#pragma omp parallel for schedule(dynamic) num_threads(threads_or_default(threads))
  for (int b = 0; b < B; ++b) {
    const size_t kb = static_cast<size_t>(b) * K * M, nb = static_cast<size_t>(b) * n;
    const int s = build_one(w, ids + kb, vals + kb, M, n, max_depth, T, h0 + static_cast<size_t>(b) * H,
                            tokens + nb, parents + nb, depth + nb, scores + nb, mask + nb * n, gaps + nb);
    if (s != ORC_OK) {
#pragma omp critical
      status = s;
    }
  }
  return status;
}

// Marginal-scored (DDTree) trees of B requests from their top-M candidates; no GRU, no correction.
int orc_build_trees_marginal(int B, int K, int M, int n, int max_depth, double T, const int32_t* ids,
                             const double* vals, int32_t* tokens, int32_t* parents, int32_t* depth, double* scores,
                             uint8_t* mask, double* gaps, int threads) {
  if (!ids || !vals || !tokens || !parents || !depth || !scores || !mask || !gaps || B < 0 || K < 1 || M < 1 ||
      n < 1 || max_depth < 1 || max_depth > K || !(T >= 0.0))
    return ORC_ERR_ARG;
  if (tree_size(M, max_depth, n) < n) return ORC_ERR_BUDGET;
  int status = ORC_OK;
#pragma omp parallel for schedule(dynamic) num_threads(threads_or_default(threads))
  for (int b = 0; b < B; ++b) {
    const size_t kb = static_cast<size_t>(b) * K * M, nb = static_cast<size_t>(b) * n;
    const int s = build_one_marginal(ids + kb, vals + kb, M, n, max_depth, T, tokens + nb, parents + nb, depth + nb,
                                     scores + nb, mask + nb * n, gaps + nb);
    if (s != ORC_OK) {
#pragma omp critical
      status = s;
    }
  }
  return status;
}

// Accepted paths of B verified trees: tokens/parents [B,n], target_next [B,n+1] -> accept_len [B], path [B,n]
// (node indices in path order, then -1), bonus [B].
int orc_accept_paths(int B, int n, const int32_t* tokens, const int32_t* parents, const int32_t* target_next,
                     int32_t* accept_len, int32_t* path, int32_t* bonus) {
  if (!tokens || !parents || !target_next || !accept_len || !path || !bonus || B < 0 || n < 1) return ORC_ERR_ARG;
  for (int b = 0; b < B; ++b) {
    const size_t nb = static_cast<size_t>(b) * n;
    const int s = accept_one(n, tokens + nb, parents + nb, target_next + static_cast<size_t>(b) * (n + 1),
                             accept_len + b, path + nb, bonus + b);
    if (s != ORC_OK) return s;
  }
  return ORC_OK;
}

// Scores of given trees (tokens/parents/depth [B,n], in any valid prefix order), recomputed in fp64.
int orc_rescore(int B, int K, int M, int n, int max_depth, double T, const int32_t* ids, const double* vals,
                const double* h0, int H, int E, int wdtype, const void* emb, const void* w_ih, const void* w_hh,
                const void* b_ih, const void* b_hh, const void* w_c, const int32_t* tokens, const int32_t* parents,
                const int32_t* depth, double* scores, int threads) {
  if (!ids || !vals || !h0 || !emb || !w_ih || !w_hh || !w_c || !tokens || !parents || !depth || !scores || B < 0 ||
      K < 1 || M < 1 || n < 1 || max_depth < 1 || max_depth > K || H < 1 || E < 1 || !(T >= 0.0))
    return ORC_ERR_ARG;
  const Weights w{H, E, wdtype, emb, w_ih, w_hh, b_ih, b_hh, w_c};
  int status = ORC_OK;
#pragma omp parallel for schedule(dynamic) num_threads(threads_or_default(threads))
  for (int b = 0; b < B; ++b) {
    const size_t kb = static_cast<size_t>(b) * K * M, nb = static_cast<size_t>(b) * n;
    const int s = rescore_one(w, ids + kb, vals + kb, M, n, max_depth, T, h0 + static_cast<size_t>(b) * H,
                              tokens + nb, parents + nb, depth + nb, scores + nb);
    if (s != ORC_OK) {
#pragma omp critical
      status = s;
    }
  }
  return status;
}

long long orc_tree_size(int M, int max_depth, long long cap) { return tree_size(M, max_depth, cap); }

}  // extern "C"
