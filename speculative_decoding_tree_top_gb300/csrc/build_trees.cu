// dt_build_trees — conditional best-first draft trees (one persistent cooperative launch per round).
//
// Method: blog.captcha.la, "Methodology — deep read" (DDTree's best-first max-priority queue keyed by cumulative
// conditional log-probability; the GRU state is carried along each root-to-node path; the correction is applied to
// the gathered top-M rows only; fixed node budget / max depth; prefix-closed tree + ancestor-only mask);
// gist.science, "Composants Clés" (only the light GRU correction and correction head are recomputed per node).
//
// GB300 design. The pages' builder replays a CUDA graph per node while a host-side heap decides the next pop
// (gist.science, "Constructeur Natif GPU"); here the whole round is one launch with no host round-trip:
//   * all B requests advance in lockstep: step s pops the s-th node of every request;
//   * phase A (all CTAs): the GRU step of the nodes popped in the previous step, as tiles of
//     [16 requests x 16 hidden units] over K = E (embedding row) then K = H (parent state), fp32 accumulation;
//   * grid barrier;
//   * phase B (one CTA per request): gather the M correction rows of the node's block position and dot them with
//     h (one warp per row), restricted log-softmax (warp reductions), merge the children into the request's
//     frontier keeping only the n - s entries that can still be popped, pop the best, write the node's output row
//     and its ancestor-mask row;
//   * grid barrier; next step.
// Every reduction has a fixed order (no floating-point atomics), so the output is bit-identical run to run.
#include <cuda_runtime.h>
#include <math.h>

#include "build_common.cuh"

namespace dt {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTB = 16;   // requests per GRU tile
constexpr int kTU = 16;   // hidden units per GRU tile
constexpr int kKC = 64;   // K-chunk of the GRU tile
constexpr int kPad = kKC + 1;

// ---- phase A: GRU step of every request whose last pop is expanded --------------------------------------------
__device__ void gru_phase(const Params& p, int node, float* smem) {
  float* xs = smem;                  // [kTB][kPad]
  float* ws = smem + kTB * kPad;     // [3][kTU][kPad]
  __shared__ int s_tok[kTB], s_par[kTB], s_exp[kTB];
  const int t = threadIdx.x, lb = t / kTU, lu = t % kTU;
  const int ublocks = (p.H + kTU - 1) / kTU;
  const int rblocks = (p.B + kTB - 1) / kTB;
  const int tiles = ublocks * rblocks;
  for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int rb = tile / ublocks, ub = tile % ublocks;
    __syncthreads();
    if (t < kTB) {
      const int b = rb * kTB + t;
      const bool ok = b < p.B && p.state[b].expand;
      s_exp[t] = ok;
      s_tok[t] = ok ? p.state[b].token : 0;
      s_par[t] = ok ? p.state[b].parent : -1;
    }
    __syncthreads();
    if (!__syncthreads_or(t < kTB && s_exp[t])) continue;
    const int b = rb * kTB + lb, k = ub * kTU + lu;
    float acc_r = 0.f, acc_u = 0.f, acc_ni = 0.f, acc_nh = 0.f;
    // input side: W_ih[gate rows] . emb[token]
    for (int e0 = 0; e0 < p.E; e0 += kKC) {
      for (int i = t; i < kTB * kKC; i += kThreads) {
        const int r = i / kKC, c = i % kKC, e = e0 + c;
        xs[r * kPad + c] = (s_exp[r] && e < p.E) ? ldw(p.emb, p.bf16, static_cast<size_t>(s_tok[r]) * p.E + e) : 0.f;
      }
      for (int i = t; i < 3 * kTU * kKC; i += kThreads) {
        const int g = i / (kTU * kKC), u = (i / kKC) % kTU, c = i % kKC, e = e0 + c, kk = ub * kTU + u;
        ws[(g * kTU + u) * kPad + c] =
            (kk < p.H && e < p.E) ? ldw(p.w_ih, p.bf16, (static_cast<size_t>(g) * p.H + kk) * p.E + e) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int c = 0; c < kKC; ++c) {
        const float x = xs[lb * kPad + c];
        acc_r = fmaf(ws[(0 * kTU + lu) * kPad + c], x, acc_r);
        acc_u = fmaf(ws[(1 * kTU + lu) * kPad + c], x, acc_u);
        acc_ni = fmaf(ws[(2 * kTU + lu) * kPad + c], x, acc_ni);
      }
      __syncthreads();
    }
    // hidden side: W_hh[gate rows] . h_parent
    for (int j0 = 0; j0 < p.H; j0 += kKC) {
      for (int i = t; i < kTB * kKC; i += kThreads) {
        const int r = i / kKC, c = i % kKC, j = j0 + c;
        float v = 0.f;
        if (s_exp[r] && j < p.H) {
          const int bb = rb * kTB + r, par = s_par[r];
          const float* hp = par < 0 ? p.h0 + static_cast<size_t>(bb) * p.H
                                    : p.hs + (static_cast<size_t>(bb) * p.n + par) * p.H;
          v = par < 0 ? __ldg(hp + j) : hp[j];
        }
        xs[r * kPad + c] = v;
      }
      for (int i = t; i < 3 * kTU * kKC; i += kThreads) {
        const int g = i / (kTU * kKC), u = (i / kKC) % kTU, c = i % kKC, j = j0 + c, kk = ub * kTU + u;
        ws[(g * kTU + u) * kPad + c] =
            (kk < p.H && j < p.H) ? ldw(p.w_hh, p.bf16, (static_cast<size_t>(g) * p.H + kk) * p.H + j) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int c = 0; c < kKC; ++c) {
        const float x = xs[lb * kPad + c];
        acc_r = fmaf(ws[(0 * kTU + lu) * kPad + c], x, acc_r);
        acc_u = fmaf(ws[(1 * kTU + lu) * kPad + c], x, acc_u);
        acc_nh = fmaf(ws[(2 * kTU + lu) * kPad + c], x, acc_nh);
      }
      __syncthreads();
    }
    if (b < p.B && k < p.H && s_exp[lb]) {
      const size_t g0 = k, g1 = static_cast<size_t>(p.H) + k, g2 = 2 * static_cast<size_t>(p.H) + k;
      const float bir = p.b_ih ? ldw(p.b_ih, p.bf16, g0) : 0.f, bhr = p.b_hh ? ldw(p.b_hh, p.bf16, g0) : 0.f;
      const float biu = p.b_ih ? ldw(p.b_ih, p.bf16, g1) : 0.f, bhu = p.b_hh ? ldw(p.b_hh, p.bf16, g1) : 0.f;
      const float bin = p.b_ih ? ldw(p.b_ih, p.bf16, g2) : 0.f, bhn = p.b_hh ? ldw(p.b_hh, p.bf16, g2) : 0.f;
      const float r = sigmoidf_(acc_r + bir + bhr);
      const float u = sigmoidf_(acc_u + biu + bhu);
      const float g = tanhf((acc_ni + bin) + r * (acc_nh + bhn));
      const int par = s_par[lb];
      const float hprev = par < 0 ? __ldg(p.h0 + static_cast<size_t>(b) * p.H + k)
                                  : p.hs[(static_cast<size_t>(b) * p.n + par) * p.H + k];
      p.hs[(static_cast<size_t>(b) * p.n + node) * p.H + k] = (1.f - u) * g + u * hprev;
    }
  }
}

// ---- phase B: expand, merge, pop (one CTA per request) ----------------------------------------------------------
__device__ void frontier_phase(const Params& p, int s, float* smem) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int M = p.M, n = p.n, H = p.H;
  float* h = smem;                                          // [H]
  float* z = h + H;                                         // [M]
  Entry* cand = reinterpret_cast<Entry*>(z + ((M + 3) & ~3));  // [n + M]
  Entry* sorted = cand + (n + M);                           // [n + M]
  __shared__ float s_red[2];
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    __syncthreads();
    NodeState st;
    bool expand;
    int node_depth, parent_idx;
    float node_score;
    const float* hsrc;
    if (s == 0) {
      expand = true;
      node_depth = 0;
      parent_idx = -1;
      node_score = 0.f;
      hsrc = p.h0 + static_cast<size_t>(b) * H;
      st.seq_next = 0;
      st.fcount = 0;
    } else {
      st = p.state[b];
      expand = st.expand != 0;
      node_depth = st.depth;
      parent_idx = s - 1;
      node_score = st.score;
      hsrc = p.hs + (static_cast<size_t>(b) * n + (s - 1)) * H;
    }
    const int F = st.fcount;
    const int C = expand ? M : 0;
    Entry* fr = p.frontier + static_cast<size_t>(b) * n;
    for (int i = t; i < F; i += kThreads) cand[i] = fr[i];
    if (expand) {
      for (int k = t; k < H; k += kThreads) h[k] = (s == 0) ? __ldg(hsrc + k) : hsrc[k];
      __syncthreads();
      const size_t pos = (static_cast<size_t>(b) * p.K + node_depth) * M;
      for (int m = warp; m < M; m += kWarps) {
        const int id = valid_id(p, __ldg(p.ids + pos + m));
        const float d = warp_row_dot(p.w_c, p.bf16, id, h, H);
        if (lane == 0) z[m] = (__ldg(p.vals + pos + m) + d) / p.T_eff;
      }
      __syncthreads();
      if (warp == 0) {
        float mx = -INFINITY;
        for (int m = lane; m < M; m += 32) mx = fmaxf(mx, z[m]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        float sum = 0.f;
        for (int m = lane; m < M; m += 32) sum += expf(z[m] - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        if (lane == 0) {
          s_red[0] = mx;
          s_red[1] = logf(sum);
        }
      }
      __syncthreads();
      const float mx = s_red[0], lse = s_red[1];
      for (int m = t; m < M; m += kThreads) {
        Entry e;
        e.score = node_score + ((z[m] - mx) - lse);
        e.token = valid_id(p, __ldg(p.ids + pos + m));
        e.parent = static_cast<short>(parent_idx);
        e.depth = static_cast<short>(node_depth + 1);
        e.seq = st.seq_next + m;
        cand[F + m] = e;
      }
    }
    __syncthreads();
    // Keep the R = n - s best: nothing ranked below them can be popped in the n - s pops left.
    const int N = F + C;
    const int R = min(n - s, N);
    for (int i = t; i < N; i += kThreads) {
      const Entry ei = cand[i];
      int r = 0;
      for (int j = 0; j < N; ++j) r += before(cand[j], ei);
      if (r < R) sorted[r] = ei;
    }
    __syncthreads();
    const Entry pop = sorted[0];
    for (int i = t + 1; i < R; i += kThreads) fr[i - 1] = sorted[i];
    const size_t o = static_cast<size_t>(b) * n + s;
    uint8_t* mrow = p.mask + o * n;
    const uint8_t* prow = pop.parent >= 0 ? p.mask + (static_cast<size_t>(b) * n + pop.parent) * n : nullptr;
    for (int j = t; j < n; j += kThreads) mrow[j] = (j == s) ? 1 : ((j < s && prow) ? prow[j] : 0);
    if (t == 0) {
      p.tokens[o] = pop.token;
      p.parents[o] = pop.parent;
      p.depth[o] = pop.depth;
      p.scores[o] = pop.score;
      NodeState ns;
      ns.token = pop.token;
      ns.parent = pop.parent;
      ns.depth = pop.depth;
      ns.expand = (s + 1 < n) && (pop.depth < p.max_depth);
      ns.score = pop.score;
      ns.seq_next = st.seq_next + C;
      ns.fcount = R - 1;
      ns.pad = 0;
      p.state[b] = ns;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) build_kernel(Params p) {
  extern __shared__ float4 smem_f4[];
  float* smem = reinterpret_cast<float*>(smem_f4);
  __shared__ int s_flag;
  const unsigned G = gridDim.x;
  for (int s = 0; s < p.n; ++s) {
    if (s > 0) {
      gru_phase(p, s - 1, smem);
      if (!grid_barrier(p.hdr, G, p.timeout_ns, &s_flag)) return;
    }
    frontier_phase(p, s, smem);
    if (s + 1 < p.n && !grid_barrier(p.hdr, G, p.timeout_ns, &s_flag)) return;
  }
}

size_t smem_bytes(int M, int n, int H) {
  const size_t a = sizeof(float) * (kTB * kPad + 3 * kTU * kPad);
  const size_t b = sizeof(float) * (H + ((M + 3) & ~3)) + 2 * sizeof(Entry) * static_cast<size_t>(n + M);
  return a > b ? a : b;
}

}  // namespace
}  // namespace dt

extern "C" size_t dt_build_workspace_bytes(int B, int K, int V, int M, int n, int H, int E) {
  (void)E;
  if (B < 0 || K < 1 || V < 1 || M < 1 || n < 1 || H < 1) return 0;
  return dt::build_layout(B, K, V, M, n, H).bytes;
}

extern "C" dt_status dt_build_trees(int B, int K, int V, int M, int n, int max_depth, float T,
                                    const int32_t* topm_ids, const float* topm_vals, const float* h0,
                                    const dt_weights* w, int32_t* out_tokens, int32_t* out_parents,
                                    int32_t* out_depth, float* out_scores, uint8_t* out_mask, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream) {
  using namespace dt;
  if (!w) return DT_ERR_INVALID_ARG;
  const int H = w->H, E = w->E;
  if (B < 0 || K < 1 || V < 1 || M < 1 || M > V || n < 1 || max_depth < 1 || max_depth > K) return DT_ERR_INVALID_ARG;
  if (!(T >= 0.0f) || !isfinite(T)) return DT_ERR_INVALID_ARG;
  if (H < 1 || E < 1 || H % 8 || E % 8) return DT_ERR_INVALID_ARG;
  if (w->dtype != DT_F32 && w->dtype != DT_BF16) return DT_ERR_INVALID_ARG;
  {  // n must not exceed the number of nodes of the depth-limited M-ary tree
    long long total = 0, level = 1;
    for (int d = 1; d <= max_depth && total < n; ++d) {
      level = level > n ? level : level * M;
      total += level;
    }
    if (total < n) return DT_ERR_INVALID_ARG;
  }
  if (M > DT_MAX_M || n > DT_MAX_N || H > DT_MAX_H || E > DT_MAX_E) return DT_ERR_UNSUPPORTED;
  if (B == 0) return DT_OK;  // nothing to read or write
  const void* ptrs[] = {topm_ids, topm_vals, h0, w->emb, w->w_ih, w->w_hh, w->w_c, out_tokens, out_parents,
                        out_depth, out_scores, out_mask, workspace};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return DT_ERR_INVALID_ARG;
  if ((w->b_ih && !aligned16(w->b_ih)) || (w->b_hh && !aligned16(w->b_hh))) return DT_ERR_INVALID_ARG;
  const BuildLayout L = build_layout(B, K, V, M, n, H);
  if (workspace_bytes < L.bytes) return DT_ERR_INVALID_ARG;

  char* ws = static_cast<char*>(workspace);
  Params p{};
  p.B = B; p.K = K; p.V = V; p.M = M; p.n = n; p.max_depth = max_depth; p.H = H; p.E = E;
  p.T_eff = T > 0.f ? T : 1.f;
  p.bf16 = w->dtype == DT_BF16;
  p.ids = topm_ids; p.vals = topm_vals; p.h0 = h0;
  p.emb = w->emb; p.w_ih = w->w_ih; p.w_hh = w->w_hh; p.b_ih = w->b_ih; p.b_hh = w->b_hh; p.w_c = w->w_c;
  p.tokens = out_tokens; p.parents = out_parents; p.depth = out_depth; p.scores = out_scores; p.mask = out_mask;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.state = reinterpret_cast<NodeState*>(ws + L.state);
  p.frontier = reinterpret_cast<Entry*>(ws + L.frontier);
  p.hs = reinterpret_cast<float*>(ws + L.hs);
  p.acc = B <= kSmallMaxB ? reinterpret_cast<long long*>(ws + L.acc) : nullptr;
  p.timeout_ns = barrier_timeout_ns();

  const size_t smem = smem_bytes(M, n, H);
  int dev = 0, sms = 0, coop = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (e != cudaSuccess) return DT_ERR_CUDA;
  if (!coop) return DT_ERR_UNSUPPORTED;
  if (small_builder_fits(p, sms)) return cuda_status(launch_small_builder(p, stream));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, build_kernel, kThreads, smem);
  if (e != cudaSuccess) return DT_ERR_CUDA;
  if (!coop || per_sm < 1) return DT_ERR_UNSUPPORTED;
  const unsigned grid = static_cast<unsigned>(sms);  // one CTA per SM; co-resident under a cooperative launch
  void* args[] = {&p};
  e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(build_kernel), dim3(grid), dim3(kThreads), args, smem,
                                  stream);
  return cuda_status(e);
}
