// dt_build_trees_marginal — DDTree's factorised (marginal) scoring on the same best-first builder.
//
// Method: blog.captcha.la, "Methodology — deep read" (DDTree scores tree nodes by factorised marginal
// log-probabilities; DominoTree replaces them with the GRU-corrected conditional ones) and "Key findings" (the
// ablation that swaps only the scoring function: conditional scoring gains +9.2% throughput); zhichai.top,
// "两条路线的困境" (DDTree's factorised scoring); gist.science, "Énoncé du Problème" (a token's score depends only on
// its position, not on the path that reached it).
//
// A node's children at block position d score parent + log-softmax over the M candidates of (base logits / T_eff):
// no hidden state, no correction, so no request depends on another and nothing crosses SMs. One CTA per request
// keeps the request's best-first state in shared memory for the whole launch and runs the same lookahead waves as
// the conditional builders: the children lists of the wave's expansions (one warp per expansion: restricted
// log-softmax, then the siblings ranked by 64-bit keys), then one warp pops and picks (request_step). The per-node
// arithmetic is the conditional builders' with a zero correction, so the trees equal theirs at W_c = 0 bit for bit.
#include <cuda_runtime.h>
#include <math.h>

#include "build_common.cuh"

namespace dt {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct MargSmem {
  size_t state, kraw, keys, bytes;
  int batch;  // expansions whose children are computed together
};
__host__ __device__ inline MargSmem marg_smem(int n, int M, int kla, size_t budget) {
  MargSmem S{};
  const int X = expansion_slots(n), KM = M < n ? M : n;
  S.state = 0;
  const size_t st = req_layout(n, X, KM, kla).bytes;
  const size_t per_job = (sizeof(Node) + sizeof(unsigned long long)) * static_cast<size_t>(M);
  int batch = kla < kWarps ? kla : kWarps;
  while (batch > 1 && st + per_job * batch > budget) --batch;
  S.batch = batch;
  S.kraw = st;
  S.keys = st + sizeof(Node) * static_cast<size_t>(M) * batch;
  S.bytes = S.keys + sizeof(unsigned long long) * static_cast<size_t>(M) * batch;
  return S;
}

__global__ void __launch_bounds__(kThreads, 1) marginal_builder(Params p, MargSmem S) {
  extern __shared__ float4 smem_f4[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(smem_f4);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int b = blockIdx.x, M = p.M, n = p.n, K = p.K, X = p.xslots, KM = M < n ? M : n, kla = p.lookahead;
  const ReqLayout RL = req_layout(n, X, KM, kla);
  const ReqView R = req_view(smem + S.state, RL);
  Job* jobs = reinterpret_cast<Job*>(smem + S.state + RL.jobs);
  Node* kraw = reinterpret_cast<Node*>(smem + S.kraw);                            // [batch][M]
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem + S.keys);  // [batch][M]

  // the root is expanded in the first wave; its children take insertion indices 0 .. M - 1
  if (t == 0) {
    *R.ctl = ReqCtl{0, 0, M, 1, 1, {0, 0, 0}};
    jobs[0] = Job{b, 0, -1, 0, 0, 0.f, {0, 0}};
  }
  if (t < 32) R.lanes[t] = t == 0 ? LaneSrc{-2, 0, 0, 0, -1, {0, 0, 0}} : t == 1 ? LaneSrc{0, 0, -1, 0, 1, {0, 0, 0}} : LaneSrc{-1, 0, 0, 0, -1, {0, 0, 0}};
  for (int i = t; i < X; i += kThreads) {
    R.kcount[i] = 0;
    R.popidx[i] = i == 0 ? -1 : -2;
    R.sdepth[i] = 0;
  }
  for (int i = t; i < n; i += kThreads) R.pops[i] = PopRec{0, 0, 0, -INFINITY};
  __syncthreads();

  for (int w = 0; w < X; ++w) {
    const ReqCtl st0 = *R.ctl;
    if (st0.s >= n || st0.njobs == 0) break;
    for (int q0 = 0; q0 < st0.njobs; q0 += S.batch) {
      const int nq = min(S.batch, st0.njobs - q0);
      // one warp per expansion: the restricted log-softmax of its block position's candidates, its children
      if (warp < nq) {
        const Job jb = jobs[q0 + warp];
        const size_t pos = (static_cast<size_t>(b) * K + jb.depth) * M;
        float mx = -INFINITY;
        for (int m = lane; m < M; m += 32) mx = fmaxf(mx, __ldg(p.vals + pos + m) / p.T_eff);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        float sum = 0.f;
        for (int m = lane; m < M; m += 32) sum += expf(__ldg(p.vals + pos + m) / p.T_eff - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        const float lse = logf(sum);
        for (int m = lane; m < M; m += 32) {
          Node e;
          e.score = jb.score + ((__ldg(p.vals + pos + m) / p.T_eff - mx) - lse);
          e.token = valid_id(p, __ldg(p.ids + pos + m));
          e.seq = m;  // the candidate index until the node is popped
          e.pslot = static_cast<short>(jb.xslot);
          e.xslot = -1;
          kraw[warp * M + m] = e;
          keys[warp * M + m] = (static_cast<unsigned long long>(key_of_f32(__float_as_uint(e.score))) << 32) |
                               static_cast<unsigned long long>(~static_cast<uint32_t>(e.token));
        }
      }
      __syncthreads();
      // siblings ranked (score, then token, then candidate index); the first kc kept: at most n - s - 1 can still
      // be popped after the node itself (n for the root's children)
      for (int i = t; i < nq * M; i += kThreads) {
        const int q = i / M, mi = i % M;
        const Job jb = jobs[q0 + q];
        const unsigned long long ki = keys[i];
        const unsigned long long* sib = keys + q * M;
        int r = 0;
#pragma unroll 8
        for (int c = 0; c < M; ++c) {
          const unsigned long long kk = sib[c];
          r += (kk > ki) | ((kk == ki) & (c < mi));
        }
        const int kc = min(KM, jb.pslot < 0 ? n : n - st0.s - 1);
        if (r < kc) R.kids[static_cast<size_t>(jb.xslot) * KM + r] = kraw[i];
        if (mi == 0) R.kcount[jb.xslot] = kc;
      }
      __syncthreads();
    }
    if (warp == 0) request_step(R, b, n, M, p.max_depth, X, KM, kla, jobs, p.hdr);
    __syncthreads();
  }

  // outputs, and each node's ancestor-mask row by walking its parent chain
  resolve_parents(R.pops, R.popidx, n, t, kThreads);
  __syncthreads();
  const size_t o = static_cast<size_t>(b) * n;
  for (int i = t; i < n; i += kThreads) {
    const PopRec r = R.pops[i];
    p.tokens[o + i] = r.token;
    p.parents[o + i] = r.parent;
    p.depth[o + i] = r.depth;
    p.scores[o + i] = r.score;
  }
  for (int i = t; i < n * n; i += kThreads) {
    const int row = i / n, c = i % n;
    int a = row;
    for (int hops = 0; a > c && hops < n; ++hops) a = R.pops[a].parent;  // parents precede their children
    p.mask[(o + row) * n + c] = a == c;
  }
}

}  // namespace
}  // namespace dt

extern "C" dt_status dt_build_trees_marginal(int B, int K, int V, int M, int n, int max_depth, float T,
                                             const int32_t* topm_ids, const float* topm_vals, int32_t* out_tokens,
                                             int32_t* out_parents, int32_t* out_depth, float* out_scores,
                                             uint8_t* out_mask, void* workspace, size_t workspace_bytes,
                                             cudaStream_t stream) {
  using namespace dt;
  if (B < 0 || K < 1 || V < 1 || M < 1 || M > V || n < 1 || max_depth < 1 || max_depth > K) return DT_ERR_INVALID_ARG;
  if (!(T >= 0.0f) || !isfinite(T)) return DT_ERR_INVALID_ARG;
  {  // n must not exceed the number of nodes of the depth-limited M-ary tree
    long long total = 0, level = 1;
    for (int d = 1; d <= max_depth && total < n; ++d) {
      level = level > n ? level : level * M;
      total += level;
    }
    if (total < n) return DT_ERR_INVALID_ARG;
  }
  if (M > DT_MAX_M || n > DT_MAX_N) return DT_ERR_UNSUPPORTED;
  if (B == 0) return DT_OK;
  const void* ptrs[] = {topm_ids, topm_vals, out_tokens, out_parents, out_depth, out_scores, out_mask, workspace};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return DT_ERR_INVALID_ARG;
  if (workspace_bytes < sizeof(WsHeader)) return DT_ERR_INVALID_ARG;
  DeviceInfo di{};
  if (current_device_info(&di) != cudaSuccess) return DT_ERR_CUDA;
  Params p{};
  p.B = B; p.K = K; p.V = V; p.M = M; p.n = n; p.max_depth = max_depth;
  p.T_eff = T > 0.f ? T : 1.f;
  p.ids = topm_ids; p.vals = topm_vals;
  p.tokens = out_tokens; p.parents = out_parents; p.depth = out_depth; p.scores = out_scores; p.mask = out_mask;
  p.hdr = static_cast<WsHeader*>(workspace);
  p.xslots = expansion_slots(n);
  const int k = lookahead_setting();
  p.lookahead = k > 0 ? (k < kLargeLookahead ? k : kLargeLookahead) : kLargeLookahead;
  const size_t budget = static_cast<size_t>(di.optin) - 1024;  // static shared memory is a few bytes
  const MargSmem S = marg_smem(n, M, p.lookahead, budget);
  if (S.bytes > budget) return DT_ERR_UNSUPPORTED;
  const void* fn = reinterpret_cast<const void*>(marginal_builder);
  if (ensure_dynamic_smem(fn, S.bytes) != cudaSuccess) return DT_ERR_CUDA;
  void* args[] = {&p, const_cast<MargSmem*>(&S)};
  return cuda_status(cudaLaunchKernel(fn, dim3(static_cast<unsigned>(B)), dim3(kThreads), args, S.bytes, stream));
}
