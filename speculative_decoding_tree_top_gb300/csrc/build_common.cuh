// Pieces shared by the two tree-builder kernels of libdominotree (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <math.h>

#include "dt_internal.cuh"

namespace dt {

constexpr int kSmallMaxB = 8;  // batches up to this size use the all-SM, one-barrier-per-step builder

struct alignas(16) Entry {  // a frontier node; 16 bytes
  float score;
  int token;
  short parent;  // index of the parent among the popped nodes, -1 for a child of the root
  short depth;
  int seq;       // insertion order
};

// Pop order: higher score, then lower token id, then earlier insertion (branch-free).
__device__ __forceinline__ bool before(const Entry& a, const Entry& b) {
  const bool seq_first = a.seq < b.seq;
  const bool tok_first = (a.token < b.token) | ((a.token == b.token) & seq_first);
  return (a.score > b.score) | ((a.score == b.score) & tok_first);
}

struct NodeState {  // the node popped last by a request, as phase A of the next step needs it
  int token;
  int parent;
  int depth;
  int expand;  // 1 if the node is expanded in the next step
  float score;
  int seq_next;
  int fcount;  // entries in the request's frontier
  int pad;
};

struct Params {
  int B, K, V, M, n, max_depth, H, E;
  float T_eff;
  bool bf16;
  const int32_t* ids;
  const float* vals;
  const float* h0;
  const void* emb;
  const void* w_ih;
  const void* w_hh;
  const void* b_ih;
  const void* b_hh;
  const void* w_c;
  int32_t* tokens;
  int32_t* parents;
  int32_t* depth;
  float* scores;
  uint8_t* mask;
  WsHeader* hdr;
  NodeState* state;
  Entry* frontier;  // [B][n]
  float* hs;        // [B][n][H]
  long long* acc;   // [n][B][M] fixed-point correction accumulators, acc_stride words apart (small-batch builder)
  int acc_stride;
  uint64_t timeout_ns;
  bool rows_smem;   // large-batch builder: the M gathered correction rows of a node are staged in shared memory
};

__device__ __forceinline__ float ldw(const void* p, bool bf16, size_t i) {
  if (bf16) {
    const unsigned short u = __ldg(static_cast<const unsigned short*>(p) + i);
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
  }
  return __ldg(static_cast<const float*>(p) + i);
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

// Candidate ids come from the caller (normally dt_topm); one outside [0, V) is recorded as DT_ERR_INVALID_ARG and
// replaced by 0, so that no gather ever leaves the weight arrays.
__device__ __forceinline__ int valid_id(const Params& p, int id) {
  if (static_cast<unsigned>(id) >= static_cast<unsigned>(p.V)) {
    record_error(p.hdr, DT_ERR_INVALID_ARG);
    return 0;
  }
  return id;
}

// Keeps the first R entries, in pop order, of the union of a request's frontier and a node's new children:
// cand[0, F) is the frontier, already in pop order (it was written that way), cand[F, F + C) the children in any
// order. The children are ranked among themselves by counting (tpe threads per child), then every entry's place in
// the union is its place in its own list plus a binary search in the other one: O((F + C) log) instead of counting
// every pair. `before` is a strict total order, so the places are distinct. sc[0, C) is scratch; sorted[0, R) the
// result. Called by the whole block (kThreads threads); ends synchronised.
template <int kThreads>
__device__ void merge_rank(const Entry* cand, int F, int C, int R, Entry* sc, Entry* sorted) {
  const int t = threadIdx.x;
  int tpe = 1;
  while (tpe < 32 && tpe * 2 * C <= kThreads) tpe *= 2;
  for (int base = 0; base < C * tpe; base += kThreads) {  // uniform bounds: every lane reaches the shuffles
    const int slot = base + t, i = slot / tpe, part = slot % tpe;
    int r = 0;
    Entry ei{};
    if (i < C) {
      ei = cand[F + i];
#pragma unroll 4
      for (int q = part; q < C; q += tpe) r += before(cand[F + q], ei);
    }
    for (int o = 1; o < tpe; o <<= 1) r += __shfl_xor_sync(0xFFFFFFFFu, r, o);
    if (i < C && part == 0) sc[r] = ei;
  }
  __syncthreads();
  for (int k = t; k < F + C; k += kThreads) {
    const bool old = k < F;
    const Entry e = old ? cand[k] : sc[k - F];
    const Entry* other = old ? sc : cand;
    int lo = 0, hi = old ? C : F;  // entries of the other list that come before e
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (before(other[mid], e)) lo = mid + 1;
      else hi = mid;
    }
    const int r = (old ? k : k - F) + lo;
    if (r < R) sorted[r] = e;
  }
  __syncthreads();
}

// One warp: the dot products of 8 consecutive rows m0 .. m0 + 7 (those < M) with h, for the rows of a gathered slice
// in shared memory (`rows`, [M][H]) or, when rows == nullptr, the correction rows w[ids[m]] in global memory. The
// lane's share of h is loaded once and used for all 8 rows, whose sums are 8 independent chains (same per-lane order
// and shuffle tree as one row at a time, so the results are identical). out[j] is valid in every lane.
__device__ __forceinline__ void warp_dot_rows8(const void* rows, const void* w, const int* ids, bool bf16, int m0,
                                               int M, const float* h, int H, float (&out)[8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 8; ++j) out[j] = 0.f;
  if (bf16) {
    const int G = H / 8;  // 16-byte groups per row
    for (int g = lane; g < G; g += 32) {
      const float4 ha = *reinterpret_cast<const float4*>(h + g * 8), hb = *reinterpret_cast<const float4*>(h + g * 8 + 4);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int m = m0 + j;
        if (m >= M) break;
        const uint4 v = rows ? reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(rows) +
                                                              static_cast<size_t>(m) * H)[g]
                             : __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(w) +
                                                                    static_cast<size_t>(ids[m]) * H) + g);
        float a = out[j];
        a = fmaf(__uint_as_float(v.x << 16), ha.x, a);
        a = fmaf(__uint_as_float(v.x & 0xFFFF0000u), ha.y, a);
        a = fmaf(__uint_as_float(v.y << 16), ha.z, a);
        a = fmaf(__uint_as_float(v.y & 0xFFFF0000u), ha.w, a);
        a = fmaf(__uint_as_float(v.z << 16), hb.x, a);
        a = fmaf(__uint_as_float(v.z & 0xFFFF0000u), hb.y, a);
        a = fmaf(__uint_as_float(v.w << 16), hb.z, a);
        a = fmaf(__uint_as_float(v.w & 0xFFFF0000u), hb.w, a);
        out[j] = a;
      }
    }
  } else {
    const int G = H / 4;
    for (int g = lane; g < G; g += 32) {
      const float4 hv = *reinterpret_cast<const float4*>(h + g * 4);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int m = m0 + j;
        if (m >= M) break;
        const float4 v = rows ? reinterpret_cast<const float4*>(static_cast<const float*>(rows) +
                                                                static_cast<size_t>(m) * H)[g]
                              : __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(w) +
                                                                      static_cast<size_t>(ids[m]) * H) + g);
        float a = out[j];
        a = fmaf(v.x, hv.x, a);
        a = fmaf(v.y, hv.y, a);
        a = fmaf(v.z, hv.z, a);
        a = fmaf(v.w, hv.w, a);
        out[j] = a;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int j = 0; j < 8; ++j) out[j] += __shfl_xor_sync(0xFFFFFFFFu, out[j], o);
}

// Builder region of the workspace, after the top-M region (one workspace serves the whole round): per-request
// last-pop state, pruned frontiers [B][n], hidden states [B][n][H] fp32, and for small batches the per-step
// fixed-point correction accumulators [n][B][M] int64 and the hidden-state publication counters [B][n].
struct BuildLayout {
  size_t state, frontier, hs, acc, bytes;
};

// Words between two correction accumulators: one 128-byte line each, so that the shares of a step (every SM adds
// one to every candidate's slot) spread over the L2 slices, unless that takes more than 64 MB.
__host__ __device__ inline int acc_stride(int B, int M, int n) {
  return static_cast<size_t>(n) * B * M * 128u <= (64u << 20) ? 16 : 1;
}

inline BuildLayout build_layout(int B, int K, int V, int M, int n, int H) {
  BuildLayout L{};
  L.state = topm_layout(B, K, V, M).bytes;
  L.frontier = align_up(L.state + sizeof(NodeState) * static_cast<size_t>(B));
  L.hs = align_up(L.frontier + sizeof(Entry) * static_cast<size_t>(B) * n);
  L.acc = align_up(L.hs + sizeof(float) * static_cast<size_t>(B) * n * H);
  // per-step per-candidate accumulators [n][B][M] int64 (acc_stride words apart), then per-node publication
  // counters [B][n] int32
  const size_t acc_bytes =
      B <= kSmallMaxB ? sizeof(long long) * (static_cast<size_t>(n) * B * M * acc_stride(B, M, n) +
                                             (static_cast<size_t>(B) * n + 1) / 2)
                      : 0;
  L.bytes = align_up(L.acc + acc_bytes);
  return L;
}


// The small-batch builder (build_small.cu). Returns false when its shared-memory plan does not fit this device
// (the caller then uses the general builder).
bool small_builder_fits(const Params& p, int sms);
cudaError_t launch_small_builder(const Params& p, cudaStream_t stream);

}  // namespace dt
