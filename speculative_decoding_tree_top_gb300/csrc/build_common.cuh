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
  long long* acc;   // [n][B][M] fixed-point correction accumulators (small-batch builder)
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

// One warp: w_c[row] . h (h in shared memory), lanes over 16-byte groups, fixed-order shuffle reduction.
__device__ __forceinline__ float warp_row_dot(const void* w, bool bf16, int row, const float* h, int H) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  if (bf16) {
    const uint4* r = reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(w) + static_cast<size_t>(row) * H);
    for (int g = lane; g < H / 8; g += 32) {
      const uint4 v = __ldg(r + g);
      const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(__uint_as_float(q[e] << 16), h[g * 8 + 2 * e], acc);
        acc = fmaf(__uint_as_float(q[e] & 0xFFFF0000u), h[g * 8 + 2 * e + 1], acc);
      }
    }
  } else {
    const float4* r = reinterpret_cast<const float4*>(static_cast<const float*>(w) + static_cast<size_t>(row) * H);
    for (int g = lane; g < H / 4; g += 32) {
      const float4 v = __ldg(r + g);
      acc = fmaf(v.x, h[g * 4 + 0], acc);
      acc = fmaf(v.y, h[g * 4 + 1], acc);
      acc = fmaf(v.z, h[g * 4 + 2], acc);
      acc = fmaf(v.w, h[g * 4 + 3], acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  return acc;
}

// The same dot product with the row in shared memory (plain loads: ld.global.nc does not apply to shared memory).
__device__ __forceinline__ float warp_row_dot_shared(const void* rows, bool bf16, int row, const float* h, int H) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  if (bf16) {
    const uint4* r = reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(rows) + static_cast<size_t>(row) * H);
    for (int g = lane; g < H / 8; g += 32) {
      const uint4 v = r[g];
      const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(__uint_as_float(q[e] << 16), h[g * 8 + 2 * e], acc);
        acc = fmaf(__uint_as_float(q[e] & 0xFFFF0000u), h[g * 8 + 2 * e + 1], acc);
      }
    }
  } else {
    const float4* r = reinterpret_cast<const float4*>(static_cast<const float*>(rows) + static_cast<size_t>(row) * H);
    for (int g = lane; g < H / 4; g += 32) {
      const float4 v = r[g];
      acc = fmaf(v.x, h[g * 4 + 0], acc);
      acc = fmaf(v.y, h[g * 4 + 1], acc);
      acc = fmaf(v.z, h[g * 4 + 2], acc);
      acc = fmaf(v.w, h[g * 4 + 3], acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  return acc;
}

// Builder region of the workspace, after the top-M region (one workspace serves the whole round): per-request
// last-pop state, pruned frontiers [B][n], hidden states [B][n][H] fp32, and for small batches the per-step
// fixed-point correction accumulators [n][B][M] int64 and the hidden-state publication counters [B][n].
struct BuildLayout {
  size_t state, frontier, hs, acc, bytes;
};

inline BuildLayout build_layout(int B, int K, int V, int M, int n, int H) {
  BuildLayout L{};
  L.state = topm_layout(B, K, V, M).bytes;
  L.frontier = align_up(L.state + sizeof(NodeState) * static_cast<size_t>(B));
  L.hs = align_up(L.frontier + sizeof(Entry) * static_cast<size_t>(B) * n);
  L.acc = align_up(L.hs + sizeof(float) * static_cast<size_t>(B) * n * H);
  // per-step per-candidate accumulators [n][B][M] int64, then per-node publication counters [B][n] int32
  const size_t acc_bytes =
      B <= kSmallMaxB ? sizeof(long long) * (static_cast<size_t>(n) * B * M + (static_cast<size_t>(B) * n + 1) / 2)
                      : 0;
  L.bytes = align_up(L.acc + acc_bytes);
  return L;
}


// The small-batch builder (build_small.cu). Returns false when its shared-memory plan does not fit this device
// (the caller then uses the general builder).
bool small_builder_fits(const Params& p, int sms);
cudaError_t launch_small_builder(const Params& p, cudaStream_t stream);

}  // namespace dt
