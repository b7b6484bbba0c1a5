// dt_topm — top-M candidate restriction over the drafter's marginal logits.
//
// Method: blog.captcha.la, "Methodology — deep read" / "Technical innovations" (the per-node correction only sees
// the M highest-marginal tokens of each depth); gist.science, "Composants Clés — Restriction de Candidats".
//
// GB300 design. The op is a pure HBM stream (every logit is read once, nothing is reused), so the kernel is laid
// out for bandwidth, not for tensor cores:
//   * grid = (chunks of 8192 logits) x (B*K rows): even one request (16 rows of 151936) gives 304 CTAs, two per
//     SM of the 152, and each CTA issues all its 16-byte loads up front (64 B/thread of bf16 in flight);
//   * each logit becomes an order-preserving integer key in registers; the chunk's top-M is found without sorting
//     the chunk: the M-th largest per-thread maximum is a lower bound of the chunk's M-th largest value (the M
//     threads above it each own a distinct element at least that large), found by a 16- or 32-step bisection of
//     block-wide counts; only the ~1% of elements at or above it are compacted into shared memory and ranked;
//   * the last CTA of a row (atomic ticket, fences) merges the row's chunk lists the same way: the largest M-th
//     entry over the sorted chunk lists bounds the row's M-th candidate from below;
//   * every comparison is on 64-bit words (key << 32 | ~id), all distinct, so the result is exact and
//     deterministic, ties broken by the lower id.
// A chunk whose bound admits more than TOPM_CAP elements (heavy ties) takes an exact bisection over the 64-bit
// words instead; slower, same result.
#include <cuda_runtime.h>

#include <mutex>

#include "dt_internal.cuh"

namespace dt {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPerThread = 32;
constexpr int kChunk = kThreads * kPerThread;  // 8192 logits per CTA
static_assert(kChunk == kTopmChunk, "chunk size shared with the workspace layout");
constexpr int kCap = 1024;                     // shared-memory candidate buffer

struct TopmSmem {
  uint64_t cand[kCap];
  uint64_t wmax[kWarps];
  int warp[kWarps];
  int flag;
};

// Local index (within the chunk) of the j-th key of thread t: 16-byte groups t, t+256, ... of 8 (bf16) or 4 (f32).
template <bool kBf16>
__device__ __forceinline__ int local_index(int t, int j) {
  constexpr int per = kBf16 ? 8 : 4;
  return (t + kThreads * (j / per)) * per + (j % per);
}

template <bool kBf16>
__device__ __forceinline__ void load_keys(const void* logits, long long row_off, int c0, int len, bool vec_ok,
                                          uint32_t (&key)[kPerThread], bool& nan) {
  constexpr int per = kBf16 ? 8 : 4;
  constexpr int groups = kPerThread / per;
  const int t = threadIdx.x;
  uint32_t raw[kPerThread];
#pragma unroll
  for (int g = 0; g < groups; ++g) {
    const int li0 = (t + kThreads * g) * per;
    if (vec_ok && li0 + per <= len) {
      const char* p = static_cast<const char*>(logits) +
                      (row_off + c0 + li0) * static_cast<long long>(kBf16 ? 2 : 4);
      const uint4 v = ld_stream_v4(p);
      if (kBf16) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) raw[g * 8 + e] = (w[e / 2] >> (16 * (e & 1))) & 0xFFFFu;
      } else {
        raw[g * 4 + 0] = v.x;
        raw[g * 4 + 1] = v.y;
        raw[g * 4 + 2] = v.z;
        raw[g * 4 + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < per; ++e) {
        const int li = li0 + e;
        uint32_t r = 0xFFFFFFFFu;  // marks padding
        if (li < len) {
          if (kBf16)
            r = static_cast<const uint16_t*>(logits)[row_off + c0 + li];
          else
            r = static_cast<const uint32_t*>(logits)[row_off + c0 + li];
        }
        raw[g * per + e] = r;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int li = local_index<kBf16>(t, j);
    if (li < len) {
      nan |= kBf16 ? is_nan_bf16(raw[j]) : is_nan_f32(raw[j]);
      key[j] = kBf16 ? key_of_bf16(raw[j]) : key_of_f32(raw[j]);
    } else {
      key[j] = 0u;
    }
  }
}

// Exact M-th largest word among `count(x)` candidates spread over the block, by bisection on the 64-bit words.
// `count_ge(c)` returns how many of this thread's words are >= c.
template <typename CountGe>
__device__ uint64_t block_kth_largest(int M, int hi_bit, CountGe count_ge, int* s_warp) {
  uint64_t prefix = 0;
  for (int bit = hi_bit; bit >= 0; --bit) {
    const uint64_t c = prefix | (1ull << bit);
    if (block_sum<kWarps>(count_ge(c), s_warp) >= M) prefix = c;
  }
  return prefix;
}

// Ranks the `total` words of s.cand (all distinct) and writes the M largest, in descending order, to out[0..M).
// Slots past `total` get 0.
__device__ __forceinline__ void rank_and_emit(TopmSmem& s, int total, int M, uint64_t* out) {
  for (int i = threadIdx.x; i < total; i += kThreads) {
    const uint64_t ci = s.cand[i];
    int r = 0;
    for (int j = 0; j < total; ++j) r += s.cand[j] > ci;
    if (r < M) out[r] = ci;
  }
  for (int i = total + threadIdx.x; i < M; i += kThreads) out[i] = 0;
}

template <bool kBf16>
__device__ __forceinline__ void emit_final(const uint64_t* sorted, int M, int32_t* ids, float* vals) {
  for (int m = threadIdx.x; m < M; m += kThreads) {
    const uint64_t c = sorted[m];
    ids[m] = static_cast<int32_t>(candidate_id(c));
    vals[m] = kBf16 ? value_of_key_bf16(candidate_key(c)) : value_of_key_f32(candidate_key(c));
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads) topm_kernel(const void* __restrict__ logits, int V, int M, int chunks,
                                                        bool vec_ok, uint64_t* __restrict__ lists,
                                                        unsigned* __restrict__ tickets, int32_t* __restrict__ out_ids,
                                                        float* __restrict__ out_vals, WsHeader* hdr) {
  __shared__ TopmSmem s;
  __shared__ uint64_t s_out[1024];  // the row's final sorted list when chunks == 1 or in the merge
  constexpr int kKeyBits = kBf16 ? 16 : 32;
  const int row = blockIdx.y, chunk = blockIdx.x, t = threadIdx.x;
  const long long row_off = static_cast<long long>(row) * V;
  const int c0 = chunk * kChunk;
  const int len = min(kChunk, V - c0);

  uint32_t key[kPerThread];
  bool nan = false;
  load_keys<kBf16>(logits, row_off, c0, len, vec_ok, key, nan);
  if (__syncthreads_or(nan) && t == 0) record_error(hdr, DT_ERR_NUMERIC);

  // Lower bound: the M-th largest of the per-thread maxima (0 when fewer than M threads hold an element).
  uint32_t tmax = 0;
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) tmax = max(tmax, key[j]);
  uint32_t theta = 0;
  for (int bit = kKeyBits - 1; bit >= 0; --bit) {
    const uint32_t c = theta | (1u << bit);
    if (__syncthreads_count(tmax >= c) >= M) theta = c;
  }
  const uint32_t thr = theta > 0 ? theta : 1u;

  int mine = 0;
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) mine += key[j] >= thr;
  int total;
  int off = block_exclusive_scan<kWarps>(mine, &total, s.warp);
  if (total <= kCap) {
#pragma unroll
    for (int j = 0; j < kPerThread; ++j)
      if (key[j] >= thr) s.cand[off++] = pack_candidate(key[j], static_cast<uint32_t>(c0 + local_index<kBf16>(t, j)));
  } else {
    // Heavy ties at the bound: find the exact M-th largest word, then keep exactly the words at or above it.
    auto word = [&](int j) {
      return key[j] ? pack_candidate(key[j], static_cast<uint32_t>(c0 + local_index<kBf16>(t, j))) : 0ull;
    };
    const uint64_t kth = block_kth_largest(
        M, 32 + kKeyBits - 1,
        [&](uint64_t c) {
          int n = 0;
#pragma unroll
          for (int j = 0; j < kPerThread; ++j) n += word(j) >= c;
          return n;
        },
        s.warp);
    mine = 0;
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) mine += key[j] != 0 && word(j) >= kth;
    off = block_exclusive_scan<kWarps>(mine, &total, s.warp);
#pragma unroll
    for (int j = 0; j < kPerThread; ++j)
      if (key[j] != 0 && word(j) >= kth) s.cand[off++] = word(j);
  }
  __syncthreads();

  const long long row_out = static_cast<long long>(row) * M;
  if (chunks == 1) {
    rank_and_emit(s, total, M, s_out);
    __syncthreads();
    emit_final<kBf16>(s_out, M, out_ids + row_out, out_vals + row_out);
    return;
  }

  uint64_t* my_list = lists + (static_cast<long long>(row) * chunks + chunk) * M;
  rank_and_emit(s, total, M, my_list);

  // The last CTA of the row to finish merges the row's chunk lists.
  __threadfence();
  __syncthreads();
  if (t == 0) s.flag = (atomicAdd(&tickets[row], 1u) == static_cast<unsigned>(chunks - 1));
  __syncthreads();
  if (!s.flag) return;
  __threadfence();
  if (t == 0) tickets[row] = 0u;

  const uint64_t* row_lists = lists + static_cast<long long>(row) * chunks * M;
  const int entries = chunks * M;
  // Every chunk list is sorted and chunk 0 holds at least M elements, so the largest M-th entry is >= 1 and at
  // least M words reach it.
  uint64_t bound = 0;
  for (int c = t; c < chunks; c += kThreads) {
    const uint64_t v = __ldcg(row_lists + static_cast<long long>(c) * M + (M - 1));
    bound = v > bound ? v : bound;
  }
  bound = block_max_u64<kWarps>(bound, s.wmax);

  mine = 0;
  for (int i = t; i < entries; i += kThreads) mine += __ldcg(row_lists + i) >= bound;
  off = block_exclusive_scan<kWarps>(mine, &total, s.warp);
  if (total <= kCap) {
    for (int i = t; i < entries; i += kThreads) {
      const uint64_t v = __ldcg(row_lists + i);
      if (v >= bound) s.cand[off++] = v;
    }
  } else {
    const uint64_t kth = block_kth_largest(
        M, 63,
        [&](uint64_t c) {
          int n = 0;
          for (int i = t; i < entries; i += kThreads) n += __ldcg(row_lists + i) >= c;
          return n;
        },
        s.warp);
    mine = 0;
    for (int i = t; i < entries; i += kThreads) mine += __ldcg(row_lists + i) >= kth;
    off = block_exclusive_scan<kWarps>(mine, &total, s.warp);
    for (int i = t; i < entries; i += kThreads) {
      const uint64_t v = __ldcg(row_lists + i);
      if (v >= kth) s.cand[off++] = v;
    }
  }
  __syncthreads();
  rank_and_emit(s, total, M, s_out);
  __syncthreads();
  emit_final<kBf16>(s_out, M, out_ids + row_out, out_vals + row_out);
}

}  // namespace
}  // namespace dt

extern "C" size_t dt_topm_workspace_bytes(int B, int K, int V, int M) {
  if (B < 0 || K < 1 || V < 1 || M < 1) return 0;
  return dt::topm_layout(B, K, V, M).bytes;
}

extern "C" dt_status dt_topm(const void* logits, dt_dtype dtype, int B, int K, int V, int M, int32_t* out_ids,
                             float* out_vals, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  using namespace dt;
  if (B < 0 || K < 1 || V < 1 || M < 1 || M > V) return DT_ERR_INVALID_ARG;
  if (dtype != DT_F32 && dtype != DT_BF16) return DT_ERR_INVALID_ARG;
  if (M > DT_MAX_M) return DT_ERR_UNSUPPORTED;
  if (B == 0) return DT_OK;  // nothing to read or write
  if (!logits || !out_ids || !out_vals || !workspace) return DT_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(out_ids) || !aligned16(out_vals) || !aligned16(workspace))
    return DT_ERR_INVALID_ARG;
  const TopmLayout L = topm_layout(B, K, V, M);
  if (workspace_bytes < L.bytes) return DT_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * K;
  if (rows > 65535) return DT_ERR_UNSUPPORTED;  // grid.y limit of one launch
  char* ws = static_cast<char*>(workspace);
  auto* hdr = reinterpret_cast<WsHeader*>(ws);
  auto* tickets = reinterpret_cast<unsigned*>(ws + L.tickets);
  auto* lists = reinterpret_cast<uint64_t*>(ws + L.lists);
  const size_t esize = dtype == DT_BF16 ? 2 : 4;
  const bool vec_ok = (static_cast<size_t>(V) * esize) % 16 == 0;
  const dim3 grid(static_cast<unsigned>(L.chunks), static_cast<unsigned>(rows));
  if (dtype == DT_BF16)
    topm_kernel<true><<<grid, kThreads, 0, stream>>>(logits, V, M, L.chunks, vec_ok, lists, tickets, out_ids,
                                                     out_vals, hdr);
  else
    topm_kernel<false><<<grid, kThreads, 0, stream>>>(logits, V, M, L.chunks, vec_ok, lists, tickets, out_ids,
                                                      out_vals, hdr);
  return cuda_status(cudaGetLastError());
}

// ---- dt_topm_static: the same top-M with no caller workspace ----------------------------------------------------
// For callers that cannot call cudaMalloc (see dominotree.h). Its scratch is this file-scope device array: every GPU
// that loads the library holds it until the process exits. Host code must not pass `g_topm_scratch` itself to a
// kernel (on the host that name is only a stand-in); the device address comes from cudaGetSymbolAddress, taken once
// per device with that device current, on the first call made on it.
namespace dt {
namespace {
__device__ __align__(256) unsigned char g_topm_scratch[DT_TOPM_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

dt_status static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topm_scratch) != cudaSuccess || !p) return DT_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DT_OK;
}
}  // namespace
}  // namespace dt

extern "C" dt_status dt_topm_static(const void* logits, dt_dtype dtype, int B, int K, int V, int M,
                                    int32_t* out_ids, float* out_vals, cudaStream_t stream) {
  using namespace dt;
  if (B < 0 || K < 1 || V < 1 || M < 1 || M > V) return DT_ERR_INVALID_ARG;
  if (dtype != DT_F32 && dtype != DT_BF16) return DT_ERR_INVALID_ARG;
  if (M > DT_MAX_M) return DT_ERR_UNSUPPORTED;
  if (B == 0) return DT_OK;
  if (!logits || !out_ids || !out_vals) return DT_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(out_ids) || !aligned16(out_vals)) return DT_ERR_INVALID_ARG;
  const TopmLayout L = topm_layout(B, K, V, M);
  if (L.bytes > DT_TOPM_STATIC_SCRATCH_BYTES) return DT_ERR_UNSUPPORTED;  // beyond the fixed scratch array
  const long long rows = static_cast<long long>(B) * K;
  if (rows > 65535) return DT_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const dt_status st = static_scratch(&scratch);
  if (st != DT_OK) return st;
  char* ws = static_cast<char*>(scratch);
  // The array keeps the previous call's contents: the header and the per-row tickets must start at zero.
  if (cudaMemsetAsync(ws, 0, L.lists, stream) != cudaSuccess) return DT_ERR_CUDA;
  auto* hdr = reinterpret_cast<WsHeader*>(ws);
  auto* tickets = reinterpret_cast<unsigned*>(ws + L.tickets);
  auto* lists = reinterpret_cast<uint64_t*>(ws + L.lists);
  const size_t esize = dtype == DT_BF16 ? 2 : 4;
  const bool vec_ok = (static_cast<size_t>(V) * esize) % 16 == 0;
  const dim3 grid(static_cast<unsigned>(L.chunks), static_cast<unsigned>(rows));
  if (dtype == DT_BF16)
    topm_kernel<true><<<grid, kThreads, 0, stream>>>(logits, V, M, L.chunks, vec_ok, lists, tickets, out_ids,
                                                     out_vals, hdr);
  else
    topm_kernel<false><<<grid, kThreads, 0, stream>>>(logits, V, M, L.chunks, vec_ok, lists, tickets, out_ids,
                                                      out_vals, hdr);
  return cuda_status(cudaGetLastError());
}
