// dt_topm — top-M candidate restriction over the drafter's marginal logits.
//
// Method: blog.captcha.la, "Methodology — deep read" / "Technical innovations" (the per-node correction only sees
// the M highest-marginal tokens of each depth); gist.science, "Composants Clés — Restriction de Candidats".
//
// GB300 design. The op is a pure HBM stream (every logit is read once, nothing is reused), so the kernel is laid
// out for bandwidth and for few instructions per logit, not for tensor cores:
//   * grid = (chunks of 16384 logits) x (B*K rows), 256 threads; every thread issues its eight (bf16) 16-byte loads
//     up front (64 logits in registers), consecutive threads on consecutive 16 bytes;
//   * the chunk's top-M is found without sorting the chunk. Lower bound: every warp takes the ceil(M / 8)-th largest
//     of its lane maxima (ballot bisection, all warps at once) and the smallest of those bounds is kept. Maxima use
//     the packed bf16x2 max, candidates the packed bf16x2 compare-to-mask: one instruction per two logits in the
//     common "nothing here" case. Only the ~1% of logits at or above the bound are re-read, appended to shared
//     memory and ranked (32-bit chunk-local words for bf16: key << 16 | ~local index);
//   * the last CTA of a row (atomic ticket, fences) merges the row's sorted chunk lists. Lower bound: the M-th
//     largest among the first ceil(M / chunks) words of every list (chunks * ceil(M / chunks) >= M distinct words);
//   * every comparison is on distinct integer words (value key, then inverted id), so the result is exact and
//     deterministic, ties broken by the lower id.
// A chunk whose bound admits more than kCap logits (heavy ties) takes an exact bisection over its words instead,
// re-reading the chunk; slower, same result.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <type_traits>

#include "dt_internal.cuh"

namespace dt {
namespace {

constexpr int kPer = 64;          // logits per thread
constexpr int kCap = 1024;        // shared-memory candidate buffer of a chunk
constexpr int kMergeSmem = 2048;  // chunk-list words the merge keeps in shared memory

__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t v) { return *reinterpret_cast<__nv_bfloat162*>(&v); }

template <bool kBf16, int kThreads>
struct Topm {
  static constexpr int kWarps = kThreads / 32;
  static constexpr int kChunk = kThreads * kPer;
  static constexpr int kPer16 = kBf16 ? 8 : 4;  // logits per 16-byte load
  static constexpr int kGroups = kPer / kPer16;
  static constexpr int kKeyBits = kBf16 ? 16 : 32;
  // A chunk-local word: value key in the high part, 0xFFFF / 0xFFFFFFFF minus the local index in the low part.
  using CWord = typename std::conditional<kBf16, uint32_t, uint64_t>::type;
  static constexpr int kIdxBits = kBf16 ? 16 : 32;
  static_assert(kChunk <= 65536, "chunk-local index must fit 16 bits");

  struct Smem {
    union alignas(16) {
      CWord cand[kCap];       // chunk stage: chunk-local candidate words
      uint64_t mcand[kCap];   // merge: candidate words of the row
    };
    uint64_t lists[kMergeSmem];
    uint64_t wmax[kWarps];
    uint32_t tmax[kThreads];
    uint32_t wkey[kWarps];
    int warp[kWarps];
    uint32_t theta;
    int n;
    int flag;
    uint64_t beta;
  };

  uint4 g[kGroups];  // this thread's 64 logits, as loaded

  __device__ static __forceinline__ CWord cword(uint32_t bits, int li) {
    const uint32_t key = kBf16 ? key_of_bf16(bits) : key_of_f32(bits);
    return (static_cast<CWord>(key) << kIdxBits) | static_cast<CWord>((kBf16 ? 0xFFFFu : 0xFFFFFFFFu) - li);
  }
  __device__ static __forceinline__ uint64_t global_word(CWord w, int c0) {
    const uint32_t key = static_cast<uint32_t>(w >> kIdxBits);
    const uint32_t low = kBf16 ? (static_cast<uint32_t>(w) & 0xFFFFu) : static_cast<uint32_t>(w);
    const int li = static_cast<int>((kBf16 ? 0xFFFFu : 0xFFFFFFFFu) - low);
    return pack_candidate(key, static_cast<uint32_t>(c0 + li));
  }

  // Loads this thread's logits (16-byte groups t, t + kThreads, ...). Past the end of the row the slots hold -inf,
  // which never changes a maximum and is kept out of the candidates by its index. Reports NaNs among real logits
  // (fp32 here; bf16 in max_key).
  __device__ __forceinline__ void load(const void* logits, long long row_off, int c0, int len, bool vec_ok,
                                       bool& nan) {
    const int t = threadIdx.x;
    constexpr uint32_t kPad = kBf16 ? 0xFF80FF80u : 0xFF800000u;
#pragma unroll
    for (int k = 0; k < kGroups; ++k) {
      const int li0 = (t + kThreads * k) * kPer16;
      if (vec_ok && li0 + kPer16 <= len) {
        g[k] = ld_stream_v4(static_cast<const char*>(logits) +
                            (row_off + c0 + li0) * static_cast<long long>(kBf16 ? 2 : 4));
      } else {
        uint32_t w[4] = {kPad, kPad, kPad, kPad};
        for (int e = 0; e < kPer16 && li0 + e < len; ++e) {
          if (kBf16) {
            const uint32_t b = static_cast<const uint16_t*>(logits)[row_off + c0 + li0 + e];
            w[e / 2] = (e & 1) ? ((w[e / 2] & 0x0000FFFFu) | (b << 16)) : ((w[e / 2] & 0xFFFF0000u) | b);
          } else {
            w[e] = static_cast<const uint32_t*>(logits)[row_off + c0 + li0 + e];
          }
        }
        g[k] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    if (!kBf16) {
#pragma unroll
      for (int k = 0; k < kGroups; ++k)
        nan |= is_nan_f32(g[k].x) | is_nan_f32(g[k].y) | is_nan_f32(g[k].z) | is_nan_f32(g[k].w);
    }
  }

  // Key of this thread's largest non-NaN logit (0 if none); sets `nan` when a NaN is present (bf16).
  __device__ __forceinline__ uint32_t max_key(bool& nan) const {
    if (kBf16) {
      __nv_bfloat162 m = as_bf2(g[0].x);
#pragma unroll
      for (int k = 0; k < kGroups; ++k) {
        m = __hmax2_nan(m, as_bf2(g[k].x));
        m = __hmax2_nan(m, as_bf2(g[k].y));
        m = __hmax2_nan(m, as_bf2(g[k].z));
        m = __hmax2_nan(m, as_bf2(g[k].w));
      }
      uint32_t mw = as_u32(__hmax2_nan(m, __lowhigh2highlow(m))) & 0xFFFFu;
      if (is_nan_bf16(mw)) {  // rare: a NaN is present; take the maximum without it
        nan = true;
        m = as_bf2(0xFF80FF80u);
#pragma unroll
        for (int k = 0; k < kGroups; ++k) {
          m = __hmax2(m, as_bf2(g[k].x));
          m = __hmax2(m, as_bf2(g[k].y));
          m = __hmax2(m, as_bf2(g[k].z));
          m = __hmax2(m, as_bf2(g[k].w));
        }
        mw = as_u32(__hmax2(m, __lowhigh2highlow(m))) & 0xFFFFu;
        if (is_nan_bf16(mw)) return 0u;
      }
      return key_of_bf16(mw);
    } else {
      float m = -INFINITY;
#pragma unroll
      for (int k = 0; k < kGroups; ++k) {
        m = fmaxf(m, __uint_as_float(g[k].x));
        m = fmaxf(m, __uint_as_float(g[k].y));
        m = fmaxf(m, __uint_as_float(g[k].z));
        m = fmaxf(m, __uint_as_float(g[k].w));
      }
      return is_nan_f32(__float_as_uint(m)) ? 0u : key_of_f32(__float_as_uint(m));
    }
  }

  // Bit k of the result is set when 16-byte group k of this thread holds a logit >= the threshold value (NaN never
  // does; padding may, and is dropped by index later). Fully unrolled, the logits stay in registers; for bf16 one
  // packed compare covers two logits and the common "nothing here" group costs five instructions.
  __device__ __forceinline__ unsigned group_mask(uint32_t thr_bits) const {
    unsigned sel = 0;
    if (kBf16) {
      const __nv_bfloat162 th = as_bf2(thr_bits | (thr_bits << 16));
#pragma unroll
      for (int k = 0; k < kGroups; ++k) {
        const unsigned any = __hge2_mask(as_bf2(g[k].x), th) | __hge2_mask(as_bf2(g[k].y), th) |
                             __hge2_mask(as_bf2(g[k].z), th) | __hge2_mask(as_bf2(g[k].w), th);
        sel |= (any != 0u) << k;
      }
    } else {
      const float th = __uint_as_float(thr_bits);
#pragma unroll
      for (int k = 0; k < kGroups; ++k) {
        const bool any = __uint_as_float(g[k].x) >= th || __uint_as_float(g[k].y) >= th ||
                         __uint_as_float(g[k].z) >= th || __uint_as_float(g[k].w) >= th;
        sel |= static_cast<unsigned>(any) << k;
      }
    }
    return sel;
  }
  // Group k of this thread's registers, for a run-time k (a select chain, no local memory).
  __device__ __forceinline__ uint4 group(int k) const {
    uint4 v = g[0];
#pragma unroll
    for (int j = 1; j < kGroups; ++j)
      if (k == j) v = g[j];
    return v;
  }
  __device__ static __forceinline__ int local_index(int e) {
    return (static_cast<int>(threadIdx.x) + kThreads * (e / kPer16)) * kPer16 + (e % kPer16);
  }
};

// The M-th largest of kN keys in shared memory (kN a multiple of 32), by one warp: bisection on the key bits,
// counting with ballots.
template <int kKeyBits, int kN>
__device__ __forceinline__ uint32_t warp_kth_key(const uint32_t* keys, int M) {
  const int lane = threadIdx.x & 31;
  uint32_t v[kN / 32];
#pragma unroll
  for (int i = 0; i < kN / 32; ++i) v[i] = keys[lane + 32 * i];
  uint32_t th = 0;
  for (int bit = kKeyBits - 1; bit >= 0; --bit) {
    const uint32_t c = th | (1u << bit);
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < kN / 32; ++i) cnt += __popc(__ballot_sync(0xFFFFFFFFu, v[i] >= c));
    if (cnt >= M) th = c;
  }
  return th;
}

// The k-th largest of the 32 lane values of a warp (k <= 32), by bisection on the key bits with ballots.
template <int kKeyBits>
__device__ __forceinline__ uint32_t warp_kth_lane_key(uint32_t v, int k) {
  uint32_t th = 0;
#pragma unroll
  for (int bit = kKeyBits - 1; bit >= 0; --bit) {
    const uint32_t c = th | (1u << bit);
    if (__popc(__ballot_sync(0xFFFFFFFFu, v >= c)) >= k) th = c;
  }
  return th;
}

// Exact M-th largest word among words spread over the block, by bisection on the word bits.
template <int kWarps, typename Word, typename CountGe>
__device__ Word block_kth_largest(int M, int hi_bit, CountGe count_ge, int* s_warp) {
  Word prefix = 0;
  for (int bit = hi_bit; bit >= 0; --bit) {
    const Word c = prefix | (static_cast<Word>(1) << bit);
    if (block_sum<kWarps>(count_ge(c), s_warp) >= M) prefix = c;
  }
  return prefix;
}

// Ranks the `total` distinct words of cand; the M largest, in descending order, go to out[0..M) converted by
// conv(word). Slots past `total` get 0.
template <int kThreads, typename Word, typename Conv>
__device__ __forceinline__ void rank_and_emit(const Word* cand, int total, int M, uint64_t* out, Conv conv) {
  for (int i = threadIdx.x; i < total; i += kThreads) {
    const Word ci = cand[i];
    int r = 0;
    if (sizeof(Word) == 4) {  // four words per shared-memory load
      const uint4* c4 = reinterpret_cast<const uint4*>(cand);
      int j = 0;
      for (; j + 4 <= total; j += 4) {
        const uint4 q = c4[j / 4];
        r += (q.x > ci) + (q.y > ci) + (q.z > ci) + (q.w > ci);
      }
      for (; j < total; ++j) r += cand[j] > ci;
    } else {
      for (int j = 0; j < total; ++j) r += cand[j] > ci;
    }
    if (r < M) out[r] = conv(ci);
  }
  for (int i = total + threadIdx.x; i < M; i += kThreads) out[i] = 0;
}

template <bool kBf16, int kThreads>
__device__ __forceinline__ void emit_final(const uint64_t* sorted, int M, int32_t* ids, float* vals) {
  for (int m = threadIdx.x; m < M; m += kThreads) {
    const uint64_t c = sorted[m];
    // 0 = no element (only possible for rows made of NaNs): keep the id in range
    ids[m] = c ? static_cast<int32_t>(candidate_id(c)) : 0;
    vals[m] = c ? (kBf16 ? value_of_key_bf16(candidate_key(c)) : value_of_key_f32(candidate_key(c))) : -INFINITY;
  }
}

template <bool kBf16, int kThreads>
__global__ void __launch_bounds__(kThreads) topm_kernel(const void* __restrict__ logits, int V, int M, int chunks,
                                                        bool vec_ok, uint64_t* __restrict__ lists,
                                                        unsigned* __restrict__ tickets, int32_t* __restrict__ out_ids,
                                                        float* __restrict__ out_vals, WsHeader* hdr) {
  using T = Topm<kBf16, kThreads>;
  using CWord = typename T::CWord;
  constexpr int kWarps = T::kWarps;
  __shared__ typename T::Smem s;
  const int row = blockIdx.y, chunk = blockIdx.x, t = threadIdx.x, warp = t >> 5;
  const long long row_off = static_cast<long long>(row) * V;
  const int c0 = chunk * T::kChunk;
  const int len = min(T::kChunk, V - c0);

  T x;
  bool nan = false;
  x.load(logits, row_off, c0, len, vec_ok, nan);
  const uint32_t my_max = x.max_key(nan);
  s.tmax[t] = my_max;
  if (t == 0) s.n = 0;
  if (__syncthreads_or(nan) && t == 0) record_error(hdr, DT_ERR_NUMERIC);

  // Lower bound of the chunk's M-th largest logit. Each warp takes the k-th largest of its 32 lane maxima,
  // k = ceil(M / warps): the warps' k lanes at or above their own bound are kWarps * k >= M distinct logits at or above
  // the smallest of those bounds. (A lane holding only padding has the maximum -inf and can pull that bound down to
  // -inf, which admits every logit: still a lower bound.) With k > 32 one warp takes the M-th largest of all maxima.
  const int k = (M + kWarps - 1) / kWarps;
  if (k <= 32) {
    const uint32_t th = warp_kth_lane_key<T::kKeyBits>(my_max, k);
    if ((t & 31) == 0) s.wkey[warp] = th;
    __syncthreads();
    if (t == 0) {
      uint32_t mn = s.wkey[0];
      for (int w = 1; w < kWarps; ++w) mn = min(mn, s.wkey[w]);
      s.theta = mn;
    }
  } else if (warp == 0) {
    const uint32_t th = warp_kth_key<T::kKeyBits, kThreads>(s.tmax, M);
    if (t == 0) s.theta = th;
  }
  __syncthreads();
  const uint32_t theta = s.theta;
  const uint32_t thr_bits =
      theta ? (kBf16 ? ((theta & 0x8000u) ? (theta & 0x7FFFu) : (~theta & 0xFFFFu))
                     : ((theta & 0x80000000u) ? (theta & 0x7FFFFFFFu) : ~theta))
            : (kBf16 ? 0xFF80u : 0xFF800000u);  // -inf: every non-NaN logit
  // Groups holding a selected logit are rare (a few percent): visit only those.
  for (unsigned sel = x.group_mask(thr_bits); sel; sel &= sel - 1) {
    const int k = __ffs(sel) - 1;
    const uint4 v = x.group(k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const int li0 = (t + kThreads * k) * T::kPer16;
#pragma unroll
    for (int e = 0; e < T::kPer16; ++e) {
      const uint32_t bits = kBf16 ? ((w[e / 2] >> (16 * (e & 1))) & 0xFFFFu) : w[e];
      const bool ok = kBf16 ? (__bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(bits))) >=
                               __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(thr_bits))))
                            : (__uint_as_float(bits) >= __uint_as_float(thr_bits));
      if (ok && li0 + e < len) {
        const int idx = atomicAdd(&s.n, 1);
        if (idx < kCap) s.cand[idx] = T::cword(bits, li0 + e);
      }
    }
  }
  __syncthreads();
  int total = s.n;
  if (total > kCap) {
    // Heavy ties at the bound (rare): the exact M-th largest word by bisection, re-reading the chunk from memory so
    // that this path leaves the registers of the main path alone; then exactly the words at or above it.
    auto word_at = [&](int li) -> CWord {
      const uint32_t bits = kBf16 ? static_cast<uint32_t>(static_cast<const uint16_t*>(logits)[row_off + c0 + li])
                                  : static_cast<const uint32_t*>(logits)[row_off + c0 + li];
      const bool ok = kBf16 ? !is_nan_bf16(bits) : !is_nan_f32(bits);
      return ok ? T::cword(bits, li) : static_cast<CWord>(0);
    };
    const CWord kth = block_kth_largest<kWarps, CWord>(
        M, T::kIdxBits + T::kKeyBits - 1,
        [&](CWord c) {
          int n = 0;
          for (int li = t; li < len; li += kThreads) n += word_at(li) >= c;
          return n;
        },
        s.warp);
    __syncthreads();
    if (t == 0) s.n = 0;
    __syncthreads();
    for (int li = t; li < len; li += kThreads) {
      const CWord w = word_at(li);
      if (w && w >= kth) s.cand[atomicAdd(&s.n, 1)] = w;
    }
    __syncthreads();
    total = s.n;
  }

  const long long row_out = static_cast<long long>(row) * M;
  auto to_global = [&](CWord w) { return T::global_word(w, c0); };
  if (chunks == 1) {
    rank_and_emit<kThreads>(s.cand, total, M, s.lists, to_global);
    __syncthreads();
    emit_final<kBf16, kThreads>(s.lists, M, out_ids + row_out, out_vals + row_out);
    return;
  }
  uint64_t* my_list = lists + (static_cast<long long>(row) * chunks + chunk) * M;
  rank_and_emit<kThreads>(s.cand, total, M, my_list, to_global);

  // The last CTA of the row to finish merges the row's chunk lists. The barrier orders every thread's list writes
  // before thread 0's fence, which publishes them at device scope before the ticket.
  __syncthreads();
  if (t == 0) {
    __threadfence();
    s.flag = (atomicAdd(&tickets[row], 1u) == static_cast<unsigned>(chunks - 1));
  }
  __syncthreads();
  if (!s.flag) return;
  if (t == 0) {
    __threadfence();
    tickets[row] = 0u;
    s.beta = 0;
  }
  const uint64_t* row_lists = lists + static_cast<long long>(row) * chunks * M;
  const int entries = chunks * M;
  const bool in_smem = entries <= kMergeSmem;
  if (in_smem)
    for (int i = t; i < entries; i += kThreads) s.lists[i] = __ldcg(row_lists + i);
  __syncthreads();
  auto entry = [&](int i) { return in_smem ? s.lists[i] : __ldcg(row_lists + i); };

  // Lower bound of the row's M-th word: the M-th largest among the first q = ceil(M / chunks) words of every
  // (sorted) chunk list, which are chunks * q >= M distinct words. 0 if fewer than M of them exist.
  const int q = (M + chunks - 1) / chunks;
  const int pn = chunks * q;
  for (int i = t; i < pn; i += kThreads) {
    const uint64_t wi = entry((i / q) * M + (i % q));
    if (wi == 0) continue;
    int r = 0;
    for (int j = 0; j < pn; ++j) r += entry((j / q) * M + (j % q)) > wi;
    if (r == M - 1) s.beta = wi;
  }
  __syncthreads();
  const uint64_t bound = s.beta ? s.beta : 1ull;

  int mine = 0;
  for (int i = t; i < entries; i += kThreads) mine += entry(i) >= bound;
  int off = block_exclusive_scan<kWarps>(mine, &total, s.warp);
  uint64_t* mcand = s.mcand;
  if (total <= kCap) {
    for (int i = t; i < entries; i += kThreads) {
      const uint64_t v = entry(i);
      if (v >= bound) mcand[off++] = v;
    }
  } else {
    const uint64_t kth = block_kth_largest<kWarps, uint64_t>(
        M, 63,
        [&](uint64_t c) {
          int n = 0;
          for (int i = t; i < entries; i += kThreads) n += entry(i) >= c;
          return n;
        },
        s.warp);
    mine = 0;
    for (int i = t; i < entries; i += kThreads) mine += entry(i) >= kth;
    off = block_exclusive_scan<kWarps>(mine, &total, s.warp);
    for (int i = t; i < entries; i += kThreads) {
      const uint64_t v = entry(i);
      if (v >= kth) mcand[off++] = v;
    }
  }
  __syncthreads();
  uint64_t* sorted = s.lists;  // the chunk lists are no longer needed
  rank_and_emit<kThreads>(mcand, total, M, sorted, [](uint64_t w) { return w; });
  __syncthreads();
  emit_final<kBf16, kThreads>(sorted, M, out_ids + row_out, out_vals + row_out);
}

dt_status launch_topm(const void* logits, dt_dtype dtype, int B, int K, int V, int M, int32_t* out_ids,
                      float* out_vals, char* ws, const TopmLayout& L, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * K;
  auto* hdr = reinterpret_cast<WsHeader*>(ws);
  auto* tickets = reinterpret_cast<unsigned*>(ws + L.tickets);
  auto* lists = reinterpret_cast<uint64_t*>(ws + L.lists);
  const size_t esize = dtype == DT_BF16 ? 2 : 4;
  const bool vec_ok = (static_cast<size_t>(V) * esize) % 16 == 0;
  const dim3 grid(static_cast<unsigned>(L.chunks), static_cast<unsigned>(rows));
  constexpr int kThreads = 256;  // Topm<.., 256>::kChunk == topm_chunk()
  if (dtype == DT_BF16)
    topm_kernel<true, kThreads><<<grid, kThreads, 0, stream>>>(logits, V, M, L.chunks, vec_ok, lists, tickets,
                                                               out_ids, out_vals, hdr);
  else
    topm_kernel<false, kThreads><<<grid, kThreads, 0, stream>>>(logits, V, M, L.chunks, vec_ok, lists, tickets,
                                                                out_ids, out_vals, hdr);
  return cuda_status(cudaGetLastError());
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
  if (static_cast<long long>(B) * K > 65535) return DT_ERR_UNSUPPORTED;  // grid.y limit of one launch
  return launch_topm(logits, dtype, B, K, V, M, out_ids, out_vals, static_cast<char*>(workspace), L, stream);
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
  if (static_cast<long long>(B) * K > 65535) return DT_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const dt_status st = static_scratch(&scratch);
  if (st != DT_OK) return st;
  char* ws = static_cast<char*>(scratch);
  // The array keeps the previous call's contents: the header and the per-row tickets must start at zero.
  if (cudaMemsetAsync(ws, 0, L.lists, stream) != cudaSuccess) return DT_ERR_CUDA;
  return launch_topm(logits, dtype, B, K, V, M, out_ids, out_vals, ws, L, stream);
}
