// dt_topm — top-M candidate restriction over the drafter's marginal logits.
//
// Method: blog.captcha.la, "Methodology — deep read" / "Technical innovations" (the per-node correction only sees
// the M highest-marginal tokens of each depth); gist.science, "Composants Clés — Restriction de Candidats".
//
// GB300 design. The op is a pure HBM stream (every logit is read once, nothing is reused), so the kernel is laid
// out for bandwidth and for few instructions per logit, not for tensor cores:
//   * grid = (chunks of 16384 logits) x (B*K rows), 256 threads; every thread issues its eight (bf16) 16-byte loads
//     up front (64 logits in registers), consecutive threads on consecutive 16 bytes;
//   * the chunk's top-M is found without sorting the chunk. Lower bound: the M-th largest of the 256 lane maxima
//     (one warp, ballot bisection). Maxima use the packed bf16x2 max, candidates the packed bf16x2
//     compare-to-mask: one instruction per two logits in the common "nothing here" case. Only the logits at or
//     above the bound (about M of the 16384) are appended to shared memory and ranked (32-bit chunk-local words
//     for bf16: key << 16 | ~local index);
//   * the last CTA of a row (atomic ticket, fences) merges the row's sorted chunk lists. Lower bound: the M-th
//     largest among the first ceil(M / chunks) words of every list (chunks * ceil(M / chunks) >= M distinct words);
//   * every comparison is on distinct integer words (value key, then inverted id), so the result is exact and
//     deterministic, ties broken by the lower id.
// A chunk whose bound admits more than kCap logits (heavy ties) takes an exact bisection over its words instead,
// re-reading the chunk; slower, same result.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
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
      // four independent chains (x, y, z, w words), then combined: short dependency chains
      __nv_bfloat162 m0 = as_bf2(g[0].x), m1 = as_bf2(g[0].y), m2 = as_bf2(g[0].z), m3 = as_bf2(g[0].w);
#pragma unroll
      for (int k = 1; k < kGroups; ++k) {
        m0 = __hmax2_nan(m0, as_bf2(g[k].x));
        m1 = __hmax2_nan(m1, as_bf2(g[k].y));
        m2 = __hmax2_nan(m2, as_bf2(g[k].z));
        m3 = __hmax2_nan(m3, as_bf2(g[k].w));
      }
      __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(m0, m1), __hmax2_nan(m2, m3));
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

// Merges the `lists` sorted candidate lists of one row (entry(i) = word i % M of list i / M; 0 = empty) into the
// row's final top-M. Lower bound of the row's M-th word: the M-th largest among the first q = ceil(M / lists) words
// of every list, which are lists * q >= M distinct words (0 if fewer than M exist); only the words at or above it
// are ranked. mcand holds kCapW words of shared memory and sorted M; `sorted` may be the buffer entry() reads,
// which is no longer read once the candidates are in mcand.
template <bool kBf16, int kThreads, int kCapW, typename EntryFn>
__device__ void merge_lists(EntryFn entry, int lists, int M, uint64_t* mcand, uint64_t* sorted, int* s_warp,
                            uint64_t* s_beta, int32_t* ids, float* vals) {
  constexpr int kWarps = kThreads / 32;
  const int t = threadIdx.x;
  const int entries = lists * M;
  if (t == 0) *s_beta = 0;
  __syncthreads();
  const int q = (M + lists - 1) / lists;
  const int pn = lists * q;
  for (int i = t; i < pn; i += kThreads) {
    const uint64_t wi = entry((i / q) * M + (i % q));
    if (wi == 0) continue;
    int r = 0;
    for (int j = 0; j < pn; ++j) r += entry((j / q) * M + (j % q)) > wi;
    if (r == M - 1) *s_beta = wi;
  }
  __syncthreads();
  const uint64_t bound = *s_beta ? *s_beta : 1ull;

  int total = 0;
  int mine = 0;
  for (int i = t; i < entries; i += kThreads) mine += entry(i) >= bound;
  int off = block_exclusive_scan<kWarps>(mine, &total, s_warp);
  if (total <= kCapW) {
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
        s_warp);
    mine = 0;
    for (int i = t; i < entries; i += kThreads) mine += entry(i) >= kth;
    off = block_exclusive_scan<kWarps>(mine, &total, s_warp);
    for (int i = t; i < entries; i += kThreads) {
      const uint64_t v = entry(i);
      if (v >= kth) mcand[off++] = v;
    }
  }
  __syncthreads();
  rank_and_emit<kThreads>(mcand, total, M, sorted, [](uint64_t w) { return w; });
  __syncthreads();
  emit_final<kBf16, kThreads>(sorted, M, ids, vals);
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

  // Lower bound of the chunk's M-th largest logit: the M-th largest of the kThreads lane maxima (M distinct logits
  // are at or above it), found by one warp with ballot bisection while the others wait. It admits little more than
  // the M lanes' maxima, so the ranking below stays small. (A lane holding only padding has the maximum -inf and
  // can pull the bound down to -inf, which admits every logit: still a lower bound.) With M > kThreads there is no
  // such bound and every logit is a candidate (the exact path below).
  if (warp == 0) {
    const uint32_t th = M <= kThreads ? warp_kth_key<T::kKeyBits, kThreads>(s.tmax, M) : 0u;
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
  }
  const uint64_t* row_lists = lists + static_cast<long long>(row) * chunks * M;
  const int entries = chunks * M;
  const bool in_smem = entries <= kMergeSmem;
  if (in_smem)
    for (int i = t; i < entries; i += kThreads) s.lists[i] = __ldcg(row_lists + i);
  __syncthreads();
  merge_lists<kBf16, kThreads, kCap>([&](int i) { return in_smem ? s.lists[i] : __ldcg(row_lists + i); }, chunks, M,
                                     s.mcand, s.lists, s.warp, &s.beta, out_ids + row_out, out_vals + row_out);
}


// ---- streaming top-M: persistent CTAs, a bulk-copy ring, a running threshold ----------------------------------
// The per-chunk kernel above pays a fixed cost per 16384 logits (bound, ranking, a list, a share of a merge) and
// keeps no load in flight while a CTA computes. Here (bf16 rows whose byte length is a multiple of 16, M <= 128)
// the B*K*chunks stages of 16384 logits are split into G equal contiguous ranges, one per persistent CTA (two per
// SM). A CTA walks its range through a ring of kSStages shared-memory stages, each filled by one cp.async.bulk of
// 32 KB that completes on the stage's mbarrier, so (kSStages - 1) x 32 KB of HBM reads stay in flight whatever it
// is computing. The part of a row inside one CTA's range is a segment; over a segment the CTA keeps every logit at
// or above a running lower bound of the segment's M-th largest (the M-th largest lane maximum of the segment's
// first stage, then the M-th largest candidate after each compaction), so after the first stage most stages cost
// one packed compare per two logits. A segment ends with its exact top-M; a row split over several CTAs is merged
// by the last of them (ticket), as in the per-chunk kernel.
constexpr int kSThreads = 256;
constexpr int kSStages = 3;
constexpr int kSElems = 16384;  // logits per stage, = the per-chunk kernel's chunk (same workspace layout)
constexpr int kSCap = 1024;     // candidate words of a segment
constexpr int kSMaxM = 128;     // the first bound takes the M-th of 256 lane maxima: keep M <= half of them

struct StreamSmem {
  uint4 ring[kSStages][kSElems * 2 / 16];
  uint64_t cand[kSCap];
  uint64_t tmp[kSMaxM];
  uint64_t full[kSStages];  // mbarriers
  uint32_t tmax[kSThreads];
  unsigned hist[256];
  int warp[kSThreads / 32];
  unsigned sel[2];
  uint64_t beta;
  uint32_t theta;
  int n;
  int flag;
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// Waits for the phase of `bar` with the given parity, at most `budget_ns`; false when the budget ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, uint64_t budget_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > budget_ns) return false;
  return true;
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// The M-th largest 16-bit key among the candidate words cand[0, n), n >= M (block-wide, two 8-bit histogram
// passes: the high byte, then the low byte within the chosen high byte).
template <int kThreads>
__device__ uint32_t kth_key16(const uint64_t* cand, int n, int M, unsigned* hist, unsigned* sel) {
  const int t = threadIdx.x, lane = t & 31;
  uint32_t prefix = 0;
  int need = M;
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 8 : 0;
    for (int i = t; i < 256; i += kThreads) hist[i] = 0u;
    __syncthreads();
    for (int i = t; i < n; i += kThreads) {
      const uint32_t key = candidate_key(cand[i]);
      if (pass == 0 || (key >> 8) == (prefix >> 8)) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (t < 32) {  // lane L holds bins 255 - 8L down to 248 - 8L: counts from the top
      unsigned c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        sum += c[j];
      }
      unsigned incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned excl = incl - sum;
      if (excl < static_cast<unsigned>(need) && incl >= static_cast<unsigned>(need)) {
        unsigned acc = excl;
        int j = 0;
        while (j < 7 && acc + c[j] < static_cast<unsigned>(need)) acc += c[j++];
        sel[0] = static_cast<unsigned>(255 - 8 * lane - j);
        sel[1] = acc;
      }
    }
    __syncthreads();
    prefix |= sel[0] << shift;
    need -= static_cast<int>(sel[1]);
    __syncthreads();
  }
  return prefix;
}

constexpr uint64_t kStageWaitNs = 4000000000ull;  // a 32 KB copy takes microseconds; this only stops a lost one

__global__ void __launch_bounds__(kSThreads, 2)
    topm_stream_kernel(const uint16_t* __restrict__ logits, int V, int M, int S, unsigned long long T,
                       uint64_t* __restrict__ lists, unsigned* __restrict__ tickets, int32_t* __restrict__ out_ids,
                       float* __restrict__ out_vals, WsHeader* hdr) {
  using X = Topm<true, kSThreads>;
  extern __shared__ uint4 smem_u4[];
  StreamSmem& s = *reinterpret_cast<StreamSmem*>(smem_u4);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const unsigned long long G = gridDim.x, c = blockIdx.x;
  const unsigned long long q0 = c * T / G, q1 = (c + 1) * T / G;  // this CTA's stages [q0, q1)
  // the CTA whose range holds stage q
  auto owner = [&](unsigned long long q) { return ((q + 1) * G + T - 1) / T - 1; };
  auto issue = [&](unsigned long long q) {
    const int st = static_cast<int>((q - q0) % kSStages);
    const unsigned long long row = q / S;
    const int c0 = static_cast<int>(q % S) * kSElems;
    const unsigned bytes = static_cast<unsigned>(min(kSElems, V - c0)) * 2u;  // a multiple of 16 (V % 8 == 0)
    mbar_expect_tx(&s.full[st], bytes);
    bulk_load(s.ring[st], logits + row * V + c0, bytes, &s.full[st]);
  };
  if (t == 0) {
    for (int i = 0; i < kSStages; ++i) mbar_init(&s.full[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (unsigned long long q = q0; q < q1 && q < q0 + kSStages; ++q) issue(q);
  }
  __syncthreads();

  bool nan = false;
  unsigned long long q = q0;
  for (; q < q1; ++q) {
    const unsigned long long row = q / S;
    const int j = static_cast<int>(q % S);
    const int st = static_cast<int>((q - q0) % kSStages);
    const unsigned parity = static_cast<unsigned>((q - q0) / kSStages) & 1u;
    const int c0 = j * kSElems, len = min(kSElems, V - c0);
    const bool seg_first = q == q0 || j == 0, seg_last = q + 1 == q1 || j == S - 1;
    const bool landed = mbar_wait(&s.full[st], parity, kStageWaitNs);
    if (__syncthreads_or(!landed)) break;
    X x;
#pragma unroll
    for (int k = 0; k < X::kGroups; ++k) {
      const int gi = t + kSThreads * k;
      x.g[k] = gi * 8 < len ? s.ring[st][gi] : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    }
    // Candidates before this stage, read while nobody can append: every thread must see the same count, since
    // branches that hold barriers depend on it.
    const int n0 = seg_first ? 0 : s.n;
    unsigned live = 0;  // groups of this thread inside the stage (whole groups: len is a multiple of 8)
#pragma unroll
    for (int k = 0; k < X::kGroups; ++k) live |= static_cast<unsigned>((t + kSThreads * k) * 8 < len) << k;
    __syncthreads();  // every thread holds its logits: the stage is refilled
    if (t == 0 && q + kSStages < q1) issue(q + kSStages);

    const uint32_t mx = x.max_key(nan);
    if (seg_first) {
      s.tmax[t] = mx;
      if (t == 0) s.n = 0;
      __syncthreads();
      if (warp == 0) {
        const uint32_t th = warp_kth_key<16, kSThreads>(s.tmax, M);
        if (t == 0) s.theta = th;
      }
      __syncthreads();
    }
    // Appends this stage's logits at or above theta. Per thread an 8-bit mask per selected group; one shared
    // atomic per warp reserves the warp's slots (lane offsets by a shuffle scan); positions past kSCap are dropped
    // and show up as s.n > kSCap.
    auto append = [&](uint32_t theta) {
      const uint32_t thr = theta ? ((theta & 0x8000u) ? (theta & 0x7FFFu) : (~theta & 0xFFFFu)) : 0xFF80u;
      const __nv_bfloat162 th2 = as_bf2(thr | (thr << 16));
      const unsigned sel = x.group_mask(thr) & live;
      uint64_t em = 0;
      int cnt = 0;
#pragma unroll
      for (int k = 0; k < X::kGroups; ++k) {
        if ((sel >> k) & 1u) {
          const uint4 v = x.g[k];
          const uint32_t q0m = __hge2_mask(as_bf2(v.x), th2), q1m = __hge2_mask(as_bf2(v.y), th2);
          const uint32_t q2m = __hge2_mask(as_bf2(v.z), th2), q3m = __hge2_mask(as_bf2(v.w), th2);
          const uint32_t m8 = (q0m & 1u) | ((q0m >> 15) & 2u) | ((q1m & 1u) << 2) | ((q1m >> 13) & 8u) |
                              ((q2m & 1u) << 4) | ((q2m >> 11) & 32u) | ((q3m & 1u) << 6) | ((q3m >> 9) & 128u);
          em |= static_cast<uint64_t>(m8) << (8 * k);
          cnt += __popc(m8);
        }
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const int wtotal = __shfl_sync(0xFFFFFFFFu, incl, 31);
      if (wtotal == 0) return;
      int base = 0;
      if (lane == 31) base = atomicAdd(&s.n, wtotal);
      int pos = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - cnt;
#pragma unroll
      for (int k = 0; k < X::kGroups; ++k) {
        uint32_t m = static_cast<uint32_t>(em >> (8 * k)) & 255u;
        if (m == 0u) continue;
        const uint4 v = x.g[k];
        const int li0 = (t + kSThreads * k) * 8;
        for (; m; m &= m - 1u, ++pos) {
          const int e = __ffs(m) - 1;
          const uint32_t word = e < 4 ? (e < 2 ? v.x : v.y) : (e < 6 ? v.z : v.w);
          const uint32_t bits = (word >> (16 * (e & 1))) & 0xFFFFu;
          if (pos < kSCap) s.cand[pos] = pack_candidate(key_of_bf16(bits), static_cast<uint32_t>(c0 + li0 + e));
        }
      }
    };
    // Raises theta to the exact M-th largest key of the n >= M candidates (radix select) and, when `filter`, keeps
    // only the candidates at or above it (M plus the ties at theta), in their order. Both are O(n).
    auto tighten = [&](bool filter) {
      const int n = s.n;
      const uint32_t th = kth_key16<kSThreads>(s.cand, n, M, s.hist, s.sel);
      if (t == 0) s.theta = max(s.theta, th);
      if (!filter) return;
      uint64_t w[kSCap / kSThreads];
      int mine = 0;
#pragma unroll
      for (int k = 0; k < kSCap / kSThreads; ++k) {
        const int i = t + kSThreads * k;
        w[k] = i < n ? s.cand[i] : 0ull;
        if (w[k] && candidate_key(w[k]) < th) w[k] = 0ull;
        mine += w[k] != 0ull;
      }
      int total = 0;
      int off = block_exclusive_scan<kSThreads / 32>(mine, &total, s.warp);  // its barriers order reads before writes
#pragma unroll
      for (int k = 0; k < kSCap / kSThreads; ++k)
        if (w[k]) s.cand[off++] = w[k];
      if (t == 0) s.n = total;
      __syncthreads();
    };
    append(s.theta);
    __syncthreads();
    if (s.n > kSCap) {
      // The stage overflowed the buffer: drop its candidates, tighten the bound on the earlier ones, try again.
      __syncthreads();
      if (t == 0) s.n = n0;
      __syncthreads();
      if (n0 >= M) tighten(true);
      const int n1 = s.n;
      __syncthreads();  // every thread has read n1 before anyone appends
      append(s.theta);
      __syncthreads();
      if (s.n > kSCap) {
        // Heavy ties at the bound: the exact M-th largest word of the segment so far (candidates + this stage,
        // re-read from memory) by bisection; keep exactly the words at or above it.
        __syncthreads();
        const long long row_off = static_cast<long long>(row) * V + c0;
        auto word_at = [&](int li) -> uint64_t {
          const uint32_t bits = logits[row_off + li];
          return is_nan_bf16(bits) ? 0ull : pack_candidate(key_of_bf16(bits), static_cast<uint32_t>(c0 + li));
        };
        const uint64_t kth = block_kth_largest<kSThreads / 32, uint64_t>(
            M, 63,
            [&](uint64_t cw) {
              int cnt = 0;
              for (int i = t; i < n1; i += kSThreads) cnt += s.cand[i] >= cw;
              for (int li = t; li < len; li += kSThreads) cnt += word_at(li) >= cw;
              return cnt;
            },
            s.warp);
        if (t == 0) s.n = 0;
        __syncthreads();
        for (int i = t; i < n1; i += kSThreads)
          if (s.cand[i] >= kth) s.tmp[atomicAdd(&s.n, 1)] = s.cand[i];
        for (int li = t; li < len; li += kSThreads) {
          const uint64_t w = word_at(li);
          if (w && w >= kth) s.tmp[atomicAdd(&s.n, 1)] = w;
        }
        __syncthreads();
        const int got = s.n;
        for (int i = t; i < got; i += kSThreads) s.cand[i] = s.tmp[i];
        if (t == 0 && kth) s.theta = max(s.theta, candidate_key(kth));
        __syncthreads();
      }
    } else if (!seg_last && s.n > 2 * M) {
      tighten(true);  // the bound rises with what has been seen; the buffer stays small
    }

    if (seg_last) {
      if (s.n > M) tighten(true);  // exactly the M-th key: M words plus its ties remain to be ranked
      const int n = s.n;
      rank_and_emit<kSThreads>(s.cand, n, M, s.tmp, [](uint64_t w) { return w; });
      __syncthreads();
      const long long cf = static_cast<long long>(owner(row * S)), cl = static_cast<long long>(owner(row * S + S - 1));
      const int nseg = static_cast<int>(cl - cf + 1);
      const long long row_out = static_cast<long long>(row) * M;
      if (nseg == 1) {
        emit_final<true, kSThreads>(s.tmp, M, out_ids + row_out, out_vals + row_out);
      } else {
        uint64_t* row_lists = lists + static_cast<long long>(row) * S * M;
        uint64_t* my_list = row_lists + (static_cast<long long>(c) - cf) * M;
        for (int i = t; i < M; i += kSThreads) my_list[i] = s.tmp[i];
        __syncthreads();
        if (t == 0) {
          __threadfence();
          s.flag = atomicAdd(&tickets[row], 1u) == static_cast<unsigned>(nseg - 1);
        }
        __syncthreads();
        if (s.flag) {
          if (t == 0) {
            __threadfence();
            tickets[row] = 0u;
          }
          const int entries = nseg * M;
          if (entries <= kSCap) {
            // The row's lists into shared memory, then the merge bound (M-th largest of the first q words of every
            // list), an in-place filter and the exact ranking, all on shared memory.
            for (int i = t; i < entries; i += kSThreads) s.cand[i] = __ldcg(row_lists + i);
            if (t == 0) s.beta = 0;
            __syncthreads();
            const int qh = (M + nseg - 1) / nseg, pn = nseg * qh;
            for (int i = t; i < pn; i += kSThreads) {
              const uint64_t wi = s.cand[(i / qh) * M + (i % qh)];
              if (wi == 0) continue;
              int r = 0;
              for (int jj = 0; jj < pn; ++jj) r += s.cand[(jj / qh) * M + (jj % qh)] > wi;
              if (r == M - 1) s.beta = wi;
            }
            __syncthreads();
            const uint64_t bound = s.beta ? s.beta : 1ull;
            uint64_t w[kSCap / kSThreads];
            int mine = 0;
#pragma unroll
            for (int k = 0; k < kSCap / kSThreads; ++k) {
              const int i = t + kSThreads * k;
              w[k] = i < entries ? s.cand[i] : 0ull;
              if (w[k] < bound) w[k] = 0ull;
              mine += w[k] != 0ull;
            }
            int kept = 0;
            int off = block_exclusive_scan<kSThreads / 32>(mine, &kept, s.warp);
#pragma unroll
            for (int k = 0; k < kSCap / kSThreads; ++k)
              if (w[k]) s.cand[off++] = w[k];
            __syncthreads();
            rank_and_emit<kSThreads>(s.cand, kept, M, s.tmp, [](uint64_t x) { return x; });
            __syncthreads();
            emit_final<true, kSThreads>(s.tmp, M, out_ids + row_out, out_vals + row_out);
          } else {
            merge_lists<true, kSThreads, kSCap>([&](int i) { return __ldcg(row_lists + i); }, nseg, M, s.cand,
                                                s.tmp, s.warp, &s.beta, out_ids + row_out, out_vals + row_out);
          }
        }
      }
      __syncthreads();
    }
  }
  if (q < q1) {
    // A stage copy never landed: report it, give the copies still in flight a bounded wait, and stop.
    if (t == 0) {
      record_error(hdr, DT_ERR_TIMEOUT);
      for (unsigned long long r = q; r < q1 && r < q + kSStages; ++r)
        mbar_wait(&s.full[(r - q0) % kSStages], static_cast<unsigned>((r - q0) / kSStages) & 1u, kStageWaitNs);
    }
    __syncthreads();
    return;
  }
  if (__syncthreads_or(nan) && t == 0) record_error(hdr, DT_ERR_NUMERIC);
}

// The streaming kernel needs its shared-memory size allowed once per device; the SM count sizes its grid.
constexpr int kMaxStreamDevices = 64;
std::atomic<int> g_stream_sms[kMaxStreamDevices];

bool stream_kernel_ready(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxStreamDevices) return false;
  int n = g_stream_sms[dev].load(std::memory_order_acquire);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return false;
    if (cudaFuncSetAttribute(topm_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(StreamSmem))) != cudaSuccess)
      return false;
    g_stream_sms[dev].store(n, std::memory_order_release);
  }
  *sms = n;
  return true;
}

dt_status launch_topm(const void* logits, dt_dtype dtype, int B, int K, int V, int M, int32_t* out_ids,
                      float* out_vals, char* ws, const TopmLayout& L, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * K;
  auto* hdr = reinterpret_cast<WsHeader*>(ws);
  auto* tickets = reinterpret_cast<unsigned*>(ws + L.tickets);
  auto* lists = reinterpret_cast<uint64_t*>(ws + L.lists);
  const size_t esize = dtype == DT_BF16 ? 2 : 4;
  const bool vec_ok = (static_cast<size_t>(V) * esize) % 16 == 0;
  if (dtype == DT_BF16 && vec_ok && M <= kSMaxM) {
    int sms = 0;
    if (!stream_kernel_ready(&sms)) return DT_ERR_CUDA;
    const unsigned long long T = static_cast<unsigned long long>(rows) * L.chunks;  // stages of the whole call
    const unsigned long long G = std::min<unsigned long long>(2ull * sms, T);
    topm_stream_kernel<<<static_cast<unsigned>(G), kSThreads, sizeof(StreamSmem), stream>>>(
        static_cast<const uint16_t*>(logits), V, M, L.chunks, T, lists, tickets, out_ids, out_vals, hdr);
    return cuda_status(cudaGetLastError());
  }
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
