// The exact top-M of a row from a few lists of candidate words: shared by dt_topm's selection and the fused
// projection top-M. Every comparison is on distinct 64-bit words (value key, then inverted id), so the result is
// exact and deterministic, ties broken by the lower id.
#pragma once

#include <cuda_runtime.h>

#include "dt_internal.cuh"

namespace dt {
namespace {

// Lane L of warp 0 holds the counts cb[0..7] of bins 255 - 8L down to 248 - 8L, and `excl` words in the bins above
// them. Returns the first j with excl + cb[0] + ... + cb[j] >= need (7 if none before the last), and sets `acc` to
// the words above bin j and `at` to cb[j] (no run-time indexing of cb: it stays in registers).
__device__ __forceinline__ int pick_bin(const unsigned (&cb)[8], unsigned excl, unsigned need, unsigned& acc,
                                        unsigned& at) {
  acc = excl;
  int j = 0;
  bool stop = false;
#pragma unroll
  for (int i = 0; i < 7; ++i) {
    stop = stop || acc + cb[i] >= need;
    if (!stop) {
      acc += cb[i];
      j = i + 1;
    }
  }
  at = cb[0];
#pragma unroll
  for (int i = 1; i < 8; ++i)
    if (i == j) at = cb[i];
  return j;
}

// Ranks the `total` distinct words of cand; the M largest, in descending order, go to out[0..M). Slots past `total`
// get 0.
template <int kThreads>
__device__ __forceinline__ void rank_and_emit(const uint64_t* cand, int total, int M, uint64_t* out) {
  for (int i = threadIdx.x; i < total; i += kThreads) {
    const uint64_t ci = cand[i];
    int r = 0;
    for (int j = 0; j < total; ++j) r += cand[j] > ci;
    if (r < M) out[r] = ci;
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

// ---- the row's final selection (run by the row's last filter CTA) -----------------------------------------------
// The row's candidates (a few hundred words) as 64-bit words (value key, inverted row index), gathered into shared
// memory (the chunks' counts, their offsets by a scan, then the words). The M-th largest word is then bracketed by one histogram of the keys relative to the smallest candidate key (256 bins,
// as fine as the key range allows): the words of the bins at and above the bin holding the M-th largest are ranked
// by counting, and the first M are written out in order. When that bin holds too many words, the M-th largest word
// is found by radix select instead (8-bit digits from the top; stops once a digit's bin is taken whole, or once the
// key digits are fixed and the ties fit the ranking buffer). Candidates written by other CTAs are read through L2.
constexpr int kSelThreads = 256;
constexpr int kSelCap = 2048;                 // candidate words of a row kept in shared memory (more: re-read)
constexpr int kChunksPerThread = 1;
constexpr int kMaxChunks = kChunksPerThread * kSelThreads;  // chunk offsets kept in shared memory up to this many
struct SelectSmem {                           // lives in the caller's shared memory (the filter's chunk buffer)
  uint64_t w[kSelCap];
  uint64_t top[DT_MAX_M];                     // the words ranked by counting
  int off[kMaxChunks + 1];
  unsigned hist[256];
  unsigned sel[2];
  unsigned red[2][16];                        // per-warp key minima and maxima (up to 512 threads)
};

// The row's selection over `chunks` lists of candidate words: count(c) words in list c, word i of list c given by
// load(c, i) as a 64-bit row word (value key << 32 | ~id). kBf16: the keys are bf16 keys (16 bits), else fp32 keys.
// Writes the row's M ids and values (in order) to ids[0..M), vals[0..M). Called by all kThreads threads (256 or 512;
// s_warp holds kThreads / 32 ints).
template <bool kBf16, int kThreads, class Count, class Load>
__device__ void select_words(Count count, int chunks, int M, Load load, int32_t* __restrict__ ids,
                             float* __restrict__ vals, SelectSmem& S, int* s_warp, int* s_n_ptr) {
  static_assert(kThreads >= 256 && kThreads <= 512 && kThreads % 32 == 0, "one histogram bin per thread at most");
  constexpr int kWarps = kThreads / 32;
  constexpr int kTopDigit = kBf16 ? 5 : 7;  // bf16 keys are 16 bits: word bits 48..63 are zero
  uint64_t* w = S.w;
  uint64_t* top = S.top;
  int* s_off = S.off;
  unsigned* hist = S.hist;
  unsigned* sel = S.sel;
  int& s_n = *s_n_ptr;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  int total = 0;
  const bool few = chunks <= kMaxChunks;
  if (few) {  // per-chunk offsets of the row's candidates, one parallel load and a scan
    int mine = 0, c_of[kChunksPerThread];
#pragma unroll
    for (int j = 0; j < kChunksPerThread; ++j) {
      const int c = kChunksPerThread * t + j;
      c_of[j] = c < chunks ? count(c) : 0;
      mine += c_of[j];
    }
    int off = block_exclusive_scan<kWarps>(mine, &total, s_warp);
#pragma unroll
    for (int j = 0; j < kChunksPerThread; ++j) {
      const int c = kChunksPerThread * t + j;
      if (c <= chunks) s_off[c] = off;
      off += c_of[j];
    }
  } else {
    int mine = 0;
    for (int c = t; c < chunks; c += kThreads) mine += count(c);
    total = block_sum<kWarps>(mine, s_warp);
  }
  if (t == 0) s_n = 0;
  __syncthreads();
  const bool in_smem = few && total <= kSelCap;
  if (in_smem) {
    for (int i = t; i < total; i += kThreads) {
      int lo = 0, hi = chunks - 1;  // the chunk holding candidate i: the last offset <= i
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= i) lo = mid;
        else hi = mid - 1;
      }
      w[i] = load(lo, i - s_off[lo]);
    }
  }
  __syncthreads();
  auto for_each = [&](auto&& f) {
    if (in_smem) {
      for (int i = t; i < total; i += kThreads) f(w[i]);
    } else {
      for (int c = 0; c < chunks; ++c) {
        const int nc = count(c);
        for (int i = t; i < nc; i += kThreads) f(load(c, i));
      }
    }
  };
  uint64_t thresh = 0;  // take every word >= thresh
  bool bracketed = false;
  if (total > M && in_smem) {
    // the candidates' key range, then one histogram relative to its minimum
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
    for (int i = t; i < total; i += kThreads) {
      const uint32_t k = candidate_key(w[i]);
      kmin = min(kmin, k);
      kmax = max(kmax, k);
    }
    kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
    kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
    if (lane == 0) {
      S.red[0][warp] = kmin;
      S.red[1][warp] = kmax;
    }
    if (t < 256) hist[t] = 0u;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kWarps; ++i) {
      kmin = min(kmin, S.red[0][i]);
      kmax = max(kmax, S.red[1][i]);
    }
    int shift = 0;
    while (((kmax - kmin) >> shift) > 255u) ++shift;
    for (int i = t; i < total; i += kThreads) atomicAdd(&hist[(candidate_key(w[i]) - kmin) >> shift], 1u);
    __syncthreads();
    if (t < 32) {  // lane L holds bins 255 - 8L down to 248 - 8L: counts from the top
      unsigned cb[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cb[j] = hist[255 - 8 * lane - j];
        sum += cb[j];
      }
      unsigned incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned excl = incl - sum;
      if (excl < static_cast<unsigned>(M) && incl >= static_cast<unsigned>(M)) {
        unsigned acc, at;
        const int j = pick_bin(cb, excl, static_cast<unsigned>(M), acc, at);
        sel[0] = static_cast<unsigned>(255 - 8 * lane - j);  // the bin holding the M-th largest
        sel[1] = acc + at;                                    // words at or above it
      }
    }
    __syncthreads();
    if (sel[1] <= static_cast<unsigned>(DT_MAX_M)) {
      thresh = static_cast<uint64_t>(kmin + (sel[0] << shift)) << 32;  // the bin's smallest key, any index
      bracketed = true;
    }
  }
  if (total > M && !bracketed) {
    uint64_t prefix = 0, pmask = 0;
    int need = M;
    for (int d = kTopDigit; d >= 0; --d) {
      for (int i = t; i < 256; i += kThreads) hist[i] = 0u;
      __syncthreads();
      for_each([&](uint64_t wd) {
        if ((wd & pmask) == prefix) atomicAdd(&hist[(wd >> (8 * d)) & 255u], 1u);
      });
      __syncthreads();
      if (t < 32) {  // lane L holds bins 255 - 8L down to 248 - 8L: counts from the top
        unsigned cb[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          cb[j] = hist[255 - 8 * lane - j];
          sum += cb[j];
        }
        unsigned incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        const unsigned excl = incl - sum;
        if (excl < static_cast<unsigned>(need) && incl >= static_cast<unsigned>(need)) {
          unsigned acc, at;
          const int j = pick_bin(cb, excl, static_cast<unsigned>(need), acc, at);
          sel[0] = static_cast<unsigned>(255 - 8 * lane - j);
          sel[1] = acc;
        }
      }
      __syncthreads();
      const unsigned b = sel[0];
      prefix |= static_cast<uint64_t>(b) << (8 * d);
      pmask |= 0xFFull << (8 * d);
      need -= static_cast<int>(sel[1]);
      // Done when the bin is taken whole, or once the key digits are fixed and the words at or above the M-th key
      // (M - need above it, hist[b] at it) fit the ranking buffer: the ranking orders the ties by index.
      const bool whole = hist[b] == static_cast<unsigned>(need) ||
                         (d == 4 && M - need + static_cast<int>(hist[b]) <= DT_MAX_M);
      __syncthreads();
      if (whole) break;
    }
    thresh = prefix;
  }
  for_each([&](uint64_t wd) {
    if (wd >= thresh) top[atomicAdd(&s_n, 1)] = wd;
  });
  __syncthreads();
  const int m = s_n;  // the words ranked: min(M, total) up to the ranking buffer
  uint64_t* sorted = w;  // the row's words are no longer needed
  __syncthreads();
  rank_and_emit<kThreads>(top, m, M, sorted);
  __syncthreads();
  emit_final<kBf16, kThreads>(sorted, M, ids, vals);
}

}  // namespace
}  // namespace dt
