// The top-M filter of one chunk of a logits row (dt_topm's filter kernel). Not part of the C ABI.
//
// A chunk is kThreads threads x kGroups 16-byte groups of logits, staged once into shared memory by cp.async (every
// group in flight together, no registers held). It keeps every logit at or above a lower bound of its row's M-th
// largest and appends those candidates, unsorted, to the row's per-chunk list in the workspace; the row's selection
// (topm_select.cuh) then ranks the few hundred candidates of all chunks. Every comparison is on distinct integer
// words, so the result is exact and deterministic, ties broken by the lower id.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "dt_internal.cuh"
#include "topm_select.cuh"

namespace dt {
namespace {

__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t v) { return *reinterpret_cast<__nv_bfloat162*>(&v); }

template <bool kBf16, int kThreads, int kGroups_ = 16>
struct Topm {
  static constexpr int kPer16 = kBf16 ? 8 : 4;  // logits per 16-byte load
  static constexpr int kGroups = kGroups_;      // 16-byte groups per thread (16 KB of shared memory per 256 threads x 4)
  static_assert(kGroups % 4 == 0 && kGroups <= 16, "whole parts; one 64-bit mask word holds half the groups");
  static constexpr int kParts = 4;              // copy groups committed per thread, waited for one by one
  static constexpr int kPartGroups = kGroups / kParts;
  static constexpr int kPer = kGroups * kPer16;  // logits per thread
  static constexpr int kChunk = kThreads * kPer;
  static constexpr int kKeyBits = kBf16 ? 16 : 32;
  // A chunk-local word: value key in the high part, 0xFFFF / 0xFFFFFFFF minus the local index in the low part.
  using CWord = typename std::conditional<kBf16, uint32_t, uint64_t>::type;
  static constexpr int kIdxBits = kBf16 ? 16 : 32;
  static_assert(kChunk <= 65536, "chunk-local index must fit 16 bits");

  // The chunk in shared memory, as loaded: thread t's 16-byte groups are s_[t + kThreads * k], k < kGroups.
  uint4* s_;
  __device__ __forceinline__ uint4 g_(int k) const { return s_[threadIdx.x + kThreads * k]; }

  // Bit pattern of the smallest value whose key is >= key (key 0: no bound, -inf).
  __device__ static __forceinline__ uint32_t thr_of(uint32_t key) {
    constexpr uint32_t kNegInf = kBf16 ? 0xFF80u : 0xFF800000u;
    constexpr uint32_t kMinKey = kBf16 ? 0x7Fu : 0x7FFFFFu;  // key of -inf: every real logit has a key >= it
    if (key <= kMinKey) return kNegInf;
    return kBf16 ? ((key & 0x8000u) ? (key & 0x7FFFu) : (~key & 0xFFFFu))
                 : ((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
  }
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

  // Stages this thread's logits into the shared chunk (16-byte groups t, t + kThreads, ...): whole groups inside
  // the row by cp.async (no registers held while the bytes are in flight), the rest element by element. Past the
  // end of the row the slots hold -inf, which never changes a maximum and is kept out of the candidates by its
  // index. The copies are committed in kParts groups of kPartGroups; a thread waits for its parts (wait_part) and
  // reads only the groups it staged itself, so no barrier is needed before it computes on them.
  __device__ __forceinline__ void stage(const void* logits, long long row_off, int c0, int len, bool vec_ok) const {
    const int t = threadIdx.x;
    constexpr uint32_t kPad = kBf16 ? 0xFF80FF80u : 0xFF800000u;
    constexpr long long kEsize = kBf16 ? 2 : 4;
    const char* src0 = static_cast<const char*>(logits) + (row_off + c0 + static_cast<long long>(t) * kPer16) * kEsize;
    const unsigned dst0 = static_cast<unsigned>(__cvta_generic_to_shared(s_ + t));
    if (vec_ok && len == kChunk) {  // a whole chunk: constant offsets, no tests
#pragma unroll
      for (int k = 0; k < kGroups; ++k) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                     ::"r"(dst0 + 16u * kThreads * k), "l"(src0 + 16ll * kThreads * k)
                     : "memory");
        if (k % kPartGroups == kPartGroups - 1) asm volatile("cp.async.commit_group;" ::: "memory");
      }
    } else {
#pragma unroll
      for (int k = 0; k < kGroups; ++k) {
        const int li0 = (t + kThreads * k) * kPer16;
        if (vec_ok && li0 + kPer16 <= len) {
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                       ::"r"(dst0 + 16u * kThreads * k), "l"(src0 + 16ll * kThreads * k)
                       : "memory");
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
          s_[t + kThreads * k] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (k % kPartGroups == kPartGroups - 1) asm volatile("cp.async.commit_group;" ::: "memory");
      }
    }
  }
  // Waits until the copies of this thread's parts 0 .. p have landed (a thread reads only its own staged groups).
  template <int p>
  __device__ static __forceinline__ void wait_part() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kParts - 1 - p) : "memory");
  }
  __device__ __forceinline__ bool any_nan_f32() const {
    bool nan = false;
#pragma unroll
    for (int k = 0; k < kGroups; ++k) {
      const uint4 v = g_(k);
      nan |= is_nan_f32(v.x) | is_nan_f32(v.y) | is_nan_f32(v.z) | is_nan_f32(v.w);
    }
    return nan;
  }

  // Key of this thread's largest non-NaN logit (0 if none); sets `nan` when a NaN is present (bf16).
  __device__ __forceinline__ uint32_t max_key(bool& nan) const {
    if (kBf16) {
      // four independent chains (x, y, z, w words), then combined: short dependency chains
      const uint4 v0 = g_(0);
      __nv_bfloat162 m0 = as_bf2(v0.x), m1 = as_bf2(v0.y), m2 = as_bf2(v0.z), m3 = as_bf2(v0.w);
#pragma unroll
      for (int k = 1; k < kGroups; ++k) {
        const uint4 v = g_(k);
        m0 = __hmax2_nan(m0, as_bf2(v.x));
        m1 = __hmax2_nan(m1, as_bf2(v.y));
        m2 = __hmax2_nan(m2, as_bf2(v.z));
        m3 = __hmax2_nan(m3, as_bf2(v.w));
      }
      __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(m0, m1), __hmax2_nan(m2, m3));
      uint32_t mw = as_u32(__hmax2_nan(m, __lowhigh2highlow(m))) & 0xFFFFu;
      if (is_nan_bf16(mw)) {  // rare: a NaN is present; take the maximum without it
        nan = true;
        m = as_bf2(0xFF80FF80u);
#pragma unroll
        for (int k = 0; k < kGroups; ++k) {
          const uint4 v = g_(k);
          m = __hmax2(m, as_bf2(v.x));
          m = __hmax2(m, as_bf2(v.y));
          m = __hmax2(m, as_bf2(v.z));
          m = __hmax2(m, as_bf2(v.w));
        }
        mw = as_u32(__hmax2(m, __lowhigh2highlow(m))) & 0xFFFFu;
        if (is_nan_bf16(mw)) return 0u;
      }
      return key_of_bf16(mw);
    } else {
      float m = -INFINITY;
#pragma unroll
      for (int k = 0; k < kGroups; ++k) {
        const uint4 v = g_(k);
        m = fmaxf(fmaxf(m, __uint_as_float(v.x)), fmaxf(__uint_as_float(v.y), fmaxf(__uint_as_float(v.z), __uint_as_float(v.w))));
      }
      return is_nan_f32(__float_as_uint(m)) ? 0u : key_of_f32(__float_as_uint(m));
    }
  }

  // Bit k of the result is set when 16-byte group k of this thread holds a logit >= the threshold value (NaN never
  // does; padding may, and is dropped by index later). Fully unrolled, the logits stay in registers; for bf16 one
  // packed compare covers two logits and the common "nothing here" group costs five instructions.
  // With kNan (bf16), the same pass also folds the groups into a NaN-propagating maximum and sets `nan` when a NaN
  // is present: one pass over the chunk when the bound is known in advance.
  template <bool kNan = false, int kFrom = 0, int kTo = kGroups>
  __device__ __forceinline__ unsigned group_mask(uint32_t thr_bits, bool* nan = nullptr) const {
    unsigned sel = 0;
    if (kBf16) {
      const __nv_bfloat162 th = as_bf2(thr_bits | (thr_bits << 16));
      __nv_bfloat162 mx = as_bf2(0xFF80FF80u);
#pragma unroll
      for (int k = kFrom; k < kTo; ++k) {
        const uint4 v = g_(k);
        const unsigned any = __hge2_mask(as_bf2(v.x), th) | __hge2_mask(as_bf2(v.y), th) |
                             __hge2_mask(as_bf2(v.z), th) | __hge2_mask(as_bf2(v.w), th);
        sel |= (any != 0u) << k;
        if (kNan)
          mx = __hmax2_nan(mx, __hmax2_nan(__hmax2_nan(as_bf2(v.x), as_bf2(v.y)), __hmax2_nan(as_bf2(v.z), as_bf2(v.w))));
      }
      if (kNan) {
        const uint32_t w = as_u32(mx);
        *nan |= is_nan_bf16(w) | is_nan_bf16(w >> 16);
      }
    } else {
      const float th = __uint_as_float(thr_bits);
#pragma unroll
      for (int k = kFrom; k < kTo; ++k) {
        const uint4 v = g_(k);
        const bool any = __uint_as_float(v.x) >= th || __uint_as_float(v.y) >= th || __uint_as_float(v.z) >= th ||
                         __uint_as_float(v.w) >= th;
        sel |= static_cast<unsigned>(any) << k;
      }
    }
    return sel;
  }
  // Bits of element e (0 <= e < kPer16) of group k (k, e compile-time after unrolling, or a short select chain).
  __device__ __forceinline__ uint32_t element_bits(int k, int e) const {
    const uint4 v = g_(k);
    if (kBf16) {
      const uint32_t w = e < 4 ? (e < 2 ? v.x : v.y) : (e < 6 ? v.z : v.w);
      return (w >> (16 * (e & 1))) & 0xFFFFu;
    }
    return e < 2 ? (e == 0 ? v.x : v.y) : (e == 2 ? v.z : v.w);
  }
  // Bit e: element e of group k lies inside the row (local index < len) and its value is >= (kEq: ==) the value
  // with bit pattern thr. NaNs never qualify; -0.0 and +0.0 compare equal. For bf16 four packed compares.
  template <bool kEq>
  __device__ __forceinline__ uint32_t elem_mask(int k, uint32_t thr, int len) const {
    const int li0 = (static_cast<int>(threadIdx.x) + kThreads * k) * kPer16;
    const uint4 v = g_(k);
    uint32_t m;
    if (kBf16) {
      const __nv_bfloat162 th = as_bf2(thr | (thr << 16));
      const uint32_t a = kEq ? __heq2_mask(as_bf2(v.x), th) : __hge2_mask(as_bf2(v.x), th);
      const uint32_t b = kEq ? __heq2_mask(as_bf2(v.y), th) : __hge2_mask(as_bf2(v.y), th);
      const uint32_t c = kEq ? __heq2_mask(as_bf2(v.z), th) : __hge2_mask(as_bf2(v.z), th);
      const uint32_t d = kEq ? __heq2_mask(as_bf2(v.w), th) : __hge2_mask(as_bf2(v.w), th);
      m = (a & 1u) | ((a >> 15) & 2u) | ((b & 1u) << 2) | ((b >> 13) & 8u) | ((c & 1u) << 4) | ((c >> 11) & 32u) |
          ((d & 1u) << 6) | ((d >> 9) & 128u);
    } else {
      const float th = __uint_as_float(thr);
      auto q = [&](uint32_t bits) -> uint32_t {
        const float f = __uint_as_float(bits);
        return kEq ? (f == th) : (f >= th);
      };
      m = q(v.x) | (q(v.y) << 1) | (q(v.z) << 2) | (q(v.w) << 3);
    }
    const int valid = len - li0;
    return valid >= kPer16 ? m : (valid > 0 ? (m & ((1u << valid) - 1u)) : 0u);
  }
  // Group k of this thread's registers, for a run-time k (a select chain, no local memory).
  __device__ __forceinline__ uint4 group(int k) const {
    uint4 v = g_(0);
#pragma unroll
    for (int j = 1; j < kGroups; ++j)
      if (k == j) v = g_(j);
    return v;
  }
  __device__ static __forceinline__ int local_index(int e) {
    return (static_cast<int>(threadIdx.x) + kThreads * (e / kPer16)) * kPer16 + (e % kPer16);
  }
};

// Warp 0 (threads 0..31): the 256-bin histogram `hist`, read from the top, places the need-th largest key in bin
// s_sel[0], with s_sel[1] keys in the bins above it. Requires at least `need` keys in the histogram.
__device__ __forceinline__ void pick_from_top(const unsigned* hist, int need, unsigned* s_sel) {
  const int lane = threadIdx.x & 31;
  unsigned cb[8], sum = 0;  // lane L holds bins 255 - 8L down to 248 - 8L: counts from the top
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
    s_sel[0] = static_cast<unsigned>(255 - 8 * lane - j);
    s_sel[1] = acc;
  }
}

// The M-th largest of the block's keys, one per thread (1 <= M <= kThreads), in every thread: radix select with
// 8-bit digits from the top, one 256-bin shared histogram per digit over the keys that share the digits found so far.
template <int kKeyBits, int kThreads>
__device__ __forceinline__ uint32_t block_kth_key(uint32_t key, int M, unsigned* hist, unsigned* s_sel) {
  static_assert(kThreads >= 256, "one histogram bin per thread");
  const int t = threadIdx.x, lane = t & 31;
  uint32_t prefix = 0;
  int need = M;
#pragma unroll
  for (int d = kKeyBits / 8 - 1; d >= 0; --d) {
    if (t < 256) hist[t] = 0u;
    __syncthreads();
    const bool match = d == kKeyBits / 8 - 1 || (key >> (8 * (d + 1))) == prefix;
    // lanes with the same digit add together (the keys are lane maxima of one row: few distinct top digits)
    const unsigned digit = (key >> (8 * d)) & 255u;
    const unsigned active = __ballot_sync(0xFFFFFFFFu, match);
    if (match) {
      const unsigned peers = __match_any_sync(active, digit);
      if (lane == __ffs(peers) - 1) atomicAdd(&hist[digit], static_cast<unsigned>(__popc(peers)));
    }
    __syncthreads();
    if (t < 32) pick_from_top(hist, need, s_sel);
    __syncthreads();
    prefix = (prefix << 8) | s_sel[0];
    need -= static_cast<int>(s_sel[1]);
    __syncthreads();  // s_sel and hist are rewritten by the next digit
  }
  return prefix;
}

constexpr int kCandMax = 1024;  // >= topm_cap(M) for every supported M

// The filter's shared state besides the staged chunk.
template <bool kBf16, int kThreads>
struct FilterShared {
  using CWord = typename std::conditional<kBf16, uint32_t, uint64_t>::type;
  CWord cand[kCandMax];
  unsigned tmax[256];  // the bound's digit histogram
  unsigned s_sel[2];
  int s_warp[kThreads / 32];
  uint32_t s_theta;
  int s_n;
};

// Keeps the chunk's candidates: every logit at or above the bound key F.s_theta (0: no bound), appended unsorted to
// F.cand as chunk-local words (value key << bits | inverted local index), their count in F.s_n. `sel_known`, when
// `have_sel` (bf16): the groups already found to hold a logit at or above the bound. More than `cap` survivors (ties,
// or sorted runs that put the large logits in few lanes): exactly the chunk's top M instead, by bisection over the
// staged chunk and the lowest-index ties. A NaN among the logits (`nan` in any thread) sets DT_ERR_NUMERIC. Called by
// all kThreads threads after a barrier that follows the write of F.s_theta; returns the count in every thread.
template <bool kBf16, int kThreads, int kGroups>
__device__ int chunk_keep(const Topm<kBf16, kThreads, kGroups>& x, int M, int len, int cap, bool have_sel,
                          unsigned sel_known, bool nan, WsHeader* hdr, FilterShared<kBf16, kThreads>& F) {
  using T = Topm<kBf16, kThreads, kGroups>;
  constexpr int kWarps = kThreads / 32;
  constexpr int kHalf = T::kGroups / 2;  // groups per 64-bit mask word
  auto* cand = F.cand;
  const int t = threadIdx.x, lane = t & 31;
  // Appends the elements whose bits are set in e0 (groups 0..kHalf-1) and e1 (the rest), kPer16 bits per group. One
  // shared atomic per warp reserves the warp's slots; slots past cap are dropped (and show up as s_n > cap). The
  // chunk is in shared memory, so groups are visited by run-time index (no unrolling, few registers).
  auto append = [&](uint64_t e0, uint64_t e1) {
    const int cnt = __popcll(e0) + __popcll(e1);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const int wtotal = __shfl_sync(0xFFFFFFFFu, incl, 31);
    if (wtotal == 0) return;
    int base = 0;
    if (lane == 31) base = atomicAdd(&F.s_n, wtotal);
    int pos = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - cnt;
    constexpr uint32_t kGroupBits = (1u << T::kPer16) - 1u;
    unsigned gm = 0;  // groups that hold candidates
#pragma unroll
    for (int k = 0; k < T::kGroups; ++k)
      gm |= static_cast<unsigned>(((k < kHalf ? e0 : e1) >> (T::kPer16 * (k % kHalf))) & kGroupBits ? 1u : 0u) << k;
#pragma unroll 1
    for (; gm; gm &= gm - 1u) {
      const int k = __ffs(gm) - 1;
      uint32_t m = static_cast<uint32_t>((k < kHalf ? e0 : e1) >> (T::kPer16 * (k % kHalf))) & kGroupBits;
      const int li0 = (t + kThreads * k) * T::kPer16;
      for (; m; m &= m - 1u, ++pos) {
        const int e = __ffs(m) - 1;
        if (pos < cap) cand[pos] = T::cword(x.element_bits(k, e), li0 + e);
      }
    }
  };
  // e0 / e1 of the elements at or above (kEq: equal to) thr in the groups whose bits are set in sel.
  auto masks = [&](unsigned sel, uint32_t thr, bool eq, uint64_t& e0, uint64_t& e1) {
    e0 = e1 = 0;
#pragma unroll 1
    for (; sel; sel &= sel - 1u) {
      const int k = __ffs(sel) - 1;
      const uint64_t m = eq ? x.template elem_mask<true>(k, thr, len) : x.template elem_mask<false>(k, thr, len);
      if (k < kHalf) e0 |= m << (T::kPer16 * k);
      else e1 |= m << (T::kPer16 * (k - kHalf));
    }
  };
  constexpr unsigned kAllGroups = (1u << T::kGroups) - 1u;

  {
    const uint32_t thr = T::thr_of(F.s_theta);
    uint64_t e0, e1;
    // cheap "anything here" test first, unless the caller's pass already found the groups
    const unsigned sel = have_sel ? sel_known : x.group_mask(thr);
    masks(sel, thr, false, e0, e1);
    append(e0, e1);
  }
  if (__syncthreads_or(nan) && t == 0) record_error(hdr, DT_ERR_NUMERIC);
  int n = F.s_n;
  if (n > cap) {
    // Exactly the top M. kth: the largest key with at least M elements at or above it (bisection, counts from the
    // staged chunk); then all elements above kth and the lowest-index ties at kth, layer by layer in index order.
    auto count_ge = [&](uint32_t key) {
      const uint32_t thr = T::thr_of(key);
      int c = 0;
#pragma unroll 1
      for (int k = 0; k < T::kGroups; ++k) c += __popc(x.template elem_mask<false>(k, thr, len));
      return c;
    };
    uint32_t kth = 0;
    for (int bit = T::kKeyBits - 1; bit >= 0; --bit) {
      const uint32_t cnd = kth | (1u << bit);
      if (block_sum<kWarps>(count_ge(cnd), F.s_warp) >= M) kth = cnd;
    }
    int need = M - block_sum<kWarps>(count_ge(kth + 1u), F.s_warp);  // ties at kth still to take (>= 1)
    if (t == 0) F.s_n = 0;
    __syncthreads();
    {
      uint64_t e0, e1;
      masks(kAllGroups, T::thr_of(kth + 1u), false, e0, e1);
      append(e0, e1);
    }
    const uint32_t thr_eq = T::thr_of(kth);
#pragma unroll 1
    for (int k = 0; k < T::kGroups; ++k) {  // layer k holds indices [k * kThreads * kPer16, (k + 1) * ...)
      if (need <= 0) break;                  // uniform
      uint32_t m = x.template elem_mask<true>(k, thr_eq, len);
      int layer = 0;
      const int before = block_exclusive_scan<kWarps>(__popc(m), &layer, F.s_warp);
      const int take = max(0, min(__popc(m), need - before));
      for (int i = __popc(m) - take; i > 0; --i) m &= ~(1u << (31 - __clz(m)));  // keep the `take` lowest
      const uint64_t em = static_cast<uint64_t>(m) << (T::kPer16 * (k % kHalf));
      append(k < kHalf ? em : 0ull, k < kHalf ? 0ull : em);
      need -= layer;
    }
    __syncthreads();
    n = F.s_n;
  }
  return n;
}

// Filters chunk `chunk` of row `row` (logits [row][V]): the chunk keeps every logit at or above the M-th largest of
// its kThreads lane maxima, or at or above the row's bound already published by another chunk (`bounds[row]`, the
// largest such bound so far; read before the copies are issued, so the load does not queue behind them), and
// publishes its own bound with atomicMax (chunk_keep does the rest). Writes the chunk's candidate words and their
// count to the row's list `chunk` in `words` / `counts` (rows x chunks lists of `cap` words). Called by all kThreads
// threads; `chunk_s` holds kThreads * kGroups 16-byte groups.
template <bool kBf16, int kThreads, int kGroups>
__device__ void filter_chunk(const void* __restrict__ logits, int V, int M, int row, int chunk, int chunks, int cap,
                             bool vec_ok, uint32_t* __restrict__ bounds, void* __restrict__ words,
                             int* __restrict__ counts, WsHeader* hdr, uint4* chunk_s, FilterShared<kBf16, kThreads>& F) {
  using T = Topm<kBf16, kThreads, kGroups>;
  using CWord = typename T::CWord;
  const int t = threadIdx.x;
  const long long row_off = static_cast<long long>(row) * V;
  const int c0 = chunk * T::kChunk;
  const int len = min(T::kChunk, V - c0);
  __syncthreads();  // the previous user of the shared state is done with it
  if (t == 0) {
    F.s_n = 0;
    F.s_theta = M <= kThreads ? *reinterpret_cast<volatile uint32_t*>(bounds + row) : 0u;
  }
  T x{chunk_s};
  x.stage(logits, row_off, c0, len, vec_ok);
  __syncthreads();
  const bool known = F.s_theta != 0u;  // uniform: written by thread 0 before the barrier
  bool nan = false;
  unsigned sel_known = 0;  // with a known bound (bf16): the groups holding candidates, found part by part
  if (kBf16 && known) {
    // each part is scanned as soon as this thread's copies of it have landed, while the later parts are in flight
    const uint32_t thr = T::thr_of(F.s_theta);
    T::template wait_part<0>();
    sel_known |= x.template group_mask<true, 0, T::kPartGroups>(thr, &nan);
    T::template wait_part<1>();
    sel_known |= x.template group_mask<true, T::kPartGroups, 2 * T::kPartGroups>(thr, &nan);
    T::template wait_part<2>();
    sel_known |= x.template group_mask<true, 2 * T::kPartGroups, 3 * T::kPartGroups>(thr, &nan);
    T::template wait_part<3>();
    sel_known |= x.template group_mask<true, 3 * T::kPartGroups, T::kGroups>(thr, &nan);
  } else {
    T::template wait_part<T::kParts - 1>();
    if (!kBf16) nan = x.any_nan_f32();
  }
  if (!known) {  // this chunk computes (and publishes) the bound
    const uint32_t mk = x.max_key(nan);
    if (M <= kThreads) {
      __syncthreads();  // every thread has read s_theta
      const uint32_t th = block_kth_key<T::kKeyBits, kThreads>(mk, M, F.tmax, F.s_sel);
      if (t == 0) {
        F.s_theta = th;
        if (th) atomicMax(bounds + row, th);
      }
      __syncthreads();
    }
  }
  const int n = chunk_keep(x, M, len, cap, kBf16 && known, sel_known, nan, hdr, F);
  CWord* out = static_cast<CWord*>(words) + (static_cast<size_t>(row) * chunks + chunk) * cap;
  for (int i = t; i < n; i += kThreads) out[i] = F.cand[i];
  if (t == 0) counts[static_cast<size_t>(row) * chunks + chunk] = n;
}

// The row's selection over the filter's per-chunk candidate lists (chunk-local words, turned into row words).
template <bool kBf16, int kThreads, int kGroups>
__device__ void select_row(int row, const void* __restrict__ words, const int* __restrict__ counts, int chunks,
                           int cap, int M, int32_t* __restrict__ out_ids, float* __restrict__ out_vals,
                           SelectSmem& S, int* s_warp, int* s_n_ptr) {
  using T = Topm<kBf16, kThreads, kGroups>;
  using CWord = typename T::CWord;
  const CWord* base = static_cast<const CWord*>(words) + static_cast<size_t>(row) * chunks * cap;
  const long long row_out = static_cast<long long>(row) * M;
  const int* cnt = counts + static_cast<size_t>(row) * chunks;
  select_words<kBf16, kThreads>(
      [&](int c) { return __ldcg(cnt + c); }, chunks, M,
      [&](int c, int i) { return T::global_word(__ldcg(base + static_cast<size_t>(c) * cap + i), c * T::kChunk); },
      out_ids + row_out, out_vals + row_out, S, s_warp, s_n_ptr);
}

}  // namespace
}  // namespace dt
