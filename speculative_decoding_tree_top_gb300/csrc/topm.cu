// dt_topm — top-M candidate restriction over the drafter's marginal logits.
//
// Method: blog.captcha.la, "Methodology — deep read" / "Technical innovations" (the per-node correction only sees
// the M highest-marginal tokens of each depth); gist.science, "Composants Clés — Restriction de Candidats".
//
// GB300 design. The op is a pure HBM stream (every logit is read once, nothing is reused), so it is laid out for
// bandwidth and for few instructions per logit, not for tensor cores. A few rows (one request's block positions)
// are latency-bound instead: each row is then one thread-block cluster that keeps everything in distributed shared
// memory (topm_cluster_kernel, below). Otherwise two launches:
//   * filter: grid = (B*K rows) x (chunks of 32768 bf16 / 16384 fp32 logits), 256 threads. Each thread stages its
//     sixteen 16-byte groups into shared memory with cp.async, committed as four parts, so all of a chunk's bytes
//     are in flight at once and no registers are held while they are. A row's first chunk computes the M-th
//     largest of its 256 lane maxima (radix over the key's bytes, one shared histogram per digit) and publishes it
//     as the row's bound; later chunks of the row read the published bound before their copies are issued and scan
//     each part as soon as it lands (packed bf16x2 compare-to-mask, one instruction per two logits). A chunk
//     appends its logits at or above the bound, unsorted, with their count (a few per chunk, M or more per row);
//   * select: one CTA per row, launched as a programmatic dependent of the filter so it takes the SMs the filter's
//     last wave leaves idle. A histogram of the candidates' keys brackets the row's exact M-th largest, and the M
//     at or above it are ranked by counting (a radix pass when the bracket holds too many).
// Every comparison is on distinct integer words (value key, then inverted index), so the result is exact and
// deterministic, ties broken by the lower id. A chunk with more survivors than its list holds (heavy ties, sorted
// runs) keeps exactly its top M instead (bisection over the staged chunk): slower, same result.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <mutex>
#include <type_traits>

#include "dt_internal.cuh"
#include "topm_filter.cuh"
#include "topm_select.cuh"

namespace dt {
namespace {

// ---- kernel 1: filter ----------------------------------------------------------------------------------------------
// One CTA per (chunk, row); a chunk is 256 threads x 16 groups of 16 bytes (32768 bf16 or 16384 fp32 logits), filtered
// by filter_chunk (topm_filter.cuh).
constexpr int kFThreads = 256;
constexpr int kFGroups = 16;
constexpr size_t kChunkSmem = static_cast<size_t>(kFThreads) * kFGroups * 16;  // 64 KB: the staged chunk

static_assert(sizeof(SelectSmem) <= kChunkSmem, "the selection fits the filter's chunk buffer");

// kFuse: the row's last CTA (ticket) runs the selection itself: one launch, best for small grids; with many rows
// the per-CTA fence and ticket cost more than a second launch (topm_select_kernel).
template <bool kBf16, bool kFuse>
__global__ void __launch_bounds__(kFThreads, 3)
    topm_filter_kernel(const void* __restrict__ logits, int V, int M, int chunks, int cap, bool vec_ok,
                       uint32_t* __restrict__ bounds, unsigned* __restrict__ tickets, void* __restrict__ words,
                       int* __restrict__ counts, int32_t* __restrict__ out_ids, float* __restrict__ out_vals,
                       WsHeader* hdr) {
  extern __shared__ uint4 chunk_s[];
  __shared__ FilterShared<kBf16, kFThreads> F;
  // rows vary fastest: a row's first chunk runs (and publishes the row's bound) before its later chunks start
  const int row = blockIdx.x, chunk = blockIdx.y, t = threadIdx.x;
  // every CTA of the grid has started once all have passed here: the selection launch may then take the SMs that
  // the filter's last wave leaves free (it waits for the filter's completion before reading anything)
  if (!kFuse) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  filter_chunk<kBf16, kFThreads, kFGroups>(logits, V, M, row, chunk, chunks, cap, vec_ok, bounds, words, counts, hdr,
                                           chunk_s, F);
  if (!kFuse) return;

  // The last CTA of the row to finish selects the row's top M. The barrier orders every thread's writes before
  // thread 0's fence, which publishes them at device scope before the ticket.
  __syncthreads();
  if (t == 0) {
    __threadfence();
    F.s_theta = atomicAdd(tickets + row, 1u) == static_cast<unsigned>(chunks - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (F.s_theta == 0u) return;
  if (t == 0) {
    __threadfence();
    tickets[row] = 0u;  // both zero for the next call
    bounds[row] = 0u;
  }
  select_row<kBf16, kFThreads, kFGroups>(row, words, counts, chunks, cap, M, out_ids, out_vals,
                                         *reinterpret_cast<SelectSmem*>(chunk_s), F.s_warp, &F.s_n);
}

template <bool kBf16>
__global__ void __launch_bounds__(kSelThreads, 7) topm_select_kernel(const void* __restrict__ words,
                                                                  const int* __restrict__ counts, int chunks, int cap,
                                                                  int M, uint32_t* __restrict__ bounds,
                                                                  int32_t* __restrict__ out_ids,
                                                                  float* __restrict__ out_vals) {
  extern __shared__ uint4 smem_u4[];
  __shared__ int s_warp[kSelThreads / 32];
  __shared__ int s_n;
  // Launched as a programmatic dependent of the filter: the CTAs may start while its last CTAs still run, and wait
  // here until that launch has completed and its writes are visible (a no-op after an ordinary launch).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) bounds[blockIdx.x] = 0u;  // the filter launch has finished with it: zero for the next call
  select_row<kBf16, kSelThreads, kFGroups>(blockIdx.x, words, counts, chunks, cap, M, out_ids, out_vals,
                                           *reinterpret_cast<SelectSmem*>(smem_u4), s_warp, &s_n);
}

// ---- one cluster per row: small grids ---------------------------------------------------------------------------
// For few rows (a single request's block positions) the chunk-list path is a chain of global round trips: the
// published bound, the candidate lists, the ticket, the last CTA's selection over words read back from L2. Here a
// row is one thread-block cluster of C CTAs (C <= 8), CTA c holding the slice [c * slice, (c + 1) * slice) of the
// row in shared memory, and the CTAs write into each other's shared memory (two cluster barriers in all):
//   1. each CTA bulk-copies its slice in (TMA, one mbarrier) and pads the rest of its chunk buffer with -inf;
//   2. each warp sorts its lanes' maxima (bitonic, in registers) and keeps its P largest; after a cluster barrier
//      every CTA reads the row's C * 8 * P >= M keys (at most 256, one per thread) and finds the same bound, the
//      M-th largest of those keys to 16 key bits (bisection, one block-wide count per bit). M
//      distinct logits lie at or above it, so it is at most the row's M-th largest; and unless one warp holds more
//      than P of the row's largest lane maxima it is the M-th largest lane maximum itself, which few other logits
//      reach;
//   3. each CTA keeps its logits at or above the bound (chunk_keep: its exact top M if it would keep too many) and
//      writes them, as row words, to its region of every CTA's candidate buffer;
//   4. each CTA ranks its own candidates among the row's by counting: the row's M largest are all candidates, so a
//      candidate's rank among them is its rank in the row when below M, and it is written straight to out[rank].
// No workspace and no global atomics; the row's CTAs compute the bound redundantly rather than wait for one another.
constexpr uint64_t kTopmCopyBudgetNs = 4000000000ull;  // the slice copy takes a microsecond: this stops a lost one
constexpr int kMaxClusterCtas = 8;

// Dynamic shared memory of the cluster kernel: the slice, then the row's candidates.
inline size_t cluster_smem_bytes(int C, int cap) { return kChunkSmem + sizeof(uint64_t) * static_cast<size_t>(C) * cap; }

// The M-th largest of the keys held one per thread (0: none), to the top 16 key bits, in every thread: the largest
// v with at least M keys whose top 16 bits are >= v, shifted back (exact for 16-bit keys, a lower bound otherwise).
// Bisection over v, one block-wide count per bit. Called by all threads, convergently.
template <int kKeyBits>
__device__ __forceinline__ uint32_t block_kth_bound16(uint32_t key, int M) {
  constexpr int kShift = kKeyBits - 16;
  const uint32_t k16 = key >> kShift;
  uint32_t v = 0;
#pragma unroll
  for (int bit = 15; bit >= 0; --bit) {
    const uint32_t cand = v | (1u << bit);
    if (__syncthreads_count(k16 >= cand) >= M) v = cand;
  }
  return v << kShift;
}

// Descending bitonic sort of one key per lane: lane i ends with the i-th largest of the warp's keys.
__device__ __forceinline__ uint32_t warp_sort_desc(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xFFFFFFFFu, v, j);
      const bool desc = (lane & k) == 0, lower = (lane & j) == 0;
      v = (desc == lower) ? max(v, o) : min(v, o);
    }
  }
  return v;
}

template <bool kBf16>
__global__ void __launch_bounds__(kFThreads, 2)
    topm_cluster_kernel(const void* __restrict__ logits, int V, int M, int slice, int cap,
                        int32_t* __restrict__ out_ids, float* __restrict__ out_vals, WsHeader* hdr) {
  using T = Topm<kBf16, kFThreads, kFGroups>;
  constexpr int kWarps = kFThreads / 32;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int C = static_cast<int>(gridDim.x);  // the cluster spans the grid's x dimension: one row
  const int c = static_cast<int>(cluster_rank());
  const int row = blockIdx.y;
  extern __shared__ uint4 chunk_s[];                                            // the slice
  uint64_t* rw = reinterpret_cast<uint64_t*>(chunk_s + kFThreads * kFGroups);  // [C][cap] the row's candidates
  __shared__ FilterShared<kBf16, kFThreads> F;
  __shared__ uint32_t s_keys[kFThreads];  // [warps][P] this CTA's warps' largest lane maxima
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ int s_cnt[kMaxClusterCtas];  // candidates of each CTA of the row
  const int c0 = c * slice;
  const int len = min(slice, V - c0);  // > 0 and whole 16-byte groups (host-checked)
  const int ngroups = len / T::kPer16;
  if (t == 0) {  // the copies go out first; the barrier below orders the barrier's initialisation before any wait
    mbar_init(&s_bar, 1);
    mbar_fence_init();
    F.s_n = 0;
    const char* src =
        static_cast<const char*>(logits) + (static_cast<long long>(row) * V + c0) * static_cast<long long>(kBf16 ? 2 : 4);
    const unsigned bytes = static_cast<unsigned>(ngroups) * 16u;
    mbar_expect_tx(&s_bar, bytes);
    constexpr unsigned kPiece = 8192;
    for (unsigned o = 0; o < bytes; o += kPiece)
      bulk_g2s(reinterpret_cast<char*>(chunk_s) + o, src + o, min(kPiece, bytes - o), &s_bar);
  }
  constexpr uint32_t kPad = kBf16 ? 0xFF80FF80u : 0xFF800000u;  // -inf: raises no maximum, dropped by index
  for (int g = ngroups + t; g < kFThreads * kFGroups; g += kFThreads) chunk_s[g] = make_uint4(kPad, kPad, kPad, kPad);
  __syncthreads();  // the barrier is initialised; the padding is in place
  const bool ok = __syncthreads_and(mbar_wait(&s_bar, 0, kTopmCopyBudgetNs));
  if (!ok && t == 0) record_error(hdr, DT_ERR_TIMEOUT);
  T x{chunk_s};
  bool nan = false;
  if (!kBf16) nan = x.any_nan_f32();
  const uint32_t mk = x.max_key(nan);
  // keys per warp: at least 4, and enough that the row's warps send M or more (C * kWarps * P <= kFThreads)
  const int P = min(32, max(4, (M + C * kWarps - 1) / (C * kWarps)));
  const uint32_t sk = warp_sort_desc(mk);
  if (lane < P) s_keys[warp * P + lane] = sk;
  cluster_sync();  // 1: every CTA of the row runs and its keys are in place
  uint32_t key = 0;  // thread t reads key t of the row's C * kWarps * P
  if (t < C * kWarps * P)
    key = ld_dsmem_u32(dsmem_addr(&s_keys[t % (kWarps * P)], static_cast<unsigned>(t / (kWarps * P))));
  const uint32_t theta = block_kth_bound16<T::kKeyBits>(key, M);
  if (t == 0) F.s_theta = theta;
  __syncthreads();
  const int n = chunk_keep(x, M, len, cap, false, 0u, nan, hdr, F);
  for (int i = t; i < n; i += kFThreads) {
    const uint64_t w = T::global_word(F.cand[i], c0);
    for (int q = 0; q < C; ++q) st_dsmem_u64(dsmem_addr(&rw[static_cast<size_t>(c) * cap + i], static_cast<unsigned>(q)), w);
  }
  if (t < C) st_dsmem_u32(dsmem_addr(&s_cnt[c], static_cast<unsigned>(t)), static_cast<uint32_t>(n));
  cluster_sync();  // 2: the row's candidates are in every CTA; no CTA touches another's memory after this
  int total = 0;
  for (int q = 0; q < C; ++q) total += s_cnt[q];
  // Ranks: a warp takes four of this CTA's candidates at a time, its lanes splitting the row's words.
  const long long row_out = static_cast<long long>(row) * M;
  const uint64_t* mine = rw + static_cast<size_t>(c) * cap;
  for (int i0 = 4 * warp; i0 < n; i0 += 4 * kWarps) {
    uint64_t w[4];
    int r[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      w[k] = i0 + k < n ? mine[i0 + k] : ~0ull;
      r[k] = 0;
    }
    for (int q = 0; q < C; ++q) {
      const uint64_t* src = rw + static_cast<size_t>(q) * cap;
      const int nq = s_cnt[q];
      for (int j = lane; j < nq; j += 32) {
        const uint64_t v = src[j];
#pragma unroll
        for (int k = 0; k < 4; ++k) r[k] += v > w[k];
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) r[k] = __reduce_add_sync(0xFFFFFFFFu, r[k]);
    if (lane < 4 && i0 + lane < n) {
      const int rank = lane == 0 ? r[0] : lane == 1 ? r[1] : lane == 2 ? r[2] : r[3];
      const uint64_t wd = lane == 0 ? w[0] : lane == 1 ? w[1] : lane == 2 ? w[2] : w[3];
      if (rank < M) {
        out_ids[row_out + rank] = static_cast<int32_t>(candidate_id(wd));
        out_vals[row_out + rank] = kBf16 ? value_of_key_bf16(candidate_key(wd)) : value_of_key_f32(candidate_key(wd));
      }
    }
  }
  if (c == 0)  // fewer candidates than M only for rows of NaNs: the missing slots as the chunk-list path fills them
    for (int m = total + t; m < M; m += kFThreads) {
      out_ids[row_out + m] = 0;
      out_vals[row_out + m] = -INFINITY;
    }
  if (!ok) mbar_wait(&s_bar, 0, kTopmCopyBudgetNs);  // a late copy must not land after the CTA has left
}

dt_status launch_topm(const void* logits, dt_dtype dtype, int B, int K, int V, int M, int32_t* out_ids,
                      float* out_vals, char* ws, const TopmLayout& L, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * K;
  auto* hdr = reinterpret_cast<WsHeader*>(ws);
  auto* bounds = reinterpret_cast<uint32_t*>(ws + L.bounds);
  auto* tickets = reinterpret_cast<unsigned*>(ws + L.tickets);
  auto* counts = reinterpret_cast<int*>(ws + L.counts);
  void* words = ws + L.words;
  const size_t esize = dtype == DT_BF16 ? 2 : 4;
  const bool vec_ok = (static_cast<size_t>(V) * esize) % 16 == 0;
  // the staged chunk (and the selection's buffers) exceed the default 48 KB of dynamic shared memory
  DeviceInfo di{};
  if (current_device_info(&di) != cudaSuccess) return DT_ERR_CUDA;
  const int sms = di.sms;
  auto run = [&](auto bf16_tag) {
    constexpr bool kB = decltype(bf16_tag)::value;
    constexpr int kChunk = Topm<kB, kFThreads, kFGroups>::kChunk;
    const int chunks = (V + kChunk - 1) / kChunk;  // <= L.chunks: the layout is sized for the smaller fp32 chunk
    const dim3 grid(static_cast<unsigned>(rows), static_cast<unsigned>(chunks));
    // one cluster per row: whole 16-byte groups in every row, M <= 256 (the candidate buffers stay small), a slice
    // of at least 8192 bf16 / 4096 fp32 logits per CTA, the row in at most 8 slices, all in one wave
    if (topm_cluster_setting() && vec_ok && M <= kFThreads && di.cluster) {
      constexpr int kPer16 = kB ? 8 : 4;
      constexpr int kMinSlice = kFThreads * kPer16 * 4;
      int C = 1;
      while (C < kMaxClusterCtas && static_cast<long long>(C) * kMinSlice < V) C *= 2;
      const int slice = ((V + C - 1) / C + kPer16 - 1) / kPer16 * kPer16;
      if (slice <= kChunk && static_cast<long long>(C - 1) * slice < V && rows * C <= 2LL * sms && rows <= 65535) {
        const size_t smem = cluster_smem_bytes(C, L.cap);
        if (ensure_dynamic_smem(reinterpret_cast<const void*>(topm_cluster_kernel<kB>), smem) != cudaSuccess)
          return false;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(C), static_cast<unsigned>(rows));
        cfg.blockDim = dim3(kFThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(C);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, topm_cluster_kernel<kB>, logits, V, M, slice, L.cap, out_ids, out_vals, hdr) ==
               cudaSuccess;
      }
    }
    // about two waves of three CTAs per SM or fewer: fuse the selection into the launch
    const bool fuse = rows * chunks <= 6LL * sms;
    if (ensure_dynamic_smem(reinterpret_cast<const void*>(topm_filter_kernel<kB, true>), kChunkSmem) != cudaSuccess ||
        ensure_dynamic_smem(reinterpret_cast<const void*>(topm_filter_kernel<kB, false>), kChunkSmem) != cudaSuccess ||
        ensure_dynamic_smem(reinterpret_cast<const void*>(topm_select_kernel<kB>), sizeof(SelectSmem)) != cudaSuccess)
      return false;
    if (fuse) {
      topm_filter_kernel<kB, true><<<grid, kFThreads, kChunkSmem, stream>>>(
          logits, V, M, chunks, L.cap, vec_ok, bounds, tickets, words, counts, out_ids, out_vals, hdr);
    } else {
      topm_filter_kernel<kB, false><<<grid, kFThreads, kChunkSmem, stream>>>(
          logits, V, M, chunks, L.cap, vec_ok, bounds, tickets, words, counts, out_ids, out_vals, hdr);
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(static_cast<unsigned>(rows));
      cfg.blockDim = dim3(kSelThreads);
      cfg.dynamicSmemBytes = sizeof(SelectSmem);
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, topm_select_kernel<kB>, static_cast<const void*>(words),
                             static_cast<const int*>(counts), chunks, L.cap, M, bounds, out_ids, out_vals) !=
          cudaSuccess)
        return false;
    }
    return true;
  };
  const bool ok = dtype == DT_BF16 ? run(std::true_type{}) : run(std::false_type{});
  if (!ok) return DT_ERR_CUDA;
  return cuda_status(cudaGetLastError());
}

// Bytes of a topm_layout workspace that one launch touches: the layout's offsets are those of the fp32 chunk (the
// most chunks); a bf16 launch has fewer, larger chunks whose candidate words are 4 bytes instead of 8.
size_t topm_launch_bytes(const TopmLayout& L, dt_dtype dtype, int B, int K, int V) {
  const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(K);
  if (dtype != DT_BF16) return L.bytes;
  constexpr int kChunk = Topm<true, kFThreads, kFGroups>::kChunk;
  const size_t chunks = (static_cast<size_t>(V) + kChunk - 1) / kChunk;
  return align_up(L.words + sizeof(uint32_t) * rows * chunks * static_cast<size_t>(L.cap));
}

}  // namespace
}  // namespace dt

extern "C" size_t dt_topm_workspace_bytes(int B, int K, int V, int M) {
  if (B < 0 || K < 1 || V < 1 || M < 1) return 0;
  return dt::topm_layout(B, K, V, M).bytes;
}

namespace dt {
// Every check of dt_topm's arguments, host-side only: nothing is launched.
dt_status topm_check(const void* logits, dt_dtype dtype, int B, int K, int V, int M, const int32_t* out_ids,
                     const float* out_vals, const void* workspace, size_t workspace_bytes) {
  if (B < 0 || K < 1 || V < 1 || M < 1 || M > V) return DT_ERR_INVALID_ARG;
  if (dtype != DT_F32 && dtype != DT_BF16) return DT_ERR_INVALID_ARG;
  if (M > DT_MAX_M) return DT_ERR_UNSUPPORTED;
  if (B == 0) return DT_OK;  // nothing to read or write
  if (!logits || !out_ids || !out_vals || !workspace) return DT_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(out_ids) || !aligned16(out_vals) || !aligned16(workspace))
    return DT_ERR_INVALID_ARG;
  const TopmLayout L = topm_layout(B, K, V, M);
  if (workspace_bytes < L.bytes) return DT_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * K > INT_MAX || L.chunks > 65535) return DT_ERR_UNSUPPORTED;  // grid limits
  return DT_OK;
}
}  // namespace dt

extern "C" dt_status dt_topm(const void* logits, dt_dtype dtype, int B, int K, int V, int M, int32_t* out_ids,
                             float* out_vals, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  using namespace dt;
  const dt_status st = topm_check(logits, dtype, B, K, V, M, out_ids, out_vals, workspace, workspace_bytes);
  if (st != DT_OK || B == 0) return st;
  return launch_topm(logits, dtype, B, K, V, M, out_ids, out_vals, static_cast<char*>(workspace),
                     topm_layout(B, K, V, M), stream);
}

// ---- dt_topm_static: the same top-M with no caller workspace ----------------------------------------------------
// For callers that cannot call cudaMalloc (see dominotree.h). Its scratch is this file-scope device array: every GPU
// that loads the library holds it until the process exits. Host code must not pass `g_topm_scratch` itself to a
// kernel (on the host that name is only a stand-in); the device address comes from cudaGetSymbolAddress, taken with
// the device current, on the first call made in that device's current context. The address is cached per device
// together with the context's unique id: a context created anew (after cudaDeviceReset, say) reloads the module,
// whose array may then sit elsewhere, so a new id takes the address again.
namespace dt {
namespace {
__device__ __align__(256) unsigned char g_topm_scratch[DT_TOPM_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
struct ScratchAddr {
  unsigned long long ctx_id;
  void* ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

// The unique id of the calling thread's current context (the driver's cuCtxGetCurrent / cuCtxGetId, reached through
// the runtime's entry-point query, so the library does not link the driver library). False if either is missing.
bool current_context_id(unsigned long long* id) {
  using GetCurrent = int (*)(void**);
  using GetId = int (*)(void*, unsigned long long*);
  static std::mutex mu;
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static bool looked = false;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!looked) {
      looked = true;
      void* f = nullptr;
      cudaDriverEntryPointQueryResult q{};
      if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
          q == cudaDriverEntryPointSuccess)
        get_current = reinterpret_cast<GetCurrent>(f);
      f = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
          q == cudaDriverEntryPointSuccess)
        get_id = reinterpret_cast<GetId>(f);
    }
  }
  void* ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != 0 || !ctx) return false;
  return get_id(ctx, id) == 0;
}

dt_status static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DT_ERR_UNSUPPORTED;
  unsigned long long ctx_id = 0;
  const bool have_id = current_context_id(&ctx_id);  // false before the runtime made any context current
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  ScratchAddr& a = g_scratch[dev];
  if (have_id && a.ptr && a.ctx_id == ctx_id) {
    *out = a.ptr;
    return DT_OK;
  }
  // the lookup makes the device's primary context current if none was, and loads the module if it was not loaded yet
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_topm_scratch) != cudaSuccess || !p) return DT_ERR_CUDA;
  if (!have_id && !current_context_id(&ctx_id)) return DT_ERR_CUDA;
  a = ScratchAddr{ctx_id, p};
  *out = p;
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
  if (static_cast<long long>(B) * K > INT_MAX || L.chunks > 65535) return DT_ERR_UNSUPPORTED;
  if (topm_launch_bytes(L, dtype, B, K, V) > DT_TOPM_STATIC_SCRATCH_BYTES) return DT_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const dt_status st = static_scratch(&scratch);
  if (st != DT_OK) return st;
  char* ws = static_cast<char*>(scratch);
  // The array keeps the previous call's contents: the header, the per-row bounds and the per-row tickets must start
  // at zero (everything before the per-chunk counts, which each call writes before reading).
  if (cudaMemsetAsync(ws, 0, L.counts, stream) != cudaSuccess) return DT_ERR_CUDA;
  return launch_topm(logits, dtype, B, K, V, M, out_ids, out_vals, ws, L, stream);
}
