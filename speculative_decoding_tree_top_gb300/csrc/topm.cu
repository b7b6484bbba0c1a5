// dt_topm — top-M candidate restriction over the drafter's marginal logits.
//
// Method: blog.captcha.la, "Methodology — deep read" / "Technical innovations" (the per-node correction only sees
// the M highest-marginal tokens of each depth); gist.science, "Composants Clés — Restriction de Candidats".
//
// GB300 design. The op is a pure HBM stream (every logit is read once, nothing is reused), so it is laid out for
// bandwidth and for few instructions per logit, not for tensor cores. Two launches:
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
