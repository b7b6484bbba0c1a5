// Internal helpers shared by the CUDA translation units of libdominotree (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dominotree.h"

namespace dt {

// Every workspace starts with this 256-byte header. It is zeroed once (dt_workspace_init); kernels leave it zeroed
// again except for `status`, which holds the first device-side problem until dt_get_error clears it.
struct WsHeader {
  unsigned status;     // dt_status of the first device-side problem, 0 if none
  unsigned abort;      // set when a barrier wait ran out: every CTA leaves at its next barrier
  unsigned bar_count;  // grid barrier: CTAs arrived at the current barrier
  unsigned bar_gen;    // grid barrier: generation, bumped by the last CTA to arrive
  unsigned long long sync_count;  // step barrier: arrivals ever made (monotonic, never reset)
  // statistics of the last dt_build_trees launch (dt_build_stats): cleared by CTA 0 before the launch's first grid
  // barrier, raised after it
  unsigned long long stat_launch_ns;    // CTA 0: its start to its end
  unsigned long long stat_gather_ns;    // the longest time one CTA spent gathering correction rows
  unsigned long long stat_gather_bytes; // correction-row bytes the launch gathered (rows x H x element size)
  unsigned stat_waves;                  // waves run
  unsigned stat_expansions;             // expansions computed (the roots included)
  unsigned reserved[50];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr size_t kAlign = 256;
__host__ __device__ inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

__device__ __forceinline__ void record_error(WsHeader* hdr, unsigned code) { atomicCAS(&hdr->status, 0u, code); }

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Grid-wide barrier of a cooperative launch. Every wait is bounded: when the budget runs out, or when another CTA's
// wait already ran out (the header's abort word), the CTA records DT_ERR_TIMEOUT (first problem wins), raises the
// abort word, and the barrier returns false in every thread of the CTA, which must then leave the kernel. Other
// recorded problems do not stop the kernel. Memory written before the barrier by any CTA is visible after it
// (release by the arrivals and the last arrival, acquire by the waiters).
__device__ __forceinline__ bool grid_barrier(WsHeader* hdr, unsigned nblocks, uint64_t timeout_ns, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned gen = ld_acquire_gpu(&hdr->bar_gen);
    const unsigned arrived = atom_add_acq_rel_gpu(&hdr->bar_count, 1u) + 1u;
    if (arrived == nblocks) {
      atomicExch(&hdr->bar_count, 0u);
      st_release_gpu(&hdr->bar_gen, gen + 1u);
    } else if (timeout_ns == 0) {  // test hook: a zero budget gives up at the first wait
      ok = 0;
    } else {
      const uint64_t t0 = global_timer_ns();
      unsigned polls = 0;
      while (ld_acquire_gpu(&hdr->bar_gen) == gen) {
        if ((++polls & 15u) == 0u &&
            (ld_acquire_gpu(&hdr->abort) != 0u || global_timer_ns() - t0 > timeout_ns)) {
          ok = 0;
          break;
        }
      }
    }
    if (!ok) {
      record_error(hdr, DT_ERR_TIMEOUT);
      atomicExch(&hdr->abort, 1u);
    }
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// One-hop grid barrier for a launch that crosses many barriers: every CTA adds 1 to a monotonic 64-bit counter
// with a release reduction (no round trip) and waits until the counter reaches `target` = base + G * k for its k-th
// crossing, base being the counter's value read by every CTA before the launch's first grid_barrier (no CTA can
// arrive here before all have read it). Bounded like grid_barrier: a run-out budget or the abort word stops it.
__device__ __forceinline__ void counter_arrive(WsHeader* hdr) {
  __syncthreads();  // every thread of the CTA is done with the phase; thread 0 releases their writes
  if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(&hdr->sync_count) : "memory");
}

// Waiting half: thread 0 polls (acquire) until `target` arrivals, then the whole CTA proceeds. Between the two halves
// a CTA may do work that reads nothing the other CTAs write in the phase (prefetches).
__device__ __forceinline__ bool counter_wait(WsHeader* hdr, unsigned long long target, uint64_t timeout_ns,
                                             int* s_flag) {
  if (threadIdx.x == 0) {
    int ok = 1;
    if (timeout_ns == 0) {
      ok = 0;
    } else {
      const uint64_t t0 = global_timer_ns();
      unsigned polls = 0;
      while (ld_acquire_gpu_u64(&hdr->sync_count) < target) {
        if ((++polls & 15u) == 0u &&
            (ld_acquire_gpu(&hdr->abort) != 0u || global_timer_ns() - t0 > timeout_ns)) {
          ok = 0;
          break;
        }
      }
    }
    if (!ok) {
      record_error(hdr, DT_ERR_TIMEOUT);
      atomicExch(&hdr->abort, 1u);
    }
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

__device__ __forceinline__ bool counter_barrier(WsHeader* hdr, unsigned long long target, uint64_t timeout_ns,
                                                int* s_flag) {
  counter_arrive(hdr);
  return counter_wait(hdr, target, timeout_ns, s_flag);
}

// ---- shared-memory barriers and bulk copies (TMA, 1-D) -------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
// Arrives once on `bar` and expects `bytes` more of asynchronous copies in the current phase.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// Adds `bytes` to the asynchronous copies the current phase of `bar` expects, without arriving (several threads may
// each announce their own copies; one arrival then closes the phase's count).
__device__ __forceinline__ void mbar_expect_tx_only(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// Arrives once on `bar`, with no transaction bytes.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
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
// Global -> shared bulk copy completing on `bar` (both addresses 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// ---- thread-block clusters: distributed shared memory and the cluster barrier ------------------------------------
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address, in the cluster's shared window, of the variable at `p` (this CTA's shared memory) in CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, unsigned rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t ld_dsmem_u64(uint32_t a) {
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void st_dsmem_u32(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_u64(uint32_t a, uint64_t v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
// Every thread of every CTA of the cluster arrives (release), then waits for all (acquire): shared-memory writes
// made before it, in any CTA of the cluster, are visible after it. Called by all threads, convergently.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- order-preserving unsigned keys of logits -------------------------------------------------------------------
// Larger key <=> larger value. -0.0 is folded onto +0.0 so that both compare equal (the id then decides). Every
// non-padding element gets a key >= 1, so key 0 marks "no element".
__device__ __forceinline__ uint32_t key_of_bf16(uint32_t bits) {
  bits &= 0xFFFFu;
  if (bits == 0x8000u) bits = 0u;
  const uint32_t k = (bits & 0x8000u) ? (~bits & 0xFFFFu) : (bits | 0x8000u);
  return k > 1u ? k : 1u;
}
__device__ __forceinline__ uint32_t key_of_f32(uint32_t bits) {
  if (bits == 0x80000000u) bits = 0u;
  const uint32_t k = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
  return k > 1u ? k : 1u;
}
__device__ __forceinline__ bool is_nan_bf16(uint32_t bits) { return (bits & 0x7FFFu) > 0x7F80u; }
__device__ __forceinline__ bool is_nan_f32(uint32_t bits) { return (bits & 0x7FFFFFFFu) > 0x7F800000u; }

__device__ __forceinline__ float value_of_key_bf16(uint32_t k) {
  const uint32_t bits = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
  return __uint_as_float(bits << 16);
}
__device__ __forceinline__ float value_of_key_f32(uint32_t k) {
  const uint32_t bits = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(bits);
}

// A candidate as one 64-bit word: key in the high half, bit-inverted id in the low half, so that the larger word is
// the larger value and, among equal values, the smaller id. Distinct ids make every word distinct; 0 = empty.
__device__ __forceinline__ uint64_t pack_candidate(uint32_t key, uint32_t id) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint64_t>(~id);
}
__device__ __forceinline__ uint32_t candidate_id(uint64_t c) { return ~static_cast<uint32_t>(c); }
__device__ __forceinline__ uint32_t candidate_key(uint64_t c) { return static_cast<uint32_t>(c >> 32); }

// ---- block-wide helpers (blockDim.x == 32 * kWarps) -------------------------------------------------------------
template <int kWarps>
__device__ __forceinline__ int block_sum(int v, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_add_sync(0xFFFFFFFFu, v);
  if (lane == 0) s_warp[warp] = v;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += s_warp[w];
  __syncthreads();
  return t;
}

template <int kWarps>
__device__ __forceinline__ int block_exclusive_scan(int v, int* total, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int s = s_warp[w];
    base += (w < warp) ? s : 0;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return base + incl - v;
}

template <int kWarps>
__device__ __forceinline__ uint64_t block_max_u64(uint64_t v, uint64_t* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t y = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = y > v ? y : v;
  }
  if (lane == 0) s_warp[warp] = v;
  __syncthreads();
  uint64_t m = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) m = s_warp[w] > m ? s_warp[w] : m;
  __syncthreads();
  return m;
}

// Streaming 16-byte load that does not allocate in L1 (the logits are read exactly once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

inline dt_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DT_OK : DT_ERR_CUDA; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Workspace layout of dt_topm: header | per-row bound of the row's M-th largest key | per-row ticket (both zero
// between calls) | per-(row, chunk) candidate counts | per-(row, chunk) candidate words, room for `cap` 8-byte words each. dt_build_trees puts its own region after this one, so that one workspace can serve
// both calls of a round. A filter CTA reads one chunk of 16384 logits of a row (256 threads x 64).
inline int topm_chunk(int B, int K) {
  (void)B;
  (void)K;
  return 16384;
}
// Candidate words a chunk may keep: all of its logits at or above the chunk's bound when there are at most 4M of
// them (M <= 256; at least 64), else exactly its top M.
__host__ __device__ inline int topm_cap(int M) { return M <= 256 ? (4 * M < 64 ? 64 : 4 * M) : M; }
struct TopmLayout {
  size_t bounds, tickets, counts, words, bytes;
  int chunks, chunk, cap;
};
inline TopmLayout topm_layout(int B, int K, int V, int M) {
  TopmLayout L{};
  const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(K);
  L.chunk = topm_chunk(B, K);
  L.chunks = (V + L.chunk - 1) / L.chunk;
  L.cap = topm_cap(M);
  L.bounds = sizeof(WsHeader);
  L.tickets = align_up(L.bounds + sizeof(uint32_t) * rows);
  L.counts = align_up(L.tickets + sizeof(uint32_t) * rows);
  L.words = align_up(L.counts + sizeof(int) * rows * static_cast<size_t>(L.chunks));
  L.bytes = align_up(L.words + sizeof(uint64_t) * rows * static_cast<size_t>(L.chunks) * L.cap);
  return L;
}

// Host-side process-wide settings (dt_set_barrier_timeout_ns, dt_set_lookahead).
uint64_t barrier_timeout_ns();
int lookahead_setting();  // 0 = automatic
bool topm_cluster_setting();  // dt_set_topm_cluster

// Attributes of the current device, queried once per device and cached (a launch then costs one runtime call).
struct DeviceInfo {
  int dev, sms, coop, optin, cluster;
};
cudaError_t current_device_info(DeviceInfo* out);
// Raises the dynamic shared-memory limit of kernel `fn` on the current device to at least `bytes`; the runtime is
// called only when a larger size than any set before for this (device, kernel) is asked for.
cudaError_t ensure_dynamic_smem(const void* fn, size_t bytes);
// dt_topm's argument checks without the launch (dt_round checks a whole round before its first launch)
dt_status topm_check(const void* logits, dt_dtype dtype, int B, int K, int V, int M, const int32_t* out_ids,
                     const float* out_vals, const void* workspace, size_t workspace_bytes);

}  // namespace dt
