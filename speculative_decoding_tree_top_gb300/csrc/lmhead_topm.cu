// dt_lmhead_topm — the drafter's full-vocabulary projection and its top-M in one launch, the logits never written.
//
// Method: blog.captcha.la, "Methodology — deep read" (the costly full-vocabulary projection; the per-node work only
// sees the M highest-marginal tokens of each depth); gist.science, "Composants Clés — Restriction de Candidats"
// (re-running the projection W2 over the whole vocabulary is what the top-M restriction avoids). The marginal
// logits of a row are hidden_r . W2^T (no bias), of which the M largest are kept, ties to the lower id.
//
// GB300 design: one persistent cooperative launch, one CTA per SM, logits kept in tensor memory.
//   * GEMM on tcgen05: CTA c owns vocabulary tiles c, c + G, ... (128 head rows each, at most 512 / Rp of them);
//     the head rows are the MMA's M side, the R hidden rows (padded to Rp, a multiple of 16) its N side. Both
//     operands arrive by 2-D TMA (128-byte swizzle, 64-column K blocks) through an 8-stage mbarrier ring; one lane
//     issues TMA, one lane the MMAs; tile i accumulates in TMEM columns [i Rp, (i + 1) Rp), so the CTA's whole slice
//     of logits stays on chip. The head is read once from HBM: at small R the launch is an HBM stream of V x D bf16.
//   * Bound: per row, every warp quarter (32 TMEM lanes: 32 head rows of every tile) offers its two largest logits
//     to a pool in the workspace; after a grid barrier every CTA takes the M-th largest of the row's pool (G x 8
//     values, a subset of the row's logits, so a lower bound of its M-th largest logit, and tight because the row's
//     top M are spread over many quarters).
//   * Filter: every logit at or above its row's bound is appended, as a 64-bit row word (value key, inverted id),
//     to the CTA's list for the row (room for all of the CTA's values: exact whatever the data).
//   * Grid barrier; then CTA r selects row r from the G lists (the selection shared with dt_topm).
// Every comparison is on integer words, so the result is deterministic and exact for the logits as computed (fp32
// accumulation of bf16 products in the tensor cores).
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>

#include "dt_internal.cuh"
#include "topm_select.cuh"
#include "umma.cuh"

namespace dt {
namespace {

constexpr int kThreads = 256;
constexpr int kTileV = 128;           // head rows per tile (the MMA's M)
constexpr int kBK = 64;               // K block: 64 bf16 = one 128-byte swizzle row
constexpr int kMaxStages = 12;
constexpr int kMaxRp = 64;            // padded hidden rows (the MMA's N): a multiple of 16
constexpr int kTmemMax = 512;
constexpr int kMaxTiles = kTmemMax / 16;  // tiles per CTA at most (each takes Rp >= 16 TMEM columns)
constexpr int kPoolPerQuarter = 2;    // logits a warp quarter offers per row
constexpr int kPoolPerCta = 4 * kPoolPerQuarter;
constexpr int kPoolPerThread = 8;     // pool values per thread in the bound's selection: G x kPoolPerCta <= 2048
constexpr uint64_t kBudgetNs = 4000000000ull;  // copies and MMAs take microseconds: this stops a lost one
constexpr size_t kStaticReserve = 3072;        // shared memory kept for the kernel's static variables

struct LhParams {
  int R, Rp, D, V, M, rpc, tpc, last, G;  // head rows per CTA, tiles per CTA, rows of a CTA's last tile
  int stages, kbps;  // ring stages, and K blocks per stage (a divisor of D / 64)
  uint32_t* pool;   // [Rp][G * kPoolPerCta] value keys (0: none)
  uint32_t* bounds; // [R] each row's bound (a key)
  uint64_t* cand;   // [R][G][rpc] each CTA's candidates of each row as row words
  int* counts;      // [R][G]
  int32_t* ids;     // [R][M]
  float* vals;      // [R][M]
  WsHeader* hdr;
  uint64_t timeout_ns;
};
struct LhMaps {
  CUtensorMap w;    // head [V][D] bf16, box 64 x 128
  CUtensorMap wl;   // the same, box 64 x last (a CTA's last tile)
  CUtensorMap h;    // hidden [R][D] bf16, box 64 x Rp
};

// One K block of a stage: the head tile's 128 rows x 64 columns, then the hidden rows' Rp x 64 (both 1 KB-aligned).
__host__ __device__ inline size_t lh_block_bytes(int Rp) {
  return static_cast<size_t>(kTileV) * kBK * 2 + static_cast<size_t>(Rp) * kBK * 2;
}
__host__ __device__ inline size_t lh_smem_bytes(int Rp, int stages, int kbps) {
  const size_t ring = static_cast<size_t>(stages) * kbps * lh_block_bytes(Rp);
  return 1024 + (ring > sizeof(SelectSmem) ? ring : sizeof(SelectSmem));
}

// Sixteen consecutive TMEM columns of this warp's 32 lanes, and the wait for them, in one statement.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Two groups of sixteen TMEM columns of this warp's 32 lanes, and one wait for both.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
        "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),
        "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]),
        "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
      : "r"(ta), "r"(tb)
      : "memory");
}

// The M-th largest of n keys (np values of a row's pool, kPer per thread at most, read from global memory) in
// every thread of the block, 0 when n < M: radix select with 8-bit digits from the top, one 256-bin shared
// histogram per digit over the keys that share the digits found so far.
template <int kPer>
__device__ uint32_t block_kth_of(const uint32_t* __restrict__ keys, int n, int M, unsigned* hist, unsigned* s_sel) {
  const int t = threadIdx.x, lane = t & 31;
  if (n < M) return 0u;
  uint32_t v[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) v[k] = t + kThreads * k < n ? __ldcg(keys + t + kThreads * k) : 0u;
  uint32_t prefix = 0;
  int need = M;
#pragma unroll 1
  for (int d = 3; d >= 0; --d) {
    hist[t] = 0u;  // kThreads == 256 bins
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const bool in = t + kThreads * k < n && (d == 3 || (v[k] >> (8 * (d + 1))) == prefix);
      if (in) atomicAdd(&hist[(v[k] >> (8 * d)) & 255u], 1u);
    }
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
        s_sel[0] = static_cast<unsigned>(255 - 8 * lane - j);
        s_sel[1] = acc;
      }
    }
    __syncthreads();
    prefix = (prefix << 8) | s_sel[0];
    need -= static_cast<int>(s_sel[1]);
    __syncthreads();  // s_sel and hist are rewritten by the next digit
  }
  return prefix;
}

__global__ void __launch_bounds__(kThreads, 1) lmhead_topm_kernel(LhParams p, const __grid_constant__ LhMaps maps) {
  extern __shared__ float4 smem_f4[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_f4) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kMaxStages], empty[kMaxStages], done, tdone[kMaxTiles];
  __shared__ uint32_t s_tmem;
  __shared__ uint32_t s_bound[kMaxRp];
  __shared__ int s_cnt[kMaxRp];
  __shared__ int s_flag, s_warp[kThreads / 32], s_n;
  __shared__ unsigned s_hist[256], s_sel[2];
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int G = static_cast<int>(gridDim.x), bid = static_cast<int>(blockIdx.x);
  const int R = p.R, Rp = p.Rp, nst = p.D / kBK / p.kbps, S = p.stages, kbps = p.kbps;
  // this CTA's head rows: [row0, row0 + nrows), in tiles of 128 (the last one of `last` rows)
  const int row0 = bid * p.rpc, nrows = min(p.rpc, p.V - row0);
  const int my_tiles = nrows > 0 ? (nrows + kTileV - 1) / kTileV : 0;
  const uint32_t cols = static_cast<uint32_t>(p.tpc * Rp) <= 32u ? 32u
                        : static_cast<uint32_t>(p.tpc * Rp) <= 64u ? 64u
                        : static_cast<uint32_t>(p.tpc * Rp) <= 128u ? 128u
                        : static_cast<uint32_t>(p.tpc * Rp) <= 256u ? 256u : 512u;
  if (t == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&done, 1);
    for (int i = 0; i < kMaxTiles; ++i) mbar_init(&tdone[i], 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(cols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;
  const size_t blk = lh_block_bytes(Rp), stage = blk * kbps;
  bool ok = true;

  // ---- GEMM: tile i of this CTA (vocabulary rows (bid + i G) * 128 ...) into TMEM columns [i Rp, (i + 1) Rp) ----
  if (warp == 0 && lane == 0) {  // TMA producer: stage s of tile i holds K blocks [s kbps, (s + 1) kbps)
    for (int i = 0; i < my_tiles && ok; ++i) {
      const bool lastt = i == p.tpc - 1;  // the CTA's last tile reads `last` head rows
      const CUtensorMap* wm = lastt ? &maps.wl : &maps.w;
      const uint32_t tx = static_cast<uint32_t>(kbps * ((lastt ? p.last : kTileV) + Rp) * kBK * 2);
      for (int sk = 0; sk < nst; ++sk) {
        const unsigned n = static_cast<unsigned>(i * nst + sk), st = n % S, use = n / S;
        if (use > 0) ok = mbar_wait(&empty[st], (use - 1) & 1u, kBudgetNs);
        if (!ok) break;
        unsigned char* a = base + st * stage;
        mbar_expect_tx(&full[st], tx);
        for (int j = 0; j < kbps; ++j) {
          const int kb = sk * kbps + j;
          tma_load_2d(a + j * blk, wm, kb * kBK, row0 + i * kTileV, &full[st]);
          tma_load_2d(a + j * blk + kTileV * kBK * 2, &maps.h, kb * kBK, 0, &full[st]);
        }
      }
    }
  } else if (warp == 1 && lane == 0) {  // MMA issuer
    const uint32_t idesc = umma_idesc(Rp, kTileV);
    for (int i = 0; i < my_tiles && ok; ++i) {
      for (int sk = 0; sk < nst; ++sk) {
        const unsigned n = static_cast<unsigned>(i * nst + sk), st = n % S, use = n / S;
        ok = mbar_wait(&full[st], use & 1u, kBudgetNs);
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        for (int j = 0; j < kbps; ++j) {
          const uint32_t a = smem_u32(base + st * stage + j * blk), b = a + kTileV * kBK * 2;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            umma_f16(tmem + static_cast<uint32_t>(i * Rp), umma_desc_sw128(a + 32 * k), umma_desc_sw128(b + 32 * k),
                     idesc, (sk > 0 || j > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&empty[st]);  // the stage is free once these MMAs have read it
      }
      if (ok) umma_commit(&tdone[i]);  // tile i's accumulator is complete after these MMAs
    }
    if (ok && my_tiles > 0) umma_commit(&done);  // every accumulator is complete after the last MMAs
  }
  // Warps 4..7 (TMEM lanes 32 (w % 4) .. + 31: head row 32 (w % 4) + lane of every tile) fold each tile into the
  // running two largest logits of rows 0..15 as soon as its accumulator is complete, while the GEMM goes on.
  const int q = warp & 3, half = warp >> 2;
  const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16);
  const int np = G * kPoolPerCta;
  bool nan = false;
  uint32_t b1[16], b2[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) b1[j] = b2[j] = 0u;
  if (warp >= 4) {
    for (int i = 0; i < my_tiles && ok; ++i) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&tdone[i], 0u, kBudgetNs));  // the TMEM load below is warp-wide
      if (!ok) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      uint32_t v[16];
      tmem_ld16(tq + static_cast<uint32_t>(i * Rp), v);
      const bool valid = i * kTileV + 32 * q + lane < nrows;  // rows past the range hold stale shared memory
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const bool isnan = (v[j] & 0x7FFFFFFFu) > 0x7F800000u;
        nan |= valid && isnan && j < R;
        const uint32_t k = valid && !isnan ? key_of_f32(v[j]) : 0u;
        if (k > b1[j]) {
          b2[j] = b1[j];
          b1[j] = k;
        } else if (k > b2[j]) {
          b2[j] = k;
        }
      }
    }
  }
  ok = __syncthreads_and(ok);
  if (ok && my_tiles > 0) ok = mbar_wait(&done, 0u, kBudgetNs);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  ok = __syncthreads_and(ok);

  if (ok) {
    // ---- pool: every quarter's two largest logits of each row (rows 0..15 already folded by warps 4..7; the other
    // row groups now, warps w and w + 4 taking alternate groups) ----
    for (int g = half ? 0 : 1; g < Rp / 16; g += 2) {
      if (g > 0) {
#pragma unroll
        for (int j = 0; j < 16; ++j) b1[j] = b2[j] = 0u;
      }
      for (int i = 0; i < (g > 0 ? my_tiles : 0); ++i) {
        uint32_t v[16];
        tmem_ld16(tq + static_cast<uint32_t>(i * Rp + 16 * g), v);
        const bool valid = i * kTileV + 32 * q + lane < nrows;  // rows past the range hold stale shared memory
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const bool isnan = (v[j] & 0x7FFFFFFFu) > 0x7F800000u;
          nan |= valid && isnan && 16 * g + j < R;
          const uint32_t k = valid && !isnan ? key_of_f32(v[j]) : 0u;
          if (k > b1[j]) {
            b2[j] = b1[j];
            b1[j] = k;
          } else if (k > b2[j]) {
            b2[j] = k;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t m1 = __reduce_max_sync(0xFFFFFFFFu, b1[j]);
        const int win = __ffs(__ballot_sync(0xFFFFFFFFu, b1[j] == m1)) - 1;
        const uint32_t m2 = __reduce_max_sync(0xFFFFFFFFu, lane == win ? b2[j] : b1[j]);
        if (lane == 0) {
          uint32_t* pr = p.pool + static_cast<size_t>(16 * g + j) * np + bid * kPoolPerCta + q * kPoolPerQuarter;
          pr[0] = m1;
          pr[1] = m2;
        }
      }
    }
  }
  if (__syncthreads_or(nan) && t == 0) record_error(p.hdr, DT_ERR_NUMERIC);
  if (ok) ok = grid_barrier(p.hdr, static_cast<unsigned>(G), p.timeout_ns, &s_flag);

  if (ok) {
    // ---- bound: CTA r takes row r's pool and publishes its M-th largest key (0: fewer than M values in the pool,
    // take every logit); after a grid barrier every CTA reads all the rows' bounds ----
    for (int r = bid; r < R; r += G) {
      const uint32_t th = block_kth_of<kPoolPerThread>(p.pool + static_cast<size_t>(r) * np, np, p.M, s_hist, s_sel);
      if (t == 0) p.bounds[r] = th;
    }
    ok = grid_barrier(p.hdr, static_cast<unsigned>(G), p.timeout_ns, &s_flag);
  }
  if (ok) {
    for (int r = t; r < R; r += kThreads) s_bound[r] = __ldcg(p.bounds + r);
    for (int r = t; r < R; r += kThreads) s_cnt[r] = 0;
    __syncthreads();
    // ---- filter: the logits at or above their row's bound, as row words, into this CTA's list of the row; warps w
    // and w + 4 take alternate tiles, two tiles per TMEM wait ----
    auto keep = [&](const uint32_t (&v)[16], int i, int g) {
      const int loc = i * kTileV + 32 * q + lane;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int r = 16 * g + j;
        const bool isnan = (v[j] & 0x7FFFFFFFu) > 0x7F800000u;
        if (loc < nrows && r < R && !isnan) {
          const uint32_t k = key_of_f32(v[j]);
          if (k >= s_bound[r]) {
            const int pos = atomicAdd(&s_cnt[r], 1);  // < rpc: the CTA holds at most rpc logits of a row
            p.cand[(static_cast<size_t>(r) * G + bid) * p.rpc + pos] = pack_candidate(k, static_cast<uint32_t>(row0 + loc));
          }
        }
      }
    };
    for (int g = 0; g < Rp / 16; ++g) {
      for (int i = half; i < my_tiles; i += 4) {
        uint32_t v0[16], v1[16];
        const bool two = i + 2 < my_tiles;
        tmem_ld16x2(tq + static_cast<uint32_t>(i * Rp + 16 * g), tq + static_cast<uint32_t>((two ? i + 2 : i) * Rp + 16 * g),
                    v0, v1);
        keep(v0, i, g);
        if (two) keep(v1, i + 2, g);
      }
    }
    __syncthreads();
    for (int r = t; r < R; r += kThreads) p.counts[static_cast<size_t>(r) * G + bid] = s_cnt[r];
    ok = grid_barrier(p.hdr, static_cast<unsigned>(G), p.timeout_ns, &s_flag);
  }

  if (ok) {
    // ---- selection: CTA r takes row r from the G lists ----
    SelectSmem& S = *reinterpret_cast<SelectSmem*>(base);
    for (int r = bid; r < R; r += G) {
      const uint64_t* rc = p.cand + static_cast<size_t>(r) * G * p.rpc;
      const int cap = p.rpc;
      const int* rn = p.counts + static_cast<size_t>(r) * G;
      select_words<false, kSelThreads>(
          [&](int c) { return __ldcg(rn + c); }, G, p.M,
          [&](int c, int i) { return __ldcg(rc + static_cast<size_t>(c) * cap + i); },
          p.ids + static_cast<size_t>(r) * p.M, p.vals + static_cast<size_t>(r) * p.M, S, s_warp, &s_n);
      __syncthreads();
    }
  } else if (t == 0) {
    record_error(p.hdr, DT_ERR_TIMEOUT);
    atomicExch(&p.hdr->abort, 1u);
  }

  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(cols) : "memory");
}

// ---- more than 64 rows: blocked passes -------------------------------------------------------------------------
// Past 64 hidden rows a CTA's slice of the logits no longer fits its tensor memory, so the GEMM runs twice, over
// work items of (vocabulary tile of 128 head rows, up to W = 256 hidden rows), each accumulating in one of two TMEM
// buffers while the epilogue warps drain the other:
//   1. pool pass: every CTA's first tile only (128 x G head rows, a sample of the vocabulary): every warp quarter
//      offers each row's two largest logits to the row's pool, as above;
//   2. lh_bound_kernel: a warp per row takes the M-th largest of the row's pool, to the top 16 key bits (a lower
//      bound of the row's M-th largest logit: the pool is a subset of the row's logits);
//   3. filter pass: every tile; the epilogue keeps every logit at or above its row's bound (one float compare per
//      logit; NaNs take the rare path too) in the CTA's list of the row (room for all of the CTA's values: exact
//      whatever the data);
//   4. lh_select_kernel: a CTA per row selects the row's top M from the G lists (the selection shared with dt_topm).
// The CTAs form groups of gs (a divisor of the hidden blocks and of the grid, at most 4) that walk the same
// vocabulary tiles in step, CTA k of a group taking hidden blocks k, k + gs, ...: a head tile comes from HBM once
// and from L2 for the group's other CTAs, at about the same time, and no CTA reads a tile twice unless it has more
// than one hidden block. A row's candidates of a group are all found by one CTA: the lists are (row, group).
constexpr int kItemMax = 256;                                      // hidden rows per work item: the MMA's N
constexpr size_t kAStage = static_cast<size_t>(kTileV) * kBK * 2;  // 16 KB: one K block of the head tile

struct LbParams {
  int R, D, V, M, G, rpc, tpc, last;  // rpc, tpc, last: head rows, tiles and rows of the last tile of a group
  int W, nitem, gs, stages;  // hidden rows per block (a multiple of 16), blocks, CTAs per group, ring stages
  uint32_t* pool;   // [Rp][G * kPoolPerCta] value keys (0: none)
  uint32_t* bounds; // [R]
  uint64_t* cand;   // [R][G / gs][rpc]
  int* counts;      // [R][G / gs]
  WsHeader* hdr;
};
struct LbMaps {
  CUtensorMap w;    // head [V][D] bf16, box 64 x 128
  CUtensorMap wl;   // the same, box 64 x last (a CTA's last tile)
  CUtensorMap h;    // hidden [R][D] bf16, box 64 x W
};
// One stage: one K block of the head tile (16 KB) and of the hidden block (W rows x 128 bytes), 1 KB-aligned.
__host__ __device__ inline size_t lb_stage_bytes(int W) { return kAStage + static_cast<size_t>(W) * kBK * 2; }
// Dynamic shared memory: alignment slack, the ring, and (filter pass) every row's threshold and count.
__host__ __device__ inline size_t lb_smem_bytes(int W, int stages, int R) {
  return 1024 + stages * lb_stage_bytes(W) + 8 * static_cast<size_t>(R);
}
template <bool kPool>
__global__ void __launch_bounds__(kThreads, 1) lh_block_kernel(LbParams p, const __grid_constant__ LbMaps maps) {
  extern __shared__ float4 smem_f4[];
  unsigned char* ring =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_f4) + 1023) & ~uintptr_t(1023));
  const size_t stage = lb_stage_bytes(p.W);
  float* s_thr = reinterpret_cast<float*>(ring + p.stages * stage);  // [R] each row's bound as a value
  int* s_cnt = reinterpret_cast<int*>(s_thr + p.R);                  // [R]
  __shared__ uint64_t full[kMaxStages], empty[kMaxStages], tfull[2], tempty[2];
  __shared__ uint32_t s_tmem;
  __shared__ unsigned s_issued, s_used;  // stage loads issued and waited for (failure drain)
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int G = static_cast<int>(gridDim.x), bid = static_cast<int>(blockIdx.x);
  const int R = p.R, W = p.W, S = p.stages, nkb = p.D / kBK, nitem = p.nitem, gs = p.gs;
  const int grp = bid / gs, rk = bid % gs, ngroups = G / gs;
  const int row0 = grp * p.rpc, nrows = min(p.rpc, p.V - row0);  // the group's head rows
  const int my_tiles = nrows > 0 ? (nrows + kTileV - 1) / kTileV : 0;
  // Filter pass: item it is (tile it / nb, hidden block rk + gs (it % nb)), nb = nitem / gs blocks per CTA. Pool
  // pass: the CTA's sample tile, the group's tile rk (zero-filled or another group's rows past the group's end: not
  // valid, keys 0; every pool slot is written and no logit is offered twice), against every hidden block.
  const int nb = kPool ? nitem : nitem / gs;
  const int items = kPool ? nitem : my_tiles * nb;
  auto tile_of = [&](int it) { return kPool ? rk : it / nb; };
  auto block_of = [&](int it) { return kPool ? it : rk + gs * (it % nb); };
  const uint32_t cols = 2 * W <= 32 ? 32u : 2 * W <= 64 ? 64u : 2 * W <= 128 ? 128u : 2 * W <= 256 ? 256u : 512u;
  if (t == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);  // one arrival per epilogue warp
    }
    mbar_fence_init();
    s_issued = s_used = 0u;
  }
  if (!kPool) {
    for (int r = t; r < R; r += kThreads) {
      const uint32_t b = __ldcg(p.bounds + r);
      s_thr[r] = b <= 0x007FFFFFu ? -INFINITY : value_of_key_f32(b);  // at or below the key of -inf: no bound
      s_cnt[r] = 0;
    }
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(cols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;
  bool ok = true, nan = false;

  if (warp == 0 && lane == 0) {  // TMA producer: K block kb of item it (its tile and its hidden block) into a stage
    unsigned n = 0;
    for (int it = 0; it < items && ok; ++it) {
      const int i = tile_of(it), j = block_of(it);
      const bool lastt = !kPool && i == p.tpc - 1;  // the group's last tile reads `last` head rows
      const CUtensorMap* wm = lastt ? &maps.wl : &maps.w;
      const uint32_t tx = static_cast<uint32_t>(((lastt ? p.last : kTileV) + W) * kBK * 2);
      for (int kb = 0; kb < nkb; ++kb, ++n) {
        const unsigned st = n % S, use = n / S;
        if (use > 0) ok = mbar_wait(&empty[st], (use - 1) & 1u, kBudgetNs);
        if (!ok) break;
        unsigned char* a = ring + st * stage;
        mbar_expect_tx(&full[st], tx);
        tma_load_2d(a, wm, kb * kBK, row0 + i * kTileV, &full[st]);
        tma_load_2d(a + kAStage, &maps.h, kb * kBK, j * W, &full[st]);
        s_issued = n + 1u;
      }
    }
  } else if (warp == 1 && lane == 0) {  // MMA issuer: item it accumulates in TMEM buffer it % 2
    const uint32_t idesc = umma_idesc(W, kTileV);
    unsigned n = 0;
    for (int it = 0; it < items && ok; ++it) {
      const int buf = it & 1;
      if (it >= 2) ok = mbar_wait(&tempty[buf], static_cast<unsigned>((it >> 1) - 1) & 1u, kBudgetNs);
      if (!ok) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      for (int kb = 0; kb < nkb; ++kb, ++n) {
        const unsigned st = n % S, use = n / S;
        ok = mbar_wait(&full[st], use & 1u, kBudgetNs);
        if (!ok) break;
        s_used = n + 1u;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a = smem_u32(ring + st * stage), bb = a + static_cast<uint32_t>(kAStage);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          umma_f16(tmem + static_cast<uint32_t>(buf * W), umma_desc_sw128(a + 32 * k), umma_desc_sw128(bb + 32 * k),
                   idesc, (kb > 0 || k > 0) ? 1u : 0u);
        umma_commit(&empty[st]);  // the stage is free once these MMAs have read it
      }
      if (ok) umma_commit(&tfull[buf]);  // the item's accumulator is complete after these MMAs
    }
  } else if (warp >= 4) {  // epilogue: warp 4 + q drains TMEM lanes 32 q .. 32 q + 31 (head rows of the tile)
    const int q = warp & 3;
    const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16);
    const int np = G * kPoolPerCta;
    for (int it = 0; it < items && ok; ++it) {
      const int i = tile_of(it), j = block_of(it), buf = it & 1;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&tfull[buf], static_cast<unsigned>(it >> 1) & 1u, kBudgetNs));
      if (!ok) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int loc = i * kTileV + 32 * q + lane;
      const bool valid = loc < nrows;  // rows past the range hold stale shared memory (or zero fill)
      const int r0 = j * W;            // hidden row of column 0
      const uint32_t tb = tq + static_cast<uint32_t>(buf * W);
      for (int c0 = 0; c0 < W; c0 += 32) {
        uint32_t v0[16], v1[16];
        tmem_ld16x2(tb + static_cast<uint32_t>(c0), tb + static_cast<uint32_t>(c0 + 16), v0, v1);
        if (kPool) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const uint32_t x = jj < 16 ? v0[jj] : v1[jj - 16];
            const int c = c0 + jj, r = r0 + c;
            const bool isnan = (x & 0x7FFFFFFFu) > 0x7F800000u;
            const uint32_t k = valid && !isnan && c < W && r < R ? key_of_f32(x) : 0u;
            const uint32_t m1 = __reduce_max_sync(0xFFFFFFFFu, k);
            const int win = __ffs(__ballot_sync(0xFFFFFFFFu, k == m1)) - 1;
            const uint32_t m2 = __reduce_max_sync(0xFFFFFFFFu, lane == win ? 0u : k);
            if (lane == 0 && c < W && r < R) {
              uint32_t* pr = p.pool + static_cast<size_t>(r) * np + bid * kPoolPerCta + q * kPoolPerQuarter;
              pr[0] = m1;
              pr[1] = m2;
            }
          }
        } else if (valid) {
          // fast path: one compare per logit against its row's threshold (NaN fails `<` and takes the rare path)
          unsigned hit = 0;
#pragma unroll
          for (int jj = 0; jj < 32; jj += 4) {
            const int c = c0 + jj, r = r0 + c;
            float4 th = make_float4(INFINITY, INFINITY, INFINITY, INFINITY);
            if (c < W && r + 3 < R) {
              th = *reinterpret_cast<const float4*>(s_thr + r);
            } else {
              if (c < W && r < R) th.x = s_thr[r];
              if (c < W && r + 1 < R) th.y = s_thr[r + 1];
              if (c < W && r + 2 < R) th.z = s_thr[r + 2];
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t x = jj + e < 16 ? v0[jj + e] : v1[jj + e - 16];
              const float te = e == 0 ? th.x : e == 1 ? th.y : e == 2 ? th.z : th.w;
              hit |= static_cast<unsigned>(!(__uint_as_float(x) < te)) << (jj + e);
            }
          }
          if (hit) {  // rare: candidates (or NaNs) among these 32 logits
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const uint32_t x = jj < 16 ? v0[jj] : v1[jj - 16];
              const int c = c0 + jj, r = r0 + c;
              if (!((hit >> jj) & 1u) || c >= W || r >= R) continue;
              if ((x & 0x7FFFFFFFu) > 0x7F800000u) {
                nan = true;
                continue;
              }
              const int pos = atomicAdd(&s_cnt[r], 1);  // < rpc: the group holds rpc logits of a row
              p.cand[(static_cast<size_t>(r) * ngroups + grp) * p.rpc + pos] =
                  pack_candidate(key_of_f32(x), static_cast<uint32_t>(row0 + loc));
            }
          }
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);  // the MMAs may overwrite this buffer
    }
  }
  ok = __syncthreads_and(ok);
  if (!ok && t == 0) {
    record_error(p.hdr, DT_ERR_TIMEOUT);
    atomicExch(&p.hdr->abort, 1u);
    // stage loads issued but never waited for must land before the CTA leaves (bounded)
    for (unsigned n = s_used; n < s_issued; ++n) mbar_wait(&full[n % S], (n / S) & 1u, kBudgetNs);
  }
  if (__syncthreads_or(nan) && t == 0) record_error(p.hdr, DT_ERR_NUMERIC);
  if (!kPool)  // the rows of this CTA's hidden blocks: their lists of this group
    for (int r = t; r < R; r += kThreads)
      if ((r / W) % gs == rk) p.counts[static_cast<size_t>(r) * ngroups + grp] = s_cnt[r];
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(cols) : "memory");
}

// A warp per row: the M-th largest key of the row's pool (np keys, 0: none), to the top 16 bits (the largest v with
// at least M pool keys whose top 16 bits are >= v, shifted back): a lower bound of the row's M-th largest logit. 0
// (every logit a candidate) when the pool holds fewer than M values.
constexpr int kBoundWarps = 8;
constexpr int kBoundPerLane = 64;  // pool keys per lane at most: np <= 2048
__global__ void __launch_bounds__(32 * kBoundWarps) lh_bound_kernel(const uint32_t* __restrict__ pool, int np, int R,
                                                                     int M, uint32_t* __restrict__ bounds) {
  __shared__ uint16_t s_pool[kBoundWarps][32 * kBoundPerLane];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kBoundWarps + warp;
  if (r >= R) return;
  const uint32_t* pr = pool + static_cast<size_t>(r) * np;
  uint16_t* sp = s_pool[warp];
  for (int i = lane; i < np; i += 32) sp[i] = static_cast<uint16_t>(__ldcg(pr + i) >> 16);
  __syncwarp();
  uint32_t v = 0;
  for (int bit = 15; bit >= 0; --bit) {
    const uint32_t cand = v | (1u << bit);
    unsigned cnt = 0;
    for (int i = lane; i < np; i += 32) cnt += sp[i] >= cand;
    if (static_cast<int>(__reduce_add_sync(0xFFFFFFFFu, cnt)) >= M) v = cand;
  }
  if (lane == 0) bounds[r] = v << 16;
}

// A CTA per row: the row's top M from the G lists of the filter pass.
__global__ void __launch_bounds__(kSelThreads) lh_select_kernel(const uint64_t* __restrict__ cand,
                                                                const int* __restrict__ counts, int G, int rpc, int M,
                                                                int32_t* __restrict__ ids, float* __restrict__ vals) {
  extern __shared__ uint4 smem_u4[];
  __shared__ int s_warp[kSelThreads / 32];
  __shared__ int s_n;
  const int r = blockIdx.x;
  const uint64_t* rc = cand + static_cast<size_t>(r) * G * rpc;
  const int* rn = counts + static_cast<size_t>(r) * G;
  select_words<false, kSelThreads>(
      [&](int c) { return __ldcg(rn + c); }, G, M,
      [&](int c, int i) { return __ldcg(rc + static_cast<size_t>(c) * rpc + i); }, ids + static_cast<size_t>(r) * M,
      vals + static_cast<size_t>(r) * M, *reinterpret_cast<SelectSmem*>(smem_u4), s_warp, &s_n);
}

constexpr int kLhKbps = 4;  // K blocks per stage (the largest divisor of D / 64 up to this): 512 bytes of a head row
inline int lh_kbps_setting(int nkb) {
  int k = kLhKbps < nkb ? kLhKbps : nkb;
  while (nkb % k) --k;
  return k;
}

struct LhLayout {
  size_t pool, bounds, counts, cand, bytes;
  int Rp, rpc, tpc, last;
};
inline LhLayout lh_layout(int R, int V, int G) {
  LhLayout L{};
  L.Rp = (R + 15) / 16 * 16;
  L.rpc = (V + G - 1) / G;                       // head rows per CTA, contiguous
  L.tpc = (L.rpc + kTileV - 1) / kTileV;         // tiles per CTA
  L.last = L.rpc - kTileV * (L.tpc - 1);         // rows of a CTA's last tile
  L.pool = align_up(sizeof(WsHeader));
  L.bounds = align_up(L.pool + sizeof(uint32_t) * static_cast<size_t>(L.Rp) * G * kPoolPerCta);
  L.counts = align_up(L.bounds + sizeof(uint32_t) * static_cast<size_t>(R));
  L.cand = align_up(L.counts + sizeof(int) * static_cast<size_t>(R) * G);
  L.bytes = align_up(L.cand + sizeof(uint64_t) * static_cast<size_t>(R) * G * L.rpc);
  return L;
}

// The blocked passes (more than 64 rows): four launches on the stream, none waiting on another CTA.
dt_status lh_blocked(int R, int D, int V, int M, const void* hidden, const void* w_head, int32_t* out_ids,
                     float* out_vals, char* ws, const LhLayout& L, const DeviceInfo& di, cudaStream_t stream) {
  const int G = di.sms;
  const int W = R < kItemMax ? (R + 15) / 16 * 16 : kItemMax;
  // the ring: as many stages as the shared memory takes beside every row's threshold and count
  const long long room = static_cast<long long>(di.optin) - static_cast<long long>(kStaticReserve) - 1024 -
                         8LL * static_cast<long long>(R);
  long long stages = room > 0 ? room / static_cast<long long>(lb_stage_bytes(W)) : 0;
  stages = stages < kMaxStages ? stages : kMaxStages;
  if (stages < 2) return DT_ERR_UNSUPPORTED;
  const int nitem = (R + W - 1) / W;
  int gs = 4;  // CTAs per group: a divisor of the hidden blocks and of the grid
  while (gs > 1 && (nitem % gs != 0 || G % gs != 0)) gs /= 2;
  const int ngroups = G / gs;
  LbParams p{};
  p.R = R; p.D = D; p.V = V; p.M = M; p.G = G;
  p.rpc = (V + ngroups - 1) / ngroups;                  // a group's head rows, contiguous
  p.tpc = (p.rpc + kTileV - 1) / kTileV;
  p.last = p.rpc - kTileV * (p.tpc - 1);
  p.W = W; p.nitem = nitem; p.gs = gs; p.stages = static_cast<int>(stages);
  p.pool = reinterpret_cast<uint32_t*>(ws + L.pool);
  p.bounds = reinterpret_cast<uint32_t*>(ws + L.bounds);
  p.counts = reinterpret_cast<int*>(ws + L.counts);
  p.cand = reinterpret_cast<uint64_t*>(ws + L.cand);
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  LbMaps maps{};
  if (!encode_bf16_2d(&maps.w, w_head, static_cast<uint64_t>(D), static_cast<uint64_t>(V), static_cast<uint64_t>(D),
                      kBK, kTileV) ||
      !encode_bf16_2d(&maps.wl, w_head, static_cast<uint64_t>(D), static_cast<uint64_t>(V), static_cast<uint64_t>(D),
                      kBK, static_cast<uint32_t>(p.last)) ||
      !encode_bf16_2d(&maps.h, hidden, static_cast<uint64_t>(D), static_cast<uint64_t>(R), static_cast<uint64_t>(D),
                      kBK, static_cast<uint32_t>(W)))
    return DT_ERR_CUDA;
  const size_t smem = lb_smem_bytes(W, p.stages, R);
  const void* fpool = reinterpret_cast<const void*>(lh_block_kernel<true>);
  const void* ffilt = reinterpret_cast<const void*>(lh_block_kernel<false>);
  if (ensure_dynamic_smem(fpool, smem) != cudaSuccess || ensure_dynamic_smem(ffilt, smem) != cudaSuccess ||
      ensure_dynamic_smem(reinterpret_cast<const void*>(lh_select_kernel), sizeof(SelectSmem)) != cudaSuccess)
    return DT_ERR_CUDA;
  lh_block_kernel<true><<<G, kThreads, smem, stream>>>(p, maps);
  lh_bound_kernel<<<(R + kBoundWarps - 1) / kBoundWarps, 32 * kBoundWarps, 0, stream>>>(p.pool, G * kPoolPerCta, R, M,
                                                                                         p.bounds);
  lh_block_kernel<false><<<G, kThreads, smem, stream>>>(p, maps);
  lh_select_kernel<<<R, kSelThreads, sizeof(SelectSmem), stream>>>(p.cand, p.counts, ngroups, p.rpc, M, out_ids,
                                                                   out_vals);
  return cuda_status(cudaGetLastError());
}

}  // namespace
}  // namespace dt

extern "C" size_t dt_lmhead_workspace_bytes(int R, int D, int V, int M) {
  if (R < 1 || D < 1 || V < 1 || M < 1) return 0;
  dt::DeviceInfo di{};
  if (dt::current_device_info(&di) != cudaSuccess) return 0;
  return dt::lh_layout(R, V, di.sms).bytes;
}

extern "C" dt_status dt_lmhead_topm(int R, int D, int V, int M, const void* hidden, const void* w_head, dt_dtype dtype,
                                    int32_t* out_ids, float* out_vals, void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream) {
  using namespace dt;
  if (R < 0 || D < 1 || V < 1 || M < 1 || M > V) return DT_ERR_INVALID_ARG;
  if (dtype != DT_F32 && dtype != DT_BF16) return DT_ERR_INVALID_ARG;
  if (R == 0) return DT_OK;
  const void* ptrs[] = {hidden, w_head, out_ids, out_vals, workspace};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return DT_ERR_INVALID_ARG;
  if (dtype != DT_BF16 || D % kBK != 0 || M > DT_MAX_M || R > DT_LMHEAD_MAX_ROWS) return DT_ERR_UNSUPPORTED;
  if (static_cast<long long>(V) + kTileV > INT_MAX) return DT_ERR_UNSUPPORTED;
  DeviceInfo di{};
  if (current_device_info(&di) != cudaSuccess) return DT_ERR_CUDA;
  const LhLayout L = lh_layout(R, V, di.sms);
  if (workspace_bytes < L.bytes) return DT_ERR_INVALID_ARG;
  if (di.sms * kPoolPerCta > kThreads * kPoolPerThread) return DT_ERR_UNSUPPORTED;  // the pool of a row in registers
  // the CTA's slice of logits must fit its tensor memory for the one-launch kernel; otherwise the blocked passes
  if (R > kMaxRp || L.tpc * L.Rp > kTmemMax)
    return lh_blocked(R, D, V, M, hidden, w_head, out_ids, out_vals, static_cast<char*>(workspace), L, di, stream);
  // the ring: K blocks per stage and as many stages as the shared memory takes (a reserve for the kernel's static
  // shared memory, about 2 KB)
  const int nkb = D / kBK;
  const int kbps = lh_kbps_setting(nkb);
  const size_t room = static_cast<size_t>(di.optin) - kStaticReserve - 1024;
  int stages = static_cast<int>(room / (kbps * lh_block_bytes(L.Rp)));
  stages = stages < kMaxStages ? stages : kMaxStages;
  if (stages < 2) return DT_ERR_UNSUPPORTED;
  const size_t smem = lh_smem_bytes(L.Rp, stages, kbps);
  if (smem + kStaticReserve > static_cast<size_t>(di.optin)) return DT_ERR_UNSUPPORTED;
  LhMaps maps{};
  if (!encode_bf16_2d(&maps.w, w_head, static_cast<uint64_t>(D), static_cast<uint64_t>(V), static_cast<uint64_t>(D),
                      kBK, kTileV) ||
      !encode_bf16_2d(&maps.wl, w_head, static_cast<uint64_t>(D), static_cast<uint64_t>(V), static_cast<uint64_t>(D),
                      kBK, static_cast<uint32_t>(L.last)) ||
      !encode_bf16_2d(&maps.h, hidden, static_cast<uint64_t>(D), static_cast<uint64_t>(R), static_cast<uint64_t>(D),
                      kBK, static_cast<uint32_t>(L.Rp)))
    return DT_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  LhParams p{};
  p.R = R; p.Rp = L.Rp; p.D = D; p.V = V; p.M = M; p.rpc = L.rpc; p.tpc = L.tpc; p.last = L.last; p.G = di.sms;
  p.stages = stages; p.kbps = kbps;
  p.pool = reinterpret_cast<uint32_t*>(ws + L.pool);
  p.bounds = reinterpret_cast<uint32_t*>(ws + L.bounds);
  p.counts = reinterpret_cast<int*>(ws + L.counts);
  p.cand = reinterpret_cast<uint64_t*>(ws + L.cand);
  p.ids = out_ids;
  p.vals = out_vals;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.timeout_ns = barrier_timeout_ns();
  const void* fn = reinterpret_cast<const void*>(lmhead_topm_kernel);
  if (ensure_dynamic_smem(fn, smem) != cudaSuccess) return DT_ERR_CUDA;
  void* args[] = {&p, &maps};
  return cuda_status(cudaLaunchCooperativeKernel(fn, dim3(static_cast<unsigned>(di.sms)), dim3(kThreads), args, smem,
                                                 stream));
}
