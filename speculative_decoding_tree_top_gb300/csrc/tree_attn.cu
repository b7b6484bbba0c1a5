// dt_tree_attention — the verify pass's attention over the prefix and the draft tree with the ancestor-only mask.
//
// Method: blog.captcha.la, "Methodology — deep read" (the prefix-closed tree is verified in a single target forward
// pass with an unmodified ancestor-only causal mask, borrowed from DDTree/SpecInfer); gist.science, "Composants
// Clés — Vérification" (standard tree attention, unchanged and lossless). For request b, query head h and tree node
// i the visible keys are the L prefix positions and the tree positions L + t with mask[b][i][t] = 1;
// out = softmax(scale q.k) v over them; query head h reads key/value head h / (Hq / Hkv).
//
// GB300 design (flash decoding on the 5th-generation tensor cores): the n tree nodes of the G = Hq / Hkv query heads
// that share a key/value head are one block of G n <= 64 query rows, so each key and value row is read once per
// (request, key/value head) and feeds 64 rows of dot products. The key blocks of all (request, key/value head)
// pairs, flattened, are split evenly over one CTA per SM (a CTA's share may span several pairs: one segment each).
// A CTA streams its keys and values by TMA, computes S = Q K^T and O += P V with tcgen05 MMAs whose accumulators
// live in tensor memory, and runs the softmax (base 2, running maximum raised lazily) from tensor memory, one thread
// per query row (tree_attn_tc below). A segment that covers its whole (request, key/value head) writes the output
// itself; a second launch, a programmatic dependent of the first, combines the segments of the rows of pairs split
// over several CTAs. Memory bound: the key and value rows are the bytes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "dt_internal.cuh"
#include "umma.cuh"

namespace dt {
namespace {

constexpr int kD = 128;           // head dimension
constexpr int kRows = 64;         // query rows per CTA: G x n, padded
constexpr int kMaxNodes = 64;

struct TaParams {
  int B, n, L, T, Hq, Hkv, G, R;
  int nb;              // key blocks of 64 per (request, key/value head)
  int grid, maxseg;    // CTAs of the partial launch; partial slots per (request, key/value head)
  int wpc;             // whole pairs per CTA: CTA c takes pairs [wpc c, wpc (c + 1)) whole
  long long rwork;     // the other pairs' key blocks, (B Hkv - wpc grid) nb, split evenly over the CTAs
  const unsigned short* q;   // [B][n][Hq][kD] bf16
  const unsigned short* k;   // [B][Hkv][T][kD] bf16
  const unsigned short* v;   // [B][Hkv][T][kD] bf16
  const uint8_t* mask;       // [B][n][n]
  float scale_log2;          // scale * log2(e)
  float* part;               // [B Hkv][maxseg][kRows][kD] unnormalised outputs of each segment
  float* ml;                 // [B Hkv][maxseg][kRows][2] running max (base 2) and sum
  float* out;                // [B][n][Hq][kD]
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The CTA whose even share of the flattened key blocks holds block x: CTA c takes [c W / G, (c + 1) W / G).
__host__ __device__ __forceinline__ int block_owner(long long x, long long W, int G) {
  return static_cast<int>(((x + 1) * G - 1) / W);
}

// ---- the partial launch on tcgen05 -------------------------------------------------------------------------------
// One CTA per SM takes an even share of the flattened (request, key/value head, block of 64 keys) space, as above;
// each run of its share within one (request, key/value head) is a segment. The roles run through all of the CTA's
// segments without stopping between them:
//   warp 2 (one thread) loads each segment's query rows by 4-D TMA (the box is the G heads x n nodes of the pair, so
//     row r = i G + gi holds node i of query head kvh G + gi) into one of two Q buffers, and streams the segment's
//     key and value blocks by 3-D TMA (rows past a pair's end read as zero) through a ring of five 32 KB stages;
//   warp 3 (one thread) issues the MMAs;
//   warps 4 and 5 run the softmax, thread r owning query row r (TMEM lane r; rows past G n are padding and are left
//     to whatever their rows of Q and P hold), so no row statistic needs a shuffle.
// Per block j:
//   S_j = Q K_j^T     M = 128 (query rows), N = 64 keys, K = 128: TMEM columns [64 (j % 2), +64), double-buffered
//                     so that S_{j+1} is computed while block j's softmax runs;
//   softmax           visibility bits (prefix keys, the node's ancestor row for tree keys, nothing past the pair's
//                     end), scale (base 2), P = 2^(s - m) rounded to bf16 into shared memory (one 128-byte swizzled
//                     row per query row, double-buffered);
//   O += P_j V_j      M = 128, N = 128 (the head dimension), K = 64 keys, V read as an MN-major operand straight
//                     from its TMA tile: TMEM columns [128 + 128 (segment % 2), +128), double-buffered per segment so
//                     that a segment's output is read out while the next one accumulates.
// The running maximum m of a row is raised only when a block's maximum exceeds it by more than 2^8 (then O is
// rescaled in TMEM, rarely): the weights stay below 2^8, and O and the row sum l are taken against the same m, which
// is what the combine kernel reads with them. The segment's O, m and l go to its partial slot.
constexpr int kTcKeys = 64;       // keys per block
constexpr int kTcStages = 5;      // key/value ring stages
constexpr int kTcThreads = 256;
constexpr float kTcLazy = 8.f;    // log2 headroom before the running maximum is raised
constexpr uint64_t kTcBudgetNs = 4000000000ull;
constexpr uint32_t kTcBox = kTcKeys * 128;          // one 64-row x 64-dim box: 8 KB
constexpr uint32_t kTcQBytes = 2 * kTcBox;          // one Q buffer: dims 0-63, then 64-127, 64 rows each
constexpr uint32_t kTcStageBytes = 4 * kTcBox;      // K (2 boxes), then V (2 boxes)
constexpr uint32_t kTcPBytes = 128 * kTcKeys * 2;   // 128 rows x 64 keys x 2 bytes
// Q buffers first: an MMA reads 128 rows of a Q box, rows 64-127 (padding) from whatever follows it, all allocated
constexpr size_t kTcSmem = 1024 + 2 * kTcQBytes + kTcStages * kTcStageBytes + 2 * kTcPBytes;

struct TaMaps {
  CUtensorMap q;     // [B][n][Hq][128] bf16, box 64 dims x G heads x n nodes x 1
  CUtensorMap k, v;  // [B Hkv][T][128] bf16, box 64 dims x 64 keys x 1
};

// 2^x by the hardware's approximate exponential (relative error about 2^-22, far below the bf16 rounding of the
// weights it feeds; subnormal results flush to zero: weights below 2^-126 of the row's maximum).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_ld16_ta(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// One segment of a CTA's share: (request, key/value head) pair, its blocks [j0, j0 + nblk), and its partial slot.
// A CTA's share is its wpc whole pairs, then its even share [rx0, rx1) of the remaining pairs' blocks (flattened);
// x runs over the share: [0, wpc nb) the whole pairs, then the rest.
struct TaSeg {
  int pair, b, kvh, j0, nblk, slot;
};
struct TaShare {
  long long rx0, len;  // the share of the remaining blocks starts at rx0; x runs over [0, len)
};
__device__ __forceinline__ TaShare ta_share(const TaParams& p) {
  const long long c = blockIdx.x;
  const long long rx0 = c * p.rwork / p.grid, rx1 = (c + 1) * p.rwork / p.grid;
  return TaShare{rx0, static_cast<long long>(p.wpc) * p.nb + (rx1 - rx0)};
}
__device__ __forceinline__ TaSeg ta_segment(const TaParams& p, const TaShare& sh, long long& x) {
  TaSeg g;
  const long long wx = static_cast<long long>(p.wpc) * p.nb;
  if (x < wx) {  // a whole pair
    g.pair = static_cast<int>(blockIdx.x) * p.wpc + static_cast<int>(x / p.nb);
    g.j0 = 0;
    g.nblk = p.nb;
    g.slot = 0;
    x += p.nb;
  } else {  // a run of the remaining pairs' blocks
    const long long rx = sh.rx0 + (x - wx), rx1 = sh.rx0 + (sh.len - wx);
    const int rp = static_cast<int>(rx / p.nb);
    const long long pfirst = static_cast<long long>(rp) * p.nb;
    const int bend = static_cast<int>(min(rx1, pfirst + p.nb) - pfirst);
    g.pair = p.wpc * p.grid + rp;
    g.j0 = static_cast<int>(rx - pfirst);
    g.nblk = bend - g.j0;
    g.slot = static_cast<int>(blockIdx.x) - block_owner(pfirst, p.rwork, p.grid);
    x += g.nblk;
  }
  g.b = g.pair / p.Hkv;
  g.kvh = g.pair % p.Hkv;
  return g;
}

__global__ void __launch_bounds__(kTcThreads, 1) tree_attn_tc(TaParams p, const __grid_constant__ TaMaps maps,
                                                              WsHeader* hdr) {
  extern __shared__ float4 smem_f4[];
  unsigned char* sq =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_f4) + 1023) & ~uintptr_t(1023));
  unsigned char* skv = sq + 2 * kTcQBytes;
  unsigned char* sp = skv + kTcStages * kTcStageBytes;
  __shared__ uint64_t kv_full[kTcStages], kv_empty[kTcStages], s_full[2], p_full[2], o_done[2];
  __shared__ uint64_t q_full[2], q_empty[2], o_free[2];
  __shared__ uint32_t s_tmem;
  __shared__ unsigned s_kv_issued, s_kv_used, s_q_issued, s_q_used;  // copies issued and consumed (failure drain)
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  if (t == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 2);  // one arrival per softmax warp
      mbar_init(&o_done[i], 1);
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&o_free[i], 2);
    }
    mbar_fence_init();
  }
  if (t == 0) s_kv_issued = s_kv_used = s_q_issued = s_q_used = 0u;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(512) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the combination may launch (it waits for us)
  bool ok = true;
  const TaShare sh = ta_share(p);

  if (warp == 2 && lane == 0) {  // TMA producer
    unsigned g = 0;
    const uint32_t qtx = static_cast<uint32_t>(2 * 128 * p.R);
    int si = 0;
    for (long long x = 0; x < sh.len && ok; ++si) {
      const TaSeg sg = ta_segment(p, sh, x);
      const unsigned qb = static_cast<unsigned>(si) & 1u;
      if (si >= 2) ok = mbar_wait(&q_empty[qb], static_cast<unsigned>((si >> 1) - 1) & 1u, kTcBudgetNs);
      if (!ok) break;
      unsigned char* qd = sq + qb * kTcQBytes;
      mbar_expect_tx(&q_full[qb], qtx);
      tma_load_4d(qd, &maps.q, 0, sg.kvh * p.G, 0, sg.b, &q_full[qb]);
      tma_load_4d(qd + kTcBox, &maps.q, 64, sg.kvh * p.G, 0, sg.b, &q_full[qb]);
      s_q_issued = static_cast<unsigned>(si) + 1u;
      for (int j = 0; j < sg.nblk && ok; ++j, ++g) {
        const unsigned st = g % kTcStages, use = g / kTcStages;
        if (use > 0) ok = mbar_wait(&kv_empty[st], (use - 1) & 1u, kTcBudgetNs);
        if (!ok) break;
        unsigned char* d = skv + st * kTcStageBytes;
        const int key = (sg.j0 + j) * kTcKeys;
        mbar_expect_tx(&kv_full[st], kTcStageBytes);
        tma_load_3d(d, &maps.k, 0, key, sg.pair, &kv_full[st]);
        tma_load_3d(d + kTcBox, &maps.k, 64, key, sg.pair, &kv_full[st]);
        tma_load_3d(d + 2 * kTcBox, &maps.v, 0, key, sg.pair, &kv_full[st]);
        tma_load_3d(d + 3 * kTcBox, &maps.v, 64, key, sg.pair, &kv_full[st]);
        s_kv_issued = g + 1u;
      }
    }
  } else if (warp == 3 && lane == 0) {  // MMA issuer
    const uint32_t id_s = umma_idesc(kTcKeys, 128), id_o = umma_idesc(kD, 128) | (1u << 16);  // O: V MN-major
    unsigned g = 0;
    int si = 0;
    for (long long x = 0; x < sh.len && ok; ++si) {
      const TaSeg sg = ta_segment(p, sh, x);
      const unsigned qb = static_cast<unsigned>(si) & 1u;
      const uint32_t aq = smem_u32(sq + qb * kTcQBytes), to = tmem + 128u + 128u * qb;
      ok = mbar_wait(&q_full[qb], static_cast<unsigned>(si >> 1) & 1u, kTcBudgetNs);
      if (ok) s_q_used = static_cast<unsigned>(si) + 1u;
      // this segment's O buffer was read out by the softmax of segment si - 2
      if (ok && si >= 2) ok = mbar_wait(&o_free[qb], static_cast<unsigned>((si >> 1) - 1) & 1u, kTcBudgetNs);
      if (!ok) break;
      auto issue_s = [&](unsigned gs) {  // S = Q K^T of block gs into TMEM columns [64 (gs % 2), +64)
        const unsigned st = gs % kTcStages;
        if (!mbar_wait(&kv_full[st], (gs / kTcStages) & 1u, kTcBudgetNs)) return false;
        s_kv_used = gs + 1u;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t bk = smem_u32(skv + st * kTcStageBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kTcBox + (kk & 3) * 32u;
          umma_f16(tmem + (gs & 1u) * kTcKeys, umma_desc_sw128(aq + off), umma_desc_sw128(bk + off), id_s,
                   kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[gs & 1u]);
        return true;
      };
      ok = issue_s(g);
      if (ok && sg.nblk == 1) umma_commit(&q_empty[qb]);  // the segment's last S: Q may be reloaded after it
      for (int j = 0; j < sg.nblk && ok; ++j, ++g) {
        const unsigned st = g % kTcStages;
        if (j + 1 < sg.nblk) {  // its S buffer was freed by block g - 1's softmax (waited for below, one block ago)
          ok = issue_s(g + 1);
          if (ok && j + 2 == sg.nblk) umma_commit(&q_empty[qb]);
        }
        if (ok) ok = mbar_wait(&p_full[g & 1u], (g >> 1) & 1u, kTcBudgetNs);  // P written, O rescaled if it had to be
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t ap = smem_u32(sp + (g & 1u) * kTcPBytes), bv = smem_u32(skv + st * kTcStageBytes + 2 * kTcBox);
#pragma unroll
        for (int kk = 0; kk < kTcKeys / 16; ++kk)
          umma_f16(to, umma_desc_sw128(ap + 32u * kk), umma_desc_sw128_mn(bv + 2048u * kk, kTcBox, 1024u), id_o,
                   (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&kv_empty[st]);  // the block's keys and values have been read
        umma_commit(&o_done[g & 1u]);
      }
    }
  } else if (warp == 4 || warp == 5) {  // softmax: thread r owns query row r (TMEM lane r)
    const int r = 32 * (warp & 3) + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const bool live = r < p.R;
    const int node = live ? r / p.G : 0, gi = live ? r % p.G : 0;  // row r = node G + gi
    unsigned g = 0;
    int si = 0;
    for (long long x = 0; x < sh.len && ok; ++si) {
      const TaSeg sg = ta_segment(p, sh, x);
      const unsigned qb = static_cast<unsigned>(si) & 1u;
      const uint32_t to = tl + 128u + 128u * qb;
      unsigned long long mbits = 0;  // bit c: tree position c is on the node's ancestor row
      if (live) {
        const uint8_t* mr = p.mask + (static_cast<size_t>(sg.b) * p.n + node) * p.n;
        for (int c = 0; c < p.n; ++c) mbits |= static_cast<unsigned long long>(mr[c] != 0) << c;
      }
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < sg.nblk && ok; ++j, ++g) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&s_full[g & 1u], (g >> 1) & 1u, kTcBudgetNs));
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        uint32_t sv[4][16];
#pragma unroll
        for (int h = 0; h < 4; ++h) tmem_ld16_ta(tl + (g & 1u) * kTcKeys + 16u * h, sv[h]);
        // bit c: key kbase + c is visible to this row; then a branch-free pass over the 64 scores
        const int kbase = (sg.j0 + j) * kTcKeys, pre = p.L - kbase, lim = p.T - kbase;
        unsigned long long visb = 0;
        if (live) {
          const unsigned long long pbits = pre >= 64 ? ~0ull : pre <= 0 ? 0ull : (1ull << pre) - 1ull;
          unsigned long long tbits = 0;
          if (pre < 64) tbits = pre >= 0 ? mbits << pre : mbits >> (-pre);  // 0 <= -pre < n <= 64
          const unsigned long long lbits = lim >= 64 ? ~0ull : lim <= 0 ? 0ull : (1ull << lim) - 1ull;
          visb = (pbits | tbits) & lbits;
        }
        float s[64];
        float bmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          s[c] = (visb >> c) & 1ull ? __uint_as_float(sv[c >> 4][c & 15]) * p.scale_log2 : -INFINITY;
          bmax = fmaxf(bmax, s[c]);
        }
        // raise the running maximum only past the headroom; O is rescaled then, unless it holds nothing yet
        const bool raise = bmax > m + kTcLazy || (m == -INFINITY && bmax > -INFINITY);
        const bool rescale_o = raise && m > -INFINITY;
        const float mn = raise ? bmax : m;
        const float alpha = rescale_o ? fast_exp2(m - mn) : 1.f;
        m = mn;
        float ls = 0.f;
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float a = m == -INFINITY ? 0.f : fast_exp2(s[c] - m), bb = m == -INFINITY ? 0.f : fast_exp2(s[c + 1] - m);
          ls += a + bb;
          pk[c >> 1] = pack_bf16(a, bb);
        }
        l = l * alpha + ls;
        // P's buffer was last read by the O MMA of block g - 2; a rescale needs block g - 1's O MMA complete (it is
        // of this segment: m was finite). Commits complete in order.
        const bool any_rescale = __any_sync(0xFFFFFFFFu, rescale_o);
        if (g >= 2 || any_rescale) {
          const unsigned gw = any_rescale ? g - 1 : g - 2;
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(&o_done[gw & 1u], (gw >> 1) & 1u, kTcBudgetNs));
          if (!ok) break;
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        }
        if (any_rescale) {
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            uint32_t ov[16];
            tmem_ld16_ta(to + 16u * h, ov);
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st16(to + 16u * h, ov);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        unsigned char* prow = sp + (g & 1u) * kTcPBytes + r * 128;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          *reinterpret_cast<uint4*>(prow + ((cc ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the MMA reads P through the async proxy
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[g & 1u]);
      }
      if (!ok) break;
      // the segment's partial: O (unnormalised, against m), m and l of each live row, at row gi n + node
      const unsigned gl = g - 1;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&o_done[gl & 1u], (gl >> 1) & 1u, kTcBudgetNs));
      if (!ok) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      // A segment that covers its whole pair is the row's only one: it writes the normalised output itself (the
      // combination of one segment: weight exp2(0) = 1, then the same reciprocal), and the combination skips it.
      const bool whole = sg.nblk == p.nb;
      const size_t unit = static_cast<size_t>(sg.pair) * p.maxseg + sg.slot;
      const int prow_out = gi * p.n + node;
      float* po = whole ? p.out + ((static_cast<size_t>(sg.b) * p.n + node) * p.Hq + sg.kvh * p.G + gi) * kD
                        : p.part + (unit * kRows + prow_out) * kD;
      const float inv = !whole ? 1.f : l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        uint32_t ov[16];
        tmem_ld16_ta(to + 16u * h, ov);
        if (live)
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(po + 16 * h + e) =
                make_float4(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv,
                            __uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv);
      }
      if (live && !whole) {
        float* pm = p.ml + (unit * kRows + prow_out) * 2;
        pm[0] = m;
        pm[1] = l;
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[qb]);  // the next segment but one may accumulate here
    }
  }
  ok = __syncthreads_and(ok);
  if (!ok && t == 0) {
    record_error(hdr, DT_ERR_TIMEOUT);
    // copies issued but never waited for must land before the CTA leaves: wait for them too (bounded)
    for (unsigned g = s_kv_used; g < s_kv_issued; ++g) mbar_wait(&kv_full[g % kTcStages], (g / kTcStages) & 1u, kTcBudgetNs);
    for (unsigned q = s_q_used; q < s_q_issued; ++q) mbar_wait(&q_full[q & 1u], (q >> 1) & 1u, kTcBudgetNs);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
}

// The segments' partials of each (request, key/value head, query row), rescaled to the row's overall maximum and
// normalised by its overall sum; a lane works on four of the 128 output columns. With few segments per row (large
// batches) one warp takes a row; with many (a request's keys spread over many CTAs) one CTA takes a row and its warps
// split the segments, reducing through shared memory. CTAs stride over the rows with the grid sized to one resident
// wave, and a row's loads (its segments' maxima and sums, then their partials) are independent of one another.
constexpr int kMaxChunks = 1024;
constexpr int kCombineThreads = 256;
constexpr int kCombineWarps = kCombineThreads / 32;
constexpr int kCombinePerSm = 2048 / kCombineThreads;  // CTAs per SM: the SM's threads
constexpr int kWarpRowSegs = 8;                        // at most this many segments per row: a warp per row
struct RowRef {
  size_t u0;  // first partial slot of the row's (request, key/value head)
  int r, b, kvh, nseg;
};
__device__ __forceinline__ RowRef row_ref(const TaParams& p, long long u) {
  RowRef q;
  q.r = static_cast<int>(u % p.R);
  const int pair = static_cast<int>(u / p.R);
  q.b = pair / p.Hkv;
  q.kvh = pair % p.Hkv;
  q.u0 = static_cast<size_t>(pair) * p.maxseg;
  q.nseg = 1;  // a whole pair
  const int rp = pair - p.wpc * p.grid;
  if (rp >= 0) {
    const long long pfirst = static_cast<long long>(rp) * p.nb;
    q.nseg = block_owner(pfirst + p.nb - 1, p.rwork, p.grid) - block_owner(pfirst, p.rwork, p.grid) + 1;
  }
  return q;
}
// Segments c0, c0 + step, ... of a row, weighted relative to the row's maximum `mx`: the weighted sum of the lane's
// four partial columns and of the segments' sums.
__device__ __forceinline__ void row_accumulate(const TaParams& p, const RowRef& q, float mx, int c0, int step,
                                               int lane, float4& num, float& den) {
#pragma unroll 4
  for (int c = c0; c < q.nseg; c += step) {
    const float2 ml = *reinterpret_cast<const float2*>(p.ml + ((q.u0 + c) * kRows + q.r) * 2);
    const float4 pv = *reinterpret_cast<const float4*>(p.part + ((q.u0 + c) * kRows + q.r) * kD + lane * 4);
    const float w = (mx == -INFINITY || ml.x == -INFINITY) ? 0.f : exp2f(ml.x - mx);
    den += w * ml.y;
    num.x += w * pv.x;
    num.y += w * pv.y;
    num.z += w * pv.z;
    num.w += w * pv.w;
  }
}
__device__ __forceinline__ void row_store(const TaParams& p, const RowRef& q, int lane, float4 num, float den) {
  const float inv = den > 0.f ? 1.f / den : 0.f;
  const int gi = q.r / p.n, i = q.r % p.n;
  *reinterpret_cast<float4*>(p.out + ((static_cast<size_t>(q.b) * p.n + i) * p.Hq + q.kvh * p.G + gi) * kD + lane * 4) =
      make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv);
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
__global__ void __launch_bounds__(kCombineThreads) tree_attn_combine(TaParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the partial launch has completed and its writes are visible
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long rows = static_cast<long long>(p.B) * p.Hkv * p.R;
  if (p.maxseg <= kWarpRowSegs) {  // a warp per row
    const long long stride = static_cast<long long>(gridDim.x) * kCombineWarps;
    for (long long u = static_cast<long long>(blockIdx.x) * kCombineWarps + warp; u < rows; u += stride) {
      const RowRef q = row_ref(p, u);
      if (q.nseg == 1) continue;  // a whole pair: its one segment wrote the output
      const float mx = warp_max(lane < q.nseg ? p.ml[((q.u0 + lane) * kRows + q.r) * 2] : -INFINITY);
      float den = 0.f;
      float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
      row_accumulate(p, q, mx, 0, 1, lane, num, den);
      row_store(p, q, lane, num, den);
    }
    return;
  }
  __shared__ float s_mx[kCombineWarps], s_den[kCombineWarps];
  __shared__ float4 s_num[kCombineWarps][32];
  for (long long u = blockIdx.x; u < rows; u += gridDim.x) {  // a CTA per row
    const RowRef q = row_ref(p, u);
    if (q.nseg == 1) continue;  // a whole pair: its one segment wrote the output
    float mx = -INFINITY;
    for (int c = threadIdx.x; c < q.nseg; c += kCombineThreads) mx = fmaxf(mx, p.ml[((q.u0 + c) * kRows + q.r) * 2]);
    mx = warp_max(mx);
    if (lane == 0) s_mx[warp] = mx;
    __syncthreads();
    mx = s_mx[0];
#pragma unroll
    for (int w = 1; w < kCombineWarps; ++w) mx = fmaxf(mx, s_mx[w]);
    float den = 0.f;
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    row_accumulate(p, q, mx, warp, kCombineWarps, lane, num, den);
    s_num[warp][lane] = num;
    if (lane == 0) s_den[warp] = den;
    __syncthreads();
    if (warp == 0) {
      float4 a = s_num[0][lane];
      float d = s_den[0];
#pragma unroll
      for (int w = 1; w < kCombineWarps; ++w) {
        const float4 b = s_num[w][lane];
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
        d += s_den[w];
      }
      row_store(p, q, lane, a, d);
    }
    __syncthreads();  // s_mx, s_num and s_den are rewritten for the next row
  }
}

struct TaPlan {
  int nb, grid, maxseg, wpc;
  long long rwork;
  size_t part, ml, bytes;
};
// The partial launch's CTAs (`per_sm` per SM) each take wpc = pairs / CTAs whole (request, key/value head) pairs,
// then an even share of the remaining pairs' blocks of `block` keys (a CTA takes at least one block); maxseg is the
// most CTAs a remaining pair is spread over, found pair by pair.
inline TaPlan ta_plan(int B, int T, int Hkv, int sms, int per_sm = 1, int block = kTcKeys) {
  TaPlan P{};
  const long long pairs = static_cast<long long>(B) * Hkv;
  P.nb = (T + block - 1) / block;
  const long long work = pairs * P.nb;
  const long long g = static_cast<long long>(per_sm) * sms;
  P.grid = static_cast<int>(g < work ? g : work);
  P.wpc = static_cast<int>(pairs / P.grid);
  const long long rest = pairs - static_cast<long long>(P.wpc) * P.grid;
  P.rwork = rest * P.nb;
  P.maxseg = 1;
  for (long long pr = 0; pr < rest; ++pr) {
    const int segs = block_owner((pr + 1) * P.nb - 1, P.rwork, P.grid) - block_owner(pr * P.nb, P.rwork, P.grid) + 1;
    P.maxseg = segs > P.maxseg ? segs : P.maxseg;
  }
  const size_t slots = static_cast<size_t>(pairs) * P.maxseg;
  P.part = align_up(sizeof(WsHeader));  // the status word first
  P.ml = align_up(P.part + sizeof(float) * slots * kRows * kD);
  P.bytes = align_up(P.ml + sizeof(float) * slots * kRows * 2);
  return P;
}

}  // namespace
}  // namespace dt

extern "C" size_t dt_tree_attention_workspace_bytes(int B, int n, int L, int Hq, int Hkv, int d) {
  if (B < 1 || n < 1 || L < 0 || Hq < 1 || Hkv < 1 || d < 1) return 0;
  dt::DeviceInfo di{};
  if (dt::current_device_info(&di) != cudaSuccess) return 0;
  return dt::ta_plan(B, L + n, Hkv, di.sms).bytes;
}

extern "C" dt_status dt_tree_attention(int B, int n, int L, int Hq, int Hkv, int d, const void* q, const void* k,
                                       const void* v, dt_dtype dtype, const uint8_t* mask, float scale, float* out,
                                       void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  using namespace dt;
  if (B < 0 || n < 1 || L < 0 || Hq < 1 || Hkv < 1 || d < 1 || Hq % Hkv != 0) return DT_ERR_INVALID_ARG;
  if (dtype != DT_F32 && dtype != DT_BF16) return DT_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return DT_ERR_INVALID_ARG;
  if (B == 0) return DT_OK;
  const void* ptrs[] = {q, k, v, out, workspace};
  for (const void* x : ptrs)
    if (!x || !aligned16(x)) return DT_ERR_INVALID_ARG;
  if (!mask) return DT_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (dtype != DT_BF16 || d != kD || G * n > kRows || n > kMaxNodes) return DT_ERR_UNSUPPORTED;
  if (static_cast<long long>(L) + n > INT_MAX / 2) return DT_ERR_UNSUPPORTED;
  DeviceInfo di{};
  if (current_device_info(&di) != cudaSuccess) return DT_ERR_CUDA;
  const int T = L + n;
  const TaPlan P = ta_plan(B, T, Hkv, di.sms);
  if (workspace_bytes < P.bytes) return DT_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * Hkv * G * n > INT_MAX || P.maxseg > kMaxChunks) return DT_ERR_UNSUPPORTED;
  TaParams p{};
  p.B = B; p.n = n; p.L = L; p.T = T; p.Hq = Hq; p.Hkv = Hkv; p.G = G; p.R = G * n;
  p.nb = P.nb; p.grid = P.grid; p.maxseg = P.maxseg; p.wpc = P.wpc; p.rwork = P.rwork;
  p.q = static_cast<const unsigned short*>(q);
  p.k = static_cast<const unsigned short*>(k);
  p.v = static_cast<const unsigned short*>(v);
  p.mask = mask;
  p.scale_log2 = scale * 1.4426950408889634f;
  char* ws = static_cast<char*>(workspace);
  p.part = reinterpret_cast<float*>(ws + P.part);
  p.ml = reinterpret_cast<float*>(ws + P.ml);
  p.out = out;
  TaMaps maps{};
  const uint64_t pairs = static_cast<uint64_t>(B) * static_cast<uint64_t>(Hkv);
  if (!encode_bf16_4d(&maps.q, q, kD, static_cast<uint64_t>(Hq), static_cast<uint64_t>(n), static_cast<uint64_t>(B),
                      64, static_cast<uint32_t>(G), static_cast<uint32_t>(n)) ||
      !encode_bf16_3d(&maps.k, k, kD, static_cast<uint64_t>(T), pairs, 64, kTcKeys) ||
      !encode_bf16_3d(&maps.v, v, kD, static_cast<uint64_t>(T), pairs, 64, kTcKeys))
    return DT_ERR_CUDA;
  const void* fa = reinterpret_cast<const void*>(tree_attn_tc);
  if (ensure_dynamic_smem(fa, kTcSmem) != cudaSuccess) return DT_ERR_CUDA;
  tree_attn_tc<<<static_cast<unsigned>(P.grid), kTcThreads, kTcSmem, stream>>>(p, maps,
                                                                               reinterpret_cast<WsHeader*>(ws));
  if (cudaGetLastError() != cudaSuccess) return DT_ERR_CUDA;
  if (P.rwork == 0) return DT_OK;  // every pair whole in one CTA's share: the partial launch wrote every output
  // the rows of pairs split over several CTAs, as a programmatic dependent of the partial launch
  const long long crows = static_cast<long long>(B) * Hkv * p.R, cper = P.maxseg <= kWarpRowSegs ? kCombineWarps : 1;
  const long long cgrid = (crows + cper - 1) / cper, ccap = static_cast<long long>(kCombinePerSm) * di.sms;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(cgrid < ccap ? cgrid : ccap));
  cfg.blockDim = dim3(kCombineThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, tree_attn_combine, p));
}
