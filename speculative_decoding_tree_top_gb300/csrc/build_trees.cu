// dt_build_trees — conditional best-first draft trees (one persistent cooperative launch per round).
//
// Method: blog.captcha.la, "Methodology — deep read" (DDTree's best-first max-priority queue keyed by cumulative
// conditional log-probability; the GRU state is carried along each root-to-node path; the correction is applied to
// the gathered top-M rows only; fixed node budget / max depth; prefix-closed tree + ancestor-only mask);
// gist.science, "Composants Clés" (only the light GRU correction and correction head are recomputed per node).
//
// GB300 design. The pages' builder replays a CUDA graph per node while a host-side heap decides the next pop
// (gist.science, "Constructeur Natif GPU"); here the whole round is one launch with no host round-trip, and all B
// requests advance in lockstep waves:
//   * a wave expands up to k nodes of every request (lookahead: the node that blocks the request's next pop, then
//     the next unexpanded nodes in the order best-first would reach them; the pops themselves stay exact, see
//     request_step), so a round takes a few waves rather than n steps;
//   * phase A (all CTAs): the GRU step of every expansion of the wave as one GEMM, rows = the packed expansions,
//     columns = the r, z, n_in, n_h gate sets of the hidden units: tcgen05 tiles for bf16 weights whose widths are
//     multiples of 64, else mma.sync or CUDA-core tiles;
//   * grid barrier;
//   * phase B1 (spread over all CTAs): for each expansion, the M correction rows of the node's block position dotted
//     with its new hidden state, the restricted log-softmax, the children ranked into the request's state block;
//   * grid barrier (unless every CTA took its own requests' expansions);
//   * phase B2 (the CTA that owns the request): its best-first state comes into shared memory as one bulk copy; one
//     warp pops and picks the next wave's expansions, which join the packed list of the next wave; the state goes
//     back as one bulk copy; a finished request writes its outputs and ancestor mask;
//   * grid barrier; next wave (none when no request added an expansion).
// Every reduction has a fixed order (no floating-point atomics), so the output is bit-identical run to run and
// does not depend on the lookahead width or on where an expansion sits in the packed list.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <mutex>

#include "build_common.cuh"
#include "umma.cuh"

namespace dt {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr uint64_t kCopyBudgetNs = 4000000000ull;
constexpr int kTB = 16;   // requests per GRU tile
constexpr int kTU = 16;   // hidden units per GRU tile
constexpr int kKC = 64;   // K-chunk of the GRU tile
constexpr int kPad = kKC + 1;

// ---- phase A: GRU step of every expansion of the wave (CUDA cores: fp32 weights, or widths that are not
// multiples of the tensor-core tile) ------------------------------------------------------------------------------
__device__ void gru_phase(const Params& p, const Job* jl, int rows, float* smem) {
  float* xs = smem;                  // [kTB][kPad]
  float* ws = smem + kTB * kPad;     // [3][kTU][kPad]
  __shared__ int s_tok[kTB], s_b[kTB], s_ps[kTB], s_xs[kTB];
  const int t = threadIdx.x, lb = t / kTU, lu = t % kTU;
  const int X = p.xslots;
  const int ublocks = (p.H + kTU - 1) / kTU;
  const int rblocks = (rows + kTB - 1) / kTB;
  const int tiles = ublocks * rblocks;
  for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int rb = tile / ublocks, ub = tile % ublocks;
    __syncthreads();
    if (t < kTB) {
      const int r = rb * kTB + t;
      const bool ok = r < rows;
      s_tok[t] = ok ? jl[r].token : -1;
      s_b[t] = ok ? jl[r].b : 0;
      s_ps[t] = ok ? jl[r].pslot : 0;
      s_xs[t] = ok ? jl[r].xslot : 0;
    }
    __syncthreads();
    const int r = rb * kTB + lb, k = ub * kTU + lu;
    float acc_r = 0.f, acc_u = 0.f, acc_ni = 0.f, acc_nh = 0.f;
    // input side: W_ih[gate rows] . emb[token]
    for (int e0 = 0; e0 < p.E; e0 += kKC) {
      for (int i = t; i < kTB * kKC; i += kThreads) {
        const int q = i / kKC, c = i % kKC, e = e0 + c;
        xs[q * kPad + c] = (s_tok[q] >= 0 && e < p.E) ? ldw(p.emb, p.bf16, static_cast<size_t>(s_tok[q]) * p.E + e) : 0.f;
      }
      for (int i = t; i < 3 * kTU * kKC; i += kThreads) {
        const int g = i / (kTU * kKC), u = (i / kKC) % kTU, c = i % kKC, e = e0 + c, kk = ub * kTU + u;
        ws[(g * kTU + u) * kPad + c] =
            (kk < p.H && e < p.E) ? ldw(p.w_ih, p.bf16, (static_cast<size_t>(g) * p.H + kk) * p.E + e) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int c = 0; c < kKC; ++c) {
        const float x = xs[lb * kPad + c];
        acc_r = fmaf(ws[(0 * kTU + lu) * kPad + c], x, acc_r);
        acc_u = fmaf(ws[(1 * kTU + lu) * kPad + c], x, acc_u);
        acc_ni = fmaf(ws[(2 * kTU + lu) * kPad + c], x, acc_ni);
      }
      __syncthreads();
    }
    // hidden side: W_hh[gate rows] . h_parent
    for (int j0 = 0; j0 < p.H; j0 += kKC) {
      for (int i = t; i < kTB * kKC; i += kThreads) {
        const int q = i / kKC, c = i % kKC, j = j0 + c;
        xs[q * kPad + c] = (s_tok[q] >= 0 && j < p.H)
                               ? __ldcg(p.hs + (static_cast<size_t>(s_b[q]) * X + s_ps[q]) * p.H + j) : 0.f;
      }
      for (int i = t; i < 3 * kTU * kKC; i += kThreads) {
        const int g = i / (kTU * kKC), u = (i / kKC) % kTU, c = i % kKC, j = j0 + c, kk = ub * kTU + u;
        ws[(g * kTU + u) * kPad + c] =
            (kk < p.H && j < p.H) ? ldw(p.w_hh, p.bf16, (static_cast<size_t>(g) * p.H + kk) * p.H + j) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int c = 0; c < kKC; ++c) {
        const float x = xs[lb * kPad + c];
        acc_r = fmaf(ws[(0 * kTU + lu) * kPad + c], x, acc_r);
        acc_u = fmaf(ws[(1 * kTU + lu) * kPad + c], x, acc_u);
        acc_nh = fmaf(ws[(2 * kTU + lu) * kPad + c], x, acc_nh);
      }
      __syncthreads();
    }
    if (r < rows && k < p.H) {
      const size_t g0 = k, g1 = static_cast<size_t>(p.H) + k, g2 = 2 * static_cast<size_t>(p.H) + k;
      const float bir = p.b_ih ? ldw(p.b_ih, p.bf16, g0) : 0.f, bhr = p.b_hh ? ldw(p.b_hh, p.bf16, g0) : 0.f;
      const float biu = p.b_ih ? ldw(p.b_ih, p.bf16, g1) : 0.f, bhu = p.b_hh ? ldw(p.b_hh, p.bf16, g1) : 0.f;
      const float bin = p.b_ih ? ldw(p.b_ih, p.bf16, g2) : 0.f, bhn = p.b_hh ? ldw(p.b_hh, p.bf16, g2) : 0.f;
      const float rg = sigmoidf_(acc_r + bir + bhr);
      const float u = sigmoidf_(acc_u + biu + bhu);
      const float g = tanhf((acc_ni + bin) + rg * (acc_nh + bhn));
      const size_t b = s_b[lb];
      const float hprev = __ldcg(p.hs + (b * X + s_ps[lb]) * p.H + k);
      p.hs[(b * X + s_xs[lb]) * p.H + k] = (1.f - u) * g + u * hprev;
    }
  }
}

// ---- phase A on the tensor cores: one GEMM per step over all expanding requests ---------------------------------
// For a tile of kRT requests x kUT hidden units the CTA computes four gate column sets per unit: r and z over
// K = E (embedding row) + H (parent state), the n gate's input side over E and its hidden side over H, which the GRU
// keeps apart (n = tanh(W_in x + b_in + r * (W_hn h + b_hn))). mma.sync m16n8k16 with bf16 operands and fp32
// accumulators: A = the requests' inputs, B = the weight rows; the fp32 parent state enters as a bf16 hi + lo pair
// (exact to 2^-16 relative). The per-step GEMM is small (B x (E + H) x 3H) and L2-bound, so the layout is chosen
// for latency: K chunks of kKc columns stream from L2 through a deep cp.async ring, and inside a chunk each warp
// takes its own k16 step for the whole tile, so a warp has kMT x (3 kUT / 8) independent accumulators in flight
// rather than one dependent chain; the eight partial tiles are summed in a fixed order in the epilogue.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lds32(const void* q) { return *static_cast<const uint32_t*>(q); }

__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
  const __nv_bfloat16 l0 = __float2bfloat16_rn(x0 - __bfloat162float(h0));
  const __nv_bfloat16 l1 = __float2bfloat16_rn(x1 - __bfloat162float(h1));
  hi = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
  lo = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// Asks L2 to fetch [src, src + bytes) (bytes a multiple of 16, src 16-byte aligned); completes on its own.
__device__ __forceinline__ void prefetch_l2(const void* src, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

template <int kRT, int kUT, int kKcT, int kStagesT>
struct GemmTile {
  static constexpr int kCols = 4 * kUT;   // r | z | n_in | n_h, kUT units each
  static constexpr int kKc = kKcT;        // K columns per pipeline stage
  static constexpr int kSteps = kKc / 16 / kWarps;  // k16 steps of each warp in every chunk
  static constexpr int kXS = kKc + 8;     // shared row stride of a bf16 chunk (elements): conflict-free fragments
  static constexpr int kHS = kKc + 8;     // shared row stride of an fp32 chunk (elements): conflict-free per half-warp
  static constexpr int kMT = kRT / 16;    // m16 tiles
  static constexpr int kNS = kUT / 8;     // n8 tiles per gate column set
  static constexpr int kNT = 4 * kNS;     // n8 tiles of the whole tile
  static constexpr int kXBytes = kRT * kHS * 4;  // the fp32 hidden-side chunk is the larger of the two inputs
  static constexpr int kWBytes = kCols * kXS * 2;
  static constexpr int kStage = kXBytes + kWBytes;
  static constexpr int kStages = kStagesT;
  static constexpr int kRS = kCols + 8;   // row stride of a warp's partial tile (floats): conflict-free float2 stores
  static constexpr int kRedBytes = kWarps * kRT * kRS * 4;
  static constexpr int kRing = kStages * kStage > kRedBytes ? kStages * kStage : kRedBytes;
  static constexpr int kInfo = kRT * 4 * 4;  // token, parent, expand per request (+ pad)
  static constexpr size_t kBytes = static_cast<size_t>(kRing) + kInfo;
  static_assert(kUT % 8 == 0 && kRT % 16 == 0, "whole mma tiles");
  static_assert(kSteps >= 1 && kSteps * 16 * kWarps == kKc, "whole k16 steps per warp per chunk");

};

// Tile shapes: 32 requests x 8 units with K chunks of 256 (B < 128; chunks of 128 through a deeper ring when the
// widths are not multiples of 256), 64 x 16 with chunks of 128 (B >= 128).
using TileS = GemmTile<32, 8, 256, 4>;
using TileS128 = GemmTile<32, 8, 128, 7>;
using TileL = GemmTile<64, 16, 128, 4>;

// Operand chunks of kKc columns stream from L2 through a ring of kStages shared-memory stages filled by 16-byte
// cp.async (one cp.async group per chunk). (Bulk copies of the 256- to 1024-byte row pieces measured 2x slower here:
// each chunk is ~56 small copies.)
template <typename GT, int kRT, int kUT>
__device__ void gemm_gru_phase(const Params& p, const Job* jl, int rows, unsigned char* smem) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int E = p.E, H = p.H, X = p.xslots;
  float* red = reinterpret_cast<float*>(smem);                // [kWarps][kRT][kRS], after the main loop
  int* info = reinterpret_cast<int*>(smem + GT::kRing);        // [kRT][4]: token (-1: no row), request, parent slot, slot
  const int rtiles = (rows + kRT - 1) / kRT, utiles = (H + kUT - 1) / kUT;
  const int nin = E / GT::kKc, nc = nin + H / GT::kKc;  // chunks: input side, then hidden side
  for (int tile = blockIdx.x; tile < rtiles * utiles; tile += gridDim.x) {
    const int b0 = (tile / utiles) * kRT, u0 = (tile % utiles) * kUT;
    __syncthreads();  // the previous tile is done with the shared buffers
    for (int r = t; r < kRT; r += kThreads) {
      const int row = b0 + r;
      const bool ok = row < rows;
      info[4 * r] = ok ? jl[row].token : -1;
      info[4 * r + 1] = ok ? jl[row].b : 0;
      info[4 * r + 2] = ok ? jl[row].pslot : 0;
      info[4 * r + 3] = ok ? jl[row].xslot : 0;
    }
    __syncthreads();

    auto issue = [&](int c) {  // chunk c -> stage c % kStages
      unsigned char* st = smem + (c % GT::kStages) * GT::kStage;
      const bool in = c < nin;
      const int k0 = (in ? c : c - nin) * GT::kKc;
      // weights: the 3 column sets of this side, kUT rows each (the other side's n set is not touched)
      const unsigned short* wsrc = static_cast<const unsigned short*>(in ? p.w_ih : p.w_hh);
      const int K = in ? E : H;
      unsigned short* wdst = reinterpret_cast<unsigned short*>(st + GT::kXBytes);
      for (int i = t; i < 3 * kUT * (GT::kKc / 8); i += kThreads) {
        const int row = i / (GT::kKc / 8), piece = i % (GT::kKc / 8);
        const int gate = row / kUT, uu = row % kUT, u = u0 + uu;
        const int set = (gate == 2 && !in) ? 3 : gate;
        cp_async16(wdst + (set * kUT + uu) * GT::kXS + piece * 8,
                   wsrc + (static_cast<size_t>(gate) * H + u) * K + k0 + piece * 8);
      }
      if (in) {  // the requests' embedding rows, bf16
        unsigned short* xdst = reinterpret_cast<unsigned short*>(st);
        for (int i = t; i < kRT * (GT::kKc / 8); i += kThreads) {
          const int r = i / (GT::kKc / 8), piece = i % (GT::kKc / 8);
          if (info[4 * r] >= 0)
            cp_async16(xdst + r * GT::kXS + piece * 8,
                       static_cast<const unsigned short*>(p.emb) + static_cast<size_t>(info[4 * r]) * E + k0 +
                           piece * 8);
        }
      } else {  // the parents' hidden states, fp32
        float* xdst = reinterpret_cast<float*>(st);
        for (int i = t; i < kRT * (GT::kKc / 4); i += kThreads) {
          const int r = i / (GT::kKc / 4), piece = i % (GT::kKc / 4);
          if (info[4 * r] >= 0) {
            const float* src = p.hs + (static_cast<size_t>(info[4 * r + 1]) * X + info[4 * r + 2]) * H;
            cp_async16(xdst + r * GT::kHS + piece * 4, src + k0 + piece * 4);
          }
        }
      }
      cp_async_commit();
    };
    auto issue_or_empty = [&](int c) {  // every thread commits one group per call, so the counts stay uniform
      if (c < nc) issue(c);
      else cp_async_commit();
    };

    float acc[GT::kMT][GT::kNT][4];
#pragma unroll
    for (int a = 0; a < GT::kMT; ++a)
#pragma unroll
      for (int b = 0; b < GT::kNT; ++b)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[a][b][q] = 0.f;

    for (int c = 0; c < GT::kStages - 1; ++c) issue_or_empty(c);
    for (int c = 0; c < nc; ++c) {
      asm volatile("cp.async.wait_group %0;" ::"n"(GT::kStages - 2) : "memory");  // chunk c has landed
      __syncthreads();  // ... for every thread; and everyone is done with chunk c - 1, whose stage is reused next
      issue_or_empty(c + GT::kStages - 1);
      const bool in = c < nin;
      const unsigned char* st = smem + (c % GT::kStages) * GT::kStage;
      const unsigned short* wsm = reinterpret_cast<const unsigned short*>(st + GT::kXBytes);
#pragma unroll
      for (int j = 0; j < GT::kSteps; ++j) {
        const int k = (j * kWarps + warp) * 16 + tig * 2;  // this warp's j-th k16 step inside the chunk
        // column sets: r, z on both sides; n_in (set 2) only on the input side, n_h (set 3) only on the hidden side
        uint32_t bfr[GT::kNT][2];
#pragma unroll
        for (int nt = 0; nt < GT::kNT; ++nt) {
          const int col = nt * 8 + g;
          bfr[nt][0] = lds32(wsm + col * GT::kXS + k);
          bfr[nt][1] = lds32(wsm + col * GT::kXS + k + 8);
        }
        if (in) {
          const unsigned short* xsm = reinterpret_cast<const unsigned short*>(st);
#pragma unroll
          for (int mt = 0; mt < GT::kMT; ++mt) {
            const int r0 = mt * 16 + g;
            const uint32_t a0 = lds32(xsm + r0 * GT::kXS + k), a1 = lds32(xsm + (r0 + 8) * GT::kXS + k);
            const uint32_t a2 = lds32(xsm + r0 * GT::kXS + k + 8), a3 = lds32(xsm + (r0 + 8) * GT::kXS + k + 8);
#pragma unroll
            for (int nt = 0; nt < 3 * GT::kNS; ++nt)
              mma_bf16_16816(acc[mt][nt], a0, a1, a2, a3, bfr[nt][0], bfr[nt][1]);
          }
        } else {
          const float* xsm = reinterpret_cast<const float*>(st);
#pragma unroll
          for (int mt = 0; mt < GT::kMT; ++mt) {
            const int r0 = mt * 16 + g;
            const float2 p0 = *reinterpret_cast<const float2*>(xsm + r0 * GT::kHS + k);
            const float2 p1 = *reinterpret_cast<const float2*>(xsm + (r0 + 8) * GT::kHS + k);
            const float2 p2 = *reinterpret_cast<const float2*>(xsm + r0 * GT::kHS + k + 8);
            const float2 p3 = *reinterpret_cast<const float2*>(xsm + (r0 + 8) * GT::kHS + k + 8);
            uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
            split_bf16x2(p0.x, p0.y, h0, l0);
            split_bf16x2(p1.x, p1.y, h1, l1);
            split_bf16x2(p2.x, p2.y, h2, l2);
            split_bf16x2(p3.x, p3.y, h3, l3);
#pragma unroll
            for (int nt = 0; nt < GT::kNT; ++nt) {
              if (nt / GT::kNS == 2) continue;  // n_in has no hidden side
              mma_bf16_16816(acc[mt][nt], h0, h1, h2, h3, bfr[nt][0], bfr[nt][1]);
              mma_bf16_16816(acc[mt][nt], l0, l1, l2, l3, bfr[nt][0], bfr[nt][1]);
            }
          }
        }
      }
    }
    cp_async_wait_all();
    __syncthreads();  // the ring is free (every chunk consumed): it now holds the warps' partial tiles
    // partial tile of this warp -> red[warp]: thread holds rows g, g + 8 and columns tig*2, tig*2 + 1 of each tile
#pragma unroll
    for (int mt = 0; mt < GT::kMT; ++mt)
#pragma unroll
      for (int nt = 0; nt < GT::kNT; ++nt) {
        const int r0 = mt * 16 + g, c0 = nt * 8 + tig * 2;
        float* q = red + (warp * kRT + r0) * GT::kRS + c0;
        *reinterpret_cast<float2*>(q) = make_float2(acc[mt][nt][0], acc[mt][nt][1]);
        *reinterpret_cast<float2*>(q + 8 * GT::kRS) = make_float2(acc[mt][nt][2], acc[mt][nt][3]);
      }
    __syncthreads();
    for (int i = t; i < kRT * kUT; i += kThreads) {  // the GRU pointwise, one (request, unit) per thread
      const int r = i / kUT, uu = i % kUT, u = u0 + uu;
      if (u >= H || info[4 * r] < 0) continue;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {  // fixed order: bit-identical run to run
        const float* q = red + (w * kRT + r) * GT::kRS + uu;
#pragma unroll
        for (int set = 0; set < 4; ++set) d[set] += q[set * kUT];
      }
      const size_t g0 = u, g1 = static_cast<size_t>(H) + u, g2 = 2 * static_cast<size_t>(H) + u;
      const float bir = p.b_ih ? ldw(p.b_ih, true, g0) : 0.f, bhr = p.b_hh ? ldw(p.b_hh, true, g0) : 0.f;
      const float biz = p.b_ih ? ldw(p.b_ih, true, g1) : 0.f, bhz = p.b_hh ? ldw(p.b_hh, true, g1) : 0.f;
      const float bin = p.b_ih ? ldw(p.b_ih, true, g2) : 0.f, bhn = p.b_hh ? ldw(p.b_hh, true, g2) : 0.f;
      const float rg = sigmoidf_(d[0] + bir + bhr);
      const float zg = sigmoidf_(d[1] + biz + bhz);
      const float ng = tanhf(d[2] + bin + rg * (d[3] + bhn));
      const size_t b = static_cast<size_t>(info[4 * r + 1]);
      const float hprev = __ldcg(p.hs + (b * X + info[4 * r + 2]) * H + u);
      p.hs[(b * X + info[4 * r + 3]) * H + u] = (1.f - zg) * ng + zg * hprev;
    }
  }
}

// ---- phases B1 / B2: shared memory --------------------------------------------------------------------------------
// The children phase holds, per expansion, [H] hidden state, [M4] logits, [M4] base logits, [M4] ids, [M] sibling
// keys, [M] children, then (when it fits) the M gathered W_c rows; the control phase holds one request's state block.
__host__ __device__ inline int round4(int x) { return (x + 3) & ~3; }
struct FrontierSmem {
  size_t h, z, vals, ids, keys, kraw, rows, bytes;
};
__host__ __device__ inline FrontierSmem frontier_smem(size_t state_bytes, int M, int H) {
  FrontierSmem F{};
  size_t o = (state_bytes + 15) / 16 * 16;
  auto take = [&o](size_t bytes) {
    const size_t at = o;
    o = (o + bytes + 15) / 16 * 16;
    return at;
  };
  F.h = take(sizeof(float) * H);
  F.z = take(sizeof(float) * round4(M));
  F.vals = take(sizeof(float) * round4(M));
  F.ids = take(sizeof(int) * round4(M));
  F.keys = take(sizeof(unsigned long long) * M);
  F.kraw = take(sizeof(Node) * M);
  F.rows = o;
  F.bytes = o;
  return F;
}
constexpr size_t kFrontierRowsCap = 160 * 1024;  // gathered rows kept in shared memory up to this size

// The children phase by groups (one request's expansions at one block position, group_mma): the J <= kLargeLookahead
// hidden states [8][H] fp32, the position's ids and base logits, the M gathered correction rows [M][H + 8] bf16 (the
// row stride padded by 16 bytes, so the MMA's row fragments fall in distinct banks), the corrected logits [8][M], and
// per expansion its children [8][M] and their sibling keys [8][M].
struct GroupSmem {
  size_t bfrag, h, ids, vals, rows, z, zpart, kraw, keys, jobs, ctl, bytes;
};
__host__ __device__ inline GroupSmem group_smem(int M, int H) {
  GroupSmem L{};
  size_t o = 0;
  auto take = [&o](size_t bytes) {
    const size_t at = o;
    o = (o + bytes + 15) / 16 * 16;
    return at;
  };
  L.bfrag = take(sizeof(uint4) * 2 * static_cast<size_t>(H));  // [H / 16 k16 steps][32 lanes]
  L.h = take(sizeof(float) * kLargeLookahead * H);
  L.ids = take(sizeof(int) * 2 * round4(M));
  L.vals = take(sizeof(float) * 2 * round4(M));
  L.rows = take(sizeof(unsigned short) * static_cast<size_t>(M) * (H + 8));
  L.z = take(sizeof(float) * kLargeLookahead * round4(M));
  L.zpart = take(sizeof(float) * kWarps * kLargeLookahead * 16);  // one 16 x 8 partial tile per warp
  L.kraw = take(sizeof(Node) * kLargeLookahead * M);
  L.keys = take(sizeof(unsigned long long) * kLargeLookahead * M);
  L.jobs = take(sizeof(Job) * 3 * kLargeLookahead);
  L.ctl = take(sizeof(ReqCtl) * 3);
  L.bytes = o;
  return L;
}

__device__ __forceinline__ void bulk_s2g(void* gdst, const void* ssrc, unsigned bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
}

// ---- the first children group of a CTA, loaded while the wave's GRU runs -------------------------------------------
// During the tensor-core GRU phase warps 2 and 3 have no role; warp 2 loads this CTA's first group of the wave (its
// entry, ids and base logits, jobs and the request's control word) into a static shared buffer and asks L2 for the
// group's correction rows, so that the children phase starts on its row copies at once.
struct GroupPrefetch {
  int valid, ngroups;
  JobGroup gr;
  ReqCtl ctl;
  Job jobs[kLargeLookahead];
  int ids[128];
  float vals[128];
};
__device__ void prefetch_first_group(const Params& p, int w, const Job* jl, GroupPrefetch* pf) {
  const int lane = threadIdx.x & 31;
  const int M = p.M, n = p.n, KM = M < n ? M : n;
  const JobGroup* gl = p.grouplist + static_cast<size_t>(w & 1) * p.B * p.lookahead;
  JobGroup gr{};
  if (static_cast<int>(blockIdx.x) < p.B * p.lookahead) gr = gl[blockIdx.x];
  const int ng = __ldcg(p.groupcount + w);
  if (static_cast<int>(blockIdx.x) >= ng || M > 128) return;  // valid stays 0
  const size_t pos = (static_cast<size_t>(gr.b) * p.K + gr.depth) * M;
  const size_t rb = static_cast<size_t>(p.H) * 2;
  for (int m = lane; m < M; m += 32) {
    const int id = valid_id(p, __ldg(p.ids + pos + m));
    pf->ids[m] = id;
    pf->vals[m] = __ldg(p.vals + pos + m);
    const char* row = static_cast<const char*>(p.w_c) + static_cast<size_t>(id) * rb;  // its row, asked of L2
    for (size_t c = 0; c < rb; c += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + c));
  }
  if (lane < gr.count) pf->jobs[lane] = jl[gr.start + lane];
  if (lane == 0) {
    const ReqLayout RL = req_layout(n, p.xslots, KM, p.lookahead);
    pf->ctl = *reinterpret_cast<const ReqCtl*>(p.rstate + static_cast<size_t>(gr.b) * RL.bytes + RL.ctl);
    pf->gr = gr;
    pf->ngroups = ng;
  }
  __syncwarp();
  if (lane == 0) pf->valid = 1;
}

// ---- phase A on the 5th-generation tensor cores (tcgen05, TMEM, 2-D TMA) ---------------------------------------
// One narrow tile = 128 expansions (rows) x 32 hidden units. The A operand is the packed activations
// [emb | hi(h) | lo(h)] of the wave (bf16, written by the control phase that picked the expansions; hi + lo carry the
// fp32 parent state to 2^-16), the B operand the gate rows [r | z | n_in | n_h] of the tile's units in W_ih / W_hh,
// both K-major, moved by TMA in 64-column blocks with 128-byte swizzle through a 6-stage ring of full / empty
// mbarriers. One lane issues the TMA loads, one lane the MMAs (kind::f16, N = 128, fp32 accumulate in TMEM); each K
// partial (below) has its own 128 columns. All eight warps read the tile back (tcgen05.ld, one row per thread, warps
// w and w + 4 on the same TMEM lanes with half of the units each) and finish the GRU step. Waves of whole tiles run
// on wide tiles instead (umma_gru_wide).
struct TmaMaps {
  CUtensorMap x;      // [rows cap][E + 2H] bf16, box 64 x 128
  CUtensorMap wih;    // [3H][E] bf16, box 64 x 32
  CUtensorMap whh;    // [3H][H] bf16, box 64 x 32
  CUtensorMap wih64;  // the same weights in boxes of 64 x 64 (wide tiles)
  CUtensorMap whh64;
};
constexpr int kUmmaRows = 128, kUmmaUnits = 32, kUmmaBK = 64, kUmmaStages = 6;
constexpr int kUmmaA = kUmmaRows * kUmmaBK * 2;            // 16 KB
// The B tile of a K block: the weight rows of the gate columns [r | z | n_in | n_h] of the tile's units, the set a
// block does not touch (n_h for an embedding block, n_in for a hidden one) read as zeros, so that one MMA of N = 128
// covers the block: the zeros add exact zeros to the other gate's sums.
constexpr int kUmmaB = 4 * kUmmaUnits * kUmmaBK * 2;       // 16 KB
constexpr int kUmmaStage = kUmmaA + kUmmaB;                // 32 KB (a multiple of 1024)
constexpr size_t kUmmaSmem = static_cast<size_t>(kUmmaStages) * kUmmaStage + 1024;  // + alignment slack
constexpr int kTmemCols = 512;  // kSplits partials of 128 columns
// Wide tiles (128 expansions x 64 units, N = 256) for waves of whole tiles: half the activation reads of two narrow
// tiles. A 4-stage ring of 48 KB stages in the same shared memory; two TMEM regions of 256 columns.
constexpr int kWideUnits = 64, kWideStages = 4;
constexpr int kWideB = 4 * kWideUnits * kUmmaBK * 2;  // 32 KB
constexpr int kWideStage = kUmmaA + kWideB;           // 48 KB
static_assert(kWideStages * kWideStage <= kUmmaStages * kUmmaStage, "the wide ring fits the narrow one's memory");

// Per-launch state of the tensor-core phase: the ring's barriers and how far each has gone (the same in every thread).
struct UmmaRing {
  uint64_t* full;    // [kUmmaStages]
  uint64_t* empty;   // [kUmmaStages]
  uint64_t* done;    // accumulator complete
  uint64_t* wfull;   // [kWideStages] the wide ring's
  uint64_t* wempty;  // [kWideStages]
  uint64_t* mid;     // wide tiles: partial 1, then partial 2, complete in TMEM
  uint64_t* r1free;  // wide tiles: the epilogue warps folded it into region 0 (4 arrivals)
  uint32_t tmem;
  unsigned blocks;   // K blocks loaded so far (ring position)
  unsigned wblocks;  // ... through the wide ring
  unsigned tiles;    // tiles finished so far (done phase)
};

// The GRU pointwise of U consecutive units u .. u + U - 1 of one expansion from its gate sums d[r | z | n_in | n_h][U].
template <int U>
__device__ __forceinline__ void gru_pointwise(const Params& p, const Job& jb, int u, const float (&d)[4][U], int X, int H) {
  const float* hprev = p.hs + (static_cast<size_t>(jb.b) * X + jb.pslot) * H + u;
  float* hout = p.hs + (static_cast<size_t>(jb.b) * X + jb.xslot) * H + u;
#pragma unroll
  for (int j = 0; j < U; ++j) {
    const size_t g0 = u + j, g1 = static_cast<size_t>(H) + g0, g2 = 2 * static_cast<size_t>(H) + g0;
    const float bir = p.b_ih ? ldw(p.b_ih, true, g0) : 0.f, bhr = p.b_hh ? ldw(p.b_hh, true, g0) : 0.f;
    const float biz = p.b_ih ? ldw(p.b_ih, true, g1) : 0.f, bhz = p.b_hh ? ldw(p.b_hh, true, g1) : 0.f;
    const float bin = p.b_ih ? ldw(p.b_ih, true, g2) : 0.f, bhn = p.b_hh ? ldw(p.b_hh, true, g2) : 0.f;
    const float rg = sigmoidf_(d[0][j] + bir + bhr);
    const float zg = sigmoidf_(d[1][j] + biz + bhz);
    const float ng = tanhf(d[2][j] + bin + rg * (d[3][j] + bhn));
    hout[j] = (1.f - zg) * ng + zg * __ldcg(hprev + j);
  }
}

// The K range of the step is summed as kSplits partials in a fixed order, whoever computes them. A wave with enough
// tiles gives each tile to one CTA, which holds all the partials in separate TMEM regions. A smaller wave gives each
// CTA `per` consecutive partials of a tile (per = 1 or 2, so that kSplits / per CTAs share it and every CTA of the
// phase has at most one). Those CTAs store their partials in the workspace, wait (bounded) for one another, and each
// then adds up all kSplits partials for its share of the tile's units. Both ways give the same bits, so the result
// of an expansion does not depend on how many share its wave.
constexpr int kSplits = kGruSplits;
static_assert(kUmmaRows == kGruTileRows && kUmmaUnits == kGruTileUnits, "workspace tiles are the MMA tiles");
__device__ __forceinline__ int split_begin(int s, int nkb) { return s * nkb / kSplits; }

// The split tile's CTAs meet, then each adds up the kSplits partials of rows [row0, row0 + 128) x units
// [u0 + uoff, + 2 U) from the workspace and runs the GRU pointwise; thread t takes row t % 128 and U units from
// uoff + U (t / 128). The pointwise's other inputs (the row's job, its parent state, the biases) are loaded before
// `epilogue` (which stores this CTA's partials) runs, so that their latency hides behind it, and all of a thread's
// partials at once after the meeting. Returns false when the epilogue or the meeting ran out of time.
template <int U, class Epilogue>  // U a multiple of 4
__device__ bool split_meet_reduce(const Params& p, const Job* jl, int rows, const float* part, int row0, int u0,
                                  int uoff, int X, int H, unsigned* ticket, int cpt, bool ok, int* s_ok,
                                  const Epilogue& epilogue) {
  const int t = threadIdx.x, r = t & (kUmmaRows - 1), q = row0 + r, c = uoff + U * (t / kUmmaRows);
  const bool mine = q < rows;
  Job jb{};
  float hp[U], bias[6][U];
  if (mine) {
    jb = jl[q];
    const float* hprev = p.hs + (static_cast<size_t>(jb.b) * X + jb.pslot) * H + u0 + c;
#pragma unroll
    for (int j = 0; j < U; ++j) {
      hp[j] = __ldcg(hprev + j);
#pragma unroll
      for (int g = 0; g < 3; ++g) {
        const size_t gi = static_cast<size_t>(g) * H + u0 + c + j;
        bias[g][j] = p.b_ih ? ldw(p.b_ih, true, gi) : 0.f;
        bias[3 + g][j] = p.b_hh ? ldw(p.b_hh, true, gi) : 0.f;
      }
    }
  }
  ok = epilogue(ok);
  // thread 0's release after the CTA barrier publishes every thread's partials; its acquire before the next barrier
  // orders every thread's reads of the others'
  ok = __syncthreads_and(ok);
  if (t == 0) {
    bool met = ok;
    if (met) {
      atom_add_acq_rel_gpu(ticket, 1u);
      const uint64_t t0 = global_timer_ns();
      while (ld_acquire_gpu(ticket) < static_cast<unsigned>(cpt)) {  // the others run now: one unit per CTA
        if (global_timer_ns() - t0 > kCopyBudgetNs || ld_acquire_gpu(&p.hdr->abort) != 0u) {
          met = false;
          break;
        }
      }
    }
    *s_ok = met;
  }
  __syncthreads();
  if (*s_ok == 0) return false;
  if (!mine) return true;
  float* hout = p.hs + (static_cast<size_t>(jb.b) * X + jb.xslot) * H + u0 + c;
#pragma unroll
  for (int j0 = 0; j0 < U; j0 += 4) {  // four units at a time: their 4 x 4 x kSplits partials loaded together
    float v[kSplits][4][4];
#pragma unroll
    for (int sp = 0; sp < kSplits; ++sp)
#pragma unroll
      for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          v[sp][g][j] = __ldcg(part + static_cast<size_t>(sp) * kUmmaRows * 128 +
                               static_cast<size_t>(g * kUmmaUnits + c + j0 + j) * kUmmaRows + r);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float d[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        d[g] = 0.f;
#pragma unroll
        for (int sp = 0; sp < kSplits; ++sp) d[g] += v[sp][g][j];  // partials in order 0 .. kSplits - 1
      }
      const int u = j0 + j;
      const float rg = sigmoidf_(d[0] + bias[0][u] + bias[3][u]);
      const float zg = sigmoidf_(d[1] + bias[1][u] + bias[4][u]);
      const float ng = tanhf(d[2] + bias[2][u] + rg * (d[3] + bias[5][u]));
      hout[u] = (1.f - zg) * ng + zg * hp[u];
    }
  }
  return true;
}

__device__ __forceinline__ void tmem_st4x8(uint32_t taddr, const float (&v)[4][8]) {  // 32 columns from taddr
#pragma unroll
  for (int g = 0; g < 4; ++g)
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 ::"r"(taddr + 8u * g), "r"(__float_as_uint(v[g][0])), "r"(__float_as_uint(v[g][1])),
                 "r"(__float_as_uint(v[g][2])), "r"(__float_as_uint(v[g][3])), "r"(__float_as_uint(v[g][4])),
                 "r"(__float_as_uint(v[g][5])), "r"(__float_as_uint(v[g][6])), "r"(__float_as_uint(v[g][7]))
                 : "memory");
}

// What partial `sp` of nkb K blocks (nE of them embedding blocks) wrote: gate slot g of its accumulator counts only
// when the partial has blocks feeding it (n_in: embedding blocks, n_h: hidden ones, r and z: any).
__device__ __forceinline__ bool partial_feeds(int sp, int g, int nkb, int nE) {
  const int sb = split_begin(sp, nkb), se = split_begin(sp + 1, nkb);
  const bool any = se > sb;
  return g < 2 ? any : g == 2 ? any && sb < nE : any && se > nE;
}

// Waves of whole tiles on wide tiles: tile = 128 expansions x 64 units, B = the four gate slots of the 64 units
// (N = 256). The K partials are still summed in order 0..3, in TMEM: partial 0 into region 0, partials 1..3 one
// after another into region 1; the four epilogue warps fold partials 1 and 2 into region 0 as each completes
// ((0 + p0) + p1, then + p2) while the MMA lane waits to reuse region 1, and the final epilogue adds partial 3.
// The sums and their order are those of the narrow tiles, so the result does not depend on the tile width.
__device__ bool umma_gru_wide(const Params& p, const TmaMaps& maps, const Job* jl, int rows, unsigned char* smem,
                              UmmaRing& ring) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int E = p.E, H = p.H, X = p.xslots;
  const int nE = E / kUmmaBK, nH = H / kUmmaBK, nkb = nE + 2 * nH;
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem) + 1023) & ~uintptr_t(1023));
  const int rtiles = (rows + kUmmaRows - 1) / kUmmaRows, utiles = H / kWideUnits, tiles = rtiles * utiles;
  const int G = static_cast<int>(gridDim.x);
  constexpr uint32_t kR1 = 256;  // region 1's first column
  bool ok = true;
  for (int tile = blockIdx.x; tile < tiles; tile += G) {
    const int row0 = (tile / utiles) * kUmmaRows, u0 = (tile % utiles) * kWideUnits;
    if (warp == 0 && lane == 0) {  // TMA producer
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the other phases' shared-memory use came first
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const unsigned n = ring.wblocks + kb, st = n % kWideStages, use = n / kWideStages;
        if (use > 0) ok = mbar_wait(&ring.wempty[st], (use - 1) & 1u, kCopyBudgetNs);
        if (!ok) break;
        unsigned char* a = base + st * kWideStage;
        unsigned char* bsm = a + kUmmaA;
        mbar_expect_tx(&ring.wfull[st], kWideStage);
        const bool emb = kb < nE;
        const int acol = emb ? kb * kUmmaBK : E + (kb - nE) * kUmmaBK;
        const int wcol = emb ? kb * kUmmaBK : ((kb - nE) % nH) * kUmmaBK;
        tma_load_2d(a, &maps.x, acol, row0, &ring.wfull[st]);
        const CUtensorMap* wm = emb ? &maps.wih64 : &maps.whh64;
        for (int g = 0; g < 4; ++g) {
          const int src = g < 2 ? g : (g == 2) == emb ? 2 : 3;
          tma_load_2d(bsm + g * kWideUnits * 128, wm, wcol, src * H + u0, &ring.wfull[st]);
        }
      }
    } else if (warp == 1 && lane == 0) {  // MMA issuer
      int sp = 0;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        while (sp + 1 < kSplits && kb >= split_begin(sp + 1, nkb)) ++sp;
        const int sb = split_begin(sp, nkb);
        if (kb == sb && sp >= 2) {  // region 1 is reused: wait until partial sp - 1 is folded into region 0
          ok = mbar_wait(ring.r1free, static_cast<unsigned>(sp - 2) & 1u, kCopyBudgetNs);
          if (!ok) break;
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        }
        const unsigned n = ring.wblocks + kb, st = n % kWideStages, use = n / kWideStages;
        ok = mbar_wait(&ring.wfull[st], use & 1u, kCopyBudgetNs);
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t d = ring.tmem + (sp == 0 ? 0u : kR1);
        const uint32_t a = smem_u32(base + st * kWideStage), bsm = a + kUmmaA;
#pragma unroll
        for (int k = 0; k < kUmmaBK / 16; ++k)
          umma_f16(d, umma_desc_sw128(a + 32 * k), umma_desc_sw128(bsm + 32 * k), umma_idesc(4 * kWideUnits),
                   (kb > sb || k > 0) ? 1u : 0u);
        umma_commit(&ring.wempty[st]);
        if ((sp == 1 || sp == 2) && kb + 1 == split_begin(sp + 1, nkb)) umma_commit(ring.mid);
      }
      if (ok) umma_commit(ring.done);
    } else if (warp >= 4) {  // fold partials 1 and 2 into region 0 as each completes
      const uint32_t trow = ring.tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
      for (int f = 0; f < 2 && ok; ++f) {
        ok = mbar_wait(ring.mid, static_cast<unsigned>(f), kCopyBudgetNs);
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        for (int c = 0; c < 4 * kWideUnits; c += 32) {
          const int g = c / kWideUnits;  // the gate slot of these 32 columns
          float a[4][8], b[4][8];
          tmem_ld4x8(trow + c, 8, a);
          tmem_ld4x8(trow + kR1 + c, 8, b);
          const bool fb = partial_feeds(f + 1, g, nkb, nE), fa = f > 0 || partial_feeds(0, g, nkb, nE);
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float pa = fa ? a[i][j] : 0.f, pb = fb ? b[i][j] : 0.f;
              a[i][j] = f == 0 ? (0.f + pa) + pb : pa + pb;
            }
          tmem_st4x8(trow + c, a);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(ring.r1free);
      }
    }
    ring.wblocks += nkb;
    ok = __syncthreads_and(ok);
    if (ok) {  // the last partial added, then the GRU pointwise: one row per thread, warps w and w + 4 half the units
      ok = mbar_wait(ring.done, ring.tiles & 1u, kCopyBudgetNs);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int r = 32 * (warp & 3) + lane, q = row0 + r;
      const uint32_t trow = ring.tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
      Job jb{};
      if (q < rows) jb = jl[q];
      bool f3[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) f3[g] = partial_feeds(3, g, nkb, nE);
      const int c0 = (warp >> 2) * (kWideUnits / 2);
      for (int c = c0; c < c0 + kWideUnits / 2; c += 8) {
        float s3[4][8], p3[4][8];
        tmem_ld4x8(trow + c, kWideUnits, s3);
        tmem_ld4x8(trow + kR1 + c, kWideUnits, p3);
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int j = 0; j < 8; ++j) s3[g][j] += f3[g] ? p3[g][j] : 0.f;
        if (q < rows && ok) gru_pointwise<8>(p, jb, u0 + c, s3, X, H);
      }
    }
    ring.tiles += 1;
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    ok = __syncthreads_and(ok);  // the accumulators are read before the next tile's first MMA overwrites them
    if (!ok) {
      record_error(p.hdr, DT_ERR_TIMEOUT);
      atomicExch(&p.hdr->abort, 1u);
      return false;
    }
  }
  return true;
}

// Returns false when a wait ran out (recorded, abort raised).
__device__ bool umma_gru_phase(const Params& p, const TmaMaps& maps, const Job* jl, int rows, unsigned char* smem,
                               UmmaRing& ring, int w, GroupPrefetch* pf) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int E = p.E, H = p.H, X = p.xslots;
  const int nE = E / kUmmaBK, nH = H / kUmmaBK, nkb = nE + 2 * nH;
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem) + 1023) & ~uintptr_t(1023));
  const int rtiles = (rows + kUmmaRows - 1) / kUmmaRows, utiles = H / kUmmaUnits, tiles = rtiles * utiles;
  const int G = static_cast<int>(gridDim.x);
  if (p.group_mma && warp == 2) prefetch_first_group(p, w, jl, pf);  // a warp with no role in either path
  if (tiles > p.gru_tiles && H % kWideUnits == 0) return umma_gru_wide(p, maps, jl, rows, smem, ring);
  const int per = tiles > p.gru_tiles ? kSplits : tiles * kSplits <= G ? 1 : tiles * (kSplits / 2) <= G ? 2 : kSplits;
  const int cpt = kSplits / per;  // CTAs per tile
  const int units = tiles * cpt;
  __shared__ int s_ok;
  bool ok = true;
  for (int unit = blockIdx.x; unit < units; unit += G) {
    const int tile = unit / cpt, part_idx = unit % cpt;
    const int s_lo = part_idx * per, s_hi = s_lo + per;
    const int row0 = (tile / utiles) * kUmmaRows, u0 = (tile % utiles) * kUmmaUnits;
    const int kb_lo = split_begin(s_lo, nkb), kb_hi = split_begin(s_hi, nkb);
    if (warp == 0 && lane == 0) {  // TMA producer
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the other phases' shared-memory use came first
      for (int kb = kb_lo; kb < kb_hi && ok; ++kb) {
        const unsigned n = ring.blocks + (kb - kb_lo), st = n % kUmmaStages, use = n / kUmmaStages;
        if (use > 0) ok = mbar_wait(&ring.empty[st], (use - 1) & 1u, kCopyBudgetNs);
        if (!ok) break;
        unsigned char* a = base + st * kUmmaStage;
        unsigned char* bsm = a + kUmmaA;
        mbar_expect_tx(&ring.full[st], kUmmaStage);
        const bool emb = kb < nE;
        const int acol = emb ? kb * kUmmaBK : E + (kb - nE) * kUmmaBK;                   // hi blocks, then lo blocks
        const int wcol = emb ? kb * kUmmaBK : ((kb - nE) % nH) * kUmmaBK;
        tma_load_2d(a, &maps.x, acol, row0, &ring.full[st]);
        // gate slot g of the tile takes weight rows g H + u0 (r, z, and n_in or n_h); the block's unused slot reads
        // rows 3 H .. past the weights' end: zeros
        const CUtensorMap* wm = emb ? &maps.wih : &maps.whh;
        for (int g = 0; g < 4; ++g) {
          const int src = g < 2 ? g : (g == 2) == emb ? 2 : 3;
          tma_load_2d(bsm + g * kUmmaUnits * 128, wm, wcol, src * H + u0, &ring.full[st]);
        }
      }
    } else if (warp == 1 && lane == 0) {  // MMA issuer: partial s into TMEM columns [128 (s - s_lo), +128)
      for (int kb = kb_lo; kb < kb_hi && ok; ++kb) {
        const unsigned n = ring.blocks + (kb - kb_lo), st = n % kUmmaStages, use = n / kUmmaStages;
        ok = mbar_wait(&ring.full[st], use & 1u, kCopyBudgetNs);
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        int sp = s_lo;  // the partial this block belongs to
        while (sp + 1 < s_hi && kb >= split_begin(sp + 1, nkb)) ++sp;
        const int sb = split_begin(sp, nkb);  // its first block
        const uint32_t d = ring.tmem + 128u * static_cast<uint32_t>(sp - s_lo);
        const uint32_t a = smem_u32(base + st * kUmmaStage), bsm = a + kUmmaA;
#pragma unroll
        for (int k = 0; k < kUmmaBK / 16; ++k)
          umma_f16(d, umma_desc_sw128(a + 32 * k), umma_desc_sw128(bsm + 32 * k), umma_idesc(4 * kUmmaUnits),
                   (kb > sb || k > 0) ? 1u : 0u);
        umma_commit(&ring.empty[st]);  // the stage is free once these MMAs have read it
      }
      if (ok) umma_commit(ring.done);  // and the partials are complete after the last block's MMAs
    }
    ring.blocks += kb_hi - kb_lo;
    ok = __syncthreads_and(ok);
    const int r = 32 * (warp & 3) + lane, q = row0 + r;  // the epilogue warps' row (expansion)
    // a tile's partials in the workspace: [split][gate column][row], so that a warp's rows are adjacent words
    float* part = p.gru_part + static_cast<size_t>(tile) * kSplits * kUmmaRows * 128;
    // epilogue: one row per thread, warps w and w + 4 (the same TMEM lanes) half of the units each
    auto epilogue = [&](bool ok) -> bool {
      if (!ok) return false;
      ok = mbar_wait(ring.done, ring.tiles & 1u, kCopyBudgetNs);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t trow = ring.tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
      Job jb{};
      if (q < rows) jb = jl[q];
      const int c0 = (warp >> 2) * (kUmmaUnits / 2);
      for (int c = c0; c < c0 + kUmmaUnits / 2; c += 8) {
        float dsum[4][8];
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int j = 0; j < 8; ++j) dsum[g][j] = 0.f;
        for (int sp = s_lo; sp < s_hi; ++sp) {
          const int sb = split_begin(sp, nkb), se = split_begin(sp + 1, nkb);
          // n_in is written only by embedding blocks, n_h only by hidden ones, nothing by an empty split (K shorter
          // than kSplits blocks): what a partial did not write contributes 0
          const bool has_any = se > sb, has_emb = has_any && sb < nE, has_hid = has_any && se > nE;
          float dv[4][8];
          tmem_ld4x8(trow + 128u * static_cast<uint32_t>(sp - s_lo) + c, kUmmaUnits, dv);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (!has_any) dv[0][j] = dv[1][j] = 0.f;
            if (!has_emb) dv[2][j] = 0.f;
            if (!has_hid) dv[3][j] = 0.f;
          }
          if (per < kSplits) {  // this CTA's partials, for the tile's CTAs to add up
            if (ok && q < rows) {
              float* pr = part + static_cast<size_t>(sp) * kUmmaRows * 128 + r;
#pragma unroll
              for (int g = 0; g < 4; ++g)
#pragma unroll
                for (int j = 0; j < 8; ++j) pr[static_cast<size_t>(g * kUmmaUnits + c + j) * kUmmaRows] = dv[g][j];
            }
          } else {  // partials in order 0 .. kSplits - 1
#pragma unroll
            for (int g = 0; g < 4; ++g)
#pragma unroll
              for (int j = 0; j < 8; ++j) dsum[g][j] += dv[g][j];
          }
        }
        if (per == kSplits && q < rows && ok) gru_pointwise<8>(p, jb, u0 + c, dsum, X, H);
      }
      return ok;
    };
    if (per < kSplits) {  // the tile's CTAs meet, then each adds up all partials for its share of the units
      const int share = kUmmaUnits / cpt;  // 8 or 16 units of this CTA, over two groups of 128 threads
      ok = share == 8 ? split_meet_reduce<4>(p, jl, rows, part, row0, u0, part_idx * share, X, H, p.gru_ticket + tile,
                                             cpt, ok, &s_ok, epilogue)
                      : split_meet_reduce<8>(p, jl, rows, part, row0, u0, part_idx * share, X, H, p.gru_ticket + tile,
                                             cpt, ok, &s_ok, epilogue);
    } else {
      ok = epilogue(ok);
    }
    ring.tiles += 1;
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    ok = __syncthreads_and(ok);  // the accumulators are read before the next unit's first MMA overwrites them
    if (!ok) {
      record_error(p.hdr, DT_ERR_TIMEOUT);
      atomicExch(&p.hdr->abort, 1u);
      return false;
    }
  }
  return true;
}

// Waits (bounded) for the current phase of `bar`; false when the wait ran out (recorded, abort raised).
__device__ __forceinline__ bool wait_copies(const Params& p, uint64_t* bar, unsigned& uses) {
  const bool ok = mbar_wait(bar, uses & 1u, kCopyBudgetNs);  // bulk copies take microseconds: this stops a lost one
  ++uses;
  if (!ok) {
    record_error(p.hdr, DT_ERR_TIMEOUT);
    atomicExch(&p.hdr->abort, 1u);
  }
  return ok;
}

// ---- phase B1 by groups: one request's expansions at one block position share that position's correction rows --
// The group's M rows W_c[ids] are gathered once and the corrections of all its J expansions come out of one
// tensor-core product Z[M][J] = W_c[ids] . [h_1 .. h_J]: mma.sync m16n8k16, the rows as A (a warp per 16 rows), the
// hidden states as the n8 B tile, split into bf16 hi + lo pairs (as the GRU's hidden side). Column j of Z depends on
// h_j alone, summed in a fixed order, so an expansion's children do not depend on which expansions share its group.
// Then one warp per expansion: the restricted log-softmax, and the children ranked by a warp sort (M <= 128) into the
// request's state block. Group g goes to CTA g mod G.
// A CTA's groups form a pipeline: once a group's product is formed, the next group's rows and hidden states are
// copied in (16-byte cp.async by every thread: a bulk copy per 1 KB row would queue on the CTA's copy engine) while
// its children are ranked. Ids and base logits are loaded a group ahead of that (registers, then one of two shared
// buffers), jobs and control words two groups ahead (three buffers), and rows are asked of L2 a group ahead.
__device__ __forceinline__ void prefetch_l2_line(const void* src) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
}
__device__ bool children_groups(const Params& p, int w, const Job* jl, unsigned char* smem, GroupPrefetch* pf) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int M = p.M, n = p.n, H = p.H, X = p.xslots, KM = M < n ? M : n;
  const ReqLayout RL = req_layout(n, X, KM, p.lookahead);
  const GroupSmem GS = group_smem(M, H);
  uint4* bfrag = reinterpret_cast<uint4*>(smem + GS.bfrag);
  float* hbuf = reinterpret_cast<float*>(smem + GS.h);
  int* ids2 = reinterpret_cast<int*>(smem + GS.ids);       // [2][M4]
  float* vals2 = reinterpret_cast<float*>(smem + GS.vals);  // [2][M4]
  unsigned short* rows_s = reinterpret_cast<unsigned short*>(smem + GS.rows);
  float* z = reinterpret_cast<float*>(smem + GS.z);
  Node* kraw = reinterpret_cast<Node*>(smem + GS.kraw);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem + GS.keys);
  Job* s_jobs = reinterpret_cast<Job*>(smem + GS.jobs);     // [3][kLargeLookahead]
  ReqCtl* s_ctl = reinterpret_cast<ReqCtl*>(smem + GS.ctl);  // [3]: the groups' requests' control words
  const int SW = H + 8;  // padded row stride of the gathered rows (elements)
  const int M4 = round4(M);
  const size_t rb = static_cast<size_t>(H) * 2;
  const int G = static_cast<int>(gridDim.x);
  const JobGroup* gl = p.grouplist + static_cast<size_t>(w & 1) * p.B * p.lookahead;
  // the wave's group count and this CTA's first group: loaded during the GRU phase (pf), else read together here
  // (the list's slot exists even when the group does not: then it holds an older wave's entry, unused)
  const bool pre = pf->valid != 0;
  JobGroup gr{};
  int ngroups;
  if (pre) {
    gr = pf->gr;
    ngroups = pf->ngroups;
  } else {
    if (static_cast<int>(blockIdx.x) < p.B * p.lookahead) gr = gl[blockIdx.x];
    ngroups = __ldcg(p.groupcount + w);
  }
  if (static_cast<int>(blockIdx.x) >= ngroups) return true;
  auto cand_pos = [&](const JobGroup& g) { return (static_cast<size_t>(g.b) * p.K + g.depth) * M; };
  // a group's jobs (32 bytes each) and its request's control word, as 16-byte copies into buffer `slot`
  static_assert(sizeof(Job) == 32 && sizeof(ReqCtl) % 16 == 0, "copied in 16-byte pieces");
  auto copy_meta = [&](const JobGroup& g, int slot) {
    if (t < 2 * g.count)
      cp_async16(reinterpret_cast<char*>(s_jobs + slot * kLargeLookahead) + 16 * t,
                 reinterpret_cast<const char*>(jl + g.start) + 16 * t);
    else if (t == 2 * kLargeLookahead)
      cp_async16(s_ctl + slot, p.rstate + static_cast<size_t>(g.b) * RL.bytes + RL.ctl);
  };
  // a group's rows (warp w: rows w, w + 8, ...; lane l: 16-byte pieces l, l + 32, ...) and its hidden states
  auto copy_inputs = [&](const JobGroup& g, const int* ids, const Job* jobs) {
    for (int m = warp; m < M; m += kWarps) {
      const char* src = static_cast<const char*>(p.w_c) + static_cast<size_t>(ids[m]) * rb;
      unsigned short* dst = rows_s + static_cast<size_t>(m) * SW;
      for (int c = lane; c < H / 8; c += 32) cp_async16(dst + 8 * c, src + 16 * c);
    }
    for (int j = warp; j < g.count; j += kWarps) {
      const float* src = p.hs + (static_cast<size_t>(g.b) * X + jobs[j].xslot) * H;
      for (int c = lane; c < H / 4; c += 32) cp_async16(hbuf + static_cast<size_t>(j) * H + 4 * c, src + 4 * c);
    }
  };
  // prologue: the first group's ids, jobs and inputs; the second's ids (registers) and jobs
  int nid = 0;
  float nval = 0.f;
  if (pre) {
    if (t < M) {
      ids2[t] = pf->ids[t];
      vals2[t] = pf->vals[t];
    }
    if (t < gr.count) s_jobs[t] = pf->jobs[t];
    if (t == 0) s_ctl[0] = pf->ctl;
  } else {
    if (t < M) {
      nid = __ldg(p.ids + cand_pos(gr) + t);
      nval = __ldg(p.vals + cand_pos(gr) + t);
    }
    copy_meta(gr, 0);
    cp_async_commit();
    if (t < M) {
      ids2[t] = valid_id(p, nid);
      vals2[t] = nval;
    }
  }
  JobGroup next{};
  if (static_cast<int>(blockIdx.x) + G < ngroups) {
    next = gl[blockIdx.x + G];
    if (t < M) {
      nid = __ldg(p.ids + cand_pos(next) + t);
      nval = __ldg(p.vals + cand_pos(next) + t);
    }
  }
  cp_async_wait_all();
  __syncthreads();
  copy_inputs(gr, ids2, s_jobs);
  if (static_cast<int>(blockIdx.x) + G < ngroups) copy_meta(next, 1);
  cp_async_commit();
  for (int g0 = blockIdx.x, k = 0; g0 < ngroups; g0 += G, ++k) {
    const int cb = k & 1, cm = k % 3, J = gr.count;
    const bool more1 = g0 + G < ngroups, more2 = g0 + 2 * G < ngroups;
    const int* ids = ids2 + cb * M4;
    cp_async_wait_all();
    __syncthreads();  // this group's rows and hidden states, the next group's jobs have landed
    // the B fragments: for k16 step s and lane l (column g = l / 4, tg = l % 4) the hi and lo bf16 pairs of
    // h_g[16 s + 2 tg, + 1] and h_g[16 s + 2 tg + 8, + 9]; columns g >= J are never read back
    for (int e = t; e < 2 * H; e += kThreads) {
      const int st = e >> 5, l = e & 31, g = l >> 2, tg = l & 3;
      if (g < J) {
        const float* hg = hbuf + static_cast<size_t>(g) * H + 16 * st + 2 * tg;
        const float2 x0 = *reinterpret_cast<const float2*>(hg), x1 = *reinterpret_cast<const float2*>(hg + 8);
        uint4 f;
        split_bf16x2(x0.x, x0.y, f.x, f.z);
        split_bf16x2(x1.x, x1.y, f.y, f.w);
        bfrag[e] = f;
      }
    }
    // the next group's rows into L2 (its ids are in registers)
    if (more1 && t < M && static_cast<unsigned>(nid) < static_cast<unsigned>(p.V)) {
      const char* src = static_cast<const char*>(p.w_c) + static_cast<size_t>(nid) * rb;
      for (size_t c = 0; c < rb; c += 128) prefetch_l2_line(src + c);
    }
    __syncthreads();
    // Z[M][8] = rows . [h_0 .. h_7], columns j >= J unused. The 16-row tiles times `ks` K parts make the warps' work
    // (ks = 8 / tiles, so every warp has a share when M < 128); each warp runs four accumulator chains (even and odd
    // k16 steps, hi and lo halves) and stores its partial tile; the partials are then added in a fixed order (part 0
    // first; even chain before odd, hi before lo), the same for every group, so Z does not depend on how many columns
    // are in use.
    {
      const int g = lane >> 2, tg = lane & 3;
      const int tiles = (M + 15) / 16, ks = tiles >= kWarps ? 1 : kWarps / tiles, steps = H / 16;
      float* zp = reinterpret_cast<float*>(smem + GS.zpart);
      for (int item = warp; item < tiles * ks; item += kWarps) {
        const int mt = item / ks, part = item % ks;
        const int s0 = steps * part / ks, s1 = steps * (part + 1) / ks;
        const int r0 = min(mt * 16 + g, M - 1), r1 = min(mt * 16 + g + 8, M - 1);
        const unsigned short* a_lo = rows_s + static_cast<size_t>(r0) * SW + tg * 2;
        const unsigned short* a_hi = rows_s + static_cast<size_t>(r1) * SW + tg * 2;
        // four accumulator chains: even and odd k16 steps, each with the hi and the lo halves apart
        float eh[4] = {0.f, 0.f, 0.f, 0.f}, el[4] = {0.f, 0.f, 0.f, 0.f};
        float oh[4] = {0.f, 0.f, 0.f, 0.f}, ol[4] = {0.f, 0.f, 0.f, 0.f};
        auto step = [&](int st, float (&dh)[4], float (&dl)[4]) {
          const int kk = st * 16;
          const uint32_t a0 = lds32(a_lo + kk), a1 = lds32(a_hi + kk), a2 = lds32(a_lo + kk + 8), a3 = lds32(a_hi + kk + 8);
          const uint4 f = bfrag[st * 32 + lane];
          mma_bf16_16816(dh, a0, a1, a2, a3, f.x, f.y);
          mma_bf16_16816(dl, a0, a1, a2, a3, f.z, f.w);
        };
        int st = s0;
        for (; st + 1 < s1; st += 2) {
          step(st, eh, el);
          step(st + 1, oh, ol);
        }
        if (st < s1) step(st, eh, el);
        // this item's partial tile: rows g, g + 8 and columns 2 tg, 2 tg + 1 of tile mt, the chains added in order
        float* zt = zp + static_cast<size_t>(item) * 16 * kLargeLookahead;
        zt[g * kLargeLookahead + 2 * tg] = (eh[0] + el[0]) + (oh[0] + ol[0]);
        zt[g * kLargeLookahead + 2 * tg + 1] = (eh[1] + el[1]) + (oh[1] + ol[1]);
        zt[(g + 8) * kLargeLookahead + 2 * tg] = (eh[2] + el[2]) + (oh[2] + ol[2]);
        zt[(g + 8) * kLargeLookahead + 2 * tg + 1] = (eh[3] + el[3]) + (oh[3] + ol[3]);
      }
      __syncthreads();
      const float* vals = vals2 + cb * M4;
      for (int i = t; i < J * M; i += kThreads) {  // the corrected logits: the parts added in order
        const int j = i / M, m = i % M, mt = m / 16, r = m % 16;
        float v = 0.f;
        for (int part = 0; part < ks; ++part)
          v += zp[static_cast<size_t>(mt * ks + part) * 16 * kLargeLookahead + r * kLargeLookahead + j];
        z[j * M4 + m] = (vals[m] + v) / p.T_eff;
      }
    }
    // the next group's ids into the other buffer; the one after it into registers
    if (more1 && t < M) {
      ids2[(cb ^ 1) * M4 + t] = valid_id(p, nid);
      vals2[(cb ^ 1) * M4 + t] = nval;
    }
    JobGroup next2{};
    if (more2) {
      next2 = gl[g0 + 2 * G];
      if (t < M) {
        nid = __ldg(p.ids + cand_pos(next2) + t);
        nval = __ldg(p.vals + cand_pos(next2) + t);
      }
    }
    __syncthreads();  // the rows, hidden states and fragments are free; the next group's ids are in place
    if (more1) {
      copy_inputs(next, ids2 + (cb ^ 1) * M4, s_jobs + ((k + 1) % 3) * kLargeLookahead);
      if (more2) copy_meta(next2, (k + 2) % 3);
      cp_async_commit();
    }
    // one warp per expansion: restricted log-softmax, children, their ranking into the request's state block (kc:
    // at most n - s - 1 of them can still be popped after the node itself, n for the root's; s from the request's
    // control word, written back by its owner before the last barrier)
    if (warp < J) {
      const Job jb = s_jobs[cm * kLargeLookahead + warp];
      const float* zj = z + warp * M4;
      Node* kr = kraw + warp * M;
      unsigned long long* kk = keys + warp * M;
      float mx = -INFINITY;
      for (int m = lane; m < M; m += 32) mx = fmaxf(mx, zj[m]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      float sum = 0.f;
      for (int m = lane; m < M; m += 32) sum += expf(zj[m] - mx);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
      const float lse = logf(sum);
      for (int m = lane; m < M; m += 32) {
        Node e;
        e.score = jb.score + ((zj[m] - mx) - lse);
        e.token = ids[m];
        e.seq = m;  // the candidate index until the node is popped
        e.pslot = static_cast<short>(jb.xslot);
        e.xslot = -1;
        kr[m] = e;
        kk[m] = (static_cast<unsigned long long>(key_of_f32(__float_as_uint(e.score))) << 32) |
                static_cast<unsigned long long>(~static_cast<uint32_t>(e.token));
      }
      __syncwarp();
      const ReqView R = req_view(p.rstate + static_cast<size_t>(jb.b) * RL.bytes, RL);
      const int kc = min(KM, jb.pslot < 0 ? n : n - s_ctl[cm].s - 1);
      Node* out = R.kids + static_cast<size_t>(jb.xslot) * KM;
      rank_children(kr, kk, M, p.V, out, kc);
      if (lane == 0) R.kcount[jb.xslot] = kc;
    }
    gr = next;
    next = next2;
  }
  // the children lists are read back through the async proxy (the owner's bulk copy of the state block)
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// ---- phase B1: the children of every expansion of the wave, spread over all CTAs ------------------------------
// Expansion q of the packed list goes to CTA q mod G: the M correction rows of the node's block position gathered
// and dotted with its new hidden state (bulk copies on an mbarrier; the next expansion's rows are asked of L2
// meanwhile), the restricted log-softmax, the siblings ranked by 64-bit keys; the first min(M, n) children and their
// count go into the request's state block in the workspace. Returns false when a copy wait ran out.
__device__ bool children_phase(const Params& p, const Job* jl, int rows, unsigned char* smem, uint64_t* bar,
                               unsigned& bar_uses) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int M = p.M, n = p.n, H = p.H, X = p.xslots, KM = M < n ? M : n;
  const size_t esize = p.bf16 ? 2 : 4;
  const ReqLayout RL = req_layout(n, X, KM, p.lookahead);
  const FrontierSmem FS = frontier_smem(0, M, H);
  float* h = reinterpret_cast<float*>(smem + FS.h);
  float* z = reinterpret_cast<float*>(smem + FS.z);
  float* vals = reinterpret_cast<float*>(smem + FS.vals);
  int* ids = reinterpret_cast<int*>(smem + FS.ids);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem + FS.keys);
  Node* kraw = reinterpret_cast<Node*>(smem + FS.kraw);
  unsigned char* rows_s = smem + FS.rows;
  const bool rows_in_smem = p.rows_smem;
  const unsigned rb = static_cast<unsigned>(H * esize);
  __shared__ float s_red[2];
  // With at least one request per CTA every CTA takes its own requests' expansions (no CTA would idle, and the
  // children lists need no grid barrier before the owner reads them); else expansion q goes to CTA q mod G.
  const bool own = p.B >= static_cast<int>(gridDim.x);
  __shared__ int s_mine[kThreads + 1];  // own mode: this CTA's expansions among the next kThreads of the list
  for (int q0 = own ? 0 : blockIdx.x; q0 < rows; q0 += own ? kThreads : gridDim.x) {
    int nmine = 1;
    if (own) {  // the owned expansions of this batch, found by every thread at once (their order does not matter)
      __syncthreads();
      if (t == 0) s_mine[kThreads] = 0;
      __syncthreads();
      if (q0 + t < rows && jl[q0 + t].b % static_cast<int>(gridDim.x) == static_cast<int>(blockIdx.x))
        s_mine[atomicAdd(&s_mine[kThreads], 1)] = q0 + t;
      __syncthreads();
      nmine = s_mine[kThreads];
    }
    for (int k = 0; k < nmine; ++k) {
      const int q = own ? s_mine[k] : q0;
      const Job jb = jl[q];
      const size_t pos = (static_cast<size_t>(jb.b) * p.K + jb.depth) * M;
      __syncthreads();  // the previous expansion is done with the shared buffers
      if (t == 0) {  // the node's hidden state (written through the generic proxy by the GRU phase): a bulk copy
        asm volatile("fence.proxy.async.global;" ::: "memory");
        mbar_expect_tx(bar, static_cast<unsigned>(H * 4));
        bulk_g2s(h, p.hs + (static_cast<size_t>(jb.b) * X + jb.xslot) * H, static_cast<unsigned>(H * 4), bar);
      }
      for (int m = t; m < M; m += kThreads) {  // ids and base logits of its block position (any M: plain loads)
        ids[m] = valid_id(p, __ldg(p.ids + pos + m));
        vals[m] = __ldg(p.vals + pos + m);
      }
      if (!own && q + static_cast<int>(gridDim.x) < rows && warp == 1) {  // the next expansion's rows, into L2
        const Job nj = jl[q + gridDim.x];
        const size_t npos = (static_cast<size_t>(nj.b) * p.K + nj.depth) * M;
        for (int m = lane; m < M; m += 32) {
          const int id = __ldg(p.ids + npos + m);
          if (static_cast<unsigned>(id) < static_cast<unsigned>(p.V))
            prefetch_l2(static_cast<const char*>(p.w_c) + static_cast<size_t>(id) * rb, rb);
        }
      }
      if (!__syncthreads_and(wait_copies(p, bar, bar_uses))) return false;
      if (rows_in_smem) {  // the M correction rows, one bulk copy each (issued by warp 0's lanes)
        if (warp == 0) {
          if (lane == 0) mbar_expect_tx(bar, rb * static_cast<unsigned>(M));
          __syncwarp();
          for (int m = lane; m < M; m += 32)
            bulk_g2s(rows_s + static_cast<size_t>(m) * rb, static_cast<const char*>(p.w_c) + static_cast<size_t>(ids[m]) * rb,
                     rb, bar);
        }
        if (!__syncthreads_and(wait_copies(p, bar, bar_uses))) return false;
      }
      for (int m0 = warp * 8; m0 < M; m0 += kWarps * 8) {  // each warp: 8 consecutive rows at a time
        float d[8];
        warp_dot_rows8(rows_in_smem ? rows_s : nullptr, p.w_c, ids, p.bf16, m0, M, h, H, d);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (lane == j && m0 + j < M) z[m0 + j] = (vals[m0 + j] + d[j]) / p.T_eff;
      }
      __syncthreads();
      if (warp == 0) {
        float mx = -INFINITY;
        for (int m = lane; m < M; m += 32) mx = fmaxf(mx, z[m]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        float sum = 0.f;
        for (int m = lane; m < M; m += 32) sum += expf(z[m] - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        if (lane == 0) {
          s_red[0] = mx;
          s_red[1] = logf(sum);
        }
      }
      __syncthreads();
      const float mx = s_red[0], lse = s_red[1];
      for (int m = t; m < M; m += kThreads) {
        Node e;
        e.score = jb.score + ((z[m] - mx) - lse);
        e.token = ids[m];
        e.seq = m;  // the candidate index until the node is popped
        e.pslot = static_cast<short>(jb.xslot);
        e.xslot = -1;
        kraw[m] = e;
        keys[m] = (static_cast<unsigned long long>(key_of_f32(__float_as_uint(e.score))) << 32) |
                  static_cast<unsigned long long>(~static_cast<uint32_t>(e.token));
      }
      __syncthreads();
      // rank among siblings (score, then token, then candidate index); the first kc kept: at most n - s - 1 of them can
      // still be popped after the node itself (n for the root's), s being the request's pops so far (its state block,
      // written back by its owner before the last barrier)
      const ReqView R = req_view(p.rstate + static_cast<size_t>(jb.b) * RL.bytes, RL);
      const int kc = min(KM, jb.pslot < 0 ? n : n - __ldcg(&R.ctl->s) - 1);
      for (int i = t; i < M; i += kThreads) {
        const unsigned long long ki = keys[i];
        int r = 0;
#pragma unroll 8
        for (int c = 0; c < M; ++c) {
          const unsigned long long kk = keys[c];
          r += (kk > ki) | ((kk == ki) & (c < i));
        }
        if (r < kc) R.kids[static_cast<size_t>(jb.xslot) * KM + r] = kraw[i];
      }
      if (t == 0) R.kcount[jb.xslot] = kc;
    }
  }
  // the children lists are read back through the async proxy (the owner's bulk copy of the state block)
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// ---- phase B2: pops and picks of every request (the CTA that owns it) -----------------------------------------
// The request's state block comes into shared memory as one bulk copy; one warp pops and picks (request_step); the
// picks join the next wave's packed list; the block goes back as one bulk copy; a finished request writes its
// outputs and ancestor-mask rows. Returns false when a copy wait ran out.
__device__ bool control_phase(const Params& p, int w, unsigned char* smem, uint64_t* bar, unsigned& bar_uses) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int M = p.M, n = p.n, X = p.xslots, KM = M < n ? M : n, kla = p.lookahead;
  const ReqLayout RL = req_layout(n, X, KM, kla);
  const size_t rstride = (RL.bytes + 127) / 128 * 128;  // one shared-memory region per request of a batch
  const int G = static_cast<int>(gridDim.x), C = p.ctl_conc;
  Job* next = p.joblist + static_cast<size_t>((w + 1) & 1) * p.B * kla;
  __shared__ int s_off[kWarps], s_cnt[kWarps];  // a batch request's place in the next wave's list, its picks
  __shared__ int s_done[kWarps];                  // the request was finished in an earlier wave
  // The requests this CTA owns (b = blockIdx.x + i G), up to C at a time: their state blocks come in by bulk copies
  // on one barrier, warp i runs request i's best-first step, and the rest follows request by request.
  for (int b0 = blockIdx.x; b0 < p.B; b0 += G * C) {
    int nb = 0;
    while (nb < C && b0 + nb * G < p.B) ++nb;
    __syncthreads();  // the previous batch (or phase) is done with the shared buffers
    if (t == 0) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      mbar_expect_tx(bar, static_cast<unsigned>(RL.bytes * nb));
      for (int i = 0; i < nb; ++i)
        bulk_g2s(smem + i * rstride, p.rstate + static_cast<size_t>(b0 + i * G) * RL.bytes,
                 static_cast<unsigned>(RL.bytes), bar);
    }
    if (!__syncthreads_and(wait_copies(p, bar, bar_uses))) return false;
    if (warp < nb) {
      const int b = b0 + warp * G;
      unsigned char* base = smem + warp * rstride;
      const ReqView R = req_view(base, RL);
      const bool done = R.ctl->s >= n;
      Job* jobs = reinterpret_cast<Job*>(base + RL.jobs);
      if (!done) {
        // each pick's embedding row is asked of L2 as soon as the pick is made: the activation rows below read it
        const auto ask_l2 = [&](int, const Job& jb) {
          if (p.xact_on) prefetch_l2(static_cast<const unsigned short*>(p.emb) + static_cast<size_t>(jb.token) * p.E,
                                     static_cast<unsigned>(p.E * 2));
        };
        request_step(R, b, n, M, p.max_depth, X, KM, kla, jobs, p.hdr, ask_l2);
      }
      // the request's picks: ordered by depth (stable: a request's expansions at one block position sit together
      // in the packed list, and each such run is a group of the children phase), their places reserved in the next
      // wave's lists; one lane per request, the batch's requests at once
      if ((t & 31) == 0) {
        s_done[warp] = done;
        s_off[warp] = 0;
        s_cnt[warp] = 0;
        const int nj = done ? 0 : R.ctl->njobs;
        if (nj > 0) {
          for (int q = 1; q < nj; ++q)
            for (int k = q; k > 0 && jobs[k - 1].depth > jobs[k].depth; --k) {
              const Job tmp = jobs[k];
              jobs[k] = jobs[k - 1];
              jobs[k - 1] = tmp;
            }
          int ng = 1;
          for (int q = 1; q < nj; ++q) ng += jobs[q].depth != jobs[q - 1].depth;
          const int off = atomicAdd(p.jobcount + w + 1, nj);
          int gi = atomicAdd(p.groupcount + w + 1, ng);
          JobGroup* gnext = p.grouplist + static_cast<size_t>((w + 1) & 1) * p.B * kla;
          for (int q = 0; q < nj;) {
            int e = q + 1;
            while (e < nj && jobs[e].depth == jobs[q].depth) ++e;
            gnext[gi++] = JobGroup{off + q, e - q, b, jobs[q].depth};
            q = e;
          }
          s_off[warp] = off;
          s_cnt[warp] = nj;
        }
      }
    }
    __syncthreads();
    int total_jobs = 0;
    for (int i = 0; i < nb; ++i) total_jobs += s_cnt[i];
    // the picks into the next wave's packed list, and their GRU inputs as the tensor-core GRU reads them
    // ([emb | hi(h_parent) | lo(h_parent)]): every pick of the batch at once, each thread's loads issued together
    for (int q = t; q < total_jobs; q += kThreads) {
      int i = 0, qq = q;
      while (qq >= s_cnt[i]) qq -= s_cnt[i++];
      next[s_off[i] + qq] = reinterpret_cast<const Job*>(smem + i * rstride + RL.jobs)[qq];
    }
    if (p.xact_on && total_jobs > 0) {
      // each pick's embedding row and parent state come into a staging slot (16-byte cp.async by the warp that owns
      // the slot, every slot of a round at once) and go out from there as its activation row; ctl_stage slots follow
      // the batch's state blocks
      const int E = p.E, H = p.H, Kx = E + 2 * H, ce = E / 8, per = ce + H / 4;
      const size_t pick_bytes = static_cast<size_t>(E) * 2 + static_cast<size_t>(H) * 4;
      unsigned char* stage = smem + static_cast<size_t>(C) * rstride;
      auto locate = [&](int q, int& r, int& qi) {  // pick q of the batch: request r's job qi
        r = 0;
        qi = q;
        while (qi >= s_cnt[r]) qi -= s_cnt[r++];
      };
      for (int q0 = 0; q0 < total_jobs; q0 += p.ctl_stage) {
        const int np = min(p.ctl_stage, total_jobs - q0);
        for (int pk = warp; pk < np; pk += kWarps) {
          int r, qi;
          locate(q0 + pk, r, qi);
          const Job jb = reinterpret_cast<const Job*>(smem + r * rstride + RL.jobs)[qi];
          const char* esrc = static_cast<const char*>(p.emb) + static_cast<size_t>(jb.token) * E * 2;
          const char* hsrc =
              reinterpret_cast<const char*>(p.hs + (static_cast<size_t>(b0 + r * G) * X + jb.pslot) * H);
          unsigned char* slot = stage + pk * pick_bytes;
          for (int c = lane; c < per; c += 32) cp_async16(slot + 16 * c, c < ce ? esrc + 16 * c : hsrc + 16 * (c - ce));
        }
        cp_async_commit();
        cp_async_wait_all();
        __syncwarp();
        for (int pk = warp; pk < np; pk += kWarps) {
          int r, qi;
          locate(q0 + pk, r, qi);
          unsigned short* xr = p.xact + static_cast<size_t>(s_off[r] + qi) * Kx;
          const unsigned char* slot = stage + pk * pick_bytes;
          for (int c = lane; c < ce; c += 32)
            reinterpret_cast<uint4*>(xr)[c] = reinterpret_cast<const uint4*>(slot)[c];
          for (int c = lane; c < H / 4; c += 32) {
            const float4 h = reinterpret_cast<const float4*>(slot + static_cast<size_t>(E) * 2)[c];
            uint2 hi, lo;
            split_bf16x2(h.x, h.y, hi.x, lo.x);
            split_bf16x2(h.z, h.w, hi.y, lo.y);
            *reinterpret_cast<uint2*>(xr + E + 4 * c) = hi;
            *reinterpret_cast<uint2*>(xr + E + H + 4 * c) = lo;
          }
        }
        __syncwarp();  // a warp's slots are read out before its next round's copies land in them
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");  // read by TMA (async proxy) after the next barrier
    }
    for (int i = 0; i < nb; ++i) {
      if (s_done[i]) continue;  // uniform
      const int b = b0 + i * G;
      unsigned char* base = smem + i * rstride;
      const ReqView R = req_view(base, RL);
      const ReqCtl st = *R.ctl;
      if (st.s >= n) {  // finished: the outputs, and each node's ancestor-mask row by walking its parent chain
        resolve_parents(R.pops, R.popidx, n, t, kThreads);
        __syncthreads();
        const size_t o = static_cast<size_t>(b) * n;
        for (int k = t; k < n; k += kThreads) {
          const PopRec rr = R.pops[k];
          p.tokens[o + k] = rr.token;
          p.parents[o + k] = rr.parent;
          p.depth[o + k] = rr.depth;
          p.scores[o + k] = rr.score;
        }
        for (int k = t; k < n * n; k += kThreads) {
          const int row = k / n, c = k % n;
          int a = row;
          for (int hops = 0; a > c && hops < n; ++hops) a = R.pops[a].parent;  // parents precede their children
          p.mask[(o + row) * n + c] = a == c;
        }
      }
      // the state block goes back but for its children lists (bulk copies; all of the batch's complete before the
      // buffers are reused): the children phase writes the lists, and the lists change here only where a lookahead
      // pick was marked as expanded, one 16-byte entry per such pick
      __syncthreads();
      if (t == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        unsigned char* gb = p.rstate + static_cast<size_t>(b) * RL.bytes;
        bulk_s2g(gb, base, static_cast<unsigned>(RL.kids));
        bulk_s2g(gb + RL.kcount, base + RL.kcount, static_cast<unsigned>(RL.bytes - RL.kcount));
        const Job* jobs = reinterpret_cast<const Job*>(base + RL.jobs);
        for (int q = 0; q < s_cnt[i]; ++q)
          if (jobs[q].aux[1] > 0) {
            const size_t at = RL.kids + static_cast<size_t>(jobs[q].aux[1] - 1) * sizeof(Node);
            bulk_s2g(gb + at, base + at, static_cast<unsigned>(sizeof(Node)));
          }
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    }
    if (t == 0) {
      asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
      asm volatile("fence.proxy.async.global;" ::: "memory");  // other CTAs write new children lists into them next
    }
  }
  return true;
}

// Before the first wave: every owned request's state block (the root expanded in wave 0 with h0, which becomes
// slot 0's hidden state), and every wave's job count at zero.
__device__ void init_requests(const Params& p, unsigned char* smem) {
  const int t = threadIdx.x;
  const int M = p.M, n = p.n, H = p.H, X = p.xslots, KM = M < n ? M : n;
  const ReqLayout RL = req_layout(n, X, KM, p.lookahead);
  // wave 0 expands the roots: its packed list holds one job per request
  for (int i = blockIdx.x * kThreads + t; i < X + 2; i += gridDim.x * kThreads) {
    p.jobcount[i] = i == 0 ? p.B : 0;
    p.groupcount[i] = i == 0 ? p.B : 0;
  }
  for (int i = blockIdx.x * kThreads + t; i < p.gru_tiles; i += gridDim.x * kThreads) p.gru_ticket[i] = 0u;
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    if (t == 0) {
      p.joblist[b] = Job{b, 0, -1, 0, 0, 0.f, {0, 0}};
      p.grouplist[b] = JobGroup{b, 1, b, 0};
    }
    const ReqView R = req_view(p.rstate + static_cast<size_t>(b) * RL.bytes, RL);
    Job* jobs = reinterpret_cast<Job*>(p.rstate + static_cast<size_t>(b) * RL.bytes + RL.jobs);
    if (t == 0) {
      *R.ctl = ReqCtl{0, 0, M, 1, 1, {0, 0, 0}};  // the root's children take insertion indices 0 .. M - 1
      jobs[0] = Job{b, 0, -1, 0, 0, 0.f, {0, 0}};
    }
    if (t < 32) R.lanes[t] = t == 0 ? LaneSrc{-2, 0, 0, 0, -1, {0, 0, 0}} : t == 1 ? LaneSrc{0, 0, -1, 0, 1, {0, 0, 0}} : LaneSrc{-1, 0, 0, 0, -1, {0, 0, 0}};
    for (int i = t; i < X; i += kThreads) {
      R.kcount[i] = 0;
      R.popidx[i] = i == 0 ? -1 : -2;
      R.sdepth[i] = 0;
    }
    for (int i = t; i < n; i += kThreads) R.pops[i] = PopRec{0, 0, 0, -INFINITY};
    for (int i = t; i < H; i += kThreads)
      p.hs[static_cast<size_t>(b) * X * H + i] = __ldg(p.h0 + static_cast<size_t>(b) * H + i);
  }
  // the state blocks are read back through the async proxy (bulk copies)
  asm volatile("fence.proxy.async.global;" ::: "memory");
  (void)smem;
}

// The waves of one launch; every way out (done, or a wait that ran out) returns here in every thread of the CTA.
template <int kGemm>
__device__ void run_waves(const Params& p, const TmaMaps& maps, unsigned char* smem, UmmaRing& ring, GroupPrefetch* pf,
                          unsigned long long base_count, uint64_t* bar, int* s_flag) {
  unsigned bar_uses = 0;
  const unsigned G = gridDim.x;
  const uint64_t t_launch = global_timer_ns();
  uint64_t gather_ns = 0, gather_bytes = 0;  // this CTA's time in the children phases; the rows read (CTA 0)
  unsigned waves = 0, expansions = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) {  // the launch's statistics start from zero, raised after the barrier
    p.hdr->stat_launch_ns = p.hdr->stat_gather_ns = p.hdr->stat_gather_bytes = 0ull;
    p.hdr->stat_waves = p.hdr->stat_expansions = 0u;
  }
  init_requests(p, smem);
  if (!grid_barrier(p.hdr, G, p.timeout_ns, s_flag)) return;
  unsigned long long target = base_count;
  for (int w = 0; w < p.xslots; ++w) {
    const int rows = __ldcg(p.jobcount + w);
    if (rows == 0) break;  // every request is finished (the same count in every CTA)
    const Job* jl = p.joblist + static_cast<size_t>(w & 1) * p.B * p.lookahead;
    if (w > 0) {  // wave 0 expands the roots, whose hidden state is h0: no GRU step
      if (kGemm == 4) {
        if (!umma_gru_phase(p, maps, jl, rows, smem, ring, w, pf)) return;
      } else if (kGemm == 1) {
        gemm_gru_phase<TileS, 32, 8>(p, jl, rows, smem);
      } else if (kGemm == 2) {
        gemm_gru_phase<TileL, 64, 16>(p, jl, rows, smem);
      } else if (kGemm == 3) {
        gemm_gru_phase<TileS128, 32, 8>(p, jl, rows, smem);
      } else {
        gru_phase(p, jl, rows, reinterpret_cast<float*>(smem));
      }
      target += G;
      if (!counter_barrier(p.hdr, target, p.timeout_ns, s_flag)) return;
      // every CTA has left the GRU phase: its meeting counters start again from zero for the next wave
      if (kGemm == 4 && blockIdx.x == 0)
        for (int i = threadIdx.x; i < p.gru_tiles; i += kThreads) p.gru_ticket[i] = 0u;
    }
    const uint64_t c0 = global_timer_ns();
    if (!(p.group_mma ? children_groups(p, w, jl, smem, pf) : children_phase(p, jl, rows, smem, bar, bar_uses))) return;
    if (threadIdx.x == 0) pf->valid = 0;  // used once (read before the barrier that follows)
    __syncthreads();
    gather_ns += global_timer_ns() - c0;
    ++waves;
    expansions += static_cast<unsigned>(rows);
    gather_bytes += static_cast<uint64_t>(p.group_mma ? __ldcg(p.groupcount + w) : rows) * p.M * p.H * (p.bf16 ? 2 : 4);
    if (p.group_mma || p.B < static_cast<int>(G)) {  // children computed by other CTAs: wait for them
      target += G;
      if (!counter_barrier(p.hdr, target, p.timeout_ns, s_flag)) return;
    } else {
      __syncthreads();  // this CTA's own children lists, stored before its fence, then read back in bulk
    }
    if (!control_phase(p, w, smem, bar, bar_uses)) return;
    target += G;
    if (!counter_barrier(p.hdr, target, p.timeout_ns, s_flag)) return;
  }
  if (threadIdx.x == 0) {
    atomicMax(&p.hdr->stat_gather_ns, static_cast<unsigned long long>(gather_ns));
    if (blockIdx.x == 0) {
      p.hdr->stat_gather_bytes = gather_bytes;
      p.hdr->stat_waves = waves;
      p.hdr->stat_expansions = expansions;
      p.hdr->stat_launch_ns = global_timer_ns() - t_launch;
    }
  }
}

// kGemm: 0 = CUDA-core GRU tiles (fp32 weights or other widths), mma.sync tensor-core tiles with 1 = TileS,
// 2 = TileL, 3 = TileS128; 4 = tcgen05 tiles (bf16, E and H multiples of 64). With kGemm = 4 the CTA holds 512 TMEM
// columns for the whole launch and frees them on every way out.
template <int kGemm>
__global__ void __launch_bounds__(kThreads, 1) build_kernel(Params p, const __grid_constant__ TmaMaps maps) {
  extern __shared__ float4 smem_f4[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(smem_f4);
  __shared__ int s_flag;
  __shared__ unsigned long long s_base;
  __shared__ uint64_t bar;  // completion of the frontier phase's bulk copies
  __shared__ uint64_t ufull[kUmmaStages], uempty[kUmmaStages], udone;
  __shared__ uint64_t wfull[kWideStages], wempty[kWideStages], umid, ur1free;
  __shared__ uint32_t s_tmem;
  __shared__ GroupPrefetch s_pf;
  if (threadIdx.x == 0) {
    s_pf.valid = 0;
    s_base = ld_relaxed_gpu_u64(&p.hdr->sync_count);  // before anyone can pass the first barrier
    mbar_init(&bar, 1);
    if (kGemm == 4) {
      for (int i = 0; i < kUmmaStages; ++i) {
        mbar_init(&ufull[i], 1);
        mbar_init(&uempty[i], 1);
      }
      mbar_init(&udone, 1);
      for (int i = 0; i < kWideStages; ++i) {
        mbar_init(&wfull[i], 1);
        mbar_init(&wempty[i], 1);
      }
      mbar_init(&umid, 1);
      mbar_init(&ur1free, 4);  // one arrival per epilogue warp
    }
    mbar_fence_init();
  }
  if (kGemm == 4 && threadIdx.x < 32) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (kGemm == 4) asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (kGemm == 4) asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  UmmaRing ring{ufull, uempty, &udone, wfull, wempty, &umid, &ur1free, kGemm == 4 ? s_tmem : 0u, 0u, 0u, 0u};
  run_waves<kGemm>(p, maps, smem, ring, &s_pf, s_base, &bar, &s_flag);
  if (kGemm == 4) {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (threadIdx.x < 32)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(ring.tmem), "r"(kTmemCols) : "memory");
  }
}

// The tcgen05 GRU's tensor maps (2-D, bf16, 128-byte swizzle): the packed activations and the two weight matrices.
// The last maps built are kept and reused while the pointers and sizes stay the same.
bool gru_tensor_maps(TmaMaps* out, const void* xact, uint64_t xrows, const void* w_ih, const void* w_hh, int E, int H) {
  static std::mutex mu;
  static TmaMaps last{};
  static const void* key[3] = {nullptr, nullptr, nullptr};
  static uint64_t key_dims[3] = {0, 0, 0};
  std::lock_guard<std::mutex> lock(mu);
  if (key[0] == xact && key[1] == w_ih && key[2] == w_hh && key_dims[0] == xrows && key_dims[1] == static_cast<uint64_t>(E) &&
      key_dims[2] == static_cast<uint64_t>(H)) {
    *out = last;
    return true;
  }
  auto map2d = [&](CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    return encode_bf16_2d(m, ptr, cols, rows, cols, kUmmaBK, box_rows);
  };
  TmaMaps m{};
  if (!map2d(&m.x, xact, static_cast<uint64_t>(E) + 2 * static_cast<uint64_t>(H), xrows, kUmmaRows) ||
      !map2d(&m.wih, w_ih, static_cast<uint64_t>(E), 3 * static_cast<uint64_t>(H), kUmmaUnits) ||
      !map2d(&m.whh, w_hh, static_cast<uint64_t>(H), 3 * static_cast<uint64_t>(H), kUmmaUnits) ||
      !map2d(&m.wih64, w_ih, static_cast<uint64_t>(E), 3 * static_cast<uint64_t>(H), kWideUnits) ||
      !map2d(&m.whh64, w_hh, static_cast<uint64_t>(H), 3 * static_cast<uint64_t>(H), kWideUnits))
    return false;
  last = m;
  key[0] = xact; key[1] = w_ih; key[2] = w_hh;
  key_dims[0] = xrows; key_dims[1] = static_cast<uint64_t>(E); key_dims[2] = static_cast<uint64_t>(H);
  *out = m;
  return true;
}

// Dynamic shared memory of the large-batch kernel; the gathered rows are staged only when they fit under both the
// cap and the device's opt-in limit (`rows_smem` reports the choice).
size_t smem_bytes(int gemm, int M, int n, int H, int kla, size_t esize, size_t optin, bool* rows_smem) {
  size_t a = sizeof(float) * (kTB * kPad + 3 * kTU * kPad);
  if (gemm == 4) a = kUmmaSmem;
  if (gemm == 1) a = TileS::kBytes;
  if (gemm == 2) a = TileL::kBytes;
  if (gemm == 3) a = TileS128::kBytes;
  const int X = expansion_slots(n), KM = M < n ? M : n;
  const size_t ctl = req_layout(n, X, KM, kla).bytes;                 // the control phase: one state block
  const FrontierSmem F = frontier_smem(0, M, H);                       // the children phase
  const size_t rows = static_cast<size_t>(M) * H * esize;
  *rows_smem = rows <= kFrontierRowsCap && F.bytes + rows <= optin;
  const size_t b = F.bytes + (*rows_smem ? rows : 0);
  size_t m = a > b ? a : b;
  return m > ctl ? m : ctl;
}

}  // namespace
}  // namespace dt

extern "C" size_t dt_build_workspace_bytes(int B, int K, int V, int M, int n, int H, int E) {
  if (B < 0 || K < 1 || V < 1 || M < 1 || n < 1 || H < 1 || E < 1) return 0;
  return dt::build_layout(B, K, V, M, n, H, E).bytes;
}

namespace dt {
namespace {

enum class BuildMode {
  kLaunch,  // validate and launch
  kCheck,   // validate only, launch nothing (dt_round checks the whole round before its first launch)
};

dt_status build_trees(int B, int K, int V, int M, int n, int max_depth, float T, const int32_t* topm_ids,
                      const float* topm_vals, const float* h0, const dt_weights* w, int32_t* out_tokens,
                      int32_t* out_parents, int32_t* out_depth, float* out_scores, uint8_t* out_mask, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream, BuildMode mode) {
  if (!w) return DT_ERR_INVALID_ARG;
  const int H = w->H, E = w->E;
  if (B < 0 || K < 1 || V < 1 || M < 1 || M > V || n < 1 || max_depth < 1 || max_depth > K) return DT_ERR_INVALID_ARG;
  if (!(T >= 0.0f) || !isfinite(T)) return DT_ERR_INVALID_ARG;
  if (H < 1 || E < 1 || H % 8 || E % 8) return DT_ERR_INVALID_ARG;
  if (w->dtype != DT_F32 && w->dtype != DT_BF16) return DT_ERR_INVALID_ARG;
  {  // n must not exceed the number of nodes of the depth-limited M-ary tree
    long long total = 0, level = 1;
    for (int d = 1; d <= max_depth && total < n; ++d) {
      level = level > n ? level : level * M;
      total += level;
    }
    if (total < n) return DT_ERR_INVALID_ARG;
  }
  if (M > DT_MAX_M || n > DT_MAX_N || H > DT_MAX_H || E > DT_MAX_E) return DT_ERR_UNSUPPORTED;
  if (B == 0) return DT_OK;  // nothing to read or write
  const void* ptrs[] = {topm_ids, topm_vals, h0, w->emb, w->w_ih, w->w_hh, w->w_c, out_tokens, out_parents,
                        out_depth, out_scores, out_mask, workspace};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return DT_ERR_INVALID_ARG;
  if ((w->b_ih && !aligned16(w->b_ih)) || (w->b_hh && !aligned16(w->b_hh))) return DT_ERR_INVALID_ARG;
  const BuildLayout L = build_layout(B, K, V, M, n, H, E);
  if (workspace_bytes < L.bytes) return DT_ERR_INVALID_ARG;

  char* ws = static_cast<char*>(workspace);
  Params p{};
  p.B = B; p.K = K; p.V = V; p.M = M; p.n = n; p.max_depth = max_depth; p.H = H; p.E = E;
  p.T_eff = T > 0.f ? T : 1.f;
  p.bf16 = w->dtype == DT_BF16;
  p.ids = topm_ids; p.vals = topm_vals; p.h0 = h0;
  p.emb = w->emb; p.w_ih = w->w_ih; p.w_hh = w->w_hh; p.b_ih = w->b_ih; p.b_hh = w->b_hh; p.w_c = w->w_c;
  p.tokens = out_tokens; p.parents = out_parents; p.depth = out_depth; p.scores = out_scores; p.mask = out_mask;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.hs = reinterpret_cast<float*>(ws + L.hs);
  p.acc = B <= kSmallMaxB ? reinterpret_cast<long long*>(ws + L.acc) : nullptr;
  p.hs_count = B <= kSmallMaxB ? reinterpret_cast<int*>(ws + L.hs_count) : nullptr;
  p.rstate = reinterpret_cast<unsigned char*>(ws + L.rstate);
  p.joblist = reinterpret_cast<Job*>(ws + L.joblist);
  p.jobcount = reinterpret_cast<int*>(ws + L.jobcount);
  p.grouplist = reinterpret_cast<JobGroup*>(ws + L.grouplist);
  p.groupcount = reinterpret_cast<int*>(ws + L.groupcount);
  p.xact = reinterpret_cast<unsigned short*>(ws + L.xact);
  p.gru_part = reinterpret_cast<float*>(ws + L.gru_part);
  p.gru_ticket = reinterpret_cast<unsigned*>(ws + L.gru_ticket);
  p.gru_tiles = L.gru_tiles;
  p.acc_stride = acc_stride(M, n);
  p.xslots = expansion_slots(n);
  p.timeout_ns = barrier_timeout_ns();
  DeviceInfo di{};
  if (current_device_info(&di) != cudaSuccess) return DT_ERR_CUDA;
  if (!di.coop) return DT_ERR_UNSUPPORTED;
  // expansions per request per wave: the setting, capped by what the builder's wave holds; by default all of the
  // small-batch builder's wave, and kLargeDefault for the large-batch builder
  const int k_set = lookahead_setting();
  {
    const int fit = kWaveJobs / (B < kWaveJobs ? B : kWaveJobs);
    p.lookahead = k_set > 0 ? (k_set < fit ? k_set : fit) : fit;
  }
  if (small_builder_fits(p, di))
    return mode == BuildMode::kCheck ? DT_OK : cuda_status(launch_small_builder(p, di, stream));
  p.lookahead = k_set > 0 ? (k_set < kLargeLookahead ? k_set : kLargeLookahead)
                          : (B >= 128 ? kLargeLookahead : kLargeDefault);

  // phase A: tcgen05 tiles when they fit (below); else mma.sync tiles for bf16 weights whose widths are multiples of
  // the pipeline chunk (the larger tile once a wave can hold 128 expansions or more); else CUDA cores
  const long long max_rows = static_cast<long long>(B) * p.lookahead;
  // tcgen05 tiles (128 expansions x 32 units) for every bf16 wave whose widths fit them: the K split makes the sums
  // independent of the wave's size, so the tree does not depend on the lookahead width
  // the kernel's static shared memory (flags, barriers, reductions, the children phase's first-group prefetch) is
  // under kStaticSmem; one CTA per SM (launch bounds), so the shared memory alone decides whether a CTA fits
  constexpr size_t kStaticSmem = 3072;
  const bool umma =
      p.bf16 && E % kUmmaBK == 0 && H % kUmmaBK == 0 && kUmmaSmem + kStaticSmem <= static_cast<size_t>(di.optin);
  const int gemm = !p.bf16 ? 0
                   : umma ? 4
                   : max_rows >= 128 ? (E % TileL::kKc == 0 && H % TileL::kKc == 0 ? 2 : 0)
                   : E % TileS::kKc == 0 && H % TileS::kKc == 0 ? 1
                   : E % TileS128::kKc == 0 && H % TileS128::kKc == 0 ? 3 : 0;
  const void* fn = gemm == 0 ? reinterpret_cast<const void*>(build_kernel<0>)
                   : gemm == 4 ? reinterpret_cast<const void*>(build_kernel<4>)
                   : gemm == 3 ? reinterpret_cast<const void*>(build_kernel<3>)
                   : gemm == 1 ? reinterpret_cast<const void*>(build_kernel<1>)
                               : reinterpret_cast<const void*>(build_kernel<2>);
  TmaMaps maps{};
  p.xact_on = gemm == 4;
  if (gemm == 4 && !gru_tensor_maps(&maps, p.xact, static_cast<uint64_t>(B) * kLargeLookahead, w->w_ih, w->w_hh, E, H))
    return DT_ERR_CUDA;
  size_t smem = smem_bytes(gemm, M, n, H, p.lookahead, p.bf16 ? 2 : 4, static_cast<size_t>(di.optin) - kStaticSmem,
                           &p.rows_smem);
  // the children phase by groups on the tensor cores when its buffers fit the same budget
  // groups spread over all CTAs (g mod G) whatever the batch: a request's groups on its owner CTA left the CTAs that
  // own two requests, and the tail waves' few groups, on one CTA each (c4: 75-85 us against a 50 us mean)
  {  // requests a CTA steps at once in the control phase: the ones it owns, as many as the shared memory holds
    const ReqLayout RL = req_layout(n, p.xslots, M < n ? M : n, p.lookahead);
    const size_t rstride = (RL.bytes + 127) / 128 * 128;
    const int owned = (B + di.sms - 1) / di.sms;
    const int fit = static_cast<int>((static_cast<size_t>(di.optin) - kStaticSmem) / rstride);
    p.ctl_conc = owned < fit ? owned : fit;
    if (p.ctl_conc > kWarps) p.ctl_conc = kWarps;
    if (p.ctl_conc < 1) p.ctl_conc = 1;
    size_t need = rstride * p.ctl_conc;
    p.ctl_stage = 0;
    if (p.xact_on) {  // staging slots for the picks' activation rows after the state blocks: all of a batch's picks
      // at once when they fit, else as many as fit (at least one)
      const size_t pick = static_cast<size_t>(E) * 2 + static_cast<size_t>(H) * 4;
      const size_t cap = static_cast<size_t>(di.optin) - kStaticSmem;
      while (p.ctl_conc > 1 && rstride * p.ctl_conc + pick > cap) --p.ctl_conc;
      if (rstride * p.ctl_conc + pick > cap) return DT_ERR_UNSUPPORTED;
      const size_t room = (cap - rstride * p.ctl_conc) / pick;
      const int want = p.ctl_conc * p.lookahead;
      p.ctl_stage = room < static_cast<size_t>(want) ? static_cast<int>(room) : want;
      need = rstride * p.ctl_conc + static_cast<size_t>(p.ctl_stage) * pick;
    }
    if (smem < need) smem = need;
  }
  p.group_mma = p.bf16 && H % 16 == 0 && M <= 128 &&
                group_smem(M, H).bytes + kStaticSmem <= static_cast<size_t>(di.optin);
  if (p.group_mma && group_smem(M, H).bytes > smem) smem = group_smem(M, H).bytes;
  if (smem + kStaticSmem > static_cast<size_t>(di.optin)) return DT_ERR_UNSUPPORTED;
  if (mode == BuildMode::kCheck) return DT_OK;
  if (ensure_dynamic_smem(fn, smem) != cudaSuccess) return DT_ERR_CUDA;
  const unsigned grid = static_cast<unsigned>(di.sms);  // one CTA per SM; co-resident under a cooperative launch
  void* args[] = {&p, &maps};
  return cuda_status(cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kThreads), args, smem, stream));
}

}  // namespace
}  // namespace dt

extern "C" dt_status dt_build_trees(int B, int K, int V, int M, int n, int max_depth, float T,
                                    const int32_t* topm_ids, const float* topm_vals, const float* h0,
                                    const dt_weights* w, int32_t* out_tokens, int32_t* out_parents,
                                    int32_t* out_depth, float* out_scores, uint8_t* out_mask, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream) {
  return dt::build_trees(B, K, V, M, n, max_depth, T, topm_ids, topm_vals, h0, w, out_tokens, out_parents, out_depth,
                         out_scores, out_mask, workspace, workspace_bytes, stream, dt::BuildMode::kLaunch);
}

extern "C" dt_status dt_round(const void* logits, dt_dtype dtype, int B, int K, int V, int M, int n, int max_depth,
                              float T, const float* h0, const dt_weights* w, int32_t* topm_ids, float* topm_vals,
                              int32_t* out_tokens, int32_t* out_parents, int32_t* out_depth, float* out_scores,
                              uint8_t* out_mask, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  using dt::BuildMode;
  // every check of both calls first (they launch nothing), so that an invalid round launches nothing at all
  dt_status st = dt::topm_check(logits, dtype, B, K, V, M, topm_ids, topm_vals, workspace, workspace_bytes);
  if (st != DT_OK) return st;
  st = dt::build_trees(B, K, V, M, n, max_depth, T, topm_ids, topm_vals, h0, w, out_tokens, out_parents,
                                 out_depth, out_scores, out_mask, workspace, workspace_bytes, stream, BuildMode::kCheck);
  if (st != DT_OK) return st;
  st = dt_topm(logits, dtype, B, K, V, M, topm_ids, topm_vals, workspace, workspace_bytes, stream);
  if (st != DT_OK) return st;
  return dt::build_trees(B, K, V, M, n, max_depth, T, topm_ids, topm_vals, h0, w, out_tokens, out_parents, out_depth,
                         out_scores, out_mask, workspace, workspace_bytes, stream, BuildMode::kLaunch);
}
