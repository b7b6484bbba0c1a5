// dt_build_trees — conditional best-first draft trees (one persistent cooperative launch per round).
//
// Method: blog.captcha.la, "Methodology — deep read" (DDTree's best-first max-priority queue keyed by cumulative
// conditional log-probability; the GRU state is carried along each root-to-node path; the correction is applied to
// the gathered top-M rows only; fixed node budget / max depth; prefix-closed tree + ancestor-only mask);
// gist.science, "Composants Clés" (only the light GRU correction and correction head are recomputed per node).
//
// GB300 design. The pages' builder replays a CUDA graph per node while a host-side heap decides the next pop
// (gist.science, "Constructeur Natif GPU"); here the whole round is one launch with no host round-trip:
//   * all B requests advance in lockstep: step s pops the s-th node of every request;
//   * phase A (all CTAs): the GRU step of the nodes popped in the previous step, as tiles of
//     [16 requests x 16 hidden units] over K = E (embedding row) then K = H (parent state), fp32 accumulation;
//   * grid barrier;
//   * phase B (one CTA per request): gather the M correction rows of the node's block position and dot them with
//     h (one warp per row), restricted log-softmax (warp reductions), merge the children into the request's
//     frontier keeping only the n - s entries that can still be popped, pop the best, write the node's output row
//     and its ancestor-mask row;
//   * grid barrier; next step.
// Every reduction has a fixed order (no floating-point atomics), so the output is bit-identical run to run.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "build_common.cuh"

namespace dt {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTB = 16;   // requests per GRU tile
constexpr int kTU = 16;   // hidden units per GRU tile
constexpr int kKC = 64;   // K-chunk of the GRU tile
constexpr int kPad = kKC + 1;

// ---- phase A: GRU step of every request whose last pop is expanded --------------------------------------------
__device__ void gru_phase(const Params& p, int node, float* smem) {
  float* xs = smem;                  // [kTB][kPad]
  float* ws = smem + kTB * kPad;     // [3][kTU][kPad]
  __shared__ int s_tok[kTB], s_par[kTB], s_exp[kTB];
  const int t = threadIdx.x, lb = t / kTU, lu = t % kTU;
  const int ublocks = (p.H + kTU - 1) / kTU;
  const int rblocks = (p.B + kTB - 1) / kTB;
  const int tiles = ublocks * rblocks;
  for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int rb = tile / ublocks, ub = tile % ublocks;
    __syncthreads();
    if (t < kTB) {
      const int b = rb * kTB + t;
      const bool ok = b < p.B && p.state[b].expand;
      s_exp[t] = ok;
      s_tok[t] = ok ? p.state[b].token : 0;
      s_par[t] = ok ? p.state[b].parent : -1;
    }
    __syncthreads();
    if (!__syncthreads_or(t < kTB && s_exp[t])) continue;
    const int b = rb * kTB + lb, k = ub * kTU + lu;
    float acc_r = 0.f, acc_u = 0.f, acc_ni = 0.f, acc_nh = 0.f;
    // input side: W_ih[gate rows] . emb[token]
    for (int e0 = 0; e0 < p.E; e0 += kKC) {
      for (int i = t; i < kTB * kKC; i += kThreads) {
        const int r = i / kKC, c = i % kKC, e = e0 + c;
        xs[r * kPad + c] = (s_exp[r] && e < p.E) ? ldw(p.emb, p.bf16, static_cast<size_t>(s_tok[r]) * p.E + e) : 0.f;
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
        const int r = i / kKC, c = i % kKC, j = j0 + c;
        float v = 0.f;
        if (s_exp[r] && j < p.H) {
          const int bb = rb * kTB + r, par = s_par[r];
          const float* hp = par < 0 ? p.h0 + static_cast<size_t>(bb) * p.H
                                    : p.hs + (static_cast<size_t>(bb) * p.n + par) * p.H;
          v = par < 0 ? __ldg(hp + j) : hp[j];
        }
        xs[r * kPad + c] = v;
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
    if (b < p.B && k < p.H && s_exp[lb]) {
      const size_t g0 = k, g1 = static_cast<size_t>(p.H) + k, g2 = 2 * static_cast<size_t>(p.H) + k;
      const float bir = p.b_ih ? ldw(p.b_ih, p.bf16, g0) : 0.f, bhr = p.b_hh ? ldw(p.b_hh, p.bf16, g0) : 0.f;
      const float biu = p.b_ih ? ldw(p.b_ih, p.bf16, g1) : 0.f, bhu = p.b_hh ? ldw(p.b_hh, p.bf16, g1) : 0.f;
      const float bin = p.b_ih ? ldw(p.b_ih, p.bf16, g2) : 0.f, bhn = p.b_hh ? ldw(p.b_hh, p.bf16, g2) : 0.f;
      const float r = sigmoidf_(acc_r + bir + bhr);
      const float u = sigmoidf_(acc_u + biu + bhu);
      const float g = tanhf((acc_ni + bin) + r * (acc_nh + bhn));
      const int par = s_par[lb];
      const float hprev = par < 0 ? __ldg(p.h0 + static_cast<size_t>(b) * p.H + k)
                                  : p.hs[(static_cast<size_t>(b) * p.n + par) * p.H + k];
      p.hs[(static_cast<size_t>(b) * p.n + node) * p.H + k] = (1.f - u) * g + u * hprev;
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
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
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
__device__ void gemm_gru_phase(const Params& p, int node, unsigned char* smem) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int E = p.E, H = p.H, B = p.B, n = p.n;
  float* red = reinterpret_cast<float*>(smem);                // [kWarps][kRT][kRS], after the main loop
  int* info = reinterpret_cast<int*>(smem + GT::kRing);        // [kRT][4]
  const int rtiles = (B + kRT - 1) / kRT, utiles = (H + kUT - 1) / kUT;
  const int nin = E / GT::kKc, nc = nin + H / GT::kKc;  // chunks: input side, then hidden side
  for (int tile = blockIdx.x; tile < rtiles * utiles; tile += gridDim.x) {
    const int b0 = (tile / utiles) * kRT, u0 = (tile % utiles) * kUT;
    __syncthreads();  // the previous tile is done with the shared buffers
    for (int r = t; r < kRT; r += kThreads) {
      const int b = b0 + r;
      const bool ok = b < B && p.state[b].expand;
      info[4 * r] = ok ? p.state[b].token : 0;
      info[4 * r + 1] = ok ? p.state[b].parent : -1;
      info[4 * r + 2] = ok;
    }
    __syncthreads();
    if (!__syncthreads_or(t < kRT && info[4 * t + 2])) continue;

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
          if (info[4 * r + 2])
            cp_async16(xdst + r * GT::kXS + piece * 8,
                       static_cast<const unsigned short*>(p.emb) + static_cast<size_t>(info[4 * r]) * E + k0 +
                           piece * 8);
        }
      } else {  // the parents' hidden states, fp32
        float* xdst = reinterpret_cast<float*>(st);
        for (int i = t; i < kRT * (GT::kKc / 4); i += kThreads) {
          const int r = i / (GT::kKc / 4), piece = i % (GT::kKc / 4);
          if (info[4 * r + 2]) {
            const int b = b0 + r, par = info[4 * r + 1];
            const float* src = par < 0 ? p.h0 + static_cast<size_t>(b) * H
                                       : p.hs + (static_cast<size_t>(b) * n + par) * H;
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
      const int r = i / kUT, uu = i % kUT, b = b0 + r, u = u0 + uu;
      if (b >= B || u >= H || !info[4 * r + 2]) continue;
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
      const int par = info[4 * r + 1];
      const float hprev = par < 0 ? __ldg(p.h0 + static_cast<size_t>(b) * H + u)
                                  : __ldcg(p.hs + (static_cast<size_t>(b) * n + par) * H + u);
      p.hs[(static_cast<size_t>(b) * n + node) * H + u] = (1.f - zg) * ng + zg * hprev;
    }
  }
}

// ---- phase B: expand, merge, pop (one CTA per request) ----------------------------------------------------------
// A CTA owns requests blockIdx.x, blockIdx.x + G, ... for the whole launch; the states of its first kSlots requests
// stay in shared memory between steps, and after each step it asks L2 for what the next step of those requests
// reads (the popped token's embedding row, the correction rows of the popped node's block position) while it waits
// at the grid barrier.
constexpr int kSlots = 8;

struct OwnedState {
  NodeState st[kSlots];
  int pf_token[kSlots];  // embedding row to prefetch, -1 for none
  int pf_pos[kSlots];    // offset of the candidate row in ids/vals to prefetch the correction rows of, -1 for none
};

// Shared memory of the frontier phase: [H] hidden state, [M4] logits, [M4] base logits, [M4] ids, 2 x [n + M]
// entries, then (when it fits) the node's M gathered W_c rows.
__host__ __device__ inline int round4(int x) { return (x + 3) & ~3; }
__host__ __device__ inline size_t frontier_rows_offset(int M, int n, int H) {
  return align_up(sizeof(float) * (H + 3 * round4(M)) + 2 * sizeof(Entry) * static_cast<size_t>(n + M), 16);
}
constexpr size_t kFrontierRowsCap = 160 * 1024;  // gathered rows kept in shared memory up to this size

__device__ void frontier_phase(const Params& p, int s, unsigned char* smem, OwnedState* own) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int M = p.M, n = p.n, H = p.H, M4 = round4(M);
  const size_t esize = p.bf16 ? 2 : 4;
  float* h = reinterpret_cast<float*>(smem);                   // [H]
  float* z = h + H;                                            // [M4]
  float* vals = z + M4;                                        // [M4]
  int* ids = reinterpret_cast<int*>(vals + M4);                // [M4]
  Entry* cand = reinterpret_cast<Entry*>(ids + M4);            // [n + M]
  Entry* sorted = cand + (n + M);                              // [n + M]
  unsigned char* rows = smem + frontier_rows_offset(M, n, H);  // [M][H]
  const bool rows_in_smem = p.rows_smem;
  __shared__ float s_red[2];
  int slot = 0;
  for (int b = blockIdx.x; b < p.B; b += gridDim.x, ++slot) {
    __syncthreads();
    NodeState st;
    bool expand;
    int node_depth, parent_idx;
    float node_score;
    const float* hsrc;
    if (s == 0) {
      expand = true;
      node_depth = 0;
      parent_idx = -1;
      node_score = 0.f;
      hsrc = p.h0 + static_cast<size_t>(b) * H;
      st.seq_next = 0;
      st.fcount = 0;
    } else {
      st = slot < kSlots ? own->st[slot] : p.state[b];
      expand = st.expand != 0;
      node_depth = st.depth;
      parent_idx = s - 1;
      node_score = st.score;
      hsrc = p.hs + (static_cast<size_t>(b) * n + (s - 1)) * H;
    }
    const int F = st.fcount;
    const int C = expand ? M : 0;
    Entry* fr = p.frontier + static_cast<size_t>(b) * n;
    const size_t pos = (static_cast<size_t>(b) * p.K + node_depth) * M;
    // first wave: everything whose address is known (state, ids, base logits, frontier), one latency
    for (int i = t; i < F; i += kThreads) cp_async16(cand + i, fr + i);
    if (expand) {
      for (int k = t; k < H / 4; k += kThreads) cp_async16(h + 4 * k, hsrc + 4 * k);
      for (int m = t; m < M; m += kThreads) {
        cp_async4(ids + m, p.ids + pos + m);
        cp_async4(vals + m, p.vals + pos + m);
      }
    }
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    if (expand) {
      for (int m = t; m < M; m += kThreads) ids[m] = valid_id(p, ids[m]);
      __syncthreads();
      if (rows_in_smem) {  // second wave: the M correction rows (L2 hits when the previous step prefetched them)
        const int pieces = static_cast<int>(H * esize / 16);
        for (int i = t; i < M * pieces; i += kThreads) {
          const int m = i / pieces, q = i % pieces;
          cp_async16(rows + (static_cast<size_t>(m) * pieces + q) * 16,
                     static_cast<const char*>(p.w_c) + (static_cast<size_t>(ids[m]) * pieces + q) * 16);
        }
        cp_async_commit();
        cp_async_wait_all();
        __syncthreads();
      }
      for (int m0 = warp * 8; m0 < M; m0 += kWarps * 8) {  // each warp: 8 consecutive rows at a time
        float d[8];
        warp_dot_rows8(rows_in_smem ? rows : nullptr, p.w_c, ids, p.bf16, m0, M, h, H, d);
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
        Entry e;
        e.score = node_score + ((z[m] - mx) - lse);
        e.token = ids[m];
        e.parent = static_cast<short>(parent_idx);
        e.depth = static_cast<short>(node_depth + 1);
        e.seq = st.seq_next + m;
        cand[F + m] = e;
      }
    }
    __syncthreads();
    // Keep the R = n - s best (nothing ranked below them can be popped in the n - s pops left): the sorted
    // frontier merged with the ranked children (sorted[n, n + M) is free: R <= n).
    const int N = F + C;
    const int R = min(n - s, N);
    merge_rank<kThreads>(cand, F, C, R, sorted + n, sorted);
    const Entry pop = sorted[0];
    for (int i = t + 1; i < R; i += kThreads) fr[i - 1] = sorted[i];
    const size_t o = static_cast<size_t>(b) * n + s;
    uint8_t* mrow = p.mask + o * n;
    const uint8_t* prow = pop.parent >= 0 ? p.mask + (static_cast<size_t>(b) * n + pop.parent) * n : nullptr;
    for (int j = t; j < n; j += kThreads) mrow[j] = (j == s) ? 1 : ((j < s && prow) ? prow[j] : 0);
    if (t == 0) {
      p.tokens[o] = pop.token;
      p.parents[o] = pop.parent;
      p.depth[o] = pop.depth;
      p.scores[o] = pop.score;
      NodeState ns;
      ns.token = pop.token;
      ns.parent = pop.parent;
      ns.depth = pop.depth;
      ns.expand = (s + 1 < n) && (pop.depth < p.max_depth);
      ns.score = pop.score;
      ns.seq_next = st.seq_next + C;
      ns.fcount = R - 1;
      ns.pad = 0;
      p.state[b] = ns;
      if (slot < kSlots) {
        own->st[slot] = ns;
        own->pf_token[slot] = ns.expand ? ns.token : -1;
        own->pf_pos[slot] = ns.expand ? static_cast<int>((static_cast<size_t>(b) * p.K + ns.depth) * M) : -1;
      }
    }
  }
}

// Runs between arriving at and waiting on the grid barrier that ends step s: the owned requests' next reads go to
// L2 (warps 1.., so that thread 0 can poll the barrier). Pure hints: nothing waits for them.
__device__ void prefetch_next(const Params& p, const OwnedState* own) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int owned = p.B > static_cast<int>(blockIdx.x) ? (p.B - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
  const unsigned esize = p.bf16 ? 2u : 4u;
  for (int slot = warp - 1; slot >= 0 && slot < min(owned, kSlots); slot += kWarps - 1) {
    const int tok = own->pf_token[slot], pos = own->pf_pos[slot];
    if (pos < 0) continue;
    if (lane == 0)
      prefetch_l2(static_cast<const char*>(p.emb) + static_cast<size_t>(tok) * p.E * esize, p.E * esize);
    for (int m = lane; m < p.M; m += 32) {
      const int id = __ldg(p.ids + pos + m);
      if (static_cast<unsigned>(id) < static_cast<unsigned>(p.V))
        prefetch_l2(static_cast<const char*>(p.w_c) + static_cast<size_t>(id) * p.H * esize, p.H * esize);
    }
  }
}

// kGemm: 0 = CUDA-core GRU tiles (fp32 weights or widths not multiples of 128), tensor cores with 1 = TileS,
// 2 = TileL, 3 = TileS128.
template <int kGemm>
__global__ void __launch_bounds__(kThreads, 1) build_kernel(Params p) {
  extern __shared__ float4 smem_f4[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(smem_f4);
  __shared__ int s_flag;
  __shared__ unsigned long long s_base;
  __shared__ OwnedState own;
  const unsigned G = gridDim.x;
  if (threadIdx.x == 0) s_base = ld_relaxed_gpu_u64(&p.hdr->sync_count);  // before anyone can pass this barrier
  if (!grid_barrier(p.hdr, G, p.timeout_ns, &s_flag)) return;
  unsigned long long target = s_base;
  for (int s = 0; s < p.n; ++s) {
    if (s > 0) {
      if (kGemm == 1) gemm_gru_phase<TileS, 32, 8>(p, s - 1, smem);
      else if (kGemm == 2) gemm_gru_phase<TileL, 64, 16>(p, s - 1, smem);
      else if (kGemm == 3) gemm_gru_phase<TileS128, 32, 8>(p, s - 1, smem);
      else gru_phase(p, s - 1, reinterpret_cast<float*>(smem));
      target += G;
      if (!counter_barrier(p.hdr, target, p.timeout_ns, &s_flag)) return;
    }
    frontier_phase(p, s, smem, &own);
    if (s + 1 < p.n) {
      counter_arrive(p.hdr);
      prefetch_next(p, &own);
      target += G;
      if (!counter_wait(p.hdr, target, p.timeout_ns, &s_flag)) return;
    }
  }
}

// Dynamic shared memory of the large-batch kernel; the gathered rows are staged only when they fit under both the
// cap and the device's opt-in limit (`rows_smem` reports the choice).
size_t smem_bytes(int gemm, int M, int n, int H, size_t esize, size_t optin, bool* rows_smem) {
  size_t a = sizeof(float) * (kTB * kPad + 3 * kTU * kPad);
  if (gemm == 1) a = TileS::kBytes;
  if (gemm == 2) a = TileL::kBytes;
  if (gemm == 3) a = TileS128::kBytes;
  const size_t rows = static_cast<size_t>(M) * H * esize;
  const size_t base = frontier_rows_offset(M, n, H);
  *rows_smem = rows <= kFrontierRowsCap && base + rows <= optin;
  const size_t b = base + (*rows_smem ? rows : 0);
  return a > b ? a : b;
}

}  // namespace
}  // namespace dt

extern "C" size_t dt_build_workspace_bytes(int B, int K, int V, int M, int n, int H, int E) {
  (void)E;
  if (B < 0 || K < 1 || V < 1 || M < 1 || n < 1 || H < 1) return 0;
  return dt::build_layout(B, K, V, M, n, H).bytes;
}

extern "C" dt_status dt_build_trees(int B, int K, int V, int M, int n, int max_depth, float T,
                                    const int32_t* topm_ids, const float* topm_vals, const float* h0,
                                    const dt_weights* w, int32_t* out_tokens, int32_t* out_parents,
                                    int32_t* out_depth, float* out_scores, uint8_t* out_mask, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream) {
  using namespace dt;
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
  const BuildLayout L = build_layout(B, K, V, M, n, H);
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
  p.state = reinterpret_cast<NodeState*>(ws + L.state);
  p.frontier = reinterpret_cast<Entry*>(ws + L.frontier);
  p.hs = reinterpret_cast<float*>(ws + L.hs);
  p.acc = B <= kSmallMaxB ? reinterpret_cast<long long*>(ws + L.acc) : nullptr;
  p.hs_count = B <= kSmallMaxB ? reinterpret_cast<int*>(ws + L.hs_count) : nullptr;
  p.acc_stride = acc_stride(M, n);
  p.xslots = expansion_slots(n);
  p.timeout_ns = barrier_timeout_ns();
  {  // expansions per request per wave: the setting, else as many as the small-batch builder's wave holds
    const int k = lookahead_setting();
    const int fit = kWaveJobs / (B < kWaveJobs ? B : kWaveJobs);
    p.lookahead = k > 0 ? (k < fit ? k : fit) : fit;
  }

  // phase A: tensor cores for bf16 weights whose widths are multiples of the 128-column pipeline chunk
  const int gemm = !p.bf16 ? 0
                   : B >= 128 ? (E % TileL::kKc == 0 && H % TileL::kKc == 0 ? 2 : 0)
                   : E % TileS::kKc == 0 && H % TileS::kKc == 0 ? 1
                   : E % TileS128::kKc == 0 && H % TileS128::kKc == 0 ? 3 : 0;
  const void* fn = gemm == 0 ? reinterpret_cast<const void*>(build_kernel<0>)
                             : gemm == 3 ? reinterpret_cast<const void*>(build_kernel<3>)
                             : gemm == 1 ? reinterpret_cast<const void*>(build_kernel<1>)
                                         : reinterpret_cast<const void*>(build_kernel<2>);
  DeviceInfo di{};
  if (current_device_info(&di) != cudaSuccess) return DT_ERR_CUDA;
  if (!di.coop) return DT_ERR_UNSUPPORTED;
  if (small_builder_fits(p, di)) return cuda_status(launch_small_builder(p, di, stream));
  // static shared memory of the kernel (flags, reductions) is well under 1 KB; one CTA per SM (launch bounds), so
  // the shared memory alone decides whether a CTA fits
  const size_t smem = smem_bytes(gemm, M, n, H, p.bf16 ? 2 : 4, static_cast<size_t>(di.optin) - 1024, &p.rows_smem);
  if (smem + 1024 > static_cast<size_t>(di.optin)) return DT_ERR_UNSUPPORTED;
  if (ensure_dynamic_smem(fn, smem) != cudaSuccess) return DT_ERR_CUDA;
  const unsigned grid = static_cast<unsigned>(di.sms);  // one CTA per SM; co-resident under a cooperative launch
  void* args[] = {&p};
  return cuda_status(cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kThreads), args, smem, stream));
}
