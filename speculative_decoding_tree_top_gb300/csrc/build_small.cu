// dt_build_trees for small batches (B <= 8): every SM works on every request; no grid barrier between steps.
//
// Method: blog.captcha.la, "Methodology — deep read" (best-first max-priority queue keyed by cumulative conditional
// log-probability; GRU state carried along each root-to-node path; correction only on the gathered top-M rows);
// gist.science, "Composants Clés" (only the light GRU correction and its head are recomputed per node).
//
// GB300 design. With one or a few requests the round is a chain of n dependent steps (pop -> GRU -> correction ->
// softmax -> pop), so the design minimises the latency of one step, not the bytes:
//   * weight-stationary: CTA j of the G = min(#SMs, H) CTAs owns hidden units [j*H/G, (j+1)*H/G) and keeps the
//     3 gate rows of W_ih and W_hh of those units in shared memory for the whole launch (9.4 MB of GRU weights
//     spread over 152 SMs: ~62 KB each at E=2560, H=512), plus the same units' columns of W_c for every candidate
//     of every position, the candidate ids and base logits (gathered once at launch);
//   * per step each CTA runs its slice of the GRU for the popped node (K-split over 512 threads: each thread reads its
//     slice of the input once and applies it to all gate rows; a recursive-halving shuffle reduce-scatter finishes
//     the sums), then its units' share of every candidate's correction W_c[id]·h;
//   * that share goes into a per-step, per-candidate 64-bit accumulator as ((fixed-point value << 8) + 1): integer
//     addition is associative (the reduction over CTAs is exact and bit-identical run to run) and never carries into
//     the low byte, which therefore counts the contributions. A CTA knows the correction of candidate m is complete
//     when that count reaches G: the slot is its own barrier, so there is no grid barrier between steps;
//   * every CTA then finishes the step for every request: corrected logits, restricted log-softmax (one warp), merge
//     of the children into the frontier kept in shared memory (rank by counting spread over the CTA, pruned to the
//     n - s that can still be popped), pop. All CTAs reach the same pop, so nothing needs publishing; CTA 0 writes the
//     outputs. The embedding row of the popped token is fetched with cp.async as soon as the pop is known;
//   * the new node's hidden state, written unit by unit by all CTAs, is published unit by unit with release
//     reductions on a counter and pulled into every CTA's shared-memory cache with cp.async, off the critical path;
//   * the embedding rows of all candidates are prefetched into L2 at launch.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "build_common.cuh"

namespace dt {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr uint64_t kCopyBudgetNs = 4000000000ull;  // the weight copies take microseconds: this stops a lost one
constexpr int kMaxRows = 16;  // gate rows per CTA, one warp each (3 * units <= 16 warps)
constexpr int kRowPad = 8;    // elements of padding per shared-memory weight row (16 bytes)

struct ReqState {  // a request's frontier bookkeeping, replicated in every CTA
  int fcount;
  int seq_next;
  int token;   // the node popped last
  int parent;
  int depth;
  int expand;
  float score;
  int pad;
};

// Shared-memory plan of one CTA (identical on host and device).
struct Plan {
  int G, umax, R;
  size_t wih, whh, bias, wc, xe, xh, req, fr, scr, z, hb, gates, ids, vals, par, hc, bytes;
};

__host__ __device__ inline size_t take(size_t& o, size_t bytes) {
  const size_t at = o;
  o = (o + bytes + 15) / 16 * 16;
  return at;
}

__host__ __device__ inline Plan make_plan(int B, int M, int n, int max_depth, int H, int E, int esize, int G) {
  Plan P{};
  P.G = G;
  P.umax = (H + G - 1) / G;
  P.R = 3 * P.umax;
  size_t o = 0;
  P.wih = take(o, static_cast<size_t>(esize) * P.R * (E + kRowPad));
  P.whh = take(o, static_cast<size_t>(esize) * P.R * (H + kRowPad));
  P.bias = take(o, sizeof(float) * 2 * P.R);
  P.wc = take(o, static_cast<size_t>(esize) * B * max_depth * M * P.umax);
  P.xe = take(o, static_cast<size_t>(esize) * B * E);  // embedding row of each request's popped token, as stored
  P.xh = take(o, sizeof(float) * H);                   // parent hidden state of the request being stepped
  P.req = take(o, sizeof(ReqState) * B);
  P.fr = take(o, sizeof(Entry) * B * n);
  P.scr = take(o, sizeof(Entry) * 2 * (n + M));
  P.z = take(o, sizeof(float) * M);
  P.hb = take(o, sizeof(float) * P.umax);
  P.gates = take(o, sizeof(float) * 2 * P.R);
  P.ids = take(o, sizeof(int) * B * max_depth * M);
  P.vals = take(o, sizeof(float) * B * max_depth * M);
  P.par = take(o, sizeof(short) * B * n);
  P.hc = take(o, sizeof(float) * B * n * H);
  P.bytes = o;
  return P;
}

template <bool kBf16>
struct WT {
  using T = typename std::conditional<kBf16, unsigned short, float>::type;
  __device__ static __forceinline__ float f(T v) {
    if (kBf16) return __uint_as_float(static_cast<uint32_t>(v) << 16);
    return static_cast<float>(v);
  }
};

// Asynchronous global -> shared copy of `bytes` (a multiple of 16, both ends 16-byte aligned), L2 only.
__device__ __forceinline__ void copy16_async(void* dst, const void* src, size_t bytes) {
  for (size_t i = threadIdx.x; i < bytes / 16; i += kThreads) {
    const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(static_cast<char*>(dst) + 16 * i));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(static_cast<const char*>(src) + 16 * i)
                 : "memory");
  }
}

__device__ __forceinline__ long long ld_relaxed_s64(const long long* p) {
  long long v;
  asm volatile("ld.relaxed.gpu.global.s64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Polls until `pred(load())` holds, within the launch's time budget; false (and the abort word raised) when the
// budget runs out or another CTA already gave up.
template <typename Load, typename Pred>
__device__ __forceinline__ bool poll(const Params& p, Load load, Pred pred) {
  if (pred(load())) return true;
  const uint64_t t0 = global_timer_ns();
  unsigned polls = 0;
  while (true) {
    if (pred(load())) return true;
    if ((++polls & 15u) == 0u &&
        (ld_acquire_gpu(&p.hdr->abort) != 0u || global_timer_ns() - t0 > p.timeout_ns || p.timeout_ns == 0)) {
      record_error(p.hdr, DT_ERR_TIMEOUT);
      atomicExch(&p.hdr->abort, 1u);
      return false;
    }
  }
}

// Correction accumulators: every CTA adds (round(v * 2^32) << 8) + 1 to the slot of each candidate. The upper 56
// bits hold the exact fixed-point sum, the low byte the number of contributions (G < 256).
constexpr float kFix = 4294967296.0f;              // 2^32
constexpr float kUnfix = 2.3283064365386963e-10f;  // 2^-32
constexpr float kMaxShare = 32768.0f;              // |share| bound: 255 shares still fit in 56 bits

__device__ __forceinline__ void add_share(const Params& p, long long* slot, float v) {
  if (!(fabsf(v) < kMaxShare)) {  // also catches NaN
    record_error(p.hdr, DT_ERR_NUMERIC);
    v = 0.f;
  }
  const unsigned long long c = (static_cast<unsigned long long>(__float2ll_rn(v * kFix)) << 8) + 1ull;
  atomicAdd(reinterpret_cast<unsigned long long*>(slot), c);
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads, 1) small_builder(Params p, Plan P) {
  using T = typename WT<kBf16>::T;
  extern __shared__ __align__(16) unsigned char smem[];
  T* wih = reinterpret_cast<T*>(smem + P.wih);               // [R][E + pad], row g*umax + u
  T* whh = reinterpret_cast<T*>(smem + P.whh);               // [R][H + pad]
  float* bias = reinterpret_cast<float*>(smem + P.bias);     // [R][2]: b_ih, b_hh
  T* wc = reinterpret_cast<T*>(smem + P.wc);                 // [B][max_depth][M][umax]
  T* xe = reinterpret_cast<T*>(smem + P.xe);                 // [B][E]
  float* xh = reinterpret_cast<float*>(smem + P.xh);         // [H]
  ReqState* rs = reinterpret_cast<ReqState*>(smem + P.req);  // [B]
  Entry* fr = reinterpret_cast<Entry*>(smem + P.fr);         // [B][n]
  Entry* cand = reinterpret_cast<Entry*>(smem + P.scr);      // [n + M]
  Entry* sorted = cand + (p.n + p.M);                        // [n + M]
  float* z = reinterpret_cast<float*>(smem + P.z);           // [M]
  float* hb = reinterpret_cast<float*>(smem + P.hb);         // [umax]: the new hidden state of the owned units
  float* gates = reinterpret_cast<float*>(smem + P.gates);   // [R][2]: input side, hidden side
  int* ids_s = reinterpret_cast<int*>(smem + P.ids);         // [B][max_depth][M] candidate ids (range-checked)
  float* vals_s = reinterpret_cast<float*>(smem + P.vals);   // [B][max_depth][M] candidate base logits
  short* par_s = reinterpret_cast<short*>(smem + P.par);     // [B][n]: parent of every popped node
  float* hc = reinterpret_cast<float*>(smem + P.hc);         // [B][n][H]: hidden state of every expanded node
  __shared__ int s_flag;
  __shared__ uint64_t wbar;  // completion of the weight rows' bulk copies

  const int B = p.B, K = p.K, M = p.M, n = p.n, H = p.H, E = p.E, maxd = p.max_depth;
  const int G = P.G, umax = P.umax;
  const int j = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int u0 = static_cast<int>((static_cast<long long>(j) * H) / G);
  const int nu = static_cast<int>((static_cast<long long>(j + 1) * H) / G) - u0;
  const size_t esize = kBf16 ? 2 : 4;
  const int AS = p.acc_stride;
  int* hs_count = reinterpret_cast<int*>(p.acc + static_cast<size_t>(n) * B * M * AS);  // [B][n]

  // ---- launch: weights of the owned units, W_c columns / ids / base logits of the candidates, L2 prefetch ----
  const int SE = E + kRowPad, SH = H + kRowPad;  // shared-memory row strides of W_ih and W_hh
  // The 3 * nu rows of W_ih and of W_hh as bulk copies (1 to 8 KB each) completing on one mbarrier, issued by warp 0;
  // waited for at the top of the first step.
  if (t == 0) {
    mbar_init(&wbar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (warp == 0) {
    if (lane == 0) mbar_expect_tx(&wbar, static_cast<unsigned>(3 * nu * (E + H) * esize));
    __syncwarp();
    for (int q = lane; q < 6 * nu; q += 32) {
      const bool hid = q >= 3 * nu;
      const int qq = hid ? q - 3 * nu : q, g = qq / nu, u = qq % nu, r = g * umax + u;
      const size_t row = static_cast<size_t>(g) * H + u0 + u;
      if (hid)
        bulk_g2s(whh + static_cast<size_t>(r) * SH, static_cast<const char*>(p.w_hh) + row * H * esize,
                 static_cast<unsigned>(esize * H), &wbar);
      else
        bulk_g2s(wih + static_cast<size_t>(r) * SE, static_cast<const char*>(p.w_ih) + row * E * esize,
                 static_cast<unsigned>(esize * E), &wbar);
    }
  }
  // A return before the first step leaves no copy in flight: this waits (bounded) for the weights.
  auto drain = [&]() {
    asm volatile("cp.async.wait_all;" ::: "memory");
    mbar_wait(&wbar, 0, kCopyBudgetNs);
  };
  for (int i = t; i < 3 * umax; i += kThreads) {
    const int g = i / umax, u = i % umax;
    const size_t row = static_cast<size_t>(g) * H + u0 + u;
    bias[2 * i] = (u < nu && p.b_ih) ? ldw(p.b_ih, kBf16, row) : 0.f;
    bias[2 * i + 1] = (u < nu && p.b_hh) ? ldw(p.b_hh, kBf16, row) : 0.f;
  }
  // candidate ids and base logits of every (request, position) first, then the owned units' W_c columns of every
  // candidate, all independent loads
  for (int i = t; i < B * maxd * M; i += kThreads) {
    const int b = i / (maxd * M), pos = (i / M) % maxd, m = i % M;
    const size_t gi = (static_cast<size_t>(b) * K + pos) * M + m;
    ids_s[i] = valid_id(p, __ldg(p.ids + gi));
    vals_s[i] = __ldg(p.vals + gi);
  }
  __syncthreads();
#pragma unroll 8
  for (int q = t; q < B * maxd * M * umax; q += kThreads) {
    const int i = q / umax, u = q % umax;
    wc[q] = u < nu ? static_cast<const T*>(p.w_c)[static_cast<size_t>(ids_s[i]) * H + u0 + u] : T(0);
  }
  {
    const size_t row_bytes = static_cast<size_t>(E) * esize;
    const size_t lines = (row_bytes + 127) / 128;
    const size_t total = static_cast<size_t>(B) * maxd * M * lines;
    for (size_t i = static_cast<size_t>(j) * kThreads + t; i < total; i += static_cast<size_t>(G) * kThreads) {
      const size_t c = i / lines, line = i % lines;
      const int b = static_cast<int>(c / (maxd * M)), pos = static_cast<int>((c / M) % maxd);
      const int m = static_cast<int>(c % M);
      const int id = __ldg(p.ids + (static_cast<size_t>(b) * K + pos) * M + m);
      if (static_cast<unsigned>(id) < static_cast<unsigned>(p.V)) {
        const char* a = static_cast<const char*>(p.emb) + static_cast<size_t>(id) * row_bytes + line * 128;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
      }
    }
  }
  // every step's accumulators and the hidden-state counters start at zero; one grid barrier orders that
  const size_t zero_words = static_cast<size_t>(n) * B * M * AS + (static_cast<size_t>(B) * n + 1) / 2;
  for (size_t i = static_cast<size_t>(j) * kThreads + t; i < zero_words; i += static_cast<size_t>(G) * kThreads)
    p.acc[i] = 0;
  for (int b = t; b < B; b += kThreads) rs[b] = ReqState{};
  if (!grid_barrier(p.hdr, G, p.timeout_ns, &s_flag)) {
    drain();
    return;
  }

  if (!mbar_wait(&wbar, 0, kCopyBudgetNs)) record_error(p.hdr, DT_ERR_TIMEOUT);  // the weight rows (bounded)
  for (int s = 0; s < n; ++s) {
    asm volatile("cp.async.wait_all;" ::: "memory");  // this thread's cache and embedding copies
    __syncthreads();                                   // ... and everyone else's
    long long* acc_s = p.acc + static_cast<size_t>(s) * B * M * AS;

    // ---- phase A: this CTA's share of the GRU and of the correction of every expanding request ----
    for (int b = 0; b < B; ++b) {
      const bool root = s == 0;
      if (!root && !rs[b].expand) continue;  // uniform across the CTA (replicated state)
      const int pos = root ? 0 : rs[b].depth;
      if (root) {
        for (int u = t; u < nu; u += kThreads) hb[u] = __ldg(p.h0 + static_cast<size_t>(b) * H + u0 + u);
      } else {
        const int par = rs[b].parent;
        const float* xhp = xh;  // the parent's hidden state: the cached copy, or h0 staged for a child of the root
        if (par < 0) {
          for (int k = t; k < H / 4; k += kThreads)
            reinterpret_cast<float4*>(xh)[k] =
                __ldg(reinterpret_cast<const float4*>(p.h0 + static_cast<size_t>(b) * H) + k);
          __syncthreads();
        } else {
          xhp = hc + (static_cast<size_t>(b) * n + par) * H;
        }
        const T* xeb = xe + static_cast<size_t>(b) * E;
        const int R = 3 * umax;
        if (warp < R) {
          // One warp per gate row (R <= 16 rows, 16 warps): the lanes stride over K with four independent
          // accumulators per side, then one shuffle tree per side. The row's input side (over E) and hidden side
          // (over H) stay apart: the n gate needs them separately.
          const int r = warp;
          constexpr int kPer = kBf16 ? 8 : 4;
          float ai[4] = {0.f, 0.f, 0.f, 0.f}, ah[4] = {0.f, 0.f, 0.f, 0.f};
          const T* wr = wih + static_cast<size_t>(r) * SE;
#pragma unroll 4
          for (int f = lane; f < E / kPer; f += 32) {
            const int c = f * kPer;
            if (kBf16) {
              const uint4 w = *reinterpret_cast<const uint4*>(wr + c), q = *reinterpret_cast<const uint4*>(xeb + c);
              ai[0] = fmaf(__uint_as_float(w.x << 16), __uint_as_float(q.x << 16), ai[0]);
              ai[1] = fmaf(__uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(q.x & 0xFFFF0000u), ai[1]);
              ai[2] = fmaf(__uint_as_float(w.y << 16), __uint_as_float(q.y << 16), ai[2]);
              ai[3] = fmaf(__uint_as_float(w.y & 0xFFFF0000u), __uint_as_float(q.y & 0xFFFF0000u), ai[3]);
              ai[0] = fmaf(__uint_as_float(w.z << 16), __uint_as_float(q.z << 16), ai[0]);
              ai[1] = fmaf(__uint_as_float(w.z & 0xFFFF0000u), __uint_as_float(q.z & 0xFFFF0000u), ai[1]);
              ai[2] = fmaf(__uint_as_float(w.w << 16), __uint_as_float(q.w << 16), ai[2]);
              ai[3] = fmaf(__uint_as_float(w.w & 0xFFFF0000u), __uint_as_float(q.w & 0xFFFF0000u), ai[3]);
            } else {
              const float4 w = *reinterpret_cast<const float4*>(wr + c), q = *reinterpret_cast<const float4*>(xeb + c);
              ai[0] = fmaf(w.x, q.x, ai[0]);
              ai[1] = fmaf(w.y, q.y, ai[1]);
              ai[2] = fmaf(w.z, q.z, ai[2]);
              ai[3] = fmaf(w.w, q.w, ai[3]);
            }
          }
          const T* hr = whh + static_cast<size_t>(r) * SH;
#pragma unroll 4
          for (int f = lane; f < H / kPer; f += 32) {
            const int c = f * kPer;
            const float4 x0 = *reinterpret_cast<const float4*>(xhp + c);
            if (kBf16) {
              const float4 x1 = *reinterpret_cast<const float4*>(xhp + c + 4);
              const uint4 w = *reinterpret_cast<const uint4*>(hr + c);
              ah[0] = fmaf(__uint_as_float(w.x << 16), x0.x, ah[0]);
              ah[1] = fmaf(__uint_as_float(w.x & 0xFFFF0000u), x0.y, ah[1]);
              ah[2] = fmaf(__uint_as_float(w.y << 16), x0.z, ah[2]);
              ah[3] = fmaf(__uint_as_float(w.y & 0xFFFF0000u), x0.w, ah[3]);
              ah[0] = fmaf(__uint_as_float(w.z << 16), x1.x, ah[0]);
              ah[1] = fmaf(__uint_as_float(w.z & 0xFFFF0000u), x1.y, ah[1]);
              ah[2] = fmaf(__uint_as_float(w.w << 16), x1.z, ah[2]);
              ah[3] = fmaf(__uint_as_float(w.w & 0xFFFF0000u), x1.w, ah[3]);
            } else {
              const float4 w = *reinterpret_cast<const float4*>(hr + c);
              ah[0] = fmaf(w.x, x0.x, ah[0]);
              ah[1] = fmaf(w.y, x0.y, ah[1]);
              ah[2] = fmaf(w.z, x0.z, ah[2]);
              ah[3] = fmaf(w.w, x0.w, ah[3]);
            }
          }
          float si = (ai[0] + ai[1]) + (ai[2] + ai[3]), sh = (ah[0] + ah[1]) + (ah[2] + ah[3]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            si += __shfl_xor_sync(0xFFFFFFFFu, si, o);
            sh += __shfl_xor_sync(0xFFFFFFFFu, sh, o);
          }
          if (lane == 0) {
            gates[2 * r] = si;
            gates[2 * r + 1] = sh;
          }
        }
        __syncthreads();
        for (int u = t; u < nu; u += kThreads) {
          const int rr = u, rz = umax + u, rn = 2 * umax + u;
          const float r = sigmoidf_(gates[2 * rr] + bias[2 * rr] + gates[2 * rr + 1] + bias[2 * rr + 1]);
          const float zg = sigmoidf_(gates[2 * rz] + bias[2 * rz] + gates[2 * rz + 1] + bias[2 * rz + 1]);
          const float g = tanhf(gates[2 * rn] + bias[2 * rn] + r * (gates[2 * rn + 1] + bias[2 * rn + 1]));
          hb[u] = (1.f - zg) * g + zg * xhp[u0 + u];
        }
      }
      __syncthreads();
      if (!root && warp == kWarps - 1) {  // publish the new units (the last warp polls nothing in phase C)
        for (int u = lane; u < nu; u += 32) {
          p.hs[(static_cast<size_t>(b) * n + (s - 1)) * H + u0 + u] = hb[u];
          // a release reduction orders the store above before the count (H units in all)
          asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(hs_count + static_cast<size_t>(b) * n + (s - 1))
                       : "memory");
        }
      }
      // this CTA's units' part of W_c[id]·h for the M candidates of position pos
      const T* wcp = wc + (static_cast<size_t>(b) * maxd + pos) * M * umax;
      for (int m = t; m < M; m += kThreads) {
        float v = 0.f;
        for (int u = 0; u < nu; ++u) v = fmaf(WT<kBf16>::f(wcp[static_cast<size_t>(m) * umax + u]), hb[u], v);
        add_share(p, acc_s + (static_cast<size_t>(b) * M + m) * AS, v);
      }
      if (B > 1) __syncthreads();  // gates / xh are reused by the next request
    }

    // ---- phase C: every CTA finishes the step for every request (the whole CTA on one request at a time) ----
    for (int b = 0; b < B; ++b) {
      const ReqState st = rs[b];
      const int F = st.fcount;
      const bool expanded = s == 0 || st.expand;
      const int C = expanded ? M : 0;
      const int pos = s == 0 ? 0 : st.depth;
      const size_t off = (static_cast<size_t>(b) * maxd + pos) * M;  // into the staged ids / base logits
      for (int i = t; i < F; i += kThreads) cand[i] = fr[static_cast<size_t>(b) * n + i];
      int ok = 1;
      if (expanded && warp == 0) {
        // All G shares of every candidate: each lane polls its slots (each on its own cache line) until all are
        // complete, every slot read of a round in flight together, then takes the corrected logits.
        auto complete = [&](long long v) { return (v & 0xFF) == (G & 0xFF); };
        const long long* slots = acc_s + static_cast<size_t>(b) * M * AS;
        float mx = -INFINITY;
        for (int m0 = lane; m0 < M; m0 += 128) {
          long long a[4];
          bool done = false;
          const uint64_t t0 = global_timer_ns();
          for (unsigned polls = 0; !done; ++polls) {
            done = true;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int m = m0 + 32 * j;
              a[j] = m < M ? ld_relaxed_s64(slots + static_cast<size_t>(m) * AS) : static_cast<long long>(G & 0xFF);
              done &= complete(a[j]);
            }
            if (!done && (polls & 15u) == 15u &&
                (ld_acquire_gpu(&p.hdr->abort) != 0u || global_timer_ns() - t0 > p.timeout_ns)) {
              record_error(p.hdr, DT_ERR_TIMEOUT);
              atomicExch(&p.hdr->abort, 1u);
              ok = 0;
              break;
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int m = m0 + 32 * j;
            if (m >= M) break;
            const float v = (vals_s[off + m] + __ll2float_rn(a[j] >> 8) * kUnfix) / p.T_eff;
            z[m] = v;
            mx = fmaxf(mx, v);
          }
        }
        ok = __all_sync(0xFFFFFFFFu, ok);
        // restricted log-softmax of this node's children, in the warp
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        float sum = 0.f;
        for (int m = lane; m < M; m += 32) sum += expf(z[m] - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        const float lse = logf(sum);
        const float base_score = s == 0 ? 0.f : st.score;
        for (int m = lane; m < M; m += 32) {
          Entry e;
          e.score = base_score + ((z[m] - mx) - lse);
          e.token = ids_s[off + m];
          e.parent = static_cast<short>(s == 0 ? -1 : s - 1);
          e.depth = static_cast<short>(pos + 1);
          e.seq = st.seq_next + m;
          cand[F + m] = e;
        }
      }
      if (expanded && s > 0 && warp == kWarps - 1) {
        // the expanded node's full hidden state (published unit by unit by every CTA) into this CTA's cache,
        // asynchronously (waited for at the next step)
        const int* cnt = hs_count + static_cast<size_t>(b) * n + (s - 1);
        if (lane == 0)
          ok &= poll(p, [&] { return static_cast<long long>(ld_acquire_gpu(reinterpret_cast<const unsigned*>(cnt))); },
                     [&](long long v) { return v >= H; });
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (ok) {
          const float* src = p.hs + (static_cast<size_t>(b) * n + (s - 1)) * H;
          float* dst = hc + (static_cast<size_t>(b) * n + (s - 1)) * H;
          for (int k = lane; k < H / 4; k += 32) {
            const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst + 4 * k));
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src + 4 * k) : "memory");
          }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
      }
      if (!__syncthreads_and(ok)) {  // a wait ran out (recorded): leave with no copy in flight
        asm volatile("cp.async.wait_all;" ::: "memory");
        return;
      }
      // Keep the R = n - s best (nothing ranked below them can be popped in the n - s pops left): the sorted
      // frontier merged with the ranked children.
      const int N = F + C;
      const int R = min(n - s, N);
      merge_rank<kThreads>(cand, F, C, R, sorted + n, sorted);
      if (N == 0 && t == 0) {  // unreachable when n <= the size of the depth-limited tree (checked on the host)
        record_error(p.hdr, DT_ERR_INVALID_ARG);
        sorted[0] = Entry{-INFINITY, 0, -1, 1, 0};
      }
      __syncthreads();
      const Entry pop = sorted[0];
      const bool will_expand = (s + 1 < n) && (pop.depth < maxd);
      if (will_expand)  // its embedding row, for the next step's GRU
        copy16_async(xe + static_cast<size_t>(b) * E,
                     static_cast<const char*>(p.emb) + static_cast<size_t>(pop.token) * E * esize, esize * E);
      asm volatile("cp.async.commit_group;" ::: "memory");
      for (int i = t + 1; i < R; i += kThreads) fr[static_cast<size_t>(b) * n + i - 1] = sorted[i];
      short* pb = par_s + static_cast<size_t>(b) * n;
      if (j == 0) {
        const size_t o = static_cast<size_t>(b) * n + s;
        uint8_t* mrow = p.mask + o * n;
        for (int c = t; c < n; c += kThreads) {  // ancestor test by walking s's parent chain (parents come first)
          int a = c < s ? pop.parent : s;
          while (a > c) a = pb[a];
          mrow[c] = a == c;
        }
        if (t == 0) {
          p.tokens[o] = pop.token;
          p.parents[o] = pop.parent;
          p.depth[o] = pop.depth;
          p.scores[o] = pop.score;
        }
      }
      if (t == 0) {  // read by others only after the next barrier
        pb[s] = pop.parent;
        ReqState ns = st;
        ns.fcount = R - 1;
        ns.seq_next += C;
        ns.token = pop.token;
        ns.parent = pop.parent;
        ns.depth = pop.depth;
        ns.score = pop.score;
        ns.expand = will_expand;
        rs[b] = ns;
      }
      if (b + 1 < B) __syncthreads();  // the next request reuses the scratch entries
    }
  }
}

int grid_size(const Params& p, int sms) { return sms < p.H ? sms : p.H; }

Plan plan_for(const Params& p, int sms) {
  return make_plan(p.B, p.M, p.n, p.max_depth, p.H, p.E, p.bf16 ? 2 : 4, grid_size(p, sms));
}

}  // namespace

bool small_builder_fits(const Params& p, int sms) {
  if (p.B > kSmallMaxB || p.B < 1 || !p.acc) return false;
  const Plan P = plan_for(p, sms);
  if (3 * P.umax > kMaxRows || P.G > 255) return false;  // GEMV rows per CTA; contribution count in one byte
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
  return P.bytes <= static_cast<size_t>(optin);
}

cudaError_t launch_small_builder(const Params& p, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const Plan P = plan_for(p, sms);
  const void* fn = p.bf16 ? reinterpret_cast<const void*>(small_builder<true>)
                          : reinterpret_cast<const void*>(small_builder<false>);
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(P.bytes));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, P.bytes);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  Params pp = p;
  Plan PP = P;
  void* args[] = {&pp, &PP};
  return cudaLaunchCooperativeKernel(fn, dim3(static_cast<unsigned>(P.G)), dim3(kThreads), args, P.bytes, stream);
}

}  // namespace dt
