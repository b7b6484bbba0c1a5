// dt_build_trees for small batches (B <= 8): every SM works on every request, one grid barrier per step.
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
//     of every position (gathered once at launch);
//   * per step each CTA runs its slice of the GRU for the popped node (one warp per gate row, 16-byte shared-memory
//     reads, fp32 accumulation), then its units' share of every candidate's correction W_c[id]·h, added into a
//     per-step accumulator as a fixed-point integer (int64, scale 2^32): integer addition is associative, so the
//     reduction over CTAs is exact and bit-identical run to run whatever the arrival order;
//   * one grid barrier; then every CTA redundantly finishes the step for every request: corrected logits,
//     restricted log-softmax (one warp), merge of the children into the frontier kept in shared memory (rank by
//     counting spread over the whole CTA, pruned to the n - s that can still be popped), pop. All CTAs reach the
//     same pop, so no second barrier is needed to publish it; CTA 0 writes the outputs;
//   * the embedding rows of all candidates are prefetched into L2 at launch.
#include <cuda_runtime.h>

#include <type_traits>

#include "build_common.cuh"

namespace dt {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

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
  size_t wih, whh, bias, wc, x, gates, hnew, req, fr, scr, z, red, ids, vals, par, hc, bytes;
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
  P.wih = take(o, static_cast<size_t>(esize) * P.R * E);
  P.whh = take(o, static_cast<size_t>(esize) * P.R * H);
  P.bias = take(o, sizeof(float) * 2 * P.R);
  P.wc = take(o, static_cast<size_t>(esize) * B * max_depth * M * P.umax);
  P.x = take(o, sizeof(float) * (E + H));
  P.gates = take(o, sizeof(float) * 2 * P.R);
  P.hnew = take(o, sizeof(float) * B * P.umax);
  P.req = take(o, sizeof(ReqState) * B);
  P.fr = take(o, sizeof(Entry) * B * n);
  P.scr = take(o, sizeof(Entry) * 2 * (n + M));
  P.z = take(o, sizeof(float) * M);
  P.red = take(o, sizeof(float) * kWarps * 32);
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

// Copies `bytes` (a multiple of 16) from global to shared memory with 16-byte loads.
__device__ __forceinline__ void copy16(void* dst, const void* src, size_t bytes) {
  const uint4* s = static_cast<const uint4*>(src);
  uint4* d = static_cast<uint4*>(dst);
#pragma unroll 8
  for (size_t i = threadIdx.x; i < bytes / 16; i += kThreads) d[i] = __ldg(s + i);
}

// a . x over `len` elements: weights in shared memory, x (fp32) in shared memory; one warp, 16-byte weight reads.
template <bool kBf16>
__device__ __forceinline__ float warp_dot(const typename WT<kBf16>::T* w, const float* x, int len) {
  const int lane = threadIdx.x & 31;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;  // independent chains: the loop is latency-, not issue-bound
  if (kBf16) {
#pragma unroll 2
    for (int c = lane; c < len / 8; c += 32) {
      const uint4 q = *reinterpret_cast<const uint4*>(w + c * 8);
      const float4 a = *reinterpret_cast<const float4*>(x + c * 8);
      const float4 b = *reinterpret_cast<const float4*>(x + c * 8 + 4);
      a0 = fmaf(__uint_as_float(q.x << 16), a.x, a0);
      a1 = fmaf(__uint_as_float(q.x & 0xFFFF0000u), a.y, a1);
      a2 = fmaf(__uint_as_float(q.y << 16), a.z, a2);
      a3 = fmaf(__uint_as_float(q.y & 0xFFFF0000u), a.w, a3);
      a0 = fmaf(__uint_as_float(q.z << 16), b.x, a0);
      a1 = fmaf(__uint_as_float(q.z & 0xFFFF0000u), b.y, a1);
      a2 = fmaf(__uint_as_float(q.w << 16), b.z, a2);
      a3 = fmaf(__uint_as_float(q.w & 0xFFFF0000u), b.w, a3);
    }
  } else {
#pragma unroll 2
    for (int c = lane; c < len / 4; c += 32) {
      const float4 q = *reinterpret_cast<const float4*>(w + c * 4);
      const float4 a = *reinterpret_cast<const float4*>(x + c * 4);
      a0 = fmaf(q.x, a.x, a0);
      a1 = fmaf(q.y, a.y, a1);
      a2 = fmaf(q.z, a.z, a2);
      a3 = fmaf(q.w, a.w, a3);
    }
  }
  float acc = (a0 + a1) + (a2 + a3);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  return acc;
}

constexpr int kMaxRows = 16;  // gate rows per CTA handled by the K-split GEMV (3 * units <= 16)

template <bool kBf16>
__device__ __forceinline__ void dot8_rows(const typename WT<kBf16>::T* w, size_t row_stride, int col, int R,
                                          const float* x8, float (&acc)[kMaxRows]) {
  constexpr int kPer = kBf16 ? 8 : 4;
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r) {
    if (r < R) {
      const typename WT<kBf16>::T* wr = w + static_cast<size_t>(r) * row_stride + col;
      if (kBf16) {
        const uint4 q = *reinterpret_cast<const uint4*>(wr);
        float a = acc[r];
        a = fmaf(__uint_as_float(q.x << 16), x8[0], a);
        a = fmaf(__uint_as_float(q.x & 0xFFFF0000u), x8[1], a);
        a = fmaf(__uint_as_float(q.y << 16), x8[2], a);
        a = fmaf(__uint_as_float(q.y & 0xFFFF0000u), x8[3], a);
        a = fmaf(__uint_as_float(q.z << 16), x8[4], a);
        a = fmaf(__uint_as_float(q.z & 0xFFFF0000u), x8[5], a);
        a = fmaf(__uint_as_float(q.w << 16), x8[6], a);
        a = fmaf(__uint_as_float(q.w & 0xFFFF0000u), x8[7], a);
        acc[r] = a;
      } else {
        const float4 q = *reinterpret_cast<const float4*>(wr);
        float a = acc[r];
        a = fmaf(q.x, x8[0], a);
        a = fmaf(q.y, x8[1], a);
        a = fmaf(q.z, x8[2], a);
        a = fmaf(q.w, x8[3], a);
        acc[r] = a;
      }
    }
  }
  (void)kPer;
}

// Sums 32 per-thread values over a warp by recursive halving: after the call, lane l holds the warp total of
// value l (31 shuffles instead of 32 x 5).
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = lane & w;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? v[i] : v[i + w];
      const float keep = upper ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, w);
    }
  }
  return v[0];
}

constexpr float kFix = 4294967296.0f;          // 2^32: fixed-point scale of the correction accumulators
constexpr float kUnfix = 2.3283064365386963e-10f;  // 2^-32

__device__ __forceinline__ void add_fixed(const Params& p, long long* slot, float v) {
  if (!(fabsf(v) < 2147483648.0f)) {  // also catches NaN: the accumulator would overflow
    record_error(p.hdr, DT_ERR_NUMERIC);
    v = 0.f;
  }
  atomicAdd(reinterpret_cast<unsigned long long*>(slot), static_cast<unsigned long long>(__float2ll_rn(v * kFix)));
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads, 1) small_builder(Params p, Plan P) {
  using T = typename WT<kBf16>::T;
  extern __shared__ __align__(16) unsigned char smem[];
  T* wih = reinterpret_cast<T*>(smem + P.wih);      // [R][E], row g*umax + u
  T* whh = reinterpret_cast<T*>(smem + P.whh);      // [R][H]
  float* bias = reinterpret_cast<float*>(smem + P.bias);  // [R][2]: b_ih, b_hh
  T* wc = reinterpret_cast<T*>(smem + P.wc);        // [B][max_depth][M][umax]
  float* xs = reinterpret_cast<float*>(smem + P.x);        // [E + H]: emb row, then parent state
  float* gates = reinterpret_cast<float*>(smem + P.gates);  // [R][2]: input side, hidden side
  float* hnew = reinterpret_cast<float*>(smem + P.hnew);    // [B][umax]
  ReqState* rs = reinterpret_cast<ReqState*>(smem + P.req);  // [B]
  Entry* fr = reinterpret_cast<Entry*>(smem + P.fr);        // [B][n]
  float* red = reinterpret_cast<float*>(smem + P.red);       // [warps][32]: GEMV reduction
  int* ids_s = reinterpret_cast<int*>(smem + P.ids);         // [B][max_depth][M] candidate ids (range-checked)
  float* vals_s = reinterpret_cast<float*>(smem + P.vals);   // [B][max_depth][M] candidate base logits
  short* par_s = reinterpret_cast<short*>(smem + P.par);     // [B][n]: parent of every popped node
  float* hc = reinterpret_cast<float*>(smem + P.hc);         // [B][n][H]: hidden state of every popped node
  __shared__ int s_flag;

  const int B = p.B, K = p.K, M = p.M, n = p.n, H = p.H, E = p.E, maxd = p.max_depth;
  const int G = P.G, umax = P.umax;
  const int j = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int u0 = static_cast<int>((static_cast<long long>(j) * H) / G);
  const int nu = static_cast<int>((static_cast<long long>(j + 1) * H) / G) - u0;
  const size_t esize = kBf16 ? 2 : 4;

  // ---- launch: weights of the owned units, W_c columns of the candidates, L2 prefetch, zeroed accumulators ----
  for (int g = 0; g < 3; ++g) {
    copy16(wih + static_cast<size_t>(g * umax) * E,
           static_cast<const char*>(p.w_ih) + (static_cast<size_t>(g) * H + u0) * E * esize, esize * nu * E);
    copy16(whh + static_cast<size_t>(g * umax) * H,
           static_cast<const char*>(p.w_hh) + (static_cast<size_t>(g) * H + u0) * H * esize, esize * nu * H);
  }
  for (int i = t; i < 3 * umax; i += kThreads) {
    const int g = i / umax, u = i % umax;
    const size_t row = static_cast<size_t>(g) * H + u0 + u;
    bias[2 * i] = (u < nu && p.b_ih) ? ldw(p.b_ih, kBf16, row) : 0.f;
    bias[2 * i + 1] = (u < nu && p.b_hh) ? ldw(p.b_hh, kBf16, row) : 0.f;
  }
#pragma unroll 4
  for (int i = t; i < B * maxd * M; i += kThreads) {
    const int b = i / (maxd * M), pos = (i / M) % maxd, m = i % M;
    const size_t gi = (static_cast<size_t>(b) * K + pos) * M + m;
    const int id = valid_id(p, __ldg(p.ids + gi));
    ids_s[i] = id;
    vals_s[i] = __ldg(p.vals + gi);
    const T* src = static_cast<const T*>(p.w_c) + static_cast<size_t>(id) * H + u0;
    for (int u = 0; u < umax; ++u) wc[static_cast<size_t>(i) * umax + u] = u < nu ? src[u] : T(0);
  }
  {
    const size_t row_bytes = static_cast<size_t>(E) * esize;
    const size_t lines = (row_bytes + 127) / 128;
    const size_t total = static_cast<size_t>(B) * maxd * M * lines;
    for (size_t i = static_cast<size_t>(j) * kThreads + t; i < total; i += static_cast<size_t>(G) * kThreads) {
      const size_t cand = i / lines, line = i % lines;
      const int b = static_cast<int>(cand / (maxd * M)), pos = static_cast<int>((cand / M) % maxd);
      const int m = static_cast<int>(cand % M);
      const int id = __ldg(p.ids + (static_cast<size_t>(b) * K + pos) * M + m);
      if (static_cast<unsigned>(id) < static_cast<unsigned>(p.V)) {
        const char* a = static_cast<const char*>(p.emb) + static_cast<size_t>(id) * row_bytes + line * 128;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
      }
    }
  }
  for (size_t i = static_cast<size_t>(j) * kThreads + t; i < static_cast<size_t>(n) * B * M;
       i += static_cast<size_t>(G) * kThreads)
    p.acc[i] = 0;
  for (int b = t; b < B; b += kThreads) {
    ReqState r{};
    rs[b] = r;
  }
  __shared__ unsigned long long s_base;
  if (t == 0) s_base = ld_relaxed_gpu_u64(&p.hdr->sync_count);  // before anyone can pass the first barrier
  if (!grid_barrier(p.hdr, G, p.timeout_ns, &s_flag)) return;
  const unsigned long long sync_base = s_base;

  for (int s = 0; s < n; ++s) {
    asm volatile("cp.async.wait_all;" ::: "memory");  // this thread's cache copies of the previous step
    __syncthreads();                                   // ... and everyone else's
    long long* acc_s = p.acc + static_cast<size_t>(s) * B * M;
    // ---- phase A: this CTA's share of the GRU and of the correction of every expanding request ----
    for (int b = 0; b < B; ++b) {
      const bool root = s == 0;
      if (!root && !rs[b].expand) continue;  // uniform across the CTA (replicated state)
      const int pos = root ? 0 : rs[b].depth;
      float* hb = hnew + b * umax;
      if (root) {
        for (int u = t; u < nu; u += kThreads) hb[u] = __ldg(p.h0 + static_cast<size_t>(b) * H + u0 + u);
      } else {
        const int tok = rs[b].token, par = rs[b].parent;
        const uint4* erow = reinterpret_cast<const uint4*>(static_cast<const char*>(p.emb) +
                                                           static_cast<size_t>(tok) * E * esize);
        constexpr int kPer16 = kBf16 ? 8 : 4;
#pragma unroll 4
        for (int c = t; c < E / kPer16; c += kThreads) {  // 16-byte loads, all in flight together
          const uint4 q = __ldg(erow + c);
          float* d = xs + c * kPer16;
          if (kBf16) {
            *reinterpret_cast<float4*>(d) = make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xFFFF0000u),
                                                        __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xFFFF0000u));
            *reinterpret_cast<float4*>(d + 4) =
                make_float4(__uint_as_float(q.z << 16), __uint_as_float(q.z & 0xFFFF0000u),
                            __uint_as_float(q.w << 16), __uint_as_float(q.w & 0xFFFF0000u));
          } else {
            *reinterpret_cast<uint4*>(d) = q;
          }
        }
        const float* hp = par < 0 ? nullptr : hc + (static_cast<size_t>(b) * n + par) * H;
        for (int k = t; k < H / 4; k += kThreads)
          reinterpret_cast<float4*>(xs + E)[k] =
              par < 0 ? __ldg(reinterpret_cast<const float4*>(p.h0 + static_cast<size_t>(b) * H) + k)
                      : reinterpret_cast<const float4*>(hp)[k];
        __syncthreads();
        {  // K-split GEMV: each thread reads its slice of x once and applies it to every gate row of this CTA
          constexpr int kPer = kBf16 ? 8 : 4;
          const int R = 3 * umax, EG = E / kPer, KG = (E + H) / kPer;
          float ai[kMaxRows], ah[kMaxRows];
#pragma unroll
          for (int r = 0; r < kMaxRows; ++r) ai[r] = ah[r] = 0.f;
          for (int f = t; f < KG; f += kThreads) {
            float x8[8];
            const float4 a = *reinterpret_cast<const float4*>(xs + f * kPer);
            x8[0] = a.x; x8[1] = a.y; x8[2] = a.z; x8[3] = a.w;
            if (kBf16) {
              const float4 b4 = *reinterpret_cast<const float4*>(xs + f * kPer + 4);
              x8[4] = b4.x; x8[5] = b4.y; x8[6] = b4.z; x8[7] = b4.w;
            }
            if (f < EG) dot8_rows<kBf16>(wih, E, f * kPer, R, x8, ai);
            else dot8_rows<kBf16>(whh, H, (f - EG) * kPer, R, x8, ah);
          }
          float v[32];
#pragma unroll
          for (int r = 0; r < kMaxRows; ++r) {
            v[r] = ai[r];
            v[kMaxRows + r] = ah[r];
          }
          red[warp * 32 + lane] = warp_reduce_scatter32(v);
          __syncthreads();
          if (t < 2 * R) {  // value t: input side of row t (t < kMaxRows) or hidden side of row t - kMaxRows
            const int vi = t < R ? t : kMaxRows + (t - R);
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) sum += red[w * 32 + vi];
            const int r = t < R ? t : t - R;
            gates[2 * r + (t < R ? 0 : 1)] = sum;
          }
        }
        __syncthreads();
        for (int u = t; u < nu; u += kThreads) {
          const int rr = u, rz = umax + u, rn = 2 * umax + u;
          const float r = sigmoidf_(gates[2 * rr] + bias[2 * rr] + gates[2 * rr + 1] + bias[2 * rr + 1]);
          const float z = sigmoidf_(gates[2 * rz] + bias[2 * rz] + gates[2 * rz + 1] + bias[2 * rz + 1]);
          const float g = tanhf(gates[2 * rn] + bias[2 * rn] + r * (gates[2 * rn + 1] + bias[2 * rn + 1]));
          const float h = (1.f - z) * g + z * xs[E + u0 + u];
          hb[u] = h;
          p.hs[(static_cast<size_t>(b) * n + (s - 1)) * H + u0 + u] = h;
        }
      }
      __syncthreads();
      // this CTA's units' part of W_c[id]·h for the M candidates of position pos
      const T* wcp = wc + (static_cast<size_t>(b) * maxd + pos) * M * umax;
      for (int m = t; m < M; m += kThreads) {
        float v = 0.f;
        for (int u = 0; u < nu; ++u) v = fmaf(WT<kBf16>::f(wcp[static_cast<size_t>(m) * umax + u]), hb[u], v);
        if (nu > 0) add_fixed(p, acc_s + static_cast<size_t>(b) * M + m, v);
      }
    }
    if (!counter_barrier(p.hdr, sync_base + static_cast<unsigned long long>(G) * (s + 1), p.timeout_ns, &s_flag))
      return;

    // hidden states of the nodes expanded this step (written unit by unit by all CTAs) into this CTA's cache, as
    // asynchronous global->shared copies that overlap phase C (waited for before the next phase A)
    if (s > 0) {
      for (int b = 0; b < B; ++b) {
        if (!rs[b].expand) continue;
        const float* src = p.hs + (static_cast<size_t>(b) * n + (s - 1)) * H;
        float* dst = hc + (static_cast<size_t>(b) * n + (s - 1)) * H;
        for (int k = t; k < H / 4; k += kThreads) {
          const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst + 4 * k));
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src + 4 * k) : "memory");
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    }

    // ---- phase C: every CTA finishes the step for every request (the whole CTA on one request at a time) ----
    Entry* cand = reinterpret_cast<Entry*>(smem + P.scr);  // [n + M]
    Entry* sorted = cand + (n + M);                          // [n + M]
    float* z = reinterpret_cast<float*>(smem + P.z);         // [M]
    __shared__ float s_red[2];
    for (int b = 0; b < B; ++b) {
      const ReqState st = rs[b];
      const int F = st.fcount;
      const bool expanded = s == 0 || st.expand;
      const int C = expanded ? M : 0;
      const int pos = s == 0 ? 0 : st.depth;
      const size_t off = (static_cast<size_t>(b) * maxd + pos) * M;  // into the staged ids/vals
      for (int i = t; i < F; i += kThreads) cand[i] = fr[static_cast<size_t>(b) * n + i];
      if (expanded) {
        for (int m = t; m < M; m += kThreads) {
          const long long a = __ldcg(acc_s + static_cast<size_t>(b) * M + m);
          z[m] = (vals_s[off + m] + __ll2float_rn(a) * kUnfix) / p.T_eff;
        }
        __syncthreads();
        if (warp == 0) {  // restricted log-softmax statistics
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
        const float base_score = s == 0 ? 0.f : st.score;
        for (int m = t; m < M; m += kThreads) {
          Entry e;
          e.score = base_score + ((z[m] - mx) - lse);
          e.token = ids_s[off + m];
          e.parent = static_cast<short>(s == 0 ? -1 : s - 1);
          e.depth = static_cast<short>(pos + 1);
          e.seq = st.seq_next + m;
          cand[F + m] = e;
        }
      }
      __syncthreads();
      // Keep the R = n - s best (nothing ranked below them can be popped in the n - s pops left). Rank by
      // counting, tpe threads per entry, each counting a stride of the others, combined with shuffles.
      const int N = F + C;
      const int R = min(n - s, N);
      int tpe = 1;
      while (tpe < 32 && tpe * 2 * N <= kThreads) tpe *= 2;
      for (int base = 0; base < N * tpe; base += kThreads) {
        const int slot = base + t, i = slot / tpe, part = slot % tpe;
        int r = 0;
        Entry ei{};
        if (i < N) {
          ei = cand[i];
#pragma unroll 4
          for (int q = part; q < N; q += tpe) r += before(cand[q], ei);
        }
        for (int o = 1; o < tpe; o <<= 1) r += __shfl_xor_sync(0xFFFFFFFFu, r, o);
        if (i < N && part == 0 && r < R) sorted[r] = ei;
      }
      if (N == 0 && t == 0) {  // unreachable when n <= the size of the depth-limited tree (checked on the host)
        record_error(p.hdr, DT_ERR_INVALID_ARG);
        sorted[0] = Entry{-INFINITY, 0, -1, 1, 0};
      }
      __syncthreads();
      const Entry pop = sorted[0];
      for (int i = t + 1; i < R; i += kThreads) fr[static_cast<size_t>(b) * n + i - 1] = sorted[i];
      short* pb = par_s + static_cast<size_t>(b) * n;
      if (t == 0) pb[s] = pop.parent;
      __syncthreads();
      if (j == 0) {
        const size_t o = static_cast<size_t>(b) * n + s;
        uint8_t* mrow = p.mask + o * n;
        for (int c = t; c < n; c += kThreads) {  // ancestor test by walking s's parent chain (parents come first)
          int a = s;
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
      if (t == 0) {
        ReqState ns = st;
        ns.fcount = R - 1;
        ns.seq_next += C;
        ns.token = pop.token;
        ns.parent = pop.parent;
        ns.depth = pop.depth;
        ns.score = pop.score;
        ns.expand = (s + 1 < n) && (pop.depth < maxd);
        rs[b] = ns;
      }
      __syncthreads();
    }
    __syncthreads();
  }
}

int grid_size(const Params& p, int sms) { return sms < p.H ? sms : p.H; }

Plan plan_for(const Params& p, int sms) {
  return make_plan(p.B, p.M, p.n, p.max_depth, p.H, p.E, p.bf16 ? 2 : 4, grid_size(p, sms));
}

}  // namespace

bool small_builder_fits(const Params& p, int sms) {
  if (p.B > kSmallMaxB || p.B < 1 || !p.acc) return false;
  if (3 * plan_for(p, sms).umax > kMaxRows) return false;  // more gate rows per CTA than the GEMV holds
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
  return plan_for(p, sms).bytes <= static_cast<size_t>(optin);
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
