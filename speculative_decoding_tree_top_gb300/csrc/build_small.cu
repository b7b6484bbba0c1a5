// dt_build_trees for small batches (B <= 8): every SM works on every request; no grid barrier between waves.
//
// Method: blog.captcha.la, "Methodology — deep read" (best-first max-priority queue keyed by cumulative conditional
// log-probability; GRU state carried along each root-to-node path; correction only on the gathered top-M rows);
// gist.science, "Composants Clés" (only the light GRU correction and its head are recomputed per node).
//
// GB300 design. With one or a few requests the round is a chain of dependent steps (pop -> GRU -> correction ->
// softmax -> pop), so the design shortens the chain rather than the bytes:
//   * lookahead waves. The expansion of a node (its GRU step and its children's scores) depends only on its own path,
//     never on the pop order, so any frontier node can be expanded before it is popped. A wave expands up to k
//     nodes of each request at once: the node that blocks the next pop, then the next unexpanded nodes in the order
//     best-first would reach them given what is known (the frontier, plus the children of nodes already expanded but
//     not yet popped). The pops themselves stay strictly best-first and exact: a node is popped only from the true
//     frontier, and its children join it only when it is popped. A wrong guess costs an unused expansion, never a
//     different tree; the outputs are bit-identical for every k. The trees of the drafting workloads are wide and
//     shallow, so k = 8 turns 16 dependent steps into 3 to 5 waves;
//   * weight-stationary: CTA j of the G = min(#SMs, H) CTAs owns hidden units [j*H/G, (j+1)*H/G) and keeps the
//     3 gate rows of W_ih and W_hh of those units in shared memory for the whole launch (9.4 MB of GRU weights
//     spread over 152 SMs: ~62 KB each at E=2560, H=512), plus the same units' columns of W_c for every candidate
//     of every position, the candidate ids and base logits (gathered once at launch);
//   * per wave each CTA runs its slice of the GRU for every job (one warp per gate row, all jobs against the row at
//     once), publishes its units of each new hidden state, then adds its units' share of every candidate's
//     correction W_c[id]·h into a per-wave, per-job, per-candidate 64-bit accumulator as ((fixed-point value << 8)
//     + 1): integer addition is associative (the reduction over CTAs is exact and bit-identical run to run) and never
//     carries into the low byte, which therefore counts the contributions. A CTA knows a candidate's correction is
//     complete when that count reaches G: the slot is its own barrier;
//   * every CTA then finishes the wave redundantly: corrected logits, restricted log-softmax and the ranked children
//     list of every job, then one warp per request pops (merging a popped node's children into the frontier, pruned
//     to what can still be popped) and picks the next wave's jobs. All CTAs reach the same decisions, so nothing is
//     exchanged but the hidden states and the correction sums; CTA 0 writes the outputs at the end.
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
constexpr int kJ = kWaveJobs;
static_assert(kJ == 8, "a wave's jobs are the n8 tile of the GRU MMA");
constexpr int kPrefetchPositions = 4;  // block positions whose candidates' embedding rows are prefetched at launch

// Shared-memory plan of one CTA (identical on host and device).
struct Plan {
  int G, umax, R, kmax;
  size_t wih, whh, bias, wc, ids, vals, xe, xh, gates, hb, z, kraw, kkey, red, jobs, ctl, lanes, merged, kids, kcount,
      popidx, sdepth, pops, bytes;
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
  P.kmax = M < n ? M : n;  // children kept per expanded node: at most n can ever be popped
  const size_t X = static_cast<size_t>(expansion_slots(n));
  size_t o = 0;
  P.wih = take(o, static_cast<size_t>(esize) * P.R * (E + kRowPad));
  P.whh = take(o, static_cast<size_t>(esize) * P.R * (H + kRowPad));
  P.bias = take(o, sizeof(float) * 2 * P.R);
  P.wc = take(o, static_cast<size_t>(esize) * B * max_depth * M * P.umax);
  P.ids = take(o, sizeof(int) * B * max_depth * M);
  P.vals = take(o, sizeof(float) * B * max_depth * M);
  P.xe = take(o, static_cast<size_t>(esize) * kJ * (E + kRowPad));  // embedding rows of the wave's jobs, as stored
  P.xh = take(o, sizeof(float) * kJ * H);                          // their parents' hidden states
  P.gates = take(o, sizeof(float) * kJ * P.R * 2);
  P.hb = take(o, sizeof(float) * kJ * P.umax);
  P.z = take(o, sizeof(float) * kJ * M);
  P.kraw = take(o, sizeof(Node) * kJ * M);
  P.kkey = take(o, sizeof(unsigned long long) * kJ * M);
  P.red = take(o, sizeof(float) * kWarps * 2 * kMaxRows * kJ);  // per-warp partial GRU tiles (tensor-core path)
  P.jobs = take(o, sizeof(Job) * kJ);
  P.ctl = take(o, sizeof(ReqCtl) * B);
  P.lanes = take(o, sizeof(LaneSrc) * B * 32);
  P.merged = take(o, sizeof(Node) * B * 2 * n);
  P.kids = take(o, sizeof(Node) * B * X * P.kmax);
  P.kcount = take(o, sizeof(int) * B * X);
  P.popidx = take(o, sizeof(int) * B * X);
  P.sdepth = take(o, sizeof(int) * B * X);
  P.pops = take(o, sizeof(PopRec) * B * n);
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

__device__ __forceinline__ long long ld_relaxed_s64(const long long* p) {
  long long v;
  asm volatile("ld.relaxed.gpu.global.s64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Correction accumulators: every CTA adds ((sum over its units of round(w * h * 2^32)) << 8) + 1 to the slot of each
// candidate. The upper 56 bits hold the exact fixed-point sum, the low byte the number of contributions (G < 256).
constexpr float kFix = 4294967296.0f;              // 2^32
constexpr float kUnfix = 2.3283064365386963e-10f;  // 2^-32
constexpr float kMaxTerm = 4096.0f;                // |w * h| bound: H <= 2048 terms of < 2^44 sum below 2^55

// One hidden unit's term of a correction, w * h, as a fixed-point integer: rounded on its own, so that a candidate's
// sum is the same however the units are spread over the CTAs (and whatever the number of SMs).
__device__ __forceinline__ long long fixed_term(const Params& p, float w, float h) {
  float v = w * h;
  if (!(fabsf(v) < kMaxTerm)) {  // also catches NaN
    record_error(p.hdr, DT_ERR_NUMERIC);
    v = 0.f;
  }
  return __float2ll_rn(v * kFix);
}
// Adds a CTA's share (the sum of its units' fixed-point terms) to a candidate's accumulator, counting one
// contribution in the low byte.
__device__ __forceinline__ void add_share(long long* slot, long long share) {
  const unsigned long long c = (static_cast<unsigned long long>(share) << 8) + 1ull;
  atomicAdd(reinterpret_cast<unsigned long long*>(slot), c);
}

// Sibling order as one 64-bit key (larger first): score, then lower token. Ties of both (only with repeated ids
// among a row's candidates) fall to the lower candidate index, as in the pop order.
__device__ __forceinline__ unsigned long long sibling_key(const Node& e) {
  return (static_cast<unsigned long long>(key_of_f32(__float_as_uint(e.score))) << 32) |
         static_cast<unsigned long long>(~static_cast<uint32_t>(e.token));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// fp32 pair -> bf16x2 high part and bf16x2 remainder (x = hi + lo to 2^-16 relative)
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
  const __nv_bfloat16 l0 = __float2bfloat16_rn(x0 - __bfloat162float(h0));
  const __nv_bfloat16 l1 = __float2bfloat16_rn(x1 - __bfloat162float(h1));
  hi = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
  lo = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
}

template <bool kBf16, bool kMma>  // kMma: bf16 weights with E and H multiples of 16 (tensor-core GRU)
__global__ void __launch_bounds__(kThreads, 1) small_builder(Params p, Plan P) {
  using T = typename WT<kBf16>::T;
  extern __shared__ __align__(16) unsigned char smem[];
  T* wih = reinterpret_cast<T*>(smem + P.wih);               // [R][E + pad], row g*umax + u
  T* whh = reinterpret_cast<T*>(smem + P.whh);               // [R][H + pad]
  float* bias = reinterpret_cast<float*>(smem + P.bias);     // [R][2]: b_ih, b_hh
  T* wc = reinterpret_cast<T*>(smem + P.wc);                 // [B][max_depth][M][umax]
  int* ids_s = reinterpret_cast<int*>(smem + P.ids);         // [B][max_depth][M] candidate ids (range-checked)
  float* vals_s = reinterpret_cast<float*>(smem + P.vals);   // [B][max_depth][M] candidate base logits
  T* xe = reinterpret_cast<T*>(smem + P.xe);                 // [kJ][E + pad]
  float* xh = reinterpret_cast<float*>(smem + P.xh);         // [kJ][H]
  float* gates = reinterpret_cast<float*>(smem + P.gates);   // [kJ][R][2]: input side, hidden side
  float* hb = reinterpret_cast<float*>(smem + P.hb);         // [kJ][umax]: the jobs' new owned units
  float* z = reinterpret_cast<float*>(smem + P.z);           // [kJ][M]
  Node* kraw = reinterpret_cast<Node*>(smem + P.kraw);       // [kJ][M] children, unsorted
  unsigned long long* kkey = reinterpret_cast<unsigned long long*>(smem + P.kkey);  // [kJ][M] their sibling keys
  float* red = reinterpret_cast<float*>(smem + P.red);       // [kWarps][2][16 rows][kJ jobs]
  Job* jobs = reinterpret_cast<Job*>(smem + P.jobs);         // [kJ]
  ReqCtl* ctl = reinterpret_cast<ReqCtl*>(smem + P.ctl);     // [B]
  LaneSrc* lanes = reinterpret_cast<LaneSrc*>(smem + P.lanes);  // [B][32]
  Node* merged = reinterpret_cast<Node*>(smem + P.merged);   // [B][2][n]
  Node* kids = reinterpret_cast<Node*>(smem + P.kids);       // [B][X][kmax] ranked children of each slot
  int* kcount = reinterpret_cast<int*>(smem + P.kcount);     // [B][X]
  int* popidx = reinterpret_cast<int*>(smem + P.popidx);     // [B][X] pop index of the slot's node (-1 root, -2 not yet)
  int* sdepth = reinterpret_cast<int*>(smem + P.sdepth);     // [B][X] depth of the slot's node
  PopRec* pops = reinterpret_cast<PopRec*>(smem + P.pops);   // [B][n]
  __shared__ int s_flag, s_J;
  __shared__ uint64_t wbar;  // completion of the weight rows' bulk copies
  __shared__ uint64_t jbar;  // completion of a wave's input copies (embedding rows, parents' states)

  const int B = p.B, K = p.K, M = p.M, n = p.n, H = p.H, E = p.E, maxd = p.max_depth;
  const int G = P.G, umax = P.umax, KM = P.kmax, X = p.xslots;
  const int kla = p.lookahead;
  const int j = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int u0 = static_cast<int>((static_cast<long long>(j) * H) / G);
  const int nu = static_cast<int>((static_cast<long long>(j + 1) * H) / G) - u0;
  const size_t esize = kBf16 ? 2 : 4;
  const int AS = p.acc_stride;
  const int SE = E + kRowPad, SH = H + kRowPad;  // shared-memory row strides of W_ih / xe and of W_hh

  // ---- launch: weights of the owned units, W_c columns / ids / base logits of the candidates, L2 prefetch ----
  // The 3 * nu rows of W_ih and of W_hh as bulk copies (1 to 8 KB each) completing on one mbarrier, issued by warp 0;
  // waited for before the first GRU step.
  const uint64_t t_launch = global_timer_ns();
  if (t == 0) {
    mbar_init(&wbar, 1);
    mbar_init(&jbar, 1);
    mbar_fence_init();
    if (j == 0) {  // the launch's statistics start from zero (before the grid barrier, after which they are raised)
      p.hdr->stat_launch_ns = p.hdr->stat_gather_ns = p.hdr->stat_gather_bytes = 0ull;
      p.hdr->stat_waves = p.hdr->stat_expansions = 0u;
    }
  }
  __syncthreads();
  uint64_t gather_ns = 0, gather_bytes = 0;  // this CTA's time in the W_c gathers; the rows they read (CTA 0)
  for (int i = t; i < 3 * umax; i += kThreads) {
    const int g = i / umax, u = i % umax;
    const size_t row = static_cast<size_t>(g) * H + u0 + u;
    bias[2 * i] = (u < nu && p.b_ih) ? ldw(p.b_ih, kBf16, row) : 0.f;
    bias[2 * i + 1] = (u < nu && p.b_hh) ? ldw(p.b_hh, kBf16, row) : 0.f;
  }
  // the candidates' ids and base logits of every request and position the tree can reach, into shared memory
  auto load_candidates = [&](int p0, int p1) {  // block positions [p0, p1)
    const int np = p1 - p0;
    for (int i = t; i < B * np * M; i += kThreads) {
      const int b = i / (np * M), pos = p0 + (i / M) % np, m = i % M;
      const size_t gi = (static_cast<size_t>(b) * K + pos) * M + m;
      const int si = (b * maxd + pos) * M + m;
      ids_s[si] = valid_id(p, __ldcg(p.ids + gi));
      vals_s[si] = __ldcg(p.vals + gi);
    }
  };
  // The owned units' W_c columns of the candidates of block positions [p0, p1): each needed row comes into L2 once
  // (one bulk prefetch per row, spread over the CTAs, so HBM serves whole rows), then every CTA takes its columns.
  auto gather_wc = [&](int p0, int p1) {
    const int np = p1 - p0;
    const uint64_t g0 = global_timer_ns();
    const unsigned rb = static_cast<unsigned>(H * esize);
    for (int i = j * kThreads + t; i < B * np * M; i += G * kThreads) {
      const int b = i / (np * M), pos = p0 + (i / M) % np, m = i % M;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                   ::"l"(static_cast<const char*>(p.w_c) + static_cast<size_t>(ids_s[(b * maxd + pos) * M + m]) * rb),
                   "r"(rb)
                   : "memory");
    }
#pragma unroll 8
    for (int q = t; q < B * np * M * umax; q += kThreads) {
      const int i = q / umax, u = q % umax;
      const int b = i / (np * M), pos = p0 + (i / M) % np, m = i % M;
      const int c = (b * maxd + pos) * M + m;
      wc[c * umax + u] = u < nu ? static_cast<const T*>(p.w_c)[static_cast<size_t>(ids_s[c]) * H + u0 + u] : T(0);
    }
    __syncthreads();  // every thread's columns are in (and the statistics see the whole gather)
    gather_ns += global_timer_ns() - g0;
    gather_bytes += static_cast<uint64_t>(B) * np * M * H * esize;
  };
  // the 3 * nu rows of W_ih and of W_hh as bulk copies (1 to 8 KB each) completing on one mbarrier, issued by warp 0;
  // waited for before the first GRU step
  auto issue_weights = [&]() {
    if (warp != 0) return;
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
  };
  // Before the CTA leaves, every bulk copy it issued must have landed (none may write shared memory after the exit):
  // this waits (bounded) for the weight rows unless the GRU step already did, and for the next wave's inputs when
  // `jobs_parity` >= 0 names the pending phase of their barrier.
  bool weights_in = false;
  auto drain = [&](int jobs_parity) {
    if (!weights_in) mbar_wait(&wbar, 0, kCopyBudgetNs);
    if (jobs_parity >= 0) mbar_wait(&jbar, static_cast<unsigned>(jobs_parity), kCopyBudgetNs);
  };
  int wc_pos = maxd < kPrefetchPositions ? maxd : kPrefetchPositions;  // positions gathered so far
  {
    // The launch's loads in the order they are needed: the candidates, then the owned units' W_c columns of every
    // candidate (they depend on the ids), then the GRU weight rows, which the first GRU step (wave 1) only needs: the
    // dependent chain is not queued behind 9.4 MB of weights.
    load_candidates(0, maxd);
    __syncthreads();
    gather_wc(0, wc_pos);
    issue_weights();
    // the embedding rows of the candidates of the first block positions (where the waves' jobs come from in the
    // shallow trees of drafting) into L2, spread over the CTAs: the wave transitions then read them from L2
    const size_t row_bytes = static_cast<size_t>(E) * esize;
    const size_t lines = (row_bytes + 127) / 128;
    const int npos = maxd < kPrefetchPositions ? maxd : kPrefetchPositions;
    const size_t total = static_cast<size_t>(B) * npos * M * lines;
    for (size_t i = static_cast<size_t>(j) * kThreads + t; i < total; i += static_cast<size_t>(G) * kThreads) {
      const size_t c = i / lines, line = i % lines;
      const int b = static_cast<int>(c / (npos * M)), pos = static_cast<int>((c / M) % npos);
      const int m = static_cast<int>(c % M);
      const int id = ids_s[(static_cast<size_t>(b) * maxd + pos) * M + m];  // range-checked
      const char* a = static_cast<const char*>(p.emb) + static_cast<size_t>(id) * row_bytes + line * 128;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
    }
  }
  // every wave's accumulators and arrival counters start at zero; one grid barrier orders that
  {
    const size_t acc_words = static_cast<size_t>(X) * kJ * M;  // one word per accumulator line
    for (size_t i = static_cast<size_t>(j) * kThreads + t; i < acc_words; i += static_cast<size_t>(G) * kThreads)
      p.acc[i * AS] = 0;
    for (int i = j * kThreads + t; i < X; i += G * kThreads) p.hs_count[i] = 0;
  }
  // control state, identical in every CTA: the root of every request is expanded in wave 0. A wave has S = B * kla job
  // slots, slot b * kla + q holding request b's q-th expansion (b = -1: empty); the slot is the job's column of the
  // GRU's MMA tile and its row of the staged inputs.
  // Wave 0 also expands, speculatively, the first nspec candidates of position 0 (the root's likeliest children by
  // marginal logit) as depth-1 nodes in slots 1 .. nspec: their GRU inputs (embedding row, h0) are known before any
  // score is. As with every pick, a wrong guess costs an unused expansion, never a different tree.
  const int S = B * kla;
  const int nspec = (maxd >= 2 && n >= 2) ? min(kla - 1, M) : 0;
  for (int b = t; b < B; b += kThreads) ctl[b] = ReqCtl{0, 0, M, 1 + nspec, 0, {0, 0, 0}};  // root's children: 0 .. M-1
  for (int i = t; i < kJ; i += kThreads) {
    const int b = i / kla, q = i % kla;
    jobs[i] = i >= S ? Job{-1, 0, 0, 0, 0, 0.f, {0, 0}}
              : q == 0 ? Job{b, 0, -1, 0, 0, 0.f, {0, 0}}       // the root
              : q <= nspec ? Job{b, q, 0, 0, 1, 0.f, {q, 0}}    // candidate q - 1 of position 0 (token set below)
                           : Job{-1, 0, 0, 0, 0, 0.f, {0, 0}};
  }
  for (int i = t; i < B * n; i += kThreads) pops[i] = PopRec{0, 0, 0, -INFINITY};
  for (int i = t; i < B * 32; i += kThreads) {  // lane 0: the merged list (empty), lane 1: the root's children
    const int l = i % 32;
    lanes[i] = l == 0 ? LaneSrc{-2, 0, 0, 0, -1, {0, 0, 0}} : l == 1 ? LaneSrc{0, 0, -1, 0, 1, {0, 0, 0}} : LaneSrc{-1, 0, 0, 0, -1, {0, 0, 0}};
  }
  for (int i = t; i < B * X; i += kThreads) {
    kcount[i] = 0;
    popidx[i] = (i % X) == 0 ? -1 : -2;
    sdepth[i] = (i % X) >= 1 && (i % X) <= nspec ? 1 : 0;
  }
  if (t == 0) s_J = B;
  const unsigned erow = static_cast<unsigned>(E * esize), hrow = static_cast<unsigned>(H * sizeof(float));
  // wave 0's inputs: the speculative jobs' embedding rows and h0 as bulk copies on jbar (the candidates are staged);
  // one arrival closes the barrier's phase 0, which wave 0 waits for (at once when nothing was copied)
  auto issue_spec = [&]() {
    __syncthreads();  // the jobs and the candidates are in place
    for (int i = t; i < S; i += kThreads) {
      const int b = i / kla, q = i % kla;
      if (q < 1 || q > nspec) continue;
      const int tok = ids_s[static_cast<size_t>(b) * maxd * M + (q - 1)];
      jobs[i].token = tok;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_expect_tx_only(&jbar, erow + hrow);
      bulk_g2s(xe + static_cast<size_t>(i) * SE, static_cast<const char*>(p.emb) + static_cast<size_t>(tok) * erow,
               erow, &jbar);
      bulk_g2s(xh + static_cast<size_t>(i) * H, p.h0 + static_cast<size_t>(b) * H, hrow, &jbar);
    }
    __syncthreads();
    if (t == 0) mbar_arrive(&jbar);
  };
  issue_spec();
  if (!grid_barrier(p.hdr, G, p.timeout_ns, &s_flag)) {
    drain(0);  // the speculative jobs' copies are in flight
    return;
  }

  for (int w = 0;; ++w) {
    __syncthreads();
    const int J = s_J;  // expansions in this wave
    if (J == 0) {
      // the barrier's pending phase completes once its copies land (none were issued when nothing was picked)
      mbar_wait(&jbar, w & 1, kCopyBudgetNs);
      break;
    }
    // the jobs' inputs, copied while the previous wave picked them (wave 0: the speculative jobs' inputs, copied at
    // launch); every thread waits, and the decision to leave is taken by the whole CTA at once
    if (!__syncthreads_and(mbar_wait(&jbar, w & 1, kCopyBudgetNs))) {
      record_error(p.hdr, DT_ERR_TIMEOUT);
      atomicExch(&p.hdr->abort, 1u);
      drain(w & 1);  // the wave's input copies are still outstanding
      return;
    }
    long long* acc_w = p.acc + static_cast<size_t>(w) * kJ * M * AS;
    if (j == 0 && t == 0) {
      p.hdr->stat_waves = w + 1;
      p.hdr->stat_expansions += (w == 0 ? B * (1 + nspec) : J);
    }
    // a GRU step runs unless the wave holds roots only (roots take h = h0); wave 0 also holds the speculative jobs
    const bool gru = w > 0 || nspec > 0;
    const bool spec_wave = w == 0 && nspec > 0;
    if (gru && !weights_in) {  // the weight rows, before the first GRU step (bounded)
      if (!__syncthreads_and(mbar_wait(&wbar, 0, kCopyBudgetNs))) {  // never compute on unstaged weights: leave
        record_error(p.hdr, DT_ERR_TIMEOUT);
        atomicExch(&p.hdr->abort, 1u);
        drain(-1);
        return;
      }
      weights_in = true;
    }
    {  // a job deeper than the positions gathered so far: gather up to it and a few beyond (same in every CTA)
      int deepest = 0;
      for (int q = 0; q < S; ++q)
        if (jobs[q].b >= 0) deepest = max(deepest, jobs[q].depth);
      if (deepest >= wc_pos) {
        const int upto = min(maxd, deepest + kPrefetchPositions);
        gather_wc(wc_pos, upto);
        wc_pos = upto;
        __syncthreads();
      }
    }

    // ---- phase A: this CTA's units of every job's GRU step, then its share of every job's correction ----
    constexpr bool mma = kBf16 && kMma;  // the tensor-core GRU (else the CUDA-core one below)
    if (gru && mma) {
      // Tensor cores, mma.sync m16n8k16 (bf16 in, fp32 accumulate): D[16 gate rows][8 jobs] = W[rows][K] X[K][jobs],
      // the warps splitting the k16 steps. A = this CTA's gate rows (rows past R repeat row R - 1: their outputs are
      // not used), B = the jobs' embedding rows (input side) and the parents' fp32 states as bf16 hi + lo pairs
      // (hidden side); each side has its own accumulator, the n gate needs them apart. A job's column never mixes
      // with another's, so its sums do not depend on which jobs share the wave (an empty slot's column is computed
      // on whatever its rows hold, and never used).
      const int g = lane >> 2, tg = lane & 3, R = 3 * umax;
      float din[4] = {0.f, 0.f, 0.f, 0.f}, dh[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const unsigned short* a_lo = reinterpret_cast<const unsigned short*>(wih) + static_cast<size_t>(min(g, R - 1)) * SE;
        const unsigned short* a_hi = reinterpret_cast<const unsigned short*>(wih) + static_cast<size_t>(min(g + 8, R - 1)) * SE;
        const unsigned short* bx = reinterpret_cast<const unsigned short*>(xe) + static_cast<size_t>(g) * SE;
#pragma unroll 2
        for (int ks = warp; ks < E / 16; ks += kWarps) {
          const int k = ks * 16 + tg * 2;
          mma_bf16_16816(din, *reinterpret_cast<const uint32_t*>(a_lo + k), *reinterpret_cast<const uint32_t*>(a_hi + k),
                         *reinterpret_cast<const uint32_t*>(a_lo + k + 8), *reinterpret_cast<const uint32_t*>(a_hi + k + 8),
                         *reinterpret_cast<const uint32_t*>(bx + k), *reinterpret_cast<const uint32_t*>(bx + k + 8));
        }
      }
      {
        const unsigned short* a_lo = reinterpret_cast<const unsigned short*>(whh) + static_cast<size_t>(min(g, R - 1)) * SH;
        const unsigned short* a_hi = reinterpret_cast<const unsigned short*>(whh) + static_cast<size_t>(min(g + 8, R - 1)) * SH;
        const float* bh = xh + static_cast<size_t>(g) * H;
        for (int ks = warp; ks < H / 16; ks += kWarps) {
          const int k = ks * 16 + tg * 2;
          const uint32_t a0 = *reinterpret_cast<const uint32_t*>(a_lo + k), a1 = *reinterpret_cast<const uint32_t*>(a_hi + k);
          const uint32_t a2 = *reinterpret_cast<const uint32_t*>(a_lo + k + 8), a3 = *reinterpret_cast<const uint32_t*>(a_hi + k + 8);
          const float2 x0 = *reinterpret_cast<const float2*>(bh + k), x1 = *reinterpret_cast<const float2*>(bh + k + 8);
          uint32_t h0, l0, h1, l1;
          split_bf16x2(x0.x, x0.y, h0, l0);
          split_bf16x2(x1.x, x1.y, h1, l1);
          mma_bf16_16816(dh, a0, a1, a2, a3, h0, h1);
          mma_bf16_16816(dh, a0, a1, a2, a3, l0, l1);
        }
      }
      // this warp's partial tiles: the thread holds rows g, g + 8 and job columns 2 tg, 2 tg + 1
      float* rw = red + warp * 2 * kMaxRows * kJ;
      *reinterpret_cast<float2*>(rw + g * kJ + 2 * tg) = make_float2(din[0], din[1]);
      *reinterpret_cast<float2*>(rw + (g + 8) * kJ + 2 * tg) = make_float2(din[2], din[3]);
      *reinterpret_cast<float2*>(rw + (kMaxRows + g) * kJ + 2 * tg) = make_float2(dh[0], dh[1]);
      *reinterpret_cast<float2*>(rw + (kMaxRows + g + 8) * kJ + 2 * tg) = make_float2(dh[2], dh[3]);
    }
    if (gru && !mma && warp < 3 * umax) {
      // One warp per gate row (R <= 16 rows, 16 warps), every job slot against the row: the lanes stride over K, one
      // accumulator per slot and side, then one shuffle tree each. A job's sums do not depend on the other jobs.
      // The row's input side (over E) and hidden side (over H) stay apart: the n gate needs them separately.
      const int r = warp;
      constexpr int kPer = kBf16 ? 8 : 4;
      float ai[kJ], ah[kJ];
#pragma unroll
      for (int q = 0; q < kJ; ++q) ai[q] = ah[q] = 0.f;
      const T* wr = wih + static_cast<size_t>(r) * SE;
      for (int f = lane; f < E / kPer; f += 32) {
        const int c = f * kPer;
        if (kBf16) {
          const uint4 wv = *reinterpret_cast<const uint4*>(wr + c);
          const float w0 = __uint_as_float(wv.x << 16), w1 = __uint_as_float(wv.x & 0xFFFF0000u);
          const float w2 = __uint_as_float(wv.y << 16), w3 = __uint_as_float(wv.y & 0xFFFF0000u);
          const float w4 = __uint_as_float(wv.z << 16), w5 = __uint_as_float(wv.z & 0xFFFF0000u);
          const float w6 = __uint_as_float(wv.w << 16), w7 = __uint_as_float(wv.w & 0xFFFF0000u);
#pragma unroll
          for (int q = 0; q < kJ; ++q) {
            if (q >= S) break;
            const uint4 xv = *reinterpret_cast<const uint4*>(xe + static_cast<size_t>(q) * SE + c);
            float a = ai[q];
            a = fmaf(w0, __uint_as_float(xv.x << 16), a);
            a = fmaf(w1, __uint_as_float(xv.x & 0xFFFF0000u), a);
            a = fmaf(w2, __uint_as_float(xv.y << 16), a);
            a = fmaf(w3, __uint_as_float(xv.y & 0xFFFF0000u), a);
            a = fmaf(w4, __uint_as_float(xv.z << 16), a);
            a = fmaf(w5, __uint_as_float(xv.z & 0xFFFF0000u), a);
            a = fmaf(w6, __uint_as_float(xv.w << 16), a);
            a = fmaf(w7, __uint_as_float(xv.w & 0xFFFF0000u), a);
            ai[q] = a;
          }
        } else {
          const float4 wv = *reinterpret_cast<const float4*>(wr + c);
#pragma unroll
          for (int q = 0; q < kJ; ++q) {
            if (q >= S) break;
            const float4 xv = *reinterpret_cast<const float4*>(xe + static_cast<size_t>(q) * SE + c);
            float a = ai[q];
            a = fmaf(wv.x, xv.x, a);
            a = fmaf(wv.y, xv.y, a);
            a = fmaf(wv.z, xv.z, a);
            a = fmaf(wv.w, xv.w, a);
            ai[q] = a;
          }
        }
      }
      const T* hr = whh + static_cast<size_t>(r) * SH;
      for (int f = lane; f < H / kPer; f += 32) {
        const int c = f * kPer;
        if (kBf16) {
          const uint4 wv = *reinterpret_cast<const uint4*>(hr + c);
          const float w0 = __uint_as_float(wv.x << 16), w1 = __uint_as_float(wv.x & 0xFFFF0000u);
          const float w2 = __uint_as_float(wv.y << 16), w3 = __uint_as_float(wv.y & 0xFFFF0000u);
          const float w4 = __uint_as_float(wv.z << 16), w5 = __uint_as_float(wv.z & 0xFFFF0000u);
          const float w6 = __uint_as_float(wv.w << 16), w7 = __uint_as_float(wv.w & 0xFFFF0000u);
#pragma unroll
          for (int q = 0; q < kJ; ++q) {
            if (q >= S) break;
            const float4 x0 = *reinterpret_cast<const float4*>(xh + static_cast<size_t>(q) * H + c);
            const float4 x1 = *reinterpret_cast<const float4*>(xh + static_cast<size_t>(q) * H + c + 4);
            float a = ah[q];
            a = fmaf(w0, x0.x, a);
            a = fmaf(w1, x0.y, a);
            a = fmaf(w2, x0.z, a);
            a = fmaf(w3, x0.w, a);
            a = fmaf(w4, x1.x, a);
            a = fmaf(w5, x1.y, a);
            a = fmaf(w6, x1.z, a);
            a = fmaf(w7, x1.w, a);
            ah[q] = a;
          }
        } else {
          const float4 wv = *reinterpret_cast<const float4*>(hr + c);
#pragma unroll
          for (int q = 0; q < kJ; ++q) {
            if (q >= S) break;
            const float4 xv = *reinterpret_cast<const float4*>(xh + static_cast<size_t>(q) * H + c);
            float a = ah[q];
            a = fmaf(wv.x, xv.x, a);
            a = fmaf(wv.y, xv.y, a);
            a = fmaf(wv.z, xv.z, a);
            a = fmaf(wv.w, xv.w, a);
            ah[q] = a;
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kJ; ++q) {
        if (q >= S) break;
        float si = ai[q], sh = ah[q];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          si += __shfl_xor_sync(0xFFFFFFFFu, si, o);
          sh += __shfl_xor_sync(0xFFFFFFFFu, sh, o);
        }
        if (lane == 0) {
          gates[(q * 3 * umax + r) * 2] = si;
          gates[(q * 3 * umax + r) * 2 + 1] = sh;
        }
      }
    }
    __syncthreads();
    if (gru && mma) {  // the partial tiles summed over the warps in a fixed order
      for (int i = t; i < 2 * 3 * umax * S; i += kThreads) {
        const int side = i / (3 * umax * S), r = (i / S) % (3 * umax), q = i % S;
        float v = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kWarps; ++w2) v += red[(w2 * 2 + side) * kMaxRows * kJ + r * kJ + q];
        gates[(q * 3 * umax + r) * 2 + side] = v;
      }
    }
    __syncthreads();
    // the GRU pointwise of the owned units (root jobs: h0), stored to the slot's hidden state; the CTA's arrival on
    // the wave's counter below publishes them together with the correction shares
    for (int i = t; i < S * umax; i += kThreads) {
      const int q = i / umax, u = i % umax;
      const Job jb = jobs[q];
      if (u >= nu || jb.b < 0) continue;
      float hn;
      if (jb.pslot < 0) {  // a root
        hn = __ldg(p.h0 + static_cast<size_t>(jb.b) * H + u0 + u);
      } else {
        const float* gq = gates + q * 3 * umax * 2;
        const int rr = u, rz = umax + u, rn = 2 * umax + u;
        const float r = sigmoidf_(gq[2 * rr] + bias[2 * rr] + gq[2 * rr + 1] + bias[2 * rr + 1]);
        const float zg = sigmoidf_(gq[2 * rz] + bias[2 * rz] + gq[2 * rz + 1] + bias[2 * rz + 1]);
        const float g = tanhf(gq[2 * rn] + bias[2 * rn] + r * (gq[2 * rn + 1] + bias[2 * rn + 1]));
        hn = (1.f - zg) * g + zg * xh[static_cast<size_t>(q) * H + u0 + u];
      }
      hb[q * umax + u] = hn;
      p.hs[(static_cast<size_t>(jb.b) * X + jb.xslot) * H + u0 + u] = hn;
    }
    __syncthreads();
    // this CTA's units' part of W_c[id]·h for the M candidates of each job's block position
    for (int i = t; i < S * M; i += kThreads) {
      const int q = i / M, m = i % M;
      const Job jb = jobs[q];
      if (jb.b < 0) continue;
      const T* wcp = wc + ((static_cast<size_t>(jb.b) * maxd + jb.depth) * M + m) * umax;
      long long v = 0;
      for (int u = 0; u < nu; ++u) v += fixed_term(p, WT<kBf16>::f(wcp[u]), hb[q * umax + u]);
      add_share(acc_w + (static_cast<size_t>(q) * M + m) * AS, v);
    }
    // One arrival per CTA and wave (release: the hidden-state units and the shares above come first). A CTA that
    // sees G arrivals (acquire) sees every share of every candidate and every unit of the wave's hidden states.
    __syncthreads();
    if (t == 0) asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.hs_count + w) : "memory");
    if (t == 0) {
      int ok = 1;
      const unsigned* cnt = reinterpret_cast<const unsigned*>(p.hs_count + w);
      const uint64_t t0 = global_timer_ns();
      for (unsigned polls = 1; ld_acquire_gpu(cnt) < static_cast<unsigned>(G); ++polls)
        if ((polls & 15u) == 0u && (ld_acquire_gpu(&p.hdr->abort) != 0u || global_timer_ns() - t0 > p.timeout_ns)) {
          record_error(p.hdr, DT_ERR_TIMEOUT);
          atomicExch(&p.hdr->abort, 1u);
          ok = 0;
          break;
        }
      s_flag = ok;
    }
    __syncthreads();
    if (!s_flag) {  // a wait ran out (recorded): leave with no copy in flight
      drain(-1);
      return;
    }

    // ---- phase C: every CTA finishes the wave (replicated) ----
    // (1) one warp per job: the corrected logits from the completed sums, the restricted log-softmax, the children;
    //     for M <= 128 the same warp ranks them (a bitonic sort of 64-bit sibling keys across its lanes) and keeps the
    //     first kc: at most n - s - 1 of them can still be popped after the job's node itself (n for the root's)
    if (warp < S && jobs[warp].b >= 0) {
      const int q = warp;
      const Job jb = jobs[q];
      const size_t off = (static_cast<size_t>(jb.b) * maxd + jb.depth) * M;  // staged ids / base logits
      const long long* slots = acc_w + static_cast<size_t>(q) * M * AS;
      float mx = -INFINITY;
      for (int m0 = lane; m0 < M; m0 += 128) {
        long long a[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int m = m0 + 32 * jj;
          a[jj] = m < M ? ld_relaxed_s64(slots + static_cast<size_t>(m) * AS) : 0ll;
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int m = m0 + 32 * jj;
          if (m >= M) break;
          const float v = (vals_s[off + m] + __ll2float_rn(a[jj] >> 8) * kUnfix) / p.T_eff;
          z[q * M + m] = v;
          mx = fmaxf(mx, v);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      float sum = 0.f;
      for (int m = lane; m < M; m += 32) sum += expf(z[q * M + m] - mx);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
      const float lse = logf(sum);
      for (int m = lane; m < M; m += 32) z[q * M + m] = (z[q * M + m] - mx) - lse;  // the restricted log-softmax
    }
    // (1b) the children's scores: the node's score plus their log-probabilities. A speculative job of wave 0 takes its
    //      own score from the root's children, scored by the root's warp in (1) (score 0 + logp, as a pop sees it).
    if (spec_wave) __syncthreads();
    if (warp < S && jobs[warp].b >= 0) {
      const int q = warp;
      const Job jb = jobs[q];
      const size_t off = (static_cast<size_t>(jb.b) * maxd + jb.depth) * M;
      const int rq = jb.b * kla;  // the request's root slot in wave 0
      const float base = jb.aux[0] > 0 ? jobs[rq].score + z[rq * M + (jb.aux[0] - 1)] : jb.score;
      for (int m = lane; m < M; m += 32) {
        Node e;
        e.score = base + z[q * M + m];
        e.token = ids_s[off + m];
        e.seq = m;  // the candidate index until the node is popped
        e.pslot = static_cast<short>(jb.xslot);
        e.xslot = -1;
        kraw[q * M + m] = e;
        kkey[q * M + m] = sibling_key(e);
      }
      if (M <= 128) {
        __syncwarp();
        const int rem = jb.pslot < 0 ? n : n - ctl[jb.b].s - 1;
        const int kc = min(min(M, KM), rem);
        Node* out = kids + (static_cast<size_t>(jb.b) * X + jb.xslot) * KM;
        rank_children(kraw + q * M, kkey + q * M, M, p.V, out, kc);
        if (lane == 0) kcount[jb.b * X + jb.xslot] = kc;
      }
    }
    __syncthreads();
    // (2) M > 128: every job's children ranked among themselves by their sibling keys (tpe threads per child)
    if (M > 128) {
      int tpe = 1;
      while (tpe < 32 && tpe * 2 * S * M <= kThreads) tpe *= 2;
      for (int base = 0; base < S * M * tpe; base += kThreads) {  // uniform bounds: every lane reaches the shuffles
        const int slot = base + t, i = slot / tpe, part = slot % tpe;
        const int q = i / M, mi = i % M;
        const bool live = i < S * M && jobs[q < S ? q : 0].b >= 0;
        int r = 0;
        if (live) {
          const unsigned long long ki = kkey[i];
          const unsigned long long* sib = kkey + q * M;
#pragma unroll 8
          for (int c = part; c < M; c += tpe) {
            const unsigned long long kc = sib[c];
            r += (kc > ki) | ((kc == ki) & (c < mi));
          }
        }
        for (int o = 1; o < tpe; o <<= 1) r += __shfl_xor_sync(0xFFFFFFFFu, r, o);
        if (live && part == 0) {
          const Job jb = jobs[q];
          const int rem = jb.pslot < 0 ? n : n - ctl[jb.b].s - 1;
          const int kc = min(min(M, KM), rem);
          if (r < kc) kids[(static_cast<size_t>(jb.b) * X + jb.xslot) * KM + r] = kraw[i];
          if (r == 0) kcount[jb.b * X + jb.xslot] = kc;
        }
      }
      __syncthreads();
    }
    // (3) one warp per request: pops, then the next wave's picks. Each pick's inputs (its embedding row and its
    //     parent's hidden state) are copied into the pick's job slot as soon as the pick is made, on jbar: the copies
    //     overlap the rest of the walk. This wave's generic reads of those rows (phase A) and the other CTAs' stores
    //     of the hidden states (acquired above) are ordered before the asynchronous copies by the proxy fences.
    if (warp < B) {
      const int b = warp;
      const ReqView R{ctl + b, lanes + b * 32, merged + static_cast<size_t>(b) * 2 * n,
                      kids + static_cast<size_t>(b) * X * KM, kcount + b * X, popidx + b * X, sdepth + b * X,
                      pops + static_cast<size_t>(b) * n};
      if (spec_wave) {  // the root's children that wave 0 expanded speculatively (candidate m: slot 1 + m) are known
        const int kc0 = kcount[b * X];
        for (int i = lane; i < kc0; i += 32) {
          Node& e = kids[static_cast<size_t>(b) * X * KM + i];
          if (e.seq < nspec) e.xslot = static_cast<short>(1 + e.seq);
        }
        __syncwarp();
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("fence.proxy.async.global;" ::: "memory");
      const auto start_copies = [&](int q, const Job& jb) {
        const int slot = b * kla + q;
        mbar_expect_tx_only(&jbar, erow + hrow);
        bulk_g2s(xe + static_cast<size_t>(slot) * SE, static_cast<const char*>(p.emb) + static_cast<size_t>(jb.token) * erow,
                 erow, &jbar);
        bulk_g2s(xh + static_cast<size_t>(slot) * H, p.hs + (static_cast<size_t>(b) * X + jb.pslot) * H, hrow, &jbar);
      };
      request_step(R, b, n, M, maxd, X, KM, kla, jobs + b * kla, p.hdr, start_copies);
      __syncwarp();
      const int nj = ctl[b].njobs;
      if (lane < kla && lane >= nj) jobs[b * kla + lane].b = -1;  // the request's slots left empty next wave
    }
    __syncthreads();
    if (t == 0) {
      int J2 = 0;
      for (int b = 0; b < B; ++b) J2 += ctl[b].njobs;
      if (J2 > 0 && w + 1 >= X) {  // cannot happen: every wave expands at least one of a request's X slots
        record_error(p.hdr, DT_ERR_INVALID_ARG);
        J2 = 0;
      }
      mbar_arrive(&jbar);  // the phase completes once every copy the picks started has landed
      s_J = J2;
    }
  }

  drain(-1);  // a round without GRU steps (n = 1, or max depth 1) never waited for the weights
  if (t == 0) {
    atomicMax(&p.hdr->stat_gather_ns, static_cast<unsigned long long>(gather_ns));
    if (j == 0) {
      p.hdr->stat_gather_bytes = gather_bytes;
      p.hdr->stat_launch_ns = global_timer_ns() - t_launch;
    }
  }
  // ---- outputs (CTA 0): nodes in pop order, and the ancestor mask by walking each node's parent chain ----
  if (j == 0) {
    for (int b = 0; b < B; ++b) resolve_parents(pops + b * n, popidx + b * X, n, t, kThreads);
    __syncthreads();
    for (int i = t; i < B * n; i += kThreads) {
      const PopRec r = pops[i];
      p.tokens[i] = r.token;
      p.parents[i] = r.parent;
      p.depth[i] = r.depth;
      p.scores[i] = r.score;
    }
    for (size_t i = t; i < static_cast<size_t>(B) * n * n; i += kThreads) {
      const int b = static_cast<int>(i / (static_cast<size_t>(n) * n));
      const int row = static_cast<int>((i / n) % n), c = static_cast<int>(i % n);
      int a = row;
      for (int hops = 0; a > c && hops < n; ++hops) a = pops[b * n + a].parent;  // parents precede their children
      p.mask[i] = a == c;
    }
  }
}

int grid_size(const Params& p, int sms) { return sms < p.H ? sms : p.H; }

Plan plan_for(const Params& p, int sms) {
  return make_plan(p.B, p.M, p.n, p.max_depth, p.H, p.E, p.bf16 ? 2 : 4, grid_size(p, sms));
}

}  // namespace

bool small_builder_fits(const Params& p, const DeviceInfo& di) {
  if (p.B > kSmallMaxB || p.B < 1 || !p.acc) return false;
  if (p.B * p.lookahead > kWaveJobs) return false;
  const Plan P = plan_for(p, di.sms);
  if (3 * P.umax > kMaxRows || P.G > 255) return false;  // GEMV rows per CTA; contribution count in one byte
  return P.bytes <= static_cast<size_t>(di.optin);
}

// One CTA per SM at most (launch bounds of 512 threads, one block), so the shared-memory plan alone decides that the
// G CTAs are co-resident; the cooperative launch checks it again.
cudaError_t launch_small_builder(const Params& p, const DeviceInfo& di, cudaStream_t stream) {
  const Plan P = plan_for(p, di.sms);
  const bool mma = p.bf16 && p.E % 16 == 0 && p.H % 16 == 0;
  const void* fn = !p.bf16 ? reinterpret_cast<const void*>(small_builder<false, false>)
                   : mma   ? reinterpret_cast<const void*>(small_builder<true, true>)
                           : reinterpret_cast<const void*>(small_builder<true, false>);
  cudaError_t e = ensure_dynamic_smem(fn, P.bytes);
  if (e != cudaSuccess) return e;
  Params pp = p;
  Plan PP = P;
  void* args[] = {&pp, &PP};
  return cudaLaunchCooperativeKernel(fn, dim3(static_cast<unsigned>(P.G)), dim3(kThreads), args, P.bytes, stream);
}

}  // namespace dt
