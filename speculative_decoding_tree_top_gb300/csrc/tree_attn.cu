// dt_tree_attention — the verify pass's attention over the prefix and the draft tree with the ancestor-only mask.
//
// Method: blog.captcha.la, "Methodology — deep read" (the prefix-closed tree is verified in a single target forward
// pass with an unmodified ancestor-only causal mask, borrowed from DDTree/SpecInfer); gist.science, "Composants
// Clés — Vérification" (standard tree attention, unchanged and lossless). For request b, query head h and tree node
// i the visible keys are the L prefix positions and the tree positions L + t with mask[b][i][t] = 1;
// out = softmax(scale q.k) v over them; query head h reads key/value head h / (Hq / Hkv).
//
// GB300 design (flash decoding): the n tree nodes of the G = Hq / Hkv query heads that share a key/value head are
// one block of G n <= 64 query rows, so each key and value row is read once per (request, key/value head) and feeds
// 64 rows of dot products: a dense contraction on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate).
// The key blocks of all (request, key/value head) pairs, flattened, are split evenly over four CTAs per SM (a CTA's
// share may span two pairs: one segment each); a CTA streams a segment's key and value rows through a two-stage
// cp.async ring in blocks of 32 (55 KB, 128 registers), keeps the running max and sum of every query row
// (online softmax, base 2) and its unnormalised output in registers, and writes them as the segment's partial; a
// second launch combines the segments of each row. Memory bound: the key and value rows are the bytes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "dt_internal.cuh"

namespace dt {
namespace {

constexpr int kD = 128;           // head dimension
constexpr int kRows = 64;         // query rows per CTA: G x n, padded
constexpr int kBlockKeys = 32;    // keys per ring stage (small: four CTAs fit an SM)
constexpr int kThreadsA = 128;    // four warps, 16 query rows each
constexpr int kPitch = kD + 8;    // shared-memory row pitch in bf16 (272 bytes: conflict-free ldmatrix)
constexpr int kMaxNodes = 64;
constexpr int kStagesA = 2;      // key/value ring stages: one block in flight while one is consumed

struct TaParams {
  int B, n, L, T, Hq, Hkv, G, R;
  int nb;              // key blocks of 32 per (request, key/value head)
  int grid, maxseg;    // CTAs of the partial launch; partial slots per (request, key/value head)
  long long work;      // all key blocks: (B Hkv) nb, split evenly over the CTAs
  const unsigned short* q;   // [B][n][Hq][kD] bf16
  const unsigned short* k;   // [B][Hkv][T][kD] bf16
  const unsigned short* v;   // [B][Hkv][T][kD] bf16
  const uint8_t* mask;       // [B][n][n]
  float scale_log2;          // scale * log2(e)
  float* part;               // [B Hkv][maxseg][kRows][kD] unnormalised outputs of each segment
  float* ml;                 // [B Hkv][maxseg][kRows][2] running max (base 2) and sum
  float* out;                // [B][n][Hq][kD]
};

struct TaSmem {
  __nv_bfloat16 q[kRows * kPitch];
  __nv_bfloat16 k[kStagesA][kBlockKeys * kPitch];
  __nv_bfloat16 v[kStagesA][kBlockKeys * kPitch];
  uint8_t mask[kMaxNodes * kMaxNodes];
};

__device__ __forceinline__ void cp16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4(const void* p, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(const void* p, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The CTA whose even share of the flattened key blocks holds block x: CTA c takes [c W / G, (c + 1) W / G).
__host__ __device__ __forceinline__ int block_owner(long long x, long long W, int G) {
  return static_cast<int>(((x + 1) * G - 1) / W);
}

// Key and value rows [k0, k0 + 32) of one (request, key/value head) into ring stage s; rows past T read as zero.
__device__ __forceinline__ void load_kv(const TaParams& p, TaSmem& S, int s, size_t kvbase, int k0) {
  for (int c = threadIdx.x; c < kBlockKeys * (kD / 8); c += kThreadsA) {
    const int r = c >> 4, col = (c & 15) * 8, key = k0 + r;  // 16 chunks of 16 bytes per row
    const bool ok = key < p.T;
    const size_t off = (kvbase + (ok ? key : 0)) * kD + col;
    cp16(&S.k[s][r * kPitch + col], p.k + off, ok);
    cp16(&S.v[s][r * kPitch + col], p.v + off, ok);
  }
}

// CTA c takes an even share of the flattened (request, key/value head, key block) space; each run of its share
// within one (request, key/value head) is a segment, whose partial attention for the 64 query rows goes to that
// pair's slot (c - the owner of the pair's first block).
__global__ void __launch_bounds__(kThreadsA, 4) tree_attn_partial(TaParams p) {
  extern __shared__ float4 smem_f4[];
  TaSmem& S = *reinterpret_cast<TaSmem*>(smem_f4);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31, g = lane >> 2, tq = lane & 3;
  const long long x1 = (static_cast<long long>(blockIdx.x) + 1) * p.work / p.grid;
  for (long long x = static_cast<long long>(blockIdx.x) * p.work / p.grid; x < x1;) {
  const int pair = static_cast<int>(x / p.nb), b = pair / p.Hkv, kvh = pair % p.Hkv;
  const long long pfirst = static_cast<long long>(pair) * p.nb;
  const int bend = static_cast<int>(min(x1, pfirst + p.nb) - pfirst);
  const int k0 = static_cast<int>(x - pfirst) * kBlockKeys, k1 = min(bend * kBlockKeys, p.T);
  const int slot = static_cast<int>(blockIdx.x) - block_owner(pfirst, p.work, p.grid);
  x = pfirst + bend;
  const size_t kvbase = (static_cast<size_t>(b) * p.Hkv + kvh) * p.T;
  // query row r = gi n + i: query head kvh G + gi, tree node i (rows >= R read as zero)
  for (int c = t; c < kRows * (kD / 8); c += kThreadsA) {
    const int r = c >> 4, col = (c & 15) * 8;
    const bool ok = r < p.R;
    const int gi = ok ? r / p.n : 0, i = ok ? r % p.n : 0;
    cp16(&S.q[r * kPitch + col], p.q + ((static_cast<size_t>(b) * p.n + i) * p.Hq + kvh * p.G + gi) * kD + col, ok);
  }
  for (int c = t; c < p.n * p.n; c += kThreadsA) S.mask[c] = p.mask[static_cast<size_t>(b) * p.n * p.n + c];
  const int nblk = (k1 - k0 + kBlockKeys - 1) / kBlockKeys;
  for (int j = 0; j < kStagesA - 1; ++j) {  // the first blocks (the queries' copies join the first group)
    if (j < nblk) load_kv(p, S, j, kvbase, k0 + j * kBlockKeys);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }

  const int rw0 = 16 * warp + g, rw1 = rw0 + 8;  // this thread's two query rows
  const int node0 = rw0 < p.R ? rw0 % p.n : -1, node1 = rw1 < p.R ? rw1 % p.n : -1;
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  for (int blk = 0; blk < nblk; ++blk) {
    if (blk + kStagesA - 1 < nblk)
      load_kv(p, S, (blk + kStagesA - 1) % kStagesA, kvbase, k0 + (blk + kStagesA - 1) * kBlockKeys);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group %0;" ::"n"(kStagesA - 1) : "memory");  // block blk has landed
    __syncthreads();
    const __nv_bfloat16* Ks = S.k[blk % kStagesA];
    const __nv_bfloat16* Vs = S.v[blk % kStagesA];
    // S = Q K^T for the block's keys: tiles of 8 keys; the warp's 16 query rows re-read as A fragments per K step
    constexpr int kNT = kBlockKeys / 8;
    float s[kNT][4];
#pragma unroll
    for (int j = 0; j < kNT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kD / 16; ++ks) {
      uint32_t qa[4];
      ldsm_x4(&S.q[(16 * warp + (lane & 15)) * kPitch + ks * 16 + (lane >> 4) * 8], qa[0], qa[1], qa[2], qa[3]);
#pragma unroll
      for (int np = 0; np < kNT / 2; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(&Ks[(np * 16 + (lane & 7) + ((lane >> 4) << 3)) * kPitch + ks * 16 + ((lane >> 3) & 1) * 8], b0, b1,
                b2, b3);
        mma_bf16(s[2 * np], qa, b0, b1);
        mma_bf16(s[2 * np + 1], qa, b2, b3);
      }
    }
    // mask and scale (base 2), the rows' running maxima
    const int kb = k0 + blk * kBlockKeys;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = kb + nt * 8 + tq * 2 + e;
        const bool in = key < k1;
        const bool v0 = in && node0 >= 0 && (key < p.L || S.mask[node0 * p.n + (key - p.L)] != 0);
        const bool v1 = in && node1 >= 0 && (key < p.L || S.mask[node1 * p.n + (key - p.L)] != 0);
        s[nt][e] = v0 ? s[nt][e] * p.scale_log2 : -INFINITY;
        s[nt][2 + e] = v1 ? s[nt][2 + e] * p.scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, s[nt][e]);
        mx1 = fmaxf(mx1, s[nt][2 + e]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float a0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0), a1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
    float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        s[nt][e] = mn0 == -INFINITY ? 0.f : exp2f(s[nt][e] - mn0);
        s[nt][2 + e] = mn1 == -INFINITY ? 0.f : exp2f(s[nt][2 + e] - mn1);
        ls0 += s[nt][e];
        ls1 += s[nt][2 + e];
      }
    }
    l0 = l0 * a0 + ls0;  // this thread's share of the row sums (the quad adds them up at the end)
    l1 = l1 * a1 + ls1;
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      o[j][0] *= a0;
      o[j][1] *= a0;
      o[j][2] *= a1;
      o[j][3] *= a1;
    }
    // O += P V: P from the score registers (bf16), V by transposed ldmatrix
#pragma unroll
    for (int kp = 0; kp < kBlockKeys / 16; ++kp) {
      const uint32_t pa[4] = {pack_bf16(s[2 * kp][0], s[2 * kp][1]), pack_bf16(s[2 * kp][2], s[2 * kp][3]),
                              pack_bf16(s[2 * kp + 1][0], s[2 * kp + 1][1]),
                              pack_bf16(s[2 * kp + 1][2], s[2 * kp + 1][3])};
#pragma unroll
      for (int dp = 0; dp < kD / 16; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(&Vs[(kp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * kPitch + dp * 16 + (lane >> 4) * 8], b0, b1,
                  b2, b3);
        mma_bf16(o[2 * dp], pa, b0, b1);
        mma_bf16(o[2 * dp + 1], pa, b2, b3);
      }
    }
    __syncthreads();  // the stage is refilled by a later load
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
  l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
  l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
  l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);
  const size_t unit = static_cast<size_t>(pair) * p.maxseg + slot;
  float* po = p.part + unit * kRows * kD;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int col = j * 8 + tq * 2;
    *reinterpret_cast<float2*>(po + rw0 * kD + col) = make_float2(o[j][0], o[j][1]);
    *reinterpret_cast<float2*>(po + rw1 * kD + col) = make_float2(o[j][2], o[j][3]);
  }
  if (tq == 0) {
    float* pm = p.ml + unit * kRows * 2;
    pm[rw0 * 2] = m0;
    pm[rw0 * 2 + 1] = l0;
    pm[rw1 * 2] = m1;
    pm[rw1 * 2 + 1] = l1;
  }
  __syncthreads();  // the queries, mask and ring are reloaded for the next segment
  }
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
  const long long pfirst = static_cast<long long>(pair) * p.nb;
  q.nseg = block_owner(pfirst + p.nb - 1, p.work, p.grid) - block_owner(pfirst, p.work, p.grid) + 1;
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
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long rows = static_cast<long long>(p.B) * p.Hkv * p.R;
  if (p.maxseg <= kWarpRowSegs) {  // a warp per row
    const long long stride = static_cast<long long>(gridDim.x) * kCombineWarps;
    for (long long u = static_cast<long long>(blockIdx.x) * kCombineWarps + warp; u < rows; u += stride) {
      const RowRef q = row_ref(p, u);
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
  int nb, grid, maxseg;
  long long work;
  size_t part, ml, bytes;
};
// Four CTAs per SM share all key blocks evenly (a CTA takes at least one block); maxseg is the most CTAs any
// (request, key/value head) is spread over, found pair by pair.
inline TaPlan ta_plan(int B, int T, int Hkv, int sms) {
  TaPlan P{};
  const long long pairs = static_cast<long long>(B) * Hkv;
  P.nb = (T + kBlockKeys - 1) / kBlockKeys;
  P.work = pairs * P.nb;
  const long long g = 4LL * sms;
  P.grid = static_cast<int>(g < P.work ? g : P.work);
  P.maxseg = 1;
  for (long long pr = 0; pr < pairs; ++pr) {
    const int segs = block_owner((pr + 1) * P.nb - 1, P.work, P.grid) - block_owner(pr * P.nb, P.work, P.grid) + 1;
    P.maxseg = segs > P.maxseg ? segs : P.maxseg;
  }
  const size_t slots = static_cast<size_t>(pairs) * P.maxseg;
  P.part = 0;
  P.ml = align_up(sizeof(float) * slots * kRows * kD);
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
  p.nb = P.nb; p.grid = P.grid; p.maxseg = P.maxseg; p.work = P.work;
  p.q = static_cast<const unsigned short*>(q);
  p.k = static_cast<const unsigned short*>(k);
  p.v = static_cast<const unsigned short*>(v);
  p.mask = mask;
  p.scale_log2 = scale * 1.4426950408889634f;
  char* ws = static_cast<char*>(workspace);
  p.part = reinterpret_cast<float*>(ws + P.part);
  p.ml = reinterpret_cast<float*>(ws + P.ml);
  p.out = out;
  const void* fa = reinterpret_cast<const void*>(tree_attn_partial);
  if (ensure_dynamic_smem(fa, sizeof(TaSmem)) != cudaSuccess) return DT_ERR_CUDA;
  tree_attn_partial<<<static_cast<unsigned>(P.grid), kThreadsA, sizeof(TaSmem), stream>>>(p);
  const long long crows = static_cast<long long>(B) * Hkv * p.R, cper = P.maxseg <= kWarpRowSegs ? kCombineWarps : 1;
  const long long cgrid = (crows + cper - 1) / cper, ccap = static_cast<long long>(kCombinePerSm) * di.sms;
  tree_attn_combine<<<static_cast<unsigned>(cgrid < ccap ? cgrid : ccap), kCombineThreads, 0, stream>>>(p);
  return cuda_status(cudaGetLastError());
}
