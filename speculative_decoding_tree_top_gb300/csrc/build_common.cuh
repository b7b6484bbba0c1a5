// Pieces shared by the two tree-builder kernels of libdominotree (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <math.h>

#include "dt_internal.cuh"

namespace dt {

constexpr int kSmallMaxB = 8;  // batches up to this size use the all-SM, one-barrier-per-step builder
constexpr int kWaveJobs = 8;   // small-batch builder: expansions per wave over the whole batch
constexpr int kSpareSlots = 16;  // expansion slots per request beyond the n that best-first needs (speculation)

// Expansion slots of a request: the root (slot 0) and every node whose children were computed, speculatively or
// not. Best-first needs at most n (the root and the first n - 1 pops); the rest bound the speculative waste.
__host__ __device__ inline int expansion_slots(int n) { return n + kSpareSlots; }

// A known node of the lookahead builders: an entry of a request's frontier, or of the children list of an expanded
// node that has not been popped yet; 16 bytes.
struct alignas(16) Node {
  float score;
  int token;
  int seq;      // insertion order; in the children list of an unpopped node: the candidate index m
  short pslot;  // expansion slot of the parent (0 = the root)
  short xslot;  // expansion slot of this node, -1 while its children are unknown
};

__device__ __forceinline__ bool before(const Node& a, const Node& b) {
  const bool seq_first = a.seq < b.seq;
  const bool tok_first = (a.token < b.token) | ((a.token == b.token) & seq_first);
  return (a.score > b.score) | ((a.score == b.score) & tok_first);
}

// One expansion: the GRU step of a node (unless it is the root) and its children's scores.
struct Job {
  int b;        // request
  int xslot;    // the node's expansion slot: where its hidden state and children go
  int pslot;    // its parent's slot (-1 for the root, whose hidden state is h0)
  int token;    // its token: the GRU input
  int depth;    // its depth: the children take block position `depth`
  float score;  // its cumulative score
  int aux[2];   // aux[0], small-batch builder: 1 + the node's candidate index among the root's children when wave 0
                // expands it speculatively (its score is known only once the root's children are scored), else 0;
                // aux[1], a lookahead pick: 1 + the index of its entry in the request's children lists (its parent's
                // list), 0 when it sits in the merged list
};

// Expansions of one request at one block position, consecutive in a wave's packed list: they share the M correction
// rows of that position (large-batch builder).
struct JobGroup {
  int start;  // first expansion in the packed list
  int count;  // expansions (at most the lookahead width)
  int b;      // request
  int depth;  // depth of the expanded nodes: their children take block position `depth`
};

// Warp-wide best of one candidate per lane (`has` false: none), in pop order: higher score (-0.0 equal to +0.0),
// then lower token, then lower insertion index, then lower lane. One warp reduction picks the lane when the best
// score is held by one lane only (the common case); ties take two more reductions. Returns the lane (-1 if no lane
// has a candidate) and gives every lane the winner's `word` in `won` (one shuffle: the walk needs only a packed
// summary of the winner in every lane; the winning lane still holds its whole node).
__device__ __forceinline__ int warp_pick(bool has, const Node& e, uint32_t word, uint32_t& won) {
  const uint32_t sk = has ? key_of_f32(__float_as_uint(e.score)) : 0u;  // keys of real scores are >= 1
  const uint32_t ms = __reduce_max_sync(0xFFFFFFFFu, sk);
  if (ms == 0u) return -1;
  const bool c1 = sk == ms;
  const unsigned top = __ballot_sync(0xFFFFFFFFu, c1);
  int wl;
  if ((top & (top - 1u)) == 0u) {
    wl = __ffs(top) - 1;
  } else {
    const uint32_t mt = __reduce_min_sync(0xFFFFFFFFu, c1 ? static_cast<uint32_t>(e.token) : 0xFFFFFFFFu);
    const bool c2 = c1 && static_cast<uint32_t>(e.token) == mt;
    const uint32_t mq = __reduce_min_sync(0xFFFFFFFFu, c2 ? static_cast<uint32_t>(e.seq) : 0xFFFFFFFFu);
    const bool c3 = c2 && static_cast<uint32_t>(e.seq) == mq;
    wl = __ffs(__ballot_sync(0xFFFFFFFFu, c3)) - 1;
  }
  won = __shfl_sync(0xFFFFFFFFu, word, wl);
  return wl;
}
// The winner's summary: its expansion slot (-1: not expanded) in the low half, its depth in the high half.
__device__ __forceinline__ uint32_t pick_word(int xslot, int depth) {
  return (static_cast<uint32_t>(xslot) & 0xFFFFu) | (static_cast<uint32_t>(depth) << 16);
}
__device__ __forceinline__ int word_xslot(uint32_t w) { return static_cast<int>(static_cast<short>(w & 0xFFFFu)); }
__device__ __forceinline__ int word_depth(uint32_t w) { return static_cast<int>(w >> 16); }

// A request's best-first bookkeeping.
struct ReqCtl {
  int s;          // nodes popped
  int fb;         // which buffer of the merged list is current
  int seq_next;   // insertion index of the next child that joins the frontier
  int next_slot;  // expansion slots in use (the root holds slot 0)
  int njobs;      // expansions picked for the next wave
  int pad[3];
};

// The frontier of a request is the union of up to 32 sorted sources, one per lane of the warp that works on it:
// lane 0 walks the merged list, lane l > 0 the ranked children list of a popped node (slot `src`), whose entry m
// has insertion index base + m and depth `dep`. An idle lane has src = -1.
struct LaneSrc {
  int src;   // -2: the merged list, -1: none, >= 0: the children list of that slot
  int idx;   // next entry
  int cnt;   // entries
  int base;  // insertion index of the list's candidate 0
  int dep;   // depth of the list's entries (-1 for the merged list: read from the parent's slot)
  int pad[3];
};

struct PopRec {  // a popped node, as the outputs need it
  int token;
  int parent;  // while building: the expansion slot of the parent; resolve_parents turns it into its pop index
  int depth;
  float score;
};

// One request's state as the warp that pops and picks sees it (shared memory).
struct ReqView {
  ReqCtl* ctl;
  LaneSrc* lanes;  // [32]
  Node* merged;    // [2][n]
  Node* kids;      // [X][KM] ranked children of every expanded slot
  int* kcount;     // [X] entries kept in each children list
  int* popidx;     // [X] pop index of the slot's node (-1: the root, -2: not popped)
  int* sdepth;     // [X] depth of the slot's node
  PopRec* pops;    // [n]
};

// A lane's view of its source: the head entry, in registers.
struct Cursor {
  Node hd;
  bool has;
};

// Pop records hold the parent's expansion slot while a request is being built; once every pop is known this turns
// them into pop indices (-1 for children of the root). Called by the threads of one block, followed by a barrier.
__device__ __forceinline__ void resolve_parents(PopRec* pops, const int* popidx, int n, int t, int nthreads) {
  for (int i = t; i < n; i += nthreads) pops[i].parent = popidx[pops[i].parent];
}

// The default of request_step's pick hook: nothing happens when a pick is made.
struct NoPickHook {
  __device__ __forceinline__ void operator()(int, const Job&) const {}
};

// Called by one whole warp for request b once its wave's expansions are known. Pops best-first while the best node
// of the frontier needs no expansion (a leaf of the depth limit, or the n-th pop) or is already expanded; then walks
// on in the order best-first would follow on what is known (the frontier, plus the children of nodes expanded but
// not popped yet, with the insertion indices they would get) and picks up to `kla` unexpanded nodes for the next
// wave, the blocked best first. A pick takes an expansion slot; picks after the first keep enough slots free for
// every pop still to come. The pops are exact whatever the picks: a pick only decides when children become known.
// `on_pick(q, job)` runs in the lane that makes the q-th pick, as soon as it is made (the small-batch builder starts
// the pick's input copies there, while the walk goes on).
template <class OnPick = NoPickHook>
__device__ inline void request_step(const ReqView& R, int b, int n, int M, int maxd, int X, int KM, int kla,
                                    Job* jobs_out, WsHeader* hdr, const OnPick& on_pick = OnPick()) {
  const int lane = threadIdx.x & 31;
  ReqCtl st = *R.ctl;
  LaneSrc ls = R.lanes[lane];
  if (ls.src >= 0 && ls.cnt < 0) ls.cnt = R.kcount[ls.src];  // the root's list, attached at launch, filled in wave 0
  Node* mg = R.merged + static_cast<size_t>(st.fb) * n;
  // Every lane keeps its source's head entry and that entry's depth (its list's, or for the merged list one more
  // than its parent's) in registers. A lane whose source moved (`go`) reloads them with predicated loads: there is no
  // divergent branch in the walk's common steps, which run as one chain of warp-wide operations.
  auto reload = [&](const LaneSrc& q, Cursor& c, int& dep, bool go) {
    const bool has = q.src != -1 && q.idx < q.cnt;
    const Node* base = q.src >= 0 ? R.kids + static_cast<size_t>(q.src) * KM : mg;
    Node h = c.hd;
    if (go && has) h = base[q.idx];
    if (go && has && q.src >= 0) h.seq += q.base;
    int d = dep;
    if (go && has) d = q.dep >= 0 ? q.dep : R.sdepth[h.pslot] + 1;
    if (go) {
      c.hd = h;
      c.has = has;
      dep = d;
    }
  };
  auto live = [](const LaneSrc& q) { return q.src != -1 && q.idx < q.cnt; };
  Cursor cu;
  cu.hd = Node{0.f, 0, 0, 0, -1};
  cu.has = false;
  int hdep = 0;
  reload(ls, cu, hdep, true);
  while (st.s < n) {
    uint32_t won;
    const int wl = warp_pick(cu.has, cu.hd, pick_word(cu.hd.xslot, cu.has ? hdep : 0), won);
    if (wl < 0) {  // unreachable when n <= the size of the depth-limited tree (checked on the host)
      if (lane == 0) record_error(hdr, DT_ERR_INVALID_ARG);
      break;
    }
    const int depth = word_depth(won), xs = word_xslot(won);
    const bool need = (st.s + 1 < n) && (depth < maxd);
    if (need && xs < 0) break;  // its children are not known yet: the next wave expands it
    const bool me = lane == wl;  // the winning lane records the pop and moves on in its list
    if (me) R.pops[st.s] = PopRec{cu.hd.token, cu.hd.pslot, depth, cu.hd.score};
    if (me && need) R.popidx[xs] = st.s;
    ls.idx += me ? 1 : 0;
    bool go = me;
    if (need) {
      const int x = xs;
      const int kc = R.kcount[x];
      if (kc > 0) {
        unsigned idle = __ballot_sync(0xFFFFFFFFu, lane > 0 && !live(ls));
        if (idle == 0u) {
          // Every lane walks a live list: fold the shortest into the merged list, keeping what can still be popped.
          const unsigned rem = lane > 0 ? static_cast<unsigned>(ls.cnt - ls.idx) : 0xFFFFFFFFu;
          const unsigned key = __reduce_min_sync(0xFFFFFFFFu, lane > 0 ? (rem << 5) | lane : 0xFFFFFFFFu);
          const int L = static_cast<int>(key & 31u);
          const int i0 = __shfl_sync(0xFFFFFFFFu, ls.idx, 0), c0 = __shfl_sync(0xFFFFFFFFu, ls.cnt, 0);
          const int sL = __shfl_sync(0xFFFFFFFFu, ls.src, L), iL = __shfl_sync(0xFFFFFFFFu, ls.idx, L);
          const int cL = __shfl_sync(0xFFFFFFFFu, ls.cnt, L), bL = __shfl_sync(0xFFFFFFFFu, ls.base, L);
          const Node* la = mg + i0;
          const Node* lb = R.kids + static_cast<size_t>(sL) * KM + iL;
          const int na = c0 - i0, nb = cL - iL, limit = n - st.s - 1;
          Node* out = R.merged + static_cast<size_t>(st.fb ^ 1) * n;
          for (int k = lane; k < na + nb; k += 32) {
            Node v;
            int lo = 0, hi, pos;
            if (k < na) {
              v = la[k];
              hi = nb;
              while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                Node c = lb[mid];
                c.seq += bL;
                if (before(c, v)) lo = mid + 1;
                else hi = mid;
              }
              pos = k + lo;
            } else {
              v = lb[k - na];
              v.seq += bL;
              hi = na;
              while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (before(la[mid], v)) lo = mid + 1;
                else hi = mid;
              }
              pos = (k - na) + lo;
            }
            if (pos < limit) out[pos] = v;
          }
          __syncwarp();
          st.fb ^= 1;
          mg = out;
          if (lane == 0) ls = LaneSrc{-2, 0, min(na + nb, limit), 0, -1, {0, 0, 0}};
          if (lane == L) ls.src = -1;
          go = go || lane == 0 || lane == L;
          idle = __ballot_sync(0xFFFFFFFFu, lane > 0 && !live(ls));
        }
        const int nl = __ffs(idle) - 1;
        if (lane == nl) ls = LaneSrc{x, 0, kc, st.seq_next, depth + 1, {0, 0, 0}};
        go = go || lane == nl;
      }
      st.seq_next += M;
    }
    reload(ls, cu, hdep, go);
    ++st.s;
  }
  R.lanes[lane] = ls;
  // lookahead: the same walk on a copy of the lanes, taking unexpanded nodes as picks instead of stopping there
  int njobs = 0;
  if (st.s < n) {
    LaneSrc ss = ls;
    Cursor sc = cu;
    int sdep = hdep;
    int sseq = st.seq_next;
    for (int sim = st.s; sim < n - 1 && njobs < kla; ++sim) {
      uint32_t won;
      const int wl = warp_pick(sc.has, sc.hd, pick_word(sc.hd.xslot, sc.has ? sdep : 0), won);
      if (wl < 0) break;
      const int depth = word_depth(won), xs = word_xslot(won);
      const bool pick = depth < maxd && xs < 0;
      if (pick) {
        const bool allowed = njobs == 0 || st.next_slot + 1 + (n - 1 - st.s) <= X;
        if (!allowed || st.next_slot >= X) break;
      }
      const bool me = lane == wl;
      if (me && pick) {  // the winning lane takes the pick
        const int x = st.next_slot;
        Node* at = ss.src == -2 ? mg + ss.idx : R.kids + static_cast<size_t>(ss.src) * KM + ss.idx;
        at->xslot = static_cast<short>(x);  // marked as expanded in the list it lives in
        R.sdepth[x] = depth;
        R.popidx[x] = -2;
        R.kcount[x] = 0;
        const int kid = ss.src >= 0 ? 1 + ss.src * KM + ss.idx : 0;
        const Job jb{b, x, sc.hd.pslot, sc.hd.token, depth, sc.hd.score, {0, kid}};
        jobs_out[njobs] = jb;
        on_pick(njobs, jb);
      }
      ss.idx += me ? 1 : 0;  // and moves on in its list
      bool go = me;
      if (pick) {
        ++st.next_slot;
        ++njobs;
      }
      if (depth < maxd && xs >= 0) {  // expanded but not popped: its children join the walk
        const int kc = R.kcount[xs];
        if (kc > 0) {
          const unsigned idle = __ballot_sync(0xFFFFFFFFu, lane > 0 && !live(ss));
          if (idle == 0u) break;
          const int nl = __ffs(idle) - 1;
          if (lane == nl) ss = LaneSrc{xs, 0, kc, sseq, depth + 1, {0, 0, 0}};
          go = go || lane == nl;
        }
        sseq += M;
      }
      reload(ss, sc, sdep, go);
    }
  }
  if (st.s < n && njobs == 0 && lane == 0) record_error(hdr, DT_ERR_INVALID_ARG);  // no slot left (unreachable)
  st.njobs = njobs;
  __syncwarp();
  if (lane == 0) *R.ctl = st;
}

struct Params {
  int B, K, V, M, n, max_depth, H, E;
  float T_eff;
  bool bf16;
  const int32_t* ids;
  const float* vals;
  const float* h0;
  const void* emb;
  const void* w_ih;
  const void* w_hh;
  const void* b_ih;
  const void* b_hh;
  const void* w_c;
  int32_t* tokens;
  int32_t* parents;
  int32_t* depth;
  float* scores;
  uint8_t* mask;
  WsHeader* hdr;
  float* hs;        // [B][xslots][H] hidden state of every expansion slot (slot 0: h0)
  long long* acc;   // [xslots][kWaveJobs][M] fixed-point correction accumulators, acc_stride words apart (small)
  int acc_stride;
  unsigned char* rstate;  // [B] per-request best-first state blocks of req_layout(...).bytes (large-batch builder)
  Job* joblist;     // [2][B * lookahead] the expansions of a wave, packed (large-batch builder)
  int* jobcount;    // [xslots + 2] expansions per wave (large-batch builder)
  JobGroup* grouplist;  // [2][B * lookahead] the wave's expansions of one request at one depth (large-batch builder)
  int* groupcount;      // [xslots + 2] groups per wave (large-batch builder)
  int ctl_conc;     // large-batch builder: requests a CTA steps at once in the control phase
  int ctl_stage;    // ... and its staging slots for the picks' activation rows (tcgen05 GRU)
  bool group_mma;   // large-batch builder: a group's corrections as one tensor-core product (bf16, H % 16 == 0,
                    // M <= 128, the group's rows in shared memory)
  unsigned short* xact;  // [B * lookahead][E + 2H] bf16 GRU inputs of the next wave's expansions (tensor-core GRU)
  bool xact_on;     // the control phase writes xact (the tensor-core GRU runs)
  uint64_t timeout_ns;
  bool rows_smem;   // large-batch builder: the M gathered correction rows of a node are staged in shared memory
  int lookahead;    // expansions a request may run per wave (1 = one pop at a time)
  int xslots;       // expansion slots per request (expansion_slots(n))
  int* hs_count;    // [xslots] per wave, the CTAs whose hidden-state units and correction shares are in (small batch)
  float* gru_part;  // [gru_tiles][kGruSplits][128][128] K-split partial gate sums of the tensor-core GRU
  unsigned* gru_ticket;  // [gru_tiles] CTAs of a tile that stored their partials in the current wave (tensor-core GRU)
  int gru_tiles;
};

__device__ __forceinline__ float ldw(const void* p, bool bf16, size_t i) {
  if (bf16) {
    const unsigned short u = __ldg(static_cast<const unsigned short*>(p) + i);
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
  }
  return __ldg(static_cast<const float*>(p) + i);
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

// Candidate ids come from the caller (normally dt_topm); one outside [0, V) is recorded as DT_ERR_INVALID_ARG and
// replaced by 0, so that no gather ever leaves the weight arrays.
__device__ __forceinline__ int valid_id(const Params& p, int id) {
  if (static_cast<unsigned>(id) >= static_cast<unsigned>(p.V)) {
    record_error(p.hdr, DT_ERR_INVALID_ARG);
    return 0;
  }
  return id;
}

// One warp: the dot products of 8 consecutive rows m0 .. m0 + 7 (those < M) with h, for the rows of a gathered slice
// in shared memory (`rows`, [M][H]) or, when rows == nullptr, the correction rows w[ids[m]] in global memory. The
// lane's share of h is loaded once and used for all 8 rows, whose sums are 8 independent chains (same per-lane order
// and shuffle tree as one row at a time, so the results are identical). out[j] is valid in every lane.
__device__ __forceinline__ void warp_dot_rows8(const void* rows, const void* w, const int* ids, bool bf16, int m0,
                                               int M, const float* h, int H, float (&out)[8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 8; ++j) out[j] = 0.f;
  if (bf16) {
    const int G = H / 8;  // 16-byte groups per row
    for (int g = lane; g < G; g += 32) {
      const float4 ha = *reinterpret_cast<const float4*>(h + g * 8), hb = *reinterpret_cast<const float4*>(h + g * 8 + 4);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int m = m0 + j;
        if (m >= M) break;
        const uint4 v = rows ? reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(rows) +
                                                              static_cast<size_t>(m) * H)[g]
                             : __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(w) +
                                                                    static_cast<size_t>(ids[m]) * H) + g);
        float a = out[j];
        a = fmaf(__uint_as_float(v.x << 16), ha.x, a);
        a = fmaf(__uint_as_float(v.x & 0xFFFF0000u), ha.y, a);
        a = fmaf(__uint_as_float(v.y << 16), ha.z, a);
        a = fmaf(__uint_as_float(v.y & 0xFFFF0000u), ha.w, a);
        a = fmaf(__uint_as_float(v.z << 16), hb.x, a);
        a = fmaf(__uint_as_float(v.z & 0xFFFF0000u), hb.y, a);
        a = fmaf(__uint_as_float(v.w << 16), hb.z, a);
        a = fmaf(__uint_as_float(v.w & 0xFFFF0000u), hb.w, a);
        out[j] = a;
      }
    }
  } else {
    const int G = H / 4;
    for (int g = lane; g < G; g += 32) {
      const float4 hv = *reinterpret_cast<const float4*>(h + g * 4);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int m = m0 + j;
        if (m >= M) break;
        const float4 v = rows ? reinterpret_cast<const float4*>(static_cast<const float*>(rows) +
                                                                static_cast<size_t>(m) * H)[g]
                              : __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(w) +
                                                                      static_cast<size_t>(ids[m]) * H) + g);
        float a = out[j];
        a = fmaf(v.x, hv.x, a);
        a = fmaf(v.y, hv.y, a);
        a = fmaf(v.z, hv.z, a);
        a = fmaf(v.w, hv.w, a);
        out[j] = a;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int j = 0; j < 8; ++j) out[j] += __shfl_xor_sync(0xFFFFFFFFu, out[j], o);
}

// A job's children ranked among themselves by one warp: a bitonic sort of their sibling keys (larger first; equal
// keys, possible only when a row repeats an id, by the lower candidate index) over 32 * R elements, element i in
// register i / 32 of lane i % 32; padding (index >= M) has key 0 and sorts last. The first kc go to out[0 .. kc).
// kPacked (token ids below 2^25, M <= 128): the candidate index rides in the key's low 7 bits, under the token's 25
// (the key's order is unchanged: score, then token ascending, then index ascending), so the sort moves one 64-bit
// word per element instead of a word and an index.
constexpr int kPackTokenBits = 25;
template <int R, bool kPacked = false>
__device__ __forceinline__ void rank_children_warp(const Node* kr, const unsigned long long* kk, int M, Node* out,
                                                   int kc) {
  const int lane = threadIdx.x & 31;
  unsigned long long k[R];
  int m[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = 32 * r + lane;
    k[r] = m[r] < M ? kk[m[r]] : 0ull;
    if (kPacked && m[r] < M)  // score bits, then 2^25 - 1 - token, then 127 - index
      k[r] = (k[r] & 0xFFFFFFFF00000000ull) |
             ((k[r] & ((1ull << kPackTokenBits) - 1ull)) << 7) | static_cast<unsigned long long>(127 - m[r]);
  }
  auto first = [](unsigned long long ka, int ma, unsigned long long kb, int mb) {
    return kPacked ? ka > kb : (ka > kb) | ((ka == kb) & (ma < mb));
  };
#pragma unroll
  for (int size = 2; size <= 32 * R; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) {
      if (j >= 32) {  // both elements of every pair sit in one lane: registers r and r + j / 32
        const int jr = j >> 5;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (r & jr) continue;
          const int r2 = r | jr;
          const bool desc = ((32 * r + lane) & size) == 0;  // this block is sorted larger-first
          if (first(k[r], m[r], k[r2], m[r2]) != desc) {
            const unsigned long long tk = k[r];
            k[r] = k[r2];
            k[r2] = tk;
            if (!kPacked) {
              const int tm = m[r];
              m[r] = m[r2];
              m[r2] = tm;
            }
          }
        }
      } else {  // the pair spans lanes lane and lane ^ j, same register
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const unsigned long long ok = __shfl_xor_sync(0xFFFFFFFFu, k[r], j);
          const int om = kPacked ? 0 : __shfl_xor_sync(0xFFFFFFFFu, m[r], j);
          const bool desc = ((32 * r + lane) & size) == 0;
          const bool lower = (lane & j) == 0;
          const bool mine_first = first(k[r], m[r], ok, om);
          if (mine_first != (lower == desc)) {
            k[r] = ok;
            if (!kPacked) m[r] = om;
          }
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int mi = kPacked ? 127 - static_cast<int>(k[r] & 127ull) : m[r];
    if (32 * r + lane < kc) out[32 * r + lane] = kr[mi];
  }
}
// The ranking of M <= 128 children, packed when every token id fits the packed key.
__device__ __forceinline__ void rank_children(const Node* kr, const unsigned long long* kk, int M, int V, Node* out,
                                              int kc) {
  if (V <= (1 << kPackTokenBits)) {
    if (M <= 32) rank_children_warp<1, true>(kr, kk, M, out, kc);
    else if (M <= 64) rank_children_warp<2, true>(kr, kk, M, out, kc);
    else rank_children_warp<4, true>(kr, kk, M, out, kc);
  } else {
    if (M <= 32) rank_children_warp<1>(kr, kk, M, out, kc);
    else if (M <= 64) rank_children_warp<2>(kr, kk, M, out, kc);
    else rank_children_warp<4>(kr, kk, M, out, kc);
  }
}

// A request's best-first state as one contiguous block (the large-batch builder keeps it in the workspace between
// waves and works on it in shared memory; offsets are multiples of 16 so the block moves as one bulk copy).
struct ReqLayout {
  size_t ctl, lanes, jobs, merged, kids, kcount, popidx, sdepth, pops, bytes;
};
__host__ __device__ inline ReqLayout req_layout(int n, int X, int KM, int kla) {
  ReqLayout L{};
  size_t o = 0;
  auto take = [&o](size_t bytes) {
    const size_t at = o;
    o = (o + bytes + 15) / 16 * 16;
    return at;
  };
  L.ctl = take(sizeof(ReqCtl));
  L.lanes = take(sizeof(LaneSrc) * 32);
  L.jobs = take(sizeof(Job) * kla);
  L.merged = take(sizeof(Node) * 2 * static_cast<size_t>(n));
  L.kids = take(sizeof(Node) * static_cast<size_t>(X) * KM);
  L.kcount = take(sizeof(int) * X);
  L.popidx = take(sizeof(int) * X);
  L.sdepth = take(sizeof(int) * X);
  L.pops = take(sizeof(PopRec) * static_cast<size_t>(n));
  L.bytes = o;
  return L;
}
__host__ __device__ inline ReqView req_view(unsigned char* base, const ReqLayout& L) {
  return ReqView{reinterpret_cast<ReqCtl*>(base + L.ctl), reinterpret_cast<LaneSrc*>(base + L.lanes),
                 reinterpret_cast<Node*>(base + L.merged), reinterpret_cast<Node*>(base + L.kids),
                 reinterpret_cast<int*>(base + L.kcount), reinterpret_cast<int*>(base + L.popidx),
                 reinterpret_cast<int*>(base + L.sdepth), reinterpret_cast<PopRec*>(base + L.pops)};
}
constexpr int kLargeLookahead = 8;  // the large-batch builder's most expansions per request and wave
constexpr int kLargeDefault = 4;    // ... and its default (kLargeLookahead once a wave holds 128 requests or more)

// Builder region of the workspace, after the top-M region (one workspace serves the whole round): the hidden states
// of every expansion slot [B][X][H] fp32; for small batches the per-wave fixed-point correction accumulators and the
// per-slot publication counters; for larger ones the per-request state blocks, the packed job lists of two waves and
// the per-wave job counts.
struct BuildLayout {
  size_t hs, acc, hs_count, rstate, joblist, jobcount, grouplist, groupcount, xact, gru_part, gru_ticket, bytes;
  int gru_tiles;
};

// The tensor-core GRU of the large-batch builder sums K as kGruSplits partials in a fixed order. A wave of at most
// kGruSpreadTiles tiles (128 expansions x 32 units) spreads the partials over CTAs and adds them up from the
// workspace; the tiles a wave of B * kLargeLookahead expansions can have, capped there, size that region.
constexpr int kGruSplits = 4;
constexpr int kGruSpreadTiles = 128;
constexpr int kGruTileRows = 128, kGruTileUnits = 32;
inline int gru_spread_tiles(int B, int H) {
  const long long t = (static_cast<long long>(B) * kLargeLookahead + kGruTileRows - 1) / kGruTileRows *
                      (H / kGruTileUnits);
  return static_cast<int>(t < kGruSpreadTiles ? t : kGruSpreadTiles);
}

// Words between two correction accumulators: one 128-byte line each, so that the shares of a wave (every SM adds
// one to every candidate's slot) spread over the L2 slices, unless that takes more than 64 MB.
__host__ __device__ inline int acc_stride(int M, int n) {
  return static_cast<size_t>(expansion_slots(n)) * kWaveJobs * M * 128u <= (64u << 20) ? 16 : 1;
}

inline BuildLayout build_layout(int B, int K, int V, int M, int n, int H, int E) {
  BuildLayout L{};
  const size_t X = static_cast<size_t>(expansion_slots(n));
  const int KM = M < n ? M : n;
  L.hs = topm_layout(B, K, V, M).bytes;
  const size_t acc_bytes = B <= kSmallMaxB ? sizeof(long long) * X * kWaveJobs * M * acc_stride(M, n) : 0;
  L.acc = align_up(L.hs + sizeof(float) * static_cast<size_t>(B) * X * H);
  L.hs_count = align_up(L.acc + acc_bytes);  // the per-wave counters
  L.rstate = align_up(L.hs_count + (B <= kSmallMaxB ? sizeof(int) * X : 0));
  // both builders may run for small batches (the small one needs shared memory the device may not have)
  L.joblist = align_up(L.rstate + req_layout(n, static_cast<int>(X), KM, kLargeLookahead).bytes * B);
  L.jobcount = align_up(L.joblist + sizeof(Job) * 2 * static_cast<size_t>(B) * kLargeLookahead);
  L.grouplist = align_up(L.jobcount + sizeof(int) * (X + 2));
  L.groupcount = align_up(L.grouplist + sizeof(JobGroup) * 2 * static_cast<size_t>(B) * kLargeLookahead);
  // the tensor-core GRU's A operand: one bf16 row [emb | hi(h_parent) | lo(h_parent)] per expansion of a wave
  L.xact = align_up(L.groupcount + sizeof(int) * (X + 2));
  L.gru_part = align_up(L.xact + sizeof(unsigned short) * static_cast<size_t>(B) * kLargeLookahead * (E + 2 * H));
  L.gru_tiles = gru_spread_tiles(B, H);
  L.gru_ticket = align_up(L.gru_part + sizeof(float) * static_cast<size_t>(L.gru_tiles) * kGruSplits * kGruTileRows *
                                           4 * kGruTileUnits);
  L.bytes = align_up(L.gru_ticket + sizeof(unsigned) * static_cast<size_t>(L.gru_tiles));
  return L;
}


// The small-batch builder (build_small.cu). Returns false when its shared-memory plan does not fit this device
// (the caller then uses the general builder).
bool small_builder_fits(const Params& p, const DeviceInfo& di);
cudaError_t launch_small_builder(const Params& p, const DeviceInfo& di, cudaStream_t stream);

}  // namespace dt
