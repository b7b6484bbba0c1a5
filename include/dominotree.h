/*
 * dominotree.h — C ABI of the GB300 (sm_103a) drafting-round tree builder of DominoTree.
 *
 * One drafting round of the method described in "DominoTree: Conditional Tree-Structured Drafting with Domino for
 * Speculative Decoding" (arXiv 2607.08642), as summarised by blog.captcha.la ("Methodology — deep read",
 * "Technical innovations"), zhichai.top ("DominoTree 的破局", "GPU 原生树构建器") and gist.science ("Résumé
 * Technique — Composants Clés"):
 *
 *   dt_topm         top-M candidates at each of the K block positions, from the drafter's marginal logits over
 *                   the full vocabulary ("top-M candidate restriction");
 *   dt_build_trees  best-first growth of a prefix-closed draft tree keyed by cumulative conditional
 *                   log-probability: per expanded node one GRU step along its path, the correction W_c[ids]·h on
 *                   the gathered top-M slice, a temperature-scaled log-softmax restricted to those M; emits tokens,
 *                   parents, depths, scores and the ancestor-only attention mask of the verify pass.
 *
 * Conventions for every call below
 *   - All array pointers are DEVICE pointers owned by the caller; the library allocates nothing and keeps no
 *     pointer after a call returns. Arrays are dense, row-major, with the shapes given in brackets, and must start
 *     on a 16-byte boundary.
 *   - Calls are asynchronous on `stream`; a round is dt_topm then dt_build_trees on the same stream.
 *   - Argument errors are detected on the host before anything is launched and return DT_ERR_INVALID_ARG (or
 *     DT_ERR_UNSUPPORTED for sizes outside the supported envelope); nothing is written then. A failed launch
 *     returns DT_ERR_CUDA. Problems found on the device (a barrier wait that ran out, a NaN among the logits) are
 *     recorded in the workspace's status word and read with dt_get_error.
 *   - The workspace is caller-allocated device memory of at least the size the matching *_workspace_bytes call
 *     returns, zeroed once (dt_workspace_init) before its first use; each call leaves it ready for the next one.
 *     dt_build_trees keeps its own region after the one dt_topm uses, so a workspace of
 *     dt_build_workspace_bytes(...) bytes serves both calls of a round when they are ordered on one stream. Two
 *     calls that may run concurrently need two workspaces.
 *   - No C++ exception crosses this boundary. The calls are thread-safe for distinct workspaces.
 */
#ifndef DOMINOTREE_H
#define DOMINOTREE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DT_ABI_VERSION 1

typedef enum {
  DT_OK = 0,
  DT_ERR_INVALID_ARG = 1, /* a null or misaligned pointer, sizes that contradict each other; from the
                             device (dt_get_error): a candidate id outside [0, V) given to dt_build_trees  */
  DT_ERR_UNSUPPORTED = 2, /* valid, but outside the envelope the kernels are built for (limits below)    */
  DT_ERR_CUDA = 3,        /* a CUDA runtime call failed (launch, attribute query)                        */
  DT_ERR_TIMEOUT = 4,     /* device: a grid-barrier wait ran out of its time budget; the kernel returned  */
  DT_ERR_NUMERIC = 5      /* device: a NaN was found among the logits                                    */
} dt_status;

typedef enum { DT_F32 = 0, DT_BF16 = 1 } dt_dtype;

/* Supported envelope of dt_build_trees (DT_ERR_UNSUPPORTED beyond). */
#define DT_MAX_M 1024      /* candidates per position                */
#define DT_MAX_N 1024      /* node budget                            */
#define DT_MAX_H 2048      /* GRU hidden width                       */
#define DT_MAX_E 16384     /* token-embedding width                  */

/* Drafter correction weights, shared by every request of a round. `dtype` is the storage type of all of them.
 * The GRU follows PyTorch's GRUCell layout: gate rows r | z | n (reset, update, new), each block H rows. */
typedef struct {
  int H;              /* GRU hidden width, a multiple of 8                                           */
  int E;              /* token-embedding width, a multiple of 8                                      */
  dt_dtype dtype;     /* DT_BF16 or DT_F32                                                           */
  const void* emb;    /* [V,E]   token embeddings fed to the GRU                                     */
  const void* w_ih;   /* [3H,E]  input-to-hidden weights                                             */
  const void* w_hh;   /* [3H,H]  hidden-to-hidden weights                                            */
  const void* b_ih;   /* [3H]    input bias, or NULL for zero                                        */
  const void* b_hh;   /* [3H]    hidden bias, or NULL for zero                                       */
  const void* w_c;    /* [V,H]   correction head: the corrected logit of token v is base_v + w_c[v]·h */
} dt_weights;

/* Zero a workspace before its first use (cudaMemsetAsync on `stream`). */
dt_status dt_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------------------------------
 * dt_topm — top-M candidate restriction.
 * Source: blog.captcha.la, "Methodology — deep read" and "Technical innovations" (the per-node correction only
 * sees the M tokens with the highest marginal at each depth, M = 64 in the experiments); gist.science,
 * "Composants Clés — Restriction de Candidats".
 *
 *   logits    [B,K,V] of `dtype` (DT_BF16 or DT_F32): the drafter's marginal logits, one row per (request,
 *             block position). V·sizeof(dtype) need not be a multiple of 16, but the base must be 16-byte aligned.
 *   out_ids   [B,K,M] int32: candidate token ids of each row, ordered by logit descending, ties by id ascending
 *             (-0.0 and +0.0 compare equal; -0.0 is returned as +0.0).
 *   out_vals  [B,K,M] fp32: the candidates' logits, exact copies of the stored values.
 *   1 <= M <= V, M <= DT_MAX_M. A NaN among the logits sets DT_ERR_NUMERIC on the device (the ids of that row are
 *   then unspecified but in range).
 * ------------------------------------------------------------------------------------------------------------- */
size_t dt_topm_workspace_bytes(int B, int K, int V, int M);
dt_status dt_topm(const void* logits, dt_dtype dtype, int B, int K, int V, int M, int32_t* out_ids,
                  float* out_vals, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------------------------------
 * dt_build_trees — conditional best-first draft trees for B independent requests.
 * Source: blog.captcha.la, "Methodology — deep read" (DDTree's best-first max-priority queue keyed by cumulative
 * conditional log-probability; GRU state carried along each root-to-node path; correction applied only to the
 * gathered top-M rows; fixed node budget n or max depth; prefix-closed tree verified with the ancestor-only
 * causal mask); gist.science, "Composants Clés" and "Vérification".
 *
 * Semantics (fp32 arithmetic, fp32 accumulation over bf16 or fp32 weights):
 *   root: score 0, hidden state h0[b], depth 0. A node u at depth d < max_depth is expanded into block position
 *   d: if u is not the root, h_u = GRUCell(emb[token_u], h_parent(u)); then for m < M
 *       z_m    = (topm_vals[b,d,m] + w_c[topm_ids[b,d,m]]·h_u) / T_eff,   T_eff = T if T > 0 else 1
 *       logp_m = z_m - max(z) - log(sum_j exp(z_j - max(z)))
 *   and the children (token topm_ids[b,d,m], score score_u + logp_m) join the frontier. n nodes are popped, best
 *   first: higher score, then lower token id, then earlier insertion (children enter in m order). The n-th pop is
 *   not expanded.
 *
 *   topm_ids, topm_vals  [B,K,M] from dt_topm.
 *   h0                   [B,H] fp32, the hidden state that summarises each request's accepted prefix.
 *   out_tokens           [B,n] int32, nodes in pop order (scores non-increasing).
 *   out_parents          [B,n] int32, index of the parent node, -1 for children of the root.
 *   out_depth            [B,n] int32, in 1..max_depth.
 *   out_scores           [B,n] fp32, cumulative conditional log-probability of the node's path.
 *   out_mask             [B,n,n] uint8, 1 where column j is row i itself or one of its ancestors (the root, i.e.
 *                        the accepted prefix, is visible to every node and has no column).
 *   Requires 1 <= M <= V, 1 <= max_depth <= K, 1 <= n <= number of nodes of the depth-limited M-ary tree,
 *   T finite and >= 0, and the limits DT_MAX_*.
 * ------------------------------------------------------------------------------------------------------------- */
size_t dt_build_workspace_bytes(int B, int K, int V, int M, int n, int H, int E);
dt_status dt_build_trees(int B, int K, int V, int M, int n, int max_depth, float T, const int32_t* topm_ids,
                         const float* topm_vals, const float* h0, const dt_weights* w, int32_t* out_tokens,
                         int32_t* out_parents, int32_t* out_depth, float* out_scores, uint8_t* out_mask,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------------------------------
 * dt_round — one drafting round: dt_topm into topm_ids / topm_vals, then dt_build_trees from them, on one stream.
 * Source: blog.captcha.la, "Methodology — deep read" (the round restricts each block position to its top-M marginal
 * candidates, then grows the best-first conditional tree over them); gist.science, "Composants Clés".
 *
 * Results are bit-identical to the two calls made one after the other with the same arguments; the difference is
 * that every argument of both is checked before either is launched, so an invalid round launches nothing.
 *
 *   logits, dtype        as dt_topm (marginal logits [B,K,V]).
 *   topm_ids, topm_vals  [B,K,M], written by the top-M and read by the builder (device memory the caller owns).
 *   h0, w, out_*         as dt_build_trees.
 *   workspace            one workspace of at least dt_build_workspace_bytes(B, K, V, M, n, w->H, w->E) bytes
 *                        (which covers the top-M's part), initialised once by dt_workspace_init.
 * Errors are those of dt_topm and dt_build_trees.
 * ------------------------------------------------------------------------------------------------------------- */
dt_status dt_round(const void* logits, dt_dtype dtype, int B, int K, int V, int M, int n, int max_depth, float T,
                   const float* h0, const dt_weights* w, int32_t* topm_ids, float* topm_vals, int32_t* out_tokens,
                   int32_t* out_parents, int32_t* out_depth, float* out_scores, uint8_t* out_mask, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------------------------------
 * dt_build_trees_marginal — the same best-first draft trees scored by DDTree's factorised marginals.
 * Source: blog.captcha.la, "Methodology — deep read" (DDTree scores tree nodes by factorised marginal
 * log-probabilities) and "Key findings" (the ablation that changes only the scoring function: conditional scoring
 * +9.2% throughput over marginal scoring); zhichai.top, "两条路线的困境"; gist.science, "Énoncé du Problème" (in the
 * factorised formulations a token's score depends only on its position).
 *
 * Semantics: dt_build_trees with no correction and no hidden state: a child at block position d scores
 *     score_parent + logp_m,   logp_m = z_m - max(z) - log(sum_j exp(z_j - max(z))),   z_m = topm_vals[b,d,m] / T_eff
 * with the same pops, ties, budget, depth limit and outputs (and, on the GPU, the same fp32 arithmetic as
 * dt_build_trees with w_c = 0, so the trees are identical to those). Arguments as dt_build_trees, without h0 and
 * weights; `workspace` needs only its 256-byte header (the status word; a round's workspace serves). One CTA per
 * request keeps the request's state in shared memory: sizes whose state does not fit return DT_ERR_UNSUPPORTED.
 * ------------------------------------------------------------------------------------------------------------- */
dt_status dt_build_trees_marginal(int B, int K, int V, int M, int n, int max_depth, float T, const int32_t* topm_ids,
                                  const float* topm_vals, int32_t* out_tokens, int32_t* out_parents,
                                  int32_t* out_depth, float* out_scores, uint8_t* out_mask, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------------------------------
 * dt_accept_paths — the accepted path of each draft tree after the target model's verify pass.
 * Source: blog.captcha.la, "Methodology — deep read" (one target forward pass over the tree with the ancestor-only
 * mask; the longest accepted root-to-leaf path is kept) and "Threat model" (lossless up to floating-point ties);
 * gist.science, "Composants Clés — Vérification", "Résultats Expérimentaux" (output equal to serial greedy decoding).
 *
 * Greedy verification: target_next[b,0] is the target's next token after the accepted prefix (the root), and
 * target_next[b,1+i] its next token after tree node i. From the root, the walk steps into the child whose token is
 * the target's next token at the current node (the earlier pop if two children carry it) until none does.
 *   tokens, parents     [B,n] int32, a tree as dt_build_trees emits it (every parent precedes its children; for
 *                       other input the result is unspecified but the call terminates and stays in bounds).
 *   target_next         [B,n+1] int32.
 *   out_accept_len      [B] int32: accepted draft tokens (0..max depth); the round emits out_accept_len + 1 tokens.
 *   out_path            [B,n] int32: the accepted nodes in path order, then -1. These are also the KV-compaction
 *                       indices: the verify pass's cache entry of tree position out_path[b,j] moves to prefix + j.
 *   out_bonus           [B] int32: the target's next token after the last accepted node.
 * Pointers must be 4-byte aligned device pointers. n <= DT_MAX_N.
 * ------------------------------------------------------------------------------------------------------------- */
dt_status dt_accept_paths(int B, int n, const int32_t* tokens, const int32_t* parents, const int32_t* target_next,
                          int32_t* out_accept_len, int32_t* out_path, int32_t* out_bonus, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------------------------------
 * dt_lmhead_topm — the drafter's full-vocabulary projection fused with its top-M: the logits are never written.
 * Source: blog.captcha.la, "Methodology — deep read" (the costly full-vocabulary projection, of which the per-node
 * work keeps only the M highest-marginal tokens); gist.science, "Composants Clés — Restriction de Candidats"
 * (re-running the projection W2 over the whole vocabulary is the cost that the top-M restriction avoids).
 *
 * Semantics: for every row r < R, logits[r][v] = sum_k hidden[r][k] * w_head[v][k] (no bias), computed on the tensor
 * cores as bf16 products accumulated in fp32; out_ids[r] / out_vals[r] are the M largest of those fp32 logits in
 * descending order, ties to the lower id (as dt_topm over the logits, exactly those the kernel computed).
 *   hidden       [R,D] bf16, row-major (the backbone's hidden state of each (request, block position) row).
 *   w_head       [V,D] bf16, row-major (the LM head W2, one row per vocabulary entry).
 *   out_ids      [R,M] int32; out_vals [R,M] fp32.
 *   workspace    dt_lmhead_workspace_bytes(R,D,V,M) bytes (on the current device), header initialised by
 *                dt_workspace_init; the status word reports DT_ERR_NUMERIC for a NaN logit and DT_ERR_TIMEOUT if a
 *                grid-barrier or copy wait ran out (dt_get_error).
 * Supported: dtype DT_BF16, D a multiple of 64, M <= DT_MAX_M, R <= DT_LMHEAD_MAX_ROWS. Outside it:
 * DT_ERR_UNSUPPORTED, before any launch. Two designs, chosen by the host:
 *   - when ceil(ceil(V/128)/SMs) * (R rounded up to 16) <= 512 (V = 151936 on 152 SMs: R <= 64): one persistent
 *     cooperative launch, one CTA per SM, each CTA's slice of the logits held in tensor memory (bound from a pool of
 *     every CTA's logits, filter and selection after grid barriers);
 *   - otherwise four launches: a GEMM pass over every CTA's first vocabulary tile (a sample) whose epilogue fills
 *     each row's pool; a bound per row from its pool; the full GEMM pass (blocks of 256 hidden rows, two TMEM
 *     accumulators) whose epilogue keeps the logits at or above their row's bound; a selection per row.
 * The workspace holds room for every logit of every row as a candidate (8 bytes each: R * V * 8 bytes and a little
 * more), so that the result is exact whatever the data; only the candidates actually kept are written.
 * Pointers must be 16-byte aligned device pointers; argument errors return DT_ERR_INVALID_ARG before any launch.
 * ------------------------------------------------------------------------------------------------------------- */
#define DT_LMHEAD_MAX_ROWS 8192
size_t dt_lmhead_workspace_bytes(int R, int D, int V, int M);
dt_status dt_lmhead_topm(int R, int D, int V, int M, const void* hidden, const void* w_head, dt_dtype dtype,
                         int32_t* out_ids, float* out_vals, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/* ---------------------------------------------------------------------------------------------------------------
 * dt_tree_attention — the verify pass's attention over the accepted prefix and the draft tree.
 * Source: blog.captcha.la, "Methodology — deep read" (the prefix-closed tree is verified in one target forward pass
 * with an unmodified ancestor-only causal mask, borrowed from DDTree/SpecInfer); gist.science, "Composants Clés —
 * Vérification" (standard tree attention, unchanged and lossless).
 *
 * Semantics: for request b, query head h and tree node i, the visible keys are the L prefix positions and the tree
 * positions L + t with mask[b][i][t] = 1 (as dt_build_trees emits it: the node's ancestors and itself); query head h
 * reads key/value head h / (Hq / Hkv);  out[b][i][h] = sum_j softmax_j(scale * q[b][i][h] . k_j) v_j  over them.
 * Arithmetic: bf16 products on the tensor cores, fp32 accumulation; the softmax weights are rounded to bf16 before
 * they multiply the value rows.
 *   q          [B,n,Hq,d] bf16;  k, v [B,Hkv,L+n,d] bf16 (the prefix's cache rows, then the tree's);
 *   mask       [B,n,n] uint8 (device);  out [B,n,Hq,d] fp32;
 *   workspace  dt_tree_attention_workspace_bytes(B,n,L,Hq,Hkv,d) bytes: a 256-byte header whose status word reports
 *              DT_ERR_TIMEOUT if a copy or MMA wait ran out (dt_get_error; initialise it with dt_workspace_init),
 *              then the partials of the key blocks.
 * Two launches: the partials on the tensor cores (tcgen05: S = Q K^T and O += P V accumulated in tensor memory, one
 * CTA per SM over an even share of the (request, key/value head, 64-key block) space; a (request, key/value head)
 * inside one CTA's share is written out directly), then the combination of the pairs split over several CTAs, a
 * programmatic dependent of the first launch (left out when no pair is split).
 * Supported: dtype DT_BF16, d = 128, (Hq / Hkv) * n <= 64. Outside it DT_ERR_UNSUPPORTED; argument errors (Hq not a
 * multiple of Hkv, scale not finite and positive, null or misaligned pointers) DT_ERR_INVALID_ARG; both before any
 * launch. Pointers are 16-byte aligned device pointers (mask: any alignment).
 * ------------------------------------------------------------------------------------------------------------- */
size_t dt_tree_attention_workspace_bytes(int B, int n, int L, int Hq, int Hkv, int d);
dt_status dt_tree_attention(int B, int n, int L, int Hq, int Hkv, int d, const void* q, const void* k, const void* v,
                            dt_dtype dtype, const uint8_t* mask, float scale, float* out, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------------------------------
 * dt_topm_static — dt_topm for callers that cannot allocate device memory.
 * No counterpart in the paper: this is a deployment variant of dt_topm, with the same arguments minus the
 * workspace and bit-identical results.
 *
 * Some callers cannot call cudaMalloc or receive a scratch buffer: a backend or plugin whose host framework owns all
 * device memory and hands it only inputs and outputs, or a latency-critical path that cannot afford the implicit
 * device synchronisation of an allocation. This entry point allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library call): its scratch is one library-wide device array of DT_TOPM_STATIC_SCRATCH_BYTES bytes,
 * which every GPU that loads the library holds until the process exits. The caller still passes the logits and the
 * output arrays.
 *   - Sizes whose scratch exceeds the array return DT_ERR_UNSUPPORTED before any launch. For V = 151936 the array
 *     holds up to 3246 rows (B·K) of bf16 logits at M = 64 and 1630 at M = 128; fp32 logits need about four times
 *     as much per row (817 rows at M = 64, 409 at M = 128). One request of 16 positions at M = 64 (bf16) uses 82 KB.
 *   - The first call on a device (more precisely, in a device context) looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it with the context's unique id. That lookup
 *     makes the device's primary context current if none is, and, under CUDA's lazy module loading, loads the
 *     library's device code on that device, which is when the driver allocates the array and may synchronise the
 *     device: make that first call during set-up, before any stream capture. A context created anew (for example
 *     after cudaDeviceReset) gets a new id, so the next call looks the address up again.
 *   - Every call shares the array and it keeps the previous call's contents; each call first clears the part that
 *     must start at zero (a cudaMemsetAsync on `stream` of the 256-byte header and the per-row bounds and tickets,
 *     4 + 4 bytes per row, each part rounded up to 256 bytes). Calls that may overlap on the GPU (other streams,
 *     other host threads) race on the array and must be serialised by the caller.
 *   - A NaN among the logits is not reported (there is no caller-visible status word); use dt_topm to detect it.
 * ------------------------------------------------------------------------------------------------------------- */
#define DT_TOPM_STATIC_SCRATCH_BYTES (16u << 20)
dt_status dt_topm_static(const void* logits, dt_dtype dtype, int B, int K, int V, int M, int32_t* out_ids,
                         float* out_vals, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------------------------------
 * dt_build_stats_read — what the last dt_build_trees (or dt_round) launch on `workspace` did, for measurement.
 * No counterpart in the paper (an observability hook). Synchronises `stream`, then reads the statistics the kernel
 * recorded in the workspace's header (a few words, written on every launch at negligible cost):
 *   launch_ns      time from CTA 0's start to its end (globaltimer), about the kernel's duration;
 *   gather_ns      the longest time any one CTA spent gathering correction rows W_c[ids]: in the large-batch
 *                  builder (B > 8) the children phases, where each group of expansions gathers its position's M rows
 *                  and forms their corrections; in the small-batch builder the W_c column gathers;
 *   gather_bytes   the correction rows those gathers read, counted once per gathered row (rows x H x element size);
 *   waves          waves the launch ran; expansions: GRU steps and roots expanded.
 * gather_bytes / gather_ns is the gather stage's achieved bandwidth. Argument errors: DT_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------------------------------------------- */
typedef struct {
  uint64_t launch_ns;
  uint64_t gather_ns;
  uint64_t gather_bytes;
  int32_t waves;
  int32_t expansions;
} dt_build_stats;
dt_status dt_build_stats_read(void* workspace, dt_build_stats* out, cudaStream_t stream);

/* Synchronises `stream`, then reads and clears the status word the device wrote into `workspace`. Returns DT_OK
 * when no device-side problem was recorded. After DT_ERR_TIMEOUT the workspace must be re-initialised. */
dt_status dt_get_error(void* workspace, cudaStream_t stream);

/* Time budget of every grid-barrier wait inside dt_build_trees, in nanoseconds (default 2 s). A test hook: with a
 * budget of 0 the first wait gives up at once, the kernel records DT_ERR_TIMEOUT and returns. Process-wide. */
void dt_set_barrier_timeout_ns(uint64_t ns);

/* Lookahead width of dt_build_trees: how many nodes of one request may be expanded together in one wave (their GRU
 * steps and children's scores computed at once), process-wide. 0 (the default) lets the library choose; k >= 1 caps
 * it (the small-batch builder also caps B·k at its wave size). The pops stay strictly best-first: a node joins the
 * frontier only when its parent is popped, so every width gives bit-identical outputs and only the time changes.
 * Returns DT_ERR_INVALID_ARG for k < 0 or k > DT_MAX_LOOKAHEAD. A tuning and test hook; no counterpart in the paper,
 * whose builder expands one popped node at a time (blog.captcha.la, "Methodology — deep read"). */
#define DT_MAX_LOOKAHEAD 8
dt_status dt_set_lookahead(int k);

/* Which kernel dt_topm (and dt_topm_static, dt_round) runs for small grids, process-wide. With 1 (the default), when
 * every row is a whole number of 16-byte groups, M <= 256, and the rows fit one wave of clusters of up to 8 CTAs on
 * the device (a few rows: one request's block positions), each row is one thread-block cluster that bounds, filters
 * and ranks its candidates in distributed shared memory; with 0, every launch takes the per-chunk candidate lists and
 * the row selection. Both give bit-identical results; only the time changes. Returns DT_ERR_INVALID_ARG unless
 * enable is 0 or 1. A tuning and test hook with no counterpart in the paper. */
dt_status dt_set_topm_cluster(int enable);

const char* dt_status_string(dt_status s);
int dt_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DOMINOTREE_H */
