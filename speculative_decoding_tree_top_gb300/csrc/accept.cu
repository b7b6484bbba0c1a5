// dt_accept_paths — the accepted root-to-node path of each draft tree after the target model's verify pass.
//
// Method: blog.captcha.la, "Methodology — deep read" (a single target-model forward pass verifies the tree and the
// longest accepted root-to-leaf path is kept) and "Threat model" (lossless up to floating-point tie-breaking);
// gist.science, "Composants Clés — Vérification" and "Résultats Expérimentaux" (lossless: the output matches serial
// greedy decoding).
//
// Greedy verification: the verify pass gives, for the root (the last accepted token) and for every tree node, the
// target's next token. Starting at the root, the walk steps into the child whose token is the target's next token at
// the current node, as long as one exists; the target's next token at the last node reached is the bonus token.
// Under greedy decoding that path is the only one the target accepts, hence the longest. One warp per request: each
// step is one ballot over the nodes (children follow their parent in pop order); at most max depth steps.
#include <cuda_runtime.h>

#include "dt_internal.cuh"

namespace dt {
namespace {

constexpr int kWarpsPerCta = 8;

__global__ void __launch_bounds__(32 * kWarpsPerCta) accept_kernel(int B, int n, const int32_t* __restrict__ tokens,
                                                                    const int32_t* __restrict__ parents,
                                                                    const int32_t* __restrict__ target_next,
                                                                    int32_t* __restrict__ accept_len,
                                                                    int32_t* __restrict__ path,
                                                                    int32_t* __restrict__ bonus) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (b >= B) return;  // whole warps only
  const int32_t* tk = tokens + static_cast<size_t>(b) * n;
  const int32_t* pa = parents + static_cast<size_t>(b) * n;
  const int32_t* tn = target_next + static_cast<size_t>(b) * (n + 1);
  int32_t* out = path + static_cast<size_t>(b) * n;
  int cur = -1, len = 0;
  int want = __ldg(tn);  // the target's token after the accepted prefix
  for (int step = 0; step < n; ++step) {
    int hit = 0x7FFFFFFF;  // lowest node index that is a child of `cur` with token `want`
    for (int i = cur + 1 + lane; i < n; i += 32)
      if (__ldg(pa + i) == cur && __ldg(tk + i) == want) {
        hit = i;
        break;
      }
    hit = static_cast<int>(__reduce_min_sync(0xFFFFFFFFu, static_cast<unsigned>(hit)));
    if (hit == 0x7FFFFFFF) break;
    if (lane == 0) out[len] = hit;
    ++len;
    cur = hit;
    want = __ldg(tn + 1 + hit);
  }
  for (int i = len + lane; i < n; i += 32) out[i] = -1;
  if (lane == 0) {
    accept_len[b] = len;
    bonus[b] = want;
  }
}

}  // namespace
}  // namespace dt

extern "C" dt_status dt_accept_paths(int B, int n, const int32_t* tokens, const int32_t* parents,
                                     const int32_t* target_next, int32_t* out_accept_len, int32_t* out_path,
                                     int32_t* out_bonus, cudaStream_t stream) {
  using namespace dt;
  if (B < 0 || n < 1) return DT_ERR_INVALID_ARG;
  if (n > DT_MAX_N) return DT_ERR_UNSUPPORTED;
  if (B == 0) return DT_OK;
  const void* ptrs[] = {tokens, parents, target_next, out_accept_len, out_path, out_bonus};
  for (const void* q : ptrs)
    if (!q || (reinterpret_cast<uintptr_t>(q) & 3u)) return DT_ERR_INVALID_ARG;
  const unsigned grid = static_cast<unsigned>((B + kWarpsPerCta - 1) / kWarpsPerCta);
  accept_kernel<<<grid, 32 * kWarpsPerCta, 0, stream>>>(B, n, tokens, parents, target_next, out_accept_len, out_path,
                                                        out_bonus);
  return cuda_status(cudaGetLastError());
}
