// Candidate trees: the tree attention mask of a parent map, and the walk of
// the greedy tree verify.
//
// A tree of N candidate nodes is given by parent[i] < i (-1: hung on the
// committed prefix).  "SpecOPD: Branch-Parallel On-Policy Distillation for
// Speculative Decoding", section "树注意力(Tree Attention)": node u sees node v
// iff v is u or one of u's ancestors, so one batched target pass scores every
// node without leaking sibling branches.  "Speculative Decoding 与 MTP",
// sections 4 and 11: at T = 0 a candidate is kept when it equals the target
// argmax, the first mismatch emits the target's token, and a tree commits a
// single path.
#pragma once

#include <cstdint>

namespace ssv {

constexpr uint32_t kBadTree = 32u;  // a parent outside [-1, i): shares the ragged-offsets status bit

// mask[b][u][v] = 1 iff v is u or an ancestor of u; depth[b][u] = number of
// strict ancestors.  One thread per (row, node).
__global__ void tree_mask_kernel(const int32_t* parent, int B, int N, uint8_t* mask, int32_t* depth,
                                 uint32_t* status) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (long long)B * N) return;
  const int b = (int)(t / N), u = (int)(t - (long long)b * N);
  const int32_t* par = parent + (long long)b * N;
  uint8_t* row = mask + ((long long)b * N + u) * N;
  for (int v = 0; v < N; ++v) row[v] = 0;
  int v = u, d = -1;
  bool ok = true;
  while (v >= 0 && d < N) {  // at most N steps: parents strictly decrease
    row[v] = 1;
    ++d;
    const int p = par[v];
    if (p >= v || p < -1) {
      ok = false;
      break;
    }
    v = p;
  }
  if (depth) depth[(long long)b * N + u] = d;
  if (!ok && status) atomicOr(status, kBadTree);
}

// One thread per row: from the prefix, move to the first child (node order)
// whose token is the current slot's target argmax; emit the argmax where no
// child matches.  am[b][0] is the prefix slot, am[b][i + 1] node i's.
__global__ void tree_walk_kernel(const int32_t* am, const int32_t* parent, const int32_t* tokens, int B, int N,
                                 int32_t* path, int32_t* out_tokens, int32_t* n_accepted, uint32_t* status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int32_t* a = am + (long long)b * (N + 1);
  const int32_t* par = parent + (long long)b * N;
  const int32_t* tok = tokens + (long long)b * N;
  int32_t* pth = path + (long long)b * N;
  int32_t* out = out_tokens + (long long)b * (N + 1);
  bool ok = true;
  for (int i = 0; i < N; ++i)
    if (par[i] >= i || par[i] < -1) ok = false;
  int cur = -1, n = 0;
  if (ok) {
    while (true) {
      const int want = a[cur + 1];
      int nxt = -1;
      if (want >= 0)
        for (int c = cur + 1; c < N; ++c)
          if (par[c] == cur && tok[c] == want) {
            nxt = c;
            break;
          }
      out[n] = want;
      if (nxt < 0) break;
      pth[n] = nxt;
      ++n;
      cur = nxt;
    }
  } else if (status) {
    atomicOr(status, kBadTree);
  }
  for (int i = ok ? n + 1 : 0; i <= N; ++i) out[i] = -1;
  for (int i = ok ? n : 0; i < N; ++i) pth[i] = -1;
  n_accepted[b] = ok ? n : -1;
}

}  // namespace ssv
