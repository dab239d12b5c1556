// KV commit of one sequence by one CTA (vLLM issue 1171, void-main: "update
// block tables when you accept one candidate and release other blocks";
// mlc-llm issue 2319: the KV cache update part).  Used by the commit kernel
// and by the fused accept-and-commit kernel.
//
// With len = seq_lens[b] and the accepted path p[0..L] (strictly increasing):
// every KV head's K and V row at logical slot len + p[d] moves to slot len + d,
// seq_lens[b] becomes len + L + 1, and the blocks that hold tree scratch and
// start at or past the new length are released.
//
// Ordering: a destination len + d is never the source of a later entry d' > d
// (its source len + p[d'] has p[d'] >= d' > d), so the rows can move in passes
// of increasing d: each pass copies its source rows into a shared-memory stage
// (cp.async, all copies in flight together), the block synchronises, and the
// pass writes the stage out.  A destination that is a source of an earlier
// entry of the same pass (p = [0, 2, 3]: slot len + 2) is therefore read
// before it is written, and no pass overwrites a row a later pass reads (the
// one overlap, p[d] = d, is a row left in place and not copied).
#pragma once

#include "kernels.cuh"

namespace mt {

struct CommitSmem {
  int bt[kMaxTree + 2];                      // block-table window over slots [len, len + T)
  long long src[kMaxTree], dst[kMaxTree];    // byte offset of each path entry's source and
                                             // destination row of KV head 0
};

__device__ __forceinline__ bool commit_len_ok(const CommitParams& c, int len) {
  return len >= 0 && (long long)len + c.T <= (long long)c.max_blocks * c.P;
}

// Threads of the CTA load the block-table window of sequence b into sm.bt
// (nothing when len is invalid).  The caller synchronises before use.
__device__ __forceinline__ void commit_load_window(const CommitParams& c, int b, int len, CommitSmem& sm) {
  if (!commit_len_ok(c, len)) return;
  const int bt0 = len / c.P, nbw = (len + c.T - 1) / c.P - bt0 + 1;
  const int* btrow = c.block_tables + (size_t)b * c.max_blocks + bt0;
  for (int j = threadIdx.x; j < nbw; j += blockDim.x) sm.bt[j] = btrow[j];
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// All threads of the CTA call this with the same b, len (seq_lens[b] as read
// before the call), L and path (shared memory), after commit_load_window and a
// block synchronisation.  stage: stage_vecs 16-byte entries of shared memory.
// Any inconsistency (L out of range, a path that is not strictly increasing
// within the tree, a slot past the table or on a page outside the pool) records
// kStPages and leaves the sequence untouched.
__device__ inline void commit_sequence(const CommitParams& c, int b, int len, int L, const int* path, CommitSmem& sm,
                                       uint4* stage, int stage_vecs) {
  const int tid = threadIdx.x, nth = blockDim.x;
  const int n = L + 1;
  if (!(L >= 0 && L <= c.max_depth && L < c.T && commit_len_ok(c, len))) {  // uniform over the CTA
    if (tid == 0) set_status(c.status, kStPages);
    return;
  }
  const int bt0 = len / c.P;
  const size_t row_bytes = (size_t)c.D * c.elem_bytes;
  const size_t head_stride = (size_t)c.P * row_bytes;
  const size_t page_stride = (size_t)c.Hkv * head_stride;
  bool ok = true;
  if (tid < n) {
    const int d = tid, node = path[d];
    ok = node >= 0 && node < c.T && (d == 0 || node > path[d - 1]);
    if (ok) {
      const int ss = len + node, ds = len + d;
      const int sp = sm.bt[ss / c.P - bt0], dp = sm.bt[ds / c.P - bt0];
      ok = sp >= 0 && sp < c.num_pages && dp >= 0 && dp < c.num_pages;
      sm.src[d] = (long long)(sp * page_stride + (size_t)(ss % c.P) * row_bytes);
      sm.dst[d] = (long long)(dp * page_stride + (size_t)(ds % c.P) * row_bytes);
    }
  }
  if (!__syncthreads_and(ok)) {
    if (tid == 0) set_status(c.status, kStPages);
    return;
  }
  // the rows of entry d as 16-byte vectors f = (kvh * 2 + kv) * rv + v (rv a
  // power of two: shifts only); entries in place (p[d] = d) are skipped
  const int rv = (int)(row_bytes / 16), lrv = __ffs(rv) - 1;
  const int per_d = c.Hkv * 2 * rv;
  const int total = n * per_d;
  char* kc = static_cast<char*>(c.k_cache);
  char* vc = static_cast<char*>(c.v_cache);
  auto vec = [&](long long base, int f) -> char* {
    const int v = f & (rv - 1), kv = (f >> lrv) & 1, kvh = f >> (lrv + 1);
    return (kv ? vc : kc) + base + (size_t)kvh * head_stride + (size_t)v * 16;
  };
  for (int e0 = 0; e0 < total; e0 += stage_vecs) {
    const int e1 = min(total, e0 + stage_vecs);
    for (int d = e0 / per_d; d * per_d < e1; ++d) {  // uniform over the CTA
      if (sm.src[d] == sm.dst[d]) continue;
      const int f0 = max(e0 - d * per_d, 0), f1 = min(e1 - d * per_d, per_d);
      uint4* st = stage + (d * per_d - e0);
      for (int f = f0 + tid; f < f1; f += nth) cp_async16(st + f, vec(sm.src[d], f));
    }
    cp_async_wait_all();
    __syncthreads();  // every source row of the pass is read before any is written
    for (int d = e0 / per_d; d * per_d < e1; ++d) {
      if (sm.src[d] == sm.dst[d]) continue;
      const int f0 = max(e0 - d * per_d, 0), f1 = min(e1 - d * per_d, per_d);
      const uint4* st = stage + (d * per_d - e0);
      for (int f = f0 + tid; f < f1; f += nth) *reinterpret_cast<uint4*>(vec(sm.dst[d], f)) = st[f];
    }
    __syncthreads();  // the stage is refilled by the next pass
  }
  // lengths and released blocks (ascending, padded with -1)
  const int new_len = len + n;
  if (tid == 0) c.seq_lens[b] = new_len;
  const int first = (new_len + c.P - 1) / c.P;  // first block starting at or past new_len
  const int last = (len + c.T - 1) / c.P;       // last block holding tree scratch
  int* rel = c.released + (size_t)b * c.rel_width;
  int* btw = c.block_tables + (size_t)b * c.max_blocks;
  const int span = max(c.rel_width, last - first + 1);
  for (int j = tid; j < span; j += nth) {
    const int p = first + j;
    if (p <= last) {
      if (j < c.rel_width) rel[j] = sm.bt[p - bt0];
      btw[p] = -1;
    } else if (j < c.rel_width) {
      rel[j] = -1;
    }
  }
}

// Shared-memory stage of the commit: the rows of every path entry of every
// head, up to cap_bytes (more moves in several passes).
inline int commit_stage_vecs(const CommitParams& c, int cap_bytes) {
  const int n_max = c.max_depth + 1 < c.T ? c.max_depth + 1 : c.T;
  const long long need = (long long)n_max * c.Hkv * 2 * (c.D * c.elem_bytes / 16);
  const long long cap = cap_bytes / 16;
  return (int)(need < cap ? need : cap);
}

}  // namespace mt
