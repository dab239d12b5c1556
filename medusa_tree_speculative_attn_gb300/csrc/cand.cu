// Candidate tree tokens from the Medusa heads (lmdeploy PR 1231 "[WIP] support
// Medusa": porting `generate_candidates`; Medusa heads at top-k over a
// 64-choice tree, "medusa choices(64)").
//
// For sequence b, with the tree given by its parents (node 0 the root):
//   token[0] = argmax_v root_logits[b][v];
//   for a node i at depth d >= 1 that has r earlier siblings (children of the
//   same parent with a smaller index): token[i] = the entry of rank r of
//   head_logits[b][d - 1] in the order "larger value first, lower index first
//   among equal values".
// One CTA per (depth, sequence): CTA (0, b) takes the root's argmax, CTA (d, b)
// the top kMaxChoices of head d - 1, and each writes the tokens of its nodes.
// A row is read twice with 16-byte loads, eight in flight per thread (the
// second pass from L2): the first pass takes each thread's maximum, and tau =
// the largest over warps of each warp's k-th largest thread maximum bounds the
// k best entries from below (k thread maxima of that warp are >= tau);
// the second pass collects the entries >= tau in shared memory, and each
// candidate's rank among them (an O(n^2) count in the stated order) places the
// k best.  When ties put more than kCand entries at or above tau, the block
// falls back to per-thread sorted top-16 lists merged by warps.
#include "kernels.cuh"

namespace mt {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCand = 512;  // candidates collected above the threshold
constexpr int kBatch = 8;   // 16-byte loads in flight per thread

// (value, index) order: larger value first, lower index among equal values.
__device__ __forceinline__ bool before(float v, int i, float w, int j) {
  return v > w || (v == w && i < j);
}

// Insert (v, i) into the sorted list (lv, li) of K entries if it belongs there.
template <int K>
__device__ __forceinline__ void insert(float (&lv)[K], int (&li)[K], float v, int i) {
  if (!before(v, i, lv[K - 1], li[K - 1])) return;
  lv[K - 1] = v;
  li[K - 1] = i;
#pragma unroll
  for (int k = K - 1; k > 0; --k) {
    if (before(lv[k], li[k], lv[k - 1], li[k - 1])) {
      const float tv = lv[k];
      lv[k] = lv[k - 1];
      lv[k - 1] = tv;
      const int ti = li[k];
      li[k] = li[k - 1];
      li[k - 1] = ti;
    }
  }
}

template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ float at(const uint4& v, int e) {
    return __uint_as_float(e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w);
  }
};
template <> struct Vec<__half> {
  static constexpr int N = 8;
  static __device__ __forceinline__ float at(const uint4& v, int e) {
    return __half2float(reinterpret_cast<const __half*>(&v)[e]);
  }
};
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ float at(const uint4& v, int e) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(&v)[e]);
  }
};

template <typename T>
__global__ void __launch_bounds__(kThreads) cand_kernel(CandParams a) {
  constexpr int K = kMaxChoices;
  constexpr int EPV = Vec<T>::N;
  __shared__ int s_par0[kMaxTree], s_par[kMaxTree], s_dep[kMaxTree], s_rank[kMaxTree];
  __shared__ int s_bad, s_need;
  __shared__ float s_wv[kWarps][K];
  __shared__ int s_wi[kWarps][K];
  __shared__ int s_top[K];
  __shared__ float s_wt[kWarps];
  __shared__ float s_cv[kCand];
  __shared__ int s_ci[kCand];
  __shared__ int s_cnt;
  const int d = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nT = a.T;
  pdl_wait();

  // ---- the tree: validity, depths (pointer jumping), choice ranks ----
  if (tid == 0) {
    s_bad = 0;
    s_need = 0;
  }
  if (tid < K) s_top[tid] = -1;  // a rank past the vocab has no entry
  __syncthreads();
  int up = -1;
  if (tid < nT) {
    const int p = a.parents[(size_t)b * nT + tid];
    const bool ok = tid == 0 ? p == -1 : (p >= 0 && p < tid);
    s_par0[tid] = p;
    s_par[tid] = ok ? p : -1;
    s_dep[tid] = tid == 0 ? 0 : 1;
    up = ok ? p : -1;
    if (!ok) s_bad = 1;
  }
  __syncthreads();
  // depth = number of links to the root: add the depth of the node `up`
  // points to and jump (six rounds cover depths below 64)
  for (int round = 0; round < 6; ++round) {
    int nd = 0, nu = -1;
    if (tid < nT && up > 0) {
      nd = s_dep[up];
      nu = s_par[up];
    }
    __syncthreads();
    if (tid < nT && up > 0) {
      s_dep[tid] += nd;
      s_par[tid] = nu;  // s_par now holds the jump pointer of the node
      up = nu;
    }
    __syncthreads();
  }
  if (tid < nT) {
    // choice rank: earlier siblings
    const int p = s_par0[tid];
    int r = 0;
    for (int j = 1; j < tid; ++j) r += s_par0[j] == p;
    s_rank[tid] = tid == 0 ? 0 : r;
    if (s_dep[tid] > a.heads) s_bad = 1;
    if (tid > 0 && s_dep[tid] == d) atomicMax(&s_need, r + 1);
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0 && d == 0) set_status(a.status, kStTree);
    return;
  }
  if (d > 0 && s_need > K) {
    if (tid == 0) set_status(a.status, kStTree);
    return;
  }
  if (d > 0 && s_need == 0) return;  // no node at this depth

  // ---- top-K of the row (the root needs only the first entry) ----
  const T* row = static_cast<const T*>(d == 0 ? a.root_logits : a.head_logits) +
                 (d == 0 ? (size_t)b * a.V : ((size_t)b * a.heads + (d - 1)) * a.V);
  const int nvec = (reinterpret_cast<uintptr_t>(row) & 15) ? 0 : a.V / EPV;  // scalar if unaligned
  const int kneed = d == 0 ? 1 : s_need;  // entries this row must rank

  // ---- fast path: threshold, then the entries at or above it ----
  {
    float tm = -INFINITY;
    for (int v0 = tid; v0 < nvec; v0 += kThreads * kBatch) {
      uint4 raw[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (v0 + j * kThreads < nvec) raw[j] = reinterpret_cast<const uint4*>(row)[v0 + j * kThreads];
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (v0 + j * kThreads < nvec) {
#pragma unroll
          for (int e = 0; e < EPV; ++e) tm = fmaxf(tm, Vec<T>::at(raw[j], e));
        }
    }
    for (int i = nvec * EPV + tid; i < a.V; i += kThreads) tm = fmaxf(tm, Act<T>::to_f(row[i]));
    // tau: for each warp the kneed-th largest of its 32 thread maxima (rank by
    // value, ties by lane), then the largest of those over the warps: kneed
    // entries of one warp's slice are >= tau, and tau is at most the kneed-th
    // largest of all the maxima
    int rk = 0;
#pragma unroll
    for (int l = 0; l < 32; ++l) rk += before(__shfl_sync(0xffffffffu, tm, l), l, tm, lane);
    if (rk == kneed - 1) s_wt[warp] = tm;
    if (tid == 0) s_cnt = 0;
    __syncthreads();
    float tau = s_wt[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) tau = fmaxf(tau, s_wt[w]);
    for (int v0 = tid; v0 < nvec; v0 += kThreads * kBatch) {
      uint4 raw[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (v0 + j * kThreads < nvec) raw[j] = reinterpret_cast<const uint4*>(row)[v0 + j * kThreads];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int v = v0 + j * kThreads;
        if (v >= nvec) continue;
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const float x = Vec<T>::at(raw[j], e);
          if (x >= tau) {
            const int slot = atomicAdd(&s_cnt, 1);
            if (slot < kCand) {
              s_cv[slot] = x;
              s_ci[slot] = v * EPV + e;
            }
          }
        }
      }
    }
    for (int i = nvec * EPV + tid; i < a.V; i += kThreads) {
      const float x = Act<T>::to_f(row[i]);
      if (x >= tau) {
        const int slot = atomicAdd(&s_cnt, 1);
        if (slot < kCand) {
          s_cv[slot] = x;
          s_ci[slot] = i;
        }
      }
    }
    __syncthreads();
    const int n = s_cnt;
    if (n <= kCand) {
      for (int c = tid; c < n; c += kThreads) {
        const float x = s_cv[c];
        const int xi = s_ci[c];
        int r = 0;
        for (int u = 0; u < n; ++u) r += before(s_cv[u], s_ci[u], x, xi);
        if (r < K) s_top[r] = xi;
      }
      __syncthreads();
      if (tid < nT && s_dep[tid] == d) a.tokens[(size_t)b * nT + tid] = s_top[s_rank[tid]];
      return;
    }
  }

  // ---- fallback (heavy ties): per-thread sorted lists, merged ----
  float lv[K];
  int li[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    lv[k] = -INFINITY;
    li[k] = 0x7fffffff;
  }
  for (int v = tid; v < nvec; v += kThreads) {
    const uint4 raw = reinterpret_cast<const uint4*>(row)[v];
#pragma unroll
    for (int e = 0; e < EPV; ++e) insert<K>(lv, li, Vec<T>::at(raw, e), v * EPV + e);
  }
  for (int i = nvec * EPV + tid; i < a.V; i += kThreads)  // tail past the last full vector
    insert<K>(lv, li, Act<T>::to_f(row[i]), i);

  // warp merge: K rounds, each taking the best head among the lanes' lists
  int pos = 0;  // this lane's next unconsumed entry
  for (int k = 0; k < K; ++k) {
    float hv = pos < K ? lv[0] : -INFINITY;
    int hi = pos < K ? li[0] : 0x7fffffff;
    float bv = hv;
    int bi = hi;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (before(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      s_wv[warp][k] = bv;
      s_wi[warp][k] = bi;
    }
    if (hi == bi && pos < K) {  // this lane's head was taken (indices are unique)
#pragma unroll
      for (int m = 0; m < K - 1; ++m) {
        lv[m] = lv[m + 1];
        li[m] = li[m + 1];
      }
      lv[K - 1] = -INFINITY;
      li[K - 1] = 0x7fffffff;
      ++pos;
    }
  }
  __syncthreads();
  // block merge by warp 0: lane w < kWarps walks warp w's list
  if (warp == 0) {
    int wp = 0;
    for (int k = 0; k < K; ++k) {
      float hv = -INFINITY;
      int hi = 0x7fffffff;
      if (lane < kWarps && wp < K) {
        hv = s_wv[lane][wp];
        hi = s_wi[lane][wp];
      }
      float bv = hv;
      int bi = hi;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (before(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (lane < kWarps && wp < K && hi == bi) ++wp;
      if (lane == 0) s_top[k] = bi == 0x7fffffff ? -1 : bi;
    }
  }
  __syncthreads();

  // ---- tokens of this depth's nodes ----
  if (tid < nT && s_dep[tid] == d) a.tokens[(size_t)b * nT + tid] = s_top[s_rank[tid]];
}

}  // namespace

cudaError_t launch_cand(const CandParams& a, int dtype, cudaStream_t stream) {
  dim3 grid(a.heads + 1, a.B);
  switch (dtype) {
    case 0: return launch_pdl(cand_kernel<float>, grid, dim3(kThreads), 0, stream, a);
    case 1: return launch_pdl(cand_kernel<__half>, grid, dim3(kThreads), 0, stream, a);
    default: return launch_pdl(cand_kernel<__nv_bfloat16>, grid, dim3(kThreads), 0, stream, a);
  }
}

}  // namespace mt
