// Greedy acceptance (LM head at temperature 0; lmdeploy PR 1231 "[WIP] support
// Medusa" -- the `evaluate_posterior` step -- and vLLM issue 1171, "it uses
// the argmax result").
//
// One CTA per (sequence, node) streams the node's vocab row of target logits
// with 16-byte loads and reduces (value, index) pairs with warp shuffles:
// larger value wins, the lower index on equal values (+0 and -0 are equal).
// The last CTA of a sequence to finish (arrival counter in the workspace,
// reset to zero by that CTA) walks the tree:
//   acc[0] = 1, acc[i] = acc[parent[i]] && token[i] == argmax[parent[i]],
//   end = the deepest accepted node (lowest index among equals),
// and writes accept_len, the padded root-to-end path and next_token.
#include "kernels.cuh"

namespace mt {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) accept_kernel(AcceptParams a) {
  constexpr int EPV = 16 / sizeof(T);
  const int row = blockIdx.x;  // b * T + i
  const int b = row / a.T;
  const T* lg = static_cast<const T*>(a.logits) + (size_t)row * a.V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  float best = -INFINITY;
  int bidx = 0x7fffffff;
  const bool vec_ok = ((a.V * (int)sizeof(T)) % 16 == 0) &&
                      ((reinterpret_cast<uintptr_t>(lg) & 15) == 0);
  if (vec_ok) {
    const int nvec = a.V / EPV;
    const uint4* src = reinterpret_cast<const uint4*>(lg);
    int v = tid;
    // four independent 16-byte loads in flight per thread
    for (; v + 3 * kThreads < nvec; v += 4 * kThreads) {
      uint4 raw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) raw[u] = __ldcs(src + v + u * kThreads);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        T tmp[EPV];
        memcpy(tmp, &raw[u], 16);
        const int base = (v + u * kThreads) * EPV;
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const float x = Act<T>::to_f(tmp[e]);
          if (better(x, base + e, best, bidx)) { best = x; bidx = base + e; }
        }
      }
    }
    for (; v < nvec; v += kThreads) {
      uint4 raw = __ldcs(src + v);
      T tmp[EPV];
      memcpy(tmp, &raw, 16);
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float x = Act<T>::to_f(tmp[e]);
        if (better(x, v * EPV + e, best, bidx)) { best = x; bidx = v * EPV + e; }
      }
    }
  } else {
    for (int v = tid; v < a.V; v += kThreads) {
      const float x = Act<T>::to_f(lg[v]);
      if (better(x, v, best, bidx)) { best = x; bidx = v; }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, off);
    const int oi = __shfl_xor_sync(0xffffffffu, bidx, off);
    if (better(ov, oi, best, bidx)) { best = ov; bidx = oi; }
  }
  __shared__ float s_v[kThreads / 32];
  __shared__ int s_i[kThreads / 32];
  __shared__ bool s_last;
  if (lane == 0) { s_v[warp] = best; s_i[warp] = bidx; }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < kThreads / 32; ++w)
      if (better(s_v[w], s_i[w], best, bidx)) { best = s_v[w]; bidx = s_i[w]; }
    a.argmax_out[row] = bidx;
    __threadfence();
    const unsigned prev = atomicAdd(&a.counters[b], 1u);
    s_last = prev == (unsigned)(a.T - 1);
  }
  __syncthreads();
  if (!s_last || tid != 0) return;

  // last arrival for sequence b: path selection
  __threadfence();
  a.counters[b] = 0u;
  const int* par = a.parents + (size_t)b * a.T;
  const int* tok = a.tokens + (size_t)b * a.T;
  const volatile int* am = a.argmax_out + (size_t)b * a.T;
  int* path = a.accept_path + (size_t)b * (a.max_depth + 1);
  unsigned long long acc = 1ull;  // bit i: node i accepted
  int depth[kMaxTree];
  depth[0] = 0;
  int end = 0;
  bool ok = par[0] == -1;
  for (int i = 1; i < a.T && ok; ++i) {
    const int p = par[i];
    if (p < 0 || p >= i) { ok = false; break; }
    depth[i] = depth[p] + 1;
    if (depth[i] > a.max_depth) { ok = false; break; }
    if (((acc >> p) & 1ull) && tok[i] == am[p]) {
      acc |= 1ull << i;
      if (depth[i] > depth[end]) end = i;
    }
  }
  for (int d = 0; d <= a.max_depth; ++d) path[d] = -1;
  if (!ok) {
    set_status(a.status, kStTree);
    a.accept_len[b] = 0;
    path[0] = 0;
    a.next_token[b] = am[0];
    return;
  }
  a.accept_len[b] = depth[end];
  for (int n = end; n >= 0; n = par[n]) path[depth[n]] = n;
  a.next_token[b] = am[end];
}

}  // namespace

cudaError_t launch_accept(const AcceptParams& a, int dtype, cudaStream_t stream) {
  dim3 grid((unsigned)(a.B * a.T));
  switch (dtype) {
    case 0: accept_kernel<float><<<grid, kThreads, 0, stream>>>(a); break;
    case 1: accept_kernel<__half><<<grid, kThreads, 0, stream>>>(a); break;
    default: accept_kernel<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace mt
