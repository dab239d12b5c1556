// Greedy acceptance (LM head at temperature 0; lmdeploy PR 1231 "[WIP] support
// Medusa" -- the `evaluate_posterior` step -- and vLLM issue 1171, "it uses
// the argmax result").
//
// Two kernels: the per-node argmax over the vocab (values compared exactly;
// +0 and -0 are equal; a larger value wins, the lower index among equal
// values), streamed through shared memory by persistent CTAs; then one warp
// per sequence selects the path:
//   acc[0] = 1, acc[i] = acc[parent[i]] && token[i] == argmax[parent[i]],
//   end = the deepest accepted node (lowest index among equals),
// and writes accept_len, the padded root-to-end path and next_token.
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace mt {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Max of the 8 values of a 16-byte vector, as float.
template <typename T> struct Max8;
template <> struct Max8<__nv_bfloat16> {
  static __device__ __forceinline__ float of(const uint4& v) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
    const __nv_bfloat162 m = __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
    return fmaxf(__low2float(m), __high2float(m));
  }
};
template <> struct Max8<__half> {
  static __device__ __forceinline__ float of(const uint4& v) {
    const __half2* h = reinterpret_cast<const __half2*>(&v);
    const __half2 m = __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
    return fmaxf(__low2float(m), __high2float(m));
  }
};
template <> struct Max8<float> {  // 4 values per vector for fp32
  static __device__ __forceinline__ float of(const uint4& v) {
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
};

constexpr int kChunkBytes = 32 * 1024;
constexpr int kStages = 6;
constexpr int kVecsPerChunk = kChunkBytes / 16;
constexpr int kStreamThreads = 512;
constexpr int kStreamWarps = kStreamThreads / 32;

__device__ __forceinline__ void warp_best(float& best, int& bidx) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, off);
    const int oi = __shfl_xor_sync(0xffffffffu, bidx, off);
    if (better(ov, oi, best, bidx)) { best = ov; bidx = oi; }
  }
}

// Per-node argmax.  Persistent CTAs take rows r = blockIdx.x, + gridDim.x, ...
// and stream them in 32 KB chunks through a 6-stage shared-memory ring filled
// by 1-D bulk copies (thread 0 issues; an mbarrier per stage counts bytes).
// Each thread scans its 16-byte vectors in increasing index order keeping
// (max, first index): a vector's packed maximum is compared first and the
// vector is searched only when it beats the running maximum.  At the end of a
// row each warp leaves its (max, index) in shared memory and warp 0 merges
// them after the chunk barrier, so rows cost no extra block synchronisation.
template <typename T>
__global__ void __launch_bounds__(kStreamThreads) argmax_stream_kernel(AcceptParams a) {
  constexpr int EPV = 16 / sizeof(T);
  extern __shared__ __align__(128) uint8_t smem[];
  uint4* ring = reinterpret_cast<uint4*>(smem);  // [kStages][kVecsPerChunk]
  __shared__ uint64_t full[kStages];
  __shared__ float s_pv[2][kStreamWarps];
  __shared__ int s_pi[2][kStreamWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long row_bytes = (long long)a.V * sizeof(T);
  const int chunks_per_row = (int)((row_bytes + kChunkBytes - 1) / kChunkBytes);
  const int nrows = a.B * a.T;
  const int my_rows = blockIdx.x < nrows ? (nrows - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const long long total = (long long)my_rows * chunks_per_row;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) tc::mbar_init(&full[s], 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  const uint64_t policy = tc::policy_evict_first();
  auto issue = [&](long long k) {  // chunk k of this CTA into stage k % kStages
    const int row = blockIdx.x + (int)(k / chunks_per_row) * gridDim.x;
    const long long off = (k % chunks_per_row) * (long long)kChunkBytes;
    const uint32_t bytes = (uint32_t)min((long long)kChunkBytes, row_bytes - off);
    uint64_t* bar = &full[k % kStages];
    tc::mbar_arrive_expect_tx(bar, bytes);
    tc::bulk_load(ring + (k % kStages) * kVecsPerChunk,
                  static_cast<const uint8_t*>(a.logits) + (size_t)row * row_bytes + off, bytes, bar, policy);
  };
  long long issued = 0;  // chunks handed to the copy engine (thread 0)
  if (tid == 0) {
    for (long long k = 0; k < total && k < kStages; ++k) issue(k);
    issued = total < kStages ? total : kStages;
  }
  volatile int no_abort = 0;
  float best = -INFINITY;
  int bidx = 0x7fffffff;
  bool ok = true;
  for (long long k = 0; k < total; ++k) {
    const int stage = (int)(k % kStages);
    if (ok) ok = tc::mbar_wait(&full[stage], (uint32_t)((k / kStages) & 1), &no_abort, a.status);
    const int c = (int)(k % chunks_per_row);
    const int rowi = (int)(k / chunks_per_row);
    const long long off = (long long)c * kChunkBytes;
    const int nvec = (int)(min((long long)kChunkBytes, row_bytes - off) / 16);
    const uint4* chunk = ring + stage * kVecsPerChunk;
    if (ok) {
      const int base = (int)(off / 16);
      for (int v = tid; v < nvec; v += kStreamThreads) {
        const uint4 raw = chunk[v];
        const float m = Max8<T>::of(raw);
        if (m > best || bidx == 0x7fffffff) {
          T tmp[EPV];
          memcpy(tmp, &raw, 16);
#pragma unroll
          for (int e = EPV - 1; e >= 0; --e)
            if (Act<T>::to_f(tmp[e]) == m) bidx = (base + v) * EPV + e;
          best = m;
        }
      }
    }
    const bool row_end = c == chunks_per_row - 1;
    if (row_end) {
      warp_best(best, bidx);
      if (lane == 0) {
        s_pv[rowi & 1][warp] = best;
        s_pi[rowi & 1][warp] = bidx;
      }
      best = -INFINITY;
      bidx = 0x7fffffff;
    }
    __syncthreads();  // stage consumed; row results (if any) published
    if (tid == 0 && ok && k + kStages < total) {
      issue(k + kStages);
      issued = k + kStages + 1;
    }
    if (row_end && warp == 0) {
      // merge the row's warp results; their slots are rewritten two rows
      // later, after further chunk barriers that warp 0 must also reach
      float v = lane < kStreamWarps ? s_pv[rowi & 1][lane] : -INFINITY;
      int ix = lane < kStreamWarps ? s_pi[rowi & 1][lane] : 0x7fffffff;
      warp_best(v, ix);
      if (lane == 0) a.argmax_out[blockIdx.x + rowi * gridDim.x] = ix;
    }
  }
  // after a timed-out wait: no bulk copy may still target shared memory at exit
  if (tid == 0)
    for (long long k = issued > kStages ? issued - kStages : 0; k < issued; ++k) {
      const uint64_t t0 = tc::global_timer_ns();
      while (!tc::mbar_try_wait(&full[k % kStages], (uint32_t)((k / kStages) & 1)) &&
             tc::global_timer_ns() - t0 < tc::kWaitLimitNs) {
      }
    }
}

// Fallback for rows that are not 16-byte aligned: one CTA per row, scalar loads.
template <typename T>
__global__ void __launch_bounds__(kThreads) argmax_scalar_kernel(AcceptParams a) {
  __shared__ float s_v[kThreads / 32];
  __shared__ int s_i[kThreads / 32];
  const int row = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T* lg = static_cast<const T*>(a.logits) + (size_t)row * a.V;
  float best = -INFINITY;
  int bidx = 0x7fffffff;
  for (int v = threadIdx.x; v < a.V; v += kThreads) {
    const float x = Act<T>::to_f(lg[v]);
    if (better(x, v, best, bidx)) { best = x; bidx = v; }
  }
  warp_best(best, bidx);
  if (lane == 0) { s_v[warp] = best; s_i[warp] = bidx; }
  __syncthreads();
  if (warp == 0) {
    float v = lane < kThreads / 32 ? s_v[lane] : -INFINITY;
    int ix = lane < kThreads / 32 ? s_i[lane] : 0x7fffffff;
    warp_best(v, ix);
    if (lane == 0) a.argmax_out[row] = ix;
  }
}

// Greedy path, one warp per sequence, every step in parallel over the nodes
// (lane l owns nodes l and l + 32):
//   ancestors and depths by pointer jumping (six rounds close any depth < 64);
//   node i matches when tokens[i] == argmax[parent[i]] (the root always);
//   node i is accepted when every node on its root path matches;
//   end = the accepted node of largest depth, the lowest index among equals.
constexpr int kPathWarps = 8;
__global__ void __launch_bounds__(kPathWarps * 32) accept_path_kernel(AcceptParams a) {
  __shared__ unsigned long long s_anc[kPathWarps][kMaxTree];
  __shared__ int s_up[kPathWarps][kMaxTree], s_dep[kPathWarps][kMaxTree], s_am[kPathWarps][kMaxTree];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kPathWarps + warp;
  if (b >= a.B) return;
  const int T = a.T;
  const int* par = a.parents + (size_t)b * T;
  const int* tok = a.tokens + (size_t)b * T;
  const int* am = a.argmax_out + (size_t)b * T;
  bool good = true;
  for (int i = lane; i < T; i += 32) {
    const int p = par[i];
    const bool ok_i = i == 0 ? p == -1 : (p >= 0 && p < i);
    good = good && ok_i;
    s_anc[warp][i] = 1ull << i;
    s_up[warp][i] = (i > 0 && ok_i) ? p : -1;
    s_dep[warp][i] = (i > 0 && ok_i) ? 1 : 0;
    s_am[warp][i] = am[i];
  }
  const bool ok = __all_sync(0xffffffffu, good);
  __syncwarp();
  for (int round = 0; round < 6; ++round) {
    unsigned long long na[2];
    int nu[2], nd[2];
    for (int k = 0; k < 2; ++k) {
      const int i = lane + 32 * k;
      if (i < T) {
        const int u = s_up[warp][i];
        na[k] = s_anc[warp][i] | (u >= 0 ? s_anc[warp][u] : 0ull);
        nd[k] = s_dep[warp][i] + (u >= 0 ? s_dep[warp][u] : 0);
        nu[k] = u >= 0 ? s_up[warp][u] : -1;
      }
    }
    __syncwarp();
    for (int k = 0; k < 2; ++k) {
      const int i = lane + 32 * k;
      if (i < T) {
        s_anc[warp][i] = na[k];
        s_dep[warp][i] = nd[k];
        s_up[warp][i] = nu[k];
      }
    }
    __syncwarp();
  }
  // mismatching nodes as a 64-bit mask
  bool mis0 = false, mis1 = false;
  {
    const int i0 = lane, i1 = lane + 32;
    if (i0 < T && i0 > 0) {
      const int p = par[i0];
      mis0 = !(p >= 0 && p < i0) || tok[i0] != s_am[warp][p];
    }
    if (i1 < T) {
      const int p = par[i1];
      mis1 = !(p >= 0 && p < i1) || tok[i1] != s_am[warp][p];
    }
  }
  const unsigned long long mis = (unsigned long long)__ballot_sync(0xffffffffu, mis0) |
                                 ((unsigned long long)__ballot_sync(0xffffffffu, mis1) << 32);
  bool deep_ok = true;
  int key = -1;  // (depth, -index) of the best accepted node owned by this lane
  for (int k = 0; k < 2; ++k) {
    const int i = lane + 32 * k;
    if (i < T) {
      const int d = s_dep[warp][i];
      deep_ok = deep_ok && d <= a.max_depth;
      if ((s_anc[warp][i] & mis) == 0ull) key = max(key, (d << 8) | (255 - i));
    }
  }
  const bool all_ok = ok && __all_sync(0xffffffffu, deep_ok);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, off));
  int* path = a.accept_path + (size_t)b * (a.max_depth + 1);
  if (!all_ok) {
    if (lane == 0) {
      set_status(a.status, kStTree);
      a.accept_len[b] = 0;
      a.next_token[b] = s_am[warp][0];
    }
    for (int d = lane; d <= a.max_depth; d += 32) path[d] = d == 0 ? 0 : -1;
    return;
  }
  const int end = 255 - (key & 255);
  const unsigned long long on_path = s_anc[warp][end];
  const int len = s_dep[warp][end];
  for (int d = lane; d <= a.max_depth; d += 32)
    if (d > len) path[d] = -1;
  for (int k = 0; k < 2; ++k) {
    const int i = lane + 32 * k;
    if (i < T && ((on_path >> i) & 1ull)) path[s_dep[warp][i]] = i;
  }
  if (lane == 0) {
    a.accept_len[b] = len;
    a.next_token[b] = s_am[warp][end];
  }
}

template <typename T>
cudaError_t launch_t(const AcceptParams& a, cudaStream_t stream) {
  const int nrows = a.B * a.T;
  if (((long long)a.V * sizeof(T)) % 16 != 0 || (reinterpret_cast<uintptr_t>(a.logits) & 15) != 0) {
    argmax_scalar_kernel<T><<<nrows, kThreads, 0, stream>>>(a);
  } else {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = nrows < sms ? nrows : sms;
    const size_t smem = (size_t)kStages * kChunkBytes;
    cudaError_t e = cudaFuncSetAttribute(argmax_stream_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    argmax_stream_kernel<T><<<grid, kStreamThreads, smem, stream>>>(a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  accept_path_kernel<<<(a.B + kPathWarps - 1) / kPathWarps, kPathWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_accept(const AcceptParams& a, int dtype, cudaStream_t stream) {
  switch (dtype) {
    case 0: return launch_t<float>(a, stream);
    case 1: return launch_t<__half>(a, stream);
    default: return launch_t<__nv_bfloat16>(a, stream);
  }
}

}  // namespace mt
