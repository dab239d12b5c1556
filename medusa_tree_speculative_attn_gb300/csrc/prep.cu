// Tree preparation: validates every sequence's tree, builds the per-node
// ancestor bitmasks and the tile schedule, and writes the tree tokens' rotated
// keys and raw values into their scratch slots of the paged cache.
//
// The tree mask (vLLM issue 1171, void-main: the Medusa tree mask inside the
// cached-KV attention) is carried as one 64-bit word per node,
//   anc[i] = anc[parent[i]] | (1 << i),   anc[0] = 1,
// so node i sees tree key t exactly when bit t of anc[i] is set.  Keys are
// rotated at position L_b + depth[i] (TensorRT-LLM issue 1946, position
// offsets for Medusa tokens) and land at logical slot L_b + i.
#include "kernels.cuh"

namespace mt {

namespace {

constexpr int kPrepThreads = 256;

// Exclusive scan of n values with one block; returns the total.
__device__ int block_exclusive_scan(int* data, int n, int* warp_sums) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int beg = min(n, tid * per), end = min(n, beg + per);
  int local = 0;
  for (int i = beg; i < end; ++i) local += data[i];
  int incl = local;
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int nw = blockDim.x >> 5;
    int v = lane < nw ? warp_sums[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane < nw) warp_sums[lane] = v;  // inclusive over warps
  }
  __syncthreads();
  int offset = (warp > 0 ? warp_sums[warp - 1] : 0) + incl - local;
  int total = warp_sums[(blockDim.x >> 5) - 1];
  int run = offset;
  for (int i = beg; i < end; ++i) {
    int v = data[i];
    data[i] = run;
    run += v;
  }
  __syncthreads();
  return total;
}

template <typename T>
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(PrepParams a) {
  const int tid = threadIdx.x;
  if (blockIdx.x == gridDim.x - 1) {
    // ---- schedule block: validate trees, ancestor masks, tile prefix ----
    extern __shared__ int s_nt[];  // [B + 1]
    __shared__ int s_warp[32];
    for (int b = tid; b < a.B; b += blockDim.x) {
      const int* par = a.tree_parents + (size_t)b * a.T;
      const int* dep = a.tree_depths + (size_t)b * a.T;
      unsigned long long* anc = a.anc + (size_t)b * a.T;
      bool ok = par[0] == -1 && dep[0] == 0;
      unsigned long long m0 = 1ull;
      anc[0] = m0;
      for (int i = 1; i < a.T; ++i) {
        int p = par[i];
        bool good = p >= 0 && p < i && dep[i] == dep[p] + 1;
        ok = ok && good;
        anc[i] = good ? (anc[p] | (1ull << i)) : 0ull;
      }
      int L = a.seq_lens[b];
      bool len_ok = L >= 0 && (long long)L + a.T <= (long long)a.max_blocks * a.P;
      if (!ok) set_status(a.status, kStTree);
      if (!len_ok) set_status(a.status, kStPages);
      if (!ok || !len_ok) anc[0] = 0ull;  // marks the sequence invalid
      s_nt[b] = (ok && len_ok) ? (L + a.T + kTileKeys - 1) / kTileKeys : 0;
    }
    __syncthreads();
    int total = block_exclusive_scan(s_nt, a.B, s_warp);
    for (int b = tid; b < a.B; b += blockDim.x) a.tile_pfx[b] = s_nt[b];
    if (tid == 0) a.tile_pfx[a.B] = total;
    return;
  }
  // ---- scatter: one warp per (b, node, kv head) row ----
  const int warp = tid >> 5, lane = tid & 31;
  const long long row = (long long)blockIdx.x * (kPrepThreads / 32) + warp;
  const long long nrows = (long long)a.B * a.T * a.Hkv;
  if (row >= nrows) return;
  const int kvh = (int)(row % a.Hkv);
  const int i = (int)((row / a.Hkv) % a.T);
  const int b = (int)(row / ((long long)a.Hkv * a.T));
  const int L = a.seq_lens[b];
  const int depth = a.tree_depths[(size_t)b * a.T + i];
  const long long slot = (long long)L + i;
  const long long pos = (long long)L + depth;
  if (L < 0 || slot / a.P >= a.max_blocks) {
    if (lane == 0) set_status(a.status, kStPages);
    return;
  }
  if (depth < 0 || pos >= a.max_pos) {
    if (lane == 0) set_status(a.status, kStTree);
    return;
  }
  const int page = a.block_tables[(size_t)b * a.max_blocks + slot / a.P];
  if (page < 0 || page >= a.num_pages) {
    if (lane == 0) set_status(a.status, kStPages);
    return;
  }
  const int half = a.D / 2;
  const T* kn = static_cast<const T*>(a.k_new) + (size_t)row * a.D;
  const T* vn = static_cast<const T*>(a.v_new) + (size_t)row * a.D;
  const size_t dst = (((size_t)page * a.Hkv + kvh) * a.P + slot % a.P) * a.D;
  T* kc = static_cast<T*>(a.k_cache) + dst;
  T* vc = static_cast<T*>(a.v_cache) + dst;
  const float2* cs = a.rope + (size_t)pos * half;
  for (int j = lane; j < half; j += 32) {
    float lo = Act<T>::to_f(kn[j]), hi = Act<T>::to_f(kn[j + half]);
    float2 c = cs[j];
    float olo, ohi;
    rope_pair(lo, hi, c.x, c.y, olo, ohi);
    kc[j] = Act<T>::from_f(olo);
    kc[j + half] = Act<T>::from_f(ohi);
  }
  for (int j = lane; j < a.D; j += 32) vc[j] = vn[j];
}

}  // namespace

cudaError_t launch_prep(const PrepParams& a, int dtype, cudaStream_t stream) {
  long long nrows = (long long)a.B * a.T * a.Hkv;
  long long blocks = (nrows + kPrepThreads / 32 - 1) / (kPrepThreads / 32) + 1;
  size_t smem = sizeof(int) * (size_t)(a.B + 1);
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  dim3 grid((unsigned)blocks);
  switch (dtype) {
    case 0: prep_kernel<float><<<grid, kPrepThreads, smem, stream>>>(a); break;
    case 1: prep_kernel<__half><<<grid, kPrepThreads, smem, stream>>>(a); break;
    default: prep_kernel<__nv_bfloat16><<<grid, kPrepThreads, smem, stream>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace mt
