// Tree preparation: validates every sequence's tree, builds the per-node
// ancestor bitmasks and the tile schedule, rotates the tree tokens' queries
// into the workspace, and writes their rotated keys and raw values into their
// scratch slots of the paged cache.
//
// The tree mask (vLLM issue 1171, void-main: the Medusa tree mask inside the
// cached-KV attention) is carried as one 64-bit word per node,
//   anc[i] = anc[parent[i]] | (1 << i),   anc[0] = 1,
// so node i sees tree key t exactly when bit t of anc[i] is set.  Keys are
// rotated at position L_b + depth[i] (TensorRT-LLM issue 1946, position
// offsets for Medusa tokens); keys land at logical slot L_b + i, queries in a
// [B][T][Hq][D] workspace array read by the attention kernels.
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
  // ---- one warp per row: B*T*Hq query rows, then B*T*Hkv key/value rows ----
  const int warp = tid >> 5, lane = tid & 31;
  long long row = (long long)blockIdx.x * (kPrepThreads / 32) + warp;
  const long long nq = (long long)a.B * a.T * a.Hq;
  const long long nk = (long long)a.B * a.T * a.Hkv;
  if (row >= nq + nk) return;
  const bool is_q = row < nq;
  if (!is_q) row -= nq;
  const int H = is_q ? a.Hq : a.Hkv;
  const int i = (int)((row / H) % a.T);
  const int b = (int)(row / ((long long)H * a.T));
  const int L = a.seq_lens[b];
  const int depth = a.tree_depths[(size_t)b * a.T + i];
  const long long pos = (long long)L + depth;
  if (L < 0 || depth < 0 || pos >= a.max_pos) {
    if (lane == 0) set_status(a.status, L < 0 ? kStPages : kStTree);
    return;
  }
  const int half = a.D / 2;
  const float2* cs = a.rope + (size_t)pos * half;
  const T* src;
  T* dst;
  if (is_q) {
    src = static_cast<const T*>(a.q) + (size_t)row * a.D;
    dst = static_cast<T*>(a.q_rot) + (size_t)row * a.D;
  } else {
    const int kvh = (int)(row % a.Hkv);
    const long long slot = (long long)L + i;
    if (slot / a.P >= a.max_blocks) {
      if (lane == 0) set_status(a.status, kStPages);
      return;
    }
    const int page = a.block_tables[(size_t)b * a.max_blocks + slot / a.P];
    if (page < 0 || page >= a.num_pages) {
      if (lane == 0) set_status(a.status, kStPages);
      return;
    }
    const size_t off = (((size_t)page * a.Hkv + kvh) * a.P + slot % a.P) * a.D;
    src = static_cast<const T*>(a.k_new) + (size_t)row * a.D;
    dst = static_cast<T*>(a.k_cache) + off;
    const T* vn = static_cast<const T*>(a.v_new) + (size_t)row * a.D;
    T* vc = static_cast<T*>(a.v_cache) + off;
    for (int j = lane; j < a.D; j += 32) vc[j] = vn[j];
  }
  for (int j = lane; j < half; j += 32) {
    const float2 c = cs[j];
    float olo, ohi;
    rope_pair(Act<T>::to_f(src[j]), Act<T>::to_f(src[j + half]), c.x, c.y, olo, ohi);
    dst[j] = Act<T>::from_f(olo);
    dst[j + half] = Act<T>::from_f(ohi);
  }
}

}  // namespace

cudaError_t launch_prep(const PrepParams& a, int dtype, cudaStream_t stream) {
  long long nrows = (long long)a.B * a.T * ((long long)a.Hq + a.Hkv);
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
