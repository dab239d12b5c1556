// KV commit: keep the accepted candidates' K/V, release the rest (vLLM issue
// 1171, void-main: "update block tables when you accept one candidate and
// release other blocks"; mlc-llm issue 2319: the KV cache update part).
//
// One CTA per sequence.  The CTA first reads the K and V rows of every path
// node (logical slot len + path[d]) of every KV head into shared memory, then
// writes them to slots len + d, so a destination that is also a later source
// (e.g. path [0, 2, 3]: slot len+2 is both) is read before it is overwritten.
// Afterwards seq_lens[b] grows by accept_len + 1 and every logical block that
// starts at or past the new length and holds tree scratch is released.
#include "kernels.cuh"

namespace mt {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) commit_kernel(CommitParams a) {
  extern __shared__ uint4 stage[];  // [n][2][row_vecs]
  __shared__ int s_src[kMaxTree], s_dst[kMaxTree];
  __shared__ int s_ok;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int len = a.seq_lens[b];
  const int L = a.accept_len[b];
  const int* path = a.accept_path + (size_t)b * (a.max_depth + 1);
  const int* bt = a.block_tables + (size_t)b * a.max_blocks;
  const int n = L + 1;
  if (tid == 0)
    s_ok = L >= 0 && L <= a.max_depth && L < a.T && len >= 0 &&
           (long long)len + a.T <= (long long)a.max_blocks * a.P;
  __syncthreads();
  if (tid < n && s_ok) {
    // one thread per path entry: a root path in increasing node order whose
    // source and destination slots map to pages of the pool
    const int d = tid;
    const int node = path[d];
    bool ok = node >= 0 && node < a.T && (d == 0 || node > path[d - 1]);
    if (ok) {
      const int ss = len + node, ds = len + d;
      const int sp = bt[ss / a.P], dp = bt[ds / a.P];
      ok = sp >= 0 && sp < a.num_pages && dp >= 0 && dp < a.num_pages;
      s_src[d] = sp * a.P + ss % a.P;  // page-row index (per head stride added below)
      s_dst[d] = dp * a.P + ds % a.P;
    }
    if (!ok) s_ok = 0;
  }
  __syncthreads();
  if (tid == 0 && !s_ok) set_status(a.status, kStPages);
  __syncthreads();
  if (!s_ok) return;
  const int row_bytes = a.D * a.elem_bytes;
  const int rv = row_bytes / 16;  // 16-byte vectors per row
  const size_t head_stride = (size_t)a.P * row_bytes;        // bytes between kv heads in a page
  const size_t page_stride = (size_t)a.Hkv * head_stride;   // bytes per page
  char* kc = static_cast<char*>(a.k_cache);
  char* vc = static_cast<char*>(a.v_cache);
  // as many KV heads per pass as the staging buffer holds (all of them at the
  // usual sizes): every source row of the pass is read before any is written
  const int per_head = n * 2 * rv;
  const int heads_per_pass = max(1, min(a.Hkv, a.stage_vecs / per_head));
  for (int h0 = 0; h0 < a.Hkv; h0 += heads_per_pass) {
    const int nh = min(heads_per_pass, a.Hkv - h0);
    const int total = nh * per_head;
    for (int e = tid; e < total; e += blockDim.x) {
      const int kvh = h0 + e / per_head, r = e % per_head;
      const int d = r / (2 * rv), which = (r / rv) % 2, v = r % rv;
      const int pr = s_src[d];
      const size_t off = (size_t)(pr / a.P) * page_stride + kvh * head_stride +
                         (size_t)(pr % a.P) * row_bytes + (size_t)v * 16;
      stage[e] = *reinterpret_cast<const uint4*>((which ? vc : kc) + off);
    }
    __syncthreads();
    for (int e = tid; e < total; e += blockDim.x) {
      const int kvh = h0 + e / per_head, r = e % per_head;
      const int d = r / (2 * rv), which = (r / rv) % 2, v = r % rv;
      const int pr = s_dst[d];
      const size_t off = (size_t)(pr / a.P) * page_stride + kvh * head_stride +
                         (size_t)(pr % a.P) * row_bytes + (size_t)v * 16;
      *reinterpret_cast<uint4*>((which ? vc : kc) + off) = stage[e];
    }
    __syncthreads();
  }
  if (tid == 0) {
    const int new_len = len + n;
    a.seq_lens[b] = new_len;
    int* rel = a.released + (size_t)b * a.rel_width;
    int nrel = 0;
    int* btw = a.block_tables + (size_t)b * a.max_blocks;
    const int first = (new_len + a.P - 1) / a.P;     // first block starting at or past new_len
    const int last = (len + a.T - 1) / a.P;          // last block holding tree scratch
    for (int p = first; p <= last; ++p) {
      if (nrel < a.rel_width) rel[nrel++] = btw[p];
      btw[p] = -1;
    }
    for (; nrel < a.rel_width; ++nrel) rel[nrel] = -1;
  }
}

}  // namespace

cudaError_t launch_commit(const CommitParams& a, cudaStream_t stream) {
  const int n_max = (a.max_depth + 1 < a.T ? a.max_depth + 1 : a.T);
  const size_t per_head = (size_t)n_max * 2 * a.D * a.elem_bytes;  // bytes
  size_t smem = per_head * (size_t)a.Hkv;
  const size_t cap = 160 * 1024;
  if (smem > cap) smem = per_head > cap ? per_head : cap / per_head * per_head;
  CommitParams p = a;
  p.stage_vecs = (int)(smem / 16);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(commit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  commit_kernel<<<a.B, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mt
