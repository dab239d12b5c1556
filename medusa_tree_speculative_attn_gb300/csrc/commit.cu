// KV commit: keep the accepted candidates' K/V, release the rest (vLLM issue
// 1171, void-main: "update block tables when you accept one candidate and
// release other blocks"; mlc-llm issue 2319: the KV cache update part).
//
// One CTA per sequence: it reads the sequence's accept length, path and length
// (together), then its block-table window, and runs the per-sequence commit
// (commit_seq.cuh), which moves the rows through a shared-memory stage, grows
// seq_lens[b] by accept_len + 1 and releases every logical block that starts
// at or past the new length and holds tree scratch.
#include "commit_seq.cuh"

namespace mt {

namespace {

constexpr int kThreads = 128;
constexpr int kStageCap = 32 * 1024;

__global__ void __launch_bounds__(kThreads) commit_kernel(CommitParams a, int stage_vecs) {
  extern __shared__ uint4 stage[];
  __shared__ CommitSmem sm;
  __shared__ int s_path[kMaxTree];
  __shared__ int s_L, s_len;
  const int b = blockIdx.x, tid = threadIdx.x;
  pdl_wait();
  if (tid == 0) {
    s_L = a.accept_len[b];
    s_len = a.seq_lens[b];
  }
  const int* path = a.accept_path + (size_t)b * (a.max_depth + 1);
  for (int d = tid; d <= a.max_depth; d += blockDim.x) s_path[d] = path[d];
  __syncthreads();
  commit_load_window(a, b, s_len, sm);
  __syncthreads();
  commit_sequence(a, b, s_len, s_L, s_path, sm, stage, stage_vecs);
}

}  // namespace

cudaError_t launch_commit(const CommitParams& a, cudaStream_t stream) {
  const int sv = commit_stage_vecs(a, kStageCap);
  return launch_pdl(commit_kernel, dim3(a.B), dim3(kThreads), (size_t)sv * 16, stream, a, sv);
}

}  // namespace mt
