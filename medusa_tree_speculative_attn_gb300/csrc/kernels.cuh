// Kernel parameter blocks and launchers (internal to the library).
#pragma once

#include <utility>

#include "common.cuh"

namespace mt {

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation, so that its launch overlaps the
// completion of the kernel before it on the stream.  A kernel calls
// pdl_wait() before it reads or writes memory that an earlier kernel may
// touch: it returns once the preceding kernel has completed and its writes
// are visible (at once in a normal launch).  No kernel releases its successor
// early (griddepcontrol.launch_dependents): the release happens as its CTAs
// exit, so every earlier kernel has completed when a successor starts.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct PrepParams {
  int B, T, Hq, Hkv, D, P, max_blocks, num_pages, max_pos;
  const void* q;
  void* q_rot;  // [B][T][Hq][D] act
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  const int* block_tables;
  const int* seq_lens;
  const int* tree_parents;
  const int* tree_depths;
  const float2* rope;
  int* status;
  unsigned long long* anc;  // [B][T]
  int* tile_pfx;            // [B + 1]
  Sched sched;              // the attention kernel's schedule (tile_pfx unused)
  int* piece_table;         // count[G], padded, + PieceRec[G][kMaxPieceRecs], or null
  int cache_fp8;            // the caches hold FP8 E4M3 codes of value / scale
  float k_scale, v_scale;
};

// Candidate tree tokens from the Medusa heads (cand.cu).
constexpr int kMaxChoices = 16;  // choice ranks per depth the kernel supports

struct CandParams {
  int B, T, V, heads;
  const void* root_logits;  // [B][V]
  const void* head_logits;  // [B][heads][V]
  const int* parents;       // [B][T]
  int* tokens;              // [B][T] out
  int* status;
};

struct AcceptParams {
  int B, T, V, max_depth;
  const int* tokens;
  const void* logits;
  const int* parents;
  int* argmax_out;
  int* accept_len;
  int* accept_path;
  int* next_token;
  int* status;
  unsigned int* counters;  // [B], left at zero
  // A row split over nsplit CTAs (few rows: more CTAs than rows keep the GPU
  // busy): the slices fold their best (value, lowest index) into row_keys and
  // count themselves in row_counters; the last slice continues as the row's
  // CTA.  Both [B*T], left at zero.
  unsigned long long* row_keys;
  unsigned int* row_counters;
  int nsplit;
};

// Typical acceptance's extra arguments (accept.cu).
struct TypicalParams {
  float k;                 // log2(e) / temperature
  float epsilon, delta;    // threshold min(epsilon, delta * exp(-entropy))
  float4* stats;           // [B*T] per row (max of y, Z, threshold, unused), workspace
  int* node_accept;        // [B][T] each node's own test (1 at the root)
  // rows split over AcceptParams::nsplit CTAs: each slice's (max of y, Z, S),
  // [B*T][nsplit] (at most kTypSplitRows rows of kTypMaxSplits slices), workspace
  float4* split_stats;
};
constexpr int kTypSplitRows = 1024;  // typical-acceptance rows are split only up to this many
constexpr int kTypMaxSplits = 16;

struct CommitParams {
  int B, T, Hkv, D, P, max_blocks, num_pages, max_depth, rel_width, elem_bytes;
  const int* accept_path;
  const int* accept_len;
  void* k_cache;
  void* v_cache;
  int* block_tables;
  int* seq_lens;
  int* released;
  int* status;
};

// Persistent CTAs per SM for each attention kernel.
constexpr int kSimtRows = 64;
constexpr int kSimtCtasPerSm = 2;
constexpr int kTcRows = 256;
constexpr int kTcCtasPerSm = 1;

cudaError_t launch_prep(const PrepParams& a, int dtype, cudaStream_t stream);
// An FP8 (E4M3) KV cache for the CUDA-core kernel: codes of value / scale (the
// tensor-core kernel takes the same facts through AttnParams).
struct Fp8Cache {
  int on;
  float k_scale, v_scale;
};

cudaError_t launch_attn_simt(const AttnParams& a, const Fp8Cache& f8, int dtype, cudaStream_t stream);
// Encode TMA descriptors (128 bytes, 64-byte aligned): a paged cache, and the
// rotated queries [B*T][Hq][D] in boxes of 128 rows (128/g nodes x g heads).
cudaError_t make_cache_tmap(void* map_out, const void* base, int dtype, int num_pages, int Hkv,
                            int P, int D);
cudaError_t make_q_tmap(void* map_out, const void* base, int dtype, int BT, int Hq, int g, int D);
cudaError_t make_cache_tmap_e4m3(void* map_out, const void* base, int num_pages, int Hkv, int P, int D);
// Whether the tensor-core kernel supports a configuration.
bool tc_supported(int D, int g);
cudaError_t launch_attn_tc(const AttnParams& a, int dtype, const void* tmap_k, const void* tmap_v,
                           const void* tmap_q, cudaStream_t stream);
cudaError_t launch_combine(const AttnParams& a, int dtype, cudaStream_t stream);
cudaError_t launch_cand(const CandParams& a, int dtype, cudaStream_t stream);
cudaError_t launch_accept(const AcceptParams& a, int dtype, cudaStream_t stream);
// Acceptance and, per sequence as soon as its path is known, the KV commit.
cudaError_t launch_accept_commit(const AcceptParams& a, const CommitParams& c, int dtype, cudaStream_t stream);
cudaError_t launch_accept_typical(const AcceptParams& a, const TypicalParams& t, int dtype, cudaStream_t stream);
cudaError_t launch_commit(const CommitParams& a, cudaStream_t stream);

}  // namespace mt
