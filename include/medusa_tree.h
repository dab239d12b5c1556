/*
 * medusa_tree.h -- C ABI of the Medusa tree-verification library (sm_103a).
 *
 * One verify step of Medusa speculative decoding, for every sequence of a
 * batch, in three calls on one CUDA stream:
 *
 *   mt_tree_attn_paged    the T candidate tokens of the sequence's speculation
 *                         tree attend, in one pass, to the sequence's paged KV
 *                         cache plus their own tree ancestors (the "tree mask"),
 *                         with RoPE applied at position prefix_len + depth;
 *   mt_tree_accept_greedy per-node vocab argmax of the target logits and the
 *                         longest root path whose tokens match their parent's
 *                         argmax;
 *   mt_kv_commit          the accepted nodes' K/V move into the sequence's next
 *                         cache slots, the sequence length grows and the tree
 *                         scratch pages past the new length are released;
 *
 * or in two, with mt_tree_accept_commit doing the last two in one launch.
 * mt_tree_accept_typical replaces greedy acceptance by typical acceptance
 * (a tempered-probability threshold), and mt_tree_candidates builds the tree's
 * tokens from the Medusa heads before the step.
 *
 * What the pages fix, per call:
 *  - vLLM issue 1171 "[Discussion] Will vLLM consider using Speculative
 *    Sampling to accelerating LLM decoding?": several new tokens attend to an
 *    existing paged KV cache (comment by zhaoyang-star); the Medusa tree mask
 *    is applied inside the cached-KV attention; block tables are updated when a
 *    candidate is accepted and the other blocks released; the step returns a
 *    list of tokens (comment by void-main listing the needed changes); with
 *    several query tokens per sequence the products belong on tensor cores
 *    (void-main on PagedFlashAttention).
 *  - TensorRT-LLM issue 1946 "How to use Medusa to support non llama models?",
 *    answer by rakib-hasan: a position-offset tensor lets RoPE rotate each
 *    Medusa token at its own position.
 *  - lmdeploy PR 1231 "[WIP] support Medusa": greedy acceptance at LM-head
 *    temperature 0 over a 64-choice tree; a tree-mask kernel in the
 *    Flash-Decoding style (split keys, merge partial softmaxes).
 *  - mlc-llm issue 2319 "[Feature Request] Medusa support": tree attention and
 *    the KV cache update are the two hard parts.
 *
 * Conventions (all calls):
 *  - Every tensor is caller-owned device memory, dense, in the layouts given
 *    below, 16-byte aligned.  The library allocates device memory only in
 *    mt_rope_create.
 *  - Calls are asynchronous on `stream` and never synchronise, except
 *    mt_read_status and mt_rope_create.
 *  - Errors the host can see (null pointers, unsupported dtype / head_dim /
 *    tree size, misalignment, a workspace that is too small) return a negative
 *    mt_status before anything is launched.  Errors only the device can see
 *    (malformed trees, page ids out of range, block tables shorter than
 *    prefix + T slots, a bounded wait that gave up) are recorded in a status
 *    word inside the workspace and read with mt_read_status; the outputs of
 *    an affected sequence are then unspecified, and nothing outside the
 *    caller's buffers is touched.  No kernel traps or asserts.
 *  - Node order: node 0 is the root (parent -1, depth 0): the token chosen by
 *    the previous step, not yet in the cache.  Every other node i has
 *    0 <= parent[i] < i and depth[i] = depth[parent[i]] + 1.  T <= 64.
 *  - Paged cache layout: k_cache and v_cache are [num_pages][Hkv][P][D] in the
 *    act dtype; logical slot s of sequence b is row s % P of page
 *    block_tables[b][s / P].  block_tables is int32 [B][max_blocks_per_seq]
 *    (unused entries may hold -1); seq_lens is int32 [B], the committed prefix
 *    length L_b.  The table must cover slots 0 .. L_b + T - 1: slots
 *    L_b .. L_b + T - 1 are the tree's scratch region.
 */
#ifndef MEDUSA_TREE_H_
#define MEDUSA_TREE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MT_OK = 0,
  MT_ERR_INVALID_ARG = -1,  /* null pointer, bad size, misaligned, workspace too small */
  MT_ERR_UNSUPPORTED = -2,  /* dtype / head_dim / page size / tree size not supported */
  MT_ERR_TREE = -3,         /* (device) parents or depths violate the node-order rule */
  MT_ERR_PAGES = -4,        /* (device) page id out of range or block table too short */
  MT_ERR_CUDA = -5,         /* a CUDA runtime call failed */
  MT_ERR_TIMEOUT = -6       /* (device) a bounded pipeline wait gave up */
} mt_status;

/* MT_E4M3 is a cache element type only (see mt_attn_desc.cache_dtype). */
typedef enum { MT_F32 = 0, MT_F16 = 1, MT_BF16 = 2, MT_E4M3 = 3 } mt_dtype;

/* Kernel choice for mt_tree_attn_paged.  AUTO: tensor cores (tcgen05, TMEM,
 * TMA) for fp16/bf16, the SIMT kernel for fp32.  SIMT: the CUDA-core kernel for
 * every dtype (a second, independent implementation used by the tests). */
typedef enum { MT_KERNEL_AUTO = 0, MT_KERNEL_SIMT = 1, MT_KERNEL_TC = 2 } mt_kernel;

typedef struct {
  int batch;               /* B >= 1 */
  int tree_size;           /* T, 1..64 */
  int num_q_heads;         /* Hq, a multiple of Hkv */
  int num_kv_heads;        /* Hkv */
  int head_dim;            /* D: 64 or 128 */
  int page_size;           /* P: 16 */
  int max_blocks_per_seq;  /* columns of block_tables */
  int num_pages;           /* pages in the cache pool */
  int num_splits;          /* 0: balanced schedule over the whole batch (each
                              persistent CTA takes an equal share of all key
                              tiles); n > 0: every (sequence, KV head) is split
                              into n key chunks merged by a log-sum-exp pass */
  mt_dtype dtype;          /* q, k_new, v_new, out, and the caches unless cache_dtype says
                              otherwise */
  float sm_scale;          /* softmax scale; 0 means 1/sqrt(D) */
  int kernel;              /* an mt_kernel value */
  /* FP8 KV cache (a reading: the pages this library follows define none).
   * cache_dtype 0: the caches hold dtype.  MT_E4M3: they hold OCP FP8 E4M3
   * codes (no infinities; largest finite 448) of value / scale, one scale for
   * K and one for V, and every cached element stands for decode(code) *
   * scale, the tree's own K/V included: mt_tree_attn_paged writes the code of
   * (act-rounded rotated key or raw value) / scale, divided in fp32 and
   * rounded to nearest even with saturation to +-448, and reads every visible
   * slot back through the scale.  Runs on either kernel: the tensor-core
   * kernel (fp16/bf16 dtype) loads the codes with TMA, converts them exactly
   * to the act dtype in shared memory, and applies k_scale with the softmax
   * scale and v_scale to the output; MT_KERNEL_AUTO picks it as for a 16-bit
   * cache.  mt_kv_commit and mt_tree_accept_commit move the 1-byte elements.
   * k_scale, v_scale: positive and finite for MT_E4M3, ignored otherwise. */
  int cache_dtype;
  float k_scale;
  float v_scale;
} mt_attn_desc;

/* ---- RoPE table ----------------------------------------------------------
 * Library-owned fp32 cos/sin table [max_pos][D/2] on the current device, built
 * on the host in double precision (NeoX / LLaMA half-split form):
 *   inv_freq_j = pow(base, -(2j)/D), theta = pos * inv_freq_j (IEEE double),
 *   stored values (float)cos(theta), (float)sin(theta).
 * The rotation of a head vector x at position pos, for j < D/2, in fp32 with
 * each product and sum rounded separately (no fused multiply-add):
 *   x'[j] = x[j]*c - x[j+D/2]*s,   x'[j+D/2] = x[j+D/2]*c + x[j]*s,
 * then rounded to nearest-even in the act dtype.  Tree token i of sequence b is
 * rotated at pos = seq_lens[b] + tree_depths[b][i] (the Medusa position offset,
 * TensorRT-LLM issue 1946).  max_pos must exceed every such position.
 * mt_rope_create allocates and synchronises the current device; destroy frees. */
typedef struct mt_rope mt_rope;
int mt_rope_create(double base, int head_dim, int max_pos, mt_rope** out);
int mt_rope_destroy(mt_rope* rope);

/* ---- Tree attention -------------------------------------------------------
 * For each sequence b, tree node i and query head h (KV head h / (Hq/Hkv)):
 *   out[b][i][h] = sum_j softmax_j(q'.k_j * sm_scale) v_j
 * over the keys j = prefix slots 0 .. L_b-1 of the paged cache, plus the tree
 * keys of i's ancestors, i itself included.  q' and the tree keys are rotated
 * at position L_b + depth[i]; the prefix keys are used as stored.  Before the
 * attention, node i's rotated key and raw value are written to logical slot
 * L_b + i (the scratch region), where mt_kv_commit later finds them; slots
 * below L_b are never written.  Accumulation in fp32, output rounded to nearest
 * even in the act dtype.  Where the schedule splits a (sequence, KV head) into
 * pieces, each piece's own softmax output is rounded to the act dtype first
 * and the fp32 merge is rounded again (the same tolerance holds).
 *   q      [B][T][Hq][D]    act   (not rotated)
 *   k_new  [B][T][Hkv][D]   act   (the tree tokens' keys, not rotated)
 *   v_new  [B][T][Hkv][D]   act
 *   k_cache, v_cache        act   paged layout above (written: scratch slots)
 *   block_tables, seq_lens  int32 (read only)
 *   tree_parents, tree_depths int32 [B][T]
 *   out    [B][T][Hq][D]    act
 *   workspace: device memory of mt_tree_attn_workspace_size(desc) bytes,
 *     zero-filled before its first use; it holds the device status word, the
 *     ancestor bitmasks, the schedule and the split-KV partial results.  One
 *     workspace per stream: calls sharing a workspace must not overlap. */
size_t mt_tree_attn_workspace_size(const mt_attn_desc* desc);
int mt_tree_attn_paged(const mt_attn_desc* desc, const void* q, const void* k_new,
                       const void* v_new, void* k_cache, void* v_cache,
                       const int32_t* block_tables, const int32_t* seq_lens,
                       const int32_t* tree_parents, const int32_t* tree_depths,
                       const mt_rope* rope, void* out, void* workspace, size_t ws_bytes,
                       cudaStream_t stream);

/* ---- Tree attention without allocation -------------------------------------
 * The pages this library follows have no counterpart for this call.  It is for
 * callers that cannot allocate device memory on the calling path -- for
 * example a serving loop that must not risk the device synchronisation and
 * out-of-memory failures of cudaMalloc between steps, or code that is handed
 * only its input and output buffers by a memory pool it does not own.
 * Same computation, arguments and layouts as mt_tree_attn_paged, but no
 * workspace argument: the workspace is a fixed 64 MiB array that the library
 * reserves on every device it is loaded on, held until the process exits.
 *  - Returns MT_ERR_UNSUPPORTED when mt_tree_attn_workspace_size(desc) exceeds
 *    64 MiB (e.g. very large batches; use mt_tree_attn_paged there).
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress) and keeps it; make that
 *    first call before any stream capture.
 *  - All calls on one device share the array: calls that overlap on the GPU
 *    race, so issue them on one stream or order them with events.
 *  - Each call clears the array's device status word first; if device_status
 *    is not NULL (a device int32), the status after this call's kernels is
 *    copied there on `stream` (MT_OK or the device-detected error). */
int mt_tree_attn_paged_noalloc(const mt_attn_desc* desc, const void* q, const void* k_new,
                               const void* v_new, void* k_cache, void* v_cache,
                               const int32_t* block_tables, const int32_t* seq_lens,
                               const int32_t* tree_parents, const int32_t* tree_depths,
                               const mt_rope* rope, void* out, int32_t* device_status,
                               cudaStream_t stream);

/* ---- Greedy acceptance ----------------------------------------------------
 * Per sequence b (LM head at temperature 0):
 *   argmax_out[b][i] = argmax_v target_logits[b][i][v], the lowest index among
 *                      equal maxima (values compared exactly; +0 equals -0);
 *   node 0 is accepted; node i > 0 is accepted when its parent is and
 *     tree_tokens[b][i] == argmax_out[b][parent[i]];
 *   end = the accepted node of largest depth, the lowest index among equals;
 *   accept_len[b]  = depth of end (accepted tokens besides the root);
 *   accept_path[b] = node ids root .. end, then -1, max_depth+1 entries;
 *   next_token[b]  = argmax_out[b][end], the token the target model adds.
 *   tree_tokens int32 [B][T]; target_logits [B][T][V] in logits_dtype (no NaN);
 *   tree_parents int32 [B][T]; every depth must be <= max_depth.
 *   workspace: mt_tree_accept_workspace_size(B, T) bytes, zero-filled before
 *   first use (status word, per-sequence arrival counters, which every call
 *   leaves at zero, per-node scratch for typical acceptance, and, for rows
 *   split over several CTAs when the rows are few, a per-row key and counter,
 *   also left at zero, and per-slice statistics). */
size_t mt_tree_accept_workspace_size(int batch, int tree_size);
int mt_tree_accept_greedy(int batch, int tree_size, int vocab, int max_depth,
                          mt_dtype logits_dtype, const int32_t* tree_tokens,
                          const void* target_logits, const int32_t* tree_parents,
                          int32_t* argmax_out, int32_t* accept_len, int32_t* accept_path,
                          int32_t* next_token, void* workspace, size_t ws_bytes,
                          cudaStream_t stream);

/* ---- Typical acceptance ---------------------------------------------------
 * The "typical acceptance scheme" that the opening comment of vLLM issue 1171
 * (gesanqiu: tree attention and typical acceptance are what most inference
 * frameworks lack) names beside tree attention; the pages do not define it, and
 * the rule taken is the Medusa paper's (Cai et al. 2024, typical acceptance).
 * Per sequence b, with x the logits row of a node and tau = temperature:
 *   q_v = exp(x_v / tau) / sum_u exp(x_u / tau), H = -sum_v q_v ln q_v;
 *   node i > 0 passes when q[tree_tokens[b][i]] > min(epsilon, delta * exp(-H))
 *     under its parent's row (a token outside [0, vocab) fails); the root
 *     passes; node_accept[b][i] = 1 when node i passes (its own test);
 *   accept_len, accept_path: as in mt_tree_accept_greedy with "accepted" =
 *     every node on the root path passes;
 *   next_token[b] = argmax of the end node's row (lowest index among equal
 *     maxima): the bonus token at temperature 0, no random draw.
 * Computed in fp32: the device sums the row in an order of its own, so a
 * node whose q[token] lies within a relative 1e-5 or so of its threshold may
 * fall either way.  temperature, epsilon, delta: positive and finite
 * (MT_ERR_INVALID_ARG otherwise; also when log2(e) / temperature overflows).
 * Logits: finite, and finite after scaling by log2(e) / temperature.
 * Layouts, max_depth and the workspace as for mt_tree_accept_greedy (the
 * same mt_tree_accept_workspace_size); node_accept int32 [B][T]. */
int mt_tree_accept_typical(int batch, int tree_size, int vocab, int max_depth,
                           mt_dtype logits_dtype, const int32_t* tree_tokens,
                           const void* target_logits, const int32_t* tree_parents,
                           float temperature, float epsilon, float delta, int32_t* node_accept,
                           int32_t* accept_len, int32_t* accept_path, int32_t* next_token,
                           void* workspace, size_t ws_bytes, cudaStream_t stream);

/* ---- KV commit --------------------------------------------------------------
 * For each sequence b, with L = accept_len[b] and len = seq_lens[b]:
 *   for d = 0..L: every KV head's K and V row at logical slot
 *     len + accept_path[b][d] is copied to slot len + d (all sources of a
 *     sequence are read before any destination is written);
 *   seq_lens[b] = len + L + 1;
 *   every logical block p with p*P >= len + L + 1 and p*P < len + T (tree
 *     scratch past the new length) is released: block_tables[b][p] becomes -1
 *     and its page id is listed, in ascending p, in released_pages[b][*], a row
 *     of (T + 2P - 2) / P entries padded with -1.
 *   accept_path int32 [B][max_depth+1], accept_len int32 [B] (as produced by
 *   mt_tree_accept_greedy); k_cache, v_cache, block_tables, seq_lens are
 *   updated in place.  desc supplies B, T, Hkv, D, P, max_blocks_per_seq,
 *   num_pages and the element size: dtype's, or 1 byte when cache_dtype is
 *   MT_E4M3 (the codes move unchanged).  status_ws: at least 256 bytes of device memory whose
 *   first int32 is the device status word (the attention workspace serves). */
int mt_kv_commit(const mt_attn_desc* desc, int max_depth, const int32_t* accept_path,
                 const int32_t* accept_len, void* k_cache, void* v_cache,
                 int32_t* block_tables, int32_t* seq_lens, int32_t* released_pages,
                 void* status_ws, cudaStream_t stream);

/* ---- Greedy acceptance and KV commit in one launch ---------------------------
 * The composition mt_tree_accept_greedy then mt_kv_commit (same results, same
 * arguments and layouts as those two calls), as one kernel launch: each
 * sequence is committed as soon as its path is known, by the CTA that
 * completed its argmax rows, so the step has no launch or round trip between
 * acceptance and commit.  desc supplies B (batch), T (tree_size), Hkv, D, P,
 * max_blocks_per_seq, num_pages and the cache's element size (as for
 * mt_kv_commit); the logits have their own dtype.  workspace: mt_tree_accept_workspace_size(B, T) bytes, zero-filled
 * before first use; its first int32 is the device status word, which records
 * the acceptance errors (MT_ERR_TREE) and the commit errors (MT_ERR_PAGES) of
 * both calls.  Host errors: those of the two calls.  A sequence whose tree is
 * malformed or too deep is accepted as the root alone (accept_len 0) and
 * committed so, exactly as the two calls would do. */
int mt_tree_accept_commit(const mt_attn_desc* desc, int vocab, int max_depth, mt_dtype logits_dtype,
                          const int32_t* tree_tokens, const void* target_logits,
                          const int32_t* tree_parents, int32_t* argmax_out, int32_t* accept_len,
                          int32_t* accept_path, int32_t* next_token, void* k_cache, void* v_cache,
                          int32_t* block_tables, int32_t* seq_lens, int32_t* released_pages,
                          void* workspace, size_t ws_bytes, cudaStream_t stream);

/* ---- Candidate tree tokens ---------------------------------------------------
 * The step before verification (lmdeploy PR 1231 "[WIP] support Medusa":
 * porting `generate_candidates`, Medusa heads at top-k over a 64-choice tree):
 * the tree's tokens from the base model's logits and the Medusa heads' logits.
 * For each sequence b, with the tree given by tree_parents[b] (node 0 the
 * root; parent[0] = -1, 0 <= parent[i] < i):
 *   tree_tokens[b][0] = argmax_v root_logits[b][v] (lowest index among equal
 *                       maxima);
 *   for node i >= 1 at depth d (1 <= d <= heads) with r earlier siblings (nodes
 *   j < i with the same parent): tree_tokens[b][i] = the entry of rank r
 *   (0-based) of head_logits[b][d-1], ordered by larger value first and lower
 *   vocab index first among equal values (+0 and -0 are equal); -1 when the
 *   head has fewer than r + 1 entries (r >= V).
 * root_logits [B][V] and head_logits [B][heads][V] in logits_dtype (no NaN);
 * tree_parents int32 [B][T]; tree_tokens int32 [B][T] out.  The tree template
 * (which choice of which head each node takes) is thus the tree's own shape:
 * the r-th child of a node takes the r-th best token of the next head.
 * Host errors: MT_ERR_INVALID_ARG for null or unaligned pointers or sizes out
 * of range (heads in [1, 63], V >= 1); MT_ERR_UNSUPPORTED for T outside
 * [1, 64] or another dtype.  Device status MT_ERR_TREE (in the first int32 of
 * status_ws, at least 256 bytes, read with mt_read_status): a malformed tree,
 * a node deeper than `heads`, or a node with 16 or more earlier siblings; the
 * tokens of that sequence (malformed tree or depth) or of that depth (too many
 * siblings) are not written.  The pages do not define the tree template; this
 * rule (child rank = head rank) is the reading used here. */
int mt_tree_candidates(int batch, int tree_size, int heads, int vocab, mt_dtype logits_dtype,
                       const void* root_logits, const void* head_logits,
                       const int32_t* tree_parents, int32_t* tree_tokens, void* status_ws,
                       cudaStream_t stream);

/* ---- Status ------------------------------------------------------------------
 * Waits for `stream`, then reads and clears the device status word at the start
 * of `workspace` (MT_OK or the first device-side error since the last read). */
int mt_read_status(void* workspace, cudaStream_t stream, int* device_status);
const char* mt_status_string(int status);

/* ---- Profiling hook -----------------------------------------------------------
 * mt_profile_enable(n) creates n pairs of CUDA events (0 disables and frees
 * them).  While fewer than n pairs are used, each mt_tree_attn_paged call
 * records one pair on its stream, immediately around its main attention kernel
 * (the ancestor/scatter preparation and the split-KV combine are outside it).
 * mt_profile_read waits for the recorded pairs, writes their elapsed times in
 * milliseconds to ms[0 .. *n_out-1] and starts over.  Not thread-safe: for one
 * host thread driving the library. */
int mt_profile_enable(int max_records);
int mt_profile_read(float* ms, int max_records, int* n_out);

/* ---- Timeout test hook --------------------------------------------------------
 * Every pipeline wait of the tensor-core attention kernel (a TMA load landing,
 * an MMA completing, a softmax handing over P) gives up after a bounded time:
 * the kernel then records MT_ERR_TIMEOUT in the status word, lets its other
 * warps stop, waits for its own copies and MMAs in flight, frees its tensor
 * memory and returns, leaving the context usable.  mt_debug_set_wait sets that
 * bound for later mt_tree_attn_paged calls (limit_ns 0 restores the default of
 * 2 s); stall = 1 makes the kernel first wait on a barrier that nothing
 * completes, so that the bound always expires (for tests of the timeout path;
 * stall = 0 is normal operation).  Process-wide, not thread-safe.  Returns
 * MT_ERR_INVALID_ARG for a stall other than 0 or 1.  Not on the pages: the
 * wait bound is how this library reports a stalled pipeline instead of
 * hanging the GPU. */
int mt_debug_set_wait(unsigned long long limit_ns, int stall);

/* Version of this ABI: major * 10000 + minor * 100 + patch. */
int mt_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MEDUSA_TREE_H_ */
