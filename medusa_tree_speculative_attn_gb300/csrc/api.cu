// C ABI of the Medusa tree-verification library: host-side validation,
// workspace layout, the RoPE table, and the kernel launches.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/medusa_tree.h"
#include "kernels.cuh"

// One NVTX range per library call, named after its C entry point, for a
// timeline tool (nothing is recorded unless such a tool is attached).
struct mt_call_range {
  explicit mt_call_range(const char* name) { nvtxRangePushA(name); }
  ~mt_call_range() { nvtxRangePop(); }
  mt_call_range(const mt_call_range&) = delete;
  mt_call_range& operator=(const mt_call_range&) = delete;
};

// Bound of the tensor-core kernel's pipeline waits, and the timeout test hook
// (mt_debug_set_wait); read by every attention call.
static unsigned long long g_wait_limit_ns = 0;  // 0: the default (2 s)
static int g_wait_stall = 0;

// Optional timing of the main attention kernel (profiling hook, one host thread).
static cudaEvent_t* g_prof_ev = nullptr;  // [cap][2]
static int g_prof_cap = 0;
static int g_prof_n = 0;

struct mt_rope {
  float2* table;  // [max_pos][D/2] (cos, sin)
  int head_dim;
  int max_pos;
  int device;
};

namespace {

using namespace mt;

constexpr size_t kAlign = 256;
constexpr int kMaxBatch = 8192;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int elem_bytes(mt_dtype dt) { return dt == MT_F32 ? 4 : 2; }

bool fp8_cache(const mt_attn_desc* d) { return d->cache_dtype == MT_E4M3; }

// Bytes of one cache element.
int cache_elem_bytes(const mt_attn_desc* d) { return fp8_cache(d) ? 1 : elem_bytes(d->dtype); }

// Which attention kernel a descriptor runs (an FP8 cache included: the
// tensor-core kernel converts its codes to the act dtype in shared memory).
int select_kernel(const mt_attn_desc* d) {
  if (d->kernel == MT_KERNEL_SIMT) return MT_KERNEL_SIMT;
  if (d->kernel == MT_KERNEL_TC) return MT_KERNEL_TC;
  if (d->dtype == MT_F32) return MT_KERNEL_SIMT;
  return tc_supported(d->head_dim, d->num_q_heads / d->num_kv_heads) ? MT_KERNEL_TC : MT_KERNEL_SIMT;
}

struct WsLayout {
  size_t anc, pfx, pieces, qrot, ml, o, total;
  int rows, rows_per_group, part_rows, nrg, G, nslots;
};

int device_sm_count(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MT_ERR_CUDA;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MT_ERR_CUDA;
  return MT_OK;
}

int layout_for(const mt_attn_desc* d, int kernel, WsLayout* w) {
  int sms = 0;
  int st = device_sm_count(&sms);
  if (st != MT_OK) return st;
  const int g = d->num_q_heads / d->num_kv_heads;
  w->rows = d->tree_size * g;
  w->rows_per_group = kernel == MT_KERNEL_SIMT ? kSimtRows : kTcRows;
  w->nrg = (w->rows + w->rows_per_group - 1) / w->rows_per_group;
  w->part_rows = w->rows < w->rows_per_group ? w->rows : w->rows_per_group;
  w->G = sms * (kernel == MT_KERNEL_SIMT ? kSimtCtasPerSm : kTcCtasPerSm);
  const long long nseg = (long long)d->batch * d->num_kv_heads * w->nrg;
  const long long nslots = d->num_splits > 0 ? nseg * d->num_splits : nseg + w->G;
  if (nslots > (1ll << 30)) return MT_ERR_INVALID_ARG;
  w->nslots = (int)nslots;
  size_t off = kAlign;  // status word and padding
  w->anc = off;
  off = align_up(off + sizeof(unsigned long long) * (size_t)d->batch * d->tree_size);
  w->pfx = off;
  off = align_up(off + sizeof(int) * (size_t)(d->batch + 1));
  w->pieces = off;  // the tensor-core kernel's per-CTA piece lists
  if (kernel != MT_KERNEL_SIMT)
    off = align_up(off + sizeof(int) * (size_t)piece_rec_offset(w->G) + sizeof(PieceRec) * kMaxPieceRecs * (size_t)w->G);
  w->qrot = off;
  off = align_up(off + (size_t)elem_bytes(d->dtype) * d->batch * d->tree_size * d->num_q_heads *
                           d->head_dim);
  w->ml = off;
  off = align_up(off + sizeof(float2) * (size_t)nslots * w->part_rows);
  w->o = off;
  off = align_up(off + (size_t)elem_bytes(d->dtype) * nslots * w->part_rows * d->head_dim);
  w->total = off;
  return MT_OK;
}

int check_desc(const mt_attn_desc* d) {
  if (!d) return MT_ERR_INVALID_ARG;
  if (d->batch < 1 || d->batch > kMaxBatch) return MT_ERR_INVALID_ARG;
  if (d->tree_size < 1 || d->tree_size > kMaxTree) return MT_ERR_UNSUPPORTED;
  if (d->num_kv_heads < 1 || d->num_q_heads < 1 || d->num_q_heads % d->num_kv_heads)
    return MT_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128) return MT_ERR_UNSUPPORTED;
  if (d->page_size != 16) return MT_ERR_UNSUPPORTED;
  if (d->max_blocks_per_seq < 1 || d->num_pages < 1) return MT_ERR_INVALID_ARG;
  if ((long long)d->num_pages * d->num_kv_heads * d->page_size >= (1ll << 31))
    return MT_ERR_UNSUPPORTED;
  if (d->num_splits < 0 || d->num_splits > 4096) return MT_ERR_INVALID_ARG;
  if (d->dtype != MT_F32 && d->dtype != MT_F16 && d->dtype != MT_BF16) return MT_ERR_UNSUPPORTED;
  if (d->kernel < MT_KERNEL_AUTO || d->kernel > MT_KERNEL_TC) return MT_ERR_INVALID_ARG;
  if (d->kernel == MT_KERNEL_TC &&
      (d->dtype == MT_F32 || !tc_supported(d->head_dim, d->num_q_heads / d->num_kv_heads)))
    return MT_ERR_UNSUPPORTED;
  if (!(d->sm_scale >= 0.f) || std::isinf(d->sm_scale)) return MT_ERR_INVALID_ARG;
  if (d->cache_dtype != 0 && d->cache_dtype != MT_E4M3) return MT_ERR_UNSUPPORTED;
  if (fp8_cache(d)) {
    if (!(d->k_scale > 0.f) || std::isinf(d->k_scale) || !(d->v_scale > 0.f) || std::isinf(d->v_scale))
      return MT_ERR_INVALID_ARG;
  }
  return MT_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MT_OK : MT_ERR_CUDA; }

}  // namespace

extern "C" {

int mt_version(void) { return 10000; }

const char* mt_status_string(int s) {
  switch (s) {
    case MT_OK: return "ok";
    case MT_ERR_INVALID_ARG: return "invalid argument";
    case MT_ERR_UNSUPPORTED: return "unsupported configuration";
    case MT_ERR_TREE: return "malformed tree (parents/depths)";
    case MT_ERR_PAGES: return "page id out of range or block table too short";
    case MT_ERR_CUDA: return "CUDA runtime error";
    case MT_ERR_TIMEOUT: return "bounded device wait gave up";
    default: return "unknown status";
  }
}

int mt_rope_create(double base, int head_dim, int max_pos, mt_rope** out) {
  if (!out || !(base > 0.0) || (head_dim != 64 && head_dim != 128) || max_pos < 1 ||
      (long long)max_pos * head_dim > (1ll << 31))
    return MT_ERR_INVALID_ARG;
  *out = nullptr;
  const int half = head_dim / 2;
  std::vector<float2> host((size_t)max_pos * half);
  for (int pos = 0; pos < max_pos; ++pos) {
    for (int j = 0; j < half; ++j) {
      const double inv_freq = std::pow(base, -(2.0 * (double)j) / (double)head_dim);
      const double theta = (double)pos * inv_freq;
      host[(size_t)pos * half + j] = make_float2((float)std::cos(theta), (float)std::sin(theta));
    }
  }
  mt_rope* r = new mt_rope();
  r->head_dim = head_dim;
  r->max_pos = max_pos;
  if (cudaGetDevice(&r->device) != cudaSuccess ||
      cudaMalloc(&r->table, host.size() * sizeof(float2)) != cudaSuccess) {
    delete r;
    return MT_ERR_CUDA;
  }
  if (cudaMemcpy(r->table, host.data(), host.size() * sizeof(float2), cudaMemcpyHostToDevice) !=
      cudaSuccess) {
    cudaFree(r->table);
    delete r;
    return MT_ERR_CUDA;
  }
  *out = r;
  return MT_OK;
}

int mt_rope_destroy(mt_rope* r) {
  if (!r) return MT_OK;
  cudaError_t e = cudaFree(r->table);
  delete r;
  return cuda_status(e);
}

size_t mt_tree_attn_workspace_size(const mt_attn_desc* d) {
  if (check_desc(d) != MT_OK) return 0;
  WsLayout w;
  if (layout_for(d, select_kernel(d), &w) != MT_OK) return 0;
  return w.total;
}

int mt_tree_attn_paged(const mt_attn_desc* d, const void* q, const void* k_new, const void* v_new,
                       void* k_cache, void* v_cache, const int32_t* block_tables,
                       const int32_t* seq_lens, const int32_t* tree_parents,
                       const int32_t* tree_depths, const mt_rope* rope, void* out,
                       void* workspace, size_t ws_bytes, cudaStream_t stream) {
  const mt_call_range range("mt_tree_attn_paged");
  int st = check_desc(d);
  if (st != MT_OK) return st;
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !block_tables || !seq_lens ||
      !tree_parents || !tree_depths || !rope || !out || !workspace)
    return MT_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) % kAlign))
    return MT_ERR_INVALID_ARG;
  if (rope->head_dim != d->head_dim) return MT_ERR_INVALID_ARG;
  const int kernel = select_kernel(d);
  WsLayout w;
  st = layout_for(d, kernel, &w);
  if (st != MT_OK) return st;
  if (ws_bytes < w.total) return MT_ERR_INVALID_ARG;

  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  PrepParams pp{};
  pp.B = d->batch; pp.T = d->tree_size; pp.Hq = d->num_q_heads; pp.Hkv = d->num_kv_heads;
  pp.D = d->head_dim;
  pp.P = d->page_size; pp.max_blocks = d->max_blocks_per_seq; pp.num_pages = d->num_pages;
  pp.max_pos = rope->max_pos;
  pp.q = q; pp.q_rot = ws + w.qrot;
  pp.k_new = k_new; pp.v_new = v_new; pp.k_cache = k_cache; pp.v_cache = v_cache;
  pp.block_tables = block_tables; pp.seq_lens = seq_lens;
  pp.tree_parents = tree_parents; pp.tree_depths = tree_depths;
  pp.rope = rope->table; pp.status = status;
  pp.cache_fp8 = fp8_cache(d); pp.k_scale = d->k_scale; pp.v_scale = d->v_scale;
  pp.anc = reinterpret_cast<unsigned long long*>(ws + w.anc);
  pp.tile_pfx = reinterpret_cast<int*>(ws + w.pfx);
  Sched sched{};
  sched.B = d->batch; sched.T = d->tree_size; sched.Hkv = d->num_kv_heads;
  sched.nrg = w.nrg; sched.G = w.G; sched.splits = d->num_splits;
  // fixed work of a piece in tile units: the tensor-core kernel streams a
  // tile in about 1 us and spends a few us on a piece's queries, epilogue
  // and pipeline refill, more with two M tiles (measured best: 5 with two,
  // 4 with one); the SIMT kernel's tiles are far slower
  sched.seg_cost = kernel == MT_KERNEL_SIMT ? 1 : (w.rows_per_group > 128 && w.rows > 128 ? 5 : 4);
  sched.tile_pfx = pp.tile_pfx;
  pp.sched = sched;
  pp.piece_table = kernel == MT_KERNEL_SIMT ? nullptr : reinterpret_cast<int*>(ws + w.pieces);
  st = cuda_status(launch_prep(pp, d->dtype, stream));
  if (st != MT_OK) return st;

  AttnParams ap{};
  ap.B = d->batch; ap.T = d->tree_size; ap.Hq = d->num_q_heads; ap.Hkv = d->num_kv_heads;
  ap.D = d->head_dim; ap.P = d->page_size; ap.max_blocks = d->max_blocks_per_seq;
  ap.num_pages = d->num_pages; ap.g = d->num_q_heads / d->num_kv_heads;
  ap.rows = w.rows; ap.rows_per_group = w.rows_per_group; ap.part_rows = w.part_rows;
  const float scale = d->sm_scale > 0.f ? d->sm_scale : (float)(1.0 / std::sqrt((double)d->head_dim));
  ap.scale_log2 = scale * 1.4426950408889634f;
  ap.q_rot = ws + w.qrot; ap.k_cache = k_cache; ap.v_cache = v_cache;
  ap.block_tables = block_tables; ap.seq_lens = seq_lens; ap.tree_depths = tree_depths;
  ap.out = out; ap.status = status;
  ap.anc = pp.anc;
  ap.part_o = ws + w.o;
  ap.part_ml = reinterpret_cast<float2*>(ws + w.ml);
  ap.sched = sched;
  ap.piece_table = pp.piece_table;
  ap.wait_limit_ns = g_wait_limit_ns ? g_wait_limit_ns : 2000000000ull;
  ap.test_stall = g_wait_stall;
  bool prof = g_prof_n < g_prof_cap;
  if (kernel == MT_KERNEL_SIMT) {
    if (prof) cudaEventRecord(g_prof_ev[2 * g_prof_n], stream);
    st = cuda_status(launch_attn_simt(ap, Fp8Cache{fp8_cache(d), d->k_scale, d->v_scale}, d->dtype, stream));
  } else {
    alignas(64) unsigned char tmap_k[128], tmap_v[128], tmap_q[128];
    const bool f8 = fp8_cache(d);
    cudaError_t ek, ev;
    if (f8) {
      ek = make_cache_tmap_e4m3(tmap_k, k_cache, d->num_pages, d->num_kv_heads, d->page_size, d->head_dim);
      ev = make_cache_tmap_e4m3(tmap_v, v_cache, d->num_pages, d->num_kv_heads, d->page_size, d->head_dim);
    } else {
      ek = make_cache_tmap(tmap_k, k_cache, d->dtype, d->num_pages, d->num_kv_heads, d->page_size, d->head_dim);
      ev = make_cache_tmap(tmap_v, v_cache, d->dtype, d->num_pages, d->num_kv_heads, d->page_size, d->head_dim);
    }
    // an FP8 cache: the K scale joins the softmax scale, the V scale the output
    AttnParams apt = ap;
    apt.cache_fp8 = f8 ? 1 : 0;
    apt.v_scale = f8 ? d->v_scale : 1.f;
    if (f8) apt.scale_log2 = (float)((double)ap.scale_log2 * (double)d->k_scale);
    if (ek != cudaSuccess || ev != cudaSuccess ||
        make_q_tmap(tmap_q, ws + w.qrot, d->dtype, d->batch * d->tree_size, d->num_q_heads, ap.g,
                    d->head_dim) != cudaSuccess) {
      st = MT_ERR_CUDA;
      prof = false;
    } else {
      // the start event goes in after the descriptors are encoded, so that
      // host time spent on them stays out of the kernel's window
      if (prof) cudaEventRecord(g_prof_ev[2 * g_prof_n], stream);
      st = cuda_status(launch_attn_tc(apt, d->dtype, tmap_k, tmap_v, tmap_q, stream));
    }
  }
  if (prof) cudaEventRecord(g_prof_ev[2 * g_prof_n++ + 1], stream);
  if (st != MT_OK) return st;
  return cuda_status(launch_combine(ap, d->dtype, stream));
}

// Acceptance workspace: status word, arrival counters [B], then (typical
// acceptance) each row's argmax [B*T] int32 and statistics [B*T] float4, then
// (rows split over several CTAs) each row's key [B*T] uint64 and slice
// counter [B*T] uint32.
struct AcceptWs {
  size_t counters, argmax, stats, row_keys, row_counters, split_stats, total;
};

AcceptWs accept_ws(int batch, int tree_size) {
  AcceptWs w;
  const size_t rows = (size_t)batch * tree_size;
  w.counters = kAlign;
  w.argmax = align_up(w.counters + sizeof(unsigned) * (size_t)batch);
  w.stats = align_up(w.argmax + sizeof(int) * rows);
  w.row_keys = align_up(w.stats + sizeof(float4) * rows);
  w.row_counters = align_up(w.row_keys + sizeof(unsigned long long) * rows);
  w.split_stats = align_up(w.row_counters + sizeof(unsigned) * rows);
  const size_t split_rows = rows < (size_t)kTypSplitRows ? rows : (size_t)kTypSplitRows;
  w.total = align_up(w.split_stats + sizeof(float4) * split_rows * kTypMaxSplits);
  return w;
}

// The split-row scratch of an acceptance workspace.
void set_row_scratch(AcceptParams& a, char* ws, int batch, int tree_size) {
  const AcceptWs w = accept_ws(batch, tree_size);
  a.row_keys = reinterpret_cast<unsigned long long*>(ws + w.row_keys);
  a.row_counters = reinterpret_cast<unsigned*>(ws + w.row_counters);
}

size_t mt_tree_accept_workspace_size(int batch, int tree_size) {
  if (batch < 1 || tree_size < 1) return 0;
  return accept_ws(batch, tree_size).total;
}

int mt_tree_accept_greedy(int batch, int tree_size, int vocab, int max_depth,
                          mt_dtype logits_dtype, const int32_t* tree_tokens,
                          const void* target_logits, const int32_t* tree_parents,
                          int32_t* argmax_out, int32_t* accept_len, int32_t* accept_path,
                          int32_t* next_token, void* workspace, size_t ws_bytes,
                          cudaStream_t stream) {
  const mt_call_range range("mt_tree_accept_greedy");
  if (batch < 1 || batch > (1 << 24) / kMaxTree) return MT_ERR_INVALID_ARG;
  if (tree_size < 1 || tree_size > kMaxTree) return MT_ERR_UNSUPPORTED;
  if (vocab < 1 || max_depth < 0 || max_depth >= kMaxTree) return MT_ERR_INVALID_ARG;
  if (logits_dtype != MT_F32 && logits_dtype != MT_F16 && logits_dtype != MT_BF16)
    return MT_ERR_UNSUPPORTED;
  if (!tree_tokens || !target_logits || !tree_parents || !argmax_out || !accept_len ||
      !accept_path || !next_token || !workspace)
    return MT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) % kAlign) ||
      ws_bytes < mt_tree_accept_workspace_size(batch, tree_size))
    return MT_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace);
  AcceptParams a{};
  a.B = batch; a.T = tree_size; a.V = vocab; a.max_depth = max_depth;
  a.tokens = tree_tokens; a.logits = target_logits; a.parents = tree_parents;
  a.argmax_out = argmax_out; a.accept_len = accept_len; a.accept_path = accept_path;
  a.next_token = next_token;
  a.status = reinterpret_cast<int*>(ws);
  set_row_scratch(a, ws, batch, tree_size);
  a.counters = reinterpret_cast<unsigned*>(ws + accept_ws(batch, tree_size).counters);
  return cuda_status(launch_accept(a, logits_dtype, stream));
}

int mt_tree_accept_typical(int batch, int tree_size, int vocab, int max_depth,
                           mt_dtype logits_dtype, const int32_t* tree_tokens,
                           const void* target_logits, const int32_t* tree_parents,
                           float temperature, float epsilon, float delta, int32_t* node_accept,
                           int32_t* accept_len, int32_t* accept_path, int32_t* next_token,
                           void* workspace, size_t ws_bytes, cudaStream_t stream) {
  const mt_call_range range("mt_tree_accept_typical");
  if (batch < 1 || batch > (1 << 24) / kMaxTree) return MT_ERR_INVALID_ARG;
  if (tree_size < 1 || tree_size > kMaxTree) return MT_ERR_UNSUPPORTED;
  if (vocab < 1 || max_depth < 0 || max_depth >= kMaxTree) return MT_ERR_INVALID_ARG;
  if (logits_dtype != MT_F32 && logits_dtype != MT_F16 && logits_dtype != MT_BF16)
    return MT_ERR_UNSUPPORTED;
  const float k = (float)(1.4426950408889634 / (double)temperature);
  if (!(temperature > 0.f) || !std::isfinite(temperature) || !std::isfinite(k) || !(epsilon > 0.f) ||
      !std::isfinite(epsilon) || !(delta > 0.f) || !std::isfinite(delta))
    return MT_ERR_INVALID_ARG;
  if (!tree_tokens || !target_logits || !tree_parents || !node_accept || !accept_len ||
      !accept_path || !next_token || !workspace)
    return MT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) % kAlign) ||
      ws_bytes < mt_tree_accept_workspace_size(batch, tree_size))
    return MT_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace);
  const AcceptWs w = accept_ws(batch, tree_size);
  AcceptParams a{};
  a.B = batch; a.T = tree_size; a.V = vocab; a.max_depth = max_depth;
  a.tokens = tree_tokens; a.logits = target_logits; a.parents = tree_parents;
  a.argmax_out = reinterpret_cast<int*>(ws + w.argmax);
  a.accept_len = accept_len; a.accept_path = accept_path; a.next_token = next_token;
  a.status = reinterpret_cast<int*>(ws);
  set_row_scratch(a, ws, batch, tree_size);
  a.counters = reinterpret_cast<unsigned*>(ws + w.counters);
  TypicalParams t{};
  t.k = k; t.epsilon = epsilon; t.delta = delta;
  t.stats = reinterpret_cast<float4*>(ws + w.stats);
  t.split_stats = reinterpret_cast<float4*>(ws + w.split_stats);
  t.node_accept = node_accept;
  return cuda_status(launch_accept_typical(a, t, logits_dtype, stream));
}

int mt_kv_commit(const mt_attn_desc* d, int max_depth, const int32_t* accept_path,
                 const int32_t* accept_len, void* k_cache, void* v_cache, int32_t* block_tables,
                 int32_t* seq_lens, int32_t* released_pages, void* status_ws,
                 cudaStream_t stream) {
  const mt_call_range range("mt_kv_commit");
  int st = check_desc(d);
  if (st != MT_OK) return st;
  if (max_depth < 0 || max_depth >= kMaxTree) return MT_ERR_INVALID_ARG;
  if (!accept_path || !accept_len || !k_cache || !v_cache || !block_tables || !seq_lens ||
      !released_pages || !status_ws)
    return MT_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(status_ws))
    return MT_ERR_INVALID_ARG;
  CommitParams c{};
  c.B = d->batch; c.T = d->tree_size; c.Hkv = d->num_kv_heads; c.D = d->head_dim;
  c.P = d->page_size; c.max_blocks = d->max_blocks_per_seq; c.num_pages = d->num_pages;
  c.max_depth = max_depth;
  c.rel_width = (d->tree_size + 2 * d->page_size - 2) / d->page_size;
  c.elem_bytes = cache_elem_bytes(d);
  c.accept_path = accept_path; c.accept_len = accept_len;
  c.k_cache = k_cache; c.v_cache = v_cache; c.block_tables = block_tables;
  c.seq_lens = seq_lens; c.released = released_pages;
  c.status = static_cast<int*>(status_ws);
  return cuda_status(launch_commit(c, stream));
}

int mt_tree_accept_commit(const mt_attn_desc* d, int vocab, int max_depth, mt_dtype logits_dtype,
                          const int32_t* tree_tokens, const void* target_logits,
                          const int32_t* tree_parents, int32_t* argmax_out, int32_t* accept_len,
                          int32_t* accept_path, int32_t* next_token, void* k_cache, void* v_cache,
                          int32_t* block_tables, int32_t* seq_lens, int32_t* released_pages,
                          void* workspace, size_t ws_bytes, cudaStream_t stream) {
  const mt_call_range range("mt_tree_accept_commit");
  int st = check_desc(d);
  if (st != MT_OK) return st;
  const int batch = d->batch, tree_size = d->tree_size;
  if (batch > (1 << 24) / kMaxTree) return MT_ERR_INVALID_ARG;
  if (vocab < 1 || max_depth < 0 || max_depth >= kMaxTree) return MT_ERR_INVALID_ARG;
  if (logits_dtype != MT_F32 && logits_dtype != MT_F16 && logits_dtype != MT_BF16)
    return MT_ERR_UNSUPPORTED;
  if (!tree_tokens || !target_logits || !tree_parents || !argmax_out || !accept_len ||
      !accept_path || !next_token || !k_cache || !v_cache || !block_tables || !seq_lens ||
      !released_pages || !workspace)
    return MT_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || (reinterpret_cast<uintptr_t>(workspace) % kAlign) ||
      ws_bytes < mt_tree_accept_workspace_size(batch, tree_size))
    return MT_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace);
  AcceptParams a{};
  a.B = batch; a.T = tree_size; a.V = vocab; a.max_depth = max_depth;
  a.tokens = tree_tokens; a.logits = target_logits; a.parents = tree_parents;
  a.argmax_out = argmax_out; a.accept_len = accept_len; a.accept_path = accept_path;
  a.next_token = next_token;
  a.status = reinterpret_cast<int*>(ws);
  set_row_scratch(a, ws, batch, tree_size);
  a.counters = reinterpret_cast<unsigned*>(ws + accept_ws(batch, tree_size).counters);
  CommitParams c{};
  c.B = batch; c.T = tree_size; c.Hkv = d->num_kv_heads; c.D = d->head_dim;
  c.P = d->page_size; c.max_blocks = d->max_blocks_per_seq; c.num_pages = d->num_pages;
  c.max_depth = max_depth;
  c.rel_width = (tree_size + 2 * d->page_size - 2) / d->page_size;
  c.elem_bytes = cache_elem_bytes(d);
  c.accept_path = accept_path; c.accept_len = accept_len;
  c.k_cache = k_cache; c.v_cache = v_cache; c.block_tables = block_tables;
  c.seq_lens = seq_lens; c.released = released_pages;
  c.status = a.status;
  return cuda_status(launch_accept_commit(a, c, logits_dtype, stream));
}

int mt_tree_candidates(int batch, int tree_size, int heads, int vocab, mt_dtype logits_dtype,
                       const void* root_logits, const void* head_logits,
                       const int32_t* tree_parents, int32_t* tree_tokens, void* status_ws,
                       cudaStream_t stream) {
  const mt_call_range range("mt_tree_candidates");
  if (batch < 1 || batch > kMaxBatch || heads < 1 || heads >= kMaxTree || vocab < 1)
    return MT_ERR_INVALID_ARG;
  if (tree_size < 1 || tree_size > kMaxTree) return MT_ERR_UNSUPPORTED;
  if (logits_dtype != MT_F32 && logits_dtype != MT_F16 && logits_dtype != MT_BF16)
    return MT_ERR_UNSUPPORTED;
  if (!root_logits || !head_logits || !tree_parents || !tree_tokens || !status_ws)
    return MT_ERR_INVALID_ARG;
  if (!aligned16(root_logits) || !aligned16(head_logits) || !aligned16(status_ws))
    return MT_ERR_INVALID_ARG;
  CandParams c{};
  c.B = batch; c.T = tree_size; c.V = vocab; c.heads = heads;
  c.root_logits = root_logits; c.head_logits = head_logits;
  c.parents = tree_parents; c.tokens = tree_tokens;
  c.status = static_cast<int*>(status_ws);
  return cuda_status(launch_cand(c, logits_dtype, stream));
}

int mt_profile_enable(int max_records) {
  if (max_records < 0 || max_records > (1 << 16)) return MT_ERR_INVALID_ARG;
  for (int i = 0; i < 2 * g_prof_cap; ++i) cudaEventDestroy(g_prof_ev[i]);
  delete[] g_prof_ev;
  g_prof_ev = nullptr;
  g_prof_cap = g_prof_n = 0;
  if (max_records == 0) return MT_OK;
  g_prof_ev = new cudaEvent_t[2 * (size_t)max_records];
  for (int i = 0; i < 2 * max_records; ++i) {
    if (cudaEventCreate(&g_prof_ev[i]) != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(g_prof_ev[j]);
      delete[] g_prof_ev;
      g_prof_ev = nullptr;
      return MT_ERR_CUDA;
    }
  }
  g_prof_cap = max_records;
  return MT_OK;
}

int mt_profile_read(float* ms, int max_records, int* n_out) {
  if (!ms || !n_out || max_records < 0) return MT_ERR_INVALID_ARG;
  int n = g_prof_n < max_records ? g_prof_n : max_records;
  for (int i = 0; i < n; ++i) {
    if (cudaEventSynchronize(g_prof_ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms[i], g_prof_ev[2 * i], g_prof_ev[2 * i + 1]) != cudaSuccess)
      return MT_ERR_CUDA;
  }
  *n_out = n;
  g_prof_n = 0;
  return MT_OK;
}

int mt_debug_set_wait(unsigned long long limit_ns, int stall) {
  if (stall != 0 && stall != 1) return MT_ERR_INVALID_ARG;
  g_wait_limit_ns = limit_ns;
  g_wait_stall = stall;
  return MT_OK;
}

int mt_read_status(void* workspace, cudaStream_t stream, int* device_status) {
  if (!workspace || !device_status) return MT_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MT_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MT_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(workspace, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return MT_ERR_CUDA;
  *device_status = v;
  return MT_OK;
}

}  // extern "C"
