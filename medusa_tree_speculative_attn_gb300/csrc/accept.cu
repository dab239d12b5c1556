// Greedy acceptance (LM head at temperature 0; lmdeploy PR 1231 "[WIP] support
// Medusa" -- the `evaluate_posterior` step -- and vLLM issue 1171, "it uses
// the argmax result"), optionally fused with the KV commit.
//
// One launch: a CTA per node takes the argmax over the vocab of its logits row
// (values compared exactly; +0 and -0 are equal; a larger value wins, the
// lower index among equal values), publishes it and counts itself in its
// sequence's arrival counter.  The CTA that completes a sequence resets the
// counter and selects the path with one warp:
//   acc[0] = 1, acc[i] = acc[parent[i]] && token[i] == argmax[parent[i]],
//   end = the deepest accepted node (lowest index among equals),
// writes accept_len, the padded root-to-end path and next_token, and, in the
// fused form, commits the sequence's K/V (commit_seq.cuh) right away.
//
// Typical acceptance (the scheme named beside tree attention in the opening
// comment of vLLM issue 1171; the rule of the Medusa paper) has the same shape:
// each row's CTA streams its logits once for the argmax and the tempered distribution's statistics, and
// node i > 0 passes when its token's probability under its parent's row is
// above min(epsilon, delta * exp(-entropy)).
#include <atomic>

#include "commit_seq.cuh"

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

__device__ __forceinline__ void warp_best(float& best, int& bidx) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, off);
    const int oi = __shfl_xor_sync(0xffffffffu, bidx, off);
    if (better(ov, oi, best, bidx)) { best = ov; bidx = oi; }
  }
}

// Counts one arrival at a counter in global memory and returns the count
// before it.  The read-modify-write is acquire-release at GPU scope: the
// caller's earlier writes (and atomics) become visible to whichever thread
// later acquires through this counter, and the caller sees everything the
// earlier arrivals released.  A CTA that finds itself last passes that view
// on to its other threads through a block barrier.
__device__ __forceinline__ unsigned count_arrival(unsigned* counter) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
  return old;
}

// Shared state of a sequence's path selection (one warp) and commit.
struct FinishSmem {
  unsigned long long anc[kMaxTree];
  int up[kMaxTree], dep[kMaxTree], am[kMaxTree];
  int par[kMaxTree], tok[kMaxTree];  // the sequence's tree and tokens
  int path[kMaxTree];
  int len;      // accepted length
  int seq_len;  // seq_lens[b] before the commit
  int last;
  CommitSmem commit;
};

// The sequence's parents, tokens and (for the commit) length, loaded by every
// row's CTA at its start so that their latency hides behind the row's logits;
// only the CTA that completes the sequence uses them.
struct SeqPrefetch {
  int par, tok, len;
  __device__ __forceinline__ void load(const AcceptParams& a, const CommitParams& c, int b, bool commit) {
    const int t = threadIdx.x;
    par = t < a.T ? a.parents[(size_t)b * a.T + t] : 0;
    tok = t < a.T ? a.tokens[(size_t)b * a.T + t] : 0;
    len = commit && t == 0 ? c.seq_lens[b] : 0;
  }
  __device__ __forceinline__ void store(const AcceptParams& a, FinishSmem& sm) const {
    const int t = threadIdx.x;
    if (t < a.T) {
      sm.par[t] = par;
      sm.tok[t] = tok;
    }
    if (t == 0) sm.seq_len = len;
  }
};

struct GreedyTest {
  __device__ __forceinline__ bool operator()(const FinishSmem& sm, int i, int p) const {
    return sm.tok[i] != sm.am[p];
  }
};

// Greedy path of sequence b by one warp, every step in parallel over the nodes
// (lane l owns nodes l and l + 32):
//   ancestors and depths by pointer jumping (six rounds close any depth < 64);
//   node i matches when tokens[i] == argmax[parent[i]] (the root always);
//   node i is accepted when every node on its root path matches;
//   end = the accepted node of largest depth, the lowest index among equals.
// The argmax values were written by other CTAs: read through L2.  Parents and
// tokens come from shared memory (SeqPrefetch).  fails(sm, i, p) says whether
// node i > 0 with the valid parent p fails its own test (greedy: tokens[i] !=
// argmax[p]).
template <class Fails = GreedyTest>
__device__ void select_path(const AcceptParams& a, int b, FinishSmem& sm, Fails fails = Fails()) {
  const int lane = threadIdx.x & 31;
  const int T = a.T;
  const int* par = sm.par;
  const int* am = a.argmax_out + (size_t)b * T;
  bool good = true;
  for (int i = lane; i < T; i += 32) {
    const int p = par[i];
    const bool ok_i = i == 0 ? p == -1 : (p >= 0 && p < i);
    good = good && ok_i;
    sm.anc[i] = 1ull << i;
    sm.up[i] = (i > 0 && ok_i) ? p : -1;
    sm.dep[i] = (i > 0 && ok_i) ? 1 : 0;
    sm.am[i] = __ldcg(am + i);
  }
  const bool ok = __all_sync(0xffffffffu, good);
  __syncwarp();
  for (int round = 0; round < 6; ++round) {
    unsigned long long na[2];
    int nu[2], nd[2];
    for (int k = 0; k < 2; ++k) {
      const int i = lane + 32 * k;
      if (i < T) {
        const int u = sm.up[i];
        na[k] = sm.anc[i] | (u >= 0 ? sm.anc[u] : 0ull);
        nd[k] = sm.dep[i] + (u >= 0 ? sm.dep[u] : 0);
        nu[k] = u >= 0 ? sm.up[u] : -1;
      }
    }
    __syncwarp();
    for (int k = 0; k < 2; ++k) {
      const int i = lane + 32 * k;
      if (i < T) {
        sm.anc[i] = na[k];
        sm.dep[i] = nd[k];
        sm.up[i] = nu[k];
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
      mis0 = !(p >= 0 && p < i0) || fails(sm, i0, p);
    }
    if (i1 < T) {
      const int p = par[i1];
      mis1 = !(p >= 0 && p < i1) || fails(sm, i1, p);
    }
  }
  const unsigned long long mis = (unsigned long long)__ballot_sync(0xffffffffu, mis0) |
                                 ((unsigned long long)__ballot_sync(0xffffffffu, mis1) << 32);
  bool deep_ok = true;
  int key = -1;  // (depth, -index) of the best accepted node owned by this lane
  for (int k = 0; k < 2; ++k) {
    const int i = lane + 32 * k;
    if (i < T) {
      const int d = sm.dep[i];
      deep_ok = deep_ok && d <= a.max_depth;
      if ((sm.anc[i] & mis) == 0ull) key = max(key, (d << 8) | (255 - i));
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
      a.next_token[b] = sm.am[0];
      sm.len = 0;
      sm.path[0] = 0;
    }
    for (int d = lane; d <= a.max_depth; d += 32) path[d] = d == 0 ? 0 : -1;
    __syncwarp();
    return;
  }
  const int end = 255 - (key & 255);
  const unsigned long long on_path = sm.anc[end];
  const int len = sm.dep[end];
  for (int d = lane; d <= a.max_depth; d += 32)
    if (d > len) path[d] = -1;
  for (int k = 0; k < 2; ++k) {
    const int i = lane + 32 * k;
    if (i < T && ((on_path >> i) & 1ull)) {
      path[sm.dep[i]] = i;
      sm.path[sm.dep[i]] = i;
    }
  }
  if (lane == 0) {
    a.accept_len[b] = len;
    a.next_token[b] = sm.am[end];
    sm.len = len;
  }
  __syncwarp();
}

// Called by every thread of a row's CTA once thread 0 holds the row's argmax
// ix and the prefetched sequence data is in shared memory (after a block
// synchronisation): publish the argmax; the CTA that completes its sequence
// selects the path and, when kCommit, commits the sequence.  The block-table
// window for the commit is loaded before the arrival, so that its latency
// overlaps the arrival's.
template <bool kCommit>
__device__ void finish_row(const AcceptParams& a, const CommitParams& c, int row, int ix, FinishSmem& sm,
                           uint4* stage, int stage_vecs) {
  const int b = row / a.T;
  if (kCommit) commit_load_window(c, b, sm.seq_len, sm.commit);
  if (threadIdx.x == 0) {
    a.argmax_out[row] = ix;  // released by the arrival
    sm.last = count_arrival(&a.counters[b]) == (unsigned)(a.T - 1);
  }
  __syncthreads();  // the last CTA's threads see every row's argmax past this point
  if (!sm.last) return;
  if (threadIdx.x == 0) a.counters[b] = 0;  // left at zero for the next call
  if (threadIdx.x < 32) select_path(a, b, sm);
  if (kCommit) {
    __syncthreads();
    commit_sequence(c, b, sm.seq_len, sm.len, sm.path, sm.commit, stage, stage_vecs);
  }
}

// Per-node argmax for rows of 16-byte vectors, one CTA per row, or, when the
// rows are few, a.nsplit CTAs per row, each taking one contiguous slice of the
// row's vectors.  Each thread takes its slice's vectors tid, tid +
// kRowThreads, ... in increasing index order, kBatch of them per round with
// all their loads issued before any is used (streaming loads: the logits are
// read once), keeping (max, first index): a vector's packed maximum is
// compared first and the vector is searched only when it beats the running
// maximum.  Warps, then the block, merge the threads' results in the same
// order.  The slices of a split row meet in a 64-bit key (below); the last
// slice to arrive continues as the row's CTA.
constexpr int kRowThreads = 128;
constexpr int kBatch = 8;

// (value, index) as a key whose unsigned order is the argmax order: a larger
// value first, then a lower index; -0 counts as +0.  No NaN (precondition).
__device__ __forceinline__ unsigned long long argmax_key(float v, int ix) {
  if (v == 0.f) v = 0.f;
  const uint32_t bits = __float_as_uint(v);
  const uint32_t ord = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
  return ((unsigned long long)ord << 32) | (0xffffffffu - (uint32_t)ix);
}

template <typename T, bool kCommit>
__global__ void __launch_bounds__(kRowThreads, 8) argmax_rows_kernel(AcceptParams a, CommitParams c, int stage_vecs) {
  constexpr int EPV = 16 / sizeof(T);
  extern __shared__ uint4 stage[];  // the commit's row stage (kCommit)
  __shared__ float s_v[kRowThreads / 32];
  __shared__ int s_i[kRowThreads / 32];
  __shared__ FinishSmem sm;
  __shared__ int s_slice_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x / a.nsplit, slice = blockIdx.x % a.nsplit;
  pdl_wait();
  SeqPrefetch pf;
  pf.load(a, c, row / a.T, kCommit);
  const int nvec = a.V / EPV;
  const int per = (nvec + a.nsplit - 1) / a.nsplit;
  const int vbeg = slice * per, vend = min(nvec, vbeg + per);
  const uint4* lg = reinterpret_cast<const uint4*>(static_cast<const T*>(a.logits) + (size_t)row * a.V);
  float best = -INFINITY;
  int bidx = 0x7fffffff;
  for (int v0 = vbeg + tid; v0 < vend; v0 += kRowThreads * kBatch) {
    uint4 raw[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int v = v0 + j * kRowThreads;
      if (v < vend) raw[j] = __ldcs(lg + v);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int v = v0 + j * kRowThreads;
      if (v < vend) {
        const float m = Max8<T>::of(raw[j]);
        if (m > best || bidx == 0x7fffffff) {
          T tmp[EPV];
          memcpy(tmp, &raw[j], 16);
#pragma unroll
          for (int e = EPV - 1; e >= 0; --e)
            if (Act<T>::to_f(tmp[e]) == m) bidx = v * EPV + e;
          best = m;
        }
      }
    }
  }
  warp_best(best, bidx);
  if (lane == 0) {
    s_v[warp] = best;
    s_i[warp] = bidx;
  }
  pf.store(a, sm);
  __syncthreads();
  float v = lane < kRowThreads / 32 ? s_v[lane] : -INFINITY;
  int ix = lane < kRowThreads / 32 ? s_i[lane] : 0x7fffffff;
  warp_best(v, ix);  // every warp merges; thread 0's result is used
  if (a.nsplit > 1) {
    // fold this slice into the row's key and count it; the row's last slice
    // takes the key (leaving it and the counter at zero) and goes on
    if (tid == 0) {
      atomicMax(&a.row_keys[row], argmax_key(v, ix));  // released by the arrival
      const bool last = count_arrival(&a.row_counters[row]) == (unsigned)(a.nsplit - 1);
      if (last) {
        // every slice's key update is ordered before this exchange
        ix = (int)(0xffffffffu - (uint32_t)atomicExch(&a.row_keys[row], 0ull));
        a.row_counters[row] = 0;
      }
      s_slice_last = last;
    }
    __syncthreads();
    if (!s_slice_last) return;
  }
  finish_row<kCommit>(a, c, row, ix, sm, stage, stage_vecs);
}

// Rows that are not 16-byte aligned: one CTA per row, scalar loads.
template <typename T, bool kCommit>
__global__ void __launch_bounds__(kThreads) argmax_scalar_kernel(AcceptParams a, CommitParams c, int stage_vecs) {
  extern __shared__ uint4 stage[];  // the commit's row stage (kCommit)
  __shared__ float s_v[kThreads / 32];
  __shared__ int s_i[kThreads / 32];
  __shared__ FinishSmem sm;
  const int row = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_wait();
  SeqPrefetch pf;
  pf.load(a, c, row / a.T, kCommit);
  const T* lg = static_cast<const T*>(a.logits) + (size_t)row * a.V;
  float best = -INFINITY;
  int bidx = 0x7fffffff;
  for (int v = threadIdx.x; v < a.V; v += kThreads) {
    const float x = Act<T>::to_f(lg[v]);
    if (better(x, v, best, bidx)) { best = x; bidx = v; }
  }
  warp_best(best, bidx);
  if (lane == 0) { s_v[warp] = best; s_i[warp] = bidx; }
  pf.store(a, sm);
  __syncthreads();
  float v = lane < kThreads / 32 ? s_v[lane] : -INFINITY;
  int ix = lane < kThreads / 32 ? s_i[lane] : 0x7fffffff;
  warp_best(v, ix);
  finish_row<kCommit>(a, c, row, ix, sm, stage, stage_vecs);
}

// ---- typical acceptance ----------------------------------------------------
//
// Per row, in base-2 units y = logit * k with k = log2(e) / temperature:
//   m = max y,  Z = sum 2^(y - m),  S = sum 2^(y - m) (y - m),
// so that the tempered distribution is q_v = 2^(y_v - m) / Z and its entropy
// in bits is H = log2 Z - S / Z (H ln 2 in nats, and exp(-H ln 2) = 2^-H).
// Each thread keeps a running (m, Z, S), moved to a larger m by scaling
// (Z, S) -> (c Z, c (S + (m_old - m) Z)), c = 2^(m_old - m).
// 2^x on the MUFU pipe (results below 2^-126 flush to zero: such terms add
// nothing measurable to a row's Z and S).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct RowStats {
  float m = -INFINITY, z = 0.f, s = 0.f;
  __device__ __forceinline__ void rebase(float nm) {  // nm >= m
    if (z > 0.f) {
      const float d = m - nm;
      const float c = exp2f(d);
      s = c * (s + d * z);
      z *= c;
    }
    m = nm;
  }
  __device__ __forceinline__ void add(float y) {  // y <= m
    const float t = y - m;
    const float e = exp2f(t);
    z += e;
    s += e > 0.f ? e * t : 0.f;
  }
  __device__ __forceinline__ void merge(RowStats o) {
    const float nm = fmaxf(m, o.m);
    if (nm == -INFINITY) return;
    rebase(nm);
    o.rebase(nm);
    z += o.z;
    s += o.s;
  }
  __device__ __forceinline__ void warp_merge() {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      RowStats o;
      o.m = __shfl_xor_sync(0xffffffffu, m, off);
      o.z = __shfl_xor_sync(0xffffffffu, z, off);
      o.s = __shfl_xor_sync(0xffffffffu, s, off);
      merge(o);
    }
  }
};

// A node's test, read by the warp that selects the path (typ_ok, filled first).
struct TypicalTest {
  const int* ok;
  __device__ __forceinline__ bool operator()(const FinishSmem&, int i, int) const { return ok[i] == 0; }
};

// The typical row pass's end, for every thread of the row's CTA: thread 0
// holds the row's argmax ix and statistics st.  Publish both; the CTA that
// completes the sequence fills each node's test (one warp, two nodes a lane:
// the token's logit is read again from its parent's row), writes node_accept
// and selects the path.
template <typename T>
__device__ void finish_typical(const AcceptParams& a, const TypicalParams& t, int row, int ix, RowStats st,
                               FinishSmem& sm, int* typ_ok) {
  const int b = row / a.T;
  if (threadIdx.x == 0) {
    const float h = log2f(st.z) - st.s / st.z;  // entropy in bits
    const float thr = fminf(t.epsilon, t.delta * exp2f(-h));
    t.stats[row] = make_float4(st.m, st.z, thr, 0.f);
    a.argmax_out[row] = ix;  // both released by the arrival
    sm.last = count_arrival(&a.counters[b]) == (unsigned)(a.T - 1);
  }
  __syncthreads();  // the last CTA's threads see every row's results past this point
  if (!sm.last) return;
  if (threadIdx.x == 0) a.counters[b] = 0;
  if (threadIdx.x >= 32) return;
  const T* lg = static_cast<const T*>(a.logits);
  for (int i = threadIdx.x; i < a.T; i += 32) {
    int ok = 1;
    if (i > 0) {
      const int p = sm.par[i], tok = sm.tok[i];
      ok = 0;
      if (p >= 0 && p < i && tok >= 0 && tok < a.V) {
        const size_t prow = (size_t)b * a.T + p;
        const float4 ps = __ldcg(t.stats + prow);
        const float y = Act<T>::to_f(lg[prow * a.V + tok]) * t.k;
        ok = exp2f(y - ps.x) / ps.y > ps.z;
      }
    }
    typ_ok[i] = ok;
    t.node_accept[(size_t)b * a.T + i] = ok;
  }
  __syncwarp();
  select_path(a, b, sm, TypicalTest{typ_ok});
}

// Rows of 16-byte vectors (same loads as argmax_rows_kernel), or any row with
// kVec false (scalar loads).  Every element enters the statistics; the argmax
// keeps the raw values' order (the lowest index among equal maxima).
template <typename T, bool kVec>
__global__ void __launch_bounds__(kRowThreads, 8) typical_rows_kernel(AcceptParams a, TypicalParams t) {
  constexpr int EPV = kVec ? 16 / sizeof(T) : 1;
  __shared__ float s_v[kRowThreads / 32];
  __shared__ int s_i[kRowThreads / 32];
  __shared__ float s_m[kRowThreads / 32], s_z[kRowThreads / 32], s_s[kRowThreads / 32];
  __shared__ int typ_ok[kMaxTree];
  __shared__ FinishSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ int s_slice_last;
  const int row = blockIdx.x / a.nsplit, slice = blockIdx.x % a.nsplit;
  pdl_wait();
  SeqPrefetch pf;
  pf.load(a, CommitParams{}, row / a.T, false);
  const T* base = static_cast<const T*>(a.logits) + (size_t)row * a.V;
  float best = -INFINITY;
  int bidx = 0x7fffffff;
  RowStats st;
  const int nvec = a.V / EPV;
  const int per = (nvec + a.nsplit - 1) / a.nsplit;
  const int vbeg = min(nvec, slice * per), vend = min(nvec, vbeg + per);
  for (int v0 = vbeg + tid; v0 < vend; v0 += kRowThreads * kBatch) {
    // all of the round's loads first (raw vectors, or scalars already widened)
    uint4 raw[kVec ? kBatch : 1];
    float xs[kVec ? 1 : kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int v = v0 + j * kRowThreads;
      if (v < vend) {
        if constexpr (kVec) raw[j] = __ldcs(reinterpret_cast<const uint4*>(base) + v);
        else xs[j] = Act<T>::to_f(base[v]);
      }
    }
    if constexpr (kVec) {
      // pass 1, per vector: its packed maximum decides the argmax (searched
      // only when it beats the running one, as in the greedy kernel) and the
      // round's largest y (k > 0, so max of x * k is k * max of x, exactly)
      float bm = -INFINITY;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int v = v0 + j * kRowThreads;
        if (v < vend) {
          const float m8 = Max8<T>::of(raw[j]);
          if (m8 > best || bidx == 0x7fffffff) {
            T tmp[EPV];
            memcpy(tmp, &raw[j], 16);
#pragma unroll
            for (int e = EPV - 1; e >= 0; --e)
              if (Act<T>::to_f(tmp[e]) == m8) bidx = v * EPV + e;
            best = m8;
          }
          bm = fmaxf(bm, m8);
        }
      }
      // pass 2: the round's terms under the running maximum, d = y - m in one
      // rounding, two accumulator pairs (a term that underflows adds 0 to both)
      bm *= t.k;
      if (bm > st.m) st.rebase(bm);
      const float neg_m = -st.m;
      float z0 = 0.f, z1 = 0.f, s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int v = v0 + j * kRowThreads;
        if (v < vend) {
          T tmp[EPV];
          memcpy(tmp, &raw[j], 16);
#pragma unroll
          for (int e = 0; e < EPV; e += 2) {
            const float d0 = fmaf(Act<T>::to_f(tmp[e]), t.k, neg_m);
            const float d1 = fmaf(Act<T>::to_f(tmp[e + 1]), t.k, neg_m);
            const float e0 = fast_exp2(d0), e1 = fast_exp2(d1);
            z0 += e0;
            z1 += e1;
            s0 = fmaf(e0, d0, s0);
            s1 = fmaf(e1, d1, s1);
          }
        }
      }
      st.z += z0 + z1;
      st.s += s0 + s1;
    } else {
      // pass 1: argmax and the round's largest y
      float bm = -INFINITY;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int v = v0 + j * kRowThreads;
        if (v < vend) {
          if (xs[j] > best || bidx == 0x7fffffff) {  // indices rise within a thread: the first maximum stays
            best = xs[j];
            bidx = v;
          }
          bm = fmaxf(bm, xs[j] * t.k);
        }
      }
      // pass 2: the round's terms, under the running maximum
      if (bm > st.m) st.rebase(bm);
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int v = v0 + j * kRowThreads;
        if (v < vend) st.add(xs[j] * t.k);
      }
    }
  }
  warp_best(best, bidx);
  st.warp_merge();
  if (lane == 0) {
    s_v[warp] = best;
    s_i[warp] = bidx;
    s_m[warp] = st.m;
    s_z[warp] = st.z;
    s_s[warp] = st.s;
  }
  pf.store(a, sm);
  __syncthreads();
  float v = lane < kRowThreads / 32 ? s_v[lane] : -INFINITY;
  int ix = lane < kRowThreads / 32 ? s_i[lane] : 0x7fffffff;
  RowStats all;
  if (lane < kRowThreads / 32) {
    all.m = s_m[lane];
    all.z = s_z[lane];
    all.s = s_s[lane];
  }
  warp_best(v, ix);  // every warp merges; thread 0's results are used
  all.warp_merge();
  if (a.nsplit > 1) {
    // fold this slice into the row: the argmax through the row's key, the
    // statistics through the slice's workspace entry; the row's last slice
    // merges the entries in slice order (leaving key and counter at zero) and
    // goes on as the row's CTA
    if (tid == 0) {
      atomicMax(&a.row_keys[row], argmax_key(v, ix));
      t.split_stats[(size_t)row * a.nsplit + slice] = make_float4(all.m, all.z, all.s, 0.f);
      // the key update and the entry are released by the arrival
      const bool last = count_arrival(&a.row_counters[row]) == (unsigned)(a.nsplit - 1);
      if (last) {
        // every slice's key update and entry are ordered before what follows
        ix = (int)(0xffffffffu - (uint32_t)atomicExch(&a.row_keys[row], 0ull));
        a.row_counters[row] = 0;
        RowStats acc;
        for (int q = 0; q < a.nsplit; ++q) {
          const float4 o = __ldcg(t.split_stats + (size_t)row * a.nsplit + q);
          RowStats ro;
          ro.m = o.x;
          ro.z = o.y;
          ro.s = o.z;
          acc.merge(ro);
        }
        all = acc;
      }
      s_slice_last = last;
    }
    __syncthreads();
    if (!s_slice_last) return;
  }
  finish_typical<T>(a, t, row, ix, all, sm, typ_ok);
}

inline int row_splits(int nrows, int nvec);

template <typename T>
cudaError_t launch_typical_t(const AcceptParams& a, const TypicalParams& t, cudaStream_t stream) {
  const int nrows = a.B * a.T;
  AcceptParams p = a;
  p.nsplit = 1;
  if (((long long)a.V * sizeof(T)) % 16 != 0 || (reinterpret_cast<uintptr_t>(a.logits) & 15) != 0)
    return launch_pdl(typical_rows_kernel<T, false>, dim3(nrows), dim3(kRowThreads), 0, stream, p, t);
  // split rows as the greedy kernel does, within the workspace's split entries
  if (nrows <= kTypSplitRows) {
    const int ns = row_splits(nrows, (int)(a.V / (16 / sizeof(T))));
    p.nsplit = ns < kTypMaxSplits ? ns : kTypMaxSplits;
  }
  return launch_pdl(typical_rows_kernel<T, true>, dim3((unsigned)((long long)nrows * p.nsplit)), dim3(kRowThreads),
                    0, stream, p, t);
}

// The fused kernel's commit stage: every row's CTA carries it, so it stays
// small enough for 7 CTAs per SM (the serving trees' five path entries of 8
// bf16 heads of 128 fit in one pass).  A grid that fits 5 CTAs per SM in one
// wave takes a stage twice that size, so that a sequence with more heads (32
// heads of 128: 80 KB) moves in two passes instead of four.
constexpr int kStageCap = 20 * 1024;
constexpr int kStageCapWide = 40 * 1024;
constexpr int kWideCtasPerSm = 5;

// CTAs per row for the vector kernel: one, unless the rows are fewer than
// about four CTAs per SM; then enough slices to reach that, each of at least
// 256 vectors (two rounds of loads per thread).
inline int sm_count() {
  static std::atomic<int> sms_cached{0};
  int sms = sms_cached.load(std::memory_order_relaxed);
  if (sms <= 0) {
    int dev = 0;
    sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    sms_cached.store(sms, std::memory_order_relaxed);
  }
  return sms;
}

inline int row_splits(int nrows, int nvec) {
  const int sms = sm_count();
  const long long target = 4LL * sms;
  if (nrows >= target) return 1;
  const int want = (int)((target + nrows - 1) / nrows);
  const int most = nvec / 256;
  return most < 2 ? 1 : (want < most ? want : most);
}

// The commit's stage (16-byte entries) for a grid of nblocks CTAs.
template <bool kCommit>
int stage_vecs_for(const CommitParams& c, long long nblocks) {
  if (!kCommit) return 0;
  return commit_stage_vecs(c, nblocks <= (long long)kWideCtasPerSm * sm_count() ? kStageCapWide : kStageCap);
}

template <typename T, bool kCommit>
cudaError_t launch_t(const AcceptParams& a, const CommitParams& c, cudaStream_t stream) {
  const int nrows = a.B * a.T;
  AcceptParams p = a;
  p.nsplit = 1;
  if (((long long)a.V * sizeof(T)) % 16 != 0 || (reinterpret_cast<uintptr_t>(a.logits) & 15) != 0) {
    const int sv = stage_vecs_for<kCommit>(c, nrows);
    return launch_pdl(argmax_scalar_kernel<T, kCommit>, dim3(nrows), dim3(kThreads), (size_t)sv * 16, stream, p,
                      c, sv);
  }
  p.nsplit = row_splits(nrows, (int)(a.V / (16 / sizeof(T))));
  const long long nblocks = (long long)nrows * p.nsplit;
  const int sv = stage_vecs_for<kCommit>(c, nblocks);
  return launch_pdl(argmax_rows_kernel<T, kCommit>, dim3((unsigned)nblocks), dim3(kRowThreads), (size_t)sv * 16,
                    stream, p, c, sv);
}

template <bool kCommit>
cudaError_t launch_dtype(const AcceptParams& a, const CommitParams& c, int dtype, cudaStream_t stream) {
  switch (dtype) {
    case 0: return launch_t<float, kCommit>(a, c, stream);
    case 1: return launch_t<__half, kCommit>(a, c, stream);
    default: return launch_t<__nv_bfloat16, kCommit>(a, c, stream);
  }
}

}  // namespace

cudaError_t launch_accept(const AcceptParams& a, int dtype, cudaStream_t stream) {
  return launch_dtype<false>(a, CommitParams{}, dtype, stream);
}

cudaError_t launch_accept_commit(const AcceptParams& a, const CommitParams& c, int dtype, cudaStream_t stream) {
  return launch_dtype<true>(a, c, dtype, stream);
}

cudaError_t launch_accept_typical(const AcceptParams& a, const TypicalParams& t, int dtype, cudaStream_t stream) {
  switch (dtype) {
    case 0: return launch_typical_t<float>(a, t, stream);
    case 1: return launch_typical_t<__half>(a, t, stream);
    default: return launch_typical_t<__nv_bfloat16>(a, t, stream);
  }
}

}  // namespace mt
