// Tree preparation: validates every sequence's tree, builds the per-node
// ancestor bitmasks and the tile schedule, rotates the tree tokens' queries
// into the workspace, and writes their rotated keys and raw values into their
// scratch slots of the paged cache.
//
// The tree mask (vLLM issue 1171, void-main: the Medusa tree mask inside the
// cached-KV attention) is carried as one 64-bit word per node, the set of the
// node's ancestors and itself (equivalently anc[i] = anc[parent[i]] | (1 << i)),
// so node i sees tree key t exactly when bit t of anc[i] is set.  Keys are
// rotated at position L_b + depth[i] (TensorRT-LLM issue 1946, position
// offsets for Medusa tokens); keys land at logical slot L_b + i, queries in a
// [B][T][Hq][D] workspace array read by the attention kernels.
#include <cuda_fp8.h>

#include <atomic>

#include "kernels.cuh"

namespace mt {

namespace {

constexpr int kPrepThreads = 256;
constexpr int kMaxDevices = 64;

// 8 consecutive act-dtype elements as one aligned vector.
template <typename T> struct Vec8 {
  struct type { uint4 a, b; };  // fp32: 32 bytes
  static __device__ __forceinline__ type load(const T* p) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
    return type{q[0], q[1]};
  }
  static __device__ __forceinline__ void store(T* p, const type& v) {
    uint4* q = reinterpret_cast<uint4*>(p);
    q[0] = v.a;
    q[1] = v.b;
  }
};
template <> struct Vec8<__half> {
  using type = uint4;
  static __device__ __forceinline__ type load(const __half* p) { return *reinterpret_cast<const uint4*>(p); }
  static __device__ __forceinline__ void store(__half* p, const type& v) { *reinterpret_cast<uint4*>(p) = v; }
};
template <> struct Vec8<__nv_bfloat16> {
  using type = uint4;
  static __device__ __forceinline__ type load(const __nv_bfloat16* p) {
    return *reinterpret_cast<const uint4*>(p);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const type& v) {
    *reinterpret_cast<uint4*>(p) = v;
  }
};

// Eight act-dtype values into an FP8 cache: the E4M3 codes of value / scale
// (fp32 division, nearest-even, saturated to +-448), one 8-byte store.
template <typename T>
__device__ __forceinline__ void store_e4m3x8(uint8_t* p, const typename Vec8<T>::type& v, float scale) {
  T x[8];
  memcpy(x, &v, sizeof(x));
  uint8_t c[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) c[e] = __nv_cvt_float_to_fp8(Act<T>::to_f(x[e]) / scale, __NV_SATFINITE, __NV_E4M3);
  uint2 w;
  memcpy(&w, c, 8);
  *reinterpret_cast<uint2*>(p) = w;
}

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

// Sequences whose trees block 0 checks per round (their parents and depths
// staged in shared memory, every load of a round issued together).
constexpr int kSchedSeqs = 16;

// Ancestor masks of sequence b by one warp.  Lane l owns nodes l and l + 32;
// the sets come from pointer jumping in shared memory: start from {i} and the
// parent link, then six rounds of  anc[i] |= anc[up[i]], up[i] = up[up[i]]
// close them for any depth < 64.  An invalid tree or prefix length writes 0
// masks (the attention kernels skip such sequences).
__device__ void ancestor_masks(const PrepParams& a, int b, unsigned long long* s_anc, int* s_up) {
  const int lane = threadIdx.x & 31;
  const int* par = a.tree_parents + (size_t)b * a.T;
  const int* dep = a.tree_depths + (size_t)b * a.T;
  const int L = a.seq_lens[b];
  bool good = true;
  for (int i = lane; i < a.T; i += 32) {
    const int p = par[i];
    const bool ok_i = i == 0 ? (p == -1 && dep[0] == 0) : (p >= 0 && p < i && dep[i] == dep[p] + 1);
    good = good && ok_i;
    s_anc[i] = 1ull << i;
    s_up[i] = ok_i ? p : -1;
  }
  const bool ok = __all_sync(0xffffffffu, good);
  __syncwarp();
  for (int round = 0; round < 6; ++round) {
    unsigned long long na[2];
    int nu[2];
    for (int k = 0; k < 2; ++k) {
      const int i = lane + 32 * k;
      if (i < a.T) {
        const int u = s_up[i];
        na[k] = s_anc[i] | (u >= 0 ? s_anc[u] : 0ull);
        nu[k] = u >= 0 ? s_up[u] : -1;
      }
    }
    __syncwarp();
    for (int k = 0; k < 2; ++k) {
      const int i = lane + 32 * k;
      if (i < a.T) {
        s_anc[i] = na[k];
        s_up[i] = nu[k];
      }
    }
    __syncwarp();
  }
  const bool len_ok = L >= 0 && (long long)L + a.T <= (long long)a.max_blocks * a.P;
  for (int i = lane; i < a.T; i += 32)
    a.anc[(size_t)b * a.T + i] = (ok && len_ok) ? s_anc[i] : 0ull;  // 0 marks invalid
  __syncwarp();
}

// Where one query or key/value row of the rotation loop goes: index() finds
// the row's sequence and node, place() loads its prefix length and depth.
struct RowPlace {
  int b, i, L, depth;
  bool live, is_q;

  __device__ __forceinline__ void index(const PrepParams& a, long long grow, long long nq, long long nrows) {
    live = grow < nrows;
    if (!live) return;
    is_q = grow < nq;
    const long long row = is_q ? grow : grow - nq;
    const int H = is_q ? a.Hq : a.Hkv;
    if (row <= 0xffffffffLL && (long long)H * a.T <= 0xffffffffLL) {  // 32-bit division
      const unsigned r32 = (unsigned)row, h = (unsigned)H;
      i = (int)((r32 / h) % (unsigned)a.T);
      b = (int)(r32 / (h * (unsigned)a.T));
    } else {
      i = (int)((row / H) % a.T);
      b = (int)(row / ((long long)H * a.T));
    }
  }
  __device__ __forceinline__ void place(const PrepParams& a) {
    if (!live) return;
    L = a.seq_lens[b];
    depth = a.tree_depths[(size_t)b * a.T + i];
  }
};

// Rotates one row as lane k of its lane group (the pairs (j, j + D/2) for j in
// [8k, 8k + 8)) and stores it: a query into the workspace, a key (and its
// value, unrotated) into its slot of the cache.
template <typename T>
__device__ __forceinline__ void rotate_row(const PrepParams& a, const RowPlace& pl, long long grow, long long nq,
                                           int k, int half) {
  if (!pl.live) return;
  const bool is_q = pl.is_q;
  const long long row = is_q ? grow : grow - nq;
  const int b = pl.b, i = pl.i, L = pl.L, depth = pl.depth;
  const T* src = static_cast<const T*>(is_q ? a.q : a.k_new) + (size_t)row * a.D;
  const typename Vec8<T>::type lo = Vec8<T>::load(src + 8 * k);
  const typename Vec8<T>::type hi = Vec8<T>::load(src + half + 8 * k);
  typename Vec8<T>::type vlo, vhi;
  if (!is_q) {
    const T* vn = static_cast<const T*>(a.v_new) + (size_t)row * a.D;
    vlo = Vec8<T>::load(vn + 8 * k);
    vhi = Vec8<T>::load(vn + half + 8 * k);
  }
  const long long pos = (long long)L + depth;
  if (L < 0 || depth < 0 || pos >= a.max_pos) {
    if (k == 0) set_status(a.status, L < 0 ? kStPages : kStTree);
    return;
  }
  T* dst = nullptr;         // act-dtype destination of the rotated row
  uint8_t* dst8 = nullptr;  // FP8 cache destination of a rotated key
  if (is_q) {
    dst = static_cast<T*>(a.q_rot) + (size_t)row * a.D;
  } else {
    const int kvh = (int)(row % a.Hkv);
    const unsigned slot = (unsigned)L + (unsigned)i;  // L >= 0 and i < 64: no wrap
    const unsigned pg = slot / (unsigned)a.P;
    const int page = pg < (unsigned)a.max_blocks ? a.block_tables[(size_t)b * a.max_blocks + pg] : -1;
    if (page < 0 || page >= a.num_pages) {
      if (k == 0) set_status(a.status, kStPages);
      return;
    }
    const size_t off = (((size_t)page * a.Hkv + kvh) * a.P + slot % (unsigned)a.P) * a.D;
    if (a.cache_fp8) {
      // FP8 cache: the codes of the raw value and (below) of the rotated key
      dst8 = static_cast<uint8_t*>(a.k_cache) + off;
      uint8_t* vc8 = static_cast<uint8_t*>(a.v_cache) + off;
      store_e4m3x8<T>(vc8 + 8 * k, vlo, a.v_scale);
      store_e4m3x8<T>(vc8 + half + 8 * k, vhi, a.v_scale);
    } else {
      dst = static_cast<T*>(a.k_cache) + off;
      // raw value: this lane's two 8-element chunks
      T* vc = static_cast<T*>(a.v_cache) + off;
      Vec8<T>::store(vc + 8 * k, vlo);
      Vec8<T>::store(vc + half + 8 * k, vhi);
    }
  }
  const float4* cs = reinterpret_cast<const float4*>(a.rope + (size_t)pos * half + 8 * k);
  T xl[8], xh[8], ol[8], oh[8];
  memcpy(xl, &lo, sizeof(xl));
  memcpy(xh, &hi, sizeof(xh));
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const float4 c = cs[e / 2];  // (cos, sin) of pairs e and e + 1
    float l0, h0, l1, h1;
    rope_pair(Act<T>::to_f(xl[e]), Act<T>::to_f(xh[e]), c.x, c.y, l0, h0);
    rope_pair(Act<T>::to_f(xl[e + 1]), Act<T>::to_f(xh[e + 1]), c.z, c.w, l1, h1);
    ol[e] = Act<T>::from_f(l0);
    ol[e + 1] = Act<T>::from_f(l1);
    oh[e] = Act<T>::from_f(h0);
    oh[e + 1] = Act<T>::from_f(h1);
  }
  typename Vec8<T>::type wl, wh;
  memcpy(&wl, ol, sizeof(ol));
  memcpy(&wh, oh, sizeof(oh));
  if (dst8) {
    store_e4m3x8<T>(dst8 + 8 * k, wl, a.k_scale);
    store_e4m3x8<T>(dst8 + half + 8 * k, wh, a.k_scale);
  } else {
    Vec8<T>::store(dst + 8 * k, wl);
    Vec8<T>::store(dst + half + 8 * k, wh);
  }
}

// Whether every product and quotient of the piece walk fits in 32 bits: the
// balanced schedule's total cost X (split mode: its unit count) times G + 1,
// and split mode's tile counts times splits + 1.  total = tiles per segment,
// summed over the sequences.
__device__ __forceinline__ bool sched_fits_int(const Sched& s, int total) {
  const long long HR = (long long)s.Hkv * s.nrg;
  const long long lim = 1LL << 31;
  if (s.splits == 0) return ((long long)total * HR + (long long)s.seg_cost * s.B * HR) * (s.G + 1) < lim;
  return (long long)s.B * HR * s.splits * (s.G + 1) < lim && (long long)total * (s.splits + 1) < lim;
}

// Each CTA's piece list (one thread per CTA), with the index type I of the
// schedule arithmetic; a record is two 16-byte stores.
template <typename I>
__device__ void walk_pieces(const PrepParams& a, const Sched& sc, const int* s_len) {
  PieceRec* recs = reinterpret_cast<PieceRec*>(a.piece_table + piece_rec_offset(sc.G));
  for (int c = threadIdx.x; c < sc.G; c += blockDim.x) {
    PieceIterT<I> it;
    it.init(sc, c);
    Piece p;
    int n = 0;
    while (it.next(p)) {
      if (n == kMaxPieceRecs) {
        n = -1;
        break;
      }
      PieceRec r;
      r.b = p.b; r.kvh = p.kvh; r.rg = p.rg; r.seg = p.seg;
      r.tile_begin = p.tile_begin; r.tile_end = p.tile_end; r.slot = p.slot;
      r.L = s_len[p.b];
      recs[(size_t)c * kMaxPieceRecs + n] = r;
      ++n;
    }
    a.piece_table[c] = n;
  }
}

template <typename T>
__global__ void __launch_bounds__(kPrepThreads, sizeof(T) == 4 ? 3 : 4) prep_kernel(PrepParams a) {
  const int tid = threadIdx.x;
  pdl_wait();
  if (blockIdx.x == 0) {
    // ---- schedule block (block 0: dispatched first): tree and length
    // checks, tiles per segment, their prefix, and the CTAs' piece lists.
    // The same checks as ancestor_masks: a parent earlier than its child and
    // depth[i] = depth[parent[i]] + 1 (the root at depth 0 with parent -1).
    extern __shared__ int s_nt[];  // [B + 1] tiles per segment, then [B] prefix lengths
    int* s_len = s_nt + a.B + 1;
    __shared__ int s_warp[32];
    __shared__ int s_par[kSchedSeqs * kMaxTree], s_dep[kSchedSeqs * kMaxTree];
    __shared__ int s_ok[kSchedSeqs];
    constexpr int kPer = kSchedSeqs * kMaxTree / kPrepThreads;
    for (int b0 = 0; b0 < a.B; b0 += kSchedSeqs) {
      const int nb = min(kSchedSeqs, a.B - b0);
      const int n = nb * a.T;
      const int* par = a.tree_parents + (size_t)b0 * a.T;
      const int* dep = a.tree_depths + (size_t)b0 * a.T;
      int pv[kPer], dv[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int e = tid + k * kPrepThreads;
        if (e < n) {
          pv[k] = par[e];
          dv[k] = dep[e];
        }
      }
      if (tid < nb) {
        s_len[b0 + tid] = a.seq_lens[b0 + tid];
        s_ok[tid] = 1;
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int e = tid + k * kPrepThreads;
        if (e < n) {
          s_par[e] = pv[k];
          s_dep[e] = dv[k];
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int e = tid + k * kPrepThreads;
        if (e < n) {
          const int sb = e / a.T, i = e % a.T;
          const int p = s_par[e];
          const bool ok_i = i == 0 ? (p == -1 && s_dep[e] == 0)
                                   : (p >= 0 && p < i && s_dep[e] == s_dep[sb * a.T + p] + 1);
          if (!ok_i) s_ok[sb] = 0;
        }
      }
      __syncthreads();
      if (tid < nb) {
        const int b = b0 + tid;
        const int L = s_len[b];
        const bool ok = s_ok[tid] != 0;
        const bool len_ok = L >= 0 && (long long)L + a.T <= (long long)a.max_blocks * a.P;
        if (!ok) set_status(a.status, kStTree);
        if (!len_ok) set_status(a.status, kStPages);
        s_nt[b] = (ok && len_ok) ? (L + a.T + kTileKeys - 1) / kTileKeys : 0;
      }
      __syncthreads();
    }
    int total = block_exclusive_scan(s_nt, a.B, s_warp);
    for (int b = tid; b < a.B; b += blockDim.x) a.tile_pfx[b] = s_nt[b];
    if (tid == 0) {
      a.tile_pfx[a.B] = total;
      s_nt[a.B] = total;
    }
    if (a.piece_table) {
      // each CTA's piece list, walked over the prefix in shared memory
      __syncthreads();
      Sched sc = a.sched;
      sc.tile_pfx = s_nt;
      if (sched_fits_int(sc, total)) walk_pieces<int>(a, sc, s_len);
      else walk_pieces<long long>(a, sc, s_len);
    }
    return;
  }
  // ---- ancestor masks: one warp per sequence, before its rotation rows ----
  const long long nwarps = (long long)(gridDim.x - 1) * (kPrepThreads / 32);
  const long long gwarp = (long long)(blockIdx.x - 1) * (kPrepThreads / 32) + (tid >> 5);
  {
    __shared__ unsigned long long s_anc[kPrepThreads / 32][kMaxTree];
    __shared__ int s_up[kPrepThreads / 32][kMaxTree];
    for (long long b = gwarp; b < a.B; b += nwarps) ancestor_masks(a, (int)b, s_anc[tid >> 5], s_up[tid >> 5]);
  }
  // ---- rotations: B*T*Hq query rows, then B*T*Hkv key/value rows ----
  // A row is handled by D/16 lanes; lane k rotates the pairs (j, j + D/2) for
  // j in [8k, 8k + 8) with 16-byte (8-element) loads and stores.  The prefix
  // length and depth that place a lane group's next row are loaded while the
  // current row is rotated, so each trip waits on one round of loads.
  const int lanes_per_row = a.D / 16;
  const int rows_per_warp = 32 / lanes_per_row;
  const int lane = tid & 31;
  const int sub = lane / lanes_per_row, k = lane % lanes_per_row;
  const long long nq = (long long)a.B * a.T * a.Hq;
  const long long nrows = nq + (long long)a.B * a.T * a.Hkv;
  const int half = a.D / 2;
  const long long stride = nwarps * rows_per_warp;
  long long row0 = gwarp * rows_per_warp + sub;
  RowPlace cur;
  cur.index(a, row0, nq, nrows);
  cur.place(a);
  for (; row0 < nrows; row0 += stride) {
    RowPlace nxt;
    nxt.index(a, row0 + stride, nq, nrows);
    nxt.place(a);
    rotate_row<T>(a, cur, row0, nq, k, half);
    cur = nxt;
  }
}

template <typename T>
cudaError_t launch_t(const PrepParams& a, cudaStream_t stream) {
  const long long nrows = (long long)a.B * a.T * ((long long)a.Hq + a.Hkv);
  const long long rows_per_block = (long long)(kPrepThreads / 32) * (32 / (a.D / 16));
  size_t smem = sizeof(int) * (size_t)(2 * a.B + 1);
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  // One resident wave: the rotation loop strides over the grid, so blocks
  // beyond what the SMs hold at once would only form a second, short wave.
  // The number resident per SM is looked up once per device.
  static std::atomic<int> resident[kMaxDevices];
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  int per_sm = dev >= 0 && dev < kMaxDevices ? resident[dev].load(std::memory_order_relaxed) : 0;
  if (per_sm <= 0) {
    // without the dynamic part (block 0's per-sequence arrays, a few KB up to
    // batches in the thousands): a batch so large that it lowers residency
    // only gets a short extra wave, which is correct, as no block waits for
    // another
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prep_kernel<T>, kPrepThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    if (dev >= 0 && dev < kMaxDevices) resident[dev].store(per_sm, std::memory_order_relaxed);
  }
  long long blocks = (nrows + rows_per_block - 1) / rows_per_block + 1;  // + block 0 (the schedule)
  const long long wave = (long long)per_sm * sms;
  if (blocks > wave) blocks = wave;
  if (blocks < 2) blocks = 2;
  return launch_pdl(prep_kernel<T>, dim3((unsigned)blocks), dim3(kPrepThreads), smem, stream, a);
}

}  // namespace

cudaError_t launch_prep(const PrepParams& a, int dtype, cudaStream_t stream) {
  switch (dtype) {
    case 0: return launch_t<float>(a, stream);
    case 1: return launch_t<__half>(a, stream);
    default: return launch_t<__nv_bfloat16>(a, stream);
  }
}

}  // namespace mt
