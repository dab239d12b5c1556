// Split-KV combine: merges the partial softmax results of the pieces of one
// segment (the Flash-Decoding style split that lmdeploy PR 1231 "[WIP] support
// Medusa" plans for its tree-mask kernel).  For piece k with running maximum
// m_k (base-2 units), sum l_k and output x_k = O_k / l_k (its own softmax
// average, stored in the act dtype):
//   M = max_k m_k,  w_k = 2^(m_k - M) l_k,  out = sum_k w_k x_k / sum_k w_k,
// evaluated in one pass with a running maximum (pieces that saw no key of a
// row, m_k = -inf, are skipped).
// Segments covered by a single piece were written directly and are skipped.
#include "kernels.cuh"

namespace mt {

namespace {

// One partial entry: 8 consecutive columns of one row in the act dtype, as
// loaded (one 16-byte word, two for fp32).
template <typename T>
struct Chunk8 {
  static constexpr int kWords = 8 * (int)sizeof(T) / 16;
  uint4 w[kWords];
  __device__ __forceinline__ void load(const T* p) {
#pragma unroll
    for (int k = 0; k < kWords; ++k) w[k] = reinterpret_cast<const uint4*>(p)[k];
  }
  __device__ __forceinline__ void to_f(float (&x)[8]) const {
    T v[8];
    memcpy(v, w, sizeof(v));
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = Act<T>::to_f(v[e]);
  }
};

// Fold one piece (max ml.x, sum ml.y, its output columns v) into the running
// result; a piece that saw no key of the row (ml.x = -inf) is skipped.
template <typename T, int PER>
__device__ __forceinline__ void merge(float& M, float& lsum, float (&acc)[PER][8], float2 ml,
                                      const Chunk8<T> (&v)[PER]) {
  if (ml.x == -INFINITY) return;
  const float m_new = fmaxf(M, ml.x);
  const float c_old = exp2f(M - m_new), c_new = exp2f(ml.x - m_new) * ml.y;
  lsum = lsum * c_old + c_new;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    float x[8];
    v[e].to_f(x);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[e][j] = acc[e][j] * c_old + x[j] * c_new;
  }
  M = m_new;
}

// Eight results times inv, rounded to the act dtype, as one 16-byte (16-bit
// types) or two (fp32) shared-memory writes.
template <typename T>
__device__ __forceinline__ void store8(T* p, const float (&x)[8], float inv) {
  T v[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) v[e] = Act<T>::from_f(x[e] * inv);
  uint4 w[8 * sizeof(T) / 16];
  memcpy(w, v, sizeof(v));
#pragma unroll
  for (int k = 0; k < (int)(8 * sizeof(T) / 16); ++k) reinterpret_cast<uint4*>(p)[k] = w[k];
}

constexpr int kWarps = 8;
constexpr int kPfxCached = 2048;  // tile prefixes copied to shared memory up to this batch

// What a block needs to merge one item (segment, 32-row block).
struct ItemInfo {
  int seg, row0, nt;
  int slot0, count;  // partial slots slot0 .. slot0 + count - 1; count 0: nothing to merge
  int all;           // every one of those slots holds a piece
};

// Persistent blocks over the items, the tile prefix copied to shared memory
// once.  One warp works out the next 32 items of the block at a time, a lane
// per item (which CTAs hold pieces of the segment: 64-bit schedule arithmetic
// in parallel instead of on every item's critical path), so that an item
// whose segment was written directly costs nothing.  For an item, thread
// (warp w, lane l) merges row l for the 8-column entries w, w + 8, ... (partial
// reads coalesced along rows), ROUND pieces per round with all their loads
// in flight; the block stages the merged rows in shared memory and writes them
// out in 16-byte chunks along each row.  BLOCKS blocks are resident per SM.
template <typename T, int D, int ROUND, int BLOCKS>
__global__ void __launch_bounds__(kWarps * 32, BLOCKS) combine_kernel(AttnParams a) {
  constexpr int C8 = D / 8;                    // 8-column partial entries per row
  constexpr int PER = C8 / kWarps;             // entries per thread
  constexpr int CH = D * (int)sizeof(T) / 16;  // 16-byte output chunks per row
  __shared__ int s_pfx[kPfxCached + 1];
  __shared__ ItemInfo s_info[32];
  __shared__ __align__(16) T s_out[32][D + 16 / (int)sizeof(T)];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  Sched s = a.sched;
  if (s.B <= kPfxCached) {
    for (int i = tid; i <= s.B; i += blockDim.x) s_pfx[i] = s.tile_pfx[i];
    __syncthreads();
    s.tile_pfx = s_pfx;
  }
  const int RG = a.rows_per_group;
  const int HR = s.Hkv * s.nrg;
  const int PR = a.part_rows;
  const int nrb = (PR + 31) / 32;
  const long long items = (long long)s.B * HR * nrb;
  const long long W = s.splits == 0 ? sched_total_cost(s) : 0;  // balanced mode works in cost units
  // does partial slot slot0 + k of segment seg (nt tiles) hold a piece?
  auto piece_exists = [&](const ItemInfo& in, int k) -> bool {
    if (in.all) return true;
    if (s.splits == 0) {
      // the segment's tiles are one contiguous stretch of the cost axis: its
      // first and last owners hold tiles of it, and a CTA in between covers its
      // whole cost range inside it, so it holds tiles exactly when that range
      // is not empty
      if (k == 0 || k == in.count - 1) return true;
      const int c = in.slot0 - in.seg + k;
      return W * (c + 1) / s.G > W * c / s.G;
    }
    // split mode: key chunk k is [nt k / n, nt (k + 1) / n), empty (and never
    // written) when the segment has fewer tiles than chunks
    return (long long)in.nt * k / s.splits < (long long)in.nt * (k + 1) / s.splits;
  };
  for (long long base = blockIdx.x; base < items; base += 32LL * gridDim.x) {
    __syncthreads();  // the previous batch's descriptions are no longer read
    if (warp == 0) {
      ItemInfo in{0, 0, 0, 0, 0, 1};
      const long long item = base + (long long)lane * gridDim.x;
      if (item < items) {
        in.seg = (int)(item / nrb);
        in.row0 = (int)(item % nrb) * 32;
        const int b = in.seg / HR, seg_in_b = in.seg % HR;
        in.nt = s.tile_pfx[b + 1] - s.tile_pfx[b];
        if (in.nt > 0 && s.splits == 0) {  // nt = 0: invalid sequence, nothing to merge
          const long long t0 = (long long)s.tile_pfx[b] * HR + (long long)seg_in_b * in.nt;
          const int c0 = sched_cta_of(sched_tile_cost(s, t0, in.seg), W, s.G);
          const int c1 = sched_cta_of(sched_tile_cost(s, t0 + in.nt - 1, in.seg), W, s.G);
          if (c0 != c1) {  // else written directly by its only CTA
            in.slot0 = in.seg + c0;
            in.count = c1 - c0 + 1;
            in.all = W >= s.G;  // every CTA's cost range is non-empty
          }
        } else if (in.nt > 0 && s.splits > 1) {
          in.slot0 = in.seg * s.splits;
          in.count = s.splits;
          in.all = in.nt >= s.splits;  // every key chunk is non-empty
        }
      }
      s_info[lane] = in;
    }
    __syncthreads();
    for (int i = 0; i < 32; ++i) {
      const ItemInfo in = s_info[i];
      if (in.count == 0) continue;  // block-uniform
      const int seg_in_b = in.seg % HR;
      const int b = in.seg / HR, kvh = seg_in_b / s.nrg, rg = seg_in_b % s.nrg;
      float M = -INFINITY, lsum = 0.f;
      float acc[PER][8];
#pragma unroll
      for (int e = 0; e < PER; ++e)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[e][j] = 0.f;
      const T* part = static_cast<const T*>(a.part_o);
      const int r = in.row0 + lane;
      const bool row_ok = r < PR && rg * RG + r < a.rows;
      if (row_ok && !in.all && s.splits == 0) {
        // a sparse schedule (fewer cost units than CTAs): most CTAs between the
        // segment's first and last owners hold nothing, so walk the segment's
        // tiles and take each distinct owner's partial slot once
        const long long t0 = (long long)s.tile_pfx[b] * HR + (long long)seg_in_b * in.nt;
        int prev = -1;
        for (int t = 0; t < in.nt; ++t) {
          const int cta = sched_cta_of(sched_tile_cost(s, t0 + t, in.seg), W, s.G);
          if (cta == prev) continue;
          prev = cta;
          const size_t slot = (size_t)in.seg + cta;
          Chunk8<T> v1[PER];
          const float2 ml1 = a.part_ml[slot * PR + r];
#pragma unroll
          for (int e = 0; e < PER; ++e) v1[e].load(part + ((slot * C8 + warp + kWarps * e) * PR + r) * 8);
          merge<T, PER>(M, lsum, acc, ml1, v1);
        }
      } else if (row_ok) {
        for (int k = 0; k < in.count; k += ROUND) {
          float2 ml[ROUND];
          Chunk8<T> v[ROUND][PER];
#pragma unroll
          for (int j = 0; j < ROUND; ++j) {
            ml[j] = make_float2(-INFINITY, 0.f);
            if (k + j < in.count && piece_exists(in, k + j)) {
              const size_t slot = (size_t)in.slot0 + k + j;
              ml[j] = a.part_ml[slot * PR + r];
#pragma unroll
              for (int e = 0; e < PER; ++e) v[j][e].load(part + ((slot * C8 + warp + kWarps * e) * PR + r) * 8);
            }
          }
#pragma unroll
          for (int j = 0; j < ROUND; ++j) merge<T, PER>(M, lsum, acc, ml[j], v[j]);
        }
      }
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
      for (int e = 0; e < PER; ++e) store8<T>(&s_out[lane][8 * (warp + kWarps * e)], acc[e], inv);
      __syncthreads();
      // 32 rows x CH chunks, consecutive threads along a row
      for (int idx = tid; idx < 32 * CH; idx += blockDim.x) {
        const int lr = idx / CH, ch = idx % CH;
        const int rr = in.row0 + lr;
        const int row = rg * RG + rr;
        if (rr >= PR || row >= a.rows) continue;
        const int node = row / a.g, h = kvh * a.g + row % a.g;
        T* dst = static_cast<T*>(a.out) + (((size_t)b * a.T + node) * a.Hq + h) * D;
        reinterpret_cast<uint4*>(dst)[ch] = *reinterpret_cast<const uint4*>(&s_out[lr][ch * (16 / sizeof(T))]);
      }
      __syncthreads();  // s_out is rewritten by the next item
    }
  }
}

template <typename T, int D, int ROUND, int BLOCKS>
cudaError_t launch_v(const AttnParams& a, int sms, cudaStream_t stream) {
  const long long items = (long long)a.B * a.Hkv * a.sched.nrg * ((a.part_rows + 31) / 32);
  const long long grid = items < (long long)BLOCKS * sms ? items : (long long)BLOCKS * sms;
  return launch_pdl(combine_kernel<T, D, ROUND, BLOCKS>, dim3((unsigned)(grid > 0 ? grid : 1)), dim3(kWarps * 32), 0,
                    stream, a);
}

// A balanced schedule with at least a quarter as many segments as CTAs cuts a
// segment into a few pieces (serving and 32k-token workloads: up to 3 and 4):
// two pieces per round, at 3 blocks per SM, keep more items in flight.  With
// no more items than SMs (batch 1: 64 items of about 5 pieces), every block
// has an SM to itself and takes 8 pieces per round.  Otherwise (key chunks,
// or many items of many pieces) 4 pieces per round at 2 blocks per SM.
template <typename T, int D>
cudaError_t launch_t(const AttnParams& a, cudaStream_t stream) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long nseg = (long long)a.B * a.Hkv * a.sched.nrg;
  const long long items = nseg * ((a.part_rows + 31) / 32);
  if (a.sched.splits == 0 && 4 * nseg >= a.sched.G) return launch_v<T, D, 2, 3>(a, sms, stream);
  if (items <= sms) return launch_v<T, D, 8, 1>(a, sms, stream);
  return launch_v<T, D, 4, 2>(a, sms, stream);
}

}  // namespace

cudaError_t launch_combine(const AttnParams& a, int dtype, cudaStream_t stream) {
  if (a.D == 64) {
    switch (dtype) {
      case 0: return launch_t<float, 64>(a, stream);
      case 1: return launch_t<__half, 64>(a, stream);
      default: return launch_t<__nv_bfloat16, 64>(a, stream);
    }
  }
  switch (dtype) {
    case 0: return launch_t<float, 128>(a, stream);
    case 1: return launch_t<__half, 128>(a, stream);
    default: return launch_t<__nv_bfloat16, 128>(a, stream);
  }
}

}  // namespace mt
