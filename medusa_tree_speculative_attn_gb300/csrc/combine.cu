// Split-KV combine: merges the partial softmax results of the pieces of one
// segment (the Flash-Decoding style split that lmdeploy PR 1231 "[WIP] support
// Medusa" plans for its tree-mask kernel).  For piece k with running maximum
// m_k (base-2 units), sum l_k and unnormalised output O_k:
//   M = max_k m_k,  w_k = 2^(m_k - M),  out = sum_k w_k O_k / sum_k w_k l_k.
// Segments covered by a single piece were written directly and are skipped.
#include "kernels.cuh"

namespace mt {

namespace {

constexpr int kWarps = 8;

// Block: 32 rows (one per lane) x 8 warps, warp w handles the 4-column groups
// w, w + 8, ...; partial reads are coalesced along rows.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) combine_kernel(AttnParams a) {
  constexpr int C4 = D / 4;                 // 4-column groups per row
  constexpr int PER = C4 / kWarps;          // groups per thread
  const Sched& s = a.sched;
  const int seg = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * 32 + lane;
  const int RG = a.rows_per_group;
  const int HR = s.Hkv * s.nrg;
  const int b = seg / HR, seg_in_b = seg % HR;
  const int kvh = seg_in_b / s.nrg, rg = seg_in_b % s.nrg;
  const int row = rg * RG + r;
  if (r >= RG || row >= a.rows) return;
  const int nt = s.tile_pfx[b + 1] - s.tile_pfx[b];
  if (nt == 0) return;

  // the slots holding this segment's pieces
  int slot0, count;
  long long t0 = 0, W = 0;
  if (s.splits == 0) {
    W = sched_total_tiles(s);
    t0 = (long long)s.tile_pfx[b] * HR + (long long)seg_in_b * nt;
    const int c0 = sched_cta_of(t0, W, s.G), c1 = sched_cta_of(t0 + nt - 1, W, s.G);
    if (c0 == c1) return;
    slot0 = seg + c0;
    count = c1 - c0 + 1;
  } else {
    if (s.splits == 1) return;
    slot0 = seg * s.splits;
    count = s.splits;
  }
  auto piece_exists = [&](int k) -> bool {
    if (s.splits == 0) {
      const int c = slot0 - seg + k;
      const long long cb = W * c / s.G, ce = W * (c + 1) / s.G;
      return (cb > t0 ? cb : t0) < (ce < t0 + nt ? ce : t0 + nt);
    }
    return (long long)nt * k / s.splits < (long long)nt * (k + 1) / s.splits;
  };

  float M = -INFINITY;
  for (int k = 0; k < count; ++k)
    if (piece_exists(k)) M = fmaxf(M, a.part_ml[(size_t)(slot0 + k) * RG + r].x);
  float4 acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  float lsum = 0.f;
  if (M != -INFINITY) {
    for (int k = 0; k < count; ++k) {
      if (!piece_exists(k)) continue;
      const size_t slot = (size_t)(slot0 + k);
      const float2 ml = a.part_ml[slot * RG + r];
      const float w = exp2f(ml.x - M);
      lsum += w * ml.y;
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const float4 v = a.part_o[(slot * C4 + warp + kWarps * e) * RG + r];
        acc[e].x = fmaf(w, v.x, acc[e].x);
        acc[e].y = fmaf(w, v.y, acc[e].y);
        acc[e].z = fmaf(w, v.z, acc[e].z);
        acc[e].w = fmaf(w, v.w, acc[e].w);
      }
    }
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  const int node = row / a.g, h = kvh * a.g + row % a.g;
  T* dst = static_cast<T*>(a.out) + (((size_t)b * a.T + node) * a.Hq + h) * D;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int c = 4 * (warp + kWarps * e);
    dst[c] = Act<T>::from_f(acc[e].x * inv);
    dst[c + 1] = Act<T>::from_f(acc[e].y * inv);
    dst[c + 2] = Act<T>::from_f(acc[e].z * inv);
    dst[c + 3] = Act<T>::from_f(acc[e].w * inv);
  }
}

template <typename T, int D>
cudaError_t launch_t(const AttnParams& a, cudaStream_t stream) {
  const int nseg = a.B * a.Hkv * a.sched.nrg;
  dim3 grid(nseg, (a.rows_per_group + 31) / 32);
  combine_kernel<T, D><<<grid, kWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
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
