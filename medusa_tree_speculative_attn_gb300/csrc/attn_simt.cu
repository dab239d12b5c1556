// SIMT (CUDA-core) tree attention over the paged KV cache.
//
// The fp32 path, the FP8 (E4M3) cache path, and for fp16/bf16 an independent
// second implementation that the tests hold against the tensor-core kernel.  Per piece of the schedule
// (see common.cuh) a CTA takes one 64-row group of (node, head) query rows of
// one (sequence, KV head) and streams that piece's 64-slot key tiles through
// shared memory: scores, online softmax in base 2, then P.V, all in fp32.
//
// Visibility of key slot k to the row of node i (the Medusa tree mask, vLLM
// issue 1171): k < L_b (a committed prefix token), or L_b <= k < L_b + T and
// bit (k - L_b) of anc[i] is set (a tree ancestor of i, or i itself).
#include <cuda_fp8.h>

#include "kernels.cuh"

namespace mt {

namespace {

constexpr int kThreads = 256;

template <typename T, int D>
__device__ __forceinline__ void load_kv_tile(const T* __restrict__ cache, float* dst, int b,
                                             int kvh, int k0, int nkeys, const AttnParams& a) {
  constexpr int LD = D + 1;
  constexpr int EPV = 16 / sizeof(T);
  constexpr int VPR = D / EPV;
  for (int v = threadIdx.x; v < kTileKeys * VPR; v += blockDim.x) {
    const int key = v / VPR, part = v % VPR;
    const int slot = k0 + key;
    float vals[EPV];
#pragma unroll
    for (int e = 0; e < EPV; ++e) vals[e] = 0.f;
    if (slot < nkeys) {
      const int page = a.block_tables[(size_t)b * a.max_blocks + slot / a.P];
      if (page >= 0 && page < a.num_pages) {
        const T* src = cache + (((size_t)page * a.Hkv + kvh) * a.P + slot % a.P) * D + part * EPV;
        uint4 raw = __ldg(reinterpret_cast<const uint4*>(src));
        T tmp[EPV];
        memcpy(tmp, &raw, 16);
#pragma unroll
        for (int e = 0; e < EPV; ++e) vals[e] = Act<T>::to_f(tmp[e]);
      } else {
        set_status(a.status, kStPages);
      }
    }
#pragma unroll
    for (int e = 0; e < EPV; ++e) dst[key * LD + part * EPV + e] = vals[e];
  }
}

// The same tile from an FP8 cache: 16 E4M3 codes per 16-byte load, each
// decoded exactly (through fp16, which holds every E4M3 value) and scaled.
template <int D>
__device__ __forceinline__ void load_kv_tile_e4m3(const uint8_t* __restrict__ cache, float* dst, int b,
                                                  int kvh, int k0, int nkeys, float scale, const AttnParams& a) {
  constexpr int LD = D + 1;
  constexpr int EPV = 16;
  constexpr int VPR = D / EPV;
  for (int v = threadIdx.x; v < kTileKeys * VPR; v += blockDim.x) {
    const int key = v / VPR, part = v % VPR;
    const int slot = k0 + key;
    float vals[EPV];
#pragma unroll
    for (int e = 0; e < EPV; ++e) vals[e] = 0.f;
    if (slot < nkeys) {
      const int page = a.block_tables[(size_t)b * a.max_blocks + slot / a.P];
      if (page >= 0 && page < a.num_pages) {
        const uint8_t* src = cache + (((size_t)page * a.Hkv + kvh) * a.P + slot % a.P) * D + part * EPV;
        uint4 raw = __ldg(reinterpret_cast<const uint4*>(src));
        uint8_t codes[EPV];
        memcpy(codes, &raw, 16);
#pragma unroll
        for (int e = 0; e < EPV; ++e)
          vals[e] = __half2float(__half(__nv_cvt_fp8_to_halfraw(codes[e], __NV_E4M3))) * scale;
      } else {
        set_status(a.status, kStPages);
      }
    }
#pragma unroll
    for (int e = 0; e < EPV; ++e) dst[key * LD + part * EPV + e] = vals[e];
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, kSimtCtasPerSm) attn_simt_kernel(AttnParams a, Fp8Cache f8) {
  constexpr int R = kSimtRows;
  constexpr int LD = D + 1;
  constexpr int PLD = kTileKeys + 1;
  constexpr int NC = D / 16;
  extern __shared__ float smem[];
  float* Qs = smem;               // [R][LD]
  float* KV = Qs + R * LD;        // [64][LD]
  float* Ps = KV + kTileKeys * LD;  // [R][PLD]
  __shared__ unsigned long long s_anc[R];
  pdl_wait();

  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const T* __restrict__ q = static_cast<const T*>(a.q_rot);
  const T* __restrict__ kc = static_cast<const T*>(a.k_cache);
  const T* __restrict__ vc = static_cast<const T*>(a.v_cache);

  PieceIter it;
  it.init(a.sched, blockIdx.x);
  Piece pc;
  while (it.next(pc)) {
    const int b = pc.b, kvh = pc.kvh;
    const int L = a.seq_lens[b];
    const int nkeys = L + a.T;
    const int row0 = pc.rg * R;
    for (int r = tid; r < R; r += blockDim.x) {
      const int row = row0 + r;
      s_anc[r] = row < a.rows ? a.anc[(size_t)b * a.T + row / a.g] : ~0ull;
    }
    // query rows (rotated at L_b + depth and rounded by the prep kernel)
    for (int e = tid; e < R * D; e += blockDim.x) {
      const int r = e / D, d = e % D;
      const int row = row0 + r;
      float v = 0.f;
      if (row < a.rows) {
        const int node = row / a.g, h = kvh * a.g + row % a.g;
        v = Act<T>::to_f(q[(((size_t)b * a.T + node) * a.Hq + h) * D + d]);
      }
      Qs[r * LD + d] = v;
    }
    float m[4], l[4], o[4][NC];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      m[i] = -INFINITY;
      l[i] = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c) o[i][c] = 0.f;
    }
    __syncthreads();

    for (int jt = pc.tile_begin; jt < pc.tile_end; ++jt) {
      const int k0 = jt * kTileKeys;
      if (f8.on)
        load_kv_tile_e4m3<D>(static_cast<const uint8_t*>(a.k_cache), KV, b, kvh, k0, nkeys, f8.k_scale, a);
      else
        load_kv_tile<T, D>(kc, KV, b, kvh, k0, nkeys, a);
      __syncthreads();
      float s[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[i][c] = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) {
        float qv[4], kv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) qv[i] = Qs[(ty * 4 + i) * LD + d];
#pragma unroll
        for (int c = 0; c < 4; ++c) kv[c] = KV[(tx + 16 * c) * LD + d];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c = 0; c < 4; ++c) s[i][c] = fmaf(qv[i], kv[c], s[i][c]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = ty * 4 + i;
        const unsigned long long anc = s_anc[r];
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int slot = k0 + tx + 16 * c;
          const bool vis = slot < nkeys && (slot < L || ((anc >> (slot - L)) & 1ull));
          s[i][c] = vis ? s[i][c] * a.scale_log2 : -INFINITY;
          mx = fmaxf(mx, s[i][c]);
        }
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m[i], mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = exp2f(m[i] - m_use);
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float p = exp2f(s[i][c] - m_use);
          Ps[r * PLD + tx + 16 * c] = p;
          rs += p;
        }
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
        l[i] = l[i] * alpha + rs;
        m[i] = m_new;
#pragma unroll
        for (int c = 0; c < NC; ++c) o[i][c] *= alpha;
      }
      __syncthreads();
      if (f8.on)
        load_kv_tile_e4m3<D>(static_cast<const uint8_t*>(a.v_cache), KV, b, kvh, k0, nkeys, f8.v_scale, a);
      else
        load_kv_tile<T, D>(vc, KV, b, kvh, k0, nkeys, a);
      __syncthreads();
#pragma unroll 4
      for (int k = 0; k < kTileKeys; ++k) {
        float pv[4], vv[NC];
#pragma unroll
        for (int i = 0; i < 4; ++i) pv[i] = Ps[(ty * 4 + i) * PLD + k];
#pragma unroll
        for (int c = 0; c < NC; ++c) vv[c] = KV[k * LD + tx + 16 * c];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c = 0; c < NC; ++c) o[i][c] = fmaf(pv[i], vv[c], o[i][c]);
      }
      __syncthreads();
    }

    // epilogue: direct output (whole segment) or a partial for the combine
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = ty * 4 + i;
      const int row = row0 + r;
      if (row >= a.rows) continue;
      if (pc.slot < 0) {
        const int node = row / a.g, h = kvh * a.g + row % a.g;
        T* dst = static_cast<T*>(a.out) + (((size_t)b * a.T + node) * a.Hq + h) * D;
        const float inv = 1.f / l[i];
#pragma unroll
        for (int c = 0; c < NC; ++c) dst[tx + 16 * c] = Act<T>::from_f(o[i][c] * inv);
      } else {
        // the partial output O / l in the act dtype, [slot][D/8][rows][8]
        // (a row that saw no key of this piece has l = 0 and m = -inf: the
        // combine skips it)
        T* dst = static_cast<T*>(a.part_o);
        const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int col = tx + 16 * c;
          dst[(((size_t)pc.slot * (D / 8) + col / 8) * a.part_rows + r) * 8 + col % 8] = Act<T>::from_f(o[i][c] * inv);
        }
        if (tx == 0) a.part_ml[(size_t)pc.slot * a.part_rows + r] = make_float2(m[i], l[i]);
      }
    }
    __syncthreads();
  }
}

template <typename T, int D>
cudaError_t launch_simt_t(const AttnParams& a, const Fp8Cache& f8, cudaStream_t stream) {
  constexpr int LD = D + 1;
  const size_t smem = sizeof(float) * (size_t)(kSimtRows * LD + kTileKeys * LD + kSimtRows * (kTileKeys + 1));
  cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_simt_kernel<T, D>, dim3(a.sched.G), dim3(kThreads), smem, stream, a, f8);
}

}  // namespace

cudaError_t launch_attn_simt(const AttnParams& a, const Fp8Cache& f8, int dtype, cudaStream_t stream) {
  if (a.D == 64) {
    switch (dtype) {
      case 0: return launch_simt_t<float, 64>(a, f8, stream);
      case 1: return launch_simt_t<__half, 64>(a, f8, stream);
      default: return launch_simt_t<__nv_bfloat16, 64>(a, f8, stream);
    }
  }
  switch (dtype) {
    case 0: return launch_simt_t<float, 128>(a, f8, stream);
    case 1: return launch_simt_t<__half, 128>(a, f8, stream);
    default: return launch_simt_t<__nv_bfloat16, 128>(a, f8, stream);
  }
}

}  // namespace mt
