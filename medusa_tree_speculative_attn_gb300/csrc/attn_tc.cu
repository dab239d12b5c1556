// Tensor-core tree attention over the paged KV cache (sm_103a: tcgen05 + TMEM
// + TMA), fp16/bf16.
//
// With T tree tokens and g query heads per KV head, each (sequence, KV head)
// has T*g query rows against the same keys: a real dense contraction, which
// belongs on tensor cores (vLLM issue 1171, void-main on PagedFlashAttention:
// with several candidates per sequence the "m dimension" is no longer 1).
// The split-KV structure follows the Flash-Decoding plan of lmdeploy PR 1231
// "[WIP] support Medusa"; the tree mask is the per-node ancestor bitmask.
//
// Persistent CTAs (one per SM) walk the balanced schedule of common.cuh.  A
// CTA holds up to 256 query rows (two 128-row M tiles) of one segment and
// streams its 64-slot key tiles:
//   producer warp  TMA 2-D loads of each tile's four 16-slot pages of K and V
//                  (page id from the block table; 128-byte swizzle) into a
//                  ring of stages; absent pages use an out-of-range
//                  coordinate, which TMA fills with zeros;
//   MMA warp       one thread issues S = Q K^T (M 128, N 64, K D) into TMEM,
//                  then O += P V (M 128, N D, K 64) once softmax wrote P;
//   softmax warps  one thread per query row: S from TMEM, tree/prefix mask,
//                  online softmax in base 2 with a lazy rescale (O in TMEM is
//                  rescaled only when the running max grows by more than 8),
//                  P to shared memory; at the end of a piece O / l goes to the
//                  output (whole segment) or O, m, l to a partial slot.
// Every mbarrier wait is bounded (2 s); on a timeout the kernel records
// MT_ERR_TIMEOUT, lets the other roles bail out, waits for its own TMA loads
// and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <type_traits>

#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace mt {

namespace {

constexpr int kSmemLimit = 232448;  // opt-in dynamic shared memory per CTA

__host__ __device__ constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

template <int D, int MT>
struct Cfg {
  static constexpr int NH = D / 64;                     // 64-element halves of a head row
  static constexpr int kQBytes = MT * NH * 128 * 128;   // [m][half][128 rows x 128 B]
  static constexpr int kPBytes = 2 * MT * 128 * 128;    // [buf][m][128 rows x 128 B]
  static constexpr int kHalfTile = kTileKeys * 128;     // 64 keys x 128 B
  static constexpr int kStageBytes = 2 * NH * kHalfTile;  // K and V halves
  static constexpr int kBarBytes = 1024;
  static constexpr int kStagesFit = (kSmemLimit - 1024 - kBarBytes - kQBytes - kPBytes) / kStageBytes;
  static constexpr int STAGES = kStagesFit > 6 ? 6 : kStagesFit;
  static constexpr int kSmemBytes = 1024 + kQBytes + kPBytes + STAGES * kStageBytes + kBarBytes;
  static constexpr int kSoftmaxWarps = 4 * MT;
  static constexpr int kProducerWarp = kSoftmaxWarps;
  static constexpr int kMmaWarp = kSoftmaxWarps + 1;
  static constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
  static constexpr int kTmemCols = pow2_at_least(MT * (D + 2 * kTileKeys));
  static_assert(STAGES >= 2, "shared memory budget");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
  __device__ static constexpr uint32_t o_col(int m) { return (uint32_t)(m * D); }
  __device__ static constexpr uint32_t s_col(int buf, int m) {
    return (uint32_t)(MT * D + (buf * MT + m) * kTileKeys);
  }
};

template <typename T> struct Pack2;
template <> struct Pack2<__half> {
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};
template <> struct Pack2<__nv_bfloat16> {
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* status) {
  const uint64_t t0 = tc::global_timer_ns();
  while (!tc::mbar_try_wait(bar, parity)) {
    if (tc::global_timer_ns() - t0 > tc::kWaitLimitNs) {
      set_status(status, kStTimeout);
      return;
    }
  }
}

// Visibility of the 64 slots [k0, k0 + 64) to a row whose node has ancestor
// mask anc: prefix slots (< L) always, tree slot L + t when bit t of anc is set.
__device__ __forceinline__ unsigned long long tile_visibility(int L, int k0,
                                                              unsigned long long anc) {
  const int base = L - k0;  // tile column of the first tree slot
  unsigned long long pre, tree;
  if (base >= 64) return ~0ull;
  if (base <= 0) pre = 0ull; else pre = (1ull << base) - 1ull;
  if (base >= 0) tree = anc << base;
  else if (base > -64) tree = anc >> (-base);
  else tree = 0ull;
  return pre | tree;
}

template <typename T, int D, int MT>
__global__ void __launch_bounds__(Cfg<D, MT>::kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const AttnParams a) {
  using C = Cfg<D, MT>;
  constexpr int S = C::STAGES;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t kIdescQK = tc::idesc_f16(kBf16, false, 128, kTileKeys);
  constexpr uint32_t kIdescPV = tc::idesc_f16(kBf16, true, 128, D);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sP = sQ + C::kQBytes;
  uint8_t* sKV = sP + C::kPBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + S * C::kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = full + S;
  uint64_t* s_full = empty + S;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;  // [2][MT]
  uint64_t* pv_done = p_full + 2 * MT;
  uint64_t* q_full = pv_done + 2;
  uint64_t* o_free = q_full + 1;
  uint64_t* fin = o_free + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&s_full[b], 1);
      tc::mbar_init(&s_free[b], C::kSoftmaxWarps);
      tc::mbar_init(&pv_done[b], 1);
      for (int m = 0; m < MT; ++m) tc::mbar_init(&p_full[b * MT + m], 4);
    }
    tc::mbar_init(q_full, C::kSoftmaxWarps);
    tc::mbar_init(o_free, C::kSoftmaxWarps);
    tc::mbar_init(fin, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == C::kMmaWarp) {
    tc::tmem_alloc(tmem_slot, C::kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == C::kProducerWarp && lane == 0) {
    tc::prefetch_tmap(&tmap_k);
    tc::prefetch_tmap(&tmap_v);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sQ_u = tc::smem_u32(sQ), sP_u = tc::smem_u32(sP), sKV_u = tc::smem_u32(sKV);

  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t policy = tc::policy_evict_first();
      const int oob_row = a.num_pages * a.Hkv * a.P;
      PieceIter pi;
      pi.init(a.sched, blockIdx.x);
      Piece pc;
      uint32_t it = 0;
      bool ok = true;
      while (ok && pi.next(pc)) {
        const int nkeys = a.seq_lens[pc.b] + a.T;
        const int* bt = a.block_tables + (size_t)pc.b * a.max_blocks;
        for (int j = pc.tile_begin; j < pc.tile_end; ++j, ++it) {
          const uint32_t stage = it % S;
          if (it >= (uint32_t)S) {
            ok = tc::mbar_wait(&empty[stage], ((it / S) - 1) & 1, abort_flag, a.status);
            if (!ok) break;
          }
          tc::mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
          uint8_t* kdst = sKV + stage * C::kStageBytes;
          uint8_t* vdst = kdst + C::NH * C::kHalfTile;
#pragma unroll
          for (int p = 0; p < kTileKeys / 16; ++p) {
            const int slot0 = j * kTileKeys + p * 16;
            int y = oob_row;
            if (slot0 < nkeys) {
              const int page = bt[slot0 / 16];
              if (page >= 0 && page < a.num_pages) y = (page * a.Hkv + pc.kvh) * 16;
              else set_status(a.status, kStPages);
            }
#pragma unroll
            for (int h = 0; h < C::NH; ++h) {
              tc::tma_load_2d(kdst + h * C::kHalfTile + p * 2048, &tmap_k, h * 64, y, &full[stage], policy);
              tc::tma_load_2d(vdst + h * C::kHalfTile + p * 2048, &tmap_v, h * 64, y, &full[stage], policy);
            }
          }
        }
      }
      // no TMA load may still be writing shared memory when the CTA exits
      const uint32_t first = it > (uint32_t)S ? it - S : 0;
      for (uint32_t t = first; t < it; ++t) drain_wait(&full[t % S], (t / S) & 1, a.status);
    }
  } else if (warp == C::kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    PieceIter pi;
    pi.init(a.sched, blockIdx.x);
    Piece pc;
    uint32_t it = 0, npieces = 0;
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      bool r = tc::mbar_wait(bar, parity, abort_flag, a.status);
      ok = __all_sync(0xffffffffu, r) && ok;
    };
    auto issue_pv = [&](uint32_t t, bool first_of_piece) {
      const uint32_t buf = t & 1, stage = t % S;
      if (first_of_piece && npieces > 0) {
        wait_all(o_free, (npieces - 1) & 1);
        if (!ok) return;
      }
      const uint32_t v_u = sKV_u + stage * C::kStageBytes + C::NH * C::kHalfTile;
      for (int m = 0; m < MT; ++m) {
        wait_all(&p_full[buf * MT + m], (t >> 1) & 1);
        if (!ok) return;
        tc::tc_fence_after();
        if (lane == 0) {
          const uint32_t p_u = sP_u + (buf * MT + m) * (128 * 128);
#pragma unroll
          for (int kk = 0; kk < kTileKeys / 16; ++kk) {
            const uint64_t ad = tc::smem_desc(p_u + kk * 32, 16, 1024);
            const uint64_t bd = tc::smem_desc(v_u + kk * 2048, C::kHalfTile, 1024);
            tc::mma_f16_ss(tmem + C::o_col(m), ad, bd, kIdescPV, (first_of_piece && kk == 0) ? 0u : 1u);
          }
        }
        __syncwarp();
      }
      if (lane == 0) {
        tc::mma_commit(&pv_done[buf]);
        tc::mma_commit(&empty[stage]);
      }
      __syncwarp();
    };
    while (ok && pi.next(pc)) {
      wait_all(q_full, npieces & 1);
      if (!ok) break;
      tc::tc_fence_after();
      const int nkeys = a.seq_lens[pc.b] + a.T;
      for (int j = pc.tile_begin; j < pc.tile_end; ++j, ++it) {
        const uint32_t stage = it % S, buf = it & 1;
        wait_all(&full[stage], (it / S) & 1);
        if (!ok) break;
        const int valid = nkeys - j * kTileKeys;
        if (valid < kTileKeys) {
          // slots past the sequence hold stale data (possibly NaN): zero the V
          // rows so that 0-probability columns contribute exactly 0
          uint8_t* vbase = sKV + stage * C::kStageBytes + C::NH * C::kHalfTile;
          const int nvec = (kTileKeys - valid) * 8;
          for (int h = 0; h < C::NH; ++h)
            for (int e = lane; e < nvec; e += 32)
              reinterpret_cast<uint4*>(vbase + h * C::kHalfTile + valid * 128)[e] = make_uint4(0, 0, 0, 0);
          tc::fence_proxy_async_smem();
          __syncwarp();
        }
        if (it >= 2) {
          wait_all(&s_free[buf], ((it >> 1) - 1) & 1);
          if (!ok) break;
        }
        tc::tc_fence_after();
        if (lane == 0) {
          const uint32_t k_u = sKV_u + stage * C::kStageBytes;
          for (int m = 0; m < MT; ++m) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t h = kk / 4, k4 = kk % 4;
              const uint64_t ad = tc::smem_desc(sQ_u + (m * C::NH + h) * (128 * 128) + k4 * 32, 16, 1024);
              const uint64_t bd = tc::smem_desc(k_u + h * C::kHalfTile + k4 * 32, 16, 1024);
              tc::mma_f16_ss(tmem + C::s_col(buf, m), ad, bd, kIdescQK, kk > 0 ? 1u : 0u);
            }
          }
          tc::mma_commit(&s_full[buf]);
        }
        __syncwarp();
        if (j > pc.tile_begin) {
          issue_pv(it - 1, j - 1 == pc.tile_begin);
          if (!ok) break;
        }
      }
      if (!ok) break;
      if (pc.tile_end > pc.tile_begin) issue_pv(it - 1, pc.tile_end - 1 == pc.tile_begin);
      ++npieces;
    }
    // every MMA issued by this warp has completed before TMEM is released
    if (lane == 0) {
      tc::mma_commit(fin);
      drain_wait(fin, 0, a.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int m = warp >> 2;               // M tile of this warpgroup
    const int quad = warp & 3;             // TMEM lane quadrant
    const int r = quad * 32 + lane;        // row within the M tile
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const T* __restrict__ q = static_cast<const T*>(a.q);
    const unsigned long long tmask = a.T == 64 ? ~0ull : ((1ull << a.T) - 1ull);
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      bool rr = tc::mbar_wait(bar, parity, abort_flag, a.status);
      ok = __all_sync(0xffffffffu, rr) && ok;
    };
    // rotated, rounded query row -> Q tile (K-major, 128-byte swizzle)
    auto load_q = [&](const Piece& p) {
      const int row = p.rg * kTcRows + m * 128 + r;
      uint8_t* qdst = sQ + m * C::NH * (128 * 128) + r * 128;
      const int L = a.seq_lens[p.b];
      constexpr int H = D / 2;
      if (row < a.rows) {
        const int node = row / a.g, h = p.kvh * a.g + row % a.g;
        const T* src = q + (((size_t)p.b * a.T + node) * a.Hq + h) * D;
        const int pos = L + a.tree_depths[(size_t)p.b * a.T + node];
        const bool pos_ok = pos >= 0 && pos < a.max_pos;
        if (!pos_ok) set_status(a.status, kStTree);
        const float2* cs = a.rope + (size_t)(pos_ok ? pos : 0) * H;
#pragma unroll
        for (int c = 0; c < H / 8; ++c) {
          uint4 lo_raw = *reinterpret_cast<const uint4*>(src + 8 * c);
          uint4 hi_raw = *reinterpret_cast<const uint4*>(src + H + 8 * c);
          T lo[8], hi[8], olo[8], ohi[8];
          memcpy(lo, &lo_raw, 16);
          memcpy(hi, &hi_raw, 16);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 t = cs[8 * c + e];
            float rl, rh;
            rope_pair(Act<T>::to_f(lo[e]), Act<T>::to_f(hi[e]), t.x, t.y, rl, rh);
            olo[e] = Act<T>::from_f(pos_ok ? rl : 0.f);
            ohi[e] = Act<T>::from_f(pos_ok ? rh : 0.f);
          }
          uint4 wl, wh;
          memcpy(&wl, olo, 16);
          memcpy(&wh, ohi, 16);
          const int cl = c, ch = H / 8 + c;  // 16-byte chunk index within the row
          *reinterpret_cast<uint4*>(qdst + (cl / 8) * (128 * 128) + (((cl % 8) ^ (r & 7)) << 4)) = wl;
          *reinterpret_cast<uint4*>(qdst + (ch / 8) * (128 * 128) + (((ch % 8) ^ (r & 7)) << 4)) = wh;
        }
      } else {
#pragma unroll
        for (int c = 0; c < D / 8; ++c)
          *reinterpret_cast<uint4*>(qdst + (c / 8) * (128 * 128) + (((c % 8) ^ (r & 7)) << 4)) =
              make_uint4(0, 0, 0, 0);
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(q_full);
    };

    PieceIter pi;
    pi.init(a.sched, blockIdx.x);
    Piece pc, nxt;
    uint32_t it = 0;
    bool have = pi.next(pc);
    if (have) load_q(pc);
    while (have && ok) {
      const int row = pc.rg * kTcRows + m * 128 + r;
      const bool row_ok = row < a.rows;
      const int node = row_ok ? row / a.g : 0;
      const unsigned long long anc = row_ok ? a.anc[(size_t)pc.b * a.T + node] : tmask;
      const int L = a.seq_lens[pc.b];
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = pc.tile_begin; j < pc.tile_end; ++j, ++it) {
        const uint32_t buf = it & 1;
        wait_all(&s_full[buf], (it >> 1) & 1);
        if (!ok) break;
        tc::tc_fence_after();
        uint32_t sr[64];
        tc::tmem_ld_x64(tmem + lane_addr + C::s_col(buf, m), sr);
        tc::tmem_ld_wait();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&s_free[buf]);
        const unsigned long long vis = tile_visibility(L, j * kTileKeys, anc);
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float x = __uint_as_float(sr[c]) * a.scale_log2;
          const float sv = ((vis >> c) & 1ull) ? x : -INFINITY;
          sr[c] = __float_as_uint(sv);
          mx = fmaxf(mx, sv);
        }
        // lazy rescale: the running max moves (and O in TMEM is rescaled) only
        // when the tile max exceeds it by more than 8, i.e. p <= 2^8 otherwise
        const bool grow = mx > m_run + 8.f;
        const bool need_o = grow && m_run != -INFINITY;
        const float m_new = grow ? mx : m_run;
        const float sc = need_o ? fast_exp2(m_run - m_new) : 1.f;
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        // P buffer `buf` was last read by the P.V of tile it - 2
        if (it >= 2) {
          wait_all(&pv_done[buf], ((it >> 1) - 1) & 1);
          if (!ok) break;
        }
        uint8_t* prow = sP + (buf * MT + m) * (128 * 128) + r * 128;
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float p[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            p[e] = fast_exp2(__uint_as_float(sr[8 * c + e]) - m_use);
            rs += p[e];
          }
          uint4 w;
          w.x = Pack2<T>::pack(p[0], p[1]);
          w.y = Pack2<T>::pack(p[2], p[3]);
          w.z = Pack2<T>::pack(p[4], p[5]);
          w.w = Pack2<T>::pack(p[6], p[7]);
          *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) = w;
        }
        if (__any_sync(0xffffffffu, need_o)) {
          // O holds the P.V sum up to tile it - 1: wait for it, then rescale
          wait_all(&pv_done[(it - 1) & 1], ((it - 1) >> 1) & 1);
          if (!ok) break;
          tc::tc_fence_after();
#pragma unroll 1
          for (int hh = 0; hh < D / 64; ++hh) {
            uint32_t o[64];
            tc::tmem_ld_x64(tmem + lane_addr + C::o_col(m) + 64 * hh, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 64; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * sc);
            tc::tmem_st_x64(tmem + lane_addr + C::o_col(m) + 64 * hh, o);
          }
          tc::tmem_st_wait();
        }
        l_run = l_run * sc + rs;
        m_run = m_new;
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&p_full[buf * MT + m]);
      }
      if (!ok) break;
      // next piece's Q goes in while the last P.V of this piece runs
      const bool have_next = pi.next(nxt);
      if (have_next) load_q(nxt);
      // epilogue
      wait_all(&pv_done[(it - 1) & 1], ((it - 1) >> 1) & 1);
      if (!ok) break;
      tc::tc_fence_after();
      const int seg_row = m * 128 + r;
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
      for (int hh = 0; hh < D / 64; ++hh) {
        uint32_t o[64];
        tc::tmem_ld_x64(tmem + lane_addr + C::o_col(m) + 64 * hh, o);
        tc::tmem_ld_wait();
        if (row_ok) {
          if (pc.slot < 0) {
            const int h = pc.kvh * a.g + row % a.g;
            T* dst = static_cast<T*>(a.out) + (((size_t)pc.b * a.T + node) * a.Hq + h) * D + 64 * hh;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              T v[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] = Act<T>::from_f(__uint_as_float(o[8 * c + e]) * inv);
              uint4 w;
              memcpy(&w, v, 16);
              reinterpret_cast<uint4*>(dst)[c] = w;
            }
          } else {
            float* dst = a.part_o + ((size_t)pc.slot * kTcRows + seg_row) * D + 64 * hh;
#pragma unroll
            for (int c = 0; c < 16; ++c)
              reinterpret_cast<uint4*>(dst)[c] = make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
          }
        }
      }
      if (row_ok && pc.slot >= 0)
        a.part_ml[(size_t)pc.slot * kTcRows + seg_row] = make_float2(m_run, l_run);
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(o_free);
      pc = nxt;
      have = have_next;
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == C::kMmaWarp) tc::tmem_dealloc(tmem, C::kTmemCols);
}

template <typename T, int D, int MT>
cudaError_t launch_t(const AttnParams& a, const CUtensorMap* tk, const CUtensorMap* tv,
                     cudaStream_t stream) {
  using C = Cfg<D, MT>;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<T, D, MT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  attn_tc_kernel<T, D, MT><<<a.sched.G, C::kThreads, C::kSmemBytes, stream>>>(*tk, *tv, a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dtype(const AttnParams& a, const CUtensorMap* tk, const CUtensorMap* tv,
                         cudaStream_t stream) {
  const bool one = a.rows <= 128;
  if (a.D == 64) return one ? launch_t<T, 64, 1>(a, tk, tv, stream) : launch_t<T, 64, 2>(a, tk, tv, stream);
  return one ? launch_t<T, 128, 1>(a, tk, tv, stream) : launch_t<T, 128, 2>(a, tk, tv, stream);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

// A paged cache [num_pages][Hkv][16][D] as a 2-D tensor of num_pages*Hkv*16
// rows by D columns; boxes of 16 rows (one page of one KV head) by 64 columns,
// 128-byte swizzle, zero fill outside.
cudaError_t make_cache_tmap(void* map_out, const void* base, int dtype, int num_pages, int Hkv,
                            int P, int D) {
  CUtensorMap* map = static_cast<CUtensorMap*>(map_out);
  auto enc = get_encode();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)num_pages * Hkv * P};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)P};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dtype == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_attn_tc(const AttnParams& a, int dtype, const void* tmap_k, const void* tmap_v,
                           cudaStream_t stream) {
  const CUtensorMap* tk = static_cast<const CUtensorMap*>(tmap_k);
  const CUtensorMap* tv = static_cast<const CUtensorMap*>(tmap_v);
  if (dtype == 1) return launch_dtype<__half>(a, tk, tv, stream);
  return launch_dtype<__nv_bfloat16>(a, tk, tv, stream);
}

}  // namespace mt
