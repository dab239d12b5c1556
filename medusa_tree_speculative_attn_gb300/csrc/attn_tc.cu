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
// streams its 64-slot key tiles.  Warp roles:
//   producers  four warps, one per SM sub-partition; producer p issues the TMA
//              loads of page p of every tile (K and V, 128-byte swizzle, page
//              ids from the block table; absent pages use an out-of-range row,
//              which TMA fills with zeros).  A single issuing thread cannot
//              keep HBM busy with 2 KB boxes; four can.  A piece's rotated
//              queries go through the same ring, one slot per M tile ahead of
//              the piece's tiles, their boxes shared out over the producers;
//   QK issuer  one thread copies each piece's queries from shared memory into
//              TMEM and issues S = Q K^T (M 128, N 64, K D; A = Q from TMEM)
//              into TMEM, for M tile m as soon as the softmax has read S_m;
//   PV issuer  one thread issues O += P V (M 128, N D, K 64), P and V from
//              shared memory; separate from the QK issuer so that neither
//              waits behind the other's dependencies;
//   softmax    one thread per query row: S from TMEM, tree/prefix mask (only
//              on tiles that reach past the prefix), online softmax in base 2
//              with a lazy rescale (O in TMEM is rescaled only when the
//              running max grows by more than 8), P written as 16-bit values
//              to a 128-byte-swizzled shared-memory tile; at the end of a
//              piece O / l goes to the output (whole segment) or O, m, l to a
//              partial slot.
// Shared memory holds P (16 KB per M tile) and a ring of 32 KB slots (a
// tile's K and V, or an M tile's queries); TMEM holds O (2 x 128 columns),
// S (2 x 64) and Q (2 x 64 packed 16-bit pairs).
// Tensor-core instructions are issued by the elected lane of a converged warp
// (tc::elect_one), which issues about twice as fast as a lane-0 branch.
// Every mbarrier wait is bounded (2 s unless the caller set another limit);
// on a timeout the kernel records MT_ERR_TIMEOUT, lets the other roles bail
// out, waits for its own TMA loads and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <atomic>
#include <type_traits>

#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace mt {

namespace {

constexpr int kSmemLimit = 232448;  // opt-in dynamic shared memory per CTA
constexpr int kMaxDevices = 64;

__host__ __device__ constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

template <int D, int MT, bool FP8 = false>
struct Cfg {
  static constexpr int NH = D / 64;                     // 64-element halves of a head row
  // A piece's queries travel through the K/V ring: M tile m's 128 rows x D
  // (the [half][128 rows x 128 B] boxes) fill one ring slot, which is exactly
  // one stage (K and V of 64 keys), so no shared memory is set aside for them
  // and the next piece's queries are prefetched in ring order.
  static constexpr int kPTile = 128 * kTileKeys * 2;     // P of one M tile: 128 rows x 128 B
  // P buffers per M tile.  Two would let the softmax of tile t wait for the
  // P.V of tile t - 2 instead of t - 1, but measured slower on every
  // workload (serving 78.2 against 75.6 us at four stages, 84.8 against 76.8
  // when it cost a stage), so there is one.
  static constexpr int NPB = 1;
  static constexpr int kPBytes = MT * NPB * kPTile;      // [m][buffer]
  static constexpr int kHalfTile = kTileKeys * 128;     // 64 keys x 128 B
  static constexpr int kStageBytes = 2 * NH * kHalfTile;  // K and V halves
  static constexpr int kBarBytes = 2048;  // barriers (first 1 KB) + the CTA's piece list
  // An FP8 (E4M3) cache: each producer TMAs its page's codes (K then V,
  // 16 rows x D bytes each) into a private ring of kF8Depth slots and converts
  // them into the ring stage the MMAs read.
  static constexpr int kF8Depth = 4;
  static constexpr int kF8PageBytes = 2 * 16 * D;
  static constexpr int kF8Bytes = FP8 ? (kTileKeys / 16) * kF8Depth * kF8PageBytes : 0;
  static constexpr int kStagesFit = (kSmemLimit - 1024 - kBarBytes - kPBytes - kF8Bytes) / kStageBytes;
  // ring depth: two M tiles run best with four stages (more stages measured
  // slower: the loads in flight then compete with the MMAs and P for shared
  // memory bandwidth); one M tile streams faster with more
  static constexpr int kStageCap = MT == 2 ? 4 : 8;
  static constexpr int STAGES = kStagesFit > kStageCap ? kStageCap : kStagesFit;
  static constexpr int kSmemBytes = 1024 + kPBytes + STAGES * kStageBytes + kF8Bytes + kBarBytes;
  static constexpr int kSoftmaxWarps = 4 * MT;
  static constexpr int kQkWarp = kSoftmaxWarps;
  static constexpr int kPvWarp = kSoftmaxWarps + 1;
  // four producer warps, one per SM sub-partition (warp w runs on w % 4):
  // producer p loads page p of each tile's four
  static constexpr int kProducer0 = kSoftmaxWarps + 2;
  static constexpr int kProducers = kTileKeys / 16;
  static constexpr int kProducerBytes = 2 * NH * 16 * 128;  // K and V of one page
  static constexpr int kThreads = (kSoftmaxWarps + 2 + kProducers) * 32;
  // TMEM: O (D fp32 columns per M tile), S (64 per M tile), Q (D/2 packed
  // 16-bit pairs per M tile)
  static constexpr int kTmemCols = pow2_at_least(MT * (D + kTileKeys + D / 2));
  static_assert(STAGES >= 2, "shared memory budget");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
  __device__ static constexpr uint32_t o_col(int m) { return (uint32_t)(m * D); }
  __device__ static constexpr uint32_t s_col(int m) { return (uint32_t)(MT * D + m * kTileKeys); }
  __device__ static constexpr uint32_t q_col(int m) { return (uint32_t)(MT * (D + kTileKeys) + m * (D / 2)); }
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

// Eight E4M3 codes (8 bytes, first element lowest) as eight act-dtype values
// (16 bytes).  Every E4M3 value is exact in fp16, fp32 and bf16: codes go
// pairwise to f16x2, and for bf16 on through fp32.
template <typename T>
__device__ __forceinline__ uint4 e4m3x8_to_act(uint2 c8) {
  uint32_t h[4];
  const uint32_t w[2] = {c8.x, c8.y};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint16_t pair = (uint16_t)(w[i / 2] >> (16 * (i % 2)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[i]) : "h"(pair));
  }
  if (std::is_same<T, __nv_bfloat16>::value) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 x;
      memcpy(&x, &h[i], 4);
      const float2 f = __half22float2(x);
      __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
      memcpy(&h[i], &b, 4);
    }
  }
  return make_uint4(h[0], h[1], h[2], h[3]);
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* status) {
  const uint64_t t0 = tc::global_timer_ns();
  while (!tc::mbar_try_wait(bar, parity)) {
    if (tc::global_timer_ns() - t0 > tc::kDrainLimitNs) {
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

template <typename T, int D, int MT, bool FP8>
__global__ void __launch_bounds__(Cfg<D, MT, FP8>::kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v,
                   const __grid_constant__ CUtensorMap tmap_q, const AttnParams a) {
  using C = Cfg<D, MT, FP8>;
  constexpr int S = C::STAGES;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t kIdescQK = tc::idesc_f16(kBf16, false, 128, kTileKeys);
  constexpr uint32_t kIdescPV = tc::idesc_f16(kBf16, true, 128, D);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr int NPB = C::NPB;
  uint8_t* sP = smem;                // [m][buffer] P tiles, 128-byte swizzled, K-major
  uint8_t* sKV = sP + C::kPBytes;
  uint8_t* sF8 = sKV + S * C::kStageBytes;  // [producer][kF8Depth] FP8 code pages (FP8 caches)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sF8 + C::kF8Bytes);
  uint64_t* full = bars;                // [S] ring slot landed (a tile's K/V, or an M tile's queries)
  uint64_t* empty = full + S;           // [S] ring slot consumed (by its P.V, or its copy into TMEM)
  // per M tile, one phase per tile:
  uint64_t* s_full = empty + S;         // [MT] S computed
  uint64_t* p_full = s_full + MT;       // [MT][NPB] P written (and O rescaled), one phase per use
  uint64_t* pv_done = p_full + MT * NPB;  // [MT][NPB] O += P V done, one phase per use
  uint64_t* s_free = pv_done + MT * NPB;  // [MT] S read out by the softmax
  uint64_t* o_free = s_free + MT;       // O of the previous piece read out
  uint64_t* fin = o_free + 1;           // [2] every MMA of each issuer done
  uint64_t* never = fin + 2;            // nothing arrives here (timeout test hook)
  uint64_t* f8_full = never + 1;        // [producer][kF8Depth] FP8 code page landed (FP8 caches)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(f8_full + C::kProducers * C::kF8Depth);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_npieces = const_cast<int*>(abort_flag + 1);
  uint32_t* s_f8pos = reinterpret_cast<uint32_t*>(s_npieces + 1);  // [producer][kF8Depth] ring positions
  static_assert((2 * 8 + 8 * 2 + 6 + C::kProducers * C::kF8Depth) * 8 + 12 +
                    C::kProducers * C::kF8Depth * 4 <= 1024, "barrier area");
  PieceRec* s_pieces = reinterpret_cast<PieceRec*>(reinterpret_cast<uint8_t*>(bars) + 1024);
  static_assert(kMaxPieceRecs * sizeof(PieceRec) <= C::kBarBytes - 1024, "piece list");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], C::kProducers);
      tc::mbar_init(&empty[s], 1);
    }
    for (int m = 0; m < MT; ++m) {
      tc::mbar_init(&s_full[m], 1);
      for (int b = 0; b < NPB; ++b) {
        tc::mbar_init(&p_full[m * NPB + b], 4);
        tc::mbar_init(&pv_done[m * NPB + b], 1);
      }
      tc::mbar_init(&s_free[m], 4);
    }
    tc::mbar_init(&fin[0], 1);
    tc::mbar_init(&fin[1], 1);
    tc::mbar_init(never, 1);
    for (int k = 0; k < C::kProducers * C::kF8Depth; ++k) tc::mbar_init(&f8_full[k], 1);
    tc::mbar_init(o_free, C::kSoftmaxWarps);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == C::kQkWarp) {
    tc::tmem_alloc(tmem_slot, C::kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == C::kProducer0 && lane == 0) {
    tc::prefetch_tmap(&tmap_k);
    tc::prefetch_tmap(&tmap_v);
    tc::prefetch_tmap(&tmap_q);
  }
  // everything above overlaps the end of the preceding kernel; the piece
  // table, queries, masks and block tables are read only past this wait
  pdl_wait();
  if (warp == C::kPvWarp) {
    // this CTA's piece list (written by the prep kernel) into shared memory:
    // the first four records are loaded with the count, the rest (rare) after
    const int* src = a.piece_table + piece_rec_offset(a.sched.G) + (size_t)blockIdx.x * kMaxPieceRecs * 8;
    const int first = src[lane];
    const int n = a.piece_table[blockIdx.x];
    int* dst = reinterpret_cast<int*>(s_pieces);
    dst[lane] = first;
    if (lane == 0) *s_npieces = n;
    for (int e = 32 + lane; e < (n > 0 ? n : 0) * 8; e += 32) dst[e] = src[e];
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sKV_u = tc::smem_u32(sKV), sP_u = tc::smem_u32(sP);
  const uint64_t limit = a.wait_limit_ns;

  if (warp >= C::kProducer0) {
    // ----------------------------------------------------------- producers
    // Each producer warp walks the schedule (page ids fetched warp-wide ahead
    // of use) and its lane 0 issues the K and V copies of its page of every
    // tile: one thread's TMA issue rate cannot keep up with HBM, four can.
    // Each piece's queries take the ring's next MT slots before its tiles.
    const int pid = warp - C::kProducer0;
    const uint64_t policy = tc::policy_evict_first();
    const uint64_t q_policy = tc::policy_evict_last();
    const int oob_row = a.num_pages * a.Hkv * a.P;
    PieceSrc pi;
    pi.init(s_pieces, *s_npieces, a.sched, blockIdx.x, a.seq_lens);
    Piece pc;
    int pL = 0;
    uint32_t pos = 0;  // ring position: MT query slots per piece, then one slot per tile
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      bool r = tc::mbar_wait(bar, parity, abort_flag, a.status, limit);
      ok = __all_sync(0xffffffffu, r) && ok;
    };
    // FP8 caches: tiles whose codes were issued (f8_issued) and converted
    // into their stages (f8_done); slot f of this producer's FP8 ring holds
    // the codes of tile f8_done + ((f - f8_done) mod depth), whose ring
    // position is in s_f8pos.
    uint32_t f8_issued = 0, f8_done = 0;
    unsigned long long q_slots = 0;  // bit p % 64: ring position p held queries (FP8 drain)
    // Convert the oldest issued tile: wait for its codes and for its stage,
    // then each lane turns half a row (D/2 codes of K, then of V) into act
    // values in the stage's 128-byte-swizzled layout (row pid * 16 + r), and
    // the warp arrives on the stage's barrier (all four producers do).
    auto f8_convert_oldest = [&]() {
      const uint32_t f = f8_done % C::kF8Depth;
      wait_all(&f8_full[pid * C::kF8Depth + f], (f8_done / C::kF8Depth) & 1);
      if (!ok) return;
      const uint32_t p = s_f8pos[pid * C::kF8Depth + f];
      const uint32_t st = p % S;
      if (p >= (uint32_t)S) {
        wait_all(&empty[st], ((p / S) - 1) & 1);
        if (!ok) return;
      }
      const uint8_t* codes = sF8 + (pid * C::kF8Depth + f) * C::kF8PageBytes;
      // 16-byte chunks of codes: consecutive lanes read consecutive chunks
      // (no bank conflicts); chunk q is row q / (D/16), columns 16 (q % (D/16))
      // on, and becomes two 8-column chunks of the stage's row pid * 16 + row
      constexpr int kChunksPerRow = D / 16;
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        uint8_t* dst = sKV + st * C::kStageBytes + kv * C::NH * C::kHalfTile;
#pragma unroll
        for (int i = 0; i < 16 * kChunksPerRow / 32; ++i) {
          const int q = i * 32 + lane;
          const int r = q / kChunksPerRow, col = (q % kChunksPerRow) * 16;
          const uint4 c16 = *reinterpret_cast<const uint4*>(codes + kv * 16 * D + q * 16);
          const int row = pid * 16 + r;
          uint8_t* drow = dst + (col / 64) * C::kHalfTile + row * 128;
          const int c0 = (col % 64) / 8;
          *reinterpret_cast<uint4*>(drow + ((c0 ^ (row & 7)) << 4)) = e4m3x8_to_act<T>(make_uint2(c16.x, c16.y));
          *reinterpret_cast<uint4*>(drow + (((c0 + 1) ^ (row & 7)) << 4)) =
              e4m3x8_to_act<T>(make_uint2(c16.z, c16.w));
        }
      }
      tc::fence_proxy_async_smem();  // the stage is read by the tensor core; the codes' slot is refilled by TMA
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&full[st]);
      ++f8_done;
    };
    // convert every issued tile at ring position <= p - S, before a wait on
    // position p's stage (which can depend on them)
    auto f8_flush_until = [&](uint32_t p) {
      while (ok && f8_done < f8_issued && p >= (uint32_t)S &&
             s_f8pos[pid * C::kF8Depth + f8_done % C::kF8Depth] <= p - S)
        f8_convert_oldest();
    };
    while (ok && pi.next(pc, pL)) {
      // the piece's queries, one slot per M tile; the slot's boxes (one per
      // 64-column half) are shared out over the producers, and every
      // producer arrives once on every slot
      for (int m = 0; m < MT && ok; ++m, ++pos) {
        const uint32_t slot = pos % S;
        if (FP8) f8_flush_until(pos);
        if (pos >= (uint32_t)S && ok) {
          wait_all(&empty[slot], ((pos / S) - 1) & 1);
          if (!ok) break;
        }
        q_slots |= 1ull << (pos % 64);
        if (lane == 0) {
          int mine = 0;
          for (int h = 0; h < C::NH; ++h) mine += ((m * C::NH + h) % C::kProducers) == pid;
          if (mine > 0) {
            tc::mbar_arrive_expect_tx(&full[slot], (uint32_t)(mine * 128 * 128));
            const int z = pc.b * a.T + (pc.rg * kTcRows + m * 128) / a.g;
            for (int h = 0; h < C::NH; ++h)
              if (((m * C::NH + h) % C::kProducers) == pid)
                tc::tma_load_3d(sKV + slot * C::kStageBytes + h * (128 * 128), &tmap_q, h * 64, pc.kvh * a.g, z,
                                &full[slot], q_policy);
          } else {
            tc::mbar_arrive(&full[slot]);
          }
        }
        __syncwarp();
      }
      if (!ok) break;
      const int nkeys = pL + a.T;
      PageWindow pw;
      pw.init(a.block_tables + (size_t)pc.b * a.max_blocks, nkeys, a.max_blocks,
              pc.tile_begin * (kTileKeys / 16), lane);
      for (int j = pc.tile_begin; j < pc.tile_end; ++j, ++pos) {
        const int y = pw.page(j * (kTileKeys / 16) + pid, lane);
        const uint32_t stage = pos % S;
        if (FP8) {
          // the codes go to this producer's FP8 ring; converting them into
          // the stage waits for the stage, later
          if (f8_issued - f8_done == (uint32_t)C::kF8Depth) f8_convert_oldest();
          if (!ok) break;
          q_slots &= ~(1ull << (pos % 64));
          const uint32_t f = f8_issued % C::kF8Depth;
          if (lane == 0) {
            uint64_t* bar = &f8_full[pid * C::kF8Depth + f];
            tc::mbar_arrive_expect_tx(bar, C::kF8PageBytes);
            uint8_t* kdst = sF8 + (pid * C::kF8Depth + f) * C::kF8PageBytes;
            int row = oob_row;
            if (y >= 0 && y < a.num_pages) row = (y * a.Hkv + pc.kvh) * 16;
            else if (j * kTileKeys + pid * 16 < nkeys) set_status(a.status, kStPages);
            tc::tma_load_2d(kdst, &tmap_k, 0, row, bar, policy);
            tc::tma_load_2d(kdst + 16 * D, &tmap_v, 0, row, bar, policy);
            s_f8pos[pid * C::kF8Depth + f] = pos;
          }
          __syncwarp();
          ++f8_issued;
          continue;
        }
        if (pos >= (uint32_t)S) {
          wait_all(&empty[stage], ((pos / S) - 1) & 1);
          if (!ok) break;
        }
        if (lane == 0) {
          tc::mbar_arrive_expect_tx(&full[stage], C::kProducerBytes);
          uint8_t* kdst = sKV + stage * C::kStageBytes + pid * 2048;
          uint8_t* vdst = kdst + C::NH * C::kHalfTile;
          int row = oob_row;
          if (y >= 0 && y < a.num_pages) row = (y * a.Hkv + pc.kvh) * 16;
          else if (j * kTileKeys + pid * 16 < nkeys) set_status(a.status, kStPages);
#pragma unroll
          for (int h = 0; h < C::NH; ++h) {
            tc::tma_load_2d(kdst + h * C::kHalfTile, &tmap_k, h * 64, row, &full[stage], policy);
            tc::tma_load_2d(vdst + h * C::kHalfTile, &tmap_v, h * 64, row, &full[stage], policy);
          }
        }
        __syncwarp();
      }
    }
    if (FP8)
      while (ok && f8_done < f8_issued) f8_convert_oldest();
    // no TMA load may still be writing shared memory when the CTA exits
    if (lane == 0) {
      if (FP8) {
        // codes never converted (after an abort), then the query slots
        for (uint32_t u = f8_done; u < f8_issued; ++u)
          drain_wait(&f8_full[pid * C::kF8Depth + u % C::kF8Depth], (u / C::kF8Depth) & 1, a.status);
      }
      // the last S positions' loads (with FP8 codes, only query slots are
      // loaded into stages by TMA; the rest were written by the warps)
      const uint32_t first = pos > (uint32_t)S ? pos - S : 0;
      for (uint32_t t = first; t < pos; ++t)
        if (!FP8 || ((q_slots >> (t % 64)) & 1ull)) drain_wait(&full[t % S], (t / S) & 1, a.status);
    }
    __syncwarp();
  } else if (warp == C::kQkWarp) {
    // ---------------------------------------------------------- QK issuer
    PieceSrc pi;
    pi.init(s_pieces, *s_npieces, a.sched, blockIdx.x, a.seq_lens);
    Piece pc;
    int pL = 0;
    uint32_t it = 0, pos = 0;  // tiles so far; ring position (as the producers count it)
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      bool r = tc::mbar_wait(bar, parity, abort_flag, a.status, limit);
      ok = __all_sync(0xffffffffu, r) && ok;
    };
    if (a.test_stall) wait_all(never, 0);  // test hook: a wait that can only time out
    while (ok && pi.next(pc, pL)) {
      // the piece's queries: ring slots -> TMEM (after every Q K^T of the
      // previous piece, in issue order); each slot is free once copied
      for (int m = 0; m < MT && ok; ++m) wait_all(&full[(pos + m) % S], ((pos + m) / S) & 1);
      if (!ok) break;
      tc::tc_fence_after();
      for (int m = 0; m < MT; ++m) {
        const uint32_t q_u = sKV_u + ((pos + m) % S) * C::kStageBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t h = kk / 4, k4 = kk % 4;
          if (tc::elect_one())
            tc::tmem_cp_128x256b(tmem + C::q_col(m) + kk * 8,
                                 tc::smem_desc(q_u + h * (128 * 128) + k4 * 32, 16, 1024));
        }
        if (tc::elect_one()) tc::mma_commit(&empty[(pos + m) % S]);
      }
      __syncwarp();
      pos += MT;
      for (int j = pc.tile_begin; j < pc.tile_end; ++j, ++it, ++pos) {
        const uint32_t stage = pos % S;
        wait_all(&full[stage], (pos / S) & 1);
        if (!ok) break;
        const uint32_t k_u = sKV_u + stage * C::kStageBytes;
        // one descriptor per stage; a K slice is a constant offset (16-byte
        // units in the address field, which cannot carry: addresses < 256 KB)
        const uint64_t kd0 = tc::smem_desc(k_u, 16, 1024);
        for (int m = 0; m < MT; ++m) {
          // S_m held the scores of tile it - 1 until the softmax read them
          if (it >= 1) {
            wait_all(&s_free[m], (it - 1) & 1);
            if (!ok) break;
          }
          tc::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t h = kk / 4, k4 = kk % 4;
            const uint64_t bd = kd0 + (uint64_t)((h * C::kHalfTile + k4 * 32) >> 4);
            if (kk == 0) {
              if (tc::elect_one()) tc::mma_f16_ts<false>(tmem + C::s_col(m), tmem + C::q_col(m), bd, kIdescQK);
            } else {
              if (tc::elect_one()) tc::mma_f16_ts<true>(tmem + C::s_col(m), tmem + C::q_col(m) + kk * 8, bd, kIdescQK);
            }
          }
          if (tc::elect_one()) tc::mma_commit(&s_full[m]);
          __syncwarp();
        }
        if (!ok) break;
      }
    }
    if (tc::elect_one()) tc::mma_commit(&fin[0]);
    __syncwarp();
    if (lane == 0) drain_wait(&fin[0], 0, a.status);
    __syncwarp();
  } else if (warp == C::kPvWarp) {
    // ---------------------------------------------------------- PV issuer
    PieceSrc pi;
    pi.init(s_pieces, *s_npieces, a.sched, blockIdx.x, a.seq_lens);
    Piece pc;
    int pL = 0;
    uint32_t it = 0, npieces = 0, pos = 0;  // tiles, pieces, ring position
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      bool r = tc::mbar_wait(bar, parity, abort_flag, a.status, limit);
      ok = __all_sync(0xffffffffu, r) && ok;
    };
    while (ok && pi.next(pc, pL)) {
      const int nkeys = pL + a.T;
      pos += MT;  // the piece's query slots
      for (int j = pc.tile_begin; j < pc.tile_end; ++j, ++it, ++pos) {
        const uint32_t stage = pos % S;
        const bool first = j == pc.tile_begin;
        if (first && npieces > 0) {
          wait_all(o_free, (npieces - 1) & 1);
          if (!ok) break;
        }
        const int valid = nkeys - j * kTileKeys;
        if (valid < kTileKeys) {
          // slots past the sequence hold stale data (possibly NaN): zero the V
          // rows so that 0-probability columns contribute exactly 0
          wait_all(&full[stage], (pos / S) & 1);
          if (!ok) break;
          uint8_t* vbase = sKV + stage * C::kStageBytes + C::NH * C::kHalfTile;
          const int nvec = (kTileKeys - valid) * 8;
          for (int h = 0; h < C::NH; ++h)
            for (int e = lane; e < nvec; e += 32)
              reinterpret_cast<uint4*>(vbase + h * C::kHalfTile + valid * 128)[e] = make_uint4(0, 0, 0, 0);
          tc::fence_proxy_async_smem();
          __syncwarp();
        }
        const uint32_t v_u = sKV_u + stage * C::kStageBytes + C::NH * C::kHalfTile;
        for (int m = 0; m < MT; ++m) {
          const int pb = (int)(it % NPB);
          wait_all(&p_full[m * NPB + pb], (it / NPB) & 1);
          if (!ok) break;
          tc::tc_fence_after();
          const uint32_t d_t = tmem + C::o_col(m);
          const uint32_t p_u = sP_u + (m * NPB + pb) * C::kPTile;
          const uint64_t pd0 = tc::smem_desc(p_u, 16, 1024), vd0 = tc::smem_desc(v_u, C::kHalfTile, 1024);
          if (first) {
            if (tc::elect_one()) tc::mma_f16_ss<false>(d_t, pd0, vd0, kIdescPV);
          } else {
            if (tc::elect_one()) tc::mma_f16_ss<true>(d_t, pd0, vd0, kIdescPV);
          }
#pragma unroll
          for (int kk = 1; kk < kTileKeys / 16; ++kk)  // next 16 keys: P +32 B, V +2048 B
            if (tc::elect_one()) tc::mma_f16_ss<true>(d_t, pd0 + (uint64_t)(kk * 2), vd0 + (uint64_t)(kk * 128), kIdescPV);
          if (tc::elect_one()) tc::mma_commit(&pv_done[m * NPB + pb]);
          __syncwarp();
        }
        if (!ok) break;
        if (tc::elect_one()) tc::mma_commit(&empty[stage]);
        __syncwarp();
      }
      ++npieces;
    }
    if (tc::elect_one()) tc::mma_commit(&fin[1]);
    __syncwarp();
    if (lane == 0) drain_wait(&fin[1], 0, a.status);
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int m = warp >> 2;               // M tile of this warpgroup
    const int quad = warp & 3;             // TMEM lane quadrant
    const int r = quad * 32 + lane;        // row within the M tile
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const unsigned long long tmask = a.T == 64 ? ~0ull : ((1ull << a.T) - 1ull);
    const float scale = a.scale_log2;
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      bool rr = tc::mbar_wait(bar, parity, abort_flag, a.status, limit);
      ok = __all_sync(0xffffffffu, rr) && ok;
    };
    PieceSrc pi;
    pi.init(s_pieces, *s_npieces, a.sched, blockIdx.x, a.seq_lens);
    Piece pc;
    int L = 0;
    uint32_t it = 0;
    // this row's ancestor mask in piece (b, rg), tmask for rows past the end
    auto row_anc = [&](int b, int rg) -> unsigned long long {
      const int row = rg * kTcRows + m * 128 + r;
      return row < a.rows ? a.anc[(size_t)b * a.T + row / a.g] : tmask;
    };
    bool have_next = false;
    unsigned long long next_anc = 0ull;
    while (ok && pi.next(pc, L)) {
      const int row = pc.rg * kTcRows + m * 128 + r;
      const bool row_ok = row < a.rows;
      const int node = row_ok ? row / a.g : 0;
      const unsigned long long anc = have_next ? next_anc : row_anc(pc.b, pc.rg);
      // the next piece's mask is loaded now, long before it is needed
      const PieceRec* nx = pi.peek();
      have_next = nx != nullptr;
      if (have_next) next_anc = row_anc(nx->b, nx->rg);
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = pc.tile_begin; j < pc.tile_end; ++j, ++it) {
        const uint32_t s_addr = tmem + lane_addr + C::s_col(m);
        wait_all(&s_full[m], it & 1);
        if (!ok) break;
        tc::tc_fence_after();
        uint32_t sr[64];
        tc::tmem_ld_x64(s_addr, sr);
        tc::tmem_ld_wait();
        // the scores are in registers: S may take the next tile's scores
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&s_free[m]);
        const int k0 = j * kTileKeys;
        if (k0 + kTileKeys > L) {
          // the tile reaches past the prefix: tree mask and sequence end
          // halves wholly inside the prefix need nothing; only slots of the
          // tree part take the per-slot test
          const unsigned long long vis = tile_visibility(L, k0, anc);
#pragma unroll
          for (int hw = 0; hw < 2; ++hw) {
            const uint32_t bits = (uint32_t)(vis >> (32 * hw));
            if (bits == 0xffffffffu) continue;
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (!((bits >> c) & 1u)) sr[32 * hw + c] = 0xff800000u;  // -inf
          }
        }
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          mx0 = fmaxf(mx0, __uint_as_float(sr[c]));
          mx1 = fmaxf(mx1, __uint_as_float(sr[c + 1]));
          mx2 = fmaxf(mx2, __uint_as_float(sr[c + 2]));
          mx3 = fmaxf(mx3, __uint_as_float(sr[c + 3]));
        }
        const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * scale;
        // lazy rescale: the running max moves (and O in TMEM is rescaled) only
        // when the tile max exceeds it by more than 8, i.e. p <= 2^8 otherwise
        const bool grow = mx > m_run + 8.f;
        const bool need_o = grow && m_run != -INFINITY;
        const float m_new = grow ? mx : m_run;
        const float sc = need_o ? fast_exp2(m_run - m_new) : 1.f;
        const float neg_m = m_new == -INFINITY ? 0.f : -m_new;
        float rs0 = 0.f, rs1 = 0.f;
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(sr[2 * c]), scale, neg_m));
          const float p1 = fast_exp2(fmaf(__uint_as_float(sr[2 * c + 1]), scale, neg_m));
          rs0 += p0;
          rs1 += p1;
          pk[c] = Pack2<T>::pack(p0, p1);
        }
        // P into buffer it % NPB of this M tile, once the P.V of tile it - NPB
        // (which read it) is done: row r is 128 B (64 keys) in an 8-row,
        // 128-byte swizzle atom (16-byte chunk c at c ^ (r % 8)).  A
        // buffer's barriers complete once per use, and its next use needs
        // this thread's P, so neither runs two phases ahead of these waits
        const int pb = (int)(it % NPB);
        if (it >= (uint32_t)NPB) {
          wait_all(&pv_done[m * NPB + pb], ((it / NPB) - 1) & 1);
          if (!ok) break;
        }
        {
          uint8_t* prow = sP + (m * NPB + pb) * C::kPTile + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          tc::fence_proxy_async_smem();  // visible to the tensor core's reads
        }
        if (__any_sync(0xffffffffu, need_o)) {
          // O must hold the P.V sum up to tile it - 1 (with one buffer that
          // P.V was waited for above)
          if (NPB > 1) {
            wait_all(&pv_done[m * NPB + (int)((it - 1) % NPB)], ((it - 1) / NPB) & 1);
            if (!ok) break;
          }
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
        }
        tc::tmem_st_wait();
        l_run = l_run * sc + (rs0 + rs1);
        m_run = m_new;
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&p_full[m * NPB + pb]);
      }
      if (!ok) break;
      // epilogue, once the piece's last P.V is done
      wait_all(&pv_done[m * NPB + (int)((it - 1) % NPB)], ((it - 1) / NPB) & 1);
      if (!ok) break;
      tc::tc_fence_after();
      const int seg_row = m * 128 + r;
      // the output, or the piece's partial output O / l (the combine weighs it by
      // l), in the act dtype; an FP8 cache's V scale multiplies both
      const float vs = FP8 ? a.v_scale : 1.f;
      const float inv = (l_run > 0.f ? 1.f / l_run : 0.f) * vs;
#pragma unroll 1
      for (int hh = 0; hh < D / 64; ++hh) {
        uint32_t o[64];
        tc::tmem_ld_x64(tmem + lane_addr + C::o_col(m) + 64 * hh, o);
        tc::tmem_ld_wait();
        if (row_ok) {
          // 16-byte chunks of 8 columns: along the output row, or (a partial,
          // [slot][D/8][rows]) chunk-major, so that consecutive rows (threads)
          // write consecutive 16 B
          uint4* dst;
          size_t step;
          if (pc.slot < 0) {
            const int h = pc.kvh * a.g + row % a.g;
            dst = reinterpret_cast<uint4*>(static_cast<T*>(a.out) + (((size_t)pc.b * a.T + node) * a.Hq + h) * D +
                                           64 * hh);
            step = 1;
          } else {
            dst = static_cast<uint4*>(a.part_o) + ((size_t)pc.slot * (D / 8) + 8 * hh) * a.part_rows + seg_row;
            step = a.part_rows;
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            T v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = Act<T>::from_f(__uint_as_float(o[8 * c + e]) * inv);
            uint4 w;
            memcpy(&w, v, 16);
            dst[c * step] = w;
          }
        }
      }
      if (row_ok && pc.slot >= 0)
        a.part_ml[(size_t)pc.slot * a.part_rows + seg_row] = make_float2(m_run, l_run);
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(o_free);
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == C::kQkWarp) tc::tmem_dealloc(tmem, C::kTmemCols);
}

template <typename T, int D, int MT, bool FP8>
cudaError_t launch_t(const AttnParams& a, const CUtensorMap* tk, const CUtensorMap* tv,
                     const CUtensorMap* tq, cudaStream_t stream) {
  using C = Cfg<D, MT, FP8>;
  // the shared-memory opt-in, once per kernel instance and device (outside
  // the hot path of later calls)
  static std::atomic<bool> opted[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !opted[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(attn_tc_kernel<T, D, MT, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) opted[dev].store(true, std::memory_order_release);
  }
  return launch_pdl(attn_tc_kernel<T, D, MT, FP8>, dim3(a.sched.G), dim3(C::kThreads), (size_t)C::kSmemBytes,
                    stream, *tk, *tv, *tq, a);
}

template <typename T, bool FP8>
cudaError_t launch_dtype(const AttnParams& a, const CUtensorMap* tk, const CUtensorMap* tv,
                         const CUtensorMap* tq, cudaStream_t stream) {
  const bool one = a.rows <= 128;
  if (a.D == 64)
    return one ? launch_t<T, 64, 1, FP8>(a, tk, tv, tq, stream) : launch_t<T, 64, 2, FP8>(a, tk, tv, tq, stream);
  return one ? launch_t<T, 128, 1, FP8>(a, tk, tv, tq, stream) : launch_t<T, 128, 2, FP8>(a, tk, tv, tq, stream);
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

// An FP8 (E4M3) paged cache [num_pages][Hkv][16][D] of 1-byte codes as a 2-D
// tensor of num_pages*Hkv*16 rows by D columns; boxes of 16 rows (one page of
// one KV head) by D columns, no swizzle (the producers convert the codes into
// the swizzled stage), zero fill outside.
cudaError_t make_cache_tmap_e4m3(void* map_out, const void* base, int num_pages, int Hkv, int P, int D) {
  CUtensorMap* map = static_cast<CUtensorMap*>(map_out);
  auto enc = get_encode();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)num_pages * Hkv * P};
  cuuint64_t strides[1] = {(cuuint64_t)D};
  cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)P};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The rotated queries [B*T][Hq][D] as a 3-D tensor (D, Hq, B*T); a box of 64
// columns x g heads x 128/g nodes is one 128-row M tile half (row = node * g +
// head in group), 128-byte swizzle.  Rows past the last node read zeros.
cudaError_t make_q_tmap(void* map_out, const void* base, int dtype, int BT, int Hq, int g, int D) {
  auto enc = get_encode();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap* map = static_cast<CUtensorMap*>(map_out);
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)BT};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)g, (cuuint32_t)(128 / g)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dtype == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool tc_supported(int D, int g) { return (D == 64 || D == 128) && g >= 1 && g <= 128 && 128 % g == 0; }

cudaError_t launch_attn_tc(const AttnParams& a, int dtype, const void* tmap_k, const void* tmap_v,
                           const void* tmap_q, cudaStream_t stream) {
  const CUtensorMap* tk = static_cast<const CUtensorMap*>(tmap_k);
  const CUtensorMap* tv = static_cast<const CUtensorMap*>(tmap_v);
  const CUtensorMap* tq = static_cast<const CUtensorMap*>(tmap_q);
  if (a.cache_fp8) {
    if (dtype == 1) return launch_dtype<__half, true>(a, tk, tv, tq, stream);
    return launch_dtype<__nv_bfloat16, true>(a, tk, tv, tq, stream);
  }
  if (dtype == 1) return launch_dtype<__half, false>(a, tk, tv, tq, stream);
  return launch_dtype<__nv_bfloat16, false>(a, tk, tv, tq, stream);
}

}  // namespace mt
