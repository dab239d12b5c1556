// Shared device-side definitions of the Medusa tree-verification kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace mt {

constexpr int kTileKeys = 64;   // logical slots per attention key tile
constexpr int kMaxTree = 64;    // one uint64 ancestor mask per node

// Device status codes (match mt_status in the public header).
enum : int { kStOk = 0, kStTree = -3, kStPages = -4, kStTimeout = -6 };

// First error wins; later ones are dropped.
__device__ __forceinline__ void set_status(int* status, int code) { atomicCAS(status, 0, code); }

// ---------------------------------------------------------------------------
// act dtype traits: exact widening to fp32, round-to-nearest-even narrowing.
// ---------------------------------------------------------------------------
template <typename T> struct Act;
template <> struct Act<float> {
  static __device__ __forceinline__ float to_f(float x) { return x; }
  static __device__ __forceinline__ float from_f(float x) { return x; }
};
template <> struct Act<__half> {
  static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};
template <> struct Act<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// RoPE on one (j, j + D/2) pair, each product and difference rounded on its
// own (no fused multiply-add), so the result is bit-identical to the plain
// fp32 definition: lo' = lo*c - hi*s, hi' = hi*c + lo*s.
__device__ __forceinline__ void rope_pair(float lo, float hi, float c, float s, float& out_lo,
                                          float& out_hi) {
  out_lo = __fsub_rn(__fmul_rn(lo, c), __fmul_rn(hi, s));
  out_hi = __fadd_rn(__fmul_rn(hi, c), __fmul_rn(lo, s));
}

// ---------------------------------------------------------------------------
// Work schedule shared by the prep, attention and combine kernels.
//
// A segment is (sequence b, KV head, row group): the rows_per_group query rows
// (node i, head-in-group hh) -> row i*g + hh of one KV head, against the
// sequence's n_b = L_b + T logical key slots, cut into ceil(n_b / 64) tiles.
// Segments are numbered b-major: s = (b * Hkv + kvh) * nrg + rg, and the tiles
// of all segments form one global list in that order.  tile_pfx[b] is the
// number of tiles of one segment of every sequence before b (so sequence b's
// segments start at tile_pfx[b] * Hkv * nrg).
//
// splits == 0 (balanced): the tiles are dealt out evenly in cost, where a
//   segment costs its tiles plus seg_cost (the fixed work of starting a
//   piece: loading its queries, writing its result, refilling the pipeline,
//   in tile units).  Tile t of segment s sits at cost x(t) = t + seg_cost *
//   (s + 1); of the total X = W + seg_cost * nseg, CTA c of G takes the tiles
//   with x in [c*X/G, (c+1)*X/G), a contiguous run of the global list, so a
//   CTA whose run crosses several short segments gets fewer tiles.
//   The part of one segment that a CTA takes is a piece; a piece that is a
//   whole segment writes the output directly, any other piece writes a
//   partial result to slot s + c (unique: CTAs touching a later segment never
//   have a smaller index).
// splits == n > 0: segment s is cut into n key chunks of equal tile counts;
//   chunk k is a piece with partial slot s*n + k (direct output when n == 1);
//   the U = nseg*n pieces are dealt to CTAs in contiguous runs.
// ---------------------------------------------------------------------------
struct Sched {
  int B, T, Hkv, nrg, G, splits;
  int seg_cost;         // balanced mode: per-segment overhead in tile units
  const int* tile_pfx;  // [B + 1]
};

struct Piece {
  int b, kvh, rg, seg;
  int tile_begin, tile_end;  // tiles of the segment covered by this piece
  int slot;                  // partial slot, or -1 for a direct write
};

// The schedule's arithmetic is written over an index type I: 64-bit in the
// attention kernels, and 32-bit in the prep kernel's table walk once it has
// checked that the total cost times (G + 1) fits in 31 bits (every product
// and quotient below is then the same in either type).
template <typename I = long long>
__device__ __forceinline__ I sched_total_tiles(const Sched& s) {
  return (I)s.tile_pfx[s.B] * s.Hkv * s.nrg;
}

// Largest b with tile_pfx[b] * HR <= t (the sequence owning global tile t).
template <typename I>
__device__ __forceinline__ int sched_find_seq(const Sched& s, I t) {
  const I HR = (I)s.Hkv * s.nrg;
  int lo = 0, hi = s.B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((I)s.tile_pfx[mid] * HR <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Balanced mode: total cost, cost of a global tile, and the first global
// tile at or past a cost (the total tile count W when there is none).
template <typename I = long long>
__device__ __forceinline__ I sched_total_cost(const Sched& s) {
  return sched_total_tiles<I>(s) + (I)s.seg_cost * s.B * s.Hkv * s.nrg;
}

__device__ __forceinline__ long long sched_tile_cost(const Sched& s, long long t, long long seg) {
  return t + (long long)s.seg_cost * (seg + 1);
}

template <typename I>
__device__ __forceinline__ I sched_first_tile_at(const Sched& s, I y) {
  const I HR = (I)s.Hkv * s.nrg;
  // sequence b's segments start at cost tile_pfx[b] * HR + seg_cost * HR * b
  int lo = 0, hi = s.B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((I)s.tile_pfx[mid] * HR + (I)s.seg_cost * HR * mid <= y) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const I base = (I)s.tile_pfx[b] * HR + (I)s.seg_cost * HR * b;
  const I nt = s.tile_pfx[b + 1] - s.tile_pfx[b];
  const I per = nt + s.seg_cost;  // cost of one segment of sequence b
  const I off = y > base ? y - base : 0;
  if (per == 0) return (I)s.tile_pfx[b] * HR;
  const I k = off / per;
  if (k >= HR) return (I)s.tile_pfx[b + 1] * HR;
  const I r = off % per;
  const I j = r < s.seg_cost ? 0 : r - s.seg_cost;
  return (I)s.tile_pfx[b] * HR + k * nt + j;
}

// CTA whose cost range holds cost x in balanced mode (X the total cost).
__device__ __forceinline__ int sched_cta_of(long long x, long long X, int G) {
  return (int)(((x + 1) * (long long)G - 1) / X);
}

// Iterator over the pieces of one CTA.
template <typename I>
struct PieceIterT {
  Sched s;
  int cta;
  I cur, end;  // balanced: global tile cursor; split mode: unit cursor
  I W;
  int bcur;    // balanced: the sequence owning cur, once found (-1 before)

  __device__ void init(const Sched& sc, int c) {
    s = sc;
    cta = c;
    bcur = -1;
    if (s.splits == 0) {
      W = sched_total_tiles<I>(s);
      const I X = sched_total_cost<I>(s);
      cur = sched_first_tile_at<I>(s, X * c / s.G);
      end = sched_first_tile_at<I>(s, X * (c + 1) / s.G);
    } else {
      W = (I)s.B * s.Hkv * s.nrg * s.splits;
      cur = W * c / s.G;
      end = W * (c + 1) / s.G;
    }
  }

  // Returns false when the CTA has no more work.
  __device__ bool next(Piece& p) {
    const I HR = (I)s.Hkv * s.nrg;
    while (cur < end) {
      if (s.splits == 0) {
        // the cursor only moves forward: after the first search, step to the
        // largest sequence whose segments start at or before it
        if (bcur < 0) bcur = sched_find_seq<I>(s, cur);
        else
          while (bcur + 1 < s.B && (I)s.tile_pfx[bcur + 1] * HR <= cur) ++bcur;
        const int b = bcur;
        int nt = s.tile_pfx[b + 1] - s.tile_pfx[b];
        I local = cur - (I)s.tile_pfx[b] * HR;
        int seg_in_b = (int)(local / nt);
        int j0 = (int)(local % nt);
        I seg_begin = cur - j0;
        I seg_end = seg_begin + nt;
        I stop = end < seg_end ? end : seg_end;
        p.b = b;
        p.kvh = seg_in_b / s.nrg;
        p.rg = seg_in_b % s.nrg;
        p.seg = (int)((I)b * HR + seg_in_b);
        p.tile_begin = j0;
        p.tile_end = j0 + (int)(stop - cur);
        p.slot = (j0 == 0 && stop == seg_end) ? -1 : p.seg + cta;
        cur = stop;
        return true;
      } else {
        I u = cur++;
        int k = (int)(u % s.splits);
        int seg = (int)(u / s.splits);
        int b = (int)(seg / HR);
        int nt = s.tile_pfx[b + 1] - s.tile_pfx[b];
        int j0 = (int)((I)nt * k / s.splits);
        int j1 = (int)((I)nt * (k + 1) / s.splits);
        if (j0 >= j1) continue;
        int seg_in_b = (int)(seg - (I)b * HR);
        p.b = b;
        p.kvh = seg_in_b / s.nrg;
        p.rg = seg_in_b % s.nrg;
        p.seg = seg;
        p.tile_begin = j0;
        p.tile_end = j1;
        p.slot = s.splits == 1 ? -1 : seg * s.splits + k;
        return true;
      }
    }
    return false;
  }
};
using PieceIter = PieceIterT<long long>;

// Arguments shared by both attention kernels and the combine kernel.
struct AttnParams {
  int B, T, Hq, Hkv, D, P, max_blocks, num_pages, g;
  int rows;            // T * g query rows per (b, kvh)
  int rows_per_group;  // RG: query rows per segment (row group)
  int part_rows;       // rows per partial slot: min(rows, RG)
  float scale_log2;    // sm_scale * log2(e)
  const void* q_rot;   // [B][T][Hq][D] act, rotated and rounded (written by prep)
  const void* k_cache;
  const void* v_cache;
  const int* block_tables;
  const int* seq_lens;
  const int* tree_depths;
  void* out;
  int* status;
  const unsigned long long* anc;  // [B][T]
  void* part_o;                   // [slots][D/8][part_rows] entries of 8 act values: O / l of the piece
  float2* part_ml;                // [slots][part_rows] (max in log2 units, sum)
  Sched sched;
  const int* piece_table;         // count[G], padded, + PieceRec[G][kMaxPieceRecs] (tensor-core kernel)
  unsigned long long wait_limit_ns;  // bound of every pipeline wait (tensor-core kernel)
  int test_stall;                    // tensor-core kernel: first wait on a barrier nothing completes
  int cache_fp8;                     // tensor-core kernel: the caches hold E4M3 codes of value / scale
  float v_scale;                     // their V scale (the K scale is folded into scale_log2)
};

// A CTA's pieces, listed ahead of time by the prep kernel (up to
// kMaxPieceRecs; more is recorded as a count of -1), with the sequence's
// prefix length, so that the attention kernel starts a piece without
// dependent global loads.  Table layout: int count[G] (padded to a multiple
// of 4), then PieceRec rec[G][kMaxPieceRecs], 16-byte aligned when the table
// is.
constexpr int kMaxPieceRecs = 32;

struct __align__(16) PieceRec {
  int b, kvh, rg, seg, tile_begin, tile_end, slot, L;
};

// Offset of the records in the table, in ints.
__host__ __device__ __forceinline__ int piece_rec_offset(int G) { return (G + 3) & ~3; }

// Pieces from a shared-memory copy of the table, or from the schedule itself
// when the table overflowed (n < 0).
struct PieceSrc {
  const PieceRec* rec;
  int n, idx;
  PieceIter iter;
  const int* seq_lens;

  __device__ __forceinline__ void init(const PieceRec* r, int count, const Sched& s, int cta, const int* lens) {
    rec = r;
    n = count;
    idx = 0;
    seq_lens = lens;
    if (n < 0) iter.init(s, cta);
  }
  __device__ __forceinline__ bool next(Piece& p, int& L) {
    if (n >= 0) {
      if (idx >= n) return false;
      const PieceRec& r = rec[idx++];
      p.b = r.b;
      p.kvh = r.kvh;
      p.rg = r.rg;
      p.seg = r.seg;
      p.tile_begin = r.tile_begin;
      p.tile_end = r.tile_end;
      p.slot = r.slot;
      L = r.L;
      return true;
    }
    if (!iter.next(p)) return false;
    L = seq_lens[p.b];
    return true;
  }
  // The record after the one last returned (table mode only), or null.
  __device__ __forceinline__ const PieceRec* peek() const { return n >= 0 && idx < n ? &rec[idx] : nullptr; }
};

// Page ids of one sequence's block table as seen by a TMA producer warp.  The
// warp fetches 32 consecutive entries (eight 64-slot tiles of 16-slot pages)
// with one coalesced load, and the following 32 are already in flight while
// the current ones are used, so issuing a tile's copies never waits on a
// global load.  Entries at or past the sequence's last slot, or past the
// table's width, read as -1.  Every lane of the warp must call page() with the
// same, non-decreasing page index.
struct PageWindow {
  const int* bt;
  int nkeys, max_blocks, base, cur, nxt;

  __device__ __forceinline__ int fetch(int first, int lane) const {
    const int q = first + lane;
    return (q < max_blocks && q * 16 < nkeys) ? __ldg(bt + q) : -1;
  }
  __device__ __forceinline__ void init(const int* bt_, int nkeys_, int max_blocks_, int first_page, int lane) {
    bt = bt_;
    nkeys = nkeys_;
    max_blocks = max_blocks_;
    base = first_page;
    cur = fetch(base, lane);
    nxt = fetch(base + 32, lane);
  }
  __device__ __forceinline__ int page(int pg, int lane) {
    while (pg - base >= 32) {
      cur = nxt;
      base += 32;
      nxt = fetch(base + 32, lane);
    }
    return __shfl_sync(0xffffffffu, cur, pg - base);
  }
};

}  // namespace mt
