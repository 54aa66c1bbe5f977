// block_rules.h -- per-block mask rules of the forward kernels (the ring's
// step kernel and its one-launch lap variant): for a query tile of shard r
// against K/V block j, which key tiles it visits, which of them need the
// element mask, and the per-row key bounds.  Included by the .cu files that
// use it; everything is device code in an anonymous namespace.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace ringattn {
namespace {

// ------------------------------------------------------------- work items
struct Tile {
  int t;                  // query tile index within the shard
  int jb, je;             // loop indices [jb, je) this tile computes
  int mask_lo, mask_from;  // loop indices below mask_lo or from mask_from take the mask
  int klim;               // mask: key k allowed iff kmin(i) <= k, k < klim and k <= kmax(i)
  int q;                  // kmax(i) = floor((i + b) / q); kmin(i) = floor((i + bl) / q) + 1
  long long b, bl;        // (bl very negative: no lower bound)
  // key-tile space, before decode_item makes them loop indices
  int kt_lo, kt_hi, full_lo, full_hi;
};

constexpr long long kNoLowerBound = -(1LL << 50);

__device__ __forceinline__ long long floor_div(long long x, int q) {
  return x >= 0 ? x / q : -((-x + q - 1) / q);
}
__device__ __forceinline__ long long tile_kmax(const Tile& w, long long i) {
  return w.q == 1 ? i + w.b : floor_div(i + w.b, w.q);
}
__device__ __forceinline__ long long tile_kmin(const Tile& w, long long i) {
  return (w.q == 1 ? i + w.bl : floor_div(i + w.bl, w.q)) + 1;
}

struct WorkItem {
  int bh, kvh, r, j, slot;  // kvh: the K/V head that query head bh reads
  int sr;                   // state slot of this CTA's rows: r, or r * ksplit + piece for split keys
  Tile tile[2];
  int lo, nk;          // loop index j < nk visits key tile lo + ((j + rot) mod nk)
  int rot;
  int ext0;            // loop indices from nk on load key tiles ext0, ext0 + 1, .. (sending only)
  int np_send;         // loop indices in all when the CTA sends
  int fwd_lo, fwd_hi;  // key tiles this CTA sends along the ring
};

__device__ __forceinline__ int key_tile(const StepArgs& a, const WorkItem& w, int j) {
  if (j >= w.nk) return w.ext0 + (j - w.nk);
  const int kt = j + w.rot;
  return w.lo + (kt >= w.nk ? kt - w.nk : kt);
}

// The mask rule of the block for the rows in half h of the shard (see the
// planner): kmax(i) = floor((i + b) / q) and, with a sliding window W,
// kmin(i) = floor((i + bl) / q) + 1; key limit klim.
template <bool kWin>
__device__ __forceinline__ void block_rule(const StepArgs& a, int r, int j, int h, Tile* w) {
  const long long n = a.n;
  w->klim = a.n;
  w->b = n;
  w->bl = kNoLowerBound;
  w->q = 1;
  if (!a.causal) return;
  const long long W = kWin ? a.window : 0;
  if (a.decode_pos0 >= 0) {
    // Short queries at global positions pos0 + i against the cache read as
    // one contiguous block (key k at position k): key k is allowed iff
    // k <= pos0 + i; a window drops positions W or more behind the query.
    w->b = a.decode_pos0;
    if (W > 0) w->bl = w->b - W;
    return;
  }
  if (a.layout == RING_LAYOUT_ZIGZAG) {
    if (j < r) {
      w->klim = a.n / 2;
    } else if (j == r) {
      w->b = 0;
    } else if (h == 0) {
      w->klim = 0;
    }
    return;
  }
  // contiguous: pos_q - pos_k = (r - j) n + i - k; striped: (i - k) P + (r - j)
  const bool striped = a.layout == RING_LAYOUT_STRIPED;
  const long long dl = striped ? (j <= r ? 0 : -1) : (long long)(r - j) * n;
  if (dl <= -n) {
    w->klim = 0;
  } else if (dl < n - 1) {
    w->b = dl;
  }
  if (W > 0) w->bl = striped ? floor_div((long long)(r - j) - W, a.P) : (long long)(r - j) * n - W;
}

// Sequence packing: the keys of block j that local query row i of shard r
// may see lie in its document [ds, de) of natural positions.  Keys of block
// j sit at j n + k (contiguous) or k P + j (striped); queries at r n + i,
// i P + r, or pos0 + i for short queries.  Inclusive local key bounds.
__device__ __forceinline__ void seg_bounds(const StepArgs& a, int r, int j, long long i, long long& lo,
                                           long long& hi) {
  const long long pos = a.decode_pos0 >= 0 ? a.decode_pos0 + i
                                           : (a.layout == RING_LAYOUT_STRIPED ? i * a.P + r : (long long)r * a.n + i);
  const long long ds = a.seg_lo[pos], de = a.seg_hi[pos];
  if (a.layout == RING_LAYOUT_STRIPED) {
    lo = floor_div(ds - j + a.P - 1, a.P);
    hi = floor_div(de - 1 - j, a.P);
  } else {
    lo = ds - (long long)j * a.n;
    hi = de - 1 - (long long)j * a.n;
  }
}

// Zigzag with a sliding window or documents.  A shard (or a
// block) holds chunk r then chunk 2P-1-r of c = n/2 tokens, so its positions
// increase with the local index; the positions a query may see form one
// interval [L, U] (causal: up to itself; a window: from W-1 tokens back; a
// document: inside it), so its keys in a block form one local interval.
// zz_local_interval maps [L, U] to that interval [lo, hi] (lo > hi: none)
// for the chunks starting at positions A0 < B0.
__device__ __forceinline__ void zz_local_interval(long long c, long long A0, long long B0, long long L,
                                                  long long U, long long& lo, long long& hi) {
  hi = U >= B0 ? c + min(U - B0, c - 1) : (U >= A0 ? min(U - A0, c - 1) : -1);
  lo = L <= A0 ? 0 : (L < A0 + c ? L - A0 : (L <= B0 ? c : (L < B0 + c ? c + L - B0 : 2 * c)));
}

// Global position of local query row i of zigzag shard r.
__device__ __forceinline__ long long zz_query_pos(const StepArgs& a, int r, long long i) {
  const long long c = a.n / 2;
  return i < c ? (long long)r * c + i : (long long)(2 * a.P - 1 - r) * c + (i - c);
}

// The keys of zigzag block j (local, inclusive) that the query at position t may see.
__device__ __forceinline__ void zz_key_bounds(const StepArgs& a, int j, long long t, long long& lo, long long& hi) {
  const long long c = a.n / 2;
  long long L = 0, U = (long long)a.n * a.P - 1;
  if (a.causal) {
    U = t;
    if (a.window > 0) L = t - a.window + 1;
  }
  if (a.seg_lo) {
    L = max(L, (long long)a.seg_lo[t]);
    U = min(U, (long long)a.seg_hi[t] - 1);
  }
  zz_local_interval(c, (long long)j * c, (long long)(2 * a.P - 1 - j) * c, L, U, lo, hi);
}

template <bool kWin>
__device__ __forceinline__ Tile tile_work(const StepArgs& a, int r, int j, int t) {
  Tile w{};
  w.t = t;
  w.q = 1;
  if (t >= a.T) return w;
  const long long n = a.n;
  const long long i_min = (long long)t * kTileM;
  const long long i_max = min((long long)a.nq - 1, i_min + kTileM - 1);
  long long last_key, first_key, common_hi, common_lo;
  if (kWin && a.layout == RING_LAYOUT_ZIGZAG) {
    // per-row bounds from positions (row_key_bounds); the tile's rows have
    // consecutive positions, so the bounds are non-decreasing over it
    w.klim = a.n;
    w.b = n;
    w.bl = kNoLowerBound;
    long long lo0, hi0, lo1, hi1;
    zz_key_bounds(a, j, zz_query_pos(a, r, i_min), lo0, hi0);
    zz_key_bounds(a, j, zz_query_pos(a, r, i_max), lo1, hi1);
    last_key = min(n - 1, hi1);
    first_key = max(0LL, lo0);
    common_hi = min(n, hi0 + 1);
    common_lo = max(0LL, lo1);
  } else {
    const int h = (a.layout == RING_LAYOUT_ZIGZAG && i_min >= n / 2) ? 1 : 0;
    block_rule<kWin>(a, r, j, h, &w);
    // kmin and kmax are non-decreasing in i: the last row bounds the tiles
    // from above, the first row from below, and the tiles every row may use
    // in full lie between the first row's kmax and the last row's kmin.
    last_key = min((long long)w.klim - 1, tile_kmax(w, i_max));
    first_key = kWin ? max(0LL, tile_kmin(w, i_min)) : 0;
    common_hi = min((long long)w.klim, tile_kmax(w, i_min) + 1);  // keys < this for every row
    common_lo = kWin ? max(0LL, tile_kmin(w, i_max)) : 0;          // keys >= this for every row
  }
  if (kWin && a.seg_lo && a.layout != RING_LAYOUT_ZIGZAG) {
    // the document bounds are non-decreasing in i too
    long long lo0, hi0, lo1, hi1;
    seg_bounds(a, r, j, i_min, lo0, hi0);
    seg_bounds(a, r, j, i_max, lo1, hi1);
    first_key = max(first_key, lo0);
    last_key = min(last_key, hi1);
    common_lo = max(common_lo, lo1);
    common_hi = min(common_hi, hi0 + 1);
  }
  w.kt_hi = last_key < 0 ? 0 : (int)min((long long)a.KT, last_key / kTileN + 1);
  w.kt_lo = (int)min((long long)w.kt_hi, first_key / kTileN);
  w.full_hi = common_hi <= 0 ? 0 : (int)min((long long)w.kt_hi, common_hi / kTileN);
  w.full_lo = (int)min((long long)w.kt_hi, (common_lo + kTileN - 1) / kTileN);
  return w;
}

// This row's allowed keys [kmin_row, kmax_row] of block j (tw: its tile's
// rule from tile_work); kmin_row is 0 without row-dependent lower bounds.
template <bool kWin>
__device__ __forceinline__ void row_key_bounds(const StepArgs& a, const Tile& tw, int r, int j, long long i_row,
                                               int& kmin_row, int& kmax_row) {
  if (kWin && a.layout == RING_LAYOUT_ZIGZAG) {
    long long lo, hi;
    zz_key_bounds(a, j, zz_query_pos(a, r, min(i_row, (long long)a.nq - 1)), lo, hi);
    kmin_row = (int)max(0LL, min((long long)a.n, lo));
    kmax_row = (int)max(-1LL, min((long long)a.n - 1, hi));
    return;
  }
  kmax_row = (int)max(-1LL, min((long long)tw.klim - 1, tile_kmax(tw, i_row)));
  kmin_row = kWin ? (int)max(0LL, min((long long)a.n, tile_kmin(tw, i_row))) : 0;
  if (kWin && a.seg_lo) {
    long long slo, shi;
    seg_bounds(a, r, j, min(i_row, (long long)a.nq - 1), slo, shi);
    kmin_row = max(kmin_row, (int)max(0LL, min((long long)a.n, slo)));
    kmax_row = min(kmax_row, (int)max(-1LL, min((long long)a.n, shi)));
  }
}

}  // namespace
}  // namespace ringattn
