// planner.cpp -- host-side layout and mask planner (no GPU).
//
// For every ring step s and shard r it records the block j = (r - s) mod P
// that shard r holds ([GRA] "One lap around the ring"; [RA-CN] "环是怎样工作的"),
// the block's class under the causal mask ([RA-CN] "Causal Attention
// 让环不再完全对称": skip a strictly-future block, mask a block crossing the
// diagonal, run the rest unmasked) and the diagonal offset used for the mask,
// plus per-shard and per-step work counts ([GRA] "The causal mask wrecks the
// load balance"; [RA-CN] "如何判断通信是否真的被覆盖": valid/skipped blocks).
#include <algorithm>
#include <cstdio>

#include "internal.h"

namespace ringattn {

int block_of(int P, int r, int step) {
  int j = (r - step) % P;
  return j < 0 ? j + P : j;
}

static long long floor_div(long long x, long long q) { return x >= 0 ? x / q : -((-x + q - 1) / q); }

BlockPlan classify(int layout, int causal, long long n, int r, int j, int P, long long window) {
  BlockPlan b{j, RING_BLOCK_FULL, n, {n, n}, {n, n}, kNoLowerOffset};
  if (!causal) return b;
  if (window > 0 && layout != RING_LAYOUT_ZIGZAG) {
    // (zigzag windows: zz_key_bounds) a key W or more positions behind the query is dropped: contiguous
    // (r-j) n + i - k < W  <=>  k - i >= (r-j) n - W + 1; striped
    // (i-k) P + (r-j) < W  <=>  k - i >= floor((r-j-W)/P) + 1
    b.lodelta = layout == RING_LAYOUT_STRIPED ? floor_div((long long)(r - j) - window, P) + 1
                                              : (long long)(r - j) * n - window + 1;
  }
  if (layout == RING_LAYOUT_ZIGZAG) {
    // Shard r holds chunks r and 2P-1-r (c = n/2 tokens each), rows in that
    // order; block j likewise.  Comparing chunk ids (all of r, j < P <= the
    // late chunks): early rows see block j's early chunk entirely if j < r,
    // up to the diagonal if j = r, never if j > r, and never its late chunk;
    // late rows see the early chunk entirely, and the late chunk entirely
    // if j > r, up to the diagonal if j = r, never if j < r.  In block
    // columns that is k < c for both halves (j < r), k - i <= 0 (j = r; for
    // a late row it also admits the whole early chunk), and for j > r
    // nothing for early rows and everything for late ones.
    const long long c = n / 2;
    if (j < r) {
      b.klim[0] = b.klim[1] = c;
      b.cls = RING_BLOCK_PARTIAL;
    } else if (j == r) {
      b.hdelta[0] = b.hdelta[1] = b.delta = 0;
      b.cls = RING_BLOCK_DIAG;
    } else {
      b.klim[0] = 0;
      b.cls = RING_BLOCK_PARTIAL;
    }
    return b;
  }
  if (layout == RING_LAYOUT_STRIPED) {
    // token positions i*P + r (queries) and k*P + j (keys): k*P + j <= i*P + r
    // <=> k - i <= 0 when j <= r, and k - i <= -1 when j > r.
    b.delta = (j <= r) ? 0 : -1;
  } else {
    b.delta = (long long)(r - j) * n;
  }
  if (b.delta >= n - 1) {
    b.cls = RING_BLOCK_FULL;  // the offset admits every pair: no diagonal
  } else if (b.delta <= -n) {
    b.cls = RING_BLOCK_SKIP;
    b.klim[0] = b.klim[1] = 0;
  } else {
    b.cls = RING_BLOCK_DIAG;
  }
  b.hdelta[0] = b.hdelta[1] = b.delta;
  return b;
}

long long block_pairs(int layout, long long n, const BlockPlan& b) {
  // row i allows columns max(0, i + lodelta) .. min(klim, i + hdelta + 1) - 1
  long long total = 0;
  for (long long i = 0; i < n; ++i) {
    const int h = row_half(layout, n, i);
    const long long hi = std::min(b.klim[h], std::max(0LL, i + b.hdelta[h] + 1));
    const long long lo = std::max(0LL, i + b.lodelta);
    total += std::max(0LL, hi - lo);
  }
  return total;
}

void tile_range(int layout, long long n, int KT, const BlockPlan& b, int t, int* nk, int* full_kt) {
  // The rows of a tile are in one half (the zigzag layout needs n/2 to be a
  // multiple of the tile), so one (klim, hdelta) rule covers the tile.
  const long long i_min = (long long)t * kTileM;
  const long long i_max = std::min(n - 1, i_min + kTileM - 1);
  const int h = row_half(layout, n, i_min);
  const long long klim = b.klim[h], hd = b.hdelta[h];
  const long long last_key = std::min(klim - 1, i_max + hd);  // largest allowed key of the tile
  int cnt = last_key < 0 ? 0 : (int)std::min<long long>(KT, last_key / kTileN + 1);
  // key tiles allowed for every row of the tile: below klim and i_min + hd
  const long long common = std::min(klim, i_min + hd + 1);
  // a sliding window starts the tile's keys at i_min + lodelta
  const int first = (int)std::min<long long>(cnt, std::max(0LL, i_min + b.lodelta) / kTileN);
  *nk = cnt - first;  // key tiles visited
  *full_kt = common <= 0 ? 0 : (int)std::min<long long>(cnt, common / kTileN);
}

void seg_key_bounds(const Plan& p, int r, int j, long long i, long long* lo, long long* hi) {
  // the query's document [ds, de); keys of block j at j n + k (contiguous)
  // or k P + j (striped)
  const long long pos = p.layout == RING_LAYOUT_STRIPED ? i * p.P + r : (long long)r * p.n + i;
  const long long ds = p.seg_lo[(size_t)pos], de = p.seg_hi[(size_t)pos];
  if (p.layout == RING_LAYOUT_STRIPED) {
    *lo = floor_div(ds - j + p.P - 1, p.P);
    *hi = floor_div(de - 1 - j, p.P);
  } else {
    *lo = ds - (long long)j * p.n;
    *hi = de - 1 - (long long)j * p.n;
  }
}

// Zigzag with a window or documents.  Shard r and block j each hold chunk
// x then chunk 2P-1-x (c = n/2 tokens), positions increasing with the local
// index, so the positions a query may see ([t - W + 1, t] under the causal
// mask and a window, cut to its document) are one interval of block keys.
// Local keys lo..hi of block j that the query at position t may see.
void zz_key_bounds(const Plan& p, int j, long long t, long long* lo, long long* hi) {
  const long long c = p.n / 2;
  long long L = 0, U = p.N - 1;
  if (p.causal) {
    U = t;
    if (p.window > 0) L = t - p.window + 1;
  }
  if (!p.seg_lo.empty()) {
    L = std::max(L, (long long)p.seg_lo[(size_t)t]);
    U = std::min(U, (long long)p.seg_hi[(size_t)t] - 1);
  }
  const long long A0 = (long long)j * c, B0 = (long long)(2 * p.P - 1 - j) * c;
  *hi = U >= B0 ? c + std::min(U - B0, c - 1) : (U >= A0 ? std::min(U - A0, c - 1) : -1);
  *lo = L <= A0 ? 0 : (L < A0 + c ? L - A0 : (L <= B0 ? c : (L < B0 + c ? c + L - B0 : 2 * c)));
}

long long zz_position(const Plan& p, int r, long long i) {
  const long long c = p.n / 2;
  return i < c ? (long long)r * c + i : (long long)(2 * p.P - 1 - r) * c + (i - c);
}

// Allowed pairs and computed tiles of zigzag block (r, j) under those bounds.
static std::pair<long long, long long> zigzag_work(const Plan& p, int r, int j) {
  const long long n = p.n;
  long long pairs = 0, tiles = 0;
  for (long long i = 0; i < n; ++i) {
    long long lo, hi;
    zz_key_bounds(p, j, zz_position(p, r, i), &lo, &hi);
    pairs += std::max(0LL, hi - lo + 1);
  }
  for (int t = 0; t < p.T; ++t) {
    const long long i_min = (long long)t * kTileM, i_max = std::min(n - 1, i_min + kTileM - 1);
    long long lo0, hi0, lo1, hi1;
    zz_key_bounds(p, j, zz_position(p, r, i_min), &lo0, &hi0);
    zz_key_bounds(p, j, zz_position(p, r, i_max), &lo1, &hi1);
    const long long first = std::max(0LL, lo0), last = std::min(n - 1, hi1);
    if (first <= last) tiles += last / kTileN - first / kTileN + 1;
  }
  return {pairs, tiles};
}

// Allowed pairs and computed 128x128 tiles of block (r, j) with segments:
// row i allows columns max(0, i + lodelta, slo(i)) .. min(klim, i + hdelta
// + 1, shi(i) + 1) - 1; the bounds are non-decreasing in i, so a tile's key
// tiles run from its first row's lower bound to its last row's upper bound.
static std::pair<long long, long long> segment_work(const Plan& p, const BlockPlan& b, int r) {
  const long long n = p.n;
  long long pairs = 0, tiles = 0;
  auto lo_of = [&](long long i) {
    long long slo, shi;
    seg_key_bounds(p, r, b.j, i, &slo, &shi);
    return std::max({0LL, i + b.lodelta, slo});
  };
  auto hi_of = [&](long long i) {  // exclusive
    long long slo, shi;
    seg_key_bounds(p, r, b.j, i, &slo, &shi);
    return std::min({b.klim[0], std::max(0LL, i + b.hdelta[0] + 1), shi + 1});
  };
  for (long long i = 0; i < n; ++i) pairs += std::max(0LL, hi_of(i) - lo_of(i));
  for (int t = 0; t < p.T; ++t) {
    const long long i_min = (long long)t * kTileM, i_max = std::min(n - 1, i_min + kTileM - 1);
    const long long last = std::min<long long>(hi_of(i_max), n) - 1;
    if (last < 0) continue;
    const long long first = std::min(lo_of(i_min), last + 1);
    if (first > last) continue;
    tiles += last / kTileN - first / kTileN + 1;
  }
  return {pairs, tiles};
}

int build_plan(Plan* p, int B, int H, long long N, int d, int P, int causal, int layout,
               std::string* err, long long window, const std::vector<long long>* segments) {
  char buf[256];
  if (B <= 0 || H <= 0 || N <= 0 || d <= 0 || P <= 0) {
    std::snprintf(buf, sizeof buf, "sizes must be positive (B=%d H=%d N=%lld d=%d P=%d)", B, H, N, d, P);
    *err = buf;
    return RING_ERR_INVALID_ARG;
  }
  if (causal != 0 && causal != 1) {
    *err = "causal must be 0 or 1";
    return RING_ERR_INVALID_ARG;
  }
  if (layout != RING_LAYOUT_CONTIGUOUS && layout != RING_LAYOUT_STRIPED && layout != RING_LAYOUT_ZIGZAG) {
    *err = "layout must be RING_LAYOUT_CONTIGUOUS, RING_LAYOUT_STRIPED or RING_LAYOUT_ZIGZAG";
    return RING_ERR_INVALID_ARG;
  }
  if ((long long)P > N) {
    std::snprintf(buf, sizeof buf, "P=%d exceeds N=%lld", P, N);
    *err = buf;
    return RING_ERR_INVALID_ARG;
  }
  if (P > kMaxShards) {
    std::snprintf(buf, sizeof buf, "P=%d exceeds the supported maximum %d", P, kMaxShards);
    *err = buf;
    return RING_ERR_UNSUPPORTED;
  }
  if (N % P != 0) {
    std::snprintf(buf, sizeof buf, "N=%lld is not a multiple of P=%d (padding is not supported)", N, P);
    *err = buf;
    return RING_ERR_UNSUPPORTED;
  }
  if (d != 64 && d != 128) {
    std::snprintf(buf, sizeof buf, "head dim d=%d unsupported (64 or 128)", d);
    *err = buf;
    return RING_ERR_UNSUPPORTED;
  }
  const long long n = N / P;
  const long long bh = (long long)B * H;
  if (window < 0 || (window > 0 && !causal)) {
    *err = "a sliding window needs the causal mask";
    return window < 0 ? RING_ERR_INVALID_ARG : RING_ERR_UNSUPPORTED;
  }
  if (layout == RING_LAYOUT_ZIGZAG && (n % (2 * kTileM)) != 0) {
    std::snprintf(buf, sizeof buf,
                  "zigzag needs chunks N/2P that are multiples of %d tokens (N=%lld, P=%d)", kTileM, N, P);
    *err = buf;
    return RING_ERR_UNSUPPORTED;
  }
  if (n > (1LL << 30) || bh > (1LL << 30)) {
    *err = "shard length or B*H too large";
    return RING_ERR_UNSUPPORTED;
  }
  const bool packed = segments && !segments->empty();
  if (packed) {
    const std::vector<long long>& sb = *segments;
    bool ok = sb.size() >= 2 && sb.front() == 0 && sb.back() == N;
    for (size_t x = 1; ok && x < sb.size(); ++x) ok = sb[x] > sb[x - 1];
    if (!ok) {
      *err = "segment boundaries must rise strictly from 0 to N";
      return RING_ERR_INVALID_ARG;
    }
    if (N > (1LL << 31) - 1) {
      *err = "segments need N < 2^31";
      return RING_ERR_UNSUPPORTED;
    }
  }
  p->B = B;
  p->H = H;
  p->N = N;
  p->d = d;
  p->P = P;
  p->causal = causal;
  p->layout = layout;
  p->Hkv = H;
  p->window = window;
  p->n = n;
  p->T = (int)((n + kTileM - 1) / kTileM);
  p->KT = (int)((n + kTileN - 1) / kTileN);
  p->blocks.assign((size_t)P * P, BlockPlan{});
  p->shard_pairs.assign(P, 0);
  p->shard_tiles.assign(P, 0);
  p->step_pairs.assign(P, 0);
  p->step_tiles.assign(P, 0);
  p->active.assign(P, {});
  p->seg_bounds.clear();
  p->seg_lo.clear();
  p->seg_hi.clear();
  if (packed) {
    p->seg_bounds = *segments;
    p->seg_lo.resize((size_t)N);
    p->seg_hi.resize((size_t)N);
    for (size_t x = 0; x + 1 < segments->size(); ++x)
      for (long long t = (*segments)[x]; t < (*segments)[x + 1]; ++t) {
        p->seg_lo[(size_t)t] = (int)(*segments)[x];
        p->seg_hi[(size_t)t] = (int)(*segments)[x + 1];
      }
  }
  // Work per distinct mask rule: every layout has at most four rules, so a
  // small cache suffices.
  std::vector<std::pair<std::vector<long long>, std::pair<long long, long long>>> cache;
  auto work = [&](const BlockPlan& b) {
    const std::vector<long long> key{b.klim[0], b.klim[1], b.hdelta[0], b.hdelta[1], b.lodelta};
    for (auto& e : cache)
      if (e.first == key) return e.second;
    long long tiles = 0;
    for (int t = 0; t < p->T; ++t) {
      int nk, full;
      tile_range(layout, n, p->KT, b, t, &nk, &full);
      tiles += nk;
    }
    std::pair<long long, long long> w{block_pairs(layout, n, b), tiles};
    cache.push_back({key, w});
    return w;
  };
  for (int s = 0; s < P; ++s) {
    for (int r = 0; r < P; ++r) {
      BlockPlan b = classify(layout, causal, n, r, block_of(P, r, s), P, window);
      const bool zz_general = layout == RING_LAYOUT_ZIGZAG && (packed || window > 0);
      auto w = zz_general ? zigzag_work(*p, r, b.j) : (packed ? segment_work(*p, b, r) : work(b));
      if (zz_general && w.first == 0) b.cls = RING_BLOCK_SKIP;  // nothing left inside the window / documents
      p->blocks[(size_t)s * P + r] = b;
      p->shard_pairs[r] += w.first * bh;
      p->shard_tiles[r] += w.second * bh;
      p->step_pairs[s] += w.first * bh;
      p->step_tiles[s] += w.second * bh;
      // The last step finalizes every shard, so it lists them all.
      if (w.first > 0 || s == P - 1) p->active[s].push_back((unsigned short)r);
    }
  }
  return RING_OK;
}

}  // namespace ringattn
