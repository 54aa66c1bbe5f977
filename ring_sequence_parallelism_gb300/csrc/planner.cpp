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

BlockPlan classify(int layout, int causal, long long n, int r, int j) {
  BlockPlan b{j, RING_BLOCK_FULL, n};
  if (!causal) return b;
  if (layout == RING_LAYOUT_STRIPED) {
    // token positions i*P + r (queries) and k*P + j (keys): k*P + j <= i*P + r
    // <=> k - i <= 0 when j <= r, and k - i <= -1 when j > r.
    b.delta = (j <= r) ? 0 : -1;
  } else {
    b.delta = (long long)(r - j) * n;
  }
  if (b.delta >= n - 1) {
    b.cls = RING_BLOCK_FULL;
  } else if (b.delta <= -n) {
    b.cls = RING_BLOCK_SKIP;
  } else {
    b.cls = RING_BLOCK_DIAG;
  }
  return b;
}

long long block_pairs(long long n, const BlockPlan& b) {
  if (b.cls == RING_BLOCK_SKIP) return 0;
  if (b.cls == RING_BLOCK_FULL) return n * n;
  // rows i = 0..n-1 allow columns 0..min(n-1, i+delta)
  long long total = 0;
  for (long long i = 0; i < n; ++i) {
    long long c = std::min(n, std::max(0LL, i + b.delta + 1));
    total += c;
  }
  return total;
}

void tile_range(long long n, int KT, const BlockPlan& b, int t, int* nk, int* full_kt) {
  const bool ragged = (n % kTileN) != 0;
  if (b.cls == RING_BLOCK_SKIP) {
    *nk = 0;
    *full_kt = 0;
    return;
  }
  if (b.cls == RING_BLOCK_FULL) {
    *nk = KT;
    *full_kt = ragged ? KT - 1 : KT;
    return;
  }
  const long long i_min = (long long)t * kTileM;
  const long long i_max = std::min(n - 1, i_min + kTileM - 1);
  const long long last_key = i_max + b.delta;  // largest allowed key of the tile
  int cnt = last_key < 0 ? 0 : (int)std::min<long long>(KT, last_key / kTileN + 1);
  const long long first_row_keys = i_min + b.delta + 1;  // keys allowed for every row
  int full = first_row_keys <= 0 ? 0 : (int)std::min<long long>(cnt, first_row_keys / kTileN);
  if (ragged && full == KT) full = KT - 1;
  *nk = cnt;
  *full_kt = full;
}

int build_plan(Plan* p, int B, int H, long long N, int d, int P, int causal, int layout,
               std::string* err) {
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
  if (layout != RING_LAYOUT_CONTIGUOUS && layout != RING_LAYOUT_STRIPED) {
    *err = "layout must be RING_LAYOUT_CONTIGUOUS or RING_LAYOUT_STRIPED";
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
  if (n > (1LL << 30) || bh > (1LL << 30)) {
    *err = "shard length or B*H too large";
    return RING_ERR_UNSUPPORTED;
  }
  p->B = B;
  p->H = H;
  p->N = N;
  p->d = d;
  p->P = P;
  p->causal = causal;
  p->layout = layout;
  p->n = n;
  p->T = (int)((n + kTileM - 1) / kTileM);
  p->KT = (int)((n + kTileN - 1) / kTileN);
  p->blocks.assign((size_t)P * P, BlockPlan{});
  p->shard_pairs.assign(P, 0);
  p->shard_tiles.assign(P, 0);
  p->step_pairs.assign(P, 0);
  p->step_tiles.assign(P, 0);
  p->active.assign(P, {});
  // Work per distinct (class, delta): the striped layout has two deltas, the
  // contiguous one FULL/SKIP plus the diagonal, so a small cache suffices.
  std::vector<std::pair<long long, std::pair<long long, long long>>> cache;
  auto work = [&](const BlockPlan& b) {
    long long key = b.cls == RING_BLOCK_DIAG ? b.delta : (b.cls == RING_BLOCK_FULL ? (1LL << 62) : -(1LL << 62));
    for (auto& e : cache)
      if (e.first == key) return e.second;
    long long tiles = 0;
    for (int t = 0; t < p->T; ++t) {
      int nk, full;
      tile_range(n, p->KT, b, t, &nk, &full);
      tiles += nk;
    }
    std::pair<long long, long long> w{block_pairs(n, b), tiles};
    cache.push_back({key, w});
    return w;
  };
  for (int s = 0; s < P; ++s) {
    for (int r = 0; r < P; ++r) {
      BlockPlan b = classify(layout, causal, n, r, block_of(P, r, s));
      p->blocks[(size_t)s * P + r] = b;
      auto w = work(b);
      p->shard_pairs[r] += w.first * bh;
      p->shard_tiles[r] += w.second * bh;
      p->step_pairs[s] += w.first * bh;
      p->step_tiles[s] += w.second * bh;
      // The last step finalizes every shard, so it lists them all.
      if (b.cls != RING_BLOCK_SKIP || s == P - 1) p->active[s].push_back((unsigned short)r);
    }
  }
  return RING_OK;
}

}  // namespace ringattn
