// internal.h -- definitions shared by the library's translation units.
// Not part of the C ABI (that is include/ringattn.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "../../include/ringattn.h"

namespace ringattn {

constexpr int kTileM = 128;       // query rows per tile (one TMEM lane each)
constexpr int kTileN = 128;       // keys per k-tile
constexpr int kMaxShards = 1024;  // P limit (kernel parameter table size)

// ---------------------------------------------------------------- planner
// Unified mask rule: inside block (query shard r, key block j) the pair
// (local row i, local column k) is allowed iff k < klim[h] and
// k - i <= hdelta[h], h the half of the shard that row i is in (zigzag:
// i >= n/2; the other layouts use half 0 only):
//   contiguous: pos(j,k) <= pos(r,i)  <=>  k - i <= (r - j) n
//   striped:    k P + j <= i P + r    <=>  k - i <= 0 if j <= r, else -1
//   zigzag:     j < r: k < n/2; j = r: k - i <= 0; j > r: half 1 every key
//   non-causal: every pair (FULL).
// "No diagonal" is hdelta = n; a skipped row set has klim = 0.
struct BlockPlan {
  int j;            // key block held by shard r at this step
  int cls;          // ring_block_class_t
  long long delta;  // diagonal offset of the block (n when it has none)
  long long klim[2];
  long long hdelta[2];
  long long lodelta;  // sliding window: also k - i >= lodelta (kNoLowerOffset without one)
};
constexpr long long kNoLowerOffset = -(1LL << 50);

struct Plan {
  int B = 0, H = 0, d = 0, P = 0, causal = 0, layout = 0;
  int Hkv = 0;  // K/V heads (H for plain multi-head attention)
  long long window = 0;  // causal sliding window (0: none)
  long long N = 0, n = 0;
  int T = 0;   // query tiles per shard, ceil(n / kTileM)
  int KT = 0;  // key tiles per block,  ceil(n / kTileN)
  std::vector<BlockPlan> blocks;       // [step * P + r]
  std::vector<long long> shard_pairs;  // [P] allowed pairs over all steps
  std::vector<long long> shard_tiles;  // [P] computed 128x128 tiles
  std::vector<long long> step_pairs;   // [P]
  std::vector<long long> step_tiles;   // [P]
  std::vector<std::vector<unsigned short>> active;  // [step] shards with work
  // Sequence packing: document boundaries [0, .., N] (empty: one document)
  // and, per natural position, the first and one-past-last position of its
  // document.
  std::vector<long long> seg_bounds;
  std::vector<int> seg_lo, seg_hi;

  const BlockPlan& at(int step, int r) const { return blocks[(size_t)step * P + r]; }
};

// Local key bounds (inclusive) that the segments allow row i of shard r in
// block j (contiguous or striped layout); lo > hi when none.
void seg_key_bounds(const Plan& p, int r, int j, long long i, long long* lo, long long* hi);
// Zigzag layout with a window or segments: local keys lo..hi of block j that
// the query at global position t may see; zz_position: position of shard r's
// local row i.
void zz_key_bounds(const Plan& p, int j, long long t, long long* lo, long long* hi);
long long zz_position(const Plan& p, int r, long long i);

int block_of(int P, int r, int step);  // (r - step) mod P
BlockPlan classify(int layout, int causal, long long n, int r, int j, int P = 1, long long window = 0);
// Half of the shard that local row i is in (1 only for the zigzag layout's late chunk).
inline int row_half(int layout, long long n, long long i) {
  return (layout == RING_LAYOUT_ZIGZAG && i >= n / 2) ? 1 : 0;
}
long long block_pairs(int layout, long long n, const BlockPlan& b);
// Key tiles a query tile t needs (a prefix of the block: count) and how many
// of them need no mask.
void tile_range(int layout, long long n, int KT, const BlockPlan& b, int t, int* nk, int* full_kt);
int build_plan(Plan* plan, int B, int H, long long N, int d, int P, int causal, int layout,
               std::string* err, long long window = 0, const std::vector<long long>* segments = nullptr);

// ---------------------------------------------------------------- kernels
// Query tensor addressing modes for the TMA map of Q.
enum QMode : int {
  kQShardMajor = 0,  // [BH][n][d], map dims (d, n, 1, BH), coords (c, i, 0, bh)
  kQContiguous = 1,  // natural [BH][N][d] with pos = r n + i, dims (d, n, P, BH)
  kQStriped = 2,     // natural with pos = i P + r, dims (d, P, n, BH)
  kQZigzag = 3       // natural, chunks of c = n/2: dims (d, c, 2P, BH), chunk r then 2P-1-r
};
// Which slot of the K/V map holds the block of shard r at step s.
enum KvMode : int {
  kKvSlotR = 0,  // rotation buffer: slot r holds block (r - s) mod P
  kKvSlotJ = 1,  // direct: slot j holds block j
  kKvSingle = 2   // one block only (slot 0)
};

struct StepArgs {
  float* o_state;  // O~ rows, d floats each
  float* m_state;  // m rows (natural-log units of the scaled score)
  float* l_state;  // l rows
  float* out;      // finalize target: normalised rows
  float* lse;      // finalize target: m + ln l
  long long row_bh, row_r, row_i;  // state/out row = bh*row_bh + r*row_r + i*row_i
  int* err;                        // device error words [0] flags, [1] site
  unsigned long long wait_limit_ns;
  int n, P, BH, T, KT;
  int q_mode, kv_mode;
  int causal, layout, step;
  int accumulate;  // continue from the stored state
  int finalize;    // write out/lse instead of the state
  int n_active;    // shards in `active`
  int fixed_r;     // >= 0: single shard (block partial); ignores `active`
  int debug_drop_v;  // test hook: issue no V loads (see RING_OPT_DEBUG_DROP_V_LOADS)
  int forward;       // send the CTA's key tiles 2u, 2u+1 to slot r+1 of the next maps
  int state_tiled;   // state in [BH][P][T][D/8][128][8] (O~) and [BH][P][T][128] (m, l) blocks
  int G;             // query heads per K/V head: query head bh reads K/V head bh / G
  int nq;            // query rows per shard (n for the ring; the short query length otherwise)
  long long window;  // > 0: causal sliding window, a query sees itself and the window-1 tokens before it
  long long decode_pos0;  // >= 0: short queries at global positions pos0 + i against the keys of
                          //       the natural-order cache, read as one contiguous block (P = 1, key k
                          //       at position k; see ring_attn_decode)
  int bh0;                // first query head of this launch (launches cover at most 65535 head groups)
  int head_lg;            // log2 of the heads whose CTAs interleave (set by the launch)
  int ksplit;             // >= 1: pieces the block's key tiles are cut into (short queries only); piece p
                          //       keeps its state in slot p
  float scale_log2;  // log2(e) / sqrt(d)
  // sequence packing (nullptr: one document): per natural position, the
  // first and one-past-last position of its document; a pair is allowed
  // only inside one document
  const int* seg_lo;
  const int* seg_hi;
  unsigned short active[kMaxShards];
};

// Arguments of the backward step kernels (one ring step, every shard).
// Natural-order tensors are [BH][N][d]; the row of (shard r, local i) within
// a head is r * row_r + i * row_i.  Shard-major vectors are [BH][P][n_pad].
struct BwdArgs {
  const float* nlse2;  // -lse * log2(e) of every query row, shard-major
  const float* nD;     // -D = -rowsum(dO * out) of every query row, shard-major
  float* dq;          // natural: the running dQ (unscaled) between steps, scale * dQ after the last
  const float* acc_in_k;  // [P][BH][n][d]: the dK~ and dV~ accumulators held by shard r (slot r)
  const float* acc_in_v;
  float* acc_out_k;  // the other buffer: shard r passes its block's accumulators to slot r + 1
  float* acc_out_v;
  float* dk;  // natural, written at the last step (dK scaled, dV as is)
  float* dv;
  long long N, row_r, row_i;
  int* err;  // device error words [0] flags, [1] site
  unsigned long long wait_limit_ns;
  int n, n_pad, P, BH, T, KT;
  int BHkv, G;  // K/V heads, and query heads per K/V head (query head bh reads K/V head bh / G)
  int q_mode;  // kQContiguous, kQStriped or kQZigzag: Q, dO, K and V through the same shard view
  int causal, layout, step;
  int accumulate;  // step > 0: continue the accumulators
  int last;        // step P - 1: write the gradients
  int lap;         // one launch for the whole ring: each CTA visits every shard in step order,
                   // its accumulators staying on chip (then step 0, accumulate 0, last 1)
  long long window;
  float scale, scale_log2;
  const int* seg_lo;  // sequence packing, as in StepArgs (nullptr: one document)
  const int* seg_hi;
};

// Device error flags.
constexpr int kErrTimeout = 1;

struct TensorMaps;  // opaque here (holds CUtensorMap values)

// Launchers (return a cudaError_t as int).
// k_next_map / v_next_map: the other rotation buffer, used only when
// a.forward is set (the kernel then sends its blocks there, slot r -> r+1).
int launch_block_partial(const StepArgs& a, const void* q_map, const void* k_map, const void* v_map,
                         int d, int grid, void* stream, const void* k_next_map = nullptr,
                         const void* v_next_map = nullptr);
int launch_state_init(float* m, float* l, float* o, long long rows, int d, void* stream);
// SMs of the current device (1 when there is none)
int sm_count();
int launch_merge(float* ma, float* la, float* oa, const float* mb, const float* lb, const float* ob,
                 long long rows, int d, void* stream);
int launch_merge_shards(const float* m, const float* l, const float* o, float* out, float* lse, long long rows,
                        int d, int P, void* stream);
int launch_finalize(const float* m, const float* l, const float* o, float* out, float* lse, int BH,
                    long long n, int d, int P, int r, int layout, long long N, void* stream);
int launch_pack_kv(const void* k, const void* v, void* kbuf, void* vbuf, int BH, long long n, int d,
                   int P, int layout, void* stream);
// Error reporting and TMA descriptors shared across translation units:
// report_error sets ring_attn_last_error() and returns `code`;
// tensor_map_4d encodes a 4-D bf16 map (box 64 x box1 x box2 x 1, 128-byte
// swizzle) into `map` (a CUtensorMap), dims innermost first, strides in bytes.
int report_error(int code, const char* msg);
int tensor_map_4d(void* map, const void* base, const unsigned long long dims[4],
                  const unsigned long long strides[3], unsigned box1, unsigned box2);
// The handle's plan and wait limit, for translation units outside api.cu.
const Plan& handle_plan(const ring_attn* h);
unsigned long long handle_wait_limit(const ring_attn* h);
int handle_debug_drop_v(const ring_attn* h);  // RING_OPT_DEBUG_DROP_V_LOADS
int block_partial_smem_bytes(int d);
// The ring forward in one launch (block_lap.cu): a.out / a.lse receive the
// result; K/V maps as for kKvSlotJ.
int launch_fwd_lap(const StepArgs& a, const void* q_map, const void* k_map, const void* v_map, int d, void* stream);
int prepare_fwd_lap_kernels();
// CTAs of one block-partial launch: one per (pair of query tiles, shard, head).
int block_partial_grid(int T, int n_active, int BH);
int prepare_block_partial_kernels();
// Backward (block_backward.cu).  The maps are shard views of natural-order
// bf16 tensors (box 64 x 128 rows), coordinates as for kQContiguous/kQStriped.
int launch_bwd_prep(const float* out, const float* lse, const void* dout, float* nlse2, float* nD, int BH,
                    long long n, int n_pad, int d, int P, long long row_r, long long row_i, long long N,
                    int zigzag, void* stream);
int launch_bwd_dkdv(const BwdArgs& a, const void* q_map, const void* do_map, const void* k_map, const void* v_map,
                    int d, void* stream);
int launch_bwd_dq(const BwdArgs& a, const void* q_map, const void* do_map, const void* k_map, const void* v_map,
                  int d, void* stream);
int prepare_backward_kernels();

}  // namespace ringattn
