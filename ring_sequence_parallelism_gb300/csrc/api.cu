// api.cu -- the C ABI (include/ringattn.h): handle, argument checks, TMA
// tensor maps and the P-step ring scheduler with the double-buffered K/V
// rotation on a side stream.
//
// Ring forward on one device ([RA-CN] "环是怎样工作的" forward loop;
// "双缓冲是重叠成立的基础": buffer A is read by the attention kernel while
// buffer B receives the next block, roles swap, streams and events order the
// two; [GRA] "Hiding the ring behind the GEMMs"):
//
//   compute stream: pack K,V -> X          record packed
//   side stream:    wait packed;      Y <- rotate(X);   record landed[1]
//   compute stream: step 0 on X;                        record released[0]
//   side stream:    wait released[0]; X <- rotate(Y);   record landed[2]
//   compute stream: wait landed[1]; step 1 on Y;        record released[1]
//   ...
// rotate(src): dst slot r <- src slot (r - 1) mod P, i.e. every shard sends
// its block to shard r + 1 and receives from r - 1 ([GRA] "One lap around
// the ring").
//
// Rotation modes (RING_OPT_ROTATION):
//   2 (default) the step kernel sends: each CTA stores the key/value tiles on
//     its diagonal from shared memory into slot r+1 of the other buffer, so
//     every block a step computes on is also moved by that step.  Only the
//     slots of shards with no work at step s (skipped causal blocks) are
//     copied, with cudaMemcpyAsync on the side stream:
//       side stream:    wait released[s-1]; copy those slots;  record landed[s+1]
//       compute stream: wait landed[s+1] before step s+1 (only if copied).
//     The kernel reads buffer s&1 and writes the other one, so kernels in
//     stream order need no events between them.
//   1 two cudaMemcpyAsync device-to-device copies per tensor per step on the
//     side stream (the schedule above).
//   0 no rotation: every step reads its block straight from the packed buffer.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>

#include "internal.h"

using namespace ringattn;

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  std::string msg = std::string(what) + ": " + cudaGetErrorString(e);
  cudaGetLastError();  // clear a sticky launch error where possible
  return fail(RING_ERR_CUDA, msg);
}

#define RA_CUDA(call, what)                     \
  do {                                          \
    cudaError_t _e = (call);                    \
    if (_e != cudaSuccess) return cuda_fail(_e, what); \
  } while (0)

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encoder() {
  if (g_encode) return RING_OK;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  void* fn = nullptr;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
    return fail(RING_ERR_CUDA, "cannot resolve cuTensorMapEncodeTiled from the driver");
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return RING_OK;
}

// 4-D bf16 tensor map, box (64, b1, b2, 1), 128-byte swizzle, zero fill out
// of bounds.  dims/strides are innermost first; strides in bytes for dims 1..3.
int encode_map(CUtensorMap* map, const void* base, const cuuint64_t dims[4], const cuuint64_t strides[3],
               cuuint32_t b1, cuuint32_t b2) {
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0) return fail(RING_ERR_INVALID_ARG, "tensor not 16-byte aligned");
  cuuint32_t box[4] = {64, b1, b2, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[128];
    std::snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return fail(RING_ERR_CUDA, buf);
  }
  return RING_OK;
}

}  // namespace

namespace ringattn {
// Shared with other translation units of the library (declared in internal.h).
int report_error(int code, const char* msg) { return fail(code, msg); }

int tensor_map_4d(void* map, const void* base, const unsigned long long dims[4],
                  const unsigned long long strides[3], unsigned box1, unsigned box2) {
  int rc = get_encoder();
  if (rc) return rc;
  cuuint64_t d4[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t s3[3] = {strides[0], strides[1], strides[2]};
  return encode_map(static_cast<CUtensorMap*>(map), base, d4, s3, box1, box2);
}
}  // namespace ringattn

struct ring_attn;

// ring_attn_fwd_host's pipeline over head groups (made on first use):
// device copies of the inputs and outputs of all heads, a handle with its
// own workspace for each (lane, group size) in use, a stream each for the
// copies in and out, and a stream for the second compute lane.
struct HostPipe {
  std::vector<int> sizes;       // K/V heads of each group, in head order
  std::vector<int> group_sub;   // the handle each group runs on
  std::vector<ring_attn*> subs;  // one per (lane, group size)
  std::vector<int> sub_units;   // K/V heads of each handle
  std::vector<int> sub_lane;    // the lane each handle runs on
  std::vector<size_t> sub_ws;   // workspace offset of each handle
  int lanes = 1;
  uint8_t* dev = nullptr;
  size_t q_off = 0, k_off = 0, v_off = 0, o_off = 0, l_off = 0;
  cudaStream_t in = nullptr, out = nullptr, lane1 = nullptr;
  std::vector<cudaEvent_t> ev_in, ev_comp;
  cudaEvent_t ev_start = nullptr, ev_done = nullptr, ev_lane = nullptr;
  bool have_done = false;  // ev_done recorded by an earlier call
};

// Events of one timed ring_attn_fwd (RING_OPT_TIMING).
struct FwdTiming {
  std::vector<cudaEvent_t> k0, k1;  // [s]: around the step kernel (lap: the launch, entry 0)
  std::vector<cudaEvent_t> c0, c1;  // [s]: around the side-stream copy that feeds step s
  std::vector<cudaEvent_t> w0, w1;  // [s]: around the compute stream's wait for that copy
  std::vector<cudaEvent_t> r0;      // [s]: side stream, before its wait for the buffer (then c0)
  cudaEvent_t p0 = nullptr, p1 = nullptr;  // around the pack
  std::vector<char> copied;         // [s]: a copy fed step s
};
// The timing getters average over the timed forwards since the previous
// read, the latest kTimedCalls of them.
constexpr int kTimedCalls = 64;

struct ring_attn {
  Plan plan;
  int rotation = 2;
  int timing = 0;
  int bwd_lap = 1;       // RING_OPT_BWD_LAP
  int fwd_lap = 0;       // RING_OPT_FWD_LAP
  int debug_drop_v = 0;
  unsigned long long wait_limit_ns = 2000000000ULL;
  // device resources, made on first use
  bool ready = false;
  int device = -1;
  cudaStream_t side = nullptr;
  cudaEvent_t packed = nullptr;
  std::vector<cudaEvent_t> landed, released;
  std::vector<FwdTiming> tsets;  // event sets of timed forwards, used in turn
  int t_next = 0;                // set of the next timed forward
  int t_count = 0;               // timed forwards recorded (at most kTimedCalls)
  bool t_read = false;           // a getter has read them: the next timed forward starts anew
  std::vector<cudaEvent_t> tbk0, tbk1, tbq0, tbq1;  // backward: dK/dV and dQ kernels per step
  cudaEvent_t tbp0 = nullptr, tbp1 = nullptr;          // backward preprocessing
  bool bwd_timed_valid = false;
  bool bwd_timed_lap = false;  // the timed backward ran in lap mode (one launch each)
  std::vector<char> copied;  // [s]: the side stream filled slots for step s (this forward)
  int* d_err = nullptr;  // [0] flags, [1] first failing site
  int* d_seg = nullptr;  // segments: first / one-past-last position of each position's document, [2][N]
  long long d_seg_n = 0;
  bool seg_dirty = false;
  HostPipe* pipe = nullptr;  // ring_attn_fwd_host
};

namespace ringattn {
const Plan& handle_plan(const ring_attn* h) { return h->plan; }
unsigned long long handle_wait_limit(const ring_attn* h) { return h->wait_limit_ns; }
int handle_debug_drop_v(const ring_attn* h) { return h->debug_drop_v; }
}  // namespace ringattn

namespace {

void destroy_pipe(HostPipe* hp) {
  if (!hp) return;
  for (cudaStream_t st : {hp->in, hp->out, hp->lane1})
    if (st) cudaStreamSynchronize(st);
  for (auto* v : {&hp->ev_in, &hp->ev_comp})
    for (auto e : *v)
      if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : {hp->ev_start, hp->ev_done, hp->ev_lane})
    if (e) cudaEventDestroy(e);
  for (cudaStream_t st : {hp->in, hp->out, hp->lane1})
    if (st) cudaStreamDestroy(st);
  if (hp->dev) cudaFree(hp->dev);
  for (ring_attn* sub : hp->subs) ring_attn_destroy(sub);
  delete hp;
}
int make_events(std::vector<cudaEvent_t>& v, int n, unsigned flags) {
  v.assign(n, nullptr);
  for (int i = 0; i < n; ++i) RA_CUDA(cudaEventCreateWithFlags(&v[i], flags), "cudaEventCreate");
  return RING_OK;
}

// The event set for the next timed forward (made on first use).
int begin_timed_call(ring_attn* h, FwdTiming** out) {
  if (h->t_read) {
    h->t_count = 0;
    h->t_next = 0;
    h->t_read = false;
  }
  if ((int)h->tsets.size() <= h->t_next) {
    FwdTiming T;
    const int P = h->plan.P;
    int rc = RING_OK;
    for (auto* v : {&T.k0, &T.k1, &T.c0, &T.c1, &T.w0, &T.w1, &T.r0})
      if (!rc) rc = make_events(*v, P, cudaEventDefault);
    if (!rc && cudaEventCreate(&T.p0) != cudaSuccess) rc = fail(RING_ERR_CUDA, "cudaEventCreate");
    if (!rc && cudaEventCreate(&T.p1) != cudaSuccess) rc = fail(RING_ERR_CUDA, "cudaEventCreate");
    if (rc) {  // release what was made; the set is not kept
      for (auto* v : {&T.k0, &T.k1, &T.c0, &T.c1, &T.w0, &T.w1, &T.r0})
        for (auto e : *v)
          if (e) cudaEventDestroy(e);
      for (cudaEvent_t e : {T.p0, T.p1})
        if (e) cudaEventDestroy(e);
      return rc;
    }
    h->tsets.push_back(std::move(T));
  }
  *out = &h->tsets[h->t_next];
  return RING_OK;
}

void end_timed_call(ring_attn* h) {
  h->tsets[h->t_next].copied = h->copied;
  h->t_next = (h->t_next + 1) % kTimedCalls;
  if (h->t_count < kTimedCalls) ++h->t_count;
}

int ensure_device(ring_attn* h) {
  int dev = -1;
  RA_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (h->ready) {
    if (dev != h->device) return fail(RING_ERR_INVALID_ARG, "handle used on a different device than its first use");
    return RING_OK;
  }
  int major = 0, minor = 0;
  RA_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "cudaDeviceGetAttribute");
  RA_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3) {
    char buf[96];
    std::snprintf(buf, sizeof buf, "this library is built for sm_103a; device %d is sm_%d%d", dev, major, minor);
    return fail(RING_ERR_UNSUPPORTED, buf);
  }
  int rc = get_encoder();
  if (rc) return rc;
  RA_CUDA((cudaError_t)prepare_block_partial_kernels(), "cudaFuncSetAttribute");
  RA_CUDA((cudaError_t)prepare_backward_kernels(), "cudaFuncSetAttribute (backward)");
  RA_CUDA((cudaError_t)prepare_fwd_lap_kernels(), "cudaFuncSetAttribute (lap)");
  RA_CUDA(cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking), "cudaStreamCreate");
  const int P = h->plan.P;
  RA_CUDA(cudaEventCreateWithFlags(&h->packed, cudaEventDisableTiming), "cudaEventCreate");
  if ((rc = make_events(h->landed, P, cudaEventDisableTiming))) return rc;
  if ((rc = make_events(h->released, P, cudaEventDisableTiming))) return rc;
  for (auto* v : {&h->tbk0, &h->tbk1, &h->tbq0, &h->tbq1})
    if ((rc = make_events(*v, P, cudaEventDefault))) return rc;
  RA_CUDA(cudaEventCreate(&h->tbp0), "cudaEventCreate");
  RA_CUDA(cudaEventCreate(&h->tbp1), "cudaEventCreate");
  RA_CUDA(cudaMalloc(&h->d_err, 2 * sizeof(int)), "cudaMalloc(error word)");
  RA_CUDA(cudaMemset(h->d_err, 0, 2 * sizeof(int)), "cudaMemset");
  h->device = dev;
  h->ready = true;
  return RING_OK;
}

bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

// Device copy of the segment table (after ensure_device): seg_lo at d_seg,
// seg_hi at d_seg + N, or nullptr without segments.  Copied once per change.
int device_segments(ring_attn* h, const int** lo, const int** hi) {
  const Plan& p = h->plan;
  *lo = *hi = nullptr;
  if (p.seg_bounds.empty()) return RING_OK;
  if (h->seg_dirty || !h->d_seg) {
    if (h->d_seg && h->d_seg_n != p.N) {
      RA_CUDA(cudaFree(h->d_seg), "cudaFree(segments)");
      h->d_seg = nullptr;
    }
    if (!h->d_seg) {
      RA_CUDA(cudaMalloc(&h->d_seg, (size_t)2 * p.N * sizeof(int)), "cudaMalloc(segments)");
      h->d_seg_n = p.N;
    }
    RA_CUDA(cudaMemcpy(h->d_seg, p.seg_lo.data(), (size_t)p.N * sizeof(int), cudaMemcpyHostToDevice),
            "cudaMemcpy(segments)");
    RA_CUDA(cudaMemcpy(h->d_seg + p.N, p.seg_hi.data(), (size_t)p.N * sizeof(int), cudaMemcpyHostToDevice),
            "cudaMemcpy(segments)");
    h->seg_dirty = false;
  }
  *lo = h->d_seg;
  *hi = h->d_seg + p.N;
  return RING_OK;
}

// ring_attn_fwd's workspace: rotation buffers X and Y (K and V each, bf16
// [P][B][H][n][d]), then the running state between steps in 128-row tile
// blocks (O~ [BH][P][T][D/8][128][8] fp32, m and l [BH][P][T][128] fp32).
struct FwdWorkspace {
  size_t tensor_bytes, o_off, m_off, l_off, total;
};
FwdWorkspace fwd_workspace(const Plan& p) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  FwdWorkspace f;
  f.tensor_bytes = (size_t)p.B * p.Hkv * (size_t)p.N * p.d * 2;  // one K or V buffer (K/V heads)
  const size_t rows = (size_t)p.B * p.H * p.P * (size_t)p.T * kTileM;  // padded to whole tiles
  f.o_off = 4 * f.tensor_bytes;
  f.m_off = f.o_off + up(rows * p.d * 4);
  f.l_off = f.m_off + up(rows * 4);
  f.total = f.l_off + up(rows * 4);
  return f;
}

StepArgs base_args(const ring_attn* h) {
  StepArgs a;
  std::memset(&a, 0, sizeof a);
  const Plan& p = h->plan;
  a.err = h->d_err;
  a.wait_limit_ns = h->wait_limit_ns;
  a.n = (int)p.n;
  a.P = p.P;
  a.BH = p.B * p.H;
  a.G = p.H / p.Hkv;
  a.nq = (int)p.n;
  a.decode_pos0 = -1;
  a.window = p.window;
  a.T = p.T;
  a.KT = p.KT;
  a.causal = p.causal;
  a.layout = p.layout;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p.d));
  a.fixed_r = -1;
  a.debug_drop_v = h->debug_drop_v;
  a.ksplit = 1;
  return a;
}

}  // namespace

extern "C" {

const char* ring_attn_last_error(void) { return g_last_error.c_str(); }

int ring_attn_create(ring_attn_t* out, int B, int H, long long N, int d, int P, int causal, int layout) {
  return ring_attn_create_gqa(out, B, H, H, N, d, P, causal, layout);
}

int ring_attn_create_gqa(ring_attn_t* out, int B, int H, int Hkv, long long N, int d, int P, int causal,
                         int layout) {
  if (!out) return fail(RING_ERR_INVALID_ARG, "out handle pointer is NULL");
  *out = nullptr;
  if (Hkv <= 0 || H <= 0 || H % Hkv != 0)
    return fail(RING_ERR_INVALID_ARG, "the query heads H must be a positive multiple of the K/V heads Hkv");
  ring_attn* h = new (std::nothrow) ring_attn();
  if (!h) return fail(RING_ERR_OOM, "out of host memory");
  std::string err;
  int rc = build_plan(&h->plan, B, H, N, d, P, causal, layout, &err);
  if (rc != RING_OK) {
    delete h;
    return fail(rc, err);
  }
  h->plan.Hkv = Hkv;
  *out = h;
  g_last_error.clear();
  return RING_OK;
}

int ring_attn_destroy(ring_attn_t h) {
  if (!h) return RING_OK;
  destroy_pipe(h->pipe);
  h->pipe = nullptr;
  if (h->ready) {
    int prev = -1;
    cudaGetDevice(&prev);
    if (prev != h->device) cudaSetDevice(h->device);
    for (auto* v : {&h->landed, &h->released, &h->tbk0, &h->tbk1, &h->tbq0, &h->tbq1})
      for (auto e : *v)
        if (e) cudaEventDestroy(e);
    for (FwdTiming& T : h->tsets) {
      for (auto* v : {&T.k0, &T.k1, &T.c0, &T.c1, &T.w0, &T.w1, &T.r0})
        for (auto e : *v)
          if (e) cudaEventDestroy(e);
      for (cudaEvent_t e : {T.p0, T.p1})
        if (e) cudaEventDestroy(e);
    }
    if (h->tbp0) cudaEventDestroy(h->tbp0);
    if (h->tbp1) cudaEventDestroy(h->tbp1);
    if (h->packed) cudaEventDestroy(h->packed);
    if (h->side) cudaStreamDestroy(h->side);
    if (h->d_err) cudaFree(h->d_err);
    if (h->d_seg) cudaFree(h->d_seg);
    if (prev >= 0 && prev != h->device) cudaSetDevice(prev);
  }
  delete h;
  return RING_OK;
}

int ring_attn_workspace_size(ring_attn_t h, size_t* bytes) {
  if (!h || !bytes) return fail(RING_ERR_INVALID_ARG, "NULL argument");
  *bytes = fwd_workspace(h->plan).total;
  return RING_OK;
}

int ring_attn_plan_block(ring_attn_t h, int r, int step, int* j, int* cls, long long* delta) {
  if (!h) return fail(RING_ERR_INVALID_ARG, "NULL handle");
  const Plan& p = h->plan;
  if (r < 0 || r >= p.P || step < 0 || step >= p.P) return fail(RING_ERR_INVALID_ARG, "r or step out of range");
  const BlockPlan& b = p.at(step, r);
  if (j) *j = b.j;
  if (cls) *cls = b.cls;
  if (delta) *delta = b.delta;
  return RING_OK;
}

int ring_attn_plan_mask(ring_attn_t h, int r, int step, long long row, long long* key_limit, long long* delta) {
  if (!h) return fail(RING_ERR_INVALID_ARG, "NULL handle");
  const Plan& p = h->plan;
  if (r < 0 || r >= p.P || step < 0 || step >= p.P) return fail(RING_ERR_INVALID_ARG, "r or step out of range");
  if (row < 0 || row >= p.n) return fail(RING_ERR_INVALID_ARG, "row out of range");
  const BlockPlan& b = p.at(step, r);
  const int half = row_half(p.layout, p.n, row);
  if (key_limit) *key_limit = b.klim[half];
  if (delta) *delta = b.hdelta[half];
  return RING_OK;
}

int ring_attn_plan_key_range(ring_attn_t h, int r, int step, long long row, long long* first, long long* last) {
  if (!h) return fail(RING_ERR_INVALID_ARG, "NULL handle");
  const Plan& p = h->plan;
  if (r < 0 || r >= p.P || step < 0 || step >= p.P) return fail(RING_ERR_INVALID_ARG, "r or step out of range");
  if (row < 0 || row >= p.n) return fail(RING_ERR_INVALID_ARG, "row out of range");
  const BlockPlan& b = p.at(step, r);
  if (p.layout == RING_LAYOUT_ZIGZAG && (p.window > 0 || !p.seg_bounds.empty())) {
    long long lo, hi;
    zz_key_bounds(p, b.j, zz_position(p, r, row), &lo, &hi);
    if (first) *first = lo;
    if (last) *last = hi;
    return RING_OK;
  }
  const int half = row_half(p.layout, p.n, row);
  long long lo = std::max(0LL, row + b.lodelta);
  long long hi = std::min(b.klim[half], std::max(0LL, row + b.hdelta[half] + 1)) - 1;
  if (!p.seg_bounds.empty()) {
    long long slo, shi;
    seg_key_bounds(p, r, b.j, row, &slo, &shi);
    lo = std::max(lo, slo);
    hi = std::min(hi, shi);
  }
  if (first) *first = lo;
  if (last) *last = hi;
  return RING_OK;
}

int ring_attn_shard_work(ring_attn_t h, long long* pairs, long long* tiles) {
  if (!h) return fail(RING_ERR_INVALID_ARG, "NULL handle");
  for (int r = 0; r < h->plan.P; ++r) {
    if (pairs) pairs[r] = h->plan.shard_pairs[r];
    if (tiles) tiles[r] = h->plan.shard_tiles[r];
  }
  return RING_OK;
}

int ring_attn_step_work(ring_attn_t h, int step, long long* pairs, long long* tiles) {
  if (!h) return fail(RING_ERR_INVALID_ARG, "NULL handle");
  if (step < 0 || step >= h->plan.P) return fail(RING_ERR_INVALID_ARG, "step out of range");
  if (pairs) *pairs = h->plan.step_pairs[step];
  if (tiles) *tiles = h->plan.step_tiles[step];
  return RING_OK;
}

int ring_attn_set_segments(ring_attn_t h, const long long* bounds, int num_segments) {
  if (!h) return fail(RING_ERR_INVALID_ARG, "NULL handle");
  if (num_segments < 0 || (num_segments > 0 && !bounds)) return fail(RING_ERR_INVALID_ARG, "bad segment list");
  std::vector<long long> sb;
  if (num_segments > 0) sb.assign(bounds, bounds + num_segments + 1);
  const Plan& p = h->plan;
  Plan np;
  std::string err;
  int rc = build_plan(&np, p.B, p.H, p.N, p.d, p.P, p.causal, p.layout, &err, p.window, &sb);
  if (rc != RING_OK) return fail(rc, err);
  np.Hkv = p.Hkv;
  h->plan = std::move(np);
  h->seg_dirty = true;
  return RING_OK;
}

int ring_attn_set_option(ring_attn_t h, int option, long long value) {
  if (!h) return fail(RING_ERR_INVALID_ARG, "NULL handle");
  switch (option) {
    case RING_OPT_ROTATION:
      if (value < 0 || value > 2) return fail(RING_ERR_INVALID_ARG, "rotation must be 0, 1 or 2");
      h->rotation = (int)value;
      return RING_OK;
    case RING_OPT_TIMING:
      if (value != 0 && value != 1) return fail(RING_ERR_INVALID_ARG, "timing must be 0 or 1");
      h->timing = (int)value;
      return RING_OK;
    case RING_OPT_WAIT_LIMIT_NS:
      if (value <= 0) return fail(RING_ERR_INVALID_ARG, "wait limit must be positive");
      h->wait_limit_ns = (unsigned long long)value;
      return RING_OK;
    case RING_OPT_WINDOW: {
      if (value < 0) return fail(RING_ERR_INVALID_ARG, "window must be >= 0");
      Plan np;
      std::string err;
      const Plan& p = h->plan;
      int rc = build_plan(&np, p.B, p.H, p.N, p.d, p.P, p.causal, p.layout, &err, value, &p.seg_bounds);
      if (rc != RING_OK) return fail(rc, err);
      np.Hkv = p.Hkv;
      h->plan = std::move(np);
      return RING_OK;
    }
    case RING_OPT_BWD_LAP:
      if (value != 0 && value != 1) return fail(RING_ERR_INVALID_ARG, "backward lap must be 0 or 1");
      h->bwd_lap = (int)value;
      return RING_OK;
    case RING_OPT_FWD_LAP:
      if (value != 0 && value != 1) return fail(RING_ERR_INVALID_ARG, "forward lap must be 0 or 1");
      h->fwd_lap = (int)value;
      return RING_OK;
    case RING_OPT_DEBUG_DROP_V_LOADS:
      if (value != 0 && value != 1) return fail(RING_ERR_INVALID_ARG, "debug option must be 0 or 1");
      h->debug_drop_v = (int)value;
      return RING_OK;
    default:
      return fail(RING_ERR_INVALID_ARG, "unknown option");
  }
}

int ring_attn_state_init(ring_attn_t h, ring_state_t s, void* stream) {
  if (!h || !s.m || !s.l || !s.o) return fail(RING_ERR_INVALID_ARG, "NULL argument");
  if (!aligned16(s.o)) return fail(RING_ERR_INVALID_ARG, "state.o not 16-byte aligned");
  int rc = ensure_device(h);
  if (rc) return rc;
  const Plan& p = h->plan;
  RA_CUDA((cudaError_t)launch_state_init(s.m, s.l, s.o, (long long)p.B * p.H * p.n, p.d, stream),
          "state_init launch");
  return RING_OK;
}

int ring_attn_merge(ring_attn_t h, ring_state_t a, ring_state_t b, void* stream) {
  if (!h || !a.m || !a.l || !a.o || !b.m || !b.l || !b.o) return fail(RING_ERR_INVALID_ARG, "NULL argument");
  if (!aligned16(a.o) || !aligned16(b.o)) return fail(RING_ERR_INVALID_ARG, "state.o not 16-byte aligned");
  int rc = ensure_device(h);
  if (rc) return rc;
  const Plan& p = h->plan;
  RA_CUDA((cudaError_t)launch_merge(a.m, a.l, a.o, b.m, b.l, b.o, (long long)p.B * p.H * p.n, p.d, stream),
          "merge launch");
  return RING_OK;
}

int ring_attn_finalize(ring_attn_t h, int r, ring_state_t s, float* out, float* lse, void* stream) {
  if (!h || !s.m || !s.l || !s.o || !out || !lse) return fail(RING_ERR_INVALID_ARG, "NULL argument");
  const Plan& p = h->plan;
  if (r < 0 || r >= p.P) return fail(RING_ERR_INVALID_ARG, "r out of range");
  if (!aligned16(s.o) || !aligned16(out)) return fail(RING_ERR_INVALID_ARG, "tensor not 16-byte aligned");
  int rc = ensure_device(h);
  if (rc) return rc;
  RA_CUDA((cudaError_t)launch_finalize(s.m, s.l, s.o, out, lse, p.B * p.H, p.n, p.d, p.P, r, p.layout, p.N, stream),
          "finalize launch");
  return RING_OK;
}

int ring_attn_block_partial(ring_attn_t h, int r, int step, const void* q_shard, const void* k_block,
                            const void* v_block, ring_state_t state, int accumulate, void* stream) {
  if (!h || !q_shard || !k_block || !v_block || !state.m || !state.l || !state.o)
    return fail(RING_ERR_INVALID_ARG, "NULL argument");
  const Plan& p = h->plan;
  if (r < 0 || r >= p.P || step < 0 || step >= p.P) return fail(RING_ERR_INVALID_ARG, "r or step out of range");
  if (accumulate != 0 && accumulate != 1) return fail(RING_ERR_INVALID_ARG, "accumulate must be 0 or 1");
  if (!aligned16(q_shard) || !aligned16(k_block) || !aligned16(v_block) || !aligned16(state.o))
    return fail(RING_ERR_INVALID_ARG, "tensor not 16-byte aligned");
  int rc = ensure_device(h);
  if (rc) return rc;
  const int BH = p.B * p.H;
  const BlockPlan& b = p.at(step, r);
  if (b.cls == RING_BLOCK_SKIP && accumulate) return RING_OK;  // nothing to merge
  CUtensorMap qm, km, vm;
  const cuuint64_t d = (cuuint64_t)p.d, n = (cuuint64_t)p.n;
  const cuuint64_t row_b = d * 2;
  {
    cuuint64_t dims[4] = {d, n, 1, (cuuint64_t)BH};
    cuuint64_t str[3] = {row_b, row_b * n, row_b * n};
    if ((rc = encode_map(&qm, q_shard, dims, str, kTileM, 1))) return rc;
  }
  {
    const cuuint64_t BHkv = (cuuint64_t)p.B * p.Hkv;  // K/V blocks carry the K/V heads
    cuuint64_t dims[4] = {d, n, BHkv, 1};
    cuuint64_t str[3] = {row_b, row_b * n, row_b * n * BHkv};
    if ((rc = encode_map(&km, k_block, dims, str, kTileN, 1))) return rc;
    if ((rc = encode_map(&vm, v_block, dims, str, kTileN, 1))) return rc;
  }
  StepArgs a = base_args(h);
  if ((rc = device_segments(h, &a.seg_lo, &a.seg_hi))) return rc;
  a.o_state = state.o;
  a.m_state = state.m;
  a.l_state = state.l;
  a.out = nullptr;
  a.lse = nullptr;
  a.row_bh = (long long)p.n;
  a.row_r = 0;
  a.row_i = 1;
  a.q_mode = kQShardMajor;
  a.kv_mode = kKvSingle;
  a.step = step;
  a.accumulate = accumulate;
  a.finalize = 0;
  a.fixed_r = r;
  a.n_active = 1;
  const int grid = block_partial_grid(p.T, 1, BH);
  RA_CUDA((cudaError_t)launch_block_partial(a, &qm, &km, &vm, p.d, grid, stream), "block_partial launch");
  return RING_OK;
}

int ring_attn_fwd(ring_attn_t h, const void* q, const void* k, const void* v, float* out, float* lse,
                  void* workspace, void* stream) {
  if (!h || !q || !k || !v || !out || !lse || !workspace) return fail(RING_ERR_INVALID_ARG, "NULL argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return fail(RING_ERR_INVALID_ARG, "tensor not 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(RING_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  int rc = ensure_device(h);
  if (rc) return rc;
  const Plan& p = h->plan;
  const int P = p.P, BH = p.B * p.H;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const FwdWorkspace fw = fwd_workspace(p);
  const size_t tensor_bytes = fw.tensor_bytes;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* kbuf[2] = {ws, ws + 2 * tensor_bytes};
  void* vbuf[2] = {ws + tensor_bytes, ws + 3 * tensor_bytes};
  const int mode = P > 1 ? h->rotation : 0;
  const bool rotate = mode != 0;

  // tensor maps: Q in natural order (strided per shard), K/V rotation buffers
  const cuuint64_t d = (cuuint64_t)p.d, n = (cuuint64_t)p.n, row_b = d * 2;
  CUtensorMap qm, km[2], vm[2];
  if (p.layout == RING_LAYOUT_STRIPED) {
    cuuint64_t dims[4] = {d, (cuuint64_t)P, n, (cuuint64_t)BH};
    cuuint64_t str[3] = {row_b, row_b * P, row_b * (cuuint64_t)p.N};
    if ((rc = encode_map(&qm, q, dims, str, 1, kTileM))) return rc;
  } else if (p.layout == RING_LAYOUT_ZIGZAG) {
    // chunks of c = n/2 tokens: dims (d, c, 2P chunks, BH)
    cuuint64_t dims[4] = {d, n / 2, (cuuint64_t)(2 * P), (cuuint64_t)BH};
    cuuint64_t str[3] = {row_b, row_b * (n / 2), row_b * (cuuint64_t)p.N};
    if ((rc = encode_map(&qm, q, dims, str, kTileM, 1))) return rc;
  } else {
    cuuint64_t dims[4] = {d, n, (cuuint64_t)P, (cuuint64_t)BH};
    cuuint64_t str[3] = {row_b, row_b * n, row_b * (cuuint64_t)p.N};
    if ((rc = encode_map(&qm, q, dims, str, kTileM, 1))) return rc;
  }
  const int BHkv = p.B * p.Hkv;  // the rotation buffers hold the K/V heads only
  for (int x = 0; x < 2; ++x) {
    cuuint64_t dims[4] = {d, n, (cuuint64_t)BHkv, (cuuint64_t)P};
    cuuint64_t str[3] = {row_b, row_b * n, row_b * n * BHkv};
    if ((rc = encode_map(&km[x], kbuf[x], dims, str, kTileN, 1))) return rc;
    if ((rc = encode_map(&vm[x], vbuf[x], dims, str, kTileN, 1))) return rc;
  }
  // The lap (no rotation) reads the blocks in place from the caller's
  // natural-order K/V, with the same coordinates as the packed buffer
  // (d column, row k of block j, head, j): key k of block j is token j n + k
  // (contiguous) or k P + j (striped), so it needs no packing pass.  The
  // step schedule packs the blocks into rotation buffer A, from which the
  // ring moves them; zigzag blocks are two chunks (not one strided map), so
  // the lap packs them too.
  const bool in_place = h->fwd_lap && p.layout != RING_LAYOUT_ZIGZAG;
  CUtensorMap kn_map, vn_map;
  if (in_place) {
    const bool striped = p.layout == RING_LAYOUT_STRIPED;
    const cuuint64_t Nn = (cuuint64_t)p.N;
    cuuint64_t dims[4] = {d, n, (cuuint64_t)BHkv, (cuuint64_t)P};
    cuuint64_t str[3] = {striped ? row_b * P : row_b, row_b * Nn, striped ? row_b : row_b * n};
    if ((rc = encode_map(&kn_map, k, dims, str, kTileN, 1))) return rc;
    if ((rc = encode_map(&vn_map, v, dims, str, kTileN, 1))) return rc;
  }

  const bool timing = h->timing != 0;
  FwdTiming* T = nullptr;
  if (timing && (rc = begin_timed_call(h, &T))) return rc;
  if (timing) RA_CUDA(cudaEventRecord(T->p0, cs), "cudaEventRecord");
  if (!in_place)
    RA_CUDA((cudaError_t)launch_pack_kv(k, v, kbuf[0], vbuf[0], BHkv, p.n, p.d, P, p.layout, cs), "pack launch");
  if (timing) RA_CUDA(cudaEventRecord(T->p1, cs), "cudaEventRecord");
  if (rotate) RA_CUDA(cudaEventRecord(h->packed, cs), "cudaEventRecord");

  const size_t slot_bytes = (size_t)BHkv * (size_t)p.n * p.d * 2;
  StepArgs a = base_args(h);
  if ((rc = device_segments(h, &a.seg_lo, &a.seg_hi))) return rc;
  a.o_state = reinterpret_cast<float*>(ws + fw.o_off);  // the running state, tile blocks
  a.m_state = reinterpret_cast<float*>(ws + fw.m_off);
  a.l_state = reinterpret_cast<float*>(ws + fw.l_off);
  a.state_tiled = 1;
  a.out = out;  // natural order, written by the last step
  a.lse = lse;
  a.row_bh = p.N;
  a.row_r = p.layout == RING_LAYOUT_STRIPED ? 1 : p.n;
  a.row_i = p.layout == RING_LAYOUT_STRIPED ? P : 1;
  a.q_mode = p.layout == RING_LAYOUT_STRIPED ? kQStriped : (p.layout == RING_LAYOUT_ZIGZAG ? kQZigzag : kQContiguous);
  a.kv_mode = rotate ? kKvSlotR : kKvSlotJ;
  h->copied.assign((size_t)P, 0);

  if (h->fwd_lap) {
    // the whole ring in one launch, blocks read in place (slot j = block j)
    a.kv_mode = kKvSlotJ;
    a.finalize = 1;
    a.n_active = P;
    if (timing) RA_CUDA(cudaEventRecord(T->k0[0], cs), "cudaEventRecord");
    RA_CUDA((cudaError_t)launch_fwd_lap(a, &qm, in_place ? &kn_map : &km[0], in_place ? &vn_map : &vm[0], p.d, cs),
            "lap kernel launch");
    if (timing) {
      for (int s = 0; s < P; ++s) {
        if (s > 0) RA_CUDA(cudaEventRecord(T->k0[s], cs), "cudaEventRecord");
        RA_CUDA(cudaEventRecord(T->k1[s], cs), "cudaEventRecord");
      }
      end_timed_call(h);
    }
    return RING_OK;
  }

  // side-stream copy of slots [r0, r0 + cnt) of buffer `cur` to [dst0, dst0 + cnt) of the other
  auto copy_slots = [&](int cur, int r0, int dst0, int cnt) -> int {
    for (int t = 0; t < 2; ++t) {
      uint8_t* dst = static_cast<uint8_t*>(t == 0 ? kbuf[cur ^ 1] : vbuf[cur ^ 1]);
      const uint8_t* src = static_cast<const uint8_t*>(t == 0 ? kbuf[cur] : vbuf[cur]);
      RA_CUDA(cudaMemcpyAsync(dst + (size_t)dst0 * slot_bytes, src + (size_t)r0 * slot_bytes,
                              (size_t)cnt * slot_bytes, cudaMemcpyDeviceToDevice, h->side),
              "rotation copy");
    }
    return RING_OK;
  };

  for (int s = 0; s < P; ++s) {
    const int cur = rotate ? (s & 1) : 0;
    if (rotate && s >= 1 && h->copied[s]) {
      if (timing) RA_CUDA(cudaEventRecord(T->w0[s], cs), "cudaEventRecord");
      RA_CUDA(cudaStreamWaitEvent(cs, h->landed[s], 0), "cudaStreamWaitEvent");
      if (timing) RA_CUDA(cudaEventRecord(T->w1[s], cs), "cudaEventRecord");
    }
    const auto& act = p.active[s];
    a.step = s;
    a.accumulate = s > 0 ? 1 : 0;
    a.finalize = s == P - 1 ? 1 : 0;
    a.forward = (mode == 2 && s + 1 < P) ? 1 : 0;
    a.n_active = (int)act.size();
    for (size_t x = 0; x < act.size(); ++x) a.active[x] = act[x];
    const int grid = block_partial_grid(p.T, a.n_active, BH);
    if (timing) RA_CUDA(cudaEventRecord(T->k0[s], cs), "cudaEventRecord");
    RA_CUDA((cudaError_t)launch_block_partial(a, &qm, &km[cur], &vm[cur], p.d, grid, cs, &km[cur ^ 1],
                                              &vm[cur ^ 1]),
            "step kernel launch");
    if (timing) RA_CUDA(cudaEventRecord(T->k1[s], cs), "cudaEventRecord");
    if (rotate) RA_CUDA(cudaEventRecord(h->released[s], cs), "cudaEventRecord");
    if (!rotate || s + 1 >= P) continue;
    // slots the side stream moves for step s+1: all of them (mode 1), or
    // those of shards the step kernel did not run (mode 2)
    std::vector<char> send((size_t)P, mode == 1 ? 1 : 0);
    if (mode == 2) {
      std::vector<char> ran((size_t)P, 0);
      for (unsigned short r : act) ran[r] = 1;
      for (int r = 0; r < P; ++r) send[r] = !ran[r];
    }
    bool any = false;
    for (int r = 0; r < P; ++r) any = any || send[r];
    if (!any) continue;
    // fill the other buffer once step s-1 has released it (and written it)
    if (timing) RA_CUDA(cudaEventRecord(T->r0[s + 1], h->side), "cudaEventRecord");
    RA_CUDA(cudaStreamWaitEvent(h->side, s == 0 ? h->packed : h->released[s - 1], 0), "cudaStreamWaitEvent");
    if (timing) RA_CUDA(cudaEventRecord(T->c0[s + 1], h->side), "cudaEventRecord");
    // runs of consecutive slots r0..r1 (r1 < P-1) go to r0+1..r1+1; slot P-1 goes to 0
    for (int r = 0; r < P - 1;) {
      if (!send[r]) { ++r; continue; }
      int r1 = r;
      while (r1 + 1 < P - 1 && send[r1 + 1]) ++r1;
      if ((rc = copy_slots(cur, r, r + 1, r1 - r + 1))) return rc;
      r = r1 + 1;
    }
    if (send[P - 1] && (rc = copy_slots(cur, P - 1, 0, 1))) return rc;
    if (timing) RA_CUDA(cudaEventRecord(T->c1[s + 1], h->side), "cudaEventRecord");
    RA_CUDA(cudaEventRecord(h->landed[s + 1], h->side), "cudaEventRecord");
    h->copied[s + 1] = 1;
  }
  if (timing) end_timed_call(h);
  return RING_OK;
}

// ------------------------------------------------------- from host memory
// ring_attn_fwd_host: the heads are independent problems, so they run in
// groups of whole K/V heads with their query heads.  The inputs of every
// group are copied in on stream `in`, in group order; each group is one
// ring_attn_fwd of a handle for the group's heads, on one of two compute
// lanes (the caller's stream and `lane1`, alternately), as soon as its
// inputs are in; its outputs are copied out on stream `out` as soon as it
// is done.  The two lanes run at the same time, so the SMs one group's step
// kernel leaves idle in its last wave take the other group's blocks.  The
// first two and the last two groups hold one K/V head each, which shortens
// the copy-in before the first kernel and the copy-out after the last.  The
// results are those of one ring_attn_fwd over all heads.

}  // extern "C"

namespace {

// K/V heads of each group: with 8 or more K/V heads in all batches, one in
// each of the first two and last two groups and the rest in an even number
// of near-equal groups of at most a quarter of them; with fewer, one each.
std::vector<int> host_group_sizes(int units) {
  if (units < 8) return std::vector<int>(units, 1);
  const int mid = units - 4, cap = (units + 3) / 4;
  int m = (mid + cap - 1) / cap;
  m += m & 1;
  std::vector<int> sizes = {1, 1};
  for (int i = 0; i < m; ++i) sizes.push_back(mid / m + (i < mid % m ? 1 : 0));
  sizes.push_back(1);
  sizes.push_back(1);
  return sizes;
}

// The group handles follow the parent's options (window, documents,
// rotation, wait limit); their plans are rebuilt when those changed.
int sync_group_handles(ring_attn* h) {
  HostPipe* hp = h->pipe;
  const Plan& p = h->plan;
  const int G = p.H / p.Hkv;
  for (size_t i = 0; i < hp->subs.size(); ++i) {
    ring_attn* sub = hp->subs[i];
    if (sub->plan.window != p.window || sub->plan.seg_bounds != p.seg_bounds) {
      const int units = hp->sub_units[i];
      Plan np;
      std::string err;
      int rc = build_plan(&np, 1, units * G, p.N, p.d, p.P, p.causal, p.layout, &err, p.window, &p.seg_bounds);
      if (rc != RING_OK) return fail(rc, err);
      np.Hkv = units;
      sub->plan = std::move(np);
      sub->seg_dirty = true;
    }
    sub->rotation = h->rotation;
    sub->fwd_lap = h->fwd_lap;
    sub->wait_limit_ns = h->wait_limit_ns;
  }
  return RING_OK;
}

int build_pipe(ring_attn* h, HostPipe* hp);

// The pipeline is attached to the handle only once every part of it exists.
int ensure_pipe(ring_attn* h) {
  if (h->pipe) return sync_group_handles(h);
  HostPipe* hp = new (std::nothrow) HostPipe();
  if (!hp) return fail(RING_ERR_OOM, "out of host memory");
  h->pipe = hp;  // sync_group_handles reads it
  const int rc = build_pipe(h, hp);
  if (rc) {
    h->pipe = nullptr;
    destroy_pipe(hp);
  }
  return rc;
}

int build_pipe(ring_attn* h, HostPipe* hp) {
  const Plan& p = h->plan;
  const int G = p.H / p.Hkv;
  hp->sizes = host_group_sizes(p.B * p.Hkv);
  const int groups = (int)hp->sizes.size();
  hp->lanes = groups > 1 ? 2 : 1;
  // one handle per (lane, group size)
  for (int g = 0; g < groups; ++g) {
    const int lane = g % hp->lanes, units = hp->sizes[g];
    int found = -1;
    for (size_t i = 0; i < hp->subs.size(); ++i)
      if (hp->sub_lane[i] == lane && hp->sub_units[i] == units) found = (int)i;
    if (found < 0) {
      ring_attn* sub = nullptr;
      int rc = ring_attn_create_gqa(&sub, 1, units * G, units, p.N, p.d, p.P, p.causal, p.layout);
      if (rc) return rc;
      sub->plan.window = -1;  // forces the first sync to build the plan with the options
      found = (int)hp->subs.size();
      hp->subs.push_back(sub);
      hp->sub_units.push_back(units);
      hp->sub_lane.push_back(lane);
    }
    hp->group_sub.push_back(found);
  }
  int rc = sync_group_handles(h);
  if (rc) return rc;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t q_bytes = (size_t)p.B * p.H * (size_t)p.N * p.d * 2;
  const size_t kv_bytes = (size_t)p.B * p.Hkv * (size_t)p.N * p.d * 2;
  const size_t o_bytes = (size_t)p.B * p.H * (size_t)p.N * p.d * 4;
  const size_t l_bytes = (size_t)p.B * p.H * (size_t)p.N * 4;
  hp->q_off = 0;
  hp->k_off = up(q_bytes);
  hp->v_off = hp->k_off + up(kv_bytes);
  hp->o_off = hp->v_off + up(kv_bytes);
  hp->l_off = hp->o_off + up(o_bytes);
  size_t total = hp->l_off + up(l_bytes);
  for (ring_attn* sub : hp->subs) {
    hp->sub_ws.push_back(total);
    total += up(fwd_workspace(sub->plan).total);
  }
  RA_CUDA(cudaMalloc(&hp->dev, total), "cudaMalloc(host-call buffers)");
  RA_CUDA(cudaStreamCreateWithFlags(&hp->in, cudaStreamNonBlocking), "cudaStreamCreate");
  RA_CUDA(cudaStreamCreateWithFlags(&hp->out, cudaStreamNonBlocking), "cudaStreamCreate");
  RA_CUDA(cudaStreamCreateWithFlags(&hp->lane1, cudaStreamNonBlocking), "cudaStreamCreate");
  if ((rc = make_events(hp->ev_in, groups, cudaEventDisableTiming))) return rc;
  if ((rc = make_events(hp->ev_comp, groups, cudaEventDisableTiming))) return rc;
  for (cudaEvent_t* e : {&hp->ev_start, &hp->ev_done, &hp->ev_lane})
    RA_CUDA(cudaEventCreateWithFlags(e, cudaEventDisableTiming), "cudaEventCreate");
  return RING_OK;
}

}  // namespace

extern "C" {

int ring_attn_fwd_host(ring_attn_t h, const void* q, const void* k, const void* v, float* out, float* lse,
                       void* stream) {
  if (!h || !q || !k || !v || !out || !lse) return fail(RING_ERR_INVALID_ARG, "NULL argument");
  int rc = ensure_device(h);
  if (rc) return rc;
  if ((rc = ensure_pipe(h))) return rc;
  HostPipe* hp = h->pipe;
  const Plan& p = h->plan;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int groups = (int)hp->sizes.size();
  const size_t G = p.H / p.Hkv, rows = (size_t)p.N;
  const size_t kv_head = rows * p.d * 2, q_head = G * rows * p.d * 2;  // bytes per K/V head
  const size_t o_head = G * rows * p.d * 4, l_head = G * rows * 4;
  uint8_t* dev = hp->dev;
  // the copies start after the caller's earlier work on its stream, and
  // after the previous call's outputs have left the device buffers
  RA_CUDA(cudaEventRecord(hp->ev_start, cs), "cudaEventRecord");
  RA_CUDA(cudaStreamWaitEvent(hp->in, hp->ev_start, 0), "cudaStreamWaitEvent");
  if (hp->have_done) RA_CUDA(cudaStreamWaitEvent(hp->in, hp->ev_done, 0), "cudaStreamWaitEvent");
  for (int g = 0, u0 = 0; g < groups; u0 += hp->sizes[g++]) {
    const size_t u = hp->sizes[g];
    // K and V first: the forward's first kernel packs them
    RA_CUDA(cudaMemcpyAsync(dev + hp->k_off + u0 * kv_head, static_cast<const uint8_t*>(k) + u0 * kv_head,
                            u * kv_head, cudaMemcpyHostToDevice, hp->in),
            "cudaMemcpyAsync(k)");
    RA_CUDA(cudaMemcpyAsync(dev + hp->v_off + u0 * kv_head, static_cast<const uint8_t*>(v) + u0 * kv_head,
                            u * kv_head, cudaMemcpyHostToDevice, hp->in),
            "cudaMemcpyAsync(v)");
    RA_CUDA(cudaMemcpyAsync(dev + hp->q_off + u0 * q_head, static_cast<const uint8_t*>(q) + u0 * q_head,
                            u * q_head, cudaMemcpyHostToDevice, hp->in),
            "cudaMemcpyAsync(q)");
    RA_CUDA(cudaEventRecord(hp->ev_in[g], hp->in), "cudaEventRecord");
  }
  // Every group's forward on its lane, and its output copies.  Whatever
  // happens, the other streams are closed out below, so the caller's stream
  // and the next call order after everything this call queued.
  rc = RING_OK;
  for (int g = 0, u0 = 0; g < groups && rc == RING_OK; u0 += hp->sizes[g++]) {
    const size_t u = hp->sizes[g];
    const int si = hp->group_sub[g];
    const cudaStream_t ls = hp->sub_lane[si] == 0 ? cs : hp->lane1;
    float* o_dev = reinterpret_cast<float*>(dev + hp->o_off + u0 * o_head);
    float* l_dev = reinterpret_cast<float*>(dev + hp->l_off + u0 * l_head);
    cudaError_t e = cudaStreamWaitEvent(ls, hp->ev_in[g], 0);
    if (e != cudaSuccess) {
      rc = fail(RING_ERR_CUDA, std::string("cudaStreamWaitEvent: ") + cudaGetErrorString(e));
      break;
    }
    if ((rc = ring_attn_fwd(hp->subs[si], dev + hp->q_off + u0 * q_head, dev + hp->k_off + u0 * kv_head,
                            dev + hp->v_off + u0 * kv_head, o_dev, l_dev, dev + hp->sub_ws[si], ls)))
      break;
    if ((e = cudaEventRecord(hp->ev_comp[g], ls)) == cudaSuccess &&
        (e = cudaStreamWaitEvent(hp->out, hp->ev_comp[g], 0)) == cudaSuccess &&
        (e = cudaMemcpyAsync(reinterpret_cast<uint8_t*>(out) + u0 * o_head, o_dev, u * o_head,
                             cudaMemcpyDeviceToHost, hp->out)) == cudaSuccess)
      e = cudaMemcpyAsync(reinterpret_cast<uint8_t*>(lse) + u0 * l_head, l_dev, u * l_head,
                          cudaMemcpyDeviceToHost, hp->out);
    if (e != cudaSuccess) rc = fail(RING_ERR_CUDA, std::string("output copy: ") + cudaGetErrorString(e));
  }
  // the caller's stream completes after the last output copy and after the
  // second lane (and after the copy-in stream, in case a failure left
  // copies there unwaited)
  RA_CUDA(cudaEventRecord(hp->ev_done, hp->out), "cudaEventRecord");
  hp->have_done = true;
  RA_CUDA(cudaStreamWaitEvent(cs, hp->ev_done, 0), "cudaStreamWaitEvent");
  RA_CUDA(cudaEventRecord(hp->ev_lane, hp->lane1), "cudaEventRecord");
  RA_CUDA(cudaStreamWaitEvent(cs, hp->ev_lane, 0), "cudaStreamWaitEvent");
  if (rc != RING_OK) {
    RA_CUDA(cudaEventRecord(hp->ev_start, hp->in), "cudaEventRecord");
    RA_CUDA(cudaStreamWaitEvent(cs, hp->ev_start, 0), "cudaStreamWaitEvent");
  }
  return rc;
}

// ---------------------------------------------------------------- backward
// Workspace of ring_attn_bwd: -lse*log2(e) and -D shard-major [BH][P][n_pad] fp32,
// then (one launch per ring step only) the dK~ and dV~ accumulator buffers X
// and Y, [P][BHkv][n][d] fp32 each.
struct BwdWorkspace {
  size_t lse_off, d_off, acc_bytes, acc_off, total;
  int n_pad;
};
// whether ring_attn_bwd runs one launch per ring step (and so needs the
// accumulator buffers): RING_OPT_BWD_LAP 0 with more than one shard
static bool bwd_per_step(const ring_attn* h) { return h->bwd_lap == 0 && h->plan.P > 1; }
static BwdWorkspace bwd_workspace(const Plan& p, bool per_step) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  BwdWorkspace w;
  w.n_pad = p.T * kTileM;
  const size_t vec = up((size_t)p.B * p.H * p.P * (size_t)w.n_pad * 4);
  w.lse_off = 0;
  w.d_off = vec;
  w.acc_bytes = up((size_t)p.B * p.Hkv * (size_t)p.N * p.d * 4);  // dK~ or dV~ of the K/V heads
  w.acc_off = 2 * vec;
  w.total = w.acc_off + (per_step ? 4 * w.acc_bytes : 0);
  return w;
}

int ring_attn_bwd_workspace_size(ring_attn_t h, size_t* bytes) {
  if (!h || !bytes) return fail(RING_ERR_INVALID_ARG, "NULL argument");
  *bytes = bwd_workspace(h->plan, bwd_per_step(h)).total;
  return RING_OK;
}

int ring_attn_bwd(ring_attn_t h, const void* q, const void* k, const void* v, const float* out, const float* lse,
                  const void* dout, float* dq, float* dk, float* dv, void* workspace, void* stream) {
  if (!h || !q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv || !workspace)
    return fail(RING_ERR_INVALID_ARG, "NULL argument");
  const Plan& p = h->plan;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(RING_ERR_INVALID_ARG, "tensor not 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(RING_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  int rc = ensure_device(h);
  if (rc) return rc;
  const int P = p.P, BH = p.B * p.H;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const bool lap = !bwd_per_step(h);
  const BwdWorkspace w = bwd_workspace(p, !lap);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* nlse2 = reinterpret_cast<float*>(ws + w.lse_off);
  float* nD = reinterpret_cast<float*>(ws + w.d_off);
  // the accumulator buffers exist in the per-step schedule's workspace only
  float* acc_k[2] = {nullptr, nullptr};
  float* acc_v[2] = {nullptr, nullptr};
  if (!lap) {
    acc_k[0] = reinterpret_cast<float*>(ws + w.acc_off);
    acc_k[1] = reinterpret_cast<float*>(ws + w.acc_off + 2 * w.acc_bytes);
    acc_v[0] = reinterpret_cast<float*>(ws + w.acc_off + w.acc_bytes);
    acc_v[1] = reinterpret_cast<float*>(ws + w.acc_off + 3 * w.acc_bytes);
  }

  // shard views of the natural-order bf16 tensors (box 64 columns x 128 rows)
  const bool striped = p.layout == RING_LAYOUT_STRIPED;
  const bool zigzag = p.layout == RING_LAYOUT_ZIGZAG;
  const cuuint64_t d = (cuuint64_t)p.d, n = (cuuint64_t)p.n, row_b = d * 2;
  CUtensorMap maps[4];
  const void* src[4] = {q, dout, k, v};
  const int BHkv = p.B * p.Hkv;
  for (int x = 0; x < 4; ++x) {
    const cuuint64_t heads = (cuuint64_t)(x < 2 ? BH : BHkv);  // q, dout: query heads; k, v: K/V heads
    if (striped) {
      cuuint64_t dims[4] = {d, (cuuint64_t)P, n, heads};
      cuuint64_t str[3] = {row_b, row_b * P, row_b * (cuuint64_t)p.N};
      if ((rc = encode_map(&maps[x], src[x], dims, str, 1, kTileM))) return rc;
    } else if (zigzag) {
      // chunks of n/2 tokens: dims (d, n/2, 2P, heads)
      cuuint64_t dims[4] = {d, n / 2, (cuuint64_t)(2 * P), heads};
      cuuint64_t str[3] = {row_b, row_b * (n / 2), row_b * (cuuint64_t)p.N};
      if ((rc = encode_map(&maps[x], src[x], dims, str, kTileM, 1))) return rc;
    } else {
      cuuint64_t dims[4] = {d, n, (cuuint64_t)P, heads};
      cuuint64_t str[3] = {row_b, row_b * n, row_b * (cuuint64_t)p.N};
      if ((rc = encode_map(&maps[x], src[x], dims, str, kTileM, 1))) return rc;
    }
  }
  const long long row_r = striped ? 1 : p.n, row_i = striped ? P : 1;
  const bool timing = h->timing != 0;
  if (timing) RA_CUDA(cudaEventRecord(h->tbp0, cs), "cudaEventRecord");
  RA_CUDA((cudaError_t)launch_bwd_prep(out, lse, dout, nlse2, nD, BH, p.n, w.n_pad, p.d, P, row_r, row_i, p.N,
                                       zigzag ? 1 : 0, cs),
          "backward prep launch");
  if (timing) RA_CUDA(cudaEventRecord(h->tbp1, cs), "cudaEventRecord");
  BwdArgs a;
  std::memset(&a, 0, sizeof a);
  if ((rc = device_segments(h, &a.seg_lo, &a.seg_hi))) return rc;
  a.nlse2 = nlse2;
  a.nD = nD;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.N = p.N;
  a.row_r = row_r;
  a.row_i = row_i;
  a.err = h->d_err;
  a.wait_limit_ns = h->wait_limit_ns;
  a.n = (int)p.n;
  a.n_pad = w.n_pad;
  a.P = P;
  a.BH = BH;
  a.BHkv = BHkv;
  a.G = p.H / p.Hkv;
  a.T = p.T;
  a.KT = p.KT;
  a.q_mode = striped ? kQStriped : (zigzag ? kQZigzag : kQContiguous);
  a.causal = p.causal;
  a.layout = p.layout;
  a.window = p.window;
  a.scale = (float)(1.0 / std::sqrt((double)p.d));
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p.d));
  if (lap) {
    // one launch per kernel: each CTA makes its tile's whole lap
    a.lap = 1;
    a.step = 0;
    a.accumulate = 0;
    a.last = 1;
    if (timing) RA_CUDA(cudaEventRecord(h->tbk0[0], cs), "cudaEventRecord");
    RA_CUDA((cudaError_t)launch_bwd_dkdv(a, &maps[0], &maps[1], &maps[2], &maps[3], p.d, cs), "backward dK/dV launch");
    if (timing) RA_CUDA(cudaEventRecord(h->tbk1[0], cs), "cudaEventRecord");
    if (timing) RA_CUDA(cudaEventRecord(h->tbq0[0], cs), "cudaEventRecord");
    RA_CUDA((cudaError_t)launch_bwd_dq(a, &maps[0], &maps[1], &maps[2], &maps[3], p.d, cs), "backward dQ launch");
    if (timing) RA_CUDA(cudaEventRecord(h->tbq1[0], cs), "cudaEventRecord");
  }
  for (int s = 0; s < P && !lap; ++s) {
    const int cur = s & 1;
    a.step = s;
    a.accumulate = s > 0 ? 1 : 0;
    a.last = s == P - 1 ? 1 : 0;
    a.acc_in_k = acc_k[cur];
    a.acc_in_v = acc_v[cur];
    a.acc_out_k = acc_k[cur ^ 1];
    a.acc_out_v = acc_v[cur ^ 1];
    if (timing) RA_CUDA(cudaEventRecord(h->tbk0[s], cs), "cudaEventRecord");
    RA_CUDA((cudaError_t)launch_bwd_dkdv(a, &maps[0], &maps[1], &maps[2], &maps[3], p.d, cs), "backward dK/dV launch");
    if (timing) RA_CUDA(cudaEventRecord(h->tbk1[s], cs), "cudaEventRecord");
    if (timing) RA_CUDA(cudaEventRecord(h->tbq0[s], cs), "cudaEventRecord");
    RA_CUDA((cudaError_t)launch_bwd_dq(a, &maps[0], &maps[1], &maps[2], &maps[3], p.d, cs), "backward dQ launch");
    if (timing) RA_CUDA(cudaEventRecord(h->tbq1[s], cs), "cudaEventRecord");
  }
  h->bwd_timed_valid = timing;
  h->bwd_timed_lap = lap;
  return RING_OK;
}

int ring_attn_get_bwd_timing(ring_attn_t h, float* dkdv_ms, float* dq_ms, float* prep_ms) {
  if (!h) return fail(RING_ERR_INVALID_ARG, "NULL handle");
  if (!h->ready || !h->bwd_timed_valid)
    return fail(RING_ERR_INVALID_ARG, "no timed backward (set RING_OPT_TIMING before ring_attn_bwd)");
  const int P = h->plan.P;
  const int timed = h->bwd_timed_lap ? 1 : P;  // lap mode: one launch each, in entry 0
  for (int s = 0; s < P; ++s) {
    if (s >= timed) {
      if (dkdv_ms) dkdv_ms[s] = 0.0f;
      if (dq_ms) dq_ms[s] = 0.0f;
      continue;
    }
    if (dkdv_ms) RA_CUDA(cudaEventElapsedTime(&dkdv_ms[s], h->tbk0[s], h->tbk1[s]), "cudaEventElapsedTime");
    if (dq_ms) RA_CUDA(cudaEventElapsedTime(&dq_ms[s], h->tbq0[s], h->tbq1[s]), "cudaEventElapsedTime");
  }
  if (prep_ms) RA_CUDA(cudaEventElapsedTime(prep_ms, h->tbp0, h->tbp1), "cudaEventElapsedTime");
  return RING_OK;
}

// ---------------------------------------------------------------- decode
// ring_attn_decode reads the cache in place, in natural order, as one block
// of N keys per K/V head (whatever the layout of the ring: its shards are a
// partition of these keys, and any partition merges to the same result).
// Short queries leave few CTAs, so the keys are cut into ksplit contiguous
// pieces, each piece of each query tile pair one CTA with a state of its
// own; merge_shards_kernel folds the ksplit states of each row exactly, by
// the same rule that folds the shards' states.  ksplit is the smallest
// count that fills at least 90 % of the SMs in whole waves (one wave of
// long pieces when the queries are few, so each CTA's set-up is paid once
// per SM), with at least 4 key tiles a piece.
// Workspace: m and l [ksplit][B][H][Lq] and O~ [ksplit][B][H][Lq][d] fp32.
static int decode_ksplit(const Plan& p, long long Lq) {
  const long long T = (Lq + kTileM - 1) / kTileM;
  const long long units = (long long)p.B * p.H * ((T + 1) / 2);
  const long long KT = ((long long)p.N + kTileN - 1) / kTileN;
  const long long cap = std::max(1LL, KT / 4);
  const long long sms = sm_count();
  for (long long ks = 1; ks <= cap; ++ks) {
    const long long ctas = units * ks, waves = (ctas + sms - 1) / sms;
    if (ctas * 10 >= sms * waves * 9) return (int)ks;
  }
  return (int)cap;
}

static size_t decode_ws(const Plan& p, long long Lq) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = (size_t)decode_ksplit(p, Lq) * p.B * p.H * (size_t)Lq;
  return up(rows * p.d * 4) + 2 * up(rows * 4);
}

int ring_attn_decode_workspace_size(ring_attn_t h, long long Lq, size_t* bytes) {
  if (!h || !bytes) return fail(RING_ERR_INVALID_ARG, "NULL argument");
  if (Lq < 1 || Lq > h->plan.N) return fail(RING_ERR_INVALID_ARG, "Lq must be in [1, N]");
  *bytes = decode_ws(h->plan, Lq);
  return RING_OK;
}

int ring_attn_decode(ring_attn_t h, const void* q, const void* k, const void* v, long long Lq, float* out,
                     float* lse, void* workspace, void* stream) {
  if (!h || !q || !k || !v || !out || !lse || !workspace) return fail(RING_ERR_INVALID_ARG, "NULL argument");
  const Plan& p = h->plan;
  if (Lq < 1 || Lq > p.N) return fail(RING_ERR_INVALID_ARG, "Lq must be in [1, N]");
  if (Lq > (1LL << 30)) return fail(RING_ERR_UNSUPPORTED, "Lq too large");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return fail(RING_ERR_INVALID_ARG, "tensor not 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(RING_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  int rc = ensure_device(h);
  if (rc) return rc;
  const int BH = p.B * p.H, BHkv = p.B * p.Hkv;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const cuuint64_t d = (cuuint64_t)p.d, Nn = (cuuint64_t)p.N, row_b = d * 2, lq = (cuuint64_t)Lq;
  CUtensorMap qm, km, vm;
  {
    cuuint64_t dims[4] = {d, lq, 1, (cuuint64_t)BH};
    cuuint64_t str[3] = {row_b, row_b * lq, row_b * lq};
    if ((rc = encode_map(&qm, q, dims, str, kTileM, 1))) return rc;
  }
  {
    // the cache in natural order, one block of N keys per K/V head: dims (d, N, BHkv, 1)
    cuuint64_t dims[4] = {d, Nn, (cuuint64_t)BHkv, 1};
    cuuint64_t str[3] = {row_b, row_b * Nn, row_b * Nn * (cuuint64_t)BHkv};
    if ((rc = encode_map(&km, k, dims, str, kTileN, 1))) return rc;
    if ((rc = encode_map(&vm, v, dims, str, kTileN, 1))) return rc;
  }
  const int ksplit = decode_ksplit(p, Lq);
  const size_t rows = (size_t)ksplit * BH * (size_t)Lq;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  float* o_st = reinterpret_cast<float*>(ws);
  float* m_st = reinterpret_cast<float*>(ws + up(rows * p.d * 4));
  float* l_st = reinterpret_cast<float*>(ws + up(rows * p.d * 4) + up(rows * 4));

  StepArgs a = base_args(h);
  if ((rc = device_segments(h, &a.seg_lo, &a.seg_hi))) return rc;
  // one contiguous block (P = 1): key k is at position k
  a.n = p.N;
  a.P = 1;
  a.KT = (int)((p.N + kTileN - 1) / kTileN);
  a.layout = RING_LAYOUT_CONTIGUOUS;
  a.o_state = o_st;  // the states of key piece x: rows [x][bh][i]
  a.m_state = m_st;
  a.l_state = l_st;
  a.out = nullptr;
  a.lse = nullptr;
  a.row_bh = Lq;
  a.row_r = (long long)BH * Lq;
  a.row_i = 1;
  a.nq = (int)Lq;
  a.T = (int)((Lq + kTileM - 1) / kTileM);
  a.decode_pos0 = p.N - Lq;
  a.q_mode = kQShardMajor;
  a.kv_mode = kKvSlotJ;  // block 0 of the one-block map
  a.ksplit = ksplit;
  a.step = 0;
  a.accumulate = 0;
  a.finalize = 0;
  a.n_active = 1;
  a.active[0] = 0;
  const int grid = block_partial_grid(a.T, 1, BH) * ksplit;
  RA_CUDA((cudaError_t)launch_block_partial(a, &qm, &km, &vm, p.d, grid, cs), "decode block launch");
  RA_CUDA((cudaError_t)launch_merge_shards(m_st, l_st, o_st, out, lse, (long long)BH * Lq, p.d, ksplit, cs),
          "decode merge launch");
  return RING_OK;
}

int ring_attn_get_timing(ring_attn_t h, float* kernel_ms, float* copy_ms, float* wait_ms, float* pack_ms) {
  if (!h) return fail(RING_ERR_INVALID_ARG, "NULL handle");
  const int n = h->t_count;
  if (n == 0) return fail(RING_ERR_INVALID_ARG, "no timed ring_attn_fwd recorded (set RING_OPT_TIMING)");
  const int P = h->plan.P;
  // elapsed time between two events of one set, synchronising on the later one
  auto elapsed = [](cudaEvent_t e0, cudaEvent_t e1, float* ms) -> int {
    RA_CUDA(cudaEventSynchronize(e1), "cudaEventSynchronize");
    RA_CUDA(cudaEventElapsedTime(ms, e0, e1), "cudaEventElapsedTime");
    return RING_OK;
  };
  int rc;
  for (int s = 0; s < P; ++s) {
    double k = 0, c = 0, w = 0;
    for (int x = 0; x < n; ++x) {
      const FwdTiming& T = h->tsets[x];
      const bool copied = s < (int)T.copied.size() && T.copied[s];
      float ms = 0.f;
      if (kernel_ms) {
        if ((rc = elapsed(T.k0[s], T.k1[s], &ms))) return rc;
        k += ms;
      }
      if (copy_ms && copied) {
        if ((rc = elapsed(T.c0[s], T.c1[s], &ms))) return rc;
        c += ms;
      }
      if (wait_ms && copied) {
        if ((rc = elapsed(T.w0[s], T.w1[s], &ms))) return rc;
        w += ms;
      }
    }
    if (kernel_ms) kernel_ms[s] = (float)(k / n);
    if (copy_ms) copy_ms[s] = (float)(c / n);
    if (wait_ms) wait_ms[s] = (float)(w / n);
  }
  if (pack_ms) {
    double pk = 0;
    for (int x = 0; x < n; ++x) {
      float ms = 0.f;
      if ((rc = elapsed(h->tsets[x].p0, h->tsets[x].p1, &ms))) return rc;
      pk += ms;
    }
    *pack_ms = (float)(pk / n);
  }
  h->t_read = true;
  return RING_OK;
}

int ring_attn_get_release_wait(ring_attn_t h, float* release_wait_ms) {
  if (!h || !release_wait_ms) return fail(RING_ERR_INVALID_ARG, "NULL argument");
  const int n = h->t_count;
  if (n == 0) return fail(RING_ERR_INVALID_ARG, "no timed ring_attn_fwd recorded (set RING_OPT_TIMING)");
  for (int s = 0; s < h->plan.P; ++s) {
    double sum = 0;
    for (int x = 0; x < n; ++x) {
      const FwdTiming& T = h->tsets[x];
      if (s < (int)T.copied.size() && T.copied[s]) {
        float ms = 0.f;
        RA_CUDA(cudaEventSynchronize(T.c0[s]), "cudaEventSynchronize");
        RA_CUDA(cudaEventElapsedTime(&ms, T.r0[s], T.c0[s]), "cudaEventElapsedTime");
        sum += ms;
      }
    }
    release_wait_ms[s] = (float)(sum / n);
  }
  h->t_read = true;
  return RING_OK;
}

int ring_attn_check(ring_attn_t h, void* stream) {
  if (!h) return fail(RING_ERR_INVALID_ARG, "NULL handle");
  if (!h->ready) return RING_OK;
  RA_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "cudaStreamSynchronize");
  RA_CUDA(cudaStreamSynchronize(h->side), "cudaStreamSynchronize");
  if (h->pipe) {
    // ring_attn_fwd_host: its copy streams, its second lane, and the group
    // handles' kernels
    for (cudaStream_t st : {h->pipe->in, h->pipe->out, h->pipe->lane1})
      RA_CUDA(cudaStreamSynchronize(st), "cudaStreamSynchronize");
    for (ring_attn* sub : h->pipe->subs) {
      int rc = ring_attn_check(sub, stream);
      if (rc) return rc;
    }
  }
  int words[2] = {0, 0};
  RA_CUDA(cudaMemcpy(words, h->d_err, sizeof words, cudaMemcpyDeviceToHost), "cudaMemcpy(error word)");
  if (words[0] != 0) {
    RA_CUDA(cudaMemset(h->d_err, 0, sizeof words), "cudaMemset");
    char buf[128];
    std::snprintf(buf, sizeof buf, "device-side wait ran out (flags 0x%x, site %d)", words[0], words[1]);
    return fail(RING_ERR_TIMEOUT, buf);
  }
  return RING_OK;
}

}  // extern "C"
