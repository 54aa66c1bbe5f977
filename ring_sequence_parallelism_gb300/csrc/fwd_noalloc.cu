// fwd_noalloc.cu -- ring_attn_fwd_noalloc: the ring forward for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a plug-in running inside a host
// application that owns every byte of device memory through its own pool
// and forbids libraries from allocating, or code on a latency-critical path
// where cudaMalloc/cudaFree may synchronise the whole device.  ring_attn_fwd
// needs scratch memory beyond its inputs and outputs (the shard-major K/V
// buffer the step kernels read, and the running l state), which its callers
// pass in as a workspace they allocated.  This entry point keeps that
// scratch in a file-scope __device__ array instead, so the call itself
// allocates nothing.
//
// Differences from ring_attn_fwd, all deliberate:
//   - the scratch is the fixed array below (kScratchBytes = 64 MiB): every
//     GPU that loads the library holds it until the process exits, and a
//     problem whose scratch does not fit is rejected with
//     RING_ERR_UNSUPPORTED;
//   - every step reads its K/V block straight from the packed buffer (no
//     double-buffered rotation, so no side stream and no events are needed;
//     the results are the same bit for bit);
//   - the device-side error word lives in the same array and is copied to
//     the caller's `status` (a device int) at the end of the call.
// Every call shares the array: calls that overlap on the GPU (on different
// streams, or from different threads) race on it and must be serialised by
// the caller.  The error word is cleared at the start of each call; the
// packed K/V and the l state are fully written before they are read.
//
// Set-up: the first call on each device, with that device current, checks
// the device, sets the kernels' shared-memory limit and takes the array's
// device address with cudaGetSymbolAddress (host code cannot use the
// array's name as a device address).  That first call should come before
// any stream capture.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace ringattn {
namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr size_t kErrBytes = 256;                   // error words [0] flags, [1] site
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceSetup {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
};

std::mutex g_setup_mutex;
DeviceSetup g_setup[kMaxDevices];

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

int cuda_error(cudaError_t e, const char* what) {
  char buf[160];
  std::snprintf(buf, sizeof buf, "%s: %s", what, cudaGetErrorString(e));
  cudaGetLastError();
  return report_error(RING_ERR_CUDA, buf);
}

// Once per device, with the device current.
int setup_device(int dev, unsigned char** scratch) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSetup& s = g_setup[dev];
  if (!s.ready) {
    int major = 0, minor = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3) {
      char buf[96];
      std::snprintf(buf, sizeof buf, "this library is built for sm_103a; device %d is sm_%d%d", dev, major, minor);
      return report_error(RING_ERR_UNSUPPORTED, buf);
    }
    e = (cudaError_t)prepare_block_partial_kernels();
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute");
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) return cuda_error(e, "cudaGetSymbolAddress(scratch)");
    s.scratch = static_cast<unsigned char*>(ptr);
    s.ready = true;
  }
  *scratch = s.scratch;
  return RING_OK;
}

bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

}  // namespace
}  // namespace ringattn

using namespace ringattn;

extern "C" int ring_attn_fwd_noalloc(ring_attn_t h, const void* q, const void* k, const void* v, float* out,
                                     float* lse, int* status, void* stream) {
  if (!h || !q || !k || !v || !out || !lse) return report_error(RING_ERR_INVALID_ARG, "NULL argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) ||
      (status && reinterpret_cast<uintptr_t>(status) % 4 != 0))
    return report_error(RING_ERR_INVALID_ARG, "tensor not 16-byte aligned");
  const Plan& p = handle_plan(h);
  if (!p.seg_bounds.empty())
    return report_error(RING_ERR_UNSUPPORTED,
                        "segments need a device table of document bounds; use ring_attn_fwd");
  const int P = p.P, BH = p.B * p.H, BHkv = p.B * p.Hkv;
  const size_t elems = (size_t)BHkv * (size_t)p.N * p.d;  // one of K, V (K/V heads)
  const size_t kv_bytes = round256(elems * 2);
  const size_t l_bytes = round256((size_t)BH * (size_t)p.N * 4);
  const size_t need = kErrBytes + 2 * kv_bytes + l_bytes;
  if (need > kScratchBytes) {
    char buf[240];
    // per query row (B*H*N of them): its l (4 bytes) and 1/G of a K/V head
    // row of K and V (2 tensors x d bf16 values), G query heads per K/V head
    const size_t G = (size_t)(p.H / p.Hkv);
    const size_t max_rows = (kScratchBytes - kErrBytes - 3 * 256) * G / (4 * G + (size_t)p.d * 4);
    std::snprintf(buf, sizeof buf,
                  "ring_attn_fwd_noalloc: this problem needs %zu bytes of scratch, more than the fixed %zu-byte "
                  "array (B*H*N up to about %zu at d=%d with %zu query heads per K/V head); use ring_attn_fwd "
                  "with a workspace",
                  need, kScratchBytes, max_rows, p.d, G);
    return report_error(RING_ERR_UNSUPPORTED, buf);
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return report_error(RING_ERR_UNSUPPORTED, "device index above 63");
  unsigned char* scratch = nullptr;
  int rc = setup_device(dev, &scratch);
  if (rc) return rc;

  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  int* err = reinterpret_cast<int*>(scratch);
  unsigned char* kbuf = scratch + kErrBytes;
  unsigned char* vbuf = kbuf + kv_bytes;
  float* l_state = reinterpret_cast<float*>(vbuf + kv_bytes);
  e = cudaMemsetAsync(err, 0, 2 * sizeof(int), cs);
  if (e != cudaSuccess) return cuda_error(e, "cudaMemsetAsync(error word)");

  // TMA maps: Q in natural order (strided per shard), packed K/V slot j = block j
  const unsigned long long d = (unsigned long long)p.d, n = (unsigned long long)p.n, row_b = d * 2;
  alignas(64) unsigned char qm[128], km[128], vm[128];
  if (p.layout == RING_LAYOUT_STRIPED) {
    unsigned long long dims[4] = {d, (unsigned long long)P, n, (unsigned long long)BH};
    unsigned long long str[3] = {row_b, row_b * P, row_b * (unsigned long long)p.N};
    if ((rc = tensor_map_4d(qm, q, dims, str, 1, kTileM))) return rc;
  } else if (p.layout == RING_LAYOUT_ZIGZAG) {
    unsigned long long dims[4] = {d, n / 2, 2ULL * P, (unsigned long long)BH};
    unsigned long long str[3] = {row_b, row_b * (n / 2), row_b * (unsigned long long)p.N};
    if ((rc = tensor_map_4d(qm, q, dims, str, kTileM, 1))) return rc;
  } else {
    unsigned long long dims[4] = {d, n, (unsigned long long)P, (unsigned long long)BH};
    unsigned long long str[3] = {row_b, row_b * n, row_b * (unsigned long long)p.N};
    if ((rc = tensor_map_4d(qm, q, dims, str, kTileM, 1))) return rc;
  }
  {
    unsigned long long dims[4] = {d, n, (unsigned long long)BHkv, (unsigned long long)P};
    unsigned long long str[3] = {row_b, row_b * n, row_b * n * BHkv};
    if ((rc = tensor_map_4d(km, kbuf, dims, str, kTileN, 1))) return rc;
    if ((rc = tensor_map_4d(vm, vbuf, dims, str, kTileN, 1))) return rc;
  }

  e = (cudaError_t)launch_pack_kv(k, v, kbuf, vbuf, BHkv, p.n, p.d, P, p.layout, cs);
  if (e != cudaSuccess) return cuda_error(e, "pack launch");

  StepArgs a;
  std::memset(&a, 0, sizeof a);
  a.o_state = out;  // O~ lives in `out` between steps
  a.m_state = lse;  // m lives in `lse` between steps
  a.l_state = l_state;
  a.out = out;
  a.lse = lse;
  a.row_bh = p.N;
  a.row_r = p.layout == RING_LAYOUT_STRIPED ? 1 : p.n;
  a.row_i = p.layout == RING_LAYOUT_STRIPED ? P : 1;
  a.err = err;
  a.wait_limit_ns = handle_wait_limit(h);
  a.debug_drop_v = handle_debug_drop_v(h);  // the bounded-wait test hook, as in ring_attn_fwd
  a.n = (int)p.n;
  a.P = P;
  a.BH = BH;
  a.G = p.H / p.Hkv;
  a.nq = (int)p.n;
  a.decode_pos0 = -1;
  a.window = p.window;
  a.T = p.T;
  a.KT = p.KT;
  a.q_mode = p.layout == RING_LAYOUT_STRIPED ? kQStriped : (p.layout == RING_LAYOUT_ZIGZAG ? kQZigzag : kQContiguous);
  a.kv_mode = kKvSlotJ;
  a.causal = p.causal;
  a.layout = p.layout;
  a.fixed_r = -1;
  a.ksplit = 1;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p.d));
  for (int s = 0; s < P; ++s) {
    const auto& act = p.active[s];
    a.step = s;
    a.accumulate = s > 0 ? 1 : 0;
    a.finalize = s == P - 1 ? 1 : 0;
    a.n_active = (int)act.size();
    for (size_t x = 0; x < act.size(); ++x) a.active[x] = act[x];
    e = (cudaError_t)launch_block_partial(a, qm, km, vm, p.d, block_partial_grid(p.T, a.n_active, BH), cs);
    if (e != cudaSuccess) return cuda_error(e, "step kernel launch");
  }
  if (status) {
    e = cudaMemcpyAsync(status, err, sizeof(int), cudaMemcpyDeviceToDevice, cs);
    if (e != cudaSuccess) return cuda_error(e, "cudaMemcpyAsync(status)");
  }
  return RING_OK;
}
