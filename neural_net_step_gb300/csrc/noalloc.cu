// mlp_op_wgrad_noalloc: the weight-gradient operation of mlp_op_wgrad for
// callers that cannot hand the library a workspace.
//
// Some callers cannot call cudaMalloc: an application whose device memory is
// owned by another allocator (a framework's caching pool, a fixed up-front
// reservation) has no way to obtain an extra buffer, and a latency-critical
// loop must not call cudaMalloc/cudaFree at all, since both may synchronise
// the device and can fail under memory pressure.  For them, this entry point
// keeps the split-K partial sums in a file-scope device array of fixed size
// instead of a caller-supplied workspace; it allocates nothing.
#include <stdio.h>

#include <map>
#include <mutex>

#include "common.cuh"
#include "mlp.h"
#include "mlp_ops.h"
#include "ops.h"

using namespace mlpk;

namespace {

// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kScratchBytes = size_t(16) << 20;   // 16 MiB
static __device__ __align__(256) float g_wgrad_scratch[kScratchBytes / sizeof(float)];

// Reports through mlp_last_error() (defined with the rest of the C ABI).
mlp_status noalloc_fail(mlp_status st, const char* msg) {
  mlpk::set_last_error(msg);
  return st;
}

// In host code `g_wgrad_scratch` names a host-side stand-in, not a device
// address.  The device address is looked up with the device current: on the
// first call on each device (which should come before any stream capture),
// and again on every later call whose stream is not capturing, so that the
// address stays right after cudaDeviceReset tears the context down and a new
// one loads the module elsewhere.  A call on a capturing stream makes no
// lookup and reuses the address the last lookup on that device found.
std::mutex g_mu;
std::map<int, void*> g_addr;

cudaError_t scratch_address(cudaStream_t stream, void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_addr.find(dev);
  if (cs != cudaStreamCaptureStatusNone) {
    if (it == g_addr.end()) return cudaErrorStreamCaptureUnsupported;   // no set-up call before the capture
    *out = it->second;
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_wgrad_scratch);
  if (e != cudaSuccess) return e;
  g_addr[dev] = p;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" {

mlp_status mlp_op_wgrad_noalloc(int dtype, int64_t N, int64_t K, int64_t B, const void* dY, int64_t ldy,
                                const void* X, int64_t ldx, float* dW, int64_t lddw, float* db, uint32_t* err_dev,
                                void* stream) {
  if (dtype != MLP_F32 && dtype != MLP_BF16 && dtype != MLP_F32X3) return noalloc_fail(MLP_ERR_DTYPE, "bad dtype");
  if (!dY || !X || !dW) return noalloc_fail(MLP_ERR_ARG, "null pointer");
  if (N < 1 || K < 1 || B < 1 || ldy < N || ldx < K || lddw < K)
    return noalloc_fail(MLP_ERR_SHAPE, "bad shape or leading dimension");
  char msg[512];
  const int splits = wgrad_splits(dtype, N, K, B);
  const size_t need = wgrad_workspace_bytes(dtype, N, K, B, splits);
  if (need > kScratchBytes) {
    snprintf(msg, sizeof(msg),
             "wgrad %lld x %lld over %lld rows needs %zu bytes of scratch; the built-in scratch holds %zu",
             (long long)N, (long long)K, (long long)B, need, kScratchBytes);
    return noalloc_fail(MLP_ERR_SHAPE, msg);
  }
  void* scratch = nullptr;
  if (need > 0) {
    cudaError_t e = scratch_address((cudaStream_t)stream, &scratch);
    if (e != cudaSuccess) {
      snprintf(msg, sizeof(msg), "scratch address lookup: %s%s", cudaGetErrorString(e),
               e == cudaErrorStreamCaptureUnsupported ? " (make one call on this device before capturing)" : "");
      return noalloc_fail(MLP_ERR_CUDA, msg);
    }
  }
  GemmOp op;
  op.dtype = dtype; op.kind = GEMM_WGRAD;
  op.a_plane = B * ldy; op.b_plane = B * ldx;   // MLP_F32X3: the three planes of each operand
  op.M = N; op.N = K; op.K = B;
  op.A = dY; op.lda = ldy; op.a_kmajor = false;
  op.B = X; op.ldb = ldx; op.b_kmajor = false;
  op.dW = dW; op.ld_dw = lddw; op.db = db;
  op.ws = (float*)scratch; op.ws_bytes = need > 0 ? kScratchBytes : 0;
  op.splits = splits;
  op.err = err_dev;
  LaunchRec r[2];
  int n = gemm_plan(op, r, msg, sizeof(msg));
  if (n < 0) return noalloc_fail(MLP_ERR_SHAPE, msg);
  for (int i = 0; i < n; ++i) {
    cudaError_t e = launch_rec(r[i], (cudaStream_t)stream);
    if (e != cudaSuccess) {
      snprintf(msg, sizeof(msg), "launch of %s failed: %s", r[i].name, cudaGetErrorString(e));
      return noalloc_fail(MLP_ERR_CUDA, msg);
    }
  }
  mlpk::set_last_error("");
  return MLP_OK;
}

}  // extern "C"
