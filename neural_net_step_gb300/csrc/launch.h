// A kernel launch described as data, so that the same step can be launched
// eagerly on a stream or recorded as nodes of an explicitly built CUDA graph
// (and re-pointed later by updating a node's arguments).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

namespace mlpk {

constexpr unsigned kMaxArgBytes = 1024;

struct LaunchRec {
  const void* func = nullptr;
  dim3 grid{1, 1, 1};
  dim3 block{1, 1, 1};
  unsigned smem = 0;
  unsigned args_size = 0;
  const char* name = "";
  // Graph dependencies: indices of earlier records in the same plan that this
  // launch must follow; ndeps < 0 means "the record just before it".  Eager
  // launches run the records in order and ignore this.
  static constexpr int kMaxDeps = 4;
  int deps[kMaxDeps] = {0, 0, 0, 0};
  int ndeps = -1;
  // May be scheduled before its predecessor ends (programmatic edge from the
  // first dependency): worth it for kernels with a real prologue (barriers,
  // TMEM) and at most one wave of CTAs.  Kernels of many small CTAs would
  // crowd onto the SMs the predecessor leaves idle and then run there, so
  // they keep full edges.
  bool early = false;
  // Tensors this launch writes that a traced step copies aside (the step's
  // intermediate results; the graph and eager paths ignore them).
  struct Out {
    int kind = 0, layer = 0;        // MLP_TRACE_* and the layer it belongs to
    const void* ptr = nullptr;
    int64_t rows = 0, cols = 0, ld = 0, plane_stride = 0;
    int planes = 1, elem_bytes = 0;
  };
  static constexpr int kMaxOuts = 2;
  Out outs[kMaxOuts];
  int nouts = 0;
  alignas(128) unsigned char args[kMaxArgBytes];

  void add_out(int kind, int layer, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int elem_bytes,
               int planes = 1, int64_t plane_stride = 0) {
    if (nouts >= kMaxOuts) return;
    Out& o = outs[nouts++];
    o.kind = kind; o.layer = layer; o.ptr = ptr;
    o.rows = rows; o.cols = cols; o.ld = ld; o.elem_bytes = elem_bytes;
    o.planes = planes; o.plane_stride = plane_stride;
  }

  void depend_on(const int* d, int n) {
    ndeps = 0;
    for (int i = 0; i < n; ++i)
      if (d[i] >= 0 && ndeps < kMaxDeps) deps[ndeps++] = d[i];
  }
  bool same_deps(const LaunchRec& o) const {
    if (ndeps != o.ndeps) return false;
    for (int i = 0; i < ndeps; ++i)
      if (deps[i] != o.deps[i]) return false;
    return true;
  }

  template <typename P>
  void set_args(const P& p) {
    static_assert(sizeof(P) <= kMaxArgBytes, "kernel parameter block too large");
    static_assert(alignof(P) <= 128, "over-aligned kernel parameter block");
    memcpy(args, &p, sizeof(P));
    args_size = sizeof(P);
  }
  bool same_as(const LaunchRec& o) const {
    return func == o.func && grid.x == o.grid.x && grid.y == o.grid.y && grid.z == o.grid.z &&
           block.x == o.block.x && block.y == o.block.y && block.z == o.block.z &&
           smem == o.smem && args_size == o.args_size && memcmp(args, o.args, args_size) == 0;
  }
};

inline cudaError_t launch_rec(const LaunchRec& r, cudaStream_t s) {
  void* argp[1] = {const_cast<unsigned char*>(r.args)};
  return cudaLaunchKernel(r.func, r.grid, r.block, argp, r.smem, s);
}

inline cudaKernelNodeParams node_params(const LaunchRec& r, void** argp) {
  cudaKernelNodeParams kp;
  memset(&kp, 0, sizeof(kp));
  kp.func = const_cast<void*>(r.func);
  kp.gridDim = r.grid;
  kp.blockDim = r.block;
  kp.sharedMemBytes = r.smem;
  argp[0] = const_cast<unsigned char*>(r.args);
  kp.kernelParams = argp;
  kp.extra = nullptr;
  return kp;
}

}  // namespace mlpk
