// Bandwidth-bound kernels of the step: the one-pass softmax cross-entropy
// (forward loss and backward dz from a single read of each logits row, the
// fused form described on devpost "Orthon", "Selected Orthon vs. PyTorch
// results"), the batch-mean loss, the flat multi-tensor AdamW update over
// co-located parameter/gradient/moment planes (noeira.ai "Neural networks",
// "The design in one page": a Param is four tensors), the row argmax, and
// small copies.
#include <math.h>
#include <stdio.h>

#include "common.cuh"
#include "ops.h"

namespace mlpk {

// ---------------------------------------------------------------------------
// Softmax cross-entropy.
//   m = max_j z_j;  s = sum_j exp(z_j - m);  loss_i = m + log(s) - z[y_i];
//   dz_j = (exp(z_j - m) / s - [j == y_i]) * grad_scale.
// ---------------------------------------------------------------------------
struct CeParams {
  const void* z; int64_t ldz;
  const int32_t* labels;
  void* dz; int64_t lddz;
  float* loss_rows;
  int B, C;
  float grad_scale;
  uint32_t* err;
};

template <typename T>
__device__ __forceinline__ void ce_finish_row(const CeParams& p, int row, int y, float m, float s,
                                              bool bad_label, int lane_or_tid) {
  if (lane_or_tid == 0) {
    const T* zr = reinterpret_cast<const T*>(p.z) + (int64_t)row * p.ldz;
    float zy = bad_label ? 0.f : to_f32(zr[y]);
    p.loss_rows[row] = bad_label ? 0.f : (m + logf(s)) - zy;
    if (bad_label && p.err) atomicOr(p.err, ERRBIT_LABEL_RANGE);
  }
}

// Four consecutive elements as fp32 (16-byte fp32 / 8-byte bf16 accesses).
template <typename T>
__device__ __forceinline__ void load4(const T* src, float* v) {
  if constexpr (sizeof(T) == 4) {
    const float4 a = *reinterpret_cast<const float4*>(src);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  } else {
    const uint2 a = *reinterpret_cast<const uint2*>(src);
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&a.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&a.y);
    v[0] = __low2float(lo); v[1] = __high2float(lo); v[2] = __low2float(hi); v[3] = __high2float(hi);
  }
}
template <typename T>
__device__ __forceinline__ void store4(T* dst, const float* v) {
  if constexpr (sizeof(T) == 4) {
    *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
  } else {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&lo);
    o.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = o;
  }
}

// One warp per row; the row lives in registers (C <= 32 * VPL).
template <typename T, int VPL>
__global__ void __launch_bounds__(256) ce_warp_kernel(const __grid_constant__ CeParams p) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= p.B) return;
  const T* zr = reinterpret_cast<const T*>(p.z) + (int64_t)row * p.ldz;
  float v[VPL];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    int j = lane + 32 * i;
    v[i] = j < p.C ? to_f32(zr[j]) : -INFINITY;
    m = fmaxf(m, v[i]);
  }
  m = warp_max(m);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    int j = lane + 32 * i;
    v[i] = j < p.C ? __expf(v[i] - m) : 0.f;
    s += v[i];
  }
  s = warp_sum(s);
  const int y = p.labels[row];
  const bool bad = y < 0 || y >= p.C;
  const float inv_s = 1.0f / s;
  T* dr = reinterpret_cast<T*>(p.dz) + (int64_t)row * p.lddz;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    int j = lane + 32 * i;
    if (j < p.C) dr[j] = from_f32<T>((v[i] * inv_s - (j == y ? 1.f : 0.f)) * p.grad_scale);
  }
  ce_finish_row<T>(p, row, y, m, s, bad, lane);
}

// One warp per row with 4 consecutive elements a lane (C % 4 == 0, rows
// 8- / 16-byte aligned; C <= 128 * SLOTS): one vector load and store per
// lane and slot; exp(z - m) = 2^(z log2e - m log2e) (one FFMA, one ex2).
__device__ __forceinline__ float pow2_approx(float t);
constexpr float kLog2e = 1.4426950408889634f;

template <typename T, int SLOTS>
__global__ void __launch_bounds__(256) ce_warp4_kernel(const __grid_constant__ CeParams p) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= p.B) return;
  const T* zr = reinterpret_cast<const T*>(p.z) + (int64_t)row * p.ldz;
  float v[SLOTS][4];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    const int j = 4 * lane + 128 * i;
    if (j < p.C) {
      load4<T>(zr + j, v[i]);
    } else {
      v[i][0] = v[i][1] = v[i][2] = v[i][3] = -INFINITY;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) m = fmaxf(m, v[i][k]);
  }
  const int y = p.labels[row];
  m = warp_max(m);
  const float ml = m * kLog2e;
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < SLOTS; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[i][k] = 4 * lane + 128 * i < p.C ? pow2_approx(fmaf(v[i][k], kLog2e, -ml)) : 0.f;
      s += v[i][k];
    }
  s = warp_sum(s);
  const bool bad = y < 0 || y >= p.C;
  const float a = (1.0f / s) * p.grad_scale;
  T* dr = reinterpret_cast<T*>(p.dz) + (int64_t)row * p.lddz;
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    const int j = 4 * lane + 128 * i;
    if (j < p.C) {
      float d[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) d[k] = v[i][k] * a - (j + k == y ? p.grad_scale : 0.f);
      store4<T>(dr + j, d);
    }
  }
  ce_finish_row<T>(p, row, y, m, s, bad, lane);
}

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = is_max ? warp_max(v) : warp_sum(v);
  __syncthreads();   // protect red from a previous use
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float r = lane < nw ? red[lane] : (is_max ? -INFINITY : 0.f);
  r = is_max ? warp_max(r) : warp_sum(r);
  return r;
}

// One CTA per row, the row held in registers as 16-byte vectors:
// C % (16 / sizeof(T)) == 0 and C <= blockDim * VPT * (16 / sizeof(T)).
template <typename T, int VPT>
__global__ void __launch_bounds__(512) ce_block_kernel(const __grid_constant__ CeParams p) {
  pdl_enter();
  constexpr int E = 16 / sizeof(T);   // elements per vector
  __shared__ float red[32];
  const int row = blockIdx.x;
  const int nvec = p.C / E;
  const uint4* zr = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.z) + (int64_t)row * p.ldz);
  uint4 raw[VPT];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    int vi = threadIdx.x + i * blockDim.x;
    if (vi < nvec) {
      raw[i] = __ldg(zr + vi);
      const T* e = reinterpret_cast<const T*>(&raw[i]);
#pragma unroll
      for (int k = 0; k < E; ++k) m = fmaxf(m, to_f32(e[k]));
    }
  }
  m = block_reduce(m, true, red);
  // e = exp(z - m), computed once and kept in registers (__expf: one MUFU op)
  float ex[VPT][E];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    int vi = threadIdx.x + i * blockDim.x;
    const T* e = reinterpret_cast<const T*>(&raw[i]);
#pragma unroll
    for (int k = 0; k < E; ++k) {
      ex[i][k] = vi < nvec ? __expf(to_f32(e[k]) - m) : 0.f;
      s += ex[i][k];
    }
  }
  s = block_reduce(s, false, red);
  const int y = p.labels[row];
  const bool bad = y < 0 || y >= p.C;
  const float inv_s = 1.0f / s;
  uint4* dr = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.dz) + (int64_t)row * p.lddz);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    int vi = threadIdx.x + i * blockDim.x;
    if (vi < nvec) {
      uint4 o;
      T* oe = reinterpret_cast<T*>(&o);
#pragma unroll
      for (int k = 0; k < E; ++k) {
        int j = vi * E + k;
        oe[k] = from_f32<T>((ex[i][k] * inv_s - (j == y ? 1.f : 0.f)) * p.grad_scale);
      }
      dr[vi] = o;
    }
  }
  ce_finish_row<T>(p, row, y, m, s, bad, threadIdx.x);
}

// Large C with 16-byte vectors, register-light: one CTA of 256 threads per
// row.  Pass 1 reads the row once from HBM (per-thread max, then one exp per
// element for the per-thread sum, combined across the CTA); pass 2 re-reads
// the row -- now resident in L2 -- and writes dz.  HBM sees one read and one
// write per element; several rows are in flight per SM.
template <typename T>
__device__ __forceinline__ void ms_combine(float& m, float& s, float m2, float s2) {
  const float mm = fmaxf(m, m2);
  s = (m == -INFINITY ? 0.f : s * __expf(m - mm)) + (m2 == -INFINITY ? 0.f : s2 * __expf(m2 - mm));
  m = mm;
}

// 2^t by the hardware's base-2 exponential (PTX ex2.approx, subnormal
// results flushed to zero); exp(x) = 2^(x log2 e), so the wide-row kernel
// forms exp(z - m) as one FFMA (z log2e - m log2e) and one ex2.
__device__ __forceinline__ float pow2_approx(float t) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
  return r;
}

template <typename T>
__global__ void __launch_bounds__(256) ce_row2_kernel(const __grid_constant__ CeParams p) {
  pdl_enter();
  constexpr int E = 16 / sizeof(T);
  __shared__ float red_m[8], red_s[8];
  const int row = blockIdx.x;
  const int nvec = p.C / E;
  const uint4* zr = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.z) + (int64_t)row * p.ldz);
  // four 16-byte loads in flight per thread (one is not enough to cover HBM
  // latency at this occupancy), consumed in index order
  constexpr int U = 4;
  float m = -INFINITY, s = 0.f;
  for (int v0 = threadIdx.x; v0 < nvec; v0 += 256 * U) {
    uint4 raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (v0 + 256 * u < nvec) raw[u] = zr[v0 + 256 * u];   // kept in L2 for the second pass
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (v0 + 256 * u >= nvec) break;
      const T* e = reinterpret_cast<const T*>(&raw[u]);
      float vmax = -INFINITY;
#pragma unroll
      for (int k = 0; k < E; ++k) vmax = fmaxf(vmax, to_f32(e[k]));
      const float vml = vmax * kLog2e;
      float vs = 0.f;
#pragma unroll
      for (int k = 0; k < E; ++k) vs += pow2_approx(fmaf(to_f32(e[k]), kLog2e, -vml));
      ms_combine<T>(m, s, vmax, vs);
    }
  }
  // combine (max, sum) across the CTA in a fixed order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    ms_combine<T>(m, s, m2, s2);
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) { red_m[wid] = m; red_s[wid] = s; }
  __syncthreads();
  m = red_m[0];
  s = red_s[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) ms_combine<T>(m, s, red_m[w], red_s[w]);
  const int y = p.labels[row];
  const bool bad = y < 0 || y >= p.C;
  // dz = exp(z - m) (1/s) grad_scale, minus grad_scale at the label (one
  // element of the row, fixed up in the vector that holds it)
  const float a = (1.0f / s) * p.grad_scale, ml = m * kLog2e;
  const int yv = y / E, yk = y - yv * E;
  uint4* dr = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.dz) + (int64_t)row * p.lddz);
  for (int v0 = threadIdx.x; v0 < nvec; v0 += 256 * U) {
    uint4 raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (v0 + 256 * u < nvec) raw[u] = __ldcs(zr + v0 + 256 * u);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int vi = v0 + 256 * u;
      if (vi >= nvec) break;
      const T* e = reinterpret_cast<const T*>(&raw[u]);
      float d[E];
#pragma unroll
      for (int k = 0; k < E; ++k) d[k] = pow2_approx(fmaf(to_f32(e[k]), kLog2e, -ml)) * a;
      if (vi == yv) {
#pragma unroll
        for (int k = 0; k < E; ++k)
          if (k == yk) d[k] -= p.grad_scale;
      }
      uint4 o;
      T* oe = reinterpret_cast<T*>(&o);
#pragma unroll
      for (int k = 0; k < E; ++k) oe[k] = from_f32<T>(d[k]);
      __stcs(dr + vi, o);
    }
  }
  ce_finish_row<T>(p, row, y, m, s, bad, threadIdx.x);
}

// Any C: one CTA per row, three passes over the row (max, sum, write).
template <typename T>
__global__ void __launch_bounds__(256) ce_generic_kernel(const __grid_constant__ CeParams p) {
  pdl_enter();
  __shared__ float red[32];
  const int row = blockIdx.x;
  const T* zr = reinterpret_cast<const T*>(p.z) + (int64_t)row * p.ldz;
  float m = -INFINITY;
  for (int j = threadIdx.x; j < p.C; j += blockDim.x) m = fmaxf(m, to_f32(zr[j]));
  m = block_reduce(m, true, red);
  float s = 0.f;
  for (int j = threadIdx.x; j < p.C; j += blockDim.x) s += expf(to_f32(zr[j]) - m);
  s = block_reduce(s, false, red);
  const int y = p.labels[row];
  const bool bad = y < 0 || y >= p.C;
  const float inv_s = 1.0f / s;
  T* dr = reinterpret_cast<T*>(p.dz) + (int64_t)row * p.lddz;
  for (int j = threadIdx.x; j < p.C; j += blockDim.x)
    dr[j] = from_f32<T>((expf(to_f32(zr[j]) - m) * inv_s - (j == y ? 1.f : 0.f)) * p.grad_scale);
  ce_finish_row<T>(p, row, y, m, s, bad, threadIdx.x);
}

template <typename T>
static int ce_plan_t(const CeOp& op, LaunchRec* rec, const CeParams& q) {
  constexpr int E = 16 / sizeof(T);
  const int64_t C = op.C;
  rec->smem = 0;
  rec->name = "softmax_ce";
  const bool vec4 = C % 4 == 0 && op.ldz % 4 == 0 && op.lddz % 4 == 0 && (uintptr_t)op.z % (4 * sizeof(T)) == 0 &&
                    (uintptr_t)op.dz % (4 * sizeof(T)) == 0;
  if (C <= 32 * 8 && vec4) {
    rec->block = dim3(256);
    rec->grid = dim3((unsigned)ceil_div(op.B, 8));
    rec->func = C <= 128 ? (const void*)ce_warp4_kernel<T, 1> : (const void*)ce_warp4_kernel<T, 2>;
  } else if (C <= 32 * 8) {
    rec->block = dim3(256);
    rec->grid = dim3((unsigned)ceil_div(op.B, 8));
    if (C <= 32) rec->func = (const void*)ce_warp_kernel<T, 1>;
    else if (C <= 64) rec->func = (const void*)ce_warp_kernel<T, 2>;
    else if (C <= 128) rec->func = (const void*)ce_warp_kernel<T, 4>;
    else rec->func = (const void*)ce_warp_kernel<T, 8>;
  } else {
    const bool vec_ok = (C % E == 0) && (op.ldz % E == 0) && (op.lddz % E == 0) &&
                        ((uintptr_t)op.z % 16 == 0) && ((uintptr_t)op.dz % 16 == 0);
    const int64_t nvec = C / E;
    rec->grid = dim3((unsigned)op.B);
    if (vec_ok && nvec > 256 * 4) {
      rec->block = dim3(256);
      rec->func = (const void*)ce_row2_kernel<T>;
    } else if (vec_ok && nvec <= 512 * 8) {
      rec->block = dim3(nvec <= 128 * 8 ? 128 : nvec <= 256 * 8 ? 256 : 512);
      rec->func = (const void*)ce_block_kernel<T, 8>;
    } else {
      rec->block = dim3(256);
      rec->func = (const void*)ce_generic_kernel<T>;
    }
  }
  rec->set_args(q);
  return 1;
}

int ce_plan(const CeOp& op, LaunchRec* rec, char* err, size_t errlen) {
  if (op.B <= 0 || op.C <= 0 || op.B > INT32_MAX || op.C > INT32_MAX || op.ldz < op.C || op.lddz < op.C) {
    snprintf(err, errlen, "softmax_ce: bad shape B=%lld C=%lld", (long long)op.B, (long long)op.C);
    return -1;
  }
  CeParams q{op.z, op.ldz, op.labels, op.dz, op.lddz, op.loss_rows, (int)op.B, (int)op.C, op.grad_scale, op.err};
  if (op.dtype == DT_F32) return ce_plan_t<float>(op, rec, q);
  return ce_plan_t<__nv_bfloat16>(op, rec, q);
}

// ---------------------------------------------------------------------------
// Squared error against real targets (the MSE loss):
//   d = z - t;  loss_rows[i] = sum_j d_ij^2;  dz = d * grad_scale.
// One warp per row: lanes stride over the row (4 elements a lane when rows
// are 16-byte aligned), the row sum by a warp tree.
// ---------------------------------------------------------------------------
struct MseParams {
  const void* z; int64_t ldz;
  const float* t; int64_t ldt;
  void* dz; int64_t lddz;
  float* loss_rows;
  int B, C;
  float grad_scale;
};

template <typename T, bool VEC>
__global__ void __launch_bounds__(256) mse_kernel(const __grid_constant__ MseParams p) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= p.B) return;
  const T* zr = reinterpret_cast<const T*>(p.z) + (int64_t)row * p.ldz;
  const float* tr = p.t + (int64_t)row * p.ldt;
  T* dr = reinterpret_cast<T*>(p.dz) + (int64_t)row * p.lddz;
  float s = 0.f;
  if (VEC) {
    for (int j = 4 * lane; j < p.C; j += 128) {
      float zv[4], d[4];
      load4<T>(zr + j, zv);
      const float4 tv = __ldcs(reinterpret_cast<const float4*>(tr + j));
      d[0] = zv[0] - tv.x; d[1] = zv[1] - tv.y; d[2] = zv[2] - tv.z; d[3] = zv[3] - tv.w;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        s += d[k] * d[k];
        d[k] *= p.grad_scale;
      }
      store4<T>(dr + j, d);
    }
  } else {
    for (int j = lane; j < p.C; j += 32) {
      const float d = to_f32(zr[j]) - tr[j];
      s += d * d;
      dr[j] = from_f32<T>(d * p.grad_scale);
    }
  }
  s = warp_sum(s);
  if (lane == 0) p.loss_rows[row] = s;
}

int mse_plan(const MseOp& op, LaunchRec* rec, char* err, size_t errlen) {
  if (op.B <= 0 || op.C <= 0 || op.B > INT32_MAX || op.C > INT32_MAX || op.ldz < op.C || op.ldt < op.C ||
      op.lddz < op.C) {
    snprintf(err, errlen, "mse: bad shape B=%lld C=%lld", (long long)op.B, (long long)op.C);
    return -1;
  }
  if (!op.z || !op.t || !op.dz || !op.loss_rows) { snprintf(err, errlen, "mse: null pointer"); return -1; }
  MseParams q{op.z, op.ldz, op.t, op.ldt, op.dz, op.lddz, op.loss_rows, (int)op.B, (int)op.C, op.grad_scale};
  const size_t es = op.dtype == DT_F32 ? 4 : 2;
  const bool vec = op.C % 4 == 0 && op.ldz % 4 == 0 && op.ldt % 4 == 0 && op.lddz % 4 == 0 &&
                   (uintptr_t)op.t % 16 == 0 && (uintptr_t)op.z % (4 * es) == 0 && (uintptr_t)op.dz % (4 * es) == 0;
  if (op.dtype == DT_F32)
    rec->func = vec ? (const void*)mse_kernel<float, true> : (const void*)mse_kernel<float, false>;
  else
    rec->func = vec ? (const void*)mse_kernel<__nv_bfloat16, true> : (const void*)mse_kernel<__nv_bfloat16, false>;
  rec->grid = dim3((unsigned)ceil_div(op.B, 8));
  rec->block = dim3(256);
  rec->smem = 0;
  rec->name = "mse";
  rec->set_args(q);
  return 1;
}

// ---------------------------------------------------------------------------
// Softmax-CE row statistics from the forward GEMM's per-group partials (one
// warp per row; lanes stride over the groups, then fixed warp trees).
// ---------------------------------------------------------------------------
struct CeCombineParams {
  const float2* stats; const float* zy; const int32_t* labels;
  float2* rowstat; float* loss_rows; uint32_t* err;
  int B, C, G;
};

__global__ void __launch_bounds__(256) ce_combine_kernel(const __grid_constant__ CeCombineParams p) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= p.B) return;
  const float2* st = p.stats + (int64_t)row * p.G;
  float m = -INFINITY;
  for (int g = lane; g < p.G; g += 32) m = fmaxf(m, st[g].x);
  m = warp_max(m);
  float s = 0.f;
  for (int g = lane; g < p.G; g += 32) {
    const float2 v = st[g];
    s += v.y * __expf(v.x - m);
  }
  s = warp_sum(s);
  if (lane == 0) {
    const int y = p.labels[row];
    const bool bad = y < 0 || y >= p.C;
    p.rowstat[row] = make_float2(m, 1.0f / s);
    p.loss_rows[row] = bad ? 0.f : (m + logf(s)) - p.zy[row];
    if (bad && p.err) atomicOr(p.err, ERRBIT_LABEL_RANGE);
  }
}

int ce_combine_plan(const CeCombineOp& op, LaunchRec* rec, char* err, size_t errlen) {
  if (op.B <= 0 || op.C <= 0 || op.B > INT32_MAX || op.C > INT32_MAX || !op.stats || !op.zy || !op.labels ||
      !op.rowstat || !op.loss_rows) {
    snprintf(err, errlen, "ce_combine: bad arguments");
    return -1;
  }
  CeCombineParams q{op.stats, op.zy, op.labels, op.rowstat, op.loss_rows, op.err, (int)op.B, (int)op.C,
                    (int)ce_groups(op.C)};
  rec->func = (const void*)ce_combine_kernel;
  rec->grid = dim3((unsigned)ceil_div(op.B, 8));
  rec->block = dim3(256);
  rec->smem = 0;
  rec->name = "ce_combine";
  rec->set_args(q);
  return 1;
}

// ---------------------------------------------------------------------------
// Mean of the row losses (fixed-order fp32 sums), step counter, finiteness.
// ---------------------------------------------------------------------------
struct LossMeanParams {
  const float* loss_rows; int64_t B; float count;
  float* loss;
  int64_t* step_counter;
  uint32_t* err;
  float* bias_corr;
  float beta1, beta2;
};

// fp32 sums in a fixed order (per-thread strided sums, then a pairwise tree):
// error ~ (B/1024 + 10) ulp of the sum, far below the loss tolerance, and
// no fp64 (slow on this part) in the step.
__global__ void __launch_bounds__(1024) loss_mean_kernel(const __grid_constant__ LossMeanParams p) {
  pdl_enter();
  __shared__ float red[1024];
  float s = 0.f;
#pragma unroll 8   // loads in flight; the additions keep their order
  for (int64_t i = threadIdx.x; i < p.B; i += blockDim.x) s += p.loss_rows[i];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    float L = red[0] / p.count;
    if (p.loss) *p.loss = L;
    if (p.step_counter) advance_step(p.step_counter, p.bias_corr, p.beta1, p.beta2);
    if (p.err && !isfinite(L)) atomicOr(p.err, ERRBIT_NONFINITE);
  }
}

int loss_mean_plan(const LossMeanOp& op, LaunchRec* rec, char* err, size_t errlen) {
  if (op.B <= 0) { snprintf(err, errlen, "loss_mean: empty batch"); return -1; }
  LossMeanParams q{op.loss_rows, op.B, (float)(op.count > 0 ? op.count : (double)op.B), op.loss,
                   op.step_counter, op.err, op.bias_corr, op.beta1, op.beta2};
  rec->func = (const void*)loss_mean_kernel;
  rec->grid = dim3(1);
  rec->block = dim3(1024);
  rec->smem = 0;
  rec->name = "loss_mean";
  rec->set_args(q);
  return 1;
}

// ---------------------------------------------------------------------------
// Optimizer update over flat planes (p, g, m, v at one index).
//   AdamW (PyTorch / Loshchilov-Hutter form):
//     m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
//     p = p - lr * (m/(1-b1^t) / (sqrt(v/(1-b2^t)) + eps) + wd * p_old).
//   Adam, decay as L2: g' = g + wd p, then the same moments and
//     p = p - lr * m/(1-b1^t) / (sqrt(v/(1-b2^t)) + eps).
//   SGD, momentum b1, L2 wd: buf = b1 buf + (g + wd p) (buf in m, zero
//     before the first step), p = p - lr buf.
// With global-norm clipping every g above is c g, c = min(1, max_norm /
// (||g||_2 + 1e-6)) over the whole flat gradient.
// ---------------------------------------------------------------------------
struct AdamWParams {
  float* p; float* g; float* m; float* v;
  __nv_bfloat16* w16; int64_t w16_plane;   // w16_plane > 0: three planes (hi, mid, lo)
  const int64_t* step_counter; int64_t t;
  const float* bias_corr;
  int64_t n;
  float lr, beta1, beta2, eps, wd;
  // gradient segments as partial sums (added here in a fixed order, written to g)
  AdamWOp::Seg seg[AdamWOp::kMaxSegs];
  int nseg;
  // batch loss = sum(loss_parts) * loss_scale, by one warp (nullable)
  const float* loss_parts; int loss_n; float loss_scale; float* loss; uint32_t* err;
  // clipping: per-block sums of squares (written by the norm kernel, read by
  // the update), their count, the threshold and the norm's destination
  float* norm_ws; int norm_n; float max_norm; float* norm_out;
};

// The gradient element g[f]: from its segment's partial sums, else the plane.
__device__ __forceinline__ float grad_elem(const AdamWParams& q, int64_t f, bool& from_parts) {
  from_parts = false;
  for (int k = 0; k < q.nseg; ++k) {
    const AdamWOp::Seg& sg = q.seg[k];
    if (f >= sg.off && f < sg.off + sg.len) {
      from_parts = true;
      float a = 0.f;
      for (int b = 0; b < sg.n; ++b) a += __ldcg(sg.parts + (int64_t)b * sg.stride + (f - sg.off));
      return a;
    }
  }
  return q.g[f];
}

// Gradient elements 4i .. 4i+3: from the plane, or summed from their
// segment's partials (16-byte loads, up to 16 in flight, added in partial
// order) and then written to the plane.  Lanes past the segment keep the
// plane's own value (padding).
__device__ __forceinline__ float4 load_grad4(const AdamWParams& q, int64_t i) {
  const int64_t f = 4 * i;
  int si = -1;
  for (int k = 0; k < q.nseg; ++k)
    if (f >= q.seg[k].off && f < q.seg[k].off + q.seg[k].len) si = k;
  if (si < 0) return reinterpret_cast<const float4*>(q.g)[i];
  const AdamWOp::Seg& sg = q.seg[si];
  const float* src = sg.parts + (f - sg.off);
  float4 part[16];
#pragma unroll
  for (int b = 0; b < 16; ++b)
    part[b] = b < sg.n ? __ldcg(reinterpret_cast<const float4*>(src + (int64_t)b * sg.stride))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 g = part[0];
#pragma unroll
  for (int b = 1; b < 16; ++b) {
    g.x += part[b].x; g.y += part[b].y; g.z += part[b].z; g.w += part[b].w;
  }
  for (int b0 = 16; b0 < sg.n; b0 += 16) {
#pragma unroll
    for (int b = 0; b < 16; ++b)
      part[b] = b0 + b < sg.n ? __ldcg(reinterpret_cast<const float4*>(src + (int64_t)(b0 + b) * sg.stride))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int b = 0; b < 16; ++b) {
      g.x += part[b].x; g.y += part[b].y; g.z += part[b].z; g.w += part[b].w;
    }
  }
  const int64_t end = sg.off + sg.len;
  if (f + 4 > end) {
    const float4 own = reinterpret_cast<const float4*>(q.g)[i];
    if (f + 1 >= end) g.y = own.y;
    if (f + 2 >= end) g.z = own.z;
    if (f + 3 >= end) g.w = own.w;
  }
  reinterpret_cast<float4*>(q.g)[i] = g;   // the gradient plane holds the summed gradient
  return g;
}

template <int KIND>
__device__ __forceinline__ void update_one(float& p, float g, float& m, float& v, const AdamWParams& q,
                                           float inv_bc1, float inv_sqrt_bc2) {
  if (KIND == OPTIM_ADAMW) {
    m = q.beta1 * m + (1.f - q.beta1) * g;
    v = q.beta2 * v + (1.f - q.beta2) * g * g;
    const float mhat = m * inv_bc1;
    const float denom = sqrtf(v) * inv_sqrt_bc2 + q.eps;
    p = p - q.lr * (mhat / denom + q.wd * p);
  } else if (KIND == OPTIM_ADAM) {
    g = g + q.wd * p;
    m = q.beta1 * m + (1.f - q.beta1) * g;
    v = q.beta2 * v + (1.f - q.beta2) * g * g;
    const float mhat = m * inv_bc1;
    const float denom = sqrtf(v) * inv_sqrt_bc2 + q.eps;
    p = p - q.lr * (mhat / denom);
  } else {
    g = g + q.wd * p;
    m = q.beta1 * m + g;
    p = p - q.lr * m;
  }
}

// bf16 planes of x: hi = bf16(x), mid = bf16(x - hi), lo = bf16(x - hi - mid)
// (hi + mid + lo = x for fp32 x in the normal range; each difference is
// exact in fp32).
__device__ __forceinline__ void split3(float x, __nv_bfloat16& hi, __nv_bfloat16& mid, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  const float r = x - __bfloat162float(hi);
  mid = __float2bfloat16_rn(r);
  lo = __float2bfloat16_rn(r - __bfloat162float(mid));
}
__device__ __forceinline__ void store_planes4(__nv_bfloat16* dst, int64_t plane, float4 v) {
  __nv_bfloat16 h[4], m[4], l[4];
  split3(v.x, h[0], m[0], l[0]);
  split3(v.y, h[1], m[1], l[1]);
  split3(v.z, h[2], m[2], l[2]);
  split3(v.w, h[3], m[3], l[3]);
  *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(h);
  *reinterpret_cast<uint2*>(dst + plane) = *reinterpret_cast<const uint2*>(m);
  *reinterpret_cast<uint2*>(dst + 2 * plane) = *reinterpret_cast<const uint2*>(l);
}

// Sum over a 256-thread block in a fixed order (warp trees, then a tree over
// the eight warp sums); every thread gets the result.
__device__ __forceinline__ float block_sum256(float a, float* red) {
  a = warp_sum(a);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  float b = (threadIdx.x & 31) < 8 ? red[threadIdx.x & 31] : 0.f;
  b = warp_sum(b);
  __syncthreads();   // red may be reused after this
  return b;
}

// Clipping, first pass: finish the gradient (segments added and written to
// g) and leave this block's sum of squares in norm_ws[blockIdx.x].
__global__ void __launch_bounds__(256) grad_norm_kernel(const __grid_constant__ AdamWParams q) {
  __shared__ float red[8];
  pdl_enter();
  const int64_t n4 = q.n / 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  float a = 0.f;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 g = load_grad4(q, i);
    a += g.x * g.x + g.y * g.y + g.z * g.z + g.w * g.w;
  }
  for (int64_t i = n4 * 4 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < q.n; i += stride) {
    bool fp = false;
    const float g = q.nseg ? grad_elem(q, i, fp) : q.g[i];
    if (fp) q.g[i] = g;
    a += g * g;
  }
  a = block_sum256(a, red);
  if (threadIdx.x == 0 && q.norm_ws) q.norm_ws[blockIdx.x] = a;
  if (q.loss_parts && blockIdx.x == 0 && threadIdx.x < 32) {
    // the batch loss from the output layer's partials (a gradient step that
    // leaves the update to a later launch): as in the update kernel
    float l = 0.f;
    for (int c = threadIdx.x; c < q.loss_n; c += 32) l += __ldcg(q.loss_parts + c);
    l = warp_sum(l);
    const float L = l * q.loss_scale;
    if (threadIdx.x == 0) {
      if (q.loss) *q.loss = L;
      if (q.err && !isfinite(L)) atomicOr(q.err, ERRBIT_NONFINITE);
    }
  }
}

template <int KIND, bool CLIP>
__global__ void __launch_bounds__(256) adamw_kernel(const __grid_constant__ AdamWParams q) {
  pdl_enter();
  // bias corrections: precomputed for the step (read by every thread, in
  // flight with its first parameter loads), else computed here
  float inv_bc1 = 1.f, inv_sqrt_bc2 = 1.f;
  if (KIND != OPTIM_SGD) {
    if (q.bias_corr) {
      inv_bc1 = __ldg(q.bias_corr);
      inv_sqrt_bc2 = __ldg(q.bias_corr + 1);
    } else {
      const int64_t t = q.t > 0 ? q.t : *q.step_counter;
      inv_bc1 = 1.0f / one_minus_pow(q.beta1, t);
      inv_sqrt_bc2 = 1.0f / sqrtf(one_minus_pow(q.beta2, t));
    }
  }
  float clip = 1.f;
  if (CLIP) {
    // every block adds the same partials in the same order: the same factor
    __shared__ float red[8];
    float a = 0.f;
    for (int c = threadIdx.x; c < q.norm_n; c += blockDim.x) a += __ldcg(q.norm_ws + c);
    const float norm = sqrtf(block_sum256(a, red));
    clip = fminf(1.f, q.max_norm / (norm + 1e-6f));
    if (blockIdx.x == 0 && threadIdx.x == 0 && q.norm_out) *q.norm_out = norm;
  }
  const int64_t n4 = q.n / 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 p = reinterpret_cast<float4*>(q.p)[i];
    float4 g = load_grad4(q, i);
    if (CLIP) { g.x *= clip; g.y *= clip; g.z *= clip; g.w *= clip; }
    float4 m = reinterpret_cast<float4*>(q.m)[i];
    float4 v = KIND == OPTIM_SGD ? make_float4(0.f, 0.f, 0.f, 0.f) : reinterpret_cast<float4*>(q.v)[i];
    update_one<KIND>(p.x, g.x, m.x, v.x, q, inv_bc1, inv_sqrt_bc2);
    update_one<KIND>(p.y, g.y, m.y, v.y, q, inv_bc1, inv_sqrt_bc2);
    update_one<KIND>(p.z, g.z, m.z, v.z, q, inv_bc1, inv_sqrt_bc2);
    update_one<KIND>(p.w, g.w, m.w, v.w, q, inv_bc1, inv_sqrt_bc2);
    reinterpret_cast<float4*>(q.p)[i] = p;
    reinterpret_cast<float4*>(q.m)[i] = m;
    if (KIND != OPTIM_SGD) reinterpret_cast<float4*>(q.v)[i] = v;
    if (q.w16 && q.w16_plane > 0) {
      store_planes4(q.w16 + 4 * i, q.w16_plane, p);
    } else if (q.w16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(p.x, p.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(p.z, p.w);
      uint2 o;
      o.x = *reinterpret_cast<uint32_t*>(&lo);
      o.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(q.w16)[i] = o;
    }
  }
  // tail (n not a multiple of 4)
  for (int64_t i = n4 * 4 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < q.n; i += stride) {
    float p = q.p[i], m = q.m[i], v = KIND == OPTIM_SGD ? 0.f : q.v[i];
    bool fp = false;
    float g = q.nseg ? grad_elem(q, i, fp) : q.g[i];
    if (fp) q.g[i] = g;
    if (CLIP) g *= clip;
    update_one<KIND>(p, g, m, v, q, inv_bc1, inv_sqrt_bc2);
    q.p[i] = p; q.m[i] = m;
    if (KIND != OPTIM_SGD) q.v[i] = v;
    if (q.w16 && q.w16_plane > 0) split3(p, q.w16[i], q.w16[i + q.w16_plane], q.w16[i + 2 * q.w16_plane]);
    else if (q.w16) q.w16[i] = __float2bfloat16_rn(p);
  }
  if (q.loss_parts && blockIdx.x == 0 && threadIdx.x < 32) {
    // the batch loss: lane c adds partials c, c + 32, ...; then a fixed-order warp tree
    float a = 0.f;
    for (int c = threadIdx.x; c < q.loss_n; c += 32) a += __ldcg(q.loss_parts + c);
    a = warp_sum(a);
    const float L = a * q.loss_scale;   // loss_scale = 1/B: the batch mean
    if (threadIdx.x == 0) {
      if (q.loss) *q.loss = L;
      if (q.err && !isfinite(L)) atomicOr(q.err, ERRBIT_NONFINITE);
    }
  }
}

template <bool CLIP>
const void* update_kernel(int kind) {
  return kind == OPTIM_ADAM ? (const void*)adamw_kernel<OPTIM_ADAM, CLIP>
         : kind == OPTIM_SGD ? (const void*)adamw_kernel<OPTIM_SGD, CLIP>
                             : (const void*)adamw_kernel<OPTIM_ADAMW, CLIP>;
}

int grad_finish_plan(const AdamWOp& op, LaunchRec* rec, char* err, size_t errlen) {
  if (op.n < 0 || op.nseg < 0 || op.nseg > AdamWOp::kMaxSegs || ((uintptr_t)op.g % 16)) {
    snprintf(err, errlen, "gradient finish: bad plane or segments");
    return -1;
  }
  AdamWParams q{};
  q.g = op.g; q.n = op.n;
  for (int k = 0; k < op.nseg; ++k) q.seg[k] = op.seg[k];
  q.nseg = op.nseg;
  q.loss_parts = op.loss_parts; q.loss_n = op.loss_n; q.loss_scale = op.loss_scale; q.loss = op.loss; q.err = op.err;
  q.norm_ws = op.norm_ws;
  int64_t blocks = ceil_div(op.n / 4 + 1, 256);
  if (blocks > AdamWOp::kNormParts) blocks = AdamWOp::kNormParts;
  if (blocks < 1) blocks = 1;
  rec->func = (const void*)grad_norm_kernel;
  rec->grid = dim3((unsigned)blocks);
  rec->block = dim3(256);
  rec->smem = 0;
  rec->name = "grad_finish";
  rec->set_args(q);
  return 1;
}

int adamw_plan(const AdamWOp& op, LaunchRec* rec, char* err, size_t errlen) {
  if (op.n < 0) { snprintf(err, errlen, "adamw: negative size"); return -1; }
  if (op.kind < OPTIM_ADAMW || op.kind > OPTIM_SGD) { snprintf(err, errlen, "adamw: unknown optimizer"); return -1; }
  if (op.kind != OPTIM_SGD && op.t <= 0 && !op.step_counter) { snprintf(err, errlen, "adamw: no step"); return -1; }
  auto al = [](const void* ptr, int a) { return ((uintptr_t)ptr % a) == 0; };
  if (!al(op.p, 16) || !al(op.g, 16) || !al(op.m, 16) || !al(op.v, 16) || (op.w16 && !al(op.w16, 8)) ||
      op.w16_plane % 4 || (op.w16_plane > 0 && op.w16_plane < op.n)) {
    snprintf(err, errlen, "adamw: planes must be 16-byte aligned (w16: 8, plane pitch >= n, multiple of 4)");
    return -1;
  }
  if (op.nseg < 0 || op.nseg > AdamWOp::kMaxSegs) {
    snprintf(err, errlen, "adamw: too many gradient segments");
    return -1;
  }
  for (int k = 0; k < op.nseg; ++k) {
    const AdamWOp::Seg& sg = op.seg[k];
    if (sg.n < 1 || sg.len < 1 || sg.off % 4 || sg.stride % 4 || sg.stride < sg.len || (uintptr_t)sg.parts % 16 ||
        sg.off + sg.len > op.n) {
      snprintf(err, errlen, "adamw: bad gradient segment %d", k);
      return -1;
    }
  }
  const bool clip = op.max_norm > 0.f;
  if (clip && !op.norm_ws) { snprintf(err, errlen, "adamw: clipping needs a norm workspace"); return -1; }
  if (!(op.max_norm >= 0.f) || !(op.max_norm < INFINITY)) {
    snprintf(err, errlen, "adamw: max_norm must be finite and >= 0");
    return -1;
  }
  AdamWParams q{};
  q.p = op.p; q.g = op.g; q.m = op.m; q.v = op.v;
  q.w16 = (__nv_bfloat16*)op.w16; q.w16_plane = op.w16_plane;
  q.step_counter = op.step_counter; q.t = op.t; q.bias_corr = op.bias_corr;
  q.n = op.n; q.lr = op.lr; q.beta1 = op.beta1; q.beta2 = op.beta2; q.eps = op.eps; q.wd = op.wd;
  for (int k = 0; k < op.nseg; ++k) q.seg[k] = op.seg[k];
  q.nseg = op.nseg;
  q.loss_parts = op.loss_parts; q.loss_n = op.loss_n; q.loss_scale = op.loss_scale; q.loss = op.loss; q.err = op.err;
  int64_t blocks = ceil_div(op.n / 4 + 1, 256);
  if (blocks > AdamWOp::kNormParts) blocks = AdamWOp::kNormParts;
  if (blocks < 1) blocks = 1;
  int nrec = 0;
  if (clip) {
    // first pass: the finished gradient and its per-block sums of squares
    AdamWParams qn = q;
    qn.loss_parts = nullptr;
    qn.norm_ws = op.norm_ws;
    LaunchRec& r = rec[nrec++];
    r.func = (const void*)grad_norm_kernel;
    r.grid = dim3((unsigned)blocks);
    r.block = dim3(256);
    r.smem = 0;
    r.name = "grad_norm";
    r.set_args(qn);
    q.nseg = 0;   // the update reads the gradient the first pass wrote
    q.norm_ws = op.norm_ws; q.norm_n = (int)blocks; q.max_norm = op.max_norm; q.norm_out = op.norm_out;
  }
  LaunchRec& r = rec[nrec++];
  r.func = clip ? update_kernel<true>(op.kind) : update_kernel<false>(op.kind);
  r.grid = dim3((unsigned)blocks);
  r.block = dim3(256);
  r.smem = 0;
  r.name = op.kind == OPTIM_ADAM ? "adam_l2_flat" : op.kind == OPTIM_SGD ? "sgd_flat" : "adamw_flat";
  r.set_args(q);
  return nrec;
}

// ---------------------------------------------------------------------------
// Row argmax (lowest index on ties).
// ---------------------------------------------------------------------------
struct ArgmaxParams {
  const void* z; int64_t ldz; int B, C; int32_t* out;
};

__device__ __forceinline__ void argmax_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i) || (v != v && v2 == v2)) { v = v2; i = i2; }
}

template <typename T>
__global__ void __launch_bounds__(256) argmax_kernel(const __grid_constant__ ArgmaxParams p) {
  pdl_enter();
  __shared__ float sv[32];
  __shared__ int si[32];
  const int row = blockIdx.x;
  const T* zr = reinterpret_cast<const T*>(p.z) + (int64_t)row * p.ldz;
  float v = -INFINITY;
  int idx = 0x7fffffff;
  for (int j = threadIdx.x; j < p.C; j += blockDim.x) argmax_merge(v, idx, to_f32(zr[j]), j);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    argmax_merge(v, idx, v2, i2);
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (lane == 0) { sv[wid] = v; si[wid] = idx; }
  __syncthreads();
  if (wid == 0) {
    v = lane < nw ? sv[lane] : -INFINITY;
    idx = lane < nw ? si[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float v2 = __shfl_xor_sync(0xffffffffu, v, o);
      int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
      argmax_merge(v, idx, v2, i2);
    }
    if (lane == 0) p.out[row] = idx == 0x7fffffff ? 0 : idx;
  }
}

int argmax_plan(const ArgmaxOp& op, LaunchRec* rec, char* err, size_t errlen) {
  if (op.B <= 0 || op.C <= 0 || op.B > INT32_MAX || op.C > INT32_MAX) {
    snprintf(err, errlen, "argmax: bad shape");
    return -1;
  }
  ArgmaxParams q{op.z, op.ldz, (int)op.B, (int)op.C, op.out};
  rec->func = op.dtype == DT_F32 ? (const void*)argmax_kernel<float> : (const void*)argmax_kernel<__nv_bfloat16>;
  rec->grid = dim3((unsigned)op.B);
  rec->block = dim3(op.C <= 32 ? 32 : op.C <= 1024 ? 128 : 256);
  rec->smem = 0;
  rec->name = "argmax";
  rec->set_args(q);
  return 1;
}

// ---------------------------------------------------------------------------
// Copies.
// ---------------------------------------------------------------------------
struct CopyRowsParams {
  const unsigned char* src; int64_t lds_bytes;
  unsigned char* dst; int64_t ldd_bytes;
  int64_t B, row_bytes;
};

__global__ void copy_rows_kernel(const __grid_constant__ CopyRowsParams p) {
  pdl_enter();
  const int64_t total = p.B * p.row_bytes;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = i / p.row_bytes, c = i % p.row_bytes;
    p.dst[r * p.ldd_bytes + c] = p.src[r * p.lds_bytes + c];
  }
}

int copy_rows_plan(const CopyRowsOp& op, LaunchRec* rec, char* err, size_t errlen) {
  if (op.B <= 0 || op.C <= 0) { snprintf(err, errlen, "copy_rows: bad shape"); return -1; }
  int64_t es = op.dtype == DT_F32 ? 4 : 2;
  CopyRowsParams q{(const unsigned char*)op.src, op.lds * es, (unsigned char*)op.dst, op.ldd * es, op.B, op.C * es};
  rec->func = (const void*)copy_rows_kernel;
  int64_t blocks = ceil_div(op.B * op.C * es, 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  rec->grid = dim3((unsigned)blocks);
  rec->block = dim3(256);
  rec->smem = 0;
  rec->name = "copy_rows";
  rec->set_args(q);
  return 1;
}

struct CastParams { const float* p; __nv_bfloat16* w16; int64_t n; };

__global__ void cast_bf16_kernel(const __grid_constant__ CastParams q) {
  pdl_enter();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < q.n; i += (int64_t)gridDim.x * blockDim.x)
    q.w16[i] = __float2bfloat16_rn(q.p[i]);
}

int cast_bf16_plan(int64_t n, const float* p, void* w16, LaunchRec* rec, char* err, size_t errlen) {
  if (n <= 0) { snprintf(err, errlen, "cast: empty"); return -1; }
  CastParams q{p, (__nv_bfloat16*)w16, n};
  rec->func = (const void*)cast_bf16_kernel;
  int64_t blocks = ceil_div(n, 256);
  if (blocks > 152 * 8) blocks = 152 * 8;
  rec->grid = dim3((unsigned)blocks);
  rec->block = dim3(256);
  rec->smem = 0;
  rec->name = "cast_bf16";
  rec->set_args(q);
  return 1;
}

// ---------------------------------------------------------------------------
// fp32 matrix -> its three bf16 planes (the fp32 model's operands for the
// tensor cores).  Streaming: one read of x, three bf16 writes.
// ---------------------------------------------------------------------------
struct Split3Params {
  const float* src; int64_t lds;
  __nv_bfloat16* dst; int64_t ldd, plane;
  int64_t rows, cols;
  int vec;   // 1: 4-wide loads/stores are aligned
};

__global__ void __launch_bounds__(256) split3_kernel(const __grid_constant__ Split3Params q) {
  pdl_enter();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  if (q.vec) {
    const int64_t c4 = q.cols / 4;
    const int64_t n = q.rows * c4;
    // two 16-byte loads in flight per thread and iteration
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += 2 * stride) {
      const int64_t i2 = i + stride;
      const int64_t r = i / c4, c = (i - r * c4) * 4;
      const int64_t r2 = i2 / c4, c2 = (i2 - r2 * c4) * 4;
      const float4 v = __ldcs(reinterpret_cast<const float4*>(q.src + r * q.lds + c));
      float4 v2 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i2 < n) v2 = __ldcs(reinterpret_cast<const float4*>(q.src + r2 * q.lds + c2));
      store_planes4(q.dst + r * q.ldd + c, q.plane, v);
      if (i2 < n) store_planes4(q.dst + r2 * q.ldd + c2, q.plane, v2);
    }
  } else {
    const int64_t n = q.rows * q.cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride) {
      const int64_t r = i / q.cols, c = i - r * q.cols;
      __nv_bfloat16* d = q.dst + r * q.ldd + c;
      split3(q.src[r * q.lds + c], d[0], d[q.plane], d[2 * q.plane]);
    }
  }
}

// The inverse: an fp32 matrix from its three bf16 planes, (hi + mid) + lo in
// fp32 -- exact, since the three planes hold the value's 24 significant bits
// in three 8-bit pieces.
struct Join3Params {
  const __nv_bfloat16* src; int64_t lds, plane;
  float* dst; int64_t ldd;
  int64_t rows, cols;
};

__global__ void __launch_bounds__(256) join3_kernel(const __grid_constant__ Join3Params q) {
  pdl_enter();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t n = q.rows * q.cols;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t r = i / q.cols, c = i - r * q.cols;
    const __nv_bfloat16* s = q.src + r * q.lds + c;
    q.dst[r * q.ldd + c] = (__bfloat162float(s[0]) + __bfloat162float(s[q.plane])) + __bfloat162float(s[2 * q.plane]);
  }
}

int join3_plan(int64_t rows, int64_t cols, const void* src, int64_t lds, int64_t plane, float* dst, int64_t ldd,
               LaunchRec* rec, char* err, size_t errlen) {
  if (rows <= 0 || cols <= 0 || lds < cols || ldd < cols || plane < rows * lds || !src || !dst) {
    snprintf(err, errlen, "join3: bad shape");
    return -1;
  }
  Join3Params q{(const __nv_bfloat16*)src, lds, plane, dst, ldd, rows, cols};
  int64_t blocks = ceil_div(rows * cols, 256);
  if (blocks > 152 * 8) blocks = 152 * 8;
  rec->func = (const void*)join3_kernel;
  rec->grid = dim3((unsigned)blocks);
  rec->block = dim3(256);
  rec->smem = 0;
  rec->name = "join3";
  rec->set_args(q);
  return 1;
}

int split3_plan(int64_t rows, int64_t cols, const float* src, int64_t lds, void* dst, int64_t ldd, int64_t plane,
                LaunchRec* rec, char* err, size_t errlen) {
  if (rows <= 0 || cols <= 0 || lds < cols || ldd < cols || plane < rows * ldd || !src || !dst) {
    snprintf(err, errlen, "split3: bad shape");
    return -1;
  }
  Split3Params q{src, lds, (__nv_bfloat16*)dst, ldd, plane, rows, cols, 0};
  q.vec = cols % 4 == 0 && lds % 4 == 0 && ldd % 4 == 0 && plane % 4 == 0 && (uintptr_t)src % 16 == 0 &&
          (uintptr_t)dst % 8 == 0;
  const int64_t work = q.vec ? rows * (cols / 4) : rows * cols;
  int64_t blocks = ceil_div(work, 256);
  if (blocks > 152 * 8) blocks = 152 * 8;
  rec->func = (const void*)split3_kernel;
  rec->grid = dim3((unsigned)blocks);
  rec->block = dim3(256);
  rec->smem = 0;
  rec->name = "split3";
  rec->set_args(q);
  return 1;
}

}  // namespace mlpk
