// The output layer of the step fused into one kernel for the 10-class,
// 128-input layer of the MNIST-shaped MLP: logits z = h W^T + b, softmax
// cross-entropy (loss and dz), the dgrad of the layer with the hidden
// activation's VJP (dY = (dz W) * act'), and the layer's weight and bias
// gradients (dW = dz^T h, db = sum dz) with the batch-mean loss.  Each row of
// h is read once; W lives in shared memory.  This is the single-read
// cross-entropy of devpost "Orthon" ("Selected Orthon vs. PyTorch results")
// extended to the whole output layer, with the layer's VJPs written out as in
// noeira.ai "Neural networks" ("The design in one page": forward and vjp per
// module).
//
// Each CTA takes 32-row tiles: the h tile is staged in shared memory, then
// logits (one thread per row and class), softmax and dz (one thread per row),
// dY (one thread per input column, looping over the tile's rows) and the
// dW / db partial sums (one thread per weight) come from shared memory.
// CTAs run in clusters of 8: after a cluster barrier, rank 0 adds its
// cluster's partials through distributed shared memory in rank order, and
// the last cluster leader to finish (an atomic ticket) adds the cluster
// partials in cluster order -- deterministic -- writes dW, db and the mean
// loss, advances the step counter and re-arms the ticket.  No CTA spins on
// another.
#include <cooperative_groups.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "ops.h"

namespace cg = cooperative_groups;

namespace mlpk {

constexpr int kHC = 10, kHK = 128;        // classes, inputs
constexpr int kHR = 32;                   // rows per tile
constexpr int kHT = 256;                  // threads
constexpr int kHCluster = 8;
constexpr int kHKP = kHK + 4;             // padded smem pitch (keeps 16-byte rows)
constexpr int kHPart = kHC * kHK + kHC;   // dW + db partial length

struct HeadParams {
  const void* h; int64_t ldh;          // [B, 128] model dtype (input of the output layer)
  const void* W;                       // [10, 128] model dtype
  const float* bias;                   // [10]
  const int32_t* labels;               // [B]
  const void* aux; int64_t ld_aux;     // stored u of the layer below (GELU only)
  void* dY; int64_t ldy;               // [B, 128] model dtype
  float* dW; float* db;                // [10, 128], [10] fp32 (gradient plane)
  float* loss;
  int64_t* step_counter;
  uint32_t* err;
  float* ws;                           // [clusters][kHPart] fp32, then [clusters] fp64 loss partials
  unsigned int* ticket;                // zero before the first launch; re-armed by the last leader
  int B, act;
  float grad_scale;
  float* bias_corr;
  float beta1, beta2;
  int64_t h_plane, dy_plane;           // fp32 h / dY held as three bf16 planes (X3 variant)
};

struct HeadSmem {
  float W[kHC][kHKP];
  float h[kHR][kHKP];
  float z[kHR][kHC];        // logits, then dz
  float part[kHPart];       // this CTA's dW / db partial
  double loss_rows[kHR];
  double loss;              // this CTA's loss partial
};

// X3: h and dY are fp32 values held as bf16 planes hi + mid + lo (the sum is
// the fp32 value exactly); the arithmetic is the fp32 kernel's.
template <bool X3>
__device__ __forceinline__ float load_h(const HeadParams& p, int64_t i) {
  if (!X3) return reinterpret_cast<const float*>(p.h)[i];
  const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(p.h);
  return (__bfloat162float(b[i]) + __bfloat162float(b[i + p.h_plane])) + __bfloat162float(b[i + 2 * p.h_plane]);
}
template <bool X3>
__device__ __forceinline__ void store_dy(const HeadParams& p, int64_t i, float v) {
  if (!X3) {
    reinterpret_cast<float*>(p.dY)[i] = v;
    return;
  }
  __nv_bfloat16* b = reinterpret_cast<__nv_bfloat16*>(p.dY);
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  const float r = v - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r);
  b[i] = hi;
  b[i + p.dy_plane] = mid;
  b[i + 2 * p.dy_plane] = __float2bfloat16_rn(r - __bfloat162float(mid));
}

template <typename T, bool X3 = false>
__global__ void __cluster_dims__(kHCluster, 1, 1) __launch_bounds__(kHT)
head_kernel(const __grid_constant__ HeadParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  HeadSmem& s = *reinterpret_cast<HeadSmem*>(smem_raw);
  __shared__ bool is_last;
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x;
  for (int i = tid; i < kHC * kHK; i += kHT) s.W[i / kHK][i % kHK] = to_f32(reinterpret_cast<const T*>(p.W)[i]);
  if (tid < kHR) s.loss_rows[tid] = 0.0;

  // this thread's fixed column for dY and its five dW elements
  const int kcol = tid % kHK;           // dY: column kcol, rows tid/128, +2, +4, ...
  const int rsub = tid / kHK;           // 0 or 1
  float acc[kHPart / kHT + 1];
#pragma unroll
  for (int j = 0; j < kHPart / kHT + 1; ++j) acc[j] = 0.f;

  const int ntiles = (p.B + kHR - 1) / kHR;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int r0 = tile * kHR;
    const int nr = min(kHR, p.B - r0);
    __syncthreads();   // W loaded / previous tile finished with h and z
#pragma unroll
    for (int j = 0; j < kHR * kHK / kHT; ++j) {
      const int i = tid + j * kHT;
      const int r = i / kHK, k = i % kHK;
      if (X3) s.h[r][k] = r < nr ? load_h<true>(p, (int64_t)(r0 + r) * p.ldh + k) : 0.f;
      else s.h[r][k] = r < nr ? to_f32(reinterpret_cast<const T*>(p.h)[(int64_t)(r0 + r) * p.ldh + k]) : 0.f;
    }
    __syncthreads();
    // logits rounded to the model dtype (the value a stored logits tensor holds)
    for (int t = tid; t < kHR * kHC; t += kHT) {
      const int r = t / kHC, c = t % kHC;
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
      for (int k = 0; k < kHK; k += 4) {
        const float4 hv = *reinterpret_cast<const float4*>(&s.h[r][k]);
        const float4 wv = *reinterpret_cast<const float4*>(&s.W[c][k]);
        a0 = fmaf(hv.x, wv.x, a0); a1 = fmaf(hv.y, wv.y, a1);
        a2 = fmaf(hv.z, wv.z, a2); a3 = fmaf(hv.w, wv.w, a3);
      }
      s.z[r][c] = to_f32(from_f32<T>((a0 + a1) + (a2 + a3) + p.bias[c]));
    }
    __syncthreads();
    // softmax cross-entropy per row: loss and dz (dz replaces z)
    if (tid < kHR) {
      const int r = tid;
      if (r < nr) {
        const int y = p.labels[r0 + r];
        const bool bad = y < 0 || y >= kHC;
        float m = -INFINITY, zy = 0.f;
#pragma unroll
        for (int c = 0; c < kHC; ++c) {
          m = fmaxf(m, s.z[r][c]);
          if (c == y) zy = s.z[r][c];
        }
        float e[kHC], se = 0.f;
#pragma unroll
        for (int c = 0; c < kHC; ++c) {
          e[c] = expf(s.z[r][c] - m);
          se += e[c];
        }
        const float inv = 1.0f / se;
#pragma unroll
        for (int c = 0; c < kHC; ++c)
          s.z[r][c] = to_f32(from_f32<T>((e[c] * inv - (c == y ? 1.f : 0.f)) * p.grad_scale));
        if (bad) {
          if (p.err) atomicOr(p.err, ERRBIT_LABEL_RANGE);
        } else {
          s.loss_rows[r] += (double)((m + logf(se)) - zy);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kHC; ++c) s.z[r][c] = 0.f;
      }
    }
    __syncthreads();
    // dY = (dz W) * act': column kcol, rows rsub, rsub + 2, ...
    {
      float wcol[kHC];
#pragma unroll
      for (int c = 0; c < kHC; ++c) wcol[c] = s.W[c][kcol];
      for (int r = rsub; r < nr; r += kHT / kHK) {
        float a = 0.f;
#pragma unroll
        for (int c = 0; c < kHC; ++c) a = fmaf(s.z[r][c], wcol[c], a);
        float g = 1.f;
        if (p.act == ACT_RELU) g = s.h[r][kcol] > 0.f ? 1.f : 0.f;   // this tile's h is the stored h
        else if (p.act == ACT_GELU_TANH)
          g = gelu_tanh_grad(to_f32(reinterpret_cast<const T*>(p.aux)[(int64_t)(r0 + r) * p.ld_aux + kcol]));
        if (X3) store_dy<true>(p, (int64_t)(r0 + r) * p.ldy + kcol, a * g);
        else reinterpret_cast<T*>(p.dY)[(int64_t)(r0 + r) * p.ldy + kcol] = from_f32<T>(a * g);
      }
    }
    // dW += dz^T h, db += sum dz over the tile's rows (zero rows add 0)
#pragma unroll
    for (int j = 0; j < kHPart / kHT + 1; ++j) {
      const int e = tid + j * kHT;
      if (e < kHC * kHK) {
        const int c = e / kHK, k = e % kHK;
        float a = acc[j];
#pragma unroll 8
        for (int r = 0; r < kHR; ++r) a = fmaf(s.z[r][c], s.h[r][k], a);
        acc[j] = a;
      } else if (e < kHPart) {
        const int c = e - kHC * kHK;
        float a = acc[j];
#pragma unroll 8
        for (int r = 0; r < kHR; ++r) a += s.z[r][c];
        acc[j] = a;
      }
    }
  }
  // ---- this CTA's partial into its shared memory ----
#pragma unroll
  for (int j = 0; j < kHPart / kHT + 1; ++j) {
    const int e = tid + j * kHT;
    if (e < kHPart) s.part[e] = acc[j];
  }
  __syncthreads();
  if (tid == 0) {
    double a = 0.0;
    for (int r = 0; r < kHR; ++r) a += s.loss_rows[r];
    s.loss = a;
  }
  // ---- cluster: rank 0 adds the cluster's partials in rank order ----
  cluster.sync();
  const unsigned rank = cluster.block_rank();
  const int nclusters = gridDim.x / kHCluster;
  const int cid = blockIdx.x / kHCluster;
  double* lws = reinterpret_cast<double*>(p.ws + round_up((int64_t)nclusters * kHPart, 2));
  if (rank == 0) {
    for (int e = tid; e < kHPart; e += kHT) {
      float a = 0.f;
#pragma unroll
      for (int q = 0; q < kHCluster; ++q) a += cluster.map_shared_rank(&s, q)->part[e];
      p.ws[(int64_t)cid * kHPart + e] = a;
    }
    if (tid == 0) {
      double a = 0.0;
      for (int q = 0; q < kHCluster; ++q) a += cluster.map_shared_rank(&s, q)->loss;
      lws[cid] = a;
    }
  }
  cluster.sync();   // the other CTAs keep their shared memory until rank 0 has read it
  if (rank != 0) return;
  // ---- the last cluster leader adds the cluster partials in order ----
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = atomicAdd(p.ticket, 1u) == (unsigned)nclusters - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int e = tid; e < kHPart; e += kHT) {
    float a = 0.f;
#pragma unroll 4
    for (int b = 0; b < nclusters; ++b) a += __ldcg(p.ws + (int64_t)b * kHPart + e);
    if (e < kHC * kHK) p.dW[e] = a;
    else p.db[e - kHC * kHK] = a;
  }
  if (tid == 0) {
    double a = 0.0;
    for (int b = 0; b < nclusters; ++b) a += __ldcg(lws + b);
    const float L = (float)(a / (double)p.B);
    if (p.loss) *p.loss = L;
    if (p.step_counter) advance_step(p.step_counter, p.bias_corr, p.beta1, p.beta2);
    if (p.err && !isfinite(L)) atomicOr(p.err, ERRBIT_NONFINITE);
    *p.ticket = 0u;
  }
}

namespace {
int head_grid(int64_t B) {
  const int64_t tiles = ceil_div(B, kHR);
  int64_t g = round_up(tiles, kHCluster);
  const int64_t gmax = (152 / kHCluster) * kHCluster;   // 144: one wave
  return (int)(g > gmax ? gmax : g);
}
}  // namespace

size_t head_workspace_bytes(int64_t B, int64_t C, int64_t K) {
  (void)C; (void)K;
  const int nc = head_grid(B) / kHCluster;
  return (size_t)round_up((int64_t)nc * kHPart, 2) * 4 + (size_t)nc * 8;
}

bool head_supported(int64_t C, int64_t K) { return C == kHC && K == kHK; }

int head_plan(const HeadOp& op, LaunchRec* rec, char* err, size_t errlen) {
  if (!head_supported(op.C, op.K) || op.B < 1 || op.B > INT32_MAX) {
    snprintf(err, errlen, "fused output layer: unsupported C=%lld K=%lld", (long long)op.C, (long long)op.K);
    return -1;
  }
  const bool x3 = op.dtype == DT_F32X3;
  if (x3 && (op.act == ACT_GELU_TANH || op.h_plane < op.B * op.ldh || op.dy_plane < op.B * op.ldy)) {
    snprintf(err, errlen, "fused output layer: planes need ReLU/none below and full plane pitches");
    return -1;
  }
  if (op.ws_bytes < head_workspace_bytes(op.B, op.C, op.K)) {
    snprintf(err, errlen, "fused output layer: workspace too small");
    return -1;
  }
  HeadParams q;
  q.h = op.h; q.ldh = op.ldh; q.W = op.W; q.bias = op.bias; q.labels = op.labels;
  q.aux = op.aux; q.ld_aux = op.ld_aux; q.dY = op.dY; q.ldy = op.ldy;
  q.dW = op.dW; q.db = op.db; q.loss = op.loss; q.step_counter = op.step_counter; q.err = op.err;
  q.ws = op.ws; q.ticket = op.ticket;
  q.B = (int)op.B; q.act = op.act;
  q.grad_scale = op.grad_scale;
  q.bias_corr = op.bias_corr; q.beta1 = op.beta1; q.beta2 = op.beta2;
  q.h_plane = op.h_plane; q.dy_plane = op.dy_plane;
  const void* fns[3] = {(const void*)head_kernel<float>, (const void*)head_kernel<__nv_bfloat16>,
                        (const void*)head_kernel<float, true>};
  static std::once_flag once;
  std::call_once(once, [&] {
    for (const void* f : fns)
      cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(HeadSmem));
  });
  rec->func = fns[x3 ? 2 : op.dtype == DT_F32 ? 0 : 1];
  rec->grid = dim3(head_grid(op.B));
  rec->block = dim3(kHT);
  rec->smem = (unsigned)sizeof(HeadSmem);
  rec->name = "head_ce";
  rec->set_args(q);
  return 1;
}

}  // namespace mlpk
