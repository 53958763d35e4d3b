// The output layer of the step fused into one kernel for the 10-class,
// 128-input layer of the MNIST-shaped MLP: logits z = h W^T + b, softmax
// cross-entropy (loss and dz; or the squared error against real targets,
// the MSE of pypi "munet-nn", "Python training"), the dgrad of the layer with the hidden
// activation's VJP (dY = (dz W) * act'), and the partial sums of the layer's
// weight and bias gradients (dW = dz^T h, db = sum dz) and of the batch loss.
// Each row of h is read once; W lives in shared memory.  This is the
// single-read cross-entropy of devpost "Orthon" ("Selected Orthon vs.
// PyTorch results") extended to the whole output layer, with the layer's
// VJPs written out as in noeira.ai "Neural networks" ("The design in one
// page": forward and vjp per module).
//
// Each CTA takes 32-row tiles: the h tile is staged in shared memory (16-byte
// loads, the next tile's in flight during the current one), then logits and
// softmax / dz (8 threads per row), dY (one thread per 4 columns x 4 rows,
// 8- or 16-byte stores) and the dW / db partial sums (one thread per column
// and 5 classes) come from shared memory.  CTAs run in clusters of 8: after a cluster barrier, CTA
// rank q adds slice q of the cluster's dW / db partials through distributed
// shared memory in rank order and writes it to the workspace; the optimizer
// adds the cluster partials (and the loss partials) in cluster order, so the
// result is deterministic and no CTA waits for another.  Block 0 advances
// the step counter and stores AdamW's bias corrections on entry.
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
constexpr int kHPartPitch = 1292;         // kHPart rounded up to 16 bytes

struct HeadParams {
  const void* h; int64_t ldh;          // [B, 128] model dtype (input of the output layer)
  const void* W;                       // [10, 128] model dtype
  const float* bias;                   // [10]
  const int32_t* labels;               // [B] (softmax CE)
  const float* targets; int64_t ldt;   // [B, 10] fp32 (MSE)
  const void* aux; int64_t ld_aux;     // stored u of the layer below (GELU only)
  void* dY; int64_t ldy;               // [B, 128] model dtype
  int64_t* step_counter;
  uint32_t* err;
  float* ws;                           // [clusters][kHPartPitch] fp32, then [clusters] fp32 loss partials
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
  float loss_rows[kHR];
  float loss;               // this CTA's loss partial
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = __bfloat162float(e[i]);
}

// 16 consecutive elements of h at element index i (16-byte aligned) as fp32.
// X3: h is held as bf16 planes hi + mid + lo whose fp32 sum is h exactly.
template <typename T, bool X3>
__device__ __forceinline__ void load_h16(const HeadParams& p, int64_t i, float* f) {
  if (X3) {
    const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(p.h) + i;
    uint4 u[6];
#pragma unroll
    for (int pl = 0; pl < 3; ++pl) {
      u[2 * pl] = __ldg(reinterpret_cast<const uint4*>(b + pl * p.h_plane));
      u[2 * pl + 1] = __ldg(reinterpret_cast<const uint4*>(b + pl * p.h_plane) + 1);
    }
    float hi[16], mid[16], lo[16];
    bf16x8_to_f32(u[0], hi); bf16x8_to_f32(u[1], hi + 8);
    bf16x8_to_f32(u[2], mid); bf16x8_to_f32(u[3], mid + 8);
    bf16x8_to_f32(u[4], lo); bf16x8_to_f32(u[5], lo + 8);
#pragma unroll
    for (int j = 0; j < 16; ++j) f[j] = (hi[j] + mid[j]) + lo[j];
  } else if (sizeof(T) == 4) {
    const float4* q = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.h) + i);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 v = __ldg(q + j);
      f[4 * j] = v.x; f[4 * j + 1] = v.y; f[4 * j + 2] = v.z; f[4 * j + 3] = v.w;
    }
  } else {
    const uint4* q = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.h) + i);
    bf16x8_to_f32(__ldg(q), f);
    bf16x8_to_f32(__ldg(q + 1), f + 8);
  }
}

// 4 consecutive dY elements at element index i (aligned to 4 elements).
template <typename T, bool X3>
__device__ __forceinline__ void store_dy4(const HeadParams& p, int64_t i, const float* v) {
  if (X3) {
    __nv_bfloat16 hi[4], mid[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      hi[j] = __float2bfloat16_rn(v[j]);
      const float r = v[j] - __bfloat162float(hi[j]);
      mid[j] = __float2bfloat16_rn(r);
      lo[j] = __float2bfloat16_rn(r - __bfloat162float(mid[j]));
    }
    __nv_bfloat16* b = reinterpret_cast<__nv_bfloat16*>(p.dY) + i;
    *reinterpret_cast<uint2*>(b) = *reinterpret_cast<const uint2*>(hi);
    *reinterpret_cast<uint2*>(b + p.dy_plane) = *reinterpret_cast<const uint2*>(mid);
    *reinterpret_cast<uint2*>(b + 2 * p.dy_plane) = *reinterpret_cast<const uint2*>(lo);
  } else if (sizeof(T) == 4) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.dY) + i) = make_float4(v[0], v[1], v[2], v[3]);
  } else {
    __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&a);
    o.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.dY) + i) = o;
  }
}

template <typename T, bool X3 = false, bool MSE = false>
__global__ void __cluster_dims__(kHCluster, 1, 1) __launch_bounds__(kHT)
head_kernel(const __grid_constant__ HeadParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  HeadSmem& s = *reinterpret_cast<HeadSmem*>(smem_raw);
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x;
  pdl_enter();
  // nothing else in the step reads the counter before the optimizer
  if (blockIdx.x == 0 && tid == 0 && p.step_counter)
    advance_step(p.step_counter, p.bias_corr, p.beta1, p.beta2);
  // h tile staging: row hr, columns hc..hc+15
  const int hr = tid >> 3, hc = 16 * (tid & 7);
  const int ntiles = (p.B + kHR - 1) / kHR;
  float hv[16];
  int label = 0;   // the label of row tid / 8 of the tile (logits / softmax mapping below)
  float tq[2] = {0.f, 0.f};   // MSE: targets of classes tid % 8 and tid % 8 + 8 of that row
  auto load_tile = [&](int tile) {   // this thread's 16 elements of the tile (zeros past the last row)
    const int r0 = tile * kHR;
    if (tile < ntiles && r0 + hr < p.B) {
      load_h16<T, X3>(p, (int64_t)(r0 + hr) * p.ldh + hc, hv);
      if (MSE) {
        const float* tr = p.targets + (int64_t)(r0 + hr) * p.ldt;
        const int c0 = tid & 7;
        tq[0] = __ldg(tr + c0);
        tq[1] = c0 + 8 < kHC ? __ldg(tr + c0 + 8) : 0.f;
      } else {
        label = __ldg(p.labels + r0 + hr);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) hv[j] = 0.f;
    }
  };
  load_tile(blockIdx.x);   // in flight while W is staged
  {   // W: 4 consecutive elements per load (rows of 128 are 4-aligned)
    float wv[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int i = 4 * (tid + j * kHT);
      if (i < kHC * kHK) {
        if (sizeof(T) == 4) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.W) + i));
          wv[j][0] = v.x; wv[j][1] = v.y; wv[j][2] = v.z; wv[j][3] = v.w;
        } else {
          const uint2 u = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(p.W) + i));
          const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
          for (int k = 0; k < 4; ++k) wv[j][k] = __bfloat162float(e[k]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int i = 4 * (tid + j * kHT);
      if (i < kHC * kHK)
        *reinterpret_cast<float4*>(&s.W[i / kHK][i % kHK]) = make_float4(wv[j][0], wv[j][1], wv[j][2], wv[j][3]);
    }
  }
  if (tid < kHR) s.loss_rows[tid] = 0.f;
  float bias[kHC];   // every thread needs all ten
#pragma unroll
  for (int c = 0; c < kHC; ++c) bias[c] = __ldg(p.bias + c);

  // dY: this thread's 4 columns kq..kq+3 and rows rq, rq + 8, rq + 16, rq + 24
  const int kq = 4 * (tid & 31);
  const int rq = tid >> 5;
  // logits: 8 threads per row (lr = tid / 8); thread `sub` takes the float4
  // columns sub, sub + 8, sub + 16, sub + 24 (conflict-free in shared memory)
  const int lr = tid >> 3, sub = tid & 7;
  // dW: this thread's column kw and classes 2 j + cw (j < 5); db: tid < 10
  const int kw = tid & (kHK - 1), cw = tid >> 7;
  float acc[5], accb = 0.f;
#pragma unroll
  for (int j = 0; j < 5; ++j) acc[j] = 0.f;

  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int r0 = tile * kHR;
    const int nr = min(kHR, p.B - r0);
    __syncthreads();   // W loaded / previous tile finished with h and z
#pragma unroll
    for (int j = 0; j < 16; j += 4)
      *reinterpret_cast<float4*>(&s.h[hr][hc + j]) = make_float4(hv[j], hv[j + 1], hv[j + 2], hv[j + 3]);
    const int y = label;   // row lr == hr of this tile
    const float t0 = tq[0], t1 = tq[1];
    __syncthreads();
    load_tile(tile + gridDim.x);   // the next tile's h, in flight during this one
    // logits (partial dot products over this thread's 16 columns, then a
    // fixed xor tree over the row's 8 threads), rounded to the model dtype
    // (the value a stored logits tensor holds); then softmax cross-entropy:
    // dz replaces z, thread sub writes classes sub and sub + 8
    {
      float zc[kHC];
#pragma unroll
      for (int c = 0; c < kHC; ++c) zc[c] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = 4 * (sub + 8 * i);
        const float4 h4 = *reinterpret_cast<const float4*>(&s.h[lr][k]);
#pragma unroll
        for (int c = 0; c < kHC; ++c) {
          const float4 w4 = *reinterpret_cast<const float4*>(&s.W[c][k]);
          zc[c] = fmaf(h4.x, w4.x, zc[c]);
          zc[c] = fmaf(h4.y, w4.y, zc[c]);
          zc[c] = fmaf(h4.z, w4.z, zc[c]);
          zc[c] = fmaf(h4.w, w4.w, zc[c]);
        }
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1)
#pragma unroll
        for (int c = 0; c < kHC; ++c) zc[c] += __shfl_xor_sync(0xffffffffu, zc[c], o);
      if (MSE) {
        // d = z - t for classes sub and sub + 8; the row's squared error by
        // a fixed xor tree over its 8 threads
        float sq = 0.f;
        if (lr < nr) {
#pragma unroll
          for (int c = 0; c < kHC; ++c) {
            if (c == sub || c == sub + 8) {
              const float d = to_f32(from_f32<T>(zc[c] + bias[c])) - (c == sub ? t0 : t1);
              sq = fmaf(d, d, sq);
              s.z[lr][c] = to_f32(from_f32<T>(d * p.grad_scale));
            }
          }
        } else {
          if (sub < kHC) s.z[lr][sub] = 0.f;
          if (sub + 8 < kHC) s.z[lr][sub + 8] = 0.f;
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        if (lr < nr && sub == 0) s.loss_rows[lr] += sq;
      } else if (lr < nr) {
        float m = -INFINITY, zy = 0.f;
#pragma unroll
        for (int c = 0; c < kHC; ++c) {
          zc[c] = to_f32(from_f32<T>(zc[c] + bias[c]));
          m = fmaxf(m, zc[c]);
          if (c == y) zy = zc[c];
        }
        float se = 0.f;
#pragma unroll
        for (int c = 0; c < kHC; ++c) {
          zc[c] = expf(zc[c] - m);
          se += zc[c];
        }
        const float inv = 1.0f / se;
#pragma unroll
        for (int c = 0; c < kHC; ++c)
          if (c == sub || c == sub + 8)
            s.z[lr][c] = to_f32(from_f32<T>((zc[c] * inv - (c == y ? 1.f : 0.f)) * p.grad_scale));
        if (sub == 0) {
          if (y < 0 || y >= kHC) {
            if (p.err) atomicOr(p.err, ERRBIT_LABEL_RANGE);
          } else {
            s.loss_rows[lr] += (m + logf(se)) - zy;
          }
        }
      } else {
        if (sub < kHC) s.z[lr][sub] = 0.f;
        if (sub + 8 < kHC) s.z[lr][sub + 8] = 0.f;
      }
    }
    __syncthreads();
    // dY = (dz W) * act'
    {
      float4 wq[kHC];
#pragma unroll
      for (int c = 0; c < kHC; ++c) wq[c] = *reinterpret_cast<const float4*>(&s.W[c][kq]);
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int r = rq + 8 * rr;
        if (r < nr) {
          float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int c = 0; c < kHC; ++c) {
            const float d = s.z[r][c];
            a[0] = fmaf(d, wq[c].x, a[0]); a[1] = fmaf(d, wq[c].y, a[1]);
            a[2] = fmaf(d, wq[c].z, a[2]); a[3] = fmaf(d, wq[c].w, a[3]);
          }
          if (p.act == ACT_RELU) {   // this tile's h is the stored h
#pragma unroll
            for (int j = 0; j < 4; ++j) a[j] *= s.h[r][kq + j] > 0.f ? 1.f : 0.f;
          } else if (p.act == ACT_GELU_TANH) {
            const T* u = reinterpret_cast<const T*>(p.aux) + (int64_t)(r0 + r) * p.ld_aux + kq;
#pragma unroll
            for (int j = 0; j < 4; ++j) a[j] *= gelu_tanh_grad(to_f32(u[j]));
          }
          store_dy4<T, X3>(p, (int64_t)(r0 + r) * p.ldy + kq, a);
        }
      }
    }
    // dW += dz^T h, db += sum dz over the tile's rows (zero rows add 0):
    // one h load and one dz row per row serve all five classes
#pragma unroll 4
    for (int r = 0; r < kHR; ++r) {
      const float hk = s.h[r][kw];
      float zr[kHC];
#pragma unroll
      for (int c = 0; c < kHC; ++c) zr[c] = s.z[r][c];
#pragma unroll
      for (int j = 0; j < 5; ++j) acc[j] = fmaf(cw ? zr[2 * j + 1] : zr[2 * j], hk, acc[j]);
      if (tid < kHC) accb += s.z[r][tid];
    }
  }
  // ---- this CTA's partial into its shared memory ----
#pragma unroll
  for (int j = 0; j < 5; ++j) s.part[(2 * j + cw) * kHK + kw] = acc[j];
  if (tid < kHC) s.part[kHC * kHK + tid] = accb;
  __syncthreads();
  if (tid < 32) {   // this CTA's loss partial: a fixed-order tree over the 32 row slots
    static_assert(kHR == 32, "one loss slot per lane");
    const float a = warp_sum(s.loss_rows[tid]);
    if (tid == 0) s.loss = a;
  }
  // ---- cluster: CTA rank q adds slice q of the partial vector over the
  //      cluster's CTAs (in rank order) through distributed shared memory ----
  cluster.sync();
  const unsigned rank = cluster.block_rank();
  const int nclusters = gridDim.x / kHCluster;
  const int cid = blockIdx.x / kHCluster;
  constexpr int kSlice = (kHPart + kHCluster - 1) / kHCluster;
  const int e_end = min(kHPart, (int)(rank + 1) * kSlice);
  for (int e = (int)rank * kSlice + tid; e < e_end; e += kHT) {
    float a = 0.f;
#pragma unroll
    for (int q = 0; q < kHCluster; ++q) a += cluster.map_shared_rank(&s, q)->part[e];
    p.ws[(int64_t)cid * kHPartPitch + e] = a;
  }
  if (rank == 0 && tid == 0) {
    float a = 0.f;
    for (int q = 0; q < kHCluster; ++q) a += cluster.map_shared_rank(&s, q)->loss;
    p.ws[(int64_t)nclusters * kHPartPitch + cid] = a;
  }
  cluster.sync();   // every CTA keeps its shared memory until the cluster has read it
}

namespace {
int head_grid(int64_t B) {
  const int64_t tiles = ceil_div(B, kHR);
  int64_t g = round_up(tiles, kHCluster);
  const int64_t gmax = (152 / kHCluster) * kHCluster;   // 144: one wave
  return (int)(g > gmax ? gmax : g);
}
}  // namespace

HeadPartials head_partials(int64_t B, int64_t C, int64_t K) {
  (void)C; (void)K;
  const int nc = head_grid(B) / kHCluster;
  return HeadPartials{nc, kHPartPitch, (int64_t)nc * kHPartPitch};
}

size_t head_workspace_bytes(int64_t B, int64_t C, int64_t K) {
  // room for this kernel's cluster partials or for those of the same layer
  // folded into the forward GEMM below it (tc_fused_head_partials)
  const HeadPartials hp = head_partials(B, C, K), fp = tc_fused_head_partials(B);
  const int64_t a = hp.loss_off + hp.n, b = fp.loss_off + fp.n;
  return (size_t)(a > b ? a : b) * 4;
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
  const int64_t al = x3 || op.dtype == DT_BF16 ? 8 : 4;   // 16-byte h rows, 8/16-byte dY stores
  if (op.ldh % al || op.ldy % al || ((uintptr_t)op.h & 15) || ((uintptr_t)op.dY & 15) ||
      (x3 && (op.h_plane % 8 || op.dy_plane % 8))) {
    snprintf(err, errlen, "fused output layer: h / dY need 16-byte aligned rows");
    return -1;
  }
  if (op.ws_bytes < head_workspace_bytes(op.B, op.C, op.K)) {
    snprintf(err, errlen, "fused output layer: workspace too small");
    return -1;
  }
  const bool mse = op.targets != nullptr;
  if (mse && op.ldt < op.C) {
    snprintf(err, errlen, "fused output layer: target pitch below C");
    return -1;
  }
  HeadParams q;
  q.h = op.h; q.ldh = op.ldh; q.W = op.W; q.bias = op.bias; q.labels = op.labels;
  q.targets = op.targets; q.ldt = op.ldt;
  q.aux = op.aux; q.ld_aux = op.ld_aux; q.dY = op.dY; q.ldy = op.ldy;
  q.step_counter = op.step_counter; q.err = op.err;
  q.ws = op.ws;
  q.B = (int)op.B; q.act = op.act;
  q.grad_scale = op.grad_scale;
  q.bias_corr = op.bias_corr; q.beta1 = op.beta1; q.beta2 = op.beta2;
  q.h_plane = op.h_plane; q.dy_plane = op.dy_plane;
  const void* fns[6] = {(const void*)head_kernel<float>, (const void*)head_kernel<__nv_bfloat16>,
                        (const void*)head_kernel<float, true>, (const void*)head_kernel<float, false, true>,
                        (const void*)head_kernel<__nv_bfloat16, false, true>,
                        (const void*)head_kernel<float, true, true>};
  static std::once_flag once;
  std::call_once(once, [&] {
    for (const void* f : fns)
      cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(HeadSmem));
  });
  rec->func = fns[(mse ? 3 : 0) + (x3 ? 2 : op.dtype == DT_F32 ? 0 : 1)];
  rec->grid = dim3(head_grid(op.B));
  rec->block = dim3(kHT);
  rec->smem = (unsigned)sizeof(HeadSmem);
  rec->name = mse ? "head_mse" : "head_ce";
  // at most one wave of CTAs: scheduled early, they wait beside the
  // predecessor at a few CTAs per SM
  rec->early = true;
  rec->set_args(q);
  return 1;
}

}  // namespace mlpk
