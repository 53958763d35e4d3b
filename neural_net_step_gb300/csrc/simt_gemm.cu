// fp32 GEMMs of the training step on the FP32 FFMA pipes (no TF32), with the
// step's epilogues fused: bias + activation for the forward LinearAct
// (noeira.ai "Neural networks", "The design in one page": MatMul+Bias+
// Activation in one kernel), the activation VJP mask for dgrad, and the bias
// gradient (row sum of dY^T) for wgrad.  Register-blocked 8x8 outputs per
// thread, 16-deep K slices double-buffered through shared memory.
#include <stdio.h>

#include "common.cuh"
#include "ops.h"

namespace mlpk {

struct SimtGemmParams {
  const float* A; int64_t lda;
  const float* B; int64_t ldb;
  int M, N, K;
  int k_chunk;           // K range per blockIdx.z (multiple of the K slice)
  int kind, act;
  const float* bias;
  float* out; int64_t ldo;
  float* out_u; int64_t ldu;
  const float* aux; int64_t ld_aux;
  float* db;             // wgrad bias gradient (splits == 1)
  float* ws;             // wgrad partials [splits][M][N] then [splits][M] (splits > 1)
};

constexpr int SK = 16;   // K slice

template <int BM, int BN, bool AK, bool BKM>
__global__ void __launch_bounds__((BM / 8) * (BN / 8))
simt_gemm_kernel(const __grid_constant__ SimtGemmParams p) {
  pdl_enter();
  constexpr int NT = (BM / 8) * (BN / 8);
  constexpr int A_PER = BM * SK / NT;
  constexpr int B_PER = BN * SK / NT;
  constexpr int LDA_S = BM + 4, LDB_S = BN + 4;
  __shared__ __align__(16) float As[2][SK][LDA_S];
  __shared__ __align__(16) float Bs[2][SK][LDB_S];

  const int tid = threadIdx.x;
  const int tx = tid % (BN / 8), ty = tid / (BN / 8);
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int kbeg = blockIdx.z * p.k_chunk;
  const int kend = min(p.K, kbeg + p.k_chunk);
  const int ntiles = kend > kbeg ? (kend - kbeg + SK - 1) / SK : 0;
  const bool do_db = (p.kind == GEMM_WGRAD) && blockIdx.x == 0 && p.db != nullptr;

  float ra[A_PER], rb[B_PER];
  auto load = [&](int t) {
    const int k0 = kbeg + t * SK;
#pragma unroll
    for (int i = 0; i < A_PER; ++i) {
      int idx = tid + i * NT;
      int m, k;
      if (AK) { m = idx / SK; k = idx % SK; } else { m = idx % BM; k = idx / BM; }
      int gm = m0 + m, gk = k0 + k;
      float v = 0.f;
      if (gm < p.M && gk < kend) v = AK ? p.A[(int64_t)gm * p.lda + gk] : p.A[(int64_t)gk * p.lda + gm];
      ra[i] = v;
    }
#pragma unroll
    for (int i = 0; i < B_PER; ++i) {
      int idx = tid + i * NT;
      int n, k;
      if (BKM) { n = idx / SK; k = idx % SK; } else { n = idx % BN; k = idx / BN; }
      int gn = n0 + n, gk = k0 + k;
      float v = 0.f;
      if (gn < p.N && gk < kend) v = BKM ? p.B[(int64_t)gn * p.ldb + gk] : p.B[(int64_t)gk * p.ldb + gn];
      rb[i] = v;
    }
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int i = 0; i < A_PER; ++i) {
      int idx = tid + i * NT;
      int m, k;
      if (AK) { m = idx / SK; k = idx % SK; } else { m = idx % BM; k = idx / BM; }
      As[buf][k][m] = ra[i];
    }
#pragma unroll
    for (int i = 0; i < B_PER; ++i) {
      int idx = tid + i * NT;
      int n, k;
      if (BKM) { n = idx / SK; k = idx % SK; } else { n = idx % BN; k = idx / BN; }
      Bs[buf][k][n] = rb[i];
    }
  };

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  float rowsum = 0.f;

  if (ntiles > 0) {
    load(0);
    store(0);
  }
  __syncthreads();
  for (int t = 0; t < ntiles; ++t) {
    const int cur = t & 1;
    if (t + 1 < ntiles) load(t + 1);
#pragma unroll
    for (int kk = 0; kk < SK; ++kk) {
      float a[8], b[8];
      float4 a0 = *reinterpret_cast<const float4*>(&As[cur][kk][ty * 4]);
      float4 a1 = *reinterpret_cast<const float4*>(&As[cur][kk][BM / 2 + ty * 4]);
      float4 b0 = *reinterpret_cast<const float4*>(&Bs[cur][kk][tx * 4]);
      float4 b1 = *reinterpret_cast<const float4*>(&Bs[cur][kk][BN / 2 + tx * 4]);
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
      a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
      b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (do_db && tid < BM) {
#pragma unroll
      for (int kk = 0; kk < SK; ++kk) rowsum += As[cur][kk][tid];
    }
    if (t + 1 < ntiles) store(cur ^ 1);
    __syncthreads();
  }

  // Epilogue.
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + (i < 4 ? ty * 4 + i : BM / 2 + ty * 4 + (i - 4));
    if (gm >= p.M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int gn = n0 + (j < 4 ? tx * 4 + j : BN / 2 + tx * 4 + (j - 4));
      if (gn >= p.N) continue;
      float c = acc[i][j];
      if (p.kind == GEMM_FWD) {
        float u = c + p.bias[gn];
        if (p.out_u) p.out_u[(int64_t)gm * p.ldu + gn] = u;
        p.out[(int64_t)gm * p.ldo + gn] = apply_act(u, p.act);
      } else if (p.kind == GEMM_DGRAD) {
        float s = p.act == ACT_NONE ? 1.f : p.aux[(int64_t)gm * p.ld_aux + gn];
        p.out[(int64_t)gm * p.ldo + gn] = c * act_grad_from_stored(s, p.act);
      } else {
        if (p.ws) p.ws[((int64_t)blockIdx.z * p.M + gm) * p.N + gn] = c;
        else p.out[(int64_t)gm * p.ldo + gn] = c;
      }
    }
  }
  if (do_db && tid < BM && m0 + tid < p.M) {
    if (p.ws) p.ws[(int64_t)gridDim.z * p.M * p.N + (int64_t)blockIdx.z * p.M + m0 + tid] = rowsum;
    else p.db[m0 + tid] = rowsum;
  }
}

// Fixed-order sum of split-K partials: dW[m, n] = sum_s ws[s][m][n]; db[m]
// likewise.  Shared by the SIMT and tensor-core wgrad paths.
struct SplitReduceParams {
  const float* ws; int splits; int M, N;
  float* dW; int64_t ld_dw;
  float* db;
};

__global__ void split_reduce_kernel(const __grid_constant__ SplitReduceParams p) {
  pdl_enter();
  const int64_t MN = (int64_t)p.M * p.N;
  const int64_t total = MN + p.M;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < MN) {
      float s = 0.f;
      for (int k = 0; k < p.splits; ++k) s += p.ws[k * MN + i];
      int64_t m = i / p.N, n = i % p.N;
      p.dW[m * p.ld_dw + n] = s;
    } else if (p.db) {
      int64_t m = i - MN;
      float s = 0.f;
      for (int k = 0; k < p.splits; ++k) s += p.ws[p.splits * MN + k * (int64_t)p.M + m];
      p.db[m] = s;
    }
  }
}

int split_reduce_plan(const float* ws, int splits, int64_t M, int64_t N, float* dW, int64_t ld_dw,
                      float* db, LaunchRec* rec) {
  SplitReduceParams q{ws, splits, (int)M, (int)N, dW, ld_dw, db};
  rec->func = (const void*)split_reduce_kernel;
  int64_t total = M * N + M;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  rec->grid = dim3((unsigned)blocks);
  rec->block = dim3(256);
  rec->smem = 0;
  rec->name = "split_reduce";
  rec->set_args(q);
  return 1;
}

namespace {
constexpr int kSMs = 152;

template <int BM, int BN>
const void* pick(bool ak, bool bk) {
  if (ak && bk) return (const void*)simt_gemm_kernel<BM, BN, true, true>;
  if (ak && !bk) return (const void*)simt_gemm_kernel<BM, BN, true, false>;
  if (!ak && !bk) return (const void*)simt_gemm_kernel<BM, BN, false, false>;
  return (const void*)simt_gemm_kernel<BM, BN, false, true>;
}
}  // namespace

int simt_gemm_splits(int64_t M, int64_t N, int64_t K) {
  int64_t tiles = ceil_div(M, 64) * ceil_div(N, 64);
  int64_t s = 1;
  while (tiles * s < 4 * kSMs && K / (s * 2) >= 256) s *= 2;
  return (int)s;
}

int simt_gemm_plan(const GemmOp& op, LaunchRec* recs, char* err, size_t errlen) {
  if (op.dtype != DT_F32) { snprintf(err, errlen, "SIMT GEMM is fp32 only"); return -1; }
  if (op.M <= 0 || op.N <= 0 || op.K <= 0 || op.M > INT32_MAX || op.N > INT32_MAX || op.K > INT32_MAX) {
    snprintf(err, errlen, "bad GEMM shape %lld x %lld x %lld", (long long)op.M, (long long)op.N, (long long)op.K);
    return -1;
  }
  SimtGemmParams p{};
  p.A = (const float*)op.A; p.lda = op.lda;
  p.B = (const float*)op.B; p.ldb = op.ldb;
  p.M = (int)op.M; p.N = (int)op.N; p.K = (int)op.K;
  p.kind = op.kind; p.act = op.act;
  p.bias = op.bias;
  p.out = (float*)(op.kind == GEMM_WGRAD ? (void*)op.dW : op.out);
  p.ldo = op.kind == GEMM_WGRAD ? op.ld_dw : op.ldo;
  p.out_u = (float*)op.out_u; p.ldu = op.ldu;
  p.aux = (const float*)op.aux; p.ld_aux = op.ld_aux;
  p.db = op.db;
  int splits = 1;
  if (op.kind == GEMM_WGRAD) {
    splits = op.splits > 0 ? op.splits : simt_gemm_splits(op.M, op.N, op.K);
    if (splits > 1) {
      size_t need = wgrad_workspace_bytes(DT_F32, op.M, op.N, op.K, splits);
      if (!op.ws || op.ws_bytes < need) {
        snprintf(err, errlen, "wgrad workspace too small (%zu < %zu)", op.ws_bytes, need);
        return -1;
      }
      p.ws = op.ws;
    }
  }
  int64_t chunk = round_up(ceil_div(op.K, splits), SK);
  p.k_chunk = (int)chunk;
  splits = (int)ceil_div(op.K, chunk);
  constexpr int BM = 64, BN = 64;
  recs[0].func = pick<BM, BN>(op.a_kmajor, op.b_kmajor);
  recs[0].grid = dim3((unsigned)ceil_div(op.N, BN), (unsigned)ceil_div(op.M, BM), (unsigned)splits);
  recs[0].block = dim3((BM / 8) * (BN / 8));
  recs[0].smem = 0;
  recs[0].name = op.kind == GEMM_FWD ? "simt_gemm_fwd" : op.kind == GEMM_DGRAD ? "simt_gemm_dgrad" : "simt_gemm_wgrad";
  recs[0].set_args(p);
  if (op.splits_out) *op.splits_out = splits;
  if (op.kind == GEMM_WGRAD && splits > 1 && !op.defer_reduce) {
    split_reduce_plan(op.ws, splits, op.M, op.N, op.dW, op.ld_dw, op.db, &recs[1]);
    return 2;
  }
  return 1;
}

}  // namespace mlpk
