// Internal interface between the step runtime and the kernels.  Every op is
// turned into one or more LaunchRec's; the runtime decides whether to launch
// them on a stream or to record them into a CUDA graph.
#pragma once
#include <stddef.h>
#include <stdint.h>

#include "launch.h"

namespace mlpk {

enum GemmKind : int { GEMM_FWD = 0, GEMM_DGRAD = 1, GEMM_WGRAD = 2 };

// C[m, n] = sum_k A(m, k) * B(k, n), with the epilogue chosen by `kind`.
//   A(m, k) = A[m*lda + k] if a_kmajor else A[k*lda + m]
//   B(k, n) = B[n*ldb + k] if b_kmajor else B[k*ldb + n]
// GEMM_FWD   : out[m, n] = act(C + bias[n]); out_u (optional) = C + bias[n]
// GEMM_DGRAD : out[m, n] = C * act'(aux[m, n])   (aux = stored h for ReLU,
//              stored u for GELU)
// GEMM_WGRAD : dW[m, n] = C (fp32);  db[m] = sum_k A(m, k) (fp32), the bias
//              gradient fused in.  With splits > 1 the K range is cut into
//              `splits` chunks whose fp32 partials go to `ws` and are summed
//              in a fixed order by a second kernel (deterministic).
//
// With dtype DT_F32X3 every fp32 operand and fp32 result is held as three
// bf16 planes (hi, mid, lo; hi + mid + lo = the fp32 value) `a_plane`,
// `b_plane`, `out_plane` elements apart, and the tensor cores accumulate the
// six significant plane products in fp32.  aux is then the hi plane of the
// stored activation (ReLU mask only).
struct GemmOp {
  int dtype = 0;            // DT_F32, DT_BF16 or DT_F32X3 (A, B, out, aux)
  int kind = GEMM_FWD;
  int act = 0;
  int64_t M = 0, N = 0, K = 0;
  const void* A = nullptr; int64_t lda = 0; bool a_kmajor = true;
  const void* B = nullptr; int64_t ldb = 0; bool b_kmajor = true;
  const float* bias = nullptr;
  void* out = nullptr; int64_t ldo = 0;
  void* out_u = nullptr; int64_t ldu = 0;
  const void* aux = nullptr; int64_t ld_aux = 0;
  float* dW = nullptr; int64_t ld_dw = 0;
  float* db = nullptr;
  float* ws = nullptr; size_t ws_bytes = 0;
  int splits = 0;           // 0 = choose
  uint32_t* err = nullptr;  // device error word (bounded-wait timeouts)
  int64_t a_plane = 0, b_plane = 0, out_plane = 0;   // DT_F32X3 plane pitches (elements)
  // GEMM_WGRAD with splits > 1: leave the partial sums in ws ([splits][M*N],
  // then [splits][M] for db) for the optimizer to add instead of planning the
  // reduce kernel; the number of splits used goes to *splits_out.
  bool defer_reduce = false;
  int* splits_out = nullptr;
  // Softmax-CE around a bf16 output layer (tensor cores):
  //   GEMM_FWD with ce_stats: besides the logits (stored bf16), each row's
  //     (max, sum exp(z - max)) over every 128-column group of the stored
  //     logits goes to ce_stats [M][ceil(N / 128)] (float2), and the logit at
  //     ce_labels[row] to ce_zy [M].
  //   GEMM_DGRAD (A = z, K-major) / GEMM_WGRAD (A = z as [K rows, M]) with
  //     ce_rowstat: the operand is dz = (exp(z - M_r) invS_r - [c == y_r])
  //     ce_scale, formed from the stored logits in shared memory;
  //     (M_r, invS_r) = ce_rowstat[r] for batch row r.
  // ReLU as one bit per element (bf16, tensor cores, one CTA per tile):
  // GEMM_FWD with ACT_RELU also writes bits, GEMM_DGRAD with ACT_RELU reads
  // its mask from them instead of the stored h (aux).  Layout: 64-column
  // groups, each [rows] of 64-bit words (pitch ld_bits >= M words), so a
  // warp's rows are contiguous: bit n % 64 of word (n / 64) * ld_bits + m is
  // "stored h[m, n] > 0".
  uint64_t* relu_bits = nullptr; int64_t ld_bits = 0;
  // bf16 forward / dgrad on CTA pairs with 2-SM MMAs (256 x 256 tiles):
  // -1 where there is at least one full wave of pair tiles, 0 never, 1
  // wherever the form allows (N and M of at least 256, no softmax-CE)
  int cg2 = -1;
  float2* ce_stats = nullptr; float* ce_zy = nullptr;
  const float2* ce_rowstat = nullptr;
  const int32_t* ce_labels = nullptr;
  float ce_scale = 0.f;
  // The 10-class, 128-input softmax-CE output layer folded into the forward
  // of the last hidden layer (fp32 planes, CTA pairs, N = 128; head_W != 0):
  // from each row's fp32 h (never stored) the epilogue forms the logits
  // z = h W_out^T + b_out, the loss, dz = (softmax(z) - onehot(y)) head_scale
  // and writes dY = (dz W_out) * act'(h) to `out` (planes) in place of h; the
  // partial sums over each CTA's rows of dW_out = dz^T h, db_out = sum dz
  // and the loss go to head_ws (tc_fused_head_partials layout), and block 0
  // advances the step counter (AdamW's bias corrections to bias_corr).
  const float* head_W = nullptr;       // fp32 [10, 128]
  const float* head_bias = nullptr;    // fp32 [10]
  const int32_t* head_labels = nullptr;
  float* head_ws = nullptr;
  float head_scale = 0.f;
  int64_t* step_counter = nullptr;
  float* bias_corr = nullptr;
  float beta1 = 0.9f, beta2 = 0.999f;
};

// Number of K splits the wgrad of this shape uses, and the workspace bytes.
int wgrad_splits(int dtype, int64_t M, int64_t N, int64_t K);
size_t wgrad_workspace_bytes(int dtype, int64_t M, int64_t N, int64_t K, int splits);
// The largest workspace any kernel choice for this shape uses (one-SM or CTA
// pairs, whatever GemmOp::cg2 says): a layout sized by it fits either.
size_t wgrad_workspace_bytes_any(int dtype, int64_t M, int64_t N, int64_t K);

// Plans: fill recs[0..n) and return n (<= 2), or -1 with a message in err.
int simt_gemm_plan(const GemmOp& op, LaunchRec* recs, char* err, size_t errlen);
int tc_gemm_plan(const GemmOp& op, LaunchRec* recs, char* err, size_t errlen);
// The kernel used by the model: tcgen05 for bf16, SIMT FFMA for fp32.
int gemm_plan(const GemmOp& op, LaunchRec* recs, char* err, size_t errlen);

// Softmax cross-entropy, forward and backward in one pass over each row.
struct CeOp {
  int dtype = 0;
  int64_t B = 0, C = 0;
  const void* z = nullptr; int64_t ldz = 0;
  const int32_t* labels = nullptr;
  void* dz = nullptr; int64_t lddz = 0;
  float* loss_rows = nullptr;
  float grad_scale = 1.0f;   // 1/B for a batch-mean loss
  uint32_t* err = nullptr;
};
int ce_plan(const CeOp& op, LaunchRec* rec, char* err, size_t errlen);

// Squared error against fp32 targets t [B, C] (ldt):  loss_rows[i] =
// sum_j (z_ij - t_ij)^2 (fp32), dz_ij = (z_ij - t_ij) * grad_scale (dtype;
// grad_scale = 2 / (B C) gives the gradient of the element-mean loss).
struct MseOp {
  int dtype = 0;
  int64_t B = 0, C = 0;
  const void* z = nullptr; int64_t ldz = 0;
  const float* t = nullptr; int64_t ldt = 0;
  void* dz = nullptr; int64_t lddz = 0;
  float* loss_rows = nullptr;
  float grad_scale = 0.f;
};
int mse_plan(const MseOp& op, LaunchRec* rec, char* err, size_t errlen);

// Softmax-CE row statistics from the per-group partials of the forward
// GEMM: M_r = max_g m_rg, S_r = sum_g s_rg exp(m_rg - M_r) (fixed order);
// rowstat[r] = (M_r, 1 / S_r), loss_rows[r] = M_r + log S_r - zy[r]; a label
// outside [0, C) sets the error bit (loss 0).
struct CeCombineOp {
  int64_t B = 0, C = 0;
  const float2* stats = nullptr; const float* zy = nullptr; const int32_t* labels = nullptr;
  float2* rowstat = nullptr; float* loss_rows = nullptr; uint32_t* err = nullptr;
};
int ce_combine_plan(const CeCombineOp& op, LaunchRec* rec, char* err, size_t errlen);
inline int64_t ce_groups(int64_t C) { return (C + 127) / 128; }

// loss = sum(loss_rows) / count in a fixed order (count = B when 0);
// optionally bumps the step counter and latches a non-finite loss into the
// error word.
struct LossMeanOp {
  int64_t B = 0;
  double count = 0;
  const float* loss_rows = nullptr;
  float* loss = nullptr;
  int64_t* step_counter = nullptr;   // nullable
  uint32_t* err = nullptr;           // nullable
  float* bias_corr = nullptr;        // nullable: AdamW bias corrections for the new step
  float beta1 = 0.9f, beta2 = 0.999f;
};
int loss_mean_plan(const LossMeanOp& op, LaunchRec* rec, char* err, size_t errlen);

// AdamW over flat fp32 planes (one launch for every parameter).
struct AdamWOp {
  int64_t n = 0;
  float* p = nullptr; float* g = nullptr; float* m = nullptr; float* v = nullptr;
  void* w16 = nullptr;                 // bf16 copy of p written after the update (nullable)
  int64_t w16_plane = 0;               // > 0: write the three bf16 planes of p, this many apart
  const int64_t* step_counter = nullptr;   // t read from device (already incremented)...
  int64_t t = 0;                       // ...or given explicitly when > 0
  const float* bias_corr = nullptr;    // precomputed [1/(1-b1^t), 1/sqrt(1-b2^t)] (nullable)
  float lr = 0, beta1 = 0, beta2 = 0, eps = 0, wd = 0;
  // Optional: gradient segments left as partial sums: g[off + e] for
  // e < len is parts[0][e] + parts[1][e] + ... + parts[n-1][e] (rows `stride`
  // floats apart), added in that order, written to g and used.  off and
  // stride must be multiples of 4, parts 16-byte aligned, and each partial
  // row readable up to the next multiple of 4 past len.
  static constexpr int kMaxSegs = 16;
  struct Seg { int64_t off, len; const float* parts; int n; int64_t stride; };
  Seg seg[kMaxSegs];
  int nseg = 0;
  // Optional: loss = sum(loss_parts[0 .. loss_n)) * loss_scale (one thread;
  // a non-finite loss sets the error bit in err).
  const float* loss_parts = nullptr; int loss_n = 0; float loss_scale = 1.f;
  float* loss = nullptr; uint32_t* err = nullptr;
  // The update rule (OPTIM_*): AdamW; Adam with the decay as L2 added to the
  // gradient; SGD with momentum beta1 (buffer in m, v untouched), L2 wd.
  int kind = 0;
  // Global-norm clipping when max_norm > 0: a first kernel adds the segments,
  // writes g and leaves one partial sum of squares per block in norm_ws
  // (kNormParts floats); the update scales g by min(1, max_norm / (||g|| +
  // 1e-6)) and block 0 writes ||g|| to norm_out (nullable).
  float max_norm = 0.f;
  float* norm_ws = nullptr;
  float* norm_out = nullptr;
  static constexpr int kNormParts = 152 * 8;
};
enum { OPTIM_ADAMW = 0, OPTIM_ADAM = 1, OPTIM_SGD = 2 };
// One or two records (clipping: norm, then update) into rec[0..1].
int adamw_plan(const AdamWOp& op, LaunchRec* rec, char* err, size_t errlen);
// The gradient finished without an update: the segments added and written
// to g, and the loss formed from loss_parts (both as the update would).
int grad_finish_plan(const AdamWOp& op, LaunchRec* rec, char* err, size_t errlen);

// Row argmax, lowest index among equal maxima.
struct ArgmaxOp {
  int dtype = 0;
  int64_t B = 0, C = 0;
  const void* z = nullptr; int64_t ldz = 0;
  int32_t* out = nullptr;
};
int argmax_plan(const ArgmaxOp& op, LaunchRec* rec, char* err, size_t errlen);

// Copy rows of a padded [B, ld] matrix into a dense [B, C] one.
struct CopyRowsOp {
  int dtype = 0;
  int64_t B = 0, C = 0;
  const void* src = nullptr; int64_t lds = 0;
  void* dst = nullptr; int64_t ldd = 0;
};
int copy_rows_plan(const CopyRowsOp& op, LaunchRec* rec, char* err, size_t errlen);

// w16[i] = bf16_rne(p[i]).
int cast_bf16_plan(int64_t n, const float* p, void* w16, LaunchRec* rec, char* err, size_t errlen);

// The three bf16 planes of an fp32 [rows, cols] matrix (row pitch lds):
// dst[pl * plane + r * ldd + c] for pl = 0 (hi), 1 (mid), 2 (lo), with
// hi = bf16(x), mid = bf16(x - hi), lo = bf16(x - hi - mid).
// fp32 [rows, cols] (ldd) from its three bf16 planes (lds, `plane` apart).
int join3_plan(int64_t rows, int64_t cols, const void* src, int64_t lds, int64_t plane, float* dst, int64_t ldd,
               LaunchRec* rec, char* err, size_t errlen);
int split3_plan(int64_t rows, int64_t cols, const float* src, int64_t lds, void* dst, int64_t ldd, int64_t plane,
                LaunchRec* rec, char* err, size_t errlen);

// The output layer fused with softmax-CE for the 10-class, 128-input head:
// logits, per-row loss, dz, dY = (dz W) * act'(aux), and per-cluster partial
// sums of dW, db and the loss in the workspace (head_partials), which the
// optimizer adds in a fixed order.  Block 0 advances the step counter.
struct HeadOp {
  int dtype = 0;
  int act = 0;                          // activation of the hidden layer below (for its VJP)
  int64_t B = 0, C = 0, K = 0;
  const void* h = nullptr; int64_t ldh = 0;
  const void* W = nullptr;              // [C, K], row pitch K
  const float* bias = nullptr;
  const int32_t* labels = nullptr;
  // MSE instead of softmax CE when set: fp32 targets [B, C] (row pitch ldt);
  // dz = (z - t) * grad_scale, loss partials are sums of (z - t)^2
  const float* targets = nullptr; int64_t ldt = 0;
  const void* aux = nullptr; int64_t ld_aux = 0;
  void* dY = nullptr; int64_t ldy = 0;
  int64_t* step_counter = nullptr;
  uint32_t* err = nullptr;
  float* ws = nullptr; size_t ws_bytes = 0;
  float grad_scale = 1.0f;
  float* bias_corr = nullptr;           // nullable: AdamW bias corrections for the new step
  float beta1 = 0.9f, beta2 = 0.999f;
  int64_t h_plane = 0, dy_plane = 0;    // DT_F32X3: h and dY as bf16 planes this far apart; W fp32
};
bool head_supported(int64_t C, int64_t K);
size_t head_workspace_bytes(int64_t B, int64_t C, int64_t K);
// What the fused output layer leaves in its workspace for the optimizer:
// n partial sums of [dW (C*K, row-major), db (C)] with row pitch `stride`
// floats, then n loss partials starting at float offset `loss_off`.
struct HeadPartials { int n; int64_t stride; int64_t loss_off; };
HeadPartials head_partials(int64_t B, int64_t C, int64_t K);
// The same output layer folded into the forward GEMM of the layer below
// (GemmOp::head_W): possible for an M x N x K fp32-as-planes forward that
// runs on CTA pairs with N = 128 and C = 10; one partial per 128-row tile.
bool tc_fused_head_ok(int64_t M, int64_t N, int64_t K, int64_t C);
HeadPartials tc_fused_head_partials(int64_t M);
int head_plan(const HeadOp& op, LaunchRec* rec, char* err, size_t errlen);

// One thread waits, through the bounded wait every tcgen05 kernel uses, for
// an mbarrier phase that nothing completes: after limit_ns it marks
// ERRBIT_TIMEOUT in err_dev and returns (the error path, exercised).
int wait_timeout_check_plan(uint32_t* err_dev, uint64_t limit_ns, LaunchRec* rec);

// Set the message mlp_last_error() returns on the calling thread.
void set_last_error(const char* msg);

}  // namespace mlpk
