// Step runtime behind the C ABI: arena layout, parameter initialisation,
// the per-step launch plan, CUDA-graph construction/replay, and the
// op-level entry points.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "common.cuh"
#include "mlp.h"
#include "mlp_ops.h"
#include "ops.h"

using namespace mlpk;

// ---------------------------------------------------------------------------
// Errors.
// ---------------------------------------------------------------------------
static thread_local char g_err[1024] = "";

static mlp_status fail(mlp_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
static mlp_status fail(mlp_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}
static mlp_status ok() {
  g_err[0] = 0;
  return MLP_OK;
}
void mlpk::set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }
#define CUDA_TRY(expr)                                                                       \
  do {                                                                                       \
    cudaError_t e_ = (expr);                                                                 \
    if (e_ != cudaSuccess) return fail(MLP_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

struct DevGuard {
  int prev = -1;
  bool changed = false;
  explicit DevGuard(int d) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != d) changed = cudaSetDevice(d) == cudaSuccess;
  }
  ~DevGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

// ---------------------------------------------------------------------------
// Arena layout.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  int L = 0;
  int dtype = 0;
  int64_t B = 0;
  std::vector<int64_t> dims;
  std::vector<int> acts;          // per hidden layer
  int64_t n_params = 0;           // dense count
  int64_t plane_n = 0;            // elements per plane (padded)
  std::vector<int64_t> woff, boff;
  size_t off_P = 0, off_G = 0, off_M = 0, off_V = 0, off_W16 = 0;
  // fp32 models whose GEMMs can run on the tensor cores with operands as
  // three bf16 planes: W16 holds the weight planes, xs the input's planes,
  // h / dY buffers hold planes (6 bytes per element, room for fp32 too)
  bool x3_ok = false;
  size_t off_xs = 0;
  int64_t ld_x = 0;               // row pitch of the input planes
  int64_t max_ld = 8;             // row pitch bound of the dY ping-pong buffers
  std::vector<size_t> off_h, off_u;
  std::vector<size_t> off_bits;   // bf16 ReLU layers: the activation's mask as bits, [N / 64][B] words
  std::vector<int64_t> ld_bits;
  std::vector<int64_t> ld_h;
  size_t off_z = 0, off_dz = 0;
  int64_t ldz = 0;
  size_t off_dy[2] = {0, 0};
  size_t off_loss_rows = 0, off_ctl = 0;
  // Split-K partial sums of the weight gradients.  In fp32 models small ones
  // (defer_l: at most 24 MB per layer, 64 MB in all, so they stay in L2) are
  // left for the optimizer to add, in a region per layer since all are read
  // at the end; the others share one region and are reduced right after
  // their GEMM.
  std::vector<size_t> off_wws, wws_bytes;
  std::vector<char> defer_l;
  size_t off_hws = 0, hws_bytes = 0;   // the fused output layer's partials (read by the optimizer)
  size_t off_xin[2] = {0, 0}, off_yin[2] = {0, 0};   // device inputs of mlp_train_step_host (two slots)
  size_t yin_bytes = 0;   // labels, or MSE targets where B * C * 4 <= 64 MiB
  size_t off_norm = 0;   // per-block sums of squares of the gradient (clipping)
  // softmax-CE fused around a wide bf16 output layer: per-row, per-128-column
  // (max, sum) partials, the label logits, and the rows' (max, 1 / sum)
  size_t off_cest = 0, off_cezy = 0, off_cerow = 0;
  size_t total = 0;
};

// Output layers at least this wide (bf16) take softmax-CE inside their GEMMs
// instead of a separate pass over the logits.
constexpr int64_t kCeGemmMinClasses = 1024;

struct Ctl {   // control block at off_ctl
  int64_t step;
  uint32_t err;
  float loss_slot;
  float bias_corr[2];     // AdamW 1/(1-b1^t), 1/sqrt(1-b2^t) of the current step
  float grad_norm;        // ||g||_2 of the last step that clipped
};

mlp_status plan_layout(const int64_t* dims, int n_dims, const int* acts, int act, int dtype, int64_t batch,
                       Layout* Lo) {
  if (!dims || n_dims < 2) return fail(MLP_ERR_ARG, "need at least 2 dims");
  if (dtype != MLP_F32 && dtype != MLP_BF16) return fail(MLP_ERR_DTYPE, "dtype must be MLP_F32 or MLP_BF16");
  if (batch < 1 || batch > (1ll << 30)) return fail(MLP_ERR_SHAPE, "batch out of range");
  Layout& L = *Lo;
  L.L = n_dims - 1;
  L.dtype = dtype;
  L.B = batch;
  L.dims.assign(dims, dims + n_dims);
  for (int i = 0; i < n_dims; ++i)
    if (dims[i] < 1 || dims[i] > (1ll << 30)) return fail(MLP_ERR_SHAPE, "dims[%d] out of range", i);
  L.acts.resize(n_dims - 2);
  for (int i = 0; i < n_dims - 2; ++i) {
    int a = acts ? acts[i] : act;
    if (a < MLP_ACT_NONE || a > MLP_ACT_GELU_TANH) return fail(MLP_ERR_ARG, "bad activation %d", a);
    L.acts[i] = a;
  }
  if (dtype == MLP_BF16)
    for (int i = 0; i < n_dims - 1; ++i)
      if (dims[i] % 8) return fail(MLP_ERR_SHAPE, "bf16 models need input/hidden widths that are multiples of 8");
  // parameter planes
  int64_t off = 0;
  for (int l = 0; l < L.L; ++l) {
    L.woff.push_back(off);
    off += (dims[l + 1] * dims[l] + 63) / 64 * 64;
    L.boff.push_back(off);
    off += (dims[l + 1] + 63) / 64 * 64;
    L.n_params += dims[l + 1] * dims[l] + dims[l + 1];
  }
  L.plane_n = off;
  // tensor cores for an fp32 model: ReLU / none below a fused output layer,
  // 16-byte TMA rows for every GEMM operand
  L.x3_ok = dtype == MLP_F32 && L.L >= 2 && head_supported(dims[L.L], dims[L.L - 1]);
  for (int i = 0; i < n_dims - 2 && L.x3_ok; ++i) L.x3_ok = L.acts[i] != MLP_ACT_GELU_TANH;
  for (int i = 0; i < L.L - 1 && L.x3_ok; ++i) L.x3_ok = dims[i] % 8 == 0;
  const size_t es = dtype == MLP_F32 ? (L.x3_ok ? 6 : 4) : 2;   // activation buffers
  size_t cur = 0;
  auto take = [&](size_t bytes) {
    size_t o = cur;
    cur = align_up(cur + bytes);
    return o;
  };
  L.off_P = take(L.plane_n * 4);
  L.off_G = take(L.plane_n * 4);
  L.off_M = take(L.plane_n * 4);
  L.off_V = take(L.plane_n * 4);
  L.off_W16 = dtype == MLP_BF16 ? take(L.plane_n * 2) : L.x3_ok ? take(L.plane_n * 6) : 0;
  L.ld_x = (dims[0] + 7) / 8 * 8;
  L.off_xs = L.x3_ok ? take(batch * L.ld_x * 6) : 0;
  int64_t max_ld = 8;
  for (int l = 0; l < L.L - 1; ++l) {
    int64_t ld = (dims[l + 1] + 7) / 8 * 8;
    L.ld_h.push_back(ld);
    max_ld = ld > max_ld ? ld : max_ld;
    L.off_h.push_back(take(batch * ld * es));
    L.off_u.push_back(L.acts[l] == MLP_ACT_GELU_TANH ? take(batch * ld * es) : 0);
    const bool bits = dtype == MLP_BF16 && L.acts[l] == MLP_ACT_RELU;
    L.ld_bits.push_back(bits ? batch : 0);
    L.off_bits.push_back(bits ? take((dims[l + 1] + 63) / 64 * batch * 8) : 0);
  }
  L.ldz = (dims[L.L] + 7) / 8 * 8;
  L.off_z = take(batch * L.ldz * es);
  L.off_dz = take(batch * L.ldz * es);
  L.max_ld = max_ld;
  L.off_dy[0] = take(batch * max_ld * es);
  L.off_dy[1] = take(batch * max_ld * es);
  L.off_loss_rows = take(batch * 4);
  size_t shared_ws = 0, deferred = 0;
  std::vector<size_t> need(L.L);
  for (int l = 0; l < L.L; ++l) {
    int s = wgrad_splits(dtype, dims[l + 1], dims[l], batch);
    size_t b = wgrad_workspace_bytes_any(dtype, dims[l + 1], dims[l], batch);
    if (L.x3_ok) {
      s = wgrad_splits(DT_F32X3, dims[l + 1], dims[l], batch);
      const size_t b3 = wgrad_workspace_bytes(DT_F32X3, dims[l + 1], dims[l], batch, s);
      b = b3 > b ? b3 : b;
    }
    need[l] = b;
    const int64_t M = dims[l + 1], MN = dims[l + 1] * dims[l];
    // deferred while the partials stay small enough to live in L2 until the
    // optimizer runs -- for fp32 models, whose short, latency-bound step
    // gains from one kernel less per layer; in bf16 steps the reduce kernel
    // overlaps the next dgrad and deferring measured slower
    const bool d = dtype == MLP_F32 && b > 0 && MN % 4 == 0 && M % 4 == 0 && b <= (24u << 20) &&
                   deferred + b <= (64u << 20);
    if (d) deferred += b;
    L.defer_l.push_back(d);
    if (!d) shared_ws = b > shared_ws ? b : shared_ws;
  }
  const size_t shared_off = shared_ws ? take(shared_ws) : 0;
  for (int l = 0; l < L.L; ++l) {
    if (L.defer_l[l]) {   // 16 bytes of slack: the optimizer reads partial rows 4 floats at a time
      L.wws_bytes.push_back(need[l] + 16);
      L.off_wws.push_back(take(need[l] + 16));
    } else {
      L.wws_bytes.push_back(need[l] ? shared_ws : 0);
      L.off_wws.push_back(shared_off);
    }
  }
  if (n_dims >= 3 && head_supported(dims[L.L], dims[L.L - 1])) {
    L.hws_bytes = head_workspace_bytes(batch, dims[L.L], dims[L.L - 1]);
    L.off_hws = take(L.hws_bytes);
  }
  L.yin_bytes = batch * 4;
  if (batch * dims[L.L] * 4 <= (64ll << 20)) L.yin_bytes = batch * dims[L.L] * 4;
  for (int k = 0; k < 2; ++k) {
    L.off_xin[k] = take(batch * dims[0] * (dtype == MLP_F32 ? 4 : 2));
    L.off_yin[k] = take(L.yin_bytes);
  }
  L.off_norm = take(AdamWOp::kNormParts * sizeof(float));
  if (dtype == MLP_BF16 && dims[L.L] >= kCeGemmMinClasses) {
    L.off_cest = take(batch * ce_groups(dims[L.L]) * 8);
    L.off_cezy = take(batch * 4);
    L.off_cerow = take(batch * 8);
  }
  L.off_ctl = take(sizeof(Ctl));
  L.total = cur;
  return MLP_OK;
}

// splitmix64 + Box-Muller: host generator for the Kaiming-normal draw.
struct HostRng {
  uint64_t s;
  uint64_t next() {
    uint64_t z = (s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
  double uniform() { return ((next() >> 11) + 0.5) * (1.0 / 9007199254740992.0); }   // (0, 1)
  bool have = false;
  double spare = 0;
  double normal() {
    if (have) { have = false; return spare; }
    double u1 = uniform(), u2 = uniform();
    double r = sqrt(-2.0 * log(u1)), th = 6.283185307179586 * u2;
    spare = r * sin(th);
    have = true;
    return r * cos(th);
  }
};

struct GraphCache {
  int n_steps = 0;
  bool pdl = false;   // built with programmatic (early-launch) edges
  cudaGraphExec_t exec = nullptr;
  cudaGraph_t graph = nullptr;
  std::vector<cudaGraphNode_t> nodes;
  std::vector<LaunchRec> recs;
};

}  // namespace

struct mlp {
  int device = 0;
  Layout lay;
  uint8_t* arena = nullptr;
  size_t arena_bytes = 0;
  bool use_graph = true;
  bool fuse_head = true;     // fused output layer + CE where the shape allows
  bool f32_tc = true;        // fp32 GEMMs on the tensor cores (three bf16 planes) where the model allows
  bool pdl = true;           // graph edges let each kernel launch before its predecessor ends
  int optim = MLP_OPTIM_ADAMW;
  int loss = MLP_LOSS_CE;
  bool ce_gemm = false;      // softmax-CE inside the GEMMs of a wide bf16 output layer (slower on this part)
  bool relu_bits = true;     // bf16 ReLU masks as bits between the forward and the dgrad
  bool head_in_gemm = true;  // fp32 planes: the fused output layer inside the forward GEMM below it
  int gemm_2sm = -1;         // bf16 forward / dgrad on CTA pairs with 2-SM MMAs (GemmOp::cg2)
  float max_grad_norm = 0.f; // > 0: global-norm clipping of the gradient before the update
  std::mutex mu;
  std::vector<GraphCache> graphs;
  int kernels_per_step = 0;
  // mlp_train_step_host: copy streams and two input slots, so the copies of
  // step i+1 run while step i computes
  // x is copied in this many pieces, one per stream (copy engine).  One: the
  // step then waits on a single event (each cross-stream wait between two
  // graph launches idles the GPU for a moment), and one copy engine moves a
  // 4096-row fp32 batch well within a step (measured: 2 % more end to end
  // than with two streams)
  static constexpr int kCopyStreams = 1;
  cudaStream_t copy_stream[kCopyStreams] = {};
  cudaEvent_t copied[2][kCopyStreams] = {}, consumed[2] = {nullptr, nullptr};
  int host_calls = 0;

  float* plane(int which) const {
    size_t off = which == MLP_PLANE_P ? lay.off_P : which == MLP_PLANE_G ? lay.off_G
               : which == MLP_PLANE_M ? lay.off_M : lay.off_V;
    return reinterpret_cast<float*>(arena + off);
  }
  void* w16() const { return lay.dtype == MLP_BF16 || lay.x3_ok ? (void*)(arena + lay.off_W16) : nullptr; }
  // the training step's GEMMs take fp32 operands as bf16 planes
  bool x3() const { return lay.x3_ok && f32_tc && fuse_head; }
  Ctl* ctl() const { return reinterpret_cast<Ctl*>(arena + lay.off_ctl); }
  size_t es() const { return lay.dtype == MLP_F32 ? 4 : 2; }
  void* at(size_t off) const { return arena + off; }
  // weight operand of layer l in the compute dtype
  const void* weight(int l) const {
    return lay.dtype == MLP_BF16 ? (const void*)((const uint16_t*)w16() + lay.woff[l])
                                 : (const void*)(plane(MLP_PLANE_P) + lay.woff[l]);
  }
  // weight of layer l as three bf16 planes (plane pitch lay.plane_n)
  const void* weight_planes(int l) const { return (const void*)((const uint16_t*)w16() + lay.woff[l]); }
  ~mlp() {
    for (int k = 0; k < 2; ++k) {
      for (int c = 0; c < kCopyStreams; ++c)
        if (copied[k][c]) cudaEventDestroy(copied[k][c]);
      if (consumed[k]) cudaEventDestroy(consumed[k]);
    }
    for (int c = 0; c < kCopyStreams; ++c)
      if (copy_stream[c]) cudaStreamDestroy(copy_stream[c]);
    for (auto& g : graphs) {
      if (g.exec) cudaGraphExecDestroy(g.exec);
      if (g.graph) cudaGraphDestroy(g.graph);
    }
  }
};

namespace {

mlp_status add(std::vector<LaunchRec>& out, int n, const LaunchRec* recs) {
  for (int i = 0; i < n; ++i) out.push_back(recs[i]);
  return MLP_OK;
}

#define PLAN_TRY(call)                                              \
  do {                                                              \
    char e_[512] = "";                                              \
    LaunchRec r_[2];                                                \
    int n_ = (call);                                                \
    if (n_ < 0) return fail(MLP_ERR_SHAPE, "%s", e_);               \
    add(out, n_, r_);                                               \
  } while (0)

// Forward GEMMs of layers [0, n_layers) (all layers: logits into the arena's
// z buffer).  x3: fp32 model with operands as bf16 planes (the input is
// split into the arena's xs planes first; hidden outputs are planes).
mlp_status plan_forward(const mlp* m, const void* x, std::vector<LaunchRec>& out, int n_layers = -1,
                        bool x3 = false, const int32_t* ce_labels = nullptr, const GemmOp* head_fold = nullptr) {
  const Layout& L = m->lay;
  const void* X = x;
  int64_t ldx = L.dims[0], xplane = 0;
  if (n_layers < 0) n_layers = L.L;
  if (x3) {
    char e_[512] = "";
    LaunchRec r;
    if (split3_plan(L.B, L.dims[0], (const float*)x, L.dims[0], m->at(L.off_xs), L.ld_x, L.B * L.ld_x, &r, e_,
                    sizeof(e_)) < 0)
      return fail(MLP_ERR_SHAPE, "%s", e_);
    out.push_back(r);
    X = m->at(L.off_xs); ldx = L.ld_x; xplane = L.B * L.ld_x;
  }
  for (int l = 0; l < n_layers; ++l) {
    GemmOp op;
    op.dtype = x3 ? DT_F32X3 : L.dtype;
    op.kind = GEMM_FWD;
    op.M = L.B; op.N = L.dims[l + 1]; op.K = L.dims[l];
    op.A = X; op.lda = ldx; op.a_kmajor = true; op.a_plane = xplane;
    op.B = x3 ? m->weight_planes(l) : m->weight(l); op.ldb = L.dims[l]; op.b_kmajor = true;
    op.b_plane = L.plane_n;
    op.bias = m->plane(MLP_PLANE_P) + L.boff[l];
    op.err = &m->ctl()->err;
    op.cg2 = m->gemm_2sm;
    if (l < L.L - 1) {
      op.act = L.acts[l];
      op.out = m->at(L.off_h[l]); op.ldo = L.ld_h[l]; op.out_plane = L.B * L.ld_h[l];
      if (op.act == MLP_ACT_GELU_TANH) { op.out_u = m->at(L.off_u[l]); op.ldu = L.ld_h[l]; }
      if (m->relu_bits && L.ld_bits[l] && !x3) {
        op.relu_bits = (uint64_t*)m->at(L.off_bits[l]); op.ld_bits = L.ld_bits[l];
      }
      X = op.out; ldx = L.ld_h[l]; xplane = op.out_plane;
      if (head_fold && l == n_layers - 1) {   // the output layer in this epilogue: it writes dY, not h
        op.head_W = head_fold->head_W; op.head_bias = head_fold->head_bias; op.head_labels = head_fold->head_labels;
        op.head_ws = head_fold->head_ws; op.head_scale = head_fold->head_scale;
        op.step_counter = head_fold->step_counter; op.bias_corr = head_fold->bias_corr;
        op.beta1 = head_fold->beta1; op.beta2 = head_fold->beta2;
        op.out = head_fold->out; op.ldo = head_fold->ldo; op.out_plane = head_fold->out_plane;
      }
    } else {
      op.act = MLP_ACT_NONE;
      op.out = m->at(L.off_z); op.ldo = L.ldz;
      if (ce_labels) {   // softmax-CE statistics from the logits' epilogue
        op.ce_stats = (float2*)m->at(L.off_cest); op.ce_zy = (float*)m->at(L.off_cezy); op.ce_labels = ce_labels;
      }
    }
    PLAN_TRY(gemm_plan(op, r_, e_, sizeof(e_)));
    // what a traced step copies aside
    LaunchRec& r = out.back();
    const int planes = x3 ? 3 : 1, eb = x3 ? 2 : (int)m->es();
    if (l == L.L - 1) {
      r.add_out(MLP_TRACE_Z, l, op.out, L.B, L.dims[l + 1], op.ldo, eb);
    } else if (head_fold && l == n_layers - 1) {
      r.add_out(MLP_TRACE_DY, l, op.out, L.B, L.dims[l + 1], op.ldo, eb, planes, op.out_plane);
    } else {
      r.add_out(MLP_TRACE_H, l, op.out, L.B, L.dims[l + 1], op.ldo, eb, planes, op.out_plane);
      if (op.out_u) r.add_out(MLP_TRACE_U, l, op.out_u, L.B, L.dims[l + 1], op.ldu, eb);
    }
  }
  return MLP_OK;
}

struct Hyper { float lr, b1, b2, eps, wd; };

// A step's plan.  grad_only: forward and backward only, the gradient left
// finished in G (no update; the update is planned by plan_update).
// scale_batch > 0: the loss and its gradient are those of a mean over
// scale_batch rows of which this batch is a part (a data-parallel shard);
// 0: over this batch.
mlp_status plan_step(const mlp* m, const void* x, const void* y, const Hyper& hp, float* loss,
                     std::vector<LaunchRec>& out, bool grad_only = false, int64_t scale_batch = 0) {
  const Layout& L = m->lay;
  const bool mse = m->loss == MLP_LOSS_MSE;
  const double Bs = (double)(scale_batch > 0 ? scale_batch : L.B);   // the batch the loss is a mean over
  const bool fuse = m->fuse_head && L.L >= 2 && head_supported(L.dims[L.L], L.dims[L.L - 1]);
  const bool x3 = m->x3();   // implies fuse
  // a wide bf16 output layer: softmax-CE inside its GEMMs (statistics from the
  // forward's epilogue, dz formed from the stored logits by dgrad and wgrad)
  const bool ce_gemm = !mse && !fuse && m->ce_gemm && L.dtype == MLP_BF16 && L.dims[L.L] >= kCeGemmMinClasses;
  const int64_t dy_plane = L.B * L.max_ld;
  Ctl* ctl = m->ctl();
  // fp32 planes: the fused output layer inside the epilogue of the forward
  // below it, where that forward runs on CTA pairs
  const bool head_gemm = fuse && x3 && !mse && m->head_in_gemm &&
                         tc_fused_head_ok(L.B, L.dims[L.L - 1], L.dims[L.L - 2], L.dims[L.L]);
  GemmOp hf;
  if (head_gemm) {
    const int l = L.L - 1;
    hf.head_W = (const float*)m->weight(l);   // fp32 master weights (an fp32 model)
    hf.head_bias = m->plane(MLP_PLANE_P) + L.boff[l];
    hf.head_labels = (const int32_t*)y;
    hf.head_ws = (float*)m->at(L.off_hws);
    hf.head_scale = (float)(1.0 / Bs);
    hf.step_counter = &ctl->step;
    hf.bias_corr = ctl->bias_corr; hf.beta1 = hp.b1; hf.beta2 = hp.b2;
    hf.out = m->at(L.off_dy[0]); hf.ldo = L.ld_h[l - 1]; hf.out_plane = dy_plane;
  }
  mlp_status st = plan_forward(m, x, out, fuse ? L.L - 1 : L.L, x3, ce_gemm ? (const int32_t*)y : nullptr,
                               head_gemm ? &hf : nullptr);
  if (st != MLP_OK) return st;
  const void* dY = m->at(L.off_dz);
  int64_t ldy = L.ldz;
  int buf = 0;
  int top = L.L - 1;   // highest layer whose wgrad/dgrad still has to be planned
  if (head_gemm) {
    dY = hf.out; ldy = hf.ldo;
    buf = 1;
    top = L.L - 2;
  } else if (fuse) {
    // output layer + CE + its VJPs in one kernel; dY of the last hidden layer
    // goes to the first ping-pong buffer
    const int l = L.L - 1;
    HeadOp hd;
    hd.dtype = x3 ? DT_F32X3 : L.dtype; hd.act = L.acts[l - 1];
    hd.B = L.B; hd.C = L.dims[L.L]; hd.K = L.dims[l];
    hd.h = m->at(L.off_h[l - 1]); hd.ldh = L.ld_h[l - 1];
    hd.h_plane = L.B * L.ld_h[l - 1]; hd.dy_plane = dy_plane;
    hd.W = m->weight(l);   // fp32 master weights for an fp32 model
    hd.bias = m->plane(MLP_PLANE_P) + L.boff[l];
    if (mse) {
      hd.targets = (const float*)y; hd.ldt = L.dims[L.L];
    } else {
      hd.labels = (const int32_t*)y;
    }
    hd.aux = hd.act == MLP_ACT_GELU_TANH ? m->at(L.off_u[l - 1]) : m->at(L.off_h[l - 1]);
    hd.ld_aux = L.ld_h[l - 1];
    hd.dY = m->at(L.off_dy[0]); hd.ldy = L.ld_h[l - 1];
    hd.step_counter = &ctl->step;
    hd.err = &ctl->err;
    hd.ws = (float*)m->at(L.off_hws); hd.ws_bytes = L.hws_bytes;
    hd.grad_scale = (float)((mse ? 2.0 / (double)L.dims[L.L] : 1.0) / Bs);
    hd.bias_corr = ctl->bias_corr; hd.beta1 = hp.b1; hd.beta2 = hp.b2;
    char e_[512] = "";
    LaunchRec r;
    if (head_plan(hd, &r, e_, sizeof(e_)) < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
    r.add_out(MLP_TRACE_DY, l - 1, hd.dY, L.B, L.dims[l], hd.ldy, x3 ? 2 : (int)m->es(), x3 ? 3 : 1, dy_plane);
    out.push_back(r);
    dY = hd.dY; ldy = hd.ldy;
    buf = 1;
    top = L.L - 2;
  } else {
    char e_[512] = "";
    LaunchRec r;
    float* loss_rows = (float*)m->at(L.off_loss_rows);
    if (ce_gemm) {
      CeCombineOp cc;
      cc.B = L.B; cc.C = L.dims[L.L];
      cc.stats = (const float2*)m->at(L.off_cest); cc.zy = (const float*)m->at(L.off_cezy);
      cc.labels = (const int32_t*)y;
      cc.rowstat = (float2*)m->at(L.off_cerow); cc.loss_rows = loss_rows; cc.err = &ctl->err;
      if (ce_combine_plan(cc, &r, e_, sizeof(e_)) < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
      dY = m->at(L.off_z);   // the top layer's VJPs read the logits and form dz themselves
    } else if (mse) {
      MseOp op;
      op.dtype = L.dtype; op.B = L.B; op.C = L.dims[L.L];
      op.z = m->at(L.off_z); op.ldz = L.ldz;
      op.t = (const float*)y; op.ldt = L.dims[L.L];
      op.dz = m->at(L.off_dz); op.lddz = L.ldz;
      op.loss_rows = loss_rows;
      op.grad_scale = (float)(2.0 / (Bs * (double)L.dims[L.L]));
      if (mse_plan(op, &r, e_, sizeof(e_)) < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
    } else {
      CeOp ce;
      ce.dtype = L.dtype; ce.B = L.B; ce.C = L.dims[L.L];
      ce.z = m->at(L.off_z); ce.ldz = L.ldz;
      ce.labels = (const int32_t*)y;
      ce.dz = m->at(L.off_dz); ce.lddz = L.ldz;
      ce.loss_rows = loss_rows;
      ce.grad_scale = (float)(1.0 / Bs);
      ce.err = &ctl->err;
      if (ce_plan(ce, &r, e_, sizeof(e_)) < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
    }
    if (!ce_gemm) r.add_out(MLP_TRACE_DZ, L.L - 1, m->at(L.off_dz), L.B, L.dims[L.L], L.ldz, (int)m->es());
    r.add_out(MLP_TRACE_LOSS_ROWS, L.L - 1, loss_rows, L.B, 1, 1, 4);
    out.push_back(r);
    r.nouts = 0;   // the record is reused for the loss mean, which writes no traced tensor
    LossMeanOp lm;
    lm.B = L.B; lm.loss_rows = loss_rows;
    lm.count = mse ? Bs * (double)L.dims[L.L] : Bs;
    lm.loss = loss ? loss : &ctl->loss_slot;
    lm.step_counter = &ctl->step;
    lm.err = &ctl->err;
    lm.bias_corr = ctl->bias_corr; lm.beta1 = hp.b1; lm.beta2 = hp.b2;
    if (loss_mean_plan(lm, &r, e_, sizeof(e_)) < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
    out.push_back(r);
  }
  float* G = m->plane(MLP_PLANE_G);
  AdamWOp::Seg seg[AdamWOp::kMaxSegs];   // gradients the optimizer adds from partial sums
  int nseg = 0;
  // In the graph the weight gradients form a side chain: wgrad(l) runs beside
  // dgrad(l) (both only read dY_l).  dgrad(l) also waits for wgrad(l+1), the
  // last reader of the ping-pong buffer it overwrites; the optimizer joins both.
  int main_tail = (int)out.size() - 1, side_tail = -1;
  for (int l = top; l >= 0; --l) {
    const int side_prev = side_tail;
    const int wg_first = (int)out.size();
    const void* Xl = l == 0 ? (x3 ? m->at(L.off_xs) : x) : m->at(L.off_h[l - 1]);
    const int64_t ldxl = l == 0 ? (x3 ? L.ld_x : L.dims[0]) : L.ld_h[l - 1];
    GemmOp wg;
    wg.dtype = x3 ? DT_F32X3 : L.dtype; wg.kind = GEMM_WGRAD;
    wg.M = L.dims[l + 1]; wg.N = L.dims[l]; wg.K = L.B;
    wg.A = dY; wg.lda = ldy; wg.a_kmajor = false; wg.a_plane = dy_plane;
    wg.B = Xl; wg.ldb = ldxl; wg.b_kmajor = false; wg.b_plane = L.B * ldxl;
    wg.dW = G + L.woff[l]; wg.ld_dw = L.dims[l];
    wg.db = G + L.boff[l];
    wg.ws = L.wws_bytes[l] ? (float*)m->at(L.off_wws[l]) : nullptr; wg.ws_bytes = L.wws_bytes[l];
    wg.err = &ctl->err;
    wg.cg2 = m->gemm_2sm;
    const bool ce_top = ce_gemm && l == L.L - 1;
    if (ce_top) {
      wg.ce_rowstat = (const float2*)m->at(L.off_cerow); wg.ce_labels = (const int32_t*)y;
      wg.ce_scale = (float)(1.0 / Bs);
    }
    // split-K partials go to the optimizer (it reads them 4 at a time)
    const int64_t MN = wg.M * wg.N;
    int used = 0;
    wg.defer_reduce = L.defer_l[l] && nseg + 2 <= AdamWOp::kMaxSegs;
    wg.splits_out = &used;
    {
      char e_[512] = "";
      LaunchRec r_[2];
      const int n_ = gemm_plan(wg, r_, e_, sizeof(e_));
      if (n_ < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
      add(out, n_, r_);
      const int d[2] = {main_tail, side_tail};
      out[wg_first].depend_on(d, 2);   // a split-K reduce after it follows it
      side_tail = (int)out.size() - 1;
      if (n_ == 1 && used > 1) {
        seg[nseg++] = AdamWOp::Seg{L.woff[l], MN, wg.ws, used, MN};
        seg[nseg++] = AdamWOp::Seg{L.boff[l], wg.M, wg.ws + (int64_t)used * MN, used, wg.M};
      }
    }
    if (l > 0) {
      GemmOp dg;
      dg.dtype = x3 ? DT_F32X3 : L.dtype; dg.kind = GEMM_DGRAD;
      dg.act = L.acts[l - 1];
      dg.M = L.B; dg.N = L.dims[l]; dg.K = L.dims[l + 1];
      dg.A = dY; dg.lda = ldy; dg.a_kmajor = true; dg.a_plane = dy_plane;
      dg.B = x3 ? m->weight_planes(l) : m->weight(l); dg.ldb = L.dims[l]; dg.b_kmajor = false;
      dg.b_plane = L.plane_n; dg.out_plane = dy_plane;
      dg.aux = dg.act == MLP_ACT_GELU_TANH ? m->at(L.off_u[l - 1]) : m->at(L.off_h[l - 1]);
      dg.ld_aux = L.ld_h[l - 1];
      if (m->relu_bits && L.ld_bits[l - 1] && !x3) {
        dg.relu_bits = (uint64_t*)m->at(L.off_bits[l - 1]); dg.ld_bits = L.ld_bits[l - 1];
      }
      dg.out = m->at(L.off_dy[buf]); dg.ldo = L.ld_h[l - 1];
      dg.err = &ctl->err;
      dg.cg2 = m->gemm_2sm;
      if (ce_top) {
        dg.ce_rowstat = wg.ce_rowstat; dg.ce_labels = wg.ce_labels; dg.ce_scale = wg.ce_scale;
      }
      PLAN_TRY(gemm_plan(dg, r_, e_, sizeof(e_)));
      out.back().add_out(MLP_TRACE_DY, l - 1, dg.out, L.B, L.dims[l], dg.ldo, x3 ? 2 : (int)m->es(), x3 ? 3 : 1,
                         dy_plane);
      const int d[2] = {main_tail, side_prev};
      out.back().depend_on(d, 2);
      main_tail = (int)out.size() - 1;
      dY = dg.out; ldy = dg.ldo;
      buf ^= 1;
    }
  }
  AdamWOp ad;
  ad.n = L.plane_n;
  ad.p = m->plane(MLP_PLANE_P); ad.g = G; ad.m = m->plane(MLP_PLANE_M); ad.v = m->plane(MLP_PLANE_V);
  ad.w16 = L.dtype == MLP_BF16 || x3 ? m->w16() : nullptr;
  ad.w16_plane = x3 ? L.plane_n : 0;
  ad.step_counter = &ctl->step;
  ad.bias_corr = ctl->bias_corr;
  ad.lr = hp.lr; ad.beta1 = hp.b1; ad.beta2 = hp.b2; ad.eps = hp.eps; ad.wd = hp.wd;
  ad.kind = m->optim;
  ad.max_norm = m->max_grad_norm;
  ad.norm_ws = (float*)m->at(L.off_norm);
  ad.norm_out = &ctl->grad_norm;
  for (int k = 0; k < nseg; ++k) ad.seg[ad.nseg++] = seg[k];
  if (fuse) {   // the output layer's gradient and the loss arrive as partial sums
    const int l = L.L - 1;
    const HeadPartials hpart =
        head_gemm ? tc_fused_head_partials(L.B) : head_partials(L.B, L.dims[L.L], L.dims[l]);
    const float* hws = (const float*)m->at(L.off_hws);
    const int64_t nw = L.dims[L.L] * L.dims[l];
    ad.seg[ad.nseg++] = AdamWOp::Seg{L.woff[l], nw, hws, hpart.n, hpart.stride};
    ad.seg[ad.nseg++] = AdamWOp::Seg{L.boff[l], L.dims[L.L], hws + nw, hpart.n, hpart.stride};
    ad.loss_parts = hws + hpart.loss_off; ad.loss_n = hpart.n;
    ad.loss_scale = (float)(1.0 / (Bs * (mse ? (double)L.dims[L.L] : 1.0)));
    ad.loss = loss ? loss : &ctl->loss_slot;
    ad.err = &ctl->err;
  }
  char e_[512] = "";
  LaunchRec r[2];
  if (grad_only) {
    // the gradient finished where parts of it are still partial sums (and
    // the loss formed from the output layer's partials); else nothing to do
    if (ad.nseg == 0 && !ad.loss_parts) return MLP_OK;
    if (grad_finish_plan(ad, r, e_, sizeof(e_)) < 0) return fail(MLP_ERR_ARG, "%s", e_);
    const int d[1] = {side_tail >= 0 ? side_tail : main_tail};
    r[0].depend_on(d, 1);
    add(out, 1, r);
    return MLP_OK;
  }
  const int nr = adamw_plan(ad, r, e_, sizeof(e_));
  if (nr < 0) return fail(MLP_ERR_ARG, "%s", e_);
  // the last weight gradient already follows the last dgrad (a single edge
  // can be an early-launch one); with clipping the update follows the norm
  const int d[1] = {side_tail >= 0 ? side_tail : main_tail};
  r[0].depend_on(d, 1);
  add(out, nr, r);
  return MLP_OK;
}

// The update half of a split step: the model's update rule over the
// finished gradient in G, at the step counter the gradient step advanced
// (bias corrections from that t and the betas given here).
mlp_status plan_update(const mlp* m, const Hyper& hp, std::vector<LaunchRec>& out) {
  const Layout& L = m->lay;
  Ctl* ctl = m->ctl();
  const bool x3 = m->x3();
  AdamWOp ad;
  ad.n = L.plane_n;
  ad.p = m->plane(MLP_PLANE_P); ad.g = m->plane(MLP_PLANE_G);
  ad.m = m->plane(MLP_PLANE_M); ad.v = m->plane(MLP_PLANE_V);
  ad.w16 = L.dtype == MLP_BF16 || x3 ? m->w16() : nullptr;
  ad.w16_plane = x3 ? L.plane_n : 0;
  ad.step_counter = &ctl->step;
  ad.bias_corr = nullptr;
  ad.lr = hp.lr; ad.beta1 = hp.b1; ad.beta2 = hp.b2; ad.eps = hp.eps; ad.wd = hp.wd;
  ad.kind = m->optim;
  ad.max_norm = m->max_grad_norm;
  ad.norm_ws = (float*)m->at(L.off_norm);
  ad.norm_out = &ctl->grad_norm;
  char e_[512] = "";
  LaunchRec r[2];
  const int nr = adamw_plan(ad, r, e_, sizeof(e_));
  if (nr < 0) return fail(MLP_ERR_ARG, "%s", e_);
  add(out, nr, r);
  return MLP_OK;
}

// Graph-cache keys of the two halves of a split step (whole steps use n >= 1).
constexpr int kGradStepKey = -1, kUpdateKey = -2;

mlp_status launch_eager(const std::vector<LaunchRec>& recs, cudaStream_t s) {
  for (const auto& r : recs) {
    cudaError_t e = launch_rec(r, s);
    if (e != cudaSuccess) return fail(MLP_ERR_CUDA, "launch of %s failed: %s", r.name, cudaGetErrorString(e));
  }
  return MLP_OK;
}

bool same_topology(const std::vector<LaunchRec>& a, const std::vector<LaunchRec>& b) {
  if (a.size() != b.size()) return false;
  for (size_t i = 0; i < a.size(); ++i) {
    const LaunchRec &x = a[i], &y = b[i];
    if (x.func != y.func || x.grid.x != y.grid.x || x.grid.y != y.grid.y || x.grid.z != y.grid.z ||
        x.block.x != y.block.x || x.smem != y.smem || !x.same_deps(y))
      return false;
  }
  return true;
}

mlp_status launch_graph(mlp* m, int key, std::vector<LaunchRec>& recs, cudaStream_t s) {
  GraphCache* gc = nullptr;
  for (auto& g : m->graphs)
    if (g.n_steps == key) gc = &g;
  if (gc && (!same_topology(gc->recs, recs) || gc->pdl != m->pdl)) {
    cudaGraphExecDestroy(gc->exec);
    cudaGraphDestroy(gc->graph);
    gc->exec = nullptr;
    gc->graph = nullptr;
    gc->nodes.clear();
    gc->recs.clear();
  }
  if (!gc) {
    m->graphs.emplace_back();
    gc = &m->graphs.back();
    gc->n_steps = key;
  }
  if (!gc->exec) {
    CUDA_TRY(cudaGraphCreate(&gc->graph, 0));
    // Each record depends on the one before it unless it names its own
    // dependencies (the side chain of weight gradients).  With pdl the edge
    // from an early-launch record's first dependency (its predecessor on the
    // main chain) is programmatic: the kernel may be scheduled once every
    // block of that predecessor has started, and waits inside
    // (griddepcontrol.wait) for it to complete.  Its other dependencies stay
    // full edges (complete before the launch).
    cudaGraphEdgeData ed;
    memset(&ed, 0, sizeof(ed));
    ed.from_port = cudaGraphKernelNodePortProgrammatic;
    ed.type = cudaGraphDependencyTypeProgrammatic;
    for (size_t i = 0; i < recs.size(); ++i) {
      const LaunchRec& r = recs[i];
      cudaGraphNode_t dn[LaunchRec::kMaxDeps];
      int nd = 0;
      if (r.ndeps < 0) {
        if (i > 0) dn[nd++] = gc->nodes[i - 1];
      } else {
        for (int k = 0; k < r.ndeps; ++k) {
          if (r.deps[k] < 0 || r.deps[k] >= (int)i) return fail(MLP_ERR_STATE, "bad plan dependency");
          dn[nd++] = gc->nodes[r.deps[k]];
        }
      }
      void* argp[1];
      cudaKernelNodeParams kp = node_params(r, argp);
      cudaGraphNode_t node;
      if (nd >= 1 && m->pdl && r.early) {
        CUDA_TRY(cudaGraphAddKernelNode(&node, gc->graph, nullptr, 0, &kp));
        CUDA_TRY(cudaGraphAddDependencies(gc->graph, dn, &node, &ed, 1));
        for (int k = 1; k < nd; ++k) CUDA_TRY(cudaGraphAddDependencies(gc->graph, dn + k, &node, nullptr, 1));
      } else {
        CUDA_TRY(cudaGraphAddKernelNode(&node, gc->graph, nd ? dn : nullptr, nd, &kp));
      }
      gc->nodes.push_back(node);
    }
    gc->pdl = m->pdl;
    CUDA_TRY(cudaGraphInstantiate(&gc->exec, gc->graph, 0));
    gc->recs = recs;
  } else {
    for (size_t i = 0; i < recs.size(); ++i) {
      if (recs[i].same_as(gc->recs[i])) continue;
      void* argp[1];
      cudaKernelNodeParams kp = node_params(recs[i], argp);
      CUDA_TRY(cudaGraphExecKernelNodeSetParams(gc->exec, gc->nodes[i], &kp));
      gc->recs[i] = recs[i];
    }
  }
  CUDA_TRY(cudaGraphLaunch(gc->exec, s));
  return MLP_OK;
}

mlp_status run(mlp* m, int key, std::vector<LaunchRec>& recs, cudaStream_t s) {
  mlp_status st = m->use_graph ? launch_graph(m, key, recs, s) : launch_eager(recs, s);
  if (st != MLP_OK) return st;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MLP_ERR_CUDA, "after launch: %s", cudaGetErrorString(e));
  return ok();
}

// The bf16 copy of the P plane the GEMMs read: one plane for a bf16 model,
// three (hi, mid, lo) for an fp32 model that can run on the tensor cores.
// Synchronous (create, write_params, option changes).
cudaError_t refresh_w16(mlp* m) {
  const Layout& L = m->lay;
  if (L.dtype != MLP_BF16 && !L.x3_ok) return cudaSuccess;
  char eb[256];
  LaunchRec r;
  int n = L.dtype == MLP_BF16
              ? cast_bf16_plan(L.plane_n, m->plane(MLP_PLANE_P), m->w16(), &r, eb, sizeof(eb))
              : split3_plan(1, L.plane_n, m->plane(MLP_PLANE_P), L.plane_n, m->w16(), L.plane_n, L.plane_n, &r, eb,
                            sizeof(eb));
  if (n < 0) return cudaErrorInvalidValue;
  cudaError_t e = launch_rec(r, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return e;
}

}  // namespace

// ---------------------------------------------------------------------------
// C ABI: model.
// ---------------------------------------------------------------------------
extern "C" {

const char* mlp_last_error(void) { return g_err; }

size_t mlp_arena_bytes(const int64_t* dims, int n_dims, const int* acts, int act, int dtype, int64_t batch) {
  Layout L;
  if (plan_layout(dims, n_dims, acts, act, dtype, batch, &L) != MLP_OK) return 0;
  return L.total;
}

mlp_status mlp_create(const int64_t* dims, int n_dims, const int* acts, int act, int dtype, uint64_t seed,
                      int64_t batch, void* arena_dev, size_t arena_bytes, int device, mlp_t** out) {
  if (!out) return fail(MLP_ERR_ARG, "out is NULL");
  *out = nullptr;
  Layout L;
  mlp_status st = plan_layout(dims, n_dims, acts, act, dtype, batch, &L);
  if (st != MLP_OK) return st;
  if (!arena_dev) return fail(MLP_ERR_ARG, "arena is NULL");
  if ((uintptr_t)arena_dev % kAlign) return fail(MLP_ERR_ARG, "arena must be %zu-byte aligned", kAlign);
  if (arena_bytes < L.total) return fail(MLP_ERR_ARG, "arena too small (%zu < %zu)", arena_bytes, L.total);
  int ndev = 0;
  CUDA_TRY(cudaGetDeviceCount(&ndev));
  if (device < 0 || device >= ndev) return fail(MLP_ERR_ARG, "device %d not present", device);
  DevGuard g(device);
  cudaPointerAttributes pa;
  CUDA_TRY(cudaPointerGetAttributes(&pa, arena_dev));
  if (pa.type != cudaMemoryTypeDevice || pa.device != device)
    return fail(MLP_ERR_ARG, "arena is not device memory of device %d", device);
  mlp* m = new mlp();
  m->device = device;
  m->lay = L;
  m->arena = (uint8_t*)arena_dev;
  m->arena_bytes = arena_bytes;
  cudaError_t e = cudaMemset(arena_dev, 0, L.total);
  // Kaiming-normal weights, zero biases (P plane), drawn on the host.
  std::vector<float> host(L.plane_n, 0.f);
  HostRng rng{seed ^ 0x6A09E667F3BCC909ull};
  for (int l = 0; l < L.L && e == cudaSuccess; ++l) {
    const double std_ = sqrt(2.0 / (double)L.dims[l]);
    const int64_t n = L.dims[l + 1] * L.dims[l];
    for (int64_t i = 0; i < n; ++i) host[L.woff[l] + i] = (float)(rng.normal() * std_);
  }
  if (e == cudaSuccess) e = cudaMemcpy(m->plane(MLP_PLANE_P), host.data(), L.plane_n * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = refresh_w16(m);
  if (e != cudaSuccess) {
    delete m;
    return fail(MLP_ERR_CUDA, "create: %s", cudaGetErrorString(e));
  }
  std::vector<LaunchRec> recs;
  Hyper hp{1e-3f, 0.9f, 0.999f, 1e-8f, 0.f};
  st = plan_step(m, arena_dev, (const int32_t*)arena_dev, hp, nullptr, recs);
  if (st != MLP_OK) {
    delete m;
    return st;
  }
  m->kernels_per_step = (int)recs.size();
  *out = m;
  return ok();
}

void mlp_destroy(mlp_t* m) {
  if (!m) return;
  DevGuard g(m->device);
  delete m;
}

int64_t mlp_num_params(const mlp_t* m) { return m ? m->lay.n_params : -1; }
int mlp_num_layers(const mlp_t* m) { return m ? m->lay.L : -1; }
int mlp_kernels_per_step(const mlp_t* m) { return m ? m->kernels_per_step : -1; }

mlp_status mlp_set_optimizer(mlp_t* m, int kind, float max_grad_norm) {
  if (!m) return fail(MLP_ERR_ARG, "model is NULL");
  if (kind < MLP_OPTIM_ADAMW || kind > MLP_OPTIM_SGD) return fail(MLP_ERR_ARG, "unknown optimizer %d", kind);
  if (!(max_grad_norm >= 0.f) || !(max_grad_norm < INFINITY))
    return fail(MLP_ERR_ARG, "max_grad_norm must be finite and >= 0");
  std::lock_guard<std::mutex> lk(m->mu);
  m->optim = kind;
  m->max_grad_norm = max_grad_norm;
  std::vector<LaunchRec> recs;
  mlp_status st = plan_step(m, m->arena, (const int32_t*)m->arena, Hyper{1e-3f, 0.9f, 0.999f, 1e-8f, 0.f},
                            nullptr, recs);
  if (st != MLP_OK) return st;
  m->kernels_per_step = (int)recs.size();
  return ok();
}

mlp_status mlp_set_loss(mlp_t* m, int loss) {
  if (!m) return fail(MLP_ERR_ARG, "model is NULL");
  if (loss != MLP_LOSS_CE && loss != MLP_LOSS_MSE) return fail(MLP_ERR_ARG, "unknown loss %d", loss);
  std::lock_guard<std::mutex> lk(m->mu);
  m->loss = loss;
  std::vector<LaunchRec> recs;
  mlp_status st = plan_step(m, m->arena, m->arena, Hyper{1e-3f, 0.9f, 0.999f, 1e-8f, 0.f}, nullptr, recs);
  if (st != MLP_OK) return st;
  m->kernels_per_step = (int)recs.size();
  return ok();
}

mlp_status mlp_read_grad_norm(mlp_t* m, float* out) {
  if (!m || !out) return fail(MLP_ERR_ARG, "model or out is NULL");
  std::lock_guard<std::mutex> lk(m->mu);
  DevGuard g(m->device);
  CUDA_TRY(cudaDeviceSynchronize());
  CUDA_TRY(cudaMemcpy(out, &m->ctl()->grad_norm, sizeof(float), cudaMemcpyDeviceToHost));
  return ok();
}

mlp_status mlp_set_graph_mode(mlp_t* m, int enable) {
  if (!m) return fail(MLP_ERR_ARG, "model is NULL");
  std::lock_guard<std::mutex> lk(m->mu);
  m->use_graph = enable != 0;
  return ok();
}

mlp_status mlp_set_option(mlp_t* m, int option, int64_t value) {
  if (!m) return fail(MLP_ERR_ARG, "model is NULL");
  std::lock_guard<std::mutex> lk(m->mu);
  switch (option) {
    case MLP_OPT_GRAPH: m->use_graph = value != 0; break;
    case MLP_OPT_FUSE_HEAD: m->fuse_head = value != 0; break;
    case MLP_OPT_F32_TENSOR_CORES: m->f32_tc = value != 0; break;
    case MLP_OPT_PDL: m->pdl = value != 0; break;
    case MLP_OPT_CE_GEMM: m->ce_gemm = value != 0; break;
    case MLP_OPT_RELU_BITS: m->relu_bits = value != 0; break;
    case MLP_OPT_HEAD_IN_GEMM: m->head_in_gemm = value != 0; break;
    case MLP_OPT_GEMM_2SM: m->gemm_2sm = value < 0 ? -1 : value > 0 ? 1 : 0; break;
    default: return fail(MLP_ERR_ARG, "unknown option %d", option);
  }
  if (option == MLP_OPT_FUSE_HEAD || option == MLP_OPT_F32_TENSOR_CORES) {   // planes kept current only while used
    DevGuard g(m->device);
    cudaError_t e = refresh_w16(m);
    if (e != cudaSuccess) return fail(MLP_ERR_CUDA, "refreshing weight planes: %s", cudaGetErrorString(e));
  }
  std::vector<LaunchRec> recs;
  mlp_status st = plan_step(m, m->arena, (const int32_t*)m->arena, Hyper{1e-3f, 0.9f, 0.999f, 1e-8f, 0.f},
                            nullptr, recs);
  if (st != MLP_OK) return st;
  m->kernels_per_step = (int)recs.size();
  return ok();
}

// The launches of mlp_forward.
static mlp_status plan_inference(mlp_t* m, const void* x, void* logits, int32_t* argmax_out,
                                 std::vector<LaunchRec>& recs) {
  const Layout& L = m->lay;
  char e_[512] = "";
  LaunchRec r;
  mlp_status st;
  if (m->x3()) {
    // fp32 model on the tensor cores, as in the training step: the hidden
    // layers on the plane GEMMs, then the last hidden activation joined back
    // into fp32 (exactly) and the small output layer on the FFMA pipes
    st = plan_forward(m, x, recs, L.L - 1, true);
    if (st != MLP_OK) return st;
    const int l = L.L - 1;
    float* hf = (float*)m->at(L.off_dy[0]);   // free outside a step; room for fp32 rows of ld_h
    if (join3_plan(L.B, L.dims[l], m->at(L.off_h[l - 1]), L.ld_h[l - 1], L.B * L.ld_h[l - 1], hf, L.ld_h[l - 1], &r,
                   e_, sizeof(e_)) < 0)
      return fail(MLP_ERR_SHAPE, "%s", e_);
    recs.push_back(r);
    GemmOp op;
    op.dtype = MLP_F32; op.kind = GEMM_FWD; op.act = MLP_ACT_NONE;
    op.M = L.B; op.N = L.dims[L.L]; op.K = L.dims[l];
    op.A = hf; op.lda = L.ld_h[l - 1]; op.a_kmajor = true;
    op.B = m->weight(l); op.ldb = L.dims[l]; op.b_kmajor = true;
    op.bias = m->plane(MLP_PLANE_P) + L.boff[l];
    op.out = m->at(L.off_z); op.ldo = L.ldz;
    op.err = &m->ctl()->err;
    LaunchRec r2[2];
    const int n = gemm_plan(op, r2, e_, sizeof(e_));
    if (n < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
    for (int i = 0; i < n; ++i) recs.push_back(r2[i]);
  } else {
    st = plan_forward(m, x, recs);
    if (st != MLP_OK) return st;
  }
  if (logits) {
    CopyRowsOp c;
    c.dtype = L.dtype; c.B = L.B; c.C = L.dims[L.L];
    c.src = m->at(L.off_z); c.lds = L.ldz;
    c.dst = logits; c.ldd = L.dims[L.L];
    if (copy_rows_plan(c, &r, e_, sizeof(e_)) < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
    recs.push_back(r);
  }
  if (argmax_out) {
    ArgmaxOp a;
    a.dtype = L.dtype; a.B = L.B; a.C = L.dims[L.L];
    a.z = m->at(L.off_z); a.ldz = L.ldz; a.out = argmax_out;
    if (argmax_plan(a, &r, e_, sizeof(e_)) < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
    recs.push_back(r);
  }
  return MLP_OK;
}

mlp_status mlp_forward(mlp_t* m, const void* x, void* logits, int32_t* argmax_out, void* stream) {
  if (!m || !x) return fail(MLP_ERR_ARG, "model or x is NULL");
  std::lock_guard<std::mutex> lk(m->mu);
  DevGuard g(m->device);
  std::vector<LaunchRec> recs;
  mlp_status st = plan_inference(m, x, logits, argmax_out, recs);
  if (st != MLP_OK) return st;
  st = launch_eager(recs, (cudaStream_t)stream);
  if (st != MLP_OK) return st;
  return ok();
}

mlp_status mlp_profile_forward(mlp_t* m, const void* x, void* logits, int32_t* argmax_out, void* stream,
                               float* ms_out, const char** names_out, int max_kernels, int* n_out) {
  if (!m || !x || !n_out || (max_kernels > 0 && !ms_out)) return fail(MLP_ERR_ARG, "bad arguments");
  std::lock_guard<std::mutex> lk(m->mu);
  DevGuard g(m->device);
  std::vector<LaunchRec> recs;
  mlp_status st = plan_inference(m, x, logits, argmax_out, recs);
  if (st != MLP_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const int n = (int)recs.size();
  std::vector<cudaEvent_t> ev(n + 1, nullptr);
  cudaError_t e = cudaSuccess;
  for (int i = 0; i <= n && e == cudaSuccess; ++i) e = cudaEventCreate(&ev[i]);
  for (int i = 0; i < n && e == cudaSuccess; ++i) {
    if (i == 0) e = cudaEventRecord(ev[0], s);
    if (e == cudaSuccess) e = launch_rec(recs[i], s);
    if (e == cudaSuccess) e = cudaEventRecord(ev[i + 1], s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  for (int i = 0; i < n && i < max_kernels && e == cudaSuccess; ++i) {
    e = cudaEventElapsedTime(&ms_out[i], ev[i], ev[i + 1]);
    if (names_out) names_out[i] = recs[i].name;
  }
  for (auto& v : ev)
    if (v) cudaEventDestroy(v);
  if (e != cudaSuccess) return fail(MLP_ERR_CUDA, "profile: %s", cudaGetErrorString(e));
  *n_out = n;
  return ok();
}

mlp_status mlp_train_step(mlp_t* m, const void* x, const void* y, float lr, float b1, float b2, float eps,
                          float wd, float* loss, void* stream) {
  if (!m || !x || !y) return fail(MLP_ERR_ARG, "model, x or labels is NULL");
  if (!(lr >= 0) || !(b1 >= 0 && b1 < 1) || !(b2 >= 0 && b2 < 1) || !(eps >= 0) || !(wd >= 0))
    return fail(MLP_ERR_ARG, "bad hyper-parameters");
  std::lock_guard<std::mutex> lk(m->mu);
  DevGuard g(m->device);
  std::vector<LaunchRec> recs;
  mlp_status st = plan_step(m, x, y, Hyper{lr, b1, b2, eps, wd}, loss, recs);
  if (st != MLP_OK) return st;
  return run(m, 1, recs, (cudaStream_t)stream);
}

mlp_status mlp_train_step_host(mlp_t* m, const void* x_host, const void* y_host, float lr, float b1, float b2,
                               float eps, float wd, float* loss_host, void* stream) {
  if (!m || !x_host || !y_host) return fail(MLP_ERR_ARG, "model, x or labels is NULL");
  if (!(lr >= 0) || !(b1 >= 0 && b1 < 1) || !(b2 >= 0 && b2 < 1) || !(eps >= 0) || !(wd >= 0))
    return fail(MLP_ERR_ARG, "bad hyper-parameters");
  std::lock_guard<std::mutex> lk(m->mu);
  DevGuard g(m->device);
  const Layout& L = m->lay;
  cudaStream_t s = (cudaStream_t)stream;
  constexpr int NC = mlp::kCopyStreams;
  if (!m->copy_stream[0]) {
    for (int c = 0; c < NC; ++c) CUDA_TRY(cudaStreamCreateWithFlags(&m->copy_stream[c], cudaStreamNonBlocking));
    for (int k = 0; k < 2; ++k) {
      for (int c = 0; c < NC; ++c) CUDA_TRY(cudaEventCreateWithFlags(&m->copied[k][c], cudaEventDisableTiming));
      CUDA_TRY(cudaEventCreateWithFlags(&m->consumed[k], cudaEventDisableTiming));
      CUDA_TRY(cudaEventRecord(m->consumed[k], s));
    }
  }
  const int k = m->host_calls & 1;
  uint8_t* xd = (uint8_t*)m->at(L.off_xin[k]);
  void* yd = m->at(L.off_yin[k]);
  const size_t ybytes = m->loss == MLP_LOSS_MSE ? (size_t)L.B * L.dims[L.L] * 4 : (size_t)L.B * 4;
  if (ybytes > L.yin_bytes)
    return fail(MLP_ERR_SHAPE, "MSE targets of %zu bytes do not fit the host-step input slot (%zu)", ybytes,
                L.yin_bytes);
  const size_t xbytes = (size_t)L.B * L.dims[0] * (L.dtype == MLP_F32 ? 4 : 2);
  // slot k is free once the step that last read it has finished; x goes in
  // NC pieces on NC streams (several copy engines), the labels with the last
  const size_t piece = (xbytes / NC + 255) / 256 * 256;
  for (int c = 0; c < NC; ++c) {
    CUDA_TRY(cudaStreamWaitEvent(m->copy_stream[c], m->consumed[k], 0));
    const size_t o = (size_t)c * piece;
    if (o < xbytes) {
      const size_t n = o + piece <= xbytes ? piece : xbytes - o;
      CUDA_TRY(cudaMemcpyAsync(xd + o, (const uint8_t*)x_host + o, n, cudaMemcpyHostToDevice, m->copy_stream[c]));
    }
    if (c == NC - 1)
      CUDA_TRY(cudaMemcpyAsync(yd, y_host, ybytes, cudaMemcpyHostToDevice, m->copy_stream[c]));
    CUDA_TRY(cudaEventRecord(m->copied[k][c], m->copy_stream[c]));
    CUDA_TRY(cudaStreamWaitEvent(s, m->copied[k][c], 0));
  }
  std::vector<LaunchRec> recs;
  // The loss goes straight from the kernel that forms it into page-locked
  // host memory the device can address (a copy node after the step would
  // add its own latency to every step); other host memory gets a copy.
  float* loss_dev = &m->ctl()->loss_slot;
  bool copy_loss = loss_host != nullptr;
  if (loss_host) {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, loss_host) == cudaSuccess && pa.type == cudaMemoryTypeHost && pa.devicePointer) {
      loss_dev = (float*)pa.devicePointer;
      copy_loss = false;
    } else {
      cudaGetLastError();   // not registered memory: clear the query's error, copy instead
    }
  }
  mlp_status st = plan_step(m, xd, yd, Hyper{lr, b1, b2, eps, wd}, loss_dev, recs);
  if (st != MLP_OK) return st;
  st = run(m, 1, recs, s);
  if (st != MLP_OK) return st;
  CUDA_TRY(cudaEventRecord(m->consumed[k], s));
  if (copy_loss) CUDA_TRY(cudaMemcpyAsync(loss_host, &m->ctl()->loss_slot, 4, cudaMemcpyDeviceToHost, s));
  ++m->host_calls;
  return ok();
}

mlp_status mlp_grad_step(mlp_t* m, const void* x, const void* y, int64_t global_batch, float* loss, void* stream) {
  if (!m || !x || !y) return fail(MLP_ERR_ARG, "bad arguments");
  if (global_batch < m->lay.B) return fail(MLP_ERR_ARG, "global_batch (%lld) is smaller than the model's batch (%lld)",
                                           (long long)global_batch, (long long)m->lay.B);
  std::lock_guard<std::mutex> lk(m->mu);
  DevGuard g(m->device);
  std::vector<LaunchRec> recs;
  // (the betas only feed bias corrections that mlp_apply_update recomputes)
  mlp_status st = plan_step(m, x, y, Hyper{0.f, 0.9f, 0.999f, 0.f, 0.f}, loss, recs, true, global_batch);
  if (st != MLP_OK) return st;
  return run(m, kGradStepKey, recs, (cudaStream_t)stream);
}

mlp_status mlp_apply_update(mlp_t* m, float lr, float b1, float b2, float eps, float wd, void* stream) {
  if (!m) return fail(MLP_ERR_ARG, "model is NULL");
  if (!(lr >= 0) || !(b1 >= 0 && b1 < 1) || !(b2 >= 0 && b2 < 1) || !(eps >= 0) || !(wd >= 0))
    return fail(MLP_ERR_ARG, "bad hyper-parameters");
  std::lock_guard<std::mutex> lk(m->mu);
  DevGuard g(m->device);
  std::vector<LaunchRec> recs;
  mlp_status st = plan_update(m, Hyper{lr, b1, b2, eps, wd}, recs);
  if (st != MLP_OK) return st;
  return run(m, kUpdateKey, recs, (cudaStream_t)stream);
}

mlp_status mlp_grad_buffer(mlp_t* m, float** g_dev, int64_t* n) {
  if (!m || !g_dev || !n) return fail(MLP_ERR_ARG, "bad arguments");
  *g_dev = m->plane(MLP_PLANE_G);
  *n = m->lay.plane_n;
  return ok();
}

mlp_status mlp_train_steps(mlp_t* m, int n_steps, const void* const* xs, const void* const* ys, float lr,
                           float b1, float b2, float eps, float wd, float* losses, void* stream) {
  if (!m || !xs || !ys || n_steps < 1) return fail(MLP_ERR_ARG, "bad arguments");
  if (!(lr >= 0) || !(b1 >= 0 && b1 < 1) || !(b2 >= 0 && b2 < 1) || !(eps >= 0) || !(wd >= 0))
    return fail(MLP_ERR_ARG, "bad hyper-parameters");
  std::lock_guard<std::mutex> lk(m->mu);
  DevGuard g(m->device);
  std::vector<LaunchRec> recs;
  for (int i = 0; i < n_steps; ++i) {
    if (!xs[i] || !ys[i]) return fail(MLP_ERR_ARG, "null batch pointer at step %d", i);
    mlp_status st = plan_step(m, xs[i], ys[i], Hyper{lr, b1, b2, eps, wd}, losses ? losses + i : nullptr, recs);
    if (st != MLP_OK) return st;
  }
  return run(m, n_steps, recs, (cudaStream_t)stream);
}

mlp_status mlp_profile_step(mlp_t* m, const void* x, const void* y, float lr, float b1, float b2, float eps,
                            float wd, float* loss, void* stream, float* ms_out, const char** names_out,
                            int max_kernels, int* n_out) {
  if (!m || !x || !y || !n_out || (max_kernels > 0 && !ms_out)) return fail(MLP_ERR_ARG, "bad arguments");
  if (!(lr >= 0) || !(b1 >= 0 && b1 < 1) || !(b2 >= 0 && b2 < 1) || !(eps >= 0) || !(wd >= 0))
    return fail(MLP_ERR_ARG, "bad hyper-parameters");
  std::lock_guard<std::mutex> lk(m->mu);
  DevGuard g(m->device);
  std::vector<LaunchRec> recs;
  mlp_status st = plan_step(m, x, y, Hyper{lr, b1, b2, eps, wd}, loss, recs);
  if (st != MLP_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const int n = (int)recs.size();
  std::vector<cudaEvent_t> ev(n + 1, nullptr);
  cudaError_t e = cudaSuccess;
  for (int i = 0; i <= n && e == cudaSuccess; ++i) e = cudaEventCreate(&ev[i]);
  for (int i = 0; i < n && e == cudaSuccess; ++i) {
    if (i == 0) e = cudaEventRecord(ev[0], s);
    if (e == cudaSuccess) e = launch_rec(recs[i], s);
    if (e == cudaSuccess) e = cudaEventRecord(ev[i + 1], s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  for (int i = 0; i < n && i < max_kernels && e == cudaSuccess; ++i) {
    e = cudaEventElapsedTime(&ms_out[i], ev[i], ev[i + 1]);
    if (names_out) names_out[i] = recs[i].name;
  }
  for (auto& v : ev)
    if (v) cudaEventDestroy(v);
  if (e != cudaSuccess) return fail(MLP_ERR_CUDA, "profile: %s", cudaGetErrorString(e));
  *n_out = n;
  return ok();
}

mlp_status mlp_trace_step(mlp_t* m, const void* x, const void* y, float lr, float b1, float b2, float eps, float wd,
                          float* loss, void* trace_dev, size_t trace_bytes, mlp_trace_entry* entries,
                          int max_entries, int* n_entries, size_t* bytes_needed, void* stream) {
  if (!m || !x || !y) return fail(MLP_ERR_ARG, "bad arguments");
  if (!(lr >= 0) || !(b1 >= 0 && b1 < 1) || !(b2 >= 0 && b2 < 1) || !(eps >= 0) || !(wd >= 0))
    return fail(MLP_ERR_ARG, "bad hyper-parameters");
  std::lock_guard<std::mutex> lk(m->mu);
  DevGuard g(m->device);
  std::vector<LaunchRec> recs;
  mlp_status st = plan_step(m, x, y, Hyper{lr, b1, b2, eps, wd}, loss, recs);
  if (st != MLP_OK) return st;
  // the trace layout: every traced tensor as stored, 256-byte aligned
  std::vector<mlp_trace_entry> ents;
  size_t off = 0;
  for (size_t i = 0; i < recs.size(); ++i) {
    for (int k = 0; k < recs[i].nouts; ++k) {
      const LaunchRec::Out& o = recs[i].outs[k];
      mlp_trace_entry e;
      memset(&e, 0, sizeof(e));
      e.kind = o.kind; e.layer = o.layer; e.launch = (int32_t)i; e.planes = o.planes;
      e.rows = o.rows; e.cols = o.cols; e.ld = o.ld; e.plane_stride = o.plane_stride;
      e.elem_bytes = o.elem_bytes;
      e.bytes = (uint64_t)(((int64_t)(o.planes - 1) * o.plane_stride + o.rows * o.ld) * o.elem_bytes);
      e.offset = off;
      off = align_up(off + e.bytes);
      ents.push_back(e);
    }
  }
  const int n = (int)ents.size();
  if (n_entries) *n_entries = n;
  if (bytes_needed) *bytes_needed = off;
  if (entries && max_entries >= n)
    for (int i = 0; i < n; ++i) entries[i] = ents[i];
  if (!trace_dev) return ok();
  if (trace_bytes < off) return fail(MLP_ERR_ARG, "trace buffer holds %zu bytes, the step writes %zu", trace_bytes, off);
  if (!entries || max_entries < n) return fail(MLP_ERR_ARG, "%d trace entries needed", n);
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* dst = (uint8_t*)trace_dev;
  int j = 0;
  for (size_t i = 0; i < recs.size(); ++i) {
    cudaError_t e = launch_rec(recs[i], s);
    if (e != cudaSuccess) return fail(MLP_ERR_CUDA, "launch of %s failed: %s", recs[i].name, cudaGetErrorString(e));
    for (int k = 0; k < recs[i].nouts; ++k, ++j)
      CUDA_TRY(cudaMemcpyAsync(dst + ents[j].offset, recs[i].outs[k].ptr, ents[j].bytes, cudaMemcpyDeviceToDevice, s));
  }
  CUDA_TRY(cudaStreamSynchronize(s));
  return ok();
}

static mlp_status copy_plane(mlp_t* m, int plane, float* host_out, const float* host_in, size_t n) {
  if (plane < MLP_PLANE_P || plane > MLP_PLANE_V) return fail(MLP_ERR_ARG, "bad plane %d", plane);
  if ((int64_t)n != m->lay.n_params) return fail(MLP_ERR_ARG, "n must be %lld", (long long)m->lay.n_params);
  const Layout& L = m->lay;
  float* base = m->plane(plane);
  size_t pos = 0;
  for (int l = 0; l < L.L; ++l) {
    const size_t nw = L.dims[l + 1] * L.dims[l], nb = L.dims[l + 1];
    if (host_out) {
      CUDA_TRY(cudaMemcpy(host_out + pos, base + L.woff[l], nw * 4, cudaMemcpyDeviceToHost));
      CUDA_TRY(cudaMemcpy(host_out + pos + nw, base + L.boff[l], nb * 4, cudaMemcpyDeviceToHost));
    } else {
      CUDA_TRY(cudaMemcpy(base + L.woff[l], host_in + pos, nw * 4, cudaMemcpyHostToDevice));
      CUDA_TRY(cudaMemcpy(base + L.boff[l], host_in + pos + nw, nb * 4, cudaMemcpyHostToDevice));
    }
    pos += nw + nb;
  }
  return MLP_OK;
}

mlp_status mlp_read_params(mlp_t* m, int plane, float* host_out, size_t n, int64_t* step_out) {
  if (!m || !host_out) return fail(MLP_ERR_ARG, "model or buffer is NULL");
  std::lock_guard<std::mutex> lk(m->mu);
  DevGuard g(m->device);
  CUDA_TRY(cudaDeviceSynchronize());
  mlp_status st = copy_plane(m, plane, host_out, nullptr, n);
  if (st != MLP_OK) return st;
  if (step_out) CUDA_TRY(cudaMemcpy(step_out, &m->ctl()->step, sizeof(int64_t), cudaMemcpyDeviceToHost));
  return ok();
}

mlp_status mlp_write_params(mlp_t* m, int plane, const float* host_in, size_t n, int64_t step) {
  if (!m || !host_in) return fail(MLP_ERR_ARG, "model or buffer is NULL");
  if (step < 0) return fail(MLP_ERR_ARG, "negative step");
  std::lock_guard<std::mutex> lk(m->mu);
  DevGuard g(m->device);
  CUDA_TRY(cudaDeviceSynchronize());
  mlp_status st = copy_plane(m, plane, nullptr, host_in, n);
  if (st != MLP_OK) return st;
  CUDA_TRY(cudaMemcpy(&m->ctl()->step, &step, sizeof(int64_t), cudaMemcpyHostToDevice));
  if (plane == MLP_PLANE_P) CUDA_TRY(refresh_w16(m));
  CUDA_TRY(cudaDeviceSynchronize());
  return ok();
}

static mlp_status status_from_bits(uint32_t bits) {
  if (bits & ERRBIT_LABEL_RANGE) return fail(MLP_ERR_LABEL_RANGE, "a label was outside [0, C)");
  if (bits & ERRBIT_NONFINITE) return fail(MLP_ERR_NONFINITE, "non-finite batch loss");
  if (bits & ERRBIT_TIMEOUT) return fail(MLP_ERR_TIMEOUT, "a bounded device wait gave up");
  if (bits) return fail(MLP_ERR_STATE, "device error bits 0x%x", bits);
  return ok();
}

mlp_status mlp_check_errors(mlp_t* m, void* stream) {
  if (!m) return fail(MLP_ERR_ARG, "model is NULL");
  std::lock_guard<std::mutex> lk(m->mu);
  DevGuard g(m->device);
  CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
  uint32_t bits = 0;
  CUDA_TRY(cudaMemcpy(&bits, &m->ctl()->err, 4, cudaMemcpyDeviceToHost));
  CUDA_TRY(cudaMemset(&m->ctl()->err, 0, 4));
  return status_from_bits(bits);
}

// ---------------------------------------------------------------------------
// C ABI: individual operations.
// ---------------------------------------------------------------------------
static mlp_status run_ops(LaunchRec* r, int n, void* stream) {
  for (int i = 0; i < n; ++i) {
    cudaError_t e = launch_rec(r[i], (cudaStream_t)stream);
    if (e != cudaSuccess) return fail(MLP_ERR_CUDA, "launch of %s failed: %s", r[i].name, cudaGetErrorString(e));
  }
  return ok();
}

static bool dtype_ok(int d) { return d == MLP_F32 || d == MLP_BF16; }
static bool gemm_dtype_ok(int d) { return d == MLP_F32 || d == MLP_BF16 || d == MLP_F32X3; }
static bool act_ok(int a) { return a >= MLP_ACT_NONE && a <= MLP_ACT_GELU_TANH; }

mlp_status mlp_op_linear_act(int dtype, int act, int64_t M, int64_t N, int64_t K, const void* X, int64_t ldx,
                             const void* W, int64_t ldw, const float* b, void* H, int64_t ldh, void* U, int64_t ldu,
                             uint32_t* err_dev, void* stream) {
  if (!gemm_dtype_ok(dtype)) return fail(MLP_ERR_DTYPE, "bad dtype");
  if (!act_ok(act)) return fail(MLP_ERR_ARG, "bad activation");
  if (!X || !W || !b || !H) return fail(MLP_ERR_ARG, "null pointer");
  if (ldx < K || ldw < K || ldh < N || (U && ldu < N)) return fail(MLP_ERR_SHAPE, "leading dimension too small");
  GemmOp op;
  op.dtype = dtype; op.kind = GEMM_FWD; op.act = act;
  op.a_plane = M * ldx; op.b_plane = N * ldw; op.out_plane = M * ldh;
  op.M = M; op.N = N; op.K = K;
  op.A = X; op.lda = ldx; op.a_kmajor = true;
  op.B = W; op.ldb = ldw; op.b_kmajor = true;
  op.bias = b; op.out = H; op.ldo = ldh; op.out_u = U; op.ldu = ldu;
  op.err = err_dev;
  LaunchRec r[2];
  char e_[512] = "";
  int n = gemm_plan(op, r, e_, sizeof(e_));
  if (n < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
  return run_ops(r, n, stream);
}

mlp_status mlp_op_dgrad(int dtype, int act, int64_t M, int64_t N, int64_t K, const void* dY, int64_t ldy,
                        const void* W, int64_t ldw, const void* S, int64_t lds, void* dX, int64_t ldx,
                        uint32_t* err_dev, void* stream) {
  if (!gemm_dtype_ok(dtype)) return fail(MLP_ERR_DTYPE, "bad dtype");
  if (!act_ok(act)) return fail(MLP_ERR_ARG, "bad activation");
  if (!dY || !W || !dX || (act != MLP_ACT_NONE && !S)) return fail(MLP_ERR_ARG, "null pointer");
  if (ldy < N || ldw < K || ldx < K || (S && lds < K)) return fail(MLP_ERR_SHAPE, "leading dimension too small");
  GemmOp op;
  op.dtype = dtype; op.kind = GEMM_DGRAD; op.act = act;
  op.a_plane = M * ldy; op.b_plane = N * ldw; op.out_plane = M * ldx;
  op.M = M; op.N = K; op.K = N;
  op.A = dY; op.lda = ldy; op.a_kmajor = true;
  op.B = W; op.ldb = ldw; op.b_kmajor = false;
  op.aux = S; op.ld_aux = lds;
  op.out = dX; op.ldo = ldx;
  op.err = err_dev;
  LaunchRec r[2];
  char e_[512] = "";
  int n = gemm_plan(op, r, e_, sizeof(e_));
  if (n < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
  return run_ops(r, n, stream);
}

size_t mlp_op_wgrad_workspace_bytes(int dtype, int64_t N, int64_t K, int64_t B) {
  if (!gemm_dtype_ok(dtype) || N < 1 || K < 1 || B < 1) return 0;
  int s = wgrad_splits(dtype, N, K, B);
  return wgrad_workspace_bytes(dtype, N, K, B, s);
}

mlp_status mlp_op_wgrad(int dtype, int64_t N, int64_t K, int64_t B, const void* dY, int64_t ldy, const void* X,
                        int64_t ldx, float* dW, int64_t lddw, float* db, void* workspace, size_t ws_bytes,
                        uint32_t* err_dev, void* stream) {
  if (!gemm_dtype_ok(dtype)) return fail(MLP_ERR_DTYPE, "bad dtype");
  if (!dY || !X || !dW) return fail(MLP_ERR_ARG, "null pointer");
  if (ldy < N || ldx < K || lddw < K) return fail(MLP_ERR_SHAPE, "leading dimension too small");
  GemmOp op;
  op.dtype = dtype; op.kind = GEMM_WGRAD;
  op.a_plane = B * ldy; op.b_plane = B * ldx;
  op.M = N; op.N = K; op.K = B;
  op.A = dY; op.lda = ldy; op.a_kmajor = false;
  op.B = X; op.ldb = ldx; op.b_kmajor = false;
  op.dW = dW; op.ld_dw = lddw; op.db = db;
  op.ws = (float*)workspace; op.ws_bytes = ws_bytes;
  op.err = err_dev;
  LaunchRec r[2];
  char e_[512] = "";
  int n = gemm_plan(op, r, e_, sizeof(e_));
  if (n < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
  return run_ops(r, n, stream);
}

mlp_status mlp_op_split3(int64_t rows, int64_t cols, const float* X, int64_t ldx, void* P, int64_t ldp,
                         void* stream) {
  if (!X || !P) return fail(MLP_ERR_ARG, "null pointer");
  if (ldx < cols || ldp < cols) return fail(MLP_ERR_SHAPE, "leading dimension too small");
  LaunchRec r;
  char e_[512] = "";
  if (split3_plan(rows, cols, X, ldx, P, ldp, rows * ldp, &r, e_, sizeof(e_)) < 0)
    return fail(MLP_ERR_SHAPE, "%s", e_);
  return run_ops(&r, 1, stream);
}

mlp_status mlp_op_softmax_ce(int dtype, int64_t B, int64_t C, const void* z, int64_t ldz, const int32_t* labels,
                             float grad_scale, void* dz, int64_t lddz, float* loss_rows, uint32_t* err_dev,
                             void* stream) {
  if (!dtype_ok(dtype)) return fail(MLP_ERR_DTYPE, "bad dtype");
  if (!z || !labels || !dz || !loss_rows) return fail(MLP_ERR_ARG, "null pointer");
  CeOp op;
  op.dtype = dtype; op.B = B; op.C = C; op.z = z; op.ldz = ldz; op.labels = labels;
  op.dz = dz; op.lddz = lddz; op.loss_rows = loss_rows; op.grad_scale = grad_scale; op.err = err_dev;
  LaunchRec r;
  char e_[512] = "";
  if (ce_plan(op, &r, e_, sizeof(e_)) < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
  return run_ops(&r, 1, stream);
}

mlp_status mlp_op_mse(int dtype, int64_t B, int64_t C, const void* z, int64_t ldz, const float* t, int64_t ldt,
                      float grad_scale, void* dz, int64_t lddz, float* loss_rows, void* stream) {
  if (!dtype_ok(dtype)) return fail(MLP_ERR_DTYPE, "bad dtype");
  if (!z || !t || !dz || !loss_rows) return fail(MLP_ERR_ARG, "null pointer");
  MseOp op;
  op.dtype = dtype; op.B = B; op.C = C; op.z = z; op.ldz = ldz; op.t = t; op.ldt = ldt;
  op.dz = dz; op.lddz = lddz; op.loss_rows = loss_rows; op.grad_scale = grad_scale;
  LaunchRec r;
  char e_[512] = "";
  if (mse_plan(op, &r, e_, sizeof(e_)) < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
  return run_ops(&r, 1, stream);
}

static size_t ce_ws_layout(int64_t B, int64_t C, int64_t K, size_t* off_zy, size_t* off_row, size_t* off_split) {
  auto al = [](size_t v) { return (v + 255) / 256 * 256; };
  size_t o = al((size_t)B * ce_groups(C) * 8);
  *off_zy = o;
  o = al(o + (size_t)B * 4);
  *off_row = o;
  o = al(o + (size_t)B * 8);
  *off_split = o;
  return o + wgrad_workspace_bytes(DT_BF16, C, K, B, wgrad_splits(DT_BF16, C, K, B));
}

size_t mlp_op_linear_ce_workspace_bytes(int64_t B, int64_t C, int64_t K) {
  if (B < 1 || C < 1 || K < 1) return 0;
  size_t a, b, c;
  return ce_ws_layout(B, C, K, &a, &b, &c);
}

mlp_status mlp_op_linear_ce(int64_t B, int64_t C, int64_t K, const void* h, int64_t ldh, const void* W,
                            const float* bias, const int32_t* labels, int act, const void* aux, int64_t ld_aux,
                            void* z, int64_t ldz, float* loss_rows, void* dX, int64_t ldx, float* dW, int64_t lddw,
                            float* db, void* ws, size_t ws_bytes, uint32_t* err_dev, void* stream) {
  if (!h || !W || !bias || !labels || !z || !loss_rows || !dX || !dW || !db || !ws)
    return fail(MLP_ERR_ARG, "null pointer");
  if (!act_ok(act) || (act != MLP_ACT_NONE && !aux)) return fail(MLP_ERR_ARG, "bad activation or aux");
  if (B < 1 || C <= 128 || K < 1 || ldh < K || ldz < C || ldx < K || lddw < K || (act != MLP_ACT_NONE && ld_aux < K))
    return fail(MLP_ERR_SHAPE, "bad shape (C must exceed 128)");
  size_t off_zy, off_row, off_split;
  const size_t need = ce_ws_layout(B, C, K, &off_zy, &off_row, &off_split);
  if (ws_bytes < need || (uintptr_t)ws % 16) return fail(MLP_ERR_ARG, "workspace too small or misaligned");
  uint8_t* w8 = (uint8_t*)ws;
  float2* stats = (float2*)w8;
  float* zy = (float*)(w8 + off_zy);
  float2* rowstat = (float2*)(w8 + off_row);
  LaunchRec r[8];
  int n = 0;
  char e_[512] = "";
  GemmOp f;
  f.dtype = DT_BF16; f.kind = GEMM_FWD; f.act = MLP_ACT_NONE;
  f.M = B; f.N = C; f.K = K;
  f.A = h; f.lda = ldh; f.a_kmajor = true;
  f.B = W; f.ldb = K; f.b_kmajor = true;
  f.bias = bias; f.out = z; f.ldo = ldz; f.err = err_dev;
  f.ce_stats = stats; f.ce_zy = zy; f.ce_labels = labels;
  int k = gemm_plan(f, r + n, e_, sizeof(e_));
  if (k < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
  n += k;
  CeCombineOp cc;
  cc.B = B; cc.C = C; cc.stats = stats; cc.zy = zy; cc.labels = labels; cc.rowstat = rowstat;
  cc.loss_rows = loss_rows; cc.err = err_dev;
  if (ce_combine_plan(cc, r + n, e_, sizeof(e_)) < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
  ++n;
  GemmOp d;
  d.dtype = DT_BF16; d.kind = GEMM_DGRAD; d.act = act;
  d.M = B; d.N = K; d.K = C;
  d.A = z; d.lda = ldz; d.a_kmajor = true;
  d.B = W; d.ldb = K; d.b_kmajor = false;
  d.aux = aux; d.ld_aux = ld_aux;
  d.out = dX; d.ldo = ldx; d.err = err_dev;
  d.ce_rowstat = rowstat; d.ce_labels = labels; d.ce_scale = (float)(1.0 / (double)B);
  k = gemm_plan(d, r + n, e_, sizeof(e_));
  if (k < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
  n += k;
  GemmOp g;
  g.dtype = DT_BF16; g.kind = GEMM_WGRAD;
  g.M = C; g.N = K; g.K = B;
  g.A = z; g.lda = ldz; g.a_kmajor = false;
  g.B = h; g.ldb = ldh; g.b_kmajor = false;
  g.dW = dW; g.ld_dw = lddw; g.db = db;
  g.ws = (float*)(w8 + off_split); g.ws_bytes = ws_bytes - off_split;
  g.err = err_dev;
  g.ce_rowstat = rowstat; g.ce_labels = labels; g.ce_scale = d.ce_scale;
  k = gemm_plan(g, r + n, e_, sizeof(e_));
  if (k < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
  n += k;
  return run_ops(r, n, stream);
}

mlp_status mlp_op_loss_mean(int64_t B, const float* loss_rows, float* loss, uint32_t* err_dev, void* stream) {
  if (!loss_rows || !loss) return fail(MLP_ERR_ARG, "null pointer");
  LossMeanOp op;
  op.B = B; op.loss_rows = loss_rows; op.loss = loss; op.err = err_dev;
  LaunchRec r;
  char e_[512] = "";
  if (loss_mean_plan(op, &r, e_, sizeof(e_)) < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
  return run_ops(&r, 1, stream);
}

mlp_status mlp_op_adamw(int64_t n, float* p, const float* g, float* m, float* v, void* w16, int64_t t, float lr,
                        float beta1, float beta2, float eps, float wd, void* stream) {
  if (!p || !g || !m || !v) return fail(MLP_ERR_ARG, "null pointer");
  if (t < 1) return fail(MLP_ERR_ARG, "t must be >= 1");
  AdamWOp op;
  op.n = n; op.p = p; op.g = const_cast<float*>(g); op.m = m; op.v = v; op.w16 = w16; op.t = t;
  op.lr = lr; op.beta1 = beta1; op.beta2 = beta2; op.eps = eps; op.wd = wd;
  LaunchRec r[2];
  char e_[512] = "";
  const int nr = adamw_plan(op, r, e_, sizeof(e_));
  if (nr < 0) return fail(MLP_ERR_ARG, "%s", e_);
  return run_ops(r, nr, stream);
}

static_assert(AdamWOp::kNormParts == MLP_OPTIM_WS_FLOATS, "norm workspace size of the C ABI");

mlp_status mlp_op_optim(int kind, int64_t n, float* p, float* g, float* m, float* v, void* w16, int64_t t, float lr,
                        float beta1, float beta2, float eps, float wd, float max_norm, float* ws_dev,
                        float* norm_dev, void* stream) {
  if (!p || !g || !m || !v) return fail(MLP_ERR_ARG, "null pointer");
  if (kind < MLP_OPTIM_ADAMW || kind > MLP_OPTIM_SGD) return fail(MLP_ERR_ARG, "unknown optimizer %d", kind);
  if (kind != MLP_OPTIM_SGD && t < 1) return fail(MLP_ERR_ARG, "t must be >= 1");
  if (max_norm > 0 && !ws_dev) return fail(MLP_ERR_ARG, "clipping needs ws_dev");
  AdamWOp op;
  op.kind = kind;
  op.n = n; op.p = p; op.g = g; op.m = m; op.v = v; op.w16 = w16; op.t = kind == MLP_OPTIM_SGD ? 1 : t;
  op.lr = lr; op.beta1 = beta1; op.beta2 = beta2; op.eps = eps; op.wd = wd;
  op.max_norm = max_norm; op.norm_ws = ws_dev; op.norm_out = norm_dev;
  LaunchRec r[2];
  char e_[512] = "";
  const int nr = adamw_plan(op, r, e_, sizeof(e_));
  if (nr < 0) return fail(MLP_ERR_ARG, "%s", e_);
  return run_ops(r, nr, stream);
}

mlp_status mlp_op_wait_timeout_check(uint64_t limit_ns, uint32_t* err_dev, void* stream) {
  if (!err_dev) return fail(MLP_ERR_ARG, "err_dev is NULL");
  if (limit_ns == 0 || limit_ns > 1000000000ull) return fail(MLP_ERR_ARG, "limit_ns must be in (0, 1 s]");
  LaunchRec r;
  wait_timeout_check_plan(err_dev, limit_ns, &r);
  return run_ops(&r, 1, stream);
}

mlp_status mlp_op_argmax(int dtype, int64_t B, int64_t C, const void* z, int64_t ldz, int32_t* out, void* stream) {
  if (!dtype_ok(dtype)) return fail(MLP_ERR_DTYPE, "bad dtype");
  if (!z || !out) return fail(MLP_ERR_ARG, "null pointer");
  if (ldz < C) return fail(MLP_ERR_SHAPE, "ldz < C");
  ArgmaxOp op;
  op.dtype = dtype; op.B = B; op.C = C; op.z = z; op.ldz = ldz; op.out = out;
  LaunchRec r;
  char e_[512] = "";
  if (argmax_plan(op, &r, e_, sizeof(e_)) < 0) return fail(MLP_ERR_SHAPE, "%s", e_);
  return run_ops(&r, 1, stream);
}

}  // extern "C"
