/*
 * mlp_ops.h -- the individual operations of the MLP training step, callable
 * on caller-owned device buffers.  They run the same kernels mlp_train_step
 * runs; they exist so that each step of the path can be checked and timed on
 * its own at full size.
 *
 * Common conventions: device pointers on the current CUDA device; dense
 * row-major layouts with explicit leading dimensions (`ld*`, in elements);
 * dtype MLP_F32 (float) or MLP_BF16 (bfloat16 bits); `stream` is a
 * cudaStream_t.  Every call validates its arguments and returns before
 * enqueuing anything when they are invalid; it returns once its kernels are
 * enqueued.  Device-side conditions (label range, wait timeouts) are OR-ed
 * into `err_dev` (a device uint32, nullable) with the bits
 *   1 = label outside [0, C), 2 = non-finite loss, 4 = bounded wait gave up.
 * For MLP_BF16 the GEMM operands are read by TMA: every operand base must be
 * 16-byte aligned and every leading dimension a multiple of 8 elements.
 * The GEMM entry points (linear_act, dgrad, wgrad) also take MLP_F32X3:
 * every matrix argument that is fp32 under MLP_F32 (X, W, H, dY, dX) is then
 * three bf16 planes [3][rows][ld] (mlp.h), produced by mlp_op_split3; the
 * bias, dW and db stay fp32; S is read from its first (hi) plane only, so
 * only ReLU / no activation are accepted; the TMA rules of MLP_BF16 apply.
 */
#ifndef MLP_OPS_H_
#define MLP_OPS_H_

#include <stddef.h>
#include <stdint.h>

#include "mlp.h"

#ifdef __cplusplus
extern "C" {
#endif

/* LinearAct forward (noeira.ai "Neural networks", "The design in one page":
 * MatMul+Bias+Activation as one kernel, bias and activation in the GEMM
 * epilogue):  u = X W^T + b,  H = act(u),  U = u (optional, nullable).
 *   X [M, K] (ldx), W [N, K] (ldw), b fp32 [N], H [M, N] (ldh), U [M, N] (ldu).
 * Accumulation is fp32; H and U are rounded to the dtype. */
mlp_status mlp_op_linear_act(int dtype, int act, int64_t M, int64_t N, int64_t K, const void* X, int64_t ldx,
                             const void* W, int64_t ldw, const float* b, void* H, int64_t ldh, void* U, int64_t ldu,
                             uint32_t* err_dev, void* stream);

/* dgrad with the activation VJP fused (noeira "The design in one page":
 * vjp per module):  dX = (dY W) * act'(S)
 *   dY [M, N] (ldy), W [N, K] (ldw), S [M, K] (lds) = what the forward of the
 *   layer below stored: h for ReLU (mask h > 0), u for GELU, unused for
 *   MLP_ACT_NONE (nullable); dX [M, K] (ldx). */
mlp_status mlp_op_dgrad(int dtype, int act, int64_t M, int64_t N, int64_t K, const void* dY, int64_t ldy,
                        const void* W, int64_t ldw, const void* S, int64_t lds, void* dX, int64_t ldx,
                        uint32_t* err_dev, void* stream);

/* The three bf16 planes of an fp32 matrix X [rows, cols] (ldx):
 * P [3][rows][ldp] with P[0] = bf16(X), P[1] = bf16(X - P[0]),
 * P[2] = bf16(X - P[0] - P[1]) (the MLP_F32X3 encoding, mlp.h). */
mlp_status mlp_op_split3(int64_t rows, int64_t cols, const float* X, int64_t ldx, void* P, int64_t ldp,
                         void* stream);

/* Workspace bytes mlp_op_wgrad needs for this shape (0 if none). */
size_t mlp_op_wgrad_workspace_bytes(int dtype, int64_t N, int64_t K, int64_t B);

/* wgrad with the bias gradient fused:  dW = dY^T X (fp32 [N, K], lddw),
 * db = sum over rows of dY (fp32 [N], nullable).
 *   dY [B, N] (ldy), X [B, K] (ldx).  The reduction over B may be split;
 *   partial sums go to `workspace` (device, ws_bytes >= the size above) and
 *   are added in a fixed order, so results are deterministic. */
mlp_status mlp_op_wgrad(int dtype, int64_t N, int64_t K, int64_t B, const void* dY, int64_t ldy, const void* X,
                        int64_t ldx, float* dW, int64_t lddw, float* db, void* workspace, size_t ws_bytes,
                        uint32_t* err_dev, void* stream);

/* mlp_op_wgrad without a workspace argument (the pages have no counterpart:
 * this is a convenience of this library).  Some callers cannot call
 * cudaMalloc: an application whose device memory belongs to another
 * allocator (a framework's caching pool, a fixed up-front reservation) has
 * no extra buffer to pass, and a latency-critical loop must not allocate,
 * since cudaMalloc/cudaFree can synchronise the device and fail under memory
 * pressure.  This entry point allocates nothing: the split-K partial sums go
 * to a built-in device array of 16 MiB, which every GPU that loads the
 * library holds until the process exits.
 *   Same arguments, layouts and results as mlp_op_wgrad, for every dtype it
 *   takes (MLP_F32, MLP_BF16, MLP_F32X3).  Returns MLP_ERR_SHAPE, before
 *   enqueuing anything, when the shape needs more than 16 MiB of scratch
 *   (mlp_op_wgrad_workspace_bytes tells how much).
 *   The array's device address is looked up (cudaGetSymbolAddress, with the
 *   device current) by the first call on a device, which should come before
 *   any stream capture; later calls look it up again unless their stream is
 *   capturing, so a cudaDeviceReset between calls leaves no stale address.
 *   Every call shares the one array per device: calls whose kernels overlap
 *   on the GPU (other streams, other threads) race on it and must be
 *   serialised by the caller.  Each call writes every scratch element it
 *   later reads, so nothing is carried over from a previous call. */
mlp_status mlp_op_wgrad_noalloc(int dtype, int64_t N, int64_t K, int64_t B, const void* dY, int64_t ldy,
                                const void* X, int64_t ldx, float* dW, int64_t lddw, float* db, uint32_t* err_dev,
                                void* stream);

/* Softmax cross-entropy, forward and backward in one pass over each row
 * (devpost "Orthon", "Selected Orthon vs. PyTorch results": one kernel reads
 * the logits once):  loss_rows[i] = logsumexp(z_i) - z_i[y_i] (fp32),
 * dz_i = (softmax(z_i) - onehot(y_i)) * grad_scale (dtype; grad_scale = 1/B
 * gives the gradient of the batch-mean loss).
 *   z [B, C] (ldz), labels int32 [B], dz [B, C] (lddz). */
mlp_status mlp_op_softmax_ce(int dtype, int64_t B, int64_t C, const void* z, int64_t ldz, const int32_t* labels,
                             float grad_scale, void* dz, int64_t lddz, float* loss_rows, uint32_t* err_dev,
                             void* stream);

/* Squared error of outputs z [B, C] (ldz, dtype) against fp32 targets t
 * [B, C] (ldt), the MSE loss (pypi "munet-nn", "Python training":
 * mse_loss):  loss_rows[i] = sum_j (z_ij - t_ij)^2 (fp32), dz_ij = (z_ij -
 * t_ij) * grad_scale (dtype; grad_scale = 2 / (B C) gives the gradient of
 * the mean over all elements, the loss being sum(loss_rows) / (B C)). */
mlp_status mlp_op_mse(int dtype, int64_t B, int64_t C, const void* z, int64_t ldz, const float* t, int64_t ldt,
                      float grad_scale, void* dz, int64_t lddz, float* loss_rows, void* stream);

/* A bf16 output layer fused with softmax cross-entropy, its VJPs included
 * (the softmax-CE-in-GEMM path of MLP_OPT_CE_GEMM): for h [B, K] (ldh, bf16),
 * W [C, K] (bf16, row pitch K), bias [C] (fp32) and labels int32 [B]:
 *   z = h W^T + bias, stored bf16 in z [B, C] (ldz);
 *   loss_rows[i] = logsumexp(z_i) - z_i[y_i] (fp32, from the stored logits);
 *   dX = (dz W) * act'(aux) [B, K] (ldx, bf16; act of the layer below: aux is
 *     its stored h for ReLU, u for GELU; MLP_ACT_NONE: aux unused), and
 *   dW = dz^T h (fp32 [C, K], lddw), db = sum_rows dz (fp32 [C]),
 * with dz = (softmax(z) - onehot(y)) / B formed on the fly from the stored
 * logits and never written.  C > 128; K and the pitches multiples of 8; ws
 * (device, 16-byte aligned) of mlp_op_linear_ce_workspace_bytes(B, C, K)
 * bytes.  Launches the forward GEMM, the statistics combine, the dgrad and
 * the wgrad (+ its split-K reduce).  A label outside [0, C) sets the error
 * bit in err_dev (its loss row is 0). */
size_t mlp_op_linear_ce_workspace_bytes(int64_t B, int64_t C, int64_t K);
mlp_status mlp_op_linear_ce(int64_t B, int64_t C, int64_t K, const void* h, int64_t ldh, const void* W,
                            const float* bias, const int32_t* labels, int act, const void* aux, int64_t ld_aux,
                            void* z, int64_t ldz, float* loss_rows, void* dX, int64_t ldx, float* dW, int64_t lddw,
                            float* db, void* ws, size_t ws_bytes, uint32_t* err_dev, void* stream);

/* loss = mean(loss_rows[0..B)) summed in a fixed order (device float). */
mlp_status mlp_op_loss_mean(int64_t B, const float* loss_rows, float* loss, uint32_t* err_dev, void* stream);

/* AdamW at step t >= 1 over flat fp32 planes p, g, m, v of n elements
 * (MuNet "What runs today": AdamW; noeira "The design in one page": moments
 * co-located per parameter):  m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 * p = p - lr (m/(1-b1^t) / (sqrt(v/(1-b2^t)) + eps) + wd p).  w16 (nullable)
 * receives bf16(p) after the update.  Planes 16-byte aligned, w16 8-byte. */
mlp_status mlp_op_adamw(int64_t n, float* p, const float* g, float* m, float* v, void* w16, int64_t t, float lr,
                        float beta1, float beta2, float eps, float wd, void* stream);

/* One update of rule `kind` (MLP_OPTIM_ADAMW / _ADAM / _SGD of mlp.h, same
 * formulas) over flat fp32 planes of n elements, with global-norm clipping
 * when max_norm > 0: g is scaled by min(1, max_norm / (||g||_2 + 1e-6))
 * before the update (g itself is not changed) and ||g|| goes to norm_dev
 * (device float, nullable).  ws_dev (device, 16-byte aligned, at least
 * MLP_OPTIM_WS_FLOATS floats) holds per-block partial sums of squares; it is
 * needed only when clipping.  t >= 1 for the Adam rules (bias correction);
 * SGD ignores t, beta2, eps and v.  w16 (nullable) receives bf16(p).
 * Clipping launches two kernels (norm, then update), otherwise one. */
enum { MLP_OPTIM_WS_FLOATS = 1216 };
mlp_status mlp_op_optim(int kind, int64_t n, float* p, float* g, float* m, float* v, void* w16, int64_t t, float lr,
                        float beta1, float beta2, float eps, float wd, float max_norm, float* ws_dev,
                        float* norm_dev, void* stream);

/* The error path of the device waits, exercised without a fault: one thread
 * waits, through the same bounded wait every tensor-core kernel uses for its
 * pipeline barriers, for an mbarrier phase that nothing completes; after
 * limit_ns (at most 1 s) it gives up, sets the timeout bit (1 << 2, the bit
 * behind MLP_ERR_TIMEOUT) in err_dev and the kernel returns normally, so the
 * context stays usable. */
mlp_status mlp_op_wait_timeout_check(uint64_t limit_ns, uint32_t* err_dev, void* stream);

/* Row argmax of z [B, C] (ldz) into int32 out [B]; lowest index on ties. */
mlp_status mlp_op_argmax(int dtype, int64_t B, int64_t C, const void* z, int64_t ldz, int32_t* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MLP_OPS_H_ */
