/*
 * mlp.h -- C ABI of a GB300-native training step for a fused-activation MLP.
 *
 * The step (one supervised update of an L-layer perceptron) is:
 *   forward   u_l = X_l W_l^T + b_l, h_l = act(u_l) for hidden layers, logits
 *             z = h_{L-1} W_L^T + b_L (Linear layers as in pypi "munet-nn",
 *             "Python training"; the MatMul+Bias+Activation fusion of
 *             noeira.ai "Neural networks", "The design in one page");
 *   loss      mean over the batch of softmax cross-entropy with integer
 *             labels (devpost "Orthon", "Core capabilities" and "Selected
 *             Orthon vs. PyTorch results"), or mean squared error against
 *             real targets (mlp_set_loss);
 *   backward  explicit vector-Jacobian products (noeira "The design in one
 *             page": forward and vjp per module, no tape): dW_l = dY_l^T X_l,
 *             db_l = column sums of dY_l, dY_{l-1} = (dY_l W_l) * act';
 *   update    AdamW with moments stored beside each parameter (noeira "The
 *             design in one page": a Param is four tensors; MuNet "What runs
 *             today": AdamW), decoupled decay, bias-corrected moments.
 * The whole step is recorded once as a CUDA graph and replayed (noeira "What
 * is in it": optional CUDA-graph capture; MuNet "What runs today": recorded
 * command-buffer replay).
 *
 * Conventions
 *   - All device pointers are plain CUDA device addresses on the model's
 *     device; host pointers are ordinary process memory.  `stream` is a
 *     cudaStream_t (NULL = the legacy default stream).
 *   - Tensors are dense row-major.  x is [batch, dims[0]] in the model dtype
 *     (float for MLP_F32, bfloat16 bits for MLP_BF16); the training targets
 *     y are int32 labels [batch] (softmax CE, the default loss) or float
 *     targets [batch, C] (MLP_LOSS_MSE, see mlp_set_loss); logits are
 *     [batch, C] in the model dtype.
 *   - Parameters use a flat order: for l = 1..L, W_l [dims[l], dims[l-1]]
 *     row-major then b_l [dims[l]].  mlp_read_params / mlp_write_params move
 *     them densely packed in that order.
 *   - Memory: the caller allocates ONE device buffer of mlp_arena_bytes()
 *     bytes (e.g. with torch) and hands it to mlp_create; the library lays
 *     out parameters, gradients, moments, the bf16 weight copy, activations,
 *     workspace and a control block inside it and allocates no device memory
 *     of its own.  The arena must outlive the model.
 *   - One batch size per model (fixed at create; MuNet "Python training":
 *     one specialization per compiled object).  Calls on one model are
 *     serialised by a mutex; at most one step is in flight per model.
 *   - Errors: argument / shape errors return before anything is enqueued;
 *     CUDA errors return MLP_ERR_CUDA; conditions found on the device (a
 *     label outside [0, C), a non-finite loss, a device wait that gave up)
 *     are latched in the control block and returned by the next
 *     mlp_check_errors.  mlp_last_error() gives a message for the calling
 *     thread.  There is no CPU fallback: without a usable GPU every compute
 *     call fails.
 */
#ifndef MLP_H_
#define MLP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mlp mlp_t;

typedef enum {
  MLP_OK = 0,
  MLP_ERR_ARG = 1,          /* bad argument (null pointer, bad enum, ...) */
  MLP_ERR_SHAPE = 2,        /* unsupported or mismatched shape */
  MLP_ERR_DTYPE = 3,        /* unsupported dtype */
  MLP_ERR_CUDA = 4,         /* a CUDA call failed */
  MLP_ERR_LABEL_RANGE = 5,  /* device: a label outside [0, C) */
  MLP_ERR_NONFINITE = 6,    /* device: non-finite batch loss */
  MLP_ERR_STATE = 7,        /* call not valid in the model's state */
  MLP_ERR_TIMEOUT = 8       /* device: a bounded wait inside a kernel gave up */
} mlp_status;

enum { MLP_ACT_NONE = 0, MLP_ACT_RELU = 1, MLP_ACT_GELU_TANH = 2 };
/* MLP_F32: fp32 everywhere (no TF32).  The GEMMs of the training step run
 *   on the tensor cores with each fp32 operand held as three bf16 planes
 *   (see MLP_OPT_F32_TENSOR_CORES), or on the FFMA pipes.
 * MLP_BF16: bf16 x / weights copy / activations / logits / gradients of
 * activations, fp32 accumulation, fp32 bias, fp32 master weights, gradients
 * and Adam moments (MuNet "Configuration", precision="mixed"; Orthon
 * "Core capabilities", FP32 master weights). */
enum { MLP_F32 = 0, MLP_BF16 = 1 };
/* Operand encoding of the op-level GEMM entry points only (mlp_ops.h): fp32
 * values as three bf16 planes hi, mid, lo stored one after another, each
 * plane [rows, ld]:  hi = bf16(x), mid = bf16(x - hi), lo = bf16(x - hi -
 * mid), so hi + mid + lo = x exactly for fp32 x in the normal range. */
enum { MLP_F32X3 = 2 };
/* Parameter planes, all indexed by the same flat parameter order. */
enum { MLP_PLANE_P = 0, MLP_PLANE_G = 1, MLP_PLANE_M = 2, MLP_PLANE_V = 3 };

/* Bytes of device memory a model with this shape needs.  dims has n_dims
 * entries [in, h1, ..., C] (n_dims >= 2); acts has n_dims-2 entries (one per
 * hidden layer) or is NULL to use `act` on every hidden layer.  Returns 0 on
 * an invalid shape (see mlp_last_error). */
size_t mlp_arena_bytes(const int64_t* dims, int n_dims, const int* acts, int act, int dtype, int64_t batch);

/* Create a model in the caller's arena on `device`.  Weights are drawn
 * Kaiming-normal (std = sqrt(2 / fan_in), noeira "A complete example":
 * make[Kaiming]) from a host generator seeded by `seed`; biases, gradients
 * and moments are zero; the step counter is 0.  For MLP_BF16 every input and
 * hidden width must be a multiple of 8 (16-byte rows for TMA).  On success
 * *out owns no memory except host bookkeeping. */
mlp_status mlp_create(const int64_t* dims, int n_dims, const int* acts, int act, int dtype, uint64_t seed,
                      int64_t batch, void* arena_dev, size_t arena_bytes, int device, mlp_t** out);

/* Forward only: logits_dev ([batch, C], model dtype; nullable) and
 * argmax_dev (int32 [batch], lowest index among equal maxima; nullable). */
mlp_status mlp_forward(mlp_t* model, const void* x_dev, void* logits_dev, int32_t* argmax_dev, void* stream);

/* One training step on (x_dev, y_dev): forward, the loss (softmax-CE of
 * int32 labels, or MSE of float targets), backward, AdamW(lr, beta1, beta2,
 * eps, wd) (or the rule of mlp_set_optimizer) at step t = (step counter + 1).
 * The loss (batch mean; element mean for MSE) is written to loss_dev (device
 * float; nullable).  Nothing is read back; the call returns once the work is
 * enqueued on `stream`. */
mlp_status mlp_train_step(mlp_t* model, const void* x_dev, const void* y_dev, float lr, float beta1,
                          float beta2, float eps, float wd, float* loss_dev, void* stream);

/* One training step on a batch in HOST memory (page-locked, so the copies are
 * asynchronous): x_host [batch, dims[0]] in the model dtype, y_host the
 * labels or MSE targets (MSE targets from host memory need batch * C * 4 <=
 * 64 MiB, else MLP_ERR_SHAPE).  The library copies them on its own copy
 * stream into one of
 * two device input slots in the arena, so the copies for the next call
 * overlap the kernels of this one; the step waits for its own copies.  The
 * host buffers must stay valid and unchanged until their copy has completed
 * (at the latest when the step completes).  loss_host (nullable) receives
 * the step's loss when the step completes: page-locked memory the device can
 * address is written by the step's last kernel directly, other memory by a
 * copy after the step.  Returns once the copies and the step are enqueued on
 * `stream`. */
mlp_status mlp_train_step_host(mlp_t* model, const void* x_host, const void* y_host, float lr, float beta1,
                               float beta2, float eps, float wd, float* loss_host, void* stream);

/* n_steps consecutive training steps enqueued as ONE CUDA-graph launch;
 * step i reads x_devs[i] / y_devs[i] (host arrays of device pointers)
 * and writes its loss to losses_dev[i] (nullable).  The graph is built on
 * the first call for a given n_steps and re-pointed on later calls. */
mlp_status mlp_train_steps(mlp_t* model, int n_steps, const void* const* x_devs, const void* const* y_devs,
                           float lr, float beta1, float beta2, float eps, float wd, float* losses_dev,
                           void* stream);

/* Use a CUDA graph for mlp_train_step / mlp_train_steps (1, the default) or
 * launch the kernels one by one (0). */
mlp_status mlp_set_graph_mode(mlp_t* model, int enable);

/* Step options.
 *   MLP_OPT_GRAPH      (default 1): same as mlp_set_graph_mode.
 *   MLP_OPT_FUSE_HEAD  (default 1): where the output layer is small (at most
 *     16 classes, at most 256 inputs, and a hidden layer below it), run it
 *     as one kernel together with softmax-CE, its dgrad and wgrad and the
 *     loss mean (the single logits read of devpost "Orthon", "Selected
 *     Orthon vs. PyTorch results", extended to the whole layer); 0 keeps the
 *     separate GEMM / CE / loss-mean kernels.  Results agree within
 *     rounding; the arithmetic and rounding points are the same.
 * Returns MLP_ERR_ARG for an unknown option. */
/*   MLP_OPT_F32_TENSOR_CORES (default 1; MLP_F32 models): run the training
 *     step's GEMMs on the tensor cores with fp32 operands as three bf16
 *     planes (MLP_F32X3): the six plane products above 2^-24 relative
 *     (hi*hi, mid*hi, hi*mid, lo*hi, mid*mid, hi*lo) are accumulated in
 *     fp32, so each product carries fp32-level error and no TF32 rounding.
 *     Used where the model allows it: ReLU / no activation, the fused output
 *     layer (MLP_OPT_FUSE_HEAD on and supported), and input / hidden widths
 *     below the output layer that are multiples of 8.  Otherwise, or with 0,
 *     the GEMMs run on the FFMA pipes.  mlp_forward follows the same
 *     choice for the hidden layers (the small output layer takes the joined
 *     fp32 activation on the FFMA pipes). */
/*   MLP_OPT_PDL (default 1): in the step's CUDA graph, let each kernel be
 *     scheduled as soon as every block of the kernel before it has started
 *     (programmatic dependent launch); it runs its prologue (barriers, tensor
 *     memory) and then waits for that kernel to complete before touching
 *     global memory.  0 chains the kernels with full dependencies.  Results
 *     are identical either way. */
/*   MLP_OPT_CE_GEMM (default 0; MLP_BF16 models with at least 1024 classes):
 *     softmax-CE inside the output layer's GEMMs.  The forward GEMM's
 *     epilogue leaves each row's (max, sum of exponentials) over every
 *     128-column group of the stored logits and the label's logit; a row
 *     kernel combines them into the row's (max, 1 / sum) and loss; the
 *     layer's dgrad and wgrad read the logits and form dz = (softmax -
 *     onehot) / B in shared memory on the way into the tensor cores, so dz
 *     is never stored (the single logits read of devpost "Orthon", "Selected
 *     Orthon vs. PyTorch results", taken into the GEMMs).  0 runs the
 *     separate softmax-CE pass (the default: on GB300 the in-GEMM dz costs
 *     more than the pass, since every logit feeds several output tiles of
 *     the dgrad and of the wgrad and its exponential is recomputed for each).
 *     Same rounding points either way (logits and dz rounded to bf16); the
 *     sums differ in order only. */
/*   MLP_OPT_RELU_BITS (default 1; MLP_BF16 models): the forward GEMM of a
 *     ReLU layer also writes its mask (stored h > 0) as one bit per element,
 *     and the dgrad below reads the bits instead of the stored activation
 *     (16x fewer bytes).  0 reads the stored activation.  Results are
 *     identical either way. */
/*   MLP_OPT_HEAD_IN_GEMM (default 1; MLP_F32 models on the tensor cores
 *     with the fused output layer): fold that output layer (10 classes, 128
 *     inputs) into the epilogue of the forward GEMM below it, where each
 *     row's fp32 h is at hand (noeira.ai "Neural networks", "The design in
 *     one page": the epilogue as the place for fused work): logits, softmax
 *     CE, dY of the hidden layer and per-CTA partials of the output layer's
 *     weight / bias gradients and loss, without storing h.  Applies where
 *     that forward runs on CTA pairs (at most 76 row tiles of 128 and a
 *     reduction of at least 192); 0, or otherwise, keeps the separate fused
 *     output-layer kernel.  Same arithmetic in fp32; the sums differ in
 *     order only. */
/*   MLP_OPT_GEMM_2SM (default -1; MLP_BF16 models): forward, dgrad and
 *     weight-gradient GEMMs with at least 256 rows and columns on CTA pairs
 *     that share 256 x 256 output tiles through 2-SM tensor-core MMAs (each
 *     SM loads half of A's and half of B's tile; a third fewer operand bytes
 *     per FLOP than one SM on a 128 x 256 tile).  -1: forward and dgrad
 *     where the pair tiles fill the device at least once and K is at least
 *     16 stages of 64 rows, weight gradients where each K split is at least
 *     16 stages; 1: wherever the shape allows; 0: never.  The same MMA
 *     arithmetic and the same bias-gradient sums either way (results are
 *     bit for bit those of the one-SM kernels). */
enum { MLP_OPT_GRAPH = 0, MLP_OPT_FUSE_HEAD = 1, MLP_OPT_F32_TENSOR_CORES = 2, MLP_OPT_PDL = 3, MLP_OPT_CE_GEMM = 4,
       MLP_OPT_RELU_BITS = 5, MLP_OPT_HEAD_IN_GEMM = 6, MLP_OPT_GEMM_2SM = 7 };
mlp_status mlp_set_option(mlp_t* model, int option, int64_t value);

/* The update rule of the training step (default MLP_OPTIM_ADAMW) and global
 * gradient-norm clipping (MuNet "What runs today": SGD, AdamW, gradient
 * clipping; noeira "What is in it": SGD, Adam, AdamW, gradient clipping).
 * The hyper-parameters of mlp_train_step* keep their places:
 *   MLP_OPTIM_ADAMW  the AdamW step described at the top.
 *   MLP_OPTIM_ADAM   Adam with the decay as L2 in the gradient: g' = g + wd p,
 *                    the AdamW moments of g', p -= lr m_hat / (sqrt(v_hat) +
 *                    eps).
 *   MLP_OPTIM_SGD    SGD with heavy-ball momentum beta1 and L2 wd: buf =
 *                    beta1 buf + (g + wd p), p -= lr buf (no dampening; buf
 *                    is plane M, zero after create; beta2, eps and plane V
 *                    are not used).
 * max_grad_norm > 0 scales the whole gradient by min(1, max_grad_norm /
 * (||g||_2 + 1e-6)) before the update, ||g|| over every gradient element;
 * the G plane keeps the unscaled gradient and mlp_read_grad_norm returns
 * ||g|| of the last step.  0 turns clipping off.  The moments are not reset:
 * switching rules mid-run carries planes M and V over as they are.  Returns
 * MLP_ERR_ARG for an unknown kind or a negative or non-finite threshold. */
enum { MLP_OPTIM_ADAMW = 0, MLP_OPTIM_ADAM = 1, MLP_OPTIM_SGD = 2 };
mlp_status mlp_set_optimizer(mlp_t* model, int kind, float max_grad_norm);

/* The loss of the training step (default MLP_LOSS_CE):
 *   MLP_LOSS_CE   softmax cross-entropy of int32 labels [batch], mean over
 *                 the batch (the step described at the top).
 *   MLP_LOSS_MSE  mean squared error against float targets [batch, C], mean
 *                 over all batch * C elements (the PyTorch mse_loss
 *                 default): dz = 2 (z - t) / (batch C) (MuNet "Python
 *                 training": the example step trains with mse_loss; "Training
 *                 swarm": the loss is MSE).  The step takes the same kernels
 *                 as with CE (the fused output layer where MLP_OPT_FUSE_HEAD
 *                 applies, the fp32 tensor-core planes), the loss part
 *                 replaced.
 * The targets are passed where the step entry points take y. */
enum { MLP_LOSS_CE = 0, MLP_LOSS_MSE = 1 };
mlp_status mlp_set_loss(mlp_t* model, int loss);

/* ||g||_2 computed by the last training step that clipped (0 before any);
 * synchronises the model's device. */
mlp_status mlp_read_grad_norm(mlp_t* model, float* out);

/* Number of parameters (flat, densely packed) and of Linear layers. */
int64_t mlp_num_params(const mlp_t* model);
int mlp_num_layers(const mlp_t* model);

/* Synchronous copies of a parameter plane to / from host memory (n must be
 * mlp_num_params).  read also returns the step counter (nullable);
 * write sets it.  Writing plane P of an MLP_BF16 model refreshes the bf16
 * weight copy.  Both synchronise the model's device. */
mlp_status mlp_read_params(mlp_t* model, int plane, float* host_out, size_t n, int64_t* step_out);
mlp_status mlp_write_params(mlp_t* model, int plane, const float* host_in, size_t n, int64_t step);

/* Synchronise `stream`, read and clear the device error word, and return
 * the first latched condition (MLP_OK if none). */
mlp_status mlp_check_errors(mlp_t* model, void* stream);

/* Number of kernels one training step launches (graph nodes per step). */
int mlp_kernels_per_step(const mlp_t* model);

/* One training step (same arguments and effect as mlp_train_step) with every
 * kernel launched on its own and bracketed by CUDA events on `stream`
 * (MuNet "Configuration": profile=True serialises kernels and records
 * per-kernel GPU timestamps).  Writes the device time of kernel i in ms to
 * ms_out[i] and its name (a static string) to names_out[i] (nullable) for
 * i < min(*n_out, max_kernels); *n_out = kernels in the step.  Synchronises
 * the stream before returning. */
mlp_status mlp_profile_step(mlp_t* model, const void* x_dev, const void* y_dev, float lr, float beta1,
                            float beta2, float eps, float wd, float* loss_dev, void* stream, float* ms_out,
                            const char** names_out, int max_kernels, int* n_out);

/* Data-parallel training (MuNet, pypi "munet-nn", "Reliability,
 * observability and scaling": mu.DataParallel splits each batch on dim 0 and
 * averages the gradients; netcl.online "Architecture: Distributed &
 * Multi-Device Execution", data_parallel_step: shard the batch, synchronise
 * the gradients, update; noeira.ai "Neural networks", "Distributed
 * training": DDP).  A step is split at its one exchange point:
 *   1. mlp_grad_step on this rank's rows of a global batch of global_batch
 *      rows (the model's batch is the shard's row count; shards may differ
 *      by rank): forward and backward; G receives the shard's gradient of
 *      the GLOBAL mean loss (dz scaled by 1 / global_batch), so the sum of G
 *      over ranks is the gradient of the whole batch; *loss_dev (nullable)
 *      receives the shard's share, sum of its row losses / global_batch
 *      (MSE: / (global_batch C)), so those sum to the batch loss.  Advances
 *      the step counter.  global_batch < the model's batch: MLP_ERR_ARG.
 *   2. the caller sums G over the ranks in place (an NCCL all-reduce on the
 *      buffer mlp_grad_buffer names, on this stream or ordered after it).
 *   3. mlp_apply_update: the update rule of mlp_set_optimizer (clipping
 *      included) over G, at the step counter of step 1.  Exactly one update
 *      per gradient step; every rank then holds the same parameters.
 * With one rank (global_batch = the model's batch) 1 + 3 is mlp_train_step,
 * bit for bit.  Both are CUDA-graph replays like mlp_train_step. */
mlp_status mlp_grad_step(mlp_t* model, const void* x_dev, const void* y_dev, int64_t global_batch, float* loss_dev,
                         void* stream);
mlp_status mlp_apply_update(mlp_t* model, float lr, float beta1, float beta2, float eps, float wd, void* stream);
/* The gradient plane G: device address and length in floats (the flat
 * parameter layout with its padding, every tensor 64-element aligned; the
 * padding holds zeros and sums to zero).  Valid for the model's lifetime. */
mlp_status mlp_grad_buffer(mlp_t* model, float** g_dev, int64_t* n_floats);

/* mlp_forward with every kernel launched on its own and bracketed by CUDA
 * events, as mlp_profile_step does for a training step (MuNet
 * "Configuration": profile=True): device ms and name of kernel i to
 * ms_out[i] / names_out[i] (nullable) for i < min(*n_out, max_kernels).
 * Same arguments and results as mlp_forward.  Synchronises the stream. */
mlp_status mlp_profile_forward(mlp_t* model, const void* x_dev, void* logits_dev, int32_t* argmax_dev, void* stream,
                               float* ms_out, const char** names_out, int max_kernels, int* n_out);

/* Traced step: one training step (same arguments and effect as
 * mlp_train_step) whose kernels run one after another on `stream`, each
 * followed by device-to-device copies of the tensors it wrote into the
 * caller's trace buffer, so that every intermediate result of the step can be
 * read back (noeira.ai "Neural networks", "The design in one page": forward
 * and backward are explicit, every layer's output and vector-Jacobian
 * product is a tensor of its own; MuNet "Configuration": profile=True runs
 * the kernels one by one).  The kernels, their launch configurations and
 * their buffers are those of mlp_train_step; only their order is serial.
 *   trace_dev (device, caller-owned, trace_bytes long) receives the tensors
 *   back to back, each 256-byte aligned, exactly as stored (row pitch,
 *   padding columns and planes included).  entries[i] (host,
 *   max_entries long, nullable) describes tensor i; *n_entries (nullable)
 *   and *bytes_needed (nullable) receive the count and the trace size.
 *   trace_dev NULL: nothing runs; only the count and the size are returned.
 *   Tensors kept only inside a fused kernel (the fused output layer's logits
 *   and dz, softmax-CE inside the GEMMs) have no entry.
 *   Errors: MLP_ERR_ARG for a trace buffer smaller than *bytes_needed or
 *   fewer entries than tensors (before anything runs); the rest as
 *   mlp_train_step.  Synchronises the stream before returning. */
enum {
  MLP_TRACE_H = 0,          /* hidden activation h_l = act(u_l), the input of layer l + 1 */
  MLP_TRACE_U = 1,          /* GELU pre-activation u_l as stored for the dgrad */
  MLP_TRACE_Z = 2,          /* logits z (layer L - 1) */
  MLP_TRACE_DZ = 3,         /* loss gradient dz = dY_{L-1} */
  MLP_TRACE_LOSS_ROWS = 4,  /* per-row loss, fp32 [B] */
  MLP_TRACE_DY = 5          /* dY_l, gradient w.r.t. u_l, written by the dgrad of layer l + 1 */
};
typedef struct {
  int32_t kind;            /* MLP_TRACE_* */
  int32_t layer;           /* 0-based layer l */
  int32_t launch;          /* index of the kernel that wrote it (mlp_profile_step order) */
  int32_t planes;          /* 1, or 3: an fp32 tensor as three bf16 planes */
  int64_t rows, cols, ld;  /* [rows, cols], row pitch ld elements */
  int64_t plane_stride;    /* elements from one plane to the next */
  int32_t elem_bytes;      /* bytes of one element of one plane: 2 (bf16) or 4 (fp32) */
  int32_t reserved;
  uint64_t offset;         /* byte offset of the tensor in trace_dev */
  uint64_t bytes;          /* bytes copied */
} mlp_trace_entry;
mlp_status mlp_trace_step(mlp_t* model, const void* x_dev, const void* y_dev, float lr, float beta1, float beta2,
                          float eps, float wd, float* loss_dev, void* trace_dev, size_t trace_bytes,
                          mlp_trace_entry* entries, int max_entries, int* n_entries, size_t* bytes_needed,
                          void* stream);

/* Message for the last failed call on this thread ("" if none). */
const char* mlp_last_error(void);

/* Destroy the model (the arena is the caller's and is not freed). */
void mlp_destroy(mlp_t* model);

#ifdef __cplusplus
}
#endif
#endif /* MLP_H_ */
