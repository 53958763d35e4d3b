// bf16 GEMMs of the training step on the sm_103a tensor cores: tcgen05.mma
// with the fp32 accumulator in tensor memory (TMEM), operands staged in
// shared memory by TMA (cp.async.bulk.tensor, 128-byte swizzle) through an
// mbarrier ring, and the step's epilogue fused after the TMEM read-back:
//   forward : h = act(acc + b) (and u = acc + b for GELU), bf16 out
//             (noeira.ai "Neural networks", "The design in one page":
//             MatMul+Bias+Activation in one kernel, bias and activation in
//             the GEMM epilogue);
//   dgrad   : dY_prev = acc * act'(stored h or u), bf16 out;
//   wgrad   : dW = acc in fp32, plus db = row sums of the A tile (dY^T) read
//             from shared memory by the otherwise idle epilogue warps.
// Mixed precision as in MuNet (pypi "munet-nn", "Configuration",
// precision="mixed"): rounded low-precision inputs, fp32 accumulation.
//
// One 128 x BN output tile per CTA; 6 warps: warp 0 issues TMA, warp 1 owns
// TMEM and issues the MMAs (one elected lane), warps 2..5 run the epilogue
// (warp w reads TMEM lanes 32*(w%4) .. +31).  Every mbarrier wait is bounded
// by a wall-clock limit; on expiry the kernel latches ERRBIT_TIMEOUT in the
// error word, drains its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <stdio.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "ops.h"

namespace mlpk {

int split_reduce_plan(const float* ws, int splits, int64_t M, int64_t N, float* dW, int64_t ld_dw,
                      float* db, LaunchRec* rec);
int simt_gemm_splits(int64_t M, int64_t N, int64_t K);

namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;                       // 64 bf16 = 128 bytes = one swizzle row
constexpr int A_STAGE_BYTES = BM * BK * 2;   // 16 KB
constexpr int NUM_THREADS = 192;
constexpr uint64_t kWaitLimitNs = 500000000ull;   // 0.5 s (a legitimate wait is microseconds)

template <int BN> struct Cfg {
  static constexpr int B_STAGE_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
  static constexpr int STAGES = BN >= 256 ? 4 : BN >= 128 ? 6 : 8;
  static constexpr int TMEM_COLS = BN <= 32 ? 32 : BN;   // power of two >= 32
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align slack*/ + 256 /*barriers*/;
};

struct Params {
  CUtensorMap tmA;
  CUtensorMap tmB;
  int M, N, K;
  int kb_per_split;     // k-blocks per blockIdx.z
  int num_kb;           // total k-blocks
  int a_mn, b_mn;       // 1: operand is MN-major in memory
  int kind, act;
  uint32_t idesc;
  const float* bias;
  __nv_bfloat16* out; int64_t ldo;
  __nv_bfloat16* out_u; int64_t ldu;
  const __nv_bfloat16* aux; int64_t ld_aux;
  float* dW; int64_t ld_dw;
  float* db;
  float* ws;            // split-K partials (splits > 1)
  uint32_t* err;
};

// ---------------------------------------------------------------------------
// PTX wrappers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: true when the phase completed, false after limit_ns (the
// error word is then marked).
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, uint32_t* err, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer() - t0 > limit_ns) {
      if (err) atomicOr(err, ERRBIT_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* err) {
  return mbar_wait_for(bar, parity, err, kWaitLimitNs);
}

// The error path of every device wait, exercised on purpose: one thread
// waits, through the same bounded wait, for the phase of an mbarrier that
// nothing arrives on; it gives up after limit_ns, marks the error word and
// the kernel returns normally.
// (One parameter block, like every kernel here: launches pass a single
// argument pointer.)
struct WaitCheckParams { uint32_t* err; uint64_t limit_ns; };
__global__ void wait_timeout_check_kernel(const __grid_constant__ WaitCheckParams q) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  mbar_wait_for(b, 0u, q.err, q.limit_ns);
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"((uint64_t)tm), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)tm) : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// 32 lanes x 32 bits, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format:
// start>>4 in [0,14), LBO>>4 in [16,30), SBO>>4 in [32,46), version 1 at
// [46,48), layout type 2 = SWIZZLE_128B at [61,64)).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int BN>
__global__ void __launch_bounds__(NUM_THREADS, 1) tc_gemm_kernel(const __grid_constant__ Params p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t a_base = base;
  const uint32_t b_base = base + C::STAGES * A_STAGE_BYTES;
  const uint32_t bar_base = b_base + C::STAGES * C::B_STAGE_BYTES;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (C::STAGES + s); };
  const uint32_t acc_bar = bar_base + 8u * (2 * C::STAGES);
  const uint32_t tmem_slot = acc_bar + 8u;
  volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int kb0 = blockIdx.z * p.kb_per_split;
  const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
  const int nkb = max(kb1 - kb0, 0);
  const bool do_db = p.kind == GEMM_WGRAD && blockIdx.x == 0 && p.db != nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), do_db ? 5 : 1);
    }
    mbar_init(acc_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot_ptr;
  pdl_enter();   // shared memory and TMEM are set up: now wait for the inputs

  const uint32_t b_bytes = C::B_STAGE_BYTES;
  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&p.tmA);
      prefetch_tmap(&p.tmB);
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < nkb && ok; ++i) {
        const int s = i % C::STAGES;
        const uint32_t ph = (uint32_t)(i / C::STAGES) & 1u;
        if (!mbar_wait(empty_bar(s), ph ^ 1u, p.err)) { ok = false; break; }
        mbar_expect_tx(full_bar(s), A_STAGE_BYTES + b_bytes);
        const int k0 = (kb0 + i) * BK;
        const uint32_t sa = a_base + s * A_STAGE_BYTES;
        const uint32_t sb = b_base + s * C::B_STAGE_BYTES;
        if (!p.a_mn) {
          tma_load_2d(sa, &p.tmA, k0, m0, full_bar(s));
        } else {
          tma_load_2d(sa, &p.tmA, m0, k0, full_bar(s));
          tma_load_2d(sa + 8192, &p.tmA, m0 + 64, k0, full_bar(s));
        }
        if (!p.b_mn) {
          tma_load_2d(sb, &p.tmB, k0, n0, full_bar(s));
        } else {
#pragma unroll
          for (int c = 0; c < BN / 64; ++c) tma_load_2d(sb + 8192 * c, &p.tmB, n0 + 64 * c, k0, full_bar(s));
        }
        ++issued;
      }
      // Drain: every issued copy must land before the CTA may exit.
      for (int i = max(0, issued - C::STAGES); i < issued; ++i)
        mbar_wait(full_bar(i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u, p.err);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      // K advance per 16-deep MMA: K-major -> 32 bytes inside the swizzle
      // row; MN-major -> 16 rows of 128 bytes.
      const uint32_t a_kstep = p.a_mn ? 2048u : 32u;
      const uint32_t b_kstep = p.b_mn ? 2048u : 32u;
      const uint32_t a_lbo = p.a_mn ? 8192u : 16u, b_lbo = p.b_mn ? 8192u : 16u;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % C::STAGES;
        const uint32_t ph = (uint32_t)(i / C::STAGES) & 1u;
        if (!mbar_wait(full_bar(s), ph, p.err)) break;
        tc_fence_after();
        const uint32_t sa = a_base + s * A_STAGE_BYTES;
        const uint32_t sb = b_base + s * C::B_STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          uint64_t ad = sdesc(sa + kk * a_kstep, a_lbo, 1024);
          uint64_t bd = sdesc(sb + kk * b_kstep, b_lbo, 1024);
          mma_bf16(tmem, ad, bd, p.idesc, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(empty_bar(s));
      }
      // Always signal the epilogue (also after an early exit) once every
      // issued MMA has completed.
      mma_commit(acc_bar);
    }
  } else {
    // ---------------- epilogue warps 2..5 ----------------
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int row_in_tile = q * 32 + lane;
    const int gm = m0 + row_in_tile;
    bool ok = true;
    if (do_db) {
      // db[m] = sum over this split's K range of A(m, k) = dY[k, m]; A is
      // MN-major: two 64(m) x 64(k) boxes, 128-byte rows, 128B swizzle.
      float colsum = 0.f;
      const int t = threadIdx.x - 64;       // 0..127 -> m within the tile
      const int box = t >> 6, mi = t & 63;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % C::STAGES;
        const uint32_t ph = (uint32_t)(i / C::STAGES) & 1u;
        ok = __all_sync(0xffffffffu, mbar_wait(full_bar(s), ph, p.err));
        if (!ok) break;
        const uint8_t* tile = base_ptr + (a_base - base) + s * A_STAGE_BYTES + box * 8192;
#pragma unroll 8
        for (int r = 0; r < BK; ++r) {
          const int off = r * 128 + ((((mi >> 3) ^ (r & 7))) << 4) + ((mi & 7) << 1);
          colsum += __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + off));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(s));
      }
      const int m = m0 + t;
      if (ok && m < p.M) {
        if (p.ws) p.ws[(int64_t)gridDim.z * p.M * p.N + (int64_t)blockIdx.z * p.M + m] = colsum;
        else p.db[m] = colsum;
      }
    }
    ok = __all_sync(0xffffffffu, mbar_wait(acc_bar, 0, p.err) && ok);
    tc_fence_after();
    if (ok && nkb > 0) {
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16];
        tmem_ld16(trow + c0, v);
        const int gn0 = n0 + c0;
        if (gm >= p.M || gn0 >= p.N) continue;
        const bool full = gn0 + 16 <= p.N;
        if (p.kind == GEMM_WGRAD) {
          float* dst = p.ws ? p.ws + ((int64_t)blockIdx.z * p.M + gm) * p.N + gn0
                            : p.dW + (int64_t)gm * p.ld_dw + gn0;
          const bool vec = full && (((uintptr_t)dst & 15) == 0);
          if (vec) {
#pragma unroll
            for (int j = 0; j < 16; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
          } else {
            for (int j = 0; j < 16 && gn0 + j < p.N; ++j) dst[j] = v[j];
          }
          continue;
        }
        float o[16];
        if (p.kind == GEMM_FWD) {
          float u[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int gn = gn0 + j;
            u[j] = v[j] + (gn < p.N ? __ldg(p.bias + gn) : 0.f);
            o[j] = apply_act(u[j], p.act);
          }
          if (p.out_u) {
            __nv_bfloat16* du = p.out_u + (int64_t)gm * p.ldu + gn0;
            if (full && (((uintptr_t)du & 15) == 0)) {
              __align__(16) __nv_bfloat16 tmp[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) tmp[j] = __float2bfloat16_rn(u[j]);
              reinterpret_cast<uint4*>(du)[0] = reinterpret_cast<uint4*>(tmp)[0];
              reinterpret_cast<uint4*>(du)[1] = reinterpret_cast<uint4*>(tmp)[1];
            } else {
              for (int j = 0; j < 16 && gn0 + j < p.N; ++j) du[j] = __float2bfloat16_rn(u[j]);
            }
          }
        } else {  // GEMM_DGRAD
          const __nv_bfloat16* ar = p.aux + (int64_t)gm * p.ld_aux + gn0;
          if (p.act == ACT_NONE) {
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] = v[j];
          } else if (full && (((uintptr_t)ar & 15) == 0)) {
            __align__(16) __nv_bfloat16 tmp[16];
            reinterpret_cast<uint4*>(tmp)[0] = __ldg(reinterpret_cast<const uint4*>(ar));
            reinterpret_cast<uint4*>(tmp)[1] = __ldg(reinterpret_cast<const uint4*>(ar) + 1);
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] = v[j] * act_grad_from_stored(__bfloat162float(tmp[j]), p.act);
          } else {
            for (int j = 0; j < 16; ++j)
              o[j] = gn0 + j < p.N ? v[j] * act_grad_from_stored(__bfloat162float(ar[j]), p.act) : 0.f;
          }
        }
        __nv_bfloat16* dst = p.out + (int64_t)gm * p.ldo + gn0;
        if (full && (((uintptr_t)dst & 15) == 0)) {
          __align__(16) __nv_bfloat16 tmp[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) tmp[j] = __float2bfloat16_rn(o[j]);
          reinterpret_cast<uint4*>(dst)[0] = reinterpret_cast<uint4*>(tmp)[0];
          reinterpret_cast<uint4*>(dst)[1] = reinterpret_cast<uint4*>(tmp)[1];
        } else {
          for (int j = 0; j < 16 && gn0 + j < p.N; ++j) dst[j] = __float2bfloat16_rn(o[j]);
        }
      }
    }
    if (ok && nkb == 0 && gm < p.M) {
      // Empty K range (only possible for a trailing split): contribute zeros.
      for (int gn = n0; gn < min(n0 + BN, p.N); ++gn) {
        if (p.kind == GEMM_WGRAD) {
          if (p.ws) p.ws[((int64_t)blockIdx.z * p.M + gm) * p.N + gn] = 0.f;
          else p.dW[(int64_t)gm * p.ld_dw + gn] = 0.f;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Persistent variant for the forward and dgrad GEMMs (bf16 out).
//
// One CTA per SM walks output tiles t = blockIdx.x, +gridDim.x, ... in
// m-major order (concurrent CTAs share A row blocks in L2).  The TMA ring runs
// across tile boundaries; the MMA warp accumulates tile i into TMEM buffer
// i % 2 while the epilogue warps drain buffer (i - 1) % 2; the epilogue
// stages each 32-row x 64-column bf16 chunk in 128B-swizzled shared memory
// (two buffers per warp) and writes it with a TMA bulk-tensor store, which
// also clips the ragged edges of the output.
// ---------------------------------------------------------------------------
constexpr int P_EPI_WARPS = 8;
constexpr int P_THREADS = 64 + 32 * P_EPI_WARPS;   // producer warp, MMA warp, 8 epilogue warps
// epilogue staging: per warp, 1 or 2 buffers of 32 rows x 128 B
//
// A k-block's loads take about a microsecond to land (L2 across the two
// dies), so a stage must buy enough MMA time: bf16 stages are 32-48 KB, four
// or five deep; with fp32 operands as planes (X3) a stage holds all three
// planes of A and of B (96 KB, two deep) and feeds six MMA groups.  X3 keeps
// two accumulators per TMEM buffer: hi x hi, and the five smaller products.

template <int BN, bool X3 = false> struct PCfg {
  static constexpr int NPL = X3 ? 3 : 1;                 // operand planes per stage
  static constexpr int A_BYTES = NPL * A_STAGE_BYTES;
  static constexpr int B_PLANE_BYTES = BN * BK * 2;
  static constexpr int B_BYTES = NPL * B_PLANE_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = X3 ? 2 : (BN >= 256 ? 4 : 5);
  static constexpr int EPI_BUFS = (X3 || BN >= 256) ? 1 : 2;   // staging buffers per epilogue warp
  static constexpr int EPI_BYTES = P_EPI_WARPS * EPI_BUFS * 4096;
  static constexpr int ACC_COLS = X3 ? 2 * BN : BN;      // TMEM columns per accumulator buffer
  static constexpr int TMEM_COLS = 2 * ACC_COLS;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + 1024 + 256;
  static_assert(TMEM_COLS <= 512, "TMEM holds 512 columns");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

// fp32 operands on the tensor cores: an fp32 value x is stored as three bf16
// planes hi + mid + lo (= x to 24 bits); an fp32 GEMM accumulates the six
// significant plane products in fp32.  Every bf16 x bf16 product is exact in
// fp32, so the result carries fp32-level error.  Phase f of the K loop uses
// planes (pa, pb) below, smallest products first: the accumulator is still
// small while the small phases are added, so its rounding at each step costs
// them nothing, and the hi x hi phase accumulates like a plain GEMM.
__device__ __forceinline__ void prod6_planes(int f, int& pa, int& pb) {
  // (1,1) (2,0) (0,2) (1,0) (0,1) (0,0)
  pa = (0x001021 >> (4 * f)) & 0xF;
  pb = (0x010201 >> (4 * f)) & 0xF;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(dst),
      "l"((uint64_t)tm), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

struct PParams {
  CUtensorMap tmA;
  CUtensorMap tmB;
  CUtensorMap tmOut;     // bf16 [M rows, N cols] (2-D, or 3-D with 3 planes), box {64, 32}, 128B swizzle
  CUtensorMap tmU;       // the GELU pre-activation out_u like tmOut (CTA pairs, when u_tma)
  int u_tma;
  int M, N, K;
  int num_kb, tiles_n, num_tiles;
  // tile order: m_fast = 1 walks the row tiles of a column tile first (CTAs
  // running at the same time share B's columns; chosen when A is the smaller
  // operand, so B is read from DRAM once and A stays in L2), else the column
  // tiles of a row tile first
  int tiles_m, m_fast;
  int b_mn;
  int kind, act;
  uint32_t idesc;
  const float* bias;
  __nv_bfloat16* out_u; int64_t ldu;
  const __nv_bfloat16* aux; int64_t ld_aux;
  uint32_t* err;
  // softmax-CE around the output layer (bf16, 256-wide tiles):
  //   forward: each row's (max, sum exp(z - max)) over every 128-column group
  //   of the stored logits -> ce_stats [M][ce_groups], z[row, label] -> ce_zy;
  //   dgrad: A holds the logits z; dz = (exp(z - M_r) invS_r - [c == y_r])
  //   ce_scale is formed in shared memory before the MMA reads the stage.
  float2* ce_stats; float* ce_zy; int ce_groups;
  const float2* ce_rowstat; const int32_t* ce_labels; float ce_scale;
  // ReLU mask as bits (bf16, one CTA per tile): written by the forward,
  // read by the dgrad in place of the stored activation
  uint64_t* relu_bits; int64_t ld_bits;
  // The 10-class output layer folded into this forward (CTA pairs, X3,
  // N = 128): `out` receives dY of this layer; the sums over each 128-row
  // tile (a pair) of dW_out (row-major [10][128]) and db_out go to
  // head_ws + tile * kFhPitch, the tile's loss sum to head_ws +
  // head_loss_off + tile
  const float* head_W; const float* head_bias; const int32_t* head_labels;
  float* head_ws; int64_t head_loss_off; float head_scale;
  int64_t* step_counter; float* bias_corr; float beta1, beta2;
};

// Output tile t of a persistent walk: its first row and column.
__device__ __forceinline__ void tile_origin(const PParams& p, int t, int bm, int bn, int& m0, int& n0) {
  if (p.m_fast) {
    m0 = (t % p.tiles_m) * bm;
    n0 = (t / p.tiles_m) * bn;
  } else {
    m0 = (t / p.tiles_n) * bm;
    n0 = (t % p.tiles_n) * bn;
  }
}

constexpr int kFhC = 10, kFhK = 128;   // classes, inputs of the folded output layer
constexpr int kFhPart = kFhC * kFhK + kFhC;   // dW_out + db_out partial length
constexpr int kFhPitch = 1292;                 // partial pitch, rounded up to 16 bytes
constexpr int kFhZ = 11;                // padded pitch of a row's 10 logits / dz in shared memory

// dz of softmax-CE from a stored logit: (exp(z - M) invS - onehot) scale, or 0
// outside the batch rows / classes.
__device__ __forceinline__ float ce_dz(float z, float M, float inv_s, bool hot, float scale, bool valid) {
  return valid ? (__expf(z - M) * inv_s - (hot ? 1.f : 0.f)) * scale : 0.f;
}

// Eight bf16 logits of one 16-byte unit (classes c0 .. c0 + 7) turned into dz
// in place.
__device__ __forceinline__ void ce_unit(uint8_t* unit, int c0, int C, int y, float M, float inv_s, float scale,
                                        bool row_ok) {
  uint4 w = *reinterpret_cast<const uint4*>(unit);
  __nv_bfloat162* w2 = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const float2 z = __bfloat1622float2(w2[h]);
    const int c = c0 + 2 * h;
    w2[h] = __floats2bfloat162_rn(ce_dz(z.x, M, inv_s, c == y, scale, row_ok && c < C),
                                  ce_dz(z.y, M, inv_s, c + 1 == y, scale, row_ok && c + 1 < C));
  }
  *reinterpret_cast<uint4*>(unit) = w;
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v, int off) {
  uint32_t r[32];
  // load and wait in one statement: the outputs are defined only after the wait
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr + (uint32_t)off)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 64 consecutive TMEM columns of this warp's 32 lanes: two x32 loads and one
// wait in a single statement (the outputs are defined only after the wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr), "r"(taddr + 32u)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* tm, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"((uint64_t)tm),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
// The activation of a 64-value chunk, the choice made once for the chunk
// (the epilogue's straight-line code runs once per tile, so keeping the ReLU
// path short and contiguous saves instruction fetch).
__device__ __forceinline__ void act_chunk(float (&v)[64], int act) {
  if (act == ACT_RELU) {
#pragma unroll
    for (int j = 0; j < 64; ++j) v[j] = fmaxf(v[j], 0.0f);
  } else if (act == ACT_GELU_TANH) {
#pragma unroll
    for (int j = 0; j < 64; ++j) v[j] = gelu_tanh(v[j]);
  }
}
// The ReLU mask of a 64-column chunk as two 32-bit words: bit j set where
// the bf16 rounding of v[j] is positive.  v is the ReLU output (>= 0, or
// -0), and bf16's smallest positive value is 2^-133, so the rounding is
// positive exactly when v > 2^-134 (2^-134 itself ties to the even zero):
// one compare per element where the chunk lies inside N; columns at or
// beyond N get no bit.
__device__ __forceinline__ void relu_mask_bits(const float (&v)[64], int gn0, int N, uint32_t& b0, uint32_t& b1) {
  constexpr float kMinPos = 0x1p-134f;
  if (gn0 + 64 <= N) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      b0 |= (v[j] > kMinPos ? 1u : 0u) << j;
      b1 |= (v[32 + j] > kMinPos ? 1u : 0u) << j;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      b0 |= (gn0 + j < N && v[j] > kMinPos ? 1u : 0u) << j;
      b1 |= (gn0 + 32 + j < N && v[32 + j] > kMinPos ? 1u : 0u) << j;
    }
  }
}
// One output plane of a warp's 32 rows x 64 columns into 128B-swizzled
// shared memory (16-byte unit u of row r at r*128 + ((u ^ (r & 7)) * 16)):
// the bf16 rounding of v; with `rest`, v then keeps the remainder v - plane,
// so that successive calls write hi, mid and lo (x = hi + mid + lo; each
// difference is exact in fp32).  One packed conversion per pair of values.
__device__ __forceinline__ void stage_plane(uint8_t* srow, int lane, float (&v)[64], bool rest) {
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * u + 2 * h], v[8 * u + 2 * h + 1]);
      w[h] = *reinterpret_cast<const uint32_t*>(&b2);
      if (rest) {
        v[8 * u + 2 * h] -= __uint_as_float(w[h] << 16);
        v[8 * u + 2 * h + 1] -= __uint_as_float(w[h] & 0xFFFF0000u);
      }
    }
    *reinterpret_cast<uint4*>(srow + ((u ^ (lane & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}
// Thread-block cluster helpers (the CTA pair of tc_gemm_pair_kernel).
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA in the cluster: release this thread's prior
// writes (including to other CTAs' shared memory) and wait for all threads.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// The shared::cluster address of this CTA's shared::cta address `a` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_cluster(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t a, float x, float y, float z, float w) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(x), "f"(y), "f"(z), "f"(w)
               : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t a, float x) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(x) : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"((uint64_t)tm),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// Named barrier `id` over `n` threads (whole warps) of this CTA.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// X3: fp32 operands as three bf16 planes (3-D maps, six K-loop phases) and
// an fp32 result written as its three planes.
// PAIR: the CTAs of a 2-CTA cluster share one output tile, each taking half of
// the K stages; after both main loops each CTA hands the accumulator rows the
// other finishes (64 of the 128) to it through distributed shared memory and
// finishes its own 64 rows.  Used when there are at most half as many tiles
// as SMs, so every CTA has one tile and its pipeline memory is free at the end.
template <int BN, bool X3, bool PAIR>
__device__ __forceinline__ void persistent_body(const PParams& p) {
  using C = PCfg<BN, X3>;
  constexpr int OUT_PLANES = X3 ? 3 : 1;
  // X3 epilogue of a CTA's last tile: 4 KB buffers per epilogue warp (one
  // per plane of each of its 64-column chunks), taken from pipeline memory
  constexpr int kX3LastBufs = (BN / 128) * OUT_PLANES;
  static_assert(!X3 || P_EPI_WARPS * kX3LastBufs * 4096 <= C::STAGES * C::STAGE_BYTES, "X3 staging");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t a_base = base;
  const uint32_t b_base = base + C::STAGES * C::A_BYTES;
  const uint32_t epi_base = b_base + C::STAGES * C::B_BYTES;
  const uint32_t bar_base = epi_base + C::EPI_BYTES;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int b) { return bar_base + 8u * (2 * C::STAGES + b); };
  auto tempty_bar = [&](int b) { return bar_base + 8u * (2 * C::STAGES + 2 + b); };
  // softmax-CE dgrad: stage s formed into dz by the epilogue warps
  auto formed_bar = [&](int s) { return bar_base + 8u * (2 * C::STAGES + 4 + s); };
  const uint32_t tmem_slot = bar_base + 8u * (3 * C::STAGES + 4);
  volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));
  // the logits of a softmax-CE dgrad are turned into dz between TMA and MMA
  const bool ce_a = !X3 && !PAIR && p.ce_rowstat != nullptr;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(formed_bar(s), P_EPI_WARPS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), P_EPI_WARPS);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot_ptr;
  pdl_enter();   // shared memory and TMEM are set up: now wait for the inputs
  // the folded output layer takes over the step counter (nothing before the
  // optimizer reads it)
  if (PAIR && p.step_counter && blockIdx.x == 0 && threadIdx.x == 0)
    advance_step(p.step_counter, p.bias_corr, p.beta1, p.beta2);
  const uint32_t stage_tx = C::STAGE_BYTES;
  // tiles walked by this CTA (a pair walks them together) and its K stages
  const int pr = PAIR ? (int)cluster_ctarank() : 0;
  // a pair handles exactly one tile; a launch with more tiles than pairs does nothing
  const bool bad_pair = PAIR && p.num_tiles > (int)(gridDim.x >> 1);
  if (bad_pair && threadIdx.x == 0 && blockIdx.x == 0 && p.err) atomicOr(p.err, ERRBIT_BAD_LAUNCH);
  const int t0 = bad_pair ? p.num_tiles : PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int tstep = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int kh = PAIR ? (p.num_kb + 1) / 2 : p.num_kb;
  const int kb_lo = PAIR ? pr * kh : 0;
  const int kb_hi = PAIR ? min(p.num_kb, kb_lo + kh) : p.num_kb;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&p.tmA);
      prefetch_tmap(&p.tmB);
      prefetch_tmap(&p.tmOut);   // the epilogue's first TMA store need not fetch it
      int it = 0;
      bool ok = true;
      for (int t = t0; t < p.num_tiles && ok; t += tstep) {
        int m0, n0;
        tile_origin(p, t, BM, BN, m0, n0);
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, p.err)) { ok = false; break; }
          mbar_expect_tx(full_bar(s), stage_tx);
          const int k0 = kb * BK;
          const uint32_t sa = a_base + s * C::A_BYTES;
          const uint32_t sb = b_base + s * C::B_BYTES;
          if (!X3) {
            tma_load_2d(sa, &p.tmA, k0, m0, full_bar(s));
            if (!p.b_mn) {
              tma_load_2d(sb, &p.tmB, k0, n0, full_bar(s));
            } else {
#pragma unroll
              for (int c = 0; c < BN / 64; ++c) tma_load_2d(sb + 8192 * c, &p.tmB, n0 + 64 * c, k0, full_bar(s));
            }
          } else {
#pragma unroll
            for (int pl = 0; pl < 3; ++pl) {   // every plane of A and B once
              tma_load_3d(sa + pl * A_STAGE_BYTES, &p.tmA, k0, m0, pl, full_bar(s));
              const uint32_t sbp = sb + pl * C::B_PLANE_BYTES;
              if (!p.b_mn) {
                tma_load_3d(sbp, &p.tmB, k0, n0, pl, full_bar(s));
              } else {
#pragma unroll
                for (int c = 0; c < BN / 64; ++c) tma_load_3d(sbp + 8192 * c, &p.tmB, n0 + 64 * c, k0, pl, full_bar(s));
              }
            }
          }
        }
      }
      for (int i = max(0, it - C::STAGES); i < it; ++i)
        mbar_wait(full_bar(i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u, p.err);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t b_kstep = p.b_mn ? 2048u : 32u;
      const uint32_t b_lbo = p.b_mn ? 8192u : 16u;
      int it = 0, tc = 0;
      bool ok = true;
      for (int t = t0; t < p.num_tiles && ok; t += tstep, ++tc) {
        const int buf = tc & 1;
        if (!mbar_wait(tempty_bar(buf), (((uint32_t)tc >> 1) & 1u) ^ 1u, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * C::ACC_COLS);
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
          if (!mbar_wait(ce_a ? formed_bar(s) : full_bar(s), ph, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = a_base + s * C::A_BYTES;
          const uint32_t sb = b_base + s * C::B_BYTES;
          if (!X3) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = sdesc(sa + kk * 32u, 16u, 1024u);
              const uint64_t bd = sdesc(sb + kk * b_kstep, b_lbo, 1024u);
              mma_bf16(d, ad, bd, p.idesc, (kb > kb_lo || kk > 0) ? 1u : 0u);
            }
          } else {
            // five small products into the second accumulator (smallest
            // first), then hi x hi into the first
#pragma unroll
            for (int f = 0; f < 6; ++f) {
              int pa, pb;
              prod6_planes(f, pa, pb);
              const uint32_t dd = f < 5 ? d + BN : d;
              const uint32_t spa = sa + pa * A_STAGE_BYTES, spb = sb + pb * C::B_PLANE_BYTES;
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                const uint64_t ad = sdesc(spa + kk * 32u, 16u, 1024u);
                const uint64_t bd = sdesc(spb + kk * b_kstep, b_lbo, 1024u);
                const bool first = kb == kb_lo && kk == 0 && (f == 0 || f == 5);
                mma_bf16(dd, ad, bd, p.idesc, first ? 0u : 1u);
              }
            }
          }
          mma_commit(empty_bar(s));
        }
        mma_commit(tfull_bar(buf));
      }
    }
  } else if (!PAIR) {
    // ---------------- epilogue warps 2..9 ----------------
    // warp w reads TMEM lanes 32*(w%4)..+31 (its lane quarter) and the
    // columns of its half of the tile: two warps share each quarter
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t stage0 = epi_base + (uint32_t)((warp - 2) * C::EPI_BUFS * 4096);
    int tc = 0, chunk = 0, it = 0;
    bool ok = true;
    for (int t = t0; t < p.num_tiles && ok; t += tstep, ++tc) {
      int m0, n0;
        tile_origin(p, t, BM, BN, m0, n0);
      const int buf = tc & 1;
      const bool last_tile = t + tstep >= p.num_tiles;
      if (ce_a) {
        // softmax-CE dgrad: every landed A stage (128 rows x 64 logits,
        // 128B-swizzled) becomes dz in place before the MMA reads it; thread
        // e takes row e / 2 and its 16-byte units 4 (e % 2) .. 4 (e % 2) + 3
        const int e = threadIdx.x - 64;
        const int r = e >> 1, hb = e & 1;
        const int gr = m0 + r;
        const bool rok = gr < p.M;
        float2 st = make_float2(0.f, 0.f);
        int y = -1;
        if (rok) {
          st = __ldg(p.ce_rowstat + gr);
          y = __ldg(p.ce_labels + gr);
        }
        for (int kb = kb_lo; kb < kb_hi && ok; ++kb, ++it) {
          const int s = it % C::STAGES;
          ok = __all_sync(0xffffffffu, mbar_wait(full_bar(s), (uint32_t)(it / C::STAGES) & 1u, p.err));
          if (!ok) break;
          uint8_t* row = base_ptr + (a_base - base) + s * C::A_BYTES + r * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            // logical unit j (columns 8 j .. 8 j + 7) sits at physical unit
            // j ^ (r & 7): the eight lanes of a shared-memory phase hit eight
            // different bank groups
            const int j = 4 * hb + i;
            ce_unit(row + 16 * (j ^ (r & 7)), kb * BK + 8 * j, p.K, y, st.x, st.y, p.ce_scale, rok);
          }
          fence_async_smem();   // the generic-proxy writes, visible to the tensor cores
          __syncwarp();
          if (lane == 0) mbar_arrive(formed_bar(s));
        }
        if (!ok) break;
      }
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * C::ACC_COLS);
      const int gm = m0 + q * 32 + lane;
      const bool row_ok = gm < p.M;
      // softmax-CE forward: this row's label, and the running (max, sum) of
      // its 128-column group (this warp's half of the 256-wide tile)
      const bool ce_f = !X3 && !PAIR && p.ce_stats != nullptr;
      int ce_y = -1;
      if (ce_f && row_ok) ce_y = __ldg(p.ce_labels + gm);
      float ce_m = -INFINITY, ce_s = 0.f;
      // 64-column chunks of this warp's half of the tile: read from TMEM once,
      // finished in registers, then each output plane is staged in
      // 128B-swizzled shared memory (16-byte unit u of row r at
      // r*128 + ((u ^ (r & 7)) * 16)) and written by a TMA store.  The
      // accumulator wait comes after the first chunk's bias / mask loads, so
      // their latency overlaps the MMAs.
      bool acc_ready = false;
#pragma unroll 1
      for (int c0 = half * (BN / 2); c0 < (half + 1) * (BN / 2); c0 += 64) {
        const int gn0 = n0 + c0;
        // the chunk's bias (lane j: columns j and 32 + j) or ReLU mask of the
        // stored activation, loaded before the TMEM read
        float bias0 = 0.f, bias1 = 0.f;
        uint32_t mask0 = 0u, mask1 = 0u;
        if (p.kind == GEMM_FWD) {
          if (gn0 + lane < p.N) bias0 = __ldg(p.bias + gn0 + lane);
          if (gn0 + 32 + lane < p.N) bias1 = __ldg(p.bias + gn0 + 32 + lane);
        } else if (p.act == ACT_RELU && row_ok && !X3 && !PAIR && p.relu_bits) {
          // the forward's bits of these 64 columns: 8 bytes instead of 128
          // (a chunk wholly beyond N has no bit group: its mask stays 0)
          const uint2 w = gn0 < p.N ? __ldg(reinterpret_cast<const uint2*>(p.relu_bits + (int64_t)(gn0 / 64) * p.ld_bits + gm))
                                    : make_uint2(0u, 0u);
          mask0 = w.x;
          mask1 = w.y;
        } else if (p.act == ACT_RELU && row_ok) {
          const __nv_bfloat16* ar = p.aux + (int64_t)gm * p.ld_aux + gn0;
          if (gn0 + 64 <= p.N) {
            uint4 a[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) a[u] = __ldg(reinterpret_cast<const uint4*>(ar) + u);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&a[u]);
              uint32_t bits = 0u;
#pragma unroll
              for (int h = 0; h < 8; ++h) bits |= (__bfloat162float(e[h]) > 0.f ? 1u : 0u) << h;
              if (u < 4) mask0 |= bits << (8 * u);
              else mask1 |= bits << (8 * (u - 4));
            }
          } else {
            for (int j = 0; j < 32; ++j) {
              if (gn0 + j < p.N && __bfloat162float(ar[j]) > 0.f) mask0 |= 1u << j;
              if (gn0 + 32 + j < p.N && __bfloat162float(ar[32 + j]) > 0.f) mask1 |= 1u << j;
            }
          }
        }
        if (!acc_ready) {
          ok = __all_sync(0xffffffffu, mbar_wait(tfull_bar(buf), ((uint32_t)tc >> 1) & 1u, p.err));
          if (!ok) break;
          tc_fence_after();
          acc_ready = true;
        }
        float v[64];
        tmem_ld64(trow + (uint32_t)c0, v);
        if (X3) {   // hi x hi + the five smaller products
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float w[32];
            tmem_ld32(trow + (uint32_t)(BN + c0 + 32 * hh), w, 0);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[32 * hh + j] += w[j];
          }
        }
        if (c0 + 64 >= (half + 1) * (BN / 2)) {
          // this warp's part of the TMEM buffer is drained: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(buf));
        }
        if (p.kind == GEMM_FWD) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] += __shfl_sync(0xffffffffu, bias0, j);
            v[32 + j] += __shfl_sync(0xffffffffu, bias1, j);
          }
          if (p.out_u && row_ok) {
            __nv_bfloat16* du = p.out_u + (int64_t)gm * p.ldu + gn0;
            if (gn0 + 64 <= p.N) {
#pragma unroll
              for (int j = 0; j < 64; j += 8) {
                uint4 w;
                __nv_bfloat162* w2 = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
                for (int h = 0; h < 4; ++h) w2[h] = __floats2bfloat162_rn(v[j + 2 * h], v[j + 2 * h + 1]);
                *reinterpret_cast<uint4*>(du + j) = w;
              }
            } else {
#pragma unroll
              for (int j = 0; j < 64; ++j)
                if (gn0 + j < p.N) du[j] = __float2bfloat16_rn(v[j]);
            }
          }
          act_chunk(v, p.act);
          if (!X3 && !PAIR && p.relu_bits && row_ok && gn0 < p.N) {
            // bit j: the stored (bf16) activation is positive
            uint32_t b0 = 0u, b1 = 0u;
            relu_mask_bits(v, gn0, p.N, b0, b1);
            // a warp's 32 rows are 32 consecutive words: one coalesced store
            *reinterpret_cast<uint2*>(p.relu_bits + (int64_t)(gn0 / 64) * p.ld_bits + gm) = make_uint2(b0, b1);
          }
          if (ce_f) {
            // the logits as stored (bf16): the chunk maximum folded into the
            // group's running maximum, then the exponentials added; the
            // label's logit is kept when it falls in this chunk
            // (rounding v in place: the store below rounds it to the same value)
            float mc = -INFINITY, zy = 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
              v[j] = __bfloat162float(__float2bfloat16_rn(v[j]));
              if (gn0 + j < p.N) mc = fmaxf(mc, v[j]);
              if (gn0 + j == ce_y) zy = v[j];
            }
            if (mc > ce_m) {
              ce_s *= __expf(ce_m - mc);
              ce_m = mc;
            }
#pragma unroll
            for (int j = 0; j < 64; ++j)
              if (gn0 + j < p.N) ce_s += __expf(v[j] - ce_m);
            if (row_ok && ce_y >= gn0 && ce_y < gn0 + 64 && ce_y < p.N) p.ce_zy[gm] = zy;
            const int gc0 = n0 + half * (BN / 2);   // first column of this warp's group (BN = 256)
            if (c0 + 64 >= (half + 1) * (BN / 2) && row_ok && gc0 < p.N)
              p.ce_stats[(int64_t)gm * p.ce_groups + gc0 / 128] = make_float2(ce_m, ce_s);
          }
        } else if (p.act == ACT_RELU) {   // dgrad: dX * 1[h > 0]
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] *= (float)((mask0 >> j) & 1u);
            v[32 + j] *= (float)((mask1 >> j) & 1u);
          }
        } else if (p.act == ACT_GELU_TANH) {   // dgrad: dX * gelu'(u) (bf16 only)
          const __nv_bfloat16* ar = p.aux + (int64_t)gm * p.ld_aux + gn0;
          if (row_ok && gn0 + 64 <= p.N) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint4 a = __ldg(reinterpret_cast<const uint4*>(ar) + u);
              const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&a);
#pragma unroll
              for (int h = 0; h < 8; ++h) v[8 * u + h] *= gelu_tanh_grad(__bfloat162float(e[h]));
            }
          } else {
#pragma unroll
            for (int j = 0; j < 64; ++j)
              v[j] *= (row_ok && gn0 + j < p.N) ? gelu_tanh_grad(__bfloat162float(ar[j])) : 0.f;
          }
        }
#pragma unroll 1
        for (int pl = 0; pl < OUT_PLANES; ++pl, ++chunk) {
          // X3, last tile of this CTA: its MMAs are done and no load follows,
          // so the pipeline memory holds every plane of every chunk of this
          // warp at once and the stores go out back to back; otherwise the
          // warp's staging buffers are reused once a store has read them
          uint32_t sbuf_addr;
          if (X3 && last_tile) {
            sbuf_addr = a_base + (uint32_t)((((warp - 2) * kX3LastBufs) + (c0 - half * (BN / 2)) / 64 * OUT_PLANES + pl) * 4096);
          } else {
            const int sbuf = chunk % C::EPI_BUFS;
            if (lane == 0) {   // the store that last used this buffer has read it
              if (C::EPI_BUFS == 1) bulk_wait_read0();
              else bulk_wait_read1();
            }
            sbuf_addr = stage0 + (uint32_t)(sbuf * 4096);
          }
          __syncwarp();
          uint8_t* srow = base_ptr + (sbuf_addr - base) + lane * 128;
          stage_plane(srow, lane, v, pl + 1 < OUT_PLANES);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (!X3) tma_store_2d(&p.tmOut, sbuf_addr, gn0, m0 + q * 32);
            else tma_store_3d(&p.tmOut, sbuf_addr, gn0, m0 + q * 32, pl);
            bulk_commit();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  if (PAIR) {
    // ---------------- the pair's epilogue (every thread of both CTAs) ----------------
    // CTA rank r finishes rows 64 r .. 64 r + 63 (TMEM lane quarters 2r, 2r+1)
    // and sends the other 64 rows (big + small accumulators added) to its
    // peer's pipeline memory, padded rows of kRP floats.  Each epilogue warp
    // holds one 32-row x 64-column chunk; the finishing warps load their bias
    // / mask before the accumulator is ready and read their own TMEM while
    // the peer's rows are in flight.
    static_assert(!PAIR || BN == 128, "one 64-column chunk per epilogue warp");
    constexpr int kRP = BN + 4;
    const bool have = t0 < p.num_tiles;   // the same for both CTAs of the pair
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const bool mine = warp >= 2 && (q >> 1) == pr;
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    const int m0 = have ? (t0 / p.tiles_n) * BM : 0, n0 = have ? (t0 % p.tiles_n) * BN : 0;
    const int c0 = half * (BN / 2);
    const int gn0 = n0 + c0;
    const int gm = m0 + q * 32 + lane;
    const bool row_ok = gm < p.M;
    float bias0 = 0.f, bias1 = 0.f;
    uint32_t mask0 = 0u, mask1 = 0u;
    if (mine && have) {
      if (p.kind == GEMM_FWD) {
        if (gn0 + lane < p.N) bias0 = __ldg(p.bias + gn0 + lane);
        if (gn0 + 32 + lane < p.N) bias1 = __ldg(p.bias + gn0 + 32 + lane);
      } else if (p.act == ACT_RELU && row_ok) {
        const __nv_bfloat16* ar = p.aux + (int64_t)gm * p.ld_aux + gn0;
        if (gn0 + 64 <= p.N) {
          uint4 a[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) a[u] = __ldg(reinterpret_cast<const uint4*>(ar) + u);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&a[u]);
            uint32_t bits = 0u;
#pragma unroll
            for (int h = 0; h < 8; ++h) bits |= (__bfloat162float(e[h]) > 0.f ? 1u : 0u) << h;
            if (u < 4) mask0 |= bits << (8 * u);
            else mask1 |= bits << (8 * (u - 4));
          }
        } else {
          for (int j = 0; j < 32; ++j) {
            if (gn0 + j < p.N && __bfloat162float(ar[j]) > 0.f) mask0 |= 1u << j;
            if (gn0 + 32 + j < p.N && __bfloat162float(ar[32 + j]) > 0.f) mask1 |= 1u << j;
          }
        }
      }
    }
    // the folded output layer: its weights into shared memory (the epilogue
    // staging area, which the pair does not use), its bias and this row's
    // label, all before the accumulator is ready
    const bool fh = PAIR && p.head_W != nullptr;
    // its partial sums: this CTA's (sP) and, in rank 0, rank 1's (sP2)
    const uint32_t fh_p_addr = epi_base + (uint32_t)((kFhC * kFhK + 2 * 64 * kFhZ + 64) * 4);
    const uint32_t fh_p2_addr = fh_p_addr + (uint32_t)(kFhPitch * 4);
    float hbias[kFhC];
#pragma unroll
    for (int c = 0; c < kFhC; ++c) hbias[c] = 0.f;
    int hy = 0;
    if (fh && have && warp >= 2) {
      const int e = (int)threadIdx.x - 64;   // 0 .. 255 over the epilogue warps
      float* sW = reinterpret_cast<float*>(base_ptr + (epi_base - base));
      for (int i = e; i < kFhC * kFhK / 4; i += 256)
        reinterpret_cast<float4*>(sW)[i] = __ldg(reinterpret_cast<const float4*>(p.head_W) + i);
      if (e < 64) {   // the softmax of row e (below): its bias and label
#pragma unroll
        for (int c = 0; c < kFhC; ++c) hbias[c] = __ldg(p.head_bias + c);
        if (m0 + 64 * pr + e < p.M) hy = __ldg(p.head_labels + m0 + 64 * pr + e);
      }
    }
    bool ok = true;
    if (warp >= 2 && have) {
      ok = __all_sync(0xffffffffu, mbar_wait(tfull_bar(0), 0u, p.err));
      tc_fence_after();
    }
    // one decision for the whole CTA: the finishing warps below meet at named
    // barriers, so either all of them run or none
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    cluster_sync_all();   // both CTAs' MMAs are done: their pipeline memory is free
    const uint32_t recv = a_base;   // [64][kRP] fp32
    float v[64];
    if (warp >= 2 && have && ok) {   // this warp's chunk: hi x hi + the five smaller products
      tmem_ld64(trow + (uint32_t)c0, v);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float w[32];
        tmem_ld32(trow + (uint32_t)(BN + c0 + 32 * hh), w, 0);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[32 * hh + j] += w[j];
      }
      if (!mine) {   // the peer finishes these rows
        const uint32_t peer =
            mapa_cluster(recv, (uint32_t)(pr ^ 1)) + (uint32_t)((((q & 1) * 32 + lane) * kRP + c0) * 4);
#pragma unroll
        for (int j = 0; j < 64; j += 4) st_cluster_v4(peer + (uint32_t)(j * 4), v[j], v[j + 1], v[j + 2], v[j + 3]);
      }
    }
    cluster_sync_all();   // the peer's rows have landed
    // staging: every plane of a finishing warp's chunk at once, in the B half
    // of the (now idle) pipeline memory; the peer's rows sit in the A half
    static_assert(!PAIR || P_EPI_WARPS * kX3LastBufs * 4096 <= C::STAGES * C::B_BYTES, "pair staging");
    static_assert(!PAIR || 64 * kRP * 4 <= C::STAGES * C::A_BYTES, "pair exchange");
    const uint32_t stage0 = b_base + (uint32_t)((warp - 2) * kX3LastBufs * 4096);
    float* sD = reinterpret_cast<float*>(base_ptr + (recv - base));   // [64][kRP]: the peer's rows, then dY
    if (mine && have && ok) {
      const float* rrow = sD + ((q & 1) * 32 + lane) * kRP;
#pragma unroll
      for (int j = 0; j < 64; j += 4) {   // + the peer's partial sums of these rows
        const float4 r4 = *reinterpret_cast<const float4*>(rrow + c0 + j);
        v[j] += r4.x; v[j + 1] += r4.y; v[j + 2] += r4.z; v[j + 3] += r4.w;
      }
      if (p.kind == GEMM_FWD) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          v[j] += __shfl_sync(0xffffffffu, bias0, j);
          v[32 + j] += __shfl_sync(0xffffffffu, bias1, j);
        }
        act_chunk(v, p.act);
      } else if (p.act == ACT_RELU) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          v[j] *= (float)((mask0 >> j) & 1u);
          v[32 + j] *= (float)((mask1 >> j) & 1u);
        }
      }
    }
    if (fh && have && ok && warp >= 2) {
      // the folded output layer over this CTA's 64 rows (row r = 32 (q % 2) +
      // lane of a finishing warp; batch row m0 + 64 rank + r), shared by all
      // eight epilogue warps (thread e).  It runs once per CTA: short rolled
      // loops over rows held in shared memory (h in sH; dY into sD, whose
      // peer rows have been added).
      static_assert(!PAIR || (kFhC * kFhK + 2 * 64 * kFhZ + 64 + 2 * kFhPitch) * 4 <= C::EPI_BYTES, "head smem");
      static_assert(!PAIR || 2 * 64 * kRP * 4 <= C::STAGES * C::A_BYTES, "head rows");
      const float* sW = reinterpret_cast<const float*>(base_ptr + (epi_base - base));   // [10][128]
      float* sZ = reinterpret_cast<float*>(base_ptr + (epi_base - base)) + kFhC * kFhK;  // [64][kFhZ]: logits
      float* sDz = sZ + 64 * kFhZ;                                                      // [64][kFhZ]: dz
      float* sL = sDz + 64 * kFhZ;                                                      // [64]: row losses
      float* sH = sD + 64 * kRP;                                                        // [64][kRP]: h
      const int e = (int)threadIdx.x - 64;
      if (mine) {
        float* hrow = sH + ((q & 1) * 32 + lane) * kRP + c0;
#pragma unroll
        for (int j = 0; j < 64; j += 4) *reinterpret_cast<float4*>(hrow + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
      }
      named_bar_sync(1, 256);   // h and the weights are in shared memory
      {   // logits of row e % 64, classes e / 64, + 4, + 8
        const int r = e & 63, g = e >> 6;
        const bool g3 = g + 8 < kFhC;
        const float* hr = sH + r * kRP;
        const float* w0 = sW + g * kFhK;
        const float* w1 = sW + (g + 4) * kFhK;
        const float* w2 = sW + (g3 ? g + 8 : g) * kFhK;
        float z0 = 0.f, z1 = 0.f, z2 = 0.f;
#pragma unroll 2
        for (int k = 0; k < kFhK; k += 4) {
          const float4 h4 = *reinterpret_cast<const float4*>(hr + k);
          const float4 a = *reinterpret_cast<const float4*>(w0 + k);
          const float4 b = *reinterpret_cast<const float4*>(w1 + k);
          const float4 c = *reinterpret_cast<const float4*>(w2 + k);
          z0 = fmaf(h4.x, a.x, z0); z0 = fmaf(h4.y, a.y, z0); z0 = fmaf(h4.z, a.z, z0); z0 = fmaf(h4.w, a.w, z0);
          z1 = fmaf(h4.x, b.x, z1); z1 = fmaf(h4.y, b.y, z1); z1 = fmaf(h4.z, b.z, z1); z1 = fmaf(h4.w, b.w, z1);
          z2 = fmaf(h4.x, c.x, z2); z2 = fmaf(h4.y, c.y, z2); z2 = fmaf(h4.z, c.z, z2); z2 = fmaf(h4.w, c.w, z2);
        }
        sZ[r * kFhZ + g] = z0;
        sZ[r * kFhZ + g + 4] = z1;
        if (g3) sZ[r * kFhZ + g + 8] = z2;
      }
      named_bar_sync(1, 256);
      if (e < 64) {   // softmax cross-entropy of row e: dz (0 past the batch) and its loss
        const bool rok = m0 + 64 * pr + e < p.M;
        float z[kFhC];
#pragma unroll
        for (int c = 0; c < kFhC; ++c) z[c] = sZ[e * kFhZ + c] + hbias[c];
        float mx = z[0], zy = 0.f;
#pragma unroll
        for (int c = 0; c < kFhC; ++c) {
          mx = fmaxf(mx, z[c]);
          if (c == hy) zy = z[c];
        }
        float se = 0.f;
#pragma unroll
        for (int c = 0; c < kFhC; ++c) {
          z[c] = expf(z[c] - mx);
          se += z[c];
        }
        const float inv = 1.0f / se;
#pragma unroll
        for (int c = 0; c < kFhC; ++c)
          sDz[e * kFhZ + c] = rok ? (z[c] * inv - (c == hy ? 1.f : 0.f)) * p.head_scale : 0.f;
        float lr = 0.f;
        if (rok) {
          if (hy < 0 || hy >= kFhC) {
            if (p.err) atomicOr(p.err, ERRBIT_LABEL_RANGE);
          } else {
            lr = (mx + logf(se)) - zy;
          }
        }
        sL[e] = lr;
      }
      named_bar_sync(1, 256);   // dz and the losses are in shared memory
      {   // dY = (dz W) * act'(h) of row e % 64, columns 32 (e / 64) .. + 31, into sD
          // (a warp reads the same weights: broadcast)
        const int r = e & 63, cq = (e >> 6) * 32;
        float dz[kFhC];
#pragma unroll
        for (int c = 0; c < kFhC; ++c) dz[c] = sDz[r * kFhZ + c];
        const float* hr = sH + r * kRP + cq;
        float* dr = sD + r * kRP + cq;
#pragma unroll 1
        for (int j = 0; j < 32; j += 4) {
          float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int c = 0; c < kFhC; ++c) {
            const float4 w = *reinterpret_cast<const float4*>(sW + c * kFhK + cq + j);
            a.x = fmaf(dz[c], w.x, a.x);
            a.y = fmaf(dz[c], w.y, a.y);
            a.z = fmaf(dz[c], w.z, a.z);
            a.w = fmaf(dz[c], w.w, a.w);
          }
          if (p.act == ACT_RELU) {
            const float4 h4 = *reinterpret_cast<const float4*>(hr + j);
            a.x = h4.x > 0.f ? a.x : 0.f;
            a.y = h4.y > 0.f ? a.y : 0.f;
            a.z = h4.z > 0.f ? a.z : 0.f;
            a.w = h4.w > 0.f ? a.w : 0.f;
          }
          *reinterpret_cast<float4*>(dr + j) = a;
        }
      }
      {   // this CTA's partial sums over its 64 rows: dW_out at column e % 128
          // for classes 5 (e / 128) .. + 4; db_out (e < 10) and the loss
          // (e = 10).  Rank 0 keeps its partial (sP), rank 1 writes its own
          // into rank 0's sP2; rank 0 adds the two below.
        const int col = e & 127, ch = e >> 7;
        float acc[5];
#pragma unroll
        for (int k = 0; k < 5; ++k) acc[k] = 0.f;
#pragma unroll 2
        for (int r = 0; r < 64; ++r) {
          const float h = sH[r * kRP + col];
#pragma unroll
          for (int k = 0; k < 5; ++k) acc[k] = fmaf(sDz[r * kFhZ + 5 * ch + k], h, acc[k]);
        }
        const uint32_t dst = pr == 0 ? fh_p_addr : mapa_cluster(fh_p2_addr, 0u);
#pragma unroll
        for (int k = 0; k < 5; ++k) st_cluster_f32(dst + 4u * (uint32_t)((5 * ch + k) * kFhK + col), acc[k]);
        if (e < kFhC) {
          float a = 0.f;
          for (int r = 0; r < 64; ++r) a += sDz[r * kFhZ + e];
          st_cluster_f32(dst + 4u * (uint32_t)(kFhC * kFhK + e), a);
        } else if (e == kFhC) {
          float a = 0.f;
          for (int r = 0; r < 64; ++r) a += sL[r];
          st_cluster_f32(dst + 4u * (uint32_t)kFhPart, a);
        }
      }
      named_bar_sync(1, 256);   // every dY row is in sD
      if (mine) {   // this warp's dY chunk back into v for the planes
        const float* drow = sD + ((q & 1) * 32 + lane) * kRP + c0;
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
          const float4 a = *reinterpret_cast<const float4*>(drow + j);
          v[j] = a.x; v[j + 1] = a.y; v[j + 2] = a.z; v[j + 3] = a.w;
        }
      }
    }
    if (mine && have && ok) {
#pragma unroll 1
      for (int pl = 0; pl < OUT_PLANES; ++pl) {
        const uint32_t sbuf_addr = stage0 + (uint32_t)(pl * 4096);
        uint8_t* srow = base_ptr + (sbuf_addr - base) + lane * 128;
        stage_plane(srow, lane, v, pl + 1 < OUT_PLANES);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (!X3) tma_store_2d(&p.tmOut, sbuf_addr, gn0, m0 + q * 32);
          else tma_store_3d(&p.tmOut, sbuf_addr, gn0, m0 + q * 32, pl);
          bulk_commit();
        }
      }
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
    if (fh && have) {
      // the pair's partial sums: rank 1's have landed in rank 0's sP2 (the
      // barrier orders them); rank 0 adds them to its own and writes the
      // tile's partial (row-major dW_out, then db_out) and loss sum
      cluster_sync_all();
      if (pr == 0) {
        const float* sP = reinterpret_cast<const float*>(base_ptr + (fh_p_addr - base));
        const float* sP2 = reinterpret_cast<const float*>(base_ptr + (fh_p2_addr - base));
        const int tile = (int)(blockIdx.x >> 1);
        for (int i = threadIdx.x; i <= kFhPart; i += blockDim.x) {
          const float a = sP[i] + sP2[i];
          if (i < kFhPart) p.head_ws[(int64_t)tile * kFhPitch + i] = a;
          else p.head_ws[p.head_loss_off + tile] = a;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int BN, bool X3>
__global__ void __launch_bounds__(P_THREADS, 1) tc_gemm_persistent_kernel(const __grid_constant__ PParams p) {
  persistent_body<BN, X3, false>(p);
}

// fp32-as-planes forward / dgrad with each 128x128 tile shared by a CTA pair
// (split K, exchange through distributed shared memory).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
tc_gemm_pair_kernel(const __grid_constant__ PParams p) {
  persistent_body<128, true, true>(p);
}

// ---------------------------------------------------------------------------
// 2-SM variant of the bf16 forward / dgrad (tcgen05.mma.cta_group::2).
//
// A cluster of two CTAs on two SMs computes 256 x 256 output tiles.  CTA r
// keeps rows 128 r .. 128 r + 127 of the tile's A rows and columns
// 128 r .. 128 r + 127 of its B columns in its own shared memory; one thread
// of CTA 0 issues the MMAs (M = 256, N = 256), which read both CTAs' halves
// and accumulate rows 128 r .. 128 r + 127 of the tile into CTA r's TMEM.
// Per SM a 64-deep stage is then 32 KB for a 128 x 256 x 64 share of the
// work, against 48 KB for the same work in a one-SM 128 x 256 tile: a third
// fewer operand bytes from L2 per FLOP.
//   Both CTAs' loads complete on CTA 0's "full" barriers (a TMA load with
// .cta_group::2 may signal the peer's barrier); the MMA commits signal the
// "empty" and "accumulator full" barriers of both CTAs at once (multicast),
// and both CTAs' epilogue warps arrive on CTA 0's "accumulator empty"
// barrier.  The epilogue is the one-SM kernel's for bf16 (bias + activation,
// GELU pre-activation, ReLU bits; dgrad masks) on this CTA's 128 rows.
// ---------------------------------------------------------------------------
struct G2Cfg {
  static constexpr int TBM = 2 * BM, TBN = 256;          // the pair's output tile
  static constexpr int A_BYTES = BM * BK * 2;            // this CTA's 128 rows of A
  static constexpr int B_BYTES = (TBN / 2) * BK * 2;     // this CTA's 128 columns of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 32 KB
  static constexpr int STAGES = 6;
  static constexpr int EPI_BYTES = P_EPI_WARPS * 4096;   // one 32 x 64 staging buffer per epilogue warp
  static constexpr int ACC_COLS = TBN;
  static constexpr int TMEM_COLS = 2 * ACC_COLS;         // double-buffered accumulator
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + 1024 + 256;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(TMEM_COLS <= 512, "TMEM holds 512 columns");
};

__device__ __forceinline__ void tmem_alloc_cg2(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_cg2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_bf16_cg2(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum));
}
// Arrive on the barrier at shared offset `bar` of both CTAs of the pair once
// the MMAs issued so far have completed.
__device__ __forceinline__ void mma_commit_cg2(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
// TMA load into this CTA's shared memory, its bytes counted on a barrier of
// either CTA of the pair (a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_cg2(uint32_t dst, const CUtensorMap* tm, int c0, int c1,
                                                uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"((uint64_t)tm), "r"(c0), "r"(c1), "r"(bar_cluster)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (arrivals from the peer CTA).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint32_t* err) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (globaltimer() - t0 > kWaitLimitNs) {
      if (err) atomicOr(err, ERRBIT_TIMEOUT);
      return false;
    }
  }
}

// FWD: the forward epilogue (bias, activation, pre-activation or ReLU bits),
// else the dgrad's (activation derivative); separate instances so that each
// epilogue has the registers to itself.
template <bool FWD>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
tc_gemm_cg2_kernel(const __grid_constant__ PParams p) {
  using C = G2Cfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t a_base = base;
  const uint32_t b_base = base + C::STAGES * C::A_BYTES;
  const uint32_t epi_base = b_base + C::STAGES * C::B_BYTES;
  const uint32_t bar_base = epi_base + C::EPI_BYTES;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int b) { return bar_base + 8u * (2 * C::STAGES + b); };
  auto tempty_bar = [&](int b) { return bar_base + 8u * (2 * C::STAGES + 2 + b); };
  const uint32_t tmem_slot = bar_base + 8u * (2 * C::STAGES + 4);
  volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // 0: the CTA whose thread issues the MMAs
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * P_EPI_WARPS);   // the epilogue warps of both CTAs
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc_cg2(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  cluster_sync_all();   // both CTAs' barriers exist before either signals the other's
  tc_fence_after();
  const uint32_t tmem = *tmem_slot_ptr;
  pdl_enter();   // shared memory and TMEM are set up: now wait for the inputs
  const uint32_t lead_full0 = mapa_cluster(full_bar(0), 0);
  const uint32_t lead_tempty0 = mapa_cluster(tempty_bar(0), 0);
  const int t0 = (int)(blockIdx.x >> 1), tstep = (int)(gridDim.x >> 1);

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      prefetch_tmap(&p.tmA);
      prefetch_tmap(&p.tmB);
      prefetch_tmap(&p.tmOut);
      int it = 0;
      bool ok = true;
      for (int t = t0; t < p.num_tiles && ok; t += tstep) {
        int m0, n0;
        tile_origin(p, t, C::TBM, C::TBN, m0, n0);
        m0 += (int)rank * BM;                             // this CTA's rows of A
        const int nb = n0 + (int)rank * (C::TBN / 2);     // this CTA's columns of B
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, p.err)) { ok = false; break; }
          if (rank == 0) mbar_expect_tx(full_bar(s), 2u * C::STAGE_BYTES);   // both CTAs' bytes
          const uint32_t fb = lead_full0 + 8u * (uint32_t)s;
          const int k0 = kb * BK;
          const uint32_t sa = a_base + s * C::A_BYTES;
          const uint32_t sb = b_base + s * C::B_BYTES;
          tma_load_2d_cg2(sa, &p.tmA, k0, m0, fb);
          if (!p.b_mn) {
            tma_load_2d_cg2(sb, &p.tmB, k0, nb, fb);
          } else {
            tma_load_2d_cg2(sb, &p.tmB, nb, k0, fb);
            tma_load_2d_cg2(sb + 8192u, &p.tmB, nb + 64, k0, fb);
          }
        }
      }
      // every stage this CTA filled has been read by the MMAs (its empty
      // barrier completed), so no copy into this CTA's memory is in flight
      for (int i = max(0, it - C::STAGES); i < it; ++i)
        mbar_wait(empty_bar(i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u, p.err);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (CTA 0) ----------------
    if (rank == 0 && lane == 0) {
      const uint32_t b_kstep = p.b_mn ? 2048u : 32u;
      const uint32_t b_lbo = p.b_mn ? 8192u : 16u;
      int it = 0, tc = 0;
      bool ok = true;
      for (int t = t0; t < p.num_tiles && ok; t += tstep, ++tc) {
        const int buf = tc & 1;
        if (!mbar_wait_cluster(tempty_bar(buf), (((uint32_t)tc >> 1) & 1u) ^ 1u, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * C::ACC_COLS);
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const int s = it % C::STAGES;
          if (!mbar_wait(full_bar(s), (uint32_t)(it / C::STAGES) & 1u, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = a_base + s * C::A_BYTES;
          const uint32_t sb = b_base + s * C::B_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16_cg2(d, sdesc(sa + kk * 32u, 16u, 1024u), sdesc(sb + kk * b_kstep, b_lbo, 1024u), p.idesc,
                         (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit_cg2(empty_bar(s));
        }
        mma_commit_cg2(tfull_bar(buf));
      }
    }
  } else {
    // ---------------- epilogue warps 2..9: this CTA's 128 rows ----------------
    // warp w reads TMEM lanes 32 (w % 4) .. +31 and the 128 columns of its
    // half of the tile, 64 at a time
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t stage0 = epi_base + (uint32_t)((warp - 2) * 4096);
    uint8_t* srow = base_ptr + (stage0 - base) + lane * 128;
    int tc = 0;
    bool ok = true;
    for (int t = t0; t < p.num_tiles && ok; t += tstep, ++tc) {
      int m0, n0;
      tile_origin(p, t, C::TBM, C::TBN, m0, n0);
      m0 += (int)rank * BM;
      const int buf = tc & 1;
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * C::ACC_COLS);
      const int gm = m0 + q * 32 + lane;
      const bool row_ok = gm < p.M;
      bool acc_ready = false;
#pragma unroll 1
      for (int c0 = half * (C::TBN / 2); c0 < (half + 1) * (C::TBN / 2); c0 += 64) {
        const int gn0 = n0 + c0;
        // the chunk's bias (lane j: columns j and 32 + j) or ReLU mask, loaded
        // before the accumulator wait
        float bias0 = 0.f, bias1 = 0.f;
        uint32_t mask0 = 0u, mask1 = 0u;
        if (FWD) {
          if (gn0 + lane < p.N) bias0 = __ldg(p.bias + gn0 + lane);
          if (gn0 + 32 + lane < p.N) bias1 = __ldg(p.bias + gn0 + 32 + lane);
        } else if (p.act == ACT_RELU && row_ok && p.relu_bits && gn0 < p.N) {
          // (a chunk wholly beyond N has no bit group: its mask stays 0)
          const uint2 w = __ldg(reinterpret_cast<const uint2*>(p.relu_bits + (int64_t)(gn0 / 64) * p.ld_bits + gm));
          mask0 = w.x;
          mask1 = w.y;
        } else if (p.act == ACT_RELU && row_ok) {
          const __nv_bfloat16* ar = p.aux + (int64_t)gm * p.ld_aux + gn0;
          for (int j = 0; j < 32; ++j) {
            if (gn0 + j < p.N && __bfloat162float(ar[j]) > 0.f) mask0 |= 1u << j;
            if (gn0 + 32 + j < p.N && __bfloat162float(ar[32 + j]) > 0.f) mask1 |= 1u << j;
          }
        }
        if (!acc_ready) {
          ok = __all_sync(0xffffffffu, mbar_wait_cluster(tfull_bar(buf), ((uint32_t)tc >> 1) & 1u, p.err));
          if (!ok) break;
          tc_fence_after();
          acc_ready = true;
        }
        float v[64];
        tmem_ld64(trow + (uint32_t)c0, v);
        const bool last = c0 + 64 >= (half + 1) * (C::TBN / 2);
        if (last) {
          // this warp's part of the accumulator is drained: hand it back to CTA 0
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(lead_tempty0 + 8u * (uint32_t)buf);
        }
        if (FWD) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] += __shfl_sync(0xffffffffu, bias0, j);
            v[32 + j] += __shfl_sync(0xffffffffu, bias1, j);
          }
          if (p.out_u && p.u_tma) {
            // the pre-activation through the staging buffer and a TMA store
            // (it clips the ragged edges), like the activation below
            if (gn0 < p.N) {
              if (lane == 0) bulk_wait_read0();
              __syncwarp();
              stage_plane(srow, lane, v, false);
              fence_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&p.tmU, stage0, gn0, m0 + q * 32);
                bulk_commit();
              }
            }
          } else if (p.out_u && row_ok) {
            __nv_bfloat16* du = p.out_u + (int64_t)gm * p.ldu + gn0;
            if (gn0 + 64 <= p.N) {
#pragma unroll
              for (int j = 0; j < 64; j += 8) {
                uint4 w;
                __nv_bfloat162* w2 = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
                for (int h = 0; h < 4; ++h) w2[h] = __floats2bfloat162_rn(v[j + 2 * h], v[j + 2 * h + 1]);
                *reinterpret_cast<uint4*>(du + j) = w;
              }
            } else {
#pragma unroll
              for (int j = 0; j < 64; ++j)
                if (gn0 + j < p.N) du[j] = __float2bfloat16_rn(v[j]);
            }
          }
          act_chunk(v, p.act);
          if (p.relu_bits && row_ok && gn0 < p.N) {
            // bit j: the stored (bf16) activation is positive
            uint32_t b0 = 0u, b1 = 0u;
            relu_mask_bits(v, gn0, p.N, b0, b1);
            *reinterpret_cast<uint2*>(p.relu_bits + (int64_t)(gn0 / 64) * p.ld_bits + gm) = make_uint2(b0, b1);
          }
        } else if (p.act == ACT_RELU) {   // dgrad: dX * 1[h > 0]
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] *= (float)((mask0 >> j) & 1u);
            v[32 + j] *= (float)((mask1 >> j) & 1u);
          }
        } else if (p.act == ACT_GELU_TANH) {   // dgrad: dX * gelu'(u)
          const __nv_bfloat16* ar = p.aux + (int64_t)gm * p.ld_aux + gn0;
          if (row_ok && gn0 + 64 <= p.N) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint4 a = __ldg(reinterpret_cast<const uint4*>(ar) + u);
              const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&a);
#pragma unroll
              for (int h = 0; h < 8; ++h) v[8 * u + h] *= gelu_tanh_grad(__bfloat162float(e[h]));
            }
          } else {
#pragma unroll
            for (int j = 0; j < 64; ++j)
              v[j] *= (row_ok && gn0 + j < p.N) ? gelu_tanh_grad(__bfloat162float(ar[j])) : 0.f;
          }
        }
        // stage the chunk (128B-swizzled) once the previous store has read
        // the buffer, then one TMA store (it clips the ragged edges); a chunk
        // wholly beyond N stores nothing
        if (gn0 >= p.N) continue;
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
        stage_plane(srow, lane, v, false);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&p.tmOut, stage0, gn0, m0 + q * 32);
          bulk_commit();
        }
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  // neither CTA leaves while the other may still signal its barriers, or the
  // MMAs may still read this CTA's shared memory or write its TMEM
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_cg2(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Persistent split-K weight gradient: dW[m, n] = sum_k A(m, k) B(k, n), with
// A = dY^T and B = X both MN-major in memory, fp32 out. The bias gradient
// db[m] = sum_k A(m, k): for bf16 by the epilogue warps on the CUDA cores
// from the landed A stages (db_stage_add: they are idle while a long unit's
// MMAs run, and a second narrow MMA per K step would lengthen those units by
// about a third), in the units db_part picks; for fp32 planes and the
// softmax-CE forming by a second MMA of the same A tile against a constant
// 16 x 64 tile of ones (N = 16) into spare TMEM columns, in one unit per row
// tile.
//
// Work units are (tile, K split) pairs, tile index fastest, so CTAs running
// at the same time share K ranges in L2.  Each unit's fp32 result goes out
// through TMA stores to the gradient plane (one split) or to a split-K
// workspace that a fixed-order reduce kernel sums (several splits).
// ---------------------------------------------------------------------------
constexpr int W_BN = 128;
constexpr int W_EPI_BUFS = 2;
constexpr int W_EPI_BYTES = P_EPI_WARPS * W_EPI_BUFS * 4096;
constexpr int W_ONES_BYTES = 16 * 128;                          // 16 rows x 64 bf16
constexpr int W_TMEM_COLS = 512;                                // 2 x (128 dW + 32 db), stride 256
// X3 (fp32 operands as three bf16 planes): a stage holds every plane of a
// 32-row K slice of A and B (48 KB, three deep) and feeds the six products,
// smallest first, into one accumulator per work unit.
// WBN = 256 (bf16, long K per work unit): 128x256 tiles halve the operand
// bytes per MMA; the accumulator then fills TMEM with the bias gradient
// beside it, so it is single-buffered (the epilogue does not overlap the next
// unit, which long units amortise).
template <bool X3, int WBN = W_BN> struct WCfg {
  static constexpr int NPL = X3 ? 3 : 1;
  static constexpr int BKW = X3 ? 32 : 64;                 // K rows per stage
  static constexpr int CHUNK_BYTES = 64 * BKW * 2;         // one 64-wide MN chunk of a plane
  static constexpr int A_PLANE_BYTES = (BM / 64) * CHUNK_BYTES;
  static constexpr int B_PLANE_BYTES = (WBN / 64) * CHUNK_BYTES;
  static constexpr int A_BYTES = NPL * A_PLANE_BYTES;
  static constexpr int B_BYTES = NPL * B_PLANE_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = X3 ? 3 : (WBN >= 256 ? 3 : 4);
  static constexpr int NBUF = WBN >= 256 ? 1 : 2;          // TMEM accumulator buffers (stride 256 columns)
  static_assert(!(X3 && WBN >= 256), "planes use 128-wide tiles");
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + W_EPI_BYTES + W_ONES_BYTES + 1024 + 256;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

struct WParams {
  CUtensorMap tmA;       // A^T storage: inner M, outer K; box {64, 64}
  CUtensorMap tmB;       // inner N, outer K; box {64, 64}
  CUtensorMap tmOut;     // fp32 3-D {N, M, splits}; box {32, 32, 1}; 128B swizzle
  int M, N, K;
  int num_kb, kb_per_split, splits;   // K stages (32 or 64 rows each), split into units
  int tiles_n, num_tiles, num_units;
  int db_share;          // bf16 bias gradient: see db_part
  uint32_t idesc, idesc_db;
  float* db_out;         // [splits][M] (nullable: no bias gradient)
  uint32_t* err;
  // softmax-CE weight gradient (bf16): A^T holds the logits z [K rows
  // (batch), M (classes)]; each stage is formed into dz in shared memory
  // (dz = (exp(z - M_k) invS_k - [m == y_k]) ce_scale) before the MMA
  const float2* ce_rowstat; const int32_t* ce_labels; float ce_scale;
};

__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r)
      : "r"(taddr)
      : "memory");
  return __uint_as_float(r);
}

// Bias gradient of a bf16 weight-gradient unit on the CUDA cores: the column
// sums of dY over the unit's K rows, taken from the landed A stages (dY^T,
// MN-major: two 64-column chunks of 64 K rows, 128B-swizzled) by the
// epilogue warps, which the long units otherwise leave idle.  Epilogue warp
// w (0..7) owns columns 16 w .. 16 w + 15 as 8 bf16 pairs; lane l takes
// pair l % 8 and the 16 rows 16 g + ((i + 2 g) mod 16), i = 0..15, g = l / 8,
// in that order (the row offset puts a warp's four row groups on distinct
// banks).  A stage's 16 rows are summed first and then added to the running
// pair; rows beyond K are zero-filled by the copy.
__device__ __forceinline__ void db_stage_add(const uint8_t* stage_a, int w, int lane, float& acc0, float& acc1) {
  const int mp = 8 * w + (lane & 7);   // columns 2 mp and 2 mp + 1 of the CTA's 128
  const int g = lane >> 3;
  const uint8_t* chunk = stage_a + (mp >> 5) * 8192;
  const int unit = (mp & 31) >> 2, byte = (mp & 3) * 4;
  float t0 = 0.f, t1 = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int r = 16 * g + ((i + 2 * g) & 15);
    const uint32_t x = *reinterpret_cast<const uint32_t*>(chunk + r * 128 + ((unit ^ (r & 7)) << 4) + byte);
    t0 += __uint_as_float(x << 16);
    t1 += __uint_as_float(x & 0xFFFF0000u);
  }
  acc0 += t0;
  acc1 += t1;
}
// The unit's bias gradient for columns m0 + 16 w + 2 (lane % 8) + {0, 1}:
// the four row groups added as (g0 + g1) + (g2 + g3) and stored by lanes
// 0..7 (row m0 + c of the [splits][M] output).
__device__ __forceinline__ void db_finish_store(float acc0, float acc1, int w, int lane, int m0, int M, int split,
                                                float* db_out) {
  acc0 += __shfl_xor_sync(0xffffffffu, acc0, 8);
  acc1 += __shfl_xor_sync(0xffffffffu, acc1, 8);
  acc0 += __shfl_xor_sync(0xffffffffu, acc0, 16);
  acc1 += __shfl_xor_sync(0xffffffffu, acc1, 16);
  const int m = m0 + 16 * w + 2 * lane;
  if (lane < 8) {
    if (m < M) db_out[(int64_t)split * M + m] = acc0;
    if (m + 1 < M) db_out[(int64_t)split * M + m + 1] = acc1;
  }
}
// Which units sum the bias gradient of a row tile (each epilogue warp's
// sums are the same whichever unit forms them, so this changes no result).
// share = 0 (several waves of units): the unit of column tile
// ti_m mod tiles_n, all eight warps (part 0), spreading such units over
// the CTAs.  share = 1 (one wave: the slowest unit sets the time): the
// rows are shared among the row tile's column tiles, P = min(tiles_n, 8)
// parts; the unit of column tile ti_n takes part (ti_n + ti_m) mod tiles_n
// (none if that is >= P), part j being the rows of the warps w with
// w P / 8 == j.  Returns the part, or -1.
__device__ __forceinline__ int db_part(const float* db_out, int ti_m, int ti_n, int tiles_n, int share) {
  if (db_out == nullptr) return -1;
  if (!share) return ti_n == ti_m % tiles_n ? 0 : -1;
  const int j = (ti_n + ti_m) % tiles_n;
  return j < min(tiles_n, 8) ? j : -1;
}
__device__ __forceinline__ bool db_warp_in_part(int w, int part, int tiles_n, int share) {
  return !share || w * min(tiles_n, 8) / 8 == part;
}

template <bool X3, int WBN>
__global__ void __launch_bounds__(P_THREADS, 1) tc_wgrad_persistent_kernel(const __grid_constant__ WParams p) {
  using C = WCfg<X3, WBN>;
  constexpr int W_STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t a_base = base;
  const uint32_t b_base = base + W_STAGES * C::A_BYTES;
  const uint32_t epi_base = b_base + W_STAGES * C::B_BYTES;
  const uint32_t ones_base = epi_base + W_EPI_BYTES;
  const uint32_t bar_base = ones_base + W_ONES_BYTES;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (W_STAGES + s); };
  auto tfull_bar = [&](int b) { return bar_base + 8u * (2 * W_STAGES + b); };
  auto tempty_bar = [&](int b) { return bar_base + 8u * (2 * W_STAGES + 2 + b); };
  auto formed_bar = [&](int s) { return bar_base + 8u * (2 * W_STAGES + 4 + s); };
  auto dbdone_bar = [&](int s) { return bar_base + 8u * (3 * W_STAGES + 4 + s); };
  const uint32_t tmem_slot = bar_base + 8u * (4 * W_STAGES + 4);
  volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));
  const bool ce_a = !X3 && p.ce_rowstat != nullptr;
  // bf16 without the softmax-CE forming: the bias gradient is summed by the
  // epilogue warps from the landed stages (db_stage_add), and the producer
  // refills such a stage only after they arrive on its dbdone barrier
  const bool db_cc = !X3 && !ce_a && p.db_out != nullptr;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  {   // the constant ones tile (bf16 1.0 = 0x3F80)
    uint32_t* ones = reinterpret_cast<uint32_t*>(base_ptr + (ones_base - base));
    for (int i = threadIdx.x; i < W_ONES_BYTES / 4; i += blockDim.x) ones[i] = 0x3F803F80u;
    fence_async_smem();   // visible to the tensor cores (async proxy)
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < W_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(formed_bar(s), P_EPI_WARPS);
      mbar_init(dbdone_bar(s), P_EPI_WARPS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), P_EPI_WARPS);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, W_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot_ptr;
  pdl_enter();   // shared memory and TMEM are set up: now wait for the inputs
  auto unit_coords = [&](int u, int& m0, int& n0, int& split, int& kb0, int& kb1) {
    const int tile = u % p.num_tiles;
    split = u / p.num_tiles;
    m0 = (tile / p.tiles_n) * BM;
    n0 = (tile % p.tiles_n) * WBN;
    kb0 = split * p.kb_per_split;
    kb1 = min(p.num_kb, kb0 + p.kb_per_split);
  };
  // the units that form the bias gradient on the tensor cores (fp32 planes,
  // softmax-CE forming): row tile i in column tile i mod tiles_n
  auto db_unit = [&](int m0, int n0) { return p.db_out != nullptr && n0 / WBN == (m0 / BM) % p.tiles_n; };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&p.tmA);
      prefetch_tmap(&p.tmB);
      prefetch_tmap(&p.tmOut);   // the epilogue's first TMA store need not fetch it
      int it = 0;
      bool ok = true;
      // bit s: the last fill of stage s feeds a bias-gradient sum / the
      // parity of that stage's next dbdone completion
      uint32_t db_prev = 0u, db_ph = 0u;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
        int m0, n0, split, kb0, kb1;
        unit_coords(u, m0, n0, split, kb0, kb1);
        const bool sum_db = db_cc && db_part(p.db_out, m0 / BM, n0 / WBN, p.tiles_n, p.db_share) >= 0;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % W_STAGES;
          const uint32_t ph = (uint32_t)(it / W_STAGES) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, p.err)) { ok = false; break; }
          if ((db_prev >> s) & 1u) {
            if (!mbar_wait(dbdone_bar(s), (db_ph >> s) & 1u, p.err)) { ok = false; break; }
            db_ph ^= 1u << s;
          }
          db_prev = sum_db ? (db_prev | (1u << s)) : (db_prev & ~(1u << s));
          mbar_expect_tx(full_bar(s), C::STAGE_BYTES);
          const int k0 = kb * C::BKW;
          const uint32_t sa = a_base + s * C::A_BYTES;
          const uint32_t sb = b_base + s * C::B_BYTES;
          if (!X3) {
            tma_load_2d(sa, &p.tmA, m0, k0, full_bar(s));
            tma_load_2d(sa + C::CHUNK_BYTES, &p.tmA, m0 + 64, k0, full_bar(s));
#pragma unroll
            for (int c = 0; c < WBN / 64; ++c) tma_load_2d(sb + c * C::CHUNK_BYTES, &p.tmB, n0 + 64 * c, k0, full_bar(s));
          } else {
#pragma unroll
            for (int pl = 0; pl < 3; ++pl) {   // every plane of A and B once
              const uint32_t spa = sa + pl * C::A_PLANE_BYTES, spb = sb + pl * C::B_PLANE_BYTES;
              tma_load_3d(spa, &p.tmA, m0, k0, pl, full_bar(s));
              tma_load_3d(spa + C::CHUNK_BYTES, &p.tmA, m0 + 64, k0, pl, full_bar(s));
              tma_load_3d(spb, &p.tmB, n0, k0, pl, full_bar(s));
              tma_load_3d(spb + C::CHUNK_BYTES, &p.tmB, n0 + 64, k0, pl, full_bar(s));
            }
          }
        }
      }
      for (int i = max(0, it - W_STAGES); i < it; ++i)
        mbar_wait(full_bar(i % W_STAGES), (uint32_t)(i / W_STAGES) & 1u, p.err);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int it = 0, tc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++tc) {
        int m0, n0, split, kb0, kb1;
        unit_coords(u, m0, n0, split, kb0, kb1);
        const bool do_db = db_unit(m0, n0) && !db_cc;   // on the tensor cores
        const int buf = C::NBUF == 2 ? (tc & 1) : 0;
        const uint32_t tph = C::NBUF == 2 ? (((uint32_t)tc >> 1) & 1u) : ((uint32_t)tc & 1u);
        if (!mbar_wait(tempty_bar(buf), tph ^ 1u, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * 256);
        bool db_started = false;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % W_STAGES;
          const uint32_t ph = (uint32_t)(it / W_STAGES) & 1u;
          if (!mbar_wait(ce_a ? formed_bar(s) : full_bar(s), ph, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = a_base + s * C::A_BYTES;
          const uint32_t sb = b_base + s * C::B_BYTES;
          // products (pa, pb) of the planes, smallest first; the bias
          // gradient sums each plane of A once, in the products that pair it
          // with B's first plane
#pragma unroll
          for (int f = 0; f < (X3 ? 6 : 1); ++f) {
            int pa = 0, pb = 0;
            if (X3) prod6_planes(f, pa, pb);
            const bool db_here = do_db && pb == 0;
            const uint32_t spa = sa + pa * C::A_PLANE_BYTES, spb = sb + pb * C::B_PLANE_BYTES;
#pragma unroll
            for (int kk = 0; kk < C::BKW / 16; ++kk) {
              const uint64_t ad = sdesc(spa + kk * 2048u, (uint32_t)C::CHUNK_BYTES, 1024u);
              const uint64_t bd = sdesc(spb + kk * 2048u, (uint32_t)C::CHUNK_BYTES, 1024u);
              const uint32_t acc = (kb > kb0 || f > 0 || kk > 0) ? 1u : 0u;
              mma_bf16(d, ad, bd, p.idesc, acc);
              if (db_here) {
                mma_bf16(d + (uint32_t)WBN, ad, sdesc(ones_base + kk * 32u, 16u, 1024u), p.idesc_db,
                         db_started ? 1u : 0u);
                db_started = true;
              }
            }
          }
          mma_commit(empty_bar(s));
        }
        mma_commit(tfull_bar(buf));
      }
    }
  } else {
    // ---------------- epilogue warps 2..9 ----------------
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t stage0 = epi_base + (uint32_t)((warp - 2) * W_EPI_BUFS * 4096);
    uint8_t* stage0_ptr = base_ptr + (stage0 - base);
    int tc = 0, chunk = 0, it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++tc) {
      int m0, n0, split, kb0, kb1;
      unit_coords(u, m0, n0, split, kb0, kb1);
      if (ce_a) {
        // softmax-CE: every landed A stage (two 64-class chunks of 64 batch
        // rows, each row 128 bytes, 128B-swizzled) becomes dz in place;
        // thread e takes chunk e / 128, row (e / 2) % 64 and the 16-byte
        // units 4 (e % 2) .. 4 (e % 2) + 3 of it
        const int e = threadIdx.x - 64;
        const int ch = e >> 7, kr = (e >> 1) & 63, hb = e & 1;
        for (int kb = kb0; kb < kb1 && ok; ++kb, ++it) {
          const int s = it % W_STAGES;
          const int b = kb * C::BKW + kr;   // batch row
          const bool rok = b < p.K;
          float2 st = make_float2(0.f, 0.f);
          int y = -1;
          if (rok) {   // in flight while the stage lands
            st = __ldg(p.ce_rowstat + b);
            y = __ldg(p.ce_labels + b);
          }
          ok = __all_sync(0xffffffffu, mbar_wait(full_bar(s), (uint32_t)(it / W_STAGES) & 1u, p.err));
          if (!ok) break;
          uint8_t* row = base_ptr + (a_base - base) + s * C::A_BYTES + ch * C::CHUNK_BYTES + kr * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = 4 * hb + i;   // logical unit j at physical unit j ^ (kr & 7)
            ce_unit(row + 16 * (j ^ (kr & 7)), m0 + 64 * ch + 8 * j, p.M, y, st.x, st.y, p.ce_scale, rok);
          }
          fence_async_smem();   // the generic-proxy writes, visible to the tensor cores
          __syncwarp();
          if (lane == 0) mbar_arrive(formed_bar(s));
        }
        if (!ok) break;
      } else if (db_cc && db_part(p.db_out, m0 / BM, n0 / WBN, p.tiles_n, p.db_share) >= 0) {
        // this warp's rows if they are in the unit's part; every warp waits
        // for each stage and arrives on its dbdone barrier
        const bool mine = db_warp_in_part(warp - 2, db_part(p.db_out, m0 / BM, n0 / WBN, p.tiles_n, p.db_share),
                                          p.tiles_n, p.db_share);
        float a0 = 0.f, a1 = 0.f;
        for (int kb = kb0; kb < kb1 && ok; ++kb, ++it) {
          const int s = it % W_STAGES;
          ok = __all_sync(0xffffffffu, mbar_wait(full_bar(s), (uint32_t)(it / W_STAGES) & 1u, p.err));
          if (!ok) break;
          if (mine) db_stage_add(base_ptr + (a_base - base) + s * C::A_BYTES, warp - 2, lane, a0, a1);
          __syncwarp();
          if (lane == 0) mbar_arrive(dbdone_bar(s));
        }
        if (!ok) break;
        if (mine) db_finish_store(a0, a1, warp - 2, lane, m0, p.M, split, p.db_out);
      } else {
        it += kb1 - kb0;
      }
      const bool do_db = db_unit(m0, n0) && !db_cc;   // read from TMEM
      const int buf = C::NBUF == 2 ? (tc & 1) : 0;
      const uint32_t tph = C::NBUF == 2 ? (((uint32_t)tc >> 1) & 1u) : ((uint32_t)tc & 1u);
      ok = __all_sync(0xffffffffu, mbar_wait(tfull_bar(buf), tph, p.err));
      if (!ok) break;
      tc_fence_after();
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * 256);
      const int gm = m0 + q * 32 + lane;
      float dbv = 0.f;
      if (do_db && half == 0 && kb1 > kb0) dbv = tmem_ld1(trow + (uint32_t)WBN);
      if (do_db && half == 0 && gm < p.M) p.db_out[(int64_t)split * p.M + gm] = dbv;
      // this warp's WBN/2 columns, 64 at a time, each as two 32x32 fp32 stores
#pragma unroll 1
      for (int c0 = half * (WBN / 2); c0 < (half + 1) * (WBN / 2); c0 += 64) {
        float v[64];
        tmem_ld32(trow, v, c0);
        tmem_ld32(trow, v + 32, c0 + 32);
        if (c0 + 64 >= (half + 1) * (WBN / 2)) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(buf));   // this warp's part of TMEM is read
        }
#pragma unroll
        for (int sub = 0; sub < 2; ++sub, ++chunk) {
          const int sbuf = chunk % W_EPI_BUFS;
          if (lane == 0) bulk_wait_read1();
          __syncwarp();
          uint8_t* srow = stage0_ptr + sbuf * 4096 + lane * 128;
#pragma unroll
          for (int w4 = 0; w4 < 8; ++w4) {
            const float4 f = make_float4(v[sub * 32 + 4 * w4], v[sub * 32 + 4 * w4 + 1], v[sub * 32 + 4 * w4 + 2],
                                         v[sub * 32 + 4 * w4 + 3]);
            *reinterpret_cast<float4*>(srow + ((w4 ^ (lane & 7)) << 4)) = f;
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&p.tmOut, stage0 + sbuf * 4096, n0 + c0 + sub * 32, m0 + q * 32, split);
            bulk_commit();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, W_TMEM_COLS);
  }
}


// ---------------------------------------------------------------------------
// 2-SM variant of the bf16 weight gradient: dW = dY^T X on CTA pairs with
// tcgen05.mma.cta_group::2, 256 x 256 tiles (each CTA holds 128 rows of dY^T
// and 128 columns of X per stage, 32 KB, both MN-major), split over K like
// the one-SM kernel. The bias gradient is summed on the CUDA cores by each
// CTA's epilogue warps from its own landed A stages (db_stage_add, the same
// order as the one-SM kernel), in the units db_part picks. The "full"
// barriers live in CTA 0, so the summing warps take a stage once the MMAs
// are done with it (the local "empty" barrier), and the producer refills it
// only after they arrive on its dbdone barrier. (A landed-stage signal
// passed on from CTA 0 measured no faster: the second read of the A stage
// from shared memory, not the wait, is what the bias gradient costs, about a
// third of a unit; hence db_part.) One accumulator buffer: the next unit's
// MMAs wait until both CTAs' epilogues have read it into registers (units
// are long; that read is a small part of them).
// ---------------------------------------------------------------------------
struct W2Cfg {
  static constexpr int TBM = 2 * BM, TBN = 256;                 // the pair's output tile
  static constexpr int CHUNK_BYTES = 64 * BK * 2;               // 64 (m or n) x 64 (k) bf16, 8 KB
  static constexpr int A_BYTES = 2 * CHUNK_BYTES;               // this CTA's 128 rows of dY^T
  static constexpr int B_BYTES = 2 * CHUNK_BYTES;               // this CTA's 128 columns of X
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;         // 32 KB
  static constexpr int STAGES = 6;
  static constexpr int EPI_BYTES = P_EPI_WARPS * 4096;          // one 32 x 32 fp32 box per epilogue warp
  static constexpr int TMEM_COLS = 256;                         // the dW accumulator, one buffer
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + 1024 + 256;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(8 * (3 * STAGES + 3) <= 256, "barrier slots");
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
tc_wgrad_cg2_kernel(const __grid_constant__ WParams p) {
  using C = W2Cfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t a_base = base;
  const uint32_t b_base = base + C::STAGES * C::A_BYTES;
  const uint32_t epi_base = b_base + C::STAGES * C::B_BYTES;
  const uint32_t bar_base = epi_base + C::EPI_BYTES;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (C::STAGES + s); };
  auto dbdone_bar = [&](int s) { return bar_base + 8u * (2 * C::STAGES + s); };
  const uint32_t tfull = bar_base + 8u * (3 * C::STAGES);
  const uint32_t tempty = bar_base + 8u * (3 * C::STAGES + 1);
  const uint32_t tmem_slot = bar_base + 8u * (3 * C::STAGES + 2);
  volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // 0: the CTA whose thread issues the MMAs
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(dbdone_bar(s), P_EPI_WARPS);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 2 * P_EPI_WARPS);   // the epilogue warps of both CTAs
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc_cg2(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  cluster_sync_all();   // both CTAs' barriers exist before either's use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot_ptr;
  pdl_enter();
  const uint32_t lead_full0 = mapa_cluster(full_bar(0), 0);
  const uint32_t lead_tempty = mapa_cluster(tempty, 0);
  const int u0 = (int)(blockIdx.x >> 1), ustep = (int)(gridDim.x >> 1);
  // work unit u: pair tile u % num_tiles (row tiles of a column tile in
  // turn), K split u / num_tiles
  auto unit_coords = [&](int u, int& m0, int& n0, int& split, int& kb0, int& kb1) {
    const int tile = u % p.num_tiles;
    split = u / p.num_tiles;
    m0 = (tile / p.tiles_n) * C::TBM;
    n0 = (tile % p.tiles_n) * C::TBN;
    kb0 = split * p.kb_per_split;
    kb1 = min(p.num_kb, kb0 + p.kb_per_split);
  };
  // this unit's part of its row tile's bias-gradient sums (db_part), or -1
  auto unit_part = [&](int m0, int n0) {
    return db_part(p.db_out, m0 / C::TBM, n0 / C::TBN, p.tiles_n, p.db_share);
  };

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      prefetch_tmap(&p.tmA);
      prefetch_tmap(&p.tmB);
      prefetch_tmap(&p.tmOut);
      int it = 0;
      bool ok = true;
      // bit s: the last fill of stage s feeds a bias-gradient sum / the
      // parity of that stage's next dbdone completion
      uint32_t db_prev = 0u, db_ph = 0u;
      for (int u = u0; u < p.num_units && ok; u += ustep) {
        int m0, n0, split, kb0, kb1;
        unit_coords(u, m0, n0, split, kb0, kb1);
        const bool sum_db = unit_part(m0, n0) >= 0;
        const int ma = m0 + (int)rank * BM, nb = n0 + (int)rank * (C::TBN / 2);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, p.err)) { ok = false; break; }
          if ((db_prev >> s) & 1u) {
            if (!mbar_wait(dbdone_bar(s), (db_ph >> s) & 1u, p.err)) { ok = false; break; }
            db_ph ^= 1u << s;
          }
          db_prev = sum_db ? (db_prev | (1u << s)) : (db_prev & ~(1u << s));
          if (rank == 0) mbar_expect_tx(full_bar(s), 2u * C::STAGE_BYTES);   // both CTAs' bytes
          const uint32_t fb = lead_full0 + 8u * (uint32_t)s;
          const int k0 = kb * BK;
          const uint32_t sa = a_base + s * C::A_BYTES;
          const uint32_t sb = b_base + s * C::B_BYTES;
          tma_load_2d_cg2(sa, &p.tmA, ma, k0, fb);
          tma_load_2d_cg2(sa + C::CHUNK_BYTES, &p.tmA, ma + 64, k0, fb);
          tma_load_2d_cg2(sb, &p.tmB, nb, k0, fb);
          tma_load_2d_cg2(sb + C::CHUNK_BYTES, &p.tmB, nb + 64, k0, fb);
        }
      }
      // every stage this CTA filled has been read by the MMAs
      for (int i = max(0, it - C::STAGES); i < it; ++i)
        mbar_wait(empty_bar(i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u, p.err);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (CTA 0) ----------------
    if (rank == 0 && lane == 0) {
      int it = 0, tc = 0;
      bool ok = true;
      for (int u = u0; u < p.num_units && ok; u += ustep, ++tc) {
        int m0, n0, split, kb0, kb1;
        unit_coords(u, m0, n0, split, kb0, kb1);
        if (!mbar_wait_cluster(tempty, ((uint32_t)tc & 1u) ^ 1u, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % C::STAGES;
          if (!mbar_wait(full_bar(s), (uint32_t)(it / C::STAGES) & 1u, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = a_base + s * C::A_BYTES;
          const uint32_t sb = b_base + s * C::B_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = sdesc(sa + kk * 2048u, (uint32_t)C::CHUNK_BYTES, 1024u);
            const uint64_t bd = sdesc(sb + kk * 2048u, (uint32_t)C::CHUNK_BYTES, 1024u);
            mma_bf16_cg2(d, ad, bd, p.idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_cg2(empty_bar(s));
        }
        mma_commit_cg2(tfull);
      }
    }
  } else {
    // ---------------- epilogue warps 2..9: this CTA's 128 rows ----------------
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t stage0 = epi_base + (uint32_t)((warp - 2) * 4096);
    uint8_t* srow = base_ptr + (stage0 - base) + lane * 128;
    int tc = 0, it = 0;
    bool ok = true;
    for (int u = u0; u < p.num_units && ok; u += ustep, ++tc) {
      int m0, n0, split, kb0, kb1;
      unit_coords(u, m0, n0, split, kb0, kb1);
      const int mr = m0 + (int)rank * BM;   // this CTA's rows
      const int part = unit_part(m0, n0);
      if (part >= 0) {
        // this unit's part of the bias gradient of this CTA's rows, stage by
        // stage as the MMAs finish with them (the stage's bytes have landed
        // by then); every warp waits and arrives, the part's warps sum
        const bool mine = db_warp_in_part(warp - 2, part, p.tiles_n, p.db_share);
        float a0 = 0.f, a1 = 0.f;
        for (int kb = kb0; kb < kb1 && ok; ++kb, ++it) {
          const int s = it % C::STAGES;
          ok = __all_sync(0xffffffffu, mbar_wait(empty_bar(s), (uint32_t)(it / C::STAGES) & 1u, p.err));
          if (!ok) break;
          if (mine) db_stage_add(base_ptr + (a_base - base) + s * C::A_BYTES, warp - 2, lane, a0, a1);
          __syncwarp();
          if (lane == 0) mbar_arrive(dbdone_bar(s));
        }
        if (!ok) break;
        if (mine) db_finish_store(a0, a1, warp - 2, lane, mr, p.M, split, p.db_out);
      } else {
        it += kb1 - kb0;
      }
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(tfull, (uint32_t)tc & 1u, p.err));
      if (!ok) break;
      tc_fence_after();
      // this warp's 128 columns into registers, the accumulator handed back
      // to CTA 0, then four 32 x 32 fp32 stores
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
      const int c0 = half * (C::TBN / 2);
      float v[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(trow, v + 32 * c, c0 + 32 * c);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(lead_tempty);
#pragma unroll
      for (int sub = 0; sub < 4; ++sub) {
        const int gn = n0 + c0 + sub * 32;
        if (gn >= p.N) continue;   // wholly beyond N: nothing to store
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
#pragma unroll
        for (int w4 = 0; w4 < 8; ++w4) {
          const float4 f = make_float4(v[sub * 32 + 4 * w4], v[sub * 32 + 4 * w4 + 1], v[sub * 32 + 4 * w4 + 2],
                                       v[sub * 32 + 4 * w4 + 3]);
          *reinterpret_cast<float4*>(srow + ((w4 ^ (lane & 7)) << 4)) = f;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&p.tmOut, stage0, gn, mr + q * 32, split);
          bulk_commit();
        }
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  // neither CTA leaves while the other may still signal its barriers, or the
  // MMAs may still read this CTA's shared memory or write its TMEM
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_cg2(tmem, C::TMEM_COLS);
  }
}

}  // namespace tc

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)f;
  });
  return fn;
}

// 2-D bf16 tensor map: inner extent `inner` (contiguous), outer extent
// `outer` with row pitch `ld` elements; box {box_inner, box_outer}; 128B
// swizzle; out-of-range elements read as zero.
bool make_tmap(CUtensorMap* tm, const void* ptr, int64_t inner, int64_t outer, int64_t ld, int box_inner,
               int box_outer, char* err, size_t errlen) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) { snprintf(err, errlen, "cuTensorMapEncodeTiled unavailable"); return false; }
  if (((uintptr_t)ptr & 15) || ((ld * 2) & 15)) {
    snprintf(err, errlen, "TMA operand needs a 16-byte aligned base and row pitch (ld=%lld)", (long long)ld);
    return false;
  }
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(err, errlen, "cuTensorMapEncodeTiled failed (%d) inner=%lld outer=%lld ld=%lld box=%dx%d", (int)r,
             (long long)inner, (long long)outer, (long long)ld, box_inner, box_outer);
    return false;
  }
  return true;
}

// make_tmap over three planes `plane` elements apart (fp32 operands held as
// bf16 hi/mid/lo planes): dims {inner, outer, 3}.
bool make_tmap_x3(CUtensorMap* tm, const void* ptr, int64_t inner, int64_t outer, int64_t ld, int64_t plane,
                  int box_inner, int box_outer, char* err, size_t errlen) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) { snprintf(err, errlen, "cuTensorMapEncodeTiled unavailable"); return false; }
  if (((uintptr_t)ptr & 15) || ((ld * 2) & 15) || ((plane * 2) & 15) || plane < ld * outer) {
    snprintf(err, errlen, "plane operand needs a 16-byte aligned base and pitches (ld=%lld plane=%lld)",
             (long long)ld, (long long)plane);
    return false;
  }
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, 3};
  cuuint64_t strides[2] = {(cuuint64_t)(ld * 2), (cuuint64_t)(plane * 2)};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(err, errlen, "cuTensorMapEncodeTiled (planes) failed (%d) inner=%lld outer=%lld", (int)r,
             (long long)inner, (long long)outer);
    return false;
  }
  return true;
}
// A 2-D map for bf16 operands, a 3-plane map for DT_F32X3 ones.
bool make_tmap_op(CUtensorMap* tm, bool x3, const void* ptr, int64_t inner, int64_t outer, int64_t ld, int64_t plane,
                  int box_inner, int box_outer, char* err, size_t errlen) {
  return x3 ? make_tmap_x3(tm, ptr, inner, outer, ld, plane, box_inner, box_outer, err, errlen)
            : make_tmap(tm, ptr, inner, outer, ld, box_inner, box_outer, err, errlen);
}

template <int BN>
const void* tc_kernel_ptr() {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute((const void*)tc::tc_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         tc::Cfg<BN>::SMEM_BYTES);
  });
  return (const void*)tc::tc_gemm_kernel<BN>;
}

constexpr int kSMs = 152;

int pick_bn(const GemmOp& op) {
  if (op.kind == GEMM_WGRAD) return 128;
  if (op.N <= 16 && !(!op.b_kmajor)) return 16;
  if (op.N >= 4096) return 256;
  return 128;
}

}  // namespace

// bk: K rows per pipeline stage (32 for fp32 operands held as planes); bn:
// the tile width.
int tc_wgrad_splits(int64_t M, int64_t N, int64_t K, int bk = tc::BK, int bn = tc::W_BN) {
  const int64_t tiles = ceil_div(M, tc::BM) * ceil_div(N, bn);
  const int64_t kbs = ceil_div(K, bk);
  // >= 2 work units per SM, each at least 8 stages long (4 with planes: a
  // stage then carries six products)
  const int64_t min_kb = bk >= tc::BK ? 8 : 4;
  // with planes the partial sums are also capped at 4 M floats (16 MB)
  const int64_t max_parts = bk >= tc::BK ? INT64_MAX : (int64_t)4 << 20;
  int64_t s = 1;
  while (tiles * s < 2 * kSMs && kbs / (s * 2) >= min_kb && s * 2 * M * N <= max_parts) s *= 2;
  return (int)s;
}

// Tile width and K splits of a tensor-core weight gradient.  bf16 with at
// least 256 columns: 256-wide tiles, with the split count that minimises
// waves x (stages per unit + 6), the 6 standing for the epilogue that a
// single-buffered accumulator does not overlap; else 128-wide tiles.
// The fixed-order reduce of s split-K partial sums of an M x N fp32 gradient
// (read s planes, write one: (s + 1) M N 4 bytes at about 6.7 TB/s), in the
// split cost models' unit: one 64-deep stage of a 128 x 256 tile on one SM
// (2 128 256 64 flops at about 12.5 TFLOP/s, 0.34 us).
static int64_t split_reduce_cost(int64_t s, int64_t M, int64_t N) {
  return s > 1 ? (s + 1) * M * N / 563000 : 0;
}

static void tc_wgrad_choice(int dtype, int64_t M, int64_t N, int64_t K, int* bn, int* splits) {
  if (dtype == DT_F32X3) {
    // double-buffered accumulators hide most of the epilogue (cost 2); at
    // least 4 stages per unit and at most 4 M floats of partial sums
    const int64_t tiles = ceil_div(M, tc::BM) * ceil_div(N, tc::W_BN);
    const int64_t kbs = ceil_div(K, tc::WCfg<true>::BKW);
    int64_t best_s = 1, best_cost = INT64_MAX;
    // at most 16 splits: the optimizer adds the partials of an element in
    // one batch of 16 loads (a second batch costs it more than the longer
    // work units cost this kernel); any count whose K chunks come out even
    // (kb_per_split = ceil(kbs / s) gives s chunks), so a layer can fill one
    // wave of SMs
    for (int64_t s = 1; s <= 16 && (s == 1 || (kbs / s >= 4 && s * M * N <= ((int64_t)4 << 20))); ++s) {
      if (ceil_div(kbs, ceil_div(kbs, s)) != s) continue;
      const int64_t cost = ceil_div(tiles * s, kSMs) * (ceil_div(kbs, s) + 2);
      if (cost < best_cost) { best_cost = cost; best_s = s; }
    }
    *bn = tc::W_BN;
    *splits = (int)best_s;
    return;
  }
  if (N < 256) {
    *bn = tc::W_BN;
    *splits = tc_wgrad_splits(M, N, K);
    return;
  }
  const int64_t tiles = ceil_div(M, tc::BM) * ceil_div(N, 256);
  const int64_t kbs = ceil_div(K, tc::BK);
  int64_t best_s = 1, best_cost = INT64_MAX;
  for (int64_t s = 1; s <= 256 && (s == 1 || kbs / s >= 8); s *= 2) {
    const int64_t cost = ceil_div(tiles * s, kSMs) * (ceil_div(kbs, s) + 6) + split_reduce_cost(s, M, N);
    if (cost < best_cost) { best_cost = cost; best_s = s; }
  }
  *bn = 256;
  *splits = (int)best_s;
}

namespace {
int cg2_max_clusters();   // (defined with the 2-SM plans below)
}

// K splits of a 2-SM weight gradient: the count that minimises waves x
// (stages per unit + 6) over the 256 x 256 pair tiles on the pairs that fit
// at once (the 6 stands for the epilogue a single accumulator buffer does
// not overlap), plus the reduce of the partial sums, with at least 8 stages
// per unit.
static int cg2_wgrad_splits(int64_t M, int64_t N, int64_t K) {
  const int64_t tiles = ceil_div(M, 256) * ceil_div(N, 256);
  const int64_t kbs = ceil_div(K, tc::BK);
  const int64_t cl = cg2_max_clusters();
  int64_t best_s = 1, best_cost = INT64_MAX;
  for (int64_t s = 1; s <= 256 && (s == 1 || kbs / s >= 8); s *= 2) {
    const int64_t cost = ceil_div(tiles * s, cl) * (ceil_div(kbs, s) + 6) + split_reduce_cost(s, M, N);
    if (cost < best_cost) { best_cost = cost; best_s = s; }
  }
  return (int)best_s;
}

// The default policy for a bf16 weight gradient on CTA pairs: both output
// dimensions at least 256 and work units of at least 16 stages.
static bool cg2_wgrad_default(int dtype, int64_t M, int64_t N, int64_t K) {
  if (dtype != DT_BF16 || M < 256 || N < 256) return false;
  return ceil_div(ceil_div(K, tc::BK), cg2_wgrad_splits(M, N, K)) >= 16;
}

int wgrad_splits(int dtype, int64_t M, int64_t N, int64_t K) {
  if (dtype == DT_F32) return simt_gemm_splits(M, N, K);
  if (cg2_wgrad_default(dtype, M, N, K)) return cg2_wgrad_splits(M, N, K);
  int bn, s;
  tc_wgrad_choice(dtype, M, N, K, &bn, &s);
  return s;
}

size_t wgrad_workspace_bytes_any(int dtype, int64_t M, int64_t N, int64_t K) {
  size_t b = wgrad_workspace_bytes(dtype, M, N, K, wgrad_splits(dtype, M, N, K));
  if (dtype == DT_BF16) {
    int bn, s;
    tc_wgrad_choice(dtype, M, N, K, &bn, &s);
    b = std::max(b, wgrad_workspace_bytes(dtype, M, N, K, s));
    if (M >= 256 && N >= 256) b = std::max(b, wgrad_workspace_bytes(dtype, M, N, K, cg2_wgrad_splits(M, N, K)));
  }
  return b;
}

size_t wgrad_workspace_bytes(int dtype, int64_t M, int64_t N, int64_t K, int splits) {
  (void)dtype; (void)K;
  if (splits <= 1) return 0;
  return (size_t)splits * (size_t)(M * N + M) * sizeof(float);
}

namespace {
const void* tcpair_kernel_ptr() {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute((const void*)tc::tc_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         tc::PCfg<128, true>::SMEM_BYTES);
  });
  return (const void*)tc::tc_gemm_pair_kernel;
}

template <int BN, bool X3>
const void* tcp_kernel_ptr() {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute((const void*)tc::tc_gemm_persistent_kernel<BN, X3>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, tc::PCfg<BN, X3>::SMEM_BYTES);
  });
  return (const void*)tc::tc_gemm_persistent_kernel<BN, X3>;
}

int device_sms() {
  static int n = [] {
    int d = 0, v = kSMs;
    if (cudaGetDevice(&d) != cudaSuccess || cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d) != cudaSuccess)
      v = kSMs;
    return v;
  }();
  return n;
}

// 3-D fp32 tensor map {inner, rows, planes} with row pitch `ld` elements and
// plane pitch `plane` elements; box {32, 32, 1}; 128B swizzle.
bool make_tmap_f32_3d(CUtensorMap* tm, const void* ptr, int64_t inner, int64_t rows, int64_t planes, int64_t ld,
                      int64_t plane, char* err, size_t errlen) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) { snprintf(err, errlen, "cuTensorMapEncodeTiled unavailable"); return false; }
  if (((uintptr_t)ptr & 15) || ((ld * 4) & 15) || ((plane * 4) & 15)) {
    snprintf(err, errlen, "fp32 TMA output needs 16-byte aligned base and pitches");
    return false;
  }
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)(ld * 4), (cuuint64_t)(plane * 4)};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(err, errlen, "cuTensorMapEncodeTiled (fp32 3-D) failed (%d)", (int)r);
    return false;
  }
  return true;
}

template <bool X3, int WBN>
const void* tcw_kernel_ptr() {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute((const void*)tc::tc_wgrad_persistent_kernel<X3, WBN>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, tc::WCfg<X3, WBN>::SMEM_BYTES);
  });
  return (const void*)tc::tc_wgrad_persistent_kernel<X3, WBN>;
}

const void* tcw2_kernel_ptr() {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute((const void*)tc::tc_wgrad_cg2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         tc::W2Cfg::SMEM_BYTES);
  });
  return (const void*)tc::tc_wgrad_cg2_kernel;
}

// Weight gradient on CTA pairs (2-SM MMAs, 256 x 256 tiles, split K).
int tc_wgrad_cg2_plan(const GemmOp& op, LaunchRec* recs, char* err, size_t errlen) {
  using G = tc::W2Cfg;
  tc::WParams p;
  memset(&p, 0, sizeof(p));
  if (!make_tmap(&p.tmA, op.A, op.M, op.K, op.lda, 64, tc::BK, err, errlen)) return -1;
  if (!make_tmap(&p.tmB, op.B, op.N, op.K, op.ldb, 64, tc::BK, err, errlen)) return -1;
  p.M = (int)op.M; p.N = (int)op.N; p.K = (int)op.K;
  p.num_kb = (int)ceil_div(op.K, tc::BK);
  int splits = op.splits > 0 ? op.splits : cg2_wgrad_splits(op.M, op.N, op.K);
  if (splits > p.num_kb) splits = p.num_kb;
  p.kb_per_split = (int)ceil_div(p.num_kb, splits);
  splits = (int)ceil_div(p.num_kb, p.kb_per_split);
  p.splits = splits;
  p.tiles_n = (int)ceil_div(op.N, G::TBN);
  p.num_tiles = (int)(ceil_div(op.M, G::TBM) * p.tiles_n);
  p.num_units = p.num_tiles * splits;
  // D f32, A and B bf16, both MN-major; M = 256 (two CTAs), N = 256 (the
  // bias gradient is summed on the CUDA cores)
  p.idesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) | ((uint32_t)(G::TBN >> 3) << 17) |
            ((uint32_t)(G::TBM >> 4) << 24);
  p.idesc_db = 0u;
  p.err = op.err;
  if (splits > 1) {
    const size_t need = wgrad_workspace_bytes(op.dtype, op.M, op.N, op.K, splits);
    if (!op.ws || op.ws_bytes < need) {
      snprintf(err, errlen, "wgrad workspace too small (%zu < %zu)", op.ws_bytes, need);
      return -1;
    }
    if (!make_tmap_f32_3d(&p.tmOut, op.ws, op.N, op.M, splits, op.N, op.M * op.N, err, errlen)) return -1;
    p.db_out = op.db ? op.ws + (int64_t)splits * op.M * op.N : nullptr;
  } else {
    if (!make_tmap_f32_3d(&p.tmOut, op.dW, op.N, op.M, 1, op.ld_dw, op.M * op.ld_dw, err, errlen)) return -1;
    p.db_out = op.db;
  }
  const int clusters = std::min(p.num_units, cg2_max_clusters());
  p.db_share = p.num_units <= clusters ? 1 : 0;   // one wave
  LaunchRec& r = recs[0];
  r.func = tcw2_kernel_ptr();
  r.smem = G::SMEM_BYTES;
  r.grid = dim3((unsigned)(2 * clusters));
  r.block = dim3(tc::P_THREADS);
  r.early = true;
  r.name = "tc2_gemm_wgrad";
  r.set_args(p);
  if (op.splits_out) *op.splits_out = splits;
  if (splits > 1 && !op.defer_reduce) {
    split_reduce_plan(op.ws, splits, op.M, op.N, op.dW, op.ld_dw, op.db, &recs[1]);
    return 2;
  }
  return 1;
}

// Weight gradient on the persistent split-K kernel (+ the fixed-order reduce).
int tc_wgrad_plan(const GemmOp& op, LaunchRec* recs, char* err, size_t errlen) {
  if (op.dtype == DT_BF16 && !op.ce_rowstat && op.cg2 != 0 && op.M >= 256 && op.N >= 256 &&
      (op.cg2 > 0 || cg2_wgrad_default(op.dtype, op.M, op.N, op.K)))
    return tc_wgrad_cg2_plan(op, recs, err, errlen);
  tc::WParams p;
  memset(&p, 0, sizeof(p));
  const bool x3 = op.dtype == DT_F32X3;
  const int bkw = x3 ? tc::WCfg<true>::BKW : tc::WCfg<false>::BKW;
  if (!make_tmap_op(&p.tmA, x3, op.A, op.M, op.K, op.lda, op.a_plane, 64, bkw, err, errlen)) return -1;
  if (!make_tmap_op(&p.tmB, x3, op.B, op.N, op.K, op.ldb, op.b_plane, 64, bkw, err, errlen)) return -1;
  p.M = (int)op.M; p.N = (int)op.N; p.K = (int)op.K;
  p.num_kb = (int)ceil_div(op.K, bkw);
  if (op.ce_rowstat) {
    if (x3 || !op.ce_labels) { snprintf(err, errlen, "softmax-CE wgrad: bf16 with labels only"); return -1; }
    p.ce_rowstat = op.ce_rowstat; p.ce_labels = op.ce_labels; p.ce_scale = op.ce_scale;
  }
  int wbn, splits;
  tc_wgrad_choice(op.dtype, op.M, op.N, op.K, &wbn, &splits);
  if (op.splits > 0) splits = op.splits;
  if (splits > p.num_kb) splits = p.num_kb;
  p.kb_per_split = (int)ceil_div(p.num_kb, splits);
  splits = (int)ceil_div(p.num_kb, p.kb_per_split);
  p.splits = splits;
  p.tiles_n = (int)ceil_div(op.N, wbn);
  p.num_tiles = (int)(ceil_div(op.M, tc::BM) * p.tiles_n);
  p.num_units = p.num_tiles * splits;
  p.idesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) | ((uint32_t)(wbn >> 3) << 17) |
            ((uint32_t)(tc::BM >> 4) << 24);
  p.idesc_db = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | ((uint32_t)(16 >> 3) << 17) |
               ((uint32_t)(tc::BM >> 4) << 24);
  p.err = op.err;
  if (splits > 1) {
    const size_t need = wgrad_workspace_bytes(op.dtype, op.M, op.N, op.K, splits);
    if (!op.ws || op.ws_bytes < need) {
      snprintf(err, errlen, "wgrad workspace too small (%zu < %zu)", op.ws_bytes, need);
      return -1;
    }
    if (!make_tmap_f32_3d(&p.tmOut, op.ws, op.N, op.M, splits, op.N, op.M * op.N, err, errlen)) return -1;
    p.db_out = op.db ? op.ws + (int64_t)splits * op.M * op.N : nullptr;
  } else {
    if (!make_tmap_f32_3d(&p.tmOut, op.dW, op.N, op.M, 1, op.ld_dw, op.M * op.ld_dw, err, errlen)) return -1;
    p.db_out = op.db;
  }
  LaunchRec& r = recs[0];
  r.func = x3 ? tcw_kernel_ptr<true, 128>() : wbn == 256 ? tcw_kernel_ptr<false, 256>() : tcw_kernel_ptr<false, 128>();
  r.smem = x3 ? tc::WCfg<true>::SMEM_BYTES
              : wbn == 256 ? tc::WCfg<false, 256>::SMEM_BYTES : tc::WCfg<false, 128>::SMEM_BYTES;
  const int sms = device_sms();
  p.db_share = p.num_units <= sms ? 1 : 0;   // one wave
  r.grid = dim3((unsigned)(p.num_units < sms ? p.num_units : sms));
  r.block = dim3(tc::P_THREADS);
  r.early = true;
  r.name = "tc_gemm_wgrad";
  r.set_args(p);
  if (op.splits_out) *op.splits_out = splits;
  if (splits > 1 && !op.defer_reduce) {
    split_reduce_plan(op.ws, splits, op.M, op.N, op.dW, op.ld_dw, op.db, &recs[1]);
    return 2;
  }
  return 1;
}

template <bool FWD>
const void* tcg2_kernel_ptr() {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute((const void*)tc::tc_gemm_cg2_kernel<FWD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         tc::G2Cfg::SMEM_BYTES);
  });
  return (const void*)tc::tc_gemm_cg2_kernel<FWD>;
}

// CTA pairs of the 2-SM kernel that fit on the device at once (a GPC may
// leave an SM unpaired), so that a persistent grid is one wave.
int cg2_max_clusters() {
  static int n = [] {
    const int sms = device_sms();
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)(sms & ~1));
    cfg.blockDim = dim3(tc::P_THREADS);
    cfg.dynamicSmemBytes = tc::G2Cfg::SMEM_BYTES;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2; attr.val.clusterDim.y = 1; attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(&c, tcg2_kernel_ptr<true>(), &cfg) != cudaSuccess || c < 1) {
      cudaGetLastError();
      c = sms / 2;
    }
    return c;
  }();
  return n;
}

// Forward / dgrad on the 2-SM kernel: CTA pairs walk 256 x 256 tiles.
int tc_cg2_plan(const GemmOp& op, LaunchRec* recs, char* err, size_t errlen) {
  using G = tc::G2Cfg;
  tc::PParams p;
  memset(&p, 0, sizeof(p));
  if (!make_tmap(&p.tmA, op.A, op.K, op.M, op.lda, 64, tc::BM, err, errlen)) return -1;
  if (op.b_kmajor) {
    if (!make_tmap(&p.tmB, op.B, op.K, op.N, op.ldb, 64, G::TBN / 2, err, errlen)) return -1;
  } else {
    if (!make_tmap(&p.tmB, op.B, op.N, op.K, op.ldb, 64, 64, err, errlen)) return -1;
  }
  if (!make_tmap(&p.tmOut, op.out, op.N, op.M, op.ldo, 64, 32, err, errlen)) return -1;
  p.M = (int)op.M; p.N = (int)op.N; p.K = (int)op.K;
  p.num_kb = (int)ceil_div(op.K, tc::BK);
  p.tiles_n = (int)ceil_div(op.N, G::TBN);
  p.tiles_m = (int)ceil_div(op.M, G::TBM);
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.m_fast = op.M < op.N ? 1 : 0;
  p.b_mn = op.b_kmajor ? 0 : 1;
  p.kind = op.kind; p.act = op.act;
  // D f32, A and B bf16, B MN-major for the dgrad, N = 256, M = 256 (two CTAs)
  p.idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)p.b_mn << 16) | ((uint32_t)(G::TBN >> 3) << 17) |
            ((uint32_t)(G::TBM >> 4) << 24);
  p.bias = op.bias;
  p.out_u = (__nv_bfloat16*)op.out_u; p.ldu = op.ldu;
  // the pre-activation through TMA stores where its layout allows a tensor
  // map (16-byte aligned base and pitch), else plain stores
  if (op.out_u && ((uintptr_t)op.out_u & 15) == 0 && ((op.ldu * 2) & 15) == 0) {
    char e2[256];
    p.u_tma = make_tmap(&p.tmU, op.out_u, op.N, op.M, op.ldu, 64, 32, e2, sizeof(e2)) ? 1 : 0;
  }
  p.aux = (const __nv_bfloat16*)op.aux; p.ld_aux = op.ld_aux;
  p.err = op.err;
  if (op.relu_bits && op.act == ACT_RELU) {
    if (op.ld_bits < op.M || ((uintptr_t)op.relu_bits & 7)) {
      snprintf(err, errlen, "ReLU bits: ld_bits >= M, 8-byte aligned");
      return -1;
    }
    p.relu_bits = op.relu_bits; p.ld_bits = op.ld_bits;
  }
  const int clusters = std::min(p.num_tiles, cg2_max_clusters());
  LaunchRec& r = recs[0];
  r.func = op.kind == GEMM_FWD ? tcg2_kernel_ptr<true>() : tcg2_kernel_ptr<false>();
  r.smem = G::SMEM_BYTES;
  r.grid = dim3((unsigned)(2 * clusters));
  r.block = dim3(tc::P_THREADS);
  r.early = true;
  r.name = op.kind == GEMM_FWD ? "tc2_gemm_fwd" : "tc2_gemm_dgrad";
  r.set_args(p);
  return 1;
}

// Forward / dgrad on the persistent kernel (bf16 output through TMA stores).
int tc_persistent_plan(const GemmOp& op, LaunchRec* recs, char* err, size_t errlen) {
  // 256-wide tiles where they still give every SM a tile
  const int sms = device_sms();
  const bool x3 = op.dtype == DT_F32X3;   // 128-wide tiles only (three planes per stage)
  // the softmax-CE forward groups columns by 128: one warp's half of a 256-wide tile
  const bool ce_f = op.kind == GEMM_FWD && op.ce_stats;
  const bool ce_a = op.kind == GEMM_DGRAD && op.ce_rowstat;
  if ((ce_f || ce_a) && (x3 || !op.ce_labels || (ce_f && (op.N <= 128 || !op.ce_zy)))) {
    snprintf(err, errlen, "softmax-CE GEMM: bf16, labels, and (forward) more than 128 columns");
    return -1;
  }
  // bf16 with at least 256 rows and columns: CTA pairs with 2-SM MMAs, by
  // default where the pair tiles fill the device at least once and the
  // reduction is at least 16 stages long (with fewer, the per-tile costs
  // that a pair pays together outweigh the halved operand traffic: the
  // 512-wide layers of the deep narrow net, K = 512, measured 12 % slower)
  if (!x3 && !ce_f && !ce_a && op.dtype == DT_BF16 && op.cg2 != 0 && op.M >= 256 && op.N >= 256 &&
      (op.cg2 > 0 || (ceil_div(op.M, 256) * ceil_div(op.N, 256) >= cg2_max_clusters() &&
                      ceil_div(op.K, tc::BK) >= 16)))
    return tc_cg2_plan(op, recs, err, errlen);
  const int BN = !x3 && op.N > 128 && (ce_f || ceil_div(op.M, tc::BM) * ceil_div(op.N, 256) >= sms) ? 256 : 128;
  tc::PParams p;
  memset(&p, 0, sizeof(p));
  if (!make_tmap_op(&p.tmA, x3, op.A, op.K, op.M, op.lda, op.a_plane, 64, tc::BM, err, errlen)) return -1;
  if (op.b_kmajor) {
    if (!make_tmap_op(&p.tmB, x3, op.B, op.K, op.N, op.ldb, op.b_plane, 64, BN, err, errlen)) return -1;
  } else {
    if (!make_tmap_op(&p.tmB, x3, op.B, op.N, op.K, op.ldb, op.b_plane, 64, 64, err, errlen)) return -1;
  }
  if (!make_tmap_op(&p.tmOut, x3, op.out, op.N, op.M, op.ldo, op.out_plane, 64, 32, err, errlen)) return -1;
  p.M = (int)op.M; p.N = (int)op.N; p.K = (int)op.K;
  p.num_kb = (int)ceil_div(op.K, tc::BK);
  p.tiles_n = (int)ceil_div(op.N, BN);
  p.tiles_m = (int)ceil_div(op.M, tc::BM);
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.b_mn = op.b_kmajor ? 0 : 1;
  p.kind = op.kind; p.act = op.act;
  p.idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)p.b_mn << 16) | ((uint32_t)(BN >> 3) << 17) |
            ((uint32_t)(tc::BM >> 4) << 24);
  p.bias = op.bias;
  p.out_u = (__nv_bfloat16*)op.out_u; p.ldu = op.ldu;
  p.aux = (const __nv_bfloat16*)op.aux; p.ld_aux = op.ld_aux;
  p.err = op.err;
  if (ce_f) {
    p.ce_stats = op.ce_stats; p.ce_zy = op.ce_zy; p.ce_groups = (int)ce_groups(op.N); p.ce_labels = op.ce_labels;
  }
  if (ce_a) {
    p.ce_rowstat = op.ce_rowstat; p.ce_labels = op.ce_labels; p.ce_scale = op.ce_scale;
  }
  // fp32 planes with few tiles: a CTA pair per tile, each half of K (with
  // fewer than three K stages the exchange costs more than the halved loop)
  const bool pair = x3 && 2 * p.num_tiles <= sms && p.num_kb >= 3;
  // B is the larger operand (more columns than rows): walk the row tiles of
  // a column tile first, so B is read from DRAM about once
  p.m_fast = !pair && op.M < op.N ? 1 : 0;
  if (op.relu_bits && op.act == ACT_RELU) {
    if (x3 || pair || op.ld_bits < op.M || ((uintptr_t)op.relu_bits & 7)) {
      snprintf(err, errlen, "ReLU bits: bf16 only, ld_bits >= M, 8-byte aligned");
      return -1;
    }
    p.relu_bits = op.relu_bits; p.ld_bits = op.ld_bits;
  }
  if (op.head_W) {   // the output layer folded into this forward
    if (!pair || op.kind != GEMM_FWD || op.N != tc::kFhK || BN != 128 || !op.head_bias || !op.head_labels ||
        !op.head_ws || (op.act != ACT_RELU && op.act != ACT_NONE) || ((uintptr_t)op.head_W & 15)) {
      snprintf(err, errlen, "folded output layer: fp32-plane forward on CTA pairs, N = 128, ReLU or none, "
                            "16-byte aligned weights");
      return -1;
    }
    p.head_W = op.head_W; p.head_bias = op.head_bias; p.head_labels = op.head_labels;
    p.head_ws = op.head_ws; p.head_loss_off = tc_fused_head_partials(op.M).loss_off; p.head_scale = op.head_scale;
    p.step_counter = op.step_counter; p.bias_corr = op.bias_corr; p.beta1 = op.beta1; p.beta2 = op.beta2;
  }
  LaunchRec& r = recs[0];
  if (pair) {
    r.func = tcpair_kernel_ptr();
    r.smem = tc::PCfg<128, true>::SMEM_BYTES;
  } else if (x3) {
    r.func = tcp_kernel_ptr<128, true>();
    r.smem = tc::PCfg<128, true>::SMEM_BYTES;
  } else if (BN == 256) {
    r.func = tcp_kernel_ptr<256, false>();
    r.smem = tc::PCfg<256>::SMEM_BYTES;
  } else {
    r.func = tcp_kernel_ptr<128, false>();
    r.smem = tc::PCfg<128>::SMEM_BYTES;
  }
  r.grid = dim3(pair ? (unsigned)(2 * p.num_tiles) : (unsigned)(p.num_tiles < sms ? p.num_tiles : sms));
  r.block = dim3(tc::P_THREADS);
  r.early = true;
  r.name = op.head_W ? "tc_gemm_fwd_head" : op.kind == GEMM_FWD ? "tc_gemm_fwd" : "tc_gemm_dgrad";
  r.set_args(p);
  return 1;
}
}  // namespace

bool tc_fused_head_ok(int64_t M, int64_t N, int64_t K, int64_t C) {
  // the CTA-pair condition of tc_persistent_plan for fp32 planes (N = 128:
  // one column tile, so a pair holds whole rows)
  return C == tc::kFhC && N == tc::kFhK && M >= 1 && M <= INT32_MAX && K >= 1 &&
         2 * ceil_div(M, tc::BM) <= device_sms() && ceil_div(K, tc::BK) >= 3;
}

HeadPartials tc_fused_head_partials(int64_t M) {
  const int n = (int)ceil_div(M, tc::BM);   // one per row tile (CTA pair)
  return HeadPartials{n, tc::kFhPitch, (int64_t)n * tc::kFhPitch};
}

int wait_timeout_check_plan(uint32_t* err_dev, uint64_t limit_ns, LaunchRec* rec) {
  const tc::WaitCheckParams q{err_dev, limit_ns};
  rec->func = (const void*)tc::wait_timeout_check_kernel;
  rec->grid = dim3(1);
  rec->block = dim3(1);
  rec->smem = 0;
  rec->name = "wait_timeout_check";
  rec->set_args(q);
  return 1;
}

int tc_gemm_plan(const GemmOp& op, LaunchRec* recs, char* err, size_t errlen) {
  if (op.dtype != DT_BF16 && op.dtype != DT_F32X3) {
    snprintf(err, errlen, "tensor-core GEMM takes bf16 or fp32-as-planes operands");
    return -1;
  }
  if (op.M <= 0 || op.N <= 0 || op.K <= 0 || op.M > INT32_MAX || op.N > INT32_MAX || op.K > INT32_MAX) {
    snprintf(err, errlen, "bad GEMM shape %lld x %lld x %lld", (long long)op.M, (long long)op.N, (long long)op.K);
    return -1;
  }
  if ((op.kind == GEMM_FWD || op.kind == GEMM_DGRAD) && op.a_kmajor && op.N > 16) {
    if (op.dtype == DT_F32X3 && (op.out_u || (op.kind == GEMM_DGRAD && op.act == ACT_GELU_TANH))) {
      snprintf(err, errlen, "fp32 planes: no GELU (its VJP needs the fp32 pre-activation)");
      return -1;
    }
    return tc_persistent_plan(op, recs, err, errlen);
  }
  if (op.kind == GEMM_WGRAD && !op.a_kmajor && !op.b_kmajor) return tc_wgrad_plan(op, recs, err, errlen);
  if (op.dtype == DT_F32X3) {
    snprintf(err, errlen, "fp32 planes: no tensor-core kernel for this GEMM form (N=%lld)", (long long)op.N);
    return -1;
  }
  const int BN = pick_bn(op);
  if (!op.b_kmajor && BN % 64) { snprintf(err, errlen, "MN-major B needs BN %% 64 == 0"); return -1; }
  tc::Params p;
  memset(&p, 0, sizeof(p));
  // A operand: K-major [M rows, K] or MN-major [K rows, M].
  if (op.a_kmajor) {
    if (!make_tmap(&p.tmA, op.A, op.K, op.M, op.lda, 64, 128, err, errlen)) return -1;
  } else {
    if (!make_tmap(&p.tmA, op.A, op.M, op.K, op.lda, 64, 64, err, errlen)) return -1;
  }
  if (op.b_kmajor) {
    if (!make_tmap(&p.tmB, op.B, op.K, op.N, op.ldb, 64, BN, err, errlen)) return -1;
  } else {
    if (!make_tmap(&p.tmB, op.B, op.N, op.K, op.ldb, 64, 64, err, errlen)) return -1;
  }
  p.M = (int)op.M; p.N = (int)op.N; p.K = (int)op.K;
  p.num_kb = (int)ceil_div(op.K, tc::BK);
  p.a_mn = op.a_kmajor ? 0 : 1;
  p.b_mn = op.b_kmajor ? 0 : 1;
  p.kind = op.kind; p.act = op.act;
  p.idesc = (1u << 4)                       // D: f32
          | (1u << 7) | (1u << 10)          // A, B: bf16
          | ((uint32_t)p.a_mn << 15) | ((uint32_t)p.b_mn << 16)
          | ((uint32_t)(BN >> 3) << 17)
          | ((uint32_t)(tc::BM >> 4) << 24);
  p.bias = op.bias;
  p.out = (__nv_bfloat16*)op.out; p.ldo = op.ldo;
  p.out_u = (__nv_bfloat16*)op.out_u; p.ldu = op.ldu;
  p.aux = (const __nv_bfloat16*)op.aux; p.ld_aux = op.ld_aux;
  p.dW = op.dW; p.ld_dw = op.ld_dw;
  p.db = op.db;
  p.err = op.err;
  int splits = 1;
  if (op.kind == GEMM_WGRAD) {
    splits = op.splits > 0 ? op.splits : tc_wgrad_splits(op.M, op.N, op.K);
    if (splits > p.num_kb) splits = p.num_kb;
  }
  p.kb_per_split = (int)ceil_div(p.num_kb, splits);
  splits = (int)ceil_div(p.num_kb, p.kb_per_split);
  if (splits > 1) {
    size_t need = wgrad_workspace_bytes(DT_BF16, op.M, op.N, op.K, splits);
    if (!op.ws || op.ws_bytes < need) {
      snprintf(err, errlen, "wgrad workspace too small (%zu < %zu)", op.ws_bytes, need);
      return -1;
    }
    p.ws = op.ws;
  }
  LaunchRec& r = recs[0];
  switch (BN) {
    case 16: r.func = tc_kernel_ptr<16>(); r.smem = tc::Cfg<16>::SMEM_BYTES; break;
    case 128: r.func = tc_kernel_ptr<128>(); r.smem = tc::Cfg<128>::SMEM_BYTES; break;
    default: r.func = tc_kernel_ptr<256>(); r.smem = tc::Cfg<256>::SMEM_BYTES; break;
  }
  r.grid = dim3((unsigned)ceil_div(op.N, BN), (unsigned)ceil_div(op.M, tc::BM), (unsigned)splits);
  r.block = dim3(tc::NUM_THREADS);
  r.name = op.kind == GEMM_FWD ? "tc_gemm_fwd" : op.kind == GEMM_DGRAD ? "tc_gemm_dgrad" : "tc_gemm_wgrad";
  r.set_args(p);
  if (splits > 1) {
    split_reduce_plan(op.ws, splits, op.M, op.N, op.dW, op.ld_dw, op.db, &recs[1]);
    return 2;
  }
  return 1;
}

int gemm_plan(const GemmOp& op, LaunchRec* recs, char* err, size_t errlen) {
  // fp32 on the FFMA pipes; bf16 and fp32-as-planes on the tensor cores
  return op.dtype == DT_F32 ? simt_gemm_plan(op, recs, err, errlen) : tc_gemm_plan(op, recs, err, errlen);
}

}  // namespace mlpk
