// Fifth-generation tensor-core (tcgen05) building blocks and the passes of
// padded ranks 16 and 32 that use them.
//
// At these ranks every element of M costs 2 RP multiply-adds in pass 1 (the
// lazy residual P_old Q_old^T and the projection Mbar Q) and RP in passes 2
// and 3, against a few bytes of HBM traffic, so on the fp32 pipe the
// arithmetic bounds them.  Here the contractions run as tcgen05.mma
// (kind::tf32, fp32 accumulators in tensor memory), issued by one thread from
// shared-memory descriptors, while the warps only move data.  Near-fp32
// accuracy comes from the split x = hi + lo of both operands (hi keeps the 19
// bits a tf32 operand holds, lo = x - hi exactly): a b ~ hi_a hi_b + hi_a lo_b
// + lo_a hi_b, within about 2^-20 of |a b| per product, accumulated in fp32.
//
// Operand layout: every operand tile is K-major with the 128-byte swizzle --
// rows of 32 fp32 values (128 B), the 16-byte chunk c of row r stored at chunk
// c ^ (r mod 8), 8-row groups 1024 B apart.  The factor operands are written
// once per step in exactly that layout ("images", k_images), so a tile of
// them reaches shared memory with one bulk copy (cp.async.bulk) and no warp
// work; the streamed operand (Mbar) is split and swizzled by the warps.
#pragma once

#include <stdint.h>

#include "psgd_kernels.cuh"

namespace psgd {

// cp.async that fills the destination with zeros when `valid` is false (the
// source address is then not read, but still points into the buffer).
__device__ __forceinline__ void cp_async16_z(void* smem, const void* gmem, bool valid) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async8_z(void* smem, const void* gmem, bool valid) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  const int n = valid ? 8 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}

// The pass-1 items the tensor-core kernel does not take (rows not 16-byte aligned
// in the bucket, or items the bucket does not wholly back): element path.
template <int RP, typename GT>
__global__ void __launch_bounds__(kThreads) k_pass1_rest(const StepArgs a) {
  const int cur = a.ctrl->cur;
  const bool use_init = (!a.warm_start) || (a.ctrl->warm_valid == 0);
  const float* Qc = a.Qf + (long long)cur * a.q_total;
  const float* Pc = a.Pf + (long long)cur * a.p_total;
  const float* Qp = use_init ? a.qinit : Qc;
  int bad = 0;
  for (int it = blockIdx.x; it < a.n_p1items; it += gridDim.x) {
    const Item item = a.p1items[it];
    const TensorDesc td = a.tensors[item.t];
    if (td.vec && a.vec_ok && (long long)(item.row0 + item.nrows) * td.m <= td.valid) continue;
    pass1_tile<RP, 0, GT, 1, 1>(a, td, item, Qp, Qc, Pc, cur, bad);
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(&a.ctrl->flag, 1);
}

namespace tc {

// Iterations of a bounded mbarrier wait before it gives up (each try_wait
// may itself suspend the thread for a while): far beyond any normal wait.
constexpr long kWaitIters = 1L << 22;

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Shared-memory matrix descriptor: K-major operand with the 128-byte swizzle
// starting at shared address `a` (16-byte units), 8-row groups 1024 B apart
// (stride byte offset), descriptor version 1, layout type 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t sdesc(uint32_t a) {
  return (uint64_t)((a >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::tf32: fp32 accumulator (bits 4-5 = 1), A and
// B tf32 (bits 7-9 and 10-12 = 2), both K-major, N / 8 at bit 17, M / 16 at
// bit 24.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (tensor memory) = A B^T (+ D when acc), one K = 8 step.
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
               "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// D (tensor memory) = A B^T (+ D when acc) with A in tensor memory (lane =
// row, one column per K element), one K = 8 step.
__device__ __forceinline__ void mma_ta(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
               "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}"
               ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

// 16 consecutive fp32 columns into tensor-memory lane (warp's lane quarter +
// lane id) starting at address `t`; complete after tmem_wait_st().
__device__ __forceinline__ void tmem_st16(uint32_t t, const float (&v)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
               "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
               ::"r"(t), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                 "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
                 "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                 "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
                 "r"(__float_as_uint(v[15]))
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// The mbarrier receives one arrival when every tcgen05 operation this thread
// issued so far has completed.
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(saddr(bar)) : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy shared-memory writes made visible to the tensor core (async proxy)
__device__ __forceinline__ void fence_smem_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void bar_init(uint64_t* bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count));
}
__device__ __forceinline__ void bar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// Waits until the phase of parity `parity` has completed; false if the bound
// ran out first.
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity) {
  for (long it = 0; it < kWaitIters; ++it) {
    uint32_t ok;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok) : "r"(saddr(bar)), "r"(parity) : "memory");
    if (ok) return true;
  }
  return false;
}

// One arrival that also announces `bytes` of bulk copies completing on the barrier.
__device__ __forceinline__ void bar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)), "r"(bytes) : "memory");
}

// Bulk copy global -> shared of `bytes` (multiple of 16, both 16-byte
// aligned), completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(saddr(dst)), "l"(src), "r"(bytes), "r"(saddr(bar)) : "memory");
}

// 32 consecutive fp32 columns of tensor-memory lane (warp's lane quarter +
// lane id), starting at address `t`.
__device__ __forceinline__ void tmem_ld32(uint32_t t, float (&v)[32]) {
  uint32_t r[32];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
               "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
               "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                 "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
                 "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
                 "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(t));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// tmem_ld32 without the wait: the registers are valid after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t t, float (&v)[32]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
               "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
               "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                 "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
                 "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
                 "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(t));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 16 consecutive fp32 columns (as tmem_ld32).
__device__ __forceinline__ void tmem_ld16(uint32_t t, float (&v)[16]) {
  uint32_t r[16];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
               "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                 "=r"(r[14]), "=r"(r[15])
               : "r"(t));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Tensor-memory allocation by one whole warp: `cols` columns (a power of two
// >= 32), address written to *slot; the permit is released right away so
// other CTAs on the SM can allocate.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(slot)), "r"(cols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_free(uint32_t t, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(t), "r"(cols));
}

// The tf32 part of x: sign, exponent and the top 10 mantissa bits.
__device__ __forceinline__ float hi_part(float x) { return __uint_as_float(__float_as_uint(x) & 0xffffe000u); }

// Float index of element (r, k), k < 32, in a swizzled K-major image whose
// rows are r (the image starts at a 1024-byte boundary, so r's group of 8 is
// the swizzle group).
__host__ __device__ __forceinline__ int swz(int r, int k) { return r * 32 + ((((k >> 2) ^ (r & 7))) << 2) + (k & 3); }

// Records a wait that gave up: the step reports PSGD_ETIMEOUT and is not committed.
__device__ __forceinline__ void timed_out(const StepArgs& a) { atomicExch(&a.ctrl->timeout, 1); }

}  // namespace tc

// Writers of one factor value x = X(r, k) into the operand images (hi and lo
// halves; layouts below, at k_images).  P: its row image and, when `chunk`,
// its chunk image.  Q (r = the column index): its row image or its chunk image.
template <int RP>
__device__ __forceinline__ void img_put_p(const StepArgs& a, const TensorDesc& td, long long r, int k, float x,
                                          bool chunk) {
  const float h = tc::hi_part(x), l = x - h;
  const long long rpad = (td.n + 127) / 128 * 128;
  const long long o = td.pi_off + tc::swz((int)r, k);
  a.img[o] = h;
  a.img[o + rpad * 32] = l;
  if (chunk) {
    const long long c = td.pti_off + (r >> 5) * 2 * RP * 32 + tc::swz(k, (int)(r & 31));
    a.img[c] = h;
    a.img[c + RP * 32] = l;
  }
}
template <int RP>
__device__ __forceinline__ void img_put_q(const StepArgs& a, const TensorDesc& td, long long r, int k, float x,
                                          bool chunk) {
  const float h = tc::hi_part(x), l = x - h;
  if (!chunk) {
    const long long rpad = (td.m + 127) / 128 * 128;
    const long long o = td.qi_off + tc::swz((int)r, k);
    a.img[o] = h;
    a.img[o + rpad * 32] = l;
  } else {
    const long long c = td.qti_off + (r >> 5) * 2 * RP * 32 + tc::swz(k, (int)(r & 31));
    a.img[c] = h;
    a.img[c + RP * 32] = l;
  }
}

// ---------------------------------------------------------------------------
// Operand images of the factors (ranks 16 and 32), hi and lo halves:
//   row image of X (R x RP): rows r of 32 values (zero beyond RP), the layout
//     of an MMA operand with K = rank; blocks of rows are contiguous images.
//     P's row image is the A operand of pass 3 and of pass 1's residual;
//     Q's (rows = the tensor's columns) the B operand of both.
//   chunk image of X: for each 32-row chunk of X, RP rows (one per rank) of
//     the chunk's 32 hi values followed by RP rows of its lo values, the
//     layout of an operand with K = X's rows (hi and lo stacked as one
//     operand of 2 RP rows).
//     P's chunk image is the B operand of pass 2 (K = the tensor's rows);
//     Q's the B operand of pass 1's projection (K = the tensor's columns).
// mode 0: P row and chunk images from the factors just orthogonalised (next
//         half); mode 1: Q row and chunk images from the next half's Q (the
//         chunk image is the next step's projection operand when that step
//         is warm-started); mode 2: Q chunk image from the projection Q of
//         this step (the fresh orthogonalised draw or the warm Q, decided on
//         the device as pass 1 decides it; launched only when a fresh draw
//         can be the projection Q); mode 3: P row image and Q row and chunk
//         images from the committed half (after the factors were replaced on
//         the host).  Modes 0 and 1 do nothing in a skipped step, so the
//         images keep describing the committed factors.
// ---------------------------------------------------------------------------
template <int RP>
__global__ void __launch_bounds__(kThreads) k_images(const StepArgs a, int mode) {
  // a skipped or timed-out step keeps the committed factors, and the images too
  if ((mode == 0 || mode == 1) && (a.ctrl->flag || a.ctrl->timeout)) return;
  const int cur = a.ctrl->cur;
  const int half = (mode == 3) ? cur : (cur ^ 1);
  const bool do_p = (mode == 0 || mode == 3);
  const bool do_q = (mode != 0);
  const int np = do_p ? a.n_gsp : 0;
  const int nq = do_q ? a.n_gsq : 0;
  const float* Psrc = a.Pf + (long long)half * a.p_total;
  const bool use_init = (!a.warm_start) || (a.ctrl->warm_valid == 0);
  const float* Qsrc = (mode == 2) ? (use_init ? a.qinit : a.Qf + (long long)cur * a.q_total)
                                  : a.Qf + (long long)half * a.q_total;
  for (int it = blockIdx.x; it < np + nq; it += gridDim.x) {
    const bool is_p = it < np;
    const GsItem gi = is_p ? a.gsp_items[it] : a.gsq_items[it - np];
    const TensorDesc td = a.tensors[gi.t];
    for (int idx = threadIdx.x; idx < gi.nrows * RP; idx += kThreads) {
      int r, k;
      float x;
      if (is_p) {   // row-major P: consecutive threads read consecutive values
        r = gi.row0 + idx / RP;
        k = idx % RP;
        x = Psrc[td.p_off + (long long)r * RP + k];
      } else {      // k-major Q: consecutive threads read consecutive columns
        k = idx / gi.nrows;
        r = gi.row0 + idx % gi.nrows;
        x = Qsrc[td.q_off + (long long)k * td.m + r];
      }
      // chunk images: for chunk r / 32, RP rows of hi then RP rows of lo (one
      // stacked operand)
      if (is_p) {
        img_put_p<RP>(a, td, r, k, x, mode == 0);
      } else {
        if (mode != 2) img_put_q<RP>(a, td, r, k, x, false);
        img_put_q<RP>(a, td, r, k, x, true);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Pass 3 on the tensor cores: out = P Q^T ("PowerSGD Hooks" step 3.7) for the
// tensors whose rows are 16-byte aligned in the bucket and which the bucket
// wholly backs.  Work item: 128 rows x 256 columns; each CTA walks a
// contiguous range of items (row block, then column tile).  Warp-specialised,
// with no CTA-wide barrier in the loop:
//   warp 8 (one lane) issues the bulk copies -- the row block of P's image
//     (A, hi and lo, reloaded only when the row block changes) and the 256
//     rows of Q's image for the item (B, two slots, one item ahead) -- and
//     the item's 3 x RP / 8 MMAs (M = 128, N = 256, K = 8; hi hi, hi lo,
//     lo hi) into one of two tensor-memory accumulators;
//   warps 0-7 drain the accumulators: warp w reads lane quarter w mod 4 (32
//     rows) and columns 128 (w / 4) .. + 127 in 32-column pieces, turns each
//     piece around in its own shared-memory buffer (row stride 36:
//     conflict-free) and writes 4 rows x 128 B per store instruction.
// mbarriers: bfull (copy -> MMA), bfree (MMA done -> copy), tfull (MMA done
// -> write-out), tfree (8 warps done -> MMA).  Each is polled by one lane.
// ---------------------------------------------------------------------------
template <int RP>
struct Pass3Tc {
  static constexpr int THREADS = 288;              // 8 write-out warps + 1 copy/MMA warp
  static constexpr int TN = 256;                   // columns per item
  static constexpr int OPA = 128 * 128;            // one half (hi or lo) of the A block
  static constexpr int OPB = TN * 128;             // one half of a B tile
  static constexpr int XS = 36;                    // turn-around row stride (floats)
  static constexpr int XW = 32 * XS * 4;           // one warp's turn-around buffer
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = 2 * OPA;            // two slots x (hi, lo)
  static constexpr int X_OFF = B_OFF + 4 * OPB;
  static constexpr int SMEM = X_OFF + 8 * XW + 1024;   // + alignment slack
  static constexpr int TCOLS = 512;                // two 256-column accumulators
  static constexpr uint32_t IDESC = tc::idesc_tf32(128, TN);
};

// Polls `bar` for `parity` on lane 0 only; the whole warp learns the result.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = tc::bar_wait(bar, parity) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <int RP>
__global__ void __launch_bounds__(288, 1) k_pass3_tc(const StepArgs a) {
  using T = Pass3Tc<RP>;
  // a.commit_cnt set (this kernel is the step's only pass-3 launch): the CTA
  // that finishes last commits the step, whichever way it leaves
  if (a.ctrl->flag) {
    if (a.commit_cnt) commit_last(a);
    return;
  }
  const int per = (a.n_t3 + gridDim.x - 1) / gridDim.x;
  const int first = blockIdx.x * per, last = min(a.n_t3, first + per);
  if (first >= last) {
    if (a.commit_cnt) commit_last(a);
    return;
  }
  extern __shared__ unsigned char p3_dsm[];
  __shared__ __align__(8) uint64_t bfull[2], bfree[2], tfull[2], tfree[2], afull, drain;
  __shared__ uint32_t tslot;
  __shared__ volatile int abort_s;
  unsigned char* sm = p3_dsm + (((tc::saddr(p3_dsm) + 1023u) & ~1023u) - tc::saddr(p3_dsm));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::bar_init(&bfull[i], 1);
      tc::bar_init(&bfree[i], 1);
      tc::bar_init(&tfull[i], 1);
      tc::bar_init(&tfree[i], 8);
    }
    tc::bar_init(&afull, 1);
    tc::bar_init(&drain, 1);
    tc::bar_init_fence();
    abort_s = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tslot, T::TCOLS);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tslot;
  const int n = last - first;

  if (warp == 8) {
    // ---------------- copies and MMAs (one lane)
    if (lane == 0) {
      unsigned char* A = sm + T::A_OFF;
      int a_t = -1, a_row = -1;
      uint32_t aph = 0u, dph = 0u;
      auto load_b = [&](int li) {
        const Item it = a.t3items[first + li];
        const TensorDesc td = a.tensors[it.t];
        const long long mpad = (td.m + 127) / 128 * 128;
        const int s = li & 1;
        unsigned char* dst = sm + T::B_OFF + s * 2 * T::OPB;
        // rows past mpad (a narrow last tile) are not copied; their MMA
        // columns are never written out
        const long long rows = min((long long)T::TN, mpad - it.col0);
        tc::bar_expect_tx(&bfull[s], (uint32_t)(2 * rows * 128));
        tc::bulk_g2s(dst, a.img + td.qi_off + (long long)it.col0 * 32, (uint32_t)(rows * 128), &bfull[s]);
        tc::bulk_g2s(dst + T::OPB, a.img + td.qi_off + mpad * 32 + (long long)it.col0 * 32,
                     (uint32_t)(rows * 128), &bfull[s]);
      };
      load_b(0);
      bool ok = true;
      for (int li = 0; li < n && ok; ++li) {
        const Item it = a.t3items[first + li];
        const TensorDesc td = a.tensors[it.t];
        // item li + 1's Q image into the slot item li - 1 used
        if (li + 1 < n) {
          if (li >= 1) ok = tc::bar_wait(&bfree[(li + 1) & 1], ((li - 1) >> 1) & 1);
          if (ok) load_b(li + 1);
        }
        if (ok && (it.t != a_t || it.row0 != a_row)) {
          // every MMA issued so far has to finish before A is replaced
          tc::commit(&drain);
          ok = tc::bar_wait(&drain, dph);
          dph ^= 1u;
          if (ok) {
            const long long npad = (td.n + 127) / 128 * 128;
            tc::bar_expect_tx(&afull, 2 * T::OPA);
            tc::bulk_g2s(A, a.img + td.pi_off + (long long)it.row0 * 32, T::OPA, &afull);
            tc::bulk_g2s(A + T::OPA, a.img + td.pi_off + npad * 32 + (long long)it.row0 * 32, T::OPA, &afull);
            ok = tc::bar_wait(&afull, aph);
            aph ^= 1u;
            a_t = it.t;
            a_row = it.row0;
          }
        }
        const int s = li & 1;
        if (ok) ok = tc::bar_wait(&bfull[s], (li >> 1) & 1);
        if (ok && li >= 2) ok = tc::bar_wait(&tfree[s], ((li - 2) >> 1) & 1);
        if (ok) {
          tc::fence_after();
          const uint32_t ahi = tc::saddr(A), alo = ahi + T::OPA;
          const uint32_t bhi = tc::saddr(sm + T::B_OFF + s * 2 * T::OPB), blo = bhi + T::OPB;
          const uint32_t d = tmem + (uint32_t)(s * T::TN);
          uint32_t acc = 0u;
#pragma unroll
          for (int term = 0; term < 3; ++term) {
            const uint32_t ta = term == 2 ? alo : ahi;
            const uint32_t tb = term == 1 ? blo : bhi;
#pragma unroll
            for (int ks = 0; ks < RP / 8; ++ks) {
              tc::mma(d, tc::sdesc(ta + ks * 32), tc::sdesc(tb + ks * 32), T::IDESC, acc);
              acc = 1u;
            }
          }
          tc::commit(&bfree[s]);
          tc::commit(&tfull[s]);
        }
      }
      if (!ok) {
        abort_s = 1;
        tc::timed_out(a);
      }
      // nothing may still write shared or tensor memory when the CTA ends
      tc::commit(&drain);
      tc::bar_wait(&drain, dph);
    }
  } else {
    // ---------------- write-out (warps 0-7)
    const int wq = warp & 3, hf = warp >> 2;
    float* xb = reinterpret_cast<float*>(sm + T::X_OFF + warp * T::XW);
    for (int li = 0; li < n; ++li) {
      const int s = li & 1;
      // the item's fields are read while its MMAs run
      const Item it = a.t3items[first + li];
      const TensorDesc td = a.tensors[it.t];
      const bool ok = !abort_s && warp_wait(&tfull[s], (li >> 1) & 1);
      if (!ok) {
        if (lane == 0) {
          abort_s = 1;
          tc::timed_out(a);
        }
        break;
      }
      tc::fence_after();
      float* out = a.out + td.g_off;
      // the warp's 128 columns in four 32-column loads, issued before one wait
      float v[4][32];
      const uint32_t tb = tmem + (uint32_t)(s * T::TN + hf * 128) + ((uint32_t)(32 * wq) << 16);
#pragma unroll
      for (int pc = 0; pc < 4; ++pc) tc::tmem_ld32_nowait(tb + pc * 32, v[pc]);
      tc::tmem_wait_ld();
#pragma unroll
      for (int pc = 0; pc < 4; ++pc) {
        const int cb = hf * 128 + pc * 32;
        if (cb >= it.ncols) break;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(xb + lane * T::XS + 4 * q) =
              make_float4(v[pc][4 * q], v[pc][4 * q + 1], v[pc][4 * q + 2], v[pc][4 * q + 3]);
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int rr = 4 * q + (lane >> 3), c4 = lane & 7;
          const int row = 32 * wq + rr, col = cb + 4 * c4;
          const float4 x = *reinterpret_cast<const float4*>(xb + rr * T::XS + 4 * c4);
          if (row < it.nrows && col < it.ncols)
            st_stream4(out + (long long)(it.row0 + row) * td.m + it.col0 + col, x);
        }
        __syncwarp();
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::saddr(&tfree[s])) : "memory");
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 0) tc::tmem_free(tmem, T::TCOLS);
  if (a.commit_cnt) commit_last(a);
}

// ---------------------------------------------------------------------------
// Pass 2 on the tensor cores: the partial Q' = Mbar^T P of one row block
// ("PowerSGD Hooks" steps 3.5-3.6, the replica mean folded), same partial
// layout as k_pass2 (qpart[rb][k][j]).  As an MMA, D (128 columns x RP) =
// A (columns x rows) B^T with B = P^T (ranks x rows): K runs over the rows,
// 32 at a time.  Work item: one row block x 128 columns; a CTA walks a
// contiguous range of items chunk by chunk.  Warp-specialised:
//   warps 0-7 (workers): warp w owns columns 32 (w mod 4) .. + 31 and rows
//     16 (w / 4) .. + 15 of every chunk.  It stages that piece of the source
//     (the Mbar scratch, or the store halves of W <= 2 replicas, whose mean is
//     taken here) in its own cp.async ring, S - 1 chunks ahead, then each lane
//     (one column) splits its 16 values into hi and lo and stores them into
//     its column's tensor-memory lane (A lives in tensor memory: lane = the
//     column, one tensor-memory column per row of the chunk), so the split
//     operand costs no shared-memory bandwidth;
//   warp 12 (one lane) bulk-copies P's chunk images (four chunks ahead, six
//     slots: a copy from L2 takes longer than a chunk's work) and issues the
//     chunk's MMAs.  P's chunk image stacks hi over lo (2 RP rows), so per
//     K = 8 step two MMAs do the three products: A_hi x [P_hi; P_lo] fills
//     accumulator columns [0, 2 RP) with (hi hi | hi lo), A_lo x P_hi adds
//     lo hi into [0, RP); the write-out adds the two halves.  Few, wide MMAs
//     matter: one lane issuing them is the kernel's critical path;
//   warps 8-11 write the finished accumulator of an item to qpart.
// mbarriers: aready (8 workers -> MMA), afree (MMA done -> workers, and the
// MMA lane's own P-slot reuse), pfull (copy -> MMA), tfull (MMA -> write-out),
// tfree (4 warps -> MMA).  A images and accumulators are double-buffered.
// Item fields are read once per item and kept in registers.
// ---------------------------------------------------------------------------
template <int RP, int NSRC>
struct Pass2Tc {
  static constexpr int THREADS = 416;               // 8 workers, 4 write-out warps, 1 MMA warp
  static constexpr int KR = 32;                     // rows per chunk (one K atom)
  static constexpr int S = NSRC == 1 ? 6 : 3;       // workers' ring depth (chunks)
  static constexpr int NP = 6;                      // P image slots
  static constexpr int PD = 4;                      // chunks a P image is copied ahead
  static constexpr int WPIECE = 16 * 32 * 4;        // one worker's piece of one source: 16 rows x 32 columns
  static constexpr int WRING = S * NSRC * WPIECE;   // one worker's ring
  static constexpr int OPB = 2 * RP * 128;          // one stacked P chunk image (hi over lo)
  static constexpr int B_OFF = 0;                   // NP slots
  static constexpr int R_OFF = B_OFF + NP * OPB;    // 8 worker rings
  static constexpr int SMEM = R_OFF + 8 * WRING + 1024;
  static constexpr int DC = 2 * RP;                 // accumulator columns per item
  static constexpr int A_COL = 2 * DC;              // tensor-memory column of A: 2 buffers x (hi 32, lo 32)
  static constexpr int TCOLS = 256;
  static constexpr uint32_t IDESC_W = tc::idesc_tf32(128, 2 * RP);
  static constexpr uint32_t IDESC_N = tc::idesc_tf32(128, RP);
};

// The fields of a pass-2 item its consumers need, read once per item.
struct Tc2Item {
  int row0, nrows, col0, ncols, rb, nch;
  long long base;   // mode-dependent source offset of the tensor (c_off)
  long long ld, m, pti_off, qp_off;
};

__device__ __forceinline__ Tc2Item tc2_item(const StepArgs& a, int i) {
  const Item it = a.t2items[i];
  const TensorDesc td = a.tensors[it.t];
  Tc2Item r;
  r.row0 = it.row0;
  r.nrows = it.nrows;
  r.col0 = it.col0;
  r.ncols = it.ncols;
  r.rb = it.rb;
  r.nch = (it.nrows + 31) / 32;
  r.base = td.c_off;
  r.ld = td.ld;
  r.m = td.m;
  r.pti_off = td.pti_off;
  r.qp_off = td.qp_off;
  return r;
}

template <int RP, int NSRC>
__global__ void __launch_bounds__(416, 1) k_pass2_tc(const StepArgs a, int src_mode) {
  using T = Pass2Tc<RP, NSRC>;
  if (a.ctrl->flag) return;
  const int per = (a.n_t2 + gridDim.x - 1) / gridDim.x;
  const int first = blockIdx.x * per, last = min(a.n_t2, first + per);
  if (first >= last) return;
  extern __shared__ unsigned char p2_dsm[];
  __shared__ __align__(8) uint64_t aready[2], afree[2], pfull[T::NP], tfull[2], tfree[2], drain;
  __shared__ uint32_t tslot;
  __shared__ volatile int abort_s;
  unsigned char* sm = p2_dsm + (((tc::saddr(p2_dsm) + 1023u) & ~1023u) - tc::saddr(p2_dsm));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::bar_init(&aready[i], 8);
      tc::bar_init(&afree[i], 1);
      tc::bar_init(&tfull[i], 1);
      tc::bar_init(&tfree[i], 4);
    }
    for (int i = 0; i < T::NP; ++i) tc::bar_init(&pfull[i], 1);
    tc::bar_init(&drain, 1);
    tc::bar_init_fence();
    abort_s = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tslot, T::TCOLS);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tslot;
  const int nxt = a.ctrl->cur ^ 1;
  // source row i of an item's tensor: the Mbar scratch, or replica w's store (next half)
  const float* src0 = (src_mode == 0) ? a.mbar : a.estore + (long long)nxt * a.est_half;

  if (warp < 8) {
    // ---------------- workers
    const int cq = warp & 3, h = warp >> 2;
    unsigned char* ring = sm + T::R_OFF + warp * T::WRING;
    int l_i = first, l_ch = 0;
    Tc2Item l_it = tc2_item(a, first);
    auto issue = [&](int slot) {   // the load cursor's chunk: this warp's 16 rows x 32 columns
      if (l_i < last) {
        const int r0 = l_it.row0 + l_ch * T::KR + 16 * h;
        const int rend = l_it.row0 + l_it.nrows;
        const long long col = l_it.col0 + 32 * cq + 4 * (lane & 7);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int rr = 4 * q + (lane >> 3);
          const bool ok = (r0 + rr < rend) && (col < l_it.ld);
          const long long off = l_it.base + (ok ? (long long)(r0 + rr) * l_it.ld + col : 0);
#pragma unroll
          for (int w = 0; w < NSRC; ++w)
            cp_async16_z(ring + (slot * NSRC + w) * T::WPIECE + rr * 128 + (lane & 7) * 16,
                         src0 + (long long)w * a.nc_pad + off, ok);
        }
        if (++l_ch == l_it.nch) {
          l_ch = 0;
          if (++l_i < last) l_it = tc2_item(a, l_i);
        }
      }
      cp_async_commit();
    };
    for (int j = 0; j < T::S - 1; ++j) issue(j);
    int k = 0;
    for (int i = first; i < last && !abort_s; ++i) {
      const int nch = (a.t2items[i].nrows + T::KR - 1) / T::KR;
      for (int c = 0; c < nch; ++c, ++k) {
        cp_async_wait<T::S - 2>();
        __syncwarp();
        issue((k + T::S - 1) % T::S);
        if (k >= 2 && !warp_wait(&afree[k & 1], ((k - 2) >> 1) & 1)) {
          if (lane == 0) {
            abort_s = 1;
            tc::timed_out(a);
          }
          break;
        }
        const unsigned char* piece = ring + (k % T::S) * NSRC * T::WPIECE;
        float hv[16], lv[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
          float v = reinterpret_cast<const float*>(piece + rr * 128)[lane];
          if (NSRC == 2) v = (v + reinterpret_cast<const float*>(piece + T::WPIECE + rr * 128)[lane]) * a.invW;
          hv[rr] = tc::hi_part(v);
          lv[rr] = v - hv[rr];
        }
        const uint32_t abase = tmem + (uint32_t)(T::A_COL + (k & 1) * 64 + 16 * h) + ((uint32_t)(32 * cq) << 16);
        tc::tmem_st16(abase, hv);
        tc::tmem_st16(abase + 32, lv);
        tc::tmem_wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::saddr(&aready[k & 1])) : "memory");
      }
    }
    cp_async_wait<0>();
  } else if (warp < 12) {
    // ---------------- write-out of finished accumulators (lane quarter warp - 8)
    const int q = warp - 8;
    for (int i = first, li = 0; i < last; ++i, ++li) {
      const Tc2Item it = tc2_item(a, i);   // read while the item is being computed
      const bool ok = !abort_s && warp_wait(&tfull[li & 1], (li >> 1) & 1);
      if (!ok) {
        if (lane == 0) {
          abort_s = 1;
          tc::timed_out(a);
        }
        break;
      }
      tc::fence_after();
      float v[2 * RP];
      const uint32_t taddr = tmem + (uint32_t)((li & 1) * T::DC) + ((uint32_t)(32 * q) << 16);
      if constexpr (RP == 32) {
        float* v0 = v;
        float* v1 = v + 32;
        tc::tmem_ld32_nowait(taddr, *reinterpret_cast<float(*)[32]>(v0));
        tc::tmem_ld32_nowait(taddr + 32, *reinterpret_cast<float(*)[32]>(v1));
        tc::tmem_wait_ld();
      } else {
        tc::tmem_ld32(taddr, v);
      }
      const int c = 32 * q + lane;
      if (c < it.ncols) {
        float* dst = a.qpart + it.qp_off + (long long)it.rb * RP * it.m + it.col0 + c;
#pragma unroll
        for (int kk = 0; kk < RP; ++kk) dst[(long long)kk * it.m] = v[kk] + v[RP + kk];
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::saddr(&tfree[li & 1])) : "memory");
    }
  } else if (lane == 0) {
    // ---------------- P images and MMAs (warp 12, one lane)
    // chunk k + PD's P image goes into the slot of chunk k + PD - NP, whose
    // MMAs (chunk k - 2) are known done at chunk k
    static_assert(T::PD == T::NP - 2, "slot reuse distance");
    int n_i = first, n_ch = 0, n_k = 0;   // the next chunk whose P image is copied
    Tc2Item n_it = tc2_item(a, first);
    auto next_p = [&]() {
      const long long ch = (n_it.row0 + n_ch * T::KR) / 32;
      const int b = n_k % T::NP;
      tc::bar_expect_tx(&pfull[b], T::OPB);
      tc::bulk_g2s(sm + T::B_OFF + b * T::OPB, a.img + n_it.pti_off + ch * 2 * RP * 32, T::OPB, &pfull[b]);
      ++n_k;
      if (++n_ch == n_it.nch) {
        n_ch = 0;
        if (++n_i < last) n_it = tc2_item(a, n_i);
      }
    };
    while (n_i < last && n_k < T::PD) next_p();
    bool ok = true;
    int k = 0;
    uint32_t dph = 0u;
    int nch = (a.t2items[first].nrows + T::KR - 1) / T::KR;
    for (int i = first, li = 0; i < last && ok; ++i, ++li) {
      const int nch_next = (i + 1 < last) ? (a.t2items[i + 1].nrows + T::KR - 1) / T::KR : 0;
      for (int c = 0; c < nch && ok; ++c, ++k) {
        if (n_i < last) {
          if (k >= 2) ok = tc::bar_wait(&afree[k & 1], ((k - 2) >> 1) & 1);
          if (!ok) break;
          next_p();
        }
        ok = tc::bar_wait(&aready[k & 1], (k >> 1) & 1);
        if (ok && c == 0 && li >= 2) ok = tc::bar_wait(&tfree[li & 1], ((li - 2) >> 1) & 1);
        if (ok) ok = tc::bar_wait(&pfull[k % T::NP], (k / T::NP) & 1);
        if (!ok) break;
        tc::fence_after();
        const uint32_t ahi = tmem + (uint32_t)(T::A_COL + (k & 1) * 64), alo = ahi + 32;
        const uint32_t bst = tc::saddr(sm + T::B_OFF + (k % T::NP) * T::OPB);   // [hi; lo], 2 RP rows
        const uint32_t d = tmem + (uint32_t)((li & 1) * T::DC);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          tc::mma_ta(d, ahi + ks * 8, tc::sdesc(bst + ks * 32), T::IDESC_W, (c == 0 && ks == 0) ? 0u : 1u);
          tc::mma_ta(d, alo + ks * 8, tc::sdesc(bst + ks * 32), T::IDESC_N, 1u);
        }
        tc::commit(&afree[k & 1]);
        if (c == nch - 1) tc::commit(&tfull[li & 1]);
      }
      nch = nch_next;
    }
    if (!ok) {
      abort_s = 1;
      tc::timed_out(a);
    }
    tc::commit(&drain);
    tc::bar_wait(&drain, dph);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 0) tc::tmem_free(tmem, T::TCOLS);
}

// ---------------------------------------------------------------------------
// Pass 1 on the tensor cores (ranks 16 and 32): error feedback, unscale,
// replica mean and the projection P_raw = Mbar Q ("PowerSGD Hooks" steps
// 3.2-3.3 with the error feedback of the hook's warning), for the items whose
// rows are 16-byte aligned in the bucket and which the bucket wholly backs.
// Item: 128 rows x a 512-column tile, walked in 32-column chunks; each chunk
// is W units (one per replica).  Per chunk two contractions run as MMAs:
//   correction  C = P_old Q_old^T for the chunk (M = 128 rows, N = 32
//               columns, K = RP): A = the item's rows of P_old's row image
//               (shared memory), B = Q_old's row image for the 32 columns,
//               hi stacked over lo (N = 64): A_hi x [Q_hi; Q_lo] gives
//               (hi hi | hi lo), A_lo x Q_hi adds lo hi to the first half;
//   projection P += Mbar Q_chunk (M = 128 rows, N = RP, K = 32 columns): A =
//               Mbar hi and lo in tensor memory, B = the chunk image of this
//               step's projection Q, hi stacked over lo, the same two MMAs.
// Warp-specialised:
//   warps 0-7 (workers): warp w owns rows 32 (w mod 4) .. + 31 and columns
//     16 (w / 4) .. + 15 of every chunk; lane = row.  It stages its piece of
//     every replica's gradient and store with cp.async in its own ring (rows
//     padded to 80 or 48 bytes: conflict-free), reads the correction from
//     tensor memory, forms M_w = g_w s + (store_w - C), writes M_w to the next
//     half of the store (turned around in shared memory so 4 lanes write 64
//     contiguous bytes of a row), sums Mbar, and stores its hi and lo into
//     tensor memory;
//   warp 8 (one lane) bulk-copies the operand images and issues the MMAs:
//     the correction two chunks ahead, the projection as soon as the workers
//     have stored Mbar;
//   warps 9-12 write each item's P partial (lanes = rows) to praw_part.
// Tensor memory: correction accumulators (2 x 64 columns), projection
// accumulators (2 items x 2 RP), Mbar operand (2 chunks x (hi 32, lo 32)).
// ---------------------------------------------------------------------------
template <int RP, typename GT>
struct Pass1Tc {
  static constexpr int THREADS = 416;               // 8 workers, 1 MMA warp, 4 write-out warps
  static constexpr int GB = (int)sizeof(GT);
  static constexpr int GROW = GB == 4 ? 80 : 48;    // staged gradient row: 16 values + 16 B pad
  static constexpr int EROW = 80;                   // staged store row
  static constexpr int UNIT = 32 * (GROW + EROW);   // one worker's piece of one unit
  static constexpr int S = GB == 4 ? 2 : 3;         // worker ring depth (units)
  static constexpr int WRING = S * UNIT;
  static constexpr int OPA = 128 * 128;             // one half of the P_old block
  static constexpr int CB = 64 * 128;               // stacked correction B (Q_old rows hi; lo)
  static constexpr int PB = 2 * RP * 128;           // stacked projection B (Q chunk hi; lo)
  static constexpr int NB = 4;                      // B slots (chunks)
  static constexpr int A1_OFF = 0;                  // 2 item buffers x (hi, lo)
  static constexpr int B_OFF = A1_OFF + 4 * OPA;
  static constexpr int R_OFF = B_OFF + NB * (CB + PB);
  static constexpr int SMEM = R_OFF + 8 * WRING + 1024;
  static constexpr int D1 = 0;                      // correction: 2 x 64 columns
  static constexpr int D2 = 128;                    // projection: 2 x 2 RP columns
  static constexpr int A2 = D2 + 4 * RP;            // Mbar: 2 x (hi 32, lo 32)
  static constexpr int TCOLS = 512;
  static constexpr uint32_t IDESC_C64 = tc::idesc_tf32(128, 64);
  static constexpr uint32_t IDESC_C32 = tc::idesc_tf32(128, 32);
  static constexpr uint32_t IDESC_PW = tc::idesc_tf32(128, 2 * RP);
  static constexpr uint32_t IDESC_PN = tc::idesc_tf32(128, RP);
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
  static_assert(A2 + 128 <= TCOLS, "tensor memory");
};

// The fields of a pass-1 item its consumers need.
struct Tc1Item {
  int row0, nrows, col0, ncols, ct, nch;
  long long g_off, c_off, m, ld, n, pi_off, qi_off, qti_off, pp_off;
};

__device__ __forceinline__ Tc1Item tc1_item(const StepArgs& a, int i) {
  const Item it = a.t1items[i];
  const TensorDesc td = a.tensors[it.t];
  Tc1Item r;
  r.row0 = it.row0;
  r.nrows = it.nrows;
  r.col0 = it.col0;
  r.ncols = it.ncols;
  r.ct = it.ct;
  r.nch = (it.ncols + 31) / 32;
  r.g_off = td.g_off;
  r.c_off = td.c_off;
  r.m = td.m;
  r.ld = td.ld;
  r.n = td.n;
  r.pi_off = td.pi_off;
  r.qi_off = td.qi_off;
  r.qti_off = td.qti_off;
  r.pp_off = td.pp_off;
  return r;
}

template <int RP, typename GT>
__global__ void __launch_bounds__(416, 1) k_pass1_tc(const StepArgs a) {
  using T = Pass1Tc<RP, GT>;
  const int per = (a.n_t1 + gridDim.x - 1) / gridDim.x;
  const int first = blockIdx.x * per, last = min(a.n_t1, first + per);
  if (first >= last) return;
  extern __shared__ unsigned char p1_dsm[];
  __shared__ __align__(8) uint64_t d1full[2], a2ready[2], a2free[2], d2full[2], d2free[2], a1full[2],
      bfull[T::NB], drain;
  __shared__ uint32_t tslot;
  __shared__ volatile int abort_s;
  unsigned char* sm = p1_dsm + (((tc::saddr(p1_dsm) + 1023u) & ~1023u) - tc::saddr(p1_dsm));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::bar_init(&d1full[i], 1);
      tc::bar_init(&a2ready[i], 8);
      tc::bar_init(&a2free[i], 1);
      tc::bar_init(&d2full[i], 1);
      tc::bar_init(&d2free[i], 4);
      tc::bar_init(&a1full[i], 1);
    }
    for (int i = 0; i < T::NB; ++i) tc::bar_init(&bfull[i], 1);
    tc::bar_init(&drain, 1);
    tc::bar_init_fence();
    abort_s = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tslot, T::TCOLS);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tslot;
  const int cur = a.ctrl->cur, nxt = cur ^ 1;
  const bool ef = a.ef != 0;
  const int W = a.W;

  if (warp < 8) {
    // ---------------- workers
    const int q = warp & 3, h = warp >> 2;
    unsigned char* ring = sm + T::R_OFF + warp * T::WRING;
    // load cursor over units (item, chunk, replica)
    int l_i = first, l_c = 0, l_w = 0;
    Tc1Item l_it = tc1_item(a, first);
    auto issue = [&](int slot) {
      if (l_i < last) {
        unsigned char* gdst = ring + slot * T::UNIT;
        unsigned char* edst = gdst + 32 * T::GROW;
        const long long col = l_it.col0 + 32 * l_c + 16 * h;   // first column of the piece
        const GT* g = reinterpret_cast<const GT*>(a.grads.p[l_w]) + l_it.g_off;
        // gradient: 16 values per row in pieces of 4 values (16 bytes fp32,
        // 8 bytes for 16-bit values, whose rows are only 8-byte aligned)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int rr = j * 8 + lane / 4, p4 = lane % 4;   // row of the piece; item row 32 q + rr
          const long long cc = col + p4 * 4;
          const bool ok = (32 * q + rr < l_it.nrows) && (cc < l_it.col0 + l_it.ncols);
          const GT* src = g + (ok ? (long long)(l_it.row0 + 32 * q + rr) * l_it.m + cc : 0);
          if constexpr (T::GB == 4)
            cp_async16_z(gdst + rr * T::GROW + p4 * 16, src, ok);
          else
            cp_async8_z(gdst + rr * T::GROW + p4 * 8, src, ok);
        }
        if (ef) {
          const float* e = a.estore + (long long)cur * a.est_half + (long long)l_w * a.nc_pad + l_it.c_off;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int rr = j * 8 + lane / 4, p16 = lane % 4;
            const long long cc = col + p16 * 4;
            const bool ok = (32 * q + rr < l_it.nrows) && (cc < l_it.col0 + l_it.ncols);
            const float* src = e + (ok ? (long long)(l_it.row0 + 32 * q + rr) * l_it.ld + cc : 0);
            cp_async16_z(edst + rr * T::EROW + p16 * 16, src, ok);
          }
        }
        if (++l_w == W) {
          l_w = 0;
          if (++l_c == l_it.nch) {
            l_c = 0;
            if (++l_i < last) l_it = tc1_item(a, l_i);
          }
        }
      }
      cp_async_commit();
    };
    for (int j = 0; j < T::S - 1; ++j) issue(j);
    const float scale = a.scale, invW = a.invW;
    float chk = 0.f;     // inf/NaN detector: 0 * x is 0 unless x is not finite
    int u = 0, k = 0;    // unit, chunk
    bool ok = true;
    for (int i = first; i < last && ok; ++i) {
      const Tc1Item it = tc1_item(a, i);
      const int r = 32 * q + lane;   // row within the item
      for (int c = 0; c < it.nch && ok; ++c, ++k) {
        float corr[16];
        if (ef) {
          // the correction of chunk k (issued two chunks ahead)
          ok = !abort_s && warp_wait(&d1full[k & 1], (k >> 1) & 1);
          if (!ok) break;
          tc::fence_after();
          float c0[16], c1[16];
          const uint32_t tb = tmem + (uint32_t)(T::D1 + (k & 1) * 64 + 16 * h) + ((uint32_t)(32 * q) << 16);
          tc::tmem_ld16(tb, c0);
          tc::tmem_ld16(tb + 32, c1);
#pragma unroll
          for (int j = 0; j < 16; ++j) corr[j] = c0[j] + c1[j];
        }
        float mb[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) mb[j] = 0.f;
        const long long colp = it.col0 + 32 * c + 16 * h;
        for (int w = 0; w < W; ++w, ++u) {
          cp_async_wait<T::S - 2>();
          __syncwarp();
          issue((u + T::S - 1) % T::S);
          unsigned char* gp = ring + (u % T::S) * T::UNIT;
          unsigned char* ep = gp + 32 * T::GROW;
          float gv[16];
          if constexpr (T::GB == 4) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float4 x = *reinterpret_cast<const float4*>(gp + lane * T::GROW + 16 * j);
              gv[4 * j] = x.x; gv[4 * j + 1] = x.y; gv[4 * j + 2] = x.z; gv[4 * j + 3] = x.w;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const uint4 x = *reinterpret_cast<const uint4*>(gp + lane * T::GROW + 16 * j);
              float f[4];
              cvt4<GT>(make_uint2(x.x, x.y), f);
              gv[8 * j] = f[0]; gv[8 * j + 1] = f[1]; gv[8 * j + 2] = f[2]; gv[8 * j + 3] = f[3];
              cvt4<GT>(make_uint2(x.z, x.w), f);
              gv[8 * j + 4] = f[0]; gv[8 * j + 5] = f[1]; gv[8 * j + 6] = f[2]; gv[8 * j + 7] = f[3];
            }
          }
          float mv[16];
          if (ef) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float4 x = *reinterpret_cast<const float4*>(ep + lane * T::EROW + 16 * j);
              mv[4 * j] = gv[4 * j] * scale + (x.x - corr[4 * j]);
              mv[4 * j + 1] = gv[4 * j + 1] * scale + (x.y - corr[4 * j + 1]);
              mv[4 * j + 2] = gv[4 * j + 2] * scale + (x.z - corr[4 * j + 2]);
              mv[4 * j + 3] = gv[4 * j + 3] * scale + (x.w - corr[4 * j + 3]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) mv[j] = gv[j] * scale;
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            chk += 0.f * (gv[j] * scale);
            mb[j] += mv[j];
          }
          if (ef) {
            // M_w into the next half of the store: turned around through the
            // store piece (4 lanes per row, 64 contiguous bytes)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<float4*>(ep + lane * T::EROW + 16 * j) =
                  make_float4(mv[4 * j], mv[4 * j + 1], mv[4 * j + 2], mv[4 * j + 3]);
            __syncwarp();
            float* en = a.estore + (long long)nxt * a.est_half + (long long)w * a.nc_pad + it.c_off;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int rr = j * 8 + lane / 4, p16 = lane % 4;
              const long long cc = colp + p16 * 4;
              if (32 * q + rr < it.nrows && cc < it.col0 + it.ncols)
                st_stream4(en + (long long)(it.row0 + 32 * q + rr) * it.ld + cc,
                           *reinterpret_cast<const float4*>(ep + rr * T::EROW + p16 * 16));
            }
            __syncwarp();
          }
        }
        if (W > 1) {
#pragma unroll
          for (int j = 0; j < 16; ++j) mb[j] *= invW;
        }
        if (a.mbar) {
          // Mbar (pass 2's source) turned around through the last unit's store piece
          unsigned char* gp = ring + ((u - 1) % T::S) * T::UNIT + 32 * T::GROW;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<float4*>(gp + lane * 80 + 16 * j) = make_float4(mb[4 * j], mb[4 * j + 1], mb[4 * j + 2], mb[4 * j + 3]);
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int rr = j * 8 + lane / 4, p16 = lane % 4;
            const long long cc = colp + p16 * 4;
            if (32 * q + rr < it.nrows && cc < it.col0 + it.ncols)
              st_stream4(a.mbar + it.c_off + (long long)(it.row0 + 32 * q + rr) * it.ld + cc,
                         *reinterpret_cast<const float4*>(gp + rr * 80 + p16 * 16));
          }
          __syncwarp();
        }
        // Mbar hi and lo into tensor memory (the projection's A), once the
        // projection two chunks back has read that buffer
        if (k >= 2) {
          ok = !abort_s && warp_wait(&a2free[k & 1], ((k - 2) >> 1) & 1);
          if (!ok) break;
        }
        float hv[16], lv[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float x = (r < it.nrows) ? mb[j] : 0.f;
          hv[j] = tc::hi_part(x);
          lv[j] = x - hv[j];
        }
        const uint32_t ab = tmem + (uint32_t)(T::A2 + (k & 1) * 64 + 16 * h) + ((uint32_t)(32 * q) << 16);
        tc::tmem_st16(ab, hv);
        tc::tmem_st16(ab + 32, lv);
        tc::tmem_wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::saddr(&a2ready[k & 1])) : "memory");
      }
    }
    if (!ok && lane == 0) {
      abort_s = 1;
      tc::timed_out(a);
    }
    cp_async_wait<0>();
    if (__any_sync(0xffffffffu, !(chk == 0.f)) && lane == 0) atomicOr(&a.ctrl->flag, 1);
  } else if (warp == 8) {
    // ---------------- images and MMAs (one lane)
    if (lane == 0) {
      // chunk cursors: B images are copied NB - 1 chunks ahead; the
      // correction is issued two chunks ahead of the projection
      int b_i = first, b_c = 0, b_k = 0;
      Tc1Item b_it = tc1_item(a, first);
      auto load_b = [&]() {   // chunk b_k's Q_old rows (stacked) and Q chunk image into slot b_k % NB
        const int s = b_k % T::NB;
        unsigned char* cb = sm + T::B_OFF + s * (T::CB + T::PB);
        const long long j0 = b_it.col0 + 32 * b_c;
        const long long mpad = (b_it.m + 127) / 128 * 128;
        uint32_t bytes = T::PB;
        if (ef) bytes += T::CB;
        tc::bar_expect_tx(&bfull[s], bytes);
        if (ef) {
          tc::bulk_g2s(cb, a.img + b_it.qi_off + j0 * 32, T::CB / 2, &bfull[s]);
          tc::bulk_g2s(cb + T::CB / 2, a.img + b_it.qi_off + mpad * 32 + j0 * 32, T::CB / 2, &bfull[s]);
        }
        tc::bulk_g2s(cb + T::CB, a.img + b_it.qti_off + (j0 / 32) * 2 * RP * 32, T::PB, &bfull[s]);
        ++b_k;
        if (++b_c == b_it.nch) {
          b_c = 0;
          if (++b_i < last) b_it = tc1_item(a, b_i);
        }
      };
      // P_old blocks: item index -> buffer index & 1
      int a_i = first;
      auto load_a = [&]() {
        const Tc1Item it = tc1_item(a, a_i);
        const int s = (a_i - first) & 1;
        unsigned char* dst = sm + T::A1_OFF + s * 2 * T::OPA;
        const long long npad = (it.n + 127) / 128 * 128;
        tc::bar_expect_tx(&a1full[s], 2 * T::OPA);
        tc::bulk_g2s(dst, a.img + it.pi_off + (long long)it.row0 * 32, T::OPA, &a1full[s]);
        tc::bulk_g2s(dst + T::OPA, a.img + it.pi_off + npad * 32 + (long long)it.row0 * 32, T::OPA, &a1full[s]);
        ++a_i;
      };
      // correction cursor
      int c_i = first, c_c = 0, c_k = 0;
      int c_nch = tc1_item(a, first).nch;
      bool ok = true;
      auto issue_corr = [&]() {   // chunk c_k's correction into D1[c_k & 1]
        const int li = c_i - first;
        const int s = c_k % T::NB;
        if (c_c == 0) {
          // the item's P_old block (a one-chunk item before it can leave this
          // load to here; the buffer's previous item is done by then)
          while (a_i <= c_i) load_a();
          ok = ok && tc::bar_wait(&a1full[li & 1], (li >> 1) & 1);
        }
        ok = ok && tc::bar_wait(&bfull[s], (c_k / T::NB) & 1);
        if (ok) {
          tc::fence_after();
          const uint32_t ahi = tc::saddr(sm + T::A1_OFF + (li & 1) * 2 * T::OPA), alo = ahi + T::OPA;
          const uint32_t bst = tc::saddr(sm + T::B_OFF + s * (T::CB + T::PB));
          const uint32_t d = tmem + (uint32_t)(T::D1 + (c_k & 1) * 64);
#pragma unroll
          for (int ks = 0; ks < RP / 8; ++ks) {
            tc::mma(d, tc::sdesc(ahi + ks * 32), tc::sdesc(bst + ks * 32), T::IDESC_C64, ks == 0 ? 0u : 1u);
            tc::mma(d, tc::sdesc(alo + ks * 32), tc::sdesc(bst + ks * 32), T::IDESC_C32, 1u);
          }
          tc::commit(&d1full[c_k & 1]);
        }
        ++c_k;
        if (++c_c == c_nch) {
          c_c = 0;
          if (++c_i < last) c_nch = tc1_item(a, c_i).nch;
        }
      };
      // prologue: P_old blocks of the first two items, the first NB - 1
      // chunks' B images, the first two corrections
      if (ef) {
        load_a();
        if (a_i < last) load_a();
      }
      while (b_i < last && b_k < T::NB - 1) load_b();
      if (ef) {
        if (c_i < last) issue_corr();
        if (c_i < last) issue_corr();
      }
      int k = 0;
      for (int i = first, li = 0; i < last && ok; ++i, ++li) {
        const int nch = tc1_item(a, i).nch;
        for (int c = 0; c < nch && ok; ++c, ++k) {
          // chunk k - 1's projection done: its B slot takes chunk k + NB - 1,
          // and every earlier MMA (so the P_old buffer of item li - 1) is done
          if (k >= 1) ok = tc::bar_wait(&a2free[(k - 1) & 1], ((k - 1) >> 1) & 1);
          if (!ok) break;
          if (b_i < last) load_b();
          if (ef && c == 0 && li >= 1 && a_i == i + 1 && a_i < last) load_a();   // item li + 1's P_old block
          // the projection of chunk k
          ok = tc::bar_wait(&a2ready[k & 1], (k >> 1) & 1);
          if (ok && c == 0 && li >= 2) ok = tc::bar_wait(&d2free[li & 1], ((li - 2) >> 1) & 1);
          if (ok && !ef) ok = tc::bar_wait(&bfull[k % T::NB], (k / T::NB) & 1);
          if (!ok) break;
          tc::fence_after();
          {
            const uint32_t ahi = tmem + (uint32_t)(T::A2 + (k & 1) * 64), alo = ahi + 32;
            const uint32_t bst = tc::saddr(sm + T::B_OFF + (k % T::NB) * (T::CB + T::PB) + T::CB);
            const uint32_t d = tmem + (uint32_t)(T::D2 + (li & 1) * 2 * RP);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              tc::mma_ta(d, ahi + ks * 8, tc::sdesc(bst + ks * 32), T::IDESC_PW, (c == 0 && ks == 0) ? 0u : 1u);
              tc::mma_ta(d, alo + ks * 8, tc::sdesc(bst + ks * 32), T::IDESC_PN, 1u);
            }
          }
          tc::commit(&a2free[k & 1]);
          if (c == nch - 1) tc::commit(&d2full[li & 1]);
          // the correction two chunks ahead (its D1 buffer was read for chunk k)
          if (ef && c_i < last) issue_corr();
        }
      }
      if (!ok) {
        abort_s = 1;
        tc::timed_out(a);
      }
      tc::commit(&drain);
      tc::bar_wait(&drain, 0);
    }
  } else {
    // ---------------- P partials of finished items (warps 9-12, lane quarter warp mod 4)
    const int q = warp & 3;
    for (int i = first, li = 0; i < last; ++i, ++li) {
      const Tc1Item it = tc1_item(a, i);
      const bool ok = !abort_s && warp_wait(&d2full[li & 1], (li >> 1) & 1);
      if (!ok) {
        if (lane == 0) {
          abort_s = 1;
          tc::timed_out(a);
        }
        break;
      }
      tc::fence_after();
      float v[2 * RP];
      const uint32_t tb = tmem + (uint32_t)(T::D2 + (li & 1) * 2 * RP) + ((uint32_t)(32 * q) << 16);
      if constexpr (RP == 32) {
        tc::tmem_ld32_nowait(tb, *reinterpret_cast<float(*)[32]>(v));
        tc::tmem_ld32_nowait(tb + 32, *reinterpret_cast<float(*)[32]>(v + 32));
        tc::tmem_wait_ld();
      } else {
        tc::tmem_ld32(tb, *reinterpret_cast<float(*)[32]>(v));
      }
      const int r = 32 * q + lane;
      if (r < it.nrows) {
        float* dst = a.praw_part + it.pp_off + ((long long)it.ct * it.n + it.row0 + r) * RP;
#pragma unroll
        for (int kk = 0; kk < RP; kk += 4)
          *reinterpret_cast<float4*>(dst + kk) =
              make_float4(v[kk] + v[RP + kk], v[kk + 1] + v[RP + kk + 1], v[kk + 2] + v[RP + kk + 2],
                          v[kk + 3] + v[RP + kk + 3]);
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::saddr(&d2free[li & 1])) : "memory");
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 0) tc::tmem_free(tmem, T::TCOLS);
}

}  // namespace psgd
