// Pass 1 for padded ranks 16 and 32 ("PowerSGD Hooks", powerSGD_hook steps
// 3.2-3.3 with the error feedback of the hook's warning) on the tensor cores.
//
// At these ranks pass 1 does 2 RP fused multiply-adds per element (RP for
// the lazy residual P_old Q_old^T, RP for the projection Mbar Q) against
// 8 + s_g bytes of HBM per replica, so on the fp32 pipe the arithmetic and
// the shared-memory operand traffic feeding it bound it, not HBM.  Both
// contractions run here on warp-level mma.sync (m16n8k8, tf32 operands, fp32
// accumulation).  Near-fp32 accuracy comes from the three-term split
// x = hi + lo (split_tf32): a b ~ hi_a hi_b + hi_a lo_b + lo_a hi_b, within
// about 2^-20 of |a b| per product.
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

// The items of the tensor-core pass 1: tensors whose rows are 16-byte
// aligned in the bucket, wholly backed by it.  Advances `it` (stepping by the
// grid) to the next such item and loads it.
__device__ __forceinline__ bool next_mma_item(const StepArgs& a, int& it, Item& item, TensorDesc& td) {
  for (; it < a.n_p1items; it += gridDim.x) {
    item = a.p1items[it];
    td = a.tensors[item.t];
    if (td.vec && a.vec_ok && (long long)(item.row0 + item.nrows) * td.m <= td.valid) return true;
  }
  return false;
}


// x = hi + lo: hi keeps the 19 bits a tf32 operand holds (sign, exponent,
// 10 mantissa bits; the rest cleared), lo = x - hi exactly.  The tensor core
// reads lo's top 19 bits too, so each of hi_a hi_b, hi_a lo_b, lo_a hi_b is
// exact in the accumulator up to 2^-21 of |a b|, and the dropped lo_a lo_b is
// below 2^-20 of it.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = __float_as_uint(x) & 0xffffe000u;
  lo = __float_as_uint(__fsub_rn(x, __uint_as_float(hi)));
}

// d += A (16 x 8, row) B (8 x 8, col), tf32 operands, fp32 accumulators.
// Fragment layout (lane = 4 g + c): a0 = A[g][c], a1 = A[g + 8][c],
// a2 = A[g][c + 4], a3 = A[g + 8][c + 4]; b0 = B[c][g], b1 = B[c + 4][g];
// d0 = D[g][2c], d1 = D[g][2c + 1], d2 = D[g + 8][2c], d3 = D[g + 8][2c + 1].
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A fragments of 16 rows of a row-major factor (RP floats a row), split:
// rows r0 + g and r0 + g + 8 (valid flags va, vb; invalid rows read as 0).
template <int RP>
__device__ __forceinline__ void load_afrag(const float* __restrict__ base, long long r0, bool va, bool vb,
                                           uint32_t (&hi)[RP / 8][4], uint32_t (&lo)[RP / 8][4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const float* ra = base + (r0 + g) * RP;
  const float* rb = base + (r0 + g + 8) * RP;
#pragma unroll
  for (int ks = 0; ks < RP / 8; ++ks) {
    const float v0 = va ? __ldg(ra + ks * 8 + c) : 0.f;
    const float v1 = vb ? __ldg(rb + ks * 8 + c) : 0.f;
    const float v2 = va ? __ldg(ra + ks * 8 + c + 4) : 0.f;
    const float v3 = vb ? __ldg(rb + ks * 8 + c + 4) : 0.f;
    split_tf32(v0, hi[ks][0], lo[ks][0]);
    split_tf32(v1, hi[ks][1], lo[ks][1]);
    split_tf32(v2, hi[ks][2], lo[ks][2]);
    split_tf32(v3, hi[ks][3], lo[ks][3]);
  }
}

// acc[n] = (16 rows of P) x (8 columns of Q, block n)^T for NB blocks:
// qb[n][ks][0] = Q(col g of block n, rank 8 ks + c), qb[n][ks][1] = the same
// column at rank 8 ks + c + 4 (raw floats, split here).  Per k step the
// smaller terms go first: lo_P hi_Q, hi_P lo_Q, then hi_P hi_Q; the NB
// accumulator chains are interleaved, each keeping that order.
template <int RP, int NB>
__device__ __forceinline__ void mma_pq(const uint32_t (&ahi)[RP / 8][4], const uint32_t (&alo)[RP / 8][4],
                                       const float (&qb)[NB][RP / 8][2], float (&acc)[NB][4]) {
#pragma unroll
  for (int n = 0; n < NB; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < RP / 8; ++ks) {
    uint32_t bh[NB][2], bl[NB][2];
#pragma unroll
    for (int n = 0; n < NB; ++n) {
      split_tf32(qb[n][ks][0], bh[n][0], bl[n][0]);
      split_tf32(qb[n][ks][1], bh[n][1], bl[n][1]);
    }
#pragma unroll
    for (int n = 0; n < NB; ++n) mma_tf32(acc[n], alo[ks], bh[n][0], bh[n][1]);
#pragma unroll
    for (int n = 0; n < NB; ++n) mma_tf32(acc[n], ahi[ks], bl[n][0], bl[n][1]);
#pragma unroll
    for (int n = 0; n < NB; ++n) mma_tf32(acc[n], ahi[ks], bh[n][0], bh[n][1]);
  }
}

// ---------------------------------------------------------------------------
// The kernel.  Work item: 128 rows x 512 columns of one tensor, walked in
// 32-column chunks; one CTA (16 warps) per SM over a persistent item list.
// Sources are staged with cp.async, S - 1 (chunk, replica) units ahead,
// continuing across items; the Q chunks (shared by the CTA) rotate through
// SQ buffers, published by one CTA barrier per chunk.  Warps 2b and 2b + 1
// own rows 16 b .. 16 b + 15 of the item, each one 16-column half of the
// chunk (their partial P are added at the end of the item):
//   correction  P_old (16 x RP, split once per item) x Q_old chunk^T, two
//               8-column blocks as two accumulator chains (mma_pq).  Pass 3
//               writes out with the fp32 chain of dot_chain, so here the
//               residual store - P_old Q_old^T differs from fl(M_w - out) by
//               the difference of the two roundings of P_old Q_old^T (about
//               2^-20 of the products' magnitude);
//   M_w, Mbar   in the accumulator layout: lane (g, c) holds rows g, g + 8
//               and columns 8 n + 2c, 8 n + 2c + 1 of block n;
//   projection  P_raw (16 x RP) += Mbar half (16 x 16) Q half (16 x RP):
//               the Mbar values a lane holds are its A fragment when k slot c
//               of a block stands for column 2c and slot c + 4 for 2c + 1,
//               and Q's B fragment takes the same column order.
// Staging: each warp copies its own 16 rows x 16 columns of every source into
// its region (row stride 24 floats for fp32, 12 words for 16-bit gradients:
// conflict-free fragment reads), so only the warp synchronises on them; the Q
// chunks (k-major, row stride 40) are shared, behind the chunk barrier.
// ---------------------------------------------------------------------------
constexpr int kThreads1M = 512;   // threads of the tensor-core pass 1 (16 warps)

template <int RP, typename GT>
struct Pass1Mma {
  static_assert(RP == 16 || RP == 32, "tensor-core pass 1 is for ranks 16 and 32");
  static constexpr int NW = kThreads1M / 32;                   // warps
  static constexpr int TR = kRows1High;                        // rows per item (8 row blocks x 16)
  static constexpr int CC = 32;                                // columns per chunk (2 halves x 16)
  static constexpr int GS = sizeof(GT) == 4 ? 24 : 12;         // gradient row stride, 32-bit words
  static constexpr int PB = 4 * (int)sizeof(GT);               // bytes of a 4-column piece
  static constexpr int ES = 24;                                // store row stride, floats
  static constexpr int WG_BYTES = 16 * GS * 4;                 // a warp's gradient region
  static constexpr int WE_BYTES = 16 * ES * 4;                 // a warp's store region
  static constexpr int UNIT_BYTES = NW * (WG_BYTES + WE_BYTES);
  static constexpr int S = (RP == 32 && sizeof(GT) == 4) ? 3 : 4;   // within 227 KB
  static constexpr int SQ = S;
  static constexpr int QS = 40;                                // Q chunk row stride
  static constexpr int QCH_BYTES = RP * QS * 4;
  static constexpr int XCH_BYTES = (NW / 2) * 32 * (RP / 2) * 4;   // item-end exchange of the halves
  static constexpr int SMEM = S * UNIT_BYTES + 2 * SQ * QCH_BYTES + XCH_BYTES;
  static_assert(TR == 16 * (NW / 2), "one 16-row block per warp pair");
  static_assert(RP * 8 <= kThreads1M, "one Q piece per thread");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

template <int RP, typename GT>
__global__ void __launch_bounds__(kThreads1M, 1) k_pass1_mma(const StepArgs a) {
  using T = Pass1Mma<RP, GT>;
  constexpr int S = T::S, SQ = T::SQ, NR = RP / 8;
  extern __shared__ __align__(128) char p1m_smem[];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, g = lane >> 2, c = lane & 3;
  const int rb = warp >> 1, hf = warp & 1;                     // row block, column half
  char* const wsm = p1m_smem + warp * (T::WG_BYTES + T::WE_BYTES);   // + slot * UNIT_BYTES
  char* const qsm = p1m_smem + S * T::UNIT_BYTES;
  float* const xch = reinterpret_cast<float*>(qsm + 2 * SQ * T::QCH_BYTES);

  const int cur = a.ctrl->cur, nxt = cur ^ 1;
  const bool use_init = (!a.warm_start) || (a.ctrl->warm_valid == 0);
  const float* Qc = a.Qf + (long long)cur * a.q_total;
  const float* Pc = a.Pf + (long long)cur * a.p_total;
  const float* Qp = use_init ? a.qinit : Qc;
  const bool ef = a.ef != 0;
  const bool same_q = (Qp == Qc);
  const int pq = (ef && same_q) ? 0 : 1;
  const int W = a.W;
  const bool unit_scale = (a.scale == 1.0f);
  const long long ecur = (long long)cur * W * a.nc_pad;
  const long long enx = (long long)nxt * W * a.nc_pad;

  // ---- issuer
  int i_it = blockIdx.x, i_ch = 0, i_w = 0, i_cs = 0, i_nch = 0, i_slot = 0;
  Item i_item;
  TensorDesc i_td;
  bool i_ok = next_mma_item(a, i_it, i_item, i_td);
  if (i_ok) i_nch = (i_item.ncols + T::CC - 1) / T::CC;
  auto issue = [&]() {
    if (i_ok) {
      char* reg = wsm + i_slot * T::UNIT_BYTES;
      const long long m = i_td.m, ld = i_td.ld;
      const int cend = i_item.col0 + i_item.ncols;
      const int cc0 = i_item.col0 + i_ch * T::CC + 16 * hf;
      const long long rbase = (long long)i_item.row0 + rb * 16;
      const int rlim = i_item.nrows - rb * 16;       // rows of this warp in the item
      const GT* gsrc = reinterpret_cast<const GT*>(a.grads.p[i_w]) + i_td.g_off;
      // 16 rows x 4 pieces of 4 columns (16 bytes fp32, 8 bytes 16-bit)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int pc = lane + 32 * j, row = pc >> 2, q = pc & 3;
        const int col = cc0 + q * 4;
        const bool v = row < rlim && col < cend;
        const GT* src = gsrc + (v ? (rbase + row) * m + col : 0);
        if constexpr (T::PB == 16) cp_async16_z(reg + row * T::GS * 4 + q * 16, src, v);
        else cp_async8_z(reg + row * T::GS * 4 + q * 8, src, v);
      }
      if (ef) {
        const float* esrc = a.estore + ecur + (long long)i_w * a.nc_pad + i_td.c_off;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int pc = lane + 32 * j, row = pc >> 2, q = pc & 3;
          const int col = cc0 + q * 4;
          const bool v = row < rlim && col < cend;
          cp_async16_z(reg + T::WG_BYTES + row * T::ES * 4 + q * 16, esrc + (v ? (rbase + row) * ld + col : 0), v);
        }
      }
      if (i_w == 0 && t < RP * 8) {
        const int k = t >> 3, q = t & 7;
        const int col = i_item.col0 + i_ch * T::CC + q * 4;
        const bool v = col < cend;
        const long long off = i_td.q_off + (long long)k * m + (v ? col : 0);
        char* dst = qsm + (i_cs % SQ) * 2 * T::QCH_BYTES + (k * T::QS + q * 4) * 4;
        if (ef) cp_async16_z(dst, Qc + off, v);
        if (!(ef && same_q)) cp_async16_z(dst + T::QCH_BYTES, Qp + off, v);
      }
      i_slot = (i_slot + 1 == S) ? 0 : i_slot + 1;
      if (++i_w == W) {
        i_w = 0;
        ++i_cs;
        if (++i_ch == i_nch) {
          i_ch = 0;
          i_it += gridDim.x;
          i_ok = next_mma_item(a, i_it, i_item, i_td);
          if (i_ok) i_nch = (i_item.ncols + T::CC - 1) / T::CC;
        }
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int u = 0; u < S - 1; ++u) issue();

  // ---- consumer
  int c_it = blockIdx.x, c_ch = 0, c_w = 0, c_cs = 0, c_nch = 0, c_slot = 0;
  Item item;
  TensorDesc td;
  bool c_ok = next_mma_item(a, c_it, item, td);
  if (c_ok) c_nch = (item.ncols + T::CC - 1) / T::CC;
  uint32_t phi[NR][4], plo[NR][4];      // P_old rows of this warp's row block, split
  float corr[2][4], mb[2][4], pacc[NR][4];
#pragma unroll
  for (int n = 0; n < NR; ++n) pacc[n][0] = pacc[n][1] = pacc[n][2] = pacc[n][3] = 0.f;
  float chk = 0.f;
  bool va = false, vb = false;
  while (c_ok) {
    cp_async_wait<S - 2>();
    if (c_w == 0) __syncthreads();
    else __syncwarp();
    issue();
    const long long ld = td.ld;
    const int cend = item.col0 + item.ncols;
    const int cc0 = item.col0 + c_ch * T::CC + 16 * hf;     // this warp's 16 columns
    const long long r0 = (long long)item.row0 + rb * 16;
    const char* qbuf = qsm + (c_cs % SQ) * 2 * T::QCH_BYTES;
    const float* qcs = reinterpret_cast<const float*>(qbuf);
    if (c_w == 0) {
      if (c_ch == 0) {
        va = rb * 16 + g < item.nrows;
        vb = rb * 16 + g + 8 < item.nrows;
        if (ef) load_afrag<RP>(Pc + td.p_off, r0, va, vb, phi, plo);
      }
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) { corr[n][e] = 0.f; mb[n][e] = 0.f; }
      if (ef) {
        // B fragment of block n: Q_old(col 16 hf + 8 n + g, rank 8 ks + c (+ 4))
        float qb[2][NR][2];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int ks = 0; ks < NR; ++ks) {
            qb[n][ks][0] = qcs[(ks * 8 + c) * T::QS + 16 * hf + n * 8 + g];
            qb[n][ks][1] = qcs[(ks * 8 + c + 4) * T::QS + 16 * hf + n * 8 + g];
          }
        mma_pq<RP, 2>(phi, plo, qb, corr);
      }
    }
    // M_w of this replica in the accumulator layout
    {
      const char* reg = wsm + c_slot * T::UNIT_BYTES;
      float* enxt = a.estore + enx + (long long)c_w * a.nc_pad + td.c_off;
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        const int col = cc0 + n * 8 + 2 * c;
        const bool cv = col < cend;
#pragma unroll
        for (int h = 0; h < 2; ++h) {               // rows g (h = 0) and g + 8 (h = 1)
          const int rl = g + 8 * h;
          float gv[2];
          if constexpr (sizeof(GT) == 4) {
            const float2 x = *reinterpret_cast<const float2*>(reg + rl * T::GS * 4 + (n * 8 + 2 * c) * 4);
            gv[0] = x.x; gv[1] = x.y;
          } else {
            const uint32_t raw = *reinterpret_cast<const uint32_t*>(reg + rl * T::GS * 4 + (n * 4 + c) * 4);
            float2 f;
            if constexpr (std::is_same<GT, __half>::value) f = __half22float2(*reinterpret_cast<const __half2*>(&raw));
            else f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw));
            gv[0] = f.x; gv[1] = f.y;
          }
          float mv[2];
          if (ef) {
            const float2 x = *reinterpret_cast<const float2*>(reg + T::WG_BYTES + rl * T::ES * 4 + (n * 8 + 2 * c) * 4);
            const float ev[2] = {x.x, x.y};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const float v = unit_scale ? gv[u] : gv[u] * a.scale;
              mv[u] = v + (ev[u] - corr[n][2 * h + u]);
            }
            if ((h == 0 ? va : vb) && cv) st_stream2(enxt + (r0 + rl) * ld + col, mv[0], mv[1]);
          } else {
#pragma unroll
            for (int u = 0; u < 2; ++u) mv[u] = unit_scale ? gv[u] : gv[u] * a.scale;
          }
          mb[n][2 * h] += mv[0];
          mb[n][2 * h + 1] += mv[1];
        }
      }
    }
    if (c_w == W - 1) {
      const float* qps = qcs + pq * (T::QCH_BYTES / 4);
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        const int col = cc0 + n * 8 + 2 * c;
        const bool cv = col < cend;
#pragma unroll
        for (int e = 0; e < 4; ++e) mb[n][e] = (cv && (e < 2 ? va : vb)) ? mb[n][e] * a.invW : 0.f;
        if (a.mbar && cv) {
          float* mrow = a.mbar + td.c_off + col;
          if (va) st_stream2(mrow + (r0 + g) * ld, mb[n][0], mb[n][1]);
          if (vb) st_stream2(mrow + (r0 + g + 8) * ld, mb[n][2], mb[n][3]);
        }
      }
      // projection over this warp's 16 columns: k step n = columns 8 n ..
      // 8 n + 7 of the half, slot c <-> 2c, slot c + 4 <-> 2c + 1; rank
      // block nr: B = Q_p(rank 8 nr + g, those columns)
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        uint32_t ahi[4], alo[4];
        split_tf32(mb[n][0], ahi[0], alo[0]);
        split_tf32(mb[n][2], ahi[1], alo[1]);
        split_tf32(mb[n][1], ahi[2], alo[2]);
        split_tf32(mb[n][3], ahi[3], alo[3]);
        uint32_t bh[NR][2], bl[NR][2];
#pragma unroll
        for (int nr = 0; nr < NR; ++nr) {
          const float2 x = *reinterpret_cast<const float2*>(qps + (nr * 8 + g) * T::QS + 16 * hf + n * 8 + 2 * c);
          split_tf32(x.x, bh[nr][0], bl[nr][0]);
          split_tf32(x.y, bh[nr][1], bl[nr][1]);
        }
#pragma unroll
        for (int nr = 0; nr < NR; ++nr) mma_tf32(pacc[nr], alo, bh[nr][0], bh[nr][1]);
#pragma unroll
        for (int nr = 0; nr < NR; ++nr) mma_tf32(pacc[nr], ahi, bl[nr][0], bl[nr][1]);
#pragma unroll
        for (int nr = 0; nr < NR; ++nr) mma_tf32(pacc[nr], ahi, bh[nr][0], bh[nr][1]);
      }
      if (c_ch == c_nch - 1) {
        // end of the item: the two halves' partial P of the row block are
        // added (second half's values through shared memory) and written
        float* xw = xch + (rb * 32 + lane) * (RP / 2);
        if (hf == 1) {
#pragma unroll
          for (int nr = 0; nr < NR; ++nr)
#pragma unroll
            for (int e = 0; e < 4; ++e) xw[nr * 4 + e] = pacc[nr][e];
        }
        __syncthreads();
        if (hf == 0) {
#pragma unroll
          for (int nr = 0; nr < NR; ++nr) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              pacc[nr][e] += xw[nr * 4 + e];
              chk = fmaf(pacc[nr][e], 0.f, chk);
            }
            float* dst = a.praw_part + td.pp_off + ((long long)item.ct * td.n + r0 + g) * RP + nr * 8 + 2 * c;
            if (va) *reinterpret_cast<float2*>(dst) = make_float2(pacc[nr][0], pacc[nr][1]);
            if (vb) *reinterpret_cast<float2*>(dst + 8 * RP) = make_float2(pacc[nr][2], pacc[nr][3]);
          }
        } else {
#pragma unroll
          for (int nr = 0; nr < NR; ++nr)
#pragma unroll
            for (int e = 0; e < 4; ++e) chk = fmaf(pacc[nr][e], 0.f, chk);
        }
#pragma unroll
        for (int nr = 0; nr < NR; ++nr) pacc[nr][0] = pacc[nr][1] = pacc[nr][2] = pacc[nr][3] = 0.f;
      }
    }
    c_slot = (c_slot + 1 == S) ? 0 : c_slot + 1;
    if (++c_w == W) {
      c_w = 0;
      ++c_cs;
      if (++c_ch == c_nch) {
        c_ch = 0;
        c_it += gridDim.x;
        c_ok = next_mma_item(a, c_it, item, td);
        if (c_ok) c_nch = (item.ncols + T::CC - 1) / T::CC;
      }
    }
  }
  cp_async_wait<0>();
  if (__any_sync(0xffffffffu, !(chk == 0.f)) && lane == 0) atomicOr(&a.ctrl->flag, 1);
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

// ---------------------------------------------------------------------------
// Pass 2 for padded rank 32 (16 compiles too; the fp32 kernel is faster
// there) ("PowerSGD Hooks", powerSGD_hook steps 3.5-3.6, the replica mean
// folded): the partial Q' = Mbar^T P of one row
// block on the tensor cores, same items and partial layout (qpart[rb][k][j])
// as k_pass2.  As an mma the product is D (columns x ranks) = A (columns x
// rows) B (rows x ranks): warp w owns MB 16-column blocks of the item's tile
// and all RP ranks, walking the rows 8 at a time.  Each warp streams its
// columns of Mbar (the Mbar scratch, or the single replica's store half) into
// a private ring of NS 8-row units with cp.async (row stride 16 MB + 8:
// conflict-free fragment reads); P rows are staged per 128 rows in shared
// memory (row stride RP + 8).  Sources have 16-byte aligned rows (stride ld),
// so every tensor takes this path.
// ---------------------------------------------------------------------------
template <int RP>
struct Pass2Mma {
  static constexpr int NR = RP / 8;                 // rank blocks
  static constexpr int MB = RP == 32 ? 2 : 4;       // 16-column blocks per warp
  static constexpr int WC = 16 * MB;                // columns per warp
  static constexpr int AS = WC + 8;                 // staged row stride (floats)
  static constexpr int UNIT = 8 * AS * 4;           // one 8-row unit of a warp
  static constexpr int NS = RP == 32 ? 12 : 8;      // units in a warp's ring
  static constexpr int PS = RP + 8;                 // staged P row stride
  static constexpr int SMEM = 8 * NS * UNIT + kPStage * PS * 4;
  static_assert(8 * WC == ctile_for(RP), "the 8 warps cover the column tile");
};

template <int RP>
__global__ void __launch_bounds__(kThreads, 1) k_pass2_mma(const StepArgs a) {
  using T = Pass2Mma<RP>;
  constexpr int NR = T::NR, MB = T::MB, NS = T::NS, AS = T::AS, PS = T::PS;
  extern __shared__ __align__(128) char p2m_smem[];
  if (a.ctrl->flag) return;
  const int nxt = a.ctrl->cur ^ 1;
  const float* P = a.Pf + (long long)nxt * a.p_total;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  char* const ring = p2m_smem + warp * NS * T::UNIT;
  float* const ps = reinterpret_cast<float*>(p2m_smem + 8 * NS * T::UNIT);
  // mbar scratch, or (one replica) the store half pass 1 just wrote
  const float* srcb = a.mbar ? a.mbar : a.estore + (long long)nxt * a.nc_pad;
  for (int it = blockIdx.x; it < a.n_items; it += gridDim.x) {
    const Item item = a.items[it];
    const TensorDesc td = a.tensors[item.t];
    const long long ld = td.ld;
    const int cend = item.col0 + item.ncols;
    const int wc0 = item.col0 + warp * T::WC;
    const float* src = srcb + td.c_off;
    const int nunits = (item.nrows + 7) / 8;
    // unit u: rows row0 + 8u .. + 7 of this warp's columns, WC / 4 pieces a row
    auto issue = [&](int u) {
      if (u < nunits) {
        char* dst = ring + (u % NS) * T::UNIT;
#pragma unroll
        for (int j = 0; j < 8 * (T::WC / 4) / 32; ++j) {
          const int pc = lane + 32 * j, row = pc / (T::WC / 4), q = pc % (T::WC / 4);
          const int rr = item.row0 + 8 * u + row, col = wc0 + 4 * q;
          const bool v = rr < item.row0 + item.nrows && col < cend;
          cp_async16_z(dst + (row * AS + 4 * q) * 4, src + (v ? (long long)rr * ld + col : 0), v);
        }
      }
      cp_async_commit();
    };
#pragma unroll
    for (int u = 0; u < NS - 1; ++u) issue(u);
    float acc[MB][NR][4];
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
      for (int nr = 0; nr < NR; ++nr) acc[mb][nr][0] = acc[mb][nr][1] = acc[mb][nr][2] = acc[mb][nr][3] = 0.f;
    for (int u = 0; u < nunits; ++u) {
      const int ks = (8 * u) % kPStage;             // row of the unit in the staged P block
      if (ks == 0) {
        __syncthreads();
        const int sb = 8 * u, rows = min(kPStage, item.nrows - sb);
        for (int idx = threadIdx.x; idx < kPStage * RP; idx += kThreads) {
          const int rr = idx / RP, k = idx - rr * RP;
          ps[rr * PS + k] = rr < rows ? P[td.p_off + (long long)(item.row0 + sb + rr) * RP + k] : 0.f;
        }
        __syncthreads();
      }
      cp_async_wait<NS - 2>();
      __syncwarp();
      const float* ar = reinterpret_cast<const float*>(ring + (u % NS) * T::UNIT);
      uint32_t bh[NR][2], bl[NR][2];
#pragma unroll
      for (int nr = 0; nr < NR; ++nr) {
        split_tf32(ps[(ks + c) * PS + nr * 8 + g], bh[nr][0], bl[nr][0]);
        split_tf32(ps[(ks + c + 4) * PS + nr * 8 + g], bh[nr][1], bl[nr][1]);
      }
#pragma unroll
      for (int mb = 0; mb < MB; ++mb) {
        // A[m = column][k = row]: a0 (j, r), a1 (j + 8, r), a2 (j, r + 4), a3 (j + 8, r + 4)
        uint32_t ah[4], al[4];
        split_tf32(ar[c * AS + mb * 16 + g], ah[0], al[0]);
        split_tf32(ar[c * AS + mb * 16 + g + 8], ah[1], al[1]);
        split_tf32(ar[(c + 4) * AS + mb * 16 + g], ah[2], al[2]);
        split_tf32(ar[(c + 4) * AS + mb * 16 + g + 8], ah[3], al[3]);
#pragma unroll
        for (int nr = 0; nr < NR; ++nr) mma_tf32(acc[mb][nr], al, bh[nr][0], bh[nr][1]);
#pragma unroll
        for (int nr = 0; nr < NR; ++nr) mma_tf32(acc[mb][nr], ah, bl[nr][0], bl[nr][1]);
#pragma unroll
        for (int nr = 0; nr < NR; ++nr) mma_tf32(acc[mb][nr], ah, bh[nr][0], bh[nr][1]);
      }
      __syncwarp();                                  // the unit's slot is refilled next
      issue(u + NS - 1);
    }
    cp_async_wait<0>();
    // D[j][k]: d0 (j = g, k = 2c), d1 (g, 2c + 1), d2 (g + 8, 2c), d3 (g + 8, 2c + 1)
    float* dst = a.qpart + td.qp_off + (long long)item.rb * RP * td.m;
#pragma unroll
    for (int mb = 0; mb < MB; ++mb) {
      const int j = wc0 + mb * 16 + g;
#pragma unroll
      for (int nr = 0; nr < NR; ++nr) {
        const long long k = nr * 8 + 2 * c;
        if (j < cend) {
          dst[k * td.m + j] = acc[mb][nr][0];
          dst[(k + 1) * td.m + j] = acc[mb][nr][1];
        }
        if (j + 8 < cend) {
          dst[k * td.m + j + 8] = acc[mb][nr][2];
          dst[(k + 1) * td.m + j + 8] = acc[mb][nr][3];
        }
      }
    }
  }
}

}  // namespace psgd
