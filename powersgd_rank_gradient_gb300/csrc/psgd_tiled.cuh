// Pass 1 for padded ranks 16 and 32 ("PowerSGD Hooks", powerSGD_hook steps
// 3.2-3.3 with the error feedback of the hook's warning), register-tiled.
//
// At these ranks the pass does 2 * RP fused multiply-adds per element (RP for
// the lazy residual P_old Q_old^T, RP for the projection Mbar Q) against
// 8 + s_g bytes of HBM per replica, so the FMA pipe and the shared-memory
// loads feeding it bound it, not HBM.  Each contraction therefore runs as a
// small register-tiled product with 16 FMAs per thread per pair of 16-byte
// shared-memory loads:
//
//   work item  128 rows x 512 columns of one tensor, walked in 32-column
//              chunks; one CTA (8 warps) per SM over a persistent item list.
//   layout A   thread t owns rows 4*(t/8) .. +3 and the chunk's columns
//              4*(t%8) .. +3: the residual correction P_old Q_old^T of those
//              16 elements (P_old rows through L1, the Q_old chunk in shared
//              memory, increasing-k FMA chains, bit-identical to pass 3),
//              then M_w = g_w * s + (store_w - correction) for every replica
//              (written to the next store half) and their mean Mbar.
//   M tile     Mbar of the chunk, column-major in shared memory (a warp's
//              rows are its own, so only the warp synchronises on it).
//   layout B   the same warp owns the same 16 rows x RP partial sums of
//              P_raw += Mbar Q: thread (rows 4 x ranks 4) per 4-column step
//              of the chunk; at rank 16 the two half-warps take alternate
//              halves of the chunk and are added at the end of the item.
//
// Sources are staged with cp.async into per-thread slots, S - 1 (chunk,
// replica) units ahead, continuing across items; the Q chunks (shared by the
// CTA) rotate through SQ buffers, published by one CTA barrier per chunk.
#pragma once

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

template <int RP, typename GT>
struct Pass1Tiled {
  static_assert(RP == 16 || RP == 32, "tiled pass 1 is for ranks 16 and 32");
  static_assert(kThreads == 256, "layout A maps 256 threads onto 32 row groups x 8 column quads");
  static constexpr int TR = kRows1Tiled;                      // rows per item
  static constexpr int CC = 32;                               // columns per chunk
  static constexpr int GB = 4 * (int)sizeof(GT);              // gradient bytes per thread and row
  static constexpr int G_BYTES = 4 * kThreads * GB;           // gradient part of a unit
  static constexpr int UNIT_BYTES = G_BYTES + 4 * kThreads * 16;
  static constexpr int S = 4;                                 // units in the ring
  // A Q chunk buffer may be refilled only after every thread has left the
  // chunk that last used it: with units issued S - 1 ahead, S buffers cover
  // any replica count (the bound is 2 + (S - 2) / W).
  static constexpr int SQ = S;
  static constexpr int QCH_BYTES = RP * CC * 4;               // one Q chunk, k-major
  static constexpr int MT_BYTES = CC * TR * 4;                // Mbar tile
  static constexpr int SMEM = S * UNIT_BYTES + 2 * SQ * QCH_BYTES + MT_BYTES;
  static_assert(TR == 4 * (kThreads / 8), "one row group of 4 rows per 8 threads");
};

// The items of the tiled kernel: tensors whose rows are 16-byte aligned in
// the bucket, wholly backed by it.  Advances `it` (stepping by the grid) to
// the next such item and loads it.
__device__ __forceinline__ bool tiled_item(const StepArgs& a, int& it, Item& item, TensorDesc& td) {
  for (; it < a.n_p1items; it += gridDim.x) {
    item = a.p1items[it];
    td = a.tensors[item.t];
    if (td.vec && a.vec_ok && (long long)(item.row0 + item.nrows) * td.m <= td.valid) return true;
  }
  return false;
}

// Q chunk layout in shared memory: 16-byte unit (k, column quad cq) at
// k * 8 + (cq ^ ((k >> 2) & 7)), so that both the layout-A reads (fixed k,
// eight quads) and the layout-B reads (fixed quad, eight k groups) hit eight
// different bank groups.
__device__ __forceinline__ int qunit(int k, int cq) { return k * 8 + (cq ^ ((k >> 2) & 7)); }
// Mbar tile: 16-byte unit (chunk column cl, row group g) at
// cl * 32 + (g ^ ((cl >> 2) & 7)).
__device__ __forceinline__ int munit(int cl, int g) { return cl * 32 + (g ^ ((cl >> 2) & 7)); }

template <int RP, typename GT>
__global__ void __launch_bounds__(kThreads, 1) k_pass1_tiled(const StepArgs a) {
  using T = Pass1Tiled<RP, GT>;
  constexpr int S = T::S, SQ = T::SQ, GB = T::GB;
  extern __shared__ __align__(128) char p1t_smem[];
  char* const wsm = p1t_smem;                                       // S units of per-thread slots
  char* const qsm = p1t_smem + S * T::UNIT_BYTES;                   // SQ x {correction Q, projection Q}
  float4* const mt = reinterpret_cast<float4*>(qsm + 2 * SQ * T::QCH_BYTES);

  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int g = t >> 3;          // layout A: row group (rows 4g .. 4g+3 of the item)
  const int lc = t & 7;          // layout A: column quad of the chunk
  // layout B: rank group, row group and (rank 16) chunk half of this thread
  const int lk = RP == 32 ? (lane & 7) : (lane & 3);
  const int gb = RP == 32 ? g : warp * 4 + ((lane >> 2) & 3);
  const int lh = RP == 32 ? 0 : (lane >> 4);

  const int cur = a.ctrl->cur, nxt = cur ^ 1;
  const bool use_init = (!a.warm_start) || (a.ctrl->warm_valid == 0);
  const float* Qc = a.Qf + (long long)cur * a.q_total;
  const float* Pc = a.Pf + (long long)cur * a.p_total;
  const float* Qp = use_init ? a.qinit : Qc;
  const bool ef = a.ef != 0;
  const bool same_q = (Qp == Qc);
  const int pq = (ef && same_q) ? 0 : 1;   // which Q buffer the projection reads
  const int W = a.W;
  const bool unit_scale = (a.scale == 1.0f);
  const long long ecur = (long long)cur * W * a.nc_pad;
  const long long enx = (long long)nxt * W * a.nc_pad;

  // ---- issuer: (item, chunk, replica) units, S - 1 ahead of the consumer
  int i_it = blockIdx.x, i_ch = 0, i_w = 0, i_cs = 0, i_nch = 0, i_slot = 0;
  Item i_item;
  TensorDesc i_td;
  bool i_ok = tiled_item(a, i_it, i_item, i_td);
  if (i_ok) i_nch = (i_item.ncols + T::CC - 1) / T::CC;
  auto issue = [&]() {
    if (i_ok) {
      char* slot = wsm + i_slot * T::UNIT_BYTES;
      const long long m = i_td.m, ld = i_td.ld;
      const int cend = i_item.col0 + i_item.ncols;
      const int c = i_item.col0 + i_ch * T::CC + lc * 4;
      const bool cv = c < cend;
      const GT* gbase = reinterpret_cast<const GT*>(a.grads.p[i_w]) + i_td.g_off;
      const float* ebase = a.estore + ecur + (long long)i_w * a.nc_pad + i_td.c_off;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int rl = g * 4 + q;
        const bool v = cv && rl < i_item.nrows;
        const long long row = i_item.row0 + rl;
        const GT* gs = gbase + (v ? row * m + c : 0);
        if constexpr (GB == 16) cp_async16_z(slot + q * kThreads * GB + t * GB, gs, v);
        else cp_async8_z(slot + q * kThreads * GB + t * GB, gs, v);
        if (ef) cp_async16_z(slot + T::G_BYTES + q * kThreads * 16 + t * 16, ebase + (v ? row * ld + c : 0), v);
      }
      if (i_w == 0 && t < RP * 8) {
        // this chunk's Q columns: thread t copies unit (k, cq) = (t / 8, t % 8)
        const int k = t >> 3, cq = t & 7;
        const int col = i_item.col0 + i_ch * T::CC + cq * 4;
        const bool v = col < cend;
        const long long off = i_td.q_off + (long long)k * m + (v ? col : 0);
        char* dst = qsm + (i_cs % SQ) * 2 * T::QCH_BYTES + qunit(k, cq) * 16;
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
          i_ok = tiled_item(a, i_it, i_item, i_td);
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
  bool c_ok = tiled_item(a, c_it, item, td);
  if (c_ok) c_nch = (item.ncols + T::CC - 1) / T::CC;
  float corr[4][4], mb[4][4], pacc[4][4];
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int i = 0; i < 4; ++i) pacc[q][i] = 0.f;
  float chk = 0.f;
  while (c_ok) {
    cp_async_wait<S - 2>();
    if (c_w == 0) __syncthreads();   // the chunk's Q is in; every thread has left the last chunk
    issue();
    const long long m = td.m, ld = td.ld;
    const int cend = item.col0 + item.ncols;
    const int c = item.col0 + c_ch * T::CC + lc * 4;
    const bool cv = c < cend;
    const char* qbuf = qsm + (c_cs % SQ) * 2 * T::QCH_BYTES;
    bool rv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) rv[q] = g * 4 + q < item.nrows;
    if (c_w == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) { corr[q][cc] = 0.f; mb[q][cc] = 0.f; }
      if (ef) {
        // correction = P_old Q_old^T on the 4 x 4 elements, one increasing-k
        // FMA chain each (the chain pass 3 used for `out`)
        const float* prow = Pc + td.p_off + (long long)(item.row0 + g * 4) * RP;
#pragma unroll
        for (int kb = 0; kb < RP / 4; ++kb) {
          float4 po[4], qo[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            po[q] = rv[q] ? __ldg(reinterpret_cast<const float4*>(prow + q * RP + kb * 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int i = 0; i < 4; ++i) qo[i] = *reinterpret_cast<const float4*>(qbuf + qunit(kb * 4 + i, lc) * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float p = i == 0 ? po[q].x : (i == 1 ? po[q].y : (i == 2 ? po[q].z : po[q].w));
              corr[q][0] = fmaf(p, qo[i].x, corr[q][0]);
              corr[q][1] = fmaf(p, qo[i].y, corr[q][1]);
              corr[q][2] = fmaf(p, qo[i].z, corr[q][2]);
              corr[q][3] = fmaf(p, qo[i].w, corr[q][3]);
            }
          }
        }
      }
    }
    // M_w of this replica: written to the next store half, added to the mean
    {
      const char* slot = wsm + c_slot * T::UNIT_BYTES;
      float* enxt = a.estore + enx + (long long)c_w * a.nc_pad + td.c_off;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float gv[4];
        if constexpr (GB == 16) {
          const float4 x = *reinterpret_cast<const float4*>(slot + q * kThreads * GB + t * GB);
          gv[0] = x.x; gv[1] = x.y; gv[2] = x.z; gv[3] = x.w;
        } else {
          cvt4<GT>(*reinterpret_cast<const uint2*>(slot + q * kThreads * GB + t * GB), gv);
        }
        float mv[4];
        if (ef) {
          const float4 x = *reinterpret_cast<const float4*>(slot + T::G_BYTES + q * kThreads * 16 + t * 16);
          const float ev[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const float v = unit_scale ? gv[cc] : gv[cc] * a.scale;
            mv[cc] = v + (ev[cc] - corr[q][cc]);
          }
          if (rv[q] && cv) store_f<4>(enxt + (long long)(item.row0 + g * 4 + q) * ld + c, mv);
        } else {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) mv[cc] = unit_scale ? gv[cc] : gv[cc] * a.scale;
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) mb[q][cc] += mv[cc];
      }
    }
    if (c_w == W - 1) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const bool v = rv[q] && cv;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) mb[q][cc] = v ? mb[q][cc] * a.invW : 0.f;
        if (a.mbar && v) store_f<4>(a.mbar + td.c_off + (long long)(item.row0 + g * 4 + q) * ld + c, mb[q]);
      }
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) mt[munit(lc * 4 + cc, g)] = make_float4(mb[0][cc], mb[1][cc], mb[2][cc], mb[3][cc]);
      __syncwarp();
      // layout B: pacc[row q][rank 4 lk + i] += Mbar(row, col) Q(col, rank)
      const char* qp = qbuf + pq * T::QCH_BYTES;
      constexpr int NQ = RP == 32 ? 8 : 4;     // column quads per thread
#pragma unroll 2
      for (int s = 0; s < NQ; ++s) {
        const int cq = lh * 4 + s;
        float4 mv[4], qv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) mv[j] = mt[munit(cq * 4 + j, gb)];
#pragma unroll
        for (int i = 0; i < 4; ++i) qv[i] = *reinterpret_cast<const float4*>(qp + qunit(lk * 4 + i, cq) * 16);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float m0 = q == 0 ? mv[0].x : (q == 1 ? mv[0].y : (q == 2 ? mv[0].z : mv[0].w));
          const float m1 = q == 0 ? mv[1].x : (q == 1 ? mv[1].y : (q == 2 ? mv[1].z : mv[1].w));
          const float m2 = q == 0 ? mv[2].x : (q == 1 ? mv[2].y : (q == 2 ? mv[2].z : mv[2].w));
          const float m3 = q == 0 ? mv[3].x : (q == 1 ? mv[3].y : (q == 2 ? mv[3].z : mv[3].w));
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float acc = pacc[q][i];
            acc = fmaf(m0, qv[i].x, acc);
            acc = fmaf(m1, qv[i].y, acc);
            acc = fmaf(m2, qv[i].z, acc);
            acc = fmaf(m3, qv[i].w, acc);
            pacc[q][i] = acc;
          }
        }
      }
      if (c_ch == c_nch - 1) {
        // end of the item: one partial P row slice per (row, column tile)
        if constexpr (RP == 16) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int i = 0; i < 4; ++i) pacc[q][i] += __shfl_xor_sync(0xffffffffu, pacc[q][i], 16);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int i = 0; i < 4; ++i) chk = fmaf(pacc[q][i], 0.f, chk);
          const int rl = gb * 4 + q;
          if (lh == 0 && rl < item.nrows) {
            float* dst = a.praw_part + td.pp_off + ((long long)item.ct * td.n + item.row0 + rl) * RP + lk * 4;
            *reinterpret_cast<float4*>(dst) = make_float4(pacc[q][0], pacc[q][1], pacc[q][2], pacc[q][3]);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) pacc[q][i] = 0.f;
        }
      }
    }
    // advance the consumer
    c_slot = (c_slot + 1 == S) ? 0 : c_slot + 1;
    if (++c_w == W) {
      c_w = 0;
      ++c_cs;
      if (++c_ch == c_nch) {
        c_ch = 0;
        c_it += gridDim.x;
        c_ok = tiled_item(a, c_it, item, td);
        if (c_ok) c_nch = (item.ncols + T::CC - 1) / T::CC;
      }
    }
  }
  cp_async_wait<0>();
  if (__any_sync(0xffffffffu, !(chk == 0.f)) && lane == 0) atomicOr(&a.ctrl->flag, 1);
}

// The pass-1 items the tiled kernel does not take (rows not 16-byte aligned
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

}  // namespace psgd
