// Kernels of the PowerSGD hook step, templated on the padded rank RP.
//
// The step ("DDP Communication Hooks", "PowerSGD Hooks", powerSGD_hook
// steps 3.1-3.7) runs as three streaming passes over every compressed matrix
// plus a small Gram-Schmidt stage on P:
//
//   pass 1  M_w  = g_w * s + (store_w - P_old Q_old^T)     error feedback, unscale
//           store'_w = M_w                                 (next half of the store)
//           Mbar = mean_w M_w                              allreduce of P folded:
//           P_raw = Mbar Q                                 mean_w(M_w Q) = Mbar Q
//   GS      P = orth(P_raw)                                steps 3.3-3.4
//   pass 2  Q' = Mbar^T P                                  steps 3.5-3.6 (mean folded)
//   pass 3  out = P Q'^T                                   step 3.7
//
// The residual M_w - P Q'^T is never written: the store keeps M_w and the
// factors (P, Q') of the step, and pass 1 of the next step subtracts P Q'^T
// on the fly with the same fused multiply-add chain pass 3 uses for `out`,
// so the value it sees is exactly fl(M_w - out).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "psgd_internal.h"

namespace psgd {

// ---------------------------------------------------------------------------
// Arguments
// ---------------------------------------------------------------------------
struct StepArgs {
  GradPtrs grads;
  int W;
  int gtype;          // gradient type: 0 float, 1 __half, 2 __nv_bfloat16
  float scale;        // inverse loss scale
  float invW;
  float* out;
  float* estore;      // error store: half b, replica w at b * est_half + w * nc_pad
  long long nc_pad;
  long long est_half; // offset of the store's second half: W * nc_pad, or 0 for a
                      // one-half store (both halves the same memory)
  float* mbar;        // replica-mean scratch or nullptr
  float* Pf;          // committed P, half b at b * p_total
  float* Qf;          // committed Q, half b at b * q_total
  long long p_total, q_total;
  float* qinit;       // orthogonalised fresh Q (used when no warm Q)
  float* qdraw;       // raw standard-normal draw before orthogonalisation
  float* praw_part;   // pass-1 partials
  float* praw;        // summed P_raw
  float* pgs;         // first Gram-Schmidt sweep output (P and Q share it)
  float* qpart;       // pass-2 partials
  float* qx;          // data-parallel split: k_qreduce writes this process's Q
                      // here (the exchange buffer, Q layout) instead of Qf
  float* img;         // ranks 16 and 32: tensor-core operand images of P and Q
  const Item* t3items;  // tensor-core pass 3 items (128 x 256; aligned, backed tensors)
  int n_t3;
  const Item* t2items;  // tensor-core pass 2 items (one row block x 128 columns)
  int n_t2;
  const Item* t1items;  // tensor-core pass 1 items (aligned rows, wholly backed)
  int n_t1;
  float2* gram;       // per Gram-Schmidt item RP x RP (double-float)
  float2* gram_t;     // per tensor RP x RP, the items' sum
  float* tmat;        // per tensor RP x RP transform
  float* tmat2;       // fused Gram-Schmidt stage: the second sweep's transforms
  int* gs_cnt;        // fused Gram-Schmidt stage: Gram partials counted per tensor
  int* commit_cnt;    // set: pass 3 (k_pass3, mode 0) ends the step with the commit,
                      // in the CTA that finishes last (counted here)
  int* status;        // the step's status word the commit writes
  const TensorDesc* tensors;
  const Item* items;         // tall (row block) x (column tile) items: pass 2
  int n_items;
  const Item* fitems;        // short items: pass 3 and the error views
  int n_fitems;
  const Item* p1items;       // short items of pass 1 (its own column tiles)
  int n_p1items;
  const GsItem* ps_items;    // chunks of each tensor's P for the partial reduction
  int n_ps;
  const GsItem* qr_items;    // chunks of each tensor's Q for the partial reduction
  int n_qr;
  const GsItem* gsp_items;   // rows of P
  int n_gsp;
  const GsItem* gsq_items;   // rows of Q
  int n_gsq;
  const int* gsp_first;      // per tensor: first Gram-Schmidt item over P
  const int* gsp_count;
  const int* gsq_first;      // per tensor: first item over Q
  const int* gsq_count;
  int n_tensors;
  Ctrl* ctrl;
  int ef;
  int warm_start;
  int vec_ok;          // grads/out base pointers allow 16-byte (8 for f16) accesses
  int has_aligned;     // some compressed tensor has 16-byte aligned rows
  int has_unaligned;   // some has not, or the bucket ends inside its view
  long long gn;        // elements in each replica's bucket
  float eps;
  // error get/set
  int replica;
  float* eio;          // user buffer (packed, e_off layout)
};

// ---------------------------------------------------------------------------
// Memory helpers: streamed data bypasses L1 so the small Q tiles stay there.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float4 ld_stream4(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_stream1(const float* p) {
  float v;
  asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
// The error store is read and written by the same pass (different halves),
// so it is read with a plain (coherent) load.
__device__ __forceinline__ float4 ld_cg4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_cg1(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream4(float* p, float4 v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_stream1(float* p, float v) {
  asm volatile("st.global.cs.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void st_stream2(float* p, float a, float b) {
  asm volatile("st.global.cs.v2.f32 [%0], {%1,%2};" ::"l"(p), "f"(a), "f"(b) : "memory");
}

// NC consecutive elements of a gradient bucket as floats.  NC = 4 is one
// vector access (the caller guarantees alignment); other widths go element by
// element.
template <int NC, typename GT>
__device__ __forceinline__ void load_grad(const GT* p, float (&v)[NC]) {
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    float t[1];
    load_grad<1, GT>(p + c, t);
    v[c] = t[0];
  }
}

template <>
__device__ __forceinline__ void load_grad<4, float>(const float* p, float (&v)[4]) {
  float4 x = ld_stream4(p);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
template <>
__device__ __forceinline__ void load_grad<1, float>(const float* p, float (&v)[1]) {
  v[0] = ld_stream1(p);
}
template <>
__device__ __forceinline__ void load_grad<4, __half>(const __half* p, float (&v)[4]) {
  uint2 raw;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(raw.x), "=r"(raw.y)
               : "l"(p));
  __half2 a = *reinterpret_cast<__half2*>(&raw.x);
  __half2 b = *reinterpret_cast<__half2*>(&raw.y);
  float2 fa = __half22float2(a), fb = __half22float2(b);
  v[0] = fa.x; v[1] = fa.y; v[2] = fb.x; v[3] = fb.y;
}
template <>
__device__ __forceinline__ void load_grad<1, __half>(const __half* p, float (&v)[1]) {
  unsigned short raw;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(raw) : "l"(p));
  v[0] = __half2float(__ushort_as_half(raw));
}

template <>
__device__ __forceinline__ void load_grad<4, __nv_bfloat16>(const __nv_bfloat16* p, float (&v)[4]) {
  uint2 raw;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(raw.x), "=r"(raw.y)
               : "l"(p));
  const float2 fa = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&raw.x));
  const float2 fb = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&raw.y));
  v[0] = fa.x; v[1] = fa.y; v[2] = fb.x; v[3] = fb.y;
}
template <>
__device__ __forceinline__ void load_grad<1, __nv_bfloat16>(const __nv_bfloat16* p, float (&v)[1]) {
  unsigned short raw;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(raw) : "l"(p));
  v[0] = __bfloat162float(__ushort_as_bfloat16(raw));
}

// Four 16-bit gradient values (8 bytes, e.g. from a shared-memory slot) as floats.
template <typename GT>
__device__ __forceinline__ void cvt4(uint2 raw, float (&v)[4]) {
  if constexpr (std::is_same<GT, __half>::value) {
    const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    v[0] = fa.x; v[1] = fa.y; v[2] = fb.x; v[3] = fb.y;
  } else {
    const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
    const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
    v[0] = fa.x; v[1] = fa.y; v[2] = fb.x; v[3] = fb.y;
  }
}

template <int NC>
__device__ __forceinline__ void load_f(const float* p, float (&v)[NC], bool stream) {
  if constexpr (NC == 4) {
    float4 x = stream ? ld_stream4(p) : ld_cg4(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else {
#pragma unroll
    for (int c = 0; c < NC; ++c) v[c] = stream ? ld_stream1(p + c) : ld_cg1(p + c);
  }
}
template <int NC>
__device__ __forceinline__ void store_f(float* p, const float (&v)[NC]) {
  if constexpr (NC == 4) {
    st_stream4(p, make_float4(v[0], v[1], v[2], v[3]));
  } else {
#pragma unroll
    for (int c = 0; c < NC; ++c) st_stream1(p + c, v[c]);
  }
}

// One row of a factor matrix (RP floats, 16-byte aligned when RP >= 4).
template <int RP>
__device__ __forceinline__ void load_row(const float* __restrict__ p, float (&v)[RP]) {
  if constexpr (RP >= 4) {
#pragma unroll
    for (int k = 0; k < RP; k += 4) {
      float4 x = __ldg(reinterpret_cast<const float4*>(p + k));
      v[k] = x.x; v[k + 1] = x.y; v[k + 2] = x.z; v[k + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < RP; ++k) v[k] = __ldg(p + k);
  }
}

// Columns c .. c+NC-1 of a k-major factor (element (j, k) at base + k * ld + j):
// v[cc][k].  One coalesced access per k across the warp.
// Columns c .. c+NC-1 of a k-major Q block (leading dimension ld).  AL: the
// NC = 4 columns are one aligned float4.  !AL: only the first `nvalid`
// columns are read; the rest are zero.
template <int RP, int NC, bool AL = true>
__device__ __forceinline__ void load_qcols(const float* __restrict__ base, long long ld, long long c,
                                           float (&v)[NC][RP], int nvalid = NC) {
#pragma unroll
  for (int k = 0; k < RP; ++k) {
    const float* p = base + (long long)k * ld + c;
    if constexpr (NC == 4 && AL) {
      float4 x = __ldg(reinterpret_cast<const float4*>(p));
      v[0][k] = x.x; v[1][k] = x.y; v[2][k] = x.z; v[3][k] = x.w;
    } else if constexpr (AL) {
#pragma unroll
      for (int cc = 0; cc < NC; ++cc) v[cc][k] = __ldg(p + cc);
    } else {
#pragma unroll
      for (int cc = 0; cc < NC; ++cc) v[cc][k] = cc < nvalid ? __ldg(p + cc) : 0.f;
    }
  }
}

// sum_k a[k] * b[k] as one fused multiply-add chain in increasing k.  Pass 3
// (out) and pass 1 (the lazy residual) both use it, so they agree bit for bit.
template <int RP>
__device__ __forceinline__ float dot_chain(const float (&a)[RP], const float (&b)[RP]) {
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < RP; ++k) acc = fmaf(a[k], b[k], acc);
  return acc;
}

// Packed pairs of fp32 values for fma.rn.f32x2: each half is an independent
// IEEE fused multiply-add (the bits of fmaf), two per instruction.
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Reduce RP per-lane values over the warp by recursive halving: each step
// exchanges half of the remaining values with the lane `o` apart, so after
// log2(RP) steps every lane holds one partial value, which the remaining
// steps sum.  The total of value index (lane >> (5 - log2 RP)) ends in lane
// `lane` (all 32 / RP lanes of a group hold the same total).
template <int RP>
__device__ __forceinline__ float warp_reduce_scatter(const float (&v)[RP]) {
  float x[RP];
#pragma unroll
  for (int i = 0; i < RP; ++i) x[i] = v[i];
  const int lane = threadIdx.x & 31;
  int o = 16;
#pragma unroll
  for (int n = RP; n > 1; n >>= 1, o >>= 1) {
    const int half = n >> 1;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? x[i] : x[i + half];
      const float keep = up ? x[i + half] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float t = x[0];
  for (; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

template <int RP>
__host__ __device__ constexpr int log2_rp() { return RP >= 32 ? 5 : RP >= 16 ? 4 : RP >= 8 ? 3 : RP >= 4 ? 2 : RP >= 2 ? 1 : 0; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// Pass 1: error feedback + unscale + replica mean + P_raw = Mbar Q.
// One CTA per (row block, column tile) item; a warp owns RW rows at a time,
// its lanes stride the tile's columns NC at a time.  P_raw partials of the
// tile are reduced across the warp and written per column tile.
// ---------------------------------------------------------------------------
template <int RP, int WT, typename GT, int RW, int NC>
__device__ __forceinline__ void pass1_tile(const StepArgs& a, const TensorDesc& td,
                                           const Item& item, const float* __restrict__ Qp,
                                           const float* __restrict__ Qc,
                                           const float* __restrict__ Pc, int cur, int& bad) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = WT > 0 ? WT : a.W;
  const int nxt = cur ^ 1;
  const long long m = td.m;
  const int cend = item.col0 + item.ncols;
  for (int rr = warp * RW; rr < item.nrows; rr += (kThreads / 32) * RW) {
    float po[RW][RP];
    float pacc[RW][RP];
    bool rv[RW];
#pragma unroll
    for (int q = 0; q < RW; ++q) {
      rv[q] = (rr + q) < item.nrows;
      const int i = item.row0 + (rv[q] ? rr + q : rr);
#pragma unroll
      for (int k = 0; k < RP; ++k) { pacc[q][k] = 0.f; po[q][k] = 0.f; }
      if (a.ef) load_row<RP>(Pc + td.p_off + (long long)i * RP, po[q]);
    }
    for (int c = item.col0 + lane * NC; c < cend; c += 32 * NC) {
      // residual correction P_old[i,:] . Q_old[c,:]
      float corr[RW][NC];
      if (a.ef) {
        float qo[NC][RP];
        load_qcols<RP, NC>(Qc + td.q_off, m, c, qo);
#pragma unroll
        for (int cc = 0; cc < NC; ++cc)
#pragma unroll
          for (int q = 0; q < RW; ++q) corr[q][cc] = dot_chain<RP>(po[q], qo[cc]);
      }
      float mb[RW][NC];
#pragma unroll
      for (int q = 0; q < RW; ++q)
#pragma unroll
        for (int cc = 0; cc < NC; ++cc) mb[q][cc] = 0.f;
#pragma unroll(WT > 0 ? WT : 1)
      for (int w = 0; w < W; ++w) {
        const GT* g = reinterpret_cast<const GT*>(a.grads.p[w]);
        float* ecur = a.estore + (long long)cur * a.est_half + (long long)w * a.nc_pad + td.c_off;
        float* enxt = a.estore + (long long)nxt * a.est_half + (long long)w * a.nc_pad + td.c_off;
#pragma unroll
        for (int q = 0; q < RW; ++q) {
          if (!rv[q]) continue;
          const long long i = item.row0 + rr + q;
          float gv[NC];
          if (i * m + c + NC <= td.valid) {
            load_grad<NC, GT>(g + td.g_off + i * m + c, gv);
          } else {
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
              float t1[1] = {0.f};
              if (i * m + c + cc < td.valid) load_grad<1, GT>(g + td.g_off + i * m + c + cc, t1);
              gv[cc] = t1[0];
            }
          }
          float ev[NC];
          if (a.ef) load_f<NC>(ecur + i * td.ld + c, ev, false);
          float mv[NC];
#pragma unroll
          for (int cc = 0; cc < NC; ++cc) {
            const float v = gv[cc] * a.scale;
            bad |= !isfinite(v);
            mv[cc] = a.ef ? v + (ev[cc] - corr[q][cc]) : v;
            mb[q][cc] += mv[cc];
          }
          if (a.ef) store_f<NC>(enxt + i * td.ld + c, mv);
        }
      }
#pragma unroll
      for (int q = 0; q < RW; ++q) {
#pragma unroll
        for (int cc = 0; cc < NC; ++cc) mb[q][cc] *= a.invW;
        if (a.mbar && rv[q]) store_f<NC>(a.mbar + td.c_off + (long long)(item.row0 + rr + q) * td.ld + c, mb[q]);
      }
      {
        float qv[NC][RP];
        load_qcols<RP, NC>(Qp + td.q_off, m, c, qv);
#pragma unroll
        for (int cc = 0; cc < NC; ++cc)
#pragma unroll
          for (int q = 0; q < RW; ++q)
#pragma unroll
            for (int k = 0; k < RP; ++k) pacc[q][k] = fmaf(mb[q][cc], qv[cc][k], pacc[q][k]);
      }
    }
#pragma unroll
    for (int q = 0; q < RW; ++q) {
#pragma unroll
      for (int k = 0; k < RP; ++k) pacc[q][k] = warp_sum(pacc[q][k]);
      if (rv[q] && lane == 0) {
        float* dst = a.praw_part + td.pp_off +
                     ((long long)item.ct * td.n + item.row0 + rr + q) * RP;
#pragma unroll
        for (int k = 0; k < RP; ++k) dst[k] = pacc[q][k];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// cp.async staging: a lane copies the bytes it will consume of a source row
// segment into its own slot of shared memory, several units ahead, so bytes
// in flight cost shared memory instead of registers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ---------------------------------------------------------------------------
// Pass 1, chunk-stationary (RP <= 8).  Warp w of the CTA owns chunk
// (w % nch) of the item's column tile (nch <= 8 chunks of 128 columns) and
// every (8 / nch)-th row of the item, so each lane loads the Q values of its
// 4 columns once per item and keeps them in registers.  Its
// source segments (one row x 128 columns of every replica's gradient and
// store) are staged by cp.async S rows ahead.  Each
// row's P partial over the chunk is reduced across the warp and parked in
// shared memory; at the end of the item the CTA adds the chunk partials in
// chunk order and writes one partial per (row, column tile).
// ---------------------------------------------------------------------------
template <int RP, int WT, typename GT, int MINB, bool SH = false>
struct Pass1CS {
  static constexpr int NCH = ctile1_for(RP) / 128;                // chunks per column tile
  static constexpr int GB = 4 * (int)sizeof(GT);
  static constexpr int GSEG = 32 * GB;
  static constexpr int ESEG = 32 * 16;
  // rows of any alignment (SH): after the segments, the chunk that follows
  // lane 31's, for every gradient and error segment
  static constexpr int XOFF = WT * (GSEG + ESEG);
  static constexpr int UNIT_BYTES = XOFF + (SH ? 2 * WT * 16 : 0);   // one row x 128 columns
  static constexpr int RED_BYTES = rows1_for(RP) * NCH * RP * 4;
  static constexpr int PST_BYTES = rows1_for(RP) * RP * 4;          // the item's committed P rows
  static constexpr int BUDGET = (MINB == 1 ? 200 * 1024 : 112 * 1024) - RED_BYTES - PST_BYTES;
  static constexpr int S_RAW = BUDGET / (8 * UNIT_BYTES);
  static constexpr int S = S_RAW > 8 ? 8 : (S_RAW < 2 ? 2 : S_RAW);
  static constexpr int SMEM = 8 * S * UNIT_BYTES + RED_BYTES + PST_BYTES;
};

// Four values of a row that starts r elements (0..3, warp-uniform) into the
// aligned chunk `lo`; `hi` is the next aligned chunk.
__device__ __forceinline__ void shift_sel(const float (&lo)[4], const float (&hi)[4], int r, float (&v)[4]) {
  switch (r) {
    case 0: v[0] = lo[0]; v[1] = lo[1]; v[2] = lo[2]; v[3] = lo[3]; break;
    case 1: v[0] = lo[1]; v[1] = lo[2]; v[2] = lo[3]; v[3] = hi[0]; break;
    case 2: v[0] = lo[2]; v[1] = lo[3]; v[2] = hi[0]; v[3] = hi[1]; break;
    default: v[0] = lo[3]; v[1] = hi[0]; v[2] = hi[1]; v[3] = hi[2]; break;
  }
}

// Streams v[0..nv) to p, which sits r = (address / 4) mod 4 elements past a
// 16-byte boundary: a full group of four is one 16-byte store (r = 0), two
// 8-byte stores (r = 2) or 4 + 8 + 4 bytes (r odd).
__device__ __forceinline__ void store4_split(float* p, const float (&v)[4], int nv, int r) {
  if (nv == 4) {
    if (r == 0) {
      st_stream4(p, make_float4(v[0], v[1], v[2], v[3]));
    } else if (r == 2) {
      st_stream2(p, v[0], v[1]);
      st_stream2(p + 2, v[2], v[3]);
    } else {
      st_stream1(p, v[0]);
      st_stream2(p + 1, v[1], v[2]);
      st_stream1(p + 3, v[3]);
    }
  } else {
    for (int cc = 0; cc < nv; ++cc) st_stream1(p + cc, v[cc]);
  }
}

// MODE 0: the tensor's rows are 16-byte aligned in the bucket and the item
// lies inside the bucket-backed part of the view (no bounds checks).  MODE 1:
// the bucket rows have any alignment (the base pointers are still aligned),
// and the view may end inside the item (batched hook's padding): each
// lane stages the aligned gradient chunk that holds its first column, lane 31
// also the chunk after it (at XOFF in the stage), and a lane takes its four
// values from its own chunk and the next lane's.  The error store and mbar
// rows (stride ld) are aligned in both modes.  PW: the bucket has a.W < WT
// replicas (the stage is laid out for WT; replicas a.W.. are neither read nor
// written), so one instantiation per WT serves every count up to it.
template <int RP, int WT, typename GT, int MINB, int MODE, bool PW = false>
__device__ __forceinline__ void pass1_tile_cs(const StepArgs& a, const TensorDesc& td, const Item& item,
                                              const float* __restrict__ Qp, const float* __restrict__ Qc,
                                              const float* __restrict__ Pc, int cur, float& chk,
                                              char* __restrict__ wsm, float* __restrict__ red,
                                              float* __restrict__ pst) {
  constexpr bool SH = (MODE == 1);
  using St = Pass1CS<RP, WT, GT, MINB, SH>;
  constexpr int S = St::S;
  constexpr int GB = St::GB;
  constexpr int NCH = St::NCH;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nxt = cur ^ 1;
  const long long m = td.m, ld = td.ld;
  const int cend = item.col0 + item.ncols;
  const int nch = (item.ncols + 127) / 128;
  // wpc warps per chunk (rows interleaved among them): a full tile has one
  // warp per chunk; a narrow one spreads the 8 warps over its chunks
  const int wpc = 8 / nch;
  const int ch = warp % nch;
  const int phase = warp / nch;
  const bool unit_scale = (a.scale == 1.0f);
  const bool same_q = (Qp == Qc);
  // pass-1 tiles have 8, 4, 2 or 1 chunks, so every warp has a chunk; a warp
  // without one would take no units but still meet the CTA barriers
  const bool active = warp < nch * wpc;
  {
    const int c = item.col0 + ch * 128 + lane * 4;
    const bool cin = active && c < cend;
    const int ncv = cin ? (int)min(4LL, (long long)cend - c) : 0;   // this lane's columns in the tile
    const int units = (active && phase < item.nrows) ? (item.nrows - phase + wpc - 1) / wpc : 0;
    float qc[4][RP], qp[4][RP];
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
#pragma unroll
      for (int k = 0; k < RP; ++k) { qc[cc][k] = 0.f; qp[cc][k] = 0.f; }
    if (cin) {
      if (a.ef) load_qcols<RP, 4, !SH>(Qc + td.q_off, m, c, qc, ncv);
      if (!(a.ef && same_q)) load_qcols<RP, 4, !SH>(Qp + td.q_off, m, c, qp, ncv);
    }
    // units are issued and consumed in order, wpc rows apart, the issued one
    // S - 1 units ahead of the consumed one: running offsets of the consumed
    // unit (bucket position, store offset) and rotating stage slots replace
    // per-row products.  go / eo: bucket and store offsets of the unit issued.
    const long long gstep = (long long)wpc * m, estep = (long long)wpc * ld;
    const long long row_first = (long long)item.row0 + phase;
    const long long ecur = (long long)cur * a.est_half;
    auto issue = [&](char* slot, long long go, long long eo) {
      if constexpr (!SH) {
        if (cin) {
#pragma unroll
          for (int w = 0; w < WT; ++w) {
            if (PW && w >= a.W) break;
            const GT* gsrc = reinterpret_cast<const GT*>(a.grads.p[w]) + go;
            if constexpr (GB == 16) cp_async16(slot + w * St::GSEG + lane * GB, gsrc);
            else cp_async8(slot + w * St::GSEG + lane * GB, gsrc);
            if (a.ef) cp_async16(slot + WT * St::GSEG + w * St::ESEG + lane * 16, a.estore + eo + (long long)w * a.nc_pad);
          }
        }
      } else {
        const long long gp = go;   // this lane's first element in the bucket
        const int rg = (int)(gp & 3);
        if (GB == 16 || (rg & 1) == 0) {
          // the lane's own four values straight into its slot, in pieces sized
          // to the row's offset modulo 4 (16, 8 or 4 bytes; 8 or 4 for 16-bit
          // values at an even offset), so the math reads an aligned slot as
          // in kind 0 (the bucket's last values element by element)
          if (c < cend) {
#pragma unroll
            for (int w = 0; w < WT; ++w) {
              if (PW && w >= a.W) break;
              const GT* g = reinterpret_cast<const GT*>(a.grads.p[w]);
              char* dst = slot + w * St::GSEG + lane * GB;
              if (gp + 4 <= a.gn) {
                if (rg == 0) {
                  if constexpr (GB == 16) cp_async16(dst, g + gp); else cp_async8(dst, g + gp);
                } else if (rg == 2) {
                  if constexpr (GB == 16) {
                    cp_async8(dst, g + gp);
                    cp_async8(dst + 8, g + gp + 2);
                  } else {
                    cp_async4(dst, g + gp);
                    cp_async4(dst + 4, g + gp + 2);
                  }
                } else {
#pragma unroll
                  for (int e = 0; e < 4; ++e) cp_async4(dst + 4 * e, g + gp + e);
                }
              } else {
                for (int e = 0; e < 4; ++e)
                  reinterpret_cast<GT*>(dst)[e] = (gp + e < a.gn) ? g[gp + e] : GT(0.f);
              }
              if (a.ef) cp_async16(slot + WT * St::GSEG + w * St::ESEG + lane * 16, a.estore + eo + (long long)w * a.nc_pad);
            }
          }
          cp_async_commit();
          return;
        }
        // 16-bit values at an odd offset: the aligned chunk holding this
        // lane's first column, and the next lane's, select the four values
        const bool gneed = c - rg < cend;
        const bool gx = lane == 31 && rg > 0 && c + 4 - rg < cend;
        auto gcopy = [&](char* dst, const GT* g, long long at) {
          if (at + 4 <= a.gn) {
            if constexpr (GB == 16) cp_async16(dst, g + at); else cp_async8(dst, g + at);
          } else {
            // the bucket ends inside this chunk
            for (int e = 0; e < 4; ++e)
              if (at + e < a.gn) reinterpret_cast<GT*>(dst)[e] = g[at + e];
          }
        };
#pragma unroll
        for (int w = 0; w < WT; ++w) {
          if (PW && w >= a.W) break;
          const GT* g = reinterpret_cast<const GT*>(a.grads.p[w]);
          if (gneed) gcopy(slot + w * St::GSEG + lane * GB, g, gp - rg);
          if (gx) gcopy(slot + St::XOFF + w * 16, g, gp - rg + 4);
          if (cin && a.ef) cp_async16(slot + WT * St::GSEG + w * St::ESEG + lane * 16, a.estore + eo + (long long)w * a.nc_pad);
        }
      }
      cp_async_commit();
    };
    // the item's committed P rows into shared memory, copied (one group of
    // its own) ahead of the first units and read there by every warp: the
    // unit loop then waits on no global load
    if (a.ef) {
      const float* psrc = Pc + td.p_off + (long long)item.row0 * RP;
      const int nv = item.nrows * RP;
      if constexpr (RP >= 4) {   // P rows (RP floats) are 16-byte aligned
        for (int idx = threadIdx.x * 4; idx < nv; idx += kThreads * 4) cp_async16(pst + idx, psrc + idx);
      } else {
        for (int idx = threadIdx.x; idx < nv; idx += kThreads) cp_async4(pst + idx, psrc + idx);
      }
    }
    cp_async_commit();
#pragma unroll
    for (int u = 0; u < S - 1; ++u) {
      const long long r = row_first + (long long)u * wpc;
      if (u < units) issue(wsm + u * St::UNIT_BYTES, td.g_off + r * m + c, ecur + td.c_off + r * ld + c);
      else cp_async_commit();
    }
    // Q's columns (loaded above, before the copies were issued) as column
    // pairs (0, 1) and (2, 3) for fma.rn.f32x2: packed only now, so that
    // their loads' latency overlaps the copies in flight
    uint64_t qc2[2][RP], qp2[2][RP];
#pragma unroll
    for (int k = 0; k < RP; ++k) {
      qc2[0][k] = f2pack(qc[0][k], qc[1][k]);
      qc2[1][k] = f2pack(qc[2][k], qc[3][k]);
      qp2[0][k] = f2pack(qp[0][k], qp[1][k]);
      qp2[1][k] = f2pack(qp[2][k], qp[3][k]);
    }
    cp_async_wait<S - 1>();   // this thread's P pieces have landed (the units may not)
    __syncthreads();          // and every thread's
    long long r_off = td.c_off + row_first * ld + c;   // store / mbar offset of the unit
    long long g_pos = row_first * m + c;               // its position in the tensor's view
    const long long g_ahead = td.g_off + (S - 1) * gstep, e_ahead = ecur + (S - 1) * estep;
    int s_use = 0;
    for (int u = 0; u < units; ++u) {
      cp_async_wait<S - 2>();
      if constexpr (SH) __syncwarp();   // lanes read their neighbour's chunk
      // unit u + S - 1 goes to the slot unit u - 1 used
      if (u + S - 1 < units)
        issue(wsm + (s_use == 0 ? S - 1 : s_use - 1) * St::UNIT_BYTES, g_pos + g_ahead, r_off + e_ahead);
      else
        cp_async_commit();
      const int rr = phase + u * wpc;
      const char* slot = wsm + s_use * St::UNIT_BYTES;
      s_use = (s_use + 1 == S) ? 0 : s_use + 1;
      float po[RP];
      if (a.ef) {
        if constexpr (RP >= 4) {
#pragma unroll
          for (int k = 0; k < RP; k += 4) {
            const float4 x = *reinterpret_cast<const float4*>(pst + rr * RP + k);
            po[k] = x.x; po[k + 1] = x.y; po[k + 2] = x.z; po[k + 3] = x.w;
          }
        } else {
#pragma unroll
          for (int k = 0; k < RP; ++k) po[k] = pst[rr * RP + k];
        }
      } else {
#pragma unroll
        for (int k = 0; k < RP; ++k) po[k] = 0.f;
      }
      float pacc[RP];
#pragma unroll
      for (int k = 0; k < RP; ++k) pacc[k] = 0.f;
      if (cin) {
        float corr[4] = {0.f, 0.f, 0.f, 0.f};
        if (a.ef) {
          // dot_chain of each column, two columns per instruction (same bits)
          uint64_t c01 = f2pack(0.f, 0.f), c23 = f2pack(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < RP; ++k) {
            const uint64_t pk = f2pack(po[k], po[k]);
            c01 = fma2(pk, qc2[0][k], c01);
            c23 = fma2(pk, qc2[1][k], c23);
          }
          f2unpack(c01, corr[0], corr[1]);
          f2unpack(c23, corr[2], corr[3]);
        }
        float mb[4] = {0.f, 0.f, 0.f, 0.f};
        float* enxt = a.estore + (long long)nxt * a.est_half + r_off;
        // SH: columns taken from the bucket (the tile's and the bucket's ends)
        const long long lim = SH ? td.valid - g_pos : 4;
        const int nvg = lim >= ncv ? ncv : (lim > 0 ? (int)lim : 0);
        const int rg = SH ? (int)((td.g_off + g_pos) & 3) : 0;
#pragma unroll
        for (int w = 0; w < WT; ++w) {
          if (PW && w >= a.W) break;
          float gv[4];
          if (SH && !(GB == 16 || (rg & 1) == 0)) {
            float lo[4], hi[4];
            const char* own = slot + w * St::GSEG + lane * GB;
            const char* nx = lane < 31 ? own + GB : slot + St::XOFF + w * 16;
            if constexpr (GB == 16) {
              const float4 x = *reinterpret_cast<const float4*>(own);
              const float4 y = *reinterpret_cast<const float4*>(nx);
              lo[0] = x.x; lo[1] = x.y; lo[2] = x.z; lo[3] = x.w;
              hi[0] = y.x; hi[1] = y.y; hi[2] = y.z; hi[3] = y.w;
            } else {
              cvt4<GT>(*reinterpret_cast<const uint2*>(own), lo);
              cvt4<GT>(*reinterpret_cast<const uint2*>(nx), hi);
            }
            shift_sel(lo, hi, rg, gv);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) gv[cc] = cc < nvg ? gv[cc] : 0.f;
          } else {
            if constexpr (GB == 16) {
              const float4 x = *reinterpret_cast<const float4*>(slot + w * St::GSEG + lane * GB);
              gv[0] = x.x; gv[1] = x.y; gv[2] = x.z; gv[3] = x.w;
            } else {
              cvt4<GT>(*reinterpret_cast<const uint2*>(slot + w * St::GSEG + lane * GB), gv);
            }
            if constexpr (SH) {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) gv[cc] = cc < nvg ? gv[cc] : 0.f;
            }
          }
          float mv[4];
          if (a.ef) {
            const float4 x = *reinterpret_cast<const float4*>(slot + WT * St::GSEG + w * St::ESEG + lane * 16);
            // a lane's columns past cend are the store's padding (cend is
            // m there, else a multiple of 4), which stays zero
            const float ev[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const float v = unit_scale ? gv[cc] : gv[cc] * a.scale;
              mv[cc] = v + (ev[cc] - corr[cc]);
              mb[cc] += mv[cc];
            }
            // SH: columns past m get 0 + (0 - 0), keeping the padding zero
            store_f<4>(enxt + (long long)w * a.nc_pad, mv);
          } else {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              mv[cc] = unit_scale ? gv[cc] : gv[cc] * a.scale;
              mb[cc] += mv[cc];
            }
          }
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) mb[cc] *= a.invW;
        if (a.mbar) store_f<4>(a.mbar + r_off, mb);
        // projection: rank k gets (mb0 q0 + mb2 q2) + (mb1 q1 + mb3 q3)
        const uint64_t (*qq)[RP] = (a.ef && same_q) ? qc2 : qp2;
        const uint64_t m01 = f2pack(mb[0], mb[1]), m23 = f2pack(mb[2], mb[3]);
#pragma unroll
        for (int k = 0; k < RP; ++k) {
          float x, y;
          f2unpack(fma2(m23, qq[1][k], fma2(m01, qq[0][k], f2pack(0.f, 0.f))), x, y);
          pacc[k] = x + y;
        }
      }
      const float tot = warp_reduce_scatter<RP>(pacc);
      chk = fmaf(tot, 0.f, chk);   // inf/NaN in the row's inputs reach the sums
      constexpr int SHF = 5 - log2_rp<RP>();
      if ((lane & ((1 << SHF) - 1)) == 0) red[(rr * NCH + ch) * RP + (lane >> SHF)] = tot;
      r_off += estep;
      g_pos += gstep;
    }
    cp_async_wait<0>();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < item.nrows * RP; e += kThreads) {
    const int rr = e / RP, k = e - (e / RP) * RP;
    float v = 0.f;
    for (int h = 0; h < nch; ++h) v += red[(rr * NCH + h) * RP + k];
    a.praw_part[td.pp_off + ((long long)item.ct * td.n + item.row0 + rr) * RP + k] = v;
  }
  __syncthreads();
}

// KIND 0 takes the items of tensors with 16-byte aligned rows (when the
// gradient pointers are aligned too) that lie wholly inside the bucket, and
// skips the rest; KIND 1 takes the rest: shifted chunks (MODE 1) when the
// pointers are aligned, else the element path.  Separate instantiations keep
// the aligned kernel free of the other paths' registers and checks.
template <int RP, int WT, typename GT, int MINB, int KIND, bool PW = false>
__global__ void __launch_bounds__(kThreads, MINB) k_pass1_cs(const StepArgs a) {
  extern __shared__ __align__(16) char p1smem[];
  using St = Pass1CS<RP, WT, GT, MINB, KIND == 1>;
  const int cur = a.ctrl->cur;
  const bool use_init = (!a.warm_start) || (a.ctrl->warm_valid == 0);
  const float* Qc = a.Qf + (long long)cur * a.q_total;
  const float* Pc = a.Pf + (long long)cur * a.p_total;
  const float* Qp = use_init ? a.qinit : Qc;
  char* wsm = p1smem + (threadIdx.x >> 5) * (St::S * St::UNIT_BYTES);
  float* red = reinterpret_cast<float*>(p1smem + 8 * St::S * St::UNIT_BYTES);
  float* pst = reinterpret_cast<float*>(p1smem + 8 * St::S * St::UNIT_BYTES + St::RED_BYTES);
  int bad = 0;
  float chk = 0.f;
  for (int it = blockIdx.x; it < a.n_p1items; it += gridDim.x) {
    const Item item = a.p1items[it];
    const TensorDesc td = a.tensors[item.t];
    const bool aligned = td.vec && a.vec_ok && (long long)(item.row0 + item.nrows) * td.m <= td.valid;
    if constexpr (KIND == 0) {
      if (aligned) pass1_tile_cs<RP, WT, GT, MINB, 0, PW>(a, td, item, Qp, Qc, Pc, cur, chk, wsm, red, pst);
    } else {
      if (aligned) continue;
      if (a.vec_ok)
        pass1_tile_cs<RP, WT, GT, MINB, 1, PW>(a, td, item, Qp, Qc, Pc, cur, chk, wsm, red, pst);
      else
        pass1_tile<RP, PW ? 0 : WT, GT, 1, 1>(a, td, item, Qp, Qc, Pc, cur, bad);
    }
  }
  bad |= !(chk == 0.f);
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(&a.ctrl->flag, 1);
}

template <int RP, int WT, typename GT, int RW>
__global__ void __launch_bounds__(kThreads) k_pass1(const StepArgs a) {
  const int cur = a.ctrl->cur;
  const bool use_init = (!a.warm_start) || (a.ctrl->warm_valid == 0);
  const float* Qc = a.Qf + (long long)cur * a.q_total;
  const float* Pc = a.Pf + (long long)cur * a.p_total;
  const float* Qp = use_init ? a.qinit : Qc;
  int bad = 0;
  for (int it = blockIdx.x; it < a.n_p1items; it += gridDim.x) {
    const Item item = a.p1items[it];
    const TensorDesc td = a.tensors[item.t];
    if (td.vec && a.vec_ok)
      pass1_tile<RP, WT, GT, RW, 4>(a, td, item, Qp, Qc, Pc, cur, bad);
    else
      pass1_tile<RP, WT, GT, RW, 1>(a, td, item, Qp, Qc, Pc, cur, bad);
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(&a.ctrl->flag, 1);
}

// ---------------------------------------------------------------------------
// Pass 2: partial Q' = Mbar^T P over one (row block, column tile); each thread
// owns CPT columns and accumulates CPT x RP sums over the block's rows.
// SRC 0: Mbar scratch; 1: mean of the W store halves just written; 2: mean of
// the W unscaled gradients (error feedback off).  Partials are k-major:
// qpart[rb][k][j].
// ---------------------------------------------------------------------------
constexpr int kPStage = 128;
// rows of loads issued together per thread: 32 bytes x batch per source
__host__ __device__ constexpr int row_batch_for(int rp) { return 32 / cpt_for(rp); }

// NC values of Mbar at (row, c0 ..) from the selected source; VEC: one
// 16-byte access per source (NC == 4, aligned rows), else element by element
// with bounds checks.
template <int SRC, typename GT, int WT, int NC, bool VEC>
__device__ __forceinline__ void load_mbar(const StepArgs& a, const TensorDesc& td, long long row, int c0,
                                          int cend, int nxt, float (&mv)[NC]) {
  const long long m = td.m, ld = td.ld;
  static_assert(!VEC || NC == 4, "vector path is 4 wide");
  if constexpr (SRC == 0) {
    if constexpr (VEC) {
      load_f<4>(a.mbar + td.c_off + row * ld + c0, mv, true);
    } else {
#pragma unroll
      for (int c = 0; c < NC; ++c) mv[c] = (c0 + c < cend) ? ld_stream1(a.mbar + td.c_off + row * ld + c0 + c) : 0.f;
    }
  } else {
    const int W = WT > 0 ? WT : a.W;
#pragma unroll
    for (int c = 0; c < NC; ++c) mv[c] = 0.f;
#pragma unroll(WT > 0 ? WT : 1)
    for (int w = 0; w < W; ++w) {
      float v[NC];
      if constexpr (SRC == 1) {
        const float* src = a.estore + (long long)nxt * a.est_half + (long long)w * a.nc_pad + td.c_off + row * ld + c0;
        if constexpr (VEC) {
          load_f<4>(src, v, true);
        } else {
#pragma unroll
          for (int c = 0; c < NC; ++c) v[c] = (c0 + c < cend) ? ld_stream1(src + c) : 0.f;
        }
      } else {
        const GT* src = reinterpret_cast<const GT*>(a.grads.p[w]) + td.g_off + row * m + c0;
        if (VEC && row * m + c0 + 4 <= td.valid) {
          if constexpr (VEC) load_grad<4, GT>(src, v);
        } else {
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            float t[1] = {0.f};
            if (c0 + c < cend && row * m + c0 + c < td.valid) load_grad<1, GT>(src + c, t);
            v[c] = t[0];
          }
        }
#pragma unroll
        for (int c = 0; c < NC; ++c) v[c] *= a.scale;
      }
#pragma unroll
      for (int c = 0; c < NC; ++c) mv[c] += v[c];
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) mv[c] *= a.invW;
  }
}

template <int RP, int SRC, typename GT, int WT, int NC>
__device__ __forceinline__ void pass2_tile(const StepArgs& a, const TensorDesc& td, const Item& item,
                                           const float* __restrict__ P, float (*ps)[RP]) {
  constexpr int CPT = cpt_for(RP);
  static_assert(NC == CPT || NC == 1, "columns per access");
  constexpr int NA = CPT;  // columns accumulated per thread
  constexpr int kRowBatch = row_batch_for(RP);
  const int c0 = item.col0 + threadIdx.x * CPT;
  const int nxt = a.ctrl->cur ^ 1;
  const int cend = item.col0 + item.ncols;
  float acc[NA][RP];
#pragma unroll
  for (int c = 0; c < NA; ++c)
#pragma unroll
    for (int k = 0; k < RP; ++k) acc[c][k] = 0.f;
  for (int sb = 0; sb < item.nrows; sb += kPStage) {
    const int rows = min(kPStage, item.nrows - sb);
    __syncthreads();
    for (int idx = threadIdx.x; idx < rows * RP; idx += kThreads)
      ps[idx / RP][idx % RP] = P[td.p_off + (long long)(item.row0 + sb) * RP + idx];
    __syncthreads();
    if (c0 >= cend) continue;
    int i = 0;
    for (; i + kRowBatch <= rows; i += kRowBatch) {
      float mv[kRowBatch][NA];
#pragma unroll
      for (int u = 0; u < kRowBatch; ++u)
        load_mbar<SRC, GT, WT, NA, (NC == 4)>(a, td, item.row0 + sb + i + u, c0, cend, nxt, mv[u]);
#pragma unroll
      for (int u = 0; u < kRowBatch; ++u)
#pragma unroll
        for (int c = 0; c < NA; ++c)
#pragma unroll
          for (int k = 0; k < RP; ++k) acc[c][k] = fmaf(mv[u][c], ps[i + u][k], acc[c][k]);
    }
    for (; i < rows; ++i) {
      float mv[NA];
      load_mbar<SRC, GT, WT, NA, (NC == 4)>(a, td, item.row0 + sb + i, c0, cend, nxt, mv);
#pragma unroll
      for (int c = 0; c < NA; ++c)
#pragma unroll
        for (int k = 0; k < RP; ++k) acc[c][k] = fmaf(mv[c], ps[i][k], acc[c][k]);
    }
  }
  if (c0 >= cend) return;
  float* dst = a.qpart + td.qp_off + (long long)item.rb * RP * td.m;
  const bool qvec = (td.m & 3) == 0;
#pragma unroll
  for (int k = 0; k < RP; ++k) {
    float* d = dst + (long long)k * td.m + c0;
    if (NA == 4 && NC == 4 && qvec) {
      *reinterpret_cast<float4*>(d) = make_float4(acc[0][k], acc[1][k], acc[2][k], acc[3][k]);
    } else {
#pragma unroll
      for (int c = 0; c < NA; ++c)
        if (c0 + c < cend) d[c] = acc[c][k];
    }
  }
}

// The vector path needs 16-byte aligned rows of the source: the mbar scratch
// and the store always have them (stride ld); gradients read directly need
// an aligned tensor, else the element-wise path (NC = 1): same CPT columns
// per thread, one access per element.
template <int RP, int SRC, typename GT, int WT>
__global__ void __launch_bounds__(kThreads, 3) k_pass2(const StepArgs a) {
  __shared__ __align__(16) float ps[kPStage][RP];
  if (a.ctrl->flag) return;
  const float* P = a.Pf + (long long)(a.ctrl->cur ^ 1) * a.p_total;
  constexpr int CPT = cpt_for(RP);
  for (int it = blockIdx.x; it < a.n_items; it += gridDim.x) {
    const Item item = a.items[it];
    const TensorDesc td = a.tensors[item.t];
    const bool vec = (SRC == 2) ? (td.vec && a.vec_ok) : true;
    if (vec && CPT == 4)
      pass2_tile<RP, SRC, GT, WT, CPT>(a, td, item, P, ps);
    else
      pass2_tile<RP, SRC, GT, WT, 1>(a, td, item, P, ps);
  }
}

// ---------------------------------------------------------------------------
// Pass 3: out = P Q'^T.  Each thread keeps its CPT3 columns of Q' in registers.
// MODE 0: write out (bucket layout).  MODE 1: materialise replica `a.replica`'s
// residual store - P Q^T of the committed half into a.eio.  MODE 2: set the
// store from a.eio + P Q^T.  MODE 3: fold the factors into the store in place
// (store -= P Q^T), after which the factors can be replaced.
// ---------------------------------------------------------------------------
// SHF (MODE 0, CPT 4): out rows of any alignment, written through
// store4_split.  BND: check each store against the end of the bucket.
template <int RP, int MODE, int NC, bool SHF = false, bool BND = true>
__device__ __forceinline__ void pass3_tile(const StepArgs& a, const TensorDesc& td, const Item& item,
                                           const float* __restrict__ P, const float* __restrict__ Q,
                                           float (*ps)[RP], float* __restrict__ store) {
  constexpr int CPT = cpt3_for(RP);
  static_assert(!SHF || (MODE == 0 && CPT == 4 && NC == 1), "shifted stores: out, 4 columns a thread");
  const long long m = td.m, ld = td.ld;
  const int c0 = item.col0 + threadIdx.x * CPT;
  const int cend = item.col0 + item.ncols;
  float qv[CPT][RP];
#pragma unroll
  for (int k = 0; k < RP; ++k) {
    const float* q = Q + td.q_off + (long long)k * m + c0;
    if constexpr (NC == 4 && CPT == 4) {
      if (c0 < cend) {
        float4 x = __ldg(reinterpret_cast<const float4*>(q));
        qv[0][k] = x.x; qv[1][k] = x.y; qv[2][k] = x.z; qv[3][k] = x.w;
      } else {
        qv[0][k] = qv[1][k] = qv[2][k] = qv[3][k] = 0.f;
      }
    } else {
#pragma unroll
      for (int c = 0; c < CPT; ++c) qv[c][k] = (c0 + c < cend) ? __ldg(q + c) : 0.f;
    }
  }
  for (int sb = 0; sb < item.nrows; sb += kPStage) {
    const int rows = min(kPStage, item.nrows - sb);
    __syncthreads();
    for (int idx = threadIdx.x; idx < rows * RP; idx += kThreads)
      ps[idx / RP][idx % RP] = P[td.p_off + (long long)(item.row0 + sb) * RP + idx];
    __syncthreads();
    if (c0 >= cend) continue;
#pragma unroll 4
    for (int i = 0; i < rows; ++i) {
      const long long row = item.row0 + sb + i;
      float pr[RP];
#pragma unroll
      for (int k = 0; k < RP; ++k) pr[k] = ps[i][k];
      float o[CPT];
#pragma unroll
      for (int c = 0; c < CPT; ++c) o[c] = dot_chain<RP>(pr, qv[c]);
      if constexpr (SHF) {
        const long long pos = row * m + c0;
        const long long lim = min((long long)cend - c0, td.valid - pos);
        const int nv = lim >= 4 ? 4 : (lim > 0 ? (int)lim : 0);
        const float ov[4] = {o[0], o[1], o[2], o[3]};
        store4_split(a.out + td.g_off + pos, ov, nv, (int)((td.g_off + pos) & 3));
      } else if constexpr (NC == CPT && CPT == 4) {
        if constexpr (MODE == 0) {
          if (!BND || row * m + c0 + 4 <= td.valid) {
            store_f<4>(a.out + td.g_off + row * m + c0, o);
          } else {
            // the bucket ends inside this chunk (batched hook): truncate
#pragma unroll
            for (int c = 0; c < 4; ++c)
              if (row * m + c0 + c < td.valid) st_stream1(a.out + td.g_off + row * m + c0 + c, o[c]);
          }
        } else if constexpr (MODE == 1) {
          float sv[4];
          load_f<4>(store + td.c_off + row * ld + c0, sv, true);
#pragma unroll
          for (int c = 0; c < 4; ++c) a.eio[td.e_off + row * m + c0 + c] = sv[c] - o[c];
        } else if constexpr (MODE == 2) {
#pragma unroll
          for (int c = 0; c < 4; ++c) store[td.c_off + row * ld + c0 + c] = a.eio[td.e_off + row * m + c0 + c] + o[c];
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) store[td.c_off + row * ld + c0 + c] -= o[c];
        }
      } else {
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          if (c0 + c >= cend) continue;
          const long long idx = row * m + c0 + c;        // bucket / packed view
          const long long sdx = row * ld + c0 + c;       // store
          if constexpr (MODE == 0) {
            if (idx < td.valid) st_stream1(a.out + td.g_off + idx, o[c]);
          } else if constexpr (MODE == 1) {
            a.eio[td.e_off + idx] = store[td.c_off + sdx] - o[c];
          } else if constexpr (MODE == 2) {
            store[td.c_off + sdx] = a.eio[td.e_off + idx] + o[c];
          } else {
            store[td.c_off + sdx] -= o[c];
          }
        }
      }
    }
  }
}

// The end-of-step commit (k_commit's work for a compressed step) done by the
// CTA of a pass that finishes last: every other CTA has counted itself done,
// so none still reads which half is current.  The counter is left at zero.
__device__ __forceinline__ void commit_last(const StepArgs& a) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.commit_cnt, 1) == (int)gridDim.x - 1) {
      __threadfence();
      const int bad = *reinterpret_cast<volatile int*>(&a.ctrl->flag);
      const int late = *reinterpret_cast<volatile int*>(&a.ctrl->timeout);
      if (!bad && !late) {
        a.ctrl->cur ^= 1;
        a.ctrl->warm_valid = 1;
      }
      *a.status = late ? 2 : (bad ? 1 : 0);
      *a.commit_cnt = 0;
    }
  }
}

template <int RP, int MODE>
__global__ void __launch_bounds__(kThreads) k_pass3(const StepArgs a) {
  __shared__ __align__(16) float ps[kPStage][RP];
  if (MODE == 0 && a.ctrl->flag) {   // skipped step: only the commit (if asked) is left
    if (a.commit_cnt) commit_last(a);
    return;
  }
  // MODE 0 reads the factors just computed (next half); the error views read
  // the committed half.
  const int half = (MODE == 0) ? (a.ctrl->cur ^ 1) : a.ctrl->cur;
  const float* P = a.Pf + (long long)half * a.p_total;
  const float* Q = a.Qf + (long long)half * a.q_total;
  float* store = nullptr;
  if (MODE != 0) store = a.estore + (long long)a.ctrl->cur * a.est_half + (long long)a.replica * a.nc_pad;
  constexpr int CPT = cpt3_for(RP);
  for (int it = blockIdx.x; it < a.n_fitems; it += gridDim.x) {
    const Item item = a.fitems[it];
    const TensorDesc td = a.tensors[item.t];
    const bool vec = (MODE == 0) ? (td.vec && a.vec_ok) : (td.m % 4 == 0);
    // ranks 16 and 32: the tensor-core pass 3 wrote the aligned, backed tensors
    if (MODE == 0 && RP >= 16 && a.n_t3 > 0 && vec && td.valid == (long long)td.n * td.m) continue;
    // BND: the view may end inside the item (batched hook's padding)
    const bool inside = (long long)(item.row0 + item.nrows) * td.m <= td.valid;
    if (vec && CPT == 4 && inside)
      pass3_tile<RP, MODE, CPT, false, false>(a, td, item, P, Q, ps, store);
    else if (vec && CPT == 4)
      pass3_tile<RP, MODE, CPT>(a, td, item, P, Q, ps, store);
    else if (MODE == 0 && CPT == 4 && a.vec_ok)
      pass3_tile<RP, MODE, 1, MODE == 0 && CPT == 4>(a, td, item, P, Q, ps, store);
    else
      pass3_tile<RP, MODE, 1>(a, td, item, P, Q, ps, store);
  }
  if (MODE == 0 && a.commit_cnt) commit_last(a);
}

}  // namespace psgd
