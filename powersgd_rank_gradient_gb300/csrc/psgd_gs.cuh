// Gram-Schmidt stage of the PowerSGD hook step (P and the fresh Q), and the
// reductions of the streaming passes' partial sums (k_psum for pass 1's P,
// k_qreduce for pass 2's Q), templated on the padded rank RP.  Kept apart
// from the streaming passes (psgd_kernels.cuh) so that the two evolve
// separately.
#pragma once

#include "psgd_kernels.cuh"
#include "psgd_tc.cuh"

namespace psgd {

// ---------------------------------------------------------------------------
// Gram-Schmidt stage.
//
// "PowerSGD Hooks" step 3.4 orthogonalises P column by column; "PowerSGD
// State" item 4 adds epsilon to each column norm.  Every Gram-Schmidt
// operation is a column operation, so the result is X T for an RP x RP upper
// triangular T that depends only on the Gram matrix G = X^T X.  The stage
// therefore (1) forms G per row block (k_gram) and adds the blocks per tensor
// (k_gram_sum), (2) runs modified Gram-Schmidt with epsilon symbolically on G
// to get T (k_solve, one CTA per tensor), (3) applies X T (k_apply), all
// sums and the recurrence in double-float arithmetic on the fp32 pipes.  It
// runs twice (the second sweep re-orthogonalises the first sweep's output),
// which keeps P^T P = I to fp32 rounding even when X is ill conditioned.
// ---------------------------------------------------------------------------
// P_raw = sum of pass 1's column-tile partials, in tile order (the Gram stage
// then reads dense rows).  Each work item is a chunk of one tensor's rows x RP
// values, four per thread.
template <int RP>
__device__ __forceinline__ void psum_item(const StepArgs& a, int it) {
  {
    const GsItem gi = a.ps_items[it];
    const TensorDesc td = a.tensors[gi.t];
    const long long len = (long long)td.n * RP;
    const float* src = a.praw_part + td.pp_off;
    const int f = gi.row0 + threadIdx.x * 4;
    if (f >= gi.row0 + gi.nrows) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (RP >= 4) {
      int c = 0;
      for (; c + 4 <= td.ctiles1; c += 4) {
        float4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) x[u] = *reinterpret_cast<const float4*>(src + (long long)(c + u) * len + f);
#pragma unroll
        for (int u = 0; u < 4; ++u) { acc.x += x[u].x; acc.y += x[u].y; acc.z += x[u].z; acc.w += x[u].w; }
      }
      for (; c < td.ctiles1; ++c) {
        const float4 x = *reinterpret_cast<const float4*>(src + (long long)c * len + f);
        acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
      }
      *reinterpret_cast<float4*>(a.praw + td.p_off + f) = acc;
    } else {
      for (int e = f; e < min(f + 4, gi.row0 + gi.nrows); ++e) {
        float v = 0.f;
        for (int c = 0; c < td.ctiles1; ++c) v += src[(long long)c * len + e];
        a.praw[td.p_off + e] = v;
      }
    }
  }
}

template <int RP>
__global__ void __launch_bounds__(kThreads) k_psum(const StepArgs a) {
  if (a.ctrl->flag) return;
  for (int it = blockIdx.x; it < a.n_ps; it += gridDim.x) psum_item<RP>(a, it);
}

// Q'(j, k) = sum over row blocks of the partials, written k-major into the
// next half of Qf (or, in the data-parallel split, into the exchange buffer
// a.qx, same layout).  Each work item is a chunk of kQrChunk values of one
// tensor's RP * m; four consecutive lanes share four consecutive values, lane
// q summing (in row-block order) the q-th quarter of the row blocks, and the
// quarters are added in order (((s0 + s1) + s2) + s3): a quarter of the
// dependent loads of one chain per value, eight of them in flight.
// img (ranks 16 and 32): also write Q's row and chunk images, as k_images
// mode 1 does.
template <int RP>
__global__ void __launch_bounds__(kThreads) k_qreduce(const StepArgs a, int img) {
  if (a.ctrl->flag) return;
  if (img && a.ctrl->timeout) return;   // not committed: the images keep the committed Q
  float* Q = a.qx ? a.qx : a.Qf + (long long)(a.ctrl->cur ^ 1) * a.q_total;
  const int q = threadIdx.x & 3;
  for (int it = blockIdx.x; it < a.n_qr; it += gridDim.x) {
    const GsItem gi = a.qr_items[it];
    const TensorDesc td = a.tensors[gi.t];
    const long long len = (long long)RP * td.m;
    const float* src = a.qpart + td.qp_off;
    const int f = gi.row0 + (threadIdx.x >> 2) * 4;   // this lane group's first value
    const int nb = td.rblocks;
    const int b0 = (int)((long long)nb * q / 4), b1 = (int)((long long)nb * (q + 1) / 4);
    const bool live = f < gi.row0 + gi.nrows;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live && len % 4 == 0) {
      int b = b0;
      for (; b + 8 <= b1; b += 8) {
        float4 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = ld_stream4(src + (long long)(b + u) * len + f);
#pragma unroll
        for (int u = 0; u < 8; ++u) { s.x += x[u].x; s.y += x[u].y; s.z += x[u].z; s.w += x[u].w; }
      }
      for (; b < b1; ++b) {
        const float4 x = ld_stream4(src + (long long)b * len + f);
        s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
      }
    } else if (live) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = 0.f;
        if (f + e < gi.row0 + gi.nrows)
          for (int b = b0; b < b1; ++b) v += src[(long long)b * len + f + e];
        if (e == 0) s.x = v; else if (e == 1) s.y = v; else if (e == 2) s.z = v; else s.w = v;
      }
    }
    // the quarters in order: lane q = 0 of the group adds q = 1, 2, 3
    float4 t = s;
#pragma unroll
    for (int j = 1; j < 4; ++j) {
      const float x = __shfl_down_sync(0xffffffffu, s.x, j), y = __shfl_down_sync(0xffffffffu, s.y, j);
      const float z = __shfl_down_sync(0xffffffffu, s.z, j), w = __shfl_down_sync(0xffffffffu, s.w, j);
      t.x += x; t.y += y; t.z += z; t.w += w;
    }
    if (!live || q != 0) continue;
    if constexpr (RP >= 16) {
      if (img) {
        const int ne = min(4, gi.row0 + gi.nrows - f);
        const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (e < ne) {
            img_put_q<RP>(a, td, (f + e) % td.m, (f + e) / td.m, tv[e], false);
            img_put_q<RP>(a, td, (f + e) % td.m, (f + e) / td.m, tv[e], true);
          }
      }
    }
    if (len % 4 == 0) {
      *reinterpret_cast<float4*>(Q + td.q_off + f) = t;
    } else {
      const int ne = min(4, gi.row0 + gi.nrows - f);
      Q[td.q_off + f] = t.x;
      if (ne > 1) Q[td.q_off + f + 1] = t.y;
      if (ne > 2) Q[td.q_off + f + 2] = t.z;
      if (ne > 3) Q[td.q_off + f + 3] = t.w;
    }
  }
}

constexpr int kGramTile = 128;

// Double-float accumulation on the fp32 pipes (fp64 throughput is a small
// fraction of fp32 on this GPU): (hi, lo) holds an unevaluated sum.  The
// product's rounding error comes from one FMA and the sum's from Knuth's
// two-sum, so each term adds its exact value up to the rounding of `lo`
// (about 2^-44 relative to the total).  The explicit-rounding intrinsics keep
// the compiler from contracting the error terms into FMAs.
__device__ __forceinline__ void df_add(float& hi, float& lo, float b, float blo) {
  const float s = __fadd_rn(hi, b);
  const float bp = __fsub_rn(s, hi);
  const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(b, bp));
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(e, blo));
}
__device__ __forceinline__ void df_add_prod(float& hi, float& lo, float a, float b) {
  const float p = __fmul_rn(a, b);
  df_add(hi, lo, p, fmaf(a, b, -p));
}

// Per Gram-Schmidt item: the Gram matrix X^T X of its rows, each entry a
// double-float (hi, lo) pair.  Rows of P come dense (nparts == 1) or as
// column-tile partials (from_parts).  gram_item does one item with the
// whole CTA (tile and red are the CTA's shared buffers).
template <int RP>
__device__ __forceinline__ void gram_item(const StepArgs& a, int it, const float* __restrict__ src,
                                          float* __restrict__ dense_out, int is_q, int from_parts,
                                          float2* __restrict__ gram_out, float (*tile)[RP + 1], float2* red) {
  constexpr int PAIRS = RP * RP;
  constexpr int PPT = PAIRS > kThreads ? PAIRS / kThreads : 1;   // pairs per thread
  constexpr int GROUPS = PAIRS >= kThreads ? 1 : kThreads / PAIRS;
  const GsItem* items = is_q ? a.gsq_items : a.gsp_items;
  const GsItem gi = items[it];
  const TensorDesc td = a.tensors[gi.t];
  const long long base = is_q ? td.q_off : td.p_off;
  const int pair0 = (threadIdx.x % (PAIRS >= kThreads ? kThreads : PAIRS)) * PPT;
  const int grp = PAIRS >= kThreads ? 0 : threadIdx.x / PAIRS;
  float hi[PPT], lo[PPT];
#pragma unroll
  for (int u = 0; u < PPT; ++u) { hi[u] = 0.f; lo[u] = 0.f; }
  for (int r0 = 0; r0 < gi.nrows; r0 += kGramTile) {
    const int rows = min(kGramTile, gi.nrows - r0);
    __syncthreads();
    for (int idx = threadIdx.x; idx < rows * RP; idx += kThreads) {
      const int rr = idx / RP, k = idx % RP;
      const long long row = gi.row0 + r0 + rr;
      float v;
      if (from_parts) {
        // the column-tile partials added in tile order, four loads in flight
        const float* pp = src + td.pp_off + row * RP + k;
        const long long tstride = (long long)td.n * RP;
        v = 0.f;
        int c = 0;
        for (; c + 4 <= td.ctiles1; c += 4) {
          float x[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) x[u] = pp[(c + u) * tstride];
#pragma unroll
          for (int u = 0; u < 4; ++u) v += x[u];
        }
        for (; c < td.ctiles1; ++c) v += pp[c * tstride];
      } else if (is_q) {
        v = src[base + (long long)k * td.m + row];
      } else {
        v = src[base + row * RP + k];
      }
      if (k >= td.r) v = 0.f;
      tile[rr][k] = v;
      if (dense_out) dense_out[base + row * RP + k] = v;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < PPT; ++u) {
      const int pa = (pair0 + u) / RP, pb = (pair0 + u) % RP;
      for (int rr = grp; rr < rows; rr += GROUPS) df_add_prod(hi[u], lo[u], tile[rr][pa], tile[rr][pb]);
    }
  }
  // reduce the row groups (in group order)
#pragma unroll
  for (int u = 0; u < PPT; ++u) {
    __syncthreads();
    red[threadIdx.x] = make_float2(hi[u], lo[u]);
    __syncthreads();
    if (threadIdx.x < (PAIRS >= kThreads ? kThreads : PAIRS)) {
      float2 s = red[threadIdx.x];
      for (int g = 1; g < GROUPS; ++g) {
        const float2 x = red[threadIdx.x + g * (PAIRS >= kThreads ? kThreads : PAIRS)];
        df_add(s.x, s.y, x.x, x.y);
      }
      gram_out[(long long)it * PAIRS + pair0 + u] = s;
    }
  }
}

template <int RP>
__global__ void __launch_bounds__(kThreads) k_gram(const StepArgs a, const float* __restrict__ src,
                                                   float* __restrict__ dense_out, int is_q,
                                                   int from_parts, float2* __restrict__ gram_out) {
  __shared__ float tile[kGramTile][RP + 1];
  __shared__ float2 red[kThreads];
  const int n_items = is_q ? a.n_gsq : a.n_gsp;
  if (a.ctrl->flag) return;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x)
    gram_item<RP>(a, it, src, dense_out, is_q, from_parts, gram_out, tile, red);
}

// The items' Gram matrices of each tensor added up: CTA (tensor, block of
// EPC entries), its threads in GROUPS item groups, each summing every
// GROUPS-th item as double-floats (eight loads in flight), the groups then
// combined in group order.
constexpr int kGramSumEntries = 32;

template <int RP>
__global__ void __launch_bounds__(kThreads) k_gram_sum(const StepArgs a, int is_q) {
  constexpr int ENT = RP * RP;
  constexpr int EPC = ENT < kGramSumEntries ? ENT : kGramSumEntries;
  constexpr int GROUPS = kThreads / EPC;
  __shared__ float2 part[kThreads];
  if (a.ctrl->flag) return;
  const int t = blockIdx.x;
  const int e = blockIdx.y * EPC + threadIdx.x % EPC;
  const int g = threadIdx.x / EPC;
  const int first = is_q ? a.gsq_first[t] : a.gsp_first[t];
  const int count = is_q ? a.gsq_count[t] : a.gsp_count[t];
  const float2* src = a.gram + (long long)first * ENT + e;
  float hi[2] = {0.f, 0.f}, lo[2] = {0.f, 0.f};
  int it = g;
  for (; it + 7 * GROUPS < count; it += 8 * GROUPS) {
    float2 x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) x[u] = src[(long long)(it + u * GROUPS) * ENT];
#pragma unroll
    for (int u = 0; u < 8; ++u) df_add(hi[u & 1], lo[u & 1], x[u].x, x[u].y);
  }
  for (; it < count; it += GROUPS) {
    const float2 x = src[(long long)it * ENT];
    df_add(hi[0], lo[0], x.x, x.y);
  }
  df_add(hi[0], lo[0], hi[1], lo[1]);
  part[threadIdx.x] = make_float2(hi[0], lo[0]);
  __syncthreads();
  if (g == 0) {
    float vh = 0.f, vl = 0.f;
    for (int q = 0; q < GROUPS; ++q) df_add(vh, vl, part[q * EPC + threadIdx.x].x, part[q * EPC + threadIdx.x].y);
    a.gram_t[(long long)t * ENT + e] = make_float2(vh, vl);
  }
}

// Double-float values (hi + lo, |lo| <= ulp(hi) / 2 after normalisation) for
// the Gram-Schmidt recurrence.  fp64 runs at a small fraction of the fp32
// rate on this GPU; these operations keep about 44 bits on the fp32 pipes.
struct Dd {
  float hi, lo;
};
__device__ __forceinline__ Dd dd_norm(float s, float e) {   // Fast2Sum, |s| >= |e|
  const float h = __fadd_rn(s, e);
  return {h, __fsub_rn(e, __fsub_rn(h, s))};
}
__device__ __forceinline__ Dd dd_add(Dd a, Dd b) {
  const float s = __fadd_rn(a.hi, b.hi);
  const float bp = __fsub_rn(s, a.hi);
  const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bp)), __fsub_rn(b.hi, bp));
  return dd_norm(s, __fadd_rn(e, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ Dd dd_mul(Dd a, Dd b) {
  const float p = __fmul_rn(a.hi, b.hi);
  float e = fmaf(a.hi, b.hi, -p);
  e = fmaf(a.hi, b.lo, e);
  e = fmaf(a.lo, b.hi, e);
  return dd_norm(p, e);
}
__device__ __forceinline__ Dd dd_neg(Dd a) { return {-a.hi, -a.lo}; }
__device__ __forceinline__ Dd dd_of(float2 v) { return dd_norm(v.x, v.y); }

// sc = 1 / (sqrt(nn) + eps) for the squared column norm nn.  For eps = 0 and
// nn > 0 it is 1 / sqrt(nn): an rsqrtf seed y refined by one Newton step for
// f(y) = 1 / y^2 - nn, y <- y + y (1 - nn y^2) / 2, with the residual in
// double-float (the seed's ~23 correct bits become ~44).  Otherwise the
// square root (sqrtf seed, one Newton step s <- s + (nn - s^2) / (2 s)) and
// the reciprocal (1 / d seed, one Newton step z <- z + z (1 - d z)) are
// refined the same way.  A zero denominator gives inf, and then NaN for a
// zero column with eps = 0, as the oracle.
__device__ __forceinline__ Dd dd_gs_scale(Dd nn, float eps) {
  const Dd one = {1.f, 0.f};
  if (eps == 0.f && nn.hi > 0.f && nn.hi < 3e38f) {
    const Dd y = {rsqrtf(nn.hi), 0.f};
    const Dd r = dd_add(one, dd_neg(dd_mul(nn, dd_mul(y, y))));
    return dd_add(y, dd_mul(y, {0.5f * r.hi, 0.5f * r.lo}));
  }
  if (nn.hi != nn.hi) return nn;   // NaN
  Dd sq = {0.f, 0.f};
  if (nn.hi > 0.f) {
    const Dd s0 = {sqrtf(nn.hi), 0.f};
    if (s0.hi < 3e38f) {
      const Dd r = dd_add(nn, dd_neg(dd_mul(s0, s0)));
      sq = dd_add(s0, {__fdiv_rn(r.hi, 2.f * s0.hi), 0.f});
    } else {
      sq = s0;
    }
  }
  const Dd den = dd_add(sq, {eps, 0.f});
  if (den.hi == 0.f) return {__int_as_float(0x7f800000), 0.f};
  const Dd z = {__frcp_rn(den.hi), 0.f};
  if (!(z.hi > 0.f)) return z;     // den overflowed: sc rounds to 0
  const Dd r = dd_add(one, dd_neg(dd_mul(den, z)));
  return dd_add(z, dd_mul(z, r));
}

// Largest deviation of the first sweep's Gram matrix from I for which the
// second sweep is skipped (its T would differ from I by about as much).
constexpr float kGsSkip = 1e-5f;

// One CTA per tensor, on the tensor's Gram matrix G (k_gram_sum): modified
// Gram-Schmidt with epsilon on the coefficient matrix T (X_out = X T), in
// double-float with T and H = G T in shared memory.  Step i, with t_i still
// unscaled: ||x_i||^2 = t_i . h_i, sc_i = 1 / (||x_i|| + eps); every later
// column j loses its projection on the normalised x_i: t_j -= c t_i and
// h_j -= c h_i with c = sc_i^2 (t_i . h_j).  A step touches only the rows
// that can be nonzero (t_i has none below row i, H none at or past rank r).
// Ranks up to 8 run the steps on one warp (__syncwarp between steps), 16 and
// 32 on the CTA (__syncthreads), the work of a step spread over its threads.
// The column scalings are applied to T at the end (t_i is not read again
// after its own step).  `sweep` is 0 for the first sweep and 1 for the
// re-orthogonalising one.
template <int RP>
__device__ __forceinline__ void solve_tensor(const StepArgs& a, const float2* __restrict__ gram_in, int t,
                                             int is_q, int sweep, float* __restrict__ tout) {
  constexpr int ENT = RP * RP;
  constexpr int LD = RP + 1;                                // padded column stride
  // the steps run on one warp for ranks up to 8 and on the CTA above, thread
  // (j, p) owning rows [p R, p R + R) of column j; the PARTS threads of a
  // column add their partial dot products with shuffles
  constexpr int TEAM = ENT <= 64 ? 32 : kThreads;
  constexpr int R = ENT > TEAM ? ENT / TEAM : 1;
  constexpr int PARTS = RP / R;
  __shared__ Dd H[RP * LD];   // H[j * LD + k] = row k of column j of G T
  __shared__ Dd T[RP * LD];   // T[j * LD + k] = row k of column j
  __shared__ Dd scal[RP];
  const TensorDesc td = a.tensors[t];
  const int count = is_q ? a.gsq_count[t] : a.gsp_count[t];
  if (count == 0) return;
  __shared__ float devw[kThreads / 32];
  float dev = 0.f;   // max |G - I| over the rank's block
  for (int idx = threadIdx.x; idx < ENT; idx += kThreads) {
    const int k = idx / RP, j = idx % RP;   // G is symmetric: entry (k, j)
    H[j * LD + k] = dd_of(gram_in[(long long)t * ENT + idx]);
    T[j * LD + k] = {(k == j && j < td.r) ? 1.f : 0.f, 0.f};
    if (k < td.r && j < td.r) dev = fmaxf(dev, fabsf(H[j * LD + k].hi - (k == j ? 1.f : 0.f)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dev = fmaxf(dev, __shfl_xor_sync(0xffffffffu, dev, o));
  if ((threadIdx.x & 31) == 0) devw[threadIdx.x >> 5] = dev;
  __syncthreads();
  // the second sweep re-orthogonalises only what the first left off: when
  // the first sweep's output is already orthonormal to kGsSkip, its T is I
  if (sweep == 1) {
    float dmax = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) dmax = fmaxf(dmax, devw[w]);
    if (dmax <= kGsSkip) {
      float* Tout = tout + (long long)t * RP * RP;
      for (int idx = threadIdx.x; idx < ENT; idx += kThreads) {
        const int k = idx / RP, jj = idx % RP;
        Tout[idx] = (k == jj && jj < td.r) ? 1.f : 0.f;
      }
      return;
    }
  }
  if (threadIdx.x >= TEAM) return;
  const int r = td.r;
  const int lane = threadIdx.x & 31;
  const int j = threadIdx.x / PARTS, p = threadIdx.x % PARTS;
  const bool own = j < RP;
  for (int i = 0; i < r; ++i) {
    // ||x_i||^2 = t_i . h_i, by every warp (t_i has no entries below row i)
    Dd nn = (lane <= i && lane < RP) ? dd_mul(T[i * LD + lane], H[i * LD + lane]) : Dd{0.f, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      nn = dd_add(nn, {__shfl_xor_sync(0xffffffffu, nn.hi, o), __shfl_xor_sync(0xffffffffu, nn.lo, o)});
    const Dd sc = dd_gs_scale(nn, a.eps);
    if (threadIdx.x == 0) scal[i] = sc;
    Dd d = {0.f, 0.f};
    const bool upd = own && j > i && j < r;
    if (upd) {
#pragma unroll
      for (int q = 0; q < R; ++q) {
        const int k = p * R + q;
        if (k <= i) d = dd_add(d, dd_mul(T[i * LD + k], H[j * LD + k]));
      }
    }
#pragma unroll
    for (int o = PARTS / 2; o > 0; o >>= 1)
      d = dd_add(d, {__shfl_xor_sync(0xffffffffu, d.hi, o), __shfl_xor_sync(0xffffffffu, d.lo, o)});
    if (upd) {
      const Dd nc = dd_neg(dd_mul(dd_mul(d, sc), sc));
#pragma unroll
      for (int q = 0; q < R; ++q) {
        const int k = p * R + q;
        if (k <= i) T[j * LD + k] = dd_add(T[j * LD + k], dd_mul(nc, T[i * LD + k]));
        if (k < r) H[j * LD + k] = dd_add(H[j * LD + k], dd_mul(nc, H[i * LD + k]));
      }
    }
    if constexpr (TEAM == 32) __syncwarp(); else __syncthreads();
  }
  float* Tout = tout + (long long)t * RP * RP;
  for (int idx = threadIdx.x; idx < ENT; idx += TEAM) {
    const int k = idx / RP, jj = idx % RP;
    float v = 0.f;
    if (jj < r) {
      const Dd x = dd_mul(T[jj * LD + k], scal[jj]);
      v = __fadd_rn(x.hi, x.lo);
    }
    Tout[idx] = v;
  }
}

template <int RP>
__global__ void __launch_bounds__(kThreads) k_solve(const StepArgs a, const float2* __restrict__ gram_in,
                                                    int is_q, int sweep) {
  if (a.ctrl->flag) return;
  solve_tensor<RP>(a, gram_in, blockIdx.x, is_q, sweep, a.tmat);
}

// dst rows = src rows x T.  Each thread computes OPT consecutive output
// columns of one row (KG threads per row), each as the increasing-l FMA chain
// over the row's RP inputs.  P (row-major) puts a row's KG threads next to
// each other; Q (k-major) puts 32 consecutive rows in a warp, so its column
// reads and writes are coalesced.
// IMG (P, ranks 16 and 32): also write the output rows into P's operand
// images (row and chunk), as k_images mode 0 does.
template <int RP, bool IMG = false>
__device__ __forceinline__ void apply_item(const StepArgs& a, int it, const float* __restrict__ src,
                                           float* __restrict__ dst, int is_q, long long half_off,
                                           const float* __restrict__ tsrc, float* T) {
  constexpr int OPT = RP >= 4 ? 4 : RP;
  constexpr int KG = RP / OPT;
  const GsItem* items = is_q ? a.gsq_items : a.gsp_items;
  const GsItem gi = items[it];
  const TensorDesc td = a.tensors[gi.t];
  const long long base = is_q ? td.q_off : td.p_off;
  __syncthreads();
  for (int idx = threadIdx.x; idx < RP * RP; idx += kThreads) T[idx] = __ldcg(tsrc + (long long)gi.t * RP * RP + idx);
  __syncthreads();
  const int span = is_q ? (gi.nrows + 31) / 32 * 32 * KG : gi.nrows * KG;
  for (int idx = threadIdx.x; idx < span; idx += kThreads) {
    const int rr = is_q ? (idx / (32 * KG)) * 32 + (idx & 31) : idx / KG;
    const int kg = is_q ? (idx >> 5) % KG : idx % KG;
    if (rr >= gi.nrows) continue;
    const long long row = gi.row0 + rr;
    float x[RP], y[OPT];
    if (is_q) {
#pragma unroll
      for (int k = 0; k < RP; ++k) x[k] = src[base + (long long)k * td.m + row];
    } else {
      load_row<RP>(src + base + row * RP, x);
    }
#pragma unroll
    for (int o = 0; o < OPT; ++o) y[o] = 0.f;
#pragma unroll
    for (int l = 0; l < RP; ++l) {
      if constexpr (OPT == 4) {
        const float4 tv = *reinterpret_cast<const float4*>(&T[l * RP + kg * 4]);
        y[0] = fmaf(x[l], tv.x, y[0]);
        y[1] = fmaf(x[l], tv.y, y[1]);
        y[2] = fmaf(x[l], tv.z, y[2]);
        y[3] = fmaf(x[l], tv.w, y[3]);
      } else {
#pragma unroll
        for (int o = 0; o < OPT; ++o) y[o] = fmaf(x[l], T[l * RP + o], y[o]);
      }
    }
    if constexpr (IMG) {
      if (!is_q) {
#pragma unroll
        for (int o = 0; o < OPT; ++o) img_put_p<RP>(a, td, row, kg * OPT + o, y[o], true);
      }
    }
    if (is_q) {
#pragma unroll
      for (int o = 0; o < OPT; ++o) dst[half_off + base + (long long)(kg * OPT + o) * td.m + row] = y[o];
    } else if constexpr (OPT == 4) {
      *reinterpret_cast<float4*>(dst + half_off + base + row * RP + kg * 4) = make_float4(y[0], y[1], y[2], y[3]);
    } else {
#pragma unroll
      for (int o = 0; o < OPT; ++o) dst[half_off + base + row * RP + o] = y[o];
    }
  }
}

// dst_half >= 0: write into half (cur ^ 1) of Pf/Qf (dst is the base).
// tsrc: the transforms (a.tmat when NULL).  img (P, ranks 16 and 32): also
// write P's operand images (k_images mode 0).
template <int RP>
__global__ void __launch_bounds__(kThreads) k_apply(const StepArgs a, const float* __restrict__ src,
                                                    float* __restrict__ dst, int is_q, int dst_half,
                                                    const float* __restrict__ tsrc, int img) {
  __shared__ __align__(16) float T[RP * RP];
  const int n_items = is_q ? a.n_gsq : a.n_gsp;
  if (a.ctrl->flag) return;
  long long half_off = 0;
  if (dst_half >= 0) half_off = (long long)(a.ctrl->cur ^ 1) * (is_q ? a.q_total : a.p_total);
  if (img && a.ctrl->timeout) img = 0;   // not committed: keep the images
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    if (RP >= 16 && img)
      apply_item<RP, true>(a, it, src, dst, is_q, half_off, tsrc ? tsrc : a.tmat, T);
    else
      apply_item<RP>(a, it, src, dst, is_q, half_off, tsrc ? tsrc : a.tmat, T);
  }
}

// ---------------------------------------------------------------------------
// Fused Gram-Schmidt stage, for buckets whose tensors have few row items
// (small buckets, where the stage is a chain of short launches): every CTA
// writes its items' Gram partials and counts them per tensor with an atomic;
// the CTA whose count completes a tensor (no CTA waits for another) adds the
// tensor's partials in item order and runs the solve.  The stage is then
// three launches instead of eight: k_gs_first (Gram of X, solve of sweep 0),
// k_gs_second (X T into the scratch, its Gram, solve of sweep 1 into tmat2),
// and k_apply with tmat2.  Counters are left at zero for the next launch.
// ---------------------------------------------------------------------------
template <int RP>
__device__ __forceinline__ void gs_count_and_solve(const StepArgs& a, int it, int is_q, int sweep,
                                                   float* __restrict__ tout, int* last_s) {
  constexpr int ENT = RP * RP;
  const GsItem gi = (is_q ? a.gsq_items : a.gsp_items)[it];
  const int t = gi.t;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int cnt = is_q ? a.gsq_count[t] : a.gsp_count[t];
    *last_s = (atomicAdd(&a.gs_cnt[t], 1) == cnt - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!*last_s) return;
  __threadfence();
  const int first = is_q ? a.gsq_first[t] : a.gsp_first[t];
  const int count = is_q ? a.gsq_count[t] : a.gsp_count[t];
  for (int e = threadIdx.x; e < ENT; e += kThreads) {
    float hi = 0.f, lo = 0.f;
    // in item order, eight loads in flight
    int i = 0;
    for (; i + 8 <= count; i += 8) {
      float2 x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = __ldcg(a.gram + (long long)(first + i + u) * ENT + e);
#pragma unroll
      for (int u = 0; u < 8; ++u) df_add(hi, lo, x[u].x, x[u].y);
    }
    for (; i < count; ++i) {
      const float2 x = __ldcg(a.gram + (long long)(first + i) * ENT + e);
      df_add(hi, lo, x.x, x.y);
    }
    a.gram_t[(long long)t * ENT + e] = make_float2(hi, lo);
  }
  __syncthreads();
  solve_tensor<RP>(a, a.gram_t, t, is_q, sweep, tout);
  __syncthreads();
  if (threadIdx.x == 0) a.gs_cnt[t] = 0;
}

template <int RP>
__global__ void __launch_bounds__(kThreads) k_gs_first(const StepArgs a, const float* __restrict__ src,
                                                       float* __restrict__ dense_out, int is_q, int from_parts) {
  __shared__ float tile[kGramTile][RP + 1];
  __shared__ float2 red[kThreads];
  __shared__ int last_s;
  const int n_items = is_q ? a.n_gsq : a.n_gsp;
  if (a.ctrl->flag) return;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    gram_item<RP>(a, it, src, dense_out, is_q, from_parts, a.gram, tile, red);
    gs_count_and_solve<RP>(a, it, is_q, 0, a.tmat, &last_s);
  }
}

template <int RP>
__global__ void __launch_bounds__(kThreads) k_gs_second(const StepArgs a, const float* __restrict__ src,
                                                        float* __restrict__ mid, int is_q) {
  __shared__ float tile[kGramTile][RP + 1];
  __shared__ float2 red[kThreads];
  __shared__ __align__(16) float T[RP * RP];
  __shared__ int last_s;
  const int n_items = is_q ? a.n_gsq : a.n_gsp;
  if (a.ctrl->flag) return;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    apply_item<RP>(a, it, src, mid, is_q, 0, a.tmat, T);
    __syncthreads();   // the CTA's rows of X T are visible to its Gram
    gram_item<RP>(a, it, mid, nullptr, is_q, 0, a.gram, tile, red);
    gs_count_and_solve<RP>(a, it, is_q, 1, a.tmat2, &last_s);
  }
}

// ---------------------------------------------------------------------------
// The fused stage in one cooperative launch (all CTAs resident): the P_raw
// sum (when asked), k_gs_first's, k_gs_second's and the final apply's work
// in the same order and on the same items, with grid-wide barriers where the
// launches ended.  Each CTA takes the same items in every phase, so the rows
// a phase reads back (X, X T) are the CTA's own writes; the transforms come
// from the tensors' last CTAs through L2.
//
// grid_barrier: CTA k of the launch's b-th barrier adds one to *bar (zeroed
// before the launch) and waits until it reaches b x gridDim.x.  The wait is
// bounded: after kBarrierPolls polls it sets the step's timeout flag (the
// commit then leaves the state unchanged and the step reports PSGD_ETIMEOUT)
// and the CTA returns.
// ---------------------------------------------------------------------------
constexpr long kBarrierPolls = 1L << 22;

__device__ __forceinline__ bool grid_barrier(const StepArgs& a, unsigned int* bar, unsigned int target, int* ok_s) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    int ok = 0;
    for (long i = 0; i < kBarrierPolls; ++i) {
      unsigned int v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar) : "memory");
      if (v >= target) {
        ok = 1;
        break;
      }
      __nanosleep(32);
    }
    if (!ok) atomicExch(&a.ctrl->timeout, 1);
    __threadfence();
    *ok_s = ok;
  }
  __syncthreads();
  return *ok_s != 0;
}

template <int RP>
__global__ void __launch_bounds__(kThreads) k_gs_coop(const StepArgs a, const float* __restrict__ src,
                                                      float* __restrict__ dense_out, int is_q, int from_parts,
                                                      float* __restrict__ mid, float* __restrict__ dst,
                                                      int dst_half, int do_psum, unsigned int* bar, int img,
                                                      unsigned int skew) {
  __shared__ float tile[kGramTile][RP + 1];
  __shared__ float2 red[kThreads];
  __shared__ __align__(16) float T[RP * RP];
  __shared__ int last_s, ok_s;
  const int n_items = is_q ? a.n_gsq : a.n_gsp;
  if (a.ctrl->flag) return;   // the same for every CTA: none waits at a barrier
  // skew (tests of the bounded wait): the first barrier waits for skew more
  // arrivals than there are CTAs, so every CTA gives up and reports a timeout
  unsigned int nb = 0, extra = skew;
  if (do_psum) {
    for (int it = blockIdx.x; it < a.n_ps; it += gridDim.x) psum_item<RP>(a, it);
    if (!grid_barrier(a, bar, ++nb * gridDim.x + extra, &ok_s)) return;
    extra = 0;
  }
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    gram_item<RP>(a, it, src, dense_out, is_q, from_parts, a.gram, tile, red);
    gs_count_and_solve<RP>(a, it, is_q, 0, a.tmat, &last_s);
  }
  if (!grid_barrier(a, bar, ++nb * gridDim.x + extra, &ok_s)) return;
  const float* x = dense_out ? dense_out : src;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    apply_item<RP>(a, it, x, mid, is_q, 0, a.tmat, T);
    __syncthreads();   // the CTA's rows of X T are visible to its Gram
    gram_item<RP>(a, it, mid, nullptr, is_q, 0, a.gram, tile, red);
    gs_count_and_solve<RP>(a, it, is_q, 1, a.tmat2, &last_s);
  }
  if (!grid_barrier(a, bar, ++nb * gridDim.x, &ok_s)) return;
  long long half_off = 0;
  if (dst_half >= 0) half_off = (long long)(a.ctrl->cur ^ 1) * (is_q ? a.q_total : a.p_total);
  if (img && *reinterpret_cast<volatile int*>(&a.ctrl->timeout)) img = 0;   // not committed: keep the images
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    if (RP >= 16 && img)
      apply_item<RP, true>(a, it, mid, dst, is_q, half_off, a.tmat2, T);
    else
      apply_item<RP>(a, it, mid, dst, is_q, half_off, a.tmat2, T);
  }
}

}  // namespace psgd
