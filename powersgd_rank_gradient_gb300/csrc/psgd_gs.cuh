// Gram-Schmidt stage of the PowerSGD hook step (P and the fresh Q), templated
// on the padded rank RP.  Kept apart from the streaming passes
// (psgd_kernels.cuh) so that the two evolve separately.
#pragma once

#include "psgd_kernels.cuh"

namespace psgd {

// ---------------------------------------------------------------------------
// Gram-Schmidt stage.
//
// "PowerSGD Hooks" step 3.4 orthogonalises P column by column; "PowerSGD
// State" item 4 adds epsilon to each column norm.  Every Gram-Schmidt
// operation is a column operation, so the result is X T for an RP x RP upper
// triangular T that depends only on the Gram matrix G = X^T X.  The stage
// therefore (1) reduces G over row blocks in fp64 (k_gram), (2) runs modified
// Gram-Schmidt with epsilon symbolically on G to get T (k_solve, one CTA per
// tensor, fp64), (3) applies X T (k_apply).  It runs twice (the second sweep
// re-orthogonalises the first sweep's output), which keeps P^T P = I to fp32
// rounding even when X is ill conditioned.
// ---------------------------------------------------------------------------
// P_raw = sum of pass 1's column-tile partials, in tile order (the Gram stage
// then reads dense rows).  Each work item is a chunk of one tensor's rows x RP
// values, four per thread.
template <int RP>
__global__ void __launch_bounds__(kThreads) k_psum(const StepArgs a) {
  if (a.ctrl->flag) return;
  for (int it = blockIdx.x; it < a.n_ps; it += gridDim.x) {
    const GsItem gi = a.ps_items[it];
    const TensorDesc td = a.tensors[gi.t];
    const long long len = (long long)td.n * RP;
    const float* src = a.praw_part + td.pp_off;
    const int f = gi.row0 + threadIdx.x * 4;
    if (f >= gi.row0 + gi.nrows) continue;
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

constexpr int kGramTile = 128;

// Rows of P live as column-tile partials (nparts > 1) or dense (nparts == 1).
template <int RP>
__global__ void __launch_bounds__(kThreads) k_gram(const StepArgs a, const float* __restrict__ src,
                                                   float* __restrict__ dense_out, int is_q,
                                                   int from_parts, double* __restrict__ gram_out) {
  __shared__ float tile[kGramTile][RP + 1];
  __shared__ double red[kThreads];
  constexpr int PAIRS = RP * RP;
  constexpr int PPT = PAIRS > kThreads ? PAIRS / kThreads : 1;   // pairs per thread
  constexpr int GROUPS = PAIRS >= kThreads ? 1 : kThreads / PAIRS;
  const GsItem* items = is_q ? a.gsq_items : a.gsp_items;
  const int n_items = is_q ? a.n_gsq : a.n_gsp;
  if (a.ctrl->flag) return;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const GsItem gi = items[it];
    const TensorDesc td = a.tensors[gi.t];
    const long long base = is_q ? td.q_off : td.p_off;
    const int pair0 = (threadIdx.x % (PAIRS >= kThreads ? kThreads : PAIRS)) * PPT;
    const int grp = PAIRS >= kThreads ? 0 : threadIdx.x / PAIRS;
    double dacc[PPT];
#pragma unroll
    for (int u = 0; u < PPT; ++u) dacc[u] = 0.0;
    for (int r0 = 0; r0 < gi.nrows; r0 += kGramTile) {
      const int rows = min(kGramTile, gi.nrows - r0);
      __syncthreads();
      for (int idx = threadIdx.x; idx < rows * RP; idx += kThreads) {
        const int rr = idx / RP, k = idx % RP;
        const long long row = gi.row0 + r0 + rr;
        float v;
        if (from_parts) {
          v = 0.f;
          for (int c = 0; c < td.ctiles1; ++c) v += src[td.pp_off + ((long long)c * td.n + row) * RP + k];
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
        float facc = 0.f;
        int cnt = 0;
        for (int rr = grp; rr < rows; rr += GROUPS) {
          facc = fmaf(tile[rr][pa], tile[rr][pb], facc);
          if (++cnt == 8) { dacc[u] += (double)facc; facc = 0.f; cnt = 0; }
        }
        dacc[u] += (double)facc;
      }
    }
    // reduce the row groups
#pragma unroll
    for (int u = 0; u < PPT; ++u) {
      __syncthreads();
      red[threadIdx.x] = dacc[u];
      __syncthreads();
      if (threadIdx.x < (PAIRS >= kThreads ? kThreads : PAIRS)) {
        double s = 0.0;
        for (int g = 0; g < GROUPS; ++g) s += red[threadIdx.x + g * (PAIRS >= kThreads ? kThreads : PAIRS)];
        gram_out[(long long)it * PAIRS + pair0 + u] = s;
      }
    }
  }
}

// One CTA per tensor: the whole CTA adds up the item Gram matrices (for
// ranks up to 8 each entry split over SPLIT threads, for 16 and 32 several
// entries per thread; four accumulators each, combined in a fixed order),
// then runs modified Gram-Schmidt with epsilon on the
// coefficient matrix T (X_out = X T), in fp64 with T and H = G T in shared
// memory.  Step i, with t_i still unscaled: ||x_i||^2 = t_i . h_i, sc_i =
// 1 / (||x_i|| + eps); every later column j loses its projection on the
// normalised x_i: t_j -= c t_i and h_j -= c h_i with c = sc_i^2 (t_i . h_j).
// The column scalings are applied to T at the end (t_i is not read again
// after its own step).  Thread (j, p) of the TEAM owns rows [p R, p R + R)
// of column j; the PARTS threads of a column add their partial dot products
// with shuffles.  Ranks up to 8 fit one warp (steps end with __syncwarp),
// larger ones use the whole CTA (__syncthreads).
template <int RP>
__global__ void __launch_bounds__(kThreads) k_solve(const StepArgs a, const double* __restrict__ gram_in,
                                                    int is_q, int only_init) {
  constexpr int ENT = RP * RP;
  constexpr int SPLIT = ENT >= kThreads ? 1 : kThreads / ENT;
  constexpr int TEAM = ENT <= 64 ? 32 : kThreads;
  constexpr int R = ENT > TEAM ? ENT / TEAM : 1;            // rows per thread
  constexpr int PARTS = RP / R;                             // threads per column
  constexpr int LD = RP + 1;                                // padded column stride
  __shared__ double H[RP * LD];   // H[j * LD + k] = row k of column j of G T
  __shared__ double T[RP * LD];   // T[j * LD + k] = row k of column j
  __shared__ double scal[RP];
  __shared__ double part[kThreads];
  const int t = blockIdx.x;
  if (a.ctrl->flag) return;
  const TensorDesc td = a.tensors[t];
  const int first = is_q ? a.gsq_first[t] : a.gsp_first[t];
  const int count = is_q ? a.gsq_count[t] : a.gsp_count[t];
  if (count == 0) return;
  if constexpr (ENT >= kThreads) {
    // EPT entries per thread, four chains each, all in flight together
    constexpr int EPT = ENT / kThreads;
    double acc[EPT][4];
#pragma unroll
    for (int e = 0; e < EPT; ++e)
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[e][u] = 0.0;
    int it = 0;
    for (; it + 4 <= count; it += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < EPT; ++e)
          acc[e][u] += gram_in[(long long)(first + it + u) * ENT + threadIdx.x + e * kThreads];
    }
    for (; it < count; ++it)
#pragma unroll
      for (int e = 0; e < EPT; ++e) acc[e][0] += gram_in[(long long)(first + it) * ENT + threadIdx.x + e * kThreads];
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const int idx = threadIdx.x + e * kThreads;
      const int k = idx / RP, j = idx % RP;   // G is symmetric: entry (k, j)
      H[j * LD + k] = (acc[e][0] + acc[e][1]) + (acc[e][2] + acc[e][3]);
      T[j * LD + k] = (k == j && j < td.r) ? 1.0 : 0.0;
    }
    __syncthreads();
  } else {
    // SPLIT threads per entry, four chains each, combined in a fixed order
    const int idx = threadIdx.x / SPLIT;
    const int sp = threadIdx.x % SPLIT;
    double s0 = 0.0, s1 = 0.0, s2 = 0.0, s3 = 0.0;
    if (idx < ENT) {
      int it = sp;
      for (; it + 3 * SPLIT < count; it += 4 * SPLIT) {
        s0 += gram_in[(long long)(first + it) * ENT + idx];
        s1 += gram_in[(long long)(first + it + SPLIT) * ENT + idx];
        s2 += gram_in[(long long)(first + it + 2 * SPLIT) * ENT + idx];
        s3 += gram_in[(long long)(first + it + 3 * SPLIT) * ENT + idx];
      }
      for (; it < count; it += SPLIT) s0 += gram_in[(long long)(first + it) * ENT + idx];
    }
    part[threadIdx.x] = (s0 + s1) + (s2 + s3);
    __syncthreads();
    if (sp == 0 && idx < ENT) {
      double v = 0.0;
      for (int q = 0; q < SPLIT; ++q) v += part[threadIdx.x + q];
      const int k = idx / RP, j = idx % RP;   // G is symmetric: entry (k, j)
      H[j * LD + k] = v;
      T[j * LD + k] = (k == j && j < td.r) ? 1.0 : 0.0;
    }
    __syncthreads();
  }
  if (threadIdx.x >= TEAM) return;
  const int r = td.r;
  const double eps = (double)a.eps;
  const int lane = threadIdx.x & 31;
  const int j = threadIdx.x / PARTS, p = threadIdx.x % PARTS;
  const bool own = j < RP;
  for (int i = 0; i < r; ++i) {
    // ||x_i||^2 = t_i . h_i, by every warp (t_i has no entries below row i)
    double nn = (lane <= i) ? T[i * LD + lane] * H[i * LD + lane] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nn += __shfl_xor_sync(0xffffffffu, nn, o);
    // sc = 1 / (sqrt(nn) + eps).  For eps = 0 and nn > 0 it is 1 / sqrt(nn):
    // an fp32 rsqrtf seed refined by one Newton-Raphson step for
    // f(y) = 1 / y^2 - nn (y <- y (3 - nn y^2) / 2), which takes the seed's
    // ~24 correct bits to ~48 with three dependent fp64 operations instead of
    // an fp64 square root and division.  A zero or negative nn, and eps > 0,
    // take the direct expression (eps = 0 with a zero column gives inf and
    // then NaN, as the oracle).
    double sc;
    if (eps == 0.0 && nn > 0.0 && nn < 1e300) {
      const double y = (double)rsqrtf((float)nn);
      sc = y * (1.5 - 0.5 * nn * y * y);
    } else {
      sc = 1.0 / (sqrt(fmax(nn, 0.0)) + eps);
    }
    if (threadIdx.x == 0) scal[i] = sc;
    double d = 0.0;
    if (own && j > i && j < r) {
#pragma unroll
      for (int q = 0; q < R; ++q) {
        const int k = p * R + q;
        d += T[i * LD + k] * H[j * LD + k];
      }
    }
#pragma unroll
    for (int o = PARTS / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (own && j > i && j < r) {
      const double c = d * sc * sc;
#pragma unroll
      for (int q = 0; q < R; ++q) {
        const int k = p * R + q;
        T[j * LD + k] -= c * T[i * LD + k];
        H[j * LD + k] -= c * H[i * LD + k];
      }
    }
    if constexpr (TEAM == 32) __syncwarp(); else __syncthreads();
  }
  float* Tout = a.tmat + (long long)t * RP * RP;
  for (int idx = threadIdx.x; idx < ENT; idx += TEAM) {
    const int k = idx / RP, jj = idx % RP;
    Tout[idx] = (float)(jj < r ? T[jj * LD + k] * scal[jj] : 0.0);
  }
}

// dst rows = src rows x T (thread per row).
template <int RP>
__global__ void __launch_bounds__(kThreads) k_apply(const StepArgs a, const float* __restrict__ src,
                                                    float* __restrict__ dst, int is_q, int dst_half) {
  __shared__ float T[RP * RP];
  const GsItem* items = is_q ? a.gsq_items : a.gsp_items;
  const int n_items = is_q ? a.n_gsq : a.n_gsp;
  if (a.ctrl->flag) return;
  // dst_half >= 0: write into half (cur ^ 1) of Pf/Qf (dst is the base)
  long long half_off = 0;
  if (dst_half >= 0) half_off = (long long)(a.ctrl->cur ^ 1) * (is_q ? a.q_total : a.p_total);
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const GsItem gi = items[it];
    const TensorDesc td = a.tensors[gi.t];
    const long long base = is_q ? td.q_off : td.p_off;
    __syncthreads();
    for (int idx = threadIdx.x; idx < RP * RP; idx += kThreads) T[idx] = a.tmat[(long long)gi.t * RP * RP + idx];
    __syncthreads();
    for (int rr = threadIdx.x; rr < gi.nrows; rr += kThreads) {
      const long long row = gi.row0 + rr;
      float x[RP], y[RP];
      // P is row-major (rows x RP); Q is k-major (element (j, k) at k * m + j)
      const long long rs = is_q ? 1 : RP;
      const long long ks = is_q ? td.m : 1;
#pragma unroll
      for (int k = 0; k < RP; ++k) { x[k] = src[base + row * rs + k * ks]; y[k] = 0.f; }
#pragma unroll
      for (int l = 0; l < RP; ++l)
#pragma unroll
        for (int k = 0; k < RP; ++k) y[k] = fmaf(x[l], T[l * RP + k], y[k]);
#pragma unroll
      for (int k = 0; k < RP; ++k) dst[half_off + base + row * rs + k * ks] = y[k];
    }
  }
}

}  // namespace psgd
