// Rank-independent kernels: the replica mean of uncompressed elements, the
// end-of-step commit, and the standard-normal draw of a fresh Q.
#include <math.h>

#include "psgd_kernels.cuh"
#include "psgd_launch.h"

namespace psgd {

// out[e] = (1/W) sum_w g_w[e] * s over the listed segments.
// "DDP Communication Hooks", "PowerSGD Hooks" step 2 (uncompressed tensors
// are allreduced as a batch, without compression) and the vanilla-allreduce
// note (every element before start_powerSGD_iter); "Default Communication
// Hooks", allreduce_hook: the allreduce result is the mean over workers.
template <int WT, typename GT>
__global__ void __launch_bounds__(kThreads) k_mean(const StepArgs a, const Segment* __restrict__ segs,
                                                   int nsegs) {
  const int W = WT > 0 ? WT : a.W;
  int bad = 0;
  for (int it = blockIdx.x; it < nsegs; it += gridDim.x) {
    const Segment sg = segs[it];
    int start = 0;
    if (a.vec_ok && (sg.off % 4 == 0)) {
      const int n4 = sg.len / 4;
      for (int j = threadIdx.x; j < n4; j += kThreads) {
        const long long o = sg.off + 4LL * j;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll(WT > 0 ? WT : 1)
        for (int w = 0; w < W; ++w) {
          float v[4];
          load_grad<4, GT>(reinterpret_cast<const GT*>(a.grads.p[w]) + o, v);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float x = v[c] * a.scale;
            bad |= !isfinite(x);
            acc[c] += x;
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c] *= a.invW;
        store_f<4>(a.out + o, acc);
      }
      start = n4 * 4;
    }
    for (int j = start + threadIdx.x; j < sg.len; j += kThreads) {
      const long long o = sg.off + j;
      float acc = 0.f;
      for (int w = 0; w < W; ++w) {
        float v[1];
        load_grad<1, GT>(reinterpret_cast<const GT*>(a.grads.p[w]) + o, v);
        const float x = v[0] * a.scale;
        bad |= !isfinite(x);
        acc += x;
      }
      a.out[o] = acc * a.invW;
    }
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(&a.ctrl->flag, 1);
}

void launch_mean(const StepArgs& a, const Segment* segs, int nsegs, int grid, cudaStream_t s) {
  if (nsegs == 0) return;
  auto go = [&](auto tag) {
    using GT = decltype(tag);
    switch (a.W) {
      case 1: k_mean<1, GT><<<grid, kThreads, 0, s>>>(a, segs, nsegs); break;
      case 2: k_mean<2, GT><<<grid, kThreads, 0, s>>>(a, segs, nsegs); break;
      case 4: k_mean<4, GT><<<grid, kThreads, 0, s>>>(a, segs, nsegs); break;
      case 8: k_mean<8, GT><<<grid, kThreads, 0, s>>>(a, segs, nsegs); break;
      default: k_mean<0, GT><<<grid, kThreads, 0, s>>>(a, segs, nsegs); break;
    }
  };
  if (a.gtype == 1)
    go(__half());
  else if (a.gtype == 2)
    go(__nv_bfloat16());
  else
    go(0.0f);
}

// End of a step: a step that saw no inf/NaN makes the next half of the
// double-buffered state current; a skipped step leaves everything as it was
// (torch.cuda.amp GradScaler: a step with inf/NaN gradients is skipped).
// A bounded wait that gave up (ctrl->timeout) also leaves the state as it was
// and reports status 2.
__global__ void k_commit(Ctrl* ctrl, int compressed, int* status) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    const int bad = ctrl->flag;
    const int late = ctrl->timeout;
    if (!bad && !late && compressed) {
      ctrl->cur ^= 1;
      ctrl->warm_valid = 1;
    }
    *status = late ? 2 : (bad ? 1 : 0);
  }
}

void launch_commit(Ctrl* ctrl, int compressed, int* status, cudaStream_t s) {
  k_commit<<<1, 32, 0, s>>>(ctrl, compressed, status);
}

// ---------------------------------------------------------------------------
// Data-parallel split (one replica per process).  "PowerSGD Hooks": the hook
// allreduces the uncompressed batch (step 2), the Ps (step 3.3) and the Qs
// (step 3.6); the caller sums the exchange buffers across the processes and
// these kernels turn the sums into means ("Default Communication Hooks",
// allreduce_hook: the mean).
// ---------------------------------------------------------------------------

// dst[pos[i] + j] = g[seg_i.off + j] * s over the listed segments (this
// replica's unscaled values, packed); a non-finite value, or the pass-1 flag
// of this process (ctrl->flag), raises *xflag to 1 (when xflag is given).
template <typename GT>
__global__ void __launch_bounds__(kThreads) k_dp_pack(const StepArgs a, const Segment* __restrict__ segs,
                                                      const long long* __restrict__ pos, int nsegs,
                                                      float* __restrict__ dst, float* xflag) {
  const GT* g = reinterpret_cast<const GT*>(a.grads.p[0]);
  int bad = 0;
  for (int it = blockIdx.x; it < nsegs; it += gridDim.x) {
    const Segment sg = segs[it];
    const long long p0 = pos[it];
    for (int j = threadIdx.x; j < sg.len; j += kThreads) {
      float v[1];
      load_grad<1, GT>(g + sg.off + j, v);
      const float x = v[0] * a.scale;
      bad |= !isfinite(x);
      dst[p0 + j] = x;
    }
  }
  if (xflag) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.ctrl->flag) bad = 1;
    if (bad) *xflag = 1.f;
  }
}

// After the caller's sum of the first exchange: a raised flag on any process
// skips the step here too; otherwise P_raw = sum / W in place.
__global__ void __launch_bounds__(kThreads) k_dp_open(const StepArgs a, float* __restrict__ xp, long long n,
                                                      const float* __restrict__ xflag, float invW) {
  if (*xflag != 0.f) {
    if (blockIdx.x == 0 && threadIdx.x == 0) a.ctrl->flag = 1;
    return;
  }
  for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < n; i += (long long)gridDim.x * kThreads)
    xp[i] *= invW;
}

// After the caller's sum of the second exchange: Q = sum / W into the next
// half of Qf (when xq is given), and out = sum / W over the listed segments
// from the packed sums.  check_finite (the vanilla phase, whose exchange is
// `out` itself): a non-finite mean raises the flag, so every process skips.
__global__ void __launch_bounds__(kThreads) k_dp_close(const StepArgs a, const float* __restrict__ xq,
                                                       const Segment* __restrict__ segs,
                                                       const long long* __restrict__ pos, int nsegs,
                                                       const float* src, float invW, int check_finite) {
  if (a.ctrl->flag) return;
  if (xq) {
    float* Q = a.Qf + (long long)(a.ctrl->cur ^ 1) * a.q_total;
    for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < a.q_total;
         i += (long long)gridDim.x * kThreads)
      Q[i] = xq[i] * invW;
  }
  int bad = 0;
  for (int it = blockIdx.x; it < nsegs; it += gridDim.x) {
    const Segment sg = segs[it];
    const long long p0 = pos[it];
    for (int j = threadIdx.x; j < sg.len; j += kThreads) {
      const float x = src[p0 + j] * invW;
      bad |= !isfinite(x);
      a.out[sg.off + j] = x;
    }
  }
  if (check_finite && __any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(&a.ctrl->flag, 1);
}

void launch_dp_pack(const StepArgs& a, const Segment* segs, const long long* pos, int nsegs, float* dst,
                    float* xflag, int grid, cudaStream_t s) {
  if (nsegs == 0 && !xflag) return;
  grid = nsegs > 0 ? grid : 1;
  if (a.gtype == 1)
    k_dp_pack<__half><<<grid, kThreads, 0, s>>>(a, segs, pos, nsegs, dst, xflag);
  else if (a.gtype == 2)
    k_dp_pack<__nv_bfloat16><<<grid, kThreads, 0, s>>>(a, segs, pos, nsegs, dst, xflag);
  else
    k_dp_pack<float><<<grid, kThreads, 0, s>>>(a, segs, pos, nsegs, dst, xflag);
}

void launch_dp_open(const StepArgs& a, float* xp, long long n, const float* xflag, float invW, int grid,
                    cudaStream_t s) {
  k_dp_open<<<grid, kThreads, 0, s>>>(a, xp, n, xflag, invW);
}

void launch_dp_close(const StepArgs& a, const float* xq, const Segment* segs, const long long* pos, int nsegs,
                     const float* src, float invW, int check_finite, int grid, cudaStream_t s) {
  k_dp_close<<<grid, kThreads, 0, s>>>(a, xq, segs, pos, nsegs, src, invW, check_finite);
}

// Philox4x32 with 10 rounds (Salmon, Moraes, Dror and Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011): each round multiplies counter
// words 0 and 2 by the round constants, swaps the halves crosswise and mixes
// in the key, which is bumped by the Weyl constants between rounds.
struct Philox4 {
  unsigned int v[4];
};

__device__ __forceinline__ Philox4 philox4x32_10(Philox4 c, unsigned int k0, unsigned int k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const unsigned int lo0 = 0xD2511F53u * c.v[0];
    const unsigned int hi0 = __umulhi(0xD2511F53u, c.v[0]);
    const unsigned int lo1 = 0xCD9E8D57u * c.v[2];
    const unsigned int hi1 = __umulhi(0xCD9E8D57u, c.v[2]);
    Philox4 n;
    n.v[0] = hi1 ^ c.v[1] ^ k0;
    n.v[1] = lo1;
    n.v[2] = hi0 ^ c.v[3] ^ k1;
    n.v[3] = lo0;
    c = n;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Standard-normal draw of Q for the tensors whose mask is set ("PowerSGD
// Hooks" step 3.1: Q is initialised from a standard normal distribution).
// Element (j, k) of compressed tensor t uses counter (j * RP + k, T,
// counter_lo, counter_hi) with T = tbase + t (tbase numbers a bucket's
// tensors after those of the buckets before it in a group) and key =
// random_seed; Box-Muller on the first two words.
__global__ void __launch_bounds__(kThreads) k_randn(const StepArgs a, const int* __restrict__ mask,
                                                    unsigned long long seed, unsigned long long counter,
                                                    int tbase, int rp) {
  for (int it = blockIdx.x; it < a.n_gsq; it += gridDim.x) {
    const GsItem gi = a.gsq_items[it];
    if (!mask[gi.t]) continue;
    const TensorDesc td = a.tensors[gi.t];
    for (int idx = threadIdx.x; idx < gi.nrows * rp; idx += kThreads) {
      const long long j = gi.row0 + idx / rp;
      const int k = idx % rp;
      float z = 0.f;
      if (k < td.r) {
        Philox4 c;
        const unsigned long long e = (unsigned long long)j * rp + k;
        c.v[0] = (unsigned int)e;
        c.v[1] = (unsigned int)(e >> 32) ^ ((unsigned int)(tbase + gi.t) << 8);
        c.v[2] = (unsigned int)counter;
        c.v[3] = (unsigned int)(counter >> 32);
        const Philox4 o = philox4x32_10(c, (unsigned int)seed, (unsigned int)(seed >> 32));
        const float u1 = ((float)o.v[0] + 1.0f) * 2.3283064365386963e-10f;  // (0, 1]
        const float u2 = (float)o.v[1] * 2.3283064365386963e-10f;           // [0, 1)
        z = sqrtf(-2.0f * logf(u1)) * cosf(6.283185307179586f * u2);
      }
      a.qdraw[td.q_off + (long long)k * td.m + j] = z;  // k-major
    }
  }
}

void launch_randn(const StepArgs& a, const int* mask, unsigned long long seed,
                  unsigned long long counter, int tbase, int rp, int grid, cudaStream_t s) {
  k_randn<<<grid, kThreads, 0, s>>>(a, mask, seed, counter, tbase, rp);
}

}  // namespace psgd
