// Definitions of the per-rank launchers; included once per padded rank RP by
// kern_rp<RP>.cu, which instantiates them.
#pragma once

#include <algorithm>
#include <atomic>

#include "psgd_gs.cuh"
#include "psgd_kernels.cuh"
#include "psgd_launch.h"
#include "psgd_tc.cuh"

namespace psgd {

// Calls f with a value of the gradient type named by gtype (0 float,
// 1 __half, 2 __nv_bfloat16).
template <typename F>
inline void by_gtype(int gtype, F&& f) {
  if (gtype == 1)
    f(__half());
  else if (gtype == 2)
    f(__nv_bfloat16());
  else
    f(0.0f);
}

// cudaFuncSetAttribute applies to the current device's context: a launcher
// that raises a kernel's shared-memory limit does so once per device.  `done`
// holds one bit per device ordinal (the library handles ordinals below 64).
// States on other host threads share it: the bit is published only after
// `setup` has run, so no thread launches before the limit is raised (threads
// that race on a fresh device each run `setup`, which is idempotent).
template <typename F>
inline void once_per_device(std::atomic<unsigned long long>& done, F&& setup) {
  int dev = 0;
  cudaGetDevice(&dev);
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return;
  setup();
  done.fetch_or(bit, std::memory_order_release);
}

template <int RP, typename GT>
void launch_pass1_mma(const StepArgs& a, int grid, cudaStream_t s) {
  // the aligned, wholly backed items on the tensor cores (tcgen05), the rest
  // on the element kernel
  using T = Pass1Tc<RP, GT>;
  static std::atomic<unsigned long long> configured{0};
  once_per_device(configured, [] {
    cudaFuncSetAttribute(k_pass1_tc<RP, GT>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
  });
  if (a.vec_ok && a.n_t1 > 0) k_pass1_tc<RP, GT><<<std::min(grid, a.n_t1), T::THREADS, T::SMEM, s>>>(a);
  if (!a.vec_ok || a.has_unaligned) k_pass1_rest<RP, GT><<<grid * 2, kThreads, 0, s>>>(a);
}

// PW: a.W < WT replicas on the stage layout of WT.
template <int RP, int WT, typename GT, int MINB, bool PW = false>
void launch_pass1_cs(const StepArgs& a, int grid, cudaStream_t s) {
  using St0 = Pass1CS<RP, WT, GT, MINB, false>;
  using St1 = Pass1CS<RP, WT, GT, MINB, true>;
  static std::atomic<unsigned long long> configured{0};
  once_per_device(configured, [] {
    cudaFuncSetAttribute(k_pass1_cs<RP, WT, GT, MINB, 0, PW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         St0::SMEM);
    cudaFuncSetAttribute(k_pass1_cs<RP, WT, GT, MINB, 1, PW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         St1::SMEM);
  });
  if (a.vec_ok && a.has_aligned) k_pass1_cs<RP, WT, GT, MINB, 0, PW><<<grid * MINB, kThreads, St0::SMEM, s>>>(a);
  if (!a.vec_ok || a.has_unaligned)
    k_pass1_cs<RP, WT, GT, MINB, 1, PW><<<grid * MINB, kThreads, a.vec_ok ? St1::SMEM : 0, s>>>(a);
}

// grid = one CTA per SM; the kernels run MINB CTAs per SM.  Ranks up to 8 use
// the chunk-stationary kernel (two CTAs per SM for W <= 2, one above; W = 3
// on the four-replica stage, 5 to 8 on the eight-replica one, larger W on the
// element kernel); ranks 16 and 32 the tensor-core kernel (one CTA per SM,
// any W).
template <int RP>
void launch_pass1(const StepArgs& a, int grid, cudaStream_t s) {
  by_gtype(a.gtype, [&](auto tag) {
    using GT = decltype(tag);
    if constexpr (RP <= 8) {
      switch (a.W) {
        case 1: launch_pass1_cs<RP, 1, GT, 2>(a, grid, s); break;
        case 2: launch_pass1_cs<RP, 2, GT, 2>(a, grid, s); break;
        case 4: launch_pass1_cs<RP, 4, GT, 1>(a, grid, s); break;
        case 8: launch_pass1_cs<RP, 8, GT, 1>(a, grid, s); break;
        case 3: launch_pass1_cs<RP, 4, GT, 1, true>(a, grid, s); break;
        case 5:
        case 6:
        case 7: launch_pass1_cs<RP, 8, GT, 1, true>(a, grid, s); break;
        default: k_pass1<RP, 0, GT, 1><<<grid * 2, kThreads, 0, s>>>(a); break;
      }
    } else {
      launch_pass1_mma<RP, GT>(a, grid, s);
    }
  });
}

template <int RP>
void launch_psum(const StepArgs& a, int grid, cudaStream_t s) {
  k_psum<RP><<<grid, kThreads, 0, s>>>(a);
}

template <int RP>
void launch_gram(const StepArgs& a, const float* src, float* dense_out, int is_q, int from_parts,
                 float2* gram, int grid, cudaStream_t s) {
  k_gram<RP><<<grid, kThreads, 0, s>>>(a, src, dense_out, is_q, from_parts, gram);
}

template <int RP>
void launch_gram_sum(const StepArgs& a, int is_q, cudaStream_t s) {
  constexpr int EPC = RP * RP < kGramSumEntries ? RP * RP : kGramSumEntries;
  k_gram_sum<RP><<<dim3(a.n_tensors, (RP * RP) / EPC), kThreads, 0, s>>>(a, is_q);
}

template <int RP>
void launch_solve(const StepArgs& a, const float2* gram, int is_q, int sweep, cudaStream_t s) {
  k_solve<RP><<<a.n_tensors, kThreads, 0, s>>>(a, gram, is_q, sweep);
}

template <int RP>
void launch_apply(const StepArgs& a, const float* src, float* dst, int is_q, int dst_half, int grid,
                  cudaStream_t s, const float* tsrc, int img) {
  k_apply<RP><<<grid, kThreads, 0, s>>>(a, src, dst, is_q, dst_half, tsrc, img);
}

template <int RP>
void launch_gs_first(const StepArgs& a, const float* src, float* dense_out, int is_q, int from_parts, int grid,
                     cudaStream_t s) {
  k_gs_first<RP><<<grid, kThreads, 0, s>>>(a, src, dense_out, is_q, from_parts);
}

template <int RP>
void launch_gs_second(const StepArgs& a, const float* src, float* mid, int is_q, int grid, cudaStream_t s) {
  k_gs_second<RP><<<grid, kThreads, 0, s>>>(a, src, mid, is_q);
}

// The fused stage as one cooperative launch (every CTA resident, which the
// cooperative launch guarantees or refuses): at most `grid` CTAs and no more
// than fit on the device at once.  *bar is zeroed first on the same stream.
template <int RP>
cudaError_t launch_gs_coop(const StepArgs& a, const float* src, float* dense_out, int is_q, int from_parts,
                           float* mid, float* dst, int dst_half, int do_psum, unsigned int* bar, int img,
                           int grid, cudaStream_t s, unsigned int skew) {
  // CTAs resident at once, per device ordinal (0: not known yet, or none fit;
  // threads that race on a fresh device each compute the same value)
  static std::atomic<int> fits[64];
  int dev = 0;
  cudaGetDevice(&dev);
  int fit = fits[dev & 63].load(std::memory_order_relaxed);
  if (fit <= 0) {
    int sms = 0, per_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_gs_coop<RP>, kThreads, 0);
    fit = std::max(0, per_sm * sms);
    fits[dev & 63].store(fit, std::memory_order_relaxed);
  }
  if (fit == 0) return cudaErrorCooperativeLaunchTooLarge;
  grid = std::max(1, std::min(grid, fit));
  cudaError_t e = cudaMemsetAsync(bar, 0, sizeof(unsigned int), s);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<StepArgs*>(&a), &src, &dense_out, &is_q, &from_parts, &mid, &dst, &dst_half,
                  &do_psum, &bar, &img, &skew};
  return cudaLaunchCooperativeKernel((const void*)k_gs_coop<RP>, dim3(grid), dim3(kThreads), args, 0, s);
}

template <int RP, int NSRC>
void launch_pass2_tc(const StepArgs& a, int src_mode, cudaStream_t s) {
  using T = Pass2Tc<RP, NSRC>;
  static std::atomic<unsigned long long> configured{0};
  once_per_device(configured, [] {
    cudaFuncSetAttribute(k_pass2_tc<RP, NSRC>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
  });
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  k_pass2_tc<RP, NSRC><<<std::min(a.n_t2, sms), T::THREADS, T::SMEM, s>>>(a, src_mode);
}

template <int RP>
void launch_pass2(const StepArgs& a, int src_mode, int grid, cudaStream_t s) {
  if constexpr (RP >= 16) {
    // rank 32: the Mbar scratch, or the store halves of one or two replicas,
    // on the tensor cores (src_mode 1 is chosen only for W <= 2); at rank 16
    // the fp32 kernel is faster
    if (RP == 32 && a.n_t2 > 0 && (src_mode == 0 || (src_mode == 1 && a.W <= 2))) {
      if (src_mode == 1 && a.W == 2)
        launch_pass2_tc<RP, 2>(a, src_mode, s);
      else
        launch_pass2_tc<RP, 1>(a, src_mode, s);
      return;
    }
  }
  if (src_mode == 0) {
    k_pass2<RP, 0, float, 0><<<grid, kThreads, 0, s>>>(a);
  } else if (src_mode == 1) {
    if (a.W == 1)
      k_pass2<RP, 1, float, 1><<<grid, kThreads, 0, s>>>(a);
    else if (a.W == 2)
      k_pass2<RP, 1, float, 2><<<grid, kThreads, 0, s>>>(a);
    else
      k_pass2<RP, 1, float, 0><<<grid, kThreads, 0, s>>>(a);
  } else {
    by_gtype(a.gtype, [&](auto tag) {
      using GT = decltype(tag);
      switch (a.W) {
        case 1: k_pass2<RP, 2, GT, 1><<<grid, kThreads, 0, s>>>(a); break;
        case 2: k_pass2<RP, 2, GT, 2><<<grid, kThreads, 0, s>>>(a); break;
        case 4: k_pass2<RP, 2, GT, 4><<<grid, kThreads, 0, s>>>(a); break;
        default: k_pass2<RP, 2, GT, 0><<<grid, kThreads, 0, s>>>(a); break;
      }
    });
  }
}

template <int RP>
void launch_qreduce(const StepArgs& a, int grid, cudaStream_t s, int img) {
  k_qreduce<RP><<<grid, kThreads, 0, s>>>(a, img);
}

template <int RP>
void launch_images(const StepArgs& a, int mode, int grid, cudaStream_t s) {
  if constexpr (RP >= 16) k_images<RP><<<grid, kThreads, 0, s>>>(a, mode);
}

template <int RP>
void launch_pass3(const StepArgs& a, int mode, int grid, cudaStream_t s) {
  if constexpr (RP >= 16) {
    // the aligned, backed tensors on the tensor cores (one CTA per SM); the
    // fp32 kernel below skips them and takes the rest
    if (mode == 0 && a.vec_ok && a.n_t3 > 0) {
      using T = Pass3Tc<RP>;
      static std::atomic<unsigned long long> configured{0};
      once_per_device(configured, [] {
        cudaFuncSetAttribute(k_pass3_tc<RP>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
      });
      int dev = 0, sms = 148;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      k_pass3_tc<RP><<<std::min(a.n_t3, sms), T::THREADS, T::SMEM, s>>>(a);
      if (!a.has_unaligned) return;   // every tensor was written
    }
  }
  if (mode == 0)
    k_pass3<RP, 0><<<grid, kThreads, 0, s>>>(a);
  else if (mode == 1)
    k_pass3<RP, 1><<<grid, kThreads, 0, s>>>(a);
  else if (mode == 2)
    k_pass3<RP, 2><<<grid, kThreads, 0, s>>>(a);
  else
    k_pass3<RP, 3><<<grid, kThreads, 0, s>>>(a);
}

#define PSGD_INSTANTIATE(RPV)                                                                   \
  template void launch_pass1<RPV>(const StepArgs&, int, cudaStream_t);                          \
  template void launch_psum<RPV>(const StepArgs&, int, cudaStream_t);                           \
  template void launch_gram<RPV>(const StepArgs&, const float*, float*, int, int, float2*, int, \
                                 cudaStream_t);                                                 \
  template void launch_gram_sum<RPV>(const StepArgs&, int, cudaStream_t);                      \
  template void launch_solve<RPV>(const StepArgs&, const float2*, int, int, cudaStream_t);      \
  template void launch_apply<RPV>(const StepArgs&, const float*, float*, int, int, int,         \
                                  cudaStream_t, const float*, int);                             \
  template void launch_gs_first<RPV>(const StepArgs&, const float*, float*, int, int, int,      \
                                     cudaStream_t);                                             \
  template cudaError_t launch_gs_coop<RPV>(const StepArgs&, const float*, float*, int, int, float*, float*, \
                                            int, int, unsigned int*, int, int, cudaStream_t,            \
                                            unsigned int);                                              \
  template void launch_gs_second<RPV>(const StepArgs&, const float*, float*, int, int,          \
                                      cudaStream_t);                                            \
  template void launch_pass2<RPV>(const StepArgs&, int, int, cudaStream_t);                     \
  template void launch_qreduce<RPV>(const StepArgs&, int, cudaStream_t, int);                        \
  template void launch_pass3<RPV>(const StepArgs&, int, int, cudaStream_t);                     \
  template void launch_images<RPV>(const StepArgs&, int, int, cudaStream_t);

}  // namespace psgd
