// Host-side launchers of the kernels (one translation unit per padded rank).
#pragma once

#include <cuda_runtime.h>

#include "psgd_internal.h"

namespace psgd {

struct StepArgs;

template <int RP> void launch_pass1(const StepArgs& a, int grid, cudaStream_t s);
template <int RP> void launch_psum(const StepArgs& a, int grid, cudaStream_t s);
template <int RP> void launch_gram(const StepArgs& a, const float* src, float* dense_out, int is_q,
                                   int from_parts, float2* gram, int grid, cudaStream_t s);
template <int RP> void launch_gram_sum(const StepArgs& a, int is_q, cudaStream_t s);
template <int RP> void launch_solve(const StepArgs& a, const float2* gram, int is_q, int sweep, cudaStream_t s);
// img: ranks 16 and 32, P's operand images written too (k_images mode 0)
template <int RP> void launch_apply(const StepArgs& a, const float* src, float* dst, int is_q,
                                    int dst_half, int grid, cudaStream_t s, const float* tsrc = nullptr,
                                    int img = 0);
template <int RP> void launch_gs_first(const StepArgs& a, const float* src, float* dense_out, int is_q,
                                       int from_parts, int grid, cudaStream_t s);
template <int RP> void launch_gs_second(const StepArgs& a, const float* src, float* mid, int is_q, int grid,
                                        cudaStream_t s);
template <int RP> cudaError_t launch_gs_coop(const StepArgs& a, const float* src, float* dense_out, int is_q,
                                              int from_parts, float* mid, float* dst, int dst_half, int do_psum,
                                              unsigned int* bar, int img, int grid, cudaStream_t s,
                                              unsigned int skew = 0);
template <int RP> void launch_pass2(const StepArgs& a, int src_mode, int grid, cudaStream_t s);
// img: ranks 16 and 32, also write Q's row image (k_images mode 1)
template <int RP> void launch_qreduce(const StepArgs& a, int grid, cudaStream_t s, int img = 0);
template <int RP> void launch_pass3(const StepArgs& a, int mode, int grid, cudaStream_t s);
template <int RP> void launch_images(const StepArgs& a, int mode, int grid, cudaStream_t s);

void launch_mean(const StepArgs& a, const Segment* segs, int nsegs, int grid, cudaStream_t s);
void launch_commit(Ctrl* ctrl, int compressed, int* status, cudaStream_t s);
void launch_randn(const StepArgs& a, const int* mask, unsigned long long seed,
                  unsigned long long counter, int tbase, int rp, int grid, cudaStream_t s);
// data-parallel split: pack this replica's values for the exchange, turn the
// exchanged sums into means
void launch_dp_pack(const StepArgs& a, const Segment* segs, const long long* pos, int nsegs, float* dst,
                    float* xflag, int grid, cudaStream_t s);
void launch_dp_open(const StepArgs& a, float* xp, long long n, const float* xflag, float invW, int grid,
                    cudaStream_t s);
void launch_dp_close(const StepArgs& a, const float* xq, const Segment* segs, const long long* pos, int nsegs,
                     const float* src, float invW, int check_finite, int grid, cudaStream_t s);

}  // namespace psgd
