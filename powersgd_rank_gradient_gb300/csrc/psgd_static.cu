// psgd_project_q_static: the Q = M^T P projection of one matrix (the work of
// pass 2 for a single replica) with its per-row-block partial sums kept in a
// file-scope __device__ array instead of memory allocated by the library.
//
// It is for callers that cannot call cudaMalloc: a training job that reserved
// nearly all device memory up front (a later cudaMalloc would fail), code
// whose device memory must all come from a framework's own allocator, and
// latency-sensitive code that cannot afford the implicit device-wide
// synchronisation cudaMalloc may perform.  Such callers pass the inputs and
// the output; the scratch is the static array below, which every GPU that
// loads this library holds until the process exits.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/psgd.h"
#include "psgd_kernels.cuh"

namespace psgd {

// 2 Mi floats (8 MiB) of partial sums: row blocks x padded rank x cols.
constexpr long long kStaticScratchFloats = 2LL * 1024 * 1024;
static __device__ __align__(256) float g_static_scratch[kStaticScratchFloats];

namespace {

// Device ordinals this entry point serves (one looked-up address each).
constexpr int kMaxDevices = 64;

std::mutex g_static_mu;
float* g_static_ptr[kMaxDevices] = {nullptr};  // per device ordinal

constexpr int kStaticRows = kRowBlock;

// Partial Q = M^T P over one (row block, column tile): each thread owns CPT
// columns and sums CPT x RP products over the block's rows in row order, the
// accumulation order of pass 2.
template <int RP, bool VEC>
__global__ void __launch_bounds__(kThreads) k_projq_static(const float* __restrict__ M,
                                                           const float* __restrict__ P, long long rows,
                                                           long long cols, int rank, int ctiles,
                                                           float* __restrict__ scratch) {
  constexpr int CPT = cpt_for(RP);
  constexpr int CT = kThreads * CPT;
  __shared__ __align__(16) float ps[128][RP];
  const int b = blockIdx.x / ctiles;
  const int ct = blockIdx.x - b * ctiles;
  const long long row0 = (long long)b * kStaticRows;
  const int nrows = (int)min((long long)kStaticRows, rows - row0);
  const long long col0 = (long long)ct * CT;
  const long long cend = min(col0 + CT, cols);
  const long long c0 = col0 + (long long)threadIdx.x * CPT;
  float acc[CPT][RP];
#pragma unroll
  for (int c = 0; c < CPT; ++c)
#pragma unroll
    for (int k = 0; k < RP; ++k) acc[c][k] = 0.f;
  for (int sb = 0; sb < nrows; sb += 128) {
    const int rs = min(128, nrows - sb);
    __syncthreads();
    for (int idx = threadIdx.x; idx < rs * RP; idx += kThreads) {
      const int i = idx / RP, k = idx % RP;
      ps[i][k] = (k < rank) ? P[(row0 + sb + i) * rank + k] : 0.f;
    }
    __syncthreads();
    if (c0 >= cend) continue;
    for (int i = 0; i < rs; ++i) {
      const long long row = row0 + sb + i;
      float mv[CPT];
      if constexpr (VEC && CPT == 4) {
        load_f<4>(M + row * cols + c0, mv, true);
      } else {
#pragma unroll
        for (int c = 0; c < CPT; ++c) mv[c] = (c0 + c < cend) ? ld_stream1(M + row * cols + c0 + c) : 0.f;
      }
#pragma unroll
      for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int k = 0; k < RP; ++k) acc[c][k] = fmaf(mv[c], ps[i][k], acc[c][k]);
    }
  }
  if (c0 >= cend) return;
  float* dst = scratch + (long long)b * RP * cols;
#pragma unroll
  for (int k = 0; k < RP; ++k)
#pragma unroll
    for (int c = 0; c < CPT; ++c)
      if (c0 + c < cend) dst[(long long)k * cols + c0 + c] = acc[c][k];
}

// Q(j, k) = sum over row blocks, in row-block order; Q is cols x rank, row-major.
template <int RP>
__global__ void __launch_bounds__(kThreads) k_projq_static_sum(const float* __restrict__ scratch,
                                                               float* __restrict__ Q, long long cols,
                                                               int rank, int rblocks) {
  const long long n = cols * rank;
  for (long long e = (long long)blockIdx.x * kThreads + threadIdx.x; e < n; e += (long long)gridDim.x * kThreads) {
    const long long j = e / rank;
    const int k = (int)(e - j * rank);
    float s = 0.f;
    for (int b = 0; b < rblocks; ++b) s += scratch[((long long)b * RP + k) * cols + j];
    Q[e] = s;
  }
}

template <int RP>
void launch_projq_static(const float* M, const float* P, float* Q, long long rows, long long cols, int rank,
                         float* scratch, cudaStream_t st) {
  constexpr int CT = kThreads * cpt_for(RP);
  const int ctiles = (int)((cols + CT - 1) / CT);
  const int rblocks = (int)((rows + kStaticRows - 1) / kStaticRows);
  const bool vec = (cols % 4 == 0) && ((uintptr_t)M % 16 == 0);
  const unsigned grid = (unsigned)rblocks * ctiles;
  if (vec)
    k_projq_static<RP, true><<<grid, kThreads, 0, st>>>(M, P, rows, cols, rank, ctiles, scratch);
  else
    k_projq_static<RP, false><<<grid, kThreads, 0, st>>>(M, P, rows, cols, rank, ctiles, scratch);
  const long long n = cols * rank;
  const int grid2 = (int)std::min<long long>((n + kThreads - 1) / kThreads, 4096);
  k_projq_static_sum<RP><<<grid2, kThreads, 0, st>>>(scratch, Q, cols, rank, rblocks);
}

}  // namespace
}  // namespace psgd

int psgd_internal_set_error(int code, const char* msg);

using namespace psgd;

extern "C" int psgd_project_q_static(const float* dev_m, const float* dev_p, float* dev_q, int64_t rows,
                                     int64_t cols, int32_t rank, void* stream) {
  if (!dev_m || !dev_p || !dev_q) return psgd_internal_set_error(PSGD_EINVAL, "psgd_project_q_static: NULL pointer");
  if (rows <= 0 || cols <= 0) return psgd_internal_set_error(PSGD_EINVAL, "psgd_project_q_static: rows and cols must be > 0");
  if (rank < 1 || rank > PSGD_MAX_RANK)
    return psgd_internal_set_error(PSGD_EINVAL, "psgd_project_q_static: rank must be in [1, 32]");
  int rp = 1;
  while (rp < rank) rp <<= 1;
  const long long rblocks = (rows + kStaticRows - 1) / kStaticRows;
  // ceil(rows / 512) * rp * cols <= kStaticScratchFloats, tested by division
  // so that no product of caller-supplied sizes can overflow
  if (cols > kStaticScratchFloats / rp || rblocks > kStaticScratchFloats / (rp * cols)) {
    const std::string msg = "psgd_project_q_static: ceil(rows / 512) = " + std::to_string(rblocks) + " row blocks x " +
                            std::to_string(rp) + " x " + std::to_string(cols) +
                            " cols of partial sums exceed the static scratch of " +
                            std::to_string(kStaticScratchFloats) + " floats";
    return psgd_internal_set_error(PSGD_EINVAL, msg.c_str());
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return psgd_internal_set_error(PSGD_ECUDA, "psgd_project_q_static: no current CUDA device");
  }
  if (dev < 0 || dev >= kMaxDevices)
    return psgd_internal_set_error(PSGD_EINVAL, "psgd_project_q_static: device ordinals above 63 are not served");
  float* scratch = nullptr;
  {
    // First call on this device: look up the device address of the static
    // array with this device current (the name is only a host-side stand-in).
    // This one-time set-up should happen before any stream capture.
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return psgd_internal_set_error(
            PSGD_ECUDA, (std::string("psgd_project_q_static: cudaGetSymbolAddress: ") + cudaGetErrorString(e)).c_str());
      }
      g_static_ptr[dev] = (float*)p;
    }
    scratch = g_static_ptr[dev];
  }
  cudaStream_t st = (cudaStream_t)stream;
  switch (rp) {
    case 1: launch_projq_static<1>(dev_m, dev_p, dev_q, rows, cols, rank, scratch, st); break;
    case 2: launch_projq_static<2>(dev_m, dev_p, dev_q, rows, cols, rank, scratch, st); break;
    case 4: launch_projq_static<4>(dev_m, dev_p, dev_q, rows, cols, rank, scratch, st); break;
    case 8: launch_projq_static<8>(dev_m, dev_p, dev_q, rows, cols, rank, scratch, st); break;
    case 16: launch_projq_static<16>(dev_m, dev_p, dev_q, rows, cols, rank, scratch, st); break;
    default: launch_projq_static<32>(dev_m, dev_p, dev_q, rows, cols, rank, scratch, st); break;
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return psgd_internal_set_error(PSGD_ECUDA, (std::string("psgd_project_q_static: launch: ") + cudaGetErrorString(e)).c_str());
  return PSGD_OK;
}
