// Bucket groups: the per-bucket states of one PowerSGD state, stepped on
// several CUDA streams so that one bucket's work overlaps another's.
//
// "DDP Communication Hooks", "What Does a Communication Hook Operate On?":
// DDP splits the gradients into buckets so that communication overlaps
// computation, and calls the hook once per GradBucket; the PowerSGD state
// keeps its error-feedback residuals and warm-start Qs per bucket
// ("PowerSGD State", "PowerSGD Hooks").  Here each bucket is a psgd_state of
// its own; psgd_group_step enqueues bucket b's step on internal stream
// b mod n_streams after the work already enqueued on the caller's stream, so
// the short, latency-bound launches of one bucket (the Gram-Schmidt stage,
// the reductions) run beside the streaming passes of the next.  The buckets'
// compressed tensors are numbered across the group in bucket order, which
// keys their Q draws, so a group draws the same Qs as one state over the
// concatenated buckets.

#include <cuda_runtime.h>

#include <string>
#include <vector>

#include "psgd.h"

int psgd_internal_set_error(int code, const char* msg);  // psgd_api.cu (C++ linkage)
extern "C" int psgd_internal_set_tensor_base(psgd_state* s, int32_t base);
extern "C" int psgd_internal_compressed_count(const psgd_state* s);

struct psgd_group {
  int device = 0;
  std::vector<psgd_state*> buckets;
  std::vector<cudaStream_t> streams;
  std::vector<cudaEvent_t> done;  // per bucket: recorded after its last enqueued step
  cudaEvent_t ready = nullptr;    // the caller's stream at the last psgd_group_step
};

namespace {

struct GroupDevice {
  int prev = -1;
  explicit GroupDevice(int dev) {
    cudaGetDevice(&prev);
    if (prev != dev) cudaSetDevice(dev);
  }
  ~GroupDevice() {
    int now = -1;
    cudaGetDevice(&now);
    if (prev >= 0 && now != prev) cudaSetDevice(prev);
  }
};

int cuda_fail(const char* what, cudaError_t e) {
  return psgd_internal_set_error(PSGD_ECUDA, (std::string(what) + ": " + cudaGetErrorString(e)).c_str());
}

void release(psgd_group* g) {
  if (!g) return;
  {
    GroupDevice d(g->device);
    for (cudaStream_t st : g->streams)
      if (st) cudaStreamSynchronize(st);
    for (psgd_state* s : g->buckets) psgd_state_destroy(s);
    for (cudaEvent_t e : g->done)
      if (e) cudaEventDestroy(e);
    if (g->ready) cudaEventDestroy(g->ready);
    for (cudaStream_t st : g->streams)
      if (st) cudaStreamDestroy(st);
  }
  delete g;
}

}  // namespace

extern "C" {

int psgd_group_create(int32_t n_buckets, const int32_t* tensors_per_bucket, const int64_t* dims,
                      const int32_t* ndims, int32_t world_size, int32_t matrix_approximation_rank,
                      int64_t start_powerSGD_iter, double min_compression_rate, int32_t use_error_feedback,
                      int32_t warm_start, float orthogonalization_epsilon, uint64_t random_seed,
                      int32_t batch_tensors_with_same_shape, psgd_dtype grad_dtype, int32_t n_streams,
                      int32_t device, psgd_group** out) {
  if (!out) return psgd_internal_set_error(PSGD_EINVAL, "out is NULL");
  *out = nullptr;
  if (n_buckets < 1 || !tensors_per_bucket)
    return psgd_internal_set_error(PSGD_EINVAL, "n_buckets must be >= 1 with tensors_per_bucket given");
  if (n_streams < 1 || n_streams > PSGD_MAX_GROUP_STREAMS)
    return psgd_internal_set_error(PSGD_EINVAL, "n_streams must be in [1, 16]");
  long long n_tensors = 0;
  for (int b = 0; b < n_buckets; ++b) {
    if (tensors_per_bucket[b] < 0) return psgd_internal_set_error(PSGD_EINVAL, "tensors_per_bucket < 0");
    n_tensors += tensors_per_bucket[b];
  }
  if (n_tensors > 0 && (!dims || !ndims)) return psgd_internal_set_error(PSGD_EINVAL, "dims/ndims NULL");
  psgd_group* g = new psgd_group();
  g->device = device;
  long long t0 = 0, d0 = 0;
  int base = 0;
  for (int b = 0; b < n_buckets; ++b) {
    psgd_state* s = nullptr;
    const int nt = tensors_per_bucket[b];
    int rc = psgd_state_create(dims + d0, ndims + t0, nt, world_size, matrix_approximation_rank,
                               start_powerSGD_iter, min_compression_rate, use_error_feedback, warm_start,
                               orthogonalization_epsilon, random_seed, batch_tensors_with_same_shape,
                               grad_dtype, device, &s);
    if (rc < 0) {
      release(g);
      return rc;
    }
    g->buckets.push_back(s);
    psgd_internal_set_tensor_base(s, base);
    base += psgd_internal_compressed_count(s);
    for (int t = 0; t < nt; ++t) d0 += ndims[t0 + t];
    t0 += nt;
  }
  GroupDevice d(device);
  g->streams.assign(n_streams, nullptr);
  for (int i = 0; i < n_streams; ++i) {
    cudaError_t e = cudaStreamCreateWithFlags(&g->streams[i], cudaStreamNonBlocking);
    if (e != cudaSuccess) {
      release(g);
      return cuda_fail("psgd_group_create: stream", e);
    }
  }
  g->done.assign(n_buckets, nullptr);
  for (int b = 0; b <= n_buckets; ++b) {
    cudaEvent_t* ev = b < n_buckets ? &g->done[b] : &g->ready;
    cudaError_t e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      release(g);
      return cuda_fail("psgd_group_create: event", e);
    }
  }
  *out = g;
  return PSGD_OK;
}

void psgd_group_destroy(psgd_group* g) { release(g); }

int psgd_group_step(psgd_group* g, int32_t bucket, const void* const* grads, float* out,
                    float inv_loss_scale, void* stream) {
  if (!g) return psgd_internal_set_error(PSGD_EINVAL, "group is NULL");
  if (bucket < 0 || bucket >= (int)g->buckets.size())
    return psgd_internal_set_error(PSGD_EINVAL, "bucket index out of range");
  GroupDevice d(g->device);
  cudaStream_t st = g->streams[bucket % (int)g->streams.size()];
  cudaError_t e = cudaEventRecord(g->ready, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, g->ready, 0);
  if (e != cudaSuccess) return cuda_fail("psgd_group_step: order after the caller's stream", e);
  const int rc = psgd_step(g->buckets[bucket], grads, out, inv_loss_scale, st);
  if (rc < 0) return rc;
  e = cudaEventRecord(g->done[bucket], st);
  if (e != cudaSuccess) return cuda_fail("psgd_group_step: completion event", e);
  return rc;
}

int psgd_group_wait(psgd_group* g, void* stream) {
  if (!g) return psgd_internal_set_error(PSGD_EINVAL, "group is NULL");
  GroupDevice d(g->device);
  for (cudaEvent_t ev : g->done) {
    cudaError_t e = cudaStreamWaitEvent((cudaStream_t)stream, ev, 0);
    if (e != cudaSuccess) return cuda_fail("psgd_group_wait", e);
  }
  return PSGD_OK;
}

int psgd_group_status(psgd_group* g, void* stream) {
  int rc = psgd_group_wait(g, stream);
  if (rc < 0) return rc;
  int skipped = 0;
  for (psgd_state* s : g->buckets) {
    rc = psgd_step_status(s, stream);
    if (rc < 0) return rc;
    skipped |= (rc == PSGD_SKIPPED_NONFINITE);
  }
  return skipped ? PSGD_SKIPPED_NONFINITE : PSGD_OK;
}

int psgd_group_bucket(psgd_group* g, int32_t bucket, psgd_state** out) {
  if (!g || !out) return psgd_internal_set_error(PSGD_EINVAL, "NULL argument");
  if (bucket < 0 || bucket >= (int)g->buckets.size())
    return psgd_internal_set_error(PSGD_EINVAL, "bucket index out of range");
  *out = g->buckets[bucket];
  return PSGD_OK;
}

int32_t psgd_group_size(const psgd_group* g) { return g ? (int32_t)g->buckets.size() : 0; }

}  // extern "C"
