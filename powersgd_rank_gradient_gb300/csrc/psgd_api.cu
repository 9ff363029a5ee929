// Host side of the C ABI declared in include/psgd.h: the bucket planner, the
// state's device memory, and the order in which a step's kernels are
// enqueued.  No step of the method's arithmetic runs here.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <functional>
#include <string>
#include <vector>

#include "../../include/psgd.h"
#include "psgd_kernels.cuh"
#include "psgd_launch.h"

using namespace psgd;

namespace {
thread_local std::string g_last_error;
}  // namespace

// Records the message psgd_last_error returns (also used by psgd_static.cu).
int psgd_internal_set_error(int code, const char* msg) {
  g_last_error = msg ? msg : "";
  return code;
}

namespace {


int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

#define PSGD_CUDA_TRY(expr)                                                            \
  do {                                                                                 \
    cudaError_t e_ = (expr);                                                           \
    if (e_ != cudaSuccess)                                                             \
      return fail(PSGD_ECUDA, std::string(#expr) + ": " + cudaGetErrorString(e_));      \
  } while (0)

struct HostTensor {
  std::vector<int64_t> shape;
  long long offset = 0;
  long long numel = 0;
  int compressed = 0;
  long long rows = 0, cols = 0;
  int rank = 0;
  int cidx = -1;          // compressed ordinal
  long long e_off = -1;   // packed error offset
  long long valid = -1;   // elements backed by the bucket (-1: all)
};

int next_pow2(int r) {
  int p = 1;
  while (p < r) p <<= 1;
  return p;
}

// "DDP Communication Hooks", "PowerSGD State" item 3 and "PowerSGD Hooks"
// step 1: vectors are never compressed; a >= 2-D tensor viewed as
// (shape[0], prod(shape[1:])) is compressed iff
// (rows + cols) * rank * min_compression_rate < rows * cols.
int plan_tensors(const int64_t* dims, const int32_t* ndims, int32_t n, int32_t rank, double mcr,
                 std::vector<HostTensor>* out) {
  if (n < 0) return fail(PSGD_EINVAL, "n_tensors < 0");
  if (n > 0 && !ndims) return fail(PSGD_EINVAL, "ndims is NULL");
  long long total_dims = 0;
  for (int t = 0; t < n; ++t) total_dims += ndims[t] > 0 ? ndims[t] : 0;
  if (total_dims > 0 && !dims) return fail(PSGD_EINVAL, "dims is NULL");
  if (rank < 1 || rank > PSGD_MAX_RANK)
    return fail(PSGD_EINVAL, "matrix_approximation_rank must be in [1, 32]");
  if (!(mcr >= 0.0)) return fail(PSGD_EINVAL, "min_compression_rate must be >= 0");
  out->clear();
  long long off = 0;
  int d = 0;
  for (int t = 0; t < n; ++t) {
    HostTensor h;
    if (ndims[t] < 0) return fail(PSGD_EINVAL, "negative ndims");
    long long numel = 1;
    for (int k = 0; k < ndims[t]; ++k) {
      const int64_t v = dims[d + k];
      if (v < 0) return fail(PSGD_EINVAL, "negative dimension");
      h.shape.push_back(v);
      numel *= v;
    }
    d += ndims[t];
    h.offset = off;
    h.numel = numel;
    if (ndims[t] >= 2 && numel > 0) {
      h.rows = h.shape[0];
      h.cols = numel / h.rows;
      const double lhs = (double)((h.rows + h.cols) * (long long)rank) * mcr;
      const double rhs = (double)(h.rows * h.cols);
      if (lhs < rhs) {
        h.compressed = 1;
        h.rank = (int)std::min<long long>(rank, std::min(h.rows, h.cols));
      }
    } else if (ndims[t] >= 2) {
      h.rows = h.shape[0];
      h.cols = h.rows > 0 ? numel / h.rows : 0;
    }
    off += numel;
    out->push_back(h);
  }
  return PSGD_OK;
}

enum Kind { K_MEAN = 0, K_PASS1, K_GRAM, K_SOLVE, K_APPLY, K_PASS2, K_QREDUCE, K_PASS3, K_COMMIT, K_RANDN,
            K_PSUM, K_DP, K_IMG, K_GS, K_COUNT };
const char* kKindNames[K_COUNT] = {"mean", "pass1", "gs_gram", "gs_solve", "gs_apply",
                                   "pass2", "qreduce", "pass3", "commit", "randn", "psum", "dp_exchange",
                                   "images", "gs_stage"};

struct EventPair {
  cudaEvent_t a, b;
};

}  // namespace

struct psgd_state {
  // configuration
  int device = 0;
  int W = 1;
  int rank = 1;
  int RP = 1;
  long long start_iter = 0;
  double mcr = 2.0;
  int ef = 1;
  int warm = 1;
  float eps = 0.f;
  unsigned long long seed = 0;
  int tensor_base = 0;    // added to the compressed-tensor number in the draw's counter
  int batch = 0;
  int batched = 0;        // the batched hook's single padded square
  psgd_dtype dtype = PSGD_F32;
  // plan
  std::vector<HostTensor> tensors;
  std::vector<TensorDesc> cdesc;
  std::vector<Item> items;    // pass 2
  std::vector<Item> fitems;   // pass 3, error views
  std::vector<Item> p1items;  // pass 1
  std::vector<Item> t3items;  // tensor-core pass 3 (ranks 16 and 32)
  std::vector<Item> t2items;  // tensor-core pass 2 (ranks 16 and 32)
  std::vector<Item> t1items;  // tensor-core pass 1 (ranks 16 and 32)
  std::vector<GsItem> ps;     // P partial reduction chunks
  std::vector<GsItem> qr;     // Q partial reduction chunks
  std::vector<GsItem> gsp, gsq;
  std::vector<int> gsp_first, gsp_count, gsq_first, gsq_count;
  std::vector<Segment> unc_segs, all_segs;
  long long N = 0, Nc = 0, Nc_pad = 0, Nunc = 0, Ne = 0;
  int any_aligned = 0;     // a compressed tensor's rows are 16-byte aligned
  int any_unaligned = 0;   // some are not, or the bucket ends inside the view
  long long p_total = 0, q_total = 0, pp_total = 0, qp_total = 0;
  int pass2_src = 0;  // 0 mbar scratch, 1 error store, 2 gradients
  int row_block = kRowBlock;  // rows per pass-2 item
  int fold_psum = 0;          // the first Gram kernel adds pass 1's P partials itself
  int gs_fused = 0;           // Gram-Schmidt stage in three launches (few row items per tensor)
  // device memory
  TensorDesc* d_tensors = nullptr;
  Item* d_items = nullptr;
  Item* d_fitems = nullptr;
  Item* d_p1items = nullptr;
  Item* d_t3items = nullptr;
  Item* d_t2items = nullptr;
  Item* d_t1items = nullptr;
  float* img = nullptr;        // tensor-core operand images (ranks 16 and 32)
  long long img_total = 0;
  GsItem* d_ps = nullptr;
  GsItem* d_qr = nullptr;
  GsItem* d_gsp = nullptr;
  GsItem* d_gsq = nullptr;
  int* d_gs_index = nullptr;  // gsp_first | gsp_count | gsq_first | gsq_count
  int* d_mask = nullptr;
  Segment* d_unc = nullptr;
  Segment* d_all = nullptr;
  float* estore = nullptr;
  int est_halves = 2;       // error-store halves (1: psgd_set_error_store_halves)
  float* mbar = nullptr;
  float* Pf = nullptr;
  float* Qf = nullptr;
  float* qinit = nullptr;
  float* qdraw = nullptr;
  float* praw_part = nullptr;
  float* praw = nullptr;
  float* pgs = nullptr;
  float* qpart = nullptr;
  float* tmat = nullptr;
  float* tmat2 = nullptr;   // fused Gram-Schmidt stage: second sweep's transforms
  int* gs_cnt = nullptr;    // fused Gram-Schmidt stage: per-tensor partial counters
  unsigned int* gs_bar = nullptr;   // its cooperative launch: the grid barrier's counter
  int* p3_cnt = nullptr;    // ranks <= 8: pass 3's finished CTAs (the last commits the step)
  int gs_coop = 1;          // the fused stage as one cooperative launch (0 after a refusal)
  unsigned int test_wait_skew = 0;   // tests: the next cooperative stage's first barrier never completes
  float2* gram = nullptr;   // per Gram-Schmidt item RP x RP double-float partials
  float2* gram_t = nullptr; // per tensor RP x RP summed Gram matrix (double-float)
  Ctrl* ctrl = nullptr;
  int* d_status = nullptr;
  int* h_status = nullptr;  // pinned
  size_t bytes = 0;
  std::vector<void*> allocs;
  // host staging for psgd_step_host: two sets, alternated call by call, so
  // that the next call's uploads overlap this call's compute and download
  std::vector<void*> stage_grads[2];
  float* stage_out[2] = {nullptr, nullptr};
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t ev_in[2] = {nullptr, nullptr}, ev_comp[2] = {nullptr, nullptr}, ev_free[2] = {nullptr, nullptr};
  int set_used[2] = {0, 0};
  long long host_calls = 0;
  // CUDA graph of the steady compressed step (psgd_set_graph): captured on
  // s_cap for one (grads, out, scale) key and replayed while the key holds
  int graph_mode = 0;
  cudaStream_t s_cap = nullptr;
  cudaGraphExec_t gexec = nullptr;
  std::vector<const void*> gkey_grads;
  const void* gkey_out = nullptr;
  float gkey_scale = 0.f;
  long long graph_captures = 0, graph_replays = 0;
  // data-parallel split (psgd_dp_*): this process holds one replica of a
  // dp_world-process job (0: not a data-parallel state)
  int dp_world = 0;
  float* xp = nullptr;        // first exchange: [P_raw | pad | uncompressed | flag]
  long long xp_count = 0;
  long long xp_unc = 0;       // first uncompressed value in xp
  float* xq = nullptr;        // second exchange: Q (Qf layout)
  long long* d_unc_pos = nullptr;  // packed position of each uncompressed segment
  long long* d_all_pos = nullptr;  // position of each whole-bucket segment (= its offset)
  int dp_stage = 0;           // 0 idle, 1 after begin, 2 after project
  const void* dp_grad = nullptr;
  float* dp_out = nullptr;
  float dp_scale = 1.f;
  bool dp_vanilla = false, dp_compressed = false;
  // counters
  long long iter = 0;
  long long compressed_launched = 0;
  std::vector<int> pending_draw;  // per compressed tensor
  int sms = 148;
  // profiling
  bool prof = false;
  uint32_t prof_mask = 0xffffffffu;   // kinds recorded while prof (psgd_profile_select)
  std::vector<std::vector<EventPair>> ev;
  std::vector<EventPair> ev_pool;
  double kind_bytes[K_COUNT] = {0};
};

namespace {

int dalloc(psgd_state* s, void** p, size_t bytes) {
  if (bytes == 0) {
    *p = nullptr;
    return PSGD_OK;
  }
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    *p = nullptr;
    cudaGetLastError();
    return fail(e == cudaErrorMemoryAllocation ? PSGD_ENOMEM : PSGD_ECUDA,
                std::string("cudaMalloc(") + std::to_string(bytes) + "): " + cudaGetErrorString(e));
  }
  s->allocs.push_back(*p);
  s->bytes += bytes;
  return PSGD_OK;
}

template <typename T>
int dupload(psgd_state* s, T** dst, const std::vector<T>& v) {
  int rc = dalloc(s, (void**)dst, std::max<size_t>(1, v.size()) * sizeof(T));
  if (rc) return rc;
  if (!v.empty()) PSGD_CUDA_TRY(cudaMemcpy(*dst, v.data(), v.size() * sizeof(T), cudaMemcpyHostToDevice));
  return PSGD_OK;
}

// piece: elements per segment (one CTA's work item).  The step's uncompressed
// ranges are small and scattered (biases, norms): 1024-element pieces give
// each thread one vector of every replica, so the mean costs about one load
// latency; the vanilla phase streams the whole bucket in 64K pieces.
void add_segments(std::vector<Segment>* segs, long long off, long long len, long long piece = 65536) {
  for (long long o = 0; o < len; o += piece) {
    Segment sg;
    sg.off = off + o;
    sg.len = (int)std::min(piece, len - o);
    sg.pad = 0;
    segs->push_back(sg);
  }
}

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    cudaGetDevice(&prev);
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int now = -1;
    cudaGetDevice(&now);
    if (prev >= 0 && now != prev) cudaSetDevice(prev);
  }
};

// The longest CTA load when G resident CTAs take items of the given sizes
// (elements, in the order the kernels take them) round-robin, as the
// persistent pass kernels do: an item costs its elements x bpe bytes plus c0
// (its setup loads and the fill and drain of its copy pipeline).
double rr_makespan(const std::vector<long long>& sizes, long long G, double bpe, double c0) {
  if (G < 1) G = 1;
  std::vector<double> load((size_t)std::min<long long>(G, (long long)sizes.size() + 1), 0.0);
  for (size_t i = 0; i < sizes.size(); ++i) load[i % load.size()] += (double)sizes[i] * bpe + c0;
  return *std::max_element(load.begin(), load.end());
}

// Bytes a CTA streams while its item setup stalls for t seconds, with G CTAs
// sharing about 6.8 TB/s of HBM (only the ratio between candidates matters).
double stall_bytes(double t, long long G) { return t * 6.8e12 / (double)std::max<long long>(G, 1); }

// Builds the work lists of the compressed tensors.
void build_plan(psgd_state* s) {
  const int RP = s->RP;
  const int CT = ctile_for(RP);
  const int CT1 = ctile1_for(RP);
  // Column tiles of pass 1.  Ranks up to 8: up to eight 128-column chunks a
  // tile, the rest of a row split into tiles of 4, 2 and 1 chunks, so that the
  // chunk-stationary kernel's 8 warps divide every tile's chunks evenly
  // (a 1600-column tensor: 8 + 4 + 1 chunks rather than 8 + 5).  Ranks 16 and
  // 32: CT1-column tiles.
  auto p1_tiles = [&](int m) {
    std::vector<std::pair<int, int>> v;   // (first column, columns)
    if (RP > 8) {
      for (int c0 = 0; c0 < m; c0 += CT1) v.push_back({c0, std::min(CT1, m - c0)});
      return v;
    }
    int left = (m + 127) / 128, done = 0;
    while (left > 0) {
      int p = 8;
      while (p > left) p >>= 1;
      v.push_back({done * 128, std::min(p * 128, m - done * 128)});
      done += p;
      left -= p;
    }
    return v;
  };
  s->cdesc.clear();
  s->items.clear();
  s->fitems.clear();
  s->p1items.clear();
  s->t3items.clear();
  s->t2items.clear();
  s->t1items.clear();
  s->qr.clear();
  s->ps.clear();
  s->gsp.clear();
  s->gsq.clear();
  s->gsp_first.clear();
  s->gsp_count.clear();
  s->gsq_first.clear();
  s->gsq_count.clear();
  s->unc_segs.clear();
  s->all_segs.clear();
  long long c_off = 0, p_off = 0, q_off = 0, pp_off = 0, qp_off = 0, e_off = 0, i_off = 0;
  long long unc = 0;
  // pass 2: row blocks of kRowBlock rows, shorter for small buckets so that
  // there are several items per resident CTA (one Q partial per item).  When
  // every compressed tensor has one shape the items are alike and the waves
  // can be counted: the row block (a multiple of 64) with the shortest
  // round-robin makespan, each item also paying its Q partial and its setup
  // (8192 x 8192: 192 rows at ranks <= 8, 320 at rank 16, 512 at rank 32,
  // each measured best for its kernel: the fp32 kernel at four and two
  // columns a thread, the tensor-core kernel of rank 32)
  {
    long long nc = 0;
    bool alike = true;
    long long n0 = -1, m0 = -1;
    for (auto& h : s->tensors) {
      if (!h.compressed) continue;
      nc += h.numel;
      if (n0 < 0) {
        n0 = h.rows;
        m0 = h.cols;
      }
      alike = alike && h.rows == n0 && h.cols == m0;
    }
    const long long target = (long long)s->sms * 3 * 4;
    int rb = kRowBlock;
    while (rb > 64 && nc / ((long long)rb * CT) < target) rb >>= 1;
    if (alike && n0 > 0) {
      const bool tc2 = RP == 32;   // 128-column items, one CTA per SM
      const int ctw = tc2 ? 128 : CT;
      const double bpe = s->pass2_src == 0 ? 4.0 : (s->pass2_src == 1 ? 4.0 * s->W
                                                                        : (s->dtype == PSGD_F32 ? 4.0 : 2.0) * s->W);
      double best = -1.0;
      for (int r = kRowBlock; r >= 64; r -= 64) {
        std::vector<long long> sizes;
        for (auto& h : s->tensors) {
          if (!h.compressed) continue;
          for (long long r0 = 0; r0 < h.rows; r0 += r)
            for (long long c0 = 0; c0 < h.cols; c0 += ctw)
              sizes.push_back(std::min<long long>(r, h.rows - r0) * std::min<long long>(ctw, h.cols - c0));
        }
        std::stable_sort(sizes.begin(), sizes.end(), std::greater<long long>());
        const long long G = std::min<long long>((long long)sizes.size(), (long long)s->sms * (tc2 ? 1 : 3));
        const double t = rr_makespan(sizes, G, bpe, stall_bytes(2e-6, G) + 8.0 * RP * ctw);
        if (best < 0 || t < best * 0.999) {
          best = t;
          rb = r;
        }
      }
    }
    s->row_block = rb;
  }
  // uncompressed ranges, merged
  long long run_start = -1, run_len = 0;
  for (auto& h : s->tensors) {
    if (h.compressed) {
      if (run_len) add_segments(&s->unc_segs, run_start, run_len, 1024);
      run_start = -1;
      run_len = 0;
      TensorDesc td;
      td.g_off = h.offset;
      td.c_off = c_off;
      td.p_off = p_off;
      td.q_off = q_off;
      td.n = (int)h.rows;
      td.m = (int)h.cols;
      td.ld = (int)((h.cols + 3) / 4 * 4);
      td.r = h.rank;
      td.valid = h.valid >= 0 ? h.valid : h.numel;
      td.ctiles = (int)((h.cols + CT - 1) / CT);
      td.ctiles1 = (int)p1_tiles((int)h.cols).size();
      td.rblocks = (int)((h.rows + s->row_block - 1) / s->row_block);
      td.pp_off = pp_off;
      td.qp_off = qp_off;
      td.e_off = e_off;
      td.vec = (h.cols % 4 == 0) && (h.offset % 4 == 0);
      // operand images (ranks 16 and 32): hi and lo of P's and Q's row
      // images (rows padded to 128) and chunk images (RP x 32 per 32 rows)
      td.pi_off = td.qi_off = td.pti_off = td.qti_off = 0;
      if (RP >= 16) {
        const long long npad = (h.rows + 127) / 128 * 128, mpad = (h.cols + 127) / 128 * 128;
        const long long nch = (h.rows + 31) / 32, mch = (h.cols + 31) / 32;
        td.pi_off = i_off;
        i_off += 2 * npad * 32;
        td.qi_off = i_off;
        i_off += 2 * mpad * 32;
        td.pti_off = i_off;
        i_off += 2 * nch * RP * 32;
        td.qti_off = i_off;
        i_off += 2 * mch * RP * 32;
      }
      if (td.vec) s->any_aligned = 1;
      if (!td.vec || td.valid < (long long)td.n * td.m) s->any_unaligned = 1;
      h.cidx = (int)s->cdesc.size();
      h.e_off = e_off;
      s->cdesc.push_back(td);
      c_off += (h.rows * td.ld + 31) / 32 * 32;
      auto r32 = [](long long x) { return (x + 31) / 32 * 32; };
      p_off += h.rows * RP;
      q_off += r32(h.cols * RP);
      pp_off += (long long)td.ctiles1 * h.rows * RP;
      qp_off += r32((long long)td.rblocks * h.cols * RP);
      e_off += h.numel;
    } else {
      unc += h.numel;
      if (h.numel == 0) continue;
      if (run_len == 0) run_start = h.offset;
      run_len += h.numel;
    }
  }
  if (run_len) add_segments(&s->unc_segs, run_start, run_len, 1024);
  add_segments(&s->all_segs, 0, s->N);
  s->Nc_pad = c_off;
  s->Ne = e_off;
  s->Nunc = unc;
  s->Nc = s->N - unc;
  s->p_total = p_off;
  s->q_total = q_off;
  s->img_total = i_off;
  s->pp_total = pp_off;
  s->qp_total = qp_off;

  // pass items: (row block) x (column tile)
  std::vector<int> group_of(s->cdesc.size(), 0);
  if (s->batch) {
    // batch_tensors_with_same_shape ("PowerSGD State" item 5 of the later
    // page): same-shape tensors are scheduled next to each other.
    std::vector<std::pair<int, int>> shapes;
    for (size_t c = 0; c < s->cdesc.size(); ++c) {
      std::pair<int, int> sh(s->cdesc[c].n, s->cdesc[c].m);
      auto it = std::find(shapes.begin(), shapes.end(), sh);
      group_of[c] = (int)(it - shapes.begin());
      if (it == shapes.end()) shapes.push_back(sh);
    }
  }
  // cut: end a row block at the first row the bucket does not wholly back
  // (batched hook), so that the checked kernels get only the rows that need
  // them.  Not for pass 2, whose row blocks index its partial sums.
  // ctw > 0: uniform column tiles of ctw columns; ctw == 0: pass 1's tiles
  auto make_items = [&](std::vector<Item>* out, int rows_per_item, int ctw, bool cut) {
    for (size_t c = 0; c < s->cdesc.size(); ++c) {
      const TensorDesc& td = s->cdesc[c];
      std::vector<std::pair<int, int>> tiles;
      if (ctw > 0) {
        for (int c0 = 0; c0 < td.m; c0 += ctw) tiles.push_back({c0, std::min(ctw, td.m - c0)});
      } else {
        tiles = p1_tiles(td.m);
      }
      const int nct = (int)tiles.size();
      const long long vr = td.valid / td.m;   // rows [0, vr) are wholly backed
      for (int r0 = 0, r1; r0 < td.n; r0 = r1) {
        r1 = std::min(r0 + rows_per_item, td.n);
        if (cut && r0 < vr && vr < r1) r1 = (int)vr;
        for (int ct = 0; ct < nct; ++ct) {
          Item it;
          it.t = (int)c;
          it.row0 = r0;
          it.nrows = r1 - r0;
          it.col0 = tiles[ct].first;
          it.ncols = tiles[ct].second;
          it.rb = r0 / s->row_block;
          it.ct = ct;
          it.pad = group_of[c];
          out->push_back(it);
        }
      }
    }
    // largest items first (static round-robin over a persistent grid); with
    // batching, same-shape groups stay together.
    std::stable_sort(out->begin(), out->end(), [&](const Item& x, const Item& y) {
      if (s->batch && x.pad != y.pad) return x.pad < y.pad;
      return (long long)x.nrows * x.ncols > (long long)y.nrows * y.ncols;
    });
    for (auto& it : *out) it.pad = 0;
  };
  make_items(&s->items, s->row_block, CT, false);
  make_items(&s->fitems, kFineRows3, ctile3_for(RP), true);
  // pass 1 (ranks <= 8): items of fewer rows in small buckets (down to 32
  // rows while a bucket holds fewer than six items per SM), so that the last
  // wave over the SMs is short; tall items in large buckets, so that each
  // warp's copy pipeline drains and refills (and the item's setup loads wait)
  // less often.  When every compressed tensor has the same shape the items
  // are alike and the waves can be counted: the height (16 to 128 rows, a
  // multiple of 16) with the shortest round-robin makespan is taken (8192 x
  // 8192 alone: 112 rows, 592 items over 304 CTAs, against 1024 64-row ones).
  int rows1 = rows1_for(RP);
  if (RP <= 8 && !s->cdesc.empty()) {
    long long nc = 0;
    for (auto& h : s->tensors)
      if (h.compressed) nc += h.numel;
    bool alike = true;
    for (const TensorDesc& td : s->cdesc)
      alike = alike && td.n == s->cdesc[0].n && td.m == s->cdesc[0].m;
    if (!alike) {
      while (rows1 > 32 && nc < 6LL * s->sms * rows1 * CT1) rows1 /= 2;
    } else {
      const double g = s->dtype == PSGD_F32 ? 4.0 : 2.0;
      const double bpe = s->W * (g + (s->ef ? 8.0 : 0.0)) + (s->pass2_src == 0 ? 4.0 : 0.0);
      const int minb = s->W <= 2 ? 2 : 1;   // CTAs per SM of the chunk-stationary kernel
      double best = -1.0;
      int best_rows = rows1;
      for (int r = rows1_for(RP); r >= 16; r -= 16) {
        std::vector<Item> cand;
        make_items(&cand, r, 0, true);
        std::vector<long long> sizes(cand.size());
        for (size_t i = 0; i < cand.size(); ++i) sizes[i] = (long long)cand[i].nrows * cand[i].ncols;
        const long long G = std::min<long long>((long long)cand.size(), s->sms) * minb;
        const double t = rr_makespan(sizes, G, bpe, stall_bytes(5e-6, G));
        if (best < 0 || t < best * 0.995) {
          best = t;
          best_rows = r;
        }
      }
      rows1 = best_rows;
    }
  }
  make_items(&s->p1items, rows1, 0, true);
  // tensor-core pass 3 (ranks 16 and 32): 128 x 256 items of the tensors
  // whose rows are 16-byte aligned in the bucket and which the bucket wholly
  // backs, in (tensor, row block, column tile) order so that a CTA's
  // contiguous range of items shares row blocks of P
  if (RP >= 16) {
    for (size_t c = 0; c < s->cdesc.size(); ++c) {
      const TensorDesc& td = s->cdesc[c];
      if (!td.vec || td.valid != (long long)td.n * td.m) continue;
      for (int r0 = 0; r0 < td.n; r0 += 128)
        for (int c0 = 0; c0 < td.m; c0 += 256) {
          Item it;
          it.t = (int)c;
          it.row0 = r0;
          it.nrows = std::min(128, td.n - r0);
          it.col0 = c0;
          it.ncols = std::min(256, td.m - c0);
          it.rb = 0;
          it.ct = 0;
          it.pad = 0;
          s->t3items.push_back(it);
        }
    }
    // tensor-core pass 1: the pass-1 items whose rows are 16-byte aligned in
    // the bucket and which the bucket wholly backs, in (tensor, row block,
    // column tile) order; the element kernel takes the rest
    for (const Item& it : s->p1items) {
      const TensorDesc& td = s->cdesc[it.t];
      if (td.vec && (long long)(it.row0 + it.nrows) * td.m <= td.valid) s->t1items.push_back(it);
    }
    std::stable_sort(s->t1items.begin(), s->t1items.end(), [](const Item& x, const Item& y) {
      if (x.t != y.t) return x.t < y.t;
      if (x.row0 != y.row0) return x.row0 < y.row0;
      return x.col0 < y.col0;
    });
    // tensor-core pass 2: one row block x 128 columns of every compressed
    // tensor (its sources, the Mbar scratch and the store, always have
    // 16-byte aligned rows)
    for (size_t c = 0; c < s->cdesc.size(); ++c) {
      const TensorDesc& td = s->cdesc[c];
      for (int r0 = 0; r0 < td.n; r0 += s->row_block)
        for (int c0 = 0; c0 < td.m; c0 += 128) {
          Item it;
          it.t = (int)c;
          it.row0 = r0;
          it.nrows = std::min(s->row_block, td.n - r0);
          it.col0 = c0;
          it.ncols = std::min(128, td.m - c0);
          it.rb = r0 / s->row_block;
          it.ct = 0;
          it.pad = 0;
          s->t2items.push_back(it);
        }
    }
  }
  // P_raw: with at most two column-tile partials per row on average the first
  // Gram kernel adds them as it reads P (one launch fewer); with more, a
  // separate reduction with more loads in flight is faster
  {
    long long rows = 0, tile_rows = 0;
    for (const TensorDesc& td : s->cdesc) {
      rows += td.n;
      tile_rows += (long long)td.ctiles1 * td.n;
    }
    s->fold_psum = tile_rows <= 2 * rows ? 1 : 0;
  }
  for (size_t c = 0; c < s->cdesc.size(); ++c) {
    const long long len = (long long)s->cdesc[c].m * RP;
    for (long long f = 0; f < len; f += kQrChunk)
      s->qr.push_back({(int)c, (int)f, (int)std::min<long long>(kQrChunk, len - f), 0});
    const long long plen = (long long)s->cdesc[c].n * RP;
    for (long long f = 0; f < plen; f += 1024)
      s->ps.push_back({(int)c, (int)f, (int)std::min<long long>(1024, plen - f), 0});
  }

  for (size_t c = 0; c < s->cdesc.size(); ++c) {
    const TensorDesc& td = s->cdesc[c];
    // Gram-Schmidt items (one Gram partial each): kGsRows rows, fewer for
    // large ranks so that a single tall matrix still spreads over many CTAs
    const int per_p = std::max(64, std::min(kGsRows, 2048 / RP));
    const int per_q = per_p;
    s->gsp_first.push_back((int)s->gsp.size());
    for (int r0 = 0; r0 < td.n; r0 += per_p) s->gsp.push_back({(int)c, r0, std::min(per_p, td.n - r0), 0});
    s->gsp_count.push_back((int)s->gsp.size() - s->gsp_first.back());
    s->gsq_first.push_back((int)s->gsq.size());
    for (int r0 = 0; r0 < td.m; r0 += per_q) s->gsq.push_back({(int)c, r0, std::min(per_q, td.m - r0), 0});
    s->gsq_count.push_back((int)s->gsq.size() - s->gsq_first.back());
  }
  // the fused Gram-Schmidt stage: ranks up to 16 and at most 128 row items
  // per tensor (the completing CTA adds a tensor's partials and solves by
  // itself while the others wait at the next barrier; at rank 32 the 32 x 32
  // sums and solves are long enough that the eight-launch stage, whose sums
  // spread over many CTAs, is faster: 8192 x 8192 stage 152 against 119 us)
  {
    int most = 0;
    for (size_t c = 0; c < s->cdesc.size(); ++c) most = std::max(most, std::max(s->gsp_count[c], s->gsq_count[c]));
    s->gs_fused = (RP <= 16 && most <= 128) ? 1 : 0;
  }
}

StepArgs make_args(psgd_state* s) {
  StepArgs a;
  memset(&a, 0, sizeof(a));
  a.W = s->W;
  a.gtype = s->dtype == PSGD_F16 ? 1 : (s->dtype == PSGD_BF16 ? 2 : 0);
  a.scale = 1.f;
  a.invW = 1.f / (float)s->W;
  a.estore = s->estore;
  a.nc_pad = s->Nc_pad;
  a.est_half = s->est_halves == 2 ? (long long)s->W * s->Nc_pad : 0;
  a.mbar = (s->pass2_src == 0) ? s->mbar : nullptr;
  a.Pf = s->Pf;
  a.Qf = s->Qf;
  a.p_total = s->p_total;
  a.q_total = s->q_total;
  a.qinit = s->qinit;
  a.qdraw = s->qdraw;
  a.praw_part = s->praw_part;
  a.praw = s->praw;
  a.pgs = s->pgs;
  a.qpart = s->qpart;
  a.gram = s->gram;
  a.gram_t = s->gram_t;
  a.tmat = s->tmat;
  a.tmat2 = s->tmat2;
  a.gs_cnt = s->gs_cnt;
  a.commit_cnt = nullptr;
  a.status = nullptr;
  a.tensors = s->d_tensors;
  a.items = s->d_items;
  a.n_items = (int)s->items.size();
  a.fitems = s->d_fitems;
  a.n_fitems = (int)s->fitems.size();
  a.p1items = s->d_p1items;
  a.n_p1items = (int)s->p1items.size();
  a.img = s->img;
  a.t3items = s->d_t3items;
  a.n_t3 = (int)s->t3items.size();
  a.t2items = s->d_t2items;
  a.n_t2 = (int)s->t2items.size();
  a.t1items = s->d_t1items;
  a.n_t1 = (int)s->t1items.size();
  a.ps_items = s->d_ps;
  a.n_ps = (int)s->ps.size();
  a.qr_items = s->d_qr;
  a.n_qr = (int)s->qr.size();
  a.gsp_items = s->d_gsp;
  a.n_gsp = (int)s->gsp.size();
  a.gsq_items = s->d_gsq;
  a.n_gsq = (int)s->gsq.size();
  const int nt = (int)s->cdesc.size();
  a.gsp_first = s->d_gs_index;
  a.gsp_count = s->d_gs_index + nt;
  a.gsq_first = s->d_gs_index + 2 * nt;
  a.gsq_count = s->d_gs_index + 3 * nt;
  a.n_tensors = nt;
  a.ctrl = s->ctrl;
  a.ef = s->ef;
  a.warm_start = s->warm;
  a.vec_ok = 1;
  a.has_aligned = s->any_aligned;
  a.has_unaligned = s->any_unaligned;
  a.gn = s->N;
  a.eps = s->eps;
  return a;
}

// Kernel launches, optionally bracketed by profiling events.
struct Launcher {
  psgd_state* s;
  cudaStream_t st;
  EventPair cur{};
  bool on = false;
  int kind = 0;
  void begin(int k) {
    kind = k;
    on = s->prof && ((s->prof_mask >> k) & 1u);
    if (!on) return;
    if (s->ev_pool.empty()) {
      EventPair p;
      cudaEventCreate(&p.a);
      cudaEventCreate(&p.b);
      s->ev_pool.push_back(p);
    }
    cur = s->ev_pool.back();
    s->ev_pool.pop_back();
    cudaEventRecord(cur.a, st);
  }
  void end() {
    if (!on) return;
    cudaEventRecord(cur.b, st);
    s->ev[kind].push_back(cur);
  }
};

template <int RP>
struct Ops {
  // do_psum: P_raw still has to be summed from pass 1's partials (the
  // data-parallel split sums them before its exchange instead)
  // Returns true when the stage also wrote P's operand images (ranks 16 and
  // 32, the cooperative launch), so images(mode 0) is not needed.
  static bool gs(psgd_state* s, const StepArgs& a, Launcher& L, int is_q, bool do_psum = true) {
    const int n_items = is_q ? a.n_gsq : a.n_gsp;
    const int grid = std::max(1, std::min(n_items, s->sms * 4));
    const float* src_dense = is_q ? s->qdraw : s->praw;
    const bool psum = !is_q && !s->fold_psum && do_psum;
    if (s->gs_fused && s->gs_coop) {
      // the whole stage (with the P_raw sum) in one cooperative launch
      const bool parts = !is_q && s->fold_psum;
      L.begin(K_GS);
      const cudaError_t e = launch_gs_coop<RP>(
          a, parts ? s->praw_part : src_dense, parts ? s->praw : nullptr, is_q, parts ? 1 : 0, s->pgs,
          is_q ? s->qinit : s->Pf, is_q ? -1 : 1, psum ? 1 : 0, s->gs_bar, (RP >= 16 && !is_q) ? 1 : 0,
          std::max(grid, psum ? std::min(a.n_ps, s->sms * 4) : 1), L.st, s->test_wait_skew);
      s->test_wait_skew = 0;
      L.end();
      if (e == cudaSuccess) return RP >= 16 && !is_q;
      // refused (no cooperative launch here): the three-launch stage from now on
      (void)cudaGetLastError();
      s->gs_coop = 0;
    }
    if (psum) {
      // P_raw = sum of pass 1's column-tile partials
      L.begin(K_PSUM);
      launch_psum<RP>(a, std::max(1, std::min(a.n_ps, s->sms * 8)), L.st);
      L.end();
    }
    if (s->gs_fused) {
      // Gram + solve, apply + Gram + solve, apply: three launches
      L.begin(K_GRAM);
      if (is_q || !s->fold_psum)
        launch_gs_first<RP>(a, src_dense, nullptr, is_q, 0, grid, L.st);
      else
        launch_gs_first<RP>(a, s->praw_part, s->praw, 0, 1, grid, L.st);
      L.end();
      L.begin(K_SOLVE);
      launch_gs_second<RP>(a, src_dense, s->pgs, is_q, grid, L.st);
      L.end();
      L.begin(K_APPLY);
      if (is_q)
        launch_apply<RP>(a, s->pgs, s->qinit, 1, -1, grid, L.st, s->tmat2);
      else
        launch_apply<RP>(a, s->pgs, s->Pf, 0, 1, grid, L.st, s->tmat2);
      L.end();
      return false;
    }
    L.begin(K_GRAM);
    if (is_q || !s->fold_psum) {
      launch_gram<RP>(a, src_dense, nullptr, is_q, 0, s->gram, grid, L.st);
    } else {
      // P_raw = the sum of pass 1's column-tile partials (in tile order),
      // written dense while its Gram matrices are formed
      launch_gram<RP>(a, s->praw_part, s->praw, 0, 1, s->gram, grid, L.st);
    }
    launch_gram_sum<RP>(a, is_q, L.st);
    L.end();
    L.begin(K_SOLVE);
    launch_solve<RP>(a, s->gram_t, is_q, 0, L.st);
    L.end();
    L.begin(K_APPLY);
    launch_apply<RP>(a, src_dense, s->pgs, is_q, -1, grid, L.st);
    L.end();
    L.begin(K_GRAM);
    launch_gram<RP>(a, s->pgs, nullptr, is_q, 0, s->gram, grid, L.st);
    launch_gram_sum<RP>(a, is_q, L.st);
    L.end();
    L.begin(K_SOLVE);
    launch_solve<RP>(a, s->gram_t, is_q, 1, L.st);
    L.end();
    L.begin(K_APPLY);
    if (is_q)
      launch_apply<RP>(a, s->pgs, s->qinit, 1, -1, grid, L.st);
    else
      launch_apply<RP>(a, s->pgs, s->Pf, 0, 1, grid, L.st, nullptr, RP >= 16 ? 1 : 0);   // with P's images
    L.end();
    return RP >= 16 && !is_q;
  }

  // ranks 16 and 32: the factor images the tensor-core passes read
  static void images(psgd_state* s, const StepArgs& a, Launcher& L, int mode) {
    if constexpr (RP >= 16) {
      const int n = (mode == 0) ? a.n_gsp : (mode == 3 ? a.n_gsp + a.n_gsq : a.n_gsq);
      L.begin(K_IMG);
      launch_images<RP>(a, mode, std::max(1, std::min(n, s->sms * 4)), L.st);
      L.end();
    }
  }

  static void compressed(psgd_state* s, const StepArgs& a, Launcher& L, bool need_fresh,
                         const std::vector<int>& mask) {
    const int grid_items = std::max(1, std::min(a.n_items, s->sms * 3));
    const int grid_fine = std::max(1, std::min(a.n_fitems, s->sms * 2));
    const int grid_p1 = std::max(1, std::min(a.n_p1items, s->sms));  // x CTAs per SM inside
    const int grid_ps = std::max(1, std::min(a.n_ps, s->sms * 8));
    const int grid_q = std::max(1, std::min(a.n_gsq, s->sms * 4));
    const int grid_qr = std::max(1, std::min(a.n_qr, s->sms * 8));
    if (need_fresh) {
      cudaMemcpyAsync(s->d_mask, mask.data(), mask.size() * sizeof(int), cudaMemcpyHostToDevice, L.st);
      L.begin(K_RANDN);
      launch_randn(a, s->d_mask, s->seed, (unsigned long long)s->iter, s->tensor_base, RP, grid_q, L.st);
      L.end();
      gs(s, a, L, 1);
    }
    // Q's chunk image (pass 1's projection operand): the last committed step
    // (or set_q) wrote it for a warm Q, so only a fresh draw needs it here
    if (need_fresh || !s->warm) images(s, a, L, 2);
    L.begin(K_PASS1);
    launch_pass1<RP>(a, grid_p1, L.st);
    L.end();
    if (!gs(s, a, L, 0)) images(s, a, L, 0);
    L.begin(K_PASS2);
    launch_pass2<RP>(a, s->pass2_src, grid_items, L.st);
    L.end();
    L.begin(K_QREDUCE);
    launch_qreduce<RP>(a, grid_qr, L.st, RP >= 16 ? 1 : 0);   // with Q's row image
    L.end();
    L.begin(K_PASS3);
    launch_pass3<RP>(a, 0, grid_fine, L.st);
    L.end();
  }

  // Data-parallel split, stage 1: a fresh Q when needed, pass 1 on the one
  // local replica, and this process's P_raw summed densely into the
  // exchange buffer (a.praw points into it).
  static void dp_begin(psgd_state* s, const StepArgs& a, Launcher& L, bool need_fresh,
                       const std::vector<int>& mask) {
    const int grid_p1 = std::max(1, std::min(a.n_p1items, s->sms));
    const int grid_ps = std::max(1, std::min(a.n_ps, s->sms * 8));
    const int grid_q = std::max(1, std::min(a.n_gsq, s->sms * 4));
    if (need_fresh) {
      cudaMemcpyAsync(s->d_mask, mask.data(), mask.size() * sizeof(int), cudaMemcpyHostToDevice, L.st);
      L.begin(K_RANDN);
      launch_randn(a, s->d_mask, s->seed, (unsigned long long)s->iter, s->tensor_base, RP, grid_q, L.st);
      L.end();
      gs(s, a, L, 1);
    }
    // Q's chunk image (pass 1's projection operand): the last committed step
    // (or set_q) wrote it for a warm Q, so only a fresh draw needs it here
    if (need_fresh || !s->warm) images(s, a, L, 2);
    L.begin(K_PASS1);
    launch_pass1<RP>(a, grid_p1, L.st);
    L.end();
    L.begin(K_PSUM);
    launch_psum<RP>(a, grid_ps, L.st);
    L.end();
  }

  // Stage 2 (after the exchanged P sum became the mean): orthogonalise P,
  // then this process's Q = M^T P into the second exchange buffer (a.qx).
  static void dp_project(psgd_state* s, const StepArgs& a, Launcher& L) {
    const int grid_items = std::max(1, std::min(a.n_items, s->sms * 3));
    const int grid_qr = std::max(1, std::min(a.n_qr, s->sms * 8));
    if (!gs(s, a, L, 0, false)) images(s, a, L, 0);
    L.begin(K_PASS2);
    launch_pass2<RP>(a, s->pass2_src, grid_items, L.st);
    L.end();
    L.begin(K_QREDUCE);
    launch_qreduce<RP>(a, grid_qr, L.st);
    L.end();
  }

  // Stage 3 (after the exchanged Q sum became the mean): out = P Q^T.
  static void dp_finish(psgd_state* s, const StepArgs& a, Launcher& L) {
    const int grid_fine = std::max(1, std::min(a.n_fitems, s->sms * 2));
    images(s, a, L, 1);
    L.begin(K_PASS3);
    launch_pass3<RP>(a, 0, grid_fine, L.st);
    L.end();
  }

  static void errview(psgd_state* s, const StepArgs& a, int mode, cudaStream_t st) {
    const int grid_fine = std::max(1, std::min(a.n_fitems, s->sms * 2));
    launch_pass3<RP>(a, mode, grid_fine, st);
  }
};

template <template <int> class F, typename... Args>
void by_rp(int rp, Args&&... args) {
  switch (rp) {
    case 1: F<1>::run(args...); break;
    case 2: F<2>::run(args...); break;
    case 4: F<4>::run(args...); break;
    case 8: F<8>::run(args...); break;
    case 16: F<16>::run(args...); break;
    default: F<32>::run(args...); break;
  }
}

template <int RP>
struct RunCompressed {
  static void run(psgd_state* s, const StepArgs& a, Launcher& L, bool need_fresh, const std::vector<int>& mask) {
    Ops<RP>::compressed(s, a, L, need_fresh, mask);
  }
};
template <int RP>
struct RunDpBegin {
  static void run(psgd_state* s, const StepArgs& a, Launcher& L, bool need_fresh, const std::vector<int>& mask) {
    Ops<RP>::dp_begin(s, a, L, need_fresh, mask);
  }
};
template <int RP>
struct RunDpProject {
  static void run(psgd_state* s, const StepArgs& a, Launcher& L) { Ops<RP>::dp_project(s, a, L); }
};
template <int RP>
struct RunDpFinish {
  static void run(psgd_state* s, const StepArgs& a, Launcher& L) { Ops<RP>::dp_finish(s, a, L); }
};
template <int RP>
struct RunImages {
  static void run(psgd_state* s, const StepArgs& a, Launcher& L, int mode) { Ops<RP>::images(s, a, L, mode); }
};
template <int RP>
struct RunErrView {
  static void run(psgd_state* s, const StepArgs& a, int mode, cudaStream_t st) { Ops<RP>::errview(s, a, mode, st); }
};

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const char* x = (const char*)a;
  const char* y = (const char*)b;
  return x < y + nb && y < x + na;
}

}  // namespace

namespace {
int create_common(psgd_state* s, int32_t world_size, int32_t rank, int64_t start_iter, double mcr,
                  int32_t use_error_feedback, int32_t warm_start, float eps, uint64_t random_seed,
                  int32_t batch, psgd_dtype grad_dtype, int32_t device, psgd_state** out);
}  // namespace

#ifndef PSGD_SOURCE_HASH
#define PSGD_SOURCE_HASH "unknown"
#endif

extern "C" {

const char* psgd_last_error(void) { return g_last_error.c_str(); }

const char* psgd_build_id(void) { return "psgd-source-hash:" PSGD_SOURCE_HASH; }

int psgd_plan(const int64_t* dims, const int32_t* ndims, int32_t n_tensors, int32_t rank, double mcr,
              int32_t* compressed, int32_t* ranks, int64_t* rows, int64_t* cols) {
  std::vector<HostTensor> ts;
  int rc = plan_tensors(dims, ndims, n_tensors, rank, mcr, &ts);
  if (rc) return rc;
  for (int t = 0; t < n_tensors; ++t) {
    if (compressed) compressed[t] = ts[t].compressed;
    if (ranks) ranks[t] = ts[t].rank;
    if (rows) rows[t] = ts[t].rows;
    if (cols) cols[t] = ts[t].cols;
  }
  return PSGD_OK;
}

void psgd_state_destroy(psgd_state* s) {
  if (!s) return;
  DeviceGuard g(s->device);
  for (void* p : s->allocs) cudaFree(p);
  for (int k = 0; k < 2; ++k) {
    for (void* p : s->stage_grads[k]) cudaFree(p);
    if (s->stage_out[k]) cudaFree(s->stage_out[k]);
    if (s->ev_in[k]) cudaEventDestroy(s->ev_in[k]);
    if (s->ev_comp[k]) cudaEventDestroy(s->ev_comp[k]);
    if (s->ev_free[k]) cudaEventDestroy(s->ev_free[k]);
  }
  if (s->s_in) cudaStreamDestroy(s->s_in);
  if (s->s_out) cudaStreamDestroy(s->s_out);
  if (s->gexec) cudaGraphExecDestroy(s->gexec);
  if (s->s_cap) cudaStreamDestroy(s->s_cap);
  if (s->h_status) cudaFreeHost(s->h_status);
  for (auto& v : s->ev)
    for (auto& e : v) {
      cudaEventDestroy(e.a);
      cudaEventDestroy(e.b);
    }
  for (auto& e : s->ev_pool) {
    cudaEventDestroy(e.a);
    cudaEventDestroy(e.b);
  }
  delete s;
}

int psgd_state_create(const int64_t* dims, const int32_t* ndims, int32_t n_tensors, int32_t world_size,
                      int32_t rank, int64_t start_iter, double mcr, int32_t use_error_feedback,
                      int32_t warm_start, float eps, uint64_t random_seed, int32_t batch,
                      psgd_dtype grad_dtype, int32_t device, psgd_state** out) {
  if (!out) return fail(PSGD_EINVAL, "out is NULL");
  *out = nullptr;
  if (world_size < 1 || world_size > PSGD_MAX_WORLD) return fail(PSGD_EINVAL, "world_size must be in [1, 64]");
  if (start_iter < 0) return fail(PSGD_EINVAL, "start_powerSGD_iter < 0");
  if (!(eps >= 0.f)) return fail(PSGD_EINVAL, "orthogonalization_epsilon must be >= 0");
  if (grad_dtype != PSGD_F32 && grad_dtype != PSGD_F16 && grad_dtype != PSGD_BF16)
    return fail(PSGD_EINVAL, "grad_dtype");
  psgd_state* s = new psgd_state();
  int rc = plan_tensors(dims, ndims, n_tensors, rank, mcr, &s->tensors);
  if (rc) {
    delete s;
    return rc;
  }
  for (auto& h : s->tensors) s->N += h.numel;
  return create_common(s, world_size, rank, start_iter, mcr, use_error_feedback, warm_start, eps, random_seed,
                       batch, grad_dtype, device, out);
}

// The batched hook: one compressed (side x side) view of the whole bucket,
// side = ceil(sqrt(numel)), backed by the bucket for its first `numel`
// elements and zero beyond.
int psgd_state_create_batched(int64_t numel, int32_t world_size, int32_t rank, int64_t start_iter,
                              int32_t use_error_feedback, int32_t warm_start, float eps, uint64_t random_seed,
                              psgd_dtype grad_dtype, int32_t device, psgd_state** out) {
  if (!out) return fail(PSGD_EINVAL, "out is NULL");
  *out = nullptr;
  if (numel < 1) return fail(PSGD_EINVAL, "numel must be >= 1");
  if (rank < 1 || rank > PSGD_MAX_RANK) return fail(PSGD_EINVAL, "matrix_approximation_rank must be in [1, 32]");
  if (world_size < 1 || world_size > PSGD_MAX_WORLD) return fail(PSGD_EINVAL, "world_size must be in [1, 64]");
  if (start_iter < 0) return fail(PSGD_EINVAL, "start_powerSGD_iter < 0");
  if (!(eps >= 0.f)) return fail(PSGD_EINVAL, "orthogonalization_epsilon must be >= 0");
  if (grad_dtype != PSGD_F32 && grad_dtype != PSGD_F16 && grad_dtype != PSGD_BF16)
    return fail(PSGD_EINVAL, "grad_dtype");
  long long side = (long long)std::sqrt((double)numel);
  while (side * side < numel) ++side;
  while (side > 1 && (side - 1) * (side - 1) >= numel) --side;
  if (side > 2147483647LL) return fail(PSGD_EINVAL, "bucket too large");
  psgd_state* s = new psgd_state();
  HostTensor h;
  h.shape = {side, side};
  h.offset = 0;
  h.numel = side * side;
  h.compressed = 1;
  h.rows = side;
  h.cols = side;
  h.rank = (int)std::min<long long>(rank, side);
  h.valid = numel;
  s->tensors.push_back(h);
  s->N = numel;
  s->batched = 1;
  return create_common(s, world_size, rank, start_iter, 0.0, use_error_feedback, warm_start, eps, random_seed,
                       0, grad_dtype, device, out);
}

}  // extern "C"

namespace {
int create_common(psgd_state* s, int32_t world_size, int32_t rank, int64_t start_iter, double mcr,
                  int32_t use_error_feedback, int32_t warm_start, float eps, uint64_t random_seed,
                  int32_t batch, psgd_dtype grad_dtype, int32_t device, psgd_state** out) {
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    delete s;
    return fail(PSGD_ECUDA, "no such CUDA device");
  }
  if (device >= 64) {   // per-device launch settings are kept for ordinals 0-63
    delete s;
    return fail(PSGD_EINVAL, "device ordinals from 64 up are not supported");
  }
  DeviceGuard g(device);
  s->device = device;
  s->W = world_size;
  s->rank = rank;
  s->RP = next_pow2(rank);
  s->start_iter = start_iter;
  s->mcr = mcr;
  s->ef = use_error_feedback ? 1 : 0;
  s->warm = warm_start ? 1 : 0;
  s->eps = eps;
  s->seed = random_seed;
  s->batch = batch ? 1 : 0;
  s->dtype = grad_dtype;
  cudaDeviceGetAttribute(&s->sms, cudaDevAttrMultiProcessorCount, device);
  // Where pass 2 reads the replica mean: a scratch copy written by pass 1
  // costs 8 bytes per element; re-reading the W sources costs W * 4 (store)
  // or W * sizeof(grad) (no error feedback).  Take the cheaper.
  const int gsz = grad_dtype == PSGD_F32 ? 4 : 2;
  const int reread = s->W * (s->ef ? 4 : gsz);
  s->pass2_src = (reread <= 8) ? (s->ef ? 1 : 2) : 0;
  if (s->W == 1 && s->ef) s->pass2_src = 1;
  build_plan(s);

  if (s->dp_world) s->fold_psum = 0;   // P_raw must be dense before the exchange
  const size_t RP = s->RP;
  const int nt = (int)s->cdesc.size();
  std::vector<int> gs_index;
  gs_index.insert(gs_index.end(), s->gsp_first.begin(), s->gsp_first.end());
  gs_index.insert(gs_index.end(), s->gsp_count.begin(), s->gsp_count.end());
  gs_index.insert(gs_index.end(), s->gsq_first.begin(), s->gsq_first.end());
  gs_index.insert(gs_index.end(), s->gsq_count.begin(), s->gsq_count.end());
  auto zero_now = [&](void* p, size_t n) -> int {
    if (p && n) PSGD_CUDA_TRY(cudaMemset(p, 0, n));
    return PSGD_OK;
  };
#define TRY(x)                  \
  do {                          \
    int rc_ = (x);              \
    if (rc_) {                  \
      psgd_state_destroy(s);    \
      return rc_;               \
    }                           \
  } while (0)
  TRY(dupload(s, &s->d_tensors, s->cdesc));
  TRY(dupload(s, &s->d_items, s->items));
  TRY(dupload(s, &s->d_fitems, s->fitems));
  TRY(dupload(s, &s->d_p1items, s->p1items));
  TRY(dupload(s, &s->d_t3items, s->t3items));
  TRY(dupload(s, &s->d_t2items, s->t2items));
  TRY(dupload(s, &s->d_t1items, s->t1items));
  if (s->img_total) {
    TRY(dalloc(s, (void**)&s->img, (size_t)s->img_total * sizeof(float)));
    TRY(zero_now(s->img, (size_t)s->img_total * sizeof(float)));
  }
  TRY(dupload(s, &s->d_ps, s->ps));
  TRY(dupload(s, &s->d_qr, s->qr));
  TRY(dupload(s, &s->d_gsp, s->gsp));
  TRY(dupload(s, &s->d_gsq, s->gsq));
  TRY(dupload(s, &s->d_gs_index, gs_index));
  TRY(dupload(s, &s->d_unc, s->unc_segs));
  TRY(dupload(s, &s->d_all, s->all_segs));
  TRY(dalloc(s, (void**)&s->d_mask, std::max(1, nt) * sizeof(int)));
  if (s->ef) TRY(dalloc(s, (void**)&s->estore, 2 * (size_t)s->W * s->Nc_pad * sizeof(float)));
  if (s->pass2_src == 0) TRY(dalloc(s, (void**)&s->mbar, (size_t)s->Nc_pad * sizeof(float)));
  TRY(dalloc(s, (void**)&s->Pf, 2 * (size_t)s->p_total * sizeof(float)));
  TRY(dalloc(s, (void**)&s->Qf, 2 * (size_t)s->q_total * sizeof(float)));
  TRY(dalloc(s, (void**)&s->qinit, (size_t)s->q_total * sizeof(float)));
  TRY(dalloc(s, (void**)&s->qdraw, (size_t)s->q_total * sizeof(float)));
  TRY(dalloc(s, (void**)&s->praw_part, (size_t)s->pp_total * sizeof(float)));
  if (s->dp_world) {
    // first exchange: [P_raw | pad to 32 | uncompressed values | flag]; P_raw
    // is summed straight into it.  Second exchange: Q in the Qf layout.
    s->xp_unc = (s->p_total + 31) / 32 * 32;
    s->xp_count = s->xp_unc + s->Nunc + 1;
    TRY(dalloc(s, (void**)&s->xp, (size_t)s->xp_count * sizeof(float)));
    s->praw = s->xp;
    TRY(dalloc(s, (void**)&s->xq, std::max<size_t>(1, (size_t)s->q_total) * sizeof(float)));
    std::vector<long long> upos, apos;
    long long acc = 0;
    for (const Segment& sg : s->unc_segs) {
      upos.push_back(acc);
      acc += sg.len;
    }
    for (const Segment& sg : s->all_segs) apos.push_back(sg.off);
    TRY(dupload(s, &s->d_unc_pos, upos));
    TRY(dupload(s, &s->d_all_pos, apos));
  } else {
    TRY(dalloc(s, (void**)&s->praw, (size_t)s->p_total * sizeof(float)));
  }
  TRY(dalloc(s, (void**)&s->pgs, (size_t)std::max(s->p_total, s->q_total) * sizeof(float)));
  TRY(dalloc(s, (void**)&s->qpart, (size_t)s->qp_total * sizeof(float)));
  TRY(dalloc(s, (void**)&s->tmat, std::max(1, nt) * RP * RP * sizeof(float)));
  TRY(dalloc(s, (void**)&s->tmat2, std::max(1, nt) * RP * RP * sizeof(float)));
  TRY(dalloc(s, (void**)&s->gs_cnt, std::max(1, nt) * sizeof(int)));
  TRY(dalloc(s, (void**)&s->gs_bar, 16));
  TRY(dalloc(s, (void**)&s->p3_cnt, 16));
  TRY(zero_now(s->p3_cnt, 16));
  TRY(zero_now(s->gs_cnt, std::max(1, nt) * sizeof(int)));
  TRY(dalloc(s, (void**)&s->gram, std::max<size_t>(1, std::max(s->gsp.size(), s->gsq.size())) * RP * RP * sizeof(float2)));
  TRY(dalloc(s, (void**)&s->gram_t, std::max(1, nt) * RP * RP * sizeof(float2)));
  TRY(dalloc(s, (void**)&s->ctrl, sizeof(Ctrl)));
  TRY(dalloc(s, (void**)&s->d_status, sizeof(int)));
  if (cudaMallocHost((void**)&s->h_status, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    s->h_status = nullptr;
    psgd_state_destroy(s);
    return fail(PSGD_ENOMEM, "cudaMallocHost");
  }
  *s->h_status = 0;
  // zero state: error store, factors, Q buffers, control block
  auto zero = [&](void* p, size_t n) -> int {
    if (p && n) PSGD_CUDA_TRY(cudaMemset(p, 0, n));
    return PSGD_OK;
  };
  if (s->ef) TRY(zero(s->estore, 2 * (size_t)s->W * s->Nc_pad * sizeof(float)));
  if (s->mbar) TRY(zero(s->mbar, (size_t)s->Nc_pad * sizeof(float)));
  TRY(zero(s->Pf, 2 * (size_t)s->p_total * sizeof(float)));
  TRY(zero(s->Qf, 2 * (size_t)s->q_total * sizeof(float)));
  TRY(zero(s->qinit, (size_t)s->q_total * sizeof(float)));
  TRY(zero(s->qdraw, (size_t)s->q_total * sizeof(float)));
  TRY(zero(s->praw_part, (size_t)s->pp_total * sizeof(float)));
  if (s->dp_world) {
    TRY(zero(s->xp, (size_t)s->xp_count * sizeof(float)));
    TRY(zero(s->xq, (size_t)s->q_total * sizeof(float)));
  } else {
    TRY(zero(s->praw, (size_t)s->p_total * sizeof(float)));
  }
  TRY(zero(s->ctrl, sizeof(Ctrl)));
  TRY(zero(s->d_status, sizeof(int)));
  s->pending_draw.assign(nt, 0);
  s->ev.assign(K_COUNT, {});
  // algorithmic bytes per launch of the streaming kernels
  {
    const double W = s->W;
    const double g = gsz;
    const double nc = (double)s->Nc;
    s->kind_bytes[K_PASS1] = nc * (W * (g + (s->ef ? 8.0 : 0.0)) + (s->pass2_src == 0 ? 4.0 : 0.0));
    const double src = s->pass2_src == 0 ? 4.0 : (s->pass2_src == 1 ? 4.0 * W : g * W);
    s->kind_bytes[K_PASS2] = nc * src;
    s->kind_bytes[K_PASS3] = nc * 4.0;
    s->kind_bytes[K_MEAN] = (double)s->Nunc * (W * g + 4.0);
  }
  PSGD_CUDA_TRY(cudaDeviceSynchronize());
  *out = s;
  return PSGD_OK;
#undef TRY
}
}  // namespace

extern "C" {

}  // extern "C"

namespace {

// The work of one step, enqueued on `st`; host counters are the caller's.
int enqueue_step(psgd_state* s, const StepArgs& a, cudaStream_t st, bool vanilla, bool compressed_step,
                 bool need_fresh, const std::vector<int>& mask) {
  Launcher L{s, st};
  bool committed = false;
  PSGD_CUDA_TRY(cudaMemsetAsync(&s->ctrl->flag, 0, 2 * sizeof(int), st));   // flag, timeout
  const int grid_seg = std::max(1, std::min<int>((int)s->all_segs.size(), s->sms * 4));
  if (vanilla) {
    // before start_powerSGD_iter calls the hook only averages the replicas
    // ("PowerSGD State", start_powerSGD_iter)
    L.begin(K_MEAN);
    launch_mean(a, s->d_all, (int)s->all_segs.size(), grid_seg, st);
    L.end();
  } else {
    if (!s->unc_segs.empty()) {
      L.begin(K_MEAN);
      launch_mean(a, s->d_unc, (int)s->unc_segs.size(),
                  std::max(1, std::min<int>((int)s->unc_segs.size(), s->sms * 4)), st);
      L.end();
    }
    if (compressed_step) {
      // pass 3 as one launch (ranks <= 8; at ranks 16 and 32 when the
      // tensor-core kernel covers every tensor): its last CTA commits the step
      StepArgs c = a;
      const bool one_pass3 = s->RP <= 8 || (!s->t3items.empty() && !s->any_unaligned);
      if (one_pass3) {
        c.commit_cnt = s->p3_cnt;
        c.status = s->d_status;
      }
      by_rp<RunCompressed>(s->RP, s, c, L, need_fresh, mask);
      committed = one_pass3;
    }
  }
  if (!committed) {
    L.begin(K_COMMIT);
    launch_commit(s->ctrl, compressed_step ? 1 : 0, s->d_status, st);
    L.end();
  }
  PSGD_CUDA_TRY(cudaGetLastError());
  PSGD_CUDA_TRY(cudaMemcpyAsync(s->h_status, s->d_status, sizeof(int), cudaMemcpyDeviceToHost, st));
  return PSGD_OK;
}

void drop_graph(psgd_state* s) {
  if (s->gexec) cudaGraphExecDestroy(s->gexec);
  s->gexec = nullptr;
  s->gkey_grads.clear();
  s->gkey_out = nullptr;
}

// Replays the steady step's graph on `st`, capturing it first (on the
// private stream s_cap, which executes nothing while capturing) when there is
// none for these pointers and this scale.
int step_graph(psgd_state* s, const StepArgs& a, const void* const* grads, const float* out, float scale,
               cudaStream_t st) {
  bool same = s->gexec && s->gkey_out == out && s->gkey_scale == scale && (int)s->gkey_grads.size() == s->W;
  for (int w = 0; same && w < s->W; ++w) same = s->gkey_grads[w] == grads[w];
  if (!same) {
    drop_graph(s);
    if (!s->s_cap) PSGD_CUDA_TRY(cudaStreamCreateWithFlags(&s->s_cap, cudaStreamNonBlocking));
    PSGD_CUDA_TRY(cudaStreamBeginCapture(s->s_cap, cudaStreamCaptureModeThreadLocal));
    const int rc = enqueue_step(s, a, s->s_cap, false, true, false, std::vector<int>(s->cdesc.size(), 0));
    cudaGraph_t graph = nullptr;
    const cudaError_t e = cudaStreamEndCapture(s->s_cap, &graph);
    if (rc < 0 || e != cudaSuccess || !graph) {
      if (graph) cudaGraphDestroy(graph);
      cudaGetLastError();
      return rc < 0 ? rc : fail(PSGD_ECUDA, std::string("psgd_step: graph capture: ") + cudaGetErrorString(e));
    }
    const cudaError_t ei = cudaGraphInstantiate(&s->gexec, graph, 0);
    cudaGraphDestroy(graph);
    if (ei != cudaSuccess) {
      s->gexec = nullptr;
      cudaGetLastError();
      return fail(PSGD_ECUDA, std::string("psgd_step: graph instantiate: ") + cudaGetErrorString(ei));
    }
    s->gkey_grads.assign(grads, grads + s->W);
    s->gkey_out = out;
    s->gkey_scale = scale;
    s->graph_captures++;
  }
  PSGD_CUDA_TRY(cudaGraphLaunch(s->gexec, st));
  s->graph_replays++;
  return PSGD_OK;
}

}  // namespace

extern "C" {

int psgd_step(psgd_state* s, const void* const* grads, float* out, float inv_loss_scale, void* stream) {
  if (!s) return fail(PSGD_EINVAL, "state is NULL");
  if (s->dp_world) return fail(PSGD_EINVAL, "psgd_step: a data-parallel state steps with psgd_dp_begin/project/finish");
  if (!grads || !out) return fail(PSGD_EINVAL, "grads/out is NULL");
  const size_t gsz = s->dtype == PSGD_F32 ? 4 : 2;
  for (int w = 0; w < s->W; ++w) {
    if (!grads[w]) return fail(PSGD_EINVAL, "grads[w] is NULL");
    const bool same = (grads[w] == (const void*)out);
    if (ranges_overlap(grads[w], s->N * gsz, out, s->N * 4)) {
      if (!(w == 0 && same && s->dtype == PSGD_F32))
        return fail(PSGD_EINVAL, "out overlaps a replica bucket (only out == grads[0] for F32 is allowed)");
    }
  }
  DeviceGuard g(s->device);
  cudaStream_t st = (cudaStream_t)stream;
  StepArgs a = make_args(s);
  for (int w = 0; w < s->W; ++w) a.grads.p[w] = grads[w];
  a.out = out;
  a.scale = inv_loss_scale;
  int vec_ok = ((uintptr_t)out % 16 == 0);
  for (int w = 0; w < s->W; ++w) vec_ok &= ((uintptr_t)grads[w] % (s->dtype == PSGD_F32 ? 16 : 8) == 0);
  a.vec_ok = vec_ok;
  const bool vanilla = s->iter < s->start_iter;
  const bool compressed_step = !vanilla && !s->cdesc.empty();
  const bool need_fresh = compressed_step && ((!s->warm) || s->compressed_launched == 0);
  if (s->graph_mode && !s->prof && compressed_step && !need_fresh) {
    // steady compressed step: the launch sequence no longer changes, and every
    // decision left (skip, double-buffer half, warm or fresh Q) is taken on
    // the device, so one captured graph replays it
    int rc = step_graph(s, a, grads, out, inv_loss_scale, st);
    if (rc < 0) return rc;
  } else {
    std::vector<int> mask(s->cdesc.size(), 0);
    if (need_fresh) {
      for (size_t c = 0; c < s->cdesc.size(); ++c) {
        mask[c] = s->pending_draw[c] ? 0 : 1;
        s->pending_draw[c] = 0;
      }
    }
    int rc = enqueue_step(s, a, st, vanilla, compressed_step, need_fresh, mask);
    if (rc < 0) return rc;
  }
  if (compressed_step) s->compressed_launched++;
  s->iter++;
  return PSGD_OK;
}

int psgd_set_graph(psgd_state* s, int32_t enable) {
  if (!s) return fail(PSGD_EINVAL, "state is NULL");
  s->graph_mode = enable ? 1 : 0;
  if (!enable) drop_graph(s);
  return PSGD_OK;
}

int psgd_graph_stats(const psgd_state* s, int64_t* captures, int64_t* replays) {
  if (!s) return fail(PSGD_EINVAL, "state is NULL");
  if (captures) *captures = s->graph_captures;
  if (replays) *replays = s->graph_replays;
  return PSGD_OK;
}

namespace {
// Allocates the two staging sets, the copy streams and their events.
int host_staging_init(psgd_state* s) {
  const size_t gsz = s->dtype == PSGD_F32 ? 4 : 2;
  for (int k = 0; k < 2; ++k) {
    s->stage_grads[k].assign(s->W, nullptr);
    for (int w = 0; w < s->W; ++w)
      if (cudaMalloc(&s->stage_grads[k][w], std::max<size_t>(16, s->N * gsz)) != cudaSuccess) goto oom;
    if (cudaMalloc((void**)&s->stage_out[k], std::max<size_t>(16, s->N * 4)) != cudaSuccess) goto oom;
    if (cudaEventCreateWithFlags(&s->ev_in[k], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s->ev_comp[k], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s->ev_free[k], cudaEventDisableTiming) != cudaSuccess)
      goto cuda_err;
  }
  if (cudaStreamCreateWithFlags(&s->s_in, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&s->s_out, cudaStreamNonBlocking) != cudaSuccess)
    goto cuda_err;
  return PSGD_OK;
oom:
  cudaGetLastError();
  return fail(PSGD_ENOMEM, "psgd_step_host: staging buffers");
cuda_err:
  cudaGetLastError();
  return fail(PSGD_ECUDA, "psgd_step_host: streams/events");
}

void host_staging_free(psgd_state* s) {
  for (int k = 0; k < 2; ++k) {
    for (void* p : s->stage_grads[k])
      if (p) cudaFree(p);
    s->stage_grads[k].clear();
    if (s->stage_out[k]) cudaFree(s->stage_out[k]);
    s->stage_out[k] = nullptr;
  }
}
}  // namespace

// Call k uses staging set k % 2.  Uploads run on an internal stream and wait
// only for the download that last used the same set; the step runs on the
// caller's stream after the uploads; the download runs on a second internal
// stream after the step, and the caller's stream waits for it, so host_out
// is valid once the caller's stream is synchronised.  Consecutive calls thus
// overlap the next upload with the current compute and download.
int psgd_step_host(psgd_state* s, const void* const* host_grads, float* host_out, float inv_loss_scale,
                   void* stream) {
  if (!s) return fail(PSGD_EINVAL, "state is NULL");
  if (!host_grads || !host_out) return fail(PSGD_EINVAL, "host_grads/host_out is NULL");
  for (int w = 0; w < s->W; ++w)
    if (!host_grads[w]) return fail(PSGD_EINVAL, "host_grads[w] is NULL");
  DeviceGuard g(s->device);
  const size_t gsz = s->dtype == PSGD_F32 ? 4 : 2;
  if (!s->s_in) {
    int rc = host_staging_init(s);
    if (rc) {
      host_staging_free(s);
      return rc;
    }
  }
  cudaStream_t st = (cudaStream_t)stream;
  const int k = (int)(s->host_calls & 1);
  if (s->set_used[k]) PSGD_CUDA_TRY(cudaStreamWaitEvent(s->s_in, s->ev_free[k], 0));
  for (int w = 0; w < s->W; ++w)
    PSGD_CUDA_TRY(cudaMemcpyAsync(s->stage_grads[k][w], host_grads[w], s->N * gsz, cudaMemcpyHostToDevice, s->s_in));
  PSGD_CUDA_TRY(cudaEventRecord(s->ev_in[k], s->s_in));
  PSGD_CUDA_TRY(cudaStreamWaitEvent(st, s->ev_in[k], 0));
  int rc = psgd_step(s, (const void* const*)s->stage_grads[k].data(), s->stage_out[k], inv_loss_scale, stream);
  if (rc) return rc;
  PSGD_CUDA_TRY(cudaEventRecord(s->ev_comp[k], st));
  PSGD_CUDA_TRY(cudaStreamWaitEvent(s->s_out, s->ev_comp[k], 0));
  PSGD_CUDA_TRY(cudaMemcpyAsync(host_out, s->stage_out[k], s->N * 4, cudaMemcpyDeviceToHost, s->s_out));
  PSGD_CUDA_TRY(cudaEventRecord(s->ev_free[k], s->s_out));
  PSGD_CUDA_TRY(cudaStreamWaitEvent(st, s->ev_free[k], 0));
  s->set_used[k] = 1;
  s->host_calls++;
  return PSGD_OK;
}

// ---------------------------------------------------------------------------
// Data-parallel split: one replica per process, the caller's collective sums
// the two exchange buffers between the three stages ("PowerSGD Hooks",
// powerSGD_hook steps 2, 3.3 and 3.6).
// ---------------------------------------------------------------------------
int psgd_dp_create(const int64_t* dims, const int32_t* ndims, int32_t n_tensors, int32_t world_size,
                   int32_t rank, int64_t start_iter, double mcr, int32_t use_error_feedback,
                   int32_t warm_start, float eps, uint64_t random_seed, int32_t batch,
                   psgd_dtype grad_dtype, int32_t device, psgd_state** out) {
  if (!out) return fail(PSGD_EINVAL, "out is NULL");
  *out = nullptr;
  if (world_size < 1 || world_size > PSGD_MAX_WORLD) return fail(PSGD_EINVAL, "world_size must be in [1, 64]");
  if (start_iter < 0) return fail(PSGD_EINVAL, "start_powerSGD_iter < 0");
  if (!(eps >= 0.f)) return fail(PSGD_EINVAL, "orthogonalization_epsilon must be >= 0");
  if (grad_dtype != PSGD_F32 && grad_dtype != PSGD_F16 && grad_dtype != PSGD_BF16)
    return fail(PSGD_EINVAL, "grad_dtype");
  psgd_state* s = new psgd_state();
  int rc = plan_tensors(dims, ndims, n_tensors, rank, mcr, &s->tensors);
  if (rc) {
    delete s;
    return rc;
  }
  for (auto& h : s->tensors) s->N += h.numel;
  s->dp_world = world_size;
  // the kernels see one replica (this process's); the W processes' means are
  // formed from the exchanged sums
  return create_common(s, 1, rank, start_iter, mcr, use_error_feedback, warm_start, eps, random_seed, batch,
                       grad_dtype, device, out);
}

namespace {
int dp_check(psgd_state* s, int stage, const char* who) {
  if (!s) return fail(PSGD_EINVAL, std::string(who) + ": state is NULL");
  if (!s->dp_world) return fail(PSGD_EINVAL, std::string(who) + ": not a data-parallel state (psgd_dp_create)");
  if (s->dp_stage != stage)
    return fail(PSGD_EINVAL, std::string(who) + ": called out of order (begin, project, finish, step after step)");
  return PSGD_OK;
}

StepArgs dp_args(psgd_state* s) {
  StepArgs a = make_args(s);
  a.grads.p[0] = s->dp_grad;
  a.out = s->dp_out;
  a.scale = s->dp_scale;
  a.vec_ok = ((uintptr_t)s->dp_out % 16 == 0) &&
             ((uintptr_t)s->dp_grad % (s->dtype == PSGD_F32 ? 16 : 8) == 0);
  return a;
}

int dp_grid(psgd_state* s, long long work) {
  return (int)std::max(1LL, std::min<long long>((work + kThreads - 1) / kThreads, (long long)s->sms * 4));
}
}  // namespace

int psgd_dp_begin(psgd_state* s, const void* grad, float* out, float inv_loss_scale, void* stream, float** exchange,
                  int64_t* count) {
  int rc = dp_check(s, 0, "psgd_dp_begin");
  if (rc) return rc;
  if (!grad || !out || !exchange || !count) return fail(PSGD_EINVAL, "psgd_dp_begin: NULL pointer");
  const size_t gsz = s->dtype == PSGD_F32 ? 4 : 2;
  if (ranges_overlap(grad, s->N * gsz, out, s->N * 4) && !(grad == (const void*)out && s->dtype == PSGD_F32))
    return fail(PSGD_EINVAL, "psgd_dp_begin: out overlaps grad (only out == grad for F32 is allowed)");
  DeviceGuard g(s->device);
  cudaStream_t st = (cudaStream_t)stream;
  s->dp_grad = grad;
  s->dp_out = out;
  s->dp_scale = inv_loss_scale;
  s->dp_vanilla = s->iter < s->start_iter;
  s->dp_compressed = !s->dp_vanilla && !s->cdesc.empty();
  const bool need_fresh = s->dp_compressed && ((!s->warm) || s->compressed_launched == 0);
  std::vector<int> mask(s->cdesc.size(), 0);
  if (need_fresh) {
    for (size_t c = 0; c < s->cdesc.size(); ++c) {
      mask[c] = s->pending_draw[c] ? 0 : 1;
      s->pending_draw[c] = 0;
    }
  }
  StepArgs a = dp_args(s);
  Launcher L{s, st};
  PSGD_CUDA_TRY(cudaMemsetAsync(&s->ctrl->flag, 0, 2 * sizeof(int), st));   // flag, timeout
  if (s->dp_vanilla) {
    // before start_powerSGD_iter the hook allreduces the whole bucket: the
    // exchange buffer is `out`, holding this replica's unscaled gradient
    L.begin(K_DP);
    launch_dp_pack(a, s->d_all, s->d_all_pos, (int)s->all_segs.size(), out, nullptr, dp_grid(s, s->N), st);
    L.end();
    *exchange = out;
    *count = s->N;
  } else {
    PSGD_CUDA_TRY(cudaMemsetAsync(s->xp + s->xp_count - 1, 0, sizeof(float), st));
    if (s->dp_compressed) by_rp<RunDpBegin>(s->RP, s, a, L, need_fresh, mask);
    L.begin(K_DP);
    launch_dp_pack(a, s->d_unc, s->d_unc_pos, (int)s->unc_segs.size(), s->xp + s->xp_unc,
                   s->xp + s->xp_count - 1, dp_grid(s, s->Nunc), st);
    L.end();
    *exchange = s->xp;
    *count = s->xp_count;
  }
  PSGD_CUDA_TRY(cudaGetLastError());
  if (s->dp_compressed) s->compressed_launched++;
  s->dp_stage = 1;
  return PSGD_OK;
}

int psgd_dp_project(psgd_state* s, void* stream, float** exchange, int64_t* count) {
  int rc = dp_check(s, 1, "psgd_dp_project");
  if (rc) return rc;
  if (!exchange || !count) return fail(PSGD_EINVAL, "psgd_dp_project: NULL pointer");
  DeviceGuard g(s->device);
  cudaStream_t st = (cudaStream_t)stream;
  *exchange = nullptr;
  *count = 0;
  if (!s->dp_vanilla) {
    StepArgs a = dp_args(s);
    a.qx = s->xq;
    Launcher L{s, st};
    L.begin(K_DP);
    launch_dp_open(a, s->xp, s->p_total, s->xp + s->xp_count - 1, 1.f / (float)s->dp_world,
                   dp_grid(s, s->p_total), st);
    L.end();
    if (s->dp_compressed) {
      by_rp<RunDpProject>(s->RP, s, a, L);
      *exchange = s->xq;
      *count = s->q_total;
    }
    PSGD_CUDA_TRY(cudaGetLastError());
  }
  s->dp_stage = 2;
  return PSGD_OK;
}

int psgd_dp_finish(psgd_state* s, void* stream) {
  int rc = dp_check(s, 2, "psgd_dp_finish");
  if (rc) return rc;
  DeviceGuard g(s->device);
  cudaStream_t st = (cudaStream_t)stream;
  StepArgs a = dp_args(s);
  Launcher L{s, st};
  const float invW = 1.f / (float)s->dp_world;
  L.begin(K_DP);
  if (s->dp_vanilla) {
    launch_dp_close(a, nullptr, s->d_all, s->d_all_pos, (int)s->all_segs.size(), s->dp_out, invW, 1,
                    dp_grid(s, s->N), st);
  } else {
    launch_dp_close(a, s->dp_compressed ? s->xq : nullptr, s->d_unc, s->d_unc_pos, (int)s->unc_segs.size(),
                    s->xp + s->xp_unc, invW, 0, dp_grid(s, std::max(s->q_total, s->Nunc)), st);
  }
  L.end();
  if (s->dp_compressed) by_rp<RunDpFinish>(s->RP, s, a, L);
  L.begin(K_COMMIT);
  launch_commit(s->ctrl, s->dp_compressed ? 1 : 0, s->d_status, st);
  L.end();
  PSGD_CUDA_TRY(cudaGetLastError());
  PSGD_CUDA_TRY(cudaMemcpyAsync(s->h_status, s->d_status, sizeof(int), cudaMemcpyDeviceToHost, st));
  s->iter++;
  s->dp_stage = 0;
  return PSGD_OK;
}

// Bucket groups (psgd_group.cu): the first compressed-tensor number of a
// bucket in the group's numbering, and the bucket's count of compressed tensors.
int psgd_internal_set_tensor_base(psgd_state* s, int32_t base) {
  if (!s || base < 0) return fail(PSGD_EINVAL, "tensor base");
  s->tensor_base = base;
  return PSGD_OK;
}

int psgd_internal_compressed_count(const psgd_state* s) { return s ? (int)s->cdesc.size() : 0; }

// Tests of the bounded waits: the next cooperative Gram-Schmidt launch's first
// grid barrier waits for one arrival more than the launch has CTAs (a count
// nothing completes), so every CTA gives up after its bounded polls and the
// step reports PSGD_ETIMEOUT.  Only states on the cooperative stage (small
// buckets, ranks up to 16) have that launch; returns PSGD_EINVAL otherwise.
int psgd_internal_force_wait_timeout(psgd_state* s) {
  if (!s) return fail(PSGD_EINVAL, "state is NULL");
  if (!s->gs_fused || !s->gs_coop) return fail(PSGD_EINVAL, "the state has no cooperative stage");
  s->test_wait_skew = 1;
  return PSGD_OK;
}

int psgd_step_status(psgd_state* s, void* stream) {
  if (!s) return fail(PSGD_EINVAL, "state is NULL");
  DeviceGuard g(s->device);
  PSGD_CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
  if (*s->h_status == 2) {
    if (s->img) {
      // a kernel may have written the operand images of factors that were not
      // committed: rebuild them from the committed half before the next step
      StepArgs a = make_args(s);
      Launcher L{s, (cudaStream_t)stream};
      by_rp<RunImages>(s->RP, s, a, L, 3);
      PSGD_CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
    }
    return fail(PSGD_ETIMEOUT, "a bounded device-side wait gave up; the step was not committed");
  }
  return *s->h_status ? PSGD_SKIPPED_NONFINITE : PSGD_OK;
}

int psgd_get_stats(const psgd_state* s, int64_t* before, int64_t* after, int64_t* iter) {
  if (!s) return fail(PSGD_EINVAL, "state is NULL");
  long long b = s->N, a = 0;
  for (auto& h : s->tensors) a += h.compressed ? (h.rows + h.cols) * h.rank : h.numel;
  if (before) *before = b;
  if (after) *after = a;
  if (iter) *iter = s->iter;
  return PSGD_OK;
}

int psgd_tensor_info(const psgd_state* s, int32_t t, int32_t* compressed, int64_t* rows, int64_t* cols,
                     int32_t* rank, int64_t* bucket_offset, int64_t* packed_offset) {
  if (!s) return fail(PSGD_EINVAL, "state is NULL");
  if (t < 0 || t >= (int)s->tensors.size()) return fail(PSGD_EINVAL, "tensor index out of range");
  const HostTensor& h = s->tensors[t];
  if (compressed) *compressed = h.compressed;
  if (rows) *rows = h.rows;
  if (cols) *cols = h.cols;
  if (rank) *rank = h.rank;
  if (bucket_offset) *bucket_offset = h.offset;
  if (packed_offset) *packed_offset = h.compressed ? h.e_off : -1;
  return PSGD_OK;
}

int64_t psgd_error_numel(const psgd_state* s) { return s ? s->Ne : 0; }

namespace {
int read_cur(psgd_state* s, int* cur) {
  Ctrl c;
  PSGD_CUDA_TRY(cudaMemcpy(&c, s->ctrl, sizeof(Ctrl), cudaMemcpyDeviceToHost));
  *cur = c.cur;
  return PSGD_OK;
}
int check_compressed(psgd_state* s, int t, HostTensor** h) {
  if (!s) return fail(PSGD_EINVAL, "state is NULL");
  if (t < 0 || t >= (int)s->tensors.size()) return fail(PSGD_EINVAL, "tensor index out of range");
  *h = &s->tensors[t];
  if (!(*h)->compressed) return fail(PSGD_EINVAL, "tensor is not compressed");
  return PSGD_OK;
}
}  // namespace

int psgd_set_q(psgd_state* s, int32_t t, const float* host_in, int32_t is_draw) {
  HostTensor* h;
  int rc = check_compressed(s, t, &h);
  if (rc) return rc;
  if (!host_in) return fail(PSGD_EINVAL, "host_in is NULL");
  DeviceGuard g(s->device);
  PSGD_CUDA_TRY(cudaDeviceSynchronize());
  const TensorDesc& td = s->cdesc[h->cidx];
  // k-major device layout: element (j, k) at k * cols + j
  std::vector<float> buf((size_t)td.m * s->RP, 0.f);
  for (long long j = 0; j < td.m; ++j)
    for (int k = 0; k < td.r; ++k) buf[(size_t)k * td.m + j] = host_in[j * td.r + k];
  if (is_draw) {
    PSGD_CUDA_TRY(cudaMemcpy(s->qdraw + td.q_off, buf.data(), buf.size() * 4, cudaMemcpyHostToDevice));
    s->pending_draw[h->cidx] = 1;
    return PSGD_OK;
  }
  // Warm Q: fold the current factors into the error store (the residual stays
  // the same), zero the committed P so the factors no longer correct anything,
  // then install Q as the projection of the next step.
  int cur = 0;
  rc = read_cur(s, &cur);
  if (rc) return rc;
  StepArgs a = make_args(s);
  if (s->ef) {
    for (int w = 0; w < s->W; ++w) {
      a.replica = w;
      by_rp<RunErrView>(s->RP, s, a, 3, (cudaStream_t)0);
    }
    PSGD_CUDA_TRY(cudaGetLastError());
  }
  PSGD_CUDA_TRY(cudaMemset(s->Pf + (size_t)cur * s->p_total, 0, (size_t)s->p_total * 4));
  PSGD_CUDA_TRY(cudaMemcpy(s->Qf + (size_t)cur * s->q_total + td.q_off, buf.data(), buf.size() * 4,
                           cudaMemcpyHostToDevice));
  if (s->img) {
    // the tensor-core pass 1 reads the committed factors through their images
    Launcher L{s, (cudaStream_t)0};
    by_rp<RunImages>(s->RP, s, a, L, 3);
    PSGD_CUDA_TRY(cudaGetLastError());
  }
  int one = 1;
  PSGD_CUDA_TRY(cudaMemcpy(&s->ctrl->warm_valid, &one, sizeof(int), cudaMemcpyHostToDevice));
  if (s->compressed_launched == 0) s->compressed_launched = 1;
  PSGD_CUDA_TRY(cudaDeviceSynchronize());
  return PSGD_OK;
}

static int get_factor(psgd_state* s, int t, float* host_out, bool is_q) {
  HostTensor* h;
  int rc = check_compressed(s, t, &h);
  if (rc) return rc;
  if (!host_out) return fail(PSGD_EINVAL, "host_out is NULL");
  DeviceGuard g(s->device);
  PSGD_CUDA_TRY(cudaDeviceSynchronize());
  int cur = 0;
  rc = read_cur(s, &cur);
  if (rc) return rc;
  const TensorDesc& td = s->cdesc[h->cidx];
  const long long rows = is_q ? td.m : td.n;
  std::vector<float> buf((size_t)rows * s->RP);
  const float* src = is_q ? s->Qf + (size_t)cur * s->q_total + td.q_off : s->Pf + (size_t)cur * s->p_total + td.p_off;
  PSGD_CUDA_TRY(cudaMemcpy(buf.data(), src, buf.size() * 4, cudaMemcpyDeviceToHost));
  for (long long j = 0; j < rows; ++j)
    for (int k = 0; k < td.r; ++k)
      host_out[j * td.r + k] = is_q ? buf[(size_t)k * rows + j] : buf[j * s->RP + k];
  return PSGD_OK;
}

int psgd_get_q(psgd_state* s, int32_t t, float* host_out) { return get_factor(s, t, host_out, true); }
int psgd_get_p(psgd_state* s, int32_t t, float* host_out) { return get_factor(s, t, host_out, false); }

static int err_view(psgd_state* s, int32_t replica, float* ptr, void* stream, int mode) {
  if (!s) return fail(PSGD_EINVAL, "state is NULL");
  if (!s->ef) return fail(PSGD_EINVAL, "error feedback is off");
  if (replica < 0 || replica >= s->W) return fail(PSGD_EINVAL, "replica out of range");
  if (!ptr) return fail(PSGD_EINVAL, "buffer is NULL");
  if (s->cdesc.empty()) return PSGD_OK;
  DeviceGuard g(s->device);
  StepArgs a = make_args(s);
  a.replica = replica;
  a.eio = ptr;
  by_rp<RunErrView>(s->RP, s, a, mode, (cudaStream_t)stream);
  PSGD_CUDA_TRY(cudaGetLastError());
  return PSGD_OK;
}

int psgd_get_error(psgd_state* s, int32_t replica, float* dev_out, void* stream) {
  return err_view(s, replica, dev_out, stream, 1);
}
int psgd_set_error(psgd_state* s, int32_t replica, const float* dev_in, void* stream) {
  return err_view(s, replica, (float*)dev_in, stream, 2);
}

size_t psgd_workspace_bytes(const psgd_state* s) { return s ? s->bytes : 0; }

int psgd_set_error_store_halves(psgd_state* s, int32_t halves) {
  if (!s) return fail(PSGD_EINVAL, "state is NULL");
  if (halves != 1 && halves != 2) return fail(PSGD_EINVAL, "halves must be 1 or 2");
  if (s->dp_world) return fail(PSGD_EINVAL, "a data-parallel state keeps two halves");
  if (s->iter != 0) return fail(PSGD_EINVAL, "the error store's halves are set before the first step");
  if (halves == s->est_halves || !s->ef || !s->estore) {
    if (s->ef && s->estore) s->est_halves = halves;
    return PSGD_OK;
  }
  DeviceGuard g(s->device);
  PSGD_CUDA_TRY(cudaDeviceSynchronize());
  const size_t half = (size_t)s->W * s->Nc_pad * sizeof(float);
  float* fresh = nullptr;
  int rc = dalloc(s, (void**)&fresh, (size_t)halves * half);
  if (rc) return rc;
  PSGD_CUDA_TRY(cudaMemset(fresh, 0, (size_t)halves * half));
  // the old store leaves the allocation list and the byte count
  for (size_t i = 0; i < s->allocs.size(); ++i)
    if (s->allocs[i] == (void*)s->estore) {
      cudaFree(s->allocs[i]);
      s->allocs.erase(s->allocs.begin() + (long)i);
      s->bytes -= (size_t)s->est_halves * half;
      break;
    }
  s->estore = fresh;
  s->est_halves = halves;
  drop_graph(s);
  return PSGD_OK;
}

int psgd_profile(psgd_state* s, int32_t enable) {
  if (!s) return fail(PSGD_EINVAL, "state is NULL");
  s->prof = enable != 0;
  s->prof_mask = 0xffffffffu;
  return PSGD_OK;
}

int psgd_profile_select(psgd_state* s, uint32_t kind_mask) {
  if (!s) return fail(PSGD_EINVAL, "state is NULL");
  s->prof = kind_mask != 0;
  s->prof_mask = kind_mask;
  return PSGD_OK;
}

int32_t psgd_profile_kinds(void) { return K_COUNT; }

int psgd_profile_read(psgd_state* s, int32_t kind, const char** name, int64_t* launches, double* total_ms,
                      double* bytes_per_launch) {
  if (!s) return fail(PSGD_EINVAL, "state is NULL");
  if (kind < 0 || kind >= K_COUNT) return fail(PSGD_EINVAL, "kind out of range");
  if (!launches && !total_ms) {   // the name and bytes only; the record stays
    if (name) *name = kKindNames[kind];
    if (bytes_per_launch) *bytes_per_launch = s->kind_bytes[kind];
    return PSGD_OK;
  }
  DeviceGuard g(s->device);
  PSGD_CUDA_TRY(cudaDeviceSynchronize());
  double ms = 0.0;
  for (auto& e : s->ev[kind]) {
    float x = 0.f;
    cudaEventElapsedTime(&x, e.a, e.b);
    ms += x;
    s->ev_pool.push_back(e);
  }
  if (name) *name = kKindNames[kind];
  if (launches) *launches = (int64_t)s->ev[kind].size();
  if (total_ms) *total_ms = ms;
  if (bytes_per_launch) *bytes_per_launch = s->kind_bytes[kind];
  s->ev[kind].clear();
  return PSGD_OK;
}

}  // extern "C"
