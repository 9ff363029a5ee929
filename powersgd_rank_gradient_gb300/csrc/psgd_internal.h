// Internal layout shared by the host planner (psgd_api.cu) and the kernels.
//
// HBM layout of a state (all offsets in elements):
//   error store  : 2 (current/next) x W x Nc_pad floats.  Replica w's store for
//                  tensor t starts at c_off[t] (aligned to 32 elements).  It
//                  holds M_w of the last committed step; the residual is kept
//                  in factored form, e_w = store_w - P Q^T, with (P, Q) the
//                  factors of that step (see Pf/Qf).
//   Pf[2], Qf[2] : the committed factors, rank padded to RP = next power of
//                  two (unused columns 0): P row-major (rows x RP), Q k-major
//                  (element (j, k) at k * cols + j, so a warp reading 4
//                  consecutive columns per lane makes one coalesced access).
//                  Qf[cur] is also the warm-start projection of the next step.
//   praw_part    : pass-1 partial P = Mbar Q, one slice per column tile.
//   qpart        : pass-2 partial Q = Mbar^T P, one k-major slice per row block.
//   mbar         : optional scratch holding the replica mean of M (W >= 3).
//   img          : ranks 16 and 32 only: P and Q split into tf32 hi and lo
//                  parts in the swizzled layout the tensor-core passes read
//                  (see psgd_tc.cuh).
//   ctrl         : device integers: cur, warm_valid, nonfinite flag, timeout.
#pragma once

#include <stdint.h>

namespace psgd {

constexpr int kThreads = 256;      // threads per CTA of the streaming passes
constexpr int kRowBlock = 512;     // rows per work item of pass 2 (one Q partial each)
constexpr int kFineRows = 128;     // rows per work item of pass 1 (ranks <= 8; fewer in small buckets)
constexpr int kRows1High = 128;   // rows per work item of pass 1 (ranks 16 and 32)
constexpr int kFineRows3 = 32;     // rows per work item of pass 3 and the error views
constexpr int kGsRows = 256;       // rows per work item of the Gram-Schmidt kernels
constexpr int kQrChunk = kThreads;  // values per work item of the Q reduction (64 groups of four)

// Columns per thread (CPT) and column-tile width of the streaming passes for
// a padded rank RP: the per-thread accumulators hold CPT x RP floats.
__host__ __device__ constexpr int cpt_for(int rp) { return rp <= 8 ? 4 : (rp == 16 ? 2 : 1); }
__host__ __device__ constexpr int ctile_for(int rp) { return kThreads * cpt_for(rp); }
// Pass 3 (and the error views) keeps CPT3 columns of Q in registers per
// thread: more columns than pass 2 at ranks 16 and 32 give its dot-product
// chains more independent work per staged P value.
__host__ __device__ constexpr int cpt3_for(int rp) { return rp <= 16 ? 4 : 2; }
__host__ __device__ constexpr int ctile3_for(int rp) { return kThreads * cpt3_for(rp); }
// Column tile of pass 1: 1024 columns (eight 128-column chunks, one per warp)
// for ranks up to 8; 512 columns (sixteen 32-column chunks) for ranks 16 and
// 32, whose items are 128 rows tall.
__host__ __device__ constexpr int ctile1_for(int rp) { return rp <= 8 ? 1024 : 512; }
__host__ __device__ constexpr int rows1_for(int rp) { return rp <= 8 ? kFineRows : kRows1High; }

struct TensorDesc {
  long long g_off;   // first element in the bucket
  long long c_off;   // first element in the packed error store / mbar
  long long p_off;   // first element of the tensor's P (rows x RP)
  long long q_off;   // first element of the tensor's Q (RP x cols, k-major; 32-aligned)
  long long pp_off;  // first element of praw_part (ctiles1 x rows x RP)
  long long qp_off;  // first element of qpart (rblocks x RP x cols; 32-aligned)
  long long e_off;   // first element in the user-visible packed error (no padding)
  long long valid;   // elements of the view backed by the bucket (n * m, or the bucket
                     // length for the batched hook's zero-padded square)
  // ranks 16 and 32: first floats of the tensor-core operand images (hi half;
  // the lo half follows it): P's and Q's row images (rows padded to 128) and
  // chunk images (one RP x 32 block per 32 rows)
  long long pi_off, qi_off, pti_off, qti_off;
  int n, m, r;       // rows, cols, effective rank
  int ld;            // row stride in the error store and mbar: m rounded up to a
                     // multiple of 4, so their rows are 16-byte aligned; the
                     // padding columns stay zero
  int ctiles;        // column tiles of passes 2 and 3
  int ctiles1;       // column tiles of pass 1 (praw_part slices)
  int rblocks;       // row blocks
  int vec;           // rows are 16-byte aligned in the bucket (m % 4 == 0, g_off % 4 == 0)
};

// One work item of the streaming passes: a (row block) x (column tile) tile.
struct Item {
  int t;
  int row0, nrows;
  int col0, ncols;
  int rb;   // row-block index within the tensor
  int ct;   // column-tile index within the tensor
  int pad;
};

// Row ranges of the small Gram-Schmidt kernels, over P (rows = n) or over Q
// (rows = m).
struct GsItem {
  int t;
  int row0, nrows;
  int pad;
};

// An uncompressed range of the bucket, split into pieces of <= 64K elements.
struct Segment {
  long long off;
  int len;
  int pad;
};

struct Ctrl {
  int cur;        // which half of the double-buffered state is current
  int warm_valid; // a committed compressed step exists (warm Q available)
  int flag;       // non-finite input seen in this step
  int timeout;    // a bounded device-side wait gave up in this step
};

constexpr int kMaxWorld = 64;

struct GradPtrs {
  const void* p[kMaxWorld];
};

}  // namespace psgd
