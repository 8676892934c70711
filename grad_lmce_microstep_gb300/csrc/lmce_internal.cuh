// Internal declarations shared by the lmce translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <vector>

namespace lmce {

// Kernel kinds for the timing records (same values as LMCE_KIND_* in lmce.h).
enum Kind { K_LSE = 0, K_FINISH = 1, K_DW = 2, K_DH = 3, K_LSE_DH = 4, K_LN = 5, K_COMPACT = 6, K_COUNT = 7 };

// Optional CUDA-event records around every kernel launch.
struct Prof {
  bool on = false;
  std::vector<cudaEvent_t> pool;
  size_t used = 0;
  struct Rec { int kind; cudaEvent_t a, b; };
  std::vector<Rec> recs;
  cudaEvent_t next() {
    if (used == pool.size()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      pool.push_back(e);
    }
    return pool[used++];
  }
};

// Launch context of one micro-step: stream, timing records, launch counter.
struct Launch {
  cudaStream_t st;
  Prof* prof;
  int n = 0;
  cudaEvent_t pending = nullptr;
  int pending_kind = 0;
  void begin(int kind) {
    ++n;
    if (prof && prof->on) {
      pending = prof->next();
      pending_kind = kind;
      if (pending) cudaEventRecord(pending, st);
    }
  }
  void end() {
    if (prof && prof->on && pending) {
      cudaEvent_t b = prof->next();
      if (b) {
        cudaEventRecord(b, st);
        prof->recs.push_back({pending_kind, pending, b});
      }
      pending = nullptr;
    }
  }
};

// Step accumulators kept on the device between micro-steps of one optimizer step.
struct DevAcc {
  double loss_sum;    // sum of valid row losses over the step
  double objective;   // sum_k s_k * loss_sum_k
  long long count;    // valid targets over the step
  unsigned int err;   // ERR_BIT_* flags
  unsigned int micro; // micro-steps that ran
  float scale;        // s of the micro-step being processed (read by the gradient kernels)
  float pad_;
  double scale64;     // the same s in double precision (weights the objective)
};

constexpr unsigned ERR_BIT_BAD_TARGET = 1u;
constexpr unsigned ERR_BIT_NONFINITE = 2u;
// A bounded device wait ran out (tensor-core path); bits 8..15 say which wait.
constexpr unsigned ERR_BIT_TIMEOUT = 4u;
constexpr unsigned ERR_BIT_COUNT = 8u;      // a compacted micro-step's valid count was not the caller's
// A bounds check of the debug build failed (bits 16..23 say which site); the access was skipped.
constexpr unsigned ERR_BIT_BOUNDS = 16u;

// Bounds checks of the debug build (LMCE_DEBUG_BOUNDS=1, built as liblmce_dbg.so): a check that
// fails records ERR_BIT_BOUNDS and its site in the step's error word, and the caller skips the
// access; lmce_finalize then returns LMCE_ERR_INTERNAL.  Nothing traps.  In the release build a
// check always passes and compiles to nothing.
#ifndef LMCE_DEBUG_BOUNDS
#define LMCE_DEBUG_BOUNDS 0
#endif
enum BoundsSite : unsigned {
  BS_TMA_ROW = 1,       // gradient kernels: a TMA box's row coordinate past its tensor
  BS_HIT = 2,           // dW pass: one-hot hits of a block past the list
  BS_SLOT = 3,          // gradient kernels / split combine: a partial slot past the pairs' slots
  BS_TILE_FLAG = 4,     // lse+dh pass / row post: a 128-token tile index past the flags
  BS_W_ROW = 5,         // dh passes: a one-hot row of W past V
  BS_COMPACT_POS = 6,   // compaction / fused ln_f forward: a compact position past the buffer
  BS_SCATTER_POS = 7,   // scatter / fused ln_f backward: a compact position past the valid rows
};
__device__ __forceinline__ bool dcheck(bool ok, unsigned* err, unsigned site) {
#if LMCE_DEBUG_BOUNDS
  if (!ok) atomicOr(err, ERR_BIT_BOUNDS | (site << 16));
  return ok;
#else
  (void)ok;
  (void)err;
  (void)site;
  return true;
#endif
}

// Arguments of one micro-step as the kernels see them.
struct StepArgs {
  const void* hidden;     // [N, C] dtype
  const void* W;          // [V, C] dtype
  const int32_t* targets; // [N]
  void* dh;               // [N, C] dtype
  float* dW;              // [V, C] fp32
  float* row_loss;        // [N] or nullptr
  int64_t N, C, V;
  int32_t ignore_id;
  int32_t norm;           // 0 global, 1 micro mean
  int32_t G;
  int64_t global_valid;
  int32_t beta;           // 0: dW = grad, 1: dW += grad
  int32_t bf16;           // 1: dtype bf16, 0: fp32
  int32_t tc_two_pass;    // tensor-core path: 1 = separate logsumexp pass, 0 = one-pass lse + dh
  int32_t tc_recompute = 0;  // one-pass tensor-core path: 1 = the dW pass recomputes the logits
                             // (0: it reads the stored exponentials when the scratch has them)
  int64_t test_stall_ns = 0;  // failure-detection test: > 0 makes the tensor-core gradient launches
                              // start no operand load and bounds their waits by this many ns
};

// Library-owned device scratch.
struct Scratch {
  float* lse;          // [max_N] per-row logsumexp
  double* part_loss;   // [max_parts] per-block loss partials
  int* part_cnt;       // [max_parts] per-block valid counts
  unsigned* part_err;  // [max_parts] per-block error flags
  DevAcc* acc;         // step accumulators
  int64_t max_parts;
  // tensor-core path only
  float* tc_part_m;    // [TC_MAX_SPLIT][max_N] per-slice base-2 row max
  float* tc_part_l;    // [TC_MAX_SPLIT][max_N] per-slice sum of 2^(x - max)
  float* tc_zt;        // [max_N] target logit
  float* tc_part;      // gradient passes: fp32 partial sums of split tiles, [2 * pairs][128][C]
  float* tc_part_lm;   // logsumexp + dh pass: per-slot (base-2 max, sum) of split tiles, [2 * pairs][2][128]
  unsigned* tc_tile_flag;  // logsumexp + dh pass: per 128-token tile, 1 = recompute exactly
  unsigned* ticket;    // [2] blocks finished, 0 between uses: [0] the row passes that reduce their
                       // own partials, [1] the squared dW norm
  // tensor-core path, exact repair of flagged tiles
  float* rep_part;     // [simt_repair_part_floats(C)] per-slice (max, sum) and dh partials
  unsigned* rep_ticket;  // [tiles * 8] per row group: slices finished (0 between uses)
  // tensor-core path, dW from the stored exponentials (all null: the dW pass recomputes the
  // logits instead)
  __nv_bfloat16* tc_p;     // [max_N][Vp] the one-pass kernel's bf16 operand p = 2^(z log2 e - m),
                           // Vp = V rounded up to 256; the target entry later becomes p_y - 2^(lse log2 e - m)
  float* tc_mref;          // [TC_MAX_VER][Np] base-2 reference m of each row, per segment of its tile
  __nv_bfloat16* tc_hs;    // [TC_MAX_VER][Np][C] rows of h scaled by s 2^(m - lse log2 e), per segment
  uint8_t* tc_kmap;        // [tiles][Vp / 256] segment of (128-token tile, 256-row vocabulary block)
  int64_t tc_p_rows;       // rows of tc_p (max_N)
};

// Segments of a 128-token tile (pairs of the one-pass kernel's schedule sharing it) the stored-
// exponential path keeps a reference for; a schedule with more falls back to recomputing.
constexpr int TC_MAX_VER = 8;

constexpr int TC_MAX_SPLIT = 32;

// Scratch of the valid-row compaction (allocated when the handle is created with
// LMCE_COMPACT_VALID_ROWS): the compacted rows, their targets, dh and row losses, each row's
// position, and the per-block counts and offsets.
struct CompactScratch {
  void* h_c;           // [max_N, C] dtype
  void* dh_c;          // [max_N, C] dtype
  int32_t* y_c;        // [max_N]
  float* rl_c;         // [max_N]
  int32_t* pos;        // [max_N] position of row n among the valid rows, -1 if ignored
  int* blk_cnt;        // [compact_blocks(max_N)]
  unsigned* blk_err;   // [compact_blocks(max_N)]
  int64_t* blk_off;    // [compact_blocks(max_N)]
  int64_t* total;      // [1] valid rows found
  int64_t* host_total; // pinned [1]
  int64_t rows;        // the compact buffers' rows as the debug checks see them (max_N; lowered
                       // by the debug build's test hook)
  unsigned* err;       // the step's error word (debug bounds checks)
};
int64_t compact_blocks(int64_t N);
// count + scan + gather of a.hidden / a.targets (a.N rows) into the compact buffers; the
// valid total is checked against n_valid (>= 0) and bad targets are flagged in acc->err
cudaError_t compact_rows(const StepArgs& a, const CompactScratch& cs, DevAcc* acc, int64_t n_valid, Launch& L);
// the count and scan alone (block offsets and the valid total, with the same checks)
cudaError_t compact_count_scan(const StepArgs& a, const CompactScratch& cs, DevAcc* acc, int64_t n_valid, Launch& L);
// dh / row_loss of a.N rows from the first n_valid compact rows, zero for the ignored rows
cudaError_t compact_scatter(const StepArgs& a, const CompactScratch& cs, int64_t n_valid, Launch& L);

// ln_f in front of the head (lmce_microstep_ln): forward x -> h with per-row mean / rstd, and
// backward dh -> dx with the dgamma / dbeta partials of ln_blocks(N) row blocks reduced in order.
struct LnArgs {
  const void* x;        // [N, C] dtype
  const float* gamma;   // [C]
  const float* beta;    // [C] or nullptr
  void* h;              // [N, C] dtype (forward output)
  const void* dh;       // [N, C] dtype (backward input)
  void* dx;             // [N, C] dtype
  float* mean;          // [N]
  float* rstd;          // [N]
  float* part_g;        // [ln_part_rows(), C], the first ln_blocks(N) rows used
  float* part_b;        // [ln_part_rows(), C]
  float* dgamma;        // [C]
  float* dbeta;         // [C] or nullptr
  int64_t N, C;
  int32_t rms;          // 1: RMSNorm, 0: LayerNorm
  float eps;
  int32_t bf16;
  int32_t accumulate;   // 1: dgamma / dbeta +=, 0: =
  unsigned* err;        // the step's error word (debug bounds checks)
};
int64_t ln_blocks(int64_t N);           // backward blocks (parameter-gradient partials) for N rows
int64_t ln_rows_per_block(int64_t N);
int64_t ln_part_rows();                 // the most ln_blocks(N) can be, for any N
cudaError_t ln_forward(const LnArgs& a, Launch& L);
cudaError_t ln_backward(const LnArgs& a, Launch& L);
// ln_f fused with the valid-row compaction, for rows that fit the register layout
// (ln_compact_fusable).  a.x, a.dx and a.N are the caller's rows; a.h, a.dh, a.mean and a.rstd
// hold the compact rows.  The forward (after compact_count_scan) normalises the valid rows of x
// straight into the compact head input and records their targets and positions; the backward
// writes dx of every row (zero for the rows without a compact position below n_valid), the row
// losses when row_loss is given, and the parameter gradients.
bool ln_compact_fusable(const LnArgs& a);
cudaError_t ln_gather_forward(const LnArgs& a, const int32_t* targets, int64_t V, const CompactScratch& cs, Launch& L);
cudaError_t ln_backward_scatter(const LnArgs& a, const CompactScratch& cs, int64_t n_valid, float* row_loss, Launch& L);

// Programmatic dependent launch: the kernels of a micro-step are launched so that each may be
// scheduled while the one before it on the stream drains; each kernel launched this way first
// waits (griddep_wait) until the previous grid has completed and its writes are visible, before
// it reads or writes anything.  Outside such a launch the wait returns at once.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// cudaFuncSetAttribute(func, MaxDynamicSharedMemorySize, bytes), made once per kernel and device
// for the largest size asked so far (the host cost of the attribute call is otherwise paid on
// every launch).
cudaError_t max_dyn_smem(const void* func, int bytes);

// Fixed-order reduction of the per-block partials of one micro-step into the step
// accumulators; also computes this micro-step's gradient scale.  One launch.
//   FIN_ALL  : loss, count and error partials (scale from the count)
//   FIN_COUNT: count and error partials only (sets the scale before any gradient kernel)
//   FIN_LOSS : loss and error partials, with the scale FIN_COUNT set
enum FinMode { FIN_ALL = 0, FIN_COUNT = 1, FIN_LOSS = 2 };
cudaError_t launch_finish(const StepArgs& a, const Scratch& s, int64_t nparts, Launch& L, int mode = FIN_ALL);

// The reduction itself, run by one block of FIN_T threads: thread t sums the partials t, t + FIN_T,
// ... in order, then a fixed-shape tree adds the threads; thread 0 updates the accumulators.
// Partials are read past L1 (another block may have just written them).  norm 0 is the global
// normalisation (s = 1 / global_valid), 1 the micro-step mean (s = 1 / (count * G)).
constexpr int FIN_T = 256;
__device__ __forceinline__ void finish_block(const double* part_loss, const int* part_cnt, const unsigned* part_err,
                                             int64_t nparts, int norm, int G, long long global_valid, DevAcc* acc,
                                             int mode) {
  __shared__ double fsl[FIN_T];
  __shared__ long long fsc[FIN_T];
  __shared__ unsigned fse[FIN_T];
  const int t = threadIdx.x;
  double l = 0.0;
  long long c = 0;
  unsigned e = 0;
  for (int64_t i = t; i < nparts; i += FIN_T) {
    if (mode != FIN_COUNT) l += __ldcg(part_loss + i);
    if (mode != FIN_LOSS) c += __ldcg(part_cnt + i);
    e |= __ldcg(part_err + i);
  }
  fsl[t] = l;
  fsc[t] = c;
  fse[t] = e;
  __syncthreads();
  for (int o = FIN_T / 2; o > 0; o >>= 1) {
    if (t < o) {
      fsl[t] += fsl[t + o];
      fsc[t] += fsc[t + o];
      fse[t] |= fse[t + o];
    }
    __syncthreads();
  }
  if (t == 0) {
    const double loss_k = fsl[0];
    const long long cnt_k = fsc[0];
    acc->err |= fse[0];
    if (mode != FIN_LOSS) {
      double s;
      if (norm == 0) s = global_valid > 0 ? 1.0 / (double)global_valid : 0.0;
      else s = cnt_k > 0 ? 1.0 / ((double)cnt_k * (double)G) : 0.0;
      acc->scale = (float)s;
      acc->scale64 = s;
      acc->count += cnt_k;
    }
    if (mode != FIN_COUNT) {
      acc->loss_sum += loss_k;
      acc->objective += acc->scale64 * loss_k;
      if (!isfinite(loss_k)) acc->err |= ERR_BIT_NONFINITE;
      acc->micro += 1;
    }
  }
}

// True in the one block of the grid that finishes last, once every block's earlier global writes
// are visible; the ticket returns to 0 for the next use.  A block-wide call (no thread may skip
// it); it only counts, it never waits on another block.
__device__ __forceinline__ bool last_block(unsigned* ticket) {
  __shared__ int is_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned n = gridDim.x * gridDim.y * gridDim.z;
    const unsigned k = atomicAdd(ticket, 1u);
    is_last = k == n - 1;
    if (is_last) *ticket = 0u;   // every block has counted
  }
  __syncthreads();
  if (is_last) __threadfence();
  return is_last != 0;
}
// Loads the module that holds the reduction kernel (no launch).
cudaError_t finish_load_kernel();

// SIMT path (fp32 FFMA).
int64_t simt_parts(int64_t N);
size_t simt_grad_smem(int64_t C);
cudaError_t simt_microstep(const StepArgs& a, const Scratch& s, Launch& L);
// The two gradient passes alone (lse and the scale already on the device).
cudaError_t simt_grads(const StepArgs& a, const Scratch& s, Launch& L);
// Loads the module of every SIMT kernel for both dtypes (no launch).
cudaError_t simt_load_kernels();
// Exact logsumexp and dh of the rows of the 128-token tiles whose flag is set: the repair of the
// one-pass logsumexp + dh kernel.  Two persistent launches whose blocks find the flagged tiles
// themselves and return at once when there is none; the work of the flagged tiles' rows is split
// over every SM by vocabulary slice and merged in slice order.
constexpr int TC_TILE_ROWS = 128;
cudaError_t simt_repair_lse(const StepArgs& a, const Scratch& s, Launch& L);
// store_p: also rewrite the flagged tiles' rows of the stored exponentials (normalised p, and
// the reference m = lse log2 e of every segment)
cudaError_t simt_repair_dh(const StepArgs& a, const Scratch& s, Launch& L, bool store_p = false);
size_t simt_repair_part_floats(int64_t C);

// Tensor-core path (tcgen05 + TMA).
bool tc_supported(int64_t C, int64_t V, int bf16);
int64_t tc_parts(int64_t N);
int64_t tc_pairs();
size_t tc_part_bytes(int64_t C);
size_t tc_part_lm_bytes();
cudaError_t tc_microstep(const StepArgs& a, const Scratch& s, Launch& L);
// Stored-exponential dW pass: columns of the stored operand (V rounded up to 256) and rows per
// reference segment (N rounded up to 256).
int64_t tc_p_cols(int64_t V);
int64_t tc_ver_rows(int64_t N);

}  // namespace lmce
