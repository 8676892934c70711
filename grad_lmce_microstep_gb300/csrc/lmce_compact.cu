// Valid-row compaction around a micro-step: the rows whose target is ignored contribute nothing
// to the loss, dh or dW, so both heavy passes can run over the valid rows alone.  zerotofrontier
// "GPT", section "Document boundaries, packing and masking", masks pad targets out of the loss;
// a micro-batch with long masked spans then costs work in proportion to its valid rows only.
//
//   count  : per block of CP_ROWS rows, the valid targets (0 <= y < V) and a bad-target bit
//   scan   : one block: exclusive prefix of the block counts in block order, the total checked
//            against the caller's count, the error bits folded into the step accumulators
//   gather : each valid row goes to position (block offset + rank within the block), the input
//            order kept: h_c[pos] = h[n], y_c[pos] = y[n], pos[n] = pos (-1 for an ignored row)
//   scatter: dh[n] = dh_c[pos[n]] and row_loss[n] = rl_c[pos[n]], zero for an ignored row
#include "lmce_internal.cuh"

namespace lmce {
namespace {

constexpr int CP_ROWS = 128;   // rows per block of count and gather: one per thread
constexpr int SCAN_T = 1024;

__device__ __forceinline__ bool valid_target(int y, int64_t V) { return y >= 0 && (int64_t)y < V; }

__global__ void __launch_bounds__(CP_ROWS) compact_count_kernel(const int32_t* __restrict__ y, int64_t N,
                                                               int64_t V, int32_t ignore_id,
                                                               int* __restrict__ blk_cnt,
                                                               unsigned* __restrict__ blk_err) {
  const int64_t n = (int64_t)blockIdx.x * CP_ROWS + threadIdx.x;
  int v = 0;
  unsigned e = 0;
  if (n < N) {
    const int t = y[n];
    v = valid_target(t, V);
    if (!v && t != ignore_id) e = ERR_BIT_BAD_TARGET;
  }
  const int c = __syncthreads_count(v);
  const int b = __syncthreads_or(e);
  if (threadIdx.x == 0) {
    blk_cnt[blockIdx.x] = c;
    blk_err[blockIdx.x] = (unsigned)b;
  }
}

// One block.  Chunks of SCAN_T block counts: a warp-shuffle inclusive scan per warp, the warp
// totals scanned by warp 0, and the running offset carried across chunks.
__global__ void __launch_bounds__(SCAN_T) compact_scan_kernel(const int* __restrict__ blk_cnt,
                                                             const unsigned* __restrict__ blk_err,
                                                             int64_t nblk, int64_t* __restrict__ blk_off,
                                                             int64_t* __restrict__ total, int64_t n_valid,
                                                             DevAcc* acc) {
  __shared__ long long wsum[SCAN_T / 32];
  __shared__ long long carry;
  __shared__ unsigned err_all;
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  if (t == 0) {
    carry = 0;
    err_all = 0;
  }
  __syncthreads();
  unsigned e = 0;
  for (int64_t base = 0; base < nblk; base += SCAN_T) {
    const int64_t i = base + t;
    long long x = i < nblk ? blk_cnt[i] : 0;
    if (i < nblk) e |= blk_err[i];
    for (int o = 1; o < 32; o <<= 1) {
      const long long u = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += u;
    }
    if (lane == 31) wsum[wid] = x;
    __syncthreads();
    if (wid == 0) {
      long long w = wsum[lane];
      for (int o = 1; o < 32; o <<= 1) {
        const long long u = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += u;
      }
      wsum[lane] = w;   // inclusive over warps
    }
    __syncthreads();
    const long long incl = x + (wid > 0 ? wsum[wid - 1] : 0) + carry;
    if (i < nblk) blk_off[i] = incl - (i < nblk ? blk_cnt[i] : 0);
    __syncthreads();
    if (t == SCAN_T - 1) carry = incl;
    __syncthreads();
  }
  if (e) atomicOr(&err_all, e);
  __syncthreads();
  if (t == 0) {
    *total = carry;
    unsigned bits = err_all;
    if (n_valid >= 0 && carry != n_valid) bits |= ERR_BIT_COUNT;
    acc->err |= bits;
  }
}

template <typename U>
__device__ __forceinline__ void copy_row(const char* __restrict__ src, char* __restrict__ dst, int64_t row_bytes,
                                         int lane) {
  const U* s = reinterpret_cast<const U*>(src);
  U* d = reinterpret_cast<U*>(dst);
  const int64_t n = row_bytes / (int64_t)sizeof(U);
  for (int64_t k = lane; k < n; k += 32) d[k] = s[k];
}

template <typename U>
__device__ __forceinline__ void zero_row(char* __restrict__ dst, int64_t row_bytes, int lane) {
  U* d = reinterpret_cast<U*>(dst);
  const int64_t n = row_bytes / (int64_t)sizeof(U);
  const U z = U();
  for (int64_t k = lane; k < n; k += 32) d[k] = z;
}

// vec: 16 = rows move in 16-byte words, 4 = 4-byte words, 2 = 2-byte words (the host picks the
// widest that divides the row size and both base addresses).
__device__ __forceinline__ void copy_row_w(const char* src, char* dst, int64_t row_bytes, int vec, int lane) {
  if (vec == 16) copy_row<uint4>(src, dst, row_bytes, lane);
  else if (vec == 4) copy_row<unsigned>(src, dst, row_bytes, lane);
  else copy_row<unsigned short>(src, dst, row_bytes, lane);
}
__device__ __forceinline__ void zero_row_w(char* dst, int64_t row_bytes, int vec, int lane) {
  if (vec == 16) zero_row<uint4>(dst, row_bytes, lane);
  else if (vec == 4) zero_row<unsigned>(dst, row_bytes, lane);
  else zero_row<unsigned short>(dst, row_bytes, lane);
}

__global__ void __launch_bounds__(CP_ROWS) compact_gather_kernel(const char* __restrict__ hidden,
                                                                const int32_t* __restrict__ y, int64_t N,
                                                                int64_t V, int64_t row_bytes, int vec,
                                                                const int64_t* __restrict__ blk_off,
                                                                char* __restrict__ h_c, int32_t* __restrict__ y_c,
                                                                int32_t* __restrict__ pos) {
  __shared__ int wcnt[CP_ROWS / 32];
  __shared__ int64_t rowpos[CP_ROWS];
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const int64_t n = (int64_t)blockIdx.x * CP_ROWS + t;
  const int yt = n < N ? y[n] : -1;
  const bool v = n < N && valid_target(yt, V);
  const unsigned bal = __ballot_sync(0xffffffffu, v);
  if (lane == 0) wcnt[wid] = __popc(bal);
  __syncthreads();
  int before = 0;
  for (int w = 0; w < wid; ++w) before += wcnt[w];
  const int64_t p = v ? blk_off[blockIdx.x] + before + __popc(bal & ((1u << lane) - 1u)) : -1;
  if (n < N) {
    pos[n] = (int32_t)p;
    if (v) y_c[p] = yt;
  }
  rowpos[t] = p;
  __syncthreads();
  // each warp copies the valid rows among its block's rows r = wid, wid + 4, ...
  const int64_t r0 = (int64_t)blockIdx.x * CP_ROWS;
  for (int r = wid; r < CP_ROWS; r += CP_ROWS / 32) {
    const int64_t q = rowpos[r];
    if (q < 0) continue;
    copy_row_w(hidden + (r0 + r) * row_bytes, h_c + q * row_bytes, row_bytes, vec, lane);
  }
}

// One warp per row; rows at or past n_valid (a count mismatch, already flagged) are zeroed.
constexpr int SC_T = 256;
__global__ void __launch_bounds__(SC_T) compact_scatter_kernel(const int32_t* __restrict__ pos, int64_t N,
                                                              int64_t n_valid, int64_t row_bytes, int vec,
                                                              const char* __restrict__ dh_c, char* __restrict__ dh,
                                                              const float* __restrict__ rl_c,
                                                              float* __restrict__ row_loss) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (SC_T / 32);
  for (int64_t n = (int64_t)blockIdx.x * (SC_T / 32) + (threadIdx.x >> 5); n < N; n += warps) {
    const int64_t q = pos[n];
    const bool ok = q >= 0 && q < n_valid;
    if (ok) copy_row_w(dh_c + q * row_bytes, dh + n * row_bytes, row_bytes, vec, lane);
    else zero_row_w(dh + n * row_bytes, row_bytes, vec, lane);
    if (row_loss && lane == 0) row_loss[n] = ok ? rl_c[q] : 0.f;
  }
}

int pick_vec(int64_t row_bytes, const void* a, const void* b) {
  const uintptr_t al = (uintptr_t)a | (uintptr_t)b;
  if (row_bytes % 16 == 0 && (al & 15) == 0) return 16;
  if (row_bytes % 4 == 0 && (al & 3) == 0) return 4;
  return 2;
}

}  // namespace

int64_t compact_blocks(int64_t N) { return (N + CP_ROWS - 1) / CP_ROWS; }

cudaError_t compact_rows(const StepArgs& a, const CompactScratch& cs, DevAcc* acc, int64_t n_valid,
                         Launch& L) {
  const int64_t nblk = compact_blocks(a.N);
  if (nblk > 0) {
    L.begin(K_FINISH);
    compact_count_kernel<<<(unsigned)nblk, CP_ROWS, 0, L.st>>>(a.targets, a.N, a.V, a.ignore_id, cs.blk_cnt,
                                                               cs.blk_err);
    L.end();
  }
  L.begin(K_FINISH);
  compact_scan_kernel<<<1, SCAN_T, 0, L.st>>>(cs.blk_cnt, cs.blk_err, nblk, cs.blk_off, cs.total, n_valid, acc);
  L.end();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || nblk == 0) return e;
  const int64_t esz = a.bf16 ? 2 : 4;
  const int64_t rb = a.C * esz;
  L.begin(K_FINISH);
  compact_gather_kernel<<<(unsigned)nblk, CP_ROWS, 0, L.st>>>(
      (const char*)a.hidden, a.targets, a.N, a.V, rb, pick_vec(rb, a.hidden, cs.h_c), cs.blk_off, (char*)cs.h_c,
      cs.y_c, cs.pos);
  L.end();
  return cudaGetLastError();
}

cudaError_t compact_scatter(const StepArgs& a, const CompactScratch& cs, int64_t n_valid, Launch& L) {
  if (a.N == 0) return cudaSuccess;
  const int64_t esz = a.bf16 ? 2 : 4;
  const int64_t rb = a.C * esz;
  int64_t blocks = (a.N + SC_T / 32 - 1) / (SC_T / 32);
  if (blocks > 152 * 8) blocks = 152 * 8;
  L.begin(K_FINISH);
  compact_scatter_kernel<<<(unsigned)blocks, SC_T, 0, L.st>>>(cs.pos, a.N, n_valid, rb, pick_vec(rb, a.dh, cs.dh_c),
                                                             (const char*)cs.dh_c, (char*)a.dh, cs.rl_c, a.row_loss);
  L.end();
  return cudaGetLastError();
}

}  // namespace lmce
