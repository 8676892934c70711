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

constexpr int CP_ROWS = 32;    // rows per block of count, gather and scatter
constexpr int SCAN_T = 1024;

__device__ __forceinline__ bool valid_target(int y, int64_t V) { return y >= 0 && (int64_t)y < V; }

__global__ void __launch_bounds__(CP_ROWS) compact_count_kernel(const int32_t* __restrict__ y, int64_t N,
                                                               int64_t V, int32_t ignore_id,
                                                               int* __restrict__ blk_cnt,
                                                               unsigned* __restrict__ blk_err) {
  griddep_wait();
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
  griddep_wait();
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

// Row moves are flat over words (U = 16, 4 or 2 bytes, the widest that divides the row size and
// both base addresses): a block moves the CP_ROWS rows of one count block, consecutive threads
// taking consecutive words of a row so every warp access is coalesced, each thread with CP_U
// loads in flight before its stores.  Word indices within a block fit 32 bits (CP_ROWS x the
// words of a row <= 32 x 2^21).
constexpr int CP_U = 4;
constexpr int MV_T = 256;

template <typename U>
__global__ void __launch_bounds__(MV_T) compact_gather_kernel(const U* __restrict__ hidden,
                                                             const int32_t* __restrict__ y, int64_t N, int64_t V,
                                                             unsigned w, const int64_t* __restrict__ blk_off,
                                                             U* __restrict__ h_c, int32_t* __restrict__ y_c,
                                                             int32_t* __restrict__ pos, int64_t rows,
                                                             unsigned* err) {
  griddep_wait();
  __shared__ int64_t rowpos[CP_ROWS];
  const int t = threadIdx.x;
  const int64_t r0 = (int64_t)blockIdx.x * CP_ROWS;
  if (t < 32) {   // warp 0: one row per lane
    const int64_t n = r0 + t;
    const int yt = n < N ? y[n] : -1;
    const bool v = n < N && valid_target(yt, V);
    const unsigned bal = __ballot_sync(0xffffffffu, v);
    int64_t p = v ? blk_off[blockIdx.x] + __popc(bal & ((1u << t) - 1u)) : -1;
    if (p >= 0 && !dcheck(p < rows, err, BS_COMPACT_POS)) p = -1;
    if (n < N) {
      pos[n] = (int32_t)p;
      if (v) y_c[p] = yt;
    }
    rowpos[t] = p;
  }
  __syncthreads();
  const unsigned total = CP_ROWS * w;
  for (unsigned c0 = t; c0 < total; c0 += MV_T * CP_U) {
    U v[CP_U];
    int64_t d[CP_U];
#pragma unroll
    for (int u = 0; u < CP_U; ++u) {
      const unsigned c = c0 + u * MV_T;
      d[u] = -1;
      if (c < total) {
        const unsigned r = c / w, col = c - r * w;
        const int64_t q = rowpos[r];
        if (q >= 0) {
          v[u] = hidden[(r0 + r) * w + col];
          d[u] = q * w + col;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < CP_U; ++u)
      if (d[u] >= 0) h_c[d[u]] = v[u];
  }
}

// dh[n] = dh_c[pos[n]] for the CP_ROWS rows of a block; rows without a position, or at or past
// n_valid (a count mismatch, already flagged), are zeroed.
template <typename U>
__global__ void __launch_bounds__(MV_T) compact_scatter_kernel(const int32_t* __restrict__ pos, int64_t N,
                                                              int64_t n_valid, unsigned w, const U* __restrict__ dh_c,
                                                              U* __restrict__ dh, const float* __restrict__ rl_c,
                                                              float* __restrict__ row_loss, int64_t cap,
                                                              unsigned* err) {
  griddep_wait();
  __shared__ int64_t rowpos[CP_ROWS];
  const int t = threadIdx.x;
  const int64_t r0 = (int64_t)blockIdx.x * CP_ROWS;
  const int rows = (int)(N - r0 < CP_ROWS ? N - r0 : CP_ROWS);
  if (t < rows) {
    const int64_t q = pos[r0 + t];
    const bool ok = q >= 0 && q < n_valid && dcheck(q < cap, err, BS_SCATTER_POS);
    rowpos[t] = ok ? q : -1;
    if (row_loss) row_loss[r0 + t] = ok ? rl_c[q] : 0.f;
  }
  __syncthreads();
  const unsigned total = (unsigned)rows * w;
  for (unsigned c0 = t; c0 < total; c0 += MV_T * CP_U) {
    U v[CP_U];
#pragma unroll
    for (int u = 0; u < CP_U; ++u) {
      const unsigned c = c0 + u * MV_T;
      v[u] = U();
      if (c < total) {
        const unsigned r = c / w, col = c - r * w;
        const int64_t q = rowpos[r];
        if (q >= 0) v[u] = dh_c[q * w + col];
      }
    }
#pragma unroll
    for (int u = 0; u < CP_U; ++u) {
      const unsigned c = c0 + u * MV_T;
      if (c < total) dh[r0 * w + c] = v[u];
    }
  }
}

int pick_vec(int64_t row_bytes, const void* a, const void* b) {
  const uintptr_t al = (uintptr_t)a | (uintptr_t)b;
  if (row_bytes % 16 == 0 && (al & 15) == 0) return 16;
  if (row_bytes % 4 == 0 && (al & 3) == 0) return 4;
  return 2;
}

template <typename U>
void launch_gather(const StepArgs& a, const CompactScratch& cs, int64_t nblk, int64_t rb, cudaStream_t st) {
  launch_pdl(compact_gather_kernel<U>, dim3((unsigned)nblk), dim3(MV_T), 0, st, (const U*)a.hidden, a.targets, a.N, a.V,
             (unsigned)(rb / (int64_t)sizeof(U)), (const int64_t*)cs.blk_off, (U*)cs.h_c, cs.y_c, cs.pos, cs.rows, cs.err);
}

template <typename U>
void launch_scatter(const StepArgs& a, const CompactScratch& cs, int64_t n_valid, int64_t rb, cudaStream_t st) {
  launch_pdl(compact_scatter_kernel<U>, dim3((unsigned)compact_blocks(a.N)), dim3(MV_T), 0, st, (const int32_t*)cs.pos,
             a.N, n_valid, (unsigned)(rb / (int64_t)sizeof(U)), (const U*)cs.dh_c, (U*)a.dh, (const float*)cs.rl_c,
             a.row_loss, cs.rows, cs.err);
}

}  // namespace

int64_t compact_blocks(int64_t N) { return (N + CP_ROWS - 1) / CP_ROWS; }

cudaError_t compact_count_scan(const StepArgs& a, const CompactScratch& cs, DevAcc* acc, int64_t n_valid,
                               Launch& L) {
  const int64_t nblk = compact_blocks(a.N);
  if (nblk > 0) {
    L.begin(K_COMPACT);
    launch_pdl(compact_count_kernel, dim3((unsigned)nblk), dim3(CP_ROWS), 0, L.st, a.targets, a.N, a.V, a.ignore_id,
               cs.blk_cnt, cs.blk_err);
    L.end();
  }
  L.begin(K_COMPACT);
  launch_pdl(compact_scan_kernel, dim3(1), dim3(SCAN_T), 0, L.st, (const int*)cs.blk_cnt, (const unsigned*)cs.blk_err, nblk,
             cs.blk_off, cs.total, n_valid, acc);
  L.end();
  return cudaGetLastError();
}

cudaError_t compact_rows(const StepArgs& a, const CompactScratch& cs, DevAcc* acc, int64_t n_valid,
                         Launch& L) {
  const int64_t nblk = compact_blocks(a.N);
  cudaError_t e = compact_count_scan(a, cs, acc, n_valid, L);
  if (e != cudaSuccess || nblk == 0) return e;
  const int64_t esz = a.bf16 ? 2 : 4;
  const int64_t rb = a.C * esz;
  const int vec = pick_vec(rb, a.hidden, cs.h_c);
  L.begin(K_COMPACT);
  if (vec == 16) launch_gather<uint4>(a, cs, nblk, rb, L.st);
  else if (vec == 4) launch_gather<unsigned>(a, cs, nblk, rb, L.st);
  else launch_gather<unsigned short>(a, cs, nblk, rb, L.st);
  L.end();
  return cudaGetLastError();
}

cudaError_t compact_scatter(const StepArgs& a, const CompactScratch& cs, int64_t n_valid, Launch& L) {
  if (a.N == 0) return cudaSuccess;
  const int64_t esz = a.bf16 ? 2 : 4;
  const int64_t rb = a.C * esz;
  const int vec = pick_vec(rb, a.dh, cs.dh_c);
  L.begin(K_COMPACT);
  if (vec == 16) launch_scatter<uint4>(a, cs, n_valid, rb, L.st);
  else if (vec == 4) launch_scatter<unsigned>(a, cs, n_valid, rb, L.st);
  else launch_scatter<unsigned short>(a, cs, n_valid, rb, L.st);
  L.end();
  return cudaGetLastError();
}

}  // namespace lmce
