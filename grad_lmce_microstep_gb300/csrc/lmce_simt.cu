// SIMT (fp32 FFMA) kernels of the fused LM-head + cross-entropy micro-step.
//
// This path serves fp32 inputs (the character-level model) and any shape the
// tensor-core path does not take.  Its three passes mirror the definition in
// "How I trained my own GPT-2 124M on FineWeb-Edu", section 4:
//   lse pass : logits z = h . W^T tile by tile, online max / sum-exp per row, the
//              target's logit, the per-row loss lse - z_target;
//   dW pass  : one block owns R vocabulary rows and streams every token:
//              dz = s (softmax - onehot) recomputed tile by tile, dW_v += dz^T h;
//   dh pass  : one block owns R token rows and streams the vocabulary:
//              dh_n += dz W.
// Logit tiles live only in registers and shared memory.  Every output element has
// one owning block that sums in a fixed order, so results are bitwise reproducible.
#include "lmce_internal.cuh"

namespace lmce {
namespace {

constexpr int R = 16;    // rows owned by one block
static_assert(TC_TILE_ROWS % R == 0, "a repair block walks whole R-row groups of its tile");
constexpr int BT = 64;   // streamed rows per tile
constexpr int BK = 32;   // reduction chunk
constexpr int NT = 256;  // threads per block

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float v, float* p) { *p = v; }
__device__ __forceinline__ void from_f(float v, __nv_bfloat16* p) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ bool target_valid(int y, int64_t V) { return y >= 0 && (int64_t)y < V; }

// S[r][t] = sum_c X[own0 + r][c] * Y[t0 + t][c] for the block's R owned rows and a
// tile of BT streamed rows.  Thread (r = tid / 16, q = tid % 16) returns t = q + 16 j.
template <typename T>
__device__ __forceinline__ void logit_tile(const T* __restrict__ X, int64_t own0, int64_t nown,
                                           const T* __restrict__ Y, int64_t t0, int64_t nstr,
                                           int64_t C, float (&acc)[4],
                                           float (*Xs)[R], float (*Ys)[BT + 1]) {
  const int tid = threadIdx.x;
  const int r = tid >> 4, q = tid & 15;
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = 0.f;
  for (int64_t c0 = 0; c0 < C; c0 += BK) {
    // X chunk: R x BK = 512 values, 2 per thread
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      int e = tid + i * NT;
      int rr = e / BK, k = e % BK;
      int64_t row = own0 + rr, col = c0 + k;
      Xs[k][rr] = (row < nown && col < C) ? to_f(X[row * C + col]) : 0.f;
    }
    // Y chunk: BT x BK = 2048 values, 8 per thread
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int e = tid + i * NT;
      int tt = e / BK, k = e % BK;
      int64_t row = t0 + tt, col = c0 + k;
      Ys[k][tt] = (row < nstr && col < C) ? to_f(Y[row * C + col]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < BK; ++k) {
      float xv = Xs[k][r];
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[j] = fmaf(xv, Ys[k][q + 16 * j], acc[j]);
    }
    __syncthreads();
  }
}

// Rows grp*R .. grp*R + R - 1: the lse pass of the SIMT path (lse, row loss, the group's partials
// at index grp).
template <typename T>
__device__ void simt_lse_rows(const StepArgs& a, float* __restrict__ lse_out, double* __restrict__ part_loss,
                              int* __restrict__ part_cnt, unsigned* __restrict__ part_err, int64_t grp) {
  __shared__ float Xs[BK][R];
  __shared__ float Ys[BK][BT + 1];
  __shared__ float zt[R];
  __shared__ double rl[R];
  __shared__ int rv[R];
  __shared__ unsigned re[R];
  const T* H = static_cast<const T*>(a.hidden);
  const T* W = static_cast<const T*>(a.W);
  const int tid = threadIdx.x, r = tid >> 4, q = tid & 15;
  const int64_t n0 = grp * R, n = n0 + r;
  const int y = (n < a.N) ? a.targets[n] : a.ignore_id;
  if (q == 0) zt[r] = 0.f;
  float m = -INFINITY, l = 0.f;
  for (int64_t v0 = 0; v0 < a.V; v0 += BT) {
    float s[4];
    logit_tile(H, n0, a.N, W, v0, a.V, a.C, s, Xs, Ys);
    float tmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int64_t v = v0 + q + 16 * j;
      if (v < a.V) {
        tmax = fmaxf(tmax, s[j]);
        if (v == y) zt[r] = s[j];
      }
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    float mn = fmaxf(m, tmax);
    float ts = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int64_t v = v0 + q + 16 * j;
      if (v < a.V) ts += expf(s[j] - mn);
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) ts += __shfl_xor_sync(0xffffffffu, ts, o);
    l = l * expf(m - mn) + ts;
    m = mn;
  }
  __syncthreads();
  if (q == 0) {
    double loss = 0.0;
    int valid = 0;
    unsigned err = 0;
    if (n < a.N) {
      float lse = m + logf(l);
      lse_out[n] = lse;
      if (target_valid(y, a.V)) {
        float li = lse - zt[r];
        loss = (double)li;
        valid = 1;
        if (!isfinite(li)) err |= ERR_BIT_NONFINITE;
        if (a.row_loss) a.row_loss[n] = li;
      } else {
        if (y != a.ignore_id) err |= ERR_BIT_BAD_TARGET;
        if (a.row_loss) a.row_loss[n] = 0.f;
      }
    }
    rl[r] = loss;
    rv[r] = valid;
    re[r] = err;
  }
  __syncthreads();
  if (tid == 0) {
    double t = 0.0;
    int c = 0;
    unsigned e = 0;
    for (int i = 0; i < R; ++i) { t += rl[i]; c += rv[i]; e |= re[i]; }
    part_loss[grp] = t;
    part_cnt[grp] = c;
    part_err[grp] = e;
  }
}

// The lse pass of the SIMT path, one block per R rows.
template <typename T>
__global__ void __launch_bounds__(NT) simt_lse_kernel(StepArgs a, float* __restrict__ lse_out,
                                                      double* __restrict__ part_loss,
                                                      int* __restrict__ part_cnt,
                                                      unsigned* __restrict__ part_err) {
  simt_lse_rows<T>(a, lse_out, part_loss, part_cnt, part_err, blockIdx.x);
}

// Owned rows grp*R .. grp*R + R - 1.
// DW = true : own R vocabulary rows, stream the tokens, acc = dW rows.
// DW = false: own R token rows, stream the vocabulary, acc = dh rows.
template <typename T, bool DW>
__device__ void simt_grad_rows(const StepArgs& a, const float* __restrict__ lse, const DevAcc* __restrict__ acc_dev,
                               int64_t grp) {
  __shared__ float Xs[BK][R];
  __shared__ float Ys[BK][BT + 1];
  __shared__ float dzs[R][BT];
  extern __shared__ float accs[];  // [R][C]
  const T* H = static_cast<const T*>(a.hidden);
  const T* Wt = static_cast<const T*>(a.W);
  const T* X = DW ? Wt : H;
  const T* Y = DW ? H : Wt;
  const int64_t nown = DW ? a.V : a.N;
  const int64_t nstr = DW ? a.N : a.V;
  const int tid = threadIdx.x, r = tid >> 4, q = tid & 15;
  const int64_t own0 = grp * R;
  // global normalisation: the caller's 1 / global_valid (the value the finish pass stores, and
  // available before it); micro-step mean: the scale the count pass set
  const float s = a.norm == 0 ? (float)(1.0 / (double)a.global_valid) : acc_dev->scale;
  for (int64_t i = tid; i < (int64_t)R * a.C; i += NT) accs[i] = 0.f;
  // per-owned-row constants for the dh pass
  int yown = a.ignore_id;
  float lown = 0.f;
  if (!DW && own0 + r < a.N) {
    yown = a.targets[own0 + r];
    lown = lse[own0 + r];
  }
  __syncthreads();
  for (int64_t t0 = 0; t0 < nstr; t0 += BT) {
    float sv[4];
    logit_tile(X, own0, nown, Y, t0, nstr, a.C, sv, Xs, Ys);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int t = q + 16 * j;
      int64_t o = own0 + r, st = t0 + t;
      float dz = 0.f;
      if (DW) {
        if (o < a.V && st < a.N) {
          int y = a.targets[st];
          if (target_valid(y, a.V)) dz = s * (expf(sv[j] - lse[st]) - (y == o ? 1.f : 0.f));
        }
      } else {
        if (o < a.N && st < a.V && target_valid(yown, a.V))
          dz = s * (expf(sv[j] - lown) - (yown == st ? 1.f : 0.f));
      }
      dzs[r][t] = dz;
    }
    __syncthreads();
    const int64_t tn = (nstr - t0 < BT) ? (nstr - t0) : BT;
    for (int64_t c = tid; c < a.C; c += NT) {
      float av[R];
#pragma unroll
      for (int i = 0; i < R; ++i) av[i] = accs[i * a.C + c];
      for (int t = 0; t < tn; ++t) {
        float yv = to_f(Y[(t0 + t) * a.C + c]);
#pragma unroll
        for (int i = 0; i < R; ++i) av[i] = fmaf(dzs[i][t], yv, av[i]);
      }
#pragma unroll
      for (int i = 0; i < R; ++i) accs[i * a.C + c] = av[i];
    }
    __syncthreads();
  }
  for (int64_t i = tid; i < (int64_t)R * a.C; i += NT) {
    int64_t rr = i / a.C, c = i % a.C, o = own0 + rr;
    if (o >= nown) continue;
    if (DW) {
      float* p = a.dW + o * a.C + c;
      *p = a.beta ? (*p + accs[i]) : accs[i];
    } else {
      from_f(accs[i], static_cast<T*>(a.dh) + o * a.C + c);
    }
  }
}

// The gradient passes of the SIMT path: one block per R owned rows.
template <typename T, bool DW>
__global__ void __launch_bounds__(NT) simt_grad_kernel(StepArgs a, const float* __restrict__ lse,
                                                       const DevAcc* __restrict__ acc_dev) {
  simt_grad_rows<T, DW>(a, lse, acc_dev, blockIdx.x);
}

// ---- exact repair of the one-pass tensor-core logsumexp + dh kernel -----------------------
// The rows of the 128-token tiles whose flag is set get their logsumexp and dh recomputed with
// the exact two-pass arithmetic above.  Both kernels are persistent (one block per SM): every
// block finds the flagged tiles itself (nothing flagged: every block returns after reading the
// flags), and the work items (flagged tile, R-row group, vocabulary slice) are spread over the
// blocks, the slices chosen so that about one item falls on each SM.  A row group's slices are
// merged by the block that finishes the group's last item (a ticket per group, counted, never
// waited on), in slice order: deterministic.
constexpr int REP_BLOCKS = 152;   // one per SM of a 152-SM GB300
constexpr int REP_VS_MAX = 32;    // most vocabulary slices per row group
constexpr int REP_GROUPS = TC_TILE_ROWS / R;

// Vocabulary slices per row group for `groups` groups (1 when there are enough groups to go round).
__device__ __forceinline__ int rep_slices(int groups) {
  const int nv = REP_BLOCKS / groups;
  return nv < 1 ? 1 : (nv > REP_VS_MAX ? REP_VS_MAX : nv);
}

// The flagged tiles in tile order, into list[]; returns how many.  A block-wide call.
__device__ int rep_flagged(const unsigned* __restrict__ flag, int ntiles, int* list) {
  __shared__ int wsum[NT / 32];
  __shared__ int found;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (threadIdx.x == 0) found = 0;
  __syncthreads();
  for (int b = 0; b < ntiles; b += NT) {
    const int i = b + threadIdx.x;
    const bool f = i < ntiles && flag[i] != 0u;
    const unsigned bal = __ballot_sync(0xffffffffu, f);
    if (lane == 0) wsum[w] = __popc(bal);
    __syncthreads();
    int off = found;
    for (int k = 0; k < w; ++k) off += wsum[k];
    if (f) list[off + __popc(bal & ((1u << lane) - 1u))] = i;
    __syncthreads();
    if (threadIdx.x == 0)
      for (int k = 0; k < NT / 32; ++k) found += wsum[k];
    __syncthreads();
  }
  return found;
}

// True in the block that finishes the last of a group's `nv` items (after its writes are visible
// device-wide); that block then merges the group.  The ticket returns to 0.  A block-wide call.
__device__ __forceinline__ bool rep_last_item(unsigned* ticket, int nv) {
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    last = atomicAdd(ticket, 1u) == (unsigned)nv - 1u;
    if (last) *ticket = 0u;
  }
  __syncthreads();
  if (last) __threadfence();
  return last != 0;
}

// Logsumexp of rows n0 .. n0 + R - 1 over the vocabulary rows [v0, v1): per-row running
// (max, sum) with natural-base exponentials, as the SIMT lse pass.  Thread (r, q) holds row r.
template <typename T>
__device__ void rep_lse_range(const StepArgs& a, int64_t n0, int64_t v0, int64_t v1, float& m, float& l,
                              float (*Xs)[R], float (*Ys)[BT + 1]) {
  const T* H = static_cast<const T*>(a.hidden);
  const T* W = static_cast<const T*>(a.W);
  const int q = threadIdx.x & 15;
  m = -INFINITY;
  l = 0.f;
  for (int64_t t0 = v0; t0 < v1; t0 += BT) {
    float s[4];
    logit_tile(H, n0, a.N, W, t0, v1, a.C, s, Xs, Ys);
    float tmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (t0 + q + 16 * j < v1) tmax = fmaxf(tmax, s[j]);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    const float mn = fmaxf(m, tmax);
    float ts = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (t0 + q + 16 * j < v1) ts += expf(s[j] - mn);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) ts += __shfl_xor_sync(0xffffffffu, ts, o);
    l = (m == -INFINITY ? 0.f : l * expf(m - mn)) + ts;
    m = mn;
  }
}

// part: [REP_BLOCKS][2][R] (max, sum) of the items of groups split into slices.
__global__ void __launch_bounds__(NT) repair_lse_kernel(StepArgs a, const unsigned* __restrict__ flag, int ntiles,
                                                        float* __restrict__ lse_out, float* __restrict__ part,
                                                        unsigned* __restrict__ ticket) {
  griddep_wait();
  __shared__ float Xs[BK][R];
  __shared__ float Ys[BK][BT + 1];
  extern __shared__ int rep_list[];
  const int nf = rep_flagged(flag, ntiles, rep_list);
  if (nf == 0) return;
  const int groups = nf * REP_GROUPS, nv = rep_slices(groups);
  const int64_t vw = ((a.V + nv - 1) / nv + BT - 1) / BT * BT;   // slice width, whole logit tiles
  const int r = threadIdx.x >> 4, q = threadIdx.x & 15;
  for (int it = blockIdx.x; it < groups * nv; it += gridDim.x) {
    const int gi = it / nv, v = it % nv;
    const int64_t n0 = (int64_t)rep_list[gi / REP_GROUPS] * TC_TILE_ROWS + (gi % REP_GROUPS) * R;
    if (n0 >= a.N) continue;   // the whole group lies past the rows: none of its items runs
    const int64_t v0 = (int64_t)v * vw, v1 = v0 + vw < a.V ? v0 + vw : a.V;
    float m, l;
    rep_lse_range<__nv_bfloat16>(a, n0, v0, v1, m, l, Xs, Ys);
    if (nv == 1) {
      if (q == 0 && n0 + r < a.N) lse_out[n0 + r] = m + logf(l);
      continue;
    }
    if (q == 0) {
      part[((size_t)it * 2 + 0) * R + r] = m;
      part[((size_t)it * 2 + 1) * R + r] = l;
    }
    if (rep_last_item(ticket + gi, nv) && q == 0 && n0 + r < a.N) {
      float M = -INFINITY;
      for (int k = 0; k < nv; ++k) M = fmaxf(M, __ldcg(part + ((size_t)(gi * nv + k) * 2 + 0) * R + r));
      float L = 0.f;
      for (int k = 0; k < nv; ++k) {
        const float mk = __ldcg(part + ((size_t)(gi * nv + k) * 2 + 0) * R + r);
        if (mk != -INFINITY) L += __ldcg(part + ((size_t)(gi * nv + k) * 2 + 1) * R + r) * expf(mk - M);
      }
      lse_out[n0 + r] = M + logf(L);
    }
  }
}

// part: [REP_BLOCKS][R][C] fp32 dh partials of the items of groups split into slices.  Dynamic
// shared memory: the R x C accumulator, then the flagged-tile list.
// pst (null: nothing stored): the stored exponentials [N][vp], whose flagged rows get p = softmax
// (0 for a row without a valid target), and mref [TC_MAX_VER][np] their reference lse log2 e.
__global__ void __launch_bounds__(NT) repair_dh_kernel(StepArgs a, const unsigned* __restrict__ flag, int ntiles,
                                                       const float* __restrict__ lse, const DevAcc* __restrict__ acc_dev,
                                                       float* __restrict__ part, unsigned* __restrict__ ticket,
                                                       __nv_bfloat16* __restrict__ pst, int64_t vp,
                                                       float* __restrict__ mref, int64_t np) {
  griddep_wait();
  __shared__ float Xs[BK][R];
  __shared__ float Ys[BK][BT + 1];
  __shared__ float dzs[R][BT];
  extern __shared__ float accs[];   // [R][C], then the list
  int* rep_list = reinterpret_cast<int*>(accs + (size_t)R * a.C);
  const int nf = rep_flagged(flag, ntiles, rep_list);
  if (nf == 0) return;
  const int groups = nf * REP_GROUPS, nv = rep_slices(groups);
  const int64_t vw = ((a.V + nv - 1) / nv + BT - 1) / BT * BT;
  const __nv_bfloat16* H = static_cast<const __nv_bfloat16*>(a.hidden);
  const __nv_bfloat16* W = static_cast<const __nv_bfloat16*>(a.W);
  const int tid = threadIdx.x, r = tid >> 4, q = tid & 15;
  // global normalisation: the caller's 1 / global_valid; micro-step mean: the count pass's scale
  const float s = a.norm == 0 ? (float)(1.0 / (double)a.global_valid) : acc_dev->scale;
  for (int it = blockIdx.x; it < groups * nv; it += gridDim.x) {
    const int gi = it / nv, v = it % nv;
    const int64_t n0 = (int64_t)rep_list[gi / REP_GROUPS] * TC_TILE_ROWS + (gi % REP_GROUPS) * R;
    if (n0 >= a.N) continue;
    const int64_t v0 = (int64_t)v * vw, v1 = v0 + vw < a.V ? v0 + vw : a.V;
    for (int64_t i = tid; i < (int64_t)R * a.C; i += NT) accs[i] = 0.f;
    int y = -1;
    float ln = 0.f;
    if (n0 + r < a.N) {
      const int t = a.targets[n0 + r];
      if (target_valid(t, a.V)) {
        y = t;
        ln = lse[n0 + r];
      }
    }
    if (pst && v == 0 && q == 0 && n0 + r < a.N)
      for (int k = 0; k < TC_MAX_VER; ++k) mref[(size_t)k * np + n0 + r] = ln * 1.4426950408889634f;
    __syncthreads();
    for (int64_t t0 = v0; t0 < v1; t0 += BT) {
      float sv[4];
      logit_tile(H, n0, a.N, W, t0, v1, a.C, sv, Xs, Ys);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t vv = t0 + q + 16 * j;
        const float pv = (y >= 0 && vv < v1) ? expf(sv[j] - ln) : 0.f;
        dzs[r][q + 16 * j] = (y >= 0 && vv < v1) ? s * (pv - (vv == y ? 1.f : 0.f)) : 0.f;
        if (pst && vv < v1 && n0 + r < a.N) pst[(n0 + r) * vp + vv] = __float2bfloat16_rn(pv);
      }
      __syncthreads();
      const int64_t tn = v1 - t0 < BT ? v1 - t0 : BT;
      for (int64_t c = tid; c < a.C; c += NT) {
        float av[R];
#pragma unroll
        for (int i = 0; i < R; ++i) av[i] = accs[i * a.C + c];
        for (int t = 0; t < tn; ++t) {
          const float wv = to_f(W[(t0 + t) * a.C + c]);
#pragma unroll
          for (int i = 0; i < R; ++i) av[i] = fmaf(dzs[i][t], wv, av[i]);
        }
#pragma unroll
        for (int i = 0; i < R; ++i) accs[i * a.C + c] = av[i];
      }
      __syncthreads();
    }
    __nv_bfloat16* dh = static_cast<__nv_bfloat16*>(a.dh);
    if (nv == 1) {
      for (int64_t i = tid; i < (int64_t)R * a.C; i += NT) {
        const int64_t rr = i / a.C, c = i % a.C;
        if (n0 + rr < a.N) from_f(accs[i], dh + (n0 + rr) * a.C + c);
      }
      __syncthreads();   // accs is reused by the next item
      continue;
    }
    float* mine = part + (size_t)it * R * a.C;
    for (int64_t i = tid; i < (int64_t)R * a.C; i += NT) mine[i] = accs[i];
    if (rep_last_item(ticket + gi, nv)) {
      for (int64_t i = tid; i < (int64_t)R * a.C; i += NT) {
        const int64_t rr = i / a.C, c = i % a.C;
        float sum = 0.f;
        for (int k = 0; k < nv; ++k) sum += __ldcg(part + (size_t)(gi * nv + k) * R * a.C + i);
        if (n0 + rr < a.N) from_f(sum, dh + (n0 + rr) * a.C + c);
      }
    }
    __syncthreads();
  }
}

}  // namespace

int64_t simt_parts(int64_t N) { return (N + R - 1) / R; }

size_t simt_grad_smem(int64_t C) { return (size_t)R * (size_t)C * sizeof(float); }

template <typename T>
static cudaError_t simt_grads_t(const StepArgs& a, const Scratch& sc, Launch& L) {
  const size_t smem = simt_grad_smem(a.C);
  auto kdw = simt_grad_kernel<T, true>;
  auto kdh = simt_grad_kernel<T, false>;
  // the static tiles (~15 KB) plus R*C floats can exceed the default 48 KB window
  cudaError_t e = max_dyn_smem((const void*)kdw, (int)smem);
  if (e == cudaSuccess) e = max_dyn_smem((const void*)kdh, (int)smem);
  if (e != cudaSuccess) return e;
  L.begin(K_DW);
  kdw<<<(unsigned)((a.V + R - 1) / R), NT, smem, L.st>>>(a, sc.lse, sc.acc);
  L.end();
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  L.begin(K_DH);
  kdh<<<(unsigned)simt_parts(a.N), NT, smem, L.st>>>(a, sc.lse, sc.acc);
  L.end();
  return cudaGetLastError();
}

template <typename T>
static cudaError_t simt_run(const StepArgs& a, const Scratch& sc, Launch& L) {
  const int64_t nb = simt_parts(a.N);
  L.begin(K_LSE);
  simt_lse_kernel<T><<<(unsigned)nb, NT, 0, L.st>>>(a, sc.lse, sc.part_loss, sc.part_cnt, sc.part_err);
  L.end();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_finish(a, sc, nb, L);
  if (e != cudaSuccess) return e;
  return simt_grads_t<T>(a, sc, L);
}

cudaError_t simt_microstep(const StepArgs& a, const Scratch& sc, Launch& L) {
  return a.bf16 ? simt_run<__nv_bfloat16>(a, sc, L) : simt_run<float>(a, sc, L);
}

cudaError_t simt_grads(const StepArgs& a, const Scratch& sc, Launch& L) {
  return a.bf16 ? simt_grads_t<__nv_bfloat16>(a, sc, L) : simt_grads_t<float>(a, sc, L);
}

// Exact repair of the one-pass tensor-core logsumexp + dh kernel (bf16): two persistent launches
// of REP_BLOCKS blocks whose blocks return at once when no tile is flagged.
size_t simt_repair_part_floats(int64_t C) { return (size_t)REP_BLOCKS * R * (size_t)(C > 2 ? C : 2); }

cudaError_t simt_repair_lse(const StepArgs& a, const Scratch& sc, Launch& L) {
  const int ntiles = (int)((a.N + TC_TILE_ROWS - 1) / TC_TILE_ROWS);
  L.begin(K_LSE);
  const cudaError_t e = launch_pdl(repair_lse_kernel, dim3(REP_BLOCKS), dim3(NT), sizeof(int) * (size_t)ntiles, L.st, a,
                                   sc.tc_tile_flag, ntiles, sc.lse, sc.rep_part, sc.rep_ticket);
  L.end();
  return e;
}

cudaError_t simt_repair_dh(const StepArgs& a, const Scratch& sc, Launch& L, bool store_p) {
  const int ntiles = (int)((a.N + TC_TILE_ROWS - 1) / TC_TILE_ROWS);
  const size_t smem = simt_grad_smem(a.C) + sizeof(int) * (size_t)ntiles;
  cudaError_t e = max_dyn_smem((const void*)repair_dh_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  L.begin(K_DH);
  e = launch_pdl(repair_dh_kernel, dim3(REP_BLOCKS), dim3(NT), smem, L.st, a, sc.tc_tile_flag, ntiles, sc.lse, sc.acc,
                 sc.rep_part, sc.rep_ticket, store_p ? sc.tc_p : (__nv_bfloat16*)nullptr, tc_p_cols(a.V), sc.tc_mref,
                 tc_ver_rows(a.N));
  L.end();
  return e;
}

// Loads the module of every SIMT kernel, both dtypes (with lazy module loading a module is
// otherwise loaded, and its device memory allocated, at the first launch of one of its kernels).
cudaError_t simt_load_kernels() {
  cudaFuncAttributes fa;
  cudaError_t e;
  if ((e = cudaFuncGetAttributes(&fa, simt_lse_kernel<float>)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, simt_lse_kernel<__nv_bfloat16>)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, simt_grad_kernel<float, true>)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, simt_grad_kernel<float, false>)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, simt_grad_kernel<__nv_bfloat16, true>)) != cudaSuccess) return e;
  return cudaFuncGetAttributes(&fa, simt_grad_kernel<__nv_bfloat16, false>);
}

}  // namespace lmce
