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

// Rows grp*R .. grp*R + R - 1.  repair == false: the lse pass of the SIMT path (lse, row loss,
// the group's partials at index grp); repair == true: only the logsumexp.
template <typename T>
__device__ void simt_lse_rows(const StepArgs& a, float* __restrict__ lse_out, double* __restrict__ part_loss,
                              int* __restrict__ part_cnt, unsigned* __restrict__ part_err, int64_t grp, bool repair) {
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
  if (repair) {
    if (q == 0 && n < a.N) lse_out[n] = m + logf(l);
    return;
  }
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

// gate == nullptr: the lse pass of the SIMT path, one block per R rows.
// gate != nullptr: repair mode, grid (128-token tiles, R-row groups of a tile): a block of a
// flagged tile takes the logsumexp of its R rows, so a tile's groups run on separate SMs; the
// blocks of other tiles return at once.
template <typename T>
__global__ void __launch_bounds__(NT) simt_lse_kernel(StepArgs a, float* __restrict__ lse_out,
                                                      double* __restrict__ part_loss,
                                                      int* __restrict__ part_cnt,
                                                      unsigned* __restrict__ part_err,
                                                      const unsigned* __restrict__ gate) {
  griddep_wait();
  if (!gate) {
    simt_lse_rows<T>(a, lse_out, part_loss, part_cnt, part_err, blockIdx.x, false);
    return;
  }
  if (!gate[blockIdx.x]) return;  // block-uniform
  const int64_t grp = (int64_t)blockIdx.x * (TC_TILE_ROWS / R) + blockIdx.y;
  if (grp * R >= a.N) return;
  simt_lse_rows<T>(a, lse_out, part_loss, part_cnt, part_err, grp, true);
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

// gate == nullptr: one block per R owned rows.
// gate != nullptr (dh pass only): repair mode, grid (128-token tiles, R-row groups of a tile): a
// block of a flagged tile writes the dh rows of its R rows; the blocks of other tiles return at
// once.
template <typename T, bool DW>
__global__ void __launch_bounds__(NT) simt_grad_kernel(StepArgs a, const float* __restrict__ lse,
                                                       const DevAcc* __restrict__ acc_dev,
                                                       const unsigned* __restrict__ gate) {
  griddep_wait();
  if (DW || !gate) {
    simt_grad_rows<T, DW>(a, lse, acc_dev, blockIdx.x);
    return;
  }
  if (!gate[blockIdx.x]) return;  // block-uniform
  const int64_t grp = (int64_t)blockIdx.x * (TC_TILE_ROWS / R) + blockIdx.y;
  if (grp * R >= a.N) return;
  simt_grad_rows<T, DW>(a, lse, acc_dev, grp);
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
  kdw<<<(unsigned)((a.V + R - 1) / R), NT, smem, L.st>>>(a, sc.lse, sc.acc, nullptr);
  L.end();
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  L.begin(K_DH);
  kdh<<<(unsigned)simt_parts(a.N), NT, smem, L.st>>>(a, sc.lse, sc.acc, nullptr);
  L.end();
  return cudaGetLastError();
}

template <typename T>
static cudaError_t simt_run(const StepArgs& a, const Scratch& sc, Launch& L) {
  const int64_t nb = simt_parts(a.N);
  L.begin(K_LSE);
  simt_lse_kernel<T><<<(unsigned)nb, NT, 0, L.st>>>(a, sc.lse, sc.part_loss, sc.part_cnt, sc.part_err, nullptr);
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

// Repair of the one-pass tensor-core logsumexp + dh kernel (bf16): the exact two passes,
// restricted to flagged tiles.  Both launches cover every row block; blocks outside flagged
// tiles return before touching memory, so the common case costs two near-empty launches.
cudaError_t simt_repair_lse(const StepArgs& a, const Scratch& sc, Launch& L) {
  L.begin(K_LSE);
  const unsigned ntiles = (unsigned)((a.N + TC_TILE_ROWS - 1) / TC_TILE_ROWS);
  const dim3 grid(ntiles, TC_TILE_ROWS / R);
  const cudaError_t e = launch_pdl(simt_lse_kernel<__nv_bfloat16>, grid, dim3(NT), 0, L.st, a, sc.lse, nullptr, nullptr,
                                   nullptr, sc.tc_tile_flag);
  L.end();
  return e;
}

cudaError_t simt_repair_dh(const StepArgs& a, const Scratch& sc, Launch& L) {
  const size_t smem = simt_grad_smem(a.C);
  auto kdh = simt_grad_kernel<__nv_bfloat16, false>;
  cudaError_t e = max_dyn_smem((const void*)kdh, (int)smem);
  if (e != cudaSuccess) return e;
  L.begin(K_DH);
  const unsigned ntiles = (unsigned)((a.N + TC_TILE_ROWS - 1) / TC_TILE_ROWS);
  const dim3 grid(ntiles, TC_TILE_ROWS / R);
  e = launch_pdl(kdh, grid, dim3(NT), smem, L.st, a, sc.lse, sc.acc, sc.tc_tile_flag);
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
