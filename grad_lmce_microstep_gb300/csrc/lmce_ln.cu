// The final normalisation in front of the head, forward and backward, around a micro-step.
// "How I trained my own GPT-2 124M", section 2.8: the last block's output goes through one
// LayerNorm (ln_f) before the tied head; "Reproduce GPT-2 124M" (model definition) uses an
// RMSNorm there.  Both are row-wise and memory-bound: one warp per row, the row held in
// registers (packed, with the warp's next row already in flight), statistics in float32.
//
//   forward : h = (x - mean) * rstd * gamma + beta  (RMSNorm: mean = 0, no beta), rounded to the
//             head's dtype; mean and rstd kept per row
//   backward: with xhat = (x - mean) * rstd and g = dh * gamma,
//             dx = rstd * (g - mean_c(g) - xhat * mean_c(g * xhat))  (RMSNorm: no mean_c(g) term);
//             dgamma = sum_n dh * xhat and dbeta = sum_n dh as per-block partials over contiguous
//             row ranges, then summed over blocks in a fixed order (deterministic)
#include <math.h>

#include "lmce_internal.cuh"

namespace lmce {
namespace {

constexpr int LN_T = 256;            // forward: 8 warps, one row each at a time
// backward kernels of the register layout: one block per SM, 12 warps when a lane's parameter
// sums (2 x KV x VN floats) fit beside its rows in the 168 registers that leaves, else 8
template <typename T, int KV>
constexpr int lnb_threads() {
  return KV * (16 / (int)sizeof(T)) <= 24 && KV <= 5 ? 384 : 256;
}
constexpr int LN_BWD_GRID = 152;     // backward blocks at most: one per SM of a 152-SM GB300
constexpr int LN_MAXV = 6;           // most 16-byte words per lane of a row in the register layout

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;        // 8 bf16 in 16 bytes
  __device__ static void unpack(const uint4& u, float* f) {
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(b[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ static uint4 pack(const float* f) {
    uint4 u;
    __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return u;
  }
};
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ static uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
};

// VN consecutive fp32 parameters (gamma or beta) at a multiple of VN
template <int VN>
__device__ __forceinline__ void load_param(const float* __restrict__ p, float* f) {
#pragma unroll
  for (int i = 0; i < VN; i += 4) {
    const float4 t = __ldg(reinterpret_cast<const float4*>(p + i));
    f[i] = t.x;
    f[i + 1] = t.y;
    f[i + 2] = t.z;
    f[i + 3] = t.w;
  }
}

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void from_f(float& d, float v) { d = v; }
__device__ __forceinline__ void from_f(__nv_bfloat16& d, float v) { d = __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Register layout: a row of C elements as KV 16-byte words per lane, word k of lane l holding
// columns (k * 32 + l) * VN ... + VN - 1 (words past C are zero and skipped).  Rows stay packed
// in their input dtype and are unpacked where used, so a warp can hold its current row and the
// prefetched next one.
template <typename T, int KV>
__device__ __forceinline__ void load_row(const T* __restrict__ row, int64_t C, int lane, uint4* u) {
  constexpr int VN = Vec<T>::N;
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int64_t c = ((int64_t)k * 32 + lane) * VN;
    u[k] = c < C ? *reinterpret_cast<const uint4*>(row + c) : make_uint4(0u, 0u, 0u, 0u);
  }
}

template <typename T, int KV>
__global__ void __launch_bounds__(LN_T, KV <= 3 ? 4 : 2) ln_fwd_vec_kernel(const T* __restrict__ x, const float* __restrict__ gamma,
                                                         const float* __restrict__ beta, int64_t N, int64_t C,
                                                         int rms, float eps, T* __restrict__ h,
                                                         float* __restrict__ mean_out, float* __restrict__ rstd_out) {
  griddep_wait();
  constexpr int VN = Vec<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * (LN_T / 32);
  const float inv_c = 1.0f / (float)C;
  int64_t n = (int64_t)blockIdx.x * (LN_T / 32) + (threadIdx.x >> 5);
  uint4 cur[KV], nxt[KV];
  if (n < N) load_row<T, KV>(x + n * C, C, lane, cur);
  for (; n < N; n += stride) {
    if (n + stride < N) load_row<T, KV>(x + (n + stride) * C, C, lane, nxt);   // in flight meanwhile
    float f[VN];
    float mean = 0.f;
    if (!rms) {
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        Vec<T>::unpack(cur[k], f);
#pragma unroll
        for (int i = 0; i < VN; ++i) s += f[i];
      }
      mean = warp_sum(s) * inv_c;
    }
    float q = 0.f;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      if (((int64_t)k * 32 + lane) * VN >= C) continue;
      Vec<T>::unpack(cur[k], f);
#pragma unroll
      for (int i = 0; i < VN; ++i) {
        const float d = f[i] - mean;
        q += d * d;
      }
    }
    const float rstd = 1.0f / sqrtf(warp_sum(q) * inv_c + eps);
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int64_t c = ((int64_t)k * 32 + lane) * VN;
      if (c >= C) continue;
      float g[VN], o[VN];
      Vec<T>::unpack(cur[k], f);
      load_param<VN>(gamma + c, g);
#pragma unroll
      for (int i = 0; i < VN; ++i) o[i] = (f[i] - mean) * rstd * g[i];
      if (beta) {
        load_param<VN>(beta + c, g);
#pragma unroll
        for (int i = 0; i < VN; ++i) o[i] += g[i];
      }
      *reinterpret_cast<uint4*>(h + n * C + c) = Vec<T>::pack(o);
    }
    if (lane == 0) {
      mean_out[n] = mean;
      rstd_out[n] = rstd;
    }
#pragma unroll
    for (int k = 0; k < KV; ++k) cur[k] = nxt[k];
  }
}

template <typename T>
__global__ void __launch_bounds__(LN_T) ln_fwd_rows_kernel(const T* __restrict__ x, const float* __restrict__ gamma,
                                                          const float* __restrict__ beta, int64_t N, int64_t C,
                                                          int rms, float eps, T* __restrict__ h,
                                                          float* __restrict__ mean_out,
                                                          float* __restrict__ rstd_out) {
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t n = (int64_t)blockIdx.x * (LN_T / 32) + (threadIdx.x >> 5);
  if (n >= N) return;
  const T* xr = x + n * C;
  T* hr = h + n * C;
  const float inv_c = 1.0f / (float)C;
  float mean = 0.f;
  if (!rms) {
    float s = 0.f;
    for (int64_t c = lane; c < C; c += 32) s += to_f(xr[c]);
    mean = warp_sum(s) * inv_c;
  }
  float q = 0.f;
  for (int64_t c = lane; c < C; c += 32) {
    const float d = to_f(xr[c]) - mean;
    q += d * d;
  }
  const float rstd = 1.0f / sqrtf(warp_sum(q) * inv_c + eps);
  for (int64_t c = lane; c < C; c += 32) {
    float o = (to_f(xr[c]) - mean) * rstd * gamma[c];
    if (beta) o += beta[c];
    from_f(hr[c], o);
  }
  if (lane == 0) {
    mean_out[n] = mean;
    rstd_out[n] = rstd;
  }
}

// Backward: block b owns the rows [b * rpb, (b + 1) * rpb), warp w taking rows w, w + 8, ... of
// them (the next one prefetched).  dx per row.  Each lane owns the same columns of every row in
// the register layout, so it keeps its columns' sums of dh * xhat and dh in registers over the
// warp's rows, in row order; the block's partial is then the warps' sums added in warp order,
// through one shared-memory slice per warp.  part_g / part_b: [gridDim.x][C].  In a slice,
// column (k * 32 + l) * VN + i sits at word (k * VN + i) * 32 + l, so a warp's 32 lanes hit 32
// banks (S = KV * 32 * VN words per array).  Dynamic shared memory: 2 * (NT / 32) * S floats.
// the parameter-gradient sums of one lane, written into its warp's slice, then the block's
// partial row: the warps' slices added in warp order
template <int KV, int VN, int NT>
__device__ __forceinline__ void ln_block_partial(const float* ag, const float* ab, float* ln_slices, int64_t C,
                                                 float* __restrict__ part_g, float* __restrict__ part_b) {
  constexpr int64_t S = (int64_t)KV * 32 * VN;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  float* wg = ln_slices + (int64_t)wid * 2 * S;
  float* wb = wg + S;
#pragma unroll
  for (int j = 0; j < KV * VN; ++j) {
    wg[j * 32 + lane] = ag[j];
    wb[j * 32 + lane] = ab[j];
  }
  __syncthreads();
  for (int64_t c = threadIdx.x; c < C; c += NT) {
    const int64_t slot = ((c / (32 * VN)) * VN + c % VN) * 32 + (c / VN) % 32;
    float pg = 0.f, pb = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
      pg += ln_slices[(int64_t)w * 2 * S + slot];
      pb += ln_slices[(int64_t)w * 2 * S + S + slot];
    }
    part_g[(int64_t)blockIdx.x * C + c] = pg;
    part_b[(int64_t)blockIdx.x * C + c] = pb;
  }
}

// dx of one row in the register layout, and the row's terms added to the lane's parameter sums
template <typename T, int KV>
__device__ __forceinline__ void ln_bwd_row(const uint4* cd, const uint4* cx, const float* __restrict__ gamma,
                                           float mean, float rstd, int64_t C, int rms, float inv_c,
                                           T* __restrict__ dxr, float* ag, float* ab) {
  constexpr int VN = Vec<T>::N;
  const int lane = threadIdx.x & 31;
  float sg = 0.f, sgx = 0.f;
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int64_t c = ((int64_t)k * 32 + lane) * VN;
    if (c >= C) continue;
    float d[VN], xv[VN], g[VN];
    Vec<T>::unpack(cd[k], d);
    Vec<T>::unpack(cx[k], xv);
    load_param<VN>(gamma + c, g);
#pragma unroll
    for (int i = 0; i < VN; ++i) {
      const float xi = (xv[i] - mean) * rstd;
      const float gi = d[i] * g[i];
      ag[k * VN + i] += d[i] * xi;
      ab[k * VN + i] += d[i];
      sg += gi;
      sgx += gi * xi;
    }
  }
  const float mg = rms ? 0.f : warp_sum(sg) * inv_c;
  const float mgx = warp_sum(sgx) * inv_c;
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int64_t c = ((int64_t)k * 32 + lane) * VN;
    if (c >= C) continue;
    float d[VN], xv[VN], g[VN], o[VN];
    Vec<T>::unpack(cd[k], d);
    Vec<T>::unpack(cx[k], xv);
    load_param<VN>(gamma + c, g);
#pragma unroll
    for (int i = 0; i < VN; ++i) o[i] = rstd * (d[i] * g[i] - mg - (xv[i] - mean) * rstd * mgx);
    *reinterpret_cast<uint4*>(dxr + c) = Vec<T>::pack(o);
  }
}

template <typename T, int KV, int NT = lnb_threads<T, KV>()>
__global__ void __launch_bounds__(NT, 1) ln_bwd_vec_kernel(
    const T* __restrict__ dh, const T* __restrict__ x, const float* __restrict__ gamma,
    const float* __restrict__ mean_in, const float* __restrict__ rstd_in, int64_t N, int64_t C, int rms,
    T* __restrict__ dx, float* __restrict__ part_g, float* __restrict__ part_b, int64_t rpb) {
  griddep_wait();
  constexpr int VN = Vec<T>::N;
  extern __shared__ float ln_slices[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t r0 = (int64_t)blockIdx.x * rpb, r1 = r0 + rpb < N ? r0 + rpb : N;
  const float inv_c = 1.0f / (float)C;
  float ag[KV * VN], ab[KV * VN];
#pragma unroll
  for (int j = 0; j < KV * VN; ++j) ag[j] = ab[j] = 0.f;
  uint4 cd[KV], cx[KV], nd[KV], nx[KV];
  if (r0 + wid < r1) {
    load_row<T, KV>(dh + (r0 + wid) * C, C, lane, cd);
    load_row<T, KV>(x + (r0 + wid) * C, C, lane, cx);
  }
  for (int64_t n = r0 + wid; n < r1; n += NT / 32) {
    const int64_t nn = n + NT / 32;
    if (nn < r1) {
      load_row<T, KV>(dh + nn * C, C, lane, nd);
      load_row<T, KV>(x + nn * C, C, lane, nx);
    }
    ln_bwd_row<T, KV>(cd, cx, gamma, mean_in[n], rstd_in[n], C, rms, inv_c, dx + n * C, ag, ab);
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      cd[k] = nd[k];
      cx[k] = nx[k];
    }
  }
  ln_block_partial<KV, VN, NT>(ag, ab, ln_slices, C, part_g, part_b);
}

// ---- ln_f fused with the valid-row compaction (lmce_microstep_ln_compact) ----------------------
// Forward: warps stride over the original rows.  A warp reads the targets of its row's 32-row
// block, ranks the valid ones with a ballot, and for a valid row normalises x[n] straight into
// the compact head input: h[p], mean[p], rstd[p], y_c[p] = y[n], with p = block offset + rank
// (the input order kept); pos[n] = p, or -1 for an ignored row, whose x is never read.  The next
// row's rank is found, and its x loaded, while the current row is normalised.
__device__ __forceinline__ int64_t ln_compact_pos(const int32_t* __restrict__ y, int64_t N, int64_t V,
                                                  const int64_t* __restrict__ blk_off, int64_t n, int* yn) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (n & ~(int64_t)31) + lane;
  const int yt = r < N ? y[r] : -1;
  const bool v = r < N && yt >= 0 && (int64_t)yt < V;
  const unsigned bal = __ballot_sync(0xffffffffu, v);
  const int l = (int)(n & 31);
  *yn = __shfl_sync(0xffffffffu, yt, l);
  if (!((bal >> l) & 1u)) return -1;
  return blk_off[n >> 5] + __popc(bal & ((1u << l) - 1u));
}

template <typename T, int KV>
__global__ void __launch_bounds__(LN_T, KV <= 3 ? 3 : 2) ln_gather_fwd_kernel(
    const T* __restrict__ x, const int32_t* __restrict__ y, int64_t V, const int64_t* __restrict__ blk_off,
    const float* __restrict__ gamma, const float* __restrict__ beta, int64_t N, int64_t C, int rms, float eps,
    T* __restrict__ h, float* __restrict__ mean_out, float* __restrict__ rstd_out, int32_t* __restrict__ y_c,
    int32_t* __restrict__ pos, int64_t rows, unsigned* err) {
  griddep_wait();
  constexpr int VN = Vec<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * (LN_T / 32);
  const float inv_c = 1.0f / (float)C;
  int64_t n = (int64_t)blockIdx.x * (LN_T / 32) + (threadIdx.x >> 5);
  uint4 cur[KV], nxt[KV];
  int yc = 0, yx = 0;
  int64_t p = -1, pn = -1;
  if (n < N) {
    p = ln_compact_pos(y, N, V, blk_off, n, &yc);
    if (p >= 0 && !dcheck(p < rows, err, BS_COMPACT_POS)) p = -1;
    if (p >= 0) load_row<T, KV>(x + n * C, C, lane, cur);
  }
  for (; n < N; n += stride) {
    const int64_t nn = n + stride;
    if (nn < N) {
      pn = ln_compact_pos(y, N, V, blk_off, nn, &yx);
      if (pn >= 0 && !dcheck(pn < rows, err, BS_COMPACT_POS)) pn = -1;
      if (pn >= 0) load_row<T, KV>(x + nn * C, C, lane, nxt);   // in flight meanwhile
    }
    if (lane == 0) pos[n] = (int32_t)p;
    if (p >= 0) {
      float f[VN];
      float mean = 0.f;
      if (!rms) {
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
          Vec<T>::unpack(cur[k], f);
#pragma unroll
          for (int i = 0; i < VN; ++i) s += f[i];
        }
        mean = warp_sum(s) * inv_c;
      }
      float q = 0.f;
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        if (((int64_t)k * 32 + lane) * VN >= C) continue;
        Vec<T>::unpack(cur[k], f);
#pragma unroll
        for (int i = 0; i < VN; ++i) {
          const float d = f[i] - mean;
          q += d * d;
        }
      }
      const float rstd = 1.0f / sqrtf(warp_sum(q) * inv_c + eps);
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int64_t c = ((int64_t)k * 32 + lane) * VN;
        if (c >= C) continue;
        float g[VN], o[VN];
        Vec<T>::unpack(cur[k], f);
        load_param<VN>(gamma + c, g);
#pragma unroll
        for (int i = 0; i < VN; ++i) o[i] = (f[i] - mean) * rstd * g[i];
        if (beta) {
          load_param<VN>(beta + c, g);
#pragma unroll
          for (int i = 0; i < VN; ++i) o[i] += g[i];
        }
        *reinterpret_cast<uint4*>(h + p * C + c) = Vec<T>::pack(o);
      }
      if (lane == 0) {
        mean_out[p] = mean;
        rstd_out[p] = rstd;
        y_c[p] = yc;
      }
    }
#pragma unroll
    for (int k = 0; k < KV; ++k) cur[k] = nxt[k];
    p = pn;
    yc = yx;
  }
}

// Backward, scattered: block b owns the original rows [b * rpb, (b + 1) * rpb) as in
// ln_bwd_vec_kernel.  Row n with a compact position q < n_valid takes the head's dh of q, its own
// x and the statistics of q; any other row's dx (and row loss) is zero, and it adds nothing to
// the parameter sums.
template <typename T, int KV, int NT = lnb_threads<T, KV>()>
__global__ void __launch_bounds__(NT, 1) ln_bwd_scatter_kernel(
    const T* __restrict__ dh_c, const T* __restrict__ x, const float* __restrict__ gamma,
    const float* __restrict__ mean_c, const float* __restrict__ rstd_c, const int32_t* __restrict__ pos,
    int64_t n_valid, int64_t N, int64_t C, int rms, T* __restrict__ dx, float* __restrict__ part_g,
    float* __restrict__ part_b, int64_t rpb, const float* __restrict__ rl_c, float* __restrict__ row_loss,
    int64_t rows, unsigned* err) {
  griddep_wait();
  constexpr int VN = Vec<T>::N;
  extern __shared__ float ln_slices[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t r0 = (int64_t)blockIdx.x * rpb, r1 = r0 + rpb < N ? r0 + rpb : N;
  const float inv_c = 1.0f / (float)C;
  float ag[KV * VN], ab[KV * VN];
#pragma unroll
  for (int j = 0; j < KV * VN; ++j) ag[j] = ab[j] = 0.f;
  auto qof = [&](int64_t n) -> int64_t {
    const int64_t q = pos[n];
    return q >= 0 && q < n_valid && dcheck(q < rows, err, BS_SCATTER_POS) ? q : -1;
  };
  uint4 cd[KV], cx[KV], nd[KV], nx[KV];
  int64_t q = -1, qn = -1;
  if (r0 + wid < r1) {
    q = qof(r0 + wid);
    if (q >= 0) {
      load_row<T, KV>(dh_c + q * C, C, lane, cd);
      load_row<T, KV>(x + (r0 + wid) * C, C, lane, cx);
    }
  }
  for (int64_t n = r0 + wid; n < r1; n += NT / 32) {
    const int64_t nn = n + NT / 32;
    if (nn < r1) {
      qn = qof(nn);
      if (qn >= 0) {
        load_row<T, KV>(dh_c + qn * C, C, lane, nd);
        load_row<T, KV>(x + nn * C, C, lane, nx);
      }
    }
    if (q >= 0) {
      ln_bwd_row<T, KV>(cd, cx, gamma, mean_c[q], rstd_c[q], C, rms, inv_c, dx + n * C, ag, ab);
    } else {
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int64_t c = ((int64_t)k * 32 + lane) * VN;
        if (c < C) *reinterpret_cast<uint4*>(dx + n * C + c) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (row_loss && lane == 0) row_loss[n] = q >= 0 ? rl_c[q] : 0.f;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      cd[k] = nd[k];
      cx[k] = nx[k];
    }
    q = qn;
  }
  ln_block_partial<KV, VN, NT>(ag, ab, ln_slices, C, part_g, part_b);
}

template <typename T>
__global__ void __launch_bounds__(LN_T) ln_bwd_rows_kernel(const T* __restrict__ dh, const T* __restrict__ x,
                                                          const float* __restrict__ gamma,
                                                          const float* __restrict__ mean_in,
                                                          const float* __restrict__ rstd_in, int64_t N, int64_t C,
                                                          int rms, T* __restrict__ dx, float* __restrict__ part_g,
                                                          float* __restrict__ part_b, int64_t rpb) {
  griddep_wait();
  extern __shared__ float ln_slices[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t r0 = (int64_t)blockIdx.x * rpb, r1 = r0 + rpb < N ? r0 + rpb : N;
  const float inv_c = 1.0f / (float)C;
  for (int64_t i = threadIdx.x; i < 2 * (LN_T / 32) * C; i += LN_T) ln_slices[i] = 0.f;
  __syncthreads();
  float* wg = ln_slices + (int64_t)wid * 2 * C;
  float* wb = wg + C;
  for (int64_t n = r0 + wid; n < r1; n += LN_T / 32) {
    const float mean = mean_in[n], rstd = rstd_in[n];
    const T* dr = dh + n * C;
    const T* xr = x + n * C;
    float sg = 0.f, sgx = 0.f;
    for (int64_t c = lane; c < C; c += 32) {
      const float d = to_f(dr[c]);
      const float gi = d * gamma[c];
      const float xi = (to_f(xr[c]) - mean) * rstd;
      wg[c] += d * xi;
      wb[c] += d;
      sg += gi;
      sgx += gi * xi;
    }
    const float mg = rms ? 0.f : warp_sum(sg) * inv_c;
    const float mgx = warp_sum(sgx) * inv_c;
    for (int64_t c = lane; c < C; c += 32) {
      const float gi = to_f(dr[c]) * gamma[c];
      const float xi = (to_f(xr[c]) - mean) * rstd;
      from_f(dx[n * C + c], rstd * (gi - mg - xi * mgx));
    }
  }
  __syncthreads();
  for (int64_t c = threadIdx.x; c < C; c += LN_T) {
    float pg = 0.f, pb = 0.f;
#pragma unroll
    for (int w = 0; w < LN_T / 32; ++w) {
      pg += ln_slices[(int64_t)w * 2 * C + c];
      pb += ln_slices[(int64_t)w * 2 * C + C + c];
    }
    part_g[(int64_t)blockIdx.x * C + c] = pg;
    part_b[(int64_t)blockIdx.x * C + c] = pb;
  }
}

// dgamma[c] (+)= sum over blocks b of part_g[b][c], likewise dbeta: a block per 32 columns; warp w
// sums the blocks w, w + 32, ... with four independent running sums (block k into sum
// (k / 32) mod 4), then warp 0 adds the 32 warps' results in warp order: a fixed order.
constexpr int LNR_T = 1024;
__global__ void __launch_bounds__(LNR_T) ln_param_reduce_kernel(const float* __restrict__ part_g,
                                                               const float* __restrict__ part_b, int64_t nblk,
                                                               int64_t C, int accumulate, float* __restrict__ dgamma,
                                                               float* __restrict__ dbeta) {
  griddep_wait();
  constexpr int NW = LNR_T / 32;
  __shared__ float sg[NW][32], sb[NW][32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t c = (int64_t)blockIdx.x * 32 + lane;
  float g[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
  if (c < C) {
    int64_t k = wid;
    for (; k + 3 * NW < nblk; k += 4 * NW) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        g[u] += part_g[(k + u * NW) * C + c];
        b[u] += part_b[(k + u * NW) * C + c];
      }
    }
    for (int u = 0; k < nblk; k += NW, ++u) {
      g[u] += part_g[k * C + c];
      b[u] += part_b[k * C + c];
    }
  }
  sg[wid][lane] = (g[0] + g[1]) + (g[2] + g[3]);
  sb[wid][lane] = (b[0] + b[1]) + (b[2] + b[3]);
  __syncthreads();
  if (wid == 0 && c < C) {
    float tg = 0.f, tb = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      tg += sg[w][lane];
      tb += sb[w][lane];
    }
    dgamma[c] = accumulate ? dgamma[c] + tg : tg;
    if (dbeta) dbeta[c] = accumulate ? dbeta[c] + tb : tb;
  }
}

// the register layout's words per lane, or 0 when a row does not fit it (C not a multiple of
// VN, wider than 32 * LN_MAXV * VN, or a pointer not 16-byte aligned)
template <typename T>
int ln_kv(const LnArgs& a, const void* rows_in, const void* rows_out) {
  constexpr int VN = Vec<T>::N;
  const uintptr_t al = (uintptr_t)rows_in | (uintptr_t)rows_out | (uintptr_t)a.x | (uintptr_t)a.gamma |
                       (uintptr_t)a.beta;
  if (a.C % VN != 0 || (al & 15) != 0) return 0;
  const int64_t kv = (a.C + 32 * VN - 1) / (32 * VN);
  return kv <= LN_MAXV ? (int)kv : 0;
}

constexpr int LN_FWD_BLOCKS_PER_SM = 4;

template <typename T, int KV>
void launch_fwd_vec(const LnArgs& a, cudaStream_t st) {
  int64_t blocks = (a.N + LN_T / 32 - 1) / (LN_T / 32);
  if (blocks > 152 * LN_FWD_BLOCKS_PER_SM) blocks = 152 * LN_FWD_BLOCKS_PER_SM;   // warps loop over rows
  launch_pdl(ln_fwd_vec_kernel<T, KV>, dim3((unsigned)blocks), dim3(LN_T), 0, st, (const T*)a.x, a.gamma, a.beta, a.N, a.C,
             (int)a.rms, a.eps, (T*)a.h, a.mean, a.rstd);
}

template <typename T, int KV>
cudaError_t launch_bwd_vec(const LnArgs& a, int64_t nblk, int64_t rpb, cudaStream_t st) {
  const size_t smem = sizeof(float) * 2 * (lnb_threads<T, KV>() / 32) * (size_t)KV * 32 * Vec<T>::N;
  cudaError_t e = max_dyn_smem((const void*)ln_bwd_vec_kernel<T, KV>, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(ln_bwd_vec_kernel<T, KV>, dim3((unsigned)nblk), dim3(lnb_threads<T, KV>()), smem, st, (const T*)a.dh,
                    (const T*)a.x, a.gamma, (const float*)a.mean, (const float*)a.rstd, a.N, a.C, (int)a.rms, (T*)a.dx,
                    a.part_g, a.part_b, rpb);
}

template <typename T, int KV>
void launch_gather_fwd(const LnArgs& a, const int32_t* y, int64_t V, const CompactScratch& cs, cudaStream_t st) {
  int64_t blocks = (a.N + LN_T / 32 - 1) / (LN_T / 32);
  if (blocks > 152 * LN_FWD_BLOCKS_PER_SM) blocks = 152 * LN_FWD_BLOCKS_PER_SM;   // warps loop over rows
  launch_pdl(ln_gather_fwd_kernel<T, KV>, dim3((unsigned)blocks), dim3(LN_T), 0, st, (const T*)a.x, y, V,
             (const int64_t*)cs.blk_off, a.gamma, a.beta, a.N, a.C, (int)a.rms, a.eps, (T*)a.h, a.mean, a.rstd, cs.y_c,
             cs.pos, cs.rows, cs.err);
}

template <typename T, int KV>
cudaError_t launch_bwd_scatter(const LnArgs& a, const CompactScratch& cs, int64_t n_valid, float* row_loss,
                               int64_t nblk, int64_t rpb, cudaStream_t st) {
  const size_t smem = sizeof(float) * 2 * (lnb_threads<T, KV>() / 32) * (size_t)KV * 32 * Vec<T>::N;
  cudaError_t e = max_dyn_smem((const void*)ln_bwd_scatter_kernel<T, KV>, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(ln_bwd_scatter_kernel<T, KV>, dim3((unsigned)nblk), dim3(lnb_threads<T, KV>()), smem, st,
                    (const T*)a.dh, (const T*)a.x, a.gamma, (const float*)a.mean, (const float*)a.rstd,
                    (const int32_t*)cs.pos, n_valid, a.N, a.C, (int)a.rms, (T*)a.dx, a.part_g, a.part_b, rpb,
                    (const float*)cs.rl_c, row_loss, cs.rows, cs.err);
}

template <typename T>
cudaError_t ln_gather_forward_t(const LnArgs& a, const int32_t* y, int64_t V, const CompactScratch& cs, Launch& L) {
  L.begin(K_LN);
  switch (ln_kv<T>(a, a.h, a.dx)) {
    case 1: launch_gather_fwd<T, 1>(a, y, V, cs, L.st); break;
    case 2: launch_gather_fwd<T, 2>(a, y, V, cs, L.st); break;
    case 3: launch_gather_fwd<T, 3>(a, y, V, cs, L.st); break;
    case 4: launch_gather_fwd<T, 4>(a, y, V, cs, L.st); break;
    case 5: launch_gather_fwd<T, 5>(a, y, V, cs, L.st); break;
    default: launch_gather_fwd<T, 6>(a, y, V, cs, L.st); break;
  }
  L.end();
  return cudaGetLastError();
}

template <typename T>
cudaError_t ln_backward_scatter_t(const LnArgs& a, const CompactScratch& cs, int64_t n_valid, float* row_loss,
                                  Launch& L) {
  const int64_t nblk = ln_blocks(a.N);
  const int64_t rpb = ln_rows_per_block(a.N);
  cudaError_t e;
  L.begin(K_LN);
  switch (ln_kv<T>(a, a.dh, a.dx)) {
    case 1: e = launch_bwd_scatter<T, 1>(a, cs, n_valid, row_loss, nblk, rpb, L.st); break;
    case 2: e = launch_bwd_scatter<T, 2>(a, cs, n_valid, row_loss, nblk, rpb, L.st); break;
    case 3: e = launch_bwd_scatter<T, 3>(a, cs, n_valid, row_loss, nblk, rpb, L.st); break;
    case 4: e = launch_bwd_scatter<T, 4>(a, cs, n_valid, row_loss, nblk, rpb, L.st); break;
    case 5: e = launch_bwd_scatter<T, 5>(a, cs, n_valid, row_loss, nblk, rpb, L.st); break;
    default: e = launch_bwd_scatter<T, 6>(a, cs, n_valid, row_loss, nblk, rpb, L.st); break;
  }
  L.end();
  if (e != cudaSuccess) return e;
  L.begin(K_LN);
  launch_pdl(ln_param_reduce_kernel, dim3((unsigned)((a.C + 31) / 32)), dim3(LNR_T), 0, L.st, (const float*)a.part_g,
             (const float*)a.part_b, nblk, a.C, (int)a.accumulate, a.dgamma, a.dbeta);
  L.end();
  return cudaGetLastError();
}

template <typename T>
cudaError_t ln_forward_t(const LnArgs& a, Launch& L) {
  const int kv = ln_kv<T>(a, a.x, a.h);
  L.begin(K_LN);
  switch (kv) {
    case 1: launch_fwd_vec<T, 1>(a, L.st); break;
    case 2: launch_fwd_vec<T, 2>(a, L.st); break;
    case 3: launch_fwd_vec<T, 3>(a, L.st); break;
    case 4: launch_fwd_vec<T, 4>(a, L.st); break;
    case 5: launch_fwd_vec<T, 5>(a, L.st); break;
    case 6: launch_fwd_vec<T, 6>(a, L.st); break;
    default:
      ln_fwd_rows_kernel<T><<<(unsigned)((a.N + LN_T / 32 - 1) / (LN_T / 32)), LN_T, 0, L.st>>>(
          (const T*)a.x, a.gamma, a.beta, a.N, a.C, a.rms, a.eps, (T*)a.h, a.mean, a.rstd);
  }
  L.end();
  return cudaGetLastError();
}

template <typename T>
cudaError_t ln_backward_t(const LnArgs& a, Launch& L) {
  const int64_t nblk = ln_blocks(a.N);
  const int64_t rpb = ln_rows_per_block(a.N);
  const int kv = ln_kv<T>(a, a.dh, a.dx);
  cudaError_t e = cudaSuccess;
  if (kv == 0) {
    const size_t smem = sizeof(float) * 2 * (LN_T / 32) * (size_t)a.C;
    e = max_dyn_smem((const void*)ln_bwd_rows_kernel<T>, (int)smem);
    if (e != cudaSuccess) return e;
    L.begin(K_LN);
    ln_bwd_rows_kernel<T><<<(unsigned)nblk, LN_T, smem, L.st>>>((const T*)a.dh, (const T*)a.x, a.gamma, a.mean,
                                                                a.rstd, a.N, a.C, a.rms, (T*)a.dx, a.part_g,
                                                                a.part_b, rpb);
    L.end();
  } else {
    L.begin(K_LN);
    switch (kv) {
      case 1: e = launch_bwd_vec<T, 1>(a, nblk, rpb, L.st); break;
      case 2: e = launch_bwd_vec<T, 2>(a, nblk, rpb, L.st); break;
      case 3: e = launch_bwd_vec<T, 3>(a, nblk, rpb, L.st); break;
      case 4: e = launch_bwd_vec<T, 4>(a, nblk, rpb, L.st); break;
      case 5: e = launch_bwd_vec<T, 5>(a, nblk, rpb, L.st); break;
      default: e = launch_bwd_vec<T, 6>(a, nblk, rpb, L.st); break;
    }
    L.end();
    if (e != cudaSuccess) return e;
  }
  L.begin(K_LN);
  launch_pdl(ln_param_reduce_kernel, dim3((unsigned)((a.C + 31) / 32)), dim3(LNR_T), 0, L.st, (const float*)a.part_g,
             (const float*)a.part_b, nblk, a.C, (int)a.accumulate, a.dgamma, a.dbeta);
  L.end();
  return cudaGetLastError();
}

}  // namespace

// rows per backward block and the blocks that covers (at most LN_BWD_GRID; a function of N alone,
// so the parameter gradients are summed in the same order on every call)
int64_t ln_rows_per_block(int64_t N) { return N > 0 ? (N + LN_BWD_GRID - 1) / LN_BWD_GRID : 1; }
int64_t ln_blocks(int64_t N) { return (N + ln_rows_per_block(N) - 1) / ln_rows_per_block(N); }
int64_t ln_part_rows() { return LN_BWD_GRID; }

cudaError_t ln_forward(const LnArgs& a, Launch& L) {
  if (a.N == 0) return cudaSuccess;
  return a.bf16 ? ln_forward_t<__nv_bfloat16>(a, L) : ln_forward_t<float>(a, L);
}

cudaError_t ln_backward(const LnArgs& a, Launch& L) {
  if (a.N == 0) return cudaSuccess;
  return a.bf16 ? ln_backward_t<__nv_bfloat16>(a, L) : ln_backward_t<float>(a, L);
}

bool ln_compact_fusable(const LnArgs& a) {
  return a.bf16 ? ln_kv<__nv_bfloat16>(a, a.h, a.dx) > 0 && ln_kv<__nv_bfloat16>(a, a.dh, a.dx) > 0
                : ln_kv<float>(a, a.h, a.dx) > 0 && ln_kv<float>(a, a.dh, a.dx) > 0;
}

cudaError_t ln_gather_forward(const LnArgs& a, const int32_t* targets, int64_t V, const CompactScratch& cs, Launch& L) {
  if (a.N == 0) return cudaSuccess;
  return a.bf16 ? ln_gather_forward_t<__nv_bfloat16>(a, targets, V, cs, L)
                : ln_gather_forward_t<float>(a, targets, V, cs, L);
}

cudaError_t ln_backward_scatter(const LnArgs& a, const CompactScratch& cs, int64_t n_valid, float* row_loss, Launch& L) {
  if (a.N == 0) return cudaSuccess;
  return a.bf16 ? ln_backward_scatter_t<__nv_bfloat16>(a, cs, n_valid, row_loss, L)
                : ln_backward_scatter_t<float>(a, cs, n_valid, row_loss, L);
}

}  // namespace lmce
