// C-ABI of the lmce library: handle, argument checks, status codes, dispatch, and the
// fixed-order loss/count reduction shared by both compute paths.
#include <stdlib.h>
#include <string.h>
#include <math.h>

#include <mutex>
#include <new>

#include "lmce.h"

#include "lmce_internal.cuh"

namespace lmce {
namespace {


// One block sums the per-block partials of a micro-step in a fixed order (each thread a
// fixed strided subset, then a fixed tree), then updates the step accumulators.
// The gradient scale of this micro-step is set here:
//   global norm    : s = 1 / global_valid
//   micro-mean norm: s = 1 / (valid_k * G), 0 for a micro-step without valid targets
// ("Multi-GPU calculation of gradients for accelerated training", section "Gradient
// accumulation averages across micro-steps").
static_assert(LMCE_NORM_GLOBAL == 0 && LMCE_NORM_MICRO_MEAN == 1, "finish_block's norm codes");

__global__ void __launch_bounds__(FIN_T) finish_kernel(const double* __restrict__ part_loss,
                                                       const int* __restrict__ part_cnt,
                                                       const unsigned* __restrict__ part_err,
                                                       int64_t nparts, int norm, int G,
                                                       long long global_valid, DevAcc* acc, int mode) {
  finish_block(part_loss, part_cnt, part_err, nparts, norm, G, global_valid, acc, mode);
}

// Sum of squares of n floats to float64 accuracy without float64 arithmetic per element (a
// GB300 runs float64 at a small fraction of its float32 rate): each square is split exactly
// into x*x + fma(x, x, -x*x), and a thread accumulates its terms as a double-single pair (S, E)
// with Knuth's TwoSum, in round-to-nearest intrinsics the compiler may not contract.  Block b
// takes the fixed range [b*per, (b+1)*per) in 16-byte steps, each thread a fixed strided subset
// in order; the threads' S + E are added in float64 in a fixed-shape tree, and the block that
// finishes last (a ticket, no waiting) adds the blocks' partials in block order.  The same order
// on every call.
struct DSum {
  float S = 0.f, E = 0.f;
  __device__ __forceinline__ void add_sq(float x) {
    const float p = __fmul_rn(x, x);
    const float e = __fmaf_rn(x, x, -p);             // x*x - p, exactly
    const float t = __fadd_rn(S, p);
    const float z = __fsub_rn(t, S);
    const float err = __fadd_rn(__fsub_rn(S, __fsub_rn(t, z)), __fsub_rn(p, z));   // (S + p) - t, exactly
    E = __fadd_rn(E, __fadd_rn(err, e));
    S = t;
  }
};
constexpr int SQ_T = 256, SQ_BLOCKS = 608;   // 4 blocks per SM of a 152-SM GB300
__global__ void __launch_bounds__(SQ_T) sumsq_part_kernel(const float* __restrict__ x, int64_t n, int64_t per,
                                                         double* __restrict__ part, unsigned* ticket) {
  __shared__ double sh[SQ_T];
  const int64_t b0 = (int64_t)blockIdx.x * per, b1 = b0 + per < n ? b0 + per : n;
  DSum d;
  if ((((uintptr_t)x) & 15) == 0 && (b0 & 3) == 0) {
    const int64_t v0 = b0 / 4, v1 = b1 / 4;   // whole float4 groups of the range
    const float4* x4 = reinterpret_cast<const float4*>(x);
    // eight loads in flight per thread, then their terms in the same order as a plain strided loop
    int64_t i = v0 + threadIdx.x;
    for (; i + 7 * SQ_T < v1; i += 8 * SQ_T) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = x4[i + u * SQ_T];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        d.add_sq(v[u].x);
        d.add_sq(v[u].y);
        d.add_sq(v[u].z);
        d.add_sq(v[u].w);
      }
    }
    for (; i < v1; i += SQ_T) {
      const float4 v = x4[i];
      d.add_sq(v.x);
      d.add_sq(v.y);
      d.add_sq(v.z);
      d.add_sq(v.w);
    }
    for (int64_t i = v1 * 4 + threadIdx.x; i < b1; i += SQ_T) d.add_sq(x[i]);
  } else {
    for (int64_t i = b0 + threadIdx.x; i < b1; i += SQ_T) d.add_sq(x[i]);
  }
  sh[threadIdx.x] = (double)d.S + (double)d.E;
  __syncthreads();
  for (int o = SQ_T / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) sh[threadIdx.x] += sh[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) part[blockIdx.x] = sh[0];
  // the block that finishes last adds the blocks' partials in block order into part[gridDim.x]
  if (!last_block(ticket)) return;
  double acc = 0.0;
  for (int i = threadIdx.x; i < (int)gridDim.x; i += SQ_T) acc += __ldcg(part + i);
  sh[threadIdx.x] = acc;
  __syncthreads();
  for (int o = SQ_T / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) sh[threadIdx.x] += sh[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) part[gridDim.x] = sh[0];
}

// One AdamW step over the tied matrix, each element read and written once (30 bytes: dW, p, m, v
// in; p, m, v and the bf16 copy of p out).  Decoupled weight decay and bias-corrected moments as
// torch.optim.AdamW, with the betas, eps and decay of "How I trained my own GPT-2 124M",
// section 6 "Implementing the Optimizer"; the update is one pass over the whole state, the fused
// form of "Making LLM training fast", section "The optimizer step".
struct AdamCoef {
  float clip, b1, omb1, b2, omb2, decay, step_size, sqrt_bc2, eps;
};
__device__ __forceinline__ void adamw_elem(float g, float& p, float& m, float& v, const AdamCoef& k) {
  g = k.clip * g;
  m = k.b1 * m + k.omb1 * g;
  v = k.b2 * v + k.omb2 * (g * g);
  const float den = sqrtf(v) / k.sqrt_bc2 + k.eps;
  p = p * k.decay - k.step_size * (m / den);
}
constexpr int AW_T = 256, AW_BLOCKS = 1216;   // 8 blocks per SM of a 152-SM GB300
__global__ void __launch_bounds__(AW_T) adamw_kernel(const float* __restrict__ g, float* __restrict__ p,
                                                    float* __restrict__ m, float* __restrict__ v,
                                                    __nv_bfloat16* __restrict__ w, int64_t n, int vec,
                                                    AdamCoef k) {
  const int64_t stride = (int64_t)gridDim.x * AW_T;
  int64_t i0 = (int64_t)blockIdx.x * AW_T + threadIdx.x;
  if (vec) {
    const int64_t n4 = n / 4;
    const float4* g4 = reinterpret_cast<const float4*>(g);
    float4* p4 = reinterpret_cast<float4*>(p);
    float4* m4 = reinterpret_cast<float4*>(m);
    float4* v4 = reinterpret_cast<float4*>(v);
    for (int64_t i = i0; i < n4; i += stride) {
      const float4 gg = __ldcs(g4 + i);
      float4 pp = __ldcs(p4 + i), mm = __ldcs(m4 + i), vv = __ldcs(v4 + i);
      adamw_elem(gg.x, pp.x, mm.x, vv.x, k);
      adamw_elem(gg.y, pp.y, mm.y, vv.y, k);
      adamw_elem(gg.z, pp.z, mm.z, vv.z, k);
      adamw_elem(gg.w, pp.w, mm.w, vv.w, k);
      __stcs(p4 + i, pp);
      __stcs(m4 + i, mm);
      __stcs(v4 + i, vv);
      if (w) {   // the next forward reads W: a plain store leaves it in L2
        const __nv_bfloat162 lo = __floats2bfloat162_rn(pp.x, pp.y), hi = __floats2bfloat162_rn(pp.z, pp.w);
        uint2 u;
        u.x = *reinterpret_cast<const unsigned*>(&lo);
        u.y = *reinterpret_cast<const unsigned*>(&hi);
        reinterpret_cast<uint2*>(w)[i] = u;
      }
    }
    i0 += n4 * 4;   // the ragged tail, fewer than 4 elements
    for (int64_t i = i0; i < n; i += stride) {
      float pp = p[i], mm = m[i], vv = v[i];
      adamw_elem(g[i], pp, mm, vv, k);
      p[i] = pp;
      m[i] = mm;
      v[i] = vv;
      if (w) w[i] = __float2bfloat16_rn(pp);
    }
    return;
  }
  for (int64_t i = i0; i < n; i += stride) {
    float pp = p[i], mm = m[i], vv = v[i];
    adamw_elem(g[i], pp, mm, vv, k);
    p[i] = pp;
    m[i] = mm;
    v[i] = vv;
    if (w) w[i] = __float2bfloat16_rn(pp);
  }
}

}  // namespace

cudaError_t finish_load_kernel() {
  cudaFuncAttributes fa;
  return cudaFuncGetAttributes(&fa, finish_kernel);
}

cudaError_t launch_finish(const StepArgs& a, const Scratch& s, int64_t nparts, Launch& L, int mode) {
  L.begin(K_FINISH);
  finish_kernel<<<1, FIN_T, 0, L.st>>>(s.part_loss, s.part_cnt, s.part_err, nparts, a.norm, a.G,
                                       (long long)a.global_valid, s.acc, mode);
  L.end();
  return cudaGetLastError();
}

}  // namespace lmce

namespace lmce {

cudaError_t max_dyn_smem(const void* func, int bytes) {
  // a fixed table (no heap use: the allocation-free entry point goes through here too); when it
  // is full the attribute is simply set on every call
  struct Entry {
    int dev;
    const void* func;
    int bytes;
  };
  constexpr int CAP = 256;
  static std::mutex mu;
  static Entry tab[CAP];
  static int used = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i) {
    Entry& x = tab[i];
    if (x.dev == dev && x.func == func) {
      if (x.bytes >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e == cudaSuccess) x.bytes = bytes;
      return e;
    }
  }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && used < CAP) tab[used++] = {dev, func, bytes};
  return e;
}

}  // namespace lmce

using namespace lmce;

struct lmce_handle {
  lmce_config cfg;
  float* dW;
  int device;
  int path;            // resolved: LMCE_PATH_SIMT, LMCE_PATH_TCGEN05, LMCE_PATH_TCGEN05_TWO_PASS or
                       // LMCE_PATH_TCGEN05_RECOMPUTE
  Scratch sc;
  DevAcc* host_acc;    // pinned
  bool first;          // next micro-step writes dW instead of adding (unless LMCE_ACCUMULATE_FROM_START)
  double* sumsq_part;  // lmce_dw_sumsq: per-block float64 partials, then the result
  CompactScratch cs;   // lmce_microstep_compact (LMCE_COMPACT_VALID_ROWS), else all null
  struct {             // lmce_microstep_ln (LMCE_FINAL_NORM), else all null
    void* h;           // [max_N, C] dtype: ln_f(x), the head's input
    void* dh;          // [max_N, C] dtype: the head's dh
    float* mean;       // [max_N]
    float* rstd;       // [max_N]
    float* part;       // [2][ln_part_rows()][C]
  } ln;
  int64_t test_stall_ns;  // lmce_test_stall_next_microstep: armed for the next micro-step, then cleared
  int attempted;       // micro-steps accepted since create/finalize
  int64_t launches;
  Prof prof;
};

static int check_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return LMCE_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess)
    return LMCE_ERR_CUDA;
  if (major != 10 || minor != 3) return LMCE_ERR_ARCH;
  return LMCE_OK;
}

static void free_scratch(lmce_handle* h) {
  cudaFree(h->sc.lse);
  cudaFree(h->sc.part_loss);
  cudaFree(h->sc.part_cnt);
  cudaFree(h->sc.part_err);
  cudaFree(h->sc.acc);
  cudaFree(h->sc.ticket);
  cudaFree(h->sc.tc_part_m);
  cudaFree(h->sc.tc_part_l);
  cudaFree(h->sc.tc_zt);
  cudaFree(h->sc.tc_part);
  cudaFree(h->sc.tc_part_lm);
  cudaFree(h->sc.tc_tile_flag);
  cudaFree(h->sc.rep_part);
  cudaFree(h->sc.rep_ticket);
  cudaFree(h->sc.tc_p);
  cudaFree(h->sc.tc_mref);
  cudaFree(h->sc.tc_hs);
  cudaFree(h->sc.tc_kmap);
  cudaFree(h->sumsq_part);
  h->sumsq_part = nullptr;
  cudaFree(h->cs.h_c);
  cudaFree(h->cs.dh_c);
  cudaFree(h->cs.y_c);
  cudaFree(h->cs.rl_c);
  cudaFree(h->cs.pos);
  cudaFree(h->cs.blk_cnt);
  cudaFree(h->cs.blk_err);
  cudaFree(h->cs.blk_off);
  cudaFree(h->cs.total);
  cudaFreeHost(h->cs.host_total);
  h->cs = CompactScratch{};
  cudaFree(h->ln.h);
  cudaFree(h->ln.dh);
  cudaFree(h->ln.mean);
  cudaFree(h->ln.rstd);
  cudaFree(h->ln.part);
  h->ln = {};
  if (h->host_acc) cudaFreeHost(h->host_acc);
  memset(&h->sc, 0, sizeof(h->sc));
  h->host_acc = nullptr;
}

extern "C" int lmce_create(const lmce_config* cfg, float* dW, lmce_handle** out) {
  if (!cfg || !dW || !out) return LMCE_ERR_ARG;
  *out = nullptr;
  if (cfg->C <= 0 || cfg->V <= 0 || cfg->max_N < 0 || cfg->grad_accum_steps < 1) return LMCE_ERR_ARG;
  if (cfg->C > (1 << 20) || cfg->V > (1LL << 31) || cfg->max_N > (1LL << 31)) return LMCE_ERR_ARG;
  if (cfg->dtype != LMCE_BF16 && cfg->dtype != LMCE_FP32) return LMCE_ERR_ARG;
  if (cfg->norm != LMCE_NORM_GLOBAL && cfg->norm != LMCE_NORM_MICRO_MEAN) return LMCE_ERR_ARG;
  if (cfg->path < LMCE_PATH_AUTO || cfg->path > LMCE_PATH_TCGEN05_RECOMPUTE) return LMCE_ERR_ARG;
  if (cfg->flags & ~(LMCE_ACCUMULATE_FROM_START | LMCE_COMPACT_VALID_ROWS | LMCE_FINAL_NORM)) return LMCE_ERR_ARG;
  const bool tc_ok = tc_supported(cfg->C, cfg->V, cfg->dtype == LMCE_BF16);
  const bool simt_ok = cfg->C <= 2048;
  int path;
  if (cfg->path == LMCE_PATH_TCGEN05 || cfg->path == LMCE_PATH_TCGEN05_TWO_PASS ||
      cfg->path == LMCE_PATH_TCGEN05_RECOMPUTE) {
    if (!tc_ok) return LMCE_ERR_ARG;
    path = cfg->path;
  } else if (cfg->path == LMCE_PATH_SIMT) {
    if (!simt_ok) return LMCE_ERR_ARG;
    path = LMCE_PATH_SIMT;
  } else {
    if (tc_ok) path = LMCE_PATH_TCGEN05;
    else if (simt_ok) path = LMCE_PATH_SIMT;
    else return LMCE_ERR_ARG;
  }
  int dev = 0;
  int st = check_device(&dev);
  if (st != LMCE_OK) return st;
  lmce_handle* h = new (std::nothrow) lmce_handle();
  if (!h) return LMCE_ERR_CUDA;
  h->cfg = *cfg;
  h->dW = dW;
  h->device = dev;
  h->path = path;
  h->first = true;
  const int64_t maxN = cfg->max_N > 0 ? cfg->max_N : 1;
  int64_t parts = simt_parts(maxN);
  int64_t tp = tc_parts(maxN);
  if (tp > parts) parts = tp;
  h->sc.max_parts = parts;
  bool ok = cudaMalloc(&h->sc.lse, sizeof(float) * maxN) == cudaSuccess &&
            cudaMalloc(&h->sc.part_loss, sizeof(double) * parts) == cudaSuccess &&
            cudaMalloc(&h->sc.part_cnt, sizeof(int) * parts) == cudaSuccess &&
            cudaMalloc(&h->sc.part_err, sizeof(unsigned) * parts) == cudaSuccess &&
            cudaMalloc(&h->sc.acc, sizeof(DevAcc)) == cudaSuccess &&
            cudaMalloc(&h->sc.ticket, 2 * sizeof(unsigned)) == cudaSuccess &&
            cudaMemset(h->sc.ticket, 0, 2 * sizeof(unsigned)) == cudaSuccess &&
            cudaMallocHost(&h->host_acc, sizeof(DevAcc)) == cudaSuccess &&
            cudaMemset(h->sc.acc, 0, sizeof(DevAcc)) == cudaSuccess;
  if (ok && path != LMCE_PATH_SIMT) {
    const size_t slices = sizeof(float) * (size_t)TC_MAX_SPLIT * (size_t)maxN;
    const size_t tiles = (size_t)(maxN + TC_TILE_ROWS - 1) / TC_TILE_ROWS;
    ok = cudaMalloc(&h->sc.tc_part_m, slices) == cudaSuccess && cudaMalloc(&h->sc.tc_part_l, slices) == cudaSuccess &&
         cudaMalloc(&h->sc.tc_zt, sizeof(float) * maxN) == cudaSuccess &&
         cudaMalloc(&h->sc.tc_part, tc_part_bytes(cfg->C)) == cudaSuccess &&
         cudaMalloc(&h->sc.tc_part_lm, tc_part_lm_bytes()) == cudaSuccess &&
         cudaMalloc(&h->sc.tc_tile_flag, sizeof(unsigned) * tiles) == cudaSuccess &&
         cudaMemset(h->sc.tc_tile_flag, 0, sizeof(unsigned) * tiles) == cudaSuccess &&
         cudaMalloc(&h->sc.rep_part, sizeof(float) * simt_repair_part_floats(cfg->C)) == cudaSuccess &&
         cudaMalloc(&h->sc.rep_ticket, sizeof(unsigned) * tiles * (TC_TILE_ROWS / 16)) == cudaSuccess &&
         cudaMemset(h->sc.rep_ticket, 0, sizeof(unsigned) * tiles * (TC_TILE_ROWS / 16)) == cudaSuccess;
  }
  if (ok && path == LMCE_PATH_TCGEN05) {
    // the stored exponentials of the dW pass: p [max_N][Vp], and per segment copy the row
    // references and the scaled rows of h; the per-row pass defines every element it reads
    const int64_t vp = tc_p_cols(cfg->V), np = tc_ver_rows(maxN);
    const size_t ttiles = (size_t)(maxN + TC_TILE_ROWS - 1) / TC_TILE_ROWS;
    const bool got = cudaMalloc(&h->sc.tc_p, sizeof(uint16_t) * (size_t)maxN * (size_t)vp) == cudaSuccess &&
                     cudaMalloc(&h->sc.tc_mref, sizeof(float) * (size_t)TC_MAX_VER * (size_t)np) == cudaSuccess &&
                     cudaMalloc(&h->sc.tc_hs, sizeof(uint16_t) * (size_t)TC_MAX_VER * (size_t)np * (size_t)cfg->C) ==
                         cudaSuccess &&
                     cudaMalloc(&h->sc.tc_kmap, ttiles * (size_t)(vp / 256)) == cudaSuccess;
    h->sc.tc_p_rows = maxN;
    if (!got) {
      // not enough device memory for the N x V scratch: LMCE_PATH_AUTO falls back to recomputing
      // the logits in the dW pass; an explicit LMCE_PATH_TCGEN05 reports the failure
      cudaFree(h->sc.tc_p);
      cudaFree(h->sc.tc_mref);
      cudaFree(h->sc.tc_hs);
      cudaFree(h->sc.tc_kmap);
      h->sc.tc_p = nullptr;
      h->sc.tc_mref = nullptr;
      h->sc.tc_hs = nullptr;
      h->sc.tc_kmap = nullptr;
      h->sc.tc_p_rows = 0;
      (void)cudaGetLastError();   // the failed allocation's error is not sticky; clear it
      if (cfg->path == LMCE_PATH_AUTO) h->path = LMCE_PATH_TCGEN05_RECOMPUTE;
      else ok = false;
    }
  }
  ok = ok && cudaMalloc(&h->sumsq_part, sizeof(double) * (SQ_BLOCKS + 1)) == cudaSuccess;
  if (ok && (cfg->flags & LMCE_COMPACT_VALID_ROWS)) {
    const size_t rows = (size_t)maxN * (size_t)cfg->C * (cfg->dtype == LMCE_BF16 ? 2 : 4);
    const size_t nb = (size_t)compact_blocks(maxN);
    CompactScratch& q = h->cs;
    ok = cudaMalloc(&q.h_c, rows) == cudaSuccess && cudaMalloc(&q.dh_c, rows) == cudaSuccess &&
         cudaMalloc(&q.y_c, sizeof(int32_t) * maxN) == cudaSuccess &&
         cudaMalloc(&q.rl_c, sizeof(float) * maxN) == cudaSuccess &&
         cudaMalloc(&q.pos, sizeof(int32_t) * maxN) == cudaSuccess &&
         cudaMalloc(&q.blk_cnt, sizeof(int) * nb) == cudaSuccess &&
         cudaMalloc(&q.blk_err, sizeof(unsigned) * nb) == cudaSuccess &&
         cudaMalloc(&q.blk_off, sizeof(int64_t) * nb) == cudaSuccess &&
         cudaMalloc(&q.total, sizeof(int64_t)) == cudaSuccess &&
         cudaMallocHost(&q.host_total, sizeof(int64_t)) == cudaSuccess &&
         // defined contents for rows a wrong n_valid would read: zero rows, targets -1
         cudaMemset(q.h_c, 0, rows) == cudaSuccess && cudaMemset(q.y_c, 0xff, sizeof(int32_t) * maxN) == cudaSuccess;
    q.rows = maxN;
    q.err = &h->sc.acc->err;
  }
  if (ok && (cfg->flags & LMCE_FINAL_NORM)) {
    const size_t rows = (size_t)maxN * (size_t)cfg->C * (cfg->dtype == LMCE_BF16 ? 2 : 4);
    ok = cudaMalloc(&h->ln.h, rows) == cudaSuccess && cudaMalloc(&h->ln.dh, rows) == cudaSuccess &&
         cudaMalloc(&h->ln.mean, sizeof(float) * maxN) == cudaSuccess &&
         cudaMalloc(&h->ln.rstd, sizeof(float) * maxN) == cudaSuccess &&
         cudaMalloc(&h->ln.part, sizeof(float) * 2 * (size_t)ln_part_rows() * (size_t)cfg->C) == cudaSuccess;
  }
  ok = ok && cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    free_scratch(h);
    delete h;
    return LMCE_ERR_CUDA;
  }
  *out = h;
  return LMCE_OK;
}

namespace {

// The micro-step after argument checks: hidden, dh (and the TMA-read W, dW) already validated.
int run_microstep(lmce_handle* h, const void* hidden, const void* W, const int32_t* targets, int64_t N,
                  int64_t global_valid, void* dh, float* row_loss, cudaStream_t st) {
  const lmce_config& c = h->cfg;
  const size_t esz = c.dtype == LMCE_BF16 ? 2 : 4;
  if (c.norm == LMCE_NORM_GLOBAL && global_valid <= 0) {
    if (N > 0 && cudaMemsetAsync(dh, 0, (size_t)N * c.C * esz, st) != cudaSuccess) return LMCE_ERR_CUDA;
    if (N > 0 && row_loss && cudaMemsetAsync(row_loss, 0, (size_t)N * sizeof(float), st) != cudaSuccess)
      return LMCE_ERR_CUDA;
    h->attempted += 1;  // dW untouched: the next micro-step with valid rows still writes it
    return LMCE_ERR_NO_VALID;
  }
  StepArgs a;
  a.hidden = hidden;
  a.W = W;
  a.targets = targets;
  a.dh = dh;
  a.dW = h->dW;
  a.row_loss = row_loss;
  a.N = N;
  a.C = c.C;
  a.V = c.V;
  a.ignore_id = c.ignore_id;
  a.norm = c.norm;
  a.G = c.grad_accum_steps;
  a.global_valid = global_valid;
  // the first micro-step of a step writes dW, unless the caller has already put part of the
  // step's gradient there
  const bool write_dW = h->first && !(c.flags & LMCE_ACCUMULATE_FROM_START);
  a.beta = write_dW ? 0 : 1;
  a.bf16 = c.dtype == LMCE_BF16;
  a.tc_two_pass = h->path == LMCE_PATH_TCGEN05_TWO_PASS;
  a.tc_recompute = h->path == LMCE_PATH_TCGEN05_RECOMPUTE;
  a.test_stall_ns = h->test_stall_ns;
  h->test_stall_ns = 0;
  if (N == 0) {
    // An empty micro-step still counts; the first one of a step leaves dW = 0.
    if (write_dW && cudaMemsetAsync(h->dW, 0, sizeof(float) * (size_t)c.V * c.C, st) != cudaSuccess)
      return LMCE_ERR_CUDA;
    h->first = false;
    h->attempted += 1;
    return LMCE_OK;
  }
  Launch L;
  L.st = st;
  L.prof = &h->prof;
  cudaError_t e = h->path != LMCE_PATH_SIMT ? tc_microstep(a, h->sc, L) : simt_microstep(a, h->sc, L);
  h->launches += L.n;
  if (e != cudaSuccess) return LMCE_ERR_CUDA;
  h->first = false;
  h->attempted += 1;
  return LMCE_OK;
}

}  // namespace

extern "C" int lmce_microstep(lmce_handle* h, const void* hidden, const void* W, const int32_t* targets,
                              int64_t N, int64_t global_valid, void* dh, float* row_loss, void* stream) {
  if (!h) return LMCE_ERR_ARG;
  if (N < 0 || N > h->cfg.max_N) return LMCE_ERR_ARG;
  if (N > 0 && (!hidden || !W || !targets || !dh)) return LMCE_ERR_ARG;
  if (h->path != LMCE_PATH_SIMT && N > 0) {
    if (((uintptr_t)hidden | (uintptr_t)W | (uintptr_t)dh | (uintptr_t)h->dW) & 15) return LMCE_ERR_ARG;
  }
  return run_microstep(h, hidden, W, targets, N, global_valid, dh, row_loss, (cudaStream_t)stream);
}

extern "C" int lmce_microstep_compact(lmce_handle* h, const void* hidden, const void* W, const int32_t* targets,
                                      int64_t N, int64_t n_valid, int64_t global_valid, void* dh, float* row_loss,
                                      void* stream) {
  if (!h || !h->cs.h_c) return LMCE_ERR_ARG;
  const lmce_config& c = h->cfg;
  if (N < 0 || N > c.max_N || n_valid < -1 || n_valid > N) return LMCE_ERR_ARG;
  if (N > 0 && (!hidden || !W || !targets || !dh)) return LMCE_ERR_ARG;
  const size_t esz = c.dtype == LMCE_BF16 ? 2 : 4;
  if (N > 0 && (((uintptr_t)hidden | (uintptr_t)dh) & (esz - 1))) return LMCE_ERR_ARG;
  if (h->path != LMCE_PATH_SIMT && N > 0 && (((uintptr_t)W | (uintptr_t)h->dW) & 15)) return LMCE_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (c.norm == LMCE_NORM_GLOBAL && global_valid <= 0)   // refused before any launch, as lmce_microstep
    return run_microstep(h, hidden, W, targets, N, global_valid, dh, row_loss, st);
  StepArgs a{};
  a.hidden = hidden;
  a.targets = targets;
  a.dh = dh;
  a.row_loss = row_loss;
  a.N = N;
  a.C = c.C;
  a.V = c.V;
  a.ignore_id = c.ignore_id;
  a.bf16 = c.dtype == LMCE_BF16;
  Launch L;
  L.st = st;
  L.prof = &h->prof;
  cudaError_t e = compact_rows(a, h->cs, h->sc.acc, n_valid, L);
  h->launches += L.n;
  if (e != cudaSuccess) return LMCE_ERR_CUDA;
  if (n_valid < 0) {
    if (cudaMemcpyAsync(h->cs.host_total, h->cs.total, sizeof(int64_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return LMCE_ERR_CUDA;
    n_valid = *h->cs.host_total;
  }
  const int s = run_microstep(h, h->cs.h_c, W, h->cs.y_c, n_valid, global_valid, h->cs.dh_c,
                              row_loss ? h->cs.rl_c : nullptr, st);
  if (s != LMCE_OK) return s;
  Launch L2;
  L2.st = st;
  L2.prof = &h->prof;
  e = compact_scatter(a, h->cs, n_valid, L2);
  h->launches += L2.n;
  return e == cudaSuccess ? LMCE_OK : LMCE_ERR_CUDA;
}

namespace {

// Argument checks shared by the two ln_f entry points (N rows of x / dx in the input dtype).
int check_ln_args(const lmce_handle* h, const void* x, const float* gamma, const float* beta, int32_t ln_kind,
                  float eps, const void* W, const int32_t* targets, int64_t N, void* dx, float* dgamma,
                  float* dbeta) {
  if (!h || !h->ln.h) return LMCE_ERR_ARG;
  const lmce_config& c = h->cfg;
  if (N < 0 || N > c.max_N) return LMCE_ERR_ARG;
  if (ln_kind != LMCE_LN_LAYERNORM && ln_kind != LMCE_LN_RMSNORM) return LMCE_ERR_ARG;
  if (!(eps >= 0.f) || !gamma || !dgamma || (ln_kind == LMCE_LN_RMSNORM && (beta || dbeta))) return LMCE_ERR_ARG;
  if (!beta && dbeta) return LMCE_ERR_ARG;
  if (N > 0 && (!x || !W || !targets || !dx)) return LMCE_ERR_ARG;
  const size_t esz = c.dtype == LMCE_BF16 ? 2 : 4;
  if (N > 0 && (((uintptr_t)x | (uintptr_t)dx) & (esz - 1))) return LMCE_ERR_ARG;
  if (h->path != LMCE_PATH_SIMT && N > 0 && (((uintptr_t)W | (uintptr_t)h->dW) & 15)) return LMCE_ERR_ARG;
  return LMCE_OK;
}

// GLOBAL normalisation without a valid target: refused before any launch, dx (and row_loss)
// zeroed, the parameter gradients untouched.
int refuse_no_valid(lmce_handle* h, int64_t N, void* dx, float* row_loss, cudaStream_t st) {
  const size_t esz = h->cfg.dtype == LMCE_BF16 ? 2 : 4;
  if (N > 0 && cudaMemsetAsync(dx, 0, (size_t)N * h->cfg.C * esz, st) != cudaSuccess) return LMCE_ERR_CUDA;
  if (N > 0 && row_loss && cudaMemsetAsync(row_loss, 0, (size_t)N * sizeof(float), st) != cudaSuccess)
    return LMCE_ERR_CUDA;
  h->attempted += 1;
  return LMCE_ERR_NO_VALID;
}

// ln_f forward, the micro-step on its output, ln_f backward: N rows of x (already checked).
int run_ln_step(lmce_handle* h, const void* x, const float* gamma, const float* beta, int32_t ln_kind, float eps,
                const void* W, const int32_t* targets, int64_t N, int64_t global_valid, void* dx, float* dgamma,
                float* dbeta, float* row_loss, cudaStream_t st) {
  const lmce_config& c = h->cfg;
  // the parameter gradients follow dW: written by the first micro-step of a step, then added
  const bool write = h->first && !(c.flags & LMCE_ACCUMULATE_FROM_START);
  LnArgs a{};
  a.x = x;
  a.gamma = gamma;
  a.beta = beta;
  a.h = h->ln.h;
  a.dh = h->ln.dh;
  a.dx = dx;
  a.mean = h->ln.mean;
  a.rstd = h->ln.rstd;
  a.part_g = h->ln.part;
  a.part_b = h->ln.part + (size_t)ln_part_rows() * (size_t)c.C;
  a.dgamma = dgamma;
  a.dbeta = dbeta;
  a.N = N;
  a.C = c.C;
  a.rms = ln_kind == LMCE_LN_RMSNORM;
  a.eps = eps;
  a.bf16 = c.dtype == LMCE_BF16;
  a.accumulate = write ? 0 : 1;
  a.err = &h->sc.acc->err;
  Launch L;
  L.st = st;
  L.prof = &h->prof;
  cudaError_t e = ln_forward(a, L);
  h->launches += L.n;
  if (e != cudaSuccess) return LMCE_ERR_CUDA;
  const int s = run_microstep(h, h->ln.h, W, targets, N, global_valid, h->ln.dh, row_loss, st);
  if (s != LMCE_OK) return s;
  if (N == 0) {   // an empty micro-step: the first one of a step leaves the parameter gradients 0
    if (write && (cudaMemsetAsync(dgamma, 0, sizeof(float) * c.C, st) != cudaSuccess ||
                  (dbeta && cudaMemsetAsync(dbeta, 0, sizeof(float) * c.C, st) != cudaSuccess)))
      return LMCE_ERR_CUDA;
    return LMCE_OK;
  }
  Launch L2;
  L2.st = st;
  L2.prof = &h->prof;
  e = ln_backward(a, L2);
  h->launches += L2.n;
  return e == cudaSuccess ? LMCE_OK : LMCE_ERR_CUDA;
}

}  // namespace

extern "C" int lmce_microstep_ln(lmce_handle* h, const void* x, const float* gamma, const float* beta,
                                 int32_t ln_kind, float eps, const void* W, const int32_t* targets, int64_t N,
                                 int64_t global_valid, void* dx, float* dgamma, float* dbeta, float* row_loss,
                                 void* stream) {
  const int ck = check_ln_args(h, x, gamma, beta, ln_kind, eps, W, targets, N, dx, dgamma, dbeta);
  if (ck != LMCE_OK) return ck;
  cudaStream_t st = (cudaStream_t)stream;
  if (h->cfg.norm == LMCE_NORM_GLOBAL && global_valid <= 0) return refuse_no_valid(h, N, dx, row_loss, st);
  return run_ln_step(h, x, gamma, beta, ln_kind, eps, W, targets, N, global_valid, dx, dgamma, dbeta, row_loss, st);
}

extern "C" int lmce_microstep_ln_compact(lmce_handle* h, const void* x, const float* gamma, const float* beta,
                                         int32_t ln_kind, float eps, const void* W, const int32_t* targets,
                                         int64_t N, int64_t n_valid, int64_t global_valid, void* dx,
                                         float* dgamma, float* dbeta, float* row_loss, void* stream) {
  const int ck = check_ln_args(h, x, gamma, beta, ln_kind, eps, W, targets, N, dx, dgamma, dbeta);
  if (ck != LMCE_OK) return ck;
  if (!h->cs.h_c || n_valid < -1 || n_valid > N) return LMCE_ERR_ARG;
  const lmce_config& c = h->cfg;
  cudaStream_t st = (cudaStream_t)stream;
  if (c.norm == LMCE_NORM_GLOBAL && global_valid <= 0) return refuse_no_valid(h, N, dx, row_loss, st);
  StepArgs a{};
  a.hidden = x;
  a.targets = targets;
  a.dh = dx;
  a.row_loss = row_loss;
  a.N = N;
  a.C = c.C;
  a.V = c.V;
  a.ignore_id = c.ignore_id;
  a.bf16 = c.dtype == LMCE_BF16;
  // Fused form (rows that fit ln_f's register layout): ln_f's forward reads the valid rows of x
  // in place and writes the head's compact input, its backward writes dx of every row; x is not
  // copied and dx needs no separate scatter.
  LnArgs la{};
  la.x = x;
  la.gamma = gamma;
  la.beta = beta;
  la.h = h->ln.h;
  la.dh = h->ln.dh;
  la.dx = dx;
  la.mean = h->ln.mean;
  la.rstd = h->ln.rstd;
  la.part_g = h->ln.part;
  la.part_b = h->ln.part + (size_t)ln_part_rows() * (size_t)c.C;
  la.dgamma = dgamma;
  la.dbeta = dbeta;
  la.N = N;
  la.C = c.C;
  la.rms = ln_kind == LMCE_LN_RMSNORM;
  la.eps = eps;
  la.bf16 = a.bf16;
  la.err = &h->sc.acc->err;
  const bool fused = N > 0 && ln_compact_fusable(la);
  Launch L;
  L.st = st;
  L.prof = &h->prof;
  cudaError_t e = fused ? compact_count_scan(a, h->cs, h->sc.acc, n_valid, L) : compact_rows(a, h->cs, h->sc.acc, n_valid, L);
  if (e == cudaSuccess && fused) e = ln_gather_forward(la, targets, c.V, h->cs, L);
  h->launches += L.n;
  if (e != cudaSuccess) return LMCE_ERR_CUDA;
  if (n_valid < 0) {
    if (cudaMemcpyAsync(h->cs.host_total, h->cs.total, sizeof(int64_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return LMCE_ERR_CUDA;
    n_valid = *h->cs.host_total;
  }
  if (fused) {
    // the parameter gradients follow dW: written by the first micro-step of a step, then added
    la.accumulate = h->first && !(c.flags & LMCE_ACCUMULATE_FROM_START) ? 0 : 1;
    const int s = run_microstep(h, h->ln.h, W, h->cs.y_c, n_valid, global_valid, h->ln.dh,
                                row_loss ? h->cs.rl_c : nullptr, st);
    if (s != LMCE_OK) return s;
    Launch L2;
    L2.st = st;
    L2.prof = &h->prof;
    e = ln_backward_scatter(la, h->cs, n_valid, row_loss, L2);
    h->launches += L2.n;
    return e == cudaSuccess ? LMCE_OK : LMCE_ERR_CUDA;
  }
  // otherwise: x gathered into the compact rows, ln_f and the head on them, dx scattered
  const int s = run_ln_step(h, h->cs.h_c, gamma, beta, ln_kind, eps, W, h->cs.y_c, n_valid, global_valid,
                            h->cs.dh_c, dgamma, dbeta, row_loss ? h->cs.rl_c : nullptr, st);
  if (s != LMCE_OK) return s;
  Launch L2;
  L2.st = st;
  L2.prof = &h->prof;
  e = compact_scatter(a, h->cs, n_valid, L2);
  h->launches += L2.n;
  return e == cudaSuccess ? LMCE_OK : LMCE_ERR_CUDA;
}

extern "C" int lmce_finalize(lmce_handle* h, double* loss_sum, int64_t* valid_count, double* loss_mean,
                             void* stream) {
  if (!h) return LMCE_ERR_ARG;
  if (h->attempted == 0) return LMCE_ERR_STATE;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(h->host_acc, h->sc.acc, sizeof(DevAcc), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return LMCE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return LMCE_ERR_CUDA;
  const DevAcc r = *h->host_acc;
  if (loss_sum) *loss_sum = r.loss_sum;
  if (valid_count) *valid_count = (int64_t)r.count;
  if (loss_mean) *loss_mean = r.count > 0 ? r.objective : NAN;
  h->first = true;
  h->attempted = 0;
  if (cudaMemsetAsync(h->sc.acc, 0, sizeof(DevAcc), st) != cudaSuccess) return LMCE_ERR_CUDA;
  if (r.err & ERR_BIT_BOUNDS) return LMCE_ERR_INTERNAL;  // a debug-build bounds check failed
  if (r.err & ERR_BIT_TIMEOUT) return LMCE_ERR_CUDA;  // a bounded device wait ran out
  if (r.err & ERR_BIT_COUNT) return LMCE_ERR_ARG;     // a compacted micro-step's n_valid was wrong
  if (r.err & ERR_BIT_BAD_TARGET) return LMCE_ERR_BAD_TARGET;
  if ((r.err & ERR_BIT_NONFINITE) || !isfinite(r.loss_sum)) return LMCE_ERR_NONFINITE;
  if (r.count == 0) return LMCE_ERR_NO_VALID;
  return LMCE_OK;
}

extern "C" int lmce_dw_sumsq(lmce_handle* h, double* sumsq, void* stream) {
  if (!h || !sumsq) return LMCE_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t n = h->cfg.V * h->cfg.C;
  const int64_t per = ((n + SQ_BLOCKS - 1) / SQ_BLOCKS + 3) / 4 * 4;   // a multiple of 4 elements
  Launch L;
  L.st = st;
  L.prof = &h->prof;
  L.begin(K_FINISH);
  sumsq_part_kernel<<<SQ_BLOCKS, SQ_T, 0, st>>>(h->dW, n, per, h->sumsq_part, h->sc.ticket + 1);
  L.end();
  h->launches += L.n;
  if (cudaGetLastError() != cudaSuccess) return LMCE_ERR_CUDA;
  double r = 0.0;
  if (cudaMemcpyAsync(&r, h->sumsq_part + SQ_BLOCKS, sizeof(double), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return LMCE_ERR_CUDA;
  *sumsq = r;
  return LMCE_OK;
}

extern "C" int lmce_clip_coef(double sumsq, double max_norm, float* coef) {
  if (!coef || !(sumsq >= 0.0) || !isfinite(sumsq) || !(max_norm > 0.0) || !isfinite(max_norm)) return LMCE_ERR_ARG;
  const double c = max_norm / (sqrt(sumsq) + 1e-6);   // clip_grad_norm_'s guard against a zero norm
  *coef = (float)(c < 1.0 ? c : 1.0);
  return LMCE_OK;
}

extern "C" int lmce_adamw(lmce_handle* h, float* p, float* m, float* v, void* W_out, int64_t step, float lr,
                          float beta1, float beta2, float eps, float weight_decay, float clip, void* stream) {
  if (!h || !p || !m || !v || step < 1) return LMCE_ERR_ARG;
  if (!(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f) || !(eps >= 0.f)) return LMCE_ERR_ARG;
  if (!isfinite(lr) || !isfinite(weight_decay) || !isfinite(clip)) return LMCE_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t n = h->cfg.V * h->cfg.C;
  // bias corrections in float64 on the host, then the per-element constants in float32
  const double bc1 = 1.0 - pow((double)beta1, (double)step), bc2 = 1.0 - pow((double)beta2, (double)step);
  AdamCoef k;
  k.clip = clip;
  k.b1 = beta1;
  k.omb1 = (float)(1.0 - (double)beta1);
  k.b2 = beta2;
  k.omb2 = (float)(1.0 - (double)beta2);
  k.decay = (float)(1.0 - (double)lr * (double)weight_decay);
  k.step_size = (float)((double)lr / bc1);
  k.sqrt_bc2 = (float)sqrt(bc2);
  k.eps = eps;
  const uintptr_t al = (uintptr_t)h->dW | (uintptr_t)p | (uintptr_t)m | (uintptr_t)v | (uintptr_t)W_out;
  const int vec = (al & 15) == 0;
  Launch L;
  L.st = st;
  L.prof = &h->prof;
  L.begin(K_FINISH);
  adamw_kernel<<<AW_BLOCKS, AW_T, 0, st>>>(h->dW, p, m, v, (__nv_bfloat16*)W_out, n, vec, k);
  L.end();
  h->launches += L.n;
  return cudaGetLastError() == cudaSuccess ? LMCE_OK : LMCE_ERR_CUDA;
}

extern "C" int lmce_destroy(lmce_handle* h) {
  if (!h) return LMCE_OK;
  int cur = 0;
  cudaGetDevice(&cur);
  if (cur != h->device) cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  free_scratch(h);
  for (cudaEvent_t e : h->prof.pool) cudaEventDestroy(e);
  if (cur != h->device) cudaSetDevice(cur);
  delete h;
  return LMCE_OK;
}

extern "C" const char* lmce_status_string(int s) {
  switch (s) {
    case LMCE_OK: return "ok";
    case LMCE_ERR_ARG: return "invalid argument";
    case LMCE_ERR_ARCH: return "device is not compute capability 10.3 (sm_103)";
    case LMCE_ERR_CUDA: return "CUDA error";
    case LMCE_ERR_BAD_TARGET: return "target outside [0, V) that is not the ignore id";
    case LMCE_ERR_NO_VALID: return "no valid target in the step";
    case LMCE_ERR_NONFINITE: return "loss is not finite";
    case LMCE_ERR_STATE: return "call out of order";
    case LMCE_ERR_INTERNAL: return "a bounds check of the debug build failed (library bug)";
    default: return "unknown status";
  }
}

extern "C" int lmce_debug_bounds(void) { return LMCE_DEBUG_BOUNDS ? 1 : 0; }

extern "C" int lmce_test_bounds_limit(lmce_handle* h, int64_t rows) {
  if (!h) return LMCE_ERR_ARG;
  if (!LMCE_DEBUG_BOUNDS || !h->cs.h_c) return LMCE_ERR_STATE;
  if (rows < 0 || rows > h->cfg.max_N) return LMCE_ERR_ARG;
  h->cs.rows = rows;
  return LMCE_OK;
}

extern "C" int lmce_test_stall_next_microstep(lmce_handle* h, int64_t wait_ns) {
  if (!h || wait_ns <= 0 || wait_ns > 1000000000LL) return LMCE_ERR_ARG;
  if (h->path == LMCE_PATH_SIMT) return LMCE_ERR_STATE;
  h->test_stall_ns = wait_ns;
  return LMCE_OK;
}

extern "C" int64_t lmce_launch_count(const lmce_handle* h) { return h ? h->launches : 0; }

extern "C" int lmce_selected_path(const lmce_handle* h) { return h ? h->path : -1; }

extern "C" int lmce_profile(lmce_handle* h, int enable) {
  if (!h) return LMCE_ERR_ARG;
  if (enable) {
    h->prof.recs.clear();
    h->prof.used = 0;
  }
  h->prof.on = enable != 0;
  return LMCE_OK;
}

extern "C" int lmce_profile_read(lmce_handle* h, int kind, double* total_ms, int64_t* launches) {
  if (!h || !total_ms || !launches || kind < 0 || kind >= K_COUNT) return LMCE_ERR_ARG;
  double t = 0.0;
  int64_t n = 0;
  for (const Prof::Rec& r : h->prof.recs) {
    if (r.kind != kind) continue;
    if (cudaEventSynchronize(r.b) != cudaSuccess) return LMCE_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return LMCE_ERR_CUDA;
    t += ms;
    ++n;
  }
  *total_ms = t;
  *launches = n;
  return LMCE_OK;
}
