// Tensor-core path (tcgen05 + TMA, sm_103a) of the fused LM-head + cross-entropy micro-step.
//
// Pass 1 (tc_lse_kernel): logits tiles z = h . W^T ("How I trained my own GPT-2 124M on
// FineWeb-Edu", section 4: the tied, bias-free lm_head) on CTA pairs: one cta_group::2
// MMA chain per 256-token x 256-vocab tile, K = C streamed through a TMA ring, fp32
// accumulators double-buffered in TMEM.  Four epilogue warps per CTA read each tile back
// with tcgen05.ld and keep a per-row online max / sum-exp (base 2), so no logit reaches
// device memory.  Each cluster covers one token block and a slice of the vocabulary and
// writes a partial (max, sum) per row; tc_combine_kernel merges the slices into the row
// logsumexp and loss.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <mutex>

#include "lmce_internal.cuh"
#include "tc_ptx.cuh"

namespace lmce {

using namespace ptx;

namespace {

constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s: any wait longer than this is an error


// ---- pass 1 geometry -----------------------------------------------------------------
constexpr int L_BM = 128;            // token rows per CTA (256 per pair)
constexpr int L_BN = 128;            // vocab rows per CTA (256 per pair tile)
constexpr int L_BK = 64;             // C per stage (one 128-byte swizzle atom)
constexpr int L_ST = 6;              // stages
constexpr int L_STAGE_A = L_BM * L_BK * 2;  // 16 KB
constexpr int L_STAGE_B = L_BN * L_BK * 2;  // 16 KB
constexpr int L_STAGE = L_STAGE_A + L_STAGE_B;
constexpr int L_THREADS = 192;       // warp 0 TMA, warp 1 MMA / forwarder, warps 2-5 epilogue
constexpr int L_SMEM = L_ST * L_STAGE + 1024;

struct LseParams {
  const int32_t* targets;
  float* part_m;   // [nsplit][N] base-2 running max
  float* part_l;   // [nsplit][N] sum of 2^(x - m)
  float* zt;       // [N] target logit
  unsigned* err;   // error word (timeouts)
  int N, V, C;
  int ignore_id;
  int vtiles;      // ceil(V / 256)
  int nsplit;
};

// A timed-out wait records the timeout bit and which wait gave up (bits 8..15).
__device__ __forceinline__ void record_timeout(unsigned* err, unsigned where) {
  atomicOr(err, ERR_BIT_TIMEOUT | (where << 8));
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(L_THREADS, 1)
    tc_lse_kernel(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmW, LseParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[L_ST], pfull[L_ST], empty[L_ST], acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ volatile int epi_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int nb = blockIdx.x >> 1;        // token block (256 rows per pair)
  const int split = blockIdx.y;
  const int t_begin = (int)(((long long)split * p.vtiles) / p.nsplit);
  const int t_end = (int)(((long long)(split + 1) * p.vtiles) / p.nsplit);
  const int ntiles = t_end - t_begin;
  const int kchunks = p.C / L_BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L_ST; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&pfull[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), 2);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    epi_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<2>(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish<2>();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmH);
      tma_prefetch_desc(&tmW);
      const int hrow = nb * 256 + (int)rank * L_BM;
      int it = 0;
      bool ok = true;
      for (int t = 0; t < ntiles && ok; ++t) {
        const int wrow = (t_begin + t) * 256 + (int)rank * L_BN;
        for (int kc = 0; kc < kchunks; ++kc, ++it) {
          const int s = it % L_ST;
          const uint32_t ph = ((it / L_ST) & 1) ^ 1;
          if (!mbar_wait(smem_u32(&empty[s]), ph, WAIT_NS)) { record_timeout(p.err, 1); ok = false; break; }
          const uint32_t a = smem_u32(smem + s * L_STAGE), b = a + L_STAGE_A;
          mbar_expect_tx(smem_u32(&full[s]), L_STAGE);
          tma_load_2d(a, &tmH, smem_u32(&full[s]), kc * L_BK, hrow);
          tma_load_2d(b, &tmW, smem_u32(&full[s]), kc * L_BK, wrow);
        }
      }
    }
  } else if (warp == 1) {
    if (rank == 1) {
      // ---------------- forwarder: tell the leader when this CTA's stage landed ------------
      if (lane == 0) {
        const uint32_t leader_pfull = mapa(smem_u32(&pfull[0]), 0);
        int it = 0;
        for (int t = 0; t < ntiles; ++t)
          for (int kc = 0; kc < kchunks; ++kc, ++it) {
            const int s = it % L_ST;
            if (!mbar_wait(smem_u32(&full[s]), (it / L_ST) & 1, WAIT_NS)) {
              record_timeout(p.err, 2);
              t = ntiles;
              break;
            }
            mbar_arrive_cluster(leader_pfull + s * 8);
          }
      }
    } else if (lane == 0) {
      // ---------------- MMA issuer (leader CTA) ----------------
      const uint32_t idesc = idesc_bf16(256, 256, 0, 0);
      int it = 0;
      bool ok = true;
      for (int t = 0; t < ntiles && ok; ++t) {
        const int b = t & 1;
        if (!mbar_wait_cluster(smem_u32(&acc_empty[b]), ((t >> 1) & 1) ^ 1, WAIT_NS)) {
          record_timeout(p.err, 3);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + b * 256;
        for (int kc = 0; kc < kchunks; ++kc, ++it) {
          const int s = it % L_ST;
          const uint32_t ph = (it / L_ST) & 1;
          if (!mbar_wait(smem_u32(&full[s]), ph, WAIT_NS) || !mbar_wait_cluster(smem_u32(&pfull[s]), ph, WAIT_NS)) {
            record_timeout(p.err, 4);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(smem + s * L_STAGE), bb = a + L_STAGE_A;
#pragma unroll
          for (int k = 0; k < L_BK / 16; ++k)
            mma_ss<2>(d, sdesc_sw128(a + k * 32, 16, 1024), sdesc_sw128(bb + k * 32, 16, 1024), idesc,
                      (kc | k) != 0);
          mma_commit_mc2(smem_u32(&empty[s]), 3);
        }
        if (ok) mma_commit_mc2(smem_u32(&acc_full[b]), 3);
      }
      if (!ok) {
        // give up: wait (bounded) for the MMAs already issued before TMEM is released
        mma_commit<2>(smem_u32(&drain_bar));
        mbar_wait(smem_u32(&drain_bar), 0, WAIT_NS);
      }
    }
  } else {
    // ---------------- epilogue: warps 2..5, one token row per thread ----------------
    const int q = warp & 3;
    const int row = (int)rank * L_BM + q * 32 + lane;
    const int n = nb * 256 + row;
    const int y = (n < p.N) ? p.targets[n] : p.ignore_id;
    float m2 = -INFINITY, l = 0.f;
    const uint32_t leader_acc_empty = mapa(smem_u32(&acc_empty[0]), 0);
    for (int t = 0; t < ntiles; ++t) {
      const int b = t & 1;
      if (!mbar_wait(smem_u32(&acc_full[b]), (t >> 1) & 1, WAIT_NS)) {
        record_timeout(p.err, 5);
        epi_abort = 1;
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (epi_abort) break;  // the same decision in every epilogue thread
      tc_fence_after();
      const int v0 = (t_begin + t) * 256;
      const uint32_t taddr = tmem + b * 256 + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        float v[32];
        tmem_ld32(taddr + c * 32, v);
        tmem_ld_wait();
        const int vb = v0 + c * 32;
        float cm = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (vb + j < p.V) cm = fmaxf(cm, v[j]);
          if (vb + j == y) p.zt[n] = v[j];
        }
        if (cm == -INFINITY) continue;
        const float mn = fmaxf(m2, cm * LOG2E);
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (vb + j < p.V) s += exp2f(fmaf(v[j], LOG2E, -mn));
        l = l * exp2f(m2 - mn) + s;
        m2 = mn;
      }
      tc_fence_before();
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (warp == 2 && lane == 0) {
        if (rank == 0) mbar_arrive(smem_u32(&acc_empty[b]));
        else mbar_arrive_cluster(leader_acc_empty + b * 8);
      }
    }
    if (n < p.N) {
      p.part_m[(size_t)split * p.N + n] = m2;
      p.part_l[(size_t)split * p.N + n] = l;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<2>(tmem, 512);
  }
}

// One thread per row: merge the vocabulary slices into lse, then the row loss and the
// per-block loss / count / error partials for the fixed-order reduction.
__global__ void __launch_bounds__(256) tc_combine_kernel(const float* __restrict__ part_m,
                                                         const float* __restrict__ part_l,
                                                         const float* __restrict__ zt, int nsplit,
                                                         StepArgs a, float* __restrict__ lse_out,
                                                         double* __restrict__ part_loss,
                                                         int* __restrict__ part_cnt,
                                                         unsigned* __restrict__ part_err) {
  __shared__ double sl[256];
  __shared__ int sc[256];
  __shared__ unsigned se[256];
  const int t = threadIdx.x;
  const int64_t n = (int64_t)blockIdx.x * 256 + t;
  double loss = 0.0;
  int valid = 0;
  unsigned err = 0;
  if (n < a.N) {
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part_m[(size_t)s * a.N + n]);
    float L = 0.f;
    for (int s = 0; s < nsplit; ++s) L += part_l[(size_t)s * a.N + n] * exp2f(part_m[(size_t)s * a.N + n] - M);
    const float lse = (M + log2f(L)) * LN2;
    lse_out[n] = lse;
    const int y = a.targets[n];
    if (y >= 0 && (int64_t)y < a.V) {
      const float li = lse - zt[n];
      loss = (double)li;
      valid = 1;
      if (!isfinite(li)) err |= ERR_BIT_NONFINITE;
      if (a.row_loss) a.row_loss[n] = li;
    } else {
      if (y != a.ignore_id) err |= ERR_BIT_BAD_TARGET;
      if (a.row_loss) a.row_loss[n] = 0.f;
    }
  }
  sl[t] = loss;
  sc[t] = valid;
  se[t] = err;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (t < o) {
      sl[t] += sl[t + o];
      sc[t] += sc[t + o];
      se[t] |= se[t + o];
    }
    __syncthreads();
  }
  if (t == 0) {
    part_loss[blockIdx.x] = sl[0];
    part_cnt[blockIdx.x] = sc[0];
    part_err[blockIdx.x] = se[0];
  }
}

// ---- host side ------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// bf16 matrix [rows, cols] row-major; box {64 cols, box_rows}, 128-byte swizzle, zero fill.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

// Vocabulary slices per token block: minimise waves x tiles-per-slice (+ a fixed cost).
int choose_nsplit(int nblocks, int vtiles, int pairs) {
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= vtiles && s <= TC_MAX_SPLIT; ++s) {
    const int waves = (nblocks * s + pairs - 1) / pairs;
    const int per = (vtiles + s - 1) / s;
    const double cost = waves * (per + 0.5);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

}  // namespace

// Scratch needed by the tensor-core path beyond the common buffers: per-slice partials.
bool tc_supported(int64_t C, int64_t V, int bf16) {
  return bf16 && C % 256 == 0 && C >= 256 && C <= 1024 && V >= 1 && V < (1LL << 31);
}

int64_t tc_parts(int64_t N) { return (N + 255) / 256; }


cudaError_t tc_lse(const StepArgs& a, const Scratch& sc, Launch& L) {
  CUtensorMap mh, mw;
  if (!make_map(&mh, a.hidden, (uint64_t)a.N, (uint64_t)a.C, L_BM) ||
      !make_map(&mw, a.W, (uint64_t)a.V, (uint64_t)a.C, L_BN))
    return cudaErrorInvalidValue;
  const int nblocks = (int)((a.N + 255) / 256);
  const int vtiles = (int)((a.V + 255) / 256);
  const int nsplit = choose_nsplit(nblocks, vtiles, num_sms() / 2);
  LseParams p;
  p.targets = a.targets;
  p.part_m = sc.tc_part_m;
  p.part_l = sc.tc_part_l;
  p.zt = sc.tc_zt;
  p.err = &sc.acc->err;
  p.N = (int)a.N;
  p.V = (int)a.V;
  p.C = (int)a.C;
  p.ignore_id = a.ignore_id;
  p.vtiles = vtiles;
  p.nsplit = nsplit;
  cudaFuncSetAttribute(tc_lse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L_SMEM);
  L.begin(K_LSE);
  tc_lse_kernel<<<dim3(2 * nblocks, nsplit), L_THREADS, L_SMEM, L.st>>>(mh, mw, p);
  L.end();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t nparts = tc_parts(a.N);
  L.begin(K_LSE);
  tc_combine_kernel<<<(unsigned)nparts, 256, 0, L.st>>>(sc.tc_part_m, sc.tc_part_l, sc.tc_zt, nsplit, a, sc.lse,
                                                        sc.part_loss, sc.part_cnt, sc.part_err);
  L.end();
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_finish(a, sc, nparts, L);
}

cudaError_t tc_microstep(const StepArgs& a, const Scratch& sc, Launch& L) {
  cudaError_t e = tc_lse(a, sc, L);
  if (e != cudaSuccess) return e;
  return simt_grads(a, sc, L);
}

}  // namespace lmce
