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
constexpr int L_BK = 128;            // C per stage: two 64-column swizzle atoms, one 3D TMA box each side
constexpr int L_ST = 3;              // stages
constexpr int L_STAGE_A = L_BM * L_BK * 2;  // 32 KB
constexpr int L_STAGE_B = L_BN * L_BK * 2;  // 32 KB
constexpr int L_STAGE = L_STAGE_A + L_STAGE_B;
constexpr int L_THREADS = 352;       // warps 0 and 10 TMA, warp 1 MMA, warps 2-9 epilogue (two per lane quarter)
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
  __shared__ __align__(8) uint64_t full[L_ST], empty[L_ST], acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ volatile int epi_abort;
  __shared__ float half_m[L_BM], half_l[L_BM];   // second column half's (max, sum) per row

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

  if (warp == 0 || warp == 10) {
    // ---------------- TMA producers: two warps take alternate stages (a warp's TMA issue
    // has a fixed cost, so two warps double the rate); in each, lane 0 waits and arms the
    // barrier and lanes 0 and 1 each issue one 32 KB box ----------------
    const int pw = warp == 0 ? 0 : 1;
    if (lane == 0 && pw == 0) {
      tma_prefetch_desc(&tmH);
      tma_prefetch_desc(&tmW);
    }
    const int hrow = nb * 256 + (int)rank * L_BM;
    const uint32_t lead_full = mapa(smem_u32(&full[0]), 0);  // both halves land on the leader's barrier
    int it = 0;
    bool ok = true;
    for (int t = 0; t < ntiles && ok; ++t) {
      const int wrow = (t_begin + t) * 256 + (int)rank * L_BN;
      for (int kc = 0; kc < kchunks; ++kc, ++it) {
        if ((it & 1) != pw) continue;
        const int s = it % L_ST;
        const uint32_t ph = ((it / L_ST) & 1) ^ 1;
        bool w = true;
        if (lane == 0) {
          w = mbar_wait(smem_u32(&empty[s]), ph, WAIT_NS);
          if (!w) record_timeout(p.err, 1);
          else if (rank == 0) mbar_expect_tx(smem_u32(&full[s]), 2 * L_STAGE);
        }
        if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
        const uint32_t a = smem_u32(smem + s * L_STAGE);
        if (lane == 0) tma_load_3d_cg2(a, &tmH, lead_full + s * 8, 0, hrow, kc * 2);
        else if (lane == 1) tma_load_3d_cg2(a + L_STAGE_A, &tmW, lead_full + s * 8, 0, wrow, kc * 2);
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    if (rank == 1) {
      // the peer CTA issues nothing: its TMA loads complete on the leader's barriers
    } else {
      // ---------------- MMA issuer (leader CTA): the whole warp runs the loop, waits are
      // polled by all lanes and decided together, elect.sync picks the issuing lane ----------------
      const uint32_t idesc = idesc_bf16(256, 256, 0, 0);
      const uint64_t dA = sdesc_sw128(smem_u32(smem), 16, 1024), dB = sdesc_sw128(smem_u32(smem) + L_STAGE_A, 16, 1024);
      int it = 0;
      bool ok = true;
      for (int t = 0; t < ntiles && ok; ++t) {
        const int b = t & 1;
        const bool we = __all_sync(0xffffffffu, mbar_wait_cluster(smem_u32(&acc_empty[b]), ((t >> 1) & 1) ^ 1, WAIT_NS));
        if (!we) {
          if (lane == 0) record_timeout(p.err, 3);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + b * 256;
        for (int kc = 0; kc < kchunks; ++kc, ++it) {
          const int s = it % L_ST;
          const uint32_t ph = (it / L_ST) & 1;
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[s]), ph, WAIT_NS))) {
            if (lane == 0) record_timeout(p.err, 4);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a = dA + (uint32_t)(s * (L_STAGE >> 4)), bb = dB + (uint32_t)(s * (L_STAGE >> 4));
#pragma unroll
          for (int k = 0; k < L_BK / 16; ++k) {
            // atom (64 columns, 128 rows x 128 B apart), then 16-column (32 B) steps
            const uint32_t off = ((k >> 2) * (L_BM * 128) + (k & 3) * 32) >> 4;
            mma_ss2_elect(d, a + off, bb + off, idesc, (kc | k) != 0);
          }
          mma_commit_mc2_elect(smem_u32(&empty[s]), 3);
        }
        if (ok) mma_commit_mc2_elect(smem_u32(&acc_full[b]), 3);
      }
      if (!ok) {
        // give up: wait (bounded) for the MMAs already issued before TMEM is released
        mma_commit2_elect(smem_u32(&drain_bar));
        mbar_wait(smem_u32(&drain_bar), 0, WAIT_NS);
      }
    }
  } else if (warp <= 9) {
    // ---------------- epilogue: warps 2..9 ----------------
    // warp -> TMEM lane quarter q (its token rows) and column half hf of every tile; each
    // thread keeps a base-2 running (max, sum) of its row over its half of the columns.
    const int q = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int kl = q * 32 + lane;
    const int row = (int)rank * L_BM + kl;
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
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (epi_abort) break;  // the same decision in every epilogue thread
      tc_fence_after();
      const int c0 = (t_begin + t) * 256 + hf * 128;      // first vocabulary column of my half
      const int tcol = y - c0;                            // my target's column in my half, if any
      const bool full_half = c0 + 128 <= p.V;
      const uint32_t taddr = tmem + b * 256 + hf * 128 + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(taddr + c * 32, v);
        if (tcol >= c * 32 && tcol < c * 32 + 32) {
          float zv = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) zv = (tcol - c * 32 == j) ? v[j] : zv;
          p.zt[n] = zv;
        }
        if (!full_half) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c0 + c * 32 + j >= p.V) v[j] = -INFINITY;
        }
        float cm = v[0];
#pragma unroll
        for (int j = 1; j < 32; ++j) cm = fmaxf(cm, v[j]);
        if (cm == -INFINITY) continue;
        const float mn = fmaxf(m2, cm * LOG2E);
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) sum += ex2_approx(fmaf(v[j], LOG2E, -mn));
        l = l * ex2_approx(m2 - mn) + sum;
        m2 = mn;
      }
      tc_fence_before();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (warp == 2 && lane == 0) {
        if (rank == 0) mbar_arrive(smem_u32(&acc_empty[b]));
        else mbar_arrive_cluster(leader_acc_empty + b * 8);
      }
    }
    // merge the two column halves of every row, then write this slice's partial
    if (hf == 1) {
      half_m[kl] = m2;
      half_l[kl] = l;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (hf == 0 && n < p.N) {
      const float mo = half_m[kl], lo = half_l[kl];
      const float M = fmaxf(m2, mo);
      const float L = (M == -INFINITY) ? 0.f : l * ex2_approx(m2 - M) + lo * ex2_approx(mo - M);
      p.part_m[(size_t)split * p.N + n] = M;
      p.part_l[(size_t)split * p.N + n] = L;
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

// ---- pass 2: gradients ----------------------------------------------------------------
// One kernel shape serves the three passes that contract a recomputed logit tile.  A CTA
// pair owns 128 "X" rows and streams the other operand "Y" in blocks of 256 rows:
//   dW pass     : X = W (vocabulary rows), Y = h (tokens); acc^T[c][v] = sum_n h[n][c] dz[n][v]
//   dh pass     : X = h (tokens), Y = W (vocabulary rows);  acc^T[c][n] = sum_v W[v][c] dz[n][v]
//   lse+dh pass : as the dh pass, with the softmax normaliser found on the way (below)
// with dz[n][v] = s (softmax(z_n)[v] - [v == y_n]) ("How I trained my own GPT-2 124M",
// section 4, differentiated; s from the gradient-accumulation normalisation).
// Per block: S^T = Y_blk . X^T (cta_group::2, M = 256 stream rows, N = 128, K = C) lands in
// TMEM; eight epilogue warps (two per TMEM lane quarter, one per half of the 128 columns)
// turn it into the bf16 operand of the second product and write it, already in the
// 128-byte-swizzled MN-major layout, into the CTA that supplies that half of N (its own or
// the peer's, over DSMEM).  dW and dh passes: s*softmax = 2^(z log2 e + log2 s - lse log2 e),
// one FFMA and one ex2 per element; the one-hot part is applied once per row (dW: the
// target's element of its row, from the target logit; dh: s*W[y_n] subtracted when dh is
// written).
// acc^T[C x 128] += Y_blk^T . dz (cta_group::2, M = 256 C rows per chunk, K = 256 stream
// rows) accumulates in TMEM for the whole stream, one 64-row quarter of dz at a time as
// soon as that quarter is written.  The S tile of block j+1 is computed while the epilogue
// works on block j.  Every output element has one owner: deterministic.
//
// The lse+dh pass needs no logsumexp beforehand.  It is the online softmax of flash
// attention with the stale-maximum rule of FlashAttention-4 taken to its end: each token
// column's base-2 reference m_n is fixed once, as the exact maximum over the first block of
// the pair's range (agreed between the two CTAs over DSMEM), and never moved.  The operand
// is p = 2^(z log2 e - m_n) and the epilogue also sums p per column (a butterfly over the 32
// rows of a warp, kept in two registers per lane), so at the end of the range
//   acc^T[c][n] = sum_v W[v][c] p[n][v],   l_n = sum_v p[n][v],
//   dh_n = s (acc^T[.][n] / l_n - W[y_n]),   lse_n = (m_n + log2 l_n) ln 2.
// An element above m_n + 80 (p > 2^80, where fp32 sums could start to lose range) flags its
// 128-token tile; the host then runs the exact two-pass repair on flagged tiles only.
constexpr int G_XT = 128;                  // X rows per pair (64 per CTA)
constexpr int G_YB = 256;                  // stream rows per block (128 per CTA)
constexpr int G_DZ = G_YB * 128;           // one dz buffer: 256 K-rows x 64 bf16 = 32 KB
constexpr int G_EPI_WARPS = 8;
constexpr int G_THREADS = 96 + 32 * G_EPI_WARPS;   // warps 0 and 10 TMA, 1 MMA, 2-9 epilogue
constexpr float FL_LIMIT = 80.f;           // lse+dh pass: largest exponent of p kept

enum GradMode { GM_DW = 0, GM_DH = 1, GM_FL = 2 };

// Ring geometry per mode: NST slots of SLOT bytes.  An S stage carries SK 64-column atoms of
// K = C (per CTA: 128 stream rows, then 64 X rows at SK * 16 KB); an accumulation stage
// carries AQ 64-row quarters of the stream block for every 256-row C chunk (per chunk two
// 64-column atoms, AQ * 16 KB); NDZ dz buffers.
template <int MODE>
struct Geo {
  static constexpr int NST = 3, SLOT = 49152, SK = 2, AQ = 1, NDZ = 2;
};
template <int MODE>
constexpr int geo_smem_bytes() {
  return Geo<MODE>::NST * Geo<MODE>::SLOT + Geo<MODE>::NDZ * G_DZ + 1024;
}

struct GradParams {
  const int32_t* targets;
  const float* lse;      // dW and dh passes: per-row logsumexp (natural log)
  const float* zt;       // dW pass: target logits
  const DevAcc* acc;     // scale of this micro-step
  unsigned* err;
  float* dW;             // dW pass output (fp32 [V, C])
  __nv_bfloat16* dh;     // dh / lse+dh pass output (bf16 [N, C])
  const __nv_bfloat16* Wt;  // W, for the one-hot term of dh
  float* part;           // [2 * pairs][128][C] fp32 partial sums of split tiles
  float* part_lm;        // lse+dh pass: [2 * pairs][2][128] (m, l) of split tiles
  float* lse_out;        // lse+dh pass: per-row logsumexp
  unsigned* tile_flag;   // lse+dh pass: per 128-token tile, set when the tile needs the repair
  int N, V, C;
  int ch0, nch;          // 256-row C chunks [ch0, ch0 + nch) of acc^T handled by this launch (nch <= 3)
  int beta;              // dW pass: 0 writes, 1 adds
};

// Balanced persistent schedule.  Work units are (X tile t, stream block j), t-major; pair pi
// of P takes units [U pi / P, U (pi + 1) / P).  Its range crosses X tiles in segments; a segment
// that covers a whole tile writes the output directly, a segment that covers part of a tile
// (at most the pair's first and last) writes fp32 partial sums to slot 2 pi (first segment) or
// 2 pi + 1, and the split-combine kernels add the partials of each split tile in pair order.
struct Sched {
  long long U;  // tiles * blocks per tile
  int P;        // pairs
  int nblk;     // stream blocks per tile
  __host__ __device__ long long u0(int p) const { return U * p / P; }
  __host__ __device__ int pair_of(long long u) const {
    int p = (int)((u * P) / U);
    while (p + 1 < P && u0(p + 1) <= u) ++p;
    while (p > 0 && u0(p) > u) --p;
    return p;
  }
};

__device__ __forceinline__ void st_shared_b16(uint32_t addr, uint16_t v, bool remote) {
  if (remote) asm volatile("st.shared::cluster.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
  else asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

// One halving step of the column reduction below: lanes with bit O set keep the upper H of
// their 2H values and receive the partner's upper H, the others the lower halves.
template <bool MAX, int H, int O>
__device__ __forceinline__ void col_step(float (&v)[64], bool hi) {
#pragma unroll
  for (int i = 0; i < H; ++i) {
    const float keep = hi ? v[i + H] : v[i];
    const float send = hi ? v[i] : v[i + H];
    const float got = __shfl_xor_sync(0xffffffffu, send, O);
    v[i] = MAX ? fmaxf(keep, got) : keep + got;
  }
}

// Column reduction of a 32 x 64 register tile (row = lane): afterwards lane L holds the max
// or sum over the 32 rows of columns 2L and 2L + 1 in v[0], v[1].  62 shuffles, fixed order.
template <bool MAX>
__device__ __forceinline__ void col_reduce64(float (&v)[64], int lane) {
  col_step<MAX, 32, 16>(v, lane & 16);
  col_step<MAX, 16, 8>(v, lane & 8);
  col_step<MAX, 8, 4>(v, lane & 4);
  col_step<MAX, 4, 2>(v, lane & 2);
  col_step<MAX, 2, 1>(v, lane & 1);
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(G_THREADS, 1)
    tc_grad_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmYs,
                   const __grid_constant__ CUtensorMap tmYa, GradParams p) {
  constexpr bool DW = MODE == GM_DW;
  constexpr bool FL = MODE == GM_FL;
  constexpr int NST = Geo<MODE>::NST, SLOT = Geo<MODE>::SLOT, SK = Geo<MODE>::SK, AQ = Geo<MODE>::AQ;
  constexpr int NDZ = Geo<MODE>::NDZ;
  static_assert(SK * 24576 <= SLOT && AQ * 16384 * 3 <= SLOT && 4 % AQ == 0, "stage does not fit its slot");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int KC = p.C / (64 * SK);           // S phase stages per block
  const int NCH = p.nch;                    // 256-row C chunks of acc^T in TMEM (from chunk p.ch0 on)
  uint8_t* sY = smem;                       // ring of NST slots
  uint8_t* sDZ = sY + NST * SLOT;           // [NDZ][256 rows][128 B]
  __shared__ __align__(8) uint64_t full[NST], empty[NST];
  __shared__ __align__(8) uint64_t s_full, s_empty, dz_full[NDZ][4], dz_empty[NDZ], acc_full, acc_empty, drain_bar;
  __shared__ __align__(8) uint64_t mx_full, lx_full;   // lse+dh pass: the peer's column max / sum arrived
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int epi_abort;
  __shared__ float col_c[G_XT];             // dh: log2(s) - lse log2(e) or -inf;  lse+dh: reference m_n (base 2)
  __shared__ int col_y[G_XT];               // dh, lse+dh: per-column target (or -1: no gradient)
  __shared__ float fl_q[4][G_XT];           // lse+dh: per-lane-quarter column max / sum
  __shared__ float fl_loc[G_XT];            // lse+dh: this CTA's column max / sum
  __shared__ float fl_pm[2][G_XT], fl_pl[2][G_XT];  // lse+dh: the peer's column max / sum (by segment parity)
  __shared__ float fl_L[G_XT];              // lse+dh: l_n of the pair
  __shared__ float fl_f[G_XT];              // lse+dh: s / l_n for a valid target, else 0
  __shared__ float fl_s[G_XT];              // lse+dh: s for a valid target, else 0

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int nX = DW ? p.V : p.N;
  const int nY = DW ? p.N : p.V;
  const int nblk = (nY + G_YB - 1) / G_YB;
  const int T = (nX + G_XT - 1) / G_XT;
  const Sched sch{(long long)T * nblk, (int)(gridDim.x >> 1), nblk};
  const int pi = blockIdx.x >> 1;
  const long long ub = sch.u0(pi), ue = sch.u0(pi + 1);
  const int t_first = (int)(ub / nblk), t_last = (int)((ue - 1) / nblk);
  const float s = p.acc->scale;
  const float log2s = log2f(s);             // -inf when s == 0: every dz is then 0

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    mbar_init(smem_u32(&s_full), 1);
    mbar_init(smem_u32(&s_empty), 2);
    for (int b = 0; b < NDZ; ++b) {
      for (int q = 0; q < 4; ++q) mbar_init(smem_u32(&dz_full[b][q]), 4);
      mbar_init(smem_u32(&dz_empty[b]), 1);
    }
    mbar_init(smem_u32(&acc_full), 1);
    mbar_init(smem_u32(&acc_empty), 2);
    mbar_init(smem_u32(&drain_bar), 1);
    mbar_init(smem_u32(&mx_full), 1);
    mbar_init(smem_u32(&lx_full), 1);
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
  const uint32_t tS = tmem + NCH * 128;     // S^T columns after the accumulator chunks

  if (warp == 0 || warp == 10) {
    // ---------------- TMA producers: two warps take alternate stages; in each, lane 0 waits
    // and arms the barrier and each box of the stage is issued by its own lane ----------------
    const int pw = warp == 0 ? 0 : 1;
    if (lane == 0 && pw == 0) {
      tma_prefetch_desc(&tmX);
      tma_prefetch_desc(&tmYs);
      tma_prefetch_desc(&tmYa);
    }
    // both CTAs' loads complete on the leader's barriers, which expect both halves' bytes
    const uint32_t lead_full = mapa(smem_u32(&full[0]), 0);
    int it = 0;
    bool ok = true;
    for (int t = t_first; t <= t_last && ok; ++t) {
      const int b0 = (int)(max(ub, (long long)t * nblk) - (long long)t * nblk);
      const int nb = (int)(min(ue, (long long)(t + 1) * nblk) - (long long)t * nblk) - b0;
      const int x0 = t * G_XT;
      for (int j = 0; j <= nb && ok; ++j) {
        const int nst = (j < nb ? KC : 0) + (j >= 1 ? 4 / AQ : 0);
        for (int u = 0; u < nst; ++u, ++it) {
          if ((it & 1) != pw) continue;
          const int st = it % NST;
          const bool sphase = j < nb && u < KC;
          bool w = true;
          if (lane == 0) {
            w = mbar_wait(smem_u32(&empty[st]), ((it / NST) & 1) ^ 1, WAIT_NS);
            if (!w) record_timeout(p.err, 17);
            else if (rank == 0) mbar_expect_tx(smem_u32(&full[st]), sphase ? 2 * SK * 24576 : 2 * AQ * 16384 * NCH);
          }
          if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
          const uint32_t dst = smem_u32(sY) + st * SLOT;
          const uint32_t bar = lead_full + st * 8;
          if (sphase) {
            // S phase of block b0+j: my 128 stream rows and my 64 X rows, SK atoms of K from 64 SK u
            if (lane == 0) tma_load_3d_cg2(dst, &tmYs, bar, 0, (b0 + j) * G_YB + (int)rank * 128, u * SK);
            else if (lane == 1) tma_load_3d_cg2(dst + SK * 16384, &tmX, bar, 0, x0 + (int)rank * 64, u * SK);
          } else if (lane == 0) {
            // accumulation phase of block b0+j-1, quarters AQ q .. AQ q + AQ - 1 (64 AQ stream rows):
            // my 128 C of every chunk, one 4D box [chunk][atom][64 AQ rows][64]
            const int q = u - (j < nb ? KC : 0);
            const int row = (b0 + j - 1) * G_YB + q * 64 * AQ;
            tma_load_4d_cg2(dst, &tmYa, bar, 0, row, 2 * (int)rank, p.ch0);
          }
          __syncwarp();
        }
      }
    }
  } else if (warp == 1) {
    if (rank == 0) {
      // ---------------- MMA issuer (leader CTA; the peer issues nothing) ----------------
      // The whole warp runs the loop (warp-uniform descriptors); every wait is polled by all
      // lanes and decided together; elect.sync picks the one lane that issues MMAs and commits.
      auto wait_w = [&](uint32_t bar, uint32_t parity, bool cluster, unsigned where) -> bool {
        const bool w = cluster ? mbar_wait_cluster(bar, parity, WAIT_NS) : mbar_wait(bar, parity, WAIT_NS);
        const bool all = __all_sync(0xffffffffu, w);
        if (!all && lane == 0) record_timeout(p.err, where);
        return all;
      };
      const uint32_t idS = idesc_bf16(256, G_XT, 0, 0);
      const uint32_t idA = idesc_bf16(256, G_XT, 1, 1);
      // descriptors of slot 0 / dz buffer 0; an operand elsewhere is the same descriptor plus
      // its byte offset / 16 (start-address field, no carry: shared memory < 256 KB)
      const uint64_t dYs = sdesc_sw128(smem_u32(sY), 16, 1024);             // S phase, K-major
      const uint64_t dXs = sdesc_sw128(smem_u32(sY) + SK * 16384, 16, 1024);
      const uint64_t dYa = sdesc_sw128(smem_u32(sY), AQ * 8192, 1024);      // accumulation, MN-major
      const uint64_t dDZ = sdesc_sw128(smem_u32(sDZ), 32768, 1024);
      bool ok = true;
      int it = 0, g = 0, sg = 0;              // stage counter, global block counter, segment counter
      for (int t = t_first; t <= t_last && ok; ++t, ++sg) {
        const int b0 = (int)(max(ub, (long long)t * nblk) - (long long)t * nblk);
        const int nb = (int)(min(ue, (long long)(t + 1) * nblk) - (long long)t * nblk) - b0;
        for (int j = 0; j <= nb && ok; ++j) {
          if (j < nb) {
            // S^T of block j (the epilogue must have read the previous block's)
            const int gb = g + j;
            if (!wait_w(smem_u32(&s_empty), (gb & 1) ^ 1, true, 21)) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int kc = 0; kc < KC; ++kc, ++it) {
              const int st = it % NST;
              if (!wait_w(smem_u32(&full[st]), (it / NST) & 1, false, 22)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t a = dYs + (uint32_t)(st * (SLOT >> 4));
              const uint64_t b = dXs + (uint32_t)(st * (SLOT >> 4));
              // atom (64 columns: Y 16 KB, X 8 KB apart), then 16-column (32 B) steps
#pragma unroll
              for (int k = 0; k < 4 * SK; ++k)
                mma_ss2_elect(tS, a + ((k >> 2) * 1024 + (k & 3) * 2), b + ((k >> 2) * 512 + (k & 3) * 2), idS,
                              (kc | k) != 0);
              mma_commit_mc2_elect(smem_u32(&empty[st]), 3);
            }
            if (!ok) break;
            mma_commit_mc2_elect(smem_u32(&s_full), 3);
          }
          if (j >= 1) {
            // accumulation of block j-1, one 64-row quarter of dz at a time
            const int jb = j - 1, gb = g + jb, db = gb % NDZ;
            if (jb == 0) {
              // the epilogue must have drained the previous segment's accumulator
              if (!wait_w(smem_u32(&acc_empty), (sg & 1) ^ 1, true, 28)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            for (int q = 0; q < 4 / AQ && ok; ++q) {
              for (int r = 0; r < AQ && ok; ++r) {
                if (!wait_w(smem_u32(&dz_full[db][q * AQ + r]), (gb / NDZ) & 1, true, 23)) ok = false;
              }
              if (!ok) break;
              const int st = it % NST;
              if (!wait_w(smem_u32(&full[st]), (it / NST) & 1, false, 24)) {
                ok = false;
                break;
              }
              ++it;
              tc_fence_after();
              const uint64_t a = dYa + (uint32_t)(st * (SLOT >> 4));
              const uint64_t b = dDZ + (uint32_t)((db * G_DZ + q * AQ * 8192) >> 4);
              // chunk i: AQ * 16 KB apart; K steps of 16 rows: 2 KB apart in both operands
              for (int i = 0; i < NCH; ++i) {
#pragma unroll
                for (int k = 0; k < 4 * AQ; ++k)
                  mma_ss2_elect(tmem + i * 128, a + (i * AQ * 1024 + k * 128), b + k * 128, idA, (jb | q | k) != 0);
              }
              mma_commit_mc2_elect(smem_u32(&empty[st]), 3);
            }
            if (!ok) break;
            mma_commit_mc2_elect(smem_u32(&dz_empty[db]), 3);
            if (jb == nb - 1) mma_commit_mc2_elect(smem_u32(&acc_full), 3);
          }
        }
        g += nb;
      }
      if (!ok) {
        // give up: wait (bounded) for the MMAs already issued before TMEM is released
        mma_commit2_elect(smem_u32(&drain_bar));
        mbar_wait(smem_u32(&drain_bar), 0, WAIT_NS);
      }
    }
  } else if (warp <= 9) {
    // ---------------- epilogue: warps 2..9 ----------------
    // warp -> (TMEM lane quarter q = warp % 4, column half hf); thread = one stream row
    const int q = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int et = (warp - 2) * 32 + lane;        // 0..255 within the epilogue warps
    const int kl = q * 32 + lane;                 // TMEM lane = my stream row in this CTA
    const int kb = (int)rank * 128 + kl;          // row within the 256-row block
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const uint32_t leader_s_empty = mapa(smem_u32(&s_empty), 0);
    const uint32_t leader_acc_empty = mapa(smem_u32(&acc_empty), 0);
    const uint32_t leader_dz_full = mapa(smem_u32(&dz_full[0][0]), 0) + (uint32_t)(kb >> 6) * 8;
    const bool remote = hf != (int)rank;         // column half hf is supplied by CTA hf
    const uint32_t dz_dst = remote ? mapa(smem_u32(sDZ), (uint32_t)hf) : smem_u32(sDZ);
    const uint32_t peer = rank ^ 1u;
    int g = 0, sg = 0;
    for (int t = t_first; t <= t_last; ++t, ++sg) {
      const int b0 = (int)(max(ub, (long long)t * nblk) - (long long)t * nblk);
      const int nb = (int)(min(ue, (long long)(t + 1) * nblk) - (long long)t * nblk) - b0;
      const int x0 = t * G_XT;
      float lacc0 = 0.f, lacc1 = 0.f;             // lse+dh: column sums of p, columns hf*64 + 2 lane (+1)
      if (!DW) {
        // per-column constants of this X tile (tokens): the target, and for the dh pass
        // log2(s) - lse log2(e), for the lse+dh pass the scale of a valid target
        if (et < G_XT) {
          const int n = x0 + et;
          int y = -1;
          float c = -INFINITY;
          if (n < p.N) {
            const int tg = p.targets[n];
            if (tg >= 0 && tg < p.V) {
              y = tg;
              if (!FL) c = log2s - p.lse[n] * LOG2E;
            }
          }
          col_y[et] = y;
          if (FL) fl_s[et] = y >= 0 ? s : 0.f;
          else col_c[et] = c;
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
      }
      for (int j = 0; j < nb; ++j) {
        const int gb = g + j;
        const int ys = (b0 + j) * G_YB + kb;        // my stream row
        // dW pass: my token's target, logsumexp and target logit, loaded while S is computed
        float crow = -INFINITY;                     // log2(s) - lse log2(e), -inf: no gradient
        int xt = -1;                                // my target's column in this X tile
        float fix = 0.f;                            // dz of that element: s (p_t - 1)
        if (DW && ys < p.N) {
          const int tg = p.targets[ys];
          if (tg >= 0 && tg < p.V) {
            const float l2 = p.lse[ys] * LOG2E;
            crow = log2s - l2;
            if (tg >= x0 && tg < x0 + G_XT) {
              xt = tg - x0;
              fix = s * (ex2_approx(fmaf(p.zt[ys], LOG2E, -l2)) - 1.f);
            }
          }
        }
        if (!mbar_wait(smem_u32(&s_full), gb & 1, WAIT_NS)) {
          record_timeout(p.err, 25);
          epi_abort = 1;
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (epi_abort) break;
        tc_fence_after();
        float z[64];
        {
          float v[32];
          tmem_ld32(tS + lane_off + hf * 64, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) z[e] = v[e];
          tmem_ld32(tS + lane_off + hf * 64 + 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) z[32 + e] = v[e];
        }
        tc_fence_before();
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (warp == 2 && lane == 0) {
          if (rank == 0) mbar_arrive(smem_u32(&s_empty));
          else mbar_arrive_cluster(leader_s_empty);
        }
        uint32_t packed[32];
        if (FL) {
          const bool row_ok = ys < p.V;             // rows past the vocabulary are zero-filled: no term
          if (j == 0) {
            // reference m_n: the exact column max of this first block over both CTAs' rows
            float v[64];
#pragma unroll
            for (int e = 0; e < 64; ++e) v[e] = row_ok ? z[e] : -INFINITY;
            col_reduce64<true>(v, lane);
            fl_q[q][hf * 64 + 2 * lane] = v[0];
            fl_q[q][hf * 64 + 2 * lane + 1] = v[1];
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (et < G_XT) {
              const float m = fmaxf(fmaxf(fl_q[0][et], fl_q[1][et]), fmaxf(fl_q[2][et], fl_q[3][et]));
              fl_loc[et] = m;
              st_cluster_f32(mapa(smem_u32(&fl_pm[sg & 1][et]), peer), m);
              fence_acq_rel_cluster();
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (et == 0) {
              mbar_arrive_cluster(mapa(smem_u32(&mx_full), peer));
              if (!mbar_wait_cluster(smem_u32(&mx_full), sg & 1, WAIT_NS)) {
                record_timeout(p.err, 29);
                epi_abort = 1;
              }
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (epi_abort) break;
            if (et < G_XT) col_c[et] = fmaxf(fl_loc[et], fl_pm[sg & 1][et]) * LOG2E;
            asm volatile("bar.sync 1, 256;" ::: "memory");
          }
          // p = 2^(z log2 e - m_n); rows past the vocabulary contribute nothing
          float tmax = -INFINITY;
#pragma unroll
          for (int e = 0; e < 64; ++e) {
            const float tt = fmaf(z[e], LOG2E, -col_c[hf * 64 + e]);
            tmax = fmaxf(tmax, tt);
            z[e] = row_ok ? ex2_approx(tt) : 0.f;
          }
          if (row_ok && tmax > FL_LIMIT) atomicOr(p.tile_flag + t, 1u);
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            __nv_bfloat162 pr = __floats2bfloat162_rn(z[e], z[e + 1]);
            packed[e / 2] = *reinterpret_cast<uint32_t*>(&pr);
          }
          col_reduce64<false>(z, lane);
          lacc0 += z[0];
          lacc1 += z[1];
        } else {
          // s * softmax for my row and column half; rows past the stream end get 0 (dh pass:
          // their W rows are zero-filled and contribute nothing)
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            float c0, c1;
            if (DW) {
              c0 = crow;
              c1 = crow;
            } else {
              c0 = col_c[hf * 64 + e];
              c1 = col_c[hf * 64 + e + 1];
            }
            const float d0 = ex2_approx(fmaf(z[e], LOG2E, c0));
            const float d1 = ex2_approx(fmaf(z[e + 1], LOG2E, c1));
            __nv_bfloat162 pr = __floats2bfloat162_rn(d0, d1);
            packed[e / 2] = *reinterpret_cast<uint32_t*>(&pr);
          }
        }
        // dz buffer db is free once the accumulation NDZ blocks back has completed
        const int db = gb % NDZ;
        if (!mbar_wait(smem_u32(&dz_empty[db]), ((gb / NDZ) & 1) ^ 1, WAIT_NS)) {
          record_timeout(p.err, 26);
          epi_abort = 1;
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t addr = dz_dst + db * G_DZ + sw128_offset(kb, c * 16);
          const uint32_t* w = packed + c * 4;
          if (remote)
            asm volatile("st.shared::cluster.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(w[0]), "r"(w[1]),
                         "r"(w[2]), "r"(w[3])
                         : "memory");
          else
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                         "r"(w[3])
                         : "memory");
        }
        if (DW && xt >= hf * 64 && xt < hf * 64 + 64) {
          __nv_bfloat16 fb = __float2bfloat16_rn(fix);
          st_shared_b16(dz_dst + db * G_DZ + sw128_offset(kb, (xt - hf * 64) * 2), *reinterpret_cast<uint16_t*>(&fb),
                        remote);
        }
        if (remote) fence_proxy_async();
        else fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(leader_dz_full + db * 32);
      }
      // accumulator -> output (whole tile) or partial slot (part of a tile); an abort is
      // acted on only right after a barrier, so every epilogue thread takes the same branch
      if (!mbar_wait(smem_u32(&acc_full), sg & 1, WAIT_NS)) {
        record_timeout(p.err, 27);
        epi_abort = 1;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (epi_abort) break;
      tc_fence_after();
      const bool whole = b0 == 0 && nb == nblk;
      const int slot = 2 * pi + (sg == 0 ? 0 : 1);
      if (FL) {
        // l_n: this CTA's column sums (four lane quarters), then the peer's over DSMEM
        fl_q[q][hf * 64 + 2 * lane] = lacc0;
        fl_q[q][hf * 64 + 2 * lane + 1] = lacc1;
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (et < G_XT) {
          const float l = (fl_q[0][et] + fl_q[1][et]) + (fl_q[2][et] + fl_q[3][et]);
          fl_loc[et] = l;
          st_cluster_f32(mapa(smem_u32(&fl_pl[sg & 1][et]), peer), l);
          fence_acq_rel_cluster();
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (et == 0) {
          mbar_arrive_cluster(mapa(smem_u32(&lx_full), peer));
          if (!mbar_wait_cluster(smem_u32(&lx_full), sg & 1, WAIT_NS)) {
            record_timeout(p.err, 30);
            epi_abort = 1;
          }
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (epi_abort) break;
        if (et < G_XT) {
          // both CTAs add the two halves in rank order: the same l_n in each
          const float mine = fl_loc[et], other = fl_pl[sg & 1][et];
          const float l = rank == 0 ? mine + other : other + mine;
          fl_L[et] = l;
          fl_f[et] = fl_s[et] != 0.f ? fl_s[et] / l : 0.f;
          const int n = x0 + et;
          if (rank == 0) {
            if (whole) {
              if (n < p.N) p.lse_out[n] = (col_c[et] + log2f(l)) * LN2;
            } else {
              p.part_lm[((size_t)slot * 2 + 0) * G_XT + et] = col_c[et];
              p.part_lm[((size_t)slot * 2 + 1) * G_XT + et] = l;
            }
          }
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
      }
      float* part = p.part + (size_t)slot * G_XT * p.C;
      for (int i = 0; i < NCH; ++i) {
        const int c = (p.ch0 + i) * 256 + (int)rank * 128 + kl;   // my C row of the accumulator
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          float v[32];
          tmem_ld32(tmem + i * 128 + lane_off + hf * 64 + cc * 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int xl = hf * 64 + cc * 32 + e;
            const int x = x0 + xl;
            if (!whole) {
              part[(size_t)xl * p.C + c] = v[e];
            } else if (x < nX) {
              if (DW) {
                float* o = p.dW + (size_t)x * p.C + c;
                *o = p.beta ? (*o + v[e]) : v[e];
              } else if (FL) {
                const int y = col_y[xl];
                float val = 0.f;
                if (y >= 0) val = v[e] * fl_f[xl] - fl_s[xl] * __bfloat162float(p.Wt[(size_t)y * p.C + c]);
                p.dh[(size_t)x * p.C + c] = __float2bfloat16_rn(val);
              } else {
                float val = v[e];
                const int y = col_y[xl];
                if (y >= 0) val -= s * __bfloat162float(p.Wt[(size_t)y * p.C + c]);
                p.dh[(size_t)x * p.C + c] = __float2bfloat16_rn(val);
              }
            }
          }
        }
      }
      tc_fence_before();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (warp == 2 && lane == 0) {
        if (rank == 0) mbar_arrive(smem_u32(&acc_empty));
        else mbar_arrive_cluster(leader_acc_empty);
      }
      g += nb;
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

// The X tiles the schedule split between pairs: those holding a pair boundary.
constexpr int MAX_SPLIT_TILES = 160;
struct SplitTiles {
  int n;
  int t[MAX_SPLIT_TILES];
};

// The partial slots of split tile t, in pair order (slot 2q for the pair's first segment).
__device__ __forceinline__ int split_slots(const Sched& sch, int t, int* slots) {
  const long long tb = (long long)t * sch.nblk, te = tb + sch.nblk;
  const int pa = sch.pair_of(tb), pz = sch.pair_of(te - 1);
  int n = 0;
  for (int q = pa; q <= pz && n < 16; ++q) slots[n++] = 2 * q + ((long long)t == sch.u0(q) / sch.nblk ? 0 : 1);
  return n;
}

// Adds the partial sums of every split X tile in pair order and writes the output exactly as
// the gradient kernel does for whole tiles.  grid: (split tiles, ceil(128 * 256 nch / 1024));
// each thread handles four consecutive C columns of one row of the launch's chunk range.
template <int MODE>
__global__ void __launch_bounds__(256) tc_split_combine_kernel(GradParams p, Sched sch, const __grid_constant__ SplitTiles sp) {
  constexpr bool DW = MODE == GM_DW;
  constexpr bool FL = MODE == GM_FL;
  __shared__ int slots[16];
  __shared__ int nslots;
  __shared__ float wts[16][G_XT];   // lse+dh: 2^(m_k - M) per slot and row
  __shared__ float fac[G_XT];       // lse+dh: s / l for a valid target, else 0
  const int t = sp.t[blockIdx.x];
  if (threadIdx.x == 0) nslots = split_slots(sch, t, slots);
  __syncthreads();
  const int nX = DW ? p.V : p.N;
  if (FL && threadIdx.x < G_XT) {
    // merge the slots' (m, l) of my row: M = max m_k, l = sum l_k 2^(m_k - M)
    const int xl = threadIdx.x, x = t * G_XT + xl;
    float M = -INFINITY;
    for (int k = 0; k < nslots; ++k) M = fmaxf(M, p.part_lm[((size_t)slots[k] * 2 + 0) * G_XT + xl]);
    float l = 0.f;
    for (int k = 0; k < nslots; ++k) {
      const float w = exp2f(p.part_lm[((size_t)slots[k] * 2 + 0) * G_XT + xl] - M);
      wts[k][xl] = w;
      l += p.part_lm[((size_t)slots[k] * 2 + 1) * G_XT + xl] * w;
    }
    float f = 0.f;
    if (x < p.N) {
      const int y = p.targets[x];
      if (y >= 0 && y < p.V) f = p.acc->scale / l;
      if (blockIdx.y == 0) p.lse_out[x] = (M + log2f(l)) * LN2;
    }
    fac[xl] = f;
  }
  if (FL) __syncthreads();
  const int idx4 = blockIdx.y * 256 + threadIdx.x;       // index of a group of 4 columns
  const int per_row = p.nch * 64;                         // this launch's C chunks only
  if (idx4 >= G_XT * per_row) return;
  const int xl = idx4 / per_row, c = p.ch0 * 256 + (idx4 % per_row) * 4;
  const int x = t * G_XT + xl;
  if (x >= nX) return;
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < nslots; ++k) {
    const float4 w = *reinterpret_cast<const float4*>(p.part + ((size_t)slots[k] * G_XT + xl) * p.C + c);
    const float a = FL ? wts[k][xl] : 1.f;
    v.x += FL ? w.x * a : w.x;
    v.y += FL ? w.y * a : w.y;
    v.z += FL ? w.z * a : w.z;
    v.w += FL ? w.w * a : w.w;
  }
  if (DW) {
    float4* o = reinterpret_cast<float4*>(p.dW + (size_t)x * p.C + c);
    if (p.beta) {
      const float4 d = *o;
      v.x += d.x;
      v.y += d.y;
      v.z += d.z;
      v.w += d.w;
    }
    *o = v;
  } else {
    const int y = p.targets[x];
    __nv_bfloat16* o = p.dh + (size_t)x * p.C + c;
    if (FL) {
      const float f = fac[xl];
      if (f == 0.f) {
        v = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        const float sc = p.acc->scale;
        const __nv_bfloat16* wr = p.Wt + (size_t)y * p.C + c;
        v.x = v.x * f - sc * __bfloat162float(wr[0]);
        v.y = v.y * f - sc * __bfloat162float(wr[1]);
        v.z = v.z * f - sc * __bfloat162float(wr[2]);
        v.w = v.w * f - sc * __bfloat162float(wr[3]);
      }
    } else if (y >= 0 && y < p.V) {
      const float sc = p.acc->scale;
      const __nv_bfloat16* wr = p.Wt + (size_t)y * p.C + c;
      v.x -= sc * __bfloat162float(wr[0]);
      v.y -= sc * __bfloat162float(wr[1]);
      v.z -= sc * __bfloat162float(wr[2]);
      v.w -= sc * __bfloat162float(wr[3]);
    }
    o[0] = __float2bfloat16_rn(v.x);
    o[1] = __float2bfloat16_rn(v.y);
    o[2] = __float2bfloat16_rn(v.z);
    o[3] = __float2bfloat16_rn(v.w);
  }
}

// ---- per-row pre / post passes of the lse+dh path -----------------------------------------
constexpr int PRE_ROWS = 32;   // rows per block of the pre pass (8 warps x 4 rows)

// Before the lse+dh pass: target validity, the target logit z_t = h_n . W[y_n] (fp32 sum of
// the exact bf16 products; C % 256 == 0), per-block valid counts and error flags, and the
// tile flags cleared.
__global__ void __launch_bounds__(256) rows_pre_kernel(StepArgs a, float* __restrict__ zt, int* __restrict__ part_cnt,
                                                       unsigned* __restrict__ part_err, unsigned* __restrict__ tile_flag,
                                                       int ntiles) {
  __shared__ int sc[8];
  __shared__ unsigned se[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0 && (int)blockIdx.x < ntiles) tile_flag[blockIdx.x] = 0u;
  const __nv_bfloat16* H = static_cast<const __nv_bfloat16*>(a.hidden);
  const __nv_bfloat16* W = static_cast<const __nv_bfloat16*>(a.W);
  int cnt = 0;
  unsigned err = 0;
  for (int r = 0; r < PRE_ROWS / 8; ++r) {
    const int64_t n = (int64_t)blockIdx.x * PRE_ROWS + warp * (PRE_ROWS / 8) + r;
    if (n >= a.N) break;
    const int y = a.targets[n];
    const bool valid = y >= 0 && (int64_t)y < a.V;
    float acc = 0.f;
    if (valid) {
      const uint4* hr = reinterpret_cast<const uint4*>(H + n * a.C);
      const uint4* wr = reinterpret_cast<const uint4*>(W + (int64_t)y * a.C);
      for (int64_t i = lane; i < a.C / 8; i += 32) {
        const uint4 hv = hr[i], wv = wr[i];
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&hv);
        const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&wv);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 hf = __bfloat1622float2(h2[k]), wf = __bfloat1622float2(w2[k]);
          acc = fmaf(hf.x, wf.x, acc);
          acc = fmaf(hf.y, wf.y, acc);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    }
    if (lane == 0) {
      zt[n] = acc;
      cnt += valid ? 1 : 0;
      if (!valid && y != a.ignore_id) err |= ERR_BIT_BAD_TARGET;
    }
  }
  if (lane == 0) {
    sc[warp] = cnt;
    se[warp] = err;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int c = 0;
    unsigned e = 0;
    for (int w = 0; w < 8; ++w) {
      c += sc[w];
      e |= se[w];
    }
    part_cnt[blockIdx.x] = c;
    part_err[blockIdx.x] = e;
  }
}

// After it: row loss lse - z_t and the per-block loss partials for the fixed-order sum.
__global__ void __launch_bounds__(256) rows_post_kernel(StepArgs a, const float* __restrict__ lse,
                                                        const float* __restrict__ zt, double* __restrict__ part_loss,
                                                        unsigned* __restrict__ part_err) {
  __shared__ double sl[256];
  __shared__ unsigned se[256];
  const int t = threadIdx.x;
  const int64_t n = (int64_t)blockIdx.x * 256 + t;
  double loss = 0.0;
  unsigned err = 0;
  if (n < a.N) {
    const int y = a.targets[n];
    if (y >= 0 && (int64_t)y < a.V) {
      const float li = lse[n] - zt[n];
      loss = (double)li;
      if (!isfinite(li)) err |= ERR_BIT_NONFINITE;
      if (a.row_loss) a.row_loss[n] = li;
    } else if (a.row_loss) {
      a.row_loss[n] = 0.f;
    }
  }
  sl[t] = loss;
  se[t] = err;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (t < o) {
      sl[t] += sl[t + o];
      se[t] |= se[t + o];
    }
    __syncthreads();
  }
  if (t == 0) {
    part_loss[blockIdx.x] = sl[0];
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

// The same matrix seen as [cols/64][rows][64]: box {64, box_rows, box_chunks} loads box_chunks
// consecutive 64-column swizzle atoms of box_rows rows in one instruction.
bool make_map3(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_chunks) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, rows, cols / 64};
  cuuint64_t strides[2] = {cols * 2, 128};
  cuuint32_t box[3] = {64, box_rows, box_chunks};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [cols/256][4][rows][64] view: box {64, box_rows, 2, box_chunks} loads, for box_chunks
// consecutive 256-column chunks, two 64-column atoms (this CTA's half of the chunk) of box_rows
// rows in one instruction.
bool make_map4(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_chunks) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {64, rows, 4, cols / 256};
  cuuint64_t strides[3] = {cols * 2, 128, 512};
  cuuint32_t box[4] = {64, box_rows, 2, box_chunks};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
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

int64_t tc_pairs() { return num_sms() / 2; }

size_t tc_part_bytes(int64_t C) { return (size_t)2 * (size_t)tc_pairs() * G_XT * (size_t)C * sizeof(float); }

size_t tc_part_lm_bytes() { return (size_t)2 * (size_t)tc_pairs() * 2 * G_XT * sizeof(float); }


cudaError_t tc_lse(const StepArgs& a, const Scratch& sc, Launch& L) {
  CUtensorMap mh, mw;
  if (!make_map3(&mh, a.hidden, (uint64_t)a.N, (uint64_t)a.C, L_BM, 2) ||
      !make_map3(&mw, a.W, (uint64_t)a.V, (uint64_t)a.C, L_BN, 2))
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
  L.begin(K_FINISH);
  tc_combine_kernel<<<(unsigned)nparts, 256, 0, L.st>>>(sc.tc_part_m, sc.tc_part_l, sc.tc_zt, nsplit, a, sc.lse,
                                                        sc.part_loss, sc.part_cnt, sc.part_err);
  L.end();
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_finish(a, sc, nparts, L);
}

bool tc_grad_supported(int64_t C) { return C % 256 == 0 && C >= 256 && C <= 1024; }

// TMEM holds at most three 256-row C chunks of acc^T beside the logits tile; a wider C runs the
// pass once per range of chunks (each run recomputes the logits).  Ranges as even as possible.
constexpr int TC_MAX_CHUNKS = 3;
int chunk_ranges(int64_t C, int* ch0, int* nch) {
  const int n = (int)(C / 256);
  const int runs = (n + TC_MAX_CHUNKS - 1) / TC_MAX_CHUNKS;
  for (int r = 0; r < runs; ++r) {
    ch0[r] = n * r / runs;
    nch[r] = n * (r + 1) / runs - ch0[r];
  }
  return runs;
}

template <int MODE>
cudaError_t tc_grad_range(const StepArgs& a, const Scratch& sc, Launch& L, int ch0, int nch) {
  constexpr bool DW = MODE == GM_DW;
  const void* X = DW ? a.W : a.hidden;
  const void* Y = DW ? a.hidden : a.W;
  const int64_t nX = DW ? a.V : a.N, nY = DW ? a.N : a.V;
  CUtensorMap mx, mys, mya;
  constexpr int SK = Geo<MODE>::SK, AQ = Geo<MODE>::AQ;
  if (!make_map3(&mx, X, (uint64_t)nX, (uint64_t)a.C, G_XT / 2, SK) ||
      !make_map3(&mys, Y, (uint64_t)nY, (uint64_t)a.C, 128, SK) ||
      !make_map4(&mya, Y, (uint64_t)nY, (uint64_t)a.C, 64 * AQ, (uint32_t)nch))
    return cudaErrorInvalidValue;
  GradParams p;
  p.targets = a.targets;
  p.lse = sc.lse;
  p.zt = sc.tc_zt;
  p.acc = sc.acc;
  p.err = &sc.acc->err;
  p.Wt = static_cast<const __nv_bfloat16*>(a.W);
  p.dW = a.dW;
  p.dh = static_cast<__nv_bfloat16*>(a.dh);
  p.part = sc.tc_part;
  p.part_lm = sc.tc_part_lm;
  p.lse_out = sc.lse;
  p.tile_flag = sc.tc_tile_flag;
  p.N = (int)a.N;
  p.V = (int)a.V;
  p.C = (int)a.C;
  p.ch0 = ch0;
  p.nch = nch;
  p.beta = a.beta;
  const int nblk = (int)((nY + G_YB - 1) / G_YB);
  const int T = (int)((nX + G_XT - 1) / G_XT);
  const long long U = (long long)T * nblk;
  // every pair covers at least a sixth of a tile, so a split tile has a handful of partials
  long long P = tc_pairs();
  if (P > U * 6 / nblk) P = U * 6 / nblk;
  if (P > U) P = U;  // every pair gets at least one unit
  if (P < 1) P = 1;
  const Sched sch{U, (int)P, nblk};
  const int smem = geo_smem_bytes<MODE>();
  cudaFuncSetAttribute(tc_grad_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  L.begin(MODE == GM_DW ? K_DW : MODE == GM_DH ? K_DH : K_LSE_DH);
  tc_grad_kernel<MODE><<<(unsigned)(2 * P), G_THREADS, smem, L.st>>>(mx, mys, mya, p);
  L.end();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  SplitTiles sp;
  sp.n = 0;
  for (int q = 1; q < sch.P; ++q) {
    const long long u = sch.u0(q);
    if (u % nblk == 0) continue;              // the boundary falls between tiles
    const int t = (int)(u / nblk);
    if (sp.n > 0 && sp.t[sp.n - 1] == t) continue;
    if (sp.n == MAX_SPLIT_TILES) return cudaErrorInvalidValue;
    sp.t[sp.n++] = t;
  }
  if (sp.n == 0) return cudaSuccess;
  L.begin(K_FINISH);
  tc_split_combine_kernel<MODE><<<dim3((unsigned)sp.n, (unsigned)((G_XT * 64 * nch + 255) / 256)), 256, 0, L.st>>>(p, sch, sp);
  L.end();
  return cudaGetLastError();
}

template <int MODE>
cudaError_t tc_grad(const StepArgs& a, const Scratch& sc, Launch& L) {
  int ch0[4], nch[4];
  const int runs = chunk_ranges(a.C, ch0, nch);
  for (int r = 0; r < runs; ++r) {
    const cudaError_t e = tc_grad_range<MODE>(a, sc, L, ch0[r], nch[r]);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Default order: the per-row pre pass (target logits, valid count, hence the scale), the
// one-pass logsumexp + dh, the exact repair of flagged tiles (two near-empty launches when
// none is flagged), the row losses, then the dW pass.
static cudaError_t tc_microstep_fused(const StepArgs& a, const Scratch& sc, Launch& L) {
  const int64_t npre = (a.N + PRE_ROWS - 1) / PRE_ROWS;
  const int ntiles = (int)((a.N + TC_TILE_ROWS - 1) / TC_TILE_ROWS);
  L.begin(K_FINISH);
  rows_pre_kernel<<<(unsigned)npre, 256, 0, L.st>>>(a, sc.tc_zt, sc.part_cnt, sc.part_err, sc.tc_tile_flag, ntiles);
  L.end();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if ((e = launch_finish(a, sc, npre, L, FIN_COUNT)) != cudaSuccess) return e;
  if ((e = tc_grad<GM_FL>(a, sc, L)) != cudaSuccess) return e;
  if ((e = simt_repair_lse(a, sc, L)) != cudaSuccess) return e;
  if ((e = simt_repair_dh(a, sc, L)) != cudaSuccess) return e;
  const int64_t nparts = tc_parts(a.N);
  L.begin(K_FINISH);
  rows_post_kernel<<<(unsigned)nparts, 256, 0, L.st>>>(a, sc.lse, sc.tc_zt, sc.part_loss, sc.part_err);
  L.end();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = launch_finish(a, sc, nparts, L, FIN_LOSS)) != cudaSuccess) return e;
  return tc_grad<GM_DW>(a, sc, L);
}

cudaError_t tc_microstep(const StepArgs& a, const Scratch& sc, Launch& L) {
  if (tc_grad_supported(a.C) && !a.tc_two_pass) return tc_microstep_fused(a, sc, L);
  cudaError_t e = tc_lse(a, sc, L);
  if (e != cudaSuccess) return e;
  if (!tc_grad_supported(a.C)) return simt_grads(a, sc, L);
  e = tc_grad<GM_DW>(a, sc, L);
  if (e != cudaSuccess) return e;
  return tc_grad<GM_DH>(a, sc, L);
}

}  // namespace lmce
