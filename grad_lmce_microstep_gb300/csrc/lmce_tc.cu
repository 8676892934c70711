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
// A gradient kernel that gave up waits this long for the MMAs it already issued before it
// releases TMEM, whatever its own wait limit.
constexpr uint64_t DRAIN_NS = 2000000000ull;


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
// column's base-2 reference m_n is fixed once, FL_HEADROOM above the exact maximum over the
// first block of the pair's range (agreed between the two CTAs over DSMEM), and never moved.
// The operand is p = 2^(z log2 e - m_n) and the epilogue also sums p per column (a butterfly
// over the 32 rows of a warp, kept in two registers per lane), so at the end of the range
//   acc^T[c][n] = sum_v W[v][c] p[n][v],   l_n = sum_v p[n][v],
//   dh_n = s (acc^T[.][n] / l_n - W[y_n]),   lse_n = (m_n + log2 l_n) ln 2.
// An element above m_n + fl_limit flags its 128-token tile, and the host then runs the exact
// two-pass repair on flagged tiles only.  fl_limit = 115 - ceil(log2 V) keeps every sum finite:
// l_n <= V 2^fl_limit <= 2^115 and |acc^T| <= 2^115 max|W| < 2^128 for any |W| < 8192 (99 at
// V = 50304).  The headroom moves the guard to FL_HEADROOM + fl_limit above the first block's
// maximum (131 at V = 50304; the widest rows of the logit-stress workload, 1 % of tokens x40,
// reach 100 above it).  It costs nothing in precision: p of the block maximum is 2^-FL_HEADROOM,
// far inside fp32 and bf16 range, and the terms that underflow (p < 2^-126) lie more than
// 126 - FL_HEADROOM = 94 below that maximum, a relative weight under 2^-94.
//
// dW from the stored exponentials (the default dW pass).  The lse+dh pass also writes its bf16
// operand p[n][v] = 2^(z log2 e - m_n) to device memory (one TMA store per epilogue warp and
// block, from the tile it has just written for the MMA) and each row's reference m_n.  Since
//   s (softmax(z_n)[v] - [v == y_n]) = f_n (p[n][v] - [v == y_n] 2^(lse_n log2 e - m_n)),
//   f_n = s 2^(m_n - lse_n log2 e),
// a per-row pass (tc_hs_kernel) replaces each row's target entry of p by the bracket (computed
// in fp32 from the target logit, then rounded once) and writes hs_n = f_n h_n in bf16, and
//   dW^T[c][v] = sum_n hs[n][c] p[n][v]
// is a plain product: the dW pass streams hs and p by TMA into the same accumulation as above,
// with no logits tile and no epilogue work per block.  The segments of a split tile were summed
// with different references (each pair fixes its own), so hs keeps one copy per segment and the
// dW pass takes, for each 128-token tile and 256-row vocabulary block, the copy of the segment
// that covered that pair of indices.  f_n and the target's bracket hold only while m_n lies within
// p_range(s) = min(96, 118 + log2 s) of lse_n log2 e: the bracket stays <= 2^96 and f_n >= 2^-118,
// so that f_n h_n stays a normal bf16 for any |h| >= 2^-8 (96 down to s = 2^-22).  A segment whose
// reference lies further below (its first block's maximum more than p_range + FL_HEADROOM below,
// in base 2: a row whose mass lies in other segments) flags its tile too, and the exact repair
// rewrites the rows of a flagged tile with the normalised p and m_n = lse_n log2 e.  Against recomputing the logits this trades a quarter
// of the tensor work (6 N C V flop per micro-step instead of 8) for one write and one read of
// the N x V bf16 operand, which stream at a small fraction of HBM bandwidth beside the products.
constexpr int G_XT = 128;                  // X rows per pair (64 per CTA)
constexpr int G_YB = 256;                  // stream rows per block (128 per CTA)
constexpr int G_DZ = G_YB * 128;           // one dz buffer: 256 K-rows x 64 bf16 = 32 KB
constexpr int G_EPI_WARPS = 8;
constexpr int G_THREADS = 128 + 32 * G_EPI_WARPS;  // warps 0 and 10 TMA, 1 MMA, 2-9 epilogue, 11 ring waiter

// GM_DWP4: the dW pass from p with four 256-row C chunks (C = 1024) in one run
enum GradMode { GM_DW = 0, GM_DH = 1, GM_FL = 2, GM_DWP = 3, GM_DWP4 = 4 };
// Named barriers of the gradient kernels: 1 the epilogue warps, 2 .. 2 + NST - 1 the ring slots'
// hand-offs from the waiter warp to the MMA warp, then the dz tile's hand-off.
constexpr int HB_DZ_FULL = 6;
constexpr float FL_HEADROOM = 32.f;        // lse+dh pass: reference above the first block's maximum (base 2)
// stored p: largest lse log2 e - m of a row's segment kept (s > 0: the scale)
__host__ __device__ __forceinline__ float p_range(float s) { return s > 0.f ? fminf(96.f, 118.f + log2f(s)) : 96.f; }

// Ring geometry per mode: NST slots of SLOT bytes.  An S stage carries SK 64-column atoms of
// K = C (per CTA: 128 stream rows, then 64 X rows at SK * 16 KB); an accumulation stage
// carries AQ 64-row quarters of the stream block for every 256-row C chunk (per chunk two
// 64-column atoms, AQ * 16 KB); NDZ dz buffers.
// Four 48 KB slots and one dz buffer (4 x 48 + 32 KB dynamic + 3 KB static = the 227 KB a CTA may
// have): with the epilogue finishing a block's dz well before the pipe needs it, a deeper ring
// pays more than a second dz buffer.
template <int MODE>
struct Geo {
  static constexpr int NST = 4, SLOT = 49152, SK = 2, AQ = 1, NDZ = 1, DZB = G_DZ, POFF = 0;
  static_assert(2 + NST <= HB_DZ_FULL, "ring hand-off barriers overlap the dz tile's");
};
// dW from the stored exponentials: a stage is one 64-token quarter of hs (every C chunk, 48 KB)
// and of p (this CTA's 64 vocabulary rows, 8 KB at POFF).  A stage's loads take 1-1.5 us to
// land (in-kernel clock stamps) against ~0.5 us of MMA work per stage, so the ring needs four
// slots; they take all the shared memory, and the flush goes from TMEM straight to global
// memory instead of through a staging buffer.  With four C chunks (C = 1024: TMEM holds all of
// acc^T, there being no logits tile) a stage is 72 KB and three slots cover ~1.3 us of MMA work.
template <>
struct Geo<GM_DWP> {
  static constexpr int POFF = 3 * 16384;
  static constexpr int NST = 4, SLOT = POFF + 8192, SK = 2, AQ = 1, NDZ = 1, DZB = 0;
  static_assert(2 + NST <= HB_DZ_FULL, "ring hand-off barriers overlap the dz tile's");
};
template <>
struct Geo<GM_DWP4> {
  static constexpr int POFF = 4 * 16384;
  static constexpr int NST = 3, SLOT = POFF + 8192, SK = 2, AQ = 1, NDZ = 1, DZB = 0;
  static_assert(2 + NST <= HB_DZ_FULL, "ring hand-off barriers overlap the dz tile's");
};
template <int MODE>
constexpr int geo_smem_bytes() {
  return Geo<MODE>::NST * Geo<MODE>::SLOT + Geo<MODE>::DZB;   // the buffer is declared 1024-aligned
}

struct GradParams {
  const int32_t* targets;
  const float* lse;      // dW and dh passes: per-row logsumexp (natural log)
  float* zt_out;         // lse+dh pass: target logit of each row (from the logits tile)
  const DevAcc* acc;     // scale of this micro-step (when scale_fixed < 0)
  float scale_fixed;     // >= 0: the scale, fixed by the caller's global valid count
  unsigned* err;
  float* dW;             // dW pass output (fp32 [V, C])
  __nv_bfloat16* dh;     // dh / lse+dh pass output (bf16 [N, C])
  const __nv_bfloat16* Wt;  // W, for the one-hot term of dh
  float* part;           // [2 * pairs][128][C] fp32 partial sums of split tiles
  float* part_lm;        // lse+dh pass: [2 * pairs][2][128] (m, l) of split tiles
  float* lse_out;        // lse+dh pass: per-row logsumexp
  unsigned* tile_flag;   // lse+dh pass: per 128-token tile, set when the tile needs the repair
  int N, V, C;
  int ch0, nch;          // 256-row C chunks [ch0, ch0 + nch) of acc^T handled by this launch (nch <= 3;
                         // 4 in the dW pass from p at C = 1024)
  int beta;              // dW pass: 0 writes, 1 adds
  float fl_limit;        // lse+dh pass: largest base-2 exponent of p kept (115 - ceil(log2 V))
  uint64_t wait_ns;      // limit of every bounded wait (WAIT_NS; shorter in the failure-detection test)
  int stall;             // failure-detection test: the producers start no load
  // stored exponentials
  int store_p;           // lse+dh pass: store p (tmE) and the row references
  float* mref;           // lse+dh pass: [TC_MAX_VER][np] reference m of each row per tile segment
  int np;                // rows per segment copy (N rounded up to 256)
  const uint8_t* kmap;   // dW pass from p: segment of (128-token tile, 256-row vocabulary block)
  int kmap_nblk;         // vocabulary blocks per kmap row
  int ttiles;            // 128-token tiles (kmap rows)
};

__device__ __forceinline__ float grad_scale(const GradParams& p) {
  return p.scale_fixed >= 0.f ? p.scale_fixed : p.acc->scale;
}

// Balanced persistent schedule.  Work units are (X tile t, stream block j), t-major; pair pi
// of P takes units [U pi / P, U (pi + 1) / P).  Its range crosses X tiles in segments; a segment
// that covers a whole tile writes the output directly, a segment that covers part of a tile
// (at most the pair's first and last) writes fp32 partial sums to slot 2 pi (first segment) or
// 2 pi + 1, and the split-combine kernels add the partials of each split tile in pair order.
//
// The passes whose stream is the vocabulary (dh, lse+dh), and the dW pass from p (stream: the
// tokens), visit the blocks of X tile t in the rotated order (j + rot(t)) mod nblk, j = 0, 1, ...:
// rot(t) is chosen so that the pair holding most of tile t reaches block (tau mod nblk) at its
// tau-th unit.  All pairs then sweep the stream roughly in phase, and the part of it being read
// at any time is a few blocks instead of the whole operand (every pair at its own offset), so W
// (or the scaled rows of h) is read from DRAM about once per sweep.  The
// order of the blocks within a segment changes no sum's definition: dh and the (max, sum) merge
// are order-free, and the order is a fixed function of the schedule (bitwise reproducible).
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
  __host__ __device__ int rot(int t) const {
    const long long tb = (long long)t * nblk, te = tb + nblk;
    const int pa = pair_of(tb), pz = pair_of(te - 1);
    long long best = -1, tau = 0, j = 0;
    for (int q = pa; q <= pz; ++q) {
      const long long a = u0(q) > tb ? u0(q) : tb, b = u0(q + 1) < te ? u0(q + 1) : te;
      if (b - a > best) {
        best = b - a;
        tau = a - u0(q);
        j = a - tb;
      }
    }
    return (int)(((tau - j) % nblk + nblk) % nblk);
  }
};

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(G_THREADS, 1)
    tc_grad_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmYs,
                   const __grid_constant__ CUtensorMap tmYa, const __grid_constant__ CUtensorMap tmO,
                   const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmE, GradParams p) {
  constexpr bool DW = MODE == GM_DW;
  constexpr bool FL = MODE == GM_FL;
  constexpr bool DWP = MODE == GM_DWP || MODE == GM_DWP4;   // dW from the stored exponentials: no logits tile
  constexpr int P_OFF = Geo<MODE>::POFF;
  constexpr bool DWX = DW || DWP;           // X = vocabulary rows, stream = tokens, output dW
  constexpr int NST = Geo<MODE>::NST, SLOT = Geo<MODE>::SLOT, SK = Geo<MODE>::SK, AQ = Geo<MODE>::AQ;
  constexpr int NDZ = Geo<MODE>::NDZ;
  static_assert(SK * 24576 <= SLOT && AQ * 16384 * 3 <= SLOT && 4 % AQ == 0, "stage does not fit its slot");
  static_assert(!DWP || (AQ == 1 && P_OFF + 8192 <= SLOT), "p quarter does not fit its slot");
  static_assert(!DWP || P_OFF >= 16384, "hs quarter does not fit before p");
  griddep_wait();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte-swizzled operands need 1024-byte alignment; the launch reserves no slack for
  // realigning, so a misaligned buffer is reported (both CTAs of the pair see the same layout
  // and leave together) instead of being used
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_timeout(p.err, 31);
    return;
  }
  uint8_t* smem = smem_raw;
  const int KC = DWP ? 0 : p.C / (64 * SK);   // S phase stages per block
  const int NCH = p.nch;                    // 256-row C chunks of acc^T in TMEM (from chunk p.ch0 on)
  uint8_t* sY = smem;                       // ring of NST slots
  uint8_t* sDZ = sY + NST * SLOT;           // [NDZ][4 K atoms][64 X rows][128 B], K-major
  __shared__ __align__(8) uint64_t full[NST], empty[NST];
  __shared__ __align__(8) uint64_t s_full, s_empty, dz_full[NDZ], dz_empty[NDZ], acc_full, acc_empty, drain_bar;
  __shared__ __align__(8) uint64_t lx_full;   // lse+dh pass: the peer's s / l_x arrived
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int epi_abort;
  __shared__ volatile int wt_abort;         // the ring waiter gave up on a stage
  __shared__ __align__(16) float col_c[G_YB];  // dW: per stream token log2(s) - lse log2(e), or -inf (read as float4)
  __shared__ int hit_cnt[2];                // dW: one-hot hits of the block (by block parity)
  __shared__ uint16_t hit[2][G_YB];         // dW: (token in block) << 8 | X row in tile
  __shared__ float fl_red[4][64];           // lse+dh: row max / sum over each 64-column quarter
  __shared__ float fl_f[G_XT];              // lse+dh: s / l_x for a valid target, else 0 (both CTAs' rows)
  __shared__ int col_y[G_XT];               // dh, lse+dh: target of each X row (token) of the tile, or -1
  __shared__ int s_rot;                     // dh, lse+dh: the tile's vocabulary rotation

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint64_t wait_ns = p.wait_ns;
  const int nX = DWX ? p.V : p.N;
  const int nY = DWX ? p.N : p.V;
  const int nblk = (nY + G_YB - 1) / G_YB;
  const int T = (nX + G_XT - 1) / G_XT;
  const Sched sch{(long long)T * nblk, (int)(gridDim.x >> 1), nblk};
  const int pi = blockIdx.x >> 1;
  const long long ub = sch.u0(pi), ue = sch.u0(pi + 1);
  const int t_first = (int)(ub / nblk), t_last = (int)((ue - 1) / nblk);
  const float s = grad_scale(p);
  const float log2s = log2f(s);             // -inf when s == 0: every dz is then 0

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    mbar_init(smem_u32(&s_full), 1);
    mbar_init(smem_u32(&s_empty), 2);
    for (int b = 0; b < NDZ; ++b) {
      mbar_init(smem_u32(&dz_full[b]), 16);    // every epilogue warp of both CTAs, once per block
      mbar_init(smem_u32(&dz_empty[b]), 1);
    }
    mbar_init(smem_u32(&acc_full), 1);
    mbar_init(smem_u32(&acc_empty), 2);
    mbar_init(smem_u32(&drain_bar), 1);
    mbar_init(smem_u32(&lx_full), 1);
    hit_cnt[0] = 0;
    hit_cnt[1] = 0;
    epi_abort = 0;
    wt_abort = 0;
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
  const uint32_t tS = tmem + NCH * 128;     // S tile columns after the accumulator chunks

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
    // dW from p: the hs copy of each 128-token tile of the block being loaded (lane 0, read one
    // block ahead so that the table's latency stays off the loads)
    int kv_cur0 = 0, kv_cur1 = 0, kv_nxt0 = 0, kv_nxt1 = 0;
    auto kver = [&](int t1, int vb) -> int {
      if (t1 >= p.ttiles) return 0;   // tokens past the last tile: zero rows of copy 0
      const int k = __ldg(p.kmap + (size_t)t1 * p.kmap_nblk + vb);
      return dcheck(k < TC_MAX_VER, p.err, BS_TMA_ROW) ? k : 0;
    };
    for (int t = t_first; t <= t_last && ok; ++t) {
      const int b0 = (int)(max(ub, (long long)t * nblk) - (long long)t * nblk);
      const int nb = (int)(min(ue, (long long)(t + 1) * nblk) - (long long)t * nblk) - b0;
      const int x0 = t * G_XT;
      const int rt = DW ? 0 : sch.rot(t);
      auto rblk = [&](int jj) { const int b = b0 + jj + rt; return b < nblk ? b : b - nblk; };
      if (DWP && lane == 0) {
        kv_nxt0 = kver(2 * rblk(0), t >> 1);
        kv_nxt1 = kver(2 * rblk(0) + 1, t >> 1);
      }
      for (int j = 0; j <= nb && ok; ++j) {
        const int nst = (j < nb ? KC : 0) + (j >= 1 ? 4 / AQ : 0);
        if (DWP && pw == 0 && lane == 0) {
          // p of block b0+j+1 (first also of b0+j) into L2 two blocks before its loads: p comes
          // from DRAM, and the ring covers only a block's worth of load latency
          for (int jj = (j == 0 ? 0 : j + 1); jj <= j + 1 && jj < nb; ++jj)
            for (int q = 0; q < 4; ++q) tma_prefetch_3d(&tmX, 0, rblk(jj) * G_YB + q * 64, 2 * t + (int)rank);
        }
        if (DWP && j >= 1 && lane == 0) {
          kv_cur0 = kv_nxt0;
          kv_cur1 = kv_nxt1;
          if (j < nb) {
            kv_nxt0 = kver(2 * rblk(j), t >> 1);
            kv_nxt1 = kver(2 * rblk(j) + 1, t >> 1);
          }
        }
        for (int u = 0; u < nst; ++u, ++it) {
          if ((it & 1) != pw) continue;
          const int st = it % NST;
          const bool sphase = j < nb && u < KC;
          bool w = true;
          if (lane == 0) {
            w = mbar_wait(smem_u32(&empty[st]), ((it / NST) & 1) ^ 1, wait_ns);
            if (!w) record_timeout(p.err, 17);
            else if (rank == 0)
              mbar_expect_tx(smem_u32(&full[st]), sphase ? 2 * SK * 24576 : DWP ? 2 * (16384 * NCH + 8192) : 2 * AQ * 16384 * NCH);
          }
          if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
          const uint32_t dst = smem_u32(sY) + st * SLOT;
          const uint32_t bar = lead_full + st * 8;
          if (p.stall) {
            // failure-detection test: no load starts, so every wait on this stage runs out
          } else if (sphase) {
            // S phase of block b0+j: my 128 stream rows and my 64 X rows, SK atoms of K from 64 SK u
            const int bj = b0 + j + rt;   // < 2 nblk
            if (lane == 0) dcheck(bj < 2 * nblk && t < T, p.err, BS_TMA_ROW);
            if (lane == 0) tma_load_3d_cg2(dst, &tmYs, bar, 0, (bj < nblk ? bj : bj - nblk) * G_YB + (int)rank * 128, u * SK);
            else if (lane == 1) tma_load_3d_cg2(dst + SK * 16384, &tmX, bar, 0, x0 + (int)rank * 64, u * SK);
          } else if (DWP) {
            // block b0+j-1, quarter q (64 tokens): hs rows of the quarter's segment copy, my 128 C
            // of every chunk; p rows of the same tokens, my 64 vocabulary rows of the tile
            const int q = u;
            const int bj = rblk(j - 1);
            if (lane == 0) {
              dcheck(bj < nblk && q < 4, p.err, BS_TMA_ROW);
              const int kv = (q >> 1) ? kv_cur1 : kv_cur0;
              tma_load_4d_cg2(dst, &tmYa, bar, 0, kv * p.np + bj * G_YB + q * 64, 2 * (int)rank, p.ch0);
            } else if (lane == 1) {
              tma_load_3d_cg2_hint(dst + P_OFF, &tmX, bar, 0, bj * G_YB + q * 64, 2 * t + (int)rank, policy_evict_first());
            }
          } else if (lane == 0) {
            // accumulation phase of block b0+j-1, quarters AQ q .. AQ q + AQ - 1 (64 AQ stream rows):
            // my 128 C of every chunk, one 4D box [chunk][atom][64 AQ rows][64]
            const int q = u - (j < nb ? KC : 0);
            const int bj = b0 + j - 1 + rt;   // < 2 nblk
            dcheck(bj < 2 * nblk && q < 4 / AQ, p.err, BS_TMA_ROW);
            const int row = (bj < nblk ? bj : bj - nblk) * G_YB + q * 64 * AQ;
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
        const bool w = cluster ? mbar_wait_cluster(bar, parity, wait_ns) : mbar_wait(bar, parity, wait_ns);
        const bool all = __all_sync(0xffffffffu, w);
        if (!all && lane == 0) record_timeout(p.err, where);
        return all;
      };
      // A ring stage is taken from the waiter warp through its slot's named barrier (below).
      auto ring_take = [&](int st) { asm volatile("bar.sync %0, 64;" ::"r"(2 + st) : "memory"); };
      // S = X . Y_blk^T: M = 128 X rows (64 per CTA), N = 256 stream rows (128 per CTA), K-major
      const uint32_t idS = idesc_bf16(128, G_YB, 0, 0);
      // acc^T += Y_blk^T . dz: M = 256 C rows per chunk (MN-major), N = 128 X rows (K-major dz)
      const uint32_t idA = idesc_bf16(256, G_XT, 1, 0);
      // descriptors of slot 0 / dz buffer 0; an operand elsewhere is the same descriptor plus
      // its byte offset / 16 (start-address field, no carry: shared memory < 256 KB)
      const uint64_t dYs = sdesc_sw128(smem_u32(sY), 16, 1024);             // S phase, K-major
      const uint64_t dXs = sdesc_sw128(smem_u32(sY) + SK * 16384, 16, 1024);
      const uint64_t dYa = sdesc_sw128(smem_u32(sY), AQ * 8192, 1024);      // accumulation, MN-major
      const uint64_t dDZ = sdesc_sw128(smem_u32(sDZ), 16, 1024);            // dz, K-major
      // dW from p: B = the quarter's p rows, MN-major (64 vocabulary rows of 128 B per token, one
      // 64-wide atom per CTA, K groups of 8 tokens 1 KB apart)
      const uint32_t idP = idesc_bf16(256, G_XT, 1, 1);
      const uint64_t dP = sdesc_sw128(smem_u32(sY) + P_OFF, 8192, 1024);
      // the block's dz tile, handed over by the waiter warp through named barrier HB_DZ_FULL
      auto dz_take = [&]() -> bool {
        asm volatile("bar.sync %0, 64;" ::"n"(HB_DZ_FULL) : "memory");
        return !wt_abort;
      };
      bool ok = true;
      int it = 0, g = 0, sg = 0;              // stage counter, global block counter, segment counter
      for (int t = t_first; t <= t_last && ok; ++t, ++sg) {
        const int b0 = (int)(max(ub, (long long)t * nblk) - (long long)t * nblk);
        const int nb = (int)(min(ue, (long long)(t + 1) * nblk) - (long long)t * nblk) - b0;
        for (int j = 0; j <= nb && ok; ++j) {
          if (!DWP && j < nb) {
            // S of block j (the epilogue must have read the previous block's)
            const int gb = g + j;
            if (!wait_w(smem_u32(&s_empty), (gb & 1) ^ 1, true, 21)) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int kc = 0; kc < KC; ++kc, ++it) {
              const int st = it % NST;
              ring_take(st);
              if (wt_abort) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t a = dXs + (uint32_t)(st * (SLOT >> 4));
              const uint64_t b = dYs + (uint32_t)(st * (SLOT >> 4));
              // atom (64 columns: X 8 KB, Y 16 KB apart), then 16-column (32 B) steps
#pragma unroll
              for (int k = 0; k < 4 * SK; ++k)
                mma_ss2_elect(tS, a + ((k >> 2) * 512 + (k & 3) * 2), b + ((k >> 2) * 1024 + (k & 3) * 2), idS,
                              (kc | k) != 0);
              mma_commit_mc2_elect(smem_u32(&empty[st]), 3);
            }
            if (!ok) break;
            mma_commit_mc2_elect(smem_u32(&s_full), 3);
          }
          if (j >= 1) {
            // accumulation of block j-1, AQ 64-row quarters of dz at a time
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
              // the whole dz tile of the block (one wait per block: the epilogue is far ahead)
              if (!DWP && q == 0 && !dz_take()) {
                ok = false;
                break;
              }
              const int st = it % NST;
              ring_take(st);
              if (wt_abort) {
                ok = false;
                break;
              }
              ++it;
              tc_fence_after();
              const uint64_t a = dYa + (uint32_t)(st * (SLOT >> 4));
              if (DWP) {
                // K steps of 16 tokens: A and p both 2 KB apart
                const uint64_t b = dP + (uint32_t)(st * (SLOT >> 4));
                for (int i = 0; i < NCH; ++i) {
#pragma unroll
                  for (int k = 0; k < 4; ++k)
                    mma_ss2_elect(tmem + i * 128, a + (i * 1024 + k * 128), b + k * 128, idP, (jb | q | k) != 0);
                }
              } else {
                const uint64_t b = dDZ + (uint32_t)((db * G_DZ + q * AQ * 8192) >> 4);
                // chunk i: AQ * 16 KB apart; K steps of 16 rows: A 2 KB apart, dz 32 B within its
                // 64-row K atom (atoms 8 KB apart)
                for (int i = 0; i < NCH; ++i) {
#pragma unroll
                  for (int k = 0; k < 4 * AQ; ++k)
                    mma_ss2_elect(tmem + i * 128, a + (i * AQ * 1024 + k * 128), b + ((k >> 2) * 512 + (k & 3) * 2),
                                  idA, (jb | q | k) != 0);
                }
              }
              mma_commit_mc2_elect(smem_u32(&empty[st]), 3);
            }
            if (!ok) break;
            if (!DWP) mma_commit_mc2_elect(smem_u32(&dz_empty[db]), 3);
            if (jb == nb - 1) mma_commit_mc2_elect(smem_u32(&acc_full), 3);
          }
        }
        g += nb;
      }
      if (!ok) {
        // give up: wait (bounded) for the MMAs already issued before TMEM is released
        mma_commit2_elect(smem_u32(&drain_bar));
        mbar_wait(smem_u32(&drain_bar), 0, DRAIN_NS);
      }
    }
  } else if (warp == 11) {
    // ---------------- ring waiter (leader CTA) ----------------
    // Waits on each ring stage's full barrier in the MMA warp's order and hands the stage over
    // through named barrier 2 + slot; before a block's accumulation stages it also waits for
    // that block's dz tile and hands it over through HB_DZ_FULL.  An mbarrier wait in the MMA warp
    // itself sits behind the MMAs it has just issued and took ~190 cycles even on a completed
    // phase, long enough for the tensor pipe to run dry after every stage; a named barrier does
    // not.  The waiter is at most NST stages ahead (a slot refills only after the MMA warp took
    // it) and one dz tile ahead (the next one is written only after the accumulation that the MMA
    // warp issues after taking this one), so every barrier sees one arrival per use.  (The S
    // tile's release stays an mbarrier wait of the MMA warp: handed over too, it measured slower,
    // since the waiter then stalls on it before the ring stages behind it.)  A wait that runs out
    // sets wt_abort, which the MMA warp reads after its barrier.
    if (rank == 0) {
      bool ok = true;
      int it = 0, g = 0;
      for (int t = t_first; t <= t_last && ok; ++t) {
        const int b0 = (int)(max(ub, (long long)t * nblk) - (long long)t * nblk);
        const int nb = (int)(min(ue, (long long)(t + 1) * nblk) - (long long)t * nblk) - b0;
        for (int j = 0; j <= nb && ok; ++j) {
          const int nst = (j < nb ? KC : 0) + (j >= 1 ? 4 / AQ : 0);
          for (int u = 0; u < nst; ++u, ++it) {
            if (!DWP && j >= 1 && u == (j < nb ? KC : 0)) {
              // block j - 1's dz tile, before its first accumulation stage
              const int gb = g + j - 1;
              const bool wd =
                  __all_sync(0xffffffffu, mbar_wait_cluster(smem_u32(&dz_full[gb % NDZ]), (gb / NDZ) & 1, wait_ns));
              if (!wd) {
                if (lane == 0) record_timeout(p.err, 23);
                wt_abort = 1;
                ok = false;
              }
              __syncwarp();
              asm volatile("bar.arrive %0, 64;" ::"n"(HB_DZ_FULL) : "memory");
              if (!ok) break;
            }
            const int st = it % NST;
            const bool w = __all_sync(0xffffffffu, mbar_wait(smem_u32(&full[st]), (it / NST) & 1, wait_ns));
            if (!w) {
              if (lane == 0) record_timeout(p.err, 29);
              wt_abort = 1;
              ok = false;
            }
            __syncwarp();
            asm volatile("bar.arrive %0, 64;" ::"r"(2 + st) : "memory");
            if (!ok) break;
          }
        }
        g += nb;
      }
    }
  } else if (warp <= 9) {
    // ---------------- epilogue: warps 2..9 ----------------
    // The S tile holds this CTA's 64 X rows x the block's 256 stream rows: TMEM lanes 0-63 the
    // stream columns 0-127, lanes 64-127 the columns 128-255 (128 TMEM columns).  Warp -> TMEM
    // lane quarter qd = warp % 4 and column half hf; thread = one X row and 64 stream columns,
    // i.e. one 64-column K atom of the dz operand, which it writes as one swizzled 128-byte row.
    const int qd = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int et = (warp - 2) * 32 + lane;        // 0..255 within the epilogue warps
    const int xr = 32 * (qd & 1) + lane;          // my X row in this CTA (0..63)
    const int xl = (int)rank * 64 + xr;           // my X row in the pair's 128-row tile
    const int ks = (qd >> 1) * 2 + hf;            // my 64-column quarter of the stream block
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const uint32_t leader_s_empty = mapa(smem_u32(&s_empty), 0);
    const uint32_t leader_acc_empty = mapa(smem_u32(&acc_empty), 0);
    // dz buffer b: leader's dz_full[b] (16 arrivals: every epilogue warp of both CTAs)
    const uint32_t dzf = mapa(smem_u32(&dz_full[0]), 0);
    const uint32_t dz_row = smem_u32(sDZ) + ks * 8192;   // + buffer * G_DZ, row xr
    const uint32_t peer = rank ^ 1u;
    if (et == 0) {
      tma_prefetch_desc(&tmO);
      tma_prefetch_desc(&tmP);
    }
    int g = 0, sg = 0;
    // dh passes, whole tiles: the one-hot rows W[y] of a 256-column chunk, 16 B per thread and row
    // (16 threads per 256-byte row, rows wr + 16 j), loaded one chunk ahead of their use
    const int wr = et >> 4, ws = et & 15;
    uint4 wv[8];
    auto wload = [&](int i) {
      const int c0 = (p.ch0 + i) * 256 + (int)rank * 128;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        int y = col_y[wr + 16 * j];   // rows without a target read row 0 and ignore it
        if (!dcheck(y < p.V, p.err, BS_W_ROW)) y = 0;
        wv[j] = __ldg(reinterpret_cast<const uint4*>(p.Wt + (size_t)(y >= 0 ? y : 0) * p.C + c0) + ws);
      }
    };
    for (int t = t_first; t <= t_last; ++t, ++sg) {
      const int b0 = (int)(max(ub, (long long)t * nblk) - (long long)t * nblk);
      const int nb = (int)(min(ue, (long long)(t + 1) * nblk) - (long long)t * nblk) - b0;
      const int x0 = t * G_XT;
      const int xg = x0 + xl;                     // my X row
      // the tile's vocabulary rotation, found by one thread; read after the block loop's first
      // barrier (the previous tile's readers are past the flush's barriers)
      if (!DWX && et == 0) s_rot = sch.rot(t);
      // dh / lse+dh: my token's target and (dh) log2(s) - lse log2(e); the targets of all 128
      // rows of the tile for the flush
      float crow = -INFINITY;
      int yrow = -1;
      if (!DWX) {
        if (xg < p.N) {
          const int tg = p.targets[xg];
          if (tg >= 0 && tg < p.V) {
            yrow = tg;
            if (!FL) crow = log2s - p.lse[xg] * LOG2E;
          }
        }
        if (et < G_XT) {
          const int n = x0 + et;
          int y = -1;
          if (n < p.N) {
            const int tg = p.targets[n];
            if (tg >= 0 && tg < p.V) y = tg;
          }
          col_y[et] = y;
        }
      }
      float m2 = 0.f, lacc = 0.f;                 // lse+dh: my row's reference (base 2) and sum of p
      // dW from p: no logits tile, nothing to do per block
      for (int j = 0; j < (DWP ? 0 : nb); ++j) {
        const int gb = g + j;
        // first stream row of the block (dh passes: rotated; read after the barrier below)
        const int ys0 = DW ? (b0 + j) * G_YB : 0;
        // dW: stream token et's constant and one-hot hit, loaded while S is computed
        float cc = -INFINITY;
        int hr = -1;
        if (DW) {
          const int n = ys0 + et;
          if (n < p.N) {
            const int tg = p.targets[n];
            if (tg >= 0 && tg < p.V) {
              cc = log2s - p.lse[n] * LOG2E;
              if (tg >= x0 && tg < x0 + G_XT) hr = tg - x0;
            }
          }
        }
        if (!mbar_wait(smem_u32(&s_full), gb & 1, wait_ns)) {
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
        if (DW) {
          // this block's per-token constants and hits (last block's readers are past the barrier above)
          col_c[et] = cc;
          if (et == 0) hit_cnt[(gb + 1) & 1] = 0;
          if (hr >= 0) {
            const int hi = atomicAdd(&hit_cnt[gb & 1], 1);
            if (dcheck(hi < G_YB, p.err, BS_HIT)) hit[gb & 1][hi] = (uint16_t)((et << 8) | hr);
          }
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (warp == 2 && lane == 0) {
          if (rank == 0) mbar_arrive(smem_u32(&s_empty));
          else mbar_arrive_cluster(leader_s_empty);
        }
        if (FL) {
          const int bj = b0 + j + s_rot;   // < 2 nblk
          const int ys0 = (bj < nblk ? bj : bj - nblk) * G_YB;
          // columns past the vocabulary (last block only) carry no term
          const int nvalid = min(64, p.V - (ys0 + ks * 64));
          if (j == 0) {
            // reference m: FL_HEADROOM above the exact maximum of my row over this first block
            // (four quarters)
            float mx = -INFINITY;
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (e < nvalid) mx = fmaxf(mx, z[e]);
            fl_red[ks][xr] = mx;
            asm volatile("bar.sync 1, 256;" ::: "memory");
            m2 = fmaf(fmaxf(fmaxf(fl_red[0][xr], fl_red[1][xr]), fmaxf(fl_red[2][xr], fl_red[3][xr])), LOG2E,
                      FL_HEADROOM);
          }
          // my row's target logit, when its column falls in my quarter of this block
          const int tq = yrow - (ys0 + ks * 64);
          if (tq >= 0 && tq < 64) {
            float zv = 0.f;
#pragma unroll
            for (int e = 0; e < 64; ++e) zv = (tq == e) ? z[e] : zv;
            p.zt_out[xg] = zv;
          }
          // p = 2^(z log2 e - m); its row sum in four partial accumulators (fixed order)
          float tmax = -INFINITY, ps0 = 0.f, ps1 = 0.f, ps2 = 0.f, ps3 = 0.f;
#pragma unroll
          for (int e = 0; e < 64; ++e) {
            const float tt = fmaf(z[e], LOG2E, -m2);
            const float pv = e < nvalid ? ex2_approx(tt) : 0.f;
            if (e < nvalid) tmax = fmaxf(tmax, tt);
            z[e] = pv;
            if ((e & 3) == 0) ps0 += pv;
            else if ((e & 3) == 1) ps1 += pv;
            else if ((e & 3) == 2) ps2 += pv;
            else ps3 += pv;
          }
          lacc += (ps0 + ps1) + (ps2 + ps3);
          if (tmax > p.fl_limit && dcheck(t < T, p.err, BS_TILE_FLAG)) atomicOr(p.tile_flag + t, 1u);
        } else if (DW) {
          // my columns whose token targets my row: dz there is s (p - 1)
          uint64_t fix = 0;
          const int nh = hit_cnt[gb & 1];
          for (int i = 0; i < nh; ++i) {
            const int hv = hit[gb & 1][i];
            if ((hv & 255) == xl && (hv >> 14) == ks) fix |= 1ull << ((hv >> 8) & 63);
          }
          // s * softmax per token column (its constant from the table), minus s at the hits
#pragma unroll
          for (int e = 0; e < 64; e += 4) {
            const float4 c4 = *reinterpret_cast<const float4*>(&col_c[ks * 64 + e]);
            z[e] = ex2_approx(fmaf(z[e], LOG2E, c4.x)) - ((fix >> e) & 1 ? s : 0.f);
            z[e + 1] = ex2_approx(fmaf(z[e + 1], LOG2E, c4.y)) - ((fix >> (e + 1)) & 1 ? s : 0.f);
            z[e + 2] = ex2_approx(fmaf(z[e + 2], LOG2E, c4.z)) - ((fix >> (e + 2)) & 1 ? s : 0.f);
            z[e + 3] = ex2_approx(fmaf(z[e + 3], LOG2E, c4.w)) - ((fix >> (e + 3)) & 1 ? s : 0.f);
          }
        } else {
          // s * softmax of my row (its constant); stream rows past the vocabulary have zero W
#pragma unroll
          for (int e = 0; e < 64; ++e) z[e] = ex2_approx(fmaf(z[e], LOG2E, crow));
        }
        uint32_t packed[32];
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          __nv_bfloat162 pr = __floats2bfloat162_rn(z[e], z[e + 1]);
          packed[e / 2] = *reinterpret_cast<uint32_t*>(&pr);
        }
        // dz buffer db is free once the accumulation NDZ blocks back has completed
        const int db = gb % NDZ;
        if (!mbar_wait(smem_u32(&dz_empty[db]), ((gb / NDZ) & 1) ^ 1, wait_ns)) {
          record_timeout(p.err, 26);
          epi_abort = 1;
        }
        if (FL && p.store_p) {
          // and once this warp's store of the previous block's p rows has read them
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
        }
        // my row of K atom ks, K-major, 128-byte swizzle: all in this CTA's shared memory
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t addr = dz_row + db * G_DZ + sw128_offset(xr, c * 16);
          const uint32_t* w = packed + c * 4;
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                       : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive(smem_u32(&dz_full[db]));
          else mbar_arrive_cluster(dzf + db * 8);
          const int row0 = x0 + (int)rank * 64 + 32 * (qd & 1);
          if (FL && p.store_p && row0 < p.N) {
            // the warp's 32 rows x 64 columns of p, as written for the MMA, to p[tokens][vocabulary]
            // (a box may reach past row N, clipped, but never starts there)
            const int bj = b0 + j + s_rot;
            const int vb = bj < nblk ? bj : bj - nblk;
            tma_store_3d_hint(&tmE, dz_row + db * G_DZ + (uint32_t)(qd & 1) * 4096, 0, row0, vb * 4 + ks,
                              policy_evict_first());   // read once, by the dW pass
            bulk_commit();
          }
        }
      }
      // the dz buffer also stages the flush: every store of p has read it
      if (FL && p.store_p && lane == 0) bulk_wait_read0();
      // accumulator -> output (whole tile) or partial slot (part of a tile); an abort is
      // acted on only right after a barrier, so every epilogue thread takes the same branch
      const bool whole = b0 == 0 && nb == nblk;
      if (!DWX && whole) wload(0);   // in flight while the last accumulation completes
      if (!mbar_wait(smem_u32(&acc_full), sg & 1, wait_ns)) {
        record_timeout(p.err, 27);
        epi_abort = 1;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (epi_abort) break;
      tc_fence_after();
      const int slot = 2 * pi + (sg == 0 ? 0 : 1);
      // the launch has at most tc_pairs() pairs: a slot past the partial buffer is reported and
      // its plain stores skipped (its TMA stores are clipped to the buffer's rows)
      const bool slot_ok = dcheck(slot < (int)gridDim.x, p.err, BS_SLOT);
      if (FL) {
        // l_x of my rows (four quarters, fixed order); s / l_x for both CTAs' rows via DSMEM
        fl_red[ks][xr] = lacc;
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (ks == 0) {
          const float l = (fl_red[0][xr] + fl_red[1][xr]) + (fl_red[2][xr] + fl_red[3][xr]);
          const float f = yrow >= 0 ? s / l : 0.f;
          fl_f[xl] = f;
          st_cluster_f32(mapa(smem_u32(&fl_f[xl]), peer), f);
          if (p.store_p && xg < p.N) {
            // the reference of this segment of the tile (segment k = pairs since the tile's first)
            const int kseg = pi - sch.pair_of((long long)t * nblk);
            if (dcheck(kseg < TC_MAX_VER, p.err, BS_SLOT)) p.mref[(size_t)kseg * p.np + xg] = m2;
          }
          if (whole) {
            if (xg < p.N) p.lse_out[xg] = (m2 + log2f(l)) * LN2;
            // stored p: the row's only reference must lie within p_range of its lse log2 e
            if (p.store_p && yrow >= 0 && !(log2f(l) <= p_range(s)) && dcheck(t < T, p.err, BS_TILE_FLAG))
              atomicOr(p.tile_flag + t, 1u);
          } else if (slot_ok) {
            p.part_lm[((size_t)slot * 2 + 0) * G_XT + xl] = m2;
            p.part_lm[((size_t)slot * 2 + 1) * G_XT + xl] = l;
          }
          fence_acq_rel_cluster();
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (et == 0) {
          mbar_arrive_cluster(mapa(smem_u32(&lx_full), peer));
          if (!mbar_wait_cluster(smem_u32(&lx_full), sg & 1, wait_ns)) {
            record_timeout(p.err, 30);
            epi_abort = 1;
          }
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (epi_abort) break;
      }
      // acc^T in TMEM: lane = C row, column = X row of the tile; thread: lane quarter qd (C rows
      // qd*32 + lane of this CTA's 128 per chunk), columns from hf*64.  The recomputing dW pass
      // and whole dh tiles leave through the dz buffer (idle: the segment's accumulation has
      // completed) by TMA, so the flush is not limited by the rate at which one SM retires
      // scattered stores; the dW pass from p has no such buffer (its ring takes all of shared
      // memory) and writes from registers:
      //  - dW pass: 16-column rounds through two 16 KB halves, each round two boxes of 16 X rows
      //    x 128 C (accumulating into dW: reduce-add at L2; else stores; partial tiles: stores);
      //  - bf16 dh of a whole tile: one 256-column chunk at a time; the rows W[y] of its one-hot
      //    term are first stored into the buffer (row x at 256 B x) and dh overwrites them.
      const int kl = qd * 32 + lane;
      const uint32_t stg = smem_u32(sDZ);
      if (!DWX && whole) {
        __nv_bfloat16* sw = reinterpret_cast<__nv_bfloat16*>(sDZ);
        for (int i = 0; i < NCH; ++i) {
          const int c0 = (p.ch0 + i) * 256 + (int)rank * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(sDZ + (wr + 16 * j) * 256 + ws * 16) = wv[j];
          asm volatile("bar.sync 1, 256;" ::: "memory");
          if (i + 1 < NCH) wload(i + 1);
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            float v[32];
            tmem_ld32(tmem + i * 128 + lane_off + hf * 64 + cc * 32, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int xc = hf * 64 + cc * 32 + e;
              __nv_bfloat16* q = sw + xc * 128 + kl;
              float val = 0.f;
              if (col_y[xc] >= 0) val = (FL ? v[e] * fl_f[xc] : v[e]) - s * __bfloat162float(*q);
              *q = __float2bfloat16_rn(val);
            }
          }
          fence_proxy_async_smem();
          asm volatile("bar.sync 1, 256;" ::: "memory");
          if (et == 0) {
            tma_store_2d(&tmO, stg, c0, x0);   // rows past N are clipped
            bulk_commit();
            bulk_wait_read0();                 // the next chunk's rows go to the same buffer
          }
          asm volatile("bar.sync 1, 256;" ::: "memory");
        }
      } else if (!DWX) {
        // partial tile of a dh pass: fp32 partial sums with plain stores (measured faster here
        // than the staged path, whose TMA traffic competes with this pass's operand stream)
        float* part = p.part + (size_t)slot * G_XT * p.C;
        for (int i = 0; i < NCH; ++i) {
          const int c = (p.ch0 + i) * 256 + (int)rank * 128 + kl;
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            float v[32];
            tmem_ld32(tmem + i * 128 + lane_off + hf * 64 + cc * 32, v);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (slot_ok) part[(size_t)(hf * 64 + cc * 32 + e) * p.C + c] = v[e];
          }
        }
      } else if (DWP) {
        // straight from TMEM: per 16-column round, for each of its 16 X rows, the warp's 32 C
        // columns as one 128-byte access (reduce-add into dW, or a store)
        float* part = p.part + (size_t)slot * G_XT * p.C;
        for (int i = 0; i < NCH; ++i) {
          const int c = (p.ch0 + i) * 256 + (int)rank * 128 + kl;
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            float v[16];
            tmem_ld16(tmem + i * 128 + lane_off + hf * 64 + cc * 16, v);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int xr = hf * 64 + cc * 16 + e;
              if (!whole) {
                if (slot_ok) part[(size_t)xr * p.C + c] = v[e];
              } else if (x0 + xr < nX) {
                float* d = p.dW + (size_t)(x0 + xr) * p.C + c;
                if (p.beta) atomicAdd(d, v[e]);
                else *d = v[e];
              }
            }
          }
        }
      } else {
        float* sf = reinterpret_cast<float*>(sDZ);
        int r = 0;
        for (int i = 0; i < NCH; ++i) {
          const int c0 = (p.ch0 + i) * 256 + (int)rank * 128;
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc, ++r) {
            float v[16];
            tmem_ld16(tmem + i * 128 + lane_off + hf * 64 + cc * 16, v);
            float* buf = sf + (r & 1) * 4096;           // rows hf*16 + e, 128 floats each
#pragma unroll
            for (int e = 0; e < 16; ++e) buf[(hf * 16 + e) * 128 + kl] = v[e];
            fence_proxy_async_smem();
            if (et == 0) bulk_wait_read0();             // last round's boxes have read the other half
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (et == 0) {
              const uint32_t src = stg + (uint32_t)(r & 1) * 16384;
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int xr0 = h * 64 + cc * 16;
                // a whole tile's box may reach past the last row (clipped), never start there
                if (!whole) tma_store_2d(&tmP, src + h * 8192, c0, slot * G_XT + xr0);
                else if (x0 + xr0 >= nX) continue;
                else if (p.beta) tma_reduce_add_2d(&tmO, src + h * 8192, c0, x0 + xr0);
                else tma_store_2d(&tmO, src + h * 8192, c0, x0 + xr0);
              }
              bulk_commit();
            }
          }
        }
      }
      if (et == 0) bulk_wait_read0();   // the buffer holds the next block's dz
      tc_fence_before();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (warp == 2 && lane == 0) {
        if (rank == 0) mbar_arrive(smem_u32(&acc_empty));
        else mbar_arrive_cluster(leader_acc_empty);
      }
      g += nb;
    }
    // every flush's and every store of p's global writes are performed before the CTA exits
    if (et == 0 || (FL && p.store_p && lane == 0)) bulk_wait0();
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
// the gradient kernel does for whole tiles.  grid: (split tiles, COMB_BLOCKS); a block covers a
// COMB_BLOCKS-th of the tile's (row, four-column group) pairs, COMB_U groups per thread at a time
// with every load of a batch issued before its stores.
constexpr int COMB_BLOCKS = 8, COMB_U = 4;
template <int MODE>
__global__ void __launch_bounds__(256) tc_split_combine_kernel(GradParams p, Sched sch, const __grid_constant__ SplitTiles sp) {
  constexpr bool DW = MODE == GM_DW || MODE == GM_DWP || MODE == GM_DWP4;
  constexpr bool FL = MODE == GM_FL;
  __shared__ int slots[16];
  __shared__ int nslots;
  __shared__ float wts[16][G_XT];   // lse+dh: 2^(m_k - M) per slot and row
  __shared__ float fac[G_XT];       // lse+dh: s / l for a valid target, else 0
  __shared__ int rowy[G_XT];        // dh passes: each row's target, or -1
  griddep_wait();
  const int t = sp.t[blockIdx.x];
  if (threadIdx.x == 0) {
    int ns = split_slots(sch, t, slots);
    for (int k = 0; k < ns; ++k)
      if (!dcheck(slots[k] < 2 * sch.P, p.err, BS_SLOT)) ns = k;
    nslots = ns;
  }
  __syncthreads();
  const int nX = DW ? p.V : p.N;
  const float s = grad_scale(p);
  if (!DW && threadIdx.x < G_XT) {
    const int xl = threadIdx.x, x = t * G_XT + xl;
    int y = -1;
    if (x < p.N) {
      const int tg = p.targets[x];
      if (tg >= 0 && tg < p.V) y = tg;
    }
    rowy[xl] = y;
    if (FL) {
      // merge the slots' (m, l) of my row: M = max m_k, l = sum l_k 2^(m_k - M)
      float M = -INFINITY;
      for (int k = 0; k < nslots; ++k) M = fmaxf(M, p.part_lm[((size_t)slots[k] * 2 + 0) * G_XT + xl]);
      float l = 0.f;
      for (int k = 0; k < nslots; ++k) {
        const float w = exp2f(p.part_lm[((size_t)slots[k] * 2 + 0) * G_XT + xl] - M);
        wts[k][xl] = w;
        l += p.part_lm[((size_t)slots[k] * 2 + 1) * G_XT + xl] * w;
      }
      fac[xl] = y >= 0 ? s / l : 0.f;
      if (blockIdx.y == 0 && x < p.N) p.lse_out[x] = (M + log2f(l)) * LN2;
      if (blockIdx.y == 0 && p.store_p && y >= 0) {
        // stored p: every segment's reference within p_range of the row's lse log2 e
        const float l2 = M + log2f(l), pr = p_range(s);
        bool far = false;
        for (int k = 0; k < nslots; ++k) far |= !(l2 - p.part_lm[((size_t)slots[k] * 2 + 0) * G_XT + xl] <= pr);
        if (far && dcheck(t < sch.U / sch.nblk, p.err, BS_TILE_FLAG)) atomicOr(p.tile_flag + t, 1u);
      }
    }
  }
  if (!DW) __syncthreads();
  const int per_row = p.nch * 64;                         // four-column groups per row (this launch's chunks)
  const int total = G_XT * per_row;
  const int ns = nslots;
  for (int base = (blockIdx.y * 256 + threadIdx.x) * COMB_U; base < total; base += COMB_BLOCKS * 256 * COMB_U) {
    int xl[COMB_U], c[COMB_U];
    bool ok[COMB_U];
    float4 v[COMB_U];
#pragma unroll
    for (int u = 0; u < COMB_U; ++u) {
      const int idx = base + u;                           // consecutive groups: one row, adjacent columns
      xl[u] = idx / per_row;
      c[u] = p.ch0 * 256 + (idx % per_row) * 4;
      ok[u] = idx < total && t * G_XT + xl[u] < nX;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int k = 0; k < ns; ++k) {
#pragma unroll
      for (int u = 0; u < COMB_U; ++u) {
        if (!ok[u]) continue;
        const float4 w = *reinterpret_cast<const float4*>(p.part + ((size_t)slots[k] * G_XT + xl[u]) * p.C + c[u]);
        const float a = FL ? wts[k][xl[u]] : 1.f;
        v[u].x += FL ? w.x * a : w.x;
        v[u].y += FL ? w.y * a : w.y;
        v[u].z += FL ? w.z * a : w.z;
        v[u].w += FL ? w.w * a : w.w;
      }
    }
    if (DW) {
      float4 d[COMB_U];
#pragma unroll
      for (int u = 0; u < COMB_U; ++u) {
        d[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (ok[u] && p.beta) d[u] = *reinterpret_cast<const float4*>(p.dW + (size_t)(t * G_XT + xl[u]) * p.C + c[u]);
      }
#pragma unroll
      for (int u = 0; u < COMB_U; ++u) {
        if (!ok[u]) continue;
        float4 r = v[u];
        if (p.beta) {
          r.x += d[u].x;
          r.y += d[u].y;
          r.z += d[u].z;
          r.w += d[u].w;
        }
        *reinterpret_cast<float4*>(p.dW + (size_t)(t * G_XT + xl[u]) * p.C + c[u]) = r;
      }
    } else {
      // dh: the row's one-hot term with one 8-byte load of W[y], one 8-byte store of dh
      uint2 wv[COMB_U];
#pragma unroll
      for (int u = 0; u < COMB_U; ++u) {
        wv[u] = make_uint2(0u, 0u);
        if (ok[u] && rowy[xl[u]] >= 0) wv[u] = *reinterpret_cast<const uint2*>(p.Wt + (size_t)rowy[xl[u]] * p.C + c[u]);
      }
#pragma unroll
      for (int u = 0; u < COMB_U; ++u) {
        if (!ok[u]) continue;
        const float f = FL ? fac[xl[u]] : 1.f;
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        if (rowy[xl[u]] >= 0) {
          const float2 w01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[u].x));
          const float2 w23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[u].y));
          r.x = (FL ? v[u].x * f : v[u].x) - s * w01.x;
          r.y = (FL ? v[u].y * f : v[u].y) - s * w01.y;
          r.z = (FL ? v[u].z * f : v[u].z) - s * w23.x;
          r.w = (FL ? v[u].w * f : v[u].w) - s * w23.y;
        }
        __nv_bfloat162 o01 = __floats2bfloat162_rn(r.x, r.y), o23 = __floats2bfloat162_rn(r.z, r.w);
        uint2 ov;
        ov.x = *reinterpret_cast<uint32_t*>(&o01);
        ov.y = *reinterpret_cast<uint32_t*>(&o23);
        *reinterpret_cast<uint2*>(p.dh + (size_t)(t * G_XT + xl[u]) * p.C + c[u]) = ov;
      }
    }
  }
}

// ---- per-row pre / post passes of the lse+dh path -----------------------------------------

// Before the lse+dh pass when the scale depends on this micro-step's valid count
// (normalisation by the micro-step mean): per-block valid counts and target errors; the block
// that finishes last reduces them (count mode), which sets the scale.
__global__ void __launch_bounds__(256) rows_pre_kernel(StepArgs a, int* __restrict__ part_cnt, unsigned* __restrict__ part_err,
                                                       const double* __restrict__ part_loss, DevAcc* acc,
                                                       unsigned* ticket) {
  griddep_wait();
  __shared__ int sc[256];
  __shared__ unsigned se[256];
  const int t = threadIdx.x;
  const int64_t n = (int64_t)blockIdx.x * 256 + t;
  int cnt = 0;
  unsigned err = 0;
  if (n < a.N) {
    const int y = a.targets[n];
    if (y >= 0 && (int64_t)y < a.V) cnt = 1;
    else if (y != a.ignore_id) err = ERR_BIT_BAD_TARGET;
  }
  sc[t] = cnt;
  se[t] = err;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (t < o) {
      sc[t] += sc[t + o];
      se[t] |= se[t + o];
    }
    __syncthreads();
  }
  if (t == 0) {
    part_cnt[blockIdx.x] = sc[0];
    part_err[blockIdx.x] = se[0];
  }
  if (last_block(ticket))
    finish_block(part_loss, part_cnt, part_err, gridDim.x, a.norm, a.G, (long long)a.global_valid, acc, FIN_COUNT);
}

// After the lse+dh pass and its repairs: row loss lse - z_t, per-block loss partials for the
// fixed-order sum, valid counts and target / non-finite errors; the repair flags of this
// block's two 128-token tiles are cleared for the next micro-step.  The block that finishes
// last reduces the partials into the step accumulators (fin_mode: FIN_ALL, or FIN_LOSS after
// the count pass).
__global__ void __launch_bounds__(256) rows_post_kernel(StepArgs a, const float* __restrict__ lse,
                                                        const float* __restrict__ zt, double* __restrict__ part_loss,
                                                        int* __restrict__ part_cnt, unsigned* __restrict__ part_err,
                                                        unsigned* __restrict__ tile_flag, int ntiles, DevAcc* acc,
                                                        unsigned* ticket, int fin_mode) {
  griddep_wait();
  __shared__ double sl[256];
  __shared__ int sc[256];
  __shared__ unsigned se[256];
  const int t = threadIdx.x;
  const int64_t n = (int64_t)blockIdx.x * 256 + t;
  if (t < 2 && (int)blockIdx.x * 2 + t < ntiles) tile_flag[blockIdx.x * 2 + t] = 0u;
  double loss = 0.0;
  int cnt = 0;
  unsigned err = 0;
  if (n < a.N) {
    const int y = a.targets[n];
    if (y >= 0 && (int64_t)y < a.V) {
      const float li = lse[n] - zt[n];
      loss = (double)li;
      cnt = 1;
      if (!isfinite(li)) err |= ERR_BIT_NONFINITE;
      if (a.row_loss) a.row_loss[n] = li;
    } else {
      if (y != a.ignore_id) err |= ERR_BIT_BAD_TARGET;
      if (a.row_loss) a.row_loss[n] = 0.f;
    }
  }
  sl[t] = loss;
  sc[t] = cnt;
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
  if (last_block(ticket))
    finish_block(part_loss, part_cnt, part_err, gridDim.x, a.norm, a.G, (long long)a.global_valid, acc, fin_mode);
}

// ---- dW from the stored exponentials: per-row pass ------------------------------------------
// s1 is the lse+dh pass's schedule (X = 128-token tiles, stream = 256-row vocabulary blocks in
// each tile's rotated order).  The segment of (tile t, block vb) is the number of pairs between
// the one that holds the tile's first unit and the one that holds that block's unit.
__device__ __forceinline__ int seg_of(const Sched& s1, int t, int vb, int rot) {
  const long long tb = (long long)t * s1.nblk;
  const int pos = ((vb - rot) % s1.nblk + s1.nblk) % s1.nblk;
  return s1.pair_of(tb + pos) - s1.pair_of(tb);
}
__device__ __forceinline__ int segs_of(const Sched& s1, int t) {
  const long long tb = (long long)t * s1.nblk;
  return s1.pair_of(tb + s1.nblk - 1) - s1.pair_of(tb) + 1;
}

constexpr int HS_ROWS = 32;     // rows per block iteration (a 128-token tile holds four)
constexpr int HS_BLOCKS = 608;  // four per SM

// After the lse+dh pass, its repairs and the final logsumexp of every row:
//   kmap[t][vb] = segment of (tile t, block vb);
//   hs[k][n] = f_k h_n in bf16, f_k = s 2^(m_k,n - lse_n log2 e) (0 for a row without a valid
//              target; zero rows from N to np), for each segment k of row n's tile;
//   p[n][y_n] = 2^(z_t log2 e - m) - 2^(lse_n log2 e - m) with m the reference of the segment
//              that covered (tile of n, block of y_n): p - onehot in that segment's scale.
__global__ void __launch_bounds__(256) tc_hs_kernel(StepArgs a, Sched s1, int ttiles, int np, int64_t vp,
                                                    const float* __restrict__ lse, const float* __restrict__ zt,
                                                    const float* __restrict__ mref, float scale_fixed,
                                                    const DevAcc* __restrict__ acc, __nv_bfloat16* __restrict__ hs,
                                                    __nv_bfloat16* __restrict__ pst, uint8_t* __restrict__ kmap) {
  griddep_wait();
  __shared__ float fs[HS_ROWS][TC_MAX_VER];
  __shared__ int nseg_sh;
  const int tid = threadIdx.x;
  const float s = scale_fixed >= 0.f ? scale_fixed : acc->scale;
  // the segment table
  const long long nk = (long long)ttiles * s1.nblk;
  for (long long i = (long long)blockIdx.x * blockDim.x + tid; i < nk; i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / s1.nblk), vb = (int)(i % s1.nblk);
    kmap[i] = (uint8_t)seg_of(s1, t, vb, s1.rot(t));
  }
  const int vecs = (int)(a.C / 8);   // 16-byte vectors per row
  const __nv_bfloat16* H = static_cast<const __nv_bfloat16*>(a.hidden);
  for (int g = blockIdx.x; g * HS_ROWS < np; g += gridDim.x) {
    const int n0 = g * HS_ROWS;
    const int t = n0 / TC_TILE_ROWS;
    if (tid < HS_ROWS) {
      const int n = n0 + tid;
      const int ns = t < ttiles ? segs_of(s1, t) : 1;
      if (tid == 0) nseg_sh = ns;
      int y = -1;
      if (n < a.N) {
        const int tg = a.targets[n];
        if (tg >= 0 && (int64_t)tg < a.V) y = tg;
      }
      const float l2 = y >= 0 ? lse[n] * LOG2E : 0.f;
      for (int k = 0; k < TC_MAX_VER; ++k)
        fs[tid][k] = (y >= 0 && k < ns) ? s * exp2f(mref[(size_t)k * np + n] - l2) : 0.f;
      if (y >= 0) {
        const int ky = seg_of(s1, t, y / G_YB, s1.rot(t));
        const float m = mref[(size_t)ky * np + n];
        pst[(size_t)n * vp + y] = __float2bfloat16_rn(exp2f(fmaf(zt[n], LOG2E, -m)) - exp2f(l2 - m));
      }
    }
    __syncthreads();
    const int ns = nseg_sh;
    for (int e = tid; e < HS_ROWS * vecs; e += blockDim.x) {
      const int r = e / vecs, cv = e % vecs;
      const int n = n0 + r;
      uint4 hv = make_uint4(0u, 0u, 0u, 0u);
      if (n < a.N) hv = __ldg(reinterpret_cast<const uint4*>(H + (size_t)n * a.C) + cv);
      for (int k = 0; k < ns; ++k) {
        const float f = fs[r][k];
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (f != 0.f) {
          const uint32_t* hi = reinterpret_cast<const uint32_t*>(&hv);
          uint32_t* oo = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi[w]));
            __nv_bfloat162 pr = __floats2bfloat162_rn(x.x * f, x.y * f);
            oo[w] = *reinterpret_cast<uint32_t*>(&pr);
          }
        }
        reinterpret_cast<uint4*>(hs + ((size_t)k * np + n) * a.C)[cv] = o;
      }
    }
    __syncthreads();
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

// Encoded tensor maps, reused across launches: a map is a function of its kind, base address,
// extents and box alone, so an entry stays right even after its buffer is freed and another is
// made at the same address.  A fixed table with round-robin replacement (no heap use).
struct MapKey {
  int kind;
  const void* ptr;
  uint64_t rows, cols;
  uint32_t a, b;
  bool operator==(const MapKey& o) const {
    return kind == o.kind && ptr == o.ptr && rows == o.rows && cols == o.cols && a == o.a && b == o.b;
  }
};
template <typename Enc>
bool cached_map(const MapKey& k, CUtensorMap* m, Enc encode) {
  constexpr int CAP = 64;
  static std::mutex mu;
  static MapKey keys[CAP];
  static CUtensorMap maps[CAP];
  static int used = 0, next = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (keys[i] == k) {
      *m = maps[i];
      return true;
    }
  if (!encode(m)) return false;
  const int slot = used < CAP ? used++ : next;
  if (used == CAP) next = (slot + 1) % CAP;
  keys[slot] = k;
  maps[slot] = *m;
  return true;
}

// The same matrix seen as [cols/64][rows][64]: box {64, box_rows, box_chunks} loads box_chunks
// consecutive 64-column swizzle atoms of box_rows rows in one instruction.
bool make_map3(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_chunks) {
  return cached_map({3, ptr, rows, cols, box_rows, box_chunks}, m, [&](CUtensorMap* out) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, rows, cols / 64};
    cuuint64_t strides[2] = {cols * 2, 128};
    cuuint32_t box[3] = {64, box_rows, box_chunks};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  });
}

// [cols/256][4][rows][64] view: box {64, box_rows, 2, box_chunks} loads, for box_chunks
// consecutive 256-column chunks, two 64-column atoms (this CTA's half of the chunk) of box_rows
// rows in one instruction.
bool make_map4(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_chunks) {
  return cached_map({4, ptr, rows, cols, box_rows, box_chunks}, m, [&](CUtensorMap* out) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {64, rows, 4, cols / 256};
    cuuint64_t strides[3] = {cols * 2, 128, 512};
    cuuint32_t box[4] = {64, box_rows, 2, box_chunks};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  });
}

// Row-major [rows][cols] fp32 or bf16 matrix, box {128 columns, box_rows rows}, no swizzle: the
// gradient kernels' flush writes its staged tiles through these (stores and reduce-adds).
bool make_map_rows(CUtensorMap* m, void* ptr, uint64_t rows, uint64_t cols, bool f32, uint32_t box_rows) {
  return cached_map({f32 ? 5 : 6, ptr, rows, cols, box_rows, 0}, m, [&](CUtensorMap* out) {
    auto fn = encode_fn();
    if (!fn) return false;
    const uint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * es};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t el[2] = {1, 1};
    return fn(out, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box,
              el, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  });
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

int64_t tc_p_cols(int64_t V) { return (V + G_YB - 1) / G_YB * G_YB; }

int64_t tc_ver_rows(int64_t N) { return (N + G_YB - 1) / G_YB * G_YB; }

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
  cudaError_t e = max_dyn_smem((const void*)tc_lse_kernel, L_SMEM);
  if (e != cudaSuccess) return e;
  L.begin(K_LSE);
  tc_lse_kernel<<<dim3(2 * nblocks, nsplit), L_THREADS, L_SMEM, L.st>>>(mh, mw, p);
  L.end();
  e = cudaGetLastError();
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

// The balanced schedule of a gradient launch over nX rows in 128-row X tiles and nY stream rows
// in 256-row blocks.
Sched grad_sched(int64_t nX, int64_t nY) {
  const int nblk = (int)((nY + G_YB - 1) / G_YB);
  const int T = (int)((nX + G_XT - 1) / G_XT);
  const long long U = (long long)T * nblk;
  // every pair covers at least a sixth of a tile, so a split tile has a handful of partials
  long long P = tc_pairs();
  if (P > U * 6 / nblk) P = U * 6 / nblk;
  if (P > U) P = U;  // every pair gets at least one unit
  if (P < 1) P = 1;
  return Sched{U, (int)P, nblk};
}

// Most segments (pairs) sharing one X tile of schedule s over T tiles.
int max_segments(const Sched& s, int T) {
  int best = 1;
  for (int t = 0; t < T; ++t) {
    const long long tb = (long long)t * s.nblk;
    const int n = s.pair_of(tb + s.nblk - 1) - s.pair_of(tb) + 1;
    if (n > best) best = n;
  }
  return best;
}

// Stored-exponential dW pass on this micro-step: buffers allocated and large enough, and every
// tile split over at most TC_MAX_VER pairs.  *nver = copies of hs the per-row pass writes.
bool use_stored_p(const StepArgs& a, const Scratch& sc, int* nver) {
  if (!sc.tc_p || a.tc_recompute || a.N <= 0 || a.N > sc.tc_p_rows) return false;
  const Sched s1 = grad_sched(a.N, a.V);
  *nver = max_segments(s1, (int)((a.N + G_XT - 1) / G_XT));
  return *nver <= TC_MAX_VER;
}

template <int MODE>
cudaError_t tc_grad_range(const StepArgs& a, const Scratch& sc, Launch& L, int ch0, int nch, int nver = 0) {
  constexpr bool DW = MODE == GM_DW;
  constexpr bool DWP = MODE == GM_DWP || MODE == GM_DWP4;
  constexpr bool DWX = DW || DWP;
  const void* X = DW ? a.W : a.hidden;
  const void* Y = DW ? a.hidden : a.W;
  const int64_t nX = DWX ? a.V : a.N, nY = DWX ? a.N : a.V;
  const int64_t vp = tc_p_cols(a.V), np = tc_ver_rows(a.N);
  CUtensorMap mx, mys, mya, mo, mp, me;
  constexpr int SK = Geo<MODE>::SK, AQ = Geo<MODE>::AQ;
  // lse+dh pass: stores p on the first range of C chunks when the dW pass reads it
  const bool store_p = MODE == GM_FL && nver > 0 && ch0 == 0;
  // flush targets: dW (fp32, 16-row boxes) or dh (bf16, whole 128-row tiles); the fp32 partial slots
  const bool mo_ok = DWX ? make_map_rows(&mo, a.dW, (uint64_t)a.V, (uint64_t)a.C, true, 16)
                         : make_map_rows(&mo, a.dh, (uint64_t)a.N, (uint64_t)a.C, false, G_XT);
  bool maps_ok;
  if (DWP) {
    // X: p [N][vp] as 64-column atoms, 64-token boxes of one atom; Y: the nver copies of hs
    maps_ok = make_map3(&mx, sc.tc_p, (uint64_t)a.N, (uint64_t)vp, 64, 1) &&
              make_map4(&mya, sc.tc_hs, (uint64_t)(nver * np), (uint64_t)a.C, 64, (uint32_t)nch);
    mys = mx;
    me = mx;
  } else {
    maps_ok = make_map3(&mx, X, (uint64_t)nX, (uint64_t)a.C, G_XT / 2, SK) &&
              make_map3(&mys, Y, (uint64_t)nY, (uint64_t)a.C, 128, SK) &&
              make_map4(&mya, Y, (uint64_t)nY, (uint64_t)a.C, 64 * AQ, (uint32_t)nch);
    // p as the epilogue warps store it: 32 tokens x one 64-column atom
    me = mx;
    if (store_p) maps_ok = maps_ok && make_map3(&me, sc.tc_p, (uint64_t)a.N, (uint64_t)vp, 32, 1);
  }
  if (!maps_ok || !mo_ok ||
      !make_map_rows(&mp, sc.tc_part, (uint64_t)(2 * tc_pairs() * G_XT), (uint64_t)a.C, true, 16))
    return cudaErrorInvalidValue;
  GradParams p;
  p.targets = a.targets;
  p.lse = sc.lse;
  p.zt_out = sc.tc_zt;
  p.acc = sc.acc;
  p.scale_fixed = a.norm == 0 ? (float)(1.0 / (double)a.global_valid) : -1.f;   // 0: global normalisation
  {
    int lg = 0;   // ceil(log2 V)
    while ((1LL << lg) < a.V) ++lg;
    p.fl_limit = (float)(115 - lg);
  }
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
  p.wait_ns = a.test_stall_ns > 0 ? (uint64_t)a.test_stall_ns : WAIT_NS;
  p.stall = a.test_stall_ns > 0 ? 1 : 0;
  p.store_p = store_p ? 1 : 0;
  p.mref = sc.tc_mref;
  p.np = (int)np;
  p.kmap = sc.tc_kmap;
  p.kmap_nblk = (int)(vp / G_YB);
  p.ttiles = (int)((a.N + G_XT - 1) / G_XT);
  const Sched sch = grad_sched(nX, nY);
  const int nblk = sch.nblk;
  const int smem = geo_smem_bytes<MODE>();
  cudaError_t e = max_dyn_smem((const void*)tc_grad_kernel<MODE>, smem);
  if (e != cudaSuccess) return e;
  L.begin(DWX ? K_DW : MODE == GM_DH ? K_DH : K_LSE_DH);
  e = launch_pdl(tc_grad_kernel<MODE>, dim3((unsigned)(2 * sch.P)), dim3(G_THREADS), (size_t)smem, L.st, mx, mys, mya,
                 mo, mp, me, p);
  L.end();
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
  e = launch_pdl(tc_split_combine_kernel<MODE>, dim3((unsigned)sp.n, (unsigned)COMB_BLOCKS), dim3(256), 0, L.st, p, sch,
                 sp);
  L.end();
  return e;
}

template <int MODE>
cudaError_t tc_grad(const StepArgs& a, const Scratch& sc, Launch& L, int nver = 0) {
  int ch0[4], nch[4];
  const int runs = chunk_ranges(a.C, ch0, nch);
  for (int r = 0; r < runs; ++r) {
    const cudaError_t e = tc_grad_range<MODE>(a, sc, L, ch0[r], nch[r], nver);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// The per-row pass between the lse+dh pass (with its repairs) and the dW pass from p.
cudaError_t tc_hs(const StepArgs& a, const Scratch& sc, Launch& L) {
  const int64_t np = tc_ver_rows(a.N);
  const Sched s1 = grad_sched(a.N, a.V);
  int blocks = (int)((np / HS_ROWS) < HS_BLOCKS ? np / HS_ROWS : HS_BLOCKS);
  if (blocks < 1) blocks = 1;
  L.begin(K_FINISH);
  const cudaError_t e = launch_pdl(tc_hs_kernel, dim3((unsigned)blocks), dim3(256), 0, L.st, a, s1,
                                   (int)((a.N + G_XT - 1) / G_XT), (int)np, tc_p_cols(a.V), (const float*)sc.lse,
                                   (const float*)sc.tc_zt, (const float*)sc.tc_mref,
                                   a.norm == 0 ? (float)(1.0 / (double)a.global_valid) : -1.f,
                                   (const DevAcc*)sc.acc, sc.tc_hs, sc.tc_p, sc.tc_kmap);
  L.end();
  return e;
}

// Default order.  With global normalisation the scale is the caller's 1 / global_valid and the
// one-pass logsumexp + dh runs first; with the micro-step mean, a count pass sets the scale
// before it (its last block to finish reduces the counts).  Then: the exact repair of flagged
// tiles (two near-empty launches when none is flagged), the row losses and counts with their
// fixed-order reduction (run by the pass's last block), then the dW pass: with the stored
// exponentials, the per-row pass (scaled copies of h, target entries of p) and the product
// dW += hs^T p; else the pass that recomputes the logits.
static cudaError_t tc_microstep_fused(const StepArgs& a, const Scratch& sc, Launch& L) {
  const int64_t nparts = tc_parts(a.N);   // 256 rows per partial
  const int ntiles = (int)((a.N + TC_TILE_ROWS - 1) / TC_TILE_ROWS);
  const bool global = a.norm == 0;
  cudaError_t e;
  if (!global) {
    L.begin(K_FINISH);
    e = launch_pdl(rows_pre_kernel, dim3((unsigned)nparts), dim3(256), 0, L.st, a, sc.part_cnt, sc.part_err, sc.part_loss,
                   sc.acc, sc.ticket);
    L.end();
    if (e != cudaSuccess) return e;
  }
  int nver = 0;
  const bool stored = use_stored_p(a, sc, &nver);
  if ((e = tc_grad<GM_FL>(a, sc, L, stored ? nver : 0)) != cudaSuccess) return e;
  if ((e = simt_repair_lse(a, sc, L)) != cudaSuccess) return e;
  if ((e = simt_repair_dh(a, sc, L, stored)) != cudaSuccess) return e;
  L.begin(K_FINISH);
  e = launch_pdl(rows_post_kernel, dim3((unsigned)nparts), dim3(256), 0, L.st, a, sc.lse, sc.tc_zt, sc.part_loss,
                 sc.part_cnt, sc.part_err, sc.tc_tile_flag, ntiles, sc.acc, sc.ticket, (int)(global ? FIN_ALL : FIN_LOSS));
  L.end();
  if (e != cudaSuccess) return e;
  if (!stored) return tc_grad<GM_DW>(a, sc, L);
  if ((e = tc_hs(a, sc, L)) != cudaSuccess) return e;
  // C = 1024: all four chunks in one run (p read once)
  if (a.C == 4 * 256) return tc_grad_range<GM_DWP4>(a, sc, L, 0, 4, nver);
  return tc_grad<GM_DWP>(a, sc, L, nver);
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
