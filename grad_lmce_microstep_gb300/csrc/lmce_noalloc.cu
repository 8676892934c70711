// Allocation-free micro-step entry point.
//
// Some callers cannot call cudaMalloc: a host runtime that hands out every byte of device
// memory from its own pool or arena and does not let a library allocate behind its back,
// or a code path that must not stall -- cudaFree synchronises the whole device and
// cudaMalloc may do so too.  lmce_microstep_noalloc serves them: it runs one micro-step
// with the SIMT kernels, taking the per-row logsumexp, the per-block loss/count partials
// and the step accumulators from a fixed array compiled into this library instead of from
// lmce_create's allocations.  The caller still passes every input and output buffer.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "lmce.h"
#include "lmce_internal.cuh"

namespace lmce {
namespace {

constexpr int64_t NA_MAX_N = LMCE_NOALLOC_MAX_N;
constexpr int64_t NA_PARTS = (NA_MAX_N + 15) / 16;  // one partial per 16-row SIMT block
constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
constexpr size_t OFF_LSE = 0;
constexpr size_t OFF_PLOSS = align256(OFF_LSE + sizeof(float) * NA_MAX_N);
constexpr size_t OFF_PCNT = align256(OFF_PLOSS + sizeof(double) * NA_PARTS);
constexpr size_t OFF_PERR = align256(OFF_PCNT + sizeof(int) * NA_PARTS);
constexpr size_t OFF_ACC = align256(OFF_PERR + sizeof(unsigned) * NA_PARTS);
constexpr size_t NA_BYTES = align256(OFF_ACC + sizeof(DevAcc));

// The scratch: ~360 KB that every GPU which loads this library holds until the process
// exits.  All calls on a device share it and it keeps the last call's contents.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NA_BYTES];

constexpr int NA_MAX_DEV = 64;
std::mutex g_mu;
// Per device: the context whose modules were loaded for this entry point (see setup()).
struct DevState {
  bool arch_ok;
  bool loaded;
  CUcontext ctx;
};
DevState g_dev[NA_MAX_DEV] = {};

PFN_cuCtxGetCurrent_v4000 ctx_fn() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  });
  return fn;
}

// With the caller's device current: check its architecture once, look up the device address
// of the scratch array (its name in host code is only a stand-in) on every call, so a device
// reset that moves the array is followed, and load every module this entry point launches
// from once per context.  With lazy module loading a module is loaded, and device memory
// allocated for its code, at the first launch of one of its kernels; loading them here keeps
// every later call free of allocations, whatever dtype or size it has.
int setup(unsigned char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LMCE_ERR_CUDA;
  if (dev < 0 || dev >= NA_MAX_DEV) return LMCE_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& d = g_dev[dev];
  if (!d.arch_ok) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return LMCE_ERR_CUDA;
    if (major != 10 || minor != 3) return LMCE_ERR_ARCH;
    d.arch_ok = true;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return LMCE_ERR_CUDA;
  CUcontext ctx = nullptr;
  PFN_cuCtxGetCurrent_v4000 f = ctx_fn();
  if (!f || f(&ctx) != CUDA_SUCCESS || !ctx) return LMCE_ERR_CUDA;
  if (!d.loaded || d.ctx != ctx) {
    if (simt_load_kernels() != cudaSuccess || finish_load_kernel() != cudaSuccess) return LMCE_ERR_CUDA;
    d.loaded = true;
    d.ctx = ctx;
  }
  *out = static_cast<unsigned char*>(p);
  return LMCE_OK;
}

}  // namespace
}  // namespace lmce

using namespace lmce;

extern "C" int lmce_microstep_noalloc(const lmce_config* cfg, const void* hidden, const void* W,
                                      const int32_t* targets, int64_t N, int64_t global_valid, void* dh,
                                      float* dW, int accumulate_dW, float* row_loss, double* loss_sum_out,
                                      int64_t* valid_count_out, void* stream) {
  if (!cfg || !dW) return LMCE_ERR_ARG;
  if (cfg->C <= 0 || cfg->C > 2048 || cfg->V <= 0 || cfg->V > (1LL << 31)) return LMCE_ERR_ARG;
  if (cfg->dtype != LMCE_BF16 && cfg->dtype != LMCE_FP32) return LMCE_ERR_ARG;
  if (cfg->norm != LMCE_NORM_GLOBAL && cfg->norm != LMCE_NORM_MICRO_MEAN) return LMCE_ERR_ARG;
  if (cfg->grad_accum_steps < 1 || cfg->flags != 0) return LMCE_ERR_ARG;
  if (cfg->path != LMCE_PATH_AUTO && cfg->path != LMCE_PATH_SIMT) return LMCE_ERR_ARG;
  if (N < 0 || N > NA_MAX_N || simt_parts(N) > NA_PARTS) return LMCE_ERR_ARG;
  if (N > 0 && (!hidden || !W || !targets || !dh)) return LMCE_ERR_ARG;
  const size_t esz = cfg->dtype == LMCE_BF16 ? 2 : 4;
  if (N > 0 && (((uintptr_t)hidden | (uintptr_t)W | (uintptr_t)dh) & (esz - 1))) return LMCE_ERR_ARG;
  if (((uintptr_t)dW & 3) || ((uintptr_t)targets & 3) || ((uintptr_t)row_loss & 3)) return LMCE_ERR_ARG;
  if (((uintptr_t)loss_sum_out & 7) || ((uintptr_t)valid_count_out & 7)) return LMCE_ERR_ARG;
  unsigned char* base = nullptr;
  int st = setup(&base);
  if (st != LMCE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  Scratch sc{};
  sc.lse = reinterpret_cast<float*>(base + OFF_LSE);
  sc.part_loss = reinterpret_cast<double*>(base + OFF_PLOSS);
  sc.part_cnt = reinterpret_cast<int*>(base + OFF_PCNT);
  sc.part_err = reinterpret_cast<unsigned*>(base + OFF_PERR);
  sc.acc = reinterpret_cast<DevAcc*>(base + OFF_ACC);
  sc.max_parts = NA_PARTS;
  // the accumulators are summed into by the reduction kernel: they must start at zero
  if (cudaMemsetAsync(sc.acc, 0, sizeof(DevAcc), s) != cudaSuccess) return LMCE_ERR_CUDA;
  int ret = LMCE_OK;
  if (cfg->norm == LMCE_NORM_GLOBAL && global_valid <= 0) {
    if (N > 0 && cudaMemsetAsync(dh, 0, (size_t)N * cfg->C * esz, s) != cudaSuccess) return LMCE_ERR_CUDA;
    if (N > 0 && row_loss && cudaMemsetAsync(row_loss, 0, sizeof(float) * (size_t)N, s) != cudaSuccess)
      return LMCE_ERR_CUDA;
    ret = LMCE_ERR_NO_VALID;
  } else if (N == 0) {
    if (!accumulate_dW && cudaMemsetAsync(dW, 0, sizeof(float) * (size_t)cfg->V * cfg->C, s) != cudaSuccess)
      return LMCE_ERR_CUDA;
  } else {
    StepArgs a;
    a.hidden = hidden;
    a.W = W;
    a.targets = targets;
    a.dh = dh;
    a.dW = dW;
    a.row_loss = row_loss;
    a.N = N;
    a.C = cfg->C;
    a.V = cfg->V;
    a.ignore_id = cfg->ignore_id;
    a.norm = cfg->norm;
    a.G = cfg->grad_accum_steps;
    a.global_valid = global_valid;
    a.beta = accumulate_dW ? 1 : 0;
    a.bf16 = cfg->dtype == LMCE_BF16;
    a.tc_two_pass = 0;
    Launch L;
    L.st = s;
    L.prof = nullptr;
    if (simt_microstep(a, sc, L) != cudaSuccess) return LMCE_ERR_CUDA;
  }
  if (loss_sum_out &&
      cudaMemcpyAsync(loss_sum_out, &sc.acc->loss_sum, sizeof(double), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return LMCE_ERR_CUDA;
  if (valid_count_out &&
      cudaMemcpyAsync(valid_count_out, &sc.acc->count, sizeof(int64_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return LMCE_ERR_CUDA;
  return ret;
}
