// Tensor-core path (tcgen05 + TMA) of the fused LM-head + cross-entropy micro-step.
#include "lmce_internal.cuh"

namespace lmce {

bool tc_supported(int64_t C, int64_t V, int bf16) { (void)C; (void)V; (void)bf16; return false; }
int64_t tc_parts(int64_t N) { return (N + 127) / 128; }
cudaError_t tc_microstep(const StepArgs&, const Scratch&, Launch&) {
  return cudaErrorNotSupported;
}

}  // namespace lmce
