// Tensor-core chunk attention (tcgen05 + TMEM + TMA).  Placeholder until the
// kernel lands: reports the shape as unsupported so the CUDA-core kernel runs.
#include "dev_common.cuh"

namespace la {

bool attn_tc_supported(int D, int kv_dtype) {
  (void)D;
  (void)kv_dtype;
  return false;
}

cudaError_t launch_qrot(const QrotArgs& a, cudaStream_t s) {
  (void)a;
  (void)s;
  return cudaErrorNotSupported;
}

cudaError_t launch_attn_tc(const TcAttnArgs& a, int num_sms, cudaStream_t s) {
  (void)a;
  (void)num_sms;
  (void)s;
  return cudaErrorNotSupported;
}

}  // namespace la
