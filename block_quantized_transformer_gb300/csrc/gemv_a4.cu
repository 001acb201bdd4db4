// Affine 4-bit instantiation of the decode GEMV chain (gemv_impl.cuh).
#include "gemv_impl.cuh"

namespace tq {

cudaError_t launch_gemv_chain_a4(const GemvChain& c, cudaStream_t s) {
  return gemv::launch_chain<TQ_AFFINE4>(c, s);
}

}  // namespace tq
