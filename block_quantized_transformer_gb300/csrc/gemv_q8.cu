// Q8_0 instantiations of the decode GEMV (gemv_impl.cuh).
#include "gemv_impl.cuh"

namespace tq {

namespace {
constexpr int kWT = TQ_Q8_0;

// Four groups of four consumer warps, two rows per warp and stage (SwiGLU: one
// gate and one up row); rows of more than 4 KB of codes take one row per warp
// and three groups, so that the activations and two stages per group fit.
template <int MODE>
cudaError_t by_k(int K, const GemvArgs& a, cudaStream_t s) {
  const int row = (K / 32) * 32;
  if (row > 4096) {
    if (MODE == GEMV_SWIGLU) return gemv::launch<gemv::Shape<kWT, MODE, 2, 3, 4>>(a, s);
    return gemv::launch<gemv::Shape<kWT, MODE, 1, 3, 4>>(a, s);
  }
  return gemv::launch<gemv::Shape<kWT, MODE, 2, 4, 4>>(a, s);
}
}  // namespace

cudaError_t launch_gemv_q8(int K, int mode, const GemvArgs& a, cudaStream_t s) {
  if (mode == GEMV_STORE) return by_k<GEMV_STORE>(K, a, s);
  if (mode == GEMV_SWIGLU) return by_k<GEMV_SWIGLU>(K, a, s);
  return by_k<GEMV_ARGMAX>(K, a, s);
}

}  // namespace tq
