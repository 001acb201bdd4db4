// Thread-mapping choice and dispatch of the decode GEMV (gemv_impl.cuh); the
// Q4_0 and Q8_0 instantiations live in gemv_q4.cu and gemv_q8.cu.
#include "kernels.cuh"
#include "launch.cuh"
#include "ptx.cuh"

namespace tq {

cudaError_t launch_gemv_chain_q4(const GemvChain& c, cudaStream_t s);
cudaError_t launch_gemv_chain_q8(const GemvChain& c, cudaStream_t s);

namespace {

__global__ void argmax_finish_kernel(const unsigned long long* keys, int n, int32_t* out) {
  grid_dep_launch();
  grid_dep_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = (int32_t)argmax_key_index(keys[i]);
}

// Any K that is a multiple of 256 (whole 16-byte rows of fp16 scales) whose
// activations and pipeline stages fit in shared memory.
bool pick_mapping(int K) { return K > 0 && K % 256 == 0 && K <= 12288; }

}  // namespace

bool gemv_supported(int K) { return pick_mapping(K); }

cudaError_t launch_gemv_chain(int wtype, const GemvChain& c, cudaStream_t s) {
  if (c.n < 1 || c.n > kMaxPhases) return cudaErrorInvalidValue;
  if (c.n > 1 && c.sync == nullptr) return cudaErrorInvalidValue;
  for (int p = 0; p < c.n; ++p)
    if (!pick_mapping(c.ph[p].K) || c.ph[p].N <= 0 || c.ph[p].B <= 0) return cudaErrorInvalidValue;
  return wtype == TQ_Q4_0 ? launch_gemv_chain_q4(c, s) : launch_gemv_chain_q8(c, s);
}

cudaError_t launch_gemv(int wtype, int mode, const GemvArgs& a, cudaStream_t s) {
  if (!pick_mapping(a.K)) return cudaErrorInvalidValue;
  if (a.N <= 0 || a.B <= 0) return cudaSuccess;
  GemvChain c{};
  c.ph[0] = a;
  c.mode[0] = mode;
  c.n = 1;
  return launch_gemv_chain(wtype, c, s);
}

cudaError_t launch_argmax_finish(const unsigned long long* keys, int n, int32_t* out, cudaStream_t s) {
  return launch_k(argmax_finish_kernel, dim3((n + 127) / 128), dim3(128), 0, s, keys, n, out);
}

}  // namespace tq
