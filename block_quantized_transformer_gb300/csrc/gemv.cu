// Thread-mapping choice and dispatch of the decode GEMV (gemv_impl.cuh); the
// Q4_0 and Q8_0 instantiations live in gemv_q4.cu and gemv_q8.cu.
#include "kernels.cuh"
#include "launch.cuh"
#include "ptx.cuh"

namespace tq {

cudaError_t launch_gemv_q4(int K, int mode, const GemvArgs& a, cudaStream_t s);
cudaError_t launch_gemv_q8(int K, int mode, const GemvArgs& a, cudaStream_t s);

namespace {

__global__ void argmax_finish_kernel(const unsigned long long* keys, int n, int32_t* out) {
  grid_dep_launch();
  grid_dep_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = (int32_t)argmax_key_index(keys[i]);
}

// Any K that is a multiple of 256 (whole 16-byte rows of fp16 scales) whose
// activations and pipeline stages fit in shared memory.
bool pick_mapping(int K) { return K > 0 && K % 256 == 0 && K <= 16384; }

}  // namespace

bool gemv_supported(int K) { return pick_mapping(K); }

cudaError_t launch_gemv(int wtype, int mode, const GemvArgs& a, cudaStream_t s) {
  if (!pick_mapping(a.K)) return cudaErrorInvalidValue;
  if (a.N <= 0 || a.B <= 0) return cudaSuccess;
  return wtype == TQ_Q4_0 ? launch_gemv_q4(a.K, mode, a, s) : launch_gemv_q8(a.K, mode, a, s);
}

cudaError_t launch_argmax_finish(const unsigned long long* keys, int n, int32_t* out, cudaStream_t s) {
  return launch_k(argmax_finish_kernel, dim3((n + 127) / 128), dim3(128), 0, s, keys, n, out);
}

}  // namespace tq
