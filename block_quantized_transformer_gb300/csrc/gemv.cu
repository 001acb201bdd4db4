// Thread-mapping choice and dispatch of the decode GEMV (gemv_impl.cuh); the
// Q4_0 and Q8_0 instantiations live in gemv_q4.cu and gemv_q8.cu.
#include "kernels.cuh"
#include "launch.cuh"
#include "ptx.cuh"

namespace tq {

cudaError_t launch_gemv_chain_q4(const GemvChain& c, cudaStream_t s);
cudaError_t launch_gemv_chain_q8(const GemvChain& c, cudaStream_t s);
cudaError_t launch_gemv_chain_a4(const GemvChain& c, cudaStream_t s);

namespace {

__global__ void argmax_finish_kernel(const unsigned long long* keys, int n, int32_t* out) {
  grid_dep_launch();
  grid_dep_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = (int32_t)argmax_key_index(keys[i]);
}

// out[b] = index of the largest of logits[b][0..V), the lowest index on ties
// (the same 64-bit keys as the GEMV's argmax epilogue).  One CTA per row.
__global__ void __launch_bounds__(256) argmax_rows_kernel(float* logits, int V, float softcap, int32_t* out) {
  grid_dep_launch();
  grid_dep_wait();
  float* row = logits + (int64_t)blockIdx.x * V;
  unsigned long long best = 0ull;
  for (int i = threadIdx.x; i < V; i += 256) {
    float v = row[i];
    if (softcap > 0.f) {
      v = softcap * tanhf(v / softcap);
      row[i] = v;
    }
    const unsigned long long k = argmax_key(v, (uint32_t)i);
    best = k > best ? k : best;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
    best = other > best ? other : best;
  }
  __shared__ unsigned long long sh[8];
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long m = sh[0];
    for (int w = 1; w < 8; ++w) m = sh[w] > m ? sh[w] : m;
    out[blockIdx.x] = (int32_t)argmax_key_index(m);
  }
}

// out[b] = x[rows[b]] for b < n, rows of H floats (H a multiple of 4); a row
// index outside [0, n_rows) sets the KV-overflow status bit and yields zeros.
__global__ void __launch_bounds__(256) gather_rows_kernel(const float* x, int H, int n_rows, const int32_t* rows,
                                                          float* out, uint32_t* status) {
  grid_dep_launch();
  grid_dep_wait();
  const int b = blockIdx.x;
  const int r = rows[b];
  const bool ok = r >= 0 && r < n_rows;
  if (!ok && threadIdx.x == 0) set_status(status, TQ_DEV_KV_OVERFLOW);
  const float4* src = reinterpret_cast<const float4*>(x + (int64_t)(ok ? r : 0) * H);
  float4* dst = reinterpret_cast<float4*>(out + (int64_t)b * H);
  for (int i = threadIdx.x; i < H / 4; i += 256) dst[i] = ok ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
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
  if (wtype == TQ_AFFINE4) return launch_gemv_chain_a4(c, s);
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

cudaError_t launch_argmax_rows(float* logits, int n, int V, float softcap, int32_t* out, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  return launch_k(argmax_rows_kernel, dim3(n), dim3(256), 0, s, logits, V, softcap, out);
}

cudaError_t launch_gather_rows(const float* x, int H, int n_rows, const int32_t* rows, int n, float* out,
                               uint32_t* status, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  return launch_k(gather_rows_kernel, dim3(n), dim3(256), 0, s, x, H, n_rows, rows, out, status);
}

cudaError_t launch_argmax_finish(const unsigned long long* keys, int n, int32_t* out, cudaStream_t s) {
  return launch_k(argmax_finish_kernel, dim3((n + 127) / 128), dim3(128), 0, s, keys, n, out);
}

}  // namespace tq
