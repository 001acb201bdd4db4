// tq_lm_head_static: the greedy LM head (RMSNorm + vocabulary GEMV + argmax)
// for callers that cannot allocate device memory.
//
// tq_lm_head needs 8 bytes of scratch per row for its argmax keys, which the
// caller passes in.  Some callers have no way to obtain that memory: a plugin
// running inside a host framework whose allocator owns the whole device pool,
// or a latency-critical thread that must not call cudaMalloc because it can
// synchronize the device.  This entry point takes its scratch from a
// file-scope device array instead, so it allocates nothing.
//
// Limits and sharing rules:
//  - at most TQ_LM_HEAD_STATIC_MAX_BATCH rows per call (32 KB of keys,
//    resident on every GPU that loads the library until the process exits);
//  - the array is shared by every call on a device and keeps the last call's
//    keys; each call clears the rows it uses before the GEMV runs;
//  - calls whose GPU work overlaps (two streams, or two threads) race on the
//    array and may return wrong argmax values: serialize them;
//  - the first call on a device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current) and caches it; make the
//    first call before any stream capture.
#include <mutex>

#include "kernels.cuh"

namespace {

__device__ __align__(256) unsigned long long g_lm_head_keys[TQ_LM_HEAD_STATIC_MAX_BATCH];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
unsigned long long* g_keys_addr[kMaxDevices] = {};

// Device address of g_lm_head_keys on the current device (host code may not
// use the symbol itself: on the host it is only a stand-in).
cudaError_t keys_on_current_device(unsigned long long** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_keys_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_lm_head_keys);
    if (e != cudaSuccess) return e;
    g_keys_addr[dev] = static_cast<unsigned long long*>(p);
  }
  *out = g_keys_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" tq_status tq_lm_head_static(int32_t wtype, tq_qmat w, int32_t vocab, int32_t hidden,
                                       const float* x, int32_t batch, const float* gain, float eps,
                                       float* logits, int32_t* argmax, void* stream) {
  if (wtype != TQ_Q4_0 && wtype != TQ_AFFINE4 && wtype != TQ_Q8_0) {
    tq::record_error("tq_lm_head_static: wtype must be 2, 4 or 8");
    return TQ_REFUSED;
  }
  if (batch < 1 || batch > TQ_LM_HEAD_STATIC_MAX_BATCH) {
    tq::record_error("tq_lm_head_static: batch must be in [1, TQ_LM_HEAD_STATIC_MAX_BATCH]");
    return TQ_REFUSED;
  }
  if (vocab < 1 || !tq::gemv_supported(hidden)) {
    tq::record_error("tq_lm_head_static: vocab must be >= 1 and hidden have a GEMV mapping");
    return TQ_REFUSED;
  }
  if (!w.qs_dev || !w.d_dev || !x || !gain || !argmax) {
    tq::record_error("tq_lm_head_static: pointers must not be NULL");
    return TQ_REFUSED;
  }
  if (((reinterpret_cast<uintptr_t>(w.qs_dev) | reinterpret_cast<uintptr_t>(w.d_dev) |
        reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(gain)) & 15u) != 0) {
    tq::record_error("tq_lm_head_static: qs, d, x and gain must be 16-byte aligned");
    return TQ_REFUSED;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long* keys = nullptr;
  cudaError_t e = keys_on_current_device(&keys);
  if (e == cudaSuccess) e = cudaMemsetAsync(keys, 0, (size_t)batch * sizeof(unsigned long long), s);
  if (e == cudaSuccess) {
    tq::GemvArgs h{};
    h.seg[0] = tq::GemvSeg{static_cast<const uint8_t*>(w.qs_dev), w.d_dev, vocab};
    h.nseg = 1;
    h.K = hidden;
    h.N = vocab;
    h.B = batch;
    h.x = x;
    h.gain = gain;
    h.eps = eps;
    h.y = logits;
    h.argmax_keys = keys;
    e = tq::launch_gemv(wtype, tq::GEMV_ARGMAX, h, s);
  }
  if (e == cudaSuccess) e = tq::launch_argmax_finish(keys, batch, argmax, s);
  if (e != cudaSuccess) {
    tq::record_error("tq_lm_head_static: CUDA error");
    (void)cudaGetLastError();
    return TQ_INTERNAL;
  }
  return TQ_OK;
}
