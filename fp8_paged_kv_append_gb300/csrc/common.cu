// Host-side status helpers of the k16v8 C ABI.
#include "k16v8_device.cuh"

extern "C" int32_t k16v8_read_device_error(const int32_t *dev_error, void *stream,
                                           int32_t *host_value) {
  if (!dev_error || !host_value) return K16V8_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, dev_error, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return K16V8_ERR_CUDA;
  *host_value = v;
  return v == 0 ? K16V8_OK : K16V8_ERR_DEVICE_BOUNDS;
}

extern "C" const char *k16v8_status_string(int32_t status) {
  switch (status) {
    case K16V8_OK: return "ok";
    case K16V8_ERR_INVALID_ARG: return "invalid argument";
    case K16V8_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case K16V8_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case K16V8_ERR_CUDA: return "CUDA error";
    case K16V8_ERR_DEVICE_BOUNDS: return "out-of-range index met on the device";
    case K16V8_ERR_STATIC_SCRATCH_LIMIT:
      return "problem needs more than the library's built-in scratch";
    default: return "unknown status";
  }
}
