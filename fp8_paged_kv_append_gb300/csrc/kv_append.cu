// kv_append: FP16 key store plus E4M3 value quantisation into the paged pool.
//
// "Phi-4: quality transfer and interrupted throughput studies": the intro
// fixes the format (FP16 keys, E4M3 FP8 values, model-specific scales);
// "Matched diagnostic profiles" names this step ("gathers values and writes
// the compressed cache").
//
// HBM-bound copy/convert.  One thread moves 8 elements of one (token, KV
// head) row: a 16-byte K load/store, a 16-byte (fp16) or 32-byte (fp32) V load
// and an 8-byte E4M3 store, so 16 consecutive threads cover a 128-wide row
// with fully coalesced transactions.  The grid is a grid-stride loop sized to
// a multiple of the SM count.
#include "k16v8_device.cuh"

namespace k16v8 {

// kVF32: fp32 input values.  kV16: the FP16-KV control -- values are copied
// as fp16 into a 2-byte value cache (no scale, no quantisation).
template <bool kVF32, bool kV16 = false>
__global__ void __launch_bounds__(256) kv_append_kernel(
    const __half *__restrict__ k, int64_t k_ts, const void *__restrict__ v, int64_t v_ts,
    const int64_t *__restrict__ slot_mapping, int32_t num_tokens,
    const float *__restrict__ v_scale, __half *__restrict__ k_cache,
    uint8_t *__restrict__ v_cache, int32_t num_pages, int32_t hkv, int32_t *dev_error) {
  constexpr int kVecPerRow = kHeadDim / 8;  // 16 threads per row
  pdl_wait();
  pdl_launch_dependents();
  const int64_t units = static_cast<int64_t>(num_tokens) * hkv * kVecPerRow;
  const int64_t n_slots = static_cast<int64_t>(num_pages) * kPage;
  for (int64_t u = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; u < units;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(u % kVecPerRow);
    const int64_t row = u / kVecPerRow;
    const int h = static_cast<int>(row % hkv);
    const int64_t t = row / hkv;
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;  // padding token
    if (slot >= n_slots) {
      if (c == 0 && h == 0) flag_error(dev_error, K16V8_DEVERR_SLOT);
      continue;
    }
    const int64_t page = slot / kPage;
    const int off = static_cast<int>(slot % kPage);
    const int64_t dst = ((page * hkv + h) * kPage + off) * kHeadDim + c * 8;

    // K: straight 16-byte copy.
    const uint4 kv = __ldg(reinterpret_cast<const uint4 *>(k + t * k_ts + h * kHeadDim + c * 8));
    *reinterpret_cast<uint4 *>(k_cache + dst) = kv;

    if constexpr (kV16) {
      const uint4 raw = __ldg(
          reinterpret_cast<const uint4 *>(static_cast<const __half *>(v) + t * v_ts +
                                          h * kHeadDim + c * 8));
      *reinterpret_cast<uint4 *>(reinterpret_cast<__half *>(v_cache) + dst) = raw;
      continue;
    }
    // V: widen to fp32, IEEE divide by the head's scale, round to E4M3.
    float x[8];
    const int64_t vsrc = t * v_ts + h * kHeadDim + c * 8;
    if constexpr (kVF32) {
      const float4 a = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(v) + vsrc));
      const float4 b =
          __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(v) + vsrc + 4));
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
      const uint4 raw =
          __ldg(reinterpret_cast<const uint4 *>(static_cast<const __half *>(v) + vsrc));
      const __half2 *h2 = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h2[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
      }
    }
    const float s = __ldg(v_scale + h);
    uint32_t w0 = 0, w1 = 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t lo = e4m3x2_from_f32(__fdiv_rn(x[2 * i], s), __fdiv_rn(x[2 * i + 1], s));
      const uint32_t hi =
          e4m3x2_from_f32(__fdiv_rn(x[2 * i + 4], s), __fdiv_rn(x[2 * i + 5], s));
      w0 |= lo << (16 * i);
      w1 |= hi << (16 * i);
    }
    *reinterpret_cast<uint2 *>(v_cache + dst) = make_uint2(w0, w1);
  }
}

}  // namespace k16v8

using namespace k16v8;

extern "C" int32_t k16v8_kv_append(const void *k, int64_t k_token_stride, const void *v,
                                   int32_t v_dtype, int64_t v_token_stride,
                                   const int64_t *slot_mapping, int32_t num_tokens,
                                   const float *v_scale, void *k_cache, uint8_t *v_cache,
                                   int32_t num_pages, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t *dev_error, void *stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || num_pages <= 0) return K16V8_ERR_INVALID_ARG;
  if (head_dim != kHeadDim) return K16V8_ERR_UNSUPPORTED_SHAPE;
  if (v_dtype != K16V8_F16 && v_dtype != K16V8_F32) return K16V8_ERR_INVALID_ARG;
  if (num_tokens == 0) return K16V8_OK;
  if (!k || !v || !slot_mapping || !v_scale || !k_cache || !v_cache) return K16V8_ERR_INVALID_ARG;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (k_token_stride == 0) k_token_stride = row;
  if (v_token_stride == 0) v_token_stride = row;
  if (k_token_stride < row || v_token_stride < row) return K16V8_ERR_INVALID_ARG;
  if (k_token_stride % 8 || v_token_stride % 8) return K16V8_ERR_INVALID_ARG;
  if (!k16v8_aligned(k, 16) || !k16v8_aligned(v, 16) || !k16v8_aligned(k_cache, 16) ||
      !k16v8_aligned(v_cache, 16) || !k16v8_aligned(slot_mapping, 8) ||
      !k16v8_aligned(v_scale, 4))
    return K16V8_ERR_INVALID_ARG;

  const int sms = k16v8_sm_count();
  if (sms <= 0) return K16V8_ERR_CUDA;
  const int64_t units = static_cast<int64_t>(num_tokens) * num_kv_heads * (kHeadDim / 8);
  const int threads = 256;
  int64_t blocks = (units + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sms) * 8;  // 8 resident CTAs of 256 per SM
  if (blocks > cap) blocks = cap;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dim3 grid(static_cast<unsigned>(blocks)), block(threads);
  if (v_dtype == K16V8_F32)
    return k16v8_launch_pdl(kv_append_kernel<true>, grid, block, 0, s,
                            static_cast<const __half *>(k), k_token_stride, v, v_token_stride,
                            slot_mapping, num_tokens, v_scale, static_cast<__half *>(k_cache),
                            v_cache, num_pages, num_kv_heads, dev_error);
  return k16v8_launch_pdl(kv_append_kernel<false>, grid, block, 0, s,
                          static_cast<const __half *>(k), k_token_stride, v, v_token_stride,
                          slot_mapping, num_tokens, v_scale, static_cast<__half *>(k_cache),
                          v_cache, num_pages, num_kv_heads, dev_error);
}

extern "C" int32_t k16v8_kv_append_v16(const void *k, int64_t k_token_stride, const void *v,
                                       int64_t v_token_stride, const int64_t *slot_mapping,
                                       int32_t num_tokens, void *k_cache, void *v_cache16,
                                       int32_t num_pages, int32_t num_kv_heads, int32_t head_dim,
                                       int32_t *dev_error, void *stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || num_pages <= 0) return K16V8_ERR_INVALID_ARG;
  if (head_dim != kHeadDim) return K16V8_ERR_UNSUPPORTED_SHAPE;
  if (num_tokens == 0) return K16V8_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache16) return K16V8_ERR_INVALID_ARG;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (k_token_stride == 0) k_token_stride = row;
  if (v_token_stride == 0) v_token_stride = row;
  if (k_token_stride < row || v_token_stride < row || k_token_stride % 8 || v_token_stride % 8)
    return K16V8_ERR_INVALID_ARG;
  if (!k16v8_aligned(k, 16) || !k16v8_aligned(v, 16) || !k16v8_aligned(k_cache, 16) ||
      !k16v8_aligned(v_cache16, 16) || !k16v8_aligned(slot_mapping, 8))
    return K16V8_ERR_INVALID_ARG;
  const int sms = k16v8_sm_count();
  if (sms <= 0) return K16V8_ERR_CUDA;
  const int64_t units = static_cast<int64_t>(num_tokens) * num_kv_heads * (kHeadDim / 8);
  int64_t blocks = (units + 255) / 256;
  if (blocks > static_cast<int64_t>(sms) * 8) blocks = static_cast<int64_t>(sms) * 8;
  return k16v8_launch_pdl(kv_append_kernel<false, true>, dim3(static_cast<unsigned>(blocks)),
                          dim3(256), 0, static_cast<cudaStream_t>(stream),
                          static_cast<const __half *>(k), k_token_stride, v, v_token_stride,
                          slot_mapping, num_tokens, static_cast<const float *>(nullptr),
                          static_cast<__half *>(k_cache), static_cast<uint8_t *>(v_cache16),
                          num_pages, num_kv_heads, dev_error);
}
