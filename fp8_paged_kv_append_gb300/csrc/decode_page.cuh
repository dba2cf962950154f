// Per-page work shared by the decode kernels: the per-warp staging ring, the
// group query in registers, and one 16-token page of Q.K, online softmax and
// P.V for the four query heads of a GQA group.
//
// "Phi-4: quality transfer and interrupted throughput studies", intro: FP16
// keys, E4M3 values with a per-(layer, KV head) FP32 scale, 40 query heads
// over 10 KV heads, d = 128, 16-token pages.
//
//  * Q.K on the tensor core: one m16n8k16 MMA per 16 dims (fp16 operands,
//    fp32 accumulation) with the page's 16 tokens as M and the 4 heads
//    (padded to 8 with zero columns) as N, so the scores land one (token,
//    head) per accumulator register.  Each lane owns the same 32 dims of
//    the key rows (tokens g, g + 8) and of the query column (head g); the
//    dot product does not depend on how dims are assigned to the MMA's K
//    index, only that key and query use the same assignment.
//  * Online softmax in the log2 domain per page (running max / sum), on the
//    accumulator layout: lanes 4g + t (t < 2) hold heads 2t, 2t + 1 of
//    tokens g and g + 8.
//  * P.V: each lane owns 4 dims of every token; E4M3 -> fp16 pairs by the
//    hardware cvt, fp16x2 FMAs summed over one 16-token page (p <= 1 and
//    |v| <= 448 keep a page sum below 7168), folded into fp32 state per
//    page.  The per-head value scale is applied by the caller once, to the
//    final state (it factors out of the sum).
#pragma once

#include <math.h>

#include "k16v8_device.cuh"

namespace k16v8 {

constexpr int kWarps = 4;
constexpr int kStages = 2;
constexpr int kMinBlocks = 4;
constexpr int kKPageBytes = kPage * kHeadDim * 2;  // 4096
constexpr int kVPageBytes = kPage * kHeadDim;      // 2048
constexpr unsigned kFull = 0xffffffffu;

template <int kVBytes>
struct __align__(128) WarpRingT {
  uint8_t k[kStages][kKPageBytes];
  uint8_t v[kStages][kVBytes];
  uint32_t p[kPage * kGroup];  // p[token][head] as a duplicated fp16 pair (p, p)
  float alpha[kGroup];         // rescale factor of the running state
  uint64_t bar[kStages];
  int32_t live[kStages];       // slot holds a page (0: the page id was rejected)
};
using WarpRing = WarpRingT<kVPageBytes>;        // E4M3 values
using WarpRing16 = WarpRingT<2 * kVPageBytes>;  // FP16 values (the FP16-KV control)

// d += A (16x16, row-major fp16) * B (16x8, column-major fp16), fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The 16-byte chunks of a 128-dim fp16 row owned by lane group t (= lane & 3):
// dims [16t, 16t+16) and [64+16t, 64+16t+16).  Word w (= 2 dims) of the
// concatenated chunks feeds K index pair (w & 1 ? 2t+8 : 2t) of MMA step w / 2.
__device__ __forceinline__ int qk_chunk(int i, int t) { return (i >> 1) * 8 + 2 * t + (i & 1); }

// Query of the group's 4 heads as the MMA's B operand: lane 4g + t holds the
// 16 words of head g's dims (zero for g >= 4, the padding columns).
// `qb` points at the group's first head row.
__device__ __forceinline__ void load_group_query(const __half *qb, uint32_t (&qf)[16]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (g < kGroup)
      raw = __ldg(reinterpret_cast<const uint4 *>(qb + g * kHeadDim) + qk_chunk(i, t));
    qf[4 * i + 0] = raw.x;
    qf[4 * i + 1] = raw.y;
    qf[4 * i + 2] = raw.z;
    qf[4 * i + 3] = raw.w;
  }
}

// Running attention state of one warp for the 4 heads of a group.  During
// the page loop: mh / lh for heads 2t, 2t+1 (t = lane & 3 < 2), lh summed
// over this lane's tokens only; o for dims [4*lane, 4*lane+4) of each head.
// After finish(): m and l (summed over the page tokens) for head
// (lane & 7) >> 1 in every lane.
struct WarpState {
  float m, l;
  float mh[2], lh[2];
  float2 o[kGroup][2];
  __device__ __forceinline__ void reset() {
    mh[0] = mh[1] = -INFINITY;
    lh[0] = lh[1] = 0.f;
#pragma unroll
    for (int h = 0; h < kGroup; ++h) o[h][0] = o[h][1] = make_float2(0.f, 0.f);
  }
  __device__ __forceinline__ void finish() {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      lh[e] += __shfl_xor_sync(kFull, lh[e], 4);
      lh[e] += __shfl_xor_sync(kFull, lh[e], 8);
      lh[e] += __shfl_xor_sync(kFull, lh[e], 16);
    }
    const int hsel = (lane & 7) >> 1;  // held by lane hsel >> 1, element hsel & 1
    const float m0 = __shfl_sync(kFull, mh[0], hsel >> 1);
    const float m1 = __shfl_sync(kFull, mh[1], hsel >> 1);
    const float l0 = __shfl_sync(kFull, lh[0], hsel >> 1);
    const float l1 = __shfl_sync(kFull, lh[1], hsel >> 1);
    m = (hsel & 1) ? m1 : m0;
    l = (hsel & 1) ? l1 : l0;
  }
};

// A decode step's new token for one (sequence, KV head): lanes 0-15 each take
// 8 dims of k_src / v_src (fp16), quantise V as the cache append does (IEEE
// division by the scale, round to nearest even, saturation), put the row into
// row `row` of the staged page (slot s) -- the staged copy may predate the
// store -- and, when tile >= 0, into that cache tile (page id * hkv + head).
template <typename Ring>
__device__ __forceinline__ void append_new_row(Ring &ring, int s, int row,
                                               const __half *__restrict__ k_src,
                                               const __half *__restrict__ v_src, float scale,
                                               __half *k_cache, uint8_t *v_cache, int64_t tile) {
  const int lane = threadIdx.x & 31;
  if (lane < kHeadDim / 8) {
    const uint4 kv = __ldg(reinterpret_cast<const uint4 *>(k_src) + lane);
    const uint4 vraw = __ldg(reinterpret_cast<const uint4 *>(v_src) + lane);
    const __half2 *vh = reinterpret_cast<const __half2 *>(&vraw);
    uint32_t w[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float2 a = __half22float2(vh[2 * u]);
      const float2 c = __half22float2(vh[2 * u + 1]);
      w[u] = static_cast<uint32_t>(e4m3x2_from_f32(__fdiv_rn(a.x, scale), __fdiv_rn(a.y, scale))) |
             (static_cast<uint32_t>(e4m3x2_from_f32(__fdiv_rn(c.x, scale), __fdiv_rn(c.y, scale)))
              << 16);
    }
    *reinterpret_cast<uint4 *>(ring.k[s] + row * 256 + lane * 16) = kv;
    *reinterpret_cast<uint2 *>(ring.v[s] + row * kHeadDim + lane * 8) = make_uint2(w[0], w[1]);
    if (tile >= 0) {
      const int64_t dst = (tile * kPage + row) * kHeadDim + lane * 8;
      *reinterpret_cast<uint4 *>(k_cache + dst) = kv;
      *reinterpret_cast<uint2 *>(v_cache + dst) = make_uint2(w[0], w[1]);
    }
  }
  __syncwarp();
}

// Fold one staged page (slot s of `ring`, its first `valid` tokens) into the
// warp's state.  qs = softmax scale * log2(e).
template <bool kVF16, typename Ring>
__device__ __forceinline__ void attend_page(Ring &ring, int s, int valid,
                                            const uint32_t (&qf)[16], float qs,
                                            WarpState &st) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  // ---- scores: S[token][head] = K Q^T, tokens g / g+8 x heads 2t, 2t+1 ----
  const uint8_t *kp = ring.k[s];
  uint4 ka[4], kb[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ka[i] = *reinterpret_cast<const uint4 *>(kp + g * 256 + qk_chunk(i, t) * 16);
    kb[i] = *reinterpret_cast<const uint4 *>(kp + (g + 8) * 256 + qk_chunk(i, t) * 16);
  }
  float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint4 &x = ka[ks >> 1], &y = kb[ks >> 1];
    if (ks & 1)
      mma_16816(sacc, x.z, y.z, x.w, y.w, qf[2 * ks], qf[2 * ks + 1]);
    else
      mma_16816(sacc, x.x, y.x, x.y, y.y, qf[2 * ks], qf[2 * ks + 1]);
  }
  // ---- online softmax (log2 domain) ----
  float sc[4];
  sc[0] = g < valid ? sacc[0] * qs : -INFINITY;
  sc[1] = g < valid ? sacc[1] * qs : -INFINITY;
  sc[2] = g + 8 < valid ? sacc[2] * qs : -INFINITY;
  sc[3] = g + 8 < valid ? sacc[3] * qs : -INFINITY;
  float pm[2] = {fmaxf(sc[0], sc[2]), fmaxf(sc[1], sc[3])};
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    pm[e] = fmaxf(pm[e], __shfl_xor_sync(kFull, pm[e], 4));
    pm[e] = fmaxf(pm[e], __shfl_xor_sync(kFull, pm[e], 8));
    pm[e] = fmaxf(pm[e], __shfl_xor_sync(kFull, pm[e], 16));
  }
  float alpha[2], p[4];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const float m_new = fmaxf(st.mh[e], pm[e]);  // finite: token 0 is valid
    alpha[e] = ex2(st.mh[e] - m_new);
    p[e] = ex2(sc[e] - m_new);
    p[e + 2] = ex2(sc[e + 2] - m_new);
    st.lh[e] = st.lh[e] * alpha[e] + (p[e] + p[e + 2]);
    st.mh[e] = m_new;
  }
  if (t < 2) {
    uint32_t ph[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      ph[e] = __half_as_ushort(__float2half_rn(p[e]));
      ph[e] |= ph[e] << 16;
    }
    *reinterpret_cast<uint2 *>(ring.p + g * kGroup + 2 * t) = make_uint2(ph[0], ph[1]);
    *reinterpret_cast<uint2 *>(ring.p + (g + 8) * kGroup + 2 * t) = make_uint2(ph[2], ph[3]);
    if (g == 0) *reinterpret_cast<float2 *>(ring.alpha + 2 * t) = make_float2(alpha[0], alpha[1]);
  }
  __syncwarp();
  // ---- P.V over this page: lane owns 4 dims of every token ----
  __half2 acc[kGroup][2];
#pragma unroll
  for (int h = 0; h < kGroup; ++h) acc[h][0] = acc[h][1] = __float2half2_rn(0.f);
  const uint8_t *vp = ring.v[s] + lane * (kVF16 ? 8 : 4);
  auto pv_token = [&](int tok) {
    __half2 v01, v23;
    if constexpr (kVF16) {
      const uint2 raw = *reinterpret_cast<const uint2 *>(vp + tok * kHeadDim * 2);
      v01 = *reinterpret_cast<const __half2 *>(&raw.x);
      v23 = *reinterpret_cast<const __half2 *>(&raw.y);
    } else {
      const uint32_t raw = *reinterpret_cast<const uint32_t *>(vp + tok * kHeadDim);
      v01 = e4m3x2_to_half2(static_cast<uint16_t>(raw & 0xffffu));
      v23 = e4m3x2_to_half2(static_cast<uint16_t>(raw >> 16));
    }
    const uint4 pp = *reinterpret_cast<const uint4 *>(ring.p + tok * kGroup);
    const uint32_t pw[kGroup] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
    for (int h = 0; h < kGroup; ++h) {
      const __half2 ph = *reinterpret_cast<const __half2 *>(&pw[h]);
      acc[h][0] = __hfma2(ph, v01, acc[h][0]);
      acc[h][1] = __hfma2(ph, v23, acc[h][1]);
    }
  };
  if (valid == kPage) {
#pragma unroll
    for (int tok = 0; tok < kPage; ++tok) pv_token(tok);
  } else {
    for (int tok = 0; tok < valid; ++tok) pv_token(tok);
  }
  // fold the page into the fp32 state: o = o * alpha + page sum
  const float4 al = *reinterpret_cast<const float4 *>(ring.alpha);
  const float alv[kGroup] = {al.x, al.y, al.z, al.w};
#pragma unroll
  for (int h = 0; h < kGroup; ++h) {
    const float2 a2 = make_float2(alv[h], alv[h]);
    st.o[h][0] = __ffma2_rn(st.o[h][0], a2, __half22float2(acc[h][0]));
    st.o[h][1] = __ffma2_rn(st.o[h][1], a2, __half22float2(acc[h][1]));
  }
}

}  // namespace k16v8
