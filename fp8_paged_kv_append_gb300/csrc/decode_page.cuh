// Per-page work shared by the decode kernels: the per-warp staging ring, the
// group query in registers, and one 16-token page of Q.K, online softmax and
// P.V for the four query heads of a GQA group.
//
// "Phi-4: quality transfer and interrupted throughput studies", intro: FP16
// keys, E4M3 values with a per-(layer, KV head) FP32 scale, 40 query heads
// over 10 KV heads, d = 128, 16-token pages.
//
//  * Q.K: eight lanes own one token (16 dims each, conflict-free 16-byte
//    shared loads), fp16-operand FMAs with fp32 accumulation against the
//    query held as packed fp16 pairs, then a 3-step reduce-scatter so each
//    lane ends with one (token, head) score: 4 shuffles per 4 tokens.
//  * Online softmax in the log2 domain per page (running max / sum).
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

// acc += a.lo * b.lo + a.hi * b.hi with fp16 operands, fp32 accumulation
// (each product is exact in fp32; one rounding per FMA).
__device__ __forceinline__ float fma_h2(uint32_t a, uint32_t b, float acc) {
  asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
      "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
      : "+f"(acc)
      : "r"(a), "r"(b));
  return acc;
}

// Sum acc[0..3] over the 8 lanes of a token group; lane j of the group ends
// with the total of head j >> 1.
__device__ __forceinline__ float reduce_scatter8(const float (&acc)[kGroup], int j) {
  const bool up4 = j & 4;
  const float s0 = up4 ? acc[0] : acc[2];
  const float s1 = up4 ? acc[1] : acc[3];
  float k0 = up4 ? acc[2] : acc[0];
  float k1 = up4 ? acc[3] : acc[1];
  k0 += __shfl_xor_sync(kFull, s0, 4);
  k1 += __shfl_xor_sync(kFull, s1, 4);
  const bool up2 = j & 2;
  const float snd = up2 ? k0 : k1;
  float kp = up2 ? k1 : k0;
  kp += __shfl_xor_sync(kFull, snd, 2);
  kp += __shfl_xor_sync(kFull, kp, 1);
  return kp;
}

// Query of the group's 4 heads as packed fp16 pairs.  Lane j (= lane & 7) of
// a token group owns dims [8j, 8j+8) and [64+8j, 64+8j+8): qh[h][0..3],
// qh[h][4..7].  `qb` points at the group's first head row.
__device__ __forceinline__ void load_group_query(const __half *qb, int j,
                                                 uint32_t (&qh)[kGroup][8]) {
#pragma unroll
  for (int h = 0; h < kGroup; ++h) {
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const uint4 raw =
          __ldg(reinterpret_cast<const uint4 *>(qb + h * kHeadDim + part * 64 + j * 8));
      qh[h][part * 4 + 0] = raw.x;
      qh[h][part * 4 + 1] = raw.y;
      qh[h][part * 4 + 2] = raw.z;
      qh[h][part * 4 + 3] = raw.w;
    }
  }
}

// Running attention state of one warp for the 4 heads of a group: m / l for
// head (lane & 7) >> 1 (every lane holding that head has the same value once
// l is summed over the lanes), o for dims [4*lane, 4*lane+4) of each head.
struct WarpState {
  float m, l;
  float2 o[kGroup][2];
  __device__ __forceinline__ void reset() {
    m = -INFINITY;
    l = 0.f;
#pragma unroll
    for (int h = 0; h < kGroup; ++h) o[h][0] = o[h][1] = make_float2(0.f, 0.f);
  }
};

// Fold one staged page (slot s of `ring`, its first `valid` tokens) into the
// warp's state.  qs = softmax scale * log2(e).
template <bool kVF16, typename Ring>
__device__ __forceinline__ void attend_page(Ring &ring, int s, int valid,
                                            const uint32_t (&qh)[kGroup][8], float qs,
                                            WarpState &st) {
  const int lane = threadIdx.x & 31;
  const int j = lane & 7;
  const int hsel = j >> 1;
  // ---- scores of 16 tokens x 4 heads ----
  const uint8_t *kp = ring.k[s];
  float sc[4];
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int t = it * 4 + (lane >> 3);
    const uint4 a = *reinterpret_cast<const uint4 *>(kp + t * 256 + j * 16);
    const uint4 bq = *reinterpret_cast<const uint4 *>(kp + t * 256 + 128 + j * 16);
    float acc[kGroup], acc2[kGroup];
#pragma unroll
    for (int h = 0; h < kGroup; ++h) {
      acc[h] = fma_h2(qh[h][0], a.x, 0.f);
      acc2[h] = fma_h2(qh[h][4], bq.x, 0.f);
      acc[h] = fma_h2(qh[h][1], a.y, acc[h]);
      acc2[h] = fma_h2(qh[h][5], bq.y, acc2[h]);
      acc[h] = fma_h2(qh[h][2], a.z, acc[h]);
      acc2[h] = fma_h2(qh[h][6], bq.z, acc2[h]);
      acc[h] = fma_h2(qh[h][3], a.w, acc[h]);
      acc2[h] = fma_h2(qh[h][7], bq.w, acc2[h]);
      acc[h] += acc2[h];
    }
    const float v = reduce_scatter8(acc, j) * qs;
    sc[it] = t < valid ? v : -INFINITY;
  }
  // ---- online softmax (log2 domain) ----
  float pm = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
  pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 8));
  pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 16));
  const float m_new = fmaxf(st.m, pm);
  const float alpha = ex2(st.m - m_new);
  float p[4];
#pragma unroll
  for (int it = 0; it < 4; ++it) p[it] = ex2(sc[it] - m_new);
  st.l = st.l * alpha + ((p[0] + p[1]) + (p[2] + p[3]));
  st.m = m_new;
  if ((lane & 1) == 0) {
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const uint32_t ph = __half_as_ushort(__float2half_rn(p[it]));
      ring.p[(it * 4 + (lane >> 3)) * kGroup + hsel] = ph | (ph << 16);
    }
    if (lane < 8) ring.alpha[hsel] = alpha;
  }
  __syncwarp();
  // ---- P.V over this page: lane owns 4 dims of every token ----
  __half2 acc[kGroup][2];
#pragma unroll
  for (int h = 0; h < kGroup; ++h) acc[h][0] = acc[h][1] = __float2half2_rn(0.f);
  const uint8_t *vp = ring.v[s] + lane * (kVF16 ? 8 : 4);
  auto pv_token = [&](int t) {
    __half2 v01, v23;
    if constexpr (kVF16) {
      const uint2 raw = *reinterpret_cast<const uint2 *>(vp + t * kHeadDim * 2);
      v01 = *reinterpret_cast<const __half2 *>(&raw.x);
      v23 = *reinterpret_cast<const __half2 *>(&raw.y);
    } else {
      const uint32_t raw = *reinterpret_cast<const uint32_t *>(vp + t * kHeadDim);
      v01 = e4m3x2_to_half2(static_cast<uint16_t>(raw & 0xffffu));
      v23 = e4m3x2_to_half2(static_cast<uint16_t>(raw >> 16));
    }
    const uint4 pp = *reinterpret_cast<const uint4 *>(ring.p + t * kGroup);
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
    for (int t = 0; t < kPage; ++t) pv_token(t);
  } else {
    for (int t = 0; t < valid; ++t) pv_token(t);
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
