// Paged causal prefill attention over the K16/V8 cache on tcgen05 tensor
// cores.
//
// "Phi-4: quality transfer and interrupted throughput studies": the fixed
// throughput metric includes prefill ("Fixed throughput studies"), and the
// 8K profile admits fresh prompts (8/7/1) before batch-16 decode ("Matched
// diagnostic profiles"); the intro gives the FP16-K / E4M3-V format and the
// 40/10/128 geometry.
//
// One CTA per (tile of 32 query tokens, KV head, sequence).  The 4 query
// heads of the GQA group are packed into the 128 rows of one MMA tile
// (row = token*4 + head), so every K/V tile loaded serves 4 heads.
//  * Q tile: one TMA box (64 dims x 4 heads x 32 tokens, 128-byte swizzle)
//    per half of the head dimension; loaded once.
//  * K tile (64 positions = 4 pages): per page and half, one TMA box of the
//    (page, head) rows straight into the K-major SW128 operand layout;
//    double-buffered.
//  * V tile: the 4 E4M3 pages by bulk copy, then dequantised by the CTA's
//    threads (hardware E4M3 -> fp16 cvt) into an MN-major SW128 operand.
//  * S = Q K^T (M 128, N 64) and O += P V (M 128, N 128) are tcgen05.mma
//    kind::f16 (K 16 per instruction) issued by one thread, accumulating in
//    tensor memory (S: 64 columns, O: 128 columns).  112 KB of shared memory
//    and 256 tensor-memory columns per CTA let two CTAs share an SM, so one
//    CTA's softmax overlaps the other's MMAs.
//  * Softmax: thread r owns row r: it loads its S row from tensor memory,
//    applies the causal mask and the log2-domain scale, keeps a running max
//    (the O row is rescaled in tensor memory only when the max grows by more
//    than 2^8, otherwise the stale max is kept -- exact, as the final
//    normalisation uses the same max), and writes P (fp16) into a K-major
//    SW128 tile for the P.V MMA.
//  * Epilogue: O / l * v_scale -> fp16, lse = ln sum exp.
#include <math.h>

#include <cudaTypedefs.h>

#include "k16v8_device.cuh"
#include "tc_sm100.cuh"

namespace k16v8 {
namespace prefill {

constexpr int kQTok = 32;                  // query tokens per tile
constexpr int kRows = kQTok * kGroup;      // 128 MMA rows
constexpr int kKv = 64;                    // KV positions per tile
constexpr int kPagesPerTile = kKv / kPage; // 4
constexpr int kThreads = 128;

// Shared memory (112 KB + barriers: two CTAs per SM).  Operand tiles start
// on 1024-byte boundaries (the dynamic shared window is 1024-aligned; the
// kernel checks).
constexpr uint32_t kKBlk = kKv * 128;              // one 64-dim half of a K tile
constexpr uint32_t kOffQ = 0;                      // 2 K-blocks x [128 rows][64] fp16
constexpr uint32_t kOffK = 32768;                  // 2 stages x 2 K-blocks x [64 pos][64]
constexpr uint32_t kOffVst = kOffK + 2 * 2 * kKBlk;    // 2 stages x [64 pos][128] E4M3
constexpr uint32_t kOffV = kOffVst + 2 * kKv * 128;    // 2 MN-blocks x [64 pos][64] fp16
constexpr uint32_t kOffP = kOffV + 2 * kKBlk;          // 1 K-block x [128 rows][64] fp16
constexpr uint32_t kOffBar = kOffP + kRows * 128;      // mbarriers, tmem slot, abort flag
constexpr uint32_t kSmemBytes = kOffBar + 128;
constexpr uint32_t kTmemCols = 256;                // S [0,64), O [128,256)

enum { kBarQ = 0, kBarKv0 = 1, kBarKv1 = 2, kBarS = 3, kBarPv = 4 };

// Bounded wait shared by the CTA's threads.  A wait that runs out sets the
// CTA-wide abort flag (and the device error word); later waits return at
// once.  Threads only act on the flag after a __syncthreads, so every thread
// leaves the main loop at the same barrier.
__device__ __forceinline__ bool cta_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         int32_t *dev_error) {
  if (*abort_flag) return false;
  if (mbar_wait_bounded(bar, parity)) return true;
  *abort_flag = 1;
  flag_error(dev_error, K16V8_DEVERR_TIMEOUT);
  return false;
}

__global__ void __launch_bounds__(kThreads, 2) prefill_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
    const uint8_t *__restrict__ v_cache, const float *__restrict__ v_scale,
    const int32_t *__restrict__ qo_indptr, const int32_t *__restrict__ block_table, int32_t maxp,
    const int32_t *__restrict__ seq_lens, int32_t total_q, int32_t hq, int32_t hkv,
    int32_t num_pages, float sm_scale, __half *__restrict__ out, float *__restrict__ lse_out,
    int32_t *dev_error) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *base = smem_raw;
  uint8_t *sQ = base + kOffQ;
  uint8_t *sK = base + kOffK;
  uint8_t *sVst = base + kOffVst;
  uint8_t *sV = base + kOffV;
  uint8_t *sP = base + kOffP;
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + kOffBar + 64);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(base + kOffBar + 68);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int g = blockIdx.y, b = blockIdx.z;
  const int tile = gridDim.x - 1 - blockIdx.x;  // longest (latest) tiles first
  pdl_wait();
  if (smem_addr(smem_raw) & 1023u) {  // operand tiles need 1024-byte alignment
    if (tid == 0) flag_error(dev_error, K16V8_DEVERR_INTERNAL);
    return;
  }

  const int q0 = __ldg(qo_indptr + b);
  const int qlen = __ldg(qo_indptr + b + 1) - q0;
  const int L = __ldg(seq_lens + b);
  if (q0 < 0 || qlen < 0 || q0 + qlen > total_q || qlen > L || L > maxp * kPage) {
    if (tid == 0 && tile == 0 && g == 0) flag_error(dev_error, K16V8_DEVERR_SEQLEN);
    return;
  }
  const int t_lo = tile * kQTok;
  if (t_lo >= qlen) return;
  const int n_tok = min(kQTok, qlen - t_lo);
  const int pos0 = L - qlen;                 // absolute position of new token 0
  const int p_lo = pos0 + t_lo;              // first / last positions of the tile
  const int p_hi = p_lo + n_tok - 1;
  const int n_kv = p_hi / kKv + 1;
  const int32_t *bt = block_table + static_cast<int64_t>(b) * maxp;

  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 5; ++i) mbar_init(&bars[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 128;

  // Issue the loads of KV tile j into stage j & 1 (thread 0 only).
  auto load_kv = [&](int j) {
    const int s = j & 1;
    uint64_t *bar = &bars[kBarKv0 + s];
    const int first_page = j * kPagesPerTile;
    const int live_pages = min(kPagesPerTile, (L - j * kKv + kPage - 1) / kPage);
    int pid0 = -1, pid1 = -1, pid2 = -1, pid3 = -1;
    uint32_t bytes = 0;
    auto get = [&](int i) {
      if (i >= live_pages) return -1;
      int p = __ldg(bt + first_page + i);
      if (p < 0 || p >= num_pages) {
        flag_error(dev_error, K16V8_DEVERR_PAGE);
        return -1;
      }
      bytes += 3 * 2048;
      return p;
    };
    pid0 = get(0);
    pid1 = get(1);
    pid2 = get(2);
    pid3 = get(3);
    mbar_arrive_expect_tx(bar, bytes);
    uint8_t *k_dst = sK + s * 2 * kKBlk;
    uint8_t *v_dst = sVst + s * kKv * 128;
    auto issue = [&](int i, int pid) {
      if (pid < 0) return;
      const int row = (pid * hkv + g) * kPage;
      tc::tma_load_2d(k_dst + i * 2048, &tmap_k, 0, row, bar);
      tc::tma_load_2d(k_dst + kKBlk + i * 2048, &tmap_k, 64, row, bar);
      bulk_g2s(v_dst + i * 2048, v_cache + static_cast<int64_t>(row) * kHeadDim, 2048, bar);
    };
    issue(0, pid0);
    issue(1, pid1);
    issue(2, pid2);
    issue(3, pid3);
  };

  if (tid == 0) {
    tc::prefetch_tensormap(&tmap_q);
    tc::prefetch_tensormap(&tmap_k);
    mbar_arrive_expect_tx(&bars[kBarQ], 2 * 16384);
    tc::tma_load_3d(sQ, &tmap_q, 0, g * kGroup, q0 + t_lo, &bars[kBarQ]);
    tc::tma_load_3d(sQ + 16384, &tmap_q, 64, g * kGroup, q0 + t_lo, &bars[kBarQ]);
    load_kv(0);
    if (n_kv > 1) load_kv(1);
  }

  // Row state: thread tid owns MMA row tid = token*4 + head.
  const int r = tid;
  const int tok = r >> 2;
  const bool row_valid = tok < n_tok;
  const int p_r = row_valid ? p_lo + tok : 0;  // last visible position
  const float qk_scale = sm_scale * kLog2e;
  float m_used = -INFINITY, l = 0.f;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  // Phases issued on each barrier (thread 0 issues every copy and MMA).
  int n_kv_loads[2] = {n_kv > 0 ? 1 : 0, n_kv > 1 ? 1 : 0};
  int n_s = 0, n_pv = 0;

  constexpr uint32_t kIdescQK = tc::idesc_f16_f32(kRows, kKv, false, false);
  constexpr uint32_t kIdescPV = tc::idesc_f16_f32(kRows, kHeadDim, false, true);

  for (int j = 0; j < n_kv; ++j) {
    const int s = j & 1;
    const uint32_t kv_par = (j >> 1) & 1;
    // ---- S = Q K^T (one thread issues) ----
    if (tid == 0) {
      const bool ok = (j > 0 || cta_wait(&bars[kBarQ], 0, abort_flag, dev_error)) &&
                      cta_wait(&bars[kBarKv0 + s], kv_par, abort_flag, dev_error);
      if (ok) {
        tc::fence_after_sync();
        const uint8_t *k_st = sK + s * 2 * kKBlk;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad =
              tc::smem_desc_sw128(smem_addr(sQ + (kk >> 2) * 16384 + (kk & 3) * 32), 16, 1024);
          const uint64_t bd =
              tc::smem_desc_sw128(smem_addr(k_st + (kk >> 2) * kKBlk + (kk & 3) * 32), 16, 1024);
          tc::mma_f16_ss(tS, ad, bd, kIdescQK, kk > 0);
        }
      }
      tc::mma_commit(&bars[kBarS]);  // completes the phase even when nothing was issued
      ++n_s;
    }
    // ---- previous P.V done: sV, sP and O are free ----
    if (j > 0) cta_wait(&bars[kBarPv], (j - 1) & 1, abort_flag, dev_error);
    // ---- dequantise V tile j into the MN-major fp16 operand ----
    cta_wait(&bars[kBarKv0 + s], kv_par, abort_flag, dev_error);
    {
      const uint8_t *vst = sVst + s * kKv * 128;
#pragma unroll
      for (int i = 0; i < kKv * 8 / kThreads; ++i) {
        const int id = tid + kThreads * i;  // chunks of 16 E4M3 values
        const int pos = id >> 3, c16 = id & 7;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
        if (j * kKv + pos < L) {
          const uint4 raw = *reinterpret_cast<const uint4 *>(vst + pos * 128 + c16 * 16);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t hv[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const __half2 a = e4m3x2_to_half2(static_cast<uint16_t>(w[q] & 0xffffu));
            const __half2 c = e4m3x2_to_half2(static_cast<uint16_t>(w[q] >> 16));
            hv[2 * q] = *reinterpret_cast<const uint32_t *>(&a);
            hv[2 * q + 1] = *reinterpret_cast<const uint32_t *>(&c);
          }
          lo = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          hi = make_uint4(hv[4], hv[5], hv[6], hv[7]);
        }
        const uint32_t off = pos * 128 + (c16 & 3) * 32;
        uint8_t *blk = sV + (c16 >> 2) * kKBlk;
        *reinterpret_cast<uint4 *>(blk + tc::sw128(off)) = lo;
        *reinterpret_cast<uint4 *>(blk + tc::sw128(off + 16)) = hi;
      }
    }
    fence_proxy_async();
    // ---- softmax of this thread's row ----
    cta_wait(&bars[kBarS], j & 1, abort_flag, dev_error);
    tc::fence_after_sync();
    // pass 1: row max of the scaled, masked scores
    const bool need_mask = j * kKv + kKv - 1 > p_lo;
    const int lim = p_r - j * kKv;  // last visible column of this tile
    float rmax = -INFINITY;
    {
      uint32_t sa[32], sb[32];
      tc::tmem_ld32(tS + lane_base, sa);
      tc::tmem_ld32(tS + lane_base + 32, sb);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        if (!need_mask || e <= lim) rmax = fmaxf(rmax, __uint_as_float(sa[e]));
        if (!need_mask || 32 + e <= lim) rmax = fmaxf(rmax, __uint_as_float(sb[e]));
      }
    }
    rmax *= qk_scale;
    float alpha = 1.f;
    if (rmax > m_used + 8.f) {
      alpha = ex2(m_used - rmax);
      m_used = rmax;
    }
    // Rescale this warp's O rows in tensor memory when any lane's max grew.
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(tO + lane_base + c * 32, o);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tc::tmem_st32(tO + lane_base + c * 32, o);
      }
      tc::tmem_wait_st();
    }
    // pass 2: p = 2^(s*scale - m), fp16 into the P operand tile
    float psum = 0.f;
    {
      uint32_t sr[2][32];
      tc::tmem_ld32(tS + lane_base, sr[0]);
      tc::tmem_ld32(tS + lane_base + 32, sr[1]);
      tc::tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // 8 values -> one 16-byte chunk of P
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c0 = c * 32 + q * 8 + 2 * e;
            float p0 = ex2(fmaf(__uint_as_float(sr[c][q * 8 + 2 * e]), qk_scale, -m_used));
            float p1 = ex2(fmaf(__uint_as_float(sr[c][q * 8 + 2 * e + 1]), qk_scale, -m_used));
            if (need_mask && c0 > lim) p0 = 0.f;
            if (need_mask && c0 + 1 > lim) p1 = 0.f;
            psum += p0 + p1;
            const __half2 h = __floats2half2_rn(p0, p1);
            pk[e] = *reinterpret_cast<const uint32_t *>(&h);
          }
          const uint32_t off = r * 128 + (c * 32 + q * 8) * 2;
          *reinterpret_cast<uint4 *>(sP + tc::sw128(off)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
    l = l * alpha + psum;
    fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    if (*abort_flag) break;  // read after the barrier: the same for every thread
    // ---- O += P V (one thread issues), then refill this stage ----
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < kKv / 16; ++kk) {
        const uint64_t ad = tc::smem_desc_sw128(smem_addr(sP + kk * 32), 16, 1024);
        const uint64_t bd = tc::smem_desc_sw128(smem_addr(sV + kk * 2048), kKBlk, 1024);
        tc::mma_f16_ss(tO, ad, bd, kIdescPV, j > 0 || kk > 0);
      }
      tc::mma_commit(&bars[kBarPv]);
      ++n_pv;
      if (j + 2 < n_kv) {
        load_kv(j + 2);
        ++n_kv_loads[s];
      }
    }
  }
  pdl_launch_dependents();

  if (cta_wait(&bars[kBarPv], (n_kv - 1) & 1, abort_flag, dev_error)) {
    tc::fence_after_sync();
    const float inv = __ldg(v_scale + g) / l;
    const int64_t orow = static_cast<int64_t>(q0 + t_lo + tok) * hq + g * kGroup + (r & 3);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      tc::tmem_ld32(tO + lane_base + c * 32, o);
      tc::tmem_wait_ld();
      if (row_valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __half2 h = __floats2half2_rn(__uint_as_float(o[q * 8 + 2 * e]) * inv,
                                                __uint_as_float(o[q * 8 + 2 * e + 1]) * inv);
            pk[e] = *reinterpret_cast<const uint32_t *>(&h);
          }
          *reinterpret_cast<uint4 *>(out + orow * kHeadDim + c * 32 + q * 8) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
    if (row_valid && lse_out) lse_out[orow] = (m_used + lg2(l)) * kLn2;
  }
  if (tid == 0) {
    // Let every copy and MMA this CTA issued land (bounded) before the
    // shared and tensor memory are given back; immediate on the normal path.
    for (int st = 0; st < 2; ++st)
      if (n_kv_loads[st] > 0) mbar_wait_bounded(&bars[kBarKv0 + st], (n_kv_loads[st] - 1) & 1);
    if (n_s > 0) mbar_wait_bounded(&bars[kBarS], (n_s - 1) & 1);
    if (n_pv > 0) mbar_wait_bounded(&bars[kBarPv], (n_pv - 1) & 1);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---- host side ------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

static int32_t set_smem_attr() {
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return K16V8_ERR_CUDA;
  if (dev < 64 && configured[dev]) return K16V8_OK;
  if (cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes)) != cudaSuccess)
    return K16V8_ERR_CUDA;
  if (dev < 64) configured[dev] = true;
  return K16V8_OK;
}

}  // namespace prefill
}  // namespace k16v8

using namespace k16v8;
using namespace k16v8::prefill;

extern "C" int32_t k16v8_paged_prefill_attention(
    const void *q, const int32_t *qo_indptr, int32_t total_q, int32_t max_qlen,
    const void *k_cache, const uint8_t *v_cache, const float *v_scale, const int32_t *block_table,
    int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t batch, int32_t num_qo_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t num_pages, float sm_scale, void *out,
    float *lse, int32_t *dev_error, void *stream) {
  if (num_qo_heads <= 0 || num_kv_heads <= 0) return K16V8_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || num_qo_heads != kGroup * num_kv_heads)
    return K16V8_ERR_UNSUPPORTED_SHAPE;
  if (batch < 0 || total_q < 0 || max_qlen < 0 || num_pages <= 0 || max_pages_per_seq < 0)
    return K16V8_ERR_INVALID_ARG;
  if (batch > 65535 || num_kv_heads > 65535) return K16V8_ERR_INVALID_ARG;
  if (batch == 0 || total_q == 0 || max_qlen == 0) return K16V8_OK;
  if (!q || !qo_indptr || !k_cache || !v_cache || !v_scale || !block_table || !seq_lens || !out)
    return K16V8_ERR_INVALID_ARG;
  if (!k16v8_aligned(q, 16) || !k16v8_aligned(k_cache, 16) || !k16v8_aligned(v_cache, 16) ||
      !k16v8_aligned(out, 16) || !k16v8_aligned(qo_indptr, 4) || !k16v8_aligned(seq_lens, 4) ||
      !k16v8_aligned(block_table, 4) || (lse && !k16v8_aligned(lse, 4)))
    return K16V8_ERR_INVALID_ARG;
  const uint64_t k_rows = static_cast<uint64_t>(num_pages) * num_kv_heads * kPage;
  if (k_rows >= (1ull << 31)) return K16V8_ERR_INVALID_ARG;

  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
  if (!encode) return K16V8_ERR_CUDA;
  CUtensorMap mq, mk;
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim),
                                static_cast<cuuint64_t>(num_qo_heads),
                                static_cast<cuuint64_t>(total_q)};
    const cuuint64_t strides[2] = {kHeadDim * 2ull,
                                   static_cast<cuuint64_t>(num_qo_heads) * kHeadDim * 2ull};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kGroup), static_cast<cuuint32_t>(kQTok)};
    const cuuint32_t es[3] = {1, 1, 1};
    if (encode(&mq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(q), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return K16V8_ERR_CUDA;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), k_rows};
    const cuuint64_t strides[1] = {kHeadDim * 2ull};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kPage)};
    const cuuint32_t es[2] = {1, 1};
    if (encode(&mk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(k_cache), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return K16V8_ERR_CUDA;
  }
  int32_t st = set_smem_attr();
  if (st != K16V8_OK) return st;
  const dim3 grid((max_qlen + kQTok - 1) / kQTok, num_kv_heads, batch);
  return k16v8_launch_pdl(prefill_kernel, grid, dim3(kThreads), kSmemBytes,
                          static_cast<cudaStream_t>(stream), mq, mk, v_cache, v_scale, qo_indptr,
                          block_table, max_pages_per_seq, seq_lens, total_q, num_qo_heads,
                          num_kv_heads, num_pages, sm_scale, static_cast<__half *>(out), lse,
                          dev_error);
}
