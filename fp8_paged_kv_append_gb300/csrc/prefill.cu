// Paged causal prefill attention over the K16/V8 cache on tcgen05 tensor
// cores.
//
// "Phi-4: quality transfer and interrupted throughput studies": the fixed
// throughput metric includes prefill ("Fixed throughput studies"), and the
// 8K profile admits fresh prompts (8/7/1) before batch-16 decode ("Matched
// diagnostic profiles"); the intro gives the FP16-K / E4M3-V format and the
// 40/10/128 geometry.
//
// One CTA per (pair of 32-token query tiles, KV head, sequence), one CTA per
// SM.  The 4 query heads of the GQA group are packed into the 128 rows of a
// tile (row = token*4 + head); both tiles (A, B) share every 128-position
// K/V tile.  Tensor memory (512 columns): S_A, S_B (128 fp32 columns each;
// P, fp16, is written over the first 64 columns of its S), O_A, O_B (128
// each).  Warp roles:
//  * warps 0-3 / 4-7: softmax of tile A / B, one thread per row: S row from
//    tensor memory, causal mask, log2-domain scale, running max (the O row in
//    tensor memory is rescaled only when the max grows by more than 2^8,
//    otherwise the stale max is kept -- exact, as the final normalisation
//    uses the same max), fp32 row sum, P (fp16) back into tensor memory;
//    finally O / l * v_scale -> fp16 and the LSE.
//  * warps 8, 10, 11: V dequantisation, E4M3 pages -> fp16 MN-major SW128
//    tile.
//  * warp 12: loads -- Q by TMA (3-D box: 64 dims x 4 heads x 32 tokens),
//    K pages by TMA straight into the K-major SW128 operand layout, E4M3 V
//    pages by bulk copy; two stages each.
//  * warp 9: one thread issues every tcgen05.mma (kind::f16, fp32
//    accumulators): S = Q K^T with both operands in shared memory, O += P V
//    with P read from tensor memory; order S_A(0) S_B(0) | PV_A(j) S_A(j+1)
//    PV_B(j) S_B(j+1) ..., so one tile's softmax overlaps the other tile's
//    MMAs.  The MMAs of one thread execute in issue order, so S_w(j+1) lands
//    after PV_w(j) has read P_w(j) from the same columns.
// Every hand-off is an mbarrier (transaction counts for copies,
// tcgen05.commit for MMAs, thread arrivals for softmax and dequant); every
// wait is bounded.
//
// KV-split form (prefill_kernel<true>): for calls whose pairs would not fill
// the SMs in whole waves, each pair's KV tiles are cut into up to 4 parts run
// by separate CTAs; every part writes its rows normalised by its own softmax
// sum (fp16) and their LSE to a workspace and counts itself on a per-pair
// atomic counter, and the part that completes the count combines the parts
// (weights e^(lse_p - lse)) and writes the output -- no CTA waits on
// another.  The plain form is a separate instantiation without that code:
// compiled into one kernel it cost the plain form 10% through its
// instruction footprint.
#include <math.h>

#include <algorithm>
#include <cmath>

#include <cudaTypedefs.h>

#include "k16v8_device.cuh"
#include "tc_sm100.cuh"

namespace k16v8 {
namespace prefill {

constexpr int kQTok = 32;                   // query tokens per tile
constexpr int kRows = kQTok * kGroup;       // 128 MMA rows per tile
constexpr int kKv = 128;                    // KV positions per tile
constexpr int kPagesPerTile = kKv / kPage;  // 8
// Warp roles: 0-7 softmax (warp w reads tensor-memory lanes 32(w%4)..+31,
// so each group of 4 spans the 4 schedulers, warp w on scheduler w%4); 8, 10
// and 11 dequantise V; 9 issues the MMAs; 12 loads.  The MMA warp is the
// only non-softmax warp on its scheduler: every tcgen05.mma it issues needs
// an issue slot there, and a dequant warp beside it (the first layout) cost
// 2-5% (measured).
constexpr int kDequantWarps = 3;
constexpr int kMmaWarp = 9;
constexpr int kLoadWarp = 12;
constexpr int kThreads = 13 * 32;
// Rank of a dequant warp among the dequant warps, or -1.
__device__ __forceinline__ int dequant_rank(int warp) {
  return warp == 8 ? 0 : (warp == 10 ? 1 : (warp == 11 ? 2 : -1));
}

constexpr uint32_t kQBytes = kRows * 256;          // one Q tile: 2 K-blocks [128][64] fp16
constexpr uint32_t kKBlk = kKv * 128;              // [128 pos][64 dims] fp16
constexpr uint32_t kKStage = 2 * kKBlk;
constexpr uint32_t kVstStage = kKv * 128;          // [128 pos][128] E4M3
constexpr uint32_t kVStage = 2 * kKBlk;            // 2 MN-blocks [128 pos][64] fp16
constexpr uint32_t kOffQ = 0;                      // Q_A, Q_B
constexpr uint32_t kOffK = 2 * kQBytes;            // 2 stages
constexpr uint32_t kOffVst = kOffK + 2 * kKStage;  // 2 stages
constexpr uint32_t kOffV = kOffVst + 2 * kVstStage;  // 2 stages
constexpr int kMaxIdPages = 512;                   // page ids staged in shared memory
constexpr uint32_t kOffIds = kOffV + 2 * kVStage;
constexpr uint32_t kOffBar = kOffIds + kMaxIdPages * 4;
constexpr uint32_t kSmemBytes = kOffBar + 256;
constexpr uint32_t kTmemCols = 512;  // S_A [0,128) S_B [128,256) O_A [256,384) O_B [384,512)
constexpr int kMaxKvParts = 4;       // KV split of one work item, at most
constexpr int kMinPartTiles = 8;     // KV tiles per part, at least

enum {
  kBarQ = 0,
  kBarKFull = 1,    // +stage
  kBarKEmpty = 3,   // +stage
  kBarVstFull = 5,  // +stage
  kBarVstEmpty = 7, // +stage, kDequantWarps*32 arrivals
  kBarVFull = 9,    // +stage, kDequantWarps*32 arrivals
  kBarVEmpty = 11,  // +stage
  kBarSFull = 13,   // +tile
  kBarPFull = 15,   // +tile, 128 arrivals
  kBarODone = 17,   // +tile
  kBarDrain = 19,   // every MMA of the CTA complete (one commit at the end)
  kNumBars = 20
};

// Bounded wait shared by every role.  A wait that runs out sets the
// CTA-wide abort flag (and the device error word); every role leaves its
// loop when a wait fails, and a wait that starts after the flag is up
// returns at once.  The suspending waits (softmax, dequant and load warps)
// also give up as soon as they see the flag (checked every 1024 polls), so
// once one role has given up the others follow within a few polls.  The
// MMA thread's spinning waits do not check it: a check in those loops cost
// the kernel 5% (they share a scheduler with softmax warps), and that
// thread waits only on the loads and the softmax warps, whose own waits
// end.  `limit` (0: the default bound) is shortened only by the
// bounded-wait test hook.
__device__ __forceinline__ bool cta_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         int32_t *dev_error, bool spin = false,
                                         uint32_t limit = 0) {
  if (*abort_flag) return false;
  if (spin) {
    // the MMA thread spins (no suspension, so a hand-off is seen at once)
    if (mbar_spin_bounded(bar, parity, limit ? limit : kMaxSpins)) return true;
  } else {
    const uint32_t n = limit ? limit : kMaxPolls;
    for (uint32_t i = 0; i < n; ++i) {
      if (mbar_try_wait(bar, parity)) return true;
      if ((i & 1023u) == 1023u && *abort_flag) return false;
    }
  }
  *abort_flag = 1;
  flag_error(dev_error, K16V8_DEVERR_TIMEOUT);
  return false;
}

// Bounded poll until three barrier phases have all completed (c may be
// null); each is tested until seen once.  Used by the MMA thread.
__device__ __forceinline__ bool wait_all3(uint64_t *a, uint32_t pa, uint64_t *b, uint32_t pb,
                                          uint64_t *c, uint32_t pc, volatile int *abort_flag,
                                          int32_t *dev_error) {
  if (*abort_flag) return false;
  bool da = false, db = false, dc = c == nullptr;
  for (uint32_t i = 0; i < kMaxSpins; ++i) {
    if (!db) db = mbar_test_wait(b, pb);
    if (!dc) dc = mbar_test_wait(c, pc);
    if (!da) da = mbar_test_wait(a, pa);
    if (da && db && dc) return true;
  }
  *abort_flag = 1;
  flag_error(dev_error, K16V8_DEVERR_TIMEOUT);
  return false;
}

// kSplit: the KV-split form (parts of a pair's KV range, merged by the last
// part); the plain form is compiled without any of that code, which keeps
// its instruction footprint as small as it was.
template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
    const __grid_constant__ CUtensorMap tmap_o,
    const uint8_t *__restrict__ v_cache, const float *__restrict__ v_scale,
    const int32_t *__restrict__ qo_indptr, const int32_t *__restrict__ block_table, int32_t maxp,
    const int32_t *__restrict__ seq_lens, int32_t total_q, int32_t hq, int32_t hkv,
    int32_t num_pages, float sm_scale, __half *__restrict__ out, float *__restrict__ lse_out,
    int32_t *dev_error, int32_t kv_parts, uint4 *__restrict__ part_o,
    float *__restrict__ part_lse, int32_t *__restrict__ counters, int32_t test_withhold) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *base = smem_raw;
  uint8_t *sQ = base + kOffQ;
  uint8_t *sK = base + kOffK;
  uint8_t *sVst = base + kOffVst;
  uint8_t *sV = base + kOffV;
  int *page_ids = reinterpret_cast<int *>(base + kOffIds);
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + kOffBar + kNumBars * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(base + kOffBar + kNumBars * 8 + 4);
  volatile int *last_flag = reinterpret_cast<volatile int *>(base + kOffBar + kNumBars * 8 + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, b = blockIdx.z;
  const int parts = kSplit ? kv_parts : 1;
  const int max_pairs = gridDim.x / parts;
  const int slot = blockIdx.x / parts, part = blockIdx.x - slot * parts;
  const int pair = max_pairs - 1 - slot;  // longest (latest) tiles first
  pdl_wait();
  if (smem_addr(smem_raw) & 1023u) {  // operand tiles need 1024-byte alignment
    if (tid == 0) flag_error(dev_error, K16V8_DEVERR_INTERNAL);
    return;
  }

  const int q0 = __ldg(qo_indptr + b);
  const int qlen = __ldg(qo_indptr + b + 1) - q0;
  const int L = __ldg(seq_lens + b);
  if (q0 < 0 || qlen < 0 || q0 + qlen > total_q || qlen > L || L > maxp * kPage) {
    if (tid == 0 && pair == 0 && g == 0) flag_error(dev_error, K16V8_DEVERR_SEQLEN);
    return;
  }
  const int t_lo = pair * 2 * kQTok;  // first query token of tile A
  if (t_lo >= qlen) return;
  const int pos0 = L - qlen;          // absolute position of new token 0
  const int p_hi = pos0 + min(t_lo + 2 * kQTok, qlen) - 1;  // last position of the pair
  const int n_all = p_hi / kKv + 1;  // KV tiles of the pair
  // KV split: part `part` of `live_parts` takes tiles [kv0, kv0 + n_kv); the
  // last part to finish merges the parts' rows (see the epilogue)
  const int live_parts = kSplit ? max(1, min(parts, n_all / kMinPartTiles)) : 1;
  if (part >= live_parts) return;
  const bool split = kSplit && live_parts > 1;
  const int kv0 = part * n_all / live_parts;
  const int n_kv = (part + 1) * n_all / live_parts - kv0;
  const int32_t *bt = block_table + static_cast<int64_t>(b) * maxp + kv0 * kPagesPerTile;
  // Bounded-wait test hook (test_withhold != 0, never in production calls):
  // the first CTA withholds the copies of its first KV tile -- no arrival,
  // nothing in flight -- so the MMA thread's wait for that tile expires
  // after kTestSpins polls and every role takes the abort path.
  const bool withheld = test_withhold != 0 && (blockIdx.x | blockIdx.y | blockIdx.z) == 0;

  if (warp == kLoadWarp && lane == 0) {
    // The query load depends on nothing else: start it before the rest of
    // the set-up (its barrier is this thread's to initialise).
    mbar_init(&bars[kBarQ], 1);
    fence_barrier_init();
    tc::prefetch_tensormap(&tmap_q);
    tc::prefetch_tensormap(&tmap_k);
    mbar_arrive_expect_tx(&bars[kBarQ], 2 * kQBytes);
    for (int w = 0; w < 2; ++w) {
      tc::tma_load_3d(sQ + w * kQBytes, &tmap_q, 0, g * kGroup, q0 + t_lo + w * kQTok,
                      &bars[kBarQ]);
      tc::tma_load_3d(sQ + w * kQBytes + kQBytes / 2, &tmap_q, 64, g * kGroup,
                      q0 + t_lo + w * kQTok, &bars[kBarQ]);
    }
  }
  if (warp == kLoadWarp) {
    // this pair's page ids into shared memory (lane-parallel), overlapping
    // the tensor-memory and barrier set-up of the other warps
    const int n_ids = min(n_kv * kPagesPerTile, (L + kPage - 1) / kPage - kv0 * kPagesPerTile);
    for (int i = lane; i < min(n_ids, kMaxIdPages); i += 32) {
      const int p = __ldg(bt + i);
      page_ids[i] = (p >= 0 && p < num_pages) ? p : -1;
      if (p < 0 || p >= num_pages) flag_error(dev_error, K16V8_DEVERR_PAGE);
    }
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      if (i == kBarQ) continue;  // initialised by the load warp
      uint32_t count = 1;
      if (i == kBarVstEmpty || i == kBarVstEmpty + 1 || i == kBarVFull || i == kBarVFull + 1)
        count = kDequantWarps * 32;
      if (i == kBarPFull || i == kBarPFull + 1) count = kRows;
      mbar_init(&bars[i], count);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    // ================= softmax: tile w (0 = A, 1 = B) =================
    const int w = warp >> 2;
    const int r = tid & 127;  // row = token*4 + head
    const int tok = r >> 2;
    const int t_abs = t_lo + w * kQTok + tok;  // token index within the sequence
    const bool row_valid = t_abs < qlen;
    const int p_lo = pos0 + t_lo + w * kQTok;   // first position of this tile
    const int p_r = row_valid ? pos0 + t_abs : 0;
    const float qk_scale = sm_scale * kLog2e;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + w * 128;   // S_w; P_w in its first 64 columns
    const uint32_t tO = tmem + 256 + w * 128;
    float m_used = -INFINITY, l = 0.f;
    for (int j = 0; j < n_kv; ++j) {
      if (!__all_sync(0xffffffffu, cta_wait(&bars[kBarSFull + w], j & 1, abort_flag, dev_error)))
        break;
      tc::fence_after_sync();
      const bool need_mask = (kv0 + j) * kKv + kKv - 1 > p_lo;  // diagonal tile
      const int lim = p_r - (kv0 + j) * kKv;  // last visible column of this tile
      // pass 1: row max (64 columns per load round)
      float rmax = -INFINITY;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t sr[2][32];
        tc::tmem_ld32(tS + lane_base + h * 64, sr[0]);
        tc::tmem_ld32(tS + lane_base + h * 64 + 32, sr[1]);
        tc::tmem_wait_ld();
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (h * 64 + c * 32 + e <= lim) rmax = fmaxf(rmax, __uint_as_float(sr[c][e]));
        } else {
          float m4[4] = {rmax, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) m4[e & 3] = fmaxf(m4[e & 3], __uint_as_float(sr[c][e]));
          rmax = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
      }
      rmax *= qk_scale;
      float alpha = 1.f;
      if (rmax > m_used + 8.f) {
        alpha = ex2(m_used - rmax);
        m_used = rmax;
      }
      // O_w is stable once PV_w(j-1) has completed.  S_w(j) was issued after
      // PV_w(j-1) and MMAs complete in order, so that is already so; the
      // wait (free by now) only orders the O accesses of a rescale.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        if (!__all_sync(0xffffffffu,
                        cta_wait(&bars[kBarODone + w], (j - 1) & 1, abort_flag, dev_error)))
          break;
        tc::fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tc::tmem_ld32(tO + lane_base + c * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tc::tmem_st32(tO + lane_base + c * 32, o);
        }
      }
      // pass 2: p = 2^(s*scale - m) in pairs; fp32 row sum; P (fp16) over the
      // already-read S columns: positions 32c.. land in P columns 16c..
      const float2 sc2 = make_float2(qk_scale, qk_scale);
      const float2 nm2 = make_float2(-m_used, -m_used);
      float2 ps2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t sr[32];
        tc::tmem_ld32(tS + lane_base + c * 32, sr);
        tc::tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c0 = c * 32 + 2 * e;
          const float2 x = __ffma2_rn(
              make_float2(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), sc2, nm2);
          // every exponential on MUFU: an FMA-pipe polynomial for part of them
          // lengthened this latency-bound pass
          float2 pp = make_float2(ex2(x.x), ex2(x.y));
          if (need_mask) {
            if (c0 > lim) pp.x = 0.f;
            if (c0 + 1 > lim) pp.y = 0.f;
          }
          ps2 = __fadd2_rn(ps2, pp);
          const __half2 hh = __floats2half2_rn(pp.x, pp.y);
          pk[e] = *reinterpret_cast<const uint32_t *>(&hh);
        }
        tc::tmem_st16(tS + lane_base + c * 16, pk);
      }
      tc::tmem_wait_st();
      l = l * alpha + (ps2.x + ps2.y);
      tc::fence_before_sync();
      mbar_arrive(&bars[kBarPFull + w]);
    }
    pdl_launch_dependents();
    // ---- epilogue ----
    // A tile whose 32 tokens all belong to this sequence leaves through a
    // TMA store from its own Q buffer (free: its last S has completed before
    // its last P.V); a partial tile at the end of a sequence is written row
    // by row so the next sequence's rows stay untouched.
    const bool full_tile = t_lo + (w + 1) * kQTok <= qlen;  // uniform over the group
    uint8_t *stage = sQ + w * kQBytes;
    const bool o_ready = __all_sync(
        0xffffffffu, cta_wait(&bars[kBarODone + w], (n_kv - 1) & 1, abort_flag, dev_error));
    bool write_out = true;
    if constexpr (!kSplit) {
      if (o_ready) {
        tc::fence_after_sync();
        const float inv = __ldg(v_scale + g) / l;
        const int64_t orow = static_cast<int64_t>(q0 + t_abs) * hq + g * kGroup + (r & 3);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tc::tmem_ld32(tO + lane_base + c * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __half2 hh = __floats2half2_rn(__uint_as_float(o[q * 8 + 2 * e]) * inv,
                                                   __uint_as_float(o[q * 8 + 2 * e + 1]) * inv);
              pk[e] = *reinterpret_cast<const uint32_t *>(&hh);
            }
            if (full_tile) {
              // dims 32c + 8q .. +7: box half c >> 1, 16-byte chunk (c & 1) * 4 + q of row r
              const uint32_t off = static_cast<uint32_t>(r) * 128 + ((c & 1) * 4 + q) * 16;
              *reinterpret_cast<uint4 *>(stage + (c >> 1) * (kQBytes / 2) + tc::sw128(off)) =
                  make_uint4(pk[0], pk[1], pk[2], pk[3]);
            } else if (row_valid) {
              *reinterpret_cast<uint4 *>(out + orow * kHeadDim + c * 32 + q * 8) =
                  make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          }
        }
        if (row_valid && lse_out) lse_out[orow] = (m_used + lg2(l)) * kLn2;
      }
    } else {
      const int64_t orow = static_cast<int64_t>(q0 + t_abs) * hq + g * kGroup + (r & 3);
      auto put = [&](int c16, const uint32_t (&pk)[4]) {  // 8 output dims [8*c16, 8*c16+8)
        if (full_tile) {
          // box half c16 >> 3, 16-byte chunk c16 & 7 of row r
          const uint32_t off = static_cast<uint32_t>(r) * 128 + (c16 & 7) * 16;
          *reinterpret_cast<uint4 *>(stage + (c16 >> 3) * (kQBytes / 2) + tc::sw128(off)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        } else if (row_valid) {
          *reinterpret_cast<uint4 *>(out + orow * kHeadDim + c16 * 8) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      };
      // KV split: every part writes its rows normalised by its own sum (fp16)
      // and its LSE; the part that finishes last (per-item counter) combines
      // them -- o = sum_p e^(lse_p - lse) o_p, lse = log sum_p e^lse_p -- and
      // writes the output.  No part waits for another.
      const int64_t item = (static_cast<int64_t>(b) * hkv + g) * max_pairs + pair;
      auto part_base = [&](int q) { return ((item * kv_parts + q) * 2 + w) * kRows; };
      if (o_ready) {
        tc::fence_after_sync();
        const float vs = __ldg(v_scale + g);
        const float inv = split ? (l > 0.f ? vs / l : 0.f) : vs / l;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tc::tmem_ld32(tO + lane_base + c * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __half2 hh = __floats2half2_rn(__uint_as_float(o[q * 8 + 2 * e]) * inv,
                                                   __uint_as_float(o[q * 8 + 2 * e + 1]) * inv);
              pk[e] = *reinterpret_cast<const uint32_t *>(&hh);
            }
            if (split)  // [chunk][row] so a warp's 32 rows are one 512-byte run
              part_o[(part_base(part) / kRows * 16 + c * 4 + q) * kRows + r] =
                  make_uint4(pk[0], pk[1], pk[2], pk[3]);
            else
              put(c * 4 + q, pk);
          }
        }
        const float lse_row = l > 0.f ? (m_used + lg2(l)) * kLn2 : -INFINITY;
        if (split)
          part_lse[part_base(part) + r] = lse_row;
        else if (row_valid && lse_out)
          lse_out[orow] = lse_row;
      }
      if (split) {
        __threadfence();  // this part's rows are visible before it is counted
        asm volatile("bar.sync 3, %0;" ::"r"(2 * kRows) : "memory");
        if (tid == 0) *last_flag = atomicAdd(counters + item, 1) == live_parts - 1;
        asm volatile("bar.sync 3, %0;" ::"r"(2 * kRows) : "memory");
        write_out = *last_flag;
        if (write_out && o_ready) {
          __threadfence();  // the other parts' rows, counted before this one
          float lq[kMaxKvParts], wq[kMaxKvParts];
          float M = -INFINITY;
#pragma unroll
          for (int q = 0; q < kMaxKvParts; ++q) {
            lq[q] = q < live_parts ? __ldcg(part_lse + part_base(q) + r) : -INFINITY;
            M = fmaxf(M, lq[q]);
          }
          float S = 0.f;
#pragma unroll
          for (int q = 0; q < kMaxKvParts; ++q) {
            wq[q] = q < live_parts && lq[q] != -INFINITY ? ex2((lq[q] - M) * kLog2e) : 0.f;
            S += wq[q];
          }
          const float invS = S > 0.f ? 1.f / S : 0.f;
#pragma unroll
          for (int q = 0; q < kMaxKvParts; ++q) wq[q] *= invS;
#pragma unroll 1
          for (int c16 = 0; c16 < 16; ++c16) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int q = 0; q < kMaxKvParts; ++q) {
              if (q < live_parts) {
                const uint4 v = __ldcg(part_o + (part_base(q) / kRows * 16 + c16) * kRows + r);
                const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&vw[e]));
                  acc[2 * e] = fmaf(wq[q], f.x, acc[2 * e]);
                  acc[2 * e + 1] = fmaf(wq[q], f.y, acc[2 * e + 1]);
                }
              }
            }
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __half2 hh = __floats2half2_rn(acc[2 * e], acc[2 * e + 1]);
              pk[e] = *reinterpret_cast<const uint32_t *>(&hh);
            }
            put(c16, pk);
          }
          if (row_valid && lse_out) lse_out[orow] = S > 0.f ? M + lg2(S) * kLn2 : -INFINITY;
          if (tid == 0) counters[item] = 0;  // ready for the next call
        }
      }
    }
    if (full_tile) {  // every thread of the group reaches this barrier
      fence_proxy_async();
      asm volatile("bar.sync %0, %1;" ::"r"(1 + w), "r"(kRows) : "memory");
      if (r == 0 && write_out && !*abort_flag) {
        const int z = q0 + t_lo + w * kQTok;
        tc::tma_store_3d(&tmap_o, stage, 0, g * kGroup, z);
        tc::tma_store_3d(&tmap_o, stage + kQBytes / 2, 64, g * kGroup, z);
        tc::bulk_commit();
        tc::bulk_wait_read();  // the buffer must outlive the copy's reads
      }
    }
  } else if (dequant_rank(warp) >= 0) {
    // ================= V dequantisation =================
    const int dt = dequant_rank(warp) * 32 + lane;  // 0 .. 32 * kDequantWarps - 1
    for (int j = 0; j < n_kv; ++j) {
      const int s = j & 1;
      if (!cta_wait(&bars[kBarVstFull + s], (j >> 1) & 1, abort_flag, dev_error)) break;
      if (j >= 2 && !cta_wait(&bars[kBarVEmpty + s], ((j >> 1) - 1) & 1, abort_flag, dev_error))
        break;
      const uint8_t *vst = sVst + s * kVstStage;
      uint8_t *vdst = sV + s * kVStage;
#pragma unroll 2
      for (int id = dt; id < kKv * 8; id += kDequantWarps * 32) {  // chunks of 16 E4M3 values
        const int pos = id >> 3, c16 = id & 7;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
        if ((kv0 + j) * kKv + pos < L) {
          const uint4 raw = *reinterpret_cast<const uint4 *>(vst + pos * 128 + c16 * 16);
          const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t hv[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const __half2 a = e4m3x2_to_half2(static_cast<uint16_t>(wv[q] & 0xffffu));
            const __half2 c = e4m3x2_to_half2(static_cast<uint16_t>(wv[q] >> 16));
            hv[2 * q] = *reinterpret_cast<const uint32_t *>(&a);
            hv[2 * q + 1] = *reinterpret_cast<const uint32_t *>(&c);
          }
          lo = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          hi = make_uint4(hv[4], hv[5], hv[6], hv[7]);
        }
        const uint32_t off = pos * 128 + (c16 & 3) * 32;
        uint8_t *blk = vdst + (c16 >> 2) * kKBlk;
        *reinterpret_cast<uint4 *>(blk + tc::sw128(off)) = lo;
        *reinterpret_cast<uint4 *>(blk + tc::sw128(off + 16)) = hi;
      }
      fence_proxy_async();
      mbar_arrive(&bars[kBarVFull + s]);
      mbar_arrive(&bars[kBarVstEmpty + s]);
    }
  } else if (warp == kLoadWarp) {
    // ================= loads =================
    // (page ids were staged before the set-up barrier)
    // Per tile, lane i < 8 issues the three copies of page i; lane 0 first
    // posts the tile's byte count on both barriers.
    // last tile issued on each stage: a stage is refilled only after its
    // previous tile was consumed, so at most that one copy is outstanding
    int last0 = -1, last1 = -1;
    for (int j = 0; j < n_kv; ++j) {
      const int s = j & 1;
      if (j >= 2) {
        // suspending waits: the warp runs a tile ahead, and a spinning one
        // would take issue slots from the softmax warps of its scheduler
        const bool ok =
            cta_wait(&bars[kBarKEmpty + s], ((j >> 1) - 1) & 1, abort_flag, dev_error) &&
            cta_wait(&bars[kBarVstEmpty + s], ((j >> 1) - 1) & 1, abort_flag, dev_error);
        if (!__all_sync(0xffffffffu, ok)) break;  // stop issuing; drain below
      }
      if (withheld && j == 0) continue;
      if (s) last1 = j; else last0 = j;
      const int live = min(kPagesPerTile, (L - (kv0 + j) * kKv + kPage - 1) / kPage);
      int pid = -1;
      if (lane < live) {
        const int pi = j * kPagesPerTile + lane;
        if (pi < kMaxIdPages) {
          pid = page_ids[pi];
        } else {
          pid = __ldg(bt + pi);
          if (pid < 0 || pid >= num_pages) {
            flag_error(dev_error, K16V8_DEVERR_PAGE);
            pid = -1;
          }
        }
      }
      const uint32_t kbytes = __reduce_add_sync(0xffffffffu, pid >= 0 ? 2u * 2048u : 0u);
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[kBarKFull + s], kbytes);
        mbar_arrive_expect_tx(&bars[kBarVstFull + s], kbytes / 2);
      }
      __syncwarp();
      if (pid >= 0) {
        uint8_t *k_dst = sK + s * kKStage;
        uint8_t *v_dst = sVst + s * kVstStage;
        const int row = (pid * hkv + g) * kPage;
        tc::tma_load_2d(k_dst + lane * 2048, &tmap_k, 0, row, &bars[kBarKFull + s]);
        tc::tma_load_2d(k_dst + kKBlk + lane * 2048, &tmap_k, 64, row, &bars[kBarKFull + s]);
        bulk_g2s(v_dst + lane * 2048, v_cache + static_cast<int64_t>(row) * kHeadDim, 2048,
                 &bars[kBarVstFull + s]);
      }
    }
    if (lane == 0) {
      // let the copies issued last on each stage land before shared memory
      // is released (at once on the normal path, where every copy has been
      // consumed); nothing else can be outstanding
      if (last0 >= 0) {
        mbar_wait_bounded(&bars[kBarKFull], (last0 >> 1) & 1);
        mbar_wait_bounded(&bars[kBarVstFull], (last0 >> 1) & 1);
      }
      if (last1 >= 0) {
        mbar_wait_bounded(&bars[kBarKFull + 1], (last1 >> 1) & 1);
        mbar_wait_bounded(&bars[kBarVstFull + 1], (last1 >> 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ================= MMA issue =================
    if (lane == 0) {
      constexpr uint32_t kIdescQK = tc::idesc_f16_f32(kRows, kKv, false, false);
      constexpr uint32_t kIdescPV = tc::idesc_f16_f32(kRows, kHeadDim, false, true);
      // Descriptors of every operand tile, built once; an MMA's operand is
      // its tile's descriptor plus a constant step in the start-address
      // field (16-byte units): +2 per 16 fp16 along K inside a 128-byte
      // row, +kKBlk/16 (or kQBytes/32) per 64-element K-block, +128 per
      // 16 positions of the MN-major V tile.
      const uint64_t dq0 = tc::smem_desc_sw128(smem_addr(sQ), 16, 1024);
      const uint64_t dq1 = tc::smem_desc_sw128(smem_addr(sQ + kQBytes), 16, 1024);
      const uint64_t dk0 = tc::smem_desc_sw128(smem_addr(sK), 16, 1024);
      const uint64_t dk1 = tc::smem_desc_sw128(smem_addr(sK + kKStage), 16, 1024);
      const uint64_t dv0 = tc::smem_desc_sw128(smem_addr(sV), kKBlk, 1024);
      const uint64_t dv1 = tc::smem_desc_sw128(smem_addr(sV + kVStage), kKBlk, 1024);
      auto issue_s = [&](int w, int j) {
        const uint64_t a0 = w ? dq1 : dq0, b0 = (j & 1) ? dk1 : dk0;
        const uint32_t d = tmem + w * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ao = static_cast<uint64_t>((kk >> 2) * (kQBytes / 2 / 16) + (kk & 3) * 2);
          const uint64_t bo = static_cast<uint64_t>((kk >> 2) * (kKBlk / 16) + (kk & 3) * 2);
          tc::mma_f16_ss(d, a0 + ao, b0 + bo, kIdescQK, kk > 0);
        }
        tc::mma_commit(&bars[kBarSFull + w]);
      };
      auto issue_pv = [&](int w, int j) {
        const uint64_t b0 = (j & 1) ? dv1 : dv0;
        const uint32_t a = tmem + w * 128;  // P_w: 8 columns per 16 positions
        const uint32_t d = tmem + 256 + w * 128;
        const bool acc0 = j > 0;
#pragma unroll
        for (int kk = 0; kk < kKv / 16; ++kk)
          tc::mma_f16_ts(d, a + kk * 8, b0 + static_cast<uint64_t>(kk * 128), kIdescPV,
                         acc0 || kk > 0);
        tc::mma_commit(&bars[kBarODone + w]);
      };
      const bool started =
          cta_wait(&bars[kBarQ], 0, abort_flag, dev_error, true) &&
          cta_wait(&bars[kBarKFull], 0, abort_flag, dev_error, true, withheld ? kTestSpins : 0);
      if (started) {
        tc::fence_after_sync();
        issue_s(0, 0);
        issue_s(1, 0);
        tc::mma_commit(&bars[kBarKEmpty]);
        for (int j = 0; j < n_kv; ++j) {
          const int s = j & 1;
          const bool more = j + 1 < n_kv;
          // P_A(j), V(j) and K(j+1) in one polling loop: V and K are nearly
          // always in place before P_A, so once P_A lands the two MMA groups
          // go out back to back, with no wait between them.
          if (!wait_all3(&bars[kBarPFull + 0], j & 1, &bars[kBarVFull + s], (j >> 1) & 1,
                         more ? &bars[kBarKFull + ((j + 1) & 1)] : nullptr, ((j + 1) >> 1) & 1,
                         abort_flag, dev_error))
            break;
          tc::fence_after_sync();
          issue_pv(0, j);
          if (more) issue_s(0, j + 1);
          if (!cta_wait(&bars[kBarPFull + 1], j & 1, abort_flag, dev_error, true)) break;
          tc::fence_after_sync();
          issue_pv(1, j);
          tc::mma_commit(&bars[kBarVEmpty + s]);
          if (more) {
            issue_s(1, j + 1);
            tc::mma_commit(&bars[kBarKEmpty + ((j + 1) & 1)]);
          }
        }
      }
      // let every MMA this thread issued land before tensor memory is
      // released: a commit tracks all of them (none: it completes at once)
      tc::mma_commit(&bars[kBarDrain]);
      mbar_wait_bounded(&bars[kBarDrain], 0);
      // and the query copy, which an abort before its wait would leave behind
      mbar_wait_bounded(&bars[kBarQ], 0);
    }
    __syncwarp();
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
  if (cudaFuncSetAttribute(prefill_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes)) != cudaSuccess ||
      cudaFuncSetAttribute(prefill_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes)) != cudaSuccess)
    return K16V8_ERR_CUDA;
  if (dev < 64) configured[dev] = true;
  return K16V8_OK;
}

}  // namespace prefill
}  // namespace k16v8

using namespace k16v8;
using namespace k16v8::prefill;

// KV parts per work item: kv_splits if given (clamped to 1..4), else the
// count (1..4) that best fills whole waves of one CTA per SM when the items
// make less than two waves (with two or more the tail is at most a third of
// a wave and items are usually short); ties go to fewer parts.  A known
// bound on the cached length caps the count at what the longest pair can
// use (the kernel gives a pair at most one part per 8 KV tiles), so a call
// over short prefixes launches no CTAs that would find nothing to do.
static int resolve_parts(int32_t kv_splits, int64_t items, int sms, int32_t max_seq_len) {
  if (kv_splits > 0) return std::min<int32_t>(kv_splits, kMaxKvParts);
  if (items <= 0 || sms <= 0 || items >= 2LL * sms) return 1;
  int cap = kMaxKvParts;
  if (max_seq_len > 0)
    cap = static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>(kMaxKvParts,
                             ((static_cast<int64_t>(max_seq_len) + kKv - 1) / kKv) / kMinPartTiles)));
  int best = 1;
  double best_fill = 0.0;
  for (int p = 1; p <= cap; ++p) {
    const double waves = static_cast<double>(items) * p / sms;
    const double fill = waves / std::ceil(waves - 1e-9);
    if (fill > best_fill + 1e-9) {
      best_fill = fill;
      best = p;
    }
  }
  return best;
}

struct PrefillWs {
  int parts;
  size_t counters_off, lse_off, o_off, total;
};

static PrefillWs prefill_ws(int32_t kv_splits, int32_t max_qlen, int32_t batch,
                            int32_t num_kv_heads, int32_t max_seq_len) {
  PrefillWs w{1, 0, 0, 0, 0};
  const int64_t max_pairs = (static_cast<int64_t>(max_qlen) + 2 * kQTok - 1) / (2 * kQTok);
  const int64_t items = max_pairs * num_kv_heads * batch;
  w.parts = resolve_parts(kv_splits, items, k16v8_sm_count(), max_seq_len);
  if (w.parts == 1) return w;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  w.lse_off = up(static_cast<size_t>(items) * 4);
  w.o_off = w.lse_off + up(static_cast<size_t>(items) * w.parts * 2 * kRows * 4);
  w.total = w.o_off + static_cast<size_t>(items) * w.parts * 2 * 16 * kRows * 16;
  return w;
}

static int32_t prefill_launch(
    const void *q, const int32_t *qo_indptr, int32_t total_q, int32_t max_qlen,
    const void *k_cache, const uint8_t *v_cache, const float *v_scale, const int32_t *block_table,
    int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t batch, int32_t num_qo_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t num_pages, float sm_scale, void *out,
    float *lse, int32_t *dev_error, void *stream, int32_t kv_splits, int32_t max_seq_len,
    void *workspace, size_t workspace_bytes, int32_t test_withhold = 0) {
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
  CUtensorMap mo;  // the output, same geometry and box as the query
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim),
                                static_cast<cuuint64_t>(num_qo_heads),
                                static_cast<cuuint64_t>(total_q)};
    const cuuint64_t strides[2] = {kHeadDim * 2ull,
                                   static_cast<cuuint64_t>(num_qo_heads) * kHeadDim * 2ull};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kGroup), static_cast<cuuint32_t>(kQTok)};
    const cuuint32_t es[3] = {1, 1, 1};
    if (encode(&mo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, out, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return K16V8_ERR_CUDA;
  }
  int32_t st = set_smem_attr();
  if (st != K16V8_OK) return st;
  const PrefillWs w = prefill_ws(kv_splits, max_qlen, batch, num_kv_heads, max_seq_len);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  if (w.parts > 1 && (!ws || !k16v8_aligned(ws, 256) || workspace_bytes < w.total))
    return ws ? K16V8_ERR_WORKSPACE_TOO_SMALL : K16V8_ERR_INVALID_ARG;
  const int64_t max_pairs = (static_cast<int64_t>(max_qlen) + 2 * kQTok - 1) / (2 * kQTok);
  if (max_pairs * w.parts >= (1LL << 31)) return K16V8_ERR_INVALID_ARG;
  const dim3 grid(static_cast<unsigned>(max_pairs * w.parts), num_kv_heads, batch);
  return k16v8_launch_pdl(
      w.parts > 1 ? prefill_kernel<true> : prefill_kernel<false>, grid, dim3(kThreads),
      kSmemBytes, static_cast<cudaStream_t>(stream), mq, mk,
      mo, v_cache, v_scale, qo_indptr, block_table, max_pages_per_seq, seq_lens, total_q,
      num_qo_heads, num_kv_heads, num_pages, sm_scale, static_cast<__half *>(out), lse, dev_error,
      static_cast<int32_t>(w.parts),
      w.parts > 1 ? reinterpret_cast<uint4 *>(ws + w.o_off) : nullptr,
      w.parts > 1 ? reinterpret_cast<float *>(ws + w.lse_off) : nullptr,
      w.parts > 1 ? reinterpret_cast<int32_t *>(ws + w.counters_off) : nullptr, test_withhold);
}

extern "C" int32_t k16v8_paged_prefill_attention(
    const void *q, const int32_t *qo_indptr, int32_t total_q, int32_t max_qlen,
    const void *k_cache, const uint8_t *v_cache, const float *v_scale, const int32_t *block_table,
    int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t batch, int32_t num_qo_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t num_pages, float sm_scale, void *out,
    float *lse, int32_t *dev_error, void *stream) {
  return prefill_launch(q, qo_indptr, total_q, max_qlen, k_cache, v_cache, v_scale, block_table,
                        max_pages_per_seq, seq_lens, batch, num_qo_heads, num_kv_heads, head_dim,
                        num_pages, sm_scale, out, lse, dev_error, stream, 1, 0, nullptr, 0);
}

extern "C" int32_t k16v8_paged_prefill_attention_wait_test(
    const void *q, const int32_t *qo_indptr, int32_t total_q, int32_t max_qlen,
    const void *k_cache, const uint8_t *v_cache, const float *v_scale, const int32_t *block_table,
    int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t batch, int32_t num_qo_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t num_pages, float sm_scale, void *out,
    float *lse, int32_t *dev_error, void *stream) {
  return prefill_launch(q, qo_indptr, total_q, max_qlen, k_cache, v_cache, v_scale, block_table,
                        max_pages_per_seq, seq_lens, batch, num_qo_heads, num_kv_heads, head_dim,
                        num_pages, sm_scale, out, lse, dev_error, stream, 1, 0, nullptr, 0,
                        /*test_withhold=*/1);
}

extern "C" size_t k16v8_prefill_workspace_size(int32_t max_qlen, int32_t batch,
                                               int32_t num_qo_heads, int32_t num_kv_heads,
                                               int32_t head_dim, int32_t kv_splits,
                                               int32_t max_seq_len) {
  if (max_qlen <= 0 || batch <= 0 || num_kv_heads <= 0 || head_dim != kHeadDim ||
      num_qo_heads != kGroup * num_kv_heads || kv_splits < 0 || max_seq_len < 0)
    return 0;
  return prefill_ws(kv_splits, max_qlen, batch, num_kv_heads, max_seq_len).total;
}

extern "C" int32_t k16v8_paged_prefill_attention_split(
    const void *q, const int32_t *qo_indptr, int32_t total_q, int32_t max_qlen,
    const void *k_cache, const uint8_t *v_cache, const float *v_scale, const int32_t *block_table,
    int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t batch, int32_t num_qo_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t num_pages, float sm_scale, int32_t kv_splits,
    int32_t max_seq_len, void *workspace, size_t workspace_bytes, void *out, float *lse,
    int32_t *dev_error, void *stream) {
  if (kv_splits < 0 || max_seq_len < 0) return K16V8_ERR_INVALID_ARG;
  return prefill_launch(q, qo_indptr, total_q, max_qlen, k_cache, v_cache, v_scale, block_table,
                        max_pages_per_seq, seq_lens, batch, num_qo_heads, num_kv_heads, head_dim,
                        num_pages, sm_scale, out, lse, dev_error, stream, kv_splits, max_seq_len,
                        workspace, workspace_bytes);
}
