// Load-balanced paged decode attention over the K16/V8 cache: every CTA of
// one full wave gets the same number of (page, KV head) tiles, whatever the
// mix of sequence lengths, and the log-sum-exp merge touches only the
// (sequence, KV head) segments that were split between CTAs.
//
// "Phi-4: quality transfer and interrupted throughput studies", intro: the
// format (FP16 K, E4M3 V with per-head scales) and the geometry (40 query
// heads over 10 KV heads, d = 128); "Matched diagnostic profiles": split-KV
// attention kernels followed by merge kernels.  The page fixes the result
// (softmax(q.K^T * sm_scale) V per query head, plus its LSE); how the work is
// cut into pieces is this file's choice.
//
// Work split.  Order all (sequence b, KV head g, page p) tiles as one flat
// list, b-major, then g, then p, so that each (b, g) segment of
// ceil(L_b / 16) tiles is contiguous.  With T tiles and G CTAs (one full
// wave: SMs x 4), CTA i takes the flat range [i*W, min((i+1)*W, T)),
// W = max(ceil(T/G), 4).  A range cuts at most two segments -- its first and
// its last -- and holds any number of whole ones.
//  * Inside a CTA the four warps stream the range's tiles interleaved (warp w
//    takes flat tiles i*W + w, + 4, ...) through the same per-warp bulk-copy
//    rings as the chunked kernel, without a break at segment boundaries.
//  * At the end of each segment piece the warps combine: warps 1-3 stage
//    their state in shared memory and go on to the next piece; warp 0 folds
//    the staged states into its own and writes the piece.  A whole segment
//    goes straight to the fp16 output and LSE; a cut one goes to partial
//    slot 0 (the CTA's first piece) or 1 (its last piece).
//  * The CTA derives its range from the sequence lengths itself (a block
//    scan of the page counts); CTA 0 also stores the scan (T, W and the
//    per-sequence page offsets) for the merge.
//  * The merge kernel rebuilds, per (sequence, query head), which CTAs cut
//    the segment and combines their partials; segments that one CTA held
//    whole are skipped, empty sequences get a zero row and LSE -inf.
//  * kAppend: the decode step's cache write folded in -- the warp that
//    consumes the page holding position L - 1 of a (b, g) segment quantises
//    the new token, stores it in the cache and in its staged copy of the
//    page before attending to it (each page of each head is one tile, held
//    by exactly one warp of the grid).
#include "decode_page.cuh"

namespace k16v8 {

constexpr int kBalCtasPerSm = kMinBlocks;
constexpr int kBalMinTiles = kWarps;  // at least one tile per warp
constexpr int kBalMaxBatch = 8192;    // the scan's page offsets live in the ring space
constexpr int kPrefetchTiles = 2;      // per warp, into L2 before the dependency wait
constexpr int kMergeFast = 8;          // cut pieces merged from one round of loads

// Cross-warp combine staging (warps 1..3) plus a few scalars.
struct BalStage {
  float o[kWarps - 1][kGroup][kHeadDim];
  float m[kWarps - 1][kGroup];
  float l[kWarps - 1][kGroup];
  uint64_t bar[kWarps][kStages];  // outside the rings: set up while the scan scratch is live
  int32_t aux[4];
};
constexpr size_t kBalSmemBytes = kWarps * sizeof(WarpRing) + sizeof(BalStage);
static_assert(static_cast<size_t>(kBalMaxBatch + 1) * sizeof(int32_t) <=
                  kWarps * sizeof(WarpRing),
              "scan scratch must fit in the ring space");

// Workspace: [plan int32: T, W, P(0..batch)] [partial o: G x 2 x 4 x 128 fp32]
// [partial lse: G x 2 x 4 fp32], each part 256-byte aligned.
struct BalLayout {
  size_t plan_off, o_off, lse_off, total;
};
static inline size_t bal_align(size_t x) { return (x + 255) / 256 * 256; }
static BalLayout bal_layout(int32_t batch, int32_t ctas) {
  BalLayout w;
  w.plan_off = 0;
  w.o_off = bal_align((static_cast<size_t>(batch) + 3) * sizeof(int32_t));
  w.lse_off = w.o_off + bal_align(static_cast<size_t>(ctas) * 2 * kGroup * kHeadDim * sizeof(float));
  w.total = w.lse_off + bal_align(static_cast<size_t>(ctas) * 2 * kGroup * sizeof(float));
  return w;
}

__device__ __forceinline__ int clamped_len(const int32_t *seq_lens, int b, int cap) {
  const int L = __ldg(seq_lens + b);
  return max(0, min(L, cap));
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int threads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// A (sequence, KV head) segment of the flat tile list: flat tiles
// [s0, s0 + np) are pages 0..np-1 of sequence b under KV head g.
struct Segment {
  int b, g, s0, np, L;
  // Step to the next non-empty segment.  Only called while the next one
  // exists (the current one ends before the CTA's range does).
  __device__ __forceinline__ void next(const int32_t *seq_lens, int hkv, int cap) {
    s0 += np;
    if (++g == hkv) {
      g = 0;
      do {
        ++b;
        L = clamped_len(seq_lens, b, cap);
        np = (L + kPage - 1) / kPage;
      } while (np == 0);
    }
  }
};

template <bool kAppend>
__global__ void __launch_bounds__(kWarps * 32, kBalCtasPerSm) decode_balanced_kernel(
    const __half *__restrict__ q, __half *__restrict__ k_cache, uint8_t *__restrict__ v_cache,
    const float *__restrict__ v_scale,
    const int32_t *__restrict__ block_table, int32_t maxp, const int32_t *__restrict__ seq_lens,
    int32_t batch, int32_t hq, int32_t hkv, int32_t num_pages, float sm_scale,
    int32_t *__restrict__ plan, float *__restrict__ part_o, float *__restrict__ part_lse,
    __half *__restrict__ out, float *__restrict__ lse_out, const __half *__restrict__ k_new,
    const __half *__restrict__ v_new, int32_t *dev_error, int32_t flags) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  WarpRing *rings = reinterpret_cast<WarpRing *>(smem_raw);
  BalStage &stg = *reinterpret_cast<BalStage *>(smem_raw + kWarps * sizeof(WarpRing));
  int32_t *ps = reinterpret_cast<int32_t *>(smem_raw);  // scan scratch, before the rings run

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cap = maxp * kPage;
  // Block table and lengths may be read before the preceding kernel has
  // finished only when the caller says they are not written by it.
  const bool early = flags & K16V8_DECODE_METADATA_READY;
  if (!early) pdl_wait();

  // ---- exclusive scan of the per-sequence page counts ----
  int carry = 0;
  for (int base = 0; base < batch; base += kWarps * 32) {
    const int b = base + threadIdx.x;
    int np = 0;
    if (b < batch) {
      int L = __ldg(seq_lens + b);
      if (L < 0 || L > cap) {
        if (blockIdx.x == 0) flag_error(dev_error, K16V8_DEVERR_SEQLEN);
        L = max(0, min(L, cap));
      }
      np = (L + kPage - 1) / kPage;
    }
    int x = np;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(kFull, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) stg.aux[warp] = x;
    __syncthreads();
    int pre = carry, tot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int v = stg.aux[w];
      if (w < warp) pre += v;
      tot += v;
    }
    if (b < batch) ps[b] = pre + x - np;
    carry += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) ps[batch] = carry;
  __syncthreads();

  const int T = carry * hkv;
  const int G = gridDim.x;
  const int W = max((T + G - 1) / G, kBalMinTiles);
  const int a = static_cast<int>(blockIdx.x) * W;
  const int e = min(a + W, T);
  const int n_my = e - a > warp ? (e - a - warp + kWarps - 1) / kWarps : 0;

  // Segment holding flat tile f (ps scratch still live): largest b with
  // ps[b] * hkv <= f, then the KV head within it.
  auto segment_of = [&](int f) {
    int lo = 0, hi = batch;  // ps[batch] * hkv = T > f
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ps[mid] * hkv <= f) lo = mid; else hi = mid;
    }
    Segment sg;
    sg.b = lo;
    sg.np = ps[lo + 1] - ps[lo];
    sg.g = (f - ps[lo] * hkv) / sg.np;
    sg.s0 = ps[lo] * hkv + sg.g * sg.np;
    sg.L = 0;  // filled by the caller when needed
    return sg;
  };
  // Lane l of a batch describes this warp's tile number base + l (flat
  // a + warp + 4 * (base + l)) as pid * hkv + g, -1 for a rejected page id,
  // -2 past the warp's last tile.  `walk` is a segment at or before the
  // batch's first tile; on return it is the segment of the batch's last tile.
  auto describe = [&](int base, Segment &walk, bool scratch_live) {
    const int k = base + lane;
    int t = -2;
    Segment sg = walk;
    if (k < n_my) {
      const int f = a + warp + kWarps * k;
      if (scratch_live) {
        sg = segment_of(f);
      } else {
        while (f >= sg.s0 + sg.np) sg.next(seq_lens, hkv, cap);
      }
      const int pid = __ldg(block_table + static_cast<int64_t>(sg.b) * maxp + (f - sg.s0));
      if (pid < 0 || pid >= num_pages) {
        flag_error(dev_error, K16V8_DEVERR_PAGE);
        t = -1;
      } else {
        t = pid * hkv + sg.g;
      }
    }
    const int last = min(31, n_my - 1 - base);
    walk.b = __shfl_sync(kFull, sg.b, last);
    walk.g = __shfl_sync(kFull, sg.g, last);
    walk.s0 = __shfl_sync(kFull, sg.s0, last);
    walk.np = __shfl_sync(kFull, sg.np, last);
    walk.L = clamped_len(seq_lens, walk.b, cap);
    return t;
  };

  Segment seg0{0, 0, 0, 0, 0};
  if (a < T) {
    seg0 = segment_of(a);
    seg0.L = clamped_len(seq_lens, seg0.b, cap);
  }
  Segment walk = seg0;
  int desc_cur = -2, desc_nxt = -2;
  if (n_my > 0) {  // implies a < T
    desc_cur = describe(0, walk, true);
    if (n_my > 32) desc_nxt = describe(32, walk, false);
  }
  if (early && lane < kPrefetchTiles && desc_cur >= 0) {
    // While the preceding kernel finishes, start this warp's first pages on
    // their way into L2 (the copies into shared memory wait below).
    const int64_t off = static_cast<int64_t>(desc_cur) * kPage * kHeadDim;
    bulk_prefetch_l2(k_cache + off, kKPageBytes);
    bulk_prefetch_l2(v_cache + off, kVPageBytes);
  }
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(&stg.bar[warp][s], 1);
    fence_barrier_init();
  }
  if (early) pdl_wait();
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i <= batch; i += blockDim.x) plan[2 + i] = ps[i];
    if (threadIdx.x == 0) {
      plan[0] = T;
      plan[1] = W;
    }
  }
  __syncthreads();  // the scan scratch becomes ring space below
  if (a >= T) return;  // no tiles for this CTA (uniform over the CTA)

  WarpRing &ring = rings[warp];
  uint64_t *bars = stg.bar[warp];
  constexpr int64_t kTileElems = static_cast<int64_t>(kPage) * kHeadDim;
  const uint64_t policy = l2_policy_evict_first();

  // ---- issue side: warp-wide (descriptor shuffle), lane 0 copies ----
  int ki = 0;  // tiles issued
  auto issue = [&]() {
    const int s = ki % kStages;
    const int t = __shfl_sync(kFull, desc_cur, ki & 31);
    if (lane == 0) {
      if (t < 0) {
        ring.live[s] = 0;
        mbar_arrive(&bars[s]);  // nothing to load: complete the phase empty
      } else {
        ring.live[s] = t + 1;  // t < 2^31 - 1 (checked on the host)
        const int64_t off = static_cast<int64_t>(t) * kTileElems;
        mbar_arrive_expect_tx(&bars[s], kKPageBytes + kVPageBytes);
        bulk_g2s_evict_first(ring.k[s], k_cache + off, kKPageBytes, &bars[s], policy);
        bulk_g2s_evict_first(ring.v[s], v_cache + off, kVPageBytes, &bars[s], policy);
      }
    }
    ++ki;
    if ((ki & 31) == 0 && ki < n_my) {  // next batch of descriptors
      desc_cur = desc_nxt;
      if (ki + 32 < n_my) desc_nxt = describe(ki + 32, walk, false);
    }
  };
  for (int k = 0; k < min(kStages, n_my); ++k) issue();

  const int j = lane & 7;
  const int hsel = j >> 1;
  const float qs = sm_scale * kLog2e;

  Segment cs = seg0;   // segment of the current piece
  int fc = a + warp;   // this warp's next flat tile to consume
  int kc = 0;          // tiles consumed
  int fail_k = -1;     // first tile whose wait gave up
  bool ok = true;
  int piece = 0;
  while (true) {
    uint32_t qf[16];
    load_group_query(q + (static_cast<int64_t>(cs.b) * hq + cs.g * kGroup) * kHeadDim, qf);
    WarpState st;
    st.reset();
    const int seg_end = cs.s0 + cs.np;
    const int pe = min(seg_end, e);
    for (; fc < pe; fc += kWarps, ++kc) {
      const int s = kc % kStages;
      if (ok) {
        ok = __all_sync(kFull, mbar_wait_bounded(&bars[s], (kc / kStages) & 1));
        if (!ok) fail_k = kc;
      }
      if (ok) {
        if (ring.live[s]) {
          const int valid = min(kPage, cs.L - (fc - cs.s0) * kPage);
          if constexpr (kAppend) {
            if (fc - cs.s0 == (cs.L - 1) / kPage) {  // the page of position L - 1
              const int64_t src = (static_cast<int64_t>(cs.b) * hkv + cs.g) * kHeadDim;
              append_new_row(ring, s, (cs.L - 1) % kPage, k_new + src, v_new + src,
                             __ldg(v_scale + cs.g), k_cache, v_cache, ring.live[s] - 1);
            }
          }
          attend_page<false>(ring, s, valid, qf, qs, st);
        }
        __syncwarp();
        if (ki < n_my) {
          if (lane == 0) fence_proxy_async();
          issue();
        }
      }
    }
    const bool last = pe >= e;
    if (last) pdl_launch_dependents();

    // ---- combine the four warps' states for this piece ----
    st.finish();  // m, l of head hsel in every lane
    const float l_run = st.l;
    if (warp > 0) {
      if (piece > 0) named_bar_sync(2, kWarps * 32);  // warp 0 has read the last staging
#pragma unroll
      for (int h = 0; h < kGroup; ++h)
        *reinterpret_cast<float4 *>(&stg.o[warp - 1][h][lane * 4]) =
            make_float4(st.o[h][0].x, st.o[h][0].y, st.o[h][1].x, st.o[h][1].y);
      if (lane < 8 && (lane & 1) == 0) {
        stg.m[warp - 1][hsel] = st.m;
        stg.l[warp - 1][hsel] = l_run;
      }
      named_bar_arrive(1, kWarps * 32);
    } else {
      named_bar_sync(1, kWarps * 32);
      const bool whole = cs.s0 >= a && seg_end <= e;
      const int slot = piece == 0 ? 0 : 1;
      const float vs = __ldg(v_scale + cs.g);
#pragma unroll
      for (int h = 0; h < kGroup; ++h) {
        const float m0 = __shfl_sync(kFull, st.m, 2 * h);
        const float l0 = __shfl_sync(kFull, l_run, 2 * h);
        float M = m0;
#pragma unroll
        for (int w = 0; w < kWarps - 1; ++w) M = fmaxf(M, stg.m[w][h]);
        float Ls = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
          const float w0 = m0 == -INFINITY ? 0.f : ex2(m0 - M);
          Ls = w0 * l0;
          acc = make_float4(w0 * st.o[h][0].x, w0 * st.o[h][0].y, w0 * st.o[h][1].x,
                            w0 * st.o[h][1].y);
#pragma unroll
          for (int w = 0; w < kWarps - 1; ++w) {
            const float mw = stg.m[w][h];
            const float sw = mw == -INFINITY ? 0.f : ex2(mw - M);
            Ls += sw * stg.l[w][h];
            const float4 ow = *reinterpret_cast<const float4 *>(&stg.o[w][h][lane * 4]);
            acc.x += sw * ow.x;
            acc.y += sw * ow.y;
            acc.z += sw * ow.z;
            acc.w += sw * ow.w;
          }
        }
        float lse = -INFINITY;
        float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
        if (Ls > 0.f) {
          const float inv = vs / Ls;
          res = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
          lse = (M + lg2(Ls)) * kLn2;
        }
        const int qhd = cs.g * kGroup + h;
        if (whole) {
          uint2 o2;
          o2.x = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(res.x))) |
                 (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(res.y))) << 16);
          o2.y = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(res.z))) |
                 (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(res.w))) << 16);
          *reinterpret_cast<uint2 *>(out + (static_cast<int64_t>(cs.b) * hq + qhd) * kHeadDim +
                                     lane * 4) = o2;
          if (lane == 0 && lse_out) lse_out[static_cast<int64_t>(cs.b) * hq + qhd] = lse;
        } else {
          const int64_t row = (static_cast<int64_t>(blockIdx.x) * 2 + slot) * kGroup + h;
          *reinterpret_cast<float4 *>(part_o + row * kHeadDim + lane * 4) = res;
          if (lane == 0) part_lse[row] = lse;
        }
      }
      if (!last) named_bar_arrive(2, kWarps * 32);
    }
    if (last) break;
    cs.next(seq_lens, hkv, cap);
    ++piece;
  }

  if (!ok) {
    // Report, then drain the copies still in flight (bounded) so none lands
    // after the CTA exits.
    if (lane == 0) {
      flag_error(dev_error, K16V8_DEVERR_TIMEOUT);
      for (int kk = fail_k; kk < ki; ++kk)
        mbar_wait_bounded(&bars[kk % kStages], (kk / kStages) & 1);
    }
    __syncwarp();
  }
}

// One warp per (sequence, query head): combine the partials of the CTAs that
// cut this row's (sequence, KV head) segment; lane owns 4 dims.
__global__ void __launch_bounds__(128, 8) merge_balanced_kernel(
    const float *__restrict__ part_o, const float *__restrict__ part_lse,
    const int32_t *__restrict__ plan, int32_t rows, int32_t hq, int32_t hkv,
    __half *__restrict__ out, float *__restrict__ lse_out) {
  const int wid = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_launch_dependents();
  if (wid >= rows) return;
  const int b = wid / hq, h = wid % hq;
  const int g = h / kGroup, hh = h % kGroup;
  const int W = __ldg(plan + 1);
  const int pb = __ldg(plan + 2 + b);
  const int np = __ldg(plan + 3 + b) - pb;
  float M = -INFINITY, S = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (np > 0) {
    const int s0 = pb * hkv + g * np;
    const int i0 = s0 / W, i1 = (s0 + np - 1) / W;
    if (i0 == i1) return;  // held whole by one CTA, which wrote the row
    const int n = i1 - i0 + 1;
    const int slot0 = s0 == i0 * W ? 0 : 1;
    auto row_of = [&](int c) {  // partial row of the c-th cutting CTA
      return (static_cast<int64_t>(i0 + c) * 2 + (c == 0 ? slot0 : 0)) * kGroup + hh;
    };
    if (n <= kMergeFast) {
      // Every partial of the segment in one round of loads (the common
      // case: a segment is cut by a few CTAs), then the same sums in the
      // same order as the general loop below.
      const float lc = lane < n ? __ldg(part_lse + row_of(lane)) : -INFINITY;
      float4 oc[kMergeFast];
#pragma unroll
      for (int c = 0; c < kMergeFast; ++c)
        oc[c] = c < n ? __ldg(reinterpret_cast<const float4 *>(part_o + row_of(c) * kHeadDim +
                                                               lane * 4))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      float lw[kMergeFast];
#pragma unroll
      for (int c = 0; c < kMergeFast; ++c) {
        lw[c] = __shfl_sync(kFull, lc, c);
        M = fmaxf(M, lw[c]);
      }
      if (M != -INFINITY) {
#pragma unroll
        for (int c = 0; c < kMergeFast; ++c) {
          if (c < n) {
            const float wu = ex2((lw[c] - M) * kLog2e);
            S += wu;
            acc.x = fmaf(wu, oc[c].x, acc.x);
            acc.y = fmaf(wu, oc[c].y, acc.y);
            acc.z = fmaf(wu, oc[c].z, acc.z);
            acc.w = fmaf(wu, oc[c].w, acc.w);
          }
        }
      }
    } else {
      for (int c = lane; c < n; c += 32) M = fmaxf(M, __ldg(part_lse + row_of(c)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
      if (M != -INFINITY) {
        for (int c = 0; c < n; ++c) {
          const int64_t r = row_of(c);
          const float4 oc =
              __ldg(reinterpret_cast<const float4 *>(part_o + r * kHeadDim + lane * 4));
          const float wu = ex2((__ldg(part_lse + r) - M) * kLog2e);
          S += wu;
          acc.x = fmaf(wu, oc.x, acc.x);
          acc.y = fmaf(wu, oc.y, acc.y);
          acc.z = fmaf(wu, oc.z, acc.z);
          acc.w = fmaf(wu, oc.w, acc.w);
        }
      }
    }
  }
  float lse = -INFINITY;
  if (S > 0.f) {
    const float inv = rcp(S);
    acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    lse = M + lg2(S) * kLn2;
  }
  uint2 st;
  st.x = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.x))) |
         (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.y))) << 16);
  st.y = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.z))) |
         (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.w))) << 16);
  *reinterpret_cast<uint2 *>(out + static_cast<int64_t>(wid) * kHeadDim + lane * 4) = st;
  if (lane == 0 && lse_out) lse_out[wid] = lse;
}

static int32_t bal_ctas(int32_t *ctas) {
  const int sms = k16v8_sm_count();
  if (sms <= 0) return K16V8_ERR_CUDA;
  *ctas = sms * kBalCtasPerSm;
  return K16V8_OK;
}

}  // namespace k16v8

using namespace k16v8;

extern "C" size_t k16v8_decode_balanced_workspace_size(int32_t batch, int32_t num_qo_heads,
                                                       int32_t head_dim) {
  if (batch < 0 || batch > kBalMaxBatch || num_qo_heads <= 0 || head_dim != kHeadDim) return 0;
  int32_t ctas = 0;
  if (bal_ctas(&ctas) != K16V8_OK) return 0;
  return bal_layout(batch, ctas).total;
}

static int32_t bal_check(int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
                         int32_t head_dim, BalLayout *w) {
  if (num_qo_heads <= 0 || num_kv_heads <= 0) return K16V8_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || num_qo_heads != kGroup * num_kv_heads)
    return K16V8_ERR_UNSUPPORTED_SHAPE;
  if (batch < 0 || batch > kBalMaxBatch) return K16V8_ERR_INVALID_ARG;
  int32_t ctas = 0;
  const int32_t st = bal_ctas(&ctas);
  if (st != K16V8_OK) return st;
  *w = bal_layout(batch, ctas);
  return K16V8_OK;
}

template <bool kAppend>
static int32_t balanced_split(const void *q, const void *k_new, const void *v_new, void *k_cache,
                              uint8_t *v_cache, const float *v_scale, const int32_t *block_table,
                              int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t batch,
                              int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t num_pages, float sm_scale, void *workspace,
                              size_t workspace_bytes, void *out, float *lse, int32_t flags,
                              int32_t *dev_error, void *stream) {
  BalLayout w;
  int32_t st = bal_check(batch, num_qo_heads, num_kv_heads, head_dim, &w);
  if (st != K16V8_OK) return st;
  if (num_pages <= 0 || max_pages_per_seq < 0) return K16V8_ERR_INVALID_ARG;
  if (flags & ~K16V8_DECODE_METADATA_READY) return K16V8_ERR_INVALID_ARG;
  // Tile indices pid * num_kv_heads + g are int32.
  if (static_cast<int64_t>(num_pages) * num_kv_heads >= (1LL << 31) - 1)
    return K16V8_ERR_INVALID_ARG;
  // Flat tile indices are int32: batch * max_pages * num_kv_heads must fit.
  if (static_cast<int64_t>(batch) * max_pages_per_seq * num_kv_heads >= (1LL << 31) - 256 ||
      static_cast<int64_t>(max_pages_per_seq) * kPage >= (1LL << 31))
    return K16V8_ERR_INVALID_ARG;
  if (batch == 0) return K16V8_OK;
  if (!q || !k_cache || !v_cache || !v_scale || !block_table || !seq_lens || !workspace || !out)
    return K16V8_ERR_INVALID_ARG;
  if (!k16v8_aligned(q, 16) || !k16v8_aligned(k_cache, 16) || !k16v8_aligned(v_cache, 16) ||
      !k16v8_aligned(workspace, 256) || !k16v8_aligned(block_table, 4) ||
      !k16v8_aligned(seq_lens, 4) || !k16v8_aligned(v_scale, 4) || !k16v8_aligned(out, 8) ||
      (lse && !k16v8_aligned(lse, 4)))
    return K16V8_ERR_INVALID_ARG;
  if (kAppend && (!k_new || !v_new || !k16v8_aligned(k_new, 16) || !k16v8_aligned(v_new, 16)))
    return K16V8_ERR_INVALID_ARG;
  if (workspace_bytes < w.total) return K16V8_ERR_WORKSPACE_TOO_SMALL;
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return K16V8_ERR_CUDA;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    if (cudaFuncSetAttribute(decode_balanced_kernel<kAppend>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kBalSmemBytes)) != cudaSuccess)
      return K16V8_ERR_CUDA;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  int32_t ctas = 0;
  st = bal_ctas(&ctas);
  if (st != K16V8_OK) return st;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  return k16v8_launch_pdl(
      decode_balanced_kernel<kAppend>, dim3(ctas), dim3(kWarps * 32), kBalSmemBytes,
      static_cast<cudaStream_t>(stream), static_cast<const __half *>(q),
      static_cast<__half *>(k_cache), v_cache, v_scale, block_table, max_pages_per_seq, seq_lens,
      batch, num_qo_heads, num_kv_heads, num_pages, sm_scale,
      reinterpret_cast<int32_t *>(ws + w.plan_off), reinterpret_cast<float *>(ws + w.o_off),
      reinterpret_cast<float *>(ws + w.lse_off), static_cast<__half *>(out), lse,
      static_cast<const __half *>(k_new), static_cast<const __half *>(v_new), dev_error, flags);
}

extern "C" int32_t k16v8_paged_decode_balanced_split(
    const void *q, const void *k_cache, const uint8_t *v_cache, const float *v_scale,
    const int32_t *block_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
    int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t num_pages, float sm_scale, void *workspace, size_t workspace_bytes, void *out,
    float *lse, int32_t flags, int32_t *dev_error, void *stream) {
  // The kernel only reads the cache when it does not append.
  return balanced_split<false>(q, nullptr, nullptr, const_cast<void *>(k_cache),
                               const_cast<uint8_t *>(v_cache), v_scale, block_table,
                               max_pages_per_seq, seq_lens, batch, num_qo_heads, num_kv_heads,
                               head_dim, num_pages, sm_scale, workspace, workspace_bytes, out, lse,
                               flags, dev_error, stream);
}

extern "C" int32_t k16v8_paged_decode_append_balanced_split(
    const void *q, const void *k_new, const void *v_new, void *k_cache, uint8_t *v_cache,
    const float *v_scale, const int32_t *block_table, int32_t max_pages_per_seq,
    const int32_t *seq_lens, int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t num_pages, float sm_scale, void *workspace, size_t workspace_bytes,
    void *out, float *lse, int32_t flags, int32_t *dev_error, void *stream) {
  return balanced_split<true>(q, k_new, v_new, k_cache, v_cache, v_scale, block_table,
                              max_pages_per_seq, seq_lens, batch, num_qo_heads, num_kv_heads,
                              head_dim, num_pages, sm_scale, workspace, workspace_bytes, out, lse,
                              flags, dev_error, stream);
}

extern "C" int32_t k16v8_merge_balanced(const void *workspace, size_t workspace_bytes,
                                        int32_t batch, int32_t num_qo_heads,
                                        int32_t num_kv_heads, int32_t head_dim, void *out,
                                        float *lse, void *stream) {
  BalLayout w;
  const int32_t st = bal_check(batch, num_qo_heads, num_kv_heads, head_dim, &w);
  if (st != K16V8_OK) return st;
  if (batch == 0) return K16V8_OK;
  if (!workspace || !out || !k16v8_aligned(workspace, 256) || !k16v8_aligned(out, 8) ||
      (lse && !k16v8_aligned(lse, 4)))
    return K16V8_ERR_INVALID_ARG;
  if (workspace_bytes < w.total) return K16V8_ERR_WORKSPACE_TOO_SMALL;
  const uint8_t *ws = static_cast<const uint8_t *>(workspace);
  const int64_t rows = static_cast<int64_t>(batch) * num_qo_heads;
  return k16v8_launch_pdl(merge_balanced_kernel, dim3(static_cast<unsigned>((rows + 3) / 4)),
                          dim3(128), 0, static_cast<cudaStream_t>(stream),
                          reinterpret_cast<const float *>(ws + w.o_off),
                          reinterpret_cast<const float *>(ws + w.lse_off),
                          reinterpret_cast<const int32_t *>(ws + w.plan_off),
                          static_cast<int32_t>(rows), num_qo_heads, num_kv_heads,
                          static_cast<__half *>(out), lse);
}

extern "C" int32_t k16v8_paged_decode_attention_balanced(
    const void *q, const void *k_cache, const uint8_t *v_cache, const float *v_scale,
    const int32_t *block_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
    int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t num_pages, float sm_scale, void *workspace, size_t workspace_bytes, void *out,
    float *lse, int32_t flags, int32_t *dev_error, void *stream) {
  const int32_t st = k16v8_paged_decode_balanced_split(
      q, k_cache, v_cache, v_scale, block_table, max_pages_per_seq, seq_lens, batch,
      num_qo_heads, num_kv_heads, head_dim, num_pages, sm_scale, workspace, workspace_bytes, out,
      lse, flags, dev_error, stream);
  if (st != K16V8_OK || batch == 0) return st;
  return k16v8_merge_balanced(workspace, workspace_bytes, batch, num_qo_heads, num_kv_heads,
                              head_dim, out, lse, stream);
}

extern "C" int32_t k16v8_paged_decode_append_attention_balanced(
    const void *q, const void *k_new, const void *v_new, void *k_cache, uint8_t *v_cache,
    const float *v_scale, const int32_t *block_table, int32_t max_pages_per_seq,
    const int32_t *seq_lens, int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t num_pages, float sm_scale, void *workspace, size_t workspace_bytes,
    void *out, float *lse, int32_t flags, int32_t *dev_error, void *stream) {
  const int32_t st = k16v8_paged_decode_append_balanced_split(
      q, k_new, v_new, k_cache, v_cache, v_scale, block_table, max_pages_per_seq, seq_lens, batch,
      num_qo_heads, num_kv_heads, head_dim, num_pages, sm_scale, workspace, workspace_bytes, out,
      lse, flags, dev_error, stream);
  if (st != K16V8_OK || batch == 0) return st;
  return k16v8_merge_balanced(workspace, workspace_bytes, batch, num_qo_heads, num_kv_heads,
                              head_dim, out, lse, stream);
}
