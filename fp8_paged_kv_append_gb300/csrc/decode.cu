// Paged split-KV decode attention over the K16/V8 cache, and the
// log-sum-exp merge of its partials.
//
// "Phi-4: quality transfer and interrupted throughput studies": the intro
// gives the format (FP16 K, E4M3 V with per-head scales) and the geometry
// (40 query heads over 10 KV heads, d = 128); "Matched diagnostic profiles"
// names the attention and merge kernels.
//
// Design (HBM-bound; 3 bytes of cache per element pair):
//  * One CTA per (split chunk, KV head, sequence); four warps.  The four
//    query heads of the GQA group share every K/V page read.
//  * Each warp streams its own pages (pages w, w+4, ... of the chunk)
//    through a kStages-deep ring in shared memory.  One lane issues two
//    bulk-async copies per page -- the 4 KB K tile and the 2 KB V tile of one
//    (page, KV head) are contiguous in the cache layout -- completing on an
//    mbarrier; no register staging, no address arithmetic per element.
//  * Per page: Q.K, online softmax and P.V as in decode_page.cuh; the
//    per-head value scale is applied once to the final partial.
//  * The four warps' states are combined in shared memory; the CTA writes
//    one fp32 partial row per query head plus its natural-log LSE.
//  * Launched with programmatic stream serialization: griddepcontrol.wait
//    precedes every read of inputs.
#include "decode_page.cuh"

namespace k16v8 {

__host__ __device__ constexpr size_t ids_bytes(int split_chunk) {
  return ((static_cast<size_t>(split_chunk / kPage) * sizeof(int) + 15) / 16) * 16;
}
static size_t decode_smem_bytes(int split_chunk, bool vf16) {
  return kWarps * (vf16 ? sizeof(WarpRing16) : sizeof(WarpRing)) + ids_bytes(split_chunk);
}

// kAppend: also write each sequence's new token (k_new / v_new, position
// L - 1) into the cache -- the warp that consumes that page quantises the
// row, stores it, and writes it into its staged copy of the page, so the
// attention sees the quantised value without a separate append launch.
// kVF16: the FP16-KV control -- values stored as fp16 (4 KB per page
// tile), no dequantisation and no scale.
template <bool kAppend, bool kVF16>
__global__ void __launch_bounds__(kWarps * 32, kVF16 ? 3 : kMinBlocks) decode_split_kernel(
    const __half *__restrict__ q, __half *__restrict__ k_cache, uint8_t *__restrict__ v_cache,
    const float *__restrict__ v_scale, const int32_t *__restrict__ block_table, int32_t maxp,
    const int32_t *__restrict__ seq_lens, int32_t hq, int32_t hkv, int32_t num_pages,
    float sm_scale, int32_t chunk, int32_t max_chunks, float *__restrict__ part_o,
    float *__restrict__ part_lse, const __half *__restrict__ k_new,
    const __half *__restrict__ v_new, int32_t *dev_error, int32_t test_skip_page,
    __half *__restrict__ out, float *__restrict__ lse_out) {
  using Ring = WarpRingT<kVF16 ? 2 * kVPageBytes : kVPageBytes>;
  constexpr uint32_t kVTile = kVF16 ? 2 * kVPageBytes : kVPageBytes;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Ring *rings = reinterpret_cast<Ring *>(smem_raw);
  int *page_ids = reinterpret_cast<int *>(smem_raw + kWarps * sizeof(Ring));

  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();

  int L = __ldg(seq_lens + b);
  const int cap = min(maxp * kPage, max_chunks * chunk);
  if (L < 0 || L > cap) {
    if (threadIdx.x == 0 && c == 0 && g == 0) flag_error(dev_error, K16V8_DEVERR_SEQLEN);
    L = max(0, min(L, cap));
  }
  const int start = c * chunk;
  if (start >= L) {  // chunk past the end of this sequence
    // With one chunk the CTA writes the final rows (out != null): an empty
    // sequence gets zero rows and LSE -inf, as the merge would give.
    if (out) {
      const int h = threadIdx.x >> 5;
      const int64_t orow = static_cast<int64_t>(b) * hq + g * kGroup + h;
      *reinterpret_cast<uint2 *>(out + orow * kHeadDim + lane * 4) = make_uint2(0u, 0u);
      if (lane == 0 && lse_out) lse_out[orow] = -INFINITY;
    }
    return;
  }
  const int n_tok = min(chunk, L - start);
  const int n_pages = (n_tok + kPage - 1) / kPage;

  const int32_t *bt = block_table + static_cast<int64_t>(b) * maxp + start / kPage;
  for (int i = threadIdx.x; i < n_pages; i += blockDim.x) {
    int pid = __ldg(bt + i);
    if (pid < 0 || pid >= num_pages) {
      flag_error(dev_error, K16V8_DEVERR_PAGE);
      pid = -1;
    }
    page_ids[i] = pid;
  }
  // Page (within this chunk) that receives the new token, or -1.
  int patch_page = -1;
  if constexpr (kAppend) {
    if (L > 0 && (L - 1) / chunk == c) patch_page = (L - 1) / kPage - start / kPage;
  }
  Ring &ring = rings[warp];
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(&ring.bar[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  const int n_my = warp < n_pages ? (n_pages - warp + kWarps - 1) / kWarps : 0;
  const int64_t head_tile = static_cast<int64_t>(kPage) * kHeadDim;  // elements per (page, head)
  const uint64_t policy = l2_policy_evict_first();
  // Bounded-wait test hook (test_skip_page >= 0, never in production calls):
  // warp 0 of the first CTA withholds its copy of page slot test_skip_page
  // -- no arrival, nothing in flight -- so its wait for that page expires
  // after kTestPolls polls and the error path below runs.
  const bool withheld = test_skip_page >= 0 && (c | g | b | warp) == 0;
  auto issue = [&](int k) {
    if (withheld && k == test_skip_page) return;
    const int s = k % kStages;
    const int pid = page_ids[warp + k * kWarps];
    if (pid < 0) {
      mbar_arrive(&ring.bar[s]);  // nothing to load: complete the phase empty
      return;
    }
    const int64_t tile = (static_cast<int64_t>(pid) * hkv + g) * head_tile;
    mbar_arrive_expect_tx(&ring.bar[s], kKPageBytes + kVTile);
    bulk_g2s_evict_first(ring.k[s], k_cache + tile, kKPageBytes, &ring.bar[s], policy);
    bulk_g2s_evict_first(ring.v[s], v_cache + tile * (kVF16 ? 2 : 1), kVTile, &ring.bar[s],
                         policy);
  };
  if (lane == 0)
    for (int k = 0; k < min(kStages, n_my); ++k) issue(k);

  const int j = lane & 7;
  uint32_t qf[16];
  load_group_query(q + (static_cast<int64_t>(b) * hq + g * kGroup) * kHeadDim, qf);
  const float qs = sm_scale * kLog2e;  // scores in the log2 domain

  const int hsel = j >> 1;  // head whose score this lane holds
  WarpState st;
  st.reset();

  int k = 0;
  bool ok = true;
  for (; k < n_my; ++k) {
    const int s = k % kStages;
    ok = __all_sync(kFull, mbar_wait_bounded(&ring.bar[s], (k / kStages) & 1,
                                             withheld && k == test_skip_page ? kTestPolls
                                                                             : kMaxPolls));
    if (!ok) break;
    const int i = warp + k * kWarps;  // page within the chunk
    const int valid = min(kPage, n_tok - i * kPage);
    if constexpr (kAppend) {
      if (i == patch_page) {
        const int64_t src = (static_cast<int64_t>(b) * hkv + g) * kHeadDim;
        const int pid = page_ids[i];
        append_new_row(ring, s, (L - 1) % kPage, k_new + src, v_new + src, __ldg(v_scale + g),
                       k_cache, v_cache, pid >= 0 ? static_cast<int64_t>(pid) * hkv + g : -1);
      }
    }
    if (page_ids[i] >= 0) attend_page<kVF16>(ring, s, valid, qf, qs, st);
    __syncwarp();
    if (lane == 0 && k + kStages < n_my) {
      fence_proxy_async();
      issue(k + kStages);
    }
  }
  if (!ok) {
    // Give up on this chunk: report, then drain the copies still in flight
    // (bounded) so none lands after the CTA exits.  Pages k .. k+kStages-1
    // were issued (all but a withheld one); nothing later was.
    if (lane == 0) {
      flag_error(dev_error, K16V8_DEVERR_TIMEOUT);
      for (int kk = k; kk < min(k + kStages, n_my); ++kk)
        if (!(withheld && kk == test_skip_page))
          mbar_wait_bounded(&ring.bar[kk % kStages], (kk / kStages) & 1);
    }
    __syncwarp();
  }

  pdl_launch_dependents();

  st.finish();  // m, l of head hsel in every lane
  const float l_run = st.l;

  // ---- combine the four warps in shared memory (ring 0's K tiles) ----
  __syncthreads();
  float *wo = reinterpret_cast<float *>(rings[0].k);  // [warp][head][128]
  float *wm = wo + kWarps * kGroup * kHeadDim;        // [warp][head]
  float *wl = wm + kWarps * kGroup;
  if (lane < 8 && (lane & 1) == 0) {
    wm[warp * kGroup + hsel] = st.m;
    wl[warp * kGroup + hsel] = l_run;
  }
#pragma unroll
  for (int h = 0; h < kGroup; ++h)
    *reinterpret_cast<float4 *>(wo + (warp * kGroup + h) * kHeadDim + lane * 4) =
        make_float4(st.o[h][0].x, st.o[h][0].y, st.o[h][1].x, st.o[h][1].y);
  __syncthreads();
  {
    const int h = threadIdx.x >> 5;
    const int d4 = (threadIdx.x & 31) * 4;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * kGroup + h]);
    float Ls = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = wm[w * kGroup + h];
      const float sw = mw == -INFINITY ? 0.f : ex2(mw - M);
      Ls += sw * wl[w * kGroup + h];
      const float4 ow = *reinterpret_cast<const float4 *>(wo + (w * kGroup + h) * kHeadDim + d4);
      acc.x += sw * ow.x;
      acc.y += sw * ow.y;
      acc.z += sw * ow.z;
      acc.w += sw * ow.w;
    }
    const int64_t row = (static_cast<int64_t>(b) * hq + g * kGroup + h) * max_chunks + c;
    float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse = -INFINITY;
    if (Ls > 0.f) {
      const float inv = (kVF16 ? 1.f : __ldg(v_scale + g)) / Ls;
      res = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      lse = (M + lg2(Ls)) * kLn2;
    }
    if (out) {
      // one chunk: this is the final row (what the merge of a single partial
      // gives: the same values, rounded to fp16)
      const int64_t orow = static_cast<int64_t>(b) * hq + g * kGroup + h;
      uint2 o2;
      o2.x = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(res.x))) |
             (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(res.y))) << 16);
      o2.y = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(res.z))) |
             (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(res.w))) << 16);
      *reinterpret_cast<uint2 *>(out + orow * kHeadDim + d4) = o2;
      if ((threadIdx.x & 31) == 0 && lse_out) lse_out[orow] = lse;
    } else {
      *reinterpret_cast<float4 *>(part_o + row * kHeadDim + d4) = res;
      if ((threadIdx.x & 31) == 0) part_lse[row] = lse;
    }
  }
}

// One warp per (sequence, query head); lane owns 4 dims.  The live chunks'
// LSEs are loaded lane-parallel.  A row of up to kMergeOneRound chunks (a
// whole 8192-token sequence at the default 512-token chunk) has every
// partial row in flight in one round of loads; longer rows are read 4
// chunks at a time.  Either way the sums run in chunk order.
constexpr int kMergeOneRound = 16;
__global__ void __launch_bounds__(128, 5) merge_states_kernel(
    const float *__restrict__ part_o, const float *__restrict__ part_lse, int32_t rows,
    int32_t hq, int32_t max_chunks, const int32_t *__restrict__ seq_lens, int32_t chunk,
    __half *__restrict__ out, float *__restrict__ lse_out) {
  const int wid = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_launch_dependents();
  if (wid >= rows) return;
  const int b = wid / hq;
  int L = __ldg(seq_lens + b);
  L = max(0, min(L, max_chunks * chunk));
  const int nc = (L + chunk - 1) / chunk;
  const float *pl = part_lse + static_cast<int64_t>(wid) * max_chunks;
  const float *po = part_o + static_cast<int64_t>(wid) * max_chunks * kHeadDim + lane * 4;
  const float lc = lane < nc ? __ldg(pl + lane) : -INFINITY;  // LSE of chunk `lane`
  float M = lc;
  for (int c = lane + 32; c < nc; c += 32) M = fmaxf(M, __ldg(pl + c));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
  float S = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY && nc <= kMergeOneRound) {
    float4 oc[kMergeOneRound];
#pragma unroll
    for (int c = 0; c < kMergeOneRound; ++c)
      oc[c] = c < nc ? __ldg(reinterpret_cast<const float4 *>(po + static_cast<int64_t>(c) * kHeadDim))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < kMergeOneRound; ++c) {
      const float wl = __shfl_sync(kFull, lc, c);
      if (c < nc) {
        const float wu = ex2((wl - M) * kLog2e);
        S += wu;
        acc.x = fmaf(wu, oc[c].x, acc.x);
        acc.y = fmaf(wu, oc[c].y, acc.y);
        acc.z = fmaf(wu, oc[c].z, acc.z);
        acc.w = fmaf(wu, oc[c].w, acc.w);
      }
    }
  } else if (M != -INFINITY) {
    int c = 0;
    for (; c + 4 <= nc; c += 4) {
      float4 oc[4];
      float w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        oc[u] = __ldg(reinterpret_cast<const float4 *>(po + static_cast<int64_t>(c + u) * kHeadDim));
        w[u] = __ldg(pl + c + u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float wu = ex2((w[u] - M) * kLog2e);
        S += wu;
        acc.x = fmaf(wu, oc[u].x, acc.x);
        acc.y = fmaf(wu, oc[u].y, acc.y);
        acc.z = fmaf(wu, oc[u].z, acc.z);
        acc.w = fmaf(wu, oc[u].w, acc.w);
      }
    }
    for (; c < nc; ++c) {
      const float4 oc = __ldg(reinterpret_cast<const float4 *>(po + static_cast<int64_t>(c) * kHeadDim));
      const float wu = ex2((__ldg(pl + c) - M) * kLog2e);
      S += wu;
      acc.x = fmaf(wu, oc.x, acc.x);
      acc.y = fmaf(wu, oc.y, acc.y);
      acc.z = fmaf(wu, oc.z, acc.z);
      acc.w = fmaf(wu, oc.w, acc.w);
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

// ---- host side ------------------------------------------------------------

struct WsLayout {
  size_t o_off, lse_off, total;
  int chunks;
};

static inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

static bool ws_layout(int32_t batch, int32_t hq, int32_t d, int32_t max_seq_len, int32_t chunk,
                      WsLayout *w) {
  if (batch < 0 || hq <= 0 || d <= 0 || max_seq_len < 0 || chunk <= 0) return false;
  w->chunks = max(1, (max_seq_len + chunk - 1) / chunk);
  const size_t rows = static_cast<size_t>(batch) * hq * w->chunks;
  w->o_off = 0;
  w->lse_off = align256(rows * d * sizeof(float));
  w->total = w->lse_off + align256(rows * sizeof(float));
  return true;
}

template <bool kAppend, bool kVF16>
static int32_t set_smem_attr(size_t bytes) {
  // The attribute is per device; remember the largest size configured.
  static size_t configured[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return K16V8_ERR_CUDA;
  if (dev < 64 && configured[dev] >= bytes) return K16V8_OK;
  if (cudaFuncSetAttribute(decode_split_kernel<kAppend, kVF16>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes)) != cudaSuccess)
    return K16V8_ERR_CUDA;
  if (dev < 64) configured[dev] = bytes;
  return K16V8_OK;
}

static int32_t check_attention_shape(int32_t hq, int32_t hkv, int32_t head_dim) {
  if (hq <= 0 || hkv <= 0) return K16V8_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || hq != kGroup * hkv) return K16V8_ERR_UNSUPPORTED_SHAPE;
  return K16V8_OK;
}

}  // namespace k16v8

using namespace k16v8;

extern "C" size_t k16v8_decode_workspace_size(int32_t batch, int32_t num_qo_heads,
                                              int32_t head_dim, int32_t max_seq_len,
                                              int32_t split_chunk) {
  WsLayout w;
  if (split_chunk % kPage) return 0;
  if (!ws_layout(batch, num_qo_heads, head_dim, max_seq_len, split_chunk, &w)) return 0;
  return w.total;
}

extern "C" int32_t k16v8_decode_workspace_layout(int32_t batch, int32_t num_qo_heads,
                                                 int32_t head_dim, int32_t max_seq_len,
                                                 int32_t split_chunk, size_t *partial_o_offset,
                                                 size_t *partial_lse_offset,
                                                 int32_t *max_chunks) {
  WsLayout w;
  if (split_chunk % kPage || !ws_layout(batch, num_qo_heads, head_dim, max_seq_len, split_chunk, &w))
    return K16V8_ERR_INVALID_ARG;
  if (partial_o_offset) *partial_o_offset = w.o_off;
  if (partial_lse_offset) *partial_lse_offset = w.lse_off;
  if (max_chunks) *max_chunks = w.chunks;
  return K16V8_OK;
}

template <bool kAppend, bool kVF16 = false>
static int32_t launch_split(const void *q, const void *k_cache, const uint8_t *v_cache,
                            const float *v_scale, const int32_t *block_table,
                            int32_t max_pages_per_seq, const int32_t *seq_lens,
                            int32_t max_seq_len, int32_t batch, int32_t num_qo_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t num_pages,
                            float sm_scale, int32_t split_chunk, void *workspace,
                            size_t workspace_bytes, const void *k_new, const void *v_new,
                            int32_t *dev_error, void *stream, int32_t test_skip_page = -1,
                            void *out = nullptr, float *lse = nullptr) {
  int32_t st = check_attention_shape(num_qo_heads, num_kv_heads, head_dim);
  if (st != K16V8_OK) return st;
  if (batch < 0 || max_seq_len < 0 || num_pages <= 0 || max_pages_per_seq < 0)
    return K16V8_ERR_INVALID_ARG;
  if (split_chunk < kPage || split_chunk > K16V8_MAX_SPLIT_CHUNK || split_chunk % kPage)
    return K16V8_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_pages_per_seq) * kPage < max_seq_len) return K16V8_ERR_INVALID_ARG;
  if (batch > 65535 || num_kv_heads > 65535) return K16V8_ERR_INVALID_ARG;
  WsLayout w;
  if (!ws_layout(batch, num_qo_heads, head_dim, max_seq_len, split_chunk, &w))
    return K16V8_ERR_INVALID_ARG;
  if (batch == 0) return K16V8_OK;
  if (!q || !k_cache || !v_cache || (!kVF16 && !v_scale) || !block_table || !seq_lens ||
      !workspace)
    return K16V8_ERR_INVALID_ARG;
  if (kAppend && (!k_new || !v_new || !k16v8_aligned(k_new, 16) || !k16v8_aligned(v_new, 16)))
    return K16V8_ERR_INVALID_ARG;
  if (workspace_bytes < w.total) return K16V8_ERR_WORKSPACE_TOO_SMALL;
  if (!k16v8_aligned(q, 16) || !k16v8_aligned(k_cache, 16) || !k16v8_aligned(v_cache, 16) ||
      !k16v8_aligned(workspace, 256) || !k16v8_aligned(block_table, 4) ||
      !k16v8_aligned(seq_lens, 4) || !k16v8_aligned(v_scale, 4))
    return K16V8_ERR_INVALID_ARG;
  if (max_seq_len == 0) return K16V8_OK;  // every sequence empty: nothing to read
  if (w.chunks == 1 && out && (!k16v8_aligned(out, 8) || (lse && !k16v8_aligned(lse, 4))))
    return K16V8_ERR_INVALID_ARG;
  const size_t smem = decode_smem_bytes(split_chunk, kVF16);
  st = set_smem_attr<kAppend, kVF16>(smem);
  if (st != K16V8_OK) return st;
  float *po = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + w.o_off);
  float *pl = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + w.lse_off);
  const dim3 grid(w.chunks, num_kv_heads, batch);
  return k16v8_launch_pdl(
      decode_split_kernel<kAppend, kVF16>, grid, dim3(kWarps * 32), smem,
      static_cast<cudaStream_t>(stream), static_cast<const __half *>(q),
      static_cast<__half *>(const_cast<void *>(k_cache)), const_cast<uint8_t *>(v_cache), v_scale,
      block_table, max_pages_per_seq, seq_lens, num_qo_heads, num_kv_heads, num_pages, sm_scale,
      split_chunk, w.chunks, po, pl, static_cast<const __half *>(k_new),
      static_cast<const __half *>(v_new), dev_error, test_skip_page,
      w.chunks == 1 ? static_cast<__half *>(out) : nullptr, w.chunks == 1 ? lse : nullptr);
}

// A combined call whose lengths fit one chunk launches only the split
// kernel, which then writes the output rows itself (no partials, no merge).
static bool single_chunk(int32_t batch, int32_t hq, int32_t d, int32_t max_seq_len,
                         int32_t split_chunk) {
  WsLayout w;
  return batch > 0 && max_seq_len > 0 &&
         ws_layout(batch, hq, d, max_seq_len, split_chunk, &w) && w.chunks == 1;
}

extern "C" int32_t k16v8_paged_decode_split(
    const void *q, const void *k_cache, const uint8_t *v_cache, const float *v_scale,
    const int32_t *block_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
    int32_t max_seq_len, int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t num_pages, float sm_scale, int32_t split_chunk, void *workspace,
    size_t workspace_bytes, int32_t *dev_error, void *stream) {
  return launch_split<false>(q, k_cache, v_cache, v_scale, block_table, max_pages_per_seq,
                             seq_lens, max_seq_len, batch, num_qo_heads, num_kv_heads, head_dim,
                             num_pages, sm_scale, split_chunk, workspace, workspace_bytes, nullptr,
                             nullptr, dev_error, stream);
}

extern "C" int32_t k16v8_paged_decode_split_wait_test(
    const void *q, const void *k_cache, const uint8_t *v_cache, const float *v_scale,
    const int32_t *block_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
    int32_t max_seq_len, int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t num_pages, float sm_scale, int32_t split_chunk, void *workspace,
    size_t workspace_bytes, int32_t *dev_error, void *stream) {
  return launch_split<false>(q, k_cache, v_cache, v_scale, block_table, max_pages_per_seq,
                             seq_lens, max_seq_len, batch, num_qo_heads, num_kv_heads, head_dim,
                             num_pages, sm_scale, split_chunk, workspace, workspace_bytes, nullptr,
                             nullptr, dev_error, stream, /*test_skip_page=*/0);
}

extern "C" int32_t k16v8_paged_decode_append_split(
    const void *q, const void *k_new, const void *v_new, void *k_cache, uint8_t *v_cache,
    const float *v_scale, const int32_t *block_table, int32_t max_pages_per_seq,
    const int32_t *seq_lens, int32_t max_seq_len, int32_t batch, int32_t num_qo_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t num_pages, float sm_scale,
    int32_t split_chunk, void *workspace, size_t workspace_bytes, int32_t *dev_error,
    void *stream) {
  return launch_split<true>(q, k_cache, v_cache, v_scale, block_table, max_pages_per_seq,
                            seq_lens, max_seq_len, batch, num_qo_heads, num_kv_heads, head_dim,
                            num_pages, sm_scale, split_chunk, workspace, workspace_bytes, k_new,
                            v_new, dev_error, stream);
}

extern "C" int32_t k16v8_paged_decode_split_v16(
    const void *q, const void *k_cache, const void *v_cache16, const int32_t *block_table,
    int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t max_seq_len, int32_t batch,
    int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_pages,
    float sm_scale, int32_t split_chunk, void *workspace, size_t workspace_bytes,
    int32_t *dev_error, void *stream) {
  return launch_split<false, true>(
      q, k_cache, static_cast<const uint8_t *>(v_cache16), nullptr, block_table,
      max_pages_per_seq, seq_lens, max_seq_len, batch, num_qo_heads, num_kv_heads, head_dim,
      num_pages, sm_scale, split_chunk, workspace, workspace_bytes, nullptr, nullptr, dev_error,
      stream);
}

extern "C" int32_t k16v8_merge_states(const float *partial_o, const float *partial_lse,
                                      int32_t batch, int32_t num_qo_heads, int32_t max_chunks,
                                      int32_t head_dim, const int32_t *seq_lens,
                                      int32_t split_chunk, void *out, float *lse,
                                      void *stream) {
  if (batch < 0 || num_qo_heads <= 0 || max_chunks <= 0 || split_chunk <= 0)
    return K16V8_ERR_INVALID_ARG;
  if (head_dim != kHeadDim) return K16V8_ERR_UNSUPPORTED_SHAPE;
  if (batch == 0) return K16V8_OK;
  if (!partial_o || !partial_lse || !seq_lens || !out) return K16V8_ERR_INVALID_ARG;
  if (!k16v8_aligned(partial_o, 16) || !k16v8_aligned(out, 8) || !k16v8_aligned(partial_lse, 4) ||
      !k16v8_aligned(seq_lens, 4) || (lse && !k16v8_aligned(lse, 4)))
    return K16V8_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(batch) * num_qo_heads;
  if (rows > (1LL << 31) - 4) return K16V8_ERR_INVALID_ARG;
  const unsigned blocks = static_cast<unsigned>((rows + 3) / 4);
  return k16v8_launch_pdl(merge_states_kernel, dim3(blocks), dim3(128), 0,
                          static_cast<cudaStream_t>(stream), partial_o, partial_lse,
                          static_cast<int32_t>(rows), num_qo_heads, max_chunks, seq_lens,
                          split_chunk, static_cast<__half *>(out), lse);
}

extern "C" int32_t k16v8_paged_decode_attention(
    const void *q, const void *k_cache, const uint8_t *v_cache, const float *v_scale,
    const int32_t *block_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
    int32_t max_seq_len, int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t num_pages, float sm_scale, int32_t split_chunk, void *workspace,
    size_t workspace_bytes, void *out, float *lse, int32_t *dev_error, void *stream) {
  if (batch > 0 && !out) return K16V8_ERR_INVALID_ARG;
  if (single_chunk(batch, num_qo_heads, head_dim, max_seq_len, split_chunk))
    return launch_split<false>(q, k_cache, v_cache, v_scale, block_table, max_pages_per_seq,
                               seq_lens, max_seq_len, batch, num_qo_heads, num_kv_heads,
                               head_dim, num_pages, sm_scale, split_chunk, workspace,
                               workspace_bytes, nullptr, nullptr, dev_error, stream, -1, out,
                               lse);
  int32_t st = k16v8_paged_decode_split(q, k_cache, v_cache, v_scale, block_table,
                                        max_pages_per_seq, seq_lens, max_seq_len, batch,
                                        num_qo_heads, num_kv_heads, head_dim, num_pages, sm_scale,
                                        split_chunk, workspace, workspace_bytes, dev_error, stream);
  if (st != K16V8_OK || batch == 0) return st;
  WsLayout w;
  ws_layout(batch, num_qo_heads, head_dim, max_seq_len, split_chunk, &w);
  const uint8_t *base = static_cast<const uint8_t *>(workspace);
  return k16v8_merge_states(reinterpret_cast<const float *>(base + w.o_off),
                            reinterpret_cast<const float *>(base + w.lse_off), batch,
                            num_qo_heads, w.chunks, head_dim, seq_lens, split_chunk, out, lse,
                            stream);
}

extern "C" int32_t k16v8_paged_decode_append_attention(
    const void *q, const void *k_new, const void *v_new, void *k_cache, uint8_t *v_cache,
    const float *v_scale, const int32_t *block_table, int32_t max_pages_per_seq,
    const int32_t *seq_lens, int32_t max_seq_len, int32_t batch, int32_t num_qo_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t num_pages, float sm_scale,
    int32_t split_chunk, void *workspace, size_t workspace_bytes, void *out, float *lse,
    int32_t *dev_error, void *stream) {
  if (batch > 0 && !out) return K16V8_ERR_INVALID_ARG;
  if (single_chunk(batch, num_qo_heads, head_dim, max_seq_len, split_chunk))
    return launch_split<true>(q, k_cache, v_cache, v_scale, block_table, max_pages_per_seq,
                              seq_lens, max_seq_len, batch, num_qo_heads, num_kv_heads, head_dim,
                              num_pages, sm_scale, split_chunk, workspace, workspace_bytes, k_new,
                              v_new, dev_error, stream, -1, out, lse);
  int32_t st = k16v8_paged_decode_append_split(
      q, k_new, v_new, k_cache, v_cache, v_scale, block_table, max_pages_per_seq, seq_lens,
      max_seq_len, batch, num_qo_heads, num_kv_heads, head_dim, num_pages, sm_scale, split_chunk,
      workspace, workspace_bytes, dev_error, stream);
  if (st != K16V8_OK || batch == 0) return st;
  WsLayout w;
  ws_layout(batch, num_qo_heads, head_dim, max_seq_len, split_chunk, &w);
  const uint8_t *base = static_cast<const uint8_t *>(workspace);
  return k16v8_merge_states(reinterpret_cast<const float *>(base + w.o_off),
                            reinterpret_cast<const float *>(base + w.lse_off), batch,
                            num_qo_heads, w.chunks, head_dim, seq_lens, split_chunk, out, lse,
                            stream);
}

extern "C" int32_t k16v8_paged_decode_attention_v16(
    const void *q, const void *k_cache, const void *v_cache16, const int32_t *block_table,
    int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t max_seq_len, int32_t batch,
    int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_pages,
    float sm_scale, int32_t split_chunk, void *workspace, size_t workspace_bytes, void *out,
    float *lse, int32_t *dev_error, void *stream) {
  if (batch > 0 && !out) return K16V8_ERR_INVALID_ARG;
  if (single_chunk(batch, num_qo_heads, head_dim, max_seq_len, split_chunk))
    return launch_split<false, true>(
        q, k_cache, static_cast<const uint8_t *>(v_cache16), nullptr, block_table,
        max_pages_per_seq, seq_lens, max_seq_len, batch, num_qo_heads, num_kv_heads, head_dim,
        num_pages, sm_scale, split_chunk, workspace, workspace_bytes, nullptr, nullptr, dev_error,
        stream, -1, out, lse);
  int32_t st = k16v8_paged_decode_split_v16(q, k_cache, v_cache16, block_table,
                                            max_pages_per_seq, seq_lens, max_seq_len, batch,
                                            num_qo_heads, num_kv_heads, head_dim, num_pages,
                                            sm_scale, split_chunk, workspace, workspace_bytes,
                                            dev_error, stream);
  if (st != K16V8_OK || batch == 0) return st;
  WsLayout w;
  ws_layout(batch, num_qo_heads, head_dim, max_seq_len, split_chunk, &w);
  const uint8_t *base = static_cast<const uint8_t *>(workspace);
  return k16v8_merge_states(reinterpret_cast<const float *>(base + w.o_off),
                            reinterpret_cast<const float *>(base + w.lse_off), batch,
                            num_qo_heads, w.chunks, head_dim, seq_lens, split_chunk, out, lse,
                            stream);
}

// ---- no-allocation variant ---------------------------------------------------
//
// For callers that cannot allocate device memory: the split-KV partials live
// in this file-scope array instead of a caller workspace.  Host code must not
// pass the array's name to a kernel (in host code it names a host-side
// stand-in); it passes the device address looked up below.

static __device__ __align__(256) uint8_t g_static_scratch[K16V8_STATIC_SCRATCH_BYTES];

// Device address of g_static_scratch on the current device, looked up once
// per device (with that device current) and cached.
static int32_t static_scratch_address(void **ptr) {
  static void *cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return K16V8_ERR_CUDA;
  if (dev >= 0 && dev < 64 && cached[dev]) {
    *ptr = cached[dev];
    return K16V8_OK;
  }
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return K16V8_ERR_CUDA;
  if (dev >= 0 && dev < 64) cached[dev] = p;
  *ptr = p;
  return K16V8_OK;
}

extern "C" int32_t k16v8_paged_decode_attention_static(
    const void *q, const void *k_cache, const uint8_t *v_cache, const float *v_scale,
    const int32_t *block_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
    int32_t max_seq_len, int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t num_pages, float sm_scale, int32_t split_chunk, void *out,
    float *lse, int32_t *dev_error, void *stream) {
  const int32_t st0 = check_attention_shape(num_qo_heads, num_kv_heads, head_dim);
  if (st0 != K16V8_OK) return st0;
  // An empty batch needs no scratch: validate it exactly as the workspace
  // call does (which launches nothing for it).
  if (batch == 0)
    return k16v8_paged_decode_attention(q, k_cache, v_cache, v_scale, block_table,
                                        max_pages_per_seq, seq_lens, max_seq_len, batch,
                                        num_qo_heads, num_kv_heads, head_dim, num_pages,
                                        sm_scale, split_chunk, nullptr, 0, out, lse, dev_error,
                                        stream);
  const size_t need =
      k16v8_decode_workspace_size(batch, num_qo_heads, head_dim, max_seq_len, split_chunk);
  if (need == 0) return K16V8_ERR_INVALID_ARG;
  if (need > K16V8_STATIC_SCRATCH_BYTES) return K16V8_ERR_STATIC_SCRATCH_LIMIT;
  void *scratch = nullptr;
  const int32_t st = static_scratch_address(&scratch);
  if (st != K16V8_OK) return st;
  return k16v8_paged_decode_attention(q, k_cache, v_cache, v_scale, block_table,
                                      max_pages_per_seq, seq_lens, max_seq_len, batch,
                                      num_qo_heads, num_kv_heads, head_dim, num_pages, sm_scale,
                                      split_chunk, scratch, K16V8_STATIC_SCRATCH_BYTES, out, lse,
                                      dev_error, stream);
}
