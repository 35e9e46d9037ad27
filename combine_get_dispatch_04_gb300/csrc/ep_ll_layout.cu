// ep_ll_layout.cu -- the low-latency (expert-major) receive layout.
//
// "[Not ready] MSCCLPP EP implementation" (mscclpp pull request 852), the
// low-latency port (dispatch<kUseFP8,...> / combine over per-expert buffers
// indexed [local_expert * num_ranks + dst_rank]).  Every unmasked top-k slot
// (t, k) gets its own row in the buffer of expert e = topk_idx[t][k]; expert
// e owns rows [e*cap, (e+1)*cap), packed by source rank, then token, then k:
//   ll_slot[t][k] = e*cap + (slots naming e from earlier sources)
//                   + (slots of src(t) before (t, k) naming e).
// With the R ranks' tokens laid out rank after rank, that is the global order
// of slots, so one prefix over chunks of 16..128 tokens gives every offset.
//
// Three launches, no global atomics:
//   1. rank   -- one warp per chunk of 16..128 tokens (chunks never straddle two
//                source ranks) walks its slots in (token, k) order, 32 at a
//                time; __match_any_sync ranks equal experts within each step
//                and a per-expert counter in shared memory carries the rank
//                across steps.  It writes each slot's rank within the chunk
//                and the chunk's per-expert histogram.
//   2. scan   -- one warp per expert: exclusive prefix over chunks (32 per
//                step, coalesced), the per-source offsets and the count.
//   3. assign -- one thread per slot: e*cap + chunk offset + rank, with the
//                capacity check.
#include "ep_common.cuh"

namespace ep {
namespace {

// Tokens per ranking warp: 128, halved (down to 16) while the batch would
// give fewer than kMinChunks warps, so that small batches still spread over
// the GPU.  Depends on (T, R) only, so the workspace size does too.
constexpr int kMaxChunk = 128;
constexpr int kMinChunk = 16;
constexpr int kMinChunks = 1024;

struct LLGeom {
  int64_t T, Tr;
  int K, E, R;
  int chunk;    // tokens per chunk
  int ncps;     // chunks per source rank
  int nchunks;  // R * ncps
  int64_t cap;  // rows per expert
};

LLGeom make_ll_geom(int64_t T, int K, int E, int R, int64_t cap) {
  LLGeom g;
  g.T = T;
  g.Tr = T / R;
  g.K = K;
  g.E = E;
  g.R = R;
  g.chunk = kMaxChunk;
  while (g.chunk > kMinChunk && (int64_t)R * ((g.Tr + g.chunk - 1) / g.chunk) < kMinChunks)
    g.chunk /= 2;
  g.ncps = (int)((g.Tr + g.chunk - 1) / g.chunk);
  g.nchunks = R * g.ncps;
  g.cap = cap;
  return g;
}

size_t ll_ws_bytes(const LLGeom& g) { return 2 * align_up(sizeof(int32_t) * (size_t)g.nchunks * g.E, 256); }

__global__ void __launch_bounds__(32)
    ll_rank_kernel(const int64_t* __restrict__ topk_idx, LLGeom g, int32_t* __restrict__ ll_slot,
                   int32_t* __restrict__ chunk_hist, int32_t* err) {
  pdl_wait_then_release();
  extern __shared__ int32_t cnt[];  // [E]
  const int lane = threadIdx.x;
  const int ch = blockIdx.x;
  const int s = ch / g.ncps, c = ch % g.ncps;
  const int64_t t0 = (int64_t)s * g.Tr + (int64_t)c * g.chunk;
  const int64_t len = min((int64_t)g.chunk, g.Tr - (int64_t)c * g.chunk);
  const int64_t nslots = len * g.K;
  const unsigned lt = (1u << lane) - 1u;
  for (int e = lane; e < g.E; e += 32) cnt[e] = 0;
  __syncwarp();
  bool bad = false;
  const int64_t* base = topk_idx + t0 * g.K;  // the chunk's slots are contiguous
  int32_t* out = ll_slot + t0 * g.K;
  for (int64_t j00 = 0; j00 < nslots; j00 += 32 * 8) {
    int64_t ev[8];  // eight steps of ids loaded before any is used
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t j = j00 + u * 32 + lane;
      ev[u] = j < nslots ? base[j] : -1;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t j0 = j00 + u * 32;
      if (j0 >= nslots) break;  // uniform
      const int64_t j = j0 + lane;
      const int64_t e = ev[u];
      int key = -1;
      if (e >= 0 && e < g.E)
        key = (int)e;
      else if (j < nslots && e != -1)
        bad = true;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, key);
      const int before = key >= 0 ? cnt[key] : 0;
      __syncwarp();
      if (key >= 0 && lane == __ffs(peers) - 1) cnt[key] = before + __popc(peers);
      __syncwarp();
      if (j < nslots) out[j] = key >= 0 ? before + __popc(peers & lt) : -1;
    }
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && err) atomicOr(err, EP_ERRBIT_BAD_EXPERT);
  // expert-major [E][nchunks], so that the scan reads each expert's chunks
  // with coalesced loads
  for (int e = lane; e < g.E; e += 32) chunk_hist[(int64_t)e * g.nchunks + ch] = cnt[e];
}

// One warp per expert: its chunks 32 at a time (one coalesced load per
// lane, the next group loaded ahead), a warp scan per group and a running
// total carried across groups.
__global__ void __launch_bounds__(256)
    ll_scan_kernel(LLGeom g, const int32_t* __restrict__ chunk_hist, int32_t* __restrict__ chunk_off,
                   int32_t* __restrict__ ll_count, int32_t* __restrict__ ll_src_offset) {
  pdl_wait_then_release();
  const int lane = threadIdx.x & 31;
  const int e = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (e >= g.E) return;  // uniform per warp
  const int32_t* h = chunk_hist + (int64_t)e * g.nchunks;
  int32_t* off = chunk_off + (int64_t)e * g.nchunks;
  int run = 0;
  int v = lane < g.nchunks ? h[lane] : 0;
  for (int c0 = 0; c0 < g.nchunks; c0 += 32) {
    const int ch = c0 + lane;
    const int nxt = ch + 32 < g.nchunks ? h[ch + 32] : 0;
    int incl = v;
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += u;
    }
    const int excl = run + incl - v;
    if (ch < g.nchunks) {
      off[ch] = excl;
      if (ll_src_offset && ch % g.ncps == 0) ll_src_offset[(int64_t)e * g.R + ch / g.ncps] = excl;
    }
    run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    v = nxt;
  }
  if (lane == 0 && ll_count) ll_count[e] = run;
}

__global__ void __launch_bounds__(256)
    ll_assign_kernel(const int64_t* __restrict__ topk_idx, LLGeom g,
                     const int32_t* __restrict__ chunk_off, int32_t* __restrict__ ll_slot,
                     int32_t* err) {
  pdl_wait_then_release();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  bool over = false;
  if (i < g.T * g.K) {
    const int32_t rank = ll_slot[i];
    if (rank >= 0) {
      const int64_t t = i / g.K;
      const int64_t s = t / g.Tr;
      const int ch = (int)(s * g.ncps + (t - s * g.Tr) / g.chunk);
      const int e = (int)topk_idx[i];
      const int64_t pos = (int64_t)chunk_off[(int64_t)e * g.nchunks + ch] + rank;
      if (pos < g.cap) {
        ll_slot[i] = (int32_t)(e * g.cap + pos);
      } else {
        ll_slot[i] = -1;
        over = true;
      }
    }
  }
  if (__any_sync(0xFFFFFFFFu, over) && (threadIdx.x & 31) == 0 && err)
    atomicOr(err, EP_ERRBIT_CAPACITY);
}

// ---------------------------------------------------------------------------
// Single-launch form for small batches (decode-size inputs).
//
// One thread-block cluster of 16 CTAs (8 where the device does not schedule
// 16) x 8 warps computes the whole layout in one launch with no scratch
// memory.  The warps, in cluster order, own consecutive runs of G tokens of
// one source rank each (wps warps per source), so warp order is slot order.
//   - Each warp walks its slots in (token, k) order, 32 at a time, ranking
//     equal experts with __match_any_sync and a per-warp counter per expert
//     in shared memory; it keeps every slot's (expert, rank) in shared memory.
//   - Per expert, an exclusive prefix over the CTA's warps gives each warp's
//     first rank and the CTA's total.  After a cluster barrier each CTA reads
//     the totals of the CTAs before it over distributed shared memory, which
//     gives its first row in every expert (and, in CTA 0, ll_count).
//   - Each slot's row is then e*cap + (CTAs before) + (warps before) + rank,
//     with the capacity check; the CTA holding a source's first warp writes
//     that source's ll_src_offset column.  A second cluster barrier, waited
//     on only at exit, keeps shared memory alive while other CTAs read it.
// The loops over slots are not unrolled beyond one batch of eight steps: the
// kernel runs once per launch with a cold instruction cache.
// ---------------------------------------------------------------------------
constexpr int kLThreads = 256;
constexpr int kLWarps = kLThreads / 32;
constexpr int kLMaxExperts = 1024;    // per-warp counters for every expert in shared memory
constexpr int kLMaxWarpSlots = 2048;  // slots one warp walks
constexpr size_t kLMaxSmem =
    sizeof(int32_t) * ((size_t)kLWarps * kLMaxExperts + 2 * kLMaxExperts +
                       (size_t)kLWarps * kLMaxWarpSlots);

struct LLShape {
  int ctas;  // CTAs of the one cluster (= the grid)
  int wps;   // warps per source rank
  int G;     // tokens per warp
};

// The split of the batch over a cluster of at most max_ctas CTAs; false if
// the single-launch form does not take this batch.
bool ll_shape(const LLGeom& g, int max_ctas, LLShape* out) {
  if (g.T <= 0 || g.E > kLMaxExperts) return false;
  const int W = max_ctas * kLWarps;
  if (W < g.R) return false;
  const int wps = W / g.R;
  const int64_t G = (g.Tr + wps - 1) / wps;
  if (G * g.K > kLMaxWarpSlots) return false;
  const int used = (int)((g.Tr + G - 1) / G);  // warps of a source that hold tokens
  out->wps = wps;
  out->G = (int)G;
  out->ctas = ((g.R - 1) * wps + used - 1) / kLWarps + 1;
  return true;
}

// Fits with 8 CTAs, hence also with 16.
bool ll_single_fits(const LLGeom& g) {
  LLShape sh;
  return ll_shape(g, 8, &sh);
}

size_t ll_cluster_smem_bytes(const LLGeom& g, const LLShape& sh) {
  return sizeof(int32_t) *
         ((size_t)kLWarps * g.E + 2 * (size_t)g.E + (size_t)kLWarps * sh.G * g.K);
}

// EP_LAYOUT_AUTO takes the single launch whenever it fits.  Measured on
// GB300 inside the step (layout -> dispatch -> combine), single against
// multi-launch: 512 tokens 9.1 / 14.1 us; decode FP8 (4096 tokens, 32 ranks,
// 256 experts, top-8) 13.8 / 20.8 us; 8 ranks x 1024 tokens, 256 experts,
// top-8: 19.6 / 25.4 us; 8 ranks x 2048 tokens (each warp at its 2048-slot
// limit with 8 CTAs): 25.8 / 26.9 us.

__global__ void __launch_bounds__(kLThreads, 1)
    ll_cluster_kernel(const int64_t* __restrict__ topk_idx, LLGeom g, int wps, int G,
                      int32_t* __restrict__ ll_slot, int32_t* __restrict__ ll_count,
                      int32_t* __restrict__ ll_src_offset, int32_t* err) {
  pdl_wait_then_release();
  extern __shared__ int32_t smem[];
  const int E = g.E, K = g.K, R = g.R;
  const int Tr = (int)g.Tr;
  const int ws = G * K;                  // slots per warp
  int32_t* wcnt = smem;                  // [kLWarps][E] per-warp counts, then first ranks
  int32_t* tot = wcnt + kLWarps * E;     // [E] this CTA's slots per expert
  int32_t* pre = tot + E;                // [E] slots per expert in the CTAs before this one
  int32_t* er = pre + E;                 // [kLWarps][ws] expert << 16 | rank, -1 = no row
  const int c = (int)cluster_cta_rank();
  const int nc = (int)gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const int gw = c * kLWarps + warp;
  const int s = gw / wps, i = gw % wps;
  int n = 0;        // slots of this warp
  int64_t j0 = 0;   // its first slot
  if (s < R && i * G < Tr) {
    const int a = i * G, b = min(Tr, a + G);
    n = (b - a) * K;
    j0 = ((int64_t)s * Tr + a) * K;
  }
  // the warp's first eight steps of ids, loaded before the zeroing below so
  // that their memory latency overlaps it
  int64_t ev0[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int j = u * 32 + lane;
    ev0[u] = j < n ? topk_idx[j0 + j] : -1;
  }
  for (int x = tid; x < kLWarps * E; x += kLThreads) wcnt[x] = 0;
  __syncthreads();

  // --- ranks within the warp ---
  int32_t* cnt = wcnt + warp * E;
  int32_t* my = er + warp * ws;
  const int64_t* ids = topk_idx + j0;
  bool bad = false;
#pragma unroll 1
  for (int j00 = 0; j00 < n; j00 += 32 * 8) {
    int64_t ev[8];  // eight steps of ids loaded before any is used
    if (j00 == 0) {
#pragma unroll
      for (int u = 0; u < 8; ++u) ev[u] = ev0[u];
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j00 + u * 32 + lane;
        ev[u] = j < n ? ids[j] : -1;
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (j00 + u * 32 >= n) break;  // uniform
      const int j = j00 + u * 32 + lane;
      const int64_t e = ev[u];
      int key = -1;
      if (e >= 0 && e < E)
        key = (int)e;
      else if (j < n && e != -1)
        bad = true;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, key);
      const int before = key >= 0 ? cnt[key] : 0;
      __syncwarp();
      if (key >= 0 && lane == __ffs(peers) - 1) cnt[key] = before + __popc(peers);
      __syncwarp();
      if (j < n) my[j] = key >= 0 ? (key << 16) | (before + __popc(peers & lt)) : -1;
    }
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && err) atomicOr(err, EP_ERRBIT_BAD_EXPERT);
  __syncthreads();

  // --- per expert: first rank of each warp, and this CTA's total ---
  for (int e = tid; e < E; e += kLThreads) {
    int acc = 0;
#pragma unroll
    for (int w = 0; w < kLWarps; ++w) {
      const int v = wcnt[w * E + e];
      wcnt[w * E + e] = acc;
      acc += v;
    }
    tot[e] = acc;
  }
  cluster_arrive();
  cluster_wait();  // every CTA's totals are final and visible to the cluster

  // --- rows per expert taken by the CTAs before this one, and ll_count ---
  for (int e = tid; e < E; e += kLThreads) {
    const uint32_t a = smem_addr(tot + e);
    int p = 0, all = 0;
#pragma unroll 4
    for (int cc = 0; cc < nc; ++cc) {
      uint32_t ra;
      asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(cc));
      const int v = dsmem_ld(ra);
      all += v;
      p += cc < c ? v : 0;
    }
    pre[e] = p;
    if (c == 0) ll_count[e] = all;
  }
  cluster_arrive();  // this CTA no longer reads the other CTAs' shared memory
  __syncthreads();   // pre[] is written

  // --- ll_src_offset columns of the sources whose first warp is in this CTA ---
  if (ll_src_offset) {
    const int s_beg = (c * kLWarps + wps - 1) / wps;
    const int s_end = min(R, ((c + 1) * kLWarps + wps - 1) / wps);
    for (int s2 = s_beg; s2 < s_end; ++s2) {
      const int w = s2 * wps - c * kLWarps;
      for (int e = tid; e < E; e += kLThreads)
        ll_src_offset[(int64_t)e * R + s2] = pre[e] + wcnt[w * E + e];
    }
  }

  // --- rows ---
  bool over = false;
  const int32_t* first = wcnt + warp * E;
  for (int j = lane; j < n; j += 32) {
    const int v = my[j];
    int32_t row = -1;
    if (v >= 0) {
      const int e = v >> 16;
      const int64_t pos = (int64_t)pre[e] + first[e] + (v & 0xFFFF);
      if (pos < g.cap)
        row = (int32_t)(e * g.cap + pos);
      else
        over = true;
    }
    ll_slot[j0 + j] = row;
  }
  if (__any_sync(0xFFFFFFFFu, over) && lane == 0 && err) atomicOr(err, EP_ERRBIT_CAPACITY);
  cluster_wait();  // the other CTAs have finished reading this CTA's shared memory
}

ClusterSizeCache g_ll_cluster_size;  // 16 or 8 CTAs, per device

cudaError_t launch_ll_cluster(const int64_t* topk_idx, const LLGeom& g, int32_t* ll_slot,
                              int32_t* ll_count, int32_t* ll_src_offset, int32_t* err_word,
                              cudaStream_t st) {
  int max_ctas = 8;
  const cudaError_t e = g_ll_cluster_size.get(ll_cluster_kernel, kLThreads, kLMaxSmem, &max_ctas);
  if (e != cudaSuccess) return e;
  LLShape sh;
  if (!ll_shape(g, max_ctas, &sh) && !ll_shape(g, max_ctas = 8, &sh)) return cudaErrorInvalidValue;
  return launch_pdl_cluster(ll_cluster_kernel, sh.ctas, kLThreads, ll_cluster_smem_bytes(g, sh),
                            sh.ctas, st, topk_idx, g, sh.wps, sh.G, ll_slot, ll_count,
                            ll_src_offset, err_word);
}

}  // namespace
}  // namespace ep

using namespace ep;

extern "C" size_t ep_ll_workspace_bytes(int64_t num_tokens, int num_ranks, int num_experts) {
  if (!routing_ok(num_tokens, 1, num_experts, num_ranks)) return 0;
  return ll_ws_bytes(make_ll_geom(num_tokens, 1, num_experts, num_ranks, 0));
}

extern "C" int ep_ll_layout_single_launch_fits(int64_t num_tokens, int num_topk, int num_ranks,
                                               int num_experts) {
  if (!routing_ok(num_tokens, num_topk, num_experts, num_ranks)) return 0;
  return ll_single_fits(make_ll_geom(num_tokens, num_topk, num_experts, num_ranks, 0)) ? 1 : 0;
}

extern "C" int ep_ll_layout_auto_single_launch(int64_t num_tokens, int num_topk, int num_ranks,
                                               int num_experts) {
  return ep_ll_layout_single_launch_fits(num_tokens, num_topk, num_ranks, num_experts);
}

extern "C" ep_status_t ep_ll_get_dispatch_layout_path(
    const int64_t* topk_idx, int64_t num_tokens, int num_topk, int num_experts, int num_ranks,
    int64_t expert_capacity, int32_t* ll_slot, int32_t* ll_count, int32_t* ll_src_offset,
    int32_t* err_word, void* workspace, size_t workspace_bytes, int path, ep_stream_t stream) {
  if (!routing_ok(num_tokens, num_topk, num_experts, num_ranks)) return EP_ERR_INVALID_ARG;
  if (expert_capacity < 0 || expert_capacity * (int64_t)num_experts >= (int64_t(1) << 31))
    return EP_ERR_INVALID_ARG;
  if (!ll_count) return EP_ERR_INVALID_ARG;
  if (path != EP_LAYOUT_AUTO && path != EP_LAYOUT_MULTI_LAUNCH && path != EP_LAYOUT_SINGLE_LAUNCH)
    return EP_ERR_INVALID_ARG;
  const LLGeom g = make_ll_geom(num_tokens, num_topk, num_experts, num_ranks, expert_capacity);
  const bool fits = ll_single_fits(g);
  if (path == EP_LAYOUT_SINGLE_LAUNCH && !fits) return EP_ERR_INVALID_ARG;
  const bool single = path == EP_LAYOUT_SINGLE_LAUNCH || (path == EP_LAYOUT_AUTO && fits);
  if (num_tokens > 0 && (!topk_idx || !ll_slot)) return EP_ERR_INVALID_ARG;
  if (num_tokens > 0 && !single && (!workspace || !aligned16(workspace))) return EP_ERR_INVALID_ARG;
  cudaStream_t st = to_cuda(stream);
  if (single) {
    if (launch_ll_cluster(topk_idx, g, ll_slot, ll_count, ll_src_offset, err_word, st) ==
        cudaSuccess)
      return EP_OK;
    cudaGetLastError();  // clear the launch error
    // EP_LAYOUT_AUTO runs the three-launch form instead when the device
    // refused the cluster and the caller passed a usable workspace.
    if (path != EP_LAYOUT_AUTO || !workspace || !aligned16(workspace) ||
        workspace_bytes < ll_ws_bytes(g))
      return EP_ERR_CUDA;
  }
  const size_t half = align_up(sizeof(int32_t) * (size_t)g.nchunks * g.E, 256);
  if (num_tokens > 0 && workspace_bytes < ll_ws_bytes(g)) return EP_ERR_CAPACITY;
  if (num_tokens == 0) {
    // no chunks: counts and offsets are zero
    if (cudaMemsetAsync(ll_count, 0, sizeof(int32_t) * num_experts, st) != cudaSuccess)
      return EP_ERR_CUDA;
    if (ll_src_offset &&
        cudaMemsetAsync(ll_src_offset, 0, sizeof(int32_t) * (size_t)num_experts * num_ranks, st) !=
            cudaSuccess)
      return EP_ERR_CUDA;
    return EP_OK;
  }
  int32_t* hist = static_cast<int32_t*>(workspace);
  int32_t* off = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + half);
  launch_pdl(ll_rank_kernel, g.nchunks, 32, sizeof(int32_t) * g.E, st, topk_idx, g, ll_slot, hist,
             err_word);
  launch_pdl(ll_scan_kernel, (g.E * 32 + 255) / 256, 256, 0, st, g, hist, off, ll_count,
             ll_src_offset);
  const int64_t n = g.T * g.K;
  launch_pdl(ll_assign_kernel, (unsigned)((n + 255) / 256), 256, 0, st, topk_idx, g, off, ll_slot,
             err_word);
  return launch_status();
}

extern "C" ep_status_t ep_ll_get_dispatch_layout(const int64_t* topk_idx, int64_t num_tokens,
                                                 int num_topk, int num_experts, int num_ranks,
                                                 int64_t expert_capacity, int32_t* ll_slot,
                                                 int32_t* ll_count, int32_t* ll_src_offset,
                                                 int32_t* err_word, void* workspace,
                                                 size_t workspace_bytes, ep_stream_t stream) {
  return ep_ll_get_dispatch_layout_path(topk_idx, num_tokens, num_topk, num_experts, num_ranks,
                                        expert_capacity, ll_slot, ll_count, ll_src_offset,
                                        err_word, workspace, workspace_bytes, EP_LAYOUT_AUTO,
                                        stream);
}
