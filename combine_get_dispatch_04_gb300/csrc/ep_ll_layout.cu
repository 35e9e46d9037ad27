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
// of slots, so one prefix over 128-token chunks gives every offset.
//
// Three launches, no global atomics:
//   1. rank   -- one warp per 128-token chunk (chunks never straddle two
//                source ranks) walks its slots in (token, k) order, 32 at a
//                time; __match_any_sync ranks equal experts within each step
//                and a per-expert counter in shared memory carries the rank
//                across steps.  It writes each slot's rank within the chunk
//                and the chunk's per-expert histogram.
//   2. scan   -- one warp per expert: exclusive prefix over chunks, the
//                per-source offsets and the per-expert count.
//   3. assign -- one thread per slot: e*cap + chunk offset + rank, with the
//                capacity check.
#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kChunk = 128;  // tokens per ranking warp

struct LLGeom {
  int64_t T, Tr;
  int K, E, R;
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
  g.ncps = (int)((g.Tr + kChunk - 1) / kChunk);
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
  const int64_t t0 = (int64_t)s * g.Tr + (int64_t)c * kChunk;
  const int64_t len = min((int64_t)kChunk, g.Tr - (int64_t)c * kChunk);
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
  for (int e = lane; e < g.E; e += 32) chunk_hist[(int64_t)ch * g.E + e] = cnt[e];
}

// One warp per expert: lanes own contiguous runs of chunks, a warp prefix
// over the runs, then each lane writes its chunks' offsets.
__global__ void __launch_bounds__(256)
    ll_scan_kernel(LLGeom g, const int32_t* __restrict__ chunk_hist, int32_t* __restrict__ chunk_off,
                   int32_t* __restrict__ ll_count, int32_t* __restrict__ ll_src_offset) {
  pdl_wait_then_release();
  const int lane = threadIdx.x & 31;
  const int e = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (e >= g.E) return;  // uniform per warp
  const int seg = (g.nchunks + 31) / 32;
  const int lo = min(g.nchunks, lane * seg), hi = min(g.nchunks, lo + seg);
  int sum = 0;
#pragma unroll 4
  for (int ch = lo; ch < hi; ++ch) sum += chunk_hist[(int64_t)ch * g.E + e];
  int incl = sum;
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - sum;
  for (int ch = lo; ch < hi; ++ch) {
    const int v = chunk_hist[(int64_t)ch * g.E + e];
    if (ch % g.ncps == 0 && ll_src_offset) ll_src_offset[(int64_t)e * g.R + ch / g.ncps] = run;
    chunk_off[(int64_t)ch * g.E + e] = run;
    run += v;
  }
  if (lane == 31 && ll_count) ll_count[e] = incl;
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
      const int ch = (int)(s * g.ncps + (t - s * g.Tr) / kChunk);
      const int e = (int)topk_idx[i];
      const int64_t pos = (int64_t)chunk_off[(int64_t)ch * g.E + e] + rank;
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

}  // namespace
}  // namespace ep

using namespace ep;

extern "C" size_t ep_ll_workspace_bytes(int64_t num_tokens, int num_ranks, int num_experts) {
  if (!routing_ok(num_tokens, 1, num_experts, num_ranks)) return 0;
  return ll_ws_bytes(make_ll_geom(num_tokens, 1, num_experts, num_ranks, 0));
}

extern "C" ep_status_t ep_ll_get_dispatch_layout(const int64_t* topk_idx, int64_t num_tokens,
                                                 int num_topk, int num_experts, int num_ranks,
                                                 int64_t expert_capacity, int32_t* ll_slot,
                                                 int32_t* ll_count, int32_t* ll_src_offset,
                                                 int32_t* err_word, void* workspace,
                                                 size_t workspace_bytes, ep_stream_t stream) {
  if (!routing_ok(num_tokens, num_topk, num_experts, num_ranks)) return EP_ERR_INVALID_ARG;
  if (expert_capacity < 0 || expert_capacity * (int64_t)num_experts >= (int64_t(1) << 31))
    return EP_ERR_INVALID_ARG;
  if (!ll_count) return EP_ERR_INVALID_ARG;
  if (num_tokens > 0 && (!topk_idx || !ll_slot || !workspace || !aligned16(workspace)))
    return EP_ERR_INVALID_ARG;
  const LLGeom g = make_ll_geom(num_tokens, num_topk, num_experts, num_ranks, expert_capacity);
  const size_t half = align_up(sizeof(int32_t) * (size_t)g.nchunks * g.E, 256);
  if (num_tokens > 0 && workspace_bytes < ll_ws_bytes(g)) return EP_ERR_CAPACITY;
  cudaStream_t st = to_cuda(stream);
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
