// ep_layout.cu -- get_dispatch_layout and slot assignment on one GPU.
//
// "[Not ready] MSCCLPP EP implementation" (mscclpp pull request 852),
// section "Scope", Intranode: get_dispatch_layout turns top-k routing into
// per-rank / per-expert token counts and the is_token_in_rank mask; the
// internode-combine commit fixes the receive order by receiver-side prefix
// sums over (source rank, token order).  With the R logical ranks' tokens
// laid out rank after rank in one call, that order is simply token order, so
// a token's row in destination r is
//     slot[t][r] = recv_base[r] + #{t' < t : token t' is sent to r}.
//
// Three launches, no atomics on global counters and no inter-block waits:
//   1. count  -- one thread per token: rank mask (a 64-bit set), the
//                is_token_in_rank row, and per-block partial counts per rank
//                (warp ballots) and per expert (warp-aggregated shared-memory
//                histogram).  Blocks never straddle two source ranks.
//   2. scan   -- one block: per-(source, rank) and per-(source, expert)
//                totals, recv_base, and the exclusive prefix of every block's
//                count per destination.
//   3. assign -- one thread per token: ballot-based prefix within the block
//                plus the block's prefix gives the slot.
#include <mutex>

#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kTok = 512;  // tokens (= threads) per block of the count/assign kernels
constexpr int kTokWarps = kTok / 32;

struct Geom {
  int64_t T, Tr;
  int K, E, El, R;
  int nbps;  // blocks per source rank
  int nb;    // total blocks = R * nbps
};

struct Workspace {
  uint64_t* masks;      // [T]
  int32_t* blk_rank;    // [R][nb]
  int32_t* blk_off;     // [R][nb]
  int32_t* blk_expert;  // [nb][E]
  size_t bytes;
};

Geom make_geom(int64_t T, int K, int E, int R) {
  Geom g;
  g.T = T;
  g.Tr = T / R;
  g.K = K;
  g.E = E;
  g.El = E / R;
  g.R = R;
  g.nbps = (int)((g.Tr + kTok - 1) / kTok);
  g.nb = R * g.nbps;
  return g;
}

Workspace carve(const Geom& g, void* base) {
  Workspace w;
  char* p = static_cast<char*>(base);
  size_t off = 0;
  w.masks = reinterpret_cast<uint64_t*>(p + off);
  off += align_up(sizeof(uint64_t) * (size_t)g.T, 256);
  w.blk_rank = reinterpret_cast<int32_t*>(p + off);
  off += align_up(sizeof(int32_t) * (size_t)g.R * g.nb, 256);
  w.blk_off = reinterpret_cast<int32_t*>(p + off);
  off += align_up(sizeof(int32_t) * (size_t)g.R * g.nb, 256);
  w.blk_expert = reinterpret_cast<int32_t*>(p + off);
  off += align_up(sizeof(int32_t) * (size_t)g.nb * g.E, 256);
  w.bytes = off;
  return w;
}

// Writes the R flags of one is_token_in_rank row (0/1 bytes).
__device__ __forceinline__ void write_member_row(uint8_t* row, uint64_t mask, int R) {
  if ((R & 3) == 0) {
    for (int r = 0; r < R; r += 4) {
      uint32_t w = (uint32_t)((mask >> r) & 1) | ((uint32_t)((mask >> (r + 1)) & 1) << 8) |
                   ((uint32_t)((mask >> (r + 2)) & 1) << 16) |
                   ((uint32_t)((mask >> (r + 3)) & 1) << 24);
      *reinterpret_cast<uint32_t*>(row + r) = w;
    }
  } else {
    for (int r = 0; r < R; ++r) row[r] = (uint8_t)((mask >> r) & 1);
  }
}

__global__ void __launch_bounds__(kTok)
    layout_count_kernel(const int64_t* __restrict__ topk_idx, Geom g,
                        uint8_t* __restrict__ is_token_in_rank, Workspace ws, int32_t* err) {
  pdl_wait_then_release();
  extern __shared__ int32_t smem[];
  int32_t* hist = smem;                // [E]
  int32_t* warp_cnt = smem + g.E;      // [kTokWarps][R]
  const int b = blockIdx.x;
  const int s = b / g.nbps, c = b % g.nbps;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t tl = (int64_t)c * kTok + threadIdx.x;
  const bool valid = tl < g.Tr;
  const int64_t t = (int64_t)s * g.Tr + tl;

  for (int i = threadIdx.x; i < g.E; i += kTok) hist[i] = 0;
  __syncthreads();

  uint64_t mask = 0;
  bool bad = false;
  const int64_t* row = topk_idx + t * g.K;
  for (int k0 = 0; k0 < g.K; k0 += 8) {
    int64_t ev[8];  // eight ids loaded before any is used
#pragma unroll
    for (int u = 0; u < 8; ++u) ev[u] = (valid && k0 + u < g.K) ? row[k0 + u] : -1;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (k0 + u >= g.K) break;  // uniform: every lane runs the same slots
      const int64_t e = ev[u];
      int key = -1;
      if (e != -1) {
        if (e < -1 || e >= g.E) {
          bad = true;
        } else {
          key = (int)e;
          mask |= 1ull << (key / g.El);
        }
      }
      // lanes naming the same expert add once, through their lowest lane
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, key);
      if (key >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[key], __popc(peers));
    }
  }
  if (valid) {
    ws.masks[t] = mask;
    write_member_row(is_token_in_rank + t * g.R, mask, g.R);
  }
  for (int r = 0; r < g.R; ++r) {
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, (mask >> r) & 1);
    if (lane == 0) warp_cnt[warp * g.R + r] = __popc(bal);
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && err) atomicOr(err, EP_ERRBIT_BAD_EXPERT);
  __syncthreads();
  for (int r = threadIdx.x; r < g.R; r += kTok) {
    int sum = 0;
    for (int w = 0; w < kTokWarps; ++w) sum += warp_cnt[w * g.R + r];
    ws.blk_rank[(int64_t)r * g.nb + b] = sum;
  }
  for (int e = threadIdx.x; e < g.E; e += kTok) ws.blk_expert[(int64_t)b * g.E + e] = hist[e];
}

constexpr int kScanThreads = 1024;

// Sum of n int32 values at p[0], p[stride], ...: eight independent partial
// sums so that the loads are issued back to back instead of one L2 round
// trip at a time.
__device__ __forceinline__ int strided_sum(const int32_t* p, int n, int64_t stride) {
  int s[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  int i = 0;
  for (; i + 8 <= n; i += 8) {
#pragma unroll
    for (int u = 0; u < 8; ++u) s[u] += p[(int64_t)(i + u) * stride];
  }
  for (; i < n; ++i) s[0] += p[(int64_t)i * stride];
  return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

__global__ void __launch_bounds__(kScanThreads)
    layout_scan_kernel(Geom g, Workspace ws, int32_t* __restrict__ ntpr,
                       int32_t* __restrict__ ntpe, int32_t* __restrict__ recv_base) {
  pdl_wait_then_release();
  __shared__ int32_t recv_count[EP_MAX_RANKS];
  __shared__ int32_t base[EP_MAX_RANKS + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = kScanThreads / 32;

  // tokens of source s sent to r: sum of the blocks of s
  for (int i = threadIdx.x; i < g.R * g.R; i += kScanThreads) {
    const int s = i / g.R, r = i % g.R;
    ntpr[i] = strided_sum(ws.blk_rank + (int64_t)r * g.nb + (int64_t)s * g.nbps, g.nbps, 1);
  }
  // slots of source s naming expert e
  for (int64_t i = threadIdx.x; i < (int64_t)g.R * g.E; i += kScanThreads) {
    const int s = (int)(i / g.E), e = (int)(i % g.E);
    ntpe[i] = strided_sum(ws.blk_expert + (int64_t)s * g.nbps * g.E + e, g.nbps, g.E);
  }
  // rows received by each destination: one warp per rank, lanes own
  // contiguous runs of blocks
  const int seg = (g.nb + 31) / 32;
  for (int r = warp; r < g.R; r += nwarps) {
    const int32_t* p = ws.blk_rank + (int64_t)r * g.nb;
    const int lo = min(g.nb, lane * seg), hi = min(g.nb, lo + seg);
    int sum = strided_sum(p + lo, hi - lo, 1);
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane == 0) recv_count[r] = sum;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    base[0] = 0;
    for (int r = 0; r < g.R; ++r) base[r + 1] = base[r] + recv_count[r];
  }
  __syncthreads();
  for (int i = threadIdx.x; i <= g.R; i += kScanThreads) recv_base[i] = base[i];
  // exclusive prefix of block counts within each destination, offset by recv_base
  for (int r = warp; r < g.R; r += nwarps) {
    const int32_t* p = ws.blk_rank + (int64_t)r * g.nb;
    int32_t* q = ws.blk_off + (int64_t)r * g.nb;
    const int lo = min(g.nb, lane * seg), hi = min(g.nb, lo + seg);
    const int sum = strided_sum(p + lo, hi - lo, 1);
    int incl = sum;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = base[r] + incl - sum;
    for (int b = lo; b < hi; ++b) {
      const int v = p[b];
      q[b] = run;
      run += v;
    }
  }
}

// Largest R * nb for which every assign block derives its own offsets from
// the per-block counts (otherwise a separate scan kernel computes them).
constexpr int kFoldMax = 8192;

// Slots of one block of tokens.  With fold == true this kernel also does the
// scan: each block sums the per-block rank counts itself (its prefix within
// each destination and the destinations' totals), and the blocks share out
// the per-source totals and recv_base.  Otherwise the block offsets come from
// layout_scan_kernel.
__global__ void __launch_bounds__(kTok)
    layout_assign_kernel(Geom g, Workspace ws, int32_t* __restrict__ slot, bool fold,
                         int32_t* __restrict__ ntpr, int32_t* __restrict__ ntpe,
                         int32_t* __restrict__ recv_base) {
  pdl_wait_then_release();
  __shared__ int32_t warp_off[kTokWarps][EP_MAX_RANKS];
  __shared__ int32_t blk_pre[EP_MAX_RANKS];
  __shared__ int32_t tot[EP_MAX_RANKS];
  __shared__ int32_t base[EP_MAX_RANKS + 1];
  const int b = blockIdx.x;
  const int s = b / g.nbps, c = b % g.nbps;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t tl = (int64_t)c * kTok + threadIdx.x;
  const bool valid = tl < g.Tr;
  const int64_t t = (int64_t)s * g.Tr + tl;
  const uint64_t mask = valid ? ws.masks[t] : 0;
  const unsigned lt = (1u << lane) - 1u;

  if (fold) {
    // per destination: the total over all blocks and the sum over blocks before b
    for (int r = warp; r < g.R; r += kTokWarps) {
      const int32_t* p = ws.blk_rank + (int64_t)r * g.nb;
      int all = 0, pre = 0;
#pragma unroll 4
      for (int bb = lane; bb < g.nb; bb += 32) {
        const int v = p[bb];
        all += v;
        pre += bb < b ? v : 0;
      }
      for (int o = 16; o > 0; o >>= 1) {
        all += __shfl_xor_sync(0xFFFFFFFFu, all, o);
        pre += __shfl_xor_sync(0xFFFFFFFFu, pre, o);
      }
      if (lane == 0) {
        tot[r] = all;
        blk_pre[r] = pre;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      base[0] = 0;
      for (int r = 0; r < g.R; ++r) base[r + 1] = base[r] + tot[r];
    }
    __syncthreads();
    // this block's share of the per-source totals and of recv_base
    const int64_t n_rank = (int64_t)g.R * g.R, n_exp = (int64_t)g.R * g.E;
    const int64_t n_out = n_rank + n_exp + g.R + 1;
    for (int64_t i = (int64_t)b * kTok + threadIdx.x; i < n_out; i += (int64_t)g.nb * kTok) {
      if (i < n_rank) {
        const int so = (int)(i / g.R), r = (int)(i % g.R);
        ntpr[i] = strided_sum(ws.blk_rank + (int64_t)r * g.nb + (int64_t)so * g.nbps, g.nbps, 1);
      } else if (i < n_rank + n_exp) {
        const int64_t k = i - n_rank;
        const int so = (int)(k / g.E), e = (int)(k % g.E);
        ntpe[k] = strided_sum(ws.blk_expert + (int64_t)so * g.nbps * g.E + e, g.nbps, g.E);
      } else {
        const int r = (int)(i - n_rank - n_exp);
        recv_base[r] = base[r];
      }
    }
  }

  for (int r = 0; r < g.R; ++r) {
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, (mask >> r) & 1);
    if (lane == 0) warp_off[warp][r] = __popc(bal);
  }
  __syncthreads();
  if (threadIdx.x < g.R) {
    const int r = threadIdx.x;
    int run = fold ? base[r] + blk_pre[r] : ws.blk_off[(int64_t)r * g.nb + b];
    for (int w = 0; w < kTokWarps; ++w) {
      const int v = warp_off[w][r];
      warp_off[w][r] = run;
      run += v;
    }
  }
  __syncthreads();
  int32_t* dst = slot + t * g.R;
  if ((g.R & 3) == 0) {
    for (int r = 0; r < g.R; r += 4) {
      int v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool in = (mask >> (r + i)) & 1;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, in);
        v[i] = in ? warp_off[warp][r + i] + __popc(bal & lt) : -1;
      }
      if (valid) *reinterpret_cast<int4*>(dst + r) = make_int4(v[0], v[1], v[2], v[3]);
    }
  } else {
    for (int r = 0; r < g.R; ++r) {
      const bool in = (mask >> r) & 1;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, in);
      if (valid) dst[r] = in ? warp_off[warp][r] + __popc(bal & lt) : -1;
    }
  }
}

// The layout's launches on one stream, given carved scratch.
void launch_layout(const int64_t* topk_idx, const Geom& g, const Workspace& ws,
                   int32_t* ntpr, int32_t* ntpe, uint8_t* is_token_in_rank, int32_t* slot,
                   int32_t* recv_base, int32_t* err_word, cudaStream_t st) {
  if (g.nb > 0) {
    const size_t smem = sizeof(int32_t) * ((size_t)g.E + (size_t)kTokWarps * g.R);
    launch_pdl(layout_count_kernel, g.nb, kTok, smem, st, topk_idx, g, is_token_in_rank, ws, err_word);
  }
  const bool fold = g.nb > 0 && (int64_t)g.R * g.nb <= kFoldMax;
  if (!fold) launch_pdl(layout_scan_kernel, 1, kScanThreads, 0, st, g, ws, ntpr, ntpe, recv_base);
  if (g.nb > 0)
    launch_pdl(layout_assign_kernel, g.nb, kTok, 0, st, g, ws, slot, fold, ntpr, ntpe, recv_base);
}

}  // namespace
}  // namespace ep

using namespace ep;

extern "C" size_t ep_workspace_bytes(int64_t num_tokens, int num_ranks, int num_experts) {
  if (!routing_ok(num_tokens, 1, num_experts, num_ranks)) return 0;
  const Geom g = make_geom(num_tokens, 1, num_experts, num_ranks);
  return carve(g, nullptr).bytes;
}

extern "C" ep_status_t ep_get_dispatch_layout(const int64_t* topk_idx, int64_t num_tokens,
                                              int num_topk, int num_experts, int num_ranks,
                                              int32_t* num_tokens_per_rank,
                                              int32_t* num_tokens_per_expert,
                                              uint8_t* is_token_in_rank, int32_t* slot,
                                              int32_t* recv_base, int32_t* err_word,
                                              void* workspace, size_t workspace_bytes,
                                              ep_stream_t stream) {
  if (!routing_ok(num_tokens, num_topk, num_experts, num_ranks)) return EP_ERR_INVALID_ARG;
  if (!num_tokens_per_rank || !num_tokens_per_expert || !recv_base) return EP_ERR_INVALID_ARG;
  if (num_tokens > 0) {
    if (!topk_idx || !is_token_in_rank || !slot || !workspace) return EP_ERR_INVALID_ARG;
    if (!aligned16(slot) || !aligned16(is_token_in_rank) || !aligned16(workspace) ||
        !aligned16(topk_idx))
      return EP_ERR_INVALID_ARG;
  }
  const Geom g = make_geom(num_tokens, num_topk, num_experts, num_ranks);
  const Workspace ws = carve(g, workspace);
  if (num_tokens > 0 && workspace_bytes < ws.bytes) return EP_ERR_CAPACITY;
  launch_layout(topk_idx, g, ws, num_tokens_per_rank, num_tokens_per_expert, is_token_in_rank,
                slot, recv_base, err_word, to_cuda(stream));
  return launch_status();
}

extern "C" ep_status_t ep_layout_total_rows(const int32_t* recv_base, int num_ranks,
                                            int32_t* host_total_rows, ep_stream_t stream) {
  if (!recv_base || !host_total_rows || num_ranks < 1 || num_ranks > EP_MAX_RANKS)
    return EP_ERR_INVALID_ARG;
  cudaStream_t st = to_cuda(stream);
  if (cudaMemcpyAsync(host_total_rows, recv_base + num_ranks, sizeof(int32_t),
                      cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return EP_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return EP_ERR_CUDA;
  return EP_OK;
}

// ---------------------------------------------------------------------------
// Layout without caller-provided scratch.
//
// For callers that cannot allocate device memory at call time: a plugin or
// custom-op host that hands the library only the tensors it already owns, a
// C caller with no device allocator of its own, or a serving loop whose
// memory budget is fixed at start-up (cudaMalloc can also stall every stream
// on the device while it runs).  The scratch lives in the file-scope array
// below, so every GPU that loads this library holds these bytes until the
// process exits.  All calls share the one array: calls that overlap on the
// GPU (two streams, or two host threads enqueueing at once) race on it.  It
// needs no clearing between calls: every scratch word a call reads was
// written earlier in that same call.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char ep_layout_noalloc_scratch[EP_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};  // device address of the array, per device id

// Device address of the scratch array on the current device, looked up once
// per device (the host-side name of the array is not a device address).
ep_status_t noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return EP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, ep_layout_noalloc_scratch) != cudaSuccess || p == nullptr)
      return EP_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return EP_OK;
}

}  // namespace

extern "C" ep_status_t ep_get_dispatch_layout_noalloc(
    const int64_t* topk_idx, int64_t num_tokens, int num_topk, int num_experts, int num_ranks,
    int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
    int32_t* slot, int32_t* recv_base, int32_t* err_word, ep_stream_t stream) {
  if (!routing_ok(num_tokens, num_topk, num_experts, num_ranks)) return EP_ERR_INVALID_ARG;
  if (!num_tokens_per_rank || !num_tokens_per_expert || !recv_base) return EP_ERR_INVALID_ARG;
  if (num_tokens > 0) {
    if (!topk_idx || !is_token_in_rank || !slot) return EP_ERR_INVALID_ARG;
    if (!aligned16(slot) || !aligned16(is_token_in_rank) || !aligned16(topk_idx))
      return EP_ERR_INVALID_ARG;
  }
  const Geom g = make_geom(num_tokens, num_topk, num_experts, num_ranks);
  if (carve(g, nullptr).bytes > (size_t)EP_NOALLOC_SCRATCH_BYTES) return EP_ERR_CAPACITY;
  void* scratch = nullptr;
  const ep_status_t s = noalloc_scratch(&scratch);
  if (s != EP_OK) return s;
  const Workspace ws = carve(g, scratch);
  launch_layout(topk_idx, g, ws, num_tokens_per_rank, num_tokens_per_expert, is_token_in_rank,
                slot, recv_base, err_word, to_cuda(stream));
  return launch_status();
}
