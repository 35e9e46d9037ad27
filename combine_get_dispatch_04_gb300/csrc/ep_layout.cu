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
// Two forms with identical outputs.  The multi-launch form has no atomics on
// global counters and no inter-block waits:
//   1. count  -- one thread per token: rank mask (a 64-bit set), the
//                is_token_in_rank row, and per-block partial counts per rank
//                (warp ballots) and per expert (warp-aggregated shared-memory
//                histogram).  Blocks never straddle two source ranks.
//   2. scan   -- one block: per-(source, rank) and per-(source, expert)
//                totals, recv_base, and the exclusive prefix of every block's
//                count per destination.  Folded into assign when the per-block
//                counts are few enough for every block to sum them itself.
//   3. assign -- one thread per token: ballot-based prefix within the block
//                plus the block's prefix gives the slot.
// The single-launch form (small batches, further below) does all of it in
// one thread-block cluster whose CTAs exchange counts through distributed
// shared memory.
#include <mutex>

#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kTok = 512;  // tokens (= threads) per block of the count/assign kernels
constexpr int kTokWarps = kTok / 32;

struct Geom {
  int64_t T, Tr;
  int K, E, El, R;
  int S;     // source ranks: R for one call over every rank's tokens, 1 for one shard's
  int nbps;  // blocks per source rank
  int nb;    // total blocks = S * nbps
};

struct Workspace {
  uint64_t* masks;      // [T]
  int32_t* blk_rank;    // [R][nb]
  int32_t* blk_off;     // [R][nb]
  int32_t* blk_expert;  // [nb][E]
  size_t bytes;
};

Geom make_geom(int64_t T, int K, int E, int R, int S) {
  Geom g;
  g.T = T;
  g.S = S;
  g.Tr = T / S;
  g.K = K;
  g.E = E;
  g.El = E / R;
  g.R = R;
  g.nbps = (int)((g.Tr + kTok - 1) / kTok);
  g.nb = S * g.nbps;
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
      // bits r..r+3 spread to the low bit of four bytes: x * 0x00204081 puts
      // copies of x at bit offsets 0, 7, 14 and 21
      const uint32_t x = (uint32_t)(mask >> r) & 0xFu;
      *reinterpret_cast<uint32_t*>(row + r) = (x * 0x00204081u) & 0x01010101u;
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
  for (int i = threadIdx.x; i < g.S * g.R; i += kScanThreads) {
    const int s = i / g.R, r = i % g.R;
    ntpr[i] = strided_sum(ws.blk_rank + (int64_t)r * g.nb + (int64_t)s * g.nbps, g.nbps, 1);
  }
  // slots of source s naming expert e
  for (int64_t i = threadIdx.x; i < (int64_t)g.S * g.E; i += kScanThreads) {
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
    const int64_t n_rank = (int64_t)g.S * g.R, n_exp = (int64_t)g.S * g.E;
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

// ---------------------------------------------------------------------------
// Single-launch layout for small batches (decode-size inputs).
//
// At these sizes the launches above are bound by latency (each warp's chain
// of dependent instructions, and the round trips between kernels), not by
// bytes.  Here one thread-block cluster does the whole layout in one launch,
// with no scratch memory:
//   - CTA c of the cluster owns tokens [c*Tc, (c+1)*Tc), Tc = chunks*256,
//     one token per thread and chunk.  It keeps its tokens' rank masks and
//     its warps' destination ballots, and counts into its own shared memory:
//     slots per (source, expert) and tokens per (source, destination).
//     The chunk loops are not unrolled: the kernel runs once per launch with
//     a cold instruction cache, so its code size is part of its latency.
//   - After one cluster barrier every CTA reads the others' counts through
//     distributed shared memory: the destination totals of the CTAs before
//     it give its first row in every destination, and the CTA in which a
//     source rank's tokens start sums that source's rows of
//     num_tokens_per_rank and num_tokens_per_expert.
//   - Slots then follow from the stored ballots: one prefix over the CTA's
//     groups of 32 tokens, then one pass over the CTA's slot rows (a
//     contiguous run of the matrix) in which consecutive threads write
//     consecutive 16-byte pieces.  A second cluster barrier, waited on only
//     at the end, keeps every CTA's shared memory alive until the other CTAs
//     have read it.
//   - Each thread's first eight ids are loaded before the shared counters
//     are zeroed, and a warp whose 32 tokens share one source adds its
//     per-destination counts from its ballots (one add per destination, not
//     one per token).  Measured at 4096 tokens (32 ranks, 256 experts,
//     top-8) with %globaltimer stamps inside layout -> dispatch -> combine
//     steps: the body from 7.8 to 7.1 us, the step from 133.8 to 133.3 us
//     (alternating A/B runs, three each).
// ---------------------------------------------------------------------------
constexpr int kCThreads = 256;  // tokens per CTA and chunk
constexpr int kCWarps = kCThreads / 32;
constexpr int kCMaxCtas = 16;   // cluster size (above 8 where the device allows it)
constexpr int kCMaxChunks = 8;  // chunks per CTA
constexpr int kCMaxTokens = 8 * kCMaxChunks * kCThreads;  // what a cluster of 8 CTAs takes
constexpr int kCMaxHist = 16384;  // R * E counters of the per-(source, expert) histogram

bool single_launch_fits(int64_t T, int R, int E) {
  return T > 0 && T <= kCMaxTokens && (int64_t)R * E <= kCMaxHist;
}

// Largest batch for which EP_LAYOUT_AUTO takes the single launch.  Measured
// on GB300 (inside the layout -> dispatch -> combine step): 14.1 us against
// 17.8 us for the multi-launch form at 4096 tokens (32 ranks, 256 experts,
// top-8); 22.0 us against 18.8 us at 16384 tokens (8 ranks, 256 experts,
// top-8), where one cluster's 16 SMs have too many tokens each.
constexpr int kCAutoMaxTokens = 8192;

struct ClusterShape {
  int ctas;    // CTAs of the one cluster (= the grid)
  int chunks;  // 256-token chunks per CTA
};

// As many CTAs as the tokens fill (at most max_ctas), then as few chunks per
// CTA as that allows.
ClusterShape cluster_shape(int64_t T, int max_ctas) {
  const int64_t per_chunk = (int64_t)max_ctas * kCThreads;
  const int chunks = (int)((T + per_chunk - 1) / per_chunk);
  const int64_t tc = (int64_t)chunks * kCThreads;
  return {(int)((T + tc - 1) / tc), chunks};
}

size_t cluster_smem_bytes(const Geom& g, int chunks) {
  return sizeof(uint64_t) * (size_t)chunks * kCThreads +
         sizeof(int32_t) * ((size_t)g.R * g.E + (size_t)g.R * g.R + 2 * (size_t)g.R +
                            2 * (size_t)chunks * kCWarps * g.R);
}
constexpr size_t kCMaxSmem = sizeof(uint64_t) * kCMaxChunks * kCThreads +
                             sizeof(int32_t) * ((size_t)kCMaxHist + EP_MAX_RANKS * EP_MAX_RANKS +
                                                2 * EP_MAX_RANKS +
                                                2 * (size_t)kCMaxChunks * kCWarps * EP_MAX_RANKS);

// floor(e / El) as (e * el_mul) >> 24 with el_mul = ceil(2^24 / El): exact
// because e * El < 2^24 (both below EP_MAX_EXPERTS = 4096).
inline uint32_t expert_rank_mul(int El) { return (uint32_t)(((1u << 24) + El - 1) / El); }

__global__ void __launch_bounds__(kCThreads, 1)
    layout_cluster_kernel(const int64_t* __restrict__ topk_idx, Geom g, int chunks,
                          uint32_t el_mul, uint8_t* __restrict__ is_token_in_rank,
                          int32_t* __restrict__ slot, int32_t* __restrict__ ntpr,
                          int32_t* __restrict__ ntpe, int32_t* __restrict__ recv_base,
                          int32_t* err) {
  pdl_wait_then_release();
  extern __shared__ uint64_t smem64[];
  const int R = g.R, E = g.E, K = g.K;
  const int Tr = (int)g.Tr, T = (int)g.T;  // T <= kCMaxTokens
  uint64_t* msk = smem64;          // [chunks][kCThreads] rank masks of this CTA's tokens
  int32_t* smem = reinterpret_cast<int32_t*>(msk + chunks * kCThreads);
  int32_t* hist = smem;            // [R][E]  slots of source s naming expert e
  int32_t* cnt_sr = hist + R * E;  // [R][R]  tokens of source s sent to r
  int32_t* tot = cnt_sr + R * R;   // [R]     tokens of this CTA sent to r
  int32_t* run = tot + R;          // [R]     next row of r for this CTA
  int32_t* wpre = run + R;         // [chunks * kCWarps][R] first row of r for each group of 32 tokens
  uint32_t* bal = reinterpret_cast<uint32_t*>(wpre + chunks * kCWarps * R);  // [chunks * kCWarps][R]
  const int c = (int)cluster_cta_rank();
  const int nc = (int)gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tc = chunks * kCThreads;
  const int t0 = c * tc;
  const int t1 = min(T, t0 + tc);  // t0 < t1: the shape leaves no CTA empty

  // the first chunk's first eight ids, loaded before the zeroing below so
  // that their memory latency overlaps it
  int64_t pre[8];
  {
    const int t = t0 + tid;
    const bool valid = t < t1;
    const int64_t* row = topk_idx + (int64_t)t * K;
#pragma unroll
    for (int u = 0; u < 8; ++u) pre[u] = (valid && u < K) ? row[u] : -1;
  }
  // only the rows of the sources this CTA holds are ever touched or read
  const int s_lo = t0 / Tr, s_hi = (t1 - 1) / Tr;
  for (int i = tid; i < (s_hi - s_lo + 1) * E; i += kCThreads) hist[s_lo * E + i] = 0;
  for (int i = tid; i < (s_hi - s_lo + 1) * R; i += kCThreads) cnt_sr[s_lo * R + i] = 0;
  __syncthreads();

  // --- masks, is_token_in_rank, this CTA's counts and its warps' ballots ---
  bool bad = false;
#pragma unroll 1
  for (int j = 0; j < chunks; ++j) {
    {
      const int t = t0 + j * kCThreads + tid;
      const bool valid = t < t1;
      const int s = valid ? t / Tr : 0;
      const int64_t* row = topk_idx + (int64_t)t * K;
      uint64_t mask = 0;
      for (int k0 = 0; k0 < K; k0 += 8) {
        int64_t ev[8];  // eight ids loaded before any is used
        if (j == 0 && k0 == 0) {
#pragma unroll
          for (int u = 0; u < 8; ++u) ev[u] = pre[u];
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) ev[u] = (valid && k0 + u < K) ? row[k0 + u] : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int64_t e = ev[u];
          if (e == -1) continue;
          if (e < -1 || e >= E) {
            bad = true;
          } else {
            atomicAdd(&hist[s * E + (int)e], 1);
            mask |= 1ull << (int)(((uint64_t)e * el_mul) >> 24);
          }
        }
      }
      msk[j * kCThreads + tid] = mask;
      if (valid) {
        write_member_row(is_token_in_rank + (int64_t)t * R, mask, R);
      }
      // lane r keeps this warp's ballot of destination r (and of r + 32)
      uint32_t b0 = 0, b1 = 0;
      for (int r = 0; r < R; ++r) {
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, (mask >> r) & 1);
        b0 = r == lane ? b : b0;
        b1 = r == lane + 32 ? b : b1;
      }
      uint32_t* wb = bal + (j * kCWarps + warp) * R;
      if (lane < R) wb[lane] = b0;
      if (lane + 32 < R) wb[lane + 32] = b1;
      // tokens per (source, destination): when the warp's tokens share one
      // source (always when Tr is a multiple of 32), one add per destination
      // from the ballots; else one add per destination of every token.  The
      // valid tokens are a prefix of the warp, so lane 0's source is theirs.
      const int s0 = __shfl_sync(0xFFFFFFFFu, s, 0);
      if (__all_sync(0xFFFFFFFFu, !valid || s == s0)) {
        if (lane < R && b0) atomicAdd(&cnt_sr[s0 * R + lane], __popc(b0));
        if (lane + 32 < R && b1) atomicAdd(&cnt_sr[s0 * R + lane + 32], __popc(b1));
      } else if (valid) {
        for (uint64_t m = mask; m != 0; m &= m - 1)
          atomicAdd(&cnt_sr[s * R + (__ffsll((long long)m) - 1)], 1);
      }
    }
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && err) atomicOr(err, EP_ERRBIT_BAD_EXPERT);
  __syncthreads();
  for (int r = tid; r < R; r += kCThreads) {
    int v = 0;
    for (int s = s_lo; s <= s_hi; ++s) v += cnt_sr[s * R + r];
    tot[r] = v;
  }
  cluster_arrive();
  cluster_wait();  // every CTA's counts are final and visible to the cluster

  // --- first row of every destination for this CTA, and recv_base ---
  if (warp == 0) {
    // lane l covers destinations l and l + 32; all loads issued before any sum
    int v[kCMaxCtas][2];
#pragma unroll
    for (int cc = 0; cc < kCMaxCtas; ++cc)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = lane + 32 * h;
        v[cc][h] = (cc < nc && r < R) ? dsmem_ld(dsmem_map(tot + r, (uint32_t)cc)) : 0;
      }
    int all[2] = {0, 0}, pre[2] = {0, 0};
#pragma unroll
    for (int cc = 0; cc < kCMaxCtas; ++cc)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        all[h] += v[cc][h];
        pre[h] += cc < c ? v[cc][h] : 0;
      }
    int inc0 = all[0], inc1 = all[1];
    for (int o = 1; o < 32; o <<= 1) {
      const int a0 = __shfl_up_sync(0xFFFFFFFFu, inc0, o);
      const int a1 = __shfl_up_sync(0xFFFFFFFFu, inc1, o);
      if (lane >= o) {
        inc0 += a0;
        inc1 += a1;
      }
    }
    const int sum0 = __shfl_sync(0xFFFFFFFFu, inc0, 31);
    const int sum1 = __shfl_sync(0xFFFFFFFFu, inc1, 31);
    const int base0 = inc0 - all[0], base1 = sum0 + inc1 - all[1];
    if (lane < R) run[lane] = base0 + pre[0];
    if (lane + 32 < R) run[lane + 32] = base1 + pre[1];
    if (c == 0) {
      if (lane < R) recv_base[lane] = base0;
      if (lane + 32 < R) recv_base[lane + 32] = base1;
      if (lane == 0) recv_base[R] = sum0 + sum1;
    }
  }

  // --- rows of num_tokens_per_rank / num_tokens_per_expert of the sources
  //     whose first token is in this CTA: sums over the CTAs holding them ---
  {
    const int s_beg = (t0 + Tr - 1) / Tr, s_end = (t1 + Tr - 1) / Tr;
    for (int s = s_beg; s < s_end; ++s) {
      const int c_last = ((s + 1) * Tr - 1) / tc;
      for (int col = tid; col < R + E; col += kCThreads) {
        const int32_t* p = col < R ? cnt_sr + s * R + col : hist + s * E + (col - R);
        int v = 0;
        for (int cc = c; cc <= c_last; ++cc) v += dsmem_ld(dsmem_map(p, (uint32_t)cc));
        if (col < R)
          ntpr[s * R + col] = v;
        else
          ntpe[s * E + (col - R)] = v;
      }
    }
  }
  cluster_arrive();  // this CTA no longer reads the other CTAs' shared memory
  __syncthreads();   // run[] is written

  // --- slots ---
  // First row of every (group of 32 tokens, destination): a prefix over the
  // CTA's groups in token order, from run[].
  const int ntok = t1 - t0;
  const int ngroups = (ntok + 31) / 32;
  for (int r = tid; r < R; r += kCThreads) {
    int acc = run[r];
    for (int w = 0; w < ngroups; ++w) {
      wpre[w * R + r] = acc;
      acc += __popc(bal[w * R + r]);
    }
  }
  __syncthreads();
  // The CTA's slot rows are one contiguous run of ntok * R entries; each
  // thread computes whole 16-byte pieces of it (R % 4 == 0) or single
  // entries, so that a warp's stores cover consecutive addresses.
  int32_t* out = slot + (int64_t)t0 * R;
  if ((R & 3) == 0) {
    const int rv = R / 4;
    for (int i = tid; i < ntok * rv; i += kCThreads) {
      const int tok = i / rv, r = (i - tok * rv) * 4;
      const uint64_t m = msk[tok] >> r;
      const uint32_t below = (1u << (tok & 31)) - 1u;  // the group's tokens before tok
      const uint32_t* b = bal + (tok >> 5) * R + r;
      const int32_t* p = wpre + (tok >> 5) * R + r;
      int sv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) sv[q] = ((m >> q) & 1) ? p[q] + __popc(b[q] & below) : -1;
      reinterpret_cast<int4*>(out)[i] = make_int4(sv[0], sv[1], sv[2], sv[3]);
    }
  } else {
    for (int i = tid; i < ntok * R; i += kCThreads) {
      const int tok = i / R, r = i - tok * R;
      const uint32_t below = (1u << (tok & 31)) - 1u;
      const int g = (tok >> 5) * R + r;
      out[i] = ((msk[tok] >> r) & 1) ? wpre[g] + __popc(bal[g] & below) : -1;
    }
  }
  cluster_wait();  // the other CTAs have finished reading this CTA's shared memory
}

ClusterSizeCache g_cluster_size;  // 16 or 8 CTAs, per device

cudaError_t launch_layout_cluster(const int64_t* topk_idx, const Geom& g, int32_t* ntpr,
                                  int32_t* ntpe, uint8_t* is_token_in_rank, int32_t* slot,
                                  int32_t* recv_base, int32_t* err_word, cudaStream_t st) {
  int max_ctas = 8;
  const cudaError_t e = g_cluster_size.get(layout_cluster_kernel, kCThreads, kCMaxSmem, &max_ctas);
  if (e != cudaSuccess) return e;
  const ClusterShape cs = cluster_shape(g.T, max_ctas);
  return launch_pdl_cluster(layout_cluster_kernel, cs.ctas, kCThreads,
                            cluster_smem_bytes(g, cs.chunks), cs.ctas, st, topk_idx, g,
                            cs.chunks, expert_rank_mul(g.El), is_token_in_rank, slot, ntpr,
                            ntpe, recv_base, err_word);
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
  const Geom g = make_geom(num_tokens, 1, num_experts, num_ranks, num_ranks);
  return carve(g, nullptr).bytes;
}

extern "C" int ep_layout_single_launch_fits(int64_t num_tokens, int num_ranks, int num_experts) {
  if (!routing_ok(num_tokens, 1, num_experts, num_ranks)) return 0;
  return single_launch_fits(num_tokens, num_ranks, num_experts) ? 1 : 0;
}

extern "C" int ep_layout_auto_single_launch(int64_t num_tokens, int num_ranks, int num_experts) {
  return ep_layout_single_launch_fits(num_tokens, num_ranks, num_experts) &&
         num_tokens <= kCAutoMaxTokens;
}

extern "C" ep_status_t ep_get_dispatch_layout_path(
    const int64_t* topk_idx, int64_t num_tokens, int num_topk, int num_experts, int num_ranks,
    int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
    int32_t* slot, int32_t* recv_base, int32_t* err_word, void* workspace,
    size_t workspace_bytes, int path, ep_stream_t stream) {
  if (!routing_ok(num_tokens, num_topk, num_experts, num_ranks)) return EP_ERR_INVALID_ARG;
  if (!num_tokens_per_rank || !num_tokens_per_expert || !recv_base) return EP_ERR_INVALID_ARG;
  if (path != EP_LAYOUT_AUTO && path != EP_LAYOUT_MULTI_LAUNCH && path != EP_LAYOUT_SINGLE_LAUNCH)
    return EP_ERR_INVALID_ARG;
  const bool fits = single_launch_fits(num_tokens, num_ranks, num_experts);
  if (path == EP_LAYOUT_SINGLE_LAUNCH && !fits) return EP_ERR_INVALID_ARG;
  const bool single = path == EP_LAYOUT_SINGLE_LAUNCH ||
                      (path == EP_LAYOUT_AUTO && fits && num_tokens <= kCAutoMaxTokens);
  if (num_tokens > 0) {
    if (!topk_idx || !is_token_in_rank || !slot) return EP_ERR_INVALID_ARG;
    if (!aligned16(slot) || !aligned16(is_token_in_rank) || !aligned16(topk_idx))
      return EP_ERR_INVALID_ARG;
    if (!single && (!workspace || !aligned16(workspace))) return EP_ERR_INVALID_ARG;
  }
  const Geom g = make_geom(num_tokens, num_topk, num_experts, num_ranks, num_ranks);
  const Workspace ws = carve(g, workspace);
  if (single) {
    if (launch_layout_cluster(topk_idx, g, num_tokens_per_rank, num_tokens_per_expert,
                              is_token_in_rank, slot, recv_base, err_word,
                              to_cuda(stream)) == cudaSuccess)
      return EP_OK;
    cudaGetLastError();  // clear the launch error
    // EP_LAYOUT_AUTO runs the multi-launch form instead when the device
    // refused the cluster (for instance a partition with too few free SMs)
    // and the caller passed a usable workspace; otherwise report the error.
    if (path != EP_LAYOUT_AUTO || !workspace || !aligned16(workspace) ||
        workspace_bytes < ws.bytes)
      return EP_ERR_CUDA;
  }
  if (num_tokens > 0 && workspace_bytes < ws.bytes) return EP_ERR_CAPACITY;
  launch_layout(topk_idx, g, ws, num_tokens_per_rank, num_tokens_per_expert, is_token_in_rank,
                slot, recv_base, err_word, to_cuda(stream));
  return launch_status();
}

extern "C" ep_status_t ep_get_dispatch_layout(const int64_t* topk_idx, int64_t num_tokens,
                                              int num_topk, int num_experts, int num_ranks,
                                              int32_t* num_tokens_per_rank,
                                              int32_t* num_tokens_per_expert,
                                              uint8_t* is_token_in_rank, int32_t* slot,
                                              int32_t* recv_base, int32_t* err_word,
                                              void* workspace, size_t workspace_bytes,
                                              ep_stream_t stream) {
  return ep_get_dispatch_layout_path(topk_idx, num_tokens, num_topk, num_experts, num_ranks,
                                     num_tokens_per_rank, num_tokens_per_expert,
                                     is_token_in_rank, slot, recv_base, err_word, workspace,
                                     workspace_bytes, EP_LAYOUT_AUTO, stream);
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
  const Geom g = make_geom(num_tokens, num_topk, num_experts, num_ranks, num_ranks);
  if (carve(g, nullptr).bytes > (size_t)EP_NOALLOC_SCRATCH_BYTES) return EP_ERR_CAPACITY;
  void* scratch = nullptr;
  const ep_status_t s = noalloc_scratch(&scratch);
  if (s != EP_OK) return s;
  const Workspace ws = carve(g, scratch);
  launch_layout(topk_idx, g, ws, num_tokens_per_rank, num_tokens_per_expert, is_token_in_rank,
                slot, recv_base, err_word, to_cuda(stream));
  return launch_status();
}

// ---------------------------------------------------------------------------
// Sharded form: one rank's layout of its own tokens, and the host-side
// offsets of the exchange.
//
// "[Not ready] MSCCLPP EP implementation" (mscclpp pull request 852):
// section "Scope", Intranode (get_dispatch_layout on each rank, then the
// dispatch over peer buffers) and the internode notify_dispatch commit (the
// count exchange that fixes the receiver-side prefix matrices).  Each rank
// lays out its own T tokens as the one source of a layout with R
// destinations: its send buffer is packed destination-major in token order,
// so the rows for destination r are one contiguous run.  After an all-gather
// of every rank's per-destination counts, each destination receives the
// runs in source-rank order, which gives exactly the rows of the
// single-call layout's destination r.
// ---------------------------------------------------------------------------
extern "C" size_t ep_shard_workspace_bytes(int64_t num_tokens, int num_ranks, int num_experts) {
  if (!routing_ok_any_t(num_tokens, 1, num_experts, num_ranks)) return 0;
  const Geom g = make_geom(num_tokens, 1, num_experts, num_ranks, 1);
  return carve(g, nullptr).bytes;
}

extern "C" ep_status_t ep_shard_layout(const int64_t* topk_idx, int64_t num_tokens, int num_topk,
                                       int num_experts, int num_ranks, int32_t* send_counts,
                                       int32_t* expert_counts, uint8_t* is_token_in_rank,
                                       int32_t* send_slot, int32_t* send_base,
                                       int32_t* err_word, void* workspace,
                                       size_t workspace_bytes, ep_stream_t stream) {
  // one source: T need not be a multiple of R
  if (!routing_ok_any_t(num_tokens, num_topk, num_experts, num_ranks)) return EP_ERR_INVALID_ARG;
  if (!send_counts || !expert_counts || !send_base) return EP_ERR_INVALID_ARG;
  const Geom g = make_geom(num_tokens, num_topk, num_experts, num_ranks, 1);
  const Workspace ws = carve(g, workspace);
  if (num_tokens > 0) {
    if (!topk_idx || !is_token_in_rank || !send_slot || !workspace) return EP_ERR_INVALID_ARG;
    if (!aligned16(send_slot) || !aligned16(is_token_in_rank) || !aligned16(topk_idx) ||
        !aligned16(workspace))
      return EP_ERR_INVALID_ARG;
    if (workspace_bytes < ws.bytes) return EP_ERR_CAPACITY;
  }
  launch_layout(topk_idx, g, ws, send_counts, expert_counts, is_token_in_rank, send_slot,
                send_base, err_word, to_cuda(stream));
  return launch_status();
}

extern "C" ep_status_t ep_shard_offsets(const int32_t* counts, int num_ranks, int rank,
                                        int64_t* send_offsets, int64_t* recv_offsets) {
  if (!counts || !send_offsets || !recv_offsets || num_ranks < 1 || num_ranks > EP_MAX_RANKS ||
      rank < 0 || rank >= num_ranks)
    return EP_ERR_INVALID_ARG;
  const int R = num_ranks;
  send_offsets[0] = 0;
  recv_offsets[0] = 0;
  for (int i = 0; i < R; ++i) {
    const int32_t out = counts[(size_t)rank * R + i];  // this rank's tokens sent to rank i
    const int32_t in = counts[(size_t)i * R + rank];   // rank i's tokens sent to this rank
    if (out < 0 || in < 0) return EP_ERR_INVALID_ARG;
    send_offsets[i + 1] = send_offsets[i] + out;
    recv_offsets[i + 1] = recv_offsets[i] + in;
  }
  return EP_OK;
}

extern "C" ep_status_t ep_shard_recv_tokens_per_expert(const int32_t* expert_counts,
                                                       int num_experts, int num_ranks, int rank,
                                                       int32_t* out) {
  if (!expert_counts || !out || num_ranks < 1 || num_ranks > EP_MAX_RANKS || num_experts < 1 ||
      num_experts > EP_MAX_EXPERTS || num_experts % num_ranks != 0 || rank < 0 ||
      rank >= num_ranks)
    return EP_ERR_INVALID_ARG;
  const int El = num_experts / num_ranks;
  for (int j = 0; j < El; ++j) {
    int64_t sum = 0;
    for (int s = 0; s < num_ranks; ++s)
      sum += expert_counts[(size_t)s * num_experts + (size_t)rank * El + j];
    if (sum > INT32_MAX) return EP_ERR_INVALID_ARG;
    out[j] = (int32_t)sum;
  }
  return EP_OK;
}
