// ep_fused.cu -- get_dispatch_layout and dispatch in one launch, for batches
// small enough that the layout is bound by latency (decode-size inputs).
//
// "[Not ready] MSCCLPP EP implementation" (mscclpp pull request 852):
// section "Scope" (get_dispatch_layout, intranode_dispatch), the internode
// cached_notify commit (the count exchange that fixes the receive offsets),
// and the low-latency port's dispatch<kUseFP8,...>.  The pages run layout,
// count exchange and data movement as separate kernels; on one GPU the count
// exchange is a wait inside one grid.
//
// The grid is the dispatch's: one warp per (token, slice) item, many
// short-lived blocks.  In addition, the first G0 blocks to start -- picked by
// an atomic ticket, not by blockIdx, so that no block ever waits on a block
// that has not started -- compute the layout's offsets:
//   A. warp w of layout block k takes 32-token group g = 8k + w (groups never
//      straddle two source ranks): each lane's rank mask, its
//      is_token_in_rank row, and one 32-bit ballot per destination, stored
//      group-major in the workspace (bal[g][r]).
//   -- the G0 layout blocks meet at a barrier (a counter in the caller's
//      state; bounded wait) --
//   B. each layout block sums the ballots per destination: the totals give
//      recv_base (written by the first layout block), and the groups before
//      each of its own give pre[g][r], the rows of destination r taken by
//      the groups before g.  The last layout block to finish releases the
//      scatter.  The layout blocks then write the rows of num_tokens_per_rank
//      and num_tokens_per_expert of the sources they are given (per-source
//      expert histograms in shared memory; num_recv_tokens_per_expert by
//      atomics), off the scatter's path.
// Every block starts with one round trip for three independent things: its
// start ticket, a first look at its release flag, and the first round of
// each warp's slice of x.  It then waits (bounded) for the release, unless it
// started after it, and each warp finds its token's rows itself: lane r
// reads bal[g][r] and pre[g][r] in one coalesced load each, so that
//     slot[t][r] = recv_base[r] + pre[g][r] + #{earlier tokens of g sent to r}.
// The warp of slice 0 writes the token's slot row; then every warp scatters
// its slice exactly as ep_dispatch does (ep_scatter.cuh).
//
// The state (EP_FUSED_SYNC_WORDS 64-bit words: the ticket, barrier, done and
// exit counters and the release flags) is zeroed once by the caller; the
// last block to leave returns it to zero.  A bounded wait that runs out sets
// EP_ERRBIT_TIMEOUT; the blocks then skip their scatter and leave.
//
// Measured on one GB300 against ep_get_dispatch_layout followed by
// ep_dispatch, per layout -> dispatch -> combine step: 16384 tokens at 8
// ranks, 7168 bf16 channels, top-8 of 256 experts: 448.5 against 450.7 us
// (8192 tokens: 238.0 against 237.5 us); every smaller batch is slower
// fused: the 4096-token FP8 decode batch at 32 ranks 150.3 against 133.5 us,
// 512 tokens at 4 ranks 27.0 against 23.4 us.  The layout phase takes about
// 10 us of the launch (its exchanges go through L2 under the other blocks'
// loads) and overlaps with nothing, whereas two launches overlap the layout
// with the dispatch's launch; and each of many short blocks pays for a
// ticket, a flag poll and an exit count on shared counters.
#include <mutex>

#include "ep_scatter.cuh"

namespace ep {
namespace {

constexpr int kFWarps = 8;                 // warps per block (one item each)
constexpr int64_t kFusedMaxTokens = 16384;

// The state's words, each counter on a 256-byte line of its own: the start
// ticket, the layout blocks' barrier, the layout blocks done, the blocks
// that have left, and kReleaseCopies copies of the release flag, so that the
// blocks waiting for the layout poll 16 lines and not one (polls of one
// line by every waiting block slowed the barrier and the release).
constexpr int kWordsPerLine = 32;
constexpr int kTicket = 0, kBarrier = 1 * kWordsPerLine, kDone = 2 * kWordsPerLine,
              kExits = 3 * kWordsPerLine, kRelease = 4 * kWordsPerLine;
constexpr int kReleaseCopies = 16;
static_assert(kRelease + kReleaseCopies * kWordsPerLine == EP_FUSED_SYNC_WORDS,
              "EP_FUSED_SYNC_WORDS must cover the counters and the release flags");

struct FusedArgs {
  ScatterArgs s;        // the scatter: dest = slot, ndest = R
  int32_t* ntpr;        // [R, R]
  int32_t* ntpe;        // [R, E]
  uint8_t* itr;         // [T, R]
  int32_t* slot;        // [T, R]
  int32_t* recv_base;   // [R + 1]
  int32_t* nrpe;        // [E] (nullable)
  uint32_t* bal;        // workspace: [W][R] ballots
  int32_t* pre;         // workspace: [W][R] rows of each destination before each group
  unsigned long long* sync;  // [EP_FUSED_SYNC_WORDS]: see kTicket ... kRelease
  int64_t Tr;           // tokens per source rank
  int gps;              // 32-token groups per source rank
  int W;                // groups, R * gps
  int G0;               // layout blocks, ceil(W / kFWarps)
  uint32_t el_mul;      // rank(e) = (e * el_mul) >> 24
  int stall;            // test hook: the layout block with ticket 0 never reaches the barrier
};

// Spins (one thread) until *p >= target; false after kWaitTimeoutNs.
__device__ __forceinline__ bool wait_at_least(const unsigned long long* p, unsigned long long target) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    if (v >= target) return true;
    if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
    __nanosleep(128);
  }
}

// Per-block shared state of the layout part.
struct LayoutSmem {
  int32_t tot[EP_MAX_RANKS];              // rows per destination, all groups
  int32_t pre[EP_MAX_RANKS];              // rows per destination before this block's groups
  int32_t cnt[kFWarps][EP_MAX_RANKS];     // rows per destination of each of this block's groups
  int32_t base[EP_MAX_RANKS + 1];         // recv_base
};

// Phase A for warp `warp` of the layout block with ticket k: one 32-token
// group's is_token_in_rank rows and its ballots (lanes past the source's end
// vote for nothing).
__device__ __forceinline__ void layout_group(const FusedArgs& f, int k, int warp, int lane,
                                             bool& bad) {
  const ScatterArgs& a = f.s;
  const int g = k * kFWarps + warp;
  if (g >= f.W) return;  // uniform per warp
  const int s = g / f.gps, gl = g % f.gps;
  const int64_t tl = (int64_t)gl * 32 + lane;
  const bool valid = tl < f.Tr;
  const int64_t t = s * f.Tr + tl;
  uint64_t mask = 0;
  const int64_t* row = a.topk_idx + t * a.K;
  for (int k0 = 0; k0 < a.K; k0 += 8) {
    int64_t ev[8];  // eight ids loaded before any is used
#pragma unroll
    for (int u = 0; u < 8; ++u) ev[u] = (valid && k0 + u < a.K) ? row[k0 + u] : -1;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t e = ev[u];
      if (e == -1) continue;
      if (e < -1 || e >= a.E)
        bad = true;
      else
        mask |= 1ull << (int)(((uint64_t)e * f.el_mul) >> 24);
    }
  }
  if (valid) {
    uint8_t* mrow = f.itr + t * a.R;
    if ((a.R & 3) == 0) {
      for (int r = 0; r < a.R; r += 4) {
        // bits r..r+3 spread to the low bit of four bytes
        const uint32_t x = (uint32_t)(mask >> r) & 0xFu;
        *reinterpret_cast<uint32_t*>(mrow + r) = (x * 0x00204081u) & 0x01010101u;
      }
    } else {
      for (int r = 0; r < a.R; ++r) mrow[r] = (uint8_t)((mask >> r) & 1);
    }
  }
  // lane r keeps this group's ballot of destination r (and of r + 32)
  uint32_t b0 = 0, b1 = 0;
  for (int r = 0; r < a.R; ++r) {
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, (mask >> r) & 1);
    b0 = r == lane ? b : b0;
    b1 = r == lane + 32 ? b : b1;
  }
  if (lane < a.R) f.bal[(int64_t)g * a.R + lane] = b0;
  if (lane + 32 < a.R) f.bal[(int64_t)g * a.R + lane + 32] = b1;
}

// Ballots each thread of a layout block loads in phase B: the whole table,
// W * R words, is read by the block in at most two unrolled rounds.
constexpr int kBallotsPerThread = 16;
constexpr int kMaxBallots = 2 * kBallotsPerThread * kFWarps * 32;  // R * W

// Phase B for the layout block with ticket k (all its threads): per
// destination, the rows of all groups (recv_base) and, for each of this
// block's groups, the rows of the groups before it (pre).  This is what the
// scatter waits for; the counts follow in layout_counts.  Thread i takes
// destination r = i % R and every (256 / R)-th group from i / R, so that a
// warp's loads of one group's ballots are contiguous, and all its loads are
// issued before any is used.
__device__ __forceinline__ void layout_offsets(const FusedArgs& f, int k, int warp, int lane,
                                               LayoutSmem& L) {
  const ScatterArgs& a = f.s;
  const int R = a.R, W = f.W;
  const int g0 = k * kFWarps;
  constexpr int kThreads = kFWarps * 32;
  for (int r = threadIdx.x; r < R; r += kThreads) {
    L.tot[r] = 0;
    L.pre[r] = 0;
  }
  __syncthreads();
  const int tpr = kThreads / R;  // threads per destination (R <= 64)
  const int r = threadIdx.x % R, gi = threadIdx.x / R;
  int all = 0, pre = 0;
  if (gi < tpr) {
    for (int j0 = 0; j0 * tpr < W; j0 += kBallotsPerThread) {
      uint32_t b[kBallotsPerThread];
#pragma unroll
      for (int j = 0; j < kBallotsPerThread; ++j) {
        const int g = gi + (j0 + j) * tpr;
        b[j] = g < W ? f.bal[(int64_t)g * R + r] : 0u;
      }
#pragma unroll
      for (int j = 0; j < kBallotsPerThread; ++j) {
        const int g = gi + (j0 + j) * tpr;
        const int c = __popc(b[j]);
        all += c;
        pre += g < g0 ? c : 0;
        if (g >= g0 && g < g0 + kFWarps && g < W) L.cnt[g - g0][r] = c;
      }
    }
    atomicAdd(&L.tot[r], all);
    atomicAdd(&L.pre[r], pre);
  }
  __syncthreads();
  if (warp == 0) {  // recv_base: exclusive prefix over destinations (R <= 64)
    const int v0 = lane < R ? L.tot[lane] : 0, v1 = lane + 32 < R ? L.tot[lane + 32] : 0;
    int i0 = v0, i1 = v1;
    for (int o = 1; o < 32; o <<= 1) {
      const int x0 = __shfl_up_sync(0xFFFFFFFFu, i0, o), x1 = __shfl_up_sync(0xFFFFFFFFu, i1, o);
      if (lane >= o) {
        i0 += x0;
        i1 += x1;
      }
    }
    const int sum0 = __shfl_sync(0xFFFFFFFFu, i0, 31), sum1 = __shfl_sync(0xFFFFFFFFu, i1, 31);
    if (lane < R) L.base[lane] = i0 - v0;
    if (lane + 32 < R) L.base[lane + 32] = sum0 + i1 - v1;
    if (lane == 0) L.base[R] = sum0 + sum1;
  }
  // pre[g][r] for this block's groups: warp w writes its group's row
  const int g = g0 + warp;
  if (g < W) {
    for (int rr = lane; rr < R; rr += 32) {
      int run = L.pre[rr];
      for (int w = 0; w < warp; ++w) run += L.cnt[w][rr];
      f.pre[(int64_t)g * R + rr] = run;
    }
  }
  __syncthreads();
  if (k == 0)
    for (int rr = threadIdx.x; rr <= R; rr += kThreads) f.recv_base[rr] = L.base[rr];
  __syncthreads();  // every write above precedes the block's release
}

// The rest of the layout's outputs, after the scatter has been released:
// the rows of num_tokens_per_rank and
// num_tokens_per_expert of the sources s with s % G0 == k, the latter from a
// per-source expert histogram in shared memory; num_recv_tokens_per_expert
// (zeroed by ticket 0 before the barrier) by atomics.
__device__ __forceinline__ void layout_counts(const FusedArgs& f, int k, int warp, int lane,
                                              int32_t* hist) {
  const ScatterArgs& a = f.s;
  const int R = a.R;
  for (int s = k; s < R; s += f.G0) {
    for (int r = warp; r < R; r += kFWarps) {
      const uint32_t* br = f.bal + (int64_t)s * f.gps * R + r;
      int c = 0;
      for (int gl = lane; gl < f.gps; gl += 32) c += __popc(br[(int64_t)gl * R]);
      for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
      if (lane == 0) f.ntpr[s * R + r] = c;
    }
    for (int e = threadIdx.x; e < a.E; e += kFWarps * 32) hist[e] = 0;
    __syncthreads();
    const int64_t* ids = a.topk_idx + s * f.Tr * a.K;
    for (int64_t i = threadIdx.x; i < f.Tr * a.K; i += kFWarps * 32) {
      const int64_t e = ids[i];
      if (e >= 0 && e < a.E) atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += kFWarps * 32) {
      const int c = hist[e];
      f.ntpe[(int64_t)s * a.E + e] = c;
      if (f.nrpe && c) atomicAdd(&f.nrpe[e], c);
    }
    __syncthreads();
  }
}

// After the release: token t's row in every destination, from its group's
// ballots and offsets (lane r takes destination r, and r + 32), as the
// destination list of ep_scatter.cuh's warp_dest_list.  The warp of slice 0
// also writes the token's slot row.
__device__ __forceinline__ int warp_slots(const FusedArgs& f, int64_t t, int slice, int lane,
                                          int32_t* dst_row, int32_t* dst_rank) {
  const ScatterArgs& a = f.s;
  const int R = a.R;
  const int64_t s = t / f.Tr, tl = t % f.Tr;
  const int64_t g = s * f.gps + tl / 32;
  const int bit = (int)(tl % 32);
  int nd = 0;
  bool over = false;
  for (int r0 = 0; r0 < R; r0 += 32) {
    const int r = r0 + lane;
    int32_t sl = -1;
    if (r < R) {
      const uint32_t b = f.bal[g * R + r];
      if ((b >> bit) & 1) sl = f.recv_base[r] + f.pre[g * R + r] + __popc(b & ((1u << bit) - 1u));
      if (slice == 0) f.slot[t * R + r] = sl;
    }
    const bool ok = sl >= 0 && sl < a.cap;
    over |= sl >= a.cap;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, ok);
    if (ok) {
      const int pos = nd + __popc(bal & ((1u << lane) - 1u));
      dst_row[pos] = sl;
      dst_rank[pos] = r;
    }
    nd += __popc(bal);
  }
  if (__any_sync(0xFFFFFFFFu, over) && lane == 0 && a.err) atomicOr(a.err, EP_ERRBIT_CAPACITY);
  __syncwarp();
  return nd;
}

template <bool kFP8>
__global__ void __launch_bounds__(kFWarps * 32, kFP8 ? 4 : 2) fused_kernel(FusedArgs f) {
  pdl_wait_then_release();
  extern __shared__ int32_t hist[];  // [E] per-source expert histogram (layout blocks)
  __shared__ int32_t dst_row[kFWarps][EP_MAX_RANKS];
  __shared__ int32_t dst_rank[kFWarps][EP_MAX_RANKS];
  __shared__ LayoutSmem L;
  __shared__ unsigned long long s_ticket;
  __shared__ int s_ok;
  const ScatterArgs& a = f.s;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // One round trip for three independent things: the start ticket (only
  // the layout role depends on it), a first look at this block's release
  // flag (blocks that start after the release never wait), and the first
  // round of this warp's slice of x (x does not depend on the layout).
  const unsigned long long* flag =
      f.sync + kRelease + (blockIdx.x % kReleaseCopies) * kWordsPerLine;
  unsigned long long seen = 0;
  if (threadIdx.x == 0) {
    s_ticket = atomicAdd(f.sync + kTicket, 1ull);
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(seen) : "l"(flag) : "memory");
    s_ok = 1;
  }
  const int nvec = a.H / 8;
  const int64_t gw = (int64_t)blockIdx.x * kFWarps + warp;
  const int64_t t = gw / a.nslices;
  const int slice = (int)(gw % a.nslices);
  const bool active = t < a.T;  // uniform per warp
  const int4* src = a.x + t * nvec;
  const int vbeg = slice * a.vps;
  const int vend = min(nvec, vbeg + a.vps);
  Round<kFP8> first;
  if (active) load_round<kFP8>(src, vbeg, vend, lane, first);
  __syncthreads();
  const unsigned long long ticket = s_ticket;
  const bool layout_block = ticket < (unsigned long long)f.G0;

  if (layout_block) {
    const int k = (int)ticket;
    bool bad = false;
    if (k == 0 && f.nrpe)
      for (int e = threadIdx.x; e < a.E; e += kFWarps * 32) f.nrpe[e] = 0;
    layout_group(f, k, warp, lane, bad);
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && a.err) atomicOr(a.err, EP_ERRBIT_BAD_EXPERT);
    __syncthreads();
    if (threadIdx.x == 0) {
      if (!(k == 0 && f.stall)) {  // the test hook leaves this block's arrival out
        __threadfence();
        atomicAdd(f.sync + kBarrier, 1ull);
      }
      if (!wait_at_least(f.sync + kBarrier, (unsigned long long)f.G0)) {
        s_ok = 0;
        if (a.err) atomicOr(a.err, EP_ERRBIT_TIMEOUT);
      }
    }
    __syncthreads();
    if (s_ok) {
      layout_offsets(f, k, warp, lane, L);
      if (threadIdx.x == 0) {
        // the slots are written; the last layout block releases the scatter
        __threadfence();
        if (atomicAdd(f.sync + kDone, 1ull) == (unsigned long long)f.G0 - 1) {
          // one fence, then plain stores: a release store per flag would
          // put a fence before each of them
          __threadfence();
          for (int j = 0; j < kReleaseCopies; ++j)
            asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(f.sync + kRelease +
                                                                    j * kWordsPerLine),
                         "l"(1ull)
                         : "memory");
        }
      }
      layout_counts(f, k, warp, lane, hist);
    }
  }

  // the scatter, once every layout block is done
  if (threadIdx.x == 0 && s_ok && seen == 0) {
    if (!wait_at_least(flag, 1ull)) {
      s_ok = 0;
      if (a.err) atomicOr(a.err, EP_ERRBIT_TIMEOUT);
    }
  }
  __syncthreads();
  if (s_ok && active) {
    const int nd = warp_slots(f, t, slice, lane, dst_row[warp], dst_rank[warp]);
    if (nd > 0) {
      if (slice == 0) warp_write_meta(a, t, nd, dst_row[warp], dst_rank[warp], lane);
      warp_scatter<kFP8>(a, src, vbeg, vend, nd, dst_row[warp], lane, first);
    }
  }

  // the last block to leave returns the state to zero for the next launch
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(f.sync + kExits, 1ull) == (unsigned long long)gridDim.x - 1) {
      __threadfence();
      f.sync[kTicket] = 0;
      f.sync[kBarrier] = 0;
      f.sync[kDone] = 0;
      for (int j = 0; j < kReleaseCopies; ++j) f.sync[kRelease + j * kWordsPerLine] = 0;
      f.sync[kExits] = 0;
    }
  }
}

// Workspace: ballots [W][R], then offsets [W][R].
size_t fused_workspace(int64_t W, int R) {
  return align_up(sizeof(uint32_t) * (size_t)W * R, 256) + sizeof(int32_t) * (size_t)W * R;
}

bool fused_fits(int64_t T, int R, int E) {
  if (!routing_ok(T, 1, E, R) || T <= 0 || T > kFusedMaxTokens) return false;
  const int64_t gps = (T / R + 31) / 32;
  return (int64_t)R * R * gps <= kMaxBallots;
}

thread_local int g_fused_stall = 0;  // set by ep_debug_set_fused_stall, used once

std::mutex g_fused_mu;
size_t g_fused_smem_limit[64] = {};  // dynamic shared memory enabled so far, per device

}  // namespace
}  // namespace ep

using namespace ep;

extern "C" int ep_layout_dispatch_fused_fits(int64_t num_tokens, int num_ranks, int num_experts) {
  return fused_fits(num_tokens, num_ranks, num_experts) ? 1 : 0;
}

extern "C" size_t ep_layout_dispatch_fused_workspace_bytes(int64_t num_tokens, int num_ranks,
                                                           int num_experts) {
  if (!fused_fits(num_tokens, num_ranks, num_experts)) return 0;
  const int64_t gps = (num_tokens / num_ranks + 31) / 32;
  return fused_workspace((int64_t)num_ranks * gps, num_ranks);
}

extern "C" void ep_debug_set_fused_stall(int on) { ep::g_fused_stall = on ? 1 : 0; }

extern "C" ep_status_t ep_layout_dispatch_fused(
    const void* x, int hidden, const int64_t* topk_idx, const float* topk_weights,
    int64_t num_tokens, int num_topk, int num_experts, int num_ranks,
    int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
    int32_t* slot, int32_t* recv_base, int64_t recv_capacity_rows, int use_fp8, void* recv_x,
    float* recv_scales, int32_t* recv_src_idx, int64_t* recv_topk_idx, float* recv_topk_weights,
    int32_t* num_recv_tokens_per_expert, void* workspace, size_t workspace_bytes,
    uint64_t* sync, int32_t* err_word, ep_stream_t stream) {
  if (!routing_ok(num_tokens, num_topk, num_experts, num_ranks)) return EP_ERR_INVALID_ARG;
  if (!fused_fits(num_tokens, num_ranks, num_experts)) return EP_ERR_INVALID_ARG;
  if (hidden < 8 || hidden % 8 != 0 || (use_fp8 && hidden % 128 != 0)) return EP_ERR_INVALID_ARG;
  if (recv_capacity_rows < 0) return EP_ERR_INVALID_ARG;
  if (!x || !topk_idx || !num_tokens_per_rank || !num_tokens_per_expert || !is_token_in_rank ||
      !slot || !recv_base || !workspace || !sync)
    return EP_ERR_INVALID_ARG;
  if ((recv_topk_idx || recv_topk_weights) && !topk_weights) return EP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(slot) || !aligned16(is_token_in_rank) ||
      !aligned16(workspace) || (reinterpret_cast<uintptr_t>(sync) & 7) != 0)
    return EP_ERR_INVALID_ARG;
  if (recv_capacity_rows > 0) {  // no receive rows: nothing is written, the buffers may be NULL
    if (!recv_x || (use_fp8 && !recv_scales) || !aligned16(recv_x)) return EP_ERR_INVALID_ARG;
  }
  const int R = num_ranks;
  const int64_t Tr = num_tokens / R;
  const int gps = (int)((Tr + 31) / 32);
  const int W = R * gps;
  if (workspace_bytes < fused_workspace(W, R)) return EP_ERR_CAPACITY;
  DeviceProps props;
  if (!device_props(&props)) return EP_ERR_CUDA;

  FusedArgs f = {};
  ScatterArgs& a = f.s;
  a.x = static_cast<const int4*>(x);
  a.T = num_tokens;
  a.H = hidden;
  a.topk_idx = topk_idx;
  a.topk_w = topk_weights;
  a.K = num_topk;
  a.E = num_experts;
  a.El = num_experts / R;
  a.R = R;
  a.dest = slot;
  a.ndest = R;
  a.rank_meta = true;
  a.ntpe = nullptr;
  a.cap = recv_capacity_rows;
  a.recv_x = recv_x;
  a.recv_scales = recv_scales;
  a.recv_src_idx = recv_src_idx;
  a.recv_topk_idx = recv_topk_idx;
  a.recv_topk_w = recv_topk_weights;
  a.nrpe = nullptr;
  a.err = err_word;
  plan_slices(a, use_fp8 != 0, props.sm_count);
  f.ntpr = num_tokens_per_rank;
  f.ntpe = num_tokens_per_expert;
  f.itr = is_token_in_rank;
  f.slot = slot;
  f.recv_base = recv_base;
  f.nrpe = num_recv_tokens_per_expert;
  f.bal = static_cast<uint32_t*>(workspace);
  f.pre = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) +
                                     align_up(sizeof(uint32_t) * (size_t)W * R, 256));
  f.sync = reinterpret_cast<unsigned long long*>(sync);
  f.Tr = Tr;
  f.gps = gps;
  f.W = W;
  f.G0 = (W + kFWarps - 1) / kFWarps;
  f.el_mul = (uint32_t)(((1u << 24) + a.El - 1) / a.El);  // floor(e / El) for e * El < 2^24
  f.stall = g_fused_stall;
  g_fused_stall = 0;

  int64_t blocks = (num_tokens * a.nslices + kFWarps - 1) / kFWarps;
  if (blocks < f.G0) blocks = f.G0;
  const size_t smem = sizeof(int32_t) * (size_t)num_experts;
  void (*kernel)(FusedArgs) = use_fp8 ? fused_kernel<true> : fused_kernel<false>;
  {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return EP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_fused_mu);
    // both variants get the largest size once (E <= EP_MAX_EXPERTS)
    if (g_fused_smem_limit[dev] == 0) {
      const int lim = (int)(sizeof(int32_t) * EP_MAX_EXPERTS);
      if (cudaFuncSetAttribute(fused_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               lim) != cudaSuccess ||
          cudaFuncSetAttribute(fused_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               lim) != cudaSuccess)
        return EP_ERR_CUDA;
      g_fused_smem_limit[dev] = (size_t)lim;
    }
  }
  launch_pdl(kernel, (unsigned)blocks, kFWarps * 32, smem, to_cuda(stream), f);
  return launch_status();
}
