// ep_combine.cu -- weighted gather-reduce of expert outputs back to tokens.
//
// "[Not ready] MSCCLPP EP implementation" (mscclpp pull request 852):
// section "Scope", Intranode (intranode_combine); the bench-accounting commit
// (combine moves one copy per dispatched (token, rank) row back to its
// owner); and the bulk-copy primitives PR (1-D cp.async.bulk loads into
// shared memory tracked by an mbarrier, the "multi-source pull and reduce,
// double buffered" pattern).  For every token t:
//     out[t] = bf16_rne( sum_k w[t][k] * y[slot[t][rank(e_k)]] )   (float32)
// or, without weights, the rank sum of DeepEP's high-throughput combine:
//     out[t] = bf16_rne( sum over ranks r with slot[t][r] >= 0 of y[slot[t][r]] )
//
// Design: persistent CTAs, several per SM, three warp roles per CTA, all
// communication through mbarriers in shared memory.
//   - Tokens go out in batches of a few (up to 32).  Each CTA's first batch
//     is fixed; with a scheduling counter (the _sched entry points) every
//     further batch is claimed from it with one atomic, so CTAs that the
//     memory system serves faster take more batches and all finish within
//     about a batch of each other.  Without it (and when every CTA has only
//     its first batch) CTA b takes every grid-th batch.  The last CTA to
//     exit returns the counter to zero.
//   - warp 1 (routing): claims the next batch before it needs it, and for
//     each batch each lane gathers one token's routing into a
//     double-buffered table (headed by the batch's first token and size):
//     the token's distinct destination rows (each row is read from HBM once,
//     however many of the token's slots name that rank) and, per row, the
//     sum of the weights of the slots naming its rank.  Loads are issued
//     eight at a time, and the warp runs one batch ahead of the copies.
//   - warp 0 (copies): per (token, channel chunk) it waits for a free stage,
//     posts the byte count on the stage's "full" barrier and issues one 1-D
//     bulk copy per distinct row (lane j copies row j), with an L2
//     evict-first policy (every row is read once).
//   - warps 2..5 (reduce): wait on "full", accumulate the weighted rows in
//     float32 from shared memory (8 channels per thread and pass; the D
//     16-byte shared loads of a pass are independent and issued together),
//     store 16 bytes of bf16 per thread, release the stage on its "empty"
//     barrier, and a table once its batch is done.
// Each slot contributes w_k * y_row; slots naming the same rank share one
// staged row, so their weights are summed first (the same sum, with the
// float32 rounding applied in a different order).
// Sizing: on GB300 one CTA's bulk-copy ring sustains about one stage per
// memory round trip, so bandwidth comes from large stages (2048-channel
// chunks, wider when min(K, R) is small) and from 3-4 CTAs per SM, not from
// deep rings; the host picks the chunk, the stage count (2 or 3) and the
// CTAs per SM from the shared-memory budget.
// Every wait is bounded (1 s).  On a timeout the CTA records
// EP_ERRBIT_TIMEOUT, stops issuing, waits (bounded) for the copies it has in
// flight, and returns.
#include <cuda_bf16.h>

#include <cmath>

#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 2) * 32;
constexpr int kMaxStages = 3;
constexpr int kBatch = 32;              // tokens per routing table
constexpr int kTargetStageBytes = 16384;  // bytes a stage should carry at least
constexpr int kMaxCtasPerSm = 4;

struct Args {
  const uint16_t* y;
  uint16_t* out;
  int64_t T;
  int H;
  const int64_t* topk_idx;
  const float* topk_w;
  int K, E, El, R;
  const int32_t* slot;
  const int32_t* ll_slot;  // non-null: expert-major rows, one per top-k slot
  int32_t* err;
  int C;       // channels per chunk (multiple of 8)
  int nchunk;  // chunks per token
  int S;       // pipeline stages
  int dmax;    // rows per stage = min(K, R)
  uint32_t stage_bytes;
  int stall_unit;  // test hook: CTA 0 never arms this pipeline unit (-1: off)
  unsigned long long* sched;  // [2] claimed-batch and exited-block counters (null: static batches)
  int claim;                  // tokens per batch
  int64_t nbatches;           // ceil(T / claim): the claims one launch makes when it runs alone
};

// Offsets of the shared-memory regions that follow the S row tiles.
struct SmemLayout {
  size_t bars, rows, w, D, hdr, abort, total;
};

__host__ __device__ inline size_t al(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline SmemLayout smem_layout(int S, uint32_t stage_bytes, int dmax) {
  SmemLayout L;
  size_t off = (size_t)S * stage_bytes;
  L.bars = off;
  off += sizeof(uint64_t) * (2 * (size_t)S + 4);
  L.rows = off;
  off += sizeof(int32_t) * 2 * kBatch * (size_t)dmax;
  L.w = off;
  off += sizeof(float) * 2 * kBatch * (size_t)dmax;
  L.D = off;
  off += sizeof(int32_t) * 2 * kBatch;
  off = al(off, 8);
  L.hdr = off;
  off += sizeof(int64_t) * 2 + sizeof(int32_t) * 2;
  off = al(off, 16);
  L.abort = off;
  off += 16;
  L.total = al(off, 128);
  return L;
}

__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  const bool got = mbar_wait_bounded(bar, parity, abort);
  return __all_sync(0xFFFFFFFFu, got);
}

// One lane's token: its distinct source rows (in order of first appearance
// over k) and, per row, the sum of the weights of the slots that name its
// rank.  Global loads are issued eight slots at a time before any is used.
__device__ __forceinline__ int gather_token(const Args& a, int64_t t, int32_t* rows, float* W,
                                            bool& bad) {
  const float* wt = a.topk_w ? a.topk_w + t * a.K : nullptr;  // null: unweighted
  int D = 0;
  if (a.ll_slot) {  // expert-major: each live slot has its own row
    const int32_t* ls = a.ll_slot + t * a.K;
    for (int k0 = 0; k0 < a.K; k0 += 8) {
      int32_t p[8];
      float wv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = k0 + u;
        p[u] = k < a.K ? ls[k] : -1;
        wv[u] = k < a.K ? (wt ? wt[k] : 1.0f) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (p[u] >= 0) {
          rows[D] = p[u];
          W[D++] = wv[u];
        }
      }
    }
    return D;
  }
  const int64_t* idx = a.topk_idx + t * a.K;
  for (int k0 = 0; k0 < a.K; k0 += 8) {
    int64_t e[8];
    float wv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int k = k0 + u;
      e[u] = k < a.K ? idx[k] : -1;
      wv[u] = k < a.K ? (wt ? wt[k] : 1.0f) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (k0 + u >= a.K) break;
      if (e[u] >= 0 && e[u] < a.E) {
        const int r = (int)(e[u] / a.El);
        int jj = -1;
        for (int q = 0; q < D; ++q)
          if (rows[q] == r) jj = q;
        if (jj < 0) {
          rows[D] = r;  // a rank for now; replaced by its row below
          W[D++] = wv[u];
        } else if (wt) {
          W[jj] += wv[u];  // unweighted: each rank's row counts once
        }
      } else if (e[u] != -1) {
        bad = true;
      }
    }
  }
  const int32_t* srow = a.slot + t * a.R;
  for (int q0 = 0; q0 < D; q0 += 8) {
    int32_t v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = q0 + u < D ? srow[rows[q0 + u]] : 0;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (q0 + u < D) rows[q0 + u] = v[u];
  }
  return D;
}

// kP passes of one staged (token, chunk): for ch = ch0 + p*step (p < kP,
// ch < clen), out[ch..ch+8) = sum over the token's D staged rows of
// W[d] * row_d, in float32, stored as bf16.  With kDMax > 0 (D <= kDMax) the
// shared loads of all kP passes are issued together from unrolled code;
// kDMax == 0 is the general loop.
template <int kDMax, int kP>
__device__ __forceinline__ void reduce_rows(const uint8_t* stage, int C, int ch0, int step,
                                            int clen, int D, const float* Wreg, const float* Wsm,
                                            uint16_t* orow) {
  if constexpr (kDMax > 0) {
    int4 v[kP][kDMax];
#pragma unroll
    for (int p = 0; p < kP; ++p) {
      const int ch = ch0 + p * step;
#pragma unroll
      for (int d = 0; d < kDMax; ++d)
        if (ch < clen && d < D) v[p][d] = *reinterpret_cast<const int4*>(stage + ((size_t)d * C + ch) * 2);
    }
#pragma unroll
    for (int p = 0; p < kP; ++p) {
      const int ch = ch0 + p * step;
      if (ch >= clen) break;
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
      for (int d = 0; d < kDMax; ++d) {
        if (d < D) {
          float f[8];
          unpack_bf16x8(v[p][d], f);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] = fmaf(Wreg[d], f[q], acc[q]);
        }
      }
      int4 o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
        ow[q] = *reinterpret_cast<const uint32_t*>(&b);
      }
      st_stream_v4(reinterpret_cast<int4*>(orow + ch), o);
    }
  } else {
    for (int p = 0; p < kP; ++p) {
      const int ch = ch0 + p * step;
      if (ch >= clen) break;
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
      for (int d = 0; d < D; ++d) {
        const int4 v = *reinterpret_cast<const int4*>(stage + ((size_t)d * C + ch) * 2);
        const float wd = Wsm[d];
        float f[8];
        unpack_bf16x8(v, f);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = fmaf(wd, f[q], acc[q]);
      }
      int4 o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
        ow[q] = *reinterpret_cast<const uint32_t*>(&b);
      }
      st_stream_v4(reinterpret_cast<int4*>(orow + ch), o);
    }
  }
}

template <int kDMax, int kP>
__global__ void __launch_bounds__(kThreads, 4) combine_kernel(Args a) {
  // The grid is persistent (every block resident from the start), so an
  // early release would gain no launch overlap; it would only let the next
  // kernel's blocks take SMs as this grid drains, unevenly.  On one GB300
  // an early release here cost the following step 54 us on 131072 skewed
  // tokens (1584 against 1638 us) and 48 us on Mixtral, and saved nothing
  // on the others.
  pdl_wait();
  extern __shared__ __align__(128) uint8_t smem[];
  const SmemLayout lay = smem_layout(a.S, a.stage_bytes, a.dmax);
  uint8_t* tiles = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bars);
  uint64_t* empty = full + a.S;
  uint64_t* tfull = empty + a.S;  // [2] routing table ready
  uint64_t* tempty = tfull + 2;   // [2] routing table released by the reducers
  int32_t* trows = reinterpret_cast<int32_t*>(smem + lay.rows);  // [2][kBatch][dmax]
  float* tW = reinterpret_cast<float*>(smem + lay.w);            // [2][kBatch][dmax]
  int32_t* tD = reinterpret_cast<int32_t*>(smem + lay.D);        // [2][kBatch]
  int64_t* tT0 = reinterpret_cast<int64_t*>(smem + lay.hdr);      // [2] first token of the batch
  int32_t* tN = reinterpret_cast<int32_t*>(tT0 + 2);              // [2] its tokens (0: no more)
  volatile int* abort = reinterpret_cast<volatile int*>(smem + lay.abort);
  uint32_t* nclaims = reinterpret_cast<uint32_t*>(smem + lay.abort + 4);  // this CTA's claims
  uint32_t* overclaim = nclaims + 1;  // a claim beyond what a lone launch hands out
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 32);
      mbar_init(&tempty[b], kConsumerWarps);
    }
    *abort = 0;
    *nclaims = 0;
    *overclaim = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // Batches of a.claim tokens: block b's first is [b * claim, (b + 1) * claim).
  // With a.sched the rest are claimed from a.sched[0] (offset by
  // gridDim.x * claim), so blocks that are served faster take more of them;
  // without it block b takes every gridDim.x-th batch after its first.
  const int64_t claim = a.claim;
  const int64_t dyn0 = (int64_t)gridDim.x * claim;

  if (warp == 1) {
    // ------------------------------------------------------------ routing
    bool ok = true, bad = false;
    uint32_t claims = 0;
    bool over = false;
    int64_t t0 = (int64_t)blockIdx.x * claim;
    for (uint32_t bi = 0;; ++bi) {
      const int buf = bi & 1;
      const uint32_t use = bi >> 1;
      unsigned long long nxt = 0;  // the next batch, claimed before it is needed
      const bool claimed = a.sched && t0 < a.T;
      if (claimed && lane == 0) {
        nxt = atomicAdd(a.sched, (unsigned long long)claim);
        ++claims;
      }
      if (use > 0 && !wait_warp(&tempty[buf], (use - 1) & 1, abort)) {
        ok = false;
        break;
      }
      const int n = t0 < a.T ? (int)(a.T - t0 < claim ? a.T - t0 : claim) : 0;
      if (lane == 0) {
        tT0[buf] = t0;
        tN[buf] = n;
      }
      if (lane < n) {
        const size_t e = (size_t)buf * kBatch + lane;
        tD[e] = gather_token(a, t0 + lane, trows + e * a.dmax, tW + e * a.dmax, bad);
      }
      mbar_arrive(&tfull[buf]);  // every lane releases its own table writes
      // a launch alone hands out exactly nbatches claims, 0 .. nbatches-1.
      // Checked only here, so that the claim's round trip (all blocks claim
      // at once at the start) overlaps the gather instead of delaying it.
      if (claimed && lane == 0)
        over |= nxt >= (unsigned long long)a.nbatches * (unsigned long long)claim;
      if (n == 0) break;
      t0 = a.sched ? dyn0 + (int64_t)__shfl_sync(0xFFFFFFFFu, nxt, 0) : t0 + dyn0;
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && a.err) atomicOr(a.err, EP_ERRBIT_BAD_EXPERT);
    if (lane == 0) {
      *nclaims = claims;
      *overclaim = over ? 1u : 0u;
    }
    if (!ok && lane == 0) {
      *abort = 1;
      if (a.err) atomicOr(a.err, EP_ERRBIT_TIMEOUT);
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ copies
    const uint64_t policy = l2_policy_evict_first();
    uint32_t it = 0, bi = 0;
    bool ok = true;
    for (; ok; ++bi) {
      const int buf = bi & 1;
      if (!wait_warp(&tfull[buf], (bi >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      const int n = tN[buf];
      if (n == 0) break;
      for (int i = 0; i < n && ok; ++i) {
        const size_t e = (size_t)buf * kBatch + i;
        const int D = tD[e];
        const int64_t row = lane < D ? trows[e * a.dmax + lane] : 0;
        for (int c = 0; c < a.nchunk; ++c) {
          const uint32_t s = it % a.S, use = it / a.S;
          if (use > 0 && !wait_warp(&empty[s], (use - 1) & 1, abort)) {
            ok = false;
            break;
          }
          const int c0 = c * a.C;
          const int clen = min(a.C, a.H - c0);
          if (blockIdx.x == 0 && (int)it == a.stall_unit) {  // test hook: leave it unarmed
            ++it;
            continue;
          }
          if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(D * clen * 2));
          __syncwarp();
          if (lane < D)
            bulk_load_g2s(tiles + (size_t)s * a.stage_bytes + (size_t)lane * a.C * 2,
                          a.y + row * a.H + c0, (uint32_t)clen * 2, &full[s], policy);
          ++it;
        }
      }
    }
    if (!ok && lane == 0) {
      *abort = 1;
      if (a.err) atomicOr(a.err, EP_ERRBIT_TIMEOUT);
    }
    // Copies still in flight must land before the CTA may exit: wait for the
    // last fill of every stage (bounded, and regardless of the abort flag).
    const int zero = 0;
    const uint32_t first = it > (uint32_t)a.S ? it - (uint32_t)a.S : 0u;
    for (uint32_t u = first; u < it; ++u)
      (void)mbar_wait_bounded(&full[u % a.S], (u / a.S) & 1, &zero);
  } else {
    // ------------------------------------------------------------ reduce
    const int ct = threadIdx.x - 64;
    uint32_t it = 0, bi = 0;
    bool ok = true;
    for (; ok; ++bi) {
      const int buf = bi & 1;
      if (!wait_warp(&tfull[buf], (bi >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      const int n = tN[buf];
      const int64_t t0 = tT0[buf];
      if (n == 0) break;
      for (int i = 0; i < n && ok; ++i) {
        const size_t e = (size_t)buf * kBatch + i;
        const float* Wsm = tW + e * a.dmax;
        float Wreg[kDMax > 0 ? kDMax : 1];
        int D = 0;
        uint16_t* orow = a.out + (t0 + i) * a.H;
        for (int c = 0; c < a.nchunk; ++c) {
          const uint32_t s = it % a.S;
          if (!wait_warp(&full[s], (it / a.S) & 1, abort)) {
            ok = false;
            break;
          }
          if (c == 0) {  // the table entry is visible once the token's first stage is
            D = tD[e];
#pragma unroll
            for (int d = 0; d < (kDMax > 0 ? kDMax : 1); ++d) Wreg[d] = d < D ? Wsm[d] : 0.0f;
          }
          const int c0 = c * a.C;
          const int clen = min(a.C, a.H - c0);
          const uint8_t* stage = tiles + (size_t)s * a.stage_bytes;
          constexpr int kStep = kConsumerWarps * 32 * 8;
          for (int ch = ct * 8; ch < clen; ch += kP * kStep)
            reduce_rows<kDMax, kP>(stage, a.C, ch, kStep, clen, D, Wreg, Wsm, orow + c0);
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
          ++it;
        }
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&tempty[buf]);
    }
    if (!ok && lane == 0) {
      *abort = 1;
      if (a.err) atomicOr(a.err, EP_ERRBIT_TIMEOUT);
    }
  }
  // The last block to leave resets the counters for the next launch: every
  // block has stopped claiming by then.  sched[1] packs the blocks that have
  // left (bits 0..31), the claims they made (bits 32..62) and whether any of
  // them ran out of a bounded wait (bit 63).  A launch that had the counters
  // to itself, from zero, leaves with exactly nbatches claims and
  // sched[0] == nbatches * claim, every claim below that and every exit index
  // below gridDim.x.  Anything else means that another launch shared the
  // counters, or that they were not zero at launch: some tokens may have been
  // skipped, so the launch reports EP_ERRBIT_SCHED.
  if (!a.sched) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    constexpr unsigned long long kLeft = 0xFFFFFFFFull, kAbort = 1ull << 63;
    const unsigned long long mine =
        1ull + ((unsigned long long)*nclaims << 32) + (*abort ? kAbort : 0ull);
    __threadfence();
    const unsigned long long prev = atomicAdd(a.sched + 1, mine);
    bool shared = *overclaim != 0 || (prev & kLeft) >= (unsigned long long)gridDim.x;
    if ((prev & kLeft) == (unsigned long long)gridDim.x - 1) {
      __threadfence();
      const unsigned long long all = prev + mine;
      const unsigned long long claimed = *reinterpret_cast<volatile unsigned long long*>(a.sched);
      // a launch that timed out loses claims on purpose: it reports EP_ERRBIT_TIMEOUT
      if (!(all & kAbort))
        shared |= ((all >> 32) & 0x7FFFFFFFull) != (unsigned long long)a.nbatches ||
                  claimed != (unsigned long long)a.nbatches * (unsigned long long)a.claim;
      a.sched[0] = 0;
      a.sched[1] = 0;
    }
    if (shared && a.err) atomicOr(a.err, EP_ERRBIT_SCHED);
  }
}

struct Plan {
  int C, S, ctas_per_sm;
  uint32_t stage_bytes;
  size_t smem;
};

// Chunk, stage count and CTAs per SM for a shape: stages of at least
// kTargetStageBytes when min(K,R) rows are staged, as many CTAs per SM (up
// to 4) as the shared memory allows, and 3 stages where they still fit.
bool make_plan(int H, int K, int R, const DeviceProps& p, Plan* out) {
  const int dmax = K < R ? K : R;
  const int reserve = 1024;  // per-block shared memory the runtime keeps
  int c = kTargetStageBytes / (2 * dmax);
  c = c < 2048 ? 2048 : c;
  c = (c + 7) / 8 * 8;
  if (c > H) c = H;
  for (; c >= 8; c = (c / 2 + 7) / 8 * 8) {
    const uint32_t sb = (uint32_t)al((size_t)dmax * c * 2, 128);
    for (int cps = kMaxCtasPerSm; cps >= 1; --cps) {
      const long per_cta = (long)p.smem_per_sm / cps - reserve;
      for (int S = kMaxStages; S >= 2; --S) {
        const size_t need = smem_layout(S, sb, dmax).total;
        if ((long)need <= per_cta && (long)need <= (long)p.smem_optin) {
          out->C = c;
          out->S = S;
          out->ctas_per_sm = cps;
          out->stage_bytes = sb;
          out->smem = need;
          return true;
        }
      }
    }
    if (c == 8) break;
  }
  return false;
}

}  // namespace

// Plan, occupancy-sized persistent grid and launch, shared by the rank-major
// and expert-major combine.
thread_local int g_stall_unit = -1;  // set by ep_debug_set_combine_stall, used once

// Per device and kernel variant: the dynamic shared-memory limit set so far
// and the blocks per SM at the last queried size.  Set-up calls run only
// when the size grows or changes, so that steady-state launches make no
// host calls besides the launch itself (and can be captured in a graph).
struct Residency {
  size_t smem_limit = 0;     // cudaFuncAttributeMaxDynamicSharedMemorySize set so far
  size_t smem_queried = 0;   // size the occupancy below was computed for
  int resident = 0;
};
constexpr int kResidencyDevices = 64;
std::mutex g_residency_mu;
Residency g_residency[kResidencyDevices][4];

cudaError_t kernel_residency(void (*kernel)(Args), int which, size_t smem, int* resident) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kResidencyDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_residency_mu);
  Residency& r = g_residency[dev][which];
  if (smem > r.smem_limit) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    r.smem_limit = smem;
  }
  if (smem != r.smem_queried || r.resident == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r.resident, kernel, kThreads, smem);
    if (e != cudaSuccess) return e;
    r.smem_queried = smem;
  }
  *resident = r.resident;
  return cudaSuccess;
}

// Tokens per batch for a grid of `ctas` blocks.  At least T / (64 * ctas),
// so that every block takes many batches and the faster blocks absorb the
// slower ones' share.  And at least enough that the claims on the one
// counter stay under about 100 per microsecond: same-address atomics on
// GB300 saturated between 130 and 170 per us (batches of one token took
// skewed routing from 1544 to 1720 us per step).  The rate is estimated
// from a 6.6 TB/s gather of 1 + min(K, R) rows of H channels per token,
// over at least 10 us.
int claim_tokens(int64_t T, int64_t ctas, int H, int dmax) {
  int64_t c = T / (ctas * 64);
  const double us = fmax(10.0, (double)T * 2.0 * H * (1 + dmax) / 6.6e6);
  const int64_t by_rate = (int64_t)ceil((double)T / us / 100.0);
  if (c < by_rate) c = by_rate;
  return (int)(c < 1 ? 1 : c > kBatch ? kBatch : c);
}

ep_status_t launch_combine(Args& a, const DeviceProps& props, ep_stream_t stream) {
  a.stall_unit = g_stall_unit;
  g_stall_unit = -1;
  Plan plan;
  if (!make_plan(a.H, a.dmax, a.dmax, props, &plan)) return EP_ERR_INVALID_ARG;
  a.C = plan.C;
  a.S = plan.S;
  a.stage_bytes = plan.stage_bytes;
  a.nchunk = (a.H + a.C - 1) / a.C;
  // unrolled reductions for up to 8 rows per token (every workload here),
  // with more passes in flight when there are fewer rows
  const int which = a.dmax <= 2 ? 0 : a.dmax <= 4 ? 1 : a.dmax <= 8 ? 2 : 3;
  void (*kernel)(Args) = which == 0   ? combine_kernel<2, 4>
                         : which == 1 ? combine_kernel<4, 2>
                         : which == 2 ? combine_kernel<8, 1>
                                      : combine_kernel<0, 1>;
  int resident = 0;
  if (kernel_residency(kernel, which, plan.smem, &resident) != cudaSuccess) return EP_ERR_CUDA;
  if (resident < 1) return EP_ERR_CUDA;
  const int64_t ctas =
      (int64_t)props.sm_count * (resident < plan.ctas_per_sm ? resident : plan.ctas_per_sm);
  a.claim = claim_tokens(a.T, ctas, a.H, a.dmax);
  const int64_t batches = (a.T + a.claim - 1) / a.claim;
  a.nbatches = batches;
  const int64_t grid = batches < ctas ? batches : ctas;
  // One batch per CTA leaves nothing to claim: the static schedule then
  // spares every CTA its failed claim and its exit count on the shared
  // counters (same-address atomics; measured on the 512-token batch: combine
  // 12.3 -> 10.3 us, step as a CUDA-graph replay 23.7 -> 21.5 us).  The
  // counters are left untouched.
  if (batches <= grid) a.sched = nullptr;
  launch_pdl(kernel, (unsigned)grid, kThreads, plan.smem, to_cuda(stream), a);
  return launch_status();
}

}  // namespace ep

using namespace ep;

namespace {

bool sched_ok(const uint64_t* sched) {
  return sched == nullptr || (reinterpret_cast<uintptr_t>(sched) & 7) == 0;
}

ep_status_t combine_rank_major(const void* y, int hidden, const int64_t* topk_idx,
                               const float* topk_weights, int64_t num_tokens, int num_topk,
                               int num_experts, int num_ranks, const int32_t* slot, void* out,
                               uint64_t* sched, int32_t* err_word, ep_stream_t stream) {
  if (!routing_ok_any_t(num_tokens, num_topk, num_experts, num_ranks)) return EP_ERR_INVALID_ARG;
  if (hidden < 8 || hidden % 8 != 0) return EP_ERR_INVALID_ARG;
  if (num_tokens == 0) return EP_OK;
  if (!y || !topk_idx || !slot || !out) return EP_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(out) || !sched_ok(sched)) return EP_ERR_INVALID_ARG;
  DeviceProps props;
  if (!device_props(&props)) return EP_ERR_CUDA;
  Args a = {};
  a.y = static_cast<const uint16_t*>(y);
  a.out = static_cast<uint16_t*>(out);
  a.T = num_tokens;
  a.H = hidden;
  a.topk_idx = topk_idx;
  a.topk_w = topk_weights;
  a.K = num_topk;
  a.E = num_experts;
  a.El = num_experts / num_ranks;
  a.R = num_ranks;
  a.slot = slot;
  a.ll_slot = nullptr;
  a.err = err_word;
  a.dmax = num_topk < num_ranks ? num_topk : num_ranks;
  a.sched = reinterpret_cast<unsigned long long*>(sched);
  return launch_combine(a, props, stream);
}

ep_status_t combine_expert_major(const void* y, int hidden, const float* topk_weights,
                                 int64_t num_tokens, int num_topk, const int32_t* ll_slot,
                                 void* out, uint64_t* sched, int32_t* err_word,
                                 ep_stream_t stream) {
  if (num_tokens < 0 || num_topk < 1 || num_topk > EP_MAX_TOPK) return EP_ERR_INVALID_ARG;
  if (hidden < 8 || hidden % 8 != 0) return EP_ERR_INVALID_ARG;
  if (num_tokens == 0) return EP_OK;
  if (!y || !ll_slot || !out) return EP_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(out) || !sched_ok(sched)) return EP_ERR_INVALID_ARG;
  DeviceProps props;
  if (!device_props(&props)) return EP_ERR_CUDA;
  Args a = {};
  a.y = static_cast<const uint16_t*>(y);
  a.out = static_cast<uint16_t*>(out);
  a.T = num_tokens;
  a.H = hidden;
  a.topk_w = topk_weights;
  a.K = num_topk;
  a.ll_slot = ll_slot;
  a.err = err_word;
  a.dmax = num_topk;
  a.sched = reinterpret_cast<unsigned long long*>(sched);
  return launch_combine(a, props, stream);
}

}  // namespace

extern "C" ep_status_t ep_combine(const void* y, int hidden, const int64_t* topk_idx,
                                  const float* topk_weights, int64_t num_tokens, int num_topk,
                                  int num_experts, int num_ranks, const int32_t* slot, void* out,
                                  int32_t* err_word, ep_stream_t stream) {
  return combine_rank_major(y, hidden, topk_idx, topk_weights, num_tokens, num_topk, num_experts,
                            num_ranks, slot, out, nullptr, err_word, stream);
}

extern "C" ep_status_t ep_combine_sched(const void* y, int hidden, const int64_t* topk_idx,
                                        const float* topk_weights, int64_t num_tokens,
                                        int num_topk, int num_experts, int num_ranks,
                                        const int32_t* slot, void* out, uint64_t* sched,
                                        int32_t* err_word, ep_stream_t stream) {
  return combine_rank_major(y, hidden, topk_idx, topk_weights, num_tokens, num_topk, num_experts,
                            num_ranks, slot, out, sched, err_word, stream);
}

extern "C" ep_status_t ep_ll_combine(const void* y, int hidden, const float* topk_weights,
                                     int64_t num_tokens, int num_topk, const int32_t* ll_slot,
                                     void* out, int32_t* err_word, ep_stream_t stream) {
  return combine_expert_major(y, hidden, topk_weights, num_tokens, num_topk, ll_slot, out,
                              nullptr, err_word, stream);
}

extern "C" ep_status_t ep_ll_combine_sched(const void* y, int hidden, const float* topk_weights,
                                           int64_t num_tokens, int num_topk,
                                           const int32_t* ll_slot, void* out, uint64_t* sched,
                                           int32_t* err_word, ep_stream_t stream) {
  return combine_expert_major(y, hidden, topk_weights, num_tokens, num_topk, ll_slot, out, sched,
                              err_word, stream);
}

extern "C" void ep_debug_set_combine_stall(int unit) { ep::g_stall_unit = unit; }
