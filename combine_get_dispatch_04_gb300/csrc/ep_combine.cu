// ep_combine.cu -- weighted gather-reduce of expert outputs back to tokens.
//
// "[Not ready] MSCCLPP EP implementation" (mscclpp pull request 852):
// section "Scope", Intranode (intranode_combine); the bench-accounting commit
// (combine moves one copy per dispatched (token, rank) row back to its
// owner); and the bulk-copy primitives PR (1-D cp.async.bulk loads into
// shared memory tracked by an mbarrier, the "multi-source pull and reduce,
// double buffered" pattern).  For every token t:
//     out[t] = bf16_rne( sum_k w[t][k] * y[slot[t][rank(e_k)]] )   (float32)
//
// Design (one persistent CTA per SM, warp-specialised):
//   - warp 0 is the producer.  For a batch of 32 tokens each lane gathers
//     one token's routing: its distinct destination ranks (each row is read
//     from HBM once, however many of the token's slots name that rank), the
//     row index of every top-k slot inside the staged tile, and the
//     weights.  Then, per (token, channel chunk), it waits for a free stage,
//     publishes the slot->row map and weights, arrives on the stage's "full"
//     mbarrier (all 32 lanes; lane 0 also posts the byte count) and issues
//     one 1-D bulk copy per distinct row (lane j copies row j).
//   - warps 1..8 are consumers: they wait on "full", accumulate the weighted
//     rows in float32 from shared memory (8 channels per thread, one 16-byte
//     shared load per slot), store 16 bytes of bf16 per thread, and release
//     the stage on its "empty" mbarrier.
//   - every wait is bounded (1 s); on a timeout the CTA records
//     EP_ERRBIT_TIMEOUT, stops issuing, waits (bounded) for the copies it has
//     in flight, and returns.
#include <cuda_bf16.h>

#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kChunkMax = kConsumerWarps * 32 * 8;  // channels covered by one pass
constexpr int kMaxStages = 16;
constexpr int kBatch = 32;  // tokens gathered per producer round
constexpr int kTabStride = EP_MAX_TOPK + 1;

struct StageDesc {
  float w[EP_MAX_TOPK];
  int8_t j[EP_MAX_TOPK];  // staged row of each top-k slot, -1 = masked
};

struct Args {
  const uint16_t* y;
  uint16_t* out;
  int64_t T;
  int H;
  const int64_t* topk_idx;
  const float* topk_w;
  int K, E, El, R;
  const int32_t* slot;
  int32_t* err;
  int C;       // channels per chunk (multiple of 8)
  int nchunk;  // chunks per token
  int S;       // pipeline stages
  uint32_t stage_bytes;
};

// dynamic shared memory layout after the S row tiles
struct Tail {
  StageDesc desc[kMaxStages];
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  float tw[kBatch][kTabStride];
  int32_t trow[kBatch][kTabStride];
  int8_t tj[kBatch][kTabStride];
  int32_t tD[kBatch];
  int abort;
};

__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  const bool got = mbar_wait_bounded(bar, parity, abort);
  return __all_sync(0xFFFFFFFFu, got);
}

__global__ void __launch_bounds__(kThreads, 1) combine_kernel(Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* tiles = smem;
  Tail& tl = *reinterpret_cast<Tail*>(smem + (size_t)a.S * a.stage_bytes);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.S; ++s) {
      mbar_init(&tl.full[s], 32);  // every producer lane arrives (releasing its writes)
      mbar_init(&tl.empty[s], kConsumerWarps);
    }
    tl.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  volatile int* abort = &tl.abort;
  const int64_t tb = a.T * blockIdx.x / gridDim.x;
  const int64_t te = a.T * (blockIdx.x + 1) / gridDim.x;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = l2_policy_evict_first();
    uint32_t it = 0;
    bool ok = true, bad = false;
    for (int64_t t0 = tb; t0 < te && ok; t0 += kBatch) {
      const int n = (int)(te - t0 < kBatch ? te - t0 : kBatch);
      if (lane < n) {
        const int64_t t = t0 + lane;
        int D = 0;
        for (int k = 0; k < a.K; ++k) {
          const int64_t e = a.topk_idx[t * a.K + k];
          int j = -1;
          if (e >= 0 && e < a.E) {
            const int r = (int)(e / a.El);
            for (int q = 0; q < D; ++q)
              if (tl.trow[lane][q] == r) j = q;
            if (j < 0) {
              j = D++;
              tl.trow[lane][j] = r;
            }
          } else if (e != -1) {
            bad = true;
          }
          tl.tj[lane][k] = (int8_t)j;
          tl.tw[lane][k] = a.topk_w[t * a.K + k];
        }
        for (int q = 0; q < D; ++q) tl.trow[lane][q] = a.slot[t * a.R + tl.trow[lane][q]];
        tl.tD[lane] = D;
      }
      __syncwarp();
      for (int i = 0; i < n && ok; ++i) {
        const int D = tl.tD[i];
        const int64_t t = t0 + i;
        (void)t;
        for (int c = 0; c < a.nchunk; ++c) {
          const uint32_t s = it % a.S, use = it / a.S;
          if (use > 0 && !wait_warp(&tl.empty[s], (use - 1) & 1, abort)) {
            ok = false;
            break;
          }
          if (lane < a.K) {
            tl.desc[s].j[lane] = tl.tj[i][lane];
            tl.desc[s].w[lane] = tl.tw[i][lane];
          }
          __syncwarp();
          const int c0 = c * a.C;
          const int clen = min(a.C, a.H - c0);
          if (lane == 0)
            mbar_arrive_expect_tx(&tl.full[s], (uint32_t)(D * clen * 2));
          else
            mbar_arrive(&tl.full[s]);
          __syncwarp();
          if (lane < D)
            bulk_load_g2s(tiles + (size_t)s * a.stage_bytes + (size_t)lane * a.C * 2,
                          a.y + (int64_t)tl.trow[i][lane] * a.H + c0, (uint32_t)clen * 2,
                          &tl.full[s], policy);
          ++it;
        }
      }
      __syncwarp();
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && a.err) atomicOr(a.err, EP_ERRBIT_BAD_EXPERT);
    if (!ok) {
      if (lane == 0) {
        *abort = 1;
        if (a.err) atomicOr(a.err, EP_ERRBIT_TIMEOUT);
      }
    }
    // Copies still in flight must land before the CTA may exit: wait for the
    // last fill of every stage (bounded, and regardless of the abort flag).
    const int zero = 0;
    const uint32_t first = it > (uint32_t)a.S ? it - (uint32_t)a.S : 0u;
    for (uint32_t u = first; u < it; ++u)
      (void)mbar_wait_bounded(&tl.full[u % a.S], (u / a.S) & 1, &zero);
  } else {
    // ------------------------------------------------------------ consumers
    const int ct = threadIdx.x - 32;
    uint32_t it = 0;
    bool ok = true;
    for (int64_t t = tb; t < te && ok; ++t) {
      uint16_t* orow = a.out + t * a.H;
      for (int c = 0; c < a.nchunk; ++c) {
        const uint32_t s = it % a.S;
        if (!wait_warp(&tl.full[s], (it / a.S) & 1, abort)) {
          ok = false;
          break;
        }
        const int c0 = c * a.C;
        const int clen = min(a.C, a.H - c0);
        const uint8_t* stage = tiles + (size_t)s * a.stage_bytes;
        for (int ch = ct * 8; ch < clen; ch += kConsumerWarps * 32 * 8) {
          float acc[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
          for (int k = 0; k < a.K; ++k) {
            const int j = tl.desc[s].j[k];
            if (j < 0) continue;
            const float w = tl.desc[s].w[k];
            const int4 v = *reinterpret_cast<const int4*>(stage + ((size_t)j * a.C + ch) * 2);
            float f[8];
            unpack_bf16x8(v, f);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(w, f[i], acc[i]);
          }
          int4 o;
          uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 p = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
            ow[i] = *reinterpret_cast<const uint32_t*>(&p);
          }
          *reinterpret_cast<int4*>(orow + c0 + ch) = o;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&tl.empty[s]);
        ++it;
      }
    }
    if (!ok && lane == 0) {
      *abort = 1;
      if (a.err) atomicOr(a.err, EP_ERRBIT_TIMEOUT);
    }
  }
}

size_t tail_bytes() { return align_up(sizeof(Tail), 128); }

}  // namespace

bool combine_plan(int H, int K, int R, int smem_optin, int* C, int* S, uint32_t* stage_bytes) {
  const int dmax = K < R ? K : R;
  const long budget = (long)smem_optin - (long)tail_bytes();
  if (budget <= 0) return false;
  int c = H < kChunkMax ? H : kChunkMax;
  long sb = (long)dmax * c * 2;
  while (sb * 4 > budget && c > 256) {
    c = (c / 2 + 7) / 8 * 8;
    sb = (long)dmax * c * 2;
  }
  long s = budget / sb;
  if (s > kMaxStages) s = kMaxStages;
  if (s < 2) return false;
  *C = c;
  *S = (int)s;
  *stage_bytes = (uint32_t)align_up((size_t)sb, 128);
  // recheck with the aligned tile size
  if ((long)*stage_bytes * *S > budget) *S = (int)(budget / *stage_bytes);
  return *S >= 2;
}

}  // namespace ep

using namespace ep;

extern "C" ep_status_t ep_combine(const void* y, int hidden, const int64_t* topk_idx,
                                  const float* topk_weights, int64_t num_tokens, int num_topk,
                                  int num_experts, int num_ranks, const int32_t* slot, void* out,
                                  int32_t* err_word, ep_stream_t stream) {
  if (!routing_ok(num_tokens, num_topk, num_experts, num_ranks)) return EP_ERR_INVALID_ARG;
  if (hidden < 8 || hidden % 8 != 0) return EP_ERR_INVALID_ARG;
  if (num_tokens == 0) return EP_OK;
  if (!y || !topk_idx || !topk_weights || !slot || !out) return EP_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(out)) return EP_ERR_INVALID_ARG;
  DeviceProps props;
  if (!device_props(&props)) return EP_ERR_CUDA;
  Args a;
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
  a.err = err_word;
  if (!combine_plan(hidden, num_topk, num_ranks, props.smem_optin, &a.C, &a.S, &a.stage_bytes))
    return EP_ERR_INVALID_ARG;
  a.nchunk = (hidden + a.C - 1) / a.C;
  const size_t smem = (size_t)a.S * a.stage_bytes + tail_bytes();
  if (cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return EP_ERR_CUDA;
  const int64_t grid = num_tokens < props.sm_count ? num_tokens : props.sm_count;
  combine_kernel<<<(unsigned)grid, kThreads, smem, to_cuda(stream)>>>(a);
  return launch_status();
}
