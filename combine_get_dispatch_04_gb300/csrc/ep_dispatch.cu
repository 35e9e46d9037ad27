// ep_dispatch.cu -- token scatter into the packed per-destination receive
// buffer, bf16 or FP8 E4M3 with per-128-channel float32 scales.
//
// "[Not ready] MSCCLPP EP implementation" (mscclpp pull request 852):
// section "Scope", Intranode (intranode_dispatch), and the low-latency port
// (dispatch<kUseFP8,...>, the FP8 payload cast).  On one GPU the scatter is
// a memory-bound copy: each token row is read once from HBM and written once
// per destination rank.
//
// One warp per token, or per slice of a token when the batch is too small
// to fill the GPU (slices of a multiple of 32 vectors); a warp's work is the
// scatter of ep_scatter.cuh.  Many short-lived blocks: the block scheduler
// balances them over the SMs better than a persistent grid did (measured).
// Blocks of 4 warps: a block holds its SM slot until its slowest warp ends,
// and smaller blocks free the slots sooner.  Against 8 warps (alternating
// A/B runs, three each) the FP8 decode dispatch went from 45.8 to 43.7 us and
// the bf16 dispatch from 768.5 to 766.8 us (skewed), 429.4 to 427.2 us
// (DSV3) and 463.9 to 462.2 us (Mixtral); 16 warps were slower, 1 and 2
// warps no faster.
#include "ep_scatter.cuh"

namespace ep {
namespace {

constexpr int kWarps = 4;  // warps (tokens or token slices) per block
using Args = ScatterArgs;

template <bool kFP8>
__global__ void __launch_bounds__(kWarps * 32) dispatch_kernel(Args a) {
  pdl_wait_then_release();
  __shared__ int32_t dst_row[kWarps][EP_MAX_RANKS];
  __shared__ int32_t dst_rank[kWarps][EP_MAX_RANKS];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // receiver-side rows per local expert (column sums of the per-source counts)
  if (blockIdx.x == 0 && a.nrpe && a.ntpe) {
    for (int e = threadIdx.x; e < a.E; e += kWarps * 32) {
      int sum = 0;
      for (int s = 0; s < a.R; ++s) sum += a.ntpe[(int64_t)s * a.E + e];
      a.nrpe[e] = sum;  // [R, E_l] row-major == expert index e
    }
  }

  const int64_t gw = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t t = gw / a.nslices;
  const int slice = (int)(gw % a.nslices);
  if (t >= a.T) return;  // uniform per warp

  const int nvec = a.H / 8;  // 16-byte vectors per row
  const int4* src = a.x + t * nvec;
  // this warp's slice of the row: [vbeg, vend), vbeg a multiple of 32 vectors
  const int vbeg = slice * a.vps;
  const int vend = min(nvec, vbeg + a.vps);
  // The payload does not depend on the slots: its first round is in flight
  // while the slot row is read (two round trips overlap instead of following
  // one another; measured 0.5-1% faster on bf16 prefill batches).
  Round<kFP8> first;
  load_round<kFP8>(src, vbeg, vend, lane, first);

  const int nd = warp_dest_list(a, t, lane, dst_row[warp], dst_rank[warp]);
  if (nd == 0) return;
  if (slice == 0) warp_write_meta(a, t, nd, dst_row[warp], dst_rank[warp], lane);
  warp_scatter<kFP8>(a, src, vbeg, vend, nd, dst_row[warp], lane, first);
}

}  // namespace

// Slicing and launch shared by the rank-major and expert-major dispatch.
// Small batches: several warps share a token (each a run of a multiple of
// 32 vectors, one or more rounds of 32 * kUnroll), aiming at four waves of
// 64 warps per SM.
ep_status_t launch_dispatch(Args& a, bool fp8, ep_stream_t stream) {
  DeviceProps props;
  if (!device_props(&props)) return EP_ERR_CUDA;
  const int64_t num_tokens = a.T;
  plan_slices(a, fp8, props.sm_count);
  int64_t blocks = (num_tokens * a.nslices + kWarps - 1) / kWarps;
  if (blocks == 0) {
    if (!a.nrpe) return EP_OK;
    blocks = 1;
  }
  cudaStream_t st = to_cuda(stream);
  if (fp8)
    launch_pdl(dispatch_kernel<true>, (unsigned)blocks, kWarps * 32, 0, st, a);
  else
    launch_pdl(dispatch_kernel<false>, (unsigned)blocks, kWarps * 32, 0, st, a);
  return launch_status();
}

}  // namespace ep

using namespace ep;

extern "C" ep_status_t ep_dispatch(const void* x, int hidden, const int64_t* topk_idx,
                                   const float* topk_weights, int64_t num_tokens, int num_topk,
                                   int num_experts, int num_ranks, const int32_t* slot,
                                   const int32_t* num_tokens_per_expert,
                                   int64_t recv_capacity_rows, int use_fp8, void* recv_x,
                                   float* recv_scales, int32_t* recv_src_idx,
                                   int64_t* recv_topk_idx, float* recv_topk_weights,
                                   int32_t* num_recv_tokens_per_expert, int32_t* err_word,
                                   ep_stream_t stream) {
  if (!routing_ok_any_t(num_tokens, num_topk, num_experts, num_ranks)) return EP_ERR_INVALID_ARG;
  if (hidden < 8 || hidden % 8 != 0 || (use_fp8 && hidden % 128 != 0)) return EP_ERR_INVALID_ARG;
  if (recv_capacity_rows < 0) return EP_ERR_INVALID_ARG;
  if (num_tokens > 0) {
    if (!x || !topk_idx || !slot) return EP_ERR_INVALID_ARG;
    if ((recv_topk_idx || recv_topk_weights) && !topk_weights) return EP_ERR_INVALID_ARG;
    if (!aligned16(x)) return EP_ERR_INVALID_ARG;
  }
  // with no receive rows nothing is written (every slot is out of capacity),
  // so the receive buffers may then be NULL
  if (num_tokens > 0 && recv_capacity_rows > 0) {
    if (!recv_x || (use_fp8 && !recv_scales) || !aligned16(recv_x)) return EP_ERR_INVALID_ARG;
  }
  if (num_recv_tokens_per_expert && !num_tokens_per_expert) return EP_ERR_INVALID_ARG;
  Args a = {};
  a.x = static_cast<const int4*>(x);
  a.T = num_tokens;
  a.H = hidden;
  a.topk_idx = topk_idx;
  a.topk_w = topk_weights;
  a.K = num_topk;
  a.E = num_experts;
  a.El = num_experts / num_ranks;
  a.R = num_ranks;
  a.dest = slot;
  a.ndest = num_ranks;
  a.rank_meta = true;
  a.ntpe = num_tokens_per_expert;
  a.cap = recv_capacity_rows;
  a.recv_x = recv_x;
  a.recv_scales = recv_scales;
  a.recv_src_idx = recv_src_idx;
  a.recv_topk_idx = recv_topk_idx;
  a.recv_topk_w = recv_topk_weights;
  a.nrpe = num_recv_tokens_per_expert;
  a.err = err_word;
  return launch_dispatch(a, use_fp8 != 0, stream);
}

extern "C" ep_status_t ep_ll_dispatch(const void* x, int hidden, int64_t num_tokens, int num_topk,
                                      const int32_t* ll_slot, int64_t recv_capacity_rows,
                                      int use_fp8, void* recv_x, float* recv_scales,
                                      int32_t* recv_src_idx, int32_t* err_word,
                                      ep_stream_t stream) {
  if (num_tokens < 0 || num_topk < 1 || num_topk > EP_MAX_TOPK) return EP_ERR_INVALID_ARG;
  if (hidden < 8 || hidden % 8 != 0 || (use_fp8 && hidden % 128 != 0)) return EP_ERR_INVALID_ARG;
  if (recv_capacity_rows < 0 || recv_capacity_rows >= (int64_t(1) << 31)) return EP_ERR_INVALID_ARG;
  if (num_tokens > 0) {
    if (!x || !ll_slot || !aligned16(x)) return EP_ERR_INVALID_ARG;
  }
  if (num_tokens > 0 && recv_capacity_rows > 0) {  // no receive rows: nothing is written
    if (!recv_x || (use_fp8 && !recv_scales) || !aligned16(recv_x)) return EP_ERR_INVALID_ARG;
  }
  Args a = {};
  a.x = static_cast<const int4*>(x);
  a.T = num_tokens;
  a.H = hidden;
  a.K = num_topk;
  a.dest = ll_slot;
  a.ndest = num_topk;
  a.rank_meta = false;
  a.cap = recv_capacity_rows;
  a.recv_x = recv_x;
  a.recv_scales = recv_scales;
  a.recv_src_idx = recv_src_idx;
  a.err = err_word;
  return launch_dispatch(a, use_fp8 != 0, stream);
}
