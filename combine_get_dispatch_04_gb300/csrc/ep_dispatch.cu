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
// to fill the GPU (slices of a multiple of 32 vectors).  Lanes hold 16-byte
// vectors of the row (8 bf16 channels); kUnroll vectors per lane are loaded
// before the stores, so each warp keeps 16 x 512 bytes (bf16) or 4 x 512
// bytes (FP8) of reads in flight.
// Loads bypass L1, stores use the streaming policy.  In the FP8 variant each
// lane holds two adjacent vectors and 8 lanes hold one block of 128
// channels: its amax is taken on the raw bf16 bits (per-halfword unsigned
// max of |x|, then a 3-step xor-shuffle), one lane per block computes the
// block's two divisions (a warp's 8 blocks in one instruction sequence), and
// the block is quantised in registers and written to every destination in
// 16-byte stores, with the 8 scales of a round in one 32-byte run.  The
// quantiser rounds exactly as the format definition requires: 448/a and a/448
// are single correctly rounded divisions (__fdiv_rn), x * (448/a) is a single
// multiply (__fmul_rn), and the E4M3 conversion is the hardware's
// round-to-nearest-even, saturate-to-finite conversion.
#include <cuda_fp8.h>

#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kWarps = 8;  // tokens per block
// 16-byte vectors each lane loads before it stores them: 16 for the bf16
// copy (a whole 4096-channel row per warp in flight; measured faster than 8
// and 4 although it leaves 2 blocks per SM), 4 for the FP8 kernel, whose
// quantiser needs the registers.
template <bool kFP8>
constexpr int kUnrollOf = kFP8 ? 4 : 16;

struct Args {
  const int4* x;
  int64_t T;
  int H;
  const int64_t* topk_idx;
  const float* topk_w;
  int K, E, El, R;
  const int32_t* dest;  // [T, ndest] destination rows, -1 = none
  int ndest;            // R (rank-major layout) or K (expert-major layout)
  bool rank_meta;       // write the per-row top-k metadata of the rank-major layout
  const int32_t* ntpe;
  int64_t cap;
  void* recv_x;
  float* recv_scales;
  int32_t* recv_src_idx;
  int64_t* recv_topk_idx;
  float* recv_topk_w;
  int32_t* nrpe;
  int32_t* err;
  int nslices;  // warps per token
  int vps;      // 16-byte vectors per slice (a multiple of 32)
};

__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

template <bool kFP8>
__global__ void __launch_bounds__(kWarps * 32) dispatch_kernel(Args a) {
  constexpr int kUnroll = kUnrollOf<kFP8>;
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

  // destinations of this token, in column order
  int nd = 0;
  bool over = false;
  for (int r0 = 0; r0 < a.ndest; r0 += 32) {
    const int r = r0 + lane;
    const int32_t sl = r < a.ndest ? a.dest[t * a.ndest + r] : -1;
    const bool ok = sl >= 0 && sl < a.cap;
    over |= sl >= a.cap;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, ok);
    if (ok) {
      const int pos = nd + __popc(bal & ((1u << lane) - 1u));
      dst_row[warp][pos] = sl;
      dst_rank[warp][pos] = r;
    }
    nd += __popc(bal);
  }
  if (__any_sync(0xFFFFFFFFu, over) && lane == 0 && a.err) atomicOr(a.err, EP_ERRBIT_CAPACITY);
  __syncwarp();
  if (nd == 0) return;

  // per-row metadata: source token, and the top-k entries that are local to
  // the destination (local expert id and weight), -1 / 0 elsewhere
  if (slice == 0 && !a.rank_meta && a.recv_src_idx) {
    for (int d = lane; d < nd; d += 32) a.recv_src_idx[dst_row[warp][d]] = (int32_t)t;
  }
  if (slice == 0 && a.rank_meta && (a.recv_src_idx || a.recv_topk_idx || a.recv_topk_w)) {
    // keep the small metadata rows in L2 (evict-last) until neighbouring
    // rows, written by other warps, have filled their sectors
    const uint64_t keep = l2_policy_evict_last();
    const int64_t e = lane < a.K ? a.topk_idx[t * a.K + lane] : -1;
    const float w = (lane < a.K && a.topk_w) ? a.topk_w[t * a.K + lane] : 0.0f;
    const int er = (e >= 0 && e < a.E) ? (int)(e / a.El) : -1;
    for (int d = 0; d < nd; ++d) {
      const int64_t row = dst_row[warp][d];
      const int r = dst_rank[warp][d];
      if (lane == 0 && a.recv_src_idx) st_hint_b32(a.recv_src_idx + row, (uint32_t)t, keep);
      if (lane < a.K) {
        const bool here = er == r;
        if (a.recv_topk_idx)
          st_hint_b64(a.recv_topk_idx + row * a.K + lane,
                      (uint64_t)(here ? e - (int64_t)r * a.El : -1), keep);
        if (a.recv_topk_w)
          st_hint_b32(a.recv_topk_w + row * a.K + lane, __float_as_uint(here ? w : 0.0f), keep);
      }
    }
  }

  const int nvec = a.H / 8;  // 16-byte vectors per row
  const int4* src = a.x + t * nvec;
  // this warp's slice of the row: [vbeg, vend), vbeg a multiple of 32 vectors
  const int vbeg = slice * a.vps;
  const int vend = min(nvec, vbeg + a.vps);
  if constexpr (!kFP8) {
    int4* out = reinterpret_cast<int4*>(a.recv_x);
    for (int v0 = vbeg; v0 < vend; v0 += 32 * kUnroll) {
      int4 buf[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < vend) buf[u] = ld_stream_v4(src + v);
      }
      for (int d = 0; d < nd; ++d) {
        int4* dst = out + (int64_t)dst_row[warp][d] * nvec;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < vend) st_stream_v4(dst + v, buf[u]);
        }
      }
    }
  } else {
    // Each lane holds two adjacent vectors (16 channels), so a 128-channel
    // block is 8 lanes and its 16 E4M3 codes per lane go out in one 16-byte
    // store.  H % 128 == 0 and vbeg % 32 == 0 make vend % 16 == 0, so blocks
    // are wholly in or out of the slice.
    uint8_t* out = reinterpret_cast<uint8_t*>(a.recv_x);
    const int nblk = a.H / 128;
    constexpr int kPairs = kUnroll / 2;  // vector pairs per lane and round
    for (int v0 = vbeg; v0 < vend; v0 += 32 * kUnroll) {
      int4 raw[kUnroll];
      uint32_t mbits[kPairs];  // amax of the lane's block, as bf16 bits
#pragma unroll
      for (int u = 0; u < kPairs; ++u) {
        const int v = v0 + u * 64 + 2 * lane;
        const bool in = v < vend;
        raw[2 * u] = in ? ld_stream_v4(src + v) : make_int4(0, 0, 0, 0);
        raw[2 * u + 1] = in ? ld_stream_v4(src + v + 1) : make_int4(0, 0, 0, 0);
        // for finite bf16 the order of |x| is the unsigned order of the low
        // 15 bits, so a per-halfword unsigned max gives the exact amax bits
        const int4& p = raw[2 * u];
        const int4& q = raw[2 * u + 1];
        uint32_t m = __vmaxu2(
            __vmaxu2(__vmaxu2((uint32_t)p.x & 0x7FFF7FFFu, (uint32_t)p.y & 0x7FFF7FFFu),
                     __vmaxu2((uint32_t)p.z & 0x7FFF7FFFu, (uint32_t)p.w & 0x7FFF7FFFu)),
            __vmaxu2(__vmaxu2((uint32_t)q.x & 0x7FFF7FFFu, (uint32_t)q.y & 0x7FFF7FFFu),
                     __vmaxu2((uint32_t)q.z & 0x7FFF7FFFu, (uint32_t)q.w & 0x7FFF7FFFu)));
        m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        mbits[u] = m;
      }
      // one correctly rounded division pair for the round's 8 blocks: lane
      // i < 8 takes block i (pair u = i / 4, lane group i % 4), in row order
      const uint32_t m0 = __shfl_sync(0xFFFFFFFFu, mbits[0], 8 * (lane & 3));
      const uint32_t m1 = __shfl_sync(0xFFFFFFFFu, mbits[1], 8 * (lane & 3));
      const uint32_t mine = (lane & 4) ? m1 : m0;
      const float am = fmaxf(__uint_as_float(mine << 16), 1e-4f);
      const float sc = __fdiv_rn(am, 448.0f);
      const float iv = __fdiv_rn(448.0f, am);
      uint4 qv[kPairs];
#pragma unroll
      for (int u = 0; u < kPairs; ++u) {
        const float inv = __shfl_sync(0xFFFFFFFFu, iv, 4 * u + (lane >> 3));
        float f[8];
        unpack_bf16x8(raw[2 * u], f);
        qv[u].x = cvt_e4m3x4(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv), __fmul_rn(f[2], inv),
                             __fmul_rn(f[3], inv));
        qv[u].y = cvt_e4m3x4(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv), __fmul_rn(f[6], inv),
                             __fmul_rn(f[7], inv));
        unpack_bf16x8(raw[2 * u + 1], f);
        qv[u].z = cvt_e4m3x4(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv), __fmul_rn(f[2], inv),
                             __fmul_rn(f[3], inv));
        qv[u].w = cvt_e4m3x4(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv), __fmul_rn(f[6], inv),
                             __fmul_rn(f[7], inv));
      }
      // lanes 0..7 hold the round's 8 scales in row order
      const bool scale_lane = lane < 8 && v0 + 16 * lane < vend;
      for (int d = 0; d < nd; ++d) {
        const int64_t row = dst_row[warp][d];
        uint8_t* dst = out + row * a.H;
#pragma unroll
        for (int u = 0; u < kPairs; ++u) {
          const int v = v0 + u * 64 + 2 * lane;
          if (v < vend) st_stream_v4(reinterpret_cast<int4*>(dst + (int64_t)v * 8),
                                     *reinterpret_cast<const int4*>(&qv[u]));
        }
        if (scale_lane) a.recv_scales[row * nblk + (v0 >> 4) + lane] = sc;
      }
    }
  }
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
  const int nvec = a.H / 8;
  const int unroll = fp8 ? kUnrollOf<true> : kUnrollOf<false>;
  const int max_slices = (nvec + 32 * unroll - 1) / (32 * unroll);
  const int64_t want_warps = (int64_t)props.sm_count * 64 * 4;
  int64_t ns = num_tokens > 0 ? (want_warps + num_tokens - 1) / num_tokens : 1;
  a.nslices = (int)(ns < 1 ? 1 : (ns > max_slices ? max_slices : ns));
  a.vps = ((nvec + a.nslices - 1) / a.nslices + 31) / 32 * 32;
  a.nslices = (nvec + a.vps - 1) / a.vps;  // no empty slice
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
  if (!routing_ok(num_tokens, num_topk, num_experts, num_ranks)) return EP_ERR_INVALID_ARG;
  if (hidden < 8 || hidden % 8 != 0 || (use_fp8 && hidden % 128 != 0)) return EP_ERR_INVALID_ARG;
  if (recv_capacity_rows < 0) return EP_ERR_INVALID_ARG;
  if (num_tokens > 0) {
    if (!x || !topk_idx || !slot || !recv_x) return EP_ERR_INVALID_ARG;
    if ((recv_topk_idx || recv_topk_weights) && !topk_weights) return EP_ERR_INVALID_ARG;
    if (use_fp8 && !recv_scales) return EP_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(recv_x)) return EP_ERR_INVALID_ARG;
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
    if (!x || !ll_slot || !recv_x || (use_fp8 && !recv_scales)) return EP_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(recv_x)) return EP_ERR_INVALID_ARG;
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
