// ep_scatter.cuh -- one warp's share of the token scatter, shared by the
// dispatch kernel (ep_dispatch.cu) and the fused layout + dispatch kernel
// (ep_fused.cu).
//
// "[Not ready] MSCCLPP EP implementation" (mscclpp pull request 852):
// section "Scope", Intranode (intranode_dispatch), and the low-latency port
// (dispatch<kUseFP8,...>, the FP8 payload cast).  A warp handles one token,
// or one slice of a token's row (a multiple of 32 16-byte vectors): it
// finds the token's destination rows, writes the per-row metadata (slice 0)
// and copies or quantises its slice into every destination row.
//
// Lanes hold 16-byte vectors of the row (8 bf16 channels); kUnroll vectors
// per lane are loaded before the stores, so each warp keeps 16 x 512 bytes
// (bf16) or 4 x 512 bytes (FP8) of reads in flight.  Loads bypass L1, stores
// use the streaming policy.  In the FP8 variant each lane holds two adjacent
// vectors and 8 lanes hold one block of 128 channels: its amax is taken on
// the raw bf16 bits (per-halfword unsigned max of |x|, then a 3-step
// xor-shuffle), one lane per block computes the block's two divisions (a
// warp's 8 blocks in one instruction sequence), and the block is quantised
// in registers and written to every destination in 16-byte stores, with the
// 8 scales of a round in one 32-byte run.  The quantiser rounds exactly as
// the format definition requires: 448/a and a/448 are single correctly
// rounded divisions (__fdiv_rn), x * (448/a) is a single multiply
// (__fmul_rn), and the E4M3 conversion is the hardware's
// round-to-nearest-even, saturate-to-finite conversion.
#pragma once

#include <cuda_fp8.h>

#include "ep_common.cuh"

namespace ep {

// 16-byte vectors each lane loads before it stores them: 16 for the bf16
// copy (a whole 4096-channel row per warp in flight; measured faster than 8
// and 4 although it leaves 2 blocks per SM), 4 for the FP8 kernel, whose
// quantiser needs the registers.
template <bool kFP8>
constexpr int kUnrollOf = kFP8 ? 4 : 16;

struct ScatterArgs {
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

// Destinations of token t, in column order: the entries of dest[t][.] that
// are >= 0 go to dst_row (their row) and dst_rank (their column); an entry
// at or beyond the capacity is skipped and sets EP_ERRBIT_CAPACITY.
// Returns their number.  dst_row / dst_rank: this warp's shared arrays.
__device__ __forceinline__ int warp_dest_list(const ScatterArgs& a, int64_t t, int lane,
                                              int32_t* dst_row, int32_t* dst_rank) {
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
      dst_row[pos] = sl;
      dst_rank[pos] = r;
    }
    nd += __popc(bal);
  }
  if (__any_sync(0xFFFFFFFFu, over) && lane == 0 && a.err) atomicOr(a.err, EP_ERRBIT_CAPACITY);
  __syncwarp();
  return nd;
}

// Per-row metadata of token t's nd rows: the source token, and the top-k
// entries that are local to the destination (local expert id and weight),
// -1 / 0 elsewhere.
__device__ __forceinline__ void warp_write_meta(const ScatterArgs& a, int64_t t, int nd,
                                                const int32_t* dst_row, const int32_t* dst_rank,
                                                int lane) {
  if (!a.rank_meta && a.recv_src_idx) {
    for (int d = lane; d < nd; d += 32) a.recv_src_idx[dst_row[d]] = (int32_t)t;
  }
  if (a.rank_meta && (a.recv_src_idx || a.recv_topk_idx || a.recv_topk_w)) {
    // keep the small metadata rows in L2 (evict-last) until neighbouring
    // rows, written by other warps, have filled their sectors
    const uint64_t keep = l2_policy_evict_last();
    const int64_t e = lane < a.K ? a.topk_idx[t * a.K + lane] : -1;
    const float w = (lane < a.K && a.topk_w) ? a.topk_w[t * a.K + lane] : 0.0f;
    const int er = (e >= 0 && e < a.E) ? (int)(e / a.El) : -1;
    for (int d = 0; d < nd; ++d) {
      const int64_t row = dst_row[d];
      const int r = dst_rank[d];
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
}

// One round of a warp's slice: kUnroll vectors per lane of the source row.
template <bool kFP8>
struct Round {
  int4 v[kUnrollOf<kFP8>];
};

// Loads the round starting at vector v0 (vectors at or beyond vend are left
// out: bf16 keeps them unset and never stores them, FP8 reads zeros).
template <bool kFP8>
__device__ __forceinline__ void load_round(const int4* src, int v0, int vend, int lane,
                                           Round<kFP8>& r) {
  constexpr int kUnroll = kUnrollOf<kFP8>;
  if constexpr (!kFP8) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = v0 + u * 32 + lane;
      if (v < vend) r.v[u] = ld_stream_v4(src + v);
    }
  } else {
#pragma unroll
    for (int u = 0; u < kUnroll / 2; ++u) {
      const int v = v0 + u * 64 + 2 * lane;
      const bool in = v < vend;
      r.v[2 * u] = in ? ld_stream_v4(src + v) : make_int4(0, 0, 0, 0);
      r.v[2 * u + 1] = in ? ld_stream_v4(src + v + 1) : make_int4(0, 0, 0, 0);
    }
  }
}

// Writes one loaded round to the token's nd destination rows: a bf16 copy,
// or the FP8 codes and the round's scales.
template <bool kFP8>
__device__ __forceinline__ void store_round(const ScatterArgs& a, const Round<kFP8>& r, int v0,
                                            int vend, int nd, const int32_t* dst_row, int lane) {
  constexpr int kUnroll = kUnrollOf<kFP8>;
  const int nvec = a.H / 8;
  if constexpr (!kFP8) {
    int4* out = reinterpret_cast<int4*>(a.recv_x);
    for (int d = 0; d < nd; ++d) {
      int4* dst = out + (int64_t)dst_row[d] * nvec;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < vend) st_stream_v4(dst + v, r.v[u]);
      }
    }
  } else {
    // Each lane holds two adjacent vectors (16 channels), so a 128-channel
    // block is 8 lanes and its 16 E4M3 codes per lane go out in one 16-byte
    // store.  H % 128 == 0 and slices of a multiple of 32 vectors make blocks
    // wholly in or out of the slice.
    uint8_t* out = reinterpret_cast<uint8_t*>(a.recv_x);
    const int nblk = a.H / 128;
    constexpr int kPairs = kUnroll / 2;  // vector pairs per lane and round
    uint32_t mbits[kPairs];              // amax of the lane's block, as bf16 bits
#pragma unroll
    for (int u = 0; u < kPairs; ++u) {
      // for finite bf16 the order of |x| is the unsigned order of the low
      // 15 bits, so a per-halfword unsigned max gives the exact amax bits
      const int4& p = r.v[2 * u];
      const int4& q = r.v[2 * u + 1];
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
    static_assert(kPairs == 2, "the division lanes below assume two vector pairs per lane");
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
      unpack_bf16x8(r.v[2 * u], f);
      qv[u].x = cvt_e4m3x4(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv), __fmul_rn(f[2], inv),
                           __fmul_rn(f[3], inv));
      qv[u].y = cvt_e4m3x4(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv), __fmul_rn(f[6], inv),
                           __fmul_rn(f[7], inv));
      unpack_bf16x8(r.v[2 * u + 1], f);
      qv[u].z = cvt_e4m3x4(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv), __fmul_rn(f[2], inv),
                           __fmul_rn(f[3], inv));
      qv[u].w = cvt_e4m3x4(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv), __fmul_rn(f[6], inv),
                           __fmul_rn(f[7], inv));
    }
    // lanes 0..7 hold the round's 8 scales in row order
    const bool scale_lane = lane < 8 && v0 + 16 * lane < vend;
    for (int d = 0; d < nd; ++d) {
      const int64_t row = dst_row[d];
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

// The warp's slice [vbeg, vend) of token row `src`, written to its nd
// destination rows round by round; `first` holds the round at vbeg, already
// loaded by the caller.
template <bool kFP8>
__device__ __forceinline__ void warp_scatter(const ScatterArgs& a, const int4* src, int vbeg,
                                             int vend, int nd, const int32_t* dst_row, int lane,
                                             const Round<kFP8>& first) {
  constexpr int kStep = 32 * kUnrollOf<kFP8>;
  store_round<kFP8>(a, first, vbeg, vend, nd, dst_row, lane);
  for (int v0 = vbeg + kStep; v0 < vend; v0 += kStep) {
    Round<kFP8> r;
    load_round<kFP8>(src, v0, vend, lane, r);
    store_round<kFP8>(a, r, v0, vend, nd, dst_row, lane);
  }
}

// Slices of a token's row so that a batch of T tokens makes about four
// waves of 64 warps per SM: a.nslices warps per token, a.vps vectors each
// (a multiple of 32, one or more rounds of 32 * kUnroll).
inline void plan_slices(ScatterArgs& a, bool fp8, int sm_count) {
  const int nvec = a.H / 8;
  const int unroll = fp8 ? kUnrollOf<true> : kUnrollOf<false>;
  const int max_slices = (nvec + 32 * unroll - 1) / (32 * unroll);
  const int64_t want_warps = (int64_t)sm_count * 64 * 4;
  const int64_t ns = a.T > 0 ? (want_warps + a.T - 1) / a.T : 1;
  a.nslices = (int)(ns < 1 ? 1 : (ns > max_slices ? max_slices : ns));
  a.vps = ((nvec + a.nslices - 1) / a.nslices + 31) / 32 * 32;
  a.nslices = (nvec + a.vps - 1) / a.vps;  // no empty slice
}

}  // namespace ep
