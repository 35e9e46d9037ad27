/*
 * ep_oracle.c -- plain, slow, single-threaded CPU oracle for the MoE
 * expert-parallel token shuffle (get_dispatch_layout -> dispatch -> combine).
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. The CUDA library never
 * calls it, and the two share no code: this file includes nothing from the
 * CUDA sources and writes its own bfloat16 and FP8 E4M3 conversions from the
 * format definitions.
 *
 * Source: "[Not ready] MSCCLPP EP implementation" (mscclpp pull request 852).
 *   - Section "Scope", Intranode: get_dispatch_layout, intranode_dispatch and
 *     intranode_combine are DeepEP's high-throughput kernels with the
 *     torch::Tensor ABI preserved (per-rank / per-expert token counts and the
 *     is_token_in_rank mask).
 *   - The commit on the internode combine: combine runs in the reverse
 *     direction of dispatch and must use the receiver-side prefix matrices,
 *     i.e. slots are defined by prefix sums over (source rank, token order).
 *   - The intranode validation commit: every rank recovers its token
 *     payloads with "combine diff=0".
 *   - The low-latency port: dispatch<kUseFP8,...> optionally casts the
 *     payload to FP8.
 *   - The bench accounting commit: combine moves one copy per dispatched
 *     (token, rank) row back to its owner.
 * The pages name these steps but never write out their arithmetic. Where
 * they are silent, the plainest reading is taken (listed next to each
 * function).
 *
 * Notation: R ranks, T tokens (T % R == 0, T_r = T / R tokens per rank),
 * K top-k slots, E experts (E % R == 0, E_l = E / R experts per rank),
 * H hidden channels.  src(t) = t / T_r, rank(e) = e / E_l.
 *
 * Parity status: every function here is pinned by the CPU test suite
 * (brute force on tiny inputs, invariants, closed forms, and library
 * routines for the number formats).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEMORY 2

/* error bits reported for data problems (same meaning as the product's) */
#define ORACLE_ERR_BAD_EXPERT 1

/* ---------------------------------------------------------------------- */
/* bfloat16: sign bit, 8 exponent bits (bias 127), 7 fraction bits.         */
/* ---------------------------------------------------------------------- */

double oracle_bf16_to_double(uint16_t h) {
  int sign = h >> 15;
  int e = (h >> 7) & 0xFF;
  int m = h & 0x7F;
  double v;
  if (e == 0)
    v = ldexp((double)m, -126 - 7); /* subnormal: m * 2^-133 */
  else if (e == 0xFF)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(128 + m), e - 127 - 7); /* (1 + m/128) * 2^(e-127) */
  return sign ? -v : v;
}

/* Round a double to the nearest bfloat16, ties to even, in one rounding. */
uint16_t oracle_double_to_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int e = ilogb(a);                 /* 2^e <= a < 2^(e+1) */
  int q = (e < -126) ? -133 : e - 7; /* exponent of one unit in the last place */
  double M = rint(ldexp(a, -q));    /* ties to even (default rounding mode) */
  if (e < -126) {
    /* subnormal: the code is the integer significand; M == 128 is the
       smallest normal (exponent field 1, fraction 0), which is code 128 too */
    return sign | (uint16_t)M;
  }
  if (M == 256.0) { /* rounded up to the next binade */
    e += 1;
    M = 128.0;
  }
  int ef = e + 127;
  if (ef >= 0xFF) return sign | 0x7F80; /* overflow rounds to infinity */
  return sign | (uint16_t)(ef << 7) | (uint16_t)((int)M - 128);
}

/* ---------------------------------------------------------------------- */
/* FP8 E4M3 (OCP 8-bit floating point, E4M3 variant): sign bit, 4 exponent  */
/* bits (bias 7), 3 fraction bits; no infinities; S.1111.111 is NaN, so the */
/* largest finite value is 1.75 * 2^8 = 448; subnormals are m * 2^-9.       */
/* Conversion here: round to nearest even, saturating to +-448.             */
/* ---------------------------------------------------------------------- */

double oracle_e4m3_to_double(uint8_t c) {
  int sign = c >> 7;
  int e = (c >> 3) & 0xF;
  int m = c & 0x7;
  double v;
  if (e == 0xF && m == 0x7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp((double)(8 + m), e - 7 - 3);
  return sign ? -v : v;
}

uint8_t oracle_e4m3_from_float(float x) {
  uint8_t sign = signbit(x) ? 0x80 : 0;
  if (isnan(x)) return sign | 0x7F;
  double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E; /* saturate (also +-inf) */
  if (a == 0.0) return sign;
  int e = ilogb(a);
  if (e < -6) e = -6;                       /* subnormal range shares 2^-6's ulp */
  double M = rint(ldexp(a, 3 - e));         /* significand in units of 2^(e-3) */
  if (M == 16.0) { /* rounded up to the next binade */
    e += 1;
    M = 8.0;
  }
  if (M < 8.0) return sign | (uint8_t)M; /* subnormal: exponent field 0 */
  return sign | (uint8_t)((e + 7) << 3) | (uint8_t)((int)M - 8);
}

/* ---------------------------------------------------------------------- */
/* get_dispatch_layout + slot assignment                                    */
/* ---------------------------------------------------------------------- */

/*
 * From top-k routing to the layout of the receive buffers.
 *
 *   is_token_in_rank[t][r]     = 1 if some slot k of token t names an expert
 *                                e with rank(e) == r (masked slots, -1, and
 *                                ids outside [0,E) name nothing; the latter
 *                                also raise ORACLE_ERR_BAD_EXPERT)
 *   num_tokens_per_rank[s][r]  = sum over tokens t of source rank s of
 *                                is_token_in_rank[t][r]
 *   num_tokens_per_expert[s][e]= number of slots (t,k) with src(t) == s and
 *                                topk_idx[t][k] == e
 *   recv_base[r]               = exclusive prefix over destination ranks of
 *                                the tokens each receives; recv_base[R] = P
 *   rank_prefix[s][r]          = exclusive prefix over source ranks
 *   slot[t][r]                 = recv_base[r] + rank_prefix[src(t)][r]
 *                                + #{t' of src(t), t' < t, in rank r}
 *                                if is_token_in_rank[t][r], else -1
 *
 * Readings: experts are laid out contiguously per rank; the T tokens of one
 * call are the R ranks' tokens, rank s owning [s*T_r, (s+1)*T_r); within a
 * destination, rows are ordered by source rank and then by token, which is
 * the order the receiver-side prefix matrices describe; destinations are
 * packed one after the other into one buffer of P rows.
 */
int oracle_layout(const int64_t* topk_idx, int64_t T, int K, int E, int R,
                  uint8_t* is_token_in_rank, int32_t* num_tokens_per_rank,
                  int32_t* num_tokens_per_expert, int32_t* slot,
                  int32_t* recv_base, int32_t* err_bits) {
  if (T < 0 || K < 1 || E < 1 || R < 1 || E % R || T % R) return ORACLE_BAD_ARG;
  const int El = E / R;
  const int64_t Tr = T / R;
  *err_bits = 0;
  memset(num_tokens_per_rank, 0, sizeof(int32_t) * (size_t)R * R);
  memset(num_tokens_per_expert, 0, sizeof(int32_t) * (size_t)R * E);
  memset(is_token_in_rank, 0, (size_t)T * R);

  for (int64_t t = 0; t < T; ++t) {
    int64_t s = t / Tr;
    for (int k = 0; k < K; ++k) {
      int64_t e = topk_idx[t * K + k];
      if (e == -1) continue;
      if (e < -1 || e >= E) {
        *err_bits |= ORACLE_ERR_BAD_EXPERT;
        continue;
      }
      is_token_in_rank[t * R + e / El] = 1;
      num_tokens_per_expert[s * E + e] += 1;
    }
  }
  for (int64_t t = 0; t < T; ++t)
    for (int r = 0; r < R; ++r)
      num_tokens_per_rank[(t / Tr) * R + r] += is_token_in_rank[t * R + r];

  recv_base[0] = 0;
  for (int r = 0; r < R; ++r) {
    int64_t recv_count = 0;
    for (int s = 0; s < R; ++s) recv_count += num_tokens_per_rank[s * R + r];
    recv_base[r + 1] = (int32_t)(recv_base[r] + recv_count);
  }

  int32_t* rank_prefix = (int32_t*)calloc((size_t)R * R, sizeof(int32_t));
  int32_t* seen = (int32_t*)calloc((size_t)R * R, sizeof(int32_t));
  if (!rank_prefix || !seen) {
    free(rank_prefix);
    free(seen);
    return ORACLE_NO_MEMORY;
  }
  for (int r = 0; r < R; ++r)
    for (int s = 1; s < R; ++s)
      rank_prefix[s * R + r] = rank_prefix[(s - 1) * R + r] + num_tokens_per_rank[(s - 1) * R + r];

  for (int64_t t = 0; t < T; ++t) {
    int64_t s = t / Tr;
    for (int r = 0; r < R; ++r) {
      if (is_token_in_rank[t * R + r]) {
        slot[t * R + r] = recv_base[r] + rank_prefix[s * R + r] + seen[s * R + r];
        seen[s * R + r] += 1;
      } else {
        slot[t * R + r] = -1;
      }
    }
  }
  free(rank_prefix);
  free(seen);
  return ORACLE_OK;
}

/*
 * The sharded form: one rank's layout of its own T tokens over R
 * destination ranks ("Scope", Intranode: get_dispatch_layout runs on every
 * rank over its own tokens).  With one source, the definitions above become
 *   is_token_in_rank[t][r] as above
 *   send_counts[r]         = sum over t of is_token_in_rank[t][r]
 *   expert_counts[e]       = number of slots (t,k) with topk_idx[t][k] == e
 *   send_base[r]           = exclusive prefix of send_counts; send_base[R]
 *                            = rows of the send buffer
 *   send_slot[t][r]        = send_base[r] + #{t' < t in rank r}
 *                            if is_token_in_rank[t][r], else -1
 * (any T >= 0).  Reading: the send buffer is packed destination-major in
 * token order, so destination r's rows are one contiguous run; the receiver
 * stores the runs in source-rank order, which is the slot order above.
 */
int oracle_shard_layout(const int64_t* topk_idx, int64_t T, int K, int E, int R,
                        uint8_t* is_token_in_rank, int32_t* send_counts,
                        int32_t* expert_counts, int32_t* send_slot, int32_t* send_base,
                        int32_t* err_bits) {
  if (T < 0 || K < 1 || E < 1 || R < 1 || E % R) return ORACLE_BAD_ARG;
  const int El = E / R;
  *err_bits = 0;
  memset(send_counts, 0, sizeof(int32_t) * (size_t)R);
  memset(expert_counts, 0, sizeof(int32_t) * (size_t)E);
  memset(is_token_in_rank, 0, (size_t)T * R);
  for (int64_t t = 0; t < T; ++t) {
    for (int k = 0; k < K; ++k) {
      int64_t e = topk_idx[t * K + k];
      if (e == -1) continue;
      if (e < -1 || e >= E) {
        *err_bits |= ORACLE_ERR_BAD_EXPERT;
        continue;
      }
      is_token_in_rank[t * R + e / El] = 1;
      expert_counts[e] += 1;
    }
  }
  for (int64_t t = 0; t < T; ++t)
    for (int r = 0; r < R; ++r) send_counts[r] += is_token_in_rank[t * R + r];
  send_base[0] = 0;
  for (int r = 0; r < R; ++r) send_base[r + 1] = send_base[r] + send_counts[r];
  for (int r = 0; r < R; ++r) {
    int32_t seen = 0;
    for (int64_t t = 0; t < T; ++t) {
      if (is_token_in_rank[t * R + r])
        send_slot[t * R + r] = send_base[r] + seen++;
      else
        send_slot[t * R + r] = -1;
    }
  }
  return ORACLE_OK;
}

/* num_recv_tokens_per_expert[r][j]: slots that destination rank r receives
   for its local expert j, summed over source ranks. */
int oracle_num_recv_tokens_per_expert(const int32_t* num_tokens_per_expert, int E, int R,
                                      int32_t* out) {
  if (E < 1 || R < 1 || E % R) return ORACLE_BAD_ARG;
  const int El = E / R;
  for (int r = 0; r < R; ++r)
    for (int j = 0; j < El; ++j) {
      int64_t sum = 0;
      for (int s = 0; s < R; ++s) sum += num_tokens_per_expert[s * E + r * El + j];
      out[r * El + j] = (int32_t)sum;
    }
  return ORACLE_OK;
}

/* ---------------------------------------------------------------------- */
/* dispatch                                                                 */
/* ---------------------------------------------------------------------- */

/*
 * FP8 quantisation of one block of 128 channels (the kUseFP8 variant of the
 * low-latency dispatch).  Reading of the constants:
 *   amax  = max |x_i| over the block (float32, exact)
 *   a     = max(amax, 1e-4f)
 *   scale = a / 448           (one correctly rounded float32 division)
 *   inv   = 448 / a           (one correctly rounded float32 division)
 *   q_i   = E4M3_rne_satfinite(x_i * inv)  (one float32 multiply, no FMA)
 * The stored scale dequantises: x_i ~ q_i * scale.
 */
void oracle_quantize_block_e4m3(const uint16_t* x, int n, uint8_t* q, float* scale) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float v = (float)fabs(oracle_bf16_to_double(x[i]));
    if (v > amax) amax = v;
  }
  float a = amax > 1e-4f ? amax : 1e-4f;
  volatile float s = a / 448.0f;
  volatile float inv = 448.0f / a;
  for (int i = 0; i < n; ++i) {
    volatile float xi = (float)oracle_bf16_to_double(x[i]);
    volatile float p = xi * inv;
    q[i] = oracle_e4m3_from_float(p);
  }
  *scale = s;
}

/*
 * Dispatch tokens t in [t_begin, t_end) of T:
 *   recv_x[slot[t][r]]          = x[t]  (bf16 bits), or its E4M3 codes with
 *   recv_scales[slot[t][r]][b]  = the scale of channel block b (FP8 only)
 *   recv_src_idx[slot[t][r]]    = t
 *   recv_topk_idx[slot][k]      = e - r*E_l if rank(e) == r else -1
 *   recv_topk_weights[slot][k]  = w[t][k]   if rank(e) == r else 0
 * for every rank r with slot[t][r] >= 0.  Rows are written at their slot, so
 * the receive buffers must hold recv_base[R] rows.  With use_fp8 the caller
 * passes H % 128 == 0.  recv_x has H bytes per row for FP8, 2H otherwise.
 */
int oracle_dispatch(const uint16_t* x, int64_t T, int64_t H, const int64_t* topk_idx,
                    const float* topk_weights, int K, int E, int R, const int32_t* slot,
                    int64_t t_begin, int64_t t_end, int use_fp8, void* recv_x,
                    float* recv_scales, int32_t* recv_src_idx, int64_t* recv_topk_idx,
                    float* recv_topk_weights) {
  if (T < 0 || H < 1 || K < 1 || E < 1 || R < 1 || E % R) return ORACLE_BAD_ARG;
  if (t_begin < 0 || t_end > T || t_begin > t_end) return ORACLE_BAD_ARG;
  if (use_fp8 && H % 128) return ORACLE_BAD_ARG;
  const int El = E / R;
  const int64_t nb = H / 128;
  uint8_t* q = NULL;
  float* scales = NULL;
  if (use_fp8) {
    q = (uint8_t*)malloc((size_t)H);
    scales = (float*)malloc(sizeof(float) * (size_t)(nb ? nb : 1));
    if (!q || !scales) {
      free(q);
      free(scales);
      return ORACLE_NO_MEMORY;
    }
  }
  for (int64_t t = t_begin; t < t_end; ++t) {
    const uint16_t* row = x + t * H;
    if (use_fp8)
      for (int64_t b = 0; b < nb; ++b) oracle_quantize_block_e4m3(row + b * 128, 128, q + b * 128, scales + b);
    for (int r = 0; r < R; ++r) {
      int64_t p = slot[t * R + r];
      if (p < 0) continue;
      if (use_fp8) {
        memcpy((uint8_t*)recv_x + p * H, q, (size_t)H);
        memcpy(recv_scales + p * nb, scales, sizeof(float) * (size_t)nb);
      } else {
        memcpy((uint16_t*)recv_x + p * H, row, sizeof(uint16_t) * (size_t)H);
      }
      if (recv_src_idx) recv_src_idx[p] = (int32_t)t;
      for (int k = 0; k < K; ++k) {
        int64_t e = topk_idx[t * K + k];
        int here = (e >= 0 && e < E && e / El == r);
        if (recv_topk_idx) recv_topk_idx[p * K + k] = here ? e - (int64_t)r * El : -1;
        if (recv_topk_weights) recv_topk_weights[p * K + k] = here ? topk_weights[t * K + k] : 0.0f;
      }
    }
  }
  free(q);
  free(scales);
  return ORACLE_OK;
}

/* ---------------------------------------------------------------------- */
/* combine                                                                  */
/* ---------------------------------------------------------------------- */

/*
 * Combine tokens t in [t_begin, t_end):
 *   out[t][h] = bf16_rne( sum over unmasked k of w[t][k] * y[slot[t][rank(e_k)]][h] )
 * where y has dispatch's row layout (one expert-output row per (token, rank)
 * pair).  The sum is taken in float64 (exact products of a float32 and a
 * bfloat16, k ascending) and rounded once to bfloat16; a token with every
 * slot masked gives +0.  Reading: each top-k slot contributes its own
 * weighted copy of its rank's row, so a rank named twice counts twice.
 */
int oracle_combine(const uint16_t* y, int64_t H, const int64_t* topk_idx,
                   const float* topk_weights, int64_t T, int K, int E, int R,
                   const int32_t* slot, int64_t t_begin, int64_t t_end, uint16_t* out) {
  if (T < 0 || H < 1 || K < 1 || E < 1 || R < 1 || E % R) return ORACLE_BAD_ARG;
  if (t_begin < 0 || t_end > T || t_begin > t_end) return ORACLE_BAD_ARG;
  const int El = E / R;
  double* acc = (double*)malloc(sizeof(double) * (size_t)H);
  if (!acc) return ORACLE_NO_MEMORY;
  for (int64_t t = t_begin; t < t_end; ++t) {
    for (int64_t h = 0; h < H; ++h) acc[h] = 0.0;
    for (int k = 0; k < K; ++k) {
      int64_t e = topk_idx[t * K + k];
      if (e < 0 || e >= E) continue;
      int64_t p = slot[t * R + e / El];
      if (p < 0) continue; /* cannot happen for a consistent layout */
      double w = (double)topk_weights[t * K + k];
      const uint16_t* row = y + p * H;
      for (int64_t h = 0; h < H; ++h) acc[h] += w * oracle_bf16_to_double(row[h]);
    }
    for (int64_t h = 0; h < H; ++h) out[t * H + h] = oracle_double_to_bf16(acc[h]);
  }
  free(acc);
  return ORACLE_OK;
}

/*
 * Unweighted rank-sum combine for tokens t in [t_begin, t_end) (DeepEP's
 * high-throughput combine, where each receiving rank's expert stage has
 * already applied the top-k weights and summed its local experts):
 *   out[t][h] = bf16_rne( sum over ranks r with slot[t][r] >= 0 of y[slot[t][r]][h] )
 * Each destination rank's row is added once, in rank order, in float64; a
 * token sent nowhere gives +0.
 */
int oracle_combine_ranksum(const uint16_t* y, int64_t H, int64_t T, int R, const int32_t* slot,
                           int64_t t_begin, int64_t t_end, uint16_t* out) {
  if (T < 0 || H < 1 || R < 1) return ORACLE_BAD_ARG;
  if (t_begin < 0 || t_end > T || t_begin > t_end) return ORACLE_BAD_ARG;
  double* acc = (double*)malloc(sizeof(double) * (size_t)H);
  if (!acc) return ORACLE_NO_MEMORY;
  for (int64_t t = t_begin; t < t_end; ++t) {
    for (int64_t h = 0; h < H; ++h) acc[h] = 0.0;
    for (int r = 0; r < R; ++r) {
      int64_t p = slot[t * R + r];
      if (p < 0) continue;
      const uint16_t* row = y + p * H;
      for (int64_t h = 0; h < H; ++h) acc[h] += oracle_bf16_to_double(row[h]);
    }
    for (int64_t h = 0; h < H; ++h) out[t * H + h] = oracle_double_to_bf16(acc[h]);
  }
  free(acc);
  return ORACLE_OK;
}

/* ---------------------------------------------------------------------- */
/* low-latency (expert-major) layout                                        */
/* ---------------------------------------------------------------------- */

/*
 * The low-latency kernels' receive layout ("[Not ready] MSCCLPP EP
 * implementation", the low-latency port: dispatch<kUseFP8,...> and combine
 * address per-expert buffers, [local_expert * num_ranks + dst_rank]): every
 * unmasked top-k slot (t, k) gets its own row in the buffer of expert
 * e = topk_idx[t][k].  Expert e owns rows [e*cap, (e+1)*cap); inside it the
 * rows are packed by source rank, then by token, then by k:
 *   ll_slot[t][k]       = e*cap + ll_src_offset[e][src(t)]
 *                         + #{(t', k') of src(t) before (t, k), topk_idx[t'][k'] == e}
 *   ll_count[e]         = slots naming e (over all sources)
 *   ll_src_offset[e][s] = slots naming e from sources before s
 * Masked slots and ids outside [0, E) get -1 (the latter set the error bit);
 * a slot whose position is >= cap gets -1 and sets ORACLE_ERR_CAPACITY.
 */
#define ORACLE_ERR_CAPACITY 2
int oracle_ll_layout(const int64_t* topk_idx, int64_t T, int K, int E, int R, int64_t cap,
                     int32_t* ll_slot, int32_t* ll_count, int32_t* ll_src_offset,
                     int32_t* err_bits) {
  if (T < 0 || K < 1 || E < 1 || R < 1 || E % R || T % R || cap < 0) return ORACLE_BAD_ARG;
  const int64_t Tr = T / R;
  *err_bits = 0;
  int64_t* per_src = (int64_t*)calloc((size_t)E * R, sizeof(int64_t));  /* [e][s] */
  int64_t* seen = (int64_t*)calloc((size_t)E * R, sizeof(int64_t));
  if (!per_src || !seen) {
    free(per_src);
    free(seen);
    return ORACLE_NO_MEMORY;
  }
  for (int64_t t = 0; t < T; ++t)
    for (int k = 0; k < K; ++k) {
      int64_t e = topk_idx[t * K + k];
      if (e == -1) continue;
      if (e < -1 || e >= E) {
        *err_bits |= ORACLE_ERR_BAD_EXPERT;
        continue;
      }
      per_src[e * R + t / Tr] += 1;
    }
  for (int e = 0; e < E; ++e) {
    int64_t run = 0;
    for (int s = 0; s < R; ++s) {
      ll_src_offset[e * R + s] = (int32_t)run;
      run += per_src[e * R + s];
    }
    ll_count[e] = (int32_t)run;
  }
  for (int64_t t = 0; t < T; ++t) {
    const int64_t s = t / Tr;
    for (int k = 0; k < K; ++k) {
      int64_t e = topk_idx[t * K + k];
      if (e < 0 || e >= E) {
        ll_slot[t * K + k] = -1;
        continue;
      }
      int64_t pos = ll_src_offset[e * R + s] + seen[e * R + s];
      seen[e * R + s] += 1;
      if (pos >= cap) {
        ll_slot[t * K + k] = -1;
        *err_bits |= ORACLE_ERR_CAPACITY;
      } else {
        ll_slot[t * K + k] = (int32_t)(e * cap + pos);
      }
    }
  }
  free(per_src);
  free(seen);
  return ORACLE_OK;
}

/* Low-latency dispatch of tokens in [t_begin, t_end): recv_x[ll_slot[t][k]]
   = x[t] (bf16) or its E4M3 codes with recv_scales (per 128 channels, as in
   oracle_dispatch), recv_src_idx[ll_slot[t][k]] = t, for every slot >= 0. */
int oracle_ll_dispatch(const uint16_t* x, int64_t T, int64_t H, int K, const int32_t* ll_slot,
                       int64_t t_begin, int64_t t_end, int use_fp8, void* recv_x,
                       float* recv_scales, int32_t* recv_src_idx) {
  if (T < 0 || H < 1 || K < 1) return ORACLE_BAD_ARG;
  if (t_begin < 0 || t_end > T || t_begin > t_end) return ORACLE_BAD_ARG;
  if (use_fp8 && H % 128) return ORACLE_BAD_ARG;
  const int64_t nb = H / 128;
  uint8_t* q = NULL;
  float* scales = NULL;
  if (use_fp8) {
    q = (uint8_t*)malloc((size_t)H);
    scales = (float*)malloc(sizeof(float) * (size_t)(nb ? nb : 1));
    if (!q || !scales) {
      free(q);
      free(scales);
      return ORACLE_NO_MEMORY;
    }
  }
  for (int64_t t = t_begin; t < t_end; ++t) {
    const uint16_t* row = x + t * H;
    if (use_fp8)
      for (int64_t b = 0; b < nb; ++b) oracle_quantize_block_e4m3(row + b * 128, 128, q + b * 128, scales + b);
    for (int k = 0; k < K; ++k) {
      int64_t p = ll_slot[t * K + k];
      if (p < 0) continue;
      if (use_fp8) {
        memcpy((uint8_t*)recv_x + p * H, q, (size_t)H);
        memcpy(recv_scales + p * nb, scales, sizeof(float) * (size_t)nb);
      } else {
        memcpy((uint16_t*)recv_x + p * H, row, sizeof(uint16_t) * (size_t)H);
      }
      if (recv_src_idx) recv_src_idx[p] = (int32_t)t;
    }
  }
  free(q);
  free(scales);
  return ORACLE_OK;
}

/* Low-latency combine of tokens in [t_begin, t_end): out[t] = bf16_rne( sum
   over slots k with ll_slot[t][k] >= 0 of w[t][k] * y[ll_slot[t][k]] ), in
   float64, k ascending; with w == NULL every slot weighs 1. */
int oracle_ll_combine(const uint16_t* y, int64_t H, const float* w, int64_t T, int K,
                      const int32_t* ll_slot, int64_t t_begin, int64_t t_end, uint16_t* out) {
  if (T < 0 || H < 1 || K < 1) return ORACLE_BAD_ARG;
  if (t_begin < 0 || t_end > T || t_begin > t_end) return ORACLE_BAD_ARG;
  double* acc = (double*)malloc(sizeof(double) * (size_t)H);
  if (!acc) return ORACLE_NO_MEMORY;
  for (int64_t t = t_begin; t < t_end; ++t) {
    for (int64_t h = 0; h < H; ++h) acc[h] = 0.0;
    for (int k = 0; k < K; ++k) {
      int64_t p = ll_slot[t * K + k];
      if (p < 0) continue;
      double wk = w ? (double)w[t * K + k] : 1.0;
      const uint16_t* row = y + p * H;
      for (int64_t h = 0; h < H; ++h) acc[h] += wk * oracle_bf16_to_double(row[h]);
    }
    for (int64_t h = 0; h < H; ++h) out[t * H + h] = oracle_double_to_bf16(acc[h]);
  }
  free(acc);
  return ORACLE_OK;
}

/* Vector helpers so the number-format pins can sweep many values per call. */
void oracle_e4m3_from_float_n(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_from_float(x[i]);
}

void oracle_double_to_bf16_n(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_double_to_bf16(x[i]);
}

void oracle_bf16_to_double_n(const uint16_t* x, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_double(x[i]);
}

void oracle_e4m3_to_double_n(const uint8_t* x, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_double(x[i]);
}
