/*
 * Plain C use of libep.so: no PyTorch, only the CUDA runtime for memory.
 * Two ranks, 8 tokens (4 per rank), 4 experts (2 per rank), top-2.  The
 * expected layout is worked out by hand below; dispatch must copy each token
 * to its slots, and combine with identity experts and weights 0.5 + 0.5 must
 * return x exactly.  The sharded form's layout of one rank's tokens and its
 * host offsets are worked out by hand too.  Prints "ok" and exits 0 on
 * success.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "ep.h"

#define CHECK(cond, msg)                                   \
  do {                                                     \
    if (!(cond)) {                                         \
      fprintf(stderr, "FAILED: %s (line %d)\n", msg, __LINE__); \
      return 1;                                            \
    }                                                      \
  } while (0)

#define CUDA(call) CHECK((call) == cudaSuccess, #call)
#define EP(call) CHECK((call) == EP_OK, #call)

enum { T = 8, K = 2, E = 4, R = 2, H = 64 };

int main(void) {
  /* experts 0,1 live on rank 0 and experts 2,3 on rank 1 */
  const int64_t idx[T][K] = {{0, 1}, {2, 3}, {0, 2}, {-1, 3}, {1, 0}, {3, -1}, {-1, -1}, {2, 0}};
  const float w[T][K] = {{0.5f, 0.5f}, {0.5f, 0.5f}, {0.5f, 0.5f}, {0.0f, 1.0f},
                         {0.5f, 0.5f}, {1.0f, 0.0f}, {0.0f, 0.0f}, {0.5f, 0.5f}};
  /* by hand: token -> ranks it is sent to */
  const int in_rank[T][R] = {{1, 0}, {0, 1}, {1, 1}, {0, 1}, {1, 0}, {0, 1}, {0, 0}, {1, 1}};
  /* rank 0 receives tokens 0,2,4,7 (rows 0..3), rank 1 receives 1,2,3,5,7 (rows 4..8) */
  const int32_t want_slot[T][R] = {{0, -1}, {-1, 4}, {1, 5}, {-1, 6},
                                   {2, -1}, {-1, 7}, {-1, -1}, {3, 8}};
  const int32_t want_base[R + 1] = {0, 4, 9};
  uint16_t x[T][H];
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h) x[t][h] = (uint16_t)(0x3F80 + 8 * t + (h & 7)); /* bf16 ~ 1.0..1.5 */

  int64_t* d_idx; float* d_w; uint16_t* d_x; int32_t *d_ntpr, *d_ntpe, *d_slot, *d_base, *d_err;
  uint8_t* d_in; void* d_ws; uint16_t *d_recv, *d_out; int32_t* d_src;
  const size_t ws_bytes = ep_workspace_bytes(T, R, E);
  CHECK(ws_bytes > 0, "workspace size");
  const int cap = T * (K < R ? K : R);
  CUDA(cudaMalloc((void**)&d_idx, sizeof idx));
  CUDA(cudaMalloc((void**)&d_w, sizeof w));
  CUDA(cudaMalloc((void**)&d_x, sizeof x));
  CUDA(cudaMalloc((void**)&d_ntpr, sizeof(int32_t) * R * R));
  CUDA(cudaMalloc((void**)&d_ntpe, sizeof(int32_t) * R * E));
  CUDA(cudaMalloc((void**)&d_slot, sizeof(int32_t) * T * R));
  CUDA(cudaMalloc((void**)&d_base, sizeof(int32_t) * (R + 1)));
  CUDA(cudaMalloc((void**)&d_err, sizeof(int32_t)));
  CUDA(cudaMalloc((void**)&d_in, (size_t)T * R));
  CUDA(cudaMalloc(&d_ws, ws_bytes));
  CUDA(cudaMalloc((void**)&d_recv, sizeof(uint16_t) * cap * H));
  CUDA(cudaMalloc((void**)&d_src, sizeof(int32_t) * cap));
  CUDA(cudaMalloc((void**)&d_out, sizeof x));
  CUDA(cudaMemcpy(d_idx, idx, sizeof idx, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_w, w, sizeof w, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_x, x, sizeof x, cudaMemcpyHostToDevice));
  CUDA(cudaMemset(d_err, 0, sizeof(int32_t)));

  for (int path = EP_LAYOUT_MULTI_LAUNCH; path <= EP_LAYOUT_SINGLE_LAUNCH; ++path) {
    CUDA(cudaMemset(d_slot, 0x7F, sizeof(int32_t) * T * R)); /* poison */
    EP(ep_get_dispatch_layout_path(d_idx, T, K, E, R, d_ntpr, d_ntpe, d_in, d_slot, d_base, d_err,
                                   d_ws, ws_bytes, path, NULL));
    int32_t slot[T][R], base[R + 1], total = -1;
    uint8_t in[T][R];
    CUDA(cudaMemcpy(slot, d_slot, sizeof slot, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(base, d_base, sizeof base, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(in, d_in, sizeof in, cudaMemcpyDeviceToHost));
    EP(ep_layout_total_rows(d_base, R, &total, NULL));
    CHECK(total == 9, "P = 9 rows");
    CHECK(memcmp(slot, want_slot, sizeof slot) == 0, "slot table");
    CHECK(memcmp(base, want_base, sizeof base) == 0, "recv_base");
    for (int t = 0; t < T; ++t)
      for (int r = 0; r < R; ++r) CHECK(in[t][r] == in_rank[t][r], "is_token_in_rank");
  }

  EP(ep_dispatch(d_x, H, d_idx, d_w, T, K, E, R, d_slot, d_ntpe, cap, 0, d_recv, NULL, d_src, NULL,
                 NULL, NULL, d_err, NULL));
  uint16_t recv[T * (K < R ? K : R)][H];
  int32_t src[T * (K < R ? K : R)];
  CUDA(cudaMemcpy(recv, d_recv, sizeof recv, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(src, d_src, sizeof src, cudaMemcpyDeviceToHost));
  for (int t = 0; t < T; ++t)
    for (int r = 0; r < R; ++r)
      if (want_slot[t][r] >= 0) {
        CHECK(memcmp(recv[want_slot[t][r]], x[t], sizeof x[t]) == 0, "dispatched row");
        CHECK(src[want_slot[t][r]] == t, "recv_src_idx");
      }

  /* identity experts: y = recv; weights per token sum to 1 (token 6 has none) */
  EP(ep_combine(d_recv, H, d_idx, d_w, T, K, E, R, d_slot, d_out, d_err, NULL));
  uint16_t out[T][H];
  int32_t err = -1;
  CUDA(cudaMemcpy(out, d_out, sizeof out, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(&err, d_err, sizeof err, cudaMemcpyDeviceToHost));
  CHECK(err == 0, "device error word");
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h) CHECK(out[t][h] == (t == 6 ? 0 : x[t][h]), "combined row");

  /* the dynamically scheduled combine: counters zeroed once, zero again after each launch */
  uint64_t* d_sched;
  CUDA(cudaMalloc((void**)&d_sched, sizeof(uint64_t) * EP_COMBINE_SCHED_WORDS));
  CUDA(cudaMemset(d_sched, 0, sizeof(uint64_t) * EP_COMBINE_SCHED_WORDS));
  for (int rep = 0; rep < 2; ++rep) {
    CUDA(cudaMemset(d_out, 0xFF, sizeof x));
    EP(ep_combine_sched(d_recv, H, d_idx, d_w, T, K, E, R, d_slot, d_out, d_sched, d_err, NULL));
    uint16_t out2[T][H];
    uint64_t sched[EP_COMBINE_SCHED_WORDS];
    CUDA(cudaMemcpy(out2, d_out, sizeof out2, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(sched, d_sched, sizeof sched, cudaMemcpyDeviceToHost));
    CHECK(memcmp(out2, out, sizeof out) == 0, "scheduled combine");
    CHECK(sched[0] == 0 && sched[1] == 0, "counters back to zero");
  }

  /* the sharded form: rank 1 of 2 holds tokens 4..7 and lays them out alone.
     By hand: token 4 -> rank 0, 5 -> rank 1, 6 -> nowhere, 7 -> ranks 0 and 1,
     so its send buffer is [4, 7 | 5, 7]. */
  {
    enum { TS = 4 };
    int32_t *d_cnt, *d_ecnt, *d_sslot, *d_sbase;
    uint8_t* d_sin;
    void* d_sws;
    const size_t sws = ep_shard_workspace_bytes(TS, R, E);
    CHECK(sws > 0, "shard workspace size");
    CUDA(cudaMalloc((void**)&d_cnt, sizeof(int32_t) * R));
    CUDA(cudaMalloc((void**)&d_ecnt, sizeof(int32_t) * E));
    CUDA(cudaMalloc((void**)&d_sslot, sizeof(int32_t) * TS * R));
    CUDA(cudaMalloc((void**)&d_sbase, sizeof(int32_t) * (R + 1)));
    CUDA(cudaMalloc((void**)&d_sin, (size_t)TS * R));
    CUDA(cudaMalloc(&d_sws, sws));
    EP(ep_shard_layout(d_idx + 4 * K, TS, K, E, R, d_cnt, d_ecnt, d_sin, d_sslot, d_sbase, d_err,
                       d_sws, sws, NULL));
    int32_t sslot[TS][R], sbase[R + 1], cnt[R], ecnt[E];
    CUDA(cudaMemcpy(sslot, d_sslot, sizeof sslot, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(sbase, d_sbase, sizeof sbase, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(cnt, d_cnt, sizeof cnt, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(ecnt, d_ecnt, sizeof ecnt, cudaMemcpyDeviceToHost));
    const int32_t want_sslot[TS][R] = {{0, -1}, {-1, 2}, {-1, -1}, {1, 3}};
    const int32_t want_sbase[R + 1] = {0, 2, 4}, want_cnt[R] = {2, 2}, want_ecnt[E] = {2, 1, 1, 1};
    CHECK(memcmp(sslot, want_sslot, sizeof sslot) == 0, "send slots");
    CHECK(memcmp(sbase, want_sbase, sizeof sbase) == 0, "send_base");
    CHECK(memcmp(cnt, want_cnt, sizeof cnt) == 0, "send counts");
    CHECK(memcmp(ecnt, want_ecnt, sizeof ecnt) == 0, "expert counts");
    /* rank 0 (tokens 0..3) sends 2 tokens to itself and 3 to rank 1 */
    const int32_t counts[R][R] = {{2, 3}, {2, 2}};
    int64_t so[R + 1], ro[R + 1];
    EP(ep_shard_offsets(&counts[0][0], R, 1, so, ro));
    CHECK(so[0] == 0 && so[1] == 2 && so[2] == 4, "send offsets");
    /* rank 1 receives rank 0's 3 rows, then its own 2: rows 4..8 of the single-call layout */
    CHECK(ro[0] == 0 && ro[1] == 3 && ro[2] == 5, "receive offsets");
    const int32_t ec[R][E] = {{2, 1, 2, 2}, {2, 1, 1, 1}};
    int32_t per[E / R];
    EP(ep_shard_recv_tokens_per_expert(&ec[0][0], E, R, 1, per));
    CHECK(per[0] == 3 && per[1] == 3, "per-expert receive counts");
  }

  printf("ok\n");
  return 0;
}
