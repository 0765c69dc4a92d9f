/*
 * ep_abi_client.c — a plain C caller of libep_gb300.so through include/ep_plan.h
 * (no Python, no C++): plan, BF16 dispatch, FP8 dispatch (quantised inside),
 * and the weighted combine of the dispatched rows, on the legacy default
 * stream.  Test driver for tests/test_gpu_c_abi.py, which writes the input
 * file, runs this program and compares what it writes with the oracle.
 *
 * usage: ep_abi_client IN OUT
 *   IN : int64 S, P, K, E, A, H; int64 topk_idx[T*K]; uint16 x[T*H] (bf16
 *        bits); float32 topk_weights[T*K]                 (T = P*S)
 *   OUT: int64 N_exp, N_recv; int32 slot[T*K]; int32 exp_src[N_exp];
 *        uint16 recv_bf16[N_exp*H]; uint8 recv_fp8[N_exp*H];
 *        float32 recv_scales[N_exp*H/128]; uint16 out[T*H]
 * Exit status 0 on success; otherwise a message on stderr.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ep_plan.h"

#define CHECK_CUDA(call)                                                           \
  do {                                                                             \
    cudaError_t e_ = (call);                                                       \
    if (e_ != cudaSuccess) {                                                       \
      fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #call, cudaGetErrorString(e_)); \
      exit(2);                                                                     \
    }                                                                              \
  } while (0)

#define CHECK_EP(call)                                                             \
  do {                                                                             \
    ep_status_t s_ = (call);                                                       \
    if (s_ != EP_OK) {                                                             \
      fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #call, ep_status_string(s_)); \
      exit(3);                                                                     \
    }                                                                              \
  } while (0)

static void read_all(FILE* f, void* dst, size_t bytes) {
  if (bytes && fread(dst, 1, bytes, f) != bytes) {
    fprintf(stderr, "short input\n");
    exit(4);
  }
}

static void write_all(FILE* f, const void* src, size_t bytes) {
  if (bytes && fwrite(src, 1, bytes, f) != bytes) {
    fprintf(stderr, "short output\n");
    exit(5);
  }
}

static void* dev_alloc(size_t bytes) {
  void* p = NULL;
  CHECK_CUDA(cudaMalloc(&p, bytes ? bytes : 16));
  return p;
}

static void* host_alloc(size_t bytes) {
  void* p = malloc(bytes ? bytes : 16);
  if (!p) {
    fprintf(stderr, "out of host memory\n");
    exit(6);
  }
  return p;
}

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s IN OUT\n", argv[0]);
    return 1;
  }
  FILE* in = fopen(argv[1], "rb");
  if (!in) {
    perror(argv[1]);
    return 1;
  }
  int64_t shape[6];
  read_all(in, shape, sizeof shape);
  const int64_t S = shape[0], H = shape[5];
  const int P = (int)shape[1], K = (int)shape[2], E = (int)shape[3], A = (int)shape[4];
  const int64_t T = (int64_t)P * S;
  int64_t* idx = host_alloc(sizeof(int64_t) * T * K);
  uint16_t* x = host_alloc(sizeof(uint16_t) * T * H);
  float* w = host_alloc(sizeof(float) * T * K);
  read_all(in, idx, sizeof(int64_t) * T * K);
  read_all(in, x, sizeof(uint16_t) * T * H);
  read_all(in, w, sizeof(float) * T * K);
  fclose(in);

  int64_t* idx_d = dev_alloc(sizeof(int64_t) * T * K);
  uint16_t* x_d = dev_alloc(sizeof(uint16_t) * T * H);
  float* w_d = dev_alloc(sizeof(float) * T * K);
  CHECK_CUDA(cudaMemcpy(idx_d, idx, sizeof(int64_t) * T * K, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(x_d, x, sizeof(uint16_t) * T * H, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(w_d, w, sizeof(float) * T * K, cudaMemcpyHostToDevice));

  /* the plan, and its exact sizes */
  ep_handle_t h = NULL;
  CHECK_EP(ep_plan(idx_d, S, P, K, E, A, 0, NULL, &h));
  int64_t n_exp = 0, n_recv = 0;
  CHECK_EP(ep_plan_sizes(h, NULL, &n_exp, &n_recv));

  /* dispatch into buffers of the worst-case size, zero padding */
  const int64_t cap = ep_worst_expanded_rows(T, K, E, A);
  if (cap < n_exp) {
    fprintf(stderr, "worst case %lld below N_exp %lld\n", (long long)cap, (long long)n_exp);
    return 7;
  }
  uint16_t* recv_d = dev_alloc(sizeof(uint16_t) * cap * H);
  uint8_t* q_d = dev_alloc((size_t)(cap * H));
  float* sc_d = dev_alloc(sizeof(float) * cap * (H / 128));
  CHECK_EP(ep_dispatch(h, x_d, EP_DTYPE_BF16, NULL, H, EP_DTYPE_BF16, EP_DISPATCH_ZERO_PAD, recv_d, NULL, cap, NULL));
  CHECK_EP(ep_dispatch(h, x_d, EP_DTYPE_BF16, NULL, H, EP_DTYPE_FP8_E4M3, EP_DISPATCH_ZERO_PAD, q_d, sc_d, cap, NULL));

  /* combine of the dispatched rows (the identity expert) */
  uint16_t* out_d = dev_alloc(sizeof(uint16_t) * T * H);
  CHECK_EP(ep_combine(h, recv_d, n_exp, w_d, NULL, H, out_d, NULL));
  CHECK_EP(ep_sync_status(h, NULL));

  /* plan arrays by their field pointers */
  const void* slot_d = NULL;
  const void* exp_src_d = NULL;
  int64_t shp[3];
  int nd = 0;
  CHECK_EP(ep_handle_get(h, EP_FIELD_SLOT, &slot_d, shp, &nd));
  CHECK_EP(ep_handle_get(h, EP_FIELD_EXP_SRC, &exp_src_d, shp, &nd));

  int32_t* slot = host_alloc(sizeof(int32_t) * T * K);
  int32_t* exp_src = host_alloc(sizeof(int32_t) * n_exp);
  uint16_t* recv = host_alloc(sizeof(uint16_t) * n_exp * H);
  uint8_t* q = host_alloc((size_t)(n_exp * H));
  float* sc = host_alloc(sizeof(float) * n_exp * (H / 128));
  uint16_t* out = host_alloc(sizeof(uint16_t) * T * H);
  CHECK_CUDA(cudaMemcpy(slot, slot_d, sizeof(int32_t) * T * K, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(exp_src, exp_src_d, sizeof(int32_t) * n_exp, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(recv, recv_d, sizeof(uint16_t) * n_exp * H, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(q, q_d, (size_t)(n_exp * H), cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(sc, sc_d, sizeof(float) * n_exp * (H / 128), cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(out, out_d, sizeof(uint16_t) * T * H, cudaMemcpyDeviceToHost));
  CHECK_EP(ep_handle_destroy(h, NULL));
  CHECK_CUDA(cudaDeviceSynchronize());

  FILE* o = fopen(argv[2], "wb");
  if (!o) {
    perror(argv[2]);
    return 1;
  }
  const int64_t sizes[2] = {n_exp, n_recv};
  write_all(o, sizes, sizeof sizes);
  write_all(o, slot, sizeof(int32_t) * T * K);
  write_all(o, exp_src, sizeof(int32_t) * n_exp);
  write_all(o, recv, sizeof(uint16_t) * n_exp * H);
  write_all(o, q, (size_t)(n_exp * H));
  write_all(o, sc, sizeof(float) * n_exp * (H / 128));
  write_all(o, out, sizeof(uint16_t) * T * H);
  fclose(o);

  cudaFree(idx_d);
  cudaFree(x_d);
  cudaFree(w_d);
  cudaFree(recv_d);
  cudaFree(q_d);
  cudaFree(sc_d);
  cudaFree(out_d);
  free(idx);
  free(x);
  free(w);
  free(slot);
  free(exp_src);
  free(recv);
  free(q);
  free(sc);
  free(out);
  return 0;
}
