/*
 * A client of the library written in plain C99 against include/cpattn.h
 * and the CUDA runtime API: no Python, no C++. tests/test_c_client.py
 * builds and runs it.
 *
 *   c_abi_client                      host-only calls (no device needed)
 *   c_abi_client gpu DIR b s hq hkv d cp
 *       reads DIR/q.bin, k.bin, v.bin, do.bin (bf16, [b, s, h, d]),
 *       runs cpattn_fwd and cpattn_bwd on device buffers it allocates, and
 *       writes DIR/o.bin (bf16), lse.bin (fp32 [b, hq, s]), dq.bin, dk.bin,
 *       dv.bin (bf16).
 * Prints one line per check; exits non-zero on the first failure.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "cpattn.h"

static int fail(const char* what, int rc) {
  fprintf(stderr, "FAIL %s: %d (%s)\n", what, rc, cpattn_strerror(rc));
  return 1;
}

static int host_checks(void) {
  int64_t idx[8];
  int rc;
  printf("version %d\n", cpattn_version());
  /* s = 8, cp = 2: rank 0 holds chunks 0 and 3, rank 1 chunks 1 and 2 */
  rc = cpattn_zigzag_index(8, 2, idx);
  if (rc) return fail("cpattn_zigzag_index", rc);
  printf("zigzag %lld %lld %lld %lld %lld %lld %lld %lld\n", (long long)idx[0], (long long)idx[1],
         (long long)idx[2], (long long)idx[3], (long long)idx[4], (long long)idx[5], (long long)idx[6],
         (long long)idx[7]);
  /* argument errors come back before any device work */
  rc = cpattn_fwd(NULL, NULL, NULL, NULL, NULL, 1, 256, 2, 2, 64, 2, 1, NULL);
  printf("null pointers -> %d %s\n", rc, cpattn_strerror(rc));
  if (rc != CPATTN_ERR_NULL_PTR) return 1;
  rc = cpattn_zigzag_index(10, 3, idx);
  printf("s not divisible by 2cp -> %d %s\n", rc, cpattn_strerror(rc));
  if (rc != CPATTN_ERR_INVALID_ARG) return 1;
  printf("bwd workspace for b1 s4096 h8/2 d128 cp4: %zu bytes\n", cpattn_bwd_workspace_bytes(1, 4096, 8, 2, 128, 4));
  return 0;
}

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* buf = malloc(bytes);
  if (buf && fread(buf, 1, bytes, f) != bytes) {
    free(buf);
    buf = NULL;
  }
  fclose(f);
  return buf;
}

static int write_file(const char* dir, const char* name, const void* buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  const int bad = fwrite(buf, 1, bytes, f) != bytes;
  fclose(f);
  return bad;
}

static int gpu_run(const char* dir, int b, int s, int hq, int hkv, int d, int cp) {
  const size_t nq = (size_t)b * s * hq * d * 2, nk = (size_t)b * s * hkv * d * 2, nl = (size_t)b * hq * s * 4;
  const char* in_names[4] = {"q.bin", "k.bin", "v.bin", "do.bin"};
  const size_t in_bytes[4] = {nq, nk, nk, nq};
  void* host[4];
  void* dev_in[4];
  void *o, *lse, *dq, *dk, *dv, *ws;
  int status = 0, rc, i;
  const size_t nws = cpattn_bwd_workspace_bytes(b, s, hq, hkv, d, cp);
  if (nws == 0) return fail("cpattn_bwd_workspace_bytes", CPATTN_ERR_INVALID_ARG);
  for (i = 0; i < 4; ++i) {
    host[i] = read_file(dir, in_names[i], in_bytes[i]);
    if (!host[i]) return fail(in_names[i], -100);
    if (cudaMalloc(&dev_in[i], in_bytes[i]) != cudaSuccess) return fail("cudaMalloc", -101);
    if (cudaMemcpy(dev_in[i], host[i], in_bytes[i], cudaMemcpyHostToDevice) != cudaSuccess)
      return fail("cudaMemcpy", -102);
  }
  if (cudaMalloc(&o, nq) || cudaMalloc(&lse, nl) || cudaMalloc(&dq, nq) || cudaMalloc(&dk, nk) ||
      cudaMalloc(&dv, nk) || cudaMalloc(&ws, nws))
    return fail("cudaMalloc", -101);
  rc = cpattn_fwd(dev_in[0], dev_in[1], dev_in[2], o, (float*)lse, b, s, hq, hkv, d, cp, 1, NULL);
  if (rc) return fail("cpattn_fwd", rc);
  rc = cpattn_bwd(dev_in[0], dev_in[1], dev_in[2], o, (const float*)lse, dev_in[3], dq, dk, dv, ws, nws, b, s, hq,
                  hkv, d, cp, 1, NULL);
  if (rc) return fail("cpattn_bwd", rc);
  rc = cpattn_device_status(NULL, &status);
  if (rc || status) return fail("cpattn_device_status", status);
  {
    void* out[5];
    const char* out_names[5] = {"o.bin", "lse.bin", "dq.bin", "dk.bin", "dv.bin"};
    void* out_dev[5] = {o, lse, dq, dk, dv};
    const size_t out_bytes[5] = {nq, nl, nq, nk, nk};
    for (i = 0; i < 5; ++i) {
      out[i] = malloc(out_bytes[i]);
      if (!out[i] || cudaMemcpy(out[i], out_dev[i], out_bytes[i], cudaMemcpyDeviceToHost) != cudaSuccess)
        return fail("cudaMemcpy", -102);
      if (write_file(dir, out_names[i], out[i], out_bytes[i])) return fail(out_names[i], -103);
      free(out[i]);
    }
  }
  for (i = 0; i < 4; ++i) {
    cudaFree(dev_in[i]);
    free(host[i]);
  }
  cudaFree(o);
  cudaFree(lse);
  cudaFree(dq);
  cudaFree(dk);
  cudaFree(dv);
  cudaFree(ws);
  printf("gpu run ok\n");
  return 0;
}

int main(int argc, char** argv) {
  if (host_checks()) return 1;
  if (argc >= 9 && strcmp(argv[1], "gpu") == 0)
    return gpu_run(argv[2], atoi(argv[3]), atoi(argv[4]), atoi(argv[5]), atoi(argv[6]), atoi(argv[7]),
                   atoi(argv[8]));
  return 0;
}
