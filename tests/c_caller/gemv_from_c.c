/* A caller of the library written in plain C (no Python, no torch): it reads the operands of one
 * batched GEMV from raw files, runs nvfp4_gemv_batched on a stream of its own through the C ABI,
 * and writes c (fp16 bits) to a file.  It also checks that a misaligned pointer is refused with
 * NVFP4_ERR_MISALIGNED before any device work, and that the planner answers for the shape.
 *
 * usage: gemv_from_c M K L g_a g_b A.bin sfa.bin b.bin sfb.bin c_out.bin
 * Exit status 0 on success; a message on stderr otherwise. */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "nvfp4_gemv.h"

static void* read_file(const char* path, size_t n) {
  FILE* f = fopen(path, "rb");
  void* p = malloc(n ? n : 1);
  if (!f || !p || fread(p, 1, n, f) != n) {
    fprintf(stderr, "cannot read %zu bytes from %s\n", n, path);
    exit(2);
  }
  fclose(f);
  return p;
}

static void* to_device(const void* host, size_t n) {
  void* d = NULL;
  if (cudaMalloc(&d, n ? n : 1) != cudaSuccess ||
      cudaMemcpy(d, host, n, cudaMemcpyHostToDevice) != cudaSuccess) {
    fprintf(stderr, "device copy of %zu bytes failed\n", n);
    exit(3);
  }
  return d;
}

int main(int argc, char** argv) {
  if (argc != 11) {
    fprintf(stderr, "usage: %s M K L g_a g_b A sfa b sfb c_out\n", argv[0]);
    return 1;
  }
  const int64_t M = atoll(argv[1]), K = atoll(argv[2]), L = atoll(argv[3]);
  const float g_a = (float)atof(argv[4]), g_b = (float)atof(argv[5]);
  const size_t nA = (size_t)(L * M * (K / 2)), nSA = (size_t)(L * M * (K / 16));
  const size_t nB = (size_t)(L * (K / 2)), nSB = (size_t)(L * (K / 16)), nC = (size_t)(L * M);
  void* hA = read_file(argv[6], nA);
  void* hSA = read_file(argv[7], nSA);
  void* hB = read_file(argv[8], nB);
  void* hSB = read_file(argv[9], nSB);
  const uint8_t* A = (const uint8_t*)to_device(hA, nA);
  const uint8_t* sfa = (const uint8_t*)to_device(hSA, nSA);
  const uint8_t* b = (const uint8_t*)to_device(hB, nB);
  const uint8_t* sfb = (const uint8_t*)to_device(hSB, nSB);
  uint16_t* c = NULL;
  if (cudaMalloc((void**)&c, 2 * nC) != cudaSuccess) return 3;

  nvfp4_plan plan;
  int st = nvfp4_gemv_plan(M, K, L, &plan);
  if (st != NVFP4_OK) {
    fprintf(stderr, "plan: %s (%s)\n", nvfp4_status_string(st), nvfp4_last_error());
    return 4;
  }
  /* a misaligned A: refused on the host, nothing enqueued (unless the shape takes the kernels
     that accept any alignment, which only happens for K % 256 != 0 here) */
  if (K % 256 == 0 && M * L >= 1) {
    nvfp4_plan forced = plan;
    forced.kernel = NVFP4_KERNEL_TMA;
    st = nvfp4_gemv_batched_ex(A + 1, sfa, g_a, b, sfb, g_b, c, M, K, L, 0, &forced);
    if (st != NVFP4_ERR_MISALIGNED) {
      fprintf(stderr, "misaligned A with a forced TMA plan gave status %d\n", st);
      return 5;
    }
  }
  cudaStream_t stream;
  if (cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking) != cudaSuccess) return 3;
  st = nvfp4_gemv_batched(A, sfa, g_a, b, sfb, g_b, c, M, K, L, stream);
  if (st != NVFP4_OK) {
    fprintf(stderr, "gemv: %s (%s)\n", nvfp4_status_string(st), nvfp4_last_error());
    return 6;
  }
  uint16_t* hC = (uint16_t*)malloc(2 * nC);
  if (!hC || cudaStreamSynchronize(stream) != cudaSuccess ||
      cudaMemcpy(hC, c, 2 * nC, cudaMemcpyDeviceToHost) != cudaSuccess) {
    fprintf(stderr, "gemv execution or copy-back failed\n");
    return 7;
  }
  FILE* f = fopen(argv[10], "wb");
  if (!f || fwrite(hC, 2, nC, f) != nC) return 8;
  fclose(f);
  printf("kernel %d, %d CTAs per batch, %d consumer warps\n", plan.kernel, plan.ctas_per_batch,
         plan.warps_per_cta);
  cudaStreamDestroy(stream);
  cudaFree((void*)A);
  cudaFree((void*)sfa);
  cudaFree((void*)b);
  cudaFree((void*)sfb);
  cudaFree(c);
  free(hA);
  free(hSA);
  free(hB);
  free(hSB);
  free(hC);
  return 0;
}
