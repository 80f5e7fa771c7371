// umma_probe.cu — test-only check of the tcgen05 operand layouts, descriptors and TMEM
// access patterns used by the chunked prefill kernel: one M=128 MMA chain D = A B over
// K in steps of 16 with A and B in each layout the kernel uses, compared on the host
// with a plain matrix product. Built by tests/test_umma_probe_gpu.py.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../packed_linear_attention_gb300/csrc/ptx_sm103.cuh"

using namespace gdn::ptx;

namespace {

// mode bits: 1 = A MN-major (else K-major), 2 = B MN-major (else K-major), 4 = A in TMEM,
// 8 = negate B through the instruction descriptor.
__global__ void __launch_bounds__(128) probe_kernel(int mode, const __half* A, const __half* B,
                                                    float* D, int M, int N, int K,
                                                    int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                 // 32 KB
  uint8_t* sB = smem + 32768;         // 32 KB
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base_sh;
  const int tid = threadIdx.x, warp = tid >> 5;
  const bool a_mn = mode & 1, b_mn = mode & 2, a_tm = mode & 4, neg = mode & 8;

  // stage operands (A is M x K, B is K x N, both row-major in global memory)
  for (int i = tid; i < M * K; i += 128) {
    const int m = i / K, k = i % K;
    const uint32_t off = a_mn ? sw128_offset(k, m, K) : sw128_offset(m, k, M);
    *reinterpret_cast<__half*>(sA + off) = A[i];
  }
  for (int i = tid; i < K * N; i += 128) {
    const int k = i / N, n = i % N;
    const uint32_t off = b_mn ? sw128_offset(k, n, K) : sw128_offset(n, k, N);
    *reinterpret_cast<__half*>(sB + off) = B[i];
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, 256);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_sh;
  const uint32_t lane_off = (uint32_t)(32 * warp) << 16;

  if (a_tm) {  // A row m (thread m) packed two halves per column at columns 128..
    for (int c0 = 0; c0 < K / 2; c0 += 16) {
      uint32_t r[16];
      for (int j = 0; j < 16; ++j) {
        const __half lo = A[tid * K + 2 * (c0 + j)], hi = A[tid * K + 2 * (c0 + j) + 1];
        r[j] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
      }
      tmem_st16(tbase + lane_off + 128 + c0, r);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  if (tid == 0) {
    const uint32_t idesc = idesc_f16(M, N, a_mn ? 1 : 0, b_mn ? 1 : 0, 0, neg ? 1 : 0);
    for (int s = 0; s < K / 16; ++s) {
      uint64_t bd = b_mn ? smem_desc_sw128(smem_u32(sB) + s * 2048, K * 128, 1024)
                         : smem_desc_sw128(smem_u32(sB) + (s / 4) * (N * 128) + (s % 4) * 32,
                                           16, 1024);
      if (a_tm) {
        mma_f16_ts(tbase, tbase + 128 + s * 8, bd, idesc, s > 0);
      } else {
        uint64_t ad = a_mn ? smem_desc_sw128(smem_u32(sA) + s * 2048, K * 128, 1024)
                           : smem_desc_sw128(smem_u32(sA) + (s / 4) * (M * 128) + (s % 4) * 32,
                                             16, 1024);
        mma_f16_ss(tbase, ad, bd, idesc, s > 0);
      }
    }
    mma_commit(&bar);
  }
  __syncwarp();
  const bool ok = mbar_wait_bounded(&bar, 0, 1u << 26);
  tc_fence_after();
  if (!ok) {
    if (tid == 0) atomicExch(status, 1);
  } else {
    for (int c0 = 0; c0 < N; c0 += 16) {
      uint32_t r[16];
      tmem_ld16(tbase + lane_off + c0, r);
      tmem_ld_wait();
      for (int j = 0; j < 16; ++j) D[tid * N + c0 + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 256);
}

}  // namespace

extern "C" int umma_probe(int mode, const void* A, const void* B, float* D, int M, int N, int K,
                          int* status) {
  if (M != 128 || N < 16 || N > 128 || N % 16 || K < 16 || K > 128 || K % 64) return -1;
  const int smem = 65536 + 1024;
  cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  probe_kernel<<<1, 128, smem>>>(mode, static_cast<const __half*>(A),
                                 static_cast<const __half*>(B), D, M, N, K, status);
  cudaError_t e = cudaDeviceSynchronize();
  return e == cudaSuccess ? 0 : (int)e;
}
