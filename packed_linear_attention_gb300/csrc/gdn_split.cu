// gdn_split.cu — state kernels of sequence splitting (prompts cut into segments that run
// in parallel).
//
// Over a segment the recurrence is affine in the segment's initial state: with the chunk
// form S <- S (gamma_L I - W^T diag(dec) K) + U^T diag(dec) K, a segment maps its initial
// state S0 to S0 M + B, where B is the segment's final state from a zero start and M its
// final state from the identity with v taken as zero. The split path runs every segment
// from those two starts in parallel, composes the maps in order here, and runs the
// segments once more from their true initial states.
//
//  * fill_states: the initial states of a pass (copies of the caller's, zeros, identities);
//  * compose_maps: per (split prompt, value head), S_start(p+1) = S_start(p) M_p + B_p in
//    fp32, in segment order;
//  * gather_states: final states from the passes' scratch into the caller's array.
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;

// One block per (state, value head): dst[i][h] = zero / identity / src[mode][h].
__global__ void __launch_bounds__(kThreads) fill_states_kernel(float* dst, const float* src,
                                                               const int32_t* mode, int hv,
                                                               int d) {
  const int i = blockIdx.x / hv, h = blockIdx.x % hv;
  const size_t per = (size_t)d * d;
  float* out = dst + ((size_t)i * hv + h) * per;
  const int m = mode[i];
  const float* in = m >= 0 && src ? src + ((size_t)m * hv + h) * per : nullptr;
  for (int e = threadIdx.x; e < d * d; e += kThreads) {
    float x = 0.f;
    if (in) x = in[e];
    else if (m == kSplitIdentity && e / d == e % d) x = 1.f;
    out[e] = x;
  }
}

// One block per (split prompt, value head); S and the current M in shared memory (fp32,
// 2 D x D). Thread t owns row t / (256 / D) and D^2 / 256 consecutive columns of S M.
template <int D>
__global__ void __launch_bounds__(kThreads) compose_maps_kernel(const SplitCompose* jobs,
                                                                const float* finals_a,
                                                                float* inits_c, int hv) {
  constexpr int kPerRow = kThreads / D, kCols = D / kPerRow;
  extern __shared__ float4 smem4[];
  float* S = reinterpret_cast<float*>(smem4);  // [D][D]
  float* M = S + D * D;                          // [D][D]
  const SplitCompose job = jobs[blockIdx.x / hv];
  const int h = blockIdx.x % hv;
  const size_t per = (size_t)D * D;
  const int tid = threadIdx.x, r = tid / kPerRow, c0 = kCols * (tid % kPerRow);
  auto state = [&](const float* base, int i) { return base + ((size_t)i * hv + h) * per; };
  auto state_mut = [&](float* base, int i) { return base + ((size_t)i * hv + h) * per; };

  // S = final state of segment 0 (run from the caller's initial state)
  const float4* s0 = reinterpret_cast<const float4*>(state(finals_a, job.first_final));
  for (int e = tid; e < D * D / 4; e += kThreads) reinterpret_cast<float4*>(S)[e] = s0[e];
  __syncthreads();
  for (int p = 1; p < job.num_segments; ++p) {
    // initial state of segment p
    float4* dst = reinterpret_cast<float4*>(state_mut(inits_c, job.first_init + p - 1));
    for (int e = tid; e < D * D / 4; e += kThreads)
      dst[e] = reinterpret_cast<const float4*>(S)[e];
    if (p + 1 == job.num_segments) break;
    // S <- S M_p + B_p (B_p at first_map + 2 (p - 1), M_p right after it)
    const float4* m =
        reinterpret_cast<const float4*>(state(finals_a, job.first_map + 2 * p - 1));
    for (int e = tid; e < D * D / 4; e += kThreads) reinterpret_cast<float4*>(M)[e] = m[e];
    __syncthreads();
    float acc[kCols];
#pragma unroll
    for (int j = 0; j < kCols; ++j) acc[j] = 0.f;
    for (int k = 0; k < D; ++k) {
      const float s = S[r * D + k];
      const float4* mrow = reinterpret_cast<const float4*>(M + k * D + c0);
#pragma unroll
      for (int j = 0; j < kCols / 4; ++j) {
        const float4 x = mrow[j];
        acc[4 * j] += s * x.x;
        acc[4 * j + 1] += s * x.y;
        acc[4 * j + 2] += s * x.z;
        acc[4 * j + 3] += s * x.w;
      }
    }
    const float* b = state(finals_a, job.first_map + 2 * p - 2) + (size_t)r * D + c0;
    __syncthreads();  // every read of S and M done
#pragma unroll
    for (int j = 0; j < kCols; ++j) S[r * D + c0 + j] = acc[j] + b[j];
    __syncthreads();
  }
}

// One block per (prompt, value head): dst[n][h] = src[index[n]][h], src chosen per prompt.
__global__ void __launch_bounds__(kThreads)
gather_states_kernel(float* dst, const float* src_a, const float* src_c, const int32_t* index,
                     int hv, int d) {
  const int n = blockIdx.x / hv, h = blockIdx.x % hv;
  const size_t per = (size_t)d * d;
  const int32_t i = index[n];
  const float* src = i >= 0 ? src_a + ((size_t)i * hv + h) * per
                            : src_c + ((size_t)(-1 - i) * hv + h) * per;
  float4* out = reinterpret_cast<float4*>(dst + ((size_t)n * hv + h) * per);
  const float4* in = reinterpret_cast<const float4*>(src);
  for (int e = threadIdx.x; e < d * d / 4; e += kThreads) out[e] = in[e];
}

}  // namespace

int launch_fill_states(float* dst, const float* src, const int32_t* mode, int count, int hv,
                       int d, void* stream) {
  if (count == 0) return 0;
  fill_states_kernel<<<count * hv, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      dst, src, mode, hv, d);
  return (int)cudaGetLastError();
}

int launch_compose_maps(const SplitCompose* jobs, int num_jobs, const float* finals_a,
                        float* inits_c, int hv, int d, void* stream) {
  if (num_jobs == 0) return 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int smem = 2 * d * d * (int)sizeof(float);
  if (d == 128) {
    static bool configured = false;
    if (!configured) {
      const cudaError_t e = cudaFuncSetAttribute(
          compose_maps_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return (int)e;
      configured = true;
    }
    compose_maps_kernel<128><<<num_jobs * hv, kThreads, smem, st>>>(jobs, finals_a, inits_c,
                                                                    hv);
  } else if (d == 64) {
    compose_maps_kernel<64><<<num_jobs * hv, kThreads, smem, st>>>(jobs, finals_a, inits_c,
                                                                   hv);
  } else {
    return (int)cudaErrorInvalidValue;
  }
  return (int)cudaGetLastError();
}

int launch_gather_states(float* dst, const float* src_a, const float* src_c,
                         const int32_t* index, int num_seqs, int hv, int d, void* stream) {
  if (num_seqs == 0) return 0;
  gather_states_kernel<<<num_seqs * hv, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      dst, src_a, src_c, index, hv, d);
  return (int)cudaGetLastError();
}

}  // namespace gdn
