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
//  * compose_maps: per (split prompt, value head, block of rows),
//    S_start(p+1) = S_start(p) M_p + B_p in fp32, in segment order;
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

// Rows of S M + B depend only on the same rows of S, so one block owns kRows rows of S for
// one (split prompt, value head): grid = jobs x heads x D / kRows. Shared memory holds the
// block's rows of S and the whole current M (fp32). Thread t owns kRpt rows and the 4
// columns 4 (t mod D/4) .. +3: at D = 128 a warp reads one S entry (broadcast) and 512
// contiguous bytes of an M row per k. Each entry sums its products from zero in k order
// and then adds B's.
constexpr int kRows = 16;

template <int D>
__global__ void __launch_bounds__(kThreads) compose_maps_kernel(const SplitCompose* jobs,
                                                                const float* finals_a,
                                                                float* inits_c, int hv) {
  constexpr int kGroups = D / 4, kRpt = kRows * kGroups / kThreads;
  constexpr int kBlocks = D / kRows;
  extern __shared__ float4 smem4[];
  float* M = reinterpret_cast<float*>(smem4);  // [D][D]
  float* S = M + D * D;                          // [kRows][D]
  const int per_job = hv * kBlocks;
  const SplitCompose job = jobs[blockIdx.x / per_job];
  const int h = (blockIdx.x % per_job) / kBlocks, row0 = (blockIdx.x % kBlocks) * kRows;
  const size_t per = (size_t)D * D;
  const int tid = threadIdx.x, cg = tid % kGroups, rg = tid / kGroups;
  auto state = [&](const float* base, int i) { return base + ((size_t)i * hv + h) * per; };
  auto rows = [&](int i) { return row0 * D + i; };  // offset of this block's rows

  // S = final state of segment 0 (run from the caller's initial state), this block's rows
  const float4* s0 = reinterpret_cast<const float4*>(state(finals_a, job.first_final) + rows(0));
  for (int e = tid; e < kRows * D / 4; e += kThreads) reinterpret_cast<float4*>(S)[e] = s0[e];
  __syncthreads();
  for (int p = 1; p < job.num_segments; ++p) {
    // initial state of segment p
    float4* dst = reinterpret_cast<float4*>(
        const_cast<float*>(state(inits_c, job.first_init + p - 1)) + rows(0));
    for (int e = tid; e < kRows * D / 4; e += kThreads)
      dst[e] = reinterpret_cast<const float4*>(S)[e];
    if (p + 1 == job.num_segments) break;
    // S <- S M_p + B_p (B_p at first_map + 2 (p - 1), M_p right after it)
    const float4* m =
        reinterpret_cast<const float4*>(state(finals_a, job.first_map + 2 * p - 1));
    for (int e = tid; e < D * D / 4; e += kThreads) smem4[e] = m[e];
    const float* b = state(finals_a, job.first_map + 2 * p - 2) + rows(0);
    float4 acc[kRpt], bv[kRpt];
#pragma unroll
    for (int i = 0; i < kRpt; ++i) {
      bv[i] = reinterpret_cast<const float4*>(b + (rg * kRpt + i) * D)[cg];
      acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
#pragma unroll 4
    for (int k = 0; k < D; ++k) {
      const float4 x = reinterpret_cast<const float4*>(M + k * D)[cg];
#pragma unroll
      for (int i = 0; i < kRpt; ++i) {
        const float sv = S[(rg * kRpt + i) * D + k];
        acc[i].x += sv * x.x;
        acc[i].y += sv * x.y;
        acc[i].z += sv * x.z;
        acc[i].w += sv * x.w;
      }
    }
    __syncthreads();  // every read of S and M done
#pragma unroll
    for (int i = 0; i < kRpt; ++i)
      reinterpret_cast<float4*>(S + (rg * kRpt + i) * D)[cg] =
          make_float4(acc[i].x + bv[i].x, acc[i].y + bv[i].y, acc[i].z + bv[i].z,
                      acc[i].w + bv[i].w);
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
  const int smem = (d * d + kRows * d) * (int)sizeof(float);
  const unsigned grid = (unsigned)(num_jobs * hv * (d / kRows));
  if (d == 128) {
    static std::atomic<int> configured[kMaxDevices];
    const int ce = configure_once(configured, [smem] {
      return (int)cudaFuncSetAttribute(compose_maps_kernel<128>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (ce != 0) return ce;
    compose_maps_kernel<128><<<grid, kThreads, smem, st>>>(jobs, finals_a, inits_c, hv);
  } else if (d == 64) {
    compose_maps_kernel<64><<<grid, kThreads, smem, st>>>(jobs, finals_a, inits_c, hv);
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
