// gdn_decode.cu — one-token gated-delta-rule update for a batch of decoding sequences.
//
// Each decoding sequence keeps its fp32 state in a caller-owned pool; the step reads the
// state once, applies one token of the recurrence (Gated Delta Networks, Yang, Kautz &
// Hatamizadeh, 2024) and writes it back in place: the "packed GDN decode" of vllm.cpp
// "vLLM, online serving" (lever 2b). The step is bound by HBM: every state byte is read
// and written once, nothing else is re-read.
//
// One block owns 32 rows of one (sequence, value head) state; 4 threads share a row and
// hold D/4 fp32 entries each, loaded and stored as float4 chunks c = sub + 4 m so a warp's
// 32 lanes touch 8 whole rows per instruction group.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 128;

template <typename T>
__device__ __forceinline__ float ld_f32(const T* p);
template <>
__device__ __forceinline__ float ld_f32<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void st_out(T* p, float x);
template <>
__device__ __forceinline__ void st_out<float>(float* p, float x) { *p = x; }
template <>
__device__ __forceinline__ void st_out<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) decode_kernel(DecodeArgs p) {
  constexpr int kVec = D / 16;
  __shared__ __align__(16) float sk[D];
  __shared__ __align__(16) float sq[D];
  const int tiles = D / 32;
  const int b = blockIdx.x / (p.hv_heads * tiles);
  const int rem = blockIdx.x % (p.hv_heads * tiles);
  const int h = rem / tiles;
  const int row0 = (rem % tiles) * 32;
  const int hk = h / p.group;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const T* q = static_cast<const T*>(p.q) + ((size_t)b * p.hk_heads + hk) * D;
  const T* k = static_cast<const T*>(p.k) + ((size_t)b * p.hk_heads + hk) * D;

  // this thread's state chunks first: their loads overlap warp 0's q/k work below
  const int r = tid >> 2, sub = tid & 3, row = row0 + r;
  const size_t slot = (size_t)p.slot[b];
  float4* srow = reinterpret_cast<float4*>(p.pool + ((slot * p.hv_heads + h) * D + row) * D);
  float4 S[kVec];
#pragma unroll
  for (int m = 0; m < kVec; ++m) S[m] = srow[sub + 4 * m];
  float ga = p.a[(size_t)b * p.hv_heads + h], bb = p.beta[(size_t)b * p.hv_heads + h];
  const float vi = ld_f32(static_cast<const T*>(p.v) + ((size_t)b * p.hv_heads + h) * D + row);
  if (warp == 0) {
    float qv[D / 32], kv[D / 32], qq = 0.f, kk = 0.f;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      qv[e] = ld_f32(q + lane + 32 * e);
      kv[e] = ld_f32(k + lane + 32 * e);
      qq += qv[e] * qv[e];
      kk += kv[e] * kv[e];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      qq += __shfl_xor_sync(0xffffffffu, qq, off);
      kk += __shfl_xor_sync(0xffffffffu, kk, off);
    }
    const float qs = p.l2norm ? rsqrtf(qq + kL2NormEps) : 1.f;
    const float ks = p.l2norm ? rsqrtf(kk + kL2NormEps) : 1.f;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      sq[lane + 32 * e] = qv[e] * qs;
      sk[lane + 32 * e] = kv[e] * ks;
    }
  }
  if (p.gate_mode == 1) gate_from_raw(p.a_log[h], p.dt_bias[h], ga, bb);
  const float g = __expf(ga);
  __syncthreads();

  const float4* kr = reinterpret_cast<const float4*>(sk);
  const float4* qr = reinterpret_cast<const float4*>(sq);
  float dot = 0.f;
#pragma unroll
  for (int m = 0; m < kVec; ++m) {
    const float4 k4 = kr[sub + 4 * m];
    S[m].x *= g; S[m].y *= g; S[m].z *= g; S[m].w *= g;
    dot += S[m].x * k4.x + S[m].y * k4.y + S[m].z * k4.z + S[m].w * k4.w;
  }
  dot += __shfl_xor_sync(0xffffffffu, dot, 1);
  dot += __shfl_xor_sync(0xffffffffu, dot, 2);
  const float delta = bb * (vi - dot);
  float outv = 0.f;
#pragma unroll
  for (int m = 0; m < kVec; ++m) {
    const float4 k4 = kr[sub + 4 * m];
    const float4 q4 = qr[sub + 4 * m];
    S[m].x += delta * k4.x; S[m].y += delta * k4.y;
    S[m].z += delta * k4.z; S[m].w += delta * k4.w;
    outv += S[m].x * q4.x + S[m].y * q4.y + S[m].z * q4.z + S[m].w * q4.w;
    srow[sub + 4 * m] = S[m];
  }
  outv += __shfl_xor_sync(0xffffffffu, outv, 1);
  outv += __shfl_xor_sync(0xffffffffu, outv, 2);
  if (sub == 0)
    st_out(static_cast<T*>(p.o) + ((size_t)b * p.hv_heads + h) * D + row, p.scale * outv);
}

}  // namespace

int launch_decode(const DecodeArgs& a, int head_dim, bool bf16, void* stream) {
  if (a.batch == 0) return 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int tiles = head_dim / 32;
  dim3 grid((unsigned)(a.batch * a.hv_heads * tiles)), block(kThreads);
  if (head_dim == 128) {
    if (bf16) decode_kernel<__nv_bfloat16, 128><<<grid, block, 0, s>>>(a);
    else decode_kernel<float, 128><<<grid, block, 0, s>>>(a);
  } else if (head_dim == 64) {
    if (bf16) decode_kernel<__nv_bfloat16, 64><<<grid, block, 0, s>>>(a);
    else decode_kernel<float, 64><<<grid, block, 0, s>>>(a);
  } else {
    return (int)cudaErrorInvalidValue;
  }
  return (int)cudaGetLastError();
}

}  // namespace gdn
