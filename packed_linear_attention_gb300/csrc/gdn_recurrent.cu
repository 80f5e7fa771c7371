// gdn_recurrent.cu — token-serial gated-delta-rule prefill on CUDA cores (fp32 state).
//
// The general path: any io dtype (fp32 or bf16), head dims 64 or 128, any GQA group. It
// evaluates the recurrence of Gated Delta Networks (Yang, Kautz & Hatamizadeh, 2024) one
// token at a time, exactly in the order of the definition:
//     S <- g S;  delta = beta (v - S k);  S <- S + delta k^T;  o = scale S q
// over packed prompts with per-prompt initial states and prefix-cache checkpoints
// (sparkinfer v0.6.28 release notes: packed passes, checkpoint bullets).
//
// Decomposition: rows of S (the value dim) evolve independently, so one block owns
// 32 rows of one (prompt, value head) pair; 4 threads share a row, each holding D/4
// state entries in registers in fp32. Tokens are staged 32 at a time in shared memory,
// with q and k L2-normalised once per token for the whole block.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kStage = 32;            // tokens staged per round
constexpr int kThreads = 128;         // 32 rows x 4 threads

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
recurrent_prefill_kernel(PrefillArgs p) {
  constexpr int kPer = D / 4;          // state entries per thread
  constexpr int kVec = kPer / 4;       // float4 chunks per thread
  __shared__ __align__(16) float sk[kStage][D];
  __shared__ __align__(16) float sq[kStage][D];
  __shared__ float sv[kStage][32];
  __shared__ float sg[kStage];
  __shared__ float sb[kStage];

  const GdnUnit u = p.units[blockIdx.x];
  const GdnSeq sd = p.seqs[u.seq];
  const int h = u.head;
  const int hk = h / p.group;
  const int tid = threadIdx.x;
  const int r = tid >> 2;              // row within the block
  const int sub = tid & 3;             // quarter of the row
  const int row = u.row0 + r;
  const bool row_ok = r < u.nrows;
  // the prompt's state slot (its index in the pack, or its pool slot)
  const size_t state_row = (((size_t)sd.state_slot * p.hv_heads + h) * D + row) * D;
  const bool have_init = p.init != nullptr && !(sd.flags & kSeqZeroInit);

  // thread owns float4 chunks c = sub + 4 m of its row (conflict-free smem reads)
  float4 S[kVec];
#pragma unroll
  for (int m = 0; m < kVec; ++m) {
    const int c = sub + 4 * m;
    S[m] = (have_init && row_ok) ? reinterpret_cast<const float4*>(p.init + state_row)[c]
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  const T* v = static_cast<const T*>(p.v);
  T* o = static_cast<T*>(p.o);
  int c_next = sd.ckpt_begin;
  const int warp = tid >> 5, lane = tid & 31;

  for (int t0 = 0; t0 < sd.len; t0 += kStage) {
    const int nt = min(kStage, sd.len - t0);
    __syncthreads();
    // stage q, k (normalised), v rows of this block, gates
    for (int j = warp; j < nt; j += kThreads / 32) {
      const size_t tok = (size_t)sd.tok_start + t0 + j;
      const T* qr = q + (tok * p.hk_heads + hk) * D;
      const T* kr = k + (tok * p.hk_heads + hk) * D;
      float qv[D / 32], kv[D / 32];
      float qq = 0.f, kk = 0.f;
#pragma unroll
      for (int e = 0; e < D / 32; ++e) {
        qv[e] = to_f32(qr[lane + 32 * e]);
        kv[e] = to_f32(kr[lane + 32 * e]);
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
        sq[j][lane + 32 * e] = qv[e] * qs;
        sk[j][lane + 32 * e] = kv[e] * ks;
      }
      if (u.row0 + lane < u.row0 + u.nrows)
        sv[j][lane] = (sd.flags & kSeqZeroV) ? 0.f
                                              : to_f32(v[(tok * p.hv_heads + h) * D + u.row0 + lane]);
      if (lane == 0) {
        float a = p.a[tok * p.hv_heads + h], b = p.beta[tok * p.hv_heads + h];
        if (p.gate_mode == 1) gate_from_raw(p.a_log[h], p.dt_bias[h], a, b);
        sg[j] = __expf(a);
        sb[j] = b;
      }
    }
    __syncthreads();

    for (int j = 0; j < nt; ++j) {
      const float g = sg[j], b = sb[j];
      const float4* kr = reinterpret_cast<const float4*>(sk[j]);
      const float4* qr = reinterpret_cast<const float4*>(sq[j]);
      float dot = 0.f;
#pragma unroll
      for (int m = 0; m < kVec; ++m) {
        const float4 kk4 = kr[sub + 4 * m];
        S[m].x *= g; S[m].y *= g; S[m].z *= g; S[m].w *= g;
        dot += S[m].x * kk4.x + S[m].y * kk4.y + S[m].z * kk4.z + S[m].w * kk4.w;
      }
      dot += __shfl_xor_sync(0xffffffffu, dot, 1);
      dot += __shfl_xor_sync(0xffffffffu, dot, 2);
      const float delta = b * (sv[j][r] - dot);
      float outv = 0.f;
#pragma unroll
      for (int m = 0; m < kVec; ++m) {
        const float4 kk4 = kr[sub + 4 * m];
        const float4 qq4 = qr[sub + 4 * m];
        S[m].x += delta * kk4.x; S[m].y += delta * kk4.y;
        S[m].z += delta * kk4.z; S[m].w += delta * kk4.w;
        outv += S[m].x * qq4.x + S[m].y * qq4.y + S[m].z * qq4.z + S[m].w * qq4.w;
      }
      outv += __shfl_xor_sync(0xffffffffu, outv, 1);
      outv += __shfl_xor_sync(0xffffffffu, outv, 2);
      const size_t tok = (size_t)sd.tok_start + t0 + j;
      if (sub == 0 && row_ok) o[(tok * p.hv_heads + h) * D + row] = from_f32<T>(p.scale * outv);
      if (c_next < sd.ckpt_end && p.ckpt_pos[c_next] == t0 + j + 1) {
        if (row_ok) {
          float4* dst = reinterpret_cast<float4*>(
              p.ckpt + (((size_t)c_next * p.hv_heads + h) * D + row) * D);
#pragma unroll
          for (int m = 0; m < kVec; ++m) dst[sub + 4 * m] = S[m];
        }
        ++c_next;
      }
    }
  }
  if (row_ok) {
    float4* dst = reinterpret_cast<float4*>(p.final_state + state_row);
#pragma unroll
    for (int m = 0; m < kVec; ++m) dst[sub + 4 * m] = S[m];
  }
  // this block's checkpoint rows are all stored (the token loop has ended)
  if (p.ckpt_ready) signal_ckpt_ready(p.ckpt_ready, u.seq, 0, kThreads, tid == 0);
}

}  // namespace

int launch_recurrent_prefill(const PrefillArgs& a, int head_dim, bool bf16, void* stream) {
  if (a.num_units == 0) return 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dim3 grid(a.num_units), block(kThreads);
  if (head_dim == 128) {
    if (bf16) recurrent_prefill_kernel<__nv_bfloat16, 128><<<grid, block, 0, s>>>(a);
    else recurrent_prefill_kernel<float, 128><<<grid, block, 0, s>>>(a);
  } else if (head_dim == 64) {
    if (bf16) recurrent_prefill_kernel<__nv_bfloat16, 64><<<grid, block, 0, s>>>(a);
    else recurrent_prefill_kernel<float, 64><<<grid, block, 0, s>>>(a);
  } else {
    return (int)cudaErrorInvalidValue;
  }
  return (int)cudaGetLastError();
}

}  // namespace gdn
