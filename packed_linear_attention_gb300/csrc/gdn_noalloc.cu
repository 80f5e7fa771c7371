// gdn_noalloc.cu — gdn_prefill_packed_noalloc: packed prefill for callers that cannot
// allocate memory when they call in.
//
// gdn_prefill_packed needs a caller-provided device workspace for its work list, and its
// handle may grow pinned staging buffers. Some callers cannot do either at call time: a
// serving engine that hands all device memory to its own pool at start-up and forbids
// allocation on the request path, or a plugin whose host framework owns every buffer.
// This entry point takes no workspace and no handle. The work list lives in a file-scope
// device array of fixed size (GDN_NOALLOC_SCRATCH_BYTES), which every GPU that loads the
// library holds until the process exits; the host image is built in a fixed host buffer
// and copied with one cudaMemcpyAsync. No call allocates anything.
//
// Sharing: all calls share the one device array per GPU. Each call rewrites the whole
// work list, including the status word at its start (cleared to zero). Two calls whose
// device work overlaps in time (e.g. on two streams) race on the array; serialise them.
//
// Set-up: the first call on each device looks up the array's device address with
// cudaGetSymbolAddress while that device is current, and caches it. Make that first call
// before any stream capture begins. The cached address belongs to the device's primary
// context: after a cudaDeviceReset in the same process this entry point must not be used.
//
// Status: the array starts with the status word that the chunked kernels set when a
// bounded device-side wait gives up; gdn_noalloc_read_status copies it into the caller's
// int32 (no allocation either).
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace {

using gdn::kMaxDevices;

// The scratch every call on this device shares (work list + status word).
static __device__ __align__(256) uint8_t g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

std::mutex g_lock;
void* g_scratch_addr[kMaxDevices] = {};
std::atomic<int32_t> g_test_hook{0};  // gdn_noalloc_set_test_hook

// The device address of this device's array (set-up on the first use per device, with that
// device current). Called with g_lock held.
gdn_status scratch_address(int dev, char** out) {
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<char*>(g_scratch_addr[dev]);
  return GDN_OK;
}
// Host image of the work list, copied from pageable memory: cudaMemcpyAsync returns only
// after the driver has taken the bytes, so the buffer is free again when the lock drops.
alignas(256) uint8_t g_host_image[GDN_NOALLOC_SCRATCH_BYTES];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return a && b && na && nb && x < y + nb && y < x + na;
}

}  // namespace

extern "C" gdn_status gdn_prefill_packed_noalloc(const gdn_config* cfg, int32_t num_seqs,
                                                 const int32_t* cu, const void* q,
                                                 const void* k, const void* v, const float* a,
                                                 const float* beta, const float* init,
                                                 const int32_t* ckpt_cu,
                                                 const int32_t* ckpt_pos, void* o,
                                                 float* ckpt_states, float* final_states,
                                                 void* stream) {
  gdn::PrefillPlan plan;
  gdn_status s = gdn::plan_prefill(nullptr, cfg, num_seqs, cu, ckpt_cu, ckpt_pos, &plan);
  if (s != GDN_OK) return s;
  if (plan.bytes > GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_UNSUPPORTED;

  // the buffer rules of gdn_prefill_packed
  const int64_t T = cu[num_seqs];
  const int D = cfg->head_dim_k;
  const size_t es = cfg->io_dtype == GDN_BF16 ? 2 : 4;
  if (T > 0 && (!q || !k || !v || !a || !beta || !o)) return GDN_ERR_INVALID_ARGUMENT;
  if (!final_states || (plan.num_ckpt > 0 && !ckpt_states)) return GDN_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {q, k, v, a, beta, init, o, ckpt_states, final_states};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_INVALID_ARGUMENT;
  const size_t sb = (size_t)cfg->num_v_heads * D * D * 4;
  const void* outs[] = {o, ckpt_states, final_states};
  const size_t out_n[] = {(size_t)T * cfg->num_v_heads * D * es, (size_t)plan.num_ckpt * sb,
                          (size_t)num_seqs * sb};
  const void* ins[] = {q, k, v, a, beta};
  const size_t in_n[] = {(size_t)T * cfg->num_k_heads * D * es,
                         (size_t)T * cfg->num_k_heads * D * es,
                         (size_t)T * cfg->num_v_heads * D * es, (size_t)T * cfg->num_v_heads * 4,
                         (size_t)T * cfg->num_v_heads * 4};
  for (int i = 0; i < 3; ++i) {
    for (int j = i + 1; j < 3; ++j)
      if (overlap(outs[i], out_n[i], outs[j], out_n[j])) return GDN_ERR_INVALID_ARGUMENT;
    for (int j = 0; j < 5; ++j)
      if (overlap(outs[i], out_n[i], ins[j], in_n[j])) return GDN_ERR_INVALID_ARGUMENT;
    if (init && static_cast<const void*>(init) != static_cast<const void*>(final_states) &&
        overlap(outs[i], out_n[i], init, (size_t)num_seqs * sb))
      return GDN_ERR_INVALID_ARGUMENT;
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> guard(g_lock);
  char* scratch = nullptr;
  const gdn_status sa = scratch_address(dev, &scratch);
  if (sa != GDN_OK) return sa;
  gdn::write_worklist(g_host_image, plan, cfg, num_seqs, cu, ckpt_cu, ckpt_pos);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(scratch, g_host_image, plan.bytes, cudaMemcpyHostToDevice, st) !=
      cudaSuccess)
    return GDN_ERR_CUDA;

  gdn::PrefillArgs pa;
  pa.q = q; pa.k = k; pa.v = v; pa.a = a; pa.beta = beta; pa.init = init;
  pa.o = o; pa.ckpt = ckpt_states; pa.final_state = final_states;
  pa.units = reinterpret_cast<const gdn::GdnUnit*>(scratch + plan.units_off);
  pa.seqs = reinterpret_cast<const gdn::GdnSeq*>(scratch + plan.seqs_off);
  pa.ckpt_pos = reinterpret_cast<const int32_t*>(scratch + plan.pos_off);
  pa.num_units = plan.num_units;
  pa.hk_heads = cfg->num_k_heads;
  pa.hv_heads = cfg->num_v_heads;
  pa.group = cfg->num_v_heads / cfg->num_k_heads;
  pa.head_dim = cfg->head_dim_k;
  pa.scale = cfg->scale;
  pa.l2norm = cfg->qk_l2norm ? 1 : 0;
  pa.status = reinterpret_cast<int32_t*>(scratch);
  pa.gate_mode = cfg->gate_mode;
  pa.a_log = cfg->a_log;
  pa.dt_bias = cfg->dt_bias;
  pa.test_skip_first_copy = g_test_hook.load(std::memory_order_relaxed);
  const int e = plan.family == 2
                    ? gdn::launch_chunked_prefill(pa, T, gdn::kChunkedAuto,
                                                  gdn::chunk_load(cu, num_seqs, cfg->num_v_heads),
                                                  stream)
                    : gdn::launch_recurrent_prefill(pa, D, cfg->io_dtype == GDN_BF16, stream);
  return e == 0 ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status gdn_noalloc_read_status(int32_t* status_out, void* stream) {
  if (!status_out) return GDN_ERR_INVALID_ARGUMENT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
  char* scratch = nullptr;
  {
    std::lock_guard<std::mutex> guard(g_lock);
    const gdn_status sa = scratch_address(dev, &scratch);
    if (sa != GDN_OK) return sa;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, scratch, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return GDN_ERR_CUDA;
  *status_out = v;
  return GDN_OK;
}

extern "C" gdn_status gdn_noalloc_set_test_hook(int32_t hook) {
  if (hook < 0 || hook > 1) return GDN_ERR_INVALID_ARGUMENT;
  g_test_hook.store(hook, std::memory_order_relaxed);
  return GDN_OK;
}
