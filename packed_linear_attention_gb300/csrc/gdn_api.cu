// gdn_api.cu — the C ABI: validation, the varlen work-list scheduler, launches, the
// pinned snapshot pool and the side-stream checkpoint copy.
//
// Conventions (see include/gdn.h): every argument is checked on the host before anything
// is enqueued ("reject unsupported combinations before model loading", pegainfer PR #786,
// Changes); device work is asynchronous on the caller's stream; the handle owns only host
// resources, a side stream and events, and destroying it drains that stream first.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/gdn.h"
#include "gdn_internal.h"

using gdn::GdnSeq;
using gdn::GdnUnit;

namespace {

constexpr int kStagingSlots = 4;
constexpr int kMaxHostGroups = 64;  // prompt groups of one gdn_prefill_packed_host call
constexpr size_t kAlign = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct StagingSlot {
  void* host = nullptr;   // pinned
  size_t bytes = 0;
  cudaEvent_t done = nullptr;  // recorded after the H2D copy out of this slot
  bool used = false;
};

}  // namespace

struct gdn_handle {
  int device = 0;
  void* pool = nullptr;
  size_t pool_bytes = 0;
  cudaStream_t side = nullptr;
  cudaEvent_t compute_ready = nullptr;
  cudaEvent_t copy_done = nullptr;
  bool copy_pending = false;
  StagingSlot slots[kStagingSlots];
  int next_slot = 0;
  int32_t kernel_pref = 0;
  int32_t test_hook = 0;  // gdn_set_test_hook
  int32_t launches = 0;   // kernels enqueued by the last prefill call (gdn_prefill_launch_count)
  // the owned prefill stream: at most one prefill in flight on it
  cudaStream_t prefill_stream = nullptr;
  cudaEvent_t prefill_ready = nullptr;  // caller stream -> prefill stream
  cudaEvent_t prefill_done = nullptr;
  bool prefill_inflight = false;
  // host-resident prefill: copy-in and copy-out streams, one event pair per prompt group
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t host_start = nullptr, host_done = nullptr;
  cudaEvent_t group_in[kMaxHostGroups] = {};
  cudaEvent_t group_out[kMaxHostGroups] = {};
};

namespace {

gdn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

// cuStreamWaitValue32 through the runtime's driver entry-point query (once per process).
using WaitValueFn = CUresult (*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
WaitValueFn wait_value_fn() {
  static WaitValueFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<WaitValueFn>(f);
  });
  return fn;
}

// Work-list layout inside the workspace (each array on a 256-byte boundary):
//   header {int32 status; int32 num_units;} | units | seqs | ckpt_pos | ready
// (ready: one int32 per prompt, zeroed by the upload; gdn_prefill_packed_snapshot's
// per-prompt checkpoint counters)
struct ListLayout {
  size_t units_off, seqs_off, pos_off, ready_off, total;
  int32_t num_units;
};

enum KernelFamily { kRecurrent = 1, kChunked = 2 };

// bf16 io, d = 64 or 128, C = 64 (d = 64 heads run zero-padded to 128 in the same kernels)
bool chunked_supported(const gdn_config* c) {
  return c->io_dtype == GDN_BF16 && (c->head_dim_k == 128 || c->head_dim_k == 64) &&
         c->head_dim_v == c->head_dim_k && c->chunk_size == 64;
}

KernelFamily pick_kernel(const gdn_handle* h, const gdn_config* c) {
  if (h && h->kernel_pref == 1) return kRecurrent;
  if (gdn::kChunkedReady && chunked_supported(c)) return kChunked;
  return kRecurrent;
}

int32_t units_per_head(KernelFamily f, int head_dim) {
  return f == kRecurrent ? head_dim / gdn::kRecurrentRows : 1;
}

ListLayout layout_for(int32_t num_seqs, int32_t num_units, int32_t num_ckpt) {
  ListLayout L;
  L.num_units = num_units;
  L.units_off = kAlign;
  L.seqs_off = align_up(L.units_off + sizeof(GdnUnit) * (size_t)num_units, kAlign);
  L.pos_off = align_up(L.seqs_off + sizeof(GdnSeq) * (size_t)num_seqs, kAlign);
  L.ready_off = align_up(L.pos_off + sizeof(int32_t) * (size_t)std::max(num_ckpt, 1), kAlign);
  L.total = align_up(L.ready_off + sizeof(int32_t) * (size_t)std::max(num_seqs, 1), kAlign);
  return L;
}

gdn_status check_config(const gdn_config* c) {
  if (!c) return GDN_ERR_INVALID_ARGUMENT;
  if (c->num_k_heads <= 0 || c->num_v_heads <= 0 || c->head_dim_k <= 0 || c->head_dim_v <= 0 ||
      c->chunk_size <= 0)
    return GDN_ERR_INVALID_ARGUMENT;
  if (c->num_v_heads % c->num_k_heads != 0) return GDN_ERR_INVALID_ARGUMENT;
  if (c->io_dtype != GDN_F32 && c->io_dtype != GDN_BF16) return GDN_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(c->scale)) return GDN_ERR_INVALID_ARGUMENT;
  if (c->gate_mode != GDN_GATES_DIRECT && c->gate_mode != GDN_GATES_RAW)
    return GDN_ERR_INVALID_ARGUMENT;
  if (c->gate_mode == GDN_GATES_RAW && (!c->a_log || !c->dt_bias))
    return GDN_ERR_INVALID_ARGUMENT;
  if (c->head_dim_k != c->head_dim_v) return GDN_ERR_UNSUPPORTED;
  if (c->head_dim_k != 64 && c->head_dim_k != 128) return GDN_ERR_UNSUPPORTED;
  if (c->chunk_size != 64) return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

// Checks the pack description; fills *num_ckpt.
gdn_status check_pack(const gdn_config* c, int32_t num_seqs, const int32_t* cu,
                      const int32_t* ckpt_cu, const int32_t* ckpt_pos, int32_t* num_ckpt) {
  if (num_seqs < 1 || !cu) return GDN_ERR_INVALID_ARGUMENT;
  if (cu[0] != 0) return GDN_ERR_INVALID_ARGUMENT;
  for (int32_t n = 0; n < num_seqs; ++n)
    if (cu[n + 1] < cu[n]) return GDN_ERR_INVALID_ARGUMENT;
  *num_ckpt = 0;
  if (!ckpt_cu) return GDN_OK;
  if (ckpt_cu[0] != 0) return GDN_ERR_INVALID_ARGUMENT;
  for (int32_t n = 0; n < num_seqs; ++n)
    if (ckpt_cu[n + 1] < ckpt_cu[n]) return GDN_ERR_INVALID_ARGUMENT;
  const int32_t total = ckpt_cu[num_seqs];
  if (total > 0 && !ckpt_pos) return GDN_ERR_INVALID_ARGUMENT;
  gdn_status soft = GDN_OK;
  for (int32_t n = 0; n < num_seqs; ++n) {
    const int32_t len = cu[n + 1] - cu[n];
    for (int32_t j = ckpt_cu[n]; j < ckpt_cu[n + 1]; ++j) {
      const int32_t p = ckpt_pos[j];
      if (p < 1 || p > len) return GDN_ERR_INVALID_ARGUMENT;
      if (j > ckpt_cu[n] && p <= ckpt_pos[j - 1]) return GDN_ERR_INVALID_ARGUMENT;
      if (p % c->chunk_size != 0 && p != len) soft = GDN_ERR_UNSUPPORTED;
    }
  }
  *num_ckpt = total;
  return soft;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  uintptr_t lo, hi;
};
bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

// Fills the host image of the work list. Units: every (prompt, value head, row block),
// ordered by prompt length, longest first (stable, so equal lengths keep pack order).
// Prompt n's state is slot slot_idx[n] of the initial / final state arrays (n without
// slot_idx); start_zero[n] != 0 makes it start from a zero state.
void build_worklist(void* dst, const ListLayout& L, KernelFamily fam, const gdn_config* c,
                    int32_t num_seqs, const int32_t* cu, const int32_t* ckpt_cu,
                    const int32_t* ckpt_pos, int32_t num_ckpt,
                    const int32_t* slot_idx = nullptr, const int32_t* start_zero = nullptr) {
  std::memset(dst, 0, L.total);
  char* base = static_cast<char*>(dst);
  int32_t* header = reinterpret_cast<int32_t*>(base);
  header[0] = 0;  // device status word
  header[1] = L.num_units;
  GdnSeq* seqs = reinterpret_cast<GdnSeq*>(base + L.seqs_off);
  for (int32_t n = 0; n < num_seqs; ++n) {
    seqs[n].tok_start = cu[n];
    seqs[n].len = cu[n + 1] - cu[n];
    seqs[n].ckpt_begin = ckpt_cu ? ckpt_cu[n] : 0;
    seqs[n].ckpt_end = ckpt_cu ? ckpt_cu[n + 1] : 0;
    seqs[n].flags = start_zero && start_zero[n] ? gdn::kSeqZeroInit : 0;
    seqs[n].state_slot = slot_idx ? slot_idx[n] : n;
  }
  if (num_ckpt > 0)
    std::memcpy(base + L.pos_off, ckpt_pos, sizeof(int32_t) * (size_t)num_ckpt);
  std::vector<int32_t> order(num_seqs);
  for (int32_t n = 0; n < num_seqs; ++n) order[n] = n;
  std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) {
    return (cu[x + 1] - cu[x]) > (cu[y + 1] - cu[y]);
  });
  GdnUnit* units = reinterpret_cast<GdnUnit*>(base + L.units_off);
  const int32_t per_head = units_per_head(fam, c->head_dim_v);
  const int32_t rows = c->head_dim_v / per_head;
  int32_t u = 0;
  for (int32_t n : order)
    for (int32_t h = 0; h < c->num_v_heads; ++h)
      for (int32_t r = 0; r < per_head; ++r) units[u++] = GdnUnit{n, h, r * rows, rows};
}

gdn_status plan(const gdn_handle* h, const gdn_config* c, int32_t num_seqs, const int32_t* cu,
                const int32_t* ckpt_cu, const int32_t* ckpt_pos, KernelFamily* fam,
                ListLayout* L, int32_t* num_ckpt) {
  gdn_status s = check_config(c);
  if (s != GDN_OK) return s;
  s = check_pack(c, num_seqs, cu, ckpt_cu, ckpt_pos, num_ckpt);
  if (s != GDN_OK) return s;
  *fam = pick_kernel(h, c);
  const int64_t units =
      (int64_t)num_seqs * c->num_v_heads * units_per_head(*fam, c->head_dim_v);
  if (units > INT32_MAX) return GDN_ERR_UNSUPPORTED;
  *L = layout_for(num_seqs, (int32_t)units, *num_ckpt);
  return GDN_OK;
}

// Takes the next pinned staging slot, growing it if needed, after its previous copy.
gdn_status take_slot(gdn_handle* h, size_t bytes, StagingSlot** out) {
  StagingSlot& s = h->slots[h->next_slot];
  h->next_slot = (h->next_slot + 1) % kStagingSlots;
  if (s.used) {
    if (cudaEventSynchronize(s.done) != cudaSuccess) return GDN_ERR_CUDA;
  }
  if (s.bytes < bytes) {
    if (s.host) cudaFreeHost(s.host);
    s.host = nullptr;
    s.bytes = 0;
    const size_t want = std::max(bytes, (size_t)1 << 16);
    if (cudaHostAlloc(&s.host, want, cudaHostAllocDefault) != cudaSuccess) return GDN_ERR_CUDA;
    s.bytes = want;
  }
  *out = &s;
  return GDN_OK;
}

}  // namespace

extern "C" {

int32_t gdn_abi_version(void) { return GDN_ABI_VERSION; }

const char* gdn_status_string(int32_t s) {
  switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARGUMENT: return "invalid argument";
    case GDN_ERR_UNSUPPORTED: return "unsupported configuration";
    case GDN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case GDN_ERR_CUDA: return "CUDA error";
    case GDN_ERR_DEVICE_TIMEOUT: return "device wait timed out or not finished";
    case GDN_ERR_POOL_EXHAUSTED: return "range outside the pinned snapshot pool";
    case GDN_ERR_BUSY: return "a prefill is already in flight on the handle's stream";
    default: return "unknown status";
  }
}

gdn_status gdn_handle_create(int32_t device, size_t pinned_pool_bytes, gdn_handle** out) {
  if (!out) return GDN_ERR_INVALID_ARGUMENT;
  *out = nullptr;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess) return GDN_ERR_CUDA;
  if (device < 0 || device >= count) return GDN_ERR_INVALID_ARGUMENT;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaSetDevice(device) != cudaSuccess) return GDN_ERR_CUDA;
  gdn_handle* h = new (std::nothrow) gdn_handle();
  if (!h) return GDN_ERR_CUDA;
  h->device = device;
  bool ok = cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&h->prefill_stream, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&h->compute_ready, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&h->copy_done, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&h->prefill_ready, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&h->prefill_done, cudaEventDisableTiming) == cudaSuccess &&
            cudaStreamCreateWithFlags(&h->h2d, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&h->d2h, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&h->host_start, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&h->host_done, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < kMaxHostGroups; ++i)
    ok = cudaEventCreateWithFlags(&h->group_in[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&h->group_out[i], cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < kStagingSlots; ++i)
    ok = cudaEventCreateWithFlags(&h->slots[i].done, cudaEventDisableTiming) == cudaSuccess;
  if (ok && pinned_pool_bytes > 0) {
    ok = cudaHostAlloc(&h->pool, pinned_pool_bytes, cudaHostAllocDefault) == cudaSuccess;
    if (ok) h->pool_bytes = pinned_pool_bytes;
  }
  cudaSetDevice(prev);
  if (!ok) {
    gdn_handle_destroy(h);
    return GDN_ERR_CUDA;
  }
  *out = h;
  return GDN_OK;
}

gdn_status gdn_handle_destroy(gdn_handle* h) {
  if (!h) return GDN_OK;
  gdn_status st = GDN_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(h->device);
  if (h->prefill_stream && cudaStreamSynchronize(h->prefill_stream) != cudaSuccess)
    st = GDN_ERR_CUDA;
  if (h->side && cudaStreamSynchronize(h->side) != cudaSuccess) st = GDN_ERR_CUDA;
  for (cudaStream_t s : {h->h2d, h->d2h})
    if (s && cudaStreamSynchronize(s) != cudaSuccess) st = GDN_ERR_CUDA;
  for (int i = 0; i < kMaxHostGroups; ++i) {
    if (h->group_in[i]) cudaEventDestroy(h->group_in[i]);
    if (h->group_out[i]) cudaEventDestroy(h->group_out[i]);
  }
  for (cudaEvent_t e : {h->host_start, h->host_done})
    if (e) cudaEventDestroy(e);
  for (cudaStream_t s : {h->h2d, h->d2h})
    if (s) cudaStreamDestroy(s);
  for (int i = 0; i < kStagingSlots; ++i) {
    StagingSlot& s = h->slots[i];
    if (s.used && s.done) cudaEventSynchronize(s.done);
    if (s.done) cudaEventDestroy(s.done);
    if (s.host) cudaFreeHost(s.host);
  }
  if (h->prefill_ready) cudaEventDestroy(h->prefill_ready);
  if (h->prefill_done) cudaEventDestroy(h->prefill_done);
  if (h->prefill_stream) cudaStreamDestroy(h->prefill_stream);
  if (h->compute_ready) cudaEventDestroy(h->compute_ready);
  if (h->copy_done) cudaEventDestroy(h->copy_done);
  if (h->side) cudaStreamDestroy(h->side);
  if (h->pool) cudaFreeHost(h->pool);
  cudaSetDevice(prev);
  delete h;
  return st;
}

gdn_status gdn_pool_info(gdn_handle* h, void** host_ptr, size_t* bytes) {
  if (!h || !host_ptr || !bytes) return GDN_ERR_INVALID_ARGUMENT;
  *host_ptr = h->pool;
  *bytes = h->pool_bytes;
  return GDN_OK;
}

gdn_status gdn_set_kernel_preference(gdn_handle* h, int32_t pref) {
  if (!h || pref < 0 || pref > 3) return GDN_ERR_INVALID_ARGUMENT;
  h->kernel_pref = pref;
  return GDN_OK;
}

gdn_status gdn_set_test_hook(gdn_handle* h, int32_t hook) {
  if (!h || hook < 0 || hook > 1) return GDN_ERR_INVALID_ARGUMENT;
  h->test_hook = hook;
  return GDN_OK;
}

gdn_status gdn_chunked_schedule(int32_t num_seqs, const int32_t* cu, int32_t num_v_heads,
                                int32_t num_sms, int32_t* schedule) {
  if (num_seqs < 0 || (num_seqs > 0 && !cu) || num_v_heads < 1 || num_sms < 1 || !schedule)
    return GDN_ERR_INVALID_ARGUMENT;
  for (int32_t n = 0; n < num_seqs; ++n)
    if (cu[n + 1] < cu[n]) return GDN_ERR_INVALID_ARGUMENT;
  if (num_seqs > 0 && cu[0] != 0) return GDN_ERR_INVALID_ARGUMENT;
  *schedule = gdn::plan_schedule(gdn::chunk_load(cu, num_seqs, num_v_heads), num_sms);
  return GDN_OK;
}

gdn_status gdn_prefill_workspace_size(const gdn_config* cfg, int32_t num_seqs,
                                      const int32_t* cu_seqlens_host,
                                      const int32_t* ckpt_cu_host, size_t* bytes) {
  if (!bytes) return GDN_ERR_INVALID_ARGUMENT;
  gdn_status s = check_config(cfg);
  if (s != GDN_OK) return s;
  if (num_seqs < 1 || !cu_seqlens_host) return GDN_ERR_INVALID_ARGUMENT;
  if (cu_seqlens_host[0] != 0) return GDN_ERR_INVALID_ARGUMENT;
  for (int32_t n = 0; n < num_seqs; ++n)
    if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return GDN_ERR_INVALID_ARGUMENT;
  int32_t num_ckpt = 0;
  if (ckpt_cu_host) {
    if (ckpt_cu_host[0] != 0) return GDN_ERR_INVALID_ARGUMENT;
    for (int32_t n = 0; n < num_seqs; ++n)
      if (ckpt_cu_host[n + 1] < ckpt_cu_host[n]) return GDN_ERR_INVALID_ARGUMENT;
    num_ckpt = ckpt_cu_host[num_seqs];
  }
  // sized for the family with the most units, so the answer does not depend on a handle
  const int64_t units = (int64_t)num_seqs * cfg->num_v_heads *
                        units_per_head(kRecurrent, cfg->head_dim_v);
  if (units > INT32_MAX) return GDN_ERR_UNSUPPORTED;
  *bytes = layout_for(num_seqs, (int32_t)units, num_ckpt).total;
  return GDN_OK;
}

namespace {

// Pointer, alignment and overlap checks shared by the prefill entry points.
// `state_slots`: states in the initial / final arrays (num_seqs, or a pool's slot count).
gdn_status check_buffers(const gdn_config* cfg, int32_t num_seqs, int64_t T, int32_t num_ckpt,
                         const void* q, const void* k, const void* v, const float* a,
                         const float* beta, const float* init, void* o, float* ckpt_states,
                         float* final_states, void* workspace, size_t workspace_bytes,
                         size_t workspace_needed, int64_t state_slots = -1) {
  if (state_slots < 0) state_slots = num_seqs;
  const int D = cfg->head_dim_k;
  const size_t es = cfg->io_dtype == GDN_BF16 ? 2 : 4;
  if (T > 0 && (!q || !k || !v || !a || !beta || !o)) return GDN_ERR_INVALID_ARGUMENT;
  if (!final_states) return GDN_ERR_INVALID_ARGUMENT;
  if (num_ckpt > 0 && !ckpt_states) return GDN_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {q, k, v, a, beta, init, o, ckpt_states, final_states};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_INVALID_ARGUMENT;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
    return GDN_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < workspace_needed) return GDN_ERR_WORKSPACE_TOO_SMALL;

  // outputs must not overlap each other, the inputs or the workspace (final may == init)
  const size_t state_bytes = (size_t)cfg->num_v_heads * D * D * 4;
  auto rng = [](const void* p, size_t n) {
    return Range{reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + n};
  };
  const Range outs[] = {rng(o, (size_t)T * cfg->num_v_heads * D * es),
                        rng(ckpt_states, (size_t)num_ckpt * state_bytes),
                        rng(final_states, (size_t)state_slots * state_bytes)};
  const Range ins[] = {rng(q, (size_t)T * cfg->num_k_heads * D * es),
                       rng(k, (size_t)T * cfg->num_k_heads * D * es),
                       rng(v, (size_t)T * cfg->num_v_heads * D * es),
                       rng(a, (size_t)T * cfg->num_v_heads * 4),
                       rng(beta, (size_t)T * cfg->num_v_heads * 4),
                       rng(workspace, workspace_needed)};
  for (int i = 0; i < 3; ++i) {
    if (outs[i].lo == 0 || outs[i].hi == outs[i].lo) continue;
    for (int j = i + 1; j < 3; ++j)
      if (outs[j].lo && overlaps(outs[i], outs[j])) return GDN_ERR_INVALID_ARGUMENT;
    for (const Range& r : ins)
      if (r.lo && r.hi > r.lo && overlaps(outs[i], r)) return GDN_ERR_INVALID_ARGUMENT;
  }
  if (init && static_cast<const void*>(init) != static_cast<const void*>(final_states)) {
    const Range ir = rng(init, (size_t)state_slots * state_bytes);
    for (const Range& r : outs)
      if (r.lo && r.hi > r.lo && overlaps(ir, r)) return GDN_ERR_INVALID_ARGUMENT;
  }
  return GDN_OK;
}

// Kernel arguments of one prefill launch over a work list at `list` (layout L).
gdn::PrefillArgs prefill_args(const gdn_config* cfg, const ListLayout& L, char* list,
                              int32_t* status, const void* q, const void* k, const void* v,
                              const float* a, const float* beta, const float* init, void* o,
                              float* ckpt_states, float* final_states) {
  gdn::PrefillArgs pa;
  pa.q = q; pa.k = k; pa.v = v; pa.a = a; pa.beta = beta; pa.init = init;
  pa.o = o; pa.ckpt = ckpt_states; pa.final_state = final_states;
  pa.units = reinterpret_cast<const GdnUnit*>(list + L.units_off);
  pa.seqs = reinterpret_cast<const GdnSeq*>(list + L.seqs_off);
  pa.ckpt_pos = reinterpret_cast<const int32_t*>(list + L.pos_off);
  pa.num_units = L.num_units;
  pa.hk_heads = cfg->num_k_heads;
  pa.hv_heads = cfg->num_v_heads;
  pa.group = cfg->num_v_heads / cfg->num_k_heads;
  pa.head_dim = cfg->head_dim_k;
  pa.scale = cfg->scale;
  pa.l2norm = cfg->qk_l2norm ? 1 : 0;
  pa.status = status;
  pa.gate_mode = cfg->gate_mode;
  pa.a_log = cfg->a_log;
  pa.dt_bias = cfg->dt_bias;
  return pa;
}

// `load`: the pack's chunk counts, for the chunked kernel's automatic schedule choice.
int launch_prefill(KernelFamily fam, gdn_handle* h, const gdn_config* cfg,
                   const gdn::PrefillArgs& pa, int64_t T, const gdn::ChunkLoad& load,
                   void* stream) {
  if (h && pa.num_units > 0) ++h->launches;  // one kernel launch either way
  if (fam == kChunked) {
    const int schedule = h && h->kernel_pref >= 2 ? h->kernel_pref : gdn::kChunkedAuto;
    gdn::PrefillArgs args = pa;
    args.test_skip_first_copy = h ? h->test_hook : 0;
    return gdn::launch_chunked_prefill(args, T, schedule, load, stream);
  }
  return gdn::launch_recurrent_prefill(pa, cfg->head_dim_k, cfg->io_dtype == GDN_BF16, stream);
}

}  // namespace

gdn_status gdn_prefill_packed(gdn_handle* h, const gdn_config* cfg, int32_t num_seqs,
                              const int32_t* cu, const void* q, const void* k, const void* v,
                              const float* a, const float* beta, const float* init,
                              const int32_t* ckpt_cu, const int32_t* ckpt_pos, void* o,
                              float* ckpt_states, float* final_states, void* workspace,
                              size_t workspace_bytes, void* stream) {
  KernelFamily fam;
  ListLayout L;
  int32_t num_ckpt = 0;
  gdn_status s = plan(h, cfg, num_seqs, cu, ckpt_cu, ckpt_pos, &fam, &L, &num_ckpt);
  if (s != GDN_OK) return s;
  const int64_t T = cu[num_seqs];
  s = check_buffers(cfg, num_seqs, T, num_ckpt, q, k, v, a, beta, init, o, ckpt_states,
                    final_states, workspace, workspace_bytes, L.total);
  if (s != GDN_OK) return s;
  if (!h) return GDN_ERR_INVALID_ARGUMENT;
  h->launches = 0;

  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return GDN_ERR_CUDA;
  if (prev != h->device && cudaSetDevice(h->device) != cudaSuccess) return GDN_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  StagingSlot* slot = nullptr;
  s = take_slot(h, L.total, &slot);
  if (s == GDN_OK) {
    build_worklist(slot->host, L, fam, cfg, num_seqs, cu, ckpt_cu, ckpt_pos, num_ckpt);
    cudaError_t e = cudaMemcpyAsync(workspace, slot->host, L.total, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaEventRecord(slot->done, st);
    slot->used = true;
    if (e != cudaSuccess) s = GDN_ERR_CUDA;
  }
  if (s == GDN_OK) {
    char* ws = static_cast<char*>(workspace);
    const gdn::PrefillArgs pa =
        prefill_args(cfg, L, ws, reinterpret_cast<int32_t*>(ws), q, k, v, a, beta, init, o,
                     ckpt_states, final_states);
    if (launch_prefill(fam, h, cfg, pa, T, gdn::chunk_load(cu, num_seqs, cfg->num_v_heads),
                       stream) != 0)
      s = GDN_ERR_CUDA;
  }
  if (prev != h->device) cudaSetDevice(prev);
  return s;
}

gdn_status gdn_prefill_packed_pool(gdn_handle* h, const gdn_config* cfg, int32_t num_seqs,
                                   const int32_t* cu, const void* q, const void* k,
                                   const void* v, const float* a, const float* beta,
                                   float* state_pool, int32_t num_slots,
                                   const int32_t* slot_idx, const int32_t* start_zero,
                                   const int32_t* ckpt_cu, const int32_t* ckpt_pos, void* o,
                                   float* ckpt_states, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  KernelFamily fam;
  ListLayout L;
  int32_t num_ckpt = 0;
  gdn_status s = plan(h, cfg, num_seqs, cu, ckpt_cu, ckpt_pos, &fam, &L, &num_ckpt);
  if (s != GDN_OK) return s;
  if (!state_pool || num_slots < 1 || !slot_idx) return GDN_ERR_INVALID_ARGUMENT;
  std::vector<char> taken((size_t)num_slots, 0);
  for (int32_t n = 0; n < num_seqs; ++n) {
    const int32_t sl = slot_idx[n];
    if (sl < 0 || sl >= num_slots || taken[(size_t)sl]) return GDN_ERR_INVALID_ARGUMENT;
    taken[(size_t)sl] = 1;
  }
  const int64_t T = cu[num_seqs];
  // the pool is both the initial and the final state array (updated in place)
  s = check_buffers(cfg, num_seqs, T, num_ckpt, q, k, v, a, beta, state_pool, o, ckpt_states,
                    state_pool, workspace, workspace_bytes, L.total, num_slots);
  if (s != GDN_OK) return s;
  if (!h) return GDN_ERR_INVALID_ARGUMENT;
  h->launches = 0;

  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return GDN_ERR_CUDA;
  if (prev != h->device && cudaSetDevice(h->device) != cudaSuccess) return GDN_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  StagingSlot* slot = nullptr;
  s = take_slot(h, L.total, &slot);
  if (s == GDN_OK) {
    build_worklist(slot->host, L, fam, cfg, num_seqs, cu, ckpt_cu, ckpt_pos, num_ckpt, slot_idx,
                   start_zero);
    cudaError_t e = cudaMemcpyAsync(workspace, slot->host, L.total, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaEventRecord(slot->done, st);
    slot->used = true;
    if (e != cudaSuccess) s = GDN_ERR_CUDA;
  }
  if (s == GDN_OK) {
    char* ws = static_cast<char*>(workspace);
    const gdn::PrefillArgs pa =
        prefill_args(cfg, L, ws, reinterpret_cast<int32_t*>(ws), q, k, v, a, beta, state_pool, o,
                     ckpt_states, state_pool);
    if (launch_prefill(fam, h, cfg, pa, T, gdn::chunk_load(cu, num_seqs, cfg->num_v_heads),
                       stream) != 0)
      s = GDN_ERR_CUDA;
  }
  if (prev != h->device) cudaSetDevice(prev);
  return s;
}

gdn_status gdn_prefill_packed_snapshot(gdn_handle* h, const gdn_config* cfg, int32_t num_seqs,
                                       const int32_t* cu, const void* q, const void* k,
                                       const void* v, const float* a, const float* beta,
                                       const float* init, const int32_t* ckpt_cu,
                                       const int32_t* ckpt_pos, void* o, float* ckpt_states,
                                       float* final_states, size_t pool_offset, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  KernelFamily fam;
  ListLayout L;
  int32_t num_ckpt = 0;
  gdn_status s = plan(h, cfg, num_seqs, cu, ckpt_cu, ckpt_pos, &fam, &L, &num_ckpt);
  if (s != GDN_OK) return s;
  const int64_t T = cu[num_seqs];
  s = check_buffers(cfg, num_seqs, T, num_ckpt, q, k, v, a, beta, init, o, ckpt_states,
                    final_states, workspace, workspace_bytes, L.total);
  if (s != GDN_OK) return s;
  if (!h) return GDN_ERR_INVALID_ARGUMENT;
  const size_t sb = (size_t)cfg->num_v_heads * cfg->head_dim_v * cfg->head_dim_k * 4;
  const size_t total = (size_t)num_ckpt * sb;
  if (pool_offset > h->pool_bytes || total > h->pool_bytes - pool_offset)
    return GDN_ERR_POOL_EXHAUSTED;
  WaitValueFn wait = wait_value_fn();
  h->launches = 0;

  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return GDN_ERR_CUDA;
  if (prev != h->device && cudaSetDevice(h->device) != cudaSuccess) return GDN_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  StagingSlot* slot = nullptr;
  s = take_slot(h, L.total, &slot);
  cudaError_t e = cudaSuccess;
  if (s == GDN_OK) {
    build_worklist(slot->host, L, fam, cfg, num_seqs, cu, ckpt_cu, ckpt_pos, num_ckpt);
    e = cudaMemcpyAsync(workspace, slot->host, L.total, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaEventRecord(slot->done, st);
    slot->used = true;
    // the side stream starts after the upload, which zeroed the prompts' counters
    if (e == cudaSuccess) e = cudaEventRecord(h->compute_ready, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->side, h->compute_ready, 0);
  }
  int32_t* ready = reinterpret_cast<int32_t*>(ws + L.ready_off);
  if (s == GDN_OK && e == cudaSuccess) {
    gdn::PrefillArgs pa = prefill_args(cfg, L, ws, reinterpret_cast<int32_t*>(ws), q, k, v, a,
                                       beta, init, o, ckpt_states, final_states);
    // with the driver's stream wait, every block counts its prompt's stored checkpoints
    if (wait && num_ckpt > 0) pa.ckpt_ready = ready;
    if (launch_prefill(fam, h, cfg, pa, T, gdn::chunk_load(cu, num_seqs, cfg->num_v_heads),
                       stream) != 0)
      s = GDN_ERR_CUDA;
  }
  if (s == GDN_OK && e == cudaSuccess && num_ckpt > 0) {
    char* dst = static_cast<char*>(h->pool) + pool_offset;
    const char* src = reinterpret_cast<const char*>(ckpt_states);
    if (!wait) {
      // no stream wait on memory: one copy after the whole pass
      e = cudaEventRecord(h->compute_ready, st);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(h->side, h->compute_ready, 0);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(dst, src, total, cudaMemcpyDeviceToHost, h->side);
    } else {
      // prompts in work-list order (longest first, the order in which their blocks start),
      // runs of consecutive prompt indices (contiguous checkpoint slots) merged up to 8 MiB
      // per copy; each copy waits until every block of its prompts counted its checkpoints
      std::vector<int32_t> order(num_seqs);
      for (int32_t n = 0; n < num_seqs; ++n) order[n] = n;
      std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) {
        return (cu[x + 1] - cu[x]) > (cu[y + 1] - cu[y]);
      });
      const cuuint32_t target =
          (cuuint32_t)(cfg->num_v_heads * units_per_head(fam, cfg->head_dim_v));
      constexpr size_t kCopyBytes = (size_t)8 << 20;
      size_t i = 0;
      while (e == cudaSuccess && i < order.size()) {
        const int32_t n0 = order[i];
        int32_t n1 = n0 + 1;  // prompts [n0, n1) in this copy
        size_t j = i + 1;
        while (j < order.size() && order[j] == n1 &&
               (size_t)(ckpt_cu[n1 + 1] - ckpt_cu[n0]) * sb <= kCopyBytes) {
          ++n1;
          ++j;
        }
        const int32_t c0 = ckpt_cu[n0], c1 = ckpt_cu[n1];
        if (c1 > c0) {
          for (int32_t n = n0; e == cudaSuccess && n < n1; ++n)
            if (ckpt_cu[n + 1] > ckpt_cu[n] &&
                wait(reinterpret_cast<CUstream>(h->side),
                     reinterpret_cast<CUdeviceptr>(ready + n), target,
                     CU_STREAM_WAIT_VALUE_GEQ) != CUDA_SUCCESS)
              e = cudaErrorUnknown;
          if (e == cudaSuccess)
            e = cudaMemcpyAsync(dst + (size_t)c0 * sb, src + (size_t)c0 * sb,
                                (size_t)(c1 - c0) * sb, cudaMemcpyDeviceToHost, h->side);
        }
        i = j;
      }
    }
    if (e == cudaSuccess) e = cudaEventRecord(h->copy_done, h->side);
    if (e == cudaSuccess) h->copy_pending = true;
  }
  if (prev != h->device) cudaSetDevice(prev);
  if (s != GDN_OK) return s;
  return cuda_status(e);
}

gdn_status gdn_checkpoint_copy_event(gdn_handle* h, void** event_out) {
  if (!h || !event_out) return GDN_ERR_INVALID_ARGUMENT;
  *event_out = static_cast<void*>(h->copy_done);
  return GDN_OK;
}

gdn_status gdn_checkpoint_copy_join(gdn_handle* h, void* stream) {
  if (!h) return GDN_ERR_INVALID_ARGUMENT;
  if (!h->copy_pending) return GDN_OK;
  return cuda_status(
      cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), h->copy_done, 0));
}

gdn_status gdn_prefill_launch_count(gdn_handle* h, int32_t* count) {
  if (!h || !count) return GDN_ERR_INVALID_ARGUMENT;
  *count = h->launches;
  return GDN_OK;
}

// ---- prefill from host memory --------------------------------------------------------------

namespace {

// One prompt group of gdn_prefill_packed_host: prompts [n0, n1), its sub-pack offsets and
// the place of its work list in the workspace.
struct HostGroup {
  int32_t n0, n1, c0, c1;
  std::vector<int32_t> cu, ck;
  KernelFamily fam;
  ListLayout L;
  size_t off;
};

// Splits the pack into groups and lays their work lists out one after another. With
// `sizing_only` the lists are sized for the family with the most units and the checkpoint
// positions are not looked at.
gdn_status plan_groups(const gdn_handle* h, const gdn_config* cfg, int32_t num_seqs,
                       const int32_t* cu, const int32_t* ckpt_cu, const int32_t* ckpt_pos,
                       int32_t group_prompts, bool sizing_only, std::vector<HostGroup>* out,
                       size_t* total) {
  if (group_prompts < 1) return GDN_ERR_INVALID_ARGUMENT;
  gdn_status s = check_config(cfg);
  if (s != GDN_OK) return s;
  if (num_seqs < 1 || !cu || cu[0] != 0) return GDN_ERR_INVALID_ARGUMENT;
  for (int32_t n = 0; n < num_seqs; ++n)
    if (cu[n + 1] < cu[n]) return GDN_ERR_INVALID_ARGUMENT;
  // Group sizes: 1, 2, 4, ... up to group_prompts at the start, group_prompts in the middle,
  // and the same ramp reversed at the end. The copy-in before the first prefill and the
  // prefill and copy-out after the last copy-in are the parts of the call that nothing
  // overlaps, so the end groups are small; the middle ones are large, for fewer copies.
  std::vector<int32_t> sizes;
  {
    std::vector<int32_t> ramp;
    for (int64_t g = 1; g < group_prompts; g *= 2) ramp.push_back((int32_t)g);
    int32_t left = num_seqs;
    std::vector<int32_t> head, tail;
    for (int32_t g : ramp) {
      if (left <= 2 * g) break;
      head.push_back(g);
      tail.push_back(g);
      left -= 2 * g;
    }
    for (int32_t g : head) sizes.push_back(g);
    while (left > 0) {
      const int32_t g = std::min(left, group_prompts);
      sizes.push_back(g);
      left -= g;
    }
    for (auto it = tail.rbegin(); it != tail.rend(); ++it) sizes.push_back(*it);
  }
  std::vector<int32_t> bounds{0};
  for (int32_t g : sizes) bounds.push_back(bounds.back() + g);
  const int32_t groups = (int32_t)bounds.size() - 1;
  if (groups > kMaxHostGroups) return GDN_ERR_UNSUPPORTED;
  out->clear();
  *total = 0;
  for (int32_t g = 0; g < groups; ++g) {
    HostGroup G;
    G.n0 = bounds[g];
    G.n1 = bounds[g + 1];
    G.c0 = ckpt_cu ? ckpt_cu[G.n0] : 0;
    G.c1 = ckpt_cu ? ckpt_cu[G.n1] : 0;
    if (G.c1 < G.c0) return GDN_ERR_INVALID_ARGUMENT;
    for (int32_t n = G.n0; n <= G.n1; ++n) G.cu.push_back(cu[n] - cu[G.n0]);
    if (ckpt_cu)
      for (int32_t n = G.n0; n <= G.n1; ++n) G.ck.push_back(ckpt_cu[n] - G.c0);
    const int32_t ng = G.n1 - G.n0;
    if (sizing_only) {
      G.fam = kRecurrent;
      const int64_t units = (int64_t)ng * cfg->num_v_heads * units_per_head(kRecurrent,
                                                                            cfg->head_dim_v);
      if (units > INT32_MAX) return GDN_ERR_UNSUPPORTED;
      G.L = layout_for(ng, (int32_t)units, G.c1 - G.c0);
    } else {
      int32_t nck = 0;
      s = plan(h, cfg, ng, G.cu.data(), ckpt_cu ? G.ck.data() : nullptr,
               ckpt_pos ? ckpt_pos + G.c0 : nullptr, &G.fam, &G.L, &nck);
      if (s != GDN_OK) return s;
    }
    G.off = *total;
    *total += G.L.total;
    out->push_back(std::move(G));
  }
  return GDN_OK;
}

}  // namespace

gdn_status gdn_prefill_host_workspace_size(const gdn_config* cfg, int32_t num_seqs,
                                           const int32_t* cu_seqlens_host,
                                           const int32_t* ckpt_cu_host, int32_t group_prompts,
                                           size_t* bytes) {
  if (!bytes) return GDN_ERR_INVALID_ARGUMENT;
  std::vector<HostGroup> groups;
  size_t total = 0;
  const gdn_status s = plan_groups(nullptr, cfg, num_seqs, cu_seqlens_host, ckpt_cu_host,
                                   nullptr, group_prompts, true, &groups, &total);
  if (s != GDN_OK) return s;
  *bytes = total;
  return GDN_OK;
}

gdn_status gdn_prefill_packed_host(gdn_handle* h, const gdn_config* cfg, int32_t num_seqs,
                                   const int32_t* cu, const int32_t* ckpt_cu,
                                   const int32_t* ckpt_pos, const gdn_prefill_buffers* host,
                                   const gdn_prefill_buffers* dev, int32_t group_prompts,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  if (!h || !host || !dev) return GDN_ERR_INVALID_ARGUMENT;
  // the whole pack is validated up front, as one gdn_prefill_packed call would be
  KernelFamily fam;
  ListLayout L;
  int32_t num_ckpt = 0;
  gdn_status s = plan(h, cfg, num_seqs, cu, ckpt_cu, ckpt_pos, &fam, &L, &num_ckpt);
  if (s != GDN_OK) return s;
  std::vector<HostGroup> groups;
  size_t lists = 0;
  s = plan_groups(h, cfg, num_seqs, cu, ckpt_cu, ckpt_pos, group_prompts, false, &groups,
                  &lists);
  if (s != GDN_OK) return s;
  const int64_t T = cu[num_seqs];
  s = check_buffers(cfg, num_seqs, T, num_ckpt, dev->q, dev->k, dev->v, dev->a, dev->beta,
                    dev->initial_state, dev->o, dev->ckpt_states, dev->final_states, workspace,
                    workspace_bytes, lists);
  if (s != GDN_OK) return s;
  if (T > 0 && (!host->q || !host->k || !host->v || !host->a || !host->beta || !host->o))
    return GDN_ERR_INVALID_ARGUMENT;
  if (!host->final_states || (num_ckpt > 0 && !host->ckpt_states)) return GDN_ERR_INVALID_ARGUMENT;
  if (!host->initial_state != !dev->initial_state) return GDN_ERR_INVALID_ARGUMENT;
  h->launches = 0;

  const size_t es = cfg->io_dtype == GDN_BF16 ? 2 : 4;
  const int D = cfg->head_dim_k;
  const size_t qrow = (size_t)cfg->num_k_heads * D * es, vrow = (size_t)cfg->num_v_heads * D * es;
  const size_t grow = (size_t)cfg->num_v_heads * 4, sb = (size_t)cfg->num_v_heads * D * D * 4;
  auto at = [](const void* p, size_t off) {
    return static_cast<char*>(const_cast<void*>(p)) + off;
  };
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return GDN_ERR_CUDA;
  if (prev != h->device && cudaSetDevice(h->device) != cudaSuccess) return GDN_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);

  // every group's work list in one copy, queued ahead of the bulk copies
  StagingSlot* slot = nullptr;
  s = take_slot(h, lists, &slot);
  cudaError_t e = cudaSuccess;
  if (s == GDN_OK) {
    char* img = static_cast<char*>(slot->host);
    for (const HostGroup& G : groups)
      build_worklist(img + G.off, G.L, G.fam, cfg, G.n1 - G.n0, G.cu.data(),
                     ckpt_cu ? G.ck.data() : nullptr, ckpt_pos ? ckpt_pos + G.c0 : nullptr,
                     G.c1 - G.c0);
    e = cudaMemcpyAsync(ws, img, lists, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaEventRecord(slot->done, st);
    slot->used = true;
  }
  // copies into the device buffers start after the work already queued on the caller's stream
  if (s == GDN_OK && e == cudaSuccess) e = cudaEventRecord(h->host_start, st);
  if (s == GDN_OK && e == cudaSuccess) e = cudaStreamWaitEvent(h->h2d, h->host_start, 0);
  if (s == GDN_OK && e == cudaSuccess) e = cudaStreamWaitEvent(h->d2h, h->host_start, 0);
  for (size_t g = 0; s == GDN_OK && e == cudaSuccess && g < groups.size(); ++g) {
    const HostGroup& G = groups[g];
    const size_t t0 = (size_t)cu[G.n0], nt = (size_t)(cu[G.n1] - cu[G.n0]);
    // copy in: this group's token rows and initial states
    auto in = [&](void* d, const void* hs, size_t off, size_t n) {
      if (e == cudaSuccess && n > 0)
        e = cudaMemcpyAsync(at(d, off), at(hs, off), n, cudaMemcpyHostToDevice, h->h2d);
    };
    in(dev->q, host->q, t0 * qrow, nt * qrow);
    in(dev->k, host->k, t0 * qrow, nt * qrow);
    in(dev->v, host->v, t0 * vrow, nt * vrow);
    in(dev->a, host->a, t0 * grow, nt * grow);
    in(dev->beta, host->beta, t0 * grow, nt * grow);
    if (dev->initial_state)
      in(dev->initial_state, host->initial_state, G.n0 * sb, (G.n1 - G.n0) * sb);
    if (e == cudaSuccess) e = cudaEventRecord(h->group_in[g], h->h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, h->group_in[g], 0);
    if (e != cudaSuccess) break;
    // the group's prefill: a sub-pack over the same buffers, rows and state slots offset
    const gdn::PrefillArgs pa = prefill_args(
        cfg, G.L, ws + G.off, reinterpret_cast<int32_t*>(ws), at(dev->q, t0 * qrow),
        at(dev->k, t0 * qrow), at(dev->v, t0 * vrow),
        reinterpret_cast<const float*>(at(dev->a, t0 * grow)),
        reinterpret_cast<const float*>(at(dev->beta, t0 * grow)),
        dev->initial_state ? reinterpret_cast<const float*>(at(dev->initial_state, G.n0 * sb))
                           : nullptr,
        at(dev->o, t0 * vrow),
        G.c1 > G.c0 ? reinterpret_cast<float*>(at(dev->ckpt_states, G.c0 * sb)) : nullptr,
        reinterpret_cast<float*>(at(dev->final_states, G.n0 * sb)));
    if (launch_prefill(G.fam, h, cfg, pa, (int64_t)nt,
                       gdn::chunk_load(cu + G.n0, G.n1 - G.n0, cfg->num_v_heads),
                       stream) != 0) {
      s = GDN_ERR_CUDA;
      break;
    }
    // copy out once the group's prefill is done
    e = cudaEventRecord(h->group_out[g], st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->d2h, h->group_out[g], 0);
    auto out = [&](void* hd, const void* ds, size_t off, size_t n) {
      if (e == cudaSuccess && n > 0)
        e = cudaMemcpyAsync(at(hd, off), at(ds, off), n, cudaMemcpyDeviceToHost, h->d2h);
    };
    out(host->o, dev->o, t0 * vrow, nt * vrow);
    if (G.c1 > G.c0) out(host->ckpt_states, dev->ckpt_states, G.c0 * sb, (G.c1 - G.c0) * sb);
    out(host->final_states, dev->final_states, G.n0 * sb, (G.n1 - G.n0) * sb);
  }
  // the caller's stream completes after the last copy out
  if (s == GDN_OK && e == cudaSuccess) e = cudaEventRecord(h->host_done, h->d2h);
  if (s == GDN_OK && e == cudaSuccess) e = cudaStreamWaitEvent(st, h->host_done, 0);
  if (prev != h->device) cudaSetDevice(prev);
  if (s != GDN_OK) return s;
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// ---- sequence splitting ------------------------------------------------------------------

namespace {

struct VSeq {
  int32_t tok_start, len, ckpt_begin, ckpt_end, flags;
};

gdn::ChunkLoad vseq_load(const std::vector<VSeq>& vs, int32_t units_per_prompt) {
  gdn::ChunkLoad l;
  for (const VSeq& x : vs) {
    if (x.len <= 1) {
      l.short_units += units_per_prompt;
      continue;
    }
    const int32_t c = (x.len + 63) / 64;
    l.total += (int64_t)c * units_per_prompt;
    l.units += units_per_prompt;
    l.longest = std::max(l.longest, c);
  }
  return l;
}

// Work-list image for a list of virtual prompts (same layout and longest-first order as
// build_worklist); ckpt positions are copied as given.
void build_vworklist(void* dst, const ListLayout& L, KernelFamily fam, const gdn_config* c,
                     const std::vector<VSeq>& vs, const std::vector<int32_t>& pos) {
  std::memset(dst, 0, L.total);
  char* base = static_cast<char*>(dst);
  int32_t* header = reinterpret_cast<int32_t*>(base);
  header[1] = L.num_units;
  GdnSeq* seqs = reinterpret_cast<GdnSeq*>(base + L.seqs_off);
  for (size_t n = 0; n < vs.size(); ++n)
    seqs[n] = GdnSeq{vs[n].tok_start, vs[n].len, vs[n].ckpt_begin, vs[n].ckpt_end, vs[n].flags,
                     (int32_t)n};
  if (!pos.empty()) std::memcpy(base + L.pos_off, pos.data(), sizeof(int32_t) * pos.size());
  std::vector<int32_t> order(vs.size());
  for (size_t n = 0; n < vs.size(); ++n) order[n] = (int32_t)n;
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t x, int32_t y) { return vs[x].len > vs[y].len; });
  GdnUnit* units = reinterpret_cast<GdnUnit*>(base + L.units_off);
  const int32_t per_head = units_per_head(fam, c->head_dim_v);
  const int32_t rows = c->head_dim_v / per_head;
  int32_t u = 0;
  for (int32_t n : order)
    for (int32_t h = 0; h < c->num_v_heads; ++h)
      for (int32_t r = 0; r < per_head; ++r) units[u++] = GdnUnit{n, h, r * rows, rows};
}

// The split plan. Pass A runs, in one launch, segment 0 of every prompt from the caller's
// initial state (unsplit prompts entirely), then for every middle segment p of a split
// prompt B_p (zero start) and M_p (identity start, v taken as zero). The maps compose into
// the initial states of segments 1 .. P-1, which pass C runs with their checkpoints.
struct SplitPlan {
  std::vector<VSeq> va, vc;
  std::vector<int32_t> fill;    // pass A initial states: caller's prompt i, zero, identity
  std::vector<gdn::SplitCompose> jobs;
  std::vector<int32_t> gather;  // per prompt: final state in pass A (i) or C (-1 - i)
  std::vector<int32_t> pos;     // checkpoint positions relative to their segment
  ListLayout la, lc;
  size_t off_c, off_fill, off_jobs, off_gather, host_bytes;
  size_t off_init_a, off_fin_a, off_init_c, off_fin_c, total;
};

// `pref`: the handle's kernel preference (1 sizes for the token-serial family, which has
// the most units).
gdn_status plan_split(int32_t pref, const gdn_config* cfg, int32_t num_seqs, const int32_t* cu,
                      const int32_t* ckpt_cu, const int32_t* ckpt_pos, int32_t seg,
                      bool have_init, KernelFamily* fam, SplitPlan* sp) {
  gdn_status s = check_config(cfg);
  if (s != GDN_OK) return s;
  if (seg < 64 || seg % 64 != 0) return GDN_ERR_INVALID_ARGUMENT;
  int32_t num_ckpt = 0;
  s = check_pack(cfg, num_seqs, cu, ckpt_cu, ckpt_pos, &num_ckpt);
  if (s != GDN_OK) return s;
  *fam = pref == 1 || !(gdn::kChunkedReady && chunked_supported(cfg)) ? kRecurrent : kChunked;
  SplitPlan& P = *sp;
  P.pos.assign(ckpt_pos ? ckpt_pos : nullptr, ckpt_pos ? ckpt_pos + num_ckpt : nullptr);
  auto segs_of = [&](int32_t n) {
    const int32_t len = cu[n + 1] - cu[n];
    return len > seg ? (len + seg - 1) / seg : 1;
  };
  // checkpoint range [j0, j1) of prompt n inside segment p, positions made segment-relative
  auto ckpt_range = [&](int32_t n, int32_t p, int32_t* j0, int32_t* j1) {
    *j0 = *j1 = 0;
    if (!ckpt_cu) return;
    int32_t j = ckpt_cu[n];
    while (j < ckpt_cu[n + 1] && (ckpt_pos[j] - 1) / seg < p) ++j;
    *j0 = j;
    while (j < ckpt_cu[n + 1] && (ckpt_pos[j] - 1) / seg == p) {
      P.pos[j] = ckpt_pos[j] - p * seg;
      ++j;
    }
    *j1 = j;
  };
  // pass A: segment 0 of every prompt (index n), then the maps of split prompts
  for (int32_t n = 0; n < num_seqs; ++n) {
    const int32_t len = cu[n + 1] - cu[n];
    int32_t j0, j1;
    ckpt_range(n, 0, &j0, &j1);
    P.va.push_back(VSeq{cu[n], std::min(len, seg), j0, j1, 0});
    P.fill.push_back(have_init ? n : gdn::kSplitZero);
  }
  for (int32_t n = 0; n < num_seqs; ++n) {
    const int32_t np = segs_of(n);
    if (np == 1) {
      P.gather.push_back(n);
      continue;
    }
    gdn::SplitCompose job;
    job.num_segments = np;
    job.first_final = n;
    job.first_map = (int32_t)P.va.size();
    job.first_init = (int32_t)P.vc.size();
    for (int32_t p = 1; p + 1 < np; ++p) {
      P.va.push_back(VSeq{cu[n] + p * seg, seg, 0, 0, 0});                // B_p
      P.fill.push_back(gdn::kSplitZero);
      P.va.push_back(VSeq{cu[n] + p * seg, seg, 0, 0, gdn::kSeqZeroV});   // M_p
      P.fill.push_back(gdn::kSplitIdentity);
    }
    for (int32_t p = 1; p < np; ++p) {
      int32_t j0, j1;
      ckpt_range(n, p, &j0, &j1);
      P.vc.push_back(VSeq{cu[n] + p * seg, std::min(seg, cu[n + 1] - cu[n] - p * seg), j0, j1,
                          0});
    }
    P.gather.push_back(-1 - (int32_t)(P.vc.size() - 1));
    P.jobs.push_back(job);
  }
  const int32_t per_head = units_per_head(*fam, cfg->head_dim_v);
  const int64_t ua = (int64_t)P.va.size() * cfg->num_v_heads * per_head;
  const int64_t uc = (int64_t)P.vc.size() * cfg->num_v_heads * per_head;
  if (ua > INT32_MAX || uc > INT32_MAX) return GDN_ERR_UNSUPPORTED;
  P.la = layout_for((int32_t)P.va.size(), (int32_t)ua, num_ckpt);
  P.lc = layout_for(std::max<int32_t>((int32_t)P.vc.size(), 1), (int32_t)uc, num_ckpt);
  P.off_c = P.la.total;
  P.off_fill = align_up(P.off_c + P.lc.total, kAlign);
  P.off_jobs = align_up(P.off_fill + sizeof(int32_t) * P.fill.size(), kAlign);
  P.off_gather = align_up(
      P.off_jobs + sizeof(gdn::SplitCompose) * std::max<size_t>(P.jobs.size(), 1), kAlign);
  P.host_bytes = align_up(P.off_gather + sizeof(int32_t) * P.gather.size(), kAlign);
  const size_t sb = (size_t)cfg->num_v_heads * cfg->head_dim_v * cfg->head_dim_k * 4;
  P.off_init_a = P.host_bytes;
  P.off_fin_a = align_up(P.off_init_a + sb * P.va.size(), kAlign);
  P.off_init_c = align_up(P.off_fin_a + sb * P.va.size(), kAlign);
  P.off_fin_c = align_up(P.off_init_c + sb * P.vc.size(), kAlign);
  P.total = align_up(P.off_fin_c + sb * P.vc.size(), kAlign);
  return GDN_OK;
}

}  // namespace

gdn_status gdn_split_segment_auto(int32_t num_seqs, const int32_t* cu, int32_t num_v_heads,
                                  int32_t num_sms, int32_t* segment_len) {
  if (num_seqs < 0 || (num_seqs > 0 && !cu) || num_v_heads < 1 || num_sms < 1 || !segment_len)
    return GDN_ERR_INVALID_ARGUMENT;
  if (num_seqs > 0 && cu[0] != 0) return GDN_ERR_INVALID_ARGUMENT;
  for (int32_t n = 0; n < num_seqs; ++n)
    if (cu[n + 1] < cu[n]) return GDN_ERR_INVALID_ARGUMENT;
  *segment_len = gdn::choose_split_segment(cu, num_seqs, num_v_heads, num_sms);
  return GDN_OK;
}

gdn_status gdn_prefill_split_workspace_size(const gdn_config* cfg, int32_t num_seqs,
                                            const int32_t* cu_seqlens_host,
                                            const int32_t* ckpt_cu_host,
                                            const int32_t* ckpt_pos_host, int32_t segment_len,
                                            size_t* bytes) {
  if (!bytes) return GDN_ERR_INVALID_ARGUMENT;
  KernelFamily fam;
  SplitPlan sp;
  // sized for the family with the most units, so the answer does not depend on a handle
  const gdn_status s = plan_split(1, cfg, num_seqs, cu_seqlens_host, ckpt_cu_host,
                                  ckpt_pos_host, segment_len, true, &fam, &sp);
  if (s != GDN_OK) return s;
  *bytes = sp.total;
  return GDN_OK;
}

gdn_status gdn_prefill_packed_split(gdn_handle* h, const gdn_config* cfg, int32_t num_seqs,
                                    const int32_t* cu, const void* q, const void* k,
                                    const void* v, const float* a, const float* beta,
                                    const float* init, const int32_t* ckpt_cu,
                                    const int32_t* ckpt_pos, void* o, float* ckpt_states,
                                    float* final_states, int32_t segment_len, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  KernelFamily fam;
  SplitPlan P;
  gdn_status s = plan_split(h ? h->kernel_pref : 0, cfg, num_seqs, cu, ckpt_cu, ckpt_pos,
                            segment_len, init != nullptr, &fam, &P);
  if (s != GDN_OK) return s;
  const int64_t T = cu[num_seqs];
  const int32_t num_ckpt = ckpt_cu ? ckpt_cu[num_seqs] : 0;
  s = check_buffers(cfg, num_seqs, T, num_ckpt, q, k, v, a, beta, init, o, ckpt_states,
                    final_states, workspace, workspace_bytes, P.total);
  if (s != GDN_OK) return s;
  if (!h) return GDN_ERR_INVALID_ARGUMENT;
  h->launches = 0;

  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return GDN_ERR_CUDA;
  if (prev != h->device && cudaSetDevice(h->device) != cudaSuccess) return GDN_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  const int hv = cfg->num_v_heads, d = cfg->head_dim_v;
  float* init_a = reinterpret_cast<float*>(ws + P.off_init_a);
  float* fin_a = reinterpret_cast<float*>(ws + P.off_fin_a);
  float* init_c = reinterpret_cast<float*>(ws + P.off_init_c);
  float* fin_c = reinterpret_cast<float*>(ws + P.off_fin_c);

  StagingSlot* slot = nullptr;
  s = take_slot(h, P.host_bytes, &slot);
  if (s == GDN_OK) {
    char* img = static_cast<char*>(slot->host);
    build_vworklist(img, P.la, fam, cfg, P.va, P.pos);
    build_vworklist(img + P.off_c, P.lc, fam, cfg, P.vc, P.pos);
    std::memcpy(img + P.off_fill, P.fill.data(), sizeof(int32_t) * P.fill.size());
    if (!P.jobs.empty())
      std::memcpy(img + P.off_jobs, P.jobs.data(), sizeof(gdn::SplitCompose) * P.jobs.size());
    std::memcpy(img + P.off_gather, P.gather.data(), sizeof(int32_t) * P.gather.size());
    cudaError_t e = cudaMemcpyAsync(ws, img, P.host_bytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaEventRecord(slot->done, st);
    slot->used = true;
    if (e != cudaSuccess) s = GDN_ERR_CUDA;
  }
  int e = 0;
  if (s == GDN_OK) {
    // pass A: segment 0 of every prompt and the segment maps of split prompts
    e = gdn::launch_fill_states(init_a, init, reinterpret_cast<const int32_t*>(ws + P.off_fill),
                                (int)P.va.size(), hv, d, stream);
    if (!P.va.empty()) ++h->launches;
    if (e == 0)
      e = launch_prefill(fam, h, cfg,
                         prefill_args(cfg, P.la, ws, status, q, k, v, a, beta, init_a, o,
                                      ckpt_states, fin_a),
                         T, vseq_load(P.va, hv), stream);
    // the initial states of segments 1 .. P-1, then pass C
    if (e == 0)
      e = gdn::launch_compose_maps(reinterpret_cast<const gdn::SplitCompose*>(ws + P.off_jobs),
                                   (int)P.jobs.size(), fin_a, init_c, hv, d, stream);
    if (e == 0 && !P.jobs.empty()) ++h->launches;
    if (e == 0 && !P.vc.empty())
      e = launch_prefill(fam, h, cfg,
                         prefill_args(cfg, P.lc, ws + P.off_c, status, q, k, v, a, beta, init_c,
                                      o, ckpt_states, fin_c),
                         T, vseq_load(P.vc, hv), stream);
    if (e == 0)
      e = gdn::launch_gather_states(final_states, fin_a, fin_c,
                                    reinterpret_cast<const int32_t*>(ws + P.off_gather),
                                    num_seqs, hv, d, stream);
    if (e == 0) ++h->launches;
    if (e != 0) s = GDN_ERR_CUDA;
  }
  if (prev != h->device) cudaSetDevice(prev);
  return s;
}

gdn_status gdn_prefill_worklist_host(gdn_handle* h, const gdn_config* cfg, int32_t num_seqs,
                                     const int32_t* cu, const int32_t* ckpt_cu,
                                     const int32_t* ckpt_pos, void* out, size_t out_bytes,
                                     size_t* bytes_needed) {
  KernelFamily fam;
  ListLayout L;
  int32_t num_ckpt = 0;
  gdn_status s = plan(h, cfg, num_seqs, cu, ckpt_cu, ckpt_pos, &fam, &L, &num_ckpt);
  if (s != GDN_OK) return s;
  if (bytes_needed) *bytes_needed = L.total;
  if (!out) return GDN_OK;
  if (out_bytes < L.total) return GDN_ERR_WORKSPACE_TOO_SMALL;
  build_worklist(out, L, fam, cfg, num_seqs, cu, ckpt_cu, ckpt_pos, num_ckpt);
  return GDN_OK;
}

gdn_status gdn_read_device_status(const void* workspace, int32_t* status_out, void* stream) {
  if (!workspace || !status_out) return GDN_ERR_INVALID_ARGUMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return GDN_ERR_CUDA;
  *status_out = v;
  return GDN_OK;
}

gdn_status gdn_checkpoint_copy(gdn_handle* h, const float* src, size_t bytes,
                               size_t pool_offset, void* stream) {
  if (!h || (!src && bytes > 0)) return GDN_ERR_INVALID_ARGUMENT;
  if (pool_offset > h->pool_bytes || bytes > h->pool_bytes - pool_offset)
    return GDN_ERR_POOL_EXHAUSTED;
  if (bytes == 0) return GDN_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaEventRecord(h->compute_ready, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->side, h->compute_ready, 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(static_cast<char*>(h->pool) + pool_offset, src, bytes,
                        cudaMemcpyDeviceToHost, h->side);
  if (e == cudaSuccess) e = cudaEventRecord(h->copy_done, h->side);
  if (e == cudaSuccess) h->copy_pending = true;
  return cuda_status(e);
}

gdn_status gdn_checkpoint_copy_query(gdn_handle* h) {
  if (!h) return GDN_ERR_INVALID_ARGUMENT;
  if (!h->copy_pending) return GDN_OK;
  cudaError_t e = cudaEventQuery(h->copy_done);
  if (e == cudaSuccess) return GDN_OK;
  if (e == cudaErrorNotReady) return GDN_ERR_DEVICE_TIMEOUT;
  return GDN_ERR_CUDA;
}

gdn_status gdn_checkpoint_copy_wait(gdn_handle* h) {
  if (!h) return GDN_ERR_INVALID_ARGUMENT;
  if (!h->copy_pending) return GDN_OK;
  return cuda_status(cudaEventSynchronize(h->copy_done));
}

gdn_status gdn_prefill_packed_async(gdn_handle* h, const gdn_config* cfg, int32_t num_seqs,
                                    const int32_t* cu, const void* q, const void* k,
                                    const void* v, const float* a, const float* beta,
                                    const float* init, const int32_t* ckpt_cu,
                                    const int32_t* ckpt_pos, void* o, float* ckpt_states,
                                    float* final_states, void* workspace,
                                    size_t workspace_bytes, void* after_stream) {
  if (!h) return GDN_ERR_INVALID_ARGUMENT;
  if (h->prefill_inflight) {
    const cudaError_t q0 = cudaEventQuery(h->prefill_done);
    if (q0 == cudaErrorNotReady) return GDN_ERR_BUSY;
    if (q0 != cudaSuccess) return GDN_ERR_CUDA;
    h->prefill_inflight = false;
  }
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return GDN_ERR_CUDA;
  if (prev != h->device && cudaSetDevice(h->device) != cudaSuccess) return GDN_ERR_CUDA;
  // the owned stream starts once the work already queued on after_stream is done
  cudaError_t e = cudaEventRecord(h->prefill_ready, static_cast<cudaStream_t>(after_stream));
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->prefill_stream, h->prefill_ready, 0);
  if (prev != h->device) cudaSetDevice(prev);
  if (e != cudaSuccess) return GDN_ERR_CUDA;
  gdn_status s = gdn_prefill_packed(h, cfg, num_seqs, cu, q, k, v, a, beta, init, ckpt_cu,
                                    ckpt_pos, o, ckpt_states, final_states, workspace,
                                    workspace_bytes, h->prefill_stream);
  if (s != GDN_OK) return s;
  if (cudaEventRecord(h->prefill_done, h->prefill_stream) != cudaSuccess) return GDN_ERR_CUDA;
  h->prefill_inflight = true;
  return GDN_OK;
}

gdn_status gdn_prefill_async_query(gdn_handle* h) {
  if (!h) return GDN_ERR_INVALID_ARGUMENT;
  if (!h->prefill_inflight) return GDN_OK;
  const cudaError_t e = cudaEventQuery(h->prefill_done);
  if (e == cudaErrorNotReady) return GDN_ERR_DEVICE_TIMEOUT;
  if (e != cudaSuccess) return GDN_ERR_CUDA;
  h->prefill_inflight = false;
  return GDN_OK;
}

gdn_status gdn_prefill_async_wait(gdn_handle* h) {
  if (!h) return GDN_ERR_INVALID_ARGUMENT;
  if (!h->prefill_inflight) return GDN_OK;
  if (cudaEventSynchronize(h->prefill_done) != cudaSuccess) return GDN_ERR_CUDA;
  h->prefill_inflight = false;
  return GDN_OK;
}

gdn_status gdn_prefill_async_join(gdn_handle* h, void* stream) {
  if (!h) return GDN_ERR_INVALID_ARGUMENT;
  if (!h->prefill_inflight) return GDN_OK;
  return cuda_status(
      cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), h->prefill_done, 0));
}

gdn_status gdn_decode_step(gdn_handle* h, const gdn_config* cfg, int32_t batch, const void* q,
                           const void* k, const void* v, const float* a, const float* beta,
                           float* pool, int32_t num_slots, const int32_t* slot_idx, void* o,
                           void* stream) {
  gdn_status s = check_config(cfg);
  if (s != GDN_OK) return s;
  if (batch < 0 || num_slots < 0) return GDN_ERR_INVALID_ARGUMENT;
  if (batch == 0) return GDN_OK;
  if (!q || !k || !v || !a || !beta || !pool || !slot_idx || !o || num_slots < 1)
    return GDN_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {q, k, v, a, beta, pool, o};
  for (const void* p : ptrs)
    if (!aligned16(p)) return GDN_ERR_INVALID_ARGUMENT;
  if ((int64_t)batch * cfg->num_v_heads * (cfg->head_dim_v / 32) > INT32_MAX)
    return GDN_ERR_UNSUPPORTED;
  if (!h) return GDN_ERR_INVALID_ARGUMENT;
  gdn::DecodeArgs da;
  da.q = q; da.k = k; da.v = v; da.a = a; da.beta = beta;
  da.pool = pool; da.slot = slot_idx; da.o = o;
  da.batch = batch;
  da.hk_heads = cfg->num_k_heads;
  da.hv_heads = cfg->num_v_heads;
  da.group = cfg->num_v_heads / cfg->num_k_heads;
  da.scale = cfg->scale;
  da.l2norm = cfg->qk_l2norm ? 1 : 0;
  da.gate_mode = cfg->gate_mode;
  da.a_log = cfg->a_log;
  da.dt_bias = cfg->dt_bias;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return GDN_ERR_CUDA;
  if (prev != h->device && cudaSetDevice(h->device) != cudaSuccess) return GDN_ERR_CUDA;
  int e = gdn::launch_decode(da, cfg->head_dim_k, cfg->io_dtype == GDN_BF16, stream);
  if (prev != h->device) cudaSetDevice(prev);
  return e == 0 ? GDN_OK : GDN_ERR_CUDA;
}

int32_t gdn_ckpt_position(int32_t len, int32_t block, int32_t tail) {
  if (len <= 0 || block <= 0 || tail < 0) return 0;
  int32_t p = (len / block) * block;
  if (p > len - tail) p -= block;
  return p > 0 ? p : 0;
}

int32_t gdn_mixed_budget(int32_t num_waiting, const int32_t* remaining, int32_t budget,
                         int32_t max_prompts, int32_t* take) {
  if (num_waiting < 0 || budget < 0 || max_prompts < 0) return -1;
  if (num_waiting > 0 && (!remaining || !take)) return -1;
  int32_t left = budget, served = 0;
  for (int32_t i = 0; i < num_waiting; ++i) {
    take[i] = 0;
    if (remaining[i] < 0) return -1;
    if (i >= max_prompts || left <= 0) continue;
    const int32_t t = std::min(remaining[i], left);
    take[i] = t;
    left -= t;
    if (t > 0) ++served;
  }
  return served;
}

}  // extern "C"

// ---- planning helpers for the allocation-free entry point (gdn_noalloc.cu) -------------

namespace gdn {

gdn_status plan_prefill(const gdn_handle* h, const gdn_config* cfg, int32_t num_seqs,
                        const int32_t* cu, const int32_t* ckpt_cu, const int32_t* ckpt_pos,
                        PrefillPlan* out) {
  KernelFamily fam;
  ListLayout L;
  int32_t num_ckpt = 0;
  gdn_status s = plan(const_cast<gdn_handle*>(h), cfg, num_seqs, cu, ckpt_cu, ckpt_pos, &fam,
                      &L, &num_ckpt);
  if (s != GDN_OK) return s;
  out->family = fam;
  out->units_off = L.units_off;
  out->seqs_off = L.seqs_off;
  out->pos_off = L.pos_off;
  out->ready_off = L.ready_off;
  out->bytes = L.total;
  out->num_units = L.num_units;
  out->num_ckpt = num_ckpt;
  return GDN_OK;
}

void write_worklist(void* dst, const PrefillPlan& plan, const gdn_config* cfg, int32_t num_seqs,
                    const int32_t* cu, const int32_t* ckpt_cu, const int32_t* ckpt_pos) {
  ListLayout L;
  L.units_off = plan.units_off;
  L.seqs_off = plan.seqs_off;
  L.pos_off = plan.pos_off;
  L.ready_off = plan.ready_off;
  L.total = plan.bytes;
  L.num_units = plan.num_units;
  build_worklist(dst, L, static_cast<KernelFamily>(plan.family), cfg, num_seqs, cu, ckpt_cu,
                 ckpt_pos, plan.num_ckpt);
}

}  // namespace gdn
