// gqa_decode_attn_static: the decode step without a plan, on a fixed array of static
// device memory instead of an allocated workspace.
//
// The source pages have no such call.  It serves callers that may not allocate device
// memory when they run the step: a serving loop that has given every free byte of HBM to
// its own KV pool (a cudaMalloc there would fail), a host runtime that does not let a
// library own device memory, or a step that must not pay the allocator's implicit
// synchronisation.  It runs the same kernels as gqa_decode_attn; only the place of
// the workspace differs.
//
// The array is one per device (the runtime gives every device its own copy of a
// __device__ variable) and lives while the library is loaded.  Each call lays out its
// workspace in it from offset 0 (RoPE tables first, then rotated queries and partials),
// so all calls on a device share it: they must not overlap on the device.  No
// region has to start at zero -- every one is written by the call before it is read --
// and the device error word is the caller's (or a scratch word nobody reads), so the
// array is never cleared.
#include <mutex>

#include "launch.h"

using namespace gqa;

namespace {

static_assert(GQA_STATIC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte regions");

// Per-device bookkeeping of the scratch: its device address once looked up, and which
// RoPE tables (theta, capacity in positions) its first bytes hold.
struct ScratchState {
  bool ready = false;
  void *base = nullptr;
  bool tab_valid = false;
  float tab_theta = 0.f;
  int tab_rows = 0;
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
ScratchState g_state[kMaxDevices];

}  // namespace

// The workspace of every gqa_decode_attn_static call on a device.
static __device__ __align__(256) unsigned char g_scratch[GQA_STATIC_SCRATCH_BYTES];

namespace {

// First call on the current device: the scratch's address and the kernels' shared-memory
// limits (the same limits gqa_plan_create sets).  Called with g_mu held.
gqa_status_t set_up(ScratchState &s) {
  if (s.ready) return GQA_OK;
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return GQA_ERR_CUDA;
  }
  if (attn_configure(8) != cudaSuccess || attn_configure(16) != cudaSuccess ||
      configure_small_kernels() != cudaSuccess) {
    cudaGetLastError();
    return GQA_ERR_CUDA;
  }
  s.base = p;
  s.ready = true;
  return GQA_OK;
}

}  // namespace

extern "C" gqa_status_t gqa_decode_attn_static(const gqa_plan_desc_t *desc, const void *q_new, const void *k_new,
                                               const void *v_new, void *k_cache, void *v_cache,
                                               const int32_t *page_table, const int32_t *seq_lens,
                                               const int32_t *positions, const void *q_norm_w, const void *k_norm_w,
                                               float rope_theta, float eps, void *out, uint32_t *device_errors,
                                               void *stream) {
  if (!desc) return GQA_ERR_INVALID_ARG;
  const gqa_plan_desc_t d = *desc;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) return GQA_ERR_CUDA;
  if (d.device < 0 || d.device >= ndev) return GQA_ERR_INVALID_ARG;
  if (d.device >= kMaxDevices) return GQA_ERR_UNSUPPORTED;
  DeviceGuard guard(d.device);
  if (!guard.ok) return GQA_ERR_CUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d.device) != cudaSuccess) return GQA_ERR_CUDA;

  std::lock_guard<std::mutex> lk(g_mu);
  ScratchState &s = g_state[d.device];
  gqa_status_t st = set_up(s);  // before the layout: the step's form depends on the kernels' limits
  if (st != GQA_OK) return st;
  StepLayout lay;
  st = step_layout(d, sms, &lay);
  if (st != GQA_OK) return st;
  if (lay.total > GQA_STATIC_SCRATCH_BYTES) return GQA_ERR_SCRATCH_LIMIT;
  uint32_t *err = device_errors ? device_errors : reinterpret_cast<uint32_t *>(static_cast<char *>(s.base) + lay.off_err);
  // The binary32 table follows the binary64 one, so its place depends on max_seq_len:
  // reuse the tables only for the same theta and the same capacity.
  const bool table_ready = s.tab_valid && s.tab_theta == rope_theta && s.tab_rows == d.max_seq_len;
  st = run_step_at(d, lay, s.base, err, table_ready, q_new, k_new, v_new, k_cache, v_cache, page_table, seq_lens,
                   positions, q_norm_w, k_norm_w, rope_theta, eps, out, static_cast<cudaStream_t>(stream));
  if (st == GQA_OK) {
    // the tables now hold this theta for a max_seq_len capacity
    s.tab_valid = true;
    s.tab_theta = rope_theta;
    s.tab_rows = d.max_seq_len;
  } else if (st != GQA_ERR_INVALID_ARG) {
    s.tab_valid = false;  // a launch may have failed half-way through a rebuild
  }
  return st;
}
