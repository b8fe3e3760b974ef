// decode_no_alloc.cu -- decode attention for callers that cannot allocate
// device memory.
//
// pkx_decode_attention_fwd needs a caller-provided workspace (the device-built
// work list and the split-KV partial results).  Some callers have no way to
// provide one: a plugin inside a host framework that owns every device
// allocation and hands out no allocator, code that must not call cudaMalloc
// because cudaMalloc synchronises the device and stalls a latency-critical
// decode loop, or a runtime whose memory is fixed at start-up.  This entry
// point takes the same inputs and outputs but no workspace: its scratch is
// the file-scope device array below, of fixed size kNoAllocScratchBytes.
//
// Properties:
//  * The array lives in this library's device image: every GPU that loads
//    this code holds its 96 MiB until the process exits.
//  * Host code cannot use the array's name as a device address; the first
//    call on each device (with that device current) looks the address up with
//    cudaGetSymbolAddress and caches it.  Make that first call before any
//    stream capture begins.
//  * Every call shares the one array, and the array keeps the last call's
//    contents.  The only state a call relies on being reset (the status word
//    and the work-list header) is rewritten by the call's own first kernel,
//    so a call never sees a previous call's data.  Two calls whose kernels
//    overlap on the GPU (different streams, or threads without ordering)
//    race on the array and corrupt each other's results: serialise them.
//  * Problems whose scratch would not fit are rejected before anything is
//    enqueued, with PKX_EWORKSPACE and a message giving both sizes.
//  * No cudaMalloc, cudaFree or other allocating routine is called.
//  * Device-side errors (an index outside the pool, a bounded wait that ran
//    out) land in the status word at the start of the array, as they do in
//    a caller's workspace; pkx_decode_no_alloc_status reads it back.
//  * The cached address belongs to the device's primary context.  After
//    cudaDeviceReset (or anything else that destroys and re-creates that
//    context) it is stale, and this entry point must not be called again in
//    the process.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "pkx_internal.h"

namespace pkx {

constexpr size_t kNoAllocScratchBytes = size_t(96) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_no_alloc_scratch[kNoAllocScratchBytes];

static std::mutex g_scratch_mu;
static void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device).  Returns PKX_OK or an error code with the message set.
static int scratch_for_current_device(void **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(PKX_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(PKX_EUNSUPPORTED, "device index %d beyond %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
    if (e != cudaSuccess || !p)
      return set_error(PKX_ECUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PKX_OK;
}

}  // namespace pkx

using namespace pkx;

extern "C" int pkx_decode_attention_fwd_no_alloc(
    const void *q, void *o, const void *k_buffer, const void *v_buffer,
    const int32_t *kv_indptr, const int32_t *kv_indices, int batch, int hq, int hkv, int lq,
    int lv, int64_t kb_ss, int64_t kb_sh, int64_t vb_ss, int64_t vb_sh, int64_t num_slots,
    float sm_scale, float logit_cap, int sliding_window, float *lse_out, void *stream) {
  if (batch < 0) return set_error(PKX_EINVAL, "negative batch");
  if (batch == 0) return PKX_OK;
  // the smallest workspace decode takes (one key stream per unit); the
  // call runs two streams when the scratch also holds their slots
  const size_t need = pkx_decode_workspace_min_size(batch, hq, hkv, lq, lv);
  if (need == 0) return set_error(PKX_EINVAL, "bad head configuration (hq=%d, hkv=%d)", hq, hkv);
  if (need > kNoAllocScratchBytes)
    return set_error(PKX_EWORKSPACE,
                     "decode problem needs %zu bytes of scratch; the built-in scratch holds %zu",
                     need, kNoAllocScratchBytes);
  void *scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc != PKX_OK) return rc;
  return pkx_decode_attention_fwd(q, o, k_buffer, v_buffer, kv_indptr, kv_indices, batch, hq, hkv,
                                  lq, lv, kb_ss, kb_sh, vb_ss, vb_sh, num_slots, sm_scale,
                                  logit_cap, sliding_window, 0, 1.0f, 1.0f, lse_out, scratch,
                                  kNoAllocScratchBytes, stream);
}

// The built-in scratch starts with the same header as a caller's workspace,
// so its status word is read the way pkx_workspace_status reads one.  On a
// device where no allocation-free call has run yet there is nothing to
// report.
extern "C" int pkx_decode_no_alloc_status(void *stream) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(PKX_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(PKX_EUNSUPPORTED, "device index %d beyond %d", dev, kMaxDevices);
  void *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    scratch = g_scratch_ptr[dev];
  }
  if (!scratch) return PKX_OK;
  return pkx_workspace_status(scratch, stream);
}
