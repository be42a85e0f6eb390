// rx_decode_attn_noalloc: decode attention that allocates nothing and needs no caller workspace.
//
// Some callers cannot allocate device memory when they run attention: a host framework that hands
// a custom operator only its input and output buffers (no allocator handle), or a serving runtime
// that owns all device memory under a fixed budget and forbids allocation while requests are in
// flight.  For them this entry point keeps the decode plan's tables and partial results in a
// scratch array that is part of the library's own module: file-scope device memory, created when
// the library is loaded on a GPU and held by that GPU until the process exits.
//
// Set-up: the first call on a device, with that device current, looks up the array's device
// address with cudaGetSymbolAddress (a host-side name of the array is not a device address) and
// caches it for later calls on that device.  Make that first call before any stream capture.
//
// Sharing: every call uses the same array.  Each call first copies the plan's tables into it
// (through the plan's pinned staging buffer, as rx_plan_upload does for a workspace), which also
// resets the device status word to zero; the partial results need no clearing (each is written
// before it is read).  Two calls whose work overlaps on the GPU (different streams, or different
// host threads) race on the array and must not be issued.  A call's device-side errors stay in
// the array's status word until the next call: rx_noalloc_read_status reads them.
#include <cuda_runtime.h>

#include <mutex>

#include "rx_internal.h"

namespace {

constexpr size_t kScratchBytes = RX_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_setup;

// Device address of the scratch array on the current device (looked up once per device).
rx_status scratch_of_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return rx::set_error(RX_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return rx::set_error(RX_ERR_UNSUPPORTED, "rx_decode_attn_noalloc: device ordinal >= 64");
  std::lock_guard<std::mutex> lock(g_setup);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return rx::set_error(RX_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e)
                                                         : "scratch address is NULL");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return RX_OK;
}

}  // namespace

extern "C" rx_status rx_decode_attn_noalloc(const rx_plan* plan, const rx_kv_desc* desc,
                                            const void* k_pool, const void* v_pool,
                                            const void* q, void* o, float* lse,
                                            rx_stream_t stream) {
  void* scratch = nullptr;
  rx_status st = scratch_of_current_device(&scratch);
  if (st) return st;
  rx::PlanHeader h;
  st = rx::plan_for_noalloc(plan, desc, k_pool, v_pool, q, o, lse, scratch, kScratchBytes, &h);
  if (st) return st;
  // the tables go in from pinned memory, so the copy does not hold the host until the stream
  // drains (a copy straight from the plan's pageable buffer would)
  st = rx_plan_upload(plan, scratch, kScratchBytes, stream);
  if (st) return st;
  rx::AuxStream aux;
  st = rx::plan_aux_stream(plan, &aux);
  if (st) return st;
  const int le = rx::launch_decode(desc, &h, k_pool, v_pool, q, o, lse, scratch, stream, &aux);
  if (le) return rx::set_error(RX_ERR_CUDA, cudaGetErrorString((cudaError_t)le));
  return RX_OK;
}

extern "C" rx_status rx_noalloc_read_status(int32_t* status, rx_stream_t stream) {
  if (!status) return rx::set_error(RX_ERR_INVALID, "status is NULL");
  void* scratch = nullptr;
  rx_status st = scratch_of_current_device(&scratch);
  if (st) return st;
  return rx_read_status(scratch, status, stream);
}

extern "C" size_t rx_noalloc_scratch_bytes(void) { return kScratchBytes; }
