// mla_static.cu — hs_sparse_mla_fwd_static: the sparse MLA forward with its scratch in a
// fixed device array that belongs to the library, for callers that cannot allocate device
// memory themselves.
//
// The split-work path of hs_sparse_mla_fwd keeps, for every query whose tiles are divided between
// SMs, per-SM partial results that a merge kernel combines; that scratch normally comes from the
// caller (hs_mla_args.workspace). Some callers cannot provide it: their device memory belongs to
// another allocator (a serving engine's pooled allocator, a runtime with a fixed memory budget),
// or they run where an allocation, which may synchronise the device, is not allowed. This entry
// point takes the scratch from g_scratch below instead and allocates nothing.
//
// Rules of the array:
//  - kStaticScratchBytes (24 MiB) on every GPU that loads the library, held until the process
//    exits; a call whose split path would need more (a device with more SMs than 24 MiB covers)
//    is rejected with HS_ERR_UNSUPPORTED.
//  - All calls share it and it keeps the last call's contents. Nothing in it has to start at zero:
//    a call writes every slot it reads before reading it. Calls that overlap on the GPU (two
//    streams, or two host threads) race on it; a caller must order them.
//  - The host needs the array's device address, which is not the address of the host-side symbol.
//    The first call on each device looks it up with cudaGetSymbolAddress while that device is
//    current and caches it; make that first call before capturing a stream. The cache is keyed
//    by device ordinal for the life of the process: after cudaDeviceReset, or from a different
//    driver context on the same device, the cached address is stale, so this entry point must not
//    be used in a process that does either.
#include <mutex>

#include "common.cuh"

namespace hs {
uint64_t mla_workspace_bytes(int32_t H, int sms);
hs_status set_last_error(hs_status s, const char* fmt, ...);  // hs_last_error() text; returns s
}  // namespace hs

namespace {

constexpr uint64_t kStaticScratchBytes = 24ull << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_scratch[kStaticScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices];  // device address of g_scratch on each device, once looked up

}  // namespace

extern "C" {

hs_status hs_sparse_mla_fwd_static(const hs_mla_args* a, hs_stream_t stream) {
  if (!a) return hs::set_last_error(HS_ERR_INVALID, "args is NULL");
  if (a->H < 1 || a->H > 64) return hs::set_last_error(HS_ERR_INVALID, "H must be in [1, 64] (got %d)", a->H);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return hs::set_last_error(HS_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return hs::set_last_error(HS_ERR_UNSUPPORTED, "device ordinal %d is beyond the %d this call serves", dev,
                              kMaxDevices);
  const uint64_t need = hs::mla_workspace_bytes(a->H, sms);
  if (need > kStaticScratchBytes)
    return hs::set_last_error(HS_ERR_UNSUPPORTED,
                              "H = %d on %d SMs needs %llu bytes of scratch; the static scratch holds %llu", a->H,
                              sms, (unsigned long long)need, (unsigned long long)kStaticScratchBytes);
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {  // first call on this device: its address of the array
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_scratch);
      if (e != cudaSuccess || !p)
        return hs::set_last_error(HS_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed: %s",
                                  cudaGetErrorString(e));
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  // everything else (argument checks, launches) is hs_sparse_mla_fwd with this workspace
  hs_mla_args b = *a;
  b.workspace = scratch;
  b.workspace_bytes = kStaticScratchBytes;
  return hs_sparse_mla_fwd(&b, stream);
}

}  // extern "C"
