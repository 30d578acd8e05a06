// moe_dispatch_noalloc: the dispatch (capacity drop + pack) for callers that cannot allocate
// device memory, so cannot hold a workspace. Its scratch (per-chunk histograms and queue bases,
// per-expert totals and offsets) lives in a fixed array inside this library instead.
//
// The array is a file-scope __device__ object: every GPU that loads the library holds its own
// copy until the process exits. Host code cannot use the array's name as a device address, so the
// first call on each device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it; kernels get that pointer. Every region of the array is fully written by
// one kernel of a call before a later kernel of the same call reads it, and the scan's ticket
// counter returns to zero at the end of each call, so no clearing is needed; two calls that
// overlap on the GPU share the array and race.
#include <mutex>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB per device
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_dispatch_scratch[kNoAllocScratchBytes];

static std::mutex g_scratch_mu;
static void* g_scratch_ptr[kNoAllocMaxDevices] = {nullptr};

static size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// Device address of this device's scratch array (looked up once per device).
static cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace moe

using namespace moe;

extern "C" MOE_API moe_status_t moe_dispatch_noalloc(const moe_config_t* cfg, const void* x,
                                                     const int32_t* topk_idx, int32_t* counts,
                                                     int32_t* offsets, int32_t* slot_of,
                                                     int32_t* row_token, void* x_packed,
                                                     moe_stream_t stream) {
  Problem p;
  const moe_status_t st = make_problem(cfg, &p);
  if (st != MOE_OK) return st;
  if (!offsets) return MOE_ERR_INVALID_ARG;
  if (p.Tu > 0 && (!x || !topk_idx || !slot_of || !row_token || !x_packed)) return MOE_ERR_INVALID_ARG;
  const size_t E = (size_t)p.E;
  const size_t hist_bytes = align256((size_t)p.nchunks * E * 4);
  // [ticket (256 B) | counts | offsets | chunk histograms | chunk bases]; the ticket is zero at
  // load time and the scan's last block resets it, so it is zero at the start of every call
  const size_t off_ticket = 0, off_counts = 256, off_offsets = off_counts + align256(E * 4);
  const size_t off_hist = off_offsets + align256((E + 1) * 4);
  const size_t off_base = off_hist + hist_bytes;
  if (off_base + hist_bytes > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;

  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return MOE_ERR_CUDA;
  char* sc = static_cast<char*>(base);
  DispatchScratch d;
  d.ticket = reinterpret_cast<unsigned int*>(sc + off_ticket);
  d.counts = reinterpret_cast<int32_t*>(sc + off_counts);
  d.offsets = reinterpret_cast<int32_t*>(sc + off_offsets);
  d.chunk_hist = reinterpret_cast<int32_t*>(sc + off_hist);
  d.chunk_base = reinterpret_cast<int32_t*>(sc + off_base);
  d.status = nullptr;  // no workspace, so no status word: bad picks only get slot -1
  return launch_dispatch_from_idx(p, x, topk_idx, counts, offsets, slot_of, row_token, x_packed, d,
                                  (cudaStream_t)stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
