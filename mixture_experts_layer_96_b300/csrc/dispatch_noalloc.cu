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

// Kernels of the regular dispatch (dispatch.cu), launched here on the static scratch.
__global__ void dispatch_hist_kernel(const int32_t* __restrict__ idx, int64_t Tu, int K, int E,
                                     int32_t* __restrict__ chunk_hist, uint32_t* status);
__global__ void dispatch_scan_kernel(const int32_t* __restrict__ chunk_hist, int64_t nchunks, int E,
                                     int64_t C, int32_t* __restrict__ chunk_base,
                                     int32_t* __restrict__ counts_ws, int32_t* __restrict__ offsets_ws,
                                     int32_t* counts_out, int32_t* offsets_out, unsigned int* ticket);
__global__ void dispatch_rank_kernel(const int32_t* __restrict__ idx, int64_t Tu, int K, int E, int64_t C,
                                     const int32_t* __restrict__ chunk_base,
                                     const int32_t* __restrict__ offsets, int32_t* __restrict__ slot_of,
                                     int32_t* __restrict__ row_token, int64_t rows);
__global__ void dispatch_gather_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ row_token,
                                       const int32_t* __restrict__ offsets, int E, int64_t row_vecs,
                                       uint4* __restrict__ x_packed);
__global__ void dispatch_gather_scalar_kernel(const unsigned char* __restrict__ x,
                                              const int32_t* __restrict__ row_token,
                                              const int32_t* __restrict__ offsets, int E,
                                              int64_t row_bytes, unsigned char* __restrict__ x_packed);

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
  unsigned int* ticket = reinterpret_cast<unsigned int*>(sc + off_ticket);
  int32_t* counts_ws = reinterpret_cast<int32_t*>(sc + off_counts);
  int32_t* offsets_ws = reinterpret_cast<int32_t*>(sc + off_offsets);
  int32_t* chunk_hist = reinterpret_cast<int32_t*>(sc + off_hist);
  int32_t* chunk_base = reinterpret_cast<int32_t*>(sc + off_base);
  const cudaStream_t s = (cudaStream_t)stream;

  const unsigned nch = (unsigned)(p.nchunks > 0 ? p.nchunks : 0);
  if (nch > 0) {
    dispatch_hist_kernel<<<nch, kChunk, 0, s>>>(topk_idx, p.Tu, p.K, p.E, chunk_hist, nullptr);
    note_launch();
  }
  dispatch_scan_kernel<<<p.E, 256, 0, s>>>(chunk_hist, p.nchunks, p.E, p.C, chunk_base, counts_ws,
                                          offsets_ws, counts, offsets, ticket);
  note_launch();
  dispatch_rank_kernel<<<nch > 0 ? nch : 1, kChunk, 0, s>>>(topk_idx, p.Tu, p.K, p.E, p.C, chunk_base,
                                                           offsets_ws, slot_of, row_token, p.rows);
  note_launch();
  if (p.rows > 0) {
    const int64_t row_bytes = (int64_t)p.hu * (int64_t)p.elt;
    int64_t blocks = (p.rows * (row_bytes / 16) + 1023) / 1024;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks < 1) blocks = 1;
    if (blocks > cap) blocks = cap;
    if (row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(x_packed) & 15) == 0) {
      dispatch_gather_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint4*>(x), row_token,
                                                             offsets_ws, p.E, row_bytes / 16,
                                                             static_cast<uint4*>(x_packed));
    } else {
      dispatch_gather_scalar_kernel<<<(unsigned)blocks, 256, 0, s>>>(
          static_cast<const unsigned char*>(x), row_token, offsets_ws, p.E, row_bytes,
          static_cast<unsigned char*>(x_packed));
    }
    note_launch();
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
