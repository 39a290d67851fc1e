// noalloc.cu -- kda_chunk_forward_split_noalloc: the split chunked forward for callers that
// cannot allocate device memory while it runs.
//
// Some callers cannot allocate during the call: a serving loop that carves its memory up once
// at start-up, code running where an allocation could stall, fail or be forbidden at the wrong
// moment.  For them the split form's per-chunk operands go to one fixed array in device memory
// instead of cudaMallocAsync scratch.  The array lives in this translation unit alone, so under
// the runtime's lazy module loading only a process that calls this entry point reserves it (on
// each GPU where it is called, until the process exits); it is kept modest, inputs longer than
// it holds run as consecutive segments of chunks, and only the number of sequences B * H is
// bounded (see kda_chunk_forward_split_noalloc in kda.h).
#include <mutex>

#include "common.cuh"

namespace kda {

bool chunk_split_fits(const ChunkArgs& a, size_t bytes);
cudaError_t run_chunk_split_in(const ChunkArgs& a, cudaStream_t s, void* scratch, size_t bytes);
cudaError_t current_context_id(unsigned long long* id);

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
static __device__ __align__(256) uint8_t g_kda_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of the array on the current device.  In host code the array's name stands
// for a host-side shadow, not a device address, so the address is looked up with
// cudaGetSymbolAddress with the device current: once per device, on the first call made with
// it, and again only if that device's context has since been destroyed and created anew
// (cudaDeviceReset), since the array can then sit at another address.
cudaError_t noalloc_scratch(void** p) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    static unsigned long long ctx_of[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    unsigned long long ctx = 0;
    if ((e = current_context_id(&ctx)) != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || ctx == 0 || ctx != ctx_of[dev]) {
        void* q = nullptr;
        e = cudaGetSymbolAddress(&q, g_kda_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if ((e = current_context_id(&ctx)) != cudaSuccess) return e;  // now surely current
        addr[dev] = q;
        ctx_of[dev] = ctx;
    }
    *p = addr[dev];
    return cudaSuccess;
}

}  // namespace

// The split form on the fixed array.  *fits = false (nothing launched) when one segment of a
// chunk per sequence does not fit in it.  Nothing in the array needs clearing: every byte a
// call reads was written earlier by the same call.
cudaError_t launch_chunk_split_noalloc(const ChunkArgs& a, cudaStream_t s, bool* fits) {
    *fits = chunk_split_fits(a, kNoAllocScratchBytes);  // checked before any CUDA call
    if (!*fits) return cudaSuccess;
    void* p = nullptr;
    const cudaError_t e = noalloc_scratch(&p);
    if (e != cudaSuccess) return e;
    return run_chunk_split_in(a, s, p, kNoAllocScratchBytes);
}

}  // namespace kda
