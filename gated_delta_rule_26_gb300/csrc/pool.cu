// pool.cu -- device scratch of the library's calls: one stream-ordered memory pool of its own per
// device.  The pool's release threshold is set so that freed blocks stay reserved for the next
// call: the device's default pool hands its free blocks back to the system at every
// synchronisation, so a caller that synchronises between calls had every call map its scratch
// again (the 6 GB of the prefill backward took as long as the kernel itself).  Calls on
// different streams still get separate blocks; a freed block is reused in stream order only.
#include <stdint.h>

#include <mutex>

#include "common.cuh"

namespace kda {

cudaError_t current_context_id(unsigned long long* id);  // chunk_tc.cu

namespace {

constexpr int kMaxDevices = 64;
struct PoolSlot {
    unsigned long long ctx = 0;  // the context the pool was created in
    cudaMemPool_t pool = nullptr;
};
std::mutex g_pool_mu;
PoolSlot g_pools[kMaxDevices];

// The pool of the current device, created on first use in this context.  A pool from a context
// that no longer exists (cudaDeviceReset) is replaced; it was destroyed with that context.
cudaError_t scratch_pool(cudaMemPool_t* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    unsigned long long ctx = 0;
    if ((e = current_context_id(&ctx)) != cudaSuccess) return e;
    if (ctx == 0) {  // no context yet on this thread: make the device's primary one current
        if ((e = cudaFree(nullptr)) != cudaSuccess) return e;
        if ((e = current_context_id(&ctx)) != cudaSuccess) return e;
    }
    std::lock_guard<std::mutex> lock(g_pool_mu);
    PoolSlot& slot = g_pools[dev];
    if (slot.pool && slot.ctx == ctx) {
        *out = slot.pool;
        return cudaSuccess;
    }
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if ((e = cudaMemPoolCreate(&pool, &props)) != cudaSuccess) return e;
    uint64_t keep = UINT64_MAX;
    if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
        cudaMemPoolDestroy(pool);
        return e;
    }
    slot.pool = pool;
    slot.ctx = ctx;
    *out = pool;
    return cudaSuccess;
}

}  // namespace

cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t s) {
    cudaMemPool_t pool = nullptr;
    const cudaError_t e = scratch_pool(&pool);
    if (e != cudaSuccess) return e;
    return cudaMallocFromPoolAsync(p, bytes, pool, s);
}

cudaError_t scratch_free(void* p, cudaStream_t s) { return cudaFreeAsync(p, s); }

cudaError_t scratch_release() {
    cudaMemPool_t pool = nullptr;
    cudaError_t e = scratch_pool(&pool);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return e;
    return cudaMemPoolTrimTo(pool, 0);
}

}  // namespace kda
