// common.cuh -- small device helpers shared by the libkda kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// I/O element loads and stores for the two supported dtypes.
__device__ __forceinline__ float ld_io(const float* p) { return *p; }
__device__ __forceinline__ float ld_io(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_io(float* p, float x) { *p = x; }
__device__ __forceinline__ void st_io(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// softplus(x) = log(1 + e^x) = max(x, 0) + log1p(e^{-|x|}); neither term overflows.
__device__ __forceinline__ float softplus_f32(float x) {
    return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x)));
}

// The KDA decay gate, log domain: g = -exp(A_log) * softplus(z + dt_bias) <= 0
// (kdafix-2026-10-02, "Fix 1": softplus first, then the -exp(A_log) multiplier).
__device__ __forceinline__ float kda_log_decay(float z, float dt_bias, float exp_A) {
    return -(exp_A * softplus_f32(z + dt_bias));
}

// Launch-side argument bundle used by the internal launchers.
struct ChunkArgs {
    int B, H, T, K, V, chunk;
    kda_dtype io;
    const void *q, *k, *v, *z, *beta;
    const float *A_log, *dt_bias, *h0;
    float scale;
    void* out;
    float* hT;
};

struct StepArgs {
    int B, H, K, V;
    kda_dtype io;
    const void *q, *k, *v, *z, *beta;
    const float *A_log, *dt_bias;
    float scale;
    float* state;
    void* out;
};

// Arguments of the backward (chunk_bwd.cu); gradients are float32.
struct BwdLaunch {
    int B, H, T, K, V;
    kda_dtype io;
    const void *q, *k, *v, *z, *beta, *d_o;
    const float *A_log, *dt_bias, *h0, *dhT;
    float scale;
    float *dq, *dk, *dv, *dz, *dbeta, *dA_log, *ddt_bias, *dh0;
};

// Count `n` kernel launches (read through kda_launch_count()).
void count_launches(int n);

// Scratch of the library's calls, stream-ordered on `s`, from the library's own pool of the
// current device, which keeps freed blocks for the next call (pool.cu); scratch_release hands
// the pool's unused blocks back to the system.
cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t s);
cudaError_t scratch_free(void* p, cudaStream_t s);
cudaError_t scratch_release();

// Internal launchers (one per kernel family); each returns a cudaError_t from the launch.
cudaError_t launch_gate(int B, int H, int T, int K, kda_dtype zdt, const void* z,
                        const float* A_log, const float* dt_bias, int chunk, float* g,
                        cudaStream_t s);
cudaError_t launch_decode(const StepArgs& a, cudaStream_t s);
cudaError_t launch_recurrent(const StepArgs& a, int T, cudaStream_t s);
cudaError_t launch_chunk_simt(const ChunkArgs& a, cudaStream_t s);
cudaError_t launch_chunk_backward(const BwdLaunch& L, cudaStream_t s);

}  // namespace kda
