// gate.cu -- the KDA decay gate and its in-chunk cumulative sum.
//
// g[b,h,t,c] = -exp(A_log[h]) * softplus(z[b,h,t,c] + dt_bias[h,c])
// (kdafix-2026-10-02, "Fix 1 -- decay form"), optionally followed by the
// inclusive prefix sum over the tokens of each chunk, G_t = sum_{s<=t} g_s,
// the in-chunk cumulative log decay that the chunked form is written in
// (kda-adjoint-2026-10-01, section 2).
//
// One CTA per (b*h, chunk); thread c walks the chunk's tokens for key channel
// c, so every load and store of a token row is coalesced across the CTA.
// Bound: HBM (read z, write 4-byte g per element).
#include "common.cuh"

namespace kda {

template <typename IO>
__global__ void __launch_bounds__(128) gate_kernel(int H, int T, int K, const IO* __restrict__ z,
                                                   const float* __restrict__ A_log,
                                                   const float* __restrict__ dt_bias, int span,
                                                   int cumulative, float* __restrict__ g) {
    const int c = threadIdx.x;
    if (c >= K) return;
    const int bh = blockIdx.x;
    const int h = bh % H;
    const int t0 = blockIdx.y * span;
    const int t1 = min(t0 + span, T);
    const float exp_A = expf(A_log[h]);
    const float dt = dt_bias[(size_t)h * K + c];
    const size_t base = (size_t)bh * T * K;
    float acc = 0.0f;
    for (int t = t0; t < t1; ++t) {
        const size_t idx = base + (size_t)t * K + c;
        float gv = kda_log_decay(ld_io(z + idx), dt, exp_A);
        if (cumulative) {
            acc += gv;
            gv = acc;
        }
        g[idx] = gv;
    }
}

cudaError_t launch_gate(int B, int H, int T, int K, kda_dtype zdt, const void* z,
                        const float* A_log, const float* dt_bias, int chunk, float* g,
                        cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int span = chunk > 0 ? chunk : 64;
    dim3 grid(B * H, (T + span - 1) / span);
    if (zdt == KDA_BF16)
        gate_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(H, T, K, (const __nv_bfloat16*)z, A_log,
                                                        dt_bias, span, chunk > 0, g);
    else
        gate_kernel<float><<<grid, 128, 0, s>>>(H, T, K, (const float*)z, A_log, dt_bias, span,
                                                chunk > 0, g);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
