// decode.cu -- one KDA decode token per (b, h), state updated in place.
//
// Per (b, h) with state S (K x V, fp32, row c = key channel):
//     alpha = exp(-exp(A_log) softplus(z + dt_bias))           (kdafix "Fix 1")
//     S' = diag(alpha) S
//     u  = v - S'^T k
//     S'' = S' + beta k u^T
//     o  = S''^T (scale q) = S'^T (scale q) + beta u (k . scale q)   (kdafix "Fix 2")
// The two reductions over the key channels (S'^T k and S'^T q) share one pass
// over S, so S is read once and written once: 2 * K * V * 4 bytes per (b, h),
// the HBM floor of this step.
//
// Layout: the value columns of S are independent, so each (b, h) is split into
// two CTAs of 256 threads (8 warps), one per half of the V columns.  Lane l owns
// the two columns [2l, 2l + 2) of its half (one float2; a warp covers 256
// contiguous bytes of a row, fully coalesced), warp w owns the key rows
// [w * R, (w + 1) * R) with R = ceil(K / 8) <= 16, so a thread keeps at most 16
// float2 of S in registers between the read and the write.  The small register
// footprint lets four CTAs share an SM, so one CTA's reads overlap another's
// writes.  The per-column partial sums of the eight warps are combined through
// shared memory; k . q is a warp-shuffle reduction.
// State loads and stores use the streaming cache hints (the state is larger
// than L2 and touched once per step).
//
// A second kernel with the same layout runs T > 1 consecutive tokens per launch
// (the fused recurrent form): the state is read once, kept in registers across the
// tokens and written once, so HBM sees 2 K V 4 bytes per (b, h) however many tokens
// are applied.  The single-token kernel stays separate: the token loop costs it
// registers and a barrier per token, which the bandwidth-bound T = 1 step cannot afford.
#include "common.cuh"

namespace kda {

namespace {
constexpr int kDecodeThreads = 256;
constexpr int kDecodeWarps = kDecodeThreads / 32;
constexpr int kMaxRowsPerWarp = 16;  // K <= 128

__device__ __forceinline__ float2 f2_scale(float2 a, float s) { return make_float2(a.x * s, a.y * s); }
__device__ __forceinline__ float2 f2_fma(float2 a, float s, float2 c) {
    return make_float2(fmaf(a.x, s, c.x), fmaf(a.y, s, c.y));
}
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
}  // namespace

// Single token (T = 1): the bandwidth-critical decode step.
template <typename IO>
__global__ void __launch_bounds__(kDecodeThreads, 4)
    decode_kernel(int H, int K, int V, const IO* __restrict__ q, const IO* __restrict__ k,
                  const IO* __restrict__ v, const IO* __restrict__ z, const IO* __restrict__ beta,
                  const float* __restrict__ A_log, const float* __restrict__ dt_bias, float scale,
                  float* __restrict__ state, IO* __restrict__ out) {
    __shared__ float s_k[128], s_q[128], s_alpha[128], s_v[64];
    __shared__ float2 s_red_k[kDecodeWarps][32], s_red_q[kDecodeWarps][32];
    __shared__ float s_kq;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t bh = blockIdx.x >> 1;
    const int h = (int)(bh % H);
    const int Vh = V >> 1, j0 = (blockIdx.x & 1) * Vh;  // this CTA's half of the columns
    const int rows = (K + kDecodeWarps - 1) / kDecodeWarps;
    const int r0 = warp * rows;
    const bool col_ok = lane * 2 < Vh;
    float* S = state + bh * (size_t)K * V + j0;

    // Issue the state loads first: they are the long-latency part of the step.
    float2 s[kMaxRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kMaxRowsPerWarp; ++i) {
        const int r = r0 + i;
        if (i < rows && r < K && col_ok)
            s[i] = __ldcs(reinterpret_cast<const float2*>(S + (size_t)r * V + lane * 2));
        else
            s[i] = make_float2(0.f, 0.f);
    }

    if (tid < K) {
        const size_t idx = bh * K + tid;
        const float g = kda_log_decay(ld_io(z + idx), dt_bias[(size_t)h * K + tid], expf(A_log[h]));
        s_alpha[tid] = expf(g);
        s_k[tid] = ld_io(k + idx);
        s_q[tid] = scale * ld_io(q + idx);  // the read scale is folded into q
    }
    if (tid < Vh) s_v[tid] = ld_io(v + bh * V + j0 + tid);
    const float b = ld_io(beta + bh);
    __syncthreads();

    if (warp == 0) {
        float kq = 0.f;
        for (int c = lane; c < K; c += 32) kq = fmaf(s_k[c], s_q[c], kq);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
        if (lane == 0) s_kq = kq;
    }

    // S' = diag(alpha) S and the two partial column reductions of this warp's rows.
    float2 pk = make_float2(0.f, 0.f), pq = pk;
#pragma unroll
    for (int i = 0; i < kMaxRowsPerWarp; ++i) {
        const int r = r0 + i;
        if (i < rows && r < K) {
            s[i] = f2_scale(s[i], s_alpha[r]);
            pk = f2_fma(s[i], s_k[r], pk);
            pq = f2_fma(s[i], s_q[r], pq);
        }
    }
    s_red_k[warp][lane] = pk;
    s_red_q[warp][lane] = pq;
    __syncthreads();

    float2 tk = s_red_k[0][lane], tq = s_red_q[0][lane];
#pragma unroll
    for (int w = 1; w < kDecodeWarps; ++w) {
        tk = f2_add(tk, s_red_k[w][lane]);
        tq = f2_add(tq, s_red_q[w][lane]);
    }
    if (!col_ok) return;
    const float2 bu = make_float2(b * (s_v[lane * 2] - tk.x), b * (s_v[lane * 2 + 1] - tk.y));

#pragma unroll
    for (int i = 0; i < kMaxRowsPerWarp; ++i) {
        const int r = r0 + i;
        if (i < rows && r < K)
            __stcs(reinterpret_cast<float2*>(S + (size_t)r * V + lane * 2), f2_fma(bu, s_k[r], s[i]));
    }
    if (warp == 0) {
        const float2 o = f2_fma(bu, s_kq, tq);
        IO* op = out + bh * V + j0 + lane * 2;
        st_io(op + 0, o.x);
        st_io(op + 1, o.y);
    }
}

// T > 1 tokens per launch, state kept in registers between tokens.
template <typename IO>
__global__ void __launch_bounds__(kDecodeThreads, 3)
    recurrent_kernel(int H, int T, int K, int V, const IO* __restrict__ q,
                     const IO* __restrict__ k, const IO* __restrict__ v,
                     const IO* __restrict__ z, const IO* __restrict__ beta,
                     const float* __restrict__ A_log, const float* __restrict__ dt_bias,
                     float scale, float* __restrict__ state, IO* __restrict__ out) {
    __shared__ float s_k[128], s_q[128], s_alpha[128], s_v[64];
    __shared__ float2 s_red_k[kDecodeWarps][32], s_red_q[kDecodeWarps][32];
    __shared__ float s_kq, s_b;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t bh = blockIdx.x >> 1;
    const int h = (int)(bh % H);
    const int Vh = V >> 1, j0 = (blockIdx.x & 1) * Vh;  // this CTA's half of the columns
    const int rows = (K + kDecodeWarps - 1) / kDecodeWarps;
    const int r0 = warp * rows;
    const bool col_ok = lane * 2 < Vh;
    float* S = state + bh * (size_t)K * V + j0;
    const float exp_A = expf(A_log[h]);
    const float dt = tid < K ? dt_bias[(size_t)h * K + tid] : 0.f;

    // Issue the state loads first: they are the long-latency part of the step.  The state
    // stays in registers for all T tokens and is written back once.
    float2 s[kMaxRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kMaxRowsPerWarp; ++i) {
        const int r = r0 + i;
        if (i < rows && r < K && col_ok)
            s[i] = __ldcs(reinterpret_cast<const float2*>(S + (size_t)r * V + lane * 2));
        else
            s[i] = make_float2(0.f, 0.f);
    }

    for (int t = 0; t < T; ++t) {
        const size_t tok = bh * T + t;
        if (t > 0) __syncthreads();  // the previous token's vectors are no longer read
        if (tid < K) {
            const size_t idx = tok * K + tid;
            s_alpha[tid] = expf(kda_log_decay(ld_io(z + idx), dt, exp_A));
            s_k[tid] = ld_io(k + idx);
            s_q[tid] = scale * ld_io(q + idx);  // the read scale is folded into q
        }
        if (tid < Vh) s_v[tid] = ld_io(v + tok * V + j0 + tid);
        if (tid == 0) s_b = ld_io(beta + tok);
        __syncthreads();

        if (warp == 0) {
            float kq = 0.f;
            for (int c = lane; c < K; c += 32) kq = fmaf(s_k[c], s_q[c], kq);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
            if (lane == 0) s_kq = kq;
        }

        // S' = diag(alpha) S and the two partial column reductions of this warp's rows.
        float2 pk = make_float2(0.f, 0.f), pq = pk;
#pragma unroll
        for (int i = 0; i < kMaxRowsPerWarp; ++i) {
            const int r = r0 + i;
            if (i < rows && r < K) {
                s[i] = f2_scale(s[i], s_alpha[r]);
                pk = f2_fma(s[i], s_k[r], pk);
                pq = f2_fma(s[i], s_q[r], pq);
            }
        }
        s_red_k[warp][lane] = pk;
        s_red_q[warp][lane] = pq;
        __syncthreads();

        float2 tk = s_red_k[0][lane], tq = s_red_q[0][lane];
#pragma unroll
        for (int w = 1; w < kDecodeWarps; ++w) {
            tk = f2_add(tk, s_red_k[w][lane]);
            tq = f2_add(tq, s_red_q[w][lane]);
        }
        const float b = s_b;
        const float2 bu = col_ok ? make_float2(b * (s_v[lane * 2] - tk.x), b * (s_v[lane * 2 + 1] - tk.y))
                                 : make_float2(0.f, 0.f);
        // S'' = S' + beta k u^T
#pragma unroll
        for (int i = 0; i < kMaxRowsPerWarp; ++i) {
            const int r = r0 + i;
            if (i < rows && r < K) s[i] = f2_fma(bu, s_k[r], s[i]);
        }
        if (warp == 0 && col_ok) {
            const float2 o = f2_fma(bu, s_kq, tq);
            IO* op = out + tok * V + j0 + lane * 2;
            st_io(op + 0, o.x);
            st_io(op + 1, o.y);
        }
    }

    if (!col_ok) return;
#pragma unroll
    for (int i = 0; i < kMaxRowsPerWarp; ++i) {
        const int r = r0 + i;
        if (i < rows && r < K)
            __stcs(reinterpret_cast<float2*>(S + (size_t)r * V + lane * 2), s[i]);
    }
}

cudaError_t launch_recurrent(const StepArgs& a, int T, cudaStream_t s) {
    const unsigned grid = (unsigned)(a.B * a.H) * 2u;
    if (a.io == KDA_BF16)
        recurrent_kernel<__nv_bfloat16><<<grid, kDecodeThreads, 0, s>>>(
            a.H, T, a.K, a.V, (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k,
            (const __nv_bfloat16*)a.v, (const __nv_bfloat16*)a.z, (const __nv_bfloat16*)a.beta,
            a.A_log, a.dt_bias, a.scale, a.state, (__nv_bfloat16*)a.out);
    else
        recurrent_kernel<float><<<grid, kDecodeThreads, 0, s>>>(
            a.H, T, a.K, a.V, (const float*)a.q, (const float*)a.k, (const float*)a.v,
            (const float*)a.z, (const float*)a.beta, a.A_log, a.dt_bias, a.scale, a.state,
            (float*)a.out);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_decode(const StepArgs& a, cudaStream_t s) {
    const unsigned grid = (unsigned)(a.B * a.H) * 2u;
    if (a.io == KDA_BF16)
        decode_kernel<__nv_bfloat16><<<grid, kDecodeThreads, 0, s>>>(
            a.H, a.K, a.V, (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k,
            (const __nv_bfloat16*)a.v, (const __nv_bfloat16*)a.z, (const __nv_bfloat16*)a.beta,
            a.A_log, a.dt_bias, a.scale, a.state, (__nv_bfloat16*)a.out);
    else
        decode_kernel<float><<<grid, kDecodeThreads, 0, s>>>(
            a.H, a.K, a.V, (const float*)a.q, (const float*)a.k, (const float*)a.v,
            (const float*)a.z, (const float*)a.beta, a.A_log, a.dt_bias, a.scale, a.state,
            (float*)a.out);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
