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
// For K = V = 128 a persistent streaming kernel replaces it: one CTA of 16 warps per SM walks
// its share of the (b, h) pairs, and each pair's state (64 KB, contiguous) passes through a
// ring of three shared-memory stages: a bulk copy (TMA) brings pair i + 1 in and a bulk copy
// takes pair i - 1 out while pair i is computed in place, so the HBM sees reads and writes at
// all times instead of one CTA's burst of loads followed by its burst of stores.
//
// A second kernel with the same layout runs T > 1 consecutive tokens per launch
// (the fused recurrent form): the state is read once, kept in registers across the
// tokens and written once, so HBM sees 2 K V 4 bytes per (b, h) however many tokens
// are applied.  The single-token kernel stays separate: the token loop costs it
// registers and a barrier per token, which the bandwidth-bound T = 1 step cannot afford.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace kda {

__device__ int g_kda_decode_timeout;

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

namespace {
constexpr int kStreamThreads = 512;
constexpr int kStages = 3;
constexpr int kPairFloats = 128 * 128;
constexpr uint32_t kPairBytes = kPairFloats * 4u;
constexpr uint32_t kStreamSmem = kStages * kPairBytes + 5 * 128 * 4 + 2 * 16 * 32 * 16 + 64 + 1024;
}  // namespace

// The decode step for K = V = 128, streamed: CTA b takes pairs b, b + gridDim.x, ...  Thread
// (warp w, lane l) owns rows 8w .. 8w + 7 and columns 4l .. 4l + 3 of the pair's state in
// shared memory; the column sums over the key rows (S'^T k and S'^T q) combine the sixteen
// warps' partial sums through shared memory.
template <typename IO>
__global__ void __launch_bounds__(kStreamThreads, 1)
    decode_stream_kernel(int BH, int H, const IO* __restrict__ q, const IO* __restrict__ k,
                         const IO* __restrict__ v, const IO* __restrict__ z,
                         const IO* __restrict__ beta, const float* __restrict__ A_log,
                         const float* __restrict__ dt_bias, float scale, float* __restrict__ state,
                         IO* __restrict__ out) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    float* stages = reinterpret_cast<float*>(sm);
    float* s_alpha = reinterpret_cast<float*>(sm + kStages * kPairBytes);
    float* s_k = s_alpha + 128;
    float* s_q = s_k + 128;
    float* s_v = s_q + 128;
    float* s_bu = s_v + 128;
    float4* s_red = reinterpret_cast<float4*>(s_bu + 128);  // [2][16][32]: S'^T k, S'^T q partials
    uint64_t* bar = reinterpret_cast<uint64_t*>(s_red + 2 * 16 * 32);  // one per stage
    float* s_misc = reinterpret_cast<float*>(bar + kStages);          // k.q, beta, S'^T q spill

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int npairs = ((int)blockIdx.x < BH) ? (BH - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    auto pair_of = [&](int i) { return (size_t)blockIdx.x + (size_t)i * gridDim.x; };
    // pair i's state into stage i % kStages (thread 0 only), in four 16 KB pieces on one barrier
    auto issue_load = [&](int i) {
        const int st = i % kStages;
        float* dst = stages + (size_t)st * kPairFloats;
        const float* src = state + pair_of(i) * kPairFloats;
        tc::mbar_arrive_expect_tx(&bar[st], kPairBytes);
#pragma unroll
        for (int part = 0; part < 4; ++part)
            tc::bulk_load(dst + part * 4096, src + part * 4096, 16384u, &bar[st]);
    };
    if (tid == 0) {
        for (int st = 0; st < kStages; ++st) tc::mbar_init(&bar[st], 1);
        tc::fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0 && npairs > 0) issue_load(0);

    bool failed = false;
    int i = 0;
    for (; i < npairs; ++i) {
        const int st = i % kStages;
        const size_t bh = pair_of(i);
        const int h = (int)(bh % H);
        // the next pair's load goes to the stage pair i - 2 used: its store must have finished
        // reading shared memory (all store groups but pair i - 1's)
        if (tid == 0 && i + 1 < npairs) {
            tc::bulk_wait_read_all_but_one();
            issue_load(i + 1);
        }
        // this pair's vectors, while its state is in flight
        if (tid < 128) {
            const size_t idx = bh * 128 + tid;
            s_alpha[tid] = expf(kda_log_decay(ld_io(z + idx), dt_bias[(size_t)h * 128 + tid], expf(A_log[h])));
            s_k[tid] = ld_io(k + idx);
            s_q[tid] = scale * ld_io(q + idx);  // the read scale is folded into q
            s_v[tid] = ld_io(v + idx);
        } else if (tid == 128) {
            s_misc[1] = ld_io(beta + bh);
        }
        const bool ok = tid != 0 || tc::mbar_wait(&bar[st], (uint32_t)((i / kStages) & 1));
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        if (warp == 15) {
            float kq = 0.f;
#pragma unroll
            for (int c = lane; c < 128; c += 32) kq = fmaf(s_k[c], s_q[c], kq);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
            if (lane == 0) s_misc[0] = kq;
        }
        // S' = diag(alpha) S, kept in registers, and this warp's partial column sums
        float* S = stages + (size_t)st * kPairFloats;
        float4 x[8];
        float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int r = 8 * warp + j;
            const float4 sv = *reinterpret_cast<const float4*>(S + r * 128 + 4 * lane);
            const float a = s_alpha[r], kr = s_k[r], qr = s_q[r];
            x[j] = make_float4(sv.x * a, sv.y * a, sv.z * a, sv.w * a);
            pk.x = fmaf(x[j].x, kr, pk.x); pk.y = fmaf(x[j].y, kr, pk.y);
            pk.z = fmaf(x[j].z, kr, pk.z); pk.w = fmaf(x[j].w, kr, pk.w);
            pq.x = fmaf(x[j].x, qr, pq.x); pq.y = fmaf(x[j].y, qr, pq.y);
            pq.z = fmaf(x[j].z, qr, pq.z); pq.w = fmaf(x[j].w, qr, pq.w);
        }
        s_red[warp * 32 + lane] = pk;
        s_red[(16 + warp) * 32 + lane] = pq;
        __syncthreads();
        // column c: beta u_c = beta (v_c - (S'^T k)_c) and (S'^T q)_c
        float oq = 0.f;
        if (tid < 256) {
            const int which = tid >> 7, c = tid & 127;
            const float* red = reinterpret_cast<const float*>(s_red) + which * 16 * 128 + c;
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < 16; ++w) sum += red[w * 128];
            if (which == 0) s_bu[c] = s_misc[1] * (s_v[c] - sum);
            else oq = sum;
        }
        __syncthreads();
        // o = S''^T (scale q) = S'^T q + beta u (k . q); S'' = S' + beta k u^T, in place
        if (tid >= 128 && tid < 256) {
            const int c = tid - 128;
            st_io(out + bh * 128 + c, fmaf(s_bu[c], s_misc[0], oq));
        }
        const float4 bu = *reinterpret_cast<const float4*>(s_bu + 4 * lane);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int r = 8 * warp + j;
            const float kr = s_k[r];
            *reinterpret_cast<float4*>(S + r * 128 + 4 * lane) =
                make_float4(fmaf(bu.x, kr, x[j].x), fmaf(bu.y, kr, x[j].y), fmaf(bu.z, kr, x[j].z),
                            fmaf(bu.w, kr, x[j].w));
        }
        tc::fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            float* dst = state + bh * kPairFloats;
#pragma unroll
            for (int part = 0; part < 4; ++part) tc::bulk_store(dst + part * 4096, S + part * 4096, 16384u);
            tc::bulk_commit();
        }
    }
    if (tid == 0) {
        if (failed) {
            atomicExch(&g_kda_decode_timeout, 1);
            // the load issued for the next pair may still be in flight: a bounded wait for it
            if (i + 1 < npairs)
                tc::mbar_wait(&bar[(i + 1) % kStages], (uint32_t)(((i + 1) / kStages) & 1), 200000000ull);
        }
        tc::bulk_wait_all();  // every store has completed before the CTA's shared memory goes
    }
}

cudaError_t read_and_clear_decode_timeout(int* timed_out) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_kda_decode_timeout, sizeof(int));
    if (e != cudaSuccess) return e;
    *timed_out = v;
    if (v) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_kda_decode_timeout, &zero, sizeof(int));
    }
    return e;
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
    if (a.K == 128 && a.V == 128) {
        int dev = 0, nsm = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        const int BH = a.B * a.H;
        const unsigned sgrid = (unsigned)(BH < nsm ? BH : nsm);
        if (a.io == KDA_BF16) {
            e = cudaFuncSetAttribute(decode_stream_kernel<__nv_bfloat16>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStreamSmem);
            if (e != cudaSuccess) return e;
            decode_stream_kernel<__nv_bfloat16><<<sgrid, kStreamThreads, kStreamSmem, s>>>(
                BH, a.H, (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k,
                (const __nv_bfloat16*)a.v, (const __nv_bfloat16*)a.z, (const __nv_bfloat16*)a.beta,
                a.A_log, a.dt_bias, a.scale, a.state, (__nv_bfloat16*)a.out);
        } else {
            e = cudaFuncSetAttribute(decode_stream_kernel<float>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStreamSmem);
            if (e != cudaSuccess) return e;
            decode_stream_kernel<float><<<sgrid, kStreamThreads, kStreamSmem, s>>>(
                BH, a.H, (const float*)a.q, (const float*)a.k, (const float*)a.v,
                (const float*)a.z, (const float*)a.beta, a.A_log, a.dt_bias, a.scale, a.state,
                (float*)a.out);
        }
        count_launches(1);
        return cudaGetLastError();
    }
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
