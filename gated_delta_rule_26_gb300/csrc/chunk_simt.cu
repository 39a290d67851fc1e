// chunk_simt.cu -- the KDA chunked (WY) forward in fp32 on CUDA cores.
//
// This is the full-precision path: fp32 I/O shapes (tolerance 1e-4) and every
// shape the tensor-core path does not take.  All arithmetic is fp32 FFMA; no
// TF32, whose 10-bit mantissa cannot hold a 1e-4 relative bar.
//
// One CTA per (b, h, V-tile) walks the chunks of its sequence in order.  Per
// chunk of C tokens, with S (K x Vt, fp32) the state entering the chunk and
// G_t the in-chunk cumulative log decay (kda-adjoint-2026-10-01, section 2):
//   1. g = -exp(A_log) softplus(z + dt_bias), G = in-chunk prefix sum of g;
//   2. A[t,i] = beta_t sum_c k[t,c] k[i,c] exp(G[t,c] - G[i,c])   (i < t)
//      M[t,i] =        sum_c q[t,c] k[i,c] exp(G[t,c] - G[i,c])   (i <= t)
//      (every exponent is <= 0: the pairwise factor is formed directly, so
//      nothing overflows however strong the decay);
//   3. (I + A) [W | U] = [diag(beta)(K * Gamma) | diag(beta) V] by forward
//      substitution, one thread per column (columns are independent);
//   4. Delta = U - W S;  o = scale ((Q * Gamma) S + M Delta);
//   5. S <- diag(Gamma_last) S + (K * exp(G_last - G))^T Delta.
// A short last chunk is padded with k = q = v = beta = g = 0, which leaves
// every quantity of the real tokens unchanged.
#include <algorithm>

#include "common.cuh"

namespace kda {

namespace {
constexpr int kSimtThreads = 256;
constexpr int kMaxPerThread = 16;  // C * Vt / 256 <= 64 * 64 / 256

struct SimtSmem {
    int C, K, Vt, ldk;
    size_t off_k, off_q, off_g, off_w, off_v, off_a, off_m, off_s, off_b, off_gl, total_floats;
    __host__ __device__ SimtSmem(int C_, int K_, int Vt_) : C(C_), K(K_), Vt(Vt_) {
        ldk = K + 1;  // odd stride: column walks over rows hit distinct banks
        size_t o = 0;
        off_k = o; o += (size_t)C * ldk;
        off_q = o; o += (size_t)C * ldk;
        off_g = o; o += (size_t)C * ldk;
        off_w = o; o += (size_t)C * ldk;
        off_v = o; o += (size_t)C * Vt;
        off_a = o; o += (size_t)C * (C + 1);
        off_m = o; o += (size_t)C * (C + 1);
        off_s = o; o += (size_t)K * Vt;
        off_b = o; o += C;
        off_gl = o; o += K;
        total_floats = o;
    }
};
}  // namespace

template <typename IO>
__global__ void __launch_bounds__(kSimtThreads)
    chunk_simt_kernel(int H, int T, int K, int V, int C, int Vt, const IO* __restrict__ q,
                      const IO* __restrict__ k, const IO* __restrict__ v, const IO* __restrict__ z,
                      const IO* __restrict__ beta, const float* __restrict__ A_log,
                      const float* __restrict__ dt_bias, float scale, const float* __restrict__ h0,
                      IO* __restrict__ out, float* __restrict__ hT) {
    extern __shared__ float smem[];
    const SimtSmem L(C, K, Vt);
    float* sK = smem + L.off_k;   // k, then K * exp(G_last - G)
    float* sQ = smem + L.off_q;   // q, then Q * Gamma
    float* sG = smem + L.off_g;   // z -> g -> G
    float* sW = smem + L.off_w;   // W
    float* sV = smem + L.off_v;   // v -> U -> Delta
    float* sA = smem + L.off_a;
    float* sM = smem + L.off_m;
    float* sS = smem + L.off_s;   // state tile, fp32
    float* sB = smem + L.off_b;
    float* sGl = smem + L.off_gl; // G_last per channel
    const int ldk = L.ldk, lda = C + 1;

    const int tid = threadIdx.x;
    const size_t bh = blockIdx.x;
    const int h = (int)(bh % H);
    const int j0 = blockIdx.y * Vt;
    const int vt = min(Vt, V - j0);
    const float exp_A = expf(A_log[h]);

    for (int e = tid; e < K * Vt; e += kSimtThreads) {
        const int c = e / Vt, j = e % Vt;
        float s0 = 0.f;
        if (h0 && j < vt) s0 = h0[(bh * K + c) * V + j0 + j];
        sS[c * Vt + j] = s0;
    }

    for (int t0 = 0; t0 < T; t0 += C) {
        const int cn = min(C, T - t0);
        __syncthreads();  // previous chunk fully consumed
        // ---- 1. load and gate
        for (int e = tid; e < C * K; e += kSimtThreads) {
            const int t = e / K, c = e % K;
            float kv = 0.f, qv = 0.f, gv = 0.f;
            if (t < cn) {
                const size_t idx = (bh * T + t0 + t) * K + c;
                kv = ld_io(k + idx);
                qv = ld_io(q + idx);
                gv = kda_log_decay(ld_io(z + idx), dt_bias[(size_t)h * K + c], exp_A);
            }
            sK[t * ldk + c] = kv;
            sQ[t * ldk + c] = qv;
            sG[t * ldk + c] = gv;
        }
        for (int e = tid; e < C * Vt; e += kSimtThreads) {
            const int t = e / Vt, j = e % Vt;
            float vv = 0.f;
            if (t < cn && j < vt) vv = ld_io(v + (bh * T + t0 + t) * V + j0 + j);
            sV[t * Vt + j] = vv;
        }
        for (int t = tid; t < C; t += kSimtThreads) sB[t] = t < cn ? ld_io(beta + bh * T + t0 + t) : 0.f;
        __syncthreads();
        for (int c = tid; c < K; c += kSimtThreads) {
            float acc = 0.f;
            for (int t = 0; t < C; ++t) {
                acc += sG[t * ldk + c];
                sG[t * ldk + c] = acc;
            }
            sGl[c] = acc;
        }
        __syncthreads();

        // ---- 2. decay-folded strictly lower A (with beta) and lower M
        for (int p = tid; p < C * C; p += kSimtThreads) {
            const int t = p / C, i = p % C;
            float a = 0.f, m = 0.f;
            if (i <= t) {
                const float* kt = sK + t * ldk;
                const float* ki = sK + i * ldk;
                const float* qt = sQ + t * ldk;
                const float* gt = sG + t * ldk;
                const float* gi = sG + i * ldk;
                for (int c = 0; c < K; ++c) {
                    const float kd = ki[c] * expf(gt[c] - gi[c]);
                    a = fmaf(kt[c], kd, a);
                    m = fmaf(qt[c], kd, m);
                }
            }
            sA[t * lda + i] = (i < t) ? sB[t] * a : 0.f;
            sM[t * lda + i] = m;
        }
        __syncthreads();

        // ---- 3. forward substitution: columns of W (j < K) and U (j < Vt)
        for (int col = tid; col < K + Vt; col += kSimtThreads) {
            if (col < K) {
                const int c = col;
                for (int t = 0; t < C; ++t) {
                    float x = sB[t] * sK[t * ldk + c] * expf(sG[t * ldk + c]);
                    for (int i = 0; i < t; ++i) x = fmaf(-sA[t * lda + i], sW[i * ldk + c], x);
                    sW[t * ldk + c] = x;
                }
            } else {
                const int j = col - K;
                for (int t = 0; t < C; ++t) {
                    float x = sB[t] * sV[t * Vt + j];
                    for (int i = 0; i < t; ++i) x = fmaf(-sA[t * lda + i], sV[i * Vt + j], x);
                    sV[t * Vt + j] = x;
                }
            }
        }
        __syncthreads();
        // K~ = K * exp(G_last - G), Q * Gamma (the scale is applied at the output)
        for (int e = tid; e < C * K; e += kSimtThreads) {
            const int t = e / K, c = e % K;
            const float G = sG[t * ldk + c];
            sK[t * ldk + c] *= expf(sGl[c] - G);
            sQ[t * ldk + c] *= expf(G);
        }
        __syncthreads();

        // ---- 4. Delta = U - W S (in place over U), inter-chunk read (Q*Gamma) S
        float qs[kMaxPerThread];
#pragma unroll
        for (int r = 0; r < kMaxPerThread; ++r) {
            const int e = tid + r * kSimtThreads;
            qs[r] = 0.f;
            if (e < C * Vt) {
                const int t = e / Vt, j = e % Vt;
                float ws = 0.f, rq = 0.f;
                for (int c = 0; c < K; ++c) {
                    const float sv = sS[c * Vt + j];
                    ws = fmaf(sW[t * ldk + c], sv, ws);
                    rq = fmaf(sQ[t * ldk + c], sv, rq);
                }
                sV[t * Vt + j] -= ws;
                qs[r] = rq;
            }
        }
        __syncthreads();
        // o = scale ((Q Gamma) S + M Delta)
#pragma unroll
        for (int r = 0; r < kMaxPerThread; ++r) {
            const int e = tid + r * kSimtThreads;
            if (e < C * Vt) {
                const int t = e / Vt, j = e % Vt;
                float acc = qs[r];
                for (int i = 0; i <= t; ++i) acc = fmaf(sM[t * lda + i], sV[i * Vt + j], acc);
                if (t < cn && j < vt) st_io(out + (bh * T + t0 + t) * V + j0 + j, scale * acc);
            }
        }
        // ---- 5. S <- diag(Gamma_last) S + K~^T Delta
        for (int e = tid; e < K * Vt; e += kSimtThreads) {
            const int c = e / Vt, j = e % Vt;
            float acc = expf(sGl[c]) * sS[c * Vt + j];
            for (int t = 0; t < C; ++t) acc = fmaf(sK[t * ldk + c], sV[t * Vt + j], acc);
            sS[c * Vt + j] = acc;
        }
    }
    __syncthreads();
    if (hT) {
        for (int e = tid; e < K * Vt; e += kSimtThreads) {
            const int c = e / Vt, j = e % Vt;
            if (j < vt) hT[(bh * K + c) * V + j0 + j] = sS[c * Vt + j];
        }
    }
}

cudaError_t launch_chunk_simt(const ChunkArgs& a, cudaStream_t s) {
    // Widest V tile (<= 64) whose working set fits in shared memory.
    int Vt = std::min(a.V, 64);
    size_t bytes = 0;
    for (;;) {
        bytes = SimtSmem(a.chunk, a.K, Vt).total_floats * sizeof(float);
        if (bytes <= 227u * 1024u || Vt <= 8) break;
        Vt /= 2;
    }
    if (a.chunk * Vt > kSimtThreads * kMaxPerThread) return cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)(a.B * a.H), (unsigned)((a.V + Vt - 1) / Vt));
    cudaError_t err;
    if (a.io == KDA_BF16) {
        auto kern = chunk_simt_kernel<__nv_bfloat16>;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (err != cudaSuccess) return err;
        kern<<<grid, kSimtThreads, bytes, s>>>(
            a.H, a.T, a.K, a.V, a.chunk, Vt, (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k,
            (const __nv_bfloat16*)a.v, (const __nv_bfloat16*)a.z, (const __nv_bfloat16*)a.beta,
            a.A_log, a.dt_bias, a.scale, a.h0, (__nv_bfloat16*)a.out, a.hT);
    } else {
        auto kern = chunk_simt_kernel<float>;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (err != cudaSuccess) return err;
        kern<<<grid, kSimtThreads, bytes, s>>>(
            a.H, a.T, a.K, a.V, a.chunk, Vt, (const float*)a.q, (const float*)a.k,
            (const float*)a.v, (const float*)a.z, (const float*)a.beta, a.A_log, a.dt_bias,
            a.scale, a.h0, (float*)a.out, a.hT);
    }
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
