// chunk_bwd.cu -- the backward of the KDA forward: from dL/do and dL/dhT, the gradients of
// q, k, v, z, beta, A_log, dt_bias and h0 (the kda-adjoint-2026-10-01 page names this
// backward and its gradients dq, dk, dv, dg, dbeta and the state gradient; each step below
// is the chain rule applied to the chunked form of the forward).
//
// Two forms walk the same equations in chunks of 16 tokens.  Phase 1 walks a sequence's chunks
// forward and keeps the state entering each chunk, and the chunk's R and Delta, in a scratch
// buffer; phase 2 walks them in reverse with dS, the adjoint of the state leaving the chunk.
// kda_chunk_bwd_kernel (any K, V): one CTA of 512 threads per (b, h), fp32 on the CUDA cores.
// kda_chunk_bwd_tc_kernel (K = V = 128): the state products on the tensor cores, one
// persistent CTA per SM taking the walks as work items (its own comment below).  Per chunk,
// with S the state entering it, G the in-chunk cumulative log decay, Gamma = e^G,
// gamma = e^{G_last}, Kg = K Gamma, Qg = Q Gamma, Kt = K e^{G_last - G},
// A'[t,i] = sum_c k_tc k_ic e^{G_tc - G_ic} (i < t), M[t,i] = sum_c q_tc k_ic e^{G_tc - G_ic}
// (i <= t), T = (I + diag(beta) A')^{-1}, R = V - Kg S, Delta = T diag(beta) R, the forward is
//     o = scale (Qg S + M Delta),   S_out = diag(gamma) S + Kt^T Delta,
// and the adjoints are, in order:
//     dDelta = Kt dS + scale M^T dO            dY = T^T dDelta
//     dKt = Delta dS^T                         dgamma = rowsum(S .* dS)
//     dQg = scale dO S^T                       P = dY S^T  (dKg = -diag(beta) P)
//     dM = scale dO Delta^T (i <= t)           dB = -dY Delta^T (i < t), dA' = diag(beta) dB
//     dbeta_t = sum_v R_tv dY_tv + sum_{i<t} A'_ti dB_ti          dV = diag(beta) dY
//     the pairwise terms of dA' and dM into dq, dk and dG (exact e^{G_t - G_i} per pair),
//     the Gamma factors into dq, dk and dG,
//     dS <- diag(gamma) dS + scale Qg^T dO - Kg^T diag(beta) dY,
// then dg = the reverse in-chunk cumulative sum of dG and the gate's own derivative:
//     dz = dg (-e^{A_log}) sigmoid(z + dt_bias), ddt_bias += dz, dA_log += dg g.
// In the CUDA-core form the state and its adjoint sit in shared memory (rows of odd pitch, so
// that both row and column walks are free of bank conflicts); in both forms every
// per-(token, channel) gradient term is produced by the same thread, so dq, dk and dG
// accumulate in registers.
#include <algorithm>
#include <functional>
#include <queue>
#include <type_traits>
#include <vector>

#include "chunk_tiles.cuh"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace kda {

// Set by the tensor-core backward when one of its bounded waits gives up.
__device__ int g_kda_bwd_timeout;

namespace {

constexpr int BC = 16;    // tokens per chunk
constexpr int BNT = 512;  // threads per CTA
constexpr int KM = 128, VM = 128;

// shared memory map (floats)
constexpr int SP = VM + 1;                // row pitch of S and dS
constexpr int O_S = 0;                    // S   [KM][SP], (c, v) at sw(c, v)
constexpr int O_DS = O_S + KM * SP;       // dS  [KM][SP]
constexpr int GP = BC + 1;                // row pitch of the channel-major q, k, G tiles
constexpr int O_Q = O_DS + KM * SP;       // q   [KM][GP]: (c, t) at ci(c, t)
constexpr int O_K = O_Q + KM * GP;        // k   [KM][GP]
constexpr int O_G = O_K + KM * GP;        // G   [KM][GP] (natural log units)
constexpr int O_KGT = O_G + KM * GP;      // Kg  [KM][BC]
constexpr int O_QGT = O_KGT + BC * KM;    // Qg  [KM][BC]
constexpr int O_KTT = O_QGT + BC * KM;    // Kt  [KM][BC]
constexpr int O_R = O_KTT + BC * KM;      // R = V - Kg S [BC][VM] (phase 1: v first)
constexpr int O_DO = O_R + BC * VM;       // dO  [BC][VM]
constexpr int O_DL = O_DO + BC * VM;      // Delta [BC][VM]
constexpr int O_DY = O_DL + BC * VM;      // dDelta, then dY [BC][VM]
constexpr int O_XT = O_DY + BC * VM;      // one C x V array transposed [VM][BC]; dG [BC][KM]
constexpr int O_AP = O_XT + BC * VM;      // A'  [BC][BC]
constexpr int O_TM = O_AP + BC * BC;      // T
constexpr int O_MM = O_TM + BC * BC;      // M
constexpr int O_DB = O_MM + BC * BC;      // dB
constexpr int O_DM = O_DB + BC * BC;      // dM
constexpr int O_BET = O_DM + BC * BC;     // beta [BC]
constexpr int O_GAM = O_BET + BC;         // gamma [KM]
constexpr int O_RED = O_GAM + KM;         // [4][KM] partial sums
constexpr int SMEM_FLOATS = O_RED + 4 * KM;
constexpr size_t BWD_SMEM_BYTES = sizeof(float) * SMEM_FLOATS;
static_assert(BWD_SMEM_BYTES <= 232448, "backward shared memory");

// S and dS rows have an odd pitch: a warp walking one row (32 v) or one column (32 c) hits
// 32 distinct banks, and every walk is a constant stride.
__device__ __forceinline__ int sw(int c, int v) { return c * SP + v; }
// q, k and G: channel-major with an odd pitch, so that a warp over 32 channels of one token
// and a warp over (2 channels x 16 tokens) both hit distinct banks
__device__ __forceinline__ int ci(int c, int t) { return c * GP + t; }
static_assert(O_KGT % 4 == 0, "16-byte aligned channel-major operands");

template <typename IO>
struct BwdArgs {
    int H, T, K, V;
    const IO *q, *k, *v, *z, *beta, *d_o;
    const float *A_log, *dt_bias, *h0, *dhT;
    float scale;
    float *dq, *dk, *dv, *dz, *dbeta, *dh0;
    float* ckpt;      // (B H, N, K, V): the state entering each chunk
    float* rd;        // (B H, N, 2, BC, V): R and Delta of each chunk, phase 1 -> phase 2
    float* dA_part;   // (B H)
    float* ddt_part;  // (B H, K)
};

// 4-byte asynchronous global -> shared copies (the state of the next chunk to process lands
// while the current one finishes)
__device__ __forceinline__ void cp_async4(float* dst_smem, const float* src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst_smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Reduce-scatter over a warp: on entry every lane holds 32 partial values; on exit v[0] of
// lane l is the sum over the 32 lanes of their value l (31 shuffles).
__device__ __forceinline__ void warp_reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
    for (int off = 16, w = 16; off >= 1; off >>= 1, w >>= 1) {
        const bool hi = (lane & off) != 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (j < w) {
                const float send = hi ? v[j] : v[j + w];
                const float keep = hi ? v[j + w] : v[j];
                v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
        }
    }
}

__device__ __forceinline__ float sigmoid_f32(float x) {
    return x >= 0.f ? 1.f / (1.f + expf(-x)) : expf(x) / (1.f + expf(x));
}

// KC = 128: the instance for K = V = 128, where every loop bound and size guard is a
// constant; KC = 0: any K, V in the supported range.
template <typename IO, int KC>
__global__ void __launch_bounds__(BNT, 1) kda_chunk_bwd_kernel(const BwdArgs<IO> a) {
    extern __shared__ float4 smem_f4[];
    float* sm = reinterpret_cast<float*>(smem_f4);
    float* S = sm + O_S;
    float* dS = sm + O_DS;
    float* Qr = sm + O_Q;
    float* Kr = sm + O_K;
    float* Gc = sm + O_G;
    float* KgT = sm + O_KGT;
    float* QgT = sm + O_QGT;
    float* KtT = sm + O_KTT;
    float* Rv = sm + O_R;
    float* dO = sm + O_DO;
    float* Dl = sm + O_DL;
    float* dY = sm + O_DY;
    float* XT = sm + O_XT;
    float* Ap = sm + O_AP;
    float* Tm = sm + O_TM;
    float* Mm = sm + O_MM;
    float* dB = sm + O_DB;
    float* dM = sm + O_DM;
    float* bet = sm + O_BET;
    float* gam = sm + O_GAM;
    float* red = sm + O_RED;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = KC ? KC : a.K, V = KC ? KC : a.V, T = a.T;
    const size_t bh = blockIdx.x;
    const int h = (int)(bh % a.H);
    const int N = (T + BC - 1) / BC;
    const float eA = expf(a.A_log[h]);
    const size_t KV = (size_t)K * V;
    // thread roles: (v or c) = tid % 128, quarter = tid / 128
    const int col = tid & 127, qtr = tid >> 7;

    // Copy a (K, V) float32 matrix from global memory into a padded shared one (zero when
    // src is null): every load is issued before the first store.
    auto load_kv = [&](float* dst, const float* src) {
        float x[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int c = qtr + 4 * j;
            x[j] = (src && c < K && col < V) ? __ldcg(src + (size_t)c * V + col) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int c = qtr + 4 * j;
            if (c < K && col < V) dst[sw(c, col)] = x[j];
        }
    };
    // ---- the state entering the sequence
    load_kv(S, a.h0 ? a.h0 + bh * KV : nullptr);
    __syncthreads();

    // Ask L2 for the inputs of chunk n (one 128-byte line per thread): k, z, and v (phase 1)
    // or q, dO, R and Delta (phase 2, `full`); issued one chunk ahead of load_chunk.
    auto prefetch_chunk = [&](int n, bool full) {
        if (n < 0 || n >= N) return;
        const int t0 = n * BC, cn = min(BC, T - t0);
        const int io = (int)sizeof(IO);
        const int lk = (cn * K * io + 127) / 128, lv = (cn * V * io + 127) / 128;
        const int lrd = (2 * BC * V * 4 + 127) / 128;
        int i = tid;
        const char* p = nullptr;
        if (i < lk) p = reinterpret_cast<const char*>(a.k + ((bh * T) + t0) * K) + 128 * i;
        else if ((i -= lk) < lk) p = reinterpret_cast<const char*>(a.z + ((bh * T) + t0) * K) + 128 * i;
        else if (full && (i -= lk) < lk) p = reinterpret_cast<const char*>(a.q + ((bh * T) + t0) * K) + 128 * i;
        else if (full && (i -= lk) < lv) p = reinterpret_cast<const char*>(a.d_o + ((bh * T) + t0) * V) + 128 * i;
        else if (full && (i -= lv) < lrd) p = reinterpret_cast<const char*>(a.rd + (bh * N + n) * (size_t)(2 * BC * V)) + 128 * i;
        else if (!full && (i -= lk) < lv) p = reinterpret_cast<const char*>(a.v + ((bh * T) + t0) * V) + 128 * i;
        if (p) prefetch_l2(p);
    };
    // Load chunk n: k, beta and G (from z), then recompute A' and T; phase 1 (`full` false)
    // also computes R and Delta from v and S, phase 2 loads q and dO, takes R and Delta as
    // phase 1 stored them, and computes M.  Every exit follows a barrier.
    auto load_chunk = [&](int n, bool full) {
        const int t0 = n * BC, cn = min(BC, T - t0);
        constexpr int PER = BC * KM / BNT;  // elements per thread of a (BC, K) or (BC, V) tile
        float kx[PER], qx[PER], zx[PER], dtx[PER], vx[PER], ox[PER], dx[PER];
        const float* rdn = a.rd + (bh * N + n) * (size_t)(2 * BC * V);
        float bx = 0.f;
        // every global load first (they overlap), then the shared-memory stores
#pragma unroll
        for (int r = 0; r < PER; ++r) {
            const int idx = tid + r * BNT, t = idx / K, c = idx - t * K;
            const bool in = idx < BC * K && t < cn;
            const size_t gi = ((bh * T) + t0 + t) * K + c;
            kx[r] = in ? ld_io(a.k + gi) : 0.f;
            qx[r] = (full && in) ? ld_io(a.q + gi) : 0.f;
            zx[r] = in ? ld_io(a.z + gi) : 0.f;
            dtx[r] = in ? __ldg(a.dt_bias + (size_t)h * K + c) : 0.f;
        }
#pragma unroll
        for (int r = 0; r < PER; ++r) {
            const int idx = tid + r * BNT, t = idx / V, vv = idx - t * V;
            const bool in = idx < BC * V && t < cn;
            const size_t gi = ((bh * T) + t0 + t) * V + vv;
            // phase 2 takes R and Delta as phase 1 left them; phase 1 starts from v
            if (full) {
                vx[r] = idx < BC * V ? __ldcg(rdn + idx) : 0.f;
                dx[r] = idx < BC * V ? __ldcg(rdn + BC * V + idx) : 0.f;
            } else {
                vx[r] = in ? ld_io(a.v + gi) : 0.f;
                dx[r] = 0.f;
            }
            ox[r] = (full && in) ? ld_io(a.d_o + gi) : 0.f;
        }
        if (tid < BC && tid < cn) bx = ld_io(a.beta + bh * T + t0 + tid);
#pragma unroll
        for (int r = 0; r < PER; ++r) {
            const int idx = tid + r * BNT, t = idx / K, c = idx - t * K;
            if (idx < BC * K) {
                const bool in = t < cn;
                Kr[ci(c, t)] = kx[r];
                if (full) Qr[ci(c, t)] = qx[r];
                Gc[ci(c, t)] = in ? kda_log_decay(zx[r], dtx[r], eA) : 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < PER; ++r) {
            const int idx = tid + r * BNT, t = idx / V, vv = idx - t * V;
            if (idx < BC * V) {
                Rv[t * VM + vv] = vx[r];
                if (full) {
                    dO[t * VM + vv] = ox[r];
                    Dl[t * VM + vv] = dx[r];
                }
            }
        }
        if (tid < BC) bet[tid] = bx;
        __syncthreads();
        if (tid < K) {  // in-chunk cumulative sum of the log decay
            float run = 0.f;
            for (int t = 0; t < BC; ++t) {
                run += Gc[ci(tid, t)];
                Gc[ci(tid, t)] = run;
            }
            gam[tid] = expf(run);
        }
        __syncthreads();
        // the decay-scaled operands, channel-major
        for (int idx = tid; idx < BC * K; idx += BNT) {
            const int c = idx >> 4, t = idx & 15;
            const float g = Gc[ci(c, t)], gl = Gc[ci(c, (BC - 1))];
            const float kk = Kr[ci(c, t)];
            KgT[c * BC + t] = kk * expf(g);
            KtT[c * BC + t] = kk * expf(gl - g);
            if (full) QgT[c * BC + t] = Qr[ci(c, t)] * expf(g);
        }
        // A' (i < t) and M (i <= t), exact pairwise decay: warp t, lanes over channels; the
        // 2 x 16 sums of the row are reduced together
        {
            const int t = warp;
            float gt[4], kt[4], qt[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = lane + 32 * u;
                const bool ok = c < K;
                gt[u] = ok ? Gc[ci(c, t)] : 0.f;
                kt[u] = ok ? Kr[ci(c, t)] : 0.f;
                qt[u] = (ok && full) ? Qr[ci(c, t)] : 0.f;
            }
            float w[32];
#pragma unroll
            for (int i = 0; i < BC; ++i) {
                float sa = 0.f, sq = 0.f;
                if (i <= t) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int c = lane + 32 * u;
                        if (c < K) {
                            const float kiE = Kr[ci(c, i)] * __expf(gt[u] - Gc[ci(c, i)]);
                            sa = fmaf(kt[u], kiE, sa);
                            sq = fmaf(qt[u], kiE, sq);
                        }
                    }
                }
                w[i] = sa;
                w[BC + i] = sq;
            }
            warp_reduce_scatter32(w, lane);
            if (lane < BC) Ap[t * BC + lane] = lane < t ? w[0] : 0.f;
            else if (full) Mm[t * BC + lane - BC] = lane - BC <= t ? w[0] : 0.f;
        }
        __syncthreads();
        // T = (I + diag(beta) A')^{-1} by forward substitution, one column per thread
        if (tid < BC) {
            const int j = tid;
            float x[BC];
#pragma unroll
            for (int t = 0; t < BC; ++t) {
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < t; ++i) acc = fmaf(Ap[t * BC + i], x[i], acc);
                x[t] = (t == j ? 1.f : 0.f) - bet[t] * acc;
                Tm[t * BC + j] = x[t];
            }
        }
        // R = V - Kg S: thread (v = col, tokens 4 qtr ..)  (phase 1 only)
        if (!full && col < V) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
            for (int c = 0; c < K; ++c) {
                const float s = S[sw(c, col)];
                const float4 kg = *reinterpret_cast<const float4*>(KgT + c * BC + 4 * qtr);
                acc[0] = fmaf(kg.x, s, acc[0]);
                acc[1] = fmaf(kg.y, s, acc[1]);
                acc[2] = fmaf(kg.z, s, acc[2]);
                acc[3] = fmaf(kg.w, s, acc[3]);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) Rv[(4 * qtr + r) * VM + col] -= acc[r];
        }
        __syncthreads();
        if (full) return;
        // Delta = T diag(beta) R
        if (col < V) {
            float rb[BC];
#pragma unroll
            for (int i = 0; i < BC; ++i) rb[i] = bet[i] * Rv[i * VM + col];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * qtr + r;
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < BC; ++i)
                    if (i <= t) acc = fmaf(Tm[t * BC + i], rb[i], acc);
                Dl[t * VM + col] = acc;
            }
        }
        __syncthreads();
    };

    // ======================================================= phase 1: chunk states forward
    for (int n = 0; n < N; ++n) {
        float* ck = a.ckpt + (bh * N + n) * KV;
        for (int j = 0; j < 32; ++j) {
            const int c = qtr + 4 * j;
            if (c < K && col < V) ck[(size_t)c * V + col] = S[sw(c, col)];
        }
        load_chunk(n, false);
        prefetch_chunk(n + 1, false);
        {  // R and Delta for phase 2
            float* rdn = a.rd + (bh * N + n) * (size_t)(2 * BC * V);
            for (int idx = tid; idx < BC * V; idx += BNT) {
                const int t = idx / V, vv = idx - t * V;
                rdn[idx] = Rv[t * VM + vv];
                rdn[BC * V + idx] = Dl[t * VM + vv];
            }
        }
        // S <- diag(gamma) S + Kt^T Delta: thread (v = col, channels qtr + 4 j)
        if (col < V) {
            float d[BC];
#pragma unroll
            for (int t = 0; t < BC; ++t) d[t] = Dl[t * VM + col];
#pragma unroll 4
            for (int j = 0; j < 32; ++j) {
                const int c = qtr + 4 * j;
                if (c >= K) continue;
                const float4* kt = reinterpret_cast<const float4*>(KtT + c * BC);
                float acc = S[sw(c, col)] * gam[c];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 x = kt[u];
                    acc = fmaf(x.x, d[4 * u], acc);
                    acc = fmaf(x.y, d[4 * u + 1], acc);
                    acc = fmaf(x.z, d[4 * u + 2], acc);
                    acc = fmaf(x.w, d[4 * u + 3], acc);
                }
                S[sw(c, col)] = acc;
            }
        }
        __syncthreads();
    }

    // ======================================================= phase 2: reverse
    load_kv(dS, a.dhT ? a.dhT + bh * KV : nullptr);
    // the state entering the last chunk, asynchronously (each later one is requested as soon
    // as the chunk after it has finished reading S)
    auto prefetch_state = [&](int n) {
        const float* ck = a.ckpt + (bh * N + n) * KV;
        for (int j = 0; j < 32; ++j) {
            const int c = qtr + 4 * j;
            if (c < K && col < V) cp_async4(S + sw(c, col), ck + (size_t)c * V + col);
        }
        cp_async_commit();
    };
    if (N > 0) prefetch_state(N - 1);
    float dA_acc = 0.f, ddt_acc = 0.f;  // this thread's channel col, tokens of quarter qtr
    // Transposed copy of a [BC][VM] array into dst ([VM][BC]).
    auto transpose_cv = [&](float* dst, const float* src) {
        for (int idx = tid; idx < BC * V; idx += BNT) {
            const int vv = idx >> 4, t = idx & 15;
            dst[vv * BC + t] = src[t * VM + vv];
        }
    };
    // out[r] = sum_v X[v][4 qtr + r] M[c][v] for this thread's channel c = col (M = S or dS,
    // X transposed [VM][BC]).
    auto contract_v = [&](const float* Mat, const float* X, float (&out)[4]) {
        out[0] = out[1] = out[2] = out[3] = 0.f;
#pragma unroll 8
        for (int vv = 0; vv < V; ++vv) {
            const float m = Mat[sw(col, vv)];
            const float4 x = *reinterpret_cast<const float4*>(X + vv * BC + 4 * qtr);
            out[0] = fmaf(x.x, m, out[0]);
            out[1] = fmaf(x.y, m, out[1]);
            out[2] = fmaf(x.z, m, out[2]);
            out[3] = fmaf(x.w, m, out[3]);
        }
    };
    // The same for two transposed operands against one pass over M.
    auto contract_v2 = [&](const float* Mat, const float* X1, const float* X2, float (&o1)[4],
                           float (&o2)[4]) {
#pragma unroll
        for (int r = 0; r < 4; ++r) o1[r] = o2[r] = 0.f;
#pragma unroll 8
        for (int vv = 0; vv < V; ++vv) {
            const float m = Mat[sw(col, vv)];
            const float4 x = *reinterpret_cast<const float4*>(X1 + vv * BC + 4 * qtr);
            const float4 y = *reinterpret_cast<const float4*>(X2 + vv * BC + 4 * qtr);
            o1[0] = fmaf(x.x, m, o1[0]);
            o1[1] = fmaf(x.y, m, o1[1]);
            o1[2] = fmaf(x.z, m, o1[2]);
            o1[3] = fmaf(x.w, m, o1[3]);
            o2[0] = fmaf(y.x, m, o2[0]);
            o2[1] = fmaf(y.y, m, o2[1]);
            o2[2] = fmaf(y.z, m, o2[2]);
            o2[3] = fmaf(y.w, m, o2[3]);
        }
    };

    for (int n = N - 1; n >= 0; --n) {
        const int t0 = n * BC, cn = min(BC, T - t0);
        cp_async_wait_all();  // this chunk's entering state (prefetch_state)
        load_chunk(n, true);  // its first barrier publishes S
        prefetch_chunk(n - 1, true);


        // dDelta = Kt dS + scale M^T dO  -> dY buffer; and this thread's share of dgamma
        if (col < V) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
            for (int c = 0; c < K; ++c) {
                const float s = dS[sw(c, col)];
                const float4 kt = *reinterpret_cast<const float4*>(KtT + c * BC + 4 * qtr);
                acc[0] = fmaf(kt.x, s, acc[0]);
                acc[1] = fmaf(kt.y, s, acc[1]);
                acc[2] = fmaf(kt.z, s, acc[2]);
                acc[3] = fmaf(kt.w, s, acc[3]);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * qtr + r;
                float m = 0.f;
                for (int s2 = t; s2 < BC; ++s2) m = fmaf(Mm[s2 * BC + t], dO[s2 * VM + col], m);
                dY[t * VM + col] = acc[r] + a.scale * m;
            }
        }
        if (col < K) {  // dgamma_c partial over the value quarter qtr, times gamma_c
            float sacc = 0.f;
            const int v0 = 32 * qtr;
#pragma unroll 8
            for (int vv = v0; vv < min(V, v0 + 32); ++vv) sacc = fmaf(S[sw(col, vv)], dS[sw(col, vv)], sacc);
            red[qtr * KM + col] = sacc * gam[col];
        }
        __syncthreads();
        // dY = T^T dDelta (in place: the column is read into registers first)
        {
            float dd[BC];
            if (col < V) {
#pragma unroll
                for (int t = 0; t < BC; ++t) dd[t] = dY[t * VM + col];
            }
            __syncthreads();
            if (col < V) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int i = 4 * qtr + r;
                    float acc = 0.f;
#pragma unroll
                    for (int t = 0; t < BC; ++t)
                        if (t >= i) acc = fmaf(Tm[t * BC + i], dd[t], acc);
                    dY[i * VM + col] = acc;
                }
            }
        }
        // the contractions over v, thread (c = col, tokens 4 qtr + r)
        float dq_r[4] = {0.f, 0.f, 0.f, 0.f}, dk_r[4] = {0.f, 0.f, 0.f, 0.f};
        float dG_r[4] = {0.f, 0.f, 0.f, 0.f};
        float dgl_part = 0.f;
        transpose_cv(XT, Dl);
        __syncthreads();
        if (col < K) {  // dKt = Delta dS^T
            float x[4];
            contract_v(dS, XT, x);
            const float gl = Gc[ci(col, (BC - 1))];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * qtr + r;
                const float eL = expf(gl - Gc[ci(col, t)]);
                const float kk = Kr[ci(col, t)];
                dk_r[r] += x[r] * eL;
                dG_r[r] -= x[r] * kk * eL;
                dgl_part += x[r] * kk * eL;
            }
        }
        {  // the first part of dbeta_t, sum_v R_tv dY_tv (warp t), into the M slot (M is done)
            const int t = warp;
            float sr = 0.f;
            for (int vv = lane; vv < V; vv += 32) sr = fmaf(Rv[t * VM + vv], dY[t * VM + vv], sr);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sr += __shfl_xor_sync(0xffffffffu, sr, off);
            if (lane == 0) Mm[t] = sr;
        }
        __syncthreads();
        // dO^T and dY^T (the latter in the R slot, R is done) for one pass over S
        transpose_cv(XT, dO);
        transpose_cv(Rv, dY);
        __syncthreads();
        if (col < K) {  // dQg = scale dO S^T and P = dY S^T, dKg = -diag(beta) P
            float x[4], y[4];
            contract_v2(S, XT, Rv, x, y);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * qtr + r;
                const float Ga = expf(Gc[ci(col, t)]);
                const float dqg = a.scale * x[r];
                const float dkg = -bet[t] * y[r];
                dq_r[r] += dqg * Ga;
                dk_r[r] += dkg * Ga;
                dG_r[r] += (dqg * Qr[ci(col, t)] + dkg * Kr[ci(col, t)]) * Ga;
            }
        }
        // dM (i <= t) and dB (i < t): warp t, lanes over value columns, reduced together
        {
            const int t = warp;
            float ot[4], yt[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int vv = lane + 32 * u;
                const bool ok = vv < V;
                ot[u] = ok ? dO[t * VM + vv] : 0.f;
                yt[u] = ok ? dY[t * VM + vv] : 0.f;
            }
            float w[32];
#pragma unroll
            for (int i = 0; i < BC; ++i) {
                float sm_ = 0.f, sb = 0.f;
                if (i <= t) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int vv = lane + 32 * u;
                        if (vv < V) {
                            const float dl = Dl[i * VM + vv];
                            sm_ = fmaf(ot[u], dl, sm_);
                            sb = fmaf(yt[u], dl, sb);
                        }
                    }
                }
                w[i] = sm_;
                w[BC + i] = sb;
            }
            warp_reduce_scatter32(w, lane);
            if (lane < BC) dM[t * BC + lane] = lane <= t ? a.scale * w[0] : 0.f;
            else dB[t * BC + lane - BC] = lane - BC < t ? -w[0] : 0.f;
        }
        __syncthreads();
        if (n > 0) prefetch_state(n - 1);  // S is not read again in this chunk
        // dbeta_t = sum_v R_tv dY_tv (above) + sum_{i<t} A'_ti dB_ti;  dV = diag(beta) dY
        if (tid < cn) {
            const int t = tid;
            float s = Mm[t];
            for (int i = 0; i < t; ++i) s = fmaf(Ap[t * BC + i], dB[t * BC + i], s);
            a.dbeta[bh * T + t0 + t] = s;
        }
        for (int idx = tid; idx < cn * V; idx += BNT) {
            const int t = idx / V, vv = idx - t * V;
            a.dv[((bh * T) + t0 + t) * V + vv] = bet[t] * dY[t * VM + vv];
        }
        // pairwise terms of dA' = diag(beta) dB and dM, thread (c = col, tokens 4 qtr + r)
        if (col < K) {
            const int c = col;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * qtr + r;
                const float gt = Gc[ci(c, t)], kt = Kr[ci(c, t)], qt = Qr[ci(c, t)];
                float rowA = 0.f, rowM = 0.f, colA = 0.f, colM = 0.f;
#pragma unroll
                for (int i = 0; i < BC; ++i) {  // t as the row (later) token
                    if (i <= t) {
                        const float kiE = Kr[ci(c, i)] * __expf(gt - Gc[ci(c, i)]);
                        rowM = fmaf(dM[t * BC + i], kiE, rowM);
                        rowA = fmaf(bet[t] * dB[t * BC + i], kiE, rowA);  // dB[t][t] = 0
                    }
                }
#pragma unroll
                for (int s2 = 0; s2 < BC; ++s2) {  // t as the column (earlier) token
                    if (s2 >= t) {
                        const float E = __expf(Gc[ci(c, s2)] - gt);
                        colM = fmaf(dM[s2 * BC + t], Qr[ci(c, s2)] * E, colM);
                        colA = fmaf(bet[s2] * dB[s2 * BC + t], Kr[ci(c, s2)] * E, colA);  // dB[t][t] = 0
                    }
                }
                dq_r[r] += rowM;
                dk_r[r] += rowA + colA + colM;
                dG_r[r] += kt * rowA + qt * rowM - kt * (colA + colM);
            }
        }
        // dS <- diag(gamma) dS + scale Qg^T dO - Kg^T diag(beta) dY  (thread (v = col, c = qtr + 4 j))
        if (col < V) {
            float dov[BC], dyv[BC];
#pragma unroll
            for (int t = 0; t < BC; ++t) {
                dov[t] = a.scale * dO[t * VM + col];
                dyv[t] = bet[t] * dY[t * VM + col];
            }
#pragma unroll 2
            for (int j = 0; j < 32; ++j) {
                const int c = qtr + 4 * j;
                if (c >= K) continue;
                const float4* qg = reinterpret_cast<const float4*>(QgT + c * BC);
                const float4* kg = reinterpret_cast<const float4*>(KgT + c * BC);
                float acc = dS[sw(c, col)] * gam[c];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 x = qg[u], y = kg[u];
                    acc = fmaf(x.x, dov[4 * u], acc);
                    acc = fmaf(x.y, dov[4 * u + 1], acc);
                    acc = fmaf(x.z, dov[4 * u + 2], acc);
                    acc = fmaf(x.w, dov[4 * u + 3], acc);
                    acc = fmaf(-y.x, dyv[4 * u], acc);
                    acc = fmaf(-y.y, dyv[4 * u + 1], acc);
                    acc = fmaf(-y.z, dyv[4 * u + 2], acc);
                    acc = fmaf(-y.w, dyv[4 * u + 3], acc);
                }
                dS[sw(c, col)] = acc;
            }
        }
        __syncthreads();  // every read of XT and of red is done
        // dG exchange ([BC][KM] in XT), the last token's share of d(G_last), reverse cumsum,
        // gate derivative; dq and dk out
        if (col < K) {
#pragma unroll
            for (int r = 0; r < 4; ++r) XT[(4 * qtr + r) * KM + col] = dG_r[r];
            red[qtr * KM + col] += dgl_part;
        }
        __syncthreads();
        if (col < K) {
            const int c = col;
            const float dgl = red[c] + red[KM + c] + red[2 * KM + c] + red[3 * KM + c];
            float suffix = dgl;  // d(G_last) enters G_{BC-1}
            for (int t = BC - 1; t > 4 * qtr + 3; --t) suffix += XT[t * KM + c];
            const float dtc = a.dt_bias[(size_t)h * K + c];
            float zr[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * qtr + r;
                zr[r] = t < cn ? ld_io(a.z + ((bh * T) + t0 + t) * K + c) : 0.f;
            }
#pragma unroll
            for (int r = 3; r >= 0; --r) {
                const int t = 4 * qtr + r;
                suffix += XT[t * KM + c];
                if (t < cn) {
                    const size_t gi = ((bh * T) + t0 + t) * K + c;
                    const float x = zr[r] + dtc;
                    const float g = -(eA * softplus_f32(x));
                    const float dz = suffix * (-eA) * sigmoid_f32(x);
                    a.dz[gi] = dz;
                    ddt_acc += dz;
                    dA_acc = fmaf(suffix, g, dA_acc);
                    a.dq[gi] = dq_r[r];
                    a.dk[gi] = dk_r[r];
                }
            }
        }
        __syncthreads();
    }

    // ---- dh0, and the per-(b, h) partial sums of dA_log and ddt_bias
    if (a.dh0) {
        for (int j = 0; j < 32; ++j) {
            const int c = qtr + 4 * j;
            if (c < K && col < V) a.dh0[bh * KV + (size_t)c * V + col] = dS[sw(c, col)];
        }
    }
    if (col < K) red[qtr * KM + col] = ddt_acc;
    for (int off = 16; off > 0; off >>= 1) dA_acc += __shfl_xor_sync(0xffffffffu, dA_acc, off);
    __syncthreads();
    if (lane == 0) XT[warp] = dA_acc;
    if (tid < K) a.ddt_part[bh * K + tid] = red[tid] + red[KM + tid] + red[2 * KM + tid] + red[3 * KM + tid];
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int w = 0; w < BNT / 32; ++w) s += XT[w];
        a.dA_part[bh] = s;
    }
}

// ============================================================== tensor-core form, K = V = 128
// The same chunk walk and adjoint equations, with the state (phase 1) and its adjoint (phase 2)
// resident in TMEM as fp32 and every contraction with them on tcgen05 (M = 128 over c or v):
//   phase 1   R^T = V^T - S^T Kg^T                                  N = 16 tokens, K = c
//             S <- diag(gamma) S + Kt^T Delta                       N = v, K = 16 tokens
//   phase 2   dDelta^T = dS^T Kt^T + dO^T (scale M)                 N = 16, K = c, then 16
//             dKt^T = dS Delta^T                                    N = 16, K = v
//             [dQg^T | P^T] = S [dO ; dY]^T                         N = 32 (dQg = scale x)
//             [dM | dB] from [dO ; dY] Delta^T                      N = 16, K = v
//             dS <- diag(gamma) dS + [scale Qg ; -beta Kg]^T [dO ; dY]   K = 32 tokens
// Every operand x is split into bf16 x_hi = bf16(x) and x_lo = bf16(x - x_hi), within 2^-16 |x|
// of x together, and a product A B is accumulated in fp32 as the four products of the halves.
// The small operand's halves are stacked along N ([B_hi ; B_lo], doubling the N above), so
// each K step of the state is read by two MMAs (A_hi, A_lo) and the epilogue adds the two
// column blocks; each product term is within about 2 * 2^-16 of its exact value, and the state
// and its adjoint stay fp32 in TMEM.  The operand copy of the state (hi and lo, 64 KB) is also
// what phase 1 keeps per chunk, with the chunk's R, Delta, A', T, M and g: phase 2 brings them
// back by bulk copy, the state already in the operand layout.  The pairwise terms, the T
// solve, the gate and the per-token outputs run on the CUDA cores as in the kernel above.
// One persistent CTA per SM takes the walks as work items (BwdSched below).
namespace bwdtc {
constexpr int NT = 512;
// shared memory (bytes from a 1024-byte aligned base): tensor-core operand tiles, each a
// K-major 128-byte-swizzled tile (read MN-major where a product needs its transpose); the
// small tiles hold the hi rows first, then the lo rows
constexpr uint32_t OFF_ST = 0;                 // state / adjoint copy [c][v], 128 rows: hi
constexpr uint32_t ST_LO = 32768;              //   lo
constexpr uint32_t OFF_KT = 65536;             // Kt [t][c]: 32 rows (hi 0..15, lo 16..31)
constexpr uint32_t OFF_DLT = OFF_KT + 8192;    // Delta [t][v]: 32 rows
constexpr uint32_t OFF_DOY = OFF_DLT + 8192;   // [dO ; dY] [t'][v]: 64 rows (hi 0..31, lo 32..63)
constexpr uint32_t OFF_AQK = OFF_DOY + 16384;  // phase 2 [scale Qg ; -beta Kg] [t'][c]: 64 rows
                                               // (until the first products: scale M^T [t][s], 32
                                               // rows); phase 1 Kg [t][c]: 32 rows
constexpr uint32_t OFF_F = OFF_AQK + 16384;    // fp32 area (float offsets below)
// R, Delta, A', T, M are contiguous: phase 2 brings them back with one bulk copy
constexpr int F_Q = 0, F_K = F_Q + KM * GP, F_G = F_K + KM * GP;
constexpr int F_R = F_G + KM * GP, F_DL = F_R + BC * VM;
constexpr int F_AP = F_DL + BC * VM, F_TM = F_AP + BC * BC, F_MM = F_TM + BC * BC;
constexpr int F_DO = F_MM + BC * BC, F_DY = F_DO + BC * VM, F_XT = F_DY + BC * VM;
constexpr int F_DB = F_XT + BC * KM, F_DM = F_DB + BC * BC;
constexpr int F_BET = F_DM + BC * BC, F_GAM = F_BET + BC, F_RED = F_GAM + KM;
constexpr int F_GT = F_RED + 4 * KM;            // g (the per-token log decay) [KM][GP]
constexpr int F_END = F_GT + KM * GP;
constexpr uint32_t OFF_MISC = OFF_F + 4u * F_END;  // four mbarriers, TMEM base, failure flag
// staging of the next chunk's rows, bulk-copied: three I/O tiles (q, k, then z in phase 1 or
// dO in phase 2) and an 8 KB slot (v in phase 1, the fp32 g phase 1 kept in phase 2)
constexpr uint32_t OFF_STG = OFF_MISC + 64;
template <typename IO>
constexpr uint32_t stg_tile() { return (uint32_t)(BC * KM * sizeof(IO)); }
template <typename IO>
constexpr uint32_t off_gslot() { return OFF_STG + 3 * stg_tile<IO>(); }
template <typename IO>
constexpr size_t smem_bytes() { return off_gslot<IO>() + BC * KM * 4 + 1024; }  // + alignment slack
static_assert((OFF_F + 4u * F_R) % 16 == 0 && (OFF_F + 4u * F_DL) % 16 == 0 &&
              (OFF_F + 4u * F_DO) % 16 == 0 && (OFF_F + 4u * F_DY) % 16 == 0, "float4 rows");
static_assert(OFF_MISC % 16 == 0 && OFF_STG % 16 == 0, "mbarriers and bulk-copy destinations");
static_assert(smem_bytes<float>() <= 232448, "backward tensor-core shared memory");
// TMEM columns: the state or its adjoint, and the accumulators of the N = 32 / 64 products
// (one column block per half of the small operand)
constexpr uint32_t TM_M = 0, TM_A = 128, TM_B = 160, TM_C = 192, TM_COLS = 256;
constexpr uint32_t ID_MN_K32 = tc::idesc_bf16(128, 32, 1, 0);
constexpr uint32_t ID_K_K32 = tc::idesc_bf16(128, 32, 0, 0);
constexpr uint32_t ID_K_K64 = tc::idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_MN_MN128 = tc::idesc_bf16(128, 128, 1, 1);
constexpr uint32_t kStateBytes = 65536;        // one operand copy of the state (hi + lo)
// floats phase 1 keeps per chunk for phase 2: R, Delta [BC][V], A', T, M [BC][BC] (contiguous in
// shared memory, RD_SM floats), then g [BC][K]
constexpr int RD_SM = 2 * BC * VM + 3 * BC * BC;
constexpr int RD = RD_SM + BC * KM;
static_assert(F_DL == F_R + BC * VM && F_AP == F_DL + BC * VM && F_TM == F_AP + BC * BC &&
              F_MM == F_TM + BC * BC && F_MM + BC * BC == F_R + RD_SM, "R, Delta, A', T, M contiguous");
}  // namespace bwdtc

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi), eight values at a time
__device__ __forceinline__ void split8(const float (&f)[8], uint4& hi, uint4& lo) {
    hi = tile::pack8(f);
    float h[8], r[8];
    tile::unpack8(hi, h);
#pragma unroll
    for (int j = 0; j < 8; ++j) r[j] = f[j] - h[j];
    lo = tile::pack8(r);
}

// Work items of the tensor-core backward, taken from *counter in order by one CTA per SM at
// most: first the forward walk's segments (every sequence's segment 0, then segment 1, ...),
// then the reverse walk's (every sequence's last segment first).  A segment is seg_len chunks
// of one sequence.  The state passes between a sequence's forward segments through s_hand and
// its adjoint between reverse segments through ds_hand; flags[2 bh] counts the sequence's
// finished forward segments, flags[2 bh + 1] its finished reverse ones.  An item waits only for
// items earlier in the order, which CTAs that are already running have taken, so the schedule
// cannot deadlock; every wait is bounded.
struct BwdSched {
    int nseg, seg_len, n_items;
    int* counter;
    unsigned* flags;
    float* s_hand;
    float* ds_hand;
};

template <typename IO>
__global__ void __launch_bounds__(bwdtc::NT, 1) kda_chunk_bwd_tc_kernel(const BwdArgs<IO> a,
                                                                          const BwdSched sc) {
    using namespace bwdtc;
    extern __shared__ uint8_t smem_bwd_raw[];
    uint8_t* sm8 = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_bwd_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float* F = reinterpret_cast<float*>(sm8 + OFF_F);
    float* Qr = F + F_Q;
    float* Kr = F + F_K;
    float* Gc = F + F_G;
    float* Rv = F + F_R;
    float* dO = F + F_DO;
    float* Dl = F + F_DL;
    float* dY = F + F_DY;
    float* XT = F + F_XT;
    float* Ap = F + F_AP;
    float* Tm = F + F_TM;
    float* Mm = F + F_MM;
    float* dB = F + F_DB;
    float* dM = F + F_DM;
    float* bet = F + F_BET;
    float* gam = F + F_GAM;
    float* red = F + F_RED;
    float* Gt = F + F_GT;
    uint64_t* bar_mma = reinterpret_cast<uint64_t*>(sm8 + OFF_MISC);
    uint64_t* bar_ld = bar_mma + 1;   // the state copy (phase 2)
    uint64_t* bar_in = bar_mma + 2;   // a chunk's staged raw rows
    uint64_t* bar_rd = bar_mma + 3;   // a chunk's R, Delta, A', T, M (phase 2)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm8 + OFF_MISC + 32);
    volatile int* s_fail = reinterpret_cast<volatile int*>(sm8 + OFF_MISC + 36);
    volatile int* s_item = reinterpret_cast<volatile int*>(sm8 + OFF_MISC + 40);
    const uint32_t sb = tc::smem_u32(sm8);

    constexpr int K = KM, V = VM;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T;
    const int N = (T + BC - 1) / BC;
    const size_t KV = (size_t)K * V;
    // the current work item: sequence bh (head h), chunks [n_lo, n_hi)
    size_t bh = 0;
    int h = 0, n_lo = 0, n_hi = 0;
    float eA = 1.f, ieA = 1.f, dtc = 0.f;
    // thread roles: channel or value column col (= the TMEM lane this warp reaches), and the
    // quarter qtr (tokens 4 qtr .. + 3, or TMEM columns 32 qtr .. + 31 of a 128-column matrix)
    const int col = tid & 127, qtr = tid >> 7;

    if (tid == 0) {
        tc::mbar_init(bar_mma, 1);
        tc::mbar_init(bar_ld, 1);
        tc::mbar_init(bar_in, 1);
        tc::mbar_init(bar_rd, 1);
        *s_fail = 0;
        tc::fence_barrier_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, TM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = *tmem_slot;
    uint32_t ph_mma = 0, ph_ld = 0, ph_in = 0, ph_rd = 0;
    auto fail = [&]() {
        *s_fail = 1;
        atomicExch(&g_kda_bwd_timeout, 1);
    };
    auto wait_mma = [&]() {
        if (!tc::mbar_wait(bar_mma, ph_mma)) fail();
        ph_mma ^= 1u;
        tc::fence_after_sync();
    };
    auto wait_ld = [&]() {
        if (!tc::mbar_wait(bar_ld, ph_ld)) fail();
        ph_ld ^= 1u;
    };
    const uint32_t t_m0 = tile::taddr(tm + TM_M, warp, 32 * qtr);
    auto master_ld = [&](uint32_t (&r0)[16], uint32_t (&r1)[16]) {
        tc::tmem_ld16(t_m0, r0);
        tc::tmem_ld16(t_m0 + 16, r1);
        tc::tmem_ld_wait();
    };
    auto master_st = [&](const uint32_t (&r0)[16], const uint32_t (&r1)[16]) {
        tc::tmem_st16(t_m0, r0);
        tc::tmem_st16(t_m0 + 16, r1);
        tc::tmem_st_wait();
    };
    // TMEM matrix <- src (K, V) row-major, or zero: row col, columns 32 qtr .. + 31
    auto master_init = [&](const float* src) {
        uint32_t r0[16], r1[16];
        const float* p = src ? src + (size_t)col * V + 32 * qtr : nullptr;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            r0[j] = __float_as_uint(p ? __ldcg(p + j) : 0.f);
            r1[j] = __float_as_uint(p ? __ldcg(p + 16 + j) : 0.f);
        }
        master_st(r0, r1);
    };
    // The operand copy (hi, lo) of the TMEM matrix.
    auto master_copy = [&]() {
        uint32_t r0[16], r1[16];
        master_ld(r0, r1);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = __uint_as_float(g < 2 ? r0[8 * g + j] : r1[8 * (g - 2) + j]);
            uint4 hi, lo;
            split8(f, hi, lo);
            const uint32_t off = tile::kmaj_off(col, 32 * qtr + 8 * g, 128);
            *reinterpret_cast<uint4*>(sm8 + OFF_ST + off) = hi;
            *reinterpret_cast<uint4*>(sm8 + OFF_ST + ST_LO + off) = lo;
        }
        tc::fence_proxy_async_smem();
    };
    // The TMEM matrix scaled by gamma in place, row col.
    auto master_decay = [&]() {
        uint32_t r0[16], r1[16];
        master_ld(r0, r1);
        const float gm = gam[col];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            r0[j] = __float_as_uint(__uint_as_float(r0[j]) * gm);
            r1[j] = __float_as_uint(__uint_as_float(r1[j]) * gm);
        }
        master_st(r0, r1);
    };

    // Ask L2 for the state copy phase 1 kept for chunk n, one 128-byte line per thread.
    auto prefetch_state = [&](int n) {
        if (n >= n_lo && n < n_hi) prefetch_l2(reinterpret_cast<const char*>(a.ckpt + (bh * N + n) * KV) + 128 * tid);
    };
    // Request chunk n's raw rows into the staging tiles (bulk copies on bar_in, issued by thread
    // 0): q, k, and z, v (phase 1) or dO (phase 2); and its beta into bnext (threads < BC).
    float bnext = 0.f;
    auto request = [&](int n, bool full) {
        const int t0 = n * BC, cn = min(BC, T - t0);
        if (tid == 0) {
            const uint32_t bytes = (uint32_t)(cn * K * sizeof(IO));
            const size_t g0 = (bh * T + t0) * (size_t)K;
            tc::mbar_arrive_expect_tx(bar_in, (full ? 3 : 4) * bytes);
            tc::bulk_load(sm8 + OFF_STG, a.q + g0, bytes, bar_in);
            tc::bulk_load(sm8 + OFF_STG + stg_tile<IO>(), a.k + g0, bytes, bar_in);
            tc::bulk_load(sm8 + OFF_STG + 2 * stg_tile<IO>(), (full ? a.d_o : a.z) + g0, bytes, bar_in);
            if (!full) tc::bulk_load(sm8 + off_gslot<IO>(), a.v + g0, bytes, bar_in);
        }
        if (tid < BC) bnext = tid < cn ? ld_io(a.beta + bh * T + t0 + tid) : 0.f;
    };
    // Request chunk n's record from phase 2: R, Delta, A', T, M into place and g into the
    // staging slot (two bulk copies on bar_rd).
    auto request_rd = [&](int n) {
        if (tid == 0) {
            const float* src = a.rd + (bh * N + n) * (size_t)RD;
            tc::mbar_arrive_expect_tx(bar_rd, RD * 4);
            tc::bulk_load(Rv, src, RD_SM * 4, bar_rd);
            tc::bulk_load(sm8 + off_gslot<IO>(), src + RD_SM, BC * KM * 4, bar_rd);
        }
    };
    // Chunk n's staged rows into the fp32 tiles: q, k, beta, g (phase 1: from z, and kept in XT
    // for the chunk's record; phase 2: as phase 1 kept it), v (phase 1, into R) or dO (phase 2,
    // whose R, Delta, A', T, M arrive by request_rd); the staging is then free and the next
    // chunk's rows are requested; then G, the in-chunk cumulative sum of g, and gamma.
    auto load_inputs = [&](int n, bool full) {
        const int t0 = n * BC, cn = min(BC, T - t0);
        if (!tc::mbar_wait(bar_in, ph_in)) fail();
        ph_in ^= 1u;
        if (full) {
            if (!tc::mbar_wait(bar_rd, ph_rd)) fail();
            ph_rd ^= 1u;
        }
        const IO* sq = reinterpret_cast<const IO*>(sm8 + OFF_STG);
        const IO* sk = sq + BC * K;
        const IO* s2 = sk + BC * K;  // z (phase 1) or dO (phase 2)
        const IO* sv = reinterpret_cast<const IO*>(sm8 + off_gslot<IO>());
        const float* sg = reinterpret_cast<const float*>(sm8 + off_gslot<IO>());
        float run[4];  // this thread's tokens 4 qtr + r: prefix sums of g within the four
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int t = 4 * qtr + r, idx = t * K + col;
            const bool in = t < cn;
            const float g = full ? sg[idx] : (in ? kda_log_decay(ld_io(s2 + idx), dtc, eA) : 0.f);
            Kr[ci(col, t)] = in ? ld_io(sk + idx) : 0.f;
            Qr[ci(col, t)] = in ? ld_io(sq + idx) : 0.f;
            Gt[ci(col, t)] = g;
            run[r] = r ? run[r - 1] + g : g;
            if (full) {
                dO[idx] = in ? ld_io(s2 + idx) : 0.f;
            } else {
                Rv[idx] = in ? ld_io(sv + idx) : 0.f;
                XT[idx] = g;
            }
        }
        red[qtr * KM + col] = run[3];
        if (tid < BC) bet[tid] = bnext;
        tc::fence_proxy_async_smem();
        __syncthreads();
        const int nx = full ? n - 1 : n + 1;
        if (nx >= n_lo && nx < n_hi) request(nx, full);
        {  // G = the in-chunk cumulative sum: the earlier quarters' totals, then the prefix
            float off = 0.f;
#pragma unroll
            for (int q2 = 0; q2 < 3; ++q2)
                if (q2 < qtr) off += red[q2 * KM + col];
#pragma unroll
            for (int r = 0; r < 4; ++r) Gc[ci(col, 4 * qtr + r)] = off + run[r];
            if (qtr == 3) gam[col] = expf(off + run[3]);
        }
        __syncthreads();
    };
    // The decay-scaled operand tiles of the chunk (hi, lo): Kt = K e^{G_last - G} always;
    // phase 1 Kg = K e^G; phase 2 (with aqk) [scale Qg ; -beta Kg], else Delta, the dO half of
    // [dO ; dY] and scale M^T (B[t][s] = scale M[s][t], where [scale Qg ; -beta Kg] goes later).
    auto build_tiles = [&](bool full, bool aqk) {
        if (tid < 256) {
            const int t = tid & 15, c0 = 8 * (tid >> 4);
            float kt[8], kg[8], qg[8];
            // Kt unless this is the [scale Qg ; -beta Kg] pass; K e^G (and Q e^G) unless this is
            // phase 2's first pass, which writes Kt and scale M^T only
            const bool need_kt = !aqk, need_kg = !full || aqk;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int c = c0 + j;
                const float g = Gc[ci(c, t)], kk = Kr[ci(c, t)];
                kt[j] = need_kt ? kk * __expf(Gc[ci(c, BC - 1)] - g) : 0.f;
                const float eg = need_kg ? __expf(g) : 0.f;
                kg[j] = kk * eg;
                qg[j] = (full && aqk) ? Qr[ci(c, t)] * eg : 0.f;
            }
            uint4 hi, lo;
            if (!aqk) {
                split8(kt, hi, lo);
                *reinterpret_cast<uint4*>(sm8 + OFF_KT + tile::kmaj_off(t, c0, 32)) = hi;
                *reinterpret_cast<uint4*>(sm8 + OFF_KT + tile::kmaj_off(16 + t, c0, 32)) = lo;
            }
            if (full && !aqk) {
                if (tid < 32) {  // scale M^T: row t = tid & 15, columns s = 8 (tid >> 4) ..
                    const int s0 = 8 * (tid >> 4);
                    float m[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) m[j] = a.scale * Mm[(s0 + j) * BC + t];
                    split8(m, hi, lo);
                    *reinterpret_cast<uint4*>(sm8 + OFF_AQK + tile::kmaj_off(t, s0, 32)) = hi;
                    *reinterpret_cast<uint4*>(sm8 + OFF_AQK + tile::kmaj_off(16 + t, s0, 32)) = lo;
                }
            } else if (!full) {
                split8(kg, hi, lo);
                *reinterpret_cast<uint4*>(sm8 + OFF_AQK + tile::kmaj_off(t, c0, 32)) = hi;
                *reinterpret_cast<uint4*>(sm8 + OFF_AQK + tile::kmaj_off(16 + t, c0, 32)) = lo;
            } else {
                const float nb = -bet[t];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    qg[j] *= a.scale;
                    kg[j] *= nb;
                }
                split8(qg, hi, lo);
                *reinterpret_cast<uint4*>(sm8 + OFF_AQK + tile::kmaj_off(t, c0, 64)) = hi;
                *reinterpret_cast<uint4*>(sm8 + OFF_AQK + tile::kmaj_off(32 + t, c0, 64)) = lo;
                split8(kg, hi, lo);
                *reinterpret_cast<uint4*>(sm8 + OFF_AQK + tile::kmaj_off(16 + t, c0, 64)) = hi;
                *reinterpret_cast<uint4*>(sm8 + OFF_AQK + tile::kmaj_off(48 + t, c0, 64)) = lo;
            }
        } else if (full && !aqk) {
            const int i = tid - 256, t = i & 15, v0 = 8 * (i >> 4);
            float d[8], o[8];
            const float4 d0 = *reinterpret_cast<const float4*>(Dl + t * VM + v0);
            const float4 d1 = *reinterpret_cast<const float4*>(Dl + t * VM + v0 + 4);
            const float4 o0 = *reinterpret_cast<const float4*>(dO + t * VM + v0);
            const float4 o1 = *reinterpret_cast<const float4*>(dO + t * VM + v0 + 4);
            d[0] = d0.x; d[1] = d0.y; d[2] = d0.z; d[3] = d0.w; d[4] = d1.x; d[5] = d1.y; d[6] = d1.z; d[7] = d1.w;
            o[0] = o0.x; o[1] = o0.y; o[2] = o0.z; o[3] = o0.w; o[4] = o1.x; o[5] = o1.y; o[6] = o1.z; o[7] = o1.w;
            uint4 hi, lo;
            split8(d, hi, lo);
            *reinterpret_cast<uint4*>(sm8 + OFF_DLT + tile::kmaj_off(t, v0, 32)) = hi;
            *reinterpret_cast<uint4*>(sm8 + OFF_DLT + tile::kmaj_off(16 + t, v0, 32)) = lo;
            split8(o, hi, lo);
            *reinterpret_cast<uint4*>(sm8 + OFF_DOY + tile::kmaj_off(t, v0, 64)) = hi;
            *reinterpret_cast<uint4*>(sm8 + OFF_DOY + tile::kmaj_off(32 + t, v0, 64)) = lo;
        }
        tc::fence_proxy_async_smem();
    };
    // Rows of a [BC][VM] fp32 tile into rows row0 .. (hi) and row0 + lo_row .. (lo) of a 32- or
    // 64-row operand tile, one (row, 8 columns) item per thread of the first 256.
    auto tile_rows = [&](const float* src, uint32_t off, int rows, int lo_row, int row0) {
        if (tid < 256) {
            const int t = tid & 15, v0 = 8 * (tid >> 4);
            const float4 x0 = *reinterpret_cast<const float4*>(src + t * VM + v0);
            const float4 x1 = *reinterpret_cast<const float4*>(src + t * VM + v0 + 4);
            float f[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            uint4 hi, lo;
            split8(f, hi, lo);
            *reinterpret_cast<uint4*>(sm8 + off + tile::kmaj_off(row0 + t, v0, rows)) = hi;
            *reinterpret_cast<uint4*>(sm8 + off + tile::kmaj_off(row0 + lo_row + t, v0, rows)) = lo;
        }
        tc::fence_proxy_async_smem();
    };
    // A' (i < t) and M (i <= t) with the exact pairwise decay: warp t
    auto arows = [&]() {
        const int t = warp;
        float gt[4], kt[4], qt[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = lane + 32 * u;
            gt[u] = Gc[ci(c, t)];
            kt[u] = Kr[ci(c, t)];
            qt[u] = Qr[ci(c, t)];
        }
        float w[32];
#pragma unroll
        for (int i = 0; i < BC; ++i) {
            float sa = 0.f, sq = 0.f;
            if (i <= t) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = lane + 32 * u;
                    const float kiE = i == t ? kt[u] : Kr[ci(c, i)] * __expf(gt[u] - Gc[ci(c, i)]);
                    sa = fmaf(kt[u], kiE, sa);
                    sq = fmaf(qt[u], kiE, sq);
                }
            }
            w[i] = sa;
            w[BC + i] = sq;
        }
        warp_reduce_scatter32(w, lane);
        if (lane < BC) Ap[t * BC + lane] = lane < t ? w[0] : 0.f;
        else Mm[t * BC + lane - BC] = lane - BC <= t ? w[0] : 0.f;
    };
    // T = (I + diag(beta) A')^{-1} by forward substitution, one column per thread of warp 4
    auto t_solve = [&]() {
        if (tid >= 128 && tid < 128 + BC) {
            const int j = tid - 128;
            float x[BC];
#pragma unroll
            for (int t = 0; t < BC; ++t) {
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < t; ++i) acc = fmaf(Ap[t * BC + i], x[i], acc);
                x[t] = (t == j ? 1.f : 0.f) - bet[t] * acc;
                Tm[t * BC + j] = x[t];
            }
        }
    };

    // ======================================================= work items
    const int BHs = sc.n_items / (2 * sc.nseg);
    float dA_acc = 0.f, ddt_acc = 0.f;  // reverse walk: this thread's channel col, tokens of qtr
    for (;;) {
        if (tid == 0) *s_item = atomicAdd(sc.counter, 1);
        __syncthreads();
        const int item = *s_item;
        if (item >= sc.n_items || *s_fail) break;
        const bool fwd = item < BHs * sc.nseg;
        const int idx = fwd ? item : item - BHs * sc.nseg;
        const int seg = fwd ? idx / BHs : sc.nseg - 1 - idx / BHs;
        bh = (size_t)(idx % BHs);
        h = (int)(bh % a.H);
        eA = expf(a.A_log[h]);
        ieA = expf(-a.A_log[h]);
        dtc = __ldg(a.dt_bias + (size_t)h * KM + col);
        n_lo = min(N, seg * sc.seg_len);
        n_hi = min(N, n_lo + sc.seg_len);
        if (tid == 0) {  // the item this one continues
            bool ok = true;
            if (fwd && seg > 0) ok = tc::flag_wait_geq(sc.flags + 2 * bh, (unsigned)seg);
            else if (!fwd && seg == sc.nseg - 1) ok = tc::flag_wait_geq(sc.flags + 2 * bh, (unsigned)sc.nseg);
            else if (!fwd) ok = tc::flag_wait_geq(sc.flags + 2 * bh + 1, (unsigned)(sc.nseg - 1 - seg));
            if (!ok) fail();
            // what it wrote by bulk copy is read here by bulk copy
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        __syncthreads();
        if (fwd) {
            // ============================================= forward walk: chunk states
            master_init(seg == 0 ? (a.h0 ? a.h0 + bh * KV : nullptr) : sc.s_hand + bh * KV);
            if (n_lo < n_hi) request(n_lo, false);
            tc::fence_before_sync();
            __syncthreads();
            for (int n = n_lo; n < n_hi && !*s_fail; ++n) {
                load_inputs(n, false);
                if (n > n_lo) wait_mma();  // the previous chunk's state update has read Kt and Delta
                if (tid == 0) tc::bulk_wait_read_all();  // the previous state copy has gone out
                __syncthreads();
                master_copy();  // S as an operand
                build_tiles(false, false);
                arows();
                tc::fence_before_sync();
                __syncthreads();
                if (tid == 0) {
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int p = 0; p < 2; ++p) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_bf16(tm + TM_A, tile::desc_mn(sb + OFF_ST + p * ST_LO, 16384, ks),
                                         tile::desc_k(sb + OFF_AQK, 32, ks), ID_MN_K32, (p | ks) != 0);
                    }
                    tc::mma_commit(bar_mma);
                }
                master_decay();  // S <- diag(gamma) S in TMEM, and T, under the R products
                t_solve();
                wait_mma();
                __syncthreads();  // T is published
                // R = V - Kg S and Delta = T diag(beta) R, value column v = tid on warps 0..3
                if (warp < 4) {
                    uint32_t r[16], r2[16];
                    tc::tmem_ld16(tile::taddr(tm + TM_A, warp, 0), r);
                    tc::tmem_ld16(tile::taddr(tm + TM_A, warp, 16), r2);
                    tc::tmem_ld_wait();
                    float rr[BC];
#pragma unroll
                    for (int t = 0; t < BC; ++t)
                        rr[t] = Rv[t * VM + tid] - (__uint_as_float(r[t]) + __uint_as_float(r2[t]));
#pragma unroll
                    for (int t = 0; t < BC; ++t) {
                        float acc = 0.f;
#pragma unroll
                        for (int i = 0; i <= t; ++i) acc = fmaf(Tm[t * BC + i], bet[i] * rr[i], acc);
                        Rv[t * VM + tid] = rr[t];
                        Dl[t * VM + tid] = acc;
                    }
                }
                tc::fence_proxy_async_smem();
                __syncthreads();
                if (tid == 0) {  // R, Delta, A', T and M (contiguous), and g, for phase 2
                    float* dst = a.rd + (bh * N + n) * (size_t)RD;
                    tc::bulk_store(dst, Rv, RD_SM * 4);
                    tc::bulk_store(dst + RD_SM, XT, BC * KM * 4);
                    tc::bulk_commit();
                }
                tile_rows(Dl, OFF_DLT, 32, 16, 0);
                if (tid == 0) tc::bulk_wait_read_all();  // before the next chunk's v and g land in R, XT
                tc::fence_before_sync();
                __syncthreads();
                if (tid == 0) {  // S += Kt^T Delta (K step 0 the hi rows, 1 the lo rows)
                    tc::fence_after_sync();
#pragma unroll
                    for (int p = 0; p < 4; ++p)
                        tc::mma_bf16(tm + TM_M, tile::desc_mn(sb + OFF_KT, 4096, p >> 1),
                                     tile::desc_mn(sb + OFF_DLT, 4096, p & 1), ID_MN_MN128, 1u);
                    tc::mma_commit(bar_mma);
                    // the state copy is the chunk's checkpoint
                    tc::bulk_store(a.ckpt + (bh * N + n) * KV, sm8 + OFF_ST, kStateBytes);
                    tc::bulk_commit();
                }
            }
            if (n_hi > n_lo && !*s_fail) wait_mma();
            if (seg < sc.nseg - 1) {  // the state for the sequence's next segment
                uint32_t r0[16], r1[16];
                master_ld(r0, r1);
                float* ps = sc.s_hand + bh * KV + (size_t)col * V + 32 * qtr;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    ps[j] = __uint_as_float(r0[j]);
                    ps[16 + j] = __uint_as_float(r1[j]);
                }
            }
            if (tid == 0) tc::bulk_wait_all();  // every checkpoint and record is in global memory
            // they are read back by bulk copies, and the tiles the next item fills by bulk copy
            // were last written by generic stores
            asm volatile("fence.proxy.async.global;" ::: "memory");
            tc::fence_proxy_async_smem();
            __threadfence();
            tc::fence_before_sync();
            __syncthreads();
            if (tid == 0) tc::st_release_gpu(sc.flags + 2 * bh, (unsigned)(seg + 1));
        } else {
            // ============================================= reverse walk
            master_init(seg == sc.nseg - 1 ? (a.dhT ? a.dhT + bh * KV : nullptr) : sc.ds_hand + bh * KV);
            if (n_lo < n_hi) {
                request(n_hi - 1, true);
                request_rd(n_hi - 1);
                prefetch_state(n_hi - 1);
            }
            tc::fence_before_sync();
            __syncthreads();
            dA_acc = 0.f;
            ddt_acc = 0.f;
    for (int n = n_hi - 1; n >= n_lo && !*s_fail; --n) {
                const int t0 = n * BC, cn = min(BC, T - t0);
                load_inputs(n, true);
                prefetch_state(n - 1);
                if (n < n_hi - 1) wait_mma();  // the previous chunk's dS update has read its tiles
                build_tiles(true, false);
                if (tid == 0) tc::bulk_wait_read_all();  // the previous chunk's dq, dk, dz have left
                __syncthreads();
                master_copy();  // dS as an operand
                tc::fence_before_sync();
                __syncthreads();
                if (tid == 128) {  // dDelta^T = dS^T Kt^T + dO^T (scale M), dKt^T = dS Delta^T
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int p = 0; p < 2; ++p) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_bf16(tm + TM_A, tile::desc_mn(sb + OFF_ST + p * ST_LO, 16384, ks),
                                         tile::desc_k(sb + OFF_KT, 32, ks), ID_MN_K32, (p | ks) != 0);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_bf16(tm + TM_B, tile::desc_k(sb + OFF_ST + p * ST_LO, 128, ks),
                                         tile::desc_k(sb + OFF_DLT, 32, ks), ID_K_K32, (p | ks) != 0);
                        // A = dO^T (rows 0..15 hi, 32..47 lo of [dO ; dY] read MN-major), B = scale M^T
                        tc::mma_bf16(tm + TM_A, tile::desc_mn(sb + OFF_DOY, 8192, 2 * p),
                                     tile::desc_k(sb + OFF_AQK, 32, 0), ID_MN_K32, 1u);
                    }
                    tc::mma_commit(bar_mma);
                }
                wait_mma();
                if (tid == 0) {  // the state entering this chunk, as phase 1 kept it
                    tc::mbar_arrive_expect_tx(bar_ld, kStateBytes);
                    tc::bulk_load(sm8 + OFF_ST, a.ckpt + (bh * N + n) * KV, kStateBytes, bar_ld);
                }
                if (warp < 4) {  // dDelta, then dY = T^T dDelta
                    uint32_t r[16], r2[16];
                    tc::tmem_ld16(tile::taddr(tm + TM_A, warp, 0), r);
                    tc::tmem_ld16(tile::taddr(tm + TM_A, warp, 16), r2);
                    tc::tmem_ld_wait();
                    float dd[BC];
#pragma unroll
                    for (int t = 0; t < BC; ++t) dd[t] = __uint_as_float(r[t]) + __uint_as_float(r2[t]);
#pragma unroll
                    for (int i = 0; i < BC; ++i) {
                        float acc = 0.f;
#pragma unroll
                        for (int t = i; t < BC; ++t) acc = fmaf(Tm[t * BC + i], dd[t], acc);
                        dY[i * VM + tid] = acc;
                    }
                }
                float dq_r[4] = {0.f, 0.f, 0.f, 0.f}, dk_r[4] = {0.f, 0.f, 0.f, 0.f};
                float dG_r[4] = {0.f, 0.f, 0.f, 0.f};
                float dgl_part = 0.f;
                {  // dKt = Delta dS^T: channel col, tokens 4 qtr ..
                    uint32_t r[4], r2[4];
                    tc::tmem_ld4(tile::taddr(tm + TM_B, warp, 4 * qtr), r);
                    tc::tmem_ld4(tile::taddr(tm + TM_B, warp, 16 + 4 * qtr), r2);
                    tc::tmem_ld_wait();
                    const float gl = Gc[ci(col, (BC - 1))];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int t = 4 * qtr + u;
                        const float x = __uint_as_float(r[u]) + __uint_as_float(r2[u]);
                        const float eL = expf(gl - Gc[ci(col, t)]);
                        const float kk = Kr[ci(col, t)];
                        dk_r[u] += x * eL;
                        dG_r[u] -= x * kk * eL;
                        dgl_part += x * kk * eL;
                    }
                }
                build_tiles(true, true);  // scale M^T has been read
                __syncthreads();
                tile_rows(dY, OFF_DOY, 64, 32, 16);
                {  // the first part of dbeta_t, sum_v R_tv dY_tv (warp t), into the M slot (M is done)
                    const int t = warp;
                    float sr = 0.f;
                    for (int vv = lane; vv < V; vv += 32) sr = fmaf(Rv[t * VM + vv], dY[t * VM + vv], sr);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) sr += __shfl_xor_sync(0xffffffffu, sr, off);
                    if (lane == 0) Mm[t] = sr;
                }
                tc::fence_before_sync();
                __syncthreads();
                wait_ld();
                if (tid == 0) {  // [dQg^T | P^T] = S [dO ; dY]^T
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int p = 0; p < 2; ++p) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_bf16(tm + TM_C, tile::desc_k(sb + OFF_ST + p * ST_LO, 128, ks),
                                         tile::desc_k(sb + OFF_DOY, 64, ks), ID_K_K64, (p | ks) != 0);
                    }
                    // [dO ; dY] Delta^T (rows 0..63 of D; the M = 128 read's rows 64..127 are ignored)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_bf16(tm + TM_B, tile::desc_k(sb + OFF_DOY, 64, ks),
                                     tile::desc_k(sb + OFF_DLT, 32, ks), ID_K_K32, ks != 0);
                    tc::mma_commit(bar_mma);
                }
                {  // dgamma_c partial over the value quarter qtr (times gamma_c), then dS <- gamma dS
                    uint32_t r0[16], r1[16];
                    master_ld(r0, r1);
                    float sacc = 0.f;
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const uint32_t off = tile::kmaj_off(col, 32 * qtr + 8 * g, 128);
                        float shi[8], slo[8];
                        tile::unpack8(*reinterpret_cast<const uint4*>(sm8 + OFF_ST + off), shi);
                        tile::unpack8(*reinterpret_cast<const uint4*>(sm8 + OFF_ST + ST_LO + off), slo);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float d = __uint_as_float(g < 2 ? r0[8 * g + j] : r1[8 * (g - 2) + j]);
                            sacc = fmaf(shi[j] + slo[j], d, sacc);
                        }
                    }
                    const float gm = gam[col];
                    red[qtr * KM + col] = sacc * gm;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        r0[j] = __float_as_uint(__uint_as_float(r0[j]) * gm);
                        r1[j] = __float_as_uint(__uint_as_float(r1[j]) * gm);
                    }
                    master_st(r0, r1);
                }
                // dV = diag(beta) dY
                for (int idx = tid; idx < BC * V; idx += NT) XT[idx] = bet[idx >> 7] * dY[idx];  // dV, staged
                wait_mma();
                if (warp < 2) {  // dM = scale dO Delta^T (i <= t), dB = -dY Delta^T (i < t): rows of D
                    uint32_t r0[16], r1[16];
                    tc::tmem_ld16(tile::taddr(tm + TM_B, warp, 0), r0);
                    tc::tmem_ld16(tile::taddr(tm + TM_B, warp, 16), r1);
                    tc::tmem_ld_wait();
                    float x[BC];
#pragma unroll
                    for (int i = 0; i < BC; ++i) x[i] = __uint_as_float(r0[i]) + __uint_as_float(r1[i]);
                    float* dst = lane < 16 ? dM + lane * BC : dB + (lane - 16) * BC;
                    if (warp == 1) {  // the lo rows' share
#pragma unroll
                        for (int i = 0; i < BC; ++i) dst[i] = x[i];
                    }
                    tc::named_sync(1, 64);
                    if (warp == 0) {
                        const int t = lane & 15;
#pragma unroll
                        for (int i = 0; i < BC; ++i) {
                            const float v = x[i] + dst[i];
                            dst[i] = lane < 16 ? (i <= t ? a.scale * v : 0.f) : (i < t ? -v : 0.f);
                        }
                        __syncwarp();
                        // dbeta_t = sum_v R_tv dY_tv + sum_{i<t} A'_ti dB_ti
                        if (lane < cn) {
                            float sb2 = Mm[lane];
                            for (int i = 0; i < lane; ++i) sb2 = fmaf(Ap[lane * BC + i], dB[lane * BC + i], sb2);
                            a.dbeta[bh * T + t0 + lane] = sb2;
                        }
                    }
                }
                {  // dQg = scale dO S^T and P = dY S^T, dKg = -diag(beta) P
                    uint32_t rx[4], ry[4], rx2[4], ry2[4];
                    tc::tmem_ld4(tile::taddr(tm + TM_C, warp, 4 * qtr), rx);
                    tc::tmem_ld4(tile::taddr(tm + TM_C, warp, 16 + 4 * qtr), ry);
                    tc::tmem_ld4(tile::taddr(tm + TM_C, warp, 32 + 4 * qtr), rx2);
                    tc::tmem_ld4(tile::taddr(tm + TM_C, warp, 48 + 4 * qtr), ry2);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int t = 4 * qtr + u;
                        const float Ga = expf(Gc[ci(col, t)]);
                        const float dqg = a.scale * (__uint_as_float(rx[u]) + __uint_as_float(rx2[u]));
                        const float dkg = -bet[t] * (__uint_as_float(ry[u]) + __uint_as_float(ry2[u]));
                        dq_r[u] += dqg * Ga;
                        dk_r[u] += dkg * Ga;
                        dG_r[u] += (dqg * Qr[ci(col, t)] + dkg * Kr[ci(col, t)]) * Ga;
                    }
                }
                tc::fence_proxy_async_smem();  // R, Delta, A', T, M are done: the next chunk's may land
                tc::fence_before_sync();
                __syncthreads();
                if (n > n_lo) request_rd(n - 1);
                if (tid == 0) {
                    tc::bulk_store(a.dv + (bh * T + t0) * (size_t)V, XT, (uint32_t)(cn * V * 4));
                    tc::bulk_commit();
                }
                if (tid == 0) {  // dS += [scale Qg ; -beta Kg]^T [dO ; dY] (K steps 0, 1 hi; 2, 3 lo)
                    tc::fence_after_sync();
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks)
                            tc::mma_bf16(tm + TM_M, tile::desc_mn(sb + OFF_AQK, 8192, 2 * (p >> 1) + ks),
                                         tile::desc_mn(sb + OFF_DOY, 8192, 2 * (p & 1) + ks), ID_MN_MN128, 1u);
                    }
                    tc::mma_commit(bar_mma);
                }
                // pairwise terms of dA' = diag(beta) dB and dM, each pair's decay E = e^{G_s - G_t} (t < s)
                // taken once: thread (c = col) takes the rows s in {qtr, 7 - qtr, 8 + qtr, 15 - qtr} (30
                // pairs below the diagonal each) and sums the row terms of s and the column terms of every
                // t <= s; the sums meet in the state-copy region (free until the next chunk's copy)
                float* colP = reinterpret_cast<float*>(sm8 + OFF_ST);  // [4][BC][KM]
                float* rowP = colP + 4 * BC * KM;                       // [BC][2][KM]
                {
                    const int c = col;
                    float gs[4], ks[4], qs[4], bs[4], dMd[4], rM[4], rA[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int s = u == 0 ? qtr : u == 1 ? 7 - qtr : u == 2 ? 8 + qtr : 15 - qtr;
                        gs[u] = Gc[ci(c, s)];
                        ks[u] = Kr[ci(c, s)];
                        qs[u] = Qr[ci(c, s)];
                        bs[u] = bet[s];
                        dMd[u] = dM[s * BC + s];
                        rM[u] = dMd[u] * ks[u];  // the diagonal pair (E = 1, dB[s][s] = 0)
                        rA[u] = 0.f;
                    }
#pragma unroll
                    for (int t = 0; t < BC; ++t) {
                        const float gt = Gc[ci(c, t)], kt = Kr[ci(c, t)];
                        float cs = 0.f;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int s = u == 0 ? qtr : u == 1 ? 7 - qtr : u == 2 ? 8 + qtr : 15 - qtr;
                            if (t < s) {
                                const float E = __expf(gs[u] - gt);
                                const float w = dM[s * BC + t] * E, x = bs[u] * dB[s * BC + t] * E;
                                rM[u] = fmaf(w, kt, rM[u]);
                                rA[u] = fmaf(x, kt, rA[u]);
                                cs = fmaf(w, qs[u], fmaf(x, ks[u], cs));
                            } else if (t == s) {
                                cs = fmaf(dMd[u], qs[u], cs);
                            }
                        }
                        colP[(qtr * BC + t) * KM + c] = cs;
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int s = u == 0 ? qtr : u == 1 ? 7 - qtr : u == 2 ? 8 + qtr : 15 - qtr;
                        rowP[(2 * s) * KM + c] = rM[u];
                        rowP[(2 * s + 1) * KM + c] = rA[u];
                    }
                }
                if (tid == 0) tc::bulk_wait_read_all();  // dV has left XT
                __syncthreads();
                // this thread's tokens t = 4 qtr + r: dq += rowM, dk += rowA + col, dG += k rowA + q rowM
                // - k col (col = the column terms of dM and dA', summed over the four row owners)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int t = 4 * qtr + r;
                    const float kt = Kr[ci(col, t)], qt = Qr[ci(col, t)];
                    const float cs = (colP[t * KM + col] + colP[(BC + t) * KM + col]) +
                                     (colP[(2 * BC + t) * KM + col] + colP[(3 * BC + t) * KM + col]);
                    const float rM = rowP[(2 * t) * KM + col], rA = rowP[(2 * t + 1) * KM + col];
                    dq_r[r] += rM;
                    dk_r[r] += rA + cs;
                    dG_r[r] += kt * rA + qt * rM - kt * cs;
                }
                // dG exchange ([BC][KM] in XT), the last token's share of d(G_last), reverse cumsum,
                // gate derivative; dq and dk out
#pragma unroll
                for (int r = 0; r < 4; ++r) XT[(4 * qtr + r) * KM + col] = dG_r[r];
                red[qtr * KM + col] += dgl_part;
                __syncthreads();
                float* ost = reinterpret_cast<float*>(sm8 + OFF_ST);  // dq, dk, dz [BC][KM] each, staged
                {
                    const int c = col;
                    const float dgl = red[c] + red[KM + c] + red[2 * KM + c] + red[3 * KM + c];
                    float suffix = dgl;
                    for (int t = BC - 1; t > 4 * qtr + 3; --t) suffix += XT[t * KM + c];
#pragma unroll
                    for (int r = 3; r >= 0; --r) {
                        const int t = 4 * qtr + r;
                        suffix += XT[t * KM + c];
                        if (t < cn) {
                            // g = -e^{A_log} softplus(x) with x = z + dt_bias, and sigmoid(x) =
                            // 1 - e^{-softplus(x)} = -expm1(g e^{-A_log})
                            const float g = Gt[ci(c, t)];
                            const float dz = suffix * (-eA) * -expm1f(g * ieA);
                            ost[t * KM + c] = dq_r[r];
                            ost[(BC + t) * KM + c] = dk_r[r];
                            ost[(2 * BC + t) * KM + c] = dz;
                            ddt_acc += dz;
                            dA_acc = fmaf(suffix, g, dA_acc);
                        }
                    }
                }
                tc::fence_proxy_async_smem();
                __syncthreads();
                if (tid == 0) {
                    const size_t g0 = (bh * T + t0) * (size_t)K;
                    const uint32_t bytes = (uint32_t)(cn * K * 4);
                    tc::bulk_store(a.dq + g0, ost, bytes);
                    tc::bulk_store(a.dk + g0, ost + BC * KM, bytes);
                    tc::bulk_store(a.dz + g0, ost + 2 * BC * KM, bytes);
                    tc::bulk_commit();
                }
            }
            if (n_hi > n_lo && !*s_fail) wait_mma();  // the segment's last dS update
            if (tid == 0) tc::bulk_wait_all();  // the gradients are in global memory
            // the adjoint for the sequence's earlier segment, or dh0
            float* dst = seg > 0 ? sc.ds_hand + bh * KV : (a.dh0 ? a.dh0 + bh * KV : nullptr);
            if (dst) {
                uint32_t r0[16], r1[16];
                master_ld(r0, r1);
                float* pd = dst + (size_t)col * V + 32 * qtr;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    pd[j] = __uint_as_float(r0[j]);
                    pd[16 + j] = __uint_as_float(r1[j]);
                }
            }
            // the segment's partial sums of dA_log and ddt_bias
            const size_t ps = bh * sc.nseg + seg;
            red[qtr * KM + col] = ddt_acc;
            for (int off = 16; off > 0; off >>= 1) dA_acc += __shfl_xor_sync(0xffffffffu, dA_acc, off);
            __syncthreads();
            if (lane == 0) XT[warp] = dA_acc;
            if (tid < K) a.ddt_part[ps * K + tid] = red[tid] + red[KM + tid] + red[2 * KM + tid] + red[3 * KM + tid];
            __syncthreads();
            if (tid == 0) {
                float sacc = 0.f;
                for (int w = 0; w < NT / 32; ++w) sacc += XT[w];
                a.dA_part[ps] = sacc;
            }
            __threadfence();
            tc::fence_before_sync();
            __syncthreads();
            if (tid == 0 && seg > 0) tc::st_release_gpu(sc.flags + 2 * bh + 1, (unsigned)(sc.nseg - seg));
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tm, TM_COLS);
    }
}

// dA_log[h] = sum over b and segments of dA_part[b, h, seg];  ddt_bias[h, c] likewise of
// ddt_part[b, h, seg, c]
__global__ void kda_bwd_reduce_kernel(int B, int H, int K, int nseg, const float* __restrict__ dA_part,
                                      const float* __restrict__ ddt_part, float* __restrict__ dA_log,
                                      float* __restrict__ ddt_bias) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < H) {
        float s = 0.f;
        for (int b = 0; b < B; ++b)
            for (int g = 0; g < nseg; ++g) s += dA_part[((size_t)b * H + i) * nseg + g];
        dA_log[i] = s;
    }
    if (i < H * K) {
        const int hh = i / K, c = i - hh * K;
        float s = 0.f;
        for (int b = 0; b < B; ++b)
            for (int g = 0; g < nseg; ++g) s += ddt_part[(((size_t)b * H + hh) * nseg + g) * K + c];
        ddt_bias[i] = s;
    }
}

}  // namespace

namespace {

// Makespan, in units of one sequence's backward, of the tensor-core backward's work items taken
// in kernel order by `nsm` CTAs: the forward walk 0.37 and the reverse walk 0.63 of a sequence
// (as measured per chunk), each split evenly over nseg segments, plus 0.002 per segment for its
// handoff (the state or adjoint through global memory, a flag, the first chunk's rows).
double bwd_makespan(long long BH, int nseg, int nsm) {
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    const long long items = 2 * BH * nseg;
    for (long long i = 0; i < std::min<long long>(nsm, items); ++i) free_at.push(0.0);
    const double f = 0.37 / nseg, r = 0.63 / nseg, hand = nseg > 1 ? 0.002 : 0.0;
    std::vector<double> fdone((size_t)BH, 0.0), rdone((size_t)BH, 0.0);
    double end = 0.0;
    auto take = [&](double ready, double dur) {
        const double t = std::max(free_at.top(), ready) + dur;
        free_at.pop();
        free_at.push(t);
        end = std::max(end, t);
        return t;
    };
    for (int g = 0; g < nseg; ++g)
        for (long long b = 0; b < BH; ++b) fdone[b] = take(fdone[b], f + hand);
    for (int g = nseg - 1; g >= 0; --g)
        for (long long b = 0; b < BH; ++b) rdone[b] = take(g == nseg - 1 ? fdone[b] : rdone[b], r + hand);
    return end;
}

// Segments per walk for the tensor-core backward: of 1, 2, 4 and 8 (segments of at least 8
// chunks), the count whose schedule finishes first by at least 2 %.
int bwd_segments(long long BH, int N, int nsm) {
    if (nsm < 1 || BH > 64LL * nsm) return 1;  // many waves: little to gain
    int best = 1;
    double bm = bwd_makespan(BH, 1, nsm);
    for (int g = 2; g <= 8; g *= 2) {
        if (N < 8 * g) break;
        const double m = bwd_makespan(BH, g, nsm);
        if (m < 0.98 * bm) {
            bm = m;
            best = g;
        }
    }
    return best;
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

cudaError_t launch_chunk_backward(const BwdLaunch& L, cudaStream_t s) {
    const int B = L.B, H = L.H, T = L.T, K = L.K, V = L.V;
    const int N = (T + BC - 1) / BC;
    const size_t BH = (size_t)B * H;
    const size_t KV = (size_t)K * V;
    const bool fixed = K == 128 && V == 128;
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // the tensor-core form's schedule: nseg segments of seg_len chunks per walk
    const int nseg = fixed ? bwd_segments((long long)BH, N, nsm) : 1;
    const int seg_len = std::max(1, (N + nseg - 1) / nseg);
    const long long n_items = 2LL * (long long)BH * nseg;
    if (fixed && n_items > 0x7fffffffLL) return cudaErrorInvalidValue;
    // scratch: partial sums, the schedule's counter and flags, the handoffs, the chunk states and
    // the chunk records
    const size_t part_bytes = round256(sizeof(float) * BH * (size_t)nseg * (1 + K));
    const size_t sched_bytes = fixed ? round256(sizeof(unsigned) * (1 + 2 * BH)) : 0;
    const size_t hand_bytes = nseg > 1 ? 2 * sizeof(float) * BH * KV : 0;
    const size_t ck_bytes = sizeof(float) * BH * (size_t)N * KV;
    const size_t rd_bytes = sizeof(float) * BH * (size_t)N * (fixed ? (size_t)bwdtc::RD : (size_t)(2 * BC * V));
    char* scratch = nullptr;
    e = scratch_alloc(reinterpret_cast<void**>(&scratch),
                      part_bytes + sched_bytes + hand_bytes + ck_bytes + rd_bytes, s);
    if (e != cudaSuccess) return e;
    float* dA_part = reinterpret_cast<float*>(scratch);
    float* ddt_part = dA_part + BH * nseg;
    unsigned* sched = reinterpret_cast<unsigned*>(scratch + part_bytes);
    float* hand = reinterpret_cast<float*>(scratch + part_bytes + sched_bytes);
    float* ckpt = reinterpret_cast<float*>(scratch + part_bytes + sched_bytes + hand_bytes);
    float* rd = ckpt + BH * (size_t)N * KV;
    auto run = [&](auto io_tag, auto kc_tag) -> cudaError_t {
        using IO = decltype(io_tag);
        constexpr int KC = decltype(kc_tag)::value;
        BwdArgs<IO> a;
        a.H = H; a.T = T; a.K = K; a.V = V;
        a.q = static_cast<const IO*>(L.q); a.k = static_cast<const IO*>(L.k);
        a.v = static_cast<const IO*>(L.v); a.z = static_cast<const IO*>(L.z);
        a.beta = static_cast<const IO*>(L.beta); a.d_o = static_cast<const IO*>(L.d_o);
        a.A_log = L.A_log; a.dt_bias = L.dt_bias; a.h0 = L.h0; a.dhT = L.dhT; a.scale = L.scale;
        a.dq = L.dq; a.dk = L.dk; a.dv = L.dv; a.dz = L.dz; a.dbeta = L.dbeta; a.dh0 = L.dh0;
        a.ckpt = ckpt; a.rd = rd; a.dA_part = dA_part; a.ddt_part = ddt_part;
        cudaError_t err = cudaFuncSetAttribute(kda_chunk_bwd_kernel<IO, KC>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)BWD_SMEM_BYTES);
        if (err != cudaSuccess) return err;
        kda_chunk_bwd_kernel<IO, KC><<<(unsigned)BH, BNT, BWD_SMEM_BYTES, s>>>(a);
        return cudaGetLastError();
    };
    // K = V = 128: the tensor-core form (its state copies are the same 64 KB as an fp32 state),
    // one CTA per SM at most taking the work items of BwdSched
    auto run_tc = [&](auto io_tag) -> cudaError_t {
        using IO = decltype(io_tag);
        BwdArgs<IO> a;
        a.H = H; a.T = T; a.K = K; a.V = V;
        a.q = static_cast<const IO*>(L.q); a.k = static_cast<const IO*>(L.k);
        a.v = static_cast<const IO*>(L.v); a.z = static_cast<const IO*>(L.z);
        a.beta = static_cast<const IO*>(L.beta); a.d_o = static_cast<const IO*>(L.d_o);
        a.A_log = L.A_log; a.dt_bias = L.dt_bias; a.h0 = L.h0; a.dhT = L.dhT; a.scale = L.scale;
        a.dq = L.dq; a.dk = L.dk; a.dv = L.dv; a.dz = L.dz; a.dbeta = L.dbeta; a.dh0 = L.dh0;
        a.ckpt = ckpt; a.rd = rd; a.dA_part = dA_part; a.ddt_part = ddt_part;
        constexpr size_t smem = bwdtc::smem_bytes<IO>();
        cudaError_t err = cudaFuncSetAttribute(kda_chunk_bwd_tc_kernel<IO>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        if ((err = cudaMemsetAsync(sched, 0, sched_bytes, s)) != cudaSuccess) return err;
        const BwdSched sc{nseg, seg_len, (int)n_items, reinterpret_cast<int*>(sched), sched + 1,
                          nseg > 1 ? hand : nullptr, nseg > 1 ? hand + BH * KV : nullptr};
        const unsigned grid = (unsigned)std::min<long long>(n_items, nsm);
        kda_chunk_bwd_tc_kernel<IO><<<grid, bwdtc::NT, smem, s>>>(a, sc);
        return cudaGetLastError();
    };
    using Any = std::integral_constant<int, 0>;
    if (L.io == KDA_BF16)
        e = fixed ? run_tc(__nv_bfloat16{}) : run(__nv_bfloat16{}, Any{});
    else
        e = fixed ? run_tc(float{}) : run(float{}, Any{});
    if (e == cudaSuccess) {
        const int n = H * K;
        kda_bwd_reduce_kernel<<<(n + 255) / 256, 256, 0, s>>>(B, H, K, nseg, dA_part, ddt_part,
                                                               L.dA_log, L.ddt_bias);
        e = cudaGetLastError();
        count_launches(2);
    }
    const cudaError_t ef = scratch_free(scratch, s);
    return e != cudaSuccess ? e : ef;
}

cudaError_t read_and_clear_bwd_timeout(int* timed_out) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_kda_bwd_timeout, sizeof(int));
    if (e != cudaSuccess) return e;
    *timed_out = v;
    if (v) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_kda_bwd_timeout, &zero, sizeof(int));
    }
    return e;
}

}  // namespace kda
