// chunk_carry.cu -- the sequential half of the split KDA chunked forward (bf16 I/O,
// K = V = 128, chunk C = 64): the inter-chunk state carry and the output, fed by the
// per-chunk operands that the chunk-parallel prep kernel wrote.
//
// Per (b, h) sequence one CTA (16 warps) keeps the fp32 state S (K x V) in TMEM and walks
// the chunks of a segment in order; per chunk n (kda-adjoint-2026-10-01, section 2, with
// the read scale of kdafix-2026-10-02 "Fix 2"):
//
//   C1  D = [(W S)^T | (Q Gamma S)^T]: S^T W^T and S^T (Q Gamma)^T, the latter with Q Gamma
//       as a K-major operand [t][c]                                 tcgen05, S as a bf16 operand
//   C2  Delta^T = U^T - (W S)^T
//   C3  (M Delta)^T onto (Q Gamma S)^T, then o = scale (Q Gamma S + M Delta) -> bf16 to HBM,
//       and S <- diag(Gamma_last) S + K~^T Delta,  K~ = K e^{G_last - G}  tcgen05, fp32 in TMEM
//
// which is the chunked WY form of the per-token recurrence S <- diag(alpha) S,
// u = v - S^T k, S <- S + beta k u^T, o = S^T (scale q): with Q' = Q Gamma - M W and U' = M U
// the output scale (Q' S + U') of the WY form is scale (Q Gamma S + M Delta).  The operands of
// a chunk arrive by TMA into one of two stages while the previous chunk is processed.
//
// The chunk-parallel state scan.  Per chunk the carry is affine in the state,
//     S_{n+1} = P_n S_n + Z_n,   P_n = diag(Gamma_last) - K~^T W,   Z_n = K~^T U,
// so a run of chunks maps its entering state S to P S + Z with P the product of the P_n and
// Z the state the run reaches from S = 0.  The kernel below therefore also runs
// sub-segments of a sequence in parallel (grid = sequences x sub-segments), in three roles:
// the plain carry from a given entering state (writing o), the carry from S = 0 (giving Z,
// no o) and the carry of the K x K matrix P from the identity with U = 0 (giving P, no o).
// kda_carry_combine_kernel then walks the sub-segments of each sequence in order,
// S_{j+1} = P_j S_j + Z_j in fp32, and the plain carry runs every sub-segment from its S_j.
#include <cuda.h>
#include <stddef.h>

#include "chunk_tiles.cuh"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace kda {

__device__ int g_kda_carry_timeout;

namespace {

using namespace tile;
constexpr int NT2 = 512;

// ---- shared memory map (bytes from a 1024-byte aligned base)
constexpr uint32_t K2_S = 0;            // 32 KB S bf16, MN-major [c][v] (2 atoms)
constexpr uint32_t K2_DELTA = 32768;    // 16 KB Delta^T, K-major [v][t]
constexpr uint32_t K2_STAGE = 49152;    // two operand stages
// one stage: W^T (MN-major [c][t]), Q Gamma (K-major [t][c], 2 atoms of 8 KB), U^T (K-major
// [v][t]), K~ (MN-major [t][c], 2 atoms of 8 KB), M (K-major [t][s]), Gamma_last.
constexpr uint32_t ST_WQ = 0, ST_UU = 32768, ST_KT = 49152, ST_MM = 65536, ST_GL = 73728;
constexpr uint32_t ST_BYTES = 74752;  // 73 KB, a multiple of 1024
constexpr uint32_t ST_TX = (uint32_t)kItemBytes;
constexpr uint32_t K2_MISC = K2_STAGE + 2 * ST_BYTES;

struct CarryMisc {
    alignas(8) uint64_t bar_full[2];  // TMA: one stage's operands
    uint64_t bar_mma;                 // tensor-core commits (C1, C3 alternate)
    uint64_t bar_o;                   // tensor-core commit: M Delta (before C3)
    uint32_t tmem_base;
};
constexpr uint32_t K2_SMEM = K2_MISC + sizeof(CarryMisc) + 1024;
static_assert(K2_SMEM <= 227 * 1024, "carry kernel shared memory");
static_assert(ST_TX <= ST_BYTES && ST_GL + kItemGL <= ST_BYTES && ST_MM + kItemMM <= ST_GL &&
                  ST_KT + kItemKT <= ST_MM && ST_UU + kItemUU <= ST_KT,
              "stage layout");

constexpr uint32_t TM_S2 = 0;    // fp32 state, lanes = key channel c, cols = v   (128)
constexpr uint32_t TM_D2 = 128;  // [(W S)^T | (Q Gamma S)^T], + (M Delta)^T above (128)
constexpr uint32_t IDESC_SW2 = tc::idesc_bf16(128, 64, 1, 1);  // C1, W half (B MN-major)
constexpr uint32_t IDESC_SG2 = tc::idesc_bf16(128, 64, 1, 0);  // C1, Q Gamma half (B K-major)
constexpr uint32_t IDESC_SK2 = tc::idesc_bf16(128, 128, 1, 0);
constexpr uint32_t IDESC_MD2 = tc::idesc_bf16(128, 64, 0, 0);

}  // namespace

__global__ void __launch_bounds__(NT2, 1)
    kda_chunk_carry_kernel(const __grid_constant__ CUtensorMap tm_wq,
                           const __grid_constant__ CUtensorMap tm_qg,
                           const __grid_constant__ CUtensorMap tm_uu,
                           const __grid_constant__ CUtensorMap tm_kt,
                           const uint8_t* __restrict__ mm, const float* __restrict__ gl, int T,
                           int seg_n0, int seg_len,
                           float scale, const float* h_in, __nv_bfloat16* __restrict__ out,
                           float* h_out, CarryGrid cg) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    const uint32_t sb = tc::smem_u32(sm);
    CarryMisc& ms = *reinterpret_cast<CarryMisc*>(sm + K2_MISC);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // warp w reaches TMEM lanes 32 (w & 3) ..; the four warps of a quarter split the columns
    const int q4 = warp & 3, part = warp >> 2, row = q4 * 32 + lane;
    // this CTA: sequence bh, sub-segment sub of the segment's chunks [j0, j1), and its role
    const int nbs = cg.BH * cg.nsub;
    const int role = cg.scan_roles ? 1 + (int)blockIdx.x / nbs : 0;  // 0: plain, 1: Z, 2: P
    const int rid = (int)blockIdx.x % nbs;
    const size_t bh = rid % cg.BH;
    const int sub = rid / cg.BH;
    const int j0 = min(seg_len, sub * cg.sub_len), j1 = min(seg_len, j0 + cg.sub_len);
    const bool zero_u = role == 2, write_o = role == 0 && out != nullptr;
    // entering state (plain role: h_in laid out [sub][bh]; Z role: zero; P role: identity) and
    // where the leaving state goes (plain role: h_out of the sequence, last sub-segment only;
    // Z and P roles: their [sub][bh] buffers)
    const float* sin = role == 0 && h_in ? h_in + ((size_t)sub * cg.BH + bh) * KD * VD : nullptr;
    float* sout = role == 0 ? (sub == cg.nsub - 1 && h_out ? h_out + bh * KD * VD : nullptr)
                            : (role == 1 ? cg.zbuf : cg.pbuf) + ((size_t)sub * cg.BH + bh) * KD * VD;

    if (tid == 0) {
        tc::mbar_init(&ms.bar_full[0], 1);
        tc::mbar_init(&ms.bar_full[1], 1);
        tc::mbar_init(&ms.bar_mma, 1);
        tc::mbar_init(&ms.bar_o, 1);
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&tm_wq);
        tc::tma_prefetch_desc(&tm_qg);
        tc::tma_prefetch_desc(&tm_uu);
        tc::tma_prefetch_desc(&tm_kt);
    }
    if (warp == 0) {
        tc::tmem_alloc(&ms.tmem_base, 256);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = ms.tmem_base;

    // the operands of chunk j of the segment into stage s
    auto issue = [&](int j, int s) {
        uint8_t* st = sm + K2_STAGE + s * ST_BYTES;
        const int item = (int)bh * seg_len + j;
        uint64_t* bar = &ms.bar_full[s];
        // the P role carries U = 0; only the plain role makes o (and reads M)
        tc::mbar_arrive_expect_tx(bar, ST_TX - (zero_u ? (uint32_t)kItemUU : 0u) -
                                           (write_o ? 0u : (uint32_t)kItemMM));
        tc::tma_load_3d(st + ST_WQ, &tm_wq, 0, 0, 2 * item, bar);
        tc::tma_load_3d(st + ST_WQ + 16384, &tm_qg, 0, 0, 4 * item + 2, bar);
        tc::tma_load_3d(st + ST_WQ + 24576, &tm_qg, 0, 0, 4 * item + 3, bar);
        if (!zero_u) tc::tma_load_3d(st + ST_UU, &tm_uu, 0, 0, item, bar);
        tc::tma_load_3d(st + ST_KT, &tm_kt, 0, 0, item, bar);
        tc::tma_load_3d(st + ST_KT + 8192, &tm_kt, 64, 0, item, bar);
        if (write_o) tc::bulk_load(st + ST_MM, mm + (size_t)item * kItemMM, (uint32_t)kItemMM, bar);
        tc::bulk_load(st + ST_GL, gl + (size_t)item * KD, (uint32_t)kItemGL, bar);
    };
    if (tid == 0 && j1 > j0) {
        issue(j0, 0);
        if (j1 > j0 + 1) issue(j0 + 1, 1);
    }

    // Initial state: fp32 into TMEM (lane c), bf16 copy as the MN-major operand [c][v].
    {
        const int c = row;
#pragma unroll 1
        for (int v0 = 32 * part; v0 < 32 * part + 32; v0 += 16) {
            float f[16];
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (sin) x = *reinterpret_cast<const float4*>(sin + (size_t)c * VD + v0 + j);
                f[j] = x.x; f[j + 1] = x.y; f[j + 2] = x.z; f[j + 3] = x.w;
            }
            if (role == 2) {  // the identity
#pragma unroll
                for (int j = 0; j < 16; ++j) f[j] = (c == v0 + j) ? 1.f : 0.f;
            }
            uint32_t r[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(f[j]);
            tc::tmem_st16(taddr(tmem, warp, TM_S2 + v0), r);
            store16_mn(sm + K2_S, c, v0, 16384, f);
        }
        tc::tmem_st_wait();
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    uint32_t ph_full = 0u, ph_m = 0u, ph_o = 0u;  // ph_full: bit s = parity of stage s
    bool failed = false;
#define KDA_CARRY_WAIT(bar, ph)                                          \
    do {                                                                 \
        const bool ok_ = tid != 0 || tc::mbar_wait(&(bar), ph);          \
        ph ^= 1u;                                                        \
        if (__syncthreads_or(!ok_)) failed = true;                       \
        tc::fence_after_sync();                                          \
    } while (0)

    // The operands of chunk j are waited for at the barrier that ends chunk j - 1 (or here).
    if (j1 > j0) {
        const bool ok = tid != 0 || tc::mbar_wait(&ms.bar_full[0], 0u);
        ph_full ^= 1u;
        if (__syncthreads_or(!ok)) failed = true;
        tc::fence_after_sync();
    }
    for (int j = j0; j < j1 && !failed; ++j) {
        const int s = (j - j0) & 1;
        uint8_t* st = sm + K2_STAGE + s * ST_BYTES;
        const uint32_t stb = sb + K2_STAGE + s * ST_BYTES;
        const int t0 = (seg_n0 + j) * C, cn = min(C, T - t0);
        // ---------------------------------------------------------------- K2: C1 + decay
        // stage s ^ 1 was consumed by the previous chunk: refill it two chunks ahead of that one
        // (a thread of warp 1, so that thread 0 issues C1 at once)
        if (tid == 32 && j >= j0 + 1 && j + 1 < j1) issue(j + 1, s ^ 1);
        // C1: D[v][t'] = sum_c S[c][v] W^T[c][t'] (t' < 64) under its own commit (Delta waits
        // for it), then sum_c S[c][v] QG[t'][c] above, which runs beside Delta (only the plain
        // role writes o; M Delta's commit covers it)
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_bf16(tmem + TM_D2, desc_mn(sb + K2_S, 16384, ks),
                             desc_mn(stb + ST_WQ, 16384, ks), IDESC_SW2, ks > 0);
            tc::mma_commit(&ms.bar_mma);
            if (write_o) {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_bf16(tmem + TM_D2 + 64, desc_mn(sb + K2_S, 16384, ks),
                                 desc_k(stb + ST_WQ + 16384, 64, ks), IDESC_SG2, ks > 0);
            }
        }
        // meanwhile: S <- diag(Gamma_last) S in TMEM (row c, this warp's 32 columns)
        {
            const float g = reinterpret_cast<const float*>(st + ST_GL)[row];
            {
                const int v0 = 32 * part;
                uint32_t d0[16], d1[16];
                tc::tmem_ld16(taddr(tmem, warp, TM_S2 + v0), d0);
                tc::tmem_ld16(taddr(tmem, warp, TM_S2 + v0 + 16), d1);
                tc::tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    d0[i] = __float_as_uint(__uint_as_float(d0[i]) * g);
                    d1[i] = __float_as_uint(__uint_as_float(d1[i]) * g);
                }
                tc::tmem_st16(taddr(tmem, warp, TM_S2 + v0), d0);
                tc::tmem_st16(taddr(tmem, warp, TM_S2 + v0 + 16), d1);
            }
            tc::tmem_st_wait();
        }
        tc::fence_before_sync();
        KDA_CARRY_WAIT(ms.bar_mma, ph_m);
        if (failed) break;
        // ---------------------------------------------------------------- K2: C2
        // C2: lane v, tokens 16 part ..: Delta^T -> K-major [v][t] (C3 waits for it)
        const int v = row, tb = 16 * part;
        {
            uint32_t dw[16];
            tc::tmem_ld16(taddr(tmem, warp, TM_D2 + tb), dw);
            float u[16];
            if (zero_u) {
#pragma unroll
                for (int i = 0; i < 16; ++i) u[i] = 0.f;
            } else {
                load16_k(st + ST_UU, v, tb, 128, u);
            }
            tc::tmem_ld_wait();
            float f[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) f[i] = u[i] - __uint_as_float(dw[i]);
            store16_k(sm + K2_DELTA, v, tb, 128, f);
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        // ---------------------------------------------------------------- K2: C3 + o out
        // (M Delta)^T onto (Q Gamma S)^T (its own commit), then C3: S += K~^T Delta, while
        // this thread's o values go out
        if (tid == 0) {
            if (write_o) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + TM_D2 + 64, desc_k(sb + K2_DELTA, 128, ks),
                                 desc_k(stb + ST_MM, 64, ks), IDESC_MD2, 1u);
                tc::mma_commit(&ms.bar_o);
            }
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_bf16(tmem + TM_S2, desc_mn(stb + ST_KT, 8192, ks),
                             desc_k(sb + K2_DELTA, 128, ks), IDESC_SK2, 1u);
            tc::mma_commit(&ms.bar_mma);
        }
        bool ok_o = true;
        if (write_o) {
            // every thread waits for M Delta itself (no CTA barrier in between); a timeout,
            // made warp-uniform for the lane exchange of the stores, skips them and is
            // counted at the barrier after C3
            ok_o = __all_sync(0xffffffffu, tc::mbar_wait(&ms.bar_o, ph_o));
            ph_o ^= 1u;
            if (ok_o) {
                tc::fence_after_sync();
                uint32_t d[16];
                tc::tmem_ld16(taddr(tmem, warp, TM_D2 + 64 + tb), d);
                tc::tmem_ld_wait();
                float o[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) o[i] = scale * __uint_as_float(d[i]);
                store_o16_pairs(out + (bh * T + t0 + tb) * VD, v, lane, cn - tb, o);
            }
        }
        {
            const bool ok = tid != 0 || tc::mbar_wait(&ms.bar_mma, ph_m);
            ph_m ^= 1u;
            if (__syncthreads_or(!ok || !ok_o)) failed = true;
            tc::fence_after_sync();
        }
        if (failed) break;

        // ---------------------------------------------------------------- K2: S to bf16
        // S (fp32, TMEM) -> bf16 operand [c][v]
        {
            const int c = row;
            {
                const int v0 = 32 * part;
                uint32_t d0[16], d1[16];
                tc::tmem_ld16(taddr(tmem, warp, TM_S2 + v0), d0);
                tc::tmem_ld16(taddr(tmem, warp, TM_S2 + v0 + 16), d1);
                tc::tmem_ld_wait();
                float f[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(d0[i]);
                store16_mn(sm + K2_S, c, v0, 16384, f);
#pragma unroll
                for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(d1[i]);
                store16_mn(sm + K2_S, c, v0 + 16, 16384, f);
            }
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        {
            // S is ready for the next C1; the next chunk's operands are waited for here too
            bool ok = true;
            if (j + 1 < j1) {
                ok = tid != 0 || tc::mbar_wait(&ms.bar_full[s ^ 1], (ph_full >> (s ^ 1)) & 1u);
                ph_full ^= 1u << (s ^ 1);
            }
            if (__syncthreads_or(!ok)) failed = true;
        }
        tc::fence_after_sync();
    }
#undef KDA_CARRY_WAIT

    if (!failed && sout) {
        const int c = row;
#pragma unroll 1
        for (int v0 = 32 * part; v0 < 32 * part + 32; v0 += 16) {
            uint32_t d[16];
            tc::tmem_ld16(taddr(tmem, warp, TM_S2 + v0), d);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(sout + (size_t)c * VD + v0 + i) =
                    make_float4(__uint_as_float(d[i]), __uint_as_float(d[i + 1]),
                                __uint_as_float(d[i + 2]), __uint_as_float(d[i + 3]));
        }
    }
    if (failed && tid == 0) {
        atomicExch(&g_kda_carry_timeout, 1);
        // give the tensor-core and TMA work still in flight a bounded chance to finish
        tc::mbar_wait(&ms.bar_mma, ph_m, 200000000ull);
        if (write_o) tc::mbar_wait(&ms.bar_o, ph_o, 200000000ull);
        tc::mbar_wait(&ms.bar_full[0], ph_full & 1u, 200000000ull);
        tc::mbar_wait(&ms.bar_full[1], (ph_full >> 1) & 1u, 200000000ull);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

cudaError_t launch_chunk_carry(const SplitOperands& ops, int BH, int T, int seg_n0, int seg_len,
                               float scale, const float* h_in, __nv_bfloat16* out, float* h_out,
                               cudaStream_t s) {
    return launch_chunk_carry_grid(ops, T, seg_n0, seg_len, scale, h_in, out, h_out,
                                   CarryGrid{BH, 1, seg_len, 0, nullptr, nullptr}, s);
}

cudaError_t launch_chunk_carry_grid(const SplitOperands& ops, int T, int seg_n0, int seg_len,
                                    float scale, const float* h_in, __nv_bfloat16* out,
                                    float* h_out, const CarryGrid& cg, cudaStream_t s) {
    cudaError_t err = cudaFuncSetAttribute(kda_chunk_carry_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)K2_SMEM);
    if (err != cudaSuccess) return err;
    const int grid = cg.BH * cg.nsub * (cg.scan_roles ? 2 : 1);
    if (grid < 1) return cudaSuccess;
    kda_chunk_carry_kernel<<<grid, NT2, K2_SMEM, s>>>(ops.wq, ops.qg, ops.uu, ops.kt, ops.mm, ops.gl, T,
                                                       seg_n0, seg_len, scale, h_in, out, h_out, cg);
    count_launches(1);
    return cudaGetLastError();
}

// The sequential half of the scan: per sequence (blockIdx.x / 8) and 16-column slice of the
// state (blockIdx.x % 8), S_0 = the segment's entering state (h_in, or zero when it is null),
// then S_{j+1} = P_j S_j + Z_j for j = 0 .. nsub - 2, every S_j written to s_out [j][bh] for
// the plain carry of sub-segment j.  fp32 throughout: P_j and Z_j come from the carry's TMEM
// state, and S is kept in shared memory between steps.  Thread (rb, cb) = (tid / 8, tid % 8)
// owns the 4 x 2 block of rows 4 rb .. and slice columns 2 cb ..; P_j sits transposed in
// shared memory (Pt[k][c]), so a step reads one float4 of P and one float2 of S per 8 FMAs,
// and P_{j+1} and Z_{j+1} are loaded into registers while step j computes.  Each output is Z
// plus the products over k in ascending order.
constexpr int kCmbThreads = 256, kCmbSlices = 8, kCmbW = VD / kCmbSlices;
constexpr size_t kCmbSmem = (size_t)KD * KD * sizeof(float) + (size_t)KD * kCmbW * sizeof(float);
static_assert(kCmbW == 16 && (KD / 4) * (kCmbW / 2) == kCmbThreads, "combine blocking");
__global__ void __launch_bounds__(kCmbThreads)
    kda_carry_combine_kernel(int BH, int nsub, const float* __restrict__ h_in,
                             const float* __restrict__ pbuf, const float* __restrict__ zbuf,
                             float* __restrict__ s_out) {
    extern __shared__ float4 cmb_smem[];
    float* Pt = reinterpret_cast<float*>(cmb_smem);  // [k][c], 128 x 128
    float* Ss = Pt + KD * KD;                         // [k][slice column], 128 x 16
    const int tid = threadIdx.x;
    const size_t bh = blockIdx.x / kCmbSlices;
    const int v0 = kCmbW * (blockIdx.x % kCmbSlices);
    const size_t KV = (size_t)KD * VD;
    const int r0 = 4 * (tid >> 3), c0 = 2 * (tid & 7);
    // P_j into registers: float4 f = tid + 256 m holds row r = f % 128, columns 4 (f / 128) ..
    float4 pr[16];
    float2 zr[4];
    auto load_pz = [&](int j) {
        const float* P = pbuf + ((size_t)j * BH + bh) * KV;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int f = tid + kCmbThreads * m, r = f & (KD - 1), k4 = 4 * (f >> 7);
            pr[m] = __ldcg(reinterpret_cast<const float4*>(P + (size_t)r * KD + k4));
        }
        const float* Z = zbuf + ((size_t)j * BH + bh) * KV + v0 + c0;
#pragma unroll
        for (int a = 0; a < 4; ++a) zr[a] = __ldcg(reinterpret_cast<const float2*>(Z + (size_t)(r0 + a) * VD));
    };
    auto store_pt = [&]() {
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int f = tid + kCmbThreads * m, r = f & (KD - 1), k4 = 4 * (f >> 7);
            Pt[(k4 + 0) * KD + r] = pr[m].x;
            Pt[(k4 + 1) * KD + r] = pr[m].y;
            Pt[(k4 + 2) * KD + r] = pr[m].z;
            Pt[(k4 + 3) * KD + r] = pr[m].w;
        }
    };
    auto out_block = [&](int j, const float2 (&x)[4]) {
        float* dst = s_out + ((size_t)j * BH + bh) * KV + v0 + c0;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            *reinterpret_cast<float2*>(dst + (size_t)(r0 + a) * VD) = x[a];
            *reinterpret_cast<float2*>(Ss + (r0 + a) * kCmbW + c0) = x[a];
        }
    };
    {
        float2 x[4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
            x[a] = h_in ? *reinterpret_cast<const float2*>(h_in + bh * KV + (size_t)(r0 + a) * VD + v0 + c0)
                        : make_float2(0.f, 0.f);
        out_block(0, x);
    }
    if (nsub > 1) {
        load_pz(0);
        store_pt();
    }
    for (int j = 0; j + 1 < nsub; ++j) {
        __syncthreads();  // P_j and S_j are in shared memory
        float2 acc[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) acc[a] = zr[a];
        if (j + 2 < nsub) load_pz(j + 1);
#pragma unroll 4
        for (int k = 0; k < KD; ++k) {
            const float4 p = *reinterpret_cast<const float4*>(Pt + k * KD + r0);
            const float2 x = *reinterpret_cast<const float2*>(Ss + k * kCmbW + c0);
            const float pa[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                acc[a].x = fmaf(pa[a], x.x, acc[a].x);
                acc[a].y = fmaf(pa[a], x.y, acc[a].y);
            }
        }
        __syncthreads();  // every read of P_j and S_j is done
        out_block(j + 1, acc);
        if (j + 2 < nsub) store_pt();
    }
}

cudaError_t launch_carry_combine(int BH, int nsub, const float* h_in, const float* pbuf,
                                 const float* zbuf, float* s_out, cudaStream_t s) {
    cudaError_t err = cudaFuncSetAttribute(kda_carry_combine_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kCmbSmem);
    if (err != cudaSuccess) return err;
    kda_carry_combine_kernel<<<BH * kCmbSlices, kCmbThreads, kCmbSmem, s>>>(BH, nsub, h_in, pbuf,
                                                                          zbuf, s_out);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t read_and_clear_carry_timeout(int* timed_out) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_kda_carry_timeout, sizeof(int));
    if (e != cudaSuccess) return e;
    *timed_out = v;
    if (v) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_kda_carry_timeout, &zero, sizeof(int));
    }
    return e;
}

}  // namespace kda
